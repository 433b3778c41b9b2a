// tiled_launch.cuh -- launch of one instantiation of the tiled kernel
// (mxgemm_kernel.cuh), shared by the translation units that instantiate it:
// mxgemm.cu (B given K x N) and tiled_kmajor.cu (B given N x K).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "mxgemm.h"
#include "mxgemm_kernel.cuh"

namespace mxg {

// What a launch needs from the caller's handle.
struct TiledLaunch {
  bool *attr_set;         // [16], per epilogue variant: shared-memory attribute set
  cudaEvent_t before;     // optional events recorded around the launch
  cudaEvent_t after;
  int64_t *launches;      // incremented per launch
};

struct TiledMaps {
  const CUtensorMap *A, *B, *B64, *SFA, *SFB, *C;
};

template <int CG, int EPI>
int launch_tiled(TiledLaunch &L, const TiledMaps &m, const KParams &kp, int units,
                 cudaStream_t stream) {
  using C = Cfg<CG>;
  auto kern = mxgemm_kernel<CG, EPI>;
  if (!L.attr_set[EPI]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
        cudaSuccess) {
      cudaGetLastError();
      return MXGEMM_ERR_CUDA;
    }
    L.attr_set[EPI] = true;
  }
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(units * CG), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  // the kernel may start while the prepass before it finishes; it waits
  // (griddepcontrol.wait) before the global accesses that depend on it
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (CG == 2) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  if (L.before && cudaEventRecord(L.before, stream) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  if (cudaLaunchKernelEx(&cfg, kern, *m.A, *m.B, *m.B64, *m.SFA, *m.SFB, *m.C, kp) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  ++*L.launches;
  if (L.after && cudaEventRecord(L.after, stream) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  return MXGEMM_OK;
}

// The instantiation for a run's epilogue (output type, use_acc, TMA or
// direct stores) with B layout bits `BASE` (0, or kEpiBKMajor).
template <int CG, int BASE>
int launch_tiled_epi(TiledLaunch &L, const TiledMaps &m, const KParams &kp, int units,
                     cudaStream_t stream) {
  const int epi = (kp.out_bf16 ? kEpiBF16 : 0) | (kp.use_acc ? kEpiAcc : 0) | (kp.tma_store ? kEpiTma : 0);
  switch (epi) {
    case 0: return launch_tiled<CG, BASE | 0>(L, m, kp, units, stream);
    case 1: return launch_tiled<CG, BASE | 1>(L, m, kp, units, stream);
    case 2: return launch_tiled<CG, BASE | 2>(L, m, kp, units, stream);
    case 3: return launch_tiled<CG, BASE | 3>(L, m, kp, units, stream);
    case 4: return launch_tiled<CG, BASE | 4>(L, m, kp, units, stream);
    case 5: return launch_tiled<CG, BASE | 5>(L, m, kp, units, stream);
    case 6: return launch_tiled<CG, BASE | 6>(L, m, kp, units, stream);
    default: return launch_tiled<CG, BASE | 7>(L, m, kp, units, stream);
  }
}

// The variants with B given N x K (defined in tiled_kmajor.cu).
int launch_tiled_kmajor(int CG, TiledLaunch &L, const TiledMaps &m, const KParams &kp, int units,
                        cudaStream_t stream);

}  // namespace mxg
