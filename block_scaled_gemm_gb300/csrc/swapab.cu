// swapab.cu -- launches of the skinny-problem kernel (swapab_kernel.cuh),
// compiled apart from mxgemm.cu so that the two build in parallel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "swapab.h"
#include "swapab_kernel.cuh"

namespace mxg {

namespace {

template <int NT, bool BF16, bool ACC>
int launch_nt(const CUtensorMap &tBt, const CUtensorMap &tAt, const CUtensorMap &tSB,
              const CUtensorMap &tSA, const SwapParams &p, int grid, cudaStream_t stream,
              bool *attr_done) {
  using S = SwapCfg<NT>;
  auto kern = mxgemm_swapab_kernel<NT, BF16, ACC>;
  if (!*attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES) !=
        cudaSuccess) {
      cudaGetLastError();
      return 5;  // MXGEMM_ERR_CUDA
    }
    *attr_done = true;
  }
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(S::THREADS, 1, 1);
  cfg.dynamicSmemBytes = S::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  // may start while a B re-pitch before it finishes (griddepcontrol.wait
  // guards its global accesses)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.splits > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(p.splits);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  if (cudaLaunchKernelEx(&cfg, kern, tBt, tAt, tSB, tSA, p) != cudaSuccess) {
    cudaGetLastError();
    return 5;
  }
  return 0;
}

template <int NT>
int launch_epi(const CUtensorMap &tBt, const CUtensorMap &tAt, const CUtensorMap &tSB,
               const CUtensorMap &tSA, const SwapParams &p, bool bf16, int grid,
               cudaStream_t stream, bool *attr_done) {
  const int e = (bf16 ? 1 : 0) | (p.use_acc ? 2 : 0);
  switch (e) {
    case 0: return launch_nt<NT, false, false>(tBt, tAt, tSB, tSA, p, grid, stream, attr_done + 0);
    case 1: return launch_nt<NT, true, false>(tBt, tAt, tSB, tSA, p, grid, stream, attr_done + 1);
    case 2: return launch_nt<NT, false, true>(tBt, tAt, tSB, tSA, p, grid, stream, attr_done + 2);
    default: return launch_nt<NT, true, true>(tBt, tAt, tSB, tSA, p, grid, stream, attr_done + 3);
  }
}

}  // namespace

int swapab_class(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

int swapab_max_splits(int nt) {
  switch (nt) {
    case 16: return swap_max_splits<16>();
    case 32: return swap_max_splits<32>();
    case 64: return swap_max_splits<64>();
    default: return swap_max_splits<128>();
  }
}

int swapab_launch(const CUtensorMap &tBt, const CUtensorMap &tAt, const CUtensorMap &tSB,
                  const CUtensorMap &tSA, const SwapParams &p, bool bf16, int grid,
                  cudaStream_t stream, bool (*attr_done)[4]) {
  switch (swapab_class(p.M)) {
    case 16: return launch_epi<16>(tBt, tAt, tSB, tSA, p, bf16, grid, stream, attr_done[0]);
    case 32: return launch_epi<32>(tBt, tAt, tSB, tSA, p, bf16, grid, stream, attr_done[1]);
    case 64: return launch_epi<64>(tBt, tAt, tSB, tSA, p, bf16, grid, stream, attr_done[2]);
    default: return launch_epi<128>(tBt, tAt, tSB, tSA, p, bf16, grid, stream, attr_done[3]);
  }
}

}  // namespace mxg
