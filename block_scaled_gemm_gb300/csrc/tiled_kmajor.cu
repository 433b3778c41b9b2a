// tiled_kmajor.cu -- the tiled kernel's instantiations for B given N x K
// (K contiguous), compiled apart from mxgemm.cu so that the two build in
// parallel.
#include "tiled_launch.cuh"

namespace mxg {

int launch_tiled_kmajor(int CG, TiledLaunch &L, const TiledMaps &m, const KParams &kp, int units,
                        cudaStream_t stream) {
  return CG == 2 ? launch_tiled_epi<2, kEpiBKMajor>(L, m, kp, units, stream)
                 : launch_tiled_epi<1, kEpiBKMajor>(L, m, kp, units, stream);
}

}  // namespace mxg
