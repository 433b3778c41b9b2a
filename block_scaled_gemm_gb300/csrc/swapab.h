// swapab.h -- host interface of the skinny-problem (M <= 128) kernel between
// the library's translation units (not part of the C interface).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace mxg {

struct SwapParams;

// Accumulator width class of the kernel instantiation for M rows: 16, 32,
// 64 or 128 (M <= 128).
int swapab_class(int M);

// Largest cluster (K split) the instantiation of class `nt` can reduce.
int swapab_max_splits(int nt);

// Launch the kernel: grid = 128-column blocks x p.splits CTAs, clusters of
// p.splits along x.  attr_done[class][epilogue] records which
// instantiations have had their shared-memory attribute set.  Returns 0 or
// MXGEMM_ERR_CUDA.
int swapab_launch(const CUtensorMap &tBt, const CUtensorMap &tAt, const CUtensorMap &tSB,
                  const CUtensorMap &tSA, const SwapParams &p, bool bf16, int grid,
                  cudaStream_t stream, bool (*attr_done)[4]);

}  // namespace mxg
