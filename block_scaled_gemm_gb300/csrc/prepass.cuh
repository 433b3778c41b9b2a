// prepass.cuh -- the HBM-bound prepasses that run before the GEMM kernel:
// the scale repack (row-major E8M0 bytes -> the tcgen05.cp chunk layout) and
// the B row re-pitch for N % 16 != 0.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace mxg {

// ---------------------------------------------------------------- prepasses

// Scale repack (CTA-pair tiles; single CTAs build the same chunks in the
// kernel): row-major scales S[rows][kb_count] -> 512-byte chunks.  Chunk
// g = (tile * k_steps + ks) * atoms + a covers rows (tile*atoms + a)*128 + r,
// r in [0,128), and K-blocks ks*4 + j, j in [0,4); its byte
// (r % 32) * 16 + (r / 32) * 4 + j holds that scale (127 = 1.0 where the row
// or K-block is out of range).  This is the 32-row x 16-byte source shape of
// tcgen05.cp .32x128b.warpx4, which replicates it into the four TMEM lane
// quarters: TMEM column c+(r/32), lane (r%32) of every quarter, byte j.
//
// One launch repacks both operands.  A CTA takes 128 rows x 64 K-blocks of
// one operand: one 16-byte read per thread (all issued before any is used, so
// the CTA pays DRAM latency once), then coalesced 4-byte writes of the 16
// chunks they form.
struct RepackArgs {
  const uint8_t *S;   // scales, rows x kb_count
  uint32_t *out;      // chunks
  int64_t rows;
  int kb_count;
  int k_steps;
  int atoms;          // 128-row blocks per tile of this operand
  int row_blocks;     // 128-row blocks to produce (tiles * atoms)
  int kgroups;        // ceil(k_steps / 16)
};

constexpr int kRepackThreads = 512;

__global__ void __launch_bounds__(kRepackThreads)
    repack_scales_kernel(RepackArgs a0, RepackArgs a1, int blocks0) {
  __shared__ __align__(16) uint32_t tile[128 * 16];  // 128 rows x 64 bytes
  const bool second = static_cast<int>(blockIdx.x) >= blocks0;
  const RepackArgs a = second ? a1 : a0;
  const int b = second ? static_cast<int>(blockIdx.x) - blocks0 : static_cast<int>(blockIdx.x);
  griddep_launch_dependents();
  const int rb = b / a.kgroups;          // 128-row block
  const int kg = b - rb * a.kgroups;     // group of 16 K steps
  const int64_t row0 = static_cast<int64_t>(rb) * 128;
  const int kb0 = kg * 64;
  uint8_t *t8 = reinterpret_cast<uint8_t *>(tile);
  // each thread brings in 16 consecutive bytes of one row (128 rows x 64 bytes)
  const int r = threadIdx.x >> 2, c0 = (threadIdx.x & 3) * 16;
  const int64_t row = row0 + r;
  const int kb = kb0 + c0;
  uint4 v = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  if (row < a.rows) {
    const uint8_t *src = a.S + row * a.kb_count + kb;
    if (kb + 16 <= a.kb_count && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      v = *reinterpret_cast<const uint4 *>(src);
    } else {
      uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t byte = kb + j < a.kb_count ? src[j] : 127u;
        w[j >> 2] |= byte << (8 * (j & 3));
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  *reinterpret_cast<uint4 *>(t8 + r * 64 + c0) = v;
  __syncthreads();
  const int tile_idx = rb / a.atoms, at = rb - tile_idx * a.atoms;
  const int nks = min(16, a.k_steps - kg * 16);
  for (int i = threadIdx.x; i < nks * 128; i += kRepackThreads) {
    const int ksl = i >> 7, w = i & 127;
    const int r = (w & 3) * 32 + (w >> 2);
    const int ks = kg * 16 + ksl;
    const int64_t g = (static_cast<int64_t>(tile_idx) * a.k_steps + ks) * a.atoms + at;
    a.out[g * 128 + w] = tile[r * 16 + ksl];
  }
}

// The same repack by a light kernel that fits beside a GEMM CTA on one SM
// (256 threads, at most 40 registers, no shared memory), so that the GEMM
// launched after it with programmatic dependent launch becomes resident at
// once and sends its first operand loads while this runs.  Units (a unit:
// 128 rows x 16 K steps of one operand, the block of repack_scales_kernel;
// units [0, units0) are A's) go two per round: thread t takes row t % 128 of
// unit 2 * (round index) + t / 128, reads the row's 16 K steps (16-byte
// loads, 127 for rows past the matrix) and writes each step's 4 bytes to
// word (r % 32) * 4 + r / 32 of that step's chunk.  Needs 16-byte aligned
// scale rows (K % 512 == 0, aligned bases).
constexpr int kRepackLiteThreads = 256;

__global__ void __launch_bounds__(kRepackLiteThreads, 6)
    repack_scales_lite_kernel(RepackArgs a0, RepackArgs a1, int units0, int units) {
  griddep_launch_dependents();
  const int t = threadIdx.x;
  const int r = t & 127;
  const int word = (r & 31) * 4 + (r >> 5);
  for (int u = 2 * static_cast<int>(blockIdx.x) + (t >> 7); u < units; u += 2 * static_cast<int>(gridDim.x)) {
    const bool second = u >= units0;
    const RepackArgs &a = second ? a1 : a0;
    const int b = second ? u - units0 : u;
    const int rb = b / a.kgroups, kg = b - rb * a.kgroups;
    const int64_t row = static_cast<int64_t>(rb) * 128 + r;
    const int n = min(16, a.k_steps - kg * 16);
    const uint4 *src = reinterpret_cast<const uint4 *>(a.S + row * a.kb_count + kg * 64);
    uint4 seg[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      seg[q] = (4 * q < n && row < a.rows) ? __ldg(src + q)
                                           : make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    const int tile_idx = rb / a.atoms, at = rb - tile_idx * a.atoms;
    uint32_t *out = a.out + ((static_cast<int64_t>(tile_idx) * a.k_steps + kg * 16) * a.atoms + at) * 128 + word;
    const int64_t stride = static_cast<int64_t>(a.atoms) * 128;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if (k < n) {
        const uint4 &x = seg[k >> 2];
        out[k * stride] = (k & 3) == 0 ? x.x : (k & 3) == 1 ? x.y : (k & 3) == 2 ? x.z : x.w;
      }
    }
  }
}

// Re-pitch the rows of an operand into the workspace: `rows` rows of `N`
// one-byte elements become rows of `Npad` bytes (a multiple of 16, for the
// 16-byte stride rule of tensor-map loads; the pad columns are zero).  With
// nbits = 6 or 4 the elements are sub-byte codes (low bits of each byte) and
// every group of 16 consecutive elements is packed, element i at bits
// [nbits*i, nbits*i + nbits) little-endian, into the first 2*nbits bytes of
// its 16-byte group, the rest zero: the shared-memory form that the scaled
// MMA reads for 6- and 4-bit operands (one 16-byte group per 16 elements,
// as for 8-bit ones).  Each thread writes 16 bytes; it reads them with the
// widest loads the source row's alignment allows (8, 4 or 1 byte).
__global__ void pad_rows_kernel(const uint8_t *__restrict__ B, int64_t rows, int64_t N,
                                int64_t Npad, uint8_t *__restrict__ out, int nbits) {
  const int64_t per_row = Npad / 16;
  const int64_t total = rows * per_row;
  griddep_launch_dependents();
  const int align = (N % 8 == 0 && (reinterpret_cast<uintptr_t>(B) & 7) == 0) ? 8
                    : (N % 4 == 0 && (reinterpret_cast<uintptr_t>(B) & 3) == 0) ? 4 : 1;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row;
    const int64_t c0 = (i - r * per_row) * 16;
    const uint8_t *src = B + r * N + c0;
    uint32_t w[4] = {0, 0, 0, 0};
    if (c0 + 16 <= N && align == 8) {
      const uint2 a = reinterpret_cast<const uint2 *>(src)[0];
      const uint2 b = reinterpret_cast<const uint2 *>(src)[1];
      w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y;
    } else if (c0 + 16 <= N && align == 4) {
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = reinterpret_cast<const uint32_t *>(src)[j];
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t b = c0 + j < N ? src[j] : 0u;
        w[j >> 2] |= b << (8 * (j & 3));
      }
    }
    if (nbits < 8) {
      const uint64_t mask = (1ull << nbits) - 1;
      uint64_t lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint64_t v = (w[j >> 2] >> (8 * (j & 3))) & mask;
        const int pos = j * nbits;
        if (pos < 64) {
          lo |= v << pos;
          if (pos + nbits > 64) hi |= v >> (64 - pos);
        } else {
          hi |= v << (pos - 64);
        }
      }
      w[0] = static_cast<uint32_t>(lo);
      w[1] = static_cast<uint32_t>(lo >> 32);
      w[2] = static_cast<uint32_t>(hi);
      w[3] = static_cast<uint32_t>(hi >> 32);
    }
    *reinterpret_cast<uint4 *>(out + r * Npad + c0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace mxg
