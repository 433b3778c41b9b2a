// mxgemm_kernel.cuh -- the block-scaled (MXFP8) GEMM kernel for sm_103a.
//
//   C[M,N] (+)= (A * 2^(sA-127)) x (B * 2^(sB-127))
//
// Design (one CTA per SM, persistent, warp-specialised):
//   warp 0      TMA producer: per 128-deep K step loads the A tile (K-major,
//               128-byte swizzle), the B tile (N-major, 128-byte swizzle) and
//               the A/B scale chunks into a STAGES-deep shared-memory ring;
//               each stage has a "full" barrier (arrive + expected bytes) and
//               an "empty" barrier (released by the MMA's commit).
//   warp 1      allocates TMEM; one thread issues, per K step, tcgen05.cp of
//               the scale chunks SMEM -> TMEM, then four
//               tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each) into an
//               FP32 TMEM accumulator, then tcgen05.commit -> empty[stage];
//               after a tile's last step, tcgen05.commit -> acc_full.
//   warps 2..9  epilogue: wait acc_full, tcgen05.ld the whole accumulator into
//               registers, release it (acc_empty) so the next tile's MMAs
//               start, then (optionally + C_in) round to FP32/BF16 and store.
//
// Pair mode (CG = 2, cluster of 2 CTAs, tcgen05 cta_group::2): the pair
// computes a 256 x 256 tile; each CTA loads its own 128 rows of A and its own
// 128-column half of B, and BOTH CTAs load the full 256-column B scale
// chunk; only the leader CTA (rank 0) sets the expected byte count, the
// peer's loads signal the leader's barrier; the leader issues every MMA and
// commit (commits multicast to both CTAs' barriers); epilogue warps of both
// CTAs release the accumulator by arriving on the leader's barrier ("arrive
// remote, wait local").  This is the 2-CTA scaled MMA of "Tensor core
// operations" (section "2-CTA Scaled MMA": B split across CTAs, B scale full)
// with the barrier rules of "TLX API Quick Reference" (sections "2-CTA MMA
// semantics", "2-CTA barrier patterns").  No TMA multicast is used.
//
// Every barrier wait is bounded: when a wait exceeds the time limit the
// thread records MXGEMM_ERR_TIMEOUT in the status word, raises a CTA-wide
// abort flag, and every role drains and returns; TMEM is always freed.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace mxg {

constexpr int kStatusTimeout = 6;  // MXGEMM_ERR_TIMEOUT

template <int CG>
struct Cfg {
  static constexpr int BM = 128;          // accumulator rows per CTA
  static constexpr int BN = 256;          // MMA N: columns of a (pair) tile
  static constexpr int BK = 128;          // K elements (bytes) per stage
  static constexpr int BN_CTA = BN / CG;  // B columns loaded by each CTA
  static constexpr int STAGES = CG == 1 ? 4 : 6;
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BK * BN_CTA;
  static constexpr int SFA_BYTES = 512;   // 128 rows x 4 K-blocks
  static constexpr int SFB_BYTES = 1024;  // 256 columns x 4 K-blocks
  static constexpr uint32_t STAGE_TX = (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES) * CG;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 3;  // full[], empty[], acc_full, acc_empty, final
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1 KB alignment
  static constexpr int TM_ACC = 0;
  static constexpr int TM_SFA = BN;               // STAGES x 4 columns
  static constexpr int TM_SFB = BN + 4 * STAGES;  // STAGES x 8 columns
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = 32 * (2 + EPI_WARPS);
  static_assert(TM_SFB + 8 * STAGES <= (int)TM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(OFF_B % 1024 == 0 && A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "align");
};

struct KParams {
  int M, N, K;
  int m_tiles;    // tiles along M (each 128*CG rows)
  int n_tiles;    // tiles along N (each 256 columns)
  int k_steps;    // ceil(K / 128)
  int num_tiles;  // m_tiles * n_tiles
  void *C;
  int out_bf16;
  int use_acc;
  int vec_ok;     // rows of C allow 16-byte vector access
  int *status;    // [0] code, [1] detail
  unsigned long long timeout_ns;
  int stall_producer;
  int use_clc;
};

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4.block_scale:
// E4M3 x E4M3, A K-major, B N-major, UE8M0 scales, M x N, scale byte ids.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int sfa_id, int sfb_id) {
  return (uint32_t(sfb_id & 3) << 4)     // B scale-factor byte id
         | (0u << 7)                     // A format E4M3
         | (0u << 10)                    // B format E4M3
         | (0u << 15)                    // A K-major
         | (1u << 16)                    // B N-major
         | (uint32_t(N >> 3) << 17)      // N / 8
         | (1u << 23)                    // scale format UE8M0
         | (uint32_t(M >> 4) << 24)      // M / 16
         | (uint32_t(sfa_id & 3) << 29); // A scale-factor byte id
}

// Tile t -> (m tile, n tile): groups of 8 M-tiles walked N-fastest, so the
// CTAs running at one time share a few A and B strips in L2.
__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int &mt, int &nt) {
  constexpr int G = 8;
  const int per_group = G * n_tiles;
  const int g = t / per_group;
  const int first = g * G;
  const int gm = min(m_tiles - first, G);
  const int r = t - g * per_group;
  mt = first + r % gm;
  nt = r / gm;
}

struct WaitCtl {
  int *status;
  volatile int *abort_flag;
  unsigned long long timeout_ns;
};

// Bounded wait for the phase of `bar` with parity `parity`.  Returns false
// (after recording a timeout, or on a raised abort flag) instead of hanging.
template <bool CLUSTER>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtl &w,
                                        int detail) {
  if (CLUSTER ? mbar_try_wait_cluster_acquire(bar, parity) : mbar_try_wait(bar, parity))
    return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (CLUSTER ? mbar_try_wait_cluster_acquire(bar, parity) : mbar_try_wait(bar, parity))
      return true;
    if ((it & 31u) == 0) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        if (atomicCAS(w.status, 0, kStatusTimeout) == 0) atomicExch(w.status + 1, detail);
        *w.abort_flag = 1;
        return false;
      }
    }
  }
}

template <int CG>
__global__ void __launch_bounds__(Cfg<CG>::THREADS, 1)
    mxgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmSFA,
                  const __grid_constant__ CUtensorMap tmSFB, const KParams p) {
  using C = Cfg<CG>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;

  const uint32_t bar_full = base + C::OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * C::STAGES;
  const uint32_t bar_acc_full = bar_empty + 8 * C::STAGES;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  const uint32_t bar_final = bar_acc_empty + 8;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, C::EPI_WARPS * CG);
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSFA);
    tma_prefetch_desc(&tmSFB);
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  if constexpr (CG == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const WaitCtl wc{p.status, abort_flag, p.timeout_ns};
  constexpr bool CL = (CG == 2);
  const int first_tile = blockIdx.x / CG;
  const int tile_stride = gridDim.x / CG;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      if (!p.stall_producer) {
        for (int t = first_tile; ok && t < p.num_tiles; t += tile_stride) {
          int mt, nt;
          tile_coords(t, p.m_tiles, p.n_tiles, mt, nt);
          const int row0 = mt * (128 * CG) + 128 * (int)rank;  // this CTA's A rows
          const int mblk = mt * CG + (int)rank;                  // its 128-row block
          const int col0 = nt * 256;
          for (int ks = 0; ks < p.k_steps; ++ks) {
            if (!wait_phase<CL>(bar_empty + 8 * stage, phase ^ 1u, wc, 0x01 | (stage << 8))) {
              ok = false;
              break;
            }
            const uint32_t fb = bar_full + 8 * stage;
            const uint32_t sA = base + C::OFF_A + stage * C::A_BYTES;
            const uint32_t sB = base + C::OFF_B + stage * C::B_BYTES;
            const uint32_t sSA = base + C::OFF_SFA + stage * C::SFA_BYTES;
            const uint32_t sSB = base + C::OFF_SFB + stage * C::SFB_BYTES;
            const int k0 = ks * 128;
            if constexpr (CG == 1) {
              mbar_arrive_expect_tx(fb, C::STAGE_TX);
              tma_load_2d(sA, &tmA, k0, row0, fb);
              tma_load_2d(sB, &tmB, col0, k0, fb);
              tma_load_2d(sB + 16384, &tmB, col0 + 128, k0, fb);
              tma_load_2d(sSA, &tmSFA, 0, (mblk * p.k_steps + ks) * 32, fb);
              tma_load_2d(sSB, &tmSFB, 0, (nt * p.k_steps + ks) * 64, fb);
            } else {
              if (rank == 0) mbar_arrive_expect_tx(fb, C::STAGE_TX);
              const uint32_t fbl = mapa_shared(fb, 0);  // leader's barrier
              tma_load_2d_pair(sA, &tmA, k0, row0, fbl);
              tma_load_2d_pair(sB, &tmB, col0 + 128 * (int)rank, k0, fbl);
              tma_load_2d_pair(sSA, &tmSFA, 0, (mblk * p.k_steps + ks) * 32, fbl);
              tma_load_2d_pair(sSB, &tmSFB, 0, (nt * p.k_steps + ks) * 64, fbl);
            }
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Drain: every stage's last fill has been consumed (its MMA commit has
      // arrived) before this CTA may finish.
      for (int i = 0; i < C::STAGES; ++i) {
        if (!wait_phase<CL>(bar_empty + 8 * stage, phase ^ 1u, wc, 0x11 | (stage << 8))) break;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = first_tile; ok && t < p.num_tiles; t += tile_stride) {
        if (!wait_phase<CL>(bar_acc_empty, acc_phase ^ 1u, wc, 0x02 | ((t & 0xFFFF) << 16))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < p.k_steps; ++ks) {
          if (!wait_phase<CL>(bar_full + 8 * stage, phase, wc, 0x03 | (stage << 8))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = base + C::OFF_A + stage * C::A_BYTES;
          const uint32_t sB = base + C::OFF_B + stage * C::B_BYTES;
          const uint32_t sSA = base + C::OFF_SFA + stage * C::SFA_BYTES;
          const uint32_t sSB = base + C::OFF_SFB + stage * C::SFB_BYTES;
          const uint32_t tSA = tmem + C::TM_SFA + 4 * stage;
          const uint32_t tSB = tmem + C::TM_SFB + 8 * stage;
          // scale chunks: 32 rows x 16 bytes each, no swizzle, 8-row groups 128 B apart
          tmem_cp_32x128b_x4<CG>(tSA, smem_desc(sSA, 0, 128, 0));
          tmem_cp_32x128b_x4<CG>(tSB, smem_desc(sSB, 0, 128, 0));
          tmem_cp_32x128b_x4<CG>(tSB + 4, smem_desc(sSB + 512, 0, 128, 0));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // A: K-major, 128-byte swizzle, 8-row groups 1024 B apart; step 32 B per K=32
            const uint64_t ad = smem_desc(sA + 32 * k, 0, 1024, 2);
            // B: N-major, 128-byte swizzle; 128-column chunks 16 KB apart,
            // 8-row K groups 1024 B apart; step 32 rows (4 KB) per K=32
            const uint64_t bd = smem_desc(sB + 4096 * k, 16384, 1024, 2);
            mma_mxf8<CG>(tmem + C::TM_ACC, ad, bd, idesc_mxf8(128 * CG, 256, k, k), tSA, tSB,
                         (ks | k) != 0);
          }
          if constexpr (CG == 1) tc_commit(bar_empty + 8 * stage);
          else tc_commit_pair(bar_empty + 8 * stage, 0x3);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (CG == 1) tc_commit(bar_acc_full);
        else tc_commit_pair(bar_acc_full, 0x3);
        acc_phase ^= 1u;
      }
      // all issued tcgen05 work has finished before TMEM can be released
      if constexpr (CG == 1) tc_commit(bar_final);
      else tc_commit_pair(bar_final, 0x1);
      WaitCtl wf = wc;
      wf.abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 8);  // never raised
      *wf.abort_flag = 0;
      wait_phase<false>(bar_final, 0, wf, 0x04);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;  // 0..7
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    const int h = ew >> 2;    // which 128-column half
    uint32_t acc_phase = 0;
    for (int t = first_tile; t < p.num_tiles; t += tile_stride) {
      int mt, nt;
      tile_coords(t, p.m_tiles, p.n_tiles, mt, nt);
      int ok = 1;
      if (lane == 0) ok = wait_phase<CL>(bar_acc_full, acc_phase, wc, 0x05 | ((t & 0xFFFF) << 16));
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[4][32];
      const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + C::TM_ACC + 128 * h;
      tmem_ld_32x32b_x32(ta + 0, v[0]);
      tmem_ld_32x32b_x32(ta + 32, v[1]);
      tmem_ld_32x32b_x32(ta + 64, v[2]);
      tmem_ld_32x32b_x32(ta + 96, v[3]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 1) mbar_arrive(bar_acc_empty);
        else mbar_arrive_cluster(bar_acc_empty, 0);
      }
      acc_phase ^= 1u;

      const int row = mt * (128 * CG) + 128 * (int)rank + 32 * q + lane;
      const int colb = nt * 256 + 128 * h;
      if (row < p.M) {
        if (!p.out_bf16) {
          float *cp = reinterpret_cast<float *>(p.C) + static_cast<int64_t>(row) * p.N + colb;
          if (p.vec_ok && colb + 128 <= p.N) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              float4 o = make_float4(__uint_as_float(v[c >> 3][(c & 7) * 4 + 0]),
                                     __uint_as_float(v[c >> 3][(c & 7) * 4 + 1]),
                                     __uint_as_float(v[c >> 3][(c & 7) * 4 + 2]),
                                     __uint_as_float(v[c >> 3][(c & 7) * 4 + 3]));
              float4 *dst = reinterpret_cast<float4 *>(cp + 4 * c);
              if (p.use_acc) {
                const float4 old = *dst;
                o.x += old.x;
                o.y += old.y;
                o.z += old.z;
                o.w += old.w;
              }
              *dst = o;
            }
          } else {
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              if (colb + c < p.N) {
                float o = __uint_as_float(v[c >> 5][c & 31]);
                if (p.use_acc) o += cp[c];
                cp[c] = o;
              }
            }
          }
        } else {
          __nv_bfloat16 *cp =
              reinterpret_cast<__nv_bfloat16 *>(p.C) + static_cast<int64_t>(row) * p.N + colb;
          if (p.vec_ok && colb + 128 <= p.N) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              uint4 *dst = reinterpret_cast<uint4 *>(cp + 8 * c);
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[(8 * c + e) >> 5][(8 * c + e) & 31]);
              if (p.use_acc) {
                const uint4 old = *dst;
                const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  f[2 * e] += __uint_as_float(ow[e] << 16);
                  f[2 * e + 1] += __uint_as_float(ow[e] & 0xFFFF0000u);
                }
              }
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
                w[e] = *reinterpret_cast<const uint32_t *>(&b2);
              }
              *dst = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              if (colb + c < p.N) {
                float o = __uint_as_float(v[c >> 5][c & 31]);
                if (p.use_acc) o += __bfloat162float(cp[c]);
                cp[c] = __float2bfloat16_rn(o);
              }
            }
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  if constexpr (CG == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<CG>(tmem, C::TM_COLS);
}

// ---------------------------------------------------------------- prepasses

// Scale repack: row-major scales S[rows][kb_count] -> 512-byte chunks.  Chunk
// g = (tile * k_steps + ks) * atoms + a covers rows (tile*atoms + a)*128 + r,
// r in [0,128), and K-blocks ks*4 + j, j in [0,4); its byte
// (r % 32) * 16 + (r / 32) * 4 + j holds that scale (127 = 1.0 where the row
// or K-block is out of range).  This is the 32-row x 16-byte source shape of
// tcgen05.cp .32x128b.warpx4, which replicates it into the four TMEM lane
// quarters: TMEM column c+(r/32), lane (r%32) of every quarter, byte j.
__global__ void repack_scales_kernel(const uint8_t *__restrict__ S, int64_t rows, int kb_count,
                                     int k_steps, int atoms, int64_t total_words,
                                     uint32_t *__restrict__ out) {
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < total_words;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t g = w >> 7;
    const int t = static_cast<int>(w & 127);
    const int a = static_cast<int>(g % atoms);
    const int64_t rest = g / atoms;
    const int ks = static_cast<int>(rest % k_steps);
    const int64_t tile = rest / k_steps;
    const int r = (t & 3) * 32 + (t >> 2);
    const int64_t row = (tile * atoms + a) * 128 + r;
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = ks * 4 + j;
      const uint32_t byte = (row < rows && kb < kb_count) ? S[row * kb_count + kb] : 127u;
      word |= byte << (8 * j);
    }
    out[w] = word;
  }
}

// Copy B [K][N] into [K][Npad] (Npad a multiple of 16) so that its rows meet
// the 16-byte stride rule of tensor-map loads; the pad columns are zero.
__global__ void pad_rows_kernel(const uint8_t *__restrict__ B, int64_t rows, int64_t N,
                                int64_t Npad, uint8_t *__restrict__ out) {
  const int64_t per_row = Npad / 16;
  const int64_t total = rows * per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row;
    const int64_t c0 = (i - r * per_row) * 16;
    const uint8_t *src = B + r * N;
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int64_t c = c0 + j;
      const uint32_t b = c < N ? src[c] : 0u;
      w[j >> 2] |= b << (8 * (j & 3));
    }
    *reinterpret_cast<uint4 *>(out + r * Npad + c0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace mxg
