// swapab_kernel.cuh -- the block-scaled GEMM for skinny problems (M <= 128)
// on sm_103a, computed transposed ("swap-AB"):
//
//   C^T[N, M] = B^T[N, K] x A^T[K, M]     (both with their E8M0 block scales)
//
// so that the long dimension N feeds the M side of the tensor cores' MMA
// (which is 128 rows for the single-CTA block-scaled form) and the few rows
// of A become the MMA's N (M rounded up to 16, at least 16).  This is the
// same scaled product as mxgemm_kernel ("TLX API Quick Reference", section
// "Matrix Multiply (MMA)", async_dot_scaled; "Tensor core operations",
// section "TMEM-backed MX Scales"), with the operand roles exchanged:
//
//   MMA A operand : 128 columns of B, K-deep.  B is K x N with N contiguous,
//                   so the operand is M-major (transpose-A bit); in shared
//                   memory it is the 128 K rows x 128 bytes that one TMA box
//                   with 128-byte swizzle gives (8-row K groups 1 KB apart).
//   MMA B operand : the M rows of A (K contiguous, so K-major), Nm rows x
//                   128 bytes per K step, 128-byte swizzle; rows past M read
//                   as zero (TMA fills them).
//   scale of A op : B_scale rows n0 .. n0+127 (B_scale holds column j's
//                   scales in row j), one 512-byte chunk per K step.
//   scale of B op : A_scale rows 0 .. Nm-1, one 512-byte chunk per K step.
//   accumulator   : TMEM lane n (column n0+n of C) x Nm FP32 columns (row m
//                   of C), so an epilogue warp's store of one row m of C is
//                   32 consecutive columns: a whole 128-byte line for FP32.
//
// Grid: one CTA per (128-column block of N, K split).  When the column
// blocks alone leave SMs idle, each block's K steps are split over a
// cluster of `splits` CTAs (at most 8); after their main loops the other
// CTAs of the cluster write their FP32 partial accumulators into the first
// CTA's shared memory (distributed shared memory), and the first CTA adds
// them in rank order (a fixed order: the result does not depend on timing)
// and stores C.  No workspace, no flags, no second launch.
//
// Warp roles (224 threads):
//   warp 0     TMA producer: per 128-deep K step the B^T tile (16 KB) and
//              the A^T tile (Nm x 128 B) into a STAGES-deep ring; full
//              barriers take its arrive plus the bytes, empty barriers are
//              released by the MMA's tcgen05.commit.  With packed scales it
//              also copies the step's two scale chunks (bulk copies).
//   warp 1     allocates TMEM; one thread issues per K step 2 x tcgen05.cp
//              (scale chunks SMEM -> TMEM) and 4 x tcgen05.mma
//              .kind::mxf8f6f4.block_scale (K = 32 each), then commits to
//              the stage's empty barrier; after the last step, to acc_full.
//   warp 2     scale builder (row-major scales): builds each stage's two
//              chunks in the byte order that tcgen05.cp .32x128b.warpx4
//              takes, from 16-byte row segments (four K steps of one row)
//              staged by TMA into a ring of SD slots, SD groups of four K
//              steps ahead (K % 512 == 0 and 16-byte aligned scale
//              pointers), or read with byte loads; then arrives on the
//              stage's full barrier (which then expects two arrives).
//   warps 3-6  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//              lanes 32 (w % 4) .. +31), the cluster reduction, optional
//              + C_in, round to FP32 / BF16, coalesced stores.
//
// Every mbarrier wait is bounded by %globaltimer: a wait that runs out
// records MXGEMM_ERR_TIMEOUT in the status word and the roles drain and
// return; C is then incomplete.  TMEM is always freed; nothing traps.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace mxg {

struct SwapParams {
  int M, N, K;
  int nm;        // MMA N: M rounded up to 16
  int k_steps;   // ceil(K / 128)
  int splits;    // CTAs (one cluster) sharing a column block's K steps
  void *C;
  int use_acc;
  int *status;   // [0] code, [1] detail
  unsigned long long timeout_ns;
  int stall_producer;
  uint32_t idesc_fmt;  // MMA A format = B's element format, MMA B format = A's
  // row-major scales (A_scale M x kb_count, B_scale N x kb_count)
  const uint8_t *a_scale;
  const uint8_t *b_scale;
  int kb_count;
  int scale_tma;  // the staging maps describe the scales (else byte loads)
  // packed scales (the 512-byte chunks of mxgemm_scale_layout_t): the
  // producer copies them with the stage and no scale builder runs
  int packed;
  const uint8_t *a_chunks;  // A_scale chunks, row block 0: ks * 512
  const uint8_t *b_chunks;  // B_scale chunks: ((c / 2 * S + ks) * 2 + c % 2) * 512
  // B given N x K (K contiguous): the MMA's A operand is then K-major (a box
  // of 128 K bytes x 128 rows of B, no transpose bit)
  int b_kmajor;
};

template <int NT>
struct SwapCfg {
  static constexpr int BK = 128;
  static constexpr int BT_BYTES = 128 * BK;  // the MMA's A operand: 128 columns of B
  static constexpr int AT_BYTES = NT * BK;   // the MMA's B operand: up to NT rows of A
  static constexpr int SF_BYTES = 512;
  static constexpr int STAGES = NT <= 16 ? 10 : NT <= 32 ? 9 : NT <= 64 ? 8 : 6;
  static constexpr int OFF_BT = 0;
  static constexpr int OFF_AT = OFF_BT + STAGES * BT_BYTES;
  static constexpr int OFF_SF = OFF_AT + STAGES * AT_BYTES;  // per stage: A op chunk, B op chunk
  static constexpr int OFF_STG = (OFF_SF + STAGES * 2 * SF_BYTES + 1023) / 1024 * 1024;
  static constexpr int STG_BT = 128 * 16;  // B_scale segments of the block's 128 columns
  static constexpr int STG_SLOT = STG_BT + 128 * 16;  // + A_scale segments (<= 128 rows)
  // staging ring of the scale builder: one slot per group of four K steps,
  // loaded SD groups ahead of the group being read
  static constexpr int SD = 4;
  static constexpr int OFF_BAR = OFF_STG + SD * STG_SLOT;
  // full[], empty[], acc_full, final, stg[]
  static constexpr int NUM_BARS = 2 * STAGES + 2 + SD;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1 KB alignment
  // the cluster reduction reuses the operand ring: per other CTA, NT x 128
  // FP32 values
  static constexpr int RECV_BYTES = OFF_SF;
  static constexpr int TM_ACC = 0;
  static constexpr int TM_SF = 128;  // per stage 8 columns: A op scales, then B op scales
  static constexpr uint32_t TM_COLS = 256;
  static constexpr int THREADS = 7 * 32;
  static_assert(TM_SF + 8 * STAGES <= (int)TM_COLS, "TMEM budget");
  static_assert(NT <= TM_SF, "accumulator columns");
  static_assert(STAGES <= 32 && SD <= 32, "one lane per early load");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(AT_BYTES % 1024 == 0 && OFF_AT % 1024 == 0, "operand alignment");
};

// Largest number of CTAs of one cluster whose partials fit the first CTA's
// receive area.
template <int NT>
__host__ __device__ constexpr int swap_max_splits() {
  return SwapCfg<NT>::RECV_BYTES / (NT * 128 * 4) + 1 < 8 ? SwapCfg<NT>::RECV_BYTES / (NT * 128 * 4) + 1
                                                            : 8;
}

// Instruction descriptor: MMA A = B^T (M-major: transpose-A bit), MMA B =
// A^T (K-major), UE8M0 scales, M = 128, N = nm, scale byte ids.
__host__ __device__ constexpr uint32_t idesc_swap(int nm, int sf_id) {
  return (uint32_t(sf_id & 3) << 4)      // B scale-factor byte id
         | (1u << 15)                    // A is M-major
         | (0u << 16)                    // B is K-major
         | (uint32_t(nm >> 3) << 17)     // N / 8
         | (1u << 23)                    // scale format UE8M0
         | (uint32_t(128 >> 4) << 24)    // M / 16
         | (uint32_t(sf_id & 3) << 29);  // A scale-factor byte id
}

template <bool CLUSTER>
__device__ __forceinline__ bool swap_wait(uint32_t bar, uint32_t parity, int *status,
                                          volatile int *abort_flag, unsigned long long timeout_ns,
                                          int detail) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        if (atomicCAS(status, 0, 6) == 0) atomicExch(status + 1, detail);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

template <int NT, bool BF16, bool ACC>
__global__ void __launch_bounds__(SwapCfg<NT>::THREADS, 1)
    mxgemm_swapab_kernel(const __grid_constant__ CUtensorMap tmBt,
                         const __grid_constant__ CUtensorMap tmAt,
                         const __grid_constant__ CUtensorMap tmSB,
                         const __grid_constant__ CUtensorMap tmSA, const SwapParams p) {
  using S = SwapCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int splits = p.splits;
  const int split = splits > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int n0 = static_cast<int>(blockIdx.x) / splits * 128;
  const int kb = static_cast<int>(static_cast<long long>(split) * p.k_steps / splits);
  const int ke = static_cast<int>(static_cast<long long>(split + 1) * p.k_steps / splits);
  const bool packed = p.packed != 0;

  const uint32_t bar_full = base + S::OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * S::STAGES;
  const uint32_t bar_acc = bar_empty + 8 * S::STAGES;
  const uint32_t bar_final = bar_acc + 8;
  const uint32_t bar_stg = bar_final + 8;  // SD staging slots
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + S::OFF_MISC + 4);
  volatile int *never = reinterpret_cast<volatile int *>(sm + S::OFF_MISC + 8);  // never raised

  const int nm = p.nm;
  const uint32_t at_tx = static_cast<uint32_t>(nm) * 128u;
  const bool stg_tma = !packed && p.scale_tma != 0;
  const int g_first = kb >> 2, g_last = (ke - 1) >> 2;
  // The first ring round of operand loads, and the scale builder's first
  // staging loads (ahead of them), go out from the thread that initializes
  // the barriers, before the rest of the set-up (TMEM allocation, the CTA
  // barrier): the set-up then overlaps their DRAM latency.
  const int n_early = p.stall_producer ? 0 : min(S::STAGES, ke - kb);
  const int n_stg_early = stg_tma ? min(S::SD, g_last - g_first + 1) : 0;
  // one operand step: the B^T tile, the A^T tile and, with packed scales,
  // the two scale chunks, all counted on the stage's full barrier
  auto load_step = [&](int st, int ks) {
    const uint32_t fb = bar_full + 8 * st;
    mbar_arrive_expect_tx(fb, S::BT_BYTES + at_tx + (packed ? 2 * S::SF_BYTES : 0));
    if (p.b_kmajor) tma_load_2d(base + S::OFF_BT + st * S::BT_BYTES, &tmBt, ks * 128, n0, fb);
    else tma_load_2d(base + S::OFF_BT + st * S::BT_BYTES, &tmBt, n0, ks * 128, fb);
    tma_load_2d(base + S::OFF_AT + st * S::AT_BYTES, &tmAt, ks * 128, 0, fb);
    if (packed) {
      const int c = n0 / 128;
      const uint32_t sf = base + S::OFF_SF + st * 2 * S::SF_BYTES;
      bulk_load(sf, p.b_chunks + (static_cast<int64_t>((c >> 1) * p.k_steps + ks) * 2 + (c & 1)) * 512,
                512, fb);
      bulk_load(sf + S::SF_BYTES, p.a_chunks + static_cast<int64_t>(ks) * 512, 512, fb);
    }
  };
  // staging load of the scale rows' segments of group g (K steps 4g .. 4g+3)
  // into slot g % SD
  auto load_stg = [&](int g) {
    const int slot = g % S::SD;
    const uint32_t sb = base + S::OFF_STG + slot * S::STG_SLOT, bar = bar_stg + 8 * slot;
    mbar_arrive_expect_tx(bar, S::STG_BT + at_tx / 8);
    tma_load_2d(sb, &tmSB, 16 * g, n0, bar);
    tma_load_2d(sb + S::STG_BT, &tmSA, 16 * g, 0, bar);
  };

  if (warp == 0) {
    if (lane == 0) {
      // the tensor-map descriptors, fetched while the barriers are set up
      tma_prefetch_desc(&tmBt);
      tma_prefetch_desc(&tmAt);
      if (stg_tma) {
        tma_prefetch_desc(&tmSB);
        tma_prefetch_desc(&tmSA);
      }
      for (int s = 0; s < S::STAGES; ++s) {
        // full: the producer's arrive with the bytes, plus the scale
        // builder's arrive once the stage's chunks are written
        mbar_init(bar_full + 8 * s, packed ? 1 : 2);
        mbar_init(bar_empty + 8 * s, 1);
      }
      mbar_init(bar_acc, 1);
      for (int i = 0; i < S::SD; ++i) mbar_init(bar_stg + 8 * i, 1);
      mbar_init(bar_final, 1);
      *abort_flag = 0;
      *never = 0;
      fence_mbar_init();
      fence_proxy_async_smem();  // the initialized barriers, before TMA completes on them
    }
    __syncwarp();
    // a prepass before this kernel (B re-pitched for N % 16 != 0) may still
    // be finishing: no global access before it has
    griddep_wait();
    // one lane per load: the staging loads first, then the operand stages
    if (lane < n_stg_early) load_stg(g_first + lane);
    __syncwarp();
    if (lane < n_early) load_step(lane, kb + lane);
  }
  if (warp == 1) {
    tmem_alloc<1>(smem_u32(tmem_slot), S::TM_COLS);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // (returns at once: thread 0 waited before the barrier)

  uint32_t v[NT];  // epilogue warps: this lane's accumulator row (column n0 + lane of C)
  bool have_acc = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const bool leader = elect_one() != 0;
    // the first ring round went out during the set-up
    int st = n_early == S::STAGES ? 0 : n_early;
    uint32_t ph = n_early == S::STAGES ? 1u : 0u;
    for (int ks = kb + n_early; ks < ke && !p.stall_producer; ++ks) {
      if (!__all_sync(0xFFFFFFFFu, swap_wait<false>(bar_empty + 8 * st, ph ^ 1u, p.status,
                                                    abort_flag, p.timeout_ns, 0x01 | (st << 8))))
        break;
      if (leader) load_step(st, ks);
      __syncwarp();
      if (++st == S::STAGES) {
        st = 0;
        ph ^= 1u;
      }
    }
    // drain: every fill of this launch has been consumed before the CTA
    // may finish (a stage never filled passes at once)
    for (int i = 0; i < S::STAGES; ++i) {
      if (!__all_sync(0xFFFFFFFFu, swap_wait<false>(bar_empty + 8 * st, ph ^ 1u, p.status, abort_flag,
                                                    p.timeout_ns, 0x11 | (st << 8))))
        break;
      if (++st == S::STAGES) {
        st = 0;
        ph ^= 1u;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one() != 0;
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int ks = kb; ks < ke; ++ks) {
      if (!__all_sync(0xFFFFFFFFu, swap_wait<false>(bar_full + 8 * st, ph, p.status, abort_flag,
                                                    p.timeout_ns, 0x03 | (st << 8)))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (leader) {
        const uint32_t sBt = base + S::OFF_BT + st * S::BT_BYTES;
        const uint32_t sAt = base + S::OFF_AT + st * S::AT_BYTES;
        const uint32_t sSF = base + S::OFF_SF + st * 2 * S::SF_BYTES;
        const uint32_t tSA = tmem + S::TM_SF + 8 * st;
        const uint32_t tSB = tSA + 4;
        // scale chunks: 32 rows x 16 bytes, no swizzle, 8-row groups 128 B apart
        tmem_cp_32x128b_x4<1>(tSA, smem_desc(sSF, 0, 128, 0));
        tmem_cp_32x128b_x4<1>(tSB, smem_desc(sSF + S::SF_BYTES, 0, 128, 0));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          // A op: M-major, 128-byte swizzle, one 128-byte-wide column chunk,
          // 8-row K groups 1 KB apart, 32 K rows (4 KB) per K = 32.
          // B op: K-major, 128-byte swizzle, 8-row groups 1 KB apart, 32 B per K = 32.
          mma_mxf8<1>(tmem + S::TM_ACC,
                      p.b_kmajor ? smem_desc(sBt + 32 * k, 0, 1024, 2)
                                 : smem_desc(sBt + 4096 * k, 16384, 1024, 2),
                      smem_desc(sAt + 32 * k, 0, 1024, 2),
                      (idesc_swap(nm, k) | p.idesc_fmt) & (p.b_kmajor ? ~(1u << 15) : ~0u), tSA, tSB,
                      (ks != kb || k != 0) ? 1u : 0u);
        tc_commit(bar_empty + 8 * st);
      }
      __syncwarp();
      if (++st == S::STAGES) {
        st = 0;
        ph ^= 1u;
      }
    }
    if (ok && leader) tc_commit(bar_acc);
    __syncwarp();
    // every issued tcgen05 operation has finished before TMEM is freed and
    // before the ring may be reused for the cluster reduction
    if (leader) tc_commit(bar_final);
    __syncwarp();
    swap_wait<false>(bar_final, 0, p.status, never, p.timeout_ns, 0x04);
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ scale builder
    // Chunk row `lane` of a K step holds, in its 4-byte word q, the step's
    // four K-block scales of row lane + 32 q (tcgen05.cp .32x128b.warpx4
    // replicates the 32 x 16-byte chunk into the four TMEM lane quarters);
    // those four bytes are bytes 4t .. 4t+3 of the row's 16-byte segment for
    // the group of four K steps 4g .. 4g+3 (t = step - 4g).
    if (!packed) {
      const bool tma = stg_tma;
      const uint32_t stg = base + S::OFF_STG;
      uint32_t sph = 0;  // per staging slot: parity of its next completion
      // per staging slot: a load issued and not yet read (the first ones went
      // out during the set-up)
      uint32_t pending = 0;
      for (int g = g_first; g < g_first + n_stg_early; ++g) pending |= 1u << (g % S::SD);
      const int kbn = p.kb_count;
      uint4 ca[4], cb[4];  // segments of the current group: B_scale rows, A_scale rows
      auto stage = [&](int g) {
        if (lane == 0) load_stg(g);
        __syncwarp();
        pending |= 1u << (g % S::SD);
      };
      // 16 scale bytes (K-blocks 16 g .. 16 g + 15) of row `row` of Sc,
      // byte by byte; 127 (1.0) past the end of the row or the matrix
      auto load16 = [&](const uint8_t *Sc, int64_t row, int64_t rows, int g) -> uint4 {
        uint32_t x[4] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu};
        if (row < rows) {
          const uint8_t *src = Sc + row * kbn + 16 * g;
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const uint32_t val = 16 * g + b < kbn ? static_cast<uint32_t>(src[b]) : 127u;
            x[b >> 2] = (x[b >> 2] & ~(0xFFu << (8 * (b & 3)))) | (val << (8 * (b & 3)));
          }
        }
        return make_uint4(x[0], x[1], x[2], x[3]);
      };
      auto take = [&](int g) -> bool {
        if (tma) {
          const int slot = g % S::SD;
          const uint32_t sb = stg + slot * S::STG_SLOT;
          if (!__all_sync(0xFFFFFFFFu, swap_wait<false>(bar_stg + 8 * slot, (sph >> slot) & 1u, p.status,
                                                        abort_flag, p.timeout_ns, 0x0A | (slot << 8))))
            return false;
          sph ^= 1u << slot;
          pending &= ~(1u << slot);
#pragma unroll
          for (int q = 0; q < 4; ++q) ca[q] = ld_shared_v4(sb + 16 * (lane + 32 * q));
          // A_scale rows past Nm were not loaded: any finite scale serves
          // (those MMA columns are not computed)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            cb[q] = lane + 32 * q < nm ? ld_shared_v4(sb + S::STG_BT + 16 * (lane + 32 * q))
                                       : make_uint4(0u, 0u, 0u, 0u);
          // these reads come before the slot's next load writes it
          fence_proxy_async_smem();
          __syncwarp();
          if (g + S::SD <= g_last) stage(g + S::SD);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) ca[q] = load16(p.b_scale, n0 + lane + 32 * q, p.N, g);
#pragma unroll
          for (int q = 0; q < 4; ++q) cb[q] = load16(p.a_scale, lane + 32 * q, p.M, g);
        }
        return true;
      };
      auto pick = [](const uint4 &x, int t) -> uint32_t {
        return t == 0 ? x.x : t == 1 ? x.y : t == 2 ? x.z : x.w;
      };
      int st = 0;
      uint32_t ph = 0;
      for (int ks = kb; ks < ke; ++ks) {
        if (ks == kb || (ks & 3) == 0) {
          if (!take(ks >> 2)) break;
        }
        if (!__all_sync(0xFFFFFFFFu, swap_wait<false>(bar_empty + 8 * st, ph ^ 1u, p.status,
                                                      abort_flag, p.timeout_ns, 0x09 | (st << 8))))
          break;
        const int t = ks & 3;
        const uint32_t sSF = base + S::OFF_SF + st * 2 * S::SF_BYTES + 16 * lane;
        st_shared_v4(sSF, pick(ca[0], t), pick(ca[1], t), pick(ca[2], t), pick(ca[3], t));
        st_shared_v4(sSF + S::SF_BYTES, pick(cb[0], t), pick(cb[1], t), pick(cb[2], t), pick(cb[3], t));
        // tcgen05.cp reads the chunks through the async proxy
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_full + 8 * st);
        if (++st == S::STAGES) {
          st = 0;
          ph ^= 1u;
        }
      }
      // staging loads still in flight (after a failed wait) land before the
      // CTA may finish
      for (int slot = 0; slot < S::SD; ++slot)
        if ((pending >> slot) & 1u)
          __all_sync(0xFFFFFFFFu, swap_wait<false>(bar_stg + 8 * slot, (sph >> slot) & 1u, p.status, never,
                                                   p.timeout_ns, 0x0B | (slot << 8)));
    }
  } else {
    // ------------------------------------------------------------ epilogue (load)
    const int q = warp & 3;  // the TMEM lane quarter this warp may read
    have_acc = __all_sync(0xFFFFFFFFu, swap_wait<false>(bar_acc, 0, p.status, abort_flag,
                                                        p.timeout_ns, 0x05));
    if (have_acc) {
      tc_fence_after();
      const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + S::TM_ACC;
      if constexpr (NT == 16) {
        tmem_ld_32x32b_x16(ta, v);
      } else {
#pragma unroll
        for (int c = 0; c < NT / 32; ++c)
          tmem_ld_32x32b_x32(ta + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
      }
      tmem_ld_wait();
    }
  }

  // ------------------------------------------------------------ K-split reduction
  // All threads of all CTAs of the cluster take part in both barriers.  The
  // first: every CTA has finished its main loop (its MMAs completed, its
  // loads landed), so the first CTA's operand ring is free to receive.  The
  // second: the partials have been written.
  const bool epi = warp >= 3;
  const int n = 32 * (warp & 3) + lane;  // accumulator lane: column n0 + n of C
  if (splits > 1) {
    cluster_sync();
    if (epi && split > 0) {
      // [other CTA][NT / 4][128 lanes] x 16 bytes in the first CTA's ring
      const uint32_t dst = mapa_shared(base, 0) +
                           static_cast<uint32_t>(((split - 1) * (NT / 4)) * 128 + n) * 16;
#pragma unroll
      for (int j4 = 0; j4 < NT / 4; ++j4)
        st_cluster_v4(dst + j4 * 128 * 16, v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
    }
    // a CTA whose accumulator never completed has said so in the status
    // word; its partial is then not added (C is incomplete either way)
    cluster_sync();
    if (epi && split == 0 && have_acc) {
      for (int r = 1; r < splits; ++r) {
        const uint32_t src = base + static_cast<uint32_t>(((r - 1) * (NT / 4)) * 128 + n) * 16;
#pragma unroll
        for (int j4 = 0; j4 < NT / 4; ++j4) {
          const uint4 o = ld_shared_v4(src + j4 * 128 * 16);
          v[4 * j4 + 0] = __float_as_uint(__uint_as_float(v[4 * j4 + 0]) + __uint_as_float(o.x));
          v[4 * j4 + 1] = __float_as_uint(__uint_as_float(v[4 * j4 + 1]) + __uint_as_float(o.y));
          v[4 * j4 + 2] = __float_as_uint(__uint_as_float(v[4 * j4 + 2]) + __uint_as_float(o.z));
          v[4 * j4 + 3] = __float_as_uint(__uint_as_float(v[4 * j4 + 3]) + __uint_as_float(o.w));
        }
      }
    }
  }

  // ------------------------------------------------------------ epilogue (store)
  // Row m of C, columns n0 .. n0+127: lane n of the warps holds column n0+n,
  // so each warp store covers 32 consecutive columns of one row.
  if (epi && split == 0 && have_acc) {
    const int col = n0 + n;
    if (col < p.N) {
#pragma unroll
      for (int m = 0; m < NT; ++m) {
        if (m < p.M) {
          const int64_t idx = static_cast<int64_t>(m) * p.N + col;
          float x = __uint_as_float(v[m]);
          if constexpr (!BF16) {
            float *cp = reinterpret_cast<float *>(p.C);
            if constexpr (ACC) x += cp[idx];
            cp[idx] = x;
          } else {
            __nv_bfloat16 *cp = reinterpret_cast<__nv_bfloat16 *>(p.C);
            if constexpr (ACC) x += __bfloat162float(cp[idx]);
            cp[idx] = __float2bfloat16_rn(x);
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<1>(tmem, S::TM_COLS);
}

}  // namespace mxg
