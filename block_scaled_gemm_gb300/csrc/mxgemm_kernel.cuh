// mxgemm_kernel.cuh -- the block-scaled (MXFP8) GEMM kernel for sm_103a.
//
//   C[M,N] (+)= (A * 2^(sA-127)) x (B * 2^(sB-127))
//
// Design (one CTA per SM, persistent, warp-specialised):
//   warp 0      TMA producer: per 128-deep K step loads the A tile (K-major,
//               128-byte swizzle), the B tile (N-major, 128-byte swizzle) and
//               (pairs) the A/B scale chunks into a STAGES-deep shared-memory
//               ring; each stage has a "full" barrier (arrives + expected
//               bytes) and an "empty" barrier (released by the MMA's commit).
//   warp 1      allocates TMEM; one thread issues, per K step, tcgen05.cp of
//               the scale chunks SMEM -> TMEM, then four
//               tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each) into an
//               FP32 TMEM accumulator, then tcgen05.commit -> empty[stage];
//               after a tile's last step, tcgen05.commit -> acc_full.
//   warps 2..9  epilogue: wait acc_full, tcgen05.ld the whole accumulator into
//               registers, release it (acc_empty) so the next tile's MMAs
//               start, then (optionally + C_in) round to FP32/BF16 and store.
//   warp 10     (single CTAs) scale loader: when the launch asks for it
//               (fused_scales: one row of tiles, M <= 128), builds each
//               stage's A and B scale chunks in shared memory straight from
//               the row-major A_scale and B_scale, so no prepass runs before
//               the kernel; otherwise (and always for pairs) the producer
//               loads chunks that a prepass repacked.
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
  // Scale chunks come either from a repack prepass (contiguous 512-byte
  // chunks, loaded by the producer's TMA with the stage) or, for single CTAs
  // when the kernel is told so (KParams::fused_scales), from the scale
  // loader warp, which builds them in shared memory from the row-major
  // scales.  Pairs always take the prepass: a chunk written by threads of one
  // CTA and read by the MMA that the other CTA issues would need a
  // cluster-scope release and acquire on every K step (a cluster-scope wait
  // there cost ~40% of the MMA rate).
  static constexpr bool HAS_SCALE_WARP = CG == 1;
  static constexpr uint32_t STAGE_TX = (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES) * CG;
  static constexpr uint32_t CHUNK_TX = (SFA_BYTES + SFB_BYTES) * CG;  // the scale chunks
  // half-width (128-column) tile: each CTA loads half of its B columns
  static constexpr uint32_t STAGE_TX_HALF = STAGE_TX - (B_BYTES / 2) * CG;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
  static constexpr int CLC_SLOTS = 4;  // cluster-launch-control response ring
  // full[], empty[], acc_full, acc_empty, final, clc_full[], clc_empty[],
  // stg (the scale loader's staging buffer has landed), stg_go (the scale
  // loader has issued its first staging load), cin[] (per epilogue warp:
  // its C_in chunks of the CTA's last tile have landed)
  static constexpr int NUM_BARS = 2 * STAGES + 3 + 2 * CLC_SLOTS + 2 + 8;
  static constexpr int OFF_CLC = (OFF_BAR + NUM_BARS * 8 + 15) / 16 * 16;  // 16-byte responses
  static constexpr int OFF_MISC = OFF_CLC + 16 * CLC_SLOTS;
  // epilogue staging: one 32-row x 64-byte buffer per epilogue warp
  static constexpr int EPI_BUF = 2048;
  static constexpr int OFF_EPI = (OFF_MISC + 16 + 1023) / 1024 * 1024;
  // scale loader staging (fused scales): one group of four K steps of raw
  // scale rows, 16 bytes per row: the tile's 128 A rows, then its 256 B rows
  static constexpr int STG_A_BYTES = 128 * 16;
  static constexpr int STG_BYTES = HAS_SCALE_WARP ? STG_A_BYTES + 256 * 16 : 0;
  static constexpr int OFF_STG = OFF_EPI + 8 * EPI_BUF;
  static constexpr int SMEM_BYTES = OFF_STG + STG_BYTES + 1024;  // + slack for 1 KB alignment
  static constexpr int TM_ACC = 0;
  static constexpr int TM_SFA = BN;               // STAGES x 4 columns
  static constexpr int TM_SFB = BN + 4 * STAGES;  // STAGES x 8 columns
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int SCALE_WARP = 2 + EPI_WARPS;  // with HAS_SCALE_WARP
  static constexpr int THREADS = 32 * (2 + EPI_WARPS + (HAS_SCALE_WARP ? 1 : 0));
  static_assert(TM_SFB + 8 * STAGES <= (int)TM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(OFF_B % 1024 == 0 && A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "align");
  static_assert(OFF_BAR % 8 == 0 && OFF_CLC % 16 == 0, "barrier and response alignment");
  static_assert(OFF_STG % 1024 == 0, "staging alignment");
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
  int tma_store;  // C's row pitch is a multiple of 16 bytes: stores go through TMA
  int *status;    // [0] code, [1] detail
  unsigned long long timeout_ns;
  int stall_producer;
  int use_clc;
  // stream-K tail (see WorkIter)
  int dp_tiles;        // tiles [0, dp_tiles) are computed whole, one CTA (pair) each
  int sk_ctas;         // CTAs (pairs) sharing the K steps of tiles [dp_tiles, num_tiles)
  long long sk_units;  // (num_tiles - dp_tiles) * k_steps
  float *partials;     // per CTA: 128 x 256 FP32 partial accumulator
  // per CTA and epilogue warp: the epoch of the launch whose partial rows
  // that warp has written (a value never equal to this launch's epoch until
  // it has been written in this launch, whatever earlier launches left)
  unsigned *flags;
  unsigned epoch;      // this launch's number, never 0
  // half-width tail (see WorkIter): items [dp_tiles, dp_tiles + half_tiles)
  // of the whole-tile walk are 128-column halves of tiles dp_tiles, ...
  int half_tiles;
  // element formats of A and B in instruction-descriptor position (bits
  // 7-9 and 10-12); 0 for E4M3 x E4M3
  uint32_t idesc_fmt;
  // the row-major scales, read by the scale loader (single CTAs):
  // A_scale M x kb_count, B_scale N x kb_count
  const uint8_t *a_scale;
  const uint8_t *b_scale;
  int kb_count;  // K / 32
  // single CTAs: the scale loader builds the chunks (else the producer loads
  // repacked chunks)
  int fused_scales;
  // with fused_scales: the scale maps (tmSFA, tmSFB) describe the row-major
  // scales (16-byte row pitch and base) and the scale loader stages its rows
  // by TMA; else it loads them with per-lane loads
  int scale_tma;
  // The launch before this one is the library's scale repack, which waited
  // for all earlier work on the stream: A and B are complete, and only the
  // scale chunks depend on that launch.  The producers of CTA pairs then send
  // the first ring round's A and B loads before the programmatic-dependent-
  // launch wait, and its chunk loads after it.
  int early_ab;
  // B given N x K (K contiguous); the kernel variant is chosen by it
  int b_kmajor;
};

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4.block_scale:
// E4M3 x E4M3, A K-major, B N-major, UE8M0 scales, M x N, scale byte ids.
// Other element formats are OR-ed in (fmt_bits).
// Descriptor code of an element format of kind::mxf8f6f4 (PTX ISA,
// instruction descriptor): E4M3 0, E5M2 1, E2M3 3, E3M2 4, E2M1 5; the
// argument is the C interface's format number (E4M3, E5M2, E2M3, E3M2,
// E2M1 = 0..4).
__host__ __device__ constexpr uint32_t mma_format_code(int f) {
  return f == 0 ? 0u : f == 1 ? 1u : f == 2 ? 3u : f == 3 ? 4u : 5u;
}
__host__ __device__ constexpr uint32_t fmt_bits(int a_fmt, int b_fmt) {
  return (mma_format_code(a_fmt) << 7) | (mma_format_code(b_fmt) << 10);
}

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

// Tile t -> (m tile, n tile): groups of 16 M-tiles walked N-fastest, so the
// CTAs running at one time share a few A and B strips in L2.  (MLP
// up-projection, pairs: groups of 16 measured 1.6 % faster than 8, 4 and
// 32 slower; B is read from DRAM once per group, A's rows of a group stay
// in L2.)
__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int &mt, int &nt) {
  constexpr int G = 16;
  const int per_group = G * n_tiles;
  const int g = t / per_group;
  const int first = g * G;
  const int gm = min(m_tiles - first, G);
  const int r = t - g * per_group;
  mt = first + r % gm;
  nt = r / gm;
}

// Work of one CTA (or CTA pair) u of P.  When the tiles do not divide into
// whole waves, the tiles after the last full wave (the "tail") are shared
// stream-K style: their K steps, laid end to end, are cut into sk_ctas equal
// contiguous ranges, one per CTA.  A range is shorter than one tile, so it
// touches at most two tiles: the start of one (a partial this CTA writes to
// its own slot) and the end of another (which this CTA finishes: it adds the
// other contributors' partials and stores C).  Each CTA does its tail work
// first, partial before finish, and then its whole tiles dp_tiles-ward
// (u, u+P, ...): every partial is written before anyone waits for it, and an
// owner's wait for partials overlaps the MMAs of its first whole tile.
// Alternatively, when the leftover tiles fill at most half a wave, each of
// them is computed as two 128-column halves by two CTAs (pairs): the last
// wave then takes half as long and needs no partial sums.
constexpr int kFull = 0;     // whole K range: store C
constexpr int kPartial = 1;  // first part of a tile's K range: write a partial
constexpr int kOwner = 2;    // last part: add the earlier parts' partials, store C

struct WorkItem {
  int tile;
  int kb, ke;         // K steps [kb, ke)
  int kind;
  int first_contrib;  // kOwner: CTAs first_contrib .. u-1 hold this tile's partials
  int half;           // -1: all 256 columns; 0 / 1: only that 128-column half
};

// Item t of the whole-tile walk: t < dp_tiles is tile t; the items after
// them are the 128-column halves of tiles dp_tiles, dp_tiles + 1, ...
__device__ __forceinline__ void item_to_work(int t, int dp_tiles, int k_steps, WorkItem &w) {
  w.kb = 0;
  w.ke = k_steps;
  w.kind = kFull;
  w.first_contrib = 0;
  if (t < dp_tiles) {
    w.tile = t;
    w.half = -1;
  } else {
    w.tile = dp_tiles + ((t - dp_tiles) >> 1);
    w.half = (t - dp_tiles) & 1;
  }
}

struct WorkIter {
  int u, P, dp_tiles, k_steps, sk_ctas, half_tiles;
  long long sk_units;
  int i = 0;         // next whole tile: u + i * P
  int tail_pos = 0;  // next tail segment (0: later tile, 1: earlier tile, 2: done)

  __device__ WorkIter(const KParams &p, int u_, int P_)
      : u(u_), P(P_), dp_tiles(p.dp_tiles), k_steps(p.k_steps), sk_ctas(p.sk_ctas),
        half_tiles(p.half_tiles), sk_units(p.sk_units) {
    if (sk_units == 0 || u >= sk_ctas) tail_pos = 2;
  }

  __device__ bool next(WorkItem &w) {
    while (tail_pos < 2) {
      const long long S = k_steps;
      const long long beg = static_cast<long long>(u) * sk_units / sk_ctas;
      const long long end = static_cast<long long>(u + 1) * sk_units / sk_ctas;
      const long long j0 = beg / S, j1 = (end - 1) / S;
      const int pos = tail_pos++;
      if (beg >= end || (pos == 1 && j0 == j1)) continue;
      const long long j = pos == 0 ? j1 : j0;
      const long long sb = beg > j * S ? beg : j * S;
      const long long se = end < (j + 1) * S ? end : (j + 1) * S;
      w.tile = dp_tiles + static_cast<int>(j);
      w.kb = static_cast<int>(sb - j * S);
      w.ke = static_cast<int>(se - j * S);
      const bool first = w.kb == 0, last = w.ke == k_steps;
      w.kind = last ? (first ? kFull : kOwner) : kPartial;
      // the CTA whose range holds the tile's first K step
      w.first_contrib = static_cast<int>(((j * S + 1) * sk_ctas - 1) / sk_units);
      w.half = -1;
      return true;
    }
    const int t = u + i * P;
    if (t >= dp_tiles + half_tiles) return false;
    ++i;
    item_to_work(t, dp_tiles, k_steps, w);
    return true;
  }
};

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

// Epilogue variants are compile-time: each instantiation carries only the
// store path it uses (a smaller footprint keeps the MMA issue loop's
// instructions resident).
constexpr int kEpiBF16 = 1;    // BF16 output (else FP32)
constexpr int kEpiAcc = 2;     // use_acc: C_in is read and added
constexpr int kEpiTma = 4;     // C's rows are 16-byte aligned: TMA stores
// (not an epilogue choice, but compiled the same way) B given N x K, K
// contiguous: its tiles are K-major in shared memory, like A's
constexpr int kEpiBKMajor = 8;

// Bounded wait (whole warp) until the n flag slots at `slots` (written by
// other CTAs after a fence) all hold `epoch`; lane i < n polls slot i.
__device__ __forceinline__ bool wait_flags(const unsigned *slots, int n, unsigned epoch,
                                           const WaitCtl &w, int detail) {
  const int lane = threadIdx.x & 31;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    unsigned v = epoch;
    if (lane < n)
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(slots + lane) : "memory");
    if (__all_sync(0xFFFFFFFFu, v == epoch)) return true;
    if ((it & 15u) == 15u) {
      bool give_up = *w.abort_flag != 0;
      if (!give_up && globaltimer_ns() - t0 > w.timeout_ns) {
        if (lane == 0 && atomicCAS(w.status, 0, kStatusTimeout) == 0) atomicExch(w.status + 1, detail);
        *w.abort_flag = 1;
        give_up = true;
      }
      if (__any_sync(0xFFFFFFFFu, give_up)) return false;
    }
    __nanosleep(64);
  }
}

// ---------------------------------------------------------------------------
// Work source under cluster launch control ("TLX API Quick Reference",
// section "CLC (Cluster Launch Control)").  The grid has one cluster per
// work item.  A resident cluster first takes its own item, then asks the
// hardware to cancel a cluster that has not launched yet and takes that
// cluster's item instead, until none is left to cancel.  The leader CTA's
// producer warp issues each request one item ahead, in the multicast form:
// the 16-byte response and its byte count land in every CTA of the cluster.
// Every role of every CTA reads the responses in order from a ring of
// CLC_SLOTS slots; the leader reuses a slot only after all readers released
// it (producer, MMA issuer and 8 epilogue warps in the leader, producer and
// 8 epilogue warps in the peer).  At most one request is outstanding, so none
// is issued after the one that found no cluster left.
struct ClcRing {
  uint32_t resp;       // response slot 0 (16 bytes per slot)
  uint32_t full;       // per-slot barrier: the response has landed in this CTA
  uint32_t empty;      // per-slot barrier of the leader CTA: readers done
  int slot = 0;        // next slot to read, and its ring phase
  uint32_t phase = 0;
  int rslot = 0;       // next slot to request into (leader's producer)
  uint32_t rphase = 0;
  bool first = true;   // the cluster's own item has not been taken yet
};

// Whole-warp call.  Returns the next item, -1 when no work is left, -2 on a
// timed-out wait (status recorded).
template <int CG, int SLOTS>
__device__ __noinline__ int clc_fetch(ClcRing &r, bool requester, uint32_t rank, const WaitCtl &wc) {
  const int lane = threadIdx.x & 31;
  int t;
  if (r.first) {
    r.first = false;
    t = static_cast<int>(blockIdx.x) / CG;
  } else {
    if (!__all_sync(0xFFFFFFFFu, wait_phase<false>(r.full + 8 * r.slot, r.phase, wc, 0x07 | (r.slot << 8))))
      return -2;
    const int x = clc_decode_x(r.resp + 16 * r.slot);
    __syncwarp();
    if (lane == 0) {
      if constexpr (CG == 1) mbar_arrive(r.empty + 8 * r.slot);
      else mbar_arrive_cluster(r.empty + 8 * r.slot, 0);
    }
    if (++r.slot == SLOTS) {
      r.slot = 0;
      r.phase ^= 1u;
    }
    if (x < 0) return -1;
    t = x / CG;
  }
  if (requester) {
    // the item after this one; each CTA expects the 16 response bytes on
    // its own barrier, the leader issues the request once the slot is free
    if (lane == 0) mbar_arrive_expect_tx(r.full + 8 * r.rslot, 16);
    if (rank == 0) {
      if (!__all_sync(0xFFFFFFFFu,
                      wait_phase<false>(r.empty + 8 * r.rslot, r.rphase ^ 1u, wc, 0x08 | (r.rslot << 8))))
        return -2;
      if (lane == 0) {
        if constexpr (CG == 1) clc_try_cancel(r.resp + 16 * r.rslot, r.full + 8 * r.rslot);
        else clc_try_cancel_all(r.resp + 16 * r.rslot, r.full + 8 * r.rslot);
      }
      __syncwarp();
    }
    if (++r.rslot == SLOTS) {
      r.rslot = 0;
      r.rphase ^= 1u;
    }
  }
  return t;
}

// The work source of one role: the static walk, or cluster launch control
// (whose ring position lives in the caller's ClcRing; the static walk's
// state stays in registers).
template <int CG, int SLOTS>
struct Sched {
  WorkIter wi;
  ClcRing *clc;
  const WaitCtl *wc;
  int dp_tiles, k_steps;
  bool use_clc, requester;
  uint32_t rank;
  __device__ Sched(const KParams &p, int u, int P, ClcRing *r, bool req, uint32_t rk,
                   const WaitCtl *w)
      : wi(p, u, P), clc(r), wc(w), dp_tiles(p.dp_tiles), k_steps(p.k_steps),
        use_clc(p.use_clc != 0), requester(req), rank(rk) {}
  __device__ bool next(WorkItem &w) {
    if (!use_clc) return wi.next(w);
    const int t = clc_fetch<CG, SLOTS>(*clc, requester, rank, *wc);
    if (t < 0) return false;
    item_to_work(t, dp_tiles, k_steps, w);
    return true;
  }
};

template <int CG, int EPI>
__global__ void __launch_bounds__(Cfg<CG>::THREADS, 1)
    mxgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmB64,
                  const __grid_constant__ CUtensorMap tmSFA,
                  const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ CUtensorMap tmC,
                  const KParams p) {
  using C = Cfg<CG>;
  constexpr bool kBF16 = (EPI & kEpiBF16) != 0;
  constexpr bool kAcc = (EPI & kEpiAcc) != 0;
  constexpr bool kTma = (EPI & kEpiTma) != 0;
  // B K-major: a B tile is [rows of B][128 K bytes], loaded by boxes of
  // 128 K bytes x 128 (64 for pair half-width tiles) rows, and read by the
  // MMA like A (no transpose bit, 32 bytes per K = 32); else B is N-major:
  // [128-column chunk][128 K rows][128 B], 4 KB per K = 32
  constexpr bool kBKM = (EPI & kEpiBKMajor) != 0;
  constexpr uint32_t kBNoT = kBKM ? ~(1u << 16) : ~0u;  // clears the transpose-B bit
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
  const uint32_t bar_clc_full = bar_final + 8;
  const uint32_t bar_clc_empty = bar_clc_full + 8 * C::CLC_SLOTS;
  const uint32_t bar_stg = bar_clc_empty + 8 * C::CLC_SLOTS;
  const uint32_t bar_stg_go = bar_stg + 8;
  const uint32_t bar_cin = bar_stg_go + 8;  // EPI_WARPS barriers
  const bool fused = C::HAS_SCALE_WARP && p.fused_scales != 0;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // full: the producer's arrive (with the TMA bytes), and with fused
      // scales the scale loader's arrive once its chunks are written
      mbar_init(bar_full + 8 * s, fused ? 2 : 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, C::EPI_WARPS * CG);
    mbar_init(bar_final, 1);
    for (int s = 0; s < C::CLC_SLOTS; ++s) {
      mbar_init(bar_clc_full + 8 * s, 1);
      // readers of a response: producer + 8 epilogue warps per CTA, the MMA
      // issuer, and the scale loader with fused scales
      mbar_init(bar_clc_empty + 8 * s, (1 + C::EPI_WARPS) * CG + 1 + (fused ? 1 : 0));
    }
    mbar_init(bar_stg, 1);
    mbar_init(bar_stg_go, 1);
    for (int i = 0; i < C::EPI_WARPS; ++i) mbar_init(bar_cin + 8 * i, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (CG == 2 && p.half_tiles > 0) tma_prefetch_desc(&tmB64);
    if (!fused || p.scale_tma) {
      tma_prefetch_desc(&tmSFA);
      tma_prefetch_desc(&tmSFB);
    }
    if (kTma) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  if constexpr (CG == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The set-up above overlaps the tail of the prepass before the kernel, if
  // any (the scale repack, the B re-pitch; programmatic dependent
  // launch); nothing below reads or writes global memory before that grid
  // has finished, except the producer's early A and B loads (early_ab),
  // whose warp waits for it itself.
  if (!(p.early_ab && warp == 0)) griddep_wait();

  const WaitCtl wc{p.status, abort_flag, p.timeout_ns};
  // Barriers completed by TMA byte counts or tcgen05.commit arrivals are
  // observed with CTA-scope acquire; only acc_empty, which the peer CTA's
  // epilogue warps release with cluster-scope arrives, is waited on with
  // cluster scope (a cluster-scope wait on every K step cost ~40% of the
  // pair's MMA rate).
  constexpr bool CL = (CG == 2);
  const int unit = blockIdx.x / CG;    // this CTA's (pair's) index in the persistent grid
  const int units = gridDim.x / CG;
  ClcRing clc_ring;
  clc_ring.resp = base + C::OFF_CLC;
  clc_ring.full = bar_clc_full;
  clc_ring.empty = bar_clc_empty;

  // The producer and MMA loops are unrolled over the ring stages: with the
  // stage index a compile-time constant every shared-memory address, TMEM
  // column and barrier of a step is a constant offset from a base, which
  // keeps the single issuing thread fast enough to hold the tensor pipe busy
  // (a rolled loop with a runtime stage index cost about 30% of MMA rate).
  // Code size matters as much: these loops run from the instruction cache,
  // and measured 5-20% slower whenever rarely taken code (another loop, a
  // tile-switch path per stage) grew around them.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // the whole warp runs the loop in lock-step; one elected lane issues
    {
      const bool leader = elect_one() != 0;
      uint32_t phase = 0;
      int nst = 0;           // next stage to fill ...
      uint32_t nph = 0;      // ... and the ring phase it belongs to
      ClcRing ring = clc_ring;
      Sched<CG, C::CLC_SLOTS> wi(p, unit, units, &ring, true, rank, &wc);
      WorkItem w;
      bool ok = !p.stall_producer && wi.next(w);
      // fused scales: the scale loader's first staging load goes to the TMA
      // unit ahead of the stages' A and B loads (behind them it would wait
      // for a whole ring of operand bytes and hold up the first MMA)
      if (fused && ok)
        ok = __all_sync(0xFFFFFFFFu, wait_phase<false>(bar_stg_go, 0, wc, 0x0C));
      int ks = w.kb, mt = 0, nt = 0;
      if (ok) tile_coords(w.tile, p.m_tiles, p.n_tiles, mt, nt);
      // whole tiles in the unrolled loop below; half-width tiles (only ever
      // at the end of the walk) in the rolled loop after it
      bool go_half = false;
      if (ok && w.half >= 0) {
        go_half = true;
        ok = false;
      }
      // one whole-tile K step into stage st (elected lane)
      auto load_whole = [&](int st) {
        const uint32_t fb = bar_full + 8 * st;
        const uint32_t sA = base + C::OFF_A + st * C::A_BYTES;
        const uint32_t sB = base + C::OFF_B + st * C::B_BYTES;
        const uint32_t sSA = base + C::OFF_SFA + st * C::SFA_BYTES;
        const uint32_t sSB = base + C::OFF_SFB + st * C::SFB_BYTES;
        const int row0 = mt * (128 * CG) + 128 * (int)rank;  // this CTA's A rows
        const int mblk = mt * CG + (int)rank;                  // its 128-row block
        const int col0 = nt * 256;
        const int k0 = ks * 128;
        if constexpr (CG == 1) {
          // (fused: the scale chunks come from the scale loader)
          mbar_arrive_expect_tx(fb, fused ? C::STAGE_TX - C::CHUNK_TX : C::STAGE_TX);
          tma_load_2d(sA, &tmA, k0, row0, fb);
          if constexpr (kBKM) {
            tma_load_2d(sB, &tmB, k0, col0, fb);
            tma_load_2d(sB + 16384, &tmB, k0, col0 + 128, fb);
          } else {
            tma_load_2d(sB, &tmB, col0, k0, fb);
            tma_load_2d(sB + 16384, &tmB, col0 + 128, k0, fb);
          }
          if (!fused) {
            tma_load_2d(sSA, &tmSFA, 0, (mblk * p.k_steps + ks) * 4, fb);
            tma_load_2d(sSB, &tmSFB, 0, (nt * p.k_steps + ks) * 8, fb);
          }
        } else {
          if (rank == 0) mbar_arrive_expect_tx(fb, C::STAGE_TX);
          const uint32_t fbl = mapa_shared(fb, 0);  // leader's barrier
          tma_load_2d_pair(sA, &tmA, k0, row0, fbl);
          if constexpr (kBKM) tma_load_2d_pair(sB, &tmB, k0, col0 + 128 * (int)rank, fbl);
          else tma_load_2d_pair(sB, &tmB, col0 + 128 * (int)rank, k0, fbl);
          tma_load_2d_pair(sSA, &tmSFA, 0, (mblk * p.k_steps + ks) * 4, fbl);
          tma_load_2d_pair(sSB, &tmSFB, 0, (nt * p.k_steps + ks) * 8, fbl);
        }
      };
      // early_ab: the first ring round's A and B go out before the wait for
      // the scale repack, its chunks after (pairs whose first item is a
      // whole tile with more K steps than the ring has stages); otherwise the
      // wait comes first.
      int pre = 0;  // stages of the first ring round filled here
      if (p.early_ab) {
        if (CG == 2 && ok && w.ke - w.kb > C::STAGES) {
          const int row0 = mt * (128 * CG) + 128 * (int)rank;
          const int mblk = mt * CG + (int)rank;
          for (int st = 0; st < C::STAGES; ++st) {
            if (leader) {
              const uint32_t fb = bar_full + 8 * st;
              if (rank == 0) mbar_arrive_expect_tx(fb, C::STAGE_TX);
              const uint32_t fbl = mapa_shared(fb, 0);
              tma_load_2d_pair(base + C::OFF_A + st * C::A_BYTES, &tmA, (w.kb + st) * 128, row0, fbl);
              if constexpr (kBKM)
                tma_load_2d_pair(base + C::OFF_B + st * C::B_BYTES, &tmB, (w.kb + st) * 128,
                                 nt * 256 + 128 * (int)rank, fbl);
              else
                tma_load_2d_pair(base + C::OFF_B + st * C::B_BYTES, &tmB, nt * 256 + 128 * (int)rank,
                                 (w.kb + st) * 128, fbl);
            }
            __syncwarp();
          }
          griddep_wait();
          for (int st = 0; st < C::STAGES; ++st) {
            if (leader) {
              const uint32_t fbl = mapa_shared(bar_full + 8 * st, 0);
              tma_load_2d_pair(base + C::OFF_SFA + st * C::SFA_BYTES, &tmSFA, 0,
                               (mblk * p.k_steps + w.kb + st) * 4, fbl);
              tma_load_2d_pair(base + C::OFF_SFB + st * C::SFB_BYTES, &tmSFB, 0,
                               (nt * p.k_steps + w.kb + st) * 8, fbl);
            }
            __syncwarp();
          }
          pre = C::STAGES;
          ks = w.kb + C::STAGES;
        } else {
          griddep_wait();
        }
      }
      if constexpr (CG == 2) {
        // Pairs: the unrolled loop holds only the per-step work; a stage
        // that is not free yet, or a tile boundary, is handled after it
        // (measured faster for pairs; slower for single CTAs, whose 4-stage
        // ring is refilled late by the extra exit and re-entry).
        int skip = 0;  // stages of the current ring round already filled
        if (pre == C::STAGES) {  // the first ring round went out above
          phase = 1u;
          nst = 0;
          nph = 1u;
        }
        while (ok) {
          bool tile_end = false, must_wait = false;
#pragma unroll
          for (int st = 0; st < C::STAGES; ++st) {
            if (skip > 0) {
              --skip;
              continue;
            }
            if (!__all_sync(0xFFFFFFFFu, mbar_test_wait(bar_empty + 8 * st, phase ^ 1u))) {
              must_wait = true;
              break;
            }
            if (leader) load_whole(st);
            __syncwarp();
            nst = (st + 1 == C::STAGES) ? 0 : st + 1;
            nph = (st + 1 == C::STAGES) ? (phase ^ 1u) : phase;
            if (++ks == w.ke) {
              tile_end = true;
              break;
            }
          }
          if (!must_wait && !tile_end) {  // a whole ring round
            phase ^= 1u;
            continue;
          }
          // resume at stage nst of the ring round of phase nph
          phase = nph;
          skip = nst;
          if (tile_end) {
            if (!wi.next(w)) break;
            ks = w.kb;
            tile_coords(w.tile, p.m_tiles, p.n_tiles, mt, nt);
            if (w.half >= 0) {
              go_half = true;
              break;
            }
          } else {
            ok = __all_sync(0xFFFFFFFFu,
                            wait_phase<false>(bar_empty + 8 * nst, nph ^ 1u, wc, 0x01 | (nst << 8)));
          }
        }
      } else {
        while (ok) {
#pragma unroll
          for (int st = 0; st < C::STAGES; ++st) {
            if (ok) {
              if (!__all_sync(0xFFFFFFFFu,
                              wait_phase<false>(bar_empty + 8 * st, phase ^ 1u, wc, 0x01 | (st << 8)))) {
                ok = false;
              } else {
                if (leader) load_whole(st);
                __syncwarp();
                nst = (st + 1 == C::STAGES) ? 0 : st + 1;
                nph = (st + 1 == C::STAGES) ? (phase ^ 1u) : phase;
                if (++ks == w.ke) {
                  if (wi.next(w)) {
                    ks = w.kb;
                    tile_coords(w.tile, p.m_tiles, p.n_tiles, mt, nt);
                    if (w.half >= 0) {
                      go_half = true;
                      ok = false;
                    }
                  } else {
                    ok = false;
                  }
                }
              }
            }
          }
          if (ok) phase ^= 1u;
        }
      }
      // half-width tiles: rolled loop, runtime stage index (nst, nph)
      while (go_half) {
        if (!__all_sync(0xFFFFFFFFu, wait_phase<false>(bar_empty + 8 * nst, nph ^ 1u, wc, 0x01 | (nst << 8))))
          break;
        if (leader) {
          const uint32_t fb = bar_full + 8 * nst;
          const uint32_t sA = base + C::OFF_A + nst * C::A_BYTES;
          const uint32_t sB = base + C::OFF_B + nst * C::B_BYTES;
          const uint32_t sSA = base + C::OFF_SFA + nst * C::SFA_BYTES;
          const uint32_t sSB = base + C::OFF_SFB + nst * C::SFB_BYTES;
          const int row0 = mt * (128 * CG) + 128 * (int)rank;
          const int mblk = mt * CG + (int)rank;
          const int col0 = nt * 256 + 128 * w.half;
          const int k0 = ks * 128;
          if constexpr (CG == 1) {
            mbar_arrive_expect_tx(fb, fused ? C::STAGE_TX_HALF - C::CHUNK_TX : C::STAGE_TX_HALF);
            tma_load_2d(sA, &tmA, k0, row0, fb);
            if constexpr (kBKM) tma_load_2d(sB, &tmB, k0, col0, fb);
            else tma_load_2d(sB, &tmB, col0, k0, fb);
            if (!fused) {
              tma_load_2d(sSA, &tmSFA, 0, (mblk * p.k_steps + ks) * 4, fb);
              tma_load_2d(sSB, &tmSFB, 0, (nt * p.k_steps + ks) * 8, fb);
            }
          } else {
            if (rank == 0) mbar_arrive_expect_tx(fb, C::STAGE_TX_HALF);
            const uint32_t fbl = mapa_shared(fb, 0);
            tma_load_2d_pair(sA, &tmA, k0, row0, fbl);
            // 64 columns per CTA (N-major: 64-byte swizzle; K-major: 64 rows)
            if constexpr (kBKM) tma_load_2d_pair(sB, &tmB64, k0, col0 + 64 * (int)rank, fbl);
            else tma_load_2d_pair(sB, &tmB64, col0 + 64 * (int)rank, k0, fbl);
            tma_load_2d_pair(sSA, &tmSFA, 0, (mblk * p.k_steps + ks) * 4, fbl);
            tma_load_2d_pair(sSB, &tmSFB, 0, (nt * p.k_steps + ks) * 8, fbl);
          }
        }
        __syncwarp();
        if (++nst == C::STAGES) {
          nst = 0;
          nph ^= 1u;
        }
        if (++ks == w.ke) {
          if (!wi.next(w)) break;
          ks = w.kb;
          tile_coords(w.tile, p.m_tiles, p.n_tiles, mt, nt);
        }
      }
      // Drain: every stage's last fill has been consumed (its MMA commit has
      // arrived) before this CTA may finish.
      for (int i = 0; i < C::STAGES; ++i) {
        if (!__all_sync(0xFFFFFFFFu, wait_phase<false>(bar_empty + 8 * nst, nph ^ 1u, wc, 0x11 | (nst << 8))))
          break;
        if (++nst == C::STAGES) {
          nst = 0;
          nph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The tensor pipe does not run ahead of the issuing thread: every
    // instruction between two MMAs adds to the K step's time.  The whole warp
    // runs the loop in lock-step (warp-uniform control flow) and one elected
    // lane issues; the next stage's full barrier is probed right after the
    // current stage's first MMA, hiding the probe's latency behind the other
    // three.
    if (rank == 0) {
      const bool leader = elect_one() != 0;
      uint32_t phase = 0, acc_phase = 0;
      const uint32_t fmt = p.idesc_fmt;  // element formats (0: E4M3 x E4M3)
      ClcRing ring = clc_ring;
      Sched<CG, C::CLC_SLOTS> wi(p, unit, units, &ring, false, rank, &wc);
      WorkItem w;
      bool ok = wi.next(w);
      int ks = w.kb;
      // whole tiles in the unrolled loop; half-width tiles (only ever at the
      // end of the walk) in the rolled loop after it, from stage hst
      bool go_half = false;
      int hst = 0;
      uint32_t hph = 0;
      if (ok && w.half >= 0) {
        go_half = true;
        ok = false;
      }
      if (ok) {
        ok = __all_sync(0xFFFFFFFFu, wait_phase<CL>(bar_acc_empty, acc_phase ^ 1u, wc, 0x02));
        tc_fence_after();
        if (ok) ok = __all_sync(0xFFFFFFFFu, wait_phase<false>(bar_full, 0, wc, 0x03));
      }
      // one whole-tile K step from stage st (elected lane); returns whether
      // stage nst (phase nph) is already full, probed after the first MMA
      auto mma_whole = [&](int st, int nst, uint32_t nph) -> uint32_t {
        const uint32_t sA = base + C::OFF_A + st * C::A_BYTES;
        const uint32_t sB = base + C::OFF_B + st * C::B_BYTES;
        const uint32_t sSA = base + C::OFF_SFA + st * C::SFA_BYTES;
        const uint32_t sSB = base + C::OFF_SFB + st * C::SFB_BYTES;
        const uint32_t tSA = tmem + C::TM_SFA + 4 * st;
        const uint32_t tSB = tmem + C::TM_SFB + 8 * st;
        // scale chunks: 32 rows x 16 bytes each, no swizzle, 8-row groups 128 B apart
        tmem_cp_32x128b_x4<CG>(tSA, smem_desc(sSA, 0, 128, 0));
        tmem_cp_32x128b_x4<CG>(tSB, smem_desc(sSB, 0, 128, 0));
        tmem_cp_32x128b_x4<CG>(tSB + 4, smem_desc(sSB + 512, 0, 128, 0));
        // A: K-major, 128-byte swizzle, 8-row groups 1024 B apart; 32 B per K=32.
        // B: N-major, 128-byte swizzle; 128-column chunks 16 KB apart,
        // 8-row K groups 1024 B apart; 32 rows (4 KB) per K=32.
        mma_mxf8<CG>(tmem + C::TM_ACC, smem_desc(sA, 0, 1024, 2),
                     kBKM ? smem_desc(sB, 0, 1024, 2) : smem_desc(sB, 16384, 1024, 2),
                     (idesc_mxf8(128 * CG, 256, 0, 0) | fmt) & kBNoT, tSA, tSB, ks != w.kb);
        const uint32_t ready = mbar_test_wait(bar_full + 8 * nst, nph);
#pragma unroll
        for (int k = 1; k < 4; ++k)
          mma_mxf8<CG>(tmem + C::TM_ACC, smem_desc(sA + 32 * k, 0, 1024, 2),
                       kBKM ? smem_desc(sB + 32 * k, 0, 1024, 2) : smem_desc(sB + 4096 * k, 16384, 1024, 2),
                       (idesc_mxf8(128 * CG, 256, k, k) | fmt) & kBNoT, tSA,
                       tSB, 1u);
        if constexpr (CG == 1) tc_commit(bar_empty + 8 * st);
        else tc_commit_pair(bar_empty + 8 * st, 0x3);
        return ready;
      };
      if constexpr (CG == 2) {
        // Pairs: the unrolled loop holds only the per-step work.  A tile
        // boundary, or a next stage that is not full yet, leaves it for the
        // code after it (one copy instead of one per stage), which re-enters
        // the loop at that stage.
        int skip = 0;  // stages of the current ring round already done
        while (ok) {
          int exit_st = -1;  // next stage, when the loop was left early
          bool tile_end = false;
#pragma unroll
          for (int st = 0; st < C::STAGES; ++st) {
            if (skip > 0) {
              --skip;
              continue;
            }
            // stage st is full
            const int nst = (st + 1 == C::STAGES) ? 0 : st + 1;
            const uint32_t nph = (st + 1 == C::STAGES) ? (phase ^ 1u) : phase;
            uint32_t next_ready = 0;
            if (leader) next_ready = mma_whole(st, nst, nph);
            __syncwarp();
            next_ready = __shfl_sync(0xFFFFFFFFu, next_ready, __ffs(__ballot_sync(0xFFFFFFFFu, leader)) - 1);
            if (++ks == w.ke) {
              tile_end = true;
              exit_st = nst;
              break;
            }
            if (!next_ready) {
              exit_st = nst;
              break;
            }
          }
          if (exit_st < 0) {  // a whole ring round
            phase ^= 1u;
            continue;
          }
          if (exit_st == 0) phase ^= 1u;  // the round ended with its last stage
          skip = exit_st;
          if (tile_end) {
            if (leader) tc_commit_pair(bar_acc_full, 0x3);
            __syncwarp();
            acc_phase ^= 1u;
            if (!wi.next(w)) break;
            if (w.half >= 0) {
              go_half = true;
              hst = exit_st;
              hph = phase;
              break;
            }
            ks = w.kb;
            ok = __all_sync(0xFFFFFFFFu, wait_phase<CL>(bar_acc_empty, acc_phase ^ 1u, wc,
                                                        0x02 | ((w.tile & 0xFFFF) << 16)));
            if (!ok) break;
            tc_fence_after();
          }
          ok = __all_sync(0xFFFFFFFFu,
                          wait_phase<false>(bar_full + 8 * exit_st, phase, wc, 0x03 | (exit_st << 8)));
        }
      } else {
        while (ok) {
#pragma unroll
          for (int st = 0; st < C::STAGES; ++st) {
            if (ok) {
              // stage st is full
              const int nst = (st + 1 == C::STAGES) ? 0 : st + 1;
              const uint32_t nph = (st + 1 == C::STAGES) ? (phase ^ 1u) : phase;
              uint32_t next_ready = 0;
              if (leader) next_ready = mma_whole(st, nst, nph);
              __syncwarp();
              next_ready =
                  __shfl_sync(0xFFFFFFFFu, next_ready, __ffs(__ballot_sync(0xFFFFFFFFu, leader)) - 1);
              if (++ks == w.ke) {
                if (leader) tc_commit(bar_acc_full);
                __syncwarp();
                acc_phase ^= 1u;
                if (!wi.next(w)) {
                  ok = false;
                } else if (w.half >= 0) {
                  go_half = true;
                  hst = nst;
                  hph = nph;
                  ok = false;
                } else {
                  ks = w.kb;
                  ok = __all_sync(0xFFFFFFFFu, wait_phase<CL>(bar_acc_empty, acc_phase ^ 1u, wc,
                                                              0x02 | ((w.tile & 0xFFFF) << 16)));
                  if (ok) tc_fence_after();
                }
              }
              if (ok && !next_ready)
                ok = __all_sync(0xFFFFFFFFu,
                                wait_phase<false>(bar_full + 8 * nst, nph, wc, 0x03 | (nst << 8)));
            }
          }
          if (ok) phase ^= 1u;
        }
      }
      // Half-width tiles: N = 128 MMAs; B scales are the matching 128-row
      // half of the 256-column chunk.  Pairs hold 64 B columns per CTA
      // (64-byte swizzle, 8-row K groups 512 B apart).
      if (go_half) {
        int s = hst;
        uint32_t ph = hph;
        const uint64_t bdesc = kBKM    ? smem_desc(0, 0, 1024, 2)
                               : CG == 2 ? smem_desc(0, 8192, 512, 4)
                                         : smem_desc(0, 16384, 1024, 2);
        const uint32_t bstep = kBKM ? 32 : CG == 2 ? 2048 : 4096;
        bool run = true;
        while (run) {
          run = __all_sync(0xFFFFFFFFu, wait_phase<CL>(bar_acc_empty, acc_phase ^ 1u, wc,
                                                       0x02 | ((w.tile & 0xFFFF) << 16)));
          if (!run) break;
          tc_fence_after();
          // the B scales of this half: one of the chunk's two 128-row halves
          const uint32_t sfb_half = 512u * static_cast<uint32_t>(w.half);
          for (int k0 = w.kb; k0 < w.ke; ++k0) {
            if (!__all_sync(0xFFFFFFFFu, wait_phase<false>(bar_full + 8 * s, ph, wc, 0x03 | (s << 8)))) {
              run = false;
              break;
            }
            if (leader) {
              const uint32_t sA = base + C::OFF_A + s * C::A_BYTES;
              const uint32_t sB = base + C::OFF_B + s * C::B_BYTES;
              const uint32_t sSA = base + C::OFF_SFA + s * C::SFA_BYTES;
              const uint32_t sSB = base + C::OFF_SFB + s * C::SFB_BYTES;
              const uint32_t tSA = tmem + C::TM_SFA + 4 * s;
              const uint32_t tSB = tmem + C::TM_SFB + 8 * s;
              // two scale copies, not three: at N = 128 the copies are not
              // hidden behind the MMAs
              tmem_cp_32x128b_x4<CG>(tSA, smem_desc(sSA, 0, 128, 0));
              tmem_cp_32x128b_x4<CG>(tSB, smem_desc(sSB + sfb_half, 0, 128, 0));
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_mxf8<CG>(tmem + C::TM_ACC, smem_desc(sA + 32 * k, 0, 1024, 2),
                             bdesc | ((sB + bstep * k) >> 4), (idesc_mxf8(128 * CG, 128, k, k) | fmt) & kBNoT, tSA,
                             tSB, (k0 != w.kb || k != 0) ? 1u : 0u);
              if constexpr (CG == 1) tc_commit(bar_empty + 8 * s);
              else tc_commit_pair(bar_empty + 8 * s, 0x3);
            }
            __syncwarp();
            if (++s == C::STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (!run) break;
          if (leader) {
            if constexpr (CG == 1) tc_commit(bar_acc_full);
            else tc_commit_pair(bar_acc_full, 0x3);
          }
          __syncwarp();
          acc_phase ^= 1u;
          run = wi.next(w);
        }
      }
      // all issued tcgen05 work has finished before TMEM can be released
      if (leader) {
        if constexpr (CG == 1) tc_commit(bar_final);
        else tc_commit_pair(bar_final, 0x1);
      }
      __syncwarp();
      WaitCtl wf = wc;
      wf.abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 8);  // never raised
      if (lane == 0) *wf.abort_flag = 0;
      __syncwarp();
      wait_phase<false>(bar_final, 0, wf, 0x04);
    }
  } else if (C::HAS_SCALE_WARP && warp == C::SCALE_WARP) {
    // ------------------------------------------------------------ scale loader
    // Per K step, the stage's A scale chunk (the tile's 128 rows) and B scale
    // chunks (its 256 columns, as two 128-row chunks) in the byte order that
    // tcgen05.cp .32x128b.warpx4 takes: lane l writes the 16-byte row l of
    // each chunk, whose 4-byte word q holds the step's four K-block scales of
    // row l + 32 q.  Those are four consecutive bytes of that row of A_scale
    // (B_scale), so a group of four K steps needs 16 bytes of each of the
    // tile's rows, and a chunk row is one word of each of four such 16-byte
    // row segments.
    //   The segments of a group are staged by TMA (2-D boxes of 16 bytes x
    // 128 A rows and x 256 B rows; rows beyond M or N read as zero, i.e.
    // 2^-127, and meet only the zero-filled operand rows there) while the
    // previous group's chunks are written; lane l then reads its rows from
    // the staging buffer.  Per-lane global loads of the segments (32 rows per
    // load instruction) measured ~27% off the MMA rate of single-CTA tiles,
    // so they serve only scales whose row pitch or base rules out TMA (K not
    // a multiple of 512, or an unaligned pointer): byte loads, 127 past the
    // end of a row.
    //   A stage is handed to the MMA issuer by an arrive on its full barrier
    // after a proxy fence (tcgen05.cp reads the chunks through the async
    // proxy).
    if (C::HAS_SCALE_WARP && fused) {
      ClcRing ring = clc_ring;
      Sched<CG, C::CLC_SLOTS> wi(p, unit, units, &ring, false, rank, &wc);
      WorkItem w, wn;
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      const bool tma = p.scale_tma != 0;
      const uint32_t stg = base + C::OFF_STG;
      uint32_t sph = 0;     // phase of the staging barrier
      bool staged = false;  // a staging load is issued and not yet read
      const int kbn = p.kb_count;
      uint4 ca[4], cb[8];   // the current group's segments: A rows lane + 32 q, B rows
      // group g (K steps 4g .. 4g+3) of item `it`: start its staging load
      auto stage = [&](const WorkItem &it, int g) {
        if (!tma) return;
        int mt = 0, nt = 0;
        tile_coords(it.tile, p.m_tiles, p.n_tiles, mt, nt);
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_stg, C::STG_BYTES);
          tma_load_2d(stg, &tmSFA, 16 * g, mt * 128, bar_stg);
          tma_load_2d(stg + C::STG_A_BYTES, &tmSFB, 16 * g, nt * 256, bar_stg);
        }
        __syncwarp();
        staged = true;
      };
      // 16 scale bytes (K-blocks 16 g .. 16 g + 15) of row `row` of S, byte by byte
      auto load16 = [&](const uint8_t *S, int64_t row, int64_t rows, int g) -> uint4 {
        uint32_t x[4] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu};
        if (row < rows) {
          const uint8_t *src = S + row * kbn + 16 * g;
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const uint32_t v = 16 * g + b < kbn ? static_cast<uint32_t>(src[b]) : 127u;
            x[b >> 2] = (x[b >> 2] & ~(0xFFu << (8 * (b & 3)))) | (v << (8 * (b & 3)));
          }
        }
        return make_uint4(x[0], x[1], x[2], x[3]);
      };
      // make group g of item `it` the current one
      auto take = [&](const WorkItem &it, int g) -> bool {
        if (tma) {
          if (!__all_sync(0xFFFFFFFFu, wait_phase<false>(bar_stg, sph, wc, 0x0A)))
            return false;
          sph ^= 1u;
          staged = false;
#pragma unroll
          for (int q = 0; q < 4; ++q) ca[q] = ld_shared_v4(stg + 16 * (lane + 32 * q));
#pragma unroll
          for (int q = 0; q < 8; ++q) cb[q] = ld_shared_v4(stg + C::STG_A_BYTES + 16 * (lane + 32 * q));
          // the reads are ordered before the next staging load's writes
          fence_proxy_async_smem();
          __syncwarp();
        } else {
          int mt = 0, nt = 0;
          tile_coords(it.tile, p.m_tiles, p.n_tiles, mt, nt);
          const int64_t arow = static_cast<int64_t>(mt) * 128 + lane;
          const int64_t brow = static_cast<int64_t>(nt) * 256 + lane;
#pragma unroll
          for (int q = 0; q < 4; ++q) ca[q] = load16(p.a_scale, arow + 32 * q, p.M, g);
#pragma unroll
          for (int q = 0; q < 8; ++q) cb[q] = load16(p.b_scale, brow + 32 * q, p.N, g);
        }
        return true;
      };
      auto pick = [](const uint4 &x, int t) -> uint32_t {
        return t == 0 ? x.x : t == 1 ? x.y : t == 2 ? x.z : x.w;
      };
      bool have = wi.next(w), have_n = false;
      if (have) stage(w, w.kb >> 2);
      if (lane == 0) mbar_arrive(bar_stg_go);  // the producer may start
      while (ok && have) {
        for (int ks = w.kb; ks < w.ke; ++ks) {
          const int g = ks >> 2;
          if (ks == w.kb || (ks & 3) == 0) {
            // this group becomes current; the next one (of this item, else
            // the first of the next item) is staged meanwhile
            if (!take(w, g)) {
              ok = false;
              break;
            }
            if (4 * (g + 1) < w.ke) {
              stage(w, g + 1);
            } else {
              have_n = wi.next(wn);
              if (have_n) stage(wn, wn.kb >> 2);
            }
          }
          if (!__all_sync(0xFFFFFFFFu,
                          wait_phase<false>(bar_empty + 8 * st, ph ^ 1u, wc, 0x09 | (st << 8)))) {
            ok = false;
            break;
          }
          const int t = ks & 3;
          const uint32_t sSA = base + C::OFF_SFA + st * C::SFA_BYTES + 16 * lane;
          const uint32_t sSB = base + C::OFF_SFB + st * C::SFB_BYTES + 16 * lane;
          st_shared_v4(sSA, pick(ca[0], t), pick(ca[1], t), pick(ca[2], t), pick(ca[3], t));
          st_shared_v4(sSB, pick(cb[0], t), pick(cb[1], t), pick(cb[2], t), pick(cb[3], t));
          st_shared_v4(sSB + 512, pick(cb[4], t), pick(cb[5], t), pick(cb[6], t), pick(cb[7], t));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_full + 8 * st);
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
        w = wn;
        have = have_n;
      }
      // after a failed wait: a staging load still in flight lands before
      // the CTA may finish
      if (staged) {
        WaitCtl wf = wc;
        wf.abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 12);  // never raised
        if (lane == 0) *wf.abort_flag = 0;
        __syncwarp();
        __all_sync(0xFFFFFFFFu, wait_phase<false>(bar_stg, sph, wf, 0x0B));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;  // 0..7
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    const int h = ew >> 2;    // which half of the tile's columns
    uint32_t acc_phase = 0;
    ClcRing ring = clc_ring;
    Sched<CG, C::CLC_SLOTS> wi(p, unit, units, &ring, false, rank, &wc);
    WorkItem w;
    while (wi.next(w)) {
      const int t = w.tile;
      int mt, nt;
      tile_coords(t, p.m_tiles, p.n_tiles, mt, nt);
      // this warp's columns: 128 of a whole tile, 64 of a half-width tile
      const bool whole = w.half < 0;
      const int ncols = whole ? 128 : 64;
      const int tcol = whole ? 128 * h : 64 * h;  // first accumulator column
      const int colb = nt * 256 + (whole ? 128 * h : 128 * w.half + 64 * h);
      if (kAcc && kTma && w.kind != kPartial && lane == 0) {
        // pull this warp's part of C_in into L2 while the tile's MMAs run
        const int r0 = mt * (128 * CG) + 128 * (int)rank + 32 * q;
        const int cw = kBF16 ? 64 : 32;  // the store boxes: 128 bytes x 16 rows
        for (int c0 = colb; c0 < colb + ncols && c0 < p.N; c0 += cw)
          for (int rh = 0; rh < 2; ++rh)
            if (r0 + 16 * rh < p.M) tma_prefetch_l2_2d(&tmC, c0, r0 + 16 * rh);
      }
      // all lanes wait (warp-uniform control flow)
      if (!__all_sync(0xFFFFFFFFu,
                      wait_phase<false>(bar_acc_full, acc_phase, wc, 0x05 | ((t & 0xFFFF) << 16))))
        break;
      tc_fence_after();
      uint32_t v[4][32];
      const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + C::TM_ACC + tcol;
      tmem_ld_32x32b_x32(ta + 0, v[0]);
      tmem_ld_32x32b_x32(ta + 32, v[1]);
      if (whole) {
        tmem_ld_32x32b_x32(ta + 64, v[2]);
        tmem_ld_32x32b_x32(ta + 96, v[3]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 1) mbar_arrive(bar_acc_empty);
        else mbar_arrive_cluster(bar_acc_empty, 0);
      }
      acc_phase ^= 1u;

      // the accumulator row this lane holds
      const bool row_ok = mt * (128 * CG) + 128 * (int)rank + 32 * q + lane < p.M;
      if (w.kind == kPartial) {
        // first part of a split tile: the FP32 partial to this CTA's slot,
        // then this warp's flag slot set to the launch's epoch.  The slot is laid out by
        // (warp, 4-column group, lane) -- the reader uses the same warp/lane
        // to row mapping -- so every warp access covers 512 contiguous bytes.
        // Rows beyond M are neither written nor read.
        float4 *slot = reinterpret_cast<float4 *>(p.partials) +
                       static_cast<int64_t>(unit * CG + (int)rank) * (128 * 256 / 4) + ew * (32 * 32) + lane;
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < 128; c += 4)
            __stcg(slot + (c / 4) * 32,
                   make_float4(__uint_as_float(v[c >> 5][(c & 31) + 0]), __uint_as_float(v[c >> 5][(c & 31) + 1]),
                               __uint_as_float(v[c >> 5][(c & 31) + 2]), __uint_as_float(v[c >> 5][(c & 31) + 3])));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicExch(p.flags + (unit * CG + (int)rank) * C::EPI_WARPS + ew, p.epoch);
        continue;
      }
      if (w.kind == kOwner) {
        // last part: add the partials of the CTAs that computed the earlier parts
        bool got = true;
        for (int c = w.first_contrib; c < unit && got; ++c) {
          // all eight epilogue warps of contributor c have written
          const bool ready = wait_flags(p.flags + (c * CG + (int)rank) * C::EPI_WARPS, C::EPI_WARPS,
                                        p.epoch, wc, 0x06 | ((t & 0xFFFF) << 16));
          if (!ready) {
            got = false;
            break;
          }
          __threadfence();
          const float4 *slot = reinterpret_cast<const float4 *>(p.partials) +
                               static_cast<int64_t>(c * CG + (int)rank) * (128 * 256 / 4) + ew * (32 * 32) + lane;
          // the row test outside the loop, and eight loads issued before their
          // adds: with the test inside, the loads went out one after another
          // (about 2.4 us per contributor at M = 16)
          if (row_ok) {
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              float4 o[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) o[i] = __ldcg(slot + (g8 * 8 + i) * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int c4 = (g8 * 8 + i) * 4;
                v[c4 >> 5][(c4 & 31) + 0] = __float_as_uint(__uint_as_float(v[c4 >> 5][(c4 & 31) + 0]) + o[i].x);
                v[c4 >> 5][(c4 & 31) + 1] = __float_as_uint(__uint_as_float(v[c4 >> 5][(c4 & 31) + 1]) + o[i].y);
                v[c4 >> 5][(c4 & 31) + 2] = __float_as_uint(__uint_as_float(v[c4 >> 5][(c4 & 31) + 2]) + o[i].z);
                v[c4 >> 5][(c4 & 31) + 3] = __float_as_uint(__uint_as_float(v[c4 >> 5][(c4 & 31) + 3]) + o[i].w);
              }
            }
          }
        }
        if (!got) break;
      }

      const int row0w = mt * (128 * CG) + 128 * (int)rank + 32 * q;  // this warp's first row
      const int row = row0w + lane;
      if (kAcc && !kTma && row < p.M) {
        // C_in of the direct-store path (rows not 16-byte aligned): this
        // lane's row, ncols columns (the prefetch above put them in L2)
        if constexpr (!kBF16) {
          const float *cp = reinterpret_cast<const float *>(p.C) + static_cast<int64_t>(row) * p.N + colb;
#pragma unroll
          for (int c = 0; c < 128; c += 4) {
            if (c >= ncols) break;
            if (p.vec_ok && colb + c + 4 <= p.N) {
              const float4 o = *reinterpret_cast<const float4 *>(cp + c);
              v[c >> 5][(c & 31) + 0] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + 0]) + o.x);
              v[c >> 5][(c & 31) + 1] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + 1]) + o.y);
              v[c >> 5][(c & 31) + 2] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + 2]) + o.z);
              v[c >> 5][(c & 31) + 3] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + 3]) + o.w);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (colb + c + e < p.N)
                  v[c >> 5][(c & 31) + e] =
                      __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + e]) + cp[c + e]);
            }
          }
        } else {
          const __nv_bfloat16 *cp =
              reinterpret_cast<const __nv_bfloat16 *>(p.C) + static_cast<int64_t>(row) * p.N + colb;
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            if (c >= ncols) break;
            if (p.vec_ok && colb + c + 8 <= p.N) {
              const uint4 o = *reinterpret_cast<const uint4 *>(cp + c);
              const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[c >> 5][(c & 31) + 2 * e] = __float_as_uint(
                    __uint_as_float(v[c >> 5][(c & 31) + 2 * e]) + __uint_as_float(ow[e] << 16));
                v[c >> 5][(c & 31) + 2 * e + 1] = __float_as_uint(
                    __uint_as_float(v[c >> 5][(c & 31) + 2 * e + 1]) + __uint_as_float(ow[e] & 0xFFFF0000u));
              }
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (colb + c + e < p.N)
                  v[c >> 5][(c & 31) + e] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + e]) +
                                                            __bfloat162float(cp[c + e]));
            }
          }
        }
      }

      // use_acc on the CTA's last tile: the operand ring is free (the tile's
      // MMAs have read every stage), so all of this warp's C_in chunks are
      // loaded into it by TMA at once (16 KB per warp, each chunk in the
      // swizzled layout of a store box) and waited for once, instead of one
      // load round trip per chunk at the end of the kernel; each chunk is
      // then summed in place and stored from there.
      bool cin_done = false;
      if constexpr (kAcc && kTma) {
        bool last = false;
        if (!p.use_clc) {
          WorkIter peek = wi.wi;
          WorkItem nx;
          last = !peek.next(nx);
        }
        if (last && whole) {
          constexpr int CCOLS = kBF16 ? 64 : 32;  // columns per chunk: 128 bytes
          const uint32_t region = base + ew * 16384;
          const uint32_t cbar = bar_cin + 8 * ew;
          int nchunk = 0;
          for (int cc = 0; cc < 128 / CCOLS; ++cc)
            for (int rh = 0; rh < 2; ++rh)
              if (colb + cc * CCOLS < p.N && row0w + 16 * rh < p.M) ++nchunk;
          if (lane == 0) {
            mbar_arrive_expect_tx(cbar, 2048u * nchunk);
            for (int cc = 0; cc < 128 / CCOLS; ++cc)
              for (int rh = 0; rh < 2; ++rh)
                if (colb + cc * CCOLS < p.N && row0w + 16 * rh < p.M)
                  tma_load_2d(region + (2 * cc + rh) * 2048, &tmC, colb + cc * CCOLS, row0w + 16 * rh, cbar);
          }
          __syncwarp();
          if (!__all_sync(0xFFFFFFFFu, wait_phase<false>(cbar, 0, wc, 0x0E | ((t & 0xFFFF) << 16)))) break;
          const int r16 = lane & 15;
          const uint32_t swz = r16 & 7;
#pragma unroll
          for (int cc = 0; cc < 128 / CCOLS; ++cc) {
            const int c0 = colb + cc * CCOLS;
            if (c0 >= p.N) break;
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
              const int r0 = row0w + 16 * rh;
              if (r0 >= p.M) break;
              const uint32_t chunk = region + (2 * cc + rh) * 2048;
              const uint32_t rowaddr = chunk + r16 * 128;
              if ((lane >> 4) == rh) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  const uint4 o = ld_shared_v4(rowaddr + ((u ^ swz) << 4));
                  if constexpr (!kBF16) {
                    const int c = cc * 32 + 4 * u;
                    const float s0 = __uint_as_float(v[c >> 5][(c & 31) + 0]) + __uint_as_float(o.x);
                    const float s1 = __uint_as_float(v[c >> 5][(c & 31) + 1]) + __uint_as_float(o.y);
                    const float s2 = __uint_as_float(v[c >> 5][(c & 31) + 2]) + __uint_as_float(o.z);
                    const float s3 = __uint_as_float(v[c >> 5][(c & 31) + 3]) + __uint_as_float(o.w);
                    st_shared_v4(rowaddr + ((u ^ swz) << 4), __float_as_uint(s0), __float_as_uint(s1),
                                 __float_as_uint(s2), __float_as_uint(s3));
                  } else {
                    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
                    uint32_t w2[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      const int c = cc * 64 + 8 * u + 2 * e;
                      const float lo = __uint_as_float(v[c >> 5][c & 31]) + __uint_as_float(ow[e] << 16);
                      const float hi =
                          __uint_as_float(v[c >> 5][(c & 31) + 1]) + __uint_as_float(ow[e] & 0xFFFF0000u);
                      const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                      w2[e] = *reinterpret_cast<const uint32_t *>(&b2);
                    }
                    st_shared_v4(rowaddr + ((u ^ swz) << 4), w2[0], w2[1], w2[2], w2[3]);
                  }
                }
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmC, chunk, c0, r0);
                bulk_commit_group();
              }
            }
          }
          cin_done = true;
        }
      }
      if (cin_done) {
        // (stored from the ring above)
      } else if constexpr (kTma) {
        // Chunks of 16 rows x 128 bytes through this warp's 2 KB staging
        // buffer, so that every row of a TMA store is a whole 128-byte line
        // in C (64-byte-wide chunks wrote each line in two halves, from two
        // stores): the 16 lanes holding the chunk's rows write them
        // (128-byte swizzle: 16-byte unit u of row r sits at u ^ (r & 7)),
        // then one lane issues the store, which clips rows >= M and columns
        // >= N.
        const uint32_t buf = base + C::OFF_EPI + ew * C::EPI_BUF;
        const int r16 = lane & 15;
        const uint32_t rowaddr = buf + r16 * 128;
        const uint32_t swz = r16 & 7;
        constexpr int CCOLS = kBF16 ? 64 : 32;  // columns per chunk: 128 bytes
#pragma unroll
        for (int cc = 0; cc < 128 / CCOLS; ++cc) {
          if (cc * CCOLS >= ncols) break;
          const int c0 = colb + cc * CCOLS;
          if (c0 >= p.N) break;
#pragma unroll
          for (int rh = 0; rh < 2; ++rh) {
            const int r0 = row0w + 16 * rh;
            if (r0 >= p.M) break;
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            if constexpr (kAcc) {
              // C_in of the chunk, 16 rows x 128 bytes, with coalesced
              // 16-byte loads (8 lanes per row, 4 rows per instruction) into
              // the staging buffer in its swizzled order; the lanes holding
              // the rows then add it to their accumulator values below.
              // (Loads of one row per lane, 32 rows per instruction, took
              // 8x the L1 wavefronts and slowed the concurrent main loop.)
              const int u = lane & 7;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int rr = (lane >> 3) + 4 * j;  // row within the chunk
                uint4 x = make_uint4(0u, 0u, 0u, 0u);
                // C's rows are 16-byte multiples here, so a unit is wholly
                // inside or wholly past column N
                if (r0 + rr < p.M && (c0 + u * CCOLS / 8) < p.N)
                  x = __ldcg(reinterpret_cast<const uint4 *>(
                      reinterpret_cast<const uint8_t *>(p.C) +
                      (static_cast<int64_t>(r0 + rr) * p.N + c0) * (kBF16 ? 2 : 4) + 16 * u));
                st_shared_v4(buf + rr * 128 + ((u ^ (rr & 7)) << 4), x.x, x.y, x.z, x.w);
              }
              __syncwarp();
            }
            if ((lane >> 4) == rh) {
              if constexpr (!kBF16) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  const int c = cc * 32 + 4 * u;
                  if constexpr (kAcc) {
                    const uint4 o = ld_shared_v4(rowaddr + ((u ^ swz) << 4));
                    v[c >> 5][(c & 31) + 0] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + 0]) + __uint_as_float(o.x));
                    v[c >> 5][(c & 31) + 1] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + 1]) + __uint_as_float(o.y));
                    v[c >> 5][(c & 31) + 2] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + 2]) + __uint_as_float(o.z));
                    v[c >> 5][(c & 31) + 3] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + 3]) + __uint_as_float(o.w));
                  }
                  st_shared_v4(rowaddr + ((u ^ swz) << 4), v[c >> 5][c & 31], v[c >> 5][(c & 31) + 1],
                               v[c >> 5][(c & 31) + 2], v[c >> 5][(c & 31) + 3]);
                }
              } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  uint32_t w[4];
                  if constexpr (kAcc) {
                    const uint4 o = ld_shared_v4(rowaddr + ((u ^ swz) << 4));
                    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      const int c = cc * 64 + 8 * u + 2 * e;
                      v[c >> 5][c & 31] =
                          __float_as_uint(__uint_as_float(v[c >> 5][c & 31]) + __uint_as_float(ow[e] << 16));
                      v[c >> 5][(c & 31) + 1] = __float_as_uint(__uint_as_float(v[c >> 5][(c & 31) + 1]) +
                                                                __uint_as_float(ow[e] & 0xFFFF0000u));
                    }
                  }
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int c = cc * 64 + 8 * u + 2 * e;
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[c >> 5][c & 31]),
                                                                    __uint_as_float(v[c >> 5][(c & 31) + 1]));
                    w[e] = *reinterpret_cast<const uint32_t *>(&b2);
                  }
                  st_shared_v4(rowaddr + ((u ^ swz) << 4), w[0], w[1], w[2], w[3]);
                }
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, buf, c0, r0);
              bulk_commit_group();
            }
          }
        }
      } else if (row < p.M) {
        // C rows not 16-byte aligned: direct stores
        if constexpr (!kBF16) {
          float *cp = reinterpret_cast<float *>(p.C) + static_cast<int64_t>(row) * p.N + colb;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c < ncols && colb + c < p.N) cp[c] = __uint_as_float(v[c >> 5][c & 31]);
        } else {
          __nv_bfloat16 *cp =
              reinterpret_cast<__nv_bfloat16 *>(p.C) + static_cast<int64_t>(row) * p.N + colb;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c < ncols && colb + c < p.N) cp[c] = __float2bfloat16_rn(__uint_as_float(v[c >> 5][c & 31]));
        }
      }
    }
    // every store of this warp has completed before the CTA may finish
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  if constexpr (CG == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<CG>(tmem, C::TM_COLS);
}

}  // namespace mxg
