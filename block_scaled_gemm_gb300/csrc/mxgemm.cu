// mxgemm.cu -- host side of the C interface declared in include/mxgemm.h:
// argument validation, tile-mode planning, workspace, tensor-map encoding and
// the launches (scale repack, optional B row padding, the GEMM kernel).
//
// The operation is the scaled product `async_dot_scaled` of the "TLX API
// Quick Reference" (section "Matrix Multiply (MMA)"); the pair mode is the
// "2-CTA Scaled MMA" of "Tensor core operations".
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>

#include "mxgemm.h"
#include "mxgemm_kernel.cuh"
#include "prepass.cuh"
#include "quantize.cuh"
#include "swapab.h"
#include "swapab_kernel.cuh"
#include "tiled_launch.cuh"

namespace {

using mxg::Cfg;
using mxg::KParams;

struct Workspace {
  uint8_t *ptr = nullptr;
  size_t bytes = 0;
};

// Everything a run needs besides its launches, keyed by the run's arguments.
// Repeated calls on the same buffers (a serving or training loop) skip the
// pointer checks and tensor-map encoding.
struct Plan {
  bool valid = false;
  // key
  int64_t M = 0, N = 0, K = 0;
  const void *A = nullptr, *As = nullptr, *B = nullptr, *Bs = nullptr;
  void *C = nullptr;
  int use_acc = 0, out_dtype = 0, mode = 0, stall = 0, sched = 0, sk = 0, fmts = 0, layout = 0;
  long long timeout_ns = 0;
  uint8_t *ws = nullptr;
  // value
  int CG = 1;
  bool pad_b = false;
  bool pack_bk = false;  // B given N x K with a sub-byte format: packed into the workspace
  int64_t npad = 0;
  int a_bits = 8, b_bits = 8;  // element bits; below 8 the operand is packed first
  size_t off_a = 0;
  CUtensorMap tA, tB, tB64, tSA, tSB, tC;
  KParams kp;
  mxg::RepackArgs ra, rb;
  int blocks_a = 0, blocks_b = 0;
  int units = 0;     // persistent CTAs (pairs) of the GEMM grid
  bool repack = false;  // pairs: the scale chunks come from the repack prepass
  bool repack_lite = false;  // ... by repack_scales_lite_kernel
  // skinny problems (M <= 128) computed transposed by mxgemm_swapab_kernel
  bool swap = false;
  CUtensorMap tAt, tSBs, tSAs;  // A rows (MMA B operand), scale staging maps
  mxg::SwapParams swp;
  int swap_grid = 0;

  bool matches(int64_t M_, int64_t N_, int64_t K_, const void *A_, const void *As_, const void *B_,
               const void *Bs_, void *C_, int ua, int od, int md, int sl, int sc, int sk_,
               long long to, uint8_t *w, int fm, int lay) const {
    return valid && M == M_ && N == N_ && K == K_ && A == A_ && As == As_ && B == B_ &&
           Bs == Bs_ && C == C_ && use_acc == ua && out_dtype == od && mode == md &&
           stall == sl && sched == sc && sk == sk_ && timeout_ns == to && ws == w && fmts == fm &&
           layout == lay;
  }
};

constexpr int kPlanCache = 8;

// Copy streams, events and device staging of mxgemm_run_host.
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr;      // the caller's stream reached the call
  cudaEvent_t b_ready = nullptr;    // B and its scales are on the device
  static constexpr int kSlots = 3;   // device slots for the row slabs
  cudaEvent_t in_ready[kSlots] = {};   // slot s holds its slab's inputs
  cudaEvent_t gemm_done[kSlots] = {};  // slot s's GEMM has finished
  cudaEvent_t out_done[kSlots] = {};   // slot s's C rows are back on the host
  cudaEvent_t b_used[2] = {};       // the last GEMM reading B slot b has finished
  int bslot = 0;                    // B slot of the next call
  Workspace stage;
};

}  // namespace

struct mxgemm_ctx {
  int device = 0;
  int sm_count = 0;
  int *d_status = nullptr;  // [0] status code, [1] detail
  // partial-sum flags: one slot per (CTA, epilogue warp), zeroed once at
  // creation; each launch writes and waits for its own epoch (never 0)
  unsigned *flags = nullptr;
  unsigned epoch = 0;
  Workspace ws;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  long long timeout_ns = 2000000000LL;
  int mode = 0;
  int stall_producer = 0;
  int scheduler = 0;
  int stream_k = 1;
  int a_fmt = 0, b_fmt = 0;  // element formats (mxgemm_format_t)
  int scale_layout = MXGEMM_SCALES_ROW_MAJOR;
  int elem_layout = MXGEMM_ELEMS_BYTE;
  int b_major = MXGEMM_B_K_BY_N;
  bool attr_set[3][16] = {};
  bool swap_attr[4][4] = {};
  cudaEvent_t prof_before = nullptr;
  cudaEvent_t prof_after = nullptr;
  int64_t launches = 0;
  Plan plans[kPlanCache];
  int next_plan = 0;
  HostPipe hp;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      changed = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

bool on_device(const void *p, int device) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged) &&
         attr.device == device;
}

// 2-D tensor map: dims {inner, outer} in elements, row pitch in bytes, box.
int encode_2d(mxgemm_ctx *h, CUtensorMap *tm, CUtensorMapDataType dt, const void *base,
              uint64_t inner, uint64_t outer, uint64_t pitch, uint32_t box_inner,
              uint32_t box_outer, CUtensorMapSwizzle swz) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = h->encode(tm, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MXGEMM_OK : MXGEMM_ERR_CUDA;
}

int ensure_workspace(mxgemm_ctx *h, size_t bytes, cudaStream_t stream) {
  if (h->ws.bytes >= bytes) return MXGEMM_OK;
  if (h->ws.ptr) {
    // stream-ordered: earlier work on this stream still using it finishes first
    cudaFreeAsync(h->ws.ptr, stream);
    h->ws.ptr = nullptr;
    h->ws.bytes = 0;
  }
  void *p = nullptr;
  size_t want = round_up(bytes, size_t(2) << 20);
  if (cudaMallocAsync(&p, want, stream) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_OUT_OF_MEMORY;
  }
  h->ws.ptr = static_cast<uint8_t *>(p);
  h->ws.bytes = want;
  for (Plan &pl : h->plans) pl.valid = false;
  return MXGEMM_OK;
}

// The tiled kernel for this run: its epilogue variant, and its B layout.
template <int CG>
int launch_gemm(mxgemm_ctx *h, const CUtensorMap &tA, const CUtensorMap &tB,
                const CUtensorMap &tB64, const CUtensorMap &tSA, const CUtensorMap &tSB, const CUtensorMap &tC,
                const KParams &kp, int units, cudaStream_t stream) {
  mxg::TiledLaunch L{h->attr_set[CG], h->prof_before, h->prof_after, &h->launches};
  const mxg::TiledMaps m{&tA, &tB, &tB64, &tSA, &tSB, &tC};
  if (kp.b_kmajor) return mxg::launch_tiled_kmajor(CG, L, m, kp, units, stream);
  return mxg::launch_tiled_epi<CG, 0>(L, m, kp, units, stream);
}

int launch_blocks(int64_t work, int per_block) {
  int64_t b = cdiv(work, per_block);
  if (b < 1) b = 1;
  if (b > 4096) b = 4096;
  return static_cast<int>(b);
}

// How the GEMM grid covers the tiles: whole tiles in full waves, and for
// the tiles that do not fill the last wave either a stream-K tail (their K
// steps split evenly over the CTAs) or half-width tiles (each leftover tile
// computed as two 128-column halves).
struct Split {
  int units;           // persistent CTAs (pairs)
  int dp_tiles;        // tiles computed whole
  int sk_ctas;         // CTAs sharing the tail
  long long sk_units;  // K steps in the tail
  int half_tiles;      // half-width items after the whole tiles (2 per leftover tile)
};

Split plan_split(int64_t T, int64_t S, int P, bool allow_tail, bool allow_stream_k, int64_t M) {
  Split r;
  r.units = static_cast<int>(T < P ? T : P);
  r.dp_tiles = static_cast<int>(T);
  r.sk_ctas = 0;
  r.sk_units = 0;
  r.half_tiles = 0;
  if (!allow_tail || T == 0) return r;
  const int64_t W = T / P, R = T % P;
  if (R == 0) return r;
  // Skinny problems (M <= 128: one row of tiles) with fewer tiles than
  // CTAs: split every tile's K steps into s equal parts, s the largest
  // divisor of S with T * s <= P and at least 4 K steps per part, so that
  // every CTA computes one part of one tile (no CTA straddles two tiles and
  // finishes late).  The partial sums hold only the valid rows, so their
  // traffic stays small next to B's, and most SMs stream B instead of one
  // per tile.  Not below 16 rows: at M = 1 the split measured slower than
  // whole tiles (34.8 -> 41.0 us at N = K = 8192; its owners finished
  // 4-18 us after the median CTA), at M = 16..128 faster (35.9 -> 30.8 us
  // at M = 16).
  if (allow_stream_k && W == 0 && M >= 16 && M <= 128 && S >= 8) {
    int64_t parts = 1;
    for (int64_t d = 2; d <= S / 4; ++d)
      if (S % d == 0 && T * d <= P) parts = d;
    if (parts > 1) {
      r.units = static_cast<int>(T * parts);
      r.dp_tiles = 0;
      r.sk_ctas = static_cast<int>(T * parts);
      r.sk_units = T * S;
      return r;
    }
  }
  // Measured on GB300: the owners' gather of FP32 partials is slow enough
  // that stream-K pays off only with long K (64+ steps) after 1 to 8 full
  // waves, and not when the last wave is nearly full; in particular not when
  // every tile would be split (fewer tiles than CTAs).
  if (allow_stream_k && S >= 64 && W >= 1 && W <= 8 && R * 100 < static_cast<int64_t>(P) * 85) {
    const int64_t tail = R * S;
    int64_t ctas = tail / 4;  // at least 4 K steps per CTA
    if (ctas > P) ctas = P;
    if (ctas > R) {  // else no CTA would get less than a whole tile
      r.units = P;
      r.dp_tiles = static_cast<int>(W * P);
      r.sk_ctas = static_cast<int>(ctas);
      r.sk_units = tail;
      return r;
    }
  }
  // Otherwise, when the leftover tiles fill at most half a wave, halve
  // their width: twice as many CTAs (pairs) finish them in half the time.
  if (2 * R <= P) {
    r.dp_tiles = static_cast<int>(W * P);
    r.half_tiles = static_cast<int>(2 * R);
    r.units = static_cast<int>(W >= 1 ? P : 2 * R);
  }
  return r;
}

// Workspace layout of a run: repacked scales (pairs), re-pitched (or
// packed) B, stream-K partials, packed A (6- and 4-bit A formats).
struct Sizes {
  size_t off_sfb, off_b, off_part, off_a, total;
};

Sizes plan_sizes(int64_t a_chunks, int64_t b_chunks, size_t b_ws_bytes,
                 const Split &sp, int CG, size_t a_bytes) {
  Sizes z;
  z.off_sfb = round_up(static_cast<size_t>(a_chunks) * 512, 1024);
  z.off_b = round_up(z.off_sfb + static_cast<size_t>(b_chunks) * 512, 1024);
  z.off_part = round_up(z.off_b + b_ws_bytes, 1024);
  z.off_a = round_up(z.off_part + static_cast<size_t>(sp.sk_ctas) * CG * 128 * 256 * sizeof(float),
                     1024);
  z.total = round_up(z.off_a + a_bytes, 1024);
  return z;
}

// Validate-once work of a run: prepass arguments, tensor maps and kernel
// parameters, stored in `pl` under the run's key.
int build_plan(mxgemm_ctx *h, Plan *pl, int64_t M, int64_t N, int64_t K, const void *A,
               const void *A_scale, const void *B, const void *B_scale, void *C, int use_acc,
               int out_dtype, int CG, int64_t m_tiles, int64_t n_tiles, int64_t k_steps,
               int64_t num_tiles, int64_t a_chunks, int64_t b_chunks, bool pad_b, int64_t npad,
               const Split &sp, const Sizes &z, int a_bits, int b_bits, bool fused, bool packed) {
  const size_t off_sfb = z.off_sfb, off_b = z.off_b;
  const size_t esz = out_dtype == MXGEMM_OUT_F32 ? 4 : 2;
  const int64_t kb = K / 32;
  // scale chunks: repacked into the workspace, or the caller's packed scales
  const uint8_t *sfa = packed ? static_cast<const uint8_t *>(A_scale) : h->ws.ptr;
  const uint8_t *sfb = packed ? static_cast<const uint8_t *>(B_scale) : h->ws.ptr + off_sfb;
  if (packed) {
    a_chunks = cdiv(M, 128) * k_steps;  // the packed area (a pair's second block may lie past it)
    b_chunks = n_tiles * k_steps * 2;
  }
  const bool b_km = h->b_major == MXGEMM_B_N_BY_K;
  const bool pack_bk = b_km && b_bits < 8;
  const void *bsrc = pad_b || pack_bk ? static_cast<const void *>(h->ws.ptr + off_b) : B;
  const int64_t bpitch = pad_b ? npad : N;
  const void *asrc = a_bits < 8 ? static_cast<const void *>(h->ws.ptr + z.off_a) : A;
  pl->ra = mxg::RepackArgs{static_cast<const uint8_t *>(A_scale), reinterpret_cast<uint32_t *>(h->ws.ptr),
                           M, static_cast<int>(kb), static_cast<int>(k_steps), 1,
                           static_cast<int>(m_tiles * CG), static_cast<int>(cdiv(k_steps, 16))};
  pl->rb = mxg::RepackArgs{static_cast<const uint8_t *>(B_scale),
                           reinterpret_cast<uint32_t *>(h->ws.ptr + off_sfb),
                           N, static_cast<int>(kb), static_cast<int>(k_steps), 2,
                           static_cast<int>(n_tiles * 2), static_cast<int>(cdiv(k_steps, 16))};
  pl->blocks_a = pl->ra.row_blocks * pl->ra.kgroups;
  pl->blocks_b = pl->rb.row_blocks * pl->rb.kgroups;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (encode_2d(h, &pl->tA, u8, asrc, K, M, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      (b_km ? encode_2d(h, &pl->tB, u8, bsrc, K, N, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B)
            : encode_2d(h, &pl->tB, u8, bsrc, N, K, bpitch, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B)) ||
      // half-width tiles of CTA pairs: 64 columns (rows of an N x K B) per CTA
      (b_km ? encode_2d(h, &pl->tB64, u8, bsrc, K, N, K, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B)
            : encode_2d(h, &pl->tB64, u8, bsrc, N, K, bpitch, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B)))
    return MXGEMM_ERR_CUDA;
  // Repacked scale chunks are contiguous 512-byte blocks, fetched as rows of
  // 128 bytes (4 rows per chunk) so each chunk is a handful of TMA requests.
  // With fused scales (single CTAs) the kernel builds the chunks; the scale
  // maps then describe the row-major scales themselves (16-byte segments of
  // 128 A rows or 256 B rows), usable when the row pitch K/32 and both bases
  // are multiples of 16 bytes.
  std::memset(&pl->tSA, 0, sizeof(pl->tSA));
  std::memset(&pl->tSB, 0, sizeof(pl->tSB));
  pl->repack = !fused && !packed;
  const bool scale_tma = fused && kb % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(A_scale) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(B_scale) % 16 == 0;
  if (!fused &&
      (encode_2d(h, &pl->tSA, u8, sfa, 128, a_chunks * 4, 128, 128, 4, CU_TENSOR_MAP_SWIZZLE_NONE) ||
       encode_2d(h, &pl->tSB, u8, sfb, 128, b_chunks * 4, 128, 128, 8, CU_TENSOR_MAP_SWIZZLE_NONE)))
    return MXGEMM_ERR_CUDA;
  if (scale_tma &&
      (encode_2d(h, &pl->tSA, u8, A_scale, kb, M, kb, 16, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
       encode_2d(h, &pl->tSB, u8, B_scale, kb, N, kb, 16, 256, CU_TENSOR_MAP_SWIZZLE_NONE)))
    return MXGEMM_ERR_CUDA;
  // C: stored through TMA (128-byte-wide boxes, 16 rows) when its row pitch
  // allows it; otherwise the kernel stores directly and tC is unused.
  const bool tma_store = (static_cast<size_t>(N) * esz) % 16 == 0;
  std::memset(&pl->tC, 0, sizeof(pl->tC));
  if (tma_store &&
      encode_2d(h, &pl->tC,
                out_dtype == MXGEMM_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                C, N, M, static_cast<uint64_t>(N) * esz, static_cast<uint32_t>(128 / esz), 16,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return MXGEMM_ERR_CUDA;
  KParams &kp = pl->kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.M = static_cast<int>(M);
  kp.N = static_cast<int>(N);
  kp.K = static_cast<int>(K);
  kp.m_tiles = static_cast<int>(m_tiles);
  kp.n_tiles = static_cast<int>(n_tiles);
  kp.k_steps = static_cast<int>(k_steps);
  kp.num_tiles = static_cast<int>(num_tiles);
  kp.C = C;
  kp.out_bf16 = out_dtype == MXGEMM_OUT_BF16;
  kp.use_acc = use_acc;
  kp.vec_ok = (N % (out_dtype == MXGEMM_OUT_F32 ? 4 : 8)) == 0;
  kp.tma_store = tma_store;
  kp.status = h->d_status;
  kp.timeout_ns = static_cast<unsigned long long>(h->timeout_ns);
  kp.stall_producer = h->stall_producer;
  kp.use_clc = h->scheduler;
  kp.dp_tiles = sp.dp_tiles;
  kp.sk_ctas = sp.sk_ctas;
  kp.sk_units = sp.sk_units;
  kp.partials = reinterpret_cast<float *>(h->ws.ptr + z.off_part);
  kp.flags = h->flags;
  kp.epoch = 0;  // set per launch
  kp.half_tiles = sp.half_tiles;
  kp.idesc_fmt = mxg::fmt_bits(h->a_fmt, h->b_fmt);
  kp.a_scale = static_cast<const uint8_t *>(A_scale);
  kp.b_scale = static_cast<const uint8_t *>(B_scale);
  kp.kb_count = static_cast<int>(kb);
  kp.fused_scales = fused ? 1 : 0;
  kp.scale_tma = scale_tma ? 1 : 0;
  // The light repack (beside the GEMM's CTAs) needs 16-byte scale rows;
  // its GEMM then sends its first A and B loads before waiting for it.
  pl->repack_lite = pl->repack && kb % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(A_scale) % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(B_scale) % 16 == 0;
  kp.early_ab = pl->repack_lite ? 1 : 0;
  kp.b_kmajor = b_km ? 1 : 0;
  pl->units = sp.units;
  pl->CG = CG;
  pl->pad_b = pad_b;
  pl->pack_bk = pack_bk;
  pl->npad = npad;
  pl->a_bits = a_bits;
  pl->b_bits = b_bits;
  pl->off_a = z.off_a;
  pl->M = M; pl->N = N; pl->K = K;
  pl->A = A; pl->As = A_scale; pl->B = B; pl->Bs = B_scale; pl->C = C;
  pl->use_acc = use_acc; pl->out_dtype = out_dtype; pl->mode = h->mode;
  pl->stall = h->stall_producer; pl->sched = h->scheduler; pl->sk = h->stream_k;
  pl->timeout_ns = h->timeout_ns;
  pl->fmts = h->a_fmt * 8 + h->b_fmt + 64 * h->elem_layout + 128 * h->b_major;
  pl->layout = packed ? MXGEMM_SCALES_PACKED : MXGEMM_SCALES_ROW_MAJOR;
  pl->ws = h->ws.ptr;
  pl->valid = true;
  return MXGEMM_OK;
}

// Skinny problems (M <= 128, 8-bit element formats): C^T = B^T x A^T on
// mxgemm_swapab_kernel, one CTA per (128-column block of N, K split), the
// K splits of a block reduced inside their cluster.  The only workspace is a
// re-pitched B when N % 16 != 0.
int run_swapab(mxgemm_ctx *h, int64_t M, int64_t N, int64_t K, const void *A, const void *A_scale,
               const void *B, const void *B_scale, void *C, int use_acc, int out_dtype,
               bool packed, cudaStream_t stream) {
  const int64_t k_steps = cdiv(K, 128);
  const int64_t nblk = cdiv(N, 128);
  const bool b_km = h->b_major == MXGEMM_B_N_BY_K;
  const bool pad_b = !b_km && (N % 16) != 0;
  const int64_t npad = round_up(static_cast<size_t>(N), 16);
  const size_t ws_bytes = pad_b ? round_up(static_cast<size_t>(K) * npad, 1024) : 0;

  Plan *plan = nullptr;
  for (Plan &pl : h->plans)
    if (pl.matches(M, N, K, A, A_scale, B, B_scale, C, use_acc, out_dtype, h->mode,
                   h->stall_producer, h->scheduler, h->stream_k, h->timeout_ns, h->ws.ptr,
                   h->a_fmt * 8 + h->b_fmt + 64 * h->elem_layout + 128 * h->b_major, h->scale_layout) &&
        pl.swap && h->ws.bytes >= ws_bytes) {
      plan = &pl;
      break;
    }
  if (!plan) {
    if (!on_device(C, h->device) || !on_device(A, h->device) || !on_device(B, h->device) ||
        !on_device(A_scale, h->device) || !on_device(B_scale, h->device))
      return MXGEMM_ERR_INVALID_VALUE;
    int st = ensure_workspace(h, ws_bytes, stream);
    if (st != MXGEMM_OK) return st;
    plan = &h->plans[h->next_plan];
    h->next_plan = (h->next_plan + 1) % kPlanCache;
    Plan &pl = *plan;
    pl.valid = false;
    const int nt = mxg::swapab_class(static_cast<int>(M));
    const int nm = static_cast<int>(round_up(static_cast<size_t>(M), 16));
    // K splits: enough CTAs per column block to cover the SMs when the
    // blocks alone do not, within one cluster (at most 8, and what the
    // first CTA's shared memory can receive), at least 4 K steps each
    int64_t splits = 1;
    if (nblk < h->sm_count) {
      splits = h->sm_count / nblk;
      splits = std::min<int64_t>(splits, mxg::swapab_max_splits(nt));
      splits = std::min<int64_t>(splits, std::max<int64_t>(1, k_steps / 4));
      splits = std::max<int64_t>(splits, 1);
    }
    const int64_t kb = K / 32;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const void *bsrc = pad_b ? static_cast<const void *>(h->ws.ptr) : B;
    const int64_t bpitch = pad_b ? npad : N;
    const bool scale_tma = !packed && kb % 16 == 0 &&
                           reinterpret_cast<uintptr_t>(A_scale) % 16 == 0 &&
                           reinterpret_cast<uintptr_t>(B_scale) % 16 == 0;
    std::memset(&pl.tSBs, 0, sizeof(pl.tSBs));
    std::memset(&pl.tSAs, 0, sizeof(pl.tSAs));
    // B: 128 columns x 128 K rows per box (the MMA's A operand, M-major);
    // A: 128 K bytes x nm rows (the MMA's B operand, K-major), rows past M
    // filled with zero
    if ((b_km ? encode_2d(h, &pl.tB, u8, B, K, N, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B)
              : encode_2d(h, &pl.tB, u8, bsrc, N, K, bpitch, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B)) ||
        encode_2d(h, &pl.tAt, u8, A, K, M, K, 128, static_cast<uint32_t>(nm),
                  CU_TENSOR_MAP_SWIZZLE_128B))
      return MXGEMM_ERR_CUDA;
    // 16-byte row segments (four K steps) of the block's 128 B_scale rows and
    // of the nm A_scale rows
    if (scale_tma &&
        (encode_2d(h, &pl.tSBs, u8, B_scale, kb, N, kb, 16, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
         encode_2d(h, &pl.tSAs, u8, A_scale, kb, M, kb, 16, static_cast<uint32_t>(nm),
                   CU_TENSOR_MAP_SWIZZLE_NONE)))
      return MXGEMM_ERR_CUDA;
    mxg::SwapParams &p = pl.swp;
    std::memset(&p, 0, sizeof(p));
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.nm = nm;
    p.k_steps = static_cast<int>(k_steps);
    p.splits = static_cast<int>(splits);
    p.C = C;
    p.use_acc = use_acc;
    p.status = h->d_status;
    p.timeout_ns = static_cast<unsigned long long>(h->timeout_ns);
    p.stall_producer = h->stall_producer;
    // the MMA's A operand is B and its B operand is A: their formats swap
    p.idesc_fmt = (mxg::mma_format_code(h->b_fmt) << 7) | (mxg::mma_format_code(h->a_fmt) << 10);
    p.a_scale = static_cast<const uint8_t *>(A_scale);
    p.b_scale = static_cast<const uint8_t *>(B_scale);
    p.kb_count = static_cast<int>(kb);
    p.scale_tma = scale_tma ? 1 : 0;
    p.packed = packed ? 1 : 0;
    p.b_kmajor = b_km ? 1 : 0;
    p.a_chunks = static_cast<const uint8_t *>(A_scale);
    p.b_chunks = static_cast<const uint8_t *>(B_scale);
    pl.swap = true;
    pl.swap_grid = static_cast<int>(nblk * splits);
    pl.CG = 1;
    pl.pad_b = pad_b;
    pl.pack_bk = false;
    pl.npad = npad;
    pl.a_bits = 8;
    pl.b_bits = 8;
    pl.repack = false;
    pl.M = M; pl.N = N; pl.K = K;
    pl.A = A; pl.As = A_scale; pl.B = B; pl.Bs = B_scale; pl.C = C;
    pl.use_acc = use_acc; pl.out_dtype = out_dtype; pl.mode = h->mode;
    pl.stall = h->stall_producer; pl.sched = h->scheduler; pl.sk = h->stream_k;
    pl.timeout_ns = h->timeout_ns;
    pl.fmts = h->a_fmt * 8 + h->b_fmt + 64 * h->elem_layout + 128 * h->b_major;
    pl.layout = packed ? MXGEMM_SCALES_PACKED : MXGEMM_SCALES_ROW_MAJOR;
    pl.ws = h->ws.ptr;
    pl.valid = true;
  }
  if (plan->pad_b) {
    mxg::pad_rows_kernel<<<launch_blocks(K * (plan->npad / 16), 256), 256, 0, stream>>>(
        static_cast<const uint8_t *>(B), K, N, plan->npad, h->ws.ptr, 8);
    ++h->launches;
    if (cudaGetLastError() != cudaSuccess) return MXGEMM_ERR_CUDA;
  }
  if (h->prof_before && cudaEventRecord(h->prof_before, stream) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  const int st = mxg::swapab_launch(plan->tB, plan->tAt, plan->tSBs, plan->tSAs, plan->swp,
                                    out_dtype == MXGEMM_OUT_BF16, plan->swap_grid, stream,
                                    h->swap_attr);
  if (st != MXGEMM_OK) return st;
  ++h->launches;
  if (h->prof_after && cudaEventRecord(h->prof_after, stream) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  return MXGEMM_OK;
}

}  // namespace

extern "C" {

const char *mxgemm_status_string(int s) {
  switch (s) {
    case MXGEMM_OK: return "ok";
    case MXGEMM_ERR_INVALID_VALUE: return "invalid value";
    case MXGEMM_ERR_MISALIGNED: return "misaligned pointer (A, B and C need 16-byte alignment)";
    case MXGEMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case MXGEMM_ERR_OUT_OF_MEMORY: return "out of device memory";
    case MXGEMM_ERR_CUDA: return "CUDA call failed";
    case MXGEMM_ERR_TIMEOUT: return "device-side wait timed out";
    case MXGEMM_ERR_TOO_LARGE:
      return "problem needs more scratch than the fixed no-allocation buffer holds";
    default: return "unknown status";
  }
}

int mxgemm_create(mxgemm_handle_t *out, int device) {
  if (!out) return MXGEMM_ERR_INVALID_VALUE;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  if (device < 0 || device >= ndev) return MXGEMM_ERR_INVALID_VALUE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MXGEMM_ERR_CUDA;
  if (!(prop.major == 10 && prop.minor == 3)) return MXGEMM_ERR_UNSUPPORTED_DEVICE;

  DeviceGuard g(device);
  mxgemm_ctx *h = new (std::nothrow) mxgemm_ctx();
  if (!h) return MXGEMM_ERR_OUT_OF_MEMORY;
  h->device = device;
  h->sm_count = prop.multiProcessorCount;
  if (const char *t = std::getenv("MXGEMM_WAIT_TIMEOUT_NS")) {
    long long v = std::atoll(t);
    if (v > 0) h->timeout_ns = v;
  }
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    delete h;
    return MXGEMM_ERR_CUDA;
  }
  h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  if (cudaMalloc(&h->d_status, 2 * sizeof(int)) != cudaSuccess) {
    delete h;
    return MXGEMM_ERR_OUT_OF_MEMORY;
  }
  if (cudaMemset(h->d_status, 0, 2 * sizeof(int)) != cudaSuccess) {
    cudaFree(h->d_status);
    delete h;
    return MXGEMM_ERR_CUDA;
  }
  // a flag slot per epilogue warp of every CTA a grid can have
  const size_t flag_bytes = static_cast<size_t>(h->sm_count) * mxg::Cfg<1>::EPI_WARPS * sizeof(unsigned);
  if (cudaMalloc(&h->flags, flag_bytes) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->d_status);
    delete h;
    return MXGEMM_ERR_OUT_OF_MEMORY;
  }
  if (cudaMemset(h->flags, 0, flag_bytes) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->flags);
    cudaFree(h->d_status);
    delete h;
    return MXGEMM_ERR_CUDA;
  }
  *out = h;
  return MXGEMM_OK;
}

int mxgemm_set_option(mxgemm_handle_t h, int option, int64_t value) {
  if (!h) return MXGEMM_ERR_INVALID_VALUE;
  switch (option) {
    case MXGEMM_OPT_MODE:
      if (value < 0 || value > 3) return MXGEMM_ERR_INVALID_VALUE;
      h->mode = static_cast<int>(value);
      return MXGEMM_OK;
    case MXGEMM_OPT_WAIT_TIMEOUT_NS:
      if (value <= 0) return MXGEMM_ERR_INVALID_VALUE;
      h->timeout_ns = value;
      return MXGEMM_OK;
    case MXGEMM_OPT_TEST_STALL_PRODUCER:
      if (value < 0 || value > 1) return MXGEMM_ERR_INVALID_VALUE;
      h->stall_producer = static_cast<int>(value);
      return MXGEMM_OK;
    case MXGEMM_OPT_SCHEDULER:
      if (value < 0 || value > 1) return MXGEMM_ERR_INVALID_VALUE;
      h->scheduler = static_cast<int>(value);
      return MXGEMM_OK;
    case MXGEMM_OPT_STREAM_K:
      if (value < 0 || value > 1) return MXGEMM_ERR_INVALID_VALUE;
      h->stream_k = static_cast<int>(value);
      return MXGEMM_OK;
    case MXGEMM_OPT_A_FORMAT:
    case MXGEMM_OPT_B_FORMAT:
      if (value < MXGEMM_FMT_E4M3 || value > MXGEMM_FMT_E2M1) return MXGEMM_ERR_INVALID_VALUE;
      (option == MXGEMM_OPT_A_FORMAT ? h->a_fmt : h->b_fmt) = static_cast<int>(value);
      return MXGEMM_OK;
    case MXGEMM_OPT_SCALE_LAYOUT:
      if (value != MXGEMM_SCALES_ROW_MAJOR && value != MXGEMM_SCALES_PACKED)
        return MXGEMM_ERR_INVALID_VALUE;
      h->scale_layout = static_cast<int>(value);
      return MXGEMM_OK;
    case MXGEMM_OPT_ELEMENT_LAYOUT:
      if (value != MXGEMM_ELEMS_BYTE && value != MXGEMM_ELEMS_PACKED) return MXGEMM_ERR_INVALID_VALUE;
      h->elem_layout = static_cast<int>(value);
      return MXGEMM_OK;
    case MXGEMM_OPT_B_MAJOR:
      if (value != MXGEMM_B_K_BY_N && value != MXGEMM_B_N_BY_K) return MXGEMM_ERR_INVALID_VALUE;
      h->b_major = static_cast<int>(value);
      return MXGEMM_OK;
    default:
      return MXGEMM_ERR_INVALID_VALUE;
  }
}

int mxgemm_run(mxgemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A,
               const void *A_scale, const void *B, const void *B_scale, void *C, int use_acc,
               int out_dtype, mxgemm_stream_t stream_) {
  if (!h) return MXGEMM_ERR_INVALID_VALUE;
  const int64_t lim = int64_t(1) << 31;
  if (M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim) return MXGEMM_ERR_INVALID_VALUE;
  if (K % 32 != 0) return MXGEMM_ERR_INVALID_VALUE;
  if (out_dtype != MXGEMM_OUT_F32 && out_dtype != MXGEMM_OUT_BF16) return MXGEMM_ERR_INVALID_VALUE;
  if (use_acc != 0 && use_acc != 1) return MXGEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return MXGEMM_OK;
  const size_t esz = out_dtype == MXGEMM_OUT_F32 ? 4 : 2;
  if (!C) return MXGEMM_ERR_INVALID_VALUE;
  if (reinterpret_cast<uintptr_t>(C) % 16) return MXGEMM_ERR_MISALIGNED;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  DeviceGuard g(h->device);
  if (K == 0) {
    if (!on_device(C, h->device)) return MXGEMM_ERR_INVALID_VALUE;
    if (use_acc) return MXGEMM_OK;
    if (cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * esz, stream) != cudaSuccess) {
      cudaGetLastError();
      return MXGEMM_ERR_CUDA;
    }
    return MXGEMM_OK;
  }
  if (!A || !B || !A_scale || !B_scale) return MXGEMM_ERR_INVALID_VALUE;
  if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16)
    return MXGEMM_ERR_MISALIGNED;

  // Skinny problems: the transposed kernel, automatically for M <= 128 with
  // 8-bit element formats, or on request (MXGEMM_OPT_MODE = 3)
  {
    const bool sub_byte = h->a_fmt >= MXGEMM_FMT_E2M3 || h->b_fmt >= MXGEMM_FMT_E2M3;
    const bool swap_ok = M <= 128 && !sub_byte;
    if (h->mode == 3 && !swap_ok) return MXGEMM_ERR_INVALID_VALUE;
    if (h->mode == 3 || (h->mode == 0 && swap_ok)) {
      const bool pk = h->scale_layout == MXGEMM_SCALES_PACKED;
      if (pk && (reinterpret_cast<uintptr_t>(A_scale) % 16 || reinterpret_cast<uintptr_t>(B_scale) % 16))
        return MXGEMM_ERR_MISALIGNED;
      return run_swapab(h, M, N, K, A, A_scale, B, B_scale, C, use_acc, out_dtype, pk, stream);
    }
  }

  // workspace size depends only on the shape and mode
  int CG = 1;
  if (h->mode == 2) CG = 2;
  // automatic: the CTA pair halves the B traffic and TMA requests per SM
  // and measured faster on every workload with more than one 128-row block
  else if (h->mode == 0 && M > 128) CG = 2;
  const int64_t m_tiles = cdiv(M, 128 * CG);
  const int64_t n_tiles = cdiv(N, 256);
  const int64_t k_steps = cdiv(K, 128);
  const int64_t num_tiles = m_tiles * n_tiles;
  if (num_tiles >= lim) return MXGEMM_ERR_INVALID_VALUE;
  // Scale chunks: built in the kernel from the row-major scales (single
  // CTAs on one row of tiles, M <= 128: the kernel streams B and has SM time
  // to spare, and no prepass runs before it), else repacked by a prepass into
  // 512-byte chunks.  On full tiles the in-kernel build measured slower: its
  // 16-byte row segments cost TMA and shared-memory transactions that the
  // mainloop needs (1-CTA square 4096: 64.1 us against 58.0 with the prepass).
  // Caller-packed scales (MXGEMM_OPT_SCALE_LAYOUT) are loaded as they are:
  // neither a prepass nor the scale loader.
  const bool packed = h->scale_layout == MXGEMM_SCALES_PACKED;
  if (packed && (reinterpret_cast<uintptr_t>(A_scale) % 16 || reinterpret_cast<uintptr_t>(B_scale) % 16))
    return MXGEMM_ERR_MISALIGNED;
  const bool fused = !packed && CG == 1 && M <= 128;
  const int64_t a_chunks = fused || packed ? 0 : m_tiles * CG * k_steps;
  const int64_t b_chunks = fused || packed ? 0 : n_tiles * k_steps * 2;  // 2 per 256 columns
  // 6- and 4-bit formats are packed 16 elements per 16-byte group first
  // (with MXGEMM_ELEMS_PACKED they arrive in that form and are read as
  // they are: whole 16-element groups, so N % 16 == 0 for a sub-byte B)
  // B given N x K (MXGEMM_B_N_BY_K) has rows of K bytes: never re-pitched
  // (K % 32 == 0), and its sub-byte groups run along K
  const bool b_km = h->b_major == MXGEMM_B_N_BY_K;
  const bool elems_packed = h->elem_layout == MXGEMM_ELEMS_PACKED;
  if (elems_packed && h->b_fmt >= MXGEMM_FMT_E2M3 && !b_km && N % 16 != 0) return MXGEMM_ERR_INVALID_VALUE;
  const int a_bits = elems_packed ? 8 : h->a_fmt == MXGEMM_FMT_E2M1 ? 4 : h->a_fmt >= MXGEMM_FMT_E2M3 ? 6 : 8;
  const int b_bits = elems_packed ? 8 : h->b_fmt == MXGEMM_FMT_E2M1 ? 4 : h->b_fmt >= MXGEMM_FMT_E2M3 ? 6 : 8;
  const bool pad_b = !b_km && ((N % 16) != 0 || b_bits < 8);
  const bool pack_bk = b_km && b_bits < 8;  // sub-byte B, N x K: packed along K first
  const int64_t npad = round_up(static_cast<size_t>(N), 16);
  // Cluster launch control: one cluster per work item (whole tiles, then
  // half-width items), handed out by the hardware; no stream-K, whose
  // partial-sum slots belong to fixed CTAs.
  const bool clc = h->scheduler == 1;
  Split sp = plan_split(num_tiles, k_steps, h->sm_count / CG, h->stream_k != 0, !clc, M);
  if (clc) sp.units = sp.dp_tiles + sp.half_tiles;
  const Sizes z = plan_sizes(a_chunks, b_chunks,
                             pad_b ? static_cast<size_t>(K) * npad
                                   : pack_bk ? static_cast<size_t>(N) * K : 0, sp, CG,
                             a_bits < 8 ? static_cast<size_t>(M) * K : 0);
  const size_t off_b = z.off_b;
  const size_t ws_bytes = z.total;

  Plan *plan = nullptr;
  for (Plan &pl : h->plans)
    if (pl.matches(M, N, K, A, A_scale, B, B_scale, C, use_acc, out_dtype, h->mode,
                   h->stall_producer, h->scheduler, h->stream_k, h->timeout_ns, h->ws.ptr,
                   h->a_fmt * 8 + h->b_fmt + 64 * h->elem_layout + 128 * h->b_major, h->scale_layout) &&
        !pl.swap && h->ws.bytes >= ws_bytes) {
      plan = &pl;
      break;
    }
  if (!plan) {
    if (!on_device(C, h->device) || !on_device(A, h->device) || !on_device(B, h->device) ||
        !on_device(A_scale, h->device) || !on_device(B_scale, h->device))
      return MXGEMM_ERR_INVALID_VALUE;
    int st = ensure_workspace(h, ws_bytes, stream);
    if (st != MXGEMM_OK) return st;
    plan = &h->plans[h->next_plan];
    h->next_plan = (h->next_plan + 1) % kPlanCache;
    plan->valid = false;
    plan->swap = false;
    st = build_plan(h, plan, M, N, K, A, A_scale, B, B_scale, C, use_acc, out_dtype, CG, m_tiles,
                    n_tiles, k_steps, num_tiles, a_chunks, b_chunks, pad_b, npad, sp, z, a_bits,
                    b_bits, fused, packed);
    if (st != MXGEMM_OK) return st;
  }

  // ---- launches: [B re-pitch], scale repack, GEMM
  if (plan->pad_b) {
    mxg::pad_rows_kernel<<<launch_blocks(K * (plan->npad / 16), 256), 256, 0, stream>>>(
        static_cast<const uint8_t *>(B), K, N, plan->npad, h->ws.ptr + off_b, plan->b_bits);
    ++h->launches;
  } else if (plan->pack_bk) {
    mxg::pad_rows_kernel<<<launch_blocks(N * (K / 16), 256), 256, 0, stream>>>(
        static_cast<const uint8_t *>(B), N, K, K, h->ws.ptr + off_b, plan->b_bits);
    ++h->launches;
  }
  if (plan->a_bits < 8) {
    mxg::pad_rows_kernel<<<launch_blocks(M * (K / 16), 256), 256, 0, stream>>>(
        static_cast<const uint8_t *>(A), M, K, K, h->ws.ptr + plan->off_a, plan->a_bits);
    ++h->launches;
  }
  if (plan->repack_lite) {
    // one CTA per SM at most, so that each fits beside a GEMM CTA
    const int units = plan->blocks_a + plan->blocks_b;
    const int grid = std::max(1, std::min((units + 1) / 2, h->sm_count));
    mxg::repack_scales_lite_kernel<<<grid, mxg::kRepackLiteThreads, 0, stream>>>(plan->ra, plan->rb,
                                                                               plan->blocks_a, units);
    h->launches += 1;
  } else if (plan->repack) {
    mxg::repack_scales_kernel<<<plan->blocks_a + plan->blocks_b, mxg::kRepackThreads, 0, stream>>>(
        plan->ra, plan->rb, plan->blocks_a);
    h->launches += 1;
  }
  if (cudaGetLastError() != cudaSuccess) return MXGEMM_ERR_CUDA;
  mxg::KParams kp = plan->kp;
  if (++h->epoch == 0) h->epoch = 1;  // 0 is the flags' initial value
  kp.epoch = h->epoch;
  return plan->CG == 2 ? launch_gemm<2>(h, plan->tA, plan->tB, plan->tB64, plan->tSA, plan->tSB, plan->tC,
                                        kp, plan->units, stream)
                       : launch_gemm<1>(h, plan->tA, plan->tB, plan->tB64, plan->tSA, plan->tSB, plan->tC,
                                        kp, plan->units, stream);
}

int mxgemm_get_device_status(mxgemm_handle_t h, mxgemm_stream_t stream_, int *status_out,
                             int *detail_out) {
  if (!h || !status_out) return MXGEMM_ERR_INVALID_VALUE;
  DeviceGuard g(h->device);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int hostv[2] = {0, 0};
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MXGEMM_ERR_CUDA;
  if (cudaMemcpy(hostv, h->d_status, sizeof(hostv), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MXGEMM_ERR_CUDA;
  if (cudaMemset(h->d_status, 0, sizeof(hostv)) != cudaSuccess) return MXGEMM_ERR_CUDA;
  *status_out = hostv[0];
  if (detail_out) *detail_out = hostv[1];
  return MXGEMM_OK;
}

int mxgemm_set_profile_events(mxgemm_handle_t h, void *ev_before, void *ev_after) {
  if (!h) return MXGEMM_ERR_INVALID_VALUE;
  h->prof_before = static_cast<cudaEvent_t>(ev_before);
  h->prof_after = static_cast<cudaEvent_t>(ev_after);
  return MXGEMM_OK;
}

int mxgemm_get_launch_count(mxgemm_handle_t h, int64_t *count_out) {
  if (!h || !count_out) return MXGEMM_ERR_INVALID_VALUE;
  *count_out = h->launches;
  return MXGEMM_OK;
}

int mxgemm_destroy(mxgemm_handle_t h) {
  if (!h) return MXGEMM_ERR_INVALID_VALUE;
  {
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    if (h->ws.ptr) cudaFree(h->ws.ptr);
    if (h->d_status) cudaFree(h->d_status);
    if (h->flags) cudaFree(h->flags);
    HostPipe &hp = h->hp;
    if (hp.stage.ptr) cudaFree(hp.stage.ptr);
    for (cudaEvent_t e : {hp.start, hp.b_ready, hp.in_ready[0], hp.in_ready[1], hp.in_ready[2],
                          hp.gemm_done[0], hp.gemm_done[1], hp.gemm_done[2], hp.out_done[0],
                          hp.out_done[1], hp.out_done[2], hp.b_used[0], hp.b_used[1]})
      if (e) cudaEventDestroy(e);
    if (hp.h2d) cudaStreamDestroy(hp.h2d);
    if (hp.d2h) cudaStreamDestroy(hp.d2h);
  }
  delete h;
  return MXGEMM_OK;
}

}  // extern "C"

// ===========================================================================
// mxgemm_quantize: MX quantization of a real matrix on the GPU.
// ===========================================================================

namespace {

template <typename T, bool SR>
void launch_quantize(const T *x, int64_t R, int64_t C, int along_cols, const uint32_t *rbits,
                     uint8_t *cd, uint8_t *sc, int64_t S, int sms, cudaStream_t stream) {
  // grid: a few resident blocks per SM, grid-stride loops over the work
  const int threads = 256;
  if (!along_cols) {
    const int64_t nblocks = R * (C / 32);
    const int64_t warps_needed = (nblocks + 7) / 8;  // a warp takes 8 blocks
    int grid = static_cast<int>(std::min<int64_t>(cdiv(warps_needed, threads / 32), int64_t(sms) * 8));
    if (grid < 1) grid = 1;
    mxg::mx_quantize_rows_kernel<T, SR><<<grid, threads, 0, stream>>>(x, nblocks, rbits, cd, sc,
                                                                      C / 32, S);
  } else {
    // two adjacent columns per thread when C is even (wider loads and
    // stores); one with stochastic rounding, whose random words take as many
    // registers again (two columns measured slower there: spills for FP32
    // input, lower occupancy for BF16)
    constexpr bool kPairsOk = !SR;
    const bool pairs = kPairsOk && C % 2 == 0;
    const int64_t work = (R / 32) * (pairs ? C / 2 : C);
    int grid = static_cast<int>(std::min<int64_t>(cdiv(work, threads), int64_t(sms) * 8));
    if (grid < 1) grid = 1;
    if constexpr (kPairsOk) {
      if (pairs) {
        mxg::mx_quantize_cols_kernel<T, 2, SR><<<grid, threads, 0, stream>>>(x, R, C, rbits, cd, sc, S);
        return;
      }
    }
    mxg::mx_quantize_cols_kernel<T, 1, SR><<<grid, threads, 0, stream>>>(x, R, C, rbits, cd, sc, S);
  }
}

// Bytes of the scales of an R x C matrix quantized along the rows (A: M = R,
// K = C) or down the columns (B: K = R, N = C), in the given layout; -1 for
// an invalid layout.
int64_t scale_bytes(int64_t R, int64_t C, int along_cols, int layout) {
  if (layout == MXGEMM_SCALES_ROW_MAJOR) return along_cols ? C * (R / 32) : R * (C / 32);
  if (layout != MXGEMM_SCALES_PACKED) return -1;
  const int64_t K = along_cols ? R : C, S = cdiv(K, 128);
  return along_cols ? cdiv(C, 256) * S * 1024 : cdiv(R, 128) * S * 512;
}

int quantize_impl(const void *X, int x_dtype, int64_t R, int64_t C, int along_cols,
                  const void *rand_bits, bool sr, int layout, void *codes, void *scales,
                  mxgemm_stream_t stream_) {
  const int64_t lim = int64_t(1) << 31;
  if (R < 0 || C < 0 || R >= lim || C >= lim) return MXGEMM_ERR_INVALID_VALUE;
  if (layout != MXGEMM_SCALES_ROW_MAJOR && layout != MXGEMM_SCALES_PACKED)
    return MXGEMM_ERR_INVALID_VALUE;
  const bool packed = layout == MXGEMM_SCALES_PACKED;
  if (x_dtype != MXGEMM_IN_F32 && x_dtype != MXGEMM_IN_BF16) return MXGEMM_ERR_INVALID_VALUE;
  if (along_cols != 0 && along_cols != 1) return MXGEMM_ERR_INVALID_VALUE;
  if ((along_cols ? R % 32 : C % 32) != 0) return MXGEMM_ERR_INVALID_VALUE;
  if (R == 0 || C == 0) return MXGEMM_OK;
  if (!X || !codes || !scales || (sr && !rand_bits)) return MXGEMM_ERR_INVALID_VALUE;
  if (reinterpret_cast<uintptr_t>(X) % 16 || reinterpret_cast<uintptr_t>(codes) % 16 ||
      reinterpret_cast<uintptr_t>(rand_bits) % 16 || (packed && reinterpret_cast<uintptr_t>(scales) % 16))
    return MXGEMM_ERR_MISALIGNED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  if (!on_device(X, dev) || !on_device(codes, dev) || !on_device(scales, dev) ||
      (sr && !on_device(rand_bits, dev)))
    return MXGEMM_ERR_INVALID_VALUE;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t *cd = static_cast<uint8_t *>(codes), *sc = static_cast<uint8_t *>(scales);
  const uint32_t *rb = static_cast<const uint32_t *>(rand_bits);
  // packed: the padding entries (rows or columns past the matrix, K blocks
  // past the last) hold 127, the kernel then writes every real scale
  const int64_t S = packed ? cdiv(along_cols ? R : C, 128) : 0;
  if (packed && cudaMemsetAsync(sc, 127, static_cast<size_t>(scale_bytes(R, C, along_cols, layout)),
                                stream) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  if (x_dtype == MXGEMM_IN_F32) {
    const float *x = static_cast<const float *>(X);
    if (sr) launch_quantize<float, true>(x, R, C, along_cols, rb, cd, sc, S, sms, stream);
    else launch_quantize<float, false>(x, R, C, along_cols, nullptr, cd, sc, S, sms, stream);
  } else {
    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(X);
    if (sr) launch_quantize<__nv_bfloat16, true>(x, R, C, along_cols, rb, cd, sc, S, sms, stream);
    else launch_quantize<__nv_bfloat16, false>(x, R, C, along_cols, nullptr, cd, sc, S, sms, stream);
  }
  if (cudaGetLastError() != cudaSuccess) return MXGEMM_ERR_CUDA;
  return MXGEMM_OK;
}

}  // namespace

extern "C" int mxgemm_quantize(const void *X, int x_dtype, int64_t R, int64_t C, int along_cols,
                               void *codes, void *scales, mxgemm_stream_t stream) {
  return quantize_impl(X, x_dtype, R, C, along_cols, nullptr, false, MXGEMM_SCALES_ROW_MAJOR, codes,
                       scales, stream);
}

extern "C" int mxgemm_quantize_sr(const void *X, int x_dtype, int64_t R, int64_t C,
                                  int along_cols, const void *rand_bits, void *codes,
                                  void *scales, mxgemm_stream_t stream) {
  return quantize_impl(X, x_dtype, R, C, along_cols, rand_bits, true, MXGEMM_SCALES_ROW_MAJOR, codes,
                       scales, stream);
}

extern "C" int mxgemm_quantize_ex(const void *X, int x_dtype, int64_t R, int64_t C, int along_cols,
                                  const void *rand_bits, int scale_layout, void *codes,
                                  void *scales, mxgemm_stream_t stream) {
  return quantize_impl(X, x_dtype, R, C, along_cols, rand_bits, rand_bits != nullptr, scale_layout,
                       codes, scales, stream);
}

extern "C" int mxgemm_scale_bytes(int64_t R, int64_t C, int along_cols, int scale_layout,
                                  int64_t *bytes_out) {
  if (!bytes_out || R < 0 || C < 0 || (along_cols != 0 && along_cols != 1) ||
      (along_cols ? R % 32 : C % 32) != 0)
    return MXGEMM_ERR_INVALID_VALUE;
  const int64_t b = scale_bytes(R, C, along_cols, scale_layout);
  if (b < 0) return MXGEMM_ERR_INVALID_VALUE;
  *bytes_out = b;
  return MXGEMM_OK;
}

// ===========================================================================
// mxgemm_run_host: operands and result in host memory.
//
// B and its scales go to the device first; then the rows of A (and of C)
// move in slabs through three device slots, so that a slab's GEMM overlaps
// the next slab's copy in and the copies out of the two before it.  The GEMM of a slab
// is an ordinary mxgemm_run on the slot's buffers.
// ===========================================================================

namespace {

int host_pipe_init(mxgemm_ctx *h) {
  HostPipe &hp = h->hp;
  if (hp.ready) return MXGEMM_OK;
  // anything created by an earlier, failed attempt is kept, not re-created
  if ((!hp.h2d && cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) != cudaSuccess) ||
      (!hp.d2h && cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) != cudaSuccess)) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  cudaEvent_t *evs[] = {&hp.start,        &hp.b_ready,      &hp.in_ready[0],  &hp.in_ready[1],
                        &hp.in_ready[2],  &hp.gemm_done[0], &hp.gemm_done[1], &hp.gemm_done[2],
                        &hp.out_done[0],  &hp.out_done[1],  &hp.out_done[2],  &hp.b_used[0],
                        &hp.b_used[1]};
  for (cudaEvent_t *e : evs)
    if (!*e && cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return MXGEMM_ERR_CUDA;
    }
  hp.ready = true;
  return MXGEMM_OK;
}

// *grown is set when the staging area was (re)allocated on `stream`.
int ensure_stage(mxgemm_ctx *h, size_t bytes, cudaStream_t stream, bool *grown) {
  Workspace &w = h->hp.stage;
  *grown = false;
  if (w.bytes >= bytes) return MXGEMM_OK;
  *grown = true;
  if (w.ptr) {
    // every earlier use is ordered before this point of `stream`
    cudaFreeAsync(w.ptr, stream);
    w.ptr = nullptr;
    w.bytes = 0;
  }
  void *p = nullptr;
  const size_t want = round_up(bytes, size_t(2) << 20);
  if (cudaMallocAsync(&p, want, stream) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_OUT_OF_MEMORY;
  }
  w.ptr = static_cast<uint8_t *>(p);
  w.bytes = want;
  return MXGEMM_OK;
}

// one asynchronous copy; false when it could not be enqueued
bool copy_async(void *dst, const void *src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
  if (bytes == 0) return true;
  if (cudaMemcpyAsync(dst, src, bytes, kind, s) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

bool wait_event(cudaStream_t s, cudaEvent_t e) {
  if (cudaStreamWaitEvent(s, e, 0) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

bool record_event(cudaEvent_t e, cudaStream_t s) {
  if (cudaEventRecord(e, s) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

}  // namespace

extern "C" int mxgemm_run_host(mxgemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A,
                               const void *A_scale, const void *B, const void *B_scale, void *C,
                               int use_acc, int out_dtype, mxgemm_stream_t stream_) {
  if (!h) return MXGEMM_ERR_INVALID_VALUE;
  const int64_t lim = int64_t(1) << 31;
  if (M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim) return MXGEMM_ERR_INVALID_VALUE;
  if (K % 32 != 0) return MXGEMM_ERR_INVALID_VALUE;
  if (out_dtype != MXGEMM_OUT_F32 && out_dtype != MXGEMM_OUT_BF16) return MXGEMM_ERR_INVALID_VALUE;
  if (use_acc != 0 && use_acc != 1) return MXGEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return MXGEMM_OK;
  if (!C) return MXGEMM_ERR_INVALID_VALUE;
  const size_t esz = out_dtype == MXGEMM_OUT_F32 ? 4 : 2;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  DeviceGuard g(h->device);
  if (K == 0) {
    if (use_acc) return MXGEMM_OK;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
      cudaGetLastError();
      return MXGEMM_ERR_CUDA;
    }
    std::memset(C, 0, static_cast<size_t>(M) * N * esz);
    return MXGEMM_OK;
  }
  if (!A || !B || !A_scale || !B_scale) return MXGEMM_ERR_INVALID_VALUE;

  int st = host_pipe_init(h);
  if (st != MXGEMM_OK) return st;
  HostPipe &hp = h->hp;
  const int64_t kb = K / 32;
  // slab rows: about 8 slabs, whole 256-row pair tiles, at least 256 rows
  int64_t ms = round_up(static_cast<size_t>(cdiv(M, 8)), 256);
  if (ms < 256) ms = 256;
  if (ms > M) ms = M;
  const int64_t nslab = cdiv(M, ms);
  // scales: row-major, or packed (slabs are whole 128-row blocks: ms is a
  // multiple of 256, and only the last slab may end short of one)
  const bool packed = h->scale_layout == MXGEMM_SCALES_PACKED;
  const int64_t S = cdiv(K, 128);
  auto as_slab_bytes = [&](int64_t rows) -> size_t {
    return packed ? static_cast<size_t>(cdiv(rows, 128) * S * 512) : static_cast<size_t>(rows) * kb;
  };
  const size_t b_bytes = static_cast<size_t>(K) * N;
  const size_t bs_bytes = packed ? static_cast<size_t>(cdiv(N, 256) * S * 1024) : static_cast<size_t>(N) * kb;
  const size_t a_bytes = static_cast<size_t>(ms) * K, as_bytes = as_slab_bytes(ms);
  const size_t c_bytes = static_cast<size_t>(ms) * N * esz;
  // staging: two B slots (consecutive calls alternate, so that one call's
  // B copy overlaps the previous call's last slabs), then three row slots
  const size_t off_bs = round_up(b_bytes, 256);
  const size_t bslot_bytes = round_up(off_bs + bs_bytes, 256);
  const size_t off_slot = 2 * bslot_bytes;
  const size_t off_as = round_up(a_bytes, 256);
  const size_t off_c = round_up(off_as + as_bytes, 256);
  const size_t slot_bytes = round_up(off_c + c_bytes, 256);
  bool grown = false;
  st = ensure_stage(h, off_slot + HostPipe::kSlots * slot_bytes, stream, &grown);
  if (st != MXGEMM_OK) return st;
  const uint8_t *hA = static_cast<const uint8_t *>(A), *hAs = static_cast<const uint8_t *>(A_scale);
  uint8_t *hC = static_cast<uint8_t *>(C);
  const int bs = hp.bslot;
  hp.bslot ^= 1;
  uint8_t *dB = hp.stage.ptr + bs * bslot_bytes;
  uint8_t *base = hp.stage.ptr;

  // The copies do not wait for the caller's stream: the host operands are
  // ready when the call is made, and every staging slot is reused only after
  // the events of its previous use (also from earlier calls; an event never
  // recorded is no wait).  The copy streams are ordered after the caller's
  // stream only when the staging area was just (re)allocated there, or when
  // C is read (use_acc): C on the host may still be arriving from an
  // earlier call.
  if ((grown || use_acc) &&
      (!record_event(hp.start, stream) || !wait_event(hp.h2d, hp.start) || !wait_event(hp.d2h, hp.start)))
    return MXGEMM_ERR_CUDA;
  if (!wait_event(hp.h2d, hp.b_used[bs]) ||
      !copy_async(dB, B, b_bytes, cudaMemcpyHostToDevice, hp.h2d) ||
      !copy_async(dB + off_bs, B_scale, bs_bytes, cudaMemcpyHostToDevice, hp.h2d) ||
      !record_event(hp.b_ready, hp.h2d))
    return MXGEMM_ERR_CUDA;
  for (int64_t j = 0; j < nslab; ++j) {
    const int s = static_cast<int>(j % HostPipe::kSlots);
    const int64_t m0 = j * ms, mj = (M - m0 < ms) ? M - m0 : ms;
    uint8_t *dA = base + off_slot + s * slot_bytes;
    uint8_t *dAs = dA + off_as;
    uint8_t *dC = dA + off_c;
    const size_t crow = static_cast<size_t>(N) * esz;
    // inputs of slab j into slot s, once the slot's previous GEMM (and,
    // when C is read, its copy out) no longer needs it
    if (!wait_event(hp.h2d, hp.gemm_done[s]) || (use_acc && !wait_event(hp.h2d, hp.out_done[s])))
      return MXGEMM_ERR_CUDA;
    if (!copy_async(dA, hA + m0 * K, static_cast<size_t>(mj) * K, cudaMemcpyHostToDevice, hp.h2d) ||
        !copy_async(dAs, hAs + (packed ? (m0 / 128) * S * 512 : m0 * kb), as_slab_bytes(mj),
                    cudaMemcpyHostToDevice, hp.h2d) ||
        (use_acc && !copy_async(dC, hC + m0 * crow, mj * crow, cudaMemcpyHostToDevice, hp.h2d)) ||
        !record_event(hp.in_ready[s], hp.h2d))
      return MXGEMM_ERR_CUDA;
    // the GEMM of slab j on the caller's stream
    if (!wait_event(stream, hp.in_ready[s]) || (j == 0 && !wait_event(stream, hp.b_ready)) ||
        !wait_event(stream, hp.out_done[s]))
      return MXGEMM_ERR_CUDA;
    st = mxgemm_run(h, mj, N, K, dA, dAs, dB, dB + off_bs, dC, use_acc, out_dtype, stream);
    if (st != MXGEMM_OK) return st;
    if (!record_event(hp.gemm_done[s], stream)) return MXGEMM_ERR_CUDA;
    // its C rows back to the host
    if (!wait_event(hp.d2h, hp.gemm_done[s]) ||
        !copy_async(hC + m0 * crow, dC, mj * crow, cudaMemcpyDeviceToHost, hp.d2h) ||
        !record_event(hp.out_done[s], hp.d2h))
      return MXGEMM_ERR_CUDA;
  }
  // B slot bs is free once this call's last GEMM is done; the caller's
  // stream completes once every slab is back
  if (!record_event(hp.b_used[bs], stream)) return MXGEMM_ERR_CUDA;
  for (int s = 0; s < HostPipe::kSlots && s < nslab; ++s)
    if (!wait_event(stream, hp.out_done[s])) return MXGEMM_ERR_CUDA;
  return MXGEMM_OK;
}

// ===========================================================================
// mxgemm_run_noalloc: the same product without any device allocation.
//
// Callers that cannot allocate device memory where they call the GEMM (a
// plug-in whose host framework owns all device memory, code that must not
// allocate after start-up) use this entry point.  The kernel builds the scale chunks itself (fused scales), so its
// only scratch is B re-pitched when N % 16 != 0.  That lives in the
// file-scope array below, which the CUDA runtime places when it loads this
// library's device code: every GPU that loads the library holds these
// kNoAllocScratchBytes until the process exits.
// ===========================================================================

namespace {
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
static __device__ __align__(256) int g_noalloc_status[2];

namespace {

struct NoAllocDevice {
  bool ready = false;
  uint8_t *scratch = nullptr;  // this device's address of g_noalloc_scratch
  int *status = nullptr;       // this device's address of g_noalloc_status
  int sm_count = 0;
  bool attr_set[3][16] = {};
};

constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_noalloc_encode = nullptr;
// process-wide options of the no-allocation path (mxgemm_noalloc_set_option)
std::atomic<long long> g_noalloc_timeout_ns{2000000000LL};
std::atomic<int> g_noalloc_stall{0};

// Once per device, with that device current: check it, and look up the
// device addresses of the scratch arrays (in host code their names are
// host-side stand-ins, not device addresses).
int noalloc_setup(int dev, NoAllocDevice **out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MXGEMM_ERR_INVALID_VALUE;
  NoAllocDevice &d = g_noalloc_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return MXGEMM_ERR_CUDA;
    }
    if (!(major == 10 && minor == 3)) return MXGEMM_ERR_UNSUPPORTED_DEVICE;
    if (!g_noalloc_encode) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return MXGEMM_ERR_CUDA;
      }
      g_noalloc_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    void *scratch = nullptr, *status = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess ||
        cudaGetSymbolAddress(&status, g_noalloc_status) != cudaSuccess || !scratch || !status) {
      cudaGetLastError();
      return MXGEMM_ERR_CUDA;
    }
    d.scratch = static_cast<uint8_t *>(scratch);
    d.status = static_cast<int *>(status);
    d.sm_count = sms;
    d.ready = true;
  }
  *out = &d;
  return MXGEMM_OK;
}

}  // namespace

extern "C" int mxgemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A,
                                  const void *A_scale, const void *B, const void *B_scale,
                                  void *C, int use_acc, int out_dtype, mxgemm_stream_t stream_) {
  const int64_t lim = int64_t(1) << 31;
  if (M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim) return MXGEMM_ERR_INVALID_VALUE;
  if (K % 32 != 0) return MXGEMM_ERR_INVALID_VALUE;
  if (out_dtype != MXGEMM_OUT_F32 && out_dtype != MXGEMM_OUT_BF16) return MXGEMM_ERR_INVALID_VALUE;
  if (use_acc != 0 && use_acc != 1) return MXGEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return MXGEMM_OK;
  const size_t esz = out_dtype == MXGEMM_OUT_F32 ? 4 : 2;
  if (!C) return MXGEMM_ERR_INVALID_VALUE;
  if (reinterpret_cast<uintptr_t>(C) % 16) return MXGEMM_ERR_MISALIGNED;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  NoAllocDevice *nd = nullptr;
  int st = noalloc_setup(dev, &nd);
  if (st != MXGEMM_OK) return st;
  if (K == 0) {
    if (!on_device(C, dev)) return MXGEMM_ERR_INVALID_VALUE;
    if (use_acc) return MXGEMM_OK;
    if (cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * esz, stream) != cudaSuccess) {
      cudaGetLastError();
      return MXGEMM_ERR_CUDA;
    }
    return MXGEMM_OK;
  }
  if (!A || !B || !A_scale || !B_scale) return MXGEMM_ERR_INVALID_VALUE;
  if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16)
    return MXGEMM_ERR_MISALIGNED;

  // single-CTA tiles, as the automatic mode of mxgemm_run
  const int CG = 1;
  const int64_t m_tiles = cdiv(M, 128 * CG);
  const int64_t n_tiles = cdiv(N, 256);
  const int64_t k_steps = cdiv(K, 128);
  const int64_t num_tiles = m_tiles * n_tiles;
  if (num_tiles >= lim) return MXGEMM_ERR_INVALID_VALUE;
  // the kernel builds the scale chunks itself (fused scales, whatever M):
  // no repacked scales in the scratch
  const int64_t a_chunks = 0, b_chunks = 0;
  const bool pad_b = (N % 16) != 0;
  const int64_t npad = round_up(static_cast<size_t>(N), 16);
  // no stream-K split here (no partial sums or flags): the scratch holds
  // only a re-pitched B
  const Split sp = plan_split(num_tiles, k_steps, nd->sm_count / CG, false, false, M);
  const Sizes z = plan_sizes(a_chunks, b_chunks, pad_b ? static_cast<size_t>(K) * npad : 0, sp, CG, 0);
  const size_t off_b = z.off_b;
  const size_t ws_bytes = z.total;
  if (ws_bytes > kNoAllocScratchBytes) return MXGEMM_ERR_TOO_LARGE;
  if (!on_device(C, dev) || !on_device(A, dev) || !on_device(B, dev) ||
      !on_device(A_scale, dev) || !on_device(B_scale, dev))
    return MXGEMM_ERR_INVALID_VALUE;

  // A handle-shaped context on the stack that points at the fixed scratch;
  // nothing in it is allocated or freed.
  mxgemm_ctx ctx;
  ctx.device = dev;
  ctx.sm_count = nd->sm_count;
  ctx.d_status = nd->status;
  ctx.ws.ptr = nd->scratch;
  ctx.ws.bytes = kNoAllocScratchBytes;
  ctx.encode = g_noalloc_encode;
  ctx.timeout_ns = g_noalloc_timeout_ns.load();
  ctx.stall_producer = g_noalloc_stall.load();
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (int i = 0; i < 3; ++i)
      for (int j = 0; j < 16; ++j) ctx.attr_set[i][j] = nd->attr_set[i][j];
  }
  Plan plan;
  st = build_plan(&ctx, &plan, M, N, K, A, A_scale, B, B_scale, C, use_acc, out_dtype, CG, m_tiles,
                  n_tiles, k_steps, num_tiles, a_chunks, b_chunks, pad_b, npad, sp, z, 8, 8,
                  true, false);
  if (st != MXGEMM_OK) return st;
  // The status word is not cleared here: it keeps the first failure since
  // mxgemm_noalloc_get_status last read (and cleared) it, so that one read
  // after many calls still sees a failure in any of them.
  if (pad_b)
    mxg::pad_rows_kernel<<<launch_blocks(K * (npad / 16), 256), 256, 0, stream>>>(
        static_cast<const uint8_t *>(B), K, N, npad, nd->scratch + off_b, 8);
  if (cudaGetLastError() != cudaSuccess) return MXGEMM_ERR_CUDA;
  mxg::KParams kp = plan.kp;
  kp.epoch = 1;  // no partial sums: the flags are not used
  st = launch_gemm<1>(&ctx, plan.tA, plan.tB, plan.tB64, plan.tSA, plan.tSB, plan.tC, kp, plan.units,
                      stream);
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (int i = 0; i < 3; ++i)
      for (int j = 0; j < 16; ++j) nd->attr_set[i][j] = nd->attr_set[i][j] || ctx.attr_set[i][j];
  }
  return st;
}

extern "C" int mxgemm_noalloc_set_option(int option, int64_t value) {
  switch (option) {
    case MXGEMM_OPT_WAIT_TIMEOUT_NS:
      if (value <= 0) return MXGEMM_ERR_INVALID_VALUE;
      g_noalloc_timeout_ns.store(static_cast<long long>(value));
      return MXGEMM_OK;
    case MXGEMM_OPT_TEST_STALL_PRODUCER:
      if (value < 0 || value > 1) return MXGEMM_ERR_INVALID_VALUE;
      g_noalloc_stall.store(static_cast<int>(value));
      return MXGEMM_OK;
    default:
      return MXGEMM_ERR_INVALID_VALUE;
  }
}

extern "C" int mxgemm_noalloc_get_status(mxgemm_stream_t stream_, int *status_out, int *detail_out) {
  if (!status_out) return MXGEMM_ERR_INVALID_VALUE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  NoAllocDevice *nd = nullptr;
  int st = noalloc_setup(dev, &nd);
  if (st != MXGEMM_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  // a plain synchronous copy into the caller's host ints: no pinned staging
  // buffer is allocated
  int hostv[2] = {0, 0};
  if (cudaStreamSynchronize(stream) != cudaSuccess ||
      cudaMemcpy(hostv, nd->status, sizeof(hostv), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(nd->status, 0, sizeof(hostv)) != cudaSuccess) {
    cudaGetLastError();
    return MXGEMM_ERR_CUDA;
  }
  *status_out = hostv[0];
  if (detail_out) *detail_out = hostv[1];
  return MXGEMM_OK;
}
