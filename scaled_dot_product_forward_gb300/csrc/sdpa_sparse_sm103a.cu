// sdpa_sparse_sm103a.cu -- sparse top-k attention forward and its index
// preparation, for sm_103a.
//
// The DeepSeek sparse attention (DSA) forward of "FlashInfer, Cake DSA kernel
// optimization" (blog.secrett2633.cloud): every query row attends only to the
// key rows its index row lists, over one key/value head shared by all query
// heads (`out, lse = fwd(q, kv, idx, topk_length=...)`), and the index rows
// are hole-free -- the valid entries first, counted by topk_length -- after a
// single-launch preparation that turns per-document positions into global
// rows (same page, sections 1 and 3).
//
// Forward, built the way the dense kernel is, for one shared key set per query
// row instead of one per tile:
//   * a job is one query row and a group of up to 128 of its heads, which
//     share the gathered keys; groups of more than 64 heads are the 128 rows
//     of M = 128 products, one softmax thread a row; groups of at most 64
//     take M = 64 products (head h in TMEM lane 32 (h / 16) + h % 16) and two
//     softmax threads a row, so no thread works on rows the group lacks;
//   * warp 0 loads the job's Q with a 3-D TMA box; warps 8..11 gather the K
//     and V rows by index with coalesced 16-byte cp.async copies (128 keys per
//     stage) into the swizzled layout the tensor core reads, after checking
//     every index (entries past the row's count or out of range become row 0
//     and are removed in the softmax), and announce each stage through the
//     copy unit when its rows have landed; with one kv tensor the rows are
//     gathered once;
//   * warp 1 issues S = Q K^T into two alternating TMEM buffers, so S(j+1)
//     runs while the softmax works on S(j), and O += P V with P in its own
//     double-buffered TMEM columns;
//   * warpgroup 1 runs the online softmax and writes O / l and the
//     log-sum-exp.
// Every barrier wait is bounded in time; on expiry the CTA records a status
// bit (read with the dense kernel's by sdpa_last_device_status), stops and
// frees its tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sdpa_internal.h"

using namespace sdpa_dev;

__device__ unsigned int g_sdpa_sparse_status = 0;

namespace {

constexpr int kRows = 128;     // head rows per job (TMEM lanes)
constexpr int kKeys = 128;     // gathered keys per stage
constexpr int kThreads = 384;  // WG0: Q loads, MMA, 2 idle; WG1: softmax; WG2: gathers
constexpr int kGatherWarps = 4;  // warps 8..11: 32 key rows each
// Register split: the launch reserves kLaunchRegs per thread (the cap of
// __launch_bounds__(384, 1)); the softmax warpgroup takes registers from the
// other two.  128*232 + 256*136 == 384*168.
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kRegsSoftmax = 232;
constexpr uint32_t kRegsOther = 136;
static_assert(128 * kRegsSoftmax + 256 * kRegsOther <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct SLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = kKeys * 128;  // 128 rows x 64 elements
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  // K and V stages; with one kv tensor there are no V rows to hold and the
  // K ring takes both areas (2 * kStages stages).
  static constexpr int kStages = (D == 64) ? 6 : 3;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBar = kV + kStages * kTileBytes;
  static constexpr int kBarBytes = 1024;
  static constexpr int kTotal = kBar + kBarBytes + 1024;
};
static_assert(SLayout<128>::kTotal <= 227 * 1024, "shared memory over the per-CTA limit");
static_assert(SLayout<64>::kTotal <= 227 * 1024, "shared memory over the per-CTA limit");

// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+D), P0 [384,448), P1 [448,512).
constexpr uint32_t kColS0 = 0, kColO = 256, kColP = 384, kTmemCols = 512;

constexpr int kMaxStages = 12;
struct SBarriers {
  uint64_t q_full, q_empty;
  // S buffer b is refilled only after the product of the tile two before,
  // whose P the softmax stored after loading that tile's S: no release
  // barrier of its own
  uint64_t s_full[2];
  // P and O += P V double-buffered by tile parity: tile t uses P buffer t & 1,
  // p_ready[t & 1] and o_done[t & 1] (each completes once per two tiles).
  uint64_t p_ready[2], o_done[2], o_free, fin;
  uint64_t k_full[kMaxStages], k_empty[kMaxStages];
  // (a stage's K and V rows are copied as one group and announced together
  // by k_full)
  uint64_t v_empty[kMaxStages];
  // Validity of the 128 gathered keys of a tile, in the next slot of a ring
  // of stages + 2: word w bit i = key 32w + i; m_full[slot] completes when
  // all four gather warps have written their words.
  uint64_t m_full[kMaxStages + 2];
  uint32_t kmask[kMaxStages + 2][4];
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(SBarriers) <= 1024, "barrier block too large");

enum SparseSite : unsigned int {
  kSpQ = 1u << 1, kSpK = 1u << 2, kSpEmpty = 1u << 3, kSpS = 1u << 4, kSpP = 1u << 5,
  kSpO = 1u << 6, kSpDrain = 1u << 7,
};

template <class Bars>
__device__ __forceinline__ bool swait(uint64_t* bar, uint32_t parity, Bars* bars,
                                      uint64_t limit_ns, unsigned int site,
                                      bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 63u) == 0) {
      if (honour_abort && *reinterpret_cast<volatile uint32_t*>(&bars->abort_flag) != 0)
        return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *reinterpret_cast<volatile uint32_t*>(&bars->abort_flag) = 1u;
        atomicOr(&g_sdpa_sparse_status, 1u | site);
        return false;
      }
    }
  }
}
template <class Bars>
__device__ __forceinline__ bool warp_swait(uint64_t* bar, uint32_t parity, Bars* bars,
                                           uint64_t limit_ns, unsigned int site) {
  return __all_sync(0xffffffffu, swait(bar, parity, bars, limit_ns, site));
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// A job: query row `row`, heads [128 * group, +128), n_kv key tiles.
struct SJob {
  int row, group, len, n_kv;
};

// A position in a ring of n slots (the ring depths are run-time values, so
// positions advance by one instead of being divided out of a counter).
struct RingPos {
  int idx = 0;
  uint32_t phase = 0;  // completed laps, mod 2: the parity of this slot's current use
  bool lapped = false;  // some slot has been used before
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
      lapped = true;
    }
  }
};

__device__ __forceinline__ bool job_of(const sdpa_impl::SparseParams& p, int j, SJob& job) {
  if (j >= p.total_q * p.n_groups) return false;
  job.row = j / p.n_groups;
  job.group = j - job.row * p.n_groups;
  int len = p.topk;
  if (p.topk_length != nullptr) len = min(max(__ldg(p.topk_length + job.row), 0), p.topk);
  job.len = len;
  job.n_kv = (len + kKeys - 1) / kKeys;
  return true;
}

// One 128-key tile of a head row's online softmax, in the log2 domain (the
// calling thread owns the row; s holds its raw scores): keys whose bit in km
// is clear are removed, the running maximum m_used moves only when the
// tile's extremum passes it by more than 2^8 (need = true; l is then scaled
// by the returned alpha), and the exponentials are added to l and packed
// into P.  With a negative scale the extremum is the minimum (mval = +inf).
template <bool BF16>
__device__ __forceinline__ float softmax_tile(float (&s)[kKeys], const uint32_t (&km)[4],
                                              float sl2, bool pos_scale, float mval,
                                              float& m_used, float& l, bool& need,
                                              uint32_t (&pk)[kKeys / 2]) {
  const bool all_valid = (km[0] & km[1] & km[2] & km[3]) == 0xffffffffu;
  if (!all_valid) {
#pragma unroll
    for (int c = 0; c < kKeys; ++c) s[c] = ((km[c >> 5] >> (c & 31)) & 1u) ? s[c] : mval;
  }
  // row extremum: eight independent chains of three-input max / min
  float e8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) e8[i] = s[i];
  if (pos_scale) {
#pragma unroll
    for (int c = 8; c < kKeys; c += 16)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        e8[i] = max3f(e8[i], s[c + i], s[c + 8 + i < kKeys ? c + 8 + i : c + i]);
    e8[0] = max3f(e8[0], e8[1], e8[2]);
    e8[3] = max3f(e8[3], e8[4], e8[5]);
    e8[6] = fmaxf(e8[6], e8[7]);
    e8[0] = max3f(e8[0], e8[3], e8[6]);
  } else {
#pragma unroll
    for (int c = 8; c < kKeys; c += 16)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        e8[i] = min3f(e8[i], s[c + i], s[c + 8 + i < kKeys ? c + 8 + i : c + i]);
    e8[0] = min3f(e8[0], e8[1], e8[2]);
    e8[3] = min3f(e8[3], e8[4], e8[5]);
    e8[6] = fminf(e8[6], e8[7]);
    e8[0] = min3f(e8[0], e8[3], e8[6]);
  }
  const float ext = e8[0];
  const float m_tile = (ext == mval) ? -INFINITY : ext * sl2;
  need = m_tile > m_used + kRescaleLog2;
  float alpha = 1.0f;
  if (need) {
    alpha = ex2(m_used - m_tile);
    m_used = m_tile;
    l *= alpha;
  }
  const float neg_m = (m_used == -INFINITY) ? 0.0f : -m_used;
#pragma unroll
  for (int c = 0; c < kKeys; c += 2) fma2_bcast(s[c], s[c + 1], s[c], s[c + 1], sl2, neg_m);
#pragma unroll
  for (int c = 0; c < kKeys; ++c) s[c] = ex2(s[c]);
  float rs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) rs[i] = 0.0f;
#pragma unroll
  for (int c = 0; c < kKeys / 2; ++c) {
    add2_acc(rs[2 * (c & 3)], rs[2 * (c & 3) + 1], s[2 * c], s[2 * c + 1]);
    pk[c] = pack2<BF16>(s[2 * c], s[2 * c + 1]);
  }
  add2_acc(rs[0], rs[1], rs[2], rs[3]);
  add2_acc(rs[4], rs[5], rs[6], rs[7]);
  add2_acc(rs[0], rs[1], rs[4], rs[5]);
  l += rs[0] + rs[1];
  return alpha;
}

// Scales the D accumulator columns of the calling thread's TMEM lane
// (t_o: its lane and first column) by alpha.
template <int D>
__device__ __forceinline__ void rescale_row(uint32_t t_o, float alpha) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(t_o + c * 32, o);
    tmem_ld_wait();
    float* of = reinterpret_cast<float*>(o);
#pragma unroll
    for (int e = 0; e < 32; e += 2) mul2_bcast(of[e], of[e + 1], alpha);
    tmem_st32(t_o + c * 32, o);
  }
}

// Reads the calling thread's accumulator row (t_o as above) and, when
// `store`, writes it times inv_l as D elements at orow.
template <int D, bool BF16>
__device__ __forceinline__ void store_row(uint32_t t_o, float inv_l, uint16_t* orow, bool store) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(t_o + c * 32, o);
    tmem_ld_wait();
    uint32_t pw[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pw[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v)
        dst[v] = make_uint4(pw[4 * v], pw[4 * v + 1], pw[4 * v + 2], pw[4 * v + 3]);
    }
  }
}

// The no-key row: zeros and lse = -inf (the safe softmax of an empty row).
template <int D>
__device__ __forceinline__ void store_empty_row(const sdpa_impl::SparseParams& p, int row, int h) {
  uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + row * p.o_st + h * p.o_sh;
  for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
  if (p.lse != nullptr) p.lse[row * p.lse_st + h * p.lse_sh] = -INFINITY;
}

// O / l and the log-sum-exp of a finished head row.
template <int D, bool BF16>
__device__ __forceinline__ void finish_row(const sdpa_impl::SparseParams& p, uint32_t t_o, int row,
                                           int h, float m_used, float l) {
  const float inv_l = (l > 0.0f) ? (1.0f / l) : 0.0f;
  if (h < p.H && p.lse != nullptr) {
    constexpr float kLn2 = 0.693147180559945309f;
    p.lse[row * p.lse_st + h * p.lse_sh] = (l > 0.0f) ? (log2f(l) + m_used) * kLn2 : -INFINITY;
  }
  uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + row * p.o_st + h * p.o_sh;
  store_row<D, BF16>(t_o, inv_l, orow, h < p.H);
}

// ---- The half-row form (groups of at most 64 heads).  The products are
// M = 64 tcgen05.mma, which put row h of the group in TMEM lane
// 32 (h / 16) + h % 16, so each warp of the softmax warpgroup owns 16 rows
// (its quarter's first half), and threads t and t + 16 share row t: keys
// [0, 64) and [64, 128) of every tile, and the first and second halves of
// the row's accumulator columns.

// One tile's step on a half row (s: its 64 raw scores, km0 / km1: the
// validity bits of its keys).  The extremum is exchanged with the partner
// thread, so both take the same rescale decision; l is the half row's sum.
template <bool BF16>
__device__ __forceinline__ float softmax_half_tile(float (&s)[kKeys / 2], uint32_t km0,
                                                   uint32_t km1, float sl2, bool pos_scale,
                                                   float mval, float& m_used, float& l,
                                                   bool& need, uint32_t (&pk)[kKeys / 4]) {
  constexpr int kN = kKeys / 2;
  if ((km0 & km1) != 0xffffffffu) {
#pragma unroll
    for (int c = 0; c < kN; ++c)
      s[c] = (((c < 32 ? km0 : km1) >> (c & 31)) & 1u) ? s[c] : mval;
  }
  float e8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) e8[i] = s[i];
  if (pos_scale) {
#pragma unroll
    for (int c = 8; c < kN; c += 16)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        e8[i] = max3f(e8[i], s[c + i], s[c + 8 + i < kN ? c + 8 + i : c + i]);
    e8[0] = max3f(e8[0], e8[1], e8[2]);
    e8[3] = max3f(e8[3], e8[4], e8[5]);
    e8[6] = fmaxf(e8[6], e8[7]);
    e8[0] = max3f(e8[0], e8[3], e8[6]);
    e8[0] = fmaxf(e8[0], __shfl_xor_sync(0xffffffffu, e8[0], 16));
  } else {
#pragma unroll
    for (int c = 8; c < kN; c += 16)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        e8[i] = min3f(e8[i], s[c + i], s[c + 8 + i < kN ? c + 8 + i : c + i]);
    e8[0] = min3f(e8[0], e8[1], e8[2]);
    e8[3] = min3f(e8[3], e8[4], e8[5]);
    e8[6] = fminf(e8[6], e8[7]);
    e8[0] = min3f(e8[0], e8[3], e8[6]);
    e8[0] = fminf(e8[0], __shfl_xor_sync(0xffffffffu, e8[0], 16));
  }
  const float ext = e8[0];
  const float m_tile = (ext == mval) ? -INFINITY : ext * sl2;
  need = m_tile > m_used + kRescaleLog2;
  float alpha = 1.0f;
  if (need) {
    alpha = ex2(m_used - m_tile);
    m_used = m_tile;
    l *= alpha;
  }
  const float neg_m = (m_used == -INFINITY) ? 0.0f : -m_used;
#pragma unroll
  for (int c = 0; c < kN; c += 2) fma2_bcast(s[c], s[c + 1], s[c], s[c + 1], sl2, neg_m);
#pragma unroll
  for (int c = 0; c < kN; ++c) s[c] = ex2(s[c]);
  float rs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) rs[i] = 0.0f;
#pragma unroll
  for (int c = 0; c < kN / 2; ++c) {
    add2_acc(rs[2 * (c & 3)], rs[2 * (c & 3) + 1], s[2 * c], s[2 * c + 1]);
    pk[c] = pack2<BF16>(s[2 * c], s[2 * c + 1]);
  }
  add2_acc(rs[0], rs[1], rs[2], rs[3]);
  add2_acc(rs[4], rs[5], rs[6], rs[7]);
  add2_acc(rs[0], rs[1], rs[4], rs[5]);
  l += rs[0] + rs[1];
  return alpha;
}

// Scales the calling thread's half of its row's D accumulator columns (t_o:
// the warp's lane base and the first column).
template <int D>
__device__ __forceinline__ void rescale_half_row(uint32_t t_o, float alpha) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t o[32];
    tmem_ld16x2_32<D / 2>(t_o + c * 32, o);
    tmem_ld_wait();
    float* of = reinterpret_cast<float*>(o);
#pragma unroll
    for (int e = 0; e < 32; e += 2) mul2_bcast(of[e], of[e + 1], alpha);
    tmem_st16x2_32<D / 2>(t_o + c * 32, o);
  }
}

// O / l (l: the half row's sum, added to its partner's here) and the
// log-sum-exp of a finished row; each thread writes its half of the D
// elements.
template <int D, bool BF16>
__device__ __forceinline__ void finish_half_row(const sdpa_impl::SparseParams& p, uint32_t t_o,
                                                int row, int h, int half, float m_used,
                                                float l_part) {
  const float l = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);
  const float inv_l = (l > 0.0f) ? (1.0f / l) : 0.0f;
  if (h < p.H && half == 0 && p.lse != nullptr) {
    constexpr float kLn2 = 0.693147180559945309f;
    p.lse[row * p.lse_st + h * p.lse_sh] = (l > 0.0f) ? (log2f(l) + m_used) * kLn2 : -INFINITY;
  }
  uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + row * p.o_st + h * p.o_sh + half * (D / 2);
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t o[32];
    tmem_ld16x2_32<D / 2>(t_o + c * 32, o);
    tmem_ld_wait();
    uint32_t pw[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pw[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
    if (h < p.H) {
      uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v)
        dst[v] = make_uint4(pw[4 * v], pw[4 * v + 1], pw[4 * v + 2], pw[4 * v + 3]);
    }
  }
}

template <int D, bool BF16, bool HALF>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_fwd_kernel(const __grid_constant__ sdpa_impl::SparseParams p) {
  using Lay = SLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + Lay::kQ;
  uint8_t* sK = smem + Lay::kK;
  uint8_t* sV = smem + Lay::kV;
  SBarriers* bars = reinterpret_cast<SBarriers*>(smem + Lay::kBar);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = p.wait_limit_ns;
  const int step = static_cast<int>(gridDim.x);
  // ring depth (stages of K, and of V when separate) and mask slots (see the
  // softmax)
  const int nst = p.kv_shared ? 2 * Lay::kStages : Lay::kStages;
  const int n_slots = nst + 2;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->p_ready[b], kRows / 32);
      mbar_init(&bars->o_done[b], 1);
    }
    mbar_init(&bars->o_free, kRows / 32);
    mbar_init(&bars->fin, 1);
    for (int s = 0; s < kMaxStages + 2; ++s) mbar_init(&bars->m_full[s], kGatherWarps);
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&bars->k_full[s], kGatherWarps * 32);  // one arrival per gathering thread
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (HALF && p.q_rows < 64) {
    // rows H .. 63 of the Q tile (read by the M = 64 products) are never
    // loaded: zero them once, so the products read finite values there
    for (int i = threadIdx.x; i < Lay::kTileBytes / 16; i += kThreads)
      reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&p.tm_q);
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_wait();
  grid_launch_dependents();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------- softmax warps
    regs_increase<kRegsSoftmax>();
    const int wq = warp & 3;
    // head row within the group, and (half-row form) which half of it
    const int half = HALF ? (lane >> 4) : 0;
    const int r = HALF ? wq * 16 + (lane & 15) : wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 >= 0.0f;
    const float mval = pos_scale ? -INFINITY : INFINITY;
    uint32_t ns = 0;
    RingPos mslot;  // key-mask slot of the next tile
    bool ok = true;
    SJob job;
    for (int jj = static_cast<int>(blockIdx.x); ok && job_of(p, jj, job); jj += step) {
      const int h = job.group * kRows + r;
      if (job.n_kv == 0) {
        // no key: zeros and lse = -inf (the safe softmax of an empty row)
        if (HALF) {
          if (h < p.H) {
            uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + job.row * p.o_st + h * p.o_sh +
                             half * (D / 2);
            for (int c = 0; c < D / 2; c += 8)
              *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
            if (half == 0 && p.lse != nullptr)
              p.lse[job.row * p.lse_st + h * p.lse_sh] = -INFINITY;
          }
        } else if (h < p.H) {
          store_empty_row<D>(p, job.row, h);
        }
        continue;
      }
      float m_used = -INFINITY, l = 0.0f;
      for (int j = 0; j < job.n_kv; ++j) {
        // The tile's key mask first: it is written when the tile is gathered,
        // long before its S, so this read overlaps the wait for S.  The
        // gathers refill this mask slot (mask slots = stages + 2) only once
        // the stage of the tile two after this one is free again, which needs
        // that tile's P and so this tile's: m_full of the slot is at most one
        // phase ahead of this wait.
        uint32_t km[4];
        if (!warp_swait(&bars->m_full[mslot.idx], mslot.phase, bars, limit, kSpK)) {
          ok = false;
          break;
        }
        {
          const volatile uint32_t* src = bars->kmask[mslot.idx];
#pragma unroll
          for (int e = 0; e < 4; ++e) km[e] = src[e];
        }
        mslot.next(n_slots);
        const uint32_t b = ns & 1;
        if (!warp_swait(&bars->s_full[b], (ns >> 1) & 1, bars, limit, kSpS)) {
          ok = false;
          break;
        }
        ++ns;
        tc_fence_after();
        constexpr int kPer = HALF ? kKeys / 2 : kKeys;  // scores per thread
        float s[kPer];
        {
          uint32_t su[kPer];
#pragma unroll
          for (int c = 0; c < kPer / 32; ++c) {
            if (HALF)
              tmem_ld16x2_32<kKeys / 2>(tmem + kColS0 + b * 128 + lane_off + c * 32, su + c * 32);
            else
              tmem_ld32(tmem + kColS0 + b * 128 + lane_off + c * 32, su + c * 32);
          }
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kPer; ++c) s[c] = __uint_as_float(su[c]);
        }
        bool need;
        uint32_t pk[kPer / 2];
        float alpha;
        if constexpr (HALF)
          alpha = softmax_half_tile<BF16>(s, half ? km[2] : km[0], half ? km[3] : km[1], sl2,
                                          pos_scale, mval, m_used, l, need, pk);
        else
          alpha = softmax_tile<BF16>(s, km, sl2, pos_scale, mval, m_used, l, need, pk);
        // Global tile index t (all jobs of this CTA).  Each wait below is
        // on a barrier whose next phase needs this tile's P, so it can never
        // fall two phases behind.
        const uint32_t t = ns - 1;
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // O is rescaled once PV(t-1) (and so every earlier product) is done
          if (!warp_swait(&bars->o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, bars, limit, kSpO)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (HALF)
            rescale_half_row<D>(tmem + kColO + lane_off, alpha);
          else
            rescale_row<D>(tmem + kColO + lane_off, alpha);
        }
        // P buffer t & 1 is free once PV(t-2) is done, which S(t) being
        // complete implies: the issuing warp issued S(t) after PV(t-2), and a
        // commit completes only after every earlier product.  (The o_done
        // waits that remain cannot fall two phases behind: a barrier's next
        // phase needs this tile's P.)
        const uint32_t pb = t & 1;
        if constexpr (HALF) {
          tmem_st16x2_32<kKeys / 4>(tmem + kColP + pb * 64 + lane_off, pk);
        } else {
          tmem_st32(tmem + kColP + pb * 64 + lane_off, pk);
          tmem_st32(tmem + kColP + pb * 64 + lane_off + 32, pk + 32);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_ready[pb]);
      }
      // the job's last product (and so all of them) must be done
      const uint32_t t_last = ns - 1;
      if (!ok || !warp_swait(&bars->o_done[t_last & 1], (t_last >> 1) & 1, bars, limit, kSpO)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (HALF)
        finish_half_row<D, BF16>(p, tmem + kColO + lane_off, job.row, h, half, m_used, l);
      else
        finish_row<D, BF16>(p, tmem + kColO + lane_off, job.row, h, m_used, l);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free);
    }
    tc_fence_before();
  } else {
  regs_decrease<kRegsOther>();
  if (warp == 0) {
    // ---------------------------------------------------- Q loads
    const bool leader = elect_one();
    int jobs = 0;
    SJob job;
    for (int jj = static_cast<int>(blockIdx.x); job_of(p, jj, job); jj += step) {
      if (job.n_kv == 0) continue;
      if (jobs > 0 && !warp_swait(&bars->q_empty, (jobs - 1) & 1, bars, limit, kSpEmpty)) break;
      if (leader && !p.debug_withhold_q) {
        mbar_arrive_expect_tx(&bars->q_full, Lay::kChunks * p.q_rows * 128);
#pragma unroll
        for (int c = 0; c < Lay::kChunks; ++c)
          tma_load_3d(sQ + c * Lay::kChunkBytes, &p.tm_q, &bars->q_full, c * 64,
                      job.group * kRows, job.row);
      }
      ++jobs;
    }
    if (jobs > 0 && !p.debug_withhold_q)
      swait(&bars->q_full, (jobs - 1) & 1, bars, limit, kSpDrain, false);
  } else if (warp >= 8) {
    // ------------------------------------------------- key/value gathers
    // Warp w (8..11) copies key rows 32(w-8) .. +31 of every tile, 16 bytes
    // per cp.async, into the 128-byte-swizzled K-major layout the products
    // read (piece q of a 128-byte row r lands at q ^ (r & 7)); lane l loads
    // the index of row +l, and four lanes share each row (see copy_rows), so
    // one warp instruction moves 64 contiguous bytes of each of 8 rows.  Each
    // thread then arrives on the stage's k_full through the copy unit, which
    // fires once that thread's copies have landed: a tile is announced as
    // soon as it is in shared memory, and the gathers never wait for their
    // own copies (the issuing warp fences them for the tensor core's proxy
    // after its wait).
    const int wrow = (warp - 8) * 32;
    const uint8_t* kbase = reinterpret_cast<const uint8_t*>(p.k);
    const uint8_t* vbase = reinterpret_cast<const uint8_t*>(p.v);
    constexpr int kPieces = D / 8;          // 16-byte pieces per row
    RingPos stage, mslot;  // ring stage and key-mask slot of the next tile
    bool ok = true;
    SJob job;
    for (int jj = static_cast<int>(blockIdx.x); ok && job_of(p, jj, job); jj += step) {
      if (job.n_kv == 0) continue;
      const int* irow = p.idx + static_cast<int64_t>(job.row) * p.idx_st;
      auto load_idx = [&](int j) {
        const int ta = j * kKeys + wrow + lane;
        return (ta < job.len) ? __ldg(irow + ta) : -1;
      };
      int na = load_idx(0);
      for (int j = 0; j < job.n_kv; ++j) {
        const int s = stage.idx;
        // an entry past the row's count or outside [0, total_k) reads row 0
        // and is removed by the softmax through the mask
        const bool va = na >= 0 && na < p.total_k;
        const int ra = va ? na : 0;
        const uint32_t ba = __ballot_sync(0xffffffffu, va);
        if (j + 1 < job.n_kv) na = load_idx(j + 1);
        if (stage.lapped) {
          // the stage's previous use, one lap ago
          const uint32_t par = stage.phase ^ 1u;
          if (!warp_swait(&bars->k_empty[s], par, bars, limit, kSpEmpty) ||
              (!p.kv_shared && !warp_swait(&bars->v_empty[s], par, bars, limit, kSpEmpty))) {
            ok = false;
            break;
          }
        }
        if (lane == 0) {
          volatile uint32_t* dst = bars->kmask[mslot.idx];
          dst[warp - 8] = ba;  // keys wrow .. +31
          mbar_arrive(&bars->m_full[mslot.idx]);  // release: the mask is written
        }
        mslot.next(n_slots);
        // Four lanes a row: lane l copies pieces c, c + 4, ... (c = l % 4) of
        // rows l / 4 + 8 i (i < 4), so one instruction moves 64 contiguous
        // bytes of each of 8 rows, the swizzle term (row & 7) = l / 4 is the
        // lane's own, and the lane needs four row indices a tile.
        int64_t roff[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          roff[i] = static_cast<int64_t>(__shfl_sync(0xffffffffu, ra, (lane >> 2) + 8 * i));
        auto copy_rows = [&](const uint8_t* base, int64_t row_bytes, uint8_t* stage) {
          const int c4 = lane & 3, r8 = lane >> 2;
          uint8_t* sdst = stage + (wrow + r8) * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint8_t* gsrc = base + roff[i] * row_bytes + c4 * 16;
#pragma unroll
            for (int pp = 0; pp < kPieces / 4; ++pp) {
              const int q = 4 * pp + c4;  // piece of the row
              cp_async_16(sdst + i * 1024 + (q >> 3) * Lay::kChunkBytes + (((q & 7) ^ r8) << 4),
                          gsrc + pp * 64);
            }
          }
        };
        copy_rows(kbase, p.k_row_bytes, sK + s * Lay::kTileBytes);
        if (!p.kv_shared) copy_rows(vbase, p.v_row_bytes, sV + s * Lay::kTileBytes);
        cp_async_commit();
        cp_async_mbar_arrive_noinc(&bars->k_full[s]);
        stage.next(nst);
      }
    }
    cp_async_wait<0>();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issue
    // The half-row form issues M = 64 products: row r of the 64-row Q tile
    // (and of P, O) lives in TMEM lane 32 (r / 16) + r % 16.
    constexpr uint32_t idS = idesc_f16_f32acc(BF16, false, HALF ? 64 : kRows, kKeys);
    constexpr uint32_t idPV = idesc_f16_f32acc(BF16, true, HALF ? 64 : kRows, D);
    constexpr uint32_t kHi = desc_hi_sw128(1024);
    const uint32_t q_lo = desc_lo_sw128(smem_addr(sQ), 16);
    const uint32_t k_lo = desc_lo_sw128(smem_addr(sK), 16);
    // V rows: their own stages, or the K stage when one kv tensor serves both
    const uint32_t v_lo = desc_lo_sw128(smem_addr(p.kv_shared ? sK : sV), Lay::kChunkBytes);
    bool issued_any = false;
    // Four K-steps per elected issue: S over each 64-column chunk of D (32
    // bytes a step in both operands), PV over each 64-key half of the tile
    // (8 TMEM columns of P and 16 V rows a step).
    auto issue_s = [&](uint32_t buf, int s) {
      const uint32_t b0 = k_lo + static_cast<uint32_t>(s * (Lay::kTileBytes >> 4));
#pragma unroll
      for (int c = 0; c < Lay::kChunks; ++c) {
        const uint32_t off = static_cast<uint32_t>(c * Lay::kChunkBytes) >> 4;
        mma_ss_x4<kHi, kHi>(tmem + kColS0 + buf * 128, q_lo + off, b0 + off, 2u, 2u, idS,
                            c > 0 ? 1u : 0u);
      }
      mma_commit_elect(&bars->s_full[buf]);
    };
    auto issue_pv = [&](int s, uint32_t pb, bool accumulate) {
      const uint32_t b0 = v_lo + static_cast<uint32_t>(s * (Lay::kTileBytes >> 4));
#pragma unroll
      for (int h = 0; h < 2; ++h)
        mma_ts_x4<kHi>(tmem + kColO, tmem + kColP + pb * 64 + h * 32, b0 + h * ((64 * 128) >> 4),
                       8u, (16 * 128) >> 4, idPV, (accumulate || h > 0) ? 1u : 0u);
      mma_commit_elect(&bars->o_done[pb]);
    };
    int g = 0, jobs = 0;
    uint32_t ns = 0;
    RingPos s_pos, pv_pos;  // ring stages of the next S and the next PV
    bool ok = true;
    SJob job;
    // S into the buffer of S(ns).  Its previous contents, S(ns-2), are in
    // the softmax's registers: the loop below waited for P(ns-2), stored
    // after that load, before issuing PV(ns-2), which precedes this issue.
    auto s_next = [&](int s) {
      // the stage's rows were written by the gathers' copies (generic proxy)
      // and are read by the tensor core (async proxy): the k_full wait
      // acquired them, this fence orders them before the products
      fence_proxy_async_smem();
      tc_fence_after();
      issue_s(ns & 1, s);
      if (!p.kv_shared) mma_commit_elect(&bars->k_empty[s]);  // else after PV
      ++ns;
    };
    for (int jj = static_cast<int>(blockIdx.x); ok && job_of(p, jj, job); jj += step) {
      if (job.n_kv == 0) continue;
      if (!warp_swait(&bars->q_full, jobs & 1, bars, limit, kSpQ) ||
          !warp_swait(&bars->k_full[s_pos.idx], s_pos.phase, bars, limit, kSpK))
        break;
      s_next(s_pos.idx);
      s_pos.next(nst);
      issued_any = true;
      if (job.n_kv == 1) mma_commit_elect(&bars->q_empty);
      for (int j = 0; j < job.n_kv; ++j) {
        const int gj = g + j;
        if (j + 1 < job.n_kv) {
          if (!warp_swait(&bars->k_full[s_pos.idx], s_pos.phase, bars, limit, kSpK)) {
            ok = false;
            break;
          }
          s_next(s_pos.idx);
          s_pos.next(nst);
          if (j + 2 == job.n_kv) mma_commit_elect(&bars->q_empty);
        }
        // (V of this stage arrived with its K, waited for before its S)
        const int s = pv_pos.idx;
        if (!warp_swait(&bars->p_ready[gj & 1], (gj >> 1) & 1, bars, limit, kSpP)) {
          ok = false;
          break;
        }
        // The job's first product overwrites O: the previous epilogue must
        // have read it.
        if (j == 0 && jobs > 0 &&
            !warp_swait(&bars->o_free, (jobs - 1) & 1, bars, limit, kSpO)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(s, static_cast<uint32_t>(gj) & 1, j > 0);
        mma_commit_elect(p.kv_shared ? &bars->k_empty[s] : &bars->v_empty[s]);
        pv_pos.next(nst);
      }
      g += job.n_kv;
      ++jobs;
    }
    if (issued_any) {
      mma_commit_elect(&bars->fin);
      swait(&bars->fin, 0, bars, limit, kSpDrain, false);
    }
  }
  }  // warpgroups 0 and 2

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Index preparation: one warp per query row.
__global__ void __launch_bounds__(256) compact_kernel(const sdpa_impl::CompactParams p) {
  const int row = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.total_q) return;
  // Document of this row: the last b with cu_q[b] <= row (offsets assumed
  // nondecreasing; a row outside every document keeps no entry).
  int lo = 0, hi = p.n_docs;  // answer in [0, n_docs)
  while (lo + 1 < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.cu_q + mid) <= row) lo = mid; else hi = mid;
  }
  const int q0 = __ldg(p.cu_q + lo), q1 = __ldg(p.cu_q + lo + 1);
  const bool inside = row >= q0 && row < q1;
  const int pos = row - q0;
  const int k0 = __ldg(p.cu_k + lo);
  const int nk = __ldg(p.cu_k + lo + 1) - k0;
  const int* in = p.idx_local + static_cast<int64_t>(row) * p.in_st;
  int* out = p.idx_global + static_cast<int64_t>(row) * p.out_st;
  int n = 0;
  for (int t0 = 0; t0 < p.topk; t0 += 32) {
    const int t = t0 + lane;
    const int l = (t < p.topk && inside) ? __ldg(in + t) : -1;
    const bool valid = l >= 0 && l < nk && (!p.is_causal || l <= pos);
    const unsigned bal = __ballot_sync(0xffffffffu, valid);
    if (valid) out[n + __popc(bal & ((1u << lane) - 1u))] = k0 + l;
    n += __popc(bal);
  }
  for (int t = n + lane; t < p.topk; t += 32) out[t] = -1;
  if (lane == 0) p.length[row] = n;
}

template <int D, bool BF16, bool HALF>
cudaError_t launch_sparse_one(const sdpa_impl::SparseParams& p, int max_ctas,
                              cudaStream_t stream) {
  auto kern = sparse_fwd_kernel<D, BF16, HALF>;
  constexpr int smem = SLayout<D>::kTotal;
  static bool configured = false;
  if (!configured) {
    // The register split assumes kLaunchRegs per thread at launch; never
    // launch a build where that does not hold (setmaxnreg would wait).
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long jobs = static_cast<long long>(p.total_q) * p.n_groups;
  const unsigned grid = static_cast<unsigned>(jobs < max_ctas ? jobs : max_ctas);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

namespace sdpa_impl {

cudaError_t launch_sparse(const SparseParams& p, int head_dim, bool bf16, int max_ctas,
                          cudaStream_t stream) {
  if (max_ctas < 1) return cudaErrorInvalidValue;
  const bool half = p.q_half != 0;
  if (head_dim == 64) {
    if (half)
      return bf16 ? launch_sparse_one<64, true, true>(p, max_ctas, stream)
                  : launch_sparse_one<64, false, true>(p, max_ctas, stream);
    return bf16 ? launch_sparse_one<64, true, false>(p, max_ctas, stream)
                : launch_sparse_one<64, false, false>(p, max_ctas, stream);
  }
  if (half)
    return bf16 ? launch_sparse_one<128, true, true>(p, max_ctas, stream)
                : launch_sparse_one<128, false, true>(p, max_ctas, stream);
  return bf16 ? launch_sparse_one<128, true, false>(p, max_ctas, stream)
              : launch_sparse_one<128, false, false>(p, max_ctas, stream);
}

cudaError_t launch_compact(const CompactParams& p, cudaStream_t stream) {
  if (p.total_q <= 0) return cudaSuccess;
  const long long threads = static_cast<long long>(p.total_q) * 32;
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  compact_kernel<<<blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t read_and_clear_sparse_status(unsigned int* status) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_sdpa_sparse_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if (*status != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_sdpa_sparse_status, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace sdpa_impl
