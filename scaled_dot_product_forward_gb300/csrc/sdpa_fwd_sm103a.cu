// sdpa_fwd_sm103a.cu -- fused scaled dot-product attention forward for sm_103a,
// head size 128 (head size 64 has its own kernel in sdpa_fwd64_sm103a.cu).
//
// Computes, per (batch, head), out = softmax(scale * Q K^T with causal or
// boolean masking) V: the five-step attention of "Profiling attention in
// PyTorch: kernels, backends and where the time goes" (news.bpdata.com),
// section "Naiv causal attention", evaluated the way that page's "Flash
// backend" section describes -- tiles of K and V streamed past on-chip query
// tiles with an online softmax, so the [seq, seq] score matrix never reaches
// HBM -- but built for Blackwell:
//
//   * persistent: at most one CTA per SM, each walking a static share of
//     the work (sdpa_sched.cuh).  A job is a pair of adjacent 128-row query
//     tiles (A = rows 256m.., B = rows 256m+128..) of one (batch, head); a
//     unit is the causal pair P-1-k followed by pair k of the same head, so
//     every unit costs the same number of key tiles.  The next job's Q load
//     and first S products overlap the previous job's epilogue;
//   * warp 0 streams each job's Q_A, Q_B and one ring of K and V tiles that
//     runs on across jobs, with TMA (128-byte swizzled boxes of 64 x 128
//     elements), K and V with their own full/empty barriers;
//   * warp 1 issues tcgen05.mma (one elected lane) in the order
//       S_A(0) S_B(0) | PV_A(0) S_A(1) PV_B(0) S_B(1) | PV_A(1) S_A(2) ...
//     so that while one softmax warpgroup works on its tile the tensor core
//     is busy with the other tile's products; S = Q K^T lands in TMEM, and
//     P (16-bit, written over S) is read from TMEM by O += P V;
//   * warpgroup 1 owns tile A, warpgroup 2 tile B: one query row per thread
//     (TMEM lane = row), so row max and row sum are in-thread tree
//     reductions with no shuffles; scale, causal / explicit / ragged-tail
//     masks and the online softmax happen in registers, O is rescaled in
//     TMEM only when the running maximum grows by more than 2^8, and the
//     epilogue writes O / l;
//   * explicit masks: each row's 128 bits per key tile come either from the
//     mask bytes (coalesced loads and an in-warp transpose) or, for masked
//     plans, from a per-tile summary that mask_tiles_kernel writes before
//     the forward; with the summary every role skips the key tiles that
//     remove every key for both query tiles of its job.
//
// Safe softmax: a row with no admissible key ends with l = 0 and is written
// as zeros, as the math backend's _safe_softmax does (same page, "Math
// backend" section).  Every barrier wait is bounded in time; on expiry the
// CTA records a status bit in g_sdpa_device_status, stops issuing work,
// drains what it already issued and frees its tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <mutex>

#include "ptx.cuh"
#include "sdpa_internal.h"
#include "sdpa_sched.cuh"

using namespace sdpa_dev;
using namespace sdpa_sched;

// Device status word: bit 0 = some barrier wait ran out of time; the upper
// bits name the wait site.  Read and cleared by sdpa_last_device_status().
__device__ unsigned int g_sdpa_device_status = 0;

// Mask-summary scratch of sdpa_forward_masked_noalloc, for callers that
// cannot allocate device memory: the row bits of up to 32 x 32 tiles (an
// [L, L] mask with L <= 4096), then their class bytes at a fixed offset.
// A file-scope array, so every GPU that loads the library holds these
// 2,098,176 bytes until the process exits; host code gets its device
// address with cudaGetSymbolAddress (sdpa_impl::noalloc_mask_tiles).
static __device__ __align__(256) uint8_t
    g_noalloc_mask_tiles[sdpa_impl::kNoAllocMaxTiles * sdpa_impl::kNoAllocMaxTiles *
                         (128 * 16 + 1)];

namespace {

constexpr int kTilesPerCta = 2;
constexpr int kThreads = 384;  // WG0: TMA warp, MMA warp, 2 spare; WG1: tile A; WG2: tile B
// Register split: the launch reserves kLaunchRegs per thread (the cap that
// __launch_bounds__(384, 1) implies); WG0 gives registers back, the two
// softmax warpgroups take them.  128*80 + 256*208 == 384*168 (the control
// warps keep enough for the persistent job loop's counters).
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kRegsControl = 80;
constexpr uint32_t kRegsSoftmax = 208;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when max grows by > 2^8
constexpr int D = 128;

// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,384), O_B
// [384,512); P_t (16-bit pairs) is written over the first 64 columns of S_t.
__host__ __device__ constexpr uint32_t s_col(int t) { return t ? 128u : 0u; }
__host__ __device__ constexpr uint32_t o_col(int t) { return t ? 256u + D : 256u; }
constexpr uint32_t kTmemCols = 512;

enum WaitSite : unsigned int {
  kSiteQFull = 1u << 1,
  kSiteKFull = 1u << 2,
  kSiteEmpty = 1u << 3,
  kSiteSFull = 1u << 4,
  kSitePReady = 1u << 5,
  kSiteODone = 1u << 6,
  kSiteDrain = 1u << 7,
  kSiteVFull = 1u << 8,
};

struct Layout {
  static constexpr int kChunks = D / 64;               // 128-byte swizzle atoms along D
  static constexpr int kChunkBytes = kBlockM * 128;    // one 128-row x 64-element box
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  // Ring depths: five 32 KB tiles fit beside Q (64 KB).  A stage of K is
  // refilled once S of both tiles has read it and that tile is needed again
  // 2.5 product pairs later, earlier than V (refilled after PV of both
  // tiles, needed three pairs later), so K gets the third stage.
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTilesPerCta * kTileBytes;
  static constexpr int kV = kK + kKStages * kTileBytes;
  static constexpr int kBar = kV + kVStages * kTileBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kTotal = kBar + kBarBytes + 1024;  // + slack for 1 KB alignment
};

constexpr int kMaxStages = 8;
struct Barriers {
  uint64_t q_full;
  uint64_t q_empty;  // the job's Q tiles are no longer read (all its S done)
  uint64_t s_full[kTilesPerCta];
  uint64_t p_ready[kTilesPerCta];
  uint64_t o_done[kTilesPerCta];
  uint64_t o_free[kTilesPerCta];  // the job's O_t read by its epilogue
  uint64_t fin;
  uint64_t k_full[kMaxStages];
  uint64_t v_full[kMaxStages];
  uint64_t k_empty[kMaxStages];
  uint64_t v_empty[kMaxStages];
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(Barriers) <= Layout::kBarBytes, "barrier block too large");
static_assert(Layout::kTotal <= 227 * 1024, "shared memory over the per-CTA limit");
static_assert(Layout::kKStages <= kMaxStages && Layout::kVStages <= kMaxStages, "ring");

// Bounded wait on one barrier phase (sdpa_sched::wait_phase with this CTA's
// abort flag and this kernel's status word).
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, Barriers* bars,
                                           uint64_t limit_ns, unsigned int site,
                                           bool honour_abort = true) {
  return sdpa_sched::wait_phase(bar, parity, &bars->abort_flag, &g_sdpa_device_status, limit_ns,
                                site, honour_abort);
}

// Warp-uniform version: every lane polls, and the warp proceeds only if all
// lanes saw the phase complete (keeps later .sync.aligned ops convergent).
__device__ __forceinline__ bool warp_wait_phase(uint64_t* bar, uint32_t parity, Barriers* bars,
                                                uint64_t limit_ns, unsigned int site) {
  const bool ok = wait_phase(bar, parity, bars, limit_ns, site);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------ softmax role
// One warpgroup, one query tile: thread r of the group owns row r (TMEM lane r).
// Both warpgroups run this one code path (t picks the tile at run time), so
// the warps sharing an SM sub-partition also share instruction-cache lines.
// Phase counters that run across the jobs of a persistent CTA (every
// barrier's phases are consumed strictly in order).
struct SoftmaxCounters {
  uint32_t s_seen;   // completions of s_full[t] consumed
  uint32_t o_seen;   // completions of o_done[t] consumed
};

// One job of one tile.  Returns false when a wait gave up.
template <int MODE, bool BF16>
__device__ __forceinline__ bool softmax_job(const sdpa_impl::FwdParams& p, const Work<2>& w, int t,
                                            Barriers* bars, uint32_t tmem, int wq, int lane,
                                            SoftmaxCounters& cnt) {
  const int n = w.n_kv(t);
  const int qt = w.tile(t);
  if (n == 0) {
    if constexpr (MODE == sdpa_impl::kMaskExplicit) {
      // A present tile whose job visits no key tile: every key of every
      // row is removed, so the rows are zeros (and log-sum-exp -inf).
      const int row_z = qt * kBlockM + wq * 32 + lane;
      if (p.tile_class != nullptr && qt < p.n_tiles && row_z < w.len) {
        if (p.lse != nullptr)
          p.lse[w.batch * p.lse_sb + w.head * p.lse_sh +
                static_cast<int64_t>(w.row0 + row_z) * p.lse_sl] = -INFINITY;
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) +
                                              w.batch * p.o_sb + w.head * p.o_sh +
                                              static_cast<int64_t>(w.row0 + row_z) * p.o_sl);
#pragma unroll
        for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return true;
  }
  const uint64_t limit = p.wait_limit_ns;
  const uint32_t tS_base = tmem + (t ? s_col(1) : s_col(0));
  const uint32_t tO_base = tmem + (t ? o_col(1) : o_col(0));
  const int r = wq * 32 + lane;
  const int row_g = qt * kBlockM + r;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tS_base + lane_off;
  const uint32_t tO = tO_base + lane_off;
  const uint32_t tP = tS;  // P_j is written over the first 64 columns of S_j
  const float sl2 = p.scale_log2;
  const bool pos_scale = sl2 >= 0.0f;
  const float mval = pos_scale ? -INFINITY : INFINITY;  // a removed raw score
  float m_used = -INFINITY;  // running max actually used in the exponentials
  float l = 0.0f;            // running row sum of probabilities
  bool ok = true;
  KeyTileCursor kc{-1, 0u};
  // With a tile summary the next visited tile and this row's 128 bits of it
  // are fetched one tile ahead, so the load's latency overlaps a whole tile
  // of work instead of the wait for S.  (A tile that removes nothing has
  // zero bits and skips the select below.)
  int kt_next = next_key_tile<MODE, 2>(p, w, kc, 0);
  uint4 bits_next = make_uint4(0u, 0u, 0u, 0u);
  const uint4* tile_bits_row = nullptr;
  if constexpr (MODE == sdpa_impl::kMaskExplicit) {
    if (p.tile_class != nullptr) {
      tile_bits_row = p.tile_bits + static_cast<int64_t>(qt) * p.n_tiles * kBlockM + r;
      bits_next = __ldg(tile_bits_row + static_cast<int64_t>(kt_next) * kBlockM);
    }
  }

  for (int j = 0; j < n; ++j) {
    const int kt = kt_next;
    if (tile_bits_row == nullptr) kt_next = j + 1;  // every key tile in order
    const int col0 = kt * kBlockN;
    const bool tail = col0 + kBlockN > w.len;
    bool masked_tile = tail || (MODE == sdpa_impl::kMaskCausal && j == qt);
    // Explicit mask: this row's 128 mask bytes for tile j, one bit per key
    // (bit set = removed).  Loaded before waiting for S so their latency
    // hides behind the score MMA.
    uint32_t mbits[kBlockN / 32];
    if constexpr (MODE == sdpa_impl::kMaskExplicit) {
      if (tile_bits_row != nullptr) {
        // Tile summary: the bits fetched during the previous tile (a warp
        // reads 512 contiguous bytes), and the next tile's now.
        mbits[0] = bits_next.x;
        mbits[1] = bits_next.y;
        mbits[2] = bits_next.z;
        mbits[3] = bits_next.w;
        if (j + 1 < n) {
          kt_next = next_key_tile<MODE, 2>(p, w, kc, j + 1);
          bits_next = __ldg(tile_bits_row + static_cast<int64_t>(kt_next) * kBlockM);
        }
      } else {
        mask_bits_from_bytes(p, w.len, row_g, lane, col0, mbits);
      }
      // A tile where none of this warp's 32 rows removes a key needs no
      // per-element select (warp-uniform, so structured masks skip it).
      masked_tile = masked_tile ||
                    __any_sync(0xffffffffu, (mbits[0] | mbits[1] | mbits[2] | mbits[3]) != 0u);
    }
    if (!warp_wait_phase(&bars->s_full[t], cnt.s_seen & 1, bars, limit, kSiteSFull)) {
      ok = false;
      break;
    }
    ++cnt.s_seen;
    tc_fence_after();
    float s[kBlockN];
    {
      uint32_t su[kBlockN];
#pragma unroll
      for (int c = 0; c < kBlockN / 32; ++c) tmem_ld32(tS + c * 32, su + c * 32);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < kBlockN; ++c) s[c] = __uint_as_float(su[c]);
    }
    if (masked_tile) {
      if constexpr (MODE == sdpa_impl::kMaskExplicit) {
#pragma unroll
        for (int c = 0; c < kBlockN; ++c)
          s[c] = ((mbits[c >> 5] >> (c & 31)) & 1u) ? mval : s[c];
      } else {
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) {
          const bool removed =
              (col0 + c >= w.len) || (MODE == sdpa_impl::kMaskCausal && col0 + c > row_g);
          s[c] = removed ? mval : s[c];
        }
      }
    }

    // Row extremum of the raw scores (max for a positive scale): eight
    // independent chains of three-input max, then a short tree.
    float e8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e8[i] = s[i];
    if (pos_scale) {
#pragma unroll
      for (int c = 8; c < kBlockN; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) e8[i] = max3f(e8[i], s[c + i], s[c + 8 + i < kBlockN ? c + 8 + i : c + i]);
      e8[0] = max3f(e8[0], e8[1], e8[2]);
      e8[3] = max3f(e8[3], e8[4], e8[5]);
      e8[6] = fmaxf(e8[6], e8[7]);
      e8[0] = max3f(e8[0], e8[3], e8[6]);
    } else {
#pragma unroll
      for (int c = 8; c < kBlockN; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) e8[i] = min3f(e8[i], s[c + i], s[c + 8 + i < kBlockN ? c + 8 + i : c + i]);
      e8[0] = min3f(e8[0], e8[1], e8[2]);
      e8[3] = min3f(e8[3], e8[4], e8[5]);
      e8[6] = fminf(e8[6], e8[7]);
      e8[0] = min3f(e8[0], e8[3], e8[6]);
    }
    const float ext = e8[0];
    const float m_tile = (ext == mval) ? -INFINITY : ext * sl2;
    const bool need = m_tile > m_used + kRescaleLog2;
    float alpha = 1.0f;
    if (need) {
      alpha = ex2(m_used - m_tile);  // 0 when nothing was admitted before
      m_used = m_tile;
      l *= alpha;
    }
    const float neg_m = (m_used == -INFINITY) ? 0.0f : -m_used;

    // Three passes over the row so each pass is a long run of independent
    // instructions: x = s * scale*log2(e) - m (packed FMA), p = 2^x, then the
    // packed row sums and the 16-bit packing.  A removed score is +-inf with
    // the sign that makes x = -inf, so its probability is exactly 0 (the
    // multiplier is never 0: the host maps a zero scale to +-FLT_MIN, which
    // gives the same all-ones weights).
#pragma unroll
    for (int c = 0; c < kBlockN; c += 2) fma2_bcast(s[c], s[c + 1], s[c], s[c + 1], sl2, neg_m);
#pragma unroll
    for (int c = 0; c < kBlockN; ++c) s[c] = ex2(s[c]);
    uint32_t pk[kBlockN / 2];
    float rs[8];  // four packed pairs of partial row sums
#pragma unroll
    for (int i = 0; i < 8; ++i) rs[i] = 0.0f;
#pragma unroll
    for (int c = 0; c < kBlockN / 2; ++c) {
      add2_acc(rs[2 * (c & 3)], rs[2 * (c & 3) + 1], s[2 * c], s[2 * c + 1]);
      pk[c] = pack2<BF16>(s[2 * c], s[2 * c + 1]);
    }
    add2_acc(rs[0], rs[1], rs[2], rs[3]);
    add2_acc(rs[4], rs[5], rs[6], rs[7]);
    add2_acc(rs[0], rs[1], rs[4], rs[5]);
    l += rs[0] + rs[1];

    if (j > 0) {
      // PV_{j-1} must have completed before O is rescaled or P_j replaces
      // P_{j-1}: S_j was issued after PV_{j-1} and the tensor pipe completes
      // in issue order, so s_full(j) already implies it -- that phase of
      // o_done is complete and is only counted here.
      ++cnt.o_seen;
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
          float* of = reinterpret_cast<float*>(o);
#pragma unroll
          for (int e = 0; e < 32; e += 2) mul2_bcast(of[e], of[e + 1], alpha);
          tmem_st32(tO + c * 32, o);
        }
      }
    }
    // P_j goes into the first 64 columns of this tile's score buffer (free
    // again: PV_{j-1} has completed, see above).
    tmem_st32(tP + 0, pk);
    tmem_st32(tP + 32, pk + 32);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->p_ready[t]);  // one arrival per warp
  }

  if (ok && !warp_wait_phase(&bars->o_done[t], cnt.o_seen & 1, bars, limit, kSiteODone))
    ok = false;
  if (ok) {
    ++cnt.o_seen;
    tc_fence_after();
    const float inv_l = (l > 0.0f) ? (1.0f / l) : 0.0f;
    if (p.lse != nullptr && row_g < w.len) {
      // log(sum_j exp(scale * s_j)) = ln(l) + m_used * ln(2): l sums 2^(x - m_used).
      constexpr float kLn2 = 0.693147180559945309f;
      p.lse[w.batch * p.lse_sb + w.head * p.lse_sh +
            static_cast<int64_t>(w.row0 + row_g) * p.lse_sl] =
          (l > 0.0f) ? (log2f(l) + m_used) * kLn2 : -INFINITY;
    }
    uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + w.batch * p.o_sb + w.head * p.o_sh +
                     static_cast<int64_t>(w.row0 + row_g) * p.o_sl;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + c * 32, o);
      tmem_ld_wait();
      uint32_t pw[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pw[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l,
                            __uint_as_float(o[2 * e + 1]) * inv_l);
      if (row_g < w.len) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(pw[4 * v], pw[4 * v + 1], pw[4 * v + 2], pw[4 * v + 3]);
      }
    }
    // O_t has been read: the next job's first PV may overwrite it.
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->o_free[t]);
  }
  tc_fence_before();
  return ok;
}

// ------------------------------------------------------------------ kernel
template <int MODE, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    sdpa_fwd_kernel(const __grid_constant__ sdpa_impl::FwdParams p) {
  using Lay = Layout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + Lay::kQ;
  uint8_t* sK = smem + Lay::kK;
  uint8_t* sV = smem + Lay::kV;
  Barriers* bars = reinterpret_cast<Barriers*>(smem + Lay::kBar);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
#pragma unroll
    for (int t = 0; t < kTilesPerCta; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_ready[t], kBlockM / 32);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_free[t], kBlockM / 32);
    }
    mbar_init(&bars->fin, 1);
#pragma unroll
    for (int s = 0; s < Lay::kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
#pragma unroll
    for (int s = 0; s < Lay::kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.tm_q);
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Everything above (barrier set-up, TMEM allocation, descriptor prefetch)
  // may overlap the previous kernel in the stream; nothing below touches
  // global memory before that kernel has completed.
  grid_dependency_wait();
  grid_launch_dependents();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tS[kTilesPerCta] = {tmem + s_col(0), tmem + s_col(1)};
  const uint32_t tO[kTilesPerCta] = {tmem + o_col(0), tmem + o_col(1)};

  if (warp >= 4) {
    // ------------------------------------------- softmax / output warps
    regs_increase<kRegsSoftmax>();
    // warps 4..7 -> tile A, 8..11 -> tile B; the same jobs as the other roles
    const int t = (warp - 4) >> 2;
    SoftmaxCounters cnt{0, 0};
    for_each_job<MODE, VARLEN, kTilesPerCta>(p, [&](const Work<kTilesPerCta>& w) {
      return softmax_job<MODE, BF16>(p, w, t, bars, tmem, warp & 3, lane, cnt);
    });
  } else {
    regs_decrease<kRegsControl>();
  // Both control warps run their loops with all 32 lanes, so loop variables
  // and descriptors stay warp-uniform; one elected lane issues each TMA copy,
  // MMA and commit.  (Issuing from a lane-0-only branch costs about 2.5x more
  // per tcgen05.mma and starves the tensor core.)
  const bool leader = elect_one();
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    // Key/value tiles issued so far over all jobs (ring position) and jobs
    // whose Q was loaded; a give-up drains what was issued.
    int g = 0, k_end = 0, v_end = 0, jobs = 0;
    for_each_job<MODE, VARLEN, kTilesPerCta>(p, [&](const Work<kTilesPerCta>& w) -> bool {
      if (w.n_kv_max == 0) return true;  // masked out entirely: nothing to load
      // The previous job's Q must be consumed (all its S products done).
      if (jobs > 0 && !warp_wait_phase(&bars->q_empty, (jobs - 1) & 1, bars, limit, kSiteEmpty))
        return false;
      if (!p.debug_withhold_q && leader) {
        const int nq = w.n_present;
        mbar_arrive_expect_tx(&bars->q_full, nq * Lay::kTileBytes);
        for (int t = 0; t < nq; ++t)
#pragma unroll
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_tile(sQ + t * Lay::kTileBytes + c * Lay::kChunkBytes, &p.tm_q, &bars->q_full,
                     c * 64, w.row0 + w.tile(t) * kBlockM, w.head, w.batch, p.pos_q);
      }
      ++jobs;
      // Key tiles in order; with a mask summary every tile is examined and
      // the ones the job does not visit are passed over.
      const bool summary = MODE == sdpa_impl::kMaskExplicit && p.tile_class != nullptr;
      const int n_scan = summary ? p.n_tiles : w.n_kv_max;
      uint32_t visit = 0xffffffffu;
      for (int kt = 0; kt < n_scan; ++kt) {
        if (summary) {
          if ((kt & 31) == 0) visit = visit_chunk<kTilesPerCta>(p, w, kt >> 5);
          if (((visit >> (kt & 31)) & 1u) == 0u) continue;
        }
        const int s = g % Lay::kKStages;
        const int use = g / Lay::kKStages;
        if (use > 0 &&
            !warp_wait_phase(&bars->k_empty[s], (use - 1) & 1, bars, limit, kSiteEmpty))
          return false;
        if (leader) {
          mbar_arrive_expect_tx(&bars->k_full[s], Lay::kTileBytes);
#pragma unroll
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_tile(sK + s * Lay::kTileBytes + c * Lay::kChunkBytes, &p.tm_k, &bars->k_full[s],
                     c * 64, w.row0 + kt * kBlockN, w.head, w.batch, p.pos_k);
        }
        k_end = g + 1;
        const int sv = g % Lay::kVStages;
        const int use_v = g / Lay::kVStages;
        if (use_v > 0 &&
            !warp_wait_phase(&bars->v_empty[sv], (use_v - 1) & 1, bars, limit, kSiteEmpty))
          return false;
        if (leader) {
          mbar_arrive_expect_tx(&bars->v_full[sv], Lay::kTileBytes);
#pragma unroll
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_tile(sV + sv * Lay::kTileBytes + c * Lay::kChunkBytes, &p.tm_v, &bars->v_full[sv],
                     c * 64, w.row0 + kt * kBlockN, w.head, w.batch, p.pos_v);
        }
        v_end = g + 1;
        ++g;
      }
      return true;
    });
    // Drain: every load issued must have landed before shared memory is
    // released (only matters when a wait gave up).  The last tile issued into
    // a stage is the largest index below the end with that stage.
    for (int j = max(0, k_end - Lay::kKStages); j < k_end; ++j)
      wait_phase(&bars->k_full[j % Lay::kKStages], (j / Lay::kKStages) & 1, bars, limit,
                 kSiteDrain, false);
    for (int j = max(0, v_end - Lay::kVStages); j < v_end; ++j)
      wait_phase(&bars->v_full[j % Lay::kVStages], (j / Lay::kVStages) & 1, bars, limit,
                 kSiteDrain, false);
    if (jobs > 0 && !p.debug_withhold_q)
      wait_phase(&bars->q_full, (jobs - 1) & 1, bars, limit, kSiteDrain, false);
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = idesc_f16_f32acc(BF16, false, kBlockM, kBlockN);
    constexpr uint32_t idPV = idesc_f16_f32acc(BF16, true, kBlockM, D);
    // Descriptor low words of the Q, K and V bases; every operand of every
    // MMA below is one of these plus a compile-time or per-stage offset.
    constexpr uint32_t kHiKMajor = desc_hi_sw128(1024);  // 8-row groups 1 KB apart
    constexpr uint32_t kHiV = desc_hi_sw128(1024);
    const uint32_t q_lo = desc_lo_sw128(smem_addr(sQ), 16);
    const uint32_t k_lo = desc_lo_sw128(smem_addr(sK), 16);
    // V is MN-major: its 64-wide chunks of D are one box apart (LBO).
    const uint32_t v_lo = desc_lo_sw128(smem_addr(sV), Lay::kChunkBytes);
    bool issued_any = false;

    // S_t = Q_t K^T from key stage s.
    auto issue_s = [&](int t, int s) {
      const uint32_t a0 = q_lo + static_cast<uint32_t>(t * (Lay::kTileBytes >> 4));
      const uint32_t b0 = k_lo + static_cast<uint32_t>(s * (Lay::kTileBytes >> 4));
      const uint32_t d = t ? tS[1] : tS[0];
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        // chunk of D (kk / 4), then 16 elements = 32 B inside the atom
        const uint32_t off = ((kk >> 2) * Lay::kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ss_elect<kHiKMajor, kHiKMajor>(d, a0 + off, b0 + off, idS, kk > 0 ? 1u : 0u);
      }
      mma_commit_elect(&bars->s_full[t]);
    };
    // O_t (+)= P_t V from value stage s, P_t read from TMEM (keys 2c, 2c+1 in column c).
    auto issue_pv = [&](int t, int s, bool accumulate) {
      const uint32_t b0 = v_lo + static_cast<uint32_t>(s * (Lay::kTileBytes >> 4));
      const uint32_t d = t ? tO[1] : tO[0];
      const uint32_t a = t ? tS[1] : tS[0];  // P_t over the first 64 columns of S_t
#pragma unroll
      for (int kk = 0; kk < kBlockN / 16; ++kk) {
        // keys kk*16 .. +16: 16 rows of 128 B
        mma_ts_elect<kHiV>(d, a + kk * 8, b0 + ((kk * 16 * 128) >> 4), idPV,
                           (accumulate || kk > 0) ? 1u : 0u);
      }
      mma_commit_elect(&bars->o_done[t]);
    };

    // Running counters over all jobs: ring position g, jobs done, P-ready
    // phases consumed per tile and jobs per tile (for o_free).
    int g = 0, jobs = 0;
    uint32_t p_seen[kTilesPerCta] = {0, 0}, t_jobs[kTilesPerCta] = {0, 0};
    for_each_job<MODE, VARLEN, kTilesPerCta>(p, [&](const Work<kTilesPerCta>& w) -> bool {
      if (w.n_kv_max == 0) return true;  // masked out entirely: no products
      if (!warp_wait_phase(&bars->q_full, jobs & 1, bars, limit, kSiteQFull) ||
          !warp_wait_phase(&bars->k_full[g % Lay::kKStages], (g / Lay::kKStages) & 1, bars, limit,
                           kSiteKFull))
        return false;
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < kTilesPerCta; ++t) {
        if (w.n_kv(t) == 0) continue;
        issue_s(t, g % Lay::kKStages);
      }
      mma_commit_elect(&bars->k_empty[g % Lay::kKStages]);
      if (w.n_kv_max == 1) mma_commit_elect(&bars->q_empty);  // that was the job's last S
      issued_any = true;

      // The first PV_t of a job overwrites O_t: the previous job's epilogue
      // must have read it.
      auto pv_ready = [&](int t, int j) -> bool {
        if (!warp_wait_phase(&bars->p_ready[t], p_seen[t] & 1, bars, limit, kSitePReady))
          return false;
        ++p_seen[t];
        if (j == 0 && t_jobs[t] > 0 &&
            !warp_wait_phase(&bars->o_free[t], (t_jobs[t] - 1) & 1, bars, limit, kSiteODone))
          return false;
        tc_fence_after();
        return true;
      };

      bool ok = true;
      for (int j = 0; j < w.n_kv_max && ok; ++j) {
        const int gj = g + j;
        const int s = gj % Lay::kVStages;   // V(j)
        const int s1 = (gj + 1) % Lay::kKStages;  // K(j+1)
        const uint32_t ph1 = ((gj + 1) / Lay::kKStages) & 1;
        bool k_next = false;
        {
          if (!warp_wait_phase(&bars->v_full[s], (gj / Lay::kVStages) & 1, bars, limit,
                               kSiteVFull)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int t = 0; t < kTilesPerCta; ++t) {
            if (j >= w.n_kv(t)) continue;
            if (!pv_ready(t, j)) {
              ok = false;
              break;
            }
            issue_pv(t, s, j > 0);
            if (j + 1 < w.n_kv(t)) {
              if (!k_next) {
                if (!warp_wait_phase(&bars->k_full[s1], ph1, bars, limit, kSiteKFull)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                k_next = true;
              }
              issue_s(t, s1);
            }
          }
          if (!ok) break;
          mma_commit_elect(&bars->v_empty[s]);
          if (k_next) mma_commit_elect(&bars->k_empty[s1]);
          if (j + 2 == w.n_kv_max) mma_commit_elect(&bars->q_empty);  // job's last S issued
        }
      }
      if (!ok) return false;
      g += w.n_kv_max;
      ++jobs;
#pragma unroll
      for (int t = 0; t < kTilesPerCta; ++t)
        if (w.n_kv(t) > 0) ++t_jobs[t];
      return true;
    });
    if (issued_any) {
      // Everything issued must finish before TMEM is released.
      mma_commit_elect(&bars->fin);
      wait_phase(&bars->fin, 0, bars, limit, kSiteDrain, false);
    }
  }
  }  // control warpgroup

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE, bool BF16, bool VARLEN>
cudaError_t launch_one(const sdpa_impl::FwdParams& p, int max_ctas, cudaStream_t stream) {
  auto kern = sdpa_fwd_kernel<MODE, BF16, VARLEN>;
  constexpr int smem = Layout::kTotal;
  static bool configured = false;  // one attribute call per instantiation
  if (!configured) {
    // The in-kernel register split assumes the launch reserves kLaunchRegs
    // per thread; never launch a build where that does not hold (the
    // softmax warpgroups would wait forever for registers).
    cudaFuncAttributes attr{};
    cudaError_t e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  // Persistent grid: one CTA per SM at most, each walking its share of the
  // equal-cost units.
  const unsigned grid = grid_size<kTilesPerCta>(p, VARLEN, max_ctas);
  // Programmatic dependent launch: this grid's set-up may start while the
  // previous kernel in the stream drains; the kernel waits for it
  // (griddepcontrol.wait) before its first global-memory access.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
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

template <bool BF16>
cudaError_t launch_mode(const sdpa_impl::FwdParams& p, int mode, int max_ctas,
                        cudaStream_t stream) {
  if (p.cu_seqlens != nullptr) {  // packed sequences: causal or no mask
    if (mode == sdpa_impl::kMaskExplicit) return cudaErrorInvalidValue;
    return mode == sdpa_impl::kMaskCausal
               ? launch_one<sdpa_impl::kMaskCausal, BF16, true>(p, max_ctas, stream)
               : launch_one<sdpa_impl::kMaskNone, BF16, true>(p, max_ctas, stream);
  }
  switch (mode) {
    case sdpa_impl::kMaskCausal:
      return launch_one<sdpa_impl::kMaskCausal, BF16, false>(p, max_ctas, stream);
    case sdpa_impl::kMaskExplicit:
      return launch_one<sdpa_impl::kMaskExplicit, BF16, false>(p, max_ctas, stream);
    default:
      return launch_one<sdpa_impl::kMaskNone, BF16, false>(p, max_ctas, stream);
  }
}

// Mask summary: CTA (kt, qt) reads 128 x 128 tile of the byte mask once
// (16-byte loads, eight threads per 128-byte row segment), writes its rows
// as bits (keys and rows past L as removed) and classifies the tile by the
// entries inside [L, L].
__global__ void __launch_bounds__(256) mask_tiles_kernel(const sdpa_impl::MaskTilesParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int kt = static_cast<int>(blockIdx.x), qt = static_cast<int>(blockIdx.y);
  const int tid = static_cast<int>(threadIdx.x);
  const int col = kt * kBlockN + 16 * (tid & 7);
  uint16_t* dst = p.bits + (static_cast<int64_t>(qt) * p.n_tiles + kt) * (kBlockM * 8);
  bool any_removed = false, any_kept = false;
#pragma unroll
  for (int i = 0; i < kBlockM / 32; ++i) {
    const int r = i * 32 + (tid >> 3);
    const int row = qt * kBlockM + r;
    uint32_t bits = 0xffffu;
    if (row < p.L) {
      const uint8_t* src = p.mask + static_cast<int64_t>(row) * p.L + col;
      if (p.vec16 && col + 16 <= p.L) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(src));
        bits = nonzero_byte_bits(x.x) | (nonzero_byte_bits(x.y) << 4) |
               (nonzero_byte_bits(x.z) << 8) | (nonzero_byte_bits(x.w) << 12);
        any_removed = any_removed || bits != 0u;
        any_kept = any_kept || bits != 0xffffu;
      } else {
        bits = 0u;
        for (int b = 0; b < 16; ++b) {
          const bool in = col + b < p.L;
          const bool removed = !in || __ldg(src + b) != 0;
          bits |= (removed ? 1u : 0u) << b;
          if (in) {
            any_removed = any_removed || removed;
            any_kept = any_kept || !removed;
          }
        }
      }
    }
    dst[r * 8 + (tid & 7)] = static_cast<uint16_t>(bits);
  }
  const int removed = __syncthreads_or(any_removed ? 1 : 0);
  const int kept = __syncthreads_or(any_kept ? 1 : 0);
  if (tid == 0)
    p.tile_class[static_cast<int64_t>(qt) * p.n_tiles + kt] =
        !removed ? sdpa_impl::kTileKept : (!kept ? sdpa_impl::kTileRemoved : sdpa_impl::kTileMixed);
}

}  // namespace

namespace sdpa_impl {

cudaError_t launch_mask_tiles(const MaskTilesParams& p, cudaStream_t stream) {
  if (p.n_tiles < 1 || p.n_tiles > 65535) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.n_tiles), static_cast<unsigned>(p.n_tiles), 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mask_tiles_kernel, p);
}

cudaError_t launch_forward(const FwdParams& p, int head_dim, int mask_mode, bool bf16,
                           int max_ctas, cudaStream_t stream) {
  if (max_ctas < 1) return cudaErrorInvalidValue;
  if (head_dim == 64) return launch_forward64(p, mask_mode, bf16, max_ctas, stream);
  return bf16 ? launch_mode<true>(p, mask_mode, max_ctas, stream)
              : launch_mode<false>(p, mask_mode, max_ctas, stream);
}

cudaError_t noalloc_mask_tiles(int device, const uint4** tile_bits,
                               const uint8_t** tile_class) {
  // One cached device address per device, found the first time a device
  // asks (with that device current, as cudaGetSymbolAddress requires) and
  // found again whenever the device's current context is a different one:
  // after cudaDeviceReset the runtime creates a new primary context and
  // loads the module again, and the old address no longer maps anything.
  // Contexts are told apart by their process-unique ids (cuCtxGetId).
  using CtxGetCurrentFn = CUresult (*)(CUcontext*);
  using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static std::once_flag once;
  static CtxGetCurrentFn ctx_current = nullptr;
  static CtxGetIdFn ctx_id = nullptr;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  static std::mutex mu;
  static void* addr[kNoAllocMaxDevices] = {};
  static unsigned long long addr_ctx[kNoAllocMaxDevices] = {};
  if (device < 0 || device >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  if (ctx_current == nullptr || ctx_id == nullptr) return cudaErrorNotSupported;
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return e;
  if (cur != device) return cudaErrorInvalidDevice;
  // The id of the context the runtime has made current for this device; 0
  // when there is none yet (no runtime call has needed it so far) or the
  // handle left current no longer names a live context.
  auto current_id = [&]() -> unsigned long long {
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || ctx_id(ctx, &id) != CUDA_SUCCESS)
      return 0;
    return id;
  };
  unsigned long long id = current_id();
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr || id == 0 || addr_ctx[device] != id) {
    // cudaGetSymbolAddress also makes the device's primary context current
    // (creating it after a reset), so the id is read again afterwards.
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_mask_tiles);
    if (e != cudaSuccess) return e;
    id = current_id();
    if (id == 0) return cudaErrorDeviceUninitialized;
    addr[device] = ptr;
    addr_ctx[device] = id;
  }
  *tile_bits = static_cast<const uint4*>(addr[device]);
  *tile_class = static_cast<const uint8_t*>(addr[device]) +
                static_cast<size_t>(kNoAllocMaxTiles) * kNoAllocMaxTiles * kBlockM * 16;
  return cudaSuccess;
}

cudaError_t read_and_clear_device_status(cudaStream_t stream, unsigned int* status) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(status, g_sdpa_device_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if (*status != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_sdpa_device_status, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace sdpa_impl
