// sdpa_fwd64_sm103a.cu -- fused scaled dot-product attention forward for sm_103a,
// head size 64.
//
// The same computation as the head-size-128 kernel (the five-step attention
// of "Profiling attention in PyTorch: kernels, backends and where the time
// goes", news.bpdata.com, section "Naiv causal attention", evaluated with an
// online softmax over K/V tiles as that page's "Flash backend" section
// describes), with the tile plan chosen for D = 64 -- the per-shape choice
// that page credits for the cuDNN backend's speed (section "cuDNN backend"):
//
//   * two 128-row query tiles per job (sdpa_sched.cuh), 128-key K/V tiles;
//   * TMEM: with D = 64 the two output accumulators take 128 columns, which
//     leaves room for P in its own buffers -- S_A [0,128), S_B [128,256),
//     O_A [256,320), O_B [320,384), P_A [384,448), P_B [448,512) -- so
//     S(j+1) of a tile is issued as soon as its softmax has loaded S(j)
//     into registers, and the softmax runs tile after tile without waiting
//     for its own products;
//   * one MMA-issuing warp per tile (warp 1: tile A, warp 2: tile B).  At
//     D = 64 a tile's products per key tile are short (S 128x128x64 and PV
//     128x64x128), and a single issuing warp's fixed cost per tile (barrier
//     checks, fences, commits, the issue itself, sharing its SM
//     sub-partition with softmax warps) left the tensor core idle between
//     them.  Each warp issues its tile's S and PV four MMAs per elected
//     issue, and both commit to the shared ring, Q and drain barriers;
//   * warp 0 streams Q and rings of six K and six V tiles (16 KB each).
//
// Explicit masks, safe softmax, bounded waits: as in the head-size-128
// kernel; this translation unit has its own status word, g_sdpa64_status.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sdpa_internal.h"
#include "sdpa_sched.cuh"

using namespace sdpa_dev;
using namespace sdpa_sched;

// Device status word of this kernel: bit 0 = some barrier wait ran out of
// time; the upper bits name the wait site (same bits as the D = 128 kernel).
__device__ unsigned int g_sdpa64_status = 0;

namespace {

constexpr int D = 64;
constexpr int kTilesPerCta = 2;
constexpr int kMmaWarps = kTilesPerCta;  // warp 1 + t issues tile t's products
constexpr int kThreads = 384;  // WG0: TMA warp, two MMA warps, 1 spare; WG1: tile A; WG2: tile B
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kRegsControl = 80;
constexpr uint32_t kRegsSoftmax = 208;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when max grows by > 2^8

__host__ __device__ constexpr uint32_t s_col(int t) { return t ? 128u : 0u; }
__host__ __device__ constexpr uint32_t o_col(int t) { return t ? 256u + D : 256u; }
__host__ __device__ constexpr uint32_t p_col(int t) { return t ? 256u + 2 * D + 64 : 256u + 2 * D; }
static_assert(256 + 2 * D + 128 <= 512, "TMEM plan exceeds 512 columns");
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
  kSiteSFree = 1u << 9,
};

struct Layout {
  static constexpr int kTileBytes = kBlockM * 128;  // 128 rows x 64 elements (one box)
  static constexpr int kStages = 6;                 // K ring and V ring depth
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTilesPerCta * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBar = kV + kStages * kTileBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kTotal = kBar + kBarBytes + 1024;  // + slack for 1 KB alignment
};

struct Barriers {
  uint64_t q_full;
  uint64_t q_empty;  // the job's Q tiles are no longer read (all its S done)
  uint64_t s_full[kTilesPerCta];
  uint64_t s_free[kTilesPerCta];  // S_t(j) loaded by the softmax: S_t(j+1) may overwrite it
  uint64_t p_ready[kTilesPerCta];
  uint64_t o_done[kTilesPerCta];
  uint64_t o_free[kTilesPerCta];  // the job's O_t read by its epilogue
  uint64_t fin;
  uint64_t k_full[Layout::kStages];
  uint64_t v_full[Layout::kStages];
  uint64_t k_empty[Layout::kStages];
  uint64_t v_empty[Layout::kStages];
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(Barriers) <= Layout::kBarBytes, "barrier block too large");
static_assert(Layout::kTotal <= 227 * 1024, "shared memory over the per-CTA limit");

__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, Barriers* bars,
                                           uint64_t limit_ns, unsigned int site,
                                           bool honour_abort = true) {
  return sdpa_sched::wait_phase(bar, parity, &bars->abort_flag, &g_sdpa64_status, limit_ns, site,
                                honour_abort);
}

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
__device__ __forceinline__ bool softmax_job(const sdpa_impl::FwdParams& p, const Work<kTilesPerCta>& w, int t,
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
  const uint32_t tP_base = tmem + (t ? p_col(1) : p_col(0));
  const int r = wq * 32 + lane;
  const int row_g = qt * kBlockM + r;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tS_base + lane_off;
  const uint32_t tO = tO_base + lane_off;
  const uint32_t tP = tP_base + lane_off;  // P_j in its own 64 columns
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
    // S(j) is in registers: the MMA warp may overwrite it with S(j+1).
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->s_free[t]);
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
      // P_{j-1}.  S_j may have been issued before PV_{j-1}, so its phase is
      // waited for here, in order and BEFORE the p_ready arrival below: once
      // P_j is released PV_j may complete too, and a parity wait that falls
      // two phases behind its barrier would block until the next phase (a
      // timeout) instead of returning.
      if (!warp_wait_phase(&bars->o_done[t], cnt.o_seen & 1, bars, limit, kSiteODone)) {
        ok = false;
        break;
      }
      tc_fence_after();
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
    // P_j goes into this tile's P buffer (free again: PV_{j-1} has
    // completed, see above).
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
    sdpa_fwd64_kernel(const __grid_constant__ sdpa_impl::FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + Layout::kQ;
  uint8_t* sK = smem + Layout::kK;
  uint8_t* sV = smem + Layout::kV;
  Barriers* bars = reinterpret_cast<Barriers*>(smem + Layout::kBar);
  constexpr int kStages = Layout::kStages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    // The ring, Q and drain barriers take one commit from each MMA warp.
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, kMmaWarps);
#pragma unroll
    for (int t = 0; t < kTilesPerCta; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], kBlockM / 32);
      mbar_init(&bars->p_ready[t], kBlockM / 32);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_free[t], kBlockM / 32);
    }
    mbar_init(&bars->fin, kMmaWarps);
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], kMmaWarps);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], kMmaWarps);
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
  // Everything above may overlap the previous kernel in the stream; nothing
  // below touches global memory before that kernel has completed.
  grid_dependency_wait();
  grid_launch_dependents();
  const uint32_t tmem = bars->tmem_base;

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
    // The control warps run their loops with all 32 lanes; one elected lane
    // issues each TMA copy, MMA and commit.
    const bool leader = elect_one();
    if (warp == 0) {
      // ---------------------------------------------------- TMA producer
      int g = 0, k_end = 0, v_end = 0, jobs = 0;
      for_each_job<MODE, VARLEN, kTilesPerCta>(p, [&](const Work<kTilesPerCta>& w) -> bool {
        if (w.n_kv_max == 0) return true;  // masked out entirely: nothing to load
        // The previous job's Q must be consumed (all its S products done).
        if (jobs > 0 &&
            !warp_wait_phase(&bars->q_empty, (jobs - 1) & 1, bars, limit, kSiteEmpty))
          return false;
        if (!p.debug_withhold_q && leader) {
          const int nq = w.n_present;
          mbar_arrive_expect_tx(&bars->q_full, nq * Layout::kTileBytes);
#pragma unroll
          for (int t = 0; t < kTilesPerCta; ++t)
            if (t < nq)
              tma_tile(sQ + t * Layout::kTileBytes, &p.tm_q, &bars->q_full, 0,
                       w.row0 + w.tile(t) * kBlockM, w.head, w.batch, p.pos_q);
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
          const int s = g % kStages;
          const int use = g / kStages;
          if (use > 0 &&
              !warp_wait_phase(&bars->k_empty[s], (use - 1) & 1, bars, limit, kSiteEmpty))
            return false;
          if (leader) {
            mbar_arrive_expect_tx(&bars->k_full[s], Layout::kTileBytes);
            tma_tile(sK + s * Layout::kTileBytes, &p.tm_k, &bars->k_full[s], 0,
                     w.row0 + kt * kBlockN, w.head, w.batch, p.pos_k);
          }
          k_end = g + 1;
          if (use > 0 &&
              !warp_wait_phase(&bars->v_empty[s], (use - 1) & 1, bars, limit, kSiteEmpty))
            return false;
          if (leader) {
            mbar_arrive_expect_tx(&bars->v_full[s], Layout::kTileBytes);
            tma_tile(sV + s * Layout::kTileBytes, &p.tm_v, &bars->v_full[s], 0,
                     w.row0 + kt * kBlockN, w.head, w.batch, p.pos_v);
          }
          v_end = g + 1;
          ++g;
        }
        return true;
      });
      // Drain: every load issued must have landed before shared memory is
      // released (only matters when a wait gave up).
      for (int j = max(0, k_end - kStages); j < k_end; ++j)
        wait_phase(&bars->k_full[j % kStages], (j / kStages) & 1, bars, limit, kSiteDrain, false);
      for (int j = max(0, v_end - kStages); j < v_end; ++j)
        wait_phase(&bars->v_full[j % kStages], (j / kStages) & 1, bars, limit, kSiteDrain, false);
      if (jobs > 0 && !p.debug_withhold_q)
        wait_phase(&bars->q_full, (jobs - 1) & 1, bars, limit, kSiteDrain, false);
    } else if (warp <= kMmaWarps) {
      // ----------------------------------------------------- MMA issuers
      // Warp 1 + t issues tile t's products.  Both warps walk every job and
      // key tile and commit once per K stage, V stage, Q buffer and drain,
      // each after waiting for that stage's data (so a warp with nothing to
      // issue never arrives for a stage's next use before the other warp has
      // arrived for this one).
      const int t = warp - 1;
      constexpr uint32_t idS = idesc_f16_f32acc(BF16, false, kBlockM, kBlockN);  // N = 128 keys
      constexpr uint32_t idPV = idesc_f16_f32acc(BF16, true, kBlockM, D);        // N = 64 dims
      constexpr uint32_t kHi = desc_hi_sw128(1024);  // 8-row groups 1 KB apart
      const uint32_t q_lo = desc_lo_sw128(smem_addr(sQ), 16);
      const uint32_t k_lo = desc_lo_sw128(smem_addr(sK), 16);
      const uint32_t v_lo = desc_lo_sw128(smem_addr(sV), Layout::kTileBytes);
      const uint32_t tS = tmem + s_col(t), tO = tmem + o_col(t), tP = tmem + p_col(t);

      // S_t = Q_t K^T from key stage s: four K-steps of 16 elements (32 B
      // inside the swizzle atom).
      auto issue_s = [&](int s) {
        const uint32_t a0 = q_lo + static_cast<uint32_t>(t * (Layout::kTileBytes >> 4));
        const uint32_t b0 = k_lo + static_cast<uint32_t>(s * (Layout::kTileBytes >> 4));
        mma_ss_x4<kHi, kHi>(tS, a0, b0, 2u, 2u, idS, 0u);
        mma_commit_elect(&bars->s_full[t]);
      };
      // O_t (+)= P_t V from value stage s: P_t from TMEM (keys 2c, 2c+1 in
      // column c, 8 columns per 16 keys), 16 value rows of 128 B per K-step.
      auto issue_pv = [&](int s, bool accumulate) {
        const uint32_t b0 = v_lo + static_cast<uint32_t>(s * (Layout::kTileBytes >> 4));
#pragma unroll
        for (int h = 0; h < kBlockN / 64; ++h)
          mma_ts_x4<kHi>(tO, tP + h * 32, b0 + static_cast<uint32_t>(h * ((64 * 128) >> 4)), 8u,
                         128u, idPV, (accumulate || h > 0) ? 1u : 0u);
        mma_commit_elect(&bars->o_done[t]);
      };

      // Running state over all jobs: ring position g, jobs done, parities of
      // the next s_free / p_ready / o_free phases, and whether the tile had
      // an earlier job (whose last S load and epilogue gate this job).
      int g = 0, jobs = 0;
      uint32_t s_par = 0u, p_par = 0u, o_par = 0u;
      bool had = false;
      for_each_job<MODE, VARLEN, kTilesPerCta>(p, [&](const Work<kTilesPerCta>& w) -> bool {
        if (w.n_kv_max == 0) return true;  // masked out entirely: no products
        const int n = w.n_kv(t);
        if (!warp_wait_phase(&bars->q_full, jobs & 1, bars, limit, kSiteQFull) ||
            !warp_wait_phase(&bars->k_full[g % kStages], (g / kStages) & 1, bars, limit,
                             kSiteKFull))
          return false;
        tc_fence_after();
        if (n > 0) {
          // The previous job's last S_t must be in its softmax's registers.
          if (had) {
            if (!warp_wait_phase(&bars->s_free[t], s_par, bars, limit, kSiteSFree)) return false;
            s_par ^= 1u;
            tc_fence_after();
          }
          issue_s(g % kStages);
        }
        mma_commit_elect(&bars->k_empty[g % kStages]);
        if (w.n_kv_max == 1) mma_commit_elect(&bars->q_empty);  // the job's last S

        for (int j = 0; j < w.n_kv_max; ++j) {
          const int gj = g + j;
          // S(j+1) once the softmax has loaded S(j), then PV(j) once P(j) is
          // ready.
          if (j + 1 < w.n_kv_max) {
            const int s1 = (gj + 1) % kStages;
            if (!warp_wait_phase(&bars->k_full[s1], ((gj + 1) / kStages) & 1, bars, limit,
                                 kSiteKFull))
              return false;
            if (j + 1 < n) {
              if (!warp_wait_phase(&bars->s_free[t], s_par, bars, limit, kSiteSFree))
                return false;
              s_par ^= 1u;
              tc_fence_after();
              issue_s(s1);
            }
            mma_commit_elect(&bars->k_empty[s1]);
            if (j + 2 == w.n_kv_max) mma_commit_elect(&bars->q_empty);  // job's last S
          }
          const int sv = gj % kStages;
          if (!warp_wait_phase(&bars->v_full[sv], (gj / kStages) & 1, bars, limit, kSiteVFull))
            return false;
          if (j < n) {
            if (!warp_wait_phase(&bars->p_ready[t], p_par, bars, limit, kSitePReady))
              return false;
            p_par ^= 1u;
            // The first PV of a job overwrites O_t: the previous job's
            // epilogue must have read it.
            if (j == 0 && had &&
                !warp_wait_phase(&bars->o_free[t], o_par, bars, limit, kSiteODone))
              return false;
            tc_fence_after();
            issue_pv(sv, j > 0);
          }
          mma_commit_elect(&bars->v_empty[sv]);
        }
        g += w.n_kv_max;
        ++jobs;
        if (n > 0) {
          if (had) o_par ^= 1u;  // the next o_free wait is for this job's epilogue
          had = true;
        }
        return true;
      });
      // Everything issued by both warps must finish before TMEM is released
      // (a warp that issued nothing arrives at once).
      mma_commit_elect(&bars->fin);
      wait_phase(&bars->fin, 0, bars, limit, kSiteDrain, false);
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
  auto kern = sdpa_fwd64_kernel<MODE, BF16, VARLEN>;
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_size<kTilesPerCta>(p, VARLEN, max_ctas));
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

}  // namespace

namespace sdpa_impl {

cudaError_t launch_forward64(const FwdParams& p, int mask_mode, bool bf16, int max_ctas,
                             cudaStream_t stream) {
  if (max_ctas < 1) return cudaErrorInvalidValue;
  return bf16 ? launch_mode<true>(p, mask_mode, max_ctas, stream)
              : launch_mode<false>(p, mask_mode, max_ctas, stream);
}

cudaError_t read_and_clear_fwd64_status(unsigned int* status) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_sdpa64_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if (*status != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_sdpa64_status, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace sdpa_impl
