// sdpa_fwd64_sm103a.cu -- fused scaled dot-product attention forward for sm_103a,
// head size 64.
//
// The same computation as the head-size-128 kernel (the five-step attention
// of "Profiling attention in PyTorch: kernels, backends and where the time
// goes", news.bpdata.com, section "Naiv causal attention", evaluated with an
// online softmax over K/V tiles as that page's "Flash backend" section
// describes), with a tile plan chosen for D = 64 -- the per-shape choice
// that page credits for the cuDNN backend's speed (section "cuDNN backend"):
//
//   * with D = 64 the two products of a tile take half the tensor-core time
//     they take at D = 128, while the softmax of a tile costs the same, so
//     two 128-key softmax warpgroups cannot keep the tensor core busy.  Here
//     a CTA holds FOUR 128-row query tiles, each with its own softmax
//     warpgroup (640 threads), and the products and the softmax step
//     through every 128-key K/V tile in two halves of 64 keys;
//   * TMEM (512 columns): tile t has S_t (64 columns, P_t written over its
//     first 32) at 128t and O_t (64 columns) at 128t + 64;
//   * warps 1 and 2 issue the products, warp m for tiles m and m + 2: per
//     64-key half-step i, once both its tiles' P(i) are ready,
//       PV_m(i) PV_m+2(i) S_m(i+1) S_m+2(i+1)
//     (four MMAs per elected issue), so while one softmax warpgroup works on
//     its S the tensor core runs the other tiles' products.  At D = 64 a tile
//     carries only ~350 cycles of tensor work per half-step, less than one
//     warp's per-tile cost of barrier checks, fences and issue, so one
//     issuing warp for all four tiles starved the tensor core;
//   * warp 0 streams Q (four 16 KB boxes per job) and a ring of five K and
//     five V tiles of 128 keys (16 KB each) with TMA; each K tile feeds the
//     S products of both its halves, each V tile the PV products of both;
//   * a job is a group of four adjacent query tiles (sdpa_sched.cuh); units
//     pair group G-1-k with group k of the same head so causal units cost the
//     same; small problems deal jobs by falling cost in snake order;
//   * explicit masks as at D = 128: bits per row and 128-key tile from the
//     mask bytes or from a plan's tile summary (which also lets every role
//     skip key tiles that remove every key for all four query tiles).
//
// Safe softmax, bounded waits and the status word follow the head-size-128
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
constexpr int kTiles = 4;                      // query tiles per CTA
constexpr int kStepN = 64;                     // keys per product / softmax step
constexpr int kMmaWarps = 2;                   // warps 1, 2 issue the products (tiles m, m + 2)
constexpr int kThreads = 128 * (1 + kTiles);   // WG0: TMA, MMA, 2 spare; WG1..4: tiles 0..3
// Register split: __launch_bounds__(640, 1) caps a thread at 96 registers;
// the control warpgroup gives registers back and the four softmax
// warpgroups take them (128*64 + 512*104 == 640*96).
constexpr uint32_t kLaunchRegs = 96;
constexpr uint32_t kRegsControl = 64;
constexpr uint32_t kRegsSoftmax = 104;
static_assert(128 * kRegsControl + 128 * kTiles * kRegsSoftmax <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when max grows by > 2^8
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t s_col(int t) { return 128u * static_cast<uint32_t>(t); }
__host__ __device__ constexpr uint32_t o_col(int t) {
  return 128u * static_cast<uint32_t>(t) + 64u;
}

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
  static constexpr int kTileBytes = kBlockM * 128;  // 128 rows x 64 elements (one box)
  static constexpr int kStages = 5;                 // K ring and V ring depth
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTiles * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBar = kV + kStages * kTileBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kTotal = kBar + kBarBytes + 1024;  // + slack for 1 KB alignment
};

struct Barriers {
  uint64_t q_full;
  uint64_t q_empty;  // the job's Q tiles are no longer read (all its S done)
  uint64_t s_full[kTiles];
  uint64_t p_ready[kTiles];
  uint64_t o_done[kTiles];
  uint64_t o_free[kTiles];  // the job's O_t read by its epilogue
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
struct SoftmaxCounters {
  uint32_t s_seen;  // completions of s_full[t] consumed
  uint32_t o_seen;  // completions of o_done[t] consumed
};

// Whether key c of a 64-key step starting at key c0 is removed for this
// row: past the sequence, past the row (causal), or by the mask bits (mb0:
// keys c0..c0+31, mb1: c0+32..c0+63).
template <int MODE>
__device__ __forceinline__ bool removed_key(int c, int c0, uint32_t mb0, uint32_t mb1, int len,
                                            int row_g) {
  bool r = c0 + c >= len;
  if constexpr (MODE == sdpa_impl::kMaskCausal) r = r || (c0 + c > row_g);
  if constexpr (MODE == sdpa_impl::kMaskExplicit)
    r = r || (((c < 32 ? mb0 : mb1) >> (c & 31)) & 1u);
  return r;
}

// One job of tile t: every visited 128-key tile in two 64-key half-steps.
// One query row per thread (TMEM lane = row).  Returns false when a wait
// gave up.
template <int MODE, bool BF16>
__device__ __forceinline__ bool softmax_job(const sdpa_impl::FwdParams& p,
                                            const Work<kTiles>& w, int t, Barriers* bars,
                                            uint32_t tmem, int wq, int lane,
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
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + s_col(t) + lane_off;  // S_i, and P_i over its first 32 columns
  const uint32_t tO = tmem + o_col(t) + lane_off;
  const int r = wq * 32 + lane;
  const int row_g = qt * kBlockM + r;
  const float sl2 = p.scale_log2;
  const bool pos_scale = sl2 >= 0.0f;
  const float mval = pos_scale ? -INFINITY : INFINITY;  // a removed raw score
  float m_used = -INFINITY;  // running max actually used in the exponentials
  float l = 0.0f;            // running row sum of probabilities
  bool ok = true;
  KeyTileCursor kc{-1, 0u};
  // With a tile summary the next visited tile and this row's 128 bits of it
  // are fetched one tile ahead.
  int kt_next = next_key_tile<MODE, kTiles>(p, w, kc, 0);
  uint4 bits_next = make_uint4(0u, 0u, 0u, 0u);
  const uint4* tile_bits_row = nullptr;
  if constexpr (MODE == sdpa_impl::kMaskExplicit) {
    if (p.tile_class != nullptr) {
      tile_bits_row = p.tile_bits + static_cast<int64_t>(qt) * p.n_tiles * kBlockM + r;
      bits_next = __ldg(tile_bits_row + static_cast<int64_t>(kt_next) * kBlockM);
    }
  }

  for (int j = 0; j < n && ok; ++j) {
    const int kt = kt_next;
    if (tile_bits_row == nullptr) kt_next = j + 1;  // every key tile in order
    const int col0 = kt * kBlockN;
    // Explicit mask: this row's bits for the 128-key tile (bit set =
    // removed), ready before the first half's S is waited for.
    uint32_t mbits[kBlockN / 32] = {0u, 0u, 0u, 0u};
    if constexpr (MODE == sdpa_impl::kMaskExplicit) {
      if (tile_bits_row != nullptr) {
        mbits[0] = bits_next.x;
        mbits[1] = bits_next.y;
        mbits[2] = bits_next.z;
        mbits[3] = bits_next.w;
        if (j + 1 < n) {
          kt_next = next_key_tile<MODE, kTiles>(p, w, kc, j + 1);
          bits_next = __ldg(tile_bits_row + static_cast<int64_t>(kt_next) * kBlockM);
        }
      } else {
        mask_bits_from_bytes(p, w.len, row_g, lane, col0, mbits);
      }
    }
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      const int c0 = col0 + h * kStepN;
      const uint32_t mb0 = h ? mbits[2] : mbits[0];
      const uint32_t mb1 = h ? mbits[3] : mbits[1];
      bool masked = (c0 + kStepN > w.len) || (MODE == sdpa_impl::kMaskCausal && kt == qt);
      if constexpr (MODE == sdpa_impl::kMaskExplicit)
        masked = masked || __any_sync(0xffffffffu, (mb0 | mb1) != 0u);
      if (!warp_wait_phase(&bars->s_full[t], cnt.s_seen & 1, bars, limit, kSiteSFull)) {
        ok = false;
        break;
      }
      ++cnt.s_seen;
      tc_fence_after();
      // Pass 1: the 64 scores of this row, masked, for the row extremum
      // (max for a positive scale): eight chains of three-input max.
      float ext;
      {
        float s[kStepN];
        {
          uint32_t su[kStepN];
          tmem_ld32(tS, su);
          tmem_ld32(tS + 32, su + 32);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kStepN; ++c) s[c] = __uint_as_float(su[c]);
        }
        if (masked) {
#pragma unroll
          for (int c = 0; c < kStepN; ++c) s[c] = removed_key<MODE>(c, c0, mb0, mb1, w.len, row_g)
                                                      ? mval : s[c];
        }
        float e8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) e8[i] = s[i];
        if (pos_scale) {
#pragma unroll
          for (int c = 8; c < kStepN; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              e8[i] = max3f(e8[i], s[c + i], s[c + 8 + i < kStepN ? c + 8 + i : c + i]);
          e8[0] = max3f(e8[0], e8[1], e8[2]);
          e8[3] = max3f(e8[3], e8[4], e8[5]);
          e8[6] = fmaxf(e8[6], e8[7]);
          e8[0] = max3f(e8[0], e8[3], e8[6]);
        } else {
#pragma unroll
          for (int c = 8; c < kStepN; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              e8[i] = min3f(e8[i], s[c + i], s[c + 8 + i < kStepN ? c + 8 + i : c + i]);
          e8[0] = min3f(e8[0], e8[1], e8[2]);
          e8[3] = min3f(e8[3], e8[4], e8[5]);
          e8[6] = fminf(e8[6], e8[7]);
          e8[0] = min3f(e8[0], e8[3], e8[6]);
        }
        ext = e8[0];
      }
      const float m_tile = (ext == mval) ? -INFINITY : ext * sl2;
      const bool need = m_tile > m_used + kRescaleLog2;
      float alpha = 1.0f;
      if (need) {
        alpha = ex2(m_used - m_tile);  // 0 when nothing was admitted before
        m_used = m_tile;
        l *= alpha;
      }
      const float neg_m = (m_used == -INFINITY) ? 0.0f : -m_used;
      // Pass 2, 32 scores at a time (read again from TMEM, which keeps the
      // registers of the first pass free): x = s * scale*log2(e) - m (packed
      // FMA), p = 2^x, packed row sums, and P packed to 16 bits and stored
      // over the first 32 columns of S -- chunk c's P (16 columns at 16c)
      // only overwrites scores that chunks <= c have read.  A removed score
      // is +-inf with the sign that makes x = -inf, so its probability is
      // exactly 0.  The stores are waited for before P is released.
      float rs[8];  // four packed pairs of partial row sums
#pragma unroll
      for (int i = 0; i < 8; ++i) rs[i] = 0.0f;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        float s[32];
        {
          uint32_t su[32];
          tmem_ld32(tS + 32 * ch, su);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = __uint_as_float(su[c]);
        }
        if (masked) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            s[c] = removed_key<MODE>(32 * ch + c, c0, mb0, mb1, w.len, row_g) ? mval : s[c];
        }
#pragma unroll
        for (int c = 0; c < 32; c += 2) fma2_bcast(s[c], s[c + 1], s[c], s[c + 1], sl2, neg_m);
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c] = ex2(s[c]);
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          add2_acc(rs[2 * (c & 3)], rs[2 * (c & 3) + 1], s[2 * c], s[2 * c + 1]);
          pk[c] = pack2<BF16>(s[2 * c], s[2 * c + 1]);
        }
        tmem_st16(tS + 16 * ch, pk);
      }
      add2_acc(rs[0], rs[1], rs[2], rs[3]);
      add2_acc(rs[4], rs[5], rs[6], rs[7]);
      add2_acc(rs[0], rs[1], rs[4], rs[5]);
      l += rs[0] + rs[1];

      if (j > 0 || h > 0) {
        // PV of the previous half-step has completed: S of this one was
        // issued after it and the tensor pipe completes in issue order, so
        // s_full already implies that o_done phase; it is only counted.
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
      // P is in TMEM once its stores complete.
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_ready[t]);  // one arrival per warp
    }
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
    // The ring, Q and drain barriers take one commit from each issuing warp.
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, kMmaWarps);
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&bars->s_full[t], 1);
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
    // warps 4..7 -> tile 0, 8..11 -> tile 1, 12..15 -> tile 2, 16..19 -> tile 3
    const int t = (warp - 4) >> 2;
    SoftmaxCounters cnt{0, 0};
    for_each_job<MODE, VARLEN, kTiles>(p, [&](const Work<kTiles>& w) {
      return softmax_job<MODE, BF16>(p, w, t, bars, tmem, warp & 3, lane, cnt);
    });
  } else {
    regs_decrease<kRegsControl>();
    // Both control warps run their loops with all 32 lanes; one elected lane
    // issues each TMA copy, MMA and commit.
    const bool leader = elect_one();
    if (warp == 0) {
      // ---------------------------------------------------- TMA producer
      int g = 0, k_end = 0, v_end = 0, jobs = 0;
      for_each_job<MODE, VARLEN, kTiles>(p, [&](const Work<kTiles>& w) -> bool {
        if (w.n_kv_max == 0) return true;  // masked out entirely: nothing to load
        // The previous job's Q must be consumed (all its S products done).
        if (jobs > 0 &&
            !warp_wait_phase(&bars->q_empty, (jobs - 1) & 1, bars, limit, kSiteEmpty))
          return false;
        if (!p.debug_withhold_q && leader) {
          const int nq = w.n_present;  // the group's tiles inside the sequence
          mbar_arrive_expect_tx(&bars->q_full, nq * Layout::kTileBytes);
#pragma unroll
          for (int t = 0; t < kTiles; ++t)
            if (t < nq)
              tma_tile(sQ + t * Layout::kTileBytes, &p.tm_q, &bars->q_full, 0,
                       w.row0 + w.tile(t) * kBlockM, w.head, w.batch, p.pos_q);
        }
        ++jobs;
        const bool summary = MODE == sdpa_impl::kMaskExplicit && p.tile_class != nullptr;
        const int n_scan = summary ? p.n_tiles : w.n_kv_max;
        uint32_t visit = 0xffffffffu;
        for (int kt = 0; kt < n_scan; ++kt) {
          if (summary) {
            if ((kt & 31) == 0) visit = visit_chunk<kTiles>(p, w, kt >> 5);
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
    } else if (warp >= 1 && warp <= kMmaWarps) {
      // ---------------------------------------------------- MMA issuers
      // Warp 1 + m issues the products of tiles m and m + kMmaWarps.  Both
      // warps walk every job and ring tile and commit once per ring stage,
      // Q buffer and drain; a stage is released when both commits have
      // arrived.  (A warp whose tiles are absent still waits for each V tile
      // before committing, so its early arrivals never reach the next use of
      // a stage before the other warp's arrival for this one.)
      const int m = warp - 1;
      constexpr uint32_t idS = idesc_f16_f32acc(BF16, false, kBlockM, kStepN);  // N = 64 keys
      constexpr uint32_t idPV = idesc_f16_f32acc(BF16, true, kBlockM, D);       // N = 64 dims
      constexpr uint32_t kHi = desc_hi_sw128(1024);  // 8-row groups 1 KB apart
      const uint32_t q_lo = desc_lo_sw128(smem_addr(sQ), 16);
      const uint32_t k_lo = desc_lo_sw128(smem_addr(sK), 16);
      const uint32_t v_lo = desc_lo_sw128(smem_addr(sV), Layout::kTileBytes);

      // S_t = Q_t K_h^T: keys 64h..64h+63 of key stage s (8 KB into the
      // tile); four K-steps of 16 elements (32 B inside the swizzle atom).
      auto issue_s = [&](int t, int s, int h) {
        const uint32_t a0 = q_lo + static_cast<uint32_t>(t * (Layout::kTileBytes >> 4));
        const uint32_t b0 = k_lo + static_cast<uint32_t>(s * (Layout::kTileBytes >> 4)) +
                            static_cast<uint32_t>(h * ((kStepN * 128) >> 4));
        mma_ss_x4<kHi, kHi>(tmem + s_col(t), a0, b0, 2u, 2u, idS, 0u);
        mma_commit_elect(&bars->s_full[t]);
      };
      // O_t (+)= P_t V_h: P_t from TMEM (keys 2c, 2c+1 in column c; 8
      // columns per 16 keys), value rows 64h..64h+63 of value stage s (16
      // rows of 128 B per K-step).
      auto issue_pv = [&](int t, int s, int h, bool accumulate) {
        const uint32_t b0 = v_lo + static_cast<uint32_t>(s * (Layout::kTileBytes >> 4)) +
                            static_cast<uint32_t>(h * ((kStepN * 128) >> 4));
        mma_ts_x4<kHi>(tmem + o_col(t), tmem + s_col(t), b0, 8u, 128u, idPV,
                       accumulate ? 1u : 0u);
        mma_commit_elect(&bars->o_done[t]);
      };

      // Running state over all jobs: ring position g, jobs done, and per tile
      // t three bits -- bit t of p_par: parity of the next p_ready phase;
      // bit t of o_par: parity of the next o_free phase; bit t of o_any: the
      // tile had an earlier job (whose epilogue must free O_t).
      int g = 0, jobs = 0;
      uint32_t p_par = 0u, o_par = 0u, o_any = 0u;
      for_each_job<MODE, VARLEN, kTiles>(p, [&](const Work<kTiles>& w) -> bool {
        if (w.n_kv_max == 0) return true;  // masked out entirely: no products
        if (!warp_wait_phase(&bars->q_full, jobs & 1, bars, limit, kSiteQFull) ||
            !warp_wait_phase(&bars->k_full[g % kStages], (g / kStages) & 1, bars, limit,
                             kSiteKFull))
          return false;
        tc_fence_after();
#pragma unroll
        for (int k2 = 0; k2 < kTiles / kMmaWarps; ++k2) {
          const int t = m + kMmaWarps * k2;
          if (w.n_kv(t) > 0) issue_s(t, g % kStages, 0);
        }

        const int n_half = 2 * w.n_kv_max;
        bool ok = true;
        for (int i = 0; i < n_half && ok; ++i) {
          const int h = i & 1;
          const int gj = g + (i >> 1);         // ring tile of this half-step
          const int sv = gj % kStages;
          const int gk1 = g + ((i + 1) >> 1);  // ring tile of the next half-step's S
          if (h == 0 &&
              !warp_wait_phase(&bars->v_full[sv], (gj / kStages) & 1, bars, limit, kSiteVFull)) {
            ok = false;
            break;
          }
          // P(i) of this warp's active tiles (and, at a job's first PV, the
          // previous job's epilogue having read O), then one fence.
          bool ready = true;
#pragma unroll
          for (int k2 = 0; k2 < kTiles / kMmaWarps; ++k2) {
            const int t = m + kMmaWarps * k2;
            if (i >= 2 * w.n_kv(t)) continue;
            ready = ready && wait_phase(&bars->p_ready[t], (p_par >> t) & 1u, bars, limit,
                                        kSitePReady);
            p_par ^= 1u << t;
            if (i == 0 && ((o_any >> t) & 1u))
              ready = ready && wait_phase(&bars->o_free[t], (o_par >> t) & 1u, bars, limit,
                                          kSiteODone);
          }
          if (!__all_sync(0xffffffffu, ready)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k2 = 0; k2 < kTiles / kMmaWarps; ++k2) {
            const int t = m + kMmaWarps * k2;
            if (i < 2 * w.n_kv(t)) issue_pv(t, sv, h, i > 0);
          }
          bool k_ready = (h == 0);  // the next S reads the second half of this K tile
#pragma unroll
          for (int k2 = 0; k2 < kTiles / kMmaWarps; ++k2) {
            const int t = m + kMmaWarps * k2;
            if (i + 1 >= 2 * w.n_kv(t)) continue;
            if (!k_ready) {
              if (!warp_wait_phase(&bars->k_full[gk1 % kStages], (gk1 / kStages) & 1, bars, limit,
                                   kSiteKFull)) {
                ok = false;
                break;
              }
              tc_fence_after();
              k_ready = true;
            }
            issue_s(t, gk1 % kStages, (i + 1) & 1);
          }
          if (!ok) break;
          // Both halves' S of this K tile and both halves' PV of this V tile
          // are issued once the h = 0 and h = 1 steps are, respectively.
          if (h == 0) mma_commit_elect(&bars->k_empty[sv]);
          if (h == 1) mma_commit_elect(&bars->v_empty[sv]);
          if (i + 2 == n_half) mma_commit_elect(&bars->q_empty);  // job's last S issued
        }
        if (!ok) return false;
        g += w.n_kv_max;
        ++jobs;
#pragma unroll
        for (int t = 0; t < kTiles; ++t)
          if (w.n_kv(t) > 0) {
            // the next o_free wait of tile t is for this job's epilogue
            if ((o_any >> t) & 1u) o_par ^= 1u << t;
            o_any |= 1u << t;
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
  cfg.gridDim = dim3(grid_size<kTiles>(p, VARLEN, max_ctas));
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
