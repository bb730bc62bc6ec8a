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
//   * a job is one query row and a group of up to 128 of its heads: the heads
//     are the 128 rows of the tensor-core tile (M = 128; groups of fewer heads
//     are zero-padded by the tensor map), and they share the gathered keys;
//   * warp 0 loads the job's Q with a 3-D TMA box; warps 2 and 3 gather the
//     K and V rows by index with coalesced 16-byte cp.async copies (128 keys
//     per stage, a whole row per instruction group) into the swizzled layout
//     the tensor core reads, after checking every index (entries past the
//     row's count or out of range become row 0 and are removed in the
//     softmax); with one kv tensor the rows are gathered once;
//   * warp 1 issues S = Q K^T into two alternating TMEM buffers, so S(j+1)
//     runs while the softmax works on S(j), and O += P V with P in its own
//     TMEM columns;
//   * warpgroup 1 runs the online softmax, one head row per thread, as in the
//     dense kernel, and writes O / l and the log-sum-exp.
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
constexpr int kGatherWarps = 4;  // warps 8..11: one key row per thread
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
  uint64_t s_full[2], s_free[2];
  // P and O += P V double-buffered by tile parity: tile t uses P buffer t & 1,
  // p_ready[t & 1] and o_done[t & 1] (each completes once per two tiles).
  uint64_t p_ready[2], o_done[2], o_free, fin;
  uint64_t k_full[kMaxStages], k_empty[kMaxStages];
  uint64_t v_full[kMaxStages], v_empty[kMaxStages];
  // Validity of the 128 gathered keys of K tile g, in slot g % kMaskSlots:
  // word w bit i = key 32w + i; m_full[slot] completes when both gather
  // warps have written their words.
  uint64_t m_full[kMaxStages + 2];
  uint32_t kmask[kMaxStages + 2][4];
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(SBarriers) <= 1024, "barrier block too large");

enum SparseSite : unsigned int {
  kSpQ = 1u << 1, kSpK = 1u << 2, kSpEmpty = 1u << 3, kSpS = 1u << 4, kSpP = 1u << 5,
  kSpO = 1u << 6, kSpDrain = 1u << 7, kSpV = 1u << 8, kSpSFree = 1u << 9,
};

__device__ __forceinline__ bool swait(uint64_t* bar, uint32_t parity, SBarriers* bars,
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
__device__ __forceinline__ bool warp_swait(uint64_t* bar, uint32_t parity, SBarriers* bars,
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

template <int D, bool BF16>
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
      mbar_init(&bars->s_free[b], kRows / 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->p_ready[b], kRows / 32);
      mbar_init(&bars->o_done[b], 1);
    }
    mbar_init(&bars->o_free, kRows / 32);
    mbar_init(&bars->fin, 1);
    for (int s = 0; s < kMaxStages + 2; ++s) mbar_init(&bars->m_full[s], kGatherWarps);
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&bars->k_full[s], kGatherWarps);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], kGatherWarps);
      mbar_init(&bars->v_empty[s], 1);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
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
    const int r = wq * 32 + lane;  // head row within the group
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 >= 0.0f;
    const float mval = pos_scale ? -INFINITY : INFINITY;
    uint32_t ns = 0;
    int g = 0;  // K tile counter (mask slot)
    bool ok = true;
    SJob job;
    for (int jj = static_cast<int>(blockIdx.x); ok && job_of(p, jj, job); jj += step) {
      const int h = job.group * kRows + r;
      if (job.n_kv == 0) {
        // no key: zeros and lse = -inf (the safe softmax of an empty row)
        if (h < p.H) {
          uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + job.row * p.o_st + h * p.o_sh;
          for (int c = 0; c < D; c += 8)
            *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          if (p.lse != nullptr) p.lse[job.row * p.lse_st + h * p.lse_sh] = -INFINITY;
        }
        continue;
      }
      float m_used = -INFINITY, l = 0.0f;
      for (int j = 0; j < job.n_kv; ++j, ++g) {
        const uint32_t b = ns & 1;
        if (!warp_swait(&bars->s_full[b], (ns >> 1) & 1, bars, limit, kSpS)) {
          ok = false;
          break;
        }
        ++ns;
        tc_fence_after();
        float s[kKeys];
        {
          uint32_t su[kKeys];
#pragma unroll
          for (int c = 0; c < kKeys / 32; ++c)
            tmem_ld32(tmem + kColS0 + b * 128 + lane_off + c * 32, su + c * 32);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kKeys; ++c) s[c] = __uint_as_float(su[c]);
        }
        // The key mask is read before S's buffer is released: the producer
        // refills this slot only after S of a tile two later has completed,
        // which needs that release (mask slots = stages + 2), so m_full of
        // the slot is at most one phase ahead of this wait.
        uint32_t km[4];
        if (!warp_swait(&bars->m_full[g % n_slots], (g / n_slots) & 1, bars, limit,
                        kSpK)) {
          ok = false;
          break;
        }
        {
          const volatile uint32_t* src = bars->kmask[g % n_slots];
#pragma unroll
          for (int e = 0; e < 4; ++e) km[e] = src[e];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[b]);
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
        const bool need = m_tile > m_used + kRescaleLog2;
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
        uint32_t pk[kKeys / 2];
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
          {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tmem + kColO + lane_off + c * 32, o);
              tmem_ld_wait();
              float* of = reinterpret_cast<float*>(o);
#pragma unroll
              for (int e = 0; e < 32; e += 2) mul2_bcast(of[e], of[e + 1], alpha);
              tmem_st32(tmem + kColO + lane_off + c * 32, o);
            }
          }
        }
        // P buffer t & 1 is free once PV(t-2) is done.
        const uint32_t pb = t & 1;
        if (t >= 2) {
          if (!warp_swait(&bars->o_done[pb], ((t >> 1) - 1) & 1, bars, limit, kSpO)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st32(tmem + kColP + pb * 64 + lane_off, pk);
        tmem_st32(tmem + kColP + pb * 64 + lane_off + 32, pk + 32);
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
      const float inv_l = (l > 0.0f) ? (1.0f / l) : 0.0f;
      if (h < p.H && p.lse != nullptr) {
        constexpr float kLn2 = 0.693147180559945309f;
        p.lse[job.row * p.lse_st + h * p.lse_sh] = (l > 0.0f) ? (log2f(l) + m_used) * kLn2
                                                              : -INFINITY;
      }
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + job.row * p.o_st + h * p.o_sh;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + kColO + lane_off + c * 32, o);
        tmem_ld_wait();
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pw[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l,
                              __uint_as_float(o[2 * e + 1]) * inv_l);
        if (h < p.H) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pw[4 * v], pw[4 * v + 1], pw[4 * v + 2], pw[4 * v + 3]);
        }
      }
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
      if (leader) {
        mbar_arrive_expect_tx(&bars->q_full, Lay::kChunks * p.q_rows * 128);
#pragma unroll
        for (int c = 0; c < Lay::kChunks; ++c)
          tma_load_3d(sQ + c * Lay::kChunkBytes, &p.tm_q, &bars->q_full, c * 64,
                      job.group * kRows, job.row);
      }
      ++jobs;
    }
    if (jobs > 0) swait(&bars->q_full, (jobs - 1) & 1, bars, limit, kSpDrain, false);
  } else if (warp >= 8) {
    // ------------------------------------------------- key/value gathers
    // Warp w (8..11) copies key rows 32(w-8) .. +31 of every tile, 16 bytes
    // per cp.async, into the 128-byte-swizzled K-major layout the products
    // read (piece q of a 128-byte row r lands at q ^ (r & 7)); lane l loads
    // the index of row +l, and the copies are spread so that one warp
    // instruction moves whole contiguous rows (D/8 lanes per row).  A tile
    // is signalled once its copies are done, `lag` tiles behind the newest,
    // so later tiles' copies are in flight meanwhile; each thread fences its
    // completed copies for the tensor core's proxy before the warp arrives.
    const int wrow = (warp - 8) * 32;
    const uint8_t* kbase = reinterpret_cast<const uint8_t*>(p.k);
    const uint8_t* vbase = reinterpret_cast<const uint8_t*>(p.v);
    constexpr int kPieces = D / 8;          // 16-byte pieces per row
    constexpr int kRowsPerOp = 32 / kPieces;
    const int piece = lane % kPieces;
    const int pc_chunk = piece >> 3, pc_q = piece & 7;
    int g = 0, signalled = 0;
    // Copies in flight per warp: fewer than the ring's free stages (the MMA
    // holds two), and on the shared-kv ring two rather than four -- a tile
    // is announced sooner after its copies land, which the products wait
    // for (measured: 486 vs 464 TFLOP/s on the top-2048 workload; one is
    // slower again).
    const int lag = max(1, min(nst - 4, 4));
    bool ok = true;
    auto signal_oldest = [&]() {
      const int s = signalled % nst;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->k_full[s]);
        mbar_arrive(&bars->v_full[s]);
      }
      ++signalled;
    };
    SJob job;
    for (int jj = static_cast<int>(blockIdx.x); ok && job_of(p, jj, job); jj += step) {
      if (job.n_kv == 0) continue;
      const int* irow = p.idx + static_cast<int64_t>(job.row) * p.idx_st;
      auto load_idx = [&](int j) {
        const int ta = j * kKeys + wrow + lane;
        return (ta < job.len) ? __ldg(irow + ta) : -1;
      };
      int na = load_idx(0);
      for (int j = 0; j < job.n_kv; ++j, ++g) {
        const int s = g % nst;
        const int use = g / nst;
        // an entry past the row's count or outside [0, total_k) reads row 0
        // and is removed by the softmax through the mask
        const bool va = na >= 0 && na < p.total_k;
        const int ra = va ? na : 0;
        const uint32_t ba = __ballot_sync(0xffffffffu, va);
        if (j + 1 < job.n_kv) na = load_idx(j + 1);
        if (use > 0) {
          const uint32_t par = (use - 1) & 1;
          const bool free_now = __all_sync(
              0xffffffffu, mbar_test_wait(&bars->k_empty[s], par) &&
                               (p.kv_shared || mbar_test_wait(&bars->v_empty[s], par)));
          if (!free_now) {
            // About to block on a stage: first finish and signal every tile
            // still in flight, so the consumers never wait on copies that are
            // done but not yet announced.
            cp_async_wait<0>();
            while (signalled < g) signal_oldest();
            if (!warp_swait(&bars->k_empty[s], par, bars, limit, kSpEmpty) ||
                (!p.kv_shared && !warp_swait(&bars->v_empty[s], par, bars, limit, kSpEmpty))) {
              ok = false;
              break;
            }
          }
        }
        if (lane == 0) {
          volatile uint32_t* dst = bars->kmask[g % n_slots];
          dst[warp - 8] = ba;  // keys wrow .. +31
          mbar_arrive(&bars->m_full[g % n_slots]);  // release: the mask is written
        }
        auto copy_rows = [&](const uint8_t* base, int64_t row_bytes, uint8_t* stage) {
#pragma unroll 4
          for (int k = 0; k < 32 / kRowsPerOp; ++k) {
            const int m = k * kRowsPerOp + lane / kPieces;  // row within this warp's 32
            const int ridx = __shfl_sync(0xffffffffu, ra, m);
            const int r = wrow + m;
            cp_async_16(stage + pc_chunk * Lay::kChunkBytes + r * 128 + ((pc_q ^ (r & 7)) << 4),
                        base + static_cast<int64_t>(ridx) * row_bytes + piece * 16);
          }
        };
        copy_rows(kbase, p.k_row_bytes, sK + s * Lay::kTileBytes);
        if (!p.kv_shared) copy_rows(vbase, p.v_row_bytes, sV + s * Lay::kTileBytes);
        cp_async_commit();
        // Keep `lag` tiles of copies in flight (fewer than the ring depth,
        // so the next tile's stage is always one that was signalled).
        if (g + 1 - signalled > lag) {
          switch (lag) {
            case 1: cp_async_wait<1>(); break;
            case 2: cp_async_wait<2>(); break;
            case 3: cp_async_wait<3>(); break;
            default: cp_async_wait<4>(); break;
          }
          while (g + 1 - signalled > lag) signal_oldest();
        }
      }
    }
    cp_async_wait<0>();
    while (signalled < g) signal_oldest();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issue
    constexpr uint32_t idS = idesc_f16_f32acc(BF16, false, kRows, kKeys);
    constexpr uint32_t idPV = idesc_f16_f32acc(BF16, true, kRows, D);
    constexpr uint32_t kHi = desc_hi_sw128(1024);
    const uint32_t q_lo = desc_lo_sw128(smem_addr(sQ), 16);
    const uint32_t k_lo = desc_lo_sw128(smem_addr(sK), 16);
    // V rows: their own stages, or the K stage when one kv tensor serves both
    const uint32_t v_lo = desc_lo_sw128(smem_addr(p.kv_shared ? sK : sV), Lay::kChunkBytes);
    bool issued_any = false;
    auto issue_s = [&](uint32_t buf, int s) {
      const uint32_t b0 = k_lo + static_cast<uint32_t>(s * (Lay::kTileBytes >> 4));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * Lay::kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ss_elect<kHi, kHi>(tmem + kColS0 + buf * 128, q_lo + off, b0 + off, idS,
                               kk > 0 ? 1u : 0u);
      }
      mma_commit_elect(&bars->s_full[buf]);
    };
    auto issue_pv = [&](int s, uint32_t pb, bool accumulate) {
      const uint32_t b0 = v_lo + static_cast<uint32_t>(s * (Lay::kTileBytes >> 4));
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk)
        mma_ts_elect<kHi>(tmem + kColO, tmem + kColP + pb * 64 + kk * 8,
                          b0 + ((kk * 16 * 128) >> 4), idPV, (accumulate || kk > 0) ? 1u : 0u);
      mma_commit_elect(&bars->o_done[pb]);
    };
    int g = 0, jobs = 0;
    uint32_t ns = 0;
    bool ok = true;
    SJob job;
    // S into the buffer of S(ns); its previous contents (S(ns-2)) must be in
    // the softmax's registers.
    auto s_next = [&](int s) -> bool {
      const uint32_t buf = ns & 1;
      if (ns >= 2 && !warp_swait(&bars->s_free[buf], ((ns >> 1) - 1) & 1, bars, limit, kSpSFree))
        return false;
      tc_fence_after();
      issue_s(buf, s);
      if (!p.kv_shared) mma_commit_elect(&bars->k_empty[s]);  // else after PV
      ++ns;
      return true;
    };
    for (int jj = static_cast<int>(blockIdx.x); ok && job_of(p, jj, job); jj += step) {
      if (job.n_kv == 0) continue;
      if (!warp_swait(&bars->q_full, jobs & 1, bars, limit, kSpQ) ||
          !warp_swait(&bars->k_full[g % nst], (g / nst) & 1, bars, limit, kSpK) ||
          !s_next(g % nst))
        break;
      issued_any = true;
      if (job.n_kv == 1) mma_commit_elect(&bars->q_empty);
      for (int j = 0; j < job.n_kv; ++j) {
        const int gj = g + j;
        if (j + 1 < job.n_kv) {
          const int s1 = (gj + 1) % nst;
          if (!warp_swait(&bars->k_full[s1], ((gj + 1) / nst) & 1, bars, limit, kSpK) ||
              !s_next(s1)) {
            ok = false;
            break;
          }
          if (j + 2 == job.n_kv) mma_commit_elect(&bars->q_empty);
        }
        const int s = gj % nst;
        if (!warp_swait(&bars->v_full[s], (gj / nst) & 1, bars, limit, kSpV) ||
            !warp_swait(&bars->p_ready[gj & 1], (gj >> 1) & 1, bars, limit, kSpP)) {
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

template <int D, bool BF16>
cudaError_t launch_sparse_one(const sdpa_impl::SparseParams& p, int max_ctas,
                              cudaStream_t stream) {
  auto kern = sparse_fwd_kernel<D, BF16>;
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
  if (head_dim == 64)
    return bf16 ? launch_sparse_one<64, true>(p, max_ctas, stream)
                : launch_sparse_one<64, false>(p, max_ctas, stream);
  return bf16 ? launch_sparse_one<128, true>(p, max_ctas, stream)
              : launch_sparse_one<128, false>(p, max_ctas, stream);
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
