// sdpa_fwd_sm103a.cu -- fused scaled dot-product attention forward for sm_103a.
//
// Computes, per (batch, head), out = softmax(scale * Q K^T with causal or
// boolean masking) V: the five-step attention of "Profiling attention in
// PyTorch: kernels, backends and where the time goes" (news.bpdata.com),
// section "Naiv causal attention", evaluated the way that page's "Flash
// backend" section describes -- tiles of K and V streamed past an on-chip
// query tile with an online softmax, so the [seq, seq] score matrix never
// reaches HBM -- but built for Blackwell:
//
//   * one CTA per (batch*head, 128-row query tile); a head's tiles are adjacent
//     in launch order (heaviest causal tile first) so K/V stay in L2;
//   * warp 0 (one lane) streams Q once and a ring of K/V tiles with TMA
//     (128-byte swizzled boxes of 64 x 128 elements) into shared memory;
//   * warp 1 (one lane) issues tcgen05.mma: S_j = Q K_j^T into one of two TMEM
//     score buffers, and O += P_j V_j with P read straight from TMEM;
//   * warps 4..7 (one query row per thread, TMEM lane = row) load S_j from
//     TMEM, apply scale, causal / explicit / ragged-tail masks and the online
//     softmax in registers (a whole score row lives in one thread, so row max
//     and row sum need no shuffles), write P_j back over S_j as 16-bit pairs,
//     rescale O in TMEM only when the running maximum grows by more than 2^8,
//     and finally write O / l.
//
// Safe softmax: a row with no admissible key ends with l = 0 and is written
// as zeros, as the math backend's _safe_softmax does (same page, "Math
// backend" section).  Every barrier wait is bounded in time; on expiry the
// CTA records a status bit in g_sdpa_device_status, stops issuing work,
// drains what it already issued and frees its tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sdpa_internal.h"

using namespace sdpa_dev;

// Device status word: bit 0 = some barrier wait ran out of time; the upper
// bits name the wait site.  Read and cleared by sdpa_last_device_status().
__device__ unsigned int g_sdpa_device_status = 0;

namespace {

constexpr int kBlockM = 128;   // query rows per tile (TMEM lanes)
constexpr int kBlockN = 128;   // keys per tile
constexpr int kThreads = 256;  // 8 warps: TMA, MMA, 2 idle, 4 softmax
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when max grows by > 2^8
constexpr uint32_t kTmemCols = 512;

enum WaitSite : unsigned int {
  kSiteQFull = 1u << 1,
  kSiteKvFull = 1u << 2,
  kSiteKvEmpty = 1u << 3,
  kSiteSFull = 1u << 4,
  kSitePReady = 1u << 5,
  kSitePvDone = 1u << 6,
  kSiteDrain = 1u << 7,
};

template <int D>
struct Layout {
  static constexpr int kChunks = D / 64;               // 128-byte swizzle atoms along D
  static constexpr int kChunkBytes = kBlockM * 128;    // one 128-row x 64-element box
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = (D == 64) ? 4 : 3;    // K/V ring depth
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBar = kV + kStages * kTileBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kTotal = kBar + kBarBytes + 1024;  // + slack for 1 KB alignment
};

struct Barriers {
  uint64_t q_full;
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t pv_done;
  uint64_t fin;
  uint64_t k_full[4];
  uint64_t v_full[4];
  uint64_t kv_empty[4];
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(Barriers) <= 256, "barrier block too large");
static_assert(Layout<128>::kTotal <= 227 * 1024, "shared memory over the per-CTA limit");
static_assert(Layout<64>::kTotal <= 227 * 1024, "shared memory over the per-CTA limit");

// Bounded wait on one barrier phase.  Returns false when the wait gave up:
// either another role already raised the CTA abort flag (honour_abort), or
// this wait exceeded the time limit, in which case it raises the flag and
// records `site` in the device status word.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, Barriers* bars,
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
        atomicOr(&g_sdpa_device_status, 1u | site);
        return false;
      }
    }
  }
}

// Warp-uniform version: every lane polls, and the warp proceeds only if all
// lanes saw the phase complete (keeps later .sync.aligned ops convergent).
__device__ __forceinline__ bool warp_wait_phase(uint64_t* bar, uint32_t parity, Barriers* bars,
                                                uint64_t limit_ns, unsigned int site) {
  const bool ok = wait_phase(bar, parity, bars, limit_ns, site);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void tma_tile(void* dst, const CUtensorMap* map, uint64_t* bar,
                                         int d0, int row, int head, int batch,
                                         const int (&pos)[3]) {
  int c[4] = {d0, 0, 0, 0};
  c[pos[0]] = row;
  c[pos[1]] = head;
  c[pos[2]] = batch;
  tma_load_4d(dst, map, bar, c[0], c[1], c[2], c[3]);
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

// ------------------------------------------------------------------ kernel
template <int D, int MODE, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    sdpa_fwd_kernel(const __grid_constant__ sdpa_impl::FwdParams p) {
  using Lay = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + Lay::kQ;
  uint8_t* sK = smem + Lay::kK;
  uint8_t* sV = smem + Lay::kV;
  Barriers* bars = reinterpret_cast<Barriers*>(smem + Lay::kBar);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Launch order walks one head's query tiles (heaviest first) before the
  // next head, so the CTAs resident at any time share a few heads' K/V in L2.
  const int bh = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.n_tiles));
  const int batch = bh / p.H;
  const int head = bh - batch * p.H;
  const int q_tile = p.n_tiles - 1 - static_cast<int>(blockIdx.x - bh * p.n_tiles);
  const int n_kv = (MODE == sdpa_impl::kMaskCausal) ? (q_tile + 1) : p.n_tiles;
  const uint64_t limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->p_ready[0], kBlockM);
    mbar_init(&bars->p_ready[1], kBlockM);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->fin, 1);
#pragma unroll
    for (int s = 0; s < Lay::kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
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
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tS0 = tmem;        // score / probability buffer 0: columns [0, 128)
  const uint32_t tS1 = tmem + 128;  // score / probability buffer 1: columns [128, 256)
  const uint32_t tO = tmem + 256;   // output accumulator: columns [256, 256 + D)

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued[4] = {0, 0, 0, 0};
      if (!p.debug_withhold_q) {
        mbar_arrive_expect_tx(&bars->q_full, Lay::kTileBytes);
#pragma unroll
        for (int c = 0; c < Lay::kChunks; ++c)
          tma_tile(sQ + c * Lay::kChunkBytes, &p.tm_q, &bars->q_full, c * 64, q_tile * kBlockM,
                   head, batch, p.pos_q);
      }
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % Lay::kStages;
        const int use = j / Lay::kStages;
        if (use > 0 &&
            !wait_phase(&bars->kv_empty[s], (use - 1) & 1, bars, limit, kSiteKvEmpty))
          break;
        mbar_arrive_expect_tx(&bars->k_full[s], Lay::kTileBytes);
#pragma unroll
        for (int c = 0; c < Lay::kChunks; ++c)
          tma_tile(sK + s * Lay::kTileBytes + c * Lay::kChunkBytes, &p.tm_k, &bars->k_full[s],
                   c * 64, j * kBlockN, head, batch, p.pos_k);
        mbar_arrive_expect_tx(&bars->v_full[s], Lay::kTileBytes);
#pragma unroll
        for (int c = 0; c < Lay::kChunks; ++c)
          tma_tile(sV + s * Lay::kTileBytes + c * Lay::kChunkBytes, &p.tm_v, &bars->v_full[s],
                   c * 64, j * kBlockN, head, batch, p.pos_v);
        issued[s] = use + 1;
      }
      // Drain: every load issued must have landed before shared memory is
      // released (only matters when a wait gave up).
#pragma unroll
      for (int s = 0; s < Lay::kStages; ++s)
        if (issued[s] > 0) {
          wait_phase(&bars->k_full[s], (issued[s] - 1) & 1, bars, limit, kSiteDrain, false);
          wait_phase(&bars->v_full[s], (issued[s] - 1) & 1, bars, limit, kSiteDrain, false);
        }
      if (!p.debug_withhold_q)
        wait_phase(&bars->q_full, 0, bars, limit, kSiteDrain, false);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16_f32acc(BF16, false, kBlockM, kBlockN);
      constexpr uint32_t idPV = idesc_f16_f32acc(BF16, true, kBlockM, D);
      const uint32_t aQ = smem_addr(sQ);
      const uint32_t aK = smem_addr(sK);
      const uint32_t aV = smem_addr(sV);
      bool issued_any = false;

      // O += P_jp V_jp, with P_jp read from the TMEM score buffer it replaced.
      auto issue_pv = [&](int jp) -> bool {
        const int bp = jp & 1;
        const int sp = jp % Lay::kStages;
        if (!wait_phase(&bars->v_full[sp], (jp / Lay::kStages) & 1, bars, limit, kSiteKvFull))
          return false;
        if (!wait_phase(&bars->p_ready[bp], (jp >> 1) & 1, bars, limit, kSitePReady))
          return false;
        tc_fence_after();
        const uint32_t tP = bp ? tS1 : tS0;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          // V tile, keys kk*16 .. +16: 16 rows of 128 B per 64-wide chunk,
          // chunks 64 elements of D apart (LBO), 8-row groups 1 KB apart (SBO).
          const uint64_t bdesc = smem_desc_sw128(
              aV + sp * Lay::kTileBytes + kk * 16 * 128, Lay::kChunkBytes, 1024);
          mma_ts(tO, tP + kk * 8, bdesc, idPV, (jp > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->pv_done);
        mma_commit(&bars->kv_empty[sp]);
        return true;
      };

      bool ok = wait_phase(&bars->q_full, 0, bars, limit, kSiteQFull);
      if (ok) {
        tc_fence_after();
        for (int j = 0; j < n_kv && ok; ++j) {
          const int s = j % Lay::kStages;
          if (!wait_phase(&bars->k_full[s], (j / Lay::kStages) & 1, bars, limit,
                          kSiteKvFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tS = (j & 1) ? tS1 : tS0;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int c = kk >> 2;              // which 64-wide chunk of D
            const int koff = (kk & 3) * 32;     // 16 elements = 32 B inside the atom
            const uint64_t adesc = smem_desc_sw128(aQ + c * Lay::kChunkBytes + koff, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(
                aK + s * Lay::kTileBytes + c * Lay::kChunkBytes + koff, 16, 1024);
            mma_ss(tS, adesc, bdesc, idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[j & 1]);
          issued_any = true;
          if (j > 0 && !issue_pv(j - 1)) ok = false;
        }
        if (ok && n_kv > 0) ok = issue_pv(n_kv - 1);
      }
      if (issued_any) {
        // Everything issued must finish before TMEM is released.
        mma_commit(&bars->fin);
        wait_phase(&bars->fin, 0, bars, limit, kSiteDrain, false);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------- softmax / output warps
    const int wq = warp & 3;
    const int r = wq * 32 + lane;            // row in tile == TMEM lane
    const int row_g = q_tile * kBlockM + r;  // query index in [0, L) when valid
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 >= 0.0f;
    const float mval = pos_scale ? -INFINITY : INFINITY;  // a removed raw score
    float m_used = -INFINITY;  // running max actually used in the exponentials
    float l = 0.0f;            // running row sum of probabilities
    bool ok = true;

    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      const uint32_t tS = (b ? tS1 : tS0) + lane_off;
      if (!warp_wait_phase(&bars->s_full[b], (j >> 1) & 1, bars, limit, kSiteSFull)) {
        ok = false;
        break;
      }
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
      const int col0 = j * kBlockN;
      const bool tail = col0 + kBlockN > p.L;
      const bool masked_tile = (MODE == sdpa_impl::kMaskExplicit) || tail ||
                               (MODE == sdpa_impl::kMaskCausal && j == q_tile);
      if (masked_tile) {
        if constexpr (MODE == sdpa_impl::kMaskExplicit) {
          uint32_t mw[kBlockN / 4];
          if (row_g < p.L) {
            const uint8_t* mrow = p.mask + static_cast<int64_t>(row_g) * p.L + col0;
            if (p.mask_vec16 && !tail) {
#pragma unroll
              for (int v = 0; v < kBlockN / 16; ++v) {
                const uint4 x = __ldg(reinterpret_cast<const uint4*>(mrow) + v);
                mw[4 * v + 0] = x.x;
                mw[4 * v + 1] = x.y;
                mw[4 * v + 2] = x.z;
                mw[4 * v + 3] = x.w;
              }
            } else {
#pragma unroll
              for (int w = 0; w < kBlockN / 4; ++w) {
                uint32_t word = 0;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  const int c = 4 * w + t;
                  const uint32_t byte = (col0 + c < p.L) ? __ldg(mrow + c) : 1u;
                  word |= (byte != 0 ? 1u : 0u) << (8 * t);
                }
                mw[w] = word;
              }
            }
          } else {
#pragma unroll
            for (int w = 0; w < kBlockN / 4; ++w) mw[w] = 0x01010101u;
          }
#pragma unroll
          for (int c = 0; c < kBlockN; ++c) {
            const bool removed =
                (col0 + c >= p.L) || (((mw[c >> 2] >> (8 * (c & 3))) & 0xffu) != 0u);
            s[c] = removed ? mval : s[c];
          }
        } else {
#pragma unroll
          for (int c = 0; c < kBlockN; ++c) {
            const bool removed = (col0 + c >= p.L) ||
                                 (MODE == sdpa_impl::kMaskCausal && col0 + c > row_g);
            s[c] = removed ? mval : s[c];
          }
        }
      }

      // Row extremum of the raw scores (max for a positive scale).
      float ext = s[0];
      if (pos_scale) {
#pragma unroll
        for (int c = 1; c < kBlockN; ++c) ext = fmaxf(ext, s[c]);
      } else {
#pragma unroll
        for (int c = 1; c < kBlockN; ++c) ext = fminf(ext, s[c]);
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

      uint32_t pk[kBlockN / 2];
      float rs = 0.0f;
#pragma unroll
      for (int c = 0; c < kBlockN / 2; ++c) {
        float p0 = ex2(fmaf(s[2 * c], sl2, neg_m));
        float p1 = ex2(fmaf(s[2 * c + 1], sl2, neg_m));
        if (masked_tile) {
          p0 = (s[2 * c] == mval) ? 0.0f : p0;
          p1 = (s[2 * c + 1] == mval) ? 0.0f : p1;
        }
        rs += p0 + p1;
        pk[c] = pack2<BF16>(p0, p1);
      }
      l += rs;
      // P_j overwrites the first 64 columns of its own score buffer.
      tmem_st32(tS + 0, pk);
      tmem_st32(tS + 32, pk + 32);

      if (j > 0) {
        // Consume PV_{j-1}'s completion in order (keeps phase parity exact);
        // it is needed anyway before O may be rescaled.
        if (!warp_wait_phase(&bars->pv_done, (j - 1) & 1, bars, limit, kSitePvDone)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
            tmem_st32(tO + lane_off + c * 32, o);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_ready[b]);
    }

    if (ok && n_kv > 0 &&
        warp_wait_phase(&bars->pv_done, (n_kv - 1) & 1, bars, limit, kSitePvDone)) {
      tc_fence_after();
      const float inv_l = (l > 0.0f) ? (1.0f / l) : 0.0f;
      using elem_t = uint16_t;
      elem_t* orow = reinterpret_cast<elem_t*>(p.out) + batch * p.o_sb + head * p.o_sh +
                     static_cast<int64_t>(row_g) * p.o_sl;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          w[t] = pack2<BF16>(__uint_as_float(o[2 * t]) * inv_l,
                             __uint_as_float(o[2 * t + 1]) * inv_l);
        if (row_g < p.L) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int MODE, bool BF16>
cudaError_t launch_one(const sdpa_impl::FwdParams& p, cudaStream_t stream) {
  auto kern = sdpa_fwd_kernel<D, MODE, BF16>;
  constexpr int smem = Layout<D>::kTotal;
  static bool configured = false;  // one attribute call per instantiation
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(static_cast<unsigned>(p.n_tiles) * static_cast<unsigned>(p.B * p.H));
  kern<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_mode(const sdpa_impl::FwdParams& p, int mode, cudaStream_t stream) {
  switch (mode) {
    case sdpa_impl::kMaskCausal:
      return launch_one<D, sdpa_impl::kMaskCausal, BF16>(p, stream);
    case sdpa_impl::kMaskExplicit:
      return launch_one<D, sdpa_impl::kMaskExplicit, BF16>(p, stream);
    default:
      return launch_one<D, sdpa_impl::kMaskNone, BF16>(p, stream);
  }
}

}  // namespace

namespace sdpa_impl {

cudaError_t launch_forward(const FwdParams& p, int head_dim, int mask_mode, bool bf16,
                           cudaStream_t stream) {
  if (head_dim == 64)
    return bf16 ? launch_mode<64, true>(p, mask_mode, stream)
                : launch_mode<64, false>(p, mask_mode, stream);
  return bf16 ? launch_mode<128, true>(p, mask_mode, stream)
              : launch_mode<128, false>(p, mask_mode, stream);
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
