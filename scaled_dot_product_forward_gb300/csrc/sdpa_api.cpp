// sdpa_api.cpp -- C-ABI front end: argument validation, the rank-3 / rank-4
// stride normaliser, TMA descriptor encoding and the single kernel launch.
//
// Rank-3 inputs [H, L, D] become [1, H, L, D] here and then follow exactly the
// rank-4 path, so both ranks reach the same fused kernel with the same
// per-head arithmetic -- the behaviour that "PyTorch 2.14 SDPA: rank-3 inputs
// now take the fused kernels" (daker.dacon.io) describes as the fix for
// rank-3 inputs silently falling back to the slow math path.  There is no
// fallback of any kind: an unsupported layout is an error, never a slower
// route.
#include "../../include/sdpa.h"

#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include <cuda.h>
#include <cuda_runtime.h>

#include "sdpa_internal.h"

namespace {

constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;  // 1 s per barrier wait
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int> g_withhold_q{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Per-device answer to "is this an sm_103 part?" (0 unknown, 1 yes, 2 no),
// and its SM count (the persistent grid's size).
std::atomic<int> g_device_ok[64];
std::atomic<int> g_device_sms[64];

sdpa_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDPA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SDPA_ERR_DEVICE;
  int state = g_device_ok[dev].load(std::memory_order_relaxed);
  if (state == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SDPA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SDPA_ERR_CUDA;
    state = (major == 10 && minor == 3 && sms > 0) ? 1 : 2;
    g_device_sms[dev].store(sms, std::memory_order_relaxed);
    g_device_ok[dev].store(state, std::memory_order_relaxed);
  }
  return state == 1 ? SDPA_OK : SDPA_ERR_DEVICE;
}

// One operand after normalisation to rank 4: extents and element strides in
// (B, H, L, D) order.
struct View {
  const void* ptr;
  int64_t ext[4];
  int64_t str[4];
};

// Byte span [lo, hi) touched by a 16-bit view (strides are non-negative).
void span_of(const View& v, uintptr_t* lo, uintptr_t* hi) {
  uint64_t last = 0;
  for (int i = 0; i < 4; ++i) last += static_cast<uint64_t>(v.ext[i] - 1) * v.str[i];
  *lo = reinterpret_cast<uintptr_t>(v.ptr);
  *hi = *lo + 2 * (last + 1);
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
  return a0 < b1 && b0 < a1;
}

sdpa_status normalise(const void* ptr, int rank, const int64_t* shape, const int64_t* stride,
                      View* out) {
  out->ptr = ptr;
  const int off = 4 - rank;  // rank 3 -> batch extent 1
  for (int i = 0; i < 4; ++i) {
    out->ext[i] = (i < off) ? 1 : shape[i - off];
    out->str[i] = (i < off) ? 0 : stride[i - off];
  }
  return SDPA_OK;
}

sdpa_status check_layout(View* v) {
  if ((reinterpret_cast<uintptr_t>(v->ptr) & 15u) != 0) return SDPA_ERR_LAYOUT;
  if (v->str[3] != 1) return SDPA_ERR_LAYOUT;
  // Extent-1 dimensions: their stride is never used; give them a harmless
  // outermost value so the tensor map stays valid.
  int64_t outer = 8;
  for (int i = 0; i < 3; ++i)
    if (v->ext[i] > 1) {
      const int64_t s = v->str[i];
      if (s <= 0 || (s % 8) != 0) return SDPA_ERR_LAYOUT;
      if (s >= (int64_t(1) << 38)) return SDPA_ERR_LAYOUT;  // TMA stride < 2^40 bytes
      if (v->ext[i] >= (int64_t(1) << 24) && s >= (int64_t(1) << 24)) return SDPA_ERR_LAYOUT;
      if (s * v->ext[i] > outer) outer = s * v->ext[i];
    }
  for (int i = 0; i < 3; ++i)
    if (v->ext[i] == 1) v->str[i] = outer;
  return SDPA_OK;
}

// 4-D tiled TMA map over one operand.  Dimension 0 is D (contiguous); L, H and
// B follow in increasing stride order.  The box is 64 elements of D (one
// 128-byte swizzle atom) by 128 rows of L.  pos[] receives the map slot of
// (L, H, B) so the kernel can place its coordinates.
sdpa_status encode_map(const View& v, bool bf16, CUtensorMap* map, int pos[3]) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return SDPA_ERR_CUDA;
  // logical outer dims: 0 = L, 1 = H, 2 = B with extents/strides from the view
  const int64_t ext[3] = {v.ext[2], v.ext[1], v.ext[0]};
  const int64_t str[3] = {v.str[2], v.str[1], v.str[0]};
  int order[3] = {0, 1, 2};
  for (int a = 0; a < 3; ++a)  // stable insertion sort by stride
    for (int b = a + 1; b < 3; ++b)
      if (str[order[b]] < str[order[a]]) {
        const int t = order[a];
        order[a] = order[b];
        order[b] = t;
      }
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(v.ext[3]), 0, 0, 0};
  cuuint64_t gstride[3];
  cuuint32_t box[4] = {64, 1, 1, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  for (int slot = 1; slot <= 3; ++slot) {
    const int d = order[slot - 1];
    gdim[slot] = static_cast<cuuint64_t>(ext[d]);
    gstride[slot - 1] = static_cast<cuuint64_t>(str[d]) * 2u;
    box[slot] = (d == 0) ? 128u : 1u;
    pos[d] = slot;
  }
  const CUresult r =
      enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
          const_cast<void*>(v.ptr), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SDPA_OK : SDPA_ERR_LAYOUT;
}

// Host-side validation shared by every entry point.  Touches no CUDA API.
sdpa_status validate(const void* q, const void* k, const void* v, void* out, sdpa_dtype dtype,
                     int rank, const int64_t* shape, const int64_t* q_stride,
                     const int64_t* k_stride, const int64_t* v_stride, const int64_t* o_stride,
                     int is_causal, const uint8_t* mask, float scale, View views[4]) {
  if (!q || !k || !v || !out || !shape || !q_stride || !k_stride || !v_stride || !o_stride)
    return SDPA_ERR_NULL;
  if (rank != 3 && rank != 4) return SDPA_ERR_RANK;
  if (dtype != SDPA_BF16 && dtype != SDPA_FP16) return SDPA_ERR_DTYPE;
  for (int i = 0; i < rank; ++i)
    if (shape[i] < 1) return SDPA_ERR_SHAPE;
  const int64_t B = (rank == 4) ? shape[0] : 1;
  const int64_t H = shape[rank - 3], L = shape[rank - 2], D = shape[rank - 1];
  if (D != 64 && D != 128) return SDPA_ERR_SHAPE;
  if (L > 0x7fffffffLL - 127) return SDPA_ERR_SHAPE;
  if (B * H > 0x7fffffffLL / ((L + 127) / 128)) return SDPA_ERR_SHAPE;  // tile and unit counts fit in int
  const void* ptrs[4] = {q, k, v, out};
  const int64_t* strides[4] = {q_stride, k_stride, v_stride, o_stride};
  for (int t = 0; t < 4; ++t) {
    normalise(ptrs[t], rank, shape, strides[t], &views[t]);
    const sdpa_status s = check_layout(&views[t]);
    if (s != SDPA_OK) return s;
  }
  if (is_causal && mask) return SDPA_ERR_ARG;
  if (std::isinf(scale)) return SDPA_ERR_ARG;
  // out must not alias any input (the kernel reads inputs while writing out)
  uintptr_t o0, o1;
  View raw_out;
  normalise(out, rank, shape, o_stride, &raw_out);
  span_of(raw_out, &o0, &o1);
  for (int t = 0; t < 3; ++t) {
    View raw;
    normalise(ptrs[t], rank, shape, strides[t], &raw);
    uintptr_t a0, a1;
    span_of(raw, &a0, &a1);
    if (overlaps(o0, o1, a0, a1)) return SDPA_ERR_ARG;
  }
  if (mask) {
    const uintptr_t m0 = reinterpret_cast<uintptr_t>(mask);
    const uintptr_t m1 = m0 + static_cast<uintptr_t>(L) * static_cast<uintptr_t>(L);
    if (overlaps(o0, o1, m0, m1)) return SDPA_ERR_ARG;
  }
  return SDPA_OK;
}


// Optional log-sum-exp output: fp32, rank - 1 extents (the shape without D),
// element strides, 4-byte aligned, not overlapping any other operand.
sdpa_status check_lse(const float* lse, int rank, const int64_t* shape, const int64_t* stride,
                      const View views[4], const uint8_t* mask, int64_t out_stride[3]) {
  if (!stride) return SDPA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return SDPA_ERR_LAYOUT;
  const int off = 4 - rank;  // rank 3: batch extent 1
  uint64_t last = 0;
  for (int i = 0; i < 3; ++i) {
    const int64_t ext = (i < off) ? 1 : shape[i - off];
    const int64_t st = (i < off) ? 0 : stride[i - off];
    if (ext > 1 && st <= 0) return SDPA_ERR_LAYOUT;
    out_stride[i] = (ext > 1) ? st : 0;
    last += static_cast<uint64_t>(ext - 1) * static_cast<uint64_t>(out_stride[i]);
  }
  const uintptr_t l0 = reinterpret_cast<uintptr_t>(lse), l1 = l0 + 4 * (last + 1);
  for (int t = 0; t < 4; ++t) {
    uintptr_t a0, a1;
    span_of(views[t], &a0, &a1);
    if (overlaps(l0, l1, a0, a1)) return SDPA_ERR_ARG;
  }
  if (mask) {
    const int64_t L = views[0].ext[2];
    const uintptr_t m0 = reinterpret_cast<uintptr_t>(mask);
    if (overlaps(l0, l1, m0, m0 + static_cast<uintptr_t>(L) * static_cast<uintptr_t>(L)))
      return SDPA_ERR_ARG;
  }
  return SDPA_OK;
}

// Everything a launch needs, built once from validated arguments.
struct Prepared {
  sdpa_impl::FwdParams p;
  View views[4];
  int mode;
  int head_dim;
  bool bf16;
  int device;
  int sms;  // SM count of that device (persistent grid size)
};

sdpa_status build_params(const void* q, const void* k, const void* v, void* out, sdpa_dtype dtype,
                         int rank, const int64_t* shape, const int64_t* q_stride,
                         const int64_t* k_stride, const int64_t* v_stride,
                         const int64_t* o_stride, int is_causal, const uint8_t* mask, float scale,
                         Prepared* pr) {
  sdpa_status s = validate(q, k, v, out, dtype, rank, shape, q_stride, k_stride, v_stride,
                           o_stride, is_causal, mask, scale, pr->views);
  if (s != SDPA_OK) return s;
  s = check_device();
  if (s != SDPA_OK) return s;
  if (cudaGetDevice(&pr->device) != cudaSuccess) return SDPA_ERR_CUDA;
  pr->sms = g_device_sms[pr->device].load(std::memory_order_relaxed);

  pr->bf16 = (dtype == SDPA_BF16);
  const View* views = pr->views;
  const int64_t B = views[0].ext[0], H = views[0].ext[1], L = views[0].ext[2],
                D = views[0].ext[3];
  sdpa_impl::FwdParams& p = pr->p;
  std::memset(&p, 0, sizeof(p));
  if ((s = encode_map(views[0], pr->bf16, &p.tm_q, p.pos_q)) != SDPA_OK) return s;
  if ((s = encode_map(views[1], pr->bf16, &p.tm_k, p.pos_k)) != SDPA_OK) return s;
  if ((s = encode_map(views[2], pr->bf16, &p.tm_v, p.pos_v)) != SDPA_OK) return s;
  p.out = out;
  p.o_sb = views[3].str[0];
  p.o_sh = views[3].str[1];
  p.o_sl = views[3].str[2];
  p.mask = mask;
  p.B = static_cast<int>(B);
  p.H = static_cast<int>(H);
  p.L = static_cast<int>(L);
  p.n_tiles = static_cast<int>((L + 127) / 128);
  const double sc = std::isnan(scale) ? 1.0 / std::sqrt(static_cast<double>(D))
                                      : static_cast<double>(scale);
  p.scale_log2 = static_cast<float>(sc * 1.4426950408889634);  // log2(e)
  // A zero scale makes every admissible weight exp(0) = 1.  The kernel needs
  // a nonzero multiplier (a removed score is an infinity that must map to
  // -inf), so it gets the smallest normal float instead: every finite score
  // times it rounds the exponent to 0 and the weights are exactly 1.0f.
  if (p.scale_log2 == 0.0f) p.scale_log2 = std::signbit(sc) ? -FLT_MIN : FLT_MIN;
  p.mask_vec16 = (mask && (L % 16) == 0 && (reinterpret_cast<uintptr_t>(mask) & 15u) == 0);
  pr->mode = is_causal ? sdpa_impl::kMaskCausal
                       : (mask ? sdpa_impl::kMaskExplicit : sdpa_impl::kMaskNone);
  // Job order: when every head's K and V fit in L2 together (here: at most
  // 48 MB, of the 129 MB), deal jobs by falling cost for balance; beyond
  // that, keep each head's jobs together for K/V reuse in L2.
  const double kv_bytes = 2.0 * 2.0 * static_cast<double>(B) * static_cast<double>(H) *
                          static_cast<double>(L) * static_cast<double>(D);
  p.snake = kv_bytes <= 48.0 * 1024 * 1024 ? 1 : 0;
  pr->head_dim = static_cast<int>(D);
  return SDPA_OK;
}

sdpa_status launch_prepared(const Prepared& pr, void* stream) {
  sdpa_impl::FwdParams p = pr.p;
  p.debug_withhold_q = g_withhold_q.load(std::memory_order_relaxed);
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  if (p.tile_class != nullptr) {
    // The mask summary is rebuilt from the mask on every launch (the mask's
    // contents may change between launches); the forward waits for it.
    sdpa_impl::MaskTilesParams mt{};
    mt.mask = p.mask;
    mt.L = p.L;
    mt.n_tiles = p.n_tiles;
    mt.vec16 = p.mask_vec16;
    mt.bits = reinterpret_cast<uint16_t*>(const_cast<uint4*>(p.tile_bits));
    mt.tile_class = const_cast<uint8_t*>(p.tile_class);
    if (sdpa_impl::launch_mask_tiles(mt, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return SDPA_ERR_CUDA;
  }
  const cudaError_t e = sdpa_impl::launch_forward(p, pr.head_dim, pr.mode, pr.bf16, pr.sms,
                                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

// Bytes of a mask summary for an [L, L] mask: 2 KB of row bits and one class
// byte per 128 x 128 tile.
uint64_t mask_tiles_bytes(int64_t L) {
  const uint64_t n = static_cast<uint64_t>((L + 127) / 128);
  return n * n * (128u * 16u + 1u);
}

using ReplaceAddressFn = CUresult (*)(CUtensorMap*, void*);

ReplaceAddressFn get_replace_fn() {
  static std::once_flag once;
  static ReplaceAddressFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapReplaceAddress", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<ReplaceAddressFn>(ptr);
  });
  return fn;
}

// A tiled map of `rank` dims (dim 0 contiguous, 16-bit elements) with the
// given extents, byte strides of dims 1.., and box; 128-byte swizzle, zero
// fill out of bounds.
sdpa_status encode_nd(const void* ptr, bool bf16, int rank, const cuuint64_t* gdim,
                      const cuuint64_t* gstride_bytes, const cuuint32_t* box, CUtensorMap* map) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return SDPA_ERR_CUDA;
  cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  const CUresult r =
      enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
          static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), gdim, gstride_bytes, box,
          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SDPA_OK : SDPA_ERR_LAYOUT;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool stride_ok(int64_t st) { return st > 0 && (st % 8) == 0; }

// [a, a + bytes) as a span for the overlap checks.
void span(const void* a, uint64_t bytes, uintptr_t* lo, uintptr_t* hi) {
  *lo = reinterpret_cast<uintptr_t>(a);
  *hi = *lo + static_cast<uintptr_t>(bytes);
}

}  // namespace

struct sdpa_plan {
  Prepared pr;
  int64_t shape[4];
  int64_t strides[4][4];
  int rank;
  int is_causal;
  float scale;
  sdpa_dtype dtype;
  void* mask_tiles = nullptr;  // device: the mask summary (masked plans only)

  ~sdpa_plan() {
    if (mask_tiles == nullptr) return;
    int cur = -1;
    const bool restore = cudaGetDevice(&cur) == cudaSuccess && cur != pr.device;
    if (restore) cudaSetDevice(pr.device);
    cudaFree(mask_tiles);
    if (restore) cudaSetDevice(cur);
  }
};

extern "C" {

sdpa_status sdpa_forward(const void* q, const void* k, const void* v, void* out,
                         sdpa_dtype dtype, int rank, const int64_t* shape,
                         const int64_t* q_stride, const int64_t* k_stride,
                         const int64_t* v_stride, const int64_t* o_stride, int is_causal,
                         const uint8_t* mask, float scale, void* stream) {
  Prepared pr;
  const sdpa_status s = build_params(q, k, v, out, dtype, rank, shape, q_stride, k_stride,
                                     v_stride, o_stride, is_causal, mask, scale, &pr);
  if (s != SDPA_OK) return s;
  return launch_prepared(pr, stream);
}

sdpa_status sdpa_forward_masked_noalloc(const void* q, const void* k, const void* v, void* out,
                                        sdpa_dtype dtype, int rank, const int64_t* shape,
                                        const int64_t* q_stride, const int64_t* k_stride,
                                        const int64_t* v_stride, const int64_t* o_stride,
                                        const uint8_t* mask, float scale, void* stream) {
  if (!mask) return SDPA_ERR_NULL;
  Prepared pr;
  const sdpa_status s = build_params(q, k, v, out, dtype, rank, shape, q_stride, k_stride,
                                     v_stride, o_stride, 0, mask, scale, &pr);
  if (s != SDPA_OK) return s;
  if (pr.p.L > SDPA_NOALLOC_MAX_L) return SDPA_ERR_SHAPE;  // beyond the fixed scratch
  const uint4* bits = nullptr;
  const uint8_t* cls = nullptr;
  if (sdpa_impl::noalloc_mask_tiles(pr.device, &bits, &cls) != cudaSuccess) return SDPA_ERR_CUDA;
  pr.p.tile_bits = bits;
  pr.p.tile_class = cls;
  return launch_prepared(pr, stream);
}

sdpa_status sdpa_forward_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                             sdpa_dtype dtype, int rank, const int64_t* shape,
                             const int64_t* q_stride, const int64_t* k_stride,
                             const int64_t* v_stride, const int64_t* o_stride,
                             const int64_t* lse_stride, int is_causal, const uint8_t* mask,
                             float scale, void* stream) {
  if (!lse) return SDPA_ERR_NULL;
  Prepared pr;
  sdpa_status s = validate(q, k, v, out, dtype, rank, shape, q_stride, k_stride, v_stride,
                           o_stride, is_causal, mask, scale, pr.views);
  if (s != SDPA_OK) return s;
  int64_t ls[3];
  if ((s = check_lse(lse, rank, shape, lse_stride, pr.views, mask, ls)) != SDPA_OK) return s;
  s = build_params(q, k, v, out, dtype, rank, shape, q_stride, k_stride, v_stride, o_stride,
                   is_causal, mask, scale, &pr);
  if (s != SDPA_OK) return s;
  pr.p.lse = lse;
  pr.p.lse_sb = ls[0];
  pr.p.lse_sh = ls[1];
  pr.p.lse_sl = ls[2];
  return launch_prepared(pr, stream);
}

sdpa_status sdpa_forward_varlen(const void* q, const void* k, const void* v, void* out,
                                float* lse, sdpa_dtype dtype, int64_t total, int64_t n_heads,
                                int64_t head_dim, const int64_t* q_stride,
                                const int64_t* k_stride, const int64_t* v_stride,
                                const int64_t* o_stride, const int64_t* lse_stride,
                                const int32_t* cu_seqlens, int64_t n_seqs, int64_t max_seqlen,
                                int is_causal, float scale, void* stream) {
  if (!cu_seqlens || !q_stride || !k_stride || !v_stride || !o_stride) return SDPA_ERR_NULL;
  if (n_seqs < 1 || n_seqs > 0x7fffffffLL - 64 || max_seqlen < 1) return SDPA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return SDPA_ERR_LAYOUT;
  // [total, H, D] with (token, head, dim) strides is the rank-3 view
  // [H, total, D] with (head, token, dim) strides.
  const int64_t shape[3] = {n_heads, total, head_dim};
  const int64_t qs[3] = {q_stride[1], q_stride[0], q_stride[2]};
  const int64_t ks[3] = {k_stride[1], k_stride[0], k_stride[2]};
  const int64_t vs[3] = {v_stride[1], v_stride[0], v_stride[2]};
  const int64_t os[3] = {o_stride[1], o_stride[0], o_stride[2]};
  Prepared pr;
  sdpa_status s = validate(q, k, v, out, dtype, 3, shape, qs, ks, vs, os, is_causal, nullptr,
                           scale, pr.views);
  if (s != SDPA_OK) return s;
  {
    // the offsets are read by the kernel while it writes out
    uintptr_t o0, o1;
    span_of(pr.views[3], &o0, &o1);
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(cu_seqlens);
    if (overlaps(o0, o1, c0, c0 + 4 * static_cast<uintptr_t>(n_seqs + 1))) return SDPA_ERR_ARG;
  }
  int64_t ls[3] = {0, 0, 0};
  if (lse) {
    if (!lse_stride) return SDPA_ERR_NULL;
    if ((s = check_lse(lse, 3, shape, lse_stride, pr.views, nullptr, ls)) != SDPA_OK) return s;
    const uintptr_t l0 = reinterpret_cast<uintptr_t>(lse);
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(cu_seqlens);
    if (overlaps(l0, l0 + 4 * static_cast<uintptr_t>((n_heads - 1) * ls[1] + (total - 1) * ls[2] + 1),
                 c0, c0 + 4 * static_cast<uintptr_t>(n_seqs + 1)))
      return SDPA_ERR_ARG;
  }
  s = build_params(q, k, v, out, dtype, 3, shape, qs, ks, vs, os, is_causal, nullptr, scale, &pr);
  if (s != SDPA_OK) return s;
  pr.p.cu_seqlens = cu_seqlens;
  pr.p.n_seqs = static_cast<int>(n_seqs);
  // Grid bound: every sequence at most max_seqlen rows (a smaller bound only
  // means fewer CTAs, never missed work: each CTA walks all its units).
  const int64_t ml = max_seqlen < total ? max_seqlen : total;
  const int64_t uph = (((ml + 127) / 128 + 1) / 2 + 1) / 2;
  const double bound = static_cast<double>(n_seqs) * static_cast<double>(n_heads) *
                       static_cast<double>(uph);
  pr.p.max_units = bound > 2.0e9 ? 2000000000LL : static_cast<long long>(bound);
  if (lse) {
    pr.p.lse = lse;
    pr.p.lse_sb = ls[0];
    pr.p.lse_sh = ls[1];
    pr.p.lse_sl = ls[2];
  }
  return launch_prepared(pr, stream);
}

sdpa_status sdpa_sparse_forward(const void* q, const void* k, const void* v, void* out, float* lse,
                                sdpa_dtype dtype, int64_t total_q, int64_t total_k,
                                int64_t n_heads, int64_t head_dim, const int64_t* q_stride,
                                int64_t k_stride, int64_t v_stride, const int64_t* o_stride,
                                const int64_t* lse_stride, const int32_t* idx, int64_t idx_stride,
                                int64_t topk, const int32_t* topk_length, float scale,
                                void* stream) {
  if (!q || !k || !v || !out || !idx || !q_stride || !o_stride) return SDPA_ERR_NULL;
  if (lse && !lse_stride) return SDPA_ERR_NULL;
  if (dtype != SDPA_BF16 && dtype != SDPA_FP16) return SDPA_ERR_DTYPE;
  if (head_dim != 64 && head_dim != 128) return SDPA_ERR_SHAPE;
  if (total_q < 1 || total_k < 1 || n_heads < 1 || topk < 1) return SDPA_ERR_SHAPE;
  const int64_t n_groups = (n_heads + 127) / 128;
  if (total_k > 0x7fffffffLL || topk > 0x7fffffffLL - 256 || n_heads > 0x7fffffffLL ||
      total_q > 0x7fffffffLL / n_groups)
    return SDPA_ERR_SHAPE;
  // layouts: 16-byte aligned rows (TMA), 4-byte aligned index arrays
  const int64_t sq_t = q_stride[0], sq_h = (n_heads > 1) ? q_stride[1] : head_dim;
  const int64_t so_t = o_stride[0], so_h = (n_heads > 1) ? o_stride[1] : head_dim;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return SDPA_ERR_LAYOUT;
  if ((total_q > 1 && !stride_ok(sq_t)) || !stride_ok(sq_h) || !stride_ok(so_h) ||
      (total_q > 1 && !stride_ok(so_t)))
    return SDPA_ERR_LAYOUT;
  if ((total_k > 1 && (!stride_ok(k_stride) || !stride_ok(v_stride))) || !aligned4(idx) ||
      (topk_length && !aligned4(topk_length)) || (total_q > 1 && idx_stride < topk))
    return SDPA_ERR_LAYOUT;
  if (lse && (!aligned4(lse) || (n_heads > 1 && lse_stride[1] <= 0) ||
              (total_q > 1 && lse_stride[0] <= 0)))
    return SDPA_ERR_LAYOUT;
  if (std::isinf(scale)) return SDPA_ERR_ARG;
  // out (and lse) must not overlap anything the kernel reads
  {
    const uint64_t ob = 2ull * static_cast<uint64_t>((total_q - 1) * so_t + (n_heads - 1) * so_h +
                                                     head_dim);
    uintptr_t o0, o1, a0, a1;
    span(out, ob, &o0, &o1);
    const void* ins[5] = {q, k, v, idx, topk_length};
    const uint64_t inb[5] = {
        2ull * static_cast<uint64_t>((total_q - 1) * sq_t + (n_heads - 1) * sq_h + head_dim),
        2ull * static_cast<uint64_t>((total_k - 1) * k_stride + head_dim),
        2ull * static_cast<uint64_t>((total_k - 1) * v_stride + head_dim),
        4ull * static_cast<uint64_t>((total_q - 1) * idx_stride + topk),
        4ull * static_cast<uint64_t>(total_q)};
    for (int t = 0; t < 5; ++t) {
      if (!ins[t]) continue;
      span(ins[t], inb[t], &a0, &a1);
      if (overlaps(o0, o1, a0, a1)) return SDPA_ERR_ARG;
    }
    if (lse) {
      const int64_t lh = (n_heads > 1) ? lse_stride[1] : 0, lt = (total_q > 1) ? lse_stride[0] : 0;
      uintptr_t l0, l1;
      span(lse, 4ull * static_cast<uint64_t>((total_q - 1) * lt + (n_heads - 1) * lh + 1), &l0,
           &l1);
      if (overlaps(l0, l1, o0, o1)) return SDPA_ERR_ARG;
      for (int t = 0; t < 5; ++t) {
        if (!ins[t]) continue;
        span(ins[t], inb[t], &a0, &a1);
        if (overlaps(l0, l1, a0, a1)) return SDPA_ERR_ARG;
      }
    }
  }
  sdpa_status s = check_device();
  if (s != SDPA_OK) return s;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDPA_ERR_CUDA;
  const bool bf16 = (dtype == SDPA_BF16);
  sdpa_impl::SparseParams p;
  std::memset(&p, 0, sizeof(p));
  {
    // Q: (D, H, total_q); box 64 x 128 heads x 1 row (heads past H read as 0)
    const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(head_dim),
                                static_cast<cuuint64_t>(n_heads),
                                static_cast<cuuint64_t>(total_q)};
    const cuuint64_t gst[2] = {static_cast<cuuint64_t>(sq_h) * 2u,
                               static_cast<cuuint64_t>(total_q > 1 ? sq_t : sq_h * n_heads) * 2u};
    // With fewer than 128 heads the box is H rows (the tile's other rows
    // are never stored).  With at most 64, the kernel runs its half-row form
    // (M = 64 products, two softmax threads a row).
    p.q_rows = static_cast<int>(n_heads < 128 ? n_heads : 128);
    p.q_half = (n_heads <= 64) ? 1 : 0;
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(p.q_rows), 1};
    if ((s = encode_nd(q, bf16, 3, gdim, gst, box, &p.tm_q)) != SDPA_OK) return s;
  }
  p.out = out;
  p.o_st = so_t;
  p.o_sh = so_h;
  p.lse = lse;
  if (lse) {
    p.lse_st = (total_q > 1) ? lse_stride[0] : 0;
    p.lse_sh = (n_heads > 1) ? lse_stride[1] : 0;
  }
  p.kv_shared = (k == v && (total_k == 1 || k_stride == v_stride)) ? 1 : 0;
  p.k = k;
  p.v = v;
  p.k_row_bytes = 2 * (total_k > 1 ? k_stride : head_dim);
  p.v_row_bytes = 2 * (total_k > 1 ? v_stride : head_dim);
  p.idx = idx;
  p.idx_st = idx_stride;
  p.topk_length = topk_length;
  p.total_q = static_cast<int>(total_q);
  p.total_k = static_cast<int>(total_k);
  p.H = static_cast<int>(n_heads);
  p.topk = static_cast<int>(topk);
  p.n_groups = static_cast<int>(n_groups);
  const double sc = std::isnan(scale) ? 1.0 / std::sqrt(static_cast<double>(head_dim))
                                      : static_cast<double>(scale);
  p.scale_log2 = static_cast<float>(sc * 1.4426950408889634);
  if (p.scale_log2 == 0.0f) p.scale_log2 = std::signbit(sc) ? -FLT_MIN : FLT_MIN;
  p.debug_withhold_q = g_withhold_q.load(std::memory_order_relaxed);
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  const int sms = g_device_sms[dev].load(std::memory_order_relaxed);
  const cudaError_t e = sdpa_impl::launch_sparse(p, static_cast<int>(head_dim), bf16, sms,
                                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

sdpa_status sdpa_sparse_compact(const int32_t* idx_local, int64_t idx_local_stride,
                                int32_t* idx_global, int64_t idx_global_stride,
                                int32_t* topk_length, int64_t total_q, int64_t topk,
                                const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                int64_t n_docs, int is_causal, void* stream) {
  if (!idx_local || !idx_global || !topk_length || !cu_seqlens_q || !cu_seqlens_k)
    return SDPA_ERR_NULL;
  if (total_q < 1 || topk < 1 || n_docs < 1 || total_q > 0x7fffffffLL / 32 ||
      topk > 0x7fffffffLL - 64 || n_docs > 0x7fffffffLL - 1)
    return SDPA_ERR_SHAPE;
  if (!aligned4(idx_local) || !aligned4(idx_global) || !aligned4(topk_length) ||
      !aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k) ||
      (total_q > 1 && (idx_local_stride < topk || idx_global_stride < topk)))
    return SDPA_ERR_LAYOUT;
  {
    // outputs must not overlap inputs or each other
    uintptr_t g0, g1, n0, n1, a0, a1;
    span(idx_global, 4ull * static_cast<uint64_t>((total_q - 1) * idx_global_stride + topk), &g0,
         &g1);
    span(topk_length, 4ull * static_cast<uint64_t>(total_q), &n0, &n1);
    if (overlaps(g0, g1, n0, n1)) return SDPA_ERR_ARG;
    const void* ins[3] = {idx_local, cu_seqlens_q, cu_seqlens_k};
    const uint64_t inb[3] = {
        4ull * static_cast<uint64_t>((total_q - 1) * idx_local_stride + topk),
        4ull * static_cast<uint64_t>(n_docs + 1), 4ull * static_cast<uint64_t>(n_docs + 1)};
    for (int t = 0; t < 3; ++t) {
      span(ins[t], inb[t], &a0, &a1);
      if (overlaps(g0, g1, a0, a1) || overlaps(n0, n1, a0, a1)) return SDPA_ERR_ARG;
    }
  }
  const sdpa_status s = check_device();
  if (s != SDPA_OK) return s;
  sdpa_impl::CompactParams p;
  p.idx_local = idx_local;
  p.in_st = idx_local_stride;
  p.idx_global = idx_global;
  p.out_st = idx_global_stride;
  p.length = topk_length;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.total_q = static_cast<int>(total_q);
  p.topk = static_cast<int>(topk);
  p.n_docs = static_cast<int>(n_docs);
  p.is_causal = is_causal ? 1 : 0;
  return sdpa_impl::launch_compact(p, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SDPA_OK
             : SDPA_ERR_CUDA;
}

sdpa_status sdpa_plan_create(sdpa_plan** plan, const void* q, const void* k, const void* v,
                             void* out, sdpa_dtype dtype, int rank, const int64_t* shape,
                             const int64_t* q_stride, const int64_t* k_stride,
                             const int64_t* v_stride, const int64_t* o_stride, int is_causal,
                             const uint8_t* mask, float scale) {
  if (!plan) return SDPA_ERR_NULL;
  *plan = nullptr;
  sdpa_plan* pl = new (std::nothrow) sdpa_plan;
  if (!pl) return SDPA_ERR_ARG;
  const sdpa_status s = build_params(q, k, v, out, dtype, rank, shape, q_stride, k_stride,
                                     v_stride, o_stride, is_causal, mask, scale, &pl->pr);
  if (s != SDPA_OK) {
    delete pl;
    return s;
  }
  pl->rank = rank;
  pl->is_causal = is_causal;
  pl->scale = scale;
  pl->dtype = dtype;
  if (mask != nullptr && pl->pr.p.n_tiles > 65535) {
    delete pl;
    return SDPA_ERR_SHAPE;
  }
  if (mask != nullptr) {
    // A masked plan owns a summary of its mask (per 128 x 128 tile: the rows
    // as bits and whether the tile removes no, some or every key), rebuilt on
    // each launch; the forward then reads 16 bytes per row and tile instead of
    // 128, skips the select in tiles that remove nothing and skips tiles that
    // remove everything for both query tiles of a job.
    const uint64_t bytes = mask_tiles_bytes(pl->pr.p.L);
    const uint64_t n2 = bytes / (128u * 16u + 1u);
    if (cudaMalloc(&pl->mask_tiles, bytes) != cudaSuccess) {
      pl->mask_tiles = nullptr;
      delete pl;
      return SDPA_ERR_CUDA;
    }
    pl->pr.p.tile_bits = static_cast<const uint4*>(pl->mask_tiles);
    pl->pr.p.tile_class = static_cast<const uint8_t*>(pl->mask_tiles) + n2 * 128u * 16u;
  }
  const int64_t* st[4] = {q_stride, k_stride, v_stride, o_stride};
  for (int i = 0; i < rank; ++i) {
    pl->shape[i] = shape[i];
    for (int t = 0; t < 4; ++t) pl->strides[t][i] = st[t][i];
  }
  *plan = pl;
  return SDPA_OK;
}

sdpa_status sdpa_plan_set_pointers(sdpa_plan* plan, const void* q, const void* k, const void* v,
                                   void* out, const uint8_t* mask) {
  if (!plan) return SDPA_ERR_NULL;
  if ((plan->pr.p.mask != nullptr) != (mask != nullptr)) return SDPA_ERR_ARG;
  // Full validation of the new addresses against the plan's shape and strides.
  View views[4];
  sdpa_status s = validate(q, k, v, out, plan->dtype, plan->rank, plan->shape, plan->strides[0],
                           plan->strides[1], plan->strides[2], plan->strides[3],
                           plan->is_causal, mask, plan->scale, views);
  if (s != SDPA_OK) return s;
  ReplaceAddressFn rep = get_replace_fn();
  if (!rep) return SDPA_ERR_CUDA;
  sdpa_impl::FwdParams p = plan->pr.p;
  if (rep(&p.tm_q, const_cast<void*>(q)) != CUDA_SUCCESS ||
      rep(&p.tm_k, const_cast<void*>(k)) != CUDA_SUCCESS ||
      rep(&p.tm_v, const_cast<void*>(v)) != CUDA_SUCCESS)
    return SDPA_ERR_LAYOUT;
  p.out = out;
  p.mask = mask;
  p.mask_vec16 = (mask && (p.L % 16) == 0 && (reinterpret_cast<uintptr_t>(mask) & 15u) == 0);
  plan->pr.p = p;
  for (int t = 0; t < 4; ++t) plan->pr.views[t] = views[t];
  return SDPA_OK;
}

sdpa_status sdpa_plan_launch(const sdpa_plan* plan, void* stream) {
  if (!plan) return SDPA_ERR_NULL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDPA_ERR_CUDA;
  if (dev != plan->pr.device) return SDPA_ERR_ARG;
  return launch_prepared(plan->pr, stream);
}

sdpa_status sdpa_plan_set_lse(sdpa_plan* plan, float* lse, const int64_t* lse_stride) {
  if (!plan) return SDPA_ERR_NULL;
  if (!lse) {
    plan->pr.p.lse = nullptr;
    return SDPA_OK;
  }
  int64_t ls[3];
  const sdpa_status s = check_lse(lse, plan->rank, plan->shape, lse_stride, plan->pr.views,
                                  plan->pr.p.mask, ls);
  if (s != SDPA_OK) return s;
  plan->pr.p.lse = lse;
  plan->pr.p.lse_sb = ls[0];
  plan->pr.p.lse_sh = ls[1];
  plan->pr.p.lse_sl = ls[2];
  return SDPA_OK;
}

void sdpa_plan_destroy(sdpa_plan* plan) { delete plan; }

sdpa_status sdpa_mask_tiles(const uint8_t* mask, int64_t L, void* tile_bits,
                            uint8_t* tile_class, void* stream) {
  if (!mask || !tile_bits || !tile_class) return SDPA_ERR_NULL;
  if (L < 1 || (L + 127) / 128 > 65535) return SDPA_ERR_SHAPE;
  if (!aligned16(tile_bits)) return SDPA_ERR_LAYOUT;
  sdpa_impl::MaskTilesParams mt{};
  mt.mask = mask;
  mt.L = static_cast<int>(L);
  mt.n_tiles = static_cast<int>((L + 127) / 128);
  mt.vec16 = (L % 16) == 0 && aligned16(mask);
  mt.bits = static_cast<uint16_t*>(tile_bits);
  mt.tile_class = tile_class;
  return sdpa_impl::launch_mask_tiles(mt, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SDPA_OK
             : SDPA_ERR_CUDA;
}

const char* sdpa_status_string(sdpa_status status) {
  switch (status) {
    case SDPA_OK: return "SDPA_OK";
    case SDPA_ERR_NULL: return "SDPA_ERR_NULL: a required pointer is NULL";
    case SDPA_ERR_RANK: return "SDPA_ERR_RANK: rank must be 3 or 4";
    case SDPA_ERR_SHAPE: return "SDPA_ERR_SHAPE: D must be 64 or 128 and every extent >= 1";
    case SDPA_ERR_DTYPE: return "SDPA_ERR_DTYPE: dtype must be SDPA_BF16 or SDPA_FP16";
    case SDPA_ERR_LAYOUT:
      return "SDPA_ERR_LAYOUT: inner stride must be 1, other strides positive multiples of 8 "
             "elements, pointers 16-byte aligned";
    case SDPA_ERR_ARG:
      return "SDPA_ERR_ARG: causal with mask, infinite scale, or out overlapping an input";
    case SDPA_ERR_CUDA: return "SDPA_ERR_CUDA: CUDA runtime or driver error";
    case SDPA_ERR_DEVICE_TIMEOUT:
      return "SDPA_ERR_DEVICE_TIMEOUT: a kernel barrier wait ran out of time";
    case SDPA_ERR_DEVICE: return "SDPA_ERR_DEVICE: the current device is not sm_103";
  }
  return "SDPA_UNKNOWN_STATUS";
}

sdpa_status sdpa_last_device_status_detail(void* stream, uint32_t* detail) {
  unsigned int st = 0, st64 = 0, st_sparse = 0;
  if (sdpa_impl::read_and_clear_device_status(static_cast<cudaStream_t>(stream), &st) !=
          cudaSuccess ||
      sdpa_impl::read_and_clear_fwd64_status(&st64) != cudaSuccess ||
      sdpa_impl::read_and_clear_sparse_status(&st_sparse) != cudaSuccess)
    return SDPA_ERR_CUDA;
  st |= st64 | st_sparse;
  if (detail) *detail = st;
  return st == 0 ? SDPA_OK : SDPA_ERR_DEVICE_TIMEOUT;
}

sdpa_status sdpa_last_device_status(void* stream) {
  return sdpa_last_device_status_detail(stream, nullptr);
}

int sdpa_version(void) { return 100; }

void sdpa_debug_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns == 0 ? kDefaultWaitLimitNs : ns, std::memory_order_relaxed);
}

void sdpa_debug_withhold_q_load(int enable) {
  g_withhold_q.store(enable ? 1 : 0, std::memory_order_relaxed);
}

}  // extern "C"
