/*
 * sdpa.h -- C ABI of the GB300 (sm_103a) fused scaled dot-product attention
 * forward.
 *
 * OPERATION.  For every (batch b, head h) and query row i:
 *
 *     out[b,h,i,:] = sum_j softmax_j( scale * q[b,h,i,:] . k[b,h,j,:]
 *                                     with removed keys at -inf ) * v[b,h,j,:]
 *
 * i.e. the five steps matmul(q, k^T), times scale, masked_fill(mask, -inf),
 * softmax over keys, matmul(attn, v) of the NaiveCausalAttention module in
 * "Profiling attention in PyTorch: kernels, backends and where the time goes"
 * (news.bpdata.com), section "Naiv causal attention", and of section 1 of
 * "PyTorch attention profiling: Flash, cuDNN and Math backends compared"
 * (dev.smart-guide.co.kr).  The user-facing call there is
 * F.scaled_dot_product_attention(q, k, v, is_causal=True) (same pages, SDPA
 * sections); this ABI takes the same arguments as raw device pointers.
 *
 *   - causal (is_causal != 0): query i sees keys j <= i.
 *   - explicit mask: mask[i*L + j] != 0 removes key j for query i, the
 *     masked_fill polarity (1 = masked out).  One [L, L] mask serves every
 *     (b, h).
 *   - a query with no admissible key yields a zero row (the math backend's
 *     "safe softmax", same pages, math-backend sections), never NaN.
 *   - rank-3 inputs [H, L, D] are treated as rank-4 [1, H, L, D] and reach the
 *     same fused kernel ("PyTorch 2.14 SDPA: rank-3 inputs now take the fused
 *     kernels", daker.dacon.io, sections on the rank-3 problem and on what
 *     changed in 2.14); results are bit-identical to the rank-4 call.
 *
 * Computation: one GPU kernel launch per call, launched with programmatic
 * stream serialization (its set-up overlaps the previous kernel in the
 * stream, its first global-memory access waits for that kernel); 16-bit
 * inputs on tensor cores
 * with fp32 accumulation, the softmax in fp32, probabilities rounded to the
 * input type before the second product, output rounded to nearest even.
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define SDPA_API __attribute__((visibility("default")))
#else
#define SDPA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sdpa_status {
  SDPA_OK = 0,
  SDPA_ERR_NULL = 1,            /* a required pointer argument is NULL */
  SDPA_ERR_RANK = 2,            /* rank is not 3 or 4 */
  SDPA_ERR_SHAPE = 3,           /* D not 64 or 128, or a dimension < 1, or too large */
  SDPA_ERR_DTYPE = 4,           /* dtype is not SDPA_BF16 / SDPA_FP16 */
  SDPA_ERR_LAYOUT = 5,          /* inner stride != 1, other strides not multiples of 8
                                   elements (16 bytes), zero stride on a dimension > 1,
                                   or a pointer not 16-byte aligned */
  SDPA_ERR_ARG = 6,             /* causal and mask both given, or out overlaps q/k/v/mask,
                                   or a NaN/inf scale other than the NaN default */
  SDPA_ERR_CUDA = 7,            /* the CUDA runtime/driver reported an error (launch,
                                   tensor-map encoding, no device) */
  SDPA_ERR_DEVICE_TIMEOUT = 8,  /* a kernel barrier wait ran out of time (see
                                   sdpa_last_device_status) */
  SDPA_ERR_DEVICE = 9           /* the current device is not an sm_103 GPU */
} sdpa_status;

typedef enum sdpa_dtype {
  SDPA_BF16 = 0,
  SDPA_FP16 = 1
} sdpa_dtype;

/*
 * sdpa_forward -- launch the fused attention forward on `stream`.
 *
 * q, k, v, out : DEVICE pointers to 16-bit elements of type `dtype`; all four
 *                share one logical shape.  The caller owns them; the call
 *                neither frees nor retains them.
 * rank         : 3 for [H, L, D], 4 for [B, H, L, D].
 * shape        : `rank` extents (host array).  D must be 64 or 128; L >= 1
 *                (any value, including ragged ones not divisible by 128).
 * *_stride     : `rank` strides in ELEMENTS (host arrays), so any strided view
 *                (for example a [B, L, H, D] buffer viewed as [B, H, L, D])
 *                is consumed in place with no transpose.  The innermost (D)
 *                stride must be 1; every other stride must be a multiple of
 *                8 elements and non-zero unless its extent is 1.
 * is_causal    : nonzero for the causal triangle.
 * mask         : NULL, or a DEVICE pointer to a dense row-major [L, L] byte
 *                matrix (nonzero = removed).  Not allowed together with
 *                is_causal.
 * scale        : multiplier of q.k; NaN selects the default 1/sqrt(D) (the
 *                module's scale on both profiling pages).
 * stream       : a cudaStream_t (NULL = legacy default stream).
 *
 * Returns SDPA_OK once the kernel is enqueued (asynchronous: results are
 * ready when the stream reaches it), or an error code.  Argument errors are
 * detected on the host before any CUDA call and launch nothing.  No device
 * memory is allocated per call.  Thread-compatible: concurrent calls must use
 * different streams.
 */
SDPA_API sdpa_status sdpa_forward(const void* q, const void* k, const void* v, void* out,
                         sdpa_dtype dtype, int rank, const int64_t* shape,
                         const int64_t* q_stride, const int64_t* k_stride,
                         const int64_t* v_stride, const int64_t* o_stride,
                         int is_causal, const uint8_t* mask, float scale, void* stream);

/*
 * Plans -- validate and encode once, launch many times.
 *
 * sdpa_forward validates its arguments and encodes three TMA descriptors on
 * every call.  A plan does that work once for a fixed shape, dtype, strides,
 * mask mode and scale (the same arguments and the same errors as
 * sdpa_forward); sdpa_plan_launch then only launches the kernel, which keeps
 * the host cost of a call to a few microseconds.  (The pages measure 117-214
 * us of CPU time per forward for the fused PyTorch backends, most of it
 * per-call plan selection for cuDNN: "Profiling attention in PyTorch:
 * kernels, backends and where the time goes", news.bpdata.com, section
 * "cuDNN backend".)
 *
 * sdpa_plan_create      : *plan receives a new plan (host memory owned by the
 *                         caller until sdpa_plan_destroy), or NULL on error.
 *                         Binds the plan to the current device.
 * sdpa_plan_set_pointers: rebinds q, k, v, out (and mask, which must be
 *                         present iff it was at creation) to new DEVICE
 *                         buffers of the same shape and strides; validated
 *                         like sdpa_forward.  Not thread-safe with a
 *                         concurrent launch of the same plan.
 * sdpa_plan_launch      : enqueues the forward on `stream` (asynchronous);
 *                         SDPA_ERR_ARG if the current device is not the
 *                         plan's.  Safe to call from several threads on
 *                         different streams, and inside CUDA graph capture.
 *                         A plan with a mask first launches the mask summary
 *                         (see sdpa_mask_tiles) into device memory the plan
 *                         allocated at creation (n^2 * 2049 bytes for n =
 *                         ceil(L / 128); SDPA_ERR_CUDA from sdpa_plan_create
 *                         when that allocation fails), then the forward,
 *                         which skips the key tiles that remove every key
 *                         for both query tiles of its job and reads 16 bytes
 *                         of mask per row and tile.  Concurrent launches of
 *                         one plan write identical summary bytes as long as
 *                         the mask's contents do not change meanwhile.
 * sdpa_plan_destroy     : frees the plan (NULL is ignored).  Work already
 *                         enqueued is unaffected.
 */
typedef struct sdpa_plan sdpa_plan;

SDPA_API sdpa_status sdpa_plan_create(sdpa_plan** plan, const void* q, const void* k,
                                      const void* v, void* out, sdpa_dtype dtype, int rank,
                                      const int64_t* shape, const int64_t* q_stride,
                                      const int64_t* k_stride, const int64_t* v_stride,
                                      const int64_t* o_stride, int is_causal,
                                      const uint8_t* mask, float scale);
SDPA_API sdpa_status sdpa_plan_set_pointers(sdpa_plan* plan, const void* q, const void* k,
                                            const void* v, void* out, const uint8_t* mask);
SDPA_API sdpa_status sdpa_plan_launch(const sdpa_plan* plan, void* stream);
SDPA_API void sdpa_plan_destroy(sdpa_plan* plan);

/*
 * sdpa_forward_masked_noalloc -- a masked forward that allocates nothing.
 *
 * The pages have no counterpart: this entry point is for callers that
 * cannot allocate device memory -- code that runs inside another runtime
 * whose memory pool has already reserved the device's memory, or a serving
 * loop that must not call cudaMalloc/cudaFree (they can synchronise the
 * whole device) -- but still want the masked fast path that a masked plan
 * gets from its summary buffer.  Here the mask summary (see sdpa_mask_tiles)
 * lives in one fixed array inside the library instead: 2,098,176 bytes of
 * device memory on every GPU that loads the library, held until the process
 * exits, enough for L <= SDPA_NOALLOC_MAX_L.
 *
 * Arguments as sdpa_forward with an explicit mask (no is_causal): mask must
 * be non-NULL (else SDPA_ERR_NULL); L > SDPA_NOALLOC_MAX_L returns
 * SDPA_ERR_SHAPE, the scratch array's limit; other errors as sdpa_forward.
 * The caller passes and owns q, k, v, out and mask; the call allocates no
 * device or pinned memory.  The first call on a device looks up the array's
 * device address on that device (it must be current, as for every call) and
 * caches it; make that first call before any stream capture.  The cached
 * address belongs to the device's context: after cudaDeviceReset the next
 * call finds that the context changed and looks the address up again (so
 * that call, too, belongs before any capture).  Every call
 * on a device uses the same array and leaves its last summary in it:
 * nothing there needs to start at zero, because each call rewrites every
 * byte it then reads, but calls whose work overlaps on the GPU (different
 * streams, or different threads) race on the array and must be ordered by
 * the caller.
 */
#define SDPA_NOALLOC_MAX_L 4096
SDPA_API sdpa_status sdpa_forward_masked_noalloc(const void* q, const void* k, const void* v,
                                                 void* out, sdpa_dtype dtype, int rank,
                                                 const int64_t* shape, const int64_t* q_stride,
                                                 const int64_t* k_stride,
                                                 const int64_t* v_stride,
                                                 const int64_t* o_stride, const uint8_t* mask,
                                                 float scale, void* stream);

/*
 * sdpa_mask_tiles -- the tile summary of an explicit mask (the mask-tile
 * skip bitmap masked plans use), written into caller-owned memory.
 *
 * The [L, L] mask (DEVICE, row-major bytes, nonzero = removed: the
 * masked_fill polarity of "Profiling attention in PyTorch: kernels, backends
 * and where the time goes", news.bpdata.com, section "Naiv causal attention") is cut
 * into n x n tiles of 128 x 128, n = ceil(L / 128).  For tile (qt, kt):
 *   tile_bits  : DEVICE, 16-byte aligned, n*n*128*16 bytes.  Row r of the
 *                tile is four 32-bit words at byte ((qt*n + kt)*128 + r)*16;
 *                bit c of word w is 1 when key kt*128 + 32w + c is removed
 *                for query qt*128 + r.  Keys and rows past L read as removed.
 *   tile_class : DEVICE, n*n bytes at qt*n + kt: 0 = no entry inside [L, L]
 *                is removed, 1 = some are, 2 = all are.
 * Asynchronous on `stream` (PDL launch: it waits for the previous kernel in
 * the stream before reading the mask).  Errors: SDPA_ERR_NULL,
 * SDPA_ERR_SHAPE (L < 1 or n > 65535), SDPA_ERR_LAYOUT (tile_bits not 16-byte
 * aligned), SDPA_ERR_CUDA.
 */
SDPA_API sdpa_status sdpa_mask_tiles(const uint8_t* mask, int64_t L, void* tile_bits,
                                     uint8_t* tile_class, void* stream);

/*
 * sdpa_forward_lse -- sdpa_forward that also writes, per query row, the
 * log-sum-exp of the scaled, masked scores, log(sum_j exp(scale * q_i . k_j))
 * over the admissible keys (-inf for a row with none): the log of the
 * softmax denominator, the second output of the fused forward on the
 * FlashInfer pull-request page (`out, lse = fwd(...)`), which a backward
 * pass or a merge of partial results needs.
 *
 * lse        : DEVICE float32 buffer of shape [B, H, L] (rank 4) or [H, L]
 *              (rank 3), 4-byte aligned, not overlapping any other operand.
 * lse_stride : rank - 1 strides in ELEMENTS (host array); positive unless
 *              the extent is 1.
 * Everything else as sdpa_forward; SDPA_ERR_NULL if lse or lse_stride is
 * NULL.  The LSE is computed in fp32 from the same running maximum and sum
 * the softmax uses.
 */
SDPA_API sdpa_status sdpa_forward_lse(const void* q, const void* k, const void* v, void* out,
                                      float* lse, sdpa_dtype dtype, int rank,
                                      const int64_t* shape, const int64_t* q_stride,
                                      const int64_t* k_stride, const int64_t* v_stride,
                                      const int64_t* o_stride, const int64_t* lse_stride,
                                      int is_causal, const uint8_t* mask, float scale,
                                      void* stream);

/*
 * sdpa_forward_varlen -- packed variable-length sequences.  Several
 * documents are stored one after another along the token axis and
 * described by cumulative offsets, the cu_seqlens arrays that the varlen
 * kernels on the FlashInfer pull-request page take ("FlashInfer, Cake DSA
 * kernel optimization", blog.secrett2633.cloud, section 3 on varlen index
 * preparation).  Each document attends only to itself: sequence i is rows
 * [cu_seqlens[i], cu_seqlens[i+1]) of q, k and v, and its output rows are
 * exactly what sdpa_forward returns for that slice alone (the same kernel
 * and per-tile arithmetic, so bit-identical).  Queries and keys share one
 * offsets array (self-attention; causal means key j <= query i within the
 * document).
 *
 * q, k, v, out : DEVICE [total, H, D] 16-bit tensors of type `dtype`.
 * *_stride     : 3 strides in ELEMENTS in (token, head, dim) order; the dim
 *                stride must be 1, the others multiples of 8 elements.
 * lse          : NULL, or DEVICE fp32 [H, total] (lse_stride: 2 strides, head
 *                then token), the per-row log-sum-exp as in sdpa_forward_lse.
 * cu_seqlens   : DEVICE int32 [n_seqs + 1], 4-byte aligned, nondecreasing,
 *                cu_seqlens[0] = 0 and cu_seqlens[n_seqs] = total.  The
 *                kernel uses the running maximum of the offsets clamped to
 *                [0, total] (the identity for valid offsets), so bad offsets
 *                cannot make it read or write outside the buffers or make
 *                two sequences overlap; rows covered by no sequence are
 *                left unwritten.
 * max_seqlen   : an upper bound on the sequence lengths; it only sizes the
 *                grid (a smaller value gives fewer CTAs, never missed work).
 * Explicit masks are not supported here (is_causal or no mask).  Errors as
 * sdpa_forward, plus SDPA_ERR_SHAPE for n_seqs < 1 or max_seqlen < 1 and
 * SDPA_ERR_ARG when out or lse overlaps cu_seqlens.
 */
SDPA_API sdpa_status sdpa_forward_varlen(const void* q, const void* k, const void* v, void* out,
                                         float* lse, sdpa_dtype dtype, int64_t total,
                                         int64_t n_heads, int64_t head_dim,
                                         const int64_t* q_stride, const int64_t* k_stride,
                                         const int64_t* v_stride, const int64_t* o_stride,
                                         const int64_t* lse_stride, const int32_t* cu_seqlens,
                                         int64_t n_seqs, int64_t max_seqlen, int is_causal,
                                         float scale, void* stream);

/*
 * sdpa_sparse_forward -- sparse top-k attention: query row i, every head,
 * attends only to the key rows idx[i, 0 .. len_i) of one key/value head
 * shared by all query heads, len_i = topk_length[i] clamped to [0, topk]
 * (topk when topk_length is NULL).  The DeepSeek sparse attention forward
 * of "FlashInfer, Cake DSA kernel optimization" (blog.secrett2633.cloud):
 * `out, lse = fwd(q, kv, idx, topk_length=...)` over hole-free index rows
 * (sections 1 and 3 of that page); pass the same pointer as k and v for one
 * shared kv tensor.
 *
 * q, out     : DEVICE [total_q, H, D] 16-bit of type `dtype`; q_stride and
 *              o_stride give 2 strides in ELEMENTS (token, head), multiples
 *              of 8; the D stride is 1.
 * k, v       : DEVICE [total_k, D]; k_stride, v_stride = row strides in
 *              ELEMENTS (multiples of 8).  16-byte aligned pointers.
 * lse        : NULL or DEVICE fp32 [total_q, H] (lse_stride: token, head).
 * idx        : DEVICE int32 [total_q, topk] (row stride idx_stride >= topk)
 *              of global key rows; entries outside [0, total_k) inside the
 *              first len_i are treated as removed keys (no fault).
 * topk_length: NULL or DEVICE int32 [total_q].
 * A row with no admissible key gives zeros and lse = -inf.  Computation as
 * sdpa_forward (16-bit tensor-core products, fp32 softmax).  Errors: NULL,
 * DTYPE, SHAPE (D not 64/128, an extent < 1), LAYOUT (alignment, strides),
 * ARG (out or lse overlapping an input, infinite scale), CUDA, DEVICE.
 * Asynchronous on `stream`; one kernel launch.
 */
SDPA_API sdpa_status sdpa_sparse_forward(const void* q, const void* k, const void* v, void* out,
                                         float* lse, sdpa_dtype dtype, int64_t total_q,
                                         int64_t total_k, int64_t n_heads, int64_t head_dim,
                                         const int64_t* q_stride, int64_t k_stride,
                                         int64_t v_stride, const int64_t* o_stride,
                                         const int64_t* lse_stride, const int32_t* idx,
                                         int64_t idx_stride, int64_t topk,
                                         const int32_t* topk_length, float scale, void* stream);

/*
 * sdpa_sparse_compact -- the index preparation of the same page (sections 1
 * and 3) in one launch: per-document key positions become global key rows
 * with the holes removed.  Query row r of document b (rows
 * [cu_seqlens_q[b], cu_seqlens_q[b+1])) keeps, in order, every entry l of
 * idx_local[r, :] with 0 <= l < (cu_seqlens_k[b+1] - cu_seqlens_k[b]) and,
 * if is_causal, l <= r - cu_seqlens_q[b]; it is written as
 * cu_seqlens_k[b] + l to idx_global[r, 0 .. n), the rest of the row is -1,
 * and topk_length[r] = n.  Rows outside every document get n = 0.
 * All arrays DEVICE int32, 4-byte aligned; offsets nondecreasing.  Errors:
 * NULL, SHAPE, LAYOUT, ARG (outputs overlapping inputs or each other), CUDA.
 */
SDPA_API sdpa_status sdpa_sparse_compact(const int32_t* idx_local, int64_t idx_local_stride,
                                         int32_t* idx_global, int64_t idx_global_stride,
                                         int32_t* topk_length, int64_t total_q, int64_t topk,
                                         const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                         int64_t n_docs, int is_causal, void* stream);

/* Adds (lse != NULL) or removes (lse == NULL) the log-sum-exp output of a
 * plan; same layout rules as sdpa_forward_lse. */
SDPA_API sdpa_status sdpa_plan_set_lse(sdpa_plan* plan, float* lse, const int64_t* lse_stride);

/* Human-readable name of a status code (static storage, never NULL). */
SDPA_API const char* sdpa_status_string(sdpa_status status);

/*
 * sdpa_last_device_status -- synchronise `stream`, then report whether any
 * kernel since the previous query gave up on a barrier wait (every wait in
 * the kernel is bounded in time; on expiry the kernel stops, frees its
 * resources and sets a device status word instead of hanging).  Returns
 * SDPA_OK, SDPA_ERR_DEVICE_TIMEOUT (the word is then cleared), or
 * SDPA_ERR_CUDA.
 *
 * sdpa_last_device_status_detail -- the same query; when `detail` is not
 * NULL it also receives the raw status bits (bit 0: a wait ran out of time;
 * the higher bits name the kind of wait), for diagnostics.
 */
SDPA_API sdpa_status sdpa_last_device_status(void* stream);
SDPA_API sdpa_status sdpa_last_device_status_detail(void* stream, uint32_t* detail);

/* ABI version: major * 10000 + minor * 100 + patch. */
SDPA_API int sdpa_version(void);

/*
 * Test hooks (not for production use).
 * sdpa_debug_set_wait_limit_ns: bound on a single barrier wait inside the
 *   kernel (default 1e9 ns); 0 restores the default.
 * sdpa_debug_withhold_q_load: when nonzero, subsequent launches (dense,
 *   packed-document and sparse forwards) never load the query tile, so every
 *   consumer wait runs out before any product is issued: the kernel must return
 *   with SDPA_ERR_DEVICE_TIMEOUT reported by sdpa_last_device_status and the
 *   context must stay usable.
 */
SDPA_API void sdpa_debug_set_wait_limit_ns(uint64_t ns);
SDPA_API void sdpa_debug_withhold_q_load(int enable);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_GB300_H */
