// sdpa_internal.h -- shared between the C-ABI front end and the kernel
// translation unit.  Not part of the public interface.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sdpa_impl {

// Kernel arguments; passed by value as a __grid_constant__ parameter so the
// TMA descriptors live in parameter space (no device allocation per call).
struct FwdParams {
  CUtensorMap tm_q;  // 4-D maps over (D, and L/H/B in stride order); box 64 x 128 rows
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  void* out;          // [B, H, L, D] with element strides below (inner stride 1)
  int64_t o_sb, o_sh, o_sl;
  const uint8_t* mask;  // [L, L] row-major bytes, nonzero = removed; null unless mask mode
  float* lse;           // optional [B, H, L] fp32 log-sum-exp per row (element strides below)
  int64_t lse_sb, lse_sh, lse_sl;
  int B, H, L;          // packed sequences: B = 1 and L = total rows
  int n_tiles;          // ceil(L / 128)
  // Packed sequences (null: dense [B, H, L, D]): sequence i is rows
  // [cu_seqlens[i], cu_seqlens[i+1]) of the L axis, attended on its own.
  const int* cu_seqlens;
  int n_seqs;
  long long max_units;  // upper bound on the number of work units (grid size)
  int snake;            // dense only: 1 = jobs by falling cost in snake order (small problems)
  float scale_log2;     // scale * log2(e)
  int pos_q[3], pos_k[3], pos_v[3];  // tensor-map coordinate slot (1..3) of L, H, B
  int mask_vec16;       // 1: mask rows may be read as 16-byte vectors (L % 16 == 0, aligned)
  // Optional tile summary of the explicit mask (both null: read the mask
  // bytes).  Tile (qt, kt) of the n_tiles x n_tiles grid of 128 x 128 tiles:
  // class byte tile_class[qt * n_tiles + kt] (kTileKept / kTileMixed /
  // kTileRemoved) and 128 rows of 128 bits at tile_bits[(qt * n_tiles + kt) *
  // 128 + row] (bit c of word w = key 32w + c removed; keys and rows past L
  // read as removed).
  const uint4* tile_bits;
  const uint8_t* tile_class;
  int debug_withhold_q; // test hook: 1 = never load Q, so every consumer wait runs out
  uint64_t wait_limit_ns;  // bound on any single barrier wait
};

// Tile classes of a mask summary, counting only entries inside [L, L].
enum TileClass : uint8_t { kTileKept = 0, kTileMixed = 1, kTileRemoved = 2 };

// Mask summary: one CTA per 128 x 128 tile of an [L, L] byte mask.
struct MaskTilesParams {
  const uint8_t* mask;  // [L, L] row-major, nonzero = removed
  int L, n_tiles;
  int vec16;            // rows may be read as 16-byte vectors
  uint16_t* bits;       // [n_tiles^2][128 rows][8] 16-bit words (the tile_bits layout)
  uint8_t* tile_class;  // [n_tiles^2]
};

// Sparse top-k attention: query row i (all heads of head group g) attends to
// the key rows idx[i, 0 .. len_i) of one shared key/value head.
struct SparseParams {
  CUtensorMap tm_q;  // 3-D (D, H, total_q), box 64 x min(H, 128) x 1 (one head group)
  void* out;                // [total_q, H, D]
  int64_t o_st, o_sh;
  float* lse;               // optional [total_q, H]
  int64_t lse_st, lse_sh;
  const int* idx;           // [total_q, topk] global key rows
  int64_t idx_st;
  const int* topk_length;   // [total_q] valid leading entries, or null (all topk)
  int total_q, total_k, H, topk, n_groups;
  int q_rows;               // heads of a group: min(H, 128)
  // 1 (H <= 64): M = 64 products, which put head h in TMEM lane
  // 32 (h / 16) + h % 16, and two softmax threads share each row; 0: M = 128
  // products, one thread a row
  int q_half;
  int kv_shared;            // 1: k and v are one tensor (gather once, use twice)
  const void* k;            // [total_k, D] rows for the gathers
  const void* v;
  int64_t k_row_bytes, v_row_bytes;
  float scale_log2;
  int debug_withhold_q;     // test hook: 1 = never load Q, so every consumer wait runs out
  uint64_t wait_limit_ns;
};

// Index preparation: per-document key positions -> global rows, holes removed.
struct CompactParams {
  const int* idx_local;
  int64_t in_st;
  int* idx_global;
  int64_t out_st;
  int* length;
  const int* cu_q;
  const int* cu_k;
  int total_q, topk, n_docs, is_causal;
};

cudaError_t launch_sparse(const SparseParams& p, int head_dim, bool bf16, int max_ctas,
                          cudaStream_t stream);
cudaError_t launch_compact(const CompactParams& p, cudaStream_t stream);
// Reads and clears the sparse kernel's status word (its own translation unit).
cudaError_t read_and_clear_sparse_status(unsigned int* status);

enum MaskMode : int { kMaskNone = 0, kMaskCausal = 1, kMaskExplicit = 2 };

// Launches the persistent forward kernel for (head_dim, mask mode, dtype) on
// `stream` with at most max_ctas CTAs (one per SM: pass the device's SM
// count).  Returns the CUDA error of the launch.
cudaError_t launch_forward(const FwdParams& p, int head_dim, int mask_mode, bool bf16,
                           int max_ctas, cudaStream_t stream);
// The head-size-64 kernel (its own translation unit; launch_forward calls it).
cudaError_t launch_forward64(const FwdParams& p, int mask_mode, bool bf16, int max_ctas,
                             cudaStream_t stream);
// Reads and clears the head-size-64 kernel's status word.
cudaError_t read_and_clear_fwd64_status(unsigned int* status);

// Writes the tile summary of p.mask (PDL launch: waits for the previous
// kernel in the stream before reading the mask).
cudaError_t launch_mask_tiles(const MaskTilesParams& p, cudaStream_t stream);

// sdpa_forward_masked_noalloc: the mask summary lives in a fixed array in
// the library, enough for n_tiles <= kNoAllocMaxTiles.  Returns the device
// addresses of its bits and class parts for `device`, which must be current
// (looked up once per device with cudaGetSymbolAddress, then cached).
constexpr int kNoAllocMaxTiles = 32;
constexpr int kNoAllocMaxDevices = 64;
cudaError_t noalloc_mask_tiles(int device, const uint4** tile_bits, const uint8_t** tile_class);

// Reads and clears the device status word (nonzero = a barrier wait timed out).
cudaError_t read_and_clear_device_status(cudaStream_t stream, unsigned int* status);

}  // namespace sdpa_impl
