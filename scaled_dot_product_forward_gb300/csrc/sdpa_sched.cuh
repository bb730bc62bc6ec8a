// sdpa_sched.cuh -- work decomposition and small device helpers shared by the
// fused forward kernels (D = 128: two query tiles per job; D = 64: four).
//
// A job is a group of TILES adjacent 128-row query tiles of one (sequence,
// head).  A unit is group G-1-k followed by group k of the same head (G
// groups per head): under the causal mask the two together visit the same
// number of key tiles whatever k is, so units of one sequence length cost the
// same and a static round-robin assignment of units to persistent CTAs is
// balanced.  Units are numbered head-major, so the CTAs busy at one time
// share a few heads' K/V in L2.  Small problems deal jobs by falling cost in
// snake order instead; packed documents are found through a warp-wide cursor
// over cu_seqlens.  Every role of a CTA walks the same sequence of jobs.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sdpa_internal.h"

namespace sdpa_sched {

using namespace sdpa_dev;

constexpr int kBlockM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBlockN = 128;  // keys per K/V tile of the load ring

// Bounded wait on one barrier phase.  Returns false when the wait gave up:
// either another role already raised the CTA's abort flag (honour_abort), or
// this wait exceeded the time limit, in which case it raises the flag and
// records `site` (bit 0 plus the site bit) in the kernel's status word.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint32_t* abort_flag,
                                           unsigned int* status, uint64_t limit_ns,
                                           unsigned int site, bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 63u) == 0) {
      if (honour_abort && *reinterpret_cast<volatile uint32_t*>(abort_flag) != 0) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *reinterpret_cast<volatile uint32_t*>(abort_flag) = 1u;
        atomicOr(status, 1u | site);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_tile(void* dst, const CUtensorMap* map, uint64_t* bar,
                                         int d0, int row, int head, int batch,
                                         const int (&pos)[3]) {
  // pos[] holds the map slot (1..3) of L, H and B; place the coordinates.
  const int c1 = (pos[0] == 1) ? row : (pos[1] == 1) ? head : batch;
  const int c2 = (pos[0] == 2) ? row : (pos[1] == 2) ? head : batch;
  const int c3 = (pos[0] == 3) ? row : (pos[1] == 3) ? head : batch;
  tma_load_4d(dst, map, bar, d0, c1, c2, c3);
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

// Bit i (i = 0..3) set when byte i of `word` is nonzero: the bytes' sign
// bits after a per-byte "!= 0" compare, gathered by one multiply (byte i's
// bit 8i+7 times 2^(7(3-i)) lands on bit 28+i; every other product term
// falls on a distinct bit outside 28..31, so nothing carries into them).
__device__ __forceinline__ uint32_t nonzero_byte_bits(uint32_t word) {
  const uint32_t m = __vcmpne4(word, 0u) & 0x80808080u;
  return (m * 0x00204081u) >> 28;
}

// The 128 mask bits (bit set = key removed) of this thread's row for the
// 128-key tile starting at col0, read from the byte mask: word k = keys
// 32k..32k+31.  All 32 lanes of the warp take part, with consecutive rows
// (row_g - lane is the warp's first row).  When the warp's 32 rows and the
// 128 keys all lie inside [len, len] and rows may be read as 16-byte vectors
// (mask_vec_ok), lane (g, c) = (lane / 8, lane % 8) reads 16 bytes of row
// 8g + i at keys 16c.. for i = 0..7 (mask_bytes_load), so each load
// instruction covers four whole 128-byte row segments, and mask_bits_convert
// turns them into 16 bits and then, with an 8 x 8 transpose of 16-bit values
// inside each group of eight lanes (three butterfly stages), into the 128
// bits of each lane's own row.  The two halves may be split so that the
// loads of one tile are in flight while the previous tile is worked on.
// Otherwise (mask_bits_slow) each row is read byte by byte, with rows and
// keys past len counted as removed.
__device__ __forceinline__ bool mask_vec_ok(const sdpa_impl::FwdParams& p, int len, int row_g,
                                            int lane, int col0) {
  return p.mask_vec16 && col0 + kBlockN <= len && row_g - lane + 31 < len;
}

__device__ __forceinline__ void mask_bytes_load(const sdpa_impl::FwdParams& p, int row_g,
                                                int lane, int col0, uint4 (&x)[8]) {
  const int g8 = lane >> 3, c8 = lane & 7;
  const uint8_t* mbase =
      p.mask + static_cast<int64_t>(row_g - lane + 8 * g8) * p.L + col0 + 16 * c8;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    x[i] = __ldg(reinterpret_cast<const uint4*>(mbase + static_cast<int64_t>(i) * p.L));
}

__device__ __forceinline__ void mask_bits_convert(const uint4 (&x)[8], int lane,
                                                  uint32_t (&mbits)[4]) {
  const int c8 = lane & 7;
  uint32_t wv[4];
#pragma unroll
  for (int k2 = 0; k2 < 4; ++k2) {
    const uint4 a = x[2 * k2], b = x[2 * k2 + 1];
    const uint32_t ha = nonzero_byte_bits(a.x) | (nonzero_byte_bits(a.y) << 4) |
                        (nonzero_byte_bits(a.z) << 8) | (nonzero_byte_bits(a.w) << 12);
    const uint32_t hb = nonzero_byte_bits(b.x) | (nonzero_byte_bits(b.y) << 4) |
                        (nonzero_byte_bits(b.z) << 8) | (nonzero_byte_bits(b.w) << 12);
    wv[k2] = ha | (hb << 16);  // rows 8g+2k2 (low) and 8g+2k2+1 (high), keys 16c..
  }
  {  // swap the off-diagonal 4 x 4 blocks (lane bit 2 <-> element bit 2)
    const bool hi = (c8 & 4) != 0;
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, hi ? wv[0] : wv[2], 4);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, hi ? wv[1] : wv[3], 4);
    if (hi) { wv[0] = r0; wv[1] = r1; } else { wv[2] = r0; wv[3] = r1; }
  }
  {  // 2 x 2 blocks inside each (lane bit 1 <-> element bit 1)
    const bool hi = (c8 & 2) != 0;
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, hi ? wv[0] : wv[1], 2);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, hi ? wv[2] : wv[3], 2);
    if (hi) { wv[0] = r0; wv[2] = r1; } else { wv[1] = r0; wv[3] = r1; }
  }
  {  // single elements (lane bit 0 <-> the 16-bit half of a word)
    const bool hi = (c8 & 1) != 0;
    const uint32_t sel = hi ? 0x5410u : 0x7632u;
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, __byte_perm(wv[0], wv[1], sel), 1);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, __byte_perm(wv[2], wv[3], sel), 1);
    if (hi) {
      wv[0] = __byte_perm(r0, wv[0], 0x7610u);
      wv[1] = __byte_perm(r0, wv[1], 0x7632u);
      wv[2] = __byte_perm(r1, wv[2], 0x7610u);
      wv[3] = __byte_perm(r1, wv[3], 0x7632u);
    } else {
      wv[0] = __byte_perm(wv[0], r0, 0x5410u);
      wv[1] = __byte_perm(wv[1], r0, 0x7610u);
      wv[2] = __byte_perm(wv[2], r1, 0x5410u);
      wv[3] = __byte_perm(wv[3], r1, 0x7610u);
    }
  }
#pragma unroll
  for (int k2 = 0; k2 < 4; ++k2) mbits[k2] = wv[k2];
}

__device__ __forceinline__ void mask_bits_slow(const sdpa_impl::FwdParams& p, int len, int row_g,
                                               int col0, uint32_t (&mbits)[4]) {
  const bool row_ok = row_g < len;
  const uint8_t* mrow = p.mask + static_cast<int64_t>(row_ok ? row_g : 0) * p.L + col0;
#pragma unroll
  for (int w32 = 0; w32 < kBlockN / 32; ++w32) {
    uint32_t bits = 0;
    for (int e = 0; e < 32; ++e) {
      const int c = 32 * w32 + e;
      const bool removed = !row_ok || col0 + c >= len || __ldg(mrow + c) != 0;
      bits |= (removed ? 1u : 0u) << e;
    }
    mbits[w32] = bits;
  }
}

__device__ __forceinline__ void mask_bits_from_bytes(const sdpa_impl::FwdParams& p, int len,
                                                     int row_g, int lane, int col0,
                                                     uint32_t (&mbits)[4]) {
  if (mask_vec_ok(p, len, row_g, lane, col0)) {
    uint4 x[8];
    mask_bytes_load(p, row_g, lane, col0, x);
    mask_bits_convert(x, lane, mbits);
  } else {
    mask_bits_slow(p, len, row_g, col0, mbits);
  }
}

// One job.  Its tiles are tile0, tile0 + 1, ... (the first n_present of
// the TILES are inside the sequence), and tile t visits kv0 + kv_step * t key
// tiles (causal: its index + 1; otherwise all of them, or with a mask
// summary the visited count) -- an arithmetic progression in every mode, so
// the record stays small and is read by tile index without indexing an
// array by a run-time value.
template <int TILES>
struct Work {
  int batch, head;     // tensor-map coordinates (batch is 0 for packed sequences)
  int row0;            // first row of the sequence along L (packed: its offset)
  int len;             // rows (= keys) of the sequence
  int tile0;           // query tile index of the job's first tile
  int n_present;       // tiles of the group inside the sequence (1..TILES)
  int kv0, kv_step;    // key tiles visited by tile t: kv0 + kv_step * t
  int n_kv_max;        // the most any tile of the job visits
  __device__ __forceinline__ int tile(int t) const { return tile0 + t; }
  __device__ __forceinline__ int n_kv(int t) const {
    return t < n_present ? kv0 + kv_step * t : 0;
  }
};

template <int TILES>
__host__ __device__ inline int groups_per_head(int n_tiles) {
  return (n_tiles + TILES - 1) / TILES;
}
template <int TILES>
__host__ __device__ inline int units_per_head(int n_tiles) {
  return (groups_per_head<TILES>(n_tiles) + 1) >> 1;
}
__host__ __device__ inline int tiles_of(int len) { return (len + kBlockM - 1) / kBlockM; }

// Job `sub` (0 or 1) of unit k of one (sequence, head) with n_tiles tiles;
// false when the unit has no such job (the middle group of an odd group count
// stands alone).  Fills the tile fields of w.
template <int MODE, int TILES>
__device__ __forceinline__ bool job_tiles(int n_tiles, int k, int sub, Work<TILES>& w) {
  const int G = groups_per_head<TILES>(n_tiles);
  const int gr = (sub == 0) ? (G - 1 - k) : k;
  if (sub == 1 && gr == G - 1 - k) return false;
  w.tile0 = TILES * gr;
  w.n_present = min(TILES, n_tiles - w.tile0);
  if (MODE == sdpa_impl::kMaskCausal) {
    w.kv0 = w.tile0 + 1;
    w.kv_step = 1;
  } else {
    w.kv0 = n_tiles;
    w.kv_step = 0;
  }
  w.n_kv_max = w.n_kv(w.n_present - 1);
  return true;
}

// Packed sequences: a warp-wide cursor over cu_seqlens, 32 sequences per
// step.  Lane i holds sequence chunk + i (its start and length and the
// inclusive count of units up to it within the chunk); `before` counts the
// units of earlier chunks.  Units are numbered sequence by sequence, each
// sequence's heads in order.  With at most 32 sequences (one chunk) the
// order is by cost instead, since any unit can then be found in the chunk:
// first every sequence's two-job units, longest sequence first, then the
// one-job units (the middle group of an odd group count), longest first, so
// the snake deals the costly units before the cheap ones fill the gaps.  The
// offsets are used as the running maximum of their values clamped to [0,
// total], so sequences never overlap and never leave the buffers, whatever
// the array holds; for valid offsets (0 first, nondecreasing, total last)
// that is the identity.  All 32 lanes run it.
struct SeqCursor {
  int chunk, before, chunk_units;
  int carry;      // running-maximum offset where this chunk starts
  int carry_out;  // ... and where it ends
  int start, len, incl;
  int incl_half, full_units;  // one chunk only: inclusive one-job units, all two-job units
};

template <int TILES>
__device__ __forceinline__ void cursor_load(const sdpa_impl::FwdParams& p, SeqCursor& c,
                                            int lane) {
  const int seq = c.chunk + lane;
  int e = c.carry;
  if (seq < p.n_seqs) e = max(e, min(max(__ldg(p.cu_seqlens + seq + 1), 0), p.L));
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, e, off);
    if (lane >= off) e = max(e, v);
  }
  int st = __shfl_up_sync(0xffffffffu, e, 1);
  if (lane == 0) st = c.carry;
  c.start = st;
  c.len = e - st;
  c.carry_out = __shfl_sync(0xffffffffu, e, 31);
  if (p.n_seqs <= 32) {
    // Bitonic sort of the lanes by (length, then lower index) descending;
    // the keys are distinct, so every warp of every CTA gets one order.
    uint64_t key = (static_cast<uint64_t>(c.len) << 6) | static_cast<uint64_t>(31 - lane);
    int s0 = c.start;
#pragma unroll
    for (int kb = 2; kb <= 32; kb <<= 1) {
#pragma unroll
      for (int jb = kb >> 1; jb > 0; jb >>= 1) {
        const uint64_t ok = __shfl_xor_sync(0xffffffffu, key, jb);
        const int os = __shfl_xor_sync(0xffffffffu, s0, jb);
        // the lower lane of a pair keeps the larger key in a descending run
        const bool take = (((lane & jb) == 0) == ((lane & kb) == 0)) ? (ok > key) : (ok < key);
        if (take) {
          key = ok;
          s0 = os;
        }
      }
    }
    c.start = s0;
    c.len = static_cast<int>(key >> 6);
    // two-job and one-job units of this sequence (per head: groups / 2 and groups % 2)
    const int groups = groups_per_head<TILES>(tiles_of(c.len));
    int full = p.H * (groups >> 1), half = p.H * (groups & 1);
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int vf = __shfl_up_sync(0xffffffffu, full, off);
      const int vh = __shfl_up_sync(0xffffffffu, half, off);
      if (lane >= off) {
        full += vf;
        half += vh;
      }
    }
    c.incl = full;
    c.incl_half = half;
    c.full_units = __shfl_sync(0xffffffffu, full, 31);
    c.chunk_units = c.full_units + __shfl_sync(0xffffffffu, half, 31);
    return;
  }
  int incl = p.H * units_per_head<TILES>(tiles_of(c.len));
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  c.incl = incl;
  c.chunk_units = __shfl_sync(0xffffffffu, incl, 31);
}

// Locates unit u (u only grows between calls).  False when u is past the
// last unit.
template <int TILES>
__device__ __forceinline__ bool cursor_find(const sdpa_impl::FwdParams& p, SeqCursor& c, int lane,
                                            int u, int& k, int& n_tiles, Work<TILES>& w) {
  while (u >= c.before + c.chunk_units) {
    if (c.chunk + 32 >= p.n_seqs) return false;
    c.before += c.chunk_units;
    c.chunk += 32;
    c.carry = c.carry_out;
    cursor_load<TILES>(p, c, lane);
  }
  if (p.n_seqs <= 32) {
    // One chunk, ordered by cost: two-job units, then one-job units.
    const bool half = u >= c.full_units;
    const int rel = half ? u - c.full_units : u;
    const unsigned hit = __ballot_sync(0xffffffffu, rel < (half ? c.incl_half : c.incl));
    const int src = __ffs(static_cast<int>(hit)) - 1;
    const int incl = __shfl_sync(0xffffffffu, half ? c.incl_half : c.incl, src);
    const int len = __shfl_sync(0xffffffffu, c.len, src);
    const int start = __shfl_sync(0xffffffffu, c.start, src);
    n_tiles = tiles_of(len);
    const int groups = groups_per_head<TILES>(n_tiles);
    w.batch = 0;
    w.row0 = start;
    w.len = len;
    if (half) {
      w.head = rel - (incl - p.H);  // one unit per head: the middle group
      k = groups >> 1;
    } else {
      const int per_head = groups >> 1;
      const int r = rel - (incl - p.H * per_head);
      w.head = r / per_head;
      k = r - w.head * per_head;
    }
    return true;
  }
  const int rel = u - c.before;
  const unsigned hit = __ballot_sync(0xffffffffu, rel < c.incl);
  const int src = __ffs(static_cast<int>(hit)) - 1;
  const int incl = __shfl_sync(0xffffffffu, c.incl, src);
  const int len = __shfl_sync(0xffffffffu, c.len, src);
  const int start = __shfl_sync(0xffffffffu, c.start, src);
  n_tiles = tiles_of(len);
  const int uph = units_per_head<TILES>(n_tiles);
  const int r = rel - (incl - p.H * uph);  // unit index within this sequence
  w.batch = 0;
  w.head = r / uph;
  k = r - w.head * uph;
  w.row0 = start;
  w.len = len;
  return true;
}

// Dense problems: the next job of this CTA (false at the end).
//  * units (default): unit u = blockIdx.x, +gridDim.x, ...; its two jobs in
//    turn (sub 0: group G-1-k, sub 1: group k);
//  * snake (small problems whose heads' K and V all fit in L2): jobs in order
//    of falling cost -- group G-1 of every head, then group G-2, ... -- dealt
//    to the CTAs 0..C-1, then C-1..0, and so on, which balances unequal
//    causal jobs far better than whole units when there are few jobs per CTA.
struct DenseIter {
  int u, sub;  // units
  int r;       // snake round
};

template <int MODE, int TILES>
__device__ __forceinline__ bool dense_next(const sdpa_impl::FwdParams& p, DenseIter& it,
                                           Work<TILES>& w) {
  const int C = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  const int BH = p.B * p.H;
  w.row0 = 0;
  w.len = p.L;
  if (p.snake) {
    const int G = groups_per_head<TILES>(p.n_tiles);
    const int i = it.r * C + ((it.r & 1) ? C - 1 - c : c);
    if (i >= BH * G) return false;
    ++it.r;
    const int cls = i / BH;
    const int bh = i - cls * BH;
    w.batch = bh / p.H;
    w.head = bh - w.batch * p.H;
    return job_tiles<MODE, TILES>(p.n_tiles, cls, 0, w);  // job 0 of unit k is group G-1-k
  }
  const int uph = units_per_head<TILES>(p.n_tiles);
  while (it.u < BH * uph) {
    const int bh = it.u / uph;
    const int k = it.u - bh * uph;
    const int sub = it.sub;
    if (sub == 0) {
      it.sub = 1;
    } else {
      it.sub = 0;
      it.u += C;
    }
    w.batch = bh / p.H;
    w.head = bh - w.batch * p.H;
    if (job_tiles<MODE, TILES>(p.n_tiles, k, sub, w)) return true;
  }
  return false;
}

// Explicit mask with a tile summary: a job visits every key tile except
// those whose every entry is removed for all of its query tiles.  Bit i of
// the result: key tile 32 * chunk + i is visited (one ballot per 32 tiles;
// every lane of the warp takes part).
template <int TILES>
__device__ __forceinline__ uint32_t visit_chunk(const sdpa_impl::FwdParams& p,
                                                const Work<TILES>& w, int chunk) {
  const int kt = chunk * 32 + static_cast<int>(threadIdx.x & 31);
  bool visit = false;
  if (kt < p.n_tiles) {
#pragma unroll
    for (int t = 0; t < TILES; ++t)
      visit = visit || (t < w.n_present &&
                        __ldg(p.tile_class + static_cast<int64_t>(w.tile(t)) * p.n_tiles + kt) !=
                            sdpa_impl::kTileRemoved);
  }
  return __ballot_sync(0xffffffffu, visit);
}

// n_kv of each present tile (and n_kv_max) becomes the number of visited key
// tiles.  A job that visits none has n_kv = 0 for every tile: the MMA and
// load roles skip it and the softmax writes its rows as zeros.
template <int TILES>
__device__ __forceinline__ void count_visits(const sdpa_impl::FwdParams& p, Work<TILES>& w) {
  int n = 0;
  for (int c = 0; c * 32 < p.n_tiles; ++c) n += __popc(visit_chunk<TILES>(p, w, c));
  w.kv0 = n;
  w.kv_step = 0;
  w.n_kv_max = n;
}

// The visited key tiles of one job in increasing order, one per call.
struct KeyTileCursor {
  int chunk;
  uint32_t bits;  // visited tiles of `chunk` not yet returned
};

// Key tile of the j-th step of a job: j itself, or with a tile summary the
// next visited tile (the cursor is called exactly n_kv_max times per job).
template <int MODE, int TILES>
__device__ __forceinline__ int next_key_tile(const sdpa_impl::FwdParams& p, const Work<TILES>& w,
                                             KeyTileCursor& c, int j) {
  if constexpr (MODE != sdpa_impl::kMaskExplicit) {
    return j;
  } else {
    if (p.tile_class == nullptr) return j;
    const int last = (p.n_tiles - 1) >> 5;
    while (c.bits == 0u && c.chunk < last) c.bits = visit_chunk<TILES>(p, w, ++c.chunk);
    if (c.bits == 0u) return p.n_tiles - 1;  // not reached: n_kv_max tiles exist
    const int kt = c.chunk * 32 + __ffs(static_cast<int>(c.bits)) - 1;
    c.bits &= c.bits - 1u;
    return kt;
  }
}

// Calls f(work) for every job of this CTA, in order; stops when f returns
// false.  VARLEN: packed sequences described by p.cu_seqlens.
template <int MODE, bool VARLEN, int TILES, typename F>
__device__ __forceinline__ void for_each_job(const sdpa_impl::FwdParams& p, F&& f) {
  if constexpr (!VARLEN) {
    DenseIter it{static_cast<int>(blockIdx.x), 0, 0};
    Work<TILES> w;
    while (dense_next<MODE, TILES>(p, it, w)) {
      if constexpr (MODE == sdpa_impl::kMaskExplicit)
        if (p.tile_class != nullptr) count_visits<TILES>(p, w);
      if (!f(w)) return;
    }
  } else {
    const int step = static_cast<int>(gridDim.x);
    const int lane = static_cast<int>(threadIdx.x & 31);
    SeqCursor c{0, 0, 0, min(max(__ldg(p.cu_seqlens), 0), p.L), 0, 0, 0, 0};
    cursor_load<TILES>(p, c, lane);
    // Units in snake order over the CTAs (0..C-1, then C-1..0, ...): units
    // of different documents cost differently, and alternating the
    // direction evens out what each CTA collects.  The sequence still grows,
    // as the cursor needs.
    const int cta = static_cast<int>(blockIdx.x);
    for (int r = 0;; ++r) {
      const int u = r * step + ((r & 1) ? step - 1 - cta : cta);
      Work<TILES> w;
      int k, n_tiles;
      if (!cursor_find<TILES>(p, c, lane, u, k, n_tiles, w)) return;
#pragma unroll 1
      for (int sub = 0; sub < 2; ++sub)
        if (job_tiles<MODE, TILES>(n_tiles, k, sub, w) && !f(w)) return;
    }
  }
}

// Persistent grid size: one CTA per SM at most, no more than the units (or,
// in snake order, the jobs) there are.
template <int TILES>
inline unsigned grid_size(const sdpa_impl::FwdParams& p, bool varlen, int max_ctas) {
  const long long n_units =
      varlen ? p.max_units
             : static_cast<long long>(p.B) * p.H *
                   (p.snake ? groups_per_head<TILES>(p.n_tiles) : units_per_head<TILES>(p.n_tiles));
  long long g = n_units < static_cast<long long>(max_ctas) ? n_units : max_ctas;
  if (g < 1) g = 1;
  return static_cast<unsigned>(g);
}

}  // namespace sdpa_sched
