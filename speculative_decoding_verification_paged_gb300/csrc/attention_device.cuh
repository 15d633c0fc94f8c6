// Device-side pieces shared by the two verify-attention kernels and their
// host launch code: launch constants, the kernel parameter block, the
// mma.sync kernel's tile configuration and shared-memory size, the swizzled
// tile addressing, and the split of the key-tile stream over persistent CTAs
// (cursor, tiles per CTA, partial slots).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace specv {
namespace attn {

constexpr int kConsumers = 128;               // 4 consumer warps
constexpr int kWarps = kConsumers / 32;
constexpr int kThreads = kConsumers + 32;     // + 1 producer warp
constexpr int kMaxGrid = 1024;                // persistent CTAs; each owns two partial slots
constexpr int kMaxBatch = 4096;
constexpr int kSmemBudget = 200 * 1024;       // ring + query buffers
constexpr int kBarConsumers = 1;              // named barrier id of the consumer warps

struct Params {
  const int32_t* block_table;
  const int32_t* ctx_lens;
  float* out;
  int32_t* counters;  // [B * Hkv] arrival counters, zero between calls
  float* lse;         // [2 * kMaxGrid][n_rows], log2 units
  float* opart;       // [2 * kMaxGrid][n_rows][D]
  int32_t* dev_err;
  int64_t num_blocks;
  int batch, rows_per_seq, num_q_heads, num_kv_heads, gqa, n_rows;
  int block_shift, max_blocks;
  float scale_log2;
};

// Keys per pipeline stage: 64, or 32 when D = 256 and several m-tiles share the stage.
__host__ __device__ constexpr int tile_keys(int D, int MT) { return (D >= 256 && MT > 1) ? 32 : 64; }

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <int D, int MT>
struct Cfg {
  static constexpr int TK = tile_keys(D, MT);     // keys per pipeline stage
  static constexpr int WN = kWarps / MT;          // warps splitting the keys of a tile
  static constexpr int KW = TK / WN;              // keys per warp per tile
  static constexpr int NT = KW / 8;               // 8-key n-tiles per warp
  static constexpr int KSPLIT = NT >= 4 ? 1 : 2;  // independent QK^T chains per n-tile
  static constexpr int ROWS = 16 * MT;            // packed query rows (padded)
  static constexpr int SUBS = D / 64;             // 128-byte-wide column slices
  static constexpr int TILE_BYTES = TK * D * 2;   // one K (or V) tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int Q_BYTES = ROWS * D * 2;
  // Pipeline depth: three stages when they fit; a kernel that runs one CTA per
  // SM anyway takes a fourth when it fits too, for more bytes in flight per SM
  // (the per-slot tables hold up to four stages).
  static constexpr int S3 = (3 * (STAGE_BYTES + Q_BYTES) <= kSmemBudget) ? 3 : 2;
  static constexpr bool ONE_CTA_PER_SM = 2 * (1024 + S3 * (STAGE_BYTES + Q_BYTES) + 2048 + 1024) > 228 * 1024;
  static constexpr int S = (ONE_CTA_PER_SM && S3 == 3 && 4 * (STAGE_BYTES + Q_BYTES) <= kSmemBudget) ? 4 : S3;
  static constexpr int RING_BYTES = S * STAGE_BYTES;
  static constexpr int SCRATCH_BYTES = (WN - 1) * MT * 16 * D * 4;  // cross-warp merge
  // Two CTAs per SM when their shared memory fits (228 KB per SM, 1 KB reserved per CTA);
  // then registers are capped so ten warps fit the SM's four register-file partitions,
  // and the query fragments are re-read from shared memory instead of held in registers.
  static constexpr int SMEM_EST = 1024 + RING_BYTES + S * Q_BYTES + 2048;
  static constexpr int MIN_BLOCKS = 2 * (SMEM_EST + 1024) <= 228 * 1024 ? 2 : 1;
  static constexpr bool Q_IN_REGS = MIN_BLOCKS == 1 && D <= 128;
  static_assert(KW % 16 == 0, "each warp needs whole 16-key steps");
  static_assert(WN * MT == kWarps, "warp layout");
  static_assert(SCRATCH_BYTES <= STAGE_BYTES, "merge scratch reuses one ring stage");
  static_assert(S <= 4, "per-slot tables (bad-block flags) hold four stages");
};

template <int D, int MT>
size_t smem_bytes(int batch) {
  using C = Cfg<D, MT>;
  return 1024 /* alignment slack */ + (size_t)C::RING_BYTES + (size_t)C::S * C::Q_BYTES + 2 * C::S * 8 +
         2 * 64 * 4 + 16 + align256((size_t)(batch + 2) * 4) + align256((size_t)batch * 4) + 64;
}

// Byte offset of 16-byte chunk `ch` (along D) of row `row` in a tile of `rows`
// rows stored as D/64 slices of [rows][64] bf16 with the 128-byte TMA swizzle.
__device__ __forceinline__ uint32_t swz(int row, int ch, int rows) {
  return (uint32_t)((ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// Position in the stream of key tiles: unit (b, g) and tile index inside it.
struct Cursor {
  int b, g, tile, ntiles, seq;
};

__device__ __forceinline__ void cursor_advance(Cursor& c, const int32_t* s_prefix, int B, int Hkv) {
  if (++c.tile < c.ntiles) return;
  c.tile = 0;
  ++c.seq;
  if (++c.g < Hkv) return;
  c.g = 0;
  do {
    ++c.b;
  } while (c.b < B && s_prefix[c.b + 1] == s_prefix[c.b]);
  c.ntiles = c.b < B ? s_prefix[c.b + 1] - s_prefix[c.b] : 0;
}

// Tiles per CTA. Stream-K (an even split of all T tiles, units cut wherever
// the split falls) balances any mix of context lengths, but every cut unit
// costs a partial write, an arrival and a merge. When all usable units have
// the same tile count (unit_tiles > 0), CTAs take whole units instead unless
// that loads the busiest CTA too far above the even split: by at most 2.4x
// with one unit per CTA, 1.6x with several (measured on 128-512 units of 32
// tiles: whole units win by 2-11%, and lose 2% at 1.9x with two per CTA).
__device__ __forceinline__ int64_t tiles_per_cta(int64_t T, int unit_tiles, int grid) {
  if (unit_tiles > 0) {
    const int64_t units = T / unit_tiles;
    const int64_t per_cta = (units + grid - 1) / grid;
    // per_cta * grid / units is the busiest CTA's load over the even split's
    if (per_cta * grid * 5 <= units * (per_cta == 1 ? 12 : 8)) return per_cta * unit_tiles;
  }
  return (T + grid - 1) / grid;
}

__device__ __forceinline__ Cursor cursor_at(int64_t f, const int32_t* s_prefix, int B, int Hkv) {
  int lo = 0, hi = B;  // largest b with s_prefix[b] * Hkv <= f
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)s_prefix[mid] * Hkv <= f) lo = mid; else hi = mid;
  }
  while (lo < B && s_prefix[lo + 1] == s_prefix[lo]) ++lo;  // skip empty sequences
  Cursor c;
  c.b = lo;
  c.ntiles = s_prefix[lo + 1] - s_prefix[lo];
  const int64_t r = f - (int64_t)s_prefix[lo] * Hkv;
  c.g = (int)(r / c.ntiles);
  c.tile = (int)(r - (int64_t)c.g * c.ntiles);
  c.seq = 0;
  return c;
}

// What the finaliser of a unit needs once the unit's last tile in range is done.
struct Fin {
  int b, g, seq;
  int complete;   // the whole unit lies in this CTA's range: write the output directly
  int slot;       // partial slot of this CTA's piece
  int64_t u0;     // first tile of the unit in the tile stream
  int c0, nseg;   // first CTA holding a piece of the unit, number of pieces
};

// Partial slot of the piece of unit [u0, ...) held by CTA c: slot 0 for a CTA's
// first unit, slot 1 for its last one (a CTA's middle units are always whole).
__device__ __forceinline__ int piece_slot(int c, int c0, int64_t u0, int64_t W) {
  return 2 * c + ((c == c0 && u0 > (int64_t)c * W) ? 1 : 0);
}

}  // namespace attn
}  // namespace specv
