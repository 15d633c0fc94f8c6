// Paged GQA verification attention (sm_103a).
//
// The verify pass of chain speculative decoding runs the last committed token
// and the k drafts of every sequence through the target at once (the "wide
// batched verify" of onnxruntime-genai PR #2457); its attention reads a
// block-paged KV cache ("paged CuTe verification attention", lmdeploy PR
// #5019 summary). Row i of a sequence with ctx tokens (verify tokens
// included) attends to keys t <= ctx - (k+1) + i, so the rows are causal along
// the draft chain.
//
// Design (GB300):
//  * All (k+1)*G query rows that share one kv head are packed into the M
//    dimension of the tensor-core tile, so each K/V byte is read from HBM once
//    per kv head. M = 16, 32 or 64 rows (1, 2 or 4 m16 tiles).
//  * One launch, stream-K split: the key tiles of all (sequence, kv head)
//    units are laid end to end and every persistent CTA takes an equal,
//    contiguous range of that tile stream, so the load is balanced for any mix
//    of context lengths. A unit that spans several CTAs is merged by its
//    log-sum-exp: every CTA that holds a piece writes a normalised partial,
//    and the last one to finish (an atomic counter per unit, which it resets)
//    combines them. The range split is computed inside the kernel from
//    ctx_lens, so no host synchronisation and no extra launch is needed.
//    When every unit has the same length the ranges follow unit boundaries
//    instead (whole units per CTA, no partials), as long as that leaves the
//    load close enough to even (tiles_per_cta).
//  * A producer warp stages paged K/V tiles (and each unit's query rows) into
//    128-byte-swizzled shared memory with tiled TMA copies (one 3-D box per
//    KV block piece and 64-wide slice of the head dimension), completing on
//    per-stage mbarriers; the ring runs across unit boundaries and the four
//    consumer warps release each stage through a second mbarrier. Block ids
//    are range-checked before they are used; a bad or unallocated block is
//    read as zeros through an out-of-range box coordinate.
//  * QK^T and PV run on mma.sync m16n8k16 (bf16 in, fp32 accumulate), several
//    independent accumulator chains per warp. P is split into a bf16 high part
//    and a bf16 remainder and both are multiplied with V, so PV keeps ~16
//    mantissa bits of P; softmax statistics and the output stay fp32.
//  * At the end of a unit the warps that split a tile's keys write their
//    partial outputs to the freed stage and all consumer threads merge them,
//    one (row, 16-column) segment each.
//  * Head dim 128 with 32 or more packed rows runs on a second kernel in this
//    file, on 5th-generation tensor cores (tcgen05, tensor memory): see the
//    comment before namespace tc. The host picks one per call.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <cuda.h>

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

template <int D, int MT>
__global__ void __launch_bounds__(kThreads, Cfg<D, MT>::MIN_BLOCKS) verify_attention_kernel(const Params p,
                                                                    const __grid_constant__ CUtensorMap tm_q,
                                                                    const __grid_constant__ CUtensorMap tm_k,
                                                                    const __grid_constant__ CUtensorMap tm_v) {
  using C = Cfg<D, MT>;
  constexpr int TK = C::TK, WN = C::WN, KW = C::KW, NT = C::NT, KSPLIT = C::KSPLIT, S = C::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* qbuf = ring + C::RING_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(qbuf + S * C::Q_BYTES);
  uint64_t* empty = full + S;
  float* s_m = reinterpret_cast<float*>(empty + S);  // [64] cross-warp max
  float* s_l = s_m + 64;                              // [64] cross-warp sum
  int32_t* s_bad = reinterpret_cast<int32_t*>(s_l + 64);  // [S] per unit slot: a block id was bad
  int32_t* s_prefix = s_bad + 4;                           // [B + 1]
  int32_t* s_ctx = s_prefix + ((p.batch + 2 + 63) & ~63);   // [B] context lengths
  int32_t* s_misc = s_ctx + ((p.batch + 63) & ~63);          // [16]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.batch, Hkv = p.num_kv_heads, G = p.gqa, R = p.rows_per_seq;
  const int64_t max_ctx = (int64_t)p.max_blocks << p.block_shift;

  // ---- 1. split plan: per-sequence tile counts and their exclusive prefix (same in every CTA)
  {
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = tid * per;
    int mine = 0, nt_min = INT32_MAX, nt_max = 0;  // tile counts of the usable sequences
    if (tid == 0) {
      s_misc[12] = INT32_MAX;
      s_misc[13] = 0;
    }
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        const int c = p.ctx_lens[b];
        if (c >= R && (int64_t)c <= max_ctx) {
          const int nt = (c + TK - 1) / TK;
          mine += nt;
          nt_min = min(nt_min, nt);
          nt_max = max(nt_max, nt);
        }
      }
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_misc[warp] = incl;
    __syncthreads();
    if (nt_max > 0) {
      atomicMin(&s_misc[12], nt_min);
      atomicMax(&s_misc[13], nt_max);
    }
    int run = incl - mine;
    for (int w = 0; w < warp; ++w) run += s_misc[w];
    if (tid == kThreads - 1) s_prefix[B] = run + mine;
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        s_prefix[b] = run;
        const int c = p.ctx_lens[b];
        s_ctx[b] = c;
        if (c >= R && (int64_t)c <= max_ctx) run += (c + TK - 1) / TK;
      }
    }
    if (tid == 0) {
      for (int s = 0; s < S; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], kWarps);
      }
      fence_mbar_init();
    }
    __syncthreads();
  }
  // unusable sequences (ctx out of range) get zero rows, each from one CTA
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    if (s_prefix[b + 1] != s_prefix[b]) continue;
    if (tid == 0) raise_error(p.dev_err, SPEC_DEVERR_CTX_LEN);
    float4* dst = reinterpret_cast<float4*>(p.out + (int64_t)b * R * p.num_q_heads * D);
    for (int i = tid; i < R * p.num_q_heads * D / 4; i += kThreads) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int64_t T = (int64_t)s_prefix[B] * Hkv;
  if (T == 0) return;
  const int unit_tiles = s_misc[12] == s_misc[13] ? s_misc[13] : 0;  // 0: units of several lengths
  const int64_t W = tiles_per_cta(T, unit_tiles, (int)gridDim.x);
  const int64_t f0 = (int64_t)blockIdx.x * W;
  const int64_t f1 = min(T, f0 + W);
  if (f0 >= f1) return;

  const uint32_t ring_u32 = smem_u32(ring);
  const uint32_t q_u32 = smem_u32(qbuf);

  // =====================================================================
  // Producer warp: one thread issues every TMA copy, S stages ahead.
  // =====================================================================
  if (warp == kWarps) {
    // Lane 0 issues the copies. The warp keeps a window of 32 consecutive
    // block-table entries of the current sequence in its lanes (one coalesced
    // load per 32 blocks), so issuing a tile never waits on a table lookup.
    constexpr int BHmax = TK;
    const int bs = 1 << p.block_shift;
    const int BH = bs < TK ? bs : TK;  // rows per KV box
    const int pieces = TK / BH;
    Cursor ld = cursor_at(f0, s_prefix, B, Hkv);
    bool fresh = true;
    int win_b = -1, win_base = 0, win_val = 0;
    for (int64_t f = f0; f < f1; ++f) {
      const int s = (int)((f - f0) % S);
      const int64_t rnd = (f - f0) / S;
      const int b = ld.b, g = ld.g;
      const int ctx = s_ctx[b];
      const int t0 = ld.tile * TK;
      const int slot = ld.seq % S;
      int zc[BHmax / 16 > 0 ? BHmax / 16 : 1];  // box row coordinate per piece (bs >= 16)
      bool bad = false;
#pragma unroll
      for (int pc = 0; pc < BHmax / 16; ++pc) {
        if (pc >= pieces) break;
        const int t = t0 + pc * BH;
        int z = -BH;  // fully out of range: the box reads as zeros
        if (t < ctx) {
          const int n = t >> p.block_shift;  // logical block
          if (b != win_b || n < win_base || n >= win_base + 32) {
            win_b = b;
            win_base = n;
            const int nb = (ctx + bs - 1) >> p.block_shift;
            win_val = (n + lane < nb) ? __ldg(p.block_table + (int64_t)b * p.max_blocks + n + lane) : 0;
          }
          const int32_t phys = __shfl_sync(0xffffffffu, win_val, n - win_base);
          if (phys < 0 || (int64_t)phys >= p.num_blocks) {
            bad = true;
          } else {
            z = (int)(((int64_t)phys << p.block_shift) + (t & (bs - 1)));
          }
        }
        zc[pc] = z;
      }
      if (lane == 0) {
        if (rnd > 0 && !mbar_wait_bounded(&empty[s], (uint32_t)((rnd - 1) & 1)))
          raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        if (fresh) s_bad[slot] = 0;
        if (bad) s_bad[slot] = 1;
        const uint32_t q_bytes = fresh ? (uint32_t)(R * G * D * 2) : 0u;
        mbar_arrive_expect_tx(&full[s], (uint32_t)C::STAGE_BYTES + q_bytes);
        if (fresh) {
          const uint32_t qdst = q_u32 + slot * C::Q_BYTES;
#pragma unroll
          for (int sub = 0; sub < C::SUBS; ++sub)
            tma_load_3d(qdst + sub * C::ROWS * 128, &tm_q, sub * 64, g * G, b * R, &full[s]);
        }
        const uint32_t kdst = ring_u32 + s * C::STAGE_BYTES;
        const uint32_t vdst = kdst + C::TILE_BYTES;
#pragma unroll
        for (int pc = 0; pc < BHmax / 16; ++pc) {
          if (pc >= pieces) break;
#pragma unroll
          for (int sub = 0; sub < C::SUBS; ++sub) {
            const uint32_t off = sub * TK * 128 + pc * BH * 128;
            tma_load_3d(kdst + off, &tm_k, sub * 64, g, zc[pc], &full[s]);
            tma_load_3d(vdst + off, &tm_v, sub * 64, g, zc[pc], &full[s]);
          }
        }
      }
      __syncwarp();
      const int before = ld.seq;
      cursor_advance(ld, s_prefix, B, Hkv);
      fresh = ld.seq != before;
    }
    return;
  }

  // =====================================================================
  // Consumer warps.
  // =====================================================================
  const int mt = warp / WN, wn = warp % WN;
  // padded query rows stay zero in every query buffer (TMA writes rows < R*G only)
  for (int i = tid; i < S * C::SUBS * (C::ROWS - p.n_rows) * 8; i += kConsumers) {
    const int ch = i % 8, rest = i / 8;
    const int r = p.n_rows + rest % (C::ROWS - p.n_rows);
    const int bs_sub = rest / (C::ROWS - p.n_rows);
    const int buf = bs_sub / C::SUBS, sub = bs_sub % C::SUBS;
    *reinterpret_cast<uint4*>(qbuf + buf * C::Q_BYTES + sub * C::ROWS * 128 + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
  }
  named_sync(kBarConsumers, kConsumers);

  Cursor cu = cursor_at(f0, s_prefix, B, Hkv);
  bool cu_fresh = true;
  bool from_zero = true;
  float o[D / 8][4];
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  uint32_t qf[C::Q_IN_REGS ? D / 16 : 1][4];
  int ctx = 0, prefix_len = 0, lim0 = 0, lim1 = 0;
  const int row_in = lane >> 2;
  const int r0 = mt * 16 + row_in, r1 = r0 + 8;

  // Combine a finished unit: merge the key-split warps, then write the output
  // (whole unit) or a normalised partial, and let the last piece merge them all.
  auto finalize = [&](const Fin& F, float* scratch) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    named_sync(kBarConsumers, kConsumers);  // every warp is done reading the stage used as scratch
    // Parallel combine, when the freed stage holds every warp's O: each warp writes
    // its O and row statistics, then every consumer thread merges one
    // (row, 16-column) segment over the WN key-split warps and writes it with
    // 16-byte stores. Otherwise warp column 0 merges the others' O alone.
    constexpr bool kParallel = WN > 1 && (size_t)WN * MT * 16 * D * 4 <= (size_t)C::STAGE_BYTES;
    if constexpr (kParallel) {
      const int base = (wn * MT + mt) * 16;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const int d = n * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2*>(&scratch[(base + row_in) * D + d]) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(&scratch[(base + row_in + 8) * D + d]) = make_float2(o[n][2], o[n][3]);
      }
      if ((lane & 3) == 0) {
        s_m[base + row_in] = m_run[0];
        s_l[base + row_in] = l_run[0];
        s_m[base + row_in + 8] = m_run[1];
        s_l[base + row_in + 8] = l_run[1];
      }
      const bool bad = named_sync_or(kBarConsumers, kConsumers, s_bad[F.seq % S] != 0);
      constexpr int kSeg = D / 16;  // 16-column segments per row
      for (int item = tid; item < MT * 16 * kSeg; item += kConsumers) {
        const int r = item / kSeg, seg = item - r * kSeg;
        if (r >= p.n_rows) continue;
        const int rt = r >> 4, ri = r & 15;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < WN; ++w) M = fmaxf(M, s_m[(w * MT + rt) * 16 + ri]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f;
        float4 acc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < WN; ++w) {
          const int sr = (w * MT + rt) * 16 + ri;
          const float f = fast_exp2(s_m[sr] - Mu);
          L += s_l[sr] * f;
          const float4* src = reinterpret_cast<const float4*>(&scratch[sr * D + seg * 16]);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 v = src[c];
            acc[c].x += v.x * f;
            acc[c].y += v.y * f;
            acc[c].z += v.z * f;
            acc[c].w += v.w * f;
          }
        }
        const float inv = (L > 0.f && !bad) ? 1.f / L : 0.f;
        float* dst;
        if (F.complete) {
          const int i = r / G, j = r - i * G;
          dst = p.out + (((int64_t)F.b * R + i) * p.num_q_heads + F.g * G + j) * D;
        } else {
          dst = p.opart + ((int64_t)F.slot * p.n_rows + r) * D;
          if (seg == 0) {
            float lse2 = L > 0.f ? M + __log2f(L) : -INFINITY;
            if (bad) lse2 = __int_as_float(0x7fc00000);  // NaN marks an unusable piece
            __stcg(p.lse + (int64_t)F.slot * p.n_rows + r, lse2);
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          __stcg(reinterpret_cast<float4*>(dst + seg * 16) + c,
                 make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv));
      }
      if (bad && tid == 0) raise_error(p.dev_err, SPEC_DEVERR_BLOCK_ID);
    } else {
    if constexpr (WN > 1) {
        if (wn > 0) {
          const int base = ((wn - 1) * MT + mt) * 16;
#pragma unroll
          for (int n = 0; n < D / 8; ++n) {
            const int d = n * 8 + 2 * (lane & 3);
            *reinterpret_cast<float2*>(&scratch[(base + row_in) * D + d]) = make_float2(o[n][0], o[n][1]);
            *reinterpret_cast<float2*>(&scratch[(base + row_in + 8) * D + d]) = make_float2(o[n][2], o[n][3]);
          }
          if ((lane & 3) == 0) {
            s_m[base + row_in] = m_run[0];
            s_l[base + row_in] = l_run[0];
            s_m[base + row_in + 8] = m_run[1];
            s_l[base + row_in + 8] = l_run[1];
          }
        }
      }
      const bool bad = named_sync_or(kBarConsumers, kConsumers, s_bad[F.seq % S] != 0);
      if (wn == 0) {
        float M[2] = {m_run[0], m_run[1]};
        if constexpr (WN > 1) {
#pragma unroll
          for (int w = 1; w < WN; ++w) {
            const int base = ((w - 1) * MT + mt) * 16 + row_in;
            M[0] = fmaxf(M[0], s_m[base]);
            M[1] = fmaxf(M[1], s_m[base + 8]);
          }
        }
        float Mu[2], L[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          Mu[h] = M[h] == -INFINITY ? 0.f : M[h];
          const float f = fast_exp2(m_run[h] - Mu[h]);
          L[h] = l_run[h] * f;
#pragma unroll
          for (int n = 0; n < D / 8; ++n) {
            o[n][2 * h] *= f;
            o[n][2 * h + 1] *= f;
          }
        }
        if constexpr (WN > 1) {
#pragma unroll
          for (int w = 1; w < WN; ++w) {
            const int base = ((w - 1) * MT + mt) * 16 + row_in;
            const float fa = fast_exp2(s_m[base] - Mu[0]);
            const float fb = fast_exp2(s_m[base + 8] - Mu[1]);
            L[0] += s_l[base] * fa;
            L[1] += s_l[base + 8] * fb;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
              const int d = n * 8 + 2 * (lane & 3);
              const float2 va = *reinterpret_cast<const float2*>(&scratch[base * D + d]);
              const float2 vb = *reinterpret_cast<const float2*>(&scratch[(base + 8) * D + d]);
              o[n][0] += va.x * fa;
              o[n][1] += va.y * fa;
              o[n][2] += vb.x * fb;
              o[n][3] += vb.y * fb;
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = h == 0 ? r0 : r1;
          if (r < p.n_rows) {
            const float inv = (L[h] > 0.f && !bad) ? 1.f / L[h] : 0.f;
            float* dst;
            if (F.complete) {
              const int i = r / G, j = r - i * G;
              dst = p.out + (((int64_t)F.b * R + i) * p.num_q_heads + F.g * G + j) * D;
            } else {
              dst = p.opart + ((int64_t)F.slot * p.n_rows + r) * D;
              if ((lane & 3) == 0) {
                float lse2 = L[h] > 0.f ? M[h] + __log2f(L[h]) : -INFINITY;
                if (bad) lse2 = __int_as_float(0x7fc00000);  // NaN marks an unusable piece
                p.lse[(int64_t)F.slot * p.n_rows + r] = lse2;
              }
            }
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
              const int d = n * 8 + 2 * (lane & 3);
              *reinterpret_cast<float2*>(dst + d) = make_float2(o[n][2 * h] * inv, o[n][2 * h + 1] * inv);
            }
          }
        }
      }
      if (bad && tid == 0) raise_error(p.dev_err, SPEC_DEVERR_BLOCK_ID);
    }
    if (!F.complete) {
      // release: every partial store of the CTA precedes the arrival
      named_sync(kBarConsumers, kConsumers);
      const int unit = F.b * Hkv + F.g;
      if (tid == 0) {
        __threadfence();
        const int last = atomicAdd(p.counters + unit, 1) == F.nseg - 1;
        if (last) __threadfence();  // acquire: the other pieces are visible
        s_misc[8] = last;
      }
      named_sync(kBarConsumers, kConsumers);
      if (s_misc[8]) {
        // out = sum_pieces 2^(lse - M) * partial / sum_pieces 2^(lse - M), merged
        // online; a thread takes kB float4 columns at once and loads a piece's
        // values for all of them together, so each piece costs one L2 round trip
        constexpr int kB = 4;
        for (int base = tid; base < p.n_rows * (D / 4); base += kB * kConsumers) {
          float M[kB], ws[kB];
          float4 acc[kB];
          bool bad[kB];
#pragma unroll
          for (int u = 0; u < kB; ++u) {
            M[u] = -INFINITY;
            ws[u] = 0.f;
            acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            bad[u] = false;
          }
          for (int sg = 0; sg < F.nseg; ++sg) {
            const int64_t slot = piece_slot(F.c0 + sg, F.c0, F.u0, W);
            float l[kB];
            float4 v[kB];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
              const int idx = base + u * kConsumers;
              l[u] = -INFINITY;
              v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (idx < p.n_rows * (D / 4)) {
                const int r = idx / (D / 4), d4 = idx - r * (D / 4);
                l[u] = __ldcg(p.lse + slot * p.n_rows + r);
                v[u] = __ldcg(reinterpret_cast<const float4*>(p.opart + (slot * p.n_rows + r) * D) + d4);
              }
            }
#pragma unroll
            for (int u = 0; u < kB; ++u) {
              const float lv = l[u];
              bad[u] |= lv != lv;
              if (!(lv > -INFINITY)) continue;
              const float Mn = fmaxf(M[u], lv);
              const float a = exp2f(M[u] - Mn), wgt = exp2f(lv - Mn);
              acc[u].x = acc[u].x * a + wgt * v[u].x;
              acc[u].y = acc[u].y * a + wgt * v[u].y;
              acc[u].z = acc[u].z * a + wgt * v[u].z;
              acc[u].w = acc[u].w * a + wgt * v[u].w;
              ws[u] = ws[u] * a + wgt;
              M[u] = Mn;
            }
          }
#pragma unroll
          for (int u = 0; u < kB; ++u) {
            const int idx = base + u * kConsumers;
            if (idx < p.n_rows * (D / 4)) {
              const int r = idx / (D / 4), d4 = idx - r * (D / 4);
              const float sc = (bad[u] || !(ws[u] > 0.f)) ? 0.f : 1.f / ws[u];  // 0: bad piece or no key seen
              const float4 o = sc == 0.f ? make_float4(0.f, 0.f, 0.f, 0.f)
                                         : make_float4(acc[u].x * sc, acc[u].y * sc, acc[u].z * sc, acc[u].w * sc);
              const int i = r / G, j = r - i * G;
              __stcg(reinterpret_cast<float4*>(p.out + (((int64_t)F.b * R + i) * p.num_q_heads + F.g * G + j) * D) + d4,
                     o);
            }
          }
        }
        if (tid == 0) p.counters[unit] = 0;  // ready for the next call
      }
    }
    fence_proxy_async_smem();  // scratch writes before the next TMA into this stage
    named_sync(kBarConsumers, kConsumers);
  };

  for (int64_t f = f0; f < f1; ++f) {
    const int stage = (int)((f - f0) % S);
    const int64_t rnd = (f - f0) / S;
    if (!mbar_wait_bounded(&full[stage], (uint32_t)(rnd & 1)) && tid == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
    const uint32_t kbase = ring_u32 + stage * C::STAGE_BYTES;
    const uint32_t vbase = kbase + C::TILE_BYTES;
    const uint32_t qb = q_u32 + (cu.seq % S) * C::Q_BYTES;
    const int t0 = cu.tile * TK;

    if (cu_fresh) {
      from_zero = cu.tile == 0;
      ctx = s_ctx[cu.b];
      prefix_len = ctx - R;
      lim0 = prefix_len + (r0 < p.n_rows ? r0 / G : 0);
      lim1 = prefix_len + (r1 < p.n_rows ? r1 / G : 0);
#pragma unroll
      for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
      if constexpr (C::Q_IN_REGS) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int mi = lane >> 3;
          const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
          ldmatrix_x4(qb + swz(row, 2 * ks + (mi >> 1), C::ROWS), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
        }
      }
    }
    // keys past the context in the last tile may hold stale cache bytes: zero those V rows
    if (t0 + TK > ctx) {
      const int valid = ctx - t0;
      for (int i = tid; i < (TK - valid) * (D / 8); i += kConsumers) {
        const int row = valid + i / (D / 8), ch = i % (D / 8);
        *reinterpret_cast<uint4*>(ring + stage * C::STAGE_BYTES + C::TILE_BYTES + swz(row, ch, TK)) =
            make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      named_sync(kBarConsumers, kConsumers);
    }
    const int kw0 = wn * KW;

    // ---- S = Q K^T for this warp's KW keys (KSPLIT independent chains per n-tile)
    float sacc[KSPLIT][NT][4];
#pragma unroll
    for (int c = 0; c < KSPLIT; ++c)
#pragma unroll
      for (int n = 0; n < NT; ++n) sacc[c][n][0] = sacc[c][n][1] = sacc[c][n][2] = sacc[c][n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      if constexpr (C::Q_IN_REGS) {
        a[0] = qf[ks][0]; a[1] = qf[ks][1]; a[2] = qf[ks][2]; a[3] = qf[ks][3];
      } else {
        const int mi = lane >> 3;
        const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
        ldmatrix_x4(qb + swz(row, 2 * ks + (mi >> 1), C::ROWS), a[0], a[1], a[2], a[3]);
      }
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        const int mi = lane >> 3;
        const int key = kw0 + np * 16 + (mi >> 1) * 8 + (lane & 7);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kbase + swz(key, 2 * ks + (mi & 1), TK), b0, b1, b2, b3);
        mma_bf16_16816(sacc[ks % KSPLIT][2 * np], a, b0, b1);
        mma_bf16_16816(sacc[ks % KSPLIT][2 * np + 1], a, b2, b3);
      }
    }
    float s[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sacc[0][n][e];
        if constexpr (KSPLIT > 1) v += sacc[1][n][e];
        s[n][e] = v;
      }

    // ---- scale, causal mask, online softmax (log2 domain, lazy rescaling)
    const bool needs_mask = t0 + TK - 1 > prefix_len;
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[n][e] * p.scale_log2;
        if (needs_mask) {
          const int t = t0 + kw0 + n * 8 + 2 * (lane & 3) + (e & 1);
          if (t > (e < 2 ? lim0 : lim1)) x = -INFINITY;
        }
        s[n][e] = x;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], x);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
      tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
    }
    // The running max may lag the true max by up to 8 (log2 units): P <= 256 stays
    // exact enough in fp32 and in the hi/lo bf16 split, and O is rescaled rarely.
    const bool grow = tmax[0] > m_run[0] + 8.f || tmax[1] > m_run[1] + 8.f;
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float m_new = fmaxf(m_run[h], tmax[h]);
        const float alpha = m_new == -INFINITY ? 1.f : fast_exp2(m_run[h] - m_new);
        m_run[h] = m_new;
        l_run[h] *= alpha;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          o[n][2 * h] *= alpha;
          o[n][2 * h + 1] *= alpha;
        }
      }
    }
    const float m_use0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
    const float m_use1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = fast_exp2(s[n][e] - (e < 2 ? m_use0 : m_use1));
        s[n][e] = pv;
        l_run[e >> 1] += pv;
      }
    }

    // ---- O += P V with P = P_hi + P_lo (two bf16 products)
#pragma unroll
    for (int kk = 0; kk < KW / 16; ++kk) {
      uint32_t ah[4], al[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float* pp = s[2 * kk + (r >> 1)];
        const float x0 = pp[2 * (r & 1)], x1 = pp[2 * (r & 1) + 1];
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
        const float2 hf = __bfloat1622float2(h2);
        ah[r] = *reinterpret_cast<const uint32_t*>(&h2);
        al[r] = pack_bf16(x0 - hf.x, x1 - hf.y);
      }
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int mi = lane >> 3;
        const int key = kw0 + kk * 16 + (mi & 1) * 8 + (lane & 7);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vbase + swz(key, 2 * dp + (mi >> 1), TK), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], ah, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], ah, b2, b3);
        mma_bf16_16816(o[2 * dp], al, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], al, b2, b3);
      }
    }

    // ---- end of this unit's tiles in range: finalise (the stage is the scratch)
    if (f == f1 - 1 || cu.tile == cu.ntiles - 1) {
      Fin fin;
      const int64_t u0 = (int64_t)s_prefix[cu.b] * Hkv + (int64_t)cu.g * cu.ntiles;
      fin.b = cu.b;
      fin.g = cu.g;
      fin.seq = cu.seq;
      fin.complete = from_zero && cu.tile == cu.ntiles - 1;
      fin.u0 = u0;
      fin.c0 = (int)(u0 / W);
      fin.nseg = (int)((u0 + cu.ntiles - 1) / W) - fin.c0 + 1;
      fin.slot = piece_slot((int)blockIdx.x, fin.c0, u0, W);
      finalize(fin, reinterpret_cast<float*>(ring + stage * C::STAGE_BYTES));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    const int before = cu.seq;
    cursor_advance(cu, s_prefix, B, Hkv);
    cu_fresh = cu.seq != before;
  }
}

// ---------------------------------------------------------------------------
// Tensor-core (tcgen05) kernel for D = 128.
//
// The keys are the MMA's M dimension (128 per tile) and the packed query rows
// are N (16, 32 or 64), so every M = 128 MMA is fully used for any row count:
//   S^T[128 keys x N] = K[128 x 128] . Q^T            (K, Q K-major in smem)
//   O^T[128 d x N]   += V^T[128 x 128 keys] . P^T     (V and P MN-major)
// with S^T (two buffers) and O^T in tensor memory. Warp 0 stages K/V/Q with
// TMA, warp 1 issues the MMAs (one thread; QK of tile i+1 before P.V of tile
// i), warps 2-9 run the softmax in two warpgroups, each owning half of the
// rows; a warp reads the 32-lane quarter of tensor memory that its index
// selects, i.e. 32 keys of S^T and 32 dims of O^T. P is written to shared
// memory as a bf16 high part and a bf16 remainder and both are multiplied with
// V. The running row max may lag by up to 8 (log2 units); a tile that exceeds
// it takes the slow path: exact row max, and the accumulated O^T and row sums
// are rescaled in place.
// ---------------------------------------------------------------------------
namespace tc {

constexpr int D = 128;
constexpr int TK = 128;                      // keys per tile (MMA M)
constexpr int kSoftmaxWarps = 8;             // two warpgroups, each owning half the query rows
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kThreads = 64 + kSoftmaxThreads;  // producer warp, MMA warp, softmax warps
// Register budget: up to three warps share an SM sub-partition (16K registers),
// so a thread may hold at most 168 registers; declaring 384 threads caps it there.
constexpr int kRegBudgetThreads = 384;
constexpr int kBarGroup0 = 2;                // named barriers: one per softmax warpgroup,
constexpr int kBarSoftmax = 4;               // all softmax warps,
constexpr int kBarTail = 5;                  // MMA warp + softmax warps
constexpr int kTmemCols = 256;               // S^T buffers at columns 0 and N, O^T at 2N

template <int MT>
struct Cfg {
  static constexpr int N = 16 * MT;                     // packed query rows (MMA N)
  static constexpr int CW = N / 2;                      // rows (tensor-memory columns) per warpgroup
  static constexpr int TILE_BYTES = TK * D * 2;         // 32 KB: two [128][64] slices
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;    // K + V
  static constexpr int Q_BYTES = N * D * 2;             // two [N][64] slices
  static constexpr int P_BYTES = N * TK * 2;            // one of P_hi / P_lo: [128 keys][N rows]
  // P is the P.V operand B in MN-major layout: the N rows of a key are contiguous
  // (N * 2 bytes) and swizzled at that width (32, 64 or 128 bytes), so a softmax
  // thread, which owns one key, writes its rows with 16-byte stores.
  static constexpr uint32_t P_LAYOUT = N == 16 ? 6u : (N == 32 ? 4u : 2u);
  static constexpr int P_SWZ_SHIFT = N == 16 ? 2 : (N == 32 ? 1 : 0);  // key bits that pick the XOR
  static constexpr int P_SWZ_MASK = N == 16 ? 1 : (N == 32 ? 3 : 7);
};

// Dynamic shared memory: stages + query buffers, NP P buffers (hi + lo), barriers,
// reductions, output row offsets, and the per-sequence plan (which grows with the batch).
template <int MT, int S, int NP>
size_t smem_bytes(int batch) {
  using C = Cfg<MT>;
  return 1024 + (size_t)S * (C::STAGE_BYTES + C::Q_BYTES) + (size_t)NP * 2 * C::P_BYTES + 64 * 8 + 4 * 64 * 4 +
         64 * 4 + 64 * 8 + 64 + align256((size_t)(batch + 2) * 4) + align256((size_t)batch * 4) + 128;
}

// Reduction of CW columns over the 32 lanes of a warp by recursive halving: at
// level j every lane keeps half of its remaining columns (chosen by lane bit j)
// and receives the partner lane's values for that half, so CW - 1 shuffles cover
// the first log2(CW) levels; the rest is a plain butterfly on one value. Lane l
// ends with the result for column reduced_col<CW>(l); v is destroyed.
template <int CW>
__device__ __forceinline__ int reduced_col(int lane) {
  int c = 0;
#pragma unroll
  for (int j = 0; (CW >> j) > 1; ++j) c += ((lane >> j) & 1) * (CW >> (j + 1));
  return c;
}
template <int CW, bool kMax>
__device__ __forceinline__ float reduce_cols(float (&v)[CW], int lane) {
#pragma unroll
  for (int j = 0; (CW >> j) > 1; ++j) {
    const int half = (CW >> j) / 2;
    const bool upper = (lane >> j) & 1;
#pragma unroll
    for (int t = 0; t < half; ++t) {
      const float mine = upper ? v[t + half] : v[t];
      const float other = upper ? v[t] : v[t + half];
      const float recv = __shfl_xor_sync(0xffffffffu, other, 1 << j);
      v[t] = kMax ? fmaxf(mine, recv) : mine + recv;
    }
  }
  float r = v[0];
#pragma unroll
  for (int j = 0; j < 5; ++j) {
    if ((CW >> j) > 1) continue;
    const float o = __shfl_xor_sync(0xffffffffu, r, 1 << j);
    r = kMax ? fmaxf(r, o) : r + o;
  }
  return r;
}

// CW consecutive columns of this thread's lane, starting at `taddr`.
template <int CW>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float (&v)[CW]) {
  if constexpr (CW == 8) {
    tmem_ld8(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < CW / 16; ++c) tmem_ld16(taddr + c * 16, *reinterpret_cast<float(*)[16]>(&v[c * 16]));
  }
  tmem_wait_ld_regs<CW>(v);
}
template <int CW>
__device__ __forceinline__ void tmem_store_cols(uint32_t taddr, const float (&v)[CW]) {
  if constexpr (CW == 8) {
    tmem_st8(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < CW / 16; ++c) tmem_st16(taddr + c * 16, *reinterpret_cast<const float(*)[16]>(&v[c * 16]));
  }
  tmem_wait_st();
}

template <int MT, int S, int NP>
__global__ void __launch_bounds__(kRegBudgetThreads, 1) verify_attention_tc_kernel(
    const Params p, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v) {
  using C = Cfg<MT>;
  constexpr int N = C::N, CW = C::CW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* qbuf = ring + S * C::STAGE_BYTES;
  uint8_t* pbuf = qbuf + S * C::Q_BYTES;  // NP x (P_hi, P_lo)
  // K and V of a stage arrive and are released separately: K is free once QK is
  // done, a tile earlier than V, so the producer can fetch the next K sooner.
  uint64_t* full_k = reinterpret_cast<uint64_t*>(pbuf + NP * 2 * C::P_BYTES);
  uint64_t* full_v = full_k + S;
  uint64_t* empty_k = full_v + S;
  uint64_t* empty_v = empty_k + S;
  uint64_t* s_full = empty_v + S;   // [2]: S^T buffer b holds QK of the tile
  uint64_t* p_full = s_full + 2;  // [2]: P of tile i written (one arrival per softmax warp)
  uint64_t* pv_done = p_full + 2; // [NP]: P.V of the tile that used P buffer j is complete
  uint64_t* fin_bar = pv_done + NP;
  float* s_red = reinterpret_cast<float*>(full_k + 64);   // [4][64] per-quarter row reductions
  float* s_mrun = s_red + 4 * 64;                         // [64] running row max (64-row tiles)
  int64_t* s_rowoff = reinterpret_cast<int64_t*>(s_mrun + 64);  // [64] output offset of each row
  int32_t* s_bad = reinterpret_cast<int32_t*>(s_rowoff + 64);  // [4]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_bad + 4);   // tensor-memory base
  int32_t* s_prefix = reinterpret_cast<int32_t*>(s_bad + 16);
  int32_t* s_ctx = s_prefix + ((p.batch + 2 + 63) & ~63);
  int32_t* s_misc = s_ctx + ((p.batch + 63) & ~63);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.batch, Hkv = p.num_kv_heads, G = p.gqa, R = p.rows_per_seq;
  const int64_t max_ctx = (int64_t)p.max_blocks << p.block_shift;

  // ---- 1. split plan (every CTA): per-sequence tile counts and their prefix
  {
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = tid * per;
    int mine = 0, nt_min = INT32_MAX, nt_max = 0;  // tile counts of the usable sequences
    if (tid == 0) {
      s_misc[12] = INT32_MAX;
      s_misc[13] = 0;
    }
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        const int c = p.ctx_lens[b];
        if (c >= R && (int64_t)c <= max_ctx) {
          const int nt = (c + TK - 1) / TK;
          mine += nt;
          nt_min = min(nt_min, nt);
          nt_max = max(nt_max, nt);
        }
      }
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_misc[warp] = incl;
    __syncthreads();
    if (nt_max > 0) {
      atomicMin(&s_misc[12], nt_min);
      atomicMax(&s_misc[13], nt_max);
    }
    int run = incl - mine;
    for (int w = 0; w < warp; ++w) run += s_misc[w];
    if (tid == kThreads - 1) s_prefix[B] = run + mine;
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        s_prefix[b] = run;
        const int c = p.ctx_lens[b];
        s_ctx[b] = c;
        if (c >= R && (int64_t)c <= max_ctx) run += (c + TK - 1) / TK;
      }
    }
    if (tid == 0) {
      for (int s = 0; s < S; ++s) {
        mbar_init(&full_k[s], 1);
        mbar_init(&full_v[s], 1);
        mbar_init(&empty_k[s], 1);
        mbar_init(&empty_v[s], 1);
      }
      for (int j = 0; j < 2; ++j) {
        mbar_init(&s_full[j], 1);
        mbar_init(&p_full[j], kSoftmaxWarps);
      }
      for (int j = 0; j < NP; ++j) mbar_init(&pv_done[j], 1);
      mbar_init(fin_bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
  }
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    if (s_prefix[b + 1] != s_prefix[b]) continue;
    if (tid == 0) raise_error(p.dev_err, SPEC_DEVERR_CTX_LEN);
    float4* dst = reinterpret_cast<float4*>(p.out + (int64_t)b * R * p.num_q_heads * D);
    for (int i = tid; i < R * p.num_q_heads * D / 4; i += kThreads) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int64_t T = (int64_t)s_prefix[B] * Hkv;
  if (T == 0) return;
  const int unit_tiles = s_misc[12] == s_misc[13] ? s_misc[13] : 0;  // 0: units of several lengths
  const int64_t W = tiles_per_cta(T, unit_tiles, (int)gridDim.x);
  const int64_t f0 = (int64_t)blockIdx.x * W;
  const int64_t f1 = min(T, f0 + W);
  if (f0 >= f1) return;
  const int n_tiles = (int)(f1 - f0);

  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  // padded query rows stay zero in every query buffer (TMA writes rows < R*G only)
  for (int i = tid; i < S * 2 * (N - p.n_rows) * 8; i += kThreads) {
    const int ch = i % 8, rest = i / 8;
    const int r = p.n_rows + rest % (N - p.n_rows);
    const int bsub = rest / (N - p.n_rows);
    const int buf = bsub / 2, sub = bsub % 2;
    *reinterpret_cast<uint4*>(qbuf + buf * C::Q_BYTES + sub * N * 128 + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();  // zeroed rows are read by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tmem_o = tmem + 2 * N;
  const uint32_t ring_u32 = smem_u32(ring), q_u32 = smem_u32(qbuf), p_u32 = smem_u32(pbuf);

  if (warp == 0) {
    // =================== producer: TMA, S stages ahead ===================
    // Iteration j loads K (and the unit's queries) of tile j once QK of tile j-S is
    // done, then V of tile j-1 once P.V of tile j-1-S is done.
    const int bs = 1 << p.block_shift;
    const int BH = bs < TK ? bs : TK;
    const int pieces = TK / BH;
    Cursor ld = cursor_at(f0, s_prefix, B, Hkv);
    bool fresh = true;
    int win_b = -1, win_base = 0, win_val = 0;
    int zc[TK / 16] = {}, zprev[TK / 16] = {};
    int g_prev = 0;
    for (int j = 0; j <= n_tiles; ++j) {
#pragma unroll
      for (int pc = 0; pc < TK / 16; ++pc) zprev[pc] = zc[pc];
      const int g = ld.g;
      if (j < n_tiles) {
        const int b = ld.b;
        const int ctx = s_ctx[b];
        const int t0 = ld.tile * TK;
        const int slot = ld.seq % S;
        const int s = j % S;
        bool bad = false;
#pragma unroll
        for (int pc = 0; pc < TK / 16; ++pc) {
          if (pc >= pieces) break;
          const int t = t0 + pc * BH;
          int z = -BH;
          if (t < ctx) {
            const int n = t >> p.block_shift;
            if (b != win_b || n < win_base || n >= win_base + 32) {
              win_b = b;
              win_base = n;
              const int nb = (ctx + bs - 1) >> p.block_shift;
              win_val = (n + lane < nb) ? __ldg(p.block_table + (int64_t)b * p.max_blocks + n + lane) : 0;
            }
            const int32_t phys = __shfl_sync(0xffffffffu, win_val, n - win_base);
            if (phys < 0 || (int64_t)phys >= p.num_blocks) bad = true;
            else z = (int)(((int64_t)phys << p.block_shift) + (t & (bs - 1)));
          }
          zc[pc] = z;
        }
        if (lane == 0) {
          if (j >= S && !mbar_wait_bounded(&empty_k[s], (uint32_t)(((j - S) / S) & 1)))
            raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
          if (fresh) s_bad[slot] = 0;
          if (bad) s_bad[slot] = 1;
          const uint32_t q_bytes = fresh ? (uint32_t)(R * G * D * 2) : 0u;
          mbar_arrive_expect_tx(&full_k[s], (uint32_t)C::TILE_BYTES + q_bytes);
          if (fresh) {
            const uint32_t qdst = q_u32 + slot * C::Q_BYTES;
            tma_load_3d(qdst, &tm_q, 0, g * G, b * R, &full_k[s]);
            tma_load_3d(qdst + N * 128, &tm_q, 64, g * G, b * R, &full_k[s]);
          }
          const uint32_t kdst = ring_u32 + s * C::STAGE_BYTES;
#pragma unroll
          for (int pc = 0; pc < TK / 16; ++pc) {
            if (pc >= pieces) break;
#pragma unroll
            for (int sub = 0; sub < 2; ++sub)
              tma_load_3d(kdst + sub * TK * 128 + pc * BH * 128, &tm_k, sub * 64, g, zc[pc], &full_k[s]);
          }
        }
      }
      if (j >= 1 && lane == 0) {
        const int jv = j - 1, s = jv % S;
        if (jv >= S && !mbar_wait_bounded(&empty_v[s], (uint32_t)(((jv - S) / S) & 1)))
          raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        mbar_arrive_expect_tx(&full_v[s], (uint32_t)C::TILE_BYTES);
        const uint32_t vdst = ring_u32 + s * C::STAGE_BYTES + C::TILE_BYTES;
#pragma unroll
        for (int pc = 0; pc < TK / 16; ++pc) {
          if (pc >= pieces) break;
#pragma unroll
          for (int sub = 0; sub < 2; ++sub)
            tma_load_3d(vdst + sub * TK * 128 + pc * BH * 128, &tm_v, sub * 64, g_prev, zprev[pc], &full_v[s]);
        }
      }
      __syncwarp();
      g_prev = g;
      if (j < n_tiles) {
        const int before = ld.seq;
        cursor_advance(ld, s_prefix, B, Hkv);
        fresh = ld.seq != before;
      }
    }
    return;
  }

  if (warp == 1) {
    // =================== MMA issuer (one thread) ===================
    // QK of tile i+1 is issued before P.V of tile i, so it runs while the softmax
    // warps work on tile i. Descriptors differ only in their start address, so each
    // one is a precomputed base plus the operand's address / 16.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(128, N, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(128, N, 1, 1);
      const uint64_t kmaj = smem_desc_sw128(0, 16, 1024);          // K, Q: K-major
      const uint64_t vmn = smem_desc_sw128(0, TK * 128, 1024);     // V: MN-major
      const uint64_t pmn = smem_desc(0, 16, 16 * N, C::P_LAYOUT);  // P: MN-major, 8-key groups
      Cursor cq = cursor_at(f0, s_prefix, B, Hkv);  // next tile to multiply by Q
      bool pv_fresh = true;                          // tile i starts a unit (for P.V)
      int q_seq = 0;
      auto issue_qk = [&](int i) {
        const int s = i % S;
        if (!mbar_wait_bounded(&full_k[s], (uint32_t)((i / S) & 1))) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        tc_fence_after();
        const uint32_t kb = (ring_u32 + s * C::STAGE_BYTES) >> 4;
        const uint32_t qb = (q_u32 + (q_seq % S) * C::Q_BYTES) >> 4;
        const uint32_t dst = tmem + (uint32_t)((i & 1) * N);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * TK * 128 + (ks & 3) * 32) >> 4;
          const uint32_t qoff = ((ks >> 2) * N * 128 + (ks & 3) * 32) >> 4;
          umma_bf16(dst, kmaj + kb + off, kmaj + qb + qoff, idesc_qk, ks > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[i & 1]);
        umma_commit(&empty_k[s]);  // K of the stage can be refilled
        cursor_advance(cq, s_prefix, B, Hkv);
        q_seq = cq.seq;
      };
      issue_qk(0);
      Cursor cpv = cursor_at(f0, s_prefix, B, Hkv);
      for (int i = 0; i < n_tiles; ++i) {
        if (i + 1 < n_tiles) issue_qk(i + 1);
        if (!mbar_wait_bounded(&p_full[i & 1], (uint32_t)((i >> 1) & 1))) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        if (!mbar_wait_bounded(&full_v[i % S], (uint32_t)((i / S) & 1))) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        tc_fence_after();
        const uint32_t vb = (ring_u32 + (i % S) * C::STAGE_BYTES + C::TILE_BYTES) >> 4;
        const uint32_t pb = (p_u32 + (i % NP) * 2 * C::P_BYTES) >> 4;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk) {
            const uint32_t voff = (kk * 2048) >> 4;
            const uint32_t poff = (part * C::P_BYTES + kk * 32 * N) >> 4;
            umma_bf16(tmem_o, vmn + vb + voff, pmn + pb + poff, idesc_pv,
                      (pv_fresh && part == 0 && kk == 0) ? 0u : 1u);
          }
        }
        umma_commit(&pv_done[i % NP]);  // P buffer free, O^T holds tiles <= i
        umma_commit(&empty_v[i % S]);   // V of the stage can be refilled
        if (i == n_tiles - 1) umma_commit(fin_bar);
        const int before = cpv.seq;
        cursor_advance(cpv, s_prefix, B, Hkv);
        pv_fresh = cpv.seq != before;
      }
    }
    __syncwarp();
    named_sync(kBarTail, 32 + kSoftmaxThreads);  // softmax warps are done with tensor memory
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
    return;
  }

  // =================== softmax / epilogue warps ===================
  const int sw = warp - 2;             // 0..7
  const int h = sw >> 2;               // warpgroup: rows [h*CW, h*CW + CW)
  const int c0 = h * CW;
  const int q4 = warp & 3;             // tensor-memory lane quarter of this warp
  const int gt = tid - 64 - h * 128;   // thread index inside the warpgroup
  const int st = tid - 64;             // thread index over all softmax warps
  const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
  const int key_in_tile = q4 * 32 + lane;  // the S^T lane this thread reads
  const int bar_group = kBarGroup0 + h;
  // Running row max: registers, or shared memory for 64-row tiles (register budget);
  // every thread of a warpgroup holds the same values for its rows.
  constexpr bool kMaxInSmem = CW >= 32;
  float l_part[CW], m_reg[kMaxInSmem ? 1 : CW];
#pragma unroll
  for (int e = 0; e < CW; ++e) l_part[e] = 0.f;
#pragma unroll
  for (int e = 0; e < (kMaxInSmem ? 1 : CW); ++e) m_reg[e] = -INFINITY;
  auto m_get = [&](int e) -> float { return kMaxInSmem ? s_mrun[c0 + e] : m_reg[kMaxInSmem ? 0 : e]; };
  Cursor cu = cursor_at(f0, s_prefix, B, Hkv);
  bool cu_fresh = true, from_zero = true, pending = false, fin_bad = false;
  Fin fin;
  Fin pend[2];     // pieces of split units, merged when the CTA is done
  int n_pend = 0;
  int ctx = 0, prefix_len = 0;

  // Wait until P.V of tile j (local index) is complete.
  auto wait_pv = [&](int j) {
    const uint32_t parity = (uint32_t)((NP == 2 ? (j >> 1) : j) & 1);
    if (!mbar_wait_bounded(&pv_done[j % NP], parity) && st == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
    tc_fence_after();
  };

  // Write the finished unit piece: output rows (whole unit) or a normalised partial.
  // A unit split over several CTAs is merged by the last one to finish its piece.
  auto epilogue = [&](const Fin& F) {
    {
      const float lsum = reduce_cols<CW, false>(l_part, lane);  // l_part is reset after this
      if (lane < CW) s_red[q4 * 64 + c0 + reduced_col<CW>(lane)] = lsum;
    }
    if (F.complete && gt < CW && c0 + gt < p.n_rows) {
      const int r = c0 + gt, i = r / G, j = r - i * G;
      s_rowoff[r] = (((int64_t)F.b * R + i) * p.num_q_heads + F.g * G + j) * D;
    }
    named_sync(bar_group, 128);
    const bool bad = fin_bad;
    const int d = q4 * 32 + lane;  // the O^T lane this thread reads
    constexpr int CH = CW < 16 ? CW : 16;  // columns per step
#pragma unroll
    for (int c = 0; c < CW; c += CH) {
      float inv[CH];
#pragma unroll
      for (int e = 0; e < CH; ++e) {
        const int r = c0 + c + e;
        const float L = s_red[r] + s_red[64 + r] + s_red[128 + r] + s_red[192 + r];
        inv[e] = (L > 0.f && !bad) ? 1.f / L : 0.f;
        if (!F.complete && q4 == 0 && lane == 0 && r < p.n_rows) {
          float lse2 = L > 0.f ? m_get(c + e) + __log2f(L) : -INFINITY;
          if (bad) lse2 = __int_as_float(0x7fc00000);
          __stcg(p.lse + (int64_t)F.slot * p.n_rows + r, lse2);
        }
      }
      float ov[CH];
      tmem_load_cols<CH>(tmem_o + lane_off + c0 + c, ov);
#pragma unroll
      for (int e = 0; e < CH; ++e) {
        const int r = c0 + c + e;
        if (r < p.n_rows) {
          const int64_t off = F.complete ? s_rowoff[r] : ((int64_t)F.slot * p.n_rows + r) * D;
          __stcg((F.complete ? p.out : p.opart) + off + d, ov[e] * inv[e]);
        }
      }
    }
    if (bad && st == 0) raise_error(p.dev_err, SPEC_DEVERR_BLOCK_ID);
    if (!F.complete) pend[n_pend++] = F;  // arrival and merge happen when the CTA is done
    named_sync(kBarSoftmax, kSoftmaxThreads);  // s_red and s_rowoff are reused
  };

  // A unit split over several CTAs is merged by the last CTA to arrive on its
  // counter. A CTA holds at most two such pieces (its first and its last unit);
  // it arrives for both once all its tiles are done, so no epilogue in the middle
  // of the tile stream waits for an atomic. No CTA ever waits for another.
  auto arrive_and_merge = [&]() {
    named_sync(kBarSoftmax, kSoftmaxThreads);  // every partial store of the CTA is issued
    if (st == 0) {
      __threadfence();  // release the partials
      int last[2] = {0, 0};
      for (int k = 0; k < n_pend; ++k)
        last[k] = atomicAdd(p.counters + pend[k].b * Hkv + pend[k].g, 1) == pend[k].nseg - 1;
      if (last[0] | last[1]) __threadfence();  // acquire the other pieces
      s_misc[8] = last[0];
      s_misc[9] = last[1];
    }
    named_sync(kBarSoftmax, kSoftmaxThreads);
    for (int k = 0; k < n_pend; ++k) {
      if (!s_misc[8 + k]) continue;
      const Fin& F = pend[k];
      if (st < p.n_rows) {
        const int r = st, i = r / G, j = r - i * G;
        s_rowoff[r] = (((int64_t)F.b * R + i) * p.num_q_heads + F.g * G + j) * D;
      }
      named_sync(kBarSoftmax, kSoftmaxThreads);
      // out[row] = sum_pieces 2^(lse - M) * partial / sum_pieces 2^(lse - M), merged
      // online; a thread's float4 columns load up to four pieces at a time
      for (int idx = st; idx < p.n_rows * (D / 4); idx += kSoftmaxThreads) {
        const int r = idx / (D / 4), d4 = idx - r * (D / 4);
        float M = -INFINITY, wsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        bool nan = false;
        for (int sg0 = 0; sg0 < F.nseg; sg0 += 4) {
          float l[4];
          float4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            l[u] = -INFINITY;
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (sg0 + u < F.nseg) {
              const int64_t slot = piece_slot(F.c0 + sg0 + u, F.c0, F.u0, W);
              l[u] = __ldcg(p.lse + slot * p.n_rows + r);
              v[u] = __ldcg(reinterpret_cast<const float4*>(p.opart + (slot * p.n_rows + r) * D) + d4);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            nan |= l[u] != l[u];
            if (l[u] == -INFINITY) continue;
            const float Mn = fmaxf(M, l[u]);
            const float a = exp2f(M - Mn), wgt = exp2f(l[u] - Mn);
            acc.x = acc.x * a + wgt * v[u].x;
            acc.y = acc.y * a + wgt * v[u].y;
            acc.z = acc.z * a + wgt * v[u].z;
            acc.w = acc.w * a + wgt * v[u].w;
            wsum = wsum * a + wgt;
            M = Mn;
          }
        }
        const float sc = (nan || wsum == 0.f) ? 0.f : 1.f / wsum;  // 0: invalid piece or no key seen
        const float4 o = sc == 0.f ? make_float4(0.f, 0.f, 0.f, 0.f)
                                   : make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc);
        __stcg(reinterpret_cast<float4*>(p.out + s_rowoff[r]) + d4, o);
      }
      if (st == 0) p.counters[F.b * Hkv + F.g] = 0;
      named_sync(kBarSoftmax, kSoftmaxThreads);  // s_rowoff is reused
    }
  };

  for (int i = 0; i < n_tiles; ++i) {
    const int stage = i % S;
    if (!mbar_wait_bounded(&s_full[i & 1], (uint32_t)((i >> 1) & 1)) && st == 0)
      raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
    tc_fence_after();
    if (pending) {  // the previous unit ended with tile i-1: write it out
      wait_pv(i - 1);
      epilogue(fin);
      pending = false;
    }
    if (cu_fresh) {
      from_zero = cu.tile == 0;
      ctx = s_ctx[cu.b];
      prefix_len = ctx - R;
#pragma unroll
      for (int e = 0; e < CW; ++e) l_part[e] = 0.f;
      if constexpr (kMaxInSmem) {
        if (gt < CW) s_mrun[c0 + gt] = -INFINITY;
        named_sync(bar_group, 128);
      } else {
#pragma unroll
        for (int e = 0; e < CW; ++e) m_reg[kMaxInSmem ? 0 : e] = -INFINITY;
      }
    }
    const int t0 = cu.tile * TK;
    const int tkey = t0 + key_in_tile;
    // row r sees this key iff r >= rmin (rows of draft position i see keys <= prefix_len + i)
    const int rmin = tkey >= ctx ? (1 << 30) : (tkey > prefix_len ? (tkey - prefix_len) * G : 0);
    const bool edge = t0 + TK - 1 > prefix_len;  // the tile holds keys some rows must not see
    float x[CW];
    tmem_load_cols<CW>(tmem + (uint32_t)((i & 1) * N) + lane_off + c0, x);
    bool grow = false;
#pragma unroll
    for (int e = 0; e < CW; ++e) {
      x[e] *= p.scale_log2;
      if (edge && c0 + e < rmin) x[e] = -INFINITY;
      grow |= x[e] > m_get(e) + 8.f;
    }
    if (named_sync_or(bar_group, 128, grow)) {
      // ---- slow path: exact tile max per row, rescale O^T and the row sums
      {
        float tmp[CW];
#pragma unroll
        for (int e = 0; e < CW; ++e) tmp[e] = x[e];
        const float mx = reduce_cols<CW, true>(tmp, lane);
        if (lane < CW) s_red[q4 * 64 + c0 + reduced_col<CW>(lane)] = mx;
      }
      named_sync(bar_group, 128);
      // O^T holds earlier tiles of this unit unless the unit starts here: wait for the
      // last P.V before rescaling it
      if (!cu_fresh) wait_pv(i - 1);
      constexpr int CH = CW < 16 ? CW : 16;  // columns rescaled per step
#pragma unroll
      for (int c = 0; c < CW; c += CH) {
        float alpha[CH];
#pragma unroll
        for (int e = 0; e < CH; ++e) {
          const int r = c0 + c + e;
          const float tm = fmaxf(fmaxf(s_red[r], s_red[64 + r]), fmaxf(s_red[128 + r], s_red[192 + r]));
          const float mo = m_get(c + e);
          const float mn = fmaxf(mo, tm);
          alpha[e] = mo == -INFINITY ? 0.f : fast_exp2(mo - mn);
          l_part[c + e] *= alpha[e];
          if constexpr (!kMaxInSmem) m_reg[kMaxInSmem ? 0 : c + e] = mn;
        }
        if (!cu_fresh) {
          float ov[CH];
          tmem_load_cols<CH>(tmem_o + lane_off + c0 + c, ov);
#pragma unroll
          for (int e = 0; e < CH; ++e) ov[e] *= alpha[e];
          tmem_store_cols<CH>(tmem_o + lane_off + c0 + c, ov);
        }
      }
      if constexpr (kMaxInSmem) {
        named_sync(bar_group, 128);  // every thread has read the old maxima
        if (gt < CW) {
          const int r = c0 + gt;
          const float tm = fmaxf(fmaxf(s_red[r], s_red[64 + r]), fmaxf(s_red[128 + r], s_red[192 + r]));
          s_mrun[r] = fmaxf(s_mrun[r], tm);
        }
      }
      named_sync(bar_group, 128);  // s_red is reused; new maxima visible
    }
    // ---- keys past the context in the last tile may hold stale bytes: zero those V rows
    if (t0 + TK > ctx) {
      if (!mbar_wait_bounded(&full_v[stage], (uint32_t)((i / S) & 1)) && st == 0)
        raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);  // V of this tile has landed
      const int valid = ctx - t0;
      uint8_t* vt = ring + stage * C::STAGE_BYTES + C::TILE_BYTES;
      for (int j = st; j < (TK - valid) * 16; j += kSoftmaxThreads) {
        const int row = valid + j / 16, ch = j % 16;
        *reinterpret_cast<uint4*>(vt + (ch >> 3) * TK * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4)) =
            make_uint4(0, 0, 0, 0);
      }
    }
    // ---- P = exp2(x - m), row sums
#pragma unroll
    for (int e = 0; e < CW; ++e) {
      const float m = m_get(e);
      x[e] = fast_exp2(x[e] - (m == -INFINITY ? 0.f : m));
      l_part[e] += x[e];
    }
    // the P buffer is free once the P.V that last read it is done
    if (i >= NP) wait_pv(i - NP);
    // ---- store P as bf16 hi + lo: this thread's key, rows [c0, c0 + CW), 8 rows per
    // 16-byte store, chunk index XOR-ed with the key bits of the swizzle
    uint8_t* pb = pbuf + (i % NP) * 2 * C::P_BYTES;
    {
      const int k = key_in_tile;
      const int sw = (k >> C::P_SWZ_SHIFT) & C::P_SWZ_MASK;
#pragma unroll
      for (int q = 0; q < CW / 8; ++q) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float a = x[8 * q + 2 * u], bb = x[8 * q + 2 * u + 1];
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, bb);
          const float2 hf = __bfloat1622float2(h2);
          hw[u] = *reinterpret_cast<const uint32_t*>(&h2);
          lw[u] = pack_bf16(a - hf.x, bb - hf.y);
        }
        const int c = (c0 >> 3) + q;
        const uint32_t off = (uint32_t)(k * N * 2) + ((uint32_t)(c ^ sw) << 4);
        *reinterpret_cast<uint4*>(pb + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(pb + C::P_BYTES + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    fence_proxy_async_smem();  // P and zeroed V rows are read by the tensor core
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&p_full[i & 1]);
    if (i == n_tiles - 1 || cu.tile == cu.ntiles - 1) {
      const int64_t u0 = (int64_t)s_prefix[cu.b] * Hkv + (int64_t)cu.g * cu.ntiles;
      fin.b = cu.b;
      fin.g = cu.g;
      fin.seq = cu.seq;
      fin.complete = from_zero && cu.tile == cu.ntiles - 1;
      fin.u0 = u0;
      fin.c0 = (int)(u0 / W);
      fin.nseg = (int)((u0 + cu.ntiles - 1) / W) - fin.c0 + 1;
      fin.slot = piece_slot((int)blockIdx.x, fin.c0, u0, W);
      fin_bad = s_bad[cu.seq % S] != 0;  // every tile of the unit in range is loaded by now
      pending = true;
    }
    const int before = cu.seq;
    cursor_advance(cu, s_prefix, B, Hkv);
    cu_fresh = cu.seq != before;
  }
  if (!mbar_wait_bounded(fin_bar, 0) && st == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
  tc_fence_after();
  if (pending) epilogue(fin);
  tc_fence_before();
  named_sync(kBarTail, 32 + kSoftmaxThreads);  // tensor memory may be released
  if (n_pend > 0) arrive_and_merge();
}

}  // namespace tc

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct Layout {
  size_t lse_off, opart_off, total;
};

static bool desc_ok(const spec_attn_desc* d, int k_draft) {
  if (d == nullptr) return false;
  if (d->batch < 0 || d->num_q_heads < 1 || d->num_kv_heads < 1) return false;
  if (d->num_q_heads % d->num_kv_heads != 0) return false;
  if (d->max_blocks_per_seq < 1 || d->num_blocks < 1 || k_draft < 1) return false;
  return true;
}

static bool shape_supported(const spec_attn_desc* d, int k_draft) {
  const int D = d->head_dim, bs = d->block_size;
  if (D != 64 && D != 128 && D != 256) return false;
  if (bs != 16 && bs != 32 && bs != 64 && bs != 128) return false;
  const int64_t rows = (int64_t)(k_draft + 1) * (d->num_q_heads / d->num_kv_heads);
  if (rows > 64) return false;
  if (d->batch > kMaxBatch) return false;
  if ((int64_t)d->max_blocks_per_seq * bs > INT32_MAX / 2) return false;
  if ((int64_t)d->num_blocks * bs > INT32_MAX) return false;  // TMA row coordinate is 32-bit
  if ((int64_t)d->batch * (k_draft + 1) > INT32_MAX) return false;
  return true;
}

static Layout layout_for(const spec_attn_desc* d, int k_draft) {
  Layout L;
  const int64_t n_rows = (int64_t)(k_draft + 1) * (d->num_q_heads / d->num_kv_heads);
  const int64_t slots = 2 * (int64_t)kMaxGrid;
  L.lse_off = align256((size_t)d->batch * d->num_kv_heads * 4);
  L.opart_off = L.lse_off + align256((size_t)(slots * n_rows * 4));
  L.total = L.opart_off + align256((size_t)(slots * n_rows * d->head_dim * 4));
  return L;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Resolved once per process (a function-local static is initialised exactly
// once even when several host threads arrive together).
static EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// A bf16 3-D view {x: 64-wide slice of D, y: head, z: token row} with 128-byte swizzle.
static bool make_map(CUtensorMap* map, const void* base, uint64_t D, uint64_t heads, uint64_t rows,
                     uint32_t box_heads, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {D, heads, rows};
  const cuuint64_t strides[2] = {D * 2, heads * D * 2};
  const cuuint32_t box[3] = {64, box_heads, box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int MT>
static int launch_main(const Params& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream) {
  auto kern = verify_attention_kernel<D, MT>;
  const size_t smem = smem_bytes<D, MT>(p.batch);
  static LaunchMemo memo;
  const int dev = current_device();
  if (dev < 0) return SPEC_ERR_LAUNCH;
  int grid = 0;
  {
    std::lock_guard<std::mutex> lock(memo.mu);
    if (memo.grid_smem[dev] != smem) {
      if (!grant_smem_locked(memo, (const void*)kern, dev, smem)) return SPEC_ERR_LAUNCH;
      int sms = 0, per_sm = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SPEC_ERR_LAUNCH;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess)
        return SPEC_ERR_LAUNCH;
      if (per_sm < 1) return SPEC_ERR_UNSUPPORTED;
      memo.grid[dev] = sms * per_sm > kMaxGrid ? kMaxGrid : sms * per_sm;
      memo.grid_smem[dev] = smem;
    }
    grid = memo.grid[dev];
  }
  kern<<<grid, kThreads, smem, stream>>>(p, tq, tk, tv);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

template <int D>
static int launch_main_d(const Params& p, int mt, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, cudaStream_t stream) {
  switch (mt) {
    case 1: return launch_main<D, 1>(p, tq, tk, tv, stream);
    case 2: return launch_main<D, 2>(p, tq, tk, tv, stream);
    default: return launch_main<D, 4>(p, tq, tk, tv, stream);
  }
}

// The tcgen05 kernel: one CTA per SM (its grid never exceeds the mma.sync kernel's).
template <int MT, int S, int NP>
static int launch_tc(const Params& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t stream) {
  auto kern = tc::verify_attention_tc_kernel<MT, S, NP>;
  const size_t smem = tc::smem_bytes<MT, S, NP>(p.batch);
  static LaunchMemo memo;
  const int dev = current_device();
  if (dev < 0) return SPEC_ERR_LAUNCH;
  int grid = 0;
  {
    std::lock_guard<std::mutex> lock(memo.mu);
    if (memo.grid_smem[dev] != smem) {
      if (!grant_smem_locked(memo, (const void*)kern, dev, smem)) return SPEC_ERR_LAUNCH;
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SPEC_ERR_LAUNCH;
      memo.grid[dev] = sms > kMaxGrid ? kMaxGrid : sms;
      memo.grid_smem[dev] = smem;
    }
    grid = memo.grid[dev];
  }
  kern<<<grid, tc::kThreads, smem, stream>>>(p, tq, tk, tv);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

enum class Kernel { kMma, kTc };

// Which kernel runs a call. D = 128 with 32 or more packed query rows per kv head
// takes the tcgen05 kernel (its MMAs stay wide, where mma.sync tiles become
// compute-bound), 16 rows the mma.sync kernel (at that width both are bound by
// HBM and the mma.sync kernel, two CTAs per SM, hides its per-unit work better).
// The environment variable SPEC_ATTN_KERNEL=tc or =mma overrides the choice; the
// tcgen05 kernel also needs its shared-memory plan to fit the batch. Both compute
// the same result within rounding.
static Kernel choose_kernel(int D, int mt, int batch, int* stages) {
  *stages = 0;
  if (D != 128) return Kernel::kMma;
  const char* env = getenv("SPEC_ATTN_KERNEL");
  const bool force_tc = env != nullptr && strcmp(env, "tc") == 0;
  const bool force_mma = env != nullptr && strcmp(env, "mma") == 0;
  if (force_mma || (!force_tc && mt < 2)) return Kernel::kMma;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return Kernel::kMma;
  // stages x P buffers per row count, most overlap first
  size_t need3 = SIZE_MAX, need2 = SIZE_MAX;
  switch (mt) {
    case 1: need3 = tc::smem_bytes<1, 3, 2>(batch); need2 = tc::smem_bytes<1, 2, 2>(batch); break;
    case 2: need2 = tc::smem_bytes<2, 2, 2>(batch); break;
    default: need2 = tc::smem_bytes<4, 2, 1>(batch); break;
  }
  if (need3 <= (size_t)optin) *stages = 3;
  else if (need2 <= (size_t)optin) *stages = 2;
  else return Kernel::kMma;
  return Kernel::kTc;
}

// Builds the tensor maps for the chosen kernel's key tile and launches it.
static int dispatch(const Params& p, int D, int bs, const void* q, const void* k_cache, const void* v_cache,
                    int64_t num_blocks, cudaStream_t stream) {
  const int R = p.rows_per_seq, G = p.gqa;
  const int mt = R * G <= 16 ? 1 : (R * G <= 32 ? 2 : 4);
  int stages = 0;
  const Kernel kind = choose_kernel(D, mt, p.batch, &stages);
  const int tk = kind == Kernel::kTc ? tc::TK : tile_keys(D, mt);
  CUtensorMap tq, tk_map, tv_map;
  if (!make_map(&tq, q, D, p.num_q_heads, (uint64_t)p.batch * R, (uint32_t)G, (uint32_t)R) ||
      !make_map(&tk_map, k_cache, D, p.num_kv_heads, (uint64_t)num_blocks * bs, 1, (uint32_t)(bs < tk ? bs : tk)) ||
      !make_map(&tv_map, v_cache, D, p.num_kv_heads, (uint64_t)num_blocks * bs, 1, (uint32_t)(bs < tk ? bs : tk)))
    return SPEC_ERR_LAUNCH;
  if (kind == Kernel::kTc) {
    if (mt == 1) return stages == 3 ? launch_tc<1, 3, 2>(p, tq, tk_map, tv_map, stream)
                                    : launch_tc<1, 2, 2>(p, tq, tk_map, tv_map, stream);
    if (mt == 2) return launch_tc<2, 2, 2>(p, tq, tk_map, tv_map, stream);
    return launch_tc<4, 2, 1>(p, tq, tk_map, tv_map, stream);
  }
  switch (D) {
    case 64: return launch_main_d<64>(p, mt, tq, tk_map, tv_map, stream);
    case 128: return launch_main_d<128>(p, mt, tq, tk_map, tv_map, stream);
    default: return launch_main_d<256>(p, mt, tq, tk_map, tv_map, stream);
  }
}

}  // namespace attn
}  // namespace specv

using namespace specv;

extern "C" size_t spec_verify_attention_workspace(const spec_attn_desc* d, int32_t k_draft) {
  if (!attn::desc_ok(d, k_draft)) return 0;
  return attn::layout_for(d, k_draft).total;
}

extern "C" int spec_verify_attention(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* ctx_lens, int32_t k_draft,
                                     float* out, const spec_attn_desc* d, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_err, spec_stream_t stream_) {
  if (!attn::desc_ok(d, k_draft)) return SPEC_ERR_INVALID_ARG;
  if (d->batch == 0) return SPEC_OK;
  if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !out) return SPEC_ERR_INVALID_ARG;
  if (!attn::shape_supported(d, k_draft)) return SPEC_ERR_UNSUPPORTED;
  const attn::Layout L = attn::layout_for(d, k_draft);
  if (workspace == nullptr || workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return SPEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) & 15)
    return SPEC_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  const int R = k_draft + 1, G = d->num_q_heads / d->num_kv_heads, D = d->head_dim;
  const int bs = d->block_size;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  attn::Params p;
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.out = out;
  p.counters = reinterpret_cast<int32_t*>(ws);
  p.lse = reinterpret_cast<float*>(ws + L.lse_off);
  p.opart = reinterpret_cast<float*>(ws + L.opart_off);
  p.dev_err = dev_err;
  p.num_blocks = d->num_blocks;
  p.batch = d->batch;
  p.rows_per_seq = R;
  p.num_q_heads = d->num_q_heads;
  p.num_kv_heads = d->num_kv_heads;
  p.gqa = G;
  p.n_rows = R * G;
  int shift = 0;
  while ((1 << shift) < bs) ++shift;
  p.block_shift = shift;
  p.max_blocks = d->max_blocks_per_seq;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
  return attn::dispatch(p, D, bs, q, k_cache, v_cache, d->num_blocks, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of spec_verify_attention.
//
// Some callers may not allocate device memory when they call us: a serving
// engine's per-step enqueue path that must not touch the allocator, a plugin
// hook of an inference runtime whose enqueue contract forbids allocation, or a
// process that reserved all device memory up front. This entry point takes no
// workspace: its scratch is the fixed array below, which every GPU that loads
// the library keeps until the process exits.
// ---------------------------------------------------------------------------
namespace specv {
namespace attn {

constexpr size_t kNoAllocScratchBytes = 32u << 20;  // 32 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Largest persistent grid a launch can use: the mma.sync kernel's occupancy (the
// tcgen05 kernel runs one CTA per SM, never more CTAs than this).
template <int D, int MT>
static int noalloc_grid(int batch, int* grid) {
  auto kern = verify_attention_kernel<D, MT>;
  const size_t smem = smem_bytes<D, MT>(batch);
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  if (per_sm < 1) return SPEC_ERR_UNSUPPORTED;
  *grid = sms * per_sm > kMaxGrid ? kMaxGrid : sms * per_sm;
  return SPEC_OK;
}

template <int D>
static int noalloc_grid_d(int mt, int batch, int* grid) {
  switch (mt) {
    case 1: return noalloc_grid<D, 1>(batch, grid);
    case 2: return noalloc_grid<D, 2>(batch, grid);
    default: return noalloc_grid<D, 4>(batch, grid);
  }
}

}  // namespace attn
}  // namespace specv

extern "C" size_t spec_verify_attention_noalloc_limit(void) { return attn::kNoAllocScratchBytes; }

extern "C" int spec_verify_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_table, const int32_t* ctx_lens, int32_t k_draft,
                                             float* out, const spec_attn_desc* d, int32_t* dev_err,
                                             spec_stream_t stream_) {
  if (!attn::desc_ok(d, k_draft)) return SPEC_ERR_INVALID_ARG;
  if (d->batch == 0) return SPEC_OK;
  if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !out) return SPEC_ERR_INVALID_ARG;
  if (!attn::shape_supported(d, k_draft)) return SPEC_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) & 15)
    return SPEC_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  // Set-up, once per device, with that device current: the device address of
  // the scratch array (host code cannot use the symbol itself).
  static void* scratch_addr[attn::kNoAllocMaxDevices] = {};
  static std::mutex scratch_mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= attn::kNoAllocMaxDevices) return SPEC_ERR_LAUNCH;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(scratch_mu);
    if (scratch_addr[dev] == nullptr) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, attn::g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
        return SPEC_ERR_LAUNCH;
      scratch_addr[dev] = ptr;
    }
    scratch = scratch_addr[dev];
  }

  const int R = k_draft + 1, G = d->num_q_heads / d->num_kv_heads, D = d->head_dim;
  const int bs = d->block_size;
  const int mt = R * G <= 16 ? 1 : (R * G <= 32 ? 2 : 4);
  int grid = 0, rc = SPEC_OK;
  switch (D) {
    case 64: rc = attn::noalloc_grid_d<64>(mt, d->batch, &grid); break;
    case 128: rc = attn::noalloc_grid_d<128>(mt, d->batch, &grid); break;
    default: rc = attn::noalloc_grid_d<256>(mt, d->batch, &grid); break;
  }
  if (rc != SPEC_OK) return rc;
  // Scratch layout for this grid: arrival counters, then two partial slots per CTA.
  const int64_t n_rows = (int64_t)R * G;
  const int64_t slots = 2 * (int64_t)grid;
  const size_t counters_bytes = attn::align256((size_t)d->batch * d->num_kv_heads * 4);
  const size_t lse_off = counters_bytes;
  const size_t opart_off = lse_off + attn::align256((size_t)(slots * n_rows * 4));
  const size_t total = opart_off + attn::align256((size_t)(slots * n_rows * D * 4));
  if (total > attn::kNoAllocScratchBytes) return SPEC_ERR_SCRATCH_LIMIT;

  uint8_t* ws = static_cast<uint8_t*>(scratch);
  // The counters must start at zero; every call shares the array, so clear them here.
  if (cudaMemsetAsync(ws, 0, counters_bytes, stream) != cudaSuccess) return SPEC_ERR_LAUNCH;

  attn::Params p;
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.out = out;
  p.counters = reinterpret_cast<int32_t*>(ws);
  p.lse = reinterpret_cast<float*>(ws + lse_off);
  p.opart = reinterpret_cast<float*>(ws + opart_off);
  p.dev_err = dev_err;
  p.num_blocks = d->num_blocks;
  p.batch = d->batch;
  p.rows_per_seq = R;
  p.num_q_heads = d->num_q_heads;
  p.num_kv_heads = d->num_kv_heads;
  p.gqa = G;
  p.n_rows = R * G;
  int shift = 0;
  while ((1 << shift) < bs) ++shift;
  p.block_shift = shift;
  p.max_blocks = d->max_blocks_per_seq;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
  return attn::dispatch(p, D, bs, q, k_cache, v_cache, d->num_blocks, stream);
}
