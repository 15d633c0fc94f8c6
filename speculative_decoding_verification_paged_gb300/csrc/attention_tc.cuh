// Tensor-core (tcgen05) kernel for D = 128 and D = 256.
//
// The keys are the MMA's M dimension (128 per tile) and the packed query rows
// are N (16, 32 or 64), so every M = 128 MMA is fully used for any row count:
//   S^T[128 keys x N] = K[128 x D] . Q^T              (K, Q K-major in smem)
//   O^T[D x N]       += V^T[D x 128 keys] . P^T       (V and P MN-major)
// with S^T (two buffers) and O^T in tensor memory; for D = 256, O^T is two
// halves of 128 lanes (dims 0-127 and 128-255), each the accumulator of its
// own M = 128 P.V MMA, at consecutive column blocks. Warp 0 stages K/V/Q with
// TMA, warp 1 issues the MMAs (one thread; QK of tile i+1 before P.V of tile
// i), the other warps run the softmax in two warpgroups or, for 64 rows at
// D = 128 and 32 rows at D = 256, four, each owning an equal share of the
// rows; a warp reads the 32-lane quarter of tensor memory that its index
// selects, i.e. 32 keys of S^T and 32 dims of O^T. P is written to shared
// memory as a bf16 high part and a bf16 remainder and both are multiplied with
// V. The running row max may lag by up to 8 (log2 units); a tile that exceeds
// it takes the slow path: exact row max, and the accumulated O^T and row sums
// are rescaled in place.
#pragma once

#include "attention_device.cuh"

namespace specv {
namespace attn {
namespace tc {

constexpr int TK = 128;                      // keys per tile (MMA M)
constexpr int kBarSoftmax = 4;               // named barriers: all softmax warps,
constexpr int kBarTail = 5;                  // MMA warp + softmax warps,
constexpr int kBarGroup0 = 6;                // one per softmax warpgroup
constexpr int kMaxGrid = 160;                // one CTA per SM, at most; a split unit has at most this many pieces
constexpr int kTmemCols = 256;               // S^T buffers at columns 0 and N, O^T halves from 2N

template <int D, int MT>
struct Cfg {
  static constexpr int N = 16 * MT;                     // packed query rows (MMA N)
  // Softmax warpgroups: each owns N / NG rows of every tile. Four where they were
  // measured faster (D = 128 with 64 rows, D = 256 with 32): 16 softmax warps hide
  // the tensor-memory, exponential and shared-memory latency of a tile better than
  // 8 holding twice the rows each. Elsewhere the 96-register cap of 18 warps
  // spills, and two warpgroups stay.
  static constexpr int NG = (D == 128 && MT == 4) || (D == 256 && MT == 2) ? 4 : 2;
  static constexpr int CW = N / NG;                     // rows (tensor-memory columns) per warpgroup
  static constexpr int kSoftmaxWarps = 4 * NG;
  static constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
  static constexpr int kThreads = 64 + kSoftmaxThreads;  // producer warp, MMA warp, softmax warps
  // Register budget: registers are split over the four SM sub-partitions (16K each),
  // and 10 warps put up to three on one (168 registers a thread), 18 warps up to five
  // (96); declaring 384 or 576 threads caps ptxas there.
  static constexpr int kRegBudgetThreads = NG == 2 ? 384 : 576;
  static_assert(CW % 8 == 0, "a softmax thread stores its rows of P 8 at a time");
  static constexpr int SUBS = D / 64;                   // 128-byte-wide column slices
  static constexpr int HALVES = D / 128;                // O^T halves of 128 lanes
  static constexpr int TILE_BYTES = TK * D * 2;         // SUBS [128][64] slices: 32 KB (D = 128), 64 KB
  static constexpr int Q_BYTES = N * D * 2;             // SUBS [N][64] slices
  static constexpr int P_BYTES = N * TK * 2;            // one of P_hi / P_lo: [128 keys][N rows]
  // P is the P.V operand B in MN-major layout: the N rows of a key are contiguous
  // (N * 2 bytes) and swizzled at that width (32, 64 or 128 bytes), so a softmax
  // thread, which owns one key, writes its rows with 16-byte stores.
  static constexpr uint32_t P_LAYOUT = N == 16 ? 6u : (N == 32 ? 4u : 2u);
  static constexpr int P_SWZ_SHIFT = N == 16 ? 2 : (N == 32 ? 1 : 0);  // key bits that pick the XOR
  static constexpr int P_SWZ_MASK = N == 16 ? 1 : (N == 32 ? 3 : 7);
  static_assert(2 * N + HALVES * N <= kTmemCols, "S^T buffers and O^T fit the allocated columns");
};

// Dynamic shared memory: S K tiles, SV V tiles, SQ query buffers, NP P buffers
// (hi + lo), barriers, reductions, output row offsets, and the per-sequence plan
// (which grows with the batch).
template <int D, int MT, int S, int NP, int SV = S, int SQ = S>
size_t smem_bytes(int batch) {
  using C = Cfg<D, MT>;
  return 1024 + (size_t)(S + SV) * C::TILE_BYTES + (size_t)SQ * C::Q_BYTES + (size_t)NP * 2 * C::P_BYTES + 64 * 8 + 4 * 64 * 4 +
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

// S K stages, SV V stages and SQ query buffers (1, or at least S). K and V are
// released separately, so the rings may differ in depth: a K tile is refilled
// once its QK is done, a V tile once its P.V is done.
template <int D, int MT, int S, int NP, int SV = S, int SQ = S>
__global__ void __launch_bounds__(Cfg<D, MT>::kRegBudgetThreads, 1) verify_attention_tc_kernel(
    const Params p, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v) {
  using C = Cfg<D, MT>;
  constexpr int N = C::N, CW = C::CW;
  constexpr int kSoftmaxWarps = C::kSoftmaxWarps, kSoftmaxThreads = C::kSoftmaxThreads, kThreads = C::kThreads;
  static_assert(SQ == 1 || SQ >= S, "a query buffer is reused only after the K stage that covers it");
  static_assert(2 * S + 2 * SV + 2 + 2 + NP + 2 <= 64, "barriers fit their area");
  // ring, query buffers and P buffers: contiguous, idle when split units are merged
  constexpr uint32_t kMergeArea = (uint32_t)((S + SV) * C::TILE_BYTES + SQ * C::Q_BYTES + NP * 2 * C::P_BYTES);
  static_assert(kMergeArea >= 2 * N * D * 4 + 512 + kMaxGrid * N * 4 + 16, "the merge holds its rows, the weights and one piece");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;                                // S K tiles, then SV V tiles
  uint8_t* qbuf = ring + (S + SV) * C::TILE_BYTES;
  uint8_t* pbuf = qbuf + SQ * C::Q_BYTES;  // NP x (P_hi, P_lo)
  // K and V of a stage arrive and are released separately: K is free once QK is
  // done, a tile earlier than V, so the producer can fetch the next K sooner.
  uint64_t* full_k = reinterpret_cast<uint64_t*>(pbuf + NP * 2 * C::P_BYTES);
  uint64_t* full_v = full_k + S;
  uint64_t* empty_k = full_v + SV;
  uint64_t* empty_v = empty_k + S;
  uint64_t* s_full = empty_v + SV;  // [2]: S^T buffer b holds QK of the tile
  uint64_t* p_full = s_full + 2;  // [2]: P of tile i written (one arrival per softmax warp)
  uint64_t* pv_done = p_full + 2; // [NP]: P.V of the tile that used P buffer j is complete
  uint64_t* fin_bar = pv_done + NP;
  uint64_t* merge_bar = fin_bar + 1;  // pieces of a split unit landed (merge)
  float* s_red = reinterpret_cast<float*>(full_k + 64);   // [4][64] per-quarter row reductions
  float* s_mrun = s_red + 4 * 64;                         // [64] running row max (64-row tiles)
  int64_t* s_rowoff = reinterpret_cast<int64_t*>(s_mrun + 64);  // [64] output offset of each row
  int32_t* s_bad = reinterpret_cast<int32_t*>(s_rowoff + 64);  // [8] per unit (seq & 7): a block id was bad
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_bad + 8);   // tensor-memory base
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
    static_assert(kThreads / 32 <= 30, "per-warp scan slots stay below the tile-count slots");
    if (tid == 0) {
      s_misc[30] = INT32_MAX;
      s_misc[31] = 0;
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
      atomicMin(&s_misc[30], nt_min);
      atomicMax(&s_misc[31], nt_max);
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
        mbar_init(&empty_k[s], 1);
      }
      for (int s = 0; s < SV; ++s) {
        mbar_init(&full_v[s], 1);
        mbar_init(&empty_v[s], 1);
      }
      for (int j = 0; j < 2; ++j) {
        mbar_init(&s_full[j], 1);
        mbar_init(&p_full[j], kSoftmaxWarps);
      }
      for (int j = 0; j < NP; ++j) mbar_init(&pv_done[j], 1);
      mbar_init(fin_bar, 1);
      mbar_init(merge_bar, 1);
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
  const int unit_tiles = s_misc[30] == s_misc[31] ? s_misc[31] : 0;  // 0: units of several lengths
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
  for (int i = tid; i < SQ * C::SUBS * (N - p.n_rows) * 8; i += kThreads) {
    const int ch = i % 8, rest = i / 8;
    const int r = p.n_rows + rest % (N - p.n_rows);
    const int bsub = rest / (N - p.n_rows);
    const int buf = bsub / C::SUBS, sub = bsub % C::SUBS;
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
    // K and V are read once: evict them first, so that the code of the unit-boundary
    // and final paths, the block table and the queries stay in L2
    const uint64_t kv_pol = l2_evict_first_policy();
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
        const int slot = ld.seq % SQ;
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
          // one query buffer: the previous unit's last QK (tile j - 1) must be done
          // before this unit's queries overwrite it
          if (SQ == 1 && S > 1 && fresh && j >= 1 &&
              !mbar_wait_bounded(&empty_k[(j - 1) % S], (uint32_t)(((j - 1) / S) & 1)))
            raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
          if (fresh) s_bad[ld.seq & 7] = 0;
          if (bad) s_bad[ld.seq & 7] = 1;
          const uint32_t q_bytes = fresh ? (uint32_t)(R * G * D * 2) : 0u;
          mbar_arrive_expect_tx(&full_k[s], (uint32_t)C::TILE_BYTES + q_bytes);
          if (fresh) {
            const uint32_t qdst = q_u32 + slot * C::Q_BYTES;
#pragma unroll
            for (int sub = 0; sub < C::SUBS; ++sub)
              tma_load_3d(qdst + sub * N * 128, &tm_q, sub * 64, g * G, b * R, &full_k[s]);
          }
          const uint32_t kdst = ring_u32 + s * C::TILE_BYTES;
#pragma unroll
          for (int pc = 0; pc < TK / 16; ++pc) {
            if (pc >= pieces) break;
#pragma unroll
            for (int sub = 0; sub < C::SUBS; ++sub)
              tma_load_3d_hint(kdst + sub * TK * 128 + pc * BH * 128, &tm_k, sub * 64, g, zc[pc], &full_k[s], kv_pol);
          }
        }
      }
      if (j >= 1 && lane == 0) {
        const int jv = j - 1, s = jv % SV;
        if (jv >= SV && !mbar_wait_bounded(&empty_v[s], (uint32_t)(((jv - SV) / SV) & 1)))
          raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        mbar_arrive_expect_tx(&full_v[s], (uint32_t)C::TILE_BYTES);
        const uint32_t vdst = ring_u32 + (S + s) * C::TILE_BYTES;
#pragma unroll
        for (int pc = 0; pc < TK / 16; ++pc) {
          if (pc >= pieces) break;
#pragma unroll
          for (int sub = 0; sub < C::SUBS; ++sub)
            tma_load_3d_hint(vdst + sub * TK * 128 + pc * BH * 128, &tm_v, sub * 64, g_prev, zprev[pc], &full_v[s],
                           kv_pol);
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
        const uint32_t kb = (ring_u32 + s * C::TILE_BYTES) >> 4;
        const uint32_t qb = (q_u32 + (q_seq % SQ) * C::Q_BYTES) >> 4;
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
        if (!mbar_wait_bounded(&full_v[i % SV], (uint32_t)((i / SV) & 1))) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        tc_fence_after();
        const uint32_t vb = (ring_u32 + (S + i % SV) * C::TILE_BYTES) >> 4;
        const uint32_t pb = (p_u32 + (i % NP) * 2 * C::P_BYTES) >> 4;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk) {
            const uint32_t poff = (part * C::P_BYTES + kk * 32 * N) >> 4;
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h) {  // dims [128h, 128h + 128): V slices 2h, 2h + 1
              const uint32_t voff = (h * 2 * TK * 128 + kk * 2048) >> 4;
              umma_bf16(tmem_o + (uint32_t)(h * N), vmn + vb + voff, pmn + pb + poff, idesc_pv,
                        (pv_fresh && part == 0 && kk == 0) ? 0u : 1u);
            }
          }
        }
        umma_commit(&pv_done[i % NP]);  // P buffer free, O^T holds tiles <= i
        umma_commit(&empty_v[i % SV]);  // V of the stage can be refilled
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
  const int sw = warp - 2;             // 0 .. kSoftmaxWarps - 1
  const int h = sw >> 2;               // warpgroup: rows [h*CW, h*CW + CW)
  const int c0 = h * CW;
  const int q4 = warp & 3;             // tensor-memory lane quarter of this warp
  const int gt = tid - 64 - h * 128;   // thread index inside the warpgroup
  const int st = tid - 64;             // thread index over all softmax warps
  const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
  const int key_in_tile = q4 * 32 + lane;  // the S^T lane this thread reads
  const int bar_group = kBarGroup0 + h;
  // Running row max: registers, or shared memory for 16 rows a thread under the
  // 96-register cap and 32 under the 168-register one (register budget);
  // every thread of a warpgroup holds the same values for its rows.
  constexpr bool kMaxInSmem = CW >= (C::NG == 4 ? 16 : 32);
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
  int merge_phase = 0;
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
  // Where the rows fit the P buffers (free here: every P.V is done), they are
  // staged there and written by bulk copies that one thread issues, so no
  // softmax thread waits on thousands of scattered stores.
  constexpr bool kStage = D <= NP * TK;  // N rows x D fp32 fit NP x (P_hi, P_lo)
  float* s_inv = reinterpret_cast<float*>(s_rowoff);  // [64] 1 / row sum (staged form)
  auto epilogue = [&](const Fin& F) {
    {
      const float lsum = reduce_cols<CW, false>(l_part, lane);  // l_part is reset after this
      if (lane < CW) s_red[q4 * 64 + c0 + reduced_col<CW>(lane)] = lsum;
    }
    if (!kStage && F.complete && gt < CW && c0 + gt < p.n_rows) {
      const int r = c0 + gt, i = r / G, j = r - i * G;
      s_rowoff[r] = (((int64_t)F.b * R + i) * p.num_q_heads + F.g * G + j) * D;
    }
    named_sync(bar_group, 128);
    const bool bad = fin_bad;
    const int d = q4 * 32 + lane;  // the O^T lane this thread reads (in each half)
    constexpr int CH = CW < 16 ? CW : 16;  // columns per step
    if constexpr (kStage) {
      // one thread per row: 1 / L into shared memory, and the piece's log-sum-exp
      if (gt < CW) {
        const int r = c0 + gt;
        const float L = s_red[r] + s_red[64 + r] + s_red[128 + r] + s_red[192 + r];
        s_inv[r] = (L > 0.f && !bad) ? 1.f / L : 0.f;
        if (!F.complete && r < p.n_rows) {
          float m = 0.f;
          if constexpr (kMaxInSmem) {
            m = s_mrun[r];
          } else {
#pragma unroll
            for (int e = 0; e < CW; ++e)
              if (e == gt) m = m_reg[kMaxInSmem ? 0 : e];
          }
          float lse2 = L > 0.f ? m + __log2f(L) : -INFINITY;
          if (bad) lse2 = __int_as_float(0x7fc00000);
          __stcg(p.lse + (int64_t)F.slot * p.n_rows + r, lse2);
        }
      }
      named_sync(bar_group, 128);
      float* stage = reinterpret_cast<float*>(pbuf);  // [n_rows][D]
#pragma unroll
      for (int c = 0; c < CW; c += CH) {
#pragma unroll
        for (int hh = 0; hh < C::HALVES; ++hh) {
          float ov[CH];
          tmem_load_cols<CH>(tmem_o + (uint32_t)(hh * N) + lane_off + c0 + c, ov);
#pragma unroll
          for (int e = 0; e < CH; ++e) {
            const int r = c0 + c + e;
            if (r < p.n_rows) stage[r * D + hh * 128 + d] = ov[e] * s_inv[r];
          }
        }
      }
      fence_proxy_async_smem();  // the staged rows are read by the bulk copies
      named_sync(kBarSoftmax, kSoftmaxThreads);
      if (st == 0) {
        const uint32_t src = smem_u32(stage);
        if (F.complete) {
          // rows i*G .. i*G + G - 1 are the G query heads of position i: contiguous in out
          for (int i = 0; i < R; ++i)
            bulk_s2g(p.out + (((int64_t)F.b * R + i) * p.num_q_heads + F.g * G) * D,
                     src + (uint32_t)(i * G * D * 4), (uint32_t)(G * D * 4));
        } else {
          bulk_s2g(p.opart + (int64_t)F.slot * p.n_rows * D, src, (uint32_t)(p.n_rows * D * 4));
        }
        bulk_commit();
        bulk_wait_read();  // the P buffers are written again after the barrier below
      }
    } else {
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
#pragma unroll
        for (int hh = 0; hh < C::HALVES; ++hh) {
          float ov[CH];
          tmem_load_cols<CH>(tmem_o + (uint32_t)(hh * N) + lane_off + c0 + c, ov);
#pragma unroll
          for (int e = 0; e < CH; ++e) {
            const int r = c0 + c + e;
            if (r < p.n_rows) {
              const int64_t off = F.complete ? s_rowoff[r] : ((int64_t)F.slot * p.n_rows + r) * D;
              __stcg((F.complete ? p.out : p.opart) + off + hh * 128 + d, ov[e] * inv[e]);
            }
          }
        }
      }
    }
    if (bad && st == 0) raise_error(p.dev_err, SPEC_DEVERR_BLOCK_ID);
    if (!F.complete) pend[n_pend++] = F;  // arrival and merge happen when the CTA is done
    named_sync(kBarSoftmax, kSoftmaxThreads);  // s_red, s_inv, s_rowoff and the P buffers are reused
  };

  // A unit split over several CTAs is merged by the last CTA to arrive on its
  // counter. A CTA holds at most two such pieces (its first and its last unit);
  // it arrives for both once all its tiles are done, so no epilogue in the middle
  // of the tile stream waits for an atomic. No CTA ever waits for another.
  auto arrive_and_merge = [&]() {
    named_sync(kBarSoftmax, kSoftmaxThreads);  // every partial store of the CTA is issued
    if (st == 0) {
      if constexpr (kStage) {
        bulk_wait_all();             // the staged partials are written
        fence_proxy_async_global();  // ... before the release below
      }
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
      // out[row] = sum_pieces w_p[row] * partial_p[row], w_p = 2^(lse_p - M) / sum 2^(lse - M).
      // The K/V ring, query and P buffers are idle now and form one contiguous area:
      // [out rows][row max, 1/sum][lse, then weights, of every piece][a chunk of pieces].
      // Pieces arrive by bulk copies, a chunk at a time (the first while the weights
      // are worked out), and the merged rows leave the same way.
      const int nr = p.n_rows, nseg = F.nseg;
      const uint32_t piece_bytes = (uint32_t)(nr * D * 4);
      float* ostage = reinterpret_cast<float*>(ring);
      float* rmax = ostage + nr * D;
      float* rinv = rmax + 64;
      float* wts = rinv + 64;  // [nseg][nr]
      const uint32_t head = piece_bytes + 512 + (((uint32_t)(nseg * nr * 4) + 15u) & ~15u);
      const int cap = (int)((kMergeArea - head) / piece_bytes);  // >= 1: nseg <= grid <= kMaxGrid
      uint8_t* pieces = reinterpret_cast<uint8_t*>(ring) + head;
      auto load_chunk = [&](int p0) {  // one thread
        const int np_ = min(cap, nseg - p0);
        mbar_arrive_expect_tx(merge_bar, (uint32_t)np_ * piece_bytes);
        for (int q = 0; q < np_; ++q)
          bulk_g2s(smem_u32(pieces + q * piece_bytes),
                   p.opart + (int64_t)piece_slot(F.c0 + p0 + q, F.c0, F.u0, W) * nr * D, piece_bytes, merge_bar);
      };
      if (st == 0) {
        bulk_wait_read();            // the previous merge's rows have left the area
        fence_proxy_async_global();  // the acquired pieces are read by the async proxy
        load_chunk(0);
      }
      for (int t = st; t < nseg * nr; t += kSoftmaxThreads) {
        const int q = t / nr, r = t - q * nr;
        wts[t] = __ldcg(p.lse + (int64_t)piece_slot(F.c0 + q, F.c0, F.u0, W) * nr + r);
      }
      named_sync(kBarSoftmax, kSoftmaxThreads);
      if (st < nr) {  // one thread per row: max and sum of 2^lse over the pieces
        const int r = st;
        float M = -INFINITY, ws = 0.f;
        bool nan = false;
        for (int q = 0; q < nseg; ++q) {
          const float lv = wts[q * nr + r];
          nan |= lv != lv;
          if (!(lv > -INFINITY)) continue;
          const float Mn = fmaxf(M, lv);
          ws = ws * exp2f(M - Mn) + exp2f(lv - Mn);
          M = Mn;
        }
        rmax[r] = M;
        rinv[r] = (nan || ws == 0.f) ? 0.f : 1.f / ws;  // 0: invalid piece or no key seen
      }
      named_sync(kBarSoftmax, kSoftmaxThreads);
      for (int t = st; t < nseg * nr; t += kSoftmaxThreads) {
        const int r = t % nr;
        const float lv = wts[t];
        wts[t] = (rinv[r] == 0.f || !(lv > -INFINITY)) ? 0.f : exp2f(lv - rmax[r]) * rinv[r];
      }
      named_sync(kBarSoftmax, kSoftmaxThreads);  // weights are visible
      for (int p0 = 0; p0 < nseg; p0 += cap) {
        const int np_ = min(cap, nseg - p0);
        if (p0 > 0 && st == 0) load_chunk(p0);
        if (!mbar_wait_bounded(merge_bar, (uint32_t)(merge_phase & 1)) && st == 0)
          raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        ++merge_phase;
        for (int idx = st; idx < nr * (D / 4); idx += kSoftmaxThreads) {
          const int r = idx / (D / 4);
          float4 a = p0 == 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : reinterpret_cast<const float4*>(ostage)[idx];
          for (int q = 0; q < np_; ++q) {
            const float w = wts[(p0 + q) * nr + r];
            if (w == 0.f) continue;  // an invalid piece, or one that saw no key of the row
            const float4 v = reinterpret_cast<const float4*>(pieces + q * piece_bytes)[idx];
            a.x += w * v.x;
            a.y += w * v.y;
            a.z += w * v.z;
            a.w += w * v.w;
          }
          reinterpret_cast<float4*>(ostage)[idx] = a;
        }
        named_sync(kBarSoftmax, kSoftmaxThreads);  // the chunk is consumed
      }
      fence_proxy_async_smem();  // the merged rows are read by the bulk copies
      named_sync(kBarSoftmax, kSoftmaxThreads);
      if (st == 0) {
        p.counters[F.b * Hkv + F.g] = 0;
        // rows i*G .. i*G + G - 1 are the G query heads of position i: contiguous in out
        for (int i = 0; i < R; ++i)
          bulk_s2g(p.out + (((int64_t)F.b * R + i) * p.num_q_heads + F.g * G) * D,
                   smem_u32(ostage) + (uint32_t)(i * G * D * 4), (uint32_t)(G * D * 4));
        bulk_commit();
      }
    }
  };

  for (int i = 0; i < n_tiles; ++i) {
    const int vstage = i % SV;
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
#pragma unroll
          for (int h = 0; h < C::HALVES; ++h) {
            float ov[CH];
            tmem_load_cols<CH>(tmem_o + (uint32_t)(h * N) + lane_off + c0 + c, ov);
#pragma unroll
            for (int e = 0; e < CH; ++e) ov[e] *= alpha[e];
            tmem_store_cols<CH>(tmem_o + (uint32_t)(h * N) + lane_off + c0 + c, ov);
          }
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
      // With one V stage the previous tile's V may still be in flight here, and the
      // V barrier's parity would then name an earlier phase: wait until the
      // previous tile's P.V is done (its V landed and consumed) before asking for
      // this tile's V. With two or more V stages the V of tile i - SV has landed
      // before QK of tile i is issued, so the parity is already unambiguous.
      if constexpr (SV == 1) {
        if (i > 0) wait_pv(i - 1);
      }
      if (!mbar_wait_bounded(&full_v[vstage], (uint32_t)((i / SV) & 1)) && st == 0)
        raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);  // V of this tile has landed
      const int valid = ctx - t0;
      uint8_t* vt = ring + (S + vstage) * C::TILE_BYTES;
      for (int j = st; j < (TK - valid) * (D / 8); j += kSoftmaxThreads) {
        const int row = valid + j / (D / 8), ch = j % (D / 8);
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
      fin_bad = s_bad[cu.seq & 7] != 0;  // every tile of the unit in range is loaded by now
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
  if (st == 0) bulk_wait_all();  // staged rows are written before the CTA exits
}

}  // namespace tc
}  // namespace attn
}  // namespace specv
