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
//  * Work item = (sequence, key chunk, kv head). A tiny plan kernel sizes the
//    key chunk from the actual context lengths (device side, no host sync) so
//    the items cover the GPU several times over; persistent CTAs pull items
//    from an atomic counter. Partial results of a split sequence are merged
//    by their log-sum-exp in a third kernel.
//  * Paged K/V tiles are staged into swizzled shared memory with 16-byte
//    cp.async copies (3-stage ring), each key looked up through the block
//    table; the block id is range-checked before any byte is read.
//  * QK^T and PV run on mma.sync m16n8k16 (bf16 in, fp32 accumulate). P is
//    split into a bf16 high part and a bf16 remainder and both are multiplied
//    with V, so PV keeps ~16 mantissa bits of P; softmax statistics and the
//    output stay fp32.
#include <math.h>

#include "common.cuh"

namespace specv {
namespace attn {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 3;
constexpr int kTargetItems = 1216;
constexpr int kMaxBatch = 4096;
constexpr int kHeaderBytes = 256;

struct WsHeader {
  int32_t chunk_tiles;
  int32_t total_splits;
  int32_t next_item;
  int32_t pad;
};

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  float* out;
  WsHeader* hdr;
  const int32_t* prefix;
  float* lse;    // [max_items][n_rows], log2 units
  float* opart;  // [max_items][n_rows][D]
  int32_t* dev_err;
  int64_t num_blocks;
  int batch, rows_per_seq, num_q_heads, num_kv_heads, gqa, n_rows;
  int block_shift, max_blocks;
  float scale_log2;
};

// Keys per pipeline stage: 64, or 32 when D = 256 and several m-tiles share the stage.
__host__ __device__ constexpr int tile_keys(int D, int MT) { return (D >= 256 && MT > 1) ? 32 : 64; }

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// Plan: chunk size and per-sequence split prefix, from the actual ctx_lens.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ ctx_lens, int batch,
                                                    int rows_per_seq, int64_t max_ctx, int tk,
                                                    int num_kv_heads, WsHeader* hdr, int32_t* prefix,
                                                    int32_t* dev_err) {
  __shared__ int64_t warp_tiles[32];
  __shared__ int32_t warp_splits[32];
  __shared__ int32_t s_chunk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (batch + blockDim.x - 1) / blockDim.x;
  const int b0 = tid * per;
  int64_t my_tiles = 0;
  for (int i = 0; i < per; ++i) {
    const int b = b0 + i;
    if (b < batch) {
      const int c = ctx_lens[b];
      const bool ok = c >= rows_per_seq && (int64_t)c <= max_ctx;
      if (!ok) raise_error(dev_err, SPEC_DEVERR_CTX_LEN);
      my_tiles += ok ? (c + tk - 1) / tk : 0;
    }
  }
  int64_t t = my_tiles;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if (lane == 0) warp_tiles[warp] = t;
  __syncthreads();
  if (tid == 0) {
    int64_t total = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += warp_tiles[w];
    const int64_t units = total * num_kv_heads;
    int64_t chunk = (units + kTargetItems - 1) / kTargetItems;
    s_chunk = (int)(chunk < 1 ? 1 : chunk);
  }
  __syncthreads();
  const int chunk = s_chunk;
  int32_t my_splits = 0;
  for (int i = 0; i < per; ++i) {
    const int b = b0 + i;
    if (b < batch) {
      const int c = ctx_lens[b];
      const bool ok = c >= rows_per_seq && (int64_t)c <= max_ctx;
      const int nt = ok ? (c + tk - 1) / tk : 0;
      my_splits += (nt + chunk - 1) / chunk;
    }
  }
  // exclusive scan of my_splits across the block
  int32_t incl = my_splits;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_splits[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    int32_t run = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      const int32_t v = warp_splits[w];
      warp_splits[w] = run;
      run += v;
    }
    hdr->chunk_tiles = chunk;
    hdr->total_splits = run;
    hdr->next_item = 0;
    prefix[batch] = run;
  }
  __syncthreads();
  int32_t run = warp_splits[warp] + incl - my_splits;
  for (int i = 0; i < per; ++i) {
    const int b = b0 + i;
    if (b < batch) {
      prefix[b] = run;
      const int c = ctx_lens[b];
      const bool ok = c >= rows_per_seq && (int64_t)c <= max_ctx;
      const int nt = ok ? (c + tk - 1) / tk : 0;
      run += (nt + chunk - 1) / chunk;
    }
  }
}

// ---------------------------------------------------------------------------
// Main kernel.
// ---------------------------------------------------------------------------
template <int D, int MT>
struct Cfg {
  static constexpr int TK = tile_keys(D, MT);           // keys per pipeline stage
  static constexpr int WN = kWarps / MT;            // warps splitting the keys of a tile
  static constexpr int KW = TK / WN;                // keys per warp per tile
  static constexpr int ROWS = 16 * MT;              // packed query rows (padded)
  static constexpr int CPK = D / 8;                 // 16-byte chunks per key row
  static constexpr int TILE_BYTES = TK * D * 2;     // one K (or V) tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int RING_BYTES = kStages * STAGE_BYTES;
  static constexpr int Q_BYTES = ROWS * D * 2;
  static constexpr int MERGE_BYTES = 64 * D * 4 + 2 * 64 * 4;  // O, m, l of every warp
  static constexpr int SCRATCH_BYTES = RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES;
  static constexpr bool Q_IN_REGS = D <= 128;
  static_assert(KW % 16 == 0, "each warp needs whole 16-key steps");
  static_assert(WN * MT == kWarps, "warp layout");
};

template <int D, int MT>
size_t smem_bytes(int batch) {
  using C = Cfg<D, MT>;
  return align256(C::SCRATCH_BYTES) + align256(C::Q_BYTES) + align256((size_t)(batch + 1) * 4) + 256;
}

// Byte offset of 16-byte chunk `ch` of row `row` in a swizzled [rows][D] bf16 tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  return (uint32_t)(row * (D * 2) + ((ch ^ (row & 7)) << 4));
}

template <int D, int MT>
__global__ void __launch_bounds__(kThreads) verify_attention_kernel(const Params p) {
  using C = Cfg<D, MT>;
  constexpr int TK = C::TK, WN = C::WN, KW = C::KW, CPK = C::CPK;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  uint8_t* qs = smem + align256(C::SCRATCH_BYTES);
  int32_t* s_prefix = reinterpret_cast<int32_t*>(qs + align256(C::Q_BYTES));
  int32_t* s_misc = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(s_prefix) +
                                               align256((size_t)(p.batch + 1) * 4));
  float* m_o = reinterpret_cast<float*>(ring);            // [64][D] after the ring is drained
  float* m_m = m_o + 64 * D;                              // [64]
  float* m_l = m_m + 64;                                  // [64]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int mt = warp / WN, wn = warp % WN;
  const int B = p.batch, Hkv = p.num_kv_heads, G = p.gqa, R = p.rows_per_seq;

  for (int i = tid; i <= B; i += kThreads) s_prefix[i] = p.prefix[i];
  const int chunk = p.hdr->chunk_tiles;
  const int n_items = p.hdr->total_splits * Hkv;
  const uint32_t ring_u32 = smem_u32(ring);
  const uint32_t q_u32 = smem_u32(qs);

  for (;;) {
    __syncthreads();  // previous item fully done with shared memory
    if (tid == 0) s_misc[0] = atomicAdd(&p.hdr->next_item, 1);
    __syncthreads();
    const int item = s_misc[0];
    if (item >= n_items) break;
    const int us = item / Hkv, g = item - us * Hkv;
    int lo = 0, hi = B;  // find b with s_prefix[b] <= us < s_prefix[b+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_prefix[mid] <= us) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int split = us - s_prefix[b];
    const int nsplit = s_prefix[b + 1] - s_prefix[b];
    const int ctx = p.ctx_lens[b];
    const int ntiles = (ctx + TK - 1) / TK;
    const int tile_begin = split * chunk;
    const int tile_end = min(ntiles, tile_begin + chunk);
    const int n_tiles_item = tile_end - tile_begin;
    const int prefix_len = ctx - R;  // committed tokens before the verify rows
    const int32_t* table = p.block_table + (int64_t)b * p.max_blocks;
    bool bad = false;

    // ---- Q tile: packed row r = i*G + j  <-  q[b, i, g*G + j, :]
    for (int c = tid; c < C::ROWS * CPK; c += kThreads) {
      const int r = c / CPK, ch = c - r * CPK;
      const bool valid = r < p.n_rows;
      const int i = valid ? r / G : 0, j = valid ? r - i * G : 0;
      const __nv_bfloat16* src = p.q + (((int64_t)b * R + i) * p.num_q_heads + g * G + j) * D + ch * 8;
      cp_async_16(q_u32 + swz<D>(r, ch), valid ? (const void*)src : (const void*)p.q, valid ? 16u : 0u);
    }

    auto load_tile = [&](int tile, int stage) {
      const int t0 = (tile_begin + tile) * TK;
      const uint32_t kdst = ring_u32 + stage * C::STAGE_BYTES;
      const uint32_t vdst = kdst + C::TILE_BYTES;
#pragma unroll 4
      for (int c = tid; c < TK * CPK; c += kThreads) {
        const int key = c / CPK, ch = c - key * CPK;
        const int t = t0 + key;
        bool valid = t < ctx;
        int64_t off = 0;
        if (valid) {
          const int32_t phys = __ldg(table + (t >> p.block_shift));
          if (phys < 0 || (int64_t)phys >= p.num_blocks) {
            bad = true;
            valid = false;
          } else {
            off = (((int64_t)phys << p.block_shift) + (t & ((1 << p.block_shift) - 1))) * Hkv + g;
            off = off * D + ch * 8;
          }
        }
        const uint32_t so = swz<D>(key, ch);
        cp_async_16(kdst + so, p.k_cache + off, valid ? 16u : 0u);
        cp_async_16(vdst + so, p.v_cache + off, valid ? 16u : 0u);
      }
    };

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
      if (s < n_tiles_item) load_tile(s, s);
      cp_async_commit();
    }

    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    uint32_t qf[C::Q_IN_REGS ? D / 16 : 1][4];

    // rows owned by this thread inside its m16 tile, and their causal limits
    const int r0 = mt * 16 + (lane >> 2), r1 = r0 + 8;
    const int lim0 = prefix_len + (r0 < p.n_rows ? r0 / G : 0);
    const int lim1 = prefix_len + (r1 < p.n_rows ? r1 / G : 0);

    for (int tile = 0; tile < n_tiles_item; ++tile) {
      cp_async_wait<kStages - 2>();
      __syncthreads();
      if (tile + kStages - 1 < n_tiles_item) load_tile(tile + kStages - 1, (tile + kStages - 1) % kStages);
      cp_async_commit();
      if (C::Q_IN_REGS && tile == 0) {
#pragma unroll
        for (int ks = 0; ks < (C::Q_IN_REGS ? D / 16 : 1); ++ks) {
          const int mi = lane >> 3;
          const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
          ldmatrix_x4(q_u32 + swz<D>(row, 2 * ks + (mi >> 1)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
        }
      }
      const int stage = tile % kStages;
      const uint32_t kbase = ring_u32 + stage * C::STAGE_BYTES;
      const uint32_t vbase = kbase + C::TILE_BYTES;
      const int t0 = (tile_begin + tile) * TK;
      const int kw0 = wn * KW;

      // ---- S = Q K^T for this warp's KW keys
      float s[KW / 8][4];
#pragma unroll
      for (int n = 0; n < KW / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4];
        if constexpr (C::Q_IN_REGS) {
          a[0] = qf[ks][0]; a[1] = qf[ks][1]; a[2] = qf[ks][2]; a[3] = qf[ks][3];
        } else {
          const int mi = lane >> 3;
          const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
          ldmatrix_x4(q_u32 + swz<D>(row, 2 * ks + (mi >> 1)), a[0], a[1], a[2], a[3]);
        }
#pragma unroll
        for (int np = 0; np < KW / 16; ++np) {
          const int mi = lane >> 3;
          const int key = kw0 + np * 16 + (mi >> 1) * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kbase + swz<D>(key, 2 * ks + (mi & 1)), b0, b1, b2, b3);
          mma_bf16_16816(s[2 * np], a, b0, b1);
          mma_bf16_16816(s[2 * np + 1], a, b2, b3);
        }
      }

      // ---- scale, causal mask, online softmax (log2 domain)
      const bool needs_mask = t0 + TK - 1 > prefix_len;
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < KW / 8; ++n) {
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
      float alpha[2], m_use[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
        tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
        const float m_new = fmaxf(m_run[h], tmax[h]);
        m_use[h] = m_new == -INFINITY ? 0.f : m_new;
        alpha[h] = fast_exp2(m_run[h] - m_use[h]);  // exp2(-inf) = 0 on the first visible tile
        m_run[h] = m_new;
        l_run[h] *= alpha[h];
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
        o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
      }
#pragma unroll
      for (int n = 0; n < KW / 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pv = fast_exp2(s[n][e] - m_use[e >> 1]);
          s[n][e] = pv;
          l_run[e >> 1] += pv;
        }
      }

      // ---- O += P V, with P = P_hi + P_lo (two bf16 products)
#pragma unroll
      for (int kk = 0; kk < KW / 16; ++kk) {
        uint32_t ah[4], al[4];
        {
          const float* p0 = s[2 * kk];
          const float* p1 = s[2 * kk + 1];
          const float src[8] = {p0[0], p0[1], p0[2], p0[3], p1[0], p1[1], p1[2], p1[3]};
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(src[2 * r], src[2 * r + 1]);
            const float2 hf = __bfloat1622float2(h2);
            ah[r] = *reinterpret_cast<const uint32_t*>(&h2);
            al[r] = pack_bf16(src[2 * r] - hf.x, src[2 * r + 1] - hf.y);
          }
        }
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int mi = lane >> 3;
          const int key = kw0 + kk * 16 + (mi & 1) * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(vbase + swz<D>(key, 2 * dp + (mi >> 1)), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * dp], ah, b0, b1);
          mma_bf16_16816(o[2 * dp], al, b0, b1);
          mma_bf16_16816(o[2 * dp + 1], ah, b2, b3);
          mma_bf16_16816(o[2 * dp + 1], al, b2, b3);
        }
      }
    }

    // ---- combine the WN key-split warps and write the item's result
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    cp_async_wait<0>();
    bad = __syncthreads_or(bad) != 0;
    {
      const int base_row = wn * C::ROWS + mt * 16 + (lane >> 2);
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const int d = n * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2*>(&m_o[base_row * D + d]) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(&m_o[(base_row + 8) * D + d]) = make_float2(o[n][2], o[n][3]);
      }
      if ((lane & 3) == 0) {
        m_m[base_row] = m_run[0];
        m_l[base_row] = l_run[0];
        m_m[base_row + 8] = m_run[1];
        m_l[base_row + 8] = l_run[1];
      }
    }
    __syncthreads();
    if (bad && tid == 0) raise_error(p.dev_err, SPEC_DEVERR_BLOCK_ID);
    const bool direct = nsplit == 1;
    for (int idx = tid; idx < p.n_rows * (D / 4); idx += kThreads) {
      const int r = idx / (D / 4), d4 = idx - r * (D / 4);
      // r lives in m-tile r/16; the WN warps of that m-tile hold partial sums
      const int rmt = r >> 4, rin = r & 15;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < WN; ++w) M = fmaxf(M, m_m[w * C::ROWS + rmt * 16 + rin]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < WN; ++w) {
        const int row = w * C::ROWS + rmt * 16 + rin;
        const float f = fast_exp2(m_m[row] - Mu);
        L += m_l[row] * f;
        const float4 v = *reinterpret_cast<const float4*>(&m_o[row * D + d4 * 4]);
        acc.x += v.x * f; acc.y += v.y * f; acc.z += v.z * f; acc.w += v.w * f;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
      if (bad) acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (direct) {
        const int i = r / G, j = r - i * G;
        float* dst = p.out + (((int64_t)b * R + i) * p.num_q_heads + g * G + j) * D + d4 * 4;
        *reinterpret_cast<float4*>(dst) = acc;
      } else {
        *reinterpret_cast<float4*>(p.opart + ((int64_t)item * p.n_rows + r) * D + d4 * 4) = acc;
        if (d4 == 0) {
          float lse2 = L > 0.f ? M + __log2f(L) : -INFINITY;
          if (bad) lse2 = __int_as_float(0x7fc00000);  // NaN marks an unusable partial
          p.lse[(int64_t)item * p.n_rows + r] = lse2;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Merge of split partials by log-sum-exp; zero rows for unusable sequences.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) merge_kernel(const Params p, int D) {
  const int Hkv = p.num_kv_heads, G = p.gqa, R = p.rows_per_seq;
  const int b = blockIdx.x / Hkv, g = blockIdx.x - b * Hkv;
  const int first = p.prefix[b];
  const int nsplit = p.prefix[b + 1] - first;
  if (nsplit == 1) return;  // written directly by the main kernel
  const int d4n = D / 4;
  for (int idx = threadIdx.x; idx < p.n_rows * d4n; idx += blockDim.x) {
    const int r = idx / d4n, d4 = idx - r * d4n;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nsplit > 1) {
      float M = -INFINITY;
      bool bad = false;
      for (int s = 0; s < nsplit; ++s) {
        const float l = p.lse[((int64_t)(first + s) * Hkv + g) * p.n_rows + r];
        bad |= l != l;
        M = fmaxf(M, l);
      }
      if (!bad && M != -INFINITY) {
        float W = 0.f;
        for (int s = 0; s < nsplit; ++s) {
          const int64_t it = (int64_t)(first + s) * Hkv + g;
          const float f = exp2f(p.lse[it * p.n_rows + r] - M);
          if (f > 0.f) {
            const float4 v = *reinterpret_cast<const float4*>(p.opart + (it * p.n_rows + r) * D + d4 * 4);
            acc.x += f * v.x; acc.y += f * v.y; acc.z += f * v.z; acc.w += f * v.w;
          }
          W += f;
        }
        const float inv = 1.f / W;
        acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
      }
    }
    const int i = r / G, j = r - i * G;
    *reinterpret_cast<float4*>(p.out + (((int64_t)b * R + i) * p.num_q_heads + g * G + j) * D + d4 * 4) = acc;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct Layout {
  size_t prefix_off, lse_off, opart_off, total;
  int64_t max_items;
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
  return true;
}

static Layout layout_for(const spec_attn_desc* d, int k_draft) {
  Layout L;
  const int64_t n_rows = (int64_t)(k_draft + 1) * (d->num_q_heads / d->num_kv_heads);
  L.max_items = kTargetItems + (int64_t)d->num_kv_heads * d->batch;
  L.prefix_off = kHeaderBytes;
  L.lse_off = L.prefix_off + align256((size_t)(d->batch + 1) * 4);
  L.opart_off = L.lse_off + align256((size_t)(L.max_items * n_rows * 4));
  L.total = L.opart_off + align256((size_t)(L.max_items * n_rows * d->head_dim * 4));
  return L;
}

template <int D, int MT>
static int launch_main(const Params& p, int batch, cudaStream_t stream) {
  auto kern = verify_attention_kernel<D, MT>;
  const size_t smem = smem_bytes<D, MT>(batch);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  if (per_sm < 1) return SPEC_ERR_UNSUPPORTED;
  kern<<<sms * per_sm, kThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

template <int D>
static int launch_main_d(const Params& p, int mt, int batch, cudaStream_t stream) {
  switch (mt) {
    case 1: return launch_main<D, 1>(p, batch, stream);
    case 2: return launch_main<D, 2>(p, batch, stream);
    default: return launch_main<D, 4>(p, batch, stream);
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

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  attn::Params p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  p.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.out = out;
  p.hdr = reinterpret_cast<attn::WsHeader*>(ws);
  p.prefix = reinterpret_cast<const int32_t*>(ws + L.prefix_off);
  p.lse = reinterpret_cast<float*>(ws + L.lse_off);
  p.opart = reinterpret_cast<float*>(ws + L.opart_off);
  p.dev_err = dev_err;
  p.num_blocks = d->num_blocks;
  p.batch = d->batch;
  p.rows_per_seq = k_draft + 1;
  p.num_q_heads = d->num_q_heads;
  p.num_kv_heads = d->num_kv_heads;
  p.gqa = d->num_q_heads / d->num_kv_heads;
  p.n_rows = p.rows_per_seq * p.gqa;
  int shift = 0;
  while ((1 << shift) < d->block_size) ++shift;
  p.block_shift = shift;
  p.max_blocks = d->max_blocks_per_seq;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d->head_dim));

  const int D = d->head_dim;
  const int mt = p.n_rows <= 16 ? 1 : (p.n_rows <= 32 ? 2 : 4);
  const int tk = attn::tile_keys(D, mt);
  const int64_t max_ctx = (int64_t)d->max_blocks_per_seq * d->block_size;

  attn::plan_kernel<<<1, 1024, 0, stream>>>(ctx_lens, d->batch, p.rows_per_seq, max_ctx, tk, d->num_kv_heads,
                                            p.hdr, reinterpret_cast<int32_t*>(ws + L.prefix_off), dev_err);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_LAUNCH;
  int rc;
  switch (D) {
    case 64: rc = attn::launch_main_d<64>(p, mt, d->batch, stream); break;
    case 128: rc = attn::launch_main_d<128>(p, mt, d->batch, stream); break;
    default: rc = attn::launch_main_d<256>(p, mt, d->batch, stream); break;
  }
  if (rc != SPEC_OK) return rc;
  attn::merge_kernel<<<d->batch * d->num_kv_heads, 256, 0, stream>>>(p, D);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}
