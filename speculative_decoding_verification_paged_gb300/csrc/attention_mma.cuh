// The mma.sync verify-attention kernel (any supported head dim and row
// count); its design is described at the top of attention.cu.
#pragma once

#include "attention_device.cuh"

namespace specv {
namespace attn {

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
    const uint64_t kv_pol = l2_evict_first_policy();  // K and V are read once
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
            tma_load_3d_hint(kdst + off, &tm_k, sub * 64, g, zc[pc], &full[s], kv_pol);
            tma_load_3d_hint(vdst + off, &tm_v, sub * 64, g, zc[pc], &full[s], kv_pol);
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

}  // namespace attn
}  // namespace specv
