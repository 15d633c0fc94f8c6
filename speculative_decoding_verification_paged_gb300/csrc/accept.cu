// Acceptance of a chain draft: greedy prefix match or speculative sampling
// (sm_103a).
//
// Greedy speculation must reproduce greedy decoding token for token
// (onnxruntime-genai PR #2457, Qwen3.8-27B-NVFP4 validation); the sampling
// rule is speculative sampling ("speculative sampling" suite of lmdeploy PR
// #5019; reject_sampler.py of lmdeploy PR #3945): draft d_j is kept when
// u_j * q_j(d_j) < p_j(d_j), the first rejected position m draws from
// max(0, p_m - q_m), and a fully accepted chain draws a bonus token from p_k.
// The emitted row is the accepted drafts, one final token and -1 padding, as
// in the reject sampler's expected output of lmdeploy PR #3945.
//
// Design (GB300): one thread-block cluster per batch row, its CTAs splitting
// the vocabulary into contiguous slices of whole 8192-logit groups (one to
// six groups per CTA; at most 16 CTAs, 8 where the device cannot schedule a
// 16-CTA cluster).
// Positions are processed in order and the row stops at the first rejection,
// so logits past it are never read (early exit). For each position every CTA
// pulls its slice into shared memory with one bulk asynchronous copy (TMA,
// mbarrier completion; position 0's copy is issued first thing, before the row
// is validated), prefetches into L2 what comes next once the slice has landed
// (the next position, and the draft probabilities a rejection would read),
// reduces it (max / sum of exp / argmax) with warp shuffles, and publishes a
// partial that every CTA of the cluster reads through distributed shared
// memory, in rank order, so all CTAs reach bit-identical decisions without
// any global-memory round trip. The correction / bonus token is a three-level
// exponential race (groups of 8192 logits, their 256 chunks of 32, then the
// chunk's logits): every CTA sums the weights of its groups and chunks in one
// pass over the slice already in shared memory, all CTAs race the groups from
// the published sums, and only the CTA holding the winning group races its
// chunks and the winning chunk's entries, so Philox and logarithms are needed
// for ~300 candidates per draw instead of one per logit.
#include <math.h>

#include "common.cuh"
#include "launch_memo.h"

namespace specv {
namespace acc {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kGroup = 8192;         // logits per race group; a CTA's slice is whole groups
constexpr int kChunks = 256;         // chunks per group (one per thread)
constexpr int kMaxGroupsPerCta = 6;  // slice <= 48K logits (192 KB of shared memory)
constexpr int kMaxK = 31;

struct Params {
  const float* logits;
  const int32_t* drafts;
  const float* probs;
  const int32_t* mode;
  const float* temperature;
  int32_t* out_tokens;
  int32_t* accept_len;
  int32_t* dev_err;
  uint32_t seed_lo, seed_hi;
  int batch, k, vocab, slice, csize, gpc;  // gpc: race groups per CTA (slice = gpc * kGroup)
  int bulk;      // 1: rows are 16-byte aligned, use bulk copies
  int prefetch;  // 1: prefetch the next position's slice into L2
};

// Partial published by each CTA for one reduction.
struct __align__(16) Part {
  float f0;   // greedy: max logit; sampling: max logit of the slice; race: best key
  float f1;   // sampling: sum of exp relative to f0; race: sum of residual weights
  int32_t i0; // greedy / race: index of the best element
  int32_t pad;
};

struct Shared {
  // Cluster exchange, push model: each CTA writes its partials into slot
  // [its rank] of every peer before a cluster barrier, so everything read after
  // the barrier is local and no CTA touches another's memory after its last one.
  Part pos[kMaxK + 1][kMaxCluster];                   // per position: (max, sum) or (max, argmax)
  float group_w[2][kMaxCluster * kMaxGroupsPerCta];   // per race: weight sum of every group
  float chunk_w[kMaxGroupsPerCta * kChunks];          // this CTA's chunk weight sums (current race)
  float wf[kWarps];
  float wg[kWarps];
  int32_t wi[kWarps];
  int32_t draft[kMaxK];  // the row's draft tokens
  float l_draft[kMaxK];  // target logit of each draft token, read once at start
  float q_draft[kMaxK];  // draft probability of each draft token
  uint64_t bar;
};

// Block-wide (max value, lowest index) reduction; result valid in every thread.
__device__ __forceinline__ void block_argmax(Shared& sh, float& v, int& idx) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
  }
  __syncthreads();
  if (lane == 0) { sh.wf[warp] = v; sh.wi[warp] = idx; }
  __syncthreads();
  v = sh.wf[0];
  idx = sh.wi[0];
  for (int w = 1; w < kWarps; ++w) {
    const float ov = sh.wf[w];
    const int oi = sh.wi[w];
    if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
  }
}

__device__ __forceinline__ float block_max(Shared& sh, float v) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) sh.wf[warp] = v;
  __syncthreads();
  v = sh.wf[0];
  for (int w = 1; w < kWarps; ++w) v = fmaxf(v, sh.wf[w]);
  return v;
}

__device__ __forceinline__ float block_sum(Shared& sh, float v) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) sh.wg[warp] = v;
  __syncthreads();
  v = sh.wg[0];
  for (int w = 1; w < kWarps; ++w) v += sh.wg[w];
  return v;
}

// Slice values x in [0, n) are read as float4 groups when the slice is 16-byte
// aligned (always when bulk copies are used); `fn(x, v)` sees every element once.
template <typename F>
__device__ __forceinline__ void for_slice(const float* buf, int n, bool vec, F fn) {
  if (vec) {
    const float4* b4 = reinterpret_cast<const float4*>(buf);
    for (int g = threadIdx.x; g * 4 < n; g += kThreads) {
      const float4 v = b4[g];
      fn(4 * g, v.x);
      fn(4 * g + 1, v.y);
      fn(4 * g + 2, v.z);
      fn(4 * g + 3, v.w);
    }
  } else {
    for (int x = threadIdx.x; x < n; x += kThreads) fn(x, buf[x]);
  }
}

__global__ void __launch_bounds__(kThreads, 4) accept_kernel(const Params p) {
  extern __shared__ __align__(128) float buf[];
  __shared__ Shared sh;
  const int tid = threadIdx.x;
  const int csize = p.csize;
  const int rank = (int)cluster_ctarank();
  const int b = blockIdx.x / csize;
  const int k = p.k, R = k + 1, V = p.vocab;
  const int x0 = rank * p.slice;
  const int n = min(p.slice, V - x0);  // >= 1 by construction of csize
  const int lane = tid & 31;
  bool bulk = p.bulk != 0;
  const bool vec = bulk;  // 16-byte aligned slices
  uint32_t phase = 0;
  bool pending = false;  // a bulk copy was issued and not yet observed complete
  auto row_ptr = [&](int j) { return p.logits + ((int64_t)b * R + j) * V + x0; };
  auto issue_row = [&](int j) {
    if (bulk) {
      if (tid == 0) {
        mbar_arrive_expect_tx(&sh.bar, (uint32_t)n * 4u);
        bulk_g2s(smem_u32(buf), row_ptr(j), (uint32_t)n * 4u, &sh.bar);
      }
      pending = true;
    } else {
      const float* src = row_ptr(j);
      for (int x = tid; x < n; x += kThreads) buf[x] = src[x];
    }
  };
  // Position 0 is read whatever the row holds, so its copy starts before anything
  // else (the barrier is initialised by the issuing thread; the others first wait
  // on it after the block barrier below).
  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
  }
  if (bulk) issue_row(0);

  // ---- row validation (identical in every CTA of the cluster): the mode, the
  // temperature and the drafts (lane j holds d_j, k <= 31) are loaded together
  const int md = p.mode[b];
  const float t_row = p.temperature[b];
  const int d_lane = lane < k ? p.drafts[(int64_t)b * k + lane] : 0;
  const bool token_bad = __any_sync(0xffffffffu, lane < k && (d_lane < 0 || d_lane >= V));
  bool valid = md == SPEC_MODE_GREEDY || md == SPEC_MODE_SAMPLE;
  int32_t err_bit = valid ? 0 : SPEC_DEVERR_MODE;
  if (token_bad) { valid = false; err_bit |= SPEC_DEVERR_TOKEN; }
  float T = 1.f;
  if (valid && md == SPEC_MODE_SAMPLE) {
    T = t_row;
    if (!(T > 0.f) || !isfinite(T)) { valid = false; err_bit |= SPEC_DEVERR_TEMPERATURE; }
  }
  if (tid < k) sh.draft[tid] = d_lane;
  __syncthreads();
  if (!valid) {
    if (rank == 0 && tid == 0) {
      raise_error(p.dev_err, err_bit);
      for (int j = 0; j < R; ++j) p.out_tokens[(int64_t)b * R + j] = -1;
      p.accept_len[b] = -1;
    }
    // the copy of position 0 must land before this CTA's shared memory goes away
    if (pending && !mbar_wait_bounded(&sh.bar, phase) && tid == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
    return;  // uniform across the cluster: no CTA touches another's shared memory
  }
  const int32_t* d = sh.draft;
  const bool greedy = md == SPEC_MODE_GREEDY;
  const float c2 = (1.0f / T) * 1.4426950408889634f;  // logit -> log2 units of p
  // The target logit and draft probability of each draft token are first read
  // after the block barriers of position 0's reductions: they load while the
  // slice is in flight.
  if (!greedy && tid < k) {
    sh.l_draft[tid] = __ldg(p.logits + ((int64_t)b * R + tid) * V + d_lane);
    // without draft probabilities the draft distribution is one-hot at the drafted token
    sh.q_draft[tid] = p.probs ? __ldg(p.probs + ((int64_t)b * k + tid) * V + d_lane) : 1.f;
  }

  // Wait for position j's slice; once it has landed, pull what position j may
  // need next into L2 (the next position, and the draft probabilities a
  // rejection at j reads), so these prefetches never compete with the slice.
  auto wait_row = [&](int j) {
    if (bulk && pending) {
      const bool ok = mbar_wait_bounded(&sh.bar, phase);
      phase ^= 1u;
      pending = false;
      if (!ok) {
        if (tid == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        bulk = false;  // stop issuing copies; later rows use plain loads
      }
    }
    // same 16-byte alignment rule as the bulk copy
    if (bulk && p.prefetch && tid == 0 && j < k) {
      bulk_prefetch_l2(row_ptr(j + 1), (uint32_t)n * 4u);
      if (!greedy && p.probs) bulk_prefetch_l2(p.probs + ((int64_t)b * k + j) * V + x0, (uint32_t)n * 4u);
    }
    __syncthreads();
  };
  // Push this CTA's partial for position j into slot [rank] of every peer, then
  // wait for all of the cluster's partials (all reads after this are local).
  auto exchange = [&](int j, Part v) {
    if (tid < csize) st_cluster_v4(map_to_rank(smem_u32(&sh.pos[j][rank]), (uint32_t)tid), v.f0, v.f1, v.i0, 0);
    cluster_sync_all();
  };
  // (best value, lowest index) over the cluster's partials of position j, by a
  // fixed shuffle tree, so every CTA gets a bit-identical result.
  auto cluster_best = [&](int j, float& bv, int& bi) {
    float v = -INFINITY;
    int i = INT32_MAX;
    if (lane < csize) {
      v = sh.pos[j][lane].f0;
      i = sh.pos[j][lane].i0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i, o);
      if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
    }
    bv = v;
    bi = i;
  };
  // Softmax statistics of the whole row from the cluster's (slice max, slice sum) pairs.
  auto cluster_stats = [&](int j, float& M, float& Z) {
    float mr = -INFINITY, zr = 0.f;
    if (lane < csize) {
      mr = sh.pos[j][lane].f0;
      zr = sh.pos[j][lane].f1;
    }
    float mm = mr;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
    float zz = (lane < csize && mr != -INFINITY) ? zr * fast_exp2((mr - mm) * c2) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zz += __shfl_xor_sync(0xffffffffu, zz, o);
    M = mm;
    Z = zz;
  };
  // Write the row's result: accepted drafts, the final token, -1 padding.
  auto write_row = [&](int m, int token) {
    int32_t* o = p.out_tokens + (int64_t)b * R;
    for (int j = 0; j < m; ++j) o[j] = d[j];
    o[m] = token;
    for (int j = m + 1; j < R; ++j) o[j] = -1;
    p.accept_len[b] = m;
  };

  // Three-level exponential race over this row's weights at position `pos`
  // (an exact sampler of w / sum(w)): group g (8192 consecutive logits) wins
  // with key W_g / E, E = -ln U from word g%4 of Philox counter (g/4, pos, b, 2);
  // in that group chunk c = {8192g + 1024i + 4c + e} wins with key S_c / E from
  // counter ((256g+c)/4, pos, b, 3); in that chunk entry x wins with w_x / E
  // from counter (x/4, pos, b, 1). Ties go to the lowest index.
  // Weights, written over the slice in place as they are computed:
  //   residual: buf holds e_x = exp2((l - m) c2) from the statistics pass and
  //             w = max(0, e_x * f - q_x) with f = exp2((m - M) c2) / Z;
  //   plain:    buf holds logits and w = exp2((l - M) c2).
  // The CTA holding the winning group writes the output row (accept length m).
  // Returns false in every CTA if all weights are 0 (nothing written).
  auto race = [&](bool residual, float M, float f, const float* qrow, int pos, int slot, int m) -> bool {
    // ---- pass over the slice: weights (in place), chunk sums (thread t owns chunk t of each group), group sums
    for (int gl = 0; gl < p.gpc; ++gl) {
      const int gbase = gl * kGroup;
      float qv[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int off = gbase + 1024 * i + 4 * tid;
#pragma unroll
        for (int e = 0; e < 4; ++e) qv[i][e] = 0.f;
        if (residual && off < n) {
          if (qrow == nullptr) {  // one-hot draft distribution at the rejected draft token
#pragma unroll
            for (int e = 0; e < 4; ++e) qv[i][e] = (x0 + off + e == d[pos]) ? 1.f : 0.f;
          } else if (vec) {
            const float4 q4 = __ldg(reinterpret_cast<const float4*>(qrow + off));
            qv[i][0] = q4.x; qv[i][1] = q4.y; qv[i][2] = q4.z; qv[i][3] = q4.w;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) qv[i][e] = (off + e < n) ? qrow[off + e] : 0.f;
          }
        }
      }
      float cs = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int off = gbase + 1024 * i + 4 * tid;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (off + e < n) {
            const float v = buf[off + e];
            const float wt = residual ? fmaxf(v * f - qv[i][e], 0.f) : fast_exp2((v - M) * c2);
            buf[off + e] = wt;
            cs += wt;
          }
        }
      }
      sh.chunk_w[gl * kChunks + tid] = cs;
      const float gsum = block_sum(sh, cs);
      // push this group's sum to every CTA of the cluster
      if (tid < csize)
        st_cluster_f32(map_to_rank(smem_u32(&sh.group_w[slot][rank * p.gpc + gl]), (uint32_t)tid), gsum);
    }
    cluster_sync_all();
    // ---- level 1, the same in every CTA: warp 0 races the groups from the exchanged
    // sums and broadcasts (winner, total) through shared memory
    const int n_groups = (V + kGroup - 1) / kGroup;
    float gbest = -1.f, total = 0.f;
    int gwin = INT32_MAX;
    for (int gi = lane; tid < 32 && gi < ((n_groups + 31) & ~31); gi += 32) {
      const float wg = gi < n_groups ? sh.group_w[slot][gi] : 0.f;
      float key = 0.f;
      if (wg > 0.f) {
        const Philox4 w = philox4x32_10((uint32_t)gi >> 2, (uint32_t)pos, (uint32_t)b, 2u, p.seed_lo, p.seed_hi);
        key = wg / -logf(word_to_uniform(w.v[gi & 3]));
      }
      float kk = key, tt = wg;
      int ii = gi < n_groups ? gi : INT32_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, kk, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ii, o);
        tt += __shfl_xor_sync(0xffffffffu, tt, o);
        if (ok > kk || (ok == kk && oi < ii)) { kk = ok; ii = oi; }
      }
      total += tt;
      if (kk > gbest || (kk == gbest && ii < gwin)) { gbest = kk; gwin = ii; }
    }
    if (tid == 0) {
      sh.wf[0] = total;
      sh.wi[0] = gwin;
    }
    __syncthreads();
    total = sh.wf[0];
    gwin = sh.wi[0];
    __syncthreads();  // sh.wf / sh.wi are reused by the block reductions below
    if (!(total > 0.f)) return false;  // the same in every CTA
    const int owner = gwin / p.gpc, glw = gwin - owner * p.gpc;
    if (rank != owner) return true;
    // ---- level 2 (owner CTA): race the winning group's chunks
    const float sc = sh.chunk_w[glw * kChunks + tid];
    float key = 0.f;
    if (sc > 0.f) {
      const uint32_t ci = (uint32_t)(gwin * kChunks + tid);
      const Philox4 w = philox4x32_10(ci >> 2, (uint32_t)pos, (uint32_t)b, 3u, p.seed_lo, p.seed_hi);
      key = sc / -logf(word_to_uniform(w.v[ci & 3]));
    }
    int cwin = tid;
    block_argmax(sh, key, cwin);
    // ---- level 3: race the winning chunk's entries (warp 0, lane i: entries 1024 i + 4c + e)
    if (tid < 32) {
      float best = -1.f;
      int bx = INT32_MAX;
      if (tid < 8) {
        const int off = glw * kGroup + 1024 * tid + 4 * cwin;
        if (off < n) {
          const Philox4 w =
              philox4x32_10((uint32_t)((x0 + off) >> 2), (uint32_t)pos, (uint32_t)b, 1u, p.seed_lo, p.seed_hi);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (off + e < n) {
              const float wt = buf[off + e];
              if (wt > 0.f) {
                const float kx = wt / -logf(word_to_uniform(w.v[e]));
                if (kx > best) { best = kx; bx = x0 + off + e; }
              }
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bx, o);
        if (ov > best || (ov == best && oi < bx)) { best = ov; bx = oi; }
      }
      if (tid == 0) write_row(m, bx);
    }
    return true;
  };

  if (!bulk) issue_row(0);  // with bulk copies position 0 is already in flight
  for (int j = 0; j <= k; ++j) {
    wait_row(j);
    if (greedy) {
      // ---- argmax of the slice, then of the cluster (ranks are in vocab order)
      float v = -INFINITY;
      int idx = INT32_MAX;
      for_slice(buf, n, vec, [&](int x, float l) {
        if (l > v) { v = l; idx = x0 + x; }
      });
      block_argmax(sh, v, idx);
      exchange(j, Part{v, 0.f, idx, 0});
      float bv;
      int bi;
      cluster_best(j, bv, bi);
      if (j < k && d[j] == bi) {
        issue_row(j + 1);
        continue;
      }
      if (rank == 0 && tid == 0) write_row(j, bi);
      break;
    }
    if (j == k) {
      // ---- every draft accepted: bonus token from p_k, weights exp((l - max)/T)
      float mx = -INFINITY;
      for_slice(buf, n, vec, [&](int, float l) { mx = fmaxf(mx, l); });
      mx = block_max(sh, mx);
      exchange(j, Part{mx, 0.f, 0, 0});
      float M, Zunused;
      cluster_stats(j, M, Zunused);
      race(false, M, 1.f, nullptr, k, 0, k);
      break;
    }
    // ---- sampling statistics of p_j = softmax(l / T): slice max, then
    // e = exp2((l - max) c2) written over the slice (the race reuses it) and summed
    float mx = -INFINITY;
    for_slice(buf, n, vec, [&](int, float l) { mx = fmaxf(mx, l); });
    mx = block_max(sh, mx);
    float z = 0.f;
    if (vec) {
      float4* b4 = reinterpret_cast<float4*>(buf);
      for (int g4 = tid; g4 * 4 < n; g4 += kThreads) {
        float4 v = b4[g4];
        v.x = fast_exp2((v.x - mx) * c2); v.y = fast_exp2((v.y - mx) * c2);
        v.z = fast_exp2((v.z - mx) * c2); v.w = fast_exp2((v.w - mx) * c2);
        b4[g4] = v;
        z += (v.x + v.y) + (v.z + v.w);
      }
    } else {
      for (int x = tid; x < n; x += kThreads) {
        const float e = fast_exp2((buf[x] - mx) * c2);
        buf[x] = e;
        z += e;
      }
    }
    z = block_sum(sh, z);
    exchange(j, Part{mx, z, 0, 0});
    float M, Z;
    cluster_stats(j, M, Z);
    const float pd = fast_exp2((sh.l_draft[j] - M) * c2) / Z;
    const float qd = sh.q_draft[j];
    const Philox4 wu = philox4x32_10(0u, (uint32_t)j, (uint32_t)b, 0u, p.seed_lo, p.seed_hi);
    const float u = word_to_uniform(wu.v[0]);
    if (u * qd < pd) {
      issue_row(j + 1);
      continue;
    }
    // ---- rejected at j: race over max(0, p_j - q_j), or over p_j if that is all zero
    const float f = fast_exp2((mx - M) * c2) / Z;  // e_x * f = p_j(x) on this slice
    const float* qrow = p.probs ? p.probs + ((int64_t)b * k + j) * V + x0 : nullptr;
    if (!race(true, M, f, qrow, j, 0, j)) {
      // all-zero residual (rare): reload the logits over the overwritten slice and race over p_j
      __syncthreads();
      const float* src = row_ptr(j);
      for (int x = tid; x < n; x += kThreads) buf[x] = src[x];
      __syncthreads();
      race(false, M, 1.f, nullptr, j, 1, j);
    }
    break;
  }

  if (pending) {  // an issued copy must land before this CTA's shared memory goes away
    if (!mbar_wait_bounded(&sh.bar, phase) && tid == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
  }
  // No cluster barrier here: every remote access (a push) precedes the last
  // barrier, and nothing after it reads or writes another CTA's memory.
}

// Cluster size and slice: the slice is a whole number of race groups, at most
// 16 CTAs per cluster (the limit on one GPC), at most kMaxGroupsPerCta groups each.
static int pick_cluster(int vocab, int max_csize, int& slice, int& gpc) {
  const int n_groups = (vocab + kGroup - 1) / kGroup;
  int c = n_groups < max_csize ? n_groups : max_csize;
  gpc = (n_groups + c - 1) / c;
  c = (n_groups + gpc - 1) / gpc;  // every CTA owns at least one logit
  slice = gpc * kGroup;
  return c;
}

}  // namespace acc
}  // namespace specv

using namespace specv;

extern "C" int spec_accept(const float* target_logits, const int32_t* draft_tokens, const float* draft_probs,
                           uint64_t philox_seed, const int32_t* mode, const float* temperature,
                           int32_t* out_tokens, int32_t* accept_len, int32_t batch, int32_t k_draft,
                           int32_t vocab, int32_t* dev_err, spec_stream_t stream_) {
  if (batch < 0 || k_draft < 1 || vocab < 1) return SPEC_ERR_INVALID_ARG;
  if (batch == 0) return SPEC_OK;
  if (!target_logits || !draft_tokens || !mode || !temperature || !out_tokens || !accept_len)
    return SPEC_ERR_INVALID_ARG;
  if (k_draft > acc::kMaxK) return SPEC_ERR_UNSUPPORTED;
  int slice = 0, gpc = 0;
  const int csize = acc::pick_cluster(vocab, acc::kMaxCluster, slice, gpc);
  if (gpc > acc::kMaxGroupsPerCta) return SPEC_ERR_UNSUPPORTED;
  if ((int64_t)batch * csize > INT32_MAX) return SPEC_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  acc::Params p;
  p.logits = target_logits;
  p.drafts = draft_tokens;
  p.probs = draft_probs;
  p.mode = mode;
  p.temperature = temperature;
  p.out_tokens = out_tokens;
  p.accept_len = accept_len;
  p.dev_err = dev_err;
  p.seed_lo = (uint32_t)(philox_seed & 0xFFFFFFFFu);
  p.seed_hi = (uint32_t)(philox_seed >> 32);
  p.batch = batch;
  p.k = k_draft;
  p.vocab = vocab;
  p.slice = slice;
  p.csize = csize;
  p.gpc = gpc;
  const bool aligned = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(target_logits) & 15) == 0) &&
                       (draft_probs == nullptr || (reinterpret_cast<uintptr_t>(draft_probs) & 15) == 0);
  p.bulk = aligned ? 1 : 0;
  p.prefetch = 1;

  auto kern = acc::accept_kernel;
  const int dev = current_device();
  if (dev < 0) return SPEC_ERR_LAUNCH;
  // The cluster plan (size, slice, groups per CTA) depends only on the device and
  // the vocabulary: it is worked out once per (device, vocabulary), together with
  // the kernel attributes, under a lock shared by all host threads.
  static LaunchMemo memo;
  static int plan_vocab[kMaxDevices], plan_csize[kMaxDevices], plan_slice[kMaxDevices], plan_gpc[kMaxDevices];
  static bool nonportable[kMaxDevices];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(acc::kThreads, 1, 1);
  cfg.stream = stream;
  {
    std::lock_guard<std::mutex> lock(memo.mu);
    if (plan_vocab[dev] != vocab) {  // vocab >= 1, so 0 marks "no plan yet"
      // Clusters larger than 8 CTAs are not guaranteed to fit a GPC; if the
      // device cannot hold one, use 8 CTAs with larger slices.
      for (int attempt = 0; attempt < 2; ++attempt) {
        if (!grant_smem_locked(memo, (const void*)kern, dev, (size_t)p.slice * sizeof(float))) return SPEC_ERR_LAUNCH;
        if (p.csize <= 8) break;
        if (!nonportable[dev]) {
          if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return SPEC_ERR_LAUNCH;
          nonportable[dev] = true;
        }
        cfg.gridDim = dim3((unsigned)p.csize, 1, 1);
        cfg.dynamicSmemBytes = (size_t)p.slice * sizeof(float);
        attr[0].val.clusterDim.x = (unsigned)p.csize;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0) break;
        (void)cudaGetLastError();
        p.csize = acc::pick_cluster(vocab, 8, p.slice, p.gpc);
        if (p.gpc > acc::kMaxGroupsPerCta) return SPEC_ERR_UNSUPPORTED;
      }
      plan_csize[dev] = p.csize;
      plan_slice[dev] = p.slice;
      plan_gpc[dev] = p.gpc;
      plan_vocab[dev] = vocab;
    }
    p.csize = plan_csize[dev];
    p.slice = plan_slice[dev];
    p.gpc = plan_gpc[dev];
  }
  cfg.gridDim = dim3((unsigned)(batch * p.csize), 1, 1);
  cfg.dynamicSmemBytes = (size_t)p.slice * sizeof(float);
  attr[0].val.clusterDim.x = (unsigned)p.csize;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return SPEC_ERR_LAUNCH;
  return SPEC_OK;
}
