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
// the vocabulary into contiguous slices (a multiple of 4 logits each; at most
// 16 CTAs, 8 where the device cannot schedule a 16-CTA cluster). Positions are
// processed in order and the row stops at the first rejection, so logits past
// it are never read (early exit), and nothing is fetched ahead of a decision.
// For each position every CTA pulls its slice into shared memory with one
// bulk asynchronous copy (TMA engine, mbarrier completion; position 0's copy
// is issued first thing, before the row is validated). Each thread folds its
// float4 groups of the slice into one partial in a single pass (a running
// max with its sum of exponentials, or a running argmax), each warp combines
// its lanes by shuffles and pushes the result straight into an exchange slot
// of every CTA of the cluster (distributed shared memory), and one cluster
// barrier per position publishes them: there is no CTA-wide barrier on the
// path. Every warp of every CTA then combines the same partials in the same
// order, so all CTAs reach bit-identical decisions. Lane j of every warp holds
// draft j with its target logit and draft probability, read by shuffle at the
// decisions. CTAs have 128 threads where six fit an SM and the grid fills it
// (more rows resident), 256 otherwise.
//
// The correction / bonus token is the exponential race over the whole
// vocabulary: entry x has the key w_x / E_x, E_x = -ln U_x, U_x from word
// x mod 4 of Philox counter (x/4, m, b, 1), and the largest key wins. Each
// thread first computes, for every entry of its slice, the weight and the
// uniform and keeps the bounds w U / (1-U) <= w / E <= w / (1-U) (from
// 1-U <= -ln U <= (1-U)/U), writing the upper bound over the slice; the
// largest lower bound of the warp then rules out every entry whose upper bound
// falls below it, and only the few entries left get the exact key (the
// logarithm). The winner of each warp is exchanged like the statistics. A
// rejected row's draft probabilities are read only here, after the decision.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "launch_memo.h"

namespace specv {
namespace acc {

constexpr int kMaxCluster = 16;
constexpr int kMaxWarps = 8;
constexpr int kMaxK = 31;
constexpr int kMinSlice = 4096;       // logits per CTA before another CTA joins the row
constexpr int kMaxSlice = 48 * 1024;  // logits per CTA (192 KB of shared memory)
constexpr int kBatch = 4;             // float4 groups per thread whose loads are in flight together

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
  int batch, k, vocab, slice, csize;
  int bulk;  // 1: rows are 16-byte aligned, use bulk copies and float4 loads
};

// A partial pushed by one warp for one exchange.
struct __align__(16) Part {
  float f0;    // max logit, best race key, or the argmax value
  float f1;    // sum of exponentials relative to f0
  int32_t i0;  // argmax / race index
  int32_t pad;
};

struct Shared {
  // Exchange, push model: warp w of CTA r writes its partial into slot
  // [r * warps + w] of every CTA of the cluster before a cluster barrier, so
  // everything read after the barrier is local. Two slots alternate: a CTA
  // writes slot e & 1 of exchange e only after the barrier of exchange e - 1,
  // which every CTA reaches after reading exchange e - 2 from the same slot.
  Part xch[2][kMaxCluster * kMaxWarps];
  uint64_t bar;
};

// Split cluster barrier used once at start-up: every CTA arrives as soon as it
// runs and waits just before its first push into a peer's shared memory, so no
// CTA writes into a peer that has not started (the rule for distributed shared
// memory); by then the barrier has long completed.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory"); }

// Combine two (max, sum of exp2((x - max) c2)) pairs; commutative, so a
// butterfly leaves the same bits in every lane.
__device__ __forceinline__ void ms_combine(float& m, float& s, float om, float os, float c2) {
  const float nm = fmaxf(m, om);
  const float a = m == -INFINITY ? 0.f : s * fast_exp2((m - nm) * c2);
  const float b = om == -INFINITY ? 0.f : os * fast_exp2((om - nm) * c2);
  m = nm;
  s = a + b;
}

// (value, index) with the larger value, the lower index on ties.
__device__ __forceinline__ void vi_combine(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}

template <int T>
__global__ void __launch_bounds__(T, T == 128 ? 6 : 3) accept_kernel(const Params p) {
  constexpr int kWarps = T / 32;
  extern __shared__ __align__(128) float buf[];
  __shared__ Shared sh;
  float4* buf4 = reinterpret_cast<float4*>(buf);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int csize = p.csize;
  const int rank = (int)cluster_ctarank();
  const int b = blockIdx.x / csize;
  const int k = p.k, R = k + 1, V = p.vocab;
  const int x0 = rank * p.slice;              // a multiple of 4: group g holds Philox counter x0/4 + g
  const int n = min(p.slice, V - x0);         // >= 1 by construction of csize
  const int ngroups = (n + 3) >> 2;
  const bool full = (n & 3) == 0;             // every float4 group lies inside the slice
  bool bulk = p.bulk != 0;
  uint32_t phase = 0;
  bool pending = false;  // a bulk copy was issued and not yet observed complete
  int xs = 0;            // exchanges so far (slot parity)
  auto row_ptr = [&](int j) { return p.logits + ((int64_t)b * R + j) * V + x0; };
  // Copy position j's slice into shared memory. Bulk: one copy by thread 0,
  // completion on the mbarrier. Plain (unaligned rows): every thread loads the
  // groups it processes itself, so no barrier is needed; entries past the
  // slice read as -inf.
  auto issue_row = [&](int j) {
    if (bulk) {
      if (tid == 0) {
        mbar_arrive_expect_tx(&sh.bar, (uint32_t)n * 4u);
        bulk_g2s(smem_u32(buf), row_ptr(j), (uint32_t)n * 4u, &sh.bar);
      }
      pending = true;
    } else {
      const float* src = row_ptr(j);
      for (int g = tid; g < ngroups; g += T) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = 4 * g + e < n ? src[4 * g + e] : -INFINITY;
        buf4[g] = make_float4(v[0], v[1], v[2], v[3]);
      }
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
  cluster_arrive_relaxed();

  // ---- row validation (identical in every CTA of the cluster): the mode, the
  // temperature and the drafts (lane j holds d_j, k <= 31) are loaded together
  const int md = p.mode[b];
  const float t_row = p.temperature[b];
  const int d_lane = lane < k ? p.drafts[(int64_t)b * k + lane] : 0;
  const bool token_bad = __any_sync(0xffffffffu, lane < k && (d_lane < 0 || d_lane >= V));
  bool valid = md == SPEC_MODE_GREEDY || md == SPEC_MODE_SAMPLE;
  int32_t err_bit = valid ? 0 : SPEC_DEVERR_MODE;
  if (token_bad) { valid = false; err_bit |= SPEC_DEVERR_TOKEN; }
  float T_ = 1.f;
  if (valid && md == SPEC_MODE_SAMPLE) {
    T_ = t_row;
    if (!(T_ > 0.f) || !isfinite(T_)) { valid = false; err_bit |= SPEC_DEVERR_TEMPERATURE; }
  }
  const bool greedy = md == SPEC_MODE_GREEDY;
  // Lane j of every warp holds draft j, its target logit and its draft
  // probability; decisions read them by shuffle, so there is no shared copy and
  // no block barrier. The logit and probability are first used at position 0's
  // decision, so their loads arrive while the slice is in flight. Without draft
  // probabilities the draft distribution is one-hot at the drafted token.
  float l_d = 0.f, q_d = 1.f;
  if (lane < k && valid && !greedy) {
    l_d = __ldg(p.logits + ((int64_t)b * R + lane) * V + d_lane);
    if (p.probs) q_d = __ldg(p.probs + ((int64_t)b * k + lane) * V + d_lane);
  }
  // The mbarrier that thread 0 initialised is visible to every thread after this
  // wait (its init fence is a release at cluster scope, the wait an acquire).
  cluster_wait();  // every CTA of the cluster is running (see cluster_arrive_relaxed)
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
  const float c2 = (1.0f / T_) * 1.4426950408889634f;  // logit -> log2 units of p

  // Wait for the slice in flight (bulk copies; every thread observes the
  // mbarrier itself, so no block barrier follows).
  auto wait_row = [&]() {
    if (bulk && pending) {
      const bool ok = mbar_wait_bounded(&sh.bar, phase);
      phase ^= 1u;
      pending = false;
      if (!ok) {
        if (tid == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
        bulk = false;  // stop issuing copies; later rows use plain loads
      }
    }
  };
  // Push this warp's partial (the same in all its lanes) into every CTA of the
  // cluster, then wait for the cluster's partials; returns the slot to read.
  auto exchange = [&](float f0, float f1, int i0) -> const Part* {
    const int slot = xs & 1;
    ++xs;
    if (lane < csize)
      st_cluster_v4(map_to_rank(smem_u32(&sh.xch[slot][rank * kWarps + warp]), (uint32_t)lane), f0, f1, i0, 0);
    cluster_sync_all();
    return sh.xch[slot];
  };
  const int nparts = csize * kWarps;
  // Softmax statistics of the whole row from the exchanged (max, sum) partials.
  auto row_stats = [&](const Part* x, float& M, float& Z) {
    float m = -INFINITY, s = 0.f;
    for (int i = lane; i < nparts; i += 32) ms_combine(m, s, x[i].f0, x[i].f1, c2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
      ms_combine(m, s, om, os, c2);
    }
    M = m;
    Z = s;
  };
  // (best value, lowest index) over the exchanged partials.
  auto row_best = [&](const Part* x, float& bv, int& bi) {
    float v = -INFINITY;
    int i = INT32_MAX;
    for (int t = lane; t < nparts; t += 32) vi_combine(v, i, x[t].f0, x[t].i0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vi_combine(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
    bv = v;
    bi = i;
  };
  auto warp_best = [&](float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vi_combine(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
  };
  // Write the row's result (one warp, lane j writes position j): accepted
  // drafts, the final token, -1 padding.
  auto write_row = [&](int m, int token) {
    if (lane < R) p.out_tokens[(int64_t)b * R + lane] = lane < m ? d_lane : (lane == m ? token : -1);
    if (lane == 0) p.accept_len[b] = m;
  };
  // Four consecutive values at group g of a row slice in global memory (16-byte
  // loads when rows are aligned; scalar loads, zero past the slice, otherwise).
  auto load4 = [&](const float* src, int g) -> float4 {
    if (p.bulk) return __ldg(reinterpret_cast<const float4*>(src) + g);
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = 4 * g + e < n ? src[4 * g + e] : 0.f;
    return make_float4(v[0], v[1], v[2], v[3]);
  };

  // Exponential race at position `pos` over the slice's logits (in buf):
  //   residual: w = max(0, exp2((l - M) c2) * invZ - q)  (q: one-hot at the rejected draft when qrow is null)
  //   plain:    w = exp2((l - M) c2)                     (scale does not matter to the race)
  // Returns the winning index (the same in every CTA), or -1 if every weight is 0.
  // Overwrites the slice with the key upper bounds.
  auto race = [&](bool residual, float M, float invZ, const float* qrow, int pos) -> int {
    const uint32_t cbase = (uint32_t)x0 >> 2;
    const float mc2 = M * c2;
    const int dpos = __shfl_sync(0xffffffffu, d_lane, pos);  // the rejected draft (one-hot q)
    // The draft row of the rejected position is read in full below: ask L2 for
    // all of this thread's pieces of it at once, so the batched loads hit L2.
    if (residual && qrow != nullptr)
      for (int g = tid; g < ngroups; g += T) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(qrow + 4 * g));
    // One pass, kBatch groups of the thread at a time: their draft-probability
    // loads are issued first, the Philox blocks (which need no data) are
    // computed while those loads are in flight, then each group's weights and
    // key bounds are formed and the upper bounds written over the slice.
    float lb_max = 0.f;
    for (int g0 = tid; g0 < ngroups; g0 += kBatch * T) {
      float4 q4[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int g = g0 + i * T;
        q4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (residual && qrow != nullptr && g < ngroups) q4[i] = load4(qrow, g);
      }
      Philox4 r[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        r[i] = philox4x32_10(cbase + (uint32_t)(g0 + i * T), (uint32_t)pos, (uint32_t)b, 1u, p.seed_lo, p.seed_hi);
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int g = g0 + i * T;
        if (g < ngroups) {
          const float4 l4 = buf4[g];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
          const float qv[4] = {q4[i].x, q4[i].y, q4[i].z, q4[i].w};
          const bool tail = !full && g == ngroups - 1;
          float ub[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float pe = fast_exp2(fmaf(lv[e], c2, -mc2));
            float qe = qv[e];
            if (residual && qrow == nullptr) qe = (x0 + 4 * g + e == dpos) ? 1.f : 0.f;
            float w = residual ? fmaxf(pe * invZ - qe, 0.f) : pe;
            if (tail && 4 * g + e >= n) w = 0.f;
            // the word's top 23 bits j as the float 1 + j 2^-23 in [1, 2): then
            // U = (2j + 1) 2^-24 = f1 - (1 - 2^-24) and 1 - U are exact subtractions
            const float f1 = __uint_as_float(0x3F800000u | (r[i].v[e] >> 9));
            const float u = f1 - 0.999999940395355224609375f;
            const float v = 1.f - u;
            ub[e] = __fdividef(w, v);
            lb_max = fmaxf(lb_max, ub[e] * u);
          }
          buf4[g] = make_float4(ub[0], ub[1], ub[2], ub[3]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lb_max = fmaxf(lb_max, __shfl_xor_sync(0xffffffffu, lb_max, o));
    // exact keys for the entries whose upper bound reaches the warp's best lower bound
    float best = -1.f;
    int bx = INT32_MAX;
    for (int g = tid; g < ngroups; g += T) {
      const float4 u4 = buf4[g];
      const float ub[4] = {u4.x, u4.y, u4.z, u4.w};
      bool any = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) any |= ub[e] > 0.f && ub[e] >= lb_max;
      if (any) {
        const Philox4 r = philox4x32_10(cbase + (uint32_t)g, (uint32_t)pos, (uint32_t)b, 1u, p.seed_lo, p.seed_hi);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (ub[e] > 0.f && ub[e] >= lb_max) {
            const float u = word_to_uniform(r.v[e]);
            const float key = (ub[e] * (1.f - u)) / -logf(u);
            if (key > best) {
              best = key;
              bx = x0 + 4 * g + e;
            }
          }
        }
      }
    }
    warp_best(best, bx);
    const Part* x = exchange(best, 0.f, bx);
    float kv;
    int win;
    row_best(x, kv, win);
    return kv > 0.f ? win : -1;
  };

  if (!bulk) issue_row(0);  // with bulk copies position 0 is already in flight
  for (int j = 0; j <= k; ++j) {
    wait_row();
    if (greedy) {
      // ---- argmax of the slice (lowest index on ties), then of the row. Four
      // independent running maxima (one per float4 lane) keep four compare
      // chains in flight; each starts at its first element, so equal values
      // still resolve to the lowest index when the four are merged.
      float v4[4];
      int i4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v4[e] = -INFINITY;
        i4[e] = tid < ngroups ? x0 + 4 * tid + e : INT32_MAX;
      }
      for (int g = tid; g < ngroups; g += T) {
        const float4 l4 = buf4[g];
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if ((full || 4 * g + e < n) && lv[e] > v4[e]) {
            v4[e] = lv[e];
            i4[e] = x0 + 4 * g + e;
          }
        }
      }
      float v = v4[0];
      int idx = i4[0];
#pragma unroll
      for (int e = 1; e < 4; ++e) vi_combine(v, idx, v4[e], i4[e]);
      warp_best(v, idx);
      const Part* x = exchange(v, 0.f, idx);
      float bv;
      int bi;
      row_best(x, bv, bi);
      if (j < k && __shfl_sync(0xffffffffu, d_lane, j) == bi) {
        issue_row(j + 1);
        continue;
      }
      if (rank == 0 && warp == 0) write_row(j, bi);
      break;
    }
    // ---- sampling: max and sum of exp2((l - max) c2) of the slice in one pass,
    // with two running (max, sum) pairs over alternate groups (two chains in flight)
    auto fold = [&](const float4 l4, float& m, float& s) {
      const float gm = fmaxf(fmaxf(l4.x, l4.y), fmaxf(l4.z, l4.w));
      if (gm == -INFINITY) return;
      if (gm > m) {
        if (m != -INFINITY) s *= fast_exp2((m - gm) * c2);
        m = gm;
      }
      s += (fast_exp2((l4.x - m) * c2) + fast_exp2((l4.y - m) * c2)) +
           (fast_exp2((l4.z - m) * c2) + fast_exp2((l4.w - m) * c2));
    };
    float m = -INFINITY, s = 0.f, mb = -INFINITY, sb = 0.f;
    for (int g = tid; g < ngroups; g += 2 * T) {
      fold(buf4[g], m, s);
      if (g + T < ngroups) fold(buf4[g + T], mb, sb);
    }
    ms_combine(m, s, mb, sb, c2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
      ms_combine(m, s, om, os, c2);
    }
    const Part* x = exchange(m, s, 0);
    float M, Z;
    row_stats(x, M, Z);
    int token;
    if (j < k) {
      const float pd = fast_exp2((__shfl_sync(0xffffffffu, l_d, j) - M) * c2) / Z;
      const float qd = __shfl_sync(0xffffffffu, q_d, j);
      const Philox4 wu = philox4x32_10(0u, (uint32_t)j, (uint32_t)b, 0u, p.seed_lo, p.seed_hi);
      const float u = word_to_uniform(wu.v[0]);
      if (u * qd < pd) {
        issue_row(j + 1);
        continue;
      }
      // ---- rejected at j: race over max(0, p_j - q_j), or over p_j if that is all zero
      const float* qrow = p.probs ? p.probs + ((int64_t)b * k + j) * V + x0 : nullptr;
      token = race(true, M, 1.f / Z, qrow, j);
      if (token < 0) {
        // all-zero residual (rare): reload the logits over the overwritten slice, race over p_j
        const float* src = row_ptr(j);
        for (int g = tid; g < ngroups; g += T) {
          float4 v = load4(src, g);
          if (!p.bulk) {
            if (4 * g + 1 >= n) v.y = -INFINITY;
            if (4 * g + 2 >= n) v.z = -INFINITY;
            if (4 * g + 3 >= n) v.w = -INFINITY;
          }
          buf4[g] = v;
        }
        token = race(false, M, 1.f, nullptr, j);
      }
    } else {
      // ---- every draft accepted: bonus token from p_k
      token = race(false, M, 1.f, nullptr, k);
    }
    if (rank == 0 && warp == 0) write_row(j, token);
    break;
  }

  if (pending) {  // an issued copy must land before this CTA's shared memory goes away
    if (!mbar_wait_bounded(&sh.bar, phase) && tid == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
  }
  // No cluster barrier here: every remote access (a push) precedes the last
  // barrier, and nothing after it reads or writes another CTA's memory.
}

// Cluster size and slice: at most `max_csize` CTAs, slices of at least
// kMinSlice logits (fewer CTAs for small vocabularies), a multiple of 4 each.
static int pick_cluster(int vocab, int max_csize, int& slice) {
  int c = (vocab + kMinSlice - 1) / kMinSlice;
  c = c < 1 ? 1 : (c > max_csize ? max_csize : c);
  slice = (vocab + c - 1) / c;
  slice = (slice + 3) & ~3;
  return (vocab + slice - 1) / slice;  // every CTA owns at least one logit
}

// Static shared memory per CTA (the Shared struct) plus what the runtime reserves.
constexpr size_t kStaticBytes = sizeof(Shared) + 1024;

// 128 threads per CTA where six CTAs fit an SM (small slices: more rows
// resident) and the grid is large enough to use them, else 256 (more warps to
// hide each CTA's latencies). SPEC_ACCEPT_THREADS=128 or =256 overrides.
static int pick_threads(int slice, int64_t ctas, int sms) {
  const char* env = getenv("SPEC_ACCEPT_THREADS");
  if (env != nullptr && strcmp(env, "128") == 0) return 128;
  if (env != nullptr && strcmp(env, "256") == 0) return 256;
  if (ctas <= 2 * (int64_t)sms) return 256;
  return 6 * ((size_t)slice * 4 + kStaticBytes) <= 228 * 1024 ? 128 : 256;
}

struct Plan {
  int vocab = 0, csize = 0, slice = 0;
};

template <int T>
static int launch(Params p, int batch, int vocab, cudaStream_t stream) {
  auto kern = accept_kernel<T>;
  const int dev = current_device();
  if (dev < 0) return SPEC_ERR_LAUNCH;
  // The cluster plan (size, slice) depends only on the device and the
  // vocabulary: it is worked out once per (device, vocabulary) together with
  // the kernel attributes, under a lock shared by all host threads.
  static LaunchMemo memo;
  static Plan plans[kMaxDevices];
  static bool attrs_set[kMaxDevices];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(T, 1, 1);
  cfg.stream = stream;
  {
    std::lock_guard<std::mutex> lock(memo.mu);
    if (!attrs_set[dev]) {
      // 16-CTA clusters are beyond the portable size; the largest shared-memory
      // carveout keeps as many slices resident as fit
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
          cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return SPEC_ERR_LAUNCH;
      attrs_set[dev] = true;
    }
    if (plans[dev].vocab != vocab) {  // vocab >= 1, so 0 marks "no plan yet"
      // Clusters larger than 8 CTAs are not guaranteed to fit a GPC; if the
      // device cannot hold one, use 8 CTAs with larger slices.
      for (int attempt = 0; attempt < 2; ++attempt) {
        if (p.slice > kMaxSlice) return SPEC_ERR_UNSUPPORTED;
        if (!grant_smem_locked(memo, (const void*)kern, dev, (size_t)p.slice * sizeof(float))) return SPEC_ERR_LAUNCH;
        if (p.csize <= 8) break;
        cfg.gridDim = dim3((unsigned)p.csize, 1, 1);
        cfg.dynamicSmemBytes = (size_t)p.slice * sizeof(float);
        attr[0].val.clusterDim.x = (unsigned)p.csize;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0) break;
        (void)cudaGetLastError();
        p.csize = pick_cluster(vocab, 8, p.slice);
      }
      plans[dev].csize = p.csize;
      plans[dev].slice = p.slice;
      plans[dev].vocab = vocab;
    }
    p.csize = plans[dev].csize;
    p.slice = plans[dev].slice;
  }
  cfg.gridDim = dim3((unsigned)(batch * p.csize), 1, 1);
  cfg.dynamicSmemBytes = (size_t)p.slice * sizeof(float);
  attr[0].val.clusterDim.x = (unsigned)p.csize;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return SPEC_ERR_LAUNCH;
  return SPEC_OK;
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
  int slice = 0;
  const int csize = acc::pick_cluster(vocab, acc::kMaxCluster, slice);
  if (slice > acc::kMaxSlice) return SPEC_ERR_UNSUPPORTED;
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
  const bool aligned = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(target_logits) & 15) == 0) &&
                       (draft_probs == nullptr || (reinterpret_cast<uintptr_t>(draft_probs) & 15) == 0);
  p.bulk = aligned ? 1 : 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return acc::pick_threads(slice, (int64_t)batch * csize, sms) == 128 ? acc::launch<128>(p, batch, vocab, stream)
                                                                      : acc::launch<256>(p, batch, vocab, stream);
}
