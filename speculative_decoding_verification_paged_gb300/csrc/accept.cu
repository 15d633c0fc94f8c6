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
// the vocabulary into contiguous slices (a multiple of 4 logits each, at most
// 16 CTAs). Positions are processed in order and the row stops at the first
// rejection, so logits past it are never read (early exit); only when the
// batch's positions are small (B V 4 bytes at most 32 MB) is each thread's
// first batch of position j + 1 loaded while position j is decided. The logits
// stream through registers: each thread loads eight float4 groups of its slice
// at a time (128-bit loads, all in flight together) and folds them into one
// partial (the batch maximum first, then one rescale of the running sum of
// exponentials and one exponential per logit; or a running argmax). Nothing is
// staged in shared memory, so a CTA holds only its exchange slots and as many
// CTAs stay resident as the registers allow: the launch picks the CTA size and
// cluster size that give the most threads per row while every row of the batch
// is resident at once, and the clusters walk the rows (persistent) when the
// batch is larger than that. Each warp combines its lanes by shuffles and
// pushes the result straight into an exchange slot of every CTA of the cluster
// (distributed shared memory, an asynchronous store that counts its bytes on
// the receiving CTA's mbarrier), and each CTA waits on its own mbarrier until
// every partial of the exchange has landed: there is no CTA-wide or
// cluster-wide barrier on the path. Every warp of every CTA then combines the
// same partials in the same order, so all CTAs reach bit-identical decisions.
// Lane j of every warp holds draft j with its target logit, its draft
// probability and the uniform of its test, read by shuffle at the decisions.
//
// The correction / bonus token is the exponential race over the whole
// vocabulary: entry x has the key w_x / E_x, E_x = -ln U_x, U_x from word
// x mod 4 of Philox counter (x/4, m, b, 1), and the largest key wins. The race
// is one more streaming pass over the slice at the decided position (its
// logits were just read, so they come from L2; a rejected row's draft
// probabilities are read only here, after the decision). For every entry the
// thread forms the weight and the uniform and the bounds
// w U / (1-U) <= w / E <= w / (1-U) (from 1-U <= -ln U <= (1-U)/U); after each
// batch the warp takes the largest lower bound so far, and only entries whose
// upper bound reaches it get the exact key (the logarithm). The bound only
// grows, and every entry that could still win reaches it when it is seen, so
// the best exact key is the race's winner. The winner of each warp is
// exchanged like the statistics.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <type_traits>

#include "common.cuh"
#include "launch_memo.h"

namespace specv {
namespace acc {

constexpr int kMaxCluster = 16;
constexpr int kMaxWarps = 8;
constexpr int kMaxK = 31;
constexpr int kMaxVocab = 1 << 30;
constexpr int kNB = 8;  // float4 groups per thread in flight together (statistics, argmax)
constexpr int kRB = 2;  // float4 groups per thread in flight together (race: logits and draft probabilities)
constexpr int64_t kPrefetchMaxBytes = 32ll << 20;  // position reads over the batch, at most, to prefetch

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
  int vec;       // 1: rows are 16-byte aligned, use float4 loads
  int prefetch;  // 1: load position j + 1's first batch while position j is decided
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
  // [r * warps + w] of every CTA of the cluster with an asynchronous store that
  // counts its 16 bytes on that CTA's mbarrier xbar[e & 1], so everything read
  // after the wait is local. Two slots alternate: a CTA pushes exchange e only
  // after its own exchange e - 1 completed, which needs every peer's push of
  // e - 1, which each peer makes after it has read exchange e - 2 from the same
  // slot (its next push depends on what it read).
  Part xch[2][kMaxCluster * kMaxWarps];
  uint64_t xbar[2];  // phase k of xbar[s] completes with exchange 2k + s
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

// Largest of three (the three-input PTX form, sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Approximate reciprocal (rcp.approx: no refinement steps).
__device__ __forceinline__ float fast_rcp(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
  return r;
}

template <bool B>
using Flag = std::integral_constant<bool, B>;
template <int M>
using RaceKind = std::integral_constant<int, M>;
constexpr int kRacePlain = 0;     // w = p (bonus token, or an all-zero residual)
constexpr int kRaceResidual = 1;  // w = max(0, p - q)
constexpr int kRaceOneHot = 2;    // w = max(0, p - [x == d])  (no draft probabilities)

// 16-byte asynchronous store into a peer CTA's shared memory that also counts its
// bytes on the peer's mbarrier (complete_tx); both are shared::cluster addresses.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, int32_t c, int32_t d, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];\n"
               ::"r"(addr), "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(c), "r"(d), "r"(bar)
               : "memory");
}
// Wait (bounded) for the phase of this CTA's mbarrier with the given parity, with
// cluster-scope acquire: the data peers stored into this CTA is visible after it.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          long long limit_cycles = 2000000000LL) {
  auto try_wait = [&]() -> bool {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (try_wait()) return true;
  const long long start = clock64();
  while (!try_wait()) {
    if (clock64() - start > limit_cycles) return false;
  }
  return true;
}
// Registers bound the CTAs resident per SM (1024 threads at 64 registers each).
template <int T>
__global__ void __launch_bounds__(T, 1024 / T) accept_kernel(const Params p) {
  constexpr int kWarps = T / 32;
  constexpr int kStep = kNB * T;  // groups per statistics / argmax batch of the block
  constexpr int kRStep = kRB * T; // groups per race iteration of the block
  __shared__ Shared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int csize = p.csize;
  const int rank = (int)cluster_ctarank();
  const int nclusters = (int)(gridDim.x / (unsigned)csize);
  const int k = p.k, R = k + 1, V = p.vocab;
  const int x0 = rank * p.slice;       // a multiple of 4: group g holds Philox counter x0/4 + g
  const int n = min(p.slice, V - x0);  // >= 1 by construction of the slice
  const int ngroups = (n + 3) >> 2;
  const bool vec = p.vec != 0;
  const int nparts = csize * kWarps;
  const float4 kZero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  int xs = 0;           // exchanges so far (slot parity)
  bool joined = false;  // the start-up cluster barrier was waited on
  if (threadIdx.x == 0) {
    mbar_init(&sh.xbar[0], 1);  // the local arrival sets the exchange's byte count
    mbar_init(&sh.xbar[1], 1);
    fence_mbar_init();  // visible to the cluster before any peer can push
  }
  __syncthreads();
  cluster_arrive_relaxed();

  // Group g of a slice in global memory, checked: one 16-byte load when rows are
  // aligned, else scalar loads; `fill` for entries past the slice. Logits are
  // read through the non-coherent path (the race may read them again from L2);
  // draft probabilities, read once, with the streaming hint.
  auto load4 = [&](const float* src, int g, float fill) -> float4 {
    if (g >= ngroups) return make_float4(fill, fill, fill, fill);
    if (vec) return __ldg(reinterpret_cast<const float4*>(src) + g);
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = 4 * g + e < n ? __ldg(src + 4 * g + e) : fill;
    return make_float4(v[0], v[1], v[2], v[3]);
  };
  auto loadq4 = [&](const float* src, int g) -> float4 {
    if (g >= ngroups) return make_float4(0.f, 0.f, 0.f, 0.f);
    if (vec) return __ldcs(reinterpret_cast<const float4*>(src) + g);
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = 4 * g + e < n ? __ldcs(src + 4 * g + e) : 0.f;
    return make_float4(v[0], v[1], v[2], v[3]);
  };
  // The thread's groups gb + i T + tid, i < kNB (-inf past the slice); batches
  // that lie wholly inside an aligned slice load without checks.
  auto load_batch = [&](const float* src, int gb, float4 (&v)[kNB]) {
    if (vec && gb + kStep <= ngroups) {
      const float4* s4 = reinterpret_cast<const float4*>(src) + gb + tid;
#pragma unroll
      for (int i = 0; i < kNB; ++i) v[i] = __ldg(s4 + i * T);
    } else {
#pragma unroll
      for (int i = 0; i < kNB; ++i) v[i] = load4(src, gb + i * T + tid, -INFINITY);
    }
  };
  // Largest of a batch.
  auto batch_max = [&](const float4 (&v)[kNB]) -> float {
    float m4[kNB];
#pragma unroll
    for (int i = 0; i < kNB; ++i) m4[i] = max3f(max3f(v[i].x, v[i].y, v[i].z), v[i].w, -INFINITY);
#pragma unroll
    for (int w = 1; w < kNB; w *= 2)
#pragma unroll
      for (int i = 0; i + w < kNB; i += 2 * w) m4[i] = fmaxf(m4[i], m4[i + w]);
    return m4[0];
  };
  // Push this warp's partial (the same in all its lanes) into every CTA of the
  // cluster, then wait for the cluster's partials; returns the slot to read.
  // Every CTA of the cluster makes the same exchanges in the same order.
  auto exchange = [&](float f0, float f1, int i0) -> const Part* {
    const int slot = xs & 1;
    const uint32_t parity = (uint32_t)((xs >> 1) & 1);
    ++xs;
    if (tid == 0) mbar_arrive_expect_tx(&sh.xbar[slot], (uint32_t)(nparts * (int)sizeof(Part)));
    if (lane < csize)
      st_async_v4(map_to_rank(smem_u32(&sh.xch[slot][rank * kWarps + warp]), (uint32_t)lane), f0, f1, i0, 0,
                  map_to_rank(smem_u32(&sh.xbar[slot]), (uint32_t)lane));
    if (!mbar_wait_cluster_bounded(&sh.xbar[slot], parity) && lane == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
    return sh.xch[slot];
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

  for (int b = (int)(blockIdx.x / (unsigned)csize); b < p.batch; b += nclusters) {
    const float* lrow = p.logits + (int64_t)b * R * V + x0;  // position j at lrow + j V
    // ---- row validation (identical in every CTA of the cluster): the mode, the
    // temperature and the drafts (lane j holds d_j, k <= 31) are loaded first,
    // then position 0's first batch (read whatever the row holds), all in flight
    // during the validation.
    const int md = p.mode[b];
    const float t_row = p.temperature[b];
    const int d_lane = lane < k ? p.drafts[(int64_t)b * k + lane] : 0;
    float4 v[kNB];
    load_batch(lrow, 0, v);
    const bool token_bad = __any_sync(0xffffffffu, lane < k && (d_lane < 0 || d_lane >= V));
    bool valid = md == SPEC_MODE_GREEDY || md == SPEC_MODE_SAMPLE;
    int32_t err_bit = valid ? 0 : SPEC_DEVERR_MODE;
    if (token_bad) { valid = false; err_bit |= SPEC_DEVERR_TOKEN; }
    float T_ = 1.f;
    if (valid && md == SPEC_MODE_SAMPLE) {
      T_ = t_row;
      if (!(T_ > 0.f) || !isfinite(T_)) { valid = false; err_bit |= SPEC_DEVERR_TEMPERATURE; }
    }
    if (!valid) {  // uniform across the cluster: no exchange for this row
      if (rank == 0 && tid == 0) {
        raise_error(p.dev_err, err_bit);
        for (int j = 0; j < R; ++j) p.out_tokens[(int64_t)b * R + j] = -1;
        p.accept_len[b] = -1;
      }
      continue;
    }
    const bool greedy = md == SPEC_MODE_GREEDY;
    // Lane j of every warp holds draft j, its target logit, its draft
    // probability and the uniform of its test; decisions read them by shuffle.
    // They are first used at position 0's decision, so their loads arrive while
    // the slice streams in. Without draft probabilities the draft distribution
    // is one-hot at the drafted token.
    float l_d = 0.f, q_d = 1.f, u_d = 0.f;
    if (lane < k && !greedy) {
      l_d = __ldg(p.logits + ((int64_t)b * R + lane) * V + d_lane);
      if (p.probs) q_d = __ldg(p.probs + ((int64_t)b * k + lane) * V + d_lane);
      // the uniform of draft j's test, off the chain of decisions
      u_d = word_to_uniform(philox4x32_10(0u, (uint32_t)lane, (uint32_t)b, 0u, p.seed_lo, p.seed_hi).v[0]);
    }
    const float c2 = (1.0f / T_) * 1.4426950408889634f;  // logit -> log2 units of p
    if (!joined) {
      cluster_wait();  // every CTA of the cluster is running (see cluster_arrive_relaxed)
      joined = true;
    }

    // Write the row's result (one warp, lane j writes position j): accepted
    // drafts, the final token, -1 padding.
    auto write_row = [&](int m, int token) {
      if (lane < R) p.out_tokens[(int64_t)b * R + lane] = lane < m ? d_lane : (lane == m ? token : -1);
      if (lane == 0) p.accept_len[b] = m;
    };

    // Exponential race at position `pos` over the slice, with weights
    //   kRaceResidual: w = max(0, exp2((l - M) c2) * invZ - q)
    //   kRaceOneHot:   the same with q one-hot at the rejected draft
    //   kRacePlain:    w = exp2((l - M) c2)   (the scale does not matter to the race)
    // Returns the winning index (the same in every CTA), or -1 if every weight is 0.
    auto race = [&](auto kind, float M, float invZ, const float* qrow, int pos) -> int {
      constexpr int kKind = decltype(kind)::value;
      const float* src = lrow + (int64_t)pos * V;
      const uint32_t cbase = (uint32_t)x0 >> 2;
      const float mc2 = M * c2;
      const int dpos = __shfl_sync(0xffffffffu, d_lane, pos);  // the rejected draft (one-hot q)
      float thr = 0.f;  // the warp's largest key lower bound so far (the same in all lanes)
      float best = -1.f;
      int bx = INT32_MAX;
      // One iteration: the thread's groups gb + i T + tid, i < kRB. Iterations
      // that lie wholly inside an aligned slice load without checks.
      auto iteration = [&](auto checked, int gb) {
        float4 l4[kRB], q4[kRB];
#pragma unroll
        for (int i = 0; i < kRB; ++i) {
          const int g = gb + i * T + tid;
          if constexpr (decltype(checked)::value) {
            l4[i] = load4(src, g, -INFINITY);
            q4[i] = kKind == kRaceResidual ? loadq4(qrow, g) : kZero4;
          } else {
            l4[i] = __ldg(reinterpret_cast<const float4*>(src) + g);
            q4[i] = kKind == kRaceResidual ? __ldcs(reinterpret_cast<const float4*>(qrow) + g) : kZero4;
          }
        }
        // the Philox blocks need no data: they are computed while the loads are in flight
        Philox4 r[kRB];
#pragma unroll
        for (int i = 0; i < kRB; ++i)
          r[i] = philox4x32_10(cbase + (uint32_t)(gb + i * T + tid), (uint32_t)pos, (uint32_t)b, 1u, p.seed_lo,
                               p.seed_hi);
        float ub[kRB * 4];
        float lb = thr, ubm = 0.f;
#pragma unroll
        for (int i = 0; i < kRB; ++i) {
          float lbe[4];
          const float lv[4] = {l4[i].x, l4[i].y, l4[i].z, l4[i].w};
          [[maybe_unused]] const float qv[4] = {q4[i].x, q4[i].y, q4[i].z, q4[i].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float pe = fast_exp2(fmaf(lv[e], c2, -mc2));  // 0 past the slice (-inf logit)
            float w;
            if constexpr (kKind == kRaceResidual) {
              w = fmaxf(fmaf(pe, invZ, -qv[e]), 0.f);
            } else if constexpr (kKind == kRaceOneHot) {
              w = pe * invZ;
              if (x0 + 4 * (gb + i * T + tid) + e == dpos) w = fmaxf(w - 1.f, 0.f);
            } else {
              w = pe;
            }
            // the word's top 23 bits j as the float 1 + j 2^-23 in [1, 2): then
            // U = (2j + 1) 2^-24 = f1 - (1 - 2^-24) and 1 - U are exact subtractions
            const float f1 = __uint_as_float(0x3F800000u + (r[i].v[e] >> 9));
            const float u = f1 - 0.999999940395355224609375f;
            const float ube = w * fast_rcp(1.f - u);
            ub[4 * i + e] = ube;
            lbe[e] = ube * u;
          }
          lb = max3f(lb, max3f(lbe[0], lbe[1], lbe[2]), lbe[3]);
          ubm = max3f(ubm, max3f(ub[4 * i], ub[4 * i + 1], ub[4 * i + 2]), ub[4 * i + 3]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lb = fmaxf(lb, __shfl_xor_sync(0xffffffffu, lb, o));
        thr = lb;
        // exact keys for the entries whose upper bound reaches the warp's bound
        // (rare: most iterations of most threads have none)
        if (ubm > 0.f && ubm >= thr) {
#pragma unroll
          for (int i = 0; i < kRB; ++i) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float ube = ub[4 * i + e];
              if (ube > 0.f && ube >= thr) {
                const float u = word_to_uniform(r[i].v[e]);
                const float key = (ube * (1.f - u)) / -logf(u);
                if (key > best) {  // entries are visited in increasing x: ties keep the lower index
                  best = key;
                  bx = x0 + 4 * (gb + i * T + tid) + e;
                }
              }
            }
          }
        }
      };
      int gb = 0;
      if (vec)
        for (; gb + kRStep <= ngroups; gb += kRStep) iteration(Flag<false>{}, gb);
      for (; gb < ngroups; gb += kRStep) iteration(Flag<true>{}, gb);  // uniform: every lane shuffles
      warp_best(best, bx);
      const Part* xp = exchange(best, 0.f, bx);
      float kv;
      int win;
      row_best(xp, kv, win);
      return kv > 0.f ? win : -1;
    };

    bool prefetched = false;  // v holds position j's first batch already
    for (int j = 0; j <= k; ++j) {
      const float* src = lrow + (int64_t)j * V;
      if (j > 0 && !prefetched) load_batch(src, 0, v);
      prefetched = false;
      if (greedy) {
        // ---- argmax of the slice (lowest index on ties), then of the row. The
        // thread visits its entries in increasing index order; a batch whose
        // maximum beats the best so far is searched for the first entry holding
        // it (rare after the first batches), so equal values keep the lowest index.
        float bv = -INFINITY;
        int idx = tid < ngroups ? x0 + 4 * tid : INT32_MAX;
        for (int gb = 0;;) {
          const float bm = batch_max(v);
          if (bm > bv) {
            bv = bm;
            // the first entry holding the maximum: selects in reverse order, the last one wins
#pragma unroll
            for (int i = kNB - 1; i >= 0; --i) {
              const float lv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
              for (int e = 3; e >= 0; --e)
                if (lv[e] == bm) idx = x0 + 4 * (gb + i * T + tid) + e;
            }
          }
          gb += kStep;
          if (gb >= ngroups) break;
          load_batch(src, gb, v);
        }
        if (p.prefetch && j < k) {  // position j + 1's first batch, in flight while j is decided
          load_batch(src + V, 0, v);
          prefetched = true;
        }
        warp_best(bv, idx);
        const Part* x = exchange(bv, 0.f, idx);
        float rv;
        int ri;
        row_best(x, rv, ri);
        if (j < k && __shfl_sync(0xffffffffu, d_lane, j) == ri) continue;
        if (rank == 0 && warp == 0) write_row(j, ri);
        break;
      }
      // ---- sampling: max and sum of exp2((l - max) c2) of the slice in one
      // pass. Per batch: its maximum first, then at most one rescale of the
      // running sums, then one exponential per logit into four running sums.
      float m = -INFINITY, s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      for (int gb = 0;;) {
        const float bm = batch_max(v);
        if (bm > m) {
          if (m != -INFINITY) {
            const float rs = fast_exp2((m - bm) * c2);
            s0 *= rs;
            s1 *= rs;
            s2 *= rs;
            s3 *= rs;
          }
          m = bm;
        }
        if (m != -INFINITY) {
          const float mc = m * c2;
#pragma unroll
          for (int i = 0; i < kNB; ++i) {
            s0 += fast_exp2(fmaf(v[i].x, c2, -mc));
            s1 += fast_exp2(fmaf(v[i].y, c2, -mc));
            s2 += fast_exp2(fmaf(v[i].z, c2, -mc));
            s3 += fast_exp2(fmaf(v[i].w, c2, -mc));
          }
        }
        gb += kStep;
        if (gb >= ngroups) break;
        load_batch(src, gb, v);
      }
      if (p.prefetch && j < k) {  // position j + 1's first batch, in flight while j is decided
        load_batch(src + V, 0, v);
        prefetched = true;
      }
      float s = (s0 + s1) + (s2 + s3);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
        ms_combine(m, s, om, os, c2);
      }
      const Part* x = exchange(m, s, 0);
      // softmax statistics of the whole row from the exchanged (max, sum) partials
      float M = -INFINITY, Z = 0.f;
      for (int i = lane; i < nparts; i += 32) ms_combine(M, Z, x[i].f0, x[i].f1, c2);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, M, o), os = __shfl_xor_sync(0xffffffffu, Z, o);
        ms_combine(M, Z, om, os, c2);
      }
      int token;
      if (j < k) {
        const float pd = fast_exp2((__shfl_sync(0xffffffffu, l_d, j) - M) * c2) / Z;
        const float qd = __shfl_sync(0xffffffffu, q_d, j);
        const float u = __shfl_sync(0xffffffffu, u_d, j);
        if (u * qd < pd) continue;
        // ---- rejected at j: race over max(0, p_j - q_j), or over p_j if that is all zero
        if (p.probs)
          token = race(RaceKind<kRaceResidual>{}, M, 1.f / Z, p.probs + ((int64_t)b * k + j) * V + x0, j);
        else
          token = race(RaceKind<kRaceOneHot>{}, M, 1.f / Z, nullptr, j);
        if (token < 0) token = race(RaceKind<kRacePlain>{}, M, 1.f, nullptr, j);  // all-zero residual (rare)
      } else {
        // ---- every draft accepted: bonus token from p_k
        token = race(RaceKind<kRacePlain>{}, M, 1.f, nullptr, k);
      }
      if (rank == 0 && warp == 0) write_row(j, token);
      break;
    }
  }
  if (!joined) cluster_wait();
  // No cluster barrier at the end: every push into this CTA belongs to an
  // exchange it has waited for, and nothing after the last one reads or writes
  // another CTA's memory.
}

// ---------------------------------------------------------------------------
// Launch configuration
// ---------------------------------------------------------------------------

struct Config {
  int threads = 0, csize = 0, slice = 0, clusters = 0;
};

constexpr int kNumCsizes = 5;  // cluster sizes 1, 2, 4, 8, 16

// Clusters of `csize` CTAs of T threads the device can hold at once, from the
// occupancy query (0: none), worked out once per device under the caller's lock.
template <int T>
static int resident_clusters(int dev, int li) {
  static int memo[kMaxDevices][kNumCsizes];  // 0: not asked yet; -1: none
  static bool attrs_set[kMaxDevices];
  auto kern = accept_kernel<T>;
  if (!attrs_set[dev]) {
    // 16-CTA clusters are beyond the portable size
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    attrs_set[dev] = true;
  }
  if (memo[dev][li] == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1u << li;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(1u << li, 1, 1);
    cfg.blockDim = dim3(T, 1, 1);
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, kern, &cfg) != cudaSuccess || c <= 0) {
      (void)cudaGetLastError();
      c = -1;
    }
    memo[dev][li] = c;
  }
  return memo[dev][li] > 0 ? memo[dev][li] : 0;
}

// Threads per CTA and cluster size. Among the configurations whose slices give
// every thread at least one float4 group (and the one-CTA clusters), prefer
// those that hold every row of the batch at once, and among them the fewest
// groups per thread and position (the shortest chain per row); at equal
// threads per row, 128-thread CTAs (finer placement over the SMs) unless they
// need 16-CTA clusters (the cluster barrier and exchange grow with the
// cluster), then the smallest cluster. Measured: serving128 49.6 us with 8 x
// 128 against 52.1 with 4 x 256; hybrid_gdn 57.0 with 8 x 256 against 57.7
// with 16 x 128. When none holds the batch, the one closest to 32 groups per
// thread (each cluster walks several rows). SPEC_ACCEPT_CONFIG="TxC" (T in
// {128, 256}, C a power of two <= 16) forces one.
static bool choose_config(int dev, int batch, int vocab, Config& out) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int force_t = 0, force_c = 0;
  if (const char* env = getenv("SPEC_ACCEPT_CONFIG")) {
    if (sscanf(env, "%dx%d", &force_t, &force_c) != 2) force_t = force_c = 0;
  }
  bool have = false;
  long best_score = 0;
  for (int ti = 0; ti < 2; ++ti) {
    const int T = ti == 0 ? 256 : 128;
    for (int li = kNumCsizes - 1; li >= 0; --li) {
      const int c = 1 << li;
      int slice = (vocab + c - 1) / c;
      slice = (slice + 3) & ~3;
      if ((vocab + slice - 1) / slice != c) continue;  // a CTA would own no logit
      if (c > 1 && slice < 4 * T) continue;
      if (force_t != 0 && (T != force_t || c != force_c)) continue;
      const int clusters = T == 256 ? resident_clusters<256>(dev, li) : resident_clusters<128>(dev, li);
      if (clusters == 0) continue;
      const long groups = ((slice / 4) + T - 1) / T;  // float4 groups per thread and position
      const bool fits = clusters >= batch;
      const long dist = groups > 32 ? groups - 32 : 32 - groups;
      const bool preferred = T == 128 ? c <= 8 : 2 * c > 8;  // see above
      const long score = fits ? groups * 1024 + (preferred ? 0 : 512) + li * 2 + (T == 256 ? 0 : 1)
                              : (1L << 40) + ((dist * 64 + li) * 2 + (T == 128 ? 0 : 1));
      if (!have || score < best_score) {
        have = true;
        best_score = score;
        out.threads = T;
        out.csize = c;
        out.slice = slice;
        out.clusters = clusters;
      }
    }
  }
  return have;
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
  if (k_draft > acc::kMaxK || vocab > acc::kMaxVocab) return SPEC_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int dev = current_device();
  if (dev < 0) return SPEC_ERR_LAUNCH;
  acc::Config c;
  if (!acc::choose_config(dev, batch, vocab, c)) return SPEC_ERR_LAUNCH;

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
  p.slice = c.slice;
  p.csize = c.csize;
  const bool aligned = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(target_logits) & 15) == 0) &&
                       (draft_probs == nullptr || (reinterpret_cast<uintptr_t>(draft_probs) & 15) == 0);
  p.vec = aligned ? 1 : 0;
  // Fetching the next position's first batch before a decision saves a rejected
  // row nothing and an accepting row one load round trip. Where every row's
  // position reads are small (at most 32 MB per position over the batch) the
  // extra reads are free and accepting rows gain; on larger batches they
  // compete with the rows that race after rejecting at position 0.
  p.prefetch = (int64_t)batch * vocab * 4 <= acc::kPrefetchMaxBytes ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)c.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int clusters = batch < c.clusters ? batch : c.clusters;
  cfg.gridDim = dim3((unsigned)(clusters * c.csize), 1, 1);
  cfg.blockDim = dim3((unsigned)c.threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  const cudaError_t e = c.threads == 256 ? cudaLaunchKernelEx(&cfg, acc::accept_kernel<256>, p)
                                         : cudaLaunchKernelEx(&cfg, acc::accept_kernel<128>, p);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}
