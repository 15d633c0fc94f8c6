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
// the vocabulary into contiguous slices of at most 16K logits (<= 16 CTAs).
// Positions are processed in order and the row stops at the first rejection,
// so logits past it are never read (early exit). For each position every CTA
// pulls its slice into shared memory with one bulk asynchronous copy (TMA,
// mbarrier completion) while the next position's slice is prefetched into L2,
// reduces it (max / sum of exp / argmax) with warp shuffles, and publishes a
// partial that every CTA of the cluster reads through distributed shared
// memory, in rank order, so all CTAs reach bit-identical decisions without
// any global-memory round trip. The correction / bonus token is an
// exponential race over the slice already in shared memory, with Philox
// uniforms generated on the fly.
#include <math.h>

#include "common.cuh"

namespace specv {
namespace acc {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kSliceTarget = 16384;  // logits per CTA (64 KB of shared memory)
constexpr int kMaxSlice = 48 * 1024;
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
  int batch, k, vocab, slice, csize;
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
  Part pos[kMaxK + 1];
  Part race[2];
  float wf[kWarps];
  float wg[kWarps];
  int32_t wi[kWarps];
  int32_t bcast_i[4];
  float bcast_f[4];
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

__global__ void __launch_bounds__(kThreads) accept_kernel(const Params p) {
  extern __shared__ __align__(128) float buf[];
  __shared__ Shared sh;
  const int tid = threadIdx.x;
  const int csize = p.csize;
  const int rank = (int)cluster_ctarank();
  const int b = blockIdx.x / csize;
  const int k = p.k, R = k + 1, V = p.vocab;
  const int x0 = rank * p.slice;
  const int n = min(p.slice, V - x0);  // >= 1 by construction of csize
  const int32_t* d = p.drafts + (int64_t)b * k;

  // ---- row validation (identical in every CTA of the cluster)
  const int md = p.mode[b];
  bool valid = (md == SPEC_MODE_GREEDY) || (md == SPEC_MODE_SAMPLE && p.probs != nullptr);
  int32_t err_bit = valid ? 0 : SPEC_DEVERR_MODE;
  for (int j = 0; j < k; ++j) {
    const int dj = d[j];
    if (dj < 0 || dj >= V) { valid = false; err_bit |= SPEC_DEVERR_TOKEN; }
  }
  float T = 1.f;
  if (valid && md == SPEC_MODE_SAMPLE) {
    T = p.temperature[b];
    if (!(T > 0.f) || !isfinite(T)) { valid = false; err_bit |= SPEC_DEVERR_TEMPERATURE; }
  }
  if (!valid) {
    if (rank == 0 && tid == 0) {
      raise_error(p.dev_err, err_bit);
      for (int j = 0; j < R; ++j) p.out_tokens[(int64_t)b * R + j] = -1;
      p.accept_len[b] = -1;
    }
    return;  // uniform across the cluster: no CTA touches another's shared memory
  }
  const bool greedy = md == SPEC_MODE_GREEDY;
  const float c2 = (1.0f / T) * 1.4426950408889634f;  // logit -> log2 units of p
  const uint32_t sh_pos = smem_u32(&sh.pos[0]);
  const uint32_t sh_race = smem_u32(&sh.race[0]);

  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  bool bulk = p.bulk != 0;
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
    __syncthreads();
  };

  int m = k;
  int token = -1;
  issue_row(0);
  for (int j = 0; j <= k; ++j) {
    wait_row();
    // L2 prefetch needs the same 16-byte alignment as the bulk copies
    if (p.prefetch && bulk && tid == 0 && j < k) {
      bulk_prefetch_l2(row_ptr(j + 1), (uint32_t)n * 4u);
      if (!greedy) bulk_prefetch_l2(p.probs + ((int64_t)b * k + j) * V + x0, (uint32_t)n * 4u);
    }
    if (greedy) {
      // ---- argmax of the slice, then of the cluster (ranks are in vocab order)
      float v = -INFINITY;
      int idx = INT32_MAX;
      for (int x = tid; x < n; x += kThreads) {
        const float l = buf[x];
        if (l > v) { v = l; idx = x0 + x; }
      }
      block_argmax(sh, v, idx);
      if (tid == 0) sh.pos[j] = Part{v, 0.f, idx, 0};
      cluster_sync_all();
      float bv = -INFINITY;
      int bi = INT32_MAX;
      for (int r = 0; r < csize; ++r) {
        const uint32_t a = map_to_rank(sh_pos + j * sizeof(Part), (uint32_t)r);
        const float ov = ld_cluster_f32(a);
        const int oi = ld_cluster_s32(a + 8);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (j < k && d[j] == bi) {
        issue_row(j + 1);
        continue;
      }
      m = j;
      token = bi;
      break;
    }
    if (j == k) {
      // ---- every draft accepted: bonus token from p_k by exponential race,
      // compared in log2 units (log2 p - log2 E) so no normaliser is needed.
      float best = -INFINITY;
      int bidx = INT32_MAX;
      for (int g4 = tid; g4 * 4 < n; g4 += kThreads) {
        const int gx = x0 + g4 * 4;
        const Philox4 w = philox4x32_10((uint32_t)(gx >> 2), (uint32_t)k, (uint32_t)b, 1u, p.seed_lo, p.seed_hi);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int x = g4 * 4 + e;
          if (x < n) {
            const float E = -logf(word_to_uniform(w.v[e]));
            const float key = buf[x] * c2 - log2f(E);
            if (key > best) { best = key; bidx = x0 + x; }
          }
        }
      }
      block_argmax(sh, best, bidx);
      if (tid == 0) sh.race[0] = Part{best, 0.f, bidx, 0};
      cluster_sync_all();
      float bv = -INFINITY;
      int bi = INT32_MAX;
      for (int r = 0; r < csize; ++r) {
        const uint32_t a = map_to_rank(sh_race, (uint32_t)r);
        const float ov = ld_cluster_f32(a);
        const int oi = ld_cluster_s32(a + 8);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      m = k;
      token = bi;
      break;
    }
    // ---- sampling statistics of p_j = softmax(l / T): slice max, then sum of exp
    float mx = -INFINITY;
    for (int x = tid; x < n; x += kThreads) mx = fmaxf(mx, buf[x]);
    mx = block_max(sh, mx);
    float z = 0.f;
    for (int x = tid; x < n; x += kThreads) z += exp2f((buf[x] - mx) * c2);
    z = block_sum(sh, z);
    if (tid == 0) sh.pos[j] = Part{mx, z, 0, 0};
    cluster_sync_all();
    float M = -INFINITY;
    for (int r = 0; r < csize; ++r) M = fmaxf(M, ld_cluster_f32(map_to_rank(sh_pos + j * sizeof(Part), (uint32_t)r)));
    float Z = 0.f;
    for (int r = 0; r < csize; ++r) {
      const uint32_t a = map_to_rank(sh_pos + j * sizeof(Part), (uint32_t)r);
      Z += ld_cluster_f32(a + 4) * exp2f((ld_cluster_f32(a) - M) * c2);
    }
    const int dj = d[j];
    const float pd = exp2f((p.logits[((int64_t)b * R + j) * V + dj] - M) * c2) / Z;
    const float qd = p.probs[((int64_t)b * k + j) * V + dj];
    const Philox4 wu = philox4x32_10(0u, (uint32_t)j, (uint32_t)b, 0u, p.seed_lo, p.seed_hi);
    const float u = word_to_uniform(wu.v[0]);
    if (u * qd < pd) {
      issue_row(j + 1);
      continue;
    }
    // ---- rejected at j: race over max(0, p_j - q_j) (falls back to p_j if all zero)
    m = j;
    const float invZ = 1.f / Z;
    const float* qrow = p.probs + ((int64_t)b * k + j) * V + x0;
    for (int pass = 0; pass < 2; ++pass) {
      float best = -1.f, wsum = 0.f;
      int bidx = INT32_MAX;
      for (int g4 = tid; g4 * 4 < n; g4 += kThreads) {
        const int gx = x0 + g4 * 4;
        float qv[4];
        if (p.bulk && g4 * 4 + 3 < n) {
          const float4 q4 = __ldg(reinterpret_cast<const float4*>(qrow + g4 * 4));
          qv[0] = q4.x; qv[1] = q4.y; qv[2] = q4.z; qv[3] = q4.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) qv[e] = (g4 * 4 + e < n) ? qrow[g4 * 4 + e] : 0.f;
        }
        const Philox4 w = philox4x32_10((uint32_t)(gx >> 2), (uint32_t)j, (uint32_t)b, 1u, p.seed_lo, p.seed_hi);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int x = g4 * 4 + e;
          if (x < n) {
            const float px = exp2f((buf[x] - M) * c2) * invZ;
            const float wt = pass == 0 ? fmaxf(px - qv[e], 0.f) : px;
            wsum += wt;
            const float E = -logf(word_to_uniform(w.v[e]));
            const float key = wt / E;
            if (key > best) { best = key; bidx = x0 + x; }
          }
        }
      }
      block_argmax(sh, best, bidx);
      wsum = block_sum(sh, wsum);
      if (tid == 0) sh.race[pass] = Part{best, wsum, bidx, 0};
      cluster_sync_all();
      float bv = -1.f, total = 0.f;
      int bi = INT32_MAX;
      for (int r = 0; r < csize; ++r) {
        const uint32_t a = map_to_rank(sh_race + pass * sizeof(Part), (uint32_t)r);
        const float ov = ld_cluster_f32(a);
        total += ld_cluster_f32(a + 4);
        const int oi = ld_cluster_s32(a + 8);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      token = bi;
      if (total > 0.f) break;  // identical in every CTA: the same partials, the same order
    }
    break;
  }

  if (pending) {  // an issued copy must land before this CTA's shared memory goes away
    if (!mbar_wait_bounded(&sh.bar, phase) && tid == 0) raise_error(p.dev_err, SPEC_DEVERR_TIMEOUT);
  }
  if (rank == 0 && tid == 0) {
    int32_t* o = p.out_tokens + (int64_t)b * R;
    for (int j = 0; j < m; ++j) o[j] = d[j];
    o[m] = token;
    for (int j = m + 1; j < R; ++j) o[j] = -1;
    p.accept_len[b] = m;
  }
  cluster_sync_all();  // peers may still be reading this CTA's partials
}

static int pick_cluster(int vocab, int& slice) {
  int c = (vocab + kSliceTarget - 1) / kSliceTarget;
  if (c < 1) c = 1;
  if (c > kMaxCluster) c = kMaxCluster;
  slice = (vocab + c - 1) / c;
  slice = (slice + 3) & ~3;
  c = (vocab + slice - 1) / slice;  // every CTA owns at least one logit
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
  int slice = 0;
  const int csize = acc::pick_cluster(vocab, slice);
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
  p.prefetch = 1;

  auto kern = acc::accept_kernel;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  // Clusters larger than 8 CTAs are not guaranteed to fit a GPC; if the device
  // cannot hold one, use 8 CTAs with larger slices.
  for (int attempt = 0; attempt < 2; ++attempt) {
    const size_t smem = (size_t)p.slice * sizeof(float);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SPEC_ERR_LAUNCH;
    if (p.csize > 8 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return SPEC_ERR_LAUNCH;
    cfg.gridDim = dim3((unsigned)(batch * p.csize), 1, 1);
    cfg.blockDim = dim3(acc::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.csize <= 8) break;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0) break;
    (void)cudaGetLastError();
    p.csize = 8;
    p.slice = (((vocab + 7) / 8) + 3) & ~3;
    if (p.slice > acc::kMaxSlice) return SPEC_ERR_UNSUPPORTED;
  }
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return SPEC_ERR_LAUNCH;
  return SPEC_OK;
}
