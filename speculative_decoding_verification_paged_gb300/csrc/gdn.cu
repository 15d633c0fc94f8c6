// Gated delta rule over the verify chain (sm_103a): the producer of the
// recurrent-state checkpoints that the commit kernels keep or stage.
//
// The hybrid models interleave attention with GatedDeltaNet layers whose
// operators publish the state after every token of a speculative step
// (onnxruntime-genai PR #2457: GatedDeltaNet.checkpoints, V-major float32
// state, a W-slot window written at slot j after token j or with slot W-1
// after the last token; lmdeploy PR #5019: "GDR verify" kernels). The update
// is the published Gated DeltaNet rule (Yang, Kautz, Hatamizadeh, "Gated Delta
// Networks: Improving Mamba2 with Delta Rule"): per (row b, head h), with the
// state S stored V-major (S[i][c], value index i, key index c),
//
//   a_t = exp(g_t),  S_t = a_t S_{t-1} + beta_t (v_t - a_t S_{t-1} k_t) k_t^T,
//   o_t = S_t (scale q_t) = a_t S_{t-1} q'_t + beta_t u_t (k_t . q'_t).
//
// Design (GB300): the step is bound by HBM (read one dv x dk fp32 state,
// write R of them), so one 256-thread CTA owns one (b, h) state and two CTAs
// share an SM. For 128 x 128 states the state lives in registers: warp w owns
// value rows [16w, 16w+16), lane l the float4 column group l, so a row is one
// coalesced 512-byte access per warp. Per token, every lane forms the 32
// partial dot products of its rows with k_t and q'_t, and a recursive-halving
// exchange (16 + 8 + 4 + 2 + 1 shuffles) leaves lane l with complete sum l:
// S k for rows l < 16, S q' for rows l - 16. The delta term u goes through
// shared memory to the whole warp, the rank-one update runs in registers and
// the checkpoint is written with streaming float4 stores. Other sizes take a
// plain shared-memory path.
#include <math.h>

#include "common.cuh"
#include "launch_memo.h"

namespace specv {
namespace gdn {

constexpr int kThreads = 256;  // 8 warps x 16 value rows = 128 rows
constexpr int kMaxTokens = 32;
constexpr int kFastDim = 128;  // dk = dv = 128: state in registers

struct Params {
  const float* q;          // [B,R,H,dk]
  const float* k;          // [B,R,H,dk]
  const float* v;          // [B,R,H,dv]
  const float* g;          // [B,R,H] log decay
  const float* beta;       // [B,R,H]
  float scale;             // applied to q
  const float* state_in;   // contiguous: [B, H*dv*dk]
  float* snapshots;        // contiguous: [B, W, H*dv*dk]
  float* pool;             // pooled: rows of H*dv*dk floats
  const int32_t* live_row; // pooled: [B]
  const int32_t* ckpt_rows;// pooled: [B, W]
  int64_t pool_rows;
  float* out;              // [B,R,H,dv]
  int batch, tokens, heads, dk, dv, slots, base;
  int32_t* dev_err;
};

// Where unit (b, h) reads its state and writes checkpoint t (offsets of the
// head inside a row of H*dv*dk floats are added by the caller). Returns false
// (and flags it) when a pool index lies outside the pool.
__device__ __forceinline__ bool locate(const Params& p, int b, const float*& src, int64_t& row_elems) {
  row_elems = (int64_t)p.heads * p.dv * p.dk;
  if (p.live_row == nullptr) {
    src = p.state_in + (int64_t)b * row_elems;
    return true;
  }
  const int64_t lr = p.live_row[b];
  bool ok = lr >= 0 && lr < p.pool_rows;
  for (int t = 0; t < p.tokens; ++t) {
    const int64_t cr = p.ckpt_rows[(int64_t)b * p.slots + p.base + t];
    ok = ok && cr >= 0 && cr < p.pool_rows;
  }
  src = p.pool + (ok ? lr : 0) * row_elems;
  return ok;
}

__device__ __forceinline__ float* checkpoint(const Params& p, int b, int t, int64_t row_elems) {
  if (p.live_row == nullptr) return p.snapshots + ((int64_t)b * p.slots + p.base + t) * row_elems;
  return p.pool + (int64_t)p.ckpt_rows[(int64_t)b * p.slots + p.base + t] * row_elems;
}

// Recursive halving over a warp: on entry every lane holds 32 partial values;
// on exit lane l holds the warp-wide sum of value l. At each step a lane keeps
// the half of its values that its lane bit selects and adds the partner's copy
// of that half.
template <int kHalf>
__device__ __forceinline__ void halve(float (&x)[32], int lane) {
  const bool up = (lane & kHalf) != 0;
#pragma unroll
  for (int j = 0; j < kHalf; ++j) {
    const float send = up ? x[j] : x[kHalf + j];
    const float keep = up ? x[kHalf + j] : x[j];
    x[j] = keep + __shfl_xor_sync(0xffffffffu, send, kHalf);
  }
}

__global__ void __launch_bounds__(kThreads, 2) gdn_verify_fast_kernel(const Params p) {
  extern __shared__ __align__(16) float smem[];
  __shared__ __align__(16) float su[kFastDim];
  __shared__ float s_alpha[kMaxTokens], s_beta[kMaxTokens];
  __shared__ int s_ok;
  const int R = p.tokens, H = p.heads;
  float* sq = smem;                  // [R][128] scale * q
  float* sk = sq + R * kFastDim;     // [R][128]
  float* sv = sk + R * kFastDim;     // [R][128]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int64_t head_off = (int64_t)h * kFastDim * kFastDim;

  const float* src = nullptr;
  int64_t row_elems = 0;
  const bool ok = locate(p, b, src, row_elems);
  if (tid == 0) s_ok = ok;
  for (int x = tid; x < R * kFastDim; x += kThreads) {
    const int t = x / kFastDim, c = x % kFastDim;
    const int64_t tok = ((int64_t)b * R + t) * H + h;
    sq[x] = p.scale * p.q[tok * kFastDim + c];
    sk[x] = p.k[tok * kFastDim + c];
    sv[x] = p.v[tok * kFastDim + c];
  }
  if (tid < R) {
    const int64_t tok = ((int64_t)b * R + tid) * H + h;
    s_alpha[tid] = expf(p.g[tok]);
    s_beta[tid] = p.beta[tok];
  }
  __syncthreads();
  if (!s_ok) {  // a pool index out of range: zero outputs, no state touched
    if (tid == 0 && h == 0) raise_error(p.dev_err, SPEC_DEVERR_POOL_ROW);
    for (int x = tid; x < R * kFastDim; x += kThreads) {
      const int t = x / kFastDim, i = x % kFastDim;
      p.out[(((int64_t)b * R + t) * H + h) * kFastDim + i] = 0.f;
    }
    return;
  }

  const int row0 = warp * 16;
  float4 S[16];
  {
    const float4* s4 = reinterpret_cast<const float4*>(src + head_off);
#pragma unroll
    for (int r = 0; r < 16; ++r) S[r] = __ldcs(s4 + (row0 + r) * (kFastDim / 4) + lane);
  }
  for (int t = 0; t < R; ++t) {
    const float4 k4 = reinterpret_cast<const float4*>(sk + t * kFastDim)[lane];
    const float4 q4 = reinterpret_cast<const float4*>(sq + t * kFastDim)[lane];
    const float alpha = s_alpha[t], bt = s_beta[t];
    float x[32];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      x[r] = S[r].x * k4.x + S[r].y * k4.y + S[r].z * k4.z + S[r].w * k4.w;
      x[16 + r] = S[r].x * q4.x + S[r].y * q4.y + S[r].z * q4.z + S[r].w * q4.w;
    }
    halve<16>(x, lane);
    halve<8>(x, lane);
    halve<4>(x, lane);
    halve<2>(x, lane);
    halve<1>(x, lane);
    const float sum = x[0];  // lane < 16: (S k)[row0 + lane]; lane >= 16: (S q')[row0 + lane - 16]
    float kq = k4.x * q4.x + k4.y * q4.y + k4.z * q4.z + k4.w * q4.w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
    const float u = sv[t * kFastDim + row0 + (lane & 15)] - alpha * sum;  // used from lanes < 16
    const float u_row = __shfl_sync(0xffffffffu, u, lane & 15);
    if (lane < 16) {
      su[row0 + lane] = u;
    } else {
      const int64_t tok = ((int64_t)b * R + t) * H + h;
      p.out[tok * kFastDim + row0 + lane - 16] = alpha * sum + bt * u_row * kq;
    }
    __syncwarp();
    float ur[16];
#pragma unroll
    for (int r4 = 0; r4 < 4; ++r4) {
      const float4 w = reinterpret_cast<const float4*>(su + row0)[r4];
      ur[4 * r4] = w.x; ur[4 * r4 + 1] = w.y; ur[4 * r4 + 2] = w.z; ur[4 * r4 + 3] = w.w;
    }
    float4* d4 = reinterpret_cast<float4*>(checkpoint(p, b, t, row_elems) + head_off);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float bu = bt * ur[r];
      S[r].x = fmaf(bu, k4.x, alpha * S[r].x);
      S[r].y = fmaf(bu, k4.y, alpha * S[r].y);
      S[r].z = fmaf(bu, k4.z, alpha * S[r].z);
      S[r].w = fmaf(bu, k4.w, alpha * S[r].w);
      __stcs(d4 + (row0 + r) * (kFastDim / 4) + lane, S[r]);
    }
    __syncwarp();  // su is rewritten by the next token
  }
}

// Any (dk, dv) whose state fits in shared memory: the state is staged there
// and each step is a plain loop over rows or elements.
__global__ void __launch_bounds__(kThreads) gdn_verify_generic_kernel(const Params p) {
  extern __shared__ __align__(16) float smem[];
  __shared__ float s_kq;
  __shared__ int s_ok;
  const int R = p.tokens, H = p.heads, dk = p.dk, dv = p.dv;
  const int64_t E = (int64_t)dv * dk;
  float* S = smem;            // [dv][dk]
  float* sq = S + E;          // [R][dk] scale * q
  float* sk = sq + R * dk;    // [R][dk]
  float* sv = sk + R * dk;    // [R][dv]
  float* sSk = sv + R * dv;   // [dv]
  float* sSq = sSk + dv;      // [dv]
  float* su = sSq + dv;       // [dv]
  const int tid = threadIdx.x;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int64_t head_off = (int64_t)h * E;

  const float* src = nullptr;
  int64_t row_elems = 0;
  const bool ok = locate(p, b, src, row_elems);
  if (tid == 0) s_ok = ok;
  __syncthreads();
  if (!s_ok) {
    if (tid == 0 && h == 0) raise_error(p.dev_err, SPEC_DEVERR_POOL_ROW);
    for (int x = tid; x < R * dv; x += kThreads) {
      const int t = x / dv, i = x % dv;
      p.out[(((int64_t)b * R + t) * H + h) * dv + i] = 0.f;
    }
    return;
  }
  for (int64_t e = tid; e < E; e += kThreads) S[e] = src[head_off + e];
  for (int x = tid; x < R * dk; x += kThreads) {
    const int t = x / dk, c = x % dk;
    const int64_t tok = ((int64_t)b * R + t) * H + h;
    sq[x] = p.scale * p.q[tok * dk + c];
    sk[x] = p.k[tok * dk + c];
  }
  for (int x = tid; x < R * dv; x += kThreads) {
    const int t = x / dv, i = x % dv;
    sv[x] = p.v[(((int64_t)b * R + t) * H + h) * dv + i];
  }
  __syncthreads();
  for (int t = 0; t < R; ++t) {
    const int64_t tok = ((int64_t)b * R + t) * H + h;
    const float alpha = expf(p.g[tok]), bt = p.beta[tok];
    const float* kt = sk + t * dk;
    const float* qt = sq + t * dk;
    for (int i = tid; i < dv; i += kThreads) {
      float a = 0.f, c2 = 0.f;
      for (int c = 0; c < dk; ++c) {
        a = fmaf(S[(int64_t)i * dk + c], kt[c], a);
        c2 = fmaf(S[(int64_t)i * dk + c], qt[c], c2);
      }
      sSk[i] = a;
      sSq[i] = c2;
    }
    if (tid == 0) {
      float kq = 0.f;
      for (int c = 0; c < dk; ++c) kq = fmaf(kt[c], qt[c], kq);
      s_kq = kq;
    }
    __syncthreads();
    for (int i = tid; i < dv; i += kThreads) {
      const float u = sv[t * dv + i] - alpha * sSk[i];
      su[i] = u;
      p.out[tok * dv + i] = alpha * sSq[i] + bt * u * s_kq;
    }
    __syncthreads();
    float* dst = checkpoint(p, b, t, row_elems) + head_off;
    for (int64_t e = tid; e < E; e += kThreads) {
      const int64_t i = e / dk, c = e % dk;
      const float s = fmaf(bt * su[i], kt[c], alpha * S[e]);
      S[e] = s;
      dst[e] = s;
    }
    __syncthreads();
  }
}

static int launch(Params& p, cudaStream_t stream) {
  if (p.batch < 0 || p.tokens < 1 || p.tokens > kMaxTokens || p.heads < 1 || p.dk < 1 || p.dv < 1 ||
      p.slots < p.tokens)
    return SPEC_ERR_INVALID_ARG;
  if (p.batch == 0) return SPEC_OK;
  if (!p.q || !p.k || !p.v || !p.g || !p.beta || !p.out) return SPEC_ERR_INVALID_ARG;
  const int64_t units = (int64_t)p.batch * p.heads;
  if (units > INT32_MAX) return SPEC_ERR_UNSUPPORTED;
  const void* state_base = p.live_row ? static_cast<const void*>(p.pool) : static_cast<const void*>(p.state_in);
  const void* snap_base = p.live_row ? static_cast<const void*>(p.pool) : static_cast<const void*>(p.snapshots);
  const bool aligned = ((reinterpret_cast<uintptr_t>(state_base) | reinterpret_cast<uintptr_t>(snap_base)) & 15) == 0;
  if (p.dk == kFastDim && p.dv == kFastDim && aligned) {
    const size_t smem = (size_t)3 * p.tokens * kFastDim * sizeof(float);
    static LaunchMemo memo;
    if (smem > 48 * 1024) {
      const int dev = current_device();
      std::lock_guard<std::mutex> lock(memo.mu);
      if (dev < 0 || !grant_smem_locked(memo, (const void*)gdn_verify_fast_kernel, dev, smem)) return SPEC_ERR_LAUNCH;
    }
    gdn_verify_fast_kernel<<<(unsigned)units, kThreads, smem, stream>>>(p);
  } else {
    const size_t smem = sizeof(float) * ((size_t)p.dv * p.dk + (size_t)p.tokens * (2 * p.dk + p.dv) + 3 * (size_t)p.dv);
    if (smem > 200 * 1024) return SPEC_ERR_UNSUPPORTED;
    static LaunchMemo memo;
    if (smem > 48 * 1024) {
      const int dev = current_device();
      std::lock_guard<std::mutex> lock(memo.mu);
      if (dev < 0 || !grant_smem_locked(memo, (const void*)gdn_verify_generic_kernel, dev, smem))
        return SPEC_ERR_LAUNCH;
    }
    gdn_verify_generic_kernel<<<(unsigned)units, kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

static Params base_params(const float* q, const float* k, const float* v, const float* g, const float* beta,
                          float scale, float* out, int32_t batch, int32_t num_tokens, int32_t num_heads, int32_t dk,
                          int32_t dv, int32_t num_slots, int32_t alignment, int32_t* dev_err) {
  Params p = {};
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = g;
  p.beta = beta;
  p.scale = scale;
  p.out = out;
  p.batch = batch;
  p.tokens = num_tokens;
  p.heads = num_heads;
  p.dk = dk;
  p.dv = dv;
  p.slots = num_slots;
  p.base = alignment == SPEC_ALIGN_TOKEN ? 0 : num_slots - num_tokens;
  p.dev_err = dev_err;
  return p;
}

}  // namespace gdn
}  // namespace specv

using namespace specv;

extern "C" int spec_gdn_verify(const float* q, const float* k, const float* v, const float* g, const float* beta,
                               float scale, const float* state_in, float* snapshots, float* out, int32_t batch,
                               int32_t num_tokens, int32_t num_heads, int32_t dk, int32_t dv, int32_t num_slots,
                               int32_t alignment, int32_t* dev_err, spec_stream_t stream) {
  if (alignment != SPEC_ALIGN_TOKEN && alignment != SPEC_ALIGN_LAST) return SPEC_ERR_INVALID_ARG;
  gdn::Params p = gdn::base_params(q, k, v, g, beta, scale, out, batch, num_tokens, num_heads, dk, dv, num_slots,
                                   alignment, dev_err);
  if (batch > 0 && (!state_in || !snapshots)) return SPEC_ERR_INVALID_ARG;
  p.state_in = state_in;
  p.snapshots = snapshots;
  return gdn::launch(p, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int spec_gdn_verify_pooled(const float* q, const float* k, const float* v, const float* g,
                                      const float* beta, float scale, float* pool, int64_t pool_rows,
                                      const int32_t* live_row, const int32_t* ckpt_rows, float* out, int32_t batch,
                                      int32_t num_tokens, int32_t num_heads, int32_t dk, int32_t dv,
                                      int32_t num_slots, int32_t alignment, int32_t* dev_err, spec_stream_t stream) {
  if (alignment != SPEC_ALIGN_TOKEN && alignment != SPEC_ALIGN_LAST) return SPEC_ERR_INVALID_ARG;
  if (pool_rows < 1) return SPEC_ERR_INVALID_ARG;
  gdn::Params p = gdn::base_params(q, k, v, g, beta, scale, out, batch, num_tokens, num_heads, dk, dv, num_slots,
                                   alignment, dev_err);
  if (batch > 0 && (!pool || !live_row || !ckpt_rows)) return SPEC_ERR_INVALID_ARG;
  p.pool = pool;
  p.pool_rows = pool_rows;
  p.live_row = live_row;
  p.ckpt_rows = ckpt_rows;
  return gdn::launch(p, reinterpret_cast<cudaStream_t>(stream));
}
