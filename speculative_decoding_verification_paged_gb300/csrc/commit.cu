// Recurrent-state commit (sm_103a).
//
// The gated-delta-net and conv operators publish the state after every verify
// token; rolling back a partly accepted draft only needs the slot of the
// accepted prefix (onnxruntime-genai PR #2457: per-token state checkpoints,
// CommitPrefix; lmdeploy PR #5019 fix 2: CommitAcceptedRecurrentStateKernel
// writes the accepted state back). With fp32 state the commit is a bit-exact
// gather: live[l, b, :] = snapshots[l, b, accept_len[b], :].
//
// Design (GB300): a streaming copy at HBM speed. Each CTA moves one 32 KB
// piece of one (layer, row) state with 16-byte loads, 8 in flight per thread
// before the first store, reading accept_len once; the grid is
// (pieces per state) x (layers * rows), so no division sits in the copy loop.
//
// The same PR notes that a rollback only needs the state pool to stage a
// different source row: spec_commit_select moves no state at all and instead
// exchanges two int32 pool-row indices per (layer, row), the live row and the
// window slot of the accepted prefix.
#include "common.cuh"

namespace specv {
namespace cmt {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 8;
constexpr int kPiece = kThreads * kVecPerThread;  // float4 per CTA

// The kept snapshot of row b is slot base + accept_len[b] of its `slots`-slot
// window; accept_len must lie in [0, n_tokens).
__global__ void __launch_bounds__(kThreads) commit_vec_kernel(const float4* __restrict__ snaps,
                                                              const int32_t* __restrict__ accept_len,
                                                              float4* __restrict__ live, int batch,
                                                              int slots, int base, int n_tokens,
                                                              int64_t vecs_per_state, int32_t* dev_err) {
  const int64_t lb = blockIdx.y;  // layer * batch + row
  const int b = (int)(lb % batch);
  const int a = __ldg(accept_len + b);
  if (a < 0 || a >= n_tokens) {
    if (blockIdx.x == 0 && lb == b && threadIdx.x == 0) raise_error(dev_err, SPEC_DEVERR_ACCEPT_LEN);
    return;
  }
  const float4* src = snaps + (lb * slots + base + a) * vecs_per_state;
  float4* dst = live + lb * vecs_per_state;
  const int64_t start = (int64_t)blockIdx.x * kPiece + threadIdx.x;
  float4 v[kVecPerThread];
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    const int64_t e = start + (int64_t)i * kThreads;
    if (e < vecs_per_state) v[i] = __ldcs(src + e);  // streamed once: evict-first
  }
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    const int64_t e = start + (int64_t)i * kThreads;
    if (e < vecs_per_state) __stcs(dst + e, v[i]);
  }
}

// Any element count or alignment: one float per thread-iteration.
__global__ void __launch_bounds__(kThreads) commit_scalar_kernel(const float* __restrict__ snaps,
                                                                 const int32_t* __restrict__ accept_len,
                                                                 float* __restrict__ live, int batch, int slots,
                                                                 int base, int n_tokens, int64_t elems,
                                                                 int32_t* dev_err) {
  const int64_t lb = blockIdx.y;
  const int b = (int)(lb % batch);
  const int a = __ldg(accept_len + b);
  if (a < 0 || a >= n_tokens) {
    if (blockIdx.x == 0 && lb == b && threadIdx.x == 0) raise_error(dev_err, SPEC_DEVERR_ACCEPT_LEN);
    return;
  }
  const float* src = snaps + (lb * slots + base + a) * elems;
  float* dst = live + lb * elems;
  for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < elems; e += (int64_t)gridDim.x * kThreads)
    dst[e] = src[e];
}

// Zero-copy commit: thread i owns unit i = layer * batch + row and exchanges
// its live-row index with the window slot of the accepted prefix. Units are
// disjoint, so the exchanges need no atomics. For windows of up to
// kWindowRegs slots every entry is loaded together with accept_len, so the
// exchange waits for one round trip to memory instead of two.
constexpr int kWindowRegs = 8;

__global__ void __launch_bounds__(kThreads) commit_select_kernel(const int32_t* __restrict__ accept_len,
                                                                 int32_t* __restrict__ live_row,
                                                                 int32_t* __restrict__ ckpt_rows, int64_t units,
                                                                 int batch, int slots, int base, int n_tokens,
                                                                 int32_t* dev_err) {
  const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (i >= units) return;
  const int b = (int)(i % batch);
  const int a = __ldg(accept_len + b);
  const int32_t live = live_row[i];
  int32_t* win = ckpt_rows + i * slots;
  int32_t entry[kWindowRegs];
#pragma unroll
  for (int s = 0; s < kWindowRegs; ++s) entry[s] = s < slots ? win[s] : 0;
  if (a < 0 || a >= n_tokens) {
    if (i == b) raise_error(dev_err, SPEC_DEVERR_ACCEPT_LEN);  // once per row, from layer 0
    return;
  }
  const int s_keep = base + a;
  int32_t chosen = 0;
  if (slots <= kWindowRegs) {
#pragma unroll
    for (int s = 0; s < kWindowRegs; ++s)
      if (s == s_keep) chosen = entry[s];
  } else {
    chosen = win[s_keep];
  }
  win[s_keep] = live;
  live_row[i] = chosen;
}

}  // namespace cmt
}  // namespace specv

using namespace specv;

namespace specv {
namespace cmt {

static int launch(const float* snapshots, const int32_t* accept_len, float* live_state, int32_t num_layers,
                  int32_t batch, int32_t num_slots, int64_t state_elems, int32_t base, int32_t n_tokens,
                  int32_t* dev_err, cudaStream_t stream) {
  if (num_layers == 0 || batch == 0 || state_elems == 0) return SPEC_OK;
  if (!snapshots || !accept_len || !live_state) return SPEC_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)num_layers * batch;
  if (rows > 65535) return SPEC_ERR_UNSUPPORTED;
  const bool vec = (state_elems % 4 == 0) && ((reinterpret_cast<uintptr_t>(snapshots) & 15) == 0) &&
                   ((reinterpret_cast<uintptr_t>(live_state) & 15) == 0);
  if (vec) {
    const int64_t vecs = state_elems / 4;
    const int64_t pieces = (vecs + kPiece - 1) / kPiece;
    if (pieces > INT32_MAX) return SPEC_ERR_UNSUPPORTED;
    dim3 grid((unsigned)pieces, (unsigned)rows, 1);
    commit_vec_kernel<<<grid, kThreads, 0, stream>>>(reinterpret_cast<const float4*>(snapshots), accept_len,
                                                     reinterpret_cast<float4*>(live_state), batch, num_slots, base,
                                                     n_tokens, vecs, dev_err);
  } else {
    int64_t blocks = (state_elems + kThreads - 1) / kThreads;
    if (blocks > 1024) blocks = 1024;
    dim3 grid((unsigned)blocks, (unsigned)rows, 1);
    commit_scalar_kernel<<<grid, kThreads, 0, stream>>>(snapshots, accept_len, live_state, batch, num_slots, base,
                                                        n_tokens, state_elems, dev_err);
  }
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

}  // namespace cmt
}  // namespace specv

extern "C" int spec_commit_state(const float* snapshots, const int32_t* accept_len, float* live_state,
                                 int32_t num_layers, int32_t batch, int32_t num_slots, int64_t state_elems,
                                 int32_t* dev_err, spec_stream_t stream_) {
  if (num_layers < 0 || batch < 0 || num_slots < 1 || state_elems < 0) return SPEC_ERR_INVALID_ARG;
  return cmt::launch(snapshots, accept_len, live_state, num_layers, batch, num_slots, state_elems, 0, num_slots,
                     dev_err, reinterpret_cast<cudaStream_t>(stream_));
}

extern "C" int spec_commit_state_aligned(const float* snapshots, const int32_t* accept_len, float* live_state,
                                         int32_t num_layers, int32_t batch, int32_t num_slots,
                                         int64_t state_elems, int32_t num_tokens, int32_t alignment,
                                         int32_t* dev_err, spec_stream_t stream_) {
  if (num_layers < 0 || batch < 0 || num_slots < 1 || state_elems < 0) return SPEC_ERR_INVALID_ARG;
  if (num_tokens < 1 || num_tokens > num_slots) return SPEC_ERR_INVALID_ARG;
  if (alignment != SPEC_ALIGN_TOKEN && alignment != SPEC_ALIGN_LAST) return SPEC_ERR_INVALID_ARG;
  const int32_t base = alignment == SPEC_ALIGN_TOKEN ? 0 : num_slots - num_tokens;
  return cmt::launch(snapshots, accept_len, live_state, num_layers, batch, num_slots, state_elems, base, num_tokens,
                     dev_err, reinterpret_cast<cudaStream_t>(stream_));
}

extern "C" int spec_commit_select(const int32_t* accept_len, int32_t* live_row, int32_t* ckpt_rows,
                                  int32_t num_layers, int32_t batch, int32_t num_slots, int32_t num_tokens,
                                  int32_t alignment, int32_t* dev_err, spec_stream_t stream_) {
  if (num_layers < 0 || batch < 0 || num_slots < 1) return SPEC_ERR_INVALID_ARG;
  if (num_tokens < 1 || num_tokens > num_slots) return SPEC_ERR_INVALID_ARG;
  if (alignment != SPEC_ALIGN_TOKEN && alignment != SPEC_ALIGN_LAST) return SPEC_ERR_INVALID_ARG;
  const int64_t units = (int64_t)num_layers * batch;
  if (units == 0) return SPEC_OK;
  if (!accept_len || !live_row || !ckpt_rows) return SPEC_ERR_INVALID_ARG;
  const int64_t blocks = (units + cmt::kThreads - 1) / cmt::kThreads;
  if (blocks > INT32_MAX) return SPEC_ERR_UNSUPPORTED;
  const int32_t base = alignment == SPEC_ALIGN_TOKEN ? 0 : num_slots - num_tokens;
  cmt::commit_select_kernel<<<(unsigned)blocks, cmt::kThreads, 0, reinterpret_cast<cudaStream_t>(stream_)>>>(
      accept_len, live_row, ckpt_rows, units, batch, num_slots, base, num_tokens, dev_err);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

extern "C" const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported shape";
    case SPEC_ERR_LAUNCH: return "kernel launch failed";
    case SPEC_ERR_WORKSPACE: return "workspace missing or too small";
    case SPEC_ERR_SCRATCH_LIMIT: return "shape needs more than the fixed scratch of the allocation-free call";
    default: return "unknown status";
  }
}
