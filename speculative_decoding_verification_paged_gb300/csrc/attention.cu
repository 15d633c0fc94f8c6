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
//  * Head dim 128 with 32 or more packed rows runs on a second kernel, on
//    5th-generation tensor cores (tcgen05, tensor memory): see the comment
//    at the top of attention_tc.cuh. The host picks one per call.
//
// Files: attention_device.cuh (pieces both kernels and the host share),
// attention_mma.cuh (the mma.sync kernel), attention_tc.cuh (the tcgen05
// kernel); this file holds the host side: argument checks, the workspace
// layout, tensor maps, launch settings, kernel choice and the C entry points.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <cuda.h>

#include "attention_device.cuh"
#include "attention_mma.cuh"
#include "attention_tc.cuh"
#include "launch_memo.h"

namespace specv {
namespace attn {

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

// Launch settings of one kernel instance on the current device: raises its
// dynamic shared-memory limit to `smem` (never lowers it) and works out the
// persistent grid, once per (device, shared-memory size), under the instance's
// lock. Every launch of the instance, with or without a caller workspace, takes
// its grid from here, so no call can lower the limit another one relies on.
struct Settings {
  int grid = 0;
  size_t smem = 0;
};

template <typename Kern>
static int settings_for(LaunchMemo& memo, Kern kern, size_t smem, int threads, bool one_per_sm, int max_grid,
                        Settings* st) {
  const int dev = current_device();
  if (dev < 0) return SPEC_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(memo.mu);
  if (!grant_smem_locked(memo, (const void*)kern, dev, smem)) return SPEC_ERR_LAUNCH;
  if (memo.grid_smem[dev] != smem) {
    int sms = 0, per_sm = 1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SPEC_ERR_LAUNCH;
    if (!one_per_sm && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess)
      return SPEC_ERR_LAUNCH;
    if (per_sm < 1) return SPEC_ERR_UNSUPPORTED;
    memo.grid[dev] = sms * per_sm > max_grid ? max_grid : sms * per_sm;
    memo.grid_smem[dev] = smem;
  }
  st->grid = memo.grid[dev];
  st->smem = smem;
  return SPEC_OK;
}

template <int D, int MT>
static LaunchMemo& memo_main() {
  static LaunchMemo memo;
  return memo;
}

template <int D, int MT, int S, int NP, int SV, int SQ>
static LaunchMemo& memo_tc() {
  static LaunchMemo memo;
  return memo;
}

template <int D, int MT>
static int settings_main(int batch, Settings* st) {
  return settings_for(memo_main<D, MT>(), verify_attention_kernel<D, MT>, smem_bytes<D, MT>(batch), kThreads,
                      false, kMaxGrid, st);
}

// The tcgen05 kernel runs one CTA per SM (at most tc::kMaxGrid CTAs).
template <int D, int MT, int S, int NP, int SV = S, int SQ = S>
static int settings_tc(int batch, Settings* st) {
  return settings_for(memo_tc<D, MT, S, NP, SV, SQ>(), tc::verify_attention_tc_kernel<D, MT, S, NP, SV, SQ>,
                      tc::smem_bytes<D, MT, S, NP, SV, SQ>(batch), tc::Cfg<D, MT>::kThreads, true, tc::kMaxGrid, st);
}

template <int D, int MT>
static int launch_main(const Params& p, const Settings& st, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, cudaStream_t stream) {
  verify_attention_kernel<D, MT><<<st.grid, kThreads, st.smem, stream>>>(p, tq, tk, tv);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

template <int D, int MT, int S, int NP, int SV = S, int SQ = S>
static int launch_tc(const Params& p, const Settings& st, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t stream) {
  tc::verify_attention_tc_kernel<D, MT, S, NP, SV, SQ><<<st.grid, tc::Cfg<D, MT>::kThreads, st.smem, stream>>>(p, tq, tk,
                                                                                                     tv);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

enum class Kernel { kMma, kTc };

// Which kernel runs a call. D = 128 or 256 with 32 or more packed query rows
// per kv head (17 or more, padded to 32 or 64) takes the tcgen05 kernel (its
// MMAs stay wide, where mma.sync tiles become compute-bound or, at D = 256,
// register-bound), 16 rows the mma.sync kernel (at that width both are bound
// by HBM and the mma.sync kernel, two CTAs per SM at D = 128, hides its
// per-unit work better). The environment variable SPEC_ATTN_KERNEL=tc or =mma
// overrides the choice for D = 128 and 256; the tcgen05 kernel also needs its
// shared-memory plan to fit the batch. Both compute the same result within
// rounding.
struct Choice {
  Kernel kind;
  int stages;     // tcgen05: K ring stages (the V ring has as many, or two with three
                  // K stages at 64 rows; the mma.sync kernel's are fixed by Cfg)
  int p_buffers;  // tcgen05: shared-memory buffers of P
};

// Returns SPEC_OK, or SPEC_ERR_LAUNCH when the device query the tcgen05 plan needs fails.
static int choose_kernel(int D, int mt, int batch, Choice* c) {
  *c = Choice{Kernel::kMma, 0, 0};
  if (D != 128 && D != 256) return SPEC_OK;
  const char* env = getenv("SPEC_ATTN_KERNEL");
  const bool force_tc = env != nullptr && strcmp(env, "tc") == 0;
  const bool force_mma = env != nullptr && strcmp(env, "mma") == 0;
  if (force_mma || (!force_tc && mt < 2)) return SPEC_OK;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  // stages x P buffers per row count, most overlap first (the instances dispatch
  // launches). At D = 256 one 128-key K + V stage is 128 KB, so there is one.
  size_t need3 = SIZE_MAX, need2 = SIZE_MAX, need1 = SIZE_MAX;
  int np = 2;
  if (D == 128) {
    switch (mt) {
      case 1: need3 = tc::smem_bytes<128, 1, 3, 2>(batch); need2 = tc::smem_bytes<128, 1, 2, 2>(batch); break;
      case 2: need2 = tc::smem_bytes<128, 2, 2, 2>(batch); break;
      default:  // 64 rows: three K stages, two V stages, one query buffer when they fit
        need3 = tc::smem_bytes<128, 4, 3, 1, 2, 1>(batch);
        need2 = tc::smem_bytes<128, 4, 2, 1>(batch);
        np = 1;
        break;
    }
  } else {
    switch (mt) {
      case 1: need1 = tc::smem_bytes<256, 1, 1, 2>(batch); break;
      case 2: need1 = tc::smem_bytes<256, 2, 1, 2>(batch); break;
      default: need1 = tc::smem_bytes<256, 4, 1, 1>(batch); np = 1; break;
    }
  }
  if (need3 <= (size_t)optin) c->stages = 3;
  else if (need2 <= (size_t)optin) c->stages = 2;
  else if (need1 <= (size_t)optin) c->stages = 1;
  else return SPEC_OK;
  c->kind = Kernel::kTc;
  c->p_buffers = np;
  return SPEC_OK;
}

// m16 tiles that hold the packed query rows of one kv head.
static int m_tiles(int rows) { return rows <= 16 ? 1 : (rows <= 32 ? 2 : 4); }

// The plan of the mma.sync instance for head dim D (see spec_attn_plan).
template <int D, int MT>
static void plan_mma(spec_attn_plan* pl) {
  using C = Cfg<D, MT>;
  *pl = spec_attn_plan{SPEC_ATTN_KERNEL_MMA, MT, C::TK, C::S, 0, C::MIN_BLOCKS};
}

template <int D>
static void plan_mma_d(int mt, spec_attn_plan* pl) {
  switch (mt) {
    case 1: plan_mma<D, 1>(pl); break;
    case 2: plan_mma<D, 2>(pl); break;
    default: plan_mma<D, 4>(pl); break;
  }
}

template <int D>
static int settings_main_d(int mt, int batch, Settings* st) {
  switch (mt) {
    case 1: return settings_main<D, 1>(batch, st);
    case 2: return settings_main<D, 2>(batch, st);
    default: return settings_main<D, 4>(batch, st);
  }
}

template <int D>
static int launch_main_d(const Params& p, int mt, const Settings& st, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, cudaStream_t stream) {
  switch (mt) {
    case 1: return launch_main<D, 1>(p, st, tq, tk, tv, stream);
    case 2: return launch_main<D, 2>(p, st, tq, tk, tv, stream);
    default: return launch_main<D, 4>(p, st, tq, tk, tv, stream);
  }
}

// The kernel a call runs and its launch settings (grid, shared memory) on the
// current device. Both entry points call this before they lay out their
// scratch, so the allocation-free one sizes its partial slots by the grid of
// the kernel that is actually launched.
struct Prepared {
  Choice ch;
  Settings st;
  int mt = 1;
};

static int prepare(int D, int rows, int batch, Prepared* pr) {
  pr->mt = m_tiles(rows);
  const int rc = choose_kernel(D, pr->mt, batch, &pr->ch);
  if (rc != SPEC_OK) return rc;
  if (pr->ch.kind == Kernel::kTc) {
    if (D == 256) {
      if (pr->mt == 1) return settings_tc<256, 1, 1, 2>(batch, &pr->st);
      if (pr->mt == 2) return settings_tc<256, 2, 1, 2>(batch, &pr->st);
      return settings_tc<256, 4, 1, 1>(batch, &pr->st);
    }
    if (pr->mt == 1) return pr->ch.stages == 3 ? settings_tc<128, 1, 3, 2>(batch, &pr->st)
                                              : settings_tc<128, 1, 2, 2>(batch, &pr->st);
    if (pr->mt == 2) return settings_tc<128, 2, 2, 2>(batch, &pr->st);
    return pr->ch.stages == 3 ? settings_tc<128, 4, 3, 1, 2, 1>(batch, &pr->st)
                              : settings_tc<128, 4, 2, 1>(batch, &pr->st);
  }
  switch (D) {
    case 64: return settings_main_d<64>(pr->mt, batch, &pr->st);
    case 128: return settings_main_d<128>(pr->mt, batch, &pr->st);
    default: return settings_main_d<256>(pr->mt, batch, &pr->st);
  }
}

// Builds the tensor maps for the prepared kernel's key tile and launches it.
static int dispatch(const Params& p, const Prepared& pr, int D, int bs, const void* q, const void* k_cache,
                    const void* v_cache, int64_t num_blocks, cudaStream_t stream) {
  const int R = p.rows_per_seq, G = p.gqa, mt = pr.mt;
  const Choice& ch = pr.ch;
  const int tk = ch.kind == Kernel::kTc ? tc::TK : tile_keys(D, mt);
  CUtensorMap tq, tk_map, tv_map;
  if (!make_map(&tq, q, D, p.num_q_heads, (uint64_t)p.batch * R, (uint32_t)G, (uint32_t)R) ||
      !make_map(&tk_map, k_cache, D, p.num_kv_heads, (uint64_t)num_blocks * bs, 1, (uint32_t)(bs < tk ? bs : tk)) ||
      !make_map(&tv_map, v_cache, D, p.num_kv_heads, (uint64_t)num_blocks * bs, 1, (uint32_t)(bs < tk ? bs : tk)))
    return SPEC_ERR_LAUNCH;
  if (ch.kind == Kernel::kTc) {
    if (D == 256) {
      if (mt == 1) return launch_tc<256, 1, 1, 2>(p, pr.st, tq, tk_map, tv_map, stream);
      if (mt == 2) return launch_tc<256, 2, 1, 2>(p, pr.st, tq, tk_map, tv_map, stream);
      return launch_tc<256, 4, 1, 1>(p, pr.st, tq, tk_map, tv_map, stream);
    }
    if (mt == 1) return ch.stages == 3 ? launch_tc<128, 1, 3, 2>(p, pr.st, tq, tk_map, tv_map, stream)
                                    : launch_tc<128, 1, 2, 2>(p, pr.st, tq, tk_map, tv_map, stream);
    if (mt == 2) return launch_tc<128, 2, 2, 2>(p, pr.st, tq, tk_map, tv_map, stream);
    return ch.stages == 3 ? launch_tc<128, 4, 3, 1, 2, 1>(p, pr.st, tq, tk_map, tv_map, stream)
                          : launch_tc<128, 4, 2, 1>(p, pr.st, tq, tk_map, tv_map, stream);
  }
  switch (D) {
    case 64: return launch_main_d<64>(p, mt, pr.st, tq, tk_map, tv_map, stream);
    case 128: return launch_main_d<128>(p, mt, pr.st, tq, tk_map, tv_map, stream);
    default: return launch_main_d<256>(p, mt, pr.st, tq, tk_map, tv_map, stream);
  }
}

}  // namespace attn
}  // namespace specv

using namespace specv;

extern "C" size_t spec_verify_attention_workspace(const spec_attn_desc* d, int32_t k_draft) {
  if (!attn::desc_ok(d, k_draft)) return 0;
  return attn::layout_for(d, k_draft).total;
}

extern "C" int spec_verify_attention_plan(const spec_attn_desc* d, int32_t k_draft, spec_attn_plan* plan) {
  if (!attn::desc_ok(d, k_draft) || plan == nullptr) return SPEC_ERR_INVALID_ARG;
  if (!attn::shape_supported(d, k_draft)) return SPEC_ERR_UNSUPPORTED;
  const int D = d->head_dim;
  const int mt = attn::m_tiles((k_draft + 1) * (d->num_q_heads / d->num_kv_heads));
  attn::Choice ch;
  const int rc = attn::choose_kernel(D, mt, d->batch, &ch);
  if (rc != SPEC_OK) return rc;
  if (ch.kind == attn::Kernel::kTc) {
    *plan = spec_attn_plan{SPEC_ATTN_KERNEL_TC, mt, attn::tc::TK, ch.stages, ch.p_buffers, 1};
    return SPEC_OK;
  }
  switch (D) {
    case 64: attn::plan_mma_d<64>(mt, plan); break;
    case 128: attn::plan_mma_d<128>(mt, plan); break;
    default: attn::plan_mma_d<256>(mt, plan); break;
  }
  return SPEC_OK;
}

namespace specv {
namespace attn {

// Host-side checks shared by both entry points (workspace aside).
static int check_call(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                      const int32_t* ctx_lens, int k_draft, const float* out, const spec_attn_desc* d) {
  if (!desc_ok(d, k_draft)) return SPEC_ERR_INVALID_ARG;
  if (d->batch == 0) return SPEC_OK;
  if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !out) return SPEC_ERR_INVALID_ARG;
  if (!shape_supported(d, k_draft)) return SPEC_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) & 15)
    return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

// The kernel parameter block for a call whose scratch starts at `ws`
// (arrival counters at 0, log-sum-exp and partial outputs at the offsets).
static Params make_params(const int32_t* block_table, const int32_t* ctx_lens, int k_draft, float* out,
                          const spec_attn_desc* d, uint8_t* ws, size_t lse_off, size_t opart_off,
                          int32_t* dev_err) {
  const int R = k_draft + 1, G = d->num_q_heads / d->num_kv_heads;
  Params p;
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
  while ((1 << shift) < d->block_size) ++shift;
  p.block_shift = shift;
  p.max_blocks = d->max_blocks_per_seq;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d->head_dim));
  return p;
}

}  // namespace attn
}  // namespace specv

extern "C" int spec_verify_attention(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* ctx_lens, int32_t k_draft,
                                     float* out, const spec_attn_desc* d, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_err, spec_stream_t stream_) {
  if (!attn::desc_ok(d, k_draft)) return SPEC_ERR_INVALID_ARG;
  if (d->batch == 0) return SPEC_OK;
  int rc = attn::check_call(q, k_cache, v_cache, block_table, ctx_lens, k_draft, out, d);
  if (rc != SPEC_OK) return rc;
  const attn::Layout L = attn::layout_for(d, k_draft);
  if (workspace == nullptr || workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return SPEC_ERR_INVALID_ARG;
  attn::Prepared pr;
  rc = attn::prepare(d->head_dim, (k_draft + 1) * (d->num_q_heads / d->num_kv_heads), d->batch, &pr);
  if (rc != SPEC_OK) return rc;
  const attn::Params p = attn::make_params(block_table, ctx_lens, k_draft, out, d, static_cast<uint8_t*>(workspace),
                                           L.lse_off, L.opart_off, dev_err);
  return attn::dispatch(p, pr, d->head_dim, d->block_size, q, k_cache, v_cache, d->num_blocks,
                        reinterpret_cast<cudaStream_t>(stream_));
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

}  // namespace attn
}  // namespace specv

extern "C" size_t spec_verify_attention_noalloc_limit(void) { return attn::kNoAllocScratchBytes; }

extern "C" int spec_verify_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_table, const int32_t* ctx_lens, int32_t k_draft,
                                             float* out, const spec_attn_desc* d, int32_t* dev_err,
                                             spec_stream_t stream_) {
  if (!attn::desc_ok(d, k_draft)) return SPEC_ERR_INVALID_ARG;
  if (d->batch == 0) return SPEC_OK;
  int rc = attn::check_call(q, k_cache, v_cache, block_table, ctx_lens, k_draft, out, d);
  if (rc != SPEC_OK) return rc;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  // Scratch this shape needs at most: arrival counters, then two partial slots
  // per CTA of the largest persistent grid. A shape that cannot fit even then
  // is rejected before any device call.
  const int64_t n_rows = (int64_t)(k_draft + 1) * (d->num_q_heads / d->num_kv_heads);
  const size_t counters_bytes = attn::align256((size_t)d->batch * d->num_kv_heads * 4);
  auto scratch_total = [&](int64_t grid, size_t* lse_off, size_t* opart_off) {
    const int64_t slots = 2 * grid;
    *lse_off = counters_bytes;
    *opart_off = *lse_off + attn::align256((size_t)(slots * n_rows * 4));
    return *opart_off + attn::align256((size_t)(slots * n_rows * d->head_dim * 4));
  };
  size_t lse_off = 0, opart_off = 0;
  if (scratch_total(1, &lse_off, &opart_off) > attn::kNoAllocScratchBytes) return SPEC_ERR_SCRATCH_LIMIT;

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

  // The kernel this call launches and its grid, from the same per-instance
  // settings the workspace form uses; the partial slots follow that grid.
  attn::Prepared pr;
  rc = attn::prepare(d->head_dim, (int)n_rows, d->batch, &pr);
  if (rc != SPEC_OK) return rc;
  if (scratch_total(pr.st.grid, &lse_off, &opart_off) > attn::kNoAllocScratchBytes) return SPEC_ERR_SCRATCH_LIMIT;

  uint8_t* ws = static_cast<uint8_t*>(scratch);
  // The counters must start at zero; every call shares the array, so clear them here.
  if (cudaMemsetAsync(ws, 0, counters_bytes, stream) != cudaSuccess) return SPEC_ERR_LAUNCH;
  const attn::Params p = attn::make_params(block_table, ctx_lens, k_draft, out, d, ws, lse_off, opart_off, dev_err);
  return attn::dispatch(p, pr, d->head_dim, d->block_size, q, k_cache, v_cache, d->num_blocks, stream);
}
