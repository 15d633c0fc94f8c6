/*
 * spec_verify.h -- C ABI of the target-side verify step of chain speculative
 * decoding (a draft of k tokens is checked by one wide target pass).
 *
 * The step has three parts, one entry point each:
 *
 *   spec_verify_attention  paged GQA attention of the k+1 verify rows of every
 *                          sequence over a block-paged bf16 KV cache
 *                          (lmdeploy PR #5019, summary: "paged CuTe
 *                          verification attention"; onnxruntime-genai PR #2457,
 *                          fast-commit notes: the "wide batched verify").
 *   spec_accept            greedy prefix match or speculative (rejection)
 *                          sampling over vocab-sized logits, giving the number
 *                          of accepted drafts and the correction/bonus token
 *                          (lmdeploy PR #5019, summary: "speculative sampling";
 *                          lmdeploy PR #3945, review of reject_sampler.py;
 *                          onnxruntime-genai PR #2457: greedy speculation is
 *                          token-identical to greedy decoding).
 *   spec_commit_state      copies, for every row, the recurrent-state checkpoint
 *                          of the accepted prefix into the live gated-delta-net
 *                          state (onnxruntime-genai PR #2457, notes on per-token
 *                          state checkpoints and CommitPrefix; lmdeploy PR #5019,
 *                          fix 2: CommitAcceptedRecurrentStateKernel).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor argument is a DEVICE pointer owned by the caller. The library
 *    never allocates, frees or synchronises; each call only enqueues kernels on
 *    `stream` (a cudaStream_t; NULL = legacy default stream) and returns.
 *  - Return value: SPEC_OK, or a negative SPEC_ERR_* code. Arguments the host
 *    can check (null pointers, sizes, unsupported shapes, a workspace that is
 *    too small) are checked before anything is launched; on error nothing is
 *    enqueued. SPEC_ERR_LAUNCH reports a failed kernel launch.
 *  - `dev_err` (optional, may be NULL) is a device int32 that kernels OR
 *    SPEC_DEVERR_* bits into when they meet data they cannot use (for example
 *    a block id outside the cache). The offending unit is skipped: its outputs
 *    are written as documented per call and the rest of the batch is computed
 *    normally. No kernel traps, asserts or aborts. The caller clears the word.
 *  - All index tensors are int32, row-major, densely packed.
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, without requiring the CUDA headers. */
typedef struct CUstream_st* spec_stream_t;

/* Status codes. */
#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARG (-1)   /* null pointer, negative size, bad enum   */
#define SPEC_ERR_UNSUPPORTED (-2)   /* a shape this build has no kernel for    */
#define SPEC_ERR_LAUNCH (-3)        /* cudaLaunch* failed (see cudaGetLastError) */
#define SPEC_ERR_WORKSPACE (-4)     /* workspace missing or smaller than asked  */
#define SPEC_ERR_SCRATCH_LIMIT (-5) /* shape needs more than the fixed scratch of
                                       spec_verify_attention_noalloc           */

/* Bits OR-ed into *dev_err by the kernels. */
#define SPEC_DEVERR_BLOCK_ID 1     /* block_table entry outside [0, num_blocks)  */
#define SPEC_DEVERR_TOKEN 2        /* draft token outside [0, V)                 */
#define SPEC_DEVERR_ACCEPT_LEN 4   /* accept_len outside [0, S-1]                */
#define SPEC_DEVERR_CTX_LEN 8      /* ctx_len < k+1 or > max_blocks_per_seq * bs */
#define SPEC_DEVERR_TEMPERATURE 16 /* sampling row with temperature not > 0      */
#define SPEC_DEVERR_TIMEOUT 32     /* an asynchronous copy did not arrive        */
#define SPEC_DEVERR_MODE 64        /* mode not 0/1                               */
#define SPEC_DEVERR_POOL_ROW 128   /* state-pool row index outside the pool      */

/* Human-readable name of a status code (static storage, never NULL). */
const char* spec_status_string(int status);

/* ------------------------------------------------------------------------ */
/* 1. Paged GQA verification attention                                        */
/* ------------------------------------------------------------------------ */

/* Shapes of one attention call. */
typedef struct spec_attn_desc {
  int32_t batch;              /* B: sequences                                  */
  int32_t num_q_heads;        /* Hq                                            */
  int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0, G = Hq / Hkv              */
  int32_t head_dim;           /* D in {64, 128, 256}                           */
  int32_t block_size;         /* bs: tokens per KV block, in {16, 32, 64, 128} */
  int32_t max_blocks_per_seq; /* row stride of block_table                     */
  int64_t num_blocks;         /* physical blocks in k_cache / v_cache          */
} spec_attn_desc;

/*
 * Bytes of device workspace spec_verify_attention needs for `d`: room for the
 * split-KV partial results (normalised partial outputs and their log-sum-exp)
 * of the largest split plan the kernel can choose, so the caller may size it
 * once from the shapes alone. Returns 0 for an invalid descriptor.
 */
size_t spec_verify_attention_workspace(const spec_attn_desc* d, int32_t k_draft);

/*
 * out[b, i, h, :] = softmax_t( q[b,i,h,:] . K[b,t,g,:] / sqrt(D) ) . V[b,t,g,:]
 * for every sequence b, verify row i in [0, k_draft], query head h, with
 * g = h / G (contiguous GQA groups) and t over the causal window
 * t <= ctx_lens[b] - (k_draft+1) + i: row 0 is the last committed token and
 * row i also sees the first i draft tokens of its own chain.
 *
 *  q           [B, k_draft+1, Hq, D] bf16
 *  k_cache     [num_blocks, bs, Hkv, D] bf16. Token t of sequence b is stored
 *  v_cache     in physical block block_table[b, t / bs], slot t % bs. The KV of
 *              the k_draft+1 verify tokens is already in the cache.
 *  block_table [B, max_blocks_per_seq] int32
 *  ctx_lens    [B] int32, tokens in the cache per sequence, verify tokens
 *              included; must lie in [k_draft+1, max_blocks_per_seq * bs].
 *  out         [B, k_draft+1, Hq, D] fp32
 *  workspace   >= spec_verify_attention_workspace(d, k_draft) bytes, 256-byte
 *              aligned, ZERO-FILLED before its first use (it holds per-unit
 *              arrival counters that every call returns to zero; the rest is
 *              scratch). Reuse it for later calls on the same stream; two calls
 *              in flight at once need two workspaces.
 *
 * The key tiles of all (sequence, kv head) units are split evenly over the
 * CTAs (split-KV); a unit held by several CTAs is merged by its log-sum-exp
 * inside the same launch. When all units have the same length, CTAs take
 * whole units instead as long as the load stays close to even. The split is
 * chosen on the device from ctx_lens, so no host synchronisation is needed.
 * Calls may come from several host threads at once (each with its own
 * workspace and stream).
 * Kernels: D = 128 or 256 with (k_draft+1)*G >= 17 packed query rows runs on
 * the 5th-generation tensor cores (tcgen05, 128-key tiles, accumulators in
 * tensor memory) when that kernel's shared-memory plan fits the batch; other
 * shapes run on mma.sync tiles. The environment variable SPEC_ATTN_KERNEL=tc
 * or =mma overrides the choice for D = 128 and 256. Both give the same result
 * within rounding (fp32 accumulation in both).
 * Device errors: a sequence with an out-of-range ctx_len (SPEC_DEVERR_CTX_LEN)
 * or block id (SPEC_DEVERR_BLOCK_ID) gets out rows of zeros.
 * Supported: D in {64,128,256}; bs in {16,32,64,128}; (k_draft+1)*G <= 64.
 */
int spec_verify_attention(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, const int32_t* ctx_lens,
                          int32_t k_draft, float* out, const spec_attn_desc* d,
                          void* workspace, size_t workspace_bytes, int32_t* dev_err,
                          spec_stream_t stream);

/*
 * Allocation-free form of spec_verify_attention (the pages have no
 * counterpart; this is a convenience of this library).
 *
 * For callers that may not allocate device memory when they call in: a
 * serving engine's per-step enqueue path that must not touch the allocator,
 * a plugin hook of an inference runtime whose enqueue contract forbids
 * allocation, or a process that reserved all device memory up front. It
 * computes the same result as spec_verify_attention but takes no workspace:
 * its scratch is a fixed array of spec_verify_attention_noalloc_limit() bytes
 * (32 MiB) inside the library, which every GPU that loads the library holds
 * until the process exits. It never calls cudaMalloc or cudaFree.
 *
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call shares the one array and leaves its contents behind; the call
 *    clears the part that must start at zero (an asynchronous memset on
 *    `stream`). Calls whose kernels overlap on the GPU (other streams, or
 *    other host threads) race on the array: serialise them.
 *  - A shape whose scratch would exceed the array returns
 *    SPEC_ERR_SCRATCH_LIMIT before anything is launched.
 * Arguments, layouts and device errors are those of spec_verify_attention.
 */
int spec_verify_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, const int32_t* ctx_lens,
                                  int32_t k_draft, float* out, const spec_attn_desc* d,
                                  int32_t* dev_err, spec_stream_t stream);

/* Bytes of the fixed scratch array used by spec_verify_attention_noalloc. */
size_t spec_verify_attention_noalloc_limit(void);

/*
 * Which kernel spec_verify_attention (and its allocation-free form) launches
 * for `d` and `k_draft` on the current device, with the tile settings it is
 * built with (a convenience of this library, for callers that report
 * per-kernel figures). The choice follows the rule stated above
 * spec_verify_attention, SPEC_ATTN_KERNEL included.
 *
 *  plan   written on SPEC_OK; host memory owned by the caller.
 *
 * Returns SPEC_ERR_INVALID_ARG for an invalid descriptor or a null plan,
 * SPEC_ERR_UNSUPPORTED for a shape spec_verify_attention rejects the same way,
 * and SPEC_ERR_LAUNCH when a device query it needs fails (D = 128 or 256 with
 * 17 or more packed rows, or with SPEC_ATTN_KERNEL=tc, reads the current
 * device's shared-memory limit; other shapes need no device). Launches
 * nothing and touches no device memory.
 */
#define SPEC_ATTN_KERNEL_MMA 1 /* mma.sync m16n8k16 tiles                    */
#define SPEC_ATTN_KERNEL_TC 2  /* tcgen05 MMAs, accumulators in tensor memory */

typedef struct spec_attn_plan {
  int32_t kernel;        /* SPEC_ATTN_KERNEL_*                                   */
  int32_t m_tiles;       /* (k_draft+1)*G packed rows padded to 16*m_tiles: 1, 2, 4 */
  int32_t keys_per_tile; /* keys per K/V pipeline stage                          */
  int32_t stages;        /* K/V pipeline stages in shared memory (tcgen05: K ring
                            stages; its V ring has as many, or two with three K) */
  int32_t p_buffers;     /* tcgen05: shared-memory buffers of P; 0 for mma.sync  */
  int32_t ctas_per_sm;   /* resident CTAs per SM the kernel is compiled for      */
} spec_attn_plan;

int spec_verify_attention_plan(const spec_attn_desc* d, int32_t k_draft, spec_attn_plan* plan);

/* ------------------------------------------------------------------------ */
/* 2. Acceptance: greedy prefix match or speculative sampling                  */
/* ------------------------------------------------------------------------ */

#define SPEC_MODE_GREEDY 0
#define SPEC_MODE_SAMPLE 1

/*
 * For each row b (k = number of drafts, R = k+1 target positions):
 *
 *  Greedy rows (mode[b] == SPEC_MODE_GREEDY): a_j = argmax_v target_logits[b,j,v]
 *  (lowest index on ties). accept_len[b] = m = first j < k with
 *  draft_tokens[b,j] != a_j, else k. Emitted: d_0..d_{m-1}, a_m.
 *
 *  Sampling rows (mode[b] == SPEC_MODE_SAMPLE), T = temperature[b] > 0:
 *  p_j = softmax(target_logits[b,j,:] / T), q_j = draft_probs[b,j,:].
 *  Draft j is accepted iff u_j * q_j(d_j) < p_j(d_j), u_j uniform in (0,1);
 *  m = first rejected j, else k. The last emitted token is drawn from
 *  w = max(0, p_m - q_m) (from p_m itself if that is all zero) when m < k, and
 *  from p_k when m == k. The draw is an exponential race over the whole
 *  vocabulary: every entry x with w_x > 0 gets the key w_x / E_x, E_x = -ln U_x,
 *  and the largest key wins, which samples x with probability w_x / sum(w)
 *  without normalising w. Ties go to the lowest index; entries of zero weight
 *  never win.
 *
 *  Random numbers: Philox4x32-10 (Salmon et al., SC'11) keyed by
 *  (philox_seed low word, philox_seed high word). u_j uses word 0 of counter
 *  (0, j, b, 0); U_x of the race at position m uses word (x mod 4) of counter
 *  (x / 4, m, b, 1). A word w maps to ((w >> 9) + 0.5) * 2^-23.
 *
 *  target_logits [B, k+1, V] fp32
 *  draft_tokens  [B, k] int32
 *  draft_probs   [B, k, V] fp32, each row a distribution; or NULL: the
 *                drafts are then deterministic and q_j is one-hot at d_j, so
 *                draft j is kept iff u_j < p_j(d_j) and a rejection draws from
 *                p_m with d_m removed (the reject sampler of lmdeploy PR #3945
 *                is called with draft_probs = None)
 *  mode          [B] int32 (SPEC_MODE_*); temperature [B] fp32 (ignored for
 *                greedy rows)
 *  out_tokens    [B, k+1] int32: d_0..d_{m-1}, final token, then -1 padding
 *  accept_len    [B] int32: m in [0, k]
 *
 * Rows are read only up to the first rejection (early exit), so the bytes read
 * depend on the outcome; when the batch's rows are small (B * V * 4 bytes at
 * most 32 MB), the first float4 batch of each thread's slice of position j + 1
 * is also loaded while position j is decided. Each row is handled by one
 * thread-block cluster; the call picks the threads per CTA and the CTAs per
 * cluster so that every row of the batch is resident at once where that fits
 * (clusters walk several rows otherwise). The environment variable
 * SPEC_ACCEPT_CONFIG=TxC (T = 128 or 256 threads, C = 1, 2, 4, 8 or 16 CTAs
 * per cluster) forces one configuration, for tests and measurements; one the
 * vocabulary cannot use (fewer than 4T logits per CTA with C > 1) makes the
 * call return SPEC_ERR_LAUNCH.
 * Device errors: a row with a draft token outside [0, V) (SPEC_DEVERR_TOKEN),
 * a sampling row with temperature not > 0 (SPEC_DEVERR_TEMPERATURE), or a mode
 * other than 0/1 (SPEC_DEVERR_MODE) gets out_tokens all -1 and accept_len -1.
 * Supported: k_draft <= 31; vocab <= 2^30.
 */
int spec_accept(const float* target_logits, const int32_t* draft_tokens,
                const float* draft_probs, uint64_t philox_seed, const int32_t* mode,
                const float* temperature, int32_t* out_tokens, int32_t* accept_len,
                int32_t batch, int32_t k_draft, int32_t vocab, int32_t* dev_err,
                spec_stream_t stream);

/* ------------------------------------------------------------------------ */
/* 3. Recurrent-state commit                                                  */
/* ------------------------------------------------------------------------ */

/*
 * live_state[l, b, :] = snapshots[l, b, accept_len[b], :] for every layer l
 * and row b. Snapshot slot s holds the state after the verify step consumed
 * its input s (input 0 is the last committed token), so slot accept_len[b] is
 * the state of the accepted prefix.
 *
 *  snapshots  [L, B, S, state_elems] fp32
 *  accept_len [B] int32 (as written by spec_accept)
 *  live_state [L, B, state_elems] fp32
 *
 * The copy is bit-exact. A row whose accept_len lies outside [0, S-1] keeps
 * its live state unchanged and sets SPEC_DEVERR_ACCEPT_LEN.
 */
int spec_commit_state(const float* snapshots, const int32_t* accept_len,
                      float* live_state, int32_t num_layers, int32_t batch,
                      int32_t num_slots, int64_t state_elems, int32_t* dev_err,
                      spec_stream_t stream);

/* Checkpoint alignments of spec_commit_state_aligned. */
#define SPEC_ALIGN_TOKEN 0 /* slot j holds the state after the step's token j      */
#define SPEC_ALIGN_LAST 1  /* slot W-1 holds the state after the step's last token */

/*
 * Commit from a checkpoint window that may be wider than the step
 * (onnxruntime-genai PR #2457: the window is described by a checkpoint count
 * and an alignment, because the conv state writes slot j after local token j
 * while GatedDeltaNet writes slot W-1 after the last token). A step of
 * num_tokens = n tokens (k+1 for a verify step) fills a window of
 * num_slots = W >= n slots; with m = accept_len[b] drafts accepted the kept
 * state is the one after token m:
 *
 *   SPEC_ALIGN_TOKEN: live_state[l, b, :] = snapshots[l, b, m, :]
 *   SPEC_ALIGN_LAST:  live_state[l, b, :] = snapshots[l, b, W - n + m, :]
 *
 * snapshots [L, B, W, state_elems] fp32; accept_len [B] int32; live_state
 * [L, B, state_elems] fp32. With W = n both alignments equal spec_commit_state.
 * A row with accept_len outside [0, n-1] keeps its live state and sets
 * SPEC_DEVERR_ACCEPT_LEN. Returns SPEC_ERR_INVALID_ARG for n outside [1, W]
 * or another alignment.
 */
int spec_commit_state_aligned(const float* snapshots, const int32_t* accept_len,
                              float* live_state, int32_t num_layers, int32_t batch,
                              int32_t num_slots, int64_t state_elems, int32_t num_tokens,
                              int32_t alignment, int32_t* dev_err, spec_stream_t stream);

/*
 * Zero-copy commit: stage a different source row instead of copying state
 * (onnxruntime-genai PR #2457, CommitPrefix note: rolling back a rejected
 * draft only needs the state pool to stage another row, the checkpoint of the
 * accepted prefix, instead of the step's final state).
 *
 * The states are rows of a pool that the caller owns and that this call never
 * touches; two int32 tables of pool-row indices, updated in place, say where
 * each (layer l, row b) keeps its state:
 *
 *  live_row  [L, B]    int32: the row holding the live state of (l, b)
 *  ckpt_rows [L, B, W] int32: the W rows the verify step writes its
 *                      checkpoints to (slot s in ckpt_rows[l, b, s])
 *  accept_len [B] int32 (as written by spec_accept)
 *
 * With m = accept_len[b] and the slot s picked as in spec_commit_state_aligned
 * (s = m for SPEC_ALIGN_TOKEN, W - n + m for SPEC_ALIGN_LAST, n = num_tokens),
 * the call exchanges live_row[l, b] and ckpt_rows[l, b, s]: the chosen
 * checkpoint becomes the live state where it lies, and the former live row
 * becomes the window's free slot for the next step. Afterwards
 * pool[live_row[l, b]] holds exactly what spec_commit_state_aligned would have
 * copied, and each (l, b) still owns the same W + 1 rows. Cost: 16 bytes of
 * index traffic per (l, b) instead of two state copies.
 *
 * A row with accept_len outside [0, n-1] keeps both tables and sets
 * SPEC_DEVERR_ACCEPT_LEN. Returns SPEC_ERR_INVALID_ARG for n outside [1, W],
 * another alignment, negative sizes or a missing table.
 */
int spec_commit_select(const int32_t* accept_len, int32_t* live_row, int32_t* ckpt_rows,
                       int32_t num_layers, int32_t batch, int32_t num_slots,
                       int32_t num_tokens, int32_t alignment, int32_t* dev_err,
                       spec_stream_t stream);

/* ------------------------------------------------------------------------ */
/* 4. Gated delta rule over the verify chain (checkpoint producer)            */
/* ------------------------------------------------------------------------ */

/*
 * The GatedDeltaNet layers of a hybrid model publish their recurrent state
 * after every token of the speculative step (onnxruntime-genai PR #2457:
 * GatedDeltaNet.checkpoints, V-major float32 state, checkpoint windows;
 * lmdeploy PR #5019: GDR verify kernels); these calls compute that series for
 * one layer. The pages name the operator but not its update, which follows the
 * published Gated DeltaNet rule (Yang, Kautz, Hatamizadeh, "Gated Delta
 * Networks"). Per row b, head h and token t (R = num_tokens tokens, k+1 for a
 * verify step), with the state S V-major (S[i][c]: value i, key c):
 *
 *   a_t = exp(g_t)
 *   S_t = a_t S_{t-1} + beta_t (v_t - a_t S_{t-1} k_t) k_t^T
 *   o_t = S_t (scale q_t)
 *
 * S_0 is the live state; checkpoint slot base + t of a W-slot window
 * (W = num_slots >= R) receives S_{t+1}, the state after input t, with
 * base = 0 for SPEC_ALIGN_TOKEN and W - R for SPEC_ALIGN_LAST; other slots are
 * not written. The gates arrive computed (g is the log decay, typically <= 0);
 * q and k are used as given (any normalisation happens upstream).
 *
 *  q, k   [B, R, H, dk] fp32      v    [B, R, H, dv] fp32
 *  g, beta [B, R, H] fp32         out  [B, R, H, dv] fp32 (o_t)
 *  state_in  [B, H, dv, dk] fp32  (one row of E = H*dv*dk floats per b)
 *  snapshots [B, W, H, dv, dk] fp32
 *
 * Arithmetic is fp32 (the state stays fp32 between tokens). dk = dv = 128
 * runs the register-resident kernel (16-byte aligned states); other sizes run
 * a shared-memory kernel while dv*dk + R*(2dk+dv) + 3dv floats fit in 200 KB.
 * Returns SPEC_ERR_INVALID_ARG for R outside [1, 32], W < R, an unknown
 * alignment, non-positive sizes or missing pointers; SPEC_ERR_UNSUPPORTED for
 * a state too large for either kernel.
 */
int spec_gdn_verify(const float* q, const float* k, const float* v, const float* g,
                    const float* beta, float scale, const float* state_in, float* snapshots,
                    float* out, int32_t batch, int32_t num_tokens, int32_t num_heads,
                    int32_t dk, int32_t dv, int32_t num_slots, int32_t alignment,
                    int32_t* dev_err, spec_stream_t stream);

/*
 * The same step over a state pool, the companion of spec_commit_select: row b
 * reads its live state from pool row live_row[b] and writes checkpoint slot s
 * to pool row ckpt_rows[b, s]; a pool row holds E = H*dv*dk floats (all heads
 * of one (layer, row)). Pass the tables of one layer (live_row + l*B,
 * ckpt_rows + l*B*W). A row naming an index outside [0, pool_rows) writes
 * zeros to its out rows, touches no state and sets SPEC_DEVERR_POOL_ROW.
 */
int spec_gdn_verify_pooled(const float* q, const float* k, const float* v, const float* g,
                           const float* beta, float scale, float* pool, int64_t pool_rows,
                           const int32_t* live_row, const int32_t* ckpt_rows, float* out,
                           int32_t batch, int32_t num_tokens, int32_t num_heads, int32_t dk,
                           int32_t dv, int32_t num_slots, int32_t alignment, int32_t* dev_err,
                           spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
