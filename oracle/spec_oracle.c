/*
 * spec_oracle.c -- plain, slow CPU oracle of the speculative-decoding verify
 * step. TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it; the product library never does, and
 * this file shares no code, header or table with the CUDA kernels.
 *
 * Everything is computed in double precision from the stored inputs, in the
 * order of the plain definitions below; there is no tiling or fusion. Loops
 * over independent units (sequence x kv head, batch row, layer x row) are
 * spread over OpenMP threads, which changes nothing in any result.
 *
 * Sources of each definition:
 *  - attention: the verify pass runs the last committed token plus the k
 *    drafts through the target in one batched forward (onnxruntime-genai PR
 *    #2457 "Expose speculative draft proposals through Engine APIs", fast
 *    commit notes: "wide batched verify") over a paged KV cache (lmdeploy PR
 *    #5019, summary: "paged CuTe verification attention"); the attention
 *    itself is plain scaled-dot-product softmax attention, causal along the
 *    chain, keys gathered through the block table.
 *  - greedy acceptance: greedy speculation must be token-identical to greedy
 *    decoding (onnxruntime-genai PR #2457, Qwen3.8-27B-NVFP4 validation note).
 *  - sampling acceptance: speculative sampling (lmdeploy PR #5019 summary;
 *    lmdeploy PR #3945 review of spec_decode/reject_sampler.py, whose fixture
 *    pads the emitted tokens with -1), i.e. the rule of Leviathan et al. 2023
 *    and Chen et al. 2023: accept a draft d with probability min(1, p(d)/q(d)),
 *    otherwise draw from max(0, p - q) normalised; the draw is an exponential
 *    race (an exact sampler of w / sum(w)) with one uniform per vocabulary
 *    entry.
 *  - Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 *    easy as 1, 2, 3", SC'11.
 *  - state commit: the operators publish the recurrent state after every verify
 *    token and the commit picks the slot of the accepted prefix
 *    (onnxruntime-genai PR #2457, per-token state checkpoint and CommitPrefix
 *    notes; lmdeploy PR #5019, fix 2, CommitAcceptedRecurrentStateKernel).
 *  - gated delta rule over the verify chain (the checkpoints' producer): the
 *    pages name the GatedDeltaNet operator, its V-major float32 state and its
 *    checkpoint window but not the update, which follows Yang, Kautz,
 *    Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_BLOCK (-5)
#define ORACLE_ERR_CTX (-6)
#define ORACLE_ERR_ACCEPT_LEN (-7)
#define ORACLE_ERR_TOKEN (-8)
#define ORACLE_ERR_TEMPERATURE (-9)
#define ORACLE_ERR_NOMEM (-10)

static void set_threads(int n_threads) {
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11, section 5: the Philox S-box of two    */
/* 32x32->64 multiplications, a key schedule advanced by Weyl constants, 10   */
/* rounds).                                                                   */
/* ------------------------------------------------------------------------ */

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint32_t mult0 = 0xD2511F53u, mult1 = 0xCD9E8D57u;
  const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
  uint32_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { /* the key is bumped between rounds */
      k0 += weyl0;
      k1 += weyl1;
    }
    uint64_t prod0 = (uint64_t)mult0 * (uint64_t)x0;
    uint64_t prod1 = (uint64_t)mult1 * (uint64_t)x2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t y0 = hi1 ^ x1 ^ k0;
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x3 ^ k1;
    uint32_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* A 32-bit word to a uniform in (0,1): top 23 bits plus one half, times 2^-23. */
double oracle_uniform(uint32_t word) {
  return ((double)(word >> 9) + 0.5) * (1.0 / 8388608.0);
}

static uint32_t philox_word(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                            int which) {
  uint32_t ctr[4] = {c0, c1, c2, c3};
  uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return out[which];
}

/* ------------------------------------------------------------------------ */
/* Paged GQA verification attention.                                          */
/* ------------------------------------------------------------------------ */

static double bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * Gather the keys and values of sequence b, kv head g into contiguous arrays
 * (token t lives in physical block block_table[b][t / bs], slot t % bs).
 */
static int gather_sequence(const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* block_table,
                           int b, int g, int n_tokens, int Hkv, int D, int bs, int64_t num_blocks,
                           int max_blocks, double* kc, double* vc) {
  for (int t = 0; t < n_tokens; ++t) {
    int32_t phys = block_table[(int64_t)b * max_blocks + t / bs];
    if (phys < 0 || (int64_t)phys >= num_blocks) return ORACLE_ERR_BLOCK;
    int64_t base = (((int64_t)phys * bs + t % bs) * Hkv + g) * (int64_t)D;
    for (int d = 0; d < D; ++d) {
      kc[(int64_t)t * D + d] = bf16_to_double(k_cache[base + d]);
      vc[(int64_t)t * D + d] = bf16_to_double(v_cache[base + d]);
    }
  }
  return ORACLE_OK;
}

/* softmax(q . k_t / sqrt(D)) . v_t over the first n_visible contiguous keys. */
static void attend_row(const double* qrow, const double* kc, const double* vc, int n_visible, int D,
                       double* scores, double* orow) {
  const double scale = 1.0 / sqrt((double)D);
  double smax = -INFINITY;
  for (int t = 0; t < n_visible; ++t) {
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += qrow[d] * kc[(int64_t)t * D + d];
    scores[t] = s * scale;
    if (scores[t] > smax) smax = scores[t];
  }
  double denom = 0.0;
  for (int t = 0; t < n_visible; ++t) {
    scores[t] = exp(scores[t] - smax);
    denom += scores[t];
  }
  for (int d = 0; d < D; ++d) orow[d] = 0.0;
  for (int t = 0; t < n_visible; ++t) {
    double w = scores[t] / denom;
    for (int d = 0; d < D; ++d) orow[d] += w * vc[(int64_t)t * D + d];
  }
}

/*
 * q [B,R,Hq,D] bf16 bits; k_cache/v_cache [num_blocks,bs,Hkv,D] bf16 bits;
 * block_table [B,max_blocks]; ctx_lens [B] (verify tokens included).
 * Computes the sequences listed in seqs[0..n_seqs) (all B in order when seqs
 * is NULL) into out [n_seqs,R,Hq,D]. Row i of sequence b sees keys
 * t <= ctx_lens[b] - R + i. Returns 0, or a negative code for the first bad
 * sequence found (its rows are left as zeros).
 */
int oracle_verify_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* block_table, const int32_t* ctx_lens, int B, int R,
                            int Hq, int Hkv, int D, int bs, int64_t num_blocks, int max_blocks,
                            const int32_t* seqs, int n_seqs, double* out, int n_threads) {
  if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !out) return ORACLE_ERR_ARG;
  if (B < 0 || R < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || bs < 1 || max_blocks < 1)
    return ORACLE_ERR_ARG;
  if (!seqs) n_seqs = B;
  const int G = Hq / Hkv;
  const int64_t n_units = (int64_t)n_seqs * Hkv;
  memset(out, 0, sizeof(double) * (size_t)n_seqs * R * Hq * D);
  int status = ORACLE_OK;
  set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t unit = 0; unit < n_units; ++unit) {
    const int s = (int)(unit / Hkv), g = (int)(unit % Hkv);
    const int b = seqs ? seqs[s] : s;
    int err = ORACLE_OK;
    const int n = (b >= 0 && b < B) ? ctx_lens[b] : -1;
    if (b < 0 || b >= B) err = ORACLE_ERR_ARG;
    else if (n < R || (int64_t)n > (int64_t)max_blocks * bs) err = ORACLE_ERR_CTX;
    double *kc = NULL, *vc = NULL, *scores = NULL, *qrow = NULL;
    if (err == ORACLE_OK) {
      kc = (double*)malloc(sizeof(double) * (size_t)n * D);
      vc = (double*)malloc(sizeof(double) * (size_t)n * D);
      scores = (double*)malloc(sizeof(double) * (size_t)n);
      qrow = (double*)malloc(sizeof(double) * (size_t)D);
      if (!kc || !vc || !scores || !qrow) err = ORACLE_ERR_NOMEM;
    }
    if (err == ORACLE_OK)
      err = gather_sequence(k_cache, v_cache, block_table, b, g, n, Hkv, D, bs, num_blocks, max_blocks, kc, vc);
    if (err == ORACLE_OK) {
      const int prefix = n - R; /* committed tokens before the verify rows */
      for (int i = 0; i < R; ++i) {
        for (int j = 0; j < G; ++j) {
          const int h = g * G + j;
          const uint16_t* qsrc = q + (((int64_t)b * R + i) * Hq + h) * D;
          for (int d = 0; d < D; ++d) qrow[d] = bf16_to_double(qsrc[d]);
          double* orow = out + (((int64_t)s * R + i) * Hq + h) * D;
          attend_row(qrow, kc, vc, prefix + i + 1, D, scores, orow);
        }
      }
    } else {
      /* leave this unit's rows zero; report the error */
#pragma omp critical
      if (status == ORACLE_OK) status = err;
    }
    free(kc); free(vc); free(scores); free(qrow);
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* Acceptance.                                                                */
/* ------------------------------------------------------------------------ */

/* First index of the largest value (ties go to the lowest index). */
static int argmax_row(const float* row, int V) {
  int best = 0;
  for (int x = 1; x < V; ++x)
    if (row[x] > row[best]) best = x;
  return best;
}

/* Max and sum of exp of logit/T over a row: p(x) = exp(l(x)/T - mx) / z. */
static void softmax_stats(const float* row, int V, double T, double* mx, double* z) {
  double m = -INFINITY;
  for (int x = 0; x < V; ++x) {
    double v = (double)row[x] / T;
    if (v > m) m = v;
  }
  double s = 0.0;
  for (int x = 0; x < V; ++x) s += exp((double)row[x] / T - m);
  *mx = m;
  *z = s;
}

/*
 * Exponential race over the weights w (length V), an exact sampler of
 * w / sum(w) that needs no normalisation: every entry x with w_x > 0 gets the
 * key w_x / E_x, E_x = -ln U_x with U_x from word (x mod 4) of Philox counter
 * (x / 4, m, b, 1), and the entry with the largest key wins (ties go to the
 * lowest index). Since E_x is exponential with rate 1, w_x / E_x exceeds every
 * other key with probability w_x / sum(w). *gap receives the relative gap
 * between the two largest keys (+inf when fewer than two entries have a key).
 * The four words of one counter serve four consecutive entries, so each
 * Philox block is computed once.
 */
static int exponential_race(const double* w, int V, uint64_t seed, int m, int b, double* gap) {
  const uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  int best = -1;
  double best_key = -1.0, second_key = -1.0;
  for (int x0 = 0; x0 < V; x0 += 4) {
    const uint32_t ctr[4] = {(uint32_t)(x0 / 4), (uint32_t)m, (uint32_t)b, 1u};
    uint32_t words[4];
    oracle_philox4x32_10(ctr, key, words);
    for (int e = 0; e < 4 && x0 + e < V; ++e) {
      const int x = x0 + e;
      if (!(w[x] > 0.0)) continue;
      const double k = w[x] / -log(oracle_uniform(words[e]));
      if (k > best_key) {
        second_key = best_key;
        best_key = k;
        best = x;
      } else if (k > second_key) {
        second_key = k;
      }
    }
  }
  *gap = (best_key > 0.0 && second_key > 0.0) ? (best_key - second_key) / best_key : INFINITY;
  return best;
}

/* Draft probability q_j(x). Without a draft distribution (draft_probs NULL) the
 * draft is taken as deterministic: q_j is one-hot at the drafted token d_j (the
 * reject sampler of lmdeploy PR #3945 is called with draft_probs = None). */
static double draft_q(const float* Q, const int32_t* d, int j, int V, int x) {
  return Q ? (double)Q[(int64_t)j * V + x] : (x == d[j] ? 1.0 : 0.0);
}

/*
 * target_logits [B,k+1,V]; draft_tokens [B,k]; draft_probs [B,k,V] (NULL: every
 * sampling row uses one-hot q, see draft_q); mode [B] (0 greedy, 1 sampling);
 * temperature [B]. Outputs out_tokens [B,k+1], accept_len [B], and for the
 * parity bookkeeping accept_margin [B] = min over the drafts that were tested
 * of |u - p/q| (+inf for greedy rows or when every q was 0) and race_gap [B] =
 * relative gap between the two largest keys of the race (+inf for greedy
 * rows).
 * Invalid rows (draft token out of range, sampling temperature not > 0) get
 * out_tokens -1 and accept_len -1; the call then returns an error code but
 * still computes every other row.
 */
int oracle_accept(const float* target_logits, const int32_t* draft_tokens, const float* draft_probs,
                  uint64_t seed, const int32_t* mode, const float* temperature, int B, int k, int V,
                  int32_t* out_tokens, int32_t* accept_len, double* accept_margin, double* race_gap,
                  int n_threads) {
  if (!target_logits || !draft_tokens || !mode || !temperature || !out_tokens || !accept_len)
    return ORACLE_ERR_ARG;
  if (B < 0 || k < 1 || V < 1) return ORACLE_ERR_ARG;
  for (int b = 0; b < B; ++b)
    if (mode[b] != 0 && mode[b] != 1) return ORACLE_ERR_ARG;
  const int R = k + 1;
  int status = ORACLE_OK;
  set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    int32_t* tok = out_tokens + (int64_t)b * R;
    const int32_t* d = draft_tokens + (int64_t)b * k;
    const float* L = target_logits + (int64_t)b * R * V;
    double margin = INFINITY, gap = INFINITY;
    int err = ORACLE_OK;
    for (int j = 0; j < R; ++j) tok[j] = -1;
    for (int j = 0; j < k; ++j)
      if (d[j] < 0 || d[j] >= V) err = ORACLE_ERR_TOKEN;
    if (err == ORACLE_OK && mode[b] == 1 && !(temperature[b] > 0.0f && isfinite(temperature[b])))
      err = ORACLE_ERR_TEMPERATURE;
    int m = -1;
    if (err == ORACLE_OK && mode[b] == 0) {
      /* greedy: accept drafts while they equal the target argmax */
      m = k;
      for (int j = 0; j < k; ++j) {
        if (d[j] != argmax_row(L + (int64_t)j * V, V)) {
          m = j;
          break;
        }
      }
      for (int j = 0; j < m; ++j) tok[j] = d[j];
      tok[m] = argmax_row(L + (int64_t)m * V, V);
    } else if (err == ORACLE_OK) {
      const double T = (double)temperature[b];
      const float* Q = draft_probs ? draft_probs + (int64_t)b * k * V : NULL;
      double mx = 0.0, z = 1.0;
      m = k;
      for (int j = 0; j < k; ++j) {
        softmax_stats(L + (int64_t)j * V, V, T, &mx, &z);
        const double p = exp((double)L[(int64_t)j * V + d[j]] / T - mx) / z;
        const double qd = draft_q(Q, d, j, V, d[j]);
        const double u = oracle_uniform(philox_word(seed, 0u, (uint32_t)j, (uint32_t)b, 0u, 0));
        if (qd > 0.0) {
          double mg = fabs(u - p / qd);
          if (mg < margin) margin = mg;
        }
        if (!(u * qd < p)) {
          m = j;
          break;
        }
      }
      double* w = (double*)malloc(sizeof(double) * (size_t)V);
      if (!w) {
        err = ORACLE_ERR_NOMEM;
      } else {
        if (m < k) {
          /* residual max(0, p_m - q_m); p_m's statistics are still in mx, z */
          double total = 0.0;
          for (int x = 0; x < V; ++x) {
            double p = exp((double)L[(int64_t)m * V + x] / T - mx) / z;
            double r = p - draft_q(Q, d, m, V, x);
            w[x] = r > 0.0 ? r : 0.0;
            total += w[x];
          }
          if (!(total > 0.0))
            for (int x = 0; x < V; ++x) w[x] = exp((double)L[(int64_t)m * V + x] / T - mx) / z;
        } else {
          /* every draft accepted: the bonus token comes from p_k itself */
          softmax_stats(L + (int64_t)k * V, V, T, &mx, &z);
          for (int x = 0; x < V; ++x) w[x] = exp((double)L[(int64_t)k * V + x] / T - mx) / z;
        }
        for (int j = 0; j < m; ++j) tok[j] = d[j];
        tok[m] = exponential_race(w, V, seed, m, b, &gap);
        free(w);
      }
    }
    if (err != ORACLE_OK) {
      for (int j = 0; j < R; ++j) tok[j] = -1;
      m = -1;
#pragma omp critical
      if (status == ORACLE_OK) status = err;
    }
    accept_len[b] = m;
    if (accept_margin) accept_margin[b] = margin;
    if (race_gap) race_gap[b] = gap;
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* Recurrent-state commit.                                                    */
/* ------------------------------------------------------------------------ */

/*
 * live [L,B,E] <- snapshots [L,B,S,E] at slot accept_len[b], for each layer
 * and row; rows with accept_len outside [0,S-1] keep their live state and make
 * the call return ORACLE_ERR_ACCEPT_LEN.
 */
/*
 * Checkpoint windows of W >= n slots for a step of n tokens (onnxruntime-genai
 * PR #2457: a checkpoint count plus a checkpoint alignment, because the conv
 * writes slot j after local token j while GatedDeltaNet writes slot W-1 after
 * the last token). With m = accept_len[b] drafts accepted the state to keep is
 * the one after token m:
 *   alignment 0 (token-indexed): slot m
 *   alignment 1 (last at W-1):   slot W - n + m
 * live[l,b,:] = snapshots[l,b,slot,:]; rows with m outside [0, n-1] are skipped
 * and reported.
 */
int oracle_commit_state_aligned(const float* snapshots, const int32_t* accept_len, float* live, int L, int B,
                                int W, int64_t E, int n, int alignment, int n_threads) {
  if (!snapshots || !accept_len || !live || L < 0 || B < 0 || W < 1 || E < 0) return ORACLE_ERR_ARG;
  if (n < 1 || n > W || (alignment != 0 && alignment != 1)) return ORACLE_ERR_ARG;
  const int base = alignment == 0 ? 0 : W - n;
  int status = ORACLE_OK;
  for (int b = 0; b < B; ++b)
    if (accept_len[b] < 0 || accept_len[b] >= n) status = ORACLE_ERR_ACCEPT_LEN;
  set_threads(n_threads);
  const int64_t n_units = (int64_t)L * B;
#pragma omp parallel for schedule(static)
  for (int64_t unit = 0; unit < n_units; ++unit) {
    const int64_t l = unit / B;
    const int b = (int)(unit % B);
    const int m = accept_len[b];
    if (m < 0 || m >= n) continue;
    const float* src = snapshots + ((l * B + b) * W + base + m) * E;
    float* dst = live + (l * B + b) * E;
    memcpy(dst, src, sizeof(float) * (size_t)E);
  }
  return status;
}

/*
 * Commit by staging a different source row (onnxruntime-genai PR #2457,
 * CommitPrefix note: rolling back a rejected draft only needs the state pool
 * to stage another row, the checkpoint of the accepted prefix, instead of the
 * step's final state). The states are rows of a pool; live_row[l,b] names the
 * row holding the live state of (l, b) and ckpt_rows[l,b,:] the W rows of its
 * checkpoint window. Committing slot s (picked exactly as in
 * oracle_commit_state_aligned) exchanges live_row[l,b] and ckpt_rows[l,b,s]:
 * the checkpoint row becomes the live row and the old live row becomes the
 * window's free slot. No state is read or written; a row with accept_len
 * outside [0, n-1] keeps both entries.
 */
int oracle_commit_select(const int32_t* accept_len, int32_t* live_row, int32_t* ckpt_rows, int L, int B, int W,
                         int n, int alignment) {
  if (!accept_len || !live_row || !ckpt_rows || L < 0 || B < 0 || W < 1) return ORACLE_ERR_ARG;
  if (n < 1 || n > W || (alignment != 0 && alignment != 1)) return ORACLE_ERR_ARG;
  const int base = alignment == 0 ? 0 : W - n;
  int status = ORACLE_OK;
  for (int l = 0; l < L; ++l) {
    for (int b = 0; b < B; ++b) {
      const int m = accept_len[b];
      if (m < 0 || m >= n) {
        status = ORACLE_ERR_ACCEPT_LEN;
        continue;
      }
      const int64_t unit = (int64_t)l * B + b;
      int32_t* slot = ckpt_rows + unit * W + base + m;
      const int32_t chosen = *slot;
      *slot = live_row[unit];
      live_row[unit] = chosen;
    }
  }
  return status;
}

int oracle_commit_state(const float* snapshots, const int32_t* accept_len, float* live, int L, int B,
                        int S, int64_t E, int n_threads) {
  if (!snapshots || !accept_len || !live || L < 0 || B < 0 || S < 1 || E < 0) return ORACLE_ERR_ARG;
  int status = ORACLE_OK;
  for (int b = 0; b < B; ++b)
    if (accept_len[b] < 0 || accept_len[b] >= S) status = ORACLE_ERR_ACCEPT_LEN;
  set_threads(n_threads);
  const int64_t n_units = (int64_t)L * B;
#pragma omp parallel for schedule(static)
  for (int64_t unit = 0; unit < n_units; ++unit) {
    const int64_t l = unit / B;
    const int b = (int)(unit % B);
    const int a = accept_len[b];
    if (a < 0 || a >= S) continue;
    const float* src = snapshots + ((l * B + b) * S + a) * E;
    float* dst = live + (l * B + b) * E;
    memcpy(dst, src, sizeof(float) * (size_t)E);
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* Gated delta rule over the verify chain                                      */
/* ------------------------------------------------------------------------ */
/*
 * The hybrid models interleave attention with GatedDeltaNet layers whose
 * operators publish the recurrent state after every token of the step
 * (onnxruntime-genai PR #2457: GatedDeltaNet.checkpoints; V-major float32
 * state; a window of W slots written either at slot j after token j or with
 * slot W-1 after the last token; lmdeploy PR #5019: GDR verify kernels). The
 * pages do not state the recurrence; it is taken from the published method
 * (Yang, Kautz, Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with
 * Delta Rule", ICLR 2025). Per (row b, head h) the state S is dv x dk, V-major
 * (S[i][c], value index i, key index c), and token t updates it by
 *
 *   alpha_t = exp(g_t)                          (g_t <= 0: log decay)
 *   S_t     = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
 *   o_t     = S_t (scale q_t)
 *
 * which is S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T written
 * out. S_0 is the live state; slot base + t of the window receives S_{t+1}
 * (the state after input t), base = 0 (token alignment) or W - R (last).
 * Everything is computed in double; the snapshots and outputs are rounded to
 * float when stored, the running state stays in double.
 *
 * Layouts: q, k [B,R,H,dk]; v [B,R,H,dv]; g, beta [B,R,H]; state_in
 * [B,H,dv,dk]; snapshots [B,W,H,dv,dk]; out [B,R,H,dv]. All float.
 */
int oracle_gdn_verify(const float* q, const float* k, const float* v, const float* g, const float* beta,
                      double scale, const float* state_in, float* snapshots, float* out, int B, int R, int H,
                      int dk, int dv, int W, int alignment, int n_threads) {
  if (!q || !k || !v || !g || !beta || !state_in || !snapshots || !out) return ORACLE_ERR_ARG;
  if (B < 0 || R < 1 || H < 1 || dk < 1 || dv < 1 || W < R || (alignment != 0 && alignment != 1))
    return ORACLE_ERR_ARG;
  const int base = alignment == 0 ? 0 : W - R;
  const int64_t E = (int64_t)dv * dk;
  int err = ORACLE_OK;
  set_threads(n_threads);
#pragma omp parallel
  {
    double* S = (double*)malloc(sizeof(double) * (size_t)E);
    double* Sk = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!S || !Sk) {
#pragma omp critical
      err = ORACLE_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic)
    for (int64_t unit = 0; unit < (int64_t)B * H; ++unit) {
      if (!S || !Sk) continue;
      const int64_t b = unit / H, h = unit % H;
      const float* s0 = state_in + unit * E;
      for (int64_t e = 0; e < E; ++e) S[e] = s0[e];
      for (int t = 0; t < R; ++t) {
        const int64_t tok = (b * R + t) * H + h;
        const float* kt = k + tok * dk;
        const float* qt = q + tok * dk;
        const float* vt = v + tok * dv;
        const double alpha = exp((double)g[tok]);
        const double bt = beta[tok];
        for (int i = 0; i < dv; ++i) {  /* S_{t-1} k_t */
          double acc = 0.0;
          for (int c = 0; c < dk; ++c) acc += S[(int64_t)i * dk + c] * (double)kt[c];
          Sk[i] = acc;
        }
        for (int i = 0; i < dv; ++i) {
          const double u = (double)vt[i] - alpha * Sk[i];
          for (int c = 0; c < dk; ++c) S[(int64_t)i * dk + c] = alpha * S[(int64_t)i * dk + c] + bt * u * (double)kt[c];
        }
        float* o = out + tok * dv;
        for (int i = 0; i < dv; ++i) {  /* o_t = S_t (scale q_t) */
          double acc = 0.0;
          for (int c = 0; c < dk; ++c) acc += S[(int64_t)i * dk + c] * (scale * (double)qt[c]);
          o[i] = (float)acc;
        }
        float* snap = snapshots + ((b * W + base + t) * H + h) * E;
        for (int64_t e = 0; e < E; ++e) snap[e] = (float)S[e];
      }
    }
    free(S);
    free(Sk);
  }
  return err;
}
