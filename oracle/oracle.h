/*
 * oracle.h -- plain CPU reference of one MoE decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this code; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no source with the CUDA library: the
 * only code both sides use is the seeded input generator (synth/), which
 * holds none of the method's arithmetic.
 *
 * What it computes (one decode step of a parallel-residual MoE transformer,
 * batch 1..8, paged KV) follows the three pages about the persistent decode
 * megakernel for a 30B-total / 3.3B-active MoE model:
 *   - the op list: "Cohere Packs the Entire Decoding Step Into a Single CUDA
 *     Megakernel" (ainews.surl.tw), paragraph 1 (RMSNorm, QKV, attention,
 *     MoE) and "Cohere megakernel serves 30B MoE 1.58x faster than vLLM"
 *     (aiweekly.co), paragraph 2 (QKV projection, attention, MoE routing,
 *     gather, GEMMs, normalization);
 *   - attention and MoE both read the same normalized input: ainews.surl.tw,
 *     paragraph 2;
 *   - paged KV cache and ragged lengths: "Cohere speeds up North Mini Code
 *     with new megakernel" (latestnews.news), paragraph 3;
 *   - BF16 weights and KV: latestnews.news, paragraph 1.
 * Where the pages are silent (rounding points, RoPE form, routing details)
 * the readings are listed in the repository's design notes; each function
 * below names the reading it implements.
 *
 * Precision: fp32 accumulation over bf16-rounded weights and activations.
 * The accum_double argument selects the accumulation: 0 = fp32 in ascending
 * index order (the plain order of every loop), 1 = double (to measure the
 * fp32 summation-order noise against), 2 = fp32 in descending index order
 * (a second, equally faithful fp32 evaluation).
 *
 * Parity: every function here is pinned by the not-gpu tests (closed forms,
 * invariants, library routines, brute force); none is "parity unpinned".
 */
#ifndef MK_ORACLE_H
#define MK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim;
  int32_t n_experts, top_k, d_ffn, vocab, page_size;
  double rope_base;
  float rms_eps;
} orc_dims;

/* A bf16 tensor the oracle reads.  Either host data (bf16 bits, row-major),
 * a constant, or the seeded generator's values, regenerated on demand from
 * (seed, tid, sigma) so that full-scale weights need not be held in RAM. */
typedef struct {
  const uint16_t *data; /* non-NULL: materialised host data */
  uint64_t seed, tid;   /* data == NULL && !is_const: generated */
  double sigma;
  int32_t is_const;     /* 1: every element is const_bits */
  uint16_t const_bits;
} orc_tensor;

typedef struct {
  orc_tensor norm;               /* [d] */
  orc_tensor wq, wk, wv;         /* [Hq*D][d], [Hkv*D][d], [Hkv*D][d] */
  orc_tensor wo;                 /* [d][Hq*D] */
  orc_tensor wr;                 /* [E][d] */
  const float *router_bias;      /* [E] or NULL */
  orc_tensor wg, wu;             /* [E][F][d] */
  orc_tensor wd;                 /* [E][d][F] */
  orc_tensor kpool, vpool;       /* [num_pages][Hkv][P][D] (post-RoPE K) */
} orc_layer;

typedef struct {
  orc_tensor embed;              /* [V][d] */
  orc_tensor final_norm;         /* [d] */
  orc_tensor lm_head;            /* [V][d] */
  const orc_layer *layers;       /* [n_layers], copied by orc_create */
} orc_weights;

typedef struct orc_model orc_model;

/* Creates a decode state for `batch` sequences.  seq_lens[b] = cached tokens
 * L_b before the first step; page_tables = [batch][max_pages] physical page
 * ids (copied).  Returns NULL on invalid arguments. */
orc_model *orc_create(const orc_dims *dims, const orc_weights *w, int32_t batch,
                      const int32_t *seq_lens, const int32_t *page_tables,
                      int32_t max_pages, int32_t accum_double);
void orc_destroy(orc_model *m);

/* Optional per-step outputs (any pointer may be NULL). */
typedef struct {
  float *logits;            /* [B][V] */
  int32_t *next_tokens;     /* [B] argmax, ties -> lowest id */
  float *argmax_margin;     /* [B] top1 - top2 logit */
  int32_t *route_ids;       /* [L][B][k] in the order used for the sum */
  float *route_w;           /* [L][B][k] */
  float *route_margin;      /* [L][B] r_(k) - r_(k+1) of the oracle's logits */
  float *router_logits;     /* [L][B][E] fp32 (+bias) */
  uint16_t *h;              /* [L+1][B][d] residual entering each layer, then final */
  uint16_t *n;              /* [L][B][d] normed input of each layer */
  uint16_t *q;              /* [L][B][Hq*D] after RoPE */
  uint16_t *k;              /* [L][B][Hkv*D] after RoPE (the appended row) */
  uint16_t *v;              /* [L][B][Hkv*D] */
  uint16_t *o;              /* [L][B][Hq*D] attention output before Wo */
  uint16_t *attn;           /* [L][B][d] */
  uint16_t *moe;            /* [L][B][d] */
  int32_t route_mismatch;   /* out: count of (l,b) whose forced ids were rejected */
} orc_step_out;

/* One decode step: token b sits at position L_b, its K/V row is appended
 * there, and L_b advances by one.  forced_ids ([L][B][k] or NULL) is another
 * implementation's routing: at an (l, b) whose top-k margin is below
 * tie_eps the oracle adopts it if it differs from its own choice only among
 * experts within tie_eps of the k-th logit; anything else counts as a
 * mismatch and the oracle keeps its own choice.  Returns 0 on success. */
int32_t orc_step(orc_model *m, const int32_t *tokens, const int32_t *forced_ids,
                 float tie_eps, orc_step_out *out);

/* Teacher-forced evaluation, one piece of the step at a time.
 *
 * orc_layer_step: layer `layer` of the step (a1-a11) from a given residual input
 * h_in [B][d] (bf16 bits) -- another implementation's residual entering that
 * layer -- writing the residual entering the next layer to h_out [B][d].
 * Tokens sit at the current positions L_b; the attention reads the state's
 * K/V rows (cached, plus rows kept by earlier steps) and the new row.  With
 * keep = 0 the state is left unchanged; with keep = 1 the new K/V row is
 * kept (call it once per layer, then orc_advance, to replay a whole step).
 * forced_ids: this layer's [B][k] routing of the other implementation, with
 * the same near-tie rule as orc_step.  out: any of n, q, k, v, o, attn, moe,
 * router_logits, route_ids, route_w, route_margin (sized for ONE layer) and
 * route_mismatch; the other fields are ignored.
 *
 * orc_head: the final norm, LM head and argmax (a12, a13) of a given final
 * residual h_in [B][d]: out's logits, next_tokens and argmax_margin.
 *
 * orc_advance: every L_b advances by one (the end of a replayed step).
 *
 * orc_step is exactly orc_layer_step(keep = 1) for every layer, orc_head, then
 * orc_advance. */
int32_t orc_layer_step(orc_model *m, int32_t layer, const uint16_t *h_in,
                       const int32_t *forced_ids, float tie_eps, int32_t keep, uint16_t *h_out,
                       orc_step_out *out);
int32_t orc_head(orc_model *m, const uint16_t *h_in, orc_step_out *out);
int32_t orc_advance(orc_model *m);

/* Continuous batching: slot b gets a new sequence with new_len cached tokens
 * held in the pages of page_row [max_pages]; the K/V rows the slot kept from
 * earlier steps are dropped, the other slots are untouched. */
int32_t orc_reset_seq(orc_model *m, int32_t b, int32_t new_len, const int32_t *page_row);

/* ---- the building blocks, exposed for the pin tests ---------------------- */

/* out = bf16(h * (1/sqrtf(mean_fp32(h^2) + eps)) * g); all bf16 bits. */
void orc_rmsnorm(const uint16_t *h, const uint16_t *g, int32_t d, float eps,
                 int32_t accum_double, uint16_t *out);
/* out[r] = sum_k W[r][k] x[k] (fp32 or double accumulation), W bf16 [rows][cols]. */
void orc_gemv(const uint16_t *w, int32_t rows, int32_t cols, const uint16_t *x,
              int32_t accum_double, float *out);
/* In-place rotate-half RoPE on x [n_heads][D] (bf16) at position pos. */
void orc_rope(uint16_t *x, int32_t n_heads, int32_t head_dim, int64_t pos, double base);
/* One query head over n keys: o = bf16(softmax(q.K^T / sqrt(D)) V). */
void orc_attention_head(const uint16_t *q, const uint16_t *keys, const uint16_t *vals,
                        int32_t n, int32_t head_dim, int32_t accum_double, uint16_t *out);
/* Router: ids/w of the top k of logits[E] (ties -> lower id), weights
 * renormalised over the top k; margin = r_(k) - r_(k+1). */
void orc_route(const float *logits, int32_t n_experts, int32_t k, int32_t *ids,
               float *w, float *margin);
/* silu(x) = x / (1 + exp(-x)) in fp32. */
float orc_silu(float x);
/* One expert: y[d] = fp32(a . Wd^T), a = bf16(silu(bf16(n.Wg^T)) * bf16(n.Wu^T)). */
void orc_expert(const uint16_t *n, const uint16_t *wg, const uint16_t *wu,
                const uint16_t *wd, int32_t d, int32_t f, int32_t accum_double,
                float *y);

#ifdef __cplusplus
}
#endif

#endif /* MK_ORACLE_H */
