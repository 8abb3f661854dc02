/*
 * oracle.cpp -- plain CPU reference of one MoE decode step (see oracle.h).
 *
 * TEST INFRASTRUCTURE ONLY: never linked into, or called by, the product.
 *
 * Written from the method's definition, not for speed: every sum runs in
 * its plain index order, every rounding point is explicit.  OpenMP only
 * splits independent output rows / heads across threads, so the thread
 * count never changes a result.  Build with -ffp-contract=off so that each
 * product is rounded to fp32 before it is added (the textbook fp32 dot
 * product).
 */
#include "oracle.h"

#include <math.h>
#include <string.h>

#include <algorithm>
#include <limits>
#include <vector>

#include "../synth/synth_rng.h" /* the seeded input generator (inputs only) */

namespace {

/* ---- bf16 <-> fp32 (the oracle's own conversion; round to nearest even) --- */

float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0; /* NaN */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

float round_bf16(float f) { return bf16_to_f32(f32_to_bf16(f)); }

/* ---- tensor access -------------------------------------------------------- */

struct Tensor {
  orc_tensor t;
  uint64_t key;
  explicit Tensor(const orc_tensor &src = orc_tensor()) : t(src), key(0) {
    if (!t.data && !t.is_const) key = syn_key(t.seed, t.tid);
  }
  uint16_t bits(int64_t i) const {
    if (t.data) return t.data[i];
    if (t.is_const) return t.const_bits;
    return syn_normal_bf16(key, (uint64_t)i, t.sigma);
  }
  /* out[j] = element (row * cols + j) as float, j < cols. */
  void row(int64_t r, int64_t cols, float *out) const {
    const int64_t base = r * cols;
    for (int64_t j = 0; j < cols; ++j) out[j] = bf16_to_f32(bits(base + j));
  }
};

/* ---- dot product: the only accumulation primitive -------------------------
 * acc: ACC_F32 (fp32, ascending index order), ACC_F64 (double), ACC_F32_REV
 * (fp32, descending index order).  The method fixes fp32 accumulation but
 * not the order of the sum; the two fp32 orders are equally faithful, and
 * how far each lands from the double evaluation measures the method's own
 * rounding noise. */
enum { ACC_F32 = 0, ACC_F64 = 1, ACC_F32_REV = 2 };

float dot(const float *a, const float *b, int64_t n, int acc) {
  if (acc == ACC_F64) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += (double)a[i] * (double)b[i];
    return (float)s;
  }
  float s = 0.0f;
  if (acc == ACC_F32_REV)
    for (int64_t i = n - 1; i >= 0; --i) s += a[i] * b[i];
  else
    for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

/* y[r] = dot(W[row0 + r], x), r < rows; W is a [*][cols] tensor. */
void gemv(const Tensor &w, int64_t row0, int64_t rows, int64_t cols, const float *x,
          int dbl, float *y) {
#pragma omp parallel
  {
    std::vector<float> buf(cols);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      w.row(row0 + r, cols, buf.data());
      y[r] = dot(buf.data(), x, cols, dbl);
    }
  }
}

/* ---- the method's steps ------------------------------------------------------ */

/* RMSNorm (design reading R5): fp32 mean of squares, 1/sqrtf, one bf16
 * rounding of (h * r) * g. */
void rmsnorm(const float *h, const Tensor &g, int64_t d, float eps, int dbl, float *out) {
  const float ss = dot(h, h, d, dbl);
  const float mean = ss / (float)d;
  const float r = 1.0f / sqrtf(mean + eps);
  for (int64_t i = 0; i < d; ++i) out[i] = round_bf16((h[i] * r) * bf16_to_f32(g.bits(i)));
}

/* RoPE (reading R4): rotate-half pairs (i, i + D/2), inv_freq_i =
 * base^(-2i/D), angle pos * inv_freq in double, cos/sin in double then fp32;
 * the rotation itself in fp32, rounded to bf16. */
void rope(float *x, int64_t n_heads, int64_t D, int64_t pos, double base) {
  const int64_t half = D / 2;
  for (int64_t i = 0; i < half; ++i) {
    const double inv_freq = pow(base, -2.0 * (double)i / (double)D);
    const double ang = (double)pos * inv_freq;
    const float c = (float)cos(ang), s = (float)sin(ang);
    for (int64_t h = 0; h < n_heads; ++h) {
      float *xh = x + h * D;
      const float x1 = xh[i], x2 = xh[i + half];
      const float a = x1 * c;
      const float b = x2 * s;
      const float e = x2 * c;
      const float f = x1 * s;
      xh[i] = round_bf16(a - b);
      xh[i + half] = round_bf16(e + f);
    }
  }
}

/* Attention of one query head over n keys (reading R7): s_j = fp32(q.k_j) *
 * (1/sqrt(D)); softmax in fp32; o = bf16((sum_j p_j v_j) / l). */
void attention_head(const float *q, const float *keys, const float *vals, int64_t n,
                    int64_t D, int dbl, float *o) {
  const float scale = (float)(1.0 / sqrt((double)D));
  std::vector<float> s(n);
  float m = -std::numeric_limits<float>::infinity();
  for (int64_t j = 0; j < n; ++j) {
    s[j] = dot(q, keys + j * D, D, dbl) * scale;
    m = std::max(m, s[j]);
  }
  std::vector<float> p(n);
  for (int64_t j = 0; j < n; ++j) p[j] = expf(s[j] - m);
  /* Each output dim sums over j in ascending order; the j-outer loop order
   * only keeps the value rows in cache. */
  if (dbl == ACC_F64) {
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) l += (double)p[j];
    std::vector<double> acc(D, 0.0);
    for (int64_t j = 0; j < n; ++j)
      for (int64_t e = 0; e < D; ++e) acc[e] += (double)p[j] * (double)vals[j * D + e];
    for (int64_t e = 0; e < D; ++e) o[e] = round_bf16((float)(acc[e] / l));
    return;
  }
  float l = 0.0f;
  std::vector<float> acc(D, 0.0f);
  for (int64_t jj = 0; jj < n; ++jj) {
    const int64_t j = dbl == ACC_F32_REV ? n - 1 - jj : jj;
    l += p[j];
    for (int64_t e = 0; e < D; ++e) acc[e] += p[j] * vals[j * D + e];
  }
  for (int64_t e = 0; e < D; ++e) o[e] = round_bf16(acc[e] / l);
}

/* Router (reading R8): rank the fp32 logits, ties -> lower id; softmax over
 * all E; weights renormalised over the chosen k. */
void route(const float *r, int64_t E, int64_t k, int32_t *ids, float *w, float *margin) {
  std::vector<int32_t> order(E);
  for (int64_t e = 0; e < E; ++e) order[e] = (int32_t)e;
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return r[a] > r[b]; });
  float m = -std::numeric_limits<float>::infinity();
  for (int64_t e = 0; e < E; ++e) m = std::max(m, r[e]);
  std::vector<float> p(E);
  float z = 0.0f;
  for (int64_t e = 0; e < E; ++e) {
    p[e] = expf(r[e] - m);
    z += p[e];
  }
  for (int64_t e = 0; e < E; ++e) p[e] = p[e] / z;
  float sum_top = 0.0f;
  for (int64_t t = 0; t < k; ++t) sum_top += p[order[t]];
  for (int64_t t = 0; t < k; ++t) {
    ids[t] = order[t];
    w[t] = p[order[t]] / sum_top;
  }
  if (margin)
    *margin = (k < E) ? r[order[k - 1]] - r[order[k]] : std::numeric_limits<float>::infinity();
}

float silu(float x) { return x / (1.0f + expf(-x)); }

}  // namespace

/* ============================ the decode state ============================== */

struct orc_model {
  orc_dims dims;
  int dbl; /* accumulation mode (ACC_*) */
  int32_t B, max_pages;
  Tensor embed, final_norm, lm_head;
  struct Layer {
    Tensor norm, wq, wk, wv, wo, wr, wg, wu, wd, kpool, vpool;
    std::vector<float> bias; /* empty: no bias */
  };
  std::vector<Layer> layers;
  std::vector<int32_t> base_len, cur_len, page_table;
  /* appended[l][b]: post-RoPE K and V rows for positions base_len[b].. */
  std::vector<std::vector<std::vector<float>>> app_k, app_v;

  /* K or V row (all D dims of kv head h) of sequence b at position j. */
  void kv_row(int64_t l, int64_t b, int64_t h, int64_t j, bool want_v, float *out) const {
    const int64_t D = dims.head_dim, H = dims.n_kv_heads, P = dims.page_size;
    if (j >= base_len[b]) {
      const std::vector<float> &src = want_v ? app_v[l][b] : app_k[l][b];
      const float *row = src.data() + ((j - base_len[b]) * H + h) * D;
      memcpy(out, row, D * sizeof(float));
      return;
    }
    const int64_t page = page_table[b * max_pages + j / P];
    const int64_t slot = j % P;
    const Tensor &pool = want_v ? layers[l].vpool : layers[l].kpool;
    pool.row(((page * H + h) * P + slot), D, out);
  }
};

extern "C" {

orc_model *orc_create(const orc_dims *dims, const orc_weights *w, int32_t batch,
                      const int32_t *seq_lens, const int32_t *page_tables,
                      int32_t max_pages, int32_t accum_double) {
  if (!dims || !w || !w->layers || batch < 1 || !seq_lens || !page_tables) return nullptr;
  if (dims->n_q_heads % dims->n_kv_heads != 0 || dims->head_dim % 2 != 0) return nullptr;
  if (dims->top_k < 1 || dims->top_k > dims->n_experts) return nullptr;
  orc_model *m = new orc_model();
  m->dims = *dims;
  m->dbl = accum_double;
  m->B = batch;
  m->max_pages = max_pages;
  m->embed = Tensor(w->embed);
  m->final_norm = Tensor(w->final_norm);
  m->lm_head = Tensor(w->lm_head);
  m->layers.resize(dims->n_layers);
  for (int32_t l = 0; l < dims->n_layers; ++l) {
    const orc_layer &s = w->layers[l];
    orc_model::Layer &L = m->layers[l];
    L.norm = Tensor(s.norm);
    L.wq = Tensor(s.wq);
    L.wk = Tensor(s.wk);
    L.wv = Tensor(s.wv);
    L.wo = Tensor(s.wo);
    L.wr = Tensor(s.wr);
    L.wg = Tensor(s.wg);
    L.wu = Tensor(s.wu);
    L.wd = Tensor(s.wd);
    L.kpool = Tensor(s.kpool);
    L.vpool = Tensor(s.vpool);
    if (s.router_bias) L.bias.assign(s.router_bias, s.router_bias + dims->n_experts);
  }
  m->base_len.assign(seq_lens, seq_lens + batch);
  m->cur_len = m->base_len;
  m->page_table.assign(page_tables, page_tables + (int64_t)batch * max_pages);
  m->app_k.assign(dims->n_layers, std::vector<std::vector<float>>(batch));
  m->app_v.assign(dims->n_layers, std::vector<std::vector<float>>(batch));
  return m;
}

void orc_destroy(orc_model *m) { delete m; }

}  // extern "C"

namespace {

void dump16(uint16_t *dst, const float *src, int64_t n) {
  if (dst)
    for (int64_t i = 0; i < n; ++i) dst[i] = f32_to_bf16(src[i]);
}

/* One layer of the step (a1-a11) for the whole batch: h [B][d] (bf16 values
 * held as floats) is the residual entering layer l and becomes the residual
 * entering layer l + 1.  Per-(layer, token) dumps go to row `row` of out's
 * arrays.  forced_l ([B][k] or NULL) is another implementation's routing of
 * this layer (see orc_step).  Each token's new K/V row joins the state for
 * this layer's attention; unless `keep` it is taken out again afterwards, so
 * that a teacher-forced evaluation leaves the state as it found it. */
void layer_forward(orc_model *m, int64_t l, std::vector<float> &h, const int32_t *forced_l,
                   float tie_eps, orc_step_out *out, int64_t row, bool keep) {
  const orc_dims &dm = m->dims;
  const int64_t B = m->B, d = dm.d_model, Hq = dm.n_q_heads, Hkv = dm.n_kv_heads;
  const int64_t D = dm.head_dim, G = Hq / Hkv, E = dm.n_experts, K = dm.top_k;
  const int64_t F = dm.d_ffn;
  const int dbl = m->dbl;
  std::vector<float> n(B * d), q(Hq * D), kk(Hkv * D), vv(Hkv * D), o(Hq * D);
  std::vector<float> attn(B * d), moe(B * d), r(E), y(d), acc(d), a(F), g(F), u(F);
  std::vector<int32_t> ids(K);
  std::vector<float> wts(K);
  const orc_model::Layer &Ly = m->layers[l];

  for (int64_t b = 0; b < B; ++b) {
    const float *hb = &h[b * d];
    float *nb = &n[b * d];
    /* a1: one RMSNorm; attention and MoE both read nb (reading R1). */
    rmsnorm(hb, Ly.norm, d, dm.rms_eps, dbl, nb);
    if (out->n) dump16(out->n + (row * B + b) * d, nb, d);

    /* a2: QKV projections, bf16 outputs (reading R3). */
    gemv(Ly.wq, 0, Hq * D, d, nb, dbl, q.data());
    gemv(Ly.wk, 0, Hkv * D, d, nb, dbl, kk.data());
    gemv(Ly.wv, 0, Hkv * D, d, nb, dbl, vv.data());
    for (auto &x : q) x = round_bf16(x);
    for (auto &x : kk) x = round_bf16(x);
    for (auto &x : vv) x = round_bf16(x);

    /* a3: RoPE at position L_b, then append K/V there (reading R6). */
    const int64_t pos = m->cur_len[b];
    rope(q.data(), Hq, D, pos, dm.rope_base);
    rope(kk.data(), Hkv, D, pos, dm.rope_base);
    if (out->q) dump16(out->q + (row * B + b) * Hq * D, q.data(), Hq * D);
    if (out->k) dump16(out->k + (row * B + b) * Hkv * D, kk.data(), Hkv * D);
    if (out->v) dump16(out->v + (row * B + b) * Hkv * D, vv.data(), Hkv * D);
    std::vector<float> &ak = m->app_k[l][b], &av = m->app_v[l][b];
    ak.insert(ak.end(), kk.begin(), kk.end());
    av.insert(av.end(), vv.begin(), vv.end());

    /* a4+a5: attention over the pos + 1 keys (cached + the new one). */
    const int64_t nkeys = pos + 1;
    std::vector<float> keys(Hkv * nkeys * D), vals(Hkv * nkeys * D); /* [hk][j][D] */
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < nkeys; ++j)
      for (int64_t hk = 0; hk < Hkv; ++hk) {
        m->kv_row(l, b, hk, j, false, &keys[(hk * nkeys + j) * D]);
        m->kv_row(l, b, hk, j, true, &vals[(hk * nkeys + j) * D]);
      }
    /* GQA: query head i reads kv head i / G. */
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < Hq; ++i) {
      const int64_t hk = i / G;
      attention_head(&q[i * D], &keys[hk * nkeys * D], &vals[hk * nkeys * D], nkeys, D,
                     dbl, &o[i * D]);
    }
    if (out->o) dump16(out->o + (row * B + b) * Hq * D, o.data(), Hq * D);
    if (!keep) { /* a teacher-forced evaluation leaves the state as it was */
      ak.resize(ak.size() - Hkv * D);
      av.resize(av.size() - Hkv * D);
    }

    /* a6: output projection. */
    gemv(Ly.wo, 0, d, Hq * D, o.data(), dbl, &attn[b * d]);
    for (int64_t i = 0; i < d; ++i) attn[b * d + i] = round_bf16(attn[b * d + i]);

    /* a7: router logits (fp32, + bias), top-k, renormalised weights. */
    gemv(Ly.wr, 0, E, d, nb, dbl, r.data());
    if (!Ly.bias.empty())
      for (int64_t e = 0; e < E; ++e) r[e] = r[e] + Ly.bias[e];
    if (out->router_logits) memcpy(out->router_logits + (row * B + b) * E, r.data(), E * 4);
    float margin;
    route(r.data(), E, K, ids.data(), wts.data(), &margin);
    if (out->route_margin) out->route_margin[row * B + b] = margin;

    if (forced_l) {
      /* Adopt the other side's choice only where it differs among near ties. */
      const int32_t *fid = forced_l + b * K;
      const float rk = r[ids[K - 1]];
      bool same = true, ok = true;
      std::vector<char> in_own(E, 0), in_forced(E, 0);
      for (int64_t t = 0; t < K; ++t) in_own[ids[t]] = 1;
      for (int64_t t = 0; t < K; ++t) {
        if (fid[t] < 0 || fid[t] >= E || in_forced[fid[t]]) { ok = false; break; }
        in_forced[fid[t]] = 1;
      }
      if (ok)
        for (int64_t e = 0; e < E; ++e)
          if (in_own[e] != in_forced[e]) {
            same = false;
            if (!(margin < tie_eps) || fabsf(r[e] - rk) >= tie_eps) ok = false;
          }
      if (!ok) {
        out->route_mismatch += 1;
      } else if (!same) {
        /* Use the forced set, ranked by the oracle's logits (ties -> lower id). */
        std::vector<int32_t> set(fid, fid + K);
        std::stable_sort(set.begin(), set.end(), [&](int32_t x, int32_t z) {
          return r[x] > r[z] || (r[x] == r[z] && x < z);
        });
        float mx = -std::numeric_limits<float>::infinity();
        for (int64_t e = 0; e < E; ++e) mx = std::max(mx, r[e]);
        float zsum = 0.0f;
        for (int64_t e = 0; e < E; ++e) zsum += expf(r[e] - mx);
        float st = 0.0f;
        std::vector<float> p(K);
        for (int64_t t = 0; t < K; ++t) {
          p[t] = expf(r[set[t]] - mx) / zsum;
          st += p[t];
        }
        for (int64_t t = 0; t < K; ++t) {
          ids[t] = set[t];
          wts[t] = p[t] / st;
        }
      }
    }
    if (out->route_ids) memcpy(out->route_ids + (row * B + b) * K, ids.data(), K * 4);
    if (out->route_w) memcpy(out->route_w + (row * B + b) * K, wts.data(), K * 4);

    /* a8-a10: chosen experts' SwiGLU, weighted fp32 combine, one rounding. */
    for (int64_t i = 0; i < d; ++i) acc[i] = 0.0f;
    for (int64_t t = 0; t < K; ++t) {
      const int64_t e = ids[t];
      gemv(Ly.wg, e * F, F, d, nb, dbl, g.data());
      gemv(Ly.wu, e * F, F, d, nb, dbl, u.data());
      for (int64_t f = 0; f < F; ++f) {
        const float gb = round_bf16(g[f]), ub = round_bf16(u[f]);
        a[f] = round_bf16(silu(gb) * ub);
      }
      gemv(Ly.wd, e * d, d, F, a.data(), dbl, y.data());
      for (int64_t i = 0; i < d; ++i) acc[i] = acc[i] + wts[t] * y[i];
    }
    for (int64_t i = 0; i < d; ++i) moe[b * d + i] = round_bf16(acc[i]);
  }
  if (out->attn) dump16(out->attn + (row * B) * d, attn.data(), B * d);
  if (out->moe) dump16(out->moe + (row * B) * d, moe.data(), B * d);

  /* a11: residual, h <- bf16((h + attn) + moe) (reading R10). */
  for (int64_t i = 0; i < B * d; ++i) h[i] = round_bf16((h[i] + attn[i]) + moe[i]);
}

/* The final norm, LM head and greedy argmax (a12, a13) of the final
 * residual h [B][d]. */
void head_forward(orc_model *m, const std::vector<float> &h, orc_step_out *out) {
  const orc_dims &dm = m->dims;
  const int64_t B = m->B, d = dm.d_model, V = dm.vocab;
  const int dbl = m->dbl;
  std::vector<float> n(B * d), logits(V);
  for (int64_t b = 0; b < B; ++b) {
    rmsnorm(&h[b * d], m->final_norm, d, dm.rms_eps, dbl, &n[b * d]);
    gemv(m->lm_head, 0, V, d, &n[b * d], dbl, logits.data());
    if (out->logits) memcpy(out->logits + b * V, logits.data(), V * 4);
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
      if (logits[v] > logits[best]) best = v;
    float second = -std::numeric_limits<float>::infinity();
    for (int64_t v = 0; v < V; ++v)
      if (v != best) second = std::max(second, logits[v]);
    if (out->next_tokens) out->next_tokens[b] = (int32_t)best;
    if (out->argmax_margin) out->argmax_margin[b] = logits[best] - second;
  }
}

}  // namespace

extern "C" {

int32_t orc_step(orc_model *m, const int32_t *tokens, const int32_t *forced_ids,
                 float tie_eps, orc_step_out *out) {
  if (!m || !tokens) return -1;
  const orc_dims &dm = m->dims;
  const int64_t B = m->B, d = dm.d_model, K = dm.top_k, V = dm.vocab, L = dm.n_layers;
  orc_step_out dummy;
  memset(&dummy, 0, sizeof(dummy));
  if (!out) out = &dummy;
  out->route_mismatch = 0;

  for (int64_t b = 0; b < B; ++b)
    if (tokens[b] < 0 || tokens[b] >= V) return -2;

  /* a0: embedding rows. h holds bf16 values as floats. */
  std::vector<float> h(B * d);
  for (int64_t b = 0; b < B; ++b) m->embed.row(tokens[b], d, &h[b * d]);

  for (int64_t l = 0; l < L; ++l) {
    if (out->h) dump16(out->h + (l * B) * d, h.data(), B * d);
    layer_forward(m, l, h, forced_ids ? forced_ids + l * B * K : nullptr, tie_eps, out, l, true);
  }
  if (out->h) dump16(out->h + (L * B) * d, h.data(), B * d);
  head_forward(m, h, out);
  for (int64_t b = 0; b < B; ++b) m->cur_len[b] += 1;
  return 0;
}

int32_t orc_layer_step(orc_model *m, int32_t layer, const uint16_t *h_in,
                       const int32_t *forced_ids, float tie_eps, int32_t keep, uint16_t *h_out,
                       orc_step_out *out) {
  if (!m || !h_in || layer < 0 || layer >= m->dims.n_layers) return -1;
  const int64_t B = m->B, d = m->dims.d_model;
  orc_step_out dummy;
  memset(&dummy, 0, sizeof(dummy));
  if (!out) out = &dummy;
  out->route_mismatch = 0;
  std::vector<float> h(B * d);
  for (int64_t i = 0; i < B * d; ++i) h[i] = bf16_to_f32(h_in[i]);
  layer_forward(m, layer, h, forced_ids, tie_eps, out, 0, keep != 0);
  dump16(h_out, h.data(), B * d);
  return 0;
}

int32_t orc_head(orc_model *m, const uint16_t *h_in, orc_step_out *out) {
  if (!m || !h_in) return -1;
  const int64_t B = m->B, d = m->dims.d_model;
  orc_step_out dummy;
  memset(&dummy, 0, sizeof(dummy));
  if (!out) out = &dummy;
  std::vector<float> h(B * d);
  for (int64_t i = 0; i < B * d; ++i) h[i] = bf16_to_f32(h_in[i]);
  head_forward(m, h, out);
  return 0;
}

int32_t orc_reset_seq(orc_model *m, int32_t b, int32_t new_len, const int32_t *page_row) {
  if (!m || b < 0 || b >= m->B || new_len < 0 || !page_row) return -1;
  m->base_len[b] = new_len;
  m->cur_len[b] = new_len;
  memcpy(&m->page_table[(int64_t)b * m->max_pages], page_row, m->max_pages * sizeof(int32_t));
  for (int64_t l = 0; l < m->dims.n_layers; ++l) {
    m->app_k[l][b].clear();
    m->app_v[l][b].clear();
  }
  return 0;
}

int32_t orc_advance(orc_model *m) {
  if (!m) return -1;
  for (int64_t b = 0; b < m->B; ++b) m->cur_len[b] += 1;
  return 0;
}

/* ---- building blocks for the pin tests ------------------------------------ */

void orc_rmsnorm(const uint16_t *h, const uint16_t *g, int32_t d, float eps,
                 int32_t accum_double, uint16_t *out) {
  std::vector<float> hf(d), of(d);
  for (int32_t i = 0; i < d; ++i) hf[i] = bf16_to_f32(h[i]);
  orc_tensor gt;
  memset(&gt, 0, sizeof(gt));
  gt.data = g;
  rmsnorm(hf.data(), Tensor(gt), d, eps, accum_double, of.data());
  for (int32_t i = 0; i < d; ++i) out[i] = f32_to_bf16(of[i]);
}

void orc_gemv(const uint16_t *w, int32_t rows, int32_t cols, const uint16_t *x,
              int32_t accum_double, float *out) {
  std::vector<float> xf(cols);
  for (int32_t i = 0; i < cols; ++i) xf[i] = bf16_to_f32(x[i]);
  orc_tensor wt;
  memset(&wt, 0, sizeof(wt));
  wt.data = w;
  gemv(Tensor(wt), 0, rows, cols, xf.data(), accum_double, out);
}

void orc_rope(uint16_t *x, int32_t n_heads, int32_t head_dim, int64_t pos, double base) {
  const int64_t n = (int64_t)n_heads * head_dim;
  std::vector<float> xf(n);
  for (int64_t i = 0; i < n; ++i) xf[i] = bf16_to_f32(x[i]);
  rope(xf.data(), n_heads, head_dim, pos, base);
  for (int64_t i = 0; i < n; ++i) x[i] = f32_to_bf16(xf[i]);
}

void orc_attention_head(const uint16_t *q, const uint16_t *keys, const uint16_t *vals,
                        int32_t n, int32_t head_dim, int32_t accum_double, uint16_t *out) {
  const int64_t D = head_dim;
  std::vector<float> qf(D), kf(n * D), vf(n * D), of(D);
  for (int64_t i = 0; i < D; ++i) qf[i] = bf16_to_f32(q[i]);
  for (int64_t i = 0; i < n * D; ++i) {
    kf[i] = bf16_to_f32(keys[i]);
    vf[i] = bf16_to_f32(vals[i]);
  }
  attention_head(qf.data(), kf.data(), vf.data(), n, D, accum_double, of.data());
  for (int64_t i = 0; i < D; ++i) out[i] = f32_to_bf16(of[i]);
}

void orc_route(const float *logits, int32_t n_experts, int32_t k, int32_t *ids, float *w,
               float *margin) {
  route(logits, n_experts, k, ids, w, margin);
}

float orc_silu(float x) { return silu(x); }

void orc_expert(const uint16_t *n, const uint16_t *wg, const uint16_t *wu,
                const uint16_t *wd, int32_t d, int32_t f, int32_t accum_double, float *y) {
  const int dbl = accum_double;
  std::vector<float> nf(d), g(f), u(f), a(f);
  for (int32_t i = 0; i < d; ++i) nf[i] = bf16_to_f32(n[i]);
  orc_tensor t;
  memset(&t, 0, sizeof(t));
  t.data = wg;
  gemv(Tensor(t), 0, f, d, nf.data(), dbl, g.data());
  t.data = wu;
  gemv(Tensor(t), 0, f, d, nf.data(), dbl, u.data());
  for (int32_t i = 0; i < f; ++i) a[i] = round_bf16(silu(round_bf16(g[i])) * round_bf16(u[i]));
  t.data = wd;
  gemv(Tensor(t), 0, d, f, a.data(), dbl, y);
}

}  // extern "C"
