/*
 * mk_schedule.cpp -- host-side task-table builder.
 *
 * The pages describe a host-built, static, fine-grained task table that
 * assigns GEMM tiles and attention splits to the SMs, each SM running one
 * threadblock ("Cohere Packs the Entire Decoding Step Into a Single CUDA
 * Megakernel", ainews.surl.tw, paragraph 2; "Cohere speeds up North Mini
 * Code with new megakernel", latestnews.news, paragraph 3).  This builder
 * produces that table for any SM count the device reports.
 *
 * Shape of the table: one row per CTA = [header][per-layer template]
 * [final tasks].  The template is executed once per layer, so the table
 * stays small (a few hundred descriptors) for any depth.
 *
 * Per-layer phases, in the order every CTA runs them:
 *   QKV     (the [Wq | Wk | Wv] rows cut per matrix into one contiguous
 *            piece per CTA, preceded by about E / n_cta router rows; every
 *            consumer of the routing takes the top-k itself from the logits)
 *   ATTN    (split-K attention: the CTAs are shared out among the
 *            (sequence, kv head) pairs in proportion to their pages, one
 *            split of about equal size per CTA)
 *   UP      (one share per CTA of the gate/up rows of the experts the
 *            router chose; the share is resolved on the device; at batch 1
 *            the share also takes its columns of the down rows)
 *   DOWN    (batch >= 2: one share per CTA of the chosen experts' down rows)
 *   OUT     (rows of d: Wo rows, the experts' weighted down results, then
 *            the residual; this produces the next layer's input)
 * then the LM head rows, one piece per CTA.
 *
 * Deadlock freedom: a task only waits on counters fed by tasks of an
 * earlier phase (or an earlier layer), and every CTA runs its tasks in
 * phase order, so by induction over phases every wait is eventually met
 * as long as all CTAs are co-resident (the launch is cooperative).
 */
#include <algorithm>
#include <cmath>
#include <array>
#include <cstring>
#include <numeric>
#include <vector>

#include "mk.h"
#include "mk_internal.h"
#include "mk_plan.h"

namespace {

using Desc = std::array<int32_t, MK_DESC_INTS>;

Desc desc(int op) {
  Desc d;
  d.fill(0);
  d[0] = op;
  return d;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" size_t mk_misc_bytes(int nb);

int mk_nb_for(int batch) { return batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8; }

/* The scratch buffer: the largest of what the task types stage there (bf16
 * vectors at pitch K). */
static size_t xn_bytes_for(const mk_model_dims &d, int nb) {
  return align_up((size_t)nb * 2 * mk_x_pitch(d.d_model, nb), 128);
}

static size_t xbuf_bytes_for(const mk_model_dims &d, int nb) {
  const size_t HqD = (size_t)d.n_q_heads * d.head_dim, D = d.head_dim;
  size_t x = (size_t)nb * 2 * d.d_model;                         /* staged h of the norm */
  /* the attention output (Wo's input) is staged across the normed-input
   * buffer and this one, which follows it: the normed input is dead by then */
  const size_t wo_in = (size_t)nb * 2 * mk_x_pitch((int)HqD, nb), xn = xn_bytes_for(d, nb);
  x = std::max(x, wo_in > xn ? wo_in - xn : (size_t)0);
  x = std::max(x, (size_t)nb * 2 * mk_x_pitch(d.d_ffn, nb));          /* one expert's activations */
  /* attention: q (bf16 [8][D + 8]), new k and v (fp32 [D] each), merge
   * scratch fp32 [4][8][D + 8] */
  x = std::max(x, 8 * (D + 8) * 2 + 2 * D * 4 + 4 * 8 * (D + 8) * 4);
  /* cross-split merge: m and l of up to 256 splits x 8 heads, then 2 x 8 */
  x = std::max(x, (size_t)(2 * 256 * MK_MAX_GROUP + 2 * MK_MAX_GROUP) * 4);
  return align_up(x, 128); /* only the ring needs 1024-byte alignment */
}

bool mk_smem_plan(const mk_model_dims *dm, int nb, MkSmem *out) {
  const mk_model_dims &d = *dm;
  MkSmem s;
  s.misc = align_up(mk_misc_bytes(nb), 128);
  s.xbuf = xbuf_bytes_for(d, nb);
  s.xn = xn_bytes_for(d, nb);
  const size_t fixed = MK_SMEM_STATIC + s.xn + s.xbuf + s.misc;
  if (fixed >= MK_SMEM_OPTIN) return false;
  size_t sb = (MK_SMEM_OPTIN - fixed) / MK_NC_WARPS / 1024 * 1024;
  sb = std::min<size_t>(sb, MK_MAX_STAGE_BYTES);
  s.stage_bytes = (int)sb;
  s.ring_slots = MK_NC_WARPS;
  const int HqD = d.n_q_heads * d.head_dim;
  if (mk_rows_per_stage(d.d_model, s.stage_bytes, nb) < 2 ||
      mk_rows_per_stage(HqD, s.stage_bytes, nb) < 1 ||
      mk_rows_per_stage(d.d_ffn, s.stage_bytes, nb) < 1 ||
      mk_pages_per_stage(d.page_size, d.head_dim, s.stage_bytes) < 1)
    return false;
  s.total = (size_t)MK_NC_WARPS * sb + s.xn + s.xbuf + s.misc;
  s.dyn = s.total + MK_SMEM_STATIC;
  *out = s;
  return true;
}

/* Library-internal (tests): the ring geometry of the nb-token kernel --
 * stage bytes, the rows of K bf16 one stage holds, and the total dynamic
 * shared memory; 0 when the model does not fit. */
extern "C" int mk_stage_geometry(const mk_model_dims *d, int nb, int K, int32_t *stage_bytes,
                                 int32_t *rows, int64_t *dyn_bytes) {
  MkSmem sm;
  if (!d || !mk_smem_plan(d, nb, &sm)) return 0;
  if (stage_bytes) *stage_bytes = sm.stage_bytes;
  if (rows) *rows = mk_rows_per_stage(K, sm.stage_bytes, nb);
  if (dyn_bytes) *dyn_bytes = (int64_t)sm.dyn;
  return 1;
}

int mk_fold_rows(const mk_model_dims *d) {
  MkSmem sm;
  int lim = 64;
  if (mk_smem_plan(d, 1, &sm)) lim = std::min(256, sm.stage_bytes / (MK_FOLD_COLS * 2));
  /* the largest multiple of 8 that fits a stage and divides d (d is a
   * multiple of 64), so that a box never reaches into the next expert */
  for (int r = lim / 8 * 8; r >= 8; r -= 8)
    if (d->d_model % r == 0) return r;
  return 8;
}

mk_status mk_validate_dims(const mk_model_dims *dm) {
  if (!dm) return MK_ERR_INVALID_ARG;
  const mk_model_dims &d = *dm;
  if (d.n_layers < 1 || d.d_model < 1 || d.n_q_heads < 1 || d.n_kv_heads < 1 || d.head_dim < 1 ||
      d.n_experts < 1 || d.top_k < 1 || d.d_ffn < 1 || d.vocab < 1 || d.page_size < 1 ||
      d.max_batch < 1 || d.num_pages < 1 || d.max_pages_per_seq < 1)
    return MK_ERR_INVALID_ARG;
  if (d.top_k > d.n_experts) return MK_ERR_INVALID_ARG;
  if (d.n_q_heads % d.n_kv_heads != 0) return MK_ERR_INVALID_ARG;
  if (!(d.rms_eps >= 0.0f) || !(d.rope_base > 0.0f)) return MK_ERR_INVALID_ARG;
  if (d.max_batch > MK_MAX_BATCH) return MK_ERR_BATCH;
  if (d.head_dim != 32 && d.head_dim != 64 && d.head_dim != 128) return MK_ERR_UNSUPPORTED;
  /* attention runs on 16-token tensor-core tiles within a page */
  if (d.page_size % 16 || d.page_size > 256) return MK_ERR_UNSUPPORTED;
  if (d.n_q_heads / d.n_kv_heads > MK_MAX_GROUP) return MK_ERR_UNSUPPORTED;
  if (d.top_k > MK_MAX_TOPK || d.n_experts > 128) return MK_ERR_UNSUPPORTED;
  if (d.d_model % 64 || d.d_ffn % 64 || (d.n_q_heads * d.head_dim) % 64) return MK_ERR_UNSUPPORTED;
  if (d.d_model > 16384 || d.d_ffn > 16384 || d.n_q_heads * d.head_dim > 16384)
    return MK_ERR_UNSUPPORTED;
  /* every streamed unit must fit one ring slot of every batch bucket used */
  for (int nb = 1; nb <= mk_nb_for(d.max_batch); nb *= 2) {
    MkSmem sm;
    if (!mk_smem_plan(&d, nb, &sm)) return MK_ERR_UNSUPPORTED;
  }
  return MK_OK;
}

mk_status mk_build_plan(const mk_model_dims *dm, int n_cta, int batch, const int32_t *seq_lens,
                        MkPlan *out, double u_seen) {
  mk_status st = mk_validate_dims(dm);
  if (st != MK_OK) return st;
  if (n_cta < 1 || n_cta > 256 || !seq_lens || !out) return MK_ERR_INVALID_ARG;
  if (batch < 1 || batch > dm->max_batch) return MK_ERR_BATCH;
  const mk_model_dims &d = *dm;
  const int64_t cap_tokens = (int64_t)d.max_pages_per_seq * d.page_size;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] < 0 || seq_lens[b] + 1 > cap_tokens) return MK_ERR_PAGE_OOB;

  const int Hq = d.n_q_heads, Hkv = d.n_kv_heads, D = d.head_dim, P = d.page_size;
  std::vector<std::vector<Desc>> lt(n_cta), ft(n_cta);
  std::vector<std::vector<Desc>> qkv_t(n_cta), attn_t(n_cta), up_t(n_cta), down_t(n_cta),
      out_t(n_cta);
  MkPlan &p = *out;
  p = MkPlan();

  /* QKV with the router rows.  The [q | k | v] rows are cut per matrix over
   * all CTAs in proportion to its rows (largest remainder, at least one CTA
   * each), each CTA one contiguous piece (with fewer CTAs than matrices the
   * pieces wrap around the grid).  The router rows are spread over the CTAs,
   * about E / n_cta per CTA, and stream first in the CTA's first QKV task:
   * the warp that computes a router stage signals its rows at once, so the
   * logits are complete one norm and one short GEMV after the layer's input
   * is, while the other warps go on with the QKV rows.  Every consumer of the
   * routing (producers and consumers of the expert stages alike) then takes
   * the top-k itself from the logits -- no CTA does it for the others, so no
   * further hop. */
  {
    const int64_t rows[3] = {(int64_t)Hq * D, (int64_t)Hkv * D, (int64_t)Hkv * D};
    const int64_t Rq = rows[0] + rows[1] + rows[2];
    const int E = d.n_experts;
    int nq = 0;
    int share[3];
    double rem[3];
    int used = 0;
    for (int m = 0; m < 3; ++m) {
      const double q = (double)rows[m] * n_cta / (double)Rq;
      share[m] = std::max(1, (int)q);
      rem[m] = q - share[m];
      used += share[m];
    }
    while (used < n_cta) {
      const int m = (int)(std::max_element(rem, rem + 3) - rem);
      ++share[m];
      rem[m] -= 1.0;
      ++used;
    }
    int c0 = 0;
    for (int m = 0; m < 3; ++m) {
      const int pieces = (int)std::min<int64_t>(share[m], rows[m]);
      for (int c = 0; c < pieces; ++c) {
        Desc t = desc(OP_QKV);
        t[1] = m;
        t[2] = (int32_t)(rows[m] * c / pieces);
        t[3] = (int32_t)(rows[m] * (c + 1) / pieces - t[2]);
        qkv_t[(c0 + c) % n_cta].push_back(t);
        ++nq;
      }
      c0 += share[m];
    }
    const int n_rp = std::min(n_cta, E);
    for (int c = 0; c < n_rp; ++c) {
      const int cta = (int)((int64_t)c * n_cta / n_rp); /* spread over the grid */
      if (qkv_t[cta].empty()) {
        qkv_t[cta].push_back(desc(OP_QKV)); /* a router piece alone */
        ++nq;
      }
      Desc &t = qkv_t[cta].front();
      t[4] = (int32_t)((int64_t)E * c / n_rp);
      t[5] = (int32_t)((int64_t)E * (c + 1) / n_rp - t[4]);
    }
    p.n_qkv = nq;
    p.n_router = E;
  }
  /* Roles.  With enough CTAs, attention and the experts run side by side on
   * different SMs, as the pages run them from the same normed input
   * ("Cohere Packs the Entire Decoding Step Into a Single CUDA Megakernel",
   * ainews.surl.tw, paragraph 2): CTAs [0, n_acta) take the attention splits
   * (QKV, ATTN, OUT), the others the expert gate/up shares (QKV or ROUTER,
   * UP, OUT).  The split follows the time each side takes: the KV cache's
   * bytes, weighted by the attention stage's higher compute per byte, against
   * the expected distinct experts' gate/up bytes.  With few CTAs every CTA
   * does everything. */
  /* Batch 1 folds the down projection into the gate/up shares: a share is a
   * range of 64-column blocks of the chosen experts' F, whose g and u are
   * kept in shared memory and whose down partials have one slot per block --
   * so the expert path has no second phase behind a grid-wide wait.  It needs
   * the largest share's g and u to fit the scratch buffer. */
  const int fold_blocks = std::min(d.n_experts, d.top_k) * (d.d_ffn / MK_FOLD_COLS);
  int n_acta = n_cta;
  if (n_cta >= 16) {
    double kv = 0.0;
    for (int b = 0; b < batch; ++b) kv += (double)seq_lens[b] * Hkv * D * 2 * 2;
    const double E = d.n_experts, K = d.top_k;
    /* distinct experts per layer: as observed on this batch's previous
     * steps (a skewed router picks fewer), else the uniform expectation */
    const double u_exp = u_seen > 0.0 ? std::min(u_seen, E)
                                      : E * (1.0 - std::pow(1.0 - K / E, (double)batch));
    const bool fold = mk_nb_for(batch) == 1;
    const double up = u_exp * (fold ? 3.0 : 2.0) * d.d_ffn * d.d_model * 2;
    /* SM cycles of a 24 KB attention stage (48 keys x 8 query heads, both
     * products and the online softmax) over those of a gate/up stage of the
     * same bytes (~1.5, measured on GB300), plus the merge at the end of
     * the attention side */
    constexpr double kAttnCostPerByte = 1.6;
    const double frac = kAttnCostPerByte * kv / std::max(kAttnCostPerByte * kv + up, 1.0);
    const int lo = std::min(batch * Hkv, n_cta - 1), hi = n_cta - 1;
    n_acta = std::max(std::max(lo, 1), std::min(hi, (int)std::lround(n_cta * frac)));
    /* folded blocks are whole: more expert CTAs than blocks would idle */
    if (fold) n_acta = std::max(n_acta, std::min(hi, n_cta - fold_blocks));
  }
  const bool roles = n_acta < n_cta; /* attention CTAs take no expert share */
  {
    const int n_up = n_cta - (roles ? n_acta : 0);
    const int max_blocks = (fold_blocks + n_up - 1) / n_up;
    MkSmem sm;
    /* a share's g and u are staged in the scratch buffer */
    p.fold = mk_nb_for(batch) == 1 && mk_smem_plan(&d, 1, &sm) &&
             (size_t)2 * max_blocks * MK_FOLD_COLS * sizeof(float) <= sm.xbuf;
  }

  /* ATTN: split-K over pages. */
  {
    struct Split {
      int b, kvh, p0, p1, slot, slot0, ns, last;
      int gi, gn, ng, gslot0, g2slot, g2slot0; /* two-level merge */
      int64_t pages;
    };
    std::vector<Split> splits;
    int64_t T = 0;
    std::vector<int64_t> npages(batch);
    for (int b = 0; b < batch; ++b) {
      npages[b] = ceil_div(seq_lens[b], P);
      T += npages[b] * Hkv;
    }
    /* Splits per (b, kvh) in proportion to its pages (largest remainder):
     * one split of about T / n_acta pages per attention CTA, or -- when the
     * pairs are many for the CTAs, so that rounding a pair's share would
     * leave whole pairs on one CTA -- twice as many half-size splits, packed
     * below largest first. */
    const int nbh = batch * Hkv;
    const int n_splits = nbh * 4 > n_acta ? std::min(2 * n_acta, 256) : n_acta;
    std::vector<int64_t> share(nbh, 1);
    if (nbh <= n_splits && T > 0) {
      std::vector<double> rem(nbh);
      int64_t used = 0;
      for (int i = 0; i < nbh; ++i) {
        const double q = (double)npages[i / Hkv] * n_splits / (double)T;
        share[i] = std::max<int64_t>(1, (int64_t)q);
        rem[i] = q - (double)share[i];
        used += share[i];
      }
      while (used < n_splits) {
        const int best = (int)(std::max_element(rem.begin(), rem.end()) - rem.begin());
        share[best] += 1;
        rem[best] -= 1.0;
        ++used;
      }
      while (used > n_splits) {
        int best = -1;
        for (int i = 0; i < nbh; ++i)
          if (share[i] > 1 && (best < 0 || rem[i] < rem[best])) best = i;
        if (best < 0) break;
        share[best] -= 1;
        rem[best] += 1.0;
        --used;
      }
    }
    int slot = 0, slot2 = 0;
    for (int b = 0; b < batch; ++b)
      for (int h = 0; h < Hkv; ++h) {
        const int64_t n = npages[b];
        const int ns = (int)std::max<int64_t>(1, std::min<int64_t>(share[b * Hkv + h], n));
        /* up to MK_SINGLE_MERGE splits merge in one level (one round trip
         * fewer on the layer's critical path); more merge in groups */
        const int grp = ns <= MK_SINGLE_MERGE ? ns : MK_MERGE_GROUP;
        const int ng = (ns + grp - 1) / grp;
        for (int i = 0; i < ns; ++i) {
          Split s;
          s.b = b;
          s.kvh = h;
          s.p0 = (int)(n * i / ns);
          s.p1 = (int)(n * (i + 1) / ns);
          s.slot = slot + i;
          s.slot0 = slot;
          s.ns = ns;
          s.last = (i == ns - 1);
          s.gi = i / grp;
          s.gn = std::min(grp, ns - s.gi * grp);
          s.ng = ng;
          s.gslot0 = slot + s.gi * grp;
          s.g2slot = slot2 + s.gi;
          s.g2slot0 = slot2;
          s.pages = s.p1 - s.p0 + (s.last ? 1 : 0);
          splits.push_back(s);
        }
        slot += ns;
        slot2 += ng;
      }
    p.n_attn_slots = slot;
    p.n_attn = (int)splits.size();
    /* greedy: largest first onto the least-loaded CTA */
    std::vector<int> order(splits.size());
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(),
                     [&](int x, int y) { return splits[x].pages > splits[y].pages; });
    std::vector<int64_t> load(n_acta, 0);
    std::vector<std::vector<int>> mine(n_acta);
    for (int idx : order) {
      const int c = (int)(std::min_element(load.begin(), load.end()) - load.begin());
      load[c] += splits[idx].pages + 1;
      mine[c].push_back(idx);
    }
    for (int c = 0; c < n_acta; ++c) {
      std::sort(mine[c].begin(), mine[c].end());
      for (int idx : mine[c]) {
        const Split &s = splits[idx];
        Desc t = desc(OP_ATTN);
        t[1] = s.b;
        t[2] = s.kvh;
        t[3] = s.p0;
        t[4] = s.last ? -1 : s.p1;
        t[5] = s.slot;
        t[6] = s.slot0;
        t[7] = s.ns;
        t[8] = s.last;
        t[9] = s.gi;
        t[10] = s.gn;
        t[11] = s.ng;
        t[12] = s.gslot0;
        t[13] = s.g2slot;
        t[14] = s.g2slot0;
        attn_t[c].push_back(t);
      }
    }
  }

  /* UP: one share per expert CTA (every CTA without roles), resolved on the
   * device once routing is known. */
  {
    const int c0 = roles ? n_acta : 0, n = n_cta - c0;
    for (int c = c0; c < n_cta; ++c) {
      Desc t = desc(OP_UP);
      t[1] = c - c0;
      t[2] = n;
      up_t[c].push_back(t);
    }
    p.n_up = n;
  }

  /* DOWN (unfolded): the chosen experts' down rows, U x d of them, one share
   * per CTA (every CTA: the attention CTAs take theirs after their splits),
   * resolved on the device once the routing is known.  Each share streams
   * its rows against its experts' activations and leaves the dot products
   * for the OUT tasks to weight and add. */
  if (!p.fold) {
    for (int c = 0; c < n_cta; ++c) {
      Desc t = desc(OP_DOWN);
      t[1] = c;
      t[2] = n_cta;
      down_t[c].push_back(t);
    }
    p.n_down = n_cta;
  }

  /* OUT: rows of d, in units of 8 rows (the residual is published as
   * tagged pairs of rows). */
  {
    const int u8 = d.d_model / 8;
    int n = std::min(n_cta, u8);
    if (ceil_div(u8, n) * 8 > MK_MAX_OUT_ROWS) n = (int)ceil_div(u8, MK_MAX_OUT_ROWS / 8);
    for (int i = 0; i < n; ++i) {
      Desc t = desc(OP_OUT);
      const int a = 8 * (int)((int64_t)u8 * i / n), b = 8 * (int)((int64_t)u8 * (i + 1) / n);
      t[2] = a;
      t[3] = b - a;
      out_t[i % n_cta].push_back(t);
    }
    p.n_out = n;
  }

  /* LM head: vocab rows, one piece per CTA. */
  {
    const int n = std::min(n_cta, d.vocab);
    for (int i = 0; i < n; ++i) {
      Desc t = desc(OP_LM);
      const int a = (int)((int64_t)d.vocab * i / n), b = (int)((int64_t)d.vocab * (i + 1) / n);
      t[2] = a;
      t[3] = b - a;
      t[4] = i;
      ft[i].push_back(t);
    }
    p.n_lm = n;
  }

  int width = 0, lmax = 0;
  for (int c = 0; c < n_cta; ++c) {
    for (auto *v : {&qkv_t[c], &attn_t[c], &up_t[c], &down_t[c], &out_t[c]})
      lt[c].insert(lt[c].end(), v->begin(), v->end());
    width = std::max<int>(width, 1 + (int)lt[c].size() + (int)ft[c].size());
    lmax = std::max<int>(lmax, (int)lt[c].size());
  }
  p.n_cta = n_cta;
  p.tasks_per_cta = width;
  p.n_layer_tasks_max = lmax;
  p.n_attn_done = batch * Hkv;
  p.batch = batch;
  p.table.assign((size_t)n_cta * width * MK_DESC_INTS, 0);
  for (int c = 0; c < n_cta; ++c) {
    int32_t *row = &p.table[(size_t)c * width * MK_DESC_INTS];
    Desc h = desc(OP_HEADER);
    h[1] = (int)lt[c].size();
    h[2] = (int)ft[c].size();
    std::memcpy(row, h.data(), sizeof(Desc));
    int at = 1;
    for (auto &t : lt[c]) std::memcpy(row + MK_DESC_INTS * at++, t.data(), sizeof(Desc));
    for (auto &t : ft[c]) std::memcpy(row + MK_DESC_INTS * at++, t.data(), sizeof(Desc));
  }
  p.built_lens.assign(seq_lens, seq_lens + batch);
  return MK_OK;
}

/* Library-internal (tests): mk_plan with the role split taken from an
 * observed number of distinct experts per layer, as mk_build_schedule does
 * once a schedule of the same batch size has run (u_seen <= 0: the
 * uniform-routing expectation, i.e. mk_plan). */
extern "C" mk_status mk_plan_observed(const mk_model_dims *dims, int32_t n_sm, int32_t batch,
                                      const int32_t *seq_lens, double u_seen,
                                      mk_plan_info *info, int32_t *table, int64_t cap);

extern "C" mk_status mk_plan(const mk_model_dims *dims, int32_t n_sm, int32_t batch,
                             const int32_t *seq_lens, mk_plan_info *info, int32_t *table,
                             int64_t cap) {
  return mk_plan_observed(dims, n_sm, batch, seq_lens, 0.0, info, table, cap);
}

extern "C" mk_status mk_plan_observed(const mk_model_dims *dims, int32_t n_sm, int32_t batch,
                                      const int32_t *seq_lens, double u_seen,
                                      mk_plan_info *info, int32_t *table, int64_t cap) {
  MkPlan p;
  mk_status st = mk_build_plan(dims, n_sm, batch, seq_lens, &p, u_seen > 0.0 ? u_seen : 0.0);
  if (st != MK_OK) return st;
  if (info) {
    info->n_cta = p.n_cta;
    info->tasks_per_cta = p.tasks_per_cta;
    info->n_layer_tasks_max = p.n_layer_tasks_max;
    info->n_qkv = p.n_qkv;
    info->n_router = p.n_router;
    info->n_attn = p.n_attn;
    info->n_up = p.n_up;
    info->n_out = p.n_out;
    info->n_lm = p.n_lm;
    info->n_attn_slots = p.n_attn_slots;
    info->n_down = p.n_down;
  }
  if (table) {
    if (cap < (int64_t)p.table.size()) return MK_ERR_INVALID_ARG;
    std::memcpy(table, p.table.data(), p.table.size() * sizeof(int32_t));
  }
  return MK_OK;
}
