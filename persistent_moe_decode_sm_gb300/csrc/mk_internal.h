/*
 * mk_internal.h -- types shared by the host schedule builder and the kernel.
 *
 * Task descriptors are exactly 32 int32 fields (128 bytes, one cache line),
 * the size the aiweekly.co page gives for the megakernel's descriptors
 * ("Cohere megakernel serves 30B MoE 1.58x faster than vLLM", paragraph 2).
 * The per-CTA table row is: a header, the per-layer template (run once per
 * layer, in order), then the final (LM head) tasks.
 */
#ifndef MK_INTERNAL_H
#define MK_INTERNAL_H

#include <stdint.h>

#define MK_DESC_INTS 32

/* ---- opcodes ---------------------------------------------------------------- */
enum {
  OP_HEADER = 100, /* [1] n_layer_tasks, [2] n_final_tasks */
  OP_QKV = 1,      /* [1] mat (0 q, 1 k, 2 v), [2] row0, [3] nrows (may be 0),
                      [4] router row0 (expert), [5] router rows (0: none) -- the router
                      rows stream first and each stage's warp signals its rows at once */
  OP_ATTN = 3,     /* [1] b, [2] kvh, [3] page0, [4] page1 (-1: up to the live length),
                      [5] slot (partial slot), [6] slot0 of (b,kvh), [7] n_splits,
                      [8] is_last (handles and appends the new token),
                      [9] merge group, [10] splits in the group, [11] groups of (b,kvh),
                      [12] first split slot of the group, [13] the group's level-2 slot,
                      [14] first level-2 slot of (b,kvh) */
  OP_UP = 4,       /* [1] share, [2] n_shares.  With the down projection folded in
                      (batch 1), a share is a range of 64-column blocks of the chosen
                      experts' F: their gate and up rows, then the down matrix's 64
                      columns of every row of d, giving one partial down vector per block */
  OP_OUT = 5,      /* [2] row0, [3] nrows */
  OP_LM = 6,       /* [2] row0, [3] nrows, [4] lm task index */
  OP_DOWN = 7      /* [1] share, [2] n_shares (unfolded, batch >= 2): a range of the
                      chosen experts' down rows (U x d of them, in slot order), each
                      giving the weighted-free row dot products of every token */
};

/* ---- counters ----------------------------------------------------------------
 * Every counter sits in its own 32-byte sector.  Counters are epoch based:
 * in step e (0-based since the last table build) a counter that receives n
 * increments per step is complete when it reaches (e + 1) * n (compared
 * modulo 2^32), so nothing is reset between steps. */
#define MK_CTR_STRIDE 8 /* int32s per counter */
enum {
  CTR_QKV_DONE = 0,
  CTR_ROUTER_DONE = 1, /* router logits written (counts rows: E per step) */
  CTR_ATTN_DONE = 2,
  CTR_UP_DONE = 3,
  CTR_DOWN_DONE = 4, /* unfolded expert down rows done (the OUT sums wait) */
  CTR_ATTN_TICKET0 = 5 /* + (b * n_kv_heads + kvh) * (1 + MK_MAX_MERGE_GROUPS):
                          the final merge ticket, then one ticket per merge group */
};
/* after the per-layer blocks: */
enum { GCTR_LM_TICKET = 0, GCTR_EXIT = 1, GCTR_COUNT = 2 };

/* Attention splits of one (sequence, kv head) merge in one level when there
 * are at most MK_SINGLE_MERGE of them (the last to finish merges all),
 * else in two: groups of up to MK_MERGE_GROUP splits (the last to finish
 * merges its group), then the groups (the last group merger writes the
 * output). */
#define MK_MERGE_GROUP 8
#define MK_SINGLE_MERGE 16
#define MK_MAX_MERGE_GROUPS 32

static inline int mk_ctrs_per_layer(int max_batch, int n_kv_heads) {
  return CTR_ATTN_TICKET0 + max_batch * n_kv_heads * (1 + MK_MAX_MERGE_GROUPS);
}

/* ---- limits ----------------------------------------------------------------- */
#define MK_FOLD_COLS 64  /* f columns per folded block (one 128-byte swizzled box row) */
#define MK_MAX_BATCH 8
#define MK_MAX_TOPK 16
#define MK_MAX_GROUP 8          /* q heads per kv head */
#define MK_MAX_OUT_ROWS 32      /* rows of d per OUT task (more rows: more tasks) */
#define MK_NC_WARPS 8           /* consumer warps; ring slot w belongs to consumer warp w */
#define MK_NP_WARPS 4           /* producer warps; producer k fills the ring slots = k mod 4 */
#define MK_THREADS ((MK_NC_WARPS + MK_NP_WARPS) * 32)
#define MK_MAX_STAGE_ROWS 64
#ifndef MK_MAX_STAGE_BYTES
#define MK_MAX_STAGE_BYTES 32768
#endif
#define MK_MAX_STAGE_PAGES 8
#define MK_SMEM_OPTIN 232448    /* opt-in shared memory per block on sm_100-class parts */
#define MK_SMEM_STATIC 1024     /* slack to align the ring to 1024 bytes */
#define MK_SMEM_TASKS 32        /* task descriptors of a CTA kept in shared memory (more: read from global) */

/* Routing result of one layer (for the diagnostics: every CTA takes the
 * top-k itself; CTA 0 records it here). */
typedef struct {
  int32_t U;                               /* distinct experts chosen */
  int32_t pad[3];
  int32_t expert[128];                     /* slot -> expert id (ascending) */
  float slot_w[128][MK_MAX_BATCH];         /* weight of slot u for token b (0: unused) */
  int32_t ids[MK_MAX_BATCH][MK_MAX_TOPK];  /* per token, descending logit */
  float w[MK_MAX_BATCH][MK_MAX_TOPK];
} mk_routing;

/* Device-side control block. */
typedef struct {
  uint32_t epoch;            /* steps since the last table build */
  int32_t abort;             /* set by the first failing wait; every CTA polls it */
  int32_t err_code;          /* first error (mk_status), 0 = none */
  int32_t err_cta, err_task, err_op, err_layer, err_ctr;
  int32_t err_seen, err_target;
  unsigned long long sum_experts; /* sum of U over layers and steps */
} mk_ctrl;

#define MK_PARAM_LAYERS 64

/* Per-layer device pointers (a device array of n_layers of these). */
typedef struct {
  const uint16_t *norm, *wq, *wk, *wv, *wo, *wr;
  const float *bias;
  const uint16_t *wg, *wu, *wd;
  uint16_t *kc, *vc;
} mk_layer_dev;

/* Everything the kernel needs; passed by value. */
typedef struct {
  /* dims */
  int32_t L, d, Hq, Hkv, D, E, K, F, V, P, max_pages, B;
  float eps, attn_scale;
  /* model */
  const mk_layer_dev *layers;
  /* the first MK_PARAM_LAYERS layers' norm gains, router biases and K/V
   * pools again, in the parameter space: read from the constant cache, with
   * no dependent global load at a layer's start (later layers: `layers`) */
  const uint16_t *l_norm[MK_PARAM_LAYERS];
  const float *l_bias[MK_PARAM_LAYERS];
  uint16_t *l_kc[MK_PARAM_LAYERS], *l_vc[MK_PARAM_LAYERS];
  const uint16_t *embed, *final_norm, *lm_head;
  /* step io */
  const int32_t *tokens;
  float *out_logits;          /* may be NULL */
  int32_t *out_next;
  /* workspace */
  uint16_t *h;                /* [L+1][MAXB][d]  (h[0] holds the embedding rows for dumps) */
  uint16_t *qkv;              /* [L][MAXB][(Hq+2Hkv)D] pre-RoPE q, k, v */
  uint16_t *o;                /* [L][MAXB][Hq D] */
  uint16_t *am;               /* [L][2][MAXB][d] the rounded attn and moe terms of the residual */
  float *attn_part;           /* [n_slots][G][D + 4] (m, l, -, -, o[D]), reused by every layer */
  float *attn_part2;          /* [n_slots][G][D + 4] merge-group partials (both by layer
                               * parity: [2][n_slots]...) */
  float *router_logits;       /* [L][MAXB][E] */
  mk_routing *routing;        /* [L] */
  uint16_t *act;              /* [L][Umax][MAXB][F] */
  float *lm_part;             /* [n_lm][MAXB][2] (value, index as float bits) */
  int32_t *ctr;               /* counters */
  mk_ctrl *ctrl;
  int32_t *seq_lens;          /* [MAXB] live lengths (advanced by the kernel) */
  const int32_t *page_table;  /* [MAXB][max_pages] */
  const float *rope;          /* [max_pos][D/2][2] (cos, sin), or [MAXB][D/2][2] */
  int32_t rope_max_pos;
  int32_t rope_per_seq;       /* 1: rope holds one row per sequence (this step's position) */
  const int32_t *table;       /* [n_cta][tasks_per_cta][32] */
  int32_t tasks_per_cta;
  int32_t n_slots, u_max;
  /* per-step increments of each counter */
  int32_t n_qkv, n_router, n_up, n_out, n_lm, n_attn_done; /* n_router: E (rows) */
  int32_t n_down;             /* down-row shares per layer (0 when folded) */
  float *dpart;               /* [2][u_max][MAXB][d] the down rows' dot products, by layer
                               * parity (unfolded) */
  int32_t ctrs_per_layer;
  unsigned long long wait_limit_ns;
  int32_t *err_host;          /* host-mapped mirror: [code, cta, task, op, layer, ctr, seen, target] */
  int32_t stage_bytes;        /* bytes of one ring slot (a multiple of 1024) */
  int32_t ring_slots;         /* MK_NC_WARPS: stage i -> slot i % ring_slots */
  const void *kv_maps;        /* [L][2] CUtensorMap of the K and V pools (64-byte aligned) */
  int32_t xbuf_bytes;         /* shared scratch buffer */
  int32_t xn_bytes;           /* shared normed-input buffer (kept across a layer's tasks) */
  int32_t poison_layer, poison_delta; /* test hook: see mk_debug_poison_wait */
  int32_t fold;               /* 1: each gate/up share also computes its blocks' down partials */
  int32_t fold_rows;          /* rows of d per down box (the tensor maps' box height) */
  float *moe_part;            /* [2][Umax * F / 64][d] partial down vectors of the folded blocks
                               * (layer parity: a layer's writers never meet the previous
                               * layer's readers) */
  int32_t moe_part_stride;    /* floats per parity half of moe_part */
  /* Values that carry their own validity: 64-bit words {payload, step_tag}
   * written with one relaxed store and polled by their readers, so that no
   * counter round trip or release fence stands between writer and reader. */
  uint32_t step_tag;          /* this step's tag (never 0, never reused) */
  uint64_t *h_tag;            /* [L+1][MAXB][d/2]: {bf16 h[2i], bf16 h[2i+1]} */
  uint64_t *lg_tag;           /* [L][MAXB][E]: {fp32 router logit} */
  const void *wd_maps;        /* [L] CUtensorMap of each layer's down weights [E*d][F] */
  unsigned long long *trace;  /* NULL, or [n_cta][trace_cap][MK_TRACE_WORDS] task timestamps */
  int32_t trace_cap;
  unsigned long long *stage_trace; /* NULL, or one CTA's [MK_STAGE_TRACE_EVENTS][8] stage timestamps */
  int32_t stage_trace_cta;         /* the CTA that records them */
} mk_kparams;

/* Copies the first MK_PARAM_LAYERS layers' pointers into the parameter
 * space (host side, when the parameters are filled in). */
static inline void mk_param_layers(mk_kparams *p, const mk_layer_dev *ly, int n_layers) {
  for (int l = 0; l < n_layers && l < MK_PARAM_LAYERS; ++l) {
    p->l_norm[l] = ly[l].norm;
    p->l_bias[l] = ly[l].bias;
    p->l_kc[l] = ly[l].kc;
    p->l_vc[l] = ly[l].vc;
  }
}

/* One trace event (per executed task, written by consumer thread 0):
 * [0] op | layer << 8 | task << 20, [1] entry, [2] dependency satisfied,
 * [3] first stage of data available, [4] exit (globaltimer ns). */
#define MK_TRACE_WORDS 8
/* Stage events of CTA 0 (after the task events in the trace buffer), in SM
 * clock cycles: [0] stage | warp << 20 | op << 24, producer: [1] loop top,
 * [2] stage known, [3] slot free, [4] copies issued; owner warp: [5] starts
 * waiting, [6] data seen, [7] slot released.  The last event holds the
 * clock anchors (globaltimer, SM clock) at the kernel's start and end. */
#define MK_STAGE_TRACE_EVENTS 4096

#ifdef __CUDACC__
#define MK_HD __host__ __device__
#else
#define MK_HD
#endif

/* ---- ring stage geometry (the producer and the consumers must agree) -------
 * A stage of streamed rows holds whole rows of K bf16 (K a multiple of 64,
 * so a row is a multiple of 128 bytes): n plain rows as two runs, rows
 * [0, h) then [h, n) with h = (n + 1) / 2; gate/up pairs as the gate rows,
 * then the up rows.  Below batch MK_RUN_GAP_MIN_NB the runs are contiguous
 * as in memory (one bulk copy per stage, two for pairs).  From it on, the
 * second run starts 64 bytes past the end of the first (two copies) and the
 * token vectors of the activations sit K + 32 elements apart: the two rows
 * (one from each run) or two tokens that a quarter-warp reads in one 16-byte
 * operand load of the tensor-core GEMV then fall in opposite halves of the
 * 128-byte bank window, so no token has to be entered twice (see mma_rows).
 * The gap costs a copy that does not start on a 128-byte line, which only
 * pays where the activation loads dominate the stage's shared-memory reads
 * (eight tokens). */
#define MK_RUN_GAP_MIN_NB 8
static inline MK_HD int mk_run_gap(int nb) { return nb >= MK_RUN_GAP_MIN_NB ? 64 : 0; }
static inline MK_HD int mk_x_pitch(int K, int nb) { return nb >= MK_RUN_GAP_MIN_NB ? K + 32 : K; }

static inline MK_HD int mk_rows_per_stage(int K, int stage_bytes, int nb) {
  int r = (stage_bytes - mk_run_gap(nb)) / (2 * K);
  return r > MK_MAX_STAGE_ROWS ? MK_MAX_STAGE_ROWS : r;
}

/* Gate/up row pairs per stage: the n gate rows, then the n up rows. */
static inline MK_HD int mk_pairs_per_stage(int K, int stage_bytes, int nb) {
  return mk_rows_per_stage(K, stage_bytes, nb) / 2;
}

/* KV pages: one tensor-map box per page and pool covers min(D, 64) head dims
 * x D / min(D, 64) halves x P tokens; a page's K box, then its V box. */
static inline MK_HD int mk_box_inner(int D) { return D < 64 ? D : 64; }
static inline MK_HD int mk_page_stage_bytes(int P, int D) { return 2 * P * D * 2; }
static inline MK_HD int mk_pages_per_stage(int P, int D, int stage_bytes) {
  int r = stage_bytes / mk_page_stage_bytes(P, D);
  return r > MK_MAX_STAGE_PAGES ? MK_MAX_STAGE_PAGES : r;
}

#endif /* MK_INTERNAL_H */
