/*
 * mk.h -- C ABI of the persistent MoE decode megakernel library (libmk).
 *
 * One call, mk_decode_step, runs the whole batch-1..8 BF16 decode step of a
 * mixture-of-experts transformer as ONE persistent kernel: RMSNorm, QKV
 * projection, RoPE + KV append, paged split-K attention, router top-k,
 * gathered expert SwiGLU, output projection, residual, final norm, LM head
 * and greedy argmax.  The method is the one described on three pages about a
 * decode megakernel for a 30B-total / 3.3B-active MoE model:
 *   - "Cohere speeds up North Mini Code with new megakernel"
 *     (latestnews.news), paragraphs 2-3: the whole forward pass in one
 *     persistent kernel, one threadblock per SM, a host-built static
 *     schedule, global-memory counters;
 *   - "Cohere Packs the Entire Decoding Step Into a Single CUDA Megakernel"
 *     (ainews.surl.tw), paragraph 2: the task table of GEMM tiles and
 *     attention splits, dataflow start on per-dependency counters, attention
 *     and MoE from the same normalized input; paragraph 4: BF16, batch 1-8;
 *   - "Cohere megakernel serves 30B MoE 1.58x faster than vLLM"
 *     (aiweekly.co), paragraphs 2-4: 32-int32 task descriptors, O(1)
 *     counter barriers, weight prefetch ahead of dependencies.
 *
 * Conventions
 *   - Every function returns mk_status (0 = MK_OK) unless stated; nothing
 *     throws across the ABI.
 *   - Pointers passed to mk_create are DEVICE pointers owned by the caller;
 *     they must stay valid until mk_destroy.  The library never frees them.
 *     Every weight / KV pointer must be 16-byte aligned.
 *   - The library owns only its workspace (activations, partials, counters,
 *     the device task table, device copies of page tables and lengths).
 *   - Work is enqueued on the stream given to mk_create; calls are
 *     asynchronous unless stated.
 *   - Layouts: bf16 matrices are row-major W[out][in] (the input dimension is
 *     contiguous); experts are stacked [E][F][d] (gate, up) and [E][d][F]
 *     (down); the K and V pools of a layer are [num_pages][n_kv_heads]
 *     [page_size][head_dim] and hold post-RoPE keys.
 *   - Errors: argument errors are returned synchronously.  Device errors
 *     (a counter wait that ran out of time, a corrupt task) are sticky and
 *     surface from the next call (mk_sync reports them at once); the context
 *     must then be destroyed.
 */
#ifndef MK_H
#define MK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mk_status;
enum {
  MK_OK = 0,
  MK_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad dimension */
  MK_ERR_BATCH = 2,         /* batch < 1 or > max_batch (at most 8) */
  MK_ERR_PAGE_OOB = 3,      /* a page id outside [0, num_pages), or no page for position L_b */
  MK_ERR_NO_SCHEDULE = 4,   /* mk_decode_step before mk_build_schedule */
  MK_ERR_CUDA = 5,          /* a CUDA runtime call failed */
  MK_ERR_DEVICE_TIMEOUT = 6,/* a device wait exceeded the wait limit (sticky) */
  MK_ERR_BAD_TASK = 7,      /* the kernel met an unknown task opcode (sticky) */
  MK_ERR_UNSUPPORTED = 8,   /* dims this build does not support (see mk_create) */
  MK_ERR_NO_DEVICE = 9,     /* no usable sm_103 device */
  MK_ERR_SCRATCH_LIMIT = 10,/* mk_decode_step_static: workspace larger than its static scratch */
  MK_ERR_BAD_TOKEN = 11     /* a token id outside [0, vocab) reached the kernel (sticky) */
};

/* Model dimensions.  page_size tokens per KV page; num_pages pages in each
 * layer's pool; max_pages_per_seq entries per page-table row. */
typedef struct {
  int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim;
  int32_t n_experts, top_k, d_ffn, vocab;
  int32_t page_size, max_batch, num_pages, max_pages_per_seq;
  float rope_base, rms_eps;
} mk_model_dims;

/* One layer's device pointers (all bf16 unless stated). */
typedef struct {
  const void *norm;                      /* [d] RMSNorm gain (one norm: parallel block) */
  const void *wq, *wk, *wv;              /* [Hq*D][d], [Hkv*D][d], [Hkv*D][d] */
  const void *wo;                        /* [d][Hq*D] */
  const void *w_router;                  /* [E][d] */
  const float *router_bias;              /* fp32 [E] added to the router logits, or NULL */
  const void *w_gate, *w_up;             /* [E][F][d] */
  const void *w_down;                    /* [E][d][F] */
  void *k_cache, *v_cache;               /* [num_pages][Hkv][P][D]; the step appends rows */
} mk_layer_ptrs;

typedef struct {
  const void *embed;                     /* [V][d] */
  const mk_layer_ptrs *layers;           /* HOST array [n_layers], copied by mk_create */
  const void *final_norm;                /* [d] */
  const void *lm_head;                   /* [V][d]; may equal embed (tied) */
} mk_weights;

typedef struct mk_ctx mk_ctx;

/* The model and its paged KV cache ("Cohere speeds up North Mini Code with
 * new megakernel", paragraphs 1 and 3: a BF16 MoE model, paged attention,
 * ragged sequence lengths).
 * Validates dims and pointers, queries the device, allocates the workspace.
 * stream: a cudaStream_t (NULL = legacy default stream).  Supported: head_dim
 * in {32, 64, 128}; n_q_heads / n_kv_heads <= 8; top_k <= 16; n_experts <=
 * 128; d_model, d_ffn and n_q_heads*head_dim multiples of 64; max_batch <= 8.
 * Returns MK_ERR_INVALID_ARG / MK_ERR_UNSUPPORTED / MK_ERR_NO_DEVICE /
 * MK_ERR_CUDA; *out is set only on MK_OK. */
mk_status mk_create(const mk_model_dims *dims, const mk_weights *w, void *stream, mk_ctx **out);

/* The host-built task table ("Cohere Packs the Entire Decoding Step Into a
 * Single CUDA Megakernel", paragraph 2: GEMM tiles and attention splits
 * assigned to the SMs in advance; continuous batching: "Cohere speeds up
 * North Mini Code with new megakernel", paragraph 3).
 * Builds the task table for `batch` sequences: seq_lens (HOST [batch]) =
 * cached tokens L_b before the next step; page_tables (HOST
 * [batch][max_pages_per_seq]) = physical page ids, -1 where unallocated.
 * Copies both to the device, resets the counters, uploads the table.
 * Call again whenever batch membership changes (continuous batching). */
mk_status mk_build_schedule(mk_ctx *ctx, int32_t batch, const int32_t *seq_lens,
                            const int32_t *page_tables);

/* The decode step as one persistent kernel ("Cohere speeds up North Mini
 * Code with new megakernel", paragraph 2; "Cohere megakernel serves 30B MoE
 * 1.58x faster than vLLM", paragraphs 2-3: every operation of the step in
 * one kernel, dependencies through counters in global memory).
 * One decode step for the scheduled batch.  token_ids: DEVICE int32 [batch];
 * out_logits: DEVICE fp32 [batch][vocab] or NULL; out_next_tokens: DEVICE
 * int32 [batch] (greedy argmax, ties -> lowest id).  A token id outside
 * [0, vocab) fails the step with MK_ERR_BAD_TOKEN (sticky; the kernel reads
 * embedding row 0 in its place, never outside the table).  Token b is processed at
 * position L_b and its K/V row is written there; L_b then advances by one
 * (on the device and in the context).  The page covering L_b must be present
 * in the page table (MK_ERR_PAGE_OOB otherwise).  When a sequence has grown
 * far past the lengths the table was built for, the table is rebuilt first.
 * Asynchronous: returns after the launch. */
mk_status mk_decode_step(mk_ctx *ctx, const int32_t *token_ids, float *out_logits,
                         int32_t *out_next_tokens);

/* Library plumbing (no operation of the pages): waits for the stream and
 * returns the sticky device status. */
mk_status mk_sync(mk_ctx *ctx);

/* Library plumbing: releases what mk_create allocated (never the caller's
 * weights or KV pools). */
void mk_destroy(mk_ctx *ctx);

/* Library plumbing: a static name for a status code ("unknown status" for
 * any other value). */
const char *mk_status_string(mk_status s);

/* One decode step that allocates no memory of its own: no cudaMalloc,
 * cudaFree, cudaHostAlloc or allocating library routine.  The three pages
 * have no counterpart of this call; it exists for callers that cannot
 * allocate device memory themselves -- for example code whose device memory
 * is entirely owned by an arena or caching allocator, or code running under a
 * memory budget that is already handed out -- and so cannot use mk_create.
 * It runs the same kernel as mk_decode_step, with all of that kernel's scratch
 * (activations, partial sums, counters, routing, task table, page tables, one
 * RoPE row per sequence) in one static device array of 16 MiB that every GPU
 * loading the library holds until the process exits.  Workloads whose scratch
 * does not fit (deep or wide models at batch 8, very long page tables) get
 * MK_ERR_SCRATCH_LIMIT before anything is launched.
 *   dims, w      as for mk_create (w->layers is a HOST array);
 *   batch, seq_lens, page_tables   as for mk_build_schedule (HOST arrays);
 *   token_ids, out_logits (may be NULL), out_next_tokens   DEVICE, as for
 *                mk_decode_step; the new K/V rows are written at L_b;
 *   stream       a cudaStream_t (NULL = legacy default stream).
 * Synchronous: it copies its host-side tables from pageable memory and reads
 * the kernel's status back before it returns, so it must not be called while
 * its stream is being captured.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current.
 * Calls share the array: the counters are cleared by each call, and calls
 * that overlap on the GPU race (serialise them).  Every device wait gives up
 * after a fixed 1 s (there is no context to set mk_set_wait_limit_ns on) and
 * the call returns MK_ERR_DEVICE_TIMEOUT.  There is no sticky state: every
 * call stands alone.  Given the same inputs and lengths it returns the same
 * bits as mk_decode_step after mk_build_schedule for those lengths. */
mk_status mk_decode_step_static(const mk_model_dims *dims, const mk_weights *w, int32_t batch,
                                const int32_t *seq_lens, const int32_t *page_tables,
                                const int32_t *token_ids, float *out_logits,
                                int32_t *out_next_tokens, void *stream);

/* ---- diagnostics (tests / benchmark) ------------------------------------- */

/* The bound on the counter barriers ("Cohere megakernel serves 30B MoE
 * 1.58x faster than vLLM", paragraph 3).
 * Device wait limit in nanoseconds (default 1e9).  Every counter / mbarrier
 * wait in the kernel gives up after this long and reports
 * MK_ERR_DEVICE_TIMEOUT instead of hanging. */
mk_status mk_set_wait_limit_ns(mk_ctx *ctx, uint64_t ns);

/* The router's top-k of the last step ("Cohere megakernel serves 30B MoE
 * 1.58x faster than vLLM", paragraph 2: MoE routing).  The oracle replays
 * this routing at near ties instead of the library accepting a forced one.
 * Routing of the last step (synchronises): ids / w HOST [n_layers][batch][top_k]
 * in descending-logit order; either may be NULL. */
mk_status mk_debug_routing(mk_ctx *ctx, int32_t *ids, float *w);

/* The intermediate values of the step's operations ("Cohere Packs the Entire
 * Decoding Step Into a Single CUDA Megakernel", paragraph 1: RMSNorm, QKV,
 * attention, MoE), for layer-by-layer comparison with the oracle.
 * Copies a workspace buffer of the last step to HOST memory (synchronises).
 * what: 0 = residual h [n_layers+1][batch][d] bf16 (h[0] is the embedding),
 *       1 = attention output o [n_layers][batch][Hq*D] bf16,
 *       2 = router logits [n_layers][batch][E] fp32,
 *       3 = q, k, v before RoPE [n_layers][batch][(Hq + 2 Hkv) D] bf16,
 *       4 = the attention term of the residual, attn = bf16(o Wo^T)
 *           [n_layers][batch][d] bf16,
 *       5 = the MoE term of the residual [n_layers][batch][d] bf16.
 * bytes must equal the buffer size. */
mk_status mk_debug_dump(mk_ctx *ctx, int32_t what, void *host_out, uint64_t bytes);

/* Running totals since mk_build_schedule (synchronises): the distinct
 * experts streamed, which fix the step's bytes ("Cohere megakernel serves
 * 30B MoE 1.58x faster than vLLM", paragraph 4: weights streamed per step). */
typedef struct {
  uint64_t steps;          /* decode steps launched */
  uint64_t sum_experts;    /* sum over steps and layers of distinct experts U */
  uint64_t rebuilds;       /* automatic table rebuilds */
} mk_stats;
mk_status mk_get_stats(mk_ctx *ctx, mk_stats *out);

/* Failure detection of the counter barriers ("Cohere megakernel serves 30B
 * MoE 1.58x faster than vLLM", paragraph 3).
 * Test only: adds `delta` to the target of layer `layer`'s attention-done
 * counter in the next launch, making that wait unsatisfiable so that the
 * bounded-wait path (MK_ERR_DEVICE_TIMEOUT) can be exercised without a hang. */
mk_status mk_debug_poison_wait(mk_ctx *ctx, int32_t layer, int32_t delta);

/* Where the SMs idle ("Cohere megakernel serves 30B MoE 1.58x faster than
 * vLLM", paragraph 4: idle SMs, dataflow start and weight prefetch).
 * Per-task timing trace of the following steps (diagnostic; each step
 * overwrites the previous one).  events_per_cta = 0 turns it off; otherwise
 * a buffer of n_sm * events_per_cta task events plus 4096 stage events is
 * allocated.  Consumer thread 0 of every CTA records, for each task it runs:
 * [0] op | layer << 8 | task << 20, [1] entry, [2] dependency satisfied,
 * [3] first data stage available (0 if none), [4] exit, [5] ns spent
 * waiting for later stages, [6] stages seen, [7] the task's mark (0 if
 * none) -- globaltimer nanoseconds, 8 words per event, unused events zero.
 * One CTA (mk_set_stage_trace_cta, default 0) also records its first 4095
 * ring stages in SM clock cycles: [0]
 * stage | warp << 20 | op << 24; the producer's [1] loop top, [2] stage
 * known, [3] slot free, [4] copies issued; the owning warp's [5] wait start,
 * [6] data seen, [7] slot released.  Stage event 4095 holds the clock
 * anchors: [0] globaltimer and [1] SM clock at the kernel's start, [2], [3]
 * the same at its end. */
mk_status mk_set_trace(mk_ctx *ctx, int32_t events_per_cta);
/* Which CTA records the stage events (default 0). */
mk_status mk_set_stage_trace_cta(mk_ctx *ctx, int32_t cta);
/* Copies the trace (synchronises).  host_out may be NULL to query the
 * geometry; otherwise it must hold (n_cta * events_per_cta + 4096) * 8
 * words: the task events [n_cta][events_per_cta][8], then the stage events
 * [4096][8] of the CTA chosen with mk_set_stage_trace_cta. */
mk_status mk_get_trace(mk_ctx *ctx, uint64_t *host_out, uint64_t n_words, int32_t *n_cta,
                       int32_t *events_per_cta);

/* The task table ("Cohere Packs the Entire Decoding Step Into a Single CUDA
 * Megakernel", paragraph 2; 32-int32 descriptors: "Cohere megakernel serves
 * 30B MoE 1.58x faster than vLLM", paragraph 2).
 * Host-only schedule planning (no GPU needed): the task table that
 * mk_build_schedule would upload for n_sm SMs.  Writes at most cap int32s of
 * [n_cta][tasks_per_cta][32] descriptors into table (may be NULL to query)
 * and the table geometry into info.  Returns MK_ERR_INVALID_ARG /
 * MK_ERR_BATCH / MK_ERR_UNSUPPORTED / MK_ERR_PAGE_OOB on bad input. */
typedef struct {
  int32_t n_cta, tasks_per_cta;       /* table is [n_cta][tasks_per_cta][32] */
  int32_t n_layer_tasks_max;          /* per-CTA tasks of one layer (template) */
  int32_t n_qkv, n_router, n_attn, n_up, n_out, n_lm; /* tasks per layer (lm: per step) */
  int32_t n_attn_slots;               /* attention partial slots per layer */
  int32_t n_down;                     /* expert down-row shares per layer (0: folded) */
} mk_plan_info;
mk_status mk_plan(const mk_model_dims *dims, int32_t n_sm, int32_t batch, const int32_t *seq_lens,
                  mk_plan_info *info, int32_t *table, int64_t cap);

#ifdef __cplusplus
}
#endif

#endif /* MK_H */
