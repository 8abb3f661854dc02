/* mk_plan.h -- the host schedule builder's C++ interface (library-internal). */
#ifndef MK_PLAN_H
#define MK_PLAN_H

#include <stdint.h>

#include <vector>

#include "mk.h"

struct MkPlan {
  int n_cta = 0, tasks_per_cta = 0, n_layer_tasks_max = 0, batch = 0;
  int n_qkv = 0, n_router = 0, n_attn = 0, n_up = 0, n_out = 0, n_lm = 0, n_down = 0;
  int n_attn_slots = 0, n_attn_done = 0;
  int fold = 0; /* the down projection is folded into the gate/up shares (batch 1) */
  std::vector<int32_t> table;      /* [n_cta][tasks_per_cta][32] */
  std::vector<int32_t> built_lens; /* lengths the attention splits were cut for */
};

/* Dynamic shared memory of the nb-token kernel: ring_slots slots of stage_bytes,
 * the normed-input buffer, the scratch buffer, the control block (total),
 * plus MK_SMEM_STATIC bytes of slack to align the ring to 1024 bytes (dyn,
 * the launch size). */
struct MkSmem {
  int stage_bytes = 0;
  int ring_slots = 0; /* one per consumer warp */
  size_t xn = 0, xbuf = 0, misc = 0, total = 0, dyn = 0;
};
/* false if the model does not fit (a row, a row pair or a KV page larger
 * than one slot). */
bool mk_smem_plan(const mk_model_dims *d, int nb, MkSmem *out);
int mk_nb_for(int batch);

/* Encodes the 3-D TMA tensor maps of every layer's K and V pools into
 * host_out ([n_layers][2] maps of 128 bytes: K, V): dims {BI = min(head_dim,
 * 64), head_dim / BI, num_pages * n_kv_heads * page_size}, box {BI,
 * head_dim / BI, page_size} (one page of one kv head), 128-byte swizzle when
 * head_dim >= 64. */
mk_status mk_encode_kv_maps(const mk_model_dims *d, const void *const *k_pools,
                            const void *const *v_pools, void *host_out);

/* Encodes a 2-D TMA tensor map per layer over the down weights viewed as
 * [n_experts * d_model rows][d_ffn columns] into host_out ([n_layers] maps of
 * 128 bytes): box {MK_FOLD_COLS columns, box_rows rows}, 128-byte swizzle. */
mk_status mk_encode_wd_maps(const mk_model_dims *d, const void *const *w_down, int box_rows,
                            void *host_out);
/* Rows of d per down box for the batch-1 ring stages (a multiple of 8, at
 * most 256). */
int mk_fold_rows(const mk_model_dims *d);

mk_status mk_validate_dims(const mk_model_dims *d);
/* u_seen > 0: the distinct experts per layer observed at this batch size,
 * used in place of the uniform-routing expectation for the role split. */
mk_status mk_build_plan(const mk_model_dims *d, int n_cta, int batch, const int32_t *seq_lens,
                        MkPlan *out, double u_seen = 0.0);

#endif
