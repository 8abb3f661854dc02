/* mk_plan.h -- the host schedule builder's C++ interface (library-internal). */
#ifndef MK_PLAN_H
#define MK_PLAN_H

#include <stdint.h>

#include <vector>

#include "mk.h"

struct MkPlan {
  int n_cta = 0, tasks_per_cta = 0, n_layer_tasks_max = 0, batch = 0;
  int n_qkv = 0, n_router = 0, n_attn = 0, n_up = 0, n_out = 0, n_lm = 0;
  int n_attn_slots = 0, n_attn_done = 0;
  std::vector<int32_t> table;      /* [n_cta][tasks_per_cta][32] */
  std::vector<int32_t> built_lens; /* lengths the attention splits were cut for */
};

mk_status mk_validate_dims(const mk_model_dims *d);
mk_status mk_build_plan(const mk_model_dims *d, int n_cta, int batch, const int32_t *seq_lens,
                        MkPlan *out);

#endif
