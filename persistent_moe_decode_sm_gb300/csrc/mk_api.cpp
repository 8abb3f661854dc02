/*
 * mk_api.cpp -- the C ABI (include/mk.h): validation, workspace, schedule
 * upload, launch of the persistent decode kernel, sticky device errors.
 */
#include <cuda.h> /* tensor-map types; the encoder is reached through the runtime */
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "mk.h"
#include "mk_internal.h"
#include "mk_plan.h"

extern "C" size_t mk_misc_bytes(int nb);
extern "C" cudaError_t mk_kernel_prepare(int nb, size_t smem, int *blocks_per_sm);
extern "C" cudaError_t mk_launch(const mk_kparams *p, int nb, int grid, size_t smem,
                                 cudaStream_t stream);

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

/* A bump allocator over one device allocation. */
struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = align_up(off, 256);
    off = o + bytes;
    return o;
  }
};

}  // namespace

struct mk_ctx {
  mk_model_dims dims{};
  cudaStream_t stream = nullptr;
  int dev = 0, n_sm = 0;
  size_t smem_optin = 0;
  std::vector<mk_layer_dev> layers;
  mk_layer_dev *layers_dev = nullptr;
  const uint16_t *embed = nullptr, *final_norm = nullptr, *lm_head = nullptr;

  /* workspace */
  uint8_t *ws = nullptr;
  size_t ws_bytes = 0;
  uint16_t *h = nullptr, *qkv = nullptr, *o = nullptr, *act = nullptr, *am = nullptr;
  float *moe_part = nullptr;
  float *dpart = nullptr;
  int moe_part_stride = 0;
  uint64_t *h_tag = nullptr, *lg_tag = nullptr;
  void *wd_maps = nullptr;             /* device [n_layers] tensor maps of the down weights */
  int fold_rows = 0;
  float *attn_part = nullptr, *attn_part2 = nullptr, *router_logits = nullptr, *lm_part = nullptr,
        *rope = nullptr;
  mk_routing *routing = nullptr;
  int32_t *ctr = nullptr, *seq_lens_dev = nullptr, *page_table_dev = nullptr;
  mk_ctrl *ctrl = nullptr;
  int32_t *table_dev = nullptr;
  size_t table_cap = 0; /* int32s */
  int n_slots_max = 0, u_max = 0, rope_max_pos = 0, ctrs_per_layer = 0;
  size_t n_ctr = 0;

  /* host-mapped error mirror */
  int32_t *err_host = nullptr, *err_host_dev = nullptr;

  /* pinned staging for schedule uploads (two buffers, guarded by events) */
  int32_t *stage_host[2] = {nullptr, nullptr};
  size_t stage_cap[2] = {0, 0};
  cudaEvent_t stage_done[2] = {nullptr, nullptr};
  int stage_next = 0;

  /* schedule */
  bool scheduled = false;
  MkPlan plan;
  int batch = 0;
  std::vector<int32_t> lens;       /* live lengths L_b (host mirror) */
  std::vector<int32_t> page_table; /* [max_batch][max_pages] */
  uint64_t wait_limit_ns = 1000000000ULL;
  int poison_layer = -1, poison_delta = 0;
  uint64_t steps = 0, rebuilds = 0;
  /* the router's observed distinct experts per layer, for the role split */
  double u_seen = 0.0;
  int u_batch = 0;          /* batch size u_seen was observed at */
  uint64_t u_sum_base = 0;  /* the device's sum of U when the schedule was built */
  uint32_t tag_serial = 0; /* the last step tag used (never reset) */
  mk_status sticky = MK_OK;
  bool prepared[4] = {false, false, false, false}; /* kernel attributes set per batch bucket */
  unsigned long long *trace = nullptr; /* [n_sm][trace_cap][MK_TRACE_WORDS] */
  int stage_trace_cta = 0;
  void *kv_maps = nullptr;             /* device [n_layers][2] tensor maps (in ws) */
  int trace_cap = 0;
};

namespace {

mk_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MK_OK : MK_ERR_CUDA; }

mk_status check_sticky(mk_ctx *c) {
  if (c->sticky != MK_OK) return c->sticky;
  const int32_t code = *(volatile int32_t *)c->err_host;
  if (code != 0) c->sticky = code;
  return c->sticky;
}

mk_status upload_plan(mk_ctx *c, const MkPlan &p) {
  const size_t n = p.table.size();
  if (n > c->table_cap) {
    if (c->table_dev) cudaFree(c->table_dev);
    c->table_dev = nullptr;
    c->table_cap = 0;
    if (cudaMalloc(&c->table_dev, n * sizeof(int32_t)) != cudaSuccess) return MK_ERR_CUDA;
    c->table_cap = n;
  }
  const int k = c->stage_next;
  c->stage_next ^= 1;
  if (cudaEventSynchronize(c->stage_done[k]) != cudaSuccess) return MK_ERR_CUDA;
  if (n > c->stage_cap[k]) {
    if (c->stage_host[k]) cudaFreeHost(c->stage_host[k]);
    c->stage_host[k] = nullptr;
    c->stage_cap[k] = 0;
    if (cudaHostAlloc(&c->stage_host[k], n * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess)
      return MK_ERR_CUDA;
    c->stage_cap[k] = n;
  }
  std::memcpy(c->stage_host[k], p.table.data(), n * sizeof(int32_t));
  cudaError_t e = cudaMemcpyAsync(c->table_dev, c->stage_host[k], n * sizeof(int32_t),
                                  cudaMemcpyHostToDevice, c->stream);
  if (e == cudaSuccess) e = cudaEventRecord(c->stage_done[k], c->stream);
  /* new table: counters restart from zero, epoch 0 */
  if (e == cudaSuccess) e = cudaMemsetAsync(c->ctr, 0, c->n_ctr * sizeof(int32_t), c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(&c->ctrl->epoch, 0, sizeof(uint32_t), c->stream);
  return cuda_status(e);
}

mk_status rebuild(mk_ctx *c) {
  MkPlan p;
  mk_status st = mk_build_plan(&c->dims, c->n_sm, c->batch, c->lens.data(), &p,
                               c->u_batch == c->batch ? c->u_seen : 0.0);
  if (st != MK_OK) return st;
  if (p.n_attn_slots > c->n_slots_max || p.n_lm > c->n_sm) return MK_ERR_INVALID_ARG;
  st = upload_plan(c, p);
  if (st != MK_OK) return st;
  c->plan = std::move(p);
  return MK_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)ptr;
  });
  return fn;
}

}  // namespace

mk_status mk_encode_kv_maps(const mk_model_dims *dm, const void *const *k_pools,
                            const void *const *v_pools, void *host_out) {
  static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
  const mk_model_dims &d = *dm;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return MK_ERR_CUDA;
  /* 3-D view of a pool: {BI head dims, D / BI halves, token rows}; one box
   * is a whole page of one kv head */
  const int D = d.head_dim, bi = mk_box_inner(D), nbox = D / bi;
  const cuuint64_t dims[3] = {(cuuint64_t)bi, (cuuint64_t)nbox,
                              (cuuint64_t)d.num_pages * d.n_kv_heads * d.page_size};
  if (dims[2] > 0xFFFFFFFFull) return MK_ERR_UNSUPPORTED;
  const cuuint64_t strides[2] = {(cuuint64_t)bi * 2, (cuuint64_t)D * 2};
  const cuuint32_t box[3] = {(cuuint32_t)bi, (cuuint32_t)nbox, (cuuint32_t)d.page_size};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = D >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUtensorMap *out = (CUtensorMap *)host_out;
  for (int l = 0; l < d.n_layers; ++l)
    for (int kv = 0; kv < 2; ++kv) {
      void *base = const_cast<void *>(kv == 0 ? k_pools[l] : v_pools[l]);
      if (enc(&out[2 * l + kv], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MK_ERR_INVALID_ARG;
    }
  return MK_OK;
}

mk_status mk_encode_wd_maps(const mk_model_dims *dm, const void *const *w_down, int box_rows,
                            void *host_out) {
  const mk_model_dims &d = *dm;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return MK_ERR_CUDA;
  /* [E * d rows][F columns], row-major; one box = MK_FOLD_COLS columns (128
   * bytes, swizzled) of box_rows consecutive rows */
  const cuuint64_t dims[2] = {(cuuint64_t)d.d_ffn, (cuuint64_t)d.n_experts * d.d_model};
  const cuuint64_t strides[1] = {(cuuint64_t)d.d_ffn * 2};
  const cuuint32_t box[2] = {(cuuint32_t)MK_FOLD_COLS, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap *out = (CUtensorMap *)host_out;
  for (int l = 0; l < d.n_layers; ++l)
    if (enc(&out[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w_down[l]), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MK_ERR_INVALID_ARG;
  return MK_OK;
}

extern "C" {

const char *mk_status_string(mk_status s) {
  switch (s) {
    case MK_OK: return "ok";
    case MK_ERR_INVALID_ARG: return "invalid argument";
    case MK_ERR_BATCH: return "batch size out of range";
    case MK_ERR_PAGE_OOB: return "page id out of range or position without a page";
    case MK_ERR_NO_SCHEDULE: return "no schedule built";
    case MK_ERR_CUDA: return "CUDA runtime error";
    case MK_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MK_ERR_BAD_TASK: return "corrupt task descriptor";
    case MK_ERR_UNSUPPORTED: return "unsupported dimensions";
    case MK_ERR_NO_DEVICE: return "no usable sm_103 device";
    case MK_ERR_SCRATCH_LIMIT: return "workspace larger than the static scratch of mk_decode_step_static";
    case MK_ERR_BAD_TOKEN: return "token id outside the vocabulary";
    default: return "unknown status";
  }
}

mk_status mk_create(const mk_model_dims *dims, const mk_weights *w, void *stream, mk_ctx **out) {
  if (!out) return MK_ERR_INVALID_ARG;
  mk_status st = mk_validate_dims(dims);
  if (st != MK_OK) return st;
  if (!w || !w->layers || !w->embed || !w->final_norm || !w->lm_head) return MK_ERR_INVALID_ARG;
  if (!aligned16(w->embed) || !aligned16(w->final_norm) || !aligned16(w->lm_head))
    return MK_ERR_INVALID_ARG;
  const mk_model_dims &d = *dims;
  for (int l = 0; l < d.n_layers; ++l) {
    const mk_layer_ptrs &L = w->layers[l];
    const void *ps[] = {L.norm, L.wq, L.wk, L.wv, L.wo, L.w_router, L.w_gate, L.w_up, L.w_down,
                        L.k_cache, L.v_cache};
    for (const void *q : ps)
      if (!q || !aligned16(q)) return MK_ERR_INVALID_ARG;
    if (L.router_bias && ((uintptr_t)L.router_bias & 3u)) return MK_ERR_INVALID_ARG;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MK_ERR_NO_DEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MK_ERR_NO_DEVICE;
  if (prop.major != 10 || prop.minor != 3 || !prop.cooperativeLaunch) return MK_ERR_NO_DEVICE;

  mk_ctx *c = new mk_ctx();
  c->dims = d;
  c->stream = (cudaStream_t)stream;
  c->dev = dev;
  c->n_sm = prop.multiProcessorCount;
  c->smem_optin = prop.sharedMemPerBlockOptin;
  c->embed = (const uint16_t *)w->embed;
  c->final_norm = (const uint16_t *)w->final_norm;
  c->lm_head = (const uint16_t *)w->lm_head;
  c->layers.resize(d.n_layers);
  for (int l = 0; l < d.n_layers; ++l) {
    const mk_layer_ptrs &L = w->layers[l];
    mk_layer_dev &D = c->layers[l];
    D.norm = (const uint16_t *)L.norm;
    D.wq = (const uint16_t *)L.wq;
    D.wk = (const uint16_t *)L.wk;
    D.wv = (const uint16_t *)L.wv;
    D.wo = (const uint16_t *)L.wo;
    D.wr = (const uint16_t *)L.w_router;
    D.bias = L.router_bias;
    D.wg = (const uint16_t *)L.w_gate;
    D.wu = (const uint16_t *)L.w_up;
    D.wd = (const uint16_t *)L.w_down;
    D.kc = (uint16_t *)L.k_cache;
    D.vc = (uint16_t *)L.v_cache;
  }
  if (c->smem_optin < MK_SMEM_OPTIN) {
    delete c;
    return MK_ERR_NO_DEVICE;
  }

  /* workspace sizes */
  const int L = d.n_layers, MB = MK_MAX_BATCH, G = d.n_q_heads / d.n_kv_heads;
  const size_t QKVD = (size_t)(d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
  const size_t HqD = (size_t)d.n_q_heads * d.head_dim;
  c->n_slots_max = 256 + d.max_batch * d.n_kv_heads; /* splits: at most 256, one per pair */
  c->u_max = std::min(d.n_experts, d.max_batch * d.top_k);
  c->rope_max_pos = d.max_pages_per_seq * d.page_size;
  c->ctrs_per_layer = mk_ctrs_per_layer(MB, d.n_kv_heads);
  c->n_ctr = ((size_t)L * c->ctrs_per_layer + GCTR_COUNT) * MK_CTR_STRIDE;
  Carve cv;
  const size_t o_h = cv.take((size_t)(L + 1) * MB * d.d_model * 2);
  const size_t o_qkv = cv.take((size_t)L * MB * QKVD * 2);
  const size_t o_o = cv.take((size_t)L * MB * HqD * 2);
  const size_t o_am = cv.take((size_t)L * 2 * MB * d.d_model * 2);
  const size_t o_part = cv.take((size_t)2 * c->n_slots_max * G * (d.head_dim + 4) * 4);
  const size_t o_part2 = cv.take((size_t)2 * c->n_slots_max * G * (d.head_dim + 4) * 4);
  const size_t o_rl = cv.take((size_t)L * MB * d.n_experts * 4);
  const size_t o_rt = cv.take((size_t)L * sizeof(mk_routing));
  const size_t o_act = cv.take((size_t)L * c->u_max * MB * d.d_ffn * 2);
  const size_t o_dp = cv.take((size_t)2 * c->u_max * MB * d.d_model * 4);
  const size_t o_lm = cv.take((size_t)c->n_sm * MB * 2 * 4);
  const size_t o_rope = cv.take((size_t)c->rope_max_pos * (d.head_dim / 2) * 2 * 4);
  const size_t o_ctr = cv.take(c->n_ctr * 4);
  const size_t o_ctrl = cv.take(sizeof(mk_ctrl));
  const size_t o_len = cv.take((size_t)MB * 4);
  const size_t o_pt = cv.take((size_t)MB * d.max_pages_per_seq * 4);
  const size_t o_ly = cv.take((size_t)L * sizeof(mk_layer_dev));
  const size_t o_maps = cv.take((size_t)L * 2 * 128);
  const size_t o_wdm = cv.take((size_t)L * 128);
  c->moe_part_stride = std::min(d.n_experts, d.top_k) * (d.d_ffn / MK_FOLD_COLS) * d.d_model;
  const size_t o_mp = cv.take((size_t)2 * c->moe_part_stride * 4);
  const size_t o_htag = cv.take((size_t)(L + 1) * MB * (d.d_model / 2) * 8);
  const size_t o_lgtag = cv.take((size_t)L * MB * d.n_experts * 8);
  c->ws_bytes = cv.off;

  cudaError_t e = cudaMalloc(&c->ws, c->ws_bytes);
  if (e != cudaSuccess) {
    delete c;
    return MK_ERR_CUDA;
  }
  c->h = (uint16_t *)(c->ws + o_h);
  c->qkv = (uint16_t *)(c->ws + o_qkv);
  c->o = (uint16_t *)(c->ws + o_o);
  c->am = (uint16_t *)(c->ws + o_am);
  c->attn_part = (float *)(c->ws + o_part);
  c->attn_part2 = (float *)(c->ws + o_part2);
  c->router_logits = (float *)(c->ws + o_rl);
  c->routing = (mk_routing *)(c->ws + o_rt);
  c->act = (uint16_t *)(c->ws + o_act);
  c->dpart = (float *)(c->ws + o_dp);
  c->lm_part = (float *)(c->ws + o_lm);
  c->rope = (float *)(c->ws + o_rope);
  c->ctr = (int32_t *)(c->ws + o_ctr);
  c->ctrl = (mk_ctrl *)(c->ws + o_ctrl);
  c->seq_lens_dev = (int32_t *)(c->ws + o_len);
  c->page_table_dev = (int32_t *)(c->ws + o_pt);
  c->layers_dev = (mk_layer_dev *)(c->ws + o_ly);
  c->kv_maps = c->ws + o_maps;
  c->wd_maps = c->ws + o_wdm;
  c->moe_part = (float *)(c->ws + o_mp);
  c->h_tag = (uint64_t *)(c->ws + o_htag);
  c->lg_tag = (uint64_t *)(c->ws + o_lgtag);
  c->fold_rows = mk_fold_rows(&d);
  std::vector<uint8_t> maps((size_t)L * 2 * 128), wdmaps;
  {
    std::vector<const void *> kp(L), vp(L);
    for (int l = 0; l < L; ++l) {
      kp[l] = w->layers[l].k_cache;
      vp[l] = w->layers[l].v_cache;
    }
    mk_status ms = mk_encode_kv_maps(&d, kp.data(), vp.data(), maps.data());
    if (ms == MK_OK) {
      std::vector<const void *> wd(L);
      for (int l = 0; l < L; ++l) wd[l] = w->layers[l].w_down;
      wdmaps.resize((size_t)L * 128);
      ms = mk_encode_wd_maps(&d, wd.data(), c->fold_rows, wdmaps.data());
    }
    if (ms != MK_OK) {
      cudaFree(c->ws);
      delete c;
      return ms;
    }
  }

  /* RoPE table: cos / sin of pos * base^(-2i/D) in double, stored as fp32 */
  std::vector<float> rope((size_t)c->rope_max_pos * (d.head_dim / 2) * 2);
  {
    const int half = d.head_dim / 2;
    std::vector<double> inv(half);
    for (int i = 0; i < half; ++i)
      inv[i] = std::pow((double)d.rope_base, -2.0 * (double)i / (double)d.head_dim);
    for (int pos = 0; pos < c->rope_max_pos; ++pos)
      for (int i = 0; i < half; ++i) {
        const double a = (double)pos * inv[i];
        rope[((size_t)pos * half + i) * 2] = (float)std::cos(a);
        rope[((size_t)pos * half + i) * 2 + 1] = (float)std::sin(a);
      }
  }
  e = cudaMemsetAsync(c->ws, 0, c->ws_bytes, c->stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->rope, rope.data(), rope.size() * 4, cudaMemcpyHostToDevice, c->stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->layers_dev, c->layers.data(), L * sizeof(mk_layer_dev),
                        cudaMemcpyHostToDevice, c->stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->kv_maps, maps.data(), maps.size(), cudaMemcpyHostToDevice, c->stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->wd_maps, wdmaps.data(), wdmaps.size(), cudaMemcpyHostToDevice,
                        c->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
  if (e == cudaSuccess) e = cudaHostAlloc(&c->err_host, 16 * sizeof(int32_t), cudaHostAllocMapped);
  if (e == cudaSuccess) {
    std::memset(c->err_host, 0, 16 * sizeof(int32_t));
    e = cudaHostGetDevicePointer((void **)&c->err_host_dev, c->err_host, 0);
  }
  for (int k = 0; k < 2 && e == cudaSuccess; ++k)
    e = cudaEventCreateWithFlags(&c->stage_done[k], cudaEventDisableTiming);
  for (int k = 0; k < 2 && e == cudaSuccess; ++k) e = cudaEventRecord(c->stage_done[k], c->stream);
  if (e != cudaSuccess) {
    mk_destroy(c);
    return MK_ERR_CUDA;
  }
  c->page_table.assign((size_t)MB * d.max_pages_per_seq, -1);
  *out = c;
  return MK_OK;
}

mk_status mk_build_schedule(mk_ctx *c, int32_t batch, const int32_t *seq_lens,
                            const int32_t *page_tables) {
  if (!c || !seq_lens || !page_tables) return MK_ERR_INVALID_ARG;
  mk_status st = check_sticky(c);
  if (st != MK_OK) return st;
  const mk_model_dims &d = c->dims;
  if (batch < 1 || batch > d.max_batch) return MK_ERR_BATCH;
  const int mp = d.max_pages_per_seq, P = d.page_size;
  for (int b = 0; b < batch; ++b) {
    const int L = seq_lens[b];
    if (L < 0 || (int64_t)L + 1 > (int64_t)mp * P) return MK_ERR_PAGE_OOB;
    /* every page holding a cached token or the next position must exist */
    for (int j = 0; j <= L / P; ++j) {
      const int pg = page_tables[(size_t)b * mp + j];
      if (pg < 0 || pg >= d.num_pages) return MK_ERR_PAGE_OOB;
    }
    for (int j = L / P + 1; j < mp; ++j) {
      const int pg = page_tables[(size_t)b * mp + j];
      if (pg >= d.num_pages || pg < -1) return MK_ERR_PAGE_OOB;
    }
  }
  const int prev_batch = c->scheduled ? c->batch : 0;
  c->batch = batch;
  c->lens.assign(seq_lens, seq_lens + batch);
  std::fill(c->page_table.begin(), c->page_table.end(), -1);
  std::memcpy(c->page_table.data(), page_tables, (size_t)batch * mp * sizeof(int32_t));
  std::vector<int32_t> lens_dev(MK_MAX_BATCH, 0);
  std::copy(c->lens.begin(), c->lens.end(), lens_dev.begin());
  /* the host vectors are temporaries: copy and wait */
  cudaError_t e = cudaMemcpyAsync(c->seq_lens_dev, lens_dev.data(), MK_MAX_BATCH * 4,
                                  cudaMemcpyHostToDevice, c->stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->page_table_dev, c->page_table.data(), c->page_table.size() * 4,
                        cudaMemcpyHostToDevice, c->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
  /* the distinct experts per layer that the previous schedule's steps saw
   * (the stream is idle now), kept for schedules of the same batch size */
  unsigned long long sum = 0;
  if (e == cudaSuccess)
    e = cudaMemcpy(&sum, &c->ctrl->sum_experts, sizeof(sum), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return MK_ERR_CUDA;
  if (prev_batch > 0 && c->steps > 0 && sum > c->u_sum_base) {
    c->u_seen = (double)(sum - c->u_sum_base) / ((double)c->steps * d.n_layers);
    c->u_batch = prev_batch;
  }
  c->u_sum_base = sum;
  st = rebuild(c); /* uses u_seen when it was observed at this batch size */
  if (st != MK_OK) return st;
  c->scheduled = true;
  c->steps = 0;
  c->rebuilds = 0;
  return MK_OK;
}

mk_status mk_decode_step(mk_ctx *c, const int32_t *token_ids, float *out_logits,
                         int32_t *out_next_tokens) {
  if (!c || !token_ids || !out_next_tokens) return MK_ERR_INVALID_ARG;
  mk_status st = check_sticky(c);
  if (st != MK_OK) return st;
  if (!c->scheduled) return MK_ERR_NO_SCHEDULE;
  const mk_model_dims &d = c->dims;
  const int mp = d.max_pages_per_seq, P = d.page_size;
  for (int b = 0; b < c->batch; ++b) {
    const int L = c->lens[b];
    if ((int64_t)L + 1 > (int64_t)mp * P) return MK_ERR_PAGE_OOB;
    const int pg = c->page_table[(size_t)b * mp + L / P];
    if (pg < 0 || pg >= d.num_pages) return MK_ERR_PAGE_OOB;
  }
  /* Re-cut the attention splits once a sequence has outgrown them: the last
   * split of each (sequence, kv head) absorbs the new tokens meanwhile. */
  {
    bool stale = false;
    for (int b = 0; b < c->batch; ++b)
      if (c->lens[b] - c->plan.built_lens[b] >= std::max(64, 4 * P)) stale = true;
    if (stale) {
      st = rebuild(c);
      if (st != MK_OK) return st;
      ++c->rebuilds;
    }
  }
  const int nb = mk_nb_for(c->batch);
  MkSmem sm;
  if (!mk_smem_plan(&d, nb, &sm)) return MK_ERR_UNSUPPORTED;
  cudaError_t e;
  const int ki = nb == 1 ? 0 : nb == 2 ? 1 : nb == 4 ? 2 : 3;
  if (!c->prepared[ki]) {
    int blocks = 0;
    e = mk_kernel_prepare(nb, sm.dyn, &blocks);
    if (e != cudaSuccess) return MK_ERR_CUDA;
    if (blocks < 1) return MK_ERR_UNSUPPORTED;
    c->prepared[ki] = true;
  }

  mk_kparams p;
  std::memset(&p, 0, sizeof(p));
  p.L = d.n_layers;
  p.d = d.d_model;
  p.Hq = d.n_q_heads;
  p.Hkv = d.n_kv_heads;
  p.D = d.head_dim;
  p.E = d.n_experts;
  p.K = d.top_k;
  p.F = d.d_ffn;
  p.V = d.vocab;
  p.P = d.page_size;
  p.max_pages = mp;
  p.B = c->batch;
  p.eps = d.rms_eps;
  p.attn_scale = (float)(1.0 / std::sqrt((double)d.head_dim));
  p.layers = c->layers_dev;
  mk_param_layers(&p, c->layers.data(), d.n_layers);
  p.embed = c->embed;
  p.final_norm = c->final_norm;
  p.lm_head = c->lm_head;
  p.tokens = token_ids;
  p.out_logits = out_logits;
  p.out_next = out_next_tokens;
  p.h = c->h;
  p.qkv = c->qkv;
  p.o = c->o;
  p.am = c->am;
  p.attn_part = c->attn_part;
  p.attn_part2 = c->attn_part2;
  p.router_logits = c->router_logits;
  p.routing = c->routing;
  p.act = c->act;
  p.lm_part = c->lm_part;
  p.ctr = c->ctr;
  p.ctrl = c->ctrl;
  p.seq_lens = c->seq_lens_dev;
  p.page_table = c->page_table_dev;
  p.rope = c->rope;
  p.rope_max_pos = c->rope_max_pos;
  p.table = c->table_dev;
  p.tasks_per_cta = c->plan.tasks_per_cta;
  p.n_slots = c->n_slots_max;
  p.u_max = c->u_max;
  p.n_down = c->plan.n_down;
  p.dpart = c->dpart;
  p.n_qkv = c->plan.n_qkv;
  p.n_router = c->plan.n_router;
  p.n_up = c->plan.n_up;
  p.n_out = c->plan.n_out;
  p.n_lm = c->plan.n_lm;
  p.n_attn_done = c->plan.n_attn_done;
  p.ctrs_per_layer = c->ctrs_per_layer;
  p.wait_limit_ns = c->wait_limit_ns;
  p.err_host = c->err_host_dev;
  p.stage_bytes = sm.stage_bytes;
  p.ring_slots = sm.ring_slots;
  p.kv_maps = c->kv_maps;
  p.xbuf_bytes = (int32_t)sm.xbuf;
  p.xn_bytes = (int32_t)sm.xn;
  p.fold = c->plan.fold;
  p.fold_rows = c->fold_rows;
  p.moe_part = c->moe_part;
  p.moe_part_stride = c->moe_part_stride;
  p.h_tag = c->h_tag;
  p.lg_tag = c->lg_tag;
  c->tag_serial = c->tag_serial == 0xFFFFFFFFu ? 1u : c->tag_serial + 1u;
  p.step_tag = c->tag_serial;
  p.wd_maps = c->wd_maps;
  p.poison_layer = c->poison_layer;
  p.poison_delta = c->poison_delta;
  p.trace = c->trace;
  p.trace_cap = c->trace_cap;
  p.stage_trace = c->trace ? c->trace + (size_t)c->n_sm * c->trace_cap * MK_TRACE_WORDS : nullptr;
  p.stage_trace_cta = c->stage_trace_cta;
  c->poison_layer = -1;
  c->poison_delta = 0;

  e = mk_launch(&p, nb, c->n_sm, sm.dyn, c->stream);
  if (e != cudaSuccess) return MK_ERR_CUDA;
  for (int b = 0; b < c->batch; ++b) c->lens[b] += 1;
  ++c->steps;
  return MK_OK;
}

mk_status mk_sync(mk_ctx *c) {
  if (!c) return MK_ERR_INVALID_ARG;
  const cudaError_t e = cudaStreamSynchronize(c->stream);
  const mk_status st = check_sticky(c);
  if (st != MK_OK) return st;
  if (e != cudaSuccess) {
    c->sticky = MK_ERR_CUDA;
    return MK_ERR_CUDA;
  }
  return MK_OK;
}

void mk_destroy(mk_ctx *c) {
  if (!c) return;
  cudaStreamSynchronize(c->stream);
  if (c->ws) cudaFree(c->ws);
  if (c->table_dev) cudaFree(c->table_dev);
  for (int k = 0; k < 2; ++k) {
    if (c->stage_host[k]) cudaFreeHost(c->stage_host[k]);
    if (c->stage_done[k]) cudaEventDestroy(c->stage_done[k]);
  }
  if (c->err_host) cudaFreeHost(c->err_host);
  if (c->trace) cudaFree(c->trace);
  delete c;
}

mk_status mk_set_trace(mk_ctx *c, int32_t events_per_cta) {
  if (!c || events_per_cta < 0) return MK_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return MK_ERR_CUDA;
  if (c->trace) cudaFree(c->trace);
  c->trace = nullptr;
  c->trace_cap = 0;
  if (events_per_cta == 0) return MK_OK;
  const size_t bytes =
      ((size_t)c->n_sm * events_per_cta + MK_STAGE_TRACE_EVENTS) * MK_TRACE_WORDS * 8;
  if (cudaMalloc(&c->trace, bytes) != cudaSuccess) return MK_ERR_CUDA;
  if (cudaMemset(c->trace, 0, bytes) != cudaSuccess) return MK_ERR_CUDA;
  c->trace_cap = events_per_cta;
  return MK_OK;
}

mk_status mk_set_stage_trace_cta(mk_ctx *c, int32_t cta) {
  if (!c || cta < 0 || cta >= c->n_sm) return MK_ERR_INVALID_ARG;
  c->stage_trace_cta = cta;
  return MK_OK;
}

mk_status mk_get_trace(mk_ctx *c, uint64_t *host_out, uint64_t n_words, int32_t *n_cta,
                       int32_t *events_per_cta) {
  if (!c) return MK_ERR_INVALID_ARG;
  if (n_cta) *n_cta = c->n_sm;
  if (events_per_cta) *events_per_cta = c->trace_cap;
  if (!host_out) return MK_OK;
  const uint64_t need =
      ((uint64_t)c->n_sm * c->trace_cap + MK_STAGE_TRACE_EVENTS) * MK_TRACE_WORDS;
  if (!c->trace || n_words < need) return MK_ERR_INVALID_ARG;
  mk_status st = mk_sync(c);
  if (st != MK_OK) return st;
  if (cudaMemcpy(host_out, c->trace, need * 8, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MK_ERR_CUDA;
  return MK_OK;
}

mk_status mk_set_wait_limit_ns(mk_ctx *c, uint64_t ns) {
  if (!c || ns == 0) return MK_ERR_INVALID_ARG;
  c->wait_limit_ns = ns;
  return MK_OK;
}

mk_status mk_debug_poison_wait(mk_ctx *c, int32_t layer, int32_t delta) {
  if (!c || layer < 0 || layer >= c->dims.n_layers) return MK_ERR_INVALID_ARG;
  c->poison_layer = layer;
  c->poison_delta = delta;
  return MK_OK;
}

mk_status mk_debug_routing(mk_ctx *c, int32_t *ids, float *w) {
  if (!c) return MK_ERR_INVALID_ARG;
  if (!c->scheduled) return MK_ERR_NO_SCHEDULE;
  mk_status st = mk_sync(c);
  if (st != MK_OK) return st;
  const int L = c->dims.n_layers, B = c->batch, K = c->dims.top_k;
  std::vector<mk_routing> rt(L);
  if (cudaMemcpy(rt.data(), c->routing, L * sizeof(mk_routing), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return MK_ERR_CUDA;
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < B; ++b)
      for (int k = 0; k < K; ++k) {
        if (ids) ids[((size_t)l * B + b) * K + k] = rt[l].ids[b][k];
        if (w) w[((size_t)l * B + b) * K + k] = rt[l].w[b][k];
      }
  return MK_OK;
}

mk_status mk_debug_dump(mk_ctx *c, int32_t what, void *host_out, uint64_t bytes) {
  if (!c || !host_out) return MK_ERR_INVALID_ARG;
  if (!c->scheduled) return MK_ERR_NO_SCHEDULE;
  mk_status st = mk_sync(c);
  if (st != MK_OK) return st;
  const mk_model_dims &d = c->dims;
  const int L = d.n_layers, B = c->batch;
  size_t row = 0, nl = 0, esz = 0;
  const uint8_t *src = nullptr;
  switch (what) {
    case 0: row = d.d_model; nl = L + 1; esz = 2; src = (const uint8_t *)c->h; break;
    case 1: row = (size_t)d.n_q_heads * d.head_dim; nl = L; esz = 2; src = (const uint8_t *)c->o; break;
    case 2: row = d.n_experts; nl = L; esz = 4; src = (const uint8_t *)c->router_logits; break;
    case 3:
      row = (size_t)(d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
      nl = L;
      esz = 2;
      src = (const uint8_t *)c->qkv;
      break;
    case 4: row = d.d_model; nl = L; esz = 2; src = (const uint8_t *)c->am; break;
    case 5:
      row = d.d_model;
      nl = L;
      esz = 2;
      src = (const uint8_t *)(c->am + (size_t)MK_MAX_BATCH * d.d_model);
      break;
    default: return MK_ERR_INVALID_ARG;
  }
  if (bytes != nl * B * row * esz) return MK_ERR_INVALID_ARG;
  /* per layer: [MAXB][row], or [2][MAXB][row] for the attn / moe terms */
  const size_t lstride = (what >= 4 ? 2 : 1) * (size_t)MK_MAX_BATCH * row * esz;
  for (size_t l = 0; l < nl; ++l)
    if (cudaMemcpy((uint8_t *)host_out + l * B * row * esz, src + l * lstride,
                   B * row * esz, cudaMemcpyDeviceToHost) != cudaSuccess)
      return MK_ERR_CUDA;
  return MK_OK;
}

mk_status mk_get_stats(mk_ctx *c, mk_stats *out) {
  if (!c || !out) return MK_ERR_INVALID_ARG;
  mk_status st = mk_sync(c);
  if (st != MK_OK) return st;
  mk_ctrl ctrl;
  if (cudaMemcpy(&ctrl, c->ctrl, sizeof(ctrl), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MK_ERR_CUDA;
  out->steps = c->steps;
  out->sum_experts = ctrl.sum_experts;
  out->rebuilds = c->rebuilds;
  return MK_OK;
}

}  // extern "C"
