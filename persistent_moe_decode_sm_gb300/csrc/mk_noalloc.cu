/*
 * mk_noalloc.cu -- one decode step that allocates no memory of its own.
 *
 * mk_create allocates a workspace with cudaMalloc and a mapped error word
 * with cudaHostAlloc.  Some callers cannot do that: code whose GPU memory is
 * entirely owned by an arena or caching allocator that must not see stray
 * driver allocations, code running where a cudaMalloc would synchronise the
 * device or fail (for example inside a memory budget that is already fully
 * handed out), or a host process that only borrows device pointers from a
 * framework.  mk_decode_step_static serves them: it runs the same persistent
 * decode kernel as mk_decode_step, with every scratch buffer (activations,
 * partial sums, counters, routing, the task table, page tables, one RoPE row
 * per sequence) carved out of one file-scope device array, mk_static_scratch,
 * of MK_STATIC_SCRATCH_BYTES.  Nothing here calls cudaMalloc, cudaFree,
 * cudaHostAlloc or an allocating library routine.  The task table itself is
 * built in ordinary host memory of the calling thread.
 *
 * The array lives on every GPU that loads the library until the process
 * exits.  Its device address is looked up once per device with
 * cudaGetSymbolAddress, by the first call made on that device (with that
 * device current).  Every call reuses the same array and it keeps the
 * previous call's contents; the counters and the control block are cleared
 * at the start of each call.  Two calls whose work overlaps on the GPU
 * (different streams, or different host threads) race on the array and give
 * wrong results: serialise them.  Each call is synchronous (it copies from
 * pageable host memory and reads the kernel's status back), so it must not
 * be called while its stream is being captured into a graph.  The kernel's
 * waits give up after a fixed 1 s (MK_STATIC_WAIT_LIMIT_NS) and the call
 * then returns MK_ERR_DEVICE_TIMEOUT.
 */
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "mk.h"
#include "mk_internal.h"
#include "mk_plan.h"

extern "C" cudaError_t mk_kernel_prepare(int nb, size_t smem, int *blocks_per_sm);
extern "C" cudaError_t mk_launch(const mk_kparams *p, int nb, int grid, size_t smem,
                                 cudaStream_t stream);

/* 16 MiB: enough for the tiny and mid models and for short contexts of models
 * of that size; the call rejects anything larger with MK_ERR_SCRATCH_LIMIT. */
#define MK_STATIC_SCRATCH_BYTES (16u << 20)
/* Every device wait of a static step gives up after this long. */
#define MK_STATIC_WAIT_LIMIT_NS 1000000000ULL

static __device__ __align__(256) unsigned char mk_static_scratch[MK_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
unsigned char *g_scratch[kMaxDevices];      /* device address of mk_static_scratch */
bool g_prepared[kMaxDevices][4];             /* kernel attribute set per batch bucket */

size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" mk_status mk_decode_step_static(const mk_model_dims *dims, const mk_weights *w,
                                           int32_t batch, const int32_t *seq_lens,
                                           const int32_t *page_tables, const int32_t *token_ids,
                                           float *out_logits, int32_t *out_next_tokens,
                                           void *stream_ptr) {
  /* ---- arguments (the same checks as mk_create / mk_build_schedule) ---- */
  mk_status st = mk_validate_dims(dims);
  if (st != MK_OK) return st;
  if (!w || !w->layers || !w->embed || !w->final_norm || !w->lm_head || !seq_lens ||
      !page_tables || !token_ids || !out_next_tokens)
    return MK_ERR_INVALID_ARG;
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
  if (batch < 1 || batch > d.max_batch) return MK_ERR_BATCH;
  const int mp = d.max_pages_per_seq, P = d.page_size, MB = MK_MAX_BATCH;
  for (int b = 0; b < batch; ++b) {
    const int Lb = seq_lens[b];
    if (Lb < 0 || (int64_t)Lb + 1 > (int64_t)mp * P) return MK_ERR_PAGE_OOB;
    for (int j = 0; j <= Lb / P; ++j) {
      const int pg = page_tables[(size_t)b * mp + j];
      if (pg < 0 || pg >= d.num_pages) return MK_ERR_PAGE_OOB;
    }
  }

  /* ---- device and one-time set-up ---- */
  int dev = 0, n_sm = 0, major = 0, minor = 0, coop = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MK_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return MK_ERR_NO_DEVICE;
  if (major != 10 || minor != 3 || !coop) return MK_ERR_NO_DEVICE;
  unsigned char *base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch[dev]) {
      void *ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, mk_static_scratch) != cudaSuccess || !ptr)
        return MK_ERR_CUDA;
      g_scratch[dev] = (unsigned char *)ptr;
    }
    base = g_scratch[dev];
  }
  cudaStream_t stream = (cudaStream_t)stream_ptr;

  /* ---- task table (host) ---- */
  MkPlan plan;
  st = mk_build_plan(dims, n_sm, batch, seq_lens, &plan);
  if (st != MK_OK) return st;

  /* ---- carve the scratch ---- */
  const int Lyr = d.n_layers, G = d.n_q_heads / d.n_kv_heads, half = d.head_dim / 2;
  const size_t QKVD = (size_t)(d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
  const size_t HqD = (size_t)d.n_q_heads * d.head_dim;
  const int u_max = std::min(d.n_experts, d.max_batch * d.top_k);
  const int n_slots = std::max(1, plan.n_attn_slots);
  const int ctrs_per_layer = mk_ctrs_per_layer(MB, d.n_kv_heads);
  const size_t n_ctr = ((size_t)Lyr * ctrs_per_layer + GCTR_COUNT) * MK_CTR_STRIDE;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = up(off, 256);
    off = o + bytes;
    return o;
  };
  const size_t o_h = take((size_t)(Lyr + 1) * MB * d.d_model * 2);
  const size_t o_qkv = take((size_t)Lyr * MB * QKVD * 2);
  const size_t o_o = take((size_t)Lyr * MB * HqD * 2);
  const size_t o_am = take((size_t)Lyr * 2 * MB * d.d_model * 2);
  const size_t o_part = take((size_t)2 * n_slots * G * (d.head_dim + 4) * 4);
  const size_t o_part2 = take((size_t)2 * n_slots * G * (d.head_dim + 4) * 4);
  const size_t o_rl = take((size_t)Lyr * MB * d.n_experts * 4);
  const size_t o_rt = take((size_t)Lyr * sizeof(mk_routing));
  const size_t o_act = take((size_t)Lyr * u_max * MB * d.d_ffn * 2);
  const size_t o_dp = take((size_t)2 * u_max * MB * d.d_model * 4);
  const size_t o_lm = take((size_t)plan.n_lm * MB * 2 * 4);
  const size_t o_rope = take((size_t)MB * half * 2 * 4); /* one row per sequence */
  const size_t o_ctr = take(n_ctr * 4);
  const size_t o_ctrl = take(sizeof(mk_ctrl));
  const size_t o_len = take((size_t)MB * 4);
  const size_t o_pt = take((size_t)MB * mp * 4);
  const size_t o_ly = take((size_t)Lyr * sizeof(mk_layer_dev));
  const size_t o_tab = take(plan.table.size() * sizeof(int32_t));
  const size_t o_maps = take((size_t)Lyr * 2 * 128);
  const size_t o_wdm = take((size_t)Lyr * 128);
  const int moe_stride = std::min(d.n_experts, d.top_k) * (d.d_ffn / MK_FOLD_COLS) * d.d_model;
  const size_t o_mp = take((size_t)2 * moe_stride * 4);
  const size_t o_htag = take((size_t)(Lyr + 1) * MB * (d.d_model / 2) * 8);
  const size_t o_lgtag = take((size_t)Lyr * MB * d.n_experts * 8);
  if (off > MK_STATIC_SCRATCH_BYTES) return MK_ERR_SCRATCH_LIMIT;

  /* ---- shared memory plan (as for mk_decode_step) ---- */
  const int nb = mk_nb_for(batch);
  MkSmem sm;
  if (optin < MK_SMEM_OPTIN || !mk_smem_plan(dims, nb, &sm)) return MK_ERR_UNSUPPORTED;
  const size_t smem = sm.dyn;
  {
    const int ki = nb == 1 ? 0 : nb == 2 ? 1 : nb == 4 ? 2 : 3;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_prepared[dev][ki]) {
      int blocks = 0;
      if (mk_kernel_prepare(nb, smem, &blocks) != cudaSuccess) return MK_ERR_CUDA;
      if (blocks < 1) return MK_ERR_UNSUPPORTED;
      g_prepared[dev][ki] = true;
    }
  }

  /* ---- host-side contents, copied into the scratch ---- */
  std::vector<mk_layer_dev> layers(Lyr);
  for (int l = 0; l < Lyr; ++l) {
    const mk_layer_ptrs &L = w->layers[l];
    mk_layer_dev &D = layers[l];
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
  std::vector<uint8_t> maps((size_t)Lyr * 2 * 128);
  {
    std::vector<const void *> kp(Lyr), vp(Lyr);
    for (int l = 0; l < Lyr; ++l) {
      kp[l] = w->layers[l].k_cache;
      vp[l] = w->layers[l].v_cache;
    }
    st = mk_encode_kv_maps(dims, kp.data(), vp.data(), maps.data());
    if (st != MK_OK) return st;
  }
  const int fold_rows = mk_fold_rows(dims);
  std::vector<uint8_t> wdmaps((size_t)Lyr * 128);
  {
    std::vector<const void *> wd(Lyr);
    for (int l = 0; l < Lyr; ++l) wd[l] = w->layers[l].w_down;
    st = mk_encode_wd_maps(dims, wd.data(), fold_rows, wdmaps.data());
    if (st != MK_OK) return st;
  }
  std::vector<int32_t> lens(MB, 0), pt((size_t)MB * mp, -1);
  std::copy(seq_lens, seq_lens + batch, lens.begin());
  std::memcpy(pt.data(), page_tables, (size_t)batch * mp * sizeof(int32_t));
  /* only the RoPE rows of this step's positions are read */
  std::vector<float> rope_rows((size_t)batch * half * 2);
  for (int b = 0; b < batch; ++b)
    for (int i = 0; i < half; ++i) {
      const double a = (double)seq_lens[b] *
                       std::pow((double)d.rope_base, -2.0 * (double)i / (double)d.head_dim);
      rope_rows[((size_t)b * half + i) * 2] = (float)std::cos(a);
      rope_rows[((size_t)b * half + i) * 2 + 1] = (float)std::sin(a);
    }

  /* pageable sources: each copy returns once the host data is consumed */
  cudaError_t e = cudaMemsetAsync(base + o_ctr, 0, n_ctr * 4, stream);
  /* the tagged words: another call may have left any bytes there */
  if (e == cudaSuccess) e = cudaMemsetAsync(base + o_htag, 0, o_lgtag - o_htag, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(base + o_lgtag, 0, (size_t)Lyr * MB * d.n_experts * 8, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(base + o_ctrl, 0, sizeof(mk_ctrl), stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + o_ly, layers.data(), Lyr * sizeof(mk_layer_dev),
                        cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + o_maps, maps.data(), maps.size(), cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + o_wdm, wdmaps.data(), wdmaps.size(), cudaMemcpyHostToDevice,
                        stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + o_len, lens.data(), MB * 4, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + o_pt, pt.data(), pt.size() * 4, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + o_tab, plan.table.data(), plan.table.size() * 4,
                        cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + o_rope, rope_rows.data(), rope_rows.size() * 4,
                        cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return MK_ERR_CUDA;

  mk_kparams p;
  std::memset(&p, 0, sizeof(p));
  p.L = Lyr;
  p.d = d.d_model;
  p.Hq = d.n_q_heads;
  p.Hkv = d.n_kv_heads;
  p.D = d.head_dim;
  p.E = d.n_experts;
  p.K = d.top_k;
  p.F = d.d_ffn;
  p.V = d.vocab;
  p.P = P;
  p.max_pages = mp;
  p.B = batch;
  p.eps = d.rms_eps;
  p.attn_scale = (float)(1.0 / std::sqrt((double)d.head_dim));
  p.layers = (const mk_layer_dev *)(base + o_ly);
  mk_param_layers(&p, layers.data(), Lyr);
  p.embed = (const uint16_t *)w->embed;
  p.final_norm = (const uint16_t *)w->final_norm;
  p.lm_head = (const uint16_t *)w->lm_head;
  p.tokens = token_ids;
  p.out_logits = out_logits;
  p.out_next = out_next_tokens;
  p.h = (uint16_t *)(base + o_h);
  p.qkv = (uint16_t *)(base + o_qkv);
  p.o = (uint16_t *)(base + o_o);
  p.am = (uint16_t *)(base + o_am);
  p.attn_part = (float *)(base + o_part);
  p.attn_part2 = (float *)(base + o_part2);
  p.router_logits = (float *)(base + o_rl);
  p.routing = (mk_routing *)(base + o_rt);
  p.act = (uint16_t *)(base + o_act);
  p.lm_part = (float *)(base + o_lm);
  p.ctr = (int32_t *)(base + o_ctr);
  p.ctrl = (mk_ctrl *)(base + o_ctrl);
  p.seq_lens = (int32_t *)(base + o_len);
  p.page_table = (const int32_t *)(base + o_pt);
  p.rope = (const float *)(base + o_rope);
  p.rope_max_pos = mp * P;
  p.rope_per_seq = 1;
  p.table = (const int32_t *)(base + o_tab);
  p.tasks_per_cta = plan.tasks_per_cta;
  p.n_slots = n_slots;
  p.u_max = u_max;
  p.n_down = plan.n_down;
  p.dpart = (float *)(base + o_dp);
  p.n_qkv = plan.n_qkv;
  p.n_router = plan.n_router;
  p.n_up = plan.n_up;
  p.n_out = plan.n_out;
  p.n_lm = plan.n_lm;
  p.n_attn_done = plan.n_attn_done;
  p.ctrs_per_layer = ctrs_per_layer;
  p.wait_limit_ns = MK_STATIC_WAIT_LIMIT_NS;
  p.err_host = nullptr;
  p.stage_bytes = sm.stage_bytes;
  p.ring_slots = sm.ring_slots;
  p.kv_maps = base + o_maps;
  p.xbuf_bytes = (int32_t)sm.xbuf;
  p.xn_bytes = (int32_t)sm.xn;
  p.fold = plan.fold;
  p.fold_rows = fold_rows;
  p.moe_part = (float *)(base + o_mp);
  p.moe_part_stride = moe_stride;
  p.h_tag = (uint64_t *)(base + o_htag);
  p.lg_tag = (uint64_t *)(base + o_lgtag);
  {
    /* a tag no earlier call used on this scratch (it starts zeroed) */
    static std::atomic<uint32_t> serial{0};
    uint32_t t = serial.fetch_add(1u) + 1u;
    if (t == 0u) t = serial.fetch_add(1u) + 1u;
    p.step_tag = t;
  }
  p.wd_maps = base + o_wdm;
  p.poison_layer = -1;
  p.poison_delta = 0;

  if (mk_launch(&p, nb, n_sm, smem, stream) != cudaSuccess) return MK_ERR_CUDA;
  /* synchronous: read the kernel's status word back */
  int32_t code = 0;
  e = cudaMemcpyAsync(&code, base + o_ctrl + offsetof(mk_ctrl, err_code), sizeof(int32_t),
                      cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return MK_ERR_CUDA;
  return code;
}
