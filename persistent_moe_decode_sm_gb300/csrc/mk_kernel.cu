/*
 * mk_kernel.cu -- the persistent decode megakernel for sm_103a.
 *
 * One CTA per SM, launched cooperatively so every CTA is resident.  Each
 * CTA walks its row of the host-built task table: the per-layer template
 * once per layer, then the LM-head tasks.  This is the method of the pages
 * ("Cohere speeds up North Mini Code with new megakernel", latestnews.news,
 * paragraphs 2-3; "Cohere Packs the Entire Decoding Step Into a Single CUDA
 * Megakernel", ainews.surl.tw, paragraph 2), redesigned for this chip:
 *
 *   warps 0..7  consumers: wait on the task's counter, compute from shared
 *               memory, write outputs, signal the downstream counter;
 *   warp  8     producer:  streams each task's immutable bytes (weights,
 *               cached K/V pages) into a ring of shared-memory stages with
 *               cp.async.bulk (TMA) completing on mbarriers.  It runs ahead
 *               of the consumers and does NOT wait for a task's data
 *               dependency before loading its weights -- the weight
 *               prefetch ahead of dependencies that the aiweekly.co page
 *               ranks third among the method's gains (paragraph 4).  Only
 *               the expert weights wait, for the routing that names them.
 *
 * Counters ("Cohere megakernel serves 30B MoE 1.58x faster than vLLM",
 * paragraph 3): a task waits for ONE counter to reach a count, and signals
 * by one release-add, so signalling and waiting are O(1) in fan-in and
 * fan-out.  Counters are epoch-based (never reset between steps).  Every
 * wait is bounded by the context's wait limit: on timeout the kernel records
 * the failing wait, raises a global abort flag that every CTA polls, drains
 * its in-flight copies and returns; the host reports MK_ERR_DEVICE_TIMEOUT.
 *
 * Arithmetic follows the method's definition: bf16 weights and activations,
 * fp32 accumulation, bf16 rounding of q/k/v, RoPE outputs, attention output,
 * attention and MoE outputs and the residual; fp32 router logits and LM-head
 * logits.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "mk.h"
#include "mk_internal.h"

namespace mk {

constexpr int NC = MK_NC_WARPS;
constexpr int NCT = NC * 32;

/* ---------------------------------------------------------------- helpers */

__device__ __forceinline__ uint32_t saddr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ float rbf(float f) { return bf2f(f2bf(f)); }

/* 8 bf16 packed in a uint4 -> 8 floats (exact). */
__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int ld_acquire(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_volatile(const int32_t *p) {
  return *(const volatile int32_t *)p;
}

__device__ __forceinline__ void red_release_add(int32_t *p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int atom_add_acq_rel(int32_t *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_release(int32_t *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void bar_consumers() {
  asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");
}

/* mbarriers (CTA scope) */
__device__ __forceinline__ void mbar_init(uint64_t *b, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

/* 1-D TMA bulk copy global -> shared, completing on an mbarrier.  The
 * weights and cached K/V are streamed once per step: evict them first from
 * L2 so that activations and partials stay resident. */
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(saddr(dst)),
      "l"(src), "r"(bytes), "r"(saddr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

/* Sum over 32 lanes of NB values at once: after log2(NB) "transposing"
 * rounds each lane keeps one value, then plain butterfly rounds finish the
 * sum.  Lane l ends with the sum of v[l >> (5 - log2 NB)]. */
template <int NB>
__device__ __forceinline__ float transpose_reduce(float (&v)[NB], int lane) {
  constexpr int LOG = NB == 1 ? 0 : NB == 2 ? 1 : NB == 4 ? 2 : 3;
#pragma unroll
  for (int r = 0; r < LOG; ++r) {
    const int half = NB >> (r + 1);
    const int mask = 16 >> r;
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, mask);
    }
  }
  float s = v[0];
#pragma unroll
  for (int m = 16 >> LOG; m >= 1; m >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, m);
  return s;
}

template <int NB>
__device__ __forceinline__ int reduce_token(int lane) {
  constexpr int LOG = NB == 1 ? 0 : NB == 2 ? 1 : NB == 4 ? 2 : 3;
  return lane >> (5 - LOG);
}
template <int NB>
__device__ __forceinline__ bool reduce_leader(int lane) {
  constexpr int LOG = NB == 1 ? 0 : NB == 2 ? 1 : NB == 4 ? 2 : 3;
  return (lane & ((32 >> LOG) - 1)) == 0;
}

/* The DPL (= D / 32 <= 4) bf16 head dims of lane `lane` in a K or V row. */
__device__ __forceinline__ void lane_dims(const uint16_t *row, int lane, int DPL, float (&o)[4]) {
  if (DPL == 4) {
    const uint2 v = *(const uint2 *)(row + lane * 4);
    o[0] = __uint_as_float(v.x << 16);
    o[1] = __uint_as_float(v.x & 0xFFFF0000u);
    o[2] = __uint_as_float(v.y << 16);
    o[3] = __uint_as_float(v.y & 0xFFFF0000u);
  } else if (DPL == 2) {
    const uint32_t v = *(const uint32_t *)(row + lane * 2);
    o[0] = __uint_as_float(v << 16);
    o[1] = __uint_as_float(v & 0xFFFF0000u);
    o[2] = o[3] = 0.0f;
  } else {
    o[0] = bf2f(row[lane]);
    o[1] = o[2] = o[3] = 0.0f;
  }
}

/* acc[b] += w . x[b] over K elements (K % 8 == 0), w and x bf16 in shared
 * memory; lane l handles the 8-element chunks l, l + 32, ... */
template <int NB>
__device__ __forceinline__ void dot_row(const uint16_t *w, const uint16_t *x, int xstride, int K,
                                        int lane, float (&acc)[NB]) {
  for (int c = lane * 8; c < K; c += 256) {
    float wf[8];
    unpack8(*(const uint4 *)(w + c), wf);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float xf[8];
      unpack8(*(const uint4 *)(x + b * xstride + c), xf);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[b] = fmaf(wf[i], xf[i], acc[b]);
    }
  }
}

/* ----------------------------------------------------------- shared layout */

struct Misc {
  uint64_t full[MK_MAX_STAGES];
  uint64_t empty[MK_MAX_STAGES];
  int32_t dec[2];         /* collective decisions, double-buffered (0 ok, 1 abort) */
  int32_t norm_layer;     /* layer whose normed input sits in xbuf (-2: none) */
  int32_t pad0;
  float red[NC][MK_MAX_BATCH];
  float rsum[MK_MAX_BATCH];
  float part[2][512];     /* GEMV partial sums [row * S + seg][b], double-buffered */
  union {
    struct {
      float slot_w[128][MK_MAX_BATCH];
      float acc[MK_MAX_OUT_ROWS][MK_MAX_BATCH][2]; /* attn, moe */
    } out;
    struct {
      float pw[NC][8][8]; /* p of up to 8 keys x 8 head slots, per warp */
      float alpha[NC][8];
      float m[8][8], l[8][8]; /* merge exchange */
    } at;
    struct {
      float best[NC][MK_MAX_BATCH][2];
    } lm;
    struct {
      uint32_t used[4];
      int32_t ids[MK_MAX_BATCH][MK_MAX_TOPK];
      float w[MK_MAX_BATCH][MK_MAX_TOPK];
    } rt;
  } u;
};

struct Ctx {
  const mk_kparams *p;
  uint8_t *ring;
  uint8_t *xbuf;
  Misc *m;
  uint32_t epoch;
  int cta;
  int nstages;
};

__device__ __forceinline__ int32_t *lctr(const mk_kparams &p, int layer, int kind) {
  return p.ctr + ((size_t)layer * p.ctrs_per_layer + kind) * MK_CTR_STRIDE;
}
__device__ __forceinline__ int32_t *gctr(const mk_kparams &p, int kind) {
  return p.ctr + ((size_t)p.L * p.ctrs_per_layer + kind) * MK_CTR_STRIDE;
}

/* ------------------------------------------------------------ error paths */

__device__ void raise_error(const mk_kparams &p, int code, int cta, int task, int op, int layer,
                            int ctr, int seen, int target) {
  if (atomicCAS(&p.ctrl->err_code, 0, code) == 0) {
    p.ctrl->err_cta = cta;
    p.ctrl->err_task = task;
    p.ctrl->err_op = op;
    p.ctrl->err_layer = layer;
    p.ctrl->err_ctr = ctr;
    p.ctrl->err_seen = seen;
    p.ctrl->err_target = target;
    volatile int32_t *h = p.err_host;
    if (h) {
      h[1] = cta;
      h[2] = task;
      h[3] = op;
      h[4] = layer;
      h[5] = ctr;
      h[6] = seen;
      h[7] = target;
      __threadfence_system();
      h[0] = code;
      __threadfence_system();
    }
  }
  atomicExch(&p.ctrl->abort, 1);
}

/* Waits until (int)(*c - target) >= 0.  Bounded: gives up after the wait
 * limit (recording MK_ERR_DEVICE_TIMEOUT) or as soon as another CTA raised
 * the abort flag.  Returns false then. */
__device__ bool wait_counter(const Ctx &cx, int32_t *c, int target, int task, int op, int layer,
                             int ctr_kind) {
  const mk_kparams &p = *cx.p;
  int v = ld_acquire(c);
  if ((int)(v - target) >= 0) return true;
  const uint64_t t0 = gtimer();
  uint32_t spins = 0;
  while (true) {
    v = ld_acquire(c);
    if ((int)(v - target) >= 0) return true;
    if ((++spins & 31) == 0) {
      if (ld_volatile(&p.ctrl->abort)) return false;
      if (gtimer() - t0 > p.wait_limit_ns) {
        raise_error(p, MK_ERR_DEVICE_TIMEOUT, cx.cta, task, op, layer, ctr_kind, v, target);
        return false;
      }
    }
    __nanosleep(20);
  }
}

/* Waits for an mbarrier phase.  Bounded like wait_counter. */
__device__ bool wait_mbar(const Ctx &cx, uint64_t *bar, uint32_t parity, int task, int op,
                          int layer) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  uint32_t spins = 0;
  while (!mbar_test(bar, parity)) {
    if ((++spins & 127) == 0) {
      if (ld_volatile(&cx.p->ctrl->abort)) return false;
      if (gtimer() - t0 > cx.p->wait_limit_ns) {
        raise_error(*cx.p, MK_ERR_DEVICE_TIMEOUT, cx.cta, task, op, layer, -1, 0, 0);
        return false;
      }
    }
  }
  return true;
}

/* ============================================================== producer
 * One thread (lane 0 of the producer warp) walks the CTA's task list stage
 * by stage with two cursors over the same sequence:
 *   - the load cursor copies stage i into ring slot i % nstages (TMA bulk
 *     copies completing on full[slot]) once the consumers have released it;
 *   - the prefetch cursor runs up to MK_PREFETCH_STAGES stages further and
 *     asks L2 for those bytes (cp.async.bulk.prefetch.L2), so that when a
 *     slot frees the copy is served from L2 rather than paying the loaded
 *     HBM latency again.  It never waits: at a task whose bytes depend on
 *     routing that is not known yet it pauses until the load cursor passes.
 * Consumers walk the same deterministic stage sequence. */

#define MK_PREFETCH_STAGES 8

__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

struct Seg {
  const uint8_t *src;
  uint32_t off, bytes;
};

enum { IT_STAGE = 1, IT_END = 0, IT_BLOCKED = -1, IT_FAIL = -2 };

struct StageIter {
  const mk_kparams *p;
  const int32_t *row;
  int nl, nf;
  uint32_t epoch;
  int layer, k;   /* current task (layer == L: the final tasks) */
  bool started;
  long count;     /* stages produced */
  /* current task */
  int op;
  const int32_t *t;
  const mk_layer_dev *ly;
  const uint16_t *src; /* row streams */
  int r, nrows, K;
  int q, p1, b, kvh;   /* attention pages */
  int64_t v, v1;       /* gate/up share */
  int u, U;            /* OUT: u = -1 while on Wo rows, then the down slot */
  const mk_routing *rt;

  __device__ void init(const mk_kparams *pp, const int32_t *rw, uint32_t ep) {
    p = pp;
    row = rw;
    nl = rw[1];
    nf = rw[2];
    epoch = ep;
    layer = 0;
    k = 0;
    started = false;
    count = 0;
    if (nl == 0) layer = p->L; /* no layer tasks */
  }

  __device__ bool at_end() const { return layer > p->L || (layer == p->L && k >= nf); }

  __device__ void next_task() {
    started = false;
    ++k;
    if (layer < p->L && k >= nl) {
      k = 0;
      ++layer;
      if (layer < p->L && nl == 0) layer = p->L;
    }
  }

  /* Routing of this task's layer: known? (blocking: wait, bounded). */
  __device__ int routing(bool block, const Ctx &cx) {
    int32_t *c = lctr(*p, layer, CTR_ROUTED);
    if ((int)(ld_acquire(c) - (int)(epoch + 1)) >= 0) return IT_STAGE;
    if (!block) return IT_BLOCKED;
    return wait_counter(cx, c, (int)(epoch + 1), -1, OP_UP, layer, CTR_ROUTED) ? IT_STAGE : IT_FAIL;
  }

  __device__ void rows_from(const uint16_t *s0, int n, int KK) {
    src = s0;
    r = 0;
    nrows = n;
    K = KK;
  }

  __device__ int begin(bool block, const Ctx &cx) {
    t = row + MK_DESC_INTS * (1 + (layer < p->L ? k : nl + k));
    op = t[0];
    const int L = layer < p->L ? layer : p->L - 1;
    ly = p->layers + L;
    switch (op) {
      case OP_QKV: {
        const uint16_t *w = t[1] == 0 ? ly->wq : t[1] == 1 ? ly->wk : ly->wv;
        rows_from(w + (size_t)t[2] * p->d, t[3], p->d);
        return IT_STAGE;
      }
      case OP_ROUTER:
        rows_from(ly->wr + (size_t)t[2] * p->d, t[3], p->d);
        return IT_STAGE;
      case OP_LM:
        rows_from(p->lm_head + (size_t)t[2] * p->d, t[3], p->d);
        return IT_STAGE;
      case OP_ATTN:
        b = t[1];
        kvh = t[2];
        q = t[3];
        p1 = t[4] >= 0 ? t[4] : (__ldg(p->seq_lens + b) + p->P - 1) / p->P;
        return IT_STAGE;
      case OP_UP: {
        const int rs = routing(block, cx);
        if (rs != IT_STAGE) return rs;
        rt = p->routing + layer;
        U = __ldcg(&rt->U);
        const int64_t T = (int64_t)U * p->F;
        v = T * t[1] / t[2];
        v1 = T * (t[1] + 1) / t[2];
        return IT_STAGE;
      }
      case OP_OUT:
        u = -1;
        rows_from(ly->wo + (size_t)t[2] * p->Hq * p->D, t[3], p->Hq * p->D);
        return IT_STAGE;
      default:
        return IT_FAIL; /* the consumers report the bad opcode */
    }
  }

  __device__ bool row_stage(Seg *seg, int &nseg, uint32_t &total) {
    if (r >= nrows) return false;
    const uint32_t rb = (uint32_t)K * 2;
    const int cnt = min(mk_rows_per_stage(rb), nrows - r);
    seg[0].src = (const uint8_t *)(src + (size_t)r * K);
    seg[0].off = 0;
    seg[0].bytes = cnt * rb;
    nseg = 1;
    total = cnt * rb;
    r += cnt;
    return true;
  }

  /* IT_STAGE: a stage; IT_END: this task has no more; IT_BLOCKED / IT_FAIL */
  __device__ int emit(Seg *seg, int &nseg, uint32_t &total, bool block, const Ctx &cx) {
    switch (op) {
      case OP_QKV:
      case OP_ROUTER:
      case OP_LM:
        return row_stage(seg, nseg, total) ? IT_STAGE : IT_END;
      case OP_ATTN: {
        if (q >= p1) return IT_END;
        const uint32_t pb = (uint32_t)p->P * p->D * 2;
        const int cnt = min(mk_pages_per_stage(pb), p1 - q);
        for (int j = 0; j < cnt; ++j) {
          const int page = __ldg(p->page_table + b * p->max_pages + q + j);
          const size_t blk = ((size_t)page * p->Hkv + kvh) * p->P * p->D;
          seg[2 * j].src = (const uint8_t *)(ly->kc + blk);
          seg[2 * j + 1].src = (const uint8_t *)(ly->vc + blk);
          seg[2 * j].off = 2 * j * pb;
          seg[2 * j + 1].off = (2 * j + 1) * pb;
          seg[2 * j].bytes = seg[2 * j + 1].bytes = pb;
        }
        nseg = 2 * cnt;
        total = 2 * cnt * pb;
        q += cnt;
        return IT_STAGE;
      }
      case OP_UP: {
        if (v >= v1) return IT_END;
        const int F = p->F, d = p->d;
        const int uu = (int)(v / F), f0 = (int)(v % F);
        const int f1 = (int)min((int64_t)F, f0 + (v1 - v));
        const uint32_t rb = (uint32_t)d * 2;
        const int cnt = min(mk_pairs_per_stage(rb), f1 - f0);
        const int e = __ldcg(&rt->expert[uu]);
        const size_t eo = (size_t)e * F * d + (size_t)f0 * d;
        seg[0].src = (const uint8_t *)(ly->wg + eo);
        seg[1].src = (const uint8_t *)(ly->wu + eo);
        seg[0].off = 0;
        seg[1].off = cnt * rb;
        seg[0].bytes = seg[1].bytes = cnt * rb;
        nseg = 2;
        total = 2 * cnt * rb;
        v += cnt;
        return IT_STAGE;
      }
      case OP_OUT: {
        while (true) {
          if (row_stage(seg, nseg, total)) return IT_STAGE;
          if (u == -1) {
            const int rs = routing(block, cx);
            if (rs != IT_STAGE) return rs;
            rt = p->routing + layer;
            U = __ldcg(&rt->U);
          }
          ++u;
          if (u >= U) return IT_END;
          const int e = __ldcg(&rt->expert[u]);
          rows_from(ly->wd + ((size_t)e * p->d + t[2]) * p->F, t[3], p->F);
        }
      }
      default:
        return IT_FAIL;
    }
  }

  /* The next stage of the stream. */
  __device__ int next(Seg *seg, int &nseg, uint32_t &total, bool block, const Ctx &cx) {
    while (true) {
      if (at_end()) return IT_END;
      if (!started) {
        const int rs = begin(block, cx);
        if (rs != IT_STAGE) return rs;
        started = true;
      }
      const int rs = emit(seg, nseg, total, block, cx);
      if (rs == IT_STAGE) {
        ++count;
        return IT_STAGE;
      }
      if (rs != IT_END) return rs;
      next_task();
    }
  }
};

struct Producer {
  Ctx cx;
  uint64_t policy;
  int last_in_slot[MK_MAX_STAGES];

  __device__ void run(const int32_t *row) {
    for (int s = 0; s < MK_MAX_STAGES; ++s) last_in_slot[s] = -1;
    StageIter ld, pf;
    ld.init(cx.p, row, cx.epoch);
    pf.init(cx.p, row, cx.epoch);
    bool pf_end = false;
    Seg seg[16];
    int nseg;
    uint32_t total;
    while (true) {
      /* run the prefetch cursor ahead of the load cursor */
      while (!pf_end && pf.count < ld.count + MK_PREFETCH_STAGES) {
        const int rs = pf.next(seg, nseg, total, false, cx);
        if (rs == IT_STAGE) {
          if (pf.count > ld.count)
            for (int j = 0; j < nseg; ++j) prefetch_l2(seg[j].src, seg[j].bytes);
        } else {
          if (rs != IT_BLOCKED) pf_end = true;
          break;
        }
      }
      const int rs = ld.next(seg, nseg, total, true, cx);
      if (rs != IT_STAGE) break; /* end, or a failed wait (already reported) */
      const long i = ld.count - 1;
      const int slot = (int)(i % cx.nstages);
      if (i >= cx.nstages) {
        const uint32_t parity = (uint32_t)(((i / cx.nstages) - 1) & 1);
        if (!wait_mbar(cx, &cx.m->empty[slot], parity, -1, -1, -1)) break;
      }
      uint8_t *dst = cx.ring + (size_t)slot * MK_STAGE_BYTES;
      uint64_t *bar = &cx.m->full[slot];
      mbar_expect_tx(bar, total);
      for (int j = 0; j < nseg; ++j) bulk_g2s(dst + seg[j].off, seg[j].src, seg[j].bytes, bar, policy);
      last_in_slot[slot] = (int)i;
    }
    /* Every copy issued must land before the CTA exits (normally the
     * consumers have waited for all of them already). */
    for (int s = 0; s < cx.nstages; ++s) {
      const int k = last_in_slot[s];
      if (k < 0) continue;
      const uint32_t parity = (uint32_t)((k / cx.nstages) & 1);
      const uint64_t t0 = gtimer();
      while (!mbar_test(&cx.m->full[s], parity) && gtimer() - t0 < cx.p->wait_limit_ns) {
      }
    }
  }
};

/* ============================================================== consumers
 * Eight warps.  Each warp waits for, reads and releases every ring stage on
 * its own (lane 0 polls the stage's mbarrier, the warp follows), so warps
 * work on different stages at the same time and no CTA-wide barrier sits on
 * the streaming path.  Rows are owned by warps by their index within the
 * task, so every output element has one writer.  A failed wait (time limit
 * or abort) marks the warp; the consumers decide together at the next
 * collective point (a barrier with an OR reduction), so all consumer threads
 * always leave at the same point and no barrier is ever left half-arrived. */

/* Consumer-wide barrier returning the OR of every thread's predicate. */
__device__ __forceinline__ bool bar_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(NCT)
      : "memory");
  return r != 0;
}

/* acc[r][b] += w_r . x[b] over K elements for R rows sharing the x loads;
 * two accumulators per (row, token) keep the FMA chains short. */
template <int NB, int R>
__device__ __forceinline__ void dot_rows(const uint16_t *const (&w)[R], const uint16_t *x,
                                         int xstride, int K, int lane, float (&acc)[R][NB]) {
  float a2[R][NB][2];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) a2[r][b][0] = a2[r][b][1] = 0.0f;
  for (int c = lane * 8; c < K; c += 256) {
    uint4 wv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) wv[r] = *(const uint4 *)(w[r] + c);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float xf[8];
      unpack8(*(const uint4 *)(x + b * xstride + c), xf);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float wf[8];
        unpack8(wv[r], wf);
#pragma unroll
        for (int i = 0; i < 8; ++i) a2[r][b][i & 1] = fmaf(wf[i], xf[i], a2[r][b][i & 1]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[r][b] = a2[r][b][0] + a2[r][b][1];
}

__device__ __forceinline__ unsigned long long pack2(uint32_t lo, uint32_t hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ float sum2(unsigned long long v) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
  return __uint_as_float(lo) + __uint_as_float(hi);
}

/* Single-token rows against an fp32 activation (the batch-1 path): the bf16
 * weight pairs become fp32 pairs with one shift and one mask, and packed
 * f32x2 FMAs (two exact fp32 FMAs each) do the products. */
template <int NB, int R>
__device__ __forceinline__ void dot_rows(const uint16_t *const (&w)[R], const float *x, int xstride,
                                         int K, int lane, float (&acc)[R][NB]) {
  static_assert(NB == 1, "fp32 activations are the batch-1 path");
  unsigned long long a2[R][2];
#pragma unroll
  for (int r = 0; r < R; ++r) a2[r][0] = a2[r][1] = 0ULL;
  for (int c = lane * 8; c < K; c += 256) {
    const uint4 xa = *(const uint4 *)(x + c), xb = *(const uint4 *)(x + c + 4);
    const unsigned long long xp[4] = {pack2(xa.x, xa.y), pack2(xa.z, xa.w), pack2(xb.x, xb.y),
                                      pack2(xb.z, xb.w)};
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint4 wv = *(const uint4 *)(w[r] + c);
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        a2[r][j & 1] = ffma2(pack2(ww[j] << 16, ww[j] & 0xFFFF0000u), xp[j], a2[r][j & 1]);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r][0] = sum2(a2[r][0]) + sum2(a2[r][1]);
}

/* activation element type: fp32 for one token, bf16 bits otherwise */
template <class XT>
__device__ __forceinline__ XT to_x(uint16_t bits);
template <>
__device__ __forceinline__ float to_x<float>(uint16_t bits) {
  return bf2f(bits);
}
template <>
__device__ __forceinline__ uint16_t to_x<uint16_t>(uint16_t bits) {
  return bits;
}

template <int NB>
struct Consumer {
  using XT = typename std::conditional<NB == 1, float, uint16_t>::type;
  Ctx cx;
  int warp, lane, tid;
  int si;     /* stages consumed (the same sequence in every warp) */
  bool wfail; /* this warp failed a stage wait */
  unsigned long long *tr; /* this CTA's trace events, or NULL */
  int tr_n;
  uint64_t t_ready, t_stage, t_swait, t_mark;
  int n_stages;

  static constexpr int ROWS = NB <= 2 ? 2 : 1; /* rows per dot pass */

  /* Thread 0 waits on a counter; every consumer learns whether the CTA goes
   * on (false also when any warp has failed a stage wait). */
  __device__ bool cwait(int32_t *c, int target, int task, int op, int layer, int kind) {
    bool fail = wfail;
    if (tid == 0) {
      fail |= !wait_counter(cx, c, target, task, op, layer, kind);
      if (tr && !t_ready) t_ready = gtimer();
    }
    return !bar_any(fail);
  }

  /* End of a task's streaming part: a consumer barrier, false if any warp
   * failed. */
  __device__ bool task_end() { return !bar_any(wfail); }

  __device__ bool stage_wait(uint8_t *&st, int task, int op, int layer) {
    if (wfail) return false;
    const int slot = si % cx.nstages;
    const uint32_t parity = (uint32_t)((si / cx.nstages) & 1);
    int ok = 1;
    if (lane == 0) {
      const bool trace = tr && warp == 0;
      const uint64_t w0 = trace ? gtimer() : 0;
      ok = wait_mbar(cx, &cx.m->full[slot], parity, task, op, layer) ? 1 : 0;
      if (trace) {
        const uint64_t w1 = gtimer();
        if (!t_stage) t_stage = w1;
        else t_swait += w1 - w0;
        ++n_stages;
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) {
      wfail = true;
      return false;
    }
    mbar_test(&cx.m->full[slot], parity); /* completed: acquire order for this thread */
    st = cx.ring + (size_t)slot * MK_STAGE_BYTES;
    return true;
  }

  __device__ void stage_release() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&cx.m->empty[si % cx.nstages]);
    ++si;
  }

  __device__ const uint16_t *h_row(int layer, int b) const {
    const mk_kparams &p = *cx.p;
    if (layer == 0) return p.embed + (size_t)__ldg(p.tokens + b) * p.d;
    return p.h + ((size_t)layer * MK_MAX_BATCH + b) * p.d;
  }

  __device__ void block_sum(float (&v)[NB]) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float s = v[b];
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, m);
      if (lane == 0) cx.m->red[warp][b] = s;
    }
    bar_consumers();
    if (tid < NB) {
      float s = 0.0f;
      for (int w = 0; w < NC; ++w) s += cx.m->red[w][tid];
      cx.m->rsum[tid] = s;
    }
    bar_consumers();
#pragma unroll
    for (int b = 0; b < NB; ++b) v[b] = cx.m->rsum[b];
    bar_consumers();
  }

  /* xbuf[b][0..d) = bf16((h * (1/sqrtf(mean_fp32(h^2) + eps))) * g) as XT;
   * rows b >= B zero.  h is read once with 16-byte loads and staged behind
   * the output in xbuf. */
  __device__ void norm_into_xbuf(int layer_tag, const uint16_t *const *hrows, const uint16_t *g) {
    const mk_kparams &p = *cx.p;
    XT *x = (XT *)cx.xbuf;
    uint16_t *raw = (uint16_t *)(cx.xbuf + (size_t)NB * p.d * sizeof(XT));
    const int n8 = p.d / 8;
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ss[b] = 0.0f;
      if (b < p.B)
        for (int i = tid; i < n8; i += NCT) {
          const uint4 v = __ldcg((const uint4 *)hrows[b] + i);
          *(uint4 *)(raw + (size_t)b * p.d + 8 * i) = v;
          float f[8];
          unpack8(v, f);
#pragma unroll
          for (int k = 0; k < 8; ++k) ss[b] = fmaf(f[k], f[k], ss[b]);
        }
    }
    block_sum(ss);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float r = 1.0f / sqrtf(ss[b] / (float)p.d + p.eps);
      for (int i = tid; i < n8; i += NCT) {
        XT o[8];
        if (b < p.B) {
          float hf[8], gf[8];
          unpack8(*(const uint4 *)(raw + (size_t)b * p.d + 8 * i), hf);
          unpack8(__ldg((const uint4 *)g + i), gf);
#pragma unroll
          for (int k = 0; k < 8; ++k) o[k] = to_x<XT>(f2bf(__fmul_rn(__fmul_rn(hf[k], r), gf[k])));
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) o[k] = to_x<XT>(0);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) x[(size_t)b * p.d + 8 * i + k] = o[k];
      }
    }
    if (tid == 0) cx.m->norm_layer = layer_tag;
    bar_consumers();
  }

  __device__ void ensure_norm(int layer) {
    if (*(volatile int32_t *)&cx.m->norm_layer == layer) return;
    struct Mark {
      Consumer *c;
      __device__ ~Mark() {
        if (c->tr && c->tid == 0) c->t_mark = gtimer();
      }
    } mark{this};
    bar_consumers(); /* everyone has read the tag before it can change */
    const uint16_t *hr[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) hr[b] = b < cx.p->B ? h_row(layer, b) : nullptr;
    norm_into_xbuf(layer, hr, cx.p->layers[layer].norm);
  }

  __device__ void invalidate_norm() {
    bar_consumers();
    if (tid == 0) cx.m->norm_layer = -2;
  }

  /* After task_end(): thread 0 releases the downstream counter. */
  __device__ void signal(int32_t *c) {
    if (tid == 0) {
      __threadfence();
      red_release_add(c, 1);
    }
  }

  /* After task_end(): one increment of the ticket counter; true (for every
   * consumer) if this task took the last ticket of the step. */
  __device__ bool ticket(int32_t *c, int per_step) {
    bool last = false;
    if (tid == 0) {
      __threadfence();
      const int old = atom_add_acq_rel(c, 1);
      last = old == (int)((cx.epoch + 1) * (uint32_t)per_step) - 1;
    }
    return bar_any(last);
  }

  /* Reduce R rows' NB sums across the warp and hand them to epi(row, b, v)
   * on the lane that owns token b. */
  template <int R, class Epi>
  __device__ __forceinline__ void finish_rows(float (&acc)[R][NB], const int (&rows)[R], Epi &epi) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float s = transpose_reduce<NB>(acc[r], lane);
      if (reduce_leader<NB>(lane)) epi(rows[r], reduce_token<NB>(lane), s);
    }
  }

  /* nrows streamed rows of K elements; row r (index within the task) is
   * computed by warp r % 8 and handed to epi(r, b, value). */
  template <class Epi>
  __device__ void gemv_task(int nrows, int K, const XT *x, int xstride, int task, int op,
                            int layer, Epi epi) {
    const int rps = mk_rows_per_stage(K * 2);
    for (int r0 = 0; r0 < nrows; r0 += rps) {
      const int cnt = min(rps, nrows - r0);
      uint8_t *st;
      if (!stage_wait(st, task, op, layer)) return;
      const uint16_t *w = (const uint16_t *)st;
      int j = ((warp - r0) % NC + NC) % NC;
      if (ROWS == 2) {
        for (; j + NC < cnt; j += 2 * NC) {
          float acc[ROWS][NB];
          const uint16_t *wr[ROWS];
          int rr[ROWS];
#pragma unroll
          for (int r = 0; r < ROWS; ++r) {
            wr[r] = w + (size_t)(j + r * NC) * K;
            rr[r] = r0 + j + r * NC;
          }
          dot_rows<NB, ROWS>(wr, x, xstride, K, lane, acc);
          finish_rows<ROWS>(acc, rr, epi);
        }
      }
      for (; j < cnt; j += NC) {
        float acc[1][NB];
        const uint16_t *wr[1] = {w + (size_t)j * K};
        const int rr[1] = {r0 + j};
        dot_rows<NB, 1>(wr, x, xstride, K, lane, acc);
        finish_rows<1>(acc, rr, epi);
      }
      stage_release();
    }
  }

  /* ---------------------------------------------------------------- QKV */
  __device__ bool op_qkv(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    if (layer > 0 && !cwait(lctr(p, layer - 1, CTR_OUT_DONE), (int)((cx.epoch + 1) * p.n_out),
                            task, OP_QKV, layer, CTR_OUT_DONE))
      return false;
    ensure_norm(layer);
    const int QKVD = (p.Hq + 2 * p.Hkv) * p.D;
    const int base = (t[1] == 0 ? 0 : t[1] == 1 ? p.Hq * p.D : (p.Hq + p.Hkv) * p.D) + t[2];
    uint16_t *out = p.qkv + (size_t)layer * MK_MAX_BATCH * QKVD;
    const int B = p.B;
    gemv_task(t[3], p.d, (const XT *)cx.xbuf, p.d, task, OP_QKV, layer,
              [&](int r, int b, float v) {
                if (b < B) out[(size_t)b * QKVD + base + r] = f2bf(v);
              });
    if (!task_end()) return false;
    signal(lctr(p, layer, CTR_QKV_DONE));
    return true;
  }

  /* ------------------------------------------------------------- router */
  __device__ bool op_router(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    if (layer > 0 && !cwait(lctr(p, layer - 1, CTR_OUT_DONE), (int)((cx.epoch + 1) * p.n_out),
                            task, OP_ROUTER, layer, CTR_OUT_DONE))
      return false;
    ensure_norm(layer);
    const int e0 = t[2];
    float *lg = p.router_logits + (size_t)layer * MK_MAX_BATCH * p.E;
    const float *bias = p.layers[layer].bias;
    const int B = p.B, E = p.E;
    gemv_task(t[3], p.d, (const XT *)cx.xbuf, p.d, task, OP_ROUTER, layer,
              [&](int r, int b, float v) {
                if (b < B) lg[(size_t)b * E + e0 + r] = bias ? v + __ldg(bias + e0 + r) : v;
              });
    if (!task_end()) return false;
    if (!ticket(lctr(p, layer, CTR_ROUTER_TICKET), p.n_router)) return true;
    route(layer);
    bar_consumers();
    if (tid == 0) {
      __threadfence();
      st_release(lctr(p, layer, CTR_ROUTED), (int)(cx.epoch + 1));
    }
    return true;
  }

  /* The last router task: top-k per token (warp b), ties -> lower id;
   * weights = softmax over the chosen logits (the same as the softmax over
   * all E renormalised over the chosen k); then the distinct-expert slots in
   * ascending expert id. */
  __device__ void route(int layer) {
    const mk_kparams &p = *cx.p;
    mk_routing *rt = p.routing + layer;
    const float *lg = p.router_logits + (size_t)layer * MK_MAX_BATCH * p.E;
    auto &R = cx.m->u.rt;
    if (tid < 4) R.used[tid] = 0;
    bar_consumers();
    if (warp < p.B) {
      const int b = warp;
      float v[4];
      int id[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        id[i] = lane + 32 * i;
        v[i] = id[i] < p.E ? __ldcg(lg + (size_t)b * p.E + id[i]) : -INFINITY;
        if (id[i] >= p.E) id[i] = 0x40000000;
      }
      float top_v[MK_MAX_TOPK];
      int top_i[MK_MAX_TOPK];
      for (int k = 0; k < p.K; ++k) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (id[i] < 0x40000000 && (v[i] > bv || (v[i] == bv && id[i] < bi))) {
            bv = v[i];
            bi = id[i];
          }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
          const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, m);
          const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, m);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        top_v[k] = bv;
        top_i[k] = bi;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (id[i] == bi) id[i] = 0x40000000; /* taken */
      }
      if (lane == 0) {
        float z = 0.0f;
        for (int k = 0; k < p.K; ++k) z += expf(top_v[k] - top_v[0]);
        for (int k = 0; k < p.K; ++k) {
          const float w = expf(top_v[k] - top_v[0]) / z;
          R.ids[b][k] = top_i[k];
          R.w[b][k] = w;
          rt->ids[b][k] = top_i[k];
          rt->w[b][k] = w;
          atomicOr(&R.used[top_i[k] >> 5], 1u << (top_i[k] & 31));
        }
      }
    }
    bar_consumers();
    if (tid < p.E) {
      const int e = tid;
      if ((R.used[e >> 5] >> (e & 31)) & 1u) {
        int rank = __popc(R.used[e >> 5] & ((1u << (e & 31)) - 1u));
        for (int w = 0; w < (e >> 5); ++w) rank += __popc(R.used[w]);
        rt->expert[rank] = e;
        for (int b = 0; b < MK_MAX_BATCH; ++b) {
          float w = 0.0f;
          if (b < p.B)
            for (int k = 0; k < p.K; ++k)
              if (R.ids[b][k] == e) w = R.w[b][k];
          rt->slot_w[rank][b] = w;
        }
      }
    }
    if (tid == 0) {
      const int U = __popc(R.used[0]) + __popc(R.used[1]) + __popc(R.used[2]) + __popc(R.used[3]);
      rt->U = U;
      atomicAdd(&p.ctrl->sum_experts, (unsigned long long)U);
    }
  }
  /* ---------------------------------------------------------- attention
   * Split-K flash decoding over the pages of one (sequence, kv head).  Lane
   * l owns head dims [l*DPL, (l+1)*DPL) of all 8 head slots; the 8 partial
   * dot products of a key are summed across lanes in 9 shuffles, leaving
   * head slot (l >> 2) & 7 on lane l. */
  __device__ bool op_attn(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    const int b = t[1], kvh = t[2], p0 = t[3], last = t[8];
    const int D = p.D, G = p.Hq / p.Hkv, P = p.P, half = D / 2;
    const int L_now = __ldg(p.seq_lens + b);
    const int p1 = t[4] >= 0 ? t[4] : (L_now + P - 1) / P;
    if (!cwait(lctr(p, layer, CTR_QKV_DONE), (int)((cx.epoch + 1) * p.n_qkv), task, OP_ATTN,
               layer, CTR_QKV_DONE))
      return false;
    invalidate_norm();
    float *qs = (float *)cx.xbuf; /* [8][D] */
    float *ks = qs + 8 * D;       /* [D] */
    float *vs = ks + D;           /* [D] */
    float *mb = vs + D;           /* merge exchange [4][8][D] */
    const int QKVD = (p.Hq + 2 * p.Hkv) * D;
    const uint16_t *qkv = p.qkv + ((size_t)layer * MK_MAX_BATCH + b) * QKVD;
    const float *rp = p.rope + (size_t)L_now * half * 2;
    for (int i = tid; i < 8 * half; i += NCT) {
      const int g = i / half, j = i % half;
      float o1 = 0.0f, o2 = 0.0f;
      if (g < G) {
        const uint16_t *src = qkv + (size_t)(kvh * G + g) * D;
        const float x1 = bf2f(__ldcg(src + j)), x2 = bf2f(__ldcg(src + j + half));
        const float c = __ldg(rp + 2 * j), s = __ldg(rp + 2 * j + 1);
        o1 = rbf(__fmul_rn(x1, c) - __fmul_rn(x2, s));
        o2 = rbf(__fmul_rn(x2, c) + __fmul_rn(x1, s));
      }
      qs[g * D + j] = o1;
      qs[g * D + j + half] = o2;
    }
    if (last) {
      const uint16_t *ksrc = qkv + (size_t)(p.Hq + kvh) * D;
      const uint16_t *vsrc = qkv + (size_t)(p.Hq + p.Hkv + kvh) * D;
      const int page = __ldg(p.page_table + b * p.max_pages + L_now / P);
      const size_t row = (((size_t)page * p.Hkv + kvh) * P + (L_now % P)) * D;
      uint16_t *kc = p.layers[layer].kc + row, *vc = p.layers[layer].vc + row;
      for (int j = tid; j < half; j += NCT) {
        const float x1 = bf2f(__ldcg(ksrc + j)), x2 = bf2f(__ldcg(ksrc + j + half));
        const float c = __ldg(rp + 2 * j), s = __ldg(rp + 2 * j + 1);
        const uint16_t k1 = f2bf(__fmul_rn(x1, c) - __fmul_rn(x2, s));
        const uint16_t k2 = f2bf(__fmul_rn(x2, c) + __fmul_rn(x1, s));
        ks[j] = bf2f(k1);
        ks[j + half] = bf2f(k2);
        kc[j] = k1;
        kc[j + half] = k2;
      }
      for (int j = tid; j < D; j += NCT) {
        const uint16_t v = __ldcg(vsrc + j);
        vs[j] = bf2f(v);
        vc[j] = v;
      }
    }
    bar_consumers();

    const int DPL = D / 32;
    float qr[8][4], orr[8][4];
#pragma unroll
    for (int g = 0; g < 8; ++g)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qr[g][i] = i < DPL ? qs[g * D + lane * DPL + i] : 0.0f;
        orr[g][i] = 0.0f;
      }
    const int hg = (lane >> 2) & 7;
    float m_run = -INFINITY, l_run = 0.0f;
    const float scale = p.attn_scale;
    auto &A = cx.m->u.at;

    const uint16_t *kr[8], *vr[8];
    /* nt <= 8 keys, all valid: rows kr/vr in shared memory, or (newkey) the
     * new token's fp32 k and v vectors */
    auto block = [&](int nt, bool newkey) {
      float s_t[8];
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        s_t[tt] = -INFINITY;
        if (tt < nt) {
          float kv[4];
          if (newkey) {
#pragma unroll
            for (int i = 0; i < 4; ++i) kv[i] = i < DPL ? ks[lane * DPL + i] : 0.0f;
          } else {
            lane_dims(kr[tt], lane, DPL, kv);
          }
          float part[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) a = fmaf(qr[g][i], kv[i], a);
            part[g] = a;
          }
          s_t[tt] = transpose_reduce<8>(part, lane) * scale;
        }
      }
      float mnew = m_run;
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) mnew = fmaxf(mnew, s_t[tt]);
      const float alpha = (m_run == -INFINITY) ? 0.0f : expf(m_run - mnew);
      float lsum = 0.0f;
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        const float pv = (s_t[tt] == -INFINITY) ? 0.0f : expf(s_t[tt] - mnew);
        s_t[tt] = pv;
        lsum += pv;
      }
      l_run = l_run * alpha + lsum;
      m_run = mnew;
      if ((lane & 3) == 0) {
#pragma unroll
        for (int tt = 0; tt < 8; ++tt) A.pw[warp][tt][hg] = s_t[tt];
        A.alpha[warp][hg] = alpha;
      }
      __syncwarp();
      {
        const float4 a0 = *(const float4 *)&A.alpha[warp][0];
        const float4 a1 = *(const float4 *)&A.alpha[warp][4];
        const float al[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int g = 0; g < 8; ++g)
#pragma unroll
          for (int i = 0; i < 4; ++i) orr[g][i] *= al[g];
      }
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        if (tt < nt) {
          float vv[4];
          if (newkey) {
#pragma unroll
            for (int i = 0; i < 4; ++i) vv[i] = i < DPL ? vs[lane * DPL + i] : 0.0f;
          } else {
            lane_dims(vr[tt], lane, DPL, vv);
          }
          const float4 p0v = *(const float4 *)&A.pw[warp][tt][0];
          const float4 p1v = *(const float4 *)&A.pw[warp][tt][4];
          const float pg[8] = {p0v.x, p0v.y, p0v.z, p0v.w, p1v.x, p1v.y, p1v.z, p1v.w};
#pragma unroll
          for (int g = 0; g < 8; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i) orr[g][i] = fmaf(pg[g], vv[i], orr[g][i]);
        }
      }
      __syncwarp();
    };

    const uint32_t pb = (uint32_t)P * D * 2;
    const int pps = mk_pages_per_stage(pb);
    for (int q0 = p0; q0 < p1; q0 += pps) {
      const int cnt = min(pps, p1 - q0);
      uint8_t *st;
      if (!stage_wait(st, task, OP_ATTN, layer)) break;
      const int nkeys = cnt * P;
      const int valid_end = L_now - q0 * P;
      int nt = 0;
      for (int kk = warp; kk < nkeys; kk += NC) {
        if (kk < valid_end) {
          const int pg = kk / P, sl = kk % P;
          kr[nt] = (const uint16_t *)(st + 2 * pg * pb) + (size_t)sl * D;
          vr[nt] = (const uint16_t *)(st + (2 * pg + 1) * pb) + (size_t)sl * D;
          ++nt;
        }
        if (nt == 8) {
          block(8, false);
          nt = 0;
        }
      }
      if (nt > 0) block(nt, false);
      stage_release();
    }
    if (tr && tid == 0) t_mark = gtimer();
    if (last && warp == 0) block(1, true);

    /* merge warp states pairwise: 8 -> 4 -> 2 -> 1 */
    for (int hw = NC / 2; hw >= 1; hw >>= 1) {
      bar_consumers();
      if (warp >= hw && warp < 2 * hw) {
        const int s = warp - hw;
        if ((lane & 3) == 0) {
          A.m[s][hg] = m_run;
          A.l[s][hg] = l_run;
        }
#pragma unroll
        for (int g = 0; g < 8; ++g)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < DPL) mb[((size_t)s * 8 + g) * D + lane * DPL + i] = orr[g][i];
      }
      bar_consumers();
      if (warp < hw) {
        const float m2 = A.m[warp][hg], l2 = A.l[warp][hg];
        const float M = fmaxf(m_run, m2);
        const float f1 = m_run == -INFINITY ? 0.0f : expf(m_run - M);
        const float f2 = m2 == -INFINITY ? 0.0f : expf(m2 - M);
        l_run = f1 * l_run + f2 * l2;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float mg1 = __shfl_sync(0xFFFFFFFFu, m_run, g * 4);
          const float mg2 = A.m[warp][g];
          const float Mg = fmaxf(mg1, mg2);
          const float a1 = mg1 == -INFINITY ? 0.0f : expf(mg1 - Mg);
          const float a2 = mg2 == -INFINITY ? 0.0f : expf(mg2 - Mg);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < DPL)
              orr[g][i] = a1 * orr[g][i] + a2 * mb[((size_t)warp * 8 + g) * D + lane * DPL + i];
        }
        m_run = M;
      }
    }
    /* warp 0 holds this split's partial: per head [m, l, -, -, o[D]] */
    const int PS = D + 4;
    float *part = p.attn_part + ((size_t)layer * p.n_slots + t[5]) * G * PS;
    if (warp == 0) {
#pragma unroll
      for (int g = 0; g < 8; ++g)
        if (g < G) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < DPL) part[(size_t)g * PS + 4 + lane * DPL + i] = orr[g][i];
        }
      if ((lane & 3) == 0 && hg < G) {
        part[(size_t)hg * PS] = m_run;
        part[(size_t)hg * PS + 1] = l_run;
      }
    }
    /* the last split of (b, kvh) to finish merges all splits:
     * o = sum_s f_s o_s with f_s = e^{m_s - M} / sum_s' e^{m_s' - M} l_s' */
    if (!task_end()) return false;
    if (!ticket(lctr(p, layer, CTR_ATTN_TICKET0 + b * p.Hkv + kvh), t[7])) return true;
    const float *parts = p.attn_part + ((size_t)layer * p.n_slots + t[6]) * G * PS;
    uint16_t *o = p.o + ((size_t)layer * MK_MAX_BATCH + b) * p.Hq * D + (size_t)kvh * G * D;
    const int ns = t[7];
    float *fm = (float *)cx.xbuf;          /* [ns][G] m, then factors */
    float *fl = fm + ns * G;               /* [ns][G] l */
    float *hd = fl + ns * G;               /* [G] max, [G] 1 / denominator */
    for (int i = tid; i < ns * G; i += NCT) {
      fm[i] = __ldcg(parts + (size_t)i * PS);
      fl[i] = __ldcg(parts + (size_t)i * PS + 1);
    }
    bar_consumers();
    if (tid < G) {
      float M = -INFINITY;
      for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, fm[s2 * G + tid]);
      float den = 0.0f;
      for (int s2 = 0; s2 < ns; ++s2) {
        const float ms = fm[s2 * G + tid];
        if (ms != -INFINITY) den = fmaf(expf(ms - M), fl[s2 * G + tid], den);
      }
      hd[tid] = M;
      hd[G + tid] = 1.0f / den;
    }
    bar_consumers();
    for (int i = tid; i < ns * G; i += NCT) {
      const int g = i % G;
      const float ms = fm[i];
      fm[i] = ms == -INFINITY ? 0.0f : expf(ms - hd[g]) * hd[G + g];
    }
    bar_consumers();
    const int D4 = D / 4;
    for (int i = tid; i < G * D4; i += NCT) {
      const int g = i / D4, j4 = i % D4;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      const float4 *src = (const float4 *)(parts + (size_t)g * PS + 4) + j4;
      int s2 = 0;
      for (; s2 + 8 <= ns; s2 += 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (size_t)(s2 + u) * G * PS / 4);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float f = fm[(s2 + u) * G + g];
          acc.x = fmaf(f, v[u].x, acc.x);
          acc.y = fmaf(f, v[u].y, acc.y);
          acc.z = fmaf(f, v[u].z, acc.z);
          acc.w = fmaf(f, v[u].w, acc.w);
        }
      }
      for (; s2 < ns; ++s2) {
        const float4 v = __ldcg(src + (size_t)s2 * G * PS / 4);
        const float f = fm[s2 * G + g];
        acc.x = fmaf(f, v.x, acc.x);
        acc.y = fmaf(f, v.y, acc.y);
        acc.z = fmaf(f, v.z, acc.z);
        acc.w = fmaf(f, v.w, acc.w);
      }
      uint16_t *dst = o + (size_t)g * D + j4 * 4;
      dst[0] = f2bf(acc.x);
      dst[1] = f2bf(acc.y);
      dst[2] = f2bf(acc.z);
      dst[3] = f2bf(acc.w);
    }
    bar_consumers();
    signal(lctr(p, layer, CTR_ATTN_DONE));
    return true;
  }

  /* ------------------------------------------------------ expert gate/up
   * Row pair j of the share (one gate row, one up row of the same expert
   * and f) is computed by warp j % 8. */
  __device__ bool op_up(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    if (!cwait(lctr(p, layer, CTR_ROUTED), (int)(cx.epoch + 1), task, OP_UP, layer, CTR_ROUTED))
      return false;
    ensure_norm(layer);
    const mk_routing *rt = p.routing + layer;
    const int U = __ldcg(&rt->U);
    const int d = p.d, F = p.F, B = p.B;
    const int64_t T = (int64_t)U * F;
    int64_t v = T * t[1] / t[2];
    const int64_t v1 = T * (t[1] + 1) / t[2];
    const XT *x = (const XT *)cx.xbuf;
    const int rps = mk_pairs_per_stage(2 * d);
    int pair0 = 0; /* pairs of this share before the current stage */
    while (v < v1 && !wfail) {
      const int u = (int)(v / F), f0 = (int)(v % F);
      const int f1 = (int)min((int64_t)F, f0 + (v1 - v));
      uint16_t *out = p.act + (((size_t)layer * p.u_max + u) * MK_MAX_BATCH) * F;
      for (int f = f0; f < f1; f += rps) {
        const int cnt = min(rps, f1 - f);
        uint8_t *st;
        if (!stage_wait(st, task, OP_UP, layer)) break;
        const uint16_t *wg = (const uint16_t *)st, *wu = wg + (size_t)cnt * d;
        for (int j = ((warp - pair0) % NC + NC) % NC; j < cnt; j += NC) {
          float acc[2][NB];
          const uint16_t *wr[2] = {wg + (size_t)j * d, wu + (size_t)j * d};
          dot_rows<NB, 2>(wr, x, d, d, lane, acc);
          const float g = transpose_reduce<NB>(acc[0], lane);
          const float uu = transpose_reduce<NB>(acc[1], lane);
          const int b = reduce_token<NB>(lane);
          if (reduce_leader<NB>(lane) && b < B) {
            const float gb = rbf(g), ub = rbf(uu);
            const float silu = gb / (1.0f + expf(-gb));
            out[(size_t)b * F + f + j] = f2bf(silu * ub);
          }
        }
        stage_release();
        pair0 += cnt;
      }
      v += f1 - f0;
    }
    if (!task_end()) return false;
    signal(lctr(p, layer, CTR_UP_DONE));
    return true;
  }

  /* ---------------------------------- Wo, expert down + combine, residual */
  __device__ bool op_out(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    const int r0 = t[2], nr = t[3], B = p.B, d = p.d, F = p.F, HqD = p.Hq * p.D;
    const int target = (int)((cx.epoch + 1) * p.n_attn_done) +
                       (layer == p.poison_layer ? p.poison_delta : 0);
    if (!cwait(lctr(p, layer, CTR_ATTN_DONE), target, task, OP_OUT, layer, CTR_ATTN_DONE))
      return false;
    invalidate_norm();
    XT *x = (XT *)cx.xbuf;
    auto &O = cx.m->u.out;
    for (int i = tid; i < NB * HqD; i += NCT) {
      const int bb = i / HqD;
      x[i] = to_x<XT>(bb < B ? __ldcg(p.o + ((size_t)layer * MK_MAX_BATCH + bb) * HqD + (i % HqD))
                             : (uint16_t)0);
    }
    for (int i = tid; i < MK_MAX_OUT_ROWS * MK_MAX_BATCH * 2; i += NCT) (&O.acc[0][0][0])[i] = 0.0f;
    bar_consumers();
    gemv_task(nr, HqD, x, HqD, task, OP_OUT, layer,
              [&](int r, int bb, float v) { O.acc[r][bb][0] = v; });
    if (!cwait(lctr(p, layer, CTR_UP_DONE), (int)((cx.epoch + 1) * p.n_up), task, OP_OUT, layer,
               CTR_UP_DONE))
      return false;
    const mk_routing *rt = p.routing + layer;
    const int U = __ldcg(&rt->U);
    for (int i = tid; i < U * MK_MAX_BATCH; i += NCT)
      O.slot_w[i / MK_MAX_BATCH][i % MK_MAX_BATCH] =
          __ldcg(&rt->slot_w[i / MK_MAX_BATCH][i % MK_MAX_BATCH]);
    /* the experts' activations: all slots at once when they fit the buffer,
     * else two slots at a time */
    const int per = NB * F;
    const int fit = (int)min((int64_t)U, (int64_t)cx.p->xbuf_bytes / ((int64_t)sizeof(XT) * per));
    const bool all = fit >= U;
    for (int u = 0; u < U; ++u) {
      const int bufslot = all ? u : (u & 1);
      XT *xa = x + (size_t)bufslot * per;
      if (all ? u == 0 : true) {
        const int n_load = all ? U : 1;
        for (int k = 0; k < n_load; ++k) {
          const int uu = all ? k : u;
          XT *dst = x + (size_t)(all ? k : bufslot) * per;
          const uint16_t *a = p.act + (((size_t)layer * p.u_max + uu) * MK_MAX_BATCH) * F;
          for (int i = tid; i < per; i += NCT)
            dst[i] = to_x<XT>((i / F) < B ? __ldcg(a + i) : (uint16_t)0);
        }
        bar_consumers();
      }
      gemv_task(nr, F, xa, F, task, OP_OUT, layer, [&](int r, int bb, float v) {
        const float sw = O.slot_w[u][bb];
        if (bb < B && sw != 0.0f) O.acc[r][bb][1] = fmaf(sw, v, O.acc[r][bb][1]);
      });
    }
    if (!task_end()) return false;
    for (int i = tid; i < nr * B; i += NCT) {
      const int r = i / B, bb = i % B;
      const uint16_t *hin = h_row(layer, bb);
      const float hv = bf2f(__ldcg(hin + r0 + r));
      const float at = rbf(O.acc[r][bb][0]);
      const float mo = rbf(O.acc[r][bb][1]);
      p.h[((size_t)(layer + 1) * MK_MAX_BATCH + bb) * d + r0 + r] =
          f2bf(__fadd_rn(__fadd_rn(hv, at), mo));
      if (layer == 0) p.h[(size_t)bb * d + r0 + r] = __ldg(hin + r0 + r);
    }
    bar_consumers();
    signal(lctr(p, layer, CTR_OUT_DONE));
    return true;
  }

  /* ---------------------------------------------- final norm + LM head */
  __device__ bool op_lm(const int32_t *t, int task) {
    const mk_kparams &p = *cx.p;
    const int L = p.L, B = p.B;
    if (!cwait(lctr(p, L - 1, CTR_OUT_DONE), (int)((cx.epoch + 1) * p.n_out), task, OP_LM, L,
               CTR_OUT_DONE))
      return false;
    if (*(volatile int32_t *)&cx.m->norm_layer != L) {
      bar_consumers();
      const uint16_t *hr[NB];
#pragma unroll
      for (int bb = 0; bb < NB; ++bb)
        hr[bb] = bb < B ? p.h + ((size_t)L * MK_MAX_BATCH + bb) * p.d : nullptr;
      norm_into_xbuf(L, hr, p.final_norm);
    }
    const int v0 = t[2];
    float best_v = -INFINITY;
    int best_i = 0x7FFFFFFF;
    float *logits = p.out_logits;
    const int V = p.V;
    /* the lane that owns token b in each warp keeps that warp's best */
    gemv_task(t[3], p.d, (const XT *)cx.xbuf, p.d, task, OP_LM, L,
              [&](int r, int bb, float v) {
                if (bb < B) {
                  if (logits) logits[(size_t)bb * V + v0 + r] = v;
                  if (v > best_v || (v == best_v && v0 + r < best_i)) {
                    best_v = v;
                    best_i = v0 + r;
                  }
                }
              });
    auto &M = cx.m->u.lm;
    if (reduce_leader<NB>(lane)) {
      M.best[warp][reduce_token<NB>(lane)][0] = best_v;
      M.best[warp][reduce_token<NB>(lane)][1] = __int_as_float(best_i);
    }
    if (!task_end()) return false;
    if (tid < B) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
      for (int w = 0; w < NC; ++w) {
        const float v = M.best[w][tid][0];
        const int i = __float_as_int(M.best[w][tid][1]);
        if (v > bv || (v == bv && i < bi)) {
          bv = v;
          bi = i;
        }
      }
      p.lm_part[((size_t)t[4] * MK_MAX_BATCH + tid) * 2] = bv;
      p.lm_part[((size_t)t[4] * MK_MAX_BATCH + tid) * 2 + 1] = __int_as_float(bi);
    }
    bar_consumers();
    if (!ticket(gctr(p, GCTR_LM_TICKET), p.n_lm)) return true;
    if (tid < B) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
      for (int k = 0; k < p.n_lm; ++k) {
        const float v = __ldcg(p.lm_part + ((size_t)k * MK_MAX_BATCH + tid) * 2);
        const int i = __float_as_int(__ldcg(p.lm_part + ((size_t)k * MK_MAX_BATCH + tid) * 2 + 1));
        if (v > bv || (v == bv && i < bi)) {
          bv = v;
          bi = i;
        }
      }
      p.out_next[tid] = bi;
      p.seq_lens[tid] = p.seq_lens[tid] + 1;
    }
    return true;
  }

  __device__ bool dispatch(const int32_t *t, int task, int layer) {
    uint64_t t0 = 0;
    if (tr && tid == 0) {
      t0 = gtimer();
      t_ready = t_stage = t_swait = t_mark = 0;
      n_stages = 0;
    }
    bool ok;
    switch (t[0]) {
      case OP_QKV: ok = op_qkv(t, task, layer); break;
      case OP_ROUTER: ok = op_router(t, task, layer); break;
      case OP_ATTN: ok = op_attn(t, task, layer); break;
      case OP_UP: ok = op_up(t, task, layer); break;
      case OP_OUT: ok = op_out(t, task, layer); break;
      case OP_LM: ok = op_lm(t, task); break;
      default:
        if (tid == 0) raise_error(*cx.p, MK_ERR_BAD_TASK, cx.cta, task, t[0], layer, -1, 0, 0);
        ok = false;
    }
    if (tr && tid == 0 && tr_n < cx.p->trace_cap) {
      unsigned long long *e = tr + (size_t)tr_n * MK_TRACE_WORDS;
      e[0] = (unsigned long long)(t[0] | (layer << 8) | (task << 20));
      e[1] = t0;
      e[2] = t_ready ? t_ready : t0;
      e[3] = t_stage;
      e[4] = gtimer();
      e[5] = t_swait;
      e[6] = (unsigned long long)n_stages;
      e[7] = t_mark;
      ++tr_n;
    }
    return ok;
  }

  /* returns false if the CTA stopped early */
  __device__ bool run(const int32_t *row) {
    si = 0;
    wfail = false;
    const mk_kparams &p = *cx.p;
    const int nl = row[1], nf = row[2];
    for (int l = 0; l < p.L; ++l)
      for (int k = 0; k < nl; ++k)
        if (!dispatch(row + MK_DESC_INTS * (1 + k), k, l)) return false;
    for (int k = 0; k < nf; ++k)
      if (!dispatch(row + MK_DESC_INTS * (1 + nl + k), nl + k, p.L)) return false;
    return true;
  }
};

template <int NB>
__global__ void __launch_bounds__(MK_THREADS, 1) decode_kernel(const mk_kparams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctx cx;
  cx.p = &p;
  cx.nstages = p.ring_stages;
  cx.ring = smem;
  cx.xbuf = smem + (size_t)p.ring_stages * MK_STAGE_BYTES;
  cx.m = (Misc *)(cx.xbuf + p.xbuf_bytes);
  cx.cta = blockIdx.x;
  cx.epoch = *(volatile uint32_t *)&p.ctrl->epoch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int32_t s_ok;
  if (threadIdx.x == 0) {
    for (int s = 0; s < cx.nstages; ++s) {
      mbar_init(&cx.m->full[s], 1);
      mbar_init(&cx.m->empty[s], NC);
    }
    cx.m->norm_layer = -2;
    s_ok = 1;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int32_t *row = p.table + (size_t)blockIdx.x * p.tasks_per_cta * MK_DESC_INTS;
  const bool header_ok = row[0] == OP_HEADER;
  if (header_ok) {
    if (warp == NC) {
      if (lane == 0) {
        Producer pr;
        pr.cx = cx;
        pr.policy = evict_first_policy();
        pr.run(row);
      }
      __syncwarp();
    } else {
      Consumer<NB> c;
      c.cx = cx;
      c.warp = warp;
      c.lane = lane;
      c.tid = threadIdx.x;
      c.tr = p.trace ? p.trace + (size_t)blockIdx.x * p.trace_cap * MK_TRACE_WORDS : nullptr;
      c.tr_n = 0;
      const bool ok = c.run(row);
      if (threadIdx.x == 0 && !ok) s_ok = 0;
    }
  } else if (threadIdx.x == 0) {
    raise_error(p, MK_ERR_BAD_TASK, blockIdx.x, -1, row[0], -1, -1, 0, 0);
    s_ok = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_ok && !ld_volatile(&p.ctrl->abort)) {
    /* the last CTA out advances the epoch */
    __threadfence();
    const int old = atom_add_acq_rel(gctr(p, GCTR_EXIT), 1);
    if (old == (int)((cx.epoch + 1) * (uint32_t)gridDim.x) - 1)
      *(volatile uint32_t *)&p.ctrl->epoch = cx.epoch + 1;
  }
}

}  // namespace mk

/* ---- library-internal entry points (used by mk_api.cpp) ------------------ */

extern "C" size_t mk_misc_bytes() { return sizeof(mk::Misc); }

static void *mk_kernel_fn(int nb) {
  return nb == 1   ? (void *)mk::decode_kernel<1>
         : nb == 2 ? (void *)mk::decode_kernel<2>
         : nb == 4 ? (void *)mk::decode_kernel<4>
                   : (void *)mk::decode_kernel<8>;
}

extern "C" cudaError_t mk_kernel_prepare(int nb, size_t smem, int *blocks_per_sm) {
  void *fn = mk_kernel_fn(nb);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, MK_THREADS, smem);
}

extern "C" cudaError_t mk_launch(const mk_kparams *p, int nb, int grid, size_t smem,
                                 cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MK_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[] = {(void *)p};
  return cudaLaunchKernelExC(&cfg, mk_kernel_fn(nb), args);
}
