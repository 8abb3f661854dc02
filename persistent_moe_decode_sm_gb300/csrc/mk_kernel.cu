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
 * Streams every task's immutable bytes into ring slot i % nstages (stage i).
 * Consumers walk the same deterministic stage sequence. */

struct Producer {
  Ctx cx;
  int i; /* stages issued */
  uint64_t policy;
  int lane;
  int last_in_slot[MK_MAX_STAGES];

  __device__ bool acquire_slot(uint8_t *&dst, uint64_t *&bar) {
    const int slot = i % cx.nstages;
    if (i >= cx.nstages) {
      const uint32_t parity = (uint32_t)(((i / cx.nstages) - 1) & 1);
      bool ok = true;
      if (lane == 0) ok = wait_mbar(cx, &cx.m->empty[slot], parity, -1, -1, -1);
      if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) return false;
    }
    dst = cx.ring + (size_t)slot * MK_STAGE_BYTES;
    bar = &cx.m->full[slot];
    return true;
  }

  /* One stage of nseg segments; lane k issues segment k (nseg <= 32). */
  __device__ bool issue(int nseg, const uint8_t *const *src, const uint32_t *off,
                        const uint32_t *bytes, uint32_t total) {
    uint8_t *dst;
    uint64_t *bar;
    if (!acquire_slot(dst, bar)) return false;
    if (lane == 0) mbar_expect_tx(bar, total);
    __syncwarp();
    if (lane < nseg) bulk_g2s(dst + off[lane], src[lane], bytes[lane], bar, policy);
    last_in_slot[i % cx.nstages] = i;
    ++i;
    return true;
  }

  __device__ bool rows(const uint16_t *src, int nrows, int K) {
    const uint32_t rb = (uint32_t)K * 2;
    const int rps = mk_rows_per_stage(rb);
    for (int r = 0; r < nrows; r += rps) {
      const int cnt = min(rps, nrows - r);
      const uint8_t *s = (const uint8_t *)(src + (size_t)r * K);
      uint32_t off = 0, by = cnt * rb;
      if (!issue(1, &s, &off, &by, by)) return false;
    }
    return true;
  }

  /* Gate and up rows [f0, f1) of one expert: cnt gate rows then cnt up rows. */
  __device__ bool up_rows(const uint16_t *wg, const uint16_t *wu, int f0, int f1, int d) {
    const uint32_t rb = (uint32_t)d * 2;
    const int rps = mk_pairs_per_stage(rb);
    for (int f = f0; f < f1; f += rps) {
      const int cnt = min(rps, f1 - f);
      const uint8_t *s[2] = {(const uint8_t *)(wg + (size_t)f * d),
                             (const uint8_t *)(wu + (size_t)f * d)};
      uint32_t off[2] = {0, cnt * rb}, by[2] = {cnt * rb, cnt * rb};
      if (!issue(2, s, off, by, 2 * cnt * rb)) return false;
    }
    return true;
  }

  /* K and V blocks of logical pages [p0, p1) of sequence b, kv head kvh:
   * page j of a stage brings K at 2j * pb and V at (2j + 1) * pb. */
  __device__ bool pages(const mk_layer_dev &ly, int b, int kvh, int p0, int p1) {
    const mk_kparams &p = *cx.p;
    const uint32_t pb = (uint32_t)p.P * p.D * 2;
    const int pps = mk_pages_per_stage(pb);
    for (int q = p0; q < p1; q += pps) {
      const int cnt = min(pps, p1 - q);
      const uint8_t *s[16];
      uint32_t off[16], by[16];
      for (int j = 0; j < cnt; ++j) {
        const int page = __ldg(p.page_table + b * p.max_pages + q + j);
        const size_t blk = ((size_t)page * p.Hkv + kvh) * p.P * p.D;
        s[2 * j] = (const uint8_t *)(ly.kc + blk);
        s[2 * j + 1] = (const uint8_t *)(ly.vc + blk);
        off[2 * j] = 2 * j * pb;
        off[2 * j + 1] = (2 * j + 1) * pb;
        by[2 * j] = by[2 * j + 1] = pb;
      }
      if (!issue(2 * cnt, s, off, by, 2 * cnt * pb)) return false;
    }
    return true;
  }

  __device__ bool routed_wait(int layer) {
    bool ok = true;
    if (lane == 0)
      ok = wait_counter(cx, lctr(*cx.p, layer, CTR_ROUTED), (int)(cx.epoch + 1), -1, OP_UP, layer,
                        CTR_ROUTED);
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  }

  __device__ bool task(const int32_t *t, int layer) {
    const mk_kparams &p = *cx.p;
    switch (t[0]) {
      case OP_QKV: {
        const mk_layer_dev &ly = p.layers[layer];
        const uint16_t *w = t[1] == 0 ? ly.wq : t[1] == 1 ? ly.wk : ly.wv;
        return rows(w + (size_t)t[2] * p.d, t[3], p.d);
      }
      case OP_ROUTER:
        return rows(p.layers[layer].wr + (size_t)t[2] * p.d, t[3], p.d);
      case OP_ATTN: {
        const int b = t[1];
        const int p1 = t[4] >= 0 ? t[4] : (__ldg(p.seq_lens + b) + p.P - 1) / p.P;
        return pages(p.layers[layer], b, t[2], t[3], p1);
      }
      case OP_UP: {
        if (!routed_wait(layer)) return false;
        const mk_routing *rt = p.routing + layer;
        const int U = __ldcg(&rt->U);
        const mk_layer_dev &ly = p.layers[layer];
        const int64_t T = (int64_t)U * p.F;
        int64_t v = T * t[1] / t[2];
        const int64_t v1 = T * (t[1] + 1) / t[2];
        while (v < v1) {
          const int u = (int)(v / p.F), f0 = (int)(v % p.F);
          const int f1 = (int)min((int64_t)p.F, f0 + (v1 - v));
          const int e = __ldcg(&rt->expert[u]);
          const size_t eo = (size_t)e * p.F * p.d;
          if (!up_rows(ly.wg + eo, ly.wu + eo, f0, f1, p.d)) return false;
          v += f1 - f0;
        }
        return true;
      }
      case OP_OUT: {
        const mk_layer_dev &ly = p.layers[layer];
        const int HqD = p.Hq * p.D;
        if (!rows(ly.wo + (size_t)t[2] * HqD, t[3], HqD)) return false;
        if (!routed_wait(layer)) return false;
        const mk_routing *rt = p.routing + layer;
        const int U = __ldcg(&rt->U);
        for (int u = 0; u < U; ++u) {
          const int e = __ldcg(&rt->expert[u]);
          if (!rows(ly.wd + ((size_t)e * p.d + t[2]) * p.F, t[3], p.F)) return false;
        }
        return true;
      }
      case OP_LM:
        return rows(p.lm_head + (size_t)t[2] * p.d, t[3], p.d);
      default:
        return false; /* the consumers report the bad opcode */
    }
  }

  __device__ void run(const int32_t *row) {
    i = 0;
    for (int s = 0; s < MK_MAX_STAGES; ++s) last_in_slot[s] = -1;
    const int nl = row[1], nf = row[2];
    const mk_kparams &p = *cx.p;
    bool ok = true;
    for (int l = 0; l < p.L && ok; ++l)
      for (int k = 0; k < nl && ok; ++k) ok = task(row + MK_DESC_INTS * (1 + k), l);
    for (int k = 0; k < nf && ok; ++k) ok = task(row + MK_DESC_INTS * (1 + nl + k), p.L - 1);
    /* Every copy issued must land before the CTA exits (normally the
     * consumers have waited for all of them already). */
    if (lane == 0)
      for (int s = 0; s < cx.nstages; ++s) {
        const int k = last_in_slot[s];
        if (k < 0) continue;
        const uint32_t parity = (uint32_t)((k / cx.nstages) & 1);
        const uint64_t t0 = gtimer();
        while (!mbar_test(&cx.m->full[s], parity) && gtimer() - t0 < p.wait_limit_ns) {
        }
      }
    __syncwarp();
  }
};

/* ============================================================== consumers
 * Eight warps.  Every decision that can end a task early (a counter wait, a
 * stage wait) is taken by thread 0 and broadcast through a named barrier, so
 * all consumer threads always leave at the same point and no barrier can be
 * left half-arrived. */

template <int NB>
struct Consumer {
  Ctx cx;
  int warp, lane, tid;
  int si;   /* stages consumed */
  int dseq; /* collective decisions taken */

  /* Thread 0's verdict (ok) becomes everyone's. */
  __device__ bool decide(bool ok) {
    const int slot = dseq & 1;
    ++dseq;
    if (tid == 0) cx.m->dec[slot] = ok ? 0 : 1;
    bar_consumers();
    return *(volatile int32_t *)&cx.m->dec[slot] == 0;
  }

  __device__ bool cwait(int32_t *c, int target, int task, int op, int layer, int kind) {
    bool ok = true;
    if (tid == 0) ok = wait_counter(cx, c, target, task, op, layer, kind);
    return decide(ok);
  }

  __device__ bool stage_begin(uint8_t *&st, int task, int op, int layer) {
    const int slot = si % cx.nstages;
    const uint32_t parity = (uint32_t)((si / cx.nstages) & 1);
    bool ok = true;
    if (tid == 0) ok = wait_mbar(cx, &cx.m->full[slot], parity, task, op, layer);
    if (!decide(ok)) return false;
    mbar_test(&cx.m->full[slot], parity); /* completed: gives this thread acquire order */
    st = cx.ring + (size_t)slot * MK_STAGE_BYTES;
    return true;
  }

  __device__ void stage_end() {
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

  /* xbuf[b][0..d) = bf16((h * (1/sqrtf(mean_fp32(h^2) + eps))) * g); rows b >= B zero. */
  __device__ void norm_into_xbuf(int layer_tag, const uint16_t *const *hrows, const uint16_t *g) {
    const mk_kparams &p = *cx.p;
    uint16_t *x = (uint16_t *)cx.xbuf;
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ss[b] = 0.0f;
      if (b < p.B)
        for (int i = tid; i < p.d; i += NCT) {
          const float v = bf2f(__ldcg(hrows[b] + i));
          ss[b] = fmaf(v, v, ss[b]);
        }
    }
    block_sum(ss);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float r = 1.0f / sqrtf(ss[b] / (float)p.d + p.eps);
      for (int i = tid; i < p.d; i += NCT) {
        uint16_t o = 0;
        if (b < p.B) {
          const float hv = bf2f(__ldcg(hrows[b] + i));
          o = f2bf(__fmul_rn(__fmul_rn(hv, r), bf2f(__ldg(g + i))));
        }
        x[b * p.d + i] = o;
      }
    }
    if (tid == 0) cx.m->norm_layer = layer_tag;
    bar_consumers();
  }

  __device__ void ensure_norm(int layer) {
    if (*(volatile int32_t *)&cx.m->norm_layer == layer) return;
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

  __device__ void signal(int32_t *c) {
    bar_consumers();
    if (tid == 0) {
      __threadfence();
      red_release_add(c, 1);
    }
  }

  /* Adds one to the ticket counter; true (for every consumer) if this task
   * took the last ticket of the step. */
  __device__ bool ticket(int32_t *c, int per_step) {
    bar_consumers();
    bool last = false;
    if (tid == 0) {
      __threadfence();
      const int old = atom_add_acq_rel(c, 1);
      last = old == (int)((cx.epoch + 1) * (uint32_t)per_step) - 1;
    }
    return !decide(!last);
  }

  /* ---- GEMV of one stage: rows [0, cnt) of K elements at w.  S warps share
   * a row (S = largest power of two with S * cnt <= 8); each writes the
   * partial sum of its K segment to part[(row * S + seg) * NB + b]. */
  static __device__ __forceinline__ int segs(int cnt) {
    int S = 1;
    while (S * 2 * cnt <= NC) S *= 2;
    return S;
  }

  __device__ void partials(const uint16_t *w, int cnt, int K, const uint16_t *x, int xstride,
                           float *part) {
    const int S = segs(cnt);
    const int seg = warp % S, kseg = K / S, k0 = seg * kseg;
    for (int row = warp / S; row < cnt; row += NC / S) {
      float acc[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
      dot_row<NB>(w + (size_t)row * K + k0, x + k0, xstride, kseg, lane, acc);
      const float s = transpose_reduce<NB>(acc, lane);
      if (reduce_leader<NB>(lane)) part[(row * S + seg) * NB + reduce_token<NB>(lane)] = s;
    }
  }

  __device__ __forceinline__ float psum(const float *part, int row, int b, int S) const {
    float s = 0.0f;
    for (int g = 0; g < S; ++g) s += part[(row * S + g) * NB + b];
    return s;
  }

  /* nrows streamed rows of K: epi(row, b, value) for every row and b < NB,
   * run by one consumer thread per (row, b). */
  template <class Epi>
  __device__ bool gemv_task(int nrows, int K, const uint16_t *x, int xstride, int task, int op,
                            int layer, Epi epi) {
    const int rps = mk_rows_per_stage(K * 2);
    int prev_r0 = -1, prev_cnt = 0, buf = 0;
    for (int r0 = 0; r0 < nrows; r0 += rps) {
      const int cnt = min(rps, nrows - r0);
      uint8_t *st;
      if (!stage_begin(st, task, op, layer)) return false;
      if (prev_r0 >= 0) {
        const float *pp = cx.m->part[buf ^ 1];
        const int S = segs(prev_cnt);
        for (int i = tid; i < prev_cnt * NB; i += NCT)
          epi(prev_r0 + i / NB, i % NB, psum(pp, i / NB, i % NB, S));
      }
      partials((const uint16_t *)st, cnt, K, x, xstride, cx.m->part[buf]);
      stage_end();
      prev_r0 = r0;
      prev_cnt = cnt;
      buf ^= 1;
    }
    if (prev_r0 >= 0) {
      bar_consumers();
      const float *pp = cx.m->part[buf ^ 1];
      const int S = segs(prev_cnt);
      for (int i = tid; i < prev_cnt * NB; i += NCT)
        epi(prev_r0 + i / NB, i % NB, psum(pp, i / NB, i % NB, S));
    }
    return true;
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
    if (!gemv_task(t[3], p.d, (const uint16_t *)cx.xbuf, p.d, task, OP_QKV, layer,
                   [&](int r, int b, float v) {
                     if (b < B) out[(size_t)b * QKVD + base + r] = f2bf(v);
                   }))
      return false;
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
    if (!gemv_task(t[3], p.d, (const uint16_t *)cx.xbuf, p.d, task, OP_ROUTER, layer,
                   [&](int r, int b, float v) {
                     if (b < B) lg[(size_t)b * E + e0 + r] = bias ? v + __ldg(bias + e0 + r) : v;
                   }))
      return false;
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

    /* nt <= 8 keys (rows in shared memory, or fp32 vectors), all valid */
    auto block = [&](const uint16_t *const *krow, const uint16_t *const *vrow, const float *kf,
                     const float *vf, int nt) {
      float s_t[8];
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        s_t[tt] = -INFINITY;
        if (tt < nt) {
          float kv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            kv[i] = i < DPL ? (kf ? kf[lane * DPL + i] : bf2f(krow[tt][lane * DPL + i])) : 0.0f;
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
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const float a = A.alpha[warp][g];
#pragma unroll
        for (int i = 0; i < 4; ++i) orr[g][i] *= a;
      }
      for (int tt = 0; tt < nt; ++tt) {
        float vv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          vv[i] = i < DPL ? (vf ? vf[lane * DPL + i] : bf2f(vrow[tt][lane * DPL + i])) : 0.0f;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float pg = A.pw[warp][tt][g];
#pragma unroll
          for (int i = 0; i < 4; ++i) orr[g][i] = fmaf(pg, vv[i], orr[g][i]);
        }
      }
      __syncwarp();
    };

    const uint32_t pb = (uint32_t)P * D * 2;
    const int pps = mk_pages_per_stage(pb);
    for (int q0 = p0; q0 < p1; q0 += pps) {
      const int cnt = min(pps, p1 - q0);
      uint8_t *st;
      if (!stage_begin(st, task, OP_ATTN, layer)) return false;
      const int nkeys = cnt * P;
      const int valid_end = L_now - q0 * P;
      const uint16_t *kr[8], *vr[8];
      int nt = 0;
      for (int kk = warp; kk < nkeys; kk += NC) {
        if (kk < valid_end) {
          const int pg = kk / P, sl = kk % P;
          kr[nt] = (const uint16_t *)(st + 2 * pg * pb) + (size_t)sl * D;
          vr[nt] = (const uint16_t *)(st + (2 * pg + 1) * pb) + (size_t)sl * D;
          ++nt;
        }
        if (nt == 8) {
          block(kr, vr, nullptr, nullptr, 8);
          nt = 0;
        }
      }
      if (nt > 0) block(kr, vr, nullptr, nullptr, nt);
      stage_end();
    }
    if (last && warp == 0) block(nullptr, nullptr, ks, vs, 1);

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
    /* warp 0 holds this split's partial */
    float *part = p.attn_part + ((size_t)layer * p.n_slots + t[5]) * G * (D + 2);
    if (warp == 0) {
#pragma unroll
      for (int g = 0; g < 8; ++g)
        if (g < G) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < DPL) part[(size_t)g * (D + 2) + 2 + lane * DPL + i] = orr[g][i];
        }
      if ((lane & 3) == 0 && hg < G) {
        part[(size_t)hg * (D + 2)] = m_run;
        part[(size_t)hg * (D + 2) + 1] = l_run;
      }
    }
    /* the last split of (b, kvh) to finish merges all splits */
    if (!ticket(lctr(p, layer, CTR_ATTN_TICKET0 + b * p.Hkv + kvh), t[7])) return true;
    const float *parts = p.attn_part + ((size_t)layer * p.n_slots + t[6]) * G * (D + 2);
    uint16_t *o = p.o + ((size_t)layer * MK_MAX_BATCH + b) * p.Hq * D + (size_t)kvh * G * D;
    const int ns = t[7];
    for (int i = tid; i < G * D; i += NCT) {
      const int g = i / D, j = i % D;
      float M = -INFINITY;
      for (int s = 0; s < ns; ++s) M = fmaxf(M, __ldcg(parts + ((size_t)s * G + g) * (D + 2)));
      float num = 0.0f, den = 0.0f;
      for (int s = 0; s < ns; ++s) {
        const float *ps = parts + ((size_t)s * G + g) * (D + 2);
        const float ms = __ldcg(ps);
        if (ms == -INFINITY) continue;
        const float f = expf(ms - M);
        num = fmaf(f, __ldcg(ps + 2 + j), num);
        den = fmaf(f, __ldcg(ps + 1), den);
      }
      o[(size_t)g * D + j] = f2bf(num / den);
    }
    signal(lctr(p, layer, CTR_ATTN_DONE));
    return true;
  }

  /* ------------------------------------------------------ expert gate/up */
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
    const uint16_t *x = (const uint16_t *)cx.xbuf;
    const int rps = mk_pairs_per_stage(2 * d);
    int buf = 0, prev_cnt = 0;
    uint16_t *prev_out = nullptr;
    auto epi = [&](uint16_t *out, int cnt) {
      const float *pp = cx.m->part[buf ^ 1];
      const int S = segs(2 * cnt);
      for (int i = tid; i < cnt * NB; i += NCT) {
        const int j = i / NB, bb = i % NB;
        if (bb < B) {
          const float gb = rbf(psum(pp, j, bb, S)), ub = rbf(psum(pp, cnt + j, bb, S));
          const float silu = gb / (1.0f + expf(-gb));
          out[(size_t)bb * F + j] = f2bf(silu * ub);
        }
      }
    };
    while (v < v1) {
      const int u = (int)(v / F), f0 = (int)(v % F);
      const int f1 = (int)min((int64_t)F, f0 + (v1 - v));
      uint16_t *out = p.act + (((size_t)layer * p.u_max + u) * MK_MAX_BATCH) * F;
      for (int f = f0; f < f1; f += rps) {
        const int cnt = min(rps, f1 - f);
        uint8_t *st;
        if (!stage_begin(st, task, OP_UP, layer)) return false;
        if (prev_out) epi(prev_out, prev_cnt);
        partials((const uint16_t *)st, 2 * cnt, d, x, d, cx.m->part[buf]);
        stage_end();
        prev_out = out + f;
        prev_cnt = cnt;
        buf ^= 1;
      }
      v += f1 - f0;
    }
    if (prev_out) {
      bar_consumers();
      epi(prev_out, prev_cnt);
    }
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
    uint16_t *x = (uint16_t *)cx.xbuf;
    auto &O = cx.m->u.out;
    for (int i = tid; i < NB * HqD; i += NCT) {
      const int bb = i / HqD;
      x[i] = bb < B ? __ldcg(p.o + ((size_t)layer * MK_MAX_BATCH + bb) * HqD + (i % HqD)) : 0;
    }
    for (int i = tid; i < MK_MAX_OUT_ROWS * MK_MAX_BATCH * 2; i += NCT) (&O.acc[0][0][0])[i] = 0.0f;
    bar_consumers();
    if (!gemv_task(nr, HqD, x, HqD, task, OP_OUT, layer,
                   [&](int r, int bb, float v) { O.acc[r][bb][0] = v; }))
      return false;
    if (!cwait(lctr(p, layer, CTR_UP_DONE), (int)((cx.epoch + 1) * p.n_up), task, OP_OUT, layer,
               CTR_UP_DONE))
      return false;
    const mk_routing *rt = p.routing + layer;
    const int U = __ldcg(&rt->U);
    for (int i = tid; i < U * MK_MAX_BATCH; i += NCT)
      O.slot_w[i / MK_MAX_BATCH][i % MK_MAX_BATCH] =
          __ldcg(&rt->slot_w[i / MK_MAX_BATCH][i % MK_MAX_BATCH]);
    for (int u = 0; u < U; ++u) {
      uint16_t *xa = x + (size_t)(u & 1) * NB * F;
      const uint16_t *a = p.act + (((size_t)layer * p.u_max + u) * MK_MAX_BATCH) * F;
      for (int i = tid; i < NB * F; i += NCT) xa[i] = (i / F) < B ? __ldcg(a + i) : 0;
      bar_consumers();
      if (!gemv_task(nr, F, xa, F, task, OP_OUT, layer, [&](int r, int bb, float v) {
            const float sw = O.slot_w[u][bb];
            if (bb < B && sw != 0.0f) O.acc[r][bb][1] = fmaf(sw, v, O.acc[r][bb][1]);
          }))
        return false;
    }
    bar_consumers();
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
    /* one thread per (row, b) in each epilogue; NCT is a multiple of NB, so
     * the token of a thread (tid % NB) never changes and it keeps a best */
    if (!gemv_task(t[3], p.d, (const uint16_t *)cx.xbuf, p.d, task, OP_LM, L,
                   [&](int r, int bb, float v) {
                     if (bb < B) {
                       if (logits) logits[(size_t)bb * V + v0 + r] = v;
                       if (v > best_v || (v == best_v && v0 + r < best_i)) {
                         best_v = v;
                         best_i = v0 + r;
                       }
                     }
                   }))
      return false;
    auto &M = cx.m->u.lm;
    {
      const int bb = tid % NB;
#pragma unroll
      for (int m = 16; m >= NB; m >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, best_v, m);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, best_i, m);
        if (ov > best_v || (ov == best_v && oi < best_i)) {
          best_v = ov;
          best_i = oi;
        }
      }
      if (lane < NB) {
        M.best[warp][bb][0] = best_v;
        M.best[warp][bb][1] = __int_as_float(best_i);
      }
    }
    bar_consumers();
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
    switch (t[0]) {
      case OP_QKV: return op_qkv(t, task, layer);
      case OP_ROUTER: return op_router(t, task, layer);
      case OP_ATTN: return op_attn(t, task, layer);
      case OP_UP: return op_up(t, task, layer);
      case OP_OUT: return op_out(t, task, layer);
      case OP_LM: return op_lm(t, task);
      default:
        if (tid == 0) raise_error(*cx.p, MK_ERR_BAD_TASK, cx.cta, task, t[0], layer, -1, 0, 0);
        return false;
    }
  }

  /* returns false if the CTA stopped early */
  __device__ bool run(const int32_t *row) {
    si = 0;
    dseq = 0;
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
      Producer pr;
      pr.cx = cx;
      pr.lane = lane;
      pr.policy = evict_first_policy();
      pr.run(row);
    } else {
      Consumer<NB> c;
      c.cx = cx;
      c.warp = warp;
      c.lane = lane;
      c.tid = threadIdx.x;
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
