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
 *               cached K/V pages) into a ring of eight shared-memory slots
 *               with TMA (cp.async.bulk for weight rows, tensor-map boxes
 *               with a 128-byte swizzle for K/V pages) completing on
 *               mbarriers.  It runs ahead of the consumers and does NOT wait
 *               for a task's data dependency before loading its weights --
 *               the weight prefetch ahead of dependencies that the
 *               aiweekly.co page ranks third among the method's gains
 *               (paragraph 4).  Only the expert weights wait, for the
 *               routing that names them.
 *
 * Ring slot w belongs to consumer warp w: stage i of the CTA's stream lands
 * in slot i % 8 and warp i % 8 consumes all of it on its own, so the eight
 * warps work on eight stages at once with no CTA-wide barrier on the
 * streaming path.  The dense contractions run on the tensor cores
 * (mma.sync m16n8k16, bf16 in, fp32 accumulate):
 *   - every GEMV: the up-to-8 tokens are the M side (rows 8-15 are zero),
 *     eight weight rows the N side, so the fp32 sums come out of the
 *     accumulator already reduced over K;
 *   - attention: the GQA group of up to 8 query heads against 16-key tiles,
 *     S = Q K^T and O += P V with P split into a bf16 high and low part so
 *     that the probabilities keep about 16 significant bits.
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
/* Batch 1 on the CUDA cores (fp32 FMAs straight on the bf16 halves) or, like
 * batch 2..8, on the tensor cores (one token in the M rows of m16n8k16). */
constexpr bool kB1CudaCores = true;
constexpr int NCT = NC * 32;
static_assert(NC % MK_NP_WARPS == 0, "each ring slot must have one producer");
#define NEG_INF (-INFINITY)

/* ---------------------------------------------------------------- helpers */

__device__ __forceinline__ uint32_t saddr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

/* Knuth's TwoSum: s = fl(a + b) and e with s + e == a + b exactly (round to
 * nearest, no overflow).  The _rn intrinsics keep the compiler from
 * reassociating. */
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

/* (hi, lo) += x: hi takes the rounded sum, lo collects the errors */
__device__ __forceinline__ void pair_add(float &hi, float &lo, float x) {
  float s, e;
  two_sum(hi, x, s, e);
  hi = s;
  lo = __fadd_rn(lo, e);
}

/* (hi, lo) += (h2, l2), renormalised with Dekker's Fast2Sum so that
 * hi == fl(hi + lo) */
__device__ __forceinline__ void pair_merge(float &hi, float &lo, float h2, float l2) {
  float s, e;
  two_sum(hi, h2, s, e);
  e = __fadd_rn(e, __fadd_rn(lo, l2));
  hi = __fadd_rn(s, e);
  lo = __fsub_rn(e, __fsub_rn(hi, s));
}

__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ float rbf(float f) { return bf2f(f2bf(f)); }

/* two bf16 in one register, `lo` in the low half (the lower k index) */
__device__ __forceinline__ uint32_t pack_bf16(uint16_t lo, uint16_t hi) {
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

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

/* SM cycle counter: cheap enough for per-stage timestamps (the stage trace
 * converts it to globaltimer time with an anchor pair) */
__device__ __forceinline__ uint64_t sclock() { return clock64(); }

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

/* A poll of a counter other CTAs update: relaxed, so that the spin does not
 * order (and slow) anything; the successful poll is followed by one acquire
 * fence. */
__device__ __forceinline__ int ld_relaxed(const int32_t *p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

/* Tagged words: {payload, tag} in one 64-bit relaxed store / load.  A word
 * read with this step's tag is this step's value: no fence or counter is
 * needed between the writer and the reader. */
__device__ __forceinline__ void st_tag(uint64_t *a, uint32_t payload, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(a),
               "l"(((unsigned long long)tag << 32) | payload)
               : "memory");
}
__device__ __forceinline__ uint64_t ld_tag(const uint64_t *a) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ bool tag_ok(uint64_t w, uint32_t tag) { return (uint32_t)(w >> 32) == tag; }

__device__ __forceinline__ void fence_acquire_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

/* CTA-scope release / acquire on a shared-memory word. */
__device__ __forceinline__ void st_release_cta(int32_t *p, int v) {
  asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(p)),
               "r"(v)
               : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.cta.shared.b32 %0, [%1];"
               : "=r"(v)
               : "r"((uint32_t)__cvta_generic_to_shared(p))
               : "memory");
  return v;
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
/* mbarrier arrive by the lanes with p set, as one predicated instruction:
 * no branch, so the warp stays converged */
__device__ __forceinline__ void mbar_arrive_if(uint64_t *b, bool p) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.u32 q, %1, 0;\n @q mbarrier.arrive.shared::cta.b64 _, [%0];\n}\n" ::"r"(
          saddr(b)),
      "r"((uint32_t)p)
      : "memory");
}
/* 32-bit shared store by the lanes with p set (one predicated instruction) */
__device__ __forceinline__ void sts32_if(float *a, float v, bool p) {
  asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q st.shared.f32 [%0], %1;\n}\n" ::"r"(
                   saddr(a)),
               "f"(v), "r"((uint32_t)p)
               : "memory");
}
/* 64-bit global store by the lanes with p set (one predicated instruction) */
__device__ __forceinline__ void st64_if(unsigned long long *a, unsigned long long v, bool p) {
  asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q st.global.u64 [%0], %1;\n}\n" ::"l"(a),
               "l"(v), "r"((uint32_t)p)
               : "memory");
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

/* As mbar_test, but the thread may be suspended (for up to ns nanoseconds)
 * until the phase completes instead of returning at once: a waiting warp
 * then takes no issue slots from the warps computing beside it. */
__device__ __forceinline__ bool mbar_wait_hint(uint64_t *b, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity), "r"(ns)
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

/* 3-D TMA tensor-map box global -> shared at coordinates {0, 0, z}. */
__device__ __forceinline__ void tensor_g2s_3d(void *dst, const void *tmap, int z, uint64_t *bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(saddr(dst)),
      "l"(tmap), "r"(0), "r"(0), "r"(z), "r"(saddr(bar)), "l"(policy)
      : "memory");
}

/* 2-D TMA tensor-map box global -> shared at coordinates {x, y}. */
__device__ __forceinline__ void tensor_g2s_2d(void *dst, const void *tmap, int x, int y,
                                              uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(saddr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(saddr(bar)), "l"(policy)
      : "memory");
}

/* a layer's norm gain, from the parameter space when it is there */
__device__ __forceinline__ const uint16_t *lnorm(const mk_kparams &p, int layer) {
  return layer < MK_PARAM_LAYERS ? p.l_norm[layer] : p.layers[layer].norm;
}

__device__ __forceinline__ void prefetch_tensormap(const void *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

/* ldmatrix: four 8x8 b16 matrices; lane l gives the row address of matrix
 * l / 8, row l % 8.  Plain: thread (g, t) gets row g, columns 2t, 2t+1;
 * transposed: rows 2t, 2t+1 of column g. */
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

/* c += A B, m16n8k16, bf16 x bf16 -> fp32.  Thread (g = lane/4, t = lane%4)
 * holds A rows g (a0, a2) and g + 8 (a1, a3) at k-pairs 2t (a0, a1) and
 * 2t + 8 (a2, a3); B column g at k-pairs 2t (b0) and 2t + 8 (b1); C rows g
 * (c0, c1) and g + 8 (c2, c3) at columns 2t, 2t + 1. */
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

/* -------------------------------------------------------- skinny GEMV tile
 * out[v][b] = W(v) . x_b for the R (virtual) rows v of one ring stage --
 * virtual row v at byte ro(v) of the stage -- and the NB token vectors x_b
 * (pitch xp elements), on the tensor cores: the tokens are the M side of an
 * m16n8k16 tile, eight weight rows the N side, and the fp32 sums come out of
 * the accumulator already reduced over K.  Each thread reads 16-byte pieces
 * of A and B at the same column offsets of each 64-column block, so the k
 * order inside a block is a permutation of its columns, the same on both
 * sides of every product that is kept, and each sum is over all columns.
 * Four accumulators (one per k step) keep the mma chains independent.
 * epi(n0, sums of the n-tile at rows n0.., sums of the n-tile at n0 + 8..,
 * whether that second tile exists) runs on every lane; see take_out.
 *
 * A quarter-warp's load covers B columns (virtual rows) 2i and 2i + 1 at the
 * same offsets.  Two layouts keep those loads free of bank conflicts:
 *
 * - Eight tokens (the stage's second run 64 bytes out of line, activations
 *   at pitch K + 32): the two rows, and the two tokens, already sit in
 *   opposite halves of the bank window.  Token g is A row g (rows 8..15
 *   zero); thread (g, t) reads columns 8t.. and 32 + 8t.. and ends with
 *   token g against rows n0 + 2t (c0) and n0 + 2t + 1 (c1).
 * - Fewer tokens (contiguous runs, all rows in the same banks): odd-g
 *   threads read the upper half of each 128-byte block first.  That changes
 *   which columns feed which k slot on odd threads, so token b is entered
 *   twice on the M side, row 2b with the even order and row 2b + 1 with the
 *   odd one, and C[m][n] is valid where m and n have the same parity: thread
 *   (g, t) ends with row n0 + 2t + (g & 1) for token g / 2 (c0 or c1). */
template <int NB, class RowMap, class Epi>
__device__ __forceinline__ void mma_rows(const uint8_t *st, int R, int K, const uint16_t *x,
                                         int xp, int lane, RowMap &&ro, Epi &&epi) {
  static_assert(NB >= MK_RUN_GAP_MIN_NB || NB <= 4, "duplicated tokens fill at most 8 A rows");
  const int g = lane >> 2, t = lane & 3;
  constexpr bool kGap = NB >= MK_RUN_GAP_MIN_NB;
  const int q = kGap ? 0 : (g & 1);
  const int tok = kGap ? g : (g >> 1);
  const bool hx = tok < NB;
  const int f0 = 8 * t + 32 * q; /* first piece of each 64-column block */
  const int sd = q ? -32 : 32;   /* the second piece, relative to the first */
  const uint16_t *xa = x + (size_t)(hx ? tok : 0) * xp + f0;
  for (int n0 = 0; n0 < R; n0 += 16) {
    const bool two = n0 + 8 < R;
    /* rows past R: nothing loaded (eight tokens) or the last row again */
    const bool ra = !kGap || n0 + g < R, rb = !kGap || n0 + 8 + g < R;
    const uint16_t *wa = (const uint16_t *)(st + ro(min(n0 + g, R - 1))) + f0;
    const uint16_t *wb = (const uint16_t *)(st + ro(min(n0 + 8 + g, R - 1))) + f0;
    float ca[4][4], cb[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) ca[i][k] = cb[i][k] = 0.0f;
#pragma unroll 2
    for (int c0 = 0; c0 < K; c0 += 64) {
      uint4 af = make_uint4(0, 0, 0, 0), as = af, wf = af, ws = af;
      if (hx) {
        af = *(const uint4 *)(xa + c0);
        as = *(const uint4 *)(xa + c0 + sd);
      }
      if (ra) {
        wf = *(const uint4 *)(wa + c0);
        ws = *(const uint4 *)(wa + c0 + sd);
      }
      mma16816(ca[0], af.x, 0u, af.y, 0u, wf.x, wf.y);
      mma16816(ca[1], af.z, 0u, af.w, 0u, wf.z, wf.w);
      mma16816(ca[2], as.x, 0u, as.y, 0u, ws.x, ws.y);
      mma16816(ca[3], as.z, 0u, as.w, 0u, ws.z, ws.w);
      if (two) {
        uint4 vf = make_uint4(0, 0, 0, 0), vs = vf;
        if (rb) {
          vf = *(const uint4 *)(wb + c0);
          vs = *(const uint4 *)(wb + c0 + sd);
        }
        mma16816(cb[0], af.x, 0u, af.y, 0u, vf.x, vf.y);
        mma16816(cb[1], af.z, 0u, af.w, 0u, vf.z, vf.w);
        mma16816(cb[2], as.x, 0u, as.y, 0u, vs.x, vs.y);
        mma16816(cb[3], as.z, 0u, as.w, 0u, vs.z, vs.w);
      }
    }
    float sa[4], sb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      sa[k] = (ca[0][k] + ca[1][k]) + (ca[2][k] + ca[3][k]);
      sb[k] = (cb[0][k] + cb[1][k]) + (cb[2][k] + cb[3][k]);
    }
    epi(n0, sa, sb, two);
  }
}

/* The valid outputs of one n-tile of mma_rows on this lane, f(v, b, value):
 * eight tokens, token g against virtual rows n0 + 2t and n0 + 2t + 1; fewer,
 * token g / 2 against row n0 + 2t + (g & 1).  Rows < R, tokens < NB. */
template <int NB, class F>
__device__ __forceinline__ void take_out(int n0, const float (&c)[4], int R, int lane, F &&f) {
  const int g = lane >> 2, t = lane & 3;
  if (NB >= MK_RUN_GAP_MIN_NB) {
    const int v = n0 + 2 * t;
    if (g < NB) {
      if (v < R) f(v, g, c[0]);
      if (v + 1 < R) f(v + 1, g, c[1]);
    }
  } else {
    const int q = g & 1, v = n0 + 2 * t + q;
    if (v < R && (g >> 1) < NB) f(v, g >> 1, q ? c[1] : c[0]);
  }
}

/* Sum over 32 lanes of 8 values at once: three "transposing" rounds leave
 * each lane one partial, two plain butterfly rounds finish: lanes 4r..4r+3
 * end with the sum of v[r]. */
__device__ __forceinline__ float transpose_reduce8(float (&v)[8], int lane) {
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int half = 8 >> (r + 1), mask = 16 >> r;
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, mask);
    }
  }
  float s = v[0];
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
  return s;
}

/* acc + a * b on the low (H = 0) or high (H = 1) bf16 halves of the words a
 * and b, in fp32 with one rounding: a product of two bf16 values is exact in
 * fp32, so this is the fp32 fma of the two values -- with no separate
 * conversion of either operand. */
template <int H>
__device__ __forceinline__ float fma_bf16h(uint32_t a, uint32_t b, float acc) {
  float d;
  if (H == 0)
    asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
        " fma.rn.f32.bf16 %0, al, bl, %3;\n}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(acc));
  else
    asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
        " fma.rn.f32.bf16 %0, ah, bh, %3;\n}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(acc));
  return d;
}

/* 8 bytes of shared memory at a shared-window address */
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

/* NR rows (virtual n0 .. n0 + NR - 1) of one token on the CUDA cores; the
 * row count is a template parameter so that every load of the block can be
 * issued ahead of the FMAs.  st and x are shared-window addresses, read with
 * explicit shared loads.  Each 32-bit word of a row and of x holds two bf16
 * columns; four accumulators per row (low and high halves of the two words a
 * lane reads per chunk) keep the fma chains independent.  v[r] gets this
 * lane's partial sum of row r. */
template <int NR>
__device__ __forceinline__ void cc_block(uint32_t st, int n0, int pitch, int K, uint32_t x,
                                         int lane, int pairs, float (&v)[8]) {
  uint32_t w[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const int vr = n0 + r;
    const int row = pairs ? ((vr & 1) ? pairs + (vr >> 1) : (vr >> 1)) : vr;
    w[r] = st + (uint32_t)(row * pitch) + 8u * lane;
  }
  float a[NR][4];
#pragma unroll
  for (int r = 0; r < NR; ++r) a[r][0] = a[r][1] = a[r][2] = a[r][3] = 0.0f;
  const uint32_t xl = x + 8u * lane;
  const int K128 = K & ~127; /* K is a multiple of 64: a half block may remain */
#pragma unroll 2
  for (int c = 0; c < K128; c += 128) {
    const uint2 xv = lds64(xl + 2u * c);
    uint2 wv[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) wv[r] = lds64(w[r] + 2u * c);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      a[r][0] = fma_bf16h<0>(wv[r].x, xv.x, a[r][0]);
      a[r][1] = fma_bf16h<1>(wv[r].x, xv.x, a[r][1]);
      a[r][2] = fma_bf16h<0>(wv[r].y, xv.y, a[r][2]);
      a[r][3] = fma_bf16h<1>(wv[r].y, xv.y, a[r][3]);
    }
  }
  if (K128 < K && lane < 16) {
    const uint2 xv = lds64(xl + 2u * K128);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const uint2 wv = lds64(w[r] + 2u * K128);
      a[r][0] = fma_bf16h<0>(wv.x, xv.x, a[r][0]);
      a[r][1] = fma_bf16h<1>(wv.x, xv.x, a[r][1]);
      a[r][2] = fma_bf16h<0>(wv.y, xv.y, a[r][2]);
      a[r][3] = fma_bf16h<1>(wv.y, xv.y, a[r][3]);
    }
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int rr = r < NR ? r : 0;
    v[r] = r < NR ? (a[rr][0] + a[rr][1]) + (a[rr][2] + a[rr][3]) : 0.0f;
  }
}

/* One block of up to 8 rows of one token on the CUDA cores, out of line:
 * the one copy of this loop serves every task type, which keeps the
 * instruction footprint of the kernel small.  Rows are virtual rows n0 ..
 * n0 + nr - 1 mapped to stage rows by identity, or (pairs > 0) as gate row
 * v / 2 for even v and up row pairs + v / 2 for odd v.  Returns this lane's
 * share of the transposing reduction: lane l holds the sum of virtual row
 * n0 + l / 4. */
__device__ __noinline__ float cc_block_sum(uint32_t st, int n0, int nr, int pitch, int K,
                                           uint32_t x, int lane, int pairs) {
  float v[8];
  switch (nr) {
    case 1: cc_block<1>(st, n0, pitch, K, x, lane, pairs, v); break;
    case 2: cc_block<2>(st, n0, pitch, K, x, lane, pairs, v); break;
    case 3: cc_block<3>(st, n0, pitch, K, x, lane, pairs, v); break;
    case 4: cc_block<4>(st, n0, pitch, K, x, lane, pairs, v); break;
    case 5: cc_block<5>(st, n0, pitch, K, x, lane, pairs, v); break;
    case 6: cc_block<6>(st, n0, pitch, K, x, lane, pairs, v); break;
    case 7: cc_block<7>(st, n0, pitch, K, x, lane, pairs, v); break;
    default: cc_block<8>(st, n0, pitch, K, x, lane, pairs, v); break;
  }
  return transpose_reduce8(v, lane);
}

/* One token on the CUDA cores (a tensor-core tile would use 1 of its 16 M
 * rows): the rows of one ring stage (pitch bytes apart) against the bf16
 * activation x, up to eight rows per pass sharing each load of x.  Lane l
 * handles columns 4l + 128i (K a multiple of 64); each product is one fp32
 * FMA on the bf16 operands.  blk(n0, s, nr) runs on every lane with lane l
 * holding the sum of virtual row n0 + l / 4 (valid for l / 4 < nr). */
template <class Blk>
__device__ __forceinline__ void cc_rows(const uint8_t *st, int R, int pitch, int K,
                                        const uint16_t *x, int lane, int pairs, Blk &&blk) {
  const uint32_t sst = saddr(st), sx = saddr(x);
  for (int n0 = 0; n0 < R; n0 += 8) {
    const int nr = min(8, R - n0);
    blk(n0, cc_block_sum(sst, n0, nr, pitch, K, sx, lane, pairs), nr);
  }
}

/* ----------------------------------------------------------- shared layout */

enum { SK_ROWS = 0, SK_PAIRS = 1, SK_PAGES = 2, SK_BOX = 3 };

/* One stage's copies: ROWS n rows of row_bytes at a (one copy); PAIRS n gate
 * rows at a and n up rows at b (two copies); PAGES n pages of one (layer, kv
 * head) (two tensor boxes each); BOX one 2-D tensor-map box of row_bytes
 * bytes, map a, coordinates {pages[0], pages[1]}. */
struct QDesc {
  const uint8_t *a, *b;
  int32_t kind, n;
  uint32_t row_bytes;
  int32_t layer_kvh; /* PAGES: layer << 8 | kvh */
  int32_t pages[MK_MAX_STAGE_PAGES];
};

#define MK_QBATCH 16 /* descriptors a producer warp plans at once */

template <int NB>
struct Misc {
  uint64_t full[NC];
  uint64_t empty[NC];
  /* each producer warp's planned stage descriptors (offset independent of NB) */
  QDesc qd[MK_NP_WARPS][MK_QBATCH];
  /* each producer warp's routing of its current layer: slot -> expert, U */
  int32_t pexp[MK_NP_WARPS][128];
  int32_t pU[MK_NP_WARPS];
  int32_t norm_layer; /* layer whose normed input sits in xbuf (-2: none) */
  int32_t ok;         /* 0 once a consumer stopped early */
  int32_t route_layer; /* layer whose routing the consumers hold (-1: none) */
  int32_t route_U;
  int32_t route_expert[128];        /* slot -> expert id, ascending */
  float route_w[128][NB];           /* weight of slot u for token b (0: not chosen) */
  float red[NC][MK_MAX_BATCH], red_lo[NC][MK_MAX_BATCH];
  float rsum[MK_MAX_BATCH];
  float am[NC / 2][8], al[NC / 2][8]; /* attention warp-merge exchange */
  int32_t tasks[MK_SMEM_TASKS][MK_DESC_INTS]; /* this CTA's task-table row */
  union {
    struct {
      float hres[MK_MAX_OUT_ROWS][NB];          /* the layer input h at the task's rows */
      float acc_o[MK_MAX_OUT_ROWS][NB];         /* Wo rows (one writer each) */
      float acc_w[NC][MK_MAX_OUT_ROWS][NB];     /* per-warp expert-down sums */
    } out;
    struct {
      float best[NC][MK_MAX_BATCH][2];
    } lm;
  } u;
};

/* The kernel's dynamic shared memory.  Pointers into it are always formed
 * from this symbol plus an offset in the function that dereferences them,
 * so that the compiler emits shared-memory (not generic) accesses. */
extern __shared__ __align__(1024) uint8_t mk_smem[];

struct Ctx {
  const mk_kparams *p;
  uint32_t ring_off, xn_off, xbuf_off, misc_off; /* byte offsets into mk_smem */
  uint32_t epoch;
  int cta;
  int SB; /* bytes of one ring slot */
  int NS; /* ring slots: stage i uses slot i % NS and belongs to consumer warp i % NC */
  __device__ __forceinline__ uint8_t *ring() const { return mk_smem + ring_off; }
  __device__ __forceinline__ uint8_t *xbuf() const { return mk_smem + xbuf_off; }
  /* the normed layer input [NB][d] bf16, kept while the layer's QKV, router
   * and expert tasks run (the scratch buffer is reused in between) */
  __device__ __forceinline__ uint16_t *xn() const { return (uint16_t *)(mk_smem + xn_off); }
  /* the mbarriers open the control block: full[NC], then empty[NC] */
  __device__ __forceinline__ uint64_t *full() const { return (uint64_t *)(mk_smem + misc_off); }
  __device__ __forceinline__ uint64_t *empty() const { return full() + NC; }
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

/* Polls the n <= 8 words at a[0], a[stride], ... (all loads of a round in
 * flight at once) until each carries `tag`; payloads to v.  Bounded: false
 * once the wait limit passes (recording MK_ERR_DEVICE_TIMEOUT with `op`,
 * `layer`) or another CTA raised the abort flag. */
__device__ bool poll_tagged(const mk_kparams &p, int cta, const uint64_t *a, int stride, int n,
                            uint32_t tag, uint32_t *v, int op, int layer) {
  uint64_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < n) w[i] = ld_tag(a + (size_t)i * stride);
  uint64_t t0 = 0;
  uint32_t spins = 0;
  while (true) {
    bool all = true;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < n && !tag_ok(w[i], tag)) all = false;
    if (all) break;
    /* the limit and the abort flag every 16 rounds: a global load each
     * round would put a second round trip between the data and its reader */
    if (!t0) {
      t0 = gtimer();
    } else if ((++spins & 15) == 0) {
      if (gtimer() - t0 > p.wait_limit_ns) {
        raise_error(p, MK_ERR_DEVICE_TIMEOUT, cta, -1, op, layer, -1, 0, (int)tag);
        return false;
      }
      if (ld_volatile(&p.ctrl->abort)) return false;
    }
    __nanosleep(32);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < n && !tag_ok(w[i], tag)) w[i] = ld_tag(a + (size_t)i * stride);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < n) v[i] = (uint32_t)w[i];
  return true;
}


/* Waits until (int)(*c - target) >= 0.  Called by all 32 lanes of a warp
 * together: lane 0 polls and broadcasts, and every lane sleeps between
 * polls, so the warp never sits split between a spinning lane and lanes
 * parked at a convergence point (measured on GB300: a lone lane spinning
 * that way saw a completed counter ~15 us after other warps did).  Bounded:
 * gives up after the wait limit (recording MK_ERR_DEVICE_TIMEOUT) or as soon
 * as another CTA raised the abort flag.  Returns false then (on every lane). */
__device__ bool wait_counter_warp(const Ctx &cx, int32_t *c, int target, int task, int op,
                                  int layer, int ctr_kind) {
  const mk_kparams &p = *cx.p;
  const int lane = threadIdx.x & 31;
  int v = lane == 0 ? ld_acquire(c) : 0;
  v = __shfl_sync(0xFFFFFFFFu, v, 0);
  if ((int)(v - target) >= 0) return true;
  const uint64_t t0 = gtimer();
  uint32_t spins = 0;
  while (true) {
    v = lane == 0 ? ld_relaxed(c) : 0;
    v = __shfl_sync(0xFFFFFFFFu, v, 0);
    if ((int)(v - target) >= 0) {
      fence_acquire_gpu();
      return true;
    }
    if ((++spins & 31) == 0) {
      int stop = 0;
      if (lane == 0) {
        if (ld_volatile(&p.ctrl->abort)) {
          stop = 1;
        } else if (gtimer() - t0 > p.wait_limit_ns) {
          raise_error(p, MK_ERR_DEVICE_TIMEOUT, cx.cta, task, op, layer, ctr_kind, v, target);
          stop = 1;
        }
      }
      if (__shfl_sync(0xFFFFFFFFu, stop, 0)) return false;
    }
    __nanosleep(20);
  }
}

/* Waits for an mbarrier phase, suspended in hardware between checks of the
 * abort flag and the time limit.  Bounded like wait_counter. */
__device__ bool wait_mbar(const Ctx &cx, uint64_t *bar, uint32_t parity, int task, int op,
                          int layer) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!mbar_wait_hint(bar, parity, 20000)) {
    if (ld_volatile(&cx.p->ctrl->abort)) return false;
    if (gtimer() - t0 > cx.p->wait_limit_ns) {
      raise_error(*cx.p, MK_ERR_DEVICE_TIMEOUT, cx.cta, task, op, layer, -1, 0, 0);
      return false;
    }
  }
  return true;
}

/* ================================================================ routing
 * Every warp that needs a layer's routing takes it from the router logits
 * itself (the router pieces are spread over the grid and signal one
 * counter), so no CTA computes it for the others and no result has to be
 * published and polled before the expert weights can be fetched.
 *
 * route_warp: the batch's distinct chosen experts for a producer warp that
 * needs them before its CTA's consumers take the routing (a share of
 * expert down rows on a CTA whose consumers are still in attention).  One
 * warp, the NT <= 8 tokens' selections interleaved so
 * that their reduction chains overlap.  Per token: K rounds of a warp argmax
 * over the E <= 128 fp32 logits (lane l holds experts l, l + 32, l + 64,
 * l + 96), ties to the lower expert id -- the same selection as the
 * consumers' rank count.  A round is two single-instruction warp
 * reductions: the largest of the lanes' best keys (an order-preserving
 * unsigned image of the float), then the lowest expert id among the lanes
 * holding it.  Writes expert[slot] (ascending id) and *U; false on timeout
 * or abort while waiting for the logits. */
/* Unsigned keys in the order of the floats (-0 taken as +0, which compares
 * equal to it); 0 marks an expert out of the running. */
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(__fadd_rn(f, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

template <int NT>
__device__ bool route_warp(const mk_kparams &p, int cta, int layer, int lane, int32_t *expert,
                           int32_t *U_out) {
  const int E = p.E, B = p.B, K = p.K;
  const uint64_t *lgt = p.lg_tag + (size_t)layer * MK_MAX_BATCH * E;
  /* the logits as their router pieces write them (tagged words) */
  const int n = max(0, min(4, (E - lane + 31) / 32));
  uint32_t key[NT][4];
  bool ok = true;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    uint32_t v[8];
    if (ok && t < B && n > 0)
      ok = poll_tagged(p, cta, lgt + (size_t)t * E + lane, 32, n, p.step_tag, v, OP_UP, layer);
#pragma unroll
    for (int i = 0; i < 4; ++i) key[t][i] = (ok && t < B && i < n) ? order_key(__uint_as_float(v[i])) : 0u;
  }
  if (!__all_sync(0xFFFFFFFFu, ok)) return false;
  int pick[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) pick[t] = 0;
  for (int k = 0; k < K; ++k) {
    uint32_t best[NT], bi[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      best[t] = key[t][0];
      bi[t] = 0;
#pragma unroll
      for (int i = 1; i < 4; ++i)
        if (key[t][i] > best[t]) {
          best[t] = key[t][i];
          bi[t] = i;
        }
    }
    uint32_t top[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) top[t] = __reduce_max_sync(0xFFFFFFFFu, best[t]);
    uint32_t win[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t)
      win[t] = __reduce_min_sync(0xFFFFFFFFu, (best[t] == top[t] && top[t] != 0u)
                                                  ? bi[t] * 32u + (uint32_t)lane
                                                  : 0xFFFFFFFFu);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (win[t] == 0xFFFFFFFFu) continue; /* no expert left (rows of absent tokens) */
      if (lane == k) pick[t] = (int)win[t];
      if ((int)(win[t] & 31u) == lane) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if ((uint32_t)i == (win[t] >> 5)) key[t][i] = 0u;
      }
    }
  }
  /* the union of the chosen sets */
  uint32_t words[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (lane < K && t < B) words[pick[t] >> 5] |= 1u << (pick[t] & 31);
#pragma unroll
  for (int i = 0; i < 4; ++i) words[i] = __reduce_or_sync(0xFFFFFFFFu, words[i]);
  const int U = __popc(words[0]) + __popc(words[1]) + __popc(words[2]) + __popc(words[3]);
  /* slot of expert e: the chosen experts below it */
  auto rank = [&](int e) {
    int r = __popc(words[e >> 5] & ((1u << (e & 31)) - 1u));
#pragma unroll
    for (int i = 0; i < 3; ++i) r += (i < (e >> 5)) ? __popc(words[i]) : 0;
    return r;
  };
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = lane + 32 * i;
    if ((words[i] >> lane) & 1u) expert[rank(e)] = e;
  }
  if (lane == 0) *U_out = U;
  __syncwarp();
  return true;
}

/* ============================================================== producer
 * One thread (lane 0 of the producer warp) walks the CTA's task list stage
 * by stage and copies stage i into ring slot i % 8 (TMA copies completing
 * on full[slot]) as soon as warp i % 8 has released the slot; eight slots of
 * about 25 KB on each of the 152 SMs keep ~30 MB of copies in flight, more
 * than HBM needs to run at its peak.  The consumers walk the same
 * deterministic stage sequence.
 *
 * Stage contents (one bulk copy per contiguous block, since each copy
 * costs the single producer thread tens of nanoseconds to issue):
 *   ROWS   n whole rows of one matrix, consecutive as in memory (one copy);
 *   PAIRS  the n gate rows, then the n up rows, of the same expert and ffn
 *          indices (two copies);
 *   PAGES  n KV pages of one (sequence, kv head): page j at stage byte
 *          j * 4PD, its K box then its V box (P tokens x D dims, stored as
 *          128-byte rows of 64 dims, swizzled when D >= 64; two copies). */


/* Producer warp k of MK_NP_WARPS.  The stage sequence is fixed by the task
 * list (and, for the expert stages, by the layer's routing); stage i goes to
 * ring slot i % 8 and is filled by warp i % MK_NP_WARPS, so each slot has
 * one producer.  Per task, the warp's lanes compute the descriptors of the
 * warp's own stages in parallel from closed forms (rows, pages, expert
 * segments), then lane 0 issues them in order, each as soon as its slot is
 * free.  Issuing a copy costs the issuing thread tens of nanoseconds, which
 * is why there are several producer warps; planning in parallel keeps the
 * issuing thread free of everything else. */
template <int NB>
struct Producer {
  Ctx cx;
  uint64_t policy;
  int k, lane;
  QDesc *buf; /* this warp's MK_QBATCH planned descriptors (shared memory) */
  int32_t *pexp; /* this warp's slot -> expert list (shared memory) */
  int32_t *pU;
  /* the consumers' routing in shared memory: its layer, U, slot -> expert */
  const int32_t *c_layer, *c_U, *c_expert;
  int r_layer;   /* layer of the routing in pexp (-1: none) */
  uint64_t t_task, t_plan; /* stage trace: the current task's start, its plan ready */
  int last_slot[NC];
  unsigned long long *strc;

  /* The layer's routing for this warp's expert stages.  For a gate/up
   * share (from_consumers) it is the consumers' routing of the layer, which
   * consumer thread 0 publishes in shared memory as soon as the consumers
   * have taken it (they start the share right after the CTA's QKV task); it
   * stays valid while a producer warp copies it, as the consumers cannot
   * leave the share before every producer warp has issued its stages of it.
   * For a share of expert down rows (whose consumers take the routing only
   * after their attention splits) the warp takes the top-k itself from the
   * tagged logits.  Returns U, or -1 on timeout / abort. */
  __device__ int routed(int layer, bool from_consumers) {
    const mk_kparams &p = *cx.p;
    if (r_layer == layer) return *(volatile int32_t *)pU;
    if (from_consumers) {
      const uint64_t t0 = gtimer();
      uint32_t spins = 0;
      while (true) {
        const int seen = lane == 0 ? ld_acquire_cta(c_layer) == layer : 0;
        if (__shfl_sync(0xFFFFFFFFu, seen, 0)) break;
        if ((++spins & 31) == 0) {
          int stop = 0;
          if (lane == 0) {
            if (ld_volatile(&p.ctrl->abort)) {
              stop = 1;
            } else if (gtimer() - t0 > p.wait_limit_ns) {
              raise_error(p, MK_ERR_DEVICE_TIMEOUT, cx.cta, -1, OP_UP, layer, CTR_ROUTER_DONE,
                          -1, layer);
              stop = 1;
            }
          }
          if (__shfl_sync(0xFFFFFFFFu, stop, 0)) return -1;
        }
        __nanosleep(20);
      }
      const int U = *(volatile const int32_t *)c_U;
      for (int i = lane; i < U; i += 32) pexp[i] = c_expert[i];
      if (lane == 0) *pU = U;
      __syncwarp();
    } else if (!route_warp<NB>(p, cx.cta, layer, lane, pexp, pU)) {
      return -1;
    }
    r_layer = layer;
    return *(volatile int32_t *)pU;
  }

  /* issues one planned stage (lane 0); false on a failed wait */
  __device__ bool issue(const QDesc &d, int i) {
    const mk_kparams &p = *cx.p;
    const uint64_t ta = strc ? sclock() : 0;
    const int NS = cx.NS, slot = i % NS;
    if (i >= NS && !wait_mbar(cx, &cx.empty()[slot], (uint32_t)(((i / NS) - 1) & 1), -1, -1, -1))
      return false;
    const uint64_t tb = strc ? sclock() : 0;
    uint8_t *dst = cx.ring() + (size_t)slot * cx.SB;
    uint64_t *bar = &cx.full()[slot];
    if (d.kind == SK_ROWS || d.kind == SK_PAIRS) {
      /* two runs, the second mk_run_gap bytes past the first (one copy for
       * plain rows where the gap is 0) */
      const int nr = d.kind == SK_PAIRS ? 2 * d.n : d.n;
      const uint32_t rb = d.row_bytes;
      mbar_expect_tx(bar, (uint32_t)nr * rb);
      if (d.kind == SK_PAIRS) {
        bulk_g2s(dst, d.a, d.n * rb, bar, policy);
        bulk_g2s(dst + d.n * rb + mk_run_gap(NB), d.b, d.n * rb, bar, policy);
      } else if (mk_run_gap(NB) == 0) {
        bulk_g2s(dst, d.a, d.n * rb, bar, policy);
      } else {
        const uint32_t h = (uint32_t)(d.n + 1) / 2;
        bulk_g2s(dst, d.a, h * rb, bar, policy);
        if ((uint32_t)d.n > h)
          bulk_g2s(dst + h * rb + mk_run_gap(NB), d.a + (size_t)h * rb, (d.n - h) * rb, bar, policy);
      }
    } else if (d.kind == SK_BOX) {
      mbar_expect_tx(bar, d.row_bytes);
      tensor_g2s_2d(dst, d.a, d.pages[0], d.pages[1], bar, policy);
    } else {
      const int P = p.P, layer = d.layer_kvh >> 8, kvh = d.layer_kvh & 0xFF;
      const uint32_t half = (uint32_t)P * p.D * 2, pgb = 2 * half;
      const uint8_t *kmap = (const uint8_t *)p.kv_maps + (size_t)layer * 2 * 128;
      const uint8_t *vmap = kmap + 128;
      mbar_expect_tx(bar, d.n * pgb);
      for (int j = 0; j < d.n; ++j) {
        const int y = (d.pages[j] * p.Hkv + kvh) * P;
        tensor_g2s_3d(dst + j * pgb, kmap, y, bar, policy);
        tensor_g2s_3d(dst + j * pgb + half, vmap, y, bar, policy);
      }
    }
    last_slot[slot] = i;
    if (strc && i < MK_STAGE_TRACE_EVENTS - 1) {
      unsigned long long *e = strc + (size_t)i * 8;
      e[1] = t_task ? t_task : ta;
      e[2] = t_plan ? t_plan : ta;
      e[3] = tb;
      e[4] = sclock();
    }
    return true;
  }

  /* Plans and issues this warp's stages among stages [j_lo, j_hi) of a task
   * whose first stage is stream stage `base`; plan(j, d) fills stage j's
   * descriptor (called on the planning lanes). */
  template <class Plan>
  __device__ bool run_stages(int base, int j_lo, int j_hi, Plan &&plan) {
    int j0 = j_lo + ((k - (base + j_lo) % MK_NP_WARPS) % MK_NP_WARPS + MK_NP_WARPS) % MK_NP_WARPS;
    for (; j0 < j_hi; j0 += MK_QBATCH * MK_NP_WARPS) {
      const int j = j0 + lane * MK_NP_WARPS;
      if (lane < MK_QBATCH && j < j_hi) plan(j, buf[lane]);
      __syncwarp();
      int ok = 1;
      if (lane == 0)
        for (int l = 0; l < MK_QBATCH; ++l) {
          const int jj = j0 + l * MK_NP_WARPS;
          if (jj >= j_hi) break;
          if (!issue(buf[l], base + jj)) {
            ok = 0;
            break;
          }
        }
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) return false;
    }
    return true;
  }

  __device__ __forceinline__ void run(const int32_t *row) {
    const Ctx c = cx;
    const mk_kparams &p = *c.p;
    for (int s = 0; s < NC; ++s) last_slot[s] = -1;
    const int nl = row[1], nf = row[2], SB = c.SB;
    const int d = p.d, F = p.F, HqD = p.Hq * p.D, P = p.P;
    int base = 0;
    bool ok = true;
    /* the layer's weight pointers, loaded one layer ahead (a dependent L2
     * round trip before the first stage of every task otherwise); the final
     * tasks keep the last layer's */
    mk_layer_dev cur = p.layers[0], nxt = p.layers[p.L > 1 ? 1 : 0];
    for (int layer = 0; layer <= p.L && ok; ++layer) {
      const int ntask = layer < p.L ? nl : nf;
      if (layer > 0 && layer < p.L) {
        cur = nxt;
        nxt = p.layers[min(layer + 1, p.L - 1)];
      }
      if (k == 0 && lane == 0 && layer + 1 < p.L) {
        /* the next layer's tensor maps into the descriptor cache */
        const uint8_t *kmap = (const uint8_t *)p.kv_maps + (size_t)(layer + 1) * 2 * 128;
        prefetch_tensormap(kmap);
        prefetch_tensormap(kmap + 128);
        if (NB == 1 && p.fold) prefetch_tensormap((const uint8_t *)p.wd_maps + (size_t)(layer + 1) * 128);
      }
      for (int kt = 0; kt < ntask && ok; ++kt) {
        const int32_t *t = row + MK_DESC_INTS * (1 + (layer < p.L ? kt : nl + kt));
        const mk_layer_dev *ly = &cur;
        const int op = t[0];
        t_task = strc ? sclock() : 0;
        t_plan = 0;
        if (op == OP_QKV || op == OP_LM) {
          /* QKV: the router rows first, then the q / k / v rows */
          const uint16_t *w = op == OP_LM ? p.lm_head
                              : t[1] == 0 ? ly->wq
                              : t[1] == 1 ? ly->wk
                                          : ly->wv;
          const uint16_t *src = w + (size_t)t[2] * d;
          const int nrows = t[3], rps = mk_rows_per_stage(d, SB, NB);
          const int rn = op == OP_QKV ? t[5] : 0;
          const uint16_t *rsrc = ly->wr + (size_t)(op == OP_QKV ? t[4] : 0) * d;
          const int n_rst = (rn + rps - 1) / rps, n_st = n_rst + (nrows + rps - 1) / rps;
          ok = run_stages(base, 0, n_st, [&](int j, QDesc &q) {
            q.kind = SK_ROWS;
            if (j < n_rst) {
              q.n = min(rps, rn - j * rps);
              q.a = (const uint8_t *)(rsrc + (size_t)j * rps * d);
            } else {
              q.n = min(rps, nrows - (j - n_rst) * rps);
              q.a = (const uint8_t *)(src + (size_t)(j - n_rst) * rps * d);
            }
            q.row_bytes = (uint32_t)d * 2;
          });
          base += n_st;
        } else if (op == OP_ATTN) {
          const int b = t[1], kvh = t[2], p0 = t[3];
          const int p1 = t[4] >= 0 ? t[4] : (__ldg(p.seq_lens + b) + P - 1) / P;
          const int pps = mk_pages_per_stage(P, p.D, SB);
          const int n_st = (p1 - p0 + pps - 1) / pps;
          ok = run_stages(base, 0, n_st, [&](int j, QDesc &q) {
            const int q0 = p0 + j * pps, cnt = min(pps, p1 - q0);
            q.kind = SK_PAGES;
            q.n = cnt;
            q.layer_kvh = (layer << 8) | kvh;
            for (int jj = 0; jj < cnt; ++jj) q.pages[jj] = __ldg(p.page_table + b * p.max_pages + q0 + jj);
          });
          base += n_st;
        } else if (op == OP_UP && NB == 1 && p.fold) {
          /* a range of 64-column blocks of the chosen experts' F: every
           * block's 64 gate rows and 64 up rows, then its down boxes (the
           * block's 64 columns of fold_rows rows of d each) */
          const int U = routed(layer, true);
          if (U < 0) {
            ok = false;
            break;
          }
          t_plan = strc ? sclock() : 0;
          const int nbf = F / MK_FOLD_COLS, T64 = U * nbf;
          const int b0 = (int)((int64_t)T64 * t[1] / t[2]);
          const int b1 = (int)((int64_t)T64 * (t[1] + 1) / t[2]);
          const int rps = mk_rows_per_stage(d, SB, NB), ng = (MK_FOLD_COLS + rps - 1) / rps;
          const int BR = p.fold_rows, nrb = d / BR;
          const int nA = (b1 - b0) * 2 * ng, nB = (b1 - b0) * nrb;
          ok = run_stages(base, 0, nA + nB, [&](int j, QDesc &q) {
            if (j < nA) {
              const int blk = b0 + j / (2 * ng), jj = j % (2 * ng);
              const int up = jj >= ng, c = up ? jj - ng : jj;
              const int f0 = (blk % nbf) * MK_FOLD_COLS + c * rps;
              q.kind = SK_ROWS;
              q.n = min(rps, MK_FOLD_COLS - c * rps);
              q.a = (const uint8_t *)((up ? ly->wu : ly->wg) + ((size_t)pexp[blk / nbf] * F + f0) * d);
              q.row_bytes = (uint32_t)d * 2;
            } else {
              const int jb = j - nA, blk = b0 + jb / nrb, rb = jb % nrb;
              q.kind = SK_BOX;
              q.n = 1;
              q.a = (const uint8_t *)p.wd_maps + (size_t)layer * 128;
              q.pages[0] = (blk % nbf) * MK_FOLD_COLS;
              q.pages[1] = pexp[blk / nbf] * d + rb * BR;
              q.row_bytes = (uint32_t)(MK_FOLD_COLS * BR * 2);
            }
          });
          base += nA + nB;
        } else if (op == OP_UP) {
          const int U = routed(layer, true);
          if (U < 0) {
            ok = false;
            break;
          }
          t_plan = strc ? sclock() : 0;
          const int pps = mk_pairs_per_stage(d, SB, NB);
          const int64_t T = (int64_t)U * F;
          const int64_t v = T * t[1] / t[2], v1 = T * (t[1] + 1) / t[2];
          /* stages per expert segment, as the consumers walk them */
          const int u0 = (int)(v / F), u1 = v1 > v ? (int)((v1 - 1) / F) : u0 - 1;
          int n_st = 0;
          for (int u = u0; u <= u1; ++u) {
            const int64_t lo = max(v, (int64_t)u * F), hi = min(v1, (int64_t)(u + 1) * F);
            n_st += (int)((hi - lo + pps - 1) / pps);
          }
          ok = run_stages(base, 0, n_st, [&](int j, QDesc &q) {
            int u = u0, jr = j;
            int64_t lo = 0, hi = 0;
            for (; u <= u1; ++u) {
              lo = max(v, (int64_t)u * F);
              hi = min(v1, (int64_t)(u + 1) * F);
              const int ns = (int)((hi - lo + pps - 1) / pps);
              if (jr < ns) break;
              jr -= ns;
            }
            const int f0 = (int)(lo - (int64_t)u * F) + jr * pps;
            const int cnt = min(pps, (int)(hi - (int64_t)u * F) - f0);
            const int e = pexp[u];
            const size_t eo = ((size_t)e * F + f0) * d;
            q.kind = SK_PAIRS;
            q.n = cnt;
            q.a = (const uint8_t *)(ly->wg + eo);
            q.b = (const uint8_t *)(ly->wu + eo);
            q.row_bytes = (uint32_t)d * 2;
          });
          base += n_st;
        } else if (op == OP_DOWN) {
          /* a range of the chosen experts' down rows (U x d of them, slot
           * order), per expert segment in stages of whole rows of F; the
           * routing is taken here if the CTA had no gate/up share, so that
           * the rows stream while its consumers still run attention */
          const int U = routed(layer, false);
          if (U < 0) {
            ok = false;
            break;
          }
          t_plan = strc ? sclock() : 0;
          const int rps = mk_rows_per_stage(F, SB, NB);
          const int64_t T = (int64_t)U * d;
          const int64_t v = T * t[1] / t[2], v1 = T * (t[1] + 1) / t[2];
          const int u0 = (int)(v / d), u1 = v1 > v ? (int)((v1 - 1) / d) : u0 - 1;
          int n_st = 0;
          for (int u = u0; u <= u1; ++u) {
            const int64_t lo = max(v, (int64_t)u * d), hi = min(v1, (int64_t)(u + 1) * d);
            n_st += (int)((hi - lo + rps - 1) / rps);
          }
          ok = run_stages(base, 0, n_st, [&](int j, QDesc &q) {
            int u = u0, jr = j;
            int64_t lo = 0, hi = 0;
            for (; u <= u1; ++u) {
              lo = max(v, (int64_t)u * d);
              hi = min(v1, (int64_t)(u + 1) * d);
              const int ns = (int)((hi - lo + rps - 1) / rps);
              if (jr < ns) break;
              jr -= ns;
            }
            const int r0 = (int)(lo - (int64_t)u * d) + jr * rps;
            q.kind = SK_ROWS;
            q.n = min(rps, (int)(hi - (int64_t)u * d) - r0);
            q.a = (const uint8_t *)(ly->wd + ((size_t)pexp[u] * d + r0) * F);
            q.row_bytes = (uint32_t)F * 2;
          });
          base += n_st;
        } else if (op == OP_OUT) {
          /* the Wo rows (the experts' down rows are DOWN tasks, or folded
           * into the gate/up shares at batch 1) */
          const int r0 = t[2], nr = t[3];
          t_plan = strc ? sclock() : 0;
          const int rps_o = mk_rows_per_stage(HqD, SB, NB), n_wo = (nr + rps_o - 1) / rps_o;
          const uint16_t *wo = ly->wo + (size_t)r0 * HqD;
          ok = run_stages(base, 0, n_wo, [&](int jw, QDesc &q) {
            q.kind = SK_ROWS;
            q.n = min(rps_o, nr - jw * rps_o);
            q.a = (const uint8_t *)(wo + (size_t)jw * rps_o * HqD);
            q.row_bytes = (uint32_t)HqD * 2;
          });
          base += n_wo;
        } else {
          ok = false; /* the consumers report the bad opcode */
        }
      }
    }
    /* Every copy issued must land before the CTA exits (normally the
     * consumers have waited for all of them already). */
    if (lane == 0)
      for (int s = 0; s < c.NS; ++s) {
        const int kk = last_slot[s];
        if (kk < 0) continue;
        const uint32_t parity = (uint32_t)((kk / c.NS) & 1);
        const uint64_t t0 = gtimer();
        while (!mbar_test(&c.full()[s], parity) && gtimer() - t0 < p.wait_limit_ns) {
        }
      }
    __syncwarp();
  }
};

/* A producer warp's whole life, out of line so that its registers are
 * allocated apart from the consumers', with its state passed by value. */
template <int NB>
__device__ __noinline__ void produce(const Ctx cx, int k, int lane, QDesc *buf, int32_t *pexp,
                                     int32_t *pU, unsigned long long *strc,
                                     const int32_t *row) {
  Producer<NB> pr;
  pr.cx = cx;
  pr.policy = evict_first_policy();
  pr.k = k;
  pr.lane = lane;
  pr.buf = buf;
  pr.pexp = pexp;
  pr.pU = pU;
  {
    const Misc<NB> *m = (const Misc<NB> *)(mk_smem + cx.misc_off);
    pr.c_layer = &m->route_layer;
    pr.c_U = &m->route_U;
    pr.c_expert = m->route_expert;
  }
  pr.r_layer = -1;
  pr.t_task = pr.t_plan = 0;
  pr.strc = strc;
  pr.run(row);
}

/* ============================================================== consumers
 * Eight warps.  Stage i of the CTA's stream belongs to warp i % 8 alone:
 * its lane 0 polls the stage's mbarrier, the warp computes every row (or
 * key) of the stage, and lane 0 releases the slot.  Outputs are written by
 * the warp that owns their stage, so each has one writer.  A failed wait
 * (time limit or abort) marks the warp; the consumers decide together at the
 * next collective point (a barrier with an OR reduction), so all consumer
 * threads always leave at the same point and no barrier is ever left
 * half-arrived. */

template <int NB>
struct Consumer {
  Ctx cx;
  int warp, lane, tid;
  int si;     /* stages of the stream before the current task (all warps agree) */
  bool wfail; /* this warp failed a stage wait */
  unsigned long long *tr; /* this CTA's trace events, or NULL */
  int tr_n;
  uint64_t t_ready, t_stage, t_swait, t_mark;
  int n_stages;

  __device__ __forceinline__ Misc<NB> *M() const { return (Misc<NB> *)(mk_smem + cx.misc_off); }

  /* Warp 0 waits on a counter; every consumer learns whether the CTA goes
   * on (false also when any warp has failed a stage wait). */
  __device__ bool cwait(int32_t *c, int target, int task, int op, int layer, int kind) {
    bool fail = wfail;
    if (warp == 0) {
      fail |= !wait_counter_warp(cx, c, target, task, op, layer, kind);
      if (tr && tid == 0 && !t_ready) t_ready = gtimer();
    }
    return !bar_any(fail);
  }

  /* End of a task's streaming part: a consumer barrier, false if any warp
   * failed. */
  __device__ bool task_end() { return !bar_any(wfail); }

  /* The first stage index j >= 0 of a task (stream stage si + j) that this
   * warp owns. */
  __device__ int first_mine() const { return (warp - si % NC + NC) % NC; }
  /* the same for a run of stages that starts at stream stage s */
  __device__ int first_mine_at(int s) const { return (warp - s % NC + NC) % NC; }

  /* Every lane of the warp waits for the stage itself, and the stage
   * bookkeeping below is branch-free (predicated single stores and
   * arrives): a wait or a multi-instruction region run by one lane alone
   * leaves the warp split, and a split warp runs the stage's compute once
   * per lane group. */
  __device__ bool stage_wait(int i, uint8_t *&st, int task, int op, int layer) {
    if (wfail) return false;
    const int slot = i % cx.NS;
    const uint32_t parity = (uint32_t)((i / cx.NS) & 1);
    const bool trace = tr && warp == 0;
    const bool sev = tr && cx.cta == cx.p->stage_trace_cta && i < MK_STAGE_TRACE_EVENTS - 1;
    const uint64_t w0 = trace ? gtimer() : 0, c0 = sev ? sclock() : 0;
    const bool ok = wait_mbar(cx, &cx.full()[slot], parity, task, op, layer);
    if (trace) {
      const uint64_t w1 = gtimer();
      if (!t_stage) t_stage = w1;
      else t_swait += w1 - w0;
      ++n_stages;
    }
    if (sev) {
      unsigned long long *se = cx.p->stage_trace + (size_t)i * 8;
      st64_if(se, (unsigned long long)(i | (warp << 20) | (op << 24)), lane == 0);
      st64_if(se + 5, c0, lane == 0);
      st64_if(se + 6, sclock(), lane == 0);
    }
    if (!__all_sync(0xFFFFFFFFu, ok)) {
      wfail = true;
      return false;
    }
    st = cx.ring() + (size_t)slot * cx.SB;
    return true;
  }

  __device__ void stage_release(int i) {
    __syncwarp(); /* every lane's reads of the slot precede the release */
    mbar_arrive_if(&cx.empty()[i % cx.NS], lane == 0);
    if (tr && cx.cta == cx.p->stage_trace_cta && i < MK_STAGE_TRACE_EVENTS - 1)
      st64_if(cx.p->stage_trace + (size_t)i * 8 + 7, sclock(), lane == 0);
  }

  __device__ const uint16_t *h_row(int layer, int b) const {
    const mk_kparams &p = *cx.p;
    if (layer == 0) {
      /* a token id outside the vocabulary fails the step (sticky) and reads
       * row 0 instead, so nothing outside the embedding table is touched */
      int tok = __ldg(p.tokens + b);
      if ((unsigned)tok >= (unsigned)p.V) {
        raise_error(p, MK_ERR_BAD_TOKEN, cx.cta, -1, -1, 0, b, tok, p.V);
        tok = 0;
      }
      return p.embed + (size_t)tok * p.d;
    }
    return p.h + ((size_t)layer * MK_MAX_BATCH + b) * p.d;
  }

  /* The block-wide sum of every thread's (hi, lo) pair per token, exact up
   * to the pairs' own rounding; v[b] = the sum rounded once to fp32. */
  __device__ void block_sum_pair(float (&hi)[NB], float (&lo)[NB], float (&v)[NB]) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float h = hi[b], l = lo[b];
#pragma unroll
      for (int k = 16; k >= 1; k >>= 1)
        pair_merge(h, l, __shfl_xor_sync(0xFFFFFFFFu, h, k), __shfl_xor_sync(0xFFFFFFFFu, l, k));
      if (lane == 0) {
        M()->red[warp][b] = h;
        M()->red_lo[warp][b] = l;
      }
    }
    bar_consumers();
    if (tid < NB) {
      float h = 0.0f, l = 0.0f;
      for (int w = 0; w < NC; ++w) pair_merge(h, l, M()->red[w][tid], M()->red_lo[w][tid]);
      M()->rsum[tid] = __fadd_rn(h, l);
    }
    bar_consumers();
#pragma unroll
    for (int b = 0; b < NB; ++b) v[b] = M()->rsum[b];
    bar_consumers();
  }

  /* xn[b][0..d) = bf16((h * (1/sqrtf(mean_fp32(h^2) + eps))) * g); rows
   * b >= B zero.  h is read once with 16-byte loads and staged in the
   * scratch buffer.  The sum of squares is carried as an unevaluated pair of
   * floats (each square of a bf16 value is exact in fp32, and TwoSum keeps
   * every addition's error), so the fp32 mean is the exact sum rounded once:
   * the same fp32 value in any summation order, hence the same normed input
   * as any other evaluation that rounds the exact mean once. */
  __device__ bool norm_into_xbuf(int src, const uint16_t *g) {
    const mk_kparams &p = *cx.p;
    const int xp = mk_x_pitch(p.d, NB), B = p.B;
    uint16_t *x = cx.xn();
    uint16_t *raw = (uint16_t *)cx.xbuf();
    const int n8 = p.d / 8, dw = p.d / 2;
    float ss[NB], sh[NB], sl[NB];
    bool fail = false;
    /* every load of the first pass (all tokens' h and this thread's first
     * piece of the gain) is issued before any is used: one round trip */
    const uint4 g_first = tid < n8 ? __ldg((const uint4 *)g + tid) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int b = 0; b < NB; ++b) sh[b] = sl[b] = 0.0f;
    for (int i = tid; i < n8; i += NCT) {
      uint4 v[NB];
      if (src == 0) {
#pragma unroll
        for (int b = 0; b < NB; ++b)
          v[b] = b < B ? __ldcg((const uint4 *)h_row(0, b) + i) : make_uint4(0, 0, 0, 0);
      } else {
        /* the residual as the OUT tasks write it: 4 tagged words (8 values)
         * per token, polled until every word carries this step's tag */
        const uint64_t *hw = p.h_tag + (size_t)src * MK_MAX_BATCH * dw + 4 * i;
        uint64_t w[NB][4];
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int k = 0; k < 4; ++k) w[b][k] = b < B ? ld_tag(hw + (size_t)b * dw + k) : 0ULL;
        uint64_t t0 = 0;
        uint32_t spins = 0;
        while (!fail) {
          bool all = true;
#pragma unroll
          for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (b < B && !tag_ok(w[b][k], p.step_tag)) all = false;
          if (all) break;
          if (!t0) {
            t0 = gtimer();
          } else if ((++spins & 15) == 0) { /* as in poll_tagged */
            if (gtimer() - t0 > p.wait_limit_ns) {
              raise_error(p, MK_ERR_DEVICE_TIMEOUT, cx.cta, -1, OP_QKV, src, -1, 0,
                          (int)p.step_tag);
              fail = true;
            } else if (ld_volatile(&p.ctrl->abort)) {
              fail = true;
            }
          }
          __nanosleep(32);
#pragma unroll
          for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (b < B && !tag_ok(w[b][k], p.step_tag)) w[b][k] = ld_tag(hw + (size_t)b * dw + k);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b)
          v[b] = b < B ? make_uint4((uint32_t)w[b][0], (uint32_t)w[b][1], (uint32_t)w[b][2],
                                    (uint32_t)w[b][3])
                       : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        *(uint4 *)(raw + (size_t)b * p.d + 8 * i) = v[b];
        float f[8];
        unpack8(v[b], f);
#pragma unroll
        for (int k = 0; k < 8; ++k) pair_add(sh[b], sl[b], __fmul_rn(f[k], f[k]));
      }
    }
    block_sum_pair(sh, sl, ss);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float r = 1.0f / sqrtf(ss[b] / (float)p.d + p.eps);
      for (int i = tid; i < n8; i += NCT) {
        uint16_t o[8];
        if (b < B) {
          float hf[8], gf[8];
          unpack8(*(const uint4 *)(raw + (size_t)b * p.d + 8 * i), hf);
          unpack8(i == tid ? g_first : __ldg((const uint4 *)g + i), gf);
#pragma unroll
          for (int k = 0; k < 8; ++k) o[k] = f2bf(__fmul_rn(__fmul_rn(hf[k], r), gf[k]));
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) o[k] = 0;
        }
        *(uint4 *)(x + (size_t)b * xp + 8 * i) =
            make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]),
                       pack_bf16(o[6], o[7]));
      }
    }
    if (tid == 0) M()->norm_layer = src;
    return !bar_any(fail);
  }

  /* The normed input of `layer` in xn (computed unless it is there already);
   * false on timeout / abort. */
  __device__ bool ensure_norm(int layer) {
    if (*(volatile int32_t *)&M()->norm_layer == layer) return true;
    bar_consumers(); /* everyone has read the tag before it can change */
    const bool ok = norm_into_xbuf(layer, lnorm(*cx.p, layer));
    if (tr && tid == 0) t_mark = gtimer();
    return ok;
  }

  /* Copies NB vectors of n bf16 (global, row stride gstride) into dst at
   * the activation pitch mk_x_pitch(n); rows b >= B zero.  No barrier. */
  __device__ void load_x(uint16_t *dst, const uint16_t *src, size_t gstride, int n) {
    const int xp = mk_x_pitch(n, NB), n8 = n / 8, B = cx.p->B;
    for (int i = tid; i < NB * n8; i += NCT) {
      const int b = i / n8, c = i % n8;
      const uint4 v = b < B ? __ldcg((const uint4 *)(src + (size_t)b * gstride) + c)
                            : make_uint4(0, 0, 0, 0);
      *(uint4 *)(dst + (size_t)b * xp + 8 * c) = v;
    }
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

  /* The cnt rows of one ring stage (K elements each) against the
   * activations x (pitch mk_x_pitch(K)); row r of the stage handed to
   * epi(r, b, value). */
  template <class Epi>
  __device__ __forceinline__ void gemv_stage(const uint8_t *st, int cnt, int K, const uint16_t *x,
                                             Epi &&epi) {
    if (NB == 1 && kB1CudaCores) {
      cc_rows(st, cnt, 2 * K, K, x, lane, 0,
              [&](int n0, float sum, int nr) {
                if ((lane & 3) == 0 && (lane >> 2) < nr) epi(n0 + (lane >> 2), 0, sum);
              });
    } else {
      /* virtual row 2i is row i of the first run, 2i + 1 row h + i */
      const int rb = 2 * K, h = (cnt + 1) >> 1, hb = h * rb + mk_run_gap(NB);
      auto f = [&](int v, int bb, float val) { epi((v & 1) ? h + (v >> 1) : (v >> 1), bb, val); };
      mma_rows<NB>(st, cnt, K, x, mk_x_pitch(K, NB), lane,
                   [=](int v) { return (v & 1) ? hb + (v >> 1) * rb : (v >> 1) * rb; },
                   [&](int n0, const float(&a)[4], const float(&b)[4], bool two) {
                     take_out<NB>(n0, a, cnt, lane, f);
                     if (two) take_out<NB>(n0 + 8, b, cnt, lane, f);
                   });
    }
  }

  /* nrows streamed rows of K elements against the activations x; each
   * stage is computed by the warp that owns it and row r (index within the
   * task) handed to epi(r, b, value). */
  template <class Epi>
  __device__ void gemv_rows(int nrows, int K, const uint16_t *x, int task, int op, int layer,
                            Epi &&epi) {
    const int rps = mk_rows_per_stage(K, cx.SB, NB);
    const int n_st = (nrows + rps - 1) / rps;
    for (int j = first_mine(); j < n_st; j += NC) {
      uint8_t *st;
      if (!stage_wait(si + j, st, task, op, layer)) break;
      const int r0 = j * rps, cnt = min(rps, nrows - r0);
      gemv_stage(st, cnt, K, x, [&](int r, int bb, float v) { epi(r0 + r, bb, v); });
      stage_release(si + j);
    }
    si += n_st;
  }

  /* ---------------------------------------------------------------- QKV
   * The CTA's router rows (if any) stream first: the warp that computes a
   * router stage writes its fp32 logits (+ bias) and at once adds its rows
   * to the layer's router counter (E per step), so the routing every expert
   * stage waits for does not wait for the q / k / v rows.  Then the q, k or v
   * rows (bf16 outputs). */
  __device__ bool op_qkv(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    /* the layer's input: the previous layer's OUT tasks' tagged residual */
    if (!ensure_norm(layer)) return false;
    const int QKVD = (p.Hq + 2 * p.Hkv) * p.D;
    const int base = (t[1] == 0 ? 0 : t[1] == 1 ? p.Hq * p.D : (p.Hq + p.Hkv) * p.D) + t[2];
    uint16_t *out = p.qkv + (size_t)layer * MK_MAX_BATCH * QKVD;
    const int B = p.B, E = p.E, d = p.d, e0 = t[4], rn = t[5], nrows = t[3];
    float *lg = p.router_logits + (size_t)layer * MK_MAX_BATCH * E;
    uint64_t *lgt = p.lg_tag + (size_t)layer * MK_MAX_BATCH * E;
    const float *bias = layer < MK_PARAM_LAYERS ? p.l_bias[layer] : p.layers[layer].bias;
    const int rps = mk_rows_per_stage(d, cx.SB, NB);
    const int n_rst = (rn + rps - 1) / rps, n_st = n_rst + (nrows + rps - 1) / rps;
    const uint16_t *x = cx.xn();
    for (int j = first_mine(); j < n_st; j += NC) {
      uint8_t *st;
      if (!stage_wait(si + j, st, task, OP_QKV, layer)) break;
      if (j < n_rst) {
        const int r0 = j * rps, cnt = min(rps, rn - r0);
        gemv_stage(st, cnt, d, x, [&](int r, int b, float v) {
          const int e = e0 + r0 + r;
          if (b < B) {
            const float l = bias ? v + __ldg(bias + e) : v;
            lg[(size_t)b * E + e] = l; /* for the diagnostics */
            st_tag(lgt + (size_t)b * E + e, __float_as_uint(l), p.step_tag);
          }
        });
        stage_release(si + j);
      } else {
        const int r0 = (j - n_rst) * rps, cnt = min(rps, nrows - r0);
        gemv_stage(st, cnt, d, x, [&](int r, int b, float v) {
          if (b < B) out[(size_t)b * QKVD + base + r0 + r] = f2bf(v);
        });
        stage_release(si + j);
      }
    }
    si += n_st;
    if (!task_end()) return false;
    signal(lctr(p, layer, CTR_QKV_DONE));
    return true;
  }

  /* The layer's routing from the router logits, taken by all consumer
   * threads at once: each (token, expert) pair counts the token's logits
   * that rank above it (larger, or equal with a lower id), so the pairs of
   * rank < k are the token's choices in descending order -- the same
   * selection as k rounds of argmax with ties to the lower id.  The weights
   * are the softmax over the chosen logits (warp t for token t); the batch's
   * distinct experts get the slots in ascending id.  Writes route_expert,
   * route_U and route_w, and the diagnostics record when publish is set.
   * Uses the scratch buffer; ends with a consumer barrier. */
  __device__ bool route_block(int layer, mk_routing *publish) {
    const mk_kparams &p = *cx.p;
    Misc<NB> *m = M();
    const int E = p.E, B = p.B, K = p.K, E4 = (E + 3) & ~3;
    const uint64_t *lgt = p.lg_tag + (size_t)layer * MK_MAX_BATCH * E;
    uint32_t *key = (uint32_t *)cx.xbuf();                  /* [NB][128] */
    int32_t *pick = (int32_t *)(key + NB * 128);             /* [NB][MK_MAX_TOPK] */
    uint32_t *flag = (uint32_t *)(pick + NB * MK_MAX_TOPK);  /* [128]: chosen by a token */
    /* the logits as their router pieces write them: thread i polls the
     * words (t, e) = i, i + 256, ... (all in flight at once) */
    static_assert(NB * 128 <= 4 * NCT, "four logit words per thread at most");
    bool fail = false;
    {
      const int t0 = tid >> 7, e = tid & 127, n = (B - t0 + 1) / 2;
      uint32_t v[8];
      if (e < E && n > 0)
        fail = !poll_tagged(p, cx.cta, lgt + (size_t)t0 * E + e, 2 * E, n, p.step_tag, v, OP_UP,
                            layer);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = t0 + 2 * k;
        if (t < NB) key[t * 128 + e] = (!fail && k < n && e < E) ? order_key(__uint_as_float(v[k])) : 0u;
      }
    }
    for (int i = tid; i < 128; i += NCT) flag[i] = 0u;
    if (bar_any(fail)) return false;
    for (int i = tid; i < NB * 128; i += NCT) {
      const int t = i >> 7, e = i & 127;
      if (t >= B || e >= E) continue;
      const uint32_t ke = key[i];
      const uint32_t *kt = key + t * 128;
      int r = 0;
      for (int j = 0; j < E4; j += 4) {
        const uint4 q = *(const uint4 *)(kt + j);
        r += (q.x > ke) + (q.y > ke) + (q.z > ke) + (q.w > ke);
        r += (q.x == ke && j < e) + (q.y == ke && j + 1 < e) + (q.z == ke && j + 2 < e) +
             (q.w == ke && j + 3 < e);
      }
      if (r < K) {
        pick[t * MK_MAX_TOPK + r] = e;
        flag[e] = 1u;
      }
    }
    bar_consumers();
    /* the slots: experts chosen by any token, ascending */
    uint32_t words[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) words[i] = __ballot_sync(0xFFFFFFFFu, flag[lane + 32 * i] != 0u);
    const int U = __popc(words[0]) + __popc(words[1]) + __popc(words[2]) + __popc(words[3]);
    auto slot_of = [&](int e) {
      int r = __popc(words[e >> 5] & ((1u << (e & 31)) - 1u));
#pragma unroll
      for (int i = 0; i < 3; ++i) r += (i < (e >> 5)) ? __popc(words[i]) : 0;
      return r;
    };
    if (warp == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if ((words[i] >> lane) & 1u) m->route_expert[slot_of(lane + 32 * i)] = lane + 32 * i;
      if (lane == 0) m->route_U = U;
      if (publish) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if ((words[i] >> lane) & 1u) publish->expert[slot_of(lane + 32 * i)] = lane + 32 * i;
        if (lane == 0) publish->U = U;
      }
    }
    for (int i = tid; i < U * NB; i += NCT) (&m->route_w[0][0])[i] = 0.0f;
    bar_consumers();
    /* token t's weights: warp t, lane k for its k-th choice */
    if (warp < B) {
      const int t = warp;
      const int e = lane < K ? pick[t * MK_MAX_TOPK + lane] : 0;
      const float v = lane < K ? key_value(key[t * 128 + e]) : 0.0f;
      const float v0 = __shfl_sync(0xFFFFFFFFu, v, 0);
      const float ex = lane < K ? expf(v - v0) : 0.0f;
      float z = ex;
#pragma unroll
      for (int sh = 16; sh >= 1; sh >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, sh);
      const float w = z > 0.0f ? ex / z : 0.0f;
      if (lane < K) {
        m->route_w[slot_of(e)][t] = w;
        if (publish) {
          publish->ids[t][lane] = e;
          publish->w[t][lane] = w;
        }
      }
    }
    bar_consumers();
    return true;
  }

  /* The layer's routing in shared memory (route_expert, route_w, route_U),
   * taken once every router piece's logits are written; CTA 0 also records
   * it for the diagnostics, and consumer thread 0 then publishes it to the
   * producer warps.  Called by every consumer thread at the start of a task
   * that needs it (while the out union is not live).  False on timeout /
   * abort. */
  __device__ bool route_local(int layer, int task, int op) {
    const mk_kparams &p = *cx.p;
    Misc<NB> *m = M();
    if (*(volatile int32_t *)&m->route_layer == layer) return true;
    bar_consumers(); /* everyone has read the tag before it can change */
    if (tr && tid == 0 && !t_ready) t_ready = gtimer();
    if (!route_block(layer, cx.cta == 0 ? p.routing + layer : nullptr)) return false;
    if (tid == 0) {
      if (cx.cta == 0) atomicAdd(&p.ctrl->sum_experts, (unsigned long long)m->route_U);
      if (tr && !t_mark) t_mark = gtimer();
      __threadfence_block();
      st_release_cta(&m->route_layer, layer); /* the producer warps may take it from here */
    }
    bar_consumers();
    return true;
  }

  /* Merges n attention partials (consecutive slots at `parts`; per head
   * [m, l, -, -, o[D]] with o unnormalised): M = max_s m_s, L = sum_s
   * e^{m_s - M} l_s, O = sum_s e^{m_s - M} o_s.  With `out` it writes the
   * partial [M, L, -, -, O] there; otherwise bf16(O / L) to ob[g][D].
   * Each thread owns 4 columns of one head and loads every partial's m, l
   * and its columns at once (16 partials per round trip), then combines
   * them in registers: no shared memory, no barrier, one L2 round trip for
   * up to 16 partials. */
  __device__ void merge_parts(const float *parts, int n, int G, int D, float *out, uint16_t *ob) {
    const int PS = D + 4, D4 = D / 4;
    for (int i = tid; i < G * D4; i += NCT) {
      const int gg = i / D4, j4 = i % D4;
      float M = NEG_INF, den = 0.0f;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int s0 = 0; s0 < n; s0 += 16) {
        float m[16], l[16];
        float4 v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          m[u] = NEG_INF;
          l[u] = 0.0f;
          v[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (s0 + u < n) {
            const float *ps = parts + ((size_t)(s0 + u) * G + gg) * PS;
            m[u] = __ldcg(ps);
            l[u] = __ldcg(ps + 1);
            v[u] = __ldcg((const float4 *)(ps + 4) + j4);
          }
        }
        float Mc = M;
#pragma unroll
        for (int u = 0; u < 16; ++u) Mc = fmaxf(Mc, m[u]);
        if (M != NEG_INF) { /* a later chunk raised the maximum: rescale */
          const float sc = expf(M - Mc);
          den *= sc;
          acc.x *= sc;
          acc.y *= sc;
          acc.z *= sc;
          acc.w *= sc;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (m[u] != NEG_INF) {
            const float f = expf(m[u] - Mc);
            den = fmaf(f, l[u], den);
            acc.x = fmaf(f, v[u].x, acc.x);
            acc.y = fmaf(f, v[u].y, acc.y);
            acc.z = fmaf(f, v[u].z, acc.z);
            acc.w = fmaf(f, v[u].w, acc.w);
          }
        M = Mc;
      }
      if (out) {
        *((float4 *)(out + (size_t)gg * PS + 4) + j4) = acc;
        if (j4 == 0) {
          out[(size_t)gg * PS] = M;
          out[(size_t)gg * PS + 1] = den;
        }
      } else {
        const float r = 1.0f / den;
        *(uint2 *)(ob + (size_t)gg * D + j4 * 4) =
            make_uint2(pack_bf16(f2bf(acc.x * r), f2bf(acc.y * r)),
                       pack_bf16(f2bf(acc.z * r), f2bf(acc.w * r)));
      }
    }
    bar_consumers();
  }

  /* ---------------------------------------------------------- attention
   * Split-K flash decoding over the pages of one (sequence, kv head).  Each
   * warp runs the online softmax over the stages it owns on the tensor
   * cores: per 16-key tile, S = Q K^T (A = the group's query heads in rows
   * 0..G-1, B = the K tile read with ldmatrix from the swizzled boxes), then
   * O += P V (A = P in the accumulator layout of S: rows 0..7 its bf16
   * rounding, rows 8..15 the rounding error, so C rows g and g + 8 add up to
   * P V with about 16 significant bits of P; B = the V tile read with a
   * transposing ldmatrix).  Thread (g, t) owns
   * head g: S of keys 2t, 2t+1 of each 8-key half, O of dims 8n + 2t, +1. */
  template <int D>
  __device__ bool op_attn(const int32_t *t, int task, int layer) {
    constexpr int KS = D / 16;           /* k-steps of Q K^T; V n-tile pairs */
    constexpr int NT = D / 8;            /* n-tiles of O */
    constexpr int BI = D < 64 ? D : 64;  /* box inner size (head dims) */
    constexpr int NBOX = D / BI;
    constexpr int CPB = BI / 8;          /* 16-byte chunks per box row */
    constexpr int ROWB = BI * 2;         /* bytes per box row */
    constexpr bool SWZ = D >= 64;        /* 128-byte swizzle */
    constexpr int GC = 2;                /* 16-key tiles per softmax update */
    const mk_kparams &p = *cx.p;
    const int b = t[1], kvh = t[2], p0 = t[3], last = t[8];
    const int G = p.Hq / p.Hkv, P = p.P, half = D / 2;
    const int L_now = __ldg(p.seq_lens + b);
    const int p1 = t[4] >= 0 ? t[4] : (L_now + P - 1) / P;
    if (!cwait(lctr(p, layer, CTR_QKV_DONE), (int)((cx.epoch + 1) * p.n_qkv), task, OP_ATTN,
               layer, CTR_QKV_DONE))
      return false;
    constexpr int QP = D + 8;                     /* q row pitch: conflict-free fragment loads */
    uint16_t *qs = (uint16_t *)cx.xbuf();           /* [8][QP] post-RoPE q, bf16 */
    float *ks = (float *)(cx.xbuf() + 16 * QP);     /* [D] new key */
    float *vs = ks + D;                           /* [D] new value */
    float *mb = vs + D;                           /* warp merge [4][8][D + 8] */
    const int QKVD = (p.Hq + 2 * p.Hkv) * D;
    const uint16_t *qkv = p.qkv + ((size_t)layer * MK_MAX_BATCH + b) * QKVD;
    const float *rp = p.rope + (size_t)(p.rope_per_seq ? b : L_now) * half * 2;
    for (int i = tid; i < 8 * half; i += NCT) {
      const int g = i / half, j = i % half;
      uint16_t o1 = 0, o2 = 0;
      if (g < G) {
        const uint16_t *src = qkv + (size_t)(kvh * G + g) * D;
        const float x1 = bf2f(__ldcg(src + j)), x2 = bf2f(__ldcg(src + j + half));
        const float c = __ldg(rp + 2 * j), s = __ldg(rp + 2 * j + 1);
        o1 = f2bf(__fmul_rn(x1, c) - __fmul_rn(x2, s));
        o2 = f2bf(__fmul_rn(x2, c) + __fmul_rn(x1, s));
      }
      qs[g * QP + j] = o1;
      qs[g * QP + j + half] = o2;
    }
    if (last) {
      const uint16_t *ksrc = qkv + (size_t)(p.Hq + kvh) * D;
      const uint16_t *vsrc = qkv + (size_t)(p.Hq + p.Hkv + kvh) * D;
      const int page = __ldg(p.page_table + b * p.max_pages + L_now / P);
      const size_t row = (((size_t)page * p.Hkv + kvh) * P + (L_now % P)) * D;
      uint16_t *kc = (layer < MK_PARAM_LAYERS ? p.l_kc[layer] : p.layers[layer].kc) + row;
      uint16_t *vc = (layer < MK_PARAM_LAYERS ? p.l_vc[layer] : p.layers[layer].vc) + row;
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

    const int g = lane >> 2, tq = lane & 3, mi = lane >> 3, rr = lane & 7;
    /* A fragments of Q: head g, dims 16j + 2t (+1) and 16j + 2t + 8 (+9) */
    const uint32_t *qf = (const uint32_t *)(qs + g * QP + 2 * tq);
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m_run = NEG_INF, l_run = 0.0f;
    const float scale = p.attn_scale;

    const int pps = mk_pages_per_stage(P, D, cx.SB), pgb = mk_page_stage_bytes(P, D);
    const int kvb = P * D * 2; /* one page's K (or V) box */
    /* byte offset of 16-byte chunk C (head dims 8C..8C+7) of token row r in a
     * box: 128-byte rows of BI dims, row index r * NBOX + C / CPB, chunks
     * XOR-swizzled by the row index mod 8 (the TMA 128-byte pattern) */
    auto boff = [&](int r, int C) -> uint32_t {
      const int r128 = r * NBOX + C / CPB, cb = C % CPB;
      return r128 * ROWB + ((SWZ ? (cb ^ (r128 & 7)) : cb) << 4);
    };
    const int n_st = (p1 - p0 + pps - 1) / pps;
    for (int j = first_mine(); j < n_st; j += NC) {
      uint8_t *st;
      if (!stage_wait(si + j, st, task, OP_ATTN, layer)) break;
      const int q0 = p0 + j * pps, cnt = min(pps, p1 - q0);
      const int valid = min(cnt * P, L_now - q0 * P); /* cached keys in this stage */
      const uint32_t sb = saddr(st);
      for (int k0 = 0; k0 < valid; k0 += 16 * GC) {
        const int ng = min(GC, (valid - k0 + 15) / 16); /* 16-key tiles in this chunk */
        float s[GC][2][4];
#pragma unroll
        for (int gi = 0; gi < GC; ++gi) {
#pragma unroll
          for (int h = 0; h < 2; ++h) s[gi][h][0] = s[gi][h][1] = s[gi][h][2] = s[gi][h][3] = 0.0f;
          if (gi < ng) {
            const int kk0 = k0 + 16 * gi, pg = kk0 / P, r0 = kk0 % P;
            const uint32_t kb = sb + pg * pgb;
            const int kr = r0 + (mi >> 1) * 8 + rr;
#pragma unroll
            for (int jj = 0; jj < KS; ++jj) {
              uint32_t r4[4];
              ldsm4(r4, kb + boff(kr, 2 * jj + (mi & 1)));
              const uint32_t qa0 = qf[8 * jj], qa1 = qf[8 * jj + 4];
              mma16816(s[gi][0], qa0, 0u, qa1, 0u, r4[0], r4[1]);
              mma16816(s[gi][1], qa0, 0u, qa1, 0u, r4[2], r4[3]);
            }
          }
        }
        float mx = NEG_INF;
#pragma unroll
        for (int gi = 0; gi < GC; ++gi)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int key = k0 + 16 * gi + 8 * h + 2 * tq + e;
              const float v = (gi < ng && key < valid) ? s[gi][h][e] * scale : NEG_INF;
              s[gi][h][e] = v;
              mx = fmaxf(mx, v);
            }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_run == NEG_INF ? 0.0f : expf(m_run - m_new);
        l_run *= alpha;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][0] *= alpha;
          o[n][1] *= alpha;
          o[n][2] *= alpha;
          o[n][3] *= alpha;
        }
        m_run = m_new;
#pragma unroll
        for (int gi = 0; gi < GC; ++gi) {
          if (gi < ng) {
            /* A rows g: the bf16 part of P; rows g + 8: what bf16 lost */
            uint32_t ah[2], al[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint16_t hb[2], lb[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float sv = s[gi][h][e];
                const float pv = sv == NEG_INF ? 0.0f : expf(sv - m_new);
                l_run += pv;
                hb[e] = f2bf(pv);
                lb[e] = f2bf(pv - bf2f(hb[e]));
              }
              ah[h] = pack_bf16(hb[0], hb[1]);
              al[h] = pack_bf16(lb[0], lb[1]);
            }
            const int kk0 = k0 + 16 * gi, pg = kk0 / P, r0 = kk0 % P;
            const uint32_t vb = sb + pg * pgb + kvb;
            const int vr = r0 + (mi & 1) * 8 + rr;
#pragma unroll
            for (int i = 0; i < KS; ++i) {
              uint32_t v4[4];
              ldsm4_t(v4, vb + boff(vr, 2 * i + (mi >> 1)));
              if (kk0 + 16 > valid) {
                /* rows past the live length may hold anything (even NaN,
                 * which a zero probability would not cancel): zero them */
                const int ka = kk0 + 2 * tq;
                const uint32_t m0 = (ka < valid ? 0xFFFFu : 0u) | (ka + 1 < valid ? 0xFFFF0000u : 0u);
                const uint32_t m1 =
                    (ka + 8 < valid ? 0xFFFFu : 0u) | (ka + 9 < valid ? 0xFFFF0000u : 0u);
                v4[0] &= m0;
                v4[2] &= m0;
                v4[1] &= m1;
                v4[3] &= m1;
              }
              /* each tile's P V from a zero accumulator, added to O with
               * IEEE fp32 adds: the running sum over thousands of keys stays
               * out of the tensor core's internal adder */
              float t0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, t1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
              mma16816(t0, ah[0], al[0], ah[1], al[1], v4[0], v4[1]);
              mma16816(t1, ah[0], al[0], ah[1], al[1], v4[2], v4[3]);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                o[2 * i][k] += t0[k];
                o[2 * i + 1][k] += t1[k];
              }
            }
          }
        }
      }
      stage_release(si + j);
    }
    si += n_st;
    if (tr && tid == 0) t_mark = gtimer();
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      o[n][0] += o[n][2];
      o[n][1] += o[n][3];
    }
    if (last && warp == 0) {
      /* the new token's own key and value (not in the cache stream) */
      float sp = 0.0f;
      for (int d = tq; d < D; d += 4) sp = fmaf(bf2f(qs[g * QP + d]), ks[d], sp);
      sp += __shfl_xor_sync(0xFFFFFFFFu, sp, 1);
      sp += __shfl_xor_sync(0xFFFFFFFFu, sp, 2);
      const float sn = sp * scale;
      const float m_new = fmaxf(m_run, sn);
      const float alpha = m_run == NEG_INF ? 0.0f : expf(m_run - m_new);
      const float pn = expf(sn - m_new);
      l_run = l_run * alpha + (tq == 0 ? pn : 0.0f);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] = fmaf(pn, vs[8 * n + 2 * tq], o[n][0] * alpha);
        o[n][1] = fmaf(pn, vs[8 * n + 2 * tq + 1], o[n][1] * alpha);
      }
      m_run = m_new;
    }
    l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 1);
    l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 2);

    /* merge warp states pairwise: 8 -> 4 -> 2 -> 1 */
    for (int hw = NC / 2; hw >= 1; hw >>= 1) {
      bar_consumers();
      if (warp >= hw && warp < 2 * hw) {
        const int s = warp - hw;
        if (tq == 0) {
          M()->am[s][g] = m_run;
          M()->al[s][g] = l_run;
        }
        float *dst = mb + (size_t)(s * 8 + g) * (D + 8) + 2 * tq;
#pragma unroll
        for (int n = 0; n < NT; ++n) *(float2 *)(dst + 8 * n) = make_float2(o[n][0], o[n][1]);
      }
      bar_consumers();
      if (warp < hw) {
        const float m2 = M()->am[warp][g], l2 = M()->al[warp][g];
        const float M = fmaxf(m_run, m2);
        const float f1 = m_run == NEG_INF ? 0.0f : expf(m_run - M);
        const float f2 = m2 == NEG_INF ? 0.0f : expf(m2 - M);
        l_run = f1 * l_run + f2 * l2;
        const float *src = mb + (size_t)(warp * 8 + g) * (D + 8) + 2 * tq;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const float2 v = *(const float2 *)(src + 8 * n);
          o[n][0] = f1 * o[n][0] + f2 * v.x;
          o[n][1] = f1 * o[n][1] + f2 * v.y;
        }
        m_run = M;
      }
    }
    /* warp 0 holds this split's partial: per head [m, l, -, -, o[D]] */
    const int PS = D + 4;
    /* the split partials by layer parity: the next layer's splits never
     * overwrite slots this layer's merges still read (two layers apart, the
     * attention-done count of the layer between orders them) */
    const size_t par = (size_t)(layer & 1) * p.n_slots * G * PS;
    float *part = p.attn_part + par + (size_t)t[5] * G * PS;
    if (warp == 0 && g < G) {
      if (tq == 0) {
        part[(size_t)g * PS] = m_run;
        part[(size_t)g * PS + 1] = l_run;
      }
#pragma unroll
      for (int n = 0; n < NT; ++n)
        *(float2 *)(part + (size_t)g * PS + 4 + 8 * n + 2 * tq) = make_float2(o[n][0], o[n][1]);
    }
    /* merge in two levels: the last split of a group to finish merges the
     * group, the last group merger merges the groups and writes o (one
     * level when there is a single group) */
    if (!task_end()) return false;
    const int ng = t[11], bh = b * p.Hkv + kvh;
    const int tk0 = CTR_ATTN_TICKET0 + bh * (1 + MK_MAX_MERGE_GROUPS);
    uint16_t *ob = p.o + ((size_t)layer * MK_MAX_BATCH + b) * p.Hq * D + (size_t)kvh * G * D;
    const float *part1 = p.attn_part + par;
    float *part2 = p.attn_part2 + par;
    if (ng <= 1) {
      if (!ticket(lctr(p, layer, tk0), t[7])) return true;
      merge_parts(part1 + (size_t)t[6] * G * PS, t[7], G, D, nullptr, ob);
    } else {
      if (!ticket(lctr(p, layer, tk0 + 1 + t[9]), t[10])) return true;
      merge_parts(part1 + (size_t)t[12] * G * PS, t[10], G, D, part2 + (size_t)t[13] * G * PS,
                  nullptr);
      if (!ticket(lctr(p, layer, tk0), ng)) return true;
      merge_parts(part2 + (size_t)t[14] * G * PS, ng, G, D, nullptr, ob);
    }
    signal(lctr(p, layer, CTR_ATTN_DONE));
    return true;
  }

  /* ------------------------------------------------------ expert gate/up
   * A share of the (expert slot, ffn index) pairs; each stage holds gate and
   * up rows interleaved, so the thread holding gate row 2j also holds up row
   * 2j + 1 and applies SwiGLU directly. */
  /* Batch 1 with the down projection folded in: the share's blocks of 64
   * f-columns.  First every block's gate and up rows (g and u rounded to
   * bf16, kept in the scratch buffer), then a = bf16(silu(g) u), then the
   * block's down boxes: rows r of the down matrix against a over the block's
   * 64 columns, the partial written to moe_part[block][r] for the OUT tasks,
   * which weight and add the blocks in order. */
  __device__ bool op_up_fold(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    if (!route_local(layer, task, OP_UP)) return false;
    if (!ensure_norm(layer)) return false;
    const int U = M()->route_U, d = p.d;
    const int nbf = p.F / MK_FOLD_COLS, T64 = U * nbf;
    const int b0 = (int)((int64_t)T64 * t[1] / t[2]);
    const int b1 = (int)((int64_t)T64 * (t[1] + 1) / t[2]);
    const int rps = mk_rows_per_stage(d, cx.SB, NB), ng = (MK_FOLD_COLS + rps - 1) / rps;
    const int BR = p.fold_rows, nrb = d / BR;
    const int nA = (b1 - b0) * 2 * ng, nB = (b1 - b0) * nrb;
    float *gsm = (float *)cx.xbuf();
    float *usm = gsm + (b1 - b0) * MK_FOLD_COLS;
    const uint16_t *x = cx.xn();
    const int pitch = 2 * d; /* batch 1: contiguous rows */
    for (int j = first_mine(); j < nA; j += NC) {
      uint8_t *st;
      if (!stage_wait(si + j, st, task, OP_UP, layer)) break;
      const int kb = j / (2 * ng), jj = j % (2 * ng), up = jj >= ng, c = up ? jj - ng : jj;
      float *dst = (up ? usm : gsm) + kb * MK_FOLD_COLS + c * rps;
      cc_rows(st, min(rps, MK_FOLD_COLS - c * rps), pitch, d, x, lane, 0,
              [&](int n0, float sum, int nr) {
                if ((lane & 3) == 0 && (lane >> 2) < nr) dst[n0 + (lane >> 2)] = rbf(sum);
              });
      stage_release(si + j);
    }
    if (!task_end()) return false; /* every g and u of the share is in */
    for (int i = tid; i < (b1 - b0) * MK_FOLD_COLS; i += NCT) {
      const float g = gsm[i];
      gsm[i] = rbf((g / (1.0f + expf(-g))) * usm[i]);
    }
    bar_consumers();
    const int sB = si + nA;
    for (int jb = (warp - sB % NC + NC) % NC; jb < nB; jb += NC) {
      uint8_t *st;
      if (!stage_wait(sB + jb, st, task, OP_UP, layer)) break;
      const int kb = jb / nrb, r0 = (jb % nrb) * BR;
      /* the block's 64 activations (bf16 values held as floats) as bf16
       * pairs, the same on every lane */
      uint32_t a16[MK_FOLD_COLS / 2];
      const float4 *a4 = (const float4 *)(gsm + kb * MK_FOLD_COLS);
#pragma unroll
      for (int i = 0; i < MK_FOLD_COLS / 4; ++i) {
        const float4 v = a4[i];
        a16[2 * i] = (__float_as_uint(v.x) >> 16) | (__float_as_uint(v.y) & 0xFFFF0000u);
        a16[2 * i + 1] = (__float_as_uint(v.z) >> 16) | (__float_as_uint(v.w) & 0xFFFF0000u);
      }
      /* box row r: 128 bytes, 16-byte chunk c stored at (c ^ (r & 7)) */
      const uint32_t sb = saddr(st);
      float *part = p.moe_part + (size_t)(layer & 1) * p.moe_part_stride + (size_t)(b0 + kb) * d + r0;
      for (int r = lane; r < BR; r += 32) {
        float m0 = 0.0f, m1 = 0.0f, m2 = 0.0f, m3 = 0.0f;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint4 w;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                       : "r"(sb + (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4))));
          m0 = fma_bf16h<0>(w.x, a16[4 * ch], m0);
          m1 = fma_bf16h<1>(w.x, a16[4 * ch], m1);
          m2 = fma_bf16h<0>(w.y, a16[4 * ch + 1], m2);
          m3 = fma_bf16h<1>(w.y, a16[4 * ch + 1], m3);
          m0 = fma_bf16h<0>(w.z, a16[4 * ch + 2], m0);
          m1 = fma_bf16h<1>(w.z, a16[4 * ch + 2], m1);
          m2 = fma_bf16h<0>(w.w, a16[4 * ch + 3], m2);
          m3 = fma_bf16h<1>(w.w, a16[4 * ch + 3], m3);
        }
        part[r] = (m0 + m1) + (m2 + m3);
      }
      stage_release(sB + jb);
    }
    si += nA + nB;
    if (!task_end()) return false;
    signal(lctr(p, layer, CTR_UP_DONE));
    return true;
  }

  __device__ bool op_up(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    if (NB == 1 && p.fold) return op_up_fold(t, task, layer);
    if (!route_local(layer, task, OP_UP)) return false;
    if (!ensure_norm(layer)) return false;
    const int U = M()->route_U;
    const int d = p.d, F = p.F, B = p.B;
    const int64_t T = (int64_t)U * F;
    int64_t v = T * t[1] / t[2];
    const int64_t v1 = T * (t[1] + 1) / t[2];
    const uint16_t *x = cx.xn();
    const int pps = mk_pairs_per_stage(d, cx.SB, NB), rb = 2 * d, xp = mk_x_pitch(d, NB);
    int j = 0; /* stage index within the task */
    while (v < v1) {
      const int u = (int)(v / F), f0 = (int)(v % F);
      const int f1 = (int)min((int64_t)F, f0 + (v1 - v));
      uint16_t *out = p.act + (((size_t)layer * p.u_max + u) * MK_MAX_BATCH) * F;
      for (int f = f0; f < f1; f += pps, ++j) {
        if ((si + j) % NC != warp) continue;
        const int cnt = min(pps, f1 - f);
        uint8_t *st;
        if (!stage_wait(si + j, st, task, OP_UP, layer)) continue;
        auto swiglu = [&](int bb, int pr, float gv, float uv) {
          if (bb < B) {
            const float gb = rbf(gv), ub = rbf(uv);
            const float silu = gb / (1.0f + expf(-gb));
            out[(size_t)bb * F + f + pr] = f2bf(silu * ub);
          }
        };
        if (NB == 1 && kB1CudaCores) {
          /* virtual row 2j is gate row j, 2j + 1 up row j: lanes 8j'..8j'+3
           * hold the gate sum, the next four lanes the up sum */
          cc_rows(st, 2 * cnt, rb, d, x, lane, cnt, [&](int n0, float sum, int nr) {
            const float up = __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
            const int r = lane >> 2;
            if ((lane & 7) == 0 && r + 1 < nr) swiglu(0, (n0 + r) >> 1, sum, up);
          });
        } else {
          /* virtual rows 2j (gate) and 2j + 1 (up) of pair j, the up rows
           * being the stage's second run.  Eight tokens: both on one lane
           * (c0, c1 of token g, pair n0 / 2 + t); fewer: gate on even g,
           * up on odd g, four lanes apart. */
          const int ub = cnt * rb + mk_run_gap(NB);
          mma_rows<NB>(
              st, 2 * cnt, d, x, xp, lane,
              [=](int vr) { return (vr & 1) ? ub + (vr >> 1) * rb : (vr >> 1) * rb; },
              [&](int n0, const float(&a)[4], const float(&b)[4], bool two) {
                const int g = lane >> 2, tq = lane & 3;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  if (hh == 1 && !two) break;
                  const float(&c)[4] = hh ? b : a;
                  const int pr = ((n0 + 8 * hh) >> 1) + tq; /* pair within the stage */
                  if (NB >= MK_RUN_GAP_MIN_NB) {
                    if (g < NB && pr < cnt) swiglu(g, pr, c[0], c[1]);
                  } else {
                    const int q = g & 1;
                    const float va = q ? c[1] : c[0];
                    const float oa = __shfl_xor_sync(0xFFFFFFFFu, va, 4);
                    if (q == 0 && pr < cnt && (g >> 1) < NB) swiglu(g >> 1, pr, va, oa);
                  }
                }
              });
        }
        stage_release(si + j);
      }
      v += f1 - f0;
    }
    si += j;
    if (!task_end()) return false;
    signal(lctr(p, layer, CTR_UP_DONE));
    return true;
  }

  /* ------------------------------------------------ expert down rows (batch >= 2)
   * A share of the chosen experts' U x d down rows, per expert segment: the
   * expert's activations (every token's a = silu(g) u, once the gate/up
   * shares are in) staged in the scratch buffer, then its rows of F against
   * them; each row's dot product per token goes to dpart for the OUT tasks,
   * which weight and add them in slot order. */
  __device__ bool op_down(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    if (!route_local(layer, task, OP_DOWN)) return false;
    if (!cwait(lctr(p, layer, CTR_UP_DONE), (int)((cx.epoch + 1) * p.n_up), task, OP_DOWN, layer,
               CTR_UP_DONE))
      return false;
    const int U = M()->route_U, d = p.d, F = p.F, B = p.B;
    const int64_t T = (int64_t)U * d;
    int64_t v = T * t[1] / t[2];
    const int64_t v1 = T * (t[1] + 1) / t[2];
    const int rps = mk_rows_per_stage(F, cx.SB, NB), xpf = mk_x_pitch(F, NB);
    uint16_t *xa = (uint16_t *)cx.xbuf();
    float *dp = p.dpart + (size_t)(layer & 1) * p.u_max * MK_MAX_BATCH * d;
    int j = 0; /* stage index within the task */
    while (v < v1) {
      const int u = (int)(v / d), r0 = (int)(v % d);
      const int r1 = (int)min((int64_t)d, r0 + (v1 - v));
      if (j > 0) bar_consumers(); /* the previous expert's activations are consumed */
      load_x(xa, p.act + (((size_t)layer * p.u_max + u) * MK_MAX_BATCH) * F, F, F);
      bar_consumers();
      float *out = dp + (size_t)u * MK_MAX_BATCH * d;
      const int nst = (r1 - r0 + rps - 1) / rps;
      for (int jj = first_mine_at(si + j); jj < nst; jj += NC) {
        uint8_t *st;
        if (!stage_wait(si + j + jj, st, task, OP_DOWN, layer)) break;
        const int rb = r0 + jj * rps, cnt = min(rps, r1 - rb);
        gemv_stage(st, cnt, F, xa, [&](int r, int bb, float val) {
          if (bb < B) out[(size_t)bb * d + rb + r] = val;
        });
        stage_release(si + j + jj);
      }
      j += nst;
      v += r1 - r0;
    }
    si += j;
    if (!task_end()) return false;
    signal(lctr(p, layer, CTR_DOWN_DONE));
    return true;
  }

  /* ---------------------------------- Wo, expert down + combine, residual */
  __device__ bool op_out(const int32_t *t, int task, int layer) {
    const mk_kparams &p = *cx.p;
    const int r0 = t[2], nr = t[3], B = p.B, d = p.d, F = p.F, HqD = p.Hq * p.D;
    const int target = (int)((cx.epoch + 1) * p.n_attn_done) +
                       (layer == p.poison_layer ? p.poison_delta : 0);
    auto &O = M()->u.out;
    /* the layer's routing (normally known long before), then the residual
     * input rows (final since the layer began) */
    if (!route_local(layer, task, OP_OUT)) return false;
    const int U = M()->route_U;
    const float(*slot_w)[NB] = M()->route_w;
    bool hfail = false;
    for (int i = tid; i < nr * B; i += NCT) {
      const int r = i / B, bb = i % B;
      if (layer == 0) {
        O.hres[r][bb] = bf2f(__ldcg(h_row(0, bb) + r0 + r));
      } else {
        /* the tagged residual (its words are valid by now: this CTA's norm
         * saw them, or the poll waits for them) */
        uint32_t w;
        if (!poll_tagged(p, cx.cta,
                         p.h_tag + ((size_t)layer * MK_MAX_BATCH + bb) * (d / 2) + (r0 + r) / 2, 1,
                         1, p.step_tag, &w, OP_OUT, layer))
          hfail = true;
        O.hres[r][bb] = bf2f((uint16_t)(((r0 + r) & 1) ? (w >> 16) : (w & 0xFFFFu)));
      }
    }
    for (int i = tid; i < NC * MK_MAX_OUT_ROWS * NB; i += NCT) (&O.acc_w[0][0][0])[i] = 0.0f;
    if (bar_any(hfail)) return false;
    /* Wo against the attention output (its rows are in the ring already).
     * Wo's input spans the normed-input buffer and the scratch buffer after
     * it (the normed input is dead: this is the CTA's last task of the
     * layer); the next norm must recompute it. */
    auto wo = [&]() -> bool {
      if (!cwait(lctr(p, layer, CTR_ATTN_DONE), target, task, OP_OUT, layer, CTR_ATTN_DONE))
        return false;
      bar_consumers(); /* every warp is done with xbuf */
      uint16_t *xo = cx.xn();
      if (tid == 0) M()->norm_layer = -2;
      load_x(xo, p.o + (size_t)layer * MK_MAX_BATCH * HqD, HqD, HqD);
      bar_consumers();
      gemv_rows(nr, HqD, xo, task, OP_OUT, layer,
                [&](int r, int bb, float v) { O.acc_o[r][bb] = v; });
      return task_end();
    };
    const bool fold = NB == 1 && p.fold; /* down rows done by the gate/up shares */
    /* Wo first (its rows are in the ring; the attention output is normally
     * complete before the experts' results), then the experts' results of
     * this task's rows, added into acc_w[warp][row][token] in a fixed order. */
    if (!wo()) return false;
    static_assert(MK_MAX_OUT_ROWS >= 32, "a lane per row of an OUT task");
    if (fold) {
      if (!cwait(lctr(p, layer, CTR_UP_DONE), (int)((cx.epoch + 1) * p.n_up), task, OP_OUT,
                 layer, CTR_UP_DONE))
        return false;
      /* the gate/up shares' down partials of this task's rows: warp w adds
       * blocks w, w + NC, ... in that order (lane r for row r0 + r, every
       * load of a batch in flight at once), the warps' sums are added in
       * warp order with the residual below */
      const int nbf = F / MK_FOLD_COLS, T64 = U * nbf;
      constexpr int BAT = 16;
      float s = 0.0f;
      if (lane < nr) {
        const float *src = p.moe_part + (size_t)(layer & 1) * p.moe_part_stride + r0 + lane;
        for (int b0 = warp; b0 < T64; b0 += BAT * NC) {
          float v[BAT];
#pragma unroll
          for (int i = 0; i < BAT; ++i) {
            const int blk = b0 + i * NC;
            v[i] = blk < T64 ? __ldcg(src + (size_t)blk * d) : 0.0f;
          }
#pragma unroll
          for (int i = 0; i < BAT; ++i) {
            const int blk = b0 + i * NC;
            if (blk < T64) s = fmaf(slot_w[blk / nbf][0], v[i], s);
          }
        }
      }
      O.acc_w[warp][lane][0] = s; /* rows nr.. of the task: 0 */
    } else {
      if (!cwait(lctr(p, layer, CTR_DOWN_DONE), (int)((cx.epoch + 1) * p.n_down), task, OP_OUT,
                 layer, CTR_DOWN_DONE))
        return false;
      /* the DOWN tasks' dot products of this task's rows: warp w adds slots
       * w, w + NC, ... (weighted by the token's routing weight) in that
       * order, lane l for (row, token) pairs l, l + 32, ... */
      const float *dp = p.dpart + (size_t)(layer & 1) * p.u_max * MK_MAX_BATCH * d + r0;
      constexpr int BAT = 8;
      for (int q = lane; q < nr * B; q += 32) {
        const int r = q / B, bb = q % B;
        float s = 0.0f;
        for (int u0 = warp; u0 < U; u0 += BAT * NC) {
          float vv[BAT];
#pragma unroll
          for (int i = 0; i < BAT; ++i) {
            const int u = u0 + i * NC;
            vv[i] = u < U ? __ldcg(dp + ((size_t)u * MK_MAX_BATCH + bb) * d + r) : 0.0f;
          }
#pragma unroll
          for (int i = 0; i < BAT; ++i) {
            const int u = u0 + i * NC;
            if (u < U) s = fmaf(slot_w[u][bb], vv[i], s);
          }
        }
        O.acc_w[warp][r][bb] = s;
      }
    }
    bar_consumers(); /* every warp's sums before the residual */
    /* the residual entering the next layer, a pair of rows per thread: one
     * tagged word for the next layer's readers, plain copies (and the two
     * terms) for the diagnostics.  r0 and nr are even. */
    for (int i = tid; i < (nr / 2) * B; i += NCT) {
      const int r = 2 * (i / B), bb = i % B;
      uint16_t hn[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float hv = O.hres[r + q][bb];
        const uint16_t at = f2bf(O.acc_o[r + q][bb]);
        float mo = 0.0f;
#pragma unroll
        for (int w = 0; w < NC; ++w) mo += O.acc_w[w][r + q][bb];
        const uint16_t mb = f2bf(mo);
        hn[q] = f2bf(__fadd_rn(__fadd_rn(hv, bf2f(at)), bf2f(mb)));
        p.h[((size_t)(layer + 1) * MK_MAX_BATCH + bb) * d + r0 + r + q] = hn[q];
        uint16_t *am = p.am + ((size_t)layer * 2 * MK_MAX_BATCH + bb) * d + r0 + r + q;
        am[0] = at;
        am[(size_t)MK_MAX_BATCH * d] = mb;
        if (layer == 0) p.h[(size_t)bb * d + r0 + r + q] = f2bf(hv);
      }
      st_tag(p.h_tag + ((size_t)(layer + 1) * MK_MAX_BATCH + bb) * (d / 2) + (r0 + r) / 2,
             (uint32_t)hn[0] | ((uint32_t)hn[1] << 16), p.step_tag);
    }
    bar_consumers(); /* the out union is read before the next task reuses it */
    return true;
  }

  /* ---------------------------------------------- final norm + LM head */
  __device__ bool op_lm(const int32_t *t, int task) {
    const mk_kparams &p = *cx.p;
    const int L = p.L, B = p.B;
    /* the final residual (tagged, as the last OUT tasks write it) */
    if (*(volatile int32_t *)&M()->norm_layer != L) {
      bar_consumers();
      if (!norm_into_xbuf(L, p.final_norm)) return false;
    }
    const int v0 = t[2];
    /* each lane sees the rows of one token: token 0 on every lane on the
     * CUDA cores; on the tensor cores token lane / 4 with eight tokens,
     * lane / 8 with fewer */
    float best_v = NEG_INF;
    int best_i = 0x7FFFFFFF;
    float *logits = p.out_logits;
    const int V = p.V;
    gemv_rows(t[3], p.d, cx.xn(), task, OP_LM, L, [&](int r, int bb, float v) {
      if (bb < B) {
        if (logits) logits[(size_t)bb * V + v0 + r] = v;
        if (v > best_v || (v == best_v && v0 + r < best_i)) {
          best_v = v;
          best_i = v0 + r;
        }
      }
    });
    /* the lanes holding a token's rows, then the warps */
    auto &LM = M()->u.lm;
    constexpr int LANES = (NB == 1 && kB1CudaCores) ? 32 : NB >= MK_RUN_GAP_MIN_NB ? 4 : 8;
#pragma unroll
    for (int s = 1; s < LANES; s <<= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, best_v, s);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, best_i, s);
      if (ov > best_v || (ov == best_v && oi < best_i)) {
        best_v = ov;
        best_i = oi;
      }
    }
    {
      const int bb = lane / LANES;
      if (lane % LANES == 0 && bb < NB) {
        LM.best[warp][bb][0] = best_v;
        LM.best[warp][bb][1] = __int_as_float(best_i);
      }
    }
    if (!task_end()) return false;
    if (tid < B) {
      float bv = NEG_INF;
      int bi = 0x7FFFFFFF;
      for (int w = 0; w < NC; ++w) {
        const float v = LM.best[w][tid][0];
        const int i = __float_as_int(LM.best[w][tid][1]);
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
      float bv = NEG_INF;
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
      case OP_ATTN:
        ok = cx.p->D == 128 ? op_attn<128>(t, task, layer)
             : cx.p->D == 64 ? op_attn<64>(t, task, layer)
                             : op_attn<32>(t, task, layer);
        break;
      case OP_UP: ok = op_up(t, task, layer); break;
      case OP_OUT: ok = op_out(t, task, layer); break;
      case OP_DOWN: ok = op_down(t, task, layer); break;
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
__global__ void __launch_bounds__(MK_THREADS, 1) decode_kernel(const __grid_constant__ mk_kparams p) {
  /* the ring starts on a 1024-byte boundary (128-byte swizzled TMA boxes);
   * the launch adds MK_SMEM_STATIC bytes of slack for that */
  Ctx cx;
  cx.p = &p;
  cx.SB = p.stage_bytes;
  cx.NS = p.ring_slots;
  cx.ring_off = (1024u - (saddr(mk_smem) & 1023u)) & 1023u;
  cx.xn_off = cx.ring_off + (uint32_t)p.ring_slots * p.stage_bytes;
  cx.xbuf_off = cx.xn_off + (uint32_t)p.xn_bytes;
  cx.misc_off = cx.xbuf_off + (uint32_t)p.xbuf_bytes;
  Misc<NB> *misc = (Misc<NB> *)(mk_smem + cx.misc_off);
  cx.cta = blockIdx.x;
  cx.epoch = *(volatile uint32_t *)&p.ctrl->epoch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NC; ++s) {
      mbar_init(&misc->full[s], 1);
      mbar_init(&misc->empty[s], 1);
    }
    misc->norm_layer = -2;
    misc->route_layer = -1;
    misc->ok = 1;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  /* the CTA's task-table row, read by every task of every layer, is copied
   * to shared memory when it fits */
  /* the stage trace's clock anchors: (globaltimer, SM clock) at start and end */
  unsigned long long *anchor =
      (p.stage_trace && (int)blockIdx.x == p.stage_trace_cta)
          ? p.stage_trace + (size_t)(MK_STAGE_TRACE_EVENTS - 1) * 8
          : nullptr;
  if (anchor && threadIdx.x == 0) {
    anchor[0] = gtimer();
    anchor[1] = sclock();
  }
  const int32_t *grow = p.table + (size_t)blockIdx.x * p.tasks_per_cta * MK_DESC_INTS;
  const bool row_in_smem = p.tasks_per_cta <= MK_SMEM_TASKS;
  if (row_in_smem)
    for (int i = threadIdx.x; i < p.tasks_per_cta * MK_DESC_INTS; i += MK_THREADS)
      (&misc->tasks[0][0])[i] = __ldg(grow + i);
  __syncthreads();
  const int32_t *row = row_in_smem ? &misc->tasks[0][0] : grow;
  const bool header_ok = row[0] == OP_HEADER;
  if (header_ok) {
    if (warp >= NC) {
      produce<NB>(cx, warp - NC, lane, misc->qd[warp - NC], misc->pexp[warp - NC],
                  &misc->pU[warp - NC],
                  (int)blockIdx.x == p.stage_trace_cta ? p.stage_trace : nullptr, row);
    } else {
      Consumer<NB> c;
      c.cx = cx;
      c.warp = warp;
      c.lane = lane;
      c.tid = threadIdx.x;
      c.tr = p.trace ? p.trace + (size_t)blockIdx.x * p.trace_cap * MK_TRACE_WORDS : nullptr;
      c.tr_n = 0;
      const bool ok = c.run(row);
      if (threadIdx.x == 0 && !ok) misc->ok = 0;
    }
  } else if (threadIdx.x == 0) {
    raise_error(p, MK_ERR_BAD_TASK, blockIdx.x, -1, row[0], -1, -1, 0, 0);
    misc->ok = 0;
  }
  __syncthreads();
  if (anchor && threadIdx.x == 0) {
    anchor[2] = gtimer();
    anchor[3] = sclock();
  }
  if (threadIdx.x == 0 && misc->ok && !ld_volatile(&p.ctrl->abort)) {
    /* the last CTA out advances the epoch */
    __threadfence();
    const int old = atom_add_acq_rel(gctr(p, GCTR_EXIT), 1);
    if (old == (int)((cx.epoch + 1) * (uint32_t)gridDim.x) - 1)
      *(volatile uint32_t *)&p.ctrl->epoch = cx.epoch + 1;
  }
}

}  // namespace mk

/* ---- library-internal entry points (used by mk_api.cpp) ------------------ */

extern "C" size_t mk_misc_bytes(int nb) {
  return nb == 1   ? sizeof(mk::Misc<1>)
         : nb == 2 ? sizeof(mk::Misc<2>)
         : nb == 4 ? sizeof(mk::Misc<4>)
                   : sizeof(mk::Misc<8>);
}


static void *mk_kernel_fn(int nb) {
  return nb == 1   ? (void *)mk::decode_kernel<1>
         : nb == 2 ? (void *)mk::decode_kernel<2>
         : nb == 4 ? (void *)mk::decode_kernel<4>
                   : (void *)mk::decode_kernel<8>;
}

/* Sets the kernel's dynamic shared-memory limit on the current device to the
 * largest size any plan uses (MK_SMEM_OPTIN), so that every later launch of
 * this instantiation -- whatever model dims it was planned for, from any
 * context or from mk_decode_step_static -- stays within the limit, and
 * reports how many CTAs of `smem` bytes fit on an SM. */
extern "C" cudaError_t mk_kernel_prepare(int nb, size_t smem, int *blocks_per_sm) {
  void *fn = mk_kernel_fn(nb);
  if (smem > MK_SMEM_OPTIN) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MK_SMEM_OPTIN);
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
