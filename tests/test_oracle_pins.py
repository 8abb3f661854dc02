"""Pins for the oracle's building blocks (CPU).

Each test ties one step of the oracle to something other than the oracle
itself: a closed form, a textbook identity, a library routine (numpy/scipy)
or an invariant of the mathematics.  The shapes are non-square and the
values asymmetric so that a transposed operand, a swapped pair, a wrong
sign or a dropped term fails at least one of them.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from bf16util import rnd, to_bits, to_f32, ulp

RNG = np.random.default_rng(1234)


def bits(x):
    return to_bits(np.asarray(x, dtype=np.float64))


# ------------------------------------------------------------------ RMSNorm


@pytest.mark.parametrize("c", [0.5, 3.0, 1e-3, -2.25])
def test_rmsnorm_constant_vector_closed_form(c):
    d, eps = 256, 1e-6
    h = bits(np.full(d, c))
    cb = float(to_f32(h[:1])[0])
    n = to_f32(oracle.rmsnorm(h, bits(np.ones(d)), eps))
    expect = rnd(cb / math.sqrt(cb * cb + eps))
    assert np.all(np.abs(n - expect) <= ulp(expect))


def test_rmsnorm_small_vector_closed_form():
    # h = (3, 4, 0, 0): mean of squares 25/4, 1/rms = 0.4 -> (1.2, 1.6, 0, 0).
    n = to_f32(oracle.rmsnorm(bits([3, 4, 0, 0]), bits([1, 1, 1, 1]), 0.0))
    assert np.array_equal(n, rnd([1.2, 1.6, 0.0, 0.0]).astype(np.float32))
    # gains multiply element-wise, eps enters under the root
    n2 = to_f32(oracle.rmsnorm(bits([3, 4, 0, 0]), bits([2, 1, 1, -1]), 0.0))
    assert np.array_equal(n2, rnd([2.4, 1.6, 0.0, 0.0]).astype(np.float32))
    n3 = to_f32(oracle.rmsnorm(bits([3, 4, 0, 0]), bits([1, 1, 1, 1]), 18.75))
    assert np.array_equal(n3, rnd([0.6, 0.8, 0.0, 0.0]).astype(np.float32))


def test_rmsnorm_zero_and_scale_invariance():
    d = 300
    z = to_f32(oracle.rmsnorm(np.zeros(d, np.uint16), bits(np.ones(d)), 1e-6))
    assert np.all(z == 0)
    h = bits(RNG.normal(0, 1, d))
    g = bits(RNG.normal(1, 0.1, d))
    a = oracle.rmsnorm(h, g, 0.0)
    b = oracle.rmsnorm(bits(to_f32(h) * 4.0), g, 0.0)  # power of two: exact
    assert np.array_equal(a, b)


def test_rmsnorm_random_vs_float64():
    d = 2048
    h = bits(RNG.normal(0, 0.7, d))
    g = bits(RNG.normal(1, 0.2, d))
    hf, gf = to_f32(h).astype(np.float64), to_f32(g).astype(np.float64)
    expect = hf / np.sqrt(np.mean(hf ** 2) + 1e-6) * gf
    n = to_f32(oracle.rmsnorm(h, g, 1e-6)).astype(np.float64)
    assert np.all(np.abs(n - expect) <= ulp(expect) * 0.5 + 1e-6 * np.abs(expect))


# --------------------------------------------------------------------- GEMV


@pytest.mark.parametrize("rows,cols", [(37, 300), (5, 2048), (130, 7)])
def test_gemv_vs_numpy_higham_bound(rows, cols):
    w = bits(RNG.normal(0, 0.05, (rows, cols)))
    x = bits(RNG.normal(0, 1.0, cols))
    wf, xf = to_f32(w).astype(np.float64), to_f32(x).astype(np.float64)
    exact = wf @ xf
    u = 2.0 ** -24
    gamma = cols * u / (1 - cols * u)
    bound = gamma * (np.abs(wf) @ np.abs(xf))
    y = oracle.gemv(w, x)
    assert np.all(np.abs(y - exact) <= bound)
    yd = oracle.gemv(w, x, accum_double=True)
    assert np.all(np.abs(yd - exact) <= np.abs(exact) * 2 ** -23 + 1e-30)


def test_gemv_is_not_transposed():
    # W = [[1, 2, 3], [4, 5, 6]], x = (1, 0, -1) -> (-2, -2); W^T would not fit.
    y = oracle.gemv(bits([[1, 2, 3], [4, 5, 6]]), bits([1, 0, -1]))
    assert np.array_equal(y, np.array([-2.0, -2.0], np.float32))
    y = oracle.gemv(bits([[1, 2, 3], [4, 5, 7]]), bits([0, 0, 1]))
    assert np.array_equal(y, np.array([3.0, 7.0], np.float32))


# --------------------------------------------------------------------- RoPE


def test_rope_position_zero_is_identity():
    x = bits(RNG.normal(0, 1, 4 * 64))
    assert np.array_equal(oracle.rope(x, 4, 64, 0, 10000.0), x)


@pytest.mark.parametrize("D,base", [(64, 10000.0), (128, 10000.0), (8, 500.0)])
@pytest.mark.parametrize("pos", [1, 7, 1000, 262143])
def test_rope_unit_vectors_closed_form(D, base, pos):
    """Rotate-half: pair (i, i + D/2) turns by pos * base^(-2i/D)."""
    half = D // 2
    for i in (0, 1, half - 1):
        theta = pos * base ** (-2.0 * i / D)
        c, s = rnd(np.float32(math.cos(theta))), rnd(np.float32(math.sin(theta)))
        e = np.zeros(D)
        e[i] = 1.0
        out = to_f32(oracle.rope(bits(e), 1, D, pos, base))
        assert out[i] == pytest.approx(c, abs=1e-7) and out[i + half] == pytest.approx(s, abs=1e-7)
        others = np.delete(out, [i, i + half])
        assert np.all(others == 0)
        e2 = np.zeros(D)
        e2[i + half] = 1.0
        out2 = to_f32(oracle.rope(bits(e2), 1, D, pos, base))
        assert out2[i] == pytest.approx(-s, abs=1e-7) and out2[i + half] == pytest.approx(c, abs=1e-7)


def test_rope_heads_independent_and_norm_preserving():
    D, H = 64, 3
    x = bits(RNG.normal(0, 1, (H, D)))
    out = to_f32(oracle.rope(x.ravel(), H, D, 77, 10000.0)).reshape(H, D)
    for h in range(H):
        single = to_f32(oracle.rope(x[h], 1, D, 77, 10000.0))
        assert np.array_equal(out[h], single)
    xf = to_f32(x).astype(np.float64)
    half = D // 2
    n_in = xf[:, :half] ** 2 + xf[:, half:] ** 2
    n_out = out[:, :half].astype(np.float64) ** 2 + out[:, half:].astype(np.float64) ** 2
    assert np.allclose(n_in, n_out, rtol=2e-2, atol=1e-4)


def test_rope_relative_position_invariance():
    D = 128
    q = bits(RNG.normal(0, 1, D))
    k = bits(RNG.normal(0, 1, D))

    def score(p, s):
        a = to_f32(oracle.rope(q, 1, D, p, 10000.0)).astype(np.float64)
        b = to_f32(oracle.rope(k, 1, D, s, 10000.0)).astype(np.float64)
        return a @ b

    ref = score(10, 3)
    scale = np.linalg.norm(to_f32(q)) * np.linalg.norm(to_f32(k))
    for t in (1, 100, 5000):
        assert abs(score(10 + t, 3 + t) - ref) < 2e-2 * scale


# ---------------------------------------------------------------- attention


def test_attention_single_key_returns_value_row():
    D = 128
    q, k, v = (bits(RNG.normal(0, 1, (1, D))) for _ in range(3))
    assert np.array_equal(oracle.attention_head(q[0], k, v), v[0])


def test_attention_identical_keys_and_zero_query_average_values():
    D, n = 64, 7
    v = bits(RNG.normal(0, 1, (n, D)))
    k = np.tile(bits(RNG.normal(0, 1, D)), (n, 1))
    q = bits(RNG.normal(0, 1, D))
    mean = to_f32(v).astype(np.float64).mean(0)
    for qq, kk in ((q, k), (np.zeros(D, np.uint16), bits(RNG.normal(0, 1, (n, D))))):
        o = to_f32(oracle.attention_head(qq, kk, v)).astype(np.float64)
        assert np.all(np.abs(o - mean) <= ulp(mean) + 1e-6)


@pytest.mark.parametrize("t", [0.5, 3.0, -4.0])
def test_attention_two_keys_closed_form_scale(t):
    """q = t*e0, k1 = e0, k2 = 0: weights sigmoid(t / sqrt(D)), 1 - that."""
    D = 64
    q = np.zeros(D)
    q[0] = t
    k = np.zeros((2, D))
    k[0, 0] = 1.0
    v = np.zeros((2, D))
    v[0, 0] = 1.0
    v[1, 1] = 1.0
    o = to_f32(oracle.attention_head(bits(q), bits(k), bits(v)))
    w1 = 1.0 / (1.0 + math.exp(-t / math.sqrt(D)))
    assert o[0] == pytest.approx(rnd(w1), abs=1e-7)
    assert o[1] == pytest.approx(rnd(1 - w1), abs=1e-7)
    assert np.all(o[2:] == 0)


def test_attention_random_vs_scipy_softmax_and_permutation():
    D, n = 128, 333
    q = bits(RNG.normal(0, 1, D))
    k = bits(RNG.normal(0, 1, (n, D)))
    v = bits(RNG.normal(0, 1, (n, D)))
    qf, kf, vf = (to_f32(a).astype(np.float64) for a in (q, k, v))
    expect = softmax(kf @ qf / math.sqrt(D)) @ vf
    o = to_f32(oracle.attention_head(q, k, v)).astype(np.float64)
    assert np.all(np.abs(o - expect) <= ulp(expect) + 1e-5)
    perm = RNG.permutation(n)
    o2 = to_f32(oracle.attention_head(q, k[perm], v[perm])).astype(np.float64)
    assert np.all(np.abs(o2 - o) <= 2 * ulp(o) + 1e-5)


# ------------------------------------------------------------------- router


def test_router_topk_matches_full_sort_and_weights_sum_to_one():
    for trial in range(200):
        E = int(RNG.choice([8, 32, 128]))
        k = int(RNG.integers(1, min(E, 9)))
        r = RNG.normal(0, 1, E).astype(np.float32)
        ids, w, margin = oracle.route(r, k)
        order = np.lexsort((np.arange(E), -r.astype(np.float64)))
        assert np.array_equal(ids, order[:k])
        assert abs(float(w.astype(np.float64).sum()) - 1.0) < 1e-6
        # softmax over all E then renormalise == softmax over the top-k logits
        assert np.allclose(w, softmax(r[ids].astype(np.float64)), rtol=1e-5, atol=1e-7)
        assert margin == pytest.approx(float(r[order[k - 1]]) - float(r[order[k]]))


def test_router_ties_lower_id_and_k_equals_e():
    ids, w, _ = oracle.route(np.zeros(16, np.float32), 4)
    assert ids.tolist() == [0, 1, 2, 3] and np.allclose(w, 0.25)
    r = np.array([0.5, 2.0, 0.5, 1.0, 0.5], np.float32)
    ids, _, margin = oracle.route(r, 3)
    assert ids.tolist() == [1, 3, 0] and margin == 0.0
    ids, w, _ = oracle.route(r, 5)
    assert ids.tolist() == [1, 3, 0, 2, 4]
    assert np.allclose(w, softmax(r.astype(np.float64))[ids], rtol=1e-6)


# ------------------------------------------------------------- SwiGLU expert


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-6)
    assert oracle.silu(-1.0) == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-6)
    assert oracle.silu(30.0) == pytest.approx(30.0, rel=1e-6)
    assert abs(oracle.silu(-30.0)) < 1e-11


def test_expert_gate_up_down_roles():
    """Wg = I, Wu = 2I, Wd = a permutation: y = P (bf16(silu(n) * 2n))."""
    d = 16
    n = bits(RNG.normal(0, 1, d))
    nf = to_f32(n).astype(np.float64)
    perm = RNG.permutation(d)
    wd = np.zeros((d, d))
    wd[np.arange(d), perm] = 1.0  # y[i] = a[perm[i]]
    y = oracle.expert(n, bits(np.eye(d)), bits(2 * np.eye(d)), bits(wd))
    a = rnd(nf / (1 + np.exp(-nf)) * 2 * nf)
    assert np.allclose(y, a[perm], rtol=0, atol=ulp(a[perm]))


def test_expert_zero_gate_gives_zero():
    d, f = 32, 24
    n = bits(RNG.normal(0, 1, d))
    y = oracle.expert(n, np.zeros((f, d), np.uint16), bits(RNG.normal(0, 1, (f, d))),
                      bits(RNG.normal(0, 1, (d, f))))
    assert np.all(y == 0)
