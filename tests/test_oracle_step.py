"""Pins for the oracle's whole decode step (CPU).

1. A float64 brute force written here with numpy/scipy library routines
   (matmul, softmax, argsort), following the same rounding points, agrees
   with the oracle on the tiny workload, over several greedy steps.
2. Invariants of the computation: paged == contiguous KV (bit-exact), an
   empty cache makes every head's output its kv head's new V row, decoding
   is incremental (step t+1 equals a fresh run whose cache holds step t's
   rows), sequences in a batch do not interact, a MoE whose experts are all
   identical equals the single dense SwiGLU MLP, and a large router bias
   forces an expert in.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import synth
from bf16util import rnd, to_bits, to_f32, ulp

TINY = synth.TINY


def tiny_inputs(dims=TINY, seq_lens=(64,), reserve=9, shuffle=True, gen=0):
    pl = synth.page_layout(dims, list(seq_lens), reserve, shuffle=shuffle, gen=gen)
    t = {k: synth.host_tensor(s) for k, s in synth.weight_specs(dims).items()}
    t.update({k: synth.host_tensor(s) for k, s in synth.kv_specs(dims, pl.num_pages, gen).items()})
    return t, pl


# ----------------------------------------------------------- numpy brute force


class BruteForce:
    """Float64 accumulation, the same bf16 rounding points; numpy routines."""

    def __init__(self, dims, t, seq_lens, page_tables):
        self.d, self.t = dims, t
        self.lens = list(seq_lens)
        self.pt = page_tables
        D, P, H = dims.head_dim, dims.page_size, dims.n_kv_heads
        self.K, self.V = [], []
        for l in range(dims.n_layers):
            kp = to_f32(t[f"l{l}.kpool"]).astype(np.float64)
            vp = to_f32(t[f"l{l}.vpool"]).astype(np.float64)
            ks, vs = [], []
            for b, L in enumerate(self.lens):
                pages = page_tables[b, np.arange(L) // P]
                ks.append(kp[pages, :, np.arange(L) % P, :])  # [L][H][D]
                vs.append(vp[pages, :, np.arange(L) % P, :])
            self.K.append(ks)
            self.V.append(vs)

    def W(self, name):
        return to_f32(self.t[name]).astype(np.float64)

    def norm(self, h, g):
        return rnd(h / np.sqrt(np.mean(h * h) + self.d.rms_eps) * g)

    def rope(self, x, pos):
        D = self.d.head_dim
        half = D // 2
        i = np.arange(half)
        ang = pos * self.d.rope_base ** (-2.0 * i / D)
        c = np.cos(ang).astype(np.float32).astype(np.float64)
        s = np.sin(ang).astype(np.float32).astype(np.float64)
        x1, x2 = x[:, :half], x[:, half:]
        return rnd(np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=1))

    def layer(self, l, b, h):
        """Layer l for sequence b from the residual h (float64 holding bf16
        values): appends the new K/V row, returns (next residual, top-k ids)."""
        d = self.d
        D, Hq, Hkv, E, k = d.head_dim, d.n_q_heads, d.n_kv_heads, d.n_experts, d.top_k
        G = Hq // Hkv
        p = f"l{l}."
        n = self.norm(h, self.W(p + "norm"))
        q = rnd(self.W(p + "wq") @ n).reshape(Hq, D)
        kk = rnd(self.W(p + "wk") @ n).reshape(Hkv, D)
        vv = rnd(self.W(p + "wv") @ n).reshape(Hkv, D)
        pos = self.lens[b]
        q, kk = self.rope(q, pos), self.rope(kk, pos)
        self.K[l][b] = np.concatenate([self.K[l][b], kk[None]], 0)
        self.V[l][b] = np.concatenate([self.V[l][b], vv[None]], 0)
        o = np.empty((Hq, D))
        for i in range(Hq):
            Kh, Vh = self.K[l][b][:, i // G, :], self.V[l][b][:, i // G, :]
            o[i] = rnd(softmax(Kh @ q[i] / math.sqrt(D)) @ Vh)
        attn = rnd(self.W(p + "wo") @ o.ravel())
        r = self.W(p + "wr") @ n
        r32 = r.astype(np.float32)
        top = np.lexsort((np.arange(E), -r32.astype(np.float64)))[:k]
        w = softmax(r32[top].astype(np.float64))
        acc = np.zeros(d.d_model)
        wg, wu, wd = self.W(p + "wg"), self.W(p + "wu"), self.W(p + "wd")
        for e, we in zip(top, w):
            g, u = rnd(wg[e] @ n), rnd(wu[e] @ n)
            a = rnd(g / (1 + np.exp(-g)) * u)
            acc += we * (wd[e] @ a)
        moe = rnd(acc)
        return rnd(h + attn + moe), top

    def step(self, tokens):
        emb = self.W("embed")
        logits_all, ids_all = [], []
        for b, tok in enumerate(tokens):
            h = emb[tok].copy()
            ids_b = []
            for l in range(self.d.n_layers):
                h, top = self.layer(l, b, h)
                ids_b.append(top)
            nf = self.norm(h, self.W("final_norm"))
            logits_all.append(self.W("lm_head") @ nf)
            ids_all.append(ids_b)
        self.lens = [L + 1 for L in self.lens]
        return np.array(logits_all), np.array(ids_all).transpose(1, 0, 2)


def test_oracle_matches_float64_brute_force_over_greedy_steps():
    t, pl = tiny_inputs()
    orc = oracle.Oracle(TINY, t, [64], pl.page_tables)
    bf = BruteForce(TINY, t, [64], pl.page_tables)
    tok = synth.first_tokens(TINY, 1)
    for step in range(9):
        r = orc.step(tok)
        logits, ids = bf.step(tok)
        err = np.abs(r["logits"] - logits)
        assert err.max() < 2e-2, (step, err.max())
        rel = np.linalg.norm(r["logits"] - logits) / np.linalg.norm(logits)
        assert rel < 1e-2
        clear = r["route_margin"] > 1e-2
        assert np.array_equal(np.sort(r["route_ids"], -1)[clear], np.sort(ids, -1)[clear])
        if r["argmax_margin"][0] > 1e-2:
            assert r["next_tokens"][0] == int(np.argmax(logits[0]))
        tok = r["next_tokens"]


# d != F, odd group size, E not a power of two, two ragged sequences: a
# transposed or mis-strided operand cannot hide behind a square shape.
ODD = synth.Dims(2, 160, 6, 2, 32, 6, 2, 96, 300)


def test_oracle_matches_brute_force_on_odd_shapes_batch2():
    lens = [29, 3]
    t, pl = tiny_inputs(dims=ODD, seq_lens=lens, reserve=3)
    orc = oracle.Oracle(ODD, t, lens, pl.page_tables)
    bf = BruteForce(ODD, t, lens, pl.page_tables)
    tok = [7, 250]
    for step in range(3):
        r = orc.step(tok)
        logits, ids = bf.step(tok)
        assert np.abs(r["logits"] - logits).max() < 2e-2
        clear = r["route_margin"] > 1e-2
        assert np.array_equal(np.sort(r["route_ids"], -1)[clear], np.sort(ids, -1)[clear])
        tok = [int(np.argmax(x)) for x in logits]


def test_oracle_double_accumulation_agrees_with_brute_force_closely():
    t, pl = tiny_inputs()
    orc = oracle.Oracle(TINY, t, [64], pl.page_tables, accum_double=True)
    bf = BruteForce(TINY, t, [64], pl.page_tables)
    tok = synth.first_tokens(TINY, 1)
    r = orc.step(tok)
    logits, ids = bf.step(tok)
    assert np.abs(r["logits"] - logits).max() < 2e-3


def test_reverse_order_fp32_mode_is_the_same_sums_reordered():
    """The descending-order fp32 mode (used only to measure the fp32 noise
    floor) computes the same sums as the other modes: it agrees with the
    float64 brute force as closely as the ascending mode does, and it is a
    genuinely different rounding order (some logit differs in its low bits)."""
    t, pl = tiny_inputs()
    fwd = oracle.Oracle(TINY, t, [64], pl.page_tables)
    rev = oracle.Oracle(TINY, t, [64], pl.page_tables, reverse=True)
    bf = BruteForce(TINY, t, [64], pl.page_tables)
    tok = synth.first_tokens(TINY, 1)
    rf, rr = fwd.step(tok), rev.step(tok)
    logits, _ = bf.step(tok)
    assert np.abs(rr["logits"] - logits).max() < 2e-2
    assert np.linalg.norm(rr["logits"] - logits) / np.linalg.norm(logits) < 1e-2
    assert np.abs(rr["logits"] - rf["logits"]).max() < 2e-2
    assert not np.array_equal(rr["logits"], rf["logits"])


# ------------------------------------------------------------------ invariants


def test_paged_equals_contiguous_bit_exact():
    t, pl = tiny_inputs(seq_lens=(64, 40))
    # Contiguous copy: logical page j of sequence b stored at physical page
    # (running index), identity-ordered.
    t2 = dict(t)
    order = [pl.page_tables[b, j] for b in range(2) for j in range(pl.page_tables.shape[1])
             if pl.page_tables[b, j] >= 0]
    ident = np.full_like(pl.page_tables, -1)
    at = 0
    for b in range(2):
        for j in range(pl.page_tables.shape[1]):
            if pl.page_tables[b, j] >= 0:
                ident[b, j] = at
                at += 1
    for l in range(TINY.n_layers):
        for kind in ("kpool", "vpool"):
            t2[f"l{l}.{kind}"] = np.ascontiguousarray(t[f"l{l}.{kind}"][order])
    tok = synth.first_tokens(TINY, 2)
    a = oracle.Oracle(TINY, t, [64, 40], pl.page_tables).step(tok)
    b = oracle.Oracle(TINY, t2, [64, 40], ident).step(tok)
    assert np.array_equal(a["logits"], b["logits"])
    assert np.array_equal(a["route_ids"], b["route_ids"])


def test_empty_cache_head_output_is_new_value_row():
    t, pl = tiny_inputs(seq_lens=(0,))
    r = oracle.Oracle(TINY, t, [0], pl.page_tables).step([5], dumps=("o", "v"))
    D, G = TINY.head_dim, TINY.n_q_heads // TINY.n_kv_heads
    for l in range(TINY.n_layers):
        o = r["o"][l, 0].reshape(TINY.n_q_heads, D)
        v = r["v"][l, 0].reshape(TINY.n_kv_heads, D)
        for i in range(TINY.n_q_heads):
            assert np.array_equal(o[i], v[i // G])


def test_incremental_decode_equals_fresh_cache():
    """Step 2 after step 1 == a fresh state whose pool holds step 1's rows."""
    t, pl = tiny_inputs(seq_lens=(37,))
    tok1, tok2 = [11], [700]
    inc = oracle.Oracle(TINY, t, [37], pl.page_tables)
    r1 = inc.step(tok1, dumps=("k", "v"))
    r2 = inc.step(tok2)
    t2 = dict(t)
    P, D = TINY.page_size, TINY.head_dim
    page, slot = pl.page_tables[0, 37 // P], 37 % P
    for l in range(TINY.n_layers):
        kp = t[f"l{l}.kpool"].copy()
        vp = t[f"l{l}.vpool"].copy()
        kp[page, :, slot, :] = r1["k"][l, 0].reshape(TINY.n_kv_heads, D)
        vp[page, :, slot, :] = r1["v"][l, 0].reshape(TINY.n_kv_heads, D)
        t2[f"l{l}.kpool"], t2[f"l{l}.vpool"] = kp, vp
    fresh = oracle.Oracle(TINY, t2, [38], pl.page_tables).step(tok2)
    assert np.array_equal(r2["logits"], fresh["logits"])


def test_batch_rows_do_not_interact():
    t, pl = tiny_inputs(seq_lens=(64, 21, 50))
    tok = [3, 900, 3]
    both = oracle.Oracle(TINY, t, [64, 21, 50], pl.page_tables).step(tok)
    for b, L in enumerate((64, 21, 50)):
        one = oracle.Oracle(TINY, t, [L], pl.page_tables[b:b + 1]).step([tok[b]])
        assert np.array_equal(both["logits"][b], one["logits"][0])


def test_identical_experts_equal_dense_mlp():
    t, pl = tiny_inputs()
    F, d = TINY.d_ffn, TINY.d_model
    t2 = dict(t)
    for l in range(TINY.n_layers):
        for kind in ("wg", "wu", "wd"):
            a = t[f"l{l}.{kind}"]
            t2[f"l{l}.{kind}"] = np.ascontiguousarray(np.broadcast_to(a[:1], a.shape))
    r = oracle.Oracle(TINY, t2, [64], pl.page_tables).step([17], dumps=("n", "moe"))
    for l in range(TINY.n_layers):
        p = f"l{l}."
        y = oracle.expert(r["n"][l, 0], t2[p + "wg"][0], t2[p + "wu"][0], t2[p + "wd"][0])
        moe = to_f32(r["moe"][l, 0]).astype(np.float64)
        dense = rnd(y)
        assert np.all(np.abs(moe - dense) <= np.abs(dense) * 2 ** -7 + 1e-7)


def test_router_bias_forces_expert():
    t, pl = tiny_inputs()
    bias = [np.zeros(TINY.n_experts, np.float32) for _ in range(TINY.n_layers)]
    bias[1][6] = 100.0
    r = oracle.Oracle(TINY, t, [64], pl.page_tables, router_biases=bias).step([17])
    assert r["route_ids"][1, 0, 0] == 6
    assert r["route_w"][1, 0, 0] == pytest.approx(1.0, abs=1e-6)


def test_forced_routing_adoption_rules():
    t, pl = tiny_inputs()
    base = oracle.Oracle(TINY, t, [64], pl.page_tables).step([17], dumps=("router_logits",))
    ids = base["route_ids"]
    # The oracle's own choice is always accepted.
    same = oracle.Oracle(TINY, t, [64], pl.page_tables).step([17], forced_ids=ids)
    assert same["route_mismatch"] == 0 and np.array_equal(same["logits"], base["logits"])
    # A different choice away from a near tie is rejected.
    bad = ids.copy()
    r = base["router_logits"][0, 0]
    worst = int(np.argmin(r))
    bad[0, 0, -1] = worst
    rej = oracle.Oracle(TINY, t, [64], pl.page_tables).step([17], forced_ids=bad)
    assert rej["route_mismatch"] == 1
    assert np.array_equal(rej["logits"], base["logits"])
    # With a huge tie tolerance the other choice is adopted (and changes the step).
    acc = oracle.Oracle(TINY, t, [64], pl.page_tables).step([17], forced_ids=bad, tie_eps=1e3)
    assert acc["route_mismatch"] == 0
    assert sorted(acc["route_ids"][0, 0].tolist()) == sorted(bad[0, 0].tolist())


# ------------------------------------------------------ teacher-forced entry points


def test_layer_by_layer_replay_equals_the_step_bit_exact():
    """orc_layer_step (keeping the K/V rows) over every layer, orc_head and
    orc_advance reproduce orc_step exactly, over two steps of a ragged batch;
    a teacher-forced evaluation with keep=False in between changes nothing."""
    lens = [29, 3]
    t, pl = tiny_inputs(dims=ODD, seq_lens=lens, reserve=3)
    ref = oracle.Oracle(ODD, t, lens, pl.page_tables)
    rep = oracle.Oracle(ODD, t, lens, pl.page_tables)
    emb = t["embed"]
    rng = np.random.default_rng(5)
    tok = [7, 250]
    for _ in range(2):
        r = ref.step(tok, dumps=("h", "o"))
        noise = to_bits(rng.standard_normal((2, ODD.d_model)))
        for l in range(ODD.n_layers):
            rep.layer(l, noise, keep=False)  # must leave the state alone
        h = emb[np.asarray(tok)]
        for l in range(ODD.n_layers):
            assert np.array_equal(h, r["h"][l])
            y = rep.layer(l, h, keep=True, dumps=("o",))
            assert np.array_equal(y["o"], r["o"][l])
            assert np.array_equal(y["route_ids"], r["route_ids"][l])
            h = y["h_out"]
        assert np.array_equal(h, r["h"][ODD.n_layers])
        hd = rep.head(h)
        rep.advance()
        assert np.array_equal(hd["logits"], r["logits"])
        assert np.array_equal(hd["next_tokens"], r["next_tokens"])
        tok = r["next_tokens"]


def test_teacher_forced_layer_matches_brute_force_from_a_foreign_residual():
    """One layer from a residual the model never produced (bf16 ~N(0, 1)),
    against the float64 brute force's same layer: every output element within
    one bf16 ulp (the double-sum oracle differs only where a sum lands within
    rounding of a bf16 tie), routing identical where the margin is clear."""
    lens = [29, 3]
    t, pl = tiny_inputs(dims=ODD, seq_lens=lens, reserve=3)
    orc = oracle.Oracle(ODD, t, lens, pl.page_tables, accum_double=True)
    bf = BruteForce(ODD, t, lens, pl.page_tables)
    rng = np.random.default_rng(11)
    for l in range(ODD.n_layers):
        h = to_bits(rng.standard_normal((2, ODD.d_model)))
        y = orc.layer(l, h)
        for b in range(2):
            bf_lens = list(bf.lens)
            hb, top = bf.layer(l, b, to_f32(h[b]).astype(np.float64))
            bf.K[l][b], bf.V[l][b] = bf.K[l][b][:-1], bf.V[l][b][:-1]  # teacher-forced: no append
            bf.lens = bf_lens
            got = to_f32(y["h_out"][b]).astype(np.float64)
            assert np.all(np.abs(got - hb) <= ulp(hb)), (l, b, np.abs(got - hb).max())
            if y["route_margin"][b] > 1e-2:
                assert np.array_equal(np.sort(y["route_ids"][b]), np.sort(top))


def test_reset_slot_equals_a_fresh_state_and_leaves_other_slots():
    """Continuous batching: after two steps, slot 1 gets a new sequence (new
    length, pages of its own).  Its next step equals a fresh state holding
    just that sequence; slot 0 continues exactly as if nothing happened."""
    lens = [29, 3, 40]
    t, pl = tiny_inputs(dims=ODD, seq_lens=lens, reserve=4)
    cont = oracle.Oracle(ODD, t, lens[:2], pl.page_tables[:2])
    ref0 = oracle.Oracle(ODD, t, lens[:1], pl.page_tables[:1])
    tok = [7, 250]
    for _ in range(2):
        r = cont.step(tok)
        ref0.step(tok[:1])
        tok = list(r["next_tokens"])
    cont.reset_seq(1, lens[2], pl.page_tables[2])
    tok[1] = 123
    r = cont.step(tok)
    fresh = oracle.Oracle(ODD, t, [lens[2]], pl.page_tables[2:3]).step([123])
    assert np.array_equal(r["logits"][1], fresh["logits"][0])
    assert np.array_equal(r["logits"][0], ref0.step(tok[:1])["logits"][0])
