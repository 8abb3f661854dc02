"""The host task-table builder, checked on the CPU (no GPU needed).

A simulator executes each CTA's queue in order with the kernel's counter
semantics (wait on one count, signal one increment, last-ticket merges) and
checks that every step completes (no deadlock in randomised interleavings),
that every counter receives exactly the per-step increments the kernel is
told to expect, and that the tiles cover every weight row, every KV page and
every output row exactly once.
"""
import numpy as np
import pytest

import persistent_moe_decode_sm_gb300 as mk
import synth

OP_QKV, OP_ATTN, OP_UP, OP_OUT, OP_LM, OP_DOWN, OP_HEADER = 1, 3, 4, 5, 6, 7, 100


def cdims(d, max_batch, max_pages):
    return mk.make_dims(d.n_layers, d.d_model, d.n_q_heads, d.n_kv_heads, d.head_dim, d.n_experts,
                        d.top_k, d.d_ffn, d.vocab, d.page_size, max_batch, 100000, max_pages)


def decode(table):
    rows = []
    for r in table:
        assert r[0, 0] == OP_HEADER
        nl, nf = int(r[0, 1]), int(r[0, 2])
        rows.append((r[1:1 + nl], r[1 + nl:1 + nl + nf]))
    return rows


def simulate(d, info, rows, batch, rng):
    """Runs one step's worth of tasks; raises on deadlock."""
    L, Hkv = d.n_layers, d.n_kv_heads
    qkv_done = [0] * L
    router_done = [0] * L
    attn_ticket = {}
    group_ticket = {}
    attn_done = [0] * L
    up_done = [0] * L
    down_done = [0] * L
    out_done = [0] * L
    lm_ticket = [0]
    queues = [[(l, t) for l in range(L) for t in lt] + [(L, t) for t in ft] for lt, ft in rows]
    pos = [0] * len(queues)

    def ready(l, t):
        op = t[0]
        if op == OP_QKV:
            return l == 0 or out_done[l - 1] == info.n_out
        if op == OP_ATTN:
            return qkv_done[l] == info.n_qkv
        if op == OP_UP:  # every consumer takes the top-k from the complete logits
            return router_done[l] == info.n_router
        if op == OP_DOWN:  # the experts' activations are complete
            return router_done[l] == info.n_router and up_done[l] == info.n_up
        if op == OP_OUT:
            return (router_done[l] == info.n_router and attn_done[l] == batch * Hkv
                    and up_done[l] == info.n_up and down_done[l] == info.n_down)
        if op == OP_LM:
            return out_done[L - 1] == info.n_out
        raise AssertionError(op)

    def run(l, t):
        op = t[0]
        if op == OP_QKV:  # its router rows (first in the task), then q / k / v
            router_done[l] += int(t[5])
            qkv_done[l] += 1
        elif op == OP_ATTN:
            # two-level merge: the last split of a group merges the group,
            # the last group merger merges the groups
            key = (l, int(t[1]), int(t[2]))
            ng = int(t[11])
            if ng > 1:
                gkey = key + (int(t[9]),)
                group_ticket[gkey] = group_ticket.get(gkey, 0) + 1
                if group_ticket[gkey] != t[10]:
                    return
            attn_ticket[key] = attn_ticket.get(key, 0) + 1
            if attn_ticket[key] == (ng if ng > 1 else t[7]):
                attn_done[l] += 1
        elif op == OP_UP:
            up_done[l] += 1
        elif op == OP_DOWN:
            down_done[l] += 1
        elif op == OP_OUT:
            out_done[l] += 1
        elif op == OP_LM:
            lm_ticket[0] += 1

    remaining = sum(len(q) for q in queues)
    while remaining:
        progressed = False
        for c in rng.permutation(len(queues)):
            if pos[c] < len(queues[c]) and ready(*queues[c][pos[c]]):
                run(*queues[c][pos[c]])
                pos[c] += 1
                remaining -= 1
                progressed = True
        assert progressed, "deadlock: no CTA can run its next task"
    assert all(x == info.n_qkv for x in qkv_done)
    assert all(x == info.n_router for x in router_done)
    assert all(x == batch * Hkv for x in attn_done)
    assert all(x == info.n_up for x in up_done)
    assert all(x == info.n_down for x in down_done)
    assert all(x == info.n_out for x in out_done)
    assert lm_ticket[0] == info.n_lm


def check_coverage(d, info, rows, seq_lens):
    D, Hq, Hkv, P = d.head_dim, d.n_q_heads, d.n_kv_heads, d.page_size
    lt_all = [t for lt, _ in rows for t in lt]
    ft_all = [t for _, ft in rows for t in ft]
    for mat, n in ((0, Hq * D), (1, Hkv * D), (2, Hkv * D)):
        cov = np.zeros(n, int)
        for t in lt_all:
            if t[0] == OP_QKV and t[1] == mat:
                cov[t[2]:t[2] + t[3]] += 1
        assert np.all(cov == 1), mat
    cov = np.zeros(d.n_experts, int)
    for t in lt_all:
        if t[0] == OP_QKV:
            cov[t[4]:t[4] + t[5]] += 1
    assert np.all(cov == 1)
    slots = []
    slots2 = []
    for b, L in enumerate(seq_lens):
        npages = -(-L // P)
        for h in range(Hkv):
            sp = [t for t in lt_all if t[0] == OP_ATTN and t[1] == b and t[2] == h]
            assert len(sp) >= 1 and all(t[7] == len(sp) for t in sp)
            assert sum(int(t[8]) for t in sp) == 1
            cov = np.zeros(max(npages, 1), int)
            for t in sp:
                p1 = npages if t[4] < 0 else t[4]
                assert (t[4] < 0) == bool(t[8])
                cov[t[3]:p1] += 1
            assert np.all(cov[:npages] == 1)
            slot0 = {int(t[6]) for t in sp}
            assert len(slot0) == 1
            s0 = slot0.pop()
            assert sorted(int(t[5]) for t in sp) == list(range(s0, s0 + len(sp)))
            slots += [int(t[5]) for t in sp]
            # merge groups: consecutive slots, one group of all splits when
            # there are at most 16, else groups of 8
            ns = len(sp)
            grp = ns if ns <= 16 else 8
            ng = -(-ns // grp)
            g2 = {int(t[14]) for t in sp}
            assert len(g2) == 1
            g20 = g2.pop()
            for t in sp:
                gi = (int(t[5]) - s0) // grp
                assert int(t[9]) == gi and int(t[11]) == ng
                assert int(t[10]) == min(grp, ns - grp * gi) and int(t[12]) == s0 + grp * gi
                assert int(t[13]) == g20 + gi
            slots2.append((g20, ng))
    assert sorted(slots) == list(range(info.n_attn_slots))
    s2 = sorted(g + i for g, n in slots2 for i in range(n))
    assert s2 == list(range(len(s2)))  # level-2 slots distinct and dense
    ups = sorted((int(t[1]), int(t[2])) for t in lt_all if t[0] == OP_UP)
    assert ups == [(i, info.n_up) for i in range(info.n_up)]
    downs = sorted((int(t[1]), int(t[2])) for t in lt_all if t[0] == OP_DOWN)
    assert downs == [(i, info.n_down) for i in range(info.n_down)]
    cov = np.zeros(d.d_model, int)
    for t in lt_all:
        if t[0] == OP_OUT:
            assert 1 <= t[3] <= 64
            cov[t[2]:t[2] + t[3]] += 1
    assert np.all(cov == 1)
    cov = np.zeros(d.vocab, int)
    idx = []
    for t in ft_all:
        assert t[0] == OP_LM
        cov[t[2]:t[2] + t[3]] += 1
        idx.append(int(t[4]))
    assert np.all(cov == 1) and sorted(idx) == list(range(info.n_lm))


def phase_rank(t):
    return {OP_QKV: 0, OP_ATTN: 1, OP_UP: 2, OP_DOWN: 3, OP_OUT: 4}[int(t[0])]


CASES = [
    ("tiny", synth.TINY, 152, [64]),
    ("tiny_b8", synth.TINY, 152, [64, 0, 15, 16, 17, 100, 3, 31]),
    ("mid", synth.MID, 152, [2048]),
    ("full_b1_8k", synth.FULL, 152, [8192]),
    ("full_b1_8k_148sm", synth.FULL, 148, [8192]),
    ("full_b8_ragged", synth.FULL, 152, synth.workloads()["full_b8"].seq_lens),
    ("long_b1", synth.FULL, 152, [262144]),
    ("long_b2", synth.FULL, 152, [131072, 131072]),
    ("few_sms", synth.MID, 7, [300, 5]),
]


@pytest.mark.parametrize("name,d,n_sm,lens", CASES, ids=[c[0] for c in CASES])
def test_schedule_is_complete_and_deadlock_free(name, d, n_sm, lens):
    max_pages = max(-(-(L + 300) // d.page_size) for L in lens)
    info, table = mk.mk_plan(cdims(d, 8, max_pages), n_sm, len(lens), lens)
    assert info.n_cta == n_sm and table.shape == (n_sm, info.tasks_per_cta, 32)
    rows = decode(table)
    for lt, ft in rows:
        ranks = [phase_rank(t) for t in lt]
        assert ranks == sorted(ranks), "tasks of a layer must run in phase order"
    check_coverage(d, info, rows, lens)
    rng = np.random.default_rng(0)
    for _ in range(2 if d.n_layers > 8 else 4):
        simulate(d, info, rows, len(lens), rng)


def test_attention_splits_are_balanced():
    d = synth.FULL
    lens = synth.workloads()["full_b8"].seq_lens
    info, table = mk.mk_plan(cdims(d, 8, 1100), 152, 8, lens)
    pages = np.zeros(152)
    for c, (lt, _) in enumerate(decode(table)):
        for t in lt:
            if t[0] == OP_ATTN:
                npages = -(-lens[t[1]] // 16)
                p1 = npages if t[4] < 0 else t[4]
                pages[c] += p1 - t[3]
    total = sum(-(-L // 16) for L in lens) * d.n_kv_heads
    assert pages.sum() == total
    n_att = int((pages > 0).sum())  # the CTAs given attention splits
    assert pages.max() <= 1.25 * total / n_att + 2


def test_roles_balance_streamed_bytes():
    """Attention CTAs take no expert share and expert CTAs no attention
    split; the split weights the KV bytes by the attention stage's higher
    compute cost (1.5x a gate/up stage's, plus the merge), so an attention CTA streams
    somewhat fewer bytes than an expert CTA."""
    d = synth.FULL
    for lens in ([8192], [262144], synth.workloads()["full_b8"].seq_lens):
        info, table = mk.mk_plan(cdims(d, 8, 17000), 152, len(lens), lens)
        rows = decode(table)
        att = [c for c, (lt, _) in enumerate(rows) if any(t[0] == OP_ATTN for t in lt)]
        exp = [c for c, (lt, _) in enumerate(rows) if any(t[0] == OP_UP for t in lt)]
        assert not set(att) & set(exp) and len(att) + len(exp) == 152
        kv = sum(lens) * d.n_kv_heads * d.head_dim * 4 / len(att)
        e, k = d.n_experts, d.top_k
        u = e * (1 - (1 - k / e) ** len(lens))
        up = u * 2 * d.d_ffn * d.d_model * 2 / len(exp)
        assert 0.45 < kv / up < 1.1, (lens[:2], kv, up)


def test_router_rows_are_spread_and_lead_the_qkv_task():
    """The router rows are spread over the grid, at most ceil(E / n_cta) per
    CTA, and ride at the front of the CTA's first QKV task (so the routing
    every expert stage waits for is complete one norm and one short GEMV
    after the layer's input); the counter expects E rows per step."""
    d = synth.FULL
    for n_sm in (152, 148, 16, 7):
        info, table = mk.mk_plan(cdims(d, 8, 600), n_sm, 1, [8192])
        rows = decode(table)
        per = [sum(int(t[5]) for t in lt if t[0] == OP_QKV) for lt, _ in rows]
        assert sum(per) == d.n_experts and max(per) <= -(-d.n_experts // n_sm)
        assert info.n_router == d.n_experts
        for lt, _ in rows:
            qk = [t for t in lt if t[0] == OP_QKV]
            assert all(int(t[5]) == 0 for t in qk[1:])


def test_out_tasks_fit_the_per_task_row_cap():
    """OUT tasks take at most 32 rows of d (the kernel's per-warp down
    accumulators hold 32); with fewer CTAs than d / 32 the rows are cut into
    more tasks, and the tasks still cover d exactly once."""
    for d, n_sm in ((synth.FULL, 152), (synth.FULL, 16), (synth.FULL, 4)):
        info, table = mk.mk_plan(cdims(d, 1, 600), n_sm, 1, [8192])
        rows = decode(table)
        outs = [t for lt, _ in rows for t in lt if t[0] == OP_OUT]
        assert len(outs) == info.n_out
        assert all(1 <= int(t[3]) <= 32 for t in outs)
        cov = np.zeros(d.d_model, int)
        for t in outs:
            cov[t[2]:t[2] + t[3]] += 1
        assert np.all(cov == 1)


def test_stage_geometry_of_the_full_model():
    """The ring stages the shared-memory plan leaves the full-scale model:
    whole d-rows per stage (5 up to batch 4, 4 at batch 8, where the second
    run of a stage sits 64 bytes out of line), Wo rows of 4096, expert down
    rows of F, and the whole plan within the 227 KB a CTA may opt in to."""
    import ctypes
    d = synth.workloads()["full"].dims
    cd = cdims(d, 8, 1024)
    f = mk.lib().mk_stage_geometry
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(type(cd)), ctypes.c_int, ctypes.c_int,
                  ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                  ctypes.POINTER(ctypes.c_int64)]
    want_rows = {1: 5, 2: 5, 4: 5, 8: 4}
    for nb, rows_d in want_rows.items():
        sb, rows, dyn = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
        assert f(ctypes.byref(cd), nb, d.d_model, ctypes.byref(sb), ctypes.byref(rows), ctypes.byref(dyn))
        assert sb.value % 1024 == 0 and dyn.value <= 232448, (nb, sb.value, dyn.value)
        assert rows.value == rows_d, (nb, rows.value)
        gap = 64 if nb == 8 else 0
        assert rows.value * 2 * d.d_model + gap <= sb.value
        for K, least in ((d.n_q_heads * d.head_dim, 2), (d.d_ffn, 10)):
            assert f(ctypes.byref(cd), nb, K, ctypes.byref(sb), ctypes.byref(rows), None)
            assert rows.value >= least, (nb, K, rows.value)


@pytest.mark.parametrize("u_seen", [8.0, 24.0, 40.0, 64.0])
def test_schedule_from_observed_experts(u_seen):
    """The role split from an observed number of distinct experts per layer
    (a skewed router's batch of 8 picks fewer than the uniform 51.6): the
    table stays complete and deadlock-free, and fewer observed experts leave
    fewer CTAs on the expert side."""
    import ctypes
    d = synth.FULL
    lens = list(synth.workloads()["full_b8"].seq_lens)
    cd = cdims(d, 8, 17000)
    f = mk.lib().mk_plan_observed
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(type(cd)), ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                  ctypes.c_double, ctypes.POINTER(mk.mk_plan_info), ctypes.c_void_p,
                  ctypes.c_int64]
    sl = np.ascontiguousarray(lens, dtype=np.int32)

    def plan(u):
        info = mk.mk_plan_info()
        assert f(ctypes.byref(cd), 152, len(lens), sl.ctypes.data, u, ctypes.byref(info), None, 0) == 0
        table = np.empty((info.n_cta, info.tasks_per_cta, 32), np.int32)
        assert f(ctypes.byref(cd), 152, len(lens), sl.ctypes.data, u, ctypes.byref(info),
                 table.ctypes.data, table.size) == 0
        return info, table

    info, table = plan(u_seen)
    rows = decode(table)
    sim_d = d
    rng = np.random.default_rng(int(u_seen))
    simulate(sim_d, info, rows, len(lens), rng)
    check_coverage(sim_d, info, rows, lens)
    n_exp = sum(any(t[0] == OP_UP for t in lt) for lt, _ in rows)
    n_exp_uniform = sum(any(t[0] == OP_UP for t in lt) for lt, _ in decode(plan(0.0)[1]))
    if u_seen < 51.0:
        assert n_exp < n_exp_uniform, (u_seen, n_exp, n_exp_uniform)
