"""GPU-vs-oracle parity harness (used by the gpu tests and by smoke()).

The GPU side runs through the C ABI (persistent_moe_decode_sm_gb300); the
oracle side is the CPU reference in oracle/ with exact (double) sums and the
method's bf16 rounding points.  Both read the same seeded inputs from synth/.

Two comparisons per step:

Teacher-forced, layer by layer (always).  For every layer l the oracle
evaluates layer l from the GPU's own residual entering it (h_l, dumped by the
library) under the GPU's routing (adopted only at near ties, see below), and
the GPU's residual entering layer l + 1 must agree with the oracle's within
bf16 rounding: every element within 2 * (ulp(h) + ulp(attn) + ulp(moe)) of
the oracle's values (one rounding flip in each of the three roundings that
make the residual) plus one bf16 ulp of the typical size of attn and moe, at
most TF_FRAC_CHANGED of the elements changed at all, relative L2 at most
TF_REL_L2.  The attention output o of every layer is held to two ulps of
each element plus one ulp of the row's rms, the routing must match wherever the oracle's top-k
margin exceeds TIE_EPS, and the logits that the oracle's LM head makes from
the GPU's final residual must agree with the GPU's logits within the stated
max-abs / relative-L2 bound.  This comparison is not chaotic: both sides see
the same input at every layer, so it holds at any depth, batch and context.

Free-running, end to end (ParityRun(free_steps=N) for the first N steps).
The oracle runs the whole step from the token alone, keeping its own KV rows,
adopting the GPU's routing only at (layer, token) pairs whose top-k margin is
below TIE_EPS and only where the two choices differ among experts within
TIE_EPS of the k-th logit (anything else is a routing mismatch and fails);
its logits must agree with the GPU's within the case's fixed bound (the
stated 3e-2 / 1e-2 unless the test names another, derived bound).  The
greedy token must be identical where the oracle's top-1/top-2 margin exceeds
TIE_EPS, else the GPU's token must be within TIE_EPS of the oracle's
maximum; both continue with the GPU's token.  After the free-running steps
the oracle's state advances by the teacher-forced replay (its own K/V rows
computed from the GPU's residuals).
"""
from __future__ import annotations

import os
import sys
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)

import oracle  # noqa: E402
import persistent_moe_decode_sm_gb300 as mk  # noqa: E402
import synth  # noqa: E402
from bf16util import to_f32, ulp  # noqa: E402

# The parity bar: router ids and greedy tokens bit-exact wherever the
# oracle's margin exceeds 1e-2; logits max-abs 3e-2 and relative L2 1e-2.
TIE_EPS = 1e-2
LOGIT_MAX_ABS = 3e-2
LOGIT_REL_L2 = 1e-2
STATED_BOUND = (LOGIT_MAX_ABS, LOGIT_REL_L2)
# Teacher-forced layer bounds.  Two faithful fp32 evaluations of a layer
# (the oracle's two summation orders) from the same residual differ from the
# exact one in at most ~1.4 % of the residual's elements, relative L2 <=
# 2e-4, each element by at most one rounding flip of h, attn or moe
# (measured on the tiny, mid and full-scale models).  The quantitative
# criteria are the per-element bound and the relative L2; the changed
# fractions only catch an error spread over every element.  A few flipped
# attention outputs move thousands of residual sums across a rounding
# boundary when the attention width is small (mid, Hq*D = 1024: up to 27 %
# of attn and 23 % of moe elements one flip off, measured on the GPU), so the
# residual's bound is 35 %; the attention outputs of a layer, where a flip
# stays within its head, are held to 10 %.
TF_FRAC_CHANGED = 0.35
TF_O_FRAC_CHANGED = 0.10
TF_REL_L2 = 2e-3

# Free-running bound of the 8-layer mid model.  Faithful fp32 evaluations of
# the method (the oracle's two summation orders) deviate from the exact
# evaluation by 0.024-0.041 max-abs and 0.009-0.0155 relative L2 at 124 of
# the 128 greedy steps of that workload (measured on the CPU; at the other 4
# steps the drift flips a router choice whose margin exceeds 1e-2), so the
# stated 3e-2 / 1e-2 sits below the method's own fp32 noise there; the bound
# is 1.5x that floor, rounded up.
MID_FREE_BOUND = (6e-2, 2.4e-2)
# Free-running bound of the full-width model cut to 4 layers.  Faithful fp32
# evaluations reach max-abs 0.032 (batch 1, 8192 cached), 0.044 (batch 8,
# ragged, Zipf skew) and 0.031 (batch 2, 131072 cached) over 152,064 x batch
# logits, relative L2 at most 0.0077; the bound is 1.5x that, rounded up.
FULL4_FREE_BOUND = (7e-2, 1.2e-2)

# d, F and Hq*D multiples of 64, head_dim 32, group 3: an odd small shape
ODD = synth.Dims(2, 192, 6, 2, 32, 6, 2, 128, 300)

SMALL = {"tiny": synth.TINY, "mid": synth.MID, "odd": ODD, "full": synth.FULL}


def f64(bits) -> np.ndarray:
    return to_f32(bits).astype(np.float64)


def layer_check(gpu_next, gpu_o, gpu_ids, y, gpu_attn=None, gpu_moe=None) -> Dict[str, float]:
    """One teacher-forced layer: the GPU's residual entering the next layer
    and attention output against the oracle's layer evaluation y from the
    GPU's own input (oracle.Oracle.layer with dumps o, attn, moe)."""
    def rms(x):
        return np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-60)

    g, o = f64(gpu_next), f64(y["h_out"])
    at, mo = f64(y["attn"]), f64(y["moe"])
    d = np.abs(g - o)
    # one rounding flip in each of h, attn and moe, twice over, plus one bf16
    # ulp at the typical size of attn and moe (what an upstream flip moves a
    # near-zero element by)
    lim = 2.0 * (ulp(o) + ulp(at) + ulp(mo)) + 2.0 ** -8 * (rms(at) + rms(mo))
    go, oo = f64(gpu_o), f64(y["o"])
    do = np.abs(go - oo)
    # two ulps of the element plus 2^-5 of its row's rms: a flipped query
    # element moves every score of its head, and 1-3 flipped elements move
    # the head's outputs by up to 1.3 % of the row's rms at 1K-16K keys
    # (measured with the oracle), near-zero outputs by many of their own ulps
    lim_o = 2.0 * ulp(oo) + 2.0 ** -5 * rms(oo)
    clear = y["route_margin"] > TIE_EPS
    same = np.all(np.sort(gpu_ids, -1) == np.sort(y["route_ids"], -1), -1)
    extra = {}
    if gpu_attn is not None:
        extra["attn_frac"] = float(np.mean(gpu_attn != y["attn"]))
        extra["moe_frac"] = float(np.mean(gpu_moe != y["moe"]))
    return {**extra, "h_ratio": float((d / lim).max()), "h_frac": float(np.mean(d > 0)),
            "h_rel": float(np.linalg.norm(d) / max(np.linalg.norm(o), 1e-30)),
            "o_ratio": float((do / lim_o).max()), "o_frac": float(np.mean(do > 0)),
            "route_mismatch": int(y["route_mismatch"]),
            "route_clear_mismatch": int((clear & ~same).sum())}


def layers_ok(s: Dict[str, float]) -> bool:
    return (s["h_ratio"] <= 1.0 and s["h_frac"] <= TF_FRAC_CHANGED and s["h_rel"] <= TF_REL_L2
            and s["o_ratio"] <= 1.0 and s["o_frac"] <= TF_O_FRAC_CHANGED
            and s["route_mismatch"] == 0 and s["route_clear_mismatch"] == 0)


def logit_stats(gl: np.ndarray, ol: np.ndarray) -> Tuple[float, float]:
    return (float(np.abs(gl - ol).max()),
            float(np.linalg.norm(gl - ol) / max(np.linalg.norm(ol), 1e-30)))


def token_ok(gn, ol, next_tokens, margin) -> bool:
    ok = True
    for b in range(len(gn)):
        if margin[b] > TIE_EPS:
            ok &= int(gn[b]) == int(next_tokens[b])
        else:
            ok &= float(ol[b, gn[b]]) >= float(ol[b].max()) - TIE_EPS
    return bool(ok)


class ParityRun:
    """One GPU decoder and one exact oracle on the same seeded inputs.

    free_steps: how many of the first steps also run the free-running
    end-to-end comparison (None: every step).  bound: the free-running logit
    bound (max-abs, relative L2)."""

    def __init__(self, dims="tiny", seq_lens: Optional[Sequence[int]] = None, reserve_steps=9,
                 zipf_s=None, max_batch=None, materialise=None, seed=0, tokens=None,
                 free_steps: Optional[int] = None, bound: Tuple[float, float] = STATED_BOUND,
                 layout_lens: Optional[Sequence[int]] = None):
        import torch

        self.torch = torch
        if isinstance(dims, str):
            if seq_lens is None:
                wl = synth.workloads()
                seq_lens = wl[dims].seq_lens if dims in wl else [64]
            dims = SMALL[dims]
        self.dims = dims
        self.seq_lens = list(seq_lens)
        self.B = len(self.seq_lens)
        self.free_steps = free_steps
        self.bound = bound
        self.n_steps = 0
        if materialise is None:
            materialise = synth.weight_bytes_total(dims) < 2e9
        # layout_lens: allocate pages for more sequences than are scheduled
        # (the spare ones replace finished sequences later)
        self.dev = synth.device_inputs(dims, list(layout_lens or self.seq_lens), reserve_steps,
                                       zipf_s, seed)
        pl = self.dev.layout
        self.page_tables = pl.page_tables[:self.B]
        self.dec = mk.Decoder(dims, self.dev.tensors, pl.num_pages, pl.max_pages,
                              max_batch or self.B, self.dev.bias_tensors)
        self.dec.build_schedule(self.seq_lens, self.page_tables)
        self.host = synth.host_inputs(dims, pl, seed, materialise=materialise)
        self.seed = seed
        # two exact oracle states: `tf` follows the GPU (each step replayed
        # teacher-forced from the GPU's residuals, keeping the K/V rows that
        # makes), `orc` runs free from the tokens alone
        self.tf = oracle.Oracle(dims, self.host, self.seq_lens, self.page_tables,
                                self.dev.biases, accum_double=True, seed=seed)
        self.orc = oracle.Oracle(dims, self.host, self.seq_lens, self.page_tables,
                                 self.dev.biases, accum_double=True, seed=seed)
        self.tokens = (np.asarray(tokens, np.int32) if tokens is not None
                       else synth.first_tokens(dims, self.B, seed))
        self.cur_lens = list(self.seq_lens)
        self.alloc_io(self.B)

    def replace(self, slot: int, new_len: int, page_row, token: int) -> None:
        """Continuous batching: `slot` gets a new sequence of new_len cached
        tokens held in the pages of page_row, whose first token is `token`;
        the library's schedule is rebuilt for the new membership, the
        oracle's slot is reset, the other sequences continue."""
        self.cur_lens[slot] = int(new_len)
        pt = np.array(self.page_tables, copy=True)
        pt[slot] = page_row
        self.page_tables = pt
        self.dec.build_schedule(self.cur_lens, self.page_tables)
        self.orc.reset_seq(slot, new_len, page_row)
        self.tf.reset_seq(slot, new_len, page_row)
        self.tokens = np.array(self.tokens, copy=True)
        self.tokens[slot] = token

    def reset_oracle(self, seq_lens, page_tables):
        """A new oracle state for a new batch (continuous batching)."""
        self.orc = oracle.Oracle(self.dims, self.host, seq_lens, page_tables, self.dev.biases,
                                 accum_double=True, seed=self.seed)
        self.tf = oracle.Oracle(self.dims, self.host, seq_lens, page_tables, self.dev.biases,
                                accum_double=True, seed=self.seed)
        self.cur_lens = list(seq_lens)
        self.page_tables = np.asarray(page_tables, np.int32)

    def alloc_io(self, B):
        torch = self.torch
        self.B = B
        self.tok_d = torch.zeros(B, dtype=torch.int32, device="cuda")
        self.next_d = torch.zeros(B, dtype=torch.int32, device="cuda")
        self.logits_d = torch.zeros(B, self.dims.vocab, dtype=torch.float32, device="cuda")

    def step(self) -> Dict:
        torch = self.torch
        L = self.dims.n_layers
        self.tok_d.copy_(torch.from_numpy(self.tokens))
        self.dec.decode_step(self.tok_d, self.logits_d, self.next_d)
        self.dec.sync()
        gpu_ids, gpu_w = self.dec.routing()
        gh, go = self.dec.dump_h(), self.dec.dump_o()
        ga, gm = self.dec.dump_attn_moe()
        gl = self.logits_d.cpu().numpy()
        gn = self.next_d.cpu().numpy()
        free = self.free_steps is None or self.n_steps < self.free_steps
        rep: Dict = {"step": self.n_steps, "free_running": free}
        # embedding rows: the GPU's h[0] must be the embedding of the tokens
        emb_ok = np.array_equal(gh[0], np.stack([self._embed_row(t) for t in self.tokens]))
        # teacher-forced, layer by layer
        worst = {"h_ratio": 0.0, "h_frac": 0.0, "h_rel": 0.0, "o_ratio": 0.0, "o_frac": 0.0,
                 "attn_frac": 0.0, "moe_frac": 0.0, "route_mismatch": 0, "route_clear_mismatch": 0}
        per_layer = []
        for l in range(L):
            y = self.tf.layer(l, gh[l], forced_ids=gpu_ids[l], tie_eps=TIE_EPS, keep=True,
                              dumps=("o", "attn", "moe"))
            s = layer_check(gh[l + 1], go[l], gpu_ids[l], y, ga[l], gm[l])
            per_layer.append(s)
            for k in worst:
                worst[k] = max(worst[k], s[k]) if isinstance(worst[k], float) else worst[k] + s[k]
        hd = self.tf.head(gh[L])
        self.tf.advance()
        rep["tf"] = worst
        rep["tf_layers_over"] = [(l, s) for l, s in enumerate(per_layer) if not layers_ok(s)][:6]
        rep["tf_worst_layer"] = int(np.argmax([s["h_ratio"] for s in per_layer]))
        rep["tf_logits"] = logit_stats(gl, hd["logits"])
        rep["tf_token_ok"] = token_ok(gn, hd["logits"], hd["next_tokens"], hd["argmax_margin"])
        rep["embed_ok"] = bool(emb_ok)
        if free:
            r = self.orc.step(self.tokens, forced_ids=gpu_ids, tie_eps=TIE_EPS)
            ol = r["logits"]
            rep["max_abs"], rep["rel_l2"] = logit_stats(gl, ol)
            rep["bound_max_abs"], rep["bound_rel_l2"] = self.bound
            rep["route_mismatch"] = int(r["route_mismatch"])
            clear = r["route_margin"] > TIE_EPS
            same = np.all(np.sort(gpu_ids, -1) == np.sort(r["route_ids"], -1), axis=-1)
            rep["route_clear_mismatch"] = int((clear & ~same).sum())
            rep["route_w_max_err"] = float(np.abs(np.sort(gpu_w, -1) -
                                                  np.sort(r["route_w"], -1)).max())
            rep["token_ok"] = token_ok(gn, ol, r["next_tokens"], r["argmax_margin"])
            rep["oracle_token"] = r["next_tokens"].tolist()
        rep["gpu_token"] = gn.tolist()
        self.tokens = gn.astype(np.int32)
        self.cur_lens = [L + 1 for L in self.cur_lens]
        self.n_steps += 1
        return rep

    def _embed_row(self, tok: int) -> np.ndarray:
        e = self.host["embed"]
        if isinstance(e, np.ndarray):
            return e[int(tok)]
        d = self.dims.d_model
        return synth.normal_bf16(self.seed, e.tid, e.sigma, d, int(tok) * d)

    @staticmethod
    def summary(rep: Dict) -> Dict:
        return {k: v for k, v in rep.items()
                if not isinstance(v, list) or (k == "tf_layers_over" and v)}

    @staticmethod
    def ok(rep: Dict) -> bool:
        good = (rep["embed_ok"] and layers_ok(rep["tf"]) and rep["tf_token_ok"]
                and rep["tf_logits"][0] <= LOGIT_MAX_ABS and rep["tf_logits"][1] <= LOGIT_REL_L2)
        if rep["free_running"]:
            good = good and (rep["route_mismatch"] == 0 and rep["route_clear_mismatch"] == 0
                             and rep["max_abs"] <= rep["bound_max_abs"]
                             and rep["rel_l2"] <= rep["bound_rel_l2"] and rep["token_ok"])
        return bool(good)

    def close(self):
        self.dec.close()
