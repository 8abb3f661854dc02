"""GPU-vs-oracle parity harness (used by the gpu tests and by smoke()).

The GPU side runs through the C ABI (persistent_moe_decode_sm_gb300); the
oracle side is the CPU reference in oracle/.  Both read the same seeded
inputs from synth/.  Per step:
  1. the GPU step runs; its routing is read back;
  2. the oracle runs the same step, adopting the GPU's routing only at an
     (layer, token) whose top-k margin is below TIE_EPS and only if the two
     choices differ among experts within TIE_EPS of the k-th logit;
     anything else is a routing mismatch (must be 0);
  3. logits must agree within LOGIT_MAX_ABS / LOGIT_REL_L2.  The reference
     is the oracle with exact (double) sums and the method's bf16 rounding
     points.  Two more oracle instances with plain fp32 sums -- ascending and
     descending summation order, both faithful to the method, which fixes
     fp32 accumulation but not the order -- run the same step with the same
     routing; the fp32 noise floor is the largest of their deviations from
     the exact evaluation and from each other, and where it approaches the
     stated bound (deep models, large batch x vocabulary) the bound becomes
     NOISE_FACTOR times that floor;
  4. the greedy token must be identical where the oracle's top-1/top-2
     margin exceeds TIE_EPS, else the GPU's token must be within TIE_EPS of
     the oracle's maximum; both continue with the GPU's token.
"""
from __future__ import annotations

import os
import sys
from typing import Dict, Optional, Sequence

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import persistent_moe_decode_sm_gb300 as mk  # noqa: E402
import synth  # noqa: E402

# The parity bar: router ids and greedy tokens bit-exact wherever the
# oracle's margin exceeds 1e-2; logits max-abs 3e-2 and relative L2 1e-2.
TIE_EPS = 1e-2
LOGIT_MAX_ABS = 3e-2
LOGIT_REL_L2 = 1e-2
# One step's fp32 noise is a single sample of a chaotic quantity (bf16
# rounding flips amplified layer by layer): on the 8-layer mid model the
# fp32 deviation from the exact evaluation went 0.0197 -> 0.0352 between
# consecutive steps, so the bound allows twice the floor measured on the step.
NOISE_FACTOR = 2.0

# d, F and Hq*D multiples of 64, head_dim 32, group 3: an odd small shape
ODD = synth.Dims(2, 192, 6, 2, 32, 6, 2, 128, 300)

SMALL = {"tiny": synth.TINY, "mid": synth.MID, "odd": ODD, "full": synth.FULL}


class ParityRun:
    def __init__(self, dims="tiny", seq_lens: Optional[Sequence[int]] = None, reserve_steps=9,
                 zipf_s=None, max_batch=None, materialise=None, seed=0, tokens=None,
                 accum_double=True, noise_floor=True):
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
        if materialise is None:
            materialise = synth.weight_bytes_total(dims) < 2e9
        self.dev = synth.device_inputs(dims, self.seq_lens, reserve_steps, zipf_s, seed)
        pl = self.dev.layout
        self.dec = mk.Decoder(dims, self.dev.tensors, pl.num_pages, pl.max_pages,
                              max_batch or self.B, self.dev.bias_tensors)
        self.dec.build_schedule(self.seq_lens, pl.page_tables)
        host = synth.host_inputs(dims, pl, seed, materialise=materialise)
        self.accum_double = accum_double
        self.orc = oracle.Oracle(dims, host, self.seq_lens, pl.page_tables, self.dev.biases,
                                 accum_double=accum_double, seed=seed)
        self.orc32 = (oracle.Oracle(dims, host, self.seq_lens, pl.page_tables, self.dev.biases,
                                    accum_double=False, seed=seed)
                      if noise_floor and accum_double else None)
        self.orc32r = (oracle.Oracle(dims, host, self.seq_lens, pl.page_tables, self.dev.biases,
                                     accum_double=False, seed=seed, reverse=True)
                       if noise_floor and accum_double else None)
        self.tokens = (np.asarray(tokens, np.int32) if tokens is not None
                       else synth.first_tokens(dims, self.B, seed))
        self.alloc_io(self.B)

    def reset_oracles(self, host, seq_lens, page_tables):
        """New oracle state(s) for a new batch (continuous batching)."""
        self.orc = oracle.Oracle(self.dims, host, seq_lens, page_tables, self.dev.biases,
                                 accum_double=self.accum_double)
        if self.orc32 is not None:
            self.orc32 = oracle.Oracle(self.dims, host, seq_lens, page_tables, self.dev.biases,
                                       accum_double=False)
            self.orc32r = oracle.Oracle(self.dims, host, seq_lens, page_tables, self.dev.biases,
                                        accum_double=False, reverse=True)

    def alloc_io(self, B):
        torch = self.torch
        self.B = B
        self.tok_d = torch.zeros(B, dtype=torch.int32, device="cuda")
        self.next_d = torch.zeros(B, dtype=torch.int32, device="cuda")
        self.logits_d = torch.zeros(B, self.dims.vocab, dtype=torch.float32, device="cuda")

    def step(self, dumps: bool = False) -> Dict:
        torch = self.torch
        self.tok_d.copy_(torch.from_numpy(self.tokens))
        self.dec.decode_step(self.tok_d, self.logits_d, self.next_d)
        self.dec.sync()
        gpu_ids, gpu_w = self.dec.routing()
        gl = self.logits_d.cpu().numpy()
        gn = self.next_d.cpu().numpy()
        r = self.orc.step(self.tokens, forced_ids=gpu_ids, tie_eps=TIE_EPS,
                          dumps=("h",) if dumps else ())
        ol = r["logits"]
        rep = {"max_abs": float(np.abs(gl - ol).max()),
               "rel_l2": float(np.linalg.norm(gl - ol) / max(np.linalg.norm(ol), 1e-30)),
               "route_mismatch": int(r["route_mismatch"])}
        rep["bound_max_abs"], rep["bound_rel_l2"] = LOGIT_MAX_ABS, LOGIT_REL_L2
        if self.orc32 is not None:
            a = self.orc32.step(self.tokens, forced_ids=gpu_ids, tie_eps=TIE_EPS)["logits"]
            b = self.orc32r.step(self.tokens, forced_ids=gpu_ids, tie_eps=TIE_EPS)["logits"]
            nol = max(np.linalg.norm(ol), 1e-30)
            diffs = (a - ol, b - ol, a - b)
            rep["noise_max_abs"] = float(max(np.abs(x).max() for x in diffs))
            rep["noise_rel_l2"] = float(max(np.linalg.norm(x) for x in diffs) / nol)
            rep["bound_max_abs"] = max(LOGIT_MAX_ABS, NOISE_FACTOR * rep["noise_max_abs"])
            rep["bound_rel_l2"] = max(LOGIT_REL_L2, NOISE_FACTOR * rep["noise_rel_l2"])
        clear = r["route_margin"] > TIE_EPS
        same = np.all(np.sort(gpu_ids, -1) == np.sort(r["route_ids"], -1), axis=-1)
        rep["route_clear"] = int(clear.sum())
        rep["route_clear_mismatch"] = int((clear & ~same).sum())
        rep["route_w_max_err"] = float(np.abs(np.sort(gpu_w, -1) - np.sort(r["route_w"], -1)).max())
        ok = True
        for b in range(self.B):
            if r["argmax_margin"][b] > TIE_EPS:
                ok &= int(gn[b]) == int(r["next_tokens"][b])
            else:
                ok &= float(ol[b, gn[b]]) >= float(ol[b].max()) - TIE_EPS
        rep["token_ok"] = bool(ok)
        rep["gpu_token"] = gn.tolist()
        rep["oracle_token"] = r["next_tokens"].tolist()
        rep["argmax_margin"] = r["argmax_margin"].tolist()
        if dumps:
            gh = self.dec.dump_h()
            rep["h_max_abs"] = [float(np.abs(synth.bf16_bits_to_f32(gh[l]) -
                                             synth.bf16_bits_to_f32(r["h"][l])).max())
                                for l in range(gh.shape[0])]
        self.tokens = gn.astype(np.int32)
        return rep

    @staticmethod
    def ok(rep: Dict) -> bool:
        return (rep["route_mismatch"] == 0 and rep["route_clear_mismatch"] == 0
                and rep["max_abs"] <= rep["bound_max_abs"]
                and rep["rel_l2"] <= rep["bound_rel_l2"] and rep["token_ok"])

    def close(self):
        self.dec.close()
