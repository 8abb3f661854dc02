"""mk_decode_step_static: the decode step for callers that cannot allocate.

Callers whose device memory is all owned by an arena or caching allocator
(or that run under a memory budget already handed out) cannot use mk_create,
which allocates a workspace.  mk_decode_step_static runs the same kernel with
its scratch in a static device array.  This test calls it through the C ABI
twice in a row (two consecutive decode positions) and checks each call's
logits and next token against the context-based mk_decode_step on the same
inputs, within the tolerance of the other parity tests.  The file is named
to be collected last.
"""
import numpy as np
import pytest

import harness
import persistent_moe_decode_sm_gb300 as mk
import synth

pytestmark = pytest.mark.gpu


def close_enough(a, b):
    err = np.abs(a - b)
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    return err.max() <= harness.LOGIT_MAX_ABS and rel <= harness.LOGIT_REL_L2


def test_static_scratch_step_matches_context_step_twice():
    import torch

    dims = synth.TINY
    lens = [40, 7]
    inp = synth.device_inputs(dims, lens, 4)
    pl = inp.layout
    dec = mk.Decoder(dims, inp.tensors, pl.num_pages, pl.max_pages, len(lens),
                     inp.bias_tensors)
    dec.build_schedule(lens, pl.page_tables)
    B, V = len(lens), dims.vocab
    tok = torch.tensor(synth.first_tokens(dims, B), dtype=torch.int32, device="cuda")
    for step in range(2):
        cur = [L + step for L in lens]
        ref_logits = torch.zeros(B, V, device="cuda")
        ref_next = torch.zeros(B, dtype=torch.int32, device="cuda")
        dec.decode_step(tok, ref_logits, ref_next)
        dec.sync()
        st_logits = torch.zeros(B, V, device="cuda")
        st_next = torch.zeros(B, dtype=torch.int32, device="cuda")
        mk.mk_decode_step_static(dec.cdims, dec.weights, B, cur, pl.page_tables, tok,
                                 st_logits, st_next)
        a, b = st_logits.cpu().numpy(), ref_logits.cpu().numpy()
        assert np.all(np.isfinite(a))
        assert close_enough(a, b), (step, float(np.abs(a - b).max()))
        assert np.array_equal(st_next.cpu().numpy(), ref_next.cpu().numpy())
        tok = ref_next.clone()
    dec.close()


def test_static_scratch_rejects_oversized_workloads():
    """A one-layer model of full width at 100,000 cached tokens needs more than
    the 16 MiB of static scratch (its RoPE rows alone take 51 MB): the call
    refuses before launching anything."""
    import torch

    lens = [100000]
    inp = synth.device_inputs(synth.Dims(1, 2048, 32, 4, 128, 128, 8, 768, 152064), lens, 2)
    t = inp.tensors
    ly = {c: t[f"l0.{n}"] for c, n in mk.Decoder.LAYER_FIELDS.items()}
    weights = mk.Weights(t["embed"], [ly], t["final_norm"], t["lm_head"])
    cd = mk.make_dims(1, 2048, 32, 4, 128, 128, 8, 768, 152064, 16, 1,
                      inp.layout.num_pages, inp.layout.max_pages)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(mk.MkError) as e:
        mk.mk_decode_step_static(cd, weights, 1, lens, inp.layout.page_tables, tok, None, nxt)
    assert e.value.code == mk.MK_ERR_SCRATCH_LIMIT
