"""mk_decode_step_static: the decode step for callers that cannot allocate.

Callers whose device memory is all owned by an arena or caching allocator
(or that run under a memory budget already handed out) cannot use mk_create,
which allocates a workspace.  mk_decode_step_static runs the same kernel with
its scratch in a static device array.  These tests call it through the C ABI
and check it against the context-based mk_decode_step on the same inputs:
both run the same kernel on the same task table (the context's schedule is
rebuilt for each step's lengths), so logits and next tokens must be
identical bit for bit, on two calls in a row.  The file is named to be
collected last.
"""
import numpy as np
import pytest

import persistent_moe_decode_sm_gb300 as mk
import synth

pytestmark = pytest.mark.gpu


def _compare_two_steps(dims, lens):
    import torch

    inp = synth.device_inputs(dims, lens, 4)
    pl = inp.layout
    dec = mk.Decoder(dims, inp.tensors, pl.num_pages, pl.max_pages, len(lens),
                     inp.bias_tensors)
    B, V = len(lens), dims.vocab
    tok = torch.tensor(synth.first_tokens(dims, B), dtype=torch.int32, device="cuda")
    for step in range(2):
        cur = [L + step for L in lens]
        dec.build_schedule(cur, pl.page_tables)
        ref_logits = torch.zeros(B, V, device="cuda")
        ref_next = torch.zeros(B, dtype=torch.int32, device="cuda")
        dec.decode_step(tok, ref_logits, ref_next)
        dec.sync()
        st_logits = torch.full((B, V), float("nan"), device="cuda")
        st_next = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        mk.mk_decode_step_static(dec.cdims, dec.weights, B, cur, pl.page_tables, tok,
                                 st_logits, st_next)
        a, b = st_logits.cpu().numpy(), ref_logits.cpu().numpy()
        assert np.all(np.isfinite(a))
        assert np.array_equal(a, b), (step, float(np.abs(a - b).max()))
        assert np.array_equal(st_next.cpu().numpy(), ref_next.cpu().numpy())
        tok = ref_next.clone()
    dec.close()


def test_static_scratch_step_matches_context_step_twice():
    _compare_two_steps(synth.TINY, [40, 7])


def test_static_step_with_other_dims_after_a_context_of_the_same_batch_bucket():
    """A context of one model (tiny) runs first; a static call of another
    model (mid, whose shared-memory plan differs) at the same batch bucket
    must still launch and agree with its own context."""
    import torch

    inp = synth.device_inputs(synth.TINY, [12], 2)
    pl = inp.layout
    dec = mk.Decoder(synth.TINY, inp.tensors, pl.num_pages, pl.max_pages, 1, inp.bias_tensors)
    dec.build_schedule([12], pl.page_tables)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    dec.decode_step(tok, None, nxt)
    dec.sync()
    dec.close()
    _compare_two_steps(synth.MID, [300])


def test_static_scratch_rejects_oversized_workloads():
    """A page table of 600,000 entries per sequence needs more than the
    16 MiB of static scratch (batch slots x entries x 4 bytes): the call
    refuses before launching anything."""
    import torch

    dims, lens = synth.TINY, [40]
    inp = synth.device_inputs(dims, lens, 2)
    pl = inp.layout
    t = inp.tensors
    layers = [{c: t[f"l{l}.{n}"] for c, n in mk.Decoder.LAYER_FIELDS.items()}
              for l in range(dims.n_layers)]
    weights = mk.Weights(t["embed"], layers, t["final_norm"], t["lm_head"])
    mp = 600_000
    pt = np.full((1, mp), -1, np.int32)
    pt[0, :pl.max_pages] = pl.page_tables[0]
    cd = mk.make_dims(dims.n_layers, dims.d_model, dims.n_q_heads, dims.n_kv_heads,
                      dims.head_dim, dims.n_experts, dims.top_k, dims.d_ffn, dims.vocab,
                      dims.page_size, 1, pl.num_pages, mp)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    with pytest.raises(mk.MkError) as e:
        mk.mk_decode_step_static(cd, weights, 1, lens, pt, tok, None, nxt)
    assert e.value.code == mk.MK_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert int(nxt.item()) == -5  # nothing ran
