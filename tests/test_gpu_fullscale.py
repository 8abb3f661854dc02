"""Full-size parity on the GPU (needs a GB300 and ~70 GB of device memory).

The full-scale synthetic model is chaotic in depth: with bf16 rounding at
every layer, two correct evaluations that differ only in fp32 summation
order (the oracle's own fp32 and exact-sum modes, for instance) drift apart
by ~1% in the residual stream within 8 layers, flip near-tied experts soon
after, and decorrelate by layer ~12.  So the end-to-end parity bar is
applied at full width, context, vocabulary and batch with the depth cut to
4 layers (the first 4 layers of the full model: same tensor ids), and the
48-layer step is checked layer by layer over its first layers plus
properties of its output.
"""
import numpy as np
import pytest

import harness
import synth

pytestmark = pytest.mark.gpu

FULL4 = synth.Dims(4, 2048, 32, 4, 128, 128, 8, 768, 152064)


def run_steps(run, n):
    for _ in range(n):
        rep = run.step()
        print({k: v for k, v in rep.items() if not isinstance(v, list)})
        assert run.ok(rep), rep


def test_full_width_batch1_8k_context():
    run = harness.ParityRun(FULL4, seq_lens=[8192], reserve_steps=4, materialise=False)
    run_steps(run, 2)
    run.close()


def test_full_width_batch8_ragged_zipf():
    lens = synth.workloads()["full_b8"].seq_lens
    run = harness.ParityRun(FULL4, seq_lens=lens, reserve_steps=3, zipf_s=1.1,
                            materialise=False)
    run_steps(run, 2)
    st = run.dec.stats()
    assert st.sum_experts < 2 * 4 * 64  # Zipf skew: fewer distinct experts than B*k per layer
    run.close()


@pytest.mark.parametrize("lens", [[262144], [131072, 131072]], ids=["b1_262k", "b2_131k"])
def test_full_width_long_context(lens):
    run = harness.ParityRun(FULL4, seq_lens=lens, reserve_steps=3, materialise=False)
    run_steps(run, 1)
    run.close()


def test_full_depth_first_layers_and_output_properties():
    """48 layers at batch 1, 8192 cached tokens: the residual entering layers
    1..4 within 1% (relative L2) of the exact-sum oracle, routing of layers
    0..3 identical where the margin exceeds 1e-2, finite logits whose argmax
    is the returned token."""
    run = harness.ParityRun("full", reserve_steps=3, materialise=False, noise_floor=False)
    rep_h = None
    torch = run.torch
    run.tok_d.copy_(torch.from_numpy(run.tokens))
    run.dec.decode_step(run.tok_d, run.logits_d, run.next_d)
    run.dec.sync()
    gpu_ids, _ = run.dec.routing()
    gh = synth.bf16_bits_to_f32(run.dec.dump_h())
    gl = run.logits_d.cpu().numpy()
    gn = run.next_d.cpu().numpy()
    r = run.orc.step(run.tokens, forced_ids=gpu_ids, tie_eps=harness.TIE_EPS, dumps=("h",))
    oh = synth.bf16_bits_to_f32(r["h"])
    for l in range(1, 5):
        rel = np.linalg.norm(gh[l] - oh[l]) / np.linalg.norm(oh[l])
        assert rel < 1e-2, (l, rel)
    for l in range(4):
        clear = r["route_margin"][l] > harness.TIE_EPS
        same = np.all(np.sort(gpu_ids[l], -1) == np.sort(r["route_ids"][l], -1), -1)
        assert np.all(same | ~clear), l
    assert np.all(np.isfinite(gl))
    assert int(gn[0]) == int(np.argmax(gl[0]))
    run.close()
