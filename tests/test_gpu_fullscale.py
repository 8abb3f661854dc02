"""Full-size parity on the GPU (needs a GB300 and ~90 GB of device memory).

Every full-scale workload is checked at its full depth of 48 layers, layer by
layer: the oracle evaluates each layer from the GPU's own residual entering
it (teacher-forced, see harness.py) and the GPU's next residual, attention
output and routing must agree at bf16-rounding scale; the oracle's LM head
from the GPU's final residual must give the GPU's logits within max-abs 3e-2
and relative L2 1e-2, and the GPU's greedy token.  This is the comparison
that holds at depth: a free-running comparison of the 48-layer model is
chaotic (two faithful fp32 evaluations drift ~1 % apart in the residual
within 8 layers and decorrelate by layer ~12), so the free-running,
end-to-end check runs on the same workloads with the depth cut to 4 layers,
at the bound derived from the fp32 noise floor (harness.FULL4_FREE_BOUND).
"""
import numpy as np
import pytest

import harness
import synth

pytestmark = pytest.mark.gpu

FULL = synth.FULL
FULL4 = synth.Dims(4, 2048, 32, 4, 128, 128, 8, 768, 152064)


def run_steps(run, n):
    reps = []
    for _ in range(n):
        rep = run.step()
        print(run.summary(rep))
        reps.append(rep)
        assert run.ok(rep), rep
    return reps


# ------------------------------------------- 4 layers: free-running end to end


def test_full_width_batch1_8k_context_free_running():
    run = harness.ParityRun(FULL4, seq_lens=[8192], reserve_steps=4, materialise=False,
                            bound=harness.FULL4_FREE_BOUND)
    run_steps(run, 2)
    run.close()


def test_full_width_batch8_ragged_zipf_free_running():
    lens = synth.workloads()["full_b8"].seq_lens
    run = harness.ParityRun(FULL4, seq_lens=lens, reserve_steps=3, zipf_s=1.1,
                            materialise=False, bound=harness.FULL4_FREE_BOUND)
    run_steps(run, 2)
    st = run.dec.stats()
    assert st.sum_experts < 2 * 4 * 64  # Zipf skew: fewer distinct experts than B*k per layer
    run.close()


# ------------------------------- 48 layers: teacher-forced, layer by layer


def test_c3_full_depth_batch1_8k_teacher_forced():
    """The benchmarked workload: 48 layers, batch 1, 8192 cached tokens,
    three greedy steps, every layer checked."""
    run = harness.ParityRun("full", reserve_steps=4, materialise=False, free_steps=0)
    run_steps(run, 3)
    run.close()


def test_c4_full_depth_batch8_ragged_zipf_with_replacement():
    """Batch 8, ragged lengths U[1024, 16384], Zipf(1.1) router skew, 48
    layers; continuous batching at full width: after two steps slot 3 gets a
    new sequence, after one more step slot 6 does (pages never written, new
    lengths, new first tokens), and the schedule is rebuilt each time."""
    wl = synth.workloads()["full_b8"]
    spare = synth.ragged_lens(0, 2, 1024, 16384, gen=1)
    run = harness.ParityRun(FULL, seq_lens=wl.seq_lens, reserve_steps=6, zipf_s=1.1,
                            materialise=False, free_steps=0,
                            layout_lens=list(wl.seq_lens) + spare)
    pt = run.dev.layout.page_tables
    run_steps(run, 2)
    run.replace(3, spare[0], pt[8], 4242)
    run_steps(run, 1)
    run.replace(6, spare[1], pt[9], 77)
    run_steps(run, 2)
    assert run.dec.stats().steps == 2  # steps since the last schedule build
    run.close()


@pytest.mark.parametrize("lens", [[262144], [131072, 131072]], ids=["b1_262k", "b2_131k"])
def test_c5_full_depth_long_context_teacher_forced(lens):
    run = harness.ParityRun(FULL, seq_lens=lens, reserve_steps=3, materialise=False,
                            free_steps=0)
    run_steps(run, 1)
    run.close()


@pytest.mark.parametrize("lens", [[262144], [131072, 131072]], ids=["b1_262k", "b2_131k"])
def test_full_width_long_context_free_running(lens):
    run = harness.ParityRun(FULL4, seq_lens=lens, reserve_steps=3, materialise=False,
                            bound=harness.FULL4_FREE_BOUND)
    run_steps(run, 1)
    run.close()
