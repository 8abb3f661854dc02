"""Failure detection without a GPU fault (needs a GB300).

A wait that can never be met (the attention-done target of one layer raised
by the test hook) must end with MK_ERR_DEVICE_TIMEOUT once the wait limit
passes: every CTA sees the abort flag, drains its copies and returns, the
error is sticky on that context, and a new context works normally.
"""
import time

import pytest

import harness
import persistent_moe_decode_sm_gb300 as mk

pytestmark = pytest.mark.gpu


def test_unsatisfiable_wait_times_out_and_recovers():
    run = harness.ParityRun("tiny")
    rep = run.step()
    assert run.ok(rep)
    mk.mk_set_wait_limit_ns(run.dec.ctx, 200_000_000)  # 0.2 s
    mk.mk_debug_poison_wait(run.dec.ctx, 1, 1000)
    t0 = time.time()
    run.dec.decode_step(run.tok_d, run.logits_d, run.next_d)
    rc = mk.lib().mk_sync(run.dec.ctx)
    elapsed = time.time() - t0
    assert rc == mk.MK_ERR_DEVICE_TIMEOUT, mk.STATUS_NAMES.get(rc, rc)
    assert elapsed < 10.0
    # sticky: the context refuses further steps
    with pytest.raises(mk.MkError) as e:
        run.dec.decode_step(run.tok_d, run.logits_d, run.next_d)
    assert e.value.code == mk.MK_ERR_DEVICE_TIMEOUT
    run.close()
    # a fresh context on the same GPU is unaffected
    run2 = harness.ParityRun("tiny")
    for _ in range(2):
        rep = run2.step()
        assert run2.ok(rep), rep
    run2.close()


def test_out_of_vocabulary_token_fails_the_step_without_reading_outside_the_table():
    run = harness.ParityRun("tiny")
    assert run.ok(run.step())
    bad = run.tok_d.clone()
    bad[0] = run.dims.vocab + 7  # outside [0, vocab): the kernel must not index with it
    run.dec.decode_step(bad, run.logits_d, run.next_d)
    rc = mk.lib().mk_sync(run.dec.ctx)
    assert rc == mk.MK_ERR_BAD_TOKEN, mk.STATUS_NAMES.get(rc, rc)
    with pytest.raises(mk.MkError) as e:  # sticky
        run.dec.decode_step(run.tok_d, run.logits_d, run.next_d)
    assert e.value.code == mk.MK_ERR_BAD_TOKEN
    run.close()
    run2 = harness.ParityRun("tiny")
    assert run2.ok(run2.step())
    run2.close()


def test_host_side_argument_errors():
    run = harness.ParityRun("tiny", seq_lens=[62], reserve_steps=2)
    pl = run.dev.layout
    with pytest.raises(mk.MkError) as e:
        run.dec.build_schedule([62, 3], pl.page_tables.repeat(2, 0))  # batch > max_batch (1)
    assert e.value.code == mk.MK_ERR_BATCH
    bad = pl.page_tables.copy()
    bad[0, 0] = pl.num_pages + 5
    with pytest.raises(mk.MkError) as e:
        run.dec.build_schedule([62], bad)
    assert e.value.code == mk.MK_ERR_PAGE_OOB
    run.dec.build_schedule([62], pl.page_tables)
    for _ in range(2):
        assert run.ok(run.step())
    # the reserve is spent: the next position has no page
    with pytest.raises(mk.MkError) as e:
        run.dec.decode_step(run.tok_d, run.logits_d, run.next_d)
    assert e.value.code == mk.MK_ERR_PAGE_OOB
    run.close()
