"""The seeded input generator: determinism, distribution, helpers (CPU)."""
import numpy as np

import synth


def test_normal_is_deterministic_and_offset_consistent():
    a = synth.normal_bf16(0, 123, 0.02, 1000)
    b = synth.normal_bf16(0, 123, 0.02, 1000)
    assert np.array_equal(a, b)
    c = synth.normal_bf16(0, 123, 0.02, 500, offset=500)
    assert np.array_equal(a[500:], c)
    assert not np.array_equal(a, synth.normal_bf16(1, 123, 0.02, 1000))
    assert not np.array_equal(a, synth.normal_bf16(0, 124, 0.02, 1000))


def test_irwin_hall_moments_and_support():
    x = synth.normal_f64(0, 7, 2_000_000)
    assert abs(x.mean()) < 3e-3
    assert abs(x.var() - 1.0) < 3e-3
    # Irwin-Hall(12) - 6: support [-6, 6], kurtosis 3 - 1.2/12 = 2.9.
    assert x.min() >= -6.0 and x.max() <= 6.0
    kurt = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert abs(kurt - 2.9) < 0.02
    # Values are multiples of 2^-32 (the sum of twelve 32-bit integers / 2^32).
    assert np.all(x * 2.0 ** 32 == np.round(x * 2.0 ** 32))


def test_bf16_scaling_matches_rounded_f64():
    """normal_bf16 = bf16_rne(float32(normal * sigma))."""
    n = 100_000
    x = synth.normal_f64(0, 9, n)
    bits = synth.normal_bf16(0, 9, 0.02, n)
    f32 = (x * 0.02).astype(np.float32)
    u = f32.view(np.uint32).astype(np.uint64)
    expect = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(bits, expect)
    v = synth.bf16_bits_to_f32(bits)
    assert abs(v.std() - 0.02) < 2e-4


def test_uniform_int_and_permutation():
    u = synth.uniform_int(0, 3, 17, 100_000)
    assert u.min() == 0 and u.max() == 16
    counts = np.bincount(u, minlength=17)
    assert counts.min() > 100_000 / 17 * 0.9
    p = synth.permutation(0, 4, 1000)
    assert sorted(p.tolist()) == list(range(1000))
    assert not np.array_equal(p, np.arange(1000))


def test_page_layout_covers_reserved_positions():
    d = synth.TINY
    pl = synth.page_layout(d, [64, 5, 31], reserve_steps=9)
    P = d.page_size
    used = []
    for b, L in enumerate([64, 5, 31]):
        need = -(-(L + 9) // P)
        assert np.all(pl.page_tables[b, :need] >= 0)
        assert np.all(pl.page_tables[b, need:] == -1)
        used += pl.page_tables[b, :need].tolist()
    assert sorted(used) == list(range(pl.num_pages))


def test_workload_shapes():
    w = synth.workloads()
    full = w["full"].dims
    # ~30.5B parameters total for the full-scale model.
    total = synth.weight_bytes_total(full) / 2
    assert 30.0e9 < total < 31.0e9
    b8 = w["full_b8"]
    assert b8.batch == 8 and all(1024 <= L <= 16384 for L in b8.seq_lens)
    assert w["long_b1"].seq_lens == [262144] and w["long_b2"].seq_lens == [131072] * 2


def test_zipf_bias():
    b = synth.router_bias(synth.FULL, 3, 1.1)
    ranks = np.exp(-b / 1.1)
    assert np.allclose(np.sort(ranks), np.arange(1, 129), rtol=1e-5)
    assert synth.router_bias(synth.FULL, 3, None) is None
