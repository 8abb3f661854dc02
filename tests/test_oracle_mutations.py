"""The pins catch planted mistakes (CPU only).

Each case rebuilds a copy of the oracle with one plausible mistake (a dropped
term, a wrong sign or index, a transposed or mis-strided operand, a swapped
pair) and runs the oracle's pin tests against it in a subprocess; every
mutant must fail at least one pin.  The mistakes are planted in a temporary
copy of the oracle's source, never in the repository.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = {
    "rmsnorm_drops_eps": [("sqrtf(mean + eps)", "sqrtf(mean)")],
    "rmsnorm_sum_not_mean": [("const float mean = ss / (float)d;", "const float mean = ss;")],
    "rope_wrong_sign": [("xh[i] = round_bf16(a - b);", "xh[i] = round_bf16(a + b);")],
    "rope_adjacent_pairs": [("const float x1 = xh[i], x2 = xh[i + half];",
                             "const float x1 = xh[2 * i], x2 = xh[2 * i + 1];")],
    "rope_wrong_frequency": [("pow(base, -2.0 * (double)i / (double)D)",
                              "pow(base, -1.0 * (double)i / (double)D)")],
    "rope_position_off_by_one": [("const int64_t pos = m->cur_len[b];",
                                  "const int64_t pos = m->cur_len[b] + 1;")],
    "attention_scale_1_over_D": [("(float)(1.0 / sqrt((double)D))", "(float)(1.0 / (double)D)")],
    "attention_skips_new_key": [("const int64_t nkeys = pos + 1;",
                                 "const int64_t nkeys = pos > 0 ? pos : 1;")],
    "gqa_wrong_head_map": [("const int64_t hk = i / G;", "const int64_t hk = i % Hkv;")],
    "kv_wrong_slot": [("const int64_t slot = j % P;", "const int64_t slot = (j + 1) % P;")],
    "kv_cached_before_rope": [
        ("    rope(kk.data(), Hkv, D, pos, dm.rope_base);",
         "    std::vector<float> kpre(kk); rope(kk.data(), Hkv, D, pos, dm.rope_base);"),
        ("ak.insert(ak.end(), kk.begin(), kk.end());", "ak.insert(ak.end(), kpre.begin(), kpre.end());")],
    "q_not_rounded": [("for (auto &x : q) x = round_bf16(x);", "")],
    "router_no_renormalisation": [("w[t] = p[order[t]] / sum_top;", "w[t] = p[order[t]];")],
    "router_ties_to_higher_id": [("[&](int32_t a, int32_t b) { return r[a] > r[b]; });",
                                  "[&](int32_t a, int32_t b) { return r[a] > r[b] || (r[a] == r[b] && a > b); });")],
    "silu_wrong_sign": [("return x / (1.0f + expf(-x));", "return x / (1.0f + expf(x));")],
    "gate_up_swapped": [("a[f] = round_bf16(silu(gb) * ub);", "a[f] = round_bf16(silu(ub) * gb);")],
    "down_expert_stride": [("gemv(Ly.wd, e * d, d, F, a.data(), dbl, y.data());",
                            "gemv(Ly.wd, e * F, d, F, a.data(), dbl, y.data());")],
    "residual_drops_moe": [("h[i] = round_bf16((h[i] + attn[i]) + moe[i]);",
                            "h[i] = round_bf16(h[i] + attn[i]);")],
    "residual_drops_attention": [("h[i] = round_bf16((h[i] + attn[i]) + moe[i]);",
                                  "h[i] = round_bf16(h[i] + moe[i]);")],
    "residual_drops_h": [("h[i] = round_bf16((h[i] + attn[i]) + moe[i]);",
                          "h[i] = round_bf16(attn[i] + moe[i]);")],
    "final_norm_skipped": [("rmsnorm(&h[b * d], m->final_norm, d, dm.rms_eps, dbl, &n[b * d]);",
                            "for (int64_t i = 0; i < d; ++i) n[b * d + i] = h[b * d + i];")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert old in src, f"mutation site for {name} not found"
        src = src.replace(old, new)
    src = src.replace('"oracle.h"', '"' + os.path.join(ROOT, "oracle", "oracle.h") + '"')
    src = src.replace('"../synth/synth_rng.h"', '"' + os.path.join(ROOT, "synth", "synth_rng.h") + '"')
    cpp = tmp_path / "mutant.cpp"
    cpp.write_text(src)
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-shared",
                           "-fPIC", str(cpp), "-o", str(lib)])
    env = dict(os.environ, MK_ORACLE_LIB_OVERRIDE=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_step.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
