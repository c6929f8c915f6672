"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle/oracle.c (on the CPU),
builds it, routes the oracle through it and runs the pin suite: at least one
pin has to fail.  This shows the pins constrain every step of the definition
(gather address, GQA head map, scale, causal alignment, normalisation, the
log-sum-exp, the state merge, the 16-bit and E4M3 decoders, the K/V scales and the
q8_0 block scales).
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_fp8 as pins_fp8
from tests import test_oracle_pins as pins
from tests import test_oracle_q8 as pins_q8

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "kv_head_map_modulo": ("const int kvh = h / g;", "const int kvh = h % hk;"),
    "slot_and_page_swapped": ("const int64_t slot = t % page_size;", "const int64_t slot = t / page_size;"),
    "scale_dropped": ("z[t] = scale * s;", "z[t] = s;"),
    "causal_off_by_one": ("int64_t last = L - q_len + i;", "int64_t last = L - q_len + i - 1;"),
    "causal_top_left": ("int64_t last = L - q_len + i;", "int64_t last = i;"),
    "lse_missing_max": ("lse[n] = zmax + log(denom);", "lse[n] = log(denom);"),
    "not_normalised": ("o_row[e] = acc[e] / denom;", "o_row[e] = acc[e];"),
    "v_read_with_k_strides": ("(int64_t)kvh * v_sh + slot * v_st", "(int64_t)kvh * k_sh + slot * k_st"),
    "q_head_is_kv_head": ("(int64_t)h * q_stride_head", "(int64_t)kvh * q_stride_head"),
    "merge_weight_wrong_reference": ("exp(lse[(int64_t)s * rows + r] - total)", "exp(lse[(int64_t)s * rows + r] - m)"),
    "bf16_bias_off_by_one": ("expo - 134", "expo - 133"),
    "f16_subnormal_scale": ("ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    "e4m3_bias_off_by_one": ("ldexp((double)(8 + frac), expo - 10)", "ldexp((double)(8 + frac), expo - 9)"),
    "e4m3_subnormal_scale": ("ldexp((double)frac, -9)", "ldexp((double)frac, -10)"),
    "k_scale_dropped": ("(k_scale * kv_elem(k, kp, e", "(kv_elem(k, kp, e"),
    "v_scale_dropped": ("(v_scale * kv_elem(v, vp, e", "(kv_elem(v, vp, e"),
    "q8_0_block_index": ("scales[sidx + e / 32]", "scales[sidx + e / 64]"),
    "q8_0_codes_unsigned": ("(double)((const int8_t*)pool)[idx + e]", "(double)((const uint8_t*)pool)[idx + e]"),
    "q8_0_k_scales_from_v_pool": ("kv_elem(k, kp, e, kv_fmt, dec, ksc, ks)", "kv_elem(k, kp, e, kv_fmt, dec, vsc, ks)"),
    "q8_0_scale_head_and_slot_strides_swapped": ("(int64_t)kvh * vsc_sh + slot * vsc_st",
                                                 "(int64_t)kvh * vsc_st + slot * vsc_sh"),
    "last_token_dropped": ("n_vis = L;                              /* tokens", "n_vis = L - 1;                              /* tokens"),
}


def _pin_checks():
    """(name, callable) for every pin, with parametrised pins expanded."""
    checks = []
    for mod in (pins, pins_fp8, pins_q8):
        for name in dir(mod):
            if not name.startswith("test_"):
                continue
            fn = getattr(mod, name)
            marks = getattr(fn, "pytestmark", [])
            params = [m for m in marks if m.name == "parametrize"]
            if not params:
                checks.append((name, fn))
                continue
            argnames = [a.strip() for a in params[0].args[0].split(",")]
            for k, v in enumerate(params[0].args[1]):
                vals = v if len(argnames) > 1 else (v,)
                kwargs = dict(zip(argnames, vals))
                checks.append((f"{name}[{k}]", lambda fn=fn, kw=kwargs: fn(**kw)))
    return checks


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation, tmp_path):
    old, new = MUTATIONS[mutation]
    src = open(SRC).read()
    assert old in src, f"mutation anchor not found: {old!r}"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(mutant),
                    "-o", str(lib), "-lm"], check=True)
    caught = []
    with oracle.use_library(str(lib)):
        for name, check in _pin_checks():
            try:
                check()
            except (AssertionError, ValueError):
                caught.append(name)
    assert caught, f"no pin caught the planted mistake {mutation!r}"
