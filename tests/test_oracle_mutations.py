"""The oracle's pins are sharp: a slip planted anywhere in the oracle fails one.

Each mutant changes one place of a copy of oracle/oracle.cpp the way a slip
would: a wrong sign, index or constant, a dropped term, swapped operands, the
wrong tie rule, a plan in the wrong order.  The copy is compiled with the
oracle's own flags under oracle/_build/mutants/, and tests/test_oracle_pins.py and
tests/test_oracle_formats.py run against it in a subprocess (MOE_ORACLE_LIB names the build); that run must
fail.  The unaltered source, built and run the same way, must pass, so that each
failure is the slip's doing and not the harness's.  Everything happens on the
CPU; the CUDA library is not involved.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

from oracle import build as oracle_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py"),
        os.path.join(ROOT, "tests", "test_oracle_formats.py")]
OUT = os.path.join(ROOT, "oracle", "_build", "mutants")

# name -> (text in oracle.cpp, exactly once; its replacement)
MUTANTS = {
    # int4 format and fp16 scales
    "nibble_order_swapped": ("(k & 1) ? (byte >> 4) : (byte & 0xF)",
                             "(k & 1) ? (byte & 0xF) : (byte >> 4)"),
    "offset_binary_bias_7": ("return (float)(u - 8) * s;", "return (float)(u - 7) * s;"),
    "scale_group_of_64": ("row_s[k / 32]", "row_s[k / 64]"),
    "half_exponent_bias": ("(int)expo - 25", "(int)expo - 24"),
    "half_subnormal_scale": ("std::ldexp((float)mant, -24)", "std::ldexp((float)mant, -25)"),
    "half_sign_dropped": ("return sign ? -mag : mag;", "return mag;"),
    # own exponential and sigmoid
    "sigmoid_sign": ("const float t = -z;", "const float t = z;"),
    "exp_ln2_low_part_dropped": ("  r = std::fma(-n, kLn2Lo, r);\n", ""),
    "exp_series_degree_6": ("float p = kInvFact[7];", "float p = 0.0f;"),
    # router logits
    "logit_operand_reversed": ("acc = std::fma(x[k], w[k], acc);",
                               "acc = std::fma(x[k], w[H - 1 - k], acc);"),
    "logit_chunk_stride": ("for (int c = j; c < chunks; c += 32) {",
                           "for (int c = j; c < chunks; c += 16) {"),
    "logit_segments_summed_in_sequence": (
        "  for (int d = 4; d >= 1; d /= 2)\n"
        "    for (int s = 0; s < d; ++s) seg[s] = seg[s] + seg[s + d];\n"
        "  return seg[0];",
        "  float tot = seg[0];\n"
        "  for (int s = 1; s < 8; ++s) tot = tot + seg[s];\n"
        "  return tot;"),
    # noaux_tc selection and gate weights
    "group_score_max_only": ("gscore[g] = (G >= 2) ? a + b : a;", "gscore[g] = a;"),
    "group_second_largest_lost": ("} else if (key[e] > b) {", "} else if (key[e] > a) {"),
    "tie_to_higher_id": ("(va == vb && ia < ib)", "(va == vb && ia > ib)"),
    "groups_not_limited": ("if (taken[e] || !group_kept[e / G]) continue;",
                           "if (taken[e]) continue;"),
    "groups_interleaved": ("!group_kept[e / G]", "!group_kept[e % n_group]"),
    "gate_from_biased_key": ("const float g = s[ids[(size_t)t * k + j]];",
                             "const float g = key[ids[(size_t)t * k + j]];"),
    "renormalised_by_key_sum": ("sum = sum + s[best];", "sum = sum + key[best];"),
    "routed_scale_dropped": ("weights[(size_t)t * k + j] = q * rsf;",
                             "weights[(size_t)t * k + j] = q;"),
    # routing plan
    "plan_entries_descending": ("for (int i = 0; i < N; ++i)\n      if (ids[i] == e)",
                                "for (int i = N - 1; i >= 0; --i)\n      if (ids[i] == e)"),
    "plan_active_includes_empty": ("if (counts[e] > 0) active[na++] = e;",
                                   "if (counts[e] >= 0) active[na++] = e;"),
    # RMSNorm
    "rmsnorm_eps_dropped": ("std::sqrt(mean + eps)", "std::sqrt(mean)"),
    "rmsnorm_mean_over_h_minus_1": ("seg[0] / (double)H", "seg[0] / (double)(H - 1)"),
    "rmsnorm_gamma_dropped": ("out[k] = gamma ? v * gamma[k] : v;", "out[k] = v;"),
    # experts
    "silu_sign": ("g / ((Acc)1 + std::exp(-g))", "g / ((Acc)1 + std::exp(g))"),
    "swiglu_gate_and_up_swapped": (
        "const Acc silu = g / ((Acc)1 + std::exp(-g));\n    h[i] = silu * u;",
        "const Acc silu = u / ((Acc)1 + std::exp(-u));\n    h[i] = silu * g;"),
    "up_with_gate_scales": ("u = u + (Acc)dequant_fmt(ur, usr, k", "u = u + (Acc)dequant_fmt(ur, gsr, k"),
    "down_scale_row_stride": ("const size_t si = gsz == 0 ? 1 : (size_t)I / 32;",
                              "const size_t si = gsz == 0 ? 1 : (size_t)I / 64;"),
    # layer combine
    "routed_weight_dropped": ("accf[r] = accf[r] + wj * (float)o[r];",
                              "accf[r] = accf[r] + (float)o[r];"),
    "shared_expert_skipped": ("if (L->n_shared > 0) {", "if (L->n_shared > 1) {"),
    "shared_expert_scaled": ("accf[r] = accf[r] + (float)o[r];",
                             "accf[r] = accf[r] + L->rsf * (float)o[r];"),
    "residual_dropped": ("y[(size_t)t * H + r] = resid ? base + v : v;",
                         "y[(size_t)t * H + r] = v;"),
    # dropped last terms, saturation and rounding slips
    "half_implicit_bit_dropped": ("(float)(mant | 0x400u)", "(float)mant"),
    "exp_reduction_by_floor": ("std::nearbyint(t * kLog2e)", "std::floor(t * kLog2e)"),
    "sigmoid_saturates_to_0": ("if (t < -32.0f) return 1.0f;", "if (t < -32.0f) return 0.0f;"),
    "plan_offsets_start_at_count": ("offsets[0] = 0;", "offsets[0] = counts[0];"),
    "last_gate_slot_skipped": ("for (int j = 0; j < k; ++j) {\n      const float g",
                               "for (int j = 0; j + 1 < k; ++j) {\n      const float g"),
    "expert_last_k_dropped": ("for (int k = 0; k < H; ++k) {\n      g = g",
                              "for (int k = 0; k + 1 < H; ++k) {\n      g = g"),
    "down_last_i_dropped": ("for (int i = 0; i < I; ++i) o = o",
                            "for (int i = 0; i + 1 < I; ++i) o = o"),
    "layer_rows_read_token_0": ("const float* xt = xh.data() + (size_t)t * H;",
                                "const float* xt = xh.data();"),
    # the other expert formats (int8, one scale per row)
    "int8_read_unsigned": ("q = byte < 128 ? (int)byte : (int)byte - 256;", "q = (int)byte;"),
    "int8_offset_binary": ("q = byte < 128 ? (int)byte : (int)byte - 256;",
                           "q = (int)byte - 128;"),
    "int8_rows_at_int4_stride": ("const size_t qh = fmt == 1 ? (size_t)H : (size_t)H / 2;",
                                 "const size_t qh = (size_t)H / 2;"),
    "row_scales_of_row_0": ("const size_t sh = gsz == 0 ? 1 : (size_t)H / 32;",
                            "const size_t sh = gsz == 0 ? 0 : (size_t)H / 32;"),
    "row_scale_int4_offset_7": ("q = int4_code(row_q, k) - 8;", "q = int4_code(row_q, k) - 7;"),
    "layer_scale_group_dropped": ("L->wfmt, L->gsz, gq", "L->wfmt, 0, gq"),
}


def _source() -> str:
    with open(oracle_build.SRC) as f:
        return f.read()


def _run_pins(name: str, text: str) -> tuple[str, int, str]:
    """Build text as the oracle and run the pins on it; (name, exit code, tail)."""
    src = os.path.join(OUT, name + ".cpp")
    lib = os.path.join(OUT, name + ".so")
    with open(src, "w") as f:
        f.write(text)
    oracle_build.compile_source(src, lib)
    env = dict(os.environ, MOE_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    return name, r.returncode, (r.stdout + r.stderr)[-600:]


def test_each_mutant_text_occurs_once():
    src = _source()
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, name
        assert old != new, name


def test_pins_fail_on_every_planted_slip():
    src = _source()
    os.makedirs(OUT, exist_ok=True)
    jobs = {"unaltered": src}
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, name
        jobs[name] = src.replace(old, new)
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        results = {n: (rc, tail) for n, rc, tail in ex.map(lambda kv: _run_pins(*kv),
                                                             jobs.items())}
    rc, tail = results.pop("unaltered")
    assert rc == 0, "the pins fail on the unaltered oracle:\n" + tail
    survivors = sorted(n for n, (rc, _) in results.items() if rc == 0)
    assert not survivors, f"no pin catches: {survivors}"
    for name in jobs:  # keep nothing but the directory
        for ext in (".cpp", ".so"):
            p = os.path.join(OUT, name + ext)
            if os.path.exists(p):
                os.remove(p)


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
