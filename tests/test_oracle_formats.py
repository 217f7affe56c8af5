"""Pins of the oracle's other expert formats: signed int8 weights and one
fp16 scale per row.

"GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy":
- N2: the container holds symmetric int4/int8 experts with per-row or grouped
  scales.
- "G2 implementation status": Q8 applies its scale to the signed
  two's-complement byte; Colibri's whole-row scale, repeated over 32-value
  groups, leaves every dequantised value unchanged.

Each pin ties the new formats to something fixed independently of them:
closed-form byte values, the grouped int4 oracle (pinned in
test_oracle_pins.py) through the identities the pages state, and a numpy
restatement in float64.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle


def _half_bits(v):
    return np.asarray(v, np.float16).view(np.uint16)


def _rand_int4(rng, rows, cols):
    return rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)


def _rand_scales(rng, rows, n):
    # fp16 scales in [0.005, 0.02]
    return _half_bits(rng.uniform(0.005, 0.02, size=(rows, n)).astype(np.float16))


def _int4_as_int8(q4):
    """The int8 bytes holding the same values as packed offset-binary nibbles:
    element 2 j is the low nibble of byte j, 2 j + 1 the high one, value u - 8."""
    lo = (q4 & 0xF).astype(np.int16) - 8
    hi = (q4 >> 4).astype(np.int16) - 8
    out = np.empty((q4.shape[0], q4.shape[1] * 2), np.int16)
    out[:, 0::2], out[:, 1::2] = lo, hi
    return out.astype(np.int8).view(np.uint8)


def test_int8_bytes_are_twos_complement():
    q = np.array([0x80, 0x7F, 0x00, 0xFF, 0x01, 0xC0, 0x40, 0x81], np.uint8)
    want = [-128, 127, 0, -1, 1, -64, 64, -127]
    half = _half_bits([0.5])
    for k, v in enumerate(want):
        # one scale for the whole row: the scale index is 0 at every k
        assert oracle.dequant_fmt(q, half, k, oracle.FMT_INT8, 0) == v * 0.5
    # grouped: element k takes scale k / 32
    row = np.full(64, 0xFE, np.uint8)  # -2 everywhere
    sc = _half_bits([0.25, 4.0])
    assert oracle.dequant_fmt(row, sc, 31, oracle.FMT_INT8, 32) == -0.5
    assert oracle.dequant_fmt(row, sc, 32, oracle.FMT_INT8, 32) == -8.0


def test_int4_format_is_the_grouped_dequant():
    rng = np.random.default_rng(3)
    q = _rand_int4(rng, 1, 128)[0]
    s = _rand_scales(rng, 1, 4)[0]
    for k in range(128):
        assert oracle.dequant_fmt(q, s, k, oracle.FMT_INT4, 32) == oracle.dequant(q, s, k)
        # per-row: every element takes the row's (first) scale
        assert oracle.dequant_fmt(q, s, k, oracle.FMT_INT4, 0) == \
            oracle.dequant(q, np.full(4, s[0], np.uint16), k)


def _expert_mats(rng, H, I, per_row=False, scale_fn=_rand_scales):
    mats = []
    for rows, cols in ((I, H), (I, H), (H, I)):
        mats.append(_rand_int4(rng, rows, cols))
        mats.append(scale_fn(rng, rows, 1 if per_row else cols // 32))
    return mats


def _repeat_scales(mats, H, I):
    """The grouped layout of per-row scales: each row's scale in all groups."""
    out = list(mats)
    for i, cols in ((1, H), (3, H), (5, I)):
        out[i] = np.repeat(mats[i], cols // 32, axis=1)
    return out


@pytest.mark.parametrize("prec", [0, 1])
def test_row_scale_equals_repeated_group_scales(prec):
    """G2 status: the whole-row scale repeated over the 32-value groups gives
    the same dequantised values, so the same expert output, bit for bit."""
    rng = np.random.default_rng(11)
    H, I = 96, 64
    x = rng.standard_normal(H).astype(np.float32)
    mats = _expert_mats(rng, H, I, per_row=True)
    got = oracle.expert_fmt(x, I, mats, oracle.FMT_INT4, 0, prec)
    want = oracle.expert(x, I, _repeat_scales(mats, H, I), prec)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("gsz", [32, 0])
def test_int8_equals_int4_on_int4_codes(gsz):
    """An int8 expert whose bytes hold the int4 codes (-8..7) with the same
    scales computes the int4 expert exactly."""
    rng = np.random.default_rng(12)
    H, I = 64, 96
    x = rng.standard_normal(H).astype(np.float32)
    mats4 = _expert_mats(rng, H, I, per_row=gsz == 0)
    mats8 = list(mats4)
    for i in (0, 2, 4):
        mats8[i] = _int4_as_int8(mats4[i])
    for prec in (0, 1):
        a = oracle.expert_fmt(x, I, mats8, oracle.FMT_INT8, gsz, prec)
        b = oracle.expert_fmt(x, I, mats4, oracle.FMT_INT4, gsz, prec)
        assert np.array_equal(a, b)
    assert np.array_equal(oracle.expert_fmt(x, I, mats4, oracle.FMT_INT4, 32, 0)
                          if gsz == 32 else oracle.expert(x, I, _repeat_scales(mats4, H, I), 0),
                          oracle.expert_fmt(x, I, mats8, oracle.FMT_INT8, gsz, 0))


def _numpy_expert(x, mats, fmt, gsz):
    """The expert in float64 numpy: W = q * s per element, h = silu(Wg x) *
    (Wu x), o = Wd h; q from an int8 view (int8) or nibble arithmetic (int4)."""
    def deq(q, s):
        if fmt == oracle.FMT_INT8:
            w = q.view(np.int8).astype(np.float64)
        else:
            w = np.empty((q.shape[0], q.shape[1] * 2))
            w[:, 0::2] = (q & 0xF).astype(np.float64) - 8
            w[:, 1::2] = (q >> 4).astype(np.float64) - 8
        sc = s.view(np.float16).astype(np.float64)
        sc = np.repeat(sc, w.shape[1] if gsz == 0 else gsz, axis=1)
        return w * sc
    gq, gs, uq, us, dq, ds = mats
    xd = x.astype(np.float64)
    g = deq(gq, gs) @ xd
    u = deq(uq, us) @ xd
    h = g / (1.0 + np.exp(-g)) * u
    return deq(dq, ds) @ h


@pytest.mark.parametrize("fmt,gsz", [(1, 32), (1, 0), (0, 0)])
def test_formats_against_numpy(fmt, gsz):
    rng = np.random.default_rng(20 + 2 * fmt + gsz)
    H, I = 128, 64
    x = rng.standard_normal(H).astype(np.float32)
    mats = []
    for rows, cols in ((I, H), (I, H), (H, I)):
        nb = cols if fmt == oracle.FMT_INT8 else cols // 2
        mats.append(rng.integers(0, 256, size=(rows, nb), dtype=np.uint8))
        sc = rng.uniform(0.0003, 0.0012 if fmt == oracle.FMT_INT8 else 0.02,
                         size=(rows, 1 if gsz == 0 else cols // gsz))
        mats.append(_half_bits(sc.astype(np.float16)))
    got = oracle.expert_fmt(x, I, mats, fmt, gsz, prec=1)
    want = _numpy_expert(x, mats, fmt, gsz)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_layer_of_row_scaled_experts():
    """The whole layer on per-row experts equals the layer on the same
    experts with the scales repeated over the groups (routing unchanged)."""
    from workloads.configs import LayerShape
    rng = np.random.default_rng(30)
    H, I, E = 64, 64, 8
    sh_row = LayerShape(H, I, E, 2, 2, 1, 2.5, group_size=0)
    sh_grp = LayerShape(H, I, E, 2, 2, 1, 2.5)
    experts = [_expert_mats(rng, H, I, per_row=True) for _ in range(E)]
    shared = _expert_mats(rng, H, I, per_row=True)
    rw = (rng.standard_normal((E, H)) * 0.1).astype(np.float32)
    rb = (rng.uniform(-0.1, 0.1, E)).astype(np.float32)
    x = rng.standard_normal((3, H)).astype(np.float32)
    y_row, ids_row, w_row, _ = oracle.moe_forward(sh_row, rw, rb, lambda e: experts[e], shared, x)
    y_grp, ids_grp, w_grp, _ = oracle.moe_forward(
        sh_grp, rw, rb, lambda e: _repeat_scales(experts[e], H, I),
        _repeat_scales(shared, H, I), x)
    assert np.array_equal(ids_row, ids_grp) and np.array_equal(w_row, w_grp)
    assert np.array_equal(y_row, y_grp)


def test_generated_formats_have_the_stated_layout():
    """The seeded generators lay the formats out as the oracle reads them:
    int8 K bytes a row, per-row scales one a row; int4 rows unchanged."""
    from workloads.gen import gen_expert_matrix
    q4, s4 = gen_expert_matrix(5, 0, 0, [3], 16, 64)
    q8, s8 = gen_expert_matrix(5, 0, 0, [3], 16, 64, group_size=0, fmt="int8")
    assert q4.shape == (1, 16, 32) and s4.shape == (1, 16, 2)
    assert q8.shape == (1, 16, 64) and s8.shape == (1, 16, 1)
    # int8 scales: the int4 table / 16, exact in fp16
    assert float(s8.max()) <= 0.02 / 16 and float(s8.min()) >= 0.005 / 16
    q4r, s4r = gen_expert_matrix(5, 0, 0, [3], 16, 64, group_size=0)
    assert np.array_equal(q4r.numpy(), q4.numpy()) and s4r.shape == (1, 16, 1)
