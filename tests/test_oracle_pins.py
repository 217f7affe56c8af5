"""Pins of the CPU oracle against facts the pages and mathematics fix.

Nothing here compares the oracle with a retyped copy of itself: each test is
a hand-worked fixture (tests/golden, each citing its passage), a closed form,
an invariant, a brute-force search, or a special case that reduces to a
library routine.  A plausible slip anywhere in oracle.cpp (dropped term, wrong
sign or index, transposed operand, swapped nibble, biased gate weights, wrong
tie rule) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def ulp32(v):
    v = np.float32(v)
    return float(np.spacing(np.abs(v)))


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ own exp/sigmoid

def test_exp_within_2ulp_of_math_exp():
    ts = np.concatenate([np.linspace(-32, 88, 40001, dtype=np.float32),
                         np.float32([0.0, 1e-8, -1e-8, 0.5, -0.5, 0.34657359, -0.34657359])])
    worst = 0.0
    for t in ts:
        got = oracle.router_exp(float(t))
        ref = math.exp(float(t))
        err = abs(got - ref) / ulp32(ref)
        worst = max(worst, err)
    assert worst <= 2.0, worst


def test_exp_special_values():
    assert oracle.router_exp(0.0) == 1.0
    for n in range(-40, 120, 7):
        t = float(np.float32(n * math.log(2.0)))
        ref = math.exp(t)
        assert abs(oracle.router_exp(t) - ref) <= 2 * ulp32(ref)


def test_sigmoid_identities():
    assert oracle.router_sigmoid(0.0) == 0.5
    assert oracle.router_sigmoid(40.0) == 1.0
    assert oracle.router_sigmoid(-100.0) == 0.0
    rng = np.random.default_rng(0)
    for z in rng.normal(0, 3, 2000).astype(np.float32):
        s, sm = oracle.router_sigmoid(float(z)), oracle.router_sigmoid(float(-z))
        ref = 1.0 / (1.0 + math.exp(-float(z)))
        assert abs(s - ref) <= 3 * ulp32(ref)
        assert abs((s + sm) - 1.0) <= 2 * ulp32(1.0)


def test_sigmoid_monotone():
    zs = np.linspace(-20, 20, 20001, dtype=np.float32)
    s = np.array([oracle.router_sigmoid(float(z)) for z in zs])
    assert np.all(np.diff(s) >= 0)


# ------------------------------------------------------------- int4 format

def test_half_to_float_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(b)) for b in bits], np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_dequant_golden():
    g = load("int4_format.json")
    s = np.array([g["scale_f16_bits"]], np.uint16)
    assert oracle.half_to_float(g["scale_f16_bits"]) == g["scale_value"]
    for c in g["cases"]:
        row = np.array([c["byte"]], np.uint8)
        assert oracle.dequant(row, s, 0) == c["k_even"], c
        assert oracle.dequant(row, s, 1) == c["k_odd"], c


def test_dequant_all_bytes_roundtrip():
    # unpack every byte with every position, requantise, re-pack: identity
    rng = np.random.default_rng(1)
    s_bits = rng.integers(0x1C00, 0x2800, 32).astype(np.uint16)  # ~0.004..0.03
    for byte in range(256):
        row = np.full(16, byte, np.uint8)  # one group of 32 values
        for k in (0, 1, 30, 31):
            sb = s_bits[k]
            sv = float(np.uint16(sb).view(np.float16))
            v = oracle.dequant(row, np.array([sb], np.uint16), k)
            q = round(v / sv)
            assert -8 <= q <= 7 and v == q * sv
            u = q + 8
            assert u == ((byte >> 4) if k & 1 else (byte & 15))
    z = np.array([0x88], np.uint8)
    assert oracle.dequant(z, np.array([0x3C00], np.uint16), 0) == 0.0


def test_dequant_group_scale_indexing():
    # scale of group g applies to k in [32g, 32g+32)
    row = np.full(64 // 2, 0xFF, np.uint8)  # q = 7 everywhere
    sc = np.array([0x3C00, 0x4000], np.uint16)  # 1.0, 2.0
    for k in range(64):
        assert oracle.dequant(row, sc, k) == (7.0 if k < 32 else 14.0)


# ----------------------------------------------------------- router logits

def test_router_order_golden():
    for c in load("router_order.json")["cases"]:
        H = c["H"]
        x = np.zeros((1, H), np.float32)
        w = np.zeros((1, H), np.float32)
        for k, v in c["x"].items():
            x[0, int(k)] = v
        for k, v in c["w"].items():
            w[0, int(k)] = v
        got = oracle.router_logits(x, w)[0, 0]
        assert got == np.float32(c["expected"]), (c["name"], got)


def test_router_logits_exact_on_integers():
    # small integers: every partial sum is an exact integer, so any order
    # gives the exact dot product; a dropped, repeated or misplaced term fails
    rng = np.random.default_rng(2)
    for H in (32, 256, 6144):
        x = rng.integers(-3, 4, (3, H)).astype(np.float32)
        W = rng.integers(-3, 4, (5, H)).astype(np.float32)
        ref = x.astype(np.int64) @ W.astype(np.int64).T
        got = oracle.router_logits(x, W)
        assert np.array_equal(got, ref.astype(np.float32))


def test_router_logits_within_rounding_bound():
    # |fl(x.w) - x.w| <= gamma_n * sum|x_k w_k| with n = terms on the longest
    # dependency chain (H/256 chunks * 4 fmas + 5 + 3 tree adds)
    rng = np.random.default_rng(3)
    H = 6144
    x = rng.standard_normal((4, H)).astype(np.float32)
    W = (rng.standard_normal((16, H)) * 0.02).astype(np.float32)
    got = oracle.router_logits(x, W).astype(np.float64)
    exact = x.astype(np.float64) @ W.astype(np.float64).T
    n = (H // 256) * 4 + 8
    u = 2.0 ** -24
    bound = (n * u / (1 - n * u)) * (np.abs(x).astype(np.float64) @ np.abs(W).astype(np.float64).T)
    assert np.all(np.abs(got - exact) <= bound)


# ---------------------------------------------------------------- selection

def test_selection_golden():
    for c in load("selection_ties.json")["cases"]:
        lg = np.array([c["logits"]], np.float32)
        b = np.array(c["bias"], np.float32)
        ids, w = oracle.select(lg, b, c["k"], c["n_group"], c["topk_group"], c["rsf"])
        assert ids[0].tolist() == c["ids"], c["name"]
        got = w[0].astype(np.float64) * 3 / c["rsf"]
        assert np.allclose(got, c["weights_times_3_over_rsf"], rtol=3e-7, atol=0), c["name"]


def _brute_select(key, s, k, n_group, topk_group):
    """Exhaustive search: best groups by summed score, best k-set by summed key.

    Group score here is found as the best pair sum over all pairs of the
    group; the kept groups are the topk_group-subset with the largest total
    score; the ids are the k-subset of their experts with the largest key
    sum.  Inputs are tie-free, so the optima are unique.
    """
    E = len(key)
    G = E // n_group
    gsc = []
    for g in range(n_group):
        idx = range(g * G, (g + 1) * G)
        if G == 1:
            gsc.append(key[g])
        else:
            gsc.append(max(float(key[a]) + float(key[b])
                           for a, b in itertools.combinations(idx, 2)))
    best_groups = max(itertools.combinations(range(n_group), topk_group),
                      key=lambda gs: sum(gsc[g] for g in gs))
    cand = [e for g in best_groups for e in range(g * G, (g + 1) * G)]
    best = max(itertools.combinations(cand, k), key=lambda es: sum(float(key[e]) for e in es))
    ids = sorted(best, key=lambda e: -float(key[e]))
    return ids


@pytest.mark.parametrize("E,k,ng,tg", [(16, 4, 4, 2), (16, 2, 8, 3), (12, 3, 3, 2),
                                       (8, 4, 2, 1), (16, 5, 4, 4), (9, 3, 9, 3)])
def test_selection_brute_force(E, k, ng, tg):
    rng = np.random.default_rng(E * 100 + k)
    for _ in range(40):
        lg = rng.normal(0, 1.5, (1, E)).astype(np.float32)
        b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
        ids, w = oracle.select(lg, b, k, ng, tg, 2.5)
        s = np.array([oracle.router_sigmoid(float(z)) for z in lg[0]], np.float32)
        key = (s + b).astype(np.float32)
        assert ids[0].tolist() == _brute_select(key, s, k, ng, tg)


def test_selection_reduces_to_plain_topk():
    rng = np.random.default_rng(5)
    E, k = 256, 8
    for ng, tg in ((1, 1), (8, 8)):
        lg = rng.normal(0, 1.5, (8, E)).astype(np.float32)
        b = rng.uniform(-0.05, 0.05, E).astype(np.float32)
        ids, _ = oracle.select(lg, b, k, ng, tg, 2.5)
        s = np.array([[oracle.router_sigmoid(float(z)) for z in row] for row in lg], np.float32)
        key = s + b
        for t in range(8):
            order = np.argsort(-key[t].astype(np.float64), kind="stable")[:k]
            assert ids[t].tolist() == order.tolist()


def test_selection_k_equals_E():
    lg = np.random.default_rng(6).normal(0, 1, (2, 16)).astype(np.float32)
    ids, w = oracle.select(lg, np.zeros(16, np.float32), 16, 4, 4, 1.0)
    assert sorted(ids[0].tolist()) == list(range(16))


def test_selection_permutation_equivariance():
    # permuting groups as blocks and experts inside groups permutes the ids
    rng = np.random.default_rng(7)
    E, ng, G, k, tg = 16, 4, 4, 4, 2
    lg = rng.normal(0, 1.5, (6, E)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    gp = rng.permutation(ng)
    inner = [rng.permutation(G) for _ in range(ng)]
    pi = np.array([gp[e // G] * G + inner[e // G][e % G] for e in range(E)])  # old -> new
    lg2 = np.empty_like(lg)
    b2 = np.empty_like(b)
    lg2[:, pi] = lg
    b2[pi] = b
    ids, w = oracle.select(lg, b, k, ng, tg, 2.5)
    ids2, w2 = oracle.select(lg2, b2, k, ng, tg, 2.5)
    assert np.array_equal(pi[ids], ids2)
    assert np.array_equal(w, w2)


def test_gate_weights_unbiased_and_sum_to_rsf():
    # weights come from the un-biased sigmoid (bias only selects) and are
    # renormalised to sum to the routed scale
    rng = np.random.default_rng(8)
    E, k, rsf = 256, 8, 2.5
    lg = rng.normal(0, 1.5, (64, E)).astype(np.float32)
    b = rng.uniform(-0.3, 0.3, E).astype(np.float32)
    ids, w = oracle.select(lg, b, k, 8, 4, rsf)
    for t in range(64):
        s = np.array([oracle.router_sigmoid(float(lg[t, e])) for e in ids[t]], np.float64)
        assert np.all(w[t] > 0)
        assert abs(float(w[t].astype(np.float64).sum()) - rsf) <= 4 * ulp32(rsf)
        assert np.allclose(w[t] / w[t][0], s / s[0], rtol=4e-7)
    # shifting all biases by a constant changes nothing
    ids2, w2 = oracle.select(lg, b + np.float32(0.25), k, 8, 4, rsf)
    assert np.array_equal(ids, ids2) and np.array_equal(w, w2)


# --------------------------------------------------------------------- plan

def test_plan_invariants_and_stable_order():
    rng = np.random.default_rng(9)
    for T, k, E in ((1, 8, 256), (4, 8, 256), (512, 8, 256), (7, 4, 16), (0, 4, 16)):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) \
            if T else np.zeros((0, k), np.int32)
        p = oracle.plan(ids, E)
        flat = ids.reshape(-1)
        assert p["counts"].tolist() == np.bincount(flat, minlength=E).tolist()
        assert p["offsets"][0] == 0 and p["offsets"][-1] == T * k
        assert np.array_equal(np.diff(p["offsets"]), p["counts"])
        assert np.array_equal(p["perm"], np.argsort(flat, kind="stable"))
        assert p["active"].tolist() == [e for e in range(E) if p["counts"][e] > 0]


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_closed_forms():
    H = 6144
    for c in (1.0, 3.0, -0.5):
        h = np.full((1, H), c, np.float32)
        out = oracle.rmsnorm(h, None, 1e-5)
        ref = c / math.sqrt(c * c + 1e-5)
        # two fp32 roundings (r to fp32, then h * r): at most 1.5 ulp
        assert np.all(np.abs(out - ref) <= 1.5 * ulp32(ref))
    # alternating +-a: mean square a^2
    h = np.tile(np.float32([2.0, -2.0]), (1, H // 2))
    out = oracle.rmsnorm(h, None, 1e-5)
    ref = 2.0 / math.sqrt(4.0 + 1e-5)
    assert np.all(np.abs(np.abs(out) - ref) <= 1.5 * ulp32(ref)) and np.all(np.sign(out) == np.sign(h))
    g = np.linspace(0.5, 2.0, H).astype(np.float32)
    out_g = oracle.rmsnorm(h, g, 1e-5)
    assert np.array_equal(out_g, (out * g).astype(np.float32))


def test_rmsnorm_within_fp64_bound():
    rng = np.random.default_rng(10)
    h = rng.standard_normal((3, 6144)).astype(np.float32)
    out = oracle.rmsnorm(h, None, 1e-5).astype(np.float64)
    hd = h.astype(np.float64)
    ref = hd / np.sqrt((hd * hd).mean(1, keepdims=True) + 1e-5)
    assert np.all(np.abs(out - ref) <= 1.5 * np.spacing(np.abs(ref).astype(np.float32)))
    # the scaling is one fp32 multiplier per row: the fp32 rounding of
    # 1/sqrt(mean + eps), the mean taken from the exact sum of squares
    for t in range(3):
        ms = math.fsum(float(v) * float(v) for v in hd[t]) / 6144
        rf = np.float32(1.0 / math.sqrt(ms + float(np.float32(1e-5))))
        assert np.array_equal(oracle.rmsnorm(h[t:t + 1], None, float(np.float32(1e-5)))[0],
                              h[t] * rf)


# ------------------------------------------------------------------ experts

def _pack(Q):
    """Integers q in [-8, 7], [rows, K] -> offset-binary bytes, low nibble = even k."""
    U = (Q + 8).astype(np.uint8)
    return (U[:, 0::2] | (U[:, 1::2] << 4)).astype(np.uint8)


def _f16bits(v):
    return np.asarray(v, np.float16).view(np.uint16)


def test_expert_constant_weights_closed_form():
    H, I = 256, 64
    rng = np.random.default_rng(11)
    x = rng.integers(-4, 5, H).astype(np.float32)
    cg, cu, cd = 3, -2, 5
    sg, su, sd = 0.5, 0.25, 0.125
    mats = (_pack(np.full((I, H), cg)), np.full((I, H // 32), _f16bits(sg)),
            _pack(np.full((I, H), cu)), np.full((I, H // 32), _f16bits(su)),
            _pack(np.full((H, I), cd)), np.full((H, I // 32), _f16bits(sd)))
    o = oracle.expert(x, I, mats, prec=1)
    Sx = float(x.sum())
    g = cg * sg * Sx
    u = cu * su * Sx
    h = g / (1 + math.exp(-g)) * u
    ref = cd * sd * I * h
    assert np.allclose(o, ref, rtol=1e-12)


def test_expert_reduces_to_integer_matvec():
    # scales 1, integer weights and inputs: gate/up are exact integer
    # mat-vecs; down with a one-hot h pulls a single column
    H, I = 128, 32
    rng = np.random.default_rng(12)
    Qg = rng.integers(-8, 8, (I, H))
    Qu = rng.integers(-8, 8, (I, H))
    Qd = rng.integers(-8, 8, (H, I))
    x = rng.integers(-2, 3, H).astype(np.float32)
    one = np.full((I, H // 32), _f16bits(1.0))
    oned = np.full((H, I // 32), _f16bits(1.0))
    mats = (_pack(Qg), one, _pack(Qu), one, _pack(Qd), oned)
    o = oracle.expert(x, I, mats, prec=1)
    g = Qg @ x.astype(np.int64)
    u = Qu @ x.astype(np.int64)
    h = np.array([gi / (1 + math.exp(-gi)) * ui for gi, ui in zip(g.astype(float), u.astype(float))])
    ref = Qd.astype(np.float64) @ h
    assert np.allclose(o, ref, rtol=1e-11, atol=1e-9)


def test_expert_group_scales_per_row_and_matrix():
    # integer weights and power-of-two scales that differ per row, per group of
    # 32 and per matrix: every dequantised weight, product and sum is exact in
    # float64, so the expert is the plain mat-vec SwiGLU of the dense matrices
    # W[r, c] = q[r, c] * s[r, c // 32]; a scale read from the wrong row, group
    # or matrix fails
    H, I = 128, 64
    rng = np.random.default_rng(17)
    pow2 = np.array([0.25, 0.5, 1.0, 2.0])
    Qg, Qu = rng.integers(-8, 8, (I, H)), rng.integers(-8, 8, (I, H))
    Qd = rng.integers(-8, 8, (H, I))
    Sg, Su = rng.choice(pow2, (I, H // 32)), rng.choice(pow2, (I, H // 32))
    Sd = rng.choice(pow2, (H, I // 32))
    x = rng.integers(-2, 3, H).astype(np.float32)
    mats = (_pack(Qg), _f16bits(Sg), _pack(Qu), _f16bits(Su), _pack(Qd), _f16bits(Sd))
    o = oracle.expert(x, I, mats, prec=1)
    Wg = Qg * np.repeat(Sg, 32, axis=1)
    Wu = Qu * np.repeat(Su, 32, axis=1)
    Wd = Qd * np.repeat(Sd, 32, axis=1)
    g = Wg @ x.astype(np.float64)
    u = Wu @ x.astype(np.float64)
    h = np.array([gi / (1 + math.exp(-gi)) * ui for gi, ui in zip(g, u)])
    ref = Wd @ h
    assert np.allclose(o, ref, rtol=1e-11, atol=1e-9 * np.abs(ref).max())


def _scaled(s_bits: np.ndarray, f: float) -> np.ndarray:
    """fp16 scale bits multiplied by a power of two (exact for these scales)."""
    out = (s_bits.view(np.float16).astype(np.float32) * np.float32(f)).astype(np.float16)
    assert np.array_equal(out.astype(np.float32) / np.float32(f),
                          s_bits.view(np.float16).astype(np.float32))
    return out.view(np.uint16)


def test_expert_linear_in_x_and_zero():
    """Gate and up are linear maps of x: scaling x by a power of two a while
    dividing the gate and up scales by a leaves every pre-activation, and so
    the whole expert, unchanged bit for bit (each product and sum scales
    exactly).  Down is linear in h: its scales times a give a times the
    output, exactly.  x = 0 gives 0."""
    from workloads import CONFIGS
    from workloads.gen import HostExpertCache
    w = CONFIGS["tiny"]
    gq, gs, uq, us, dq, ds = HostExpertCache(w).expert(3)
    x = np.random.default_rng(5).standard_normal(256).astype(np.float32)
    base = oracle.expert(x, 128, (gq, gs, uq, us, dq, ds))
    for a in (2.0, 0.5, 4.0):
        xa = (x * np.float32(a)).astype(np.float32)
        mats = (gq, _scaled(gs, 1 / a), uq, _scaled(us, 1 / a), dq, ds)
        assert np.array_equal(oracle.expert(xa, 128, mats), base), a
        # without the compensation the result changes (SwiGLU is not linear)
        assert not np.array_equal(oracle.expert(xa, 128, (gq, gs, uq, us, dq, ds)), base)
        out = oracle.expert(x, 128, (gq, gs, uq, us, dq, _scaled(ds, a)))
        assert np.array_equal(out, base * a), a
    assert np.all(oracle.expert(np.zeros(256, np.float32), 128, (gq, gs, uq, us, dq, ds)) == 0)


def test_fp32_oracle_error_far_below_tolerance():
    from workloads import CONFIGS
    from workloads.gen import HostExpertCache
    w = CONFIGS["glm_decode"]
    mats = HostExpertCache(w).expert(17)
    x = np.random.default_rng(13).standard_normal(6144).astype(np.float32)
    o32 = oracle.expert(x, 2048, mats, prec=0)
    o64 = oracle.expert(x, 2048, mats, prec=1)
    rel = np.abs(o32 - o64).max() / np.abs(o64).max()
    assert rel < 1e-5, rel


# --------------------------------------------------------------- full layer

def _layer_from(shape, router_w, router_b, experts, shared):
    return shape, router_w, router_b, (lambda e: experts[e]), shared


def test_layer_identical_experts_sum_to_rsf():
    # every routed expert identical => y = rsf * E(x) + S(x) (weights sum to rsf)
    from workloads import CONFIGS
    from workloads.gen import HostExpertCache, gen_router
    w = CONFIGS["tiny"]
    sh = w.shape
    cache = HostExpertCache(w)
    one = cache.expert(5)
    shared = cache.expert(-1)
    rw, rb = gen_router(sh, w.seed, 0, "uniform")
    x = np.random.default_rng(14).standard_normal((3, sh.hidden)).astype(np.float32)
    # both accumulations: fp64 (tight) and the fp32 layer the kernels match
    for prec, tol in ((1, 1e-6), (0, 2e-5)):
        y, ids, wt, _ = oracle.moe_forward(sh, rw.numpy(), rb.numpy(), lambda e: one, shared,
                                           x, prec=prec)
        for t in range(3):
            e = oracle.expert(x[t], sh.inter, one, prec=1)
            s = oracle.expert(x[t], sh.i_shared, shared, prec=1)
            ref = float(wt[t].astype(np.float64).sum()) * e + s
            assert abs(float(wt[t].astype(np.float64).sum()) - 2.5) < 1e-6
            assert np.allclose(y[t], ref, rtol=tol, atol=tol * np.abs(ref).max())


def test_layer_shared_only_when_routed_experts_are_zero():
    from workloads import CONFIGS
    from workloads.gen import HostExpertCache, gen_router
    w = CONFIGS["tiny"]
    sh = w.shape
    cache = HostExpertCache(w)
    zq = np.full((sh.inter, sh.hidden // 2), 0x88, np.uint8)
    zd = np.full((sh.hidden, sh.inter // 2), 0x88, np.uint8)
    e0 = cache.expert(0)
    zero = (zq, e0[1], zq, e0[3], zd, e0[5])
    shared = cache.expert(-1)
    rw, rb = gen_router(sh, w.seed, 0, "uniform")
    x = np.random.default_rng(15).standard_normal((2, sh.hidden)).astype(np.float32)
    y, *_ = oracle.moe_forward(sh, rw.numpy(), rb.numpy(), lambda e: zero, shared, x)
    for t in range(2):
        s = oracle.expert(x[t], sh.i_shared, shared, prec=0).astype(np.float32)
        assert np.array_equal(y[t], s)


def test_layer_residual_and_rmsnorm():
    from workloads import CONFIGS
    from workloads.gen import HostExpertCache, gen_router
    w = CONFIGS["tiny"]
    sh = w.shape
    cache = HostExpertCache(w)
    rw, rb = gen_router(sh, w.seed, 0, "uniform")
    h = (np.random.default_rng(16).standard_normal((2, sh.hidden)) * 3).astype(np.float32)
    xh = oracle.rmsnorm(h, None, 1e-5)
    y0, ids0, w0, _ = oracle.moe_forward(sh, rw.numpy(), rb.numpy(), cache.expert,
                                         cache.expert(-1), xh)
    y1, ids1, w1, _ = oracle.moe_forward(sh, rw.numpy(), rb.numpy(), cache.expert,
                                         cache.expert(-1), h, eps=1e-5, resid=h)
    assert np.array_equal(ids0, ids1) and np.array_equal(w0, w1)
    assert np.array_equal(y1, (h + y0).astype(np.float32))


def test_layer_rows_stable_alone_or_batched():
    # a token's ids, weights and output are the same whether it runs alone
    # (M = 1) or inside a batch of four (M = 4): rows never mix
    from workloads import CONFIGS
    from workloads.gen import HostExpertCache, gen_router
    w = CONFIGS["tiny"]
    sh = w.shape
    cache = HostExpertCache(w)
    rw, rb = gen_router(sh, w.seed, 0, "uniform")
    x = np.random.default_rng(18).standard_normal((4, sh.hidden)).astype(np.float32)
    y4, ids4, w4, _ = oracle.moe_forward(sh, rw.numpy(), rb.numpy(), cache.expert,
                                         cache.expert(-1), x)
    for t in range(4):
        y1, ids1, w1, _ = oracle.moe_forward(sh, rw.numpy(), rb.numpy(), cache.expert,
                                             cache.expert(-1), x[t:t + 1])
        assert np.array_equal(ids1[0], ids4[t]) and np.array_equal(w1[0], w4[t])
        assert np.array_equal(y1[0], y4[t])
    assert len({tuple(r) for r in ids4.tolist()}) > 1  # the rows do differ
