"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties an oracle function to a hand-derived worked example, a closed
form of the Adam recursion, an exhaustive or property check, a conversion
done by numpy or torch, or a value printed on the pages.  None of them
re-types the oracle's per-element sequence.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import DT_BF16, DT_F16, DT_F32, MODE_ADAMW, MODE_L2, Group

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32_EPS = 2.0 ** -24  # unit roundoff of fp32


def _ulp(x):
    return np.spacing(np.abs(np.asarray(x, dtype=np.float32))).astype(np.float64)


# ---- worked examples ---------------------------------------------------------

def _worked_examples():
    rows = []
    with open(os.path.join(GOLDEN, "worked_examples.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, *kvs = line.split()
            d = dict(kv.split("=") for kv in kvs)
            rows.append((name, d))
    return rows


@pytest.mark.parametrize("name,d", _worked_examples(),
                         ids=[r[0] for r in _worked_examples()])
def test_worked_example_fp32_exact(name, d):
    mode = MODE_ADAMW if d["mode"] == "adamw" else MODE_L2
    grp = Group(mode=mode, bias_correction=int(d["bc"]), beta1=float(d["beta1"]),
                beta2=float(d["beta2"]), eps=float(d["eps"]), weight_decay=float(d["wd"]),
                lr=float(d["lr"]), grad_scale=float(d["gs"]))
    p = np.array([float(d["p"])], np.float32)
    m = np.array([float(d["m"])], np.float32)
    v = np.array([float(d["v"])], np.float32)
    g = np.array([float(d["g"])], np.float32)
    oracle.adam_f32(grp, int(d["step"]), p, m, v, g, DT_F32)
    assert p[0] == np.float32(d["p_new"]), (name, p[0])
    assert m[0] == np.float32(d["m_new"]), (name, m[0])
    assert v[0] == np.float32(d["v_new"]), (name, v[0])
    # the double evaluation reaches the same exact values
    p64, m64, v64 = (np.array([float(d[k])]) for k in ("p", "m", "v"))
    oracle.adam_f64(grp, int(d["step"]), p64, m64, v64, np.array([float(d["g"])]))
    assert (p64[0], m64[0], v64[0]) == (float(d["p_new"]), float(d["m_new"]), float(d["v_new"]))


def test_worked_example_remainder_form():
    # Example A on a master held as bf16 1.0 + remainder 0: the new master
    # 0.9609375 has 8 significant bits, so it splits into 0x3F76 and 0.
    grp = Group(mode=MODE_ADAMW, bias_correction=1, beta1=0.5, beta2=0.75, eps=0.5,
                weight_decay=0.125, lr=0.0625, grad_scale=1.0)
    hi = np.array([0x3F80], np.uint16)
    rem = np.array([0], np.int16)
    m = np.zeros(1, np.float32)
    v = np.zeros(1, np.float32)
    out = np.zeros(1, np.uint16)
    oracle.adam_rem(grp, 1, hi, rem, m, v, np.array([0.5], np.float32), DT_F32, out)
    assert out[0] == 0x3F76 and rem[0] == 0 and m[0] == 0.25 and v[0] == 0.0625


# ---- remainders --------------------------------------------------------------

def _remainder_rows():
    rows = []
    with open(os.path.join(GOLDEN, "remainder_split.txt")) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b, c = line.split()
                rows.append((int(a, 16), int(b, 16), int(c)))
    return rows


def test_remainder_golden_rows():
    rows = _remainder_rows()
    bits = np.array([r[0] for r in rows], np.uint32)
    hi, rem = oracle.rem_split(bits)
    assert hi.tolist() == [r[1] for r in rows]
    assert rem.tolist() == [r[2] for r in rows]
    back = oracle.rem_pack(np.array([r[1] for r in rows], np.uint16),
                           np.array([r[2] for r in rows], np.int16))
    assert back.tolist() == [r[0] for r in rows]


def test_remainder_roundtrip_all_2pow32():
    """pack(split(x)) == x for every one of the 2^32 fp32 bit patterns.

    A left inverse on a finite set of the same size is a bijection, so this
    also gives split(pack(h, r)) == (h, r) for every (bf16, int16) pair.
    """
    L = oracle.lib()
    chunk = 1 << 22
    x = np.empty(chunk, np.uint32)
    hi = np.empty(chunk, np.uint16)
    rem = np.empty(chunk, np.int16)
    back = np.empty(chunk, np.uint32)
    base = np.arange(chunk, dtype=np.uint32)
    for start in range(0, 1 << 32, chunk):
        np.add(base, np.uint32(start), out=x)
        L.oracle_rem_split_n(chunk, x.ctypes.data, hi.ctypes.data, rem.ctypes.data)
        L.oracle_rem_pack_n(chunk, hi.ctypes.data, rem.ctypes.data, back.ctypes.data)
        if not np.array_equal(back, x):
            bad = np.nonzero(back != x)[0][0]
            pytest.fail(f"round trip breaks at 0x{int(x[bad]):08X}")


def test_remainder_high_half_is_nearest_bf16():
    """The split's high half is a nearest bf16 to the master, ties away from 0."""
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # every midpoint and near-midpoint low half for random high halves
    hs = rng.integers(0, 1 << 16, size=4096, dtype=np.uint64).astype(np.uint32)
    lows = np.array([0x7FFF, 0x8000, 0x8001, 0x0000, 0xFFFF], np.uint32)
    bits = np.concatenate([bits, ((hs[:, None] << 16) | lows[None, :]).ravel()])
    hi, _ = oracle.rem_split(bits)
    with np.errstate(invalid="ignore"):
        x = bits.view(np.float32).astype(np.float64)
        hv = (hi.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        trunc = ((bits >> 16) << 16).view(np.float32).astype(np.float64)
        up = (((bits >> 16) + 1) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    ok = np.isfinite(x) & np.isfinite(hv) & np.isfinite(up)
    x, hv, trunc, up = x[ok], hv[ok], trunc[ok], up[ok]
    other = np.where(hv == trunc, up, trunc)
    dh, do = np.abs(x - hv), np.abs(x - other)
    assert np.all(dh <= do)
    tie = dh == do
    assert np.all(np.abs(hv[tie]) >= np.abs(x[tie]))


# ---- conversions -------------------------------------------------------------

def _special_f32_bits():
    rng = np.random.default_rng(11)
    rnd = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    # rounding-relevant low-bit patterns under every exponent
    exps = np.arange(0, 256, dtype=np.uint32)
    mhi = rng.integers(0, 1 << 23, size=64, dtype=np.uint64).astype(np.uint32) & 0x7FE000
    lows = np.array([0, 1, 0xFFF, 0x1000, 0x1001, 0x1FFF, 0x7FFF, 0x8000, 0x8001, 0xFFFF],
                    np.uint32)
    grid = ((exps[:, None, None] << 23) | mhi[None, :, None] | lows[None, None, :]).ravel()
    fixed = np.array([0, 0x7F800000, 0x7FC00000, 0x7F800001, 0x477FE000, 0x477FEFFF,
                      0x477FF000, 0x477FF001, 0x38800000, 0x387FFFFF, 0x33000000, 0x33000001,
                      0x337FFFFF, 0x33800000, 0x7F7FFFFF, 0x7F7F8000, 0x00000001], np.uint32)
    return np.concatenate([rnd, grid, grid | 0x80000000, fixed, fixed | 0x80000000])


def test_bf16_rounding_matches_torch():
    x = _special_f32_bits().view(np.float32)
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(oracle.bf16_to_f32(ours[nan])))


def test_f16_rounding_matches_numpy():
    x = _special_f32_bits().view(np.float32)
    ours = oracle.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(oracle.f16_to_f32(ours[nan])))


def test_widening_all_16bit_patterns():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref_bf = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    ref_h = h.view(np.float16).astype(np.float32)
    for ours, ref in ((oracle.bf16_to_f32(h), ref_bf), (oracle.f16_to_f32(h), ref_h)):
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(ours), nan)
        assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ---- bias correction -----------------------------------------------------------

@pytest.mark.parametrize("beta", [0.5, 0.75, 0.9, 0.95, 0.999, 0.9999])
def test_bias_correction_is_correctly_rounded(beta):
    """1 - beta^k against its exact rational value rounded once to fp32."""
    b = Fraction(float(np.float32(beta)))
    for k in list(range(1, 40)) + [100, 1000]:
        want = np.float32(float(1 - b ** k))
        got = oracle.bias_correction(beta, k)
        # double pow is within a few double ulps; after the one rounding to
        # fp32 that can move the result by at most one fp32 ulp
        assert abs(float(got) - float(want)) <= float(np.spacing(want)), (beta, k, got, want)
    assert oracle.bias_correction(0.5, 3) == np.float32(0.875)
    assert oracle.bias_correction(0.5, 24) == np.float32(1 - 2.0 ** -24)


# ---- closed forms --------------------------------------------------------------

def _rand_problem(n, seed, gscale=1e-3):
    rng = np.random.default_rng(seed)
    p = rng.standard_normal(n).astype(np.float32)
    g = (rng.standard_normal(n) * gscale).astype(np.float32)
    # a spread of magnitudes, including grads near and below eps
    g[: n // 8] *= np.float32(1e-5)
    g[n // 8: n // 4] *= np.float32(1e3)
    return p, g


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_closed_form_adamw_step1(wd):
    """AdamW, bias correction on, zero moments: m^ = sg and v^ = sg^2 at step 1,
    so p1 = p0 - lr*(sg/(|sg|+eps) + wd*p0)."""
    n = 50_000
    p0, g = _rand_problem(n, 1)
    grp = Group(mode=MODE_ADAMW, bias_correction=1, beta1=0.9, beta2=0.95, eps=1e-8,
                weight_decay=wd, lr=1.6e-3, grad_scale=0.5)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.adam_f32(grp, 1, p, m, v, g, DT_F32)
    sg = g.astype(np.float64) * 0.5
    eps = float(np.float32(1e-8))
    lr, wdd = float(np.float32(1.6e-3)), float(np.float32(wd))
    u = sg / (np.abs(sg) + eps) + wdd * p0
    want = p0 - lr * u
    tol = _ulp(want) + lr * (np.abs(u) + 1.0) * 32 * F32_EPS
    assert np.all(np.abs(p - want) <= tol)


def test_closed_form_l2_step1():
    """L2 mode at step 1: s = g*gs + wd*p0 and p1 = p0 - lr*s/(|s|+eps)."""
    n = 50_000
    p0, g = _rand_problem(n, 2, gscale=1e-2)
    grp = Group(mode=MODE_L2, bias_correction=1, beta1=0.9, beta2=0.95, eps=1e-8,
                weight_decay=0.1, lr=1e-3, grad_scale=1.0 / 65536)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.adam_f32(grp, 1, p, m, v, g, DT_F32)
    s = g.astype(np.float64) * (1.0 / 65536) + float(np.float32(0.1)) * p0
    lr = float(np.float32(1e-3))
    want = p0 - lr * s / (np.abs(s) + float(np.float32(1e-8)))
    assert np.all(np.abs(p - want) <= _ulp(want) + lr * 32 * F32_EPS)
    # the first moment is the first moving average of s
    assert np.allclose(m, (1 - float(np.float32(0.9))) * s, rtol=8 * F32_EPS, atol=0)


@pytest.mark.parametrize("bc", [1, 0])
def test_closed_form_constant_gradient_ten_steps(bc):
    """Constant gradient, zero initial moments, wd = 0: after k steps
    m_k = (1-b1^k) sg and v_k = (1-b2^k) sg^2 exactly, so each step moves p by
    lr*sg/(|sg|+eps) with bias correction, and by
    lr*(1-b1^k) sg/(sqrt(1-b2^k)|sg|+eps) without it."""
    n, K = 20_000, 10
    p0, g = _rand_problem(n, 3)
    b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))
    grp = Group(mode=MODE_ADAMW, bias_correction=bc, beta1=0.9, beta2=0.999, eps=1e-8,
                weight_decay=0.0, lr=1e-3, grad_scale=1.0)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    sg = g.astype(np.float64)
    want = p0.astype(np.float64)
    lr, eps = float(np.float32(1e-3)), float(np.float32(1e-8))
    for k in range(1, K + 1):
        oracle.adam_f32(grp, k, p, m, v, g, DT_F32)
        if bc:
            want = want - lr * sg / (np.abs(sg) + eps)
        else:
            want = want - lr * (1 - b1 ** k) * sg / (math.sqrt(1 - b2 ** k) * np.abs(sg) + eps)
        tol = K * _ulp(want) + lr * K * K * 16 * F32_EPS
        assert np.all(np.abs(p - want) <= tol), k
        assert np.allclose(m, (1 - b1 ** k) * sg, rtol=4 * k * F32_EPS, atol=1e-30)
        assert np.allclose(v, (1 - b2 ** k) * sg * sg, rtol=4 * k * F32_EPS, atol=1e-37)


def test_closed_form_adamw_decay_only():
    """Zero gradient, AdamW: the moments stay zero and the update is pure
    decay, p_k = p0 (1 - lr wd)^k."""
    n, K = 10_000, 10
    p0, _ = _rand_problem(n, 4)
    grp = Group(mode=MODE_ADAMW, bias_correction=1, beta1=0.9, beta2=0.95, eps=1e-8,
                weight_decay=0.1, lr=1.6e-3)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    g = np.zeros(n, np.float32)
    for k in range(1, K + 1):
        oracle.adam_f32(grp, k, p, m, v, g, DT_F32)
    a = float(np.float32(1.6e-3)) * float(np.float32(0.1))
    want = p0.astype(np.float64) * (1 - a) ** K
    assert np.all(np.abs(p - want) <= 2 * K * _ulp(want))
    assert not m.any() and not v.any()


def test_double_evaluation_closed_forms():
    """The double evaluation meets the AdamW recursion with m^ = sg, v^ = sg^2
    (constant gradient) to double rounding over ten steps."""
    n = 20_000
    p0, g = _rand_problem(n, 5)
    grp = Group(mode=MODE_ADAMW, bias_correction=1, beta1=0.9, beta2=0.95, eps=1e-8,
                weight_decay=0.1, lr=1e-3, grad_scale=1.0)
    lr, wd, eps = (float(np.float32(x)) for x in (1e-3, 0.1, 1e-8))
    pd, md, vd = p0.astype(np.float64), np.zeros(n), np.zeros(n)
    sg = g.astype(np.float64)
    want = p0.astype(np.float64)
    for k in range(1, 11):
        oracle.adam_f64(grp, k, pd, md, vd, sg)
        want = want - lr * (sg / (np.abs(sg) + eps) + wd * want)
        assert np.all(np.abs(pd - want) <= 1e-13 * (np.abs(want) + 1.0)), k


def test_double_evaluation_agrees_with_fp32():
    """fp32 and double evaluations stay within the fp32 rounding the
    recursion accumulates: each step rounds p at the scale of |p| and the
    moving averages at the scale of their two terms."""
    n, K = 30_000, 10
    p0, g = _rand_problem(n, 5)
    for mode in (MODE_ADAMW, MODE_L2):
        grp = Group(mode=mode, bias_correction=1, beta1=0.9, beta2=0.95, eps=1e-8,
                    weight_decay=0.1, lr=1e-3, grad_scale=1.0)
        p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        pd, md, vd = p0.astype(np.float64), np.zeros(n), np.zeros(n)
        pscale = np.abs(p0).astype(np.float64)
        sgmax = np.abs(g).astype(np.float64)
        if mode == MODE_L2:
            sgmax = sgmax + 0.1 * (np.abs(p0) + 0.02)
        for k in range(1, K + 1):
            oracle.adam_f32(grp, k, p, m, v, g, DT_F32)
            oracle.adam_f64(grp, k, pd, md, vd, g.astype(np.float64))
            pscale = np.maximum(pscale, np.abs(pd))
        assert np.all(np.abs(p - pd) <= 2 * K * F32_EPS * pscale + 1e-3 * K * 64 * F32_EPS)
        assert np.all(np.abs(m - md) <= 8 * K * F32_EPS * (np.abs(md) + sgmax))
        assert np.all(np.abs(v - vd) <= 8 * K * F32_EPS * (np.abs(vd) + sgmax ** 2))


# ---- dtypes of g and p_out -----------------------------------------------------

@pytest.mark.parametrize("out_dtype", [DT_F32, DT_BF16, DT_F16])
@pytest.mark.parametrize("g_dtype", [DT_F32, DT_BF16, DT_F16])
def test_grad_widening_and_param_out_cast(g_dtype, out_dtype):
    n = 4096
    p0, g32 = _rand_problem(n, 6)
    if g_dtype == DT_F32:
        g, g_as_f32 = g32, g32
    elif g_dtype == DT_BF16:
        gt = torch.from_numpy(g32).to(torch.bfloat16)
        g = gt.view(torch.int16).numpy().view(np.uint16)
        g_as_f32 = gt.float().numpy()
    else:
        g = g32.astype(np.float16).view(np.uint16)
        g_as_f32 = g32.astype(np.float16).astype(np.float32)
    grp = Group(mode=MODE_ADAMW, weight_decay=0.1, lr=1e-3)
    # the update with a low-precision grad equals the update with its exact fp32 value
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    out = np.zeros(n, np.float32 if out_dtype == DT_F32 else np.uint16)
    oracle.adam_f32(grp, 1, p, m, v, g, g_dtype, out, out_dtype)
    p2, m2, v2 = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.adam_f32(grp, 1, p2, m2, v2, g_as_f32, DT_F32)
    assert np.array_equal(p, p2) and np.array_equal(m, m2) and np.array_equal(v, v2)
    if out_dtype == DT_F32:
        assert np.array_equal(out, p)
    elif out_dtype == DT_BF16:
        ref = torch.from_numpy(p.copy()).to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(out, ref.view(np.uint16))
    else:
        assert np.array_equal(out, p.astype(np.float16).view(np.uint16))


def test_remainder_update_composes_pack_update_split():
    n = 8192
    rng = np.random.default_rng(8)
    hi = torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(torch.bfloat16)
    hi = hi.view(torch.int16).numpy().view(np.uint16).copy()
    rem = rng.integers(-32768, 32768, size=n).astype(np.int16)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    grp = Group(mode=MODE_ADAMW, weight_decay=0.1, beta1=0.9, beta2=0.95, lr=1e-3)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    out = np.zeros(n, np.uint16)
    r2 = rem.copy()
    oracle.adam_rem(grp, 1, hi, r2, m, v, g, DT_F32, out)
    master = oracle.rem_pack(hi, rem).view(np.float32).copy()
    m3, v3 = np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.adam_f32(grp, 1, master, m3, v3, g, DT_F32)
    h3, r3 = oracle.rem_split(master.view(np.uint32))
    assert np.array_equal(out, h3) and np.array_equal(r2, r3)
    assert np.array_equal(m, m3) and np.array_equal(v, v3)


# ---- inf/nan screen ------------------------------------------------------------

def test_nonfinite_screen_special_cases():
    f = np.ones(100, np.float32)
    assert not oracle.any_nonfinite(f, DT_F32, 1.0)
    for bad in (np.inf, -np.inf, np.nan):
        h = f.copy()
        h[57] = bad
        assert oracle.any_nonfinite(h, DT_F32, 1.0)
    big = f.copy()
    big[3] = 3e38
    assert not oracle.any_nonfinite(big, DT_F32, 1.0)
    assert oracle.any_nonfinite(big, DT_F32, 10.0)  # overflows once scaled
    bf = np.full(10, 0x3F80, np.uint16)
    assert not oracle.any_nonfinite(bf, DT_BF16, 1.0)
    bf[9] = 0x7F80
    assert oracle.any_nonfinite(bf, DT_BF16, 1.0)
    h16 = np.full(10, 0x7BFF, np.uint16)  # 65504, the largest fp16
    assert not oracle.any_nonfinite(h16, DT_F16, 1.0)
    h16[0] = 0x7C00
    assert oracle.any_nonfinite(h16, DT_F16, 1.0)
    assert not oracle.any_nonfinite(np.zeros(0, np.float32), DT_F32, 1.0)


# ---- shard step: noop and step counters ----------------------------------------

def _small_shard(seed=9, with_empty=True, shared=False):
    rng = np.random.default_rng(seed)
    groups = [Group(mode=MODE_ADAMW, weight_decay=0.01), Group(mode=MODE_L2, weight_decay=0.0)]
    if with_empty:
        groups.append(Group(mode=MODE_ADAMW))
    tensors = []
    for i, n in enumerate([1000, 4097, 3]):
        tensors.append(oracle.Tensor(group=i % 2, p=rng.standard_normal(n).astype(np.float32),
                                     m=np.zeros(n, np.float32), v=np.zeros(n, np.float32),
                                     g=(rng.standard_normal(n) * 1e-3).astype(np.float32)))
    slot = [0] * len(groups) if shared else []
    return oracle.Shard(groups=groups, tensors=tensors, step_slot=slot)


def _snapshot(shard):
    return [(t.p.copy(), t.m.copy(), t.v.copy()) for t in shard.tensors], list(shard.steps)


@pytest.mark.parametrize("capturable", [False, True])
def test_noop_leaves_everything_bit_identical(capturable):
    sh = _small_shard()
    oracle.shard_step(sh, capturable=capturable)
    before, steps = _snapshot(sh)
    assert oracle.shard_step(sh, capturable=capturable, noop=True) is True
    after, steps2 = _snapshot(sh)
    assert steps == steps2
    for a, b in zip(before, after):
        for x, y in zip(a, b):
            assert x.tobytes() == y.tobytes()


def test_nonfinite_grad_sets_noop_before_any_update():
    sh = _small_shard()
    oracle.shard_step(sh, capturable=True)
    sh.tensors[2].g[1] = np.inf  # the last tensor: a late screen would be too late
    before, steps = _snapshot(sh)
    assert oracle.shard_step(sh, capturable=True, check_finite=True) is True
    after, steps2 = _snapshot(sh)
    assert steps == steps2 == [1, 1, 1]
    for a, b in zip(before, after):
        for x, y in zip(a, b):
            assert x.tobytes() == y.tobytes()


def _golden_empty_group():
    with open(os.path.join(GOLDEN, "empty_group_steps.txt")) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    return {r[0]: (r[1], r[2]) for r in rows}


@pytest.mark.parametrize("capturable", [False, True])
def test_empty_group_advances_like_the_fixed_loop(capturable):
    want_groups, want_state = _golden_empty_group()["fixed"]
    rng = np.random.default_rng(0)
    t = oracle.Tensor(group=0, p=rng.standard_normal(4).astype(np.float32),
                      m=np.zeros(4, np.float32), v=np.zeros(4, np.float32),
                      g=np.ones(4, np.float32))
    sh = oracle.Shard(groups=[Group(), Group()], tensors=[t])
    for _ in range(3):
        oracle.shard_step(sh, capturable=capturable)
    got = ",".join(str(s) for s in oracle.group_steps(sh))
    assert got == want_groups == want_state


def test_capturable_steps_count_only_applied_steps():
    sh = _small_shard()
    for k in range(5):
        oracle.shard_step(sh, capturable=True, noop=(k == 2))
    assert oracle.group_steps(sh) == [4, 4, 4]


def test_shared_step_counter_advances_once_per_step():
    sh = _small_shard(shared=True)
    for _ in range(3):
        oracle.shard_step(sh, capturable=True)
    assert sh.steps == [3] and oracle.group_steps(sh) == [3, 3, 3]


def test_preadvanced_counter_is_used_as_is():
    a, b = _small_shard(), _small_shard()
    b.steps = [1, 1, 1]
    oracle.shard_step(a, capturable=True)
    oracle.shard_step(b, capturable=True, step_preadvanced=True)
    assert a.steps == b.steps == [1, 1, 1]
    for ta, tb in zip(a.tensors, b.tensors):
        assert ta.p.tobytes() == tb.p.tobytes()


# ---- 16-bit optimizer state (p, m, v of one dtype T) ----------------------------

@pytest.mark.parametrize("state_dtype", [DT_BF16, DT_F16])
@pytest.mark.parametrize("name,d", _worked_examples(), ids=[r[0] for r in _worked_examples()])
def test_worked_example_16bit_state_exact(name, d, state_dtype):
    """Every value of the worked examples has at most 8 significant bits, so
    it is exact in bf16 and fp16 as well and the 16-bit state path must give
    the same results bit for bit."""
    mode = MODE_ADAMW if d["mode"] == "adamw" else MODE_L2
    grp = Group(mode=mode, bias_correction=int(d["bc"]), beta1=float(d["beta1"]),
                beta2=float(d["beta2"]), eps=float(d["eps"]), weight_decay=float(d["wd"]),
                lr=float(d["lr"]), grad_scale=float(d["gs"]))
    conv = oracle.f32_to_bf16 if state_dtype == DT_BF16 else oracle.f32_to_f16
    back = oracle.bf16_to_f32 if state_dtype == DT_BF16 else oracle.f16_to_f32
    p, m, v = (conv(np.array([float(d[k])], np.float32)) for k in ("p", "m", "v"))
    g = np.array([float(d["g"])], np.float32)
    oracle.adam_state(grp, int(d["step"]), p, m, v, state_dtype, g, DT_F32)
    assert back(p)[0] == np.float32(d["p_new"]), name
    assert back(m)[0] == np.float32(d["m_new"]), name
    assert back(v)[0] == np.float32(d["v_new"]), name


@pytest.mark.parametrize("state_dtype", [DT_BF16, DT_F16])
def test_16bit_state_is_widen_update_round(state_dtype):
    """The 16-bit state update equals the fp32 update of the widened values,
    each result rounded to the state dtype by torch's own conversion."""
    n = 20_000
    rng = np.random.default_rng(12)
    tdt = torch.bfloat16 if state_dtype == DT_BF16 else torch.float16

    def to16(x):
        return torch.from_numpy(np.asarray(x, np.float32)).to(tdt).view(torch.int16).numpy().view(np.uint16)

    def to32(b):
        return torch.from_numpy(b.view(np.int16).copy()).view(tdt).float().numpy()

    p = to16(rng.standard_normal(n))
    m = to16(rng.standard_normal(n) * 1e-3)
    v = to16(np.abs(rng.standard_normal(n)) * 1e-6)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    grp = Group(mode=MODE_ADAMW, weight_decay=0.1, beta1=0.9, beta2=0.95, lr=1e-3)
    p32, m32, v32 = to32(p), to32(m), to32(v)
    out = np.zeros(n, np.uint16)
    oracle.adam_state(grp, 3, p, m, v, state_dtype, g, DT_F32, out, DT_BF16)
    oracle.adam_f32(grp, 3, p32, m32, v32, g, DT_F32)
    assert np.array_equal(p, to16(p32)) and np.array_equal(m, to16(m32))
    assert np.array_equal(v, to16(v32))
    ref_out = torch.from_numpy(p32.copy()).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(out, ref_out.view(np.uint16))


# ---- fp32 master with 16-bit moments (exp_avg_dtype = exp_avg_sq_dtype) ---------

@pytest.mark.parametrize("moment_dtype", [DT_BF16, DT_F16])
@pytest.mark.parametrize("name,d", _worked_examples(), ids=[r[0] for r in _worked_examples()])
def test_worked_example_16bit_moments_exact(name, d, moment_dtype):
    """The worked examples' moments are exact in bf16 and fp16, so an fp32
    master with 16-bit moments must reproduce them bit for bit too."""
    mode = MODE_ADAMW if d["mode"] == "adamw" else MODE_L2
    grp = Group(mode=mode, bias_correction=int(d["bc"]), beta1=float(d["beta1"]),
                beta2=float(d["beta2"]), eps=float(d["eps"]), weight_decay=float(d["wd"]),
                lr=float(d["lr"]), grad_scale=float(d["gs"]))
    conv = oracle.f32_to_bf16 if moment_dtype == DT_BF16 else oracle.f32_to_f16
    back = oracle.bf16_to_f32 if moment_dtype == DT_BF16 else oracle.f16_to_f32
    p = np.array([float(d["p"])], np.float32)
    m, v = (conv(np.array([float(d[k])], np.float32)) for k in ("m", "v"))
    g = np.array([float(d["g"])], np.float32)
    oracle.adam_moments(grp, int(d["step"]), p, m, v, moment_dtype, g, DT_F32)
    assert p[0] == np.float32(d["p_new"]), name
    assert back(m)[0] == np.float32(d["m_new"]), name
    assert back(v)[0] == np.float32(d["v_new"]), name


@pytest.mark.parametrize("moment_dtype", [DT_BF16, DT_F16])
def test_16bit_moments_are_widen_update_round(moment_dtype):
    """With 16-bit moments the fp32 master gets exactly the fp32 update of
    the widened moments, and the new moments are that update's moments
    rounded by torch's own conversion."""
    n = 20_000
    rng = np.random.default_rng(15)
    tdt = torch.bfloat16 if moment_dtype == DT_BF16 else torch.float16

    def to16(x):
        return torch.from_numpy(np.asarray(x, np.float32)).to(tdt).view(torch.int16).numpy().view(np.uint16)

    def to32(b):
        return torch.from_numpy(b.view(np.int16).copy()).view(tdt).float().numpy()

    p = rng.standard_normal(n).astype(np.float32)
    m = to16(rng.standard_normal(n) * 1e-3)
    v = to16(np.abs(rng.standard_normal(n)) * 1e-6)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    grp = Group(mode=MODE_ADAMW, weight_decay=0.1, beta1=0.9, beta2=0.95, lr=1e-3)
    p32, m32, v32 = p.copy(), to32(m), to32(v)
    out = np.zeros(n, np.uint16)
    oracle.adam_moments(grp, 3, p, m, v, moment_dtype, g, DT_F32, out, DT_BF16)
    oracle.adam_f32(grp, 3, p32, m32, v32, g, DT_F32)
    assert p.tobytes() == p32.tobytes()
    assert np.array_equal(m, to16(m32)) and np.array_equal(v, to16(v32))
    ref_out = torch.from_numpy(p32.copy()).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(out, ref_out.view(np.uint16))


def test_16bit_moments_in_a_shard_step():
    """shard_step takes the moments path for a tensor that names a moment dtype."""
    n = 300
    rng = np.random.default_rng(16)
    p = rng.standard_normal(n).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    m = np.zeros(n, np.uint16)
    v = np.zeros(n, np.uint16)
    sh = oracle.Shard(groups=[Group(mode=MODE_ADAMW, weight_decay=0.1, lr=1e-3)],
                      tensors=[oracle.Tensor(group=0, p=p, m=m, v=v, g=g,
                                             moment_dtype=DT_BF16)])
    ref = [p.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    for k in (1, 2):
        oracle.shard_step(sh, capturable=False)
        oracle.adam_f32(sh.groups[0], k, *ref, g, DT_F32)
        ref[1] = oracle.bf16_to_f32(oracle.f32_to_bf16(ref[1]))
        ref[2] = oracle.bf16_to_f32(oracle.f32_to_bf16(ref[2]))
    assert p.tobytes() == ref[0].tobytes()
    assert np.array_equal(oracle.bf16_to_f32(m), ref[1])
    assert np.array_equal(oracle.bf16_to_f32(v), ref[2])


def test_fp32_state_through_the_generic_path_matches_adam_f32():
    n = 5000
    p0, g = _rand_problem(n, 13)
    grp = Group(mode=MODE_L2, weight_decay=0.1, lr=1e-3)
    a = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    b = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    for k in (1, 2, 3):
        oracle.adam_f32(grp, k, *a, g, DT_F32)
        oracle.adam_state(grp, k, *b, DT_F32, g, DT_F32)
    for x, y in zip(a, b):
        assert x.tobytes() == y.tobytes()


# ---- gradient norm and clipping --------------------------------------------------

def test_sumsq_against_numpy_and_exact_cases():
    rng = np.random.default_rng(14)
    g = rng.standard_normal(100_003).astype(np.float32)
    want = float(np.sum(g.astype(np.float64) ** 2))  # numpy's pairwise float64 sum
    assert oracle.sumsq(g, DT_F32) == pytest.approx(want, rel=1e-13)
    # constant vectors: n * c^2 exactly
    assert oracle.sumsq(np.full(1000, 0.5, np.float32), DT_F32) == 250.0
    assert oracle.sumsq(np.full(7, 0x4000, np.uint16), DT_BF16) == 28.0  # bf16 2.0
    assert oracle.sumsq(np.full(9, 0x3C00, np.uint16), DT_F16) == 9.0    # fp16 1.0
    assert oracle.sumsq(np.zeros(0, np.float32), DT_F32) == 0.0
    bad = g.copy()
    bad[5] = np.inf
    assert oracle.sumsq(bad, DT_F32) == np.inf


def test_shard_norm_is_the_norm_of_the_scaled_concatenation():
    rng = np.random.default_rng(15)
    gs = [0.5, 2.0]
    groups = [Group(grad_scale=gs[0]), Group(grad_scale=gs[1]), Group()]
    tensors, cat = [], []
    for i, n in enumerate([1000, 17, 4096, 3]):
        g = rng.standard_normal(n).astype(np.float32)
        tensors.append(oracle.Tensor(group=i % 2, p=np.zeros(n, np.float32),
                                     m=np.zeros(n, np.float32), v=np.zeros(n, np.float32), g=g))
        cat.append(g.astype(np.float64) * gs[i % 2])
    sh = oracle.Shard(groups=groups, tensors=tensors)
    want = np.linalg.norm(np.concatenate(cat)) ** 2
    assert oracle.shard_sumsq(sh) == pytest.approx(want, rel=1e-12)


def test_clip_coefficient_cases():
    # below the threshold: coefficient clamped to 1, scale unchanged
    norm, inf, coef, gs = oracle.clip_from_sumsq(9.0, max_norm=5.0, grad_scale=0.25)
    assert norm == np.float32(3.0) and not inf and coef == np.float32(1.0) and gs == np.float32(0.25)
    # above: max_norm / (norm + 1e-6), in float
    norm, inf, coef, gs = oracle.clip_from_sumsq(100.0, max_norm=1.0, grad_scale=1.0)
    assert norm == np.float32(10.0)
    assert coef == np.float32(1.0) / (np.float32(10.0) + np.float32(1e-6))
    assert coef == pytest.approx(0.1, rel=1e-6) and gs == coef
    # a non-finite squared norm sets found_inf
    for bad in (np.inf, np.nan):
        assert oracle.clip_from_sumsq(bad, 1.0, 1.0)[1]
    assert np.isnan(oracle.clip_from_sumsq(np.nan, 1.0, 1.0)[0])
    assert np.isinf(oracle.clip_from_sumsq(np.inf, 1.0, 1.0)[0])
    # a norm beyond the float range is not finite either
    assert oracle.clip_from_sumsq(1e80, 1.0, 1.0)[1]
    # no clipping requested
    assert oracle.clip_from_sumsq(16.0, 0.0, 0.5)[2:] == (np.float32(1.0), np.float32(0.5))


# ---- the data-parallel exchange (one-GPU stand-in) -----------------------------

def _golden_reduce_rows():
    rows = []
    path = os.path.join(os.path.dirname(__file__), "golden", "reduce_sources.txt")
    with open(path) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, srcs = line.split("|")
            dt, op, expected = head.split()
            rows.append((dt, op, float(expected), [float(x) for x in srcs.split()]))
    return rows


_DT = {"f32": DT_F32, "bf16": DT_BF16, "f16": DT_F16}


def _to_dtype(x, dt):
    x = np.asarray(x, np.float32)
    if dt == DT_F32:
        return x
    return oracle.f32_to_bf16(x) if dt == DT_BF16 else oracle.f32_to_f16(x)


def _from_dtype(x, dt):
    if dt == DT_F32:
        return np.asarray(x, np.float32)
    return oracle.bf16_to_f32(x) if dt == DT_BF16 else oracle.f16_to_f32(x)


@pytest.mark.parametrize("row", _golden_reduce_rows(), ids=lambda r: f"{r[0]}-{r[1]}-{r[2]}")
def test_reduce_sources_golden_rows(row):
    dts, op, expected, values = row
    dt = _DT[dts]
    srcs = [_to_dtype([v], dt) for v in values]
    for s, v in zip(srcs, values):  # the fixture's inputs are exact in their dtype
        assert _from_dtype(s, dt)[0] == np.float32(v) or (np.isnan(v) and np.isnan(_from_dtype(s, dt)[0]))
    got = _from_dtype(oracle.reduce_sources(srcs, dt, op == "avg"), dt)[0]
    if np.isnan(expected):
        assert np.isnan(got)
    else:
        assert got == np.float32(expected) and np.signbit(got) == np.signbit(np.float32(expected))


def _round_f32_exact(q):
    """Nearest float32 to the rational q, ties to even, by exact comparison
    (independent of the oracle's float arithmetic)."""
    from fractions import Fraction
    r0 = np.float32(float(q))
    cands = [np.nextafter(r0, np.float32(-np.inf)), r0, np.nextafter(r0, np.float32(np.inf))]
    best = None
    for c in cands:
        d = abs(Fraction(float(c)) - q)
        key = (d, int(np.asarray(c, np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_reduce_sources_average_is_correctly_rounded_when_the_sum_is_exact():
    """Small-integer contributions: the float sum is exact, so the average
    must be the nearest float to the exact rational sum / R."""
    from fractions import Fraction
    rng = np.random.default_rng(16)
    for r in (3, 5, 6, 7, 12):
        srcs = [rng.integers(-1000, 1000, 500).astype(np.float32) for _ in range(r)]
        got = oracle.reduce_sources(srcs, DT_F32, True)
        total = np.sum(np.stack(srcs).astype(np.int64), axis=0)
        for i in range(0, 500, 7):
            want = _round_f32_exact(Fraction(int(total[i]), r))
            assert got[i] == want, (r, i)


def test_reduce_sources_invariants():
    rng = np.random.default_rng(17)
    x = rng.standard_normal(4096).astype(np.float32)
    # one rank, sum or average: the values themselves
    for avg in (False, True):
        assert oracle.reduce_sources([x], DT_F32, avg).tobytes() == x.tobytes()
    # two equal contributions averaged: x + x = 2x exactly, halved exactly
    assert oracle.reduce_sources([x, x], DT_F32, True).tobytes() == x.tobytes()
    # x and -x cancel to +0
    z = oracle.reduce_sources([x, -x], DT_F32, False)
    assert not np.any(z) and not np.any(np.signbit(z))
    # 16-bit: the result is the nearest-even rounding of the float result
    xb = oracle.f32_to_bf16(x)
    yb = oracle.f32_to_bf16(rng.standard_normal(4096).astype(np.float32))
    f = oracle.bf16_to_f32(xb) + oracle.bf16_to_f32(yb)
    assert np.array_equal(oracle.reduce_sources([xb, yb], DT_BF16, False), oracle.f32_to_bf16(f))


def _exchange_shard(seed, n=(3000, 17, 1024)):
    rng = np.random.default_rng(seed)
    tensors = []
    for i, k in enumerate(n):
        tensors.append(oracle.Tensor(group=i % 2, p=rng.standard_normal(k).astype(np.float32),
                                     m=np.zeros(k, np.float32), v=np.zeros(k, np.float32),
                                     g=np.zeros(k, np.uint16), g_dtype=DT_BF16,
                                     p_out=np.zeros(k, np.uint16), out_dtype=DT_BF16))
    groups = [Group(mode=MODE_ADAMW, weight_decay=0.1, lr=1e-3), Group(mode=MODE_L2, lr=1e-3)]
    return oracle.Shard(groups=groups, tensors=tensors)


def test_exchange_with_one_rank_is_the_plain_step():
    a, b = _exchange_shard(18), _exchange_shard(18)
    rng = np.random.default_rng(19)
    srcs = [[oracle.f32_to_bf16(rng.standard_normal(t.g.size).astype(np.float32) * 1e-2)]
            for t in a.tensors]
    for t, s in zip(b.tensors, srcs):
        t.g[...] = s[0]
    oracle.exchange_step(a, srcs, average=True, capturable=True)
    oracle.shard_step(b, capturable=True)
    for ta, tb in zip(a.tensors, b.tensors):
        for k in ("p", "m", "v", "g", "p_out"):
            assert getattr(ta, k).tobytes() == getattr(tb, k).tobytes()
    assert a.steps == b.steps


def test_exchange_noop_and_screen():
    rng = np.random.default_rng(20)
    sh = _exchange_shard(21)
    before = [(t.p.copy(), t.m.copy(), t.v.copy()) for t in sh.tensors]
    srcs = [[oracle.f32_to_bf16(rng.standard_normal(t.g.size).astype(np.float32))
             for _ in range(3)] for t in sh.tensors]
    # a set flag: the exchange still fills the gradient shard; nothing else moves
    assert oracle.exchange_step(sh, srcs, average=True, capturable=True, noop=True)
    for t, s, (p, m, v) in zip(sh.tensors, srcs, before):
        assert t.g.tobytes() == oracle.reduce_sources(s, DT_BF16, True).tobytes()
        assert t.p.tobytes() == p.tobytes() and t.m.tobytes() == m.tobytes()
    assert sh.steps == [0, 0]
    # an inf in one rank's contribution reaches the shard and the screen skips the step
    srcs[1][2][5] = 0x7F80  # bf16 +inf
    assert oracle.exchange_step(sh, srcs, average=True, capturable=True, check_finite=True)
    assert sh.steps == [0, 0]
    assert np.isinf(oracle.bf16_to_f32(sh.tensors[1].g)[5])


def test_gather_places_each_rank_shard():
    rng = np.random.default_rng(22)
    r, s = 4, 1000
    shards = [oracle.f32_to_bf16(rng.standard_normal(s).astype(np.float32)) for _ in range(r)]
    bucket = np.zeros(r * s, np.uint16)
    for k in range(r):
        bucket |= oracle.gather_param_out(shards[k], r, k)
    assert bucket.tobytes() == np.concatenate(shards).tobytes()


# ---- scaled optimizer state ------------------------------------------------------

def test_max_scaled_state_is_half_the_dtype_max():
    assert oracle.max_scaled_state(DT_BF16) == np.float32(torch.finfo(torch.bfloat16).max / 2)
    assert oracle.max_scaled_state(DT_F16) == np.float32(torch.finfo(torch.float16).max / 2)


def test_state_scale_hand_rows():
    # absmax 32752 * 2^-10: the scale is 2^-10 exactly, the reciprocal 1024,
    # and every scaled value is exact in fp16
    buf = np.float32([31.984375, -16.0, 2.0, 0.0])
    bits, scale = oracle.scale_state(buf, DT_F16)
    assert scale == np.float32(2.0 ** -10)
    assert list(oracle.f16_to_f32(bits)) == [32752.0, -16384.0, 2048.0, 0.0]
    # bf16: absmax (finfo.max / 2) * 2^-100 -> scale 2^-100, values exact
    top = np.float32(oracle.max_scaled_state(DT_BF16) * np.float32(2.0 ** -100))
    bits, scale = oracle.scale_state(np.float32([top, -top / 4]), DT_BF16)
    assert scale == np.float32(2.0 ** -100)
    assert list(oracle.bf16_to_f32(bits)) == [np.float32(oracle.max_scaled_state(DT_BF16)),
                                               np.float32(-oracle.max_scaled_state(DT_BF16) / 4)]
    # all zeros (of either sign): scale 0, reciprocal 0, zeros stored
    bits, scale = oracle.scale_state(np.float32([0.0, -0.0]), DT_F16)
    assert scale == 0 and not np.any(oracle.f16_to_f32(bits))
    # a NaN: the scale is NaN, the reciprocal 0; NaN stays NaN, the rest 0
    bits, scale = oracle.scale_state(np.float32([1.0, np.nan, -2.0]), DT_F16)
    v = oracle.f16_to_f32(bits)
    assert np.isnan(scale) and np.isnan(v[1]) and v[0] == 0 and v[2] == 0
    # an inf: scale inf, reciprocal 0, inf * 0 = NaN
    bits, scale = oracle.scale_state(np.float32([1.0, np.inf]), DT_BF16)
    v = oracle.bf16_to_f32(bits)
    assert np.isinf(scale) and np.isnan(v[1]) and v[0] == 0


def _page_rescale_in_torch(x: torch.Tensor, dtype: torch.dtype):
    """The page's rescale as torch operations on the CPU: absmax from aminmax,
    the scale against half the dtype's largest value, a reciprocal only
    where the scale is positive, the product, the cast."""
    lo, hi = torch.aminmax(x)
    absmax = torch.maximum(-lo, hi)
    scale = absmax / torch.tensor(torch.finfo(dtype).max / 2, dtype=torch.float32)
    rscale = torch.where(scale > 0, scale.reciprocal(), torch.zeros_like(scale))
    return (x * rscale).to(dtype), scale


@pytest.mark.parametrize("dt", [DT_BF16, DT_F16])
def test_state_scale_matches_the_pages_torch_operations(dt):
    tdt = torch.bfloat16 if dt == DT_BF16 else torch.float16
    rng = np.random.default_rng(23)
    for mag in (1e-12, 1e-3, 1.0, 1e4, 1e30):
        x = (rng.standard_normal(10_000) * mag).astype(np.float32)
        if dt == DT_F16 and mag > 1e4:
            continue
        want_bits, want_scale = _page_rescale_in_torch(torch.from_numpy(x), tdt)
        bits, scale = oracle.scale_state(x, dt)
        assert scale == np.float32(want_scale.item())
        assert bits.tobytes() == want_bits.view(torch.int16).numpy().tobytes()


@pytest.mark.parametrize("dt", [DT_BF16, DT_F16])
def test_scaled_step_is_unscale_step_rescale(dt):
    rng = np.random.default_rng(24)
    n = 5000
    tdt = torch.bfloat16 if dt == DT_BF16 else torch.float16
    # bf16's scale target (finfo.max / 2 ~ 1.7e38) leaves the reciprocal
    # finite only for absmax above ~0.5 (see the test below), so the moments
    # get magnitudes bf16 survives; fp16 takes Adam-like ones
    mm, vm = (1e-3, 1e-6) if dt == DT_F16 else (2.0, 4.0)
    p16, sp = oracle.scale_state(rng.standard_normal(n).astype(np.float32), dt)
    m16, sm = oracle.scale_state((rng.standard_normal(n) * mm).astype(np.float32), dt)
    v16, sv = oracle.scale_state((np.abs(rng.standard_normal(n)) * vm).astype(np.float32), dt)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    grp = Group(mode=MODE_ADAMW, weight_decay=0.1, beta1=0.9, beta2=0.95, lr=1e-3)
    # reference composition from pinned pieces: widen * scale, the fp32 step
    widen = oracle.bf16_to_f32 if dt == DT_BF16 else oracle.f16_to_f32
    p = widen(p16) * sp
    m = widen(m16) * sm
    v = widen(v16) * sv
    out_ref = np.zeros(n, np.uint16)
    oracle.adam_f32(grp, 4, p, m, v, g, DT_F32, out_ref, DT_BF16)
    scales = np.float32([sp, sm, sv])
    out = np.zeros(n, np.uint16)
    oracle.adam_scaled(grp, 4, p16, m16, v16, scales, dt, g, DT_F32, out, DT_BF16)
    assert out.tobytes() == out_ref.tobytes()  # param-out from the unrounded new param
    for bits, buf, k in ((p16, p, 0), (m16, m, 1), (v16, v, 2)):
        want_bits, want_scale = oracle.scale_state(buf, dt)
        assert bits.tobytes() == want_bits.tobytes()
        assert scales[k:k + 1].tobytes() == np.float32([want_scale]).tobytes()
        assert np.all(np.isfinite(widen(bits)))
        # and the stored state is the new value to within the dtype's precision
        back = widen(bits).astype(np.float64) * scales[k]
        rel = 2.0 ** -8 if dt == DT_BF16 else 2.0 ** -11
        assert np.all(np.abs(back - buf) <= rel * np.abs(buf) + 2.0 ** -24 * scales[k] * 65504)
    # an empty tensor is left alone
    e = np.zeros(0, np.uint16)
    s0 = np.float32([1, 2, 3])
    oracle.adam_scaled(grp, 1, e, e.copy(), e.copy(), s0, dt, np.zeros(0, np.float32))
    assert list(s0) == [1, 2, 3]


def test_bf16_scale_reciprocal_overflows_for_small_buffers():
    """The page's target finfo(bf16).max / 2 makes the scale of a buffer
    with absmax 1e-3 subnormal (about 5.9e-42) and its reciprocal overflow
    to inf: nonzero values are stored as inf and zeros as NaN (0 * inf),
    exactly as the page's torch operations do."""
    x = np.float32([1e-3, -5e-4, 0.0])
    bits, scale = oracle.scale_state(x, DT_BF16)
    assert 0 < scale < np.finfo(np.float32).tiny  # subnormal
    v = oracle.bf16_to_f32(bits)
    assert v[0] == np.inf and v[1] == -np.inf and np.isnan(v[2])
    want, want_scale = _page_rescale_in_torch(torch.from_numpy(x), torch.bfloat16)
    w = want.float().numpy()
    assert np.array_equal(np.isnan(v), np.isnan(w))  # NaN payloads are not compared
    assert np.array_equal(v[~np.isnan(v)], w[~np.isnan(w)])
    assert scale == np.float32(want_scale.item())
    # fp16's target 32752 keeps the same buffer exact to fp16 precision
    bits, scale = oracle.scale_state(x, DT_F16)
    assert np.all(np.isfinite(oracle.f16_to_f32(bits)))


def test_scaled_worked_example():
    """The AdamW worked example (p=1, g=0.5, m=v=0, step 1) reached through a
    power-of-two unscale: p stored as 0.5 with scale 2, m and v as zeros with
    scale 0; the fp32 step then gives the example's exact values, and the
    new param-out is their bf16 rounding."""
    rows = {r[0]: r[1] for r in _worked_examples()}
    name = next(k for k, d in rows.items() if d["mode"] == "adamw" and float(d["m"]) == 0
                and float(d["v"]) == 0 and int(d["step"]) == 1)
    d = rows[name]
    grp = Group(mode=MODE_ADAMW, bias_correction=int(d["bc"]), beta1=float(d["beta1"]),
                beta2=float(d["beta2"]), eps=float(d["eps"]), weight_decay=float(d["wd"]),
                lr=float(d["lr"]), grad_scale=float(d["gs"]))
    p16 = oracle.f32_to_f16(np.float32([float(d["p"]) / 2]))
    m16 = np.zeros(1, np.uint16)
    v16 = np.zeros(1, np.uint16)
    scales = np.float32([2.0, 0.0, 0.0])
    out = np.zeros(1, np.uint16)
    oracle.adam_scaled(grp, 1, p16, m16, v16, scales, DT_F16, np.float32([float(d["g"])]), DT_F32,
                       out, DT_BF16)
    assert out[0] == oracle.f32_to_bf16(np.float32([float(d["p_new"])]))[0]
    for bits, k, key in ((p16, 0, "p_new"), (m16, 1, "m_new"), (v16, 2, "v_new")):
        want_bits, want_scale = oracle.scale_state(np.float32([float(d[key])]), DT_F16)
        assert bits[0] == want_bits[0] and scales[k] == want_scale


def test_shard_step_dispatches_scaled_tensors():
    rng = np.random.default_rng(25)
    p16, sp = oracle.scale_state(rng.standard_normal(300).astype(np.float32), DT_F16)
    t = oracle.Tensor(group=0, p=p16, m=np.zeros(300, np.uint16), v=np.zeros(300, np.uint16),
                      g=(rng.standard_normal(300) * 1e-2).astype(np.float32), state_dtype=DT_F16,
                      scales=np.float32([sp, 0, 0]), p_out=np.zeros(300, np.uint16),
                      out_dtype=DT_BF16)
    ref = [p16.copy(), np.zeros(300, np.uint16), np.zeros(300, np.uint16), t.scales.copy()]
    grp = Group(mode=MODE_ADAMW, weight_decay=0.1, lr=1e-3)
    sh = oracle.Shard(groups=[grp], tensors=[t])
    oracle.shard_step(sh, capturable=False)
    oracle.adam_scaled(grp, 1, ref[0], ref[1], ref[2], ref[3], DT_F16, t.g, DT_F32,
                       np.zeros(300, np.uint16), DT_BF16)
    assert t.p.tobytes() == ref[0].tobytes() and t.scales.tobytes() == ref[3].tobytes()
    assert sh.steps == [1] and np.any(t.m)


@pytest.mark.parametrize("g_dtype,out_dtype", [(DT_F32, oracle.DT_NONE), (DT_BF16, DT_BF16),
                                               (DT_F16, DT_F32)])
@pytest.mark.parametrize("mode", [MODE_L2, MODE_ADAMW])
def test_timed_build_computes_what_the_parity_build_does(g_dtype, out_dtype, mode):
    """The benchmark's CPU baseline times a second build of the same oracle
    source (-O3 -fopenmp, vectorised, each tensor split across threads).  It
    must be the same function: bit-identical to the parity build, three
    steps of an odd-sized tensor, fp32 master and remainder forms."""
    rng = np.random.default_rng(31)
    n = 100_003
    grp = Group(mode=mode, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, lr=1.6e-3,
                grad_scale=0.5)
    g32 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g = {DT_F32: g32, DT_BF16: oracle.f32_to_bf16(g32), DT_F16: oracle.f32_to_f16(g32)}[g_dtype]
    p0 = rng.standard_normal(n).astype(np.float32)
    odt = {oracle.DT_NONE: None, DT_F32: np.float32, DT_BF16: np.uint16}[out_dtype]
    a = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    b = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    oa = np.zeros(n, odt) if odt else None
    ob = np.zeros(n, odt) if odt else None
    hi, rem = oracle.rem_split(p0.view(np.uint32))
    ra = [hi.copy(), rem.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    rb = [hi.copy(), rem.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    for k in (1, 2, 3):
        oracle.adam_f32(grp, k, *a, g, g_dtype, oa, out_dtype)
        oracle.adam_f32(grp, k, *b, g, g_dtype, ob, out_dtype, timed=True)
        oracle.adam_rem(grp, k, ra[0], ra[1], ra[2], ra[3], g, g_dtype, ra[0])
        oracle.adam_rem(grp, k, rb[0], rb[1], rb[2], rb[3], g, g_dtype, rb[0], timed=True)
    for x, y in zip(a + ra, b + rb):
        assert x.tobytes() == y.tobytes()
    if odt:
        assert oa.tobytes() == ob.tobytes()
    assert oracle.timed_lib().oracle_omp_threads() >= 1


# ---- gradient accumulation across reduce-scatters ---------------------------------

def _golden_accumulate_rows():
    rows = []
    path = os.path.join(os.path.dirname(__file__), "golden", "accumulate_grad.txt")
    with open(path) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, vals = line.split("|")
            dt, expected = head.split()
            old, synced = (float(x) for x in vals.split())
            rows.append((dt, float(expected), old, synced))
    return rows


@pytest.mark.parametrize("row", _golden_accumulate_rows(), ids=lambda r: f"{r[0]}-{r[1]}")
def test_accumulate_grad_golden_rows(row):
    dts, expected, old, synced = row
    dt = _DT[dts]
    a, b = _to_dtype([old], dt), _to_dtype([synced], dt)
    for x, v in ((a, old), (b, synced)):  # the fixture's inputs are exact in their dtype
        w = _from_dtype(x, dt)[0]
        assert w == np.float32(v) or (np.isnan(v) and np.isnan(w))
    got = _from_dtype(oracle.accumulate_grad(a, b, dt), dt)[0]
    if np.isnan(expected):
        assert np.isnan(got)
    else:
        assert got == np.float32(expected) and np.signbit(got) == np.signbit(np.float32(expected))


@pytest.mark.parametrize("dt", [DT_BF16, DT_F16])
def test_accumulate_grad_is_torch_add_in_the_grad_dtype(dt):
    """The page's grads_shard.add_(sync_grads_shard) on 16-bit tensors, run
    by torch on the CPU, against the oracle's accumulation."""
    rng = np.random.default_rng(41)
    tdt = torch.bfloat16 if dt == DT_BF16 else torch.float16
    a = (rng.standard_normal(20000) * 1e-2).astype(np.float32)
    b = (rng.standard_normal(20000) * 1e-2).astype(np.float32)
    ta, tb = torch.from_numpy(a).to(tdt), torch.from_numpy(b).to(tdt)
    want = ta.clone().add_(tb).view(torch.int16).numpy().view(np.uint16)
    ab = ta.view(torch.int16).numpy().view(np.uint16).copy()
    bb = tb.view(torch.int16).numpy().view(np.uint16).copy()
    assert np.array_equal(oracle.accumulate_grad(ab, bb, dt), want)


def test_reduce_into_composes_the_reduction_and_the_accumulation():
    rng = np.random.default_rng(42)
    old = oracle.f32_to_bf16(rng.standard_normal(3000).astype(np.float32))
    srcs = [oracle.f32_to_bf16(rng.standard_normal(3000).astype(np.float32)) for _ in range(3)]
    synced = oracle.reduce_sources(srcs, DT_BF16, True)
    assert np.array_equal(oracle.reduce_into(old, srcs, DT_BF16, True, False), synced)
    acc = oracle.reduce_into(old, srcs, DT_BF16, True, True)
    assert np.array_equal(acc, oracle.f32_to_bf16(oracle.bf16_to_f32(old) + oracle.bf16_to_f32(synced)))
    # accumulating a shard of +0 leaves every nonzero value as it was
    x = rng.standard_normal(3000).astype(np.float32)
    zero = np.zeros(3000, np.float32)
    assert oracle.accumulate_grad(x, zero, DT_F32).tobytes() == x.tobytes()
    # two micro-batches accumulated through the shard step equal the sum fed
    # to the plain step
    sh_a, sh_b = _exchange_shard(43), _exchange_shard(43)
    src1 = [[oracle.f32_to_bf16(rng.standard_normal(t.g.size).astype(np.float32)) for _ in range(2)]
            for t in sh_a.tensors]
    src2 = [[oracle.f32_to_bf16(rng.standard_normal(t.g.size).astype(np.float32)) for _ in range(2)]
            for t in sh_a.tensors]
    for t, s1 in zip(sh_a.tensors, src1):
        t.g[...] = oracle.reduce_sources(s1, DT_BF16, True)
    oracle.exchange_step(sh_a, src2, average=True, capturable=False, accumulate=True)
    for t, s1, s2 in zip(sh_b.tensors, src1, src2):
        t.g[...] = oracle.accumulate_grad(oracle.reduce_sources(s1, DT_BF16, True),
                                          oracle.reduce_sources(s2, DT_BF16, True), DT_BF16)
    oracle.shard_step(sh_b, capturable=False)
    for ta, tb in zip(sh_a.tensors, sh_b.tensors):
        assert ta.g.tobytes() == tb.g.tobytes() and ta.p.tobytes() == tb.p.tobytes()
