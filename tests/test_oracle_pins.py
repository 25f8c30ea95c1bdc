"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- hand-worked groups, the page's printed packing vector, closed
forms, exhaustive or exact-rational brute force, and library routines on special
cases that reduce to them.  No expected value here comes from the CUDA path."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from conftest import GOLDEN_DIR, parse_cases

CASES = parse_cases(os.path.join(GOLDEN_DIR, "hand_groups.txt"))


def _f32(bits):
    return np.array([int(bits, 16)], dtype=np.uint32).view(np.float32)[0]


def _group_from_case(case):
    vals = [_f32(b) for b in case["values"].split()]
    pad = _f32(case["pad"])
    g = np.full(128, pad, dtype=np.float32)
    g[: len(vals)] = vals
    return g, len(vals)


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_hand_worked_groups(oracle_mod, case, dtype):
    g, nv = _group_from_case(case)
    if dtype == "f16":
        if case["f16_exact"] != "1":
            pytest.skip("values not exact in fp16")
        assert np.array_equal(g.astype(np.float16).astype(np.float32), g)
        W = g.astype(np.float16)[None, :]
    else:
        W = g[None, :]
    # Put the hand-worked group second in a row of three groups, so that the
    # row/group indexing is exercised too; the other groups are plain N(0,1).
    rng = np.random.default_rng(7)
    row = rng.standard_normal(384).astype(W.dtype)
    row[128:256] = W[0]
    q, s16, z, s32 = oracle_mod.quantize_pack(row[None, :], with_fp32_scales=True)
    assert s32[0, 1].view(np.uint32) == int(case["scale_f32"], 16)
    assert s16[0, 1].view(np.uint16) == int(case["scale_f16"], 16)
    assert z[0, 1] == int(case["zero"])
    qq = oracle_mod.unpack(q, 384)[0, 128:256]
    exp_q = [int(x) for x in case["q"].split()]
    assert list(qq[:nv]) == exp_q
    assert np.all(qq[nv:] == int(case["q_pad"]))
    if "packed_prefix" in case:
        pref = [int(x, 16) for x in case["packed_prefix"].split()]
        packed = q[0, 64:128]
        assert list(packed[: len(pref)]) == pref
        assert np.all(packed[len(pref):] == int(case["packed_pad"], 16))


def test_pack_unpack_identity(oracle_mod):
    """Packing then unpacking returns the nibbles (the unpacker-integrity check of
    the pure-Python GPTQ page, 'Running and Testing It')."""
    rng = np.random.default_rng(11)
    W = (rng.standard_normal((37, 512)) * 0.3).astype(np.float32)
    q, s, z = oracle_mod.quantize_pack(W)
    nib = oracle_mod.unpack(q, 512)
    # Re-pack by the documented layout and compare bytes.
    repacked = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(repacked, q)
    assert nib.max() <= 15


def test_ranges_and_endpoints(oracle_mod):
    """zp and q in [0,15]; in an in-range group (min <= 0 <= max) the minimum maps
    to level 0 and the maximum to level 15, unless the zero-point tie pushed the top
    by exactly one level (then the max sits at 16 - 1 = 15 after the clip anyway)."""
    rng = np.random.default_rng(3)
    W = (rng.standard_normal((64, 1024)) * 0.05).astype(np.float16)
    q, s16, z, s32 = oracle_mod.quantize_pack(W, with_fp32_scales=True)
    nib = oracle_mod.unpack(q, 1024).reshape(64, 8, 128)
    Wg = W.astype(np.float32).reshape(64, 8, 128)
    assert z.max() <= 15 and nib.max() <= 15
    for n in range(64):
        for g in range(8):
            w = Wg[n, g]
            if w.min() <= 0 <= w.max() and w.min() < w.max():
                assert nib[n, g][np.argmin(w)] <= 1
                assert nib[n, g][np.argmax(w)] >= 14


def test_reconstruction_bound(oracle_mod):
    """|w - (q - zp) * s| <= s/2 (1 + 2^-20) for in-range groups, with the fp32 scale,
    and |w - (q - zp) * s16| <= s/2 (1 + 2^-20) + 15 |s - s16| with the stored one."""
    rng = np.random.default_rng(5)
    for dtype, sigma in ((np.float16, 0.02), (np.float32, 1.0)):
        W = (rng.standard_normal((96, 512)) * sigma).astype(dtype)
        q, s16, z, s32 = oracle_mod.quantize_pack(W, with_fp32_scales=True)
        nib = oracle_mod.unpack(q, 512).reshape(96, 4, 128).astype(np.float64)
        w = W.astype(np.float64).reshape(96, 4, 128)
        s = s32.astype(np.float64)[..., None]
        s_st = s16.astype(np.float64)[..., None]
        zz = z.astype(np.float64)[..., None]
        inr = (w.min(-1) <= 0) & (w.max(-1) >= 0)
        err = np.abs(w - (nib - zz) * s)
        bound = s / 2 * (1 + 2.0 ** -20)
        assert np.all(err[inr] <= np.broadcast_to(bound, err.shape)[inr])
        err16 = np.abs(w - (nib - zz) * s_st)
        b16 = bound + 15 * np.abs(s - s_st)
        assert np.all(err16[inr] <= np.broadcast_to(b16, err.shape)[inr])


def test_exact_rational_brute_force(oracle_mod):
    """For each element, with the exact rational quotient x = w/s (Fraction), the
    level q must be the integer in [0,15] nearest to x + zp (ties to even), except
    when x lies within 2^-20 |x| of a half-integer, where fp32 rounding of the
    quotient may legitimately decide.  zp is checked the same way from -min/s."""
    rng = np.random.default_rng(17)
    W = (rng.standard_normal((8, 256)) * 0.7).astype(np.float32)
    W[3, :128] += 3.0           # an all-positive group (zp clipped to 0)
    W[5, 128:] -= 4.0           # an all-negative group (zp clipped to 15)
    q, s16, z, s32 = oracle_mod.quantize_pack(W, with_fp32_scales=True)
    nib = oracle_mod.unpack(q, 256)

    def near_half(x):
        fl = math.floor(x)
        return abs(x - fl - Fraction(1, 2)) <= abs(x) * Fraction(1, 2 ** 20)

    checked = 0
    for n in range(8):
        for g in range(2):
            w = W[n, 128 * g:128 * g + 128]
            s = Fraction(float(s32[n, g]))
            mn = Fraction(float(w.min()))
            zx = -mn / s
            if not near_half(zx):
                # brute force over every level: the nearest one to the exact quotient
                cand = min(range(-64, 80), key=lambda j: (abs(zx - j), j % 2))
                assert z[n, g] == min(max(cand, 0), 15)
            for i in range(128):
                x = Fraction(float(w[i])) / s
                if near_half(x):
                    continue
                # brute force: the nearest of all integers in a window around x
                c = math.floor(x)
                r = min(range(c - 2, c + 3), key=lambda j: (abs(x - j), j % 2))
                expect = min(max(r + int(z[n, g]), 0), 15)
                assert nib[n, 128 * g + i] == expect
                checked += 1
    assert checked > 1900


def test_unit_scale_reduces_to_builtin_round(oracle_mod):
    """Groups with min 0 and max 15 have s = 1 and zp = 0, so q = round(w) with
    ties to even -- exactly Python's built-in round().  Run over every fp16 value
    in [0, 15] (exhaustive)."""
    allv = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    vals = allv[(allv >= 0) & (allv <= 15)]
    per = 126
    ng = (len(vals) + per - 1) // per
    W = np.zeros((ng, 128), np.float32)
    W[:, 1] = 15.0
    body = np.zeros(ng * per, np.float32)
    body[: len(vals)] = vals
    W[:, 2:] = body.reshape(ng, per)
    q, s16, z, s32 = oracle_mod.quantize_pack(W, with_fp32_scales=True)
    assert np.all(s32 == 1.0) and np.all(z == 0)
    nib = oracle_mod.unpack(q, 128)[:, 2:].reshape(-1)[: len(vals)]
    expect = np.array([round(float(v)) for v in vals])
    assert np.array_equal(nib, expect)


def test_constant_groups(oracle_mod):
    """Constant groups take scale 1: zp = clip(round(-c)), q = clip(round(c) + zp)."""
    cs = np.array([0.0, -0.0, 0.3, -0.3, 0.5, -0.5, 1.5, -2.6, 7.0, -20.0, 20.0], np.float32)
    W = np.repeat(cs, 128).reshape(len(cs), 128)
    q, s16, z, s32 = oracle_mod.quantize_pack(W, with_fp32_scales=True)
    nib = oracle_mod.unpack(q, 128)
    assert np.all(s32 == 1.0)
    assert np.all(s16.view(np.uint16) == 0x3C00)
    for i, c in enumerate(cs):
        zr = min(max(round(-float(c)), 0), 15)
        assert z[i, 0] == zr
        assert np.all(nib[i] == min(max(round(float(c)) + zr, 0), 15))


def test_f16_conversions_against_numpy(oracle_mod):
    """The oracle's own binary16 codecs agree with numpy's (a library routine):
    widening exhaustively over all finite patterns, narrowing on a spread of fp32
    values including ties, subnormals and overflow."""
    for bits in list(range(0, 0x7C00, 37)) + [0x0001, 0x03FF, 0x0400, 0x7BFF, 0x8001, 0xFBFF]:
        ref = float(np.array([bits], np.uint16).view(np.float16)[0])
        assert oracle_mod.f16_to_f32(bits) == ref
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * 10,
        (rng.standard_normal(500) * 1e-6).astype(np.float32),    # subnormal range
        np.array([65504, 65519, 65520, 70000, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 0.1, 1 / 15], np.float32),
    ])
    for x in xs:
        with np.errstate(over="ignore"):
            ref = int(np.array([x], np.float32).astype(np.float16).view(np.uint16)[0])
        assert oracle_mod.f32_to_f16_bits(float(x)) == ref, x


def test_matmul_integer_special_case(oracle_mod):
    """With s = 1 and zp = 0 (groups spanning exactly [0, 15] in integers) the
    dequantized weights are the integers q; with small-integer activations the fp64
    result is exact and equals numpy's int64 matmul (a library routine)."""
    rng = np.random.default_rng(23)
    N, K, M = 9, 384, 5
    Wi = rng.integers(0, 16, size=(N, K))
    Wi[:, 0::128] = 0
    Wi[:, 1::128] = 15
    q, s16, z = oracle_mod.quantize_pack(Wi.astype(np.float32))
    assert np.all(s16 == 1.0) and np.all(z == 0)
    Ai = rng.integers(-8, 9, size=(M, K))
    A_bits = (Ai.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # exact in bf16
    Y, S = oracle_mod.matmul(A_bits, q, s16, z)
    assert np.array_equal(Y, (Ai @ Wi.T).astype(np.float64))
    assert np.array_equal(S, (np.abs(Ai) @ np.abs(Wi).T).astype(np.float64))


def test_fused_matmul_equals_explicit_dequant(oracle_mod):
    """The chunked fused matmul equals dequantize-then-matmul (numpy fp64 matmul,
    a library routine) on tiny non-square shapes, relative 1e-12.  The shapes use
    more than one chunk of 256 output rows."""
    rng = np.random.default_rng(29)
    N, K, M = 300, 256, 3
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    q, s16, z = oracle_mod.quantize_pack(W)
    A = (rng.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    Y, S = oracle_mod.matmul(A, q, s16, z)
    Wd = oracle_mod.dequantize(q, s16, z, K)
    Af = (A.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Yd = Af @ Wd.T
    assert np.allclose(Y, Yd, rtol=1e-12, atol=1e-15)
    assert np.all(S >= np.abs(Y) * (1 - 1e-12))
    assert np.allclose(S, np.abs(Af) @ np.abs(Wd).T, rtol=1e-12)
    # sampled entries agree with the full result
    mi = np.array([0, 2, 1, 2]); ni = np.array([0, 299, 256, 17])
    Ye, Se = oracle_mod.matmul_entries(A, q, s16, z, mi, ni)
    assert np.array_equal(Ye, Y[mi, ni]) and np.array_equal(Se, S[mi, ni])


def test_dequant_hand_values(oracle_mod):
    """Reconstruction of the hand-worked groups: H1 (s16 = 1, zp = 8) gives q - 8;
    H4b gives -3 everywhere; H2 gives (q - 8) * 0.0999755859375."""
    by = {c["name"]: c for c in CASES}
    g1, _ = _group_from_case(by["H1"])
    g4, _ = _group_from_case(by["H4b"])
    g2, _ = _group_from_case(by["H2"])
    W = np.stack([g1, g4, g2])
    q, s16, z = oracle_mod.quantize_pack(W)
    d = oracle_mod.dequantize(q, s16, z, 128)
    assert list(d[0, :6]) == [-8.0, 0.0, 0.0, 2.0, 2.0, 7.0]
    assert np.all(d[1] == -3.0)
    assert list(d[2, :3]) == [-8 * 0.0999755859375, 7 * 0.0999755859375, 0.0]


def test_tolerance_closed_forms(oracle_mod):
    """ulp of bf16 (8 significant bits): 2^(e-7) in the binade [2^e, 2^(e+1)),
    2^-133 at zero and in the subnormal range."""
    u = oracle_mod.ulp_bf16(np.array([1.0, 1.5, 1.99, 2.0, 3.0, 0.0, 2.0 ** -130, -4.0]))
    assert list(u) == [2.0 ** -7, 2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -6,
                       2.0 ** -133, 2.0 ** -133, 2.0 ** -5]
    Yref = np.array([1.0, -3.0, 0.0])
    S = np.array([2.0, 3.0, 0.0])
    bits = np.array([0x3F80, 0xC040, 0x0000], np.uint16)   # 1.0, -3.0, 0.0 exactly
    ok, worst, _ = oracle_mod.check_y(bits, Yref, S)
    assert ok and worst == 0.0
    # one bf16 step off on 1.0 (1.0078125): error 2^-7 > 8e-3*2 + 2^-8? 0.0078 < 0.0199 -> ok
    ok, _, _ = oracle_mod.check_y(np.array([0x3F81, 0xC040, 0x0000], np.uint16), Yref, S)
    assert ok
    # error above the bound fails
    ok, _, _ = oracle_mod.check_y(np.array([0x3F90, 0xC040, 0x0000], np.uint16), Yref, S)
    assert not ok
    # a nonzero output where the reference is exactly 0 with S = 0 fails
    ok, _, _ = oracle_mod.check_y(np.array([0x3F80, 0xC040, 0x0001], np.uint16), Yref, S)
    assert not ok


# ---- symmetric variant and 16-bit dequantize ----------------------------------------
SYM_CASES = parse_cases(os.path.join(GOLDEN_DIR, "sym_groups.txt"))


@pytest.mark.parametrize("case", SYM_CASES, ids=[c["name"] for c in SYM_CASES])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_symmetric_hand_worked_groups(oracle_mod, case, dtype):
    """Hand-worked symmetric groups (tests/golden/sym_groups.txt), placed second in a
    row of three groups."""
    g, nv = _group_from_case(case)
    if dtype == "f16":
        assert case["f16_exact"] == "1"
        assert np.array_equal(g.astype(np.float16).astype(np.float32), g)
        W = g.astype(np.float16)[None, :]
    else:
        W = g[None, :]
    rng = np.random.default_rng(8)
    row = rng.standard_normal(384).astype(W.dtype)
    row[128:256] = W[0]
    q, s16, z, s32 = oracle_mod.quantize_pack(row[None, :], with_fp32_scales=True, symmetric=True)
    assert s32[0, 1].view(np.uint32) == int(case["scale_f32"], 16)
    assert s16[0, 1].view(np.uint16) == int(case["scale_f16"], 16)
    assert np.all(z == 8)
    qq = oracle_mod.unpack(q, 384)[0, 128:256]
    assert list(qq[:nv]) == [int(x) for x in case["q"].split()]
    assert np.all(qq[nv:] == int(case["q_pad"]))


def test_symmetric_odd_symmetry(oracle_mod):
    """Negating W mirrors every level about the zero point (level -> 16 - level) and
    keeps the scales: round-half-even and the clip are odd functions.  A dropped sign,
    a round-half-up or an offset other than 8 breaks it."""
    rng = np.random.default_rng(11)
    for dt in (np.float16, np.float32):
        W = (rng.standard_normal((8, 512)) * 0.02).astype(dt)
        W[rng.random(W.shape) < 0.01] *= 10
        q1, s1, z1 = oracle_mod.quantize_pack(W, symmetric=True)
        q2, s2, z2 = oracle_mod.quantize_pack(-W, symmetric=True)
        l1 = oracle_mod.unpack(q1, 512).astype(int)
        l2 = oracle_mod.unpack(q2, 512).astype(int)
        assert np.array_equal(s1.view(np.uint16), s2.view(np.uint16))
        assert np.array_equal(l2, 16 - l1)
        assert np.all(z1 == 8) and np.all(z2 == 8)


def test_symmetric_bounds(oracle_mod):
    """Levels in [1, 15]; each element within half a step (fp32 scale) of (level - 8) *
    scale, up to the fp32 quotient's rounding; the largest |w| of a group maps to level
    1 or 15 (q = -7 or 7)."""
    rng = np.random.default_rng(12)
    W = (rng.standard_normal((16, 1024)) * 0.02).astype(np.float32)
    W[rng.random(W.shape) < 0.001] *= 10
    q, s16, z, s32 = oracle_mod.quantize_pack(W, with_fp32_scales=True, symmetric=True)
    lv = oracle_mod.unpack(q, 1024).astype(np.float64)
    assert lv.min() >= 1 and lv.max() <= 15
    s = np.repeat(s32.astype(np.float64), 128, axis=1)
    err = np.abs(W.astype(np.float64) - (lv - 8) * s)
    assert np.all(err <= s * (0.5 + 2.0 ** -20))
    g = np.abs(W).reshape(16, 8, 128)
    top = np.take_along_axis(lv.reshape(16, 8, 128), g.argmax(axis=2)[..., None], axis=2)
    assert np.all((top == 1) | (top == 15))


def test_bf16_rounding_against_torch(oracle_mod):
    """binary32 -> bfloat16 rounding against torch's CPU conversion (round to nearest
    even): random magnitudes over the whole exponent range, exact ties, values that
    carry into the next binade, zeros, subnormals and overflow to infinity."""
    import torch
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(4000) * 10.0 ** rng.integers(-37, 37, 4000)).astype(np.float32)
    ties = (rng.standard_normal(1000).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    carry = np.array([0x3F7FFFFF, 0x3FFFFFFF, 0x7F7FFFFF, 0x7F7F8000, 0x00008000, 0x00018000,
                      0x00000001, 0x807FFFFF, 0x80000000, 0x00000000, 0x3F808000, 0x3F818000],
                     np.uint32)
    x = np.concatenate([x, ties.view(np.float32), carry.view(np.float32)])
    ours = oracle_mod.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("out", ["bf16", "fp16"])
def test_dequantize16_is_the_exact_product_rounded_once(oracle_mod, out):
    """The 16-bit dequantize equals the fp64 dequantize (pinned above) rounded by a
    library: numpy's float64 -> float16 and torch's float64 -> bfloat16 conversions
    (round to nearest even).  Scales span subnormal to large fp16 values, so fp16
    outputs include subnormals and overflow to infinity."""
    import torch
    rng = np.random.default_rng(9)
    N, K = 16, 512
    q = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    mag = 10.0 ** rng.integers(-7, 4, (N, K // 128))
    s = (rng.standard_normal((N, K // 128)) * mag).astype(np.float16)
    s[0, 0] = np.float16(8000.0)          # 15 * 8000 overflows fp16
    z = rng.integers(0, 16, (N, K // 128), dtype=np.uint8)
    z[0, 0] = 0
    exact = oracle_mod.dequantize(q, s, z, K)
    got = oracle_mod.dequantize16(q, s, z, K, out)
    if out == "fp16":
        with np.errstate(over="ignore"):
            ref = exact.astype(np.float16).view(np.uint16)
        assert np.isinf(got.view(np.float16)).any()
    else:
        ref = torch.from_numpy(exact).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ---- clip-range calibration ("Building a From-Scratch Group-Wise INT4 Quantization Layer
# for LLaMA Weights", Step 4) ------------------------------------------------------------
def calib_group(name):
    k = np.arange(128)
    if name == "ramp":
        return ((k + 1) / 128.0 * np.where(k % 2 == 0, 1.0, -1.0)).astype(np.float32)
    if name == "grid":
        base = np.concatenate([np.arange(1, 8), -np.arange(1, 8)]) / 64.0
        return np.resize(base, 128).astype(np.float32)
    if name == "constant":
        return (np.float32(0.3) * np.where(k % 3 == 0, -1.0, 1.0)).astype(np.float32)
    if name == "zeros":
        return np.zeros(128, np.float32)
    if name == "tie":
        w = np.zeros(128, np.float32)
        w[[0, 5]], w[1] = 1.0, -1.0
        return w
    raise KeyError(name)


CALIB_CASES = parse_cases(os.path.join(GOLDEN_DIR, "calib_groups.txt"))


@pytest.mark.parametrize("case", CALIB_CASES, ids=[c["name"] for c in CALIB_CASES])
def test_calibration_hand_worked_groups(oracle_mod, case):
    w = calib_group(case["values"])
    param = float(case["param"])
    if case["method"] == "percentile":
        r = oracle_mod.percentile_abs(w, param)
        assert r == np.float32(float(case["r"]))
        s_exp = np.float32(1.0) if r == 0 else np.float32(r) / np.float32(7.0)
    else:
        s_exp = np.float32(float(case["s"]))
        assert oracle_mod.mse_step(w, int(param)) == s_exp
    q, s16, z, s32 = oracle_mod.quantize_pack_calibrated(w[None, :], case["method"], param,
                                                         with_fp32_scales=True)
    assert s32[0, 0] == s_exp and z[0, 0] == 8
    assert s16[0, 0] == s_exp.astype(np.float16)
    lv = oracle_mod.unpack(q, 128)[0].astype(np.int64)
    if case["name"] == "grid_mse":
        assert np.array_equal(lv - 8, np.rint(w * 64).astype(np.int64))
    if case["name"] == "constant_mse":
        assert np.array_equal(lv - 8, np.sign(w).astype(np.int64))
    if case["name"] == "zeros_mse":
        assert np.all(lv == 8)
    if case["name"] == "tie_mse":
        from fractions import Fraction
        step = Fraction(float(np.float32(1.0) / np.float32(999.0)))
        half_ulp = Fraction(1, 2 ** 26)          # fl(1/3) lies in [2^-2, 2^-1): ulp 2^-25
        assert abs(333 * step - Fraction(float(s_exp))) < half_ulp
        assert lv[0] == 11 and lv[1] == 5 and lv[5] == 11 and np.all(lv[2:5] == 8)


def test_percentile_100_is_the_absmax_quantizer(oracle_mod):
    """p = 100 takes the largest |w| as the range, s = absmax / 7: the pinned symmetric
    quantizer (whose [-8, 7] clip never binds when s = absmax / 7)."""
    rng = np.random.default_rng(51)
    W = (rng.standard_normal((64, 512)) * 0.02).astype(np.float16)
    W[3, :128] = 0
    a = oracle_mod.quantize_pack_calibrated(W, "percentile", 100.0)
    b = oracle_mod.quantize_pack(W, symmetric=True)
    for x, y in zip(a, b):
        assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))


@pytest.mark.parametrize("p", [0.5, 10.0, 50.0, 90.0, 99.0, 99.9, 100.0])
def test_percentile_matches_numpy_quantile(oracle_mod, p):
    """Against numpy's linear-interpolation quantile in fp64 (a library routine): the
    fp32 evaluation differs only by roundings, far below one order-statistic gap, so
    a wrong rank, sort order or interpolation weight fails."""
    rng = np.random.default_rng(int(p * 10) + 1)
    for _ in range(50):
        w = (rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 2)).astype(np.float32)
        r = float(oracle_mod.percentile_abs(w, p))
        ref = float(np.quantile(np.abs(w).astype(np.float64), p / 100.0, method="linear"))
        assert abs(r - ref) <= 1e-6 * np.abs(w).max(), (p, r, ref)


def _mse64(w, c):
    """The search's score of step c, in fp64 with exact quotients (independent of the
    fp32 evaluation order)."""
    w = w.astype(np.float64)
    lv = np.clip(np.rint(w / c), -7, 7)
    return np.mean((lv * c - w) ** 2)


def test_mse_choice_is_optimal_in_fp64(oracle_mod):
    """The chosen step lies on the candidate grid linspace(min|w|, max|w|, n) and, with
    its score recomputed in fp64, is within rounding of the best candidate's."""
    rng = np.random.default_rng(61)
    n = 1000
    for trial in range(40):
        w = (rng.standard_normal(128) * 0.02).astype(np.float32)
        if trial % 4 == 0:
            w[rng.integers(0, 128, 2)] *= 10            # outliers
        s = float(oracle_mod.mse_step(w, n))
        lo, hi = float(np.abs(w).min()), float(np.abs(w).max())
        grid = lo + np.arange(n) * (hi - lo) / (n - 1)
        i = int(np.argmin(np.abs(grid - s)))
        assert abs(grid[i] - s) <= 4e-7 * hi
        scores = np.array([_mse64(w, c) for c in grid])
        best = scores.min()
        assert _mse64(w, s) <= best * (1 + 1e-4) + 1e-30
        # the first minimum: no candidate before the chosen one scores clearly better
        assert np.all(scores[:i] >= _mse64(w, s) * (1 - 1e-4))


def test_mse_levels_and_clamp(oracle_mod):
    """Levels are clamp(rint(w / s), -7, 7) + 8 with the chosen fp32 step: checked in
    exact arithmetic (ties excluded), including values beyond 7.5 steps that clamp."""
    from fractions import Fraction
    rng = np.random.default_rng(71)
    W = (rng.standard_normal((16, 128)) * 0.02).astype(np.float32)
    W[:, 0] = 0.3  # a large outlier per group: the search clamps it rather than widen the step
    q, _, z, s32 = oracle_mod.quantize_pack_calibrated(W, "mse", 1000, with_fp32_scales=True)
    lv = oracle_mod.unpack(q, 128).astype(np.int64) - 8
    assert np.all(z == 8)
    clamped = 0
    for r in range(16):
        s = Fraction(float(s32[r, 0]))
        for k in range(128):
            x = Fraction(float(W[r, k])) / s
            fl = x.numerator // x.denominator
            frac = x - fl
            if abs(frac - Fraction(1, 2)) < Fraction(1, 1 << 20):
                continue
            nearest = fl + (1 if frac > Fraction(1, 2) else 0)
            exp = max(-7, min(7, nearest))
            clamped += exp != nearest
            assert lv[r, k] == exp
    assert clamped > 0


# ---- W4A8 ("Hands-On Build Guide: Group-Wise INT4 Weight-Only Quantization with
# Per-Channel Scale", Step 3 and Step 5) ----------------------------------------------------
def _bf16(x):
    import synth
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_act_int8_hand_rows(oracle_mod):
    """Hand-worked rows.  amax = 127 gives s_a = 1, so a_q = rint(a) with ties to even:
    2.5 -> 2, -3.5 -> -4, 0.5 -> 0, 1.5 -> 2.  amax = 254 gives s_a = 2: 1 / 2 = 0.5 -> 0,
    3 / 2 = 1.5 -> 2, 5 / 2 = 2.5 -> 2.  An all-zero row takes s_a = fl(1e-8) / 127 and
    a_q = 0.  amax = 1: s_a = fl(1/127), and the extreme elements land on +-127."""
    rows = np.zeros((4, 128), np.float32)
    rows[0, :7] = [127, 2.5, -3.5, 0.5, -0.5, 1.5, -127]
    rows[1, :5] = [254, 1, 3, 5, -254]
    rows[3, :3] = [1.0, -1.0, 0.25]
    aq, sa = oracle_mod.quantize_act_int8(_bf16(rows))
    assert list(aq[0, :7]) == [127, 2, -4, 0, 0, 2, -127] and np.all(aq[0, 7:] == 0)
    assert list(aq[1, :5]) == [127, 0, 2, 2, -127]
    assert sa[0] == 1.0 and sa[1] == 2.0
    assert sa[2] == np.float32(1e-8) / np.float32(127) and np.all(aq[2] == 0)
    assert sa[3] == np.float32(1.0) / np.float32(127.0)
    assert aq[3, 0] == 127 and aq[3, 1] == -127 and aq[3, 2] == 32   # 0.25 * 127 = 31.75 -> 32


def test_act_int8_exact_rounding_and_bounds(oracle_mod):
    """Each level is the nearest integer to a / s_a in exact arithmetic (ties excluded),
    |a_q| <= 127, the row's largest magnitude maps to +-127, and |a - a_q s_a| <= s_a / 2."""
    from fractions import Fraction
    import synth
    rng = np.random.default_rng(91)
    A = synth.f32_to_bf16_bits((rng.standard_normal((6, 384)) * 10.0 ** rng.integers(-3, 3, (6, 1)))
                               .astype(np.float32))
    aq, sa = oracle_mod.quantize_act_int8(A)
    a = oracle_mod.bf16_bits_to_f64(A)
    assert np.all(np.abs(aq.astype(int)) <= 127)
    for m in range(6):
        s = Fraction(float(sa[m]))
        assert abs(aq[m, np.argmax(np.abs(a[m]))]) == 127
        for k in range(384):
            x = Fraction(float(a[m, k])) / s
            fl = x.numerator // x.denominator
            frac = x - fl
            # the fp32 quotient is within half an ulp (2^-24 |x|) of x: skip near-ties
            if abs(frac - Fraction(1, 2)) <= abs(x) / (1 << 22) + Fraction(1, 1 << 40):
                continue
            assert aq[m, k] == fl + (1 if frac > Fraction(1, 2) else 0)
        # near a tie the fp32 quotient (within 127.5 * 2^-24 of a / s_a) may round to the
        # farther integer: |a / s_a - a_q| <= 1/2 + 2^-17
        assert np.all(np.abs(a[m] - aq[m] * float(sa[m])) <= float(sa[m]) / 2 * (1 + 2.0 ** -15))


def test_w4a8_matmul_integer_special_case(oracle_mod):
    """Integer weights (a group spanning [0, 15] exactly: s = 1, zp = 0) and s_a = 1
    (a row whose largest magnitude is 127): Y is the integer product a_q q, exact."""
    rng = np.random.default_rng(92)
    N, K, M = 20, 256, 3
    W = rng.integers(0, 16, (N, K)).astype(np.float16)
    W[:, ::128] = 0
    W[:, 1::128] = 15
    q, s, z = oracle_mod.quantize_pack(W)
    assert np.all(z == 0) and np.all(s == 1)
    A = rng.integers(-127, 128, (M, K)).astype(np.float32)
    A[:, 0] = 127
    aq, sa = oracle_mod.quantize_act_int8(_bf16(A))
    assert np.all(sa == 1) and np.array_equal(aq.astype(np.float32), A)
    Y, S = oracle_mod.w4a8_matmul(aq, sa, q, s, z)
    qi = oracle_mod.unpack(q, K).astype(np.int64)
    assert np.array_equal(Y, (aq.astype(np.int64) @ qi.T).astype(np.float64))
    assert np.array_equal(S, (np.abs(aq.astype(np.int64)) @ qi.T).astype(np.float64))


def test_w4a8_matmul_equals_w4a16_on_representable_activations(oracle_mod):
    """With s_a a power of two (largest magnitude 127 * 2^e), a_q * s_a is an exact bf16
    value, so the W4A8 product equals the pinned W4A16 product on those activations."""
    import synth
    W, _ = synth.make_random(70, 512, 1, seed=93)
    q, s, z = oracle_mod.quantize_pack(W)
    rng = np.random.default_rng(93)
    A = rng.standard_normal((4, 512)).astype(np.float32)
    A[:, 7] = 127 * np.float32(2.0) ** np.arange(-6, -2)       # row maxima 127 * 2^e
    A = np.clip(A, -A[:, 7:8], A[:, 7:8])
    aq, sa = oracle_mod.quantize_act_int8(_bf16(A))
    assert np.array_equal(sa, np.float32(2.0) ** np.arange(-6, -2))
    A2 = _bf16(aq.astype(np.float32) * sa[:, None])
    Y1, S1 = oracle_mod.w4a8_matmul(aq, sa, q, s, z)
    Y2, S2 = oracle_mod.matmul(A2, q, s, z)
    assert np.array_equal(Y1, Y2) and np.array_equal(S1, S2)


# ---- GPTQ ("Build a GPTQ INT4 Quantization Engine in Python/NumPy", Step 3) -------------
def test_gptq_hand_worked_feed(oracle_mod):
    case = parse_cases(os.path.join(GOLDEN_DIR, "gptq_cases.txt"))[0]
    K = 128
    U = np.eye(K, dtype=np.float32)
    U[0, 0], U[0, 1] = 2.0, -4.0
    w = np.zeros((1, K), np.float32)
    w[0, :4] = [0.5625, 1.25, -1.5, 2.25]
    q, s, z = oracle_mod.gptq_quantize(w, U)
    lv = oracle_mod.unpack(q, K)[0]
    exp = [int(x) for x in case["levels"].split()]
    assert list(lv[:4]) == exp and np.all(lv[4:] == int(case["rest"]))
    assert s[0, 0] == np.float16(float(case["scale"])) and z[0, 0] == int(case["zero"])
    q_rtn = oracle_mod.unpack(oracle_mod.quantize_pack(w)[0], K)[0]
    assert q_rtn[1] == 11 and lv[1] == 12          # the fed-forward error changed the level


@pytest.mark.parametrize("diag", [False, True])
def test_gptq_without_correlation_is_round_to_nearest(oracle_mod, diag):
    """With U diagonal (uncorrelated inputs) every fed-forward term is exactly zero, so
    GPTQ reduces to the pinned round-to-nearest quantizer."""
    import synth
    W, _ = synth.make_random(48, 512, 1, seed=95)
    U = np.eye(512, dtype=np.float32)
    if diag:
        U *= np.random.default_rng(95).uniform(0.5, 3.0, 512).astype(np.float32)
    for a, b in zip(oracle_mod.gptq_quantize(W, U), oracle_mod.quantize_pack(W)):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


def test_gptq_reduces_the_layer_error(oracle_mod):
    """GPTQ minimizes the layer-output error greedily: on correlated calibration inputs
    its H-weighted reconstruction error tr((W - W_hat) H (W - W_hat)^T) is well below
    round-to-nearest's, row by row.  A sign error or a transposed U in the update
    would raise it instead."""
    import synth
    rng = np.random.default_rng(96)
    K = 512
    X = rng.standard_normal((4096, K))
    X[:, 1:] += 0.9 * X[:, :-1]
    U = oracle_mod.gptq_factor(X)
    assert np.allclose(np.triu(U), U)
    W, _ = synth.make_random(64, K, 1, seed=96)
    H = X.T @ X / X.shape[0]

    def loss(q, s, z):
        D = W.astype(np.float64) - oracle_mod.dequantize(q, s, z, K)
        return np.einsum("nk,kl,nl->n", D, H, D)

    lg, lr = loss(*oracle_mod.gptq_quantize(W, U)), loss(*oracle_mod.quantize_pack(W))
    assert lg.mean() < 0.8 * lr.mean()
    assert np.mean(lg < lr) > 0.9


def test_gptq_factor_inverts_the_hessian(oracle_mod):
    """U^T U = H^-1 for the damped Hessian (checked in fp64 against numpy's inverse)."""
    rng = np.random.default_rng(97)
    X = rng.standard_normal((1000, 256))
    U = oracle_mod.gptq_factor(X).astype(np.float64)
    H = X.T @ X / 1000
    H += 1e-4 * np.mean(np.diag(H)) * np.eye(256)
    assert np.allclose(U.T @ U @ H, np.eye(256), atol=1e-4)


def test_w4a8_entries_equal_the_full_product(oracle_mod):
    import synth
    W, A = synth.make_random(40, 384, 5, seed=98)
    q, s, z = oracle_mod.quantize_pack(W)
    aq, sa = oracle_mod.quantize_act_int8(A)
    Y, S = oracle_mod.w4a8_matmul(aq, sa, q, s, z)
    mi, ni = np.repeat(np.arange(5), 40), np.tile(np.arange(40), 5)
    Ye, Se = oracle_mod.w4a8_matmul_entries(aq, sa, q, s, z, mi, ni)
    assert np.array_equal(Ye, Y[mi, ni]) and np.array_equal(Se, S[mi, ni])
