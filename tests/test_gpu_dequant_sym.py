"""GPU parity for the symmetric quantizer (w4_quantize_pack_sym) and the explicit
dequantize (w4_dequantize): bit-exact against the CPU oracle on the same seeded
inputs, through the C ABI (ctypes binding)."""
import os

import numpy as np
import pytest

from conftest import GOLDEN_DIR, parse_cases

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    from w4a16_matmul_asym_b300 import build
    build.build()
    import w4a16_matmul_asym_b300 as w4
    w4.load_library()
    return torch, w4, oracle_mod


def to_dev_w(torch, W):
    if W.dtype == np.float16:
        return torch.from_numpy(W).cuda()
    return torch.from_numpy(np.ascontiguousarray(W, np.float32)).cuda()


def gpu_sym(env, W):
    torch, w4, _ = env
    q, s, z = w4.quantize_pack(to_dev_w(torch, W), symmetric=True)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy(), z.cpu().numpy()


def assert_sym_equal(env, W):
    _, _, orc = env
    q, s, z = gpu_sym(env, W)
    qo, so, zo = orc.quantize_pack(W, symmetric=True)
    assert np.array_equal(s.view(np.uint16), so.view(np.uint16)), "scales differ"
    assert np.array_equal(z, zo), "zeros differ"
    if not np.array_equal(q, qo):
        bad = np.argwhere(q != qo)
        raise AssertionError(f"qweight differs at {len(bad)} bytes, first {bad[:5].tolist()}")


# ---- symmetric quantize ----------------------------------------------------------
@pytest.mark.parametrize("N,K,dtype", [(1, 128, np.float16), (3, 256, np.float32), (257, 384, np.float16),
                                       (100, 1152, np.float32), (33, 4096, np.float16),
                                       (4096, 4096, np.float16)])
def test_quantize_sym_random(env, N, K, dtype):
    import synth
    W, _ = synth.make_random(N, K, 1, seed=N + K)
    assert_sym_equal(env, W.astype(dtype))


def test_quantize_sym_llama7b_shape(env):
    import synth
    W, _ = synth.make_workload("llama7b_gemv")
    assert_sym_equal(env, W)


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_quantize_sym_hand_groups(env, dtype):
    """The hand-worked symmetric groups of tests/golden/sym_groups.txt, one per row."""
    cases = parse_cases(os.path.join(GOLDEN_DIR, "sym_groups.txt"))
    rows = []
    for c in cases:
        vals = np.array([int(b, 16) for b in c["values"].split()], np.uint32).view(np.float32)
        pad = np.array([int(c["pad"], 16)], np.uint32).view(np.float32)[0]
        g = np.full(256, pad, np.float32)
        g[: len(vals)] = vals
        g[128:] = np.linspace(-1, 1, 128, dtype=np.float32)
        rows.append(g)
    W = np.stack(rows).astype(dtype)
    assert_sym_equal(env, W)
    q, _, _ = gpu_sym(env, W)
    for r, c in enumerate(cases):
        lv = np.stack([q[r, :64] & 15, q[r, :64] >> 4], axis=1).reshape(-1)
        exp = [int(x) for x in c["q"].split()]
        assert list(lv[: len(exp)]) == exp


def test_quantize_sym_edge_values(env):
    """All-zero groups, a lone +-0, fp16 subnormals, +-65504, exact ties of w / s."""
    rng = np.random.default_rng(3)
    W = np.zeros((6, 512), np.float16)
    W[1, :128] = np.float16(-0.0)
    W[2, :128] = (rng.integers(-1023, 1024, 128) * 2.0 ** -24).astype(np.float16)   # subnormals
    W[3, :128] = np.float16(65504.0) * np.sign(rng.standard_normal(128)).astype(np.float16)
    W[4, :128] = (np.arange(128) - 64).astype(np.float16) * np.float16(0.5)          # ties at s = 64/7 * 0.5
    W[5] = rng.standard_normal(512).astype(np.float16)
    assert_sym_equal(env, W)


def test_quantize_sym_fp32_wide_range(env):
    rng = np.random.default_rng(4)
    W = (rng.standard_normal((64, 1024)) * 10.0 ** rng.integers(-30, 30, (64, 1))).astype(np.float32)
    assert_sym_equal(env, W)


def test_quantize_sym_fp32_tiny_scales(env):
    """Symmetric groups with absmax below ~2e-38 (scale without a finite reciprocal),
    including exact zeros, quantize bit-exactly."""
    from test_gpu_parity import tiny_scale_rows
    assert_sym_equal(env, tiny_scale_rows(np.random.default_rng(18)))


# ---- dequantize ---------------------------------------------------------------------
def run_dequant(env, q, s, z, dtype):
    torch, w4, _ = env
    out = w4.dequantize(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(z).cuda(),
                        dtype=torch.bfloat16 if dtype == "bf16" else torch.float16)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("out", ["bf16", "fp16"])
@pytest.mark.parametrize("N,K,sym", [(1, 128, False), (5, 384, True), (257, 1152, False), (1000, 4096, True),
                                     (3, 128, True)])
def test_dequantize_matches_oracle(env, out, N, K, sym):
    import synth
    _, _, orc = env
    W, _ = synth.make_random(N, K, 1, seed=7 * N + K)
    q, s, z = orc.quantize_pack(W, symmetric=sym)
    got = run_dequant(env, q, s, z, out)
    assert np.array_equal(got, orc.dequantize16(q, s, z, K, out))


@pytest.mark.parametrize("out", ["bf16", "fp16"])
def test_dequantize_extreme_scales(env, out):
    """Random levels, zero points and fp16 scales from subnormal to 65504: fp16 output
    reaches subnormals and overflows to +-inf, bf16 keeps every value finite."""
    _, _, orc = env
    rng = np.random.default_rng(21)
    N, K = 64, 1024
    q = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    bits = rng.integers(0, 0x7C00, (N, K // 128)).astype(np.uint16)         # every finite positive fp16
    bits |= (rng.integers(0, 2, bits.shape).astype(np.uint16) << 15)        # both signs
    s = bits.view(np.float16)
    z = rng.integers(0, 16, (N, K // 128), dtype=np.uint8)
    got = run_dequant(env, q, s, z, out)
    assert np.array_equal(got, orc.dequantize16(q, s, z, K, out))


@pytest.mark.parametrize("out", ["bf16", "fp16"])
def test_dequantize_full_size(env, out):
    """Llama-7B-sized weights (11008 x 4096), every element compared."""
    import synth
    _, _, orc = env
    W, _ = synth.make_workload("llama7b_gemv")
    q, s, z = orc.quantize_pack(W)
    got = run_dequant(env, q, s, z, out)
    assert np.array_equal(got, orc.dequantize16(q, s, z, W.shape[1], out))


def test_dequantize_output_guard(env):
    """out placed inside a larger buffer: the elements around it keep their sentinel."""
    import synth
    torch, w4, orc = env
    N, K = 37, 640
    W, _ = synth.make_random(N, K, 1, seed=5)
    q, s, z = orc.quantize_pack(W)
    sentinel = 0x7F7B
    pad = 8                                    # 16 bytes: out stays 16-byte aligned
    buf = torch.full((pad + N * K + 40,), sentinel, dtype=torch.int16, device="cuda")
    out = buf[pad:pad + N * K].view(torch.bfloat16).view(N, K)
    w4.dequantize(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(z).cuda(), out=out)
    torch.cuda.synchronize()
    flat = buf.cpu().numpy().view(np.uint16)
    assert np.all(flat[:pad] == sentinel) and np.all(flat[pad + N * K:] == sentinel)
    assert np.array_equal(flat[pad:pad + N * K].reshape(N, K), orc.dequantize16(q, s, z, K, "bf16"))


# ---- the matmul on symmetric weights -------------------------------------------------
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (8, 1000, 2048), (64, 512, 1024), (1, 300, 384)])
def test_matmul_on_symmetric_weights(env, M, N, K):
    """w4_matmul consumes the symmetric quantizer's output (zero points 8) unchanged."""
    import synth
    torch, w4, orc = env
    W, A = synth.make_random(N, K, M, seed=M + N)
    q, s, z = w4.quantize_pack(to_dev_w(torch, W), symmetric=True)
    Ad = torch.from_numpy(np.ascontiguousarray(A).view(np.int16)).cuda().view(torch.bfloat16)
    Y = w4.matmul(Ad, q, s, z)
    torch.cuda.synchronize()
    Yb = Y.view(torch.int16).cpu().numpy().view(np.uint16)
    qo, so, zo = orc.quantize_pack(W, symmetric=True)
    Yref, S = orc.matmul(A, qo, so, zo)
    ok, worst, idx = orc.check_y(Yb, Yref, S)
    assert ok, f"worst ratio {worst:.3g} at {idx}"
