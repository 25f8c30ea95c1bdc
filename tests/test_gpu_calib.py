"""GPU parity of the clip-range calibrated quantizers ("Building a From-Scratch
Group-Wise INT4 Quantization Layer for LLaMA Weights", Step 4): the percentile and the
MSE-search calibrators against the CPU oracle, bit-exact in qweight, scales and zeros,
through the C ABI (via the ctypes binding).  The calibrated weights then feed
w4_matmul, whose output must meet the usual tolerance."""
import numpy as np
import pytest

from test_oracle_pins import CALIB_CASES, calib_group

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    from w4a16_matmul_asym_b300 import build
    build.build()
    import w4a16_matmul_asym_b300 as w4
    w4.load_library()
    return torch, w4, oracle_mod


def gpu_calib(env, W, method, param):
    torch, w4, _ = env
    Wd = torch.from_numpy(np.ascontiguousarray(W)).cuda()
    q, s, z = w4.quantize_pack(Wd, calibration=method, param=param)
    torch.cuda.synchronize()
    assert w4.w4_check_device_error(0) == w4.W4_OK
    return q.cpu().numpy(), s.cpu().numpy(), z.cpu().numpy()


def assert_calib_equal(env, W, method, param):
    _, _, orc = env
    q, s, z = gpu_calib(env, W, method, param)
    qo, so, zo = orc.quantize_pack_calibrated(W, method, param)
    bad_s = np.argwhere(s.view(np.uint16) != so.view(np.uint16))
    assert len(bad_s) == 0, f"scales differ at {len(bad_s)} groups, first {bad_s[:5].tolist()}"
    assert np.array_equal(z, zo), "zeros differ"
    if not np.array_equal(q, qo):
        bad = np.argwhere(q != qo)
        raise AssertionError(f"qweight differs at {len(bad)} bytes, first {bad[:5].tolist()}")


@pytest.mark.parametrize("p", [99.9, 50.0, 100.0, 0.5, 12.5, 95.0, 3.0, 99.5, 0.1])
@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_percentile_random(env, p, dtype):
    """Order statistics near the top (99.9, 100, 99.5: the two largest; 95: within 8 of the
    top), near the bottom (0.1, 0.5: the two smallest; 3: within 8) and in the middle
    (50, 12.5: the sorted path)."""
    import synth
    W, _ = synth.make_random(96, 1024, 1, seed=int(p * 10) + 3, w_dtype="f16")
    assert_calib_equal(env, W.astype(dtype), "percentile", p)


@pytest.mark.parametrize("n", [1000, 1, 2, 7, 100])
@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_mse_random(env, n, dtype):
    import synth
    W, _ = synth.make_random(24, 512, 1, seed=n + 17, w_dtype="f16")
    assert_calib_equal(env, W.astype(dtype), "mse", n)


def test_calibration_hand_worked_groups(env):
    """The golden groups of the oracle pins (ties between candidates, exact grids,
    constant and all-zero groups, the order-statistic ramps), each method with the
    parameters the fixture gives."""
    for case in CALIB_CASES:
        w = calib_group(case["values"])[None, :]
        assert_calib_equal(env, w, case["method"], float(case["param"]) if case["method"] == "percentile"
                           else int(case["param"]))


def test_calibration_edge_groups(env):
    """Zero groups, -0, constant magnitudes, fp16 subnormals, +-65504, groups with one
    outlier, and exact ties of w / s, for both methods."""
    rng = np.random.default_rng(29)
    rows = [np.zeros(128), np.full(128, -0.0), np.full(128, 0.3), np.full(128, -2.5),
            (rng.integers(-1023, 1024, 128) * 2.0 ** -24),
            np.where(rng.random(128) < 0.5, 65504.0, -65504.0),
            np.concatenate([[1.0], rng.standard_normal(127) * 0.01]),
            (np.arange(128) - 64) / 8.0,
            rng.integers(-7, 8, 128) / 4.0]
    W = np.stack(rows).astype(np.float16)
    for method, param in (("percentile", 99.9), ("percentile", 50.0), ("mse", 1000), ("mse", 3)):
        assert_calib_equal(env, W, method, param)
        assert_calib_equal(env, W.astype(np.float32), method, param)


def test_calibration_ragged_and_many_groups(env):
    """Odd row counts and more groups than warps in flight (grid-stride loop)."""
    import synth
    W, _ = synth.make_random(1031, 384, 1, seed=5)
    assert_calib_equal(env, W, "percentile", 99.0)
    W2, _ = synth.make_random(37, 896, 1, seed=6)
    assert_calib_equal(env, W2, "mse", 257)


def test_calibrated_weights_feed_the_matmul(env):
    """Both calibrated layouts are consumed by w4_matmul (zero points 8): Y within the
    usual tolerance of the fp64 dequantize-matmul, for the decode and GEMM paths."""
    import synth
    torch, w4, orc = env
    W, A = synth.make_random(256, 2048, 32, seed=8)
    for method, param in (("percentile", 99.9), ("mse", 200)):
        q, s, z = gpu_calib(env, W, method, param)
        for M in (1, 8, 32):
            Ad = torch.from_numpy(np.ascontiguousarray(A[:M]).view(np.int16)).cuda().view(torch.bfloat16)
            Y = w4.matmul(Ad, torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(z).cuda())
            torch.cuda.synchronize()
            Yref, S = orc.matmul(A[:M], q, s, z)
            ok, worst, idx = orc.check_y(Y.view(torch.int16).cpu().numpy().view(np.uint16), Yref, S)
            assert ok, (method, M, worst, idx)


def test_percentile_full_workload_sampled_rows(env):
    """The 70B-layer workload at full size in the launch configuration the benchmark
    times; 64 sampled rows compared bit-exactly with the oracle run on those rows."""
    import synth
    _, _, orc = env
    W, _ = synth.make_workload("mlp70b")
    q, s, z = gpu_calib(env, W, "percentile", 99.9)
    rows = np.random.default_rng(3).choice(W.shape[0], 64, replace=False)
    qo, so, zo = orc.quantize_pack_calibrated(W[rows], "percentile", 99.9)
    assert np.array_equal(q[rows], qo) and np.array_equal(z[rows], zo)
    assert np.array_equal(s[rows].view(np.uint16), so.view(np.uint16))


def test_mse_full_workload_sampled_rows(env):
    """The Llama-7B-shaped weights at full size through the MSE search (1000
    candidates); 8 sampled rows compared bit-exactly with the oracle on those rows."""
    import synth
    _, _, orc = env
    W, _ = synth.make_workload("llama7b_gemv")
    q, s, z = gpu_calib(env, W, "mse", 1000)
    rows = np.random.default_rng(4).choice(W.shape[0], 8, replace=False)
    qo, so, zo = orc.quantize_pack_calibrated(W[rows], "mse", 1000)
    assert np.array_equal(q[rows], qo) and np.array_equal(z[rows], zo)
    assert np.array_equal(s[rows].view(np.uint16), so.view(np.uint16))
