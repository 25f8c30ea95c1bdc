"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

qweight, scales and zeros must be bit-exact; Y must satisfy, per element,
|Y - Y_ref| <= 8e-3 * sum_k |a_k * w_hat_k| + ulp_bf16(|Y_ref|) / 2.
All calls go through the C ABI (via the thin ctypes binding)."""
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


def to_dev_bf16(torch, A_bits):
    return torch.from_numpy(np.ascontiguousarray(A_bits).view(np.int16)).cuda().view(torch.bfloat16)


def y_bits(torch, Y):
    return Y.view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_quantize(env, W):
    torch, w4, _ = env
    q, s, z = w4.quantize_pack(to_dev_w(torch, W))
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy(), z.cpu().numpy()


def assert_quant_equal(env, W):
    _, _, orc = env
    q, s, z = gpu_quantize(env, W)
    qo, so, zo = orc.quantize_pack(W)
    assert np.array_equal(s.view(np.uint16), so.view(np.uint16)), "scales differ"
    assert np.array_equal(z, zo), "zeros differ"
    if not np.array_equal(q, qo):
        bad = np.argwhere(q != qo)
        raise AssertionError(f"qweight differs at {len(bad)} bytes, first {bad[:5].tolist()}")


def run_matmul(env, A_bits, q, s, z):
    torch, w4, _ = env
    Y = w4.matmul(to_dev_bf16(torch, A_bits), torch.from_numpy(q).cuda(),
                  torch.from_numpy(s).cuda(), torch.from_numpy(z).cuda())
    torch.cuda.synchronize()
    return y_bits(torch, Y)


def assert_matmul_ok(env, A_bits, q, s, z):
    _, _, orc = env
    Yb = run_matmul(env, A_bits, q, s, z)
    Yref, S = orc.matmul(A_bits, q, s, z)
    ok, worst, idx = orc.check_y(Yb, Yref, S)
    assert ok, f"Y out of tolerance: worst ratio {worst:.3g} at {idx}"
    return worst


# ---- quantize / pack -----------------------------------------------------------------
def test_quantize_tiny_f32(env):
    import synth
    W, _ = synth.make_workload("tiny")
    assert_quant_equal(env, W)


@pytest.mark.parametrize("name", ["llama7b_gemv", "skinny_m8", "prefill_gemm", "mlp70b"])
def test_quantize_full_workloads(env, name):
    import synth
    W, _ = synth.make_workload(name, M=1)
    assert_quant_equal(env, W)


@pytest.mark.parametrize("N,K,dtype", [(1, 128, "f16"), (3, 128, "f32"), (5, 384, "f16"),
                                       (17, 256, "f32"), (7, 1152, "f16"), (9, 640, "f16")])
def test_quantize_ragged(env, N, K, dtype):
    import synth
    W, _ = synth.make_random(N, K, 1, seed=N * 1000 + K, sigma=0.5,
                             w_dtype=dtype, outliers=True)
    assert_quant_equal(env, W)


def test_quantize_hand_groups(env):
    """Every hand-worked group of tests/golden/hand_groups.txt, one per row."""
    cases = parse_cases(os.path.join(GOLDEN_DIR, "hand_groups.txt"))
    rows = []
    for c in cases:
        vals = [np.array([int(b, 16)], np.uint32).view(np.float32)[0] for b in c["values"].split()]
        g = np.full(128, np.array([int(c["pad"], 16)], np.uint32).view(np.float32)[0], np.float32)
        g[: len(vals)] = vals
        rows.append(g)
    W = np.stack(rows)
    assert_quant_equal(env, W)
    W16 = np.stack([r for r, c in zip(rows, cases) if c["f16_exact"] == "1"]).astype(np.float16)
    assert_quant_equal(env, W16)


def test_quantize_edge_values(env):
    """Constant groups, ties at every level, all-positive / all-negative groups, fp16
    subnormals, zeros, the fp16 extremes, groups that clip."""
    rng = np.random.default_rng(99)
    rows = []
    for c in (0.0, -0.0, 0.3, -2.6, 0.5, 7.0, 60000.0, -60000.0):
        rows.append(np.full(128, c, np.float32))
    # exact ties: multiples of s/2 in a group spanning [-7.5, 7.5] (s = 1)
    t = np.arange(-15, 16, dtype=np.float32) / 2
    g = np.zeros(128, np.float32); g[:31] = t; rows.append(g)
    # s = 0.1f ties (H2-like), shifted copies
    for off in range(4):
        g = np.zeros(128, np.float32); g[0] = -0.75; g[1] = 0.75
        g[2:40] = np.round(rng.uniform(-7.5, 7.5, 38) * 2) / 2 * np.float32(0.1)
        rows.append(g + np.float32(off * 0.0))
    rows.append(np.abs(rng.standard_normal(128).astype(np.float32)) + 3)      # all positive
    rows.append(-np.abs(rng.standard_normal(128).astype(np.float32)) - 3)     # all negative
    sub = (rng.integers(-1023, 1024, 128).astype(np.float32) * 2.0 ** -24)     # fp16 subnormals
    rows.append(sub.astype(np.float32))
    rows.append(np.array([65504, -65504] + [0] * 126, np.float32))
    rows.append(np.array([1000.0, 1000.125] + [1000.0625] * 126, np.float32))  # narrow, far from 0
    W = np.stack(rows)
    assert_quant_equal(env, W.astype(np.float16))
    assert_quant_equal(env, W.astype(np.float16).astype(np.float32))


def test_quantize_random_fp32_many_ties(env):
    """fp32 weights on a coarse grid, so that w/s lands on half-integers often."""
    rng = np.random.default_rng(5)
    W = (rng.integers(-60, 61, size=(64, 1024)).astype(np.float32) / 8)
    assert_quant_equal(env, W)


def tiny_scale_rows(rng):
    """fp32 groups whose scale lies below 2^-128 (no finite reciprocal): subnormal and
    tiny normal values, exact zeros among them; every range stays >= 1000 * 2^-149 so
    the scale itself is nonzero."""
    t = np.float32(2.0 ** -149)
    rows = [
        (rng.uniform(-1e-38, 1e-38, 128)).astype(np.float32),                  # subnormal s
        (rng.uniform(0, 3e-39, 128)).astype(np.float32),                       # all positive
        (rng.integers(-1000, 1001, 128).astype(np.float32) * t),               # s = 133 * 2^-149
        np.where(rng.random(128) < 0.5, 0.0, rng.uniform(-4e-38, 4e-38, 128)).astype(np.float32),
        (rng.uniform(-1e-37, 1e-37, 128)).astype(np.float32),                  # tiny normals
        (rng.integers(-7, 8, 128).astype(np.float32) * np.float32(2.0 ** -130)),  # ties on a grid
    ]
    return np.stack(rows)


def test_quantize_fp32_tiny_scales(env):
    """Groups whose fp32 scale has no finite reciprocal still quantize bit-exactly."""
    assert_quant_equal(env, tiny_scale_rows(np.random.default_rng(17)))


# ---- matmul: GEMV / skinny path (M <= 8) ----------------------------------------------
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_matmul_small_m(env, M):
    import synth
    _, _, orc = env
    W, A = synth.make_random(203, 1152, M, seed=40 + M)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


@pytest.mark.parametrize("N,K,M", [(1, 128, 1), (2, 256, 1), (31, 128, 3), (65, 384, 8),
                                   (130, 4096, 2), (1000, 256, 1)])
def test_matmul_small_m_ragged(env, N, K, M):
    import synth
    _, _, orc = env
    W, A = synth.make_random(N, K, M, seed=N + K + M)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 2048), (37, 4096), (300, 8192), (1031, 2048), (9, 6144)])
def test_matmul_streaming_gemv(env, M, N, K):
    """Shapes that take the streaming GEMV (K a multiple of 2048): activations in
    registers for M * ceil(K/4096) <= 2, in shared memory otherwise; N tails."""
    import synth
    _, _, orc = env
    W, A = synth.make_random(N, K, M, seed=7 * N + K + M)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 12, 16])
@pytest.mark.parametrize("N,K", [(1, 2048), (15, 2048), (17, 4096), (300, 8192), (1031, 2048),
                                 (9, 6144), (2500, 4096)])
def test_matmul_decode_mma(env, M, N, K):
    """The warp-MMA decode kernel (1 <= M <= 16, K a multiple of 2048): one or two
    8-column activation blocks, N tails inside a 16-row tile, CTAs with one or many
    tiles, one to four 2048-wide stages per tile."""
    import synth
    _, _, orc = env
    W, A = synth.make_random(N, K, M, seed=31 * N + K + M)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_matmul_streaming_zero_rows(env, M):
    """Rows of W that are all zero reconstruct to 0 exactly, so those outputs must be
    exactly 0 on the streaming path too; other rows stay within tolerance."""
    import synth
    _, _, orc = env
    W, A = synth.make_random(40, 4096, M, seed=11 + M)
    W[3] = 0
    W[17:25] = 0
    q, s, z = orc.quantize_pack(W)
    Yb = run_matmul(env, A, q, s, z)
    assert np.all(Yb[:, 3] == 0) and np.all(Yb[:, 17:25] == 0)
    Yref, S = orc.matmul(A, q, s, z)
    ok, worst, idx = orc.check_y(Yb, Yref, S)
    assert ok, (worst, idx)


def _bf16_bits(x):
    import synth
    return synth.f32_to_bf16_bits(np.ascontiguousarray(x, np.float32))


@pytest.mark.parametrize("K", [2048, 4096, 8192])
def test_gemv_wide_range_activations(env, K):
    """Activations whose groups each hold one huge element (2^20) next to values 2^-10
    N(0, 1): every other element lies more than 12 binades below its group maximum,
    so the decode GEMV cannot give it an exact integer digit and must carry it as a
    residual (more than four per lane: the slow path).  The weight under each huge
    element is 0, so it reconstructs to exactly 0 and the huge element contributes
    nothing: the tolerance (relative to sum |a * w_hat|) is set by the small ones."""
    import synth
    _, _, orc = env
    rng = np.random.default_rng(K + 5)
    N = 77
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    a = (rng.standard_normal(K) * 2.0 ** -10).astype(np.float32)
    big = np.arange(0, K, 128) + rng.integers(0, 128, K // 128)
    a[big] = 2.0 ** 20
    W[:, big] = 0
    q, s, z = orc.quantize_pack(W)
    A = _bf16_bits(a[None, :])
    assert_matmul_ok(env, A, q, s, z)


@pytest.mark.parametrize("K", [2048, 4096, 8192])
def test_gemv_few_small_activations(env, K):
    """One to three elements per group far below the group maximum (the register
    residual list of the decode GEMV), mixed with exact zeros and subnormals."""
    import synth
    _, _, orc = env
    rng = np.random.default_rng(K + 9)
    N = 300
    W, _ = synth.make_random(N, K, 1, seed=K + 9)
    a = rng.standard_normal(K).astype(np.float32)
    for g in range(K // 128):
        idx = g * 128 + rng.choice(128, size=rng.integers(1, 4), replace=False)
        a[idx] *= 2.0 ** -20
    a[rng.integers(0, K, 8)] = 0.0
    a[rng.integers(0, K, 4)] = 3e-39  # subnormal in bf16
    q, s, z = orc.quantize_pack(W)
    A = _bf16_bits(a[None, :])
    assert_matmul_ok(env, A, q, s, z)


@pytest.mark.parametrize("special", ["inf", "nan"])
def test_gemv_nonfinite_activation(env, special):
    """An infinite or NaN activation propagates as IEEE arithmetic would: a row whose
    reconstructed weight there is 0 gives NaN (inf * 0), others give +-inf (or NaN)."""
    import synth
    torch, _, orc = env
    K, N = 4096, 64
    W, _ = synth.make_random(N, K, 1, seed=21)
    rng = np.random.default_rng(21)
    a = rng.standard_normal(K).astype(np.float32)
    a[1000] = np.inf if special == "inf" else np.nan
    W[:10, 1000] = 0  # these rows reconstruct 0 there
    q, s, z = orc.quantize_pack(W)
    A = _bf16_bits(a[None, :])
    Yb = run_matmul(env, A, q, s, z)[0]
    y = orc.bf16_bits_to_f64(Yb)
    w_hat = orc.dequantize(q, s, z, K)
    with np.errstate(invalid="ignore", over="ignore"):
        ref = w_hat @ orc.bf16_bits_to_f64(A[0])
    assert np.array_equal(np.isnan(y), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(y[fin], ref[fin])  # both +-inf


@pytest.mark.parametrize("name", ["tiny", "llama7b_gemv", "skinny_m8", "mlp70b"])
def test_matmul_full_workloads_small_m(env, name):
    import synth
    _, _, orc = env
    W, A = synth.make_workload(name)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


def test_matmul_zero_weights_give_exact_zero(env):
    """All-zero W: every reconstructed weight is 0, so Y must be exactly 0."""
    import synth
    _, _, orc = env
    _, A = synth.make_random(8, 512, 8, seed=3)
    W = np.zeros((64, 512), np.float16)
    q, s, z = orc.quantize_pack(W)
    for M in (1, 8):
        Yb = run_matmul(env, A[:M], q, s, z)
        assert np.all(Yb == 0)


def test_matmul_k_zero_fills_zeros(env):
    torch, w4, _ = env
    A = torch.empty((3, 0), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((5, 0), dtype=torch.uint8, device="cuda")
    s = torch.empty((5, 0), dtype=torch.float16, device="cuda")
    z = torch.empty((5, 0), dtype=torch.uint8, device="cuda")
    Y = torch.full((3, 5), 7.0, dtype=torch.bfloat16, device="cuda")
    w4.matmul(A, q, s, z, out=Y)
    torch.cuda.synchronize()
    assert torch.all(Y == 0)


def test_binding_rejects_mismatched_tables(env):
    """The C ABI takes bare pointers, so the binding checks the packed tables' shapes,
    dtypes and contiguity before any launch; nothing reaches the GPU."""
    torch, w4, _ = env
    q = torch.zeros((4, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones((4, 2), dtype=torch.float16, device="cuda")
    z = torch.zeros((4, 2), dtype=torch.uint8, device="cuda")
    A = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        w4.matmul(A, q, s[:, :1].contiguous(), z)
    with pytest.raises(ValueError):
        w4.dequantize(q, s, z[:3].contiguous())
    with pytest.raises(ValueError):
        w4.quantize_pack(torch.zeros((4, 256), dtype=torch.float16, device="cuda"), out=(q, s, z.t()))
    assert w4.w4_check_device_error(0) == 0


def test_empty_problems_are_noops(env):
    torch, w4, _ = env
    W = torch.empty((0, 256), dtype=torch.float16, device="cuda")
    q, s, z = w4.quantize_pack(W)
    assert q.shape == (0, 128) and s.shape == (0, 2)
    A = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    qw = torch.zeros((4, 128), dtype=torch.uint8, device="cuda")
    Y = w4.matmul(A, qw, torch.ones((4, 2), dtype=torch.float16, device="cuda"),
                  torch.zeros((4, 2), dtype=torch.uint8, device="cuda"))
    assert Y.shape == (0, 4)
    assert w4.w4_check_device_error(0) == 0


# ---- matmul: tcgen05 tensor-core path (M >= 9) ------------------------------------------
@pytest.mark.parametrize("M,N,K", [(9, 256, 128), (15, 100, 256), (16, 256, 512), (128, 512, 1024),
                                   (129, 257, 384), (300, 1000, 1024), (64, 1, 128),
                                   (200, 777, 640), (17, 4104, 256)])
def test_matmul_gemm_shapes(env, M, N, K):
    import synth
    _, _, orc = env
    W, A = synth.make_random(N, K, M, seed=M * 7 + N + K)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


@pytest.mark.parametrize("M,N,K", [(9, 37, 2048), (12, 300, 4096), (16, 4096, 4096), (13, 1031, 2048),
                                   (10, 200, 8192), (16, 9, 6144)])
def test_matmul_9_to_16_rows(env, M, N, K):
    """9 <= M <= 16 with few 128-row tiles and K a multiple of 2048: the warp-MMA decode
    kernel (two 8-column activation blocks, odd M leaving the last column empty) where
    its activations fit in shared memory, the tcgen05 GEMM otherwise."""
    import synth
    _, _, orc = env
    W, A = synth.make_random(N, K, M, seed=900 + M + N)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


@pytest.mark.parametrize("M", [9, 10, 12, 15, 16, 20])
def test_matmul_gemm_small_m_tail(env, M):
    import synth
    _, _, orc = env
    W, A = synth.make_random(96, 768, M, seed=500 + M)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


def test_matmul_gemm_zero_weights(env):
    import synth
    _, _, orc = env
    _, A = synth.make_random(8, 512, 40, seed=4)
    q, s, z = orc.quantize_pack(np.zeros((300, 512), np.float16))
    assert np.all(run_matmul(env, A, q, s, z) == 0)


@pytest.mark.parametrize("M,N,K,offset", [(200, 264, 256, 0), (300, 1000, 512, 0), (17, 4104, 256, 0),
                                          (40, 136, 384, 1), (129, 257, 384, 0)])
def test_matmul_gemm_output_guard(env, M, N, K, offset):
    """Y placed inside a larger buffer keeps the elements around it untouched.  With
    offset 0 and N % 8 == 0, Y is 16-byte aligned and the tensor-store epilogue writes
    it (boxes clipped at N and M); offset 1 makes Y 2-byte aligned, as N % 8 != 0 does,
    which selects direct stores."""
    import synth
    torch, w4, orc = env
    W, A = synth.make_random(N, K, M, seed=M + 3 * N + K + offset)
    q, s, z = orc.quantize_pack(W)
    sentinel = 0x7F7B  # a bf16 NaN pattern the kernel never produces
    pad = N + offset
    buf = torch.full((pad + M * N + N,), sentinel, dtype=torch.int16, device="cuda")
    Y = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
    w4.matmul(to_dev_bf16(torch, A), torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(),
              torch.from_numpy(z).cuda(), out=Y)
    torch.cuda.synchronize()
    flat = buf.cpu().numpy().view(np.uint16)
    assert np.all(flat[:pad] == sentinel) and np.all(flat[pad + M * N:] == sentinel)
    Yref, S = orc.matmul(A, q, s, z)
    ok, worst, idx = orc.check_y(flat[pad:pad + M * N].reshape(M, N), Yref, S)
    assert ok, f"worst ratio {worst:.3g} at {idx}"


@pytest.mark.parametrize("M,N,K", [(1, 4000, 8192), (4, 300, 4096), (12, 1031, 2048), (64, 300, 1024)])
def test_matmul_unaligned_tables(env, M, N, K):
    """Scales and zero points that start one element past a 16-byte boundary (2- and
    1-byte aligned, which the C ABI accepts).  The streaming kernels copy the tables
    with tensor copies that need 16-byte alignment, so they step aside (the plain GEMV
    for M <= 8, the GEMM, which loads its tables directly, above), and the result still
    matches the oracle."""
    import synth
    torch, w4, orc = env
    W, A = synth.make_random(N, K, M, seed=7 * M + N + K)
    q, s, z = orc.quantize_pack(W)
    sbuf = torch.zeros(s.size + 8, dtype=torch.float16, device="cuda")
    zbuf = torch.zeros(z.size + 16, dtype=torch.uint8, device="cuda")
    s_d = sbuf[1:1 + s.size].view(s.shape)
    z_d = zbuf[1:1 + z.size].view(z.shape)
    s_d.copy_(torch.from_numpy(s))
    z_d.copy_(torch.from_numpy(z))
    assert s_d.data_ptr() % 16 == 2 and z_d.data_ptr() % 16 == 1
    Y = w4.matmul(to_dev_bf16(torch, A), torch.from_numpy(q).cuda(), s_d, z_d)
    torch.cuda.synchronize()
    Yref, S = orc.matmul(A, q, s, z)
    ok, worst, idx = orc.check_y(y_bits(torch, Y), Yref, S)
    assert ok, f"worst ratio {worst:.3g} at {idx}"


@pytest.mark.parametrize("M,N,K", [(512, 38400, 128), (300, 20000, 256)])
def test_matmul_gemm_many_tiles_full(env, M, N, K):
    """More than twice as many tiles as SMs at small K, every output compared: the
    persistent tile loop (accumulator hand-off and barrier phases across many tiles
    per CTA) checked element by element, not on a sample."""
    import synth
    _, _, orc = env
    W, A = synth.make_random(N, K, M, seed=M + N + K)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


@pytest.mark.parametrize("M,N,K", [(256, 19200, 384), (300, 19072, 1024), (768, 6400, 256)])
def test_matmul_gemm_partial_last_wave_full(env, M, N, K):
    """Tile counts (150, 298, 150 on 148 SMs) that leave a last wave of two tiles, so a
    few CTAs run one tile more than the rest (the persistent loop's end with uneven
    work), at K = 384, 1024 and 256.  Every output compared."""
    import synth
    _, _, orc = env
    W, A = synth.make_random(N, K, M, seed=M + 7 * N + K)
    q, s, z = orc.quantize_pack(W)
    assert_matmul_ok(env, A, q, s, z)


def test_matmul_prefill_workload_sampled(env):
    """Full-size prefill workload (M=2048, N=14336, K=4096) in the launch configuration
    the benchmark times; checked on 6000 sampled outputs plus one full output row and
    one full output column, each computed one by one by the oracle."""
    import synth
    torch, w4, orc = env
    W, A = synth.make_workload("prefill_gemm")
    q, s, z = orc.quantize_pack(W)
    Yb = run_matmul(env, A, q, s, z)
    M, N = A.shape[0], q.shape[0]
    rng = np.random.default_rng(123)
    mi = np.concatenate([rng.integers(0, M, 6000), np.full(N, 1537), np.arange(M)])
    ni = np.concatenate([rng.integers(0, N, 6000), np.arange(N), np.full(M, 9001)])
    Yref, S = orc.matmul_entries(A, q, s, z, mi, ni)
    ok, worst, idx = orc.check_y(Yb[mi, ni], Yref, S)
    assert ok, f"worst ratio {worst:.3g} at sample {idx}"
