"""GPU parity of W4A8 ("Hands-On Build Guide: Group-Wise INT4 Weight-Only Quantization
with Per-Channel Scale", Step 3 and Step 5): the per-token INT8 activation quantizer
bit-exact against the CPU oracle, and the W4A8 product within the library's tolerance
of the oracle's fp64 product, on the decode path (no workspace) and on the GEMM path
(int8 widened into a caller-owned workspace), through the C ABI."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    from w4a16_matmul_asym_b300 import build
    build.build()
    import w4a16_matmul_asym_b300 as w4
    w4.load_library()
    return torch, w4, oracle_mod


def to_dev_bf16(torch, A_bits):
    return torch.from_numpy(np.ascontiguousarray(A_bits).view(np.int16)).cuda().view(torch.bfloat16)


def gpu_act_int8(env, A_bits):
    torch, w4, _ = env
    aq, sa = w4.quantize_act_int8(to_dev_bf16(torch, A_bits))
    torch.cuda.synchronize()
    assert w4.w4_check_device_error(0) == w4.W4_OK
    return aq.cpu().numpy(), sa.cpu().numpy()


def assert_act_equal(env, A_bits):
    _, _, orc = env
    aq, sa = gpu_act_int8(env, A_bits)
    aqo, sao = orc.quantize_act_int8(A_bits)
    assert np.array_equal(sa.view(np.uint32), sao.view(np.uint32)), "scales differ"
    if not np.array_equal(aq, aqo):
        bad = np.argwhere(aq != aqo)
        raise AssertionError(f"levels differ at {len(bad)} positions, first {bad[:5].tolist()}")


@pytest.mark.parametrize("M,K", [(1, 4096), (3, 128), (8, 8192), (64, 1152), (2048, 4096), (5, 8), (7, 24)])
def test_act_int8_random(env, M, K):
    import synth
    rng = np.random.default_rng(M * 31 + K)
    A = (rng.standard_normal((M, K)) * 10.0 ** rng.uniform(-4, 3, (M, 1))).astype(np.float32)
    assert_act_equal(env, synth.f32_to_bf16_bits(A))


def test_act_int8_edge_rows(env):
    """Hand rows with exact ties (s_a = 1 and 2), an all-zero row, -0, subnormal bf16
    values, a lone large element, and the bf16 extremes."""
    import synth
    rows = np.zeros((8, 256), np.float32)
    rows[0, :7] = [127, 2.5, -3.5, 0.5, -0.5, 1.5, -127]
    rows[1, :5] = [254, 1, 3, 5, -254]
    rows[3, :] = -0.0
    rows[4, :] = np.arange(256) * 1e-39
    rows[5, 17] = 3e38
    rows[5, :16] = 1.0
    rows[6, :] = np.where(np.arange(256) % 2 == 0, 3.3895e38, -3.3895e38)
    rows[7, :] = (np.arange(256) - 128) / 64.0
    assert_act_equal(env, synth.f32_to_bf16_bits(rows))


def run_w4a8(env, A_bits, W, M):
    torch, w4, orc = env
    q, s, z = orc.quantize_pack(W)
    aq, sa = orc.quantize_act_int8(A_bits[:M])
    Y = w4.matmul_w4a8(torch.from_numpy(aq).cuda(), torch.from_numpy(sa).cuda(), torch.from_numpy(q).cuda(),
                       torch.from_numpy(s).cuda(), torch.from_numpy(z).cuda())
    torch.cuda.synchronize()
    assert w4.w4_check_device_error(0) == w4.W4_OK
    Yb = Y.view(torch.int16).cpu().numpy().view(np.uint16)
    return Yb, (aq, sa, q, s, z)


@pytest.mark.parametrize("M,N,K", [(1, 300, 2048), (1, 1031, 4096), (1, 77, 8192), (1, 5000, 16384),
                                   (2, 37, 4096), (8, 1031, 8192), (16, 200, 4096), (3, 1031, 2048), (8, 300, 4096),
                                   (5, 17, 6144), (12, 2500, 2048)])
def test_w4a8_decode_path(env, M, N, K):
    """Shapes the decode kernels take, with no workspace: M = 1 on integer dot products
    over the int8 digits (half-group, one-group and two-warp-per-row layouts), larger M
    on the warp-MMA kernel with the int8 activations widened while staged."""
    import synth
    torch, w4, orc = env
    assert w4.w4_matmul_w4a8_workspace_size(M, K) == 0
    W, A = synth.make_random(N, K, M, seed=N + K + M)
    Yb, (aq, sa, q, s, z) = run_w4a8(env, A, W, M)
    Yref, S = orc.w4a8_matmul(aq, sa, q, s, z)
    ok, worst, idx = orc.check_y(Yb, Yref, S)
    assert ok, (worst, idx)


@pytest.mark.parametrize("M,N,K", [(3, 100, 1152), (17, 257, 2048), (64, 1000, 1024), (300, 777, 640),
                                   (16, 64, 16384), (256, 19200, 384)])
def test_w4a8_gemm_path(env, M, N, K):
    """Shapes the decode kernel does not take: a_q widened into the workspace, then the
    tcgen05 GEMM with the per-row scale in its epilogue (256 x 19200: more tiles than
    SMs, with a partial last wave)."""
    import synth
    torch, w4, orc = env
    assert w4.w4_matmul_w4a8_workspace_size(M, K) >= M * K * 2
    W, A = synth.make_random(N, K, M, seed=3 * N + K + M)
    Yb, (aq, sa, q, s, z) = run_w4a8(env, A, W, M)
    Yref, S = orc.w4a8_matmul(aq, sa, q, s, z)
    ok, worst, idx = orc.check_y(Yb, Yref, S)
    assert ok, (worst, idx)


def test_w4a8_prefill_workload_sampled(env):
    """The prefill workload at full size (M = 2048, N = 14336, K = 4096) through the
    GPU activation quantizer and the W4A8 GEMM, on 4000 sampled outputs."""
    import synth
    torch, w4, orc = env
    W, A = synth.make_workload("prefill_gemm")
    q, s, z = orc.quantize_pack(W)
    aqd, sad = w4.quantize_act_int8(to_dev_bf16(torch, A))
    Y = w4.matmul_w4a8(aqd, sad, torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(z).cuda())
    torch.cuda.synchronize()
    aq, sa = aqd.cpu().numpy(), sad.cpu().numpy()
    aqo, sao = orc.quantize_act_int8(A)
    assert np.array_equal(aq, aqo) and np.array_equal(sa.view(np.uint32), sao.view(np.uint32))
    Yb = Y.view(torch.int16).cpu().numpy().view(np.uint16)
    rng = np.random.default_rng(7)
    mi, ni = rng.integers(0, A.shape[0], 4000), rng.integers(0, W.shape[0], 4000)
    Yref, S = orc.w4a8_matmul_entries(aq, sa, q, s, z, mi, ni)
    ok, worst, idx = orc.check_y(Yb[mi, ni], Yref, S)
    assert ok, (worst, idx)


@pytest.mark.parametrize("name", ["llama7b_gemv", "mlp70b"])
def test_w4a8_decode_full_workloads(env, name):
    """The M = 1 decode workloads at full size through the GPU activation quantizer and
    the W4A8 decode kernel, every output compared."""
    import synth
    torch, w4, orc = env
    W, A = synth.make_workload(name)
    q, s, z = orc.quantize_pack(W)
    aqd, sad = w4.quantize_act_int8(to_dev_bf16(torch, A))
    Y = w4.matmul_w4a8(aqd, sad, torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(z).cuda())
    torch.cuda.synchronize()
    aq, sa = aqd.cpu().numpy(), sad.cpu().numpy()
    Yref, S = orc.w4a8_matmul(aq, sa, q, s, z)
    ok, worst, idx = orc.check_y(Y.view(torch.int16).cpu().numpy().view(np.uint16), Yref, S)
    assert ok, (worst, idx)


def test_w4a8_small_workspace_is_rejected(env):
    torch, w4, _ = env
    M, N, K = 64, 128, 1024
    need = w4.w4_matmul_w4a8_workspace_size(M, K)
    assert need >= M * K * 2
    aq = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sa = torch.ones((M,), dtype=torch.float32, device="cuda")
    q = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    s = torch.ones((N, K // 128), dtype=torch.float16, device="cuda")
    z = torch.zeros((N, K // 128), dtype=torch.uint8, device="cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty((need - 256,), dtype=torch.uint8, device="cuda")
    rc = w4.w4_matmul_w4a8(aq.data_ptr(), sa.data_ptr(), M, N, K, 128, q.data_ptr(), s.data_ptr(), z.data_ptr(),
                           Y.data_ptr(), ws.data_ptr(), ws.numel(), 0)
    assert rc == w4.W4_ERR_INVALID_ARG
    rc = w4.w4_matmul_w4a8(aq.data_ptr(), sa.data_ptr(), M, N, K, 128, q.data_ptr(), s.data_ptr(), z.data_ptr(),
                           Y.data_ptr(), 0, 0, 0)
    assert rc == w4.W4_ERR_INVALID_ARG
