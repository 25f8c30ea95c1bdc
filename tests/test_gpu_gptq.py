"""GPU parity of GPTQ ("Build a GPTQ INT4 Quantization Engine in Python/NumPy", Step
3): the column-greedy quantization with error feedback, bit-exact against the CPU
oracle (same fp32 operations, each column's updates applied in ascending order), on
the same U factor, through the C ABI."""
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


_FACTORS = {}


def correlated_factor(orc, K, seed):
    """U from synthetic calibration activations X [K + 64, K] ~ N(0, 1) with
    neighbouring inputs correlated (x_k += 0.9 x_(k-1)): a dense factor.  Cached per
    (K, seed): the fp64 Hessian inverse of K = 8192 takes seconds."""
    if (K, seed) not in _FACTORS:
        rng = np.random.default_rng(seed)
        X = rng.standard_normal((K + 64, K))
        X[:, 1:] += 0.9 * X[:, :-1]
        _FACTORS[(K, seed)] = orc.gptq_factor(X)
    return _FACTORS[(K, seed)]


def assert_gptq_equal(env, W, U):
    torch, w4, orc = env
    q, s, z = w4.gptq_quantize(torch.from_numpy(np.ascontiguousarray(W)).cuda(), torch.from_numpy(U).cuda())
    torch.cuda.synchronize()
    assert w4.w4_check_device_error(0) == w4.W4_OK
    q, s, z = q.cpu().numpy(), s.cpu().numpy(), z.cpu().numpy()
    qo, so, zo = orc.gptq_quantize(W, U)
    assert np.array_equal(s.view(np.uint16), so.view(np.uint16)), "scales differ"
    assert np.array_equal(z, zo), "zeros differ"
    if not np.array_equal(q, qo):
        bad = np.argwhere(q != qo)
        raise AssertionError(f"qweight differs at {len(bad)} bytes, first {bad[:5].tolist()}")


@pytest.mark.parametrize("N,K", [(1, 128), (7, 512), (9, 1024), (100, 4096), (13, 2048), (9, 8192), (5, 6144)])
@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_gptq_matches_oracle(env, N, K, dtype):
    import synth
    _, _, orc = env
    W, _ = synth.make_random(N, K, 1, seed=N + K)
    assert_gptq_equal(env, W.astype(dtype), correlated_factor(orc, K, seed=K))


def test_gptq_hand_worked_case(env):
    K = 128
    U = np.eye(K, dtype=np.float32)
    U[0, 0], U[0, 1] = 2.0, -4.0
    w = np.zeros((1, K), np.float32)
    w[0, :4] = [0.5625, 1.25, -1.5, 2.25]
    assert_gptq_equal(env, w, U)


def test_gptq_identity_factor_is_round_to_nearest(env):
    """With U = I the GPU GPTQ output equals the GPU round-to-nearest quantizer's."""
    import synth
    torch, w4, _ = env
    W, _ = synth.make_random(64, 1024, 1, seed=3)
    Wd = torch.from_numpy(W).cuda()
    a = w4.gptq_quantize(Wd, torch.eye(1024, dtype=torch.float32, device="cuda"))
    b = w4.quantize_pack(Wd)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_gptq_llama7b_shape_sampled_rows(env):
    """The Llama-7B-shaped weights at full size (N = 11008, K = 4096); 6 sampled rows
    compared bit-exactly with the oracle on those rows."""
    import synth
    torch, w4, orc = env
    W, _ = synth.make_workload("llama7b_gemv")
    U = correlated_factor(orc, 4096, seed=4096)
    q, s, z = w4.gptq_quantize(torch.from_numpy(W).cuda(), torch.from_numpy(U).cuda())
    torch.cuda.synchronize()
    rows = np.random.default_rng(5).choice(W.shape[0], 6, replace=False)
    qo, so, zo = orc.gptq_quantize(W[rows], U)
    assert np.array_equal(q.cpu().numpy()[rows], qo) and np.array_equal(z.cpu().numpy()[rows], zo)
    assert np.array_equal(s.cpu().numpy()[rows].view(np.uint16), so.view(np.uint16))
