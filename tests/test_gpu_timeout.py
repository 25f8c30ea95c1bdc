"""Failure detection without a GPU fault: the consumers of the tensor-core GEMM
(M = 64), of the integer-dot decode GEMV (M = 1), of the warp-MMA decode kernel with
its activations in registers (M = 3) and in shared memory (M = 12), and of the
quantize kernel are made
to wait on a barrier that nothing signals; the bounded wait must run out, record
W4_ERR_TIMEOUT in the device error word, drain its copies, free tensor memory and
exit.  The context must stay usable (a normal call afterwards is correct)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [1, 3, 12, 64])
def test_injected_stall_times_out_and_context_survives(oracle_mod, M):
    import torch
    import synth
    from w4a16_matmul_asym_b300 import build
    build.build()
    import w4a16_matmul_asym_b300 as w4
    W, A = synth.make_random(512, 2048, M, seed=77)
    q, s, z = oracle_mod.quantize_pack(W)
    Ad = torch.from_numpy(A.view(np.int16)).cuda().view(torch.bfloat16)
    qd, sd, zd = (torch.from_numpy(x).cuda() for x in (q, s, z))
    assert w4.w4_check_device_error(0) == w4.W4_OK
    w4.w4_set_wait_timeout_ns(20_000_000)        # 20 ms
    w4.w4_debug_inject_stall(True)
    try:
        w4.matmul(Ad, qd, sd, zd)
        rc = w4.w4_check_device_error(0)
    finally:
        w4.w4_debug_inject_stall(False)
        w4.w4_set_wait_timeout_ns(0)
    assert rc == w4.W4_ERR_TIMEOUT
    assert w4.w4_check_device_error(0) == w4.W4_OK   # the word was cleared
    Y = w4.matmul(Ad, qd, sd, zd)
    torch.cuda.synchronize()
    Yref, S = oracle_mod.matmul(A, q, s, z)
    ok, worst, _ = oracle_mod.check_y(Y.view(torch.int16).cpu().numpy().view(np.uint16), Yref, S)
    assert ok, worst


def test_quantize_stall_times_out_and_context_survives(oracle_mod):
    """The quantize kernel's consumers wait on a barrier nothing signals: the bounded
    wait records W4_ERR_TIMEOUT, the producer drains its copies, and the next call is
    bit-exact."""
    import torch
    import synth
    from w4a16_matmul_asym_b300 import build
    build.build()
    import w4a16_matmul_asym_b300 as w4
    W, _ = synth.make_random(300, 4096, 1, seed=78)
    Wd = torch.from_numpy(W).cuda()
    assert w4.w4_check_device_error(0) == w4.W4_OK
    w4.w4_set_wait_timeout_ns(20_000_000)        # 20 ms
    w4.w4_debug_inject_stall(True)
    try:
        w4.quantize_pack(Wd)
        rc = w4.w4_check_device_error(0)
    finally:
        w4.w4_debug_inject_stall(False)
        w4.w4_set_wait_timeout_ns(0)
    assert rc == w4.W4_ERR_TIMEOUT
    assert w4.w4_check_device_error(0) == w4.W4_OK
    q, s, z = w4.quantize_pack(Wd)
    torch.cuda.synchronize()
    qo, so, zo = oracle_mod.quantize_pack(W)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), so.view(np.uint16))
    assert np.array_equal(z.cpu().numpy(), zo)
