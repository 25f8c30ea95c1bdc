"""Failure detection without a GPU fault: the consumers of the tensor-core GEMM
(M = 64), of the split-K tensor-core kernel (M = 12), of the integer-dot decode GEMV
(M = 1) and of the streaming GEMV with activations in shared memory (M = 3) are made
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
