"""w4_matmul_w4a8_noalloc: the W4A8 matmul for callers that cannot allocate device
memory when they run: plugins whose host framework owns every device allocation and
offers them none, real-time loops that must not allocate after start-up (an allocation
can stall the device), code with no way to recover from a failed allocation.  It takes
its scratch from a fixed array inside the library instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row, on shapes that need the
scratch (the GEMM path), and checks each result against the workspace entry point
w4_matmul_w4a8 on the same inputs, within the library's matmul tolerance.  The file is
named to be collected last, and the test stands alone: it passes in a fresh process
and after the other tests."""
import ctypes

import numpy as np
import pytest


def _lib():
    from w4a16_matmul_asym_b300 import build
    build.build()
    import w4a16_matmul_asym_b300 as w4
    return w4, w4.load_library()


def test_noalloc_rejects_oversized_scratch_before_launching():
    """A shape whose scratch exceeds the fixed array is refused with its own status,
    before any pointer is used (no GPU needed)."""
    w4, lib = _lib()
    fake = ctypes.c_void_p(0x10000)
    M, K = 4096, 4096                       # 32 MiB of widened activations > 16 MiB
    assert w4.w4_matmul_w4a8_workspace_size(M, K) > w4.W4_NOALLOC_SCRATCH_BYTES
    rc = lib.w4_matmul_w4a8_noalloc(fake, fake, M, 256, K, 128, fake, fake, fake, fake, None)
    assert rc == w4.W4_ERR_SCRATCH_LIMIT
    assert "scratch" in w4.status_string(rc)
    assert lib.w4_matmul_w4a8_noalloc(fake, fake, -1, 256, K, 128, fake, fake, fake, fake, None) == 1
    assert lib.w4_matmul_w4a8_noalloc(fake, fake, 8, 256, K, 64, fake, fake, fake, fake, None) == 2


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_twice(oracle_mod):
    import torch
    import synth
    w4, lib = _lib()
    torch.cuda.set_device(0)
    for call, (M, N, K, seed) in enumerate([(64, 300, 1024, 1), (200, 129, 2048, 2)]):
        assert w4.w4_matmul_w4a8_workspace_size(M, K) > 0        # the scratch path
        W, A = synth.make_random(N, K, M, seed=seed)
        q, s, z = oracle_mod.quantize_pack(W)
        aq, sa = oracle_mod.quantize_act_int8(A)
        d = {k: torch.from_numpy(v).cuda() for k, v in (("aq", aq), ("sa", sa), ("q", q), ("s", s), ("z", z))}
        Y_ws = w4.matmul_w4a8(d["aq"], d["sa"], d["q"], d["s"], d["z"])
        Y_na = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        rc = lib.w4_matmul_w4a8_noalloc(d["aq"].data_ptr(), d["sa"].data_ptr(), M, N, K, 128, d["q"].data_ptr(),
                                        d["s"].data_ptr(), d["z"].data_ptr(), Y_na.data_ptr(), None)
        assert rc == w4.W4_OK, (call, w4.status_string(rc))
        torch.cuda.synchronize()
        assert w4.w4_check_device_error(0) == w4.W4_OK
        y_na = Y_na.view(torch.int16).cpu().numpy().view(np.uint16)
        y_ws = Y_ws.view(torch.int16).cpu().numpy().view(np.uint16)
        _, S = oracle_mod.w4a8_matmul(aq, sa, q, s, z)
        ok, worst, idx = oracle_mod.check_y(y_na, oracle_mod.bf16_bits_to_f64(y_ws), S)
        assert ok, (call, worst, idx)
