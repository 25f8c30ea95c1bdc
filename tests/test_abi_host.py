"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
exports every function include/w4a16.h declares, and rejects invalid arguments
with the documented status before touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    from w4a16_matmul_asym_b300 import build
    build.build()
    import w4a16_matmul_asym_b300 as w4
    return w4.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("w4_quantize_pack", "w4_matmul", "w4_status_string", "w4_check_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
    import w4a16_matmul_asym_b300 as w4
    assert set(w4.EXPORTED) == set(declared_functions())


def test_status_strings(lib):
    import w4a16_matmul_asym_b300 as w4
    for code in range(6):
        s = w4.status_string(code)
        assert s and s.startswith("W4_")
    assert "unknown" in w4.status_string(99)


FAKE = 0x10000  # a 16-byte-aligned, never-dereferenced address


@pytest.mark.parametrize("args,expect", [
    ((FAKE, 0, -1, 128, 128), 1),        # negative N
    ((FAKE, 0, 4, -128, 128), 1),        # negative K
    ((FAKE, 0, 4, 130, 128), 1),         # K not a multiple of the group (checked after group)
    ((FAKE, 0, 4, 128, 64), 2),          # group 64 unsupported
    ((FAKE, 0, 4, 128, 0), 1),           # group 0
    ((FAKE, 7, 4, 128, 128), 1),         # unknown dtype
    ((0, 0, 4, 128, 128), 1),            # null W
    ((FAKE + 8, 0, 4, 128, 128), 3),     # misaligned W
    ((FAKE, 0, 0, 128, 128), 0),         # empty: N == 0
    ((FAKE, 0, 4, 0, 128), 0),           # empty: K == 0
])
def test_quantize_pack_validation(lib, args, expect):
    W, dt, N, K, G = args
    rc = lib.w4_quantize_pack(W, dt, N, K, G, FAKE, FAKE, FAKE, None)
    assert rc == expect


def test_quantize_pack_null_and_misaligned_outputs(lib):
    assert lib.w4_quantize_pack(FAKE, 0, 4, 128, 128, 0, FAKE, FAKE, None) == 1
    assert lib.w4_quantize_pack(FAKE, 0, 4, 128, 128, FAKE, 0, FAKE, None) == 1
    assert lib.w4_quantize_pack(FAKE, 0, 4, 128, 128, FAKE, FAKE, 0, None) == 1
    assert lib.w4_quantize_pack(FAKE, 0, 4, 128, 128, FAKE + 4, FAKE, FAKE, None) == 3
    assert lib.w4_quantize_pack(FAKE, 0, 4, 128, 128, FAKE, FAKE + 1, FAKE, None) == 3


@pytest.mark.parametrize("args,expect", [
    ((FAKE, -1, 4, 128, 128), 1),
    ((FAKE, 1, -4, 128, 128), 1),
    ((FAKE, 1, 4, -128, 128), 1),
    ((FAKE, 1, 4, 100, 128), 1),
    ((FAKE, 1, 4, 256, 32), 2),
    ((FAKE, 0, 4, 256, 128), 0),         # M == 0: nothing to do
    ((FAKE, 3, 0, 256, 128), 0),         # N == 0: nothing to do
    ((0, 3, 4, 256, 128), 1),            # null A
    ((FAKE + 2, 3, 4, 256, 128), 3),     # misaligned A
])
def test_matmul_validation(lib, args, expect):
    A, M, N, K, G = args
    rc = lib.w4_matmul(A, M, N, K, G, FAKE, FAKE, FAKE, FAKE, None)
    assert rc == expect


def test_matmul_null_and_misaligned(lib):
    assert lib.w4_matmul(FAKE, 2, 4, 256, 128, 0, FAKE, FAKE, FAKE, None) == 1
    assert lib.w4_matmul(FAKE, 2, 4, 256, 128, FAKE, 0, FAKE, FAKE, None) == 1
    assert lib.w4_matmul(FAKE, 2, 4, 256, 128, FAKE, FAKE, 0, FAKE, None) == 1
    assert lib.w4_matmul(FAKE, 2, 4, 256, 128, FAKE, FAKE, FAKE, 0, None) == 1
    assert lib.w4_matmul(FAKE, 2, 4, 256, 128, FAKE + 8, FAKE, FAKE, FAKE, None) == 3
    assert lib.w4_matmul(FAKE, 2, 4, 256, 128, FAKE, FAKE + 1, FAKE, FAKE, None) == 3
    assert lib.w4_matmul(FAKE, 2, 4, 256, 128, FAKE, FAKE, FAKE, FAKE + 1, None) == 3


@pytest.mark.parametrize("args,expect", [
    ((FAKE, 0, -1, 128, 128), 1),
    ((FAKE, 0, 4, 130, 128), 1),
    ((FAKE, 0, 4, 128, 64), 2),
    ((FAKE, 7, 4, 128, 128), 1),
    ((0, 0, 4, 128, 128), 1),
    ((FAKE + 8, 1, 4, 128, 128), 3),
    ((FAKE, 0, 0, 128, 128), 0),
    ((FAKE, 1, 4, 0, 128), 0),
])
def test_quantize_pack_sym_validation(lib, args, expect):
    """The symmetric quantizer validates exactly as w4_quantize_pack."""
    W, dt, N, K, G = args
    assert lib.w4_quantize_pack_sym(W, dt, N, K, G, FAKE, FAKE, FAKE, None) == expect
    assert lib.w4_quantize_pack_sym(FAKE, 0, 4, 128, 128, FAKE + 4, FAKE, FAKE, None) == 3
    assert lib.w4_quantize_pack_sym(FAKE, 0, 4, 128, 128, FAKE, FAKE, 0, None) == 1


BF16, F16, F32 = 2, 0, 1


@pytest.mark.parametrize("args,expect", [
    ((-1, 256, 128, BF16), 1),           # negative N
    ((4, -256, 128, BF16), 1),           # negative K
    ((4, 100, 128, BF16), 1),            # K not a multiple of the group
    ((4, 256, 64, BF16), 2),             # group 64 unsupported
    ((4, 256, 128, F32), 1),             # fp32 output is not offered
    ((4, 256, 128, 9), 1),               # unknown dtype
    ((0, 256, 128, F16), 0),             # empty
    ((4, 0, 128, BF16), 0),              # empty
])
def test_dequantize_validation(lib, args, expect):
    N, K, G, dt = args
    assert lib.w4_dequantize(FAKE, FAKE, FAKE, N, K, G, dt, FAKE, None) == expect


def test_dequantize_null_and_misaligned(lib):
    assert lib.w4_dequantize(0, FAKE, FAKE, 4, 256, 128, BF16, FAKE, None) == 1
    assert lib.w4_dequantize(FAKE, 0, FAKE, 4, 256, 128, BF16, FAKE, None) == 1
    assert lib.w4_dequantize(FAKE, FAKE, 0, 4, 256, 128, BF16, FAKE, None) == 1
    assert lib.w4_dequantize(FAKE, FAKE, FAKE, 4, 256, 128, BF16, 0, None) == 1
    assert lib.w4_dequantize(FAKE + 4, FAKE, FAKE, 4, 256, 128, BF16, FAKE, None) == 3
    assert lib.w4_dequantize(FAKE, FAKE + 1, FAKE, 4, 256, 128, BF16, FAKE, None) == 3
    assert lib.w4_dequantize(FAKE, FAKE, FAKE, 4, 256, 128, F16, FAKE + 8, None) == 3


def test_binding_fails_loudly_without_library(tmp_path):
    from w4a16_matmul_asym_b300 import _binding
    with pytest.raises(ImportError):
        _binding._lib_saved = _binding._lib
        try:
            _binding._lib = None
            _binding.load_library(str(tmp_path / "missing.so"))
        finally:
            _binding._lib = _binding._lib_saved


@pytest.mark.parametrize("args,expect", [
    ((FAKE, 0, -1, 128, 128), 1),
    ((FAKE, 0, 4, 130, 128), 1),
    ((FAKE, 0, 4, 128, 64), 2),
    ((FAKE, 7, 4, 128, 128), 1),
    ((0, 0, 4, 128, 128), 1),
    ((FAKE + 8, 1, 4, 128, 128), 3),
    ((FAKE, 0, 0, 128, 128), 0),
    ((FAKE, 1, 4, 0, 128), 0),
])
def test_calibrated_quantizers_validation(lib, args, expect):
    """The percentile and MSE quantizers validate as w4_quantize_pack, plus their
    parameter ranges: p in (0, 100], candidates in [1, 2^24]."""
    W, dt, N, K, G = args
    assert lib.w4_quantize_pack_percentile(W, dt, N, K, G, ctypes.c_float(99.9), FAKE, FAKE, FAKE, None) == expect
    assert lib.w4_quantize_pack_mse(W, dt, N, K, G, 1000, FAKE, FAKE, FAKE, None) == expect


@pytest.mark.parametrize("p", [0.0, -1.0, 100.5, float("nan"), float("inf")])
def test_percentile_parameter_range(lib, p):
    assert lib.w4_quantize_pack_percentile(FAKE, 0, 4, 128, 128, ctypes.c_float(p), FAKE, FAKE, FAKE, None) == 1


@pytest.mark.parametrize("n", [0, -5, (1 << 24) + 1])
def test_mse_candidate_range(lib, n):
    assert lib.w4_quantize_pack_mse(FAKE, 0, 4, 128, 128, n, FAKE, FAKE, FAKE, None) == 1


def test_act_int8_validation(lib):
    """Per-token activation quantizer: sizes, K % 8, nulls, alignment, empty."""
    assert lib.w4_quantize_act_int8(FAKE, -1, 128, FAKE, FAKE, None) == 1
    assert lib.w4_quantize_act_int8(FAKE, 4, 12, FAKE, FAKE, None) == 1
    assert lib.w4_quantize_act_int8(FAKE, 0, 128, FAKE, FAKE, None) == 0
    assert lib.w4_quantize_act_int8(0, 4, 128, FAKE, FAKE, None) == 1
    assert lib.w4_quantize_act_int8(FAKE, 4, 128, FAKE, 0, None) == 1
    assert lib.w4_quantize_act_int8(FAKE + 8, 4, 128, FAKE, FAKE, None) == 3
    assert lib.w4_quantize_act_int8(FAKE, 4, 128, FAKE + 8, FAKE, None) == 3
    assert lib.w4_quantize_act_int8(FAKE, 4, 128, FAKE, FAKE + 2, None) == 3


def test_w4a8_workspace_size(lib):
    """Decode shapes (M <= 16, K a multiple of 2048, activations fitting in shared
    memory) need no workspace; others need M * K * 2 bytes rounded up to 256."""
    assert lib.w4_matmul_w4a8_workspace_size(1, 4096) == 0
    assert lib.w4_matmul_w4a8_workspace_size(16, 4096) == 0
    assert lib.w4_matmul_w4a8_workspace_size(17, 4096) == 17 * 4096 * 2
    assert lib.w4_matmul_w4a8_workspace_size(3, 1000 // 8 * 8 + 128 * 8) == -(-3 * 2024 * 2 // 256) * 256
    assert lib.w4_matmul_w4a8_workspace_size(2048, 4096) == 2048 * 4096 * 2
    assert lib.w4_matmul_w4a8_workspace_size(0, 4096) == 0


def test_w4a8_matmul_validation(lib):
    args = (FAKE, FAKE, 2, 4, 256, 128, FAKE, FAKE, FAKE, FAKE, 0, 0, None)
    assert lib.w4_matmul_w4a8(*args[:2], -1, *args[3:]) == 1
    assert lib.w4_matmul_w4a8(*args[:5], 64, *args[6:]) == 2
    assert lib.w4_matmul_w4a8(*args[:4], 200, *args[5:]) == 1
    assert lib.w4_matmul_w4a8(*args[:2], 0, *args[3:]) == 0
    assert lib.w4_matmul_w4a8(0, *args[1:]) == 1
    assert lib.w4_matmul_w4a8(FAKE + 8, *args[1:]) == 3
    assert lib.w4_matmul_w4a8(FAKE, FAKE + 2, *args[2:]) == 3
    assert lib.w4_matmul_w4a8(*args[:9], FAKE + 1, *args[10:]) == 3


def test_gptq_validation(lib):
    args = [FAKE, 0, 4, 256, 128, FAKE, FAKE, FAKE, FAKE, None]   # never called as is: it would launch
    bad = list(args); bad[2] = -1
    assert lib.w4_gptq_quantize(*bad) == 1
    bad = list(args); bad[4] = 64
    assert lib.w4_gptq_quantize(*bad) == 2
    bad = list(args); bad[3] = 200
    assert lib.w4_gptq_quantize(*bad) == 1
    bad = list(args); bad[3] = 16384
    assert lib.w4_gptq_quantize(*bad) == 2
    bad = list(args); bad[5] = 0
    assert lib.w4_gptq_quantize(*bad) == 1
    bad = list(args); bad[5] = FAKE + 4
    assert lib.w4_gptq_quantize(*bad) == 3
    bad = list(args); bad[2] = 0
    assert lib.w4_gptq_quantize(*bad) == 0
