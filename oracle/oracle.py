"""CPU oracle for group-wise asymmetric INT4 quantization and the W4A16 matmul.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this module.  The CUDA
library never calls it and shares no code with it.

The arithmetic lives in ``w4a16_oracle.c`` (plain C, fp32 quantization steps,
fp64 matmul), compiled here with ``gcc -O2 -ffp-contract=off`` and loaded with
ctypes.  This module only marshals numpy arrays and states the output tolerance.

Sources (page titles): "From-Scratch INT4 Weight-Only Quantizer with Per-Group
Scales and Zero-Points" (Architecture Overview item 3; Steps 5-6), "From
Scratch: Building a GPTQ INT4 Quantizer in Pure Python" (Step 2, Step 4), "Build
a GPTQ INT4 Quantization Engine in Python/NumPy" (Step 4 packing, Step 5
chunked dequantize-matmul).  Each C function cites the step it follows.

Pinning: every function here is checked in ``tests/test_oracle_pins.py`` against
hand-worked groups (``tests/golden/``), the packing example printed on the
GPTQ/NumPy page, closed forms, invariants and exhaustive small cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

GROUP = 128
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "libw4a16_oracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math",
           "-std=c11", "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc) into oracle/_build and return the .so path."""
    with _lock:
        os.makedirs(_BUILD_DIR, exist_ok=True)
        stale = (not os.path.exists(_SO)
                 or os.path.getmtime(_SO) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _SO + f".tmp{os.getpid()}"
            cmd = ["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.oracle_quantize_pack.argtypes = [vp, ctypes.c_int, i64, i64, vp, vp, vp, vp]
    lib.oracle_quantize_pack.restype = ctypes.c_int
    lib.oracle_quantize_pack_sym.argtypes = [vp, ctypes.c_int, i64, i64, vp, vp, vp, vp]
    lib.oracle_quantize_pack_sym.restype = ctypes.c_int
    lib.oracle_quantize_pack_calib.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_double,
                                               vp, vp, vp, vp]
    lib.oracle_quantize_pack_calib.restype = ctypes.c_int
    lib.oracle_percentile_abs.argtypes = [vp, ctypes.c_int, ctypes.c_float]
    lib.oracle_percentile_abs.restype = ctypes.c_float
    lib.oracle_mse_step.argtypes = [vp, ctypes.c_int, ctypes.c_int]
    lib.oracle_mse_step.restype = ctypes.c_float
    lib.oracle_quantize_act_int8.argtypes = [vp, i64, i64, vp, vp]
    lib.oracle_quantize_act_int8.restype = ctypes.c_int
    lib.oracle_w4a8_matmul.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp, dp, dp]
    lib.oracle_w4a8_matmul.restype = ctypes.c_int
    lib.oracle_w4a8_matmul_entries.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp, vp, vp, i64, dp, dp]
    lib.oracle_w4a8_matmul_entries.restype = ctypes.c_int
    lib.oracle_gptq_quantize.argtypes = [vp, ctypes.c_int, i64, i64, vp, vp, vp, vp]
    lib.oracle_gptq_quantize.restype = ctypes.c_int
    lib.oracle_dequantize_16.argtypes = [vp, vp, vp, i64, i64, ctypes.c_int, vp]
    lib.oracle_dequantize_16.restype = ctypes.c_int
    lib.oracle_f32_to_bf16_bits.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16_bits.restype = ctypes.c_uint16
    lib.oracle_unpack.argtypes = [vp, i64, i64, vp]
    lib.oracle_unpack.restype = ctypes.c_int
    lib.oracle_dequantize.argtypes = [vp, vp, vp, i64, i64, dp]
    lib.oracle_dequantize.restype = ctypes.c_int
    lib.oracle_matmul.argtypes = [vp, i64, i64, i64, vp, vp, vp, dp, dp]
    lib.oracle_matmul.restype = ctypes.c_int
    lib.oracle_matmul_entries.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, vp, i64, dp, dp]
    lib.oracle_matmul_entries.restype = ctypes.c_int
    lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_f16_bits.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_f16_bits.restype = ctypes.c_uint16
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_u16_bits(x: np.ndarray) -> np.ndarray:
    """fp16 / bf16-as-uint16 arrays -> contiguous uint16 bit patterns."""
    if x.dtype == np.float16:
        return np.ascontiguousarray(x).view(np.uint16)
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x)
    raise TypeError(f"expected float16 or uint16 bit patterns, got {x.dtype}")


def quantize_pack(W: np.ndarray, with_fp32_scales: bool = False, symmetric: bool = False):
    """Quantize W[N,K] (float16 or float32) with groups of 128 along K.

    Returns (qweight uint8 [N,K/2], scales float16 [N,K/128], zeros uint8 [N,K/128])
    and, if asked, the fp32 scales [N,K/128] used for q and zp.  symmetric=True takes
    the absmax / 7 variant (levels q + 8, zero points 8).
    """
    if W.ndim != 2:
        raise ValueError("W must be 2-D [N,K]")
    N, K = W.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    if W.dtype == np.float16:
        src, dt = _as_u16_bits(W), 0
    elif W.dtype == np.float32:
        src, dt = np.ascontiguousarray(W), 1
    else:
        raise TypeError("W must be float16 or float32")
    ng = K // GROUP
    q = np.empty((N, K // 2), np.uint8)
    s = np.empty((N, ng), np.uint16)
    z = np.empty((N, ng), np.uint8)
    s32 = np.empty((N, ng), np.float32)
    fn = _load().oracle_quantize_pack_sym if symmetric else _load().oracle_quantize_pack
    rc = fn(_ptr(src), dt, N, K, _ptr(q), _ptr(s), _ptr(z), _ptr(s32))
    if rc:
        raise RuntimeError(f"oracle_quantize_pack failed ({rc})")
    out = (q, s.view(np.float16), z)
    return out + (s32,) if with_fp32_scales else out


CALIB_METHODS = {"percentile": 2, "mse": 3}


def quantize_pack_calibrated(W: np.ndarray, method: str, param: float, with_fp32_scales: bool = False):
    """Clip-range calibrated symmetric quantization of W[N,K] (float16 or float32):
    method "percentile" (param = p, the percentile of |w| taken as the clip range) or
    "mse" (param = number of linspace candidate steps).  Same outputs as
    quantize_pack: levels clamp(rint(w / s), -7, 7) + 8, zero points 8, fp16 scales."""
    if W.ndim != 2:
        raise ValueError("W must be 2-D [N,K]")
    N, K = W.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    if W.dtype == np.float16:
        src, dt = _as_u16_bits(W), 0
    elif W.dtype == np.float32:
        src, dt = np.ascontiguousarray(W), 1
    else:
        raise TypeError("W must be float16 or float32")
    ng = K // GROUP
    q = np.empty((N, K // 2), np.uint8)
    s = np.empty((N, ng), np.uint16)
    z = np.empty((N, ng), np.uint8)
    s32 = np.empty((N, ng), np.float32)
    rc = _load().oracle_quantize_pack_calib(_ptr(src), dt, N, K, CALIB_METHODS[method], float(param),
                                            _ptr(q), _ptr(s), _ptr(z), _ptr(s32))
    if rc:
        raise RuntimeError(f"oracle_quantize_pack_calib failed ({rc})")
    out = (q, s.view(np.float16), z)
    return out + (s32,) if with_fp32_scales else out


def percentile_abs(group: np.ndarray, p: float) -> np.float32:
    """The percentile calibrator's clip range for one group (fp32 values)."""
    g = np.ascontiguousarray(group, dtype=np.float32)
    return np.float32(_load().oracle_percentile_abs(_ptr(g), len(g), float(p)))


def mse_step(group: np.ndarray, n: int) -> np.float32:
    """The MSE calibrator's chosen step for one group (fp32 values)."""
    g = np.ascontiguousarray(group, dtype=np.float32)
    return np.float32(_load().oracle_mse_step(_ptr(g), len(g), int(n)))


def gptq_factor(X: np.ndarray, damp: float = 1e-4) -> np.ndarray:
    """The upper Cholesky factor U of H^-1 (H^-1 = U^T U) from calibration activations
    X [n, K], with H = X^T X / n + damp * mean(diag(H)) * I ("Build a GPTQ INT4
    Quantization Engine in Python/NumPy", Step 3, compute_hessian), computed in fp64
    with numpy's inverse and Cholesky and returned as fp32 (the quantizer's input)."""
    X = np.asarray(X, np.float64)
    H = X.T @ X / X.shape[0]
    H += damp * np.mean(np.diag(H)) * np.eye(H.shape[0])
    Hinv = np.linalg.inv(H)
    L = np.linalg.cholesky(Hinv)          # Hinv = L L^T, L lower
    return np.ascontiguousarray(L.T, dtype=np.float32)


def gptq_quantize(W: np.ndarray, U: np.ndarray):
    """GPTQ quantization of W[N,K] (float16 or float32) given U (fp32 [K,K]): returns
    (qweight, scales float16, zeros) in the layout of quantize_pack."""
    N, K = W.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    if W.dtype == np.float16:
        src, dt = _as_u16_bits(W), 0
    elif W.dtype == np.float32:
        src, dt = np.ascontiguousarray(W), 1
    else:
        raise TypeError("W must be float16 or float32")
    U = np.ascontiguousarray(U, dtype=np.float32)
    if U.shape != (K, K):
        raise ValueError("U must be [K, K]")
    ng = K // GROUP
    q = np.empty((N, K // 2), np.uint8)
    s = np.empty((N, ng), np.uint16)
    z = np.empty((N, ng), np.uint8)
    if _load().oracle_gptq_quantize(_ptr(src), dt, N, K, _ptr(U), _ptr(q), _ptr(s), _ptr(z)):
        raise RuntimeError("oracle_gptq_quantize failed")
    return q, s.view(np.float16), z


def unpack(qweight: np.ndarray, K: int) -> np.ndarray:
    """qweight uint8 [N,K/2] -> q uint8 [N,K]."""
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    N = qweight.shape[0]
    q = np.empty((N, K), np.uint8)
    if _load().oracle_unpack(_ptr(qweight), N, K, _ptr(q)):
        raise RuntimeError("oracle_unpack failed")
    return q


def dequantize(qweight, scales, zeros, K: int) -> np.ndarray:
    """(q - zp) * fp16 scale, in float64, [N,K]."""
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    s = _as_u16_bits(scales)
    z = np.ascontiguousarray(zeros, dtype=np.uint8)
    N = qweight.shape[0]
    out = np.empty((N, K), np.float64)
    if _load().oracle_dequantize(_ptr(qweight), _ptr(s), _ptr(z), N, K, _ptr(out)):
        raise RuntimeError("oracle_dequantize failed")
    return out


def dequantize16(qweight, scales, zeros, K: int, out_dtype: str = "bf16") -> np.ndarray:
    """(q - zp) * fp16 scale rounded once to bfloat16 or float16, as uint16 bit
    patterns [N,K]."""
    if out_dtype not in ("bf16", "fp16"):
        raise ValueError("out_dtype must be 'bf16' or 'fp16'")
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    s = _as_u16_bits(scales)
    z = np.ascontiguousarray(zeros, dtype=np.uint8)
    N = qweight.shape[0]
    out = np.empty((N, K), np.uint16)
    rc = _load().oracle_dequantize_16(_ptr(qweight), _ptr(s), _ptr(z), N, K,
                                      0 if out_dtype == "bf16" else 1, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_dequantize_16 failed ({rc})")
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Element-wise binary32 -> bfloat16 bit patterns (round to nearest even)."""
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    return np.array([lib.oracle_f32_to_bf16_bits(float(v)) for v in flat], np.uint16).reshape(np.shape(x))


def matmul(A_bf16: np.ndarray, qweight, scales, zeros):
    """Y = A @ W_hat^T in float64 for A given as bf16 bit patterns (uint16) [M,K].

    Returns (Y float64 [M,N], S float64 [M,N]) with S = sum_k |A[m,k] * w_hat[n,k]|.
    """
    A = _as_u16_bits(A_bf16)
    M, K = A.shape
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    s = _as_u16_bits(scales)
    z = np.ascontiguousarray(zeros, dtype=np.uint8)
    N = qweight.shape[0]
    Y = np.empty((M, N), np.float64)
    S = np.empty((M, N), np.float64)
    if _load().oracle_matmul(_ptr(A), M, N, K, _ptr(qweight), _ptr(s), _ptr(z), _ptr(Y), _ptr(S)):
        raise RuntimeError("oracle_matmul failed")
    return Y, S


def quantize_act_int8(A_bf16: np.ndarray):
    """Per-token INT8 activations of A [M,K] (bf16 bit patterns): (a_q int8 [M,K],
    s_a float32 [M]) with s_a = max(max|a|, 1e-8) / 127, a_q = clip(rint(a / s_a),
    -128, 127), all in fp32."""
    A = _as_u16_bits(A_bf16)
    M, K = A.shape
    aq = np.empty((M, K), np.int8)
    sa = np.empty((M,), np.float32)
    if _load().oracle_quantize_act_int8(_ptr(A), M, K, _ptr(aq), _ptr(sa)):
        raise RuntimeError("oracle_quantize_act_int8 failed")
    return aq, sa


def w4a8_matmul(a_q: np.ndarray, a_scale: np.ndarray, qweight, scales, zeros):
    """Y = (a_q * s_a) @ W_hat^T in float64, with S = sum_k |a_q s_a w_hat|: returns
    (Y float64 [M,N], S float64 [M,N])."""
    aq = np.ascontiguousarray(a_q, dtype=np.int8)
    sa = np.ascontiguousarray(a_scale, dtype=np.float32)
    M, K = aq.shape
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    s = _as_u16_bits(scales)
    z = np.ascontiguousarray(zeros, dtype=np.uint8)
    N = qweight.shape[0]
    Y = np.empty((M, N), np.float64)
    S = np.empty((M, N), np.float64)
    if _load().oracle_w4a8_matmul(_ptr(aq), _ptr(sa), M, N, K, _ptr(qweight), _ptr(s), _ptr(z),
                                  _ptr(Y), _ptr(S)):
        raise RuntimeError("oracle_w4a8_matmul failed")
    return Y, S


def w4a8_matmul_entries(a_q, a_scale, qweight, scales, zeros, mi, ni):
    """The W4A8 fp64 result and S for the listed (m, n) positions only."""
    aq = np.ascontiguousarray(a_q, dtype=np.int8)
    sa = np.ascontiguousarray(a_scale, dtype=np.float32)
    M, K = aq.shape
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    s = _as_u16_bits(scales)
    z = np.ascontiguousarray(zeros, dtype=np.uint8)
    N = qweight.shape[0]
    mi = np.ascontiguousarray(mi, dtype=np.int64)
    ni = np.ascontiguousarray(ni, dtype=np.int64)
    Y = np.empty(len(mi), np.float64)
    S = np.empty(len(mi), np.float64)
    if _load().oracle_w4a8_matmul_entries(_ptr(aq), _ptr(sa), M, N, K, _ptr(qweight), _ptr(s), _ptr(z),
                                          _ptr(mi), _ptr(ni), len(mi), _ptr(Y), _ptr(S)):
        raise RuntimeError("oracle_w4a8_matmul_entries failed")
    return Y, S


def matmul_entries(A_bf16, qweight, scales, zeros, mi, ni):
    """The fp64 result and S for the listed (m, n) positions only."""
    A = _as_u16_bits(A_bf16)
    M, K = A.shape
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    s = _as_u16_bits(scales)
    z = np.ascontiguousarray(zeros, dtype=np.uint8)
    N = qweight.shape[0]
    mi = np.ascontiguousarray(mi, dtype=np.int64)
    ni = np.ascontiguousarray(ni, dtype=np.int64)
    Y = np.empty(mi.shape[0], np.float64)
    S = np.empty(mi.shape[0], np.float64)
    rc = _load().oracle_matmul_entries(_ptr(A), M, N, K, _ptr(qweight), _ptr(s), _ptr(z),
                                       _ptr(mi), _ptr(ni), mi.shape[0], _ptr(Y), _ptr(S))
    if rc:
        raise RuntimeError(f"oracle_matmul_entries failed ({rc})")
    return Y, S


def f16_to_f32(bits: int) -> float:
    return float(_load().oracle_f16_to_f32(bits))


def f32_to_f16_bits(x: float) -> int:
    return int(_load().oracle_f32_to_f16_bits(x))


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(bits))


# ---- output tolerance --------------------------------------------------------
# |Y - Y_ref| <= 8e-3 * S + 0.5 * ulp_bf16(|Y_ref|), per element, where
# ulp_bf16(x) = 2^(floor(log2 x) - 7) for normal x and the smallest bf16
# subnormal 2^-133 below the normal range (and at 0).
REL_TOL = 8e-3
_BF16_MIN_SUBNORMAL = 2.0 ** -133
_BF16_MIN_NORMAL = 2.0 ** -126


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    x = np.abs(np.asarray(x, dtype=np.float64))
    out = np.full(x.shape, _BF16_MIN_SUBNORMAL)
    nz = x >= _BF16_MIN_NORMAL
    e = np.floor(np.log2(np.where(nz, x, 1.0)))
    out[nz] = np.ldexp(1.0, (e[nz] - 7).astype(np.int64))
    return out


def y_tolerance(Y_ref: np.ndarray, S: np.ndarray) -> np.ndarray:
    return REL_TOL * np.asarray(S, np.float64) + 0.5 * ulp_bf16(Y_ref)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 patterns -> float64 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def check_y(Y_bits: np.ndarray, Y_ref: np.ndarray, S: np.ndarray):
    """Compare bf16 outputs (uint16 bit patterns) with the fp64 reference.

    Returns (ok, worst_ratio, index_of_worst) where ratio = |err| / tolerance.
    """
    Y = bf16_bits_to_f64(Y_bits).reshape(np.shape(Y_ref))
    err = np.abs(Y - Y_ref)
    tol = y_tolerance(Y_ref, S)
    ratio = err / tol
    if ratio.size == 0:
        return True, 0.0, None
    idx = int(np.argmax(ratio))
    worst = float(ratio.reshape(-1)[idx])
    ok = bool(np.all(np.isfinite(Y))) and worst <= 1.0
    return ok, worst, np.unravel_index(idx, ratio.shape)
