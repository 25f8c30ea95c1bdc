"""ctypes binding of libw4a16.so: the C entry points under the same names, plus
torch-tensor conveniences that allocate outputs and pass the current stream.

Argument marshalling only: every step of quantization and of the matmul runs in
the library's CUDA kernels.  There is no CPU path; if the library is missing the
import fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libw4a16.so")

W4_OK = 0
W4_ERR_INVALID_ARG = 1
W4_ERR_UNSUPPORTED = 2
W4_ERR_MISALIGNED = 3
W4_ERR_CUDA = 4
W4_ERR_TIMEOUT = 5
W4_ERR_SCRATCH_LIMIT = 6
W4_NOALLOC_SCRATCH_BYTES = 16 << 20
W4_DTYPE_F16 = 0
W4_DTYPE_F32 = 1
W4_DTYPE_BF16 = 2
GROUP_SIZE = 128

# Symbols declared in include/w4a16.h (checked by the host-side tests).
EXPORTED = ("w4_quantize_pack", "w4_quantize_pack_sym", "w4_quantize_pack_percentile",
            "w4_quantize_pack_mse", "w4_dequantize", "w4_matmul", "w4_quantize_act_int8",
            "w4_matmul_w4a8", "w4_matmul_w4a8_workspace_size", "w4_matmul_w4a8_noalloc",
            "w4_gptq_quantize",
            "w4_status_string", "w4_check_device_error", "w4_set_wait_timeout_ns",
            "w4_debug_inject_stall")


class W4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libw4a16.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m w4a16_matmul_asym_b300.build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.w4_quantize_pack.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, vp, vp, vp, vp]
    lib.w4_quantize_pack.restype = ctypes.c_int
    lib.w4_quantize_pack_sym.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, vp, vp, vp, vp]
    lib.w4_quantize_pack_sym.restype = ctypes.c_int
    lib.w4_quantize_pack_percentile.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_float,
                                                vp, vp, vp, vp]
    lib.w4_quantize_pack_percentile.restype = ctypes.c_int
    lib.w4_quantize_pack_mse.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
    lib.w4_quantize_pack_mse.restype = ctypes.c_int
    lib.w4_dequantize.argtypes = [vp, vp, vp, i64, i64, ctypes.c_int, ctypes.c_int, vp, vp]
    lib.w4_dequantize.restype = ctypes.c_int
    lib.w4_matmul.argtypes = [vp, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp, vp]
    lib.w4_matmul.restype = ctypes.c_int
    lib.w4_quantize_act_int8.argtypes = [vp, i64, i64, vp, vp, vp]
    lib.w4_quantize_act_int8.restype = ctypes.c_int
    lib.w4_matmul_w4a8_workspace_size.argtypes = [i64, i64]
    lib.w4_matmul_w4a8_workspace_size.restype = ctypes.c_size_t
    lib.w4_matmul_w4a8.argtypes = [vp, vp, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.w4_matmul_w4a8.restype = ctypes.c_int
    lib.w4_matmul_w4a8_noalloc.argtypes = [vp, vp, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp, vp]
    lib.w4_matmul_w4a8_noalloc.restype = ctypes.c_int
    lib.w4_gptq_quantize.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, vp, vp, vp, vp, vp]
    lib.w4_gptq_quantize.restype = ctypes.c_int
    lib.w4_status_string.argtypes = [ctypes.c_int]
    lib.w4_status_string.restype = ctypes.c_char_p
    lib.w4_check_device_error.argtypes = [vp]
    lib.w4_check_device_error.restype = ctypes.c_int
    lib.w4_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.w4_set_wait_timeout_ns.restype = None
    lib.w4_debug_inject_stall.argtypes = [ctypes.c_int]
    lib.w4_debug_inject_stall.restype = None
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().w4_status_string(int(status)).decode()


# ---- raw C entry points (pointers and sizes) -------------------------------------
def w4_quantize_pack(W_ptr: int, w_dtype: int, N: int, K: int, group: int,
                     qweight_ptr: int, scales_ptr: int, zeros_ptr: int, stream: int) -> int:
    return load_library().w4_quantize_pack(W_ptr, w_dtype, N, K, group, qweight_ptr,
                                           scales_ptr, zeros_ptr, stream)


def w4_quantize_pack_sym(W_ptr: int, w_dtype: int, N: int, K: int, group: int,
                         qweight_ptr: int, scales_ptr: int, zeros_ptr: int, stream: int) -> int:
    return load_library().w4_quantize_pack_sym(W_ptr, w_dtype, N, K, group, qweight_ptr,
                                               scales_ptr, zeros_ptr, stream)


def w4_quantize_pack_percentile(W_ptr: int, w_dtype: int, N: int, K: int, group: int, p: float,
                                qweight_ptr: int, scales_ptr: int, zeros_ptr: int, stream: int) -> int:
    return load_library().w4_quantize_pack_percentile(W_ptr, w_dtype, N, K, group, p, qweight_ptr,
                                                      scales_ptr, zeros_ptr, stream)


def w4_quantize_pack_mse(W_ptr: int, w_dtype: int, N: int, K: int, group: int, candidates: int,
                         qweight_ptr: int, scales_ptr: int, zeros_ptr: int, stream: int) -> int:
    return load_library().w4_quantize_pack_mse(W_ptr, w_dtype, N, K, group, candidates, qweight_ptr,
                                               scales_ptr, zeros_ptr, stream)


def w4_dequantize(qweight_ptr: int, scales_ptr: int, zeros_ptr: int, N: int, K: int, group: int,
                  out_dtype: int, out_ptr: int, stream: int) -> int:
    return load_library().w4_dequantize(qweight_ptr, scales_ptr, zeros_ptr, N, K, group, out_dtype,
                                        out_ptr, stream)


def w4_matmul(A_ptr: int, M: int, N: int, K: int, group: int, qweight_ptr: int,
              scales_ptr: int, zeros_ptr: int, Y_ptr: int, stream: int) -> int:
    return load_library().w4_matmul(A_ptr, M, N, K, group, qweight_ptr, scales_ptr,
                                    zeros_ptr, Y_ptr, stream)


def w4_quantize_act_int8(A_ptr: int, M: int, K: int, aq_ptr: int, ascale_ptr: int, stream: int) -> int:
    return load_library().w4_quantize_act_int8(A_ptr, M, K, aq_ptr, ascale_ptr, stream)


def w4_matmul_w4a8_workspace_size(M: int, K: int) -> int:
    return int(load_library().w4_matmul_w4a8_workspace_size(M, K))


def w4_matmul_w4a8(aq_ptr: int, ascale_ptr: int, M: int, N: int, K: int, group: int, qweight_ptr: int,
                   scales_ptr: int, zeros_ptr: int, Y_ptr: int, ws_ptr: int, ws_bytes: int, stream: int) -> int:
    return load_library().w4_matmul_w4a8(aq_ptr, ascale_ptr, M, N, K, group, qweight_ptr, scales_ptr, zeros_ptr,
                                         Y_ptr, ws_ptr, ws_bytes, stream)


def w4_matmul_w4a8_noalloc(aq_ptr: int, ascale_ptr: int, M: int, N: int, K: int, group: int, qweight_ptr: int,
                           scales_ptr: int, zeros_ptr: int, Y_ptr: int, stream: int) -> int:
    """w4_matmul_w4a8 without a caller workspace: scratch from the library's fixed array."""
    return load_library().w4_matmul_w4a8_noalloc(aq_ptr, ascale_ptr, M, N, K, group, qweight_ptr, scales_ptr,
                                                 zeros_ptr, Y_ptr, stream)


def w4_gptq_quantize(W_ptr: int, w_dtype: int, N: int, K: int, group: int, U_ptr: int, qweight_ptr: int,
                     scales_ptr: int, zeros_ptr: int, stream: int) -> int:
    return load_library().w4_gptq_quantize(W_ptr, w_dtype, N, K, group, U_ptr, qweight_ptr, scales_ptr,
                                           zeros_ptr, stream)


def w4_check_device_error(stream: int = 0) -> int:
    return load_library().w4_check_device_error(stream)


def w4_set_wait_timeout_ns(ns: int) -> None:
    load_library().w4_set_wait_timeout_ns(int(ns))


def w4_debug_inject_stall(enable: bool) -> None:
    load_library().w4_debug_inject_stall(1 if enable else 0)


# ---- torch conveniences ------------------------------------------------------------
def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check_tables(qweight, scales, zeros, N: int, K: int, group: int, device) -> None:
    """The packed tables must be contiguous CUDA tensors of the documented dtypes and
    shapes on `device`: the C ABI takes bare pointers and cannot check their sizes, so a
    wrong shape here would let a kernel read or write past a buffer."""
    import torch
    ng = K // group if group > 0 else 0
    for name, t, dt, shape in (("qweight", qweight, torch.uint8, (N, K // 2)),
                               ("scales", scales, torch.float16, (N, ng)),
                               ("zeros", zeros, torch.uint8, (N, ng))):
        if t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous() or t.device != device:
            raise ValueError(f"{name} must be a contiguous {dt} tensor of shape {shape} on {device}, "
                             f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def quantize_pack(W, group: int = GROUP_SIZE, stream=None, out=None, symmetric: bool = False,
                  calibration: str | None = None, param=None):
    """Quantize a CUDA tensor W[N,K] (float16 or float32).

    Returns (qweight uint8 [N,K/2], scales float16 [N,K/128], zeros uint8 [N,K/128]),
    allocated with torch on W's device unless `out` supplies them.  symmetric=True runs
    w4_quantize_pack_sym (scale absmax / 7, zero points 8); calibration="percentile"
    (param = p, default 99.9) or "mse" (param = candidates, default 1000) runs the
    calibrated symmetric quantizers.
    """
    import torch
    if W.dim() != 2 or not W.is_cuda:
        raise ValueError("W must be a 2-D CUDA tensor")
    if W.dtype == torch.float16:
        dt = W4_DTYPE_F16
    elif W.dtype == torch.float32:
        dt = W4_DTYPE_F32
    else:
        raise TypeError("W must be float16 or float32")
    W = W.contiguous()
    N, K = W.shape
    if out is None:
        ng = K // group if group > 0 else 0
        qweight = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
        scales = torch.empty((N, ng), dtype=torch.float16, device=W.device)
        zeros = torch.empty((N, ng), dtype=torch.uint8, device=W.device)
    else:
        qweight, scales, zeros = out
        _check_tables(qweight, scales, zeros, N, K, group, W.device)
    if calibration is not None:
        if calibration == "percentile":
            rc = w4_quantize_pack_percentile(W.data_ptr(), dt, N, K, group, 99.9 if param is None else float(param),
                                             qweight.data_ptr(), scales.data_ptr(), zeros.data_ptr(),
                                             _stream_handle(stream))
        elif calibration == "mse":
            rc = w4_quantize_pack_mse(W.data_ptr(), dt, N, K, group, 1000 if param is None else int(param),
                                      qweight.data_ptr(), scales.data_ptr(), zeros.data_ptr(),
                                      _stream_handle(stream))
        else:
            raise ValueError("calibration must be None, 'percentile' or 'mse'")
        if rc != W4_OK:
            raise W4Error(rc, f"w4_quantize_pack_{calibration}")
        return qweight, scales, zeros
    fn, name = (w4_quantize_pack_sym, "w4_quantize_pack_sym") if symmetric else (w4_quantize_pack, "w4_quantize_pack")
    rc = fn(W.data_ptr(), dt, N, K, group, qweight.data_ptr(), scales.data_ptr(), zeros.data_ptr(),
            _stream_handle(stream))
    if rc != W4_OK:
        raise W4Error(rc, name)
    return qweight, scales, zeros


def dequantize(qweight, scales, zeros, dtype=None, group: int = GROUP_SIZE, stream=None, out=None):
    """W_hat[N,K] = (q - zp) * scale as a bfloat16 (default) or float16 CUDA tensor."""
    import torch
    dtype = torch.bfloat16 if dtype is None else dtype
    if dtype == torch.bfloat16:
        odt = W4_DTYPE_BF16
    elif dtype == torch.float16:
        odt = W4_DTYPE_F16
    else:
        raise TypeError("dtype must be torch.bfloat16 or torch.float16")
    if qweight.dim() != 2 or not qweight.is_cuda or qweight.dtype != torch.uint8:
        raise ValueError("qweight must be a 2-D uint8 CUDA tensor")
    if scales.dtype != torch.float16 or zeros.dtype != torch.uint8:
        raise TypeError("scales must be float16 and zeros uint8")
    N, K = qweight.shape[0], qweight.shape[1] * 2
    _check_tables(qweight, scales, zeros, N, K, group, qweight.device)
    if out is None:
        out = torch.empty((N, K), dtype=dtype, device=qweight.device)
    elif out.dtype != dtype or tuple(out.shape) != (N, K) or not out.is_contiguous() or out.device != qweight.device:
        raise ValueError(f"out must be a contiguous {dtype} tensor of shape ({N}, {K}) on {qweight.device}")
    rc = w4_dequantize(qweight.data_ptr(), scales.data_ptr(), zeros.data_ptr(), N, K, group, odt,
                       out.data_ptr(), _stream_handle(stream))
    if rc != W4_OK:
        raise W4Error(rc, "w4_dequantize")
    return out


def matmul(A, qweight, scales, zeros, group: int = GROUP_SIZE, stream=None, out=None):
    """Y[M,N] = A[M,K] (bfloat16, CUDA) times the dequantized weights, as bfloat16."""
    import torch
    if A.dim() != 2 or not A.is_cuda or A.dtype != torch.bfloat16:
        raise ValueError("A must be a 2-D bfloat16 CUDA tensor")
    A = A.contiguous()
    M, K = A.shape
    N = qweight.shape[0]
    if qweight.dtype != torch.uint8 or zeros.dtype != torch.uint8 or scales.dtype != torch.float16:
        raise TypeError("qweight/zeros must be uint8 and scales float16")
    if tuple(qweight.shape) != (N, K // 2):
        raise ValueError(f"qweight shape {tuple(qweight.shape)} does not match K={K}")
    _check_tables(qweight, scales, zeros, N, K, group, A.device)
    if out is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    else:
        if (out.dtype != torch.bfloat16 or tuple(out.shape) != (M, N) or not out.is_contiguous()
                or out.device != A.device):
            raise ValueError(f"out must be a contiguous bfloat16 tensor of shape ({M}, {N}) on {A.device}")
        Y = out
    rc = w4_matmul(A.data_ptr(), M, N, K, group, qweight.data_ptr(), scales.data_ptr(),
                   zeros.data_ptr(), Y.data_ptr(), _stream_handle(stream))
    if rc != W4_OK:
        raise W4Error(rc, "w4_matmul")
    return Y


def quantize_act_int8(A, stream=None, out=None):
    """Per-token INT8 activations of A[M,K] (bfloat16, CUDA): returns (a_q int8 [M,K],
    a_scale float32 [M]), allocated with torch unless `out` supplies them."""
    import torch
    if A.dim() != 2 or not A.is_cuda or A.dtype != torch.bfloat16:
        raise ValueError("A must be a 2-D bfloat16 CUDA tensor")
    A = A.contiguous()
    M, K = A.shape
    if out is None:
        aq = torch.empty((M, K), dtype=torch.int8, device=A.device)
        sa = torch.empty((M,), dtype=torch.float32, device=A.device)
    else:
        aq, sa = out
        if (aq.dtype != torch.int8 or tuple(aq.shape) != (M, K) or not aq.is_contiguous() or aq.device != A.device
                or sa.dtype != torch.float32 or tuple(sa.shape) != (M,) or not sa.is_contiguous()
                or sa.device != A.device):
            raise ValueError(f"out must be (int8 [{M}, {K}], float32 [{M}]) contiguous tensors on {A.device}")
    rc = w4_quantize_act_int8(A.data_ptr(), M, K, aq.data_ptr(), sa.data_ptr(), _stream_handle(stream))
    if rc != W4_OK:
        raise W4Error(rc, "w4_quantize_act_int8")
    return aq, sa


def matmul_w4a8(a_q, a_scale, qweight, scales, zeros, group: int = GROUP_SIZE, stream=None, out=None,
                workspace=None):
    """Y[M,N] = a_scale[m] * a_q[M,K] times the dequantized weights, as bfloat16.  The
    scratch workspace the call may need (w4_matmul_w4a8_workspace_size) is allocated
    with torch unless given."""
    import torch
    if a_q.dim() != 2 or not a_q.is_cuda or a_q.dtype != torch.int8:
        raise ValueError("a_q must be a 2-D int8 CUDA tensor")
    a_q = a_q.contiguous()
    M, K = a_q.shape
    if a_scale.dtype != torch.float32 or tuple(a_scale.shape) != (M,) or a_scale.device != a_q.device:
        raise ValueError(f"a_scale must be a float32 tensor of shape ({M},) on {a_q.device}")
    a_scale = a_scale.contiguous()
    N = qweight.shape[0]
    _check_tables(qweight, scales, zeros, N, K, group, a_q.device)
    if out is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=a_q.device)
    else:
        if (out.dtype != torch.bfloat16 or tuple(out.shape) != (M, N) or not out.is_contiguous()
                or out.device != a_q.device):
            raise ValueError(f"out must be a contiguous bfloat16 tensor of shape ({M}, {N}) on {a_q.device}")
        Y = out
    need = w4_matmul_w4a8_workspace_size(M, K)
    if workspace is None and need > 0:
        workspace = torch.empty((need,), dtype=torch.uint8, device=a_q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = w4_matmul_w4a8(a_q.data_ptr(), a_scale.data_ptr(), M, N, K, group, qweight.data_ptr(), scales.data_ptr(),
                        zeros.data_ptr(), Y.data_ptr(), ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != W4_OK:
        raise W4Error(rc, "w4_matmul_w4a8")
    return Y


def gptq_quantize(W, U, group: int = GROUP_SIZE, stream=None, out=None):
    """GPTQ quantization of a CUDA tensor W[N,K] (float16 or float32) given U (float32
    CUDA [K,K], the upper Cholesky factor of H^-1): returns (qweight, scales, zeros) in
    the layout of quantize_pack."""
    import torch
    if W.dim() != 2 or not W.is_cuda:
        raise ValueError("W must be a 2-D CUDA tensor")
    dt = {torch.float16: W4_DTYPE_F16, torch.float32: W4_DTYPE_F32}.get(W.dtype)
    if dt is None:
        raise TypeError("W must be float16 or float32")
    W = W.contiguous()
    N, K = W.shape
    if U.dtype != torch.float32 or tuple(U.shape) != (K, K) or U.device != W.device:
        raise ValueError(f"U must be a float32 tensor of shape ({K}, {K}) on {W.device}")
    U = U.contiguous()
    ng = K // group if group > 0 else 0
    if out is None:
        qweight = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
        scales = torch.empty((N, ng), dtype=torch.float16, device=W.device)
        zeros = torch.empty((N, ng), dtype=torch.uint8, device=W.device)
    else:
        qweight, scales, zeros = out
        _check_tables(qweight, scales, zeros, N, K, group, W.device)
    rc = w4_gptq_quantize(W.data_ptr(), dt, N, K, group, U.data_ptr(), qweight.data_ptr(), scales.data_ptr(),
                          zeros.data_ptr(), _stream_handle(stream))
    if rc != W4_OK:
        raise W4Error(rc, "w4_gptq_quantize")
    return qweight, scales, zeros
