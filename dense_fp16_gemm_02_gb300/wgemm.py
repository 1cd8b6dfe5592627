"""Python binding of libwgemm.so (ctypes): argument marshalling only.

Every name mirrors a C entry point declared in include/wgemm.h. The GEMM runs
entirely in the library's CUDA kernels; there is no fallback path: if the
library is not built, or the GPU is not an sm_103 part, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

WGEMM_OK = 0
STATUS_NAMES = {
    0: "WGEMM_OK", -1: "WGEMM_ERR_INVALID_ARG", -2: "WGEMM_ERR_ALIGNMENT", -3: "WGEMM_ERR_LAUNCH",
    -4: "WGEMM_ERR_NO_DEVICE", -5: "WGEMM_ERR_DEVICE_TIMEOUT", -6: "WGEMM_ERR_CONFIG",
    -7: "WGEMM_ERR_WORKSPACE", -8: "WGEMM_ERR_NOALLOC_TOO_LARGE",
}
MODE_DATA_PARALLEL, MODE_SPLIT_K, MODE_STREAM_K = 0, 1, 2
# Whole waves of tiles data parallel, the rest (partial last wave and `splits` − 1
# full waves before it) by stream-K.
MODE_HYBRID = 3
# Stream-K ranges with split-K's fix-up: each tile's owner zeroes it first and
# every unit adds its partial into C.
MODE_STREAM_K_ZERO = 4
WGEMM_F32, WGEMM_F16, WGEMM_BF16 = 0, 1, 2


class WgemmError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({status_string(code)})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load():
    """Load libwgemm.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "dense_fp16_gemm_02_gb300.build.build()")
        lib = ctypes.CDLL(path)
        i, p, u32, u64 = ctypes.c_int, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64
        lib.wgemm_f16f32.argtypes = [p, p, p, i, i, i, i, i, i, p]
        lib.wgemm_f16f32.restype = i
        lib.wgemm_f16f32_config.argtypes = [p, p, p, i, i, i, i, i, i, i, i, i, p]
        lib.wgemm_f16f32_config.restype = i
        lib.wgemm_f16f32_splitk_noalloc.argtypes = [p, p, p, i, i, i, i, i, i, i, p]
        lib.wgemm_f16f32_splitk_noalloc.restype = i
        lib.wgemm_f16f32_host.argtypes = [p, p, p, i, i, i, i, i, i, p, p, p, p]
        lib.wgemm_f16f32_host.restype = i
        sz = ctypes.POINTER(ctypes.c_size_t)
        lib.wgemm_host_device_elems.argtypes = [i, i, i, sz, sz, sz]
        lib.wgemm_host_device_elems.restype = i
        lib.wgemm_debug_set_host_panels.argtypes = [i]
        lib.wgemm_debug_set_host_panels.restype = i
        lib.wgemm_debug_host_panel_rows.argtypes = [i, i, i]
        lib.wgemm_debug_host_panel_rows.restype = i
        lib.wgemm_debug_set_host_blocks.argtypes = [i]
        lib.wgemm_debug_set_host_blocks.restype = i
        lib.wgemm_debug_host_block_cols.argtypes = [i, i]
        lib.wgemm_debug_host_block_cols.restype = i
        lib.wgemm_gemm.argtypes = [p, p, p, i, i, i, i, i, i, i, i, p]
        lib.wgemm_gemm.restype = i
        lib.wgemm_gemm_config.argtypes = [p, p, p, i, i, i, i, i, i, i, i, i, i, i, p]
        lib.wgemm_gemm_config.restype = i
        f = ctypes.c_float
        lib.wgemm_gemm_ex.argtypes = [p, p, p, p, p, f, f, i, i, i, i, i, i, i, i, i, p]
        lib.wgemm_gemm_ex.restype = i
        lib.wgemm_gemm_ex_config.argtypes = [p, p, p, p, p, f, f, i, i, i, i, i, i, i, i, i, i,
                                             p]
        lib.wgemm_gemm_ex_config.restype = i
        lib.wgemm_debug_config_fused.argtypes = [i]
        lib.wgemm_debug_config_fused.restype = i
        for name in ("wgemm_bf16f32", "wgemm_f16f16", "wgemm_bf16bf16"):
            getattr(lib, name).argtypes = [p, p, p, i, i, i, i, i, i, p]
            getattr(lib, name).restype = i
        lib.wgemm_set_pdl.argtypes = [i]
        lib.wgemm_set_pdl.restype = i
        lib.wgemm_num_configs.argtypes = []
        lib.wgemm_num_configs.restype = i
        lib.wgemm_config_name.argtypes = [i]
        lib.wgemm_config_name.restype = ctypes.c_char_p
        lib.wgemm_select.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i),
                                     ctypes.POINTER(i)]
        lib.wgemm_select.restype = i
        lib.wgemm_check.argtypes = [p]
        lib.wgemm_check.restype = i
        lib.wgemm_last_device_error.argtypes = [ctypes.POINTER(i)] * 4
        lib.wgemm_last_device_error.restype = i
        lib.wgemm_status_string.argtypes = [i]
        lib.wgemm_status_string.restype = ctypes.c_char_p
        lib.wgemm_workspace_bytes.argtypes = []
        lib.wgemm_workspace_bytes.restype = ctypes.c_size_t
        lib.wgemm_release_workspace.argtypes = []
        lib.wgemm_release_workspace.restype = i
        lib.wgemm_debug_set_trace.argtypes = [p, i]
        lib.wgemm_debug_set_trace.restype = i
        lib.wgemm_debug_trace_build.argtypes = []
        lib.wgemm_debug_trace_build.restype = i
        lib.wgemm_debug_max_workers.argtypes = [i]
        lib.wgemm_debug_max_workers.restype = i
        lib.wgemm_debug_predict_us.argtypes = [i] * 9
        lib.wgemm_debug_predict_us.restype = ctypes.c_double
        lib.wgemm_debug_set_flag_wait_skew.argtypes = [i]
        lib.wgemm_debug_set_flag_wait_skew.restype = i
        lib.wgemm_debug_set_cooperative.argtypes = [i]
        lib.wgemm_debug_set_cooperative.restype = i
        lib.wgemm_debug_smem_desc.argtypes = [u32]
        lib.wgemm_debug_smem_desc.restype = u64
        lib.wgemm_debug_idesc.argtypes = [i, i, i]
        lib.wgemm_debug_idesc.restype = u32
        lib.wgemm_debug_config_out.argtypes = [i]
        lib.wgemm_debug_config_out.restype = i
        lib.wgemm_debug_sw128_offset.argtypes = [u32, u32]
        lib.wgemm_debug_sw128_offset.restype = u32
        lib.wgemm_debug_plan.argtypes = [i, i, i, i, i, i, i, p, i, ctypes.POINTER(i),
                                         ctypes.POINTER(i)]
        lib.wgemm_debug_plan.restype = i
        _lib = lib
        return lib


def header_functions() -> list[str]:
    """Names of the functions include/wgemm.h declares."""
    hdr = os.path.join(os.path.dirname(_build.HERE), "include", "wgemm.h")
    text = open(hdr).read()
    return sorted(set(re.findall(r"^\s*[\w\s\*]*?\b(wgemm_\w+)\s*\(", text, re.M)))


def status_string(code: int) -> str:
    try:
        return load().wgemm_status_string(code).decode()
    except RuntimeError:
        return STATUS_NAMES.get(code, "unknown")


def wgemm_set_pdl(enable: bool) -> int:
    """Programmatic dependent launch on or off (process-wide); returns the
    previous setting."""
    rc = load().wgemm_set_pdl(1 if enable else 0)
    if rc < 0:
        raise WgemmError(rc, "wgemm_set_pdl")
    return rc


def num_configs() -> int:
    return load().wgemm_num_configs()


def config_name(config_id: int) -> str:
    return load().wgemm_config_name(config_id).decode()


def config_names() -> list[str]:
    return [config_name(i) for i in range(num_configs())]


def config_id(name: str) -> int:
    names = config_names()
    if name not in names:
        raise KeyError(name)
    return names.index(name)


def wgemm_f16f32(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                 stream: int | None) -> int:
    """The raw C call on device pointers; returns the status code."""
    return load().wgemm_f16f32(A, B, C, M, N, K, lda, ldb, ldc, stream)


def wgemm_f16f32_config(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                        ldc: int, config: int, mode: int, splits: int,
                        stream: int | None) -> int:
    return load().wgemm_f16f32_config(A, B, C, M, N, K, lda, ldb, ldc, config, mode, splits,
                                      stream)


def wgemm_gemm(A: int, B: int, C: int, ab_type: int, c_type: int, M: int, N: int, K: int,
               lda: int, ldb: int, ldc: int, stream: int | None) -> int:
    """The typed C call on device pointers; returns the status code."""
    return load().wgemm_gemm(A, B, C, ab_type, c_type, M, N, K, lda, ldb, ldc, stream)


def wgemm_gemm_config(A: int, B: int, C: int, ab_type: int, c_type: int, M: int, N: int, K: int,
                      lda: int, ldb: int, ldc: int, config: int, mode: int, splits: int,
                      stream: int | None) -> int:
    return load().wgemm_gemm_config(A, B, C, ab_type, c_type, M, N, K, lda, ldb, ldc, config,
                                    mode, splits, stream)


def wgemm_bf16f32(A, B, C, M, N, K, lda, ldb, ldc, stream) -> int:
    return load().wgemm_bf16f32(A, B, C, M, N, K, lda, ldb, ldc, stream)


def wgemm_f16f16(A, B, C, M, N, K, lda, ldb, ldc, stream) -> int:
    return load().wgemm_f16f16(A, B, C, M, N, K, lda, ldb, ldc, stream)


def wgemm_bf16bf16(A, B, C, M, N, K, lda, ldb, ldc, stream) -> int:
    return load().wgemm_bf16bf16(A, B, C, M, N, K, lda, ldb, ldc, stream)


def wgemm_gemm_ex(A, B, D, Cin, bias, alpha, beta, ab_type, c_type, M, N, K, lda, ldb, ldd,
                  ldcin, stream) -> int:
    """The fused-epilogue C call on device pointers; returns the status code."""
    return load().wgemm_gemm_ex(A, B, D, Cin, bias, alpha, beta, ab_type, c_type, M, N, K, lda,
                                ldb, ldd, ldcin, stream)


def wgemm_gemm_ex_config(A, B, D, Cin, bias, alpha, beta, ab_type, c_type, M, N, K, lda, ldb,
                         ldd, ldcin, config, stream) -> int:
    return load().wgemm_gemm_ex_config(A, B, D, Cin, bias, alpha, beta, ab_type, c_type, M, N,
                                       K, lda, ldb, ldd, ldcin, config, stream)


def config_fused(config: int) -> int:
    """1 if the configuration has the alpha/beta/bias epilogue, else 0."""
    return load().wgemm_debug_config_fused(config)


def config_out(config: int) -> int:
    """0 if the configuration writes fp32 C, 1 if 16-bit C."""
    return load().wgemm_debug_config_out(config)


def wgemm_f16f32_splitk_noalloc(A: int, B: int, C: int, M: int, N: int, K: int, lda: int,
                                ldb: int, ldc: int, splits: int, stream: int | None) -> int:
    """Split-K on device pointers with the library's fixed scratch array (no
    allocation); returns the status code."""
    return load().wgemm_f16f32_splitk_noalloc(A, B, C, M, N, K, lda, ldb, ldc, splits, stream)


def wgemm_f16f32_host(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                      ldc: int, dA: int, dB: int, dC: int, stream: int | None) -> int:
    """A, B and C in host memory (pinned for overlap), through the caller's
    device buffers dA, dB, dC (sizes from host_device_elems); returns the
    status code."""
    return load().wgemm_f16f32_host(A, B, C, M, N, K, lda, ldb, ldc, dA, dB, dC, stream)


def host_device_elems(M: int, N: int, K: int) -> tuple[int, int, int]:
    """Element counts of the device buffers wgemm_f16f32_host needs:
    (A: M·kd fp16, B: N·kd fp16, C: M·nd fp32)."""
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    rc = load().wgemm_host_device_elems(M, N, K, ctypes.byref(a), ctypes.byref(b),
                                        ctypes.byref(c))
    if rc != 0:
        raise ValueError(status_string(rc))
    return a.value, b.value, c.value


def gemm_from_host(A, B, stream=None):
    """C = A·Bᵀ for fp16 torch tensors in (pinned) host memory: C comes back
    as a new pinned fp32 host tensor; the device buffers are allocated here
    (torch) for this call. Asynchronous on `stream` (default: the current
    one): synchronise before reading C."""
    import torch

    if A.is_cuda or B.is_cuda or A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("gemm_from_host takes fp16 host tensors")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("A is M×K and B is N×K")
    if A.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("rows must be contiguous")
    M, K = A.shape
    N = B.shape[0]
    na, nb, nc = host_device_elems(M, N, K)
    dev = torch.device("cuda", torch.cuda.current_device())
    dA = torch.empty(max(na, 1), dtype=torch.float16, device=dev)
    dB = torch.empty(max(nb, 1), dtype=torch.float16, device=dev)
    dC = torch.empty(max(nc, 1), dtype=torch.float32, device=dev)
    C = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = wgemm_f16f32_host(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, A.stride(0),
                           B.stride(0), N, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                           s.cuda_stream)
    if rc != 0:
        raise RuntimeError(status_string(rc))
    # The device buffers must outlive the enqueued work.
    dA.record_stream(s)
    dB.record_stream(s)
    dC.record_stream(s)
    return C


def wgemm_select(M: int, N: int, K: int, lda: int | None = None, ldb: int | None = None,
                 c_type: int = WGEMM_F32, fused: int = 0) -> tuple[int, int, int]:
    """(configuration id, mode, splits) that the library runs for this shape,
    these row pitches (K when omitted), this C type and epilogue: fused 0
    (plain), 1 (alpha/beta/bias) or 2 (in place with beta = 1, fp32 D; a
    bool True counts as 1)."""
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    c, m, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = load().wgemm_select(M, N, K, lda, ldb, c_type, int(fused), ctypes.byref(c),
                             ctypes.byref(m), ctypes.byref(s))
    if rc != WGEMM_OK:
        raise WgemmError(rc, "wgemm_select")
    return c.value, m.value, s.value


def wgemm_check(stream: int | None = None) -> int:
    return load().wgemm_check(stream)


def wgemm_last_device_error() -> dict:
    vals = [ctypes.c_int() for _ in range(4)]
    code = load().wgemm_last_device_error(*[ctypes.byref(v) for v in vals])
    return {"code": code, "block": vals[0].value, "warp": vals[1].value,
            "site": vals[2].value, "parity": vals[3].value}


def wgemm_workspace_bytes() -> int:
    return load().wgemm_workspace_bytes()


def wgemm_release_workspace() -> int:
    return load().wgemm_release_workspace()


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _wgemm_type(dtype) -> int:
    import torch
    types = {torch.float32: WGEMM_F32, torch.float16: WGEMM_F16, torch.bfloat16: WGEMM_BF16}
    if dtype not in types:
        raise TypeError(f"unsupported element type {dtype}")
    return types[dtype]


def gemm_ex(A, B, D=None, *, Cin=None, bias=None, alpha: float = 1.0, beta: float = 0.0,
            out_dtype=None, config: int | str | None = None, stream=None):
    """D = alpha·A·Bᵀ + beta·Cin + bias[None, :] for torch tensors (the fused
    epilogue): A, B as for gemm(); Cin of D's type (M×N, may be D itself);
    bias an N-element float32 tensor. D is allocated when not given."""
    import torch
    if A.dtype not in (torch.float16, torch.bfloat16) or B.dtype != A.dtype:
        raise TypeError("A and B must both be float16 or both bfloat16")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("A must be M×K and B N×K")
    if A.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("A and B need a contiguous last dimension")
    M, K = A.shape
    N = B.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    if D.shape != (M, N) or D.stride(1) != 1:
        raise ValueError("D must be M×N with a contiguous last dimension")
    if Cin is not None and (Cin.shape != (M, N) or Cin.stride(1) != 1 or Cin.dtype != D.dtype):
        raise ValueError("Cin must be M×N of D's type with a contiguous last dimension")
    if bias is not None and (bias.dtype != torch.float32 or bias.numel() != N
                             or not bias.is_contiguous()):
        raise ValueError("bias must be N contiguous float32 values")
    ab_type, c_type = _wgemm_type(A.dtype), _wgemm_type(D.dtype)
    if M == 0 or N == 0:
        return D
    h = _stream_handle(stream)
    cid = -1 if config is None else (config_id(config) if isinstance(config, str) else int(config))
    rc = wgemm_gemm_ex_config(A.data_ptr(), B.data_ptr(), D.data_ptr(),
                              None if Cin is None else Cin.data_ptr(),
                              None if bias is None else bias.data_ptr(), float(alpha),
                              float(beta), ab_type, c_type, M, N, K, max(A.stride(0), K),
                              max(B.stride(0), K), D.stride(0),
                              N if Cin is None else Cin.stride(0), cid, h)
    if rc != WGEMM_OK:
        raise WgemmError(rc, "wgemm_gemm_ex")
    return D


def gemm(A, B, C=None, *, out_dtype=None, config: int | str | None = None, mode: int = -1,
         splits: int = 1, stream=None):
    """C = A·Bᵀ for torch tensors: A (M×K) and B (N×K) both float16 or both
    bfloat16; C (M×N) float32 (the default), float16 or bfloat16.

    A and B may have a row stride larger than K (a column slice of a wider
    tensor); their last dimension must be contiguous. C is allocated (of
    `out_dtype`, default float32) when not given. The work is enqueued on
    `stream` (default: torch's current stream).
    """
    import torch
    if A.dtype not in (torch.float16, torch.bfloat16) or B.dtype != A.dtype:
        raise TypeError("A and B must both be float16 or both bfloat16")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("A must be M×K and B N×K")
    if A.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("A and B need a contiguous last dimension")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    if C.shape != (M, N) or C.stride(1) != 1:
        raise ValueError("C must be M×N with a contiguous last dimension")
    ab_type, c_type = _wgemm_type(A.dtype), _wgemm_type(C.dtype)
    lda, ldb, ldc = A.stride(0), B.stride(0), C.stride(0)
    if M == 0 or N == 0:
        return C
    h = _stream_handle(stream)
    if config is None:
        rc = wgemm_gemm(A.data_ptr(), B.data_ptr(), C.data_ptr(), ab_type, c_type, M, N, K,
                        max(lda, K), max(ldb, K), ldc, h)
    else:
        cid = config_id(config) if isinstance(config, str) else int(config)
        rc = wgemm_gemm_config(A.data_ptr(), B.data_ptr(), C.data_ptr(), ab_type, c_type, M, N,
                               K, max(lda, K), max(ldb, K), ldc, cid, mode, splits, h)
    if rc != WGEMM_OK:
        raise WgemmError(rc, "wgemm_gemm")
    return C
