"""Python binding of the fine-grained FP8 GEMM library (``libfp8fg.so``).

Argument marshalling only: torch tensors supply device pointers, shapes and
the current CUDA stream; every step of the computation runs in the library's
CUDA kernels. The functions carry the names of the C entry points declared
in ``include/fp8fg.h``; the ``*_out`` variants write into caller-provided
tensors and allocate nothing.

The shared library is loaded on first use (so that the ``build`` submodule
can be imported before it exists); any call without the built library
raises ImportError: there is no fallback path. Build it with
``python -m fp8_fine_grained_24_b300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8fg.so")


class _Library:
    """ctypes handle of libfp8fg.so, opened (and typed) on first attribute access."""

    def __init__(self):
        self._cdll = None
        self._lock = threading.Lock()

    def _open(self):
        with self._lock:
            if self._cdll is None:
                if not os.path.exists(LIB_PATH):
                    raise ImportError(
                        f"{LIB_PATH} is missing: build it with `python -m fp8_fine_grained_24_b300.build` "
                        "(nvcc, sm_103a). The library has no non-CUDA fallback.")
                cdll = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in _SIGS.items():
                    f = getattr(cdll, name)
                    f.restype = res
                    f.argtypes = args
                self._cdll = cdll
        return self._cdll

    def __getattr__(self, name):
        if name.startswith("_"):
            raise AttributeError(name)
        return getattr(self._cdll if self._cdll is not None else self._open(), name)


lib = _Library()

# ---------------------------------------------------------------- constants
OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED_SHAPE = -2
ERR_MISALIGNED = -3
ERR_CUDA = -4
ERR_TIMEOUT = -5

BF16, FP32, E4M3 = 0, 1, 2
SCALE_BLOCK128, SCALE_ROW, SCALE_ROW_POW2 = 0, 1, 2
MASK_ROWS, MASK_K = 0, 1

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_c_vp = ctypes.c_void_p
_c_sz = ctypes.c_size_t

_SIGS = {
    "fp8fg_scale_ld": (_c_i64, [_c_i64]),
    "fp8_quant_1x128": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_int, _c_vp]),
    "fp8_quant_128x128": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_int, _c_vp]),
    "fp8_requant_128x1": (_c_int, [_c_vp, _c_int, _c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_int,
                                   _c_vp]),
    "fp8_gemm_dense": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_int, _c_int, _c_i64, _c_i64, _c_i64,
                                _c_vp, _c_sz, _c_vp]),
    "fp8fg_gemm_workspace_size": (_c_sz, [_c_i64, _c_i64, _c_i64]),
    "fp8_gemm_dgrad": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_i64, _c_i64, _c_i64, _c_vp,
                                _c_sz, _c_vp]),
    "fp8_gemm_dense_quant": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_vp, _c_vp, _c_int, _c_i64, _c_i64,
                                      _c_i64, _c_vp, _c_sz, _c_vp]),
    "fp8_gemm_grouped_contig": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_i64, _c_i64, _c_i64,
                                         _c_i64, _c_vp]),
    "fp8_gemm_grouped_masked": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_int, _c_vp, _c_int, _c_int,
                                         _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_vp]),
    "fp8fg_check": (_c_int, [_c_vp]),
    "fp8fg_last_error_string": (ctypes.c_char_p, []),
    "fp8fg_version": (ctypes.c_char_p, []),
    "fp8fg_debug_set": (_c_int, [_c_int, _c_i64]),
    "fp8_gemm_dense_noalloc": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_int, _c_int, _c_i64, _c_i64,
                                        _c_i64, _c_vp]),
    "fp8fg_study_mma_accumulation": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_vp]),
}


class Fp8fgError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"fp8fg error {code}: {msg}")
        self.code = code


def _check(rc: int):
    if rc != OK:
        raise Fp8fgError(rc, lib.fp8fg_last_error_string().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_DT = {torch.bfloat16: BF16, torch.float32: FP32, torch.uint8: E4M3, torch.float8_e4m3fn: E4M3}


def _dtype_code(t):
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _as_u8(t):
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


def scale_ld(rows: int) -> int:
    """Row stride (floats) of per-row scale arrays: rows rounded up to 4."""
    return int(lib.fp8fg_scale_ld(int(rows)))


def version() -> str:
    return lib.fp8fg_version().decode()


def check(stream=None):
    """Synchronize the stream and raise if a device-side wait timed out."""
    _check(lib.fp8fg_check(_stream(stream)))


def debug_set(key: int, value: int):
    _check(lib.fp8fg_debug_set(int(key), int(value)))


# K split of decode-sized dense GEMMs (fp8fg_debug_set key 4)
SPLIT_AUTO, SPLIT_STREAM, SPLIT_CLUSTER = 0, 1, 2


def set_split_policy(policy: int):
    """Automatic, Stream-K over the workspace only, or the cluster split wherever it applies."""
    debug_set(4, policy)


# ---------------------------------------------------------------- quantizers
def fp8_quant_1x128_out(x, q, s, pow2=False, stream=None):
    M, K = x.shape
    _check(lib.fp8_quant_1x128(_ptr(x), _dtype_code(x), M, K, x.stride(0), _ptr(q), _ptr(s), int(bool(pow2)),
                               _stream(stream)))
    return q, s


def fp8_quant_1x128(x, pow2=False, stream=None):
    """x [M, K] bf16/fp32 -> (q [M, K] uint8 E4M3, s [K/128, ld(M)] fp32)."""
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((K // 128, scale_ld(M)), dtype=torch.float32, device=x.device)
    return fp8_quant_1x128_out(x, q, s, pow2, stream)


def fp8_quant_128x128_out(w, q, s, pow2=False, stream=None):
    w3 = w if w.dim() == 3 else w.unsqueeze(0)
    G, N, K = w3.shape
    _check(lib.fp8_quant_128x128(_ptr(w3), _dtype_code(w3), G, N, K, _ptr(q), _ptr(s), int(bool(pow2)),
                                 _stream(stream)))
    return q, s


def fp8_quant_128x128(w, pow2=False, stream=None):
    """w [N, K] or [G, N, K] -> (q same shape uint8, s [(G,) ceil(N/128), K/128] fp32)."""
    assert w.is_contiguous()
    lead = w.shape[:-2]
    N, K = w.shape[-2:]
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    s = torch.empty((*lead, (N + 127) // 128, K // 128), dtype=torch.float32, device=w.device)
    return fp8_quant_128x128_out(w, q, s, pow2, stream)


def fp8_requant_128x1_out(src, s_src, qT, sT, valid_rows=None, pow2=False, stream=None):
    src3 = src if src.dim() == 3 else src.unsqueeze(0)
    G, T, C = src3.shape
    _check(lib.fp8_requant_128x1(_ptr(_as_u8(src3)), _dtype_code(src3), _ptr(s_src), G, T, C, _ptr(valid_rows),
                                 _ptr(qT), _ptr(sT), int(bool(pow2)), _stream(stream)))
    return qT, sT


def fp8_requant_128x1(src, s_src=None, valid_rows=None, pow2=False, stream=None):
    """src [(G,) T, C] E4M3 (with s_src [(G,) C/128, ld(T)]) or bf16/fp32
    -> (qT [(G,) C, T] uint8, sT [(G,) T/128, ld(C)] fp32)."""
    assert src.is_contiguous()
    lead = src.shape[:-2]
    T, C = src.shape[-2:]
    qT = torch.empty((*lead, C, T), dtype=torch.uint8, device=src.device)
    sT = torch.empty((*lead, T // 128, scale_ld(C)), dtype=torch.float32, device=src.device)
    return fp8_requant_128x1_out(src, s_src, qT, sT, valid_rows, pow2, stream)


# ---------------------------------------------------------------- GEMMs
def gemm_workspace_size(M: int, N: int, K: int) -> int:
    """Stream-K workspace bytes for a dense GEMM on the current device (0: none).

    The cluster split, which the automatic policy prefers for decode-sized
    problems, uses no workspace; the size covers the Stream-K plan that the
    policy may choose instead."""
    return int(lib.fp8fg_gemm_workspace_size(M, N, K))


def gemm_workspace(M: int, N: int, K: int, device="cuda"):
    """A zero-filled workspace tensor for fp8_gemm_dense_out, or None if not needed."""
    nbytes = gemm_workspace_size(M, N, K)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device) if nbytes else None


def fp8_gemm_dense_out(a, sa, b, sb, c, b_scale_kind=SCALE_BLOCK128, accumulate=False, workspace=None,
                       stream=None):
    M, K = a.shape
    N = b.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.fp8_gemm_dense(_ptr(_as_u8(a)), _ptr(sa), _ptr(_as_u8(b)), _ptr(sb), int(b_scale_kind), _ptr(c),
                              _dtype_code(c), int(bool(accumulate)), M, N, K, _ptr(workspace), ws_bytes,
                              _stream(stream)))
    return c


def fp8_gemm_dense(a, sa, b, sb, out_dtype=torch.bfloat16, b_scale_kind=SCALE_BLOCK128, stream=None):
    """C[M, N] = (a * sa) @ (b * sb)^T with FP32 promotion per 128-K block."""
    M, K = a.shape
    N = b.shape[0]
    c = torch.empty((M, N), dtype=out_dtype, device=a.device)
    ws = None
    nbytes = gemm_workspace_size(M, N, K)
    if nbytes:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=a.device)  # counters start at zero
    return fp8_gemm_dense_out(a, sa, b, sb, c, b_scale_kind, False, ws, stream)


def fp8_gemm_dgrad_out(dy, s_dy, w, sw, dx, accumulate=False, workspace=None, stream=None):
    """dX[M, K] (+)= dY[M, N] @ W[N, K] from dY's 1x128 and W's 128x128 quantization."""
    M, N = dy.shape
    K = w.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.fp8_gemm_dgrad(_ptr(_as_u8(dy)), _ptr(s_dy), _ptr(_as_u8(w)), _ptr(sw), _ptr(dx), _dtype_code(dx),
                              int(bool(accumulate)), M, N, K, _ptr(workspace), ws_bytes, _stream(stream)))
    return dx


def fp8_gemm_dgrad(dy, s_dy, w, sw, out_dtype=torch.bfloat16, stream=None):
    """dX = dY @ W with W read as its own transpose (no transposed copy)."""
    M = dy.shape[0]
    N, K = w.shape
    dx = torch.empty((M, K), dtype=out_dtype, device=dy.device)
    ws = gemm_workspace(M, K, N, device=dy.device)
    return fp8_gemm_dgrad_out(dy, s_dy, w, sw, dx, False, ws, stream)


def fp8_gemm_dense_quant_out(a, sa, b, sb, q, s, c=None, pow2=False, workspace=None, stream=None):
    """Dense GEMM whose BF16 result is quantized per 1x128 tile in the epilogue:
    q [M, N] uint8 E4M3, s [N/128, ld(M)] fp32; c (BF16 [M, N]) optional."""
    M, K = a.shape
    N = b.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.fp8_gemm_dense_quant(_ptr(_as_u8(a)), _ptr(sa), _ptr(_as_u8(b)), _ptr(sb), SCALE_BLOCK128, _ptr(q),
                                    _ptr(s), _ptr(c), int(bool(pow2)), M, N, K, _ptr(workspace), ws_bytes,
                                    _stream(stream)))
    return q, s


def fp8_gemm_dense_quant(a, sa, b, sb, pow2=False, with_bf16=False, stream=None):
    """(q, s) or (q, s, c): the GEMM's result quantized per 1x128 tile (and its BF16 form)."""
    M, K = a.shape
    N = b.shape[0]
    q = torch.empty((M, N), dtype=torch.uint8, device=a.device)
    s = torch.empty((N // 128, scale_ld(M)), dtype=torch.float32, device=a.device)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=a.device) if with_bf16 else None
    ws = gemm_workspace(M, N, K, device=a.device)
    fp8_gemm_dense_quant_out(a, sa, b, sb, q, s, c, pow2, ws, stream)
    return (q, s, c) if with_bf16 else (q, s)


def fp8_gemm_grouped_contig_out(a, sa, b, sb, m_indices, c, stream=None):
    M_total, K = a.shape
    E, N, _ = b.shape
    _check(lib.fp8_gemm_grouped_contig(_ptr(_as_u8(a)), _ptr(sa), _ptr(_as_u8(b)), _ptr(sb), _ptr(m_indices),
                                       _ptr(c), _dtype_code(c), M_total, N, K, E, _stream(stream)))
    return c


def fp8_gemm_grouped_contig(a, sa, b, sb, m_indices, out_dtype=torch.bfloat16, stream=None):
    """Grouped-contiguous MoE GEMM; padding rows (m_indices == -1) of C are left unwritten."""
    c = torch.empty((a.shape[0], b.shape[1]), dtype=out_dtype, device=a.device)
    return fp8_gemm_grouped_contig_out(a, sa, b, sb, m_indices, c, stream)


def fp8_gemm_grouped_masked_out(a, sa, b, sb, masked_m, c, b_scale_kind=SCALE_BLOCK128, mask_dim=MASK_ROWS,
                                accumulate=False, expected_m=0, stream=None):
    E, M_max, K = a.shape
    N = b.shape[1]
    _check(lib.fp8_gemm_grouped_masked(_ptr(_as_u8(a)), _ptr(sa), _ptr(_as_u8(b)), _ptr(sb), int(b_scale_kind),
                                       _ptr(masked_m), int(mask_dim), _ptr(c), _dtype_code(c),
                                       int(bool(accumulate)), E, M_max, N, K, int(expected_m), _stream(stream)))
    return c


def fp8_gemm_grouped_masked(a, sa, b, sb, masked_m, out_dtype=torch.bfloat16, b_scale_kind=SCALE_BLOCK128,
                            mask_dim=MASK_ROWS, expected_m=0, stream=None):
    """Grouped-masked MoE GEMM (rows >= masked_m[e] of C[e] unwritten in MASK_ROWS mode)."""
    E, M_max, _ = a.shape
    c = torch.empty((E, M_max, b.shape[1]), dtype=out_dtype, device=a.device)
    return fp8_gemm_grouped_masked_out(a, sa, b, sb, masked_m, c, b_scale_kind, mask_dim, False, expected_m,
                                       stream)


# ---------------------------------------------------------------- studies
def study_mma_accumulation(a, b, interval, stream=None):
    """D[128, N] = a[128, K] b[N, K]^T on unscaled E4M3 codes (uint8), the
    tensor-core accumulator restarted every `interval` K (see fp8fg.h)."""
    assert a.shape[0] == 128 and a.shape[1] == b.shape[1]
    d = torch.empty((128, b.shape[0]), dtype=torch.float32, device=a.device)
    _check(lib.fp8fg_study_mma_accumulation(_ptr(_as_u8(a)), _ptr(_as_u8(b)), _ptr(d), b.shape[0], a.shape[1],
                                            int(interval), _stream(stream)))
    return d


__all__ = [
    "lib", "LIB_PATH", "Fp8fgError", "scale_ld", "version", "check", "debug_set", "set_split_policy",
    "SPLIT_AUTO", "SPLIT_STREAM", "SPLIT_CLUSTER",
    "fp8_quant_1x128", "fp8_quant_1x128_out", "fp8_quant_128x128", "fp8_quant_128x128_out",
    "fp8_requant_128x1", "fp8_requant_128x1_out", "gemm_workspace_size", "gemm_workspace",
    "fp8_gemm_dense", "fp8_gemm_dense_out", "fp8_gemm_dense_quant", "fp8_gemm_dense_quant_out",
    "fp8_gemm_dgrad", "fp8_gemm_dgrad_out",
    "fp8_gemm_grouped_contig", "fp8_gemm_grouped_contig_out",
    "fp8_gemm_grouped_masked", "fp8_gemm_grouped_masked_out", "study_mma_accumulation",
]
