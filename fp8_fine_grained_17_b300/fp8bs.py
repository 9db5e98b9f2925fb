"""Python binding of libfp8bs.so (ctypes): argument marshalling only.

Every function named ``fp8bs_*`` here forwards to the C entry point of the
same name with the tensors' device pointers and sizes; all work runs in the
library's CUDA kernels. PyTorch supplies device memory and streams only.
There is no CPU fallback: if the library is missing or a tensor is not on a
CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8bs.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fp8bs.h")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
OUT_F32, OUT_BF16 = 0, 1
TILE_AUTO, TILE_128x256, TILE_128x128, TILE_PAIR_256x256, TILE_PAIR_256x128 = 0, 1, 2, 3, 4
TILES = (TILE_128x256, TILE_128x128, TILE_PAIR_256x256, TILE_PAIR_256x128)
NORM_RMS, NORM_LAYER = 0, 1
NOALLOC_SCRATCH_BYTES = 12 << 20   # FP8BS_NOALLOC_SCRATCH_BYTES in include/fp8bs.h


class Fp8bsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m fp8_fine_grained_17_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, f32p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        st = ctypes.c_int
        L.fp8bs_quantize_act_1x128.argtypes = [vp, i64, i64, i64, vp, i64, f32p, vp]
        L.fp8bs_quantize_act_1x128.restype = st
        L.fp8bs_quantize_weight_128x128.argtypes = [vp, i64, i64, i64, vp, i64, f32p, vp]
        L.fp8bs_quantize_weight_128x128.restype = st
        L.fp8bs_quantize_act_1x128_pow2.argtypes = [vp, i64, i64, i64, vp, i64, f32p, vp]
        L.fp8bs_quantize_act_1x128_pow2.restype = st
        L.fp8bs_quantize_weight_128x128_pow2.argtypes = [vp, i64, i64, i64, vp, i64, f32p, vp]
        L.fp8bs_quantize_weight_128x128_pow2.restype = st
        L.fp8bs_gemm.argtypes = [vp, f32p, vp, f32p, vp, ctypes.c_int, i64, i64, i64, i64, vp]
        L.fp8bs_gemm.restype = st
        L.fp8bs_grouped_gemm.argtypes = [vp, f32p, vp, i32, i64, vp, f32p, vp, ctypes.c_int,
                                         i64, i64, i64, vp]
        L.fp8bs_grouped_gemm.restype = st
        L.fp8bs_gemm_tiled.argtypes = [vp, f32p, vp, f32p, vp, ctypes.c_int, i64, i64, i64, i64,
                                       ctypes.c_int, vp]
        L.fp8bs_gemm_tiled.restype = st
        L.fp8bs_grouped_gemm_tiled.argtypes = [vp, f32p, vp, i32, i64, vp, f32p, vp, ctypes.c_int,
                                               i64, i64, i64, ctypes.c_int, vp]
        L.fp8bs_grouped_gemm_tiled.restype = st
        L.fp8bs_norm_quantize_act_1x128.argtypes = [vp, i64, i64, i64, vp, vp, ctypes.c_int,
                                                    ctypes.c_float, vp, i64, f32p, f32p, f32p, vp]
        L.fp8bs_norm_quantize_act_1x128.restype = st
        L.fp8bs_gemm_bf16_act.argtypes = [vp, i64, vp, f32p, vp, ctypes.c_int, i64, i64, i64, i64, vp]
        L.fp8bs_gemm_bf16_act.restype = st
        L.fp8bs_grouped_gemm_bf16_act.argtypes = [vp, i64, vp, i32, i64, vp, f32p, vp, ctypes.c_int,
                                                  i64, i64, i64, vp]
        L.fp8bs_grouped_gemm_bf16_act.restype = st
        L.fp8bs_quantize_act_and_weight.argtypes = [vp, i64, i64, i64, vp, i64, f32p, vp, i64, i64, i64,
                                                    vp, i64, f32p, vp]
        L.fp8bs_quantize_act_and_weight.restype = st
        L.fp8bs_status_string.argtypes = [ctypes.c_int]
        L.fp8bs_status_string.restype = ctypes.c_char_p
        L.fp8bs_last_device_error.argtypes = [vp]
        L.fp8bs_last_device_error.restype = st
        L.fp8bs_gemm_ws.argtypes = [vp, f32p, vp, f32p, vp, ctypes.c_int, i64, i64, i64, i64,
                                    ctypes.c_int, vp, ctypes.c_size_t, vp]
        L.fp8bs_gemm_ws.restype = st
        L.fp8bs_gemm_workspace_size.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
        L.fp8bs_gemm_workspace_size.restype = st
        L.fp8bs_gemm_noalloc.argtypes = [vp, f32p, vp, f32p, vp, ctypes.c_int, i64, i64, i64, i64,
                                         ctypes.c_int, vp]
        L.fp8bs_gemm_noalloc.restype = st
        L.fp8bs_test_inject_stall.argtypes = [i64, i64]
        L.fp8bs_test_inject_stall.restype = st
        _lib = L
    return _lib


def header_symbols() -> list[str]:
    """Names of the functions declared in include/fp8bs.h."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fp8bs_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return lib().fp8bs_status_string(int(status)).decode()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("fp8bs works on CUDA tensors only (no CPU path)")
    return t.data_ptr()


def _check(fn: str, status: int):
    if status != OK:
        raise Fp8bsError(fn, status)


def _row_stride(t: torch.Tensor) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    return t.stride(0)


def _u8(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


# ---------------------------------------------------------------- C entry points

def fp8bs_quantize_act_1x128(x: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, stream=None,
                             pow2: bool = False):
    """x bf16 [M, K] -> q e4m3/uint8 [M, K], scale fp32 [M, K/128] (contiguous).
    pow2: power-of-two scales (fp8bs_quantize_act_1x128_pow2)."""
    M, K = x.shape
    assert x.dtype == torch.bfloat16 and scale.dtype == torch.float32 and scale.is_contiguous()
    q8 = _u8(q)
    name = "fp8bs_quantize_act_1x128_pow2" if pow2 else "fp8bs_quantize_act_1x128"
    _check(name, getattr(lib(), name)(
        _ptr(x), M, K, _row_stride(x), _ptr(q8), _row_stride(q8), _ptr(scale), _stream(stream)))


def fp8bs_quantize_weight_128x128(w: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, stream=None,
                                  pow2: bool = False):
    """w bf16 [N, K] -> q [N, K], scale fp32 [ceil(N/128), K/128] (contiguous)."""
    N, K = w.shape
    assert w.dtype == torch.bfloat16 and scale.dtype == torch.float32 and scale.is_contiguous()
    q8 = _u8(q)
    name = "fp8bs_quantize_weight_128x128_pow2" if pow2 else "fp8bs_quantize_weight_128x128"
    _check(name, getattr(lib(), name)(
        _ptr(w), N, K, _row_stride(w), _ptr(q8), _row_stride(q8), _ptr(scale), _stream(stream)))


def fp8bs_norm_quantize_act_1x128(x: torch.Tensor, gamma: torch.Tensor, beta, kind: int, eps: float,
                                  q: torch.Tensor, scale: torch.Tensor, mean=None, rstd=None,
                                  stream=None):
    """RMSNorm/LayerNorm of x bf16 [M, K] (gamma, optional beta: bf16 [K]),
    rounded to bf16 and cast in 1x128 tiles: q [M, K], scale fp32 [M, K/128];
    optional fp32 [M] outputs mean (LayerNorm) and rstd."""
    M, K = x.shape
    assert x.dtype == torch.bfloat16 and gamma.dtype == torch.bfloat16 and gamma.is_contiguous()
    assert beta is None or (beta.dtype == torch.bfloat16 and beta.is_contiguous())
    assert scale.dtype == torch.float32 and scale.is_contiguous()
    for t in (mean, rstd):
        assert t is None or (t.dtype == torch.float32 and t.is_contiguous())
    q8 = _u8(q)
    _check("fp8bs_norm_quantize_act_1x128", lib().fp8bs_norm_quantize_act_1x128(
        _ptr(x), M, K, _row_stride(x), _ptr(gamma), _ptr(beta), int(kind), float(eps),
        _ptr(q8), _row_stride(q8), _ptr(scale), _ptr(mean), _ptr(rstd), _stream(stream)))


def fp8bs_quantize_act_and_weight(x, qx, sx, w, qw, sw, stream=None):
    """Both quantizers in one launch (same results as the two calls)."""
    M, K = x.shape
    N, Kw = w.shape
    assert x.dtype == torch.bfloat16 and w.dtype == torch.bfloat16
    assert sx.dtype == torch.float32 and sw.dtype == torch.float32
    assert sx.is_contiguous() and sw.is_contiguous()
    qx8, qw8 = _u8(qx), _u8(qw)
    _check("fp8bs_quantize_act_and_weight", lib().fp8bs_quantize_act_and_weight(
        _ptr(x), M, K, _row_stride(x), _ptr(qx8), _row_stride(qx8), _ptr(sx),
        _ptr(w), N, Kw, _row_stride(w), _ptr(qw8), _row_stride(qw8), _ptr(sw), _stream(stream)))


def _out_dtype(c: torch.Tensor) -> int:
    if c.dtype == torch.float32:
        return OUT_F32
    if c.dtype == torch.bfloat16:
        return OUT_BF16
    raise ValueError("output must be float32 or bfloat16")


def fp8bs_gemm(qa, sa, qw, sw, c, stream=None, tile=TILE_AUTO):
    """C[M, N] = dequant(qa, sa) @ dequant(qw, sw)^T into c (fp32 or bf16).
    A tile other than TILE_AUTO goes through fp8bs_gemm_tiled."""
    M, K = qa.shape
    N = qw.shape[0]
    for t in (qa, sa, qw, sw):
        assert t.is_contiguous()
    args = (_ptr(_u8(qa)), _ptr(sa), _ptr(_u8(qw)), _ptr(sw), _ptr(c), _out_dtype(c),
            M, N, K, _row_stride(c))
    if tile == TILE_AUTO:
        _check("fp8bs_gemm", lib().fp8bs_gemm(*args, _stream(stream)))
    else:
        _check("fp8bs_gemm_tiled", lib().fp8bs_gemm_tiled(*args, int(tile), _stream(stream)))


def fp8bs_gemm_workspace_size(M: int, N: int, K: int, tile=TILE_AUTO) -> int:
    """Workspace bytes fp8bs_gemm_ws needs on the current device (0: no split)."""
    n = ctypes.c_size_t(0)
    _check("fp8bs_gemm_workspace_size",
           lib().fp8bs_gemm_workspace_size(int(M), int(N), int(K), int(tile), ctypes.byref(n)))
    return int(n.value)


def fp8bs_gemm_ws(qa, sa, qw, sw, c, workspace, stream=None, tile=TILE_AUTO):
    """fp8bs_gemm with a workspace (uint8 CUDA tensor, zero-filled before its
    first use, or None) that lets the last wave of tiles be split along K."""
    M, K = qa.shape
    N = qw.shape[0]
    for t in (qa, sa, qw, sw):
        assert t.is_contiguous()
    ws = _ptr(workspace) if workspace is not None else None
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("fp8bs_gemm_ws", lib().fp8bs_gemm_ws(_ptr(_u8(qa)), _ptr(sa), _ptr(_u8(qw)), _ptr(sw), _ptr(c),
                                                _out_dtype(c), M, N, K, _row_stride(c), int(tile), ws,
                                                nbytes, _stream(stream)))


def fp8bs_gemm_noalloc(qa, sa, qw, sw, c, stream=None, tile=TILE_AUTO):
    """fp8bs_gemm_ws with the library's fixed device scratch as workspace:
    nothing is allocated by the call (for callers that cannot allocate)."""
    M, K = qa.shape
    N = qw.shape[0]
    for t in (qa, sa, qw, sw):
        assert t.is_contiguous()
    _check("fp8bs_gemm_noalloc", lib().fp8bs_gemm_noalloc(_ptr(_u8(qa)), _ptr(sa), _ptr(_u8(qw)), _ptr(sw),
                                                          _ptr(c), _out_dtype(c), M, N, K, _row_stride(c),
                                                          int(tile), _stream(stream)))


def fp8bs_grouped_gemm(qa, sa, expert_offsets, qw, sw, c, stream=None, tile=TILE_AUTO):
    """Per expert e: rows offsets[e]:offsets[e+1] of A times W_e^T."""
    total_M, K = qa.shape
    E, N, _ = qw.shape
    assert expert_offsets.dtype == torch.int32 and expert_offsets.numel() == E + 1
    for t in (qa, sa, qw, sw, expert_offsets):
        assert t.is_contiguous()
    args = (_ptr(_u8(qa)), _ptr(sa), _ptr(expert_offsets), E, total_M, _ptr(_u8(qw)), _ptr(sw),
            _ptr(c), _out_dtype(c), N, K, _row_stride(c))
    if tile == TILE_AUTO:
        _check("fp8bs_grouped_gemm", lib().fp8bs_grouped_gemm(*args, _stream(stream)))
    else:
        _check("fp8bs_grouped_gemm_tiled",
               lib().fp8bs_grouped_gemm_tiled(*args, int(tile), _stream(stream)))


def fp8bs_gemm_bf16_act(a, qw, sw, c, stream=None):
    """C = (1x128-quantized a) @ dequant(qw, sw)^T with the activation
    quantization inside the GEMM kernel; a is bf16 [M, K]."""
    M, K = a.shape
    N = qw.shape[0]
    assert a.dtype == torch.bfloat16
    for t in (qw, sw):
        assert t.is_contiguous()
    _check("fp8bs_gemm_bf16_act", lib().fp8bs_gemm_bf16_act(
        _ptr(a), _row_stride(a), _ptr(_u8(qw)), _ptr(sw), _ptr(c), _out_dtype(c), M, N, K,
        _row_stride(c), _stream(stream)))


def fp8bs_grouped_gemm_bf16_act(a, expert_offsets, qw, sw, c, stream=None):
    """Grouped GEMM with the activation quantization inside the kernel."""
    total_M, K = a.shape
    E, N, _ = qw.shape
    assert a.dtype == torch.bfloat16
    assert expert_offsets.dtype == torch.int32 and expert_offsets.numel() == E + 1
    for t in (qw, sw, expert_offsets):
        assert t.is_contiguous()
    _check("fp8bs_grouped_gemm_bf16_act", lib().fp8bs_grouped_gemm_bf16_act(
        _ptr(a), _row_stride(a), _ptr(expert_offsets), E, total_M, _ptr(_u8(qw)), _ptr(sw), _ptr(c),
        _out_dtype(c), N, K, _row_stride(c), _stream(stream)))


def fp8bs_last_device_error(stream=None) -> int:
    """Synchronizes the stream; returns (and clears) the device error status."""
    return lib().fp8bs_last_device_error(_stream(stream))


def fp8bs_test_inject_stall(chunk: int, wait_limit_ns: int = 0) -> None:
    """Failure-detection tests only: later GEMM launches leave out one chunk's
    copies in their first CTA and give up waiting after wait_limit_ns
    (chunk < 0 restores normal operation)."""
    _check("fp8bs_test_inject_stall", lib().fp8bs_test_inject_stall(int(chunk), int(wait_limit_ns)))


# ------------------------------------------------------ allocating conveniences

def quantize_act(x: torch.Tensor, stream=None, pow2: bool = False):
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((M, K // 128), dtype=torch.float32, device=x.device)
    fp8bs_quantize_act_1x128(x, q, s, stream, pow2)
    return q, s


def norm_quantize_act(x: torch.Tensor, gamma: torch.Tensor, beta=None, kind: int = NORM_RMS,
                      eps: float = 1e-6, stream=None):
    """Returns (q, scale, mean, rstd); mean is None for RMSNorm."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((M, K // 128), dtype=torch.float32, device=x.device)
    mean = torch.empty(M, dtype=torch.float32, device=x.device) if kind == NORM_LAYER else None
    rstd = torch.empty(M, dtype=torch.float32, device=x.device)
    fp8bs_norm_quantize_act_1x128(x, gamma, beta, kind, eps, q, s, mean, rstd, stream)
    return q, s, mean, rstd


def quantize_weight(w: torch.Tensor, stream=None, pow2: bool = False):
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=w.device)
    fp8bs_quantize_weight_128x128(w, q, s, stream, pow2)
    return q, s


def gemm(qa, sa, qw, sw, out_dtype=torch.bfloat16, stream=None, tile=TILE_AUTO):
    c = torch.empty((qa.shape[0], qw.shape[0]), dtype=out_dtype, device=qa.device)
    fp8bs_gemm(qa, sa, qw, sw, c, stream, tile)
    return c


def workspace(M: int, N: int, K: int, tile=TILE_AUTO, device=None):
    """A zero-filled workspace for fp8bs_gemm_ws (None when the shape needs none)."""
    n = fp8bs_gemm_workspace_size(M, N, K, tile)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda") if n else None


def gemm_ws(qa, sa, qw, sw, ws, out_dtype=torch.bfloat16, stream=None, tile=TILE_AUTO):
    c = torch.empty((qa.shape[0], qw.shape[0]), dtype=out_dtype, device=qa.device)
    fp8bs_gemm_ws(qa, sa, qw, sw, c, ws, stream, tile)
    return c


def gemm_bf16_act(a, qw, sw, out_dtype=torch.bfloat16, stream=None):
    c = torch.empty((a.shape[0], qw.shape[0]), dtype=out_dtype, device=a.device)
    fp8bs_gemm_bf16_act(a, qw, sw, c, stream)
    return c


def grouped_gemm_bf16_act(a, expert_offsets, qw, sw, out_dtype=torch.bfloat16, stream=None):
    c = torch.zeros((a.shape[0], qw.shape[1]), dtype=out_dtype, device=a.device)
    fp8bs_grouped_gemm_bf16_act(a, expert_offsets, qw, sw, c, stream)
    return c


def grouped_gemm(qa, sa, expert_offsets, qw, sw, out_dtype=torch.bfloat16, stream=None,
                 tile=TILE_AUTO):
    c = torch.zeros((qa.shape[0], qw.shape[1]), dtype=out_dtype, device=qa.device)
    fp8bs_grouped_gemm(qa, sa, expert_offsets, qw, sw, c, stream, tile)
    return c
