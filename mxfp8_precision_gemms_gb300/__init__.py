"""Python binding of the GB300 MXFP8 / per-tensor FP8 library (libmxfp8.so).

Argument marshalling only: every step of quantization and GEMM runs in the
library's CUDA kernels.  PyTorch supplies device memory (outputs are
allocated with ``torch.empty`` when not passed in) and the current stream.
The function names match the C ABI in ``include/mxfp8.h``.  There is no CPU
fallback: calling any op without the built library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxfp8.so")

MXFP8_OK = 0
MXFP8_ERR_INVALID_ARG = 1
MXFP8_ERR_UNSUPPORTED_SHAPE = 2
MXFP8_ERR_MISALIGNED = 3
MXFP8_ERR_CUDA = 4
MXFP8_ERR_DEVICE_CHECK = 5
MXFP8_ERR_TIMEOUT = 6

MX_ROWWISE, MX_COLWISE, MX_SCALE_FLOOR = 1, 2, 4
FP8_E4M3, FP8_E5M2 = 0, 1
GEMM_MX, GEMM_TENSOR = 0, 1

_lock = threading.Lock()
_lib = None


class MXFP8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"mxfp8 status {status}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library with argument types set.  Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I32, I, U = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                 ctypes.c_int, ctypes.c_uint)
            st = ctypes.c_int
            sigs = {
                "mxfp8_scale_bytes": (ctypes.c_size_t, [I64, I64]),
                "mxfp8_grouped_scale_bytes": (ctypes.c_size_t, [I64, I64, I32]),
                "fp8_quantize_mx": (st, [P, I64, I64, I64, U, P, P, P, P, P]),
                "fp8_quantize_mx_grouped": (st, [P, I64, I64, I64, P, I32, U, P, P, P]),
                "fp8_quantize_tensor": (st, [P, I64, I, P, P, P, P, P]),
                "mxfp8_tensor_workspace_bytes": (ctypes.c_size_t, []),
                "fp8_quantize_tensor_batch": (st, [I32, P, P, I, P, P, P, P, P]),
                "fp8_quantize_mx_batch": (st, [I32, P, P, P, P, P, P, P, P, P, P]),
                "mxfp8_debug_swiglu_f32": (st, [P, P, I64, P, P]),
                "fp8_quantize_tensor_noalloc": (st, [P, I64, I, P, P, P, P]),
                "fp8_quantize_tensor_scaled": (st, [P, I64, I, P, P, P, P, P]),
                "fp8_quantize_tensor_delayed": (st, [P, I64, I, ctypes.c_float, P, I32, P, P, P, P, P, P]),
                "fp8_requantize_tensor": (st, [P, I64, I, P, P, I, P, P, P]),
                "fp8_dequantize_mx": (st, [P, P, I64, I64, P, I32, P, I64, P]),
                "fp8_swiglu_quantize_mx": (st, [P, I64, I64, I64, P, I32, U, P, P, P]),
                "fp8_route_weight_quantize_mx": (st, [P, I64, I64, P, P, I64, I64, P, I32, U, P, P, P]),
                "fp8_route_weight_quantize_mx_tokens": (st, [P, I64, I64, I32, P, P, I64, I64, P, I32, U, P, P, P]),
                "fp8_scaled_gemm": (st, [I, I, I, P, P, P, P, I64, I64, I64, P, I64, P]),
                "fp8_scaled_gemm_pair": (st, [I] + [I, I, P, P, P, P, I64, I64, I64, P, I64] * 2 + [P]),
                "fp8_grouped_gemm": (st, [P, P, P, P, P, I32, I64, I64, I64, P, I64, P]),
                "mxfp8_last_device_status": (st, [P]),
                "mxfp8_status_string": (ctypes.c_char_p, [st]),
                "mxfp8_last_error": (ctypes.c_char_p, []),
                "mxfp8_set_wait_limit_ns": (None, [ctypes.c_uint64]),
                "mxfp8_debug_inject_wait_timeout": (None, [I]),
            }
            for name, (res, args) in sigs.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(status: int) -> None:
    if status != MXFP8_OK:
        raise MXFP8Error(status, lib().mxfp8_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _need_cuda(*ts) -> None:
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors passed to the library must live on a CUDA device")


# ------------------------------------------------------------- sizes --

def mxfp8_scale_bytes(rows: int, k: int) -> int:
    return int(lib().mxfp8_scale_bytes(rows, k))


def mxfp8_grouped_scale_bytes(total_rows: int, k: int, groups: int) -> int:
    return int(lib().mxfp8_grouped_scale_bytes(total_rows, k, groups))


# -------------------------------------------------------- quantization --

def fp8_quantize_mx(x: torch.Tensor, flags: int = MX_ROWWISE, q_row=None, s_row=None,
                    q_col=None, s_col=None, stream=None) -> dict:
    """MXFP8-quantize a 2D BF16 tensor (row stride = x.stride(0)).

    Returns {"q_row", "s_row"} and/or {"q_col", "s_col"} as uint8 tensors."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    _need_cuda(x)
    rows, cols = x.shape
    dev = x.device
    out = {}
    if flags & MX_ROWWISE:
        q_row = q_row if q_row is not None else torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        s_row = s_row if s_row is not None else torch.empty(mxfp8_scale_bytes(rows, cols), dtype=torch.uint8, device=dev)
        out["q_row"], out["s_row"] = q_row, s_row
    if flags & MX_COLWISE:
        q_col = q_col if q_col is not None else torch.empty((cols, rows), dtype=torch.uint8, device=dev)
        s_col = s_col if s_col is not None else torch.empty(mxfp8_scale_bytes(cols, rows), dtype=torch.uint8, device=dev)
        out["q_col"], out["s_col"] = q_col, s_col
    _check(lib().fp8_quantize_mx(_ptr(x), rows, cols, x.stride(0), flags, _ptr(q_row), _ptr(s_row),
                                 _ptr(q_col), _ptr(s_col), _stream(stream)))
    return out


def fp8_quantize_mx_grouped(x: torch.Tensor, offsets: torch.Tensor, flags: int = 0, q=None, s=None,
                            stream=None):
    """Rowwise MXFP8 quantization of expert-sorted rows; offsets: int32 device tensor (G+1)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert offsets.dtype == torch.int32
    _need_cuda(x, offsets)
    rows, cols = x.shape
    groups = offsets.numel() - 1
    q = q if q is not None else torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty(max(1, mxfp8_grouped_scale_bytes(rows, cols, groups)), dtype=torch.uint8,
                        device=x.device)
    _check(lib().fp8_quantize_mx_grouped(_ptr(x), rows, cols, x.stride(0), _ptr(offsets), groups,
                                         flags, _ptr(q), _ptr(s), _stream(stream)))
    return q, s


def fp8_quantize_tensor(x: torch.Tensor, fmt: int = FP8_E4M3, q=None, amax=None, scale=None,
                        workspace=None, stream=None):
    """Per-tensor FP8 quantization; returns (q uint8, amax fp32[1], scale fp32[1]).

    ``workspace``: None for the two-kernel path, or a device uint8 tensor of
    ``mxfp8_tensor_workspace_bytes()`` bytes for the single-launch path."""
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    _need_cuda(x, workspace)
    q = q if q is not None else torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    amax = amax if amax is not None else torch.empty(1, dtype=torch.float32, device=x.device)
    scale = scale if scale is not None else torch.empty(1, dtype=torch.float32, device=x.device)
    _check(lib().fp8_quantize_tensor(_ptr(x), x.numel(), fmt, _ptr(amax), _ptr(scale), _ptr(q),
                                     _ptr(workspace), _stream(stream)))
    return q, amax, scale


def fp8_quantize_tensor_scaled(x: torch.Tensor, scale: torch.Tensor, fmt: int = FP8_E4M3, q=None,
                               amax=None, sat_count=None, stream=None):
    """Cast with a device scale: returns (q, amax fp32[1], sat_count int64[1])."""
    assert x.dtype == torch.bfloat16 and x.is_contiguous() and scale.dtype == torch.float32
    _need_cuda(x, scale)
    q = q if q is not None else torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    amax = amax if amax is not None else torch.empty(1, dtype=torch.float32, device=x.device)
    sat_count = sat_count if sat_count is not None else torch.empty(1, dtype=torch.int64, device=x.device)
    _check(lib().fp8_quantize_tensor_scaled(_ptr(x), x.numel(), fmt, _ptr(scale), _ptr(q), _ptr(amax),
                                            _ptr(sat_count), _stream(stream)))
    return q, amax, sat_count


def fp8_quantize_tensor_delayed(x: torch.Tensor, history: torch.Tensor, pos: torch.Tensor,
                                fmt: int = FP8_E4M3, margin: float = 1.0, q=None, scale=None,
                                amax=None, sat_count=None, stream=None):
    """One delayed-scaling cast; history (fp32) and pos (int32[1]) are updated
    in place.  Returns (q, scale, amax, sat_count) as device tensors."""
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    assert history.dtype == torch.float32 and pos.dtype == torch.int32
    _need_cuda(x, history, pos)
    dev = x.device
    q = q if q is not None else torch.empty(x.shape, dtype=torch.uint8, device=dev)
    scale = scale if scale is not None else torch.empty(1, dtype=torch.float32, device=dev)
    amax = amax if amax is not None else torch.empty(1, dtype=torch.float32, device=dev)
    sat_count = sat_count if sat_count is not None else torch.empty(1, dtype=torch.int64, device=dev)
    _check(lib().fp8_quantize_tensor_delayed(_ptr(x), x.numel(), fmt, margin, _ptr(history),
                                             history.numel(), _ptr(pos), _ptr(scale), _ptr(q), _ptr(amax),
                                             _ptr(sat_count), _stream(stream)))
    return q, scale, amax, sat_count


def fp8_requantize_tensor(q: torch.Tensor, scale_in: torch.Tensor, scale_out: torch.Tensor,
                          fmt_in: int = FP8_E4M3, fmt_out: int = FP8_E4M3, out=None, sat_count=None,
                          stream=None):
    """Payload rescaled from scale_in to scale_out: returns (q_out, sat_count)."""
    assert q.dtype == torch.uint8 and q.is_contiguous()
    _need_cuda(q, scale_in, scale_out)
    out = out if out is not None else torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    sat_count = sat_count if sat_count is not None else torch.empty(1, dtype=torch.int64, device=q.device)
    _check(lib().fp8_requantize_tensor(_ptr(q), q.numel(), fmt_in, _ptr(scale_in), _ptr(scale_out), fmt_out,
                                       _ptr(out), _ptr(sat_count), _stream(stream)))
    return out, sat_count


def mxfp8_debug_swiglu_f32(g: torch.Tensor, u: torch.Tensor, stream=None) -> torch.Tensor:
    """Test hook: the SwiGLU fast path's fp32 g sigma(g) u per element."""
    assert g.dtype == torch.bfloat16 and u.dtype == torch.bfloat16 and g.shape == u.shape
    assert g.is_contiguous() and u.is_contiguous()
    _need_cuda(g, u)
    y = torch.empty(g.shape, dtype=torch.float32, device=g.device)
    _check(lib().mxfp8_debug_swiglu_f32(_ptr(g), _ptr(u), g.numel(), _ptr(y), _stream(stream)))
    return y


def fp8_quantize_mx_batch(xs, flags=MX_ROWWISE, outs=None, stream=None):
    """fp8_quantize_mx for several 2D BF16 tensors with as few launches as
    possible.  ``flags``: one value for all tensors or a list (one per
    tensor).  Returns a list of dicts like fp8_quantize_mx's; ``outs`` may
    supply them (the keys the flags need)."""
    count = len(xs)
    fl = [int(flags)] * count if isinstance(flags, int) else [int(f) for f in flags]
    assert len(fl) == count
    for x in xs:
        assert x.dtype == torch.bfloat16 and x.dim() == 2 and (x.numel() == 0 or x.stride(1) == 1)
    _need_cuda(*xs)
    dev = xs[0].device
    if outs is None:
        outs = []
        for x, f in zip(xs, fl):
            r, c = x.shape
            o = {}
            if f & MX_ROWWISE:
                o["q_row"] = torch.empty((r, c), dtype=torch.uint8, device=dev)
                o["s_row"] = torch.empty(mxfp8_scale_bytes(r, c), dtype=torch.uint8, device=dev)
            if f & MX_COLWISE:
                o["q_col"] = torch.empty((c, r), dtype=torch.uint8, device=dev)
                o["s_col"] = torch.empty(mxfp8_scale_bytes(c, r), dtype=torch.uint8, device=dev)
            outs.append(o)
    ptr = lambda o, k: o[k].data_ptr() if k in o else None
    keep = [(ctypes.c_void_p * count)(*[x.data_ptr() for x in xs]),
            (ctypes.c_int64 * count)(*[x.shape[0] for x in xs]),
            (ctypes.c_int64 * count)(*[x.shape[1] for x in xs]),
            (ctypes.c_int64 * count)(*[max(x.stride(0), x.shape[1]) for x in xs]),
            (ctypes.c_uint * count)(*fl)]
    keep += [(ctypes.c_void_p * count)(*[ptr(o, k) for o in outs]) for k in ("q_row", "s_row", "q_col", "s_col")]
    args = [ctypes.cast(a, ctypes.c_void_p) for a in keep]
    _check(lib().fp8_quantize_mx_batch(count, *args, _stream(stream)))
    return outs


def fp8_quantize_tensor_batch(xs, fmt: int = FP8_E4M3, workspace=None, qs=None, amax=None, scale=None,
                              stream=None):
    """Per-tensor FP8 quantization of several BF16 tensors in one launch.

    Returns (list of q, amax fp32[count], scale fp32[count]).  ``workspace``:
    a device uint8 tensor of ``mxfp8_tensor_workspace_bytes()`` bytes."""
    count = len(xs)
    dev = xs[0].device
    for x in xs:
        assert x.dtype == torch.bfloat16 and x.is_contiguous()
    _need_cuda(*xs, workspace)
    qs = qs if qs is not None else [torch.empty(x.shape, dtype=torch.uint8, device=dev) for x in xs]
    amax = amax if amax is not None else torch.empty(count, dtype=torch.float32, device=dev)
    scale = scale if scale is not None else torch.empty(count, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(mxfp8_tensor_workspace_bytes(), dtype=torch.uint8, device=dev)
    xp = (ctypes.c_void_p * count)(*[x.data_ptr() for x in xs])
    qp = (ctypes.c_void_p * count)(*[q.data_ptr() for q in qs])
    ns = (ctypes.c_int64 * count)(*[x.numel() for x in xs])
    _check(lib().fp8_quantize_tensor_batch(count, ctypes.cast(xp, ctypes.c_void_p), ctypes.cast(ns, ctypes.c_void_p),
                                           fmt, _ptr(amax), _ptr(scale), ctypes.cast(qp, ctypes.c_void_p),
                                           _ptr(workspace), _stream(stream)))
    return qs, amax, scale


def mxfp8_tensor_workspace_bytes() -> int:
    return int(lib().mxfp8_tensor_workspace_bytes())


# ------------------------------------------- routed-path conversions --

def _scales_for(rows: int, cols: int, offsets, device) -> torch.Tensor:
    if offsets is None:
        n = mxfp8_scale_bytes(rows, cols)
    else:
        n = mxfp8_grouped_scale_bytes(rows, cols, offsets.numel() - 1)
    return torch.empty(max(1, n), dtype=torch.uint8, device=device)


def _groups(offsets) -> int:
    if offsets is None:
        return 0
    assert offsets.dtype == torch.int32
    return offsets.numel() - 1


def fp8_dequantize_mx(q: torch.Tensor, s: torch.Tensor, offsets=None, out=None,
                      stream=None) -> torch.Tensor:
    """BF16 s * q of a rowwise MX operand (q: rows x cols uint8); offsets: the
    int32 group offsets of a group-padded scale array, or None."""
    assert q.dtype == torch.uint8 and q.dim() == 2 and q.is_contiguous()
    _need_cuda(q, s, offsets)
    rows, cols = q.shape
    out = out if out is not None else torch.empty((rows, cols), dtype=torch.bfloat16, device=q.device)
    assert out.dtype == torch.bfloat16 and out.stride(1) == 1
    _check(lib().fp8_dequantize_mx(_ptr(q), _ptr(s), rows, cols, _ptr(offsets), _groups(offsets),
                                   _ptr(out), out.stride(0), _stream(stream)))
    return out


def fp8_swiglu_quantize_mx(h: torch.Tensor, offsets=None, flags: int = 0, q=None, s=None,
                           stream=None):
    """Rowwise MXFP8 of SwiGLU(h): h is rows x 2f BF16 (gate | up); returns (q, s)."""
    assert h.dtype == torch.bfloat16 and h.dim() == 2 and h.stride(1) == 1
    _need_cuda(h, offsets)
    rows, width = h.shape
    f = width // 2
    q = q if q is not None else torch.empty((rows, f), dtype=torch.uint8, device=h.device)
    s = s if s is not None else _scales_for(rows, f, offsets, h.device)
    _check(lib().fp8_swiglu_quantize_mx(_ptr(h), rows, f, h.stride(0), _ptr(offsets), _groups(offsets),
                                        flags, _ptr(q), _ptr(s), _stream(stream)))
    return q, s


def fp8_route_weight_quantize_mx(dy: torch.Tensor, row_token: torch.Tensor, row_weight: torch.Tensor,
                                 offsets=None, flags: int = 0, q=None, s=None, stream=None):
    """Rowwise MXFP8 of w_i * dy[row_token[i]] for every dispatched row i;
    row_token int32, row_weight fp32 (device).  Returns (q, s)."""
    assert dy.dtype == torch.bfloat16 and dy.dim() == 2 and dy.stride(1) == 1
    assert row_token.dtype == torch.int32 and row_weight.dtype == torch.float32
    assert row_token.numel() == row_weight.numel()
    _need_cuda(dy, row_token, row_weight, offsets)
    tokens, cols = dy.shape
    rows = row_token.numel()
    q = q if q is not None else torch.empty((rows, cols), dtype=torch.uint8, device=dy.device)
    s = s if s is not None else _scales_for(rows, cols, offsets, dy.device)
    _check(lib().fp8_route_weight_quantize_mx(_ptr(dy), tokens, dy.stride(0), _ptr(row_token),
                                              _ptr(row_weight), rows, cols, _ptr(offsets),
                                              _groups(offsets), flags, _ptr(q), _ptr(s),
                                              _stream(stream)))
    return q, s


def fp8_route_weight_quantize_mx_tokens(dy: torch.Tensor, token_rows: torch.Tensor,
                                        token_weights: torch.Tensor, rows: int, offsets=None,
                                        flags: int = 0, q=None, s=None, stream=None):
    """The same conversion with the routing given per token: token_rows
    (tokens x k int32 dispatched rows, -1 for none) and token_weights
    (tokens x k fp32); each dY row is read once.  Returns (q, s)."""
    assert dy.dtype == torch.bfloat16 and dy.dim() == 2 and dy.stride(1) == 1
    assert token_rows.dtype == torch.int32 and token_weights.dtype == torch.float32
    assert token_rows.shape == token_weights.shape and token_rows.dim() == 2
    assert token_rows.is_contiguous() and token_weights.is_contiguous()
    _need_cuda(dy, token_rows, token_weights, offsets)
    tokens, cols = dy.shape
    assert token_rows.shape[0] == tokens
    k = token_rows.shape[1]
    q = q if q is not None else torch.empty((rows, cols), dtype=torch.uint8, device=dy.device)
    s = s if s is not None else _scales_for(rows, cols, offsets, dy.device)
    _check(lib().fp8_route_weight_quantize_mx_tokens(_ptr(dy), tokens, dy.stride(0), k,
                                                     _ptr(token_rows), _ptr(token_weights), rows,
                                                     cols, _ptr(offsets), _groups(offsets), flags,
                                                     _ptr(q), _ptr(s), _stream(stream)))
    return q, s


# --------------------------------------------------------------- GEMMs --

def fp8_scaled_gemm(mode: int, a: torch.Tensor, a_scale: torch.Tensor, b: torch.Tensor,
                    b_scale: torch.Tensor, c=None, a_fmt: int = FP8_E4M3, b_fmt: int = FP8_E4M3,
                    stream=None) -> torch.Tensor:
    """C = A . B^T (A: M x K, B: N x K uint8 payloads) -> BF16 M x N."""
    assert a.dtype == torch.uint8 and b.dtype == torch.uint8 and a.dim() == 2 and b.dim() == 2
    _need_cuda(a, b, a_scale, b_scale)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape[1] == K and a.is_contiguous() and b.is_contiguous()
    c = c if c is not None else torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _check(lib().fp8_scaled_gemm(mode, a_fmt, b_fmt, _ptr(a), _ptr(a_scale), _ptr(b), _ptr(b_scale),
                                 M, N, K, _ptr(c), c.stride(0), _stream(stream)))
    return c


def fp8_scaled_gemm_pair(mode: int, first, second, stream=None):
    """Two independent GEMMs of one mode in one launch.  first / second are
    dicts with a, a_scale, b, b_scale (as fp8_scaled_gemm) and optionally c,
    a_fmt, b_fmt; returns (C0, C1)."""
    args, outs = [], []
    for g in (first, second):
        a, b = g["a"], g["b"]
        assert a.dtype == torch.uint8 and b.dtype == torch.uint8 and a.dim() == 2 and b.dim() == 2
        _need_cuda(a, b, g["a_scale"], g["b_scale"])
        M, K = a.shape
        N = b.shape[0]
        assert b.shape[1] == K and a.is_contiguous() and b.is_contiguous()
        c = g.get("c")
        c = c if c is not None else torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
        args += [g.get("a_fmt", FP8_E4M3), g.get("b_fmt", FP8_E4M3), _ptr(a), _ptr(g["a_scale"]),
                 _ptr(b), _ptr(g["b_scale"]), M, N, K, _ptr(c), c.stride(0)]
        outs.append(c)
    _check(lib().fp8_scaled_gemm_pair(mode, *args, _stream(stream)))
    return outs[0], outs[1]


def fp8_grouped_gemm(a: torch.Tensor, a_scale: torch.Tensor, b: torch.Tensor, b_scale: torch.Tensor,
                     offsets: torch.Tensor, c=None, stream=None) -> torch.Tensor:
    """Per-expert MX GEMM: a (total_rows x K), b (G x N x K), offsets int32 (G+1)."""
    assert a.dtype == torch.uint8 and b.dtype == torch.uint8 and b.dim() == 3
    _need_cuda(a, a_scale, b, b_scale, offsets)
    total, K = a.shape
    G, N, Kb = b.shape
    assert Kb == K and offsets.numel() == G + 1 and offsets.dtype == torch.int32
    c = c if c is not None else torch.empty((total, N), dtype=torch.bfloat16, device=a.device)
    _check(lib().fp8_grouped_gemm(_ptr(a), _ptr(a_scale), _ptr(b), _ptr(b_scale), _ptr(offsets), G,
                                  total, N, K, _ptr(c), c.stride(0), _stream(stream)))
    return c


# -------------------------------------------------------------- status --

def mxfp8_last_device_status(stream=None) -> int:
    """Synchronize the stream and return (and clear) the device status word."""
    return int(lib().mxfp8_last_device_status(_stream(stream)))


def mxfp8_status_string(status: int) -> str:
    return lib().mxfp8_status_string(status).decode()


def mxfp8_last_error() -> str:
    return lib().mxfp8_last_error().decode()


def mxfp8_set_wait_limit_ns(ns: int) -> None:
    lib().mxfp8_set_wait_limit_ns(ns)


def mxfp8_debug_inject_wait_timeout(enable: bool) -> None:
    lib().mxfp8_debug_inject_wait_timeout(1 if enable else 0)
