"""FP64 CPU oracle for MXFP8 / per-tensor FP8 quantization and scaled GEMMs.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports this package.  Only ``tests/``, the smoke check in
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.

The arithmetic lives in ``oracle.c`` (plain C, FP64, scalar); this module
compiles it on first use with gcc and exposes numpy-level wrappers.  Each
wrapper names the passage it follows; the C file carries the full list of
sources and of the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

E4M3, E5M2 = 0, 1
ROWWISE, COLWISE, SCALE_FLOOR = 1, 2, 4


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    stale = force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I32 = ctypes.c_int32
            I = ctypes.c_int
            sig = {
                "orc_bf16_decode_array": (None, [P, I64, P]),
                "orc_fp8_decode_array": (None, [P, I64, I, P]),
                "orc_fp8_encode_array": (None, [P, I64, I, P]),
                "orc_bf16_round_array": (None, [P, I64, P]),
                "orc_e8m0_array": (None, [P, I64, I, P]),
                "orc_scale_bytes": (I64, [I64, I64]),
                "orc_swizzle_offset": (I64, [I64, I64, I64]),
                "orc_quantize_mx": (None, [P, I64, I64, I64, I, P, P, P, P]),
                "orc_quantize_mx_grouped": (None, [P, I64, I64, P, I32, I, P, P, I64]),
                "orc_quantize_tensor": (None, [P, I64, I, P, P, P]),
                "orc_gemm_mx_rows": (None, [P, P, P, P, I64, I64, I64, P, I64, P]),
                "orc_gemm_tensor_rows": (None, [P, I, ctypes.c_float, P, I, ctypes.c_float,
                                                I64, I64, I64, P, I64, P]),
                "orc_gemm_grouped_rows": (None, [P, P, P, P, P, I32, I64, I64, P, I64, P]),
                "orc_num_threads": (I, []),
                "orc_dequantize_mx": (None, [P, P, I64, I64, P, I64]),
                "orc_quantize_tensor_scaled": (None, [P, I64, I, ctypes.c_float, P, P, P]),
                "orc_delayed_scale": (ctypes.c_float, [P, I32, I, ctypes.c_float]),
                "orc_quantize_tensor_delayed": (None, [P, I64, I, ctypes.c_float, P, I32, P, P, P, P, P]),
                "orc_requantize_tensor": (None, [P, I64, I, ctypes.c_float, ctypes.c_float, I, P, P]),
                "orc_dequantize_mx_grouped": (None, [P, P, P, I32, I64, P, I64]),
                "orc_swiglu": (None, [P, I64, I64, I64, P]),
                "orc_swiglu_bf16": (None, [P, I64, I64, I64, P]),
                "orc_route_weight": (None, [P, I64, I64, P, P, I64, I64, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous arrays"
    return ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------- codecs --

def bf16_decode(bits) -> np.ndarray:
    """BF16 bit patterns -> exact float64 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().orc_bf16_decode_array(_p(b), b.size, _p(out))
    return out


def fp8_decode(codes, fmt: int = E4M3) -> np.ndarray:
    """E4M3 / E5M2 codes -> exact float64 values."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().orc_fp8_decode_array(_p(c), c.size, fmt, _p(out))
    return out


def fp8_encode(values, fmt: int = E4M3) -> np.ndarray:
    """Saturating round-to-nearest-even encode of float64 values."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    _load().orc_fp8_encode_array(_p(v), v.size, fmt, _p(out))
    return out


def bf16_round(values) -> np.ndarray:
    """Round float64 values to BF16 bit patterns (RNE)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().orc_bf16_round_array(_p(v), v.size, _p(out))
    return out


def e8m0_scale_byte(amax, floor: bool = False) -> np.ndarray:
    """E8M0 byte of the block scale for each block maximum (rceil or floor)."""
    a = np.ascontiguousarray(amax, dtype=np.float64)
    out = np.empty(a.shape, np.int32)
    _load().orc_e8m0_array(_p(a), a.size, 1 if floor else 0, _p(out))
    return out


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().orc_num_threads())


def scale_bytes(rows: int, k: int) -> int:
    return int(_load().orc_scale_bytes(rows, k))


def grouped_scale_bytes(offsets, k: int) -> int:
    off = np.asarray(offsets, dtype=np.int64)
    padded = int(sum((int(off[g + 1] - off[g]) + 127) // 128 * 128 for g in range(len(off) - 1)))
    return padded // 128 * ((k + 127) // 128) * 512


def swizzle_offset(r: int, j: int, k: int) -> int:
    return int(_load().orc_swizzle_offset(r, j, k))


# ---------------------------------------------------------- quantization --

def quantize_mx(x_bits: np.ndarray, flags: int = ROWWISE) -> dict:
    """MXFP8 quantization of a rows x cols BF16 matrix (bit patterns).

    Returns q_row (rows x cols), s_row (swizzled bytes), q_col (cols x rows)
    and s_col, for the orientations selected by ``flags``."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    out = {}
    q_row = np.zeros((rows, cols), np.uint8) if flags & ROWWISE else np.zeros(1, np.uint8)
    s_row = np.zeros(scale_bytes(rows, cols), np.uint8) if flags & ROWWISE else np.zeros(1, np.uint8)
    q_col = np.zeros((cols, rows), np.uint8) if flags & COLWISE else np.zeros(1, np.uint8)
    s_col = np.zeros(scale_bytes(cols, rows), np.uint8) if flags & COLWISE else np.zeros(1, np.uint8)
    _load().orc_quantize_mx(_p(x), rows, cols, cols, flags, _p(q_row), _p(s_row), _p(q_col), _p(s_col))
    if flags & ROWWISE:
        out["q_row"], out["s_row"] = q_row, s_row
    if flags & COLWISE:
        out["q_col"], out["s_col"] = q_col, s_col
    return out


def dequantize_mx(q, s) -> np.ndarray:
    """BF16 bit patterns of s * q for a rowwise MX operand (q: rows x cols)."""
    q = np.ascontiguousarray(q, np.uint8)
    s = np.ascontiguousarray(s, np.uint8)
    rows, cols = q.shape
    out = np.zeros((rows, cols), np.uint16)
    _load().orc_dequantize_mx(_p(q), _p(s), rows, cols, _p(out), cols)
    return out


def dequantize_mx_grouped(q, s, offsets) -> np.ndarray:
    """BF16 bit patterns of s * q for a group-padded rowwise operand."""
    q = np.ascontiguousarray(q, np.uint8)
    s = np.ascontiguousarray(s, np.uint8)
    off = np.ascontiguousarray(offsets, np.int32)
    rows, cols = q.shape
    assert int(off[-1]) == rows
    out = np.zeros((rows, cols), np.uint16)
    _load().orc_dequantize_mx_grouped(_p(q), _p(s), _p(off), off.size - 1, cols, _p(out), cols)
    return out


def swiglu(h, f: int | None = None) -> np.ndarray:
    """FP64 g * sigma(g) * u of BF16 bits h (rows x 2f: gate | up)."""
    h = np.ascontiguousarray(h, np.uint16)
    rows, width = h.shape
    f = width // 2 if f is None else f
    out = np.zeros((rows, f), np.float64)
    _load().orc_swiglu(_p(h), rows, f, width, _p(out))
    return out


def swiglu_bf16(h, f: int | None = None) -> np.ndarray:
    """BF16 bits of g * sigma(g) * u correctly rounded (never a tie: the exact
    value is irrational), h as in swiglu.  Raises if FP64 could not decide the
    rounding side of some value (never observed)."""
    h = np.ascontiguousarray(h, np.uint16)
    rows, width = h.shape
    f = width // 2 if f is None else f
    out = np.zeros((rows, f), np.uint16)
    lib = _load()
    before = ctypes.c_int64.in_dll(lib, "orc_swiglu_undecided").value
    lib.orc_swiglu_bf16(_p(h), rows, f, width, _p(out))
    after = ctypes.c_int64.in_dll(lib, "orc_swiglu_undecided").value
    if after != before:
        raise ArithmeticError(f"{after - before} SwiGLU values undecided in FP64")
    return out


def route_weight(dy, row_token, row_weight) -> np.ndarray:
    """BF16 bits of w_i * dy[tok_i], rounded once, for every dispatched row."""
    dy = np.ascontiguousarray(dy, np.uint16)
    tok = np.ascontiguousarray(row_token, np.int32)
    w = np.ascontiguousarray(row_weight, np.float32)
    tokens, cols = dy.shape
    out = np.zeros((tok.size, cols), np.uint16)
    _load().orc_route_weight(_p(dy), tokens, cols, _p(tok), _p(w), tok.size, cols, _p(out))
    return out


def quantize_mx_grouped(x_bits: np.ndarray, offsets, flags: int = ROWWISE):
    """Grouped rowwise MXFP8 quantization; returns (q, s) with group g's scale
    rows starting at its padded row."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    rows, cols = x.shape
    assert off[-1] == rows
    nb = grouped_scale_bytes(off, cols)
    q = np.zeros((rows, cols), np.uint8)
    s = np.zeros(max(nb, 1), np.uint8)
    _load().orc_quantize_mx_grouped(_p(x), cols, cols, _p(off), len(off) - 1, flags, _p(q), _p(s), nb)
    return q, s[:nb]


def quantize_tensor(x_bits: np.ndarray, fmt: int = E4M3):
    """Per-tensor current-scaling FP8 quantization: (amax, scale, q)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.zeros(x.shape, np.uint8)
    amax = np.zeros(1, np.float32)
    scale = np.zeros(1, np.float32)
    _load().orc_quantize_tensor(_p(x), x.size, fmt, _p(amax), _p(scale), _p(q))
    return amax[0], scale[0], q


def quantize_tensor_scaled(x_bits, fmt: int, scale: float):
    """Cast with a given fp32 scale: (q, amax, saturated count)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.zeros(x.shape, np.uint8)
    amax = np.zeros(1, np.float32)
    sat = np.zeros(1, np.int64)
    _load().orc_quantize_tensor_scaled(_p(x), x.size, fmt, float(np.float32(scale)), _p(q),
                                       _p(amax), _p(sat))
    return q, amax[0], int(sat[0])


def delayed_scale(history, fmt: int = E4M3, margin: float = 1.0) -> np.float32:
    h = np.ascontiguousarray(history, np.float32)
    return np.float32(_load().orc_delayed_scale(_p(h), h.size, fmt, float(np.float32(margin))))


def quantize_tensor_delayed(x_bits, fmt: int, margin: float, history, pos: int):
    """One delayed-scaling cast.  Returns (q, scale, amax, sat, history', pos')."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    hist = np.array(history, np.float32)
    p = np.array([pos], np.int32)
    q = np.zeros(x.shape, np.uint8)
    scale = np.zeros(1, np.float32)
    amax = np.zeros(1, np.float32)
    sat = np.zeros(1, np.int64)
    _load().orc_quantize_tensor_delayed(_p(x), x.size, fmt, float(np.float32(margin)), _p(hist),
                                        hist.size, _p(p), _p(scale), _p(q), _p(amax), _p(sat))
    return q, scale[0], amax[0], int(sat[0]), hist, int(p[0])


def requantize_tensor(q_in, fmt_in: int, s_in: float, s_out: float, fmt_out: int):
    """FP8 payload rescaled from s_in to s_out: (q_out, saturated count)."""
    q = np.ascontiguousarray(q_in, np.uint8)
    out = np.zeros(q.shape, np.uint8)
    sat = np.zeros(1, np.int64)
    _load().orc_requantize_tensor(_p(q), q.size, fmt_in, float(np.float32(s_in)),
                                  float(np.float32(s_out)), fmt_out, _p(out), _p(sat))
    return out, int(sat[0])


# ------------------------------------------------------------------ GEMMs --

def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, r.size


def gemm_mx(qa, sa, qb, sb, rows=None) -> np.ndarray:
    """FP64 C = A B^T on MX-dequantized operands (both K-major)."""
    qa = np.ascontiguousarray(qa, np.uint8); qb = np.ascontiguousarray(qb, np.uint8)
    sa = np.ascontiguousarray(sa, np.uint8); sb = np.ascontiguousarray(sb, np.uint8)
    M, K = qa.shape
    N = qb.shape[0]
    r, nr = _rows_arg(rows, M)
    out = np.zeros((nr, N), np.float64)
    _load().orc_gemm_mx_rows(_p(qa), _p(sa), _p(qb), _p(sb), M, N, K,
                             None if r is None else _p(r), nr, _p(out))
    return out


def gemm_tensor(qa, fa, s_a, qb, fb, s_b, rows=None) -> np.ndarray:
    """FP64 C = (sum_k q_a q_b) / (s_a s_b) for per-tensor scaled operands."""
    qa = np.ascontiguousarray(qa, np.uint8); qb = np.ascontiguousarray(qb, np.uint8)
    M, K = qa.shape
    N = qb.shape[0]
    r, nr = _rows_arg(rows, M)
    out = np.zeros((nr, N), np.float64)
    _load().orc_gemm_tensor_rows(_p(qa), fa, float(s_a), _p(qb), fb, float(s_b), M, N, K,
                                 None if r is None else _p(r), nr, _p(out))
    return out


def gemm_grouped(qa, sa, qw, sw, offsets, rows=None) -> np.ndarray:
    """FP64 grouped GEMM: C rows listed in ``rows`` (ascending global row
    indices), or all total_rows x N when rows is None."""
    qa = np.ascontiguousarray(qa, np.uint8); sa = np.ascontiguousarray(sa, np.uint8)
    qw = np.ascontiguousarray(qw, np.uint8); sw = np.ascontiguousarray(sw, np.uint8)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    G, N, K = qw.shape
    total = int(off[-1])
    r = None
    if rows is not None:
        r = np.ascontiguousarray(np.sort(np.asarray(rows, dtype=np.int64)))
        assert r.size == 0 or (r[0] >= 0 and r[-1] < total)
    nr = total if r is None else r.size
    out = np.zeros((nr, N), np.float64)
    _load().orc_gemm_grouped_rows(_p(qa), _p(sa), _p(qw), _p(sw), _p(off), G, N, K,
                                  None if r is None else _p(r), nr, _p(out))
    return out
