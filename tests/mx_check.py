"""Comparison of a GPU MX quantization with the oracle's when the BF16 values
being quantized are only known to lie in a small set.

The fused SwiGLU quantizer forms g sigma(g) u in fp32 (error below 7.5 *
2^-24 relative: checked for every BF16 gate by the fast-path test, plus an
absolute 2^-149 where fp32 underflows) before the BF16 rounding.  Where the exact value lies within that distance of a BF16
rounding midpoint either neighbour is a correct result, so the check takes,
per element, the set {bf16(y - band), bf16(y + band)} around the oracle's
FP64 value y, band = 2^-19 |y| + 2^-140 (both bounds with margin).  Blocks
whose 32 values are all unambiguous must match the oracle's bytes exactly;
an ambiguous block's scale byte must lie between the E8M0 bytes of the
smallest and the largest admissible block maximum, and each of its payload
bytes must be the encoding, under the GPU's scale, of one admissible value.
"""
import numpy as np

import oracle

BAND_REL = 2.0 ** -19
BAND_ABS = 2.0 ** -140


def bf16_candidates(y: np.ndarray):
    """(nearest, low, high) BF16 bit patterns around FP64 values y."""
    c = oracle.bf16_round(y)
    band = np.abs(y) * BAND_REL + BAND_ABS
    lo = oracle.bf16_round(y - band)
    hi = oracle.bf16_round(y + band)
    exact = (y == 0) | ~np.isfinite(y)
    return c, np.where(exact, c, lo), np.where(exact, c, hi)


def padded_rows(rows: int, offsets=None) -> np.ndarray:
    """Scale row of every payload row (identity, or the group-padded row)."""
    if offsets is None:
        return np.arange(rows, dtype=np.int64)
    off = np.asarray(offsets, np.int64)
    counts = np.diff(off)
    starts = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])[:-1]
    g = np.repeat(np.arange(counts.size), counts)
    return starts[g] + (np.arange(rows) - off[g])


def scale_positions(prow: np.ndarray, cols: int) -> np.ndarray:
    """Byte of every logical scale (row, block) in the swizzled array."""
    nkc = (cols + 127) // 128
    j = np.arange(cols // 32)[None, :]
    r = prow[:, None]
    return ((r // 128) * nkc + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4


def check_set_quantization(q_gpu, s_gpu, lo, hi, q_exp, s_exp, offsets=None, floor=False):
    rows, cols = lo.shape
    kb = cols // 32
    pos = scale_positions(padded_rows(rows, offsets), cols)
    blk = (lo != hi).reshape(rows, kb, 32).any(-1)
    s_gpu = s_gpu[: s_exp.size]
    keep = np.ones(s_exp.size, bool)
    keep[pos[blk]] = False
    bad = np.nonzero(keep & (s_gpu != s_exp))[0]
    assert bad.size == 0, f"{bad.size} scale bytes differ, first at byte {bad[:4]}"
    same = ~np.repeat(blk, 32, axis=1)
    nq = int((q_gpu[same] != q_exp[same]).sum())
    assert nq == 0, f"{nq} payload bytes differ in unambiguous blocks"
    r, j = np.nonzero(blk)
    if r.size == 0:
        return 0
    lov = oracle.bf16_decode(lo.reshape(rows, kb, 32)[r, j])
    hiv = oracle.bf16_decode(hi.reshape(rows, kb, 32)[r, j])
    bmin = oracle.e8m0_scale_byte(np.minimum(np.abs(lov), np.abs(hiv)).max(-1), floor)
    bmax = oracle.e8m0_scale_byte(np.maximum(np.abs(lov), np.abs(hiv)).max(-1), floor)
    sg = s_gpu[pos[r, j]].astype(np.int32)
    assert np.all((bmin <= sg) & (sg <= bmax)), "ambiguous block scale out of range"
    sc = np.ldexp(1.0, sg - 127)[:, None]
    qg = q_gpu.reshape(rows, kb, 32)[r, j]
    ok = (qg == oracle.fp8_encode(lov / sc)) | (qg == oracle.fp8_encode(hiv / sc))
    assert ok.all(), f"{int((~ok).sum())} payload bytes of ambiguous blocks inadmissible"
    return int(r.size)
