"""The float-float constants of the SwiGLU rounding resolver (ff_consts.h)
are the fp32 splits of ln 2, 1/6, 1/24 and e^(j/64) that their generator
computes with 60-digit decimal arithmetic; and each split sums back to its
constant within the float-float precision."""
import importlib.util
import os
import re
from decimal import Decimal, getcontext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mxfp8_precision_gemms_gb300", "csrc")


def _gen():
    spec = importlib.util.spec_from_file_location("gen_ff_consts", os.path.join(CSRC, "gen_ff_consts.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_header_is_generated_output():
    with open(os.path.join(CSRC, "ff_consts.h")) as f:
        assert f.read() == _gen().render()


def test_splits_sum_to_the_constants():
    getcontext().prec = 60
    text = open(os.path.join(CSRC, "ff_consts.h")).read()
    hexf = r"(-?0x[0-9a-f.]+p[-+]?\d+)f"
    val = lambda h: Decimal(float.fromhex(h))
    c = {n: val(h) for n, h in re.findall(r"(kLn2C[123]) = " + hexf, text)}
    assert abs(c["kLn2C1"] + c["kLn2C2"] + c["kLn2C3"] - Decimal(2).ln()) < Decimal(2) ** -64  # half a unit of kLn2C3
    assert c["kLn2C1"] * 4096 == 2839
    for name, d in (("kInv6", Decimal(1) / 6), ("kInv24", Decimal(1) / 24)):
        hi, lo = re.search(name + r"Hi = " + hexf + ", " + name + r"Lo = " + hexf, text).groups()
        assert abs(val(hi) + val(lo) - d) < d * Decimal(2) ** -48
    rows = re.findall(r"\{" + hexf + ", " + hexf + r"\},\s+// j = (-?\d+)", text)
    assert [int(r[2]) for r in rows] == list(range(-23, 24))
    for hi, lo, j in rows:
        e = (Decimal(int(j)) / 64).exp()
        assert abs(val(hi) + val(lo) - e) < e * Decimal(2) ** -48
