"""Exhaustive agreement of the hardware E2M1 / E4M3 / E5M2 conversions with
the oracle's round-to-nearest-even encoders over every non-NaN fp32 bit
pattern (E5M2: the backward oracle's numpy encoder).
The GPU reports where the code changes between neighbouring patterns; the
oracle's change points come from bisection over its monotone encoder."""
import struct

import pytest

import oracle

pytestmark = pytest.mark.gpu


def _f(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def oracle_transitions(fmt, lo, hi):
    if fmt == 2:
        import oracle.bwd as ob
        enc = lambda y: int(ob.fp8_encode(y, ob.E5M2))
    else:
        enc = oracle.e2m1_encode if fmt == 0 else oracle.e4m3_encode
    code = lambda u: enc(_f(u))
    out = [(lo, code(lo))]

    def rec(a, ca, b, cb):  # a < b, ca = code(a), cb = code(b)
        if ca == cb:
            return
        if b == a + 1:
            out.append((b, cb))
            return
        m = (a + b) // 2
        cm = code(m)
        rec(a, ca, m, cm)
        rec(m, cm, b, cb)

    rec(lo, code(lo), hi, code(hi))
    return sorted(out)


@pytest.mark.parametrize("fmt", [0, 1, 2], ids=["e2m1", "e4m3", "e5m2"])
@pytest.mark.parametrize("lo,hi", [(0x00000000, 0x7F800000), (0x80000000, 0xFF800000)], ids=["pos", "neg"])
def test_hardware_conversion_matches_oracle(fmt, lo, hi):
    import blackwell_nvfp4_quantize_gb300 as fa

    gpu = fa.debug_cvt_transitions(fmt, lo, hi)
    ref = oracle_transitions(fmt, lo, hi)
    assert gpu == ref
