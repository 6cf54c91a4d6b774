"""Pins of the DAR drift analysis (CPU): the destructive
dequantize-add-requantize merge behaves as the quantized-base numerical
analysis of the pages describes, and the overlay path does not drift."""
import numpy as np

import oracle as O
import synth as S
from oracle import dar_drift as D


def _q8_block(codes, d=0.01):
    qs = np.asarray(codes, np.int8).reshape(1, 32)
    dbits = np.array([[np.float16(d).view(np.uint16)]], np.uint16)
    return qs, dbits


def test_scale_recomputation_shift_collapses_the_other_codes():
    # one block: code 127 then 31 codes of 4; a delta makes weight 0 ten times larger.
    # The new scale is ~10 d, so 4 d / 10 d = 0.4 rounds to 0: the other weights vanish.
    qs, d = _q8_block([127] + [4] * 31)
    w0 = O.dequantize_q8_0(qs, d)
    delta = np.zeros((1, 32))
    delta[0, 0] = 9 * w0[0, 0]
    q2, d2 = D.dar_merge(O.Q8_0, qs, d, delta)
    assert q2[0, 0] == 127 and np.all(q2[0, 1:] == 0)
    assert O.f16_to_float(d2)[0, 0] > 9 * O.f16_to_float(d)[0, 0]


def test_representable_delta_merges_exactly():
    # a delta of k*d on one weight that keeps the block maximum is exact under DAR
    rng = np.random.default_rng(3)
    codes = rng.integers(-100, 101, size=32)
    codes[0] = 127
    qs, d = _q8_block(codes)
    dv = float(O.f16_to_float(d)[0, 0])
    delta = np.zeros((1, 32))
    delta[0, 5] = 7 * dv
    q2, d2 = D.dar_merge(O.Q8_0, qs, d, delta)
    want = qs.astype(np.int64).copy()
    want[0, 5] += 7
    assert np.array_equal(d2, d) and np.array_equal(q2.astype(np.int64), want)


def test_dar_switch_cycles_drift_while_the_overlay_does_not():
    rng = np.random.default_rng(5)
    m, n = 64, 512
    w = S.gaussian(rng, (m, n), 0.02)
    A = S.gaussian(rng, (8, n), 0.01)
    B = S.gaussian(rng, (m, 8), 0.01)
    delta = 2.0 * (B.astype(np.float64) @ A.astype(np.float64))
    for quant in (O.Q8_0, O.Q4_0, O.Q4_K):
        base = D.quantize(quant, w)
        after = D.dar_switch_cycles(quant, *base, delta, 3)
        # base -> A -> base by DAR does not return the base bytes
        assert D.drift(quant, base, after[1])["rel_fro"] > 0
        # the overlay path: base -> A -> base evaluates from untouched bytes, so
        # the base comes back exactly
        before = (base[0].copy(), base[1].copy())
        deq = O.dequantize(quant, *base)
        O.effective_weight(deq, [(A, B, 2.0)])
        assert np.array_equal(O.effective_weight(O.dequantize(quant, *base), []), deq)
        assert np.array_equal(base[0], before[0]) and np.array_equal(base[1], before[1])


def test_one_dar_merge_output_error_against_the_fresh_base():
    rng = np.random.default_rng(7)
    m, n = 128, 512
    w = S.gaussian(rng, (m, n), 0.02)
    A = S.gaussian(rng, (16, n), 0.01).astype(np.float64)
    B = S.gaussian(rng, (m, 16), 0.01).astype(np.float64)
    delta = 2.0 * (B @ A)
    x = S.gaussian(rng, (2, n), 1.0)
    errs = {}
    for quant in (O.Q8_0, O.Q4_0):
        base = D.quantize(quant, w)
        errs[quant] = D.output_error(quant, base, D.dar_merge(quant, *base, delta), delta, x)
    # the merged bytes miss the fresh-base output; 4-bit codes miss it by more
    assert 0 < errs[O.Q8_0] < errs[O.Q4_0]
    # and a zero delta on the untouched base has no error
    base = D.quantize(O.Q8_0, w)
    assert D.output_error(O.Q8_0, base, base, np.zeros((m, n)), x) == 0
