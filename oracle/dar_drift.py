"""Dequantize-add-requantize (DAR) drift: what the overlay design avoids.

TEST INFRASTRUCTURE AND ANALYSIS ONLY, on the CPU.  Nothing on the library's
product path reaches this module; the library never requantizes.

"Deep Technical Design: Exact, Atomic, Reversible Specialist Overlays on
Quantized Transformer Bases" §5 "Quantized-Base Numerical Analysis", The
Pathology of Dequantize-Add-Requantize (DAR) Error:

1. Scale recomputation shift: the block scale follows the block's largest
   magnitude, so one large delta inflates the scale and the other codes of the
   block collapse toward zero.
2. Repeated merge degradation: switching states by DAR applies the lossy
   quantizer again on every switch, and its errors accumulate.
3. Fresh-base oracle: the only drift-free reference is the original base plus
   the active deltas, evaluated from the untouched base bytes.

"We propose a content-addressed overlay system" report, §"Quantized-Base
Numerical Analysis" (rounding when adding the adapter back into the quantized
format) and §"Explicit Correctness and Atomicity Invariants" (no drift from
repeated applications) state the same hazard; its open question is the size of
the error for concrete formats, which `drift_table` measures on synthetic
8B-shape tensors.

Q is the quantizer the synthetic inputs use (the `synth` package: q8_0,
q4_0, q4_K with round-half-away codes and f16 scales); deq is the oracle's
exact dequantization.
"""
from __future__ import annotations

import numpy as np

import synth as S

from . import ovl_oracle as O

_QUANTIZE = {O.Q8_0: S.quantize_q8_0, O.Q4_0: S.quantize_q4_0, O.Q4_K: S.quantize_q4_k}


def quantize(quant: int, w: np.ndarray):
    """Q(w): float -> (codes, scale plane) of the given profile (fp32 input)."""
    return _QUANTIZE[quant](np.asarray(w, dtype=np.float32))


def dar_merge(quant: int, qs, d, delta) -> tuple:
    """One destructive merge: Q(deq(qs, d) + delta), the new base bytes."""
    w = O.dequantize(quant, qs, d) + np.asarray(delta, np.float64)
    return quantize(quant, w)


def dar_switch_cycles(quant: int, qs, d, delta, cycles: int):
    """base -> adapter -> base, `cycles` times, by DAR: add the delta and
    requantize, then subtract it and requantize.  Returns the list of bases
    after each full cycle (the first entry is the starting base)."""
    out = [(qs, d)]
    for _ in range(cycles):
        q1, d1 = dar_merge(quant, *out[-1], delta)
        q2, d2 = dar_merge(quant, q1, d1, -np.asarray(delta, np.float64))
        out.append((q2, d2))
    return out


def drift(quant: int, base, other) -> dict:
    """How far `other` is from the fresh `base` (both (codes, scales))."""
    w0 = O.dequantize(quant, *base)
    w1 = O.dequantize(quant, *other)
    diff = w1 - w0
    return {
        "rel_fro": float(np.linalg.norm(diff) / np.linalg.norm(w0)),
        "max_abs": float(np.abs(diff).max()),
        "weights_changed": float(np.count_nonzero(diff) / diff.size),
    }


def output_error(quant: int, fresh, merged, delta, x) -> float:
    """max_i |y_DAR - y_fresh| / sum_j |W'_ij x_j| with y_fresh the fresh-base
    oracle (untouched base plus the delta, fp64) and y_DAR from the merged bytes."""
    w_fresh = O.dequantize(quant, *fresh) + np.asarray(delta, np.float64)
    y_fresh = O.merged_path(w_fresh, x)
    y_dar = O.merged_path(O.dequantize(quant, *merged), x)
    scale = np.abs(np.asarray(x, np.float64)) @ np.abs(w_fresh).T
    return float((np.abs(y_dar - y_fresh) / scale).max())


def drift_table(shape=(4096, 4096), rank: int = 16, s: float = 2.0, cycles=(1, 2, 5, 10), seed: int = 0):
    """Drift of the base after DAR switch cycles (base -> A -> base) and the
    output error of one DAR merge against the fresh-base oracle, per format,
    for a seeded N(0, 0.02) tensor and a rank-`rank` N(0, 0.01) adapter."""
    m, n = shape
    rng = np.random.default_rng(seed)
    w = S.gaussian(rng, (m, n), 0.02)
    A = S.gaussian(rng, (rank, n), 0.01).astype(np.float64)
    B = S.gaussian(rng, (m, rank), 0.01).astype(np.float64)
    delta = s * (B @ A)
    x = S.gaussian(rng, (4, n), 1.0)
    rows = []
    for quant in (O.Q8_0, O.Q4_0, O.Q4_K):
        base = quantize(quant, w)
        merged = dar_merge(quant, *base, delta)
        bases = dar_switch_cycles(quant, *base, delta, max(cycles))
        rows.append({
            "quant": quant,
            "merge_output_error": output_error(quant, base, merged, delta, x),
            "cycles": {c: drift(quant, base, bases[c]) for c in cycles},
        })
    return rows


if __name__ == "__main__":
    names = {O.Q8_0: "q8_0", O.Q4_0: "q4_0", O.Q4_K: "q4_K"}
    table = drift_table()
    print("| format | one DAR merge: max output error / sum|W'x| | base drift after 1 / 2 / 5 / 10 cycles "
          "(relative Frobenius) | weights changed after 10 |")
    print("|---|---:|---|---:|")
    for r in table:
        c = r["cycles"]
        print(f"| {names[r['quant']]} | {r['merge_output_error']:.2e} | "
              + " / ".join(f"{c[k]['rel_fro']:.2e}" for k in sorted(c))
              + f" | {100 * c[max(c)]['weights_changed']:.1f} % |")
