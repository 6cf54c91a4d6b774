"""The byte counts behind bench.py's roofline numerators (CPU), recomputed by
hand from the 8B-shape block's shapes and the formats' block sizes."""
import os
import sys

import numpy as np

import synth as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class _Tensor:
    def __init__(self, d_out, d_in):
        self.d_out, self.d_in = d_out, d_in


class _Base:
    def __init__(self, quant):
        self.quant = quant
        self.tensors = [_Tensor(*S.SHAPES_8B[p]) for p in S.PROJ]


def test_block_weight_count_and_q8_bytes():
    w = sum(m * n for m, n in S.SHAPES_8B.values())
    assert w == 218_103_808                                   # 8B-shape decoder block
    # q8_0: 32 int8 codes + one f16 scale per 32 weights = 34 bytes per block
    assert sum(S.qs_bytes(S.Q8_0, m, n) + S.d_bytes(m, n) for m, n in S.SHAPES_8B.values()) == w // 32 * 34
    # q4_0 and q4_K: 4.5 bits per weight
    for q in (S.Q4_0, S.Q4_K):
        assert sum(S.qs_bytes(q, m, n) + S.d_bytes(m, n) for m, n in S.SHAPES_8B.values()) * 8 == w * 4.5


def test_decode_step_bytes():
    base = _Base(S.Q8_0)
    lora = sum(16 * (m + n) * 4 for m, n in S.SHAPES_8B.values())
    assert lora == 5_242_880                                  # rank-16 fp32 factors on all seven
    eff = bench.effective_bytes(base, None)
    assert eff == 218_103_808 // 32 * 34 + lora == 236_978_176
    xy = sum(2 * n + 4 * m for m, n in S.SHAPES_8B.values())  # bf16 x read, fp32 y written, per tensor
    assert bench.algorithmic_bytes(base, None) == eff + xy == 237_228_032


def test_traffic_constant_is_per_launch_of_the_same_step():
    # the measured traffic per launch (when the current kernel has been measured)
    # is within 1 % of the algorithmic bytes per launch
    alg = bench.algorithmic_bytes(_Base(S.Q8_0), None) / 4
    if bench.K1_TRAFFIC_PER_LAUNCH is not None:
        assert abs(bench.K1_TRAFFIC_PER_LAUNCH / alg - 1) < 0.01


def test_sparse_overlay_bytes_formula():
    # k pairs cost k * (4 + 2) bytes: 32-bit index, 16-bit value
    rng = np.random.default_rng(0)
    idx, val = S.dare_entries(rng, 64, 256, keep=0.1)
    sp = S.build_sparse_adapter([0], [(idx, val)])
    assert idx.nbytes + val.nbytes == 6 * sp.nnz[0]
    assert sp.payload.nbytes >= 6 * sp.nnz[0] and sp.idx_off[0] % 16 == 0 and sp.val_off[0] % 16 == 0


def test_secondary_workloads_reduce_each_line_and_survive_a_failure(monkeypatch):
    """The default line's `secondary` block: each workload's last emitted line
    reduced to value, per-token-count step time and roofline fraction; a
    workload that raises is reported, not fatal; emit is restored."""
    import argparse

    def ok(args):
        assert args.steps == 50 and args.warmup == 5
        bench.emit({"metric": "m", "value": 2.0, "unit": "u",
                    "per_T": {1: {"ms_per_step": 0.0425, "roofline": {"frac": 0.44444, "bound": "hbm"}}}})

    def flat(args):
        bench.emit({"metric": "s", "value": 88.0, "unit": "us", "roofline": {"frac": 0.1177, "bound": "tensor"}})

    def boom(args):
        raise RuntimeError("no device")

    keep = bench.emit
    monkeypatch.setattr(bench, "SECONDARY", ("a", "b", "c"))
    monkeypatch.setattr(bench, "WORKLOADS", {"a": ok, "b": flat, "c": boom})
    out = bench.secondary_workloads(argparse.Namespace(steps=200, warmup=10, gpus=1))
    assert out["a"] == {"metric": "m", "value": 2.0, "unit": "u",
                        "per_T": {"1": {"us_per_step": 42.5, "frac": 0.4444, "bound": "hbm"}}}
    assert out["b"] == {"metric": "s", "value": 88.0, "unit": "us", "frac": 0.1177, "bound": "tensor"}
    assert out["c"]["error"].startswith("RuntimeError")
    assert bench.emit is keep
