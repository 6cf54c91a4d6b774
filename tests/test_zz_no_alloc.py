"""The allocation-free dual-path forward (ovl_dualpath_forward_noalloc).

It exists for callers that can neither lend the library an arena nor allocate
device memory when they call: an embedder whose device memory belongs to its
own pooled allocator, or a latency-critical caller that cannot take the
device-wide stall a cudaMalloc may cause.  Its scratch lives in one file-scope
device array that every call reuses.  This test calls it twice in a row
through the C ABI -- the second call runs on whatever the first left in the
array -- and checks both outputs against the regular entry point
(ovl_linear_forward) and the oracle, within the same per-output tolerance as
the other parity tests.  Self-contained: it passes in a fresh process and after
the rest of the suite.  Kept last in collection order.
"""
import numpy as np
import pytest

import oracle as O
import synth as S
from gpu_common import assert_within_bound, deq_of, lora_terms, make_runtime, require_gpu, stage, torch, x_device

pytestmark = pytest.mark.gpu

CASES = [
    # quant, d_out, d_in, T, ranks, scales, x dtype, outliers
    (S.Q8_0, 1024, 4096, 1, (16,), (2.0,), "bf16", False),
    (S.Q4_0, 1000, 288, 3, (5, 7), (1.0, 0.5), "f32", False),
    # 8 tokens at an aligned d_in: linear_forward takes the tensor-core route
    # here, this entry point the decode kernel's 8-token tiles
    (S.Q8_0, 512, 2048, 8, (16, 4), (1.0, 0.5), "bf16", False),
    # 24 tokens: three launches of 8-token tiles in one call, sharing the slots
    (S.Q8_0, 512, 4096, 24, (16,), (2.0,), "bf16", False),
    # outliers ~1e7 times their block neighbours, on columns whose weights are 0
    (S.Q8_0, 300, 4096, 2, (16,), (2.0,), "f32", True),
]


def _build(case, seed):
    quant, m, n, T, ranks, scales, xdt, outliers = case
    rng = np.random.default_rng(seed)
    W = S.gaussian(rng, (m, n), 0.02)
    cols = np.array([32 * b + (5 * b) % 32 for b in range(0, n // 32, 3)])
    if outliers:
        W[:, cols] = 0.0
    base = S.build_base(quant, [(0, 0, W)])
    ads = []
    for r, s in zip(ranks, scales):
        A = S.gaussian(rng, (r, n), 0.01)
        B = S.gaussian(rng, (m, r), 0.01)
        ads.append((S.build_adapter(base, [0], [r], [(A, B)]), s))
    x = S.gaussian(rng, (T, n), 1.0)
    if outliers:
        x *= np.float32(1e-3)
        x[:, cols] = np.float32(1e4)
    return base, ads, x


def test_noalloc_forward_matches_linear_forward_on_two_calls_in_a_row():
    require_gpu()
    import quantized_base_lora_gb300 as q
    stream = torch.cuda.Stream()
    sh = int(stream.cuda_stream)
    prepared = []
    for i, case in enumerate(CASES):
        base, ads, x = _build(case, 100 + i)
        rt = make_runtime(base, arena_bytes=64 << 20)
        hs = [stage(rt, ad) for ad, _ in ads]
        assert rt.activate(hs, [s for _, s in ads])[0] == 0
        xd, x64 = x_device(x, case[6])
        y_ref = rt.forward(0, xd)                        # existing entry point
        torch.cuda.synchronize()
        A_dev = [torch.from_numpy(ad.factors[0][0]).cuda() for ad, _ in ads]
        B_dev = [torch.from_numpy(ad.factors[0][1]).cuda() for ad, _ in ads]
        t = base.tensors[0]
        y_na = torch.full((case[3], case[1]), float("nan"), device="cuda")
        prepared.append((case, base, ads, rt, xd, x64, y_ref, A_dev, B_dev, t, y_na))
    # the two calls, back to back on one stream, sharing the static scratch array
    for case, base, ads, rt, xd, x64, y_ref, A_dev, B_dev, t, y_na in prepared:
        st = q.ovl_dualpath_forward_noalloc(
            rt.base.data_ptr() + t.qs_off, rt.base.data_ptr() + t.d_off, base.quant, t.d_out, t.d_in,
            [a.data_ptr() for a in A_dev], [b.data_ptr() for b in B_dev], list(case[4]), list(case[5]),
            xd.data_ptr(), q.OVL_BF16 if case[6] == "bf16" else q.OVL_F32, case[3], y_na.data_ptr(), sh)
        assert st == q.OVL_OK, st
    stream.synchronize()
    for case, base, ads, rt, xd, x64, y_ref, A_dev, B_dev, t, y_na in prepared:
        deq = deq_of(base, 0)
        terms = lora_terms(ads, 0)
        got = y_na.cpu().numpy()
        ref = y_ref.cpu().numpy()
        assert_within_bound(got, deq, terms, x64, f"noalloc {case}")
        bound = O.error_bound(O.effective_weight(deq, terms), x64)
        assert (np.abs(got.astype(np.float64) - ref.astype(np.float64)) <= bound).all()
        rt.close()


def test_noalloc_forward_rejects_bad_arguments():
    require_gpu()
    import quantized_base_lora_gb300 as q
    y = torch.zeros(1, 64, device="cuda")
    x = torch.zeros(1, 64, device="cuda")
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    assert q.ovl_dualpath_forward_noalloc(p, p + 4096, 3, 64, 64, [], [], [], [], x.data_ptr(), q.OVL_F32, 1,
                                          y.data_ptr()) == q.OVL_E_QUANT
    assert q.ovl_dualpath_forward_noalloc(p, p + 4096, q.OVL_Q8_0, 64, 60, [], [], [], [], x.data_ptr(),
                                          q.OVL_F32, 1, y.data_ptr()) == q.OVL_E_SHAPE
    assert q.ovl_dualpath_forward_noalloc(p + 8, p + 4096, q.OVL_Q8_0, 64, 64, [], [], [], [], x.data_ptr(),
                                          q.OVL_F32, 1, y.data_ptr()) == q.OVL_E_SHAPE
    A = torch.zeros(4, 64, device="cuda")
    assert q.ovl_dualpath_forward_noalloc(p, p + 4096, q.OVL_Q8_0, 64, 64, [A.data_ptr()], [A.data_ptr()], [4],
                                          [float("nan")], x.data_ptr(), q.OVL_F32, 1, y.data_ptr()) == q.OVL_E_ARG
    assert q.ovl_dualpath_forward_noalloc(p, p + 4096, q.OVL_Q8_0, 64, 64, [], [], [], [], x.data_ptr(),
                                          q.OVL_F32, 0, y.data_ptr()) == q.OVL_OK
