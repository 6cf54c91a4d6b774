"""Shared helpers of the GPU tests: upload synthetic workloads through the C ABI
and compare library outputs with the oracle."""
import numpy as np
import pytest

import oracle as O
import synth as S

torch = pytest.importorskip("torch")


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")


def tensor_tuples(base):
    return [(t.layer, t.proj, t.d_out, t.d_in, t.qs_off, t.d_off) for t in base.tensors]


def adapter_tuples(ad):
    return list(zip(ad.targets, ad.ranks, ad.a_off, ad.b_off))


def make_runtime(base, arena_bytes=256 << 20, policy=None):
    import quantized_base_lora_gb300 as q
    from quantized_base_lora_gb300.runtime import Runtime
    rt = Runtime(arena_bytes=arena_bytes, policy=policy or q.OVL_SWITCH_REJECT)
    st = rt.load_base(base.quant, tensor_tuples(base), base.buf, S.content_digest(base.buf))
    assert st == 0, q.ovl_last_error(rt.ctx)
    return rt


def stage(rt, ad):
    import quantized_base_lora_gb300 as q
    st, h = rt.stage(ad, S.content_digest(ad.payload))
    assert st == 0, q.ovl_last_error(rt.ctx)
    return h


def x_device(x_f32, dtype):
    """x float32 numpy -> (device tensor of `dtype`, float64 values the device sees)."""
    if dtype == "bf16":
        bits = S.to_bf16_bits(x_f32)
        xd = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        return xd, S.bf16_bits_to_f32(bits).astype(np.float64)
    return torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).cuda(), x_f32.astype(np.float64)


def deq_of(base, i):
    qs, d = base.planes[i]
    return O.dequantize(base.quant, qs, d)


def lora_terms(ads_scales, tensor_index):
    """[(Adapter, s)] -> oracle terms [(A, B, s)] for one base tensor (composition order)."""
    out = []
    for ad, s in ads_scales:
        if tensor_index in ad.targets:
            A, B = ad.factors[ad.targets.index(tensor_index)]
            out.append((A, B, float(np.float32(s))))
    return out


def assert_within_bound(y_gpu, deq, terms, x64, label=""):
    """|y_gpu - y_oracle| <= 2e-3 * sum_j |W'_ij x_j| + 1e-5 per output."""
    Wp = O.effective_weight(deq, terms)
    y_ref = O.dual_path(deq, terms, x64)
    bound = O.error_bound(Wp, x64)
    err = np.abs(np.asarray(y_gpu, np.float64) - y_ref)
    ratio = float((err / bound).max()) if err.size else 0.0
    assert np.isfinite(y_gpu).all(), f"{label}: non-finite output"
    assert (err <= bound).all(), f"{label}: max err/bound = {ratio:.3g}"
    return ratio
