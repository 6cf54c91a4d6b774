"""GPU parity of the per-layer JIT path: fp32 materialization S = deq + sum s B A
(bit-exact dequantization for an empty stack) and the tcgen05 TF32 prefill GEMM
Y = X S^T, against the fp64 oracle; dual path vs JIT path on the q4_0 block
with two stacked adapters."""
import numpy as np
import pytest

import oracle as O
import synth as S
from gpu_common import (assert_within_bound, deq_of, lora_terms, make_runtime, require_gpu, stage, torch,
                        x_device)

pytestmark = pytest.mark.gpu


def jit_scratch(m, n, T):
    need = (m * n * 4 + 127) // 128 * 128 + T * n * 4
    return torch.empty(need + 256, dtype=torch.uint8, device="cuda")


def materialize(rt, i, m, n):
    import quantized_base_lora_gb300 as q
    S_dev = torch.empty((m, n), dtype=torch.float32, device="cuda")
    q.check(q.ovl_materialize_layer(rt.ctx, i, S_dev.data_ptr(), S_dev.numel() * 4,
                                    int(torch.cuda.current_stream().cuda_stream)), rt.ctx)
    torch.cuda.synchronize()
    return S_dev.cpu().numpy()


@pytest.mark.parametrize("quant", [S.Q8_0, S.Q4_0])
def test_materialize_empty_stack_is_exact_dequant(quant):
    require_gpu()
    rng = np.random.default_rng(5 + quant)
    W = S.gaussian(rng, (300, 512), 0.02)
    base = S.build_base(quant, [(0, 0, W)])
    rt = make_runtime(base, arena_bytes=32 << 20)
    got = materialize(rt, 0, 300, 512)
    want = deq_of(base, 0).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    rt.close()


def test_materialize_with_stack_within_bound():
    require_gpu()
    rng = np.random.default_rng(9)
    m, n = 257, 384
    W = S.gaussian(rng, (m, n), 0.02)
    base = S.build_base(S.Q8_0, [(0, 0, W)])
    ads = []
    for r, s in ((16, 1.0), (40, 0.5)):
        ads.append((S.build_adapter(base, [0], [r], [(S.gaussian(rng, (r, n), 0.01),
                                                      S.gaussian(rng, (m, r), 0.01))]), s))
    rt = make_runtime(base, arena_bytes=32 << 20)
    assert rt.activate([stage(rt, a) for a, _ in ads], [s for _, s in ads])[0] == 0
    got = materialize(rt, 0, m, n).astype(np.float64)
    deq = deq_of(base, 0)
    terms = lora_terms(ads, 0)
    Wp = O.effective_weight(deq, terms)
    assert (np.abs(got - Wp) <= O.materialize_bound(deq, terms)).all()
    rt.close()


JIT_CASES = [  # quant, m, n, T, ranks, xdtype
    (S.Q8_0, 256, 256, 1, (8,), "f32"),
    (S.Q8_0, 1000, 512, 17, (16,), "bf16"),
    (S.Q4_0, 384, 1024, 64, (4, 12), "bf16"),
    (S.Q8_0, 640, 768, 300, (16,), "bf16"),
    (S.Q4_0, 130, 4096, 256, (), "f32"),
]


@pytest.mark.parametrize("case", JIT_CASES, ids=[f"q{c[0]}_{c[1]}x{c[2]}_T{c[3]}" for c in JIT_CASES])
def test_jit_forward_vs_oracle(case):
    require_gpu()
    import quantized_base_lora_gb300 as q
    quant, m, n, T, ranks, xdt = case
    rng = np.random.default_rng(m + n + T)
    W = S.gaussian(rng, (m, n), 0.02)
    base = S.build_base(quant, [(0, 0, W)])
    ads = [(S.build_adapter(base, [0], [r], [(S.gaussian(rng, (r, n), 0.01), S.gaussian(rng, (m, r), 0.01))]),
            2.0) for r in ranks]
    rt = make_runtime(base, arena_bytes=32 << 20)
    assert rt.activate([stage(rt, a) for a, _ in ads], [s for _, s in ads])[0] == 0
    x = S.gaussian(rng, (T, n), 1.0)
    xd, x64 = x_device(x, xdt)
    y = rt.forward(0, xd, path=q.OVL_PATH_JIT, scratch=jit_scratch(m, n, T))
    torch.cuda.synchronize()
    assert rt.check_device() == 0
    assert_within_bound(y.cpu().numpy(), deq_of(base, 0), lora_terms(ads, 0), x64, f"jit {case}")
    rt.close()


@pytest.fixture(scope="module")
def block_q4():
    require_gpu()
    base = S.block_base(S.Q4_0, projs=("q", "k", "gate", "down"))
    a16 = S.block_adapter(base, adapter=0, rank=16)
    a64 = S.block_adapter(base, adapter=1, rank=64)
    rt = make_runtime(base, arena_bytes=512 << 20)
    assert rt.activate([stage(rt, a16), stage(rt, a64)], [1.0, 0.5])[0] == 0
    return base, a16, a64, rt


@pytest.mark.parametrize("T", [1, 4, 8])
@pytest.mark.parametrize("proj", [0, 1, 2, 3])
def test_dual_equals_jit_q4_stacked(block_q4, proj, T):
    import quantized_base_lora_gb300 as q
    base, a16, a64, rt = block_q4
    t = base.tensors[proj]
    x = S.activations(T, t.d_in)
    xd, x64 = x_device(x, "bf16")
    y_dual = rt.forward(proj, xd).cpu().numpy()
    y_jit = rt.forward(proj, xd, path=q.OVL_PATH_JIT, scratch=jit_scratch(t.d_out, t.d_in, T)).cpu().numpy()
    assert rt.check_device() == 0
    deq = deq_of(base, proj)
    terms = lora_terms([(a16, 1.0), (a64, 0.5)], proj)
    assert_within_bound(y_jit, deq, terms, x64, "jit")
    assert_within_bound(y_dual, deq, terms, x64, "dual")
    bound = O.error_bound(O.effective_weight(deq, terms), x64)
    assert (np.abs(y_dual.astype(np.float64) - y_jit) <= bound).all()


def test_prefill_512_tokens_gate_q8():
    """One projection of the 32-layer prefill workload: gate 14336x4096 q8_0,
    rank-16 adapter, T = 512 bf16 tokens, per-layer JIT."""
    require_gpu()
    import quantized_base_lora_gb300 as q
    base = S.block_base(S.Q8_0, projs=("gate",))
    ad = S.block_adapter(base, adapter=0, rank=16)
    rt = make_runtime(base, arena_bytes=256 << 20)
    assert rt.activate([stage(rt, ad)], [2.0])[0] == 0
    t = base.tensors[0]
    x = S.activations(512, t.d_in)
    xd, x64 = x_device(x, "bf16")
    y = rt.forward(0, xd, path=q.OVL_PATH_JIT, scratch=jit_scratch(t.d_out, t.d_in, 512)).cpu().numpy()
    assert rt.check_device() == 0
    assert_within_bound(y, deq_of(base, 0), lora_terms([(ad, 2.0)], 0), x64, "prefill gate")
    rt.close()
