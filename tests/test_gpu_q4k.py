"""GPU parity of the q4_K base (256-weight super-blocks: 6-bit sub-block scales
and minimums under two f16 scales) against the fp64 oracle, through the C ABI:
the 8B-shape block with a rank-16 adapter at T = 1, multi-token K1 tiles and
the tensor-core route (4 tokens and more),
multi-tensor launches, ragged shapes, a zero-B adapter, the JIT
materialization (correctly rounded dequantization for an empty stack) and the
JIT prefill GEMM, a segmented batch, and the d_in rule of the format."""
import numpy as np
import pytest

import oracle as O
import synth as S
from gpu_common import (assert_within_bound, deq_of, lora_terms, make_runtime, require_gpu, stage, tensor_tuples,
                        torch, x_device)

pytestmark = pytest.mark.gpu


def fwd(rt, i, xd):
    y = rt.forward(i, xd)
    torch.cuda.synchronize()
    assert rt.check_device() == 0
    return y.cpu().numpy()


@pytest.fixture(scope="module")
def block_q4k():
    require_gpu()
    base = S.block_base(S.Q4_K)
    ad = S.block_adapter(base, adapter=0, rank=16)
    rt = make_runtime(base, arena_bytes=512 << 20)
    assert rt.activate([stage(rt, ad)], [2.0])[0] == 0
    return base, ad, rt


@pytest.mark.parametrize("proj", list(range(7)))
def test_block_q4k_decode_bf16(block_q4k, proj):
    base, ad, rt = block_q4k
    t = base.tensors[proj]
    x = S.activations(1, t.d_in)
    xd, x64 = x_device(x, "bf16")
    y = fwd(rt, proj, xd)
    assert_within_bound(y, deq_of(base, proj), lora_terms([(ad, 2.0)], proj), x64, S.PROJ[proj])


@pytest.mark.parametrize("T", [2, 3, 4, 8, 13, 64, 100])   # 4 and up: the tensor-core route
@pytest.mark.parametrize("proj", [1, 6])
def test_block_q4k_multi_token(block_q4k, proj, T):
    base, ad, rt = block_q4k
    t = base.tensors[proj]
    x = S.activations(T, t.d_in)
    xd, x64 = x_device(x, "bf16")
    y = fwd(rt, proj, xd)
    assert y.shape == (T, t.d_out)
    assert_within_bound(y, deq_of(base, proj), lora_terms([(ad, 2.0)], proj), x64, f"{S.PROJ[proj]} T={T}")


@pytest.mark.parametrize("T", [1, 5])
def test_block_q4k_multi_tensor_launch(block_q4k, T):
    import quantized_base_lora_gb300 as q
    base, ad, rt = block_q4k
    for grp in ([0, 1, 2], [4, 5]):
        d_in = base.tensors[grp[0]].d_in
        x = S.activations(T, d_in, seed=77 + T)
        xd, x64 = x_device(x, "bf16")
        ys = [torch.full((T, base.tensors[i].d_out), float("nan"), device="cuda") for i in grp]
        st = q.ovl_linear_forward_multi(rt.ctx, grp, xd.data_ptr(), q.OVL_BF16, T, [y.data_ptr() for y in ys],
                                        int(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        assert st == 0 and rt.check_device() == 0
        for i, y in zip(grp, ys):
            assert_within_bound(y.cpu().numpy(), deq_of(base, i), lora_terms([(ad, 2.0)], i), x64,
                                f"multi {grp} tensor {i} T={T}")


RAGGED = [  # (d_out, d_in, T, ranks, xdtype)
    (1, 256, 1, (), "f32"),
    (3, 512, 2, (1,), "bf16"),
    (1000, 768, 3, (5, 7), "f32"),
    (77, 4352, 1, (3,), "bf16"),
    (513, 2048, 9, (32, 2), "bf16"),
    (4096, 256, 1, (128, 128), "f32"),
]


@pytest.mark.parametrize("case", RAGGED, ids=[f"{c[0]}x{c[1]}_T{c[2]}_r{'-'.join(map(str, c[3]))}_{c[4]}"
                                             for c in RAGGED])
def test_q4k_ragged_shapes(case):
    require_gpu()
    m, n, T, ranks, xdt = case
    rng = np.random.default_rng(m * 11 + n)
    W = S.gaussian(rng, (m, n), 0.02)
    base = S.build_base(S.Q4_K, [(0, 0, W)])
    ads = []
    for k, r in enumerate(ranks):
        A = S.gaussian(rng, (r, n), 0.01)
        B = S.gaussian(rng, (m, r), 0.01)
        ads.append((S.build_adapter(base, [0], [r], [(A, B)]), [2.0, 0.5, 1.25][k % 3]))
    rt = make_runtime(base, arena_bytes=64 << 20)
    assert rt.activate([stage(rt, ad) for ad, _ in ads], [s for _, s in ads])[0] == 0
    x = S.gaussian(rng, (T, n), 1.0)
    xd, x64 = x_device(x, xdt)
    y = fwd(rt, 0, xd)
    assert y.shape == (T, m)
    assert_within_bound(y, deq_of(base, 0), lora_terms(ads, 0), x64, str(case))
    rt.close()


def test_q4k_zero_B_adapter_gives_base_output_exactly():
    require_gpu()
    rng = np.random.default_rng(21)
    m, n = 640, 1024
    base = S.build_base(S.Q4_K, [(0, 0, S.gaussian(rng, (m, n), 0.02))])
    ad0 = S.build_adapter(base, [0], [16], [(S.gaussian(rng, (16, n), 0.01), np.zeros((m, 16), np.float32))])
    rt = make_runtime(base, arena_bytes=32 << 20)
    h = stage(rt, ad0)
    xd, x64 = x_device(S.gaussian(rng, (1, n), 1.0), "bf16")
    y_base = fwd(rt, 0, xd)
    assert rt.activate([h], [2.0])[0] == 0
    y_zero = fwd(rt, 0, xd)
    assert np.array_equal(y_base.view(np.uint32), y_zero.view(np.uint32))
    assert_within_bound(y_base, deq_of(base, 0), [], x64, "q4_K base")
    rt.close()


def test_q4k_materialize_empty_stack_is_rounded_exact_dequant():
    require_gpu()
    import quantized_base_lora_gb300 as q
    rng = np.random.default_rng(23)
    m, n = 300, 1536
    base = S.build_base(S.Q4_K, [(0, 0, S.gaussian(rng, (m, n), 0.02))])
    rt = make_runtime(base, arena_bytes=32 << 20)
    S_dev = torch.empty((m, n), dtype=torch.float32, device="cuda")
    q.check(q.ovl_materialize_layer(rt.ctx, 0, S_dev.data_ptr(), S_dev.numel() * 4,
                                    int(torch.cuda.current_stream().cuda_stream)), rt.ctx)
    torch.cuda.synchronize()
    # d*sc*code - dmin*m rounded once to fp32 (the oracle's fp64 value is exact here)
    want = deq_of(base, 0).astype(np.float32)
    assert np.array_equal(S_dev.cpu().numpy().view(np.uint32), want.view(np.uint32))
    rt.close()


@pytest.mark.parametrize("T", [1, 64, 200])
def test_q4k_jit_forward_vs_oracle(T):
    require_gpu()
    import quantized_base_lora_gb300 as q
    rng = np.random.default_rng(25 + T)
    m, n = 384, 1024
    base = S.build_base(S.Q4_K, [(0, 0, S.gaussian(rng, (m, n), 0.02))])
    ads = [(S.build_adapter(base, [0], [r], [(S.gaussian(rng, (r, n), 0.01), S.gaussian(rng, (m, r), 0.01))]), s)
           for r, s in ((16, 1.0), (64, 0.5))]
    rt = make_runtime(base, arena_bytes=32 << 20)
    assert rt.activate([stage(rt, a) for a, _ in ads], [s for _, s in ads])[0] == 0
    xd, x64 = x_device(S.gaussian(rng, (T, n), 1.0), "bf16")
    scratch = torch.empty((m * n * 4 + 127) // 128 * 128 + T * n * 4 + 256, dtype=torch.uint8, device="cuda")
    y_jit = rt.forward(0, xd, path=q.OVL_PATH_JIT, scratch=scratch)
    y_dual = rt.forward(0, xd)
    torch.cuda.synchronize()
    assert rt.check_device() == 0
    for name, y in (("jit", y_jit), ("dual", y_dual)):
        assert_within_bound(y.cpu().numpy(), deq_of(base, 0), lora_terms(ads, 0), x64, f"{name} T={T}")
    rt.close()


def test_q4k_segmented_batch():
    require_gpu()
    import quantized_base_lora_gb300 as q
    base = S.block_base(S.Q4_K, projs=("q",))
    ads = [S.block_adapter(base, adapter=a, rank=16) for a in range(4)]
    rt = make_runtime(base, arena_bytes=128 << 20)
    assert rt.activate([stage(rt, a) for a in ads], [2.0] * 4, mode=q.OVL_MODE_TABLE)[0] == 0
    T = 20
    ids = S.zipf_ids(T, 4, 1.1, seed=31)
    perm, offsets, slots = S.segments(ids)
    xd, x64 = x_device(S.activations(T, 4096, seed=32), "bf16")
    y = torch.full((T, 4096), float("nan"), device="cuda")
    st = q.ovl_segmented_forward(rt.ctx, 0, xd.data_ptr(), q.OVL_BF16, T, [int(v) for v in offsets],
                                 [int(v) for v in slots], [int(v) for v in perm], y.data_ptr(),
                                 int(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0 and rt.check_device() == 0
    y = y.cpu().numpy()
    deq = deq_of(base, 0)
    for t in range(T):
        A, B = ads[ids[t]].factors[0]
        assert_within_bound(y[t:t + 1], deq, [(A, B, 2.0)], x64[t:t + 1], f"token {t} adapter {ids[t]}")
    rt.close()


def test_q4k_base_needs_whole_super_blocks():
    require_gpu()
    import quantized_base_lora_gb300 as q
    from quantized_base_lora_gb300.runtime import Runtime
    rng = np.random.default_rng(27)
    good = S.build_base(S.Q4_K, [(0, 0, S.gaussian(rng, (8, 512), 0.02))])
    tt = tensor_tuples(good)
    bad = [(l, p, d_out, 480, qo, do) for (l, p, d_out, d_in, qo, do) in tt]   # 480: a multiple of 32, not of 256
    rt = Runtime(arena_bytes=16 << 20)
    assert rt.load_base(S.Q4_K, bad, good.buf, S.content_digest(good.buf)) == q.OVL_E_SHAPE
    assert rt.load_base(S.Q4_K, tt, good.buf, S.content_digest(good.buf)) == 0
    rt.close()
    # the allocation-free entry point does not take q4_K
    x = torch.zeros((1, 512), device="cuda")
    y = torch.zeros((1, 8), device="cuda")
    buf = torch.zeros(8192, dtype=torch.uint8, device="cuda")
    assert q.ovl_dualpath_forward_noalloc(buf.data_ptr(), buf.data_ptr() + 4096, q.OVL_Q4_K, 8, 512, [], [], [], [],
                                          x.data_ptr(), q.OVL_F32, 1, y.data_ptr(), 0) == q.OVL_E_QUANT
