"""GPU parity of the fused dual-path kernel against the fp64 oracle, through the
C ABI: the single 256x256 layer with its switch sequence, the 8B-shape q8_0
block, the q4_0 block with two stacked adapters at T = 1, 4, 8, ragged and
degenerate shapes."""
import numpy as np
import pytest

import oracle as O
import synth as S
from gpu_common import (adapter_tuples, assert_within_bound, deq_of, lora_terms, make_runtime, require_gpu,
                        stage, tensor_tuples, torch, x_device)

pytestmark = pytest.mark.gpu


def fwd(rt, i, xd):
    y = rt.forward(i, xd)
    torch.cuda.synchronize()
    assert rt.check_device() == 0
    return y.cpu().numpy()


# ----------------------------------------------------------------- single layer
@pytest.fixture(scope="module")
def layer256():
    require_gpu()
    base, ad_a, ad_b, x, s = S.single_layer_256()
    rt = make_runtime(base)
    return base, ad_a, ad_b, x, s, rt


def test_single_layer_switch_sequence(layer256):
    import quantized_base_lora_gb300 as q
    base, ad_a, ad_b, x, s, rt = layer256
    xd, x64 = x_device(x, "f32")
    deq = deq_of(base, 0)
    d0 = rt.base_digest()[1]
    ha, hb = stage(rt, ad_a), stage(rt, ad_b)
    outs = {}
    for name, handles, ads in (("base", [], []), ("A", [ha], [(ad_a, s)]), ("base2", [], []),
                               ("B", [hb], [(ad_b, s)])):
        st, cid = rt.activate(handles, [s] * len(handles))
        assert st == 0, q.ovl_last_error(rt.ctx)
        y = fwd(rt, 0, xd)
        assert_within_bound(y, deq, lora_terms(ads, 0), x64, name)
        outs[name] = y
        assert rt.base_digest()[1] == d0                       # base bytes untouched
    assert np.array_equal(outs["base"].view(np.uint32), outs["base2"].view(np.uint32))
    # reversibility: base -> A -> base -> B is bitwise base -> B in a fresh context
    rt2 = make_runtime(base)
    hb2 = stage(rt2, ad_b)
    st, cid2 = rt2.activate([hb2], [s])
    y2 = fwd(rt2, 0, xd)
    assert np.array_equal(outs["B"].view(np.uint32), y2.view(np.uint32))
    assert rt.state()["composition_id"] == rt2.state()["composition_id"] == cid2
    rt2.close()


def test_single_layer_ids_match_oracle(layer256):
    import json, os
    base, ad_a, ad_b, x, s, rt = layer256
    with open(os.path.join(os.path.dirname(__file__), "golden", "config1.json")) as f:
        g = json.load(f)
    rt3 = make_runtime(base)
    assert rt3.state()["composition_id"].hex() == g["ids"]["base"]
    ha = stage(rt3, ad_a)
    assert rt3.activate([ha], [s])[1].hex() == g["ids"]["A"]
    hb = stage(rt3, ad_b)
    assert rt3.activate([hb], [s])[1].hex() == g["ids"]["B"]
    assert rt3.state()["base_digest"].hex() == g["base_digest"]
    rt3.close()


def test_zero_B_adapter_gives_base_output_exactly(layer256):
    base, ad_a, ad_b, x, s, rt = layer256
    A, B = ad_a.factors[0]
    zb = S.build_adapter(base, [0], [8], [(A, np.zeros_like(B))])
    xd, _ = x_device(x, "f32")
    rt.activate([], [])
    y0 = fwd(rt, 0, xd)
    hz = stage(rt, zb)
    rt.activate([hz], [s])
    y1 = fwd(rt, 0, xd)
    assert np.array_equal(y0, y1)                                # fp32 ==
    assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))  # and bits (no -0 expected)
    rt.activate([], [])


def test_forward_is_deterministic(layer256):
    base, ad_a, ad_b, x, s, rt = layer256
    xd, _ = x_device(x, "f32")
    ha = stage(rt, ad_a)
    rt.activate([ha], [s])
    ys = [fwd(rt, 0, xd) for _ in range(5)]
    for y in ys[1:]:
        assert np.array_equal(ys[0].view(np.uint32), y.view(np.uint32))
    rt.activate([], [])


# ----------------------------------------------------------------- 8B-shape q8_0 block
@pytest.fixture(scope="module")
def block_q8():
    require_gpu()
    base = S.block_base(S.Q8_0)
    ad = S.block_adapter(base, adapter=0, rank=16)
    rt = make_runtime(base, arena_bytes=512 << 20)
    h = stage(rt, ad)
    st, _ = rt.activate([h], [2.0])
    assert st == 0
    return base, ad, rt


@pytest.mark.parametrize("proj", list(range(7)))
def test_block_q8_decode_bf16(block_q8, proj):
    base, ad, rt = block_q8
    t = base.tensors[proj]
    x = S.activations(1, t.d_in)
    xd, x64 = x_device(x, "bf16")
    y = fwd(rt, proj, xd)
    assert_within_bound(y, deq_of(base, proj), lora_terms([(ad, 2.0)], proj), x64, S.PROJ[proj])


# ----------------------------------------------------------------- q4_0 block, stacked adapters
@pytest.fixture(scope="module")
def block_q4():
    require_gpu()
    base = S.block_base(S.Q4_0)
    a16 = S.block_adapter(base, adapter=0, rank=16)
    a64 = S.block_adapter(base, adapter=1, rank=64)
    rt = make_runtime(base, arena_bytes=768 << 20)
    h16, h64 = stage(rt, a16), stage(rt, a64)
    st, _ = rt.activate([h16, h64], [1.0, 0.5])
    assert st == 0
    return base, a16, a64, rt


@pytest.mark.parametrize("T", [1, 4, 8])
@pytest.mark.parametrize("proj", [0, 1, 4, 6])
def test_block_q4_stacked(block_q4, proj, T):
    base, a16, a64, rt = block_q4
    t = base.tensors[proj]
    x = S.activations(T, t.d_in)
    xd, x64 = x_device(x, "bf16")
    y = fwd(rt, proj, xd)
    assert_within_bound(y, deq_of(base, proj), lora_terms([(a16, 1.0), (a64, 0.5)], proj), x64,
                        f"{S.PROJ[proj]} T={T}")


# ----------------------------------------------------------------- ragged / degenerate shapes
RAGGED = [  # (quant, d_out, d_in, T, ranks, xdtype)
    (S.Q8_0, 1, 32, 1, (), "f32"),
    (S.Q8_0, 3, 96, 2, (1,), "bf16"),
    (S.Q4_0, 1000, 288, 3, (5, 7), "f32"),
    (S.Q8_0, 1337, 1056, 5, (16,), "bf16"),
    (S.Q4_0, 77, 4128, 1, (3,), "bf16"),
    (S.Q8_0, 513, 8192, 8, (32, 2), "bf16"),
    (S.Q4_0, 257, 2048, 16, (4,), "f32"),
    (S.Q8_0, 4096, 256, 1, (128, 128), "f32"),
    (S.Q8_0, 512, 4096, 1, (64, 64), "f32"),      # long shrink chunks: the separate shrink launch
    (S.Q4_K, 100, 2048, 1, (96, 16), "bf16"),    # rank 112 on 100 CTAs: the separate shrink launch
    (S.Q8_0, 64, 20480, 1, (8,), "bf16"),        # rows too wide for 4-row stages; blocks past 16 warps in shared memory
    (S.Q4_0, 96, 20480, 1, (4,), "f32"),
]


@pytest.mark.parametrize("case", RAGGED, ids=[f"q{c[0]}_{c[1]}x{c[2]}_T{c[3]}_r{'-'.join(map(str, c[4]))}_{c[5]}"
                                             for c in RAGGED])
def test_ragged_shapes(case):
    require_gpu()
    quant, m, n, T, ranks, xdt = case
    rng = np.random.default_rng(m * 7 + n)
    W = S.gaussian(rng, (m, n), 0.02)
    base = S.build_base(quant, [(0, 0, W)])
    ads = []
    for k, r in enumerate(ranks):
        A = S.gaussian(rng, (r, n), 0.01)
        B = S.gaussian(rng, (m, r), 0.01)
        ads.append((S.build_adapter(base, [0], [r], [(A, B)]), [2.0, 0.5, 1.25][k % 3]))
    rt = make_runtime(base, arena_bytes=64 << 20)
    hs = [stage(rt, ad) for ad, _ in ads]
    assert rt.activate(hs, [s for _, s in ads])[0] == 0
    x = S.gaussian(rng, (T, n), 1.0)
    xd, x64 = x_device(x, xdt)
    y = fwd(rt, 0, xd)
    assert y.shape == (T, m)
    assert_within_bound(y, deq_of(base, 0), lora_terms(ads, 0), x64, str(case))
    rt.close()


def test_empty_token_batch_is_a_noop():
    require_gpu()
    import quantized_base_lora_gb300 as q
    base, ad_a, ad_b, x, s = S.single_layer_256()
    rt = make_runtime(base)
    y = torch.full((1, 256), 7.0, device="cuda")
    xd = torch.zeros((1, 256), device="cuda")
    st = q.ovl_linear_forward(rt.ctx, 0, xd.data_ptr(), q.OVL_F32, 0, y.data_ptr())
    torch.cuda.synchronize()
    assert st == 0 and bool((y == 7.0).all())
    rt.close()


def test_activation_scale_extremes_stay_within_bound():
    """Blocks whose activations span a wide dynamic range and all-zero blocks."""
    require_gpu()
    rng = np.random.default_rng(99)
    m, n = 64, 512
    W = S.gaussian(rng, (m, n), 0.02)
    base = S.build_base(S.Q8_0, [(0, 0, W)])
    rt = make_runtime(base)
    x = S.gaussian(rng, (4, n), 1.0)
    x[0, :32] = 0.0                                   # zero block
    x[1, 32:64] *= np.float32(1e-30)                  # tiny block
    x[2, 64:96] *= np.float32(1e20)                   # huge block
    x[3, ::7] *= np.float32(1e-6)                     # mixed magnitudes inside blocks
    x[3, 96:128] *= np.float32(1e-35)                 # below 2^-104: the block takes the fp32 route
    xd, x64 = x_device(x, "f32")
    y = fwd(rt, 0, xd)
    assert_within_bound(y, deq_of(base, 0), [], x64, "extremes")
    rt.close()


# ----------------------------------------------------------------- multi-tensor launches
@pytest.mark.parametrize("T", [1, 3, 4, 37])   # 4 and 37: one tensor-core launch over the group
def test_multi_tensor_launch_qkv_and_gate_up(block_q8, T):
    import quantized_base_lora_gb300 as q
    base, ad, rt = block_q8
    for group in ([0, 1, 2], [4, 5]):
        x = S.activations(T, 4096, seed=5000 + T)
        xd, x64 = x_device(x, "bf16")
        ys = [torch.full((T, base.tensors[i].d_out), float("nan"), device="cuda") for i in group]
        st = q.ovl_linear_forward_multi(rt.ctx, group, xd.data_ptr(), q.OVL_BF16, T, [y.data_ptr() for y in ys],
                                        int(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        assert st == 0 and rt.check_device() == 0
        for i, y in zip(group, ys):
            assert_within_bound(y.cpu().numpy(), deq_of(base, i), lora_terms([(ad, 2.0)], i), x64,
                                f"multi {S.PROJ[i]} T={T}")


def test_multi_tensor_launch_rejects_mixed_d_in(block_q8):
    import quantized_base_lora_gb300 as q
    base, ad, rt = block_q8
    xd = torch.zeros((1, 4096), device="cuda")
    ys = [torch.zeros((1, 4096), device="cuda") for _ in range(2)]
    st = q.ovl_linear_forward_multi(rt.ctx, [0, 6], xd.data_ptr(), q.OVL_F32, 1, [y.data_ptr() for y in ys])
    assert st == q.OVL_E_SHAPE
    st = q.ovl_linear_forward_multi(rt.ctx, [0, 1, 2, 3, 4], xd.data_ptr(), q.OVL_F32, 1, [ys[0].data_ptr()] * 5)
    assert st == q.OVL_E_ARG


# ----------------------------------------------------------------- tensor-core path (16+ tokens)
TC_CASES = [  # (quant, d_out, d_in, T, ranks, xdtype): token chunks of 64, ragged rows and tokens
    (S.Q8_0, 1000, 4096, 64, (16, 64), "bf16"),
    (S.Q8_0, 300, 2048, 512, (8,), "bf16"),
    (S.Q4_0, 777, 1024, 100, (5, 3), "f32"),
    (S.Q8_0, 129, 256, 16, (), "f32"),
    (S.Q4_0, 256, 512, 33, (64, 100), "bf16"),   # low-rank K-blocks over two pipeline stages
]


@pytest.mark.parametrize("case", TC_CASES, ids=[f"q{c[0]}_{c[1]}x{c[2]}_T{c[3]}_r{'-'.join(map(str, c[4]))}_{c[5]}"
                                                for c in TC_CASES])
def test_tensor_core_path(case):
    require_gpu()
    quant, m, n, T, ranks, xdt = case
    rng = np.random.default_rng(m + 31 * n + T)
    W = S.gaussian(rng, (m, n), 0.02)
    base = S.build_base(quant, [(0, 0, W)])
    ads = []
    for k, r in enumerate(ranks):
        A = S.gaussian(rng, (r, n), 0.01)
        B = S.gaussian(rng, (m, r), 0.01)
        ads.append((S.build_adapter(base, [0], [r], [(A, B)]), [2.0, 0.5][k % 2]))
    rt = make_runtime(base, arena_bytes=64 << 20)
    hs = [stage(rt, ad) for ad, _ in ads]
    assert rt.activate(hs, [s for _, s in ads])[0] == 0
    x = S.gaussian(rng, (T, n), 1.0)
    xd, x64 = x_device(x, xdt)
    y = fwd(rt, 0, xd)
    assert_within_bound(y, deq_of(base, 0), lora_terms(ads, 0), x64, str(case))
    y2 = fwd(rt, 0, xd)                                  # deterministic
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
    rt.close()


# ----------------------------------------------------------------- outliers on zero-weight columns
# A block whose largest activation meets a zero weight while its other
# activations are ~1e7 times smaller: sum_j |w_ij x_j| is made of the small
# elements only, so they must keep their own precision (the decode kernel
# takes such blocks through plain fp32).  Outlier columns vary inside the
# block; every other block carries no outlier, so marked and unmarked blocks
# meet in one launch.
OUTLIER_CASES = [  # (quant, d_out, d_in, T, ranks, xdtype)
    (S.Q8_0, 64, 32, 1, (), "f32"),
    (S.Q8_0, 64, 32, 2, (4,), "bf16"),
    (S.Q8_0, 300, 4096, 1, (16,), "bf16"),
    (S.Q8_0, 300, 4096, 1, (), "f32"),
    (S.Q8_0, 300, 4096, 2, (16,), "f32"),
    (S.Q8_0, 300, 4096, 3, (16,), "bf16"),
    (S.Q4_0, 200, 4096, 1, (8,), "bf16"),
    (S.Q4_0, 200, 4096, 3, (), "f32"),
    (S.Q8_0, 160, 14336, 1, (16,), "bf16"),      # two register records per lane
    (S.Q4_0, 96, 14336, 2, (), "f32"),
]


def outlier_layer(quant, m, n, T, ranks, seed):
    rng = np.random.default_rng(seed)
    W = S.gaussian(rng, (m, n), 0.02)
    cols = np.array([32 * b + (7 * b) % 32 for b in range(0, n // 32, 2)])
    W[:, cols] = 0.0                                 # code 0 (q8_0) / 8 (q4_0): weight exactly 0
    base = S.build_base(quant, [(0, 0, W)])
    ads = []
    for k, r in enumerate(ranks):
        A = S.gaussian(rng, (r, n), 0.01)
        B = S.gaussian(rng, (m, r), 0.01)
        ads.append((S.build_adapter(base, [0], [r], [(A, B)]), [2.0, 0.5][k % 2]))
    x = S.gaussian(rng, (T, n), 1.0) * np.float32(1e-3)
    sign = np.where(rng.standard_normal((T, cols.size)) < 0, -1.0, 1.0).astype(np.float32)
    x[:, cols] = np.float32(1e4) * sign
    return base, ads, x.astype(np.float32)


@pytest.mark.parametrize("case", OUTLIER_CASES,
                         ids=[f"q{c[0]}_{c[1]}x{c[2]}_T{c[3]}_r{'-'.join(map(str, c[4]))}_{c[5]}" for c in OUTLIER_CASES])
def test_outlier_on_zero_weight_stays_within_bound(case):
    require_gpu()
    quant, m, n, T, ranks, xdt = case
    base, ads, x = outlier_layer(quant, m, n, T, ranks, seed=m + n + T)
    rt = make_runtime(base, arena_bytes=64 << 20)
    hs = [stage(rt, ad) for ad, _ in ads]
    assert rt.activate(hs, [s for _, s in ads])[0] == 0
    xd, x64 = x_device(x, xdt)
    y = fwd(rt, 0, xd)
    assert_within_bound(y, deq_of(base, 0), lora_terms(ads, 0), x64, str(case))
    y2 = fwd(rt, 0, xd)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))   # deterministic
    rt.close()


def test_outlier_blocks_in_multi_tensor_launch(block_q8):
    """q+k+v in one launch, two blocks of x holding an outlier ~1e9 times
    their neighbours: every CTA of every tensor adds the marked blocks."""
    import quantized_base_lora_gb300 as q
    base, ad, rt = block_q8
    rng = np.random.default_rng(17)
    x = S.gaussian(rng, (1, 4096), 1.0) * np.float32(1e-4)
    x[0, 5] = np.float32(3e5)
    x[0, 4000] = np.float32(-2e6)
    xd, x64 = x_device(x, "bf16")
    group = [0, 1, 2]
    ys = [torch.full((1, base.tensors[i].d_out), float("nan"), device="cuda") for i in group]
    st = q.ovl_linear_forward_multi(rt.ctx, group, xd.data_ptr(), q.OVL_BF16, 1, [y.data_ptr() for y in ys],
                                    int(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0 and rt.check_device() == 0
    for i, y in zip(group, ys):
        assert_within_bound(y.cpu().numpy(), deq_of(base, i), lora_terms([(ad, 2.0)], i), x64, f"outlier {i}")


# ----------------------------------------------------------------- 128-token chunks (two MMA issuers, N = 128)
# Layers large enough to need no split-K (gate+up of the 8B block: 224 row
# tiles) take 128-token chunks when T >= 128: each dequantized weight feeds 128
# multiply-adds.  T = 200 is one full chunk and a ragged one of 72 tokens.
@pytest.mark.parametrize("quant", [S.Q8_0, S.Q4_0, S.Q4_K])
@pytest.mark.parametrize("T", [128, 200])
def test_wide_token_chunks_gate_up(quant, T):
    require_gpu()
    import quantized_base_lora_gb300 as q
    base = S.block_base(quant, projs=("gate", "up"))
    ad = S.block_adapter(base, adapter=0, rank=16)
    rt = make_runtime(base, arena_bytes=256 << 20)
    h = stage(rt, ad)
    assert rt.activate([h], [2.0])[0] == 0
    x = S.activations(T, 4096, seed=7000 + T)
    xd, x64 = x_device(x, "bf16")
    ys = [torch.full((T, t.d_out), float("nan"), device="cuda") for t in base.tensors]
    st = q.ovl_linear_forward_multi(rt.ctx, [0, 1], xd.data_ptr(), q.OVL_BF16, T, [y.data_ptr() for y in ys],
                                    int(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0 and rt.check_device() == 0
    rows = np.random.default_rng(T).choice(T, min(T, 24), replace=False)
    for i, y in enumerate(ys):
        got = y.cpu().numpy()
        assert np.isfinite(got).all()
        assert_within_bound(got[rows], deq_of(base, i), lora_terms([(ad, 2.0)], i), x64[rows], f"wide q{quant} {i} T={T}")
    # deterministic
    y0 = ys[0].clone()
    st = q.ovl_linear_forward_multi(rt.ctx, [0, 1], xd.data_ptr(), q.OVL_BF16, T, [y.data_ptr() for y in ys],
                                    int(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert torch.equal(y0, ys[0])
    rt.close()
