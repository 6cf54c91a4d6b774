"""GPU parity of sparse (DARE-style index-value) overlays against the fp64
oracle, through the C ABI: sparse-only and mixed low-rank + sparse stacks on
the dual path (single-token and multi-token routes, multi-tensor launches),
the JIT path (materialization and GEMM), q4_K and q8_0 bases, staging
validation (every failure changes nothing), identities, and reversibility."""
import numpy as np
import pytest

import oracle as O
import synth as S
from gpu_common import (assert_within_bound, deq_of, lora_terms, make_runtime, require_gpu, stage, tensor_tuples,
                        torch, x_device)

pytestmark = pytest.mark.gpu


def stage_sparse(rt, sp):
    import quantized_base_lora_gb300 as q
    st, h = rt.stage_sparse(sp, S.content_digest(sp.payload))
    assert st == 0, q.ovl_last_error(rt.ctx)
    return h


def sparse_terms(sp, s, tensor_index):
    if tensor_index not in sp.targets:
        return []
    idx, val = sp.entries[sp.targets.index(tensor_index)]
    return [O.SparseTerm(idx, val, float(np.float32(s)))]


def fwd(rt, i, xd, **kw):
    y = rt.forward(i, xd, **kw)
    torch.cuda.synchronize()
    assert rt.check_device() == 0
    return y.cpu().numpy()


CASES = [  # quant, m, n, T, lora ranks, keep, xdtype
    (S.Q8_0, 1, 32, 1, (), 0.5, "f32"),
    (S.Q8_0, 300, 512, 1, (), 0.01, "bf16"),
    (S.Q4_0, 1000, 288, 3, (5,), 0.03, "f32"),
    (S.Q8_0, 513, 2048, 5, (16,), 0.02, "bf16"),       # tensor-core route + sparse
    (S.Q4_K, 640, 1024, 2, (8,), 0.05, "bf16"),
    (S.Q8_0, 256, 4096, 37, (), 0.002, "bf16"),
    (S.Q4_0, 130, 256, 1, (), 1.0, "f32"),             # every weight has a pair
]


@pytest.mark.parametrize("case", CASES, ids=[f"q{c[0]}_{c[1]}x{c[2]}_T{c[3]}_r{'-'.join(map(str, c[4]))}_k{c[5]}"
                                             for c in CASES])
def test_sparse_dual_path_vs_oracle(case):
    require_gpu()
    quant, m, n, T, ranks, keep, xdt = case
    rng = np.random.default_rng(m * 13 + n + T)
    base = S.build_base(quant, [(0, 0, S.gaussian(rng, (m, n), 0.02))])
    rt = make_runtime(base, arena_bytes=64 << 20)
    handles, scales, terms = [], [], []
    for r in ranks:
        ad = S.build_adapter(base, [0], [r], [(S.gaussian(rng, (r, n), 0.01), S.gaussian(rng, (m, r), 0.01))])
        handles.append(stage(rt, ad))
        scales.append(2.0)
        terms += lora_terms([(ad, 2.0)], 0)
    sp = S.build_sparse_adapter([0], [S.dare_entries(rng, m, n, keep)])
    handles.append(stage_sparse(rt, sp))
    scales.append(0.5)
    terms += sparse_terms(sp, 0.5, 0)
    assert rt.activate(handles, scales)[0] == 0
    xd, x64 = x_device(S.gaussian(rng, (T, n), 1.0), xdt)
    y = fwd(rt, 0, xd)
    assert y.shape == (T, m)
    assert_within_bound(y, deq_of(base, 0), terms, x64, str(case))
    rt.close()


def test_sparse_before_lora_order_and_ids():
    require_gpu()
    rng = np.random.default_rng(51)
    m, n = 384, 1024
    base = S.build_base(S.Q8_0, [(0, 0, S.gaussian(rng, (m, n), 0.02))])
    ad = S.build_adapter(base, [0], [16], [(S.gaussian(rng, (16, n), 0.01), S.gaussian(rng, (m, 16), 0.01))])
    sp = S.build_sparse_adapter([0], [S.dare_entries(rng, m, n, 0.02)])
    rt = make_runtime(base, arena_bytes=64 << 20)
    ha, hs = stage(rt, ad), stage_sparse(rt, sp)
    xd, x64 = x_device(S.gaussian(rng, (1, n), 1.0), "bf16")
    st1, id1 = rt.activate([ha, hs], [2.0, 1.0])
    y1 = fwd(rt, 0, xd)
    st2, id2 = rt.activate([hs, ha], [1.0, 2.0])
    y2 = fwd(rt, 0, xd)
    assert st1 == st2 == 0 and id1 != id2
    terms = lora_terms([(ad, 2.0)], 0) + sparse_terms(sp, 1.0, 0)
    assert_within_bound(y1, deq_of(base, 0), terms, x64, "lora,sparse")
    assert_within_bound(y2, deq_of(base, 0), terms[::-1], x64, "sparse,lora")
    # identities against the oracle's byte strings
    bkey = O.base_key(S.content_digest(base.buf), base.quant, tensor_tuples(base))
    akey = O.adapter_key(S.content_digest(ad.payload), [(0, 16, ad.a_off[0], ad.b_off[0])])
    skey = O.sparse_adapter_key(S.content_digest(sp.payload), [(0, sp.nnz[0], sp.idx_off[0], sp.val_off[0])])
    assert id1 == O.composition_id(bkey, O.MODE_STACK, [(akey, 2.0), (skey, 1.0)])
    assert id2 == O.composition_id(bkey, O.MODE_STACK, [(skey, 1.0), (akey, 2.0)])
    rt.close()


def test_zero_valued_sparse_overlay_gives_base_output_exactly_and_base_is_untouched():
    require_gpu()
    rng = np.random.default_rng(53)
    m, n = 500, 768
    base = S.build_base(S.Q4_0, [(0, 0, S.gaussian(rng, (m, n), 0.02))])
    idx, _ = S.dare_entries(rng, m, n, 0.05)
    sp0 = S.build_sparse_adapter([0], [(idx, np.zeros(idx.size, np.uint16))])
    sp1 = S.build_sparse_adapter([0], [S.dare_entries(rng, m, n, 0.05)])
    rt = make_runtime(base, arena_bytes=64 << 20)
    d0 = rt.base_digest()[1]
    h0, h1 = stage_sparse(rt, sp0), stage_sparse(rt, sp1)
    xd, x64 = x_device(S.gaussian(rng, (3, n), 1.0), "f32")
    y_base = fwd(rt, 0, xd)
    assert rt.activate([h0], [3.0])[0] == 0
    y_zero = fwd(rt, 0, xd)
    assert np.array_equal(y_base.view(np.uint32), y_zero.view(np.uint32))
    # base -> sparse -> base: the base output comes back bit for bit
    assert rt.activate([h1], [1.0])[0] == 0
    fwd(rt, 0, xd)
    assert rt.activate([], [])[0] == 0
    assert np.array_equal(fwd(rt, 0, xd).view(np.uint32), y_base.view(np.uint32))
    assert rt.base_digest()[1] == d0
    rt.close()


def test_sparse_with_multi_tensor_launches():
    require_gpu()
    import quantized_base_lora_gb300 as q
    base = S.block_base(S.Q8_0, projs=("q", "k", "v"))
    ad = S.block_adapter(base, adapter=0, rank=16)
    sp = S.block_sparse_adapter(base, adapter=0, keep=0.01)
    rt = make_runtime(base, arena_bytes=256 << 20)
    assert rt.activate([stage(rt, ad), stage_sparse(rt, sp)], [2.0, 1.0])[0] == 0
    for T in (1, 4):
        xd, x64 = x_device(S.activations(T, 4096, seed=90 + T), "bf16")
        ys = [torch.full((T, t.d_out), float("nan"), device="cuda") for t in base.tensors]
        st = q.ovl_linear_forward_multi(rt.ctx, [0, 1, 2], xd.data_ptr(), q.OVL_BF16, T, [y.data_ptr() for y in ys],
                                        int(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        assert st == 0 and rt.check_device() == 0
        for i, y in enumerate(ys):
            terms = lora_terms([(ad, 2.0)], i) + sparse_terms(sp, 1.0, i)
            assert_within_bound(y.cpu().numpy(), deq_of(base, i), terms, x64, f"multi tensor {i} T={T}")
    rt.close()


def test_sparse_block_q4k_decode():
    require_gpu()
    base = S.block_base(S.Q4_K, projs=("q", "down"))
    ad = S.block_adapter(base, adapter=0, rank=16)
    sp = S.block_sparse_adapter(base, adapter=1, keep=0.01)
    rt = make_runtime(base, arena_bytes=256 << 20)
    assert rt.activate([stage(rt, ad), stage_sparse(rt, sp)], [2.0, 1.0])[0] == 0
    for i, t in enumerate(base.tensors):
        xd, x64 = x_device(S.activations(1, t.d_in), "bf16")
        y = fwd(rt, i, xd)
        assert_within_bound(y, deq_of(base, i), lora_terms([(ad, 2.0)], i) + sparse_terms(sp, 1.0, i), x64,
                            f"tensor {i}")
    rt.close()


def test_sparse_materialize_is_rounded_exact_and_jit_forward_within_bound():
    require_gpu()
    import quantized_base_lora_gb300 as q
    rng = np.random.default_rng(57)
    m, n, T = 320, 1024, 96
    base = S.build_base(S.Q8_0, [(0, 0, S.gaussian(rng, (m, n), 0.02))])
    sp = S.build_sparse_adapter([0], [S.dare_entries(rng, m, n, 0.03)])
    rt = make_runtime(base, arena_bytes=64 << 20)
    hs = stage_sparse(rt, sp)
    assert rt.activate([hs], [0.75])[0] == 0
    S_dev = torch.empty((m, n), dtype=torch.float32, device="cuda")
    q.check(q.ovl_materialize_layer(rt.ctx, 0, S_dev.data_ptr(), S_dev.numel() * 4,
                                    int(torch.cuda.current_stream().cuda_stream)), rt.ctx)
    torch.cuda.synchronize()
    # fp32 d*q is exact and one fused multiply-add rounds deq + s*v once
    want = O.effective_weight(deq_of(base, 0), sparse_terms(sp, 0.75, 0)).astype(np.float32)
    assert np.array_equal(S_dev.cpu().numpy().view(np.uint32), want.view(np.uint32))
    # JIT forward with a low-rank term in front of the sparse one
    ad = S.build_adapter(base, [0], [16], [(S.gaussian(rng, (16, n), 0.01), S.gaussian(rng, (m, 16), 0.01))])
    assert rt.activate([stage(rt, ad), hs], [2.0, 0.75])[0] == 0
    xd, x64 = x_device(S.gaussian(rng, (T, n), 1.0), "bf16")
    scratch = torch.empty((m * n * 4 + 127) // 128 * 128 + T * n * 4 + 256, dtype=torch.uint8, device="cuda")
    y = fwd(rt, 0, xd, path=q.OVL_PATH_JIT, scratch=scratch)
    assert_within_bound(y, deq_of(base, 0), lora_terms([(ad, 2.0)], 0) + sparse_terms(sp, 0.75, 0), x64, "jit")
    rt.close()


def test_sparse_staging_failures_change_nothing():
    require_gpu()
    import quantized_base_lora_gb300 as q
    rng = np.random.default_rng(59)
    m, n = 64, 256
    base = S.build_base(S.Q8_0, [(0, 0, S.gaussian(rng, (m, n), 0.02)), (0, 1, S.gaussian(rng, (m, n), 0.02))])
    rt = make_runtime(base, arena_bytes=32 << 20)
    before = rt.state()
    idx, val = S.dare_entries(rng, m, n, 0.1)

    def attempt(sp, digest=None, required=None):
        st, h = rt.stage_sparse(sp, digest or S.content_digest(sp.payload), required)
        assert h == 0
        after = rt.state()
        assert (after["arena_used"], after["n_staged"], after["composition_id"]) == \
            (before["arena_used"], before["n_staged"], before["composition_id"])
        return st

    swapped = idx.copy()
    swapped[[3, 4]] = swapped[[4, 3]]
    assert attempt(S.build_sparse_adapter([0], [(swapped, val)])) == q.OVL_E_SHAPE          # not increasing
    dup = idx.copy()
    dup[5] = dup[4]
    assert attempt(S.build_sparse_adapter([0], [(dup, val)])) == q.OVL_E_SHAPE              # repeated index
    big = idx.copy()
    big[-1] = m * n
    assert attempt(S.build_sparse_adapter([0], [(big, val)])) == q.OVL_E_SHAPE              # beyond the tensor
    nan = val.copy()
    nan[7] = 0x7E00
    assert attempt(S.build_sparse_adapter([0], [(idx, nan)])) == q.OVL_E_NONFINITE
    inf = val.copy()
    inf[0] = 0xFC00
    assert attempt(S.build_sparse_adapter([0], [(idx, inf)])) == q.OVL_E_NONFINITE
    good = S.build_sparse_adapter([0], [(idx, val)])
    assert attempt(good, digest=bytes(32)) == q.OVL_E_HASH
    assert attempt(good, required=bytes([1] * 32)) == q.OVL_E_HASH
    assert attempt(S.build_sparse_adapter([0, 0], [(idx, val), (idx, val)])) == q.OVL_E_DUPLICATE
    assert attempt(S.build_sparse_adapter([5], [(idx, val)])) == q.OVL_E_NOTARGET
    for phase in (q.OVL_PHASE_VALIDATION, q.OVL_PHASE_ALLOCATION, q.OVL_PHASE_STAGING, q.OVL_PHASE_CHECKSUM):
        assert q.ovl_debug_inject(rt.ctx, phase, q.OVL_E_CUDA) == 0
        assert attempt(good) == q.OVL_E_CUDA
    # an empty target is allowed and adds nothing
    h = stage_sparse(rt, S.build_sparse_adapter([1], [(np.zeros(0, np.uint32), np.zeros(0, np.uint16))]))
    assert rt.activate([h], [1.0])[0] == 0
    rt.close()


def test_sparse_overlay_refused_in_table_composition():
    require_gpu()
    import quantized_base_lora_gb300 as q
    rng = np.random.default_rng(61)
    base = S.build_base(S.Q8_0, [(0, 0, S.gaussian(rng, (64, 256), 0.02))])
    rt = make_runtime(base, arena_bytes=32 << 20)
    hs = stage_sparse(rt, S.build_sparse_adapter([0], [S.dare_entries(rng, 64, 256, 0.1)]))
    ad = S.build_adapter(base, [0], [4], [(S.gaussian(rng, (4, 256), 0.01), S.gaussian(rng, (64, 4), 0.01))])
    ha = stage(rt, ad)
    before = rt.state()["composition_id"]
    assert rt.activate([ha, hs], [1.0, 1.0], mode=q.OVL_MODE_TABLE)[0] == q.OVL_E_ARG
    assert rt.state()["composition_id"] == before
    assert rt.activate([hs], [1.0])[0] == 0
    st, e = q.ovl_get_entry(rt.ctx, 0)
    assert st == 0 and e["total_rank"] == 0
    rt.close()
