"""GPU parity of the segmented multi-adapter batch (TABLE composition) against
the oracle: 64 decode requests over 16 rank-16 adapters drawn from Zipf(1.1) on
a q4_0 base (4096x4096 and 14336x4096), base-only segments, ragged token
counts, empty segments and argument errors."""
import numpy as np
import pytest

import oracle as O
import synth as S
from gpu_common import deq_of, make_runtime, require_gpu, stage, torch, x_device

pytestmark = pytest.mark.gpu


def seg_forward(rt, tensor, xd, offsets, slots, perm):
    import quantized_base_lora_gb300 as q
    T = xd.shape[0]
    d_out = rt.tensors[tensor][2] if tensor < len(rt.tensors) else 16
    y = torch.full((T, d_out), float("nan"), device="cuda")
    st = q.ovl_segmented_forward(rt.ctx, tensor, xd.data_ptr(), q.OVL_BF16 if xd.dtype == torch.bfloat16 else q.OVL_F32,
                                 T, list(offsets), list(slots), list(perm), y.data_ptr(),
                                 int(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, y.cpu().numpy()


def check(y, base, i, table, x64, slot_of_token, label):
    deq = deq_of(base, i)
    ref = O.segmented(deq, table, x64, slot_of_token)
    # per-token bound with that token's effective weight
    for t in range(x64.shape[0]):
        sl = slot_of_token[t]
        Wp = O.effective_weight(deq, [table[sl]] if sl >= 0 else [])
        bound = O.error_bound(Wp, x64[t:t + 1])[0]
        err = np.abs(y[t].astype(np.float64) - ref[t])
        assert (err <= bound).all(), f"{label}: token {t} slot {sl} max err/bound {(err / bound).max():.3g}"


@pytest.fixture(scope="module")
def serving():
    require_gpu()
    import quantized_base_lora_gb300 as q
    base = S.block_base(S.Q4_0, projs=("q", "gate"))
    ads = [S.block_adapter(base, adapter=a, rank=16) for a in range(16)]
    rt = make_runtime(base, arena_bytes=256 << 20)
    hs = [stage(rt, a) for a in ads]
    assert rt.activate(hs, [2.0] * 16, mode=q.OVL_MODE_TABLE)[0] == 0
    return base, ads, rt


def table_terms(ads, i, s=2.0):
    return [(ad.factors[ad.targets.index(i)][0], ad.factors[ad.targets.index(i)][1], s) for ad in ads]


@pytest.mark.parametrize("proj", [0, 1])
def test_zipf_batch_of_64(serving, proj):
    base, ads, rt = serving
    ids = S.zipf_ids(64, 16, 1.1)
    perm, offsets, slots = S.segments(ids)
    x = S.activations(64, base.tensors[proj].d_in, seed=4000 + proj)
    xd, x64 = x_device(x, "bf16")
    st, y = seg_forward(rt, proj, xd, offsets, slots, perm)
    assert st == 0 and rt.check_device() == 0
    check(y, base, proj, table_terms(ads, proj), x64, ids, f"zipf proj {proj}")


def test_base_only_and_empty_segments(serving):
    base, ads, rt = serving
    T = 13
    rng = np.random.default_rng(77)
    x = S.gaussian(rng, (T, 4096), 1.0)
    xd, x64 = x_device(x, "f32")
    # segments: [0,4) slot 3, [4,4) slot 5 (empty), [4,9) base only, [9,13) slot 15; rows permuted
    perm = rng.permutation(T).astype(np.int32)
    offsets, slots = [0, 4, 4, 9, 13], [3, 5, -1, 15]
    slot_of = np.empty(T, dtype=np.int64)
    for s in range(4):
        slot_of[perm[offsets[s]:offsets[s + 1]]] = slots[s]
    st, y = seg_forward(rt, 0, xd, offsets, slots, perm)
    assert st == 0
    check(y, base, 0, table_terms(ads, 0), x64, slot_of, "mixed segments")


def test_segment_argument_errors(serving):
    import quantized_base_lora_gb300 as q
    base, ads, rt = serving
    xd = torch.zeros((4, 4096), device="cuda")
    assert seg_forward(rt, 0, xd, [0, 4], [0], [0, 1, 2, 2])[0] == q.OVL_E_ARG      # not a permutation
    assert seg_forward(rt, 0, xd, [0, 3], [0], [0, 1, 2, 3])[0] == q.OVL_E_ARG      # offsets do not reach T
    assert seg_forward(rt, 0, xd, [0, 2, 1, 4], [0, 0, 0], [0, 1, 2, 3])[0] == q.OVL_E_ARG   # decreasing
    assert seg_forward(rt, 0, xd, [0, 4], [16], [0, 1, 2, 3])[0] == q.OVL_E_ARG     # slot out of range
    assert seg_forward(rt, 9, xd, [0, 4], [0], [0, 1, 2, 3])[0] == q.OVL_E_ARG      # no such tensor


def test_segmented_needs_table_composition():
    require_gpu()
    import quantized_base_lora_gb300 as q
    base, ad_a, ad_b, x, s = S.single_layer_256()
    rt = make_runtime(base, arena_bytes=32 << 20)
    xd = torch.zeros((2, 256), device="cuda")
    assert seg_forward(rt, 0, xd, [0, 2], [0], [0, 1])[0] == q.OVL_E_STATE
    rt.close()
