"""Activating compositions from manifests ([OVR] Composition Identity and
Manifest Schema; [DTD] §11): adapters found among the staged ones by their
content digest and applied in load order with their merge weights, the same
composition id and outputs as ovl_activate with that list, and every
mismatch against the context rejected with the state unchanged."""
import json

import numpy as np
import pytest

import oracle as O
import synth as S
from gpu_common import assert_within_bound, deq_of, make_runtime, require_gpu, stage, torch, x_device

pytestmark = pytest.mark.gpu


def h(b: bytes) -> str:
    return "sha256:" + b.hex()


@pytest.fixture()
def env():
    require_gpu()
    import quantized_base_lora_gb300 as q
    base, ad_a, ad_b, x, s = S.single_layer_256()
    rng = np.random.default_rng(8)
    sp = S.build_sparse_adapter([0], [S.dare_entries(rng, 256, 256, keep=0.02)])
    rt = make_runtime(base, arena_bytes=64 << 20)
    ha = stage(rt, ad_a)
    st, hs = rt.stage_sparse(sp, S.content_digest(sp.payload))
    assert st == 0, q.ovl_last_error(rt.ctx)
    yield q, base, ad_a, ad_b, sp, x, rt, ha, hs
    rt.close()


def manifest(base, entries, **over):
    d = {"base_model_hash": h(S.content_digest(base.buf)), "quantization": "q8_0",
         "runtime": {"name": "ovl-gb300", "version": "v1"}, "adapters": entries}
    d.update(over)
    return json.dumps(d)


def snapshot(rt):
    st = rt.state()
    return (st["composition_id"], st["epoch"], st["n_entries"], st["has_previous"])


def test_two_entry_manifest_matches_ovl_activate_and_the_oracle(env):
    q, base, ad_a, ad_b, sp, x, rt, ha, hs = env
    # the sparse overlay is listed first in the document but loads second
    text = manifest(base, [
        {"name": "dare", "file_hash": h(S.content_digest(sp.payload)), "load_order": 20, "merge_weight": 0.75,
         "type": "sparse", "targets": [0]},
        {"name": "lora-a", "file_hash": h(S.content_digest(ad_a.payload)), "load_order": 10, "merge_weight": 2.0,
         "rank": 8, "targets": [0], "required_base_hash": h(S.content_digest(base.buf))}])
    st, cid = q.ovl_activate_manifest(rt.ctx, text)
    assert st == 0, q.ovl_last_error(rt.ctx)
    xd, x64 = x_device(x, "f32")
    y = rt.forward(0, xd)
    torch.cuda.synchronize()
    assert rt.check_device() == 0
    # the same list through ovl_activate in a fresh context: same id, same bits
    rt2 = make_runtime(base, arena_bytes=64 << 20)
    ha2 = stage(rt2, ad_a)
    st, hs2 = rt2.stage_sparse(sp, S.content_digest(sp.payload))
    st, cid2 = rt2.activate([ha2, hs2], [2.0, 0.75])
    assert st == 0 and cid2 == cid
    y2 = rt2.forward(0, xd)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    rt2.close()
    # and the oracle: LoRA then the sparse delta, in load order
    A, B = ad_a.factors[0]
    idx, val = sp.entries[0]
    terms = [(A, B, 2.0), O.SparseTerm(idx, val, float(np.float32(0.75)))]
    assert_within_bound(y.cpu().numpy(), deq_of(base, 0), terms, x64, "manifest composition")
    # activating the same manifest again is the idempotent no-op
    ep = rt.state()["epoch"]
    assert q.ovl_activate_manifest(rt.ctx, text) == (0, cid) and rt.state()["epoch"] == ep


def test_context_mismatches_change_nothing(env):
    q, base, ad_a, ad_b, sp, x, rt, ha, hs = env
    good_a = {"name": "lora-a", "file_hash": h(S.content_digest(ad_a.payload)), "load_order": 1, "merge_weight": 2.0}
    assert rt.activate([ha], [2.0])[0] == 0
    before = snapshot(rt)
    cases = [
        (manifest(base, [good_a], base_model_hash="sha256:" + "00" * 32), q.OVL_E_HASH),
        (manifest(base, [good_a], quantization="q4_0"), q.OVL_E_QUANT),
        (manifest(base, [dict(good_a, file_hash=h(S.content_digest(ad_b.payload)))]), q.OVL_E_HASH),   # not staged
        (manifest(base, [dict(good_a, type="sparse")]), q.OVL_E_ARG),
        (manifest(base, [dict(good_a, rank=16)]), q.OVL_E_SHAPE),
        (manifest(base, [dict(good_a, targets=[1])]), q.OVL_E_SHAPE),
        (manifest(base, [dict(good_a, required_base_hash="sha256:" + "11" * 32)]), q.OVL_E_HASH),
        (manifest(base, [good_a, dict(good_a, name="again")]), q.OVL_E_DUPLICATE),
        (manifest(base, [good_a], runtime={"name": "ovl-gb300", "version": "v0"}), q.OVL_E_ARG),
        ("{not json", q.OVL_E_ARG),
    ]
    for text, code in cases:
        st, _ = q.ovl_activate_manifest(rt.ctx, text)
        assert st == code, (text, st, q.ovl_last_error(rt.ctx))
        assert q.ovl_last_error(rt.ctx)
        assert snapshot(rt) == before
    # an empty adapter list is the base-only composition; rollback restores the previous one
    st, cid = q.ovl_activate_manifest(rt.ctx, manifest(base, []))
    assert st == 0 and rt.state()["n_entries"] == 0
    assert rt.rollback()[1] == before[0]
