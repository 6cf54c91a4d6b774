"""Activation state machine through the C ABI on a GPU: every failure leaves the
state unchanged, injected faults at each phase roll back, rollback is one
level deep, activation is idempotent, switches are refused while forward work
is in flight, and the switch transcript matches the oracle's model."""
import json
import os

import numpy as np
import pytest

import oracle as O
import synth as S
from gpu_common import adapter_tuples, make_runtime, require_gpu, stage, tensor_tuples, torch

pytestmark = pytest.mark.gpu


@pytest.fixture()
def env():
    require_gpu()
    import quantized_base_lora_gb300 as q
    base, ad_a, ad_b, x, s = S.single_layer_256()
    rt = make_runtime(base, arena_bytes=32 << 20)
    yield q, base, ad_a, ad_b, s, rt
    rt.close()


def snapshot(rt):
    st = rt.state()
    return (st["composition_id"], st["epoch"], st["n_staged"], st["arena_used"], st["has_previous"],
            st["n_entries"])


def test_staging_failures_change_nothing(env):
    q, base, ad_a, ad_b, s, rt = env
    A, B = ad_a.factors[0]
    before = snapshot(rt)
    d = S.content_digest(ad_a.payload)
    cases = []
    cases.append((q.OVL_E_HASH, dict(ad=ad_a, digest=bytes(32))))
    bad = A.copy()
    bad[3, 5] = np.nan
    nan_ad = S.build_adapter(base, [0], [8], [(bad, B)])
    cases.append((q.OVL_E_NONFINITE, dict(ad=nan_ad, digest=S.content_digest(nan_ad.payload))))
    inf_ad = S.build_adapter(base, [0], [8], [(A, np.where(B > 0.02, np.inf, B).astype(np.float32))])
    cases.append((q.OVL_E_NONFINITE, dict(ad=inf_ad, digest=S.content_digest(inf_ad.payload))))
    for code, kw in cases:
        st, h = rt.stage(kw["ad"], kw["digest"])
        assert (st, h) == (code, 0), q.ovl_last_error(rt.ctx)
        assert snapshot(rt) == before
    # descriptor errors
    P = ad_a.payload
    for code, targets, ranks, aoff, boff in [
        (q.OVL_E_NOTARGET, [1], [8], [0], [8192]),
        (q.OVL_E_DUPLICATE, [0, 0], [8, 8], [0, 0], [8192, 8192]),
        (q.OVL_E_SHAPE, [0], [0], [0], [8192]),
        (q.OVL_E_SHAPE, [0], [8], [4], [8192]),
        (q.OVL_E_SHAPE, [0], [8], [0], [P.nbytes - 16]),
        (q.OVL_E_SHAPE, [0], [200], [0], [8192]),
    ]:
        st, h = q.ovl_stage_adapter(rt.ctx, targets, ranks, aoff, boff, P, d)
        assert st == code, (code, q.ovl_last_error(rt.ctx))
        assert snapshot(rt) == before
    st, h = rt.stage(ad_a, d, required_base=b"\x01" * 32)
    assert st == q.OVL_E_HASH and snapshot(rt) == before
    st, h = rt.stage(ad_a, d, required_base=S.content_digest(base.buf))
    assert st == 0


def test_arena_budget_is_all_or_nothing():
    require_gpu()
    import quantized_base_lora_gb300 as q
    rng = np.random.default_rng(1)
    W = S.gaussian(rng, (2048, 2048), 0.02)
    base = S.build_base(S.Q8_0, [(0, 0, W)])
    rt = make_runtime(base, arena_bytes=16 << 20)            # ~7 MiB left after the workspace
    big = S.build_adapter(base, [0], [128], [(S.gaussian(rng, (128, 2048), 0.01),
                                              S.gaussian(rng, (2048, 128), 0.01))])   # 2 MiB
    hs = []
    while True:
        before = snapshot(rt)
        st, h = rt.stage(big, S.content_digest(big.payload))
        if st != 0:
            assert st == q.OVL_E_OOM and snapshot(rt) == before
            break
        hs.append(h)
    assert len(hs) >= 2
    assert rt.unstage(hs[-1]) == 0
    st, h = rt.stage(big, S.content_digest(big.payload))
    assert st == 0
    rt.close()


@pytest.mark.parametrize("phase", [1, 2, 3, 4])
def test_injected_stage_faults_roll_back(env, phase):
    q, base, ad_a, ad_b, s, rt = env
    before = snapshot(rt)
    assert q.ovl_debug_inject(rt.ctx, phase, q.OVL_E_CUDA) == 0
    st, h = rt.stage(ad_a, S.content_digest(ad_a.payload))
    assert st == q.OVL_E_CUDA and h == 0
    assert snapshot(rt) == before
    st, h = rt.stage(ad_a, S.content_digest(ad_a.payload))   # injection was one-shot
    assert st == 0


def test_injected_swap_faults_roll_back(env):
    q, base, ad_a, ad_b, s, rt = env
    ha = stage(rt, ad_a)
    before = snapshot(rt)
    for phase in (q.OVL_PHASE_VALIDATION, q.OVL_PHASE_SWAP):
        q.ovl_debug_inject(rt.ctx, phase, q.OVL_E_OOM)
        st, cid = rt.activate([ha], [s])
        assert st == q.OVL_E_OOM and snapshot(rt) == before
    st, cid = rt.activate([ha], [s])
    assert st == 0
    mid = snapshot(rt)
    q.ovl_debug_inject(rt.ctx, q.OVL_PHASE_SWAP, q.OVL_E_STATE)
    assert rt.rollback()[0] == q.OVL_E_STATE and snapshot(rt) == mid
    assert rt.rollback()[0] == 0 and snapshot(rt)[0] == before[0]


def test_activation_errors_and_idempotency(env):
    q, base, ad_a, ad_b, s, rt = env
    ha, hb = stage(rt, ad_a), stage(rt, ad_b)
    before = snapshot(rt)
    assert rt.activate([999], [1.0])[0] == q.OVL_E_ARG
    assert rt.activate([ha, ha], [1.0, 1.0])[0] == q.OVL_E_DUPLICATE
    assert rt.activate([ha], [float("nan")])[0] == q.OVL_E_ARG
    assert rt.activate([ha], [float("inf")])[0] == q.OVL_E_ARG
    assert rt.activate([ha], [1.0], mode=7)[0] == q.OVL_E_ARG
    assert snapshot(rt) == before
    st, ida = rt.activate([ha], [s])
    ep = rt.state()["epoch"]
    st2, ida2 = rt.activate([ha], [s])                      # same composition: no-op
    assert st2 == 0 and ida2 == ida and rt.state()["epoch"] == ep
    st, idab = rt.activate([ha, hb], [s, s])
    st, idba = rt.activate([hb, ha], [s, s])
    assert idab != idba                                      # order is part of the identity
    assert q.ovl_get_entry(rt.ctx, 0)[1]["handle"] == hb
    assert rt.unstage(ha) == q.OVL_E_STATE                    # active
    st, _ = rt.activate([], [])                               # deactivate
    assert rt.unstage(ha) == q.OVL_E_STATE                    # rollback target still holds it
    assert rt.rollback()[0] == 0 and rt.rollback()[0] == q.OVL_E_NO_PREVIOUS
    assert rt.activate([], [])[0] == 0
    assert rt.rollback()[0] == 0
    assert rt.activate([], [])[0] == 0


def test_switch_refused_while_forward_in_flight(env):
    q, base, ad_a, ad_b, s, rt = env
    ha = stage(rt, ad_a)
    xd = torch.randn(1, 256, device="cuda")
    rt.forward(0, xd)                  # first use loads the kernel (lazy module loading waits for the device)
    torch.cuda.synchronize()
    torch.cuda._sleep(400_000_000)                           # keeps the stream busy (~0.2 s)
    rt.forward(0, xd)
    before = snapshot(rt)
    st, _ = rt.activate([ha], [s])
    assert st == q.OVL_E_BUSY and snapshot(rt) == before
    torch.cuda.synchronize()
    assert rt.activate([ha], [s])[0] == 0


def test_drain_policy_waits():
    require_gpu()
    import quantized_base_lora_gb300 as q
    base, ad_a, ad_b, x, s = S.single_layer_256()
    rt = make_runtime(base, arena_bytes=32 << 20, policy=q.OVL_SWITCH_DRAIN)
    ha = stage(rt, ad_a)
    xd = torch.randn(1, 256, device="cuda")
    torch.cuda._sleep(200_000_000)
    rt.forward(0, xd)
    assert rt.activate([ha], [s])[0] == 0
    rt.close()


def test_base_load_errors():
    require_gpu()
    import quantized_base_lora_gb300 as q
    from quantized_base_lora_gb300.runtime import Runtime
    base, ad_a, ad_b, x, s = S.single_layer_256()
    tt = tensor_tuples(base)
    rt = Runtime(arena_bytes=32 << 20)
    assert rt.load_base(base.quant, tt, base.buf, bytes(32)) == q.OVL_E_HASH
    for unknown in (0, 4, 9):
        assert rt.load_base(unknown, tt, base.buf, S.content_digest(base.buf)) == q.OVL_E_QUANT
    bad = [(0, 0, 256, 256, 0, base.buf.nbytes)]
    assert rt.load_base(base.quant, bad, base.buf, S.content_digest(base.buf)) == q.OVL_E_SHAPE
    bad = [(0, 0, 256, 250, 0, 65536)]
    assert rt.load_base(base.quant, bad, base.buf, S.content_digest(base.buf)) == q.OVL_E_SHAPE
    assert rt.state()["base_loaded"] == 0
    assert rt.load_base(base.quant, tt, base.buf, S.content_digest(base.buf)) == 0
    assert rt.load_base(base.quant, tt, base.buf, S.content_digest(base.buf)) == q.OVL_E_STATE
    rt.close()


def test_table_composition_refuses_stack_forward(env):
    q, base, ad_a, ad_b, s, rt = env
    ha = stage(rt, ad_a)
    assert rt.activate([ha], [s], mode=q.OVL_MODE_TABLE)[0] == 0
    with pytest.raises(q.OvlError) as e:
        rt.forward(0, torch.zeros(1, 256, device="cuda"))
    assert e.value.status == q.OVL_E_STATE


def test_switch_transcript_matches_oracle():
    require_gpu()
    import quantized_base_lora_gb300 as q
    with open(os.path.join(os.path.dirname(__file__), "golden", "switch_transcript.json")) as f:
        g = json.load(f)
    base, _, _, x, s = S.single_layer_256()
    rt = make_runtime(base, arena_bytes=32 << 20)
    d0 = rt.base_digest()[1]
    ads = [S.block_adapter(base, adapter=a, rank=8) for a in range(4)]
    handles = {}
    for a, ad in enumerate(ads):
        dig = S.content_digest(ad.payload)
        if a == g["corrupt"]:
            dig = bytes([dig[0] ^ 0xFF]) + dig[1:]
        st, h = rt.stage(ad, dig)
        assert st == (q.OVL_E_HASH if a == g["corrupt"] else 0)
        handles[a] = h
    got = []
    for op, a in O.switch_sequence(g["n_ops"], 4, g["corrupt"]):
        if op == "activate":
            st, cid = rt.activate([handles[a]], [g["scale"]])
        elif op == "stage_corrupt":
            dig = S.content_digest(ads[a].payload)
            st, _ = rt.stage(ads[a], bytes([dig[0] ^ 0xFF]) + dig[1:])
            cid = rt.state()["composition_id"]
        else:
            st, cid = rt.rollback()
            if st != 0:
                cid = rt.state()["composition_id"]
        got.append([op, a, st, cid.hex()])
    assert got == g["transcript"]
    assert rt.base_digest()[1] == d0
    rt.close()


@pytest.mark.parametrize("multi", [False, True])
def test_device_wait_timeout_is_reported_and_recovers(env, multi):
    """A bounded device-side wait that runs out ([OVR] TDD and Fault-Injection
    Matrix): the injected launch withholds one CTA's low-rank partial sums and
    polls about a millisecond.  Its outputs come back NaN, the status check
    reports OVL_E_DEVICE_TIMEOUT once, the state is unchanged, and the next
    forward is exact again."""
    from gpu_common import assert_within_bound, deq_of, lora_terms, x_device
    q, base, ad_a, ad_b, s, rt = env
    x = S.single_layer_256()[3]
    ha = stage(rt, ad_a)
    assert rt.activate([ha], [s])[0] == 0
    xd, x64 = x_device(x, "f32")
    sh = int(torch.cuda.current_stream().cuda_stream)
    before = snapshot(rt)
    digest = rt.base_digest()[1]
    assert q.ovl_debug_inject(rt.ctx, q.OVL_PHASE_DEVICE_WAIT, q.OVL_E_CUDA) == q.OVL_E_ARG
    assert q.ovl_debug_inject(rt.ctx, q.OVL_PHASE_DEVICE_WAIT, q.OVL_E_DEVICE_TIMEOUT) == 0
    y = torch.zeros((1, 256), device="cuda")
    if multi:
        st = q.ovl_linear_forward_multi(rt.ctx, [0], xd.data_ptr(), q.OVL_F32, 1, [y.data_ptr()], sh)
    else:
        st = q.ovl_linear_forward(rt.ctx, 0, xd.data_ptr(), q.OVL_F32, 1, y.data_ptr(), q.OVL_PATH_DUAL, 0, 0, sh)
    assert st == 0
    torch.cuda.synchronize()
    assert bool(torch.isnan(y).all()), "outputs of a timed-out launch must be NaN"
    assert rt.check_device() == q.OVL_E_DEVICE_TIMEOUT
    assert rt.check_device() == 0                       # read and cleared
    assert snapshot(rt) == before and rt.base_digest()[1] == digest
    y2 = rt.forward(0, xd)
    torch.cuda.synchronize()
    assert rt.check_device() == 0
    terms = lora_terms([(ad_a, s)], 0)
    assert_within_bound(y2.cpu().numpy(), deq_of(base, 0), terms, x64, "after timeout")
    rt.activate([], [])
