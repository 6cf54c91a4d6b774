"""GPU parity on the 32-layer stack of the 8B-shape q8_0 block (every layer
drawn from its own seeds, a rank-16 adapter with its own seeds on all 224
projections, s = 2.0), run the way the decode benchmark runs it: one decode
token through every layer as q+k+v, o, gate+up, down calls.  Sampled layers
are checked against the oracle on all seven projections; one deep layer's
projection is also run as a 512-token prefill on the per-layer JIT path."""
import numpy as np
import pytest

import synth as S
from gpu_common import assert_within_bound, deq_of, lora_terms, require_gpu, torch, x_device

pytestmark = pytest.mark.gpu

LAYERS = 32
SAMPLED = (0, 9, 22, 31)
GROUPS = [[0, 1, 2], [3], [4, 5], [6]]


@pytest.fixture(scope="module")
def stack32():
    require_gpu()
    import quantized_base_lora_gb300 as q
    from quantized_base_lora_gb300.runtime import Runtime
    from synth.stack import LayerStack, layer_stride, stack_adapter
    rt = Runtime(arena_bytes=256 << 20)
    buf = torch.empty(LAYERS * layer_stride(S.Q8_0), dtype=torch.uint8, device="cuda")

    def sink(layer, off, padded):
        buf[off:off + padded.nbytes].copy_(torch.from_numpy(padded))

    stack = LayerStack(S.Q8_0, LAYERS, sink)
    torch.cuda.synchronize()
    tensors = [(t.layer, t.proj, t.d_out, t.d_in, t.qs_off, t.d_off) for t in stack.tensors]
    assert q.ovl_load_base(rt.ctx, S.Q8_0, tensors, buf.data_ptr(), buf.numel(), stack.digest,
                           int(torch.cuda.current_stream().cuda_stream)) == 0, q.ovl_last_error(rt.ctx)
    rt.base, rt.tensors = buf, tensors
    ad = stack_adapter(stack, adapter=0, rank=16)
    st, h = rt.stage(ad, S.content_digest(ad.payload))
    assert st == 0, q.ovl_last_error(rt.ctx)
    assert rt.activate([h], [2.0])[0] == 0
    yield q, rt, stack, ad
    rt.close()


def test_decode_token_through_32_layers_matches_oracle(stack32):
    q, rt, stack, ad = stack32
    sh = int(torch.cuda.current_stream().cuda_stream)
    xs = {d: x_device(S.activations(1, d), "bf16") for d in (4096, 14336)}
    ys = [[torch.full((1, t.d_out), float("nan"), device="cuda") for t in stack.tensors[7 * l:7 * l + 7]]
          for l in range(LAYERS)]
    for l in range(LAYERS):
        for grp in GROUPS:
            xd = xs[stack.tensors[7 * l + grp[0]].d_in][0]
            if len(grp) == 1:
                st = q.ovl_linear_forward(rt.ctx, 7 * l + grp[0], xd.data_ptr(), q.OVL_BF16, 1,
                                          ys[l][grp[0]].data_ptr(), q.OVL_PATH_DUAL, 0, 0, sh)
            else:
                st = q.ovl_linear_forward_multi(rt.ctx, [7 * l + i for i in grp], xd.data_ptr(), q.OVL_BF16, 1,
                                                [ys[l][i].data_ptr() for i in grp], sh)
            assert st == 0, q.ovl_last_error(rt.ctx)
    torch.cuda.synchronize()
    assert rt.check_device() == 0
    for l in range(LAYERS):
        for y in ys[l]:
            assert bool(torch.isfinite(y).all()), f"layer {l}: unwritten output"
    for l in SAMPLED:
        one = S.block_base(S.Q8_0, layers=(l,))
        for i in range(7):
            t = one.tensors[i]
            A, B = ad.factors[7 * l + i]
            terms = [(A, B, 2.0)]
            assert_within_bound(ys[l][i].cpu().numpy(), deq_of(one, i), terms, xs[t.d_in][1],
                                f"layer {l} {S.PROJ[i]}")


def test_prefill_512_tokens_jit_on_a_deep_layer(stack32):
    """Layer 31's gate projection, T = 512, per-layer JIT (fp32 scratch, TF32
    tensor-core GEMM); 32 sampled tokens checked on every output."""
    q, rt, stack, ad = stack32
    l, i = 31, 4
    t = stack.tensors[7 * l + i]
    x = S.activations(512, t.d_in)
    xd, x64 = x_device(x, "bf16")
    need = (t.d_out * t.d_in * 4 + 127) // 128 * 128 + 512 * t.d_in * 4 + 256
    scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
    sp = (scratch.data_ptr() + 127) // 128 * 128
    y = torch.full((512, t.d_out), float("nan"), device="cuda")
    st = q.ovl_linear_forward(rt.ctx, 7 * l + i, xd.data_ptr(), q.OVL_BF16, 512, y.data_ptr(), q.OVL_PATH_JIT,
                              sp, need - (sp - scratch.data_ptr()), int(torch.cuda.current_stream().cuda_stream))
    assert st == 0, q.ovl_last_error(rt.ctx)
    torch.cuda.synchronize()
    assert rt.check_device() == 0
    one = S.block_base(S.Q8_0, layers=(l,))
    rows = np.random.default_rng(31).choice(512, 32, replace=False)
    A, B = ad.factors[7 * l + i]
    assert_within_bound(y.cpu().numpy()[rows], deq_of(one, i), [(A, B, 2.0)], x64[rows], "layer 31 gate T=512")
