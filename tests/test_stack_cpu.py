"""The 32-layer stack generator (input generation for the 32-layer decode
workload), checked on small shapes on the CPU: every layer is the seeded layer
block_base builds on its own, at its stride, and the declared digest is the
content digest of the concatenated padded layers."""
import numpy as np

import oracle as O
import synth as S
from synth.stack import LayerStack, layer_stride, stack_adapter

SMALL = {"q": (64, 64), "k": (32, 64), "v": (32, 64), "o": (64, 64), "gate": (96, 64), "up": (96, 64),
         "down": (64, 96)}


def test_stack_layers_have_their_own_seeds_and_digest():
    n_layers = 3
    stride = layer_stride(S.Q8_0, SMALL)
    assert stride % 65536 == 0
    buf = np.zeros(n_layers * stride, dtype=np.uint8)

    def sink(layer, off, padded):
        buf[off:off + padded.nbytes] = padded

    st = LayerStack(S.Q8_0, n_layers, sink, workers=2, shapes=SMALL)
    assert st.digest == O.tree_digest(buf)
    assert len(st.tensors) == 7 * n_layers
    for l in range(n_layers):
        one = S.block_base(S.Q8_0, layers=(l,), shapes=SMALL)
        assert np.array_equal(buf[l * stride:l * stride + one.buf.nbytes], one.buf)
        for i, t in enumerate(one.tensors):
            u = st.tensors[7 * l + i]
            assert (u.layer, u.proj, u.d_out, u.d_in) == (l, t.proj, t.d_out, t.d_in)
            assert (u.qs_off, u.d_off) == (l * stride + t.qs_off, l * stride + t.d_off)
    # distinct layers differ (own seeds)
    assert not np.array_equal(buf[:stride], buf[stride:2 * stride])
    ad = stack_adapter(st, adapter=0, rank=4)
    assert ad.targets == list(range(7 * n_layers))
    A, B = ad.factors[7 + 2]                       # layer 1, v
    rng = np.random.default_rng(S.adapter_seed(0, 1, 2))
    assert np.array_equal(A, S.gaussian(rng, (4, 64), 0.01)) and np.array_equal(B, S.gaussian(rng, (32, 4), 0.01))
