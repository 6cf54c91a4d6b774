"""Writes the golden fixtures of this folder.

Inputs come from the seeded generators in ``synth``; every stored expected
value is computed by ``oracle`` alone.  Re-run after a change to either that
is justified by the pages:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402
import synth as S   # noqa: E402


def base_tensor_tuples(base):
    return [(t.layer, t.proj, t.d_out, t.d_in, t.qs_off, t.d_off) for t in base.tensors]


def adapter_target_tuples(ad):
    return list(zip(ad.targets, ad.ranks, ad.a_off, ad.b_off))


def config1():
    base, ad_a, ad_b, x, s = S.single_layer_256()
    qs, d = base.planes[0]
    deq = O.dequantize_q8_0(qs, d)
    out = {"base_digest": O.tree_digest(base.buf).hex(), "y": {}, "ids": {}}
    bkey = O.base_key(O.tree_digest(base.buf), base.quant, base_tensor_tuples(base))
    for name, ad in (("base", None), ("A", ad_a), ("B", ad_b)):
        ads = [] if ad is None else [(ad.factors[0][0], ad.factors[0][1], s)]
        out["y"][name] = [float(v).hex() for v in O.dual_path(deq, ads, x)[0]]
        ent = [] if ad is None else [(O.adapter_key(O.tree_digest(ad.payload), adapter_target_tuples(ad)), s)]
        out["ids"][name] = O.composition_id(bkey, O.MODE_STACK, ent).hex()
    return out


def switch():
    base, ad_a, ad_b, x, s = S.single_layer_256()
    bkey = O.base_key(O.tree_digest(base.buf), base.quant, base_tensor_tuples(base))
    keys = []
    for a in range(4):
        ad = S.block_adapter(base, adapter=a, rank=8)
        keys.append(O.adapter_key(O.tree_digest(ad.payload), adapter_target_tuples(ad)))
    tr = O.switch_transcript(bkey, keys, 2.0, 100, 3)
    return {"base_key": bkey.hex(), "adapter_keys": [k.hex() for k in keys], "scale": 2.0,
            "n_ops": 100, "corrupt": 3, "transcript": [list(t) for t in tr]}


if __name__ == "__main__":
    with open(os.path.join(HERE, "config1.json"), "w") as f:
        json.dump(config1(), f, indent=1)
    with open(os.path.join(HERE, "switch_transcript.json"), "w") as f:
        json.dump(switch(), f, indent=0)
    print("written")
