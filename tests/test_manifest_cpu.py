"""Composition manifests parsed by the library on the CPU (no device):
the fields the pages name ([OVR] Composition Identity and Manifest Schema;
[DTD] §11 AdapterManifestV0), adapters ordered by load_order, and
deterministic rejection of malformed documents ([OVR] TDD and Fault-Injection
Matrix: invalid JSON, missing fields, wrong hashes)."""
import json

import numpy as np
import pytest

q = pytest.importorskip("quantized_base_lora_gb300")

H = {k: "sha256:" + v * 32 for k, v in (("base", "ab"), ("a", "01"), ("b", "02"), ("c", "03"))}


def doc(**over):
    d = {"base_model_hash": H["base"], "quantization": "q8_0",
         "adapters": [{"name": "medical", "file_hash": H["a"], "load_order": 2, "merge_weight": 1.0},
                      {"name": "safety", "file_hash": H["b"], "load_order": 1, "merge_weight": 0.5, "type": "lora",
                       "rank": 16, "required_base_hash": H["base"], "targets": [0, 3, 6]}]}
    d.update(over)
    return d


def parse(d):
    text = d if isinstance(d, (str, bytes)) else json.dumps(d)
    return q.ovl_manifest_parse(text)


def test_fields_and_load_order():
    st, m = parse(doc(runtime={"name": "ovl-gb300", "version": "v1"}, tokenizer_id="tok", mode="table",
                      timestamp_utc="2026-07-21T00:00:00Z"))
    assert st == q.OVL_OK
    assert m["base_digest"] == bytes.fromhex("ab" * 32)
    assert m["quant"] == q.OVL_Q8_0 and m["mode"] == q.OVL_MODE_TABLE
    names = [a["name"] for a in m["adapters"]]
    assert names == ["safety", "medical"]                       # increasing load_order
    s, med = m["adapters"]
    assert s["file_digest"] == bytes.fromhex("02" * 32) and s["rank"] == 16 and s["n_targets"] == 3
    assert s["required_base_digest"] == bytes.fromhex("ab" * 32) and s["merge_weight"] == 0.5
    assert med["type"] == q.OVL_ADAPTER_LORA and med["rank"] == 0 and med["required_base_digest"] is None


@pytest.mark.parametrize("quant,code", [("q8_0", 1), ("q4_0", 2), ("q4_K", 3)])
def test_quantization_profiles(quant, code):
    st, m = parse(doc(quantization=quant))
    assert st == q.OVL_OK and m["quant"] == code


def test_merge_weight_is_rounded_to_binary32_and_base_only_is_empty():
    st, m = parse(doc(adapters=[{"name": "x", "file_hash": H["c"], "load_order": 7, "merge_weight": 0.1,
                                 "type": "sparse"}]))
    assert st == q.OVL_OK and m["adapters"][0]["merge_weight"] == float(np.float32(0.1))
    assert m["adapters"][0]["type"] == q.OVL_ADAPTER_SPARSE
    st, m = parse(doc(adapters=[]))
    assert st == q.OVL_OK and m["adapters"] == [] and m["mode"] == q.OVL_MODE_STACK


MALFORMED = [
    ("", "empty"),
    ("{", "truncated"),
    ("[]", "not an object"),
    ('{"base_model_hash": "x",}', "trailing comma"),
    ("{'base_model_hash': 1}", "single quotes"),
    ('{"a": NaN}', "NaN literal"),
    ('{"a": 1} // note', "comment"),
    ('{"a": 01}', "leading zero"),
    ('{"a": 1} {"b": 2}', "two documents"),
    ('{"a": "\\x"}', "bad escape"),
    ('{"a": "\\ud800"}', "lone surrogate"),
    ('{"a": "tab\there"}', "raw control character"),
    ('{"a": 1, "a": 2}', "duplicate key"),
    ("[" * 40 + "]" * 40, "too deep"),
]


@pytest.mark.parametrize("text,why", MALFORMED, ids=[w for _, w in MALFORMED])
def test_malformed_json_is_rejected(text, why):
    st, m = parse(text)
    assert st == q.OVL_E_ARG and m is None, why
    assert q.ovl_last_error(None)


def drop(d, key):
    d = dict(d)
    d.pop(key)
    return d


def adapter_with(i, **over):
    d = doc()
    d["adapters"] = [dict(a) for a in d["adapters"]]
    d["adapters"][i].update(over)
    return d


def adapter_without(i, key):
    d = doc()
    d["adapters"] = [dict(a) for a in d["adapters"]]
    d["adapters"][i].pop(key)
    return d


SCHEMA = [
    (drop(doc(), "base_model_hash"), q.OVL_E_ARG, "no base hash"),
    (drop(doc(), "quantization"), q.OVL_E_ARG, "no quantization"),
    (drop(doc(), "adapters"), q.OVL_E_ARG, "no adapters"),
    (doc(base_model_hash="ab" * 32), q.OVL_E_ARG, "hash without prefix"),
    (doc(base_model_hash="sha256:" + "ab" * 31), q.OVL_E_ARG, "short hash"),
    (doc(base_model_hash="sha256:" + "AB" * 32), q.OVL_E_ARG, "uppercase hex"),
    (doc(base_model_hash="sha256:" + "zz" * 32), q.OVL_E_ARG, "not hex"),
    (doc(quantization="q4_1"), q.OVL_E_QUANT, "unknown quantization"),
    (doc(quantization=8), q.OVL_E_ARG, "quantization not a string"),
    (doc(mode="merged"), q.OVL_E_ARG, "unknown mode"),
    (doc(runtime={"name": "ovl-gb300", "version": "v2"}), q.OVL_E_ARG, "runtime version skew"),
    (doc(runtime={"name": "other", "version": "v1"}), q.OVL_E_ARG, "other runtime"),
    (doc(runtime={"name": "ovl-gb300"}), q.OVL_E_ARG, "runtime without version"),
    (doc(signature="..."), q.OVL_E_ARG, "unknown field"),
    (doc(adapters={}), q.OVL_E_ARG, "adapters not an array"),
    (doc(adapters=[1]), q.OVL_E_ARG, "adapter not an object"),
    (adapter_without(0, "name"), q.OVL_E_ARG, "no name"),
    (adapter_without(0, "file_hash"), q.OVL_E_ARG, "no file hash"),
    (adapter_without(0, "load_order"), q.OVL_E_ARG, "no load order"),
    (adapter_without(0, "merge_weight"), q.OVL_E_ARG, "no merge weight"),
    (adapter_with(0, name=""), q.OVL_E_ARG, "empty name"),
    (adapter_with(0, name="n" * 64), q.OVL_E_ARG, "long name"),
    (adapter_with(0, type="ia3"), q.OVL_E_ARG, "unknown adapter type"),
    (adapter_with(0, load_order=0), q.OVL_E_ARG, "load order 0"),
    (adapter_with(0, load_order=1.5), q.OVL_E_ARG, "fractional load order"),
    (adapter_with(0, load_order=2 ** 31), q.OVL_E_ARG, "load order too large"),
    (adapter_with(0, load_order=1), q.OVL_E_ARG, "ambiguous order"),
    (adapter_with(0, merge_weight="1.0"), q.OVL_E_ARG, "weight as a string"),
    (adapter_with(0, merge_weight=1e39), q.OVL_E_ARG, "weight overflows binary32"),
    (adapter_with(0, rank=0), q.OVL_E_ARG, "rank 0"),
    (adapter_with(0, rank=129), q.OVL_E_ARG, "rank above the limit"),
    (adapter_with(0, type="sparse", rank=4), q.OVL_E_ARG, "rank on a sparse overlay"),
    (adapter_with(0, targets=[-1]), q.OVL_E_ARG, "negative target"),
    (adapter_with(0, targets=3), q.OVL_E_ARG, "targets not an array"),
    (adapter_with(0, required_base_hash="sha256:"), q.OVL_E_ARG, "bad required base hash"),
    (adapter_with(0, scale=2.0), q.OVL_E_ARG, "unknown adapter field"),
    (adapter_with(0, name="safety"), q.OVL_E_DUPLICATE, "name twice"),
    (adapter_with(0, file_hash=H["b"]), q.OVL_E_DUPLICATE, "file hash twice"),
    (doc(adapters=[{"name": f"n{i}", "file_hash": "sha256:" + f"{i:064x}", "load_order": i + 1, "merge_weight": 1}
                   for i in range(33)]), q.OVL_E_ARG, "more than OVL_MAX_TABLE adapters"),
]


@pytest.mark.parametrize("d,code,why", SCHEMA, ids=[w for _, _, w in SCHEMA])
def test_schema_violations_are_rejected(d, code, why):
    st, m = parse(d)
    assert st == code and m is None, why
    assert q.ovl_last_error(None)


def test_rejection_is_deterministic():
    d = adapter_with(0, load_order=1)
    outs = {(parse(d)[0], q.ovl_last_error(None)) for _ in range(3)}
    assert len(outs) == 1
