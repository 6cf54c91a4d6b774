"""The C ABI on the CPU: the library loads, exports every symbol the header
declares, and its host-side SHA-256 / content digest agree with independent
implementations.  No GPU needed (no compute call touches a device)."""
import ctypes
import hashlib
import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ovl():
    lib_path = os.path.join(ROOT, "quantized_base_lora_gb300", "libovl.so")
    if not os.path.exists(lib_path):
        import importlib.util
        spec = importlib.util.spec_from_file_location(
            "qbl_build", os.path.join(ROOT, "quantized_base_lora_gb300", "build.py"))
        m = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(m)
        m.build()
    import quantized_base_lora_gb300 as q
    return q


def header_symbols():
    with open(os.path.join(ROOT, "include", "ovl.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ovl_[a-z0-9_]+)\s*\(", text)))


def test_every_entry_point_cites_its_passage_or_says_it_has_none():
    """The comment block directly above each declaration cites the passage that
    defines the operation, or states that the pages define no counterpart."""
    with open(os.path.join(ROOT, "include", "ovl.h")) as f:
        text = f.read()
    decls = list(re.finditer(r"\n(?:ovl_status|const char\*) (ovl_\w+)\(", text))
    assert len(decls) >= 20
    for i, m in enumerate(decls):
        # the doc comment: the last /* ... */ that ends before this declaration
        # and after the previous one
        lo = decls[i - 1].end() if i else 0
        head = text[lo:m.start()]
        blocks = re.findall(r"/\*.*?\*/", head, flags=re.S)
        assert blocks, m.group(1)
        doc = blocks[-1]
        assert any(t in doc for t in ("[OVR]", "[DTD]", "[MODELD]", "FIPS")) or "no counterpart" in doc.lower(), \
            m.group(1)


def test_every_declared_symbol_is_exported(ovl):
    syms = header_symbols()
    assert len(syms) >= 19
    lib = ctypes.CDLL(ovl.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), f"missing export {s}"
    assert set(syms) == set(ovl.EXPORTED)


def test_version(ovl):
    assert "sm_103a" in ovl.ovl_version()


@pytest.mark.parametrize("msg", [b"abc", b"", b"abcdbcdecdefdefgefghfghighijhijkijkljklmklmnlmnomnopnopq"])
def test_sha256_fips_vectors(ovl, msg):
    assert ovl.ovl_sha256(msg) == hashlib.sha256(msg).digest()


def test_sha256_padding_boundaries(ovl):
    rng = np.random.default_rng(0)
    for n in [1, 55, 56, 57, 63, 64, 65, 119, 120, 127, 128, 1000, 4096]:
        data = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
        assert ovl.ovl_sha256(data) == hashlib.sha256(data).digest(), n


@pytest.mark.parametrize("size", [0, 1, 65535, 65536, 65537, 5 * 65536 + 3, 3 << 20])
def test_content_digest_matches_oracle(ovl, size):
    buf = np.random.default_rng(size).integers(0, 256, size, dtype=np.uint8)
    assert ovl.ovl_content_digest(buf) == O.tree_digest(buf)


def test_create_rejects_bad_arguments_without_a_device(ovl):
    st, ctx = ovl.ovl_create(0, 0, 1 << 30)
    assert st == ovl.OVL_E_ARG and not ctx.value
    assert "arena" in ovl.ovl_last_error(None)
    st, ctx = ovl.ovl_create(0, 4096 + 3, 1 << 30)
    assert st == ovl.OVL_E_ARG
    st, ctx = ovl.ovl_create(0, 1 << 20, 1 << 20)
    assert st == ovl.OVL_E_ARG


def test_null_context_is_rejected(ovl):
    assert ovl.lib.ovl_destroy(None) == ovl.OVL_OK
    assert ovl.ovl_debug_inject(None, 1, -2) == ovl.OVL_E_ARG
    assert ovl.ovl_rollback(None)[0] == ovl.OVL_E_ARG


def test_status_codes_match_the_oracles_restatement(ovl):
    for name in ["OVL_OK", "OVL_E_ARG", "OVL_E_HASH", "OVL_E_SHAPE", "OVL_E_QUANT", "OVL_E_OOM",
                 "OVL_E_NONFINITE", "OVL_E_DUPLICATE", "OVL_E_NOTARGET", "OVL_E_BUSY",
                 "OVL_E_NO_PREVIOUS", "OVL_E_STATE"]:
        assert getattr(ovl, name) == getattr(O, name)
    with open(os.path.join(ROOT, "include", "ovl.h")) as f:
        text = f.read()
    for name, val in re.findall(r"\b(OVL_E_[A-Z_]+)\s*=\s*(-?\d+)", text):
        assert getattr(ovl, name) == int(val)
