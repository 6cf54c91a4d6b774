"""Planted mistakes in the oracle (on the CPU, through monkeypatch): each
plausible slip - a swapped nibble, a wrong offset or block index, a dropped
scale, a transposed operand, a swapped field, a wrong sign - must make at least
one of the independent pins in test_oracle_pins.py fail.  This checks the pins,
not the oracle: with no mistake planted every pin passes (that file's own run).
The golden-file pins are left out here, since they were written by the oracle."""
import numpy as np
import pytest

import oracle
import oracle.ovl_oracle as M
import test_oracle_pins as P


def plant(monkeypatch, name, fn):
    monkeypatch.setattr(M, name, fn)
    monkeypatch.setattr(oracle, name, fn, raising=False)


def caught(*pins) -> list:
    """Names of the pins that fail under the planted mistake."""
    out = []
    for pin in pins:
        try:
            pin()
        except Exception:    # an AssertionError, or a crash on the bad shapes
            out.append(pin.__name__)
    return out


F16 = M.f16_to_float
Q4_CODES = M.q4_0_codes
DEQ_Q8 = M.dequantize_q8_0
DEQ_Q4 = M.dequantize_q4_0
DEQ_Q4K = M.dequantize_q4_k
FIELDS_Q4K = M.q4_k_header_fields
EFF = M.effective_weight
DUAL = M.dual_path
SPARSE_DELTA = M.sparse_delta


def test_f16_subnormal_exponent_off_by_one(monkeypatch):
    def bad(bits):
        b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
        e = (b >> 10) & 0x1F
        v = F16(bits)
        return np.where(e == 0, 2.0 * v, v)
    plant(monkeypatch, "f16_to_float", bad)
    assert caught(P.test_f16_decode_exhaustive_vs_numpy)


def test_q4_0_nibbles_swapped(monkeypatch):
    def bad(packed):
        c = Q4_CODES(packed)
        out = c.copy()
        out[:, 0::2], out[:, 1::2] = c[:, 1::2], c[:, 0::2]
        return out
    plant(monkeypatch, "q4_0_codes", bad)
    assert caught(P.test_q4_0_nibble_order_hand_built, P.test_q4_0_dequant_every_scale_every_code)


def test_q4_0_offset_7(monkeypatch):
    plant(monkeypatch, "dequantize_q4_0", lambda p, d: DEQ_Q4(p, d) + np.repeat(
        F16(d).reshape(np.asarray(p).shape[0], -1), 32, axis=1))
    assert caught(P.test_q4_0_dequant_every_scale_every_code, P.test_q4_0_nibble_order_hand_built)


def test_q8_0_scale_of_the_wrong_block(monkeypatch):
    def bad(qs, d_bits):
        qs = np.asarray(qs).view(np.int8)
        m, n = qs.shape
        d = F16(d_bits).reshape(m, n // 32)
        d = np.roll(d, 1, axis=1)            # block b scaled by the scale of block b - 1
        return np.repeat(d, 32, axis=1) * qs.astype(np.float64)
    plant(monkeypatch, "dequantize_q8_0", bad)
    assert caught(P.test_quantizer_round_trip_through_oracle_dequant, P.test_base_gemv_exact_rationals)


def test_lora_scale_dropped(monkeypatch):
    def bad_eff(deq, adapters):
        return EFF(deq, [(a[0], a[1], 1.0) if isinstance(a, tuple) else a for a in adapters])

    def bad_dual(deq, adapters, x):
        return DUAL(deq, [(a[0], a[1], 1.0) if isinstance(a, tuple) else a for a in adapters], x)
    plant(monkeypatch, "effective_weight", bad_eff)
    plant(monkeypatch, "dual_path", bad_dual)
    assert caught(P.test_unit_outer_product_moves_one_weight_by_s, P.test_dual_equals_merged_exact_rationals)


def test_lora_factors_transposed_in_the_expand(monkeypatch):
    def bad(deq, adapters, x):
        x = np.asarray(x, np.float64)
        y = x @ np.asarray(deq, np.float64).T
        for A, B, s in adapters:
            v = x @ np.asarray(A, np.float64).T
            Bt = np.asarray(B, np.float64)
            # B read as [r][m] row-major from its [m][r] buffer
            y = y + float(s) * (v @ Bt.reshape(Bt.shape[1], Bt.shape[0]))
        return y
    plant(monkeypatch, "dual_path", bad)
    assert caught(P.test_dual_equals_merged_exact_rationals, P.test_unit_outer_product_moves_one_weight_by_s)


def test_lora_term_sign_flipped(monkeypatch):
    plant(monkeypatch, "effective_weight",
          lambda deq, ads: 2 * np.asarray(deq, np.float64) - EFF(deq, ads))
    assert caught(P.test_unit_outer_product_moves_one_weight_by_s, P.test_dual_equals_merged_exact_rationals)


def test_q4_k_scale_and_minimum_swapped(monkeypatch):
    def bad(hdr):
        d, dmin, sc, mn = FIELDS_Q4K(hdr)
        return d, dmin, mn, sc
    plant(monkeypatch, "q4_k_header_fields", bad)
    assert caught(P.test_q4_k_header_every_value_in_every_slot, P.test_q4_k_sub_block_staircase_hand_evaluated)


def test_q4_k_minimum_added(monkeypatch):
    def bad(packed, hdr):
        w = DEQ_Q4K(packed, hdr)
        m, n = w.shape
        _, dmin, _, mn = FIELDS_Q4K(np.asarray(hdr, np.uint8).reshape(m, n // 256, 16))
        return w + 2 * np.repeat((dmin[..., None] * mn).reshape(m, n // 32), 32, axis=1)
    plant(monkeypatch, "dequantize_q4_k", bad)
    assert caught(P.test_q4_k_reduces_to_q4_0, P.test_q4_k_sub_block_staircase_hand_evaluated)


def test_q4_k_sub_blocks_reversed(monkeypatch):
    def bad(hdr):
        d, dmin, sc, mn = FIELDS_Q4K(hdr)
        return d, dmin, sc[..., ::-1], mn[..., ::-1]
    plant(monkeypatch, "q4_k_header_fields", bad)
    assert caught(P.test_q4_k_header_every_value_in_every_slot, P.test_q4_k_sub_block_staircase_hand_evaluated)


def test_sparse_index_read_column_major(monkeypatch):
    def bad(term, m, n):
        D = np.zeros(m * n, dtype=np.float64)
        idx = np.asarray(term.idx, np.int64)
        D[(idx % m) * n + idx // m] = F16(term.val_bits)
        return D.reshape(m, n)
    plant(monkeypatch, "sparse_delta", bad)
    assert caught(P.test_sparse_index_is_row_major_flat)


def test_sparse_scale_dropped(monkeypatch):
    def bad(deq, adapters, x):
        return DUAL(deq, [M.SparseTerm(a.idx, a.val_bits, 1.0) if isinstance(a, M.SparseTerm) else a
                          for a in adapters], x)
    plant(monkeypatch, "dual_path", bad)
    assert caught(P.test_sparse_single_entry_moves_exactly_one_weight, P.test_sparse_dual_path_exact_rationals)


def test_composition_id_ignores_the_scale(monkeypatch):
    CID = M.composition_id
    plant(monkeypatch, "composition_id", lambda bk, mode, entries: CID(bk, mode, [(k, 1.0) for k, _ in entries]))
    assert caught(P.test_composition_id_invariants)


def test_base_key_offsets_packed_as_u32(monkeypatch):
    import hashlib
    import struct

    def bad(digest, quant, tensors):
        tensors = list(tensors)
        h = hashlib.sha256(b"OVLB" + digest + struct.pack("<II", quant, len(tensors)))
        for t in tensors:
            h.update(struct.pack("<IIIIII", *[v & 0xFFFFFFFF for v in t]))
        return h.digest()
    plant(monkeypatch, "base_key", bad)
    assert caught(P.test_base_key_field_by_field)


def test_adapter_key_rank_and_tensor_swapped(monkeypatch):
    AK = M.adapter_key
    plant(monkeypatch, "adapter_key", lambda dg, targets: AK(dg, [(r, ti, ao, bo) for ti, r, ao, bo in targets]))
    assert caught(P.test_adapter_key_field_by_field)


def test_composition_id_without_the_runtime_tag(monkeypatch):
    monkeypatch.setattr(M, "RUNTIME_TAG", b"")
    assert caught(P.test_composition_id_field_by_field)


def test_tree_digest_hashes_the_whole_buffer_once(monkeypatch):
    import hashlib
    plant(monkeypatch, "tree_digest", lambda buf, leaf=M.LEAF: hashlib.sha256(
        hashlib.sha256(bytes(memoryview(buf).cast("B"))).digest()).digest())
    assert caught(P.test_tree_digest_multi_leaf_closed_forms)


@pytest.mark.parametrize("pin", [P.test_q4_0_nibble_order_hand_built, P.test_unit_outer_product_moves_one_weight_by_s,
                                 P.test_q4_k_sub_block_staircase_hand_evaluated,
                                 P.test_sparse_single_entry_moves_exactly_one_weight,
                                 P.test_base_key_field_by_field, P.test_adapter_key_field_by_field,
                                 P.test_composition_id_field_by_field, P.test_tree_digest_multi_leaf_closed_forms])
def test_pins_pass_without_a_planted_mistake(pin):
    assert not caught(pin)
