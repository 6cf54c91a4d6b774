"""Pins of the CPU oracle against facts that do not come from the oracle itself:
library decoders, exact rational arithmetic, closed forms, published SHA-256
test vectors and the invariants the pages state.  CPU only."""
import hashlib
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import synth as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- binary16
def test_f16_decode_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.f16_to_float(bits)
    lib = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(lib)
    assert fin.sum() == 63488
    assert np.array_equal(ours[fin], lib[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(lib[fin]))     # -0 kept
    assert np.array_equal(np.isinf(ours), np.isinf(lib))
    assert np.array_equal(np.isnan(ours), np.isnan(lib))


def _finite_f16_bits():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return bits[((bits >> 10) & 0x1F) != 31]


# ---------------------------------------------------------------- dequant
def test_q8_0_dequant_every_scale_every_code():
    d = _finite_f16_bits()                                   # 63488 scales
    codes = np.arange(-128, 128, dtype=np.int16).astype(np.int8)   # all 256 codes
    qs = np.tile(codes, (d.size, 1))                         # [63488][256]: 8 blocks/row
    dq = np.repeat(d[:, None], 256 // 32, axis=1)            # same scale in every block
    ours = O.dequantize_q8_0(qs, dq)
    want = d.view(np.float16).astype(np.float64)[:, None] * codes.astype(np.float64)[None, :]
    assert np.array_equal(ours, want)                        # 11 x 8 bits: exact in fp64


def test_q4_0_dequant_every_scale_every_code():
    d = _finite_f16_bits()
    codes = np.arange(16, dtype=np.uint8)
    row = np.tile(codes, 2)                                  # 32 codes = one block
    packed = (row[0::2] | (row[1::2] << 4)).astype(np.uint8)
    qs = np.tile(packed, (d.size, 1))                        # [63488][16]
    ours = O.dequantize_q4_0(qs, d[:, None])
    want = d.view(np.float16).astype(np.float64)[:, None] * (row.astype(np.float64) - 8.0)[None, :]
    assert np.array_equal(ours, want)


def test_dequant_exact_rationals_sample():
    rng = np.random.default_rng(7)
    d = rng.choice(_finite_f16_bits(), size=400)
    q = rng.integers(-128, 128, size=(400, 32)).astype(np.int8)
    ours = O.dequantize_q8_0(q, d[:, None])
    for i in range(0, 400, 7):
        dv = Fraction(float(d[i:i + 1].view(np.float16)[0]))
        for j in range(0, 32, 5):
            assert Fraction(float(ours[i, j])) == dv * int(q[i, j])


def test_q4_0_nibble_order_hand_built():
    # byte 0 = 0x21 -> element 0 has code 1, element 1 has code 2; byte 1 = 0xF0 -> codes 0, 15
    packed = np.zeros((1, 16), dtype=np.uint8)
    packed[0, 0] = 0x21
    packed[0, 1] = 0xF0
    packed[0, 2:] = 0x88                                     # code 8 -> value 0
    d = np.array([[0x3C00]], dtype=np.uint16)                # 1.0
    w = O.dequantize_q4_0(packed, d)[0]
    assert list(w[:4]) == [-7.0, -6.0, -8.0, 7.0]
    assert not w[4:].any()


def test_quantizer_round_trip_through_oracle_dequant():
    rng = np.random.default_rng(3)
    m, n = 16, 128
    q = rng.integers(-127, 128, size=(m, n)).astype(np.int8)
    q[:, ::32] = 127                                          # max |q| = 127 in every block
    d16 = (rng.uniform(1e-4, 1e-2, size=(m, n // 32))).astype(np.float16)
    w = O.dequantize_q8_0(q, d16.view(np.uint16)).astype(np.float32)
    q2, d2 = S.quantize_q8_0(w)
    assert np.array_equal(q2, q)
    assert np.array_equal(d2, d16.view(np.uint16))


def test_quantizer_q4_round_trip_through_oracle_dequant():
    rng = np.random.default_rng(4)
    m, n = 8, 64
    c = rng.integers(0, 16, size=(m, n)).astype(np.uint8)
    c[:, ::32] = 0                                            # value -8d: |w| max = 8d
    d16 = (rng.uniform(1e-3, 1e-1, size=(m, n // 32))).astype(np.float16)
    packed = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    w = O.dequantize_q4_0(packed, d16.view(np.uint16)).astype(np.float32)
    p2, d2 = S.quantize_q4_0(w)
    assert np.array_equal(d2, d16.view(np.uint16))
    assert np.array_equal(p2, packed)


# ---------------------------------------------------------------- q4_K
def _hdr_bitwise(d_bits: int, dmin_bits: int, sc, mn) -> np.ndarray:
    """One 16-byte q4_K header built bit by bit (independent of any packer):
    value j of a 6-bit field sets bits 6j..6j+5 of its six bytes, LSB first."""
    out = [d_bits & 0xFF, d_bits >> 8, dmin_bits & 0xFF, dmin_bits >> 8] + [0] * 12
    for base, vals in ((4, sc), (10, mn)):
        for j, v in enumerate(vals):
            for b in range(6):
                if (int(v) >> b) & 1:
                    pos = 6 * j + b
                    out[base + pos // 8] |= 1 << (pos % 8)
    return np.array(out, dtype=np.uint8)


def test_q4_k_header_every_value_in_every_slot():
    hdrs, want = [], []
    for j in range(8):
        for v in range(64):
            sc = [0] * 8
            mn = [0] * 8
            sc[j] = v
            mn[7 - j] = 63 - v
            hdrs.append(_hdr_bitwise(0x3C00, 0x4000, sc, mn))
            want.append((sc, mn))
    d, dmin, sc, mn = O.q4_k_header_fields(np.stack(hdrs))
    assert np.all(d == 1.0) and np.all(dmin == 2.0)
    assert np.array_equal(sc, np.array([w[0] for w in want]))
    assert np.array_equal(mn, np.array([w[1] for w in want]))


def test_q4_k_header_random_vs_bit_string():
    rng = np.random.default_rng(11)
    h = rng.integers(0, 256, size=(300, 16)).astype(np.uint8)
    _, _, sc, mn = O.q4_k_header_fields(h)
    for i in range(300):
        for base, got in ((4, sc[i]), (10, mn[i])):
            # bit string, least significant bit of byte `base` first
            bits = "".join(format(int(b), "08b")[::-1] for b in h[i, base:base + 6])
            vals = [int(bits[6 * j:6 * j + 6][::-1], 2) for j in range(8)]
            assert list(got) == vals


def test_q4_k_reduces_to_q4_0():
    # sc_j = 1, m_j = 8 and dmin = d give d*code - 8d = d*(code - 8): q4_0 exactly
    rng = np.random.default_rng(12)
    m, n = 9, 512
    packed = rng.integers(0, 256, size=(m, n // 2)).astype(np.uint8)
    dfin = _finite_f16_bits()
    dbits = rng.choice(dfin, size=(m, n // 256))
    hdr = np.stack([np.stack([_hdr_bitwise(int(dbits[i, k]), int(dbits[i, k]), [1] * 8, [8] * 8)
                              for k in range(n // 256)]) for i in range(m)])
    d32 = np.repeat(dbits, 8, axis=1)                         # the same d for every 32-block
    assert np.array_equal(O.dequantize_q4_k(packed, hdr), O.dequantize_q4_0(packed, d32))


def test_q4_k_sub_block_staircase_hand_evaluated():
    # d = 1, dmin = 0.5, sc_j = j + 1, m_j = 2j, every code 3:
    # sub-block j of every super-block holds 3(j + 1) - j = 2j + 3
    hdr = _hdr_bitwise(0x3C00, 0x3800, [j + 1 for j in range(8)], [2 * j for j in range(8)])
    packed = np.full((1, 256), 0x33, dtype=np.uint8)          # two super-blocks
    w = O.dequantize_q4_k(packed, np.stack([hdr, hdr])[None])[0]
    want = np.repeat(np.array([2 * j + 3 for j in range(8)] * 2, dtype=np.float64), 32)
    assert np.array_equal(w, want)
    # nibble order inside a sub-block: byte 0 = 0x51 -> element 0 code 1, element 1 code 5
    packed[0, 0] = 0x51
    w = O.dequantize_q4_k(packed, np.stack([hdr, hdr])[None])[0]
    assert w[0] == 1.0 and w[1] == 5.0 and w[2] == 3.0


def test_q4_k_exact_rationals_every_scale_min_code():
    rng = np.random.default_rng(13)
    dfin = _finite_f16_bits()
    rows = []
    want = []
    for sc in range(64):
        d_bits, dm_bits = int(rng.choice(dfin)), int(rng.choice(dfin))
        dv = Fraction(float(np.array([d_bits], np.uint16).view(np.float16)[0]))
        dmv = Fraction(float(np.array([dm_bits], np.uint16).view(np.float16)[0]))
        mins = [(sc + 8 * j) % 64 for j in range(8)]          # every m over the 64 rows x 8 slots
        hdr = _hdr_bitwise(d_bits, dm_bits, [sc] * 8, mins)
        codes = np.tile(np.arange(16, dtype=np.uint8), 16)     # every code in every sub-block
        rows.append((codes[0::2] | (codes[1::2] << 4), hdr))
        want.append([dv * sc * int(codes[c]) - dmv * mins[c // 32] for c in range(256)])
    packed = np.stack([r[0] for r in rows])
    hdr = np.stack([r[1] for r in rows])[:, None, :]
    w = O.dequantize_q4_k(packed, hdr)
    for i in range(64):
        assert [Fraction(float(v)) for v in w[i]] == want[i]


def test_q4_k_is_4_5_bits_per_weight():
    m, n = 3, 1024
    qs, hdr = S.quantize_q4_k(np.zeros((m, n), np.float32))
    assert (qs.nbytes + hdr.nbytes) * 8 == 4.5 * m * n
    assert S.qs_bytes(S.Q4_K, m, n) + S.d_bytes(m, n) == qs.nbytes + hdr.nbytes


def test_q4_k_quantizer_round_trip_through_oracle_dequant():
    # weights that are exactly representable with full-range codes re-quantize
    # to the same bytes: sc = 63 and m = 63 in some sub-block fix d and dmin
    rng = np.random.default_rng(14)
    m, n = 4, 512
    codes = rng.integers(0, 16, size=(m, n)).astype(np.uint8)
    codes[:, ::32] = 0
    codes[:, 1::32] = 15                                     # every sub-block spans 0..15
    sc = rng.integers(1, 64, size=(m, n // 256, 8))
    mn = rng.integers(1, 64, size=(m, n // 256, 8))
    sc[..., 0] = 63
    mn[..., 0] = 63
    d = np.float16(0.001)
    hdr = np.stack([np.stack([_hdr_bitwise(int(d.view(np.uint16)), int(d.view(np.uint16)), sc[i, k], mn[i, k])
                              for k in range(n // 256)]) for i in range(m)])
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    w = O.dequantize_q4_k(packed, hdr)
    p2, h2 = S.quantize_q4_k(w.astype(np.float32))
    assert np.array_equal(O.dequantize_q4_k(p2, h2), w)


# ---------------------------------------------------------------- sparse overlays
def _f16(vals):
    return np.asarray(vals, np.float16).view(np.uint16)


def test_sparse_single_entry_moves_exactly_one_weight():
    rng = np.random.default_rng(41)
    m, n = 5, 64
    qs, d = S.quantize_q8_0(S.gaussian(rng, (m, n), 0.02))
    deq = O.dequantize_q8_0(qs, d)
    i, j, v, s = 3, 17, 0.375, 2.0
    term = O.SparseTerm(np.array([i * n + j], np.uint32), _f16([v]), s)
    Wp = O.effective_weight(deq, [term])
    diff = Wp - deq
    assert diff[i, j] == s * v and np.count_nonzero(diff) == 1
    x = S.gaussian(rng, (2, n), 1.0).astype(np.float64)
    y0, y1 = O.dual_path(deq, [], x), O.dual_path(deq, [term], x)
    assert np.array_equal(np.delete(y1, i, axis=1), np.delete(y0, i, axis=1))
    assert np.allclose(y1[:, i] - y0[:, i], s * v * x[:, j], rtol=1e-13, atol=0)


def test_sparse_index_is_row_major_flat():
    # idx = row * d_in + col: entries 0, 4, 7 of a 3x4 tensor are (0,0), (1,0), (1,3)
    term = O.SparseTerm(np.array([0, 4, 7], np.uint32), _f16([1.0, 2.0, -3.0]), 1.0)
    D = O.sparse_delta(term, 3, 4)
    want = np.zeros((3, 4))
    want[0, 0], want[1, 0], want[1, 3] = 1.0, 2.0, -3.0
    assert np.array_equal(D, want)


def test_sparse_outer_product_equals_rank_one_lora():
    # a dense "sparse" overlay holding u w^T (f16-exact values) is the LoRA term B = u, A = w^T
    m, n = 6, 32
    u = np.array([0.5, -1.0, 0.25, 2.0, -0.125, 1.5])
    w = (np.arange(n) % 7 - 3) * 0.0625
    idx = np.arange(m * n, dtype=np.uint32)
    term = O.SparseTerm(idx, _f16(np.outer(u, w).ravel()), 1.5)
    lora = (w[None, :], u[:, None], 1.5)
    deq = np.zeros((m, n))
    assert np.array_equal(O.effective_weight(deq, [term]), O.effective_weight(deq, [lora]))
    x = np.linspace(-1, 1, 2 * n).reshape(2, n)
    assert np.allclose(O.dual_path(deq, [term], x), O.dual_path(deq, [lora], x), rtol=1e-13, atol=1e-15)


def test_sparse_dual_path_exact_rationals():
    rng = np.random.default_rng(43)
    m, n, T = 4, 64, 2
    qs, d = S.quantize_q8_0(S.gaussian(rng, (m, n), 0.02))
    deq = O.dequantize_q8_0(qs, d)
    idx = np.sort(rng.choice(m * n, size=20, replace=False)).astype(np.uint32)
    val = _f16(rng.standard_normal(20) * 0.01)
    s = 0.75
    term = O.SparseTerm(idx, val, s)
    x = S.gaussian(rng, (T, n), 1.0).astype(np.float64)
    y = O.dual_path(deq, [term], x)
    vv = val.view(np.float16).astype(np.float64)
    for t in range(T):
        for i in range(m):
            acc = sum(Fraction(float(deq[i, j])) * Fraction(float(x[t, j])) for j in range(n))
            for k in range(20):
                if int(idx[k]) // n == i:
                    acc += Fraction(s) * Fraction(float(vv[k])) * Fraction(float(x[t, int(idx[k]) % n]))
            assert abs(Fraction(float(y[t, i])) - acc) <= Fraction(1, 10 ** 12) * (abs(acc) + 1)


def test_sparse_and_lora_mixed_dual_equals_merged():
    rng = np.random.default_rng(45)
    m, n, T = 64, 256, 3
    qs, d = S.quantize_q4_0(S.gaussian(rng, (m, n), 0.02))
    deq = O.dequantize_q4_0(qs, d)
    idx, val = S.dare_entries(rng, m, n, keep=0.05)
    terms = [(S.gaussian(rng, (8, n), 0.01), S.gaussian(rng, (m, 8), 0.01), 2.0),
             O.SparseTerm(idx, val, 0.5)]
    x = S.gaussian(rng, (T, n), 1.0).astype(np.float64)
    Wp = O.effective_weight(deq, terms)
    dual = O.dual_path(deq, terms, x)
    merged = O.merged_path(Wp, x)
    assert (np.abs(dual - merged) <= 1e-12 * (np.abs(x) @ np.abs(Wp).T)).all()
    # order of the stack does not change W' in exact arithmetic; here fp64 agrees closely
    assert np.allclose(O.effective_weight(deq, terms[::-1]), Wp, rtol=0, atol=1e-15)


def test_sparse_adapter_key_brute_recomputation():
    # the byte string of the identity, assembled field by field with hashlib
    dg = bytes(range(32))
    want = hashlib.sha256(b"OVLS" + dg + (2).to_bytes(4, "little")
                          + (3).to_bytes(4, "little") + (100).to_bytes(4, "little")
                          + (0).to_bytes(8, "little") + (512).to_bytes(8, "little")
                          + (6).to_bytes(4, "little") + (7).to_bytes(4, "little")
                          + (768).to_bytes(8, "little") + (1024).to_bytes(8, "little")).digest()
    assert O.sparse_adapter_key(dg, [(3, 100, 0, 512), (6, 7, 768, 1024)]) == want
    # a sparse overlay and a low-rank adapter with the same numbers are different identities
    assert O.sparse_adapter_key(dg, [(3, 100, 0, 512)]) != O.adapter_key(dg, [(3, 100, 0, 512)])


def test_dare_entries_shape_and_order():
    rng = np.random.default_rng(47)
    idx, val = S.dare_entries(rng, 300, 512, keep=0.02)
    assert idx.dtype == np.uint32 and val.dtype == np.uint16
    assert np.all(np.diff(idx.astype(np.int64)) > 0) and int(idx[-1]) < 300 * 512
    assert abs(idx.size / (300 * 512) - 0.02) < 0.003
    assert np.isfinite(val.view(np.float16)).all()


# ---------------------------------------------------------------- GEMV / LoRA
def _tiny_problem(seed, m=6, n=64, T=2, ranks=(2, 3)):
    rng = np.random.default_rng(seed)
    w = S.gaussian(rng, (m, n), 0.02)
    qs, d = S.quantize_q8_0(w)
    ads = []
    for r in ranks:
        A = S.gaussian(rng, (r, n), 0.01)
        B = S.gaussian(rng, (m, r), 0.01)
        ads.append((A, B, float(rng.choice([0.5, 1.0, 2.0]))))
    x = S.gaussian(rng, (T, n), 1.0)
    return qs, d, ads, x


def _exact_dual(qs, d, ads, x):
    m, n = qs.shape
    dq = [[Fraction(float(d[i, j // 32:j // 32 + 1].view(np.float16)[0])) * int(qs[i, j])
           for j in range(n)] for i in range(m)]
    xs = [[Fraction(float(v)) for v in row] for row in x]
    out = []
    for xt in xs:
        y = [sum(dq[i][j] * xt[j] for j in range(n)) for i in range(m)]
        for A, B, s in ads:
            r = A.shape[0]
            v = [sum(Fraction(float(A[t, j])) * xt[j] for j in range(n)) for t in range(r)]
            for i in range(m):
                y[i] += Fraction(s) * sum(Fraction(float(B[i, t])) * v[t] for t in range(r))
        out.append(y)
    return out


def _exact_merged(qs, d, ads, x):
    m, n = qs.shape
    W = [[Fraction(float(d[i, j // 32:j // 32 + 1].view(np.float16)[0])) * int(qs[i, j])
          for j in range(n)] for i in range(m)]
    for A, B, s in ads:
        r = A.shape[0]
        for i in range(m):
            for j in range(n):
                W[i][j] += Fraction(s) * sum(Fraction(float(B[i, t])) * Fraction(float(A[t, j]))
                                             for t in range(r))
    return [[sum(W[i][j] * Fraction(float(xt[j])) for j in range(n)) for i in range(m)] for xt in x]


def test_base_gemv_exact_rationals():
    qs, d, _, x = _tiny_problem(11, ranks=())
    exact = _exact_dual(qs, d, [], x)
    deq = O.dequantize_q8_0(qs, d)
    y = O.dual_path(deq, [], x)
    scale = np.abs(x.astype(np.float64)) @ np.abs(deq).T
    for t in range(x.shape[0]):
        for i in range(qs.shape[0]):
            assert abs(Fraction(float(y[t, i])) - exact[t][i]) <= Fraction(1e-13) * Fraction(float(scale[t, i]))


def test_dual_equals_merged_exact_rationals():
    qs, d, ads, x = _tiny_problem(12)
    ed = _exact_dual(qs, d, ads, x)
    em = _exact_merged(qs, d, ads, x)
    assert ed == em                                           # algebraic identity, exactly
    deq = O.dequantize_q8_0(qs, d)
    Wp = O.effective_weight(deq, ads)
    yd = O.dual_path(deq, ads, x)
    ym = O.merged_path(Wp, x)
    scale = np.abs(x.astype(np.float64)) @ np.abs(Wp).T
    for t in range(x.shape[0]):
        for i in range(qs.shape[0]):
            tol = Fraction(1e-13) * Fraction(float(scale[t, i]))
            assert abs(Fraction(float(yd[t, i])) - ed[t][i]) <= tol
            assert abs(Fraction(float(ym[t, i])) - ed[t][i]) <= tol


def test_dual_equals_merged_fp64_config1_size():
    base, ad_a, ad_b, x, s = S.single_layer_256()
    qs, d = base.planes[0]
    deq = O.dequantize_q8_0(qs, d)
    for ad in (ad_a, ad_b):
        A, B = ad.factors[0]
        ads = [(A, B, s)]
        Wp = O.effective_weight(deq, ads)
        diff = np.abs(O.dual_path(deq, ads, x) - O.merged_path(Wp, x))
        assert (diff <= 1e-12 * (np.abs(x.astype(np.float64)) @ np.abs(Wp).T)).all()


def test_zero_B_gives_base_output_exactly():
    qs, d, ads, x = _tiny_problem(13, ranks=(4,))
    A, B, s = ads[0]
    deq = O.dequantize_q8_0(qs, d)
    y0 = O.dual_path(deq, [], x)
    y1 = O.dual_path(deq, [(A, np.zeros_like(B), s)], x)
    assert np.array_equal(y0.view(np.uint64), y1.view(np.uint64))
    W1 = O.effective_weight(deq, [(A, np.zeros_like(B), s)])
    assert np.array_equal(W1, deq)


def test_unit_outer_product_moves_one_weight_by_s():
    qs, d, _, x = _tiny_problem(14, ranks=())
    m, n = qs.shape
    i0, j0, s = 3, 17, 2.0
    A = np.zeros((1, n), np.float32)
    A[0, j0] = 1
    B = np.zeros((m, 1), np.float32)
    B[i0, 0] = 1
    deq = O.dequantize_q8_0(qs, d)
    Wp = O.effective_weight(deq, [(A, B, s)])
    delta = Wp - deq
    assert delta[i0, j0] == s and np.count_nonzero(delta) == 1
    y0 = O.dual_path(deq, [], x)
    y1 = O.dual_path(deq, [(A, B, s)], x)
    others = np.arange(m) != i0
    assert np.array_equal(y0[:, others], y1[:, others])
    assert np.allclose(y1[:, i0] - y0[:, i0], s * x[:, j0].astype(np.float64), rtol=0, atol=1e-15)


def test_stack_order_exact_and_identity_order():
    qs, d, ads, x = _tiny_problem(15, m=3, n=32, T=1)
    fwd = _exact_dual(qs, d, ads, x)
    rev = _exact_dual(qs, d, ads[::-1], x)
    assert fwd == rev                                         # linear LoRA commutes exactly
    bk = O.base_key(b"\1" * 32, O.Q8_0, [(0, 0, 3, 32, 0, 256)])
    ka = O.adapter_key(b"\2" * 32, [(0, 2, 0, 256)])
    kb = O.adapter_key(b"\3" * 32, [(0, 3, 0, 512)])
    assert O.composition_id(bk, O.MODE_STACK, [(ka, 1.0), (kb, 0.5)]) != \
        O.composition_id(bk, O.MODE_STACK, [(kb, 0.5), (ka, 1.0)])


def test_error_bound_hand_example():
    W = np.array([[1.0, -2.0], [0.5, 0.0]])
    x = np.array([[3.0, 1.0]])
    b = O.error_bound(W, x)
    assert np.allclose(b, [[2e-3 * 5 + 1e-5, 2e-3 * 1.5 + 1e-5]], rtol=0, atol=1e-18)


def test_segmented_reduces_to_dual_per_token():
    qs, d, ads, x = _tiny_problem(16, T=5, ranks=(2, 3, 4))
    deq = O.dequantize_q8_0(qs, d)
    slots = np.array([2, 0, -1, 2, 1])
    y = O.segmented(deq, ads, x, slots)
    for t, sl in enumerate(slots):
        want = O.dual_path(deq, [ads[sl]] if sl >= 0 else [], x[t:t + 1])[0]
        assert np.array_equal(y[t], want)
    ex = _exact_dual(qs, d, [ads[2]], x[:1])
    assert abs(Fraction(float(y[0, 0])) - ex[0][0]) <= Fraction(1e-13)


def test_materialize_bound_covers_fp32_rounding_of_dequant():
    qs, d, ads, _ = _tiny_problem(17)
    deq = O.dequantize_q8_0(qs, d)
    assert np.array_equal(deq.astype(np.float32).astype(np.float64), deq)   # dequant is exact in fp32
    b = O.materialize_bound(deq, ads)
    assert (b > 0).all() and (b < 1e-5).all()


# ---------------------------------------------------------------- digests / identity
FIPS = {
    b"abc": "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad",
    b"": "e3b0c44298fc1c149afbf4c8996fb92427ae41e4649b934ca495991b7852b855",
    b"abcdbcdecdefdefgefghfghighijhijkijkljklmklmnlmnomnopnopq":
        "248d6a61d20638b8e5c026930c3e6039a33ce45964ff2167f6ecedd419db06c1",
}


def test_sha256_primitive_fips_vectors():
    for msg, hexd in FIPS.items():
        assert hashlib.sha256(msg).hexdigest() == hexd


def test_tree_digest_closed_forms():
    rng = np.random.default_rng(5)
    one = rng.integers(0, 256, size=1000, dtype=np.uint8)
    assert O.tree_digest(one) == hashlib.sha256(hashlib.sha256(one.tobytes()).digest()).digest()
    full = rng.integers(0, 256, size=O.LEAF, dtype=np.uint8)
    assert O.tree_digest(full) == hashlib.sha256(hashlib.sha256(full.tobytes()).digest()).digest()
    assert O.tree_digest(np.zeros(0, np.uint8)).hex() == FIPS[b""]


@pytest.mark.parametrize("size", [1, 65535, 65536, 65537, 3 * 65536 + 17])
def test_tree_digest_matches_caller_side_digest(size):
    buf = np.random.default_rng(size).integers(0, 256, size=size, dtype=np.uint8)
    assert O.tree_digest(buf) == S.content_digest(buf)


# The identity byte strings, assembled field by field from the C header's text
# (little-endian u32 / u64 fields, 4-byte tags, a 16-byte runtime tag) with
# int.to_bytes and hashlib: values are chosen so that a field packed at the
# wrong width, two fields swapped or a dropped field changes the digest.
def _u32(v):
    return int(v).to_bytes(4, "little")


def _u64(v):
    return int(v).to_bytes(8, "little")


ID_TENSORS = [(3, 6, 14336, 4096, 0x1_0000_0100, 0x2_0000_0200),
              (31, 2, 1024, 8192, 256, 0x3_FFFF_FF00)]
ID_TARGETS = [(5, 16, 0x1_0000_0010, 0x3_0000_0020), (9, 64, 4096, 0x7_0000_2000)]


def test_base_key_field_by_field():
    dg = bytes(range(100, 132))
    raw = b"OVLB" + dg + _u32(O.Q4_0) + _u32(len(ID_TENSORS))
    for layer, proj, d_out, d_in, qs_off, d_off in ID_TENSORS:
        raw += _u32(layer) + _u32(proj) + _u32(d_out) + _u32(d_in) + _u64(qs_off) + _u64(d_off)
    assert len(raw) == 4 + 32 + 8 + 2 * 32
    assert O.base_key(dg, O.Q4_0, ID_TENSORS) == hashlib.sha256(raw).digest()


def test_adapter_key_field_by_field():
    dg = bytes(range(200, 232))
    raw = b"OVLA" + dg + _u32(len(ID_TARGETS))
    for tensor, rank, a_off, b_off in ID_TARGETS:
        raw += _u32(tensor) + _u32(rank) + _u64(a_off) + _u64(b_off)
    assert len(raw) == 4 + 32 + 4 + 2 * 24
    assert O.adapter_key(dg, ID_TARGETS) == hashlib.sha256(raw).digest()


def test_composition_id_field_by_field():
    bk = hashlib.sha256(b"base").digest()
    k1, k2 = hashlib.sha256(b"one").digest(), hashlib.sha256(b"two").digest()
    tag = b"ovl-gb300 v1" + bytes(4)                   # 16 bytes, zero padded
    scales = [2.0, -0.75]
    raw = b"OVLC" + tag + bk + _u32(O.MODE_TABLE) + _u32(2)
    for k, sc in zip((k1, k2), scales):
        raw += k + np.float32(sc).tobytes()            # IEEE-754 binary32 bits, little-endian
    assert O.composition_id(bk, O.MODE_TABLE, list(zip((k1, k2), scales))) == hashlib.sha256(raw).digest()
    # an empty composition is recorded with mode STACK whatever mode was asked
    empty = hashlib.sha256(b"OVLC" + tag + bk + _u32(O.MODE_STACK) + _u32(0)).digest()
    assert O.composition_id(bk, O.MODE_TABLE, []) == empty
    assert O.composition_id(bk, O.MODE_STACK, []) == empty


def test_tree_digest_multi_leaf_closed_forms():
    """Two and three leaves: SHA256(SHA256(l0) | SHA256(l1) [| SHA256(l2)]),
    the last leaf short."""
    rng = np.random.default_rng(11)
    for size in (O.LEAF + 100, 2 * O.LEAF + 1):
        buf = rng.integers(0, 256, size=size, dtype=np.uint8).tobytes()
        leaves = [buf[i:i + 65536] for i in range(0, size, 65536)]
        assert len(leaves) == (2 if size < 2 * 65536 else 3)
        want = hashlib.sha256(b"".join(hashlib.sha256(l).digest() for l in leaves)).digest()
        assert O.tree_digest(np.frombuffer(buf, np.uint8)) == want


def test_composition_id_invariants():
    bk = O.base_key(b"\1" * 32, O.Q8_0, [(0, 0, 256, 256, 0, 65536)])
    ka = O.adapter_key(b"\2" * 32, [(0, 8, 0, 8192)])
    base_only = O.composition_id(bk, O.MODE_STACK, [])
    with_a = O.composition_id(bk, O.MODE_STACK, [(ka, 2.0)])
    assert base_only != with_a
    assert with_a == O.composition_id(bk, O.MODE_STACK, [(ka, 2.0)])
    assert with_a != O.composition_id(bk, O.MODE_STACK, [(ka, float(np.nextafter(np.float32(2.0), 3)))])
    assert with_a != O.composition_id(bk, O.MODE_TABLE, [(ka, 2.0)])
    bk2 = O.base_key(b"\1" * 32, O.Q4_0, [(0, 0, 256, 256, 0, 65536)])
    assert O.composition_id(bk2, O.MODE_STACK, []) != base_only
    assert O.base_key(b"\1" * 32, O.Q8_0, [(0, 0, 256, 256, 0, 65536)]) != \
        O.base_key(b"\1" * 32, O.Q8_0, [(0, 1, 256, 256, 0, 65536)])


def test_switch_model_invariants():
    bk = b"\7" * 32
    m = O.SwitchModel(bk)
    _, ha = m.stage(b"\xaa" * 32)
    _, hb = m.stage(b"\xbb" * 32)
    base_id = m.current_id()
    st, ida = m.activate([ha], [2.0])
    assert st == O.OVL_OK and ida != base_id
    ep = m.epoch
    st, ida2 = m.activate([ha], [2.0])                         # idempotent
    assert st == O.OVL_OK and ida2 == ida and m.epoch == ep
    assert m.unstage(ha) == O.OVL_E_STATE                       # active
    st, _ = m.activate([], [])                                  # deactivate = base-only
    assert m.current_id() == base_id
    st, idb = m.activate([hb], [2.0])
    # reversibility: base -> A -> base -> B has the state of base -> B
    m2 = O.SwitchModel(bk)
    m2.stage(b"\xaa" * 32)
    _, hb2 = m2.stage(b"\xbb" * 32)
    _, idb2 = m2.activate([hb2], [2.0])
    assert idb == idb2 and m.active == m2.active
    assert m.rollback() == (O.OVL_OK, base_id)
    assert m.rollback()[0] == O.OVL_E_NO_PREVIOUS               # one level deep
    assert m.activate([ha, ha], [1.0, 1.0])[0] == O.OVL_E_DUPLICATE
    assert m.activate([ha], [float("nan")])[0] == O.OVL_E_ARG
    assert m.current_id() == base_id                            # failures change nothing


def test_switch_transcript_golden():
    with open(os.path.join(GOLDEN, "switch_transcript.json")) as f:
        g = json.load(f)
    keys = [bytes.fromhex(k) for k in g["adapter_keys"]]
    tr = O.switch_transcript(bytes.fromhex(g["base_key"]), keys, g["scale"], g["n_ops"], g["corrupt"])
    assert [list(t) for t in tr] == g["transcript"]
    statuses = [t[2] for t in tr]
    assert statuses.count(O.OVL_E_HASH) == 12 and statuses.count(O.OVL_E_NO_PREVIOUS) == 12


def test_config1_golden_outputs():
    with open(os.path.join(GOLDEN, "config1.json")) as f:
        g = json.load(f)
    base, ad_a, ad_b, x, s = S.single_layer_256()
    assert S.content_digest(base.buf).hex() == g["base_digest"]
    qs, d = base.planes[0]
    deq = O.dequantize_q8_0(qs, d)
    for name, ad in (("base", None), ("A", ad_a), ("B", ad_b)):
        ads = [] if ad is None else [(ad.factors[0][0], ad.factors[0][1], s)]
        y = O.dual_path(deq, ads, x)[0]
        want = np.array([float.fromhex(h) for h in g["y"][name]])
        assert np.array_equal(y, want)
