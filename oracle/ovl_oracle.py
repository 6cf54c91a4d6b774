"""Oracle: fp64 CPU statement of what the overlay library computes.

TEST INFRASTRUCTURE ONLY (see the package docstring): the library's product
path never reaches this module, and this module never reaches the library.

Sources (cited by page title and section):

* [OVR]  "We propose a content-addressed overlay system ..." report
  (mikekappel.com/reports/runtime/we-propose-a-content-addressed-overlay-system/)
* [DTD]  "Deep Technical Design: Exact, Atomic, Reversible Specialist Overlays on
  Quantized Transformer Bases"
  (mikekappel.com/reports/runtime/quantized-adapter-runtime-architecture/)
* [MODELD] contenox modeld blueprint "LoRA adapters"
  (contenox.com/docs/development/blueprints/modeld/lora-adapters/)

Function -> pin (tests/test_oracle_pins.py):

* f16_to_float            exhaustive vs numpy's binary16 decoder (all 65536 patterns)
* dequantize_q8_0/q4_0    exhaustive (every finite scale x every code) vs exact
                          products; exact rationals on a sample; hand-built nibbles
* q4_k_header_fields      every 6-bit value in every sub-block slot vs headers
                          packed bit by bit; random headers vs a bit-string decode
* dequantize_q4_k         reduces bitwise to dequantize_q4_0 (sc = 1, m = 8,
                          dmin = d); hand-evaluated sub-block staircase; exact
                          rationals on every (sc, m, code) with sampled scales;
                          4.5 bits per weight
* dual_path / merged_path exact-rational brute force on tiny shapes; dual == merged
                          identity; zero-B and unit outer-product closed forms
* effective_weight        closed forms (zero-B, e_i e_j^T), order invariance in
                          exact arithmetic
* error_bound             hand-evaluated 2x2 example
* SparseTerm / sparse_delta and the sparse terms of effective_weight,
  dual_path            one entry moves exactly one weight by s*v (closed form);
                          a sparse overlay equal to a rank-1 outer product gives
                          the same W' and y as that LoRA term; exact-rational
                          brute force on tiny shapes; dual == merged with mixed
                          stacks
* segmented               reduces to dual_path per token (brute force)
* tree_digest             single-leaf closed form SHA256(SHA256(data)); FIPS 180
                          test vectors for the primitive
* composition_id          invariants (order, scale bits, base-only) + golden file
* SwitchModel             invariants + golden transcript of the switch sequence
No function here is "parity unpinned".
"""
from __future__ import annotations

import hashlib
import struct
from dataclasses import dataclass, field

import numpy as np

QK = 32
QK_K = 256           # weights per q4_K super-block
Q8_0 = 1
Q4_0 = 2
Q4_K = 3
MODE_STACK = 1
MODE_TABLE = 2
LEAF = 65536

# status codes of the library's boundary, restated from its specification
OVL_OK = 0
OVL_E_ARG = -1
OVL_E_HASH = -2
OVL_E_SHAPE = -3
OVL_E_QUANT = -4
OVL_E_OOM = -5
OVL_E_NONFINITE = -6
OVL_E_DUPLICATE = -7
OVL_E_NOTARGET = -8
OVL_E_BUSY = -9
OVL_E_NO_PREVIOUS = -10
OVL_E_STATE = -11

RUNTIME_TAG = b"ovl-gb300 v1\0\0\0\0"   # 16 bytes: runtime version in the identity


# --------------------------------------------------------------------------
# Block dequantization.
# [DTD] §5 "Quantized-Base Numerical Analysis": a q8_0 block is 32 weights and
# one f16 scale; the benchmark's q4_0 block is 32 4-bit codes and an f16 scale
# with value d*(code-8).  [OVR] §"Immutable base": full-precision values are
# only materialized transiently.
# --------------------------------------------------------------------------
def f16_to_float(bits) -> np.ndarray:
    """IEEE 754 binary16 -> float64, from the format's definition.

    sign s, 5-bit exponent e (bias 15), 10-bit fraction f:
      e = 0          -> (-1)^s * f * 2^-24            (zero / subnormal)
      0 < e < 31     -> (-1)^s * (1024 + f) * 2^(e-25) (normal)
      e = 31         -> +-inf (f = 0) or NaN
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(f, -24), np.ldexp(1024.0 + f, (e - 25).astype(np.int64)))
    mag = np.where(e == 31, np.where(f == 0, np.inf, np.nan), mag)
    return s * mag


def dequantize_q8_0(qs: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """w[i][j] = d[i][j/32] * q[i][j], q int8, in float64 (exact)."""
    qs = np.asarray(qs).view(np.int8)
    m, n = qs.shape
    d = f16_to_float(d_bits).reshape(m, n // QK)
    return np.repeat(d, QK, axis=1) * qs.astype(np.float64)


def q4_0_codes(packed: np.ndarray) -> np.ndarray:
    """Unpack nibbles: element 2p <- low nibble of byte p, 2p+1 <- high nibble."""
    packed = np.asarray(packed, dtype=np.uint8)
    m, half = packed.shape
    codes = np.empty((m, 2 * half), dtype=np.int64)
    codes[:, 0::2] = packed & 0x0F
    codes[:, 1::2] = packed >> 4
    return codes


def dequantize_q4_0(packed: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """w[i][j] = d[i][j/32] * (code[i][j] - 8), in float64 (exact)."""
    codes = q4_0_codes(packed)
    m, n = codes.shape
    d = f16_to_float(d_bits).reshape(m, n // QK)
    return np.repeat(d, QK, axis=1) * (codes - 8).astype(np.float64)


# --------------------------------------------------------------------------
# q4_K super-blocks.
# [DTD] §5 "Quantized-Base Numerical Analysis": a q4_K super-block holds 256
# weights in 8 sub-blocks of 32; every sub-block has a 6-bit scale and a 6-bit
# minimum (zero-point), and two f16 scales govern the whole super-block, for
# 4.5 bits per weight.  Reading: the sub-block scale multiplies the f16 scale d
# and the sub-block minimum multiplies the f16 scale dmin, and the minimum is
# subtracted, w = d*sc_j*code - dmin*m_j with a 4-bit code.  The pages give no
# byte packing; the header of each super-block is 16 bytes:
#   bytes 0-1  d (binary16), bytes 2-3 dmin (binary16),
#   bytes 4-9  the eight sc_j as one 48-bit little-endian field, sc_j in bits 6j..6j+5,
#   bytes 10-15 the eight m_j the same way.
# Codes use the q4_0 nibble order within the row.
# --------------------------------------------------------------------------
def q4_k_header_fields(hdr: np.ndarray):
    """Split 16-byte headers [..][16] into (d, dmin, sc[..][8], m[..][8]).

    d and dmin are float64 values; sc and m are integers 0..63.
    """
    h = np.asarray(hdr, dtype=np.uint8).astype(np.int64)
    d = f16_to_float(h[..., 0] + 256 * h[..., 1])
    dmin = f16_to_float(h[..., 2] + 256 * h[..., 3])

    def field48(bytes6):
        # the six bytes as one little-endian integer, then eight 6-bit slices
        v = np.zeros(bytes6.shape[:-1], dtype=np.int64)
        for k in range(6):
            v += bytes6[..., k] << (8 * k)
        return np.stack([(v >> (6 * j)) & 63 for j in range(8)], axis=-1)

    return d, dmin, field48(h[..., 4:10]), field48(h[..., 10:16])


def dequantize_q4_k(packed: np.ndarray, hdr: np.ndarray) -> np.ndarray:
    """w[i][c] = d * sc_j * code[i][c] - dmin * m_j, j = (c mod 256) / 32, in float64.

    packed: uint8 [m][n/2] codes (q4_0 nibble order); hdr: uint8 [m][n/256][16]
    (or [m][n/16]).  Exact: every product has at most 11+6+4 significant bits.
    """
    codes = q4_0_codes(packed).astype(np.float64)
    m, n = codes.shape
    d, dmin, sc, mn = q4_k_header_fields(np.asarray(hdr, np.uint8).reshape(m, n // QK_K, 16))
    scale = (d[..., None] * sc).reshape(m, n // QK)       # per 32-weight sub-block
    minimum = (dmin[..., None] * mn).reshape(m, n // QK)
    return np.repeat(scale, QK, axis=1) * codes - np.repeat(minimum, QK, axis=1)


def dequantize(quant: int, qs, d_bits) -> np.ndarray:
    if quant == Q8_0:
        return dequantize_q8_0(qs, d_bits)
    if quant == Q4_0:
        return dequantize_q4_0(qs, d_bits)
    if quant == Q4_K:
        return dequantize_q4_k(qs, d_bits)
    raise ValueError("unknown quant profile")


# --------------------------------------------------------------------------
# Effective weights and the two evaluation paths.
# [OVR] §"Explicit Correctness and Atomicity Invariants" (Compositional
# Integrity): W' = W + sum_i dW_i in load order.  [OVR] §"Quantized-Base
# Numerical Analysis": fresh-base oracle Y = W + sum_i dW_i from one dequant.
# [OVR] §"Annotated Primary-Source Bibliography" (LoRA): dW = (alpha/r) B A;
# the scale s folds alpha/r and any merge weight.
# [OVR] §"Native/WASM Kernel Implications": direct low-rank addition
# y = xW + x(BA) (two small matmuls) vs pre-merged W' = W + BA.
# --------------------------------------------------------------------------
# --------------------------------------------------------------------------
# Sparse overlays.
# [OVR] §"Runtime Strategy Comparison Matrix" (Sparse Overlay): only the
# non-zero elements of the update are stored, as indices and values, and they
# are added at those indices at use time; the base is unchanged.
# [OVR] §"Memory, Byte, and Latency Formulas" (Sparse Adapter) and [DTD] §7
# (Sparse Overlay Bytes): 32-bit indices and 16-bit (f16) values, k*(4+2)
# bytes.  [DTD] §11 (Deep Compatibility Checks): indices strictly monotonic,
# no NaN or Inf in the f16 payload.  Reading: index = row*d_in + col of the
# tensor the target names; the term's scale s multiplies every value.
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class SparseTerm:
    idx: np.ndarray        # uint32 flat indices row * d_in + col, strictly increasing
    val_bits: np.ndarray   # uint16 binary16 values
    s: float


def sparse_delta(term: SparseTerm, m: int, n: int) -> np.ndarray:
    """Dense float64 [m][n] with delta[idx[k] / n][idx[k] mod n] = f16(val[k])."""
    D = np.zeros(m * n, dtype=np.float64)
    D[np.asarray(term.idx, np.int64)] = f16_to_float(term.val_bits)
    return D.reshape(m, n)


def _term_matrix(term, m: int, n: int) -> np.ndarray:
    """s * dW of one overlay term: (A, B, s) low-rank or SparseTerm."""
    if isinstance(term, SparseTerm):
        return float(term.s) * sparse_delta(term, m, n)
    A, B, s = term
    return float(s) * (np.asarray(B, np.float64) @ np.asarray(A, np.float64))


def effective_weight(deq: np.ndarray, adapters) -> np.ndarray:
    """W' = deq + sum_k s_k * dW_k in order; a term is (A [r][n], B [m][r], s)
    (dW = B A) or a SparseTerm (dW = its scattered values)."""
    W = np.array(deq, dtype=np.float64, copy=True)
    m, n = W.shape
    for term in adapters:
        W += _term_matrix(term, m, n)
    return W


def dual_path(deq: np.ndarray, adapters, x: np.ndarray) -> np.ndarray:
    """y[t] = deq x[t] + sum_k s_k dW_k x[t]; x [T][n] -> y [T][m], float64.

    Low-rank terms go through the rank-r side product s B (A x); sparse terms
    add s * sum over the stored entries of the row of val * x[col]."""
    x = np.asarray(x, dtype=np.float64)
    deq = np.asarray(deq, np.float64)
    m, n = deq.shape
    y = x @ deq.T
    for term in adapters:
        if isinstance(term, SparseTerm):
            idx = np.asarray(term.idx, np.int64)
            rows, cols = idx // n, idx % n
            contrib = np.zeros((x.shape[0], m), dtype=np.float64)
            # entry-by-entry accumulation (np.add.at: unbuffered, repeated rows add up)
            np.add.at(contrib.T, rows, (f16_to_float(term.val_bits)[:, None] * x[:, cols].T))
            y = y + float(term.s) * contrib
            continue
        A, B, s = term
        v = x @ np.asarray(A, np.float64).T            # [T][r]   shrink
        y = y + float(s) * (v @ np.asarray(B, np.float64).T)   # [T][m] expand
    return y


def merged_path(W_eff: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y[t] = W' x[t] (the per-layer materialized path), float64."""
    return np.asarray(x, np.float64) @ np.asarray(W_eff, np.float64).T


def error_bound(W_eff: np.ndarray, x: np.ndarray, rel: float = 2e-3, abs_: float = 1e-5) -> np.ndarray:
    """Per-output tolerance rel * sum_j |W'_ij x_j| + abs_  ([T][m])."""
    return rel * (np.abs(np.asarray(x, np.float64)) @ np.abs(np.asarray(W_eff, np.float64)).T) + abs_


def materialize_bound(deq: np.ndarray, adapters, ulps: float = 4.0) -> np.ndarray:
    """Element bound for an fp32 materialization of W' = deq + sum s B A.

    Each term of the sum is formed and added in fp32; the bound is
    ulps * 2^-24 * (rank+2) * (|deq| + sum_k |s_k| |B_k| |A_k|).
    """
    mag = np.abs(np.asarray(deq, np.float64)).copy()
    m, n = mag.shape
    terms = 2
    for term in adapters:
        if isinstance(term, SparseTerm):
            mag += np.abs(_term_matrix(term, m, n))
            terms += 2
            continue
        A, B, s = term
        mag += abs(float(s)) * (np.abs(np.asarray(B, np.float64)) @ np.abs(np.asarray(A, np.float64)))
        terms += np.asarray(A).shape[0] + 1
    return ulps * 2.0 ** -24 * terms * mag


def segmented(deq: np.ndarray, table, x: np.ndarray, slot_of_token) -> np.ndarray:
    """Multi-adapter batch ([DTD] §1, SGMV): token t uses table[slot_of_token[t]].

    y[t] = deq x[t] + s B (A x[t]) with (A, B, s) = table[slot]; slot < 0 means
    base only.  Output rows in the original request order.
    """
    x = np.asarray(x, np.float64)
    y = np.empty((x.shape[0], deq.shape[0]), dtype=np.float64)
    for t in range(x.shape[0]):
        sl = int(slot_of_token[t])
        ads = [table[sl]] if sl >= 0 else []
        y[t] = dual_path(deq, ads, x[t:t + 1])[0]
    return y


# --------------------------------------------------------------------------
# Content digests and composition identity.
# [OVR] §"Composition Identity and Manifest Schema": identity = base hash,
# layout + quantization profile, ordered adapter list with hashes and merge
# coefficients, runtime version.  [DTD] §3 (same tuple, formula lost in the
# export).  [MODELD] §"Runtime Identity and Cache Safety": adapter list in
# deterministic order, each digest and scale.  [OVR] §"Checksum Verification":
# SHA-256 of every artifact.
# --------------------------------------------------------------------------
def tree_digest(buf, leaf: int = LEAF) -> bytes:
    """SHA-256 over the concatenation of SHA-256(leaf_i), leaves of `leaf` bytes."""
    mv = memoryview(np.ascontiguousarray(np.frombuffer(bytes(buf), dtype=np.uint8)
                                         if isinstance(buf, (bytes, bytearray)) else buf
                                         ).view(np.uint8)).cast("B")
    leaves = [hashlib.sha256(mv[i:i + leaf]).digest() for i in range(0, len(mv), leaf)]
    return hashlib.sha256(b"".join(leaves)).digest()


def base_key(digest: bytes, quant: int, tensors) -> bytes:
    """tensors: iterable of (layer, proj, d_out, d_in, qs_off, d_off)."""
    tensors = list(tensors)
    h = hashlib.sha256()
    h.update(b"OVLB")
    h.update(digest)
    h.update(struct.pack("<II", quant, len(tensors)))
    for (layer, proj, d_out, d_in, qs_off, d_off) in tensors:
        h.update(struct.pack("<IIIIQQ", layer, proj, d_out, d_in, qs_off, d_off))
    return h.digest()


def adapter_key(digest: bytes, targets) -> bytes:
    """targets: iterable of (tensor_index, rank, a_off, b_off)."""
    targets = list(targets)
    h = hashlib.sha256()
    h.update(b"OVLA")
    h.update(digest)
    h.update(struct.pack("<I", len(targets)))
    for (ti, r, ao, bo) in targets:
        h.update(struct.pack("<IIQQ", ti, r, ao, bo))
    return h.digest()


def sparse_adapter_key(digest: bytes, targets) -> bytes:
    """Identity of a sparse overlay; targets: iterable of (tensor_index, nnz, idx_off, val_off)."""
    targets = list(targets)
    h = hashlib.sha256()
    h.update(b"OVLS")
    h.update(digest)
    h.update(struct.pack("<I", len(targets)))
    for (ti, nnz, io, vo) in targets:
        h.update(struct.pack("<IIQQ", ti, nnz, io, vo))
    return h.digest()


def f32_bits(s: float) -> int:
    return struct.unpack("<I", struct.pack("<f", float(s)))[0]


def composition_id(bkey: bytes, mode: int, entries) -> bytes:
    """entries: ordered [(adapter_key, scale)]; empty = base only (mode STACK)."""
    entries = list(entries)
    h = hashlib.sha256()
    h.update(b"OVLC")
    h.update(RUNTIME_TAG)
    h.update(bkey)
    h.update(struct.pack("<II", mode if entries else MODE_STACK, len(entries)))
    for akey, s in entries:
        h.update(akey)
        h.update(struct.pack("<I", f32_bits(s)))
    return h.digest()


# --------------------------------------------------------------------------
# Activation state machine.
# [OVR] §"Proposed Activation/Deactivation State Machine": validate -> stage ->
# atomic swap; on error the pointer is unchanged; the old state may be kept for
# rollback; deactivation = activating the base-only manifest.
# [OVR] §"Explicit Correctness and Atomicity Invariants": idempotency (repeated
# activation of the same composition does nothing); concurrent safety (reject
# the switch while generation runs).  [DTD] §6: VALIDATION, ALLOCATION,
# STAGING, CHECKSUM, COMMIT/SWAP, ROLLBACK.
# --------------------------------------------------------------------------
@dataclass
class SwitchModel:
    """Pure-Python model of the observable switch state.

    Rollback is one level deep: it restores the composition that was active
    before the last successful swap and clears the rollback slot.
    """
    base_key: bytes
    staged: dict = field(default_factory=dict)      # handle -> adapter_key
    active: tuple = ()                              # ((handle, scale), ...)
    mode: int = MODE_STACK
    prev: object = None                             # (entries, mode) or None
    epoch: int = 0
    next_handle: int = 1

    def _id(self, entries, mode):
        return composition_id(self.base_key, mode, [(self.staged[h], s) for h, s in entries])

    def current_id(self):
        return self._id(self.active, self.mode)

    def stage(self, akey: bytes, ok: bool = True, err: int = OVL_E_HASH):
        if not ok:
            return err, None
        h = self.next_handle
        self.next_handle += 1
        self.staged[h] = akey
        return OVL_OK, h

    def activate(self, handles, scales, mode=MODE_STACK):
        handles = list(handles)
        if any(h not in self.staged for h in handles):
            return OVL_E_ARG, self.current_id()
        if len(set(handles)) != len(handles):
            return OVL_E_DUPLICATE, self.current_id()
        if any(not np.isfinite(s) for s in scales):
            return OVL_E_ARG, self.current_id()
        entries = tuple(zip(handles, [float(np.float32(s)) for s in scales]))
        mode = mode if entries else MODE_STACK
        new_id = self._id(entries, mode)
        if new_id == self.current_id():
            return OVL_OK, new_id                    # idempotent no-op
        self.prev = (self.active, self.mode)
        self.active, self.mode = entries, mode
        self.epoch += 1
        return OVL_OK, new_id

    def rollback(self):
        if self.prev is None:
            return OVL_E_NO_PREVIOUS, self.current_id()
        self.active, self.mode = self.prev
        self.prev = None
        self.epoch += 1
        return OVL_OK, self.current_id()

    def unstage(self, h):
        if h not in self.staged:
            return OVL_E_ARG
        in_use = any(hh == h for hh, _ in self.active)
        if self.prev is not None:
            in_use = in_use or any(hh == h for hh, _ in self.prev[0])
        if in_use:
            return OVL_E_STATE
        del self.staged[h]
        return OVL_OK


def switch_sequence(n_ops: int = 100, n_adapters: int = 4, corrupt: int = 3):
    """The timed switch workload: op i even -> activate adapter (i/2) mod 4
    (the corrupt one is re-staged instead and must fail its hash check);
    op i odd -> rollback.  Returns [(op, adapter_or_None)]."""
    ops = []
    for i in range(n_ops):
        if i % 2 == 0:
            a = (i // 2) % n_adapters
            ops.append(("stage_corrupt", a) if a == corrupt else ("activate", a))
        else:
            ops.append(("rollback", None))
    return ops


def switch_transcript(bkey: bytes, adapter_keys, scale: float = 2.0, n_ops: int = 100, corrupt: int = 3):
    """Expected (status, composition id hex) of every op of switch_sequence()."""
    m = SwitchModel(bkey)
    handles = {}
    for a, k in enumerate(adapter_keys):
        st, h = m.stage(k, ok=(a != corrupt))
        handles[a] = h
    out = []
    for op, a in switch_sequence(n_ops, len(adapter_keys), corrupt):
        if op == "activate":
            st, cid = m.activate([handles[a]], [scale])
        elif op == "stage_corrupt":
            st, _ = m.stage(adapter_keys[a], ok=False)
            cid = m.current_id()
        else:
            st, cid = m.rollback()
        out.append((op, a, st, cid.hex()))
    return out
