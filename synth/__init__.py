"""Seeded synthetic inputs for the dual-path overlay library and its oracle.

This module only *produces inputs*: Gaussian base weights quantized into the
q8_0 / q4_0 byte layout, fp32 LoRA factors, activations, adapter-id draws and
the byte buffers that carry them.  It holds none of the method's arithmetic
(no dequantization, no GEMV, no LoRA application): both the CUDA library and
the CPU oracle consume the bytes produced here, each with its own code.

Workload shapes follow the configurations of the benchmark: a Llama-style
decoder block at 8B shape (hidden 4096, GQA k/v 1024, MLP 14336), base
weights ~ N(0, 0.02), LoRA factors ~ N(0, 0.01), activations ~ N(0, 1).

Byte layout (the library's written format; see the header ``include/ovl.h``):

* base buffer: per tensor a ``qs`` plane and a ``d`` plane, each starting on a
  256-byte boundary.  q8_0: ``qs`` is int8 ``[d_out][d_in]`` row-major.
  q4_0: ``qs`` is uint8 ``[d_out][d_in/2]``; byte ``p`` of a row holds element
  ``2p`` in bits 0-3 and element ``2p+1`` in bits 4-7, codes 0..15.
  ``d`` is IEEE binary16 ``[d_out][d_in/32]`` (one scale per 32-block).
  q4_K: ``qs`` as q4_0; the ``d`` plane holds one 16-byte header per
  256-weight super-block, ``[d_out][d_in/256][16]``: binary16 d, binary16 dmin,
  then the eight 6-bit sub-block scales as one 48-bit little-endian field
  (scale j in bits 6j..6j+5) and the eight 6-bit sub-block minimums the same
  way.  Same plane sizes as q4_0 (4.5 bits per weight).
* adapter payload: per target an fp32 ``A [r][d_in]`` and fp32 ``B [d_out][r]``,
  each starting on a 256-byte boundary.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np

QK = 32                      # weights per quantization block
QK_K = 256                   # weights per q4_K super-block
ALIGN = 256                  # plane / factor alignment inside a buffer
LEAF = 65536                 # leaf size of the content digest (bytes)

Q8_0 = 1
Q4_0 = 2
Q4_K = 3

PROJ = ("q", "k", "v", "o", "gate", "up", "down")
# (d_out, d_in) of the seven projections of one decoder block at 8B shape
SHAPES_8B = {
    "q": (4096, 4096),
    "k": (1024, 4096),
    "v": (1024, 4096),
    "o": (4096, 4096),
    "gate": (14336, 4096),
    "up": (14336, 4096),
    "down": (4096, 14336),
}


def _align(n: int, a: int = ALIGN) -> int:
    return (n + a - 1) // a * a


# --------------------------------------------------------------------------
# seeds
# --------------------------------------------------------------------------
def base_seed(layer: int, proj: int) -> int:
    return 10_000 + 8 * layer + proj


def adapter_seed(adapter: int, layer: int, proj: int) -> int:
    return 1_000_000 + 10_000 * adapter + 8 * layer + proj


def sparse_seed(adapter: int, layer: int, proj: int) -> int:
    return 5_000_000 + 10_000 * adapter + 8 * layer + proj


def x_seed(T: int, d_in: int) -> int:
    return 2000 + 16 * T + (0 if d_in == 4096 else 1)


ZIPF_SEED = 3000


def gaussian(rng: np.random.Generator, shape, sigma: float) -> np.ndarray:
    """N(0, sigma^2) drawn in float32, row-major (sigma is a standard deviation)."""
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma)


def round_half_away(v: np.ndarray) -> np.ndarray:
    return np.sign(v) * np.floor(np.abs(v) + np.float32(0.5))


# --------------------------------------------------------------------------
# quantizers (input generation only: the library never quantizes)
# --------------------------------------------------------------------------
def quantize_q8_0(w: np.ndarray):
    """float32 [m][n] -> (qs int8 [m][n], d uint16 bits [m][n/32]).

    d = fp16(max|w_block| / 127) (fp32 division, round-to-nearest-even into
    binary16); q = clamp(round_half_away(w / d), -127, 127); an all-zero block
    gets d = 0, q = 0.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    m, n = w.shape
    assert n % QK == 0
    blk = w.reshape(m, n // QK, QK)
    amax = np.abs(blk).max(axis=2)
    d16 = (amax / np.float32(127.0)).astype(np.float16)
    d32 = d16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d32 > 0, round_half_away(blk / d32), np.float32(0))
    q = np.clip(q, -127, 127).astype(np.int8).reshape(m, n)
    return q, d16.view(np.uint16)


def quantize_q4_0(w: np.ndarray):
    """float32 [m][n] -> (qs uint8 [m][n/2] packed nibbles, d uint16 bits).

    d = fp16(max|w_block| / 8); code = clamp(round_half_away(w / d) + 8, 0, 15),
    value d * (code - 8); element 2p in the low nibble of byte p.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    m, n = w.shape
    assert n % QK == 0
    blk = w.reshape(m, n // QK, QK)
    amax = np.abs(blk).max(axis=2)
    d16 = (amax / np.float32(8.0)).astype(np.float16)
    d32 = d16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d32 > 0, round_half_away(blk / d32), np.float32(0))
    code = np.clip(q + 8, 0, 15).astype(np.uint8).reshape(m, n)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, d16.view(np.uint16)


def pack6x8(v: np.ndarray) -> np.ndarray:
    """[..][8] integers 0..63 -> [..][6] bytes: one 48-bit little-endian field,
    value j in bits 6j..6j+5."""
    v = np.asarray(v, dtype=np.uint64)
    f = np.zeros(v.shape[:-1], dtype=np.uint64)
    for j in range(8):
        f |= v[..., j] << np.uint64(6 * j)
    return np.stack([((f >> np.uint64(8 * k)) & np.uint64(0xFF)).astype(np.uint8) for k in range(6)], axis=-1)


def quantize_q4_k(w: np.ndarray):
    """float32 [m][n] -> (qs uint8 [m][n/2] packed nibbles, headers uint8 [m][n/16]).

    Per 32-weight sub-block j (fp32 arithmetic): lo_j = min(min w, 0),
    step_j = (max w - lo_j) / 15, zero-point mu_j = -lo_j.  Per super-block:
    d = fp16(max_j step_j / 63), dmin = fp16(max_j mu_j / 63),
    sc_j = clamp(round_half_away(step_j / d), 0, 63),
    m_j = clamp(round_half_away(mu_j / dmin), 0, 63) (0 where d or dmin is 0);
    code = clamp(round_half_away((w + dmin*m_j) / (d*sc_j)), 0, 15) (0 where
    d*sc_j is 0), value d*sc_j*code - dmin*m_j.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    m, n = w.shape
    assert n % QK_K == 0
    blk = w.reshape(m, n // QK_K, 8, QK)
    lo = np.minimum(blk.min(axis=3), np.float32(0))
    step = (blk.max(axis=3) - lo) / np.float32(15.0)
    mu = -lo
    d16 = (step.max(axis=2) / np.float32(63.0)).astype(np.float16)
    dm16 = (mu.max(axis=2) / np.float32(63.0)).astype(np.float16)
    d32 = d16.astype(np.float32)[..., None]
    dm32 = dm16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d32 > 0, round_half_away(step / d32), np.float32(0))
        mq = np.where(dm32 > 0, round_half_away(mu / dm32), np.float32(0))
    sc = np.clip(sc, 0, 63)
    mq = np.clip(mq, 0, 63)
    eff_scale = (d32 * sc)[..., None]
    eff_min = (dm32 * mq)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(eff_scale > 0, round_half_away((blk + eff_min) / eff_scale), np.float32(0))
    code = np.clip(q, 0, 15).astype(np.uint8).reshape(m, n)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    hdr = np.zeros((m, n // QK_K, 16), dtype=np.uint8)
    hdr[..., 0:2] = d16.view(np.uint16)[..., None].view(np.uint8).reshape(m, n // QK_K, 2)
    hdr[..., 2:4] = dm16.view(np.uint16)[..., None].view(np.uint8).reshape(m, n // QK_K, 2)
    hdr[..., 4:10] = pack6x8(sc.astype(np.int64))
    hdr[..., 10:16] = pack6x8(mq.astype(np.int64))
    return packed, hdr.reshape(m, n // 16)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# buffers
# --------------------------------------------------------------------------
@dataclass
class TensorDesc:
    layer: int
    proj: int
    d_out: int
    d_in: int
    qs_off: int
    d_off: int


@dataclass
class Base:
    quant: int
    tensors: list
    buf: np.ndarray            # uint8, the whole base
    # per-tensor views (host) for convenience of tests: (qs, d_bits)
    planes: list = field(default_factory=list)


def qs_bytes(quant: int, d_out: int, d_in: int) -> int:
    return d_out * d_in if quant == Q8_0 else d_out * d_in // 2


def d_bytes(d_out: int, d_in: int) -> int:
    return d_out * (d_in // QK) * 2


def build_base(quant: int, items) -> Base:
    """items: iterable of (layer, proj, w_float32[d_out][d_in]) -> Base."""
    qz = {Q8_0: quantize_q8_0, Q4_0: quantize_q4_0, Q4_K: quantize_q4_k}[quant]
    enc = []
    off = 0
    descs = []
    for layer, proj, w in items:
        qs, d = qz(w)
        d_out, d_in = w.shape
        qs_off = off
        off = _align(off + qs.nbytes)
        d_off = off
        off = _align(off + d.nbytes)
        descs.append(TensorDesc(layer, proj, d_out, d_in, qs_off, d_off))
        enc.append((qs, d))
    buf = np.zeros(max(off, ALIGN), dtype=np.uint8)
    for t, (qs, d) in zip(descs, enc):
        buf[t.qs_off:t.qs_off + qs.nbytes] = qs.reshape(-1).view(np.uint8)
        buf[t.d_off:t.d_off + d.nbytes] = d.reshape(-1).view(np.uint8)
    b = Base(quant, descs, buf)
    b.planes = [base_planes(b, i) for i in range(len(descs))]
    return b


def base_planes(base: Base, i: int):
    """(qs, d_bits) numpy views of tensor i inside the base buffer."""
    t = base.tensors[i]
    nq = qs_bytes(base.quant, t.d_out, t.d_in)
    qs = base.buf[t.qs_off:t.qs_off + nq]
    if base.quant == Q8_0:
        qs = qs.view(np.int8).reshape(t.d_out, t.d_in)
    else:
        qs = qs.reshape(t.d_out, t.d_in // 2)
    if base.quant == Q4_K:
        hdr = base.buf[t.d_off:t.d_off + d_bytes(t.d_out, t.d_in)]
        return qs, hdr.reshape(t.d_out, t.d_in // QK_K, 16)
    d = base.buf[t.d_off:t.d_off + d_bytes(t.d_out, t.d_in)].view(np.uint16)
    return qs, d.reshape(t.d_out, t.d_in // QK)


@dataclass
class Adapter:
    targets: list              # tensor indices into the base
    ranks: list
    a_off: list
    b_off: list
    payload: np.ndarray        # uint8
    factors: list              # [(A fp32 [r][d_in], B fp32 [d_out][r])]
    required_base: bytes = b"\0" * 32


def build_adapter(base: Base, targets, ranks, factors, required_base=None) -> Adapter:
    """Pack fp32 factors [(A, B)] for the given target tensors into one payload."""
    off = 0
    a_off, b_off = [], []
    for (A, B) in factors:
        a_off.append(off)
        off = _align(off + A.nbytes)
        b_off.append(off)
        off = _align(off + B.nbytes)
    payload = np.zeros(max(off, ALIGN), dtype=np.uint8)
    for (A, B), ao, bo in zip(factors, a_off, b_off):
        payload[ao:ao + A.nbytes] = np.ascontiguousarray(A, np.float32).reshape(-1).view(np.uint8)
        payload[bo:bo + B.nbytes] = np.ascontiguousarray(B, np.float32).reshape(-1).view(np.uint8)
    return Adapter(list(targets), list(ranks), a_off, b_off, payload,
                   [(np.ascontiguousarray(A, np.float32), np.ascontiguousarray(B, np.float32))
                    for A, B in factors],
                   required_base if required_base is not None else b"\0" * 32)


@dataclass
class SparseAdapter:
    targets: list              # tensor indices into the base
    nnz: list
    idx_off: list
    val_off: list
    payload: np.ndarray        # uint8
    entries: list              # [(idx uint32 [nnz], val_bits uint16 [nnz])] per target
    required_base: bytes = b"\0" * 32


def build_sparse_adapter(targets, entries, required_base=None) -> SparseAdapter:
    """Pack index-value pairs [(idx uint32, val_bits uint16)] per target into one
    payload: per target a uint32 index plane and a binary16 value plane, each
    starting on a 256-byte boundary."""
    off = 0
    io, vo = [], []
    for idx, val in entries:
        io.append(off)
        off = _align(off + 4 * len(idx))
        vo.append(off)
        off = _align(off + 2 * len(val))
    payload = np.zeros(max(off, ALIGN), dtype=np.uint8)
    for (idx, val), a, b in zip(entries, io, vo):
        payload[a:a + 4 * len(idx)] = np.ascontiguousarray(idx, np.uint32).view(np.uint8)
        payload[b:b + 2 * len(val)] = np.ascontiguousarray(val, np.uint16).view(np.uint8)
    return SparseAdapter(list(targets), [len(i) for i, _ in entries], io, vo, payload,
                         [(np.ascontiguousarray(i, np.uint32), np.ascontiguousarray(v, np.uint16)) for i, v in entries],
                         required_base if required_base is not None else b"\0" * 32)


def dare_entries(rng: np.random.Generator, d_out: int, d_in: int, keep: float = 0.01, sigma: float = 1e-4):
    """A DARE-style sparse task vector: a dense delta ~ N(0, sigma) of which each
    element is kept with probability `keep` (a Bernoulli process, drawn as
    geometric gaps between kept positions) and rescaled by 1/keep, stored as
    strictly increasing flat indices row*d_in + col and binary16 values."""
    total = d_out * d_in
    pos = []
    at = -1
    while True:
        gaps = rng.geometric(keep, size=max(16, int(total * keep * 1.1) + 16))
        cand = at + np.cumsum(gaps)
        pos.append(cand[cand < total])
        if cand[-1] >= total:
            break
        at = int(cand[-1])
    idx = np.concatenate(pos).astype(np.uint32)
    val = (gaussian(rng, (idx.size,), sigma) / np.float32(keep)).astype(np.float16)
    return idx, val.view(np.uint16)


def block_sparse_adapter(base: Base, adapter: int, keep: float = 0.01, which=None) -> SparseAdapter:
    """DARE-style sparse overlay (density `keep`) on every tensor of `base` (or `which`)."""
    idx = list(range(len(base.tensors))) if which is None else list(which)
    entries = []
    for i in idx:
        t = base.tensors[i]
        rng = np.random.default_rng(sparse_seed(adapter, t.layer, t.proj))
        entries.append(dare_entries(rng, t.d_out, t.d_in, keep))
    return build_sparse_adapter(idx, entries)


def content_digest(buf: np.ndarray) -> bytes:
    """Declared digest of a byte buffer: SHA-256 over the concatenated SHA-256
    digests of consecutive 64 KiB leaves (last leaf may be short).  This is the
    value a caller declares when it hands bytes to the library."""
    mv = memoryview(np.ascontiguousarray(buf).view(np.uint8)).cast("B")
    top = hashlib.sha256()
    for i in range(0, len(mv), LEAF):
        top.update(hashlib.sha256(mv[i:i + LEAF]).digest())
    return top.digest()


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
def single_layer_256(seed_a: int = 0, seed_b: int = 1, quant: int = Q8_0):
    """256x256 layer, rank-8 adapters A (rng seed 0) and B (rng seed 1), s = 2.0.

    rng(0) draws W, then adapter A's A-factor, then its B-factor, then x (fp32);
    adapter B's factors come from rng(1).
    """
    rng = np.random.default_rng(seed_a)
    W = gaussian(rng, (256, 256), 0.02)
    A1 = gaussian(rng, (8, 256), 0.01)
    B1 = gaussian(rng, (256, 8), 0.01)
    x = gaussian(rng, (1, 256), 1.0)
    rng2 = np.random.default_rng(seed_b)
    A2 = gaussian(rng2, (8, 256), 0.01)
    B2 = gaussian(rng2, (256, 8), 0.01)
    base = build_base(quant, [(0, 0, W)])
    ad_a = build_adapter(base, [0], [8], [(A1, B1)])
    ad_b = build_adapter(base, [0], [8], [(A2, B2)])
    return base, ad_a, ad_b, x, 2.0


def block_base(quant: int, layers=(0,), shapes=SHAPES_8B, projs=PROJ) -> Base:
    items = []
    for layer in layers:
        for p in projs:
            pi = PROJ.index(p)
            d_out, d_in = shapes[p]
            rng = np.random.default_rng(base_seed(layer, pi))
            items.append((layer, pi, gaussian(rng, (d_out, d_in), 0.02)))
    return build_base(quant, items)


def block_adapter(base: Base, adapter: int, rank: int, which=None) -> Adapter:
    """Rank-`rank` LoRA on every tensor of `base` (or on the indices `which`)."""
    idx = list(range(len(base.tensors))) if which is None else list(which)
    factors = []
    for i in idx:
        t = base.tensors[i]
        rng = np.random.default_rng(adapter_seed(adapter, t.layer, t.proj))
        A = gaussian(rng, (rank, t.d_in), 0.01)
        B = gaussian(rng, (t.d_out, rank), 0.01)
        factors.append((A, B))
    return build_adapter(base, idx, [rank] * len(idx), factors)


def activations(T: int, d_in: int, seed=None) -> np.ndarray:
    """x ~ N(0,1) float32 [T][d_in]."""
    rng = np.random.default_rng(x_seed(T, d_in) if seed is None else seed)
    return gaussian(rng, (T, d_in), 1.0)


def zipf_ids(n_requests: int = 64, n_adapters: int = 16, a: float = 1.1, seed: int = ZIPF_SEED):
    """Finite Zipf draw of adapter ids: p_k proportional to k^-a, k = 1..n, id = k-1."""
    k = np.arange(1, n_adapters + 1, dtype=np.float64)
    p = k ** (-a)
    p /= p.sum()
    rng = np.random.default_rng(seed)
    return rng.choice(n_adapters, size=n_requests, p=p).astype(np.int32)


def segments(ids: np.ndarray):
    """Group requests by adapter id (stable, ascending id).

    Returns (perm, seg_offsets, seg_slot): perm[j] = original request index of
    the j-th grouped row; segment s covers grouped rows seg_offsets[s] ..
    seg_offsets[s+1]-1 and uses table slot seg_slot[s].
    """
    ids = np.asarray(ids, dtype=np.int32)
    perm = np.argsort(ids, kind="stable").astype(np.int32)
    sorted_ids = ids[perm]
    slots, starts = np.unique(sorted_ids, return_index=True)
    offsets = np.append(starts, len(ids)).astype(np.int32)
    return perm, offsets, slots.astype(np.int32)
