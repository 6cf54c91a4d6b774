"""The 32-layer stack of 8B-shape decoder blocks, every layer drawn from its
own seeds (base seed 10000 + 8 layer + proj), generated layer by layer in a
process pool.

Each worker quantizes one layer and returns its bytes padded to a multiple
of the 64 KiB digest leaf, with the leaf digests; the parent hands each layer
to a sink (for example a copy into its slot of a device buffer) as it arrives,
so the whole stack never has to exist in host memory.  The declared content
digest of the stack is the SHA-256 of all leaf digests in layer order, which
is the content digest of the concatenated padded layers.

Input generation only: none of the method's arithmetic lives here.
"""
from __future__ import annotations

import hashlib
import multiprocessing as mp
import os

import numpy as np

from . import (ALIGN, LEAF, PROJ, SHAPES_8B, Base, TensorDesc, _align, block_adapter, block_base, d_bytes,
               qs_bytes)


def layer_nbytes(quant: int, shapes=SHAPES_8B, projs=PROJ) -> int:
    """Bytes of one layer's base buffer, laid out as build_base lays it out."""
    off = 0
    for p in projs:
        d_out, d_in = shapes[p]
        off = _align(off + qs_bytes(quant, d_out, d_in))
        off = _align(off + d_bytes(d_out, d_in))
    return max(off, ALIGN)


def layer_stride(quant: int, shapes=SHAPES_8B) -> int:
    """Distance between consecutive layers in the stack (whole digest leaves)."""
    return (layer_nbytes(quant, shapes) + LEAF - 1) // LEAF * LEAF


def _build_layer(args):
    quant, layer, stride, shapes = args
    b = block_base(quant, layers=(layer,), shapes=shapes)
    padded = np.zeros(stride, dtype=np.uint8)
    padded[:b.buf.nbytes] = b.buf
    mv = memoryview(padded).cast("B")
    leaves = b"".join(hashlib.sha256(mv[i:i + LEAF]).digest() for i in range(0, stride, LEAF))
    return layer, padded, leaves, [(t.layer, t.proj, t.d_out, t.d_in, t.qs_off, t.d_off) for t in b.tensors]


class LayerStack:
    """Tensors (layer-major, offsets into the stack buffer) and declared digest
    of an n-layer stack whose bytes went to `sink(layer, offset, padded_bytes)`."""

    def __init__(self, quant: int, n_layers: int, sink, workers: int | None = None, shapes=SHAPES_8B):
        self.quant = quant
        self.n_layers = n_layers
        self.stride = layer_stride(quant, shapes)
        self.nbytes = n_layers * self.stride
        workers = workers or max(1, min(8, os.cpu_count() or 1, n_layers))
        leaves = [b""] * n_layers
        tensors = [None] * n_layers
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers) as pool:
            for layer, padded, lv, tt in pool.imap_unordered(_build_layer,
                                                             [(quant, l, self.stride, shapes)
                                                              for l in range(n_layers)]):
                sink(layer, layer * self.stride, padded)
                leaves[layer] = lv
                tensors[layer] = [TensorDesc(l, p, m, n, layer * self.stride + qo, layer * self.stride + do)
                                  for (l, p, m, n, qo, do) in tt]
        self.tensors = [t for tt in tensors for t in tt]
        self.digest = hashlib.sha256(b"".join(leaves)).digest()

    def as_base(self) -> Base:
        """A Base with this stack's tensor table (no host bytes)."""
        return Base(self.quant, self.tensors, np.zeros(0, dtype=np.uint8))


def stack_adapter(stack: LayerStack, adapter: int, rank: int):
    """Rank-`rank` LoRA on all tensors of every layer, each (layer, proj) with
    its own seeds (1000000 + 10000 adapter + 8 layer + proj)."""
    return block_adapter(stack.as_base(), adapter=adapter, rank=rank)
