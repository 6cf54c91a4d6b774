"""Python binding of libovl (the C ABI declared in include/ovl.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  Importing this package loads ``libovl.so`` from this directory and
raises ImportError if it has not been built (``python
quantized_base_lora_gb300/build.py``); there is no fallback implementation.

Device buffers and streams are passed as integers (e.g. ``tensor.data_ptr()``
and ``torch.cuda.current_stream().cuda_stream``).  Functions keep the C names
and return the ovl_status code first; use :func:`check` to raise on errors.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libovl.so")

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
OVL_E_CUDA = -12
OVL_E_DEVICE_TIMEOUT = -13
STATUS_NAMES = {v: k for k, v in list(globals().items()) if k.startswith("OVL_E_") or k == "OVL_OK"}

OVL_Q8_0, OVL_Q4_0, OVL_Q4_K = 1, 2, 3
OVL_F32, OVL_BF16 = 1, 2
OVL_MODE_STACK, OVL_MODE_TABLE = 1, 2
OVL_PATH_DUAL, OVL_PATH_JIT = 1, 2
OVL_SWITCH_REJECT, OVL_SWITCH_DRAIN = 1, 2
OVL_ADAPTER_LORA, OVL_ADAPTER_SPARSE = 1, 2
(OVL_PHASE_VALIDATION, OVL_PHASE_ALLOCATION, OVL_PHASE_STAGING,
 OVL_PHASE_CHECKSUM, OVL_PHASE_SWAP, OVL_PHASE_DEVICE_WAIT) = 1, 2, 3, 4, 5, 6
OVL_MAX_STACK, OVL_MAX_TABLE, OVL_MAX_RANK, OVL_MAX_TOTAL_RANK, OVL_MAX_T, OVL_MAX_SEGMENTS = 8, 32, 128, 256, 512, 64


class ovl_tensor_desc(C.Structure):
    _fields_ = [("layer", C.c_uint32), ("proj", C.c_uint32), ("d_out", C.c_uint32), ("d_in", C.c_uint32),
                ("qs_off", C.c_uint64), ("d_off", C.c_uint64)]


class ovl_base_desc(C.Structure):
    _fields_ = [("quant", C.c_uint32), ("n_tensors", C.c_uint32), ("tensors", C.POINTER(ovl_tensor_desc))]


class ovl_adapter_desc(C.Structure):
    _fields_ = [("n_targets", C.c_uint32), ("target_tensor", C.POINTER(C.c_uint32)),
                ("rank", C.POINTER(C.c_uint32)), ("a_off", C.POINTER(C.c_uint64)),
                ("b_off", C.POINTER(C.c_uint64)), ("required_base_digest", C.c_uint8 * 32)]


class ovl_sparse_desc(C.Structure):
    _fields_ = [("n_targets", C.c_uint32), ("target_tensor", C.POINTER(C.c_uint32)),
                ("nnz", C.POINTER(C.c_uint32)), ("idx_off", C.POINTER(C.c_uint64)),
                ("val_off", C.POINTER(C.c_uint64)), ("required_base_digest", C.c_uint8 * 32)]


class ovl_state(C.Structure):
    _fields_ = [("composition_id", C.c_uint8 * 32), ("base_digest", C.c_uint8 * 32),
                ("quant", C.c_uint32), ("mode", C.c_uint32), ("n_entries", C.c_uint32),
                ("has_previous", C.c_uint32), ("epoch", C.c_uint64), ("arena_used", C.c_uint64),
                ("arena_bytes", C.c_uint64), ("n_staged", C.c_uint32), ("base_loaded", C.c_uint32)]


class ovl_entry(C.Structure):
    _fields_ = [("handle", C.c_uint64), ("adapter_key", C.c_uint8 * 32), ("scale", C.c_float),
                ("total_rank", C.c_uint32)]


class ovl_manifest_entry(C.Structure):
    _fields_ = [("name", C.c_char * 64), ("file_digest", C.c_uint8 * 32), ("required_base_digest", C.c_uint8 * 32),
                ("type", C.c_uint32), ("load_order", C.c_uint32), ("rank", C.c_uint32), ("n_targets", C.c_uint32),
                ("has_required_base", C.c_uint32), ("merge_weight", C.c_float)]


class ovl_manifest(C.Structure):
    _fields_ = [("base_digest", C.c_uint8 * 32), ("quant", C.c_uint32), ("mode", C.c_uint32),
                ("n_adapters", C.c_uint32), ("adapters", ovl_manifest_entry * 32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libovl.so is not built ({LIB_PATH}); run python quantized_base_lora_gb300/build.py")
    lib = C.CDLL(LIB_PATH)
    P, U32, U64, I32, SZ = C.c_void_p, C.c_uint32, C.c_uint64, C.c_int32, C.c_size_t
    B32 = C.POINTER(C.c_uint8)
    sig = {
        "ovl_create": ([C.POINTER(P), C.c_int, P, SZ, U32], I32),
        "ovl_destroy": ([P], I32),
        "ovl_load_base": ([P, C.POINTER(ovl_base_desc), P, SZ, B32, P], I32),
        "ovl_stage_adapter": ([P, C.POINTER(ovl_adapter_desc), P, SZ, B32, C.POINTER(U64)], I32),
        "ovl_stage_sparse": ([P, C.POINTER(ovl_sparse_desc), P, SZ, B32, C.POINTER(U64)], I32),
        "ovl_unstage_adapter": ([P, U64], I32),
        "ovl_activate": ([P, C.POINTER(U64), C.POINTER(C.c_float), U32, U32, B32], I32),
        "ovl_rollback": ([P, B32], I32),
        "ovl_linear_forward": ([P, U32, P, U32, U32, P, U32, P, SZ, P], I32),
        "ovl_materialize_layer": ([P, U32, P, SZ, P], I32),
        "ovl_linear_forward_multi": ([P, U32, C.POINTER(U32), P, U32, U32, C.POINTER(P), P], I32),
        "ovl_segmented_forward": ([P, U32, P, U32, U32, C.POINTER(I32), C.POINTER(I32), U32,
                                   C.POINTER(I32), P, P], I32),
        "ovl_base_digest": ([P, B32, P], I32),
        "ovl_get_state": ([P, C.POINTER(ovl_state)], I32),
        "ovl_get_entry": ([P, U32, C.POINTER(ovl_entry)], I32),
        "ovl_check_device": ([P, P], I32),
        "ovl_debug_inject": ([P, U32, I32], I32),
        "ovl_last_error": ([P], C.c_char_p),
        "ovl_sha256": ([P, SZ, B32], I32),
        "ovl_content_digest": ([P, SZ, B32], I32),
        "ovl_version": ([], C.c_char_p),
        "ovl_dualpath_forward_noalloc": ([P, P, U32, U32, U32, C.POINTER(P), C.POINTER(P), C.POINTER(U32),
                                          C.POINTER(C.c_float), U32, P, U32, U32, P, P], I32),
        "ovl_stage_activations": ([P, P, SZ, P], I32),
        "ovl_manifest_parse": ([C.c_char_p, SZ, C.POINTER(ovl_manifest)], I32),
        "ovl_activate_manifest": ([P, C.c_char_p, SZ, B32], I32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()
EXPORTED = ("ovl_create", "ovl_destroy", "ovl_load_base", "ovl_stage_adapter", "ovl_stage_sparse", "ovl_unstage_adapter",
            "ovl_activate", "ovl_rollback", "ovl_linear_forward", "ovl_linear_forward_multi", "ovl_materialize_layer",
            "ovl_segmented_forward", "ovl_base_digest", "ovl_get_state", "ovl_get_entry",
            "ovl_check_device", "ovl_debug_inject", "ovl_last_error", "ovl_sha256",
            "ovl_content_digest", "ovl_version", "ovl_dualpath_forward_noalloc", "ovl_stage_activations",
            "ovl_manifest_parse", "ovl_activate_manifest")


class OvlError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _b32(buf: bytes | None = None):
    arr = (C.c_uint8 * 32)()
    if buf is not None:
        if len(buf) != 32:
            raise ValueError("digest must be 32 bytes")
        C.memmove(arr, buf, 32)
    return arr


def _u32s(v):
    return (C.c_uint32 * len(v))(*[int(i) for i in v])


def _u64s(v):
    return (C.c_uint64 * len(v))(*[int(i) for i in v])


def _i32s(v):
    return (C.c_int32 * len(v))(*[int(i) for i in v])


def ovl_last_error(ctx) -> str:
    return (lib.ovl_last_error(ctx) or b"").decode()


def check(status: int, ctx=None):
    if status != OVL_OK:
        raise OvlError(status, ovl_last_error(ctx))
    return status


def ovl_version() -> str:
    return lib.ovl_version().decode()


def ovl_sha256(data: bytes) -> bytes:
    out = _b32()
    buf = C.create_string_buffer(bytes(data), len(data))
    check(lib.ovl_sha256(buf, len(data), out))
    return bytes(out)


def ovl_content_digest(data) -> bytes:
    """data: bytes or a C-contiguous numpy uint8 array (host)."""
    out = _b32()
    if isinstance(data, (bytes, bytearray)):
        buf = C.create_string_buffer(bytes(data), len(data))
        check(lib.ovl_content_digest(buf, len(data), out))
    else:
        check(lib.ovl_content_digest(data.ctypes.data, data.nbytes, out))
    return bytes(out)


def ovl_create(device: int, arena_ptr: int, arena_bytes: int, policy: int = OVL_SWITCH_REJECT):
    ctx = C.c_void_p()
    st = lib.ovl_create(C.byref(ctx), int(device), C.c_void_p(arena_ptr), int(arena_bytes), int(policy))
    return st, ctx


def ovl_destroy(ctx) -> int:
    return lib.ovl_destroy(ctx)


def ovl_load_base(ctx, quant: int, tensors, base_ptr: int, nbytes: int, digest: bytes, stream: int = 0) -> int:
    """tensors: iterable of (layer, proj, d_out, d_in, qs_off, d_off)."""
    tensors = list(tensors)
    arr = (ovl_tensor_desc * max(1, len(tensors)))()
    for i, t in enumerate(tensors):
        arr[i] = ovl_tensor_desc(*[int(v) for v in t])
    desc = ovl_base_desc(int(quant), len(tensors), arr)
    return lib.ovl_load_base(ctx, C.byref(desc), C.c_void_p(base_ptr), int(nbytes), _b32(digest),
                             C.c_void_p(stream))


def ovl_stage_adapter(ctx, targets, ranks, a_off, b_off, payload, digest: bytes, required_base: bytes | None = None):
    """payload: C-contiguous numpy uint8 array (host).  Returns (status, handle)."""
    n = len(targets)
    desc = ovl_adapter_desc(n, _u32s(targets), _u32s(ranks), _u64s(a_off), _u64s(b_off),
                            _b32(required_base or b"\0" * 32))
    h = C.c_uint64(0)
    st = lib.ovl_stage_adapter(ctx, C.byref(desc), C.c_void_p(payload.ctypes.data), int(payload.nbytes),
                               _b32(digest), C.byref(h))
    return st, int(h.value)


def ovl_stage_sparse(ctx, targets, nnz, idx_off, val_off, payload, digest: bytes, required_base: bytes | None = None):
    """payload: C-contiguous numpy uint8 array (host).  Returns (status, handle)."""
    n = len(targets)
    desc = ovl_sparse_desc(n, _u32s(targets), _u32s(nnz), _u64s(idx_off), _u64s(val_off),
                           _b32(required_base or b"\0" * 32))
    h = C.c_uint64(0)
    st = lib.ovl_stage_sparse(ctx, C.byref(desc), C.c_void_p(payload.ctypes.data), int(payload.nbytes),
                              _b32(digest), C.byref(h))
    return st, int(h.value)


def ovl_unstage_adapter(ctx, h: int) -> int:
    return lib.ovl_unstage_adapter(ctx, int(h))


def ovl_activate(ctx, handles, scales, mode: int = OVL_MODE_STACK):
    handles, scales = list(handles), list(scales)
    out = _b32()
    st = lib.ovl_activate(ctx, _u64s(handles) if handles else None,
                          (C.c_float * len(scales))(*scales) if scales else None, len(handles), int(mode), out)
    return st, bytes(out)


def ovl_rollback(ctx):
    out = _b32()
    st = lib.ovl_rollback(ctx, out)
    return st, bytes(out)


def ovl_linear_forward(ctx, tensor: int, x_ptr: int, x_dtype: int, T: int, y_ptr: int,
                       path: int = OVL_PATH_DUAL, scratch_ptr: int = 0, scratch_bytes: int = 0,
                       stream: int = 0) -> int:
    return lib.ovl_linear_forward(ctx, int(tensor), int(x_ptr), int(x_dtype), int(T), int(y_ptr), int(path),
                                  int(scratch_ptr), int(scratch_bytes), int(stream))


def ovl_linear_forward_multi(ctx, tensors, x_ptr: int, x_dtype: int, T: int, y_ptrs, stream: int = 0) -> int:
    n = len(tensors)
    return lib.ovl_linear_forward_multi(ctx, n, (C.c_uint32 * n)(*tensors), int(x_ptr), int(x_dtype), int(T),
                                        (C.c_void_p * n)(*map(int, y_ptrs)), int(stream))


def ovl_materialize_layer(ctx, tensor: int, scratch_ptr: int, scratch_bytes: int, stream: int = 0) -> int:
    return lib.ovl_materialize_layer(ctx, int(tensor), C.c_void_p(scratch_ptr), int(scratch_bytes),
                                     C.c_void_p(stream))


def ovl_segmented_forward(ctx, tensor: int, x_ptr: int, x_dtype: int, T: int, seg_offsets, seg_slot, perm,
                          y_ptr: int, stream: int = 0) -> int:
    n_seg = len(seg_slot)
    return lib.ovl_segmented_forward(ctx, int(tensor), C.c_void_p(x_ptr), int(x_dtype), int(T),
                                     _i32s(seg_offsets), _i32s(seg_slot), n_seg, _i32s(perm),
                                     C.c_void_p(y_ptr), C.c_void_p(stream))


def ovl_base_digest(ctx, stream: int = 0):
    out = _b32()
    st = lib.ovl_base_digest(ctx, out, C.c_void_p(stream))
    return st, bytes(out)


def ovl_get_state(ctx):
    s = ovl_state()
    st = lib.ovl_get_state(ctx, C.byref(s))
    d = {f: getattr(s, f) for f, _ in ovl_state._fields_}
    d["composition_id"] = bytes(s.composition_id)
    d["base_digest"] = bytes(s.base_digest)
    return st, d


def ovl_get_entry(ctx, i: int):
    e = ovl_entry()
    st = lib.ovl_get_entry(ctx, int(i), C.byref(e))
    return st, {"handle": e.handle, "adapter_key": bytes(e.adapter_key), "scale": e.scale,
                "total_rank": e.total_rank}


def ovl_check_device(ctx, stream: int = 0) -> int:
    return lib.ovl_check_device(ctx, C.c_void_p(stream))


def ovl_debug_inject(ctx, phase: int, code: int) -> int:
    return lib.ovl_debug_inject(ctx, int(phase), int(code))


def ovl_manifest_parse(text):
    """Parse a composition manifest (str or bytes) without a device: (status,
    dict with base_digest, quant, mode and the adapters in load order)."""
    raw = text.encode() if isinstance(text, str) else bytes(text)
    m = ovl_manifest()
    st = lib.ovl_manifest_parse(raw, len(raw), C.byref(m))
    if st != 0:
        return st, None
    ads = []
    for i in range(m.n_adapters):
        e = m.adapters[i]
        ads.append({"name": e.name.decode(), "file_digest": bytes(e.file_digest), "type": e.type,
                    "load_order": e.load_order, "merge_weight": e.merge_weight, "rank": e.rank,
                    "n_targets": e.n_targets,
                    "required_base_digest": bytes(e.required_base_digest) if e.has_required_base else None})
    return st, {"base_digest": bytes(m.base_digest), "quant": m.quant, "mode": m.mode, "adapters": ads}


def ovl_activate_manifest(ctx, text):
    raw = text.encode() if isinstance(text, str) else bytes(text)
    out = _b32()
    st = lib.ovl_activate_manifest(ctx, raw, len(raw), out)
    return st, bytes(out)


def ovl_stage_activations(dst_ptr: int, src_host_ptr: int, nbytes: int, stream: int = 0) -> int:
    return lib.ovl_stage_activations(C.c_void_p(dst_ptr), C.c_void_p(src_host_ptr), int(nbytes), C.c_void_p(stream))


def ovl_dualpath_forward_noalloc(qs_ptr: int, d_ptr: int, quant: int, d_out: int, d_in: int, A_ptrs, B_ptrs,
                                 ranks, scales, x_ptr: int, x_dtype: int, T: int, y_ptr: int,
                                 stream: int = 0) -> int:
    """Allocation-free dual-path forward (see include/ovl.h); factor pointers are device addresses."""
    n = len(ranks)
    Ap = (C.c_void_p * max(n, 1))(*[C.c_void_p(p) for p in A_ptrs])
    Bp = (C.c_void_p * max(n, 1))(*[C.c_void_p(p) for p in B_ptrs])
    return lib.ovl_dualpath_forward_noalloc(C.c_void_p(qs_ptr), C.c_void_p(d_ptr), int(quant), int(d_out), int(d_in),
                                            Ap, Bp, _u32s(ranks) if n else None,
                                            (C.c_float * n)(*scales) if n else None, n, C.c_void_p(x_ptr),
                                            int(x_dtype), int(T), C.c_void_p(y_ptr), C.c_void_p(stream))
