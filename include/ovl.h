/*
 * ovl.h — C ABI of the dual-path quantized-base + LoRA overlay library (libovl).
 *
 * The library evaluates the linear layers of a transformer whose base weights
 * are an immutable block-quantized buffer (q8_0, q4_0 or q4_K), with an ordered
 * stack of overlays - low-rank adapters or sparse index-value overlays - applied
 * without ever being merged into the base:
 *
 *     y = deq(W_q) x + sum_k s_k dW_k x                              (dual path)
 *     S = deq(W_q) + sum_k s_k dW_k ;  y = S x      (per-layer JIT, S discarded)
 *
 * with dW_k = B_k A_k for a low-rank adapter (evaluated as B_k (A_k x) on the
 * dual path) and dW_k = the scattered values of a sparse overlay.
 *
 * Sources, cited by page title and section:
 *   [OVR]    "We propose a content-addressed overlay system ..." report
 *            (mikekappel.com/reports/runtime/we-propose-a-content-addressed-overlay-system/)
 *   [DTD]    "Deep Technical Design: Exact, Atomic, Reversible Specialist Overlays on
 *            Quantized Transformer Bases"
 *            (mikekappel.com/reports/runtime/quantized-adapter-runtime-architecture/)
 *   [MODELD] contenox modeld blueprint "LoRA adapters"
 *            (contenox.com/docs/development/blueprints/modeld/lora-adapters/)
 *
 * Conventions for every entry point
 *   - Returns ovl_status: 0 = OVL_OK, negative = error.  Nothing throws, aborts or
 *     exits.  On error the library state is exactly what it was before the call
 *     (strong guarantee; [OVR] §"Explicit Correctness and Atomicity Invariants",
 *     Atomic Update) and ovl_last_error() describes the failure.  Errors are
 *     deterministic for a given input ([OVR] §"Checksum Verification").
 *   - "device pointer" = a CUDA global-memory address on the context's device,
 *     owned by the caller and valid for the duration stated.  "host pointer" =
 *     ordinary process memory.  Streams are cudaStream_t passed as void*
 *     (NULL = the legacy default stream).  The library never calls cudaMalloc or
 *     cudaFree: every byte of device memory it uses comes from the caller's
 *     arena (ovl_create) or the caller's argument buffers.
 *   - Work enqueued on a stream is asynchronous; a device-side failure (a bounded
 *     wait that ran out) is latched in a status word that ovl_check_device() reads.
 *   - Calls on one context are serialized by an internal mutex; forward calls
 *     must be issued on one stream (or otherwise stream-ordered) because they
 *     share the context's device workspace.
 *
 * Byte layouts (written format shared by every producer and consumer of the bytes)
 *   Base buffer (device, caller-owned, never written by the library):
 *     per tensor a qs plane at qs_off and a d plane at d_off (both multiples of 16).
 *       q8_0: qs = int8 [d_out][d_in] row-major; weight = d * q.
 *       q4_0: qs = uint8 [d_out][d_in/2]; byte p of a row holds element 2p in bits 0-3
 *             and element 2p+1 in bits 4-7; codes 0..15; weight = d * (code - 8).
 *       d   = IEEE binary16, little-endian, [d_out][d_in/32], one scale per 32 weights.
 *     ([DTD] §5 "Quantized-Base Numerical Analysis": 32-weight blocks, one f16 scale.)
 *       q4_K: qs as q4_0.  The d plane holds one 16-byte header per 256-weight
 *             super-block, [d_out][d_in/256][16]: bytes 0-1 d and bytes 2-3 dmin
 *             (IEEE binary16), bytes 4-9 the eight 6-bit sub-block scales sc_j as
 *             one 48-bit little-endian field (sc_j in bits 6j..6j+5), bytes 10-15
 *             the eight 6-bit sub-block minimums m_j the same way.  Weight c of a
 *             row = d * sc_j * code - dmin * m_j with j = (c mod 256) / 32.
 *             ([DTD] §5: 256-weight super-blocks of 8 sub-blocks of 32, a 6-bit
 *             scale and a 6-bit minimum per sub-block, two f16 super-block
 *             scales, 4.5 bits per weight; the byte packing is this library's.)
 *             d_in must be a multiple of 256.
 *     The d plane, rounded up to a multiple of 16 bytes, must lie inside the buffer
 *     (d_out * d_in / 16 bytes for every profile).
 *     d_in must be a multiple of 32.
 *   Adapter payload (host, copied into the arena by ovl_stage_adapter):
 *     per target tensor t: A_t = float32 [rank][d_in] at a_off, B_t = float32
 *     [d_out][rank] at b_off, offsets multiples of 16 ([OVR] §"Memory, Byte, and
 *     Latency Formulas": LoRA stores A (r x n) and B (m x r)).
 *   Activations x: row-major [T][d_in] float32 or bfloat16.  Outputs y: float32 [T][d_out].
 *
 * Content digest (the "declared digest" arguments)
 *   SHA-256 (FIPS 180-4) over the concatenation of the SHA-256 digests of
 *   consecutive 65536-byte leaves of the bytes (the last leaf may be shorter;
 *   zero bytes -> SHA-256 of the empty string).  ([OVR] §"Checksum Verification";
 *   [DTD] §6 CHECKSUM VERIFICATION.)
 *
 * Composition identity (32 bytes, little-endian fields)
 *   base_key    = SHA256("OVLB" | base_digest | u32 quant | u32 n_tensors |
 *                        per tensor u32 layer,proj,d_out,d_in | u64 qs_off,d_off)
 *   adapter_key = SHA256("OVLA" | payload_digest | u32 n_targets |
 *                        per target u32 tensor,rank | u64 a_off,b_off)
 *   id          = SHA256("OVLC" | runtime_tag[16] | base_key | u32 mode | u32 K |
 *                        per entry adapter_key | u32 bits_of_float(scale))
 *   runtime_tag = "ovl-gb300 v1" padded with zero bytes to 16; an empty stack has
 *   mode OVL_MODE_STACK.  ([OVR] §"Composition Identity and Manifest Schema";
 *   [DTD] §3; [MODELD] §"Runtime Identity and Cache Safety".)
 */
#ifndef OVL_H
#define OVL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ovl_ctx ovl_ctx;
typedef int32_t ovl_status;
typedef uint64_t ovl_adapter_h;   /* 0 is never a valid handle */

enum {
  OVL_OK = 0,
  OVL_E_ARG = -1,            /* bad argument / unknown handle / non-finite scale */
  OVL_E_HASH = -2,           /* declared digest does not match the bytes */
  OVL_E_SHAPE = -3,          /* dims, offsets, alignment or sizes inconsistent */
  OVL_E_QUANT = -4,          /* unknown or mismatched quantization profile */
  OVL_E_OOM = -5,            /* arena budget exceeded (all-or-nothing) */
  OVL_E_NONFINITE = -6,      /* NaN/Inf in an adapter payload */
  OVL_E_DUPLICATE = -7,      /* duplicate handle / duplicate target */
  OVL_E_NOTARGET = -8,       /* adapter targets a tensor the base does not have */
  OVL_E_BUSY = -9,           /* switch requested while forward work is in flight */
  OVL_E_NO_PREVIOUS = -10,   /* rollback with no previous composition */
  OVL_E_STATE = -11,         /* operation not valid in the current state */
  OVL_E_CUDA = -12,          /* a CUDA runtime call failed */
  OVL_E_DEVICE_TIMEOUT = -13 /* a bounded device-side wait ran out */
};

enum { OVL_Q8_0 = 1, OVL_Q4_0 = 2, OVL_Q4_K = 3 };   /* quantization profile */
enum { OVL_F32 = 1, OVL_BF16 = 2 };                  /* activation dtype */
enum { OVL_MODE_STACK = 1, OVL_MODE_TABLE = 2 };     /* composition mode */
enum { OVL_PATH_DUAL = 1, OVL_PATH_JIT = 2 };        /* evaluation path */
enum { OVL_SWITCH_REJECT = 1, OVL_SWITCH_DRAIN = 2 };/* switch vs in-flight forward */
enum {                                                /* activation phases ([DTD] §6) */
  OVL_PHASE_VALIDATION = 1, OVL_PHASE_ALLOCATION = 2, OVL_PHASE_STAGING = 3,
  OVL_PHASE_CHECKSUM = 4, OVL_PHASE_SWAP = 5,
  OVL_PHASE_DEVICE_WAIT = 6   /* a bounded device-side wait of the next decode launch (tests) */
};

enum { OVL_ADAPTER_LORA = 1, OVL_ADAPTER_SPARSE = 2 };/* adapter type in a manifest */
enum {
  OVL_MAX_STACK = 8,          /* adapters in one STACK composition */
  OVL_MAX_TABLE = 32,         /* slots in one TABLE composition */
  OVL_MAX_RANK = 128,         /* rank of one adapter target */
  OVL_MAX_TOTAL_RANK = 256,   /* sum of ranks on one tensor in a STACK */
  OVL_MAX_T = 512,            /* tokens per forward call */
  OVL_MAX_SEGMENTS = 64       /* segments per segmented call */
};

typedef struct {
  uint32_t layer, proj;       /* informational; part of the identity */
  uint32_t d_out, d_in;       /* rows (outputs) and columns (inputs) */
  uint64_t qs_off, d_off;     /* byte offsets of the two planes in the base buffer */
} ovl_tensor_desc;

typedef struct {
  uint32_t quant;             /* OVL_Q8_0, OVL_Q4_0 or OVL_Q4_K */
  uint32_t n_tensors;
  const ovl_tensor_desc* tensors;   /* host array of n_tensors, copied */
} ovl_base_desc;

typedef struct {
  uint32_t n_targets;
  const uint32_t* target_tensor;    /* host arrays of n_targets, copied */
  const uint32_t* rank;
  const uint64_t* a_off;
  const uint64_t* b_off;
  uint8_t required_base_digest[32]; /* all-zero = no requirement, else must equal the
                                       base's content digest ([DTD] §11 AdapterManifestV0) */
} ovl_adapter_desc;

typedef struct {
  uint8_t composition_id[32];
  uint8_t base_digest[32];
  uint32_t quant, mode, n_entries, has_previous;
  uint64_t epoch;             /* number of successful swaps since ovl_load_base */
  uint64_t arena_used, arena_bytes;
  uint32_t n_staged, base_loaded;
} ovl_state;

typedef struct {
  ovl_adapter_h handle;
  uint8_t adapter_key[32];
  float scale;
  uint32_t total_rank;        /* sum of ranks over the adapter's targets */
} ovl_entry;

typedef struct {
  char name[64];                    /* NUL-terminated */
  uint8_t file_digest[32];          /* content digest of the adapter's payload */
  uint8_t required_base_digest[32]; /* valid when has_required_base */
  uint32_t type;                    /* OVL_ADAPTER_LORA or OVL_ADAPTER_SPARSE */
  uint32_t load_order;
  uint32_t rank;                    /* 0 = not given */
  uint32_t n_targets;               /* 0 = not given */
  uint32_t has_required_base;
  float merge_weight;               /* binary32, the entry's scale */
} ovl_manifest_entry;

typedef struct {
  uint8_t base_digest[32];
  uint32_t quant, mode, n_adapters;
  ovl_manifest_entry adapters[OVL_MAX_TABLE];   /* in increasing load_order */
} ovl_manifest;

/* Create a context on CUDA device `device` over a caller-owned device arena of
 * arena_bytes bytes (>= 16 MiB, 256-byte aligned).  The arena holds the device
 * status word, the forward workspace, staged adapters and digest scratch; it must
 * outlive the context.  switch_policy: OVL_SWITCH_REJECT (a switch while forward
 * work is in flight fails with OVL_E_BUSY) or OVL_SWITCH_DRAIN (waits for it)
 * ([OVR] §"Explicit Correctness and Atomicity Invariants", Concurrent Safety).
 * *out receives the context; on error *out is NULL. */
ovl_status ovl_create(ovl_ctx** out, int device, void* arena_dev, size_t arena_bytes,
                      uint32_t switch_policy);

/* Destroy the context after synchronizing its internal stream.  Frees host
 * state only; the arena and the base remain the caller's.  NULL is a no-op.
 * (Housekeeping of this library; the pages define no counterpart.) */
ovl_status ovl_destroy(ovl_ctx* ctx);

/* Register the immutable base ([OVR] §"Immutable base"; [DTD] §2 Oracle
 * Invariant).  base_dev: device pointer to nbytes bytes laid out as described
 * above, read-only to the library, valid until ovl_destroy.  digest: the declared
 * content digest; the library computes the digest of the device bytes (device
 * leaf hashing on `stream`, then synchronizes) and fails with OVL_E_HASH on
 * mismatch.  Descriptor errors: OVL_E_QUANT, OVL_E_SHAPE.  Once per context
 * (OVL_E_STATE otherwise).  The base-only composition becomes active. */
ovl_status ovl_load_base(ovl_ctx* ctx, const ovl_base_desc* desc, const void* base_dev,
                         size_t nbytes, const uint8_t digest[32], void* stream);

/* Stage an adapter ([OVR] §"Proposed Activation/Deactivation State Machine";
 * [DTD] §6 VALIDATION -> ALLOCATION -> STAGING -> CHECKSUM).  payload_host: host
 * pointer to nbytes bytes (A/B factors at the descriptor's offsets), read during
 * the call only.  Validation: targets exist (OVL_E_NOTARGET), no duplicate target
 * (OVL_E_DUPLICATE), 1 <= rank <= OVL_MAX_RANK, offsets aligned and in range
 * (OVL_E_SHAPE), required base digest (OVL_E_HASH), digest of the host bytes
 * equals `digest` (OVL_E_HASH).  Allocation from the arena, all-or-nothing
 * (OVL_E_OOM).  Staging: host->device copy on the library's internal stream.
 * Checksum: the digest of the device copy must equal the host digest
 * (OVL_E_HASH) and every factor value must be finite (OVL_E_NONFINITE).  Any
 * failure frees the allocation and changes nothing.  *out receives the handle. */
ovl_status ovl_stage_adapter(ovl_ctx* ctx, const ovl_adapter_desc* desc, const void* payload_host,
                             size_t nbytes, const uint8_t digest[32], ovl_adapter_h* out);

/* Descriptor of a sparse overlay (see ovl_stage_sparse). */
typedef struct {
  uint32_t n_targets;
  const uint32_t* target_tensor;    /* host arrays of n_targets, copied */
  const uint32_t* nnz;              /* index-value pairs per target (0 allowed) */
  const uint64_t* idx_off;
  const uint64_t* val_off;
  uint8_t required_base_digest[32]; /* all-zero = no requirement */
} ovl_sparse_desc;

/* Stage a sparse overlay: only the non-zero elements of each target's weight
 * update, as index-value pairs added at their positions at use time, the base
 * unchanged ([OVR] §"Runtime Strategy Comparison Matrix", Sparse Overlay;
 * [OVR] §"Memory, Byte, and Latency Formulas", Sparse Adapter: 32-bit indices
 * and 16-bit values, k*(4+2) bytes; [DTD] §7 Sparse Overlay Bytes; [DTD] §11
 * AdapterManifestV0 adapter type Sparse (DARE)).
 * Payload (host, nbytes bytes, read during the call only): per target a uint32
 * index plane [nnz] at idx_off and an IEEE binary16 value plane [nnz] at
 * val_off (offsets multiples of 16).  Pair k adds scale * val[k] to the weight at
 * row idx[k] / d_in, column idx[k] % d_in of the target tensor.
 * Phases and errors as ovl_stage_adapter.  Validation: targets exist
 * (OVL_E_NOTARGET), no duplicate target (OVL_E_DUPLICATE), d_out * d_in < 2^32,
 * nnz <= d_out * d_in, planes aligned and inside the payload, indices strictly
 * increasing and below d_out * d_in ([DTD] §11 Deep Compatibility Checks)
 * (OVL_E_SHAPE), required base digest and payload digest (OVL_E_HASH).
 * Allocation: the payload plus the row offsets [d_out + 1] per target that the
 * library builds (OVL_E_OOM).  Checksum: device-copy digest (OVL_E_HASH), then
 * every value finite (OVL_E_NONFINITE, [DTD] §11).  Any failure frees the
 * allocation and changes nothing.  The handle is activated with ovl_activate
 * like a low-rank adapter, in STACK compositions only; ovl_get_entry reports
 * total_rank 0 for it.  adapter_key = SHA256("OVLS" | payload_digest |
 * u32 n_targets | per target u32 tensor, nnz | u64 idx_off, val_off). */
ovl_status ovl_stage_sparse(ovl_ctx* ctx, const ovl_sparse_desc* desc, const void* payload_host, size_t nbytes,
                            const uint8_t digest[32], ovl_adapter_h* out);

/* Release a staged adapter's arena block, marking it free in the arena
 * allocator (as [DTD] §6 ROLLBACK frees a staging block; [OVR] §"Proposed
 * Activation/Deactivation State Machine", Final State: staging memory that is no
 * longer needed is freed).  OVL_E_STATE if it is part of the
 * active or the rollback composition; OVL_E_BUSY (REJECT policy) if forward work
 * that read it is still in flight; OVL_E_ARG for an unknown handle. */
ovl_status ovl_unstage_adapter(ovl_ctx* ctx, ovl_adapter_h h);

/* Atomically make (h[0], scale[0]) ... (h[n-1], scale[n-1]) the active
 * composition ([OVR] §"Proposed Activation/Deactivation State Machine",
 * Activation Point; [DTD] §6 COMMIT/SWAP).  mode OVL_MODE_STACK: every entry is
 * applied to every token, in order.  mode OVL_MODE_TABLE: entries are slots that
 * ovl_segmented_forward selects per segment.  n = 0 activates the base-only
 * composition (deactivation, [OVR] same section, Deactivation).  Re-activating
 * the active composition is a no-op that returns its id ([OVR] Idempotency).
 * The replaced composition becomes the rollback target.  Errors: OVL_E_ARG
 * (unknown handle, non-finite scale, bad mode, n over the limit, a sparse
 * overlay in a TABLE composition), OVL_E_DUPLICATE,
 * OVL_E_SHAPE (total rank on a tensor over OVL_MAX_TOTAL_RANK), OVL_E_BUSY.
 * composition_id_out (host, 32 bytes, may be NULL) receives the active id. */
ovl_status ovl_activate(ovl_ctx* ctx, const ovl_adapter_h* h, const float* scale, uint32_t n,
                        uint32_t mode, uint8_t composition_id_out[32]);

/* Restore the composition that was active before the last successful swap and
 * clear the rollback slot (one level deep; [OVR] §"Proposed Activation/
 * Deactivation State Machine", Commit or Rollback).  OVL_E_NO_PREVIOUS if there
 * is none; OVL_E_BUSY as for ovl_activate. */
ovl_status ovl_rollback(ovl_ctx* ctx, uint8_t composition_id_out[32]);

/* y = layer `tensor` of the active composition applied to x.
 * x: device pointer [T][d_in] (x_dtype OVL_F32 or OVL_BF16); y: device pointer
 * float32 [T][d_out]; both valid until the work on `stream` completes.
 * path OVL_PATH_DUAL: fused dequant + low-rank kernel, y = deq(W) x + sum s B (A x)
 *   with fp32 accumulation ([OVR] §"Native/WASM Kernel Implications", Direct
 *   Low-Rank Addition; [DTD] §8 Prefill vs Decode).  scratch unused (may be NULL).
 * path OVL_PATH_JIT: materializes S = deq(W) + sum s B A into `scratch` (device,
 *   float32, >= d_out*d_in*4 bytes), then y = x S^T on the tensor cores (TF32
 *   operands, fp32 accumulation); the scratch may be reused by the next layer
 *   ([DTD] §1 Per-Layer JIT CoW Materialization; §5 Fresh-Base Oracle Definition).
 * STACK compositions only (OVL_E_STATE for TABLE).  T = 0 is a no-op.  Errors:
 * OVL_E_ARG (tensor index, dtype, path, T > OVL_MAX_T, null pointers, scratch too
 * small), OVL_E_STATE (no base), OVL_E_CUDA (launch failure).
 * Co-residency: below 4 tokens the dual path is one launch of at most one CTA
 * per SM, and every CTA waits for the low-rank partial sums of all the others
 * (single tokens with long factor rows per CTA -- stacked or high-rank terms --
 * instead run the low-rank shrink as a separate launch first, and then no CTA
 * waits for another).  It therefore assumes that all CTAs of the launch are
 * resident at the same time, which holds unless other work keeps SMs (or their shared memory) for
 * the launch's duration: a kernel on another stream that occupies SMs for
 * longer than ~2 s, or an execution context limited to fewer SMs than the
 * device has.  The wait is bounded: when it runs out, that launch's outputs
 * are NaN and ovl_check_device returns OVL_E_DEVICE_TIMEOUT; this call has
 * already returned OVL_OK, since the failure exists only on the device. */
ovl_status ovl_linear_forward(ovl_ctx* ctx, uint32_t tensor, const void* x, uint32_t x_dtype,
                              uint32_t T, float* y, uint32_t path, float* scratch,
                              size_t scratch_bytes, void* stream);

/* Dual path for up to 4 tensors that read the same activations -- the q, k and
 * v projections of a block, or gate and up -- in one launch ([DTD] §8: decode is
 * memory-bandwidth bound, so one pass streams every weight once and the fixed
 * per-launch latency is paid once).  tensors: host array of n tensor indices,
 * all with the same d_in; ys: host array of n device pointers, ys[i] float32
 * [T][d_out of tensors[i]].  Each output equals ovl_linear_forward(tensors[i],
 * path OVL_PATH_DUAL).  STACK compositions only.  Errors as ovl_linear_forward,
 * plus OVL_E_SHAPE when the d_in differ and OVL_E_ARG for n = 0 or n > 4. */
ovl_status ovl_linear_forward_multi(ovl_ctx* ctx, uint32_t n, const uint32_t* tensors, const void* x,
                                    uint32_t x_dtype, uint32_t T, float* const* ys, void* stream);

/* Materialize S = deq(W) + sum_k s_k B_k A_k (STACK composition, float32
 * [d_out][d_in] row-major) into the caller's device scratch without requantizing
 * ([DTD] §5 Fresh-Base Oracle Definition; §7 Scratch Overhead).  With an empty
 * stack S is the exact dequantized tensor. */
ovl_status ovl_materialize_layer(ovl_ctx* ctx, uint32_t tensor, float* scratch,
                                 size_t scratch_bytes, void* stream);

/* Multi-adapter batch over one base tensor (TABLE composition; [DTD] §1 SGMV).
 * x: device [T][d_in]; y: device float32 [T][d_out], rows in request order.
 * perm, seg_offsets, seg_slot: HOST arrays, copied into the launch:
 *   perm[j] (j < T) = request row of the j-th grouped row (a permutation of 0..T-1);
 *   segment s (s < n_seg) covers grouped rows seg_offsets[s] .. seg_offsets[s+1]-1
 *   (seg_offsets has n_seg+1 nondecreasing entries, first 0, last T) and uses
 *   table slot seg_slot[s] (-1 = base only).
 * y[perm[j]] = deq(W) x[perm[j]] + s_slot B_slot (A_slot x[perm[j]]).
 * Errors: OVL_E_STATE (not TABLE), OVL_E_ARG (bad segments or slots). */
ovl_status ovl_segmented_forward(ovl_ctx* ctx, uint32_t tensor, const void* x, uint32_t x_dtype,
                                 uint32_t T, const int32_t* seg_offsets, const int32_t* seg_slot,
                                 uint32_t n_seg, const int32_t* perm, float* y, void* stream);

/* Allocation-free dual-path forward.  No counterpart in the source pages: it
 * serves callers that can neither lend an arena (ovl_create) nor allocate
 * device memory when they call -- an embedder whose device memory belongs
 * entirely to its own pooled allocator (a cudaMalloc behind its back would
 * escape its budget and can stall every stream of the device while the
 * driver maps the new memory), or a caller on a latency-critical path that
 * must not take that stall at all.
 *   y = deq(W) x + sum_k scale[k] B[k] (A[k] x), exactly the computation of
 *   ovl_linear_forward on the dual path for the STACK composition (B[0..n), ...).
 * qs, d: device pointers to one tensor's planes in the layout above (16-byte
 * aligned; the d plane readable up to the next multiple of 16 bytes).  A, B,
 * rank, scale: HOST arrays of n_terms entries; A[k] float32 [rank][d_in] and
 * B[k] float32 [d_out][rank] are device pointers.  x, y as in
 * ovl_linear_forward.  Runs on the current device, on `stream`.
 * Scratch: a file-scope device array of 2 MiB per device (held by every GPU
 * that loads the library until the process exits) instead of cudaMalloc; the
 * call allocates nothing and calls no allocating routine.  The first call on a
 * device looks up the array's device address and clears it (synchronizing the
 * device), so make that first call before any stream capture.  Every call
 * then clears, on `stream`, the status word and the part of the array its
 * launches use, and numbers those launches' partial sums afresh: nothing of
 * an earlier call is read.  Calls that overlap on the GPU (different streams,
 * or other threads) race on the shared array and must be serialized by the
 * caller.
 * Errors: OVL_E_QUANT (also for OVL_Q4_K, which this entry point does not
 * take), OVL_E_SHAPE (d_in, alignment, rank, total rank), OVL_E_ARG
 * (null pointers, dtype, T > OVL_MAX_T, n_terms > OVL_MAX_STACK, non-finite
 * scale), OVL_E_OOM (the low-rank partial sums would need more than the 2 MiB
 * array), OVL_E_CUDA.  T = 0 is a no-op.  If a bounded device-side wait runs
 * out (other work holding the SMs the launch needs), the outputs it covers
 * are written as NaN. */
ovl_status ovl_dualpath_forward_noalloc(const void* qs, const void* d, uint32_t quant, uint32_t d_out,
                                        uint32_t d_in, const float* const* A, const float* const* B,
                                        const uint32_t* rank, const float* scale, uint32_t n_terms,
                                        const void* x, uint32_t x_dtype, uint32_t T, float* y, void* stream);

/* Copy one decode step's activations from page-locked host memory into device
 * memory inside the stream's programmatic launch chain.  No counterpart in the
 * source pages: a runtime helper for decode loops around the dual-path calls.
 * A plain host-to-device copy between two forwards makes the next launch wait
 * for the copy engine and start cold; this call's kernel reads `src_host`
 * before its grid dependency resolves, lets the next launch's CTAs start
 * streaming weights at once, and writes `dst` only after the preceding kernel
 * on `stream` has completed (so it never overwrites activations that earlier
 * kernels still read).  src_host: page-locked (registered) host memory, or
 * device or managed memory; dst: device (or managed or page-locked) memory;
 * nbytes: any size, with dst and src_host equally aligned modulo 16.  The call
 * allocates nothing; the caller keeps both buffers unchanged until the copy
 * has run.  Errors: OVL_E_ARG (null pointer, pageable host memory, different
 * alignment modulo 16), OVL_E_CUDA.  nbytes = 0 is a no-op.  The forward calls
 * also accept page-locked host memory for y: the kernels then write each
 * output straight to the host. */
ovl_status ovl_stage_activations(void* dst, const void* src_host, size_t nbytes, void* stream);

/* Composition manifest ([OVR] §"Composition Identity and Manifest Schema":
 * base model hash, quantization profile, runtime tag and the ordered adapter
 * list with name, file hash, load order and merge weight; [DTD] §11
 * AdapterManifestV0: adapter type, rank, required base checksum).  The
 * document is one strict JSON object (UTF-8, at most 1 MiB, no comments, no
 * duplicate keys; any key not listed is an error):
 *   "base_model_hash": "sha256:<64 lowercase hex>"          required
 *   "quantization":    "q8_0" | "q4_0" | "q4_K"             required
 *   "runtime":         {"name": "ovl-gb300", "version": "v1"} optional; another value is version skew
 *   "mode":            "stack" | "table"                     optional, default "stack"
 *   "tokenizer_id", "timestamp_utc": strings                 optional, informational
 *   "adapters": [ { "name": 1..63 bytes, unique;  "file_hash": "sha256:<hex>", unique;
 *                   "load_order": integer 1..2^31-1, unique;  "merge_weight": number;
 *                   "type": "lora" (default) | "sparse";  "rank": integer;
 *                   "required_base_hash": "sha256:<hex>";  "targets": [tensor index, ...] } ]
 * The adapters apply in increasing load_order with scale = merge_weight
 * rounded to binary32.  Parsing needs no device.
 * Errors: OVL_E_ARG (not JSON, missing or malformed field, unknown field,
 * ambiguous load_order, non-finite weight, runtime skew, more than
 * OVL_MAX_TABLE adapters), OVL_E_QUANT (unknown quantization profile),
 * OVL_E_DUPLICATE (a name or file_hash listed twice).  The message is read
 * with ovl_last_error(NULL). */
ovl_status ovl_manifest_parse(const char* text, size_t len, ovl_manifest* out);

/* Activate the composition a manifest describes: each adapter is found among
 * the context's staged adapters by its payload content digest (the content
 * address), then activated in load order with its merge weight, exactly as
 * ovl_activate would (same composition id, idempotency, rollback slot, busy
 * policy).  Checked against the context before anything changes:
 * base_model_hash against the loaded base (OVL_E_HASH), quantization against
 * its profile (OVL_E_QUANT), a file_hash with no staged adapter (OVL_E_HASH),
 * the staged adapter's type (OVL_E_ARG), rank (every target, OVL_E_SHAPE),
 * targets (same tensors in the same order, OVL_E_SHAPE) and
 * required_base_hash (OVL_E_HASH).  Any failure, at parsing or later, leaves
 * the active composition and the rollback slot unchanged ([OVR] §"TDD and
 * Fault-Injection Matrix": malformed manifests and wrong hashes are rejected
 * deterministically with no state change). */
ovl_status ovl_activate_manifest(ovl_ctx* ctx, const char* text, size_t len, uint8_t composition_id_out[32]);

/* Recompute the content digest of the base's device bytes now (device leaf
 * hashing on `stream`, synchronizes).  Used to check that the base stays
 * bit-identical across switches ([DTD] §2 Oracle Invariant). */
ovl_status ovl_base_digest(ovl_ctx* ctx, uint8_t digest_out[32], void* stream);

/* Snapshot of the observable state: composition id, base digest, quant
 * profile, mode, entry count, rollback availability, epoch, arena use ([MODELD]
 * §"Observability": which base is active, which adapters are attached). */
ovl_status ovl_get_state(ovl_ctx* ctx, ovl_state* out);

/* Entry i (< n_entries) of the active composition, in order: handle, adapter
 * key, scale, total rank (0 for a sparse overlay) ([MODELD] §"Observability":
 * adapter digests and scales). */
ovl_status ovl_get_entry(ovl_ctx* ctx, uint32_t i, ovl_entry* out);

/* Synchronize `stream`, read and clear the device status word.  Returns OVL_OK,
 * OVL_E_DEVICE_TIMEOUT (a bounded device wait ran out; outputs of that launch are
 * invalid) or OVL_E_CUDA.  (The pages define no counterpart: it reports the
 * library's own bounded device-side waits.) */
ovl_status ovl_check_device(ovl_ctx* ctx, void* stream);

/* Fault injection for tests ([OVR] §"TDD and Fault-Injection Matrix"): the next
 * stage/activate/rollback that reaches `phase` fails there with `code` (< 0),
 * with the same cleanup as a real failure.  code 0 clears a pending injection.
 * OVL_PHASE_DEVICE_WAIT (code must be OVL_E_DEVICE_TIMEOUT): the next
 * ovl_linear_forward / ovl_linear_forward_multi that runs the decode kernel
 * with a low-rank term withholds the partial sums of its first CTA and limits
 * the gather's poll to about a millisecond, so that bounded wait runs out: the
 * call returns OVL_OK, the launch's outputs are NaN, and the following
 * ovl_check_device returns OVL_E_DEVICE_TIMEOUT.  No state changes; nothing
 * faults or hangs; the next forward is normal. */
ovl_status ovl_debug_inject(ovl_ctx* ctx, uint32_t phase, ovl_status code);

/* Message of the last failed call on ctx (static storage owned by ctx; "" after
 * success).  ctx NULL returns the message of the last failed call that has no
 * context on this thread (ovl_create, ovl_manifest_parse).
 * ([MODELD] §"Observability": why an adapter failed to load.) */
const char* ovl_last_error(ovl_ctx* ctx);

/* Host utility (no device needed): FIPS 180-4 SHA-256 of n bytes, computed by
 * the library's own code. */
ovl_status ovl_sha256(const void* data, size_t n, uint8_t out[32]);

/* Host utility (no device needed): the content digest defined above (64 KiB
 * leaves), the value a caller declares for a base or a payload ([OVR]
 * §"Checksum Verification"; [DTD] §6 CHECKSUM VERIFICATION). */
ovl_status ovl_content_digest(const void* data, size_t n, uint8_t out[32]);

/* Library version string (static); the same runtime version enters every
 * composition id ([OVR] §"Composition Identity and Manifest Schema": the
 * identity includes the runtime version). */
const char* ovl_version(void);

#ifdef __cplusplus
}
#endif
#endif /* OVL_H */
