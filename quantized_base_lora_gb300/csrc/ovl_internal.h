// Internal declarations of libovl: launch arguments of the kernels and the
// launcher functions the host state machine calls.  Not part of the C ABI.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/ovl.h"

namespace ovl {

constexpr int kQK = 32;                 // weights per quantization block
constexpr int kQKK = 256;               // weights per q4_K super-block (16-byte header each)
constexpr size_t kLeaf = 65536;         // content-digest leaf size

// Device status word codes (latched by kernels, read by ovl_check_device).
enum : uint32_t {
  kDevOk = 0,
  kDevTimeoutFull = 1,      // consumer gave up waiting for a staged tile
  kDevTimeoutEmpty = 2,     // producer gave up waiting for a free stage
  kDevTimeoutShrink = 3,    // gave up waiting for the low-rank partial sums
};

// One low-rank term as the kernels see it: A [r][d_in], B [d_out][r] (fp32,
// device), applied with scale s.
struct LoraRef {
  const float* A;
  const float* B;
  uint32_t r;
  float s;
};

// Device workspace carved from the arena at context creation.  The low-rank
// partial sums are 64-bit slots {launch epoch (high word), f32 value (low
// word)}: a reader accepts a slot once it carries its own launch's epoch, so no
// slot ever needs clearing between launches.  The epoch counter is host memory
// (launcher only); epochs start at 1 and the slots are cleared when it wraps.
// An epoch is below 2^31: bit 31 of DualArgs::epoch carries a test request.
struct Workspace {
  uint32_t* status;               // one status word (device)
  float* partial;                 // partial-sum slots (device), 8 bytes each
  size_t partial_floats;          // size of that region in floats
  uint32_t* epoch_counter;        // host: last epoch handed out (wraps below 2^31)
  float* tc_scratch;              // tensor-core path scratch (device, 256-byte aligned)
  size_t tc_scratch_bytes;        // 0: the tensor-core path is not available
};

// One tensor of a (multi-tensor) dual-path launch.  All tensors of a launch
// share d_in and the activations; CTAs [g0, g0 + gn) of the grid serve this
// tensor, and its low-rank terms are lora[k0, k1) (rank offset rb0 in the
// flattened shrink space).  Filled by the launcher.
struct DualSeg {
  const uint8_t* qs;
  const uint8_t* dpl;
  float* y;
  uint32_t m;
  uint32_t g0, gn;
  uint32_t k0, k1, rb0;
};

constexpr int kMaxMulti = 4;
constexpr uint32_t kEpochWithhold = 0x80000000u;
constexpr uint32_t kTokTile = 64;       // tokens per tensor-core launch

// Fused dual-path forward over a token chunk (T <= 8).  Single-tensor callers
// fill qs/dpl/m/y; multi-tensor callers fill nseg and seg[] (qs, dpl, y, m,
// k0, k1, rb0) and leave m = total rows.
// Field order: the kernel reads its parameters through the constant cache, and
// a line first touched late in the kernel costs a memory round trip there.
// Everything the kernel reads late (epoch, workspace, token selection) shares
// the first cache lines with fields every warp reads at the start.
struct DualArgs {
  const uint8_t* qs;      // qs plane
  const uint8_t* dpl;     // d plane (binary16)
  const void* x;          // [T][n], fp32 or bf16
  float* y;               // [T][m]
  uint32_t m, n, quant;
  uint32_t xdt, T;
  uint32_t nl;            // number of low-rank terms
  uint32_t rtot;          // sum of ranks
  uint32_t epoch;         // this launch's partial-slot epoch (filled by the launcher, < 2^31);
                          // bit 31 (kEpochWithhold) is a test-only request: CTA 0 tags its partial
                          // sums with an epoch no reader accepts and the gather polls about a
                          // millisecond, so that bounded wait runs out
  uint32_t nseg;          // 0: single tensor (qs/dpl/m/y); else seg[0..nseg)
  // Per-token term selection (segmented batches): when tok_sel is set, token t
  // of the launch receives only term tok_term[t] (-1: base only).
  uint32_t tok_sel;
  int8_t tok_term[8];     // this launch's slice (filled by the launcher)
  uint32_t b_pad;         // 1: each B may be read in 16-byte granules around its rows
                          //    (arena-resident factors), so B rows can be bulk-copied
  uint32_t a16;           // 1: every A is 16-byte aligned (16-byte copies of its rows)
  Workspace ws;
  DualSeg seg[kMaxMulti];
  LoraRef lora[OVL_MAX_TABLE];
  const int8_t* tok_host;  // host array of T entries (launcher only)
};

// Dual path on the tensor cores (K4) for multi-token launches of one to four
// tensors that share x (same d_in): token chunks of kTokTile, each one widen +
// shrink launch and one fused dequantizing GEMM launch over all the tensors.
struct FusedTensor {
  const uint8_t* qs;
  const uint8_t* dpl;
  uint32_t m;
  float* y;                 // [T][m]
  uint32_t nl, rtot;
  LoraRef lora[OVL_MAX_TABLE];
};
struct FusedLaunch {
  uint32_t nt;              // tensors, 1..4; their terms together at most OVL_MAX_TABLE
  FusedTensor t[4];
  uint32_t quant, n;
  const void* x;            // [T][n], fp32 or bf16, 16-byte aligned
  uint32_t xdt, T;
  uint32_t tok_sel;         // segmented (one tensor): token t adds only term tok_host[t] (-1: none)
  const int8_t* tok_host;   // host, T entries
  float* scratch;           // widened activations + low-rank vectors
  size_t scratch_bytes;
  uint32_t* status;
};
// d_in a multiple of 256 (the f16 scale rows feed 16-byte tensor-map boxes).
bool fused_gemm_supported(uint32_t m, uint32_t n);
// vcols: the tensors' total ranks, each rounded up to a multiple of 32.
size_t fused_gemm_scratch_bytes(uint32_t T, uint32_t n, uint32_t vcols);
inline uint32_t fused_vcols(uint32_t rtot) { return (rtot + 31) / 32 * 32; }
cudaError_t launch_fused_gemm(const FusedLaunch& L, cudaStream_t st);

// Materialize S = deq(W) + sum_k s_k B_k A_k into fp32 scratch [m][n].
struct MatArgs {
  const uint8_t* qs;
  const uint8_t* dpl;
  uint32_t m, n, quant;
  uint32_t nl;
  LoraRef lora[OVL_MAX_STACK];
  float* S;
};

// One sparse overlay term on one tensor: nnz index-value pairs (flat index
// row * n + col, strictly increasing; binary16 values) and the row offsets the
// library builds at staging (rp[row] .. rp[row + 1] are the row's pairs).
struct SparseRef {
  const uint32_t* idx;
  const uint16_t* val;
  const uint32_t* rp;     // [m + 1]
  uint32_t nnz;
  float s;
};

// One tensor of a sparse launch: rows [row0, row0 + m) of the launch, output
// y [T][m], terms t[k0, k1).
struct SparseSeg {
  float* y;
  uint32_t m, row0;
  uint32_t k0, k1;
};

// y[t][row] += sum_k s_k * sum_{pairs of row in term k} val * x[t][col], terms in
// order, after the dense dual path has written y.  Up to kMaxMulti tensors that
// share x (and d_in) in one launch.
struct SparseApply {
  const void* x;          // [T][n], fp32 or bf16
  uint32_t n, T, xdt;
  uint32_t nseg, mtot;
  SparseSeg seg[kMaxMulti];
  uint32_t nt;
  SparseRef t[kMaxMulti * OVL_MAX_STACK];
};

cudaError_t launch_dualpath(const DualArgs& a, cudaStream_t st);
cudaError_t launch_sparse_apply(const SparseApply& a, cudaStream_t st);
// S[idx[k]] += s * val[k] for every pair of one term (fp32 scratch [m][n]).
cudaError_t launch_sparse_scatter(float* S, const SparseRef& t, cudaStream_t st);
cudaError_t launch_materialize(const MatArgs& a, cudaStream_t st);
// Y[T][m] = X[T][n] * S[m][n]^T with TF32 tensor-core operands, fp32 accumulate.
cudaError_t launch_jit_gemm(const float* S, const void* x, uint32_t xdt, uint32_t T, uint32_t m,
                            uint32_t n, float* y, float* xf32_scratch, const Workspace& ws,
                            cudaStream_t st);
size_t jit_gemm_x_scratch_bytes(uint32_t T, uint32_t n);

// Content digest helpers: SHA-256 of each 64 KiB leaf of a device buffer into
// `leaf_digests` (device, 32 bytes per leaf).
cudaError_t launch_leaf_digests(const uint8_t* data, size_t n, uint8_t* leaf_digests,
                                cudaStream_t st);
// Scan `n` fp32 values at `p`; increments *flag (device) if any is NaN/Inf.
cudaError_t launch_finite_scan(const float* p, size_t n, uint32_t* flag, cudaStream_t st);

// A parsed composition manifest (ovl_manifest.cu): adapters in increasing
// load_order.
struct ManifestAdapter {
  std::string name;
  uint8_t file_hash[32] = {};
  uint32_t type = OVL_ADAPTER_LORA;
  uint32_t load_order = 0;
  float merge_weight = 0.f;
  uint32_t rank = 0;                 // 0: not given
  bool has_required_base = false;
  uint8_t required_base[32] = {};
  bool has_targets = false;
  std::vector<uint32_t> targets;
};
struct Manifest {
  uint8_t base_hash[32] = {};
  uint32_t quant = 0, mode = OVL_MODE_STACK;
  std::vector<ManifestAdapter> adapters;
};
constexpr const char* kManifestRuntimeName = "ovl-gb300";
constexpr const char* kManifestRuntimeVersion = "v1";
ovl_status parse_manifest(const char* text, size_t len, Manifest* out, std::string* err);
// Message returned by ovl_last_error(NULL) (failures that have no context).
void set_context_free_error(const std::string& msg);

// Host-side digests (library's own SHA-256).
void host_sha256(const void* data, size_t n, uint8_t out[32]);
void host_content_digest(const void* data, size_t n, uint8_t out[32]);
void host_digest_of_leaves(const uint8_t* leaf_digests, size_t n_leaves, uint8_t out[32]);

}  // namespace ovl
