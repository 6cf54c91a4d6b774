// libovl host side: context, device arena, activation state machine and the
// extern "C" boundary declared in include/ovl.h.
//
// Sources: "We propose a content-addressed overlay system" report
// §"Proposed Activation/Deactivation State Machine" (validate, stage, atomic
// pointer swap, rollback restores the previous pointer, deactivation = activate
// the base-only manifest), §"Explicit Correctness and Atomicity Invariants"
// (atomic update, idempotency, bounded resources, checksum verification,
// concurrent safety), §"Composition Identity and Manifest Schema";
// "Deep Technical Design ..." §2 (Transactional Atomicity Invariant: isolated
// staging arena, pointer updated only after all checks), §3 (identity tuple
// incl. layout, quantization and runtime policy), §6 (VALIDATION, ALLOCATION,
// STAGING, CHECKSUM, COMMIT/SWAP, ROLLBACK), §11 (AdapterManifestV0 required
// base checksum; deep compatibility checks); contenox modeld blueprint
// "LoRA adapters" §"Runtime Identity and Cache Safety" and §"Validation and
// Compatibility" (digest match, finite scale, zero-match targets rejected).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "ovl_internal.h"
#include "sha256.cuh"

namespace ovl {
namespace {

constexpr size_t kArenaAlign = 256;
constexpr size_t kStatusOff = 0;
constexpr size_t kPartialOff = 1024;
// K1's partial-sum slots: at most 8 tokens x OVL_MAX_TOTAL_RANK x 152 shrink
// CTAs x 8 bytes = 2.4 MiB; then the tensor-core scratch, which holds a
// 128-token chunk of 14336-wide activations in fp32 (7.3 MB) and its s v.
constexpr size_t kPartialBytes = 3u << 20;
constexpr size_t kTcOff = kPartialOff + kPartialBytes;
constexpr size_t kTcBytes = 8u << 20;
constexpr size_t kReservedEnd = kTcOff + kTcBytes;
constexpr size_t kMinArena = 16u << 20;
constexpr uint32_t kMaxTableRank = 1024;   // sum of ranks of a TABLE composition on one tensor
constexpr char kRuntimeTag[16] = {'o', 'v', 'l', '-', 'g', 'b', '3', '0', '0', ' ', 'v', '1', 0, 0, 0, 0};

// First-fit sub-allocator over [kReservedEnd, arena_bytes) of the caller's arena.
class Arena {
 public:
  void reset(size_t begin, size_t end) {
    free_.clear();
    if (end > begin) free_[begin] = end - begin;
    used_ = 0;
  }
  bool alloc(size_t bytes, size_t* off) {
    bytes = (bytes + kArenaAlign - 1) / kArenaAlign * kArenaAlign;
    if (bytes == 0) bytes = kArenaAlign;
    for (auto it = free_.begin(); it != free_.end(); ++it) {
      if (it->second >= bytes) {
        *off = it->first;
        const size_t rest = it->second - bytes;
        const size_t base = it->first;
        free_.erase(it);
        if (rest) free_[base + bytes] = rest;
        used_ += bytes;
        sizes_[*off] = bytes;
        return true;
      }
    }
    return false;
  }
  void release(size_t off) {
    auto s = sizes_.find(off);
    if (s == sizes_.end()) return;
    size_t bytes = s->second;
    sizes_.erase(s);
    used_ -= bytes;
    size_t begin = off;
    auto next = free_.lower_bound(off);
    if (next != free_.end() && next->first == off + bytes) {
      bytes += next->second;
      free_.erase(next);
    }
    auto it = free_.lower_bound(off);
    if (it != free_.begin()) {
      auto prev = std::prev(it);
      if (prev->first + prev->second == begin) {
        begin = prev->first;
        bytes += prev->second;
        free_.erase(prev);
      }
    }
    free_[begin] = bytes;
  }
  size_t used() const { return used_; }

 private:
  std::map<size_t, size_t> free_;
  std::map<size_t, size_t> sizes_;
  size_t used_ = 0;
};

struct Target {
  uint32_t tensor, rank;
  uint64_t a_off, b_off;
};

// A sparse overlay target: index and value planes inside the payload, and the
// row offsets [d_out + 1] the library builds at staging (offset from the
// adapter's arena allocation).
struct SparseTarget {
  uint32_t tensor, nnz;
  uint64_t idx_off, val_off;
  uint64_t rp_off;
};

struct Adapter {
  ovl_adapter_h h = 0;
  bool sparse = false;               // index-value overlay instead of low-rank factors
  std::vector<SparseTarget> sp;      // sparse targets (sparse adapters only)
  std::vector<Target> targets;
  size_t off = 0, bytes = 0;
  uint8_t digest[32];
  uint8_t key[32];
  uint32_t total_rank = 0;
  bool used = false;        // read by at least one forward call
};

struct Entry {
  ovl_adapter_h h;
  float s;
};

struct Composition {
  uint32_t mode = OVL_MODE_STACK;
  std::vector<Entry> entries;
  uint8_t id[32];
};

}  // namespace
}  // namespace ovl

struct ovl_ctx {
  int device = 0;
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;
  uint32_t policy = OVL_SWITCH_REJECT;
  ovl::Arena alloc;
  std::mutex mu;
  cudaStream_t stream = nullptr;
  cudaEvent_t fwd_done = nullptr;
  bool fwd_recorded = false;
  ovl::Workspace ws{};
  uint32_t slot_epoch = 0;   // last partial-slot epoch handed to a launch
  // base
  bool base_loaded = false;
  uint32_t quant = 0;
  std::vector<ovl_tensor_desc> tensors;
  const uint8_t* base = nullptr;
  size_t base_bytes = 0;
  uint8_t base_digest[32];
  uint8_t base_key[32];
  // adapters and compositions
  std::map<ovl_adapter_h, ovl::Adapter> staged;
  ovl_adapter_h next_h = 1;
  std::shared_ptr<const ovl::Composition> active, prev;
  uint64_t epoch = 0;
  // fault injection
  uint32_t inject_phase = 0;
  ovl_status inject_code = 0;
  std::string err;
};

namespace ovl {
namespace {

thread_local std::string g_create_err;

}  // namespace

void set_context_free_error(const std::string& msg) { g_create_err = msg; }

ovl_status activate_locked(ovl_ctx* ctx, const ovl_adapter_h* h, const float* scale, uint32_t n, uint32_t mode,
                           uint8_t composition_id_out[32]);

namespace {

// Makes `dev` current for the scope of a call and restores the caller's device.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev == dev) {
      prev = -1;   // already current: nothing to restore
      ok = true;
    } else {
      ok = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

ovl_status fail(ovl_ctx* c, ovl_status code, const std::string& msg) {
  c->err = msg;
  return code;
}

ovl_status cuda_fail(ovl_ctx* c, cudaError_t e, const char* what) {
  cudaGetLastError();
  return fail(c, OVL_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Returns the injected code if a pending injection targets `phase`, consuming it.
ovl_status injected(ovl_ctx* c, uint32_t phase) {
  if (c->inject_phase == phase && c->inject_code < 0) {
    ovl_status code = c->inject_code;
    c->inject_phase = 0;
    c->inject_code = 0;
    c->err = "injected failure at phase " + std::to_string(phase);
    return code;
  }
  return OVL_OK;
}

void compute_base_key(ovl_ctx* c) {
  Sha256Stream h;
  h.update("OVLB", 4);
  h.update(c->base_digest, 32);
  h.u32(c->quant);
  h.u32(static_cast<uint32_t>(c->tensors.size()));
  for (const auto& t : c->tensors) {
    h.u32(t.layer); h.u32(t.proj); h.u32(t.d_out); h.u32(t.d_in);
    h.u64(t.qs_off); h.u64(t.d_off);
  }
  h.final(c->base_key);
}

void compute_adapter_key(Adapter& a) {
  Sha256Stream h;
  if (a.sparse) {
    h.update("OVLS", 4);
    h.update(a.digest, 32);
    h.u32(static_cast<uint32_t>(a.sp.size()));
    for (const auto& t : a.sp) {
      h.u32(t.tensor); h.u32(t.nnz); h.u64(t.idx_off); h.u64(t.val_off);
    }
    h.final(a.key);
    return;
  }
  h.update("OVLA", 4);
  h.update(a.digest, 32);
  h.u32(static_cast<uint32_t>(a.targets.size()));
  for (const auto& t : a.targets) {
    h.u32(t.tensor); h.u32(t.rank); h.u64(t.a_off); h.u64(t.b_off);
  }
  h.final(a.key);
}

void compute_composition_id(ovl_ctx* c, Composition& comp) {
  Sha256Stream h;
  h.update("OVLC", 4);
  h.update(kRuntimeTag, 16);
  h.update(c->base_key, 32);
  h.u32(comp.entries.empty() ? static_cast<uint32_t>(OVL_MODE_STACK) : comp.mode);
  h.u32(static_cast<uint32_t>(comp.entries.size()));
  for (const auto& e : comp.entries) {
    h.update(c->staged.at(e.h).key, 32);
    uint32_t bits;
    std::memcpy(&bits, &e.s, 4);
    h.u32(bits);
  }
  h.final(comp.id);
}

// Device content digest of [p, p+n): leaf hashing on the GPU, root on the host.
ovl_status device_digest(ovl_ctx* c, const uint8_t* p, size_t n, cudaStream_t st, uint8_t out[32]) {
  const size_t leaves = (n + kLeaf - 1) / kLeaf;
  if (leaves == 0) {
    host_sha256(nullptr, 0, out);
    return OVL_OK;
  }
  size_t off;
  if (!c->alloc.alloc(leaves * 32, &off)) return fail(c, OVL_E_OOM, "arena too small for digest scratch");
  uint8_t* scratch = c->arena + off;
  std::vector<uint8_t> host(leaves * 32);
  cudaError_t e = launch_leaf_digests(p, n, scratch, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(host.data(), scratch, host.size(), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  c->alloc.release(off);
  if (e != cudaSuccess) return cuda_fail(c, e, "device digest");
  host_digest_of_leaves(host.data(), leaves, out);
  return OVL_OK;
}

// REJECT: fail if forward work may still run; DRAIN: wait for it.
ovl_status busy_check(ovl_ctx* c) {
  if (!c->fwd_recorded) return OVL_OK;
  if (c->policy == OVL_SWITCH_DRAIN) {
    cudaError_t e = cudaEventSynchronize(c->fwd_done);
    if (e != cudaSuccess) return cuda_fail(c, e, "drain");
    return OVL_OK;
  }
  cudaError_t q = cudaEventQuery(c->fwd_done);
  if (q == cudaErrorNotReady) return fail(c, OVL_E_BUSY, "forward work in flight");
  if (q != cudaSuccess) return cuda_fail(c, q, "event query");
  return OVL_OK;
}

const Target* target_for(const Adapter& a, uint32_t tensor) {
  for (const auto& t : a.targets)
    if (t.tensor == tensor) return &t;
  return nullptr;
}

bool finite_f32(float v) { return std::isfinite(v); }

ovl_status ok(ovl_ctx* c) {
  c->err.clear();
  return OVL_OK;
}

}  // namespace
}  // namespace ovl

using namespace ovl;

extern "C" {

const char* ovl_version(void) { return "ovl-gb300 v1 (sm_103a)"; }

ovl_status ovl_sha256(const void* data, size_t n, uint8_t out[32]) {
  if ((!data && n) || !out) return OVL_E_ARG;
  host_sha256(data, n, out);
  return OVL_OK;
}

ovl_status ovl_content_digest(const void* data, size_t n, uint8_t out[32]) {
  if ((!data && n) || !out) return OVL_E_ARG;
  host_content_digest(data, n, out);
  return OVL_OK;
}

const char* ovl_last_error(ovl_ctx* ctx) {
  if (!ctx) return g_create_err.c_str();
  return ctx->err.c_str();
}

ovl_status ovl_create(ovl_ctx** out, int device, void* arena_dev, size_t arena_bytes,
                      uint32_t switch_policy) {
  if (!out) return OVL_E_ARG;
  *out = nullptr;
  g_create_err.clear();
  if (!arena_dev || (reinterpret_cast<uintptr_t>(arena_dev) % kArenaAlign) != 0) {
    g_create_err = "arena must be a 256-byte aligned device pointer";
    return OVL_E_ARG;
  }
  if (arena_bytes < kMinArena) {
    g_create_err = "arena must be at least 16 MiB";
    return OVL_E_ARG;
  }
  if (switch_policy != OVL_SWITCH_REJECT && switch_policy != OVL_SWITCH_DRAIN) {
    g_create_err = "unknown switch policy";
    return OVL_E_ARG;
  }
  DeviceGuard g(device);
  if (!g.ok) {
    g_create_err = "cannot select device";
    return OVL_E_CUDA;
  }
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, arena_dev) != cudaSuccess || pa.type != cudaMemoryTypeDevice ||
      pa.device != device) {
    cudaGetLastError();
    g_create_err = "arena is not device memory of the given device";
    return OVL_E_ARG;
  }
  ovl_ctx* c = new (std::nothrow) ovl_ctx();
  if (!c) return OVL_E_OOM;
  c->device = device;
  c->arena = static_cast<uint8_t*>(arena_dev);
  c->arena_bytes = arena_bytes;
  c->policy = switch_policy;
  c->alloc.reset(kReservedEnd, arena_bytes);
  cudaError_t e = cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->fwd_done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->arena, 0, kReservedEnd, c->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) {
    g_create_err = std::string("cuda: ") + cudaGetErrorString(e);
    cudaGetLastError();
    if (c->fwd_done) cudaEventDestroy(c->fwd_done);
    if (c->stream) cudaStreamDestroy(c->stream);
    delete c;
    return OVL_E_CUDA;
  }
  c->ws.status = reinterpret_cast<uint32_t*>(c->arena + kStatusOff);
  // lower half: the dual path's partial-sum slots; upper half: scratch of the
  // tensor-core path (widened activations, low-rank vectors)
  c->ws.partial = reinterpret_cast<float*>(c->arena + kPartialOff);
  c->ws.partial_floats = kPartialBytes / sizeof(float);
  c->ws.tc_scratch = reinterpret_cast<float*>(c->arena + kTcOff);
  c->ws.tc_scratch_bytes = kTcBytes;
  c->ws.epoch_counter = &c->slot_epoch;
  *out = c;
  return OVL_OK;
}

ovl_status ovl_destroy(ovl_ctx* ctx) {
  if (!ctx) return OVL_OK;
  {
    DeviceGuard g(ctx->device);
    cudaStreamSynchronize(ctx->stream);
    if (ctx->fwd_recorded) cudaEventSynchronize(ctx->fwd_done);
    cudaEventDestroy(ctx->fwd_done);
    cudaStreamDestroy(ctx->stream);
  }
  delete ctx;
  return OVL_OK;
}

ovl_status ovl_load_base(ovl_ctx* ctx, const ovl_base_desc* desc, const void* base_dev, size_t nbytes,
                         const uint8_t digest[32], void* stream) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (ctx->base_loaded) return fail(ctx, OVL_E_STATE, "base already loaded");
  if (!desc || !base_dev || !digest || (desc->n_tensors && !desc->tensors))
    return fail(ctx, OVL_E_ARG, "null argument");
  if (desc->quant != OVL_Q8_0 && desc->quant != OVL_Q4_0 && desc->quant != OVL_Q4_K)
    return fail(ctx, OVL_E_QUANT, "unknown quantization profile");
  if (desc->n_tensors == 0) return fail(ctx, OVL_E_SHAPE, "base has no tensors");
  if ((reinterpret_cast<uintptr_t>(base_dev) & 15) != 0) return fail(ctx, OVL_E_SHAPE, "base must be 16-byte aligned");
  for (uint32_t i = 0; i < desc->n_tensors; ++i) {
    const ovl_tensor_desc& t = desc->tensors[i];
    const std::string who = "tensor " + std::to_string(i) + ": ";
    if (t.d_out == 0 || t.d_in == 0 || t.d_in % kQK != 0) return fail(ctx, OVL_E_SHAPE, who + "d_in must be a positive multiple of 32");
    if (desc->quant == OVL_Q4_K && t.d_in % kQKK != 0)
      return fail(ctx, OVL_E_SHAPE, who + "q4_K: d_in must be a multiple of 256");
    if (t.qs_off % 16 || t.d_off % 16) return fail(ctx, OVL_E_SHAPE, who + "plane offsets must be multiples of 16");
    const uint64_t qsb = desc->quant == OVL_Q8_0 ? uint64_t(t.d_out) * t.d_in : uint64_t(t.d_out) * t.d_in / 2;
    const uint64_t db = (uint64_t(t.d_out) * (t.d_in / kQK) * 2 + 15) / 16 * 16;
    if (t.qs_off > nbytes || qsb > nbytes - t.qs_off || t.d_off > nbytes || db > nbytes - t.d_off)
      return fail(ctx, OVL_E_SHAPE, who + "planes exceed the base buffer");
  }
  DeviceGuard g(ctx->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t got[32];
  ovl_status s = device_digest(ctx, static_cast<const uint8_t*>(base_dev), nbytes, st, got);
  if (s != OVL_OK) return s;
  if (std::memcmp(got, digest, 32) != 0) return fail(ctx, OVL_E_HASH, "base digest mismatch");
  ctx->quant = desc->quant;
  ctx->tensors.assign(desc->tensors, desc->tensors + desc->n_tensors);
  ctx->base = static_cast<const uint8_t*>(base_dev);
  ctx->base_bytes = nbytes;
  std::memcpy(ctx->base_digest, got, 32);
  compute_base_key(ctx);
  auto comp = std::make_shared<Composition>();
  compute_composition_id(ctx, *comp);
  ctx->active = comp;
  ctx->prev.reset();
  ctx->epoch = 0;
  ctx->base_loaded = true;
  return ok(ctx);
}

ovl_status ovl_stage_adapter(ovl_ctx* ctx, const ovl_adapter_desc* desc, const void* payload_host,
                             size_t nbytes, const uint8_t digest[32], ovl_adapter_h* out) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (out) *out = 0;
  // ---- VALIDATION
  if (ovl_status s = injected(ctx, OVL_PHASE_VALIDATION)) return s;
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  if (!desc || !payload_host || !digest || !out) return fail(ctx, OVL_E_ARG, "null argument");
  if (desc->n_targets == 0 || !desc->target_tensor || !desc->rank || !desc->a_off || !desc->b_off)
    return fail(ctx, OVL_E_ARG, "adapter has no targets");
  Adapter ad;
  for (uint32_t i = 0; i < desc->n_targets; ++i) {
    Target t{desc->target_tensor[i], desc->rank[i], desc->a_off[i], desc->b_off[i]};
    const std::string who = "target " + std::to_string(i) + ": ";
    if (t.tensor >= ctx->tensors.size()) return fail(ctx, OVL_E_NOTARGET, who + "no such base tensor");
    for (const auto& o : ad.targets)
      if (o.tensor == t.tensor) return fail(ctx, OVL_E_DUPLICATE, who + "tensor targeted twice");
    if (t.rank == 0 || t.rank > OVL_MAX_RANK) return fail(ctx, OVL_E_SHAPE, who + "rank out of range");
    const ovl_tensor_desc& td = ctx->tensors[t.tensor];
    const uint64_t ab = uint64_t(t.rank) * td.d_in * 4, bb = uint64_t(td.d_out) * t.rank * 4;
    if (t.a_off % 16 || t.b_off % 16) return fail(ctx, OVL_E_SHAPE, who + "factor offsets must be multiples of 16");
    if (t.a_off > nbytes || ab > nbytes - t.a_off || t.b_off > nbytes || bb > nbytes - t.b_off)
      return fail(ctx, OVL_E_SHAPE, who + "factors exceed the payload");
    ad.targets.push_back(t);
    ad.total_rank += t.rank;
  }
  static const uint8_t zero[32] = {0};
  if (std::memcmp(desc->required_base_digest, zero, 32) != 0 &&
      std::memcmp(desc->required_base_digest, ctx->base_digest, 32) != 0)
    return fail(ctx, OVL_E_HASH, "adapter requires a different base");
  host_content_digest(payload_host, nbytes, ad.digest);
  if (std::memcmp(ad.digest, digest, 32) != 0) return fail(ctx, OVL_E_HASH, "adapter digest mismatch");
  // ---- ALLOCATION
  if (ovl_status s = injected(ctx, OVL_PHASE_ALLOCATION)) return s;
  if (!ctx->alloc.alloc(nbytes, &ad.off)) return fail(ctx, OVL_E_OOM, "arena budget exceeded");
  ad.bytes = nbytes;
  auto release = [&](ovl_status code) {
    ctx->alloc.release(ad.off);
    return code;
  };
  // ---- STAGING
  DeviceGuard g(ctx->device);
  if (ovl_status s = injected(ctx, OVL_PHASE_STAGING)) return release(s);
  cudaError_t e = cudaMemcpyAsync(ctx->arena + ad.off, payload_host, nbytes, cudaMemcpyHostToDevice, ctx->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return release(cuda_fail(ctx, e, "staging copy"));
  // ---- CHECKSUM: digest of the device copy, then finiteness of every factor
  if (ovl_status s = injected(ctx, OVL_PHASE_CHECKSUM)) return release(s);
  uint8_t dev_digest[32];
  if (ovl_status s = device_digest(ctx, ctx->arena + ad.off, nbytes, ctx->stream, dev_digest)) return release(s);
  if (std::memcmp(dev_digest, ad.digest, 32) != 0) return release(fail(ctx, OVL_E_HASH, "staged copy corrupted"));
  uint32_t* flag = ctx->ws.status + 1;
  e = cudaMemsetAsync(flag, 0, 4, ctx->stream);
  for (const auto& t : ad.targets) {
    const ovl_tensor_desc& td = ctx->tensors[t.tensor];
    if (e == cudaSuccess)
      e = launch_finite_scan(reinterpret_cast<const float*>(ctx->arena + ad.off + t.a_off), size_t(t.rank) * td.d_in, flag, ctx->stream);
    if (e == cudaSuccess)
      e = launch_finite_scan(reinterpret_cast<const float*>(ctx->arena + ad.off + t.b_off), size_t(td.d_out) * t.rank, flag, ctx->stream);
  }
  uint32_t bad = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&bad, flag, 4, cudaMemcpyDeviceToHost, ctx->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return release(cuda_fail(ctx, e, "finite scan"));
  if (bad) return release(fail(ctx, OVL_E_NONFINITE, "adapter payload holds NaN or Inf"));
  compute_adapter_key(ad);
  ad.h = ctx->next_h++;
  *out = ad.h;
  ctx->staged.emplace(ad.h, ad);
  return ok(ctx);
}

ovl_status ovl_stage_sparse(ovl_ctx* ctx, const ovl_sparse_desc* desc, const void* payload_host, size_t nbytes,
                            const uint8_t digest[32], ovl_adapter_h* out) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (out) *out = 0;
  // ---- VALIDATION: shapes, strictly increasing in-range indices ([DTD] §11
  // Deep Compatibility Checks), base requirement, digest of the host bytes
  if (ovl_status s = injected(ctx, OVL_PHASE_VALIDATION)) return s;
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  if (!desc || !payload_host || !digest || !out) return fail(ctx, OVL_E_ARG, "null argument");
  if (desc->n_targets == 0 || !desc->target_tensor || !desc->nnz || !desc->idx_off || !desc->val_off)
    return fail(ctx, OVL_E_ARG, "overlay has no targets");
  const uint8_t* P = static_cast<const uint8_t*>(payload_host);
  Adapter ad;
  ad.sparse = true;
  bool nonfinite = false;
  size_t rp_total = 0;
  std::vector<std::vector<uint32_t>> rps;
  for (uint32_t i = 0; i < desc->n_targets; ++i) {
    SparseTarget t{desc->target_tensor[i], desc->nnz[i], desc->idx_off[i], desc->val_off[i], 0};
    const std::string who = "target " + std::to_string(i) + ": ";
    if (t.tensor >= ctx->tensors.size()) return fail(ctx, OVL_E_NOTARGET, who + "no such base tensor");
    for (const auto& o : ad.sp)
      if (o.tensor == t.tensor) return fail(ctx, OVL_E_DUPLICATE, who + "tensor targeted twice");
    const ovl_tensor_desc& td = ctx->tensors[t.tensor];
    const uint64_t cells = uint64_t(td.d_out) * td.d_in;
    if (cells > 0xFFFFFFFFull) return fail(ctx, OVL_E_SHAPE, who + "tensor too large for 32-bit indices");
    if (t.nnz > cells) return fail(ctx, OVL_E_SHAPE, who + "more pairs than weights");
    if (t.idx_off % 16 || t.val_off % 16) return fail(ctx, OVL_E_SHAPE, who + "plane offsets must be multiples of 16");
    const uint64_t ib = uint64_t(t.nnz) * 4, vb = uint64_t(t.nnz) * 2;
    if (t.idx_off > nbytes || ib > nbytes - t.idx_off || t.val_off > nbytes || vb > nbytes - t.val_off)
      return fail(ctx, OVL_E_SHAPE, who + "pairs exceed the payload");
    std::vector<uint32_t> rp(size_t(td.d_out) + 1, 0);
    uint32_t prev = 0;
    for (uint32_t k = 0; k < t.nnz; ++k) {
      uint32_t idx;
      uint16_t v;
      std::memcpy(&idx, P + t.idx_off + 4ull * k, 4);
      std::memcpy(&v, P + t.val_off + 2ull * k, 2);
      if (k && idx <= prev) return fail(ctx, OVL_E_SHAPE, who + "indices must be strictly increasing");
      if (idx >= cells) return fail(ctx, OVL_E_SHAPE, who + "index beyond the tensor");
      if ((v & 0x7C00u) == 0x7C00u) nonfinite = true;   // binary16 Inf or NaN
      ++rp[idx / td.d_in + 1];
      prev = idx;
    }
    for (size_t r = 1; r < rp.size(); ++r) rp[r] += rp[r - 1];
    t.rp_off = rp_total;   // relative to the row-offset area for now
    rp_total += (rp.size() * 4 + kArenaAlign - 1) / kArenaAlign * kArenaAlign;
    ad.sp.push_back(t);
    rps.push_back(std::move(rp));
  }
  static const uint8_t zero[32] = {0};
  if (std::memcmp(desc->required_base_digest, zero, 32) != 0 &&
      std::memcmp(desc->required_base_digest, ctx->base_digest, 32) != 0)
    return fail(ctx, OVL_E_HASH, "overlay requires a different base");
  host_content_digest(payload_host, nbytes, ad.digest);
  if (std::memcmp(ad.digest, digest, 32) != 0) return fail(ctx, OVL_E_HASH, "overlay digest mismatch");
  // ---- ALLOCATION: payload, then the row offsets of every target
  if (ovl_status s = injected(ctx, OVL_PHASE_ALLOCATION)) return s;
  const size_t pay = (nbytes + kArenaAlign - 1) / kArenaAlign * kArenaAlign;
  if (!ctx->alloc.alloc(pay + rp_total, &ad.off)) return fail(ctx, OVL_E_OOM, "arena budget exceeded");
  ad.bytes = nbytes;
  for (auto& t : ad.sp) t.rp_off += pay;
  auto release = [&](ovl_status code) {
    ctx->alloc.release(ad.off);
    return code;
  };
  // ---- STAGING
  DeviceGuard g(ctx->device);
  if (ovl_status s = injected(ctx, OVL_PHASE_STAGING)) return release(s);
  cudaError_t e = cudaMemcpyAsync(ctx->arena + ad.off, payload_host, nbytes, cudaMemcpyHostToDevice, ctx->stream);
  for (size_t i = 0; i < ad.sp.size() && e == cudaSuccess; ++i)
    e = cudaMemcpyAsync(ctx->arena + ad.off + ad.sp[i].rp_off, rps[i].data(), rps[i].size() * 4,
                        cudaMemcpyHostToDevice, ctx->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return release(cuda_fail(ctx, e, "staging copy"));
  // ---- CHECKSUM: digest of the device copy; finiteness of the f16 values
  // ([DTD] §11: no NaN or Inf in the f16 payloads)
  if (ovl_status s = injected(ctx, OVL_PHASE_CHECKSUM)) return release(s);
  uint8_t dev_digest[32];
  if (ovl_status s = device_digest(ctx, ctx->arena + ad.off, nbytes, ctx->stream, dev_digest)) return release(s);
  if (std::memcmp(dev_digest, ad.digest, 32) != 0) return release(fail(ctx, OVL_E_HASH, "staged copy corrupted"));
  if (nonfinite) return release(fail(ctx, OVL_E_NONFINITE, "overlay values hold NaN or Inf"));
  compute_adapter_key(ad);
  ad.h = ctx->next_h++;
  *out = ad.h;
  ctx->staged.emplace(ad.h, ad);
  return ok(ctx);
}

ovl_status ovl_unstage_adapter(ovl_ctx* ctx, ovl_adapter_h h) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  auto it = ctx->staged.find(h);
  if (it == ctx->staged.end()) return fail(ctx, OVL_E_ARG, "unknown adapter handle");
  for (const auto* comp : {ctx->active.get(), ctx->prev.get()})
    if (comp)
      for (const auto& e : comp->entries)
        if (e.h == h) return fail(ctx, OVL_E_STATE, "adapter is part of the active or rollback composition");
  DeviceGuard g(ctx->device);
  Adapter& a = it->second;
  if (a.used && ctx->fwd_recorded) {
    if (ctx->policy == OVL_SWITCH_DRAIN) {
      cudaEventSynchronize(ctx->fwd_done);
    } else {
      cudaError_t q = cudaEventQuery(ctx->fwd_done);
      if (q == cudaErrorNotReady) return fail(ctx, OVL_E_BUSY, "forward work reading the adapter is in flight");
    }
  }
  ctx->alloc.release(a.off);
  ctx->staged.erase(it);
  return ok(ctx);
}

ovl_status ovl_activate(ovl_ctx* ctx, const ovl_adapter_h* h, const float* scale, uint32_t n, uint32_t mode,
                        uint8_t composition_id_out[32]) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  return ovl::activate_locked(ctx, h, scale, n, mode, composition_id_out);
}

ovl_status ovl_activate_manifest(ovl_ctx* ctx, const char* text, size_t len, uint8_t composition_id_out[32]) {
  using namespace ovl;
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  Manifest m;
  std::string err;
  if (ovl_status st = parse_manifest(text, len, &m, &err)) return fail(ctx, st, err);
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  if (std::memcmp(m.base_hash, ctx->base_digest, 32) != 0)
    return fail(ctx, OVL_E_HASH, "base_model_hash is not the loaded base's digest");
  if (m.quant != ctx->quant) return fail(ctx, OVL_E_QUANT, "quantization is not the loaded base's profile");
  std::vector<ovl_adapter_h> hs;
  std::vector<float> ws;
  for (const ManifestAdapter& e : m.adapters) {
    const Adapter* found = nullptr;   // staged adapters in increasing handle order
    for (const auto& kv : ctx->staged)
      if (std::memcmp(kv.second.digest, e.file_hash, 32) == 0) {
        found = &kv.second;
        break;
      }
    const std::string who = "adapter \"" + e.name + "\": ";
    if (!found) return fail(ctx, OVL_E_HASH, who + "no staged adapter has this file_hash");
    if (found->sparse != (e.type == OVL_ADAPTER_SPARSE))
      return fail(ctx, OVL_E_ARG, who + "type does not match the staged adapter");
    if (e.rank)
      for (const Target& t : found->targets)
        if (t.rank != e.rank) return fail(ctx, OVL_E_SHAPE, who + "rank does not match the staged adapter");
    if (e.has_targets) {
      std::vector<uint32_t> got;
      if (found->sparse)
        for (const SparseTarget& t : found->sp) got.push_back(t.tensor);
      else
        for (const Target& t : found->targets) got.push_back(t.tensor);
      if (got != e.targets) return fail(ctx, OVL_E_SHAPE, who + "targets do not match the staged adapter");
    }
    if (e.has_required_base && std::memcmp(e.required_base, ctx->base_digest, 32) != 0)
      return fail(ctx, OVL_E_HASH, who + "required_base_hash is not the loaded base's digest");
    hs.push_back(found->h);
    ws.push_back(e.merge_weight);
  }
  return activate_locked(ctx, hs.data(), ws.data(), static_cast<uint32_t>(hs.size()), m.mode, composition_id_out);
}

}  // extern "C"

namespace ovl {

// The body of ovl_activate with the context's lock held.
ovl_status activate_locked(ovl_ctx* ctx, const ovl_adapter_h* h, const float* scale, uint32_t n, uint32_t mode,
                           uint8_t composition_id_out[32]) {
  if (ovl_status s = injected(ctx, OVL_PHASE_VALIDATION)) return s;
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  if (n && (!h || !scale)) return fail(ctx, OVL_E_ARG, "null argument");
  if (mode != OVL_MODE_STACK && mode != OVL_MODE_TABLE) return fail(ctx, OVL_E_ARG, "unknown mode");
  if (n > (mode == OVL_MODE_STACK ? uint32_t(OVL_MAX_STACK) : uint32_t(OVL_MAX_TABLE)))
    return fail(ctx, OVL_E_ARG, "too many adapters");
  auto comp = std::make_shared<Composition>();
  comp->mode = n ? mode : static_cast<uint32_t>(OVL_MODE_STACK);
  for (uint32_t i = 0; i < n; ++i) {
    if (!ctx->staged.count(h[i])) return fail(ctx, OVL_E_ARG, "unknown adapter handle");
    for (uint32_t j = 0; j < i; ++j)
      if (h[j] == h[i]) return fail(ctx, OVL_E_DUPLICATE, "adapter listed twice");
    if (!finite_f32(scale[i])) return fail(ctx, OVL_E_ARG, "scale must be finite");
    if (mode == OVL_MODE_TABLE && ctx->staged.at(h[i]).sparse)
      return fail(ctx, OVL_E_ARG, "sparse overlays are applied in STACK compositions only");
    comp->entries.push_back({h[i], scale[i]});
  }
  if (comp->mode == OVL_MODE_STACK) {
    for (uint32_t t = 0; t < ctx->tensors.size(); ++t) {
      uint32_t r = 0;
      for (const auto& e : comp->entries)
        if (const Target* tg = target_for(ctx->staged.at(e.h), t)) r += tg->rank;
      if (r > OVL_MAX_TOTAL_RANK) return fail(ctx, OVL_E_SHAPE, "total rank on a tensor exceeds the limit");
    }
  }
  compute_composition_id(ctx, *comp);
  if (std::memcmp(comp->id, ctx->active->id, 32) == 0) {     // idempotent no-op
    if (composition_id_out) std::memcpy(composition_id_out, comp->id, 32);
    return ok(ctx);
  }
  // ---- COMMIT / SWAP
  if (ovl_status s = injected(ctx, OVL_PHASE_SWAP)) return s;
  DeviceGuard g(ctx->device);
  if (ovl_status s = busy_check(ctx)) return s;
  ctx->prev = ctx->active;
  ctx->active = comp;
  ++ctx->epoch;
  if (composition_id_out) std::memcpy(composition_id_out, comp->id, 32);
  return ok(ctx);
}

}  // namespace ovl

extern "C" {

ovl_status ovl_rollback(ovl_ctx* ctx, uint8_t composition_id_out[32]) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  if (!ctx->prev) return fail(ctx, OVL_E_NO_PREVIOUS, "no previous composition");
  if (ovl_status s = injected(ctx, OVL_PHASE_SWAP)) return s;
  DeviceGuard g(ctx->device);
  if (ovl_status s = busy_check(ctx)) return s;
  ctx->active = ctx->prev;
  ctx->prev.reset();
  ++ctx->epoch;
  if (composition_id_out) std::memcpy(composition_id_out, ctx->active->id, 32);
  return ok(ctx);
}

}  // extern "C"

namespace ovl {
namespace {

// Low-rank terms of `comp` that touch `tensor` (STACK), in composition order.
uint32_t stack_terms(ovl_ctx* c, const Composition& comp, uint32_t tensor, LoraRef* out, uint32_t* rtot,
                     std::vector<Adapter*>* used) {
  uint32_t nl = 0;
  *rtot = 0;
  for (const auto& e : comp.entries) {
    Adapter& a = c->staged.at(e.h);
    const Target* t = target_for(a, tensor);
    if (!t) continue;
    out[nl].A = reinterpret_cast<const float*>(c->arena + a.off + t->a_off);
    out[nl].B = reinterpret_cast<const float*>(c->arena + a.off + t->b_off);
    out[nl].r = t->rank;
    out[nl].s = e.s;
    *rtot += t->rank;
    ++nl;
    used->push_back(&a);
  }
  return nl;
}

// Sparse overlay terms of `comp` that touch `tensor` (STACK), in composition order.
uint32_t sparse_terms(ovl_ctx* c, const Composition& comp, uint32_t tensor, SparseRef* out,
                      std::vector<Adapter*>* used) {
  uint32_t n = 0;
  for (const auto& e : comp.entries) {
    Adapter& a = c->staged.at(e.h);
    if (!a.sparse) continue;
    for (const auto& t : a.sp) {
      if (t.tensor != tensor) continue;
      out[n].idx = reinterpret_cast<const uint32_t*>(c->arena + a.off + t.idx_off);
      out[n].val = reinterpret_cast<const uint16_t*>(c->arena + a.off + t.val_off);
      out[n].rp = reinterpret_cast<const uint32_t*>(c->arena + a.off + t.rp_off);
      out[n].nnz = t.nnz;
      out[n].s = e.s;
      ++n;
      used->push_back(&a);
    }
  }
  return n;
}

// Adds the sparse terms of tensors[0..n) (which share x) to the outputs the
// dense dual path wrote, in one launch; nothing is launched without any.
cudaError_t apply_sparse(ovl_ctx* c, const uint32_t* tensors, uint32_t n, const void* x, uint32_t xdt, uint32_t T,
                         float* const* ys, std::vector<Adapter*>* used, cudaStream_t st) {
  SparseApply sa{};
  for (uint32_t i = 0; i < n; ++i) {
    const uint32_t k0 = sa.nt;
    sa.nt += sparse_terms(c, *c->active, tensors[i], sa.t + sa.nt, used);
    if (sa.nt == k0) continue;
    const ovl_tensor_desc& td = c->tensors[tensors[i]];
    sa.seg[sa.nseg++] = SparseSeg{ys[i], td.d_out, sa.mtot, k0, sa.nt};
    sa.mtot += td.d_out;
  }
  if (sa.nt == 0) return cudaSuccess;
  sa.x = x;
  sa.n = c->tensors[tensors[0]].d_in;
  sa.T = T;
  sa.xdt = xdt;
  return launch_sparse_apply(sa, st);
}

// Adds the sparse terms of `tensor` into a materialized fp32 scratch, in order.
cudaError_t scatter_sparse(ovl_ctx* c, uint32_t tensor, float* S, std::vector<Adapter*>* used, cudaStream_t st) {
  SparseRef sp[OVL_MAX_STACK];
  const uint32_t n = sparse_terms(c, *c->active, tensor, sp, used);
  cudaError_t e = cudaSuccess;
  for (uint32_t k = 0; k < n && e == cudaSuccess; ++k) e = launch_sparse_scatter(S, sp[k], st);
  return e;
}

// Launches of four or more tokens run on the tensor cores (K4) when the shape
// allows: there the integer dot products are bound by issue slots (measured on
// the q4_0 block: 204 vs 184 us at 4 tokens, 431 vs 191 us at 8).
constexpr uint32_t kTcMinT = 4;

// The tensor-core kernel reads the activations 16 bytes at a time.
bool use_tc(const ovl_ctx* c, uint32_t T, const ovl_tensor_desc& td, uint32_t rtot, const void* x) {
  return T >= kTcMinT && (reinterpret_cast<uintptr_t>(x) & 15) == 0 && c->ws.tc_scratch_bytes > 0 &&
         fused_gemm_supported(td.d_out, td.d_in) &&
         fused_gemm_scratch_bytes(T, td.d_in, fused_vcols(rtot)) <= c->ws.tc_scratch_bytes;
}

void tc_tensor(const ovl_ctx* c, const ovl_tensor_desc& td, float* y, const LoraRef* terms, uint32_t nl,
               uint32_t rtot, FusedTensor* out) {
  out->qs = c->base + td.qs_off;
  out->dpl = c->base + td.d_off;
  out->m = td.d_out;
  out->y = y;
  out->nl = nl;
  out->rtot = rtot;
  for (uint32_t k = 0; k < nl; ++k) out->lora[k] = terms[k];
}

void tc_common(const ovl_ctx* c, uint32_t n, const void* x, uint32_t xdt, uint32_t T, FusedLaunch* L) {
  L->quant = c->quant;
  L->n = n;
  L->x = x;
  L->xdt = xdt;
  L->T = T;
  L->scratch = c->ws.tc_scratch;
  L->scratch_bytes = c->ws.tc_scratch_bytes;
  L->status = c->ws.status;
}

cudaError_t launch_tc(const ovl_ctx* c, const ovl_tensor_desc& td, const void* x, uint32_t xdt, uint32_t T, float* y,
                      const LoraRef* terms, uint32_t nl, uint32_t rtot, const int8_t* tok, cudaStream_t st) {
  FusedLaunch L{};
  L.nt = 1;
  tc_tensor(c, td, y, terms, nl, rtot, &L.t[0]);
  tc_common(c, td.d_in, x, xdt, T, &L);
  L.tok_sel = tok != nullptr;
  L.tok_host = tok;
  return launch_fused_gemm(L, st);
}

// A pending OVL_PHASE_DEVICE_WAIT injection applies to the next decode launch
// that has a low-rank term (the gather it disturbs exists only then).
uint32_t take_device_wait_injection(ovl_ctx* c, uint32_t nl) {
  if (nl == 0 || c->inject_phase != OVL_PHASE_DEVICE_WAIT || c->inject_code >= 0) return 0u;
  c->inject_phase = 0;
  c->inject_code = 0;
  return 1u;
}

// One event per forward call: forward work on a context is stream-ordered, so
// once the latest record has completed every earlier forward has too.
ovl_status record_use(ovl_ctx* c, const std::vector<Adapter*>& used, cudaStream_t st) {
  cudaError_t e = cudaEventRecord(c->fwd_done, st);
  if (e != cudaSuccess) return cuda_fail(c, e, "event record");
  c->fwd_recorded = true;
  for (Adapter* a : used) a->used = true;
  return OVL_OK;
}

}  // namespace
}  // namespace ovl

extern "C" {

ovl_status ovl_materialize_layer(ovl_ctx* ctx, uint32_t tensor, float* scratch, size_t scratch_bytes,
                                 void* stream) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  if (tensor >= ctx->tensors.size()) return fail(ctx, OVL_E_ARG, "no such tensor");
  if (ctx->active->mode != OVL_MODE_STACK) return fail(ctx, OVL_E_STATE, "TABLE composition: use ovl_segmented_forward");
  const ovl_tensor_desc& td = ctx->tensors[tensor];
  if (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 15) || scratch_bytes < size_t(td.d_out) * td.d_in * 4)
    return fail(ctx, OVL_E_ARG, "scratch must be 16-byte aligned and hold d_out*d_in floats");
  DeviceGuard g(ctx->device);
  MatArgs m{};
  m.qs = ctx->base + td.qs_off;
  m.dpl = ctx->base + td.d_off;
  m.m = td.d_out;
  m.n = td.d_in;
  m.quant = ctx->quant;
  m.S = scratch;
  uint32_t rtot;
  std::vector<Adapter*> used;
  m.nl = stack_terms(ctx, *ctx->active, tensor, m.lora, &rtot, &used);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_materialize(m, st);
  if (e == cudaSuccess) e = scatter_sparse(ctx, tensor, scratch, &used, st);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "materialize launch");
  if (ovl_status s = record_use(ctx, used, st)) return s;
  return ok(ctx);
}

ovl_status ovl_linear_forward(ovl_ctx* ctx, uint32_t tensor, const void* x, uint32_t x_dtype, uint32_t T,
                              float* y, uint32_t path, float* scratch, size_t scratch_bytes, void* stream) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  if (tensor >= ctx->tensors.size()) return fail(ctx, OVL_E_ARG, "no such tensor");
  if (x_dtype != OVL_F32 && x_dtype != OVL_BF16) return fail(ctx, OVL_E_ARG, "unknown activation dtype");
  if (path != OVL_PATH_DUAL && path != OVL_PATH_JIT) return fail(ctx, OVL_E_ARG, "unknown path");
  if (T > OVL_MAX_T) return fail(ctx, OVL_E_ARG, "T exceeds OVL_MAX_T");
  if (ctx->active->mode != OVL_MODE_STACK) return fail(ctx, OVL_E_STATE, "TABLE composition: use ovl_segmented_forward");
  if (T == 0) return ok(ctx);
  if (!x || !y) return fail(ctx, OVL_E_ARG, "null activation or output");
  const ovl_tensor_desc& td = ctx->tensors[tensor];
  DeviceGuard g(ctx->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LoraRef terms[OVL_MAX_STACK];
  uint32_t rtot;
  std::vector<Adapter*> used;
  const uint32_t nl = stack_terms(ctx, *ctx->active, tensor, terms, &rtot, &used);
  if (path == OVL_PATH_DUAL && use_tc(ctx, T, td, rtot, x)) {
    cudaError_t e = launch_tc(ctx, td, x, x_dtype, T, y, terms, nl, rtot, nullptr, st);
    if (e == cudaSuccess) e = apply_sparse(ctx, &tensor, 1, x, x_dtype, T, &y, &used, st);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "tensor-core launch");
  } else if (path == OVL_PATH_DUAL) {
    DualArgs a{};
    a.b_pad = 1;   // factors live in the arena: 16-byte aligned, allocations rounded to 256 bytes
    a.a16 = 1;
    a.qs = ctx->base + td.qs_off;
    a.dpl = ctx->base + td.d_off;
    a.m = td.d_out;
    a.n = td.d_in;
    a.quant = ctx->quant;
    a.x = x;
    a.xdt = x_dtype;
    a.T = T;
    a.y = y;
    a.nl = nl;
    a.rtot = rtot;
    for (uint32_t i = 0; i < nl; ++i) a.lora[i] = terms[i];
    a.ws = ctx->ws;
    a.epoch = take_device_wait_injection(ctx, nl) ? kEpochWithhold : 0u;
    cudaError_t e = launch_dualpath(a, st);
    if (e == cudaSuccess) e = apply_sparse(ctx, &tensor, 1, x, x_dtype, T, &y, &used, st);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "dual-path launch");
  } else {
    const size_t need = size_t(td.d_out) * td.d_in * 4;
    const size_t xneed = jit_gemm_x_scratch_bytes(T, td.d_in);
    if (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 127) || scratch_bytes < (need + 127) / 128 * 128 + xneed)
      return fail(ctx, OVL_E_ARG, "JIT scratch must be 128-byte aligned and hold the layer plus the widened activations");
    MatArgs m{};
    m.qs = ctx->base + td.qs_off;
    m.dpl = ctx->base + td.d_off;
    m.m = td.d_out;
    m.n = td.d_in;
    m.quant = ctx->quant;
    m.S = scratch;
    m.nl = nl;
    for (uint32_t i = 0; i < nl; ++i) m.lora[i] = terms[i];
    cudaError_t e = launch_materialize(m, st);
    if (e == cudaSuccess) e = scatter_sparse(ctx, tensor, scratch, &used, st);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "materialize launch");
    float* xs = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(scratch) + (need + 127) / 128 * 128);
    e = launch_jit_gemm(scratch, x, x_dtype, T, td.d_out, td.d_in, y, xs, ctx->ws, st);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "JIT GEMM launch");
  }
  if (ovl_status s = record_use(ctx, used, st)) return s;
  return ok(ctx);
}

ovl_status ovl_linear_forward_multi(ovl_ctx* ctx, uint32_t n, const uint32_t* tensors, const void* x,
                                    uint32_t x_dtype, uint32_t T, float* const* ys, void* stream) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  if (n == 0 || n > static_cast<uint32_t>(kMaxMulti) || !tensors || !ys) return fail(ctx, OVL_E_ARG, "need 1 to 4 tensors");
  if (x_dtype != OVL_F32 && x_dtype != OVL_BF16) return fail(ctx, OVL_E_ARG, "unknown activation dtype");
  if (T > OVL_MAX_T) return fail(ctx, OVL_E_ARG, "T exceeds OVL_MAX_T");
  if (ctx->active->mode != OVL_MODE_STACK) return fail(ctx, OVL_E_STATE, "TABLE composition: use ovl_segmented_forward");
  for (uint32_t i = 0; i < n; ++i) {
    if (tensors[i] >= ctx->tensors.size()) return fail(ctx, OVL_E_ARG, "no such tensor");
    if (ctx->tensors[tensors[i]].d_in != ctx->tensors[tensors[0]].d_in)
      return fail(ctx, OVL_E_SHAPE, "tensors of one launch must share d_in");
    if (T && !ys[i]) return fail(ctx, OVL_E_ARG, "null output");
  }
  if (T == 0) return ok(ctx);
  if (!x) return fail(ctx, OVL_E_ARG, "null activation");
  DeviceGuard g(ctx->device);
  {
    // multi-token: one tensor-core launch over all the tensors when every
    // tensor allows it and their s v vectors fit the scratch together
    bool tc_all = T >= kTcMinT;   // single-token decode never takes the tensor-core route: skip the term lookups
    uint32_t vcols = 0;
    for (uint32_t i = 0; i < n && tc_all; ++i) {
      LoraRef terms[OVL_MAX_STACK];
      uint32_t rt;
      std::vector<Adapter*> tmp;
      const uint32_t nl = stack_terms(ctx, *ctx->active, tensors[i], terms, &rt, &tmp);
      tc_all = use_tc(ctx, T, ctx->tensors[tensors[i]], rt, x);
      if (nl) vcols += fused_vcols(rt);
    }
    if (tc_all) tc_all = fused_gemm_scratch_bytes(T, ctx->tensors[tensors[0]].d_in, vcols) <= ctx->ws.tc_scratch_bytes;
    if (tc_all) {
      cudaStream_t st = static_cast<cudaStream_t>(stream);
      std::vector<Adapter*> used;
      FusedLaunch L{};
      L.nt = n;
      for (uint32_t i = 0; i < n; ++i) {
        LoraRef terms[OVL_MAX_STACK];
        uint32_t rt;
        const uint32_t nl = stack_terms(ctx, *ctx->active, tensors[i], terms, &rt, &used);
        tc_tensor(ctx, ctx->tensors[tensors[i]], ys[i], terms, nl, rt, &L.t[i]);
      }
      tc_common(ctx, ctx->tensors[tensors[0]].d_in, x, x_dtype, T, &L);
      cudaError_t e = launch_fused_gemm(L, st);
      if (e == cudaSuccess) e = apply_sparse(ctx, tensors, n, x, x_dtype, T, ys, &used, st);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "tensor-core launch");
      if (ovl_status s = record_use(ctx, used, st)) return s;
      return ok(ctx);
    }
  }
  DualArgs a{};
  a.b_pad = 1;   // factors live in the arena: 16-byte aligned, allocations rounded to 256 bytes
  a.a16 = 1;
  std::vector<Adapter*> used;
  for (uint32_t i = 0; i < n; ++i) {
    const ovl_tensor_desc& td = ctx->tensors[tensors[i]];
    LoraRef terms[OVL_MAX_STACK];
    uint32_t rt;
    const uint32_t nl = stack_terms(ctx, *ctx->active, tensors[i], terms, &rt, &used);
    DualSeg& sgm = a.seg[i];
    sgm.qs = ctx->base + td.qs_off;
    sgm.dpl = ctx->base + td.d_off;
    sgm.y = ys[i];
    sgm.m = td.d_out;
    sgm.k0 = a.nl;
    sgm.rb0 = a.rtot;
    for (uint32_t k = 0; k < nl; ++k) a.lora[a.nl++] = terms[k];
    sgm.k1 = a.nl;
    a.rtot += rt;
    a.m += td.d_out;
  }
  a.nseg = n;
  a.n = ctx->tensors[tensors[0]].d_in;
  a.quant = ctx->quant;
  a.x = x;
  a.xdt = x_dtype;
  a.T = T;
  a.ws = ctx->ws;
  a.epoch = take_device_wait_injection(ctx, a.nl) ? kEpochWithhold : 0u;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_dualpath(a, st);
  if (e == cudaSuccess) e = apply_sparse(ctx, tensors, n, x, x_dtype, T, ys, &used, st);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "multi-tensor launch");
  if (ovl_status s = record_use(ctx, used, st)) return s;
  return ok(ctx);
}

ovl_status ovl_segmented_forward(ovl_ctx* ctx, uint32_t tensor, const void* x, uint32_t x_dtype, uint32_t T,
                                 const int32_t* seg_offsets, const int32_t* seg_slot, uint32_t n_seg,
                                 const int32_t* perm, float* y, void* stream) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  if (ctx->active->mode != OVL_MODE_TABLE) return fail(ctx, OVL_E_STATE, "segmented forward needs a TABLE composition");
  if (tensor >= ctx->tensors.size()) return fail(ctx, OVL_E_ARG, "no such tensor");
  if (x_dtype != OVL_F32 && x_dtype != OVL_BF16) return fail(ctx, OVL_E_ARG, "unknown activation dtype");
  if (T > OVL_MAX_T) return fail(ctx, OVL_E_ARG, "T exceeds OVL_MAX_T");
  if (n_seg > OVL_MAX_SEGMENTS) return fail(ctx, OVL_E_ARG, "too many segments");
  if (T == 0) return ok(ctx);
  if (!x || !y || !seg_offsets || !seg_slot || !perm || n_seg == 0) return fail(ctx, OVL_E_ARG, "null argument");
  // segments: offsets nondecreasing from 0 to T; perm a permutation; slots valid
  const Composition& comp = *ctx->active;
  const int32_t n_slots = static_cast<int32_t>(comp.entries.size());
  if (seg_offsets[0] != 0 || seg_offsets[n_seg] != static_cast<int32_t>(T))
    return fail(ctx, OVL_E_ARG, "segment offsets must run from 0 to T");
  for (uint32_t s = 0; s < n_seg; ++s) {
    if (seg_offsets[s + 1] < seg_offsets[s]) return fail(ctx, OVL_E_ARG, "segment offsets must not decrease");
    if (seg_slot[s] < -1 || seg_slot[s] >= n_slots) return fail(ctx, OVL_E_ARG, "segment slot out of range");
  }
  std::vector<uint8_t> seen(T, 0);
  for (uint32_t j = 0; j < T; ++j) {
    if (perm[j] < 0 || perm[j] >= static_cast<int32_t>(T) || seen[perm[j]]) return fail(ctx, OVL_E_ARG, "perm is not a permutation");
    seen[perm[j]] = 1;
  }
  // low-rank terms: every table slot that targets this tensor
  const ovl_tensor_desc& td = ctx->tensors[tensor];
  DualArgs a{};
  a.b_pad = 1;   // factors live in the arena: 16-byte aligned, allocations rounded to 256 bytes
  a.a16 = 1;
  std::vector<int> slot_term(n_slots, -1);
  std::vector<Adapter*> used;
  for (int32_t sl = 0; sl < n_slots; ++sl) {
    Adapter& ad = ctx->staged.at(comp.entries[sl].h);
    const Target* tg = target_for(ad, tensor);
    if (!tg) continue;
    slot_term[sl] = static_cast<int>(a.nl);
    a.lora[a.nl].A = reinterpret_cast<const float*>(ctx->arena + ad.off + tg->a_off);
    a.lora[a.nl].B = reinterpret_cast<const float*>(ctx->arena + ad.off + tg->b_off);
    a.lora[a.nl].r = tg->rank;
    a.lora[a.nl].s = comp.entries[sl].s;
    a.rtot += tg->rank;
    ++a.nl;
    used.push_back(&ad);
  }
  if (a.rtot > kMaxTableRank) return fail(ctx, OVL_E_SHAPE, "total rank of the table on this tensor exceeds the limit");
  // request r (row r of x and y) uses the slot of the segment holding it
  std::vector<int8_t> tok(T, -1);
  for (uint32_t s = 0; s < n_seg; ++s)
    for (int32_t j = seg_offsets[s]; j < seg_offsets[s + 1]; ++j)
      tok[perm[j]] = static_cast<int8_t>(seg_slot[s] >= 0 ? slot_term[seg_slot[s]] : -1);
  DeviceGuard g(ctx->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  a.qs = ctx->base + td.qs_off;
  a.dpl = ctx->base + td.d_off;
  a.m = td.d_out;
  a.n = td.d_in;
  a.quant = ctx->quant;
  a.x = x;
  a.xdt = x_dtype;
  a.T = T;
  a.y = y;
  a.tok_sel = 1;
  a.tok_host = tok.data();
  a.ws = ctx->ws;
  cudaError_t e = use_tc(ctx, T, td, a.rtot, x)
                      ? launch_tc(ctx, td, x, x_dtype, T, y, a.lora, a.nl, a.rtot, tok.data(), st)
                      : launch_dualpath(a, st);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "segmented launch");
  if (ovl_status s = record_use(ctx, used, st)) return s;
  return ok(ctx);
}

ovl_status ovl_base_digest(ovl_ctx* ctx, uint8_t digest_out[32], void* stream) {
  if (!ctx || !digest_out) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!ctx->base_loaded) return fail(ctx, OVL_E_STATE, "no base loaded");
  DeviceGuard g(ctx->device);
  if (ovl_status s = device_digest(ctx, ctx->base, ctx->base_bytes, static_cast<cudaStream_t>(stream), digest_out))
    return s;
  return ok(ctx);
}

ovl_status ovl_get_state(ovl_ctx* ctx, ovl_state* out) {
  if (!ctx || !out) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  std::memset(out, 0, sizeof(*out));
  out->base_loaded = ctx->base_loaded;
  out->arena_bytes = ctx->arena_bytes;
  out->arena_used = ctx->alloc.used() + kReservedEnd;
  out->n_staged = static_cast<uint32_t>(ctx->staged.size());
  if (ctx->base_loaded) {
    std::memcpy(out->composition_id, ctx->active->id, 32);
    std::memcpy(out->base_digest, ctx->base_digest, 32);
    out->quant = ctx->quant;
    out->mode = ctx->active->mode;
    out->n_entries = static_cast<uint32_t>(ctx->active->entries.size());
    out->has_previous = ctx->prev ? 1u : 0u;
    out->epoch = ctx->epoch;
  }
  return ok(ctx);
}

ovl_status ovl_get_entry(ovl_ctx* ctx, uint32_t i, ovl_entry* out) {
  if (!ctx || !out) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!ctx->base_loaded || i >= ctx->active->entries.size()) return fail(ctx, OVL_E_ARG, "no such entry");
  const Entry& e = ctx->active->entries[i];
  const Adapter& a = ctx->staged.at(e.h);
  out->handle = e.h;
  std::memcpy(out->adapter_key, a.key, 32);
  out->scale = e.s;
  out->total_rank = a.total_rank;
  return ok(ctx);
}

ovl_status ovl_check_device(ovl_ctx* ctx, void* stream) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  DeviceGuard g(ctx->device);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  uint32_t st = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&st, ctx->ws.status, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "check device");
  if (st != kDevOk) {
    // Reset the status word so the next launch starts clean (the partial-sum
    // slots need nothing: every launch tags its own with a fresh epoch).
    cudaMemset(ctx->ws.status, 0, 4);
    return fail(ctx, OVL_E_DEVICE_TIMEOUT, "a bounded device wait ran out (code " + std::to_string(st) + ")");
  }
  return ok(ctx);
}

ovl_status ovl_debug_inject(ovl_ctx* ctx, uint32_t phase, ovl_status code) {
  if (!ctx) return OVL_E_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (code > 0 || phase < OVL_PHASE_VALIDATION || phase > OVL_PHASE_DEVICE_WAIT) return fail(ctx, OVL_E_ARG, "bad injection");
  if (phase == OVL_PHASE_DEVICE_WAIT && code != 0 && code != OVL_E_DEVICE_TIMEOUT)
    return fail(ctx, OVL_E_ARG, "a device-wait injection takes OVL_E_DEVICE_TIMEOUT");
  ctx->inject_phase = code ? phase : 0;
  ctx->inject_code = code;
  return ok(ctx);
}

}  // extern "C"
