// Allocation-free variant of the dual-path forward.
//
// The regular entry point (ovl_linear_forward) takes its kernel scratch -- the
// low-rank partial sums and the device status word -- from the arena that the
// caller lent to ovl_create.  Some callers have no arena to lend and cannot
// allocate device memory when they call: an embedder whose device memory is
// owned entirely by its own pooled allocator, or a caller on a latency-critical
// path that cannot take the device-wide stall a cudaMalloc may cause.  For them
// this file keeps the scratch in one file-scope device array, sized once at
// load time, so a call needs nothing but the caller's inputs and outputs.
//
// There is no counterpart to this entry point in the source pages; it is an
// interface convenience around the same kernel (k_dualpath) and computes
// exactly what ovl_linear_forward computes for a STACK composition.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "ovl_internal.h"

namespace ovl {
namespace {

// 2 MiB of scratch per device: a 512 B head holding the status word, the rest
// epoch-tagged low-rank partial-sum slots (8 bytes per T-tile x total rank x
// shrink CTA; the launch lowers the number of shrink CTAs to fit).  Every GPU
// that loads the library keeps this array until the process exits.
constexpr size_t kNoAllocBytes = 2u << 20;
constexpr size_t kNoAllocStatus = 0;
constexpr size_t kNoAllocPartial = 512;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

std::mutex g_setup_mu;
uint8_t* g_scratch_addr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

// Device address of the array on the current device, looked up (and the array
// cleared) on the first call for that device.  In host code the array's name is
// only a host-side stand-in, so the kernel receives this looked-up address.
cudaError_t scratch_for_current_device(uint8_t** out, int* sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaMemset(p, 0, kNoAllocBytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    g_sms[dev] = sms > 0 ? sms : 1;
    g_scratch_addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_addr[dev];
  *sms_out = g_sms[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace ovl

extern "C" ovl_status ovl_dualpath_forward_noalloc(const void* qs, const void* d, uint32_t quant, uint32_t d_out,
                                                   uint32_t d_in, const float* const* A, const float* const* B,
                                                   const uint32_t* rank, const float* scale, uint32_t n_terms,
                                                   const void* x, uint32_t x_dtype, uint32_t T, float* y,
                                                   void* stream) {
  using namespace ovl;
  if (quant != OVL_Q8_0 && quant != OVL_Q4_0) return OVL_E_QUANT;
  if (d_out == 0 || d_in == 0 || d_in % kQK != 0) return OVL_E_SHAPE;
  if (x_dtype != OVL_F32 && x_dtype != OVL_BF16) return OVL_E_ARG;
  if (T > OVL_MAX_T) return OVL_E_ARG;
  if (n_terms > OVL_MAX_STACK) return OVL_E_ARG;
  if (n_terms && (!A || !B || !rank || !scale)) return OVL_E_ARG;
  if (!qs || !d || (T && (!x || !y))) return OVL_E_ARG;
  if ((reinterpret_cast<uintptr_t>(qs) & 15) || (reinterpret_cast<uintptr_t>(d) & 15))
    return OVL_E_SHAPE;
  DualArgs a{};
  uint32_t rtot = 0;
  for (uint32_t k = 0; k < n_terms; ++k) {
    if (!A[k] || !B[k]) return OVL_E_ARG;
    if (rank[k] == 0 || rank[k] > OVL_MAX_RANK) return OVL_E_SHAPE;
    if (!std::isfinite(scale[k])) return OVL_E_ARG;
    a.lora[k] = LoraRef{A[k], B[k], rank[k], scale[k]};
    rtot += rank[k];
  }
  if (rtot > OVL_MAX_TOTAL_RANK) return OVL_E_SHAPE;
  if (T == 0) return OVL_OK;

  uint8_t* scratch = nullptr;
  int sms = 1;
  cudaError_t e = scratch_for_current_device(&scratch, &sms);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return OVL_E_CUDA;
  }
  // The launch fits its number of shrink CTAs to the slots; it needs at least
  // one CTA's slots for a full token tile of 8.
  const uint64_t need = kNoAllocPartial + 8ull * 8 * rtot;
  if (n_terms && need > kNoAllocBytes) return OVL_E_OOM;   // more scratch than the static array holds
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Clear the status word and every partial-sum slot this call's launches can
  // use (at most 8 tokens x total rank x one shrink CTA per SM, 8 bytes each);
  // the launches then tag their slots with epochs 1, 2, ... counted in this
  // call alone, so no slot written by an earlier call is ever accepted.
  const uint64_t used = n_terms ? kNoAllocPartial + 8ull * 8 * rtot * static_cast<uint64_t>(sms) : kNoAllocPartial;
  e = cudaMemsetAsync(scratch, 0, static_cast<size_t>(std::min<uint64_t>(used, kNoAllocBytes)), st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return OVL_E_CUDA;
  }
  uint32_t epoch = 0;
  a.qs = static_cast<const uint8_t*>(qs);
  a.dpl = static_cast<const uint8_t*>(d);
  a.m = d_out;
  a.n = d_in;
  a.quant = quant;
  a.x = x;
  a.xdt = x_dtype;
  a.T = T;
  a.y = y;
  a.nl = n_terms;
  a.rtot = rtot;
  a.ws.status = reinterpret_cast<uint32_t*>(scratch + kNoAllocStatus);
  a.ws.partial = reinterpret_cast<float*>(scratch + kNoAllocPartial);
  a.ws.partial_floats = (kNoAllocBytes - kNoAllocPartial) / sizeof(float);
  a.ws.epoch_counter = &epoch;
  // B rows are bulk-copied in 16-byte granules only when that stays inside the
  // caller's B arrays.
  a.b_pad = 1;
  a.a16 = 1;
  for (uint32_t k = 0; k < n_terms; ++k) {
    if ((reinterpret_cast<uintptr_t>(B[k]) & 15) || (static_cast<uint64_t>(d_out) * rank[k] * 4) % 16) a.b_pad = 0;
    if (reinterpret_cast<uintptr_t>(A[k]) & 15) a.a16 = 0;
  }
  e = launch_dualpath(a, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return OVL_E_CUDA;
  }
  return OVL_OK;
}
