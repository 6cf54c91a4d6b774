// Staging of a decode step's activations from pinned host memory into device
// memory, as one kernel in the stream's programmatic launch chain.
//
// A plain host-to-device copy between two forward launches makes the next
// launch wait for the copy engine and start cold.  This kernel instead reads
// the source (page-locked host memory, reached through the unified address
// space) before its grid dependency resolves, triggers its dependents at once
// so the next forward's CTAs become resident and stream their weights, and
// writes the destination only after the preceding grid has completed -- so it
// never overwrites activations that earlier kernels on the stream still read.
//
// There is no counterpart in the source pages: it is a runtime helper around
// the dual-path calls.
#include <cuda_runtime.h>

#include <algorithm>

#include "ovl_internal.h"
#include "ptx.cuh"

namespace ovl {
namespace {

// 128 threads of at most 32 registers (4096 registers a CTA): it fits on an SM
// beside two resident decode CTAs (2 x 320 threads x 96 registers), so it never
// keeps a CTA of the next launch from becoming resident early.
constexpr int kStageThreads = 128;
constexpr int kStageVec = 4;          // 16-byte words a thread holds across the dependency

// Each CTA copies chunks of kStageThreads * kStageVec 16-byte words; the first
// chunk of every CTA is loaded before the grid dependency resolves.
__global__ void __launch_bounds__(kStageThreads, 16) k_stage_copy(uint4* __restrict__ dst,
                                                              const uint4* __restrict__ src, size_t nvec,
                                                              uint8_t* __restrict__ dst_tail,
                                                              const uint8_t* __restrict__ src_tail, uint32_t ntail) {
  griddep_launch_dependents();
  const size_t chunk = static_cast<size_t>(kStageThreads) * kStageVec;
  size_t base = static_cast<size_t>(blockIdx.x) * chunk;
  uint4 v[kStageVec];
#pragma unroll
  for (int k = 0; k < kStageVec; ++k) {
    const size_t i = base + threadIdx.x + static_cast<size_t>(k) * kStageThreads;
    if (i < nvec) v[k] = src[i];
  }
  uint8_t tb = 0;
  const bool tail = blockIdx.x == 0 && threadIdx.x < ntail;
  if (tail) tb = src_tail[threadIdx.x];
  griddep_wait();
  for (;;) {
#pragma unroll
    for (int k = 0; k < kStageVec; ++k) {
      const size_t i = base + threadIdx.x + static_cast<size_t>(k) * kStageThreads;
      if (i < nvec) dst[i] = v[k];
    }
    base += static_cast<size_t>(gridDim.x) * chunk;
    if (base >= nvec) break;
#pragma unroll
    for (int k = 0; k < kStageVec; ++k) {
      const size_t i = base + threadIdx.x + static_cast<size_t>(k) * kStageThreads;
      if (i < nvec) v[k] = src[i];
    }
  }
  if (tail) dst_tail[threadIdx.x] = tb;
}

}  // namespace
}  // namespace ovl

extern "C" ovl_status ovl_stage_activations(void* dst, const void* src_host, size_t nbytes, void* stream) {
  using namespace ovl;
  if (nbytes == 0) return OVL_OK;
  if (!dst || !src_host) return OVL_E_ARG;
  // Both ends must be reachable from the device: page-locked (registered) host
  // memory, device memory or managed memory.  Pageable host memory is refused
  // before anything is launched.
  void* dptr[2] = {nullptr, nullptr};
  const void* ends[2] = {dst, src_host};
  void* const dst_in = dst;
  const void* const src_in = src_host;
  for (int k = 0; k < 2; ++k) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, ends[k]) != cudaSuccess) {
      cudaGetLastError();
      return OVL_E_ARG;
    }
    if (at.type == cudaMemoryTypeUnregistered || !at.devicePointer) return OVL_E_ARG;
    dptr[k] = at.devicePointer;
  }
  dst = dptr[0];
  src_host = dptr[1];
  const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src_host);
  if ((d & 15) != (s & 15)) return OVL_E_ARG;
  // the 16-byte aligned body [d0, d1) and up to 15 head bytes and 15 tail bytes
  const uintptr_t d0 = (d + 15) & ~static_cast<uintptr_t>(15);
  const size_t head = std::min<size_t>(nbytes, d0 - d);
  const size_t nvec = (nbytes - head) / 16;
  const size_t tail = nbytes - head - nvec * 16;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (head) {
    // an unaligned head is rare (callers pass allocations); it goes ahead as a
    // plain stream-ordered copy
    e = cudaMemcpyAsync(dst_in, src_in, head, cudaMemcpyDefault, st);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return OVL_E_CUDA;
    }
  }
  static int nsm = [] {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
  }();
  const size_t chunk = static_cast<size_t>(kStageThreads) * kStageVec;
  const uint32_t grid = static_cast<uint32_t>(std::max<size_t>(1, std::min<size_t>((nvec + chunk - 1) / chunk, nsm)));
  uint8_t* db = static_cast<uint8_t*>(dst) + head;
  const uint8_t* sb = static_cast<const uint8_t*>(src_host) + head;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStageThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_stage_copy, reinterpret_cast<uint4*>(db), reinterpret_cast<const uint4*>(sb), nvec,
                         db + nvec * 16, sb + nvec * 16, static_cast<uint32_t>(tail));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return OVL_E_CUDA;
  }
  return OVL_OK;
}
