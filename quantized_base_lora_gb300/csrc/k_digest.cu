// Content digests and payload checks.
//
// Content digest = SHA-256 over the concatenation of SHA-256(leaf_i) for
// consecutive 64 KiB leaves.  The leaves of a device buffer are hashed on the
// GPU (one thread per leaf, ~113 K independent leaves for a 7.4 GB base); the
// short root pass runs on the host.  Sources: "We propose a content-addressed
// overlay system" report §"Explicit Correctness and Atomicity Invariants"
// (Checksum Verification: SHA-256 of every artifact); "Deep Technical Design
// ..." §2 (Oracle Invariant: base bytes bit-identical from init to
// termination), §6 CHECKSUM VERIFICATION (detect in-flight corruption after
// staging), §11 Deep Compatibility Checks (no NaN/Inf in payloads).
#include <thread>
#include <vector>

#include "ovl_internal.h"
#include "sha256.cuh"

namespace ovl {
namespace {

__device__ __forceinline__ uint32_t bswap32(uint32_t v) { return __byte_perm(v, 0, 0x0123); }

__global__ void __launch_bounds__(128) k_leaf_digests(const uint8_t* __restrict__ data, size_t n,
                                                       uint8_t* __restrict__ out, size_t n_leaves) {
  const size_t leaf = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (leaf >= n_leaves) return;
  const size_t begin = leaf * kLeaf;
  const size_t len = (n - begin) < kLeaf ? (n - begin) : kLeaf;
  const uint8_t* p = data + begin;
  uint32_t h[8];
  sha256_init(h);
  uint32_t w[16];
  const size_t full = len / 64;
  const bool aligned = (reinterpret_cast<uintptr_t>(p) & 15) == 0;
  for (size_t b = 0; b < full; ++b) {
    if (aligned) {
      const uint4* q = reinterpret_cast<const uint4*>(p + 64 * b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(q + i);
        w[4 * i + 0] = bswap32(v.x);
        w[4 * i + 1] = bswap32(v.y);
        w[4 * i + 2] = bswap32(v.z);
        w[4 * i + 3] = bswap32(v.w);
      }
    } else {
      for (int i = 0; i < 16; ++i) w[i] = load_be32(p + 64 * b + 4 * i);
    }
    sha256_compress(h, w);
  }
  // tail and padding (FIPS 180-4 §5.1.1)
  uint8_t tail[128];
  const size_t rem = len - 64 * full;
  for (size_t i = 0; i < rem; ++i) tail[i] = p[64 * full + i];
  tail[rem] = 0x80;
  const size_t tl = (rem + 9 <= 64) ? 64 : 128;
  for (size_t i = rem + 1; i < tl - 8; ++i) tail[i] = 0;
  const uint64_t bits = static_cast<uint64_t>(len) * 8u;
  for (int i = 0; i < 8; ++i) tail[tl - 1 - i] = static_cast<uint8_t>(bits >> (8 * i));
  for (size_t b = 0; b < tl / 64; ++b) {
    for (int i = 0; i < 16; ++i) w[i] = load_be32(tail + 64 * b + 4 * i);
    sha256_compress(h, w);
  }
  uint8_t* o = out + leaf * 32;
  for (int i = 0; i < 8; ++i) {
    o[4 * i + 0] = static_cast<uint8_t>(h[i] >> 24);
    o[4 * i + 1] = static_cast<uint8_t>(h[i] >> 16);
    o[4 * i + 2] = static_cast<uint8_t>(h[i] >> 8);
    o[4 * i + 3] = static_cast<uint8_t>(h[i]);
  }
}

__global__ void k_finite_scan(const float* __restrict__ p, size_t n, uint32_t* flag) {
  bool bad = false;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint32_t u = __float_as_uint(__ldg(p + i));
    bad |= (u & 0x7F800000u) == 0x7F800000u;   // exponent all ones: Inf or NaN
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicAdd(flag, 1u);
}

}  // namespace

cudaError_t launch_leaf_digests(const uint8_t* data, size_t n, uint8_t* leaf_digests,
                                cudaStream_t st) {
  const size_t leaves = (n + kLeaf - 1) / kLeaf;
  if (leaves == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((leaves + 127) / 128);
  k_leaf_digests<<<blocks, 128, 0, st>>>(data, n, leaf_digests, leaves);
  return cudaGetLastError();
}

cudaError_t launch_finite_scan(const float* p, size_t n, uint32_t* flag, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  size_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  k_finite_scan<<<static_cast<unsigned>(blocks), 256, 0, st>>>(p, n, flag);
  return cudaGetLastError();
}

void host_sha256(const void* data, size_t n, uint8_t out[32]) {
  sha256_bytes(static_cast<const uint8_t*>(data), n, out);
}

void host_digest_of_leaves(const uint8_t* leaf_digests, size_t n_leaves, uint8_t out[32]) {
  sha256_bytes(leaf_digests, n_leaves * 32, out);
}

void host_content_digest(const void* data, size_t n, uint8_t out[32]) {
  const uint8_t* p = static_cast<const uint8_t*>(data);
  const size_t leaves = (n + kLeaf - 1) / kLeaf;
  std::vector<uint8_t> dig(leaves * 32);
  unsigned nt = std::thread::hardware_concurrency();
  if (nt == 0) nt = 1;
  if (nt > 32) nt = 32;
  if (leaves < 8 * nt) nt = 1;
  auto work = [&](size_t a, size_t b) {
    for (size_t i = a; i < b; ++i) {
      const size_t len = (n - i * kLeaf) < kLeaf ? (n - i * kLeaf) : kLeaf;
      sha256_bytes(p + i * kLeaf, len, dig.data() + 32 * i);
    }
  };
  if (nt == 1) {
    work(0, leaves);
  } else {
    std::vector<std::thread> th;
    for (unsigned t = 0; t < nt; ++t) th.emplace_back(work, leaves * t / nt, leaves * (t + 1) / nt);
    for (auto& x : th) x.join();
  }
  sha256_bytes(dig.data(), dig.size(), out);
}

}  // namespace ovl
