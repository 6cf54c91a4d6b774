// SHA-256 from FIPS 180-4 (Secure Hash Standard), sections 4.1.2, 4.2.2,
// 5.1.1, 5.3.3 and 6.2.  One compression routine serves the host (identity,
// staging digests) and the device (leaf hashing of the base and of staged
// adapters).  Constants: FIPS 180-4 §4.2.2 (first 32 bits of the fractional
// parts of the cube roots of the first 64 primes) and §5.3.3 (square roots of
// the first 8 primes).
#pragma once
#include <stddef.h>
#include <stdint.h>

#ifdef __CUDACC__
#define OVL_HD __host__ __device__ __forceinline__
#else
#define OVL_HD inline
#endif

namespace ovl {

#define OVL_SHA256_K_LIST                                                                      \
  0x428a2f98u, 0x71374491u, 0xb5c0fbcfu, 0xe9b5dba5u, 0x3956c25bu, 0x59f111f1u, 0x923f82a4u,   \
      0xab1c5ed5u, 0xd807aa98u, 0x12835b01u, 0x243185beu, 0x550c7dc3u, 0x72be5d74u,           \
      0x80deb1feu, 0x9bdc06a7u, 0xc19bf174u, 0xe49b69c1u, 0xefbe4786u, 0x0fc19dc6u,           \
      0x240ca1ccu, 0x2de92c6fu, 0x4a7484aau, 0x5cb0a9dcu, 0x76f988dau, 0x983e5152u,           \
      0xa831c66du, 0xb00327c8u, 0xbf597fc7u, 0xc6e00bf3u, 0xd5a79147u, 0x06ca6351u,           \
      0x14292967u, 0x27b70a85u, 0x2e1b2138u, 0x4d2c6dfcu, 0x53380d13u, 0x650a7354u,           \
      0x766a0abbu, 0x81c2c92eu, 0x92722c85u, 0xa2bfe8a1u, 0xa81a664bu, 0xc24b8b70u,           \
      0xc76c51a3u, 0xd192e819u, 0xd6990624u, 0xf40e3585u, 0x106aa070u, 0x19a4c116u,           \
      0x1e376c08u, 0x2748774cu, 0x34b0bcb5u, 0x391c0cb3u, 0x4ed8aa4au, 0x5b9cca4fu,           \
      0x682e6ff3u, 0x748f82eeu, 0x78a5636fu, 0x84c87814u, 0x8cc70208u, 0x90befffau,           \
      0xa4506cebu, 0xbef9a3f7u, 0xc67178f2u

#ifdef __CUDACC__
__constant__ static const uint32_t kSha256K_dev[64] = {OVL_SHA256_K_LIST};
#endif
static const uint32_t kSha256K_host[64] = {OVL_SHA256_K_LIST};

OVL_HD uint32_t sha_rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

OVL_HD void sha256_init(uint32_t h[8]) {
  h[0] = 0x6a09e667u; h[1] = 0xbb67ae85u; h[2] = 0x3c6ef372u; h[3] = 0xa54ff53au;
  h[4] = 0x510e527fu; h[5] = 0x9b05688cu; h[6] = 0x1f83d9abu; h[7] = 0x5be0cd19u;
}

// One compression of a 16-word big-endian message block (FIPS 180-4 §6.2.2).
// The 64-entry schedule is kept as a rolling window of 16 words.
OVL_HD void sha256_compress(uint32_t h[8], uint32_t w[16]) {
#ifdef __CUDA_ARCH__
  const uint32_t* K = kSha256K_dev;
#else
  const uint32_t* K = kSha256K_host;
#endif
  uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
#ifdef __CUDA_ARCH__
#pragma unroll
#endif
  for (int t = 0; t < 64; ++t) {
    uint32_t wt;
    if (t < 16) {
      wt = w[t];
    } else {
      uint32_t w15 = w[(t - 15) & 15], w2 = w[(t - 2) & 15];
      uint32_t s0 = sha_rotr(w15, 7) ^ sha_rotr(w15, 18) ^ (w15 >> 3);
      uint32_t s1 = sha_rotr(w2, 17) ^ sha_rotr(w2, 19) ^ (w2 >> 10);
      wt = w[t & 15] + s0 + w[(t - 7) & 15] + s1;
      w[t & 15] = wt;
    }
    uint32_t S1 = sha_rotr(e, 6) ^ sha_rotr(e, 11) ^ sha_rotr(e, 25);
    uint32_t ch = (e & f) ^ (~e & g);
    uint32_t t1 = hh + S1 + ch + K[t] + wt;
    uint32_t S0 = sha_rotr(a, 2) ^ sha_rotr(a, 13) ^ sha_rotr(a, 22);
    uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
    uint32_t t2 = S0 + maj;
    hh = g; g = f; f = e; e = d + t1; d = c; c = b; b = a; a = t1 + t2;
  }
  h[0] += a; h[1] += b; h[2] += c; h[3] += d; h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
}

OVL_HD uint32_t load_be32(const uint8_t* p) {
  return ((uint32_t)p[0] << 24) | ((uint32_t)p[1] << 16) | ((uint32_t)p[2] << 8) | (uint32_t)p[3];
}

// Byte-wise one-shot SHA-256 (padding per FIPS 180-4 §5.1.1).  Used on the host
// and for short device tails; the device leaf kernel has its own word loop.
OVL_HD void sha256_bytes(const uint8_t* data, size_t n, uint8_t out[32]) {
  uint32_t h[8];
  sha256_init(h);
  uint32_t w[16];
  size_t full = n / 64;
  for (size_t b = 0; b < full; ++b) {
    for (int i = 0; i < 16; ++i) w[i] = load_be32(data + 64 * b + 4 * i);
    sha256_compress(h, w);
  }
  uint8_t tail[128];
  size_t rem = n - 64 * full;
  for (size_t i = 0; i < rem; ++i) tail[i] = data[64 * full + i];
  tail[rem] = 0x80;
  size_t tl = (rem + 1 + 8 <= 64) ? 64 : 128;
  for (size_t i = rem + 1; i < tl - 8; ++i) tail[i] = 0;
  uint64_t bits = (uint64_t)n * 8u;
  for (int i = 0; i < 8; ++i) tail[tl - 1 - i] = (uint8_t)(bits >> (8 * i));
  for (size_t b = 0; b < tl / 64; ++b) {
    for (int i = 0; i < 16; ++i) w[i] = load_be32(tail + 64 * b + 4 * i);
    sha256_compress(h, w);
  }
  for (int i = 0; i < 8; ++i) {
    out[4 * i + 0] = (uint8_t)(h[i] >> 24);
    out[4 * i + 1] = (uint8_t)(h[i] >> 16);
    out[4 * i + 2] = (uint8_t)(h[i] >> 8);
    out[4 * i + 3] = (uint8_t)(h[i]);
  }
}

// Incremental host hasher for building identity strings.
struct Sha256Stream {
  uint32_t h[8];
  uint8_t buf[64];
  size_t len = 0;
  uint64_t total = 0;
  Sha256Stream() { sha256_init(h); }
  void update(const void* p, size_t n) {
    const uint8_t* d = static_cast<const uint8_t*>(p);
    total += n;
    while (n) {
      size_t take = 64 - len < n ? 64 - len : n;
      for (size_t i = 0; i < take; ++i) buf[len + i] = d[i];
      len += take; d += take; n -= take;
      if (len == 64) {
        uint32_t w[16];
        for (int i = 0; i < 16; ++i) w[i] = load_be32(buf + 4 * i);
        sha256_compress(h, w);
        len = 0;
      }
    }
  }
  void u32(uint32_t v) { uint8_t b[4] = {(uint8_t)v, (uint8_t)(v >> 8), (uint8_t)(v >> 16), (uint8_t)(v >> 24)}; update(b, 4); }
  void u64(uint64_t v) { u32((uint32_t)v); u32((uint32_t)(v >> 32)); }
  void final(uint8_t out[32]) {
    uint64_t bits = total * 8u;
    uint8_t pad = 0x80;
    update(&pad, 1);
    uint8_t z = 0;
    while (len != 56) update(&z, 1);
    uint8_t lb[8];
    for (int i = 0; i < 8; ++i) lb[i] = (uint8_t)(bits >> (56 - 8 * i));
    update(lb, 8);
    for (int i = 0; i < 8; ++i) {
      out[4 * i + 0] = (uint8_t)(h[i] >> 24); out[4 * i + 1] = (uint8_t)(h[i] >> 16);
      out[4 * i + 2] = (uint8_t)(h[i] >> 8);  out[4 * i + 3] = (uint8_t)(h[i]);
    }
  }
};

}  // namespace ovl
