// K2: per-layer JIT materialization  S = deq(W_q) + sum_k s_k B_k A_k  (fp32).
//
// Sources: "Deep Technical Design: Exact, Atomic, Reversible Specialist Overlays
// on Quantized Transformer Bases" §1 (Per-Layer JIT CoW Materialization: one
// layer into an f32 scratchpad, merged with the adapter, consumed, discarded),
// §5 (Fresh-Base Oracle Definition: materialize without requantizing),
// §7 (Scratch Overhead: one f32 weight matrix).
//
// One CTA writes a 32 x 128 tile: every thread dequantizes and accumulates a
// 4 x 4 patch (float4 stores, coalesced).  The low-rank terms are added adapter
// by adapter (s_k times the rank-r_k sum), with rank chunks of 32 staged in
// shared memory.  With no adapters the output is the exact dequantized tensor
// (d * q is exact in fp32).
#include <cuda_fp16.h>

#include "ovl_internal.h"

namespace ovl {
namespace {

constexpr int TR = 32, TC = 128, KC = 32;

__global__ void __launch_bounds__(256) k_materialize(const MatArgs a) {
  __shared__ float As[KC][TC];
  __shared__ float Bs[TR][KC + 1];
  const int tid = threadIdx.x;
  const int tx = tid & 31;           // column group: 4 columns each
  const int ty = tid >> 5;           // row group: 4 rows each
  const uint32_t row0 = blockIdx.y * TR, col0 = blockIdx.x * TC;
  const uint32_t c = col0 + tx * 4;
  float acc[4][4];
  // dequantized base
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t r = row0 + ty * 4 + i;
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    if (r < a.m && c < a.n && a.quant == OVL_Q4_K) {
      // 16-byte super-block header: d, dmin, 6-bit sc_j and m_j of sub-block
      // j = (c mod 256) / 32 (all four columns lie in one sub-block).
      const uint4 h = *reinterpret_cast<const uint4*>(a.dpl + static_cast<size_t>(r) * (a.n / 16) + (c / kQKK) * 16);
      const uint32_t j6 = 6u * ((c % kQKK) / kQK);
      const uint64_t scf = (static_cast<uint64_t>(h.z & 0xFFFFu) << 32) | h.y;
      const uint64_t mnf = (static_cast<uint64_t>(h.w) << 16) | (h.z >> 16);
      const float dsc = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x & 0xFFFFu))) *
                        static_cast<float>(static_cast<uint32_t>(scf >> j6) & 63u);
      const float dmn = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x >> 16))) *
                        static_cast<float>(static_cast<uint32_t>(mnf >> j6) & 63u);
      const uchar2 q = *reinterpret_cast<const uchar2*>(a.qs + static_cast<size_t>(r) * (a.n / 2) + c / 2);
      // d*sc*code (<= 21 significant bits) and dmin*m (<= 17) are exact in
      // fp32; the fused multiply-add rounds their difference once.
      acc[i][0] = fmaf(dsc, static_cast<float>(q.x & 0xF), -dmn);
      acc[i][1] = fmaf(dsc, static_cast<float>(q.x >> 4), -dmn);
      acc[i][2] = fmaf(dsc, static_cast<float>(q.y & 0xF), -dmn);
      acc[i][3] = fmaf(dsc, static_cast<float>(q.y >> 4), -dmn);
    } else if (r < a.m && c < a.n) {
      const __half dh = reinterpret_cast<const __half*>(a.dpl)[static_cast<size_t>(r) * (a.n / kQK) + c / kQK];
      const float d = __half2float(dh);
      if (a.quant == OVL_Q8_0) {
        const char4 q = *reinterpret_cast<const char4*>(a.qs + static_cast<size_t>(r) * a.n + c);
        acc[i][0] = d * static_cast<float>(q.x);
        acc[i][1] = d * static_cast<float>(q.y);
        acc[i][2] = d * static_cast<float>(q.z);
        acc[i][3] = d * static_cast<float>(q.w);
      } else {
        const uchar2 q = *reinterpret_cast<const uchar2*>(a.qs + static_cast<size_t>(r) * (a.n / 2) + c / 2);
        acc[i][0] = d * static_cast<float>(static_cast<int>(q.x & 0xF) - 8);
        acc[i][1] = d * static_cast<float>(static_cast<int>(q.x >> 4) - 8);
        acc[i][2] = d * static_cast<float>(static_cast<int>(q.y & 0xF) - 8);
        acc[i][3] = d * static_cast<float>(static_cast<int>(q.y >> 4) - 8);
      }
    }
  }
  for (uint32_t k = 0; k < a.nl; ++k) {
    const LoraRef L = a.lora[k];
    float dl[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) dl[i][j] = 0.f;
    for (uint32_t t0 = 0; t0 < L.r; t0 += KC) {
      __syncthreads();
      for (int e = tid; e < KC * TC; e += 256) {
        const int tt = e / TC, cc = e % TC;
        const uint32_t t = t0 + tt, col = col0 + cc;
        As[tt][cc] = (t < L.r && col < a.n) ? __ldg(L.A + static_cast<size_t>(t) * a.n + col) : 0.f;
      }
      for (int e = tid; e < TR * KC; e += 256) {
        const int rr = e / KC, tt = e % KC;
        const uint32_t r = row0 + rr, t = t0 + tt;
        Bs[rr][tt] = (r < a.m && t < L.r) ? __ldg(L.B + static_cast<size_t>(r) * L.r + t) : 0.f;
      }
      __syncthreads();
      const uint32_t kmax = (L.r - t0) < KC ? (L.r - t0) : KC;
      for (uint32_t tt = 0; tt < kmax; ++tt) {
        const float4 av = *reinterpret_cast<const float4*>(&As[tt][tx * 4]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float bv = Bs[ty * 4 + i][tt];
          dl[i][0] = fmaf(bv, av.x, dl[i][0]);
          dl[i][1] = fmaf(bv, av.y, dl[i][1]);
          dl[i][2] = fmaf(bv, av.z, dl[i][2]);
          dl[i][3] = fmaf(bv, av.w, dl[i][3]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(L.s, dl[i][j], acc[i][j]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t r = row0 + ty * 4 + i;
    if (r < a.m && c < a.n)
      *reinterpret_cast<float4*>(a.S + static_cast<size_t>(r) * a.n + c) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
}

}  // namespace

cudaError_t launch_materialize(const MatArgs& a, cudaStream_t st) {
  if (a.m == 0 || a.n == 0) return cudaSuccess;
  dim3 grid((a.n + TC - 1) / TC, (a.m + TR - 1) / TR);
  k_materialize<<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace ovl
