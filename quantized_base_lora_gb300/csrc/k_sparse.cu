// K7: sparse overlay terms.  A sparse overlay stores only the non-zero
// elements of a weight update, as strictly increasing 32-bit indices and f16
// values, and adds them at their positions at use time while the base stays
// unchanged ("We propose a content-addressed overlay system" report,
// §"Runtime Strategy Comparison Matrix", Sparse Overlay; "Deep Technical
// Design: Exact, Atomic, Reversible Specialist Overlays on Quantized
// Transformer Bases" §7 Sparse Overlay Bytes and §11 Deep Compatibility Checks).
//
// Dual path: k_sparse_apply adds s * (dW x) to the y the dense kernel wrote.
// One launch covers the tensors of one forward call (up to four that share x).
// A group of 4 to 32 lanes per output row (sized from the average pairs per
// row); the row's pairs come from the row offsets built at staging.  The launch
// is a programmatic dependent of the dense kernel: each group loads its row's
// first pairs (immutable) into registers, lane l of the group taking pairs l,
// l + group, ..., before the grid dependency resolves; only the gather of x and
// the update of y wait for it.  Four tokens per pass reuse the registers; the
// group folds its partial sums in a fixed butterfly order (deterministic).
//
// JIT path: k_sparse_scatter adds s * val into the fp32 scratch at each index.
// The indices of one term are distinct, so no two threads of a launch write
// the same element; terms run as successive launches in composition order.
#include <cuda_fp16.h>

#include "ovl_internal.h"
#include "ptx.cuh"

namespace ovl {
namespace {

constexpr int kThreads = 256;
constexpr int kTokPass = 4;
constexpr int kPairRegs = 8;       // pairs per lane held across the dependency wait

__device__ __forceinline__ float x_at(const void* x, uint32_t xdt, size_t i) {
  if (xdt == OVL_BF16)
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(x)[i]) << 16);
  return static_cast<const float*>(x)[i];
}

// LPR lanes (an aligned group within a warp) per output row.
template <int LPR>
__global__ void __launch_bounds__(kThreads, 4) k_sparse_apply(const SparseApply a) {
  griddep_launch_dependents();
  const uint32_t sub = threadIdx.x & (LPR - 1);
  const uint32_t gr = (blockIdx.x * kThreads + threadIdx.x) / LPR;   // global row of the launch
  // Every lane of a warp stays to the end (the folds below use the full warp
  // mask); rows past the end do no work.
  const bool live = gr < a.mtot;
  uint32_t si = 0;
  while (live && si + 1 < a.nseg && gr >= a.seg[si + 1].row0) ++si;
  const SparseSeg& sg = a.seg[si];
  const uint32_t row = live ? gr - sg.row0 : 0;
  const uint32_t base = row * a.n;   // < 2^32: checked at staging
  const uint32_t k0 = live ? sg.k0 : 0, k1 = live ? sg.k1 : 0;
  // first term: row bounds and its first LPR * kPairRegs pairs, before the wait
  uint32_t b0 = 0, e0 = 0;
  uint32_t col[kPairRegs];
  float val[kPairRegs];
#pragma unroll
  for (int j = 0; j < kPairRegs; ++j) {
    col[j] = 0;
    val[j] = 0.f;
  }
  if (k1 > k0) {
    const SparseRef& R = a.t[k0];
    b0 = R.rp[row];
    e0 = R.rp[row + 1];
#pragma unroll
    for (int j = 0; j < kPairRegs; ++j) {
      const uint32_t p = b0 + sub + LPR * j;
      if (p < e0) {
        col[j] = R.idx[p] - base;
        val[j] = __half2float(__ushort_as_half(R.val[p]));
      }
    }
  }
  griddep_wait();   // y written by the dense kernel, x by its producer
  const uint32_t T = live ? a.T : 0;
  // warp-uniform pass count: the longest of the rows in this warp
  const uint32_t Tw = __reduce_max_sync(0xffffffffu, T);
  for (uint32_t t0 = 0; t0 < Tw; t0 += kTokPass) {
    const uint32_t nt = t0 < T ? min(static_cast<uint32_t>(kTokPass), T - t0) : 0u;
    float yv[kTokPass];
#pragma unroll
    for (int u = 0; u < kTokPass; ++u)
      yv[u] = (static_cast<uint32_t>(u) < nt) ? sg.y[static_cast<size_t>(t0 + u) * sg.m + row] : 0.f;
    const uint32_t kw = __reduce_max_sync(0xffffffffu, k1 - k0);   // terms, warp-uniform bound
    for (uint32_t kk = 0; kk < kw; ++kk) {
      const uint32_t k = k0 + kk;
      const bool has = k < k1;
      float acc[kTokPass];
#pragma unroll
      for (int u = 0; u < kTokPass; ++u) acc[u] = 0.f;
      uint32_t e = 0, p0 = 0;
      if (has && kk == 0) {
#pragma unroll
        for (int j = 0; j < kPairRegs; ++j)
          if (b0 + sub + LPR * j < e0)
#pragma unroll
            for (int u = 0; u < kTokPass; ++u)
              if (static_cast<uint32_t>(u) < nt)
                acc[u] = fmaf(val[j], x_at(a.x, a.xdt, static_cast<size_t>(t0 + u) * a.n + col[j]), acc[u]);
        e = e0;
        p0 = b0 + LPR * kPairRegs;
      } else if (has) {
        p0 = a.t[k].rp[row];
        e = a.t[k].rp[row + 1];
      }
      if (has) {
        const SparseRef& R = a.t[k];
        for (uint32_t p = p0 + sub; p < e; p += LPR) {
          const uint32_t c = R.idx[p] - base;
          const float v = __half2float(__ushort_as_half(R.val[p]));
#pragma unroll
          for (int u = 0; u < kTokPass; ++u)
            if (static_cast<uint32_t>(u) < nt)
              acc[u] = fmaf(v, x_at(a.x, a.xdt, static_cast<size_t>(t0 + u) * a.n + c), acc[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kTokPass; ++u) {
#pragma unroll
        for (int o = LPR / 2; o >= 1; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
        if (has) yv[u] = fmaf(a.t[k].s, acc[u], yv[u]);
      }
    }
    if (sub == 0)
#pragma unroll
      for (int u = 0; u < kTokPass; ++u)
        if (static_cast<uint32_t>(u) < nt) sg.y[static_cast<size_t>(t0 + u) * sg.m + row] = yv[u];
  }
}

__global__ void __launch_bounds__(256) k_sparse_scatter(float* S, const SparseRef t) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t p = blockIdx.x * blockDim.x + threadIdx.x; p < t.nnz; p += stride) {
    float* dst = S + t.idx[p];
    *dst = fmaf(t.s, __half2float(__ushort_as_half(t.val[p])), *dst);
  }
}

}  // namespace

cudaError_t launch_sparse_apply(const SparseApply& a, cudaStream_t st) {
  if (a.mtot == 0 || a.T == 0 || a.nt == 0) return cudaSuccess;
  // lanes per row: enough for the average row of the first terms to sit in
  // registers with a quarter to spare, between 4 and 32
  uint64_t pairs = 0;
  for (uint32_t i = 0; i < a.nseg; ++i)
    if (a.seg[i].k1 > a.seg[i].k0) pairs += a.t[a.seg[i].k0].nnz;
  const uint64_t want = (pairs * 5 / 4 + static_cast<uint64_t>(a.mtot) * kPairRegs - 1) /
                        (static_cast<uint64_t>(a.mtot) * kPairRegs);
  int lpr = 4;
  while (lpr < 32 && static_cast<uint64_t>(lpr) < want) lpr *= 2;
  void (*fn)(const SparseApply) = lpr == 4 ? k_sparse_apply<4> : lpr == 8 ? k_sparse_apply<8>
                                  : lpr == 16 ? k_sparse_apply<16> : k_sparse_apply<32>;
  const uint64_t threads = static_cast<uint64_t>(a.mtot) * lpr;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<uint32_t>((threads + kThreads - 1) / kThreads));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

cudaError_t launch_sparse_scatter(float* S, const SparseRef& t, cudaStream_t st) {
  if (t.nnz == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const uint32_t want = (t.nnz + 255) / 256;
  const uint32_t grid = want < static_cast<uint32_t>(8 * (sms > 0 ? sms : 1)) ? want : 8u * (sms > 0 ? sms : 1);
  k_sparse_scatter<<<grid, 256, 0, st>>>(S, t);
  return cudaGetLastError();
}

}  // namespace ovl
