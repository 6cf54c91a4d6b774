// K1: fused dual-path decode kernel for one tensor of the quantized base.
//
//   y[t] = deq(W_q) x[t] + sum_k s_k B_k (A_k x[t])      (t < T <= 8 per launch)
//
// Sources: "Deep Technical Design: Exact, Atomic, Reversible Specialist Overlays
// on Quantized Transformer Bases" §1 (Dual-Path Ephemeral-Accumulation: base and
// overlay evaluated as parallel streams), §5 (q8_0: 32 weights + f16 scale),
// §8 (decode GEMV is memory-bandwidth bound; fetch adapter rows while the base
// block is live); "We propose a content-addressed overlay system" report
// §"Native/WASM Kernel Implications" (direct low-rank addition: x A^T, then B).
//
// Design (GB300):
//  * Each CTA owns a contiguous row range of W.  Because the planes are
//    row-major, that range is one contiguous byte range of the qs plane and of
//    the d plane, streamed by one producer thread with 1-D bulk copies
//    (cp.async.bulk, TMA engine, L2 evict-first) into an NS-deep shared-memory
//    ring guarded by mbarriers.  No multicast.
//  * Every consumer lane owns fixed 32-weight column blocks for the whole
//    kernel.  The activation block is rewritten once per launch as an exact
//    integer: x_j = X_j * 2^-s_b with |X_j| < 2^22 split into three byte limbs
//    (h signed, m and l unsigned).  The base dot product of a block is then
//    exact integer arithmetic on the dp4a units (no per-weight conversion):
//    P = 65536 * sum(q h) + 256 * sum(q m) + sum(q l), and acc += d * 2^-s_b * P
//    in fp32.  q4_0 codes are used unsigned with the -8 offset folded into the
//    accumulator start (-8 * sum of limbs).
//  * The low-rank shrink v = A x is a side product: each CTA reduces one
//    contiguous chunk of the flattened [sum r_k][n] factor space and publishes
//    partial sums; after its rows are streamed the CTA waits (bounded) for all
//    partials, reduces them in a fixed order and adds s_k B_k v_k to its rows in
//    the epilogue.  Every reduction has a fixed order: results are bitwise
//    deterministic, and a zero B adds exactly zero.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "ovl_internal.h"
#include "ptx.cuh"

namespace ovl {
namespace {

constexpr int kRecBytes = 112;  // per (token, block) activation record: 7 x 16 B
constexpr int kMaxNS = 4;
constexpr uint32_t kRecBudget = 128 * 1024;
constexpr uint32_t kSmemBudget = 220 * 1024;

struct DualCfg {
  uint32_t nwc;          // consumer warps
  uint32_t bpl;          // column blocks per consumer lane
  uint32_t ns;           // pipeline depth
  uint32_t rowbytes;     // qs bytes per row
  uint32_t nb;           // 32-blocks per row
  uint32_t stage_q;      // qs bytes of a full stage
  uint32_t stage_bytes;  // stride between stages
  uint32_t rows_max;     // rows of the largest CTA slice
  uint32_t gs;           // CTAs that reduce a shrink chunk
  uint32_t off_rec, off_stage, off_red, off_v, off_tmp;
  uint32_t smem;
};

__device__ __forceinline__ void latch(uint32_t* status, uint32_t code) {
  atomicCAS(status, 0u, code);
}

__device__ __forceinline__ float load_x(const void* x, uint32_t xdt, size_t i) {
  if (xdt == OVL_BF16) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(x)[i]) << 16);
  }
  return static_cast<const float*>(x)[i];
}

// Activation record of one 32-block: limbs h|m|l (32 bytes each, in the order the
// weight words are consumed), then {2^-s as f32 bits, start_h, start_m, start_l}.
template <bool Q4>
__device__ __forceinline__ void prep_record(uint8_t* rec, const void* x, uint32_t xdt, size_t idx,
                                            uint32_t lane) {
  const float v = load_x(x, xdt, idx);
  const uint32_t mx = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
  int X = 0;
  float xs = 0.f;
  if (mx != 0u) {
    const int E = ilogbf(__uint_as_float(mx));
    const int s = 21 - E;                 // |X| <= 2^22
    X = __float2int_rn(ldexpf(v, s));
    xs = ldexpf(1.0f, -s);
  }
  // q4_0 word i of a block carries elements 8i..8i+7 as nibbles: the low nibbles
  // hold the even elements, the high nibbles the odd ones.
  const uint32_t p = Q4 ? ((lane >> 3) * 8 + (lane & 1) * 4 + ((lane & 7) >> 1)) : lane;
  const int h = X >> 16;
  const int mm = (X >> 8) & 0xFF;
  const int ll = X & 0xFF;
  rec[p] = static_cast<uint8_t>(h & 0xFF);
  rec[32 + p] = static_cast<uint8_t>(mm);
  rec[64 + p] = static_cast<uint8_t>(ll);
  uint32_t* meta = reinterpret_cast<uint32_t*>(rec + 96);
  if (Q4) {
    const int sh = __reduce_add_sync(0xffffffffu, h);
    const int sm = __reduce_add_sync(0xffffffffu, mm);
    const int sl = __reduce_add_sync(0xffffffffu, ll);
    if (lane == 0) {
      meta[1] = static_cast<uint32_t>(-8 * sh);
      meta[2] = static_cast<uint32_t>(-8 * sm);
      meta[3] = static_cast<uint32_t>(-8 * sl);
    }
  } else if (lane == 0) {
    meta[1] = meta[2] = meta[3] = 0u;
  }
  if (lane == 0) meta[0] = __float_as_uint(xs);
}

__device__ __forceinline__ float limb_combine(int sh, int sm, int sl) {
  return fmaf(__int2float_rn(sh), 65536.f, __int2float_rn(sm * 256 + sl));
}

__device__ __forceinline__ float dot_q8(const uint8_t* wp, const uint4 (&r)[7]) {
  const uint4 a = *reinterpret_cast<const uint4*>(wp);
  const uint4 b = *reinterpret_cast<const uint4*>(wp + 16);
  int sh = 0, sm = 0, sl = 0;
  sh = dp4a_ss(a.x, r[0].x, sh); sh = dp4a_ss(a.y, r[0].y, sh);
  sh = dp4a_ss(a.z, r[0].z, sh); sh = dp4a_ss(a.w, r[0].w, sh);
  sh = dp4a_ss(b.x, r[1].x, sh); sh = dp4a_ss(b.y, r[1].y, sh);
  sh = dp4a_ss(b.z, r[1].z, sh); sh = dp4a_ss(b.w, r[1].w, sh);
  sm = dp4a_su(a.x, r[2].x, sm); sm = dp4a_su(a.y, r[2].y, sm);
  sm = dp4a_su(a.z, r[2].z, sm); sm = dp4a_su(a.w, r[2].w, sm);
  sm = dp4a_su(b.x, r[3].x, sm); sm = dp4a_su(b.y, r[3].y, sm);
  sm = dp4a_su(b.z, r[3].z, sm); sm = dp4a_su(b.w, r[3].w, sm);
  sl = dp4a_su(a.x, r[4].x, sl); sl = dp4a_su(a.y, r[4].y, sl);
  sl = dp4a_su(a.z, r[4].z, sl); sl = dp4a_su(a.w, r[4].w, sl);
  sl = dp4a_su(b.x, r[5].x, sl); sl = dp4a_su(b.y, r[5].y, sl);
  sl = dp4a_su(b.z, r[5].z, sl); sl = dp4a_su(b.w, r[5].w, sl);
  return limb_combine(sh, sm, sl);
}

__device__ __forceinline__ float dot_q4(const uint8_t* wp, const uint4 (&r)[7]) {
  const uint4 w = *reinterpret_cast<const uint4*>(wp);
  const uint32_t m4 = 0x0F0F0F0Fu;
  const uint32_t l0 = w.x & m4, h0 = (w.x >> 4) & m4;
  const uint32_t l1 = w.y & m4, h1 = (w.y >> 4) & m4;
  const uint32_t l2 = w.z & m4, h2 = (w.z >> 4) & m4;
  const uint32_t l3 = w.w & m4, h3 = (w.w >> 4) & m4;
  int sh = static_cast<int>(r[6].y);
  uint32_t sm = r[6].z, sl = r[6].w;
  sh = dp4a_us(l0, r[0].x, sh); sh = dp4a_us(h0, r[0].y, sh);
  sh = dp4a_us(l1, r[0].z, sh); sh = dp4a_us(h1, r[0].w, sh);
  sh = dp4a_us(l2, r[1].x, sh); sh = dp4a_us(h2, r[1].y, sh);
  sh = dp4a_us(l3, r[1].z, sh); sh = dp4a_us(h3, r[1].w, sh);
  sm = dp4a_uu(l0, r[2].x, sm); sm = dp4a_uu(h0, r[2].y, sm);
  sm = dp4a_uu(l1, r[2].z, sm); sm = dp4a_uu(h1, r[2].w, sm);
  sm = dp4a_uu(l2, r[3].x, sm); sm = dp4a_uu(h2, r[3].y, sm);
  sm = dp4a_uu(l3, r[3].z, sm); sm = dp4a_uu(h3, r[3].w, sm);
  sl = dp4a_uu(l0, r[4].x, sl); sl = dp4a_uu(h0, r[4].y, sl);
  sl = dp4a_uu(l1, r[4].z, sl); sl = dp4a_uu(h1, r[4].w, sl);
  sl = dp4a_uu(l2, r[5].x, sl); sl = dp4a_uu(h2, r[5].y, sl);
  sl = dp4a_uu(l3, r[5].z, sl); sl = dp4a_uu(h3, r[5].w, sl);
  return limb_combine(sh, static_cast<int>(sm), static_cast<int>(sl));
}

// Sum over the 32 lanes of v[lane >> (5 - log2 N)] for all N values at once
// (N - 1 + 5 - log2 N shuffles instead of 5 N).  Fixed order: deterministic.
template <int N>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], uint32_t lane) {
  int bit = 16;
#pragma unroll
  for (int half = N / 2; half >= 1; half /= 2) {
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = upper ? v[j] : v[j + half];
      const float keep = upper ? v[j + half] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
    bit >>= 1;
  }
  float r = v[0];
  for (; bit >= 1; bit >>= 1) r += __shfl_xor_sync(0xffffffffu, r, bit);
  return r;
}

template <int N>
struct Log2 { static constexpr int v = 1 + Log2<N / 2>::v; };
template <>
struct Log2<1> { static constexpr int v = 0; };

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Partial shrink sums of this CTA's chunk of the flattened [rtot][n] factor
// space: partial[(t * rtot + rho) * gs + cta] = sum_{j in chunk, row rho} A[rho][j] x[t][j].
template <int TT>
__device__ void shrink_chunk(const DualArgs& a, const DualCfg& c, uint32_t cta, float* tmp,
                             uint32_t warp, uint32_t lane) {
  if (cta >= c.gs) return;
  const uint32_t nthr = c.nwc * 32;
  const uint64_t total = static_cast<uint64_t>(a.rtot) * a.n;
  const uint64_t lo = cta * total / c.gs, hi = (cta + 1) * total / c.gs;
  const uint32_t rho_a = static_cast<uint32_t>(lo / a.n), rho_b = static_cast<uint32_t>((hi - 1) / a.n);
  for (uint32_t rho = rho_a; rho <= rho_b; ++rho) {
    uint32_t k = 0, rbase = 0;
    while (rho >= rbase + a.lora[k].r) { rbase += a.lora[k].r; ++k; }
    const float* Arow = a.lora[k].A + static_cast<size_t>(rho - rbase) * a.n;
    const uint64_t rs = static_cast<uint64_t>(rho) * a.n;
    const uint32_t j0 = static_cast<uint32_t>(max(lo, rs) - rs);
    const uint32_t j1 = static_cast<uint32_t>(min(hi, rs + a.n) - rs);
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.f;
    for (uint32_t j = j0 + threadIdx.x; j < j1; j += nthr) {
      const float av = __ldg(Arow + j);
#pragma unroll
      for (int t = 0; t < TT; ++t)
        if (t < static_cast<int>(a.T)) acc[t] = fmaf(av, load_x(a.x, a.xdt, static_cast<size_t>(t) * a.n + j), acc[t]);
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const float s = warp_sum(acc[t]);
      if (lane == 0) tmp[warp * TT + t] = s;
    }
    named_bar(1, nthr);
    if (threadIdx.x < a.T) {
      float s = 0.f;
      for (uint32_t w = 0; w < c.nwc; ++w) s += tmp[w * TT + threadIdx.x];
      a.ws.partial[(static_cast<size_t>(threadIdx.x) * a.rtot + rho) * c.gs + cta] = s;
    }
    named_bar(1, nthr);
  }
}

template <int QUANT, int TT, int RG>
__global__ void __launch_bounds__(288, 2) k_dualpath(const DualArgs a, const DualCfg c) {
  constexpr bool Q4 = QUANT == OVL_Q4_0;
  constexpr int N = TT * RG;
  constexpr int LN = Log2<N>::v;
  constexpr uint32_t kBlockBytes = Q4 ? 16 : 32;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm);
  uint64_t* empty = full + kMaxNS;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + 64);
  uint8_t* rec = sm + c.off_rec;
  uint8_t* stages = sm + c.off_stage;
  float* red = reinterpret_cast<float*>(sm + c.off_red);
  float* vsm = reinterpret_cast<float*>(sm + c.off_v);
  float* tmp = reinterpret_cast<float*>(sm + c.off_tmp);

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t G = gridDim.x, cta = blockIdx.x;
  const uint32_t row0 = static_cast<uint32_t>((static_cast<uint64_t>(cta) * a.m) / G);
  const uint32_t row1 = static_cast<uint32_t>((static_cast<uint64_t>(cta + 1) * a.m) / G);
  const uint32_t nrows = row1 - row0;
  const uint32_t nst = (nrows + RG - 1) / RG;
  const uint32_t nthr = c.nwc * 32;

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < c.ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], c.nwc);
    }
    *abort_flag = 0u;
    mbar_fence_init();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == c.nwc) {
    // ---------------- producer: stream this CTA's rows (base bytes are immutable,
    // so this may start before the preceding grid has finished).
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      uint32_t issued = 0;
      for (uint32_t s = 0; s < nst; ++s) {
        const uint32_t slot = s % c.ns;
        if (s >= c.ns && !mbar_wait_bounded(&empty[slot], ((s / c.ns) - 1) & 1)) {
          latch(a.ws.status, kDevTimeoutEmpty);
          *abort_flag = 1u;
          break;
        }
        if (*abort_flag) break;
        const uint32_t r0 = row0 + s * RG;
        const uint32_t rows = min(static_cast<uint32_t>(RG), row1 - r0);
        const size_t dstart = static_cast<size_t>(r0) * c.nb * 2;
        const size_t d0 = dstart & ~static_cast<size_t>(15);
        const size_t d1 = (dstart + static_cast<size_t>(rows) * c.nb * 2 + 15) & ~static_cast<size_t>(15);
        uint8_t* dst = stages + static_cast<size_t>(slot) * c.stage_bytes;
        const uint32_t bq = rows * c.rowbytes;
        mbar_arrive_expect_tx(&full[slot], bq + static_cast<uint32_t>(d1 - d0));
        bulk_g2s(dst, a.qs + static_cast<size_t>(r0) * c.rowbytes, bq, &full[slot], pol);
        bulk_g2s(dst + c.stage_q, a.dpl + d0, static_cast<uint32_t>(d1 - d0), &full[slot], pol);
        ++issued;
      }
      // Do not leave while copies into this CTA's shared memory may be in flight.
      const uint32_t first = issued > c.ns ? issued - c.ns : 0;
      for (uint32_t s = first; s < issued; ++s) mbar_wait_bounded(&full[s % c.ns], (s / c.ns) & 1);
    }
    return;
  }

  // ---------------- consumers
  griddep_wait();  // x, y and the workspace may be touched by the preceding grid

  // 1. activation records for the tokens of this launch
  for (uint32_t rr = warp; rr < a.T * c.nb; rr += c.nwc) {
    const uint32_t t = rr / c.nb, b = rr - t * c.nb;
    prep_record<Q4>(rec + static_cast<size_t>(rr) * kRecBytes, a.x, a.xdt,
                    static_cast<size_t>(t) * a.n + b * 32 + lane, lane);
  }
  // 2. low-rank shrink partials, published with one arrival per CTA
  if (a.nl) shrink_chunk<TT>(a, c, cta, tmp, warp, lane);
  named_bar(1, nthr);
  if (a.nl && threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&a.ws.counter[0], 1ull);
  }

  // 3. stream the base rows
  bool ok = true;
  for (uint32_t s = 0; s < nst; ++s) {
    const uint32_t slot = s % c.ns;
    // warp-uniform decision: the shuffles below need every lane
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (s / c.ns) & 1))) {
      latch(a.ws.status, kDevTimeoutFull);
      *abort_flag = 1u;
      ok = false;
      break;
    }
    const uint8_t* sq = stages + static_cast<size_t>(slot) * c.stage_bytes;
    const uint32_t r0 = row0 + s * RG;
    const size_t dstart = static_cast<size_t>(r0) * c.nb * 2;
    const __half* sd = reinterpret_cast<const __half*>(sq + c.stage_q + (dstart & 15));
    float acc[N];
#pragma unroll
    for (int i = 0; i < N; ++i) acc[i] = 0.f;
    for (uint32_t k = 0; k < c.bpl; ++k) {
      const uint32_t b = threadIdx.x + k * nthr;
      if (b < c.nb) {
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (t < static_cast<int>(a.T)) {
            const uint4* rp = reinterpret_cast<const uint4*>(rec + static_cast<size_t>(t * c.nb + b) * kRecBytes);
            uint4 r[7];
#pragma unroll
            for (int i = 0; i < 7; ++i) r[i] = rp[i];
            const float xs = __uint_as_float(r[6].x);
#pragma unroll
            for (int rr = 0; rr < RG; ++rr) {
              const uint8_t* wp = sq + rr * c.rowbytes + b * kBlockBytes;
              const float P = Q4 ? dot_q4(wp, r) : dot_q8(wp, r);
              const float d = __half2float(sd[rr * c.nb + b]);
              acc[t * RG + rr] = fmaf(d * xs, P, acc[t * RG + rr]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    const float tot = transpose_reduce<N>(acc, lane);
    if ((lane & ((32 >> LN) - 1)) == 0) {
      const uint32_t idx = lane >> (5 - LN);
      const uint32_t t = idx / RG, rr = idx - t * RG;
      const uint32_t lr = s * RG + rr;
      if (lr < nrows && t < a.T) red[(warp * TT + t) * c.rows_max + lr] = tot;
    }
  }
  named_bar(1, nthr);

  // 4. low-rank vector v = A x (sum of the published partials, fixed order)
  if (a.nl) {
    if (threadIdx.x == 0) {
      uint32_t it = 0;
      while (ld_acquire_u64(&a.ws.counter[0]) < G) {
        if (++it > (1u << 22)) {
          latch(a.ws.status, kDevTimeoutShrink);
          break;
        }
        __nanosleep(64);
      }
    }
    named_bar(1, nthr);
    const uint64_t total = static_cast<uint64_t>(a.rtot) * a.n;
    for (uint32_t i = threadIdx.x; i < a.T * a.rtot; i += nthr) {
      const uint32_t t = i / a.rtot, rho = i - t * a.rtot;
      uint64_t cf = ((static_cast<uint64_t>(rho) * a.n + 1) * c.gs + total - 1) / total;
      uint64_t cl = ((static_cast<uint64_t>(rho + 1) * a.n) * c.gs + total - 1) / total;
      cf = cf ? cf - 1 : 0;
      cl = cl ? cl - 1 : 0;
      if (cl > c.gs - 1) cl = c.gs - 1;
      const float* p = a.ws.partial + (static_cast<size_t>(t) * a.rtot + rho) * c.gs;
      float s = 0.f;
      for (uint64_t q = cf; q <= cl; ++q) s += __ldcg(p + q);
      vsm[t * a.rtot + rho] = s;
    }
    named_bar(1, nthr);
    if (threadIdx.x == 0) {
      // Last CTA out resets the arrival counters for the next launch.
      const unsigned long long old = atomicAdd(&a.ws.counter[1], 1ull);
      if (old == G - 1) {
        atomicExch(&a.ws.counter[0], 0ull);
        atomicExch(&a.ws.counter[1], 0ull);
      }
    }
  }

  // 5. epilogue: y = base + sum_k s_k (B_k v_k), one warp per row
  if (!ok) return;
  for (uint32_t lr = warp; lr < nrows; lr += c.nwc) {
    const uint32_t row = row0 + lr;
    float yv[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      float s = 0.f;
      if (t < static_cast<int>(a.T))
        for (uint32_t w = 0; w < c.nwc; ++w) s += red[(w * TT + t) * c.rows_max + lr];
      yv[t] = s;
    }
    uint32_t rbase = 0;
    for (uint32_t k = 0; k < a.nl; ++k) {
      const uint32_t r = a.lora[k].r;
      const float* Brow = a.lora[k].B + static_cast<size_t>(row) * r;
      float part[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) part[t] = 0.f;
      for (uint32_t tau = lane; tau < r; tau += 32) {
        const float bv = __ldg(Brow + tau);
#pragma unroll
        for (int t = 0; t < TT; ++t)
          if (t < static_cast<int>(a.T)) part[t] = fmaf(bv, vsm[t * a.rtot + rbase + tau], part[t]);
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) yv[t] = fmaf(a.lora[k].s, warp_sum(part[t]), yv[t]);
      rbase += r;
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < TT; ++t)
        if (t < static_cast<int>(a.T)) a.y[static_cast<size_t>(t) * a.m + row] = yv[t];
    }
  }
}

using KernelFn = void (*)(const DualArgs, const DualCfg);

KernelFn pick(uint32_t quant, int tt, int rg) {
#define OVL_K(Q, T_, R_) \
  if (quant == Q && tt == T_ && rg == R_) return k_dualpath<Q, T_, R_>;
  OVL_K(OVL_Q8_0, 1, 2) OVL_K(OVL_Q8_0, 1, 8) OVL_K(OVL_Q8_0, 2, 2) OVL_K(OVL_Q8_0, 4, 2)
  OVL_K(OVL_Q8_0, 8, 2) OVL_K(OVL_Q4_0, 1, 2) OVL_K(OVL_Q4_0, 1, 8) OVL_K(OVL_Q4_0, 2, 2)
  OVL_K(OVL_Q4_0, 4, 2) OVL_K(OVL_Q4_0, 8, 2)
#undef OVL_K
  return nullptr;
}

uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

int device_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// Shared-memory plan for one launch; returns false if it cannot fit.
bool plan(DualCfg& c, const DualArgs& a, int tt, int rg, uint32_t G) {
  c.rows_max = (a.m + G - 1) / G;
  uint32_t off = 128;
  c.off_rec = off;
  off = round_up(off + tt * c.nb * kRecBytes, 128);
  c.off_red = off;
  off = round_up(off + c.nwc * tt * c.rows_max * 4, 128);
  c.off_v = off;
  off = round_up(off + tt * a.rtot * 4 + 4, 128);
  c.off_tmp = off;
  off = round_up(off + c.nwc * tt * 4, 1024);
  c.stage_q = rg * c.rowbytes;
  c.stage_bytes = round_up(c.stage_q + round_up(rg * c.nb * 2, 16) + 32, 128);
  c.off_stage = off;
  for (uint32_t ns = kMaxNS; ns >= 2; --ns) {
    if (off + ns * c.stage_bytes <= kSmemBudget) {
      c.ns = ns;
      c.smem = off + ns * c.stage_bytes;
      return true;
    }
  }
  return false;
}

}  // namespace

cudaError_t launch_dualpath(const DualArgs& a0, cudaStream_t st) {
  if (a0.T == 0 || a0.m == 0) return cudaSuccess;
  static int nsm = device_sms();
  DualCfg c{};
  c.nb = a0.n / kQK;
  c.rowbytes = a0.quant == OVL_Q8_0 ? a0.n : a0.n / 2;
  // consumer warps: fewest idle lanes, then fewest blocks per lane
  uint32_t best_w = 1, best_b = 0, best_waste = ~0u;
  for (uint32_t w = 1; w <= 8; ++w) {
    const uint32_t b = (c.nb + 32 * w - 1) / (32 * w);
    const uint32_t waste = b * 32 * w - c.nb;
    if (b < best_b || best_b == 0 || (b == best_b && waste < best_waste)) {
      best_w = w; best_b = b; best_waste = waste;
    }
  }
  c.nwc = best_w;
  c.bpl = best_b;
  // token tile
  int tt = 1;
  const uint32_t Tneed = a0.T < 8 ? a0.T : 8;
  while (tt < static_cast<int>(Tneed)) tt *= 2;
  while (tt > 1 && tt * c.nb * kRecBytes > kRecBudget) tt /= 2;
  const int rg = (tt == 1 && c.rowbytes * 8 <= 40960) ? 8 : 2;
  KernelFn fn = pick(a0.quant, tt, rg);
  if (!fn) return cudaErrorInvalidValue;
  const uint32_t threads = (c.nwc + 1) * 32;
  // grid: co-resident CTAs, at least two rows each
  uint32_t G = static_cast<uint32_t>(nsm) * 2;
  G = std::min<uint32_t>(G, std::max<uint32_t>(1, a0.m / 2));
  int occ = 0;
  for (int iter = 0; iter < 4; ++iter) {
    if (!plan(c, a0, tt, rg, G)) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, c.smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, c.smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const uint32_t cap = static_cast<uint32_t>(nsm) * static_cast<uint32_t>(occ);
    if (G <= cap) break;
    G = cap;
  }
  if (!plan(c, a0, tt, rg, G)) return cudaErrorInvalidConfiguration;
  c.gs = a0.nl ? static_cast<uint32_t>(std::min<uint64_t>(G, static_cast<uint64_t>(a0.rtot) * a0.n)) : 0;
  if (a0.nl && static_cast<size_t>(tt) * a0.rtot * c.gs > a0.ws.partial_floats) return cudaErrorInvalidValue;

  const size_t esz = a0.xdt == OVL_BF16 ? 2 : 4;
  for (uint32_t t0 = 0; t0 < a0.T; t0 += tt) {
    DualArgs a = a0;
    a.T = std::min<uint32_t>(tt, a0.T - t0);
    a.x = static_cast<const uint8_t*>(a0.x) + static_cast<size_t>(t0) * a0.n * esz;
    a.y = a0.y + static_cast<size_t>(t0) * a0.m;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, a, c);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ovl
