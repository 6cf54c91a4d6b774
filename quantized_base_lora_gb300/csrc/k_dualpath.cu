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
//    kernel.  The activation block is rewritten once per launch on a fixed-point
//    grid: x_j ~ X_j * 2^-s_b with |X_j| <= 2^22 (22 bits below the block's
//    largest element) split into three byte limbs (h signed, m and l unsigned).
//    The base dot product of a block is then exact integer arithmetic on the
//    dp4a units (no per-weight conversion): P = 65536 * sum(q h) + 256 *
//    sum(q m) + sum(q l), and acc += d * 2^-s_b * P in fp32.  q4_0 codes are
//    used unsigned with the -8 offset folded into the accumulator start (-8 *
//    sum of limbs).  The grid represents an element exactly when it lies
//    within 2^14 of the block maximum (bf16 input) and to 2^-12 of itself when
//    it lies within 2^10 (fp32 input); a block with any smaller nonzero element
//    is marked when its record is built, and the epilogue adds its exact fp32
//    residual sum_j w_j (x_j - X_j 2^-s), so every element keeps 12 bits
//    relative to itself whatever the block's dynamic range.
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
#ifndef OVL_K1_MAX_NS
#define OVL_K1_MAX_NS 8
#endif
#ifndef OVL_K1_SOFT_BYTES
#define OVL_K1_SOFT_BYTES (150 * 1024)
#endif
#ifndef OVL_K1_STAGE_BYTES
#define OVL_K1_STAGE_BYTES 16384
#endif
#ifndef OVL_K1_PDL
#define OVL_K1_PDL 1
#endif
#ifndef OVL_K1_MAX_GROUPS
#define OVL_K1_MAX_GROUPS 4
#endif
constexpr int kMaxNS = OVL_K1_MAX_NS;
constexpr uint32_t kPreDepStages = 2;     // ring stages copied to shared memory before the grid dependency
constexpr int kMaxThreads = 18 * 32;       // up to 16 consumer warps + producer + helper

// One CTA per SM: its ring (up to 150 KB of shared memory) is as deep as the
// SM's memory latency needs, and registers are not capped for a second CTA.
// Measured on the 8B-shape decode step, one deep ring per SM beat two
// co-resident CTAs of consecutive launches with half the ring each (the next
// launch's CTA still becomes resident on each SM as soon as this grid's CTA
// there exits, and streams its ring while the rest of the grid drains).
// Up to 16 column warps cover a row of up to 16K weights with one 32-block
// per lane, so single-token launches keep one activation record per lane in
// registers (a second register record made the two-row variants spill).
template <int TT, int RG>
struct K1Shape {
  static constexpr int threads = kMaxThreads;
  static constexpr int min_blocks = 1;
  static constexpr int reg_records = 1;
};
constexpr uint32_t reg_records_of(int, int) { return 1u; }
constexpr uint32_t kRecBudget = 128 * 1024;
constexpr uint32_t kSmemBudget = 220 * 1024;

struct DualCfg {
  uint32_t nwc;          // column warps per consumer group
  uint32_t ng;           // consumer groups (each consumes every ng-th stage)
  uint32_t bpl;          // column blocks per consumer lane
  uint32_t ns;           // pipeline depth
  uint32_t rowbytes;     // qs bytes per row
  uint32_t nb;           // 32-blocks per row
  uint32_t stage_q;      // qs bytes of a full stage
  uint32_t stage_bytes;  // stride between stages
  uint32_t rows_max;     // rows of the largest CTA slice
  uint32_t gs;           // CTAs that reduce a shrink chunk
  uint32_t off_rec, off_stage, off_red, off_v, off_ep;
  uint32_t off_x, off_a, off_xw;  // staged activations, shrink chunk of A, x window
  uint32_t stage_x;              // 0: x read from global; 4 or 16: cp.async granule
  uint32_t xvec;                 // 1: x (staged or global) allows 16-byte vector loads
  uint32_t stage_a;              // 1: the shrink chunk of A is staged in shared memory
  uint32_t xwin;                 // >0: the helper stages the x window of its chunk (capacity, elements)
  uint32_t shrink_vec;           // 1: A chunk and x window share one index, 16-byte vector reads
  uint32_t b_ring;               // 1: B rows arrive as one ring stage after the last base stage
  uint32_t b_areg;               // 1: the helper copies B rows into the A/x-window area after its shrink
  uint32_t div32;                // 1: rtot * n * gs < 2^32, chunk arithmetic fits 32 bits
  uint32_t smem;
  uint32_t off_mk;               // marked-block map: 1 + TT * map_words(nb) words
  uint32_t xfull;                // 1: the helper stages all of x (single token) for a chunk read with 16-byte loads
  uint32_t shrink_only;          // 1 (instances that read v): this launch only computes v, one CTA per factor row
};

// Words per token of the marked-block map.
__host__ __device__ __forceinline__ uint32_t map_words(uint32_t nb) { return (nb + 31) / 32; }

__device__ __forceinline__ void latch(uint32_t* status, uint32_t code) {
  atomicCAS(status, 0u, code);
}

__device__ __forceinline__ float load_x(const void* x, uint32_t xdt, size_t i) {
  if (xdt == OVL_BF16) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(x)[i]) << 16);
  }
  return static_cast<const float*>(x)[i];
}

// Activation records.  Record (t, b) describes the 32-block b of token t as
// an integer vector X with x_j ~ X_j * 2^-s (|X_j| <= 2^22), split in three
// byte limbs X = 65536 h + 256 m + l with h signed (byte 2 of X) and m, l
// unsigned (bytes 1 and 0): words 0-7 = h, 8-15 = m, 16-23 = l, then
// {2^-s as f32 bits, start_h, start_m, start_l}.  Limb word k holds the four
// elements that weight word k consumes: elements 4k..4k+3 for q8_0; for q4_0
// word 2g carries the low nibbles (elements 8g, 8g+2, 8g+4, 8g+6) and word
// 2g+1 the high nibbles (8g+1, ...).  The q4_0 starts are -8 * sum of the limbs,
// which folds the code offset into the integer accumulators.
//
// Precision.  s = 21 - E with 2^E <= max|x| < 2^(E+1), so an element is
// rounded to the nearest multiple of 2^(E-21): the error is at most 2^(E-22).
// A bf16 element (8 significant bits) at or above 2^(E-14) lies on the grid
// and is exact; an fp32 element at or above 2^(E-10) keeps a rounding error of
// at most 2^-12 of itself.  A block holding a smaller nonzero element (or a
// non-finite one, or a largest magnitude below 2^-104, where the grid would
// leave the normal range) is marked: its bit is set in the CTA's marked-block
// map (word 0: any block marked; then one row of words per token) and nothing
// else changes on the integer path.  The epilogue adds, in plain fp32, the
// marked blocks' residual products sum_j w_j (x_j - X_j 2^-s) (block_residual),
// re-reading only their weights.  The residual of each element is exact in
// fp32 and no larger than the element, so the sum of the two parts keeps each
// element to fp32 precision without cancellation against the integer part.
// Typical activations mark no block, and the hot loop carries no branch for it.
struct BlockScale {
  float sc;   // 2^s (0 when the block is below 2^-104 or all zero)
  float xs;   // 2^-s
};
__device__ __forceinline__ BlockScale block_scale(uint32_t mx) {
  const int E = static_cast<int>(mx >> 23) - 127;   // mx >= 2^-104 is normal
  const int s = 21 - E;
  if (mx < 0x0B800000u) return BlockScale{0.f, 0.f};  // all zero, or marked below
  return BlockScale{__uint_as_float(static_cast<uint32_t>(s + 127) << 23),
                    __uint_as_float(static_cast<uint32_t>(127 - s) << 23)};
}

// Smallest element magnitude (as fp32 bits) that the grid of a block with
// largest magnitude mx carries to 2^-12 of itself: 2^(E-14) for bf16 input,
// 2^(E-10) for fp32 input.
__device__ __forceinline__ uint32_t grid_floor_bits(uint32_t mx, uint32_t xdt) {
  return (mx & 0x7F800000u) - ((xdt == OVL_BF16 ? 14u : 10u) << 23);
}

// True when the block must take the fp32 route: mx = largest magnitude bits,
// mn1 = (smallest nonzero magnitude bits) - 1 (0xFFFFFFFF if none).
__device__ __forceinline__ bool block_marked(uint32_t mx, uint32_t mn1, uint32_t xdt) {
  if (mx == 0) return false;
  if (mx >= 0x7F800000u || mx < 0x0B800000u) return true;   // Inf/NaN, or below 2^-104
  return mn1 + 1u < grid_floor_bits(mx, xdt);
}

// Record a marked block (t, b) in the CTA's map.
__device__ __forceinline__ void mark_block(uint32_t* mk, uint32_t mkw, uint32_t t, uint32_t b) {
  atomicOr(mk, 1u);
  atomicOr(mk + 1 + t * mkw + (b >> 5), 1u << (b & 31));
}

// Exact round-to-nearest-even of v * 2^s to an integer, |result| <= 2^22:
// adding 1.5 * 2^23 leaves the integer in the low mantissa bits.
__device__ __forceinline__ int round_scaled(float v, float sc) {
  return __float_as_int(fmaf(v, sc, 12582912.0f)) - 0x4B400000;
}

// Limb words of four rounded integers: h (byte 2), m (byte 1), l (byte 0).
__device__ __forceinline__ void limb_words(const int (&X)[4], uint32_t& hw, uint32_t& mw, uint32_t& lw) {
  const uint32_t x0 = static_cast<uint32_t>(X[0]), x1 = static_cast<uint32_t>(X[1]);
  const uint32_t x2 = static_cast<uint32_t>(X[2]), x3 = static_cast<uint32_t>(X[3]);
  hw = __byte_perm(__byte_perm(x0, x1, 0x0062), __byte_perm(x2, x3, 0x0062), 0x5410);
  mw = __byte_perm(__byte_perm(x0, x1, 0x0051), __byte_perm(x2, x3, 0x0051), 0x5410);
  lw = __byte_perm(__byte_perm(x0, x1, 0x0040), __byte_perm(x2, x3, 0x0040), 0x5410);
}

// One warp builds four records per batch and two batches at a time: lane
// k = lane & 7 of each 8-lane group produces limb word k of its record.
// Activations staged in shared memory are read with one vector load per lane.

// The four activation values that limb word k of block `row` consumes.
template <bool Q4>
__device__ __forceinline__ void load_word_inputs(const void* xsrc, uint32_t xdt, bool vec, size_t row, uint32_t k,
                                                 float (&v)[4]) {
  if (vec && xdt == OVL_BF16) {
    const uint16_t* xb = static_cast<const uint16_t*>(xsrc);
    if (!Q4) {
      const uint2 w = *reinterpret_cast<const uint2*>(xb + row + 4 * k);
      v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xFFFF0000u);
      v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xFFFF0000u);
    } else {
      const uint4 w = *reinterpret_cast<const uint4*>(xb + row + 8 * (k >> 1));
      const bool odd = k & 1;
      v[0] = __uint_as_float(odd ? (w.x & 0xFFFF0000u) : (w.x << 16));
      v[1] = __uint_as_float(odd ? (w.y & 0xFFFF0000u) : (w.y << 16));
      v[2] = __uint_as_float(odd ? (w.z & 0xFFFF0000u) : (w.z << 16));
      v[3] = __uint_as_float(odd ? (w.w & 0xFFFF0000u) : (w.w << 16));
    }
  } else if (vec) {
    const float* xf = static_cast<const float*>(xsrc);
    if (!Q4) {
      const float4 w = *reinterpret_cast<const float4*>(xf + row + 4 * k);
      v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    } else {
      const float4 w0 = *reinterpret_cast<const float4*>(xf + row + 8 * (k >> 1));
      const float4 w1 = *reinterpret_cast<const float4*>(xf + row + 8 * (k >> 1) + 4);
      const bool odd = k & 1;
      v[0] = odd ? w0.y : w0.x; v[1] = odd ? w0.w : w0.z;
      v[2] = odd ? w1.y : w1.x; v[3] = odd ? w1.w : w1.z;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t e = Q4 ? (8 * (k >> 1) + (k & 1) + 2 * i) : (4 * k + i);
      v[i] = load_x(xsrc, xdt, row + e);
    }
  }
}

template <bool Q4>
__device__ __forceinline__ void build_record(uint8_t* rec, uint32_t ri, bool live, uint32_t k, const float (&v)[4],
                                             uint32_t xdt, uint32_t* mk, uint32_t mkw, uint32_t t, uint32_t b) {
  uint32_t mx = 0, mn1 = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t av = __float_as_uint(v[i]) & 0x7FFFFFFFu;
    mx = max(mx, av);
    mn1 = min(mn1, av - 1u);
  }
#pragma unroll
  for (int o = 1; o <= 4; o <<= 1) {
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn1 = min(mn1, __shfl_xor_sync(0xffffffffu, mn1, o));
  }
  const BlockScale bs = block_scale(mx);
  int X[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) X[i] = round_scaled(v[i], bs.sc);
  const float xs = bs.xs;
  // The record is the same whether or not the block is marked; a marked
  // block only sets its bit in the map (the epilogue adds its residual).
  if (block_marked(mx, mn1, xdt) && live && k == 0) mark_block(mk, mkw, t, b);
  uint32_t hw, mw, lw;
  limb_words(X, hw, mw, lw);
  int sh = 0, sm = 0, sl = 0;
  if (Q4) {
    sh = dp4a_ss(static_cast<int>(hw), 0x01010101, 0);
    sm = static_cast<int>(dp4a_uu(mw, 0x01010101u, 0u));
    sl = static_cast<int>(dp4a_uu(lw, 0x01010101u, 0u));
#pragma unroll
    for (int o = 1; o <= 4; o <<= 1) {
      sh += __shfl_xor_sync(0xffffffffu, sh, o);
      sm += __shfl_xor_sync(0xffffffffu, sm, o);
      sl += __shfl_xor_sync(0xffffffffu, sl, o);
    }
  }
  if (live) {
    uint32_t* w = reinterpret_cast<uint32_t*>(rec + static_cast<size_t>(ri) * kRecBytes);
    w[k] = hw;
    w[8 + k] = mw;
    w[16 + k] = lw;
    if (k == 0) *reinterpret_cast<uint4*>(w + 24) = make_uint4(__float_as_uint(xs), static_cast<uint32_t>(-8 * sh),
                                                                static_cast<uint32_t>(-8 * sm),
                                                                static_cast<uint32_t>(-8 * sl));
  }
}

// The record of one block built by a single lane straight into registers
// (single-token launches) from activations staged in shared memory.
template <bool Q4>
__device__ __forceinline__ void lane_record(uint4 (&r)[7], const void* xsrc, uint32_t xdt, bool vec, size_t row,
                                            uint32_t* mk, uint32_t mkw) {
  float v[32];
  if (vec && xdt == OVL_BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(xsrc) + row);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = p[q];
      v[8 * q + 0] = __uint_as_float(w.x << 16); v[8 * q + 1] = __uint_as_float(w.x & 0xFFFF0000u);
      v[8 * q + 2] = __uint_as_float(w.y << 16); v[8 * q + 3] = __uint_as_float(w.y & 0xFFFF0000u);
      v[8 * q + 4] = __uint_as_float(w.z << 16); v[8 * q + 5] = __uint_as_float(w.z & 0xFFFF0000u);
      v[8 * q + 6] = __uint_as_float(w.w << 16); v[8 * q + 7] = __uint_as_float(w.w & 0xFFFF0000u);
    }
  } else if (vec) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(xsrc) + row);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 w = p[q];
      v[4 * q + 0] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = load_x(xsrc, xdt, row + j);
  }
  uint32_t mx = 0, mn1 = 0xFFFFFFFFu;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t av = __float_as_uint(v[j]) & 0x7FFFFFFFu;
    mx = max(mx, av);
    mn1 = min(mn1, av - 1u);
  }
  const BlockScale bs = block_scale(mx);
  const float sc = bs.sc;
  int sh = 0, sm = 0, sl = 0;
  uint32_t hw[8], mw[8], lw[8];
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    int X[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) X[i] = round_scaled(v[Q4 ? (8 * (w >> 1) + (w & 1) + 2 * i) : (4 * w + i)], sc);
    limb_words(X, hw[w], mw[w], lw[w]);
    if (Q4) {
      sh = dp4a_ss(static_cast<int>(hw[w]), 0x01010101, sh);
      sm = static_cast<int>(dp4a_uu(mw[w], 0x01010101u, static_cast<uint32_t>(sm)));
      sl = static_cast<int>(dp4a_uu(lw[w], 0x01010101u, static_cast<uint32_t>(sl)));
    }
  }
  r[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  r[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
  r[2] = make_uint4(mw[0], mw[1], mw[2], mw[3]);
  r[3] = make_uint4(mw[4], mw[5], mw[6], mw[7]);
  r[4] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  r[5] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
  const float xs = bs.xs;
  // The record is the same whether or not the block is marked; a marked
  // block only sets its bit in the map (the epilogue adds its residual).
  if (block_marked(mx, mn1, xdt)) mark_block(mk, mkw, 0, static_cast<uint32_t>(row >> 5));
  r[6] = Q4 ? make_uint4(__float_as_uint(xs), static_cast<uint32_t>(-8 * sh), static_cast<uint32_t>(-8 * sm),
                         static_cast<uint32_t>(-8 * sl))
            : make_uint4(__float_as_uint(xs), 0u, 0u, 0u);
}

template <bool Q4>
__device__ __forceinline__ void prep_records(uint8_t* rec, const DualArgs& a, const void* xsrc, bool vec, uint32_t nb,
                                             uint32_t warp, uint32_t nwarps, uint32_t lane, uint32_t* mk,
                                             uint32_t mkw) {
  const uint32_t k = lane & 7;
  const uint32_t total = a.T * nb;
  for (uint32_t base = warp * 8; base < total; base += nwarps * 8) {
    const uint32_t ri0 = base + (lane >> 3), ri1 = ri0 + 4;
    const bool live0 = ri0 < total, live1 = ri1 < total;
    const uint32_t t0 = live0 ? ri0 / nb : 0, b0 = live0 ? ri0 - t0 * nb : 0;
    const uint32_t t1 = live1 ? ri1 / nb : 0, b1 = live1 ? ri1 - t1 * nb : 0;
    float v0[4] = {0.f, 0.f, 0.f, 0.f}, v1[4] = {0.f, 0.f, 0.f, 0.f};
    if (live0) load_word_inputs<Q4>(xsrc, a.xdt, vec, static_cast<size_t>(t0) * a.n + static_cast<size_t>(b0) * 32, k, v0);
    if (live1) load_word_inputs<Q4>(xsrc, a.xdt, vec, static_cast<size_t>(t1) * a.n + static_cast<size_t>(b1) * 32, k, v1);
    build_record<Q4>(rec, ri0, live0, k, v0, a.xdt, mk, mkw, t0, b0);
    build_record<Q4>(rec, ri1, live1, k, v1, a.xdt, mk, mkw, t1, b1);
  }
}

// P = 65536 sh + 256 sm + sl from the exact limb sums (|sh| < 2^19, |sm|, |sl|
// < 2^21): U = 256 sh + sm is exact in int32 and rounds once to fp32, then
// one FMA adds sl (exact in fp32), so |P~ - P| <= 2^-24 (2 |P| + |sl|) + 2^-24
// |P|: relative to P itself plus a fraction of one unit, with no cancellation
// between limbs whatever the signs of the elements.
__device__ __forceinline__ float limb_combine(int sh, int sm, int sl) {
  return fmaf(__int2float_rn(sh * 256 + sm), 256.f, __int2float_rn(sl));
}

// d * sc_j and dmin * m_j of sub-block j (j6 = 6 j) from a q4_K super-block
// header {d, dmin (binary16), sc_0..7 (6 bits each), m_0..7 (6 bits each)}.
// Both products are exact in fp32.
__device__ __forceinline__ void q4k_scales(const uint4 h, uint32_t j6, float* dsc, float* dmn) {
  const uint64_t scf = (static_cast<uint64_t>(h.z & 0xFFFFu) << 32) | h.y;
  const uint64_t mnf = (static_cast<uint64_t>(h.w) << 16) | (h.z >> 16);
  *dsc = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x & 0xFFFFu))) *
         static_cast<float>(static_cast<uint32_t>(scf >> j6) & 63u);
  *dmn = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x >> 16))) *
         static_cast<float>(static_cast<uint32_t>(mnf >> j6) & 63u);
}

// The residual product of a marked block with one row: sum_j w_j r_j, where
// r_j = x_j - X_j 2^-s is what the block's record left out of element j (the
// record's X_j and 2^-s are recomputed from x exactly as the record was built)
// and w_j = fma(code_j, dq, -dm) (q8_0: code = q, dq = d, dm = 0; q4_0: code
// 0..15, dq = d, dm = 8 d -- both exact; q4_K: dq = d sc_j, dm = dmin m_j, one
// rounding).  r_j is exact in fp32 (a multiple of the element's own unit in the
// last place, below half a grid step) and |r_j| <= |x_j|.  Four fixed FMA chains,
// combined in a fixed order.  Error <= 10 * 2^-24 * sum|w_j r_j|.
template <bool Q4>
__device__ __forceinline__ float block_residual(const uint4 (&wq)[2], float dq, float dm, const void* xsrc,
                                                uint32_t xdt, size_t xoff) {
  uint32_t mx = 0;
  for (int j = 0; j < 32; ++j) mx = max(mx, __float_as_uint(load_x(xsrc, xdt, xoff + j)) & 0x7FFFFFFFu);
  const BlockScale bs = block_scale(mx);
  const uint32_t* wb = reinterpret_cast<const uint32_t*>(wq);
  float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int j = 0; j < 32; ++j) {
    const float v = load_x(xsrc, xdt, xoff + j);
    const float Xf = static_cast<float>(round_scaled(v, bs.sc));
    const float r = fmaf(-Xf, bs.xs, v);
    const uint32_t byte = (wb[(Q4 ? (j >> 1) : j) >> 2] >> (8 * ((Q4 ? (j >> 1) : j) & 3))) & 0xFFu;
    const float code = Q4 ? static_cast<float>((byte >> (4 * (j & 1))) & 15u)
                          : static_cast<float>(static_cast<int8_t>(static_cast<uint8_t>(byte)));
    c[j & 3] = fmaf(fmaf(code, dq, -dm), r, c[j & 3]);
  }
  return (c[0] + c[1]) + (c[2] + c[3]);
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

// q4_0: unsigned codes 0..15 against the limbs; the -8 offset is in the
// accumulator starts of the record.
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

// dot_q4 with zero accumulator starts: sum(code * X) for codes 0..15 (q4_K,
// whose minimum term needs sum(X) separately).
__device__ __forceinline__ float dot_q4_zero(const uint8_t* wp, const uint4 (&r)[7]) {
  uint4 z = r[6];
  z.y = 0u; z.z = 0u; z.w = 0u;
  const uint4 rz[7] = {r[0], r[1], r[2], r[3], r[4], r[5], z};
  return dot_q4(wp, rz);
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

// Global address of element f of the flattened [rtot][n] factor space.
__device__ __forceinline__ const float* factor_ptr(const DualArgs& a, uint64_t f) {
  const uint32_t rho = static_cast<uint32_t>(f / a.n);
  uint32_t k = 0, rbase = 0;
  while (rho >= rbase + a.lora[k].r) { rbase += a.lora[k].r; ++k; }
  return a.lora[k].A + static_cast<size_t>(rho - rbase) * a.n + (f - static_cast<uint64_t>(rho) * a.n);
}

// This CTA's chunk [lo, hi) of the flattened factor space (contiguous chunks,
// one per shrink CTA).
__device__ __forceinline__ void shrink_bounds(const DualArgs& a, const DualCfg& c, uint32_t cta, uint64_t* lo,
                                              uint64_t* hi) {
  if (c.div32) {
    const uint32_t total = a.rtot * a.n;
    *lo = cta * total / c.gs;
    *hi = (cta + 1) * total / c.gs;
  } else {
    const uint64_t total = static_cast<uint64_t>(a.rtot) * a.n;
    *lo = cta * total / c.gs;
    *hi = (cta + 1) * total / c.gs;
  }
}

// Range [cf, cl] of shrink CTAs whose chunk overlaps factor row rho.
__device__ __forceinline__ void partial_range(const DualArgs& a, const DualCfg& c, uint32_t rho, uint32_t* cf,
                                              uint32_t* cl) {
  uint32_t f, l;
  if (c.div32) {
    const uint32_t total = a.rtot * a.n;
    f = ((rho * a.n + 1) * c.gs + total - 1) / total;
    l = ((rho + 1) * a.n * c.gs + total - 1) / total;
  } else {
    const uint64_t total = static_cast<uint64_t>(a.rtot) * a.n;
    f = static_cast<uint32_t>(((static_cast<uint64_t>(rho) * a.n + 1) * c.gs + total - 1) / total);
    l = static_cast<uint32_t>(((static_cast<uint64_t>(rho + 1) * a.n) * c.gs + total - 1) / total);
  }
  f = f ? f - 1 : 0;
  l = l ? l - 1 : 0;
  *cf = f;
  *cl = l > c.gs - 1 ? c.gs - 1 : l;
}

// The part of x that a shrink chunk [lo, hi) of the flattened factor space
// touches (x index j = f mod n), widened to 16-byte granules of g elements:
// piece 1 = x[w0, w1), then, when the chunk wraps past the end of a row,
// piece 2 = x[0, w2).  A chunk of n or more elements takes the whole of x.
struct XWindow {
  uint32_t w0, w1, w2;
};
__device__ __forceinline__ XWindow x_window(uint64_t lo, uint64_t hi, uint32_t n, uint32_t g) {
  if (hi - lo >= n) return XWindow{0u, n, 0u};
  const uint32_t j0 = static_cast<uint32_t>(lo % n);
  const uint32_t je = j0 + static_cast<uint32_t>(hi - lo);
  const uint32_t w0 = j0 / g * g;
  if (je <= n) return XWindow{w0, min(n, (je + g - 1) / g * g), 0u};
  return XWindow{w0, n, (je - n + g - 1) / g * g};
}

// One low-rank term of this CTA's tensor, copied from the kernel parameters
// into shared memory at the start so that the B stage and the epilogue do not
// wait on constant-cache misses.  `here` = byte offset of this CTA's first B
// row inside the B stage.
struct EpTerm {
  const float* B;
  uint32_t r;
  float s;
  uint32_t here;
  uint32_t pad;
};

// Eight consecutive activations x[idx .. idx+8) (idx a multiple of 8, rows
// 16-byte aligned): one 16-byte load for bf16, two for fp32.
__device__ __forceinline__ void load_x8(const void* x, uint32_t xdt, size_t idx, float (&v)[8]) {
  if (xdt == OVL_BF16) {
    const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + idx);
    v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xFFFF0000u);
    v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xFFFF0000u);
    v[4] = __uint_as_float(w.z << 16); v[5] = __uint_as_float(w.z & 0xFFFF0000u);
    v[6] = __uint_as_float(w.w << 16); v[7] = __uint_as_float(w.w & 0xFFFF0000u);
  } else {
    const float4 p = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx);
    const float4 q = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx + 4);
    v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w;
    v[4] = q.x; v[5] = q.y; v[6] = q.z; v[7] = q.w;
  }
}

// Term (index into this CTA's term table) that factor row rho belongs to.
__device__ __forceinline__ uint32_t term_of_row(const EpTerm* ep, uint32_t nterm, uint32_t rho) {
  uint32_t k = 0, base = 0;
  while (k + 1 < nterm && rho >= base + ep[k].r) base += ep[k++].r;
  return k;
}

// Tokens of the launch that need factor row rho: all of them, or (segmented
// batches) those whose selected term owns the row.
__device__ __forceinline__ uint32_t row_token_mask(const DualArgs& a, const EpTerm* ep, uint32_t nterm, uint32_t rho) {
  uint32_t m = a.T >= 32 ? ~0u : ((1u << a.T) - 1u);
  if (a.tok_sel) {
    const int k = static_cast<int>(term_of_row(ep, nterm, rho));
    m = 0;
    for (uint32_t t = 0; t < a.T && t < 8; ++t)
      if (a.tok_term[t] == k) m |= 1u << t;
  }
  return m;
}

// Epoch tag of a shrink CTA's partial sums.  With the test-only withhold flag
// CTA 0 tags them with a value no reader accepts, so the gather's bounded
// wait runs out.
__device__ __forceinline__ uint32_t launch_epoch(const DualArgs& a) { return a.epoch & ~kEpochWithhold; }
__device__ __forceinline__ uint32_t slot_tag(const DualArgs& a, uint32_t cta) {
  return ((a.epoch & kEpochWithhold) && cta == 0) ? a.epoch : launch_epoch(a);
}

// Partial shrink sums of this CTA's chunk of the flattened [rtot][n] factor
// space, computed by one warp: slot (t * rtot + rho) * gs + cta receives
// sum_{j in chunk, row rho} A[rho][j] x[t][j] for every token t that needs
// row rho, tagged with the launch epoch in one 64-bit store.  Each lane takes
// groups of eight consecutive elements (one 16-byte activation load per
// token); sums run in a fixed order (per lane over its groups, then a fixed
// warp reduction).
template <int TT>
__device__ void shrink_chunk_warp(const DualArgs& a, const DualCfg& c, uint32_t cta, const float* sA,
                                  const void* xsrc, const EpTerm* ep, uint32_t nterm, uint32_t lane) {
  uint64_t lo, hi;
  shrink_bounds(a, c, cta, &lo, &hi);
  unsigned long long* slots = reinterpret_cast<unsigned long long*>(a.ws.partial);
  const uint32_t rho_a = static_cast<uint32_t>(lo / a.n), rho_b = static_cast<uint32_t>((hi - 1) / a.n);
  for (uint32_t rho = rho_a; rho <= rho_b; ++rho) {
    const uint32_t tmask = row_token_mask(a, ep, nterm, rho);
    if (!tmask) continue;
    const uint64_t rs = static_cast<uint64_t>(rho) * a.n;
    const uint32_t j0 = static_cast<uint32_t>(max(lo, rs) - rs);
    const uint32_t j1 = static_cast<uint32_t>(min(hi, rs + a.n) - rs);
    const float* Arow = c.stage_a ? sA + (static_cast<int64_t>(rs) - static_cast<int64_t>(lo)) : factor_ptr(a, rs);
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.f;
    if (c.xvec) {
      constexpr int kUnroll = TT == 1 ? 2 : 1;   // loads in flight without spilling
#pragma unroll kUnroll
      for (uint32_t jj = (j0 & ~7u) + 8 * lane; jj < j1; jj += 256) {
        float av[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) av[e] = (jj + e >= j0 && jj + e < j1) ? Arow[jj + e] : 0.f;
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (!((tmask >> t) & 1u)) continue;
          float xv[8];
          load_x8(xsrc, a.xdt, static_cast<size_t>(t) * a.n + jj, xv);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[t] = fmaf(av[e], xv[e], acc[t]);
        }
      }
    } else {
      for (uint32_t j = j0 + lane; j < j1; j += 32) {
        const float av = Arow[j];
#pragma unroll
        for (int t = 0; t < TT; ++t)
          if ((tmask >> t) & 1u) acc[t] = fmaf(av, load_x(xsrc, a.xdt, static_cast<size_t>(t) * a.n + j), acc[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      if (!((tmask >> t) & 1u)) continue;
      const float v = warp_sum(acc[t]);
      if (lane == 0)
        st_relaxed_u64(slots + (static_cast<size_t>(t) * a.rtot + rho) * c.gs + cta,
                       (static_cast<unsigned long long>(slot_tag(a, cta)) << 32) | __float_as_uint(v));
    }
  }
}

// v[t][rho] for NP factor rows per lane (pairs base + lane + 32 h): every
// shrink slot of a row, PER slots per row and round, all loads of a round in
// flight together; a round is repeated (bounded) until each slot carries this
// launch's epoch.  Each row is summed over its slots in CTA order.
template <int NP, int PER>
__device__ __forceinline__ void gather_rows(const DualArgs& a, const DualCfg& c, float* vsm, uint32_t base,
                                            const EpTerm* ept, uint32_t nterm, uint32_t lane) {
  bool ok = true;
  const unsigned long long* slots = reinterpret_cast<const unsigned long long*>(a.ws.partial);
  const uint32_t npairs = a.T * a.rtot;
  const uint32_t ep = launch_epoch(a);
  const uint32_t limit = (a.epoch & kEpochWithhold) ? (1u << 10) : (1u << 21);
  uint32_t cf[NP], cl[NP];
  bool live[NP];
  const unsigned long long* pp[NP];
  float sum[NP];
#pragma unroll
  for (int h = 0; h < NP; ++h) {
    const uint32_t i = base + lane + 32 * h;
    live[h] = i < npairs;
    const uint32_t t = live[h] ? i / a.rtot : 0, rho = live[h] ? i - t * a.rtot : 0;
    // segmented batches: a token needs only the rows of its own term
    if (live[h] && a.tok_sel && a.tok_term[t] != static_cast<int>(term_of_row(ept, nterm, rho))) live[h] = false;
    partial_range(a, c, rho, &cf[h], &cl[h]);
    pp[h] = slots + (static_cast<size_t>(t) * a.rtot + rho) * c.gs;
    sum[h] = 0.f;
  }
  for (uint32_t q = 0;; q += PER) {
    bool more = false;
#pragma unroll
    for (int h = 0; h < NP; ++h) more = more || (live[h] && cf[h] + q <= cl[h]);
    if (!more) break;
    unsigned long long v[NP][PER];
    for (uint32_t it = 0;; ++it) {
      bool all = true;
#pragma unroll
      for (int h = 0; h < NP; ++h) {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const uint32_t qq = cf[h] + q + u;
          const bool use = live[h] && qq <= cl[h];
          v[h][u] = use ? ld_relaxed_u64(pp[h] + qq) : 0ull;
          all = all && (!use || static_cast<uint32_t>(v[h][u] >> 32) == ep);
        }
      }
      if (all) break;
      if (it > limit) {
        latch(a.ws.status, kDevTimeoutShrink);
        ok = false;
        break;
      }
      __nanosleep(64);
    }
#pragma unroll
    for (int h = 0; h < NP; ++h)
#pragma unroll
      for (int u = 0; u < PER; ++u)
        if (live[h] && cf[h] + q + u <= cl[h]) sum[h] += __uint_as_float(static_cast<uint32_t>(v[h][u]));
  }
  // A row whose poll gave up is stored as NaN: every output that uses it
  // becomes NaN instead of silently missing part of its low-rank term.
#pragma unroll
  for (int h = 0; h < NP; ++h)
    if (live[h]) vsm[base + lane + 32 * h] = ok ? sum[h] : __uint_as_float(0x7FC00000u);
}

// The B rows [row0, row0 + nrows) of one low-rank term as a 16-byte aligned
// byte span (bulk-copy granularity); `skew` = offset of the first row in it.
struct BSpan {
  const uint8_t* lo;
  uint32_t bytes, skew;
};
__device__ __forceinline__ BSpan b_span(const float* B, uint32_t r, uint32_t row0, uint32_t nrows) {
  const uintptr_t s = reinterpret_cast<uintptr_t>(B + static_cast<size_t>(row0) * r);
  const uintptr_t e = s + static_cast<uintptr_t>(nrows) * r * 4u;
  const uintptr_t lo = s & ~static_cast<uintptr_t>(15);
  return BSpan{reinterpret_cast<const uint8_t*>(lo), static_cast<uint32_t>(((e + 15) & ~static_cast<uintptr_t>(15)) - lo),
               static_cast<uint32_t>(s - lo)};
}

// Sum over the marked blocks of token t (ascending block order) of their
// residual products with row `row` of the CTA's tensor, in plain fp32: each
// block's weights are re-read from the immutable base planes in global memory.
template <int QUANT>
__device__ __noinline__ float marked_sum(const uint32_t* mk, const DualArgs& a, const DualCfg& c, const DualSeg& sg,
                                         uint32_t t, uint32_t row, const void* xsrc) {
  constexpr bool QK4 = QUANT == OVL_Q4_K;
  constexpr bool Q4 = QUANT != OVL_Q8_0;
  const uint32_t mkw = map_words(c.nb);
  float sum = 0.f;
  for (uint32_t w = 0; w < mkw; ++w) {
    uint32_t bits = mk[1 + t * mkw + w];
    while (bits) {
      const uint32_t b = 32 * w + static_cast<uint32_t>(__ffs(static_cast<int>(bits)) - 1);
      bits &= bits - 1;
      const uint8_t* wp = sg.qs + static_cast<size_t>(row) * c.rowbytes + static_cast<size_t>(b) * (Q4 ? 16u : 32u);
      uint4 wq[2];
      wq[0] = *reinterpret_cast<const uint4*>(wp);
      wq[1] = Q4 ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(wp + 16);
      float dq, dm;
      if constexpr (QK4) {
        const uint4 h =
            *reinterpret_cast<const uint4*>(sg.dpl + static_cast<size_t>(row) * c.nb * 2 + (b >> 3) * 16u);
        q4k_scales(h, 6u * (b & 7u), &dq, &dm);
      } else {
        dq = __half2float(*reinterpret_cast<const __half*>(sg.dpl + (static_cast<size_t>(row) * c.nb + b) * 2));
        dm = Q4 ? 8.f * dq : 0.f;
      }
      sum += block_residual<Q4>(wq, dq, dm, xsrc, a.xdt, static_cast<size_t>(t) * a.n + static_cast<size_t>(b) * 32);
    }
  }
  return sum;
}

template <int QUANT, int TT, int RG, bool VX = false>
__global__ void __launch_bounds__(K1Shape<TT, RG>::threads, K1Shape<TT, RG>::min_blocks)
    k_dualpath(const DualArgs a, const DualCfg c) {
  constexpr int NREG = K1Shape<TT, RG>::reg_records;
  // q4_K shares q4_0's codes, records and stage layout; only the per-block
  // scale (and its minimum term) differ.
  constexpr bool QK4 = QUANT == OVL_Q4_K;
  constexpr bool Q4 = QUANT == OVL_Q4_0 || QK4;
  constexpr int N = TT * RG;
  constexpr int LN = Log2<N>::v;
  constexpr uint32_t kBlockBytes = Q4 ? 16 : 32;
  extern __shared__ __align__(1024) uint8_t sm[];
  if constexpr (VX) {
    if (c.shrink_only) {
      // v[rho] = A_rho . x for factor row rho = blockIdx.x: the shrink launch
      // of a single-token launch with long factor rows, run by this same kernel
      // so consecutive launches stay on one function.  Each thread takes 8
      // elements of every blockDim.x * 8; fixed-order warp sums, then the
      // warps' sums in warp order.
      griddep_launch_dependents();
      griddep_wait();   // x may come from the preceding grid
      float* part = reinterpret_cast<float*>(sm);
      const uint32_t rho = blockIdx.x, w = threadIdx.x >> 5, ln = threadIdx.x & 31;
      const float* Arow = factor_ptr(a, static_cast<uint64_t>(rho) * a.n);
      float acc0 = 0.f, acc1 = 0.f;
      for (uint32_t j = threadIdx.x * 8; j < a.n; j += blockDim.x * 8) {
        const float4 p = *reinterpret_cast<const float4*>(Arow + j);
        const float4 q = *reinterpret_cast<const float4*>(Arow + j + 4);
        float xv[8];
        load_x8(a.x, a.xdt, j, xv);
        acc0 = fmaf(p.x, xv[0], acc0); acc1 = fmaf(p.y, xv[1], acc1);
        acc0 = fmaf(p.z, xv[2], acc0); acc1 = fmaf(p.w, xv[3], acc1);
        acc0 = fmaf(q.x, xv[4], acc0); acc1 = fmaf(q.y, xv[5], acc1);
        acc0 = fmaf(q.z, xv[6], acc0); acc1 = fmaf(q.w, xv[7], acc1);
      }
      const float sum = warp_sum(acc0 + acc1);
      if (ln == 0) part[w] = sum;
      __syncthreads();
      if (threadIdx.x == 0) {
        float t = part[0];
        for (uint32_t i = 1; i < blockDim.x / 32; ++i) t += part[i];
        a.ws.tc_scratch[rho] = t;
      }
      return;
    }
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(sm);
  uint64_t* empty = full + kMaxNS;
  uint64_t* vbar = empty + kMaxNS;                  // low-rank vector ready
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(vbar + 1);
  uint8_t* rec = sm + c.off_rec;
  uint8_t* stages = sm + c.off_stage;
  float* red = reinterpret_cast<float*>(sm + c.off_red);
  float* vsm = reinterpret_cast<float*>(sm + c.off_v);
  EpTerm* ep = reinterpret_cast<EpTerm*>(sm + c.off_ep);
  float* sA = reinterpret_cast<float*>(sm + c.off_a);
  uint32_t* mk = reinterpret_cast<uint32_t*>(sm + c.off_mk);

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ncw = c.nwc * c.ng;               // consumer warps
  const uint32_t nthr = ncw * 32;
  const uint32_t cta = blockIdx.x;
  // this CTA's tensor and its contiguous row slice of that tensor
  uint32_t si = 0;
  while (si + 1 < a.nseg && cta >= a.seg[si + 1].g0) ++si;
  const DualSeg& sg = a.seg[si];
  const uint32_t lc = cta - sg.g0;
  const uint32_t row0 = static_cast<uint32_t>((static_cast<uint64_t>(lc) * sg.m) / sg.gn);
  const uint32_t row1 = static_cast<uint32_t>((static_cast<uint64_t>(lc + 1) * sg.m) / sg.gn);
  const uint32_t nrows = row1 - row0;
  const uint32_t nst = (nrows + RG - 1) / RG;

  for (uint32_t i = threadIdx.x; i < 1 + TT * map_words(c.nb); i += blockDim.x) mk[i] = 0u;
  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < c.ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], c.nwc);
    }
    mbar_init(vbar, 1);
    *abort_flag = 0u;
    mbar_fence_init();
  }
  if (warp == 1 % (ncw + 2) && a.nl) {
    // this tensor's low-rank terms (B stage layout: one 16-byte span per term)
    const uint32_t nt = sg.k1 - sg.k0;
    for (uint32_t k = lane; k < nt; k += 32) {
      const LoraRef L = a.lora[sg.k0 + k];
      ep[k] = EpTerm{L.B, L.r, L.s, 0u, 0u};
    }
    __syncwarp();
    if (lane == 0) {
      uint32_t off = 0;
      for (uint32_t k = 0; k < nt; ++k) {
        const BSpan sp = b_span(ep[k].B, ep[k].r, row0, nrows);
        ep[k].here = off + sp.skew;
        off += sp.bytes;
      }
    }
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == ncw) {
    if (lane == 0) {
      // ---------------- producer: stream this CTA's rows in order.  The base is
      // immutable, so this starts before the preceding grid has finished.
      const uint64_t pol = l2_evict_first_policy();
      // The B rows are copied in late (after the shrink, or after the last
      // base stage): bring them into L2 now so that copy does not wait on HBM.
      if (c.b_ring || c.b_areg)
        for (uint32_t k = 0; k < sg.k1 - sg.k0; ++k) {
          const BSpan sp = b_span(ep[k].B, ep[k].r, row0, nrows);
          bulk_prefetch_l2(sp.lo, sp.bytes);
        }
      uint32_t issued = 0;
      uint32_t slot = 0, lap = 0;   // slot = s mod ns, lap = s / ns, kept as counters
      for (uint32_t s = 0; s < nst; ++s) {
        if (s != 0 && ++slot == c.ns) {
          slot = 0;
          ++lap;
        }
        if (lap != 0 && !mbar_wait_bounded(&empty[slot], (lap - 1) & 1)) {
          latch(a.ws.status, kDevTimeoutEmpty);
          *abort_flag = 1u;
          break;
        }
        if (s == kPreDepStages) {
          // Only the first stages go to shared memory before the grid
          // dependency resolves; the rest of the ring's worth of quantized
          // rows is requested into L2.  Their copies to shared memory, issued
          // after the dependency, hit L2, and the activation reads that the
          // records need right after the dependency do not queue behind a
          // full ring of weights arriving at this SM.  (Prefetching the
          // scale rows as well measured slower.)
          const uint32_t ra = row0 + s * RG;
          const uint32_t ahead = c.ns > kPreDepStages ? c.ns - kPreDepStages : 0u;
          const size_t q0 = static_cast<size_t>(ra) * c.rowbytes;
          const uint32_t rows_ahead = min(row1 - ra, ahead * RG);
          const size_t len = static_cast<size_t>(rows_ahead) * c.rowbytes;
          for (size_t off = 0; off < len; off += 16384) {
            const uint32_t b = static_cast<uint32_t>(len - off < 16384 ? len - off : 16384);
            bulk_prefetch_l2(sg.qs + q0 + off, b);
          }
          griddep_wait();
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
        bulk_g2s(dst, sg.qs + static_cast<size_t>(r0) * c.rowbytes, bq, &full[slot], pol);
        bulk_g2s(dst + c.stage_q, sg.dpl + d0, static_cast<uint32_t>(d1 - d0), &full[slot], pol);
        ++issued;
      }
      // B rows of this CTA's low-rank terms: one more stage, read by the epilogue.
      if (c.b_ring && sg.k1 > sg.k0 && issued == nst && !*abort_flag) {
        const uint32_t s = nst, slot = s % c.ns;
        if (s >= c.ns && !mbar_wait_bounded(&empty[slot], ((s / c.ns) - 1) & 1)) {
          latch(a.ws.status, kDevTimeoutEmpty);
          *abort_flag = 1u;
        } else {
          const uint32_t nt = sg.k1 - sg.k0;
          const BSpan last = b_span(ep[nt - 1].B, ep[nt - 1].r, row0, nrows);
          mbar_arrive_expect_tx(&full[slot], ep[nt - 1].here - last.skew + last.bytes);
          uint8_t* dst = stages + static_cast<size_t>(slot) * c.stage_bytes;
          for (uint32_t k = 0; k < nt; ++k) {
            const BSpan sp = b_span(ep[k].B, ep[k].r, row0, nrows);
            bulk_g2s(dst + ep[k].here - sp.skew, sp.lo, sp.bytes, &full[slot], pol);
          }
          ++issued;
        }
      }
      // Do not leave while copies into this CTA's shared memory may be in flight.
      const uint32_t first = issued > c.ns ? issued - c.ns : 0;
      for (uint32_t s = first; s < issued; ++s) mbar_wait_bounded(&full[s % c.ns], (s / c.ns) & 1);
    }
    return;
  }
  if (warp == ncw + 1) {
    // ---------------- helper warp: the low-rank side product, off the critical
    // path.  Stage this CTA's shrink chunk of A (before the grid dependency
    // resolves: the factors are immutable) and, after it, the x window of the
    // chunk; reduce the chunk, publish the epoch-tagged partial sums, then
    // gather every partial of every factor row (bounded polling on the epochs),
    // sum them in a fixed order into v and release the epilogue.
    if (!a.nl) return;
    if constexpr (VX) {
      // The low-rank vector v = A x of this launch comes from the shrink
      // launch just before it (this kernel in its shrink-only mode, v in the
      // workspace's tensor-core scratch): read it once the grid dependency
      // has resolved.
      griddep_wait();
      const float* vsrc = a.ws.tc_scratch;
      for (uint32_t i = lane; i < a.T * a.rtot; i += 32) vsm[i] = vsrc[i];
      __syncwarp();
      if (lane == 0) mbar_arrive(vbar);
      return;
    }
    uint64_t lo = 0, hi = 0;
    if (cta < c.gs) shrink_bounds(a, c, cta, &lo, &hi);
    const bool vec = c.shrink_vec && cta < c.gs;
    uint32_t rho_a = 0, w0 = 0;
    if (vec) {
      // Element f of the chunk lives at index f - rho_a n - w0 of both the
      // staged A and the x window (w0 = the window start, a multiple of the
      // 16-byte granule); each factor row is copied as its 16-byte aligned
      // superset [j0 & ~3, (j1 + 3) & ~3).
      const uint32_t g = a.xdt == OVL_BF16 ? 8u : 4u;
      rho_a = static_cast<uint32_t>(lo / a.n);
      w0 = static_cast<uint32_t>(lo - static_cast<uint64_t>(rho_a) * a.n) / g * g;
      const uint32_t rho_b = static_cast<uint32_t>((hi - 1) / a.n);
      for (uint32_t rho = rho_a; rho <= rho_b; ++rho) {
        const uint64_t rs = static_cast<uint64_t>(rho) * a.n;
        const uint32_t j0 = static_cast<uint32_t>(max(lo, rs) - rs);
        const uint32_t j1 = static_cast<uint32_t>(min(hi, rs + a.n) - rs);
        const float* Arow = factor_ptr(a, rs);
        float* dst = sA + ((rho - rho_a) * a.n - w0);
        for (uint32_t e = (j0 >> 2) + lane; e < ((j1 + 3) >> 2); e += 32) cp_async16(dst + 4 * e, Arow + 4 * e);
      }
    } else if (c.stage_a && cta < c.gs) {
      const uint32_t rho_a = static_cast<uint32_t>(lo / a.n), rho_b = static_cast<uint32_t>((hi - 1) / a.n);
      for (uint32_t rho = rho_a; rho <= rho_b; ++rho) {
        const uint64_t rs = static_cast<uint64_t>(rho) * a.n;
        const uint32_t j0 = static_cast<uint32_t>(max(lo, rs) - rs);
        const uint32_t j1 = static_cast<uint32_t>(min(hi, rs + a.n) - rs);
        const float* Arow = factor_ptr(a, rs);
        float* dstA = sA + (static_cast<int64_t>(rs) - static_cast<int64_t>(lo));
        for (uint32_t j = j0 + lane; j < j1; j += 32) cp_async4(dstA + j, Arow + j);
      }
    }
    cp_async_commit();
    griddep_wait();
    XWindow win{0u, 0u, 0u};
    const void* xw = nullptr;
    if (c.xwin && cta < c.gs) {
      const uint32_t esz = a.xdt == OVL_BF16 ? 2u : 4u, g = 16u / esz;
      win = x_window(lo, hi, a.n, g);
      uint8_t* sXw = sm + c.off_xw;
      const uint8_t* gx = static_cast<const uint8_t*>(a.x);
      const uint32_t n1 = (win.w1 - win.w0) / g, n2 = win.w2 / g;
      for (uint32_t e = lane; e < n1; e += 32) cp_async16(sXw + e * 16, gx + static_cast<size_t>(win.w0) * esz + e * 16);
      for (uint32_t e = lane; e < n2; e += 32) cp_async16(sXw + (n1 + e) * 16, gx + e * 16);
      cp_async_commit();
      xw = sXw;
    } else if (c.xfull && cta < c.gs) {
      uint8_t* sXw = sm + c.off_xw;
      const uint8_t* gx = static_cast<const uint8_t*>(a.x);
      const uint32_t nvec = a.n * (a.xdt == OVL_BF16 ? 2u : 4u) / 16u;
      for (uint32_t e = lane; e < nvec; e += 32) cp_async16(sXw + e * 16, gx + e * 16);
      cp_async_commit();
    }
    cp_async_wait_all();
    __syncwarp();
    if (c.stage_x) named_bar(2, nthr + 32);         // the consumers have staged x
    const void* xsrc = c.stage_x ? static_cast<const void*>(sm + c.off_x)
                                 : (c.xfull ? static_cast<const void*>(sm + c.off_xw) : a.x);
    if (vec) {
      unsigned long long* slots = reinterpret_cast<unsigned long long*>(a.ws.partial);
      const uint32_t rho_b = static_cast<uint32_t>((hi - 1) / a.n);
      const uint64_t fb = static_cast<uint64_t>(rho_a) * a.n + w0;
      for (uint32_t rho = rho_a; rho <= rho_b; ++rho) {
        const uint64_t rs = static_cast<uint64_t>(rho) * a.n;
        const uint32_t i0 = static_cast<uint32_t>(max(lo, rs) - fb);
        const uint32_t i1 = static_cast<uint32_t>(min(hi, rs + a.n) - fb);
        float c4[4] = {0.f, 0.f, 0.f, 0.f};
        for (uint32_t idx = (i0 & ~3u) + 4 * lane; idx < i1; idx += 128) {
          const float4 av = *reinterpret_cast<const float4*>(sA + idx);
          float xv[4];
          if (a.xdt == OVL_BF16) {
            const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(xw) + idx);
            xv[0] = __uint_as_float(w.x << 16); xv[1] = __uint_as_float(w.x & 0xFFFF0000u);
            xv[2] = __uint_as_float(w.y << 16); xv[3] = __uint_as_float(w.y & 0xFFFF0000u);
          } else {
            const float4 w = *reinterpret_cast<const float4*>(static_cast<const float*>(xw) + idx);
            xv[0] = w.x; xv[1] = w.y; xv[2] = w.z; xv[3] = w.w;
          }
          const float aq[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (idx + q >= i0 && idx + q < i1) c4[q] = fmaf(aq[q], xv[q], c4[q]);
        }
        const float v = warp_sum((c4[0] + c4[1]) + (c4[2] + c4[3]));
        if (lane == 0)
          st_relaxed_u64(slots + static_cast<size_t>(rho) * c.gs + cta,
                         (static_cast<unsigned long long>(slot_tag(a, cta)) << 32) | __float_as_uint(v));
      }
    } else if (cta < c.gs) {
      shrink_chunk_warp<TT>(a, c, cta, sA, xsrc, ep, sg.k1 - sg.k0, lane);
    }
    if (c.b_areg) {
      // The A chunk and the x window are consumed: reuse their area for this
      // CTA's B rows (16-byte copies of each term's span), ready long before
      // the base stream ends.
      __syncwarp();
      uint8_t* dstB = sm + c.off_a;
      for (uint32_t k = 0; k < sg.k1 - sg.k0; ++k) {
        const BSpan sp = b_span(ep[k].B, ep[k].r, row0, nrows);
        uint8_t* d = dstB + ep[k].here - sp.skew;
        for (uint32_t e = lane; e < sp.bytes / 16; e += 32) cp_async16(d + e * 16, sp.lo + e * 16);
      }
      cp_async_commit();
    }
    // v[t][rho] = sum over the shrink CTAs covering row rho, in CTA order.
    for (uint32_t base = 0; base < a.T * a.rtot; base += 64) {
      if (a.T * a.rtot - base > 32) gather_rows<2, 6>(a, c, vsm, base, ep, sg.k1 - sg.k0, lane);
      else gather_rows<1, 16>(a, c, vsm, base, ep, sg.k1 - sg.k0, lane);
    }
    cp_async_wait_all();   // B rows (when copied here) land before the release
    __syncwarp();
    if (lane == 0) mbar_arrive(vbar);
    return;
  }

  // ---------------- consumers
  const uint32_t grp = warp / c.nwc;                // consumer group: stages grp, grp+ng, ...
  const uint32_t cw = warp - grp * c.nwc;           // column warp inside the group
  const uint32_t L = cw * 32 + lane;                // column lane: blocks L, L + ncol, ...
  const uint32_t ncol = c.nwc * 32;
  griddep_wait();  // x, y and the workspace may be touched by the preceding grid
  const void* xsrc = a.x;
  if (c.stage_x) {
    uint8_t* sX = sm + c.off_x;
    const uint32_t xbytes = a.T * a.n * (a.xdt == OVL_BF16 ? 2u : 4u);
    const uint8_t* gx = static_cast<const uint8_t*>(a.x);
    if (c.stage_x == 16) {
      for (uint32_t e = threadIdx.x * 16; e < xbytes; e += nthr * 16) cp_async16(sX + e, gx + e);
    } else {
      for (uint32_t e = threadIdx.x * 4; e < xbytes; e += nthr * 4) cp_async4(sX + e, gx + e);
    }
    cp_async_commit();
    cp_async_wait_all();
    xsrc = sX;
    // x staged: tell the helper warp (which reads it too) without waiting for
    // it, then make every consumer's copies visible to the others
    if (a.nl) named_bar_arrive(2, nthr + 32);
    named_bar(1, nthr);
  }

  // 1. activation records.  Single-token launches build each lane's first NREG
  //    records in registers; any further blocks (and multi-token launches) use
  //    records built cooperatively in shared memory.
  if (TT > 1 || c.bpl > static_cast<uint32_t>(NREG)) {
    prep_records<Q4>(rec, a, xsrc, c.xvec != 0, c.nb, warp, ncw, lane, mk, map_words(c.nb));
    named_bar(1, nthr);
  }
  uint4 rreg[NREG][7];
  if (TT == 1) {
#pragma unroll
    for (int k = 0; k < NREG; ++k) {
      const uint32_t b = L + k * ncol;
      if (k < static_cast<int>(c.bpl) && b < c.nb)
        lane_record<Q4>(rreg[k], xsrc, a.xdt, c.xvec != 0, static_cast<size_t>(b) * 32, mk, map_words(c.nb));
    }
  }

  // 3. stream the base rows
  bool ok = true;
  // slot = s mod ns and the barrier phase (s / ns) & 1, kept as counters
  uint32_t slot = grp, phase = 0;
  for (uint32_t s = grp; s < nst; s += c.ng) {
    if (s != grp && (slot += c.ng) >= c.ns) {
      slot -= c.ns;
      phase ^= 1u;
    }
    // warp-uniform decision: the shuffles below need every lane
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], phase))) {
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
    auto block = [&](uint32_t b, const uint4 (&r)[7], int t) {
      const float xs = __uint_as_float(r[6].x);
      if constexpr (QK4) {
        // Sub-block j = b mod 8 of a 256-weight super-block: weight
        // d*sc_j*code - dmin*m_j, so the block sum is
        // xs*(d*sc_j*sum(code*X) - dmin*m_j*sum(X)).  sum(code*X) comes from
        // zero accumulator starts; the record's starts hold -8*sum(X), so
        // xs*sum(X) is -xs/8 times their value (exact: powers of two), once
        // per block for all rows.
        const float xs0 = -0.125f * xs * limb_combine(static_cast<int>(r[6].y), static_cast<int>(r[6].z), static_cast<int>(r[6].w));
        const uint32_t j6 = 6u * (b & 7u);
        const uint8_t* hb = reinterpret_cast<const uint8_t*>(sd) + (b >> 3) * 16u;
#pragma unroll
        for (int rr = 0; rr < RG; ++rr) {
          const uint8_t* wp = sq + rr * c.rowbytes + b * kBlockBytes;
          const float P = dot_q4_zero(wp, r);                         // sum(code*X)
          const uint4 h = *reinterpret_cast<const uint4*>(hb + static_cast<size_t>(rr) * c.nb * 2);
          float dsc, dmn;
          q4k_scales(h, j6, &dsc, &dmn);
          acc[t * RG + rr] = fmaf(dsc, xs * P, acc[t * RG + rr]);
          acc[t * RG + rr] = fmaf(-dmn, xs0, acc[t * RG + rr]);
        }
      } else {
#pragma unroll
        for (int rr = 0; rr < RG; ++rr) {
          const uint8_t* wp = sq + rr * c.rowbytes + b * kBlockBytes;
          const float P = Q4 ? dot_q4(wp, r) : dot_q8(wp, r);
          const float d = __half2float(sd[rr * c.nb + b]);
          acc[t * RG + rr] = fmaf(d * xs, P, acc[t * RG + rr]);
        }
      }
    };
    if (TT == 1) {
#pragma unroll
      for (int k = 0; k < NREG; ++k) {
        const uint32_t b = L + k * ncol;
        if (k < static_cast<int>(c.bpl) && b < c.nb) block(b, rreg[k], 0);
      }
    }
    for (uint32_t k = (TT == 1 ? static_cast<uint32_t>(NREG) : 0u); k < c.bpl; ++k) {
      const uint32_t b = L + k * ncol;
      if (b < c.nb) {
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (t < static_cast<int>(a.T)) {
            const uint4* rp = reinterpret_cast<const uint4*>(rec + static_cast<size_t>(t * c.nb + b) * kRecBytes);
            uint4 r[7];
#pragma unroll
            for (int i = 0; i < 7; ++i) r[i] = rp[i];
            block(b, r, t);
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
      if (lr < nrows && t < a.T) red[(cw * TT + t) * c.rows_max + lr] = tot;
    }
  }
  // Every base stage has been consumed (so the B stage's barrier is on the
  // phase of the B copy itself).
  named_bar(1, nthr);
  const bool b_staged = (c.b_ring || c.b_areg) && sg.k1 > sg.k0;
  const uint8_t* sBst = c.b_areg ? sm + c.off_a : stages + static_cast<size_t>(nst % c.ns) * c.stage_bytes;
  const uint32_t nterm = sg.k1 - sg.k0;
  // Common single-token case: at most one output per thread and at most one
  // term of rank <= 16 with its B rows staged.  Every shared-memory read that
  // does not need v is issued before the waits below, and the B and v reads
  // after them go out in one round: a chain of dependent shared-memory rounds
  // is what an epilogue costs at the end of a memory-bound launch.
  const uint32_t r0f = nterm ? ep[0].r : 0u;
  const bool fast = TT == 1 && nrows <= nthr && !a.tok_sel && nterm <= 1 && r0f <= 16 && (nterm == 0 || b_staged);
  float rv[kMaxThreads / 32];
  EpTerm e0{};
  uint32_t rot0 = 0;
  // A stage that never arrived (the producer or a consumer warp gave up) left
  // rows of this CTA without their base sums: the flag was set before the
  // barrier above, so it is read here, off the critical path.
  if (*abort_flag) ok = false;
  const bool any_marked = mk[0] != 0u;
  float corr = 0.f;   // fast path: the marked blocks' residual products (before the waits)
  if (fast) {
    const uint32_t lr = threadIdx.x;
#pragma unroll
    for (int w = 0; w < kMaxThreads / 32; ++w)
      rv[w] = (lr < nrows && w < static_cast<int>(c.nwc)) ? red[w * c.rows_max + lr] : 0.f;
    if (nterm) {
      e0 = ep[0];
      rot0 = lr % e0.r;
    }
    if (any_marked && lr < nrows) corr = marked_sum<QUANT>(mk, a, c, sg, 0, row0 + lr, xsrc);
  }
  // 4. the low-rank vector from the helper warp and the B rows from the
  //    producer (bounded waits)
  if (a.nl && !mbar_wait_bounded(vbar, 0)) {
    latch(a.ws.status, kDevTimeoutShrink);
    ok = false;
  }
  if (ok && c.b_ring && b_staged && !mbar_wait_bounded(&full[nst % c.ns], (nst / c.ns) & 1)) {
    latch(a.ws.status, kDevTimeoutFull);
    ok = false;
  }

  // 5. epilogue, one output per thread: y = base + sum_k s_k (B_k v_k).  If
  //    any bounded wait of this CTA gave up (the status word holds the code),
  //    its outputs are written as NaN rather than left stale or partial.
  if (!ok) {
    for (uint32_t i = threadIdx.x; i < a.T * nrows; i += nthr) {
      const uint32_t t = i / nrows, lr = i - t * nrows;
      sg.y[static_cast<size_t>(t) * sg.m + row0 + lr] = __uint_as_float(0x7FC00000u);
    }
    return;
  }
  if (fast) {
    const uint32_t lr = threadIdx.x;
    if (lr >= nrows) return;
    float yv = 0.f;
#pragma unroll
    for (int w = 0; w < kMaxThreads / 32; ++w)
      if (w < static_cast<int>(c.nwc)) yv += rv[w];
    yv += corr;
    if (nterm) {
      const uint32_t r = e0.r;
      const float* Brow = reinterpret_cast<const float*>(sBst + e0.here) + lr * r;
      const float* vv = vsm + sg.rb0;
      float b16[16], v16[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        uint32_t j = u + rot0;
        j = j >= r ? j - r : j;
        b16[u] = static_cast<uint32_t>(u) < r ? Brow[j] : 0.f;
        v16[u] = static_cast<uint32_t>(u) < r ? vv[j] : 0.f;
      }
      float dot = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if (static_cast<uint32_t>(u) < r) dot = fmaf(b16[u], v16[u], dot);
      yv = fmaf(e0.s, dot, yv);
    }
    sg.y[row0 + lr] = yv;
    return;
  }
  for (uint32_t i = threadIdx.x; i < a.T * nrows; i += nthr) {
    const uint32_t t = i / nrows, lr = i - t * nrows;
    const uint32_t row = row0 + lr;
    float yv = 0.f;
    for (uint32_t w = 0; w < c.nwc; ++w) yv += red[(w * TT + t) * c.rows_max + lr];
    if (any_marked) yv += marked_sum<QUANT>(mk, a, c, sg, t, row, xsrc);
    uint32_t rbase = sg.rb0;   // global rank offset of the term
    for (uint32_t k = sg.k0; k < sg.k1; ++k) {
      const EpTerm e = ep[k - sg.k0];
      const uint32_t r = e.r;
      if (a.tok_sel && a.tok_term[t] != static_cast<int>(k)) {   // segmented: one term per token
        rbase += r;
        continue;
      }
      const float* Brow = b_staged ? reinterpret_cast<const float*>(sBst + e.here) + lr * r
                                   : e.B + static_cast<size_t>(row) * r;
      const float* vv = vsm + t * a.rtot + rbase;
      // Each row starts its dot product at a rotation of its own (lr mod r), so
      // the lanes of a warp, whose B rows are r words apart, read different
      // shared-memory banks.  The order is fixed per row: deterministic.
      const uint32_t rot = lr % r;
      float dot = 0.f;
      for (uint32_t tau = 0; tau < r; tau += 8) {   // eight loads in flight, summed in order
        float b8[8], v8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t j = tau + u + rot;
          j = j >= r ? j - r : j;
          b8[u] = (tau + u < r) ? Brow[j] : 0.f;
          v8[u] = (tau + u < r) ? vv[j] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (tau + u < r) dot = fmaf(b8[u], v8[u], dot);
      }
      yv = fmaf(e.s, dot, yv);
      rbase += r;
    }
    sg.y[static_cast<size_t>(t) * sg.m + row] = yv;
  }
}

// Single-token launches whose shrink chunks would be at least this many factor
// elements per CTA take the separate shrink launch.
constexpr uint64_t kShrinkVChunk = 2048;

using KernelFn = void (*)(const DualArgs, const DualCfg);

KernelFn pick(uint32_t quant, int tt, int rg, bool vx) {
  if (vx) {
#define OVL_KV(Q, R_) \
  if (quant == Q && tt == 1 && rg == R_) return k_dualpath<Q, 1, R_, true>;
    OVL_KV(OVL_Q8_0, 2) OVL_KV(OVL_Q8_0, 4) OVL_KV(OVL_Q8_0, 8)
    OVL_KV(OVL_Q4_0, 2) OVL_KV(OVL_Q4_0, 4) OVL_KV(OVL_Q4_0, 8)
    OVL_KV(OVL_Q4_K, 2) OVL_KV(OVL_Q4_K, 4) OVL_KV(OVL_Q4_K, 8)
#undef OVL_KV
    return nullptr;
  }
#define OVL_K(Q, T_, R_) \
  if (quant == Q && tt == T_ && rg == R_) return k_dualpath<Q, T_, R_>;
  OVL_K(OVL_Q8_0, 1, 2) OVL_K(OVL_Q8_0, 1, 4) OVL_K(OVL_Q8_0, 1, 8)
  OVL_K(OVL_Q8_0, 2, 2) OVL_K(OVL_Q8_0, 4, 2) OVL_K(OVL_Q8_0, 8, 2)
  OVL_K(OVL_Q4_0, 1, 2) OVL_K(OVL_Q4_0, 1, 4) OVL_K(OVL_Q4_0, 1, 8)
  OVL_K(OVL_Q4_0, 2, 2) OVL_K(OVL_Q4_0, 4, 2) OVL_K(OVL_Q4_0, 8, 2)
  OVL_K(OVL_Q4_K, 1, 2) OVL_K(OVL_Q4_K, 1, 4) OVL_K(OVL_Q4_K, 1, 8)
  OVL_K(OVL_Q4_K, 2, 2) OVL_K(OVL_Q4_K, 4, 2) OVL_K(OVL_Q4_K, 8, 2)
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

// Shared-memory plan for one launch; returns false if it cannot fit.  The
// soft budget (150 KB) sizes the ring: 8 stages of 4 rows for d_in = 4096,
// 4 stages of 2 rows for d_in = 14336 (q8_0).  Deeper rings (10 and 6 stages)
// and mixed plans where only some consecutive launches fit side by side on
// an SM measured slower.
constexpr uint32_t kSoftBudget = OVL_K1_SOFT_BYTES;

bool plan(DualCfg& c, const DualArgs& a, int tt, int rg, uint32_t rows_max, uint32_t b_need) {
  c.rows_max = rows_max;
  uint32_t off = round_up(2 * kMaxNS * 8 + 8 + 16, 256);   // mbarriers + abort flag
  c.off_rec = off;
  if (tt > 1 || c.bpl > reg_records_of(tt, rg)) off = round_up(off + tt * c.nb * kRecBytes, 128);
  c.off_red = off;
  off = round_up(off + c.nwc * tt * c.rows_max * 4, 128);
  c.off_v = off;
  off = round_up(off + tt * a.rtot * 4 + 4, 128);
  c.off_ep = off;
  off = round_up(off + a.nl * static_cast<uint32_t>(sizeof(EpTerm)), 128);
  c.off_mk = off;
  off = round_up(off + (1 + tt * map_words(c.nb)) * 4, 128);
  c.off_x = off;
  if (c.stage_x) off = round_up(off + tt * a.n * (a.xdt == OVL_BF16 ? 2 : 4), 128);
  c.off_a = off;
  if (c.stage_a) {
    const uint32_t chunk = static_cast<uint32_t>((static_cast<uint64_t>(a.rtot) * a.n + c.gs - 1) / std::max<uint32_t>(c.gs, 1));
    off = round_up(off + (chunk + (c.shrink_vec ? 24u : 2u)) * 4, 128);
  }
  c.off_xw = off;
  if (c.xwin) off = round_up(off + c.xwin * (a.xdt == OVL_BF16 ? 2 : 4), 128);
  else if (c.xfull) off = round_up(off + a.n * (a.xdt == OVL_BF16 ? 2 : 4), 128);
  c.stage_q = rg * c.rowbytes;
  c.stage_bytes = round_up(c.stage_q + round_up(rg * c.nb * 2, 16) + 32, 128);
  // B rows: into the A chunk + x window area after the shrink when they fit
  // there, else as one ring stage after the last base stage, else from global
  c.b_areg = a.nl && a.b_pad && b_need > 0 && b_need <= off - c.off_a;
  c.b_ring = a.nl && a.b_pad && !c.b_areg && b_need > 0 && b_need <= c.stage_bytes;
  c.off_stage = off;
  // Group g consumes the stages s = g, g+ng, ...  With ns a multiple of ng every
  // slot is consumed by one group only, in order, so a consumer is never more
  // than one barrier phase ahead of its slot (the parity wait cannot alias).
  for (uint32_t budget : {kSoftBudget, kSmemBudget}) {
    if (off + c.stage_bytes > budget) continue;
    const uint32_t max_ns = std::min<uint32_t>(kMaxNS, (budget - off) / c.stage_bytes);
    const uint32_t ng = std::min<uint32_t>(c.ng, max_ns);
    const uint32_t ns = max_ns / ng * ng;
    if (ns >= 2 * ng || budget == kSmemBudget) {
      c.ng = ng;
      c.ns = ns;
      c.smem = off + ns * c.stage_bytes;
      return true;
    }
  }
  return false;
}

}  // namespace

cudaError_t launch_dualpath(const DualArgs& a_in, cudaStream_t st) {
  if (a_in.T == 0 || a_in.m == 0) return cudaSuccess;
  DualArgs a0 = a_in;
  if (a0.nseg == 0) {
    a0.nseg = 1;
    a0.seg[0] = DualSeg{a0.qs, a0.dpl, a0.y, a0.m, 0, 0, 0, a0.nl, 0};
  }
  if (a0.nseg > static_cast<uint32_t>(kMaxMulti)) return cudaErrorInvalidValue;
  static int nsm = device_sms();
  DualCfg c{};
  c.nb = a0.n / kQK;
  c.rowbytes = a0.quant == OVL_Q8_0 ? a0.n : a0.n / 2;
  // column warps: fewest blocks per lane, then fewest idle lanes
  uint32_t best_w = 1, best_b = 0, best_waste = ~0u;
  for (uint32_t w = 1; w <= kMaxThreads / 32 - 2; ++w) {
    const uint32_t b = (c.nb + 32 * w - 1) / (32 * w);
    const uint32_t waste = b * 32 * w - c.nb;
    if (best_b == 0 || b < best_b || (b == best_b && waste < best_waste)) {
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
  int rg = 2, rg_fallback = 2;
  if (tt == 1) {
    // One kernel instance per format for single-token launches: 4 rows a
    // stage for q8_0, 8 for the 4-bit formats, whatever d_in (as long as two
    // stages fit the ring).  A decode step then runs the same kernel
    // function for every projection; a launch that follows one of another
    // function starts later (measured on the 8B-shape step, d_in 4096 and
    // 14336: 52.6 us with two instances, 49.2 us with one, although the
    // 14336-wide launch alone is slower in the larger stages).  Rows too wide for that take the
    // largest stage of at most 16 KB (q8_0) or 32 KB (4-bit) that fits.
    const uint32_t stage_target = a0.quant == OVL_Q8_0 ? OVL_K1_STAGE_BYTES : 2 * OVL_K1_STAGE_BYTES;
    while (rg < 8 && 2 * rg * c.rowbytes <= stage_target) rg *= 2;
    rg_fallback = rg;
    const int rg_uniform = a0.quant == OVL_Q8_0 ? 4 : 8;
    if (static_cast<uint64_t>(rg_uniform) * c.rowbytes <= 64 * 1024) rg = rg_uniform;
  }
  const uint32_t max_cw = kMaxThreads / 32 - 2;
  c.ng = std::max<uint32_t>(1, std::min<uint32_t>(OVL_K1_MAX_GROUPS, max_cw / c.nwc));
  const uint32_t G = std::min<uint32_t>(static_cast<uint32_t>(nsm), a0.m);
  // large factors on a single token: the shrink runs as its own launch
  const bool vx = tt == 1 && a0.nl && !a0.tok_sel && !(a0.epoch & kEpochWithhold) && a0.a16 &&
                  (reinterpret_cast<uintptr_t>(a0.x) & 15) == 0 && a0.ws.tc_scratch &&
                  a0.ws.tc_scratch_bytes >= static_cast<size_t>(a0.rtot) * 4 &&
                  static_cast<uint64_t>(a0.rtot) * a0.n >= kShrinkVChunk * G;
  KernelFn fn = pick(a0.quant, tt, rg, vx);
  if (!fn) return cudaErrorInvalidValue;
  if (G < a0.nseg) return cudaErrorInvalidValue;
  // CTAs per tensor in proportion to its rows (at least one, at most one per row)
  {
    uint32_t left = G;
    for (uint32_t i = 0; i < a0.nseg; ++i) {
      const uint32_t rest = a0.nseg - 1 - i;
      uint32_t gn = static_cast<uint32_t>((static_cast<uint64_t>(G) * a0.seg[i].m + a0.m / 2) / a0.m);
      gn = std::max<uint32_t>(1, std::min<uint32_t>(gn, a0.seg[i].m));
      gn = std::min<uint32_t>(gn, left - rest);
      if (i + 1 == a0.nseg) gn = std::min<uint32_t>(left, a0.seg[i].m);
      a0.seg[i].g0 = G - left;
      a0.seg[i].gn = gn;
      left -= gn;
    }
  }
  uint32_t G_used = 0, rows_max = 1;
  for (uint32_t i = 0; i < a0.nseg; ++i) {
    G_used += a0.seg[i].gn;
    rows_max = std::max<uint32_t>(rows_max, (a0.seg[i].m + a0.seg[i].gn - 1) / a0.seg[i].gn);
  }
  // shrink CTAs: at most one per CTA, per factor element, and per free slot
  c.gs = 0;
  if (a0.nl) {
    const uint64_t slots = a0.ws.partial_floats / 2 / (static_cast<uint64_t>(tt) * a0.rtot);
    c.gs = static_cast<uint32_t>(std::min<uint64_t>({G_used, static_cast<uint64_t>(a0.rtot) * a0.n, slots}));
    if (c.gs == 0) return cudaErrorInvalidValue;
  }
  if (vx) c.gs = 0;   // no shrink chunks, slots or gather in the dual-path launch
  c.div32 = static_cast<uint64_t>(a0.rtot) * a0.n * (static_cast<uint64_t>(c.gs) + 1) < (1ull << 32);
  if (a0.nl && static_cast<size_t>(tt) * a0.rtot * c.gs > a0.ws.partial_floats / 2) return cudaErrorInvalidValue;
  if (a0.nl && !a0.ws.epoch_counter) return cudaErrorInvalidValue;
  // operands staged in shared memory when small (immutable ones before the
  // grid dependency resolves, activations right after)
  const uint32_t esz_x = a0.xdt == OVL_BF16 ? 2 : 4;
  const uintptr_t xa = reinterpret_cast<uintptr_t>(a0.x);
  const bool x_small = static_cast<uint64_t>(tt) * a0.n * esz_x <= 32768;
  // Records built per lane in registers read x once, straight from global.
  const bool reg_only = tt == 1 && c.bpl <= reg_records_of(tt, rg);
  c.stage_x = (reg_only || !x_small) ? 0 : (xa % 16 == 0 ? 16 : (xa % 4 == 0 ? 4 : 0));
  c.xvec = c.stage_x ? 1 : (xa % 16 == 0 ? 1 : 0);
  c.stage_a = a0.nl && !vx && (static_cast<uint64_t>(a0.rtot) * a0.n / std::max<uint32_t>(c.gs, 1) + 2) * 4 <= 32768;
  // Single-token launches with x left in global memory: the helper warp stages
  // the x window of its shrink chunk (16-byte copies) when it is small.
  if (a0.nl && !vx && tt == 1 && !c.stage_x && c.xvec) {
    const uint32_t g = 16 / esz_x;
    const uint64_t chunk = (static_cast<uint64_t>(a0.rtot) * a0.n + c.gs - 1) / c.gs;
    // pieces: at most chunk + 2g elements, and at most n + g when the chunk wraps
    const uint64_t cap = std::min<uint64_t>(static_cast<uint64_t>(a0.n) + g, chunk + 2 * g);
    // one index for the A chunk and the x window: every chunk shorter than a
    // factor row (so it touches at most two), 16-byte aligned factors; other
    // launches read x from global memory (16-byte loads) in the shrink
    c.shrink_vec = cap * esz_x <= 8192 && c.stage_a && a0.a16 && chunk + g < a0.n && (chunk + 24) * 4 <= 32768;
    c.xwin = c.shrink_vec ? static_cast<uint32_t>(cap) : 0;
  }
  // Chunks over several factor rows (stacked or high-rank terms): the helper
  // stages all of x once (16-byte copies, all in flight together), so its
  // pass over the chunk reads x from shared memory instead of waiting on one
  // global load after another.
  c.xfull = 0;
  if (a0.nl && tt == 1 && !c.shrink_vec && !c.stage_x && c.xvec && c.stage_a &&
      static_cast<uint64_t>(a0.n) * esz_x <= 32768)
    c.xfull = 1;
  // Bytes of the B stage of the largest CTA slice (16-byte spans per term).
  uint32_t b_need = 0;
  for (uint32_t i = 0; a0.nl && i < a0.nseg; ++i) {
    const uint64_t rows = (a0.seg[i].m + a0.seg[i].gn - 1) / a0.seg[i].gn;
    uint64_t need = 0;
    for (uint32_t k = a0.seg[i].k0; k < a0.seg[i].k1; ++k) need += (rows * a0.lora[k].r * 4 + 15) / 16 * 16 + 16;
    b_need = static_cast<uint32_t>(std::min<uint64_t>(std::max<uint64_t>(b_need, need), 1u << 30));
  }
  if (!plan(c, a0, tt, rg, rows_max, b_need)) {
    // the uniform stage does not fit beside this launch's other buffers
    if (rg == rg_fallback) return cudaErrorInvalidConfiguration;
    rg = rg_fallback;
    fn = pick(a0.quant, tt, rg, vx);
    if (!fn || !plan(c, a0, tt, rg, rows_max, b_need)) return cudaErrorInvalidConfiguration;
  }
  if (c.ns % c.ng != 0 || c.ns > static_cast<uint32_t>(kMaxNS)) return cudaErrorInvalidConfiguration;
  const uint32_t threads = (c.nwc * c.ng + 2) * 32;   // consumers + producer + helper
  // one attribute / occupancy query per (kernel, shared-memory size)
  struct Seen { KernelFn fn; uint32_t smem; int occ; };
  static std::mutex mu;
  static Seen seen[64];
  static int nseen = 0;
  int occ = -1;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < nseen; ++i)
      if (seen[i].fn == fn && seen[i].smem == c.smem) occ = seen[i].occ;
    if (occ < 0) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
      // Always the largest shared-memory carveout: an SM configured smaller for
      // one launch would have no room for a CTA of the next, which then packs
      // two CTAs onto the SMs that drained first and leaves others idle.
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, c.smem);
      if (e != cudaSuccess) return e;
      if (nseen < 64) seen[nseen++] = {fn, c.smem, occ};
    }
  }
  if (occ < 1) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaSuccess;

  const size_t esz = a0.xdt == OVL_BF16 ? 2 : 4;
  for (uint32_t t0 = 0; t0 < a0.T; t0 += tt) {
    DualArgs a = a0;
    a.T = std::min<uint32_t>(tt, a0.T - t0);
    a.x = static_cast<const uint8_t*>(a0.x) + static_cast<size_t>(t0) * a0.n * esz;
    for (uint32_t i = 0; i < a0.nseg; ++i) a.seg[i].y = a0.seg[i].y + static_cast<size_t>(t0) * a0.seg[i].m;
    if (a0.tok_sel)
      for (uint32_t t = 0; t < 8; ++t) a.tok_term[t] = (t0 + t < a0.T) ? a0.tok_host[t0 + t] : -1;
    if (a0.nl) {
      // A fresh epoch per launch; on wrap-around clear the slots first so no
      // slot can carry a reused epoch.
      uint32_t ep = ++*a0.ws.epoch_counter;
      if (ep >= kEpochWithhold) {
        e = cudaMemsetAsync(a0.ws.partial, 0, a0.ws.partial_floats * sizeof(float), st);
        if (e != cudaSuccess) return e;
        *a0.ws.epoch_counter = 0;
        ep = ++*a0.ws.epoch_counter;
      }
      a.epoch = ep | (a0.epoch & kEpochWithhold);
    }
    if (vx) {
      // the shrink launch: the same kernel in its shrink-only mode, one CTA
      // per factor row (consecutive launches stay on one function)
      cudaLaunchConfig_t cv{};
      cv.gridDim = dim3(a.rtot);
      cv.stream = st;
      cudaLaunchAttribute av[1];
      av[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      av[0].val.programmaticStreamSerializationAllowed = 1;
      cv.attrs = av;
      cv.numAttrs = OVL_K1_PDL;
      DualCfg cvc = c;
      cvc.shrink_only = 1;
      cv.blockDim = dim3(threads);
      cv.dynamicSmemBytes = 256;   // the warps' partial sums
      e = cudaLaunchKernelEx(&cv, fn, a, cvc);
      if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(G_used);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = OVL_K1_PDL;
    e = cudaLaunchKernelEx(&cfg, fn, a, c);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ovl
