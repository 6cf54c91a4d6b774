// K4: the dual path on the tensor cores, for multi-token launches.
//
//   Y[t][i] = sum_j deq(W)[i][j] X[t][j] + sum_k s_k (B_k v_k[t])_i,   v_k[t] = A_k X[t]
//
// Sources: "Deep Technical Design: Exact, Atomic, Reversible Specialist Overlays
// on Quantized Transformer Bases" §1 (dual path: the quantized base and the
// overlay evaluated side by side, nothing merged into the stored weights), §5
// (q8_0 / q4_0: 32 weights per f16 scale), §8 (with more tokens per weight the
// layer becomes a GEMM); "We propose a content-addressed overlay system"
// report, "Native/WASM Kernel Implications" (low-rank addition: x A^T, then B).
//
// Design (sm_103a).  With T tokens each weight byte feeds T multiply-adds; past
// a few tokens the integer dot products of K1 run out of issue slots, so this
// kernel dequantizes on the way into the tensor cores instead of materializing
// the layer:
//  * one CTA per 128-row tile of W and per tile of up to 64 tokens (UMMA M = 128,
//    N = token tile rounded up to 16);
//  * producer (warp 0, one thread): every 8 K-blocks (K-block = 32 weights,
//    exactly one quantization block per row) one TMA 2-D copy of the tile's raw
//    codes for those 8 blocks (one 128 / 256-byte run per row) and one of their
//    f16 scales; per K-block the fp32 activations (128-byte swizzle);
//  * converters (warps 2..9, two per TMEM lane quarter, 16 weights of a row
//    each): d * q in fp32 (exact: 11 x 8 significant bits), stored straight
//    into tensor memory (row r in lane r, K along columns) with tcgen05.st --
//    the dequantized operand never touches shared memory;
//  * MMA issuer (warp 1, one thread): tcgen05.mma.kind::tf32 (K = 8) with A in
//    TMEM and the activations in shared memory, accumulator in TMEM;
//    tcgen05.commit frees each stage;
//  * epilogue (warps 2..5, one TMEM lane quarter each): accumulator + the
//    low-rank term from v (computed by k_shrink), stored to Y.
// TF32 keeps 10 explicit mantissa bits of d*q (|error| <= 2^-10 |w|); the
// activations (bf16, or fp32 rounded by the tensor core) likewise; fp32
// accumulation.  Every wait is bounded and latches a status code.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "ovl_internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace ovl {
namespace {

constexpr uint32_t BM = 128;              // rows of W per CTA (UMMA M)
constexpr uint32_t BK = 32;               // weights per K-block: one quantization block
constexpr uint32_t kDGroup = 8;           // K-blocks per scale tile
constexpr uint32_t kDBytes = BM * kDGroup * 2;   // one scale tile: 128 rows x 8 f16
constexpr uint32_t kMaxStages = 14;
constexpr uint32_t kSmemCap = 220 * 1024;
constexpr uint32_t kTmemCols = 512;       // accumulator at columns [0, 64), A stages at 64 + 32 s
constexpr uint32_t kAcol = 64;
constexpr uint32_t kConvWarps = 8;        // two threads per tile row
constexpr uint32_t kThreads = (2 + kConvWarps) * 32;   // producer, MMA issuer, converters
constexpr uint32_t kTimeoutFused = 5;

struct FusedArgs {
  uint32_t m, n, T, quant;
  uint32_t bn;            // UMMA N (multiple of 16, <= kTokTile)
  uint32_t ns;            // pipeline depth
  uint32_t kblocks;       // n / 32
  uint32_t qrow;          // raw code bytes per row and K-block (32 or 16)
  uint32_t b_off;         // offset of the B tile in a stage
  uint32_t gbytes;        // one code group: scales (kDBytes) then codes (BM x 8 qrow)
  uint32_t stage_bytes;
  uint32_t tmem_cols;
  uint32_t idesc;
  uint32_t lkb;           // extra K-blocks of the low-rank term (ranks in chunks of 32)
  uint32_t nl, rtot;
  float* y;
  uint32_t* status;
  LoraRef lora[OVL_MAX_TABLE];
};

// Four consecutive weights of one 32-bit word as floats, exactly: the byte goes
// into the low mantissa bits of 2^23 (one byte permute) and 2^23 + bias comes
// off again (exact); `bias` = 128 for offset-binary int8, 8 for q4 codes.
__device__ __forceinline__ float byte_value(uint32_t word, uint32_t b, float bias) {
  return __int_as_float(static_cast<int>(__byte_perm(word, 0x4B000000u, 0x7540u + b))) - (8388608.f + bias);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_fused_gemm(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmD,
                 const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmV,
                 const FusedArgs g) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  uint8_t* tiles = sm;                                   // ns x (A | B | raw codes)
  uint8_t* gring = sm + g.ns * g.stage_bytes;            // 2 code groups (scales + codes)
  uint64_t* full = reinterpret_cast<uint64_t*>(gring + 2 * g.gbytes);
  uint64_t* empty = full + kMaxStages;
  uint64_t* conv = empty + kMaxStages;
  uint64_t* dfull = conv + kMaxStages;
  uint64_t* dempty = dfull + 2;
  uint64_t* accum = dempty + 2;
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(accum + 1);

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t m0 = blockIdx.x * BM, n0 = blockIdx.y * g.bn;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_taddr)),
                 "r"(g.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (uint32_t i = 0; i < g.ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&conv[i], kConvWarps);   // one arrival per converter warp
    }
    for (uint32_t i = 0; i < 2; ++i) {
      mbar_init(&dfull[i], 1);
      mbar_init(&dempty[i], kConvWarps);
    }
    mbar_init(accum, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = *s_taddr;
  griddep_launch_dependents();

  const uint32_t ktot = g.kblocks + g.lkb;   // base K-blocks, then the low-rank ones
  // Each CTA walks the base K-blocks from its own group onwards (wrapping), so
  // the CTAs of a launch read different activation tiles at any moment
  // instead of all asking the same few L2 lines for the same tile.  d_in is a
  // multiple of 256 here: group boundaries stay aligned.  The order is fixed
  // per CTA: results are deterministic.
  const uint32_t rot = (blockIdx.x % (g.kblocks / kDGroup)) * kDGroup;
  auto kdata = [&](uint32_t kb) { return kb < g.kblocks ? (kb + rot) % g.kblocks : kb; };
  if (warp == 0 && lane == 0) {
    // ---- producer
    griddep_wait();   // the widened activations and s v come from preceding kernels
    for (uint32_t kb = 0; kb < ktot; ++kb) {
      const uint32_t st = kb % g.ns;
      const bool base = kb < g.kblocks;
      if (base && kb % kDGroup == 0) {
        const uint32_t dg = kb / kDGroup, ds = dg & 1;
        if (dg >= 2 && !mbar_wait_spin(&dempty[ds], ((dg / 2) - 1) & 1)) {
          latch_status(g.status, kTimeoutFused);
          break;
        }
        uint8_t* grp = gring + ds * g.gbytes;
        mbar_arrive_expect_tx(&dfull[ds], g.gbytes);
        const uint32_t dgd = kdata(kb) / kDGroup;   // the group's data
        tma_load_2d(grp, &tmD, static_cast<int32_t>(dgd * kDGroup), static_cast<int32_t>(m0), &dfull[ds]);
        tma_load_2d(grp + kDBytes, &tmQ, static_cast<int32_t>(dgd * kDGroup * g.qrow), static_cast<int32_t>(m0),
                    &dfull[ds]);
      }
      if (kb >= g.ns && !mbar_wait_spin(&empty[st], ((kb / g.ns) - 1) & 1)) {
        latch_status(g.status, kTimeoutFused);
        break;
      }
      uint8_t* stg = tiles + st * g.stage_bytes;
      if (base) {
        mbar_arrive_expect_tx(&full[st], g.bn * 128);
        tma_load_2d(stg + g.b_off, &tmX, 0, static_cast<int32_t>(kdata(kb) * g.T + n0), &full[st]);
      } else {
        mbar_arrive_expect_tx(&full[st], g.bn * 128);
        tma_load_2d(stg + g.b_off, &tmV, static_cast<int32_t>((kb - g.kblocks) * BK), static_cast<int32_t>(n0),
                    &full[st]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    for (uint32_t kb = 0; kb < ktot; ++kb) {
      const uint32_t st = kb % g.ns;
      if (!mbar_wait_spin(&conv[st], (kb / g.ns) & 1) || !mbar_wait_spin(&full[st], (kb / g.ns) & 1)) {
        latch_status(g.status, kTimeoutFused);
        break;
      }
      tc_fence_after();
      const uint64_t bdesc = sdesc_sw128(smem_u32(tiles + st * g.stage_bytes + g.b_off));
      const uint32_t acol = taddr + kAcol + BK * st;
#pragma unroll
      for (uint32_t k = 0; k < BK / 8; ++k)   // K = 8 tf32 per instruction: 8 TMEM columns, 32 bytes of B
        umma_tf32_ts(taddr, acol + 8 * k, bdesc + 2 * k, g.idesc, (kb | k) != 0);
      umma_commit(&empty[st]);
    }
    umma_commit(accum);
  } else if (warp >= 2) {
    // ---- converters: weights [16 h, 16 h + 16) of row r = TMEM lane r; a warp
    // may only reach its own lane quarter (warp mod 4)
    const uint32_t quarter = warp & 3u, h = (warp - 2) >> 2, r = quarter * 32 + lane;
    bool pending = false;
    uint32_t pend_st = 0;
    for (uint32_t kb = 0; kb < ktot; ++kb) {
      const uint32_t st = kb % g.ns;
      const bool base = kb < g.kblocks;
      const uint32_t dg = kb / kDGroup, ds = dg & 1;
      if (base && kb % kDGroup == 0 && !mbar_wait_spin(&dfull[ds], (dg / 2) & 1)) {
        latch_status(g.status, kTimeoutFused);
        break;
      }
      // TMEM buffer st is free once the MMAs of K-block kb - ns completed (the
      // converters never read the activation tile)
      if (kb >= g.ns && !mbar_wait_spin(&empty[st], ((kb / g.ns) - 1) & 1)) {
        latch_status(g.status, kTimeoutFused);
        break;
      }
      float w[16];
      if (base) {
        const uint8_t* grp = gring + ds * g.gbytes;
        const float d = __half2float(reinterpret_cast<const __half*>(grp)[r * kDGroup + kb % kDGroup]);
        const uint8_t* qrowp = grp + kDBytes + r * (kDGroup * g.qrow) + (kb % kDGroup) * g.qrow;
        if (g.quant == OVL_Q8_0) {
          const uint4 q = *reinterpret_cast<const uint4*>(qrowp + h * 16);
          const uint32_t words[4] = {q.x ^ 0x80808080u, q.y ^ 0x80808080u, q.z ^ 0x80808080u, q.w ^ 0x80808080u};
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int b = 0; b < 4; ++b) w[4 * i + b] = d * byte_value(words[i], b, 128.f);
        } else {
          const uint2 q = *reinterpret_cast<const uint2*>(qrowp + h * 8);
          const uint32_t words[2] = {q.x, q.y};
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint32_t lo = words[i] & 0x0F0F0F0Fu, hi = (words[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
            for (int b = 0; b < 4; ++b) {   // element 2p in the low nibble, 2p+1 in the high one
              w[8 * i + 2 * b] = d * byte_value(lo, b, 8.f);
              w[8 * i + 2 * b + 1] = d * byte_value(hi, b, 8.f);
            }
          }
        }
      } else {
        // low-rank K-block j: ranks 32 j + [16 h, 16 h + 16) of B (all terms,
        // concatenated in order), row m0 + r; zero past the ranks or the rows
        const uint32_t row = m0 + r;
        uint32_t rho = (kb - g.kblocks) * BK + 16 * h, k = 0, rb = 0;
        while (k + 1 < g.nl && rho >= rb + g.lora[k].r) rb += g.lora[k++].r;
#pragma unroll
        for (int e = 0; e < 16; ++e, ++rho) {
          while (k + 1 < g.nl && rho >= rb + g.lora[k].r) rb += g.lora[k++].r;
          w[e] = (row < g.m && rho < g.rtot) ? g.lora[k].B[static_cast<size_t>(row) * g.lora[k].r + (rho - rb)] : 0.f;
        }
      }
      __syncwarp();               // every lane is done with this group's codes and scales
      if (lane == 0 && base && (kb % kDGroup == kDGroup - 1 || kb + 1 == g.kblocks)) mbar_arrive(&dempty[ds]);
      // Software pipeline: K-block kb - 1 was stored to TMEM one iteration
      // ago; wait for that store only now (its latency overlapped this
      // conversion) and release it to the MMA issuer, then store kb.
      if (pending) {
        tmem_wait_st();
        tc_fence_before();        // the MMA issuer reads these columns after the barrier
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv[pend_st]);
      }
      uint32_t bits[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) bits[e] = __float_as_uint(w[e]);
      tmem_st16_async(taddr + ((quarter * 32u) << 16) + kAcol + BK * st + 16 * h, bits);
      pending = true;
      pend_st = st;
    }
    if (pending) {
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv[pend_st]);
    }
  }
  __syncwarp();

  // ---- epilogue (warps 2..5): TMEM lane quarter (warp mod 4) = 32 rows, column = token
  griddep_wait();   // Y may still be read by a preceding kernel
  if (warp >= 2 && warp < 6) {
    const bool ok = mbar_wait_bounded(accum, 0);
    if (!ok) latch_status(g.status, kTimeoutFused);
    tc_fence_after();
    const uint32_t quarter = warp & 3u;
    const uint32_t row = m0 + quarter * 32 + lane;
    for (uint32_t c0 = 0; c0 < g.bn; c0 += 32) {
      uint32_t acc[32];
      tmem_ld32(taddr + ((quarter * 32u) << 16) + c0, acc);
      if (!ok || row >= g.m) continue;
#pragma unroll
      for (uint32_t j = 0; j < 32; ++j) {
        const uint32_t t = n0 + c0 + j;
        if (c0 + j < g.bn && t < g.T) g.y[static_cast<size_t>(t) * g.m + row] = __uint_as_float(acc[j]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(g.tmem_cols)
                 : "memory");
  }
}

// Activations of one token chunk -> fp32 in K-block-major order:
// out[(j * T + t) * 32 + e] = x[t][32 j + e].  One K-block of every token is
// then one contiguous run (its tile is spread over many L2 slices, instead of T
// lines a row apart that every CTA asks for at once).
__global__ void __launch_bounds__(256) k_widen_kblk(const void* __restrict__ x, uint32_t xdt, uint32_t T, uint32_t n,
                                                   float* __restrict__ out) {
  griddep_launch_dependents();
  griddep_wait();
  const size_t count = static_cast<size_t>(T) * n;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint32_t e = static_cast<uint32_t>(i & 31), rest = static_cast<uint32_t>(i >> 5);
    const uint32_t t = rest % T, j = rest / T;
    const size_t src = static_cast<size_t>(t) * n + j * 32u + e;
    out[i] = xdt == OVL_BF16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(x)[src]) << 16)
                             : static_cast<const float*>(x)[src];
  }
}

// v[t][rho] = s_k A_k[rho - rb_k] . x[t] for every token and factor row (one
// warp per pair, 16-byte loads, fixed-order sums), rows padded to a multiple of
// 32 with zeros; pairs a segmented token does not use are zero as well.  The
// fused kernel multiplies these by the B rows on the tensor cores.
struct ShrinkArgs {
  const float* x;         // widened activations [T][n]
  float* v;               // [T][rpad]
  uint32_t n, T, nl, rtot, rpad, tok_sel;
  LoraRef lora[OVL_MAX_TABLE];
  int8_t tok_term[kTokTile];
};

__global__ void __launch_bounds__(256) k_shrink(const ShrinkArgs s) {
  griddep_launch_dependents();
  griddep_wait();   // the widened activations
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t pairs = s.T * s.rpad;
  for (uint32_t p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < pairs; p += (gridDim.x * blockDim.x) >> 5) {
    const uint32_t t = p / s.rpad, rho = p - t * s.rpad;
    uint32_t k = 0, rb = 0;
    while (k + 1 < s.nl && rho >= rb + s.lora[k].r) rb += s.lora[k++].r;
    float acc = 0.f;
    if (rho < s.rtot && (!s.tok_sel || s.tok_term[t] == static_cast<int>(k))) {
      const float4* a = reinterpret_cast<const float4*>(s.lora[k].A + static_cast<size_t>(rho - rb) * s.n);
      for (uint32_t j = lane; j < s.n / 4; j += 32) {
        // element 4 j of token t in the K-block-major layout
        const float4 xv = *reinterpret_cast<const float4*>(s.x + (static_cast<size_t>(j >> 3) * s.T + t) * 32 + (j & 7) * 4);
        const float4 av = a[j];
        acc = fmaf(av.x, xv.x, acc);
        acc = fmaf(av.y, xv.y, acc);
        acc = fmaf(av.z, xv.z, acc);
        acc = fmaf(av.w, xv.w, acc);
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      acc *= s.lora[k].s;
    }
    if (lane == 0) s.v[p] = acc;
  }
}

}  // namespace

bool fused_gemm_supported(uint32_t m, uint32_t n) { return m > 0 && n >= 256 && n % 256 == 0; }

size_t fused_gemm_scratch_bytes(uint32_t T, uint32_t n, uint32_t rtot) {
  const uint32_t tc = std::min<uint32_t>(T, kTokTile);
  const uint32_t rpad = (rtot + BK - 1) / BK * BK;
  return (static_cast<size_t>(tc) * n * 4 + 255) / 256 * 256 + static_cast<size_t>(tc) * rpad * 4;
}

cudaError_t launch_fused_gemm(const FusedLaunch& L, cudaStream_t st) {
  if (L.T == 0 || L.m == 0) return cudaSuccess;
  if (!fused_gemm_supported(L.m, L.n) || L.nl > OVL_MAX_TABLE) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(L.qs) & 15) || (reinterpret_cast<uintptr_t>(L.dpl) & 15) ||
      (reinterpret_cast<uintptr_t>(L.scratch) & 255) || L.scratch_bytes < fused_gemm_scratch_bytes(L.T, L.n, L.rtot))
    return cudaErrorInvalidValue;
  for (uint32_t k = 0; k < L.nl; ++k)
    if (reinterpret_cast<uintptr_t>(L.lora[k].A) & 15) return cudaErrorInvalidValue;
  const uint32_t rpad = (L.rtot + BK - 1) / BK * BK;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(k_fused_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const uint32_t qrow = L.quant == OVL_Q8_0 ? 32u : 16u;
  const uint32_t rowbytes = L.n / BK * qrow;
  CUtensorMap tmQ, tmD;
  if (!encode_map_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.qs, rowbytes, L.m, rowbytes, kDGroup * qrow, BM, false) ||
      !encode_map_2d(&tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.dpl, L.n / BK, L.m, L.n / BK * 2, kDGroup, BM, false))
    return cudaErrorInvalidValue;
  const size_t esz = L.xdt == OVL_BF16 ? 2 : 4;
  float* xf = L.scratch;
  float* v = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(L.scratch) +
                                      (static_cast<size_t>(std::min<uint32_t>(L.T, kTokTile)) * L.n * 4 + 255) / 256 * 256);
  for (uint32_t t0 = 0; t0 < L.T; t0 += kTokTile) {
    const uint32_t tc = std::min<uint32_t>(kTokTile, L.T - t0);
    const void* xc = static_cast<const uint8_t*>(L.x) + static_cast<size_t>(t0) * L.n * esz;
    cudaError_t e;
    {
      cudaLaunchConfig_t cw{};
      const size_t count = static_cast<size_t>(tc) * L.n;
      cw.gridDim = dim3(static_cast<unsigned>(std::max<size_t>(1, std::min<size_t>((count + 255) / 256, 1184))));
      cw.blockDim = dim3(256);
      cw.stream = st;
      cudaLaunchAttribute aw[1];
      aw[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      aw[0].val.programmaticStreamSerializationAllowed = 1;
      cw.attrs = aw;
      cw.numAttrs = 1;
      e = cudaLaunchKernelEx(&cw, k_widen_kblk, xc, L.xdt, tc, L.n, xf);
      if (e != cudaSuccess) return e;
    }
    FusedArgs g{};
    g.m = L.m;
    g.n = L.n;
    g.T = tc;
    g.quant = L.quant;
    g.bn = (tc + 15) / 16 * 16;
    g.kblocks = L.n / BK;
    g.qrow = qrow;
    g.b_off = 0;
    g.gbytes = kDBytes + BM * kDGroup * qrow;
    g.stage_bytes = (g.bn * 128 + 1023) / 1024 * 1024;
    g.lkb = L.nl ? rpad / BK : 0;
    g.ns = std::min<uint32_t>(kMaxStages, (kSmemCap - 1024 - 2 * g.gbytes - 512) / g.stage_bytes);
    if (g.ns < 2) return cudaErrorInvalidConfiguration;
    g.tmem_cols = kTmemCols;
    g.idesc = (1u << 4)                  // accumulator: f32
              | (2u << 7) | (2u << 10)   // A, B: tf32
              | ((g.bn >> 3) << 17)      // N
              | ((BM >> 4) << 24);       // M
    g.nl = L.nl;
    g.rtot = L.rtot;
    g.y = L.y + static_cast<size_t>(t0) * L.m;
    g.status = L.status;
    for (uint32_t k = 0; k < L.nl; ++k) g.lora[k] = L.lora[k];
    int8_t tok_term[kTokTile];
    for (uint32_t t = 0; t < kTokTile; ++t) tok_term[t] = (L.tok_sel && t < tc) ? L.tok_host[t0 + t] : -1;
    CUtensorMap tmX, tmV;
    // K-block-major activations: row j * tc + t holds x[t][32 j .. 32 j + 32)
    if (!encode_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, xf, BK, static_cast<uint64_t>(g.kblocks) * tc, BK * 4,
                       BK, g.bn, true))
      return cudaErrorInvalidValue;
    if (L.nl) {
      if (!encode_map_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, v, rpad, tc, static_cast<uint64_t>(rpad) * 4, BK, g.bn,
                         true))
        return cudaErrorInvalidValue;
    } else {
      tmV = tmX;   // no low-rank K-blocks: never read
    }
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    if (L.nl) {
      ShrinkArgs s{};
      s.x = xf;
      s.v = v;
      s.n = L.n;
      s.T = tc;
      s.nl = L.nl;
      s.rtot = L.rtot;
      s.rpad = rpad;
      s.tok_sel = L.tok_sel;
      for (uint32_t k = 0; k < L.nl; ++k) s.lora[k] = L.lora[k];
      for (uint32_t t = 0; t < kTokTile; ++t) s.tok_term[t] = tok_term[t];
      cudaLaunchConfig_t cs{};
      const uint32_t warps = tc * rpad;
      cs.gridDim = dim3(std::max<uint32_t>(1, std::min<uint32_t>((warps + 7) / 8, 1184)));
      cs.blockDim = dim3(256);
      cs.stream = st;
      cs.attrs = at;
      cs.numAttrs = 1;
      e = cudaLaunchKernelEx(&cs, k_shrink, s);
      if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((L.m + BM - 1) / BM, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = g.ns * g.stage_bytes + 2 * g.gbytes + 512 + 1024;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_fused_gemm, tmQ, tmD, tmX, tmV, g);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ovl
