// K3: prefill GEMM of the per-layer JIT path on the 5th-generation tensor cores.
//
//   Y[T][m] = X[T][n] * S[m][n]^T      (S = the fp32 materialized layer)
//
// Sources: "Deep Technical Design: Exact, Atomic, Reversible Specialist Overlays
// on Quantized Transformer Bases" §8 (Prefill vs Decode: during prefill the
// batch dimension equals the sequence length and dense GEMM favours per-layer
// JIT materialization, amortized over the tokens), §1 (the materialized layer
// is passed through the linear layer, then discarded).
//
// Design (sm_103a): one CTA per 128-row tile of S and per N-tile of tokens.
// TMA (2-D tensor maps, 128-byte swizzle, no multicast) streams K-blocks of 32
// fp32 values (one 128-byte swizzle row) of S and of the widened activations
// into an mbarrier ring; one thread issues tcgen05.mma.kind::tf32 (M=128,
// N=BN, K=8) with the accumulator in TMEM; tcgen05.commit releases each stage;
// four warps read the accumulator back with tcgen05.ld and store Y.  TF32
// keeps 10 explicit mantissa bits of S (the bf16 activations are exact in
// TF32); fp32 accumulation.  Every wait is bounded and latches a status code.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "ovl_internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace ovl {
namespace {

constexpr uint32_t BM = 128;          // rows of S per CTA (UMMA M)
constexpr uint32_t BK = 32;           // fp32 K elements per stage (128 bytes)
constexpr uint32_t kMaxStages = 8;
constexpr uint32_t kSmemCap = 220 * 1024;
constexpr uint32_t kTimeoutGemm = 4;

struct GemmArgs {
  uint32_t m, n, T;
  uint32_t bn;            // UMMA N (multiple of 16, <= 256)
  uint32_t ns;            // pipeline depth
  uint32_t kblocks;       // n / 32
  uint32_t b_bytes;       // bytes of one B tile (bn rows x 128 B)
  uint32_t stage_bytes;   // A tile + B tile
  uint32_t tmem_cols;     // power of two >= bn
  uint32_t idesc;         // instruction descriptor
  float* y;
  uint32_t* status;
};

__global__ void __launch_bounds__(128, 1)
    k_jit_gemm(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmX, const GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  // tiles on a 1024-byte boundary (the swizzle atom); one spare KiB is allocated
  uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  uint8_t* tiles = sm;                                                    // ns x (A tile | B tile)
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + g.ns * g.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  uint64_t* accum = empty + kMaxStages;
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
    }
    mbar_init(accum, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = *s_taddr;
  griddep_launch_dependents();

  if (warp == 0 && lane == 0) {
    // ---- TMA producer
    griddep_wait();   // S and the widened activations come from preceding kernels
    for (uint32_t kb = 0; kb < g.kblocks; ++kb) {
      const uint32_t st = kb % g.ns;
      if (kb >= g.ns && !mbar_wait_bounded(&empty[st], ((kb / g.ns) - 1) & 1)) {
        latch_status(g.status, kTimeoutGemm);
        break;
      }
      uint8_t* a = tiles + st * g.stage_bytes;
      mbar_arrive_expect_tx(&full[st], BM * 128 + g.b_bytes);
      tma_load_2d(a, &tmS, static_cast<int32_t>(kb * BK), static_cast<int32_t>(m0), &full[st]);
      tma_load_2d(a + BM * 128, &tmX, static_cast<int32_t>(kb * BK), static_cast<int32_t>(n0), &full[st]);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: one thread drives the tensor cores
    for (uint32_t kb = 0; kb < g.kblocks; ++kb) {
      const uint32_t st = kb % g.ns;
      if (!mbar_wait_bounded(&full[st], (kb / g.ns) & 1)) {
        latch_status(g.status, kTimeoutGemm);
        break;
      }
      tc_fence_after();
      const uint32_t a = smem_u32(tiles + st * g.stage_bytes);
      const uint64_t adesc = sdesc_sw128(a), bdesc = sdesc_sw128(a + BM * 128);
#pragma unroll
      for (uint32_t k = 0; k < BK / 8; ++k)   // K = 8 tf32 = 32 bytes per instruction
        umma_tf32(taddr, adesc + 2 * k, bdesc + 2 * k, g.idesc, (kb | k) != 0);
      umma_commit(&empty[st]);                 // stage free once these MMAs have read it
    }
    umma_commit(accum);                        // accumulator complete
  }
  __syncwarp();

  // ---- epilogue: TMEM -> registers -> Y (row = lane of TMEM, column = token)
  griddep_wait();   // Y may still be read by a preceding kernel
  const bool ok = mbar_wait_bounded(accum, 0);
  if (!ok) latch_status(g.status, kTimeoutGemm);
  tc_fence_after();
  const uint32_t row = m0 + warp * 32 + lane;
  for (uint32_t c0 = 0; c0 < g.bn; c0 += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + ((warp * 32u) << 16) + c0, r);
    if (ok && row < g.m) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t t = n0 + c0 + j;
        if (t < g.T && c0 + j < g.bn) g.y[static_cast<size_t>(t) * g.m + row] = __uint_as_float(r[j]);
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

// X (bf16 or fp32) -> fp32 rows [T][n] for the tensor-map operand.
__global__ void k_widen(const void* __restrict__ x, uint32_t xdt, size_t count, float* __restrict__ out) {
  griddep_wait();
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    out[i] = xdt == OVL_BF16
                 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(x)[i]) << 16)
                 : static_cast<const float*>(x)[i];
  }
  griddep_launch_dependents();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D fp32 tensor map: rows x cols (cols contiguous), box = box_rows x 32 cols,
// 128-byte swizzle, out-of-range elements read as zero.
bool make_map(CUtensorMap* map, const float* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * sizeof(float)};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                   uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_map_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                   const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3], bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t str[2] = {strides_bytes[0], strides_bytes[1]};
  const cuuint32_t b[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dt, 3, const_cast<void*>(base), d, str, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_widen(const void* x, uint32_t xdt, size_t count, float* out, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(std::max<size_t>(1, std::min<size_t>((count + 255) / 256, 1024))));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_widen, x, xdt, count, out);
}

size_t jit_gemm_x_scratch_bytes(uint32_t T, uint32_t n) { return static_cast<size_t>(T) * n * 4; }

cudaError_t launch_jit_gemm(const float* S, const void* x, uint32_t xdt, uint32_t T, uint32_t m, uint32_t n, float* y,
                            float* xf32, const Workspace& ws, cudaStream_t st) {
  if (T == 0 || m == 0) return cudaSuccess;
  if (n % BK != 0 || (reinterpret_cast<uintptr_t>(S) & 15) || (reinterpret_cast<uintptr_t>(xf32) & 15))
    return cudaErrorInvalidValue;
  // 1. widen the activations into the scratch tail
  {
    cudaLaunchConfig_t cfg{};
    const size_t count = static_cast<size_t>(T) * n;
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<size_t>((count + 255) / 256, 1024)));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_widen, x, xdt, count, xf32);
    if (e != cudaSuccess) return e;
  }
  // 2. GEMM
  GemmArgs g{};
  g.m = m;
  g.n = n;
  g.T = T;
  g.bn = std::min<uint32_t>(256, (T + 15) / 16 * 16);
  g.kblocks = n / BK;
  g.b_bytes = g.bn * 128;
  g.stage_bytes = BM * 128 + g.b_bytes;
  g.ns = std::min<uint32_t>(kMaxStages, (kSmemCap - 2048) / g.stage_bytes);
  if (g.ns < 2) return cudaErrorInvalidConfiguration;
  g.tmem_cols = 32;
  while (g.tmem_cols < g.bn) g.tmem_cols *= 2;
  g.idesc = (1u << 4)                  // accumulator: f32
            | (2u << 7) | (2u << 10)   // A, B: tf32
            | ((g.bn >> 3) << 17)      // N
            | ((BM >> 4) << 24);       // M
  g.y = y;
  g.status = ws.status;
  CUtensorMap tmS, tmX;
  if (!make_map(&tmS, S, m, n, BM) || !make_map(&tmX, xf32, T, n, g.bn)) return cudaErrorInvalidValue;
  const uint32_t smem = g.ns * g.stage_bytes + 2048;   // tiles + alignment slack + barriers
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(k_jit_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((m + BM - 1) / BM, (T + g.bn - 1) / g.bn);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_jit_gemm, tmS, tmX, g);
}

}  // namespace ovl
