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
//    N = token tile rounded up to 16); a pipeline stage is 4 K-blocks (128
//    weights; a K-block is one quantization block);
//  * code-group producer (one thread, own warp): every 8 K-blocks one TMA copy
//    of the tile's raw codes (128-byte swizzle, so the 32 rows a converter warp
//    reads hit different banks) and one of their f16 scales, several groups
//    ahead; the weights are immutable, so it starts before the kernels that
//    produce the activations have finished;
//  * activation producer (warp 0, one thread): one 3-D TMA box per stage, the
//    4 K-blocks' fp32 activation tiles (128-byte swizzle);
//  * converters (16 warps, four per TMEM lane quarter, one K-block each):
//    d (q - bias) in fp32, exactly (one byte permute and one FMA per weight),
//    stored straight into tensor memory (row r in lane r, K along columns) --
//    the dequantized operand never touches shared memory;
//  * MMA issuers (four threads, one warp each): a thread can issue a
//    tcgen05.mma only every ~110 cycles, while an M = 128, N = 64, K = 8 tf32
//    MMA keeps the tensor core busy for ~37, so issuer w takes K-block w of
//    every stage into its own accumulator; tcgen05.commit frees each stage;
//  * epilogue (four converter warps, one TMEM lane quarter each): the
//    accumulators summed in a fixed order, stored to Y.  The low-rank term runs
//    as extra K-blocks (A = the B factors' rows, B = s v from k_widen_shrink).
// TF32 keeps 10 explicit mantissa bits of d (q - bias) (|error| <= 2^-10 |w|);
// the activations (bf16, or fp32 rounded by the tensor core) likewise; fp32
// accumulation.  Every wait is bounded and latches a status code.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "ovl_internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace ovl {
namespace {

constexpr uint32_t BM = 128;              // rows of W per CTA (UMMA M)
constexpr uint32_t BK = 32;               // weights per K-block: one quantization block
constexpr uint32_t kSub = 4;              // K-blocks per pipeline stage (128 weights)
constexpr uint32_t kStageCols = kSub * BK;   // TMEM columns of one stage's weight operand
constexpr uint32_t kDGroup = 8;           // K-blocks per code group (two stages)
constexpr uint32_t kDBytes = BM * kDGroup * 2;   // one scale tile: 128 rows x 8 f16
// One thread can issue a tcgen05.mma only every ~110 cycles, while an M = 128,
// N = 64, K = 8 tf32 MMA takes the tensor core ~37: several issuing threads,
// each with its own accumulator over its own share of K, keep it busy.  With
// 128-token chunks (N = 128, ~74 cycles an MMA) two issuers suffice, and each
// dequantized weight feeds twice the multiply-adds.
constexpr uint32_t kIssuers = 4;          // MMA-issuing warps (lane 0 of warps 1 .. kIssuers); a launch uses nis
constexpr uint32_t kWideTile = 128;       // token chunk of the two-issuer form
constexpr uint32_t kTmemCols = 512;       // accumulators (bn columns each), then the stages' weight operands
constexpr uint32_t kMaxStages = 3;
constexpr uint32_t kMaxGroups = 4;
constexpr uint32_t kSmemCap = 220 * 1024;
constexpr uint32_t kConvWarps = 16;       // four per TMEM lane quarter: one K-block of a stage each
constexpr uint32_t kConv0 = 1 + kIssuers;   // first converter warp
constexpr uint32_t kGroupWarp = kConv0 + kConvWarps;   // code-group producer
constexpr uint32_t kThreads = (kGroupWarp + 1) * 32;   // producer, MMA issuers, converters, group producer
constexpr uint32_t kTimeoutFused = 5;
static_assert(kSub % kIssuers == 0, "stage split");
static_assert(kIssuers * kTokTile + 2 * kStageCols <= kTmemCols, "TMEM budget: two stages at the widest token tile");
static_assert(2 * kWideTile + 2 * kStageCols <= kTmemCols, "TMEM budget: two stages, two issuers at 128 tokens");

constexpr uint32_t kMaxFusedTensors = 4;   // tensors sharing x in one launch (q+k+v, gate+up)

// One tensor of a launch: its row tiles are [tile0, tile0 + ceil(m / BM)) of
// the launch's tiles; its terms lora[term0 .. term0 + nl); its s v columns are
// chunks [vchunk0, vchunk0 + lkb) of 32 of the launch's v.
struct FusedTensorArgs {
  uint32_t m, tile0, lkb, rtot, nl, term0, vchunk0;
  float* y;                 // [T][m]
};

// Tensor maps of a launch (kernel parameter, so the TMA unit reads them from
// the parameter space): codes and scales per tensor, activations, s v.
struct FusedMaps {
  CUtensorMap q[kMaxFusedTensors];
  CUtensorMap d[kMaxFusedTensors];
  CUtensorMap x, v;
};

struct FusedArgs {
  uint32_t nt;              // tensors in this launch
  uint32_t n, T, quant;
  uint32_t bn;            // UMMA N (multiple of 16, <= kWideTile)
  uint32_t nis;           // MMA issuers: 4 (bn <= 64) or 2 (bn up to 128); each owns kSub / nis K-blocks
  uint32_t ns;            // pipeline stages (activation tiles + TMEM weight operands)
  uint32_t acol;          // first TMEM column of the weight operands: nis bn
  uint32_t ng;            // code-group buffers
  uint32_t kblocks;       // n / 32
  uint32_t splits;        // CTAs (one cluster) sharing a row tile, each with kbs K-blocks
  uint32_t kbs;           // base K-blocks per CTA: kblocks / splits, a multiple of kDGroup
  uint32_t bstages;       // base stages per CTA: kbs / kSub
  uint32_t recv_bytes;    // split-K receive buffer: BM x bn fp32 (0 without splits)
  uint32_t recv_alias;    // 1: the receive buffer lies in the activation tiles
  uint32_t qrow;          // raw code bytes per row and K-block (32 or 16)
  uint32_t gbytes;        // one code group: codes (128-byte swizzled boxes) then scales
  uint32_t xbytes;        // one activation tile: bn rows x 128 bytes
  uint32_t stage_bytes;   // kSub activation tiles (one 3-D box)
  uint32_t tmem_cols;
  uint32_t idesc;
  uint32_t* status;
  FusedTensorArgs ts[kMaxFusedTensors];
  LoraRef lora[OVL_MAX_TABLE];
};

// Byte b of a 32-bit word placed at mantissa bits 8..15 of 2^15: the float
// 2^15 + byte, in one byte permute.
__device__ __forceinline__ float magic15(uint32_t word, uint32_t b) {
  return __int_as_float(static_cast<int>(__byte_perm(word, 0x47000000u, 0x7404u | (b << 4))));
}

// Byte offset of 16-byte chunk c of row r in a tile written by TMA with the
// 128-byte swizzle (rows of 128 bytes; chunk c of row r lands at c ^ (r mod 8)).
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

// One K-block (32 weights) of row r, dequantized to d (q - bias) in fp32,
// exactly: with f = 2^15 + q, fma(f, d, -d (2^15 + bias)) is d (q - bias)
// rounded once, and both d (2^15 + bias) (at most 11 + 13 significant bits)
// and d (q - bias) (at most 11 + 8) are representable.  `codes` is the group's
// code area, `kbg` the K-block within the group.
__device__ __forceinline__ void dequant_kblock(const uint8_t* codes, uint32_t quant, uint32_t r, uint32_t kbg, float d,
                                               uint32_t (&bits)[32]) {
  if (quant == OVL_Q8_0) {
    // two boxes of 4 K-blocks; a K-block is two chunks; int8 made offset-binary
    // (bias 128) by flipping the sign bits
    const float c = -d * (32768.f + 128.f);
    const uint8_t* box = codes + (kbg >> 2) * (BM * 128u);
    const uint32_t ch = 2u * (kbg & 3u);
    const uint4 q0 = *reinterpret_cast<const uint4*>(box + sw128_off(r, ch));
    const uint4 q1 = *reinterpret_cast<const uint4*>(box + sw128_off(r, ch + 1));
    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t u = words[i] ^ 0x80808080u;
#pragma unroll
      for (int b = 0; b < 4; ++b) bits[4 * i + b] = __float_as_uint(fmaf(magic15(u, b), d, c));
    }
  } else {
    // one box of 8 K-blocks; a K-block is one chunk, byte p holding elements
    // 2p (low nibble) and 2p + 1 (high nibble); bias 8
    const float c = -d * (32768.f + 8.f);
    const uint4 q = *reinterpret_cast<const uint4*>(codes + sw128_off(r, kbg));
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = words[i] & 0x0F0F0F0Fu, hi = (words[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        bits[8 * i + 2 * b] = __float_as_uint(fmaf(magic15(lo, b), d, c));
        bits[8 * i + 2 * b + 1] = __float_as_uint(fmaf(magic15(hi, b), d, c));
      }
    }
  }
}

// q4_K: sub-block kbg of the group's super-block, weight d sc code - dmin m,
// rounded once: the code is formed exactly (2^15 + code, minus 2^15) and one
// fused multiply-add applies the scale and the minimum.  `hdr` is the row's
// 16-byte super-block header (the group starts on a super-block boundary).
__device__ __forceinline__ void dequant_kblock_q4k(const uint8_t* codes, const uint8_t* hdr, uint32_t r, uint32_t kbg,
                                                   uint32_t (&bits)[32]) {
  const uint4 h4 = *reinterpret_cast<const uint4*>(hdr);
  const uint32_t j6 = 6u * kbg;
  const uint64_t scf = (static_cast<uint64_t>(h4.z & 0xFFFFu) << 32) | h4.y;
  const uint64_t mnf = (static_cast<uint64_t>(h4.w) << 16) | (h4.z >> 16);
  const float dsc = __half2float(__ushort_as_half(static_cast<unsigned short>(h4.x & 0xFFFFu))) *
                    static_cast<float>(static_cast<uint32_t>(scf >> j6) & 63u);
  const float ndm = -(__half2float(__ushort_as_half(static_cast<unsigned short>(h4.x >> 16))) *
                      static_cast<float>(static_cast<uint32_t>(mnf >> j6) & 63u));
  const uint4 q = *reinterpret_cast<const uint4*>(codes + sw128_off(r, kbg));
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = words[i] & 0x0F0F0F0Fu, hi = (words[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      bits[8 * i + 2 * b] = __float_as_uint(fmaf(magic15(lo, b) - 32768.f, dsc, ndm));
      bits[8 * i + 2 * b + 1] = __float_as_uint(fmaf(magic15(hi, b) - 32768.f, dsc, ndm));
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    k_fused_gemm(const __grid_constant__ FusedMaps maps, const __grid_constant__ FusedArgs g) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  uint8_t* tiles = sm;                                   // ns x kSub activation tiles
  uint8_t* gring = sm + g.ns * g.stage_bytes;            // ng code groups (codes, then scales)
  // split-K partials of the rows this CTA owns: their own area, or (recv_alias)
  // the activation tiles, which are free once every CTA of the cluster is past
  // its last MMA
  float* recv = reinterpret_cast<float*>(g.recv_alias ? tiles : gring + g.ng * g.gbytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(gring + g.ng * g.gbytes + (g.recv_alias ? 0u : g.recv_bytes));
  uint64_t* empty = full + kMaxStages;
  uint64_t* conv = empty + kMaxStages;     // [issuer][stage]
  uint64_t* dfull = conv + kIssuers * kMaxStages;
  uint64_t* dempty = dfull + kMaxGroups;
  uint64_t* accum = dempty + kMaxGroups;
  uint64_t* red = accum + 1;               // split-K: the owners' partials have arrived
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(red + 1);

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // split-K: the CTAs of a cluster share the row tile, CTA `split` (its rank in
  // the cluster) taking base K-blocks [split kbs, (split + 1) kbs)
  const uint32_t split = g.splits > 1 ? cluster_ctarank() : 0u;
  const uint32_t tile = blockIdx.x / g.splits;
  // this CTA's tensor (the launch's tiles are the tensors' tiles in order)
  uint32_t ti = 0;
  while (ti + 1 < g.nt && tile >= g.ts[ti + 1].tile0) ++ti;
  const uint32_t tm = g.ts[ti].m, tlkb = g.ts[ti].lkb, trtot = g.ts[ti].rtot, tnl = g.ts[ti].nl;
  const uint32_t tterm0 = g.ts[ti].term0, tvc0 = g.ts[ti].vchunk0;
  float* const ty = g.ts[ti].y;
  const LoraRef* const tlora = g.lora + tterm0;
  const CUtensorMap* const tmQ = &maps.q[ti];
  const CUtensorMap* const tmD = &maps.d[ti];
  const CUtensorMap* const tmX = &maps.x;
  const CUtensorMap* const tmV = &maps.v;
  const uint32_t m0 = (tile - g.ts[ti].tile0) * BM, n0 = blockIdx.y * g.bn, k0 = split * g.kbs;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_taddr)),
                 "r"(g.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (uint32_t i = 0; i < g.ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], g.nis);    // one commit per issuer
      for (uint32_t w = 0; w < g.nis; ++w)
        mbar_init(&conv[w * kMaxStages + i], kConvWarps / g.nis);   // the converters of its K-blocks
    }
    for (uint32_t i = 0; i < g.ng; ++i) {
      mbar_init(&dfull[i], 1);
      mbar_init(&dempty[i], kConvWarps);
    }
    mbar_init(accum, g.nis);
    mbar_init(red, 4);   // one arrival per epilogue warp (in the cluster) whose rows this CTA owns
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every CTA's barriers are initialized before any CTA of the cluster can
  // arrive on them remotely
  if (g.splits > 1) cluster_sync_all();
  const uint32_t taddr = *s_taddr;
  griddep_launch_dependents();

  // Stages: kSub K-blocks each; the base ones, then (in the cluster's last CTA)
  // the low-rank ones (the last may hold fewer K-blocks).
  const bool lowrank = split + 1 == g.splits;
  const uint32_t stot = g.bstages + (lowrank ? (tlkb + kSub - 1) / kSub : 0u);
  auto nsub = [&](uint32_t s) { return s < g.bstages ? kSub : min(kSub, tlkb - (s - g.bstages) * kSub); };
  // Each CTA walks the base K-blocks from its own group onwards (wrapping), so
  // the CTAs of a launch read different activation tiles at any moment
  // instead of all asking the same few L2 lines for the same tile.  d_in is a
  // multiple of 256 here: stages and groups stay aligned.  The order is fixed
  // per CTA: results are deterministic.
  // Slots and phase parities advance as counters (no divisions in the loops).
  const uint32_t rot = (tile % (g.kbs / kDGroup)) * kDGroup;
  if (warp == 0 && lane == 0) {
    // ---- activation producer
    prefetch_tensormap(tmX);
    prefetch_tensormap(tmV);
    griddep_wait();   // the widened activations and s v come from preceding kernels
    uint32_t st = 0, ph = 0, kd = rot;   // slot, its use parity, the stage's first K-block of data
    for (uint32_t s = 0; s < stot; ++s) {
      const bool base = s < g.bstages;
      if (s >= g.ns && !mbar_wait_spin(&empty[st], ph ^ 1u)) {
        latch_status(g.status, kTimeoutFused);
        break;
      }
      // the stage's kSub activation tiles in one box {32, bn, kSub} (token rows
      // and K-blocks past the ends read as zero)
      uint8_t* stg = tiles + st * g.stage_bytes;
      mbar_arrive_expect_tx(&full[st], g.stage_bytes);
      if (base)
        tma_load_3d(stg, tmX, 0, static_cast<int32_t>(n0), static_cast<int32_t>(k0 + kd), &full[st]);
      else
        tma_load_3d(stg, tmV, 0, static_cast<int32_t>(n0), static_cast<int32_t>(tvc0 + (s - g.bstages) * kSub),
                    &full[st]);
      kd += kSub;
      if (kd >= g.kbs) kd -= g.kbs;
      if (++st == g.ns) {
        st = 0;
        ph ^= 1u;
      }
    }
  } else if (warp == kGroupWarp && lane == 0) {
    // ---- code-group producer: raw codes and scales of two stages per group,
    // up to ng groups ahead of the converters.  The base weights are
    // immutable, so this starts before the preceding kernels have finished.
    prefetch_tensormap(tmQ);
    prefetch_tensormap(tmD);
    uint32_t ds = 0, gph = 0, kd = rot;
    for (uint32_t dg = 0; dg < g.bstages / 2; ++dg) {
      if (dg >= g.ng && !mbar_wait_bounded(&dempty[ds], gph ^ 1u)) {
        latch_status(g.status, kTimeoutFused);
        break;
      }
      uint8_t* grp = gring + ds * g.gbytes;
      mbar_arrive_expect_tx(&dfull[ds], g.gbytes);
      // the group's data starts at K-block k0 + kd, a multiple of 8
      for (uint32_t b = 0; b < g.qrow / 16; ++b)   // 128-byte boxes: q4 one, q8 two
        tma_load_2d(grp + b * (BM * 128u), tmQ, static_cast<int32_t>((k0 + kd) * g.qrow + b * 128u),
                    static_cast<int32_t>(m0), &dfull[ds]);
      tma_load_2d(grp + BM * kDGroup * g.qrow, tmD, static_cast<int32_t>(k0 + kd), static_cast<int32_t>(m0),
                  &dfull[ds]);
      kd += kDGroup;
      if (kd >= g.kbs) kd -= g.kbs;
      if (++ds == g.ng) {
        ds = 0;
        gph ^= 1u;
      }
    }
  } else if (warp >= 1 && warp <= g.nis && lane == 0) {
    // ---- MMA issuers: issuer w takes K-blocks [w kpi, (w + 1) kpi) of every
    // stage (kpi = kSub / nis) into its own accumulator (columns [w bn, (w + 1) bn))
    const uint32_t kpi = kSub / g.nis;
    const uint32_t w = warp - 1, j0 = w * kpi;
    const uint32_t dacc = taddr + w * g.bn;
    uint32_t st = 0, ph = 0;
    for (uint32_t s = 0; s < stot; ++s) {
      if (!mbar_wait_spin(&conv[w * kMaxStages + st], ph) || !mbar_wait_spin(&full[st], ph)) {
        latch_status(g.status, kTimeoutFused);
        break;
      }
      tc_fence_after();
      const uint32_t acol = taddr + g.acol + kStageCols * st;
      // K = 8 tf32 per instruction: 8 TMEM columns of A, 32 bytes of each B row
      const uint64_t b0 = sdesc_sw128(smem_u32(tiles + st * g.stage_bytes));
      const uint64_t bstep = static_cast<uint64_t>(g.xbytes >> 4);   // next tile, in descriptor address units
      if (s < g.bstages) {
        for (uint32_t i = 0; i < kpi * (BK / 8); ++i) {
          const uint32_t j = j0 + (i >> 2), kk = i & 3u;
          umma_tf32_ts(dacc, acol + BK * j + 8 * kk, b0 + j * bstep + 2u * kk, g.idesc, (s | i) != 0);
        }
      } else {
        const uint32_t nk = nsub(s);
        for (uint32_t j = j0; j < j0 + kpi && j < nk; ++j)
          for (uint32_t kk = 0; kk < BK / 8; ++kk)
            umma_tf32_ts(dacc, acol + BK * j + 8 * kk, b0 + j * bstep + 2u * kk, g.idesc, 1u);
      }
      umma_commit(&empty[st]);
      if (++st == g.ns) {
        st = 0;
        ph ^= 1u;
      }
    }
    umma_commit(accum);
  } else if (warp >= kConv0 && warp < kConv0 + kConvWarps) {
    // ---- converters: row r = TMEM lane r (a warp reaches only its own lane
    // quarter, warp mod 4); warp h of a quarter takes K-block h of each stage
    const uint32_t quarter = warp & 3u, h = (warp - kConv0) >> 2, r = quarter * 32 + lane;
    uint64_t* myconv = conv + (h / (kSub / g.nis)) * kMaxStages;
    const uint32_t lanes = taddr + ((quarter * 32u) << 16);
    uint32_t st = 0, ph = 0, ds = 0, gph = 0;   // stage slot and parity; group slot and parity
    for (uint32_t s = 0; s < stot; ++s) {
      const bool base = s < g.bstages;
      if (base && (s & 1u) == 0 && !mbar_wait_spin(&dfull[ds], gph)) {
        latch_status(g.status, kTimeoutFused);
        break;
      }
      // the weight operand of stage st is free once the MMAs of stage s - ns
      // completed (the converters never read the activation tiles)
      if (s >= g.ns && !mbar_wait_spin(&empty[st], ph ^ 1u)) {
        latch_status(g.status, kTimeoutFused);
        break;
      }
      const uint32_t col = lanes + g.acol + kStageCols * st;
      if (base) {
        const uint8_t* grp = gring + ds * g.gbytes;
        const uint32_t kbg = (s & 1u) * kSub + h;   // this warp's K-block within the group
        const uint8_t* hdr = grp + BM * kDGroup * g.qrow + r * (kDGroup * 2);   // row r's 8 scales or q4_K header
        uint32_t bits[32];
        if (g.quant == OVL_Q4_K) {
          dequant_kblock_q4k(grp, hdr, r, kbg, bits);
        } else {
          const float d = __half2float(*reinterpret_cast<const __half*>(hdr + kbg * 2));
          dequant_kblock(grp, g.quant, r, kbg, d, bits);
        }
        __syncwarp();   // every lane is done with this stage's codes and scales
        if (lane == 0 && ((s & 1u) == 1 || s + 1 == g.bstages)) mbar_arrive(&dempty[ds]);
        tmem_st32_async(col + BK * h, bits);
      } else if (h < nsub(s)) {
        // low-rank K-block h of the stage: ranks 32 c + [0, 32) of the B
        // factors (all terms, concatenated in order), row m0 + r; zero past the
        // ranks or the rows
        const uint32_t row = m0 + r;
        uint32_t rho = ((s - g.bstages) * kSub + h) * BK, k = 0, rb = 0;
        while (k + 1 < tnl && rho >= rb + tlora[k].r) rb += tlora[k++].r;
        uint32_t bits[32];
#pragma unroll
        for (int e = 0; e < 32; ++e, ++rho) {
          while (k + 1 < tnl && rho >= rb + tlora[k].r) rb += tlora[k++].r;
          bits[e] = __float_as_uint((row < tm && rho < trtot)
                                        ? tlora[k].B[static_cast<size_t>(row) * tlora[k].r + (rho - rb)]
                                        : 0.f);
        }
        tmem_st32_async(col + BK * h, bits);
      }
      // hand the stage to this K-block's issuer as soon as the store landed
      // (with two stages, deferring it would serialize conversion and MMAs)
      tmem_wait_st();
      tc_fence_before();   // the issuer reads these columns after the barrier
      __syncwarp();
      if (lane == 0) mbar_arrive(&myconv[st]);
      if (base && (s & 1u) == 1 && ++ds == g.ng) {   // the group's second stage is done
        ds = 0;
        gph ^= 1u;
      }
      if (++st == g.ns) {
        st = 0;
        ph ^= 1u;
      }
    }
  }
  __syncwarp();
  if (g.recv_alias) {
    // every CTA of the cluster past its last MMA (the tiles hold no operand
    // any more) before any partial lands in them; all waits above are bounded
    if (!mbar_wait_bounded(accum, 0)) latch_status(g.status, kTimeoutFused);
    tc_fence_after();
    cluster_sync_all();
  }

  // ---- epilogue (the first four converter warps, one per TMEM lane quarter:
  // 32 rows; column = token): the issuers' accumulators summed in a fixed order.
  // Without split-K they go to Y.  With it, row rl of the tile belongs to the
  // cluster's CTA rl / (BM / splits): every CTA sends its partial rows there
  // (distributed shared memory, slot = its own rank) and arrives on that CTA's
  // `red` barrier; the owner adds the splits' partials in rank order.
  griddep_wait();   // Y may still be read by a preceding kernel
  if (warp >= kConv0 && warp < kConv0 + 4) {
    const bool ok = mbar_wait_bounded(accum, 0);
    if (!ok) latch_status(g.status, kTimeoutFused);
    tc_fence_after();
    const uint32_t quarter = warp & 3u;
    const uint32_t rl = quarter * 32 + lane, row = m0 + rl;
    const uint32_t per = BM / g.splits;   // rows each CTA of the cluster owns
    const uint32_t own = rl / per;
    const uint32_t rs = g.bn + 4;   // recv row stride (floats): 16-byte rows, reads spread over the banks
    const uint32_t slot = (split * per + (rl - own * per)) * rs;   // in the owner's recv
    const uint32_t raddr = g.splits > 1 ? cluster_map(recv + slot, own) : 0u;
    for (uint32_t c0 = 0; c0 < g.bn; c0 += 32) {
      float sum[32];
      {
        uint32_t acc[32];
        tmem_ld32(taddr + ((quarter * 32u) << 16) + c0, acc);
#pragma unroll
        for (uint32_t j = 0; j < 32; ++j) sum[j] = __uint_as_float(acc[j]);
      }
      for (uint32_t w = 1; w < g.nis; ++w) {
        uint32_t acc[32];
        tmem_ld32(taddr + ((quarter * 32u) << 16) + w * g.bn + c0, acc);
#pragma unroll
        for (uint32_t j = 0; j < 32; ++j) sum[j] += __uint_as_float(acc[j]);
      }
      if (g.splits > 1) {
#pragma unroll
        for (uint32_t j = 0; j < 32; j += 4)
          if (c0 + j < g.bn) st_cluster_v4(raddr + (c0 + j) * 4, sum[j], sum[j + 1], sum[j + 2], sum[j + 3]);
        continue;
      }
      if (!ok || row >= tm) continue;
#pragma unroll
      for (uint32_t j = 0; j < 32; ++j) {
        const uint32_t t = n0 + c0 + j;
        if (c0 + j < g.bn && t < g.T) ty[static_cast<size_t>(t) * tm + row] = sum[j];
      }
    }
    if (g.splits > 1) {
      fence_acq_rel_cluster();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(cluster_map(red, own));
      if (own == split) {
        // this warp's rows are this CTA's: wait for all splits, add in rank order
        const bool got = mbar_wait_cluster(red, 0);
        if (!got) latch_status(g.status, kTimeoutFused);
        if (got && ok && row < tm) {
          const float* mine = recv + (rl - own * per) * rs;
          for (uint32_t c = 0; c < g.bn; c += 4) {
            float4 v = *reinterpret_cast<const float4*>(mine + c);
            for (uint32_t sp = 1; sp < g.splits; ++sp) {
              const float4 u = *reinterpret_cast<const float4*>(mine + sp * per * rs + c);
              v.x += u.x;
              v.y += u.y;
              v.z += u.z;
              v.w += u.w;
            }
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (uint32_t q = 0; q < 4; ++q) {
              const uint32_t t = n0 + c + q;
              if (t < g.T) ty[static_cast<size_t>(t) * tm + row] = vv[q];
            }
          }
        }
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

// Four activations x[idx .. idx + 4) as fp32 (idx a multiple of 4).
__device__ __forceinline__ float4 load_x4(const void* x, uint32_t xdt, size_t idx) {
  if (xdt == OVL_BF16) {
    const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + idx);
    return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u), __uint_as_float(raw.y << 16),
                       __uint_as_float(raw.y & 0xFFFF0000u));
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx);
}

// Activations of one token chunk -> fp32 in K-block-major order:
// out[(j * T + t) * 32 + e] = x[t][32 j + e].  One K-block of every token is
// then one contiguous run (its tile is spread over many L2 slices, instead of T
// lines a row apart that every CTA asks for at once).  Four elements a thread.
__global__ void __launch_bounds__(256) k_widen_kblk(const void* __restrict__ x, uint32_t xdt, uint32_t T, uint32_t n,
                                                   float* __restrict__ out) {
  griddep_launch_dependents();
  griddep_wait();
  const uint32_t count4 = T * n / 4;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < count4; i += gridDim.x * blockDim.x) {
    const uint32_t e4 = i & 7u, rest = i >> 3;
    const uint32_t t = rest % T, j = rest / T;
    *reinterpret_cast<float4*>(out + static_cast<size_t>(i) * 4) = load_x4(x, xdt, static_cast<size_t>(t) * n + j * 32u + e4 * 4);
  }
}

// The low-rank side product and the widening in one pass:
//   v[t][rho] = s_k A_k[rho - rb_k] . x[t]   (rows padded to a multiple of 32
// with zeros; pairs a segmented token does not use are zero as well), and the
// K-block-major fp32 copy of x that the fused kernel's tiles come from.
// One block per 2 factor rows x 8 tokens; warp w takes the 128-element chunks
// c = w mod W of the row, each lane 4 elements of a chunk with all 16 sums in
// registers; the sums are folded across lanes (butterfly) and then across
// warps in a fixed order: deterministic.  Each (chunk, token) of the widened
// copy is written by exactly one block.
struct ShrinkArgs {
  const void* x;          // the chunk's activations [T][n] (xdt)
  float* xw;              // widened activations, K-block-major
  float* v;               // [T][rpad]
  uint32_t xdt, n, T, nl, rtot, rpad, tok_sel;
  // the launch's terms in order, each tensor's followed by a padding term
  // (A null) up to a multiple of 32 rows; padding rows of v are zero
  LoraRef lora[OVL_MAX_TABLE + kMaxFusedTensors];
  int8_t tok_term[kWideTile];
};

constexpr uint32_t kShrinkRows = 2;     // factor rows per block
constexpr uint32_t kShrinkToks = 8;     // tokens per block
constexpr uint32_t kShrinkSums = kShrinkRows * kShrinkToks;
// W warps split K: 32 make one load round for d_in = 4096 when the grid is
// small; 8 when there are many blocks (many factor rows), most of them empty.
template <uint32_t kShrinkWarps>
__global__ void __launch_bounds__(kShrinkWarps * 32) k_widen_shrink(const ShrinkArgs a) {
  griddep_launch_dependents();
  griddep_wait();   // x may come from a preceding kernel; xw and v may still be read by one
  __shared__ float part[kShrinkWarps][kShrinkSums];
  __shared__ float ssc[kShrinkRows];
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rho0 = blockIdx.x * kShrinkRows, t0 = blockIdx.y * kShrinkToks;
  // this block's factor rows and the (token, row) pairs it computes
  const float* arow[kShrinkRows];
  float sc[kShrinkRows];
  uint32_t mask = 0;   // bit tt * kShrinkRows + i
  {
    uint32_t k = 0, rb = 0;
#pragma unroll
    for (uint32_t i = 0; i < kShrinkRows; ++i) {
      const uint32_t rho = rho0 + i;
      while (k + 1 < a.nl && rho >= rb + a.lora[k].r) rb += a.lora[k++].r;
      const bool live = rho < a.rtot && a.lora[k].A != nullptr;
      arow[i] = live ? a.lora[k].A + static_cast<size_t>(rho - rb) * a.n : nullptr;
      sc[i] = live ? a.lora[k].s : 0.f;
#pragma unroll
      for (uint32_t tt = 0; tt < kShrinkToks; ++tt) {
        const uint32_t t = t0 + tt;
        if (live && t < a.T && (!a.tok_sel || a.tok_term[t] == static_cast<int>(k))) mask |= 1u << (tt * kShrinkRows + i);
      }
    }
  }
  float acc[kShrinkSums];
#pragma unroll
  for (uint32_t i = 0; i < kShrinkSums; ++i) acc[i] = 0.f;
  const uint32_t nchunks = a.n / 128;
  for (uint32_t c = warp; c < nchunks; c += kShrinkWarps) {
    const bool widen = (c / kShrinkWarps) % gridDim.x == blockIdx.x;   // this block's share of the widened copy
    if (!mask && !widen) continue;
    const uint32_t j = c * 128 + lane * 4;
    float4 xv[kShrinkToks];
#pragma unroll
    for (uint32_t tt = 0; tt < kShrinkToks; ++tt) {
      const uint32_t t = t0 + tt;
      xv[tt] = t < a.T ? load_x4(a.x, a.xdt, static_cast<size_t>(t) * a.n + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (widen) {
#pragma unroll
      for (uint32_t tt = 0; tt < kShrinkToks; ++tt) {
        const uint32_t t = t0 + tt;
        if (t < a.T) *reinterpret_cast<float4*>(a.xw + (static_cast<size_t>(j >> 5) * a.T + t) * 32 + (j & 31)) = xv[tt];
      }
    }
    if (mask) {
#pragma unroll
      for (uint32_t i = 0; i < kShrinkRows; ++i) {
        if (!arow[i]) continue;
        const float4 av = *reinterpret_cast<const float4*>(arow[i] + j);
#pragma unroll
        for (uint32_t tt = 0; tt < kShrinkToks; ++tt) {
          float s = acc[tt * kShrinkRows + i];
          s = fmaf(av.x, xv[tt].x, s);
          s = fmaf(av.y, xv[tt].y, s);
          s = fmaf(av.z, xv[tt].z, s);
          s = fmaf(av.w, xv[tt].w, s);
          acc[tt * kShrinkRows + i] = s;
        }
      }
    }
  }
  if (!mask) {   // nothing to sum: zeros (the block still wrote its share of xw)
    if (threadIdx.x < kShrinkSums) {
      const uint32_t t = t0 + threadIdx.x / kShrinkRows, rho = rho0 + threadIdx.x % kShrinkRows;
      if (t < a.T) a.v[static_cast<size_t>(t) * a.rpad + rho] = 0.f;
    }
    return;
  }
  // fold the 16 sums across the warp: each round halves what a lane keeps;
  // lane l ends with sum l / 2 (its neighbour holds the same)
#pragma unroll
  for (uint32_t r = 0; r < 4; ++r) {
    const uint32_t off = 16u >> r, cnt = kShrinkSums >> (r + 1);
    const bool up = (lane & off) != 0;
#pragma unroll
    for (uint32_t i = 0; i < cnt; ++i) {
      const float send = up ? acc[i] : acc[i + cnt];
      const float keep = up ? acc[i + cnt] : acc[i];
      acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 1);
  if ((lane & 1) == 0) part[warp][lane >> 1] = acc[0];
  if (threadIdx.x == 0) {
#pragma unroll
    for (uint32_t i = 0; i < kShrinkRows; ++i) ssc[i] = sc[i];
  }
  __syncthreads();
  if (threadIdx.x < kShrinkSums) {
    float s = part[0][threadIdx.x];
#pragma unroll
    for (uint32_t w = 1; w < kShrinkWarps; ++w) s += part[w][threadIdx.x];
    const uint32_t tt = threadIdx.x / kShrinkRows, i = threadIdx.x % kShrinkRows, t = t0 + tt;
    if (t < a.T) a.v[static_cast<size_t>(t) * a.rpad + rho0 + i] = ((mask >> threadIdx.x) & 1) ? s * ssc[i] : 0.f;
  }
}

}  // namespace

// SMs of the current device (cached per device).
uint32_t sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (!cached[dev] && cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 152;
  return static_cast<uint32_t>(cached[dev]);
}

bool fused_gemm_supported(uint32_t m, uint32_t n) { return m > 0 && n >= 256 && n % 256 == 0; }

// Scratch of one token chunk of `tile` tokens (the widened activations, then s v).
size_t chunk_scratch_bytes(uint32_t T, uint32_t n, uint32_t vcols, uint32_t tile) {
  const uint32_t tc = std::min<uint32_t>(T, tile);
  return (static_cast<size_t>(tc) * n * 4 + 255) / 256 * 256 + static_cast<size_t>(tc) * vcols * 4;
}

size_t fused_gemm_scratch_bytes(uint32_t T, uint32_t n, uint32_t vcols) {
  return chunk_scratch_bytes(T, n, vcols, kTokTile);
}

cudaError_t launch_fused_gemm(const FusedLaunch& L, cudaStream_t st) {
  if (L.T == 0) return cudaSuccess;
  if (L.nt == 0 || L.nt > kMaxFusedTensors || (L.tok_sel && L.nt != 1)) return cudaErrorInvalidValue;
  // per tensor: its tiles, its terms in the launch's table, its s v columns
  FusedTensorArgs ta[kMaxFusedTensors] = {};
  uint32_t tiles = 0, terms = 0, vcols = 0;
  for (uint32_t i = 0; i < L.nt; ++i) {
    const FusedTensor& t = L.t[i];
    if (!fused_gemm_supported(t.m, L.n) || t.nl > OVL_MAX_TABLE || (reinterpret_cast<uintptr_t>(t.qs) & 15) ||
        (reinterpret_cast<uintptr_t>(t.dpl) & 15))
      return cudaErrorInvalidValue;
    for (uint32_t k = 0; k < t.nl; ++k)
      if (reinterpret_cast<uintptr_t>(t.lora[k].A) & 15) return cudaErrorInvalidValue;
    const uint32_t rp = t.nl ? fused_vcols(t.rtot) : 0u;
    ta[i] = FusedTensorArgs{t.m, tiles, rp / BK, t.rtot, t.nl, terms, vcols / BK, nullptr};
    tiles += (t.m + BM - 1) / BM;
    terms += t.nl;
    vcols += rp;
  }
  if (terms > OVL_MAX_TABLE || (reinterpret_cast<uintptr_t>(L.scratch) & 255) ||
      L.scratch_bytes < fused_gemm_scratch_bytes(L.T, L.n, vcols))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(k_fused_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const uint32_t qrow = L.quant == OVL_Q8_0 ? 32u : 16u;
  const uint32_t rowbytes = L.n / BK * qrow;
  FusedMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  for (uint32_t i = 0; i < L.nt; ++i) {
    // codes: 128-byte boxes (8 q4 K-blocks or 4 q8 ones) in the 128-byte
    // swizzle, so the 32 rows a converter warp reads fall in different banks
    if (!encode_map_2d(&maps.q[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, L.t[i].qs, rowbytes, L.t[i].m, rowbytes, 128, BM,
                       true) ||
        !encode_map_2d(&maps.d[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.t[i].dpl, L.n / BK, L.t[i].m, L.n / BK * 2,
                       kDGroup, BM, false))
      return cudaErrorInvalidValue;
  }
  // the shrink's table: every tensor's terms, then a padding term (no A) up to
  // its multiple of 32 rows
  ShrinkArgs s{};
  for (uint32_t i = 0; i < L.nt; ++i) {
    const FusedTensor& t = L.t[i];
    if (!t.nl) continue;
    for (uint32_t k = 0; k < t.nl; ++k) s.lora[s.nl++] = t.lora[k];
    if (fused_vcols(t.rtot) > t.rtot) s.lora[s.nl++] = LoraRef{nullptr, nullptr, fused_vcols(t.rtot) - t.rtot, 0.f};
  }
  // split-K over a cluster when the row tiles alone would leave SMs idle:
  // each CTA then walks kblocks / splits K-blocks (a whole number of code groups)
  uint32_t splits = 1;
  if (tiles * 4 <= sm_count() && L.n % (BK * kDGroup * 4) == 0)
    splits = 4;
  else if (tiles * 2 <= sm_count() && L.n % (BK * kDGroup * 2) == 0)
    splits = 2;
  // 128-token chunks (two issuers, N = 128: each dequantized weight feeds twice
  // the multiply-adds) when there are that many tokens, no per-token
  // selection, and the scratch holds a chunk; 64 otherwise.  With split-K the
  // receive buffer then shares the activation tiles.
  const uint32_t tile =
      (L.T >= kWideTile && !L.tok_sel && chunk_scratch_bytes(L.T, L.n, vcols, kWideTile) <= L.scratch_bytes)
          ? kWideTile
          : kTokTile;
  const size_t esz = L.xdt == OVL_BF16 ? 2 : 4;
  // Widening pass: as many whole token chunks as the scratch holds are
  // widened (with their s v) by one launch, then each chunk runs its fused
  // GEMM on its part of the widened copy (segmented batches: one chunk).
  uint32_t wtok = tile;
  if (!L.tok_sel)
    while (wtok + tile <= (L.T + tile - 1) / tile * tile &&
           chunk_scratch_bytes(wtok + tile, L.n, vcols, wtok + tile) <= L.scratch_bytes)
      wtok += tile;
  float* xf = L.scratch;
  float* v = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(L.scratch) +
                                      (static_cast<size_t>(std::min<uint32_t>(L.T, wtok)) * L.n * 4 + 255) / 256 * 256);
  for (uint32_t w0 = 0; w0 < L.T; w0 += wtok) {
    const uint32_t wc = std::min<uint32_t>(wtok, L.T - w0);
    const void* xc = static_cast<const uint8_t*>(L.x) + static_cast<size_t>(w0) * L.n * esz;
    cudaError_t e;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    const uint32_t tc = wc;   // tokens of the widening pass
    const uint32_t t0 = w0;
    if (vcols) {
      // widened activations and s v of every tensor in one pass
      s.x = xc;
      s.xw = xf;
      s.v = v;
      s.xdt = L.xdt;
      s.n = L.n;
      s.T = tc;
      s.rtot = vcols;
      s.rpad = vcols;
      s.tok_sel = L.tok_sel;
      for (uint32_t t = 0; t < kWideTile; ++t) s.tok_term[t] = (L.tok_sel && t < tc) ? L.tok_host[t0 + t] : -1;
      cudaLaunchConfig_t cs{};
      cs.gridDim = dim3(vcols / kShrinkRows, (tc + kShrinkToks - 1) / kShrinkToks);
      const bool wide = cs.gridDim.x * cs.gridDim.y <= 2 * sm_count();
      cs.blockDim = dim3(wide ? 1024 : 256);
      cs.stream = st;
      cs.attrs = at;
      cs.numAttrs = 1;
      e = wide ? cudaLaunchKernelEx(&cs, k_widen_shrink<32>, s) : cudaLaunchKernelEx(&cs, k_widen_shrink<8>, s);
    } else {
      cudaLaunchConfig_t cw{};
      const uint32_t count4 = tc * L.n / 4;
      cw.gridDim = dim3(std::max<uint32_t>(1, std::min<uint32_t>((count4 + 255) / 256, 1184)));
      cw.blockDim = dim3(256);
      cw.stream = st;
      cw.attrs = at;
      cw.numAttrs = 1;
      e = cudaLaunchKernelEx(&cw, k_widen_kblk, xc, L.xdt, tc, L.n, xf);
    }
    if (e != cudaSuccess) return e;
    for (uint32_t c0 = 0; c0 < wc; c0 += tile) {
    const uint32_t tc = std::min<uint32_t>(tile, wc - c0);   // tokens of this fused GEMM
    const uint32_t t0 = w0 + c0;
    FusedArgs g{};
    g.nt = L.nt;
    g.n = L.n;
    g.T = tc;
    g.quant = L.quant;
    g.bn = (tc + 15) / 16 * 16;
    g.nis = g.bn > kTokTile ? 2u : kIssuers;
    g.kblocks = L.n / BK;
    g.splits = splits;
    g.kbs = g.kblocks / g.splits;
    g.bstages = g.kbs / kSub;
    g.qrow = qrow;
    g.gbytes = BM * kDGroup * qrow + kDBytes;   // multiple of 1024: every group stays swizzle-aligned
    g.xbytes = g.bn * 128;                      // multiple of 2048
    g.stage_bytes = kSub * g.xbytes;
    g.acol = g.nis * g.bn;
    g.ns = std::min<uint32_t>(kMaxStages, (kTmemCols - g.acol) / kStageCols);
    g.recv_bytes = g.splits > 1 ? BM * (g.bn + 4) * 4 : 0u;
    g.recv_alias = g.splits > 1 && g.bn > kTokTile && g.recv_bytes <= g.ns * g.stage_bytes;
    const uint32_t own_recv = g.recv_alias ? 0u : g.recv_bytes;
    const uint32_t left = kSmemCap - 1024 - 512 - g.ns * g.stage_bytes - own_recv;
    g.ng = std::min<uint32_t>(kMaxGroups, left / g.gbytes);
    if (g.ng < 2) return cudaErrorInvalidConfiguration;
    g.tmem_cols = kTmemCols;
    g.idesc = (1u << 4)                  // accumulator: f32
              | (2u << 7) | (2u << 10)   // A, B: tf32
              | ((g.bn >> 3) << 17)      // N
              | ((BM >> 4) << 24);       // M
    g.status = L.status;
    for (uint32_t i = 0; i < L.nt; ++i) {
      g.ts[i] = ta[i];
      g.ts[i].y = L.t[i].y + static_cast<size_t>(t0) * L.t[i].m;
      for (uint32_t k = 0; k < L.t[i].nl; ++k) g.lora[ta[i].term0 + k] = L.t[i].lora[k];
    }
    // K-block-major activations of the pass as {element e, token t, K-block j}:
    // x[t][32 j + e] at ((j wc + t) 32 + e); this chunk's tokens start at c0;
    // one box = kSub tiles of bn tokens
    const uint32_t box[3] = {BK, g.bn, kSub};
    {
      const uint64_t dims[3] = {BK, tc, g.kblocks};
      const uint64_t str[2] = {BK * 4, static_cast<uint64_t>(wc) * BK * 4};
      if (!encode_map_3d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, xf + static_cast<size_t>(c0) * BK, dims, str, box,
                         true))
        return cudaErrorInvalidValue;
    }
    if (vcols) {
      // s v as {rank within a chunk of 32, token, chunk}: v[t][32 c + e]
      const uint64_t dims[3] = {BK, tc, vcols / BK};
      const uint64_t str[2] = {static_cast<uint64_t>(vcols) * 4, BK * 4};
      if (!encode_map_3d(&maps.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, v + static_cast<size_t>(c0) * vcols, dims, str,
                         box, true))
        return cudaErrorInvalidValue;
    } else {
      maps.v = maps.x;   // no low-rank K-blocks: never read
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(tiles * g.splits, 1);
    cfg.blockDim = dim3(kThreads);
    // at least 120 KiB, so that two CTAs never share an SM (each holds all of
    // its SM's tensor memory)
    cfg.dynamicSmemBytes =
        std::max<uint32_t>(g.ns * g.stage_bytes + g.ng * g.gbytes + own_recv + 512 + 1024, 120 * 1024);
    cfg.stream = st;
    cudaLaunchAttribute ak[2];
    ak[0] = at[0];
    ak[1].id = cudaLaunchAttributeClusterDimension;
    ak[1].val.clusterDim.x = g.splits;
    ak[1].val.clusterDim.y = 1;
    ak[1].val.clusterDim.z = 1;
    cfg.attrs = ak;
    cfg.numAttrs = g.splits > 1 ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, k_fused_gemm, maps, g);
    if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace ovl
