// Exact-attention backward kernels for sm_103a (tcgen05 + TMEM + TMA).
//
// What is computed: the gradients of <dO, O> for O = softmax(scale Q K^T) V,
// with the probabilities rebuilt from the forward's per-row LSE rather than
// read back ("01 · 注意力为什么是 IO 瓶颈" §7: the fused method keeps only O
// and LSE for the backward and recomputes P from them). Per (b, h):
//   P  = exp(scale Q K^T - LSE)        dV = P^T dO
//   dP = dO V^T                         dS = P * (dP - D),  D_i = dO_i . O_i
//   dQ = scale dS K                     dK = scale dS^T Q
//
// Two launches on the caller's stream:
//   bwd_prep_kernel     per query row: -D and -LSE*log2(e) into a workspace
//                       whose rows are padded to a multiple of 128; padding
//                       rows get 0 and -inf, so their probabilities are zero.
//   fa_bwd_kernel       CTAs of two roles, grouped by head (a head's
//                       key-block CTAs, then its query-block CTAs, so that
//                       both roles find the head's tiles in L2):
//     key block (bwd_dkdv_cta)   one CTA per 128 key rows of one (b, h),
//                       streaming the Q/dO blocks: S^T = K Q_i^T,
//                       dP^T = V dO_i^T, P^T, dS^T, dV += P^T dO_i,
//                       dK += dS^T Q_i;
//     query block (bwd_dq_cta)   one CTA per 128 query rows of one (b, h),
//                       streaming the K/V blocks: S = Q K_j^T, dP = dO V_j^T,
//                       dS, dQ += dS K_j.
// S and dP are formed in both roles (7 tile products per pair of blocks
// instead of 5). In exchange every accumulator stays in the TMEM of the one
// CTA that owns it: no atomics, a deterministic result, and the state fits
// TMEM (512 columns): the key-block owner holds dV and dK (2 x d columns)
// plus two 128-column score regions.
//
// The two score regions R0, R1 alternate: block i's S goes to R[i&1] and its
// dP to R[(i+1)&1]. S and dP complete on barriers of their own, so that the
// elementwise warps take the exponentials of block i as soon as its S is
// done, while the tensor core still works on block i-1's gradient products
// and block i's dP; only dS = P (dP - D) is left for after dP. Once they have
// loaded dP_i, the MMA warp issues block i+1's S into R[(i+1)&1]; they write
// the packed bf16 results (P and dS, or dS alone) over S_i in R[i&1]. The
// tile products of block i that read those results, then block i+1's dP
// (into R[i&1]), follow in issue order, which the tensor core keeps.
// (In the query-block kernel, with S and dP in regions of their own, S_{j+1}
// goes in as soon as S_j has been loaded, and dP_{j+1} once dP_j has.)
//
// In the key-block kernel Q_i and dO_i share a ring slot but each has its own
// full and empty barriers. dV_i needs only P_i^T and dO_i, so it is issued
// right behind dP_i^T as soon as the elementwise warps have stored P_i^T, and
// runs while they compute dS_i^T; dK_i follows their last hand-off. S^T of
// the next block, which needs Q alone, goes in as soon as its region is free
// and Q has landed.
//
// Warp roles (10 warps, as in the forward kernel):
//   warps 0-7  elementwise step + epilogue: warp w serves TMEM lane quarter
//              w & 3 (32 rows) and the 64 streamed-block columns
//              [64 (w >> 2), 64 (w >> 2) + 64)
//   warp 8     TMA producer (one thread)
//   warp 9     TMEM allocator and MMA issuer (the whole warp, converged; one
//              elected lane issues each tcgen05 instruction)
// Packed bf16 results of warp half h live in that half's own score columns
// [64h, 64h + 32) (and dS of the key-block kernel in [64h + 32, 64h + 64)),
// so that no warp overwrites scores another warp has yet to load. For the
// tile products that read them, key step kk (16 streamed rows) sits at
// column 64 (kk >> 2) + 8 (kk & 3).
// At d = 128 the gradients leave through shared memory, which is free once
// the CTA's last products have completed: each elementwise warp writes its
// 32 rows x 64 columns in the 128-byte swizzled layout and one lane stores
// them with a tiled TMA store, instead of every thread writing its own row.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

enum : unsigned int {
  kRoleDqProducer = 4, kRoleDqMma = 5, kRoleDqSoftmax = 6,
  kRoleDkvProducer = 7, kRoleDkvMma = 8, kRoleDkvSoftmax = 9,
};

template <int HD>
struct BwdCfg {
  static constexpr int kBlk = 128;                 // rows per block, both directions
  static constexpr int kChunks = HD / 64;          // 128-byte swizzle chunks per row
  static constexpr int kChunkBytes = 128 * 128;    // 128 rows x 128 bytes
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kPairBytes = 2 * kTileBytes;            // (Q_i, dO_i) or (K_j, V_j)
  static constexpr int kStages = (HD == 128) ? 2 : 4;          // ring slots of pairs
  static constexpr int kVecBytes = 2 * 128 * 4;                // -LSE*log2e and -D of 128 rows
  static constexpr int kSmemBytes = kPairBytes + kStages * kPairBytes + kStages * kVecBytes + 1024;
  static constexpr int kThreads = 320;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t kIdescAcc = ptx::idesc_bf16_f32(128, HD, false, true);
};

struct BwdParams {
  __nv_bfloat16* dQ;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  const float* nlse2;     // [B*H][Npad]: -LSE * log2(e); -inf on padding rows
  const float* ndelta;    // [B*H][Npad]: -D; 0 on padding rows
  int N;
  int Npad;               // N rounded up to a multiple of 128
  int H;
  int n_blocks;           // Npad / 128
  int BH;                 // B * H
  float scale_log2;       // scale * log2(e)
  float scale;
  unsigned long long timeout_ns;
  int drop_load;          // test hook: index of a tile load to skip in each kernel, -1 = none
};

// ---------------------------------------------------------------- prep
// Eight padded query rows per warp: D = dO_r . O_r (float32 sum of the exact
// products of bf16 values) and LSE_r * log2(e), both stored negated. A row is
// read as 16-byte pieces, HD / 8 lanes to a row, and every piece of the
// warp's rows is requested before the first product so that each warp keeps
// 4 KB (d = 128) of loads in flight.
template <int HD>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ O,
                                                       const __nv_bfloat16* __restrict__ dO,
                                                       const float* __restrict__ LSE, float* __restrict__ nlse2,
                                                       float* __restrict__ ndelta, int N, int Npad,
                                                       long long rows) {
  constexpr int kRowsPerWarp = 8;
  constexpr int kLanesPerRow = HD / 8;                       // 16-byte pieces per row: 16 or 8
  constexpr int kRowsPerLoad = 32 / kLanesPerRow;            // rows one warp-wide load covers: 2 or 4
  constexpr int kLoads = kRowsPerWarp / kRowsPerLoad;        // loads per lane per operand: 4 or 2
  static_assert(kLanesPerRow * kRowsPerLoad == 32 && kLoads * kRowsPerLoad == kRowsPerWarp, "row split");
  const long long row0 = ((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * kRowsPerWarp;
  if (row0 >= rows) return;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, piece = lane % kLanesPerRow;
  uint4 o4[kLoads], g4[kLoads];
  float lse[kLoads];
  bool live[kLoads];
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    const long long row = row0 + i * kRowsPerLoad + sub;
    const long long bh = row / Npad;
    const int r = static_cast<int>(row - bh * Npad);
    live[i] = row < rows && r < N;
    o4[i] = g4[i] = make_uint4(0u, 0u, 0u, 0u);
    lse[i] = 0.f;
    if (live[i]) {
      const size_t off = (static_cast<size_t>(bh) * N + r) * HD + piece * 8;
      o4[i] = __ldg(reinterpret_cast<const uint4*>(O + off));
      g4[i] = __ldg(reinterpret_cast<const uint4*>(dO + off));
      if (piece == 0) lse[i] = __ldg(LSE + static_cast<size_t>(bh) * N + r);
    }
  }
  float dsum[kLoads];
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    const uint32_t ow[4] = {o4[i].x, o4[i].y, o4[i].z, o4[i].w};
    const uint32_t gw[4] = {g4[i].x, g4[i].y, g4[i].z, g4[i].w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
      const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
      acc = fmaf(of.x, gf.x, acc);
      acc = fmaf(of.y, gf.y, acc);
    }
#pragma unroll
    for (int s = kLanesPerRow / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    dsum[i] = acc;
  }
  if (piece == 0) {
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const long long row = row0 + i * kRowsPerLoad + sub;
      if (row < rows) {
        nlse2[row] = live[i] ? -lse[i] * 1.4426950408889634074f : -INFINITY;
        ndelta[row] = -dsum[i];
      }
    }
  }
}

// The tile-product bursts of sm103a_ptx.cuh (mma_ss_k128_warp, mma_ss_k64_warp,
// mma_ts_k128_warp) with each product's descriptors formed by one 64-bit add
// to the burst's base descriptors: the offsets never carry out of the
// start-address field, so the descriptor words are the same. That takes
// fewer instructions from the issuing warp, which shares its sub-partition
// with elementwise warps; here it made the backward call 2.5 % faster, while
// the forward kernel measured no better with it.
#define FA_BURST_SS64(OA) "add.s64 ad, a0, " #OA ";\n\tadd.s64 bd, b0, " #OA ";\n\t" \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, t;\n\t"
#define FA_BURST_SS64_HEAD \
  "{\n\t.reg .pred p, e, t;\n\t.reg .b64 a0, b0, ad, bd;\n\t" \
  "setp.ne.b32 p, %5, 0;\n\tsetp.eq.u32 t, %4, %4;\n\telect.sync _|e, 0xffffffff;\n\t" \
  "mov.b64 a0, {%1, %3};\n\tmov.b64 b0, {%2, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], a0, b0, %4, p;\n\t"
#define FA_BURST_TS64(OA, OB) "add.u32 ta, %1, " #OA ";\n\tadd.s64 bd, b0, " #OB ";\n\t" \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %4, t;\n\t"
#define FA_BURST_TS64_HEAD \
  "{\n\t.reg .pred p, e, t;\n\t.reg .b32 ta;\n\t.reg .b64 b0, bd;\n\t" \
  "setp.ne.b32 p, %5, 0;\n\tsetp.eq.u32 t, %4, %4;\n\telect.sync _|e, 0xffffffff;\n\t" \
  "mov.b64 b0, {%2, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b0, %4, p;\n\t"

__device__ __forceinline__ void mma_ss_k128_warp64(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                                   uint32_t idesc, uint32_t acc0) {
  asm volatile(FA_BURST_SS64_HEAD FA_BURST_SS64(2) FA_BURST_SS64(4) FA_BURST_SS64(6) FA_BURST_SS64(1024)
               FA_BURST_SS64(1026) FA_BURST_SS64(1028) FA_BURST_SS64(1030) "}" ::"r"(d_tmem),
               "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(acc0)
               : "memory");
}
__device__ __forceinline__ void mma_ss_k64_warp64(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                                  uint32_t idesc, uint32_t acc0) {
  asm volatile(FA_BURST_SS64_HEAD FA_BURST_SS64(2) FA_BURST_SS64(4) FA_BURST_SS64(6) "}" ::"r"(d_tmem), "r"(a_lo),
               "r"(b_lo), "r"(hi), "r"(idesc), "r"(acc0)
               : "memory");
}
template <int kA4>
__device__ __forceinline__ void mma_ts_k128_warp64(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                                   uint32_t idesc, uint32_t acc0) {
  static_assert(kA4 == 32 || kA4 == 64, "A column step of the second four products");
  if constexpr (kA4 == 32) {
    asm volatile(FA_BURST_TS64_HEAD FA_BURST_TS64(8, 128) FA_BURST_TS64(16, 256) FA_BURST_TS64(24, 384)
                 FA_BURST_TS64(32, 512) FA_BURST_TS64(40, 640) FA_BURST_TS64(48, 768) FA_BURST_TS64(56, 896) "}"
                 ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc0)
                 : "memory");
  } else {
    asm volatile(FA_BURST_TS64_HEAD FA_BURST_TS64(8, 128) FA_BURST_TS64(16, 256) FA_BURST_TS64(24, 384)
                 FA_BURST_TS64(64, 512) FA_BURST_TS64(72, 640) FA_BURST_TS64(80, 768) FA_BURST_TS64(88, 896) "}"
                 ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc0)
                 : "memory");
  }
}

// S-shaped product over the model dimension: D[128 x 128] = A B^T with A and
// B two 128-row tiles in the K-major swizzled layout (k = 0 .. HD). Called by
// the whole converged issuer warp (one elected lane issues).
template <int HD>
__device__ __forceinline__ void issue_tile_qk(uint32_t d_tmem, uint32_t a_tile, uint32_t b_tile) {
  using C = BwdCfg<HD>;
  static_assert(C::kChunkBytes == 16384, "128-row tiles of 128-byte rows per chunk");
  const uint64_t a_desc = ptx::desc_kmajor_sw128(a_tile), b_desc = ptx::desc_kmajor_sw128(b_tile);
  if constexpr (HD == 128)
    mma_ss_k128_warp64(d_tmem, ptx::desc_lo(a_desc), ptx::desc_lo(b_desc), ptx::desc_hi(a_desc), C::kIdescS, 0u);
  else
    mma_ss_k64_warp64(d_tmem, ptx::desc_lo(a_desc), ptx::desc_lo(b_desc), ptx::desc_hi(a_desc), C::kIdescS, 0u);
}

// Accumulating product over the 128 streamed rows: D[128 x HD] += A B with A
// packed bf16 in TMEM (rows 64h .. 64h+63 of the streamed block at column
// a_col + kHalf * h, 16 rows per 8 columns) and B a 128 x HD tile read
// MN-major from shared memory. Called by the whole converged issuer warp.
template <int HD, int kHalf>
__device__ __forceinline__ void issue_tile_acc(uint32_t d_tmem, uint32_t a_col, uint32_t b_tile, bool accumulate) {
  using C = BwdCfg<HD>;
  const uint64_t b_desc = ptx::desc_mnmajor_sw128(b_tile, C::kChunkBytes);
  mma_ts_k128_warp64<kHalf>(d_tmem, a_col, ptx::desc_lo(b_desc), ptx::desc_hi(b_desc), C::kIdescAcc,
                               accumulate ? 1u : 0u);
}

// Epilogue helper: 32 accumulator columns of this thread's row, times `mul`,
// to bf16 at dst (64 bytes, 16-byte aligned) when `store`.
__device__ __forceinline__ void store_row32(uint32_t taddr, float mul, __nv_bfloat16* dst, bool store) {
  uint32_t v[32];
  ptx::tmem_ld32(taddr, v);
  ptx::tmem_ld_wait();
  ptx::reg_fence32(v);
  uint32_t packed[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    packed[i] = ptx::pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
  if (store) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      d4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
  }
}

// Epilogue helper for d = 128, once every product of the CTA has completed
// (its shared memory is free then): the warp's 32 rows x 64 columns of an
// accumulator, times `mul`, to bf16 in a 4 KB staging buffer at `stage`, in
// the 128-byte swizzled layout a tiled TMA store reads.
__device__ __forceinline__ void stage_rows64(uint32_t taddr, float mul, uint32_t stage, int lane) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t v[32];
    ptx::tmem_ld32(taddr + 32 * h, v);
    ptx::tmem_ld_wait();
    ptx::reg_fence32(v);
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      packed[i] = ptx::pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
    const uint32_t row_addr = stage + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t unit = 4u * h + q;      // 16-byte unit within the 128-byte row
      const uint32_t addr = row_addr + ((unit ^ static_cast<uint32_t>(lane & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(packed[4 * q]),
                   "r"(packed[4 * q + 1]), "r"(packed[4 * q + 2]), "r"(packed[4 * q + 3])
                   : "memory");
    }
  }
}

// ---------------------------------------------------------------- dQ
// Shared memory: Q and dO of the CTA's query block, a ring of kKSlots K tiles
// and one of kVSlots V tiles (K_j is read twice, by S_j early and by dQ_j
// late; V_j only by dP_j). TMEM: dQ at 0, S at HD, dP at HD + 128, and two
// 64-column slots for the packed dS of consecutive blocks at HD + 256. With
// dS outside the score regions, S_{j+1} and dP_{j+1} are issued as soon as
// the elementwise warps have loaded S_j and dP_j, and the elementwise step of
// block j+1 overlaps dQ += dS_j K_j.
template <int HD>
struct DqCfg {
  using C = BwdCfg<HD>;
  static constexpr int kKSlots = (HD == 128) ? 3 : 4;
  static constexpr int kVSlots = (HD == 128) ? 2 : 4;
  static constexpr int kSmemBytes = (2 + kKSlots + kVSlots) * C::kTileBytes + 1024;
  static constexpr uint32_t kColDQ = 0;
  static constexpr uint32_t kColS = HD;
  static constexpr uint32_t kColP = HD + 128;
  static constexpr uint32_t kColDS = HD + 256;    // + 64 * (j & 1)
};

// One CTA of the query-block role: query rows [128 blk, 128 blk + 128) of
// head bh. The tensor maps are the kernel's own (grid-constant) parameters.
template <int HD>
__device__ __forceinline__ void bwd_dq_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                           const CUtensorMap& tmdQ,
                                           const CUtensorMap& tmdO, const BwdParams& p, int blk, int bh) {
  using C = BwdCfg<HD>;
  using D = DqCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_in_full;
  __shared__ __align__(8) uint64_t bar_k_full[D::kKSlots];
  __shared__ __align__(8) uint64_t bar_k_empty[D::kKSlots];
  __shared__ __align__(8) uint64_t bar_v_full[D::kVSlots];
  __shared__ __align__(8) uint64_t bar_v_empty[D::kVSlots];
  __shared__ __align__(8) uint64_t bar_st_full;    // S_j complete
  __shared__ __align__(8) uint64_t bar_dpt_full;   // dP_j complete
  __shared__ __align__(8) uint64_t bar_s_free;     // S_j loaded (and K_{j+1} landed)
  __shared__ __align__(8) uint64_t bar_dp_free;
  __shared__ __align__(8) uint64_t bar_p_full[2];
  __shared__ __align__(8) uint64_t bar_acc_full;
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q0 = blk * C::kBlk;
  const int n = p.n_blocks;

  const uint32_t smem_base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = smem_base;
  const uint32_t sdO = smem_base + C::kTileBytes;
  const uint32_t sK = smem_base + 2 * C::kTileBytes;                    // kKSlots tiles
  const uint32_t sV = sK + D::kKSlots * C::kTileBytes;                  // kVSlots tiles

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar_in_full), 1);
    for (int s = 0; s < D::kKSlots; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bar_k_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_k_empty[s]), 1);
    }
    for (int s = 0; s < D::kVSlots; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bar_v_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_v_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bar_st_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_dpt_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_s_free), 256);
    ptx::mbar_init(ptx::smem_u32(&bar_dp_free), 256);
    ptx::mbar_init(ptx::smem_u32(&bar_p_full[0]), 256);
    ptx::mbar_init(ptx::smem_u32(&bar_p_full[1]), 256);
    ptx::mbar_init(ptx::smem_u32(&bar_acc_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_drain), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_base_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    ptx::prefetch_tmap(&tmdO);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  volatile int* abort_ptr = &abort_flag;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_once = ptx::policy_evict_first();
      const uint64_t pol_shared = ptx::policy_evict_last();
      const uint32_t in_full = ptx::smem_u32(&bar_in_full);
      ptx::mbar_arrive_expect_tx(in_full, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        ptx::tma_load_3d(sQ + c * C::kChunkBytes, &tmQ, in_full, c * 64, q0, bh, pol_once);
        ptx::tma_load_3d(sdO + c * C::kChunkBytes, &tmdO, in_full, c * 64, q0, bh, pol_once);
      }
      // Loads in the order they are needed: K_0, V_0, K_1, V_1, ...
      int issued = 0;    // loads started, counted in that order
      bool ok = true;
      for (int it = 0; it < 2 * n && ok; ++it) {
        const int j = it >> 1;
        const bool is_v = it & 1;
        const int slots = is_v ? D::kVSlots : D::kKSlots;
        const int slot = j % slots;
        uint64_t* empty = is_v ? bar_v_empty : bar_k_empty;
        uint64_t* full = is_v ? bar_v_full : bar_k_full;
        if (!wait_or_abort(ptx::smem_u32(&empty[slot]), ((j / slots) & 1) ^ 1u, abort_ptr, p.timeout_ns,
                           kRoleDqProducer)) {
          ok = false;
          break;
        }
        issued = it + 1;
        if (it == p.drop_load) continue;   // test hook: this tile never arrives
        const uint32_t fb = ptx::smem_u32(&full[slot]);
        ptx::mbar_arrive_expect_tx(fb, C::kTileBytes);
        const uint32_t dst = (is_v ? sV : sK) + slot * C::kTileBytes;
        for (int c = 0; c < C::kChunks; ++c)
          ptx::tma_load_3d(dst + c * C::kChunkBytes, is_v ? &tmV : &tmK, fb, c * 64, j * C::kBlk, bh, pol_shared);
      }
      if (!ok || *abort_ptr) {
        drain_wait(in_full, 0, p.timeout_ns);
        // Only the last kKSlots K loads and kVSlots V loads can still be in flight.
        for (int it = 0; it < issued; ++it) {
          const int j = it >> 1;
          const bool is_v = it & 1;
          const int slots = is_v ? D::kVSlots : D::kKSlots;
          const int last_j = ((issued - 1 - (is_v ? 1 : 0)) >> 1);
          if (j + slots <= last_j || it == p.drop_load) continue;
          drain_wait(ptx::smem_u32(&(is_v ? bar_v_full : bar_k_full)[j % slots]), (j / slots) & 1, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this converged (warp-uniform waits, one elected
    // lane issues each tcgen05 instruction).
    {
      auto k_tile = [&](int j) { return sK + (j % D::kKSlots) * C::kTileBytes; };
      auto v_tile = [&](int j) { return sV + (j % D::kVSlots) * C::kTileBytes; };
      // S_j = Q K_j^T and dP_j = dO V_j^T, each committed to its own barrier.
      // K_0 and V_0 are waited for here; every later K_{j+1} by the
      // elementwise warps before their s_free(j), and V_{j+1} before their
      // dp_free(j), so that this warp waits only on the hand-offs.
      auto issue_s = [&](int j) {
        ptx::tc_fence_after();
        issue_tile_qk<HD>(tmem_base + D::kColS, sQ, k_tile(j));
        ptx::mma_commit_warp(ptx::smem_u32(&bar_st_full));
      };
      auto issue_dp = [&](int j) {
        ptx::tc_fence_after();
        issue_tile_qk<HD>(tmem_base + D::kColP, sdO, v_tile(j));
        ptx::mma_commit_warp(ptx::smem_u32(&bar_v_empty[j % D::kVSlots]));
        ptx::mma_commit_warp(ptx::smem_u32(&bar_dpt_full));
      };
      bool ok = wait_warp_or_abort(ptx::smem_u32(&bar_in_full), 0, abort_ptr, p.timeout_ns, kRoleDqMma);
      if (ok) ok = wait_warp_or_abort(ptx::smem_u32(&bar_k_full[0]), 0, abort_ptr, p.timeout_ns, kRoleDqMma);
      if (ok) ok = wait_warp_or_abort(ptx::smem_u32(&bar_v_full[0]), 0, abort_ptr, p.timeout_ns, kRoleDqMma);
      if (ok) {
        issue_s(0);
        issue_dp(0);
      }
      for (int j = 0; j < n && ok; ++j) {
        if (j + 1 < n) {
          // S_{j+1} as soon as S_j has been read; dP_{j+1} once dP_j has.
          ok = wait_warp_or_abort(ptx::smem_u32(&bar_s_free), j & 1, abort_ptr, p.timeout_ns, kRoleDqMma);
          if (!ok) break;
          issue_s(j + 1);
          ok = wait_warp_or_abort(ptx::smem_u32(&bar_dp_free), j & 1, abort_ptr, p.timeout_ns, kRoleDqMma);
          if (!ok) break;
          issue_dp(j + 1);
        }
        ok = wait_warp_or_abort(ptx::smem_u32(&bar_p_full[j & 1]), (j >> 1) & 1, abort_ptr, p.timeout_ns, kRoleDqMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_tile_acc<HD, 32>(tmem_base + D::kColDQ, tmem_base + D::kColDS + 64u * (j & 1), k_tile(j), j > 0);
        ptx::mma_commit_warp(ptx::smem_u32(&bar_k_empty[j % D::kKSlots]));
      }
      if (ok) {
        ptx::mma_commit_warp(ptx::smem_u32(&bar_acc_full));
      } else {
        ptx::mma_commit_warp(ptx::smem_u32(&bar_drain));
        drain_wait(ptx::smem_u32(&bar_drain), 0, p.timeout_ns);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ dS + epilogue
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const size_t vrow = static_cast<size_t>(bh) * p.Npad + q0 + row;
    const float nl = p.nlse2[vrow];
    const float nd = p.ndelta[vrow];
    const uint64_t sl2x2 = ptx::f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t nlx2 = ptx::f2_pack(nl, nl);
    const uint64_t ndx2 = ptx::f2_pack(nd, nd);
    const uint32_t tS = tmem_base + lane_addr + D::kColS + 64u * half;
    const uint32_t tP = tmem_base + lane_addr + D::kColP + 64u * half;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = wait_warp_or_abort(ptx::smem_u32(&bar_st_full), j & 1, abort_ptr, p.timeout_ns, kRoleDqSoftmax);
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t s[2][32], dp[2][32];
      ptx::tmem_ld32(tS, s[0]);
      ptx::tmem_ld32(tS + 32, s[1]);
      ptx::tmem_ld_wait();
      ptx::reg_fence32(s[0]);
      ptx::reg_fence32(s[1]);
      if (j + 1 < n) {
        // K_{j+1} in place before the hand-off that lets S_{j+1} be issued.
        ok = wait_warp_or_abort(ptx::smem_u32(&bar_k_full[(j + 1) % D::kKSlots]), ((j + 1) / D::kKSlots) & 1,
                                abort_ptr, p.timeout_ns, kRoleDqSoftmax);
        if (!ok) break;
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bar_s_free));

      const int valid = p.N - j * C::kBlk - 64 * half;   // keys of this warp's 64 that exist
      const bool ragged = valid < 64;
      // P (float32, kept in s) while dP_j is still on the tensor core.
      if (!ragged) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float x0, x1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][2 * k]), __uint_as_float(s[c][2 * k + 1])),
                                       sl2x2, nlx2),
                           x0, x1);
            float p0 = ptx::ex2_approx(x0);
            float p1 = ptx::ex2_approx(x1);
            s[c][2 * k] = __float_as_uint(p0);
            s[c][2 * k + 1] = __float_as_uint(p1);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float x0, x1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][2 * k]), __uint_as_float(s[c][2 * k + 1])),
                                       sl2x2, nlx2),
                           x0, x1);
            float p0 = ptx::ex2_approx(x0);
            float p1 = ptx::ex2_approx(x1);
            if (32 * c + 2 * k >= valid) p0 = 0.f;   // keys past N: exact zeros whatever the fill gave
            if (32 * c + 2 * k + 1 >= valid) p1 = 0.f;
            s[c][2 * k] = __float_as_uint(p0);
            s[c][2 * k + 1] = __float_as_uint(p1);
          }
        }
      }
      ok = wait_warp_or_abort(ptx::smem_u32(&bar_dpt_full), j & 1, abort_ptr, p.timeout_ns, kRoleDqSoftmax);
      if (!ok) break;
      ptx::tc_fence_after();
      ptx::tmem_ld32(tP, dp[0]);
      ptx::tmem_ld32(tP + 32, dp[1]);
      ptx::tmem_ld_wait();
      ptx::reg_fence32(dp[0]);
      ptx::reg_fence32(dp[1]);
      if (j + 1 < n) {
        // V_{j+1} in place before the hand-off that lets dP_{j+1} be issued.
        ok = wait_warp_or_abort(ptx::smem_u32(&bar_v_full[(j + 1) % D::kVSlots]), ((j + 1) / D::kVSlots) & 1,
                                abort_ptr, p.timeout_ns, kRoleDqSoftmax);
        if (!ok) break;
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bar_dp_free));
      uint32_t pds[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint64_t t =
              ptx::f2_add(ptx::f2_pack(__uint_as_float(dp[c][2 * k]), __uint_as_float(dp[c][2 * k + 1])), ndx2);
          float d0, d1;
          ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(s[c][2 * k]), __uint_as_float(s[c][2 * k + 1])), t),
                         d0, d1);
          pds[16 * c + k] = ptx::pack_bf16x2(d0, d1);
        }
      }
      ptx::tmem_st32(tmem_base + lane_addr + D::kColDS + 64u * (j & 1) + 32u * half, pds);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bar_p_full[j & 1]));
    }
    if (ok) ok = wait_warp_or_abort(ptx::smem_u32(&bar_acc_full), 0, abort_ptr, p.timeout_ns, kRoleDqSoftmax);
    if (ok) {
      ptx::tc_fence_after();
      if constexpr (HD == 128) {
        // Through shared memory: 32 rows x 64 columns per warp, then one
        // tiled TMA store (rows past N are not written).
        const int qw = q0 + quarter * 32;
        if (qw < p.N) {
          const uint32_t stage = smem_base + static_cast<uint32_t>(warp) * 4096u;
          stage_rows64(tmem_base + lane_addr + D::kColDQ + half * 64, p.scale, stage, lane);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&tmdQ, stage, half * 64, qw, bh);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read0();
          }
          __syncwarp();
        }
      } else {
        const int q = q0 + row;
        __nv_bfloat16* dst = p.dQ + (static_cast<size_t>(bh) * p.N + q) * HD + half * (HD / 2);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c)
          store_row32(tmem_base + lane_addr + D::kColDQ + half * (HD / 2) + 32 * c, p.scale, dst + 32 * c, q < p.N);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- dK, dV
// One CTA of the key-block role: key rows [128 blk, 128 blk + 128) of head bh.
template <int HD>
__device__ __forceinline__ void bwd_dkdv_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                             const CUtensorMap& tmdK, const CUtensorMap& tmdV,
                                             const CUtensorMap& tmdO, const BwdParams& p, int blk, int bh) {
  using C = BwdCfg<HD>;
  constexpr uint32_t kColDV = 0;
  constexpr uint32_t kColDK = HD;
  constexpr uint32_t kColR = 2 * HD;    // R0 = kColR, R1 = kColR + 128
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_kv_full;
  __shared__ __align__(8) uint64_t bar_q_full[C::kStages];     // Q_i and -LSE*log2e landed
  __shared__ __align__(8) uint64_t bar_q_empty[C::kStages];    // dK(i) done with Q_i
  __shared__ __align__(8) uint64_t bar_do_full[C::kStages];    // dO_i and -D landed
  __shared__ __align__(8) uint64_t bar_do_empty[C::kStages];   // dV(i) done with dO_i
  __shared__ __align__(8) uint64_t bar_st_full;    // S^T(i) complete
  __shared__ __align__(8) uint64_t bar_dpt_full;   // dP^T(i) complete
  __shared__ __align__(8) uint64_t bar_dp_free;
  __shared__ __align__(8) uint64_t bar_p_full;
  __shared__ __align__(8) uint64_t bar_pt_stored;  // P^T(i) packed into TMEM
  __shared__ __align__(8) uint64_t bar_acc_full;
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kv0 = blk * C::kBlk;
  const int n = p.n_blocks;

  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t smem_base = (raw + 1023u) & ~1023u;
  const uint32_t sK = smem_base;
  const uint32_t sV = smem_base + C::kTileBytes;
  const uint32_t sRing = smem_base + C::kPairBytes;                  // slot s: Q_i, then dO_i
  const uint32_t sVec = sRing + C::kStages * C::kPairBytes;          // slot s: [-lse2 x 128][-D x 128]
  const float* vec = reinterpret_cast<const float*>(smem_raw + (sVec - raw));

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar_kv_full), 1);
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bar_q_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_q_empty[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_do_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_do_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bar_st_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_dpt_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_dp_free), 256);
    ptx::mbar_init(ptx::smem_u32(&bar_p_full), 256);
    ptx::mbar_init(ptx::smem_u32(&bar_pt_stored), 256);
    ptx::mbar_init(ptx::smem_u32(&bar_acc_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_drain), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_base_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    ptx::prefetch_tmap(&tmdO);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  volatile int* abort_ptr = &abort_flag;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // Every tile this CTA loads is read by other CTAs of its head too: its
      // K and V by the head's query-block CTAs, which run right after it.
      const uint64_t pol_shared = ptx::policy_evict_last();
      const uint32_t kv_full = ptx::smem_u32(&bar_kv_full);
      ptx::mbar_arrive_expect_tx(kv_full, C::kPairBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        ptx::tma_load_3d(sK + c * C::kChunkBytes, &tmK, kv_full, c * 64, kv0, bh, pol_shared);
        ptx::tma_load_3d(sV + c * C::kChunkBytes, &tmV, kv_full, c * 64, kv0, bh, pol_shared);
      }
      // Q_i (with its rows' -LSE*log2e) goes into its slot as soon as dK of
      // the slot's previous block has completed, dO_i (with -D) once dV has:
      // the issuer runs dK first, so S^T, which needs only Q, can start early.
      int issued_q = 0, issued_do = 0;
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        const int slot = i % C::kStages;
        const uint32_t par = ((i / C::kStages) & 1) ^ 1u;
        const uint32_t dst = sRing + slot * C::kPairBytes;
        const size_t voff = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(i) * C::kBlk;
        if (!wait_or_abort(ptx::smem_u32(&bar_q_empty[slot]), par, abort_ptr, p.timeout_ns, kRoleDkvProducer)) {
          ok = false;
          break;
        }
        issued_q = i + 1;
        if (i != p.drop_load) {    // test hook: this step's tiles never arrive
          const uint32_t full = ptx::smem_u32(&bar_q_full[slot]);
          ptx::mbar_arrive_expect_tx(full, C::kTileBytes + C::kBlk * 4);
          for (int c = 0; c < C::kChunks; ++c)
            ptx::tma_load_3d(dst + c * C::kChunkBytes, &tmQ, full, c * 64, i * C::kBlk, bh, pol_shared);
          ptx::bulk_load_1d(sVec + slot * C::kVecBytes, p.nlse2 + voff, C::kBlk * 4, full, pol_shared);
        }
        if (!wait_or_abort(ptx::smem_u32(&bar_do_empty[slot]), par, abort_ptr, p.timeout_ns, kRoleDkvProducer)) {
          ok = false;
          break;
        }
        issued_do = i + 1;
        if (i != p.drop_load) {
          const uint32_t full = ptx::smem_u32(&bar_do_full[slot]);
          ptx::mbar_arrive_expect_tx(full, C::kTileBytes + C::kBlk * 4);
          for (int c = 0; c < C::kChunks; ++c)
            ptx::tma_load_3d(dst + C::kTileBytes + c * C::kChunkBytes, &tmdO, full, c * 64, i * C::kBlk, bh,
                             pol_shared);
          ptx::bulk_load_1d(sVec + slot * C::kVecBytes + C::kBlk * 4, p.ndelta + voff, C::kBlk * 4, full,
                            pol_shared);
        }
      }
      if (!ok || *abort_ptr) {
        drain_wait(kv_full, 0, p.timeout_ns);
        for (int i = issued_q > C::kStages ? issued_q - C::kStages : 0; i < issued_q; ++i)
          if (i != p.drop_load)
            drain_wait(ptx::smem_u32(&bar_q_full[i % C::kStages]), (i / C::kStages) & 1, p.timeout_ns);
        for (int i = issued_do > C::kStages ? issued_do - C::kStages : 0; i < issued_do; ++i)
          if (i != p.drop_load)
            drain_wait(ptx::smem_u32(&bar_do_full[i % C::kStages]), (i / C::kStages) & 1, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this converged (warp-uniform waits, one elected
    // lane issues each tcgen05 instruction).
    {
      auto region = [&](int i) { return tmem_base + kColR + 128u * static_cast<uint32_t>(i & 1); };
      auto q_tile = [&](int i) { return sRing + (i % C::kStages) * C::kPairBytes; };
      bool ok = wait_warp_or_abort(ptx::smem_u32(&bar_kv_full), 0, abort_ptr, p.timeout_ns, kRoleDkvMma);
      if (ok) ok = wait_warp_or_abort(ptx::smem_u32(&bar_q_full[0]), 0, abort_ptr, p.timeout_ns, kRoleDkvMma);
      if (ok) {
        ptx::tc_fence_after();
        issue_tile_qk<HD>(region(0), sK, q_tile(0));                   // S_0^T = K Q_0^T
        ptx::mma_commit_warp(ptx::smem_u32(&bar_st_full));
      }
      if (ok) ok = wait_warp_or_abort(ptx::smem_u32(&bar_do_full[0]), 0, abort_ptr, p.timeout_ns, kRoleDkvMma);
      if (ok) {
        ptx::tc_fence_after();
        issue_tile_qk<HD>(region(1), sV, q_tile(0) + C::kTileBytes);   // dP_0^T = V dO_0^T
        ptx::mma_commit_warp(ptx::smem_u32(&bar_dpt_full));
        // dV_0 as soon as P_0^T is in place: it runs while dS_0^T is computed.
        ok = wait_warp_or_abort(ptx::smem_u32(&bar_pt_stored), 0, abort_ptr, p.timeout_ns, kRoleDkvMma);
        if (ok) {
          ptx::tc_fence_after();
          issue_tile_acc<HD, 64>(tmem_base + kColDV, region(0), q_tile(0) + C::kTileBytes, false);   // dV += P^T dO_0
          ptx::mma_commit_warp(ptx::smem_u32(&bar_do_empty[0]));
        }
      }
      for (int i = 0; i < n && ok; ++i) {
        // S_{i+1}^T goes in as soon as region(i+1) is free (dp_free(i)) and
        // Q_{i+1} has landed, if that happens before p_full(i); otherwise
        // after dK/dV(i). A late Q must not hold back dK/dV(i), whose commits
        // free the ring slots the next copies need.
        bool s_issued = false;
        const int s1 = (i + 1) % C::kStages;
        const uint32_t in_par = ((i + 1) / C::kStages) & 1;
        const uint32_t q_full1 = ptx::smem_u32(&bar_q_full[s1]);
        if (i + 1 < n) {
          ok = wait_warp_or_abort(ptx::smem_u32(&bar_dp_free), i & 1, abort_ptr, p.timeout_ns, kRoleDkvMma);
          if (!ok) break;
          const uint64_t t0 = ptx::globaltimer_ns();
          while (true) {
            if (__all_sync(0xffffffffu, ptx::mbar_test_wait(q_full1, in_par))) {
              ptx::tc_fence_after();
              issue_tile_qk<HD>(region(i + 1), sK, q_tile(i + 1));      // S_{i+1}^T
              ptx::mma_commit_warp(ptx::smem_u32(&bar_st_full));
              s_issued = true;
              break;
            }
            if (__all_sync(0xffffffffu, ptx::mbar_test_wait(ptx::smem_u32(&bar_p_full), i & 1))) break;
            // Out of time or aborting: the bounded wait below reports it.
            if (__any_sync(0xffffffffu, *abort_ptr != 0) || ptx::globaltimer_ns() - t0 > p.timeout_ns) break;
            // Poll less often: the elementwise warps of this sub-partition
            // need the issue slots meanwhile.
            __nanosleep(32);
          }
        }
        ok = wait_warp_or_abort(ptx::smem_u32(&bar_p_full), i & 1, abort_ptr, p.timeout_ns, kRoleDkvMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_tile_acc<HD, 64>(tmem_base + kColDK, region(i) + 32, q_tile(i), i > 0);             // dK += dS^T Q_i
        ptx::mma_commit_warp(ptx::smem_u32(&bar_q_empty[i % C::kStages]));
        if (i + 1 < n) {
          if (!s_issued) {
            ok = wait_warp_or_abort(q_full1, in_par, abort_ptr, p.timeout_ns, kRoleDkvMma);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_tile_qk<HD>(region(i + 1), sK, q_tile(i + 1));        // S_{i+1}^T
            ptx::mma_commit_warp(ptx::smem_u32(&bar_st_full));
          }
          ok = wait_warp_or_abort(ptx::smem_u32(&bar_do_full[s1]), in_par, abort_ptr, p.timeout_ns, kRoleDkvMma);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_tile_qk<HD>(region(i), sV, q_tile(i + 1) + C::kTileBytes);   // dP_{i+1}^T
          ptx::mma_commit_warp(ptx::smem_u32(&bar_dpt_full));
          // dV_{i+1} right behind it once P_{i+1}^T is in place.
          ok = wait_warp_or_abort(ptx::smem_u32(&bar_pt_stored), (i + 1) & 1, abort_ptr, p.timeout_ns, kRoleDkvMma);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_tile_acc<HD, 64>(tmem_base + kColDV, region(i + 1), q_tile(i + 1) + C::kTileBytes, true);   // dV
          ptx::mma_commit_warp(ptx::smem_u32(&bar_do_empty[(i + 1) % C::kStages]));
        }
      }
      if (ok) {
        ptx::mma_commit_warp(ptx::smem_u32(&bar_acc_full));
      } else {
        ptx::mma_commit_warp(ptx::smem_u32(&bar_drain));
        drain_wait(ptx::smem_u32(&bar_drain), 0, p.timeout_ns);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ P, dS + epilogue
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint64_t sl2x2 = ptx::f2_pack(p.scale_log2, p.scale_log2);
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      // P^T as soon as S^T(i) is complete (it overlaps the tensor core's dK/dV
      // of the previous block and dP^T of this one), then dS^T once dP^T(i) is.
      ok = wait_warp_or_abort(ptx::smem_u32(&bar_st_full), i & 1, abort_ptr, p.timeout_ns, kRoleDkvSoftmax);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tS = tmem_base + lane_addr + kColR + 128u * (i & 1) + 64u * half;
      const uint32_t tP = tmem_base + lane_addr + kColR + 128u * ((i + 1) & 1) + 64u * half;
      uint32_t s[2][32], dp[2][32];
      ptx::tmem_ld32(tS, s[0]);
      ptx::tmem_ld32(tS + 32, s[1]);
      ptx::tmem_ld_wait();
      ptx::reg_fence32(s[0]);
      ptx::reg_fence32(s[1]);
      // -LSE*log2e and -D of this warp's 64 query columns (broadcast reads).
      const float4* vl = reinterpret_cast<const float4*>(vec + (i % C::kStages) * (C::kVecBytes / 4) + 64 * half);
      const float4* vd = vl + 32;    // + 128 floats
      {
        uint32_t pp[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 l4 = vl[8 * c + u];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int e = 4 * u + 2 * h2;
              const uint64_t nl2 = h2 ? ptx::f2_pack(l4.z, l4.w) : ptx::f2_pack(l4.x, l4.y);
              float x0, x1;
              ptx::f2_unpack(
                  ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1])), sl2x2, nl2), x0,
                  x1);
              const float p0 = ptx::ex2_approx(x0);
              const float p1 = ptx::ex2_approx(x1);
              s[c][e] = __float_as_uint(p0);
              s[c][e + 1] = __float_as_uint(p1);
              pp[16 * c + 2 * u + h2] = ptx::pack_bf16x2(p0, p1);
            }
          }
        }
        ptx::tmem_st32(tS, pp);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&bar_pt_stored));
      }
      ok = wait_warp_or_abort(ptx::smem_u32(&bar_dpt_full), i & 1, abort_ptr, p.timeout_ns, kRoleDkvSoftmax);
      if (!ok) break;
      ptx::tc_fence_after();
      ptx::tmem_ld32(tP, dp[0]);
      ptx::tmem_ld32(tP + 32, dp[1]);
      ptx::tmem_ld_wait();
      ptx::reg_fence32(dp[0]);
      ptx::reg_fence32(dp[1]);
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bar_dp_free));
      uint32_t pds[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 d4 = vd[8 * c + u];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int e = 4 * u + 2 * h2;
            const uint64_t nd2 = h2 ? ptx::f2_pack(d4.z, d4.w) : ptx::f2_pack(d4.x, d4.y);
            const uint64_t t = ptx::f2_add(ptx::f2_pack(__uint_as_float(dp[c][e]), __uint_as_float(dp[c][e + 1])), nd2);
            float d0, d1;
            ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1])), t), d0, d1);
            pds[16 * c + 2 * u + h2] = ptx::pack_bf16x2(d0, d1);
          }
        }
      }
      ptx::tmem_st32(tS + 32, pds);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bar_p_full));
    }
    if (ok) ok = wait_warp_or_abort(ptx::smem_u32(&bar_acc_full), 0, abort_ptr, p.timeout_ns, kRoleDkvSoftmax);
    if (ok) {
      ptx::tc_fence_after();
      if constexpr (HD == 128) {
        // Through shared memory: per warp 32 rows x 64 columns of dV and of
        // dK, then two tiled TMA stores (rows past N are not written).
        const int kw = kv0 + quarter * 32;
        if (kw < p.N) {
          const uint32_t stage = smem_base + static_cast<uint32_t>(warp) * 8192u;
          stage_rows64(tmem_base + lane_addr + kColDV + half * 64, 1.f, stage, lane);
          stage_rows64(tmem_base + lane_addr + kColDK + half * 64, p.scale, stage + 4096u, lane);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&tmdV, stage, half * 64, kw, bh);
            ptx::tma_store_3d(&tmdK, stage + 4096u, half * 64, kw, bh);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read0();
          }
          __syncwarp();
        }
      } else {
        const int kv = kv0 + row;
        const size_t off = (static_cast<size_t>(bh) * p.N + kv) * HD + half * (HD / 2);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) {
          store_row32(tmem_base + lane_addr + kColDV + half * (HD / 2) + 32 * c, 1.f, p.dV + off + 32 * c, kv < p.N);
          store_row32(tmem_base + lane_addr + kColDK + half * (HD / 2) + 32 * c, p.scale, p.dK + off + 32 * c,
                      kv < p.N);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Both roles in one launch, on a 1-D grid: the n_blocks * B * H key-block
// CTAs first, then as many query-block CTAs. Blocks are dispatched in index
// order and a key-block CTA does four tile products per step against three,
// so the longer CTAs start first and the shorter ones fill the last wave of
// SMs, where two launches would each leave a part of their last wave idle.
template <int HD>
__global__ void __launch_bounds__(BwdCfg<HD>::kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ CUtensorMap tmdK,
                  const __grid_constant__ CUtensorMap tmdV, const BwdParams p) {
  // The CTAs of one head are consecutive: its key-block CTAs (the longer
  // role first), then its query-block CTAs. Both roles stream that head's Q,
  // K, V and dO, which then stay in L2 from one role to the other.
  const long long per_head = 2LL * p.n_blocks;
  const long long idx = blockIdx.x;
  const int bh = static_cast<int>(idx / per_head);
  const int r = static_cast<int>(idx - bh * per_head);
  const bool dkdv = r < p.n_blocks;
  const int blk = dkdv ? r : r - p.n_blocks;
  if (dkdv)
    bwd_dkdv_cta<HD>(tmQ, tmK, tmV, tmdK, tmdV, tmdO, p, blk, bh);
  else
    bwd_dq_cta<HD>(tmQ, tmK, tmV, tmdQ, tmdO, p, blk, bh);
}

}  // namespace fa
