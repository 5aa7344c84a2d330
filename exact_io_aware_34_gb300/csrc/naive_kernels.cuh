// Standard (materialising) attention on GB300: the comparator for the fused
// kernel. It runs the three steps that "01 · 注意力为什么是 IO 瓶颈" §3 and §5
// describe, each as its own kernel with its N x N intermediate in HBM:
//   1. S = bf16(scale * bf16(Q K^T))      s_gemm_kernel (tcgen05, TMEM; persistent)
//   2. P = bf16(softmax(S)) in place of S; LSE = m + ln l per row
//                                          softmax_rows_kernel
//   3. O = bf16(P V)                        gemm_bf16_kernel
// The rounding points are those of a bf16 framework running the three ops
// (the reading used for the "no worse than twice the baseline" rule).
//
// gemm_bf16_kernel computes, for every batch index z (one (b, h)):
//   C[z][m][n] = bf16(alpha * bf16(sum_k A[z][m][k] * B[z](k, n)))
// with A row-major [M][K] (K-major operand) and B either [Nc][K] (K-major)
// or [K][Nc] (MN-major, as for O = P V). One CTA computes a 128 x BN tile
// of C; warp 4 loads A and B chunks of 64 k with TMA into a ring, warp 5
// issues the tcgen05 MMAs into TMEM, warps 0-3 convert the accumulator (one
// row per thread), stage it in shared memory in the 128-byte swizzled layout
// and write it with TMA stores (each warp its own 32 rows). S = Q K^T, whose
// tiles have only K = d, runs on s_gemm_kernel below, which keeps its CTAs
// and overlaps one tile's epilogue with the next tile's products.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103a_ptx.cuh"

namespace fa {
namespace naive {

template <int BN, bool B_KMAJOR>
struct GemmCfg {
  static constexpr int kBM = 128;
  static constexpr int kBK = 64;                          // k per ring stage (one 128-byte row)
  static constexpr int kABytes = kBM * kBK * 2;           // 16 KB
  static constexpr int kBBytes = BN * kBK * 2;            // BN x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = B_KMAJOR ? 2 : 4;
  static constexpr int kCtasPerSm = B_KMAJOR ? 3 : 1;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static constexpr int kThreads = 192;                    // 6 warps
  static constexpr uint32_t kTmemCols = BN < 32 ? 32 : BN;
  static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBM, BN, false, !B_KMAJOR);
};

struct GemmParams {
  __nv_bfloat16* C;
  int M, Nc, K;
  int ldc;          // row stride of C in elements (a multiple of 8)
  float alpha;
  unsigned long long timeout_ns;
};

// Bounded single-thread wait; on timeout records the status word and
// returns false (the caller then stops issuing and drains).
__device__ __forceinline__ bool naive_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned long long timeout_ns, unsigned int role) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      if (atomicCAS(&g_status_word, 0u, 1u) == 0u) {
        g_status_info[0] = role;
        g_status_info[1] = blockIdx.x;
        g_status_info[2] = blockIdx.y;
        g_status_info[3] = blockIdx.z;
      }
      __threadfence();
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool naive_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                unsigned long long timeout_ns, unsigned int role) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = naive_wait(bar, parity, abort_flag, timeout_ns, role) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int BN, bool B_KMAJOR>
__global__ void __launch_bounds__(GemmCfg<BN, B_KMAJOR>::kThreads, GemmCfg<BN, B_KMAJOR>::kCtasPerSm)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  using C = GemmCfg<BN, B_KMAJOR>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[C::kStages];
  __shared__ __align__(8) uint64_t bar_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_acc;
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * C::kBM;
  const int z = blockIdx.z;
  const int nk = (p.K + C::kBK - 1) / C::kBK;
  const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bar_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bar_acc), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_drain), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_ptr = &abort_flag;

  if (warp == 4) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_first();
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % C::kStages;
        if (!naive_wait(ptx::smem_u32(&bar_empty[s]), ((kb / C::kStages) & 1) ^ 1u, abort_ptr, p.timeout_ns, 1))
          break;
        issued = kb + 1;
        const uint32_t full = ptx::smem_u32(&bar_full[s]);
        const uint32_t sa = base + s * C::kStageBytes;
        const uint32_t sb = sa + C::kABytes;
        ptx::mbar_arrive_expect_tx(full, C::kStageBytes);
        ptx::tma_load_3d(sa, &tmA, full, kb * C::kBK, m0, z, pol);
        if (B_KMAJOR) {
          ptx::tma_load_3d(sb, &tmB, full, kb * C::kBK, n0, z, pol);
        } else {
          // BN columns of n as BN/64 boxes of 64 n x 64 k rows (8 KB each).
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) ptx::tma_load_3d(sb + c * 8192, &tmB, full, n0 + 64 * c, kb * C::kBK, z, pol);
        }
      }
      if (*abort_ptr) {
        const int first = issued > C::kStages ? issued - C::kStages : 0;
        for (int kb = first; kb < issued; ++kb) drain_wait(ptx::smem_u32(&bar_full[kb % C::kStages]), (kb / C::kStages) & 1, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % C::kStages;
        ok = naive_wait(ptx::smem_u32(&bar_full[s]), (kb / C::kStages) & 1, abort_ptr, p.timeout_ns, 2);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t sa = base + s * C::kStageBytes;
        const uint32_t sb = sa + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < C::kBK / 16; ++kk) {
          const uint64_t adesc = ptx::desc_kmajor_sw128(sa + kk * 32);
          const uint64_t bdesc = B_KMAJOR ? ptx::desc_kmajor_sw128(sb + kk * 32)
                                          : ptx::desc_mnmajor_sw128(sb + kk * 16 * 128, 8192);
          ptx::mma_ss(tmem, adesc, bdesc, C::kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&bar_empty[s]));
      }
      if (ok) {
        ptx::mma_commit(ptx::smem_u32(&bar_acc));
      } else {
        ptx::mma_commit(ptx::smem_u32(&bar_drain));
        drain_wait(ptx::smem_u32(&bar_drain), 0, p.timeout_ns);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue: TMEM -> swizzled SMEM -> TMA store
    if (naive_wait_warp(ptx::smem_u32(&bar_acc), 0, abort_ptr, p.timeout_ns, 3)) {
      ptx::tc_fence_after();
      const int row = warp * 32 + lane;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
      // The ring is idle once the accumulator is complete: stage the tile at
      // its start as BN/64 chunks of 128 rows x 128 bytes.
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t acc[32];
        ptx::tmem_ld32(taddr + 32 * c, acc);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(acc);
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          // round the fp32 sum to bf16, then apply alpha and round again
          const float a0 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(acc[2 * i]))) * p.alpha;
          const float a1 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(acc[2 * i + 1]))) * p.alpha;
          packed[i] = ptx::pack_bf16x2(a0, a1);
        }
        const uint32_t row_addr = base + (c >> 1) * (C::kBM * 128) + row * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t unit = 4 * (c & 1) + v;       // 16-byte unit within the 128-byte row
          const uint32_t addr = row_addr + ((unit ^ static_cast<uint32_t>(row & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(packed[4 * v]),
                       "r"(packed[4 * v + 1]), "r"(packed[4 * v + 2]), "r"(packed[4 * v + 3])
                       : "memory");
        }
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        // this warp's 32 rows; rows past M and columns past Nc are not written
#pragma unroll
        for (int c = 0; c < BN / 64; ++c)
          ptx::tma_store_3d(&tmC, base + c * (C::kBM * 128) + warp * 32 * 128, n0 + 64 * c, m0 + warp * 32, z);
        ptx::bulk_commit_group();
        ptx::bulk_wait_group_read0();
      }
      __syncwarp();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// S = bf16(alpha * bf16(Q K^T)) for every (z, 128-row, 128-column) tile, as
// a persistent grid: CTA c walks tiles c, c + gridDim.x, ... (columns
// fastest, so that the CTAs in flight share the A rows and one head's B rows
// in L2). A (M x K) and B (Nc x K) are K-major with K <= 128 (d). The
// accumulator is double-buffered in TMEM (two 128-column halves), so the MMA
// of the next tile runs while the epilogue warps convert this one; the
// epilogue stages its bf16 rows in a buffer of its own (not the load ring)
// and writes them with TMA stores, each warp waiting only for its own
// previous store to have read its rows.
struct SGemmCfg {
  static constexpr int kBM = 128;
  static constexpr int kBN = 128;
  static constexpr int kBK = 64;
  static constexpr int kABytes = kBM * kBK * 2;                 // 16 KB
  static constexpr int kStageBytes = kABytes + kBN * kBK * 2;   // A and B chunks of one k step
  static constexpr int kStages = 2;
  static constexpr int kOutBytes = kBM * kBN * 2;               // 2 chunks of 128 rows x 128 bytes
  static constexpr int kSmemBytes = kStages * kStageBytes + kOutBytes + 1024;
  static constexpr int kThreads = 192;                          // 6 warps
  static constexpr int kCtasPerSm = 2;                          // 2 x 97 KB shared, 2 x 256 TMEM columns
  static constexpr uint32_t kTmemCols = 2 * kBN;
  static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBM, kBN, false, false);
};

struct SGemmParams {
  int M, Nc, K;
  int mt, nt;        // 128-row and 128-column tiles per batch index
  int tiles;         // mt * nt * batch
  float alpha;
  unsigned long long timeout_ns;
};

__global__ void __launch_bounds__(SGemmCfg::kThreads, SGemmCfg::kCtasPerSm)
    s_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmC, const SGemmParams p) {
  using C = SGemmCfg;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[C::kStages];
  __shared__ __align__(8) uint64_t bar_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_acc_full[2];
  __shared__ __align__(8) uint64_t bar_acc_empty[2];
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nk = (p.K + C::kBK - 1) / C::kBK;
  const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t out = base + C::kStages * C::kStageBytes;   // 1024-aligned staging buffer
  auto tile_coords = [&](int t, int& z, int& m0, int& n0) {
    const int per = p.mt * p.nt;
    z = t / per;
    const int r = t - z * per;
    m0 = (r / p.nt) * C::kBM;
    n0 = (r - (r / p.nt) * p.nt) * C::kBN;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bar_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_u32(&bar_acc_full[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_acc_empty[a]), 4);   // one arrival per epilogue warp
    }
    ptx::mbar_init(ptx::smem_u32(&bar_drain), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_ptr = &abort_flag;

  if (warp == 4) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_last();   // A and B tiles are read by many CTAs
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
        int z, m0, n0;
        tile_coords(t, z, m0, n0);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % C::kStages;
          if (!naive_wait(ptx::smem_u32(&bar_empty[s]), ((it / C::kStages) & 1) ^ 1u, abort_ptr, p.timeout_ns, 1)) {
            ok = false;
            break;
          }
          const uint32_t full = ptx::smem_u32(&bar_full[s]);
          const uint32_t sa = base + s * C::kStageBytes;
          ptx::mbar_arrive_expect_tx(full, C::kStageBytes);
          ptx::tma_load_3d(sa, &tmA, full, kb * C::kBK, m0, z, pol);
          ptx::tma_load_3d(sa + C::kABytes, &tmB, full, kb * C::kBK, n0, z, pol);
        }
      }
      if (!ok) {
        // Let the copies in flight land before the CTA exits.
        const int first = it > C::kStages ? it - C::kStages : 0;
        for (int k = first; k < it; ++k)
          drain_wait(ptx::smem_u32(&bar_full[k % C::kStages]), (k / C::kStages) & 1, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      int it = 0, i = 0;
      for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x, ++i) {
        const int a = i & 1;
        ok = naive_wait(ptx::smem_u32(&bar_acc_empty[a]), ((i >> 1) & 1) ^ 1u, abort_ptr, p.timeout_ns, 2);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t acc = tmem + a * C::kBN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % C::kStages;
          ok = naive_wait(ptx::smem_u32(&bar_full[s]), (it / C::kStages) & 1, abort_ptr, p.timeout_ns, 2);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t sa = base + s * C::kStageBytes;
#pragma unroll
          for (int kk = 0; kk < C::kBK / 16; ++kk)
            ptx::mma_ss(acc, ptx::desc_kmajor_sw128(sa + kk * 32), ptx::desc_kmajor_sw128(sa + C::kABytes + kk * 32),
                        C::kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(ptx::smem_u32(&bar_empty[s]));
        }
        if (ok) ptx::mma_commit(ptx::smem_u32(&bar_acc_full[a]));
      }
      if (!ok) {
        ptx::mma_commit(ptx::smem_u32(&bar_drain));
        drain_wait(ptx::smem_u32(&bar_drain), 0, p.timeout_ns);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue: TMEM -> swizzled SMEM -> TMA store
    const int row = warp * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int i = 0;
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++i) {
      const int a = i & 1;
      if (!naive_wait_warp(ptx::smem_u32(&bar_acc_full[a]), (i >> 1) & 1, abort_ptr, p.timeout_ns, 3)) break;
      ptx::tc_fence_after();
      int z, m0, n0;
      tile_coords(t, z, m0, n0);
      // This warp's rows of the staging buffer are free once its previous
      // store has read them (one tile ago, so normally long done).
      if (lane == 0) ptx::bulk_wait_group_read0();
      __syncwarp();
#pragma unroll
      for (int c = 0; c < C::kBN / 32; ++c) {
        uint32_t acc[32];
        ptx::tmem_ld32(taddr + a * C::kBN + 32 * c, acc);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(acc);
        if (c == C::kBN / 32 - 1) {
          // The accumulator half is read: it may take the tile after next.
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bar_acc_empty[a]));
        }
        uint32_t packed[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          // round the fp32 sum to bf16, then apply alpha and round again
          const float a0 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(acc[2 * k]))) * p.alpha;
          const float a1 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(acc[2 * k + 1]))) * p.alpha;
          packed[k] = ptx::pack_bf16x2(a0, a1);
        }
        const uint32_t row_addr = out + (c >> 1) * (C::kBM * 128) + row * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t unit = 4 * (c & 1) + v;       // 16-byte unit within the 128-byte row
          const uint32_t addr = row_addr + ((unit ^ static_cast<uint32_t>(row & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(packed[4 * v]),
                       "r"(packed[4 * v + 1]), "r"(packed[4 * v + 2]), "r"(packed[4 * v + 3])
                       : "memory");
        }
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        // this warp's 32 rows; rows past M and columns past Nc are not written
#pragma unroll
        for (int c = 0; c < C::kBN / 64; ++c)
          ptx::tma_store_3d(&tmC, out + c * (C::kBM * 128) + warp * 32 * 128, n0 + 64 * c, m0 + warp * 32, z);
        ptx::bulk_commit_group();
      }
    }
    if (lane == 0) ptx::bulk_wait_group_read0();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Row softmax in place: P[r] = bf16(e^{S[r] - m} / l) computed in fp32 from
// the bf16 scores, LSE[r] = m + ln l. One warp per row (8 rows per 256-thread
// block), 16-byte loads and stores; rows have n valid columns and a stride of
// ld elements (a multiple of 64). Pass 1 keeps an online max and sum per lane
// and merges them across the warp; pass 2 reads the row again and writes P
// over it. (Keeping the row in shared memory or registers to save the second
// read measured slower on GB300: fewer resident warps, less in flight.)
__device__ __forceinline__ void softmax_absorb8(const uint4& u, float& m, float& l) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
  float x[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
  float mx = x[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) mx = fmaxf(mx, x[e]);
  if (mx > m) {
    l = (m == -INFINITY) ? 0.f : l * expf(m - mx);
    m = mx;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) l += expf(x[e] - m);
}

__device__ __forceinline__ void softmax_absorb1(float x, float& m, float& l) {
  if (x > m) {
    l = (m == -INFINITY) ? 1.f : l * expf(m - x) + 1.f;
    m = x;
  } else {
    l += expf(x - m);
  }
}

__device__ __forceinline__ void softmax_warp_merge(float& m, float& l) {
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, m2);
    l = (m == -INFINITY ? 0.f : l * expf(m - mn)) + (m2 == -INFINITY ? 0.f : l2 * expf(m2 - mn));
    m = mn;
  }
}

__device__ __forceinline__ uint4 softmax_emit8(uint4 u, float m, float inv) {
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    h[e] = __floats2bfloat162_rn(expf(f.x - m) * inv, expf(f.y - m) * inv);
  }
  return u;
}

__global__ void __launch_bounds__(256) softmax_rows_kernel(__nv_bfloat16* S, float* LSE, long long rows, int n,
                                                           int ld) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * 8 + warp;
  if (r >= rows) return;
  __nv_bfloat16* row = S + r * static_cast<size_t>(ld);
  float m = -INFINITY, l = 0.f;
  const int n8 = n & ~7;
  for (int i = lane * 8; i < n8; i += 256) softmax_absorb8(*reinterpret_cast<const uint4*>(row + i), m, l);
  for (int i = n8 + lane; i < n; i += 32) softmax_absorb1(__bfloat162float(row[i]), m, l);
  softmax_warp_merge(m, l);
  const float inv = 1.f / l;
  for (int i = lane * 8; i < n8; i += 256)
    *reinterpret_cast<uint4*>(row + i) = softmax_emit8(*reinterpret_cast<const uint4*>(row + i), m, inv);
  for (int i = n8 + lane; i < n; i += 32) row[i] = __float2bfloat16_rn(expf(__bfloat162float(row[i]) - m) * inv);
  if (lane == 0) LSE[r] = m + logf(l);
}

}  // namespace naive
}  // namespace fa
