// Fused exact-attention forward kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// A unit of work is 2 query tiles of 128 rows (256 query rows) of one (b, h);
// the CTA that owns it streams every 128-row key/value block of that head
// past them:
//   "Flash Attention (FA1)", "Tiling in FlashAttention": Q in Br x d blocks,
//   K and V in Bc x d blocks, Tc = ceil(N / Bc); here Br = Bc = 128 (the
//   tcgen05 M and the key-block width). The CTA runs the query-outer order
//   ("01 · 注意力为什么是 IO 瓶颈" §5 skeleton; the FlashAttention-2 split of
//   "FlashAttention：IO 感知的精确注意力", core concepts).
//
// Per key block j and query tile t the update is the page's online softmax
// ("Flash Attention (FA1)", derivation steps 1-5) in its unnormalised form:
//   S = Q_t K_j^T                        (tcgen05.mma, fp32 in TMEM)
//   m_new = max(m, rowmax(S))            (step 2)
//   P = exp(scale*(S - m_new))           (step 1 taken against m_new)
//   l = l * e^{scale(m - m_new)} + rowsum(P)      (step 2)
//   O = O * e^{scale(m - m_new)} + P V_j          (steps 3-5, numerator form)
// and after the last block O /= l, LSE = scale*m + ln l.
//
// A negative scale: the tensor core forms -S (the A operand negated through
// the instruction descriptor) and the kernel runs with |scale|, since
// scale * S = |scale| * (-S); the maximum the softmax keeps is then that of
// the scaled scores, as it is for scale >= 0.
//
// Exactness-preserving deviation: the running maximum used for the
// exponentials is only moved when the new row maximum exceeds it by more
// than kRescaleLog2 (in log2 units of the scaled score). Until then the
// stale maximum keeps serving both l and O, so every term of O and l carries
// the same factor and O / l and (m + ln l) are unchanged; the probabilities
// stay below 2^kRescaleLog2, far inside bf16/fp32 range. This skips most of
// the O rescales (a TMEM read-modify-write of 128 x d floats).
//
// Persistent grid: one CTA per SM (shared and tensor memory allow no
// second) walks units blockIdx.x, blockIdx.x + gridDim.x, ... in (b, h,
// query block) order, so the CTAs in flight share few heads' K/V in L2. The
// ring position and the barrier phases run on across units: the next unit's
// Q is loaded as soon as the last Q K^T products of the current one have
// completed, and its first Q K^T products are issued right after the current
// unit's last P V, so they overlap that unit's epilogue.
//
// Split last round. All units cost the same, so a grid of G CTAs takes
// ceil(units / G) rounds. When the units left after the whole rounds would
// fill at most half of an even grid, the host launches clusters of two CTAs
// and each pair shares one of those units: rank r runs the r-th half of its
// key blocks and keeps an unmerged partial result (O relative to its own
// running maximum, with m, l and l'). Then rank r finalises query tile r:
// the partner's tile-r warpgroup writes its rows of the partial result into
// this CTA's Q tiles (free once this CTA's last Q K^T products completed,
// which its producer signals to the partner) through distributed shared
// memory, and this CTA merges the two by the online-softmax rule and writes
// O and LSE. The last round then takes about half as long (e.g. 512 units on
// 152 SMs: 3.5 rounds instead of 4).
//
// Warp roles (12 warps, 3 warpgroups):
//   warps 0-3   softmax + epilogue for query tile 0 (one thread per row)
//   warps 4-7   softmax + epilogue for query tile 1
//   warp 8      TMA producer (one thread)
//   warp 9      TMEM allocator and MMA issuer (the whole warp, converged; one
//               elected lane issues each tcgen05 instruction)
//   warps 10-11 idle (they complete the third warpgroup)
// With 12 warps a launch gets 168 registers per thread (3 warps per SM
// sub-partition); setmaxnreg then moves registers from the control
// warpgroup (down to 72) to the softmax warpgroups (up to 216), which hold a
// 128-score row plus its packed probabilities without spilling.
// P is handed to the issuer in two halves: once the probabilities of keys
// 0-63 are stored (and O_t rescaled, if it is), the issuer runs the first
// four K = 16 products of P V while the softmax warps exponentiate keys
// 64-127; the other four follow the second hand-off. Both halves sum in the
// same order as one burst, so the result is unchanged.
// TMEM (512 columns x 128 lanes x 32 bit): S_t at column 128*t (P_t, packed
// bf16, overwrites the first 64 of those columns), O_t at 256 + d*t.
// Shared memory: Q tiles (2 x 128 x d bf16) + a ring of K/V tiles
// (kStages x 128 x d bf16), each tile stored as d/64 chunks of 128 rows x
// 128 bytes in the 128-byte swizzled layout that TMA writes and the tensor
// core reads, + one 4 KB O staging buffer per softmax warp (32 rows x 64
// columns of bf16, the same layout): the epilogue writes O there chunk by
// chunk and one lane stores each chunk with a tiled TMA store, instead of
// every thread writing its own row to global memory.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103a_ptx.cuh"

namespace fa {

// Device status word (set on a wait timeout) and the first timeout's details.
// Read and cleared by fa_get_device_status().
__device__ unsigned int g_status_word;
__device__ unsigned int g_status_info[4];

enum : unsigned int { kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3 };

template <int HD>
struct FwdCfg {
  static constexpr int kBM = 128;        // query rows per tile (tcgen05 M)
  static constexpr int kBN = 128;        // keys per K/V block
  static constexpr int kQTiles = 2;      // query tiles per CTA
  static constexpr int kChunks = HD / 64;          // 128-byte swizzle chunks per row
  static constexpr int kChunkBytes = 128 * 128;    // 128 rows x 128 bytes
  static constexpr int kTileBytes = kChunks * kChunkBytes;   // one Q, K or V tile
  static constexpr int kStages = (HD == 128) ? 4 : 8;        // K/V ring slots
  static constexpr int kSmemQ = kQTiles * kTileBytes;
  static constexpr int kSmemKV = kStages * kTileBytes;
  static constexpr int kSmemStage = 8 * 32 * 128;  // per softmax warp: 32 rows x 64 columns of bf16 O
  static constexpr int kSmemBytes = kSmemQ + kSmemKV + kSmemStage + 1024;  // + alignment slack
  static constexpr int kThreads = 384;          // 12 warps: 3 warpgroups
  // Registers per thread after the split: the two softmax warpgroups raise
  // theirs, the control warpgroup (producer, MMA issuer, two idle warps)
  // lowers its own. The launch holds 12 warps x 32 x kRegsLaunch registers;
  // the split must not need more (the host checks the built kernel's count).
  static constexpr int kRegsLaunch = 168;
  static constexpr int kRegsSoftmax = 216;
  static constexpr int kRegsControl = 72;
  static_assert(8 * kRegsSoftmax + 4 * kRegsControl <= 12 * kRegsLaunch, "register split exceeds the launch");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;         // + 128 * t
  static constexpr uint32_t kColO = 256;       // + HD * t
  static constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, HD, false, true);
};

struct FwdParams {
  __nv_bfloat16* O;
  float* LSE;
  int N;                       // query rows per head (rows of Q, O, LSE)
  int N_kv;                    // keys per K/V head
  int H;                       // query heads
  int H_kv;                    // K/V heads; query head h reads K/V head h / (H / H_kv)
  int n_kv_blocks;
  int q_blocks;                // 256-row query blocks per head
  int num_units;               // B * H * q_blocks: the (b, h, query block) units
  int num_whole;               // units walked whole (u = blockIdx.x + k * gridDim.x < num_whole)
  int split_tail;              // 1: units [num_whole, num_units) are split over CTA pairs (clusters of 2)
  float scale_log2;            // |scale| * log2(e)
  uint32_t idesc_qk;           // instruction descriptor of S = Q K^T (A negated when scale < 0)
  unsigned long long timeout_ns;
  int drop_load;               // test hook: index of a K/V load to skip, -1 = none
};

constexpr float kRescaleLog2 = 8.0f;

// Bounded wait. Returns false when the CTA is aborting (another role gave up)
// or when this wait itself ran out of time, in which case it raises the abort
// flag and records the timeout in the device status word. The flag and the
// clock are read once per kPolls polls of the barrier: a phase that completes
// while they are being read is seen only at the next poll.
template <int kPolls = 1>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned long long timeout_ns, unsigned int role) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int r = 0; r < kPolls; ++r)
      if (ptx::mbar_try_wait(bar, parity)) return true;
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
}

// Warp-uniform bounded wait for the 32 lanes of a softmax warp: returns the
// same answer in every lane, so the warp-collective TMEM instructions that
// follow are never reached by part of a warp.
template <int kPolls = 1>
__device__ __forceinline__ bool wait_warp_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                   unsigned long long timeout_ns, unsigned int role) {
  if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  const int lane = threadIdx.x & 31;
  while (true) {
#pragma unroll 1
    for (int r = 0; r < kPolls; ++r)
      if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
    int stop = 0;
    if (lane == 0) {
      if (*abort_flag) {
        stop = 1;
      } else if (ptx::globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        if (atomicCAS(&g_status_word, 0u, 1u) == 0u) {
          g_status_info[0] = role;
          g_status_info[1] = blockIdx.x;
          g_status_info[2] = blockIdx.y;
          g_status_info[3] = blockIdx.z;
        }
        __threadfence();
        stop = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
  }
}

// wait_warp_or_abort for a barrier that another CTA of the cluster arrives
// on: the wait acquires at cluster scope, so the data that CTA wrote into
// this one before arriving is visible when it returns true.
__device__ __forceinline__ bool wait_cluster_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                      unsigned long long timeout_ns, unsigned int role) {
  if (__all_sync(0xffffffffu, ptx::mbar_try_wait_cluster(bar, parity))) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  const int lane = threadIdx.x & 31;
  while (true) {
    if (__all_sync(0xffffffffu, ptx::mbar_try_wait_cluster(bar, parity))) return true;
    int stop = 0;
    if (lane == 0) {
      if (*abort_flag) {
        stop = 1;
      } else if (ptx::globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        if (atomicCAS(&g_status_word, 0u, 1u) == 0u) {
          g_status_info[0] = role;
          g_status_info[1] = blockIdx.x;
          g_status_info[2] = blockIdx.y;
          g_status_info[3] = blockIdx.z;
        }
        __threadfence();
        stop = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
  }
}

// Bounded wait used only while cleaning up after an abort: ignores the abort
// flag, gives up silently after `timeout_ns`.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long timeout_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > timeout_ns) return;
  }
}

// The split unit of this CTA's pair and this CTA's half of its key blocks
// (rank 0 the first ceil(n/2), rank 1 the rest); valid is false when the
// grid has no split units or this pair has none.
struct TailPart {
  uint32_t rank;
  int u, kb0, kb1;
  bool valid;
};

__device__ __forceinline__ TailPart tail_part(const FwdParams& p) {
  TailPart tp;
  tp.rank = p.split_tail ? ptx::cluster_ctarank() : 0u;
  tp.u = p.num_whole + static_cast<int>(blockIdx.x >> 1);
  tp.valid = p.split_tail && tp.u < p.num_units;
  const int half = (p.n_kv_blocks + 1) >> 1;
  tp.kb0 = tp.rank ? half : 0;
  tp.kb1 = tp.rank ? p.n_kv_blocks : half;
  return tp;
}

template <int HD>
__global__ void __launch_bounds__(FwdCfg<HD>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p) {
  using C = FwdCfg<HD>;
  // Bounded waits read the abort flag and the clock once per this many polls
  // (at d = 128 the hand-offs are then seen sooner; at d = 64 one poll per
  // check measured faster).
  constexpr int kPolls = HD == 128 ? 8 : 1;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q_full;
  __shared__ __align__(8) uint64_t bar_q_empty;
  __shared__ __align__(8) uint64_t bar_kv_full[C::kStages];
  __shared__ __align__(8) uint64_t bar_kv_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_s_full[2];
  __shared__ __align__(8) uint64_t bar_p_full[2];
  __shared__ __align__(8) uint64_t bar_p_half[2];   // P_t of keys 0-63 stored (and O_t rescaled)
  __shared__ __align__(8) uint64_t bar_o_full[2];
  __shared__ __align__(8) uint64_t bar_drain;
  // Split units: the partner CTA's producer arrives on bar_peer_ready when
  // its Q tiles may be overwritten; its 128 sending threads arrive on
  // bar_xfer_full once their rows of the partial result are in this CTA.
  __shared__ __align__(8) uint64_t bar_peer_ready;
  __shared__ __align__(8) uint64_t bar_xfer_full;
  __shared__ float xch_m[C::kBM], xch_l[C::kBM], xch_lo[C::kBM];
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_kv = p.n_kv_blocks;
  // Unit u is query block u % q_blocks of head u / q_blocks; this CTA takes
  // units blockIdx.x, blockIdx.x + gridDim.x, ...
  auto unit_head = [&](int u) { return u / p.q_blocks; };
  auto unit_row0 = [&](int u) { return (u - (u / p.q_blocks) * p.q_blocks) * (C::kQTiles * C::kBM); };
  auto kv_head = [&](int bh) {
    const int b = bh / p.H;
    return b * p.H_kv + (bh - b * p.H) / (p.H / p.H_kv);
  };

  // 1024-byte aligned base: the 128-byte swizzle pattern is a function of
  // the shared-memory address bits [4, 10).
  const uint32_t smem_base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = smem_base;
  const uint32_t sKV = smem_base + C::kSmemQ;
  const uint32_t sStage = sKV + C::kSmemKV;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar_q_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_q_empty), 1);
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bar_kv_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_kv_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(ptx::smem_u32(&bar_s_full[t]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_p_full[t]), C::kBM);
      ptx::mbar_init(ptx::smem_u32(&bar_p_half[t]), C::kBM);
      ptx::mbar_init(ptx::smem_u32(&bar_o_full[t]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bar_drain), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_peer_ready), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_xfer_full), C::kBM);
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
  }
  ptx::tc_fence_before();
  __syncthreads();
  // The partner's barriers must be initialised before any arrival from here.
  if (p.split_tail) ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;

  volatile int* abort_ptr = &abort_flag;

  if (warp >= 8) ptx::setmaxnreg_dec<C::kRegsControl>();
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_last();
      const uint32_t q_full = ptx::smem_u32(&bar_q_full);
      int issued = 0;       // K/V loads issued by this CTA (the ring position runs on across units)
      int q_issued = 0;     // Q loads issued (one per unit)
      bool ok = true;
      int uc = 0;
      for (int u = blockIdx.x; u < p.num_whole && ok; u += gridDim.x, ++uc) {
        const int bh = unit_head(u), bh_kv = kv_head(bh), q_row0 = unit_row0(u);
        // The previous unit's Q tiles are free once its last Q K^T products completed.
        if (uc > 0 && !wait_or_abort<kPolls>(ptx::smem_u32(&bar_q_empty), (uc - 1) & 1, abort_ptr, p.timeout_ns,
                                     kRoleProducer)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(q_full, C::kQTiles * C::kTileBytes);
        for (int t = 0; t < C::kQTiles; ++t)
          for (int c = 0; c < C::kChunks; ++c)
            ptx::tma_load_3d(sQ + t * C::kTileBytes + c * C::kChunkBytes, &tmQ, q_full, c * 64,
                             q_row0 + t * C::kBM, bh, pol_q);
        q_issued = uc + 1;
        for (int j = 0; j < n_kv && ok; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            const int it = 2 * n_kv * uc + 2 * j + kv;
            const int slot = it % C::kStages;
            const uint32_t phase = (it / C::kStages) & 1;
            if (!wait_or_abort<kPolls>(ptx::smem_u32(&bar_kv_empty[slot]), phase ^ 1u, abort_ptr, p.timeout_ns,
                               kRoleProducer)) {
              ok = false;
              break;
            }
            issued = it + 1;
            if (it == p.drop_load) continue;   // test hook: this tile never arrives
            const uint32_t full = ptx::smem_u32(&bar_kv_full[slot]);
            ptx::mbar_arrive_expect_tx(full, C::kTileBytes);
            const void* map = kv ? static_cast<const void*>(&tmV) : static_cast<const void*>(&tmK);
            for (int c = 0; c < C::kChunks; ++c)
              ptx::tma_load_3d(sKV + slot * C::kTileBytes + c * C::kChunkBytes, map, full, c * 64,
                               j * C::kBN, bh_kv, pol_kv);
          }
        }
      }
      if (const TailPart tp = tail_part(p); ok && tp.valid) {
        // The split unit: Q, then this CTA's half of the key blocks.
        const int bh = unit_head(tp.u), bh_kv = kv_head(bh), q_row0 = unit_row0(tp.u);
        if (uc > 0 && !wait_or_abort<kPolls>(ptx::smem_u32(&bar_q_empty), (uc - 1) & 1, abort_ptr, p.timeout_ns,
                                     kRoleProducer))
          ok = false;
        if (ok) {
          ptx::mbar_arrive_expect_tx(q_full, C::kQTiles * C::kTileBytes);
          for (int t = 0; t < C::kQTiles; ++t)
            for (int c = 0; c < C::kChunks; ++c)
              ptx::tma_load_3d(sQ + t * C::kTileBytes + c * C::kChunkBytes, &tmQ, q_full, c * 64,
                               q_row0 + t * C::kBM, bh, pol_q);
          q_issued = uc + 1;
        }
        for (int j = tp.kb0; j < tp.kb1 && ok; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            const int it = 2 * n_kv * uc + 2 * (j - tp.kb0) + kv;
            const int slot = it % C::kStages;
            const uint32_t phase = (it / C::kStages) & 1;
            if (!wait_or_abort<kPolls>(ptx::smem_u32(&bar_kv_empty[slot]), phase ^ 1u, abort_ptr, p.timeout_ns,
                               kRoleProducer)) {
              ok = false;
              break;
            }
            issued = it + 1;
            if (it == p.drop_load) continue;   // test hook: this tile never arrives
            const uint32_t full = ptx::smem_u32(&bar_kv_full[slot]);
            ptx::mbar_arrive_expect_tx(full, C::kTileBytes);
            const void* map = kv ? static_cast<const void*>(&tmV) : static_cast<const void*>(&tmK);
            for (int c = 0; c < C::kChunks; ++c)
              ptx::tma_load_3d(sKV + slot * C::kTileBytes + c * C::kChunkBytes, map, full, c * 64,
                               j * C::kBN, bh_kv, pol_kv);
          }
        }
        // Once its Q K^T products have completed, the partner may write its
        // partial result over this CTA's Q tiles.
        if (ok && wait_or_abort<kPolls>(ptx::smem_u32(&bar_q_empty), uc & 1, abort_ptr, p.timeout_ns, kRoleProducer))
          ptx::mbar_arrive_remote(ptx::mapa_shared(ptx::smem_u32(&bar_peer_ready), tp.rank ^ 1u));
      }
      if (!ok || *abort_ptr) {
        // Let every copy this thread started land before the CTA exits.
        if (q_issued > 0) drain_wait(q_full, (q_issued - 1) & 1, p.timeout_ns);
        const int first = issued > C::kStages ? issued - C::kStages : 0;
        for (int it = first; it < issued; ++it) {
          if (it == p.drop_load) continue;
          drain_wait(ptx::smem_u32(&bar_kv_full[it % C::kStages]), (it / C::kStages) & 1, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this code converged: waits are warp-uniform and one
    // elected lane issues every tcgen05 instruction. A lone diverged lane
    // issues far more slowly while the softmax warps of its sub-partition
    // compete for issue slots.
    // P V for query tile t from the V tile loaded as the it-th K/V load (P_t
    // sits in the S_t columns), over keys [64 half, 64 half + 64): four
    // K = 16 products; the first product of a unit overwrites O_t.
    auto issue_pv_half = [&](int t, int it, bool accumulate, int half) {
      const uint32_t v_tile = sKV + (it % C::kStages) * C::kTileBytes;
      const uint32_t d_tmem = tmem_base + C::kColO + HD * t;
      const uint32_t a_tmem = tmem_base + C::kColS + 128 * t;
      static_assert(C::kBN == 128, "two bursts of four K = 16 products");
      const uint64_t b_desc = ptx::desc_mnmajor_sw128(v_tile, C::kChunkBytes);
      if (half == 0)
        ptx::mma_ts_k64half_warp<0>(d_tmem, a_tmem, ptx::desc_lo(b_desc), ptx::desc_hi(b_desc), C::kIdescPV,
                                    accumulate ? 1u : 0u);
      else
        ptx::mma_ts_k64half_warp<1>(d_tmem, a_tmem, ptx::desc_lo(b_desc), ptx::desc_hi(b_desc), C::kIdescPV, 1u);
    };
    // S_t = Q_t K^T with the K tile of the it-th K/V load.
    auto issue_qk = [&](int t, int it) {
      const uint32_t k_tile = sKV + (it % C::kStages) * C::kTileBytes;
      const uint32_t q_tile = sQ + t * C::kTileBytes;
      const uint32_t d_tmem = tmem_base + C::kColS + 128 * t;
      const uint64_t a_desc = ptx::desc_kmajor_sw128(q_tile), b_desc = ptx::desc_kmajor_sw128(k_tile);
      if constexpr (HD == 128)
        ptx::mma_ss_k128_warp(d_tmem, ptx::desc_lo(a_desc), ptx::desc_lo(b_desc), ptx::desc_hi(a_desc), p.idesc_qk, 0u);
      else
        ptx::mma_ss_k64_warp(d_tmem, ptx::desc_lo(a_desc), ptx::desc_lo(b_desc), ptx::desc_hi(a_desc), p.idesc_qk, 0u);
    };
    // Per unit: Q and K_0 are waited for here; every later K_{j+1} and V_j
    // is waited for by the softmax warps before their first hand-off for
    // block j (p_half), so the p_half / p_full waits below imply those tiles
    // have landed. An mbarrier wait in this warp stalls the queued
    // tensor-core work, so it does as few as it can. g counts the key blocks
    // of all units so far (the phase of s_full, p_half and p_full).
    bool ok = true;
    int g = 0, uc = 0;
    for (int u = blockIdx.x; u < p.num_whole && ok; u += gridDim.x, ++uc) {
      const int it0 = 2 * n_kv * uc;
      ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_q_full), uc & 1, abort_ptr, p.timeout_ns, kRoleMma);
      if (ok)
        ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_kv_full[it0 % C::kStages]), (it0 / C::kStages) & 1, abort_ptr,
                                p.timeout_ns, kRoleMma);
      for (int j = 0; j < n_kv && ok; ++j, ++g) {
        const int itK = it0 + 2 * j;
        ptx::tc_fence_after();
        for (int t = 0; t < 2 && ok; ++t) {
          if (j > 0) {
            ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_p_half[t]), (g - 1) & 1, abort_ptr, p.timeout_ns, kRoleMma);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_pv_half(t, itK - 1, j > 1, 0);
            ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_p_full[t]), (g - 1) & 1, abort_ptr, p.timeout_ns, kRoleMma);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_pv_half(t, itK - 1, true, 1);
            if (t == 1) ptx::mma_commit_warp(ptx::smem_u32(&bar_kv_empty[(itK - 1) % C::kStages]));
          }
          issue_qk(t, itK);
          ptx::mma_commit_warp(ptx::smem_u32(&bar_s_full[t]));
        }
        if (ok) {
          ptx::mma_commit_warp(ptx::smem_u32(&bar_kv_empty[itK % C::kStages]));
          // The unit's last Q K^T products are issued: Q is free when they complete.
          if (j == n_kv - 1) ptx::mma_commit_warp(ptx::smem_u32(&bar_q_empty));
        }
      }
      // The last key block's P V.
      const int itV = it0 + 2 * n_kv - 1;
      for (int t = 0; t < 2 && ok; ++t) {
        ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_p_half[t]), (g - 1) & 1, abort_ptr, p.timeout_ns, kRoleMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_pv_half(t, itV, n_kv > 1, 0);
        ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_p_full[t]), (g - 1) & 1, abort_ptr, p.timeout_ns, kRoleMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_pv_half(t, itV, true, 1);
        ptx::mma_commit_warp(ptx::smem_u32(&bar_o_full[t]));
        if (t == 1) ptx::mma_commit_warp(ptx::smem_u32(&bar_kv_empty[itV % C::kStages]));
      }
    }
    if (const TailPart tp = tail_part(p); ok && tp.valid) {
      // The split unit: the same sequence over this CTA's half of the key blocks.
      const int it0 = 2 * n_kv * uc;
      const int nb = tp.kb1 - tp.kb0;
      ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_q_full), uc & 1, abort_ptr, p.timeout_ns, kRoleMma);
      if (ok)
        ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_kv_full[it0 % C::kStages]), (it0 / C::kStages) & 1, abort_ptr,
                                p.timeout_ns, kRoleMma);
      for (int j = 0; j < nb && ok; ++j, ++g) {
        const int itK = it0 + 2 * j;
        ptx::tc_fence_after();
        for (int t = 0; t < 2 && ok; ++t) {
          if (j > 0) {
            ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_p_half[t]), (g - 1) & 1, abort_ptr, p.timeout_ns, kRoleMma);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_pv_half(t, itK - 1, j > 1, 0);
            ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_p_full[t]), (g - 1) & 1, abort_ptr, p.timeout_ns, kRoleMma);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_pv_half(t, itK - 1, true, 1);
            if (t == 1) ptx::mma_commit_warp(ptx::smem_u32(&bar_kv_empty[(itK - 1) % C::kStages]));
          }
          issue_qk(t, itK);
          ptx::mma_commit_warp(ptx::smem_u32(&bar_s_full[t]));
        }
        if (ok) {
          ptx::mma_commit_warp(ptx::smem_u32(&bar_kv_empty[itK % C::kStages]));
          if (j == nb - 1) ptx::mma_commit_warp(ptx::smem_u32(&bar_q_empty));
        }
      }
      const int itV = it0 + 2 * nb - 1;
      for (int t = 0; t < 2 && ok; ++t) {
        ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_p_half[t]), (g - 1) & 1, abort_ptr, p.timeout_ns, kRoleMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_pv_half(t, itV, nb > 1, 0);
        ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_p_full[t]), (g - 1) & 1, abort_ptr, p.timeout_ns, kRoleMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_pv_half(t, itV, true, 1);
        ptx::mma_commit_warp(ptx::smem_u32(&bar_o_full[t]));
        if (t == 1) ptx::mma_commit_warp(ptx::smem_u32(&bar_kv_empty[itV % C::kStages]));
      }
    }
    if (!ok) {
      // Wait for every MMA already issued before TMEM is freed.
      ptx::mma_commit_warp(ptx::smem_u32(&bar_drain));
      drain_wait(ptx::smem_u32(&bar_drain), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax + epilogue
    ptx::setmaxnreg_inc<C::kRegsSoftmax>();
    const int t = warp >> 2;                 // query tile
    const int quarter = warp & 3;            // TMEM lane quarter
    const int row = quarter * 32 + lane;     // row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem_base + lane_addr + C::kColS + 128 * t;
    const uint32_t tO = tmem_base + lane_addr + C::kColO + HD * t;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g = 0, uc = 0;      // key blocks and units so far (barrier phases)
    for (int u = blockIdx.x; u < p.num_whole && ok; u += gridDim.x, ++uc) {
    const int it0 = 2 * n_kv * uc;
    float m_use = 0.f;      // raw-score maximum the exponentials are taken against
    float l = 0.f;          // running sum of exp, relative to m_use (for LSE)
    float lo = 0.f;         // the same with each block's largest term as P V sees it (for O)
    for (int j = 0; j < n_kv; ++j, ++g) {
      // V_j and K_{j+1} must have landed before this block's hand-off (see
      // the MMA issuer); waiting here costs nothing, S_t(j) comes later.
      {
        const int itV = it0 + 2 * j + 1;
        ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_kv_full[itV % C::kStages]), (itV / C::kStages) & 1, abort_ptr,
                                p.timeout_ns, kRoleSoftmax);
        if (ok && j + 1 < n_kv)
          ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_kv_full[(itV + 1) % C::kStages]), ((itV + 1) / C::kStages) & 1,
                                  abort_ptr, p.timeout_ns, kRoleSoftmax);
        if (!ok) break;
      }
      ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_s_full[t]), g & 1, abort_ptr, p.timeout_ns, kRoleSoftmax);
      if (!ok) break;
      ptx::tc_fence_after();
      // The loads also reduce each 32-column piece to its maximum, which is
      // the row maximum of a full block. In the ragged last block the
      // columns past N hold scores of zero-filled keys, so that block masks
      // them to -inf and takes the maximum itself.
      uint32_t s[4][32];
      float mr[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32_max(tS + 32 * c, s[c], mr[c]);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        ptx::reg_fence32(s[c]);
        ptx::reg_fence1(mr[c]);
      }

      const int valid = p.N_kv - j * C::kBN;    // keys of this block that exist
      const bool ragged = valid < C::kBN;
      float mt;
      if (!ragged) {
        mt = ptx::max3(mr[0], mr[1], fmaxf(mr[2], mr[3]));
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i >= valid) s[c][i] = __float_as_uint(-INFINITY);
        // Row maximum: 8 independent chains of 3-input max, then a small tree.
        float mc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = k >> 1, b = (k & 1) * 16;
          mc[k] = fmaxf(__uint_as_float(s[c][b]), __uint_as_float(s[c][b + 1]));
#pragma unroll
          for (int i = 2; i < 16; i += 2)
            mc[k] = ptx::max3(mc[k], __uint_as_float(s[c][b + i]), __uint_as_float(s[c][b + i + 1]));
        }
        mt = ptx::max3(ptx::max3(mc[0], mc[1], mc[2]), ptx::max3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
      }

      float alpha = 1.f;
      bool rescale_o = false;
      if (j == 0) {
        m_use = mt;
      } else {
        const bool need = (mt - m_use) * sl2 > kRescaleLog2;
        rescale_o = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = ptx::ex2_approx((m_use - mt) * sl2);
          m_use = mt;
        }
      }
      // P = 2^(s*scale*log2e - m*scale*log2e): pairs through the f32x2 FMA,
      // MUFU ex2 per element, 4 independent f32x2 partial sums, bf16x2 pack.
      const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
      const float neg_m = -m_use * sl2;
      const uint64_t negmx2 = ptx::f2_pack(neg_m, neg_m);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[2][32];
      // At d = 64 the pass is written twice, with and without the ragged
      // block's masking (+6 % at d = 64; the same split cost 3 % at d = 128,
      // which keeps one loop with the test inside).
      if constexpr (HD == 64) {
        if (!ragged) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0, x1;
              ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])), sl2x2,
                                         negmx2),
                             x0, x1);
              float p0 = ptx::ex2_approx(x0);
              float p1 = ptx::ex2_approx(x1);
              acc[(i >> 1) & 3] = ptx::f2_add(acc[(i >> 1) & 3], ptx::f2_pack(p0, p1));
              pk[c >> 1][(c & 1) * 16 + (i >> 1)] = ptx::pack_bf16x2(p0, p1);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0, x1;
              ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])), sl2x2,
                                         negmx2),
                             x0, x1);
              float p0 = ptx::ex2_approx(x0);
              float p1 = ptx::ex2_approx(x1);
              if (32 * c + i >= valid) p0 = 0.f;   // keys past N: exact zeros (also when scale == 0)
              if (32 * c + i + 1 >= valid) p1 = 0.f;
              acc[(i >> 1) & 3] = ptx::f2_add(acc[(i >> 1) & 3], ptx::f2_pack(p0, p1));
              pk[c >> 1][(c & 1) * 16 + (i >> 1)] = ptx::pack_bf16x2(p0, p1);
            }
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float x0, x1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])), sl2x2,
                                       negmx2),
                           x0, x1);
            float p0 = ptx::ex2_approx(x0);
            float p1 = ptx::ex2_approx(x1);
            if (ragged) {   // exact zeros for keys past N (also when scale == 0)
              if (32 * c + i >= valid) p0 = 0.f;
              if (32 * c + i + 1 >= valid) p1 = 0.f;
            }
            acc[(i >> 1) & 3] = ptx::f2_add(acc[(i >> 1) & 3], ptx::f2_pack(p0, p1));
            pk[c >> 1][(c & 1) * 16 + (i >> 1)] = ptx::pack_bf16x2(p0, p1);
          }
        }
      }
      if (rescale_o) {
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + 32 * c, o);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          ptx::tmem_st32(tO + 32 * c, o);
        }
      }
      ptx::tmem_st32(tS, pk[0]);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bar_p_half[t]));
      if constexpr (HD == 64) {
        if (!ragged) {
#pragma unroll
          for (int c = 2; c < 4; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0, x1;
              ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])), sl2x2,
                                         negmx2),
                             x0, x1);
              float p0 = ptx::ex2_approx(x0);
              float p1 = ptx::ex2_approx(x1);
              acc[(i >> 1) & 3] = ptx::f2_add(acc[(i >> 1) & 3], ptx::f2_pack(p0, p1));
              pk[c >> 1][(c & 1) * 16 + (i >> 1)] = ptx::pack_bf16x2(p0, p1);
            }
          }
        } else {
#pragma unroll
          for (int c = 2; c < 4; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0, x1;
              ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])), sl2x2,
                                         negmx2),
                             x0, x1);
              float p0 = ptx::ex2_approx(x0);
              float p1 = ptx::ex2_approx(x1);
              if (32 * c + i >= valid) p0 = 0.f;   // keys past N: exact zeros (also when scale == 0)
              if (32 * c + i + 1 >= valid) p1 = 0.f;
              acc[(i >> 1) & 3] = ptx::f2_add(acc[(i >> 1) & 3], ptx::f2_pack(p0, p1));
              pk[c >> 1][(c & 1) * 16 + (i >> 1)] = ptx::pack_bf16x2(p0, p1);
            }
          }
        }
      } else {
#pragma unroll
        for (int c = 2; c < 4; ++c) {
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float x0, x1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])), sl2x2,
                                       negmx2),
                           x0, x1);
            float p0 = ptx::ex2_approx(x0);
            float p1 = ptx::ex2_approx(x1);
            if (ragged) {   // exact zeros for keys past N (also when scale == 0)
              if (32 * c + i >= valid) p0 = 0.f;
              if (32 * c + i + 1 >= valid) p1 = 0.f;
            }
            acc[(i >> 1) & 3] = ptx::f2_add(acc[(i >> 1) & 3], ptx::f2_pack(p0, p1));
            pk[c >> 1][(c & 1) * 16 + (i >> 1)] = ptx::pack_bf16x2(p0, p1);
          }
        }
      }
      float sum;
      {
        float a0, a1, b0, b1;
        ptx::f2_unpack(ptx::f2_add(acc[0], acc[1]), a0, a1);
        ptx::f2_unpack(ptx::f2_add(acc[2], acc[3]), b0, b1);
        sum = (a0 + a1) + (b0 + b1);
      }
      // The P V product sees every probability rounded to bf16. The largest
      // one of the block (the score equal to mt, recomputed here exactly as
      // the loop above computes it) enters the normaliser of O the same way,
      // so that a row dominated by one key weights it exactly 1; l itself,
      // which LSE needs, stays the sum of the unrounded terms.
      const float pmax = ptx::ex2_approx(fmaf(mt, sl2, neg_m));
      l = l * alpha + sum;
      lo = lo * alpha + (sum + (ptx::round_bf16(pmax) - pmax));
      ptx::tmem_st32(tS + 32, pk[1]);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bar_p_full[t]));
    }
    if (ok) ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_o_full[t]), uc & 1, abort_ptr, p.timeout_ns, kRoleSoftmax);
    if (ok) {
      ptx::tc_fence_after();
      const int bh = unit_head(u);
      const int row0 = unit_row0(u) + t * C::kBM + quarter * 32;   // this warp's first row
      const int grow = row0 + lane;
      const bool in_range = grow < p.N;
      const float inv_l = 1.f / lo;
      // O goes out through shared memory: each warp writes its 32 rows of a
      // 64-column chunk in the 128-byte swizzled layout, then one lane stores
      // them with a tiled TMA store (rows past N are not written).
      if (row0 < p.N) {
        const uint32_t stage = sStage + static_cast<uint32_t>(warp) * (32u * 128u);
#pragma unroll
        for (int k = 0; k < HD / 64; ++k) {
          // The staging rows are free once this warp's previous store has read them.
          if (lane == 0) ptx::bulk_wait_group_read0();
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + 64 * k + 32 * h, o);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(o);
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[i] = ptx::pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
            const uint32_t row_addr = stage + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint32_t unit = 4u * h + v;      // 16-byte unit within the 128-byte row
              const uint32_t addr = row_addr + ((unit ^ static_cast<uint32_t>(lane & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(packed[4 * v]),
                           "r"(packed[4 * v + 1]), "r"(packed[4 * v + 2]), "r"(packed[4 * v + 3])
                           : "memory");
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&tmO, stage, 64 * k, row0, bh);
            ptx::bulk_commit_group();
          }
        }
      }
      if (in_range) {
        // LSE = scale * m + ln l = (scale*log2(e) * m + log2 l) * ln 2
        p.LSE[static_cast<size_t>(bh) * p.N + grow] = (m_use * sl2 + __log2f(l)) * 0.69314718055994530942f;
      }
    }
    }   // units
    if (const TailPart tp = tail_part(p); ok && tp.valid) {
      // The split unit: the block loop over this CTA's half of the keys, then
      // the exchange with the partner.
      const int it0 = 2 * n_kv * uc;
      float m_use = 0.f, l = 0.f, lo = 0.f;
      for (int j = tp.kb0; j < tp.kb1; ++j, ++g) {
        // V_j and K_{j+1} must have landed before this block's hand-off (see
        // the MMA issuer); waiting here costs nothing, S_t(j) comes later.
        {
          const int itV = it0 + 2 * (j - tp.kb0) + 1;
          ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_kv_full[itV % C::kStages]), (itV / C::kStages) & 1, abort_ptr,
                                  p.timeout_ns, kRoleSoftmax);
          if (ok && j + 1 < tp.kb1)
            ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_kv_full[(itV + 1) % C::kStages]), ((itV + 1) / C::kStages) & 1,
                                    abort_ptr, p.timeout_ns, kRoleSoftmax);
          if (!ok) break;
        }
        ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_s_full[t]), g & 1, abort_ptr, p.timeout_ns, kRoleSoftmax);
        if (!ok) break;
        ptx::tc_fence_after();
        // The loads also reduce each 32-column piece to its maximum, which is
        // the row maximum of a full block. In the ragged last block the
        // columns past N hold scores of zero-filled keys, so that block masks
        // them to -inf and takes the maximum itself.
        uint32_t s[4][32];
        float mr[4];
  #pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32_max(tS + 32 * c, s[c], mr[c]);
        ptx::tmem_ld_wait();
  #pragma unroll
        for (int c = 0; c < 4; ++c) {
          ptx::reg_fence32(s[c]);
          ptx::reg_fence1(mr[c]);
        }

        const int valid = p.N_kv - j * C::kBN;    // keys of this block that exist
        const bool ragged = valid < C::kBN;
        float mt;
        if (!ragged) {
          mt = ptx::max3(mr[0], mr[1], fmaxf(mr[2], mr[3]));
        } else {
  #pragma unroll
          for (int c = 0; c < 4; ++c)
  #pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * c + i >= valid) s[c][i] = __float_as_uint(-INFINITY);
          // Row maximum: 8 independent chains of 3-input max, then a small tree.
          float mc[8];
  #pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int c = k >> 1, b = (k & 1) * 16;
            mc[k] = fmaxf(__uint_as_float(s[c][b]), __uint_as_float(s[c][b + 1]));
  #pragma unroll
            for (int i = 2; i < 16; i += 2)
              mc[k] = ptx::max3(mc[k], __uint_as_float(s[c][b + i]), __uint_as_float(s[c][b + i + 1]));
          }
          mt = ptx::max3(ptx::max3(mc[0], mc[1], mc[2]), ptx::max3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
        }

        float alpha = 1.f;
        bool rescale_o = false;
        if (j == tp.kb0) {
          m_use = mt;
        } else {
          const bool need = (mt - m_use) * sl2 > kRescaleLog2;
          rescale_o = __any_sync(0xffffffffu, need);
          if (need) {
            alpha = ptx::ex2_approx((m_use - mt) * sl2);
            m_use = mt;
          }
        }
        // P = 2^(s*scale*log2e - m*scale*log2e): pairs through the f32x2 FMA,
        // MUFU ex2 per element, 4 independent f32x2 partial sums, bf16x2 pack.
        const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
        const float neg_m = -m_use * sl2;
        const uint64_t negmx2 = ptx::f2_pack(neg_m, neg_m);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[2][32];
  #pragma unroll
        for (int c = 0; c < 2; ++c) {
  #pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float x0, x1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])), sl2x2,
                                       negmx2),
                           x0, x1);
            float p0 = ptx::ex2_approx(x0);
            float p1 = ptx::ex2_approx(x1);
            if (ragged) {   // exact zeros for keys past N (also when scale == 0)
              if (32 * c + i >= valid) p0 = 0.f;
              if (32 * c + i + 1 >= valid) p1 = 0.f;
            }
            acc[(i >> 1) & 3] = ptx::f2_add(acc[(i >> 1) & 3], ptx::f2_pack(p0, p1));
            pk[c >> 1][(c & 1) * 16 + (i >> 1)] = ptx::pack_bf16x2(p0, p1);
          }
        }
        if (rescale_o) {
  #pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + 32 * c, o);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(o);
  #pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            ptx::tmem_st32(tO + 32 * c, o);
          }
        }
        ptx::tmem_st32(tS, pk[0]);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&bar_p_half[t]));
  #pragma unroll
        for (int c = 2; c < 4; ++c) {
  #pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float x0, x1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])), sl2x2,
                                       negmx2),
                           x0, x1);
            float p0 = ptx::ex2_approx(x0);
            float p1 = ptx::ex2_approx(x1);
            if (ragged) {   // exact zeros for keys past N (also when scale == 0)
              if (32 * c + i >= valid) p0 = 0.f;
              if (32 * c + i + 1 >= valid) p1 = 0.f;
            }
            acc[(i >> 1) & 3] = ptx::f2_add(acc[(i >> 1) & 3], ptx::f2_pack(p0, p1));
            pk[c >> 1][(c & 1) * 16 + (i >> 1)] = ptx::pack_bf16x2(p0, p1);
          }
        }
        float sum;
        {
          float a0, a1, b0, b1;
          ptx::f2_unpack(ptx::f2_add(acc[0], acc[1]), a0, a1);
          ptx::f2_unpack(ptx::f2_add(acc[2], acc[3]), b0, b1);
          sum = (a0 + a1) + (b0 + b1);
        }
        // The P V product sees every probability rounded to bf16. The largest
        // one of the block (the score equal to mt, recomputed here exactly as
        // the loop above computes it) enters the normaliser of O the same way,
        // so that a row dominated by one key weights it exactly 1; l itself,
        // which LSE needs, stays the sum of the unrounded terms.
        const float pmax = ptx::ex2_approx(fmaf(mt, sl2, neg_m));
        l = l * alpha + sum;
        lo = lo * alpha + (sum + (ptx::round_bf16(pmax) - pmax));
        ptx::tmem_st32(tS + 32, pk[1]);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&bar_p_full[t]));
      }
      if (ok) ok = wait_warp_or_abort<kPolls>(ptx::smem_u32(&bar_o_full[t]), uc & 1, abort_ptr, p.timeout_ns, kRoleSoftmax);
      const int bh = unit_head(tp.u);
      const int grow = unit_row0(tp.u) + t * C::kBM + row;
      if (ok && t != static_cast<int>(tp.rank)) {
        // The tile the partner finalises: send this CTA's partial result for
        // it (unnormalised O relative to m_use, and m_use, l, lo) into the
        // partner's Q tiles (free once its producer says so), as float32
        // [d][128 rows], then arrive on its bar_xfer_full.
        ok = wait_cluster_or_abort(ptx::smem_u32(&bar_peer_ready), 0, abort_ptr, p.timeout_ns, kRoleSoftmax);
        if (ok) {
          ptx::tc_fence_after();
          const uint32_t peer = tp.rank ^ 1u;
          const uint32_t dst = ptx::mapa_shared(sQ, peer) + static_cast<uint32_t>(row) * 4u;
#pragma unroll 1
          for (int c = 0; c < HD / 8; ++c) {
            uint32_t o[8];
            ptx::tmem_ld8(tO + 8 * c, o);
            ptx::tmem_ld_wait();
            ptx::reg_fence8(o);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              ptx::st_shared_cluster_f32(dst + static_cast<uint32_t>((8 * c + i) * C::kBM * 4), __uint_as_float(o[i]));
          }
          ptx::st_shared_cluster_f32(ptx::mapa_shared(ptx::smem_u32(&xch_m[row]), peer), m_use);
          ptx::st_shared_cluster_f32(ptx::mapa_shared(ptx::smem_u32(&xch_l[row]), peer), l);
          ptx::st_shared_cluster_f32(ptx::mapa_shared(ptx::smem_u32(&xch_lo[row]), peer), lo);
          ptx::mbar_arrive_remote(ptx::mapa_shared(ptx::smem_u32(&bar_xfer_full), peer));
        }
      } else if (ok) {
        // The tile this CTA finalises: merge the partner's partial result
        // over the other half of the keys with this CTA's ("Flash Attention
        // (FA1)", derivation steps 4-5): with m = max(m_a, m_b) and
        // a_x = 2^{scale log2(e) (m_x - m)}, O = a_a O_a + a_b O_b, and l, lo
        // alike.
        ok = wait_cluster_or_abort(ptx::smem_u32(&bar_xfer_full), 0, abort_ptr, p.timeout_ns, kRoleSoftmax);
        if (ok) {
          ptx::tc_fence_after();
          const bool in_range = grow < p.N;
          __nv_bfloat16* orow = p.O + (static_cast<size_t>(bh) * p.N + grow) * HD;
          const float m_b = xch_m[row];
          const float m = fmaxf(m_use, m_b);
          const float a_a = ptx::ex2_approx((m_use - m) * sl2);
          const float a_b = ptx::ex2_approx((m_b - m) * sl2);
          const float l_all = a_a * l + a_b * xch_l[row];
          const float inv_l = 1.f / (a_a * lo + a_b * xch_lo[row]);
          const float* part = reinterpret_cast<const float*>(smem_raw + (sQ - ptx::smem_u32(smem_raw)));
#pragma unroll 1
          for (int c = 0; c < HD / 8; ++c) {
            uint32_t o[8];
            ptx::tmem_ld8(tO + 8 * c, o);
            ptx::tmem_ld_wait();
            ptx::reg_fence8(o);
            uint32_t packed[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float x0 = fmaf(a_a, __uint_as_float(o[2 * i]), a_b * part[(8 * c + 2 * i) * C::kBM + row]);
              const float x1 = fmaf(a_a, __uint_as_float(o[2 * i + 1]), a_b * part[(8 * c + 2 * i + 1) * C::kBM + row]);
              packed[i] = ptx::pack_bf16x2(x0 * inv_l, x1 * inv_l);
            }
            if (in_range)
              *reinterpret_cast<uint4*>(orow + 8 * c) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          }
          if (in_range)
            p.LSE[static_cast<size_t>(bh) * p.N + grow] = (m * sl2 + __log2f(l_all)) * 0.69314718055994530942f;
        }
      }
    }
  }

  // The O stores must have read the staging rows before the CTA's shared
  // memory is released.
  if (warp < 8 && lane == 0) ptx::bulk_wait_group_read0();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
  // Neither CTA of a pair exits while the other may still write into it.
  // Every wait above is bounded, so every thread of both CTAs gets here.
  if (p.split_tail) ptx::cluster_sync();
}

}  // namespace fa
