// Exact attention for short query blocks against long key/value sequences
// with shared K/V heads: the decode (generation) shape. sm_103a, tcgen05 +
// TMEM + TMA.
//
// What is computed is the forward's definition: for query head h and K/V
// head h / G (G = H / H_kv query heads share one K/V head, the grouping of
// "FlashAttention：IO 感知的精确注意力", "与其他知识点的关系"),
// O = softmax(scale Q K^T) V and LSE per query row, every query row
// attending to all N_kv keys.
//
// Decode is bandwidth-bound ("常见误区" on the same page): the K/V bytes
// dominate. Two things keep all SMs streaming them:
//  * Packing. The query rows of the G heads that share a K/V head fill one
//    128-row tile (hp = min(G, 128 / N_q) heads of N_q rows each; one TMA box
//    {64, N_q, hp} loads them), so each K/V tile is read once per group
//    rather than once per query head.
//  * Split keys. The key blocks of a (b, K/V head, tile) are cut into
//    num_splits contiguous ranges, one CTA each. A CTA's partial result over
//    its range (O normalised by its own l, and its LSE) goes to a float32
//    workspace, and decode_merge_kernel combines the partials with the
//    online-softmax rule of "Flash Attention (FA1)", derivation steps 4-5:
//    LSE = ln sum_s e^{LSE_s}, O = sum_s e^{LSE_s - LSE} O_s.
//    With one split the CTA writes O and LSE directly.
//
// Per CTA (256 threads, 2 warpgroups): warps 0-3 run the softmax and
// epilogue of the one tile (one thread per row), warp 4 is the TMA producer,
// warp 5 allocates TMEM and issues the MMAs (converged, one elected lane
// issuing), warps 6-7 are idle. Two CTAs per SM launch with 128 registers per
// thread; setmaxnreg moves registers from the control warpgroup (down to 56)
// to the softmax warpgroup (up to 200), which then holds a 128-score row and
// its packed probabilities without spilling. TMEM: S at
// column 0 (P, packed bf16, over its
// first 64 columns), O at column 128. The per-block update is the forward
// kernel's, including the lazy rescale. With a single tile, a CTA's QK^T,
// softmax and PV of a block run one after another; two CTAs per SM (a
// 2-slot K/V ring each) overlap one CTA's softmax with the other's loads and
// MMAs.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

enum : unsigned int { kRoleDecProducer = 10, kRoleDecMma = 11, kRoleDecSoftmax = 12 };

template <int HD>
struct DecCfg {
  static constexpr int kBM = 128;
  static constexpr int kBN = 128;
  static constexpr int kChunks = HD / 64;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = (HD == 128) ? 2 : 4;      // K/V ring slots
  static constexpr int kCtasPerSm = 2;                       // 2 x (Q + ring) fits shared memory, 2 x 256 TMEM
  static constexpr int kSmemBytes = kTileBytes + kStages * kTileBytes + 1024;
  static constexpr int kThreads = 256;                       // 8 warps: 2 warpgroups
  // Registers per thread after the split: the softmax warpgroup raises its
  // own, the control warpgroup (producer, MMA issuer, two idle warps) lowers
  // its own. Two CTAs per SM launch with 128 registers per thread; the split
  // must not need more (the host checks the built kernel's count).
  static constexpr int kRegsLaunch = 128;
  static constexpr int kRegsSoftmax = 200;
  static constexpr int kRegsControl = 56;
  static_assert(4 * kRegsSoftmax + 4 * kRegsControl <= 8 * kRegsLaunch, "register split exceeds the launch");
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = 128;
  static constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, HD, false, true);
};

struct DecParams {
  __nv_bfloat16* O;       // [B, H, N_q, d] (num_splits == 1 and !f32_out)
  float* LSE;             // [B, H, N_q]    (num_splits == 1 and !f32_out)
  float* O_part;          // [num_splits][B*H*N_q][d] (num_splits > 1 or f32_out)
  float* LSE_part;        // [num_splits][B*H*N_q]
  int f32_out;            // 1: results stay float32 (normalised O and LSE) in O_part / LSE_part
  int N_q;
  int N_kv;
  int H;
  int H_kv;
  int G;                  // H / H_kv
  int hp;                 // query heads packed per tile (1 when N_q > 128)
  int box_q;              // query rows per head in a tile: N_q, or 128 when N_q > 128
  int q_blocks;           // 128-row query blocks per head: 1, or ceil(N_q / 128) when N_q > 128
  int tiles_per_group;    // ceil(G / hp) * q_blocks
  int n_kv_blocks;
  int blocks_per_split;
  int num_splits;
  float scale_log2;            // |scale| * log2(e)
  uint32_t idesc_qk;           // instruction descriptor of S = Q K^T (A negated when scale < 0)
  unsigned long long timeout_ns;
  int drop_load;          // test hook: index of a K/V load (within a CTA's range) to skip, -1 = none
};

template <int HD>
__global__ void __launch_bounds__(DecCfg<HD>::kThreads, DecCfg<HD>::kCtasPerSm)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const DecParams p) {
  using C = DecCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q_full;
  __shared__ __align__(8) uint64_t bar_kv_full[C::kStages];
  __shared__ __align__(8) uint64_t bar_kv_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_s_full;
  __shared__ __align__(8) uint64_t bar_p_full;
  __shared__ __align__(8) uint64_t bar_o_full;
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tile = blockIdx.x / p.num_splits;
  const int split = blockIdx.x - tile * p.num_splits;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int head_tile = tile / p.q_blocks;
  const int q0 = (tile - head_tile * p.q_blocks) * C::kBM;      // first query row of the tile
  const int g0 = head_tile * p.hp;                              // first query head of the group in this tile
  const int nh = min(p.hp, p.G - g0);                           // query heads in this tile
  const int rows = p.q_blocks == 1 ? nh * p.N_q : min(C::kBM, p.N_q - q0);   // tile rows that are real
  const int j0 = split * p.blocks_per_split;
  const int j1 = min(p.n_kv_blocks, j0 + p.blocks_per_split);
  const int n = j1 - j0;                                        // key blocks of this CTA (>= 1)
  const int bh_kv = b * p.H_kv + kvh;
  const int bh_q0 = b * p.H + kvh * p.G + g0;                   // first query head, flattened

  const uint32_t smem_base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = smem_base;
  const uint32_t sKV = smem_base + C::kTileBytes;
  uint8_t* q_generic = smem_raw + (sQ - ptx::smem_u32(smem_raw));

  // Rows of the Q tile that no query fills are zero, so that their scores are
  // finite; they are never stored.
  const int box_rows = p.hp * p.box_q;
  for (int c = 0; c < C::kChunks; ++c)
    for (int i = threadIdx.x; i < (C::kBM - box_rows) * 8; i += C::kThreads)
      reinterpret_cast<uint4*>(q_generic + c * C::kChunkBytes + box_rows * 128)[i] = make_uint4(0u, 0u, 0u, 0u);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar_q_full), 1);
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bar_kv_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bar_kv_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bar_s_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_p_full), C::kBM);
    ptx::mbar_init(ptx::smem_u32(&bar_o_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bar_drain), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_base_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  volatile int* abort_ptr = &abort_flag;

  if (warp >= 4) ptx::setmaxnreg_dec<C::kRegsControl>();
  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_first();   // each K/V tile is read by one CTA
      const uint32_t q_full = ptx::smem_u32(&bar_q_full);
      ptx::mbar_arrive_expect_tx(q_full, C::kChunks * 128 * box_rows);
      for (int c = 0; c < C::kChunks; ++c)
        ptx::tma_load_3d(sQ + c * C::kChunkBytes, &tmQ, q_full, c * 64, q0, bh_q0, pol_q);
      int issued = 0;
      bool ok = true;
      for (int jj = 0; jj < n && ok; ++jj) {
        for (int kv = 0; kv < 2; ++kv) {
          const int it = 2 * jj + kv;
          const int slot = it % C::kStages;
          if (!wait_or_abort(ptx::smem_u32(&bar_kv_empty[slot]), ((it / C::kStages) & 1) ^ 1u, abort_ptr,
                             p.timeout_ns, kRoleDecProducer)) {
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
                             (j0 + jj) * C::kBN, bh_kv, pol_kv);
        }
      }
      if (!ok || *abort_ptr) {
        drain_wait(q_full, 0, p.timeout_ns);
        for (int it = issued > C::kStages ? issued - C::kStages : 0; it < issued; ++it)
          if (it != p.drop_load)
            drain_wait(ptx::smem_u32(&bar_kv_full[it % C::kStages]), (it / C::kStages) & 1, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this converged (warp-uniform waits, one elected
    // lane issues each tcgen05 instruction).
    {
      auto kv_wait = [&](int it) {
        return wait_warp_or_abort(ptx::smem_u32(&bar_kv_full[it % C::kStages]), (it / C::kStages) & 1, abort_ptr,
                             p.timeout_ns, kRoleDecMma);
      };
      bool ok = wait_warp_or_abort(ptx::smem_u32(&bar_q_full), 0, abort_ptr, p.timeout_ns, kRoleDecMma);
      for (int jj = 0; jj < n && ok; ++jj) {
        if (jj > 0) {
          // O += P V for the previous block (P sits in the S columns).
          ok = wait_warp_or_abort(ptx::smem_u32(&bar_p_full), (jj - 1) & 1, abort_ptr, p.timeout_ns, kRoleDecMma);
          if (ok) ok = kv_wait(2 * (jj - 1) + 1);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t v_tile = sKV + ((2 * (jj - 1) + 1) % C::kStages) * C::kTileBytes;
          const uint64_t b_desc = ptx::desc_mnmajor_sw128(v_tile, C::kChunkBytes);
          ptx::mma_ts_k128_warp<32>(tmem_base + C::kColO, tmem_base + C::kColS, ptx::desc_lo(b_desc),
                                    ptx::desc_hi(b_desc), C::kIdescPV, jj > 1 ? 1u : 0u);
          ptx::mma_commit_warp(ptx::smem_u32(&bar_kv_empty[(2 * (jj - 1) + 1) % C::kStages]));
        }
        ok = kv_wait(2 * jj);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t k_tile = sKV + ((2 * jj) % C::kStages) * C::kTileBytes;
        const uint64_t a_desc = ptx::desc_kmajor_sw128(sQ), b_desc = ptx::desc_kmajor_sw128(k_tile);
        if constexpr (HD == 128)
          ptx::mma_ss_k128_warp(tmem_base + C::kColS, ptx::desc_lo(a_desc), ptx::desc_lo(b_desc),
                                ptx::desc_hi(a_desc), p.idesc_qk, 0u);
        else
          ptx::mma_ss_k64_warp(tmem_base + C::kColS, ptx::desc_lo(a_desc), ptx::desc_lo(b_desc),
                               ptx::desc_hi(a_desc), p.idesc_qk, 0u);
        ptx::mma_commit_warp(ptx::smem_u32(&bar_s_full));
        ptx::mma_commit_warp(ptx::smem_u32(&bar_kv_empty[(2 * jj) % C::kStages]));
      }
      if (ok) {
        // The last block's P V.
        ok = wait_warp_or_abort(ptx::smem_u32(&bar_p_full), (n - 1) & 1, abort_ptr, p.timeout_ns, kRoleDecMma);
        if (ok) ok = kv_wait(2 * (n - 1) + 1);
        if (ok) {
          ptx::tc_fence_after();
          const uint32_t v_tile = sKV + ((2 * (n - 1) + 1) % C::kStages) * C::kTileBytes;
          const uint64_t b_desc = ptx::desc_mnmajor_sw128(v_tile, C::kChunkBytes);
          ptx::mma_ts_k128_warp<32>(tmem_base + C::kColO, tmem_base + C::kColS, ptx::desc_lo(b_desc),
                                    ptx::desc_hi(b_desc), C::kIdescPV, n > 1 ? 1u : 0u);
          ptx::mma_commit_warp(ptx::smem_u32(&bar_o_full));
          ptx::mma_commit_warp(ptx::smem_u32(&bar_kv_empty[(2 * (n - 1) + 1) % C::kStages]));
        }
      }
      if (!ok) {
        ptx::mma_commit_warp(ptx::smem_u32(&bar_drain));
        drain_wait(ptx::smem_u32(&bar_drain), 0, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax + epilogue
    ptx::setmaxnreg_inc<C::kRegsSoftmax>();
    const int quarter = warp;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem_base + lane_addr + C::kColS;
    const uint32_t tO = tmem_base + lane_addr + C::kColO;
    const float sl2 = p.scale_log2;
    float m_use = 0.f;
    float l = 0.f;          // running sum of exp, relative to m_use (for LSE)
    float lo = 0.f;         // the same with each block's largest term as P V sees it (for O)
    bool ok = true;
    for (int jj = 0; jj < n; ++jj) {
      ok = wait_warp_or_abort(ptx::smem_u32(&bar_s_full), jj & 1, abort_ptr, p.timeout_ns, kRoleDecSoftmax);
      if (!ok) break;
      ptx::tc_fence_after();
      // The loads also reduce each 32-column piece to its maximum, which is
      // the row maximum of a full block; the ragged last block masks the
      // columns past N_kv (scores of zero-filled keys) and takes its own.
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

      const int valid = p.N_kv - (j0 + jj) * C::kBN;   // keys of this block that exist
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
        float mc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = k >> 1, bb = (k & 1) * 16;
          mc[k] = fmaxf(__uint_as_float(s[c][bb]), __uint_as_float(s[c][bb + 1]));
#pragma unroll
          for (int i = 2; i < 16; i += 2)
            mc[k] = ptx::max3(mc[k], __uint_as_float(s[c][bb + i]), __uint_as_float(s[c][bb + i + 1]));
        }
        mt = ptx::max3(ptx::max3(mc[0], mc[1], mc[2]), ptx::max3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
      }
      float alpha = 1.f;
      bool rescale_o = false;
      if (jj == 0) {
        m_use = mt;
      } else {
        const bool need = (mt - m_use) * sl2 > kRescaleLog2;
        rescale_o = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = ptx::ex2_approx((m_use - mt) * sl2);
          m_use = mt;
        }
      }
      const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
      const float neg_m = -m_use * sl2;
      const uint64_t negmx2 = ptx::f2_pack(neg_m, neg_m);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float x0, x1;
          ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])), sl2x2,
                                     negmx2),
                         x0, x1);
          float p0 = ptx::ex2_approx(x0);
          float p1 = ptx::ex2_approx(x1);
          if (ragged) {
            if (32 * c + i >= valid) p0 = 0.f;
            if (32 * c + i + 1 >= valid) p1 = 0.f;
          }
          acc[(i >> 1) & 3] = ptx::f2_add(acc[(i >> 1) & 3], ptx::f2_pack(p0, p1));
          pk[c >> 1][(c & 1) * 16 + (i >> 1)] = ptx::pack_bf16x2(p0, p1);
        }
        // The first 64 probabilities are packed: store them now (over scores
        // already in registers) and free their registers.
        if (c == 1) ptx::tmem_st32(tS, pk[0]);
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
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bar_p_full));
    }
    if (ok) ok = wait_warp_or_abort(ptx::smem_u32(&bar_o_full), 0, abort_ptr, p.timeout_ns, kRoleDecSoftmax);
    if (ok) {
      ptx::tc_fence_after();
      // Row r of the tile is query row q0 + r % box_q of query head g0 + r / box_q.
      const bool in_range = row < rows;
      const int hq = row / p.box_q;
      const size_t grow = (static_cast<size_t>(bh_q0) + hq) * p.N_q + q0 + (row - hq * p.box_q);
      const float inv_l = 1.f / lo;
      const float lse = (m_use * sl2 + __log2f(l)) * 0.69314718055994530942f;
      const size_t n_rows = static_cast<size_t>(gridDim.z) * p.H * p.N_q;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + 32 * c, o);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(o);
        if (!in_range) continue;
        if (p.num_splits == 1 && !p.f32_out) {
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = ptx::pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(p.O + grow * HD + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        } else {
          float4* dst = reinterpret_cast<float4*>(p.O_part + (split * n_rows + grow) * HD + 32 * c);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                 __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
        }
      }
      if (in_range) {
        if (p.num_splits == 1 && !p.f32_out) p.LSE[grow] = lse;
        else p.LSE_part[split * n_rows + grow] = lse;
      }
    }
  }

  // The merge kernel may be scheduled now; it waits for this grid's end.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// One warp per query row: combine the num_splits partial results of the row.
// LSE = m + ln sum_s e^{LSE_s - m} with m = max_s LSE_s, and
// O = sum_s e^{LSE_s - LSE} O_s, rounded once to bf16 (OutT = __nv_bfloat16)
// or kept in float32 (OutT = float). The splits' LSE are
// read by the lanes in parallel (32 at a time) and their weights passed by
// shuffles, so the row costs two dependent rounds of loads, not 2 x splits.
template <int HD, typename OutT = __nv_bfloat16>
__global__ void __launch_bounds__(256) decode_merge_kernel(const float* __restrict__ O_part,
                                                           const float* __restrict__ LSE_part,
                                                           OutT* __restrict__ O, float* __restrict__ LSE,
                                                           long long n_rows, int num_splits) {
  // Launched as a programmatic dependent of the decode kernel: wait here until
  // that grid has finished and its partials are visible (returns at once when
  // there is no such grid).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  float m = -INFINITY;
  for (int s0 = 0; s0 < num_splits; s0 += 32) {
    const int s = s0 + lane;
    if (s < num_splits) m = fmaxf(m, LSE_part[s * n_rows + row]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  constexpr int kPer = HD / 32;     // output elements per lane: 4 or 2
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float total = 0.f;
  for (int s0 = 0; s0 < num_splits; s0 += 32) {
    const int s_me = s0 + lane;
    const float w_me = s_me < num_splits ? __expf(LSE_part[s_me * n_rows + row] - m) : 0.f;
    total += w_me;
    const int cnt = min(32, num_splits - s0);
#pragma unroll 4
    for (int i = 0; i < cnt; ++i) {
      const float w = __shfl_sync(0xffffffffu, w_me, i);
      const float* src = O_part + ((s0 + i) * n_rows + row) * HD + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, src[e], acc[e]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  const float inv = 1.f / total;
  OutT* dst = O + row * HD + lane * kPer;
  if constexpr (sizeof(OutT) == 4) {
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
      *reinterpret_cast<float2*>(dst + e) = make_float2(acc[e] * inv, acc[e + 1] * inv);
  } else {
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
      *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
  if (lane == 0) LSE[row] = m + __logf(total);
}

}  // namespace fa
