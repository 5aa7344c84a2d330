// Inline-PTX wrappers for the Blackwell (sm_100a / sm_103a) features the
// attention kernel uses: mbarriers, TMA tensor copies, tensor memory (TMEM)
// allocation, tcgen05 MMAs, commits and TMEM loads/stores.
//
// Conventions written down here once:
//  * Shared-memory addresses are 32-bit `.shared::cta` addresses.
//  * A TMEM address is (lane << 16) | column. A warp may only touch the 32
//    lanes of its quarter: lanes [32*(warp_id % 4), 32*(warp_id % 4) + 32).
//  * tcgen05.ld results are undefined until tcgen05.wait::ld; the wrappers
//    below return registers that the caller must pass through tmem_ld_wait()
//    (which also tells the compiler the registers change there).
#pragma once

#include <cstdint>

namespace fa {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// True once the phase with parity `parity` has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// True if the phase with parity `parity` has completed; never blocks.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------- clusters
// Rank of this CTA within its cluster (0 when launched without clusters).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of shared-memory location `addr` (a shared::cta
// address of this CTA) in the CTA of rank `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_shared_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster; orders this thread's
// earlier memory operations (e.g. st.shared::cluster) before the arrival at
// cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// try_wait with cluster-scope acquire: writes that another CTA of the cluster
// released before arriving are visible once this returns true.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Every thread of every CTA of the cluster arrives, then waits for all.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 3-D tiled load global -> shared, completion counted in bytes on `bar`.
// c0 is the innermost coordinate (elements) and must be a multiple of 8 for
// bf16 so that the copy starts on a 16-byte boundary.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int c0, int c1,
                                            int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// Tiled TMA store of a box from this CTA's shared memory (in the map's
// swizzled layout) to global memory; parts of the box outside the tensor are
// not written. Completion is tracked with bulk groups (commit / wait).
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk group has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the async proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Plain (untiled) bulk copy of `bytes` from global to this CTA's shared
// memory, completing on `bar` like the tensor copies. Both addresses must be
// 16-byte aligned and `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------- TMEM
// Warp-wide: allocates `ncols` columns (power of two >= 32) and writes the
// base TMEM address to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- UMMA descriptors
// Shared-memory matrix descriptor, K-major operand, 128-byte swizzle:
// rows of 128 bytes (64 bf16 along K), 8-row atoms of 1024 bytes, atoms
// stacked along M/N every 1024 bytes. The leading-byte offset is unused for
// swizzled K-major layouts. Bits: [0,14) start>>4, [16,30) LBO>>4,
// [32,46) SBO>>4, [46,48) = 1 (tcgen05 descriptor), [61,64) = 2 (128B swizzle).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// MN-major operand, 128-byte swizzle: atoms of 64 bf16 along M/N (128 bytes)
// x 8 rows along K (1024 bytes). SBO = distance between 8-row groups along K
// (1024 bytes here); LBO = distance between 64-element atoms along M/N.
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t mn_atom_stride) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((mn_atom_stride >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and f32 accumulation.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B
// format (1 = bf16), 15 A major (1 = MN), 16 B major (1 = MN), [17,23) N>>3,
// [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Bit 13 of the kind::f16 instruction descriptor negates A: the product is
// then (-A) B^T, exact for floating-point operands.
constexpr uint32_t kIdescNegateA = 1u << 13;

// ---------------------------------------------------------------- tcgen05.mma
// D[tmem] (+)= A[smem] * B[smem]^T ; accumulate when `accum` != 0.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accum)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem] ; A is read from tensor memory.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accum)
      : "memory");
}

// Bursts of products issued from a converged warp: every lane calls these and
// elect.sync picks one lane (lane 0 of a full warp) to issue. A single
// diverged lane issues tcgen05.mma far more slowly than a converged warp when
// other warps of its SM sub-partition compete for issue slots (measured on
// GB300: 252 against 151 cycles per 128x128x16 product beside 8 busy warps).
// One asm block holds the group: one elect.sync and one accumulate predicate,
// then per product only a 32-bit add on the descriptor's low word (its start
// address in 16-byte units; the shared memory window is below 256 KB, so it
// never carries into the next field) and the predicated tcgen05.mma. The
// fewer instructions per product, the less of the issuing warp's share of
// issue slots the group takes (1566 -> 1633 TFLOP/s on the 8k forward against
// one asm statement per product). The first product accumulates when
// acc0 != 0, the others always.
#define FA_BURST_SS(OA) "add.u32 al, %1, " #OA ";\n\tadd.u32 bl, %2, " #OA ";\n\t" \
  "mov.b64 ad, {al, %3};\n\tmov.b64 bd, {bl, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, t;\n\t"
#define FA_BURST_SS_HEAD \
  "{\n\t.reg .pred p, e, t;\n\t.reg .b32 al, bl;\n\t.reg .b64 ad, bd;\n\t" \
  "setp.ne.b32 p, %5, 0;\n\tsetp.eq.u32 t, %4, %4;\n\telect.sync _|e, 0xffffffff;\n\t" \
  "mov.b64 ad, {%1, %3};\n\tmov.b64 bd, {%2, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, p;\n\t"

// K = 128 over two K-major 128-byte-swizzled chunks of 16 KB, A and B alike:
// product kk starts at (kk / 4) * 16 KB + (kk % 4) * 32 B. a_lo / b_lo are the
// low words of desc_kmajor_sw128 of the tiles, `hi` their (common) high word.
__device__ __forceinline__ void mma_ss_k128_warp(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                                 uint32_t idesc, uint32_t acc0) {
  asm volatile(FA_BURST_SS_HEAD FA_BURST_SS(2) FA_BURST_SS(4) FA_BURST_SS(6) FA_BURST_SS(1024) FA_BURST_SS(1026)
               FA_BURST_SS(1028) FA_BURST_SS(1030) "}" ::"r"(d_tmem),
               "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(acc0)
               : "memory");
}

// K = 64 within one chunk: product kk starts at kk * 32 B.
__device__ __forceinline__ void mma_ss_k64_warp(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                                uint32_t idesc, uint32_t acc0) {
  asm volatile(FA_BURST_SS_HEAD FA_BURST_SS(2) FA_BURST_SS(4) FA_BURST_SS(6) "}" ::"r"(d_tmem), "r"(a_lo),
               "r"(b_lo), "r"(hi), "r"(idesc), "r"(acc0)
               : "memory");
}

// Eight products with A from TMEM and B MN-major over 128 rows of K (16 rows,
// 2 KB, per product): B of product kk starts at kk * 2 KB; A at column
// a_tmem + 8 * kk (kA4 = 32) or a_tmem + kA4 * (kk / 4) + 8 * (kk % 4).
#define FA_BURST_TS(OA, OB) "add.u32 ta, %1, " #OA ";\n\tadd.u32 bl, %2, " #OB ";\n\t" \
  "mov.b64 bd, {bl, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %4, t;\n\t"
#define FA_BURST_TS_HEAD \
  "{\n\t.reg .pred p, e, t;\n\t.reg .b32 ta, bl;\n\t.reg .b64 bd;\n\t" \
  "setp.ne.b32 p, %5, 0;\n\tsetp.eq.u32 t, %4, %4;\n\telect.sync _|e, 0xffffffff;\n\t" \
  "mov.b64 bd, {%2, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t"

// Opens a burst whose products all accumulate (no leading product that may
// overwrite D): the continuation of a burst split in two.
#define FA_BURST_TS_HEAD_ACC \
  "{\n\t.reg .pred e, t;\n\t.reg .b32 ta, bl;\n\t.reg .b64 bd;\n\t" \
  "setp.eq.u32 t, %4, %4;\n\telect.sync _|e, 0xffffffff;\n\t"

// Half of the 128-key P V burst (A columns step 8 per product): keys
// [64 kHalf, 64 kHalf + 64), four products; the second half always accumulates.
template <int kHalf>
__device__ __forceinline__ void mma_ts_k64half_warp(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                                    uint32_t idesc, uint32_t acc0) {
  if constexpr (kHalf == 0) {
    asm volatile(FA_BURST_TS_HEAD FA_BURST_TS(8, 128) FA_BURST_TS(16, 256) FA_BURST_TS(24, 384) "}" ::"r"(d_tmem),
                 "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc0)
                 : "memory");
  } else {
    asm volatile(FA_BURST_TS_HEAD_ACC FA_BURST_TS(32, 512) FA_BURST_TS(40, 640) FA_BURST_TS(48, 768)
                 FA_BURST_TS(56, 896) "}" ::"r"(d_tmem),
                 "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc0)
                 : "memory");
  }
}

template <int kA4>
__device__ __forceinline__ void mma_ts_k128_warp(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                                 uint32_t idesc, uint32_t acc0) {
  static_assert(kA4 == 32 || kA4 == 64, "A column step per four products");
  if constexpr (kA4 == 32) {
    asm volatile(FA_BURST_TS_HEAD FA_BURST_TS(8, 128) FA_BURST_TS(16, 256) FA_BURST_TS(24, 384)
                 FA_BURST_TS(32, 512) FA_BURST_TS(40, 640) FA_BURST_TS(48, 768) FA_BURST_TS(56, 896) "}" ::"r"(d_tmem),
                 "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc0)
                 : "memory");
  } else {
    asm volatile(FA_BURST_TS_HEAD FA_BURST_TS(8, 128) FA_BURST_TS(16, 256) FA_BURST_TS(24, 384)
                 FA_BURST_TS(64, 512) FA_BURST_TS(72, 640) FA_BURST_TS(80, 768) FA_BURST_TS(88, 896) "}" ::"r"(d_tmem),
                 "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc0)
                 : "memory");
  }
}

__device__ __forceinline__ uint32_t desc_lo(uint64_t d) { return static_cast<uint32_t>(d); }
__device__ __forceinline__ uint32_t desc_hi(uint64_t d) { return static_cast<uint32_t>(d >> 32); }

// mma_commit from a converged warp: the elected lane (the one that issued the
// products above) arrives.
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// ---------------------------------------------------------------- TMEM load/store
#define FA_R8(a, i) "=r"(a[i]), "=r"(a[i + 1]), "=r"(a[i + 2]), "=r"(a[i + 3]), "=r"(a[i + 4]), "=r"(a[i + 5]), \
                    "=r"(a[i + 6]), "=r"(a[i + 7])
#define FA_W8(a, i) "r"(a[i]), "r"(a[i + 1]), "r"(a[i + 2]), "r"(a[i + 3]), "r"(a[i + 4]), "r"(a[i + 5]), \
                    "r"(a[i + 6]), "r"(a[i + 7])
#define FA_M8(a, i) "+r"(a[i]), "+r"(a[i + 1]), "+r"(a[i + 2]), "+r"(a[i + 3]), "+r"(a[i + 4]), "+r"(a[i + 5]), \
                    "+r"(a[i + 6]), "+r"(a[i + 7])

// 32 lanes x 32 columns of 32-bit: thread t of the warp gets lane
// (quarter*32 + t), columns [col, col+32) in r[0..31].
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : FA_R8(r, 0), FA_R8(r, 8), FA_R8(r, 16), FA_R8(r, 24)
      : "r"(taddr));
}

// 32 lanes x 8 columns of 32-bit: r[0..7] = columns [col, col+8) of this thread's lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : FA_R8(r, 0)
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      FA_W8(r, 0), FA_W8(r, 8), FA_W8(r, 16), FA_W8(r, 24)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// After tmem_ld_wait(): marks the 32 registers as produced here, so that no
// use of them is scheduled before the wait.
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
  asm volatile("" : FA_M8(r, 0), FA_M8(r, 8), FA_M8(r, 16), FA_M8(r, 24));
}

__device__ __forceinline__ void reg_fence8(uint32_t (&r)[8]) { asm volatile("" : FA_M8(r, 0)); }

// tmem_ld32 that also returns, in `mx`, the maximum of the 32 fp32 values
// this thread loads (the load-with-reduction form of sm_103a; NaN operands
// are ignored, as by max.f32). Valid after tmem_ld_wait, like the values.
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : FA_R8(r, 0), FA_R8(r, 8), FA_R8(r, 16), FA_R8(r, 24), "=f"(mx)
      : "r"(taddr));
}

__device__ __forceinline__ void reg_fence1(float& x) { asm volatile("" : "+f"(x)); }

#undef FA_R8
#undef FA_W8
#undef FA_M8

// ---------------------------------------------------------------- math
// Hardware base-2 exponential (MUFU.EX2), flush-to-zero; ex2(-inf) = +0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (sm_100+).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed pair of floats in one 64-bit register, for the f32x2 FMA/ADD (sm_100+).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Two floats to packed bf16x2 (round to nearest even): `lo` in bits [0,16).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Per-thread register budget of the executing warpgroup (all four warps must
// execute the same instruction): raise it to N, drawing on registers other
// warpgroups released, or lower it to N.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  static_assert(N >= 24 && N <= 256 && N % 8 == 0, "setmaxnreg range");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  static_assert(N >= 24 && N <= 256 && N % 8 == 0, "setmaxnreg range");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// x rounded to bf16 by the same conversion pack_bf16x2 makes, as a float.
__device__ __forceinline__ float round_bf16(float x) { return __uint_as_float(pack_bf16x2(x, 0.f) << 16); }

}  // namespace ptx
}  // namespace fa
