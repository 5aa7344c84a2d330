// C ABI of the exact attention forward pass (declared in include/fa.h):
// argument checks, TMA descriptor encoding, the launch on the caller's
// stream, and the device status word.
//
// One launch per call ("01 · 注意力为什么是 IO 瓶颈" §6: the fused forward is a
// single kernel launch on the caller's stream). Unlike the upstream library
// described there, which allocates softmax_lse itself, the caller owns O and
// LSE here and this file allocates no device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_bwd_kernel.cuh"
#include "fa_decode_kernel.cuh"
#include "fa_fwd_kernel.cuh"
#include "naive_kernels.cuh"

// Device scratch for fa_naive_fwd_noalloc: the score/probability matrices of
// the standard-attention path live here instead of in caller memory. It is
// part of this library's device image, so every GPU that loads the library
// holds these 64 MiB until the process exits. In host code the name below is
// only a host-side stand-in; its device address comes from
// cudaGetSymbolAddress (see naive_static_scratch()).
static constexpr size_t kNaiveStaticScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_naive_static_scratch[kNaiveStaticScratchBytes];

namespace {

thread_local int t_last_cuda_error = 0;

// Bound on every device-side wait of the standard-attention kernels.
constexpr unsigned long long kNaiveTimeoutNs = 2000000000ull;

fa_status_t cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return FA_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [B*H, N, d] bf16 view of a contiguous [B, H, N, d] tensor; box = 64 x 128
// rows x 1 head, 128-byte swizzle. Rows beyond N of a head are outside the
// tensor and read as zeros, so a ragged last block never sees the next head.
bool make_map_ld(CUtensorMap* m, const void* base, int Z, int rows, int cols, long long ld, int box_cols,
                 int box_rows);
bool make_map(CUtensorMap* m, const void* base, int BH, int N, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// SM count of a device, read once per device.
int sm_count(int dev) {
  static std::once_flag once[64];
  static int count[64];
  std::call_once(once[dev], [dev] {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    count[dev] = n;
  });
  return count[dev];
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  auto x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Launch shape of the forward over `units` units of 256 query rows with
// n_kv key blocks each, on `sms` SMs of which at most `max2` clusters of two
// can be resident at once (a cluster must fit in one GPC). All units cost
// the same, so a grid of G CTAs takes ceil(units / G) rounds. When the units
// left after the whole rounds fill at most half of an even grid, clusters of
// two share them, one unit per pair, half of its key blocks each: the last
// round then takes about half as long (512 units on 152 SMs: 3.5 rounds
// instead of 4). A persistent grid must be resident as a whole, so a
// clustered grid has at most 2 * max2 CTAs, and it is used only when it
// takes fewer rounds; each half must hold at least two key blocks.
struct FwdShape {
  int grid, cluster, whole_units;
};
FwdShape fwd_shape(int units, int n_kv, int sms, int max2) {
  const int g1 = std::max(1, std::min(units, sms));
  const FwdShape plain{g1, 1, units};
  const int g2 = std::min(sms & ~1, 2 * max2);
  if (n_kv < 4 || g2 < 2) return plain;
  const int whole = units / g2 * g2, tail = units - whole;
  if (tail == 0 || 2 * tail > g2) return plain;
  // whole / g2 + 1/2 rounds against ceil(units / g1)
  return 2 * (whole / g2) + 1 < 2 * ((units + g1 - 1) / g1) ? FwdShape{g2, 2, whole} : plain;
}

// Per device and head dimension: the kernel's shared-memory opt-in, whether
// its register split fits the launch, and how many clusters of two can be
// resident at once.
struct FwdDevInfo {
  cudaError_t err;
  bool regs_ok;
  int max2;
};

template <int HD>
const FwdDevInfo* fwd_dev_info(int dev) {
  using C = fa::FwdCfg<HD>;
  static std::once_flag once[64];
  static FwdDevInfo info[64];
  if (dev < 0 || dev >= 64) return nullptr;
  std::call_once(once[dev], [&] {
    FwdDevInfo& fi = info[dev];
    fi = FwdDevInfo{cudaSuccess, false, 0};
    fi.err = cudaFuncSetAttribute(fa::fa_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    // The warpgroups' register split draws on the registers the block is
    // launched with; a split larger than that would never complete, so the
    // kernel is not launched unless the built register count covers it.
    cudaFuncAttributes fattr;
    if (fi.err == cudaSuccess) fi.err = cudaFuncGetAttributes(&fattr, fa::fa_fwd_kernel<HD>);
    fi.regs_ok = fi.err == cudaSuccess && 8 * C::kRegsSoftmax + 4 * C::kRegsControl <= 12 * fattr.numRegs;
    if (fi.err == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2u);
      cfg.blockDim = dim3(C::kThreads);
      cfg.dynamicSmemBytes = C::kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      // A failed query only disables the shared units.
      if (cudaOccupancyMaxActiveClusters(&n, fa::fa_fwd_kernel<HD>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      fi.max2 = std::max(0, n);
    }
  });
  return &info[dev];
}

// Units [0, whole_units) of a problem of total_units units run whole; the rest
// (the last, partial round) are shared by CTA pairs. A launch covering only
// part of the problem (unit_offset onwards, e.g. one head group of
// fa_fwd_host) follows the whole problem's plan, so that every unit is
// computed the same way as by one launch over everything.
struct SplitPlan {
  int total_units;
  int unit_offset;
};

template <int HD>
fa_status_t launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int H_kv, int N,
                   int N_kv, float scale, int drop_load, unsigned long long timeout_ns, cudaStream_t stream,
                   const SplitPlan* plan = nullptr) {
  using C = fa::FwdCfg<HD>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  // The dynamic shared-memory opt-in is per function and device context.
  const FwdDevInfo* fi = fwd_dev_info<HD>(dev);
  if (!fi) return FA_ERR_UNSUPPORTED;
  if (fi->err != cudaSuccess) return cuda_fail(fi->err);
  if (!fi->regs_ok) return FA_ERR_UNSUPPORTED;

  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, Q, B * H, N, HD) || !make_map(&mk, K, B * H_kv, N_kv, HD) ||
      !make_map(&mv, V, B * H_kv, N_kv, HD) || !make_map_ld(&mo, O, B * H, N, HD, HD, 64, 32))
    return cuda_fail(cudaErrorInvalidValue);

  fa::FwdParams p;
  p.O = static_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.N = N;
  p.N_kv = N_kv;
  p.H = H;
  p.H_kv = H_kv;
  p.n_kv_blocks = (N_kv + C::kBN - 1) / C::kBN;
  p.q_blocks = (N + C::kQTiles * C::kBM - 1) / (C::kQTiles * C::kBM);
  p.num_units = B * H * p.q_blocks;   // < 2^31 / 256: B*H*N < 2^31
  // scale < 0: the tensor core forms -S and the kernel runs with |scale|.
  p.scale_log2 = static_cast<float>(std::fabs(static_cast<double>(scale)) * 1.4426950408889634074);
  p.idesc_qk = C::kIdescQK | (scale < 0.f ? fa::ptx::kIdescNegateA : 0u);
  p.timeout_ns = timeout_ns;
  p.drop_load = drop_load;

  // Persistent grid: one CTA per SM (the kernel's shared memory and tensor
  // memory allow no second), each walking units blockIdx.x + k * gridDim.x.
  const FwdShape sh = fwd_shape(plan ? plan->total_units : p.num_units, p.n_kv_blocks, sm_count(dev), fi->max2);
  int grid = std::min(p.num_units, sh.grid);
  p.num_whole = p.num_units;
  p.split_tail = 0;
  if (sh.cluster == 2) {
    // This launch's units past the problem's whole rounds are shared; they
    // are a suffix of its units and at most half the grid.
    const int offset = plan ? plan->unit_offset : 0;
    const int local_whole = std::max(0, std::min(p.num_units, sh.whole_units - offset));
    if (local_whole < p.num_units) {
      p.split_tail = 1;
      p.num_whole = local_whole;
      grid = sh.grid;
    }
  }
  if (p.split_tail) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fa::fa_fwd_kernel<HD>, mq, mk, mv, mo, p);
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
  }
  fa::fa_fwd_kernel<HD><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mo, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

fa_status_t fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                     float scale, int drop_load, unsigned long long timeout_ns, cudaStream_t stream) {
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * N >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  for (const void* ptr : {Q, K, V, static_cast<const void*>(O)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(LSE) % 4 != 0) return FA_ERR_INVALID_ARG;
  const size_t n_qkv = static_cast<size_t>(B) * H * N * d * 2;
  const size_t n_lse = static_cast<size_t>(B) * H * N * 4;
  for (const void* in : {Q, K, V}) {
    if (overlaps(O, n_qkv, in, n_qkv) || overlaps(LSE, n_lse, in, n_qkv)) return FA_ERR_INVALID_ARG;
  }
  if (overlaps(O, n_qkv, LSE, n_lse)) return FA_ERR_INVALID_ARG;
  if (d == 64) return launch<64>(Q, K, V, O, LSE, B, H, H, N, N, scale, drop_load, timeout_ns, stream);
  return launch<128>(Q, K, V, O, LSE, B, H, H, N, N, scale, drop_load, timeout_ns, stream);
}

// ---------------------------------------------------------------- standard attention
// Row stride (elements) of the N x N score / probability matrices in the
// workspace: a multiple of 64 so that every row starts 128-byte aligned.
inline long long naive_ld(int N) { return (static_cast<long long>(N) + 63) / 64 * 64; }

// 3-D bf16 map [Z][rows][cols] with a row stride of ld elements.
bool make_map_ld(CUtensorMap* m, const void* base, int Z, int rows, int cols, long long ld, int box_cols,
                 int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(Z)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(ld) * rows * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool B_KMAJOR>
cudaError_t gemm_attr() {
  using G = fa::naive::GemmCfg<BN, B_KMAJOR>;
  return cudaFuncSetAttribute(fa::naive::gemm_bf16_kernel<BN, B_KMAJOR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              G::kSmemBytes);
}

// The three launches of standard attention with S / P in `ws` ([B*H][N][ld] bf16).
template <int HD>
fa_status_t naive_launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                         float scale, void* ws, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  std::call_once(once[dev], [&] {
    attr_err[dev] = cudaFuncSetAttribute(fa::naive::s_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fa::naive::SGemmCfg::kSmemBytes);
    if (attr_err[dev] == cudaSuccess) attr_err[dev] = gemm_attr<HD, false>();
  });
  if (attr_err[dev] != cudaSuccess) return cuda_fail(attr_err[dev]);

  const int BH = B * H;
  const long long ld = naive_ld(N);
  CUtensorMap mq, mk, mp, mv, ms_out, mo_out;
  if (!make_map_ld(&mq, Q, BH, N, HD, HD, 64, 128) || !make_map_ld(&mk, K, BH, N, HD, HD, 64, 128) ||
      !make_map_ld(&mp, ws, BH, N, N, ld, 64, 128) || !make_map_ld(&mv, V, BH, N, HD, HD, 64, 64) ||
      !make_map_ld(&ms_out, ws, BH, N, N, ld, 64, 32) || !make_map_ld(&mo_out, O, BH, N, HD, HD, 64, 32))
    return cuda_fail(cudaErrorInvalidValue);
  auto* S = static_cast<__nv_bfloat16*>(ws);

  // 1. S = bf16(scale * bf16(Q K^T)): a persistent grid of two CTAs per SM
  using G1 = fa::naive::SGemmCfg;
  fa::naive::SGemmParams g1;
  g1.M = N;
  g1.Nc = N;
  g1.K = HD;
  g1.mt = (N + G1::kBM - 1) / G1::kBM;
  g1.nt = (N + G1::kBN - 1) / G1::kBN;
  const long long s_tiles = static_cast<long long>(g1.mt) * g1.nt * BH;
  if (s_tiles >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  g1.tiles = static_cast<int>(s_tiles);
  g1.alpha = scale;
  g1.timeout_ns = kNaiveTimeoutNs;
  const int s_grid = static_cast<int>(std::min<long long>(s_tiles, 2LL * sm_count(dev)));
  fa::naive::s_gemm_kernel<<<s_grid, G1::kThreads, G1::kSmemBytes, stream>>>(mq, mk, ms_out, g1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  // 2. P = softmax(S) row by row, in place; LSE = m + ln l
  const long long n_rows = static_cast<long long>(BH) * N;
  fa::naive::softmax_rows_kernel<<<static_cast<unsigned>((n_rows + 7) / 8), 256, 0, stream>>>(
      S, LSE, n_rows, N, static_cast<int>(ld));
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  // 3. O = bf16(P V)
  fa::naive::GemmParams g2{static_cast<__nv_bfloat16*>(O), N, HD, N, HD, 1.0f, kNaiveTimeoutNs};
  using G2 = fa::naive::GemmCfg<HD, false>;
  fa::naive::gemm_bf16_kernel<HD, false><<<dim3(1, (N + 127) / 128, BH), G2::kThreads, G2::kSmemBytes, stream>>>(
      mp, mv, mo_out, g2);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

// Argument checks shared by every entry point of the library (host side only).
fa_status_t check_args(const void* Q, const void* K, const void* V, const void* O, const float* LSE, int B, int H,
                       int N, int d, float scale) {
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * N >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  for (const void* ptr : {Q, K, V, O})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(LSE) % 4 != 0) return FA_ERR_INVALID_ARG;
  const size_t n_qkv = static_cast<size_t>(B) * H * N * d * 2;
  const size_t n_lse = static_cast<size_t>(B) * H * N * 4;
  for (const void* in : {Q, K, V}) {
    if (overlaps(O, n_qkv, in, n_qkv) || overlaps(LSE, n_lse, in, n_qkv)) return FA_ERR_INVALID_ARG;
  }
  if (overlaps(O, n_qkv, LSE, n_lse)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Device address of g_naive_static_scratch on the current device. The first
// successful lookup on a device is kept; a failed one is not (its error is
// returned and cleared from the runtime's last-error state), so the next call
// on that device looks the address up again.
cudaError_t naive_static_scratch(int dev, void** out) {
  static std::mutex mu;
  static void* addr[64];
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_naive_static_scratch);
    if (e != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

// The standard-attention launches put B*H in gridDim.z and the 128-row block
// count of N in gridDim.y, both limited to 65535.
bool naive_grid_ok(int B, int H, int N) {
  return static_cast<long long>(B) * H <= 65535 && (static_cast<long long>(N) + 127) / 128 <= 65535;
}

// A correct pipeline never waits anywhere near this long; it only bounds
// how long a broken one can hold the GPU.
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;

// ---------------------------------------------------------------- backward
// Query rows per head in the backward workspace: N rounded up to whole
// 128-row blocks, so that every block's slice starts 512-byte aligned.
inline long long bwd_npad(int N) { return (static_cast<long long>(N) + 127) / 128 * 128; }

template <int HD>
fa_status_t bwd_launch(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                       void* dQ, void* dK, void* dV, int B, int H, int N, float scale, void* ws, int drop_load,
                       unsigned long long timeout_ns, cudaStream_t stream) {
  using C = fa::BwdCfg<HD>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  // Dynamic shared memory of the main kernel: the larger of its two roles.
  constexpr int kSmem = fa::DqCfg<HD>::kSmemBytes > C::kSmemBytes ? fa::DqCfg<HD>::kSmemBytes : C::kSmemBytes;
  std::call_once(once[dev], [&] {
    attr_err[dev] = cudaFuncSetAttribute(fa::fa_bwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err[dev] != cudaSuccess) return cuda_fail(attr_err[dev]);

  const int BH = B * H;
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  if (!make_map(&mq, Q, BH, N, HD) || !make_map(&mk, K, BH, N, HD) || !make_map(&mv, V, BH, N, HD) ||
      !make_map(&mdo, dO, BH, N, HD) || !make_map_ld(&mdq, dQ, BH, N, HD, HD, 64, 32) ||
      !make_map_ld(&mdk, dK, BH, N, HD, HD, 64, 32) || !make_map_ld(&mdv, dV, BH, N, HD, HD, 64, 32))
    return cuda_fail(cudaErrorInvalidValue);

  const long long npad = bwd_npad(N);
  const long long rows = static_cast<long long>(BH) * npad;
  fa::BwdParams p;
  p.dQ = static_cast<__nv_bfloat16*>(dQ);
  p.dK = static_cast<__nv_bfloat16*>(dK);
  p.dV = static_cast<__nv_bfloat16*>(dV);
  p.nlse2 = static_cast<const float*>(ws);
  p.ndelta = static_cast<const float*>(ws) + rows;
  p.N = N;
  p.Npad = static_cast<int>(npad);
  p.H = H;
  p.n_blocks = static_cast<int>(npad / C::kBlk);
  p.BH = BH;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  p.scale = scale;
  p.timeout_ns = timeout_ns;
  p.drop_load = drop_load;

  // 1. -LSE*log2(e) and -D per query row (eight rows per warp, 64 per block)
  fa::bwd_prep_kernel<HD><<<static_cast<unsigned>((rows + 63) / 64), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), LSE, static_cast<float*>(ws),
      static_cast<float*>(ws) + rows, N, p.Npad, rows);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  // 2. dK and dV (one CTA per 128 key rows), then dQ (one CTA per 128 query
  // rows), in one launch
  const unsigned ctas = static_cast<unsigned>(2LL * p.n_blocks * BH);
  fa::fa_bwd_kernel<HD><<<ctas, C::kThreads, kSmem, stream>>>(mq, mk, mv, mdo, mdq, mdk, mdv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

// ---------------------------------------------------------------- host buffers
// fa_fwd_host: the device copies of Q, K, V, O and LSE live in the caller's
// workspace, each part 256-byte aligned.
constexpr int kHostMaxChunks = 16;

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

size_t host_workspace_bytes(int B, int H, int N, int d) {
  const size_t n_qkv = static_cast<size_t>(B) * H * N * d * 2;
  const size_t n_lse = static_cast<size_t>(B) * H * N * 4;
  return 4 * align256(n_qkv) + align256(n_lse);
}

// Streams and events of the host path, one set per device, created on first
// use and kept for the life of the process: an upload stream, a download
// stream, and a second compute stream so that consecutive chunk kernels may
// overlap. Calls are serialised by `mu` while they enqueue, which lets them
// reuse the events: a stream wait takes the event's state when it is enqueued.
struct HostPath {
  std::mutex mu;
  cudaStream_t up = nullptr, down = nullptr, aux = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in[kHostMaxChunks] = {}, done[kHostMaxChunks] = {};
  cudaError_t err = cudaSuccess;
};

HostPath* host_path(int dev) {
  static HostPath hp[64];
  static std::once_flag once[64];
  std::call_once(once[dev], [dev] {
    HostPath& h = hp[dev];
    cudaError_t e = cudaStreamCreateWithFlags(&h.up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.down, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.aux, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.end, cudaEventDisableTiming);
    for (int c = 0; c < kHostMaxChunks && e == cudaSuccess; ++c) {
      e = cudaEventCreateWithFlags(&h.in[c], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.done[c], cudaEventDisableTiming);
    }
    h.err = e;
  });
  return &hp[dev];
}

// Heads per chunk: about 8 chunks, so that the first upload and the last
// download, which nothing overlaps, are short.
int host_chunks(int BH, int num_chunks) {
  const int nc = num_chunks > 0 ? num_chunks : 8;
  return std::max(1, std::min({nc, BH, kHostMaxChunks}));
}

fa_status_t host_impl(const void* Qh, const void* Kh, const void* Vh, void* Oh, float* LSEh, int B, int H, int N,
                      int d, float scale, int num_chunks, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  if (!Qh || !Kh || !Vh || !Oh || !LSEh) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || d < 1 || num_chunks < 0) return FA_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * N >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const size_t need = host_workspace_bytes(B, H, N, d);
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 || workspace_bytes < need)
    return FA_ERR_INVALID_ARG;
  const size_t n_qkv = static_cast<size_t>(B) * H * N * d * 2;
  const size_t n_lse = static_cast<size_t>(B) * H * N * 4;
  for (const void* a : {Qh, Kh, Vh}) {
    if (overlaps(Oh, n_qkv, a, n_qkv) || overlaps(LSEh, n_lse, a, n_qkv)) return FA_ERR_INVALID_ARG;
  }
  if (overlaps(Oh, n_qkv, LSEh, n_lse)) return FA_ERR_INVALID_ARG;
  for (const void* a : {Qh, Kh, Vh, static_cast<const void*>(Oh), static_cast<const void*>(LSEh)})
    if (overlaps(a, a == LSEh ? n_lse : n_qkv, workspace, need)) return FA_ERR_INVALID_ARG;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  HostPath* hp = host_path(dev);
  if (hp->err != cudaSuccess) return cuda_fail(hp->err);

  char* Qd = static_cast<char*>(workspace);
  char* Kd = Qd + align256(n_qkv);
  char* Vd = Kd + align256(n_qkv);
  char* Od = Vd + align256(n_qkv);
  char* Ld = Od + align256(n_qkv);
  const char* qh = static_cast<const char*>(Qh);
  const char* kh = static_cast<const char*>(Kh);
  const char* vh = static_cast<const char*>(Vh);
  char* oh = static_cast<char*>(Oh);
  char* lh = reinterpret_cast<char*>(LSEh);

  const int BH = B * H;
  const int nc = host_chunks(BH, num_chunks);
  const int per = (BH + nc - 1) / nc;
  const size_t head_bytes = static_cast<size_t>(N) * d * 2;
  const size_t head_lse = static_cast<size_t>(N) * 4;
  constexpr int kUnitRows = fa::FwdCfg<128>::kQTiles * fa::FwdCfg<128>::kBM;   // rows per unit (either d)
  const int q_blocks = (N + kUnitRows - 1) / kUnitRows;

  std::lock_guard<std::mutex> lock(hp->mu);
#define FA_TRY(x)                              \
  do {                                         \
    cudaError_t e_ = (x);                      \
    if (e_ != cudaSuccess) return cuda_fail(e_); \
  } while (0)
  // Everything below runs after the work already on `stream` (which may still
  // use the workspace), and `stream` resumes only after the last download.
  FA_TRY(cudaEventRecord(hp->start, stream));
  FA_TRY(cudaStreamWaitEvent(hp->up, hp->start, 0));
  FA_TRY(cudaStreamWaitEvent(hp->aux, hp->start, 0));
  FA_TRY(cudaStreamWaitEvent(hp->down, hp->start, 0));
  for (int c = 0; c < nc; ++c) {
    const int bh0 = c * per;
    const int nbh = std::min(per, BH - bh0);
    if (nbh <= 0) break;
    const size_t off = static_cast<size_t>(bh0) * head_bytes, bytes = static_cast<size_t>(nbh) * head_bytes;
    const size_t loff = static_cast<size_t>(bh0) * head_lse, lbytes = static_cast<size_t>(nbh) * head_lse;
    FA_TRY(cudaMemcpyAsync(Qd + off, qh + off, bytes, cudaMemcpyHostToDevice, hp->up));
    FA_TRY(cudaMemcpyAsync(Kd + off, kh + off, bytes, cudaMemcpyHostToDevice, hp->up));
    FA_TRY(cudaMemcpyAsync(Vd + off, vh + off, bytes, cudaMemcpyHostToDevice, hp->up));
    FA_TRY(cudaEventRecord(hp->in[c], hp->up));
    cudaStream_t cs = (c & 1) ? hp->aux : stream;
    FA_TRY(cudaStreamWaitEvent(cs, hp->in[c], 0));
    // The chunk's heads as a [1, nbh, N, d] problem: the same kernel and the
    // same per-head result as fa_fwd.
    // (with the whole problem's plan for the units CTA pairs share)
    const SplitPlan plan{BH * q_blocks, bh0 * q_blocks};
    const fa_status_t st =
        d == 64 ? launch<64>(Qd + off, Kd + off, Vd + off, Od + off, reinterpret_cast<float*>(Ld + loff), 1, nbh,
                             nbh, N, N, scale, -1, kDefaultTimeoutNs, cs, &plan)
                : launch<128>(Qd + off, Kd + off, Vd + off, Od + off, reinterpret_cast<float*>(Ld + loff), 1, nbh,
                              nbh, N, N, scale, -1, kDefaultTimeoutNs, cs, &plan);
    if (st != FA_OK) return st;
    FA_TRY(cudaEventRecord(hp->done[c], cs));
    FA_TRY(cudaStreamWaitEvent(hp->down, hp->done[c], 0));
    FA_TRY(cudaMemcpyAsync(oh + off, Od + off, bytes, cudaMemcpyDeviceToHost, hp->down));
    FA_TRY(cudaMemcpyAsync(lh + loff, Ld + loff, lbytes, cudaMemcpyDeviceToHost, hp->down));
  }
  // The downloads follow every chunk's kernel, so the last one covers all.
  FA_TRY(cudaEventRecord(hp->end, hp->down));
  FA_TRY(cudaStreamWaitEvent(stream, hp->end, 0));
#undef FA_TRY
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status_t fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                   float scale, cudaStream_t stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, -1, kDefaultTimeoutNs, stream);
}

fa_status_t fa_fwd_launch_shape(int B, int H, int N, int d, int* grid, int* cluster, int* whole_units) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * N >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const FwdDevInfo* fi = d == 64 ? fwd_dev_info<64>(dev) : fwd_dev_info<128>(dev);
  if (!fi) return FA_ERR_UNSUPPORTED;
  if (fi->err != cudaSuccess) return cuda_fail(fi->err);
  using C = fa::FwdCfg<128>;   // the unit and key-block sizes do not depend on d
  const int unit_rows = C::kQTiles * C::kBM;
  const int units = B * H * ((N + unit_rows - 1) / unit_rows);
  const FwdShape sh = fwd_shape(units, (N + C::kBN - 1) / C::kBN, sm_count(dev), fi->max2);
  if (grid) *grid = sh.grid;
  if (cluster) *cluster = sh.cluster;
  if (whole_units) *whole_units = sh.whole_units;
  return FA_OK;
}

size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  return host_workspace_bytes(B, H, N, d);
}

fa_status_t fa_fwd_host(const void* Qh, const void* Kh, const void* Vh, void* Oh, float* LSEh, int B, int H, int N,
                        int d, float scale, int num_chunks, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  return host_impl(Qh, Kh, Vh, Oh, LSEh, B, H, N, d, scale, num_chunks, workspace, workspace_bytes, stream);
}

fa_status_t fa_fwd_fault_test(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                              int N, int d, float scale, int drop_load, unsigned long long timeout_ns,
                              cudaStream_t stream) {
  if (timeout_ns == 0) return FA_ERR_INVALID_ARG;
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, drop_load < 0 ? -1 : drop_load, timeout_ns, stream);
}

fa_status_t fa_get_device_status(cudaStream_t stream, unsigned int* info) {
  if (info)
    for (int i = 0; i < 4; ++i) info[i] = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, fa::g_status_word, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e);
  if (word == 0) return FA_OK;
  unsigned int details[4] = {0, 0, 0, 0};
  e = cudaMemcpyFromSymbol(details, fa::g_status_info, sizeof(details));
  if (e != cudaSuccess) return cuda_fail(e);
  if (info)
    for (int i = 0; i < 4; ++i) info[i] = details[i];
  const unsigned int zeros[4] = {0, 0, 0, 0};
  e = cudaMemcpyToSymbol(fa::g_status_word, zeros, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(fa::g_status_info, zeros, sizeof(zeros));
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_ERR_TIMEOUT;
}

size_t fa_naive_workspace_bytes(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  return static_cast<size_t>(B) * H * N * naive_ld(N) * 2;
}

fa_status_t fa_naive_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                         int d, float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  fa_status_t st = check_args(Q, K, V, O, LSE, B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (!naive_grid_ok(B, H, N)) return FA_ERR_UNSUPPORTED;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 128 != 0) return FA_ERR_INVALID_ARG;
  const size_t need = fa_naive_workspace_bytes(B, H, N);
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  const size_t n_qkv = static_cast<size_t>(B) * H * N * d * 2;
  const size_t n_lse = static_cast<size_t>(B) * H * N * 4;
  for (const void* in : {Q, K, V, static_cast<const void*>(O)})
    if (overlaps(workspace, need, in, n_qkv)) return FA_ERR_INVALID_ARG;
  if (overlaps(workspace, need, LSE, n_lse)) return FA_ERR_INVALID_ARG;
  if (d == 64) return naive_launch<64>(Q, K, V, O, LSE, B, H, N, scale, workspace, stream);
  return naive_launch<128>(Q, K, V, O, LSE, B, H, N, scale, workspace, stream);
}

fa_status_t fa_naive_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                                 int N, int d, float scale, cudaStream_t stream) {
  fa_status_t st = check_args(Q, K, V, O, LSE, B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (fa_naive_workspace_bytes(B, H, N) > kNaiveStaticScratchBytes) return FA_ERR_UNSUPPORTED;
  if (!naive_grid_ok(B, H, N)) return FA_ERR_UNSUPPORTED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  e = naive_static_scratch(dev, &scratch);
  if (e != cudaSuccess) return cuda_fail(e);
  if (d == 64) return naive_launch<64>(Q, K, V, O, LSE, B, H, N, scale, scratch, stream);
  return naive_launch<128>(Q, K, V, O, LSE, B, H, N, scale, scratch, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  return 2 * static_cast<size_t>(B) * H * static_cast<size_t>(bwd_npad(N)) * 4;
}

}  // extern "C"

namespace {

fa_status_t bwd_impl(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                     void* dQ, void* dK, void* dV, int B, int H, int N, int d, float scale, void* workspace,
                     size_t workspace_bytes, int drop_load, unsigned long long timeout_ns, cudaStream_t stream) {
  fa_status_t st = check_args(Q, K, V, O, LSE, B, H, N, d, scale);
  if (st != FA_OK) return st;
  // The main launch is a 1-D grid: one CTA per 128 rows of every head, in
  // each of its two roles.
  if (2LL * (bwd_npad(N) / 128) * B * H > 2147483647LL) return FA_ERR_UNSUPPORTED;
  if (!dO || !dQ || !dK || !dV || !workspace) return FA_ERR_INVALID_ARG;
  for (const void* ptr : {dO, static_cast<const void*>(dQ), static_cast<const void*>(dK),
                          static_cast<const void*>(dV)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 128 != 0) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_bytes(B, H, N);
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  const size_t n_qkv = static_cast<size_t>(B) * H * N * d * 2;
  const size_t n_lse = static_cast<size_t>(B) * H * N * 4;
  // Every written buffer (dQ, dK, dV, workspace) is disjoint from every
  // input and from the other written buffers.
  const void* outs[4] = {dQ, dK, dV, workspace};
  const size_t out_n[4] = {n_qkv, n_qkv, n_qkv, need};
  for (int a = 0; a < 4; ++a) {
    for (const void* in : {Q, K, V, O, dO})
      if (overlaps(outs[a], out_n[a], in, n_qkv)) return FA_ERR_INVALID_ARG;
    if (overlaps(outs[a], out_n[a], LSE, n_lse)) return FA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a], out_n[a], outs[b], out_n[b])) return FA_ERR_INVALID_ARG;
  }
  if (d == 64)
    return bwd_launch<64>(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, scale, workspace, drop_load, timeout_ns, stream);
  return bwd_launch<128>(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, scale, workspace, drop_load, timeout_ns, stream);
}

// ---------------------------------------------------------------- shared K/V heads, short queries
struct KvPlan {
  int G, hp, box_q, q_blocks, tiles_per_group, n_kv_blocks, blocks_per_split, num_splits;
};

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
  return sms;
}

// Packing and key split of the short-query kernel. A tile is 128 query rows:
// for N_q <= 128 the rows of min(G, 128 / N_q) heads of a group, for
// N_q > 128 one 128-row block of one head. With num_splits <= 0 the split
// count fills one wave of CTAs (two per SM); it is capped by the number of
// key blocks, and ranges are whole blocks with no empty range.
KvPlan kv_plan(int B, int H, int H_kv, int N_q, int N_kv, int num_splits) {
  KvPlan k;
  k.G = H / H_kv;
  if (N_q <= 128) {
    k.hp = std::min(k.G, 128 / N_q);
    k.box_q = N_q;
    k.q_blocks = 1;
  } else {
    k.hp = 1;
    k.box_q = 128;
    k.q_blocks = (N_q + 127) / 128;
  }
  k.tiles_per_group = (k.G + k.hp - 1) / k.hp * k.q_blocks;
  k.n_kv_blocks = (N_kv + 127) / 128;
  int s = num_splits;
  if (s <= 0) {
    const long long base = static_cast<long long>(B) * H_kv * k.tiles_per_group;
    const int sms = device_sm_count();
    const long long slots = static_cast<long long>(sms) * 2;   // resident short-query CTAs (two per SM)
    s = base >= slots ? 1 : static_cast<int>(slots / base);
  }
  s = std::max(1, std::min(s, k.n_kv_blocks));
  k.blocks_per_split = (k.n_kv_blocks + s - 1) / s;
  k.num_splits = (k.n_kv_blocks + k.blocks_per_split - 1) / k.blocks_per_split;
  return k;
}

// Which kernel runs fa_fwd_kv. Short query blocks (N_q <= 128) take the
// short-query kernel. Long ones take the fused forward kernel (two query
// tiles per CTA, one CTA per SM, no split) when num_splits is 1, and with
// num_splits = 0 whenever its CTAs fill more than three quarters of the SMs;
// otherwise the short-query kernel with one 128-row query tile per CTA and a
// key split fills the device. Both full, the short-query kernel runs long
// query blocks at about 0.8 of the fused kernel's rate.
struct KvRoute {
  bool fused;
  KvPlan plan;
};

KvRoute kv_route(int B, int H, int H_kv, int N_q, int N_kv, int num_splits) {
  KvRoute r{false, kv_plan(B, H, H_kv, N_q, N_kv, num_splits)};
  if (N_q <= 128) return r;
  if (num_splits == 1) {
    r.fused = true;
  } else if (num_splits <= 0) {
    const long long fused_ctas = static_cast<long long>(B) * H * ((N_q + 255) / 256);
    r.fused = 4 * fused_ctas > 3LL * device_sm_count() || r.plan.num_splits <= 1;
  }
  return r;
}

size_t kv_workspace_bytes(int B, int H, int N_q, int d, const KvPlan& k) {
  if (k.num_splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N_q;
  return static_cast<size_t>(k.num_splits) * rows * (d + 1) * 4;
}

fa_status_t kv_check(const void* Q, const void* K, const void* V, const void* O, const float* LSE, int B, int H,
                     int H_kv, int N_q, int N_kv, int d, float scale, size_t o_elem_bytes) {
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || H_kv < 1 || N_q < 1 || N_kv < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * N_q >= (1LL << 31) || static_cast<long long>(B) * H_kv * N_kv >= (1LL << 31))
    return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  for (const void* ptr : {Q, K, V, O})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(LSE) % 4 != 0) return FA_ERR_INVALID_ARG;
  const size_t n_q = static_cast<size_t>(B) * H * N_q * d * 2;
  const size_t n_o = static_cast<size_t>(B) * H * N_q * d * o_elem_bytes;
  const size_t n_kv = static_cast<size_t>(B) * H_kv * N_kv * d * 2;
  const size_t n_lse = static_cast<size_t>(B) * H * N_q * 4;
  if (overlaps(O, n_o, Q, n_q) || overlaps(O, n_o, K, n_kv) || overlaps(O, n_o, V, n_kv)) return FA_ERR_INVALID_ARG;
  if (overlaps(LSE, n_lse, Q, n_q) || overlaps(LSE, n_lse, K, n_kv) || overlaps(LSE, n_lse, V, n_kv) ||
      overlaps(LSE, n_lse, O, n_o))
    return FA_ERR_INVALID_ARG;
  return FA_OK;
}

template <int HD>
fa_status_t decode_launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int H_kv,
                          int N_q, int N_kv, float scale, const KvPlan& k, void* ws, bool f32_out, int drop_load,
                          unsigned long long timeout_ns, cudaStream_t stream) {
  using C = fa::DecCfg<HD>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  static bool regs_ok[64];
  std::call_once(once[dev], [&] {
    attr_err[dev] =
        cudaFuncSetAttribute(fa::fa_decode_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    // The warpgroups' register split must fit the registers the block is
    // launched with (see the forward launch).
    cudaFuncAttributes fattr;
    if (attr_err[dev] == cudaSuccess) attr_err[dev] = cudaFuncGetAttributes(&fattr, fa::fa_decode_kernel<HD>);
    regs_ok[dev] = attr_err[dev] == cudaSuccess && 4 * C::kRegsSoftmax + 4 * C::kRegsControl <= 8 * fattr.numRegs;
  });
  if (attr_err[dev] != cudaSuccess) return cuda_fail(attr_err[dev]);
  if (!regs_ok[dev]) return FA_ERR_UNSUPPORTED;

  // Q as [B*H][N_q][d] with a box of 64 x N_q rows x hp heads: one load
  // brings the packed rows of hp query heads. K, V as [B*H_kv][N_kv][d].
  CUtensorMap mq, mk, mv;
  auto fn = encode_fn();
  if (!fn) return cuda_fail(cudaErrorInvalidValue);
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(N_q),
                          static_cast<cuuint64_t>(B) * H};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(HD) * 2, static_cast<cuuint64_t>(N_q) * HD * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(k.box_q), static_cast<cuuint32_t>(k.hp)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(Q), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cuda_fail(cudaErrorInvalidValue);
  }
  if (!make_map(&mk, K, B * H_kv, N_kv, HD) || !make_map(&mv, V, B * H_kv, N_kv, HD))
    return cuda_fail(cudaErrorInvalidValue);

  fa::DecParams p;
  const size_t rows = static_cast<size_t>(B) * H * N_q;
  p.O = f32_out ? nullptr : static_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.f32_out = f32_out ? 1 : 0;
  if (k.num_splits > 1) {
    p.O_part = static_cast<float*>(ws);
    p.LSE_part = static_cast<float*>(ws) + static_cast<size_t>(k.num_splits) * rows * HD;
  } else {
    // One split with float32 results: the kernel's partial result is the result.
    p.O_part = f32_out ? static_cast<float*>(O) : nullptr;
    p.LSE_part = f32_out ? LSE : nullptr;
  }
  p.N_q = N_q;
  p.N_kv = N_kv;
  p.H = H;
  p.H_kv = H_kv;
  p.G = k.G;
  p.hp = k.hp;
  p.box_q = k.box_q;
  p.q_blocks = k.q_blocks;
  p.tiles_per_group = k.tiles_per_group;
  p.n_kv_blocks = k.n_kv_blocks;
  p.blocks_per_split = k.blocks_per_split;
  p.num_splits = k.num_splits;
  // scale < 0: the tensor core forms -S and the kernel runs with |scale|.
  p.scale_log2 = static_cast<float>(std::fabs(static_cast<double>(scale)) * 1.4426950408889634074);
  p.idesc_qk = C::kIdescQK | (scale < 0.f ? fa::ptx::kIdescNegateA : 0u);
  p.timeout_ns = timeout_ns;
  p.drop_load = drop_load;
  const dim3 grid(static_cast<unsigned>(k.tiles_per_group * k.num_splits), H_kv, B);
  fa::fa_decode_kernel<HD><<<grid, C::kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  if (k.num_splits > 1) {
    // The merge as a programmatic dependent launch: it is scheduled while the
    // decode grid finishes and waits (griddepcontrol.wait) for its partials.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (f32_out)
      e = cudaLaunchKernelEx(&cfg, fa::decode_merge_kernel<HD, float>, static_cast<const float*>(p.O_part),
                             static_cast<const float*>(p.LSE_part), static_cast<float*>(O), LSE,
                             static_cast<long long>(rows), k.num_splits);
    else
      e = cudaLaunchKernelEx(&cfg, fa::decode_merge_kernel<HD>, static_cast<const float*>(p.O_part),
                             static_cast<const float*>(p.LSE_part), static_cast<__nv_bfloat16*>(O), LSE,
                             static_cast<long long>(rows), k.num_splits);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return FA_OK;
}

fa_status_t kv_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int H_kv,
                    int N_q, int N_kv, int d, float scale, int num_splits, void* workspace, size_t workspace_bytes,
                    bool f32_out, int drop_load, unsigned long long timeout_ns, cudaStream_t stream) {
  fa_status_t st = kv_check(Q, K, V, O, LSE, B, H, H_kv, N_q, N_kv, d, scale, f32_out ? 4 : 2);
  if (st != FA_OK) return st;
  // Float32 results come from the short-query kernel (the fused kernel
  // writes bf16).
  const KvRoute route =
      f32_out ? KvRoute{false, kv_plan(B, H, H_kv, N_q, N_kv, num_splits)} : kv_route(B, H, H_kv, N_q, N_kv, num_splits);
  if (route.fused) {
    // Long query blocks: the fused forward kernel with the K/V head mapping.
    if (d == 64) return launch<64>(Q, K, V, O, LSE, B, H, H_kv, N_q, N_kv, scale, drop_load, timeout_ns, stream);
    return launch<128>(Q, K, V, O, LSE, B, H, H_kv, N_q, N_kv, scale, drop_load, timeout_ns, stream);
  }
  const KvPlan& k = route.plan;
  if (static_cast<long long>(k.tiles_per_group) * k.num_splits > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;  // grid.x
  const size_t need = kv_workspace_bytes(B, H, N_q, d, k);
  if (need > 0) {
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 128 != 0 || workspace_bytes < need)
      return FA_ERR_INVALID_ARG;
    const size_t n_q = static_cast<size_t>(B) * H * N_q * d * 2;
    const size_t n_o = static_cast<size_t>(B) * H * N_q * d * (f32_out ? 4 : 2);
    const size_t n_kv = static_cast<size_t>(B) * H_kv * N_kv * d * 2;
    if (overlaps(workspace, need, Q, n_q) || overlaps(workspace, need, K, n_kv) ||
        overlaps(workspace, need, V, n_kv) || overlaps(workspace, need, O, n_o) ||
        overlaps(workspace, need, LSE, static_cast<size_t>(B) * H * N_q * 4))
      return FA_ERR_INVALID_ARG;
  }
  if (d == 64)
    return decode_launch<64>(Q, K, V, O, LSE, B, H, H_kv, N_q, N_kv, scale, k, workspace, f32_out, drop_load,
                             timeout_ns, stream);
  return decode_launch<128>(Q, K, V, O, LSE, B, H, H_kv, N_q, N_kv, scale, k, workspace, f32_out, drop_load,
                            timeout_ns, stream);
}

}  // namespace

extern "C" {

int fa_fwd_kv_num_splits(int B, int H, int H_kv, int N_q, int N_kv, int d) {
  if (B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || N_q < 1 || N_kv < 1 || (d != 64 && d != 128)) return 0;
  const KvRoute r = kv_route(B, H, H_kv, N_q, N_kv, 0);
  return r.fused ? 1 : r.plan.num_splits;
}

size_t fa_fwd_kv_workspace_bytes(int B, int H, int H_kv, int N_q, int N_kv, int d, int num_splits) {
  if (B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || N_q < 1 || N_kv < 1 || (d != 64 && d != 128)) return 0;
  const KvRoute r = kv_route(B, H, H_kv, N_q, N_kv, num_splits);
  return r.fused ? 0 : kv_workspace_bytes(B, H, N_q, d, r.plan);
}

fa_status_t fa_fwd_kv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int H_kv,
                      int N_q, int N_kv, int d, float scale, int num_splits, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  return kv_impl(Q, K, V, O, LSE, B, H, H_kv, N_q, N_kv, d, scale, num_splits, workspace, workspace_bytes, false, -1,
                 kDefaultTimeoutNs, stream);
}

size_t fa_fwd_kv_f32_workspace_bytes(int B, int H, int H_kv, int N_q, int N_kv, int d, int num_splits) {
  if (B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || N_q < 1 || N_kv < 1 || (d != 64 && d != 128)) return 0;
  return kv_workspace_bytes(B, H, N_q, d, kv_plan(B, H, H_kv, N_q, N_kv, num_splits));
}

fa_status_t fa_fwd_kv_f32(const void* Q, const void* K, const void* V, float* O, float* LSE, int B, int H, int H_kv,
                          int N_q, int N_kv, int d, float scale, int num_splits, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  return kv_impl(Q, K, V, O, LSE, B, H, H_kv, N_q, N_kv, d, scale, num_splits, workspace, workspace_bytes, true, -1,
                 kDefaultTimeoutNs, stream);
}

fa_status_t fa_fwd_kv_fault_test(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                                 int H_kv, int N_q, int N_kv, int d, float scale, int num_splits, void* workspace,
                                 size_t workspace_bytes, int drop_load, unsigned long long timeout_ns,
                                 cudaStream_t stream) {
  if (timeout_ns == 0) return FA_ERR_INVALID_ARG;
  return kv_impl(Q, K, V, O, LSE, B, H, H_kv, N_q, N_kv, d, scale, num_splits, workspace, workspace_bytes, false,
                 drop_load < 0 ? -1 : drop_load, timeout_ns, stream);
}

fa_status_t fa_merge_partials(const float* O_parts, const float* LSE_parts, void* O, float* LSE, int num_parts,
                              long long rows, int d, cudaStream_t stream) {
  if (!O_parts || !LSE_parts || !O || !LSE || num_parts < 1 || rows < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (rows >= (1LL << 31) / 8) return FA_ERR_INVALID_ARG;
  const void* ptrs[4] = {O_parts, LSE_parts, O, LSE};
  for (const void* ptr : ptrs)
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return FA_ERR_INVALID_ARG;
  const size_t n_op = static_cast<size_t>(num_parts) * rows * d * 4;
  const size_t n_lp = static_cast<size_t>(num_parts) * rows * 4;
  const size_t n_o = static_cast<size_t>(rows) * d * 2;
  const size_t n_l = static_cast<size_t>(rows) * 4;
  if (overlaps(O, n_o, O_parts, n_op) || overlaps(O, n_o, LSE_parts, n_lp) || overlaps(LSE, n_l, O_parts, n_op) ||
      overlaps(LSE, n_l, LSE_parts, n_lp) || overlaps(O, n_o, LSE, n_l))
    return FA_ERR_INVALID_ARG;
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  if (d == 64)
    fa::decode_merge_kernel<64><<<grid, 256, 0, stream>>>(O_parts, LSE_parts, static_cast<__nv_bfloat16*>(O), LSE,
                                                         rows, num_parts);
  else
    fa::decode_merge_kernel<128><<<grid, 256, 0, stream>>>(O_parts, LSE_parts, static_cast<__nv_bfloat16*>(O), LSE,
                                                          rows, num_parts);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

fa_status_t fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                   void* dQ, void* dK, void* dV, int B, int H, int N, int d, float scale, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, workspace, workspace_bytes, -1,
                  kDefaultTimeoutNs, stream);
}

fa_status_t fa_bwd_fault_test(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                              const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int N, int d, float scale,
                              void* workspace, size_t workspace_bytes, int drop_load, unsigned long long timeout_ns,
                              cudaStream_t stream) {
  if (timeout_ns == 0) return FA_ERR_INVALID_ARG;
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, workspace, workspace_bytes,
                  drop_load < 0 ? -1 : drop_load, timeout_ns, stream);
}

const char* fa_status_string(fa_status_t status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

int fa_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"
