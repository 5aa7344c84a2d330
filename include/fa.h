/*
 * fa.h -- C ABI of the exact attention forward pass (and its backward by
 * recomputation) for GB300 (sm_103a).
 *
 * The operation: for every batch b and head h,
 *     S = scale * Q K^T              (N x N scores, never written to memory)
 *     P = softmax(S) row by row      (safe softmax: subtract the row maximum)
 *     O = P V                         (N x d, bf16)
 *     LSE[r] = m_r + ln(sum_j e^{S_rj - m_r})   (one float per query row)
 * computed in one fused kernel launch that reads Q, K, V once per query
 * block and writes only O and LSE.
 *
 * Sources (page title, then section):
 *   - "01 · 注意力为什么是 IO 瓶颈" (ai-reference-codex FlashAttention chapter 01),
 *     §4 (the fused kernel reads Q, K, V and writes only O and LSE) and §6
 *     (softmax_lse is one float32 per query row; one kernel launch on the
 *     caller's stream).
 *   - "Flash Attention (FA1)" (languisher.top), "Naive Attention 问题分析"
 *     (the safe softmax), "Tiling in FlashAttention" (Br x d query blocks,
 *     Bc x d key/value blocks, ceil(N/B) blocks) and the derivation of the
 *     online-softmax update (steps 1-5, boxed O_new equation).
 *   - "FlashAttention：IO 感知的精确注意力" (inference.xph.ink kp-015), core
 *     concepts: exact, not approximate; FlashAttention-2 work split.
 *
 * Conventions of this library (the pages do not fix an interface):
 *   - Layout: Q, K, V and O are bf16, contiguous row-major [B, H, N, d]
 *     (d fastest). LSE is float32, contiguous [B, H, N], natural logarithm of
 *     the sum of e^{scaled score}: LSE = max_j S_rj + ln(sum_j e^{S_rj - max}).
 *   - Ownership: the caller allocates every buffer (device memory) and keeps
 *     ownership; the library allocates no device memory and keeps no pointer
 *     after the call returns.
 *   - Asynchrony: fa_fwd only validates its arguments, encodes the TMA
 *     descriptors and enqueues one kernel on `stream`. Errors found on the
 *     host are returned immediately and nothing is launched. A device-side
 *     timeout (a pipeline wait that did not finish within its limit, which a
 *     correct build never hits) is reported later by fa_get_device_status.
 *   - Supported: d in {64, 128}; B, H, N >= 1 with B <= 65535, H <= 65535,
 *     B*H*N < 2^31; scale finite, of either sign (zero gives uniform
 *     weights); non-causal (no mask).
 *   - Pointers: Q, K, V, O must be 16-byte aligned, LSE 4-byte aligned. O and
 *     LSE must not overlap Q, K, V or each other.
 */
#ifndef EXACT_IO_AWARE_34_FA_H_
#define EXACT_IO_AWARE_34_FA_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null or misaligned pointer, bad size, non-finite scale, overlap */
  FA_ERR_UNSUPPORTED = 2,  /* a valid request this build does not implement (d, a grid limit) */
  FA_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed; see fa_last_cuda_error() */
  FA_ERR_TIMEOUT = 4       /* a device-side pipeline wait ran out of time (reported after the fact) */
} fa_status_t;

/*
 * fa_fwd -- exact attention forward pass, one kernel launch.
 *   Q, K, V : device, bf16 [B, H, N, d], read only.
 *   O       : device, bf16 [B, H, N, d], written (every element).
 *   LSE     : device, float32 [B, H, N], written (every element).
 *   B, H, N, d : batch, heads, sequence length, head dimension.
 *   scale   : multiplies Q K^T before the softmax (1/sqrt(d) is usual).
 *   stream  : CUDA stream the kernel is enqueued on (0 = legacy default).
 * Returns FA_OK once the kernel is enqueued; otherwise an error code and
 * nothing is launched (FA_ERR_CUDA: the launch itself failed).
 * The launch is a persistent grid of at most one CTA per SM walking units of
 * 256 query rows; when the units of its last, partial round fill at most
 * half of the SMs, it is launched as clusters of two CTAs that share those
 * units (half of the key blocks each, merged on chip; see
 * fa_fwd_launch_shape). The result does not depend on the stream or on other
 * work on the GPU, but it does depend on the SM count (which units are
 * shared), like any reduction order.
 * Follows: "Flash Attention (FA1)" tiling and online-softmax update;
 * "01 · 注意力为什么是 IO 瓶颈" §4/§6 for the O + LSE outputs.
 */
fa_status_t fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                   int B, int H, int N, int d, float scale, cudaStream_t stream);

/*
 * fa_fwd_launch_shape -- the launch fa_fwd makes for these sizes on the
 * current device (informational; it launches nothing and reads no data).
 *   grid        : host, receives the number of CTAs (at most the SM count).
 *   cluster     : host, receives 1 (no shared units) or 2 (CTA pairs share
 *                 the units of the last, partial round).
 *   whole_units : host, receives how many units of 256 query rows are run
 *                 whole by one CTA; the other B*H*ceil(N/256) - whole_units
 *                 are shared.
 * Any of the three may be NULL. Returns FA_ERR_INVALID_ARG or
 * FA_ERR_UNSUPPORTED for sizes fa_fwd rejects, FA_ERR_CUDA if the device
 * cannot be queried, else FA_OK.
 */
fa_status_t fa_fwd_launch_shape(int B, int H, int N, int d, int* grid, int* cluster, int* whole_units);

/*
 * fa_fwd_host_workspace_bytes -- device workspace fa_fwd_host needs: room for
 * device copies of Q, K, V, O (bf16 [B, H, N, d] each) and LSE (float32
 * [B, H, N]), each part padded to 256 bytes. 0 for unsupported sizes.
 */
size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_fwd_host -- fa_fwd on HOST buffers, end to end: uploads Q, K, V, runs the
 * forward kernel and downloads O and LSE, pipelined over groups of (b, h)
 * heads so that the uploads of one group and the downloads of another overlap
 * the kernel on a third. Each head's O and LSE are bit for bit those of fa_fwd
 * (the group launches follow the whole problem's choice of the units CTA
 * pairs share).
 *   Qh, Kh, Vh : host, bf16 [B, H, N, d], read. Page-locked (pinned) memory
 *                gives full copy bandwidth; pageable memory works, slower.
 *   Oh, LSEh   : host, bf16 [B, H, N, d] and float32 [B, H, N], written.
 *   num_chunks : head groups, 0 for the default of 8; capped at B*H and at 16.
 *   workspace  : device, fa_fwd_host_workspace_bytes(B, H, N, d) bytes at
 *                least, 256-byte aligned, owned by the caller, overlapping no
 *                host buffer; its contents are overwritten.
 *   stream     : the call is ordered after the work already on `stream`, and
 *                `stream` reaches the end of the call only when Oh and LSEh
 *                are written: synchronise `stream` before reading them. The
 *                copies run on two internal streams and every second group's
 *                kernel on a third (created once per device).
 * Limits and error codes as for fa_fwd, checked on the host before anything
 * is enqueued; FA_ERR_INVALID_ARG also for a missing, misaligned, small or
 * overlapping workspace or overlapping host buffers.
 */
fa_status_t fa_fwd_host(const void* Qh, const void* Kh, const void* Vh, void* Oh, float* LSEh,
                        int B, int H, int N, int d, float scale, int num_chunks,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_get_device_status -- synchronise `stream`, then read and clear the
 * library's device status word on the current device. Returns FA_OK, or
 * FA_ERR_TIMEOUT if any kernel of this library on this device gave up on a
 * wait since the last call, or FA_ERR_CUDA if the synchronisation failed.
 * `info`, if not NULL, receives 4 words describing the first timeout:
 * {role (forward: 1 producer, 2 mma, 3 softmax/epilogue; backward dQ CTA:
 * 4, 5, 6; backward dK/dV CTA: 7, 8, 9; short-query kernel of fa_fwd_kv:
 * 10, 11, 12, in the same order), blockIdx.x, blockIdx.y,
 * blockIdx.z}; all zero when there was none. (`info` is this library's
 * addition for diagnosing a timeout; with info = NULL the call only reports
 * the status.)
 */
fa_status_t fa_get_device_status(cudaStream_t stream, unsigned int* info);

/* fa_status_string -- a static, human-readable name for a status code. */
const char* fa_status_string(fa_status_t status);

/* fa_last_cuda_error -- the cudaError_t behind the most recent FA_ERR_CUDA
 * returned on this host thread (0 if none). */
int fa_last_cuda_error(void);

/*
 * fa_naive_workspace_bytes -- bytes of device workspace fa_naive_fwd needs for
 * B x H heads of length N: the N x N score matrix of every head in bf16,
 * rows padded to a multiple of 64 elements. Returns 0 for non-positive sizes.
 */
size_t fa_naive_workspace_bytes(int B, int H, int N);

/*
 * fa_naive_fwd -- standard attention with the N x N intermediates in HBM:
 * the comparator the fused kernel is measured against. Three kernel launches
 * on `stream`, as "01 · 注意力为什么是 IO 瓶颈" §3 and §5 describe:
 *   S = bf16(scale * bf16(Q K^T))   (written to `workspace`)
 *   P = bf16(softmax(S))            (written over S; LSE = m + ln l per row)
 *   O = bf16(P V)
 * Arguments as for fa_fwd, plus `workspace`: device memory of at least
 * fa_naive_workspace_bytes(B, H, N) bytes, 128-byte aligned, owned by the
 * caller, not overlapping any other buffer; its contents are overwritten.
 * Same shape limits and error codes as fa_fwd; FA_ERR_INVALID_ARG also for
 * a missing, misaligned, too small or overlapping workspace, and
 * FA_ERR_UNSUPPORTED (before any CUDA call) when B*H > 65535 or
 * ceil(N / 128) > 65535 (the launches' grid limits).
 */
fa_status_t fa_naive_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                         int B, int H, int N, int d, float scale,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_naive_fwd_noalloc -- fa_naive_fwd for callers that cannot allocate
 * device memory, e.g. a service that reserves all of its GPU memory at
 * start-up and forbids any later cudaMalloc, or a code path where the latency
 * or possible failure of an allocation is not acceptable. (The pages have no
 * counterpart: this is an interface convenience of this library.)
 * Same arguments, results and errors as fa_naive_fwd, minus the workspace:
 * the N x N matrices live in a 64 MiB (67108864-byte) array inside the
 * library's device image, which every GPU that loads the library holds until
 * the process exits. Requests whose fa_naive_workspace_bytes() exceed
 * 64 MiB return FA_ERR_UNSUPPORTED without launching anything (for example
 * B*H = 8 heads of N = 2048, or one head of N = 5760, still fit).
 *   - The call allocates nothing (no cudaMalloc, no library allocator).
 *   - The B*H and N limits of fa_naive_fwd apply too (FA_ERR_UNSUPPORTED).
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. A failed lookup returns FA_ERR_CUDA and is
 *     not remembered: the next call on that device tries again.
 *   - Every call on a device shares the one array, and the array keeps the
 *     last call's contents (nothing in it needs to start at zero). Calls whose
 *     kernels overlap on the GPU (different streams, no ordering between them)
 *     race on it: order them, e.g. issue them on one stream.
 */
fa_status_t fa_naive_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                 int B, int H, int N, int d, float scale, cudaStream_t stream);

/*
 * fa_fwd_kv -- the forward pass with shared key/value heads (GQA) and
 * separate query and key lengths: the prefill and decode shapes of a model
 * whose H query heads share H_kv key/value heads ("FlashAttention：IO 感知的
 * 精确注意力", "与其他知识点的关系": grouped K/V heads combine with the exact,
 * IO-aware kernel; "常见误区": decode is bandwidth-bound).
 *   Q      : device, bf16 [B, H, N_q, d], read only.
 *   K, V   : device, bf16 [B, H_kv, N_kv, d], read only. H must be a multiple
 *            of H_kv; query head h attends to K/V head h / (H / H_kv).
 *   O      : device, bf16 [B, H, N_q, d], written.
 *   LSE    : device, float32 [B, H, N_q], written (natural log).
 *   Every query row attends to all N_kv keys (no mask).
 *   num_splits : the number of contiguous key ranges computed by separate
 *            CTAs and merged with the online-softmax rule ("Flash Attention
 *            (FA1)", derivation steps 4-5). 0 chooses (fa_fwd_kv_num_splits):
 *            for N_q <= 128 one wave of CTAs; for N_q > 128 no split (the
 *            fused forward kernel) unless that kernel would fill at most
 *            three quarters of the SMs, else one wave. Values above the
 *            number of 128-key blocks are capped. For N_q > 128, 1 always
 *            takes the fused forward kernel (the same result as fa_fwd when
 *            H_kv = H and N_q = N_kv).
 *   workspace, workspace_bytes : device memory of at least
 *            fa_fwd_kv_workspace_bytes(...) bytes, 128-byte aligned, not
 *            overlapping any other buffer; may be NULL when that is 0 (one
 *            split or the fused forward kernel).
 * The short-query kernel tiles 128 query rows: for N_q <= 128 the rows of
 * the heads sharing a K/V head are packed into one tile (min(H/H_kv, 128/N_q)
 * heads per tile), so each K/V tile is read once per group; for N_q > 128 a
 * tile is one 128-row block of one head. Launches: one kernel, plus one merge
 * kernel when there is more than one split (a programmatic dependent launch:
 * it is scheduled as the first grid ends and waits for it on the device). Limits as for fa_fwd;
 * FA_ERR_INVALID_ARG also when H is not a multiple of H_kv or for a missing,
 * misaligned, small or overlapping workspace.
 */
fa_status_t fa_fwd_kv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                      int B, int H, int H_kv, int N_q, int N_kv, int d, float scale,
                      int num_splits, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* fa_fwd_kv_num_splits -- the split count fa_fwd_kv uses when num_splits is 0
 * (1 when it takes the fused forward kernel); 0 for invalid sizes. Depends on
 * the current device's SM count (148 when there is no device). */
int fa_fwd_kv_num_splits(int B, int H, int H_kv, int N_q, int N_kv, int d);

/* fa_fwd_kv_workspace_bytes -- workspace bytes fa_fwd_kv needs for these sizes
 * and num_splits (0 = the automatic choice): num_splits * B*H*N_q * (d + 1)
 * float32 partial results when there is more than one split, else 0. */
size_t fa_fwd_kv_workspace_bytes(int B, int H, int H_kv, int N_q, int N_kv, int d, int num_splits);

/*
 * fa_fwd_kv_f32_workspace_bytes -- workspace bytes fa_fwd_kv_f32 needs:
 * num_splits * B*H*N_q * (d + 1) float32 partial results when the short-query
 * kernel's key split (num_splits, 0 = automatic, as for fa_fwd_kv) has more
 * than one range, else 0. 0 also for invalid sizes.
 */
size_t fa_fwd_kv_f32_workspace_bytes(int B, int H, int H_kv, int N_q, int N_kv, int d, int num_splits);

/*
 * fa_fwd_kv_f32 -- fa_fwd_kv with O kept in float32: O[r] is the softmax-
 * weighted sum of the value rows, normalised by its own l, not rounded to
 * bf16. This is the partial result one device of a sequence split hands to
 * the others: the exchange carries it in float32 and only the final merge
 * (fa_merge_partials) rounds, once ("Flash Attention (FA1)", derivation
 * steps 4-5: partial results over disjoint key sets combine exactly).
 *   O   : device, float32 [B, H, N_q, d], written.  LSE : float32 [B, H, N_q].
 *   Other arguments, limits and errors as for fa_fwd_kv. Every shape runs on
 *   the short-query kernel (128 query rows per tile); with more than one key
 *   range a merge kernel writes O and LSE (two launches), with one the kernel
 *   writes them itself.
 */
fa_status_t fa_fwd_kv_f32(const void* Q, const void* K, const void* V, float* O, float* LSE,
                          int B, int H, int H_kv, int N_q, int N_kv, int d, float scale,
                          int num_splits, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_fwd_kv_fault_test -- TEST HOOK, not for production use. fa_fwd_kv with
 * every device-side wait limited to `timeout_ns`, and, when drop_load >= 0,
 * the drop_load-th K/V tile load skipped in every CTA (in the short-query
 * kernel: K, V of a CTA's first block, then of its second, ...; in the fused
 * forward kernel as for fa_fwd_fault_test).
 */
fa_status_t fa_fwd_kv_fault_test(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                 int B, int H, int H_kv, int N_q, int N_kv, int d, float scale,
                                 int num_splits, void* workspace, size_t workspace_bytes,
                                 int drop_load, unsigned long long timeout_ns, cudaStream_t stream);

/*
 * fa_merge_partials -- combine attention results computed over disjoint key
 * sets into the result over their union, by the online-softmax rule
 * ("Flash Attention (FA1)", derivation steps 4-5, in log-sum-exp form):
 *     LSE = ln sum_p e^{LSE_p},   O = sum_p e^{LSE_p - LSE} O_p.
 * This is the exchange step of a sequence split of K/V across devices: each
 * device computes (O_p, LSE_p) for its key shard (fa_fwd / fa_fwd_kv), the
 * partial results are gathered, and one call merges them.
 *   O_parts   : device, float32 [num_parts][rows][d], each normalised by its own l_p.
 *   LSE_parts : device, float32 [num_parts][rows], natural log.
 *   O         : device, bf16 [rows][d], written.   LSE : device, float32 [rows], written.
 *   rows      : number of query rows (e.g. B*H*N_q); d in {64, 128}.
 * All pointers 16-byte aligned; outputs must not overlap inputs or each other.
 * One kernel launch on `stream`.
 */
fa_status_t fa_merge_partials(const float* O_parts, const float* LSE_parts, void* O, float* LSE,
                              int num_parts, long long rows, int d, cudaStream_t stream);

/*
 * fa_bwd_workspace_bytes -- bytes of device workspace fa_bwd needs for
 * B x H heads of length N: two float32 values per query row, rows padded to
 * a multiple of 128. Returns 0 for non-positive sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N);

/*
 * fa_bwd -- exact attention backward pass by recomputation. For every (b, h)
 * it forms the gradients of <dO, O> for O = softmax(scale Q K^T) V:
 *     P  = exp(scale Q K^T - LSE)   (rebuilt from the forward's LSE)
 *     D  = rowsum(dO * O)           (from the forward's O)
 *     dV = P^T dO,   dS = P * (dO V^T - D),   dQ = scale dS K,   dK = scale dS^T Q
 * without writing any N x N matrix to memory ("01 · 注意力为什么是 IO 瓶颈"
 * §7: only O and LSE are kept from the forward and P is recomputed instead
 * of being stored and read back; the gradient formulas are the chain rule of
 * the forward's definition, which the pages do not print).
 *   Q, K, V, O, dO : device, bf16 [B, H, N, d], read only. O and LSE are the
 *                    outputs of fa_fwd (or any forward with the same meaning).
 *   LSE            : device, float32 [B, H, N], read only, natural log.
 *   dQ, dK, dV     : device, bf16 [B, H, N, d], written (every element).
 *   workspace      : device, at least fa_bwd_workspace_bytes(B, H, N) bytes,
 *                    128-byte aligned, owned by the caller; overwritten.
 *   B, H, N, d, scale, stream : as for fa_fwd (same limits).
 * Two kernel launches on `stream`: a per-row pass over O and dO, then one
 * launch whose CTAs take one of two roles: dK/dV (one CTA per 128 key rows)
 * or dQ (one CTA per 128 query rows). Inputs must be 16-byte aligned (LSE 4-byte); dQ, dK, dV and
 * the workspace must not overlap any input or each other. Errors as for
 * fa_fwd, plus FA_ERR_INVALID_ARG for a missing, misaligned, too small or
 * overlapping output or workspace, and FA_ERR_UNSUPPORTED when
 * 2 * ceil(N / 128) * B * H exceeds 2^31 - 1 (the CTA count of the main launch).
 */
fa_status_t fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                   const float* LSE, void* dQ, void* dK, void* dV,
                   int B, int H, int N, int d, float scale,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_fwd_fault_test -- TEST HOOK, not for production use. Same as fa_fwd,
 * but (a) every device-side wait gives up after `timeout_ns` nanoseconds,
 * and (b) when `drop_load` >= 0 the producer skips the drop_load-th K/V tile
 * load (0 = K of block 0, 1 = V of block 0, 2 = K of block 1, ...) in every
 * CTA, so that its consumer's wait runs out. The kernel then stops every role,
 * waits for its own copies and tensor-core work in flight, frees its tensor
 * memory and exits normally; fa_get_device_status reports FA_ERR_TIMEOUT and
 * the CUDA context stays usable. O and LSE are unspecified after a drop.
 * Exists only to test that the timeout path ends cleanly.
 */
fa_status_t fa_fwd_fault_test(const void* Q, const void* K, const void* V, void* O, float* LSE,
                              int B, int H, int N, int d, float scale,
                              int drop_load, unsigned long long timeout_ns, cudaStream_t stream);

/*
 * fa_bwd_fault_test -- TEST HOOK, not for production use. Same as fa_bwd, but
 * every device-side wait gives up after `timeout_ns` nanoseconds, and when
 * `drop_load` >= 0 the producer of every CTA skips one tile load: in a dQ
 * CTA the drop_load-th of K_0, V_0, K_1, V_1, ...; in a dK/dV CTA the Q and
 * dO tiles of query block drop_load. The waiting
 * role then gives up, every role stops, waits for its own copies and
 * tensor-core work in flight, frees its tensor memory and exits;
 * fa_get_device_status reports FA_ERR_TIMEOUT and the CUDA context stays
 * usable. dQ, dK, dV are unspecified after a drop.
 */
fa_status_t fa_bwd_fault_test(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                              const float* LSE, void* dQ, void* dK, void* dV,
                              int B, int H, int N, int d, float scale,
                              void* workspace, size_t workspace_bytes,
                              int drop_load, unsigned long long timeout_ns, cudaStream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* EXACT_IO_AWARE_34_FA_H_ */
