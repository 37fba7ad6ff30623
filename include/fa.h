/*
 * fa.h -- C ABI of the GB300 (sm_103a) online-softmax attention library.
 *
 * The operations, all from the pages on online softmax and FlashAttention:
 *
 *  - fa_fwd / fa_fwd_dt: exact dense attention forward O = softmax(scale * Q K^T) V,
 *    computed tile by tile with the online-softmax state (row max m, denominator l,
 *    alpha = exp(m - m_new) rescaling both l and the O accumulator), so that the
 *    N x N score matrix never reaches device memory.
 *    ("Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到 FlashAttention", §七,
 *    the per-Q-tile loop; the 1/sqrt(d) factor as in "为什么 Flash Attention 算出来的
 *    结果和标准注意力有微小差异？有损但值得", section "罪魁祸首是 online softmax 里那步
 *    rescale".)
 *
 *  - fa_bwd: the gradients of that forward, recomputing the scores from the kept LSE
 *    (same page, §7.2).
 *
 *  - online_softmax_rows: the per-row softmax state (m, l), m = max_t x_t,
 *    l = sum_t exp(x_t - m), reduced thread -> warp shuffle -> shared memory -> first
 *    warp with the merge rule m = max(m_a, m_b), l = l_a e^(m_a - m) + l_b e^(m_b - m).
 *    (Same page, §四, §4.1 and §4.2.)
 *
 * Conventions common to every call:
 *  - Every pointer passed to a compute call is a DEVICE pointer owned by the caller
 *    (fa_fwd_host takes its tensors in host memory and a device workspace). The
 *    library allocates no device memory: its device state is one status word per
 *    device and the 64 MiB scratch array of fa_fwd_splitkv_static, both in static
 *    device memory.
 *  - Calls are asynchronous on `stream` (0 = the legacy default stream). The return
 *    value reports argument errors (checked on the host, nothing is launched) and
 *    launch errors only. Errors the kernels detect while running (a bounded wait that
 *    ran out) are reported by fa_last_device_error().
 *  - Concurrent calls on different streams are allowed; the library keeps no
 *    per-call host state. The exception is fa_fwd_splitkv_static, whose calls share
 *    one scratch array (see there).
 */
#ifndef ONLINE_SOFTMAX_07_GB300_FA_H
#define ONLINE_SOFTMAX_07_GB300_FA_H

#include <stddef.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID = 1,      /* a null pointer, a negative size, len == 0 with rows > 0,
                              a non-finite or non-positive scale, causal not 0/1     */
  FA_ERR_UNSUPPORTED = 2,  /* head dimension or dtype outside what is built          */
  FA_ERR_ALIGN = 3,        /* a pointer without the alignment the call needs         */
  FA_ERR_CUDA = 4,         /* the CUDA runtime or driver returned an error           */
  FA_ERR_TIMEOUT = 5,      /* a kernel gave up a bounded wait (fa_last_device_error) */
  FA_ERR_TOO_LARGE = 6     /* fa_fwd_splitkv_static: the partials exceed its scratch  */
} fa_status;

typedef enum {
  FA_BF16 = 0,             /* q, k, v, o bf16; fp32 scores, softmax state and O accumulator */
  FA_F32 = 1,              /* q, k, v, o fp32; fp32 arithmetic on CUDA cores                */
  FA_F16 = 2               /* q, k, v, o fp16; as FA_BF16 with P and O rounded to fp16      */
} fa_dtype;

/*
 * Attention forward, bf16.
 *
 * q, k, v: device, contiguous [B, H, N, d] bf16 (row-major; one N x d matrix per
 *          head; K and V have the same N as Q). 16-byte aligned.
 * o:       device, contiguous [B, H, N, d] bf16, written. 16-byte aligned.
 * lse:     device fp32 [B, H, N], written with LSE_i = m_i + ln l_i = ln sum_j
 *          exp(scale q_i.k_j) over the visible keys j; NULL = not written. 4-byte aligned.
 * B, H, N: >= 0; any of them 0 is an empty problem (FA_OK, nothing launched).
 * d:       64 or 128 (else FA_ERR_UNSUPPORTED).
 * scale:   finite, > 0; multiplies the scores before the softmax (1/sqrt(d) usually).
 * causal:  0 = no mask; 1 = key j visible to query i iff j <= i.
 * Accuracy: scores, m, l and the O accumulator in fp32; P rounded to bf16 (round to
 * nearest even) for the P.V product; O rounded to bf16 at the end.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal,
                 cudaStream_t stream);

/*
 * Attention forward with an explicit element type. fa_fwd(...) is
 * fa_fwd_dt(..., FA_BF16, stream). With FA_F16, q, k, v and o are fp16 with the same
 * layout, alignment and d as for bf16 (the tensor-core path; P is rounded to fp16, whose
 * range holds it: P <= 2^8). With FA_F32, q, k, v and o are fp32 [B, H, N, d] (4-byte
 * aligned), d may be any value in 1..128, and all arithmetic is fp32 on CUDA cores (the
 * same online-softmax tile loop, 32 keys per tile).
 */
fa_status fa_fwd_dt(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int N, int d, float scale, int causal,
                    fa_dtype dtype, cudaStream_t stream);

/*
 * Attention forward with a chosen key block: the number of keys per K/V tile, i.e. per
 * step of the online-softmax tile loop ("Softmax 数值稳定性与 IO-Aware Attention" §七)
 * and so the number of (m, l) merges per row (N / block_n).  "Flash Attention 和标准
 * Attention 输出完全一样吗" suggests a larger block (128 -> 256) to reduce the merges;
 * "为什么 Flash Attention 算出来的结果和标准注意力有微小差异？有损但值得" ("罪魁祸首是
 * online softmax 里那步 rescale") says the error grows with their number.  This entry
 * exists for that study: same operation, arguments and results as fa_fwd_dt.
 *
 * block_n: 0 or 128 = fa_fwd_dt (the kernel the library otherwise runs; any dtype fa_fwd_dt
 *          takes); 64 (d = 64 or 128), 192 or 256 (d = 64): the same tcgen05 kernel built
 *          with 64-, 192- or 256-key tiles, FA_BF16 only.  Other values: FA_ERR_INVALID;
 *          192 or 256 with d = 128, or a 16-bit type other than bf16: FA_ERR_UNSUPPORTED.
 * Errors: as fa_fwd_dt.
 */
fa_status fa_fwd_block(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                       int block_n, cudaStream_t stream);

/*
 * Split-KV attention forward.  Same operation, arguments and results as fa_fwd_dt (bf16
 * or fp16, d in {64, 128}); each query block's K/V tiles are divided into num_splits
 * contiguous chunks processed by separate thread blocks, which raises the parallelism
 * when B * H * ceil(N / 256) is small next to the number of SMs.  Each chunk's result
 * (O normalised by its own denominator, and its LSE) goes to `workspace`; a second
 * kernel (launched as a programmatic dependent of the first on the same stream, so that
 * its blocks are placed while the first drains; it reads nothing before the first has
 * completed) merges them by bringing them to a common maximum, as the lihaoran.work
 * FlashAttention note ("为什么不能平均各块的softmax") and the merge rule of "Softmax
 * 数值稳定性与 IO-Aware Attention" §4.1 prescribe (partial results are not averaged).
 *
 * num_splits: 1..64 (1 = fa_fwd_dt; the workspace is then unused).
 * workspace:  device memory of at least fa_fwd_splitkv_workspace_bytes(...) bytes,
 *             16-byte aligned, owned by the caller; its contents need no initialisation
 *             and are overwritten.  Calls that share a workspace must not overlap.
 * Errors: as fa_fwd_dt, plus FA_ERR_INVALID for num_splits out of range, a NULL or too
 * small workspace (num_splits > 1), FA_ERR_ALIGN for a misaligned workspace.
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal, int num_splits,
                         void* workspace, size_t workspace_bytes, fa_dtype dtype,
                         cudaStream_t stream);

/* Workspace bytes fa_fwd_splitkv needs: num_splits * B * H * ceil(N/256)*256 * (d + 1) * 4
 * (0 for invalid arguments).  Host-only, no CUDA call. */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits);

/* A split count for fa_fwd_splitkv on a GPU with `sms` SMs.  Causal: the last query
 * block needs about 2 SMs / blocks times the average work per SM (blocks = B * H *
 * ceil(N/256)); the split count is that ratio rounded down after adding 0.2, so the
 * longest pieces no longer set the time.  Not causal: blocks are of equal length and a
 * split pays only while every piece still runs in the first wave, so SMs / blocks rounded
 * down.  Then at least two K/V tiles per split, at most 64; 1 when no split pays or for
 * invalid arguments (causal not 0 or 1, sms < 1).  Host-only, no CUDA call. */
int fa_fwd_splitkv_splits_for(int B, int H, int N, int causal, int sms);

/* fa_fwd_splitkv_splits_for with the current device's SM count (read from the runtime);
 * 1 when the device or its SM count cannot be queried. */
int fa_fwd_splitkv_default_splits(int B, int H, int N, int causal);

/*
 * Split-KV forward for callers that cannot allocate device memory (memory pools or arenas
 * that own all device memory, plugin interfaces without an allocator, paths where a
 * cudaMalloc would synchronise the device).  The pages have no counterpart: this is a
 * deployment convenience around fa_fwd_splitkv, same arguments and results minus the
 * workspace.
 *
 * The partials go to a scratch array in the library's static device memory: 64 MiB,
 * reserved on every GPU that loads the library until it is unloaded.  Problems needing
 * more (fa_fwd_splitkv_workspace_bytes > 64 MiB) return FA_ERR_TOO_LARGE and launch
 * nothing.  The call allocates nothing.  The first call on a device looks up the array's
 * device address (once per device, with that device current); make that first call before
 * any stream capture.  All calls share the array and it keeps the last call's partials;
 * nothing needs clearing (every partial read is written by the same call), but calls that
 * overlap on the GPU (other streams or host threads) race on it.
 */
fa_status fa_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o,
                                float* lse, int B, int H, int N, int d, float scale,
                                int causal, int num_splits, fa_dtype dtype,
                                cudaStream_t stream);

/*
 * Attention forward on host-resident tensors (the end-to-end path): q, k, v, o and lse
 * as in fa_fwd_dt but in host memory.  The B * H (batch, head) slabs are processed in
 * `chunks` consecutive groups; for each group the library copies Q, K, V in on an
 * internal copy stream, runs fa_fwd_dt on `stream`, and copies O (and LSE) out on a
 * second internal copy stream, so the copies of one group overlap the kernels of its
 * neighbours.  Up to three groups' device buffers are in use at a time, in `workspace`.
 *
 * q, k, v, o: host [B, H, N, d] (bf16/fp16: d in {64, 128}; fp32: any d <= 128);
 *             should be page-locked (cudaHostAlloc / cudaHostRegister): pageable memory
 *             gives the same results but the copies then do not overlap.
 * lse:        host fp32 [B, H, N], or NULL.
 * chunks:     >= 1 (more than B * H acts as B * H).
 * workspace:  device memory owned by the caller, at least
 *             fa_fwd_host_workspace_bytes(B, H, N, d, dtype, chunks) bytes, 256-byte
 *             aligned; its contents are overwritten.
 * Ordering: the copies in start after work enqueued on `stream` before the call, and
 * work enqueued on `stream` after the call starts after the last copy out; the call
 * returns once everything is enqueued (synchronise `stream` before reading o / lse).
 * Calls from several threads are enqueued one at a time.
 * Errors: as fa_fwd_dt; FA_ERR_INVALID for chunks < 1, a NULL or too small workspace;
 * FA_ERR_ALIGN for a misaligned workspace; FA_ERR_CUDA if a copy or an enqueue fails
 * (o and lse are then undefined).
 */
fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int N, int d, float scale, int causal, fa_dtype dtype, int chunks,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Device workspace bytes fa_fwd_host needs (0 for invalid arguments).  Host-only. */
size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d, fa_dtype dtype, int chunks);

/*
 * Row online-softmax state.
 *
 * x:      device fp32 [rows, len], contiguous row-major; any 4-byte alignment (a row
 *         may start at any float offset).
 * m_out:  device fp32 [rows], written with m_r = max_t x[r, t].
 * l_out:  device fp32 [rows], written with l_r = sum_t exp(x[r, t] - m_r).
 * rows:   >= 0 (0 = nothing to do, FA_OK). len: >= 1 when rows > 0.
 */
fa_status online_softmax_rows(const float* x, float* m_out, float* l_out,
                              int rows, int len, cudaStream_t stream);

/*
 * Row softmax: y[r, t] = exp(x[r, t] - m_r) / l_r with m_r, l_r as in
 * online_softmax_rows ("Softmax 数值稳定性与 IO-Aware Attention", §三: the third pass,
 * here fused with the (m, l) reduction).  One block per row (a warp per row up to 1024
 * floats) reads the row for (m, l), then again for y; the second read normally hits L2,
 * so device memory sees one read of x and one write of y.
 *
 * x:     device fp32 [rows, len], contiguous; any 4-byte alignment.
 * y:     device fp32 [rows, len], written; may alias x (in place); any 4-byte alignment.
 * m_out, l_out: device fp32 [rows], written with the row state, or NULL.
 * rows:  >= 0 (0 = nothing to do).  len: >= 1 when rows > 0.
 */
fa_status online_softmax_forward(const float* x, float* y, float* m_out, float* l_out,
                                 int rows, int len, cudaStream_t stream);

/*
 * Attention backward (bf16 or fp16 with d = 64 or 128 on the tensor cores; fp32 with any
 * d in 1..128 on CUDA cores): the gradients dQ, dK, dV of the
 * forward above for an upstream gradient dO.  "Softmax 数值稳定性与 IO-Aware Attention"
 * §7.2: only per-row statistics of the forward are kept (here LSE) and the scores are
 * recomputed tile by tile, never stored.  With P = exp(scale Q K^T - LSE):
 *   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D_i = sum_c dO_ic O_ic,
 *   dQ = scale dS K,  dK = scale dS^T Q
 * (the chain rule through the softmax; the pages print no gradient formula).
 *
 *   q, k, v, o, dout    [B, H, N, d], dtype; o and lse as fa_fwd wrote them for q, k, v
 *                       (same scale and causal)
 *   lse                 [B, H, N] fp32, required
 *   dq, dk, dv          [B, H, N, d], dtype, written (fp32 accumulation inside)
 *   workspace           caller-owned device scratch of at least
 *                       fa_bwd_workspace_bytes_dt(B, H, N, d, dtype) bytes (per query
 *                       row: fp32 statistics, or at d = 64 with bf16/fp16 their bf16
 *                       terms and the fp32 dQ accumulator); its contents are overwritten
 * Alignment: bf16/fp16: every pointer but lse 16 bytes, lse 4; fp32: 4 bytes, the
 * workspace 16.  B*H*N == 0 is a no-op (FA_OK).
 * Determinism: dK and dV elements are each written once by one block.  dQ likewise at
 * d = 128 and for fp32; at d = 64 (bf16/fp16) each key tile's block adds its share of dQ
 * into the fp32 accumulator (TMA reduce-adds), in an order that varies from run to run,
 * so dQ may differ in its last bits between runs.  Stream order: the call is ordered on
 * `stream` like a single launch.  At d = 128 (bf16/fp16) the dQ pass runs on an internal
 * stream of the library that forks from `stream` after the statistics pass and joins it
 * after the dQ pass, so that it can overlap the dK/dV pass (stream capture sees the fork
 * and the join); at d = 64 every launch is on `stream`.  Enqueueing is serialised across
 * host threads.  Errors: FA_ERR_INVALID (null pointer, lse missing, negative size,
 * scale not finite and > 0, causal not 0/1, workspace too small), FA_ERR_UNSUPPORTED
 * (d or dtype), FA_ERR_ALIGN, FA_ERR_CUDA.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, void* workspace, size_t workspace_bytes,
                 fa_dtype dtype, cudaStream_t stream);

/* Workspace fa_bwd needs for this head dimension and dtype, in bytes, with
 * n_pad = ceil(N / 128) * 128: bf16/fp16 at d = 64: 288 * B * H * n_pad (16 bf16 row
 * statistics terms and a 64-float dQ accumulator row per padded query row); bf16/fp16 at
 * d = 128: 40 * B * H * n_pad (two fp32 statistics and the 16 bf16 terms per row); fp32
 * (1 <= d <= 128): 8 * B * H * n_pad.  0 for negative sizes, for a d or
 * dtype fa_bwd does not support, and for problems of more than INT_MAX 128-row tiles. */
size_t fa_bwd_workspace_bytes_dt(int B, int H, int N, int d, fa_dtype dtype);

/* A workspace size that serves every d and dtype of fa_bwd: the largest value of
 * fa_bwd_workspace_bytes_dt, 288 * B * H * n_pad (0 for negative sizes). */
size_t fa_bwd_workspace_bytes(int B, int H, int N);

/* Static, never-NULL description of a status code. */
const char* fa_status_str(fa_status status);

/*
 * Synchronises `stream`, then reads and clears the current device's status word.
 * Returns FA_ERR_TIMEOUT if a kernel launched since the last call gave up a bounded
 * wait (it then skipped the rest of its work, so its outputs are not valid),
 * FA_ERR_CUDA if the synchronisation failed, else FA_OK.
 */
fa_status fa_last_device_error(cudaStream_t stream);

/*
 * Self-test of the bounded-wait path: launches one block that waits on a
 * shared-memory barrier nothing ever completes, with a time limit of `limit_ns`
 * nanoseconds (1..2e9). The wait runs out, the kernel records the timeout in the
 * status word and returns, leaving the context usable; fa_last_device_error() then
 * returns FA_ERR_TIMEOUT. Not part of the method; it exists so that tests can check
 * the timeout path without faulting or hanging the GPU.
 */
fa_status fa_selftest_wait_timeout(long long limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ONLINE_SOFTMAX_07_GB300_FA_H */
