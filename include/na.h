/*
 * na.h -- C ABI of libna: multi-dimensional neighborhood attention (NA), forward and backward,
 * on one NVIDIA GB300 (sm_103a).
 *
 * What is computed.  NATTEN issue #161, "Backward pass is very slow towards much tokens and large
 * kernels" (the user's benchmark script: na2d/na3d(query, key, value, kernel_size) and the unfused
 * na*_qk -> softmax -> na*_av chain with a dilation argument) is the source of the operation; it
 * never writes the window down, so this library fixes the plainest reading:
 *   per spatial axis of length L, odd kernel size k (r = k/2) and dilation d, query index i is in
 *   residue class c = i mod d at class index j = i div d; the class has Lc = ceil((L-c)/d) positions;
 *   the window starts at class index s = clamp(j - r, 0, Lc - k) -- shifted, never truncated, at the
 *   borders -- and holds the k positions c + d*(s+t), t = 0..k-1.  A query's neighbourhood is the
 *   Cartesian product of its per-axis windows (every query sees exactly prod(k) keys).
 *   O_i = sum_j softmax_j(scale * <q_i, k_j>) v_j over that neighbourhood;
 *   LSE_i = natural-log logsumexp of the scaled logits.
 * The backward follows the maintainer's fused-kernel profile in the same issue: a ComputeDelta
 * prologue Delta_i = <dO_i, O_i>, then dQ, dK and dV from the recomputed probabilities.
 *
 * Tensor layout (all entry points).  q, k, v, o, dO, dQ, dK, dV are contiguous
 * [B, L_1, ..., L_ndim, heads, D] arrays of one element type (the layout of NATTEN's fused ops,
 * [b, (t,) h, w, heads, dim] in the user's script); lse and delta are contiguous fp32
 * [B, L_1, ..., L_ndim, heads].  Every pointer is a DEVICE pointer owned by the caller; the
 * library keeps none of them after a call returns.  All work is enqueued on `stream` (a
 * cudaStream_t passed as void*; NULL is the legacy default stream) and the calls return without
 * waiting for it.
 *
 * Errors.  Arguments are validated before anything is enqueued; on a validation error nothing is
 * written and no work is enqueued.  No entry point aborts, prints or traps.  Device-side waits
 * are bounded: a wait that runs out records NA_ERR_TIMEOUT in a per-device status word that
 * na_device_status() reports.
 */
#ifndef NA_H_
#define NA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NA_BF16 = 0, /* bfloat16 tensors; tcgen05 tensor-core kernels, fp32 accumulation */
    NA_FP32 = 1, /* float32 tensors; CUDA-core FMA kernels, fp32 throughout */
    NA_FP16 = 2  /* float16 tensors; the same tensor-core kernels as NA_BF16 with fp16 operands (P and
                    dS are rounded to fp16), fp32 accumulation.  The kernels mask keys outside a
                    window with a -65504 bias, so |scale * q.k| must stay below 3.2e4. */
} na_dtype;

typedef enum {
    NA_OK = 0,
    NA_ERR_INVALID_ARG = 1, /* bad sizes, kernel, dilation, scale or a null pointer */
    NA_ERR_UNSUPPORTED = 2, /* valid NA problem outside what the kernels implement (see below) */
    NA_ERR_ALIGNMENT = 3,   /* a tensor pointer is not 16-byte aligned */
    NA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed */
    NA_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (reported by na_device_status) */
    NA_ERR_WORKSPACE = 6    /* workspace too small, or it could not be allocated */
} na_status;

/*
 * Forward.  Writes o (same type as q) and lse (fp32, natural log).
 *   B >= 1; 1 <= ndim <= 3; spatial[a] >= 1; heads >= 1;
 *   kernel[a] odd and >= 1; dilation[a] >= 1; spatial[a] / dilation[a] >= kernel[a]
 *   (every residue class holds at least k positions); scale finite (the workloads use D^-0.5).
 *   Every tensor pointer 16-byte aligned.
 * Supported (else NA_ERR_UNSUPPORTED):
 *   NA_BF16, NA_FP16: D in {16, 32, 64, 128}; dilation[a] <= 8 (the tensor-core kernels load a dilated
 *   tile as one TMA box whose element stride is the dilation, and a TMA element stride is at most
 *   8); a tile plan must exist whose boxes span at most
 *   256 elements per axis (class positions times the dilation).
 *   NA_FP32: D in {16, 32, 64, 128}.
 */
na_status na_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int ndim, const int* spatial, int heads, int D,
                 const int* kernel, const int* dilation, float scale,
                 na_dtype dtype, void* stream);

/* Bytes of workspace na_bwd needs (the fp32 Delta array, B * prod(spatial) * heads * 4, rounded
   up to 256).  Returns 0 for invalid sizes. */
size_t na_bwd_workspace_size(int B, int ndim, const int* spatial, int heads);

/*
 * Backward = na_bwd_delta + na_bwd_dq + na_bwd_dkdv.  Reads q, k, v, o, dO and the forward's lse;
 * writes dQ, dK, dV (same type as q).  Each output element is written exactly once (no atomics),
 * so the result is bitwise deterministic.
 *   workspace: device memory of at least na_bwd_workspace_size() bytes, or NULL, in which case
 *   the call allocates it with cudaMallocAsync and frees it with cudaFreeAsync on `stream`.
 * Argument rules and support are those of na_fwd.
 */
na_status na_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dQ, void* dK, void* dV,
                 int B, int ndim, const int* spatial, int heads, int D,
                 const int* kernel, const int* dilation, float scale, na_dtype dtype,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward without any allocation.  The source pages have no counterpart for this entry point; it
 * exists for callers that cannot allocate device memory while they run: a host framework that has
 * handed out all device memory up front under a fixed budget, or a latency-critical loop where an
 * allocation may block, fail under memory pressure, or is simply forbidden by the caller's rules.
 * Such callers cannot pass workspace = NULL to na_bwd (that allocates with cudaMallocAsync), and
 * may have no spare buffer of na_bwd_workspace_size() bytes to lend either.
 *
 * It computes exactly what na_bwd computes, with the same arguments minus the workspace, and calls
 * no cudaMalloc, cudaFree or other allocating routine.  The Delta scratch is a fixed array of
 * NA_NOALLOC_MAX_ROWS floats (32 MiB) that the library reserves in device memory on every GPU
 * where it is loaded, for the life of the process.
 *   - Limit: B * prod(spatial) * heads must be <= NA_NOALLOC_MAX_ROWS; larger problems return
 *     NA_ERR_WORKSPACE before anything is enqueued (use na_bwd for them).
 *   - Set-up: the first call on each device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current).  Make that first call before any stream
 *     capture on the device.
 *   - Sharing: every call on a device uses the same array, which keeps the last call's contents.
 *     Each call overwrites every row it reads before reading it, so nothing needs clearing, but
 *     two calls whose work overlaps on the GPU (e.g. on different streams) race on the array:
 *     order them on one stream or with events.
 */
#define NA_NOALLOC_MAX_ROWS (8 * 1024 * 1024)
na_status na_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dQ, void* dK, void* dV,
                         int B, int ndim, const int* spatial, int heads, int D,
                         const int* kernel, const int* dilation, float scale, na_dtype dtype,
                         void* stream);

/*
 * Backward step 1 (the maintainer's "ComputeDelta"): delta[row] = sum_c dO[row, c] * o[row, c]
 * for every (batch, token, head) row, in fp32.  delta: fp32 [B, L.., heads].
 */
na_status na_bwd_delta(const void* o, const void* dO, float* delta,
                       int B, int ndim, const int* spatial, int heads, int D,
                       na_dtype dtype, void* stream);

/*
 * Backward step 2: dQ_i = scale * sum_{j in N(i)} P_ij (<dO_i, v_j> - delta_i) k_j, with
 * P_ij = exp(scale <q_i, k_j> - lse_i).  One pass over query tiles; writes every dQ row once.
 */
na_status na_bwd_dq(const void* q, const void* k, const void* v, const void* dO,
                    const float* lse, const float* delta, void* dQ,
                    int B, int ndim, const int* spatial, int heads, int D,
                    const int* kernel, const int* dilation, float scale,
                    na_dtype dtype, void* stream);

/*
 * Backward step 3: dV_j = sum_{i : j in N(i)} P_ij dO_i and
 * dK_j = scale * sum_{i : j in N(i)} P_ij (<dO_i, v_j> - delta_i) q_i.  One pass over key tiles,
 * each walking the queries whose windows hold its keys (the inverse neighbourhood); every dK/dV
 * row is written once, with no atomics.
 */
na_status na_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO,
                      const float* lse, const float* delta, void* dK, void* dV,
                      int B, int ndim, const int* spatial, int heads, int D,
                      const int* kernel, const int* dilation, float scale,
                      na_dtype dtype, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status word.  Returns
 * NA_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last call, NA_ERR_CUDA if the
 * stream reports an error, else NA_OK.  If raw is non-NULL it receives the raw status word
 * (0x5000 | wait site) for diagnostics.
 */
na_status na_device_status(void* stream, uint32_t* raw);
/* The library looks up, once per device, the device addresses of its file-scope arrays (this status
 * word and na_bwd_noalloc's scratch) and keeps them for the life of the process.  A cudaDeviceReset,
 * or anything else that destroys and recreates the device's primary context, invalidates those
 * addresses: do not call the library on a device after resetting it. */

/*
 * Test hook for the bounded device-side waits (the pages have no counterpart; it exists so that the
 * timeout path can be exercised without faulting a GPU).  For every later launch of the tensor-core
 * kernels (NA_BF16, NA_FP16) in this process it sets the time limit of one wait to limit_ns
 * (100 us .. 10 s; 0 restores the 2 s default) and, with withhold = 1, makes the first CTA skip the
 * copy of its first halo chunk, so that the waits on that chunk run out.  Such a call leaves its
 * outputs incomplete and na_device_status() then reports NA_ERR_TIMEOUT; the kernels stop issuing
 * work, let the copies already issued land, free their tensor memory and return.  Call it again with
 * (0, 0) to restore normal launches.  Process-wide; for tests only.
 * Errors: NA_ERR_INVALID_ARG for a limit outside the range or withhold not 0 or 1.
 */
na_status na_debug_wait_hook(unsigned long long limit_ns, int withhold);

/* Static description of a status code. */
const char* na_strerror(na_status status);

/*
 * Tile plan the tensor-core kernels (bf16 and fp16) would use for this problem, for benchmarking
 * and roofline accounting.  which: 0 = forward, 1 = dQ, 2 = dK/dV.  out[16] receives
 *   {T1, T2, T3, H1, H2, H3, G1, G2, G3, NC, chunks_per_tile_max, ctas, mma_flops,
 *    tmem_cols, smem_bytes, chunks_total}
 * (axes embedded as 3D, outermost first; mma_flops = the attention products' FLOPs that all
 * tiles issue, without the window-bias products; ctas = persistent grid size;
 * chunks_total = chunks over all tiles).
 */
na_status na_plan_info(int which, int B, int ndim, const int* spatial, int heads, int D,
                       const int* kernel, const int* dilation, int64_t* out);


/*
 * Unfused operations.  NATTEN issue #161 ("Backward pass is very slow towards much tokens and large
 * kernels") times the chain na2d_qk -> softmax -> na2d_av beside the fused op, and the maintainer's
 * profile there lists its kernels (attention logits, AV, their gradients QGRAD, KGRAD, AGRAD, VGRAD,
 * softmax forward and backward).  These entry points compute that chain: the bf16 and fp16 products
 * on warp-level tensor-core MMAs, the fp32 products and the softmax on CUDA cores.
 *
 * Attention weights attn: [B, L.., heads, K] in the dtype of q, K = kernel[0] * ... * kernel[ndim-1];
 * the weight of window offset (t_0, .., t_{n-1}) (t_a < kernel[a], first axis outermost) sits at
 * t = (t_0 * kernel[1] + t_1) * kernel[2] + ... and belongs to the key at position
 * c + dilation[a] * (s_a + t_a) along each axis (c, s_a: the query's residue class and window start).
 * Tensors of D channels: [B, L.., heads, D] as for na_fwd.  Every pointer caller-owned device
 * memory, 16-byte aligned; arithmetic in fp32.  Supported: NA_FP32, NA_BF16, NA_FP16 with
 * D in {16, 32, 64, 128} (else NA_ERR_UNSUPPORTED); sizes are validated as for na_fwd.
 */

/* attn = scale * q . k over each query's window (the logits), plus, when rpb is not null, the relative
 * positional bias of each pair.  The maintainer's profile in the same issue names the logits kernel
 * QKRPB.  rpb: fp32 [heads, 2 k_0 - 1, .., 2 k_{n-1} - 1], caller-owned device memory, 4-byte aligned;
 * the pair (query i, its window offset t) reads rpb[h, (c(key)_a - c(i)_a + k_a - 1)_a], c(.)_a the
 * position's class index along axis a (its index divided by dilation[a]). */
na_status na_qk(const void* q, const void* k, const float* rpb, void* attn, int B, int ndim, const int* spatial,
                int heads, int D, const int* kernel, const int* dilation, float scale, na_dtype dtype, void* stream);

/* o = sum over each query's window of attn * v. */
na_status na_av(const void* attn, const void* v, void* o, int B, int ndim, const int* spatial, int heads, int D,
                const int* kernel, const int* dilation, na_dtype dtype, void* stream);

/* y = softmax(x) over the K weights of every (batch, token, head) row; y may be x. */
na_status na_softmax(const void* x, void* y, int B, int ndim, const int* spatial, int heads, const int* kernel,
                     na_dtype dtype, void* stream);

/* dx = y * (dy - sum_t y dy), the softmax's gradient given its output y; dx may be dy. */
na_status na_softmax_bwd(const void* y, const void* dy, void* dx, int B, int ndim, const int* spatial, int heads,
                         const int* kernel, na_dtype dtype, void* stream);

/* Gradients of na_qk given dattn (the logits' gradient): dq = scale * sum_t dattn k over the query's
 * window; dk = scale * sum over the queries whose windows hold the key of dattn q (no atomics). */
na_status na_qk_bwd(const void* dattn, const void* q, const void* k, void* dq, void* dk, int B, int ndim,
                    const int* spatial, int heads, int D, const int* kernel, const int* dilation, float scale,
                    na_dtype dtype, void* stream);

/* Gradients of na_av given dO: dattn = dO . v over the query's window; dv = sum over the queries
 * whose windows hold the key of attn dO (no atomics). */
na_status na_av_bwd(const void* dO, const void* attn, const void* v, void* dattn, void* dv, int B, int ndim,
                    const int* spatial, int heads, int D, const int* kernel, const int* dilation, na_dtype dtype,
                    void* stream);

/* Variable windows.  The user in the same issue asks for kernel sizes that change along time; the
 * maintainer advises masking the unfused logits, which the user already does to na3d_qk's output.
 * This sets attn[row, t] = -inf, in place, for every window offset t outside the query's own window:
 * along each axis a, the window of size k_a(x_a) that the same shifted-window rule gives (nested in
 * the full window of size kernel[a]).  sizes: device int32, caller-owned, 4-byte aligned, the per-
 * position sizes of axis 0 (spatial[0] entries), then of axis 1, ...; each entry is clamped to
 * [1, kernel[a]] and an even entry is lowered by one.  Offsets inside every row's window are not
 * touched, and nothing else is read.  The softmax, the weighted sum and every gradient then treat the
 * masked weights as absent (their probability and gradient are zero). */
na_status na_mask_window(void* attn, const int* sizes, int B, int ndim, const int* spatial, int heads,
                         const int* kernel, const int* dilation, na_dtype dtype, void* stream);

/* Bytes of device workspace na_rpb_grad needs for this problem (0 on invalid arguments). */
size_t na_rpb_grad_workspace_size(int B, int ndim, const int* spatial, int heads, const int* kernel);

/* Gradient of na_qk's bias table given the logits' gradient dattn [B, L.., heads, K] (dtype):
 * drpb[h, r] = sum over batch, queries and window offsets at relative position r of dattn.
 * drpb: fp32 [heads, 2 k_0 - 1, ..], overwritten.  Two stages through the workspace (per block of
 * tokens, then over blocks in a fixed order): deterministic, no atomics.  With workspace null the
 * library allocates it on the stream (cudaMallocAsync) and frees it after use; otherwise it needs
 * na_rpb_grad_workspace_size bytes (NA_ERR_WORKSPACE if fewer), 16-byte aligned.  Every head's table
 * is reduced in one block's shared memory: heads * prod(2 k_a - 1) * 4 bytes must stay within about
 * 224 KB (8 heads of a 9x9x9 window fit, of an 11x11x11 window not), else NA_ERR_UNSUPPORTED. */
na_status na_rpb_grad(const void* dattn, float* drpb, int B, int ndim, const int* spatial, int heads,
                      const int* kernel, const int* dilation, na_dtype dtype, void* workspace, size_t workspace_bytes,
                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NA_H_ */
