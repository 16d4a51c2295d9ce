// na_internal.h -- structures shared by the host API and the kernels of libna (not installed).
//
// Problems of 1, 2 or 3 spatial axes are embedded as 3 axes, outermost first, with leading
// axes of length 1, kernel 1 and dilation 1.  All tile geometry is in *class coordinates*: along
// an axis with dilation d, residue class c holds the positions c, c+d, c+2d, ... and a tile or
// halo is a run of consecutive class indices.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace na {

// Division of 32-bit unsigned values by a divisor fixed for a launch, by multiplication (Granlund
// and Montgomery, "Division by invariant integers using multiplication", 1994): with s = ceil(log2 d)
// and m = floor(2^32 (2^s - d) / d) + 1, n / d = (t + ((n - t) >> 1)) >> (s - 1) where
// t = umulhi(m, n), exact for every 32-bit n; d = 1 is a copy.  A hardware-free division by a
// runtime divisor costs a thread ~74 cycles on this GPU, this ~10.
struct FastDiv {
    uint32_t d, m, s;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f{d, 0u, 0u};
    if (d <= 1) return f;
    uint32_t s = 0;
    while ((1ull << s) < d) ++s;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << s) - d)) / d + 1ull);
    f.s = s;
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
    if (f.d <= 1u) return n;
    const uint32_t t = __umulhi(f.m, n);
    return (t + ((n - t) >> 1)) >> (f.s - 1u);
}

struct Geom {
    int B, heads, D;
    int L[3], k[3], d[3];
};

// Static tile plan of one tensor-core kernel for one problem.
struct TilePlan {
    int T[3];        // tile extents (class coordinates), T0*T1*T2 == 128, powers of two
    int H[3];        // halo box extents: keys (fwd, dQ) or queries (dK/dV) a tile may need;
                     // H[a] == nchk[a] * G[a] along every axis
    int G[3];        // chunk box extents; G[a] <= 32 along masked axes; NC multiple of 16
    int NC;          // rows of one chunk = G0*G1*G2 (multiple of 16, <= 112)
    int nchk[3];     // chunks along each axis that cover the halo box
    int ntile[3];    // tiles per axis and residue class: ceil(ceil(L/d) / T)
    int tmem_cols;   // TMEM columns allocated per CTA (power of two)
    int sbufs;       // score buffers in TMEM: 2, or 3 (the forward at D <= 32 with NC <= 64)
    int per_sm;      // persistent CTAs per SM (the grid is per_sm x SM count, at most `ctas`)
    int smem_bytes;  // dynamic shared memory per CTA (includes alignment slack)
    int64_t ctas;    // tiles (linearised: head fastest, then tile along axes 2,1,0, class 2,1,0, batch)
};

// Kernel parameters of the tensor-core kernels (passed as __grid_constant__).
// Tensor-map roles per kernel:
//   fwd : tm[0] q tile, tm[1] k chunk, tm[2] v chunk
//   dq  : tm[0] q tile, tm[1] dO tile, tm[2] k chunk, tm[3] v chunk
//   dkdv: tm[0] k tile, tm[1] v tile, tm[2] q chunk, tm[3] dO chunk
// Outputs are written with plain 16-byte stores, one row per thread.
struct TcParams {
    CUtensorMap tm[4];
    TilePlan plan;
    int L[3], k[3], d[3];
    int B, heads, D;
    float scale;        // softmax scale (applied to q.k)
    float scale_log2;   // max(|scale|, tiny) * log2(e); a negative scale negates A of the S product
    uint32_t neg;       // 1 when scale < 0
    uint32_t rad[8];    // mixed radix of the tile index: heads, ntile2, ntile1, ntile0, d2, d1, d0, B
    uint32_t step[8];   // the grid size written in that radix (persistent CTAs step by it)
    uint16_t* out0;     // fwd: O; dQ: dQ; dK/dV: dK  ([B, L.., heads, D], 2-byte elements)
    uint16_t* out1;     // dK/dV: dV
    uint32_t f16;       // element type of every tensor of D channels: 0 bf16, 1 fp16
    float* lse_out;     // fwd: [B, L.., heads] natural-log LSE
    const float* lse;   // bwd: forward LSE
    const float* delta; // bwd: Delta = <dO, O>
    unsigned* err;      // device status word
    unsigned long long wait_ns;  // time limit of one bounded wait (kWaitLimitNs unless a test lowers it)
    uint32_t withhold;  // test hook: 1 = CTA 0 never fills its first halo chunk, so a wait runs out
    // Per-tile decode without integer division (a 32-bit division by a runtime value costs the
    // softmax warps hundreds of cycles at every tile boundary):
    int Lc_tab[3][8];   // class length ceil((L - c) / d) per axis and residue class c < d (d <= 8)
    uint32_t rcpG[3];   // floor(2^32 / G[a]) + 1 (0 for G[a] == 1): umulhi(x, rcpG[a]) == x / G[a] for x < 2^26
};

// Parameters of the CUDA-core kernels (fp32 path and the Delta prologue).
struct FmaParams {
    const void* q;
    const void* key;
    const void* value;
    const void* o;
    const void* dO;
    const float* lse;
    const float* delta;
    void* out0;         // fwd: o      dq: dQ   dkdv: dK   delta: delta (float*)
    void* out1;         // fwd: lse    dkdv: dV
    int L[3], k[3], d[3];
    int B, heads, D;
    int64_t N;          // tokens per batch entry
    float scale;
    // 32-bit row decode without division (used when B * N * heads < 2^32)
    uint32_t rows32;
    FastDiv fd_heads, fd_N, fd_L[3], fd_d[3];
    // query quads (four consecutive class positions along the innermost axis, one head): quads per
    // class (of the longest class) and their total, B * L0 * L1 * d2 * qc2 * heads
    int qc2;
    FastDiv fd_qc2;
    long long quads;
};

// Parameters of the unfused operations (na_unfused.cu).  Rows are (batch, token, head) triples;
// K = k0 k1 k2 attention weights per row.
struct UnfParams {
    const void* a;      // qk: q      av: attn   gather: dattn  scatter: dattn/attn  dattn: dO  softmax: x / y
    const void* b;      // qk: k      av: v      gather: k      scatter: q / dO      dattn: v   softmax bwd: dy
    void* out0;         // qk: attn   av: o      gather: dq     scatter: dk / dv     dattn: dattn  softmax: y / dx
    int L[3], k[3], d[3];
    int heads, D, K;
    long long rows;     // B * tokens * heads
    float scale;        // qk: scale; gather, scatter: the factor of the sum (scale, or 1)
    const float* rpb;   // qk: relative positional bias [heads, 2k0-1, 2k1-1, 2k2-1], or null
    const int* vk;      // mask: per-position kernel sizes, concatenated over the axes
    int vk_off[3];      // mask: offset of each (embedded) axis in vk, -1 for an axis without one
    int strips2;        // tensor-core logits: strips of 16 class positions along the innermost axis, summed over classes
    long long units;    // tensor-core kernels: strips of all lines, heads and batch entries (B L0 L1 strips2 heads)
    // 32-bit decodes without division (rows and units < 2^32)
    uint32_t small;
    FastDiv fd_heads, fd_strips2, fd_L[3], fd_d[3], fd_K, fd_k2, fd_k12;
    // Inverse-window gathers fed by TMA (tma = 1): per query line, the span's source rows (tm_src: the
    // [B, L.., heads * D] tensor, srows span positions) and each span query's window weights on that line
    // (tm_w: the [B, L.., heads * K] weights, a box of wb >= k2 + 7 offsets from an aligned start).
    CUtensorMap tm_src, tm_w;
    uint32_t tma, wb;
    uint32_t srows;             // span rows copied per line: the largest span of any strip, rounded up to 16
    uint32_t wrows;             // weight rows copied per line: srows (inverse-window gather) or 16 (weighted sum)
    unsigned* err;              // device status word (bounded waits)
    unsigned long long wait_ns; // time limit of one wait
};

// Tokens per block of the bias-gradient reduction's first stage, and the size of its partial sums.
int rpb_grad_tokens_per_block(int K);
size_t rpb_grad_workspace_bytes(long long tokens, int heads, int K, int table);

// Launchers (defined next to their kernels).  Return a cudaError_t as int.
int launch_fwd_tc(const TcParams& p, cudaStream_t stream);
int launch_fwd_tc_f16(const TcParams& p, cudaStream_t stream);
int launch_fwd_tc_sb3(const TcParams& p, cudaStream_t stream);   // three score buffers, D <= 32
int launch_dq_tc_f16(const TcParams& p, cudaStream_t stream);
int launch_dkdv_tc_f16(const TcParams& p, cudaStream_t stream);
int launch_dq_tc(const TcParams& p, cudaStream_t stream);
int launch_dkdv_tc(const TcParams& p, cudaStream_t stream);
int launch_fwd_fma(const FmaParams& p, cudaStream_t stream);
int launch_dq_fma(const FmaParams& p, cudaStream_t stream);
int launch_dkdv_fma(const FmaParams& p, cudaStream_t stream);
int launch_delta(const FmaParams& p, int elem, cudaStream_t stream);  // elem: 0 bf16, 1 fp32, 2 fp16
// elem: 0 bf16, 1 fp32, 2 fp16
int launch_unfused_qk(const UnfParams& p, int elem, cudaStream_t stream);
int launch_unfused_av(const UnfParams& p, int elem, cudaStream_t stream);
int launch_unfused_gather(const UnfParams& p, int elem, cudaStream_t stream);
int launch_unfused_scatter(const UnfParams& p, int elem, cudaStream_t stream);
int launch_unfused_dattn(const UnfParams& p, int elem, cudaStream_t stream);
// drpb[h, r] = sum over (batch, query, offset) at relative position r of dattn (two stages through
// `partial`, which holds rpb_grad_workspace_bytes).
int launch_unfused_rpb_grad(const UnfParams& p, int elem, long long tokens, float* partial, float* drpb,
                            cudaStream_t s);
// attn[row, t] = -inf for every offset t outside the row's variable window (p.vk).
int launch_unfused_mask_window(const UnfParams& p, int elem, cudaStream_t s);
int launch_unfused_softmax(const UnfParams& p, int elem, bool bwd, cudaStream_t stream);

// Kernel attributes that depend on the plan (dynamic smem opt-in); called before the launch.
int prepare_tc_kernel(int which, int D, int smem_bytes);

}  // namespace na
