// na_fma.cu -- CUDA-core kernels of libna: the fp32 path (forward, dQ, dK/dV; fp32 FMA, no TF32)
// and the Delta prologue shared by both paths.
//
// Neighbourhood as read from NATTEN issue #161 ("Backward pass is very slow towards much tokens and
// large kernels"): per axis, a window of k positions of the query's residue class (dilation d),
// starting at class index clamp(j - k/2, 0, Lc - k); the Cartesian product over axes.  The
// maintainer's remark in that thread that fp32 attention is limited by memory rather than by
// arithmetic, since the fp32 compute peak is low, is why this path lets L1/L2 absorb the window
// overlap instead of tiling through shared memory.
//
// Lane layout: a row of D fp32 values is D/4 chunks of 16 bytes, and each row gets D/4
// consecutive lanes, one per chunk.  Neighbouring rows (heads, then tokens) sit next to each other
// in memory, so every row load of a warp is coalesced.  Dot products over D are a lane's chunk plus
// a butterfly over the row's lanes (shuffles restricted to those lanes, so rows whose loops differ
// in length never wait on each other).
#include <cmath>

#include <cuda_fp16.h>

#include "na_device.cuh"
#include "na_internal.h"

namespace na {
using namespace dev;

namespace {

constexpr int kFmaThreads = 256;

struct RowIdx {
    long long b, tok;  // batch, spatial token index
    int h;
    int x[3];          // spatial coordinates (embedded 3D)
};

__device__ __forceinline__ RowIdx decode_row(const FmaParams& p, long long row) {
    RowIdx r;
    r.h = static_cast<int>(row % p.heads);
    long long bt = row / p.heads;
    r.b = bt / p.N;
    r.tok = bt % p.N;
    long long t = r.tok;
    for (int a = 2; a >= 0; --a) {
        r.x[a] = static_cast<int>(t % p.L[a]);
        t /= p.L[a];
    }
    return r;
}

// First neighbour (spatial index) of spatial index i along axis a.
__device__ __forceinline__ int first_nb(const FmaParams& p, int a, int i) {
    const int d = p.d[a], c = i % d, j = i / d;
    return c + d * win_start(j, class_len(p.L[a], d, c), p.k[a]);
}

// The lanes of one row: CPH = D / 4 lanes per row, 32 / CPH rows per warp.  Lanes past the last
// row repeat it and store nothing.  UNIFORM: every row of the warp runs the same loop (forward, dQ),
// so the butterflies may name the whole warp; otherwise they name only the row's lanes.
template <int D, bool UNIFORM>
struct RowLanes {
    static constexpr int CPH = D / 4;
    static constexpr int RPW = 32 / CPH;
    int c, rl;
    unsigned mask;     // the lanes that take part in a butterfly
    long long row;
    bool store;

    __device__ bool init(long long rows) {
        const int lane = threadIdx.x & 31;
        c = lane % CPH;
        rl = lane / CPH;
        mask = (UNIFORM || CPH == 32) ? 0xffffffffu : ((1u << CPH) - 1u) << (rl * CPH);
        const long long row0 = (static_cast<long long>(blockIdx.x) * kFmaThreads + (threadIdx.x & ~31)) / CPH;
        if (row0 >= rows) return false;   // the whole warp
        row = row0 + rl;
        store = row < rows;
        if (!store) row = rows - 1;
        return true;
    }
    // sum over the row's lanes
    __device__ float sum(float v) const {
#pragma unroll
        for (int m = CPH / 2; m >= 1; m >>= 1) v += __shfl_xor_sync(mask, v, m);
        return v;
    }
};

constexpr float kLog2e = 1.4426950408889634f;   // log2(e)
constexpr float kLn2 = 0.6931471805599453f;     // ln(2)

__device__ __forceinline__ float dot4(const float4& a, const float4& b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

__device__ __forceinline__ void axpy4(float4& acc, float s, const float4& x) {
    acc.x = fmaf(s, x.x, acc.x);
    acc.y = fmaf(s, x.y, acc.y);
    acc.z = fmaf(s, x.z, acc.z);
    acc.w = fmaf(s, x.w, acc.w);
}

__device__ __forceinline__ void scale4(float4& acc, float s) {
    acc.x *= s;
    acc.y *= s;
    acc.z *= s;
    acc.w *= s;
}

// The lane's chunk of a row (row-major [rows, D] fp32): a float4 pointer.
__device__ __forceinline__ const float4* chunk_ptr(const void* base, long long row, int D, int c) {
    return reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * D) + c;
}

// A row's window: the first key's row index along each line (t0, t1); keys of a line are `step` rows apart.
struct FmaWindow {
    int f[3];
    long long b;
    int h;
    __device__ void start(const FmaParams& p, const RowIdx& r) {
        b = r.b;
        h = r.h;
        for (int a = 0; a < 3; ++a) f[a] = first_nb(p, a, r.x[a]);
    }
    __device__ long long line_row(const FmaParams& p, int t0, int t1) const {
        const long long tok = ((b * p.L[0] + f[0] + p.d[0] * t0) * p.L[1] + f[1] + p.d[1] * t1) * p.L[2] + f[2];
        return tok * p.heads + h;
    }
};

// Keys per group: their loads issue together (and the forward rescales once per group).  Larger
// groups keep more loads in flight per warp but cost registers, hence resident warps; measured at
// 1024x1024 9x9 fp32, one key per group suits the forward and two the backward kernels.
constexpr int kGF = 1;
constexpr int kGB = 2;

// Forward: online softmax over the window in log2 units (the scale carries log2 e), one rescale
// per group of keys; LSE is stored in natural-log units.
template <int D>
__global__ void __launch_bounds__(kFmaThreads) fwd_fma_kernel(const FmaParams p) {
    const long long rows = static_cast<long long>(p.B) * p.N * p.heads;
    RowLanes<D, true> ln;
    if (!ln.init(rows)) return;
    const float4 qc = __ldg(chunk_ptr(p.q, ln.row, D, ln.c));
    FmaWindow win;
    win.start(p, decode_row(p, ln.row));
    const int kstep4 = p.d[2] * p.heads * (D / 4);   // float4s between consecutive keys of a line
    const float sl2 = p.scale * kLog2e;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float m = -INFINITY, l = 0.f;
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const long long r0 = win.line_row(p, t0, t1);
            const float4* kl = chunk_ptr(p.key, r0, D, ln.c);
            const float4* vl = chunk_ptr(p.value, r0, D, ln.c);
            for (int t2 = 0; t2 < p.k[2]; t2 += kGF) {
                const int n = min(kGF, p.k[2] - t2);
                float4 kc[kGF], vc[kGF];
#pragma unroll
                for (int g = 0; g < kGF; ++g) {
                    const long long o = static_cast<long long>(t2 + min(g, n - 1)) * kstep4;   // a valid key in every slot
                    kc[g] = __ldg(kl + o);
                    vc[g] = __ldg(vl + o);
                }
                float sg[kGF];
                float gm = -INFINITY;
#pragma unroll
                for (int g = 0; g < kGF; ++g) {
                    const float sv = sl2 * ln.sum(dot4(qc, kc[g]));
                    sg[g] = g < n ? sv : -INFINITY;
                    gm = fmaxf(gm, sg[g]);
                }
                const float mn = fmaxf(m, gm);
                const float corr = fast_exp2(m - mn);   // 0 on the first group (m = -inf)
                l *= corr;
                scale4(acc, corr);
#pragma unroll
                for (int g = 0; g < kGF; ++g) {
                    const float pe = fast_exp2(sg[g] - mn);   // 0 for the empty slots
                    l += pe;
                    axpy4(acc, pe, vc[g]);
                }
                m = mn;
            }
        }
    if (ln.store) {
        scale4(acc, 1.f / l);
        reinterpret_cast<float4*>(static_cast<float*>(p.out0) + ln.row * D)[ln.c] = acc;
        if (ln.c == 0) static_cast<float*>(p.out1)[ln.row] = (m + __log2f(l)) * kLn2;
    }
}

// dQ = scale * sum_j dS_ij k_j with P = exp(scale q.k - LSE), dS = P (dO.v - Delta).
template <int D>
__global__ void __launch_bounds__(kFmaThreads) dq_fma_kernel(const FmaParams p) {
    const long long rows = static_cast<long long>(p.B) * p.N * p.heads;
    RowLanes<D, true> ln;
    if (!ln.init(rows)) return;
    const float4 qc = __ldg(chunk_ptr(p.q, ln.row, D, ln.c));
    const float4 gc = __ldg(chunk_ptr(p.dO, ln.row, D, ln.c));
    const float nl2 = -p.lse[ln.row] * kLog2e, dlt = p.delta[ln.row];
    const float sl2 = p.scale * kLog2e;
    FmaWindow win;
    win.start(p, decode_row(p, ln.row));
    const int kstep4 = p.d[2] * p.heads * (D / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const long long r0 = win.line_row(p, t0, t1);
            const float4* kl = chunk_ptr(p.key, r0, D, ln.c);
            const float4* vl = chunk_ptr(p.value, r0, D, ln.c);
            for (int t2 = 0; t2 < p.k[2]; t2 += kGB) {
                const int n = min(kGB, p.k[2] - t2);
                float4 kc[kGB], vc[kGB];
#pragma unroll
                for (int g = 0; g < kGB; ++g) {
                    const long long o = static_cast<long long>(t2 + min(g, n - 1)) * kstep4;
                    kc[g] = __ldg(kl + o);
                    vc[g] = __ldg(vl + o);
                }
#pragma unroll
                for (int g = 0; g < kGB; ++g) {
                    const float s = ln.sum(dot4(qc, kc[g]));
                    const float dp = ln.sum(dot4(gc, vc[g]));
                    const float ds = g < n ? fast_exp2(fmaf(sl2, s, nl2)) * (dp - dlt) : 0.f;
                    axpy4(acc, ds, kc[g]);
                }
            }
        }
    if (ln.store) {
        scale4(acc, p.scale);
        reinterpret_cast<float4*>(static_cast<float*>(p.out0) + ln.row * D)[ln.c] = acc;
    }
}

// dK, dV: one row's lanes per key, gathering over the queries whose windows hold the key.  Per axis
// those queries form the class-index interval [i_lo, i_hi]: i_lo = 0 if j < k else j - k/2, and
// i_hi = Lc - 1 if j >= Lc - k else j + k/2 (the border keys are seen by more queries).
template <int D>
__global__ void __launch_bounds__(kFmaThreads) dkdv_fma_kernel(const FmaParams p) {
    const long long rows = static_cast<long long>(p.B) * p.N * p.heads;
    RowLanes<D, false> ln;
    if (!ln.init(rows)) return;
    const RowIdx r = decode_row(p, ln.row);
    int lo[3], hi[3], cl[3];
    for (int a = 0; a < 3; ++a) {
        const int d = p.d[a], c = r.x[a] % d, j = r.x[a] / d, Lc = class_len(p.L[a], d, c), ka = p.k[a];
        lo[a] = j < ka ? 0 : j - ka / 2;
        hi[a] = j >= Lc - ka ? Lc - 1 : j + ka / 2;
        cl[a] = c;
    }
    const float4 kc = __ldg(chunk_ptr(p.key, ln.row, D, ln.c));
    const float4 vc = __ldg(chunk_ptr(p.value, ln.row, D, ln.c));
    const float sl2 = p.scale * kLog2e;
    float4 dk = make_float4(0.f, 0.f, 0.f, 0.f), dv = make_float4(0.f, 0.f, 0.f, 0.f);
    const int qstep = p.d[2] * p.heads;
    for (int i0 = lo[0]; i0 <= hi[0]; ++i0)
        for (int i1 = lo[1]; i1 <= hi[1]; ++i1) {
            const long long tok =
                ((r.b * p.L[0] + cl[0] + p.d[0] * i0) * p.L[1] + cl[1] + p.d[1] * i1) * p.L[2] + cl[2];
            const long long qr0 = tok * p.heads + r.h;   // query row of class index 0 along axis 2
            const float4* ql = chunk_ptr(p.q, qr0, D, ln.c);
            const float4* gl = chunk_ptr(p.dO, qr0, D, ln.c);
            const float* lsl = p.lse + qr0;
            const float* dll = p.delta + qr0;
            for (int i2 = lo[2]; i2 <= hi[2]; i2 += kGB) {
                const int n = min(kGB, hi[2] - i2 + 1);
                float4 qc[kGB], gc[kGB];
                float ls[kGB], dl[kGB];
#pragma unroll
                for (int g = 0; g < kGB; ++g) {
                    const int ii = i2 + min(g, n - 1);   // a valid query in every slot
                    const long long oq = static_cast<long long>(ii) * qstep;
                    qc[g] = __ldg(ql + oq * (D / 4));
                    gc[g] = __ldg(gl + oq * (D / 4));
                    ls[g] = __ldg(lsl + oq);
                    dl[g] = __ldg(dll + oq);
                }
#pragma unroll
                for (int g = 0; g < kGB; ++g) {
                    const float s = ln.sum(dot4(kc, qc[g]));
                    const float dp = ln.sum(dot4(vc, gc[g]));
                    const float pe = g < n ? fast_exp2(fmaf(sl2, s, -ls[g] * kLog2e)) : 0.f;
                    axpy4(dv, pe, gc[g]);
                    axpy4(dk, pe * (dp - dl[g]), qc[g]);
                }
            }
        }
    if (ln.store) {
        scale4(dk, p.scale);
        reinterpret_cast<float4*>(static_cast<float*>(p.out0) + ln.row * D)[ln.c] = dk;
        reinterpret_cast<float4*>(static_cast<float*>(p.out1) + ln.row * D)[ln.c] = dv;
    }
}

// Delta = <dO, O> per row.  Each row is split over G = D*bytes/16 lanes (16 bytes each), reduced
// with warp shuffles; a warp covers 32/G rows per step of a grid-stride loop.
template <typename T>
__global__ void __launch_bounds__(256) delta_kernel(const T* __restrict__ o, const T* __restrict__ dO,
                                                    float* __restrict__ delta, long long rows, int D) {
    constexpr int kPer = 16 / sizeof(T);  // elements per 16-byte load
    const int G = D / kPer;               // lanes per row (power of two, <= 32)
    const int lane = threadIdx.x & 31;
    const int rows_per_warp = 32 / G;
    const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long base = warp_id * rows_per_warp; base < rows; base += nwarps * rows_per_warp) {
        const long long row = base + lane / G;
        float acc = 0.f;
        if (row < rows) {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + (lane % G));
            const uint4 b = __ldg(reinterpret_cast<const uint4*>(dO + row * D) + (lane % G));
            const T* ta = reinterpret_cast<const T*>(&a);
            const T* tb = reinterpret_cast<const T*>(&b);
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc = fmaf(static_cast<float>(ta[e]), static_cast<float>(tb[e]), acc);
        }
        for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (row < rows && lane % G == 0) delta[row] = acc;
    }
}


template <int D, typename F>
int launch_rows(F kernel, const FmaParams& p, cudaStream_t s) {
    const long long total = static_cast<long long>(p.B) * p.N * p.heads;
    if (total == 0) return 0;
    const long long blocks = (total * (D / 4) + kFmaThreads - 1) / kFmaThreads;
    kernel<<<dim3(static_cast<unsigned>(blocks)), dim3(kFmaThreads), 0, s>>>(p);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_fwd_fma(const FmaParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_rows<16>(fwd_fma_kernel<16>, p, s);
        case 32: return launch_rows<32>(fwd_fma_kernel<32>, p, s);
        case 64: return launch_rows<64>(fwd_fma_kernel<64>, p, s);
        case 128: return launch_rows<128>(fwd_fma_kernel<128>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dq_fma(const FmaParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_rows<16>(dq_fma_kernel<16>, p, s);
        case 32: return launch_rows<32>(dq_fma_kernel<32>, p, s);
        case 64: return launch_rows<64>(dq_fma_kernel<64>, p, s);
        case 128: return launch_rows<128>(dq_fma_kernel<128>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dkdv_fma(const FmaParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_rows<16>(dkdv_fma_kernel<16>, p, s);
        case 32: return launch_rows<32>(dkdv_fma_kernel<32>, p, s);
        case 64: return launch_rows<64>(dkdv_fma_kernel<64>, p, s);
        case 128: return launch_rows<128>(dkdv_fma_kernel<128>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_delta(const FmaParams& p, int elem, cudaStream_t s) {
    const long long rows = static_cast<long long>(p.B) * p.N * p.heads;
    if (rows == 0) return 0;
    const int per = elem == 1 ? 4 : 8;  // elements per 16-byte load
    const int G = p.D / per;
    const long long rows_per_block = (256 / 32) * (32 / G);
    long long blocks = (rows + rows_per_block - 1) / rows_per_block;
    if (blocks > 152LL * 16) blocks = 152LL * 16;  // grid-stride: 16 resident blocks per SM
    const dim3 grid(static_cast<unsigned>(blocks)), block(256);
    if (elem == 0)
        delta_kernel<__nv_bfloat16><<<grid, block, 0, s>>>(static_cast<const __nv_bfloat16*>(p.o),
                                                           static_cast<const __nv_bfloat16*>(p.dO),
                                                           static_cast<float*>(p.out0), rows, p.D);
    else if (elem == 2)
        delta_kernel<__half><<<grid, block, 0, s>>>(static_cast<const __half*>(p.o), static_cast<const __half*>(p.dO),
                                                    static_cast<float*>(p.out0), rows, p.D);
    else
        delta_kernel<float><<<grid, block, 0, s>>>(static_cast<const float*>(p.o), static_cast<const float*>(p.dO),
                                                   static_cast<float*>(p.out0), rows, p.D);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace na
