// na_fma.cu -- CUDA-core kernels of libna: the fp32 path (forward, dQ, dK/dV; fp32 FMA, no TF32)
// and the Delta prologue shared by both paths.
//
// Neighbourhood as read from NATTEN issue #161 ("Backward pass is very slow towards much tokens and
// large kernels"): per axis, a window of k positions of the query's residue class (dilation d),
// starting at class index clamp(j - k/2, 0, Lc - k); the Cartesian product over axes.  The
// maintainer's remark in that thread that fp32 attention is memory-bound ("FP32 peak FLOPS is
// usually terrible") is why this path keeps one thread per row and lets L1/L2 absorb the window
// overlap instead of tiling through shared memory.
#include <cmath>

#include <cuda_fp16.h>

#include "na_device.cuh"
#include "na_internal.h"

namespace na {
using namespace dev;

namespace {

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

__device__ __forceinline__ long long row_of(const FmaParams& p, long long b, const int* x, int h) {
    return ((b * p.L[0] + x[0]) * p.L[1] + x[1]) * static_cast<long long>(p.L[2]) * p.heads +
           static_cast<long long>(x[2]) * p.heads + h;
}

// First neighbour (spatial index) of spatial index i along axis a.
__device__ __forceinline__ int first_nb(const FmaParams& p, int a, int i) {
    const int d = p.d[a], c = i % d, j = i / d;
    return c + d * win_start(j, class_len(p.L[a], d, c), p.k[a]);
}

template <int D>
__device__ __forceinline__ void load_row(const float* base, long long row, float (&v)[D]) {
    const float4* src = reinterpret_cast<const float4*>(base + row * D);
#pragma unroll
    for (int i = 0; i < D / 4; ++i) {
        const float4 t = __ldg(src + i);
        v[4 * i] = t.x;
        v[4 * i + 1] = t.y;
        v[4 * i + 2] = t.z;
        v[4 * i + 3] = t.w;
    }
}

template <int D>
__device__ __forceinline__ float dot_row(const float (&a)[D], const float* base, long long row) {
    const float4* src = reinterpret_cast<const float4*>(base + row * D);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < D / 4; ++i) {
        const float4 t = __ldg(src + i);
        acc = fmaf(a[4 * i], t.x, acc);
        acc = fmaf(a[4 * i + 1], t.y, acc);
        acc = fmaf(a[4 * i + 2], t.z, acc);
        acc = fmaf(a[4 * i + 3], t.w, acc);
    }
    return acc;
}

template <int D>
__device__ __forceinline__ void axpy_row(float (&acc)[D], float s, const float* base, long long row) {
    const float4* src = reinterpret_cast<const float4*>(base + row * D);
#pragma unroll
    for (int i = 0; i < D / 4; ++i) {
        const float4 t = __ldg(src + i);
        acc[4 * i] = fmaf(s, t.x, acc[4 * i]);
        acc[4 * i + 1] = fmaf(s, t.y, acc[4 * i + 1]);
        acc[4 * i + 2] = fmaf(s, t.z, acc[4 * i + 2]);
        acc[4 * i + 3] = fmaf(s, t.w, acc[4 * i + 3]);
    }
}

template <int D>
__device__ __forceinline__ void store_row(float* base, long long row, const float (&v)[D], float mul) {
    float4* dst = reinterpret_cast<float4*>(base + row * D);
#pragma unroll
    for (int i = 0; i < D / 4; ++i)
        dst[i] = make_float4(v[4 * i] * mul, v[4 * i + 1] * mul, v[4 * i + 2] * mul, v[4 * i + 3] * mul);
}

// Forward: one thread per (batch, token, head) row, online softmax over the window.
template <int D>
__global__ void __launch_bounds__(128) fwd_fma_kernel(const FmaParams p) {
    const long long total = static_cast<long long>(p.B) * p.N * p.heads;
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= total) return;
    const float* q = static_cast<const float*>(p.q);
    const float* k = static_cast<const float*>(p.key);
    const float* v = static_cast<const float*>(p.value);
    const RowIdx r = decode_row(p, row);
    int f[3];
    for (int a = 0; a < 3; ++a) f[a] = first_nb(p, a, r.x[a]);
    float qv[D], acc[D];
    load_row<D>(q, row, qv);
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    float m = -INFINITY, l = 0.f;
    int x[3];
    for (int t0 = 0; t0 < p.k[0]; ++t0) {
        x[0] = f[0] + p.d[0] * t0;
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            x[1] = f[1] + p.d[1] * t1;
            for (int t2 = 0; t2 < p.k[2]; ++t2) {
                x[2] = f[2] + p.d[2] * t2;
                const long long kr = row_of(p, r.b, x, r.h);
                const float s = p.scale * dot_row<D>(qv, k, kr);
                const float mn = fmaxf(m, s);
                const float corr = expf(m - mn);  // 0 on the first key (m = -inf)
                const float pe = expf(s - mn);
                l = l * corr + pe;
#pragma unroll
                for (int c = 0; c < D; ++c) acc[c] *= corr;
                axpy_row<D>(acc, pe, v, kr);
                m = mn;
            }
        }
    }
    store_row<D>(static_cast<float*>(p.out0), row, acc, 1.f / l);
    static_cast<float*>(p.out1)[row] = m + logf(l);
}

// dQ: one thread per query row.
template <int D>
__global__ void __launch_bounds__(128) dq_fma_kernel(const FmaParams p) {
    const long long total = static_cast<long long>(p.B) * p.N * p.heads;
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= total) return;
    const float* q = static_cast<const float*>(p.q);
    const float* k = static_cast<const float*>(p.key);
    const float* v = static_cast<const float*>(p.value);
    const float* dO = static_cast<const float*>(p.dO);
    const RowIdx r = decode_row(p, row);
    int f[3];
    for (int a = 0; a < 3; ++a) f[a] = first_nb(p, a, r.x[a]);
    float qv[D], gv[D], acc[D];
    load_row<D>(q, row, qv);
    load_row<D>(dO, row, gv);
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    const float lse = p.lse[row], dlt = p.delta[row];
    int x[3];
    for (int t0 = 0; t0 < p.k[0]; ++t0) {
        x[0] = f[0] + p.d[0] * t0;
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            x[1] = f[1] + p.d[1] * t1;
            for (int t2 = 0; t2 < p.k[2]; ++t2) {
                x[2] = f[2] + p.d[2] * t2;
                const long long kr = row_of(p, r.b, x, r.h);
                const float pe = expf(p.scale * dot_row<D>(qv, k, kr) - lse);
                const float ds = pe * (dot_row<D>(gv, v, kr) - dlt);
                axpy_row<D>(acc, ds, k, kr);
            }
        }
    }
    store_row<D>(static_cast<float*>(p.out0), row, acc, p.scale);
}

// dK, dV: one thread per key row, gathering over the queries whose windows hold the key.  Per axis
// those queries form the class-index interval [i_lo, i_hi]: i_lo = 0 if j < k else j - k/2, and
// i_hi = Lc - 1 if j >= Lc - k else j + k/2 (the border keys are seen by more queries).
template <int D>
__global__ void __launch_bounds__(128) dkdv_fma_kernel(const FmaParams p) {
    const long long total = static_cast<long long>(p.B) * p.N * p.heads;
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= total) return;
    const float* q = static_cast<const float*>(p.q);
    const float* k = static_cast<const float*>(p.key);
    const float* v = static_cast<const float*>(p.value);
    const float* dO = static_cast<const float*>(p.dO);
    const RowIdx r = decode_row(p, row);
    int lo[3], hi[3], cl[3];
    for (int a = 0; a < 3; ++a) {
        const int d = p.d[a], c = r.x[a] % d, j = r.x[a] / d, Lc = class_len(p.L[a], d, c), ka = p.k[a];
        lo[a] = j < ka ? 0 : j - ka / 2;
        hi[a] = j >= Lc - ka ? Lc - 1 : j + ka / 2;
        cl[a] = c;
    }
    float kv[D], vv[D], dk[D], dv[D];
    load_row<D>(k, row, kv);
    load_row<D>(v, row, vv);
#pragma unroll
    for (int c = 0; c < D; ++c) {
        dk[c] = 0.f;
        dv[c] = 0.f;
    }
    int x[3];
    for (int i0 = lo[0]; i0 <= hi[0]; ++i0) {
        x[0] = cl[0] + p.d[0] * i0;
        for (int i1 = lo[1]; i1 <= hi[1]; ++i1) {
            x[1] = cl[1] + p.d[1] * i1;
            for (int i2 = lo[2]; i2 <= hi[2]; ++i2) {
                x[2] = cl[2] + p.d[2] * i2;
                const long long qr = row_of(p, r.b, x, r.h);
                const float pe = expf(p.scale * dot_row<D>(kv, q, qr) - p.lse[qr]);
                const float ds = pe * (dot_row<D>(vv, dO, qr) - p.delta[qr]);
                axpy_row<D>(dv, pe, dO, qr);
                axpy_row<D>(dk, ds, q, qr);
            }
        }
    }
    store_row<D>(static_cast<float*>(p.out0), row, dk, p.scale);
    store_row<D>(static_cast<float*>(p.out1), row, dv, 1.f);
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


template <typename F>
int launch_rows(F kernel, const FmaParams& p, cudaStream_t s) {
    const long long total = static_cast<long long>(p.B) * p.N * p.heads;
    if (total == 0) return 0;
    const long long blocks = (total + 127) / 128;
    kernel<<<dim3(static_cast<unsigned>(blocks)), dim3(128), 0, s>>>(p);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_fwd_fma(const FmaParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_rows(fwd_fma_kernel<16>, p, s);
        case 32: return launch_rows(fwd_fma_kernel<32>, p, s);
        case 64: return launch_rows(fwd_fma_kernel<64>, p, s);
        case 128: return launch_rows(fwd_fma_kernel<128>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dq_fma(const FmaParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_rows(dq_fma_kernel<16>, p, s);
        case 32: return launch_rows(dq_fma_kernel<32>, p, s);
        case 64: return launch_rows(dq_fma_kernel<64>, p, s);
        case 128: return launch_rows(dq_fma_kernel<128>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dkdv_fma(const FmaParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_rows(dkdv_fma_kernel<16>, p, s);
        case 32: return launch_rows(dkdv_fma_kernel<32>, p, s);
        case 64: return launch_rows(dkdv_fma_kernel<64>, p, s);
        case 128: return launch_rows(dkdv_fma_kernel<128>, p, s);
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
