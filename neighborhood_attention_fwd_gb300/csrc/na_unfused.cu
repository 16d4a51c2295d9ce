// na_unfused.cu -- the unfused neighborhood-attention operations of libna on CUDA cores: attention
// logits (QK over each query's window), a row softmax over the window, the weighted sum (AV), and
// the gradient of each.
//
// NATTEN issue #161 ("Backward pass is very slow towards much tokens and large kernels") benchmarks
// this chain -- na2d_qk, softmax, na2d_av and their backward kernels QGRAD, KGRAD, AGRAD, VGRAD --
// against the fused operation, and its maintainer notes that in fp32 the unfused chain can match the
// fused one because both are memory-bound.  These kernels keep one thread per row (a query row, or a
// key row for the gradients that gather over inverse windows) and let L1/L2 absorb the window
// overlap.
//
// Attention weights are [B, L.., heads, K] with K = k0 k1 k2; window offset t = (t0 k1 + t1) k2 + t2
// (axis 0 outermost) selects key c + d (s + t_a) along each axis a, s the window start.  Every tensor
// has the same element type (fp32, bf16 or fp16); arithmetic is fp32.
#include <cmath>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "na_device.cuh"
#include "na_internal.h"

namespace na {
using namespace dev;

namespace {

template <typename T>
__device__ __forceinline__ float to_f(T v) {
    return static_cast<float>(v);
}
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) {
    return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half from_f<__half>(float v) {
    return __float2half_rn(v);
}

// D elements of a row, widened to fp32 (16-byte loads).
template <typename T, int D>
__device__ __forceinline__ void load_row(const T* base, long long row, float (&v)[D]) {
    constexpr int kPer = 16 / sizeof(T);
    const uint4* src = reinterpret_cast<const uint4*>(base + row * D);
#pragma unroll
    for (int i = 0; i < D / kPer; ++i) {
        const uint4 u = __ldg(src + i);
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int j = 0; j < kPer; ++j) v[i * kPer + j] = to_f(e[j]);
    }
}

template <typename T, int D>
__device__ __forceinline__ float dot_row(const float (&a)[D], const T* base, long long row) {
    float v[D];
    load_row<T, D>(base, row, v);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < D; ++c) acc = fmaf(a[c], v[c], acc);
    return acc;
}

template <typename T, int D>
__device__ __forceinline__ void axpy_row(float (&acc)[D], float s, const T* base, long long row) {
    float v[D];
    load_row<T, D>(base, row, v);
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = fmaf(s, v[c], acc[c]);
}

template <typename T, int D>
__device__ __forceinline__ void store_row(T* base, long long row, const float (&v)[D], float mul) {
    constexpr int kPer = 16 / sizeof(T);
    uint4* dst = reinterpret_cast<uint4*>(base + row * D);
#pragma unroll
    for (int i = 0; i < D / kPer; ++i) {
        uint4 u;
        T* e = reinterpret_cast<T*>(&u);
#pragma unroll
        for (int j = 0; j < kPer; ++j) e[j] = from_f<T>(v[i * kPer + j] * mul);
        dst[i] = u;
    }
}

// Row decode and window geometry (embedded 3D, outermost axis first).
struct Row {
    long long b;
    int h, x[3];
};

__device__ __forceinline__ Row decode(const UnfParams& p, long long row) {
    Row r;
    r.h = static_cast<int>(row % p.heads);
    long long t = row / p.heads;
    for (int a = 2; a >= 0; --a) {
        r.x[a] = static_cast<int>(t % p.L[a]);
        t /= p.L[a];
    }
    r.b = t;
    return r;
}

__device__ __forceinline__ long long row_at(const UnfParams& p, long long b, const int (&x)[3], int h) {
    return (((b * p.L[0] + x[0]) * p.L[1] + x[1]) * p.L[2] + x[2]) * p.heads + h;
}

// First neighbour (spatial index) of spatial index i along axis a.
__device__ __forceinline__ int first_nb(const UnfParams& p, int a, int i) {
    const int d = p.d[a], c = i % d, j = i / d;
    return c + d * win_start(j, class_len(p.L[a], d, c), p.k[a]);
}

// Queries whose windows hold key index x along axis a: class indices [lo, hi] of x's class.
__device__ __forceinline__ void inverse_range(const UnfParams& p, int a, int x, int& lo, int& hi) {
    const int d = p.d[a], c = x % d, j = x / d, Lc = class_len(p.L[a], d, c), k = p.k[a];
    lo = j < k ? 0 : j - (k >> 1);
    hi = j >= Lc - k ? Lc - 1 : j + (k >> 1);
}

// attn[row, t] = scale q_row . k_(t-th neighbour)
template <typename T, int D>
__global__ void __launch_bounds__(128) qk_kernel(const UnfParams p) {
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const T* q = static_cast<const T*>(p.a);
    const T* k = static_cast<const T*>(p.b);
    T* attn = static_cast<T*>(p.out0) + row * p.K;
    const Row r = decode(p, row);
    int f[3];
    for (int a = 0; a < 3; ++a) f[a] = first_nb(p, a, r.x[a]);
    float qv[D];
    load_row<T, D>(q, row, qv);
    int t = 0, x[3];
    for (int t0 = 0; t0 < p.k[0]; ++t0) {
        x[0] = f[0] + p.d[0] * t0;
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            x[1] = f[1] + p.d[1] * t1;
            for (int t2 = 0; t2 < p.k[2]; ++t2, ++t) {
                x[2] = f[2] + p.d[2] * t2;
                attn[t] = from_f<T>(p.scale * dot_row<T, D>(qv, k, row_at(p, r.b, x, r.h)));
            }
        }
    }
}

// o_row = sum_t attn[row, t] v_(t-th neighbour)
template <typename T, int D>
__global__ void __launch_bounds__(128) av_kernel(const UnfParams p) {
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const T* attn = static_cast<const T*>(p.a) + row * p.K;
    const T* v = static_cast<const T*>(p.b);
    const Row r = decode(p, row);
    int f[3];
    for (int a = 0; a < 3; ++a) f[a] = first_nb(p, a, r.x[a]);
    float acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    int t = 0, x[3];
    for (int t0 = 0; t0 < p.k[0]; ++t0) {
        x[0] = f[0] + p.d[0] * t0;
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            x[1] = f[1] + p.d[1] * t1;
            for (int t2 = 0; t2 < p.k[2]; ++t2, ++t) {
                x[2] = f[2] + p.d[2] * t2;
                axpy_row<T, D>(acc, to_f(attn[t]), v, row_at(p, r.b, x, r.h));
            }
        }
    }
    store_row<T, D>(static_cast<T*>(p.out0), row, acc, 1.f);
}

// y = softmax(x) over each row of K weights (x and y may be the same tensor).
template <typename T>
__global__ void __launch_bounds__(128) softmax_kernel(const UnfParams p) {
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const T* x = static_cast<const T*>(p.a) + row * p.K;
    T* y = static_cast<T*>(p.out0) + row * p.K;
    float m = -INFINITY;
    for (int t = 0; t < p.K; ++t) m = fmaxf(m, to_f(x[t]));
    float l = 0.f;
    for (int t = 0; t < p.K; ++t) l += expf(to_f(x[t]) - m);
    const float inv = 1.f / l;
    for (int t = 0; t < p.K; ++t) y[t] = from_f<T>(expf(to_f(x[t]) - m) * inv);
}

// dx = y * (dy - sum_t y dy) over each row (the softmax's gradient; dx may be dy's tensor).
template <typename T>
__global__ void __launch_bounds__(128) softmax_bwd_kernel(const UnfParams p) {
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const T* y = static_cast<const T*>(p.a) + row * p.K;
    const T* dy = static_cast<const T*>(p.b) + row * p.K;
    T* dx = static_cast<T*>(p.out0) + row * p.K;
    float s = 0.f;
    for (int t = 0; t < p.K; ++t) s = fmaf(to_f(y[t]), to_f(dy[t]), s);
    for (int t = 0; t < p.K; ++t) dx[t] = from_f<T>(to_f(y[t]) * (to_f(dy[t]) - s));
}

// Gather over a query's window: out_row = mul * sum_t w[row, t] src_(t-th neighbour).
// dQ of the logits (w = dattn, src = k, mul = scale).
template <typename T, int D>
__global__ void __launch_bounds__(128) gather_kernel(const UnfParams p) {
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const T* w = static_cast<const T*>(p.a) + row * p.K;
    const T* src = static_cast<const T*>(p.b);
    const Row r = decode(p, row);
    int f[3];
    for (int a = 0; a < 3; ++a) f[a] = first_nb(p, a, r.x[a]);
    float acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    int t = 0, x[3];
    for (int t0 = 0; t0 < p.k[0]; ++t0) {
        x[0] = f[0] + p.d[0] * t0;
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            x[1] = f[1] + p.d[1] * t1;
            for (int t2 = 0; t2 < p.k[2]; ++t2, ++t) {
                x[2] = f[2] + p.d[2] * t2;
                axpy_row<T, D>(acc, to_f(w[t]), src, row_at(p, r.b, x, r.h));
            }
        }
    }
    store_row<T, D>(static_cast<T*>(p.out0), row, acc, p.scale);
}

// Gather over a key's inverse window: out_j = mul * sum over queries i whose window holds j of
// w[i, t(i, j)] src_i, t(i, j) the offset of j in i's window.  dK (w = dattn, src = q, mul = scale)
// and dV (w = attn, src = dO, mul = 1); no atomics, every key row is written once.
template <typename T, int D>
__global__ void __launch_bounds__(128) scatter_kernel(const UnfParams p) {
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const T* w = static_cast<const T*>(p.a);
    const T* src = static_cast<const T*>(p.b);
    const Row r = decode(p, row);
    int lo[3], hi[3], cl[3];
    for (int a = 0; a < 3; ++a) {
        inverse_range(p, a, r.x[a], lo[a], hi[a]);
        cl[a] = r.x[a] % p.d[a];
    }
    float acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    int x[3], ta[3];
    for (int i0 = lo[0]; i0 <= hi[0]; ++i0) {
        x[0] = cl[0] + p.d[0] * i0;
        ta[0] = (r.x[0] - first_nb(p, 0, x[0])) / p.d[0];
        for (int i1 = lo[1]; i1 <= hi[1]; ++i1) {
            x[1] = cl[1] + p.d[1] * i1;
            ta[1] = (r.x[1] - first_nb(p, 1, x[1])) / p.d[1];
            for (int i2 = lo[2]; i2 <= hi[2]; ++i2) {
                x[2] = cl[2] + p.d[2] * i2;
                ta[2] = (r.x[2] - first_nb(p, 2, x[2])) / p.d[2];
                const long long qi = row_at(p, r.b, x, r.h);
                const int t = (ta[0] * p.k[1] + ta[1]) * p.k[2] + ta[2];
                axpy_row<T, D>(acc, to_f(w[qi * p.K + t]), src, qi);
            }
        }
    }
    store_row<T, D>(static_cast<T*>(p.out0), row, acc, p.scale);
}

// dattn[row, t] = dO_row . v_(t-th neighbour)  (the weights' gradient of AV)
template <typename T, int D>
__global__ void __launch_bounds__(128) av_bwd_attn_kernel(const UnfParams p) {
    const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const T* dO = static_cast<const T*>(p.a);
    const T* v = static_cast<const T*>(p.b);
    T* dattn = static_cast<T*>(p.out0) + row * p.K;
    const Row r = decode(p, row);
    int f[3];
    for (int a = 0; a < 3; ++a) f[a] = first_nb(p, a, r.x[a]);
    float g[D];
    load_row<T, D>(dO, row, g);
    int t = 0, x[3];
    for (int t0 = 0; t0 < p.k[0]; ++t0) {
        x[0] = f[0] + p.d[0] * t0;
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            x[1] = f[1] + p.d[1] * t1;
            for (int t2 = 0; t2 < p.k[2]; ++t2, ++t) {
                x[2] = f[2] + p.d[2] * t2;
                dattn[t] = from_f<T>(dot_row<T, D>(g, v, row_at(p, r.b, x, r.h)));
            }
        }
    }
}

int launch_rows(void (*kernel)(const UnfParams), const UnfParams& p, cudaStream_t s) {
    if (p.rows == 0) return 0;
    const long long blocks = (p.rows + 127) / 128;
    kernel<<<dim3(static_cast<unsigned>(blocks)), dim3(128), 0, s>>>(p);
    return static_cast<int>(cudaGetLastError());
}

// Kernel selection by element type and head dim.
enum Op { kQK, kAV, kDQ, kDKV, kDAttn };

template <typename T, int D>
int launch_op_td(Op op, const UnfParams& p, cudaStream_t s) {
    switch (op) {
        case kQK: return launch_rows(qk_kernel<T, D>, p, s);
        case kAV: return launch_rows(av_kernel<T, D>, p, s);
        case kDQ: return launch_rows(gather_kernel<T, D>, p, s);
        case kDKV: return launch_rows(scatter_kernel<T, D>, p, s);
        case kDAttn: return launch_rows(av_bwd_attn_kernel<T, D>, p, s);
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

template <typename T>
int launch_op_t(Op op, const UnfParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_op_td<T, 16>(op, p, s);
        case 32: return launch_op_td<T, 32>(op, p, s);
        case 64: return launch_op_td<T, 64>(op, p, s);
        case 128: return launch_op_td<T, 128>(op, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_op(Op op, const UnfParams& p, int elem, cudaStream_t s) {
    if (elem == 0) return launch_op_t<__nv_bfloat16>(op, p, s);
    if (elem == 2) return launch_op_t<__half>(op, p, s);
    return launch_op_t<float>(op, p, s);
}

template <typename T>
int launch_softmax_t(bool bwd, const UnfParams& p, cudaStream_t s) {
    if (p.rows == 0) return 0;
    const long long blocks = (p.rows + 127) / 128;
    if (bwd)
        softmax_bwd_kernel<T><<<dim3(static_cast<unsigned>(blocks)), dim3(128), 0, s>>>(p);
    else
        softmax_kernel<T><<<dim3(static_cast<unsigned>(blocks)), dim3(128), 0, s>>>(p);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_unfused_qk(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kQK, p, elem, s); }
int launch_unfused_av(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kAV, p, elem, s); }
int launch_unfused_gather(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kDQ, p, elem, s); }
int launch_unfused_scatter(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kDKV, p, elem, s); }
int launch_unfused_dattn(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kDAttn, p, elem, s); }
int launch_unfused_softmax(const UnfParams& p, int elem, bool bwd, cudaStream_t s) {
    if (elem == 0) return launch_softmax_t<__nv_bfloat16>(bwd, p, s);
    if (elem == 2) return launch_softmax_t<__half>(bwd, p, s);
    return launch_softmax_t<float>(bwd, p, s);
}

}  // namespace na
