// na_unfused.cu -- the unfused neighborhood-attention operations of libna on CUDA cores: attention
// logits (QK over each query's window), a row softmax over the window, the weighted sum (AV), and
// the gradient of each.
//
// NATTEN issue #161 ("Backward pass is very slow towards much tokens and large kernels") benchmarks
// this chain -- na2d_qk, softmax, na2d_av and their backward kernels QGRAD, KGRAD, AGRAD, VGRAD --
// against the fused operation; its maintainer expects the unfused chain to hold its own in fp32,
// where both are limited by memory rather than arithmetic.
//
// Lane layout.  A [.., heads, D] row is D * s bytes, i.e. CPH = D * s / 16 chunks of 16 bytes, and
// each row gets CPH consecutive lanes, one per chunk: consecutive lanes read consecutive 16-byte
// chunks of q (and of any neighbour row, as neighbouring rows of the same offset sit next to each
// other), so every row load of a warp is coalesced.  A dot product over D is then an in-register
// sum of the lane's chunk plus a butterfly over the row's CPH lanes.  The weights of a warp's rows
// ([rows, K], contiguous in memory) pass through a per-warp shared-memory stage of 128 offsets at a
// time, so they are read and written with consecutive lanes on consecutive elements; the stage's
// row stride is an odd number of 32-bit words, so the rows' lanes hit distinct banks.
//
// Attention weights are [B, L.., heads, K] with K = k0 k1 k2; window offset t = (t0 k1 + t1) k2 + t2
// (axis 0 outermost) selects key c + d (s + t_a) along each axis a, s the window start.  Every tensor
// has the same element type (fp32, bf16 or fp16); arithmetic is fp32.
#include <cmath>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "na_device.cuh"
#include "na_internal.h"

namespace na {
using namespace dev;

namespace {

constexpr int kThreads = 256;   // 8 warps per block
constexpr int kKC = 128;        // window offsets staged per warp and pass
constexpr float kLog2eF = 1.4426950408889634f;   // log2(e): exp(x) = 2^(x log2 e)

// 16-byte chunks: EPC elements widened to fp32 and back (round to nearest even).
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int EPC = 4;
    __device__ static void unpack(const uint4& u, float (&f)[4]) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
    __device__ static float get(float v) { return v; }
    __device__ static float put(float v) { return v; }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int EPC = 8;
    // a bf16 is the upper half of the fp32 with the same bits
    __device__ static void two(uint32_t w, float& lo, float& hi) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
    __device__ static void unpack(const uint4& u, float (&f)[8]) {
        two(u.x, f[0], f[1]);
        two(u.y, f[2], f[3]);
        two(u.z, f[4], f[5]);
        two(u.w, f[6], f[7]);
    }
    __device__ static uint32_t pair(float lo, float hi) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ static uint4 pack(const float (&f)[8]) {
        return make_uint4(pair(f[0], f[1]), pair(f[2], f[3]), pair(f[4], f[5]), pair(f[6], f[7]));
    }
    __device__ static float get(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 put(float v) { return __float2bfloat16_rn(v); }
};

template <>
struct Elem<__half> {
    static constexpr int EPC = 8;
    __device__ static void two(uint32_t w, float& lo, float& hi) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        lo = f.x;
        hi = f.y;
    }
    __device__ static void unpack(const uint4& u, float (&f)[8]) {
        two(u.x, f[0], f[1]);
        two(u.y, f[2], f[3]);
        two(u.z, f[4], f[5]);
        two(u.w, f[6], f[7]);
    }
    __device__ static uint32_t pair(float lo, float hi) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ static uint4 pack(const float (&f)[8]) {
        return make_uint4(pair(f[0], f[1]), pair(f[2], f[3]), pair(f[4], f[5]), pair(f[6], f[7]));
    }
    __device__ static float get(__half v) { return __half2float(v); }
    __device__ static __half put(float v) { return __float2half_rn(v); }
};

template <typename T>
__device__ __forceinline__ uint4 ld16(const T* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// Lane layout of the row-parallel kernels (see the file comment).
template <typename T, int D>
struct Lanes {
    static constexpr int EPC = Elem<T>::EPC;
    static constexpr int CPH = D / EPC;            // lanes per row
    static constexpr int RPW = 32 / CPH;           // rows per warp
    static constexpr int SP = kKC + 4 / sizeof(T); // stage row stride (elements): an odd number of words
    static constexpr size_t kStageBytes = size_t(kThreads / 32) * RPW * SP * sizeof(T);
    static_assert(D % EPC == 0 && 32 % CPH == 0, "unsupported head dim");

    int lane, c, rl, nrows;
    long long row0, row;   // first row of the warp; this lane's row (lanes past the end repeat the last)

    // Returns false for a warp with no rows (the whole warp leaves together).
    __device__ bool init(long long rows) {
        lane = threadIdx.x & 31;
        c = lane % CPH;
        rl = lane / CPH;
        row0 = (static_cast<long long>(blockIdx.x) * kThreads + (threadIdx.x & ~31)) / CPH;
        if (row0 >= rows) return false;
        nrows = static_cast<int>(min(static_cast<long long>(RPW), rows - row0));
        row = row0 + min(rl, nrows - 1);
        return true;
    }
};

// Row decode and window geometry (embedded 3D, outermost axis first).
struct Row {
    long long b;
    int h, x[3];
};

__device__ __forceinline__ Row decode(const UnfParams& p, long long row) {
    Row r;
    if (p.small) {
        uint32_t u = static_cast<uint32_t>(row), q = fdiv(u, p.fd_heads);
        r.h = static_cast<int>(u - q * p.fd_heads.d);
        u = q;
        for (int a = 2; a >= 0; --a) {
            q = fdiv(u, p.fd_L[a]);
            r.x[a] = static_cast<int>(u - q * p.fd_L[a].d);
            u = q;
        }
        r.b = u;
        return r;
    }
    r.h = static_cast<int>(row % p.heads);
    long long t = row / p.heads;
    for (int a = 2; a >= 0; --a) {
        r.x[a] = static_cast<int>(t % p.L[a]);
        t /= p.L[a];
    }
    r.b = t;
    return r;
}

// First neighbour (spatial index) of spatial index i along axis a.
__device__ __forceinline__ int cidx(const UnfParams& p, int a, int i) {   // class index i / d
    return static_cast<int>(fdiv(static_cast<uint32_t>(i), p.fd_d[a]));
}
__device__ __forceinline__ int clen(const UnfParams& p, int a, int c) {   // length of class c
    return static_cast<int>(fdiv(static_cast<uint32_t>(p.L[a] - c + p.d[a] - 1), p.fd_d[a]));
}
__device__ __forceinline__ int first_nb(const UnfParams& p, int a, int i) {
    const int d = p.d[a], j = cidx(p, a, i), c = i - j * d;
    return c + d * win_start(j, clen(p, a, c), p.k[a]);
}

// A tensor-core warp's unit (head fastest, then strip along the innermost axis, the two outer axes,
// batch).
__device__ __forceinline__ void decode_unit(const UnfParams& p, long long unit, int& h, int& s, int& x1, int& x0,
                                            long long& b) {
    if (p.small) {
        uint32_t u = static_cast<uint32_t>(unit), q = fdiv(u, p.fd_heads);
        h = static_cast<int>(u - q * p.fd_heads.d);
        u = q;
        q = fdiv(u, p.fd_strips2);
        s = static_cast<int>(u - q * p.fd_strips2.d);
        u = q;
        q = fdiv(u, p.fd_L[1]);
        x1 = static_cast<int>(u - q * p.fd_L[1].d);
        u = q;
        q = fdiv(u, p.fd_L[0]);
        x0 = static_cast<int>(u - q * p.fd_L[0].d);
        b = q;
        return;
    }
    long long u = unit;
    h = static_cast<int>(u % p.heads);
    u /= p.heads;
    s = static_cast<int>(u % p.strips2);
    u /= p.strips2;
    x1 = static_cast<int>(u % p.L[1]);
    u /= p.L[1];
    x0 = static_cast<int>(u % p.L[0]);
    b = u / p.L[0];
}

// A row's window, walked one key line (fixed t0, t1) at a time: the line's first key row and the
// row step between consecutive keys of the line (offset order t = (t0 k1 + t1) k2 + t2).
struct Window {
    int f[3];
    int rb[3];        // per axis: relative-position index of window offset 0 (class coordinates)
    long long b;
    int h;
    long long step;   // rows between keys t2 and t2 + 1

    __device__ void start(const UnfParams& p, const Row& r) {
        b = r.b;
        h = r.h;
        for (int a = 0; a < 3; ++a) {
            f[a] = first_nb(p, a, r.x[a]);
            rb[a] = cidx(p, a, f[a]) - cidx(p, a, r.x[a]) + p.k[a] - 1;
        }
        step = static_cast<long long>(p.d[2]) * p.heads;
    }
    // Index into one head's bias table [2k0-1, 2k1-1, 2k2-1] of window offset (t0, t1, 0).
    __device__ int rpb_line(const UnfParams& p, int t0, int t1) const {
        return ((rb[0] + t0) * (2 * p.k[1] - 1) + rb[1] + t1) * (2 * p.k[2] - 1) + rb[2];
    }
    __device__ long long line_row(const UnfParams& p, int t0, int t1) const {
        const long long tok = ((b * p.L[0] + f[0] + p.d[0] * t0) * p.L[1] + f[1] + p.d[1] * t1) * p.L[2] + f[2];
        return tok * p.heads + h;
    }
};

// Keys per group in the row-parallel kernels: their loads are issued together, and the dot
// kernel reduces a group's partial sums across the row's lanes with a reduce-scatter.
template <int CPH>
struct Group {
    static constexpr int G = CPH < 8 ? CPH : 8;
};

// Stage <-> global copies of a warp's weight rows [row0, row0 + nrows) x [tc, tc + clen).
template <typename T, int SP>
__device__ __forceinline__ void stage_store(T* out, const T* stage, long long row0, int nrows, int K, int tc,
                                            int clen, int lane) {
    if (clen <= 0 || nrows <= 0) return;
    int rr = 0, j = lane;   // idx = rr * clen + j, stepped by 32 without dividing
    while (j >= clen) {
        j -= clen;
        ++rr;
    }
    for (int idx = lane; idx < nrows * clen; idx += 32) {
        out[(row0 + rr) * K + tc + j] = stage[rr * SP + j];
        for (j += 32; j >= clen; j -= clen) ++rr;
    }
}

template <typename T, int SP>
__device__ __forceinline__ void stage_load(T* stage, const T* in, long long row0, int nrows, int K, int tc, int clen,
                                           int lane) {
    if (clen <= 0 || nrows <= 0) return;
    int rr = 0, j = lane;   // idx = rr * clen + j, stepped by 32 without dividing
    while (j >= clen) {
        j -= clen;
        ++rr;
    }
    for (int idx = lane; idx < nrows * clen; idx += 32) {
        stage[rr * SP + j] = in[(row0 + rr) * K + tc + j];
        for (j += 32; j >= clen; j -= clen) ++rr;
    }
}

// Reduce-scatter of G partial sums over the row's lanes: afterwards s[0] holds, on lane c, the full
// sum (over all CPH lanes) of entry c % G.  Each round halves the entries a lane keeps: the lane
// whose bit m is set keeps the upper half and sends the lower half to its partner, which keeps
// the lower half.
template <int G, int CPH>
__device__ __forceinline__ void reduce_scatter(float (&s)[G], int c) {
#pragma unroll
    for (int m = G / 2; m >= 1; m >>= 1) {
        const bool upper = (c & m) != 0;
#pragma unroll
        for (int j = 0; j < m; ++j) {
            const float send = upper ? s[j] : s[j + m];
            const float keep = upper ? s[j + m] : s[j];
            s[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
#pragma unroll
    for (int m = G; m < CPH; m <<= 1) s[0] += __shfl_xor_sync(0xffffffffu, s[0], m);
}

// out[row, t] = scale * a_row . b_(t-th neighbour of row) (+ rpb[head, relative position of t])
// Logits (a = q, b = k, scale, optional bias) and the weights' gradient of AV (a = dO, b = v, scale 1).
template <typename T, int D, bool BIAS>
__global__ void __launch_bounds__(kThreads) dot_kernel(const UnfParams p) {
    using E = Elem<T>;
    using Ln = Lanes<T, D>;
    constexpr int EPC = Ln::EPC, CPH = Ln::CPH, SP = Ln::SP, G = Group<CPH>::G;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Ln ln;
    if (!ln.init(p.rows)) return;
    T* stage = reinterpret_cast<T*>(smem_raw) + (threadIdx.x >> 5) * Ln::RPW * SP;
    const T* A = static_cast<const T*>(p.a);
    const T* Bm = static_cast<const T*>(p.b) + ln.c * EPC;
    T* out = static_cast<T*>(p.out0);

    float af[EPC];
    E::unpack(ld16(A + ln.row * D + ln.c * EPC), af);
    Window win;
    win.start(p, decode(p, ln.row));
    const int kstep = p.d[2] * p.heads * D;   // elements between consecutive keys of a line
    const float* bias = BIAS ? p.rpb + static_cast<long long>(win.h) * (2 * p.k[0] - 1) * (2 * p.k[1] - 1) *
                                           (2 * p.k[2] - 1)
                             : nullptr;
    int t = 0, tc = 0;
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const T* kp = Bm + win.line_row(p, t0, t1) * D;
            const int bline = BIAS ? win.rpb_line(p, t0, t1) : 0;
            for (int t2 = 0; t2 < p.k[2]; t2 += G) {
                const int n = min(G, p.k[2] - t2);
                if (t + G > tc + kKC) {   // the stage is full: write it out
                    __syncwarp();
                    stage_store<T, SP>(out, stage, ln.row0, ln.nrows, p.K, tc, t - tc, ln.lane);
                    __syncwarp();
                    tc = t;
                }
                uint4 u[G];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    u[g] = g < n ? ld16(kp + static_cast<long long>(t2 + g) * kstep) : make_uint4(0, 0, 0, 0);
                float sg[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float bf[EPC];
                    E::unpack(u[g], bf);
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int e = 0; e < EPC; e += 2) {
                        s0 = fmaf(af[e], bf[e], s0);
                        s1 = fmaf(af[e + 1], bf[e + 1], s1);
                    }
                    sg[g] = s0 + s1;
                }
                reduce_scatter<G, CPH>(sg, ln.c);
                const int g = ln.c % G;
                if (ln.c < G && g < n)
                    stage[ln.rl * SP + (t - tc + g)] =
                        E::put(BIAS ? fmaf(sg[0], p.scale, __ldg(bias + bline + t2 + g)) : sg[0] * p.scale);
                t += n;
            }
        }
    __syncwarp();
    stage_store<T, SP>(out, stage, ln.row0, ln.nrows, p.K, tc, t - tc, ln.lane);
}

// out_row = scale * sum_t w[row, t] src_(t-th neighbour of row)
// AV (w = attn, src = v, scale 1) and dQ of the logits (w = dattn, src = k, scale).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) wsum_kernel(const UnfParams p) {
    using E = Elem<T>;
    using Ln = Lanes<T, D>;
    constexpr int EPC = Ln::EPC, CPH = Ln::CPH, SP = Ln::SP, G = Group<CPH>::G;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Ln ln;
    if (!ln.init(p.rows)) return;
    T* stage = reinterpret_cast<T*>(smem_raw) + (threadIdx.x >> 5) * Ln::RPW * SP;
    const T* W = static_cast<const T*>(p.a);
    const T* S = static_cast<const T*>(p.b) + ln.c * EPC;

    float acc[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) acc[e] = 0.f;
    Window win;
    win.start(p, decode(p, ln.row));
    const int kstep = p.d[2] * p.heads * D;   // elements between consecutive keys of a line
    int t = 0, tc = -kKC;
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const T* kp = S + win.line_row(p, t0, t1) * D;
            for (int t2 = 0; t2 < p.k[2]; t2 += G) {
                const int n = min(G, p.k[2] - t2);
                if (t + G > tc + kKC) {   // stage the next weights
                    tc = t;
                    __syncwarp();
                    stage_load<T, SP>(stage, W, ln.row0, ln.nrows, p.K, tc, min(kKC, p.K - tc), ln.lane);
                    __syncwarp();
                }
                uint4 u[G];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    u[g] = g < n ? ld16(kp + static_cast<long long>(t2 + g) * kstep) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float w = g < n ? E::get(stage[ln.rl * SP + (t - tc + g)]) : 0.f;
                    float sf[EPC];
                    E::unpack(u[g], sf);
#pragma unroll
                    for (int e = 0; e < EPC; ++e) acc[e] = fmaf(w, sf[e], acc[e]);
                }
                t += n;
            }
        }
    if (ln.rl < ln.nrows) {
#pragma unroll
        for (int e = 0; e < EPC; ++e) acc[e] *= p.scale;
        *reinterpret_cast<uint4*>(static_cast<T*>(p.out0) + ln.row * D + ln.c * EPC) = E::pack(acc);
    }
}

// Gather over a key's inverse window: out_j = scale * sum over queries i whose window holds j of
// w[i, t(i, j)] src_i, t(i, j) the offset of j in i's window.  dK (w = dattn, src = q, scale) and
// dV (w = attn, src = dO, scale 1); no atomics, every key row is written once.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) scatter_kernel(const UnfParams p) {
    using E = Elem<T>;
    using Ln = Lanes<T, D>;
    constexpr int EPC = Ln::EPC, G = 2;   // queries per group (larger groups cost resident warps: measured slower)
    Ln ln;
    if (!ln.init(p.rows)) return;
    if (ln.rl >= ln.nrows) return;   // no warp-wide operation follows
    const T* W = static_cast<const T*>(p.a);
    const T* S = static_cast<const T*>(p.b) + ln.c * EPC;
    const Row r = decode(p, ln.row);
    // per axis: the key's class, class index, class length and the class indices of its queries
    int cl[3], jk[3], Lc[3], lo[3], hi[3];
    for (int a = 0; a < 3; ++a) {
        const int d = p.d[a], k = p.k[a];
        jk[a] = cidx(p, a, r.x[a]);
        cl[a] = r.x[a] - jk[a] * d;
        Lc[a] = clen(p, a, cl[a]);
        lo[a] = jk[a] < k ? 0 : jk[a] - (k >> 1);
        hi[a] = jk[a] >= Lc[a] - k ? Lc[a] - 1 : jk[a] + (k >> 1);
    }
    const int qstep = p.d[2] * p.heads;   // rows between consecutive queries of a line
    float acc[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) acc[e] = 0.f;
    for (int i0 = lo[0]; i0 <= hi[0]; ++i0) {
        const int ta0 = jk[0] - win_start(i0, Lc[0], p.k[0]);
        for (int i1 = lo[1]; i1 <= hi[1]; ++i1) {
            const int ta01 = ta0 * p.k[1] + jk[1] - win_start(i1, Lc[1], p.k[1]);
            const long long q0 =
                ((r.b * p.L[0] + cl[0] + p.d[0] * i0) * p.L[1] + cl[1] + p.d[1] * i1) * p.L[2] + cl[2];
            const long long qrow0 = q0 * p.heads + r.h;   // query row of class index 0 along axis 2
            const T* wl = W + qrow0 * p.K;                 // its weights
            const T* sl = S + qrow0 * D;                   // and its row of src
            for (int i2 = lo[2]; i2 <= hi[2]; i2 += G) {
                const int n = min(G, hi[2] - i2 + 1);
                float w[G];
                uint4 u[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (g < n) {
                        const int ii = i2 + g;
                        const long long oq = static_cast<long long>(ii) * qstep;
                        const int t = ta01 * p.k[2] + jk[2] - win_start(ii, Lc[2], p.k[2]);
                        w[g] = E::get(wl[oq * p.K + t]);
                        u[g] = ld16(sl + oq * D);
                    } else {
                        w[g] = 0.f;
                        u[g] = make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float sf[EPC];
                    E::unpack(u[g], sf);
#pragma unroll
                    for (int e = 0; e < EPC; ++e) acc[e] = fmaf(w[g], sf[e], acc[e]);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EPC; ++e) acc[e] *= p.scale;
    *reinterpret_cast<uint4*>(static_cast<T*>(p.out0) + ln.row * D + ln.c * EPC) = E::pack(acc);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ float warp_maxf(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// Rows of up to kRegK weights are held in registers and read once, two rows per warp (16 lanes each,
// kRegK / 16 weights per lane); longer rows take a whole warp and are read again for each pass.
constexpr int kRegK = 128;

__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ float half_maxf(float v) {
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// y = softmax(x) over each row of K weights (x and y may be the same tensor: every read of a row
// happens before its first write).  Rows of at most kRegK weights: two per warp, lanes 16 h .. 16 h + 15
// on row 2 w + h (the warp's pair of rows, row2 = 2 w); longer rows: one per warp.
template <typename T>
__device__ __forceinline__ void softmax_pair(const UnfParams& p, long long row2, int lane) {
    using E = Elem<T>;
    constexpr int NV = kRegK / 16;
    const long long row = row2 + (lane >> 4);
    const bool live = row < p.rows;
    const int l16 = lane & 15;
    const T* x = static_cast<const T*>(p.a) + row * p.K;
    T* y = static_cast<T*>(p.out0) + row * p.K;
    float v[NV];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int t = l16 + 16 * i;
        v[i] = live && t < p.K ? E::get(x[t]) : -INFINITY;
        m = fmaxf(m, v[i]);
    }
    m = half_maxf(m);
    float l = 0.f;
    const float ml2 = m * kLog2eF;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        v[i] = live && l16 + 16 * i < p.K ? fast_exp2(fmaf(v[i], kLog2eF, -ml2)) : 0.f;
        l += v[i];
    }
    const float inv = 1.f / half_sum(l);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < NV; ++i)
        if (live && l16 + 16 * i < p.K) y[l16 + 16 * i] = E::put(v[i] * inv);
}

template <typename T>
__device__ __forceinline__ void softmax_row(const UnfParams& p, long long row, int lane) {
    using E = Elem<T>;
    const T* x = static_cast<const T*>(p.a) + row * p.K;
    T* y = static_cast<T*>(p.out0) + row * p.K;
    float m = -INFINITY;
    for (int t = lane; t < p.K; t += 32) m = fmaxf(m, E::get(x[t]));
    m = warp_maxf(m);
    float l = 0.f;
    const float ml2 = m * kLog2eF;
    for (int t = lane; t < p.K; t += 32) l += fast_exp2(fmaf(E::get(x[t]), kLog2eF, -ml2));
    const float inv = 1.f / warp_sum(l);
    __syncwarp();
    for (int t = lane; t < p.K; t += 32) y[t] = E::put(fast_exp2(fmaf(E::get(x[t]), kLog2eF, -ml2)) * inv);
    __syncwarp();
}

__device__ __forceinline__ long long warp_index() {
    return (static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) softmax_kernel(const UnfParams p) {
    const long long w = warp_index();
    if (p.K <= kRegK) {
        if (2 * w < p.rows) softmax_pair<T>(p, 2 * w, threadIdx.x & 31);   // warp-uniform
    } else if (w < p.rows) {
        softmax_row<T>(p, w, threadIdx.x & 31);
    }
}

// dx = y * (dy - sum_t y dy) over each row (dx may be dy's tensor); rows of at most kRegK weights two
// per warp as in the forward, longer rows one per warp.
template <typename T>
__device__ __forceinline__ void softmax_bwd_pair(const UnfParams& p, long long row2, int lane) {
    using E = Elem<T>;
    constexpr int NV = kRegK / 16;
    const long long row = row2 + (lane >> 4);
    const bool live = row < p.rows;
    const int l16 = lane & 15;
    const T* y = static_cast<const T*>(p.a) + row * p.K;
    const T* dy = static_cast<const T*>(p.b) + row * p.K;
    T* dx = static_cast<T*>(p.out0) + row * p.K;
    float vy[NV], vd[NV];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int t = l16 + 16 * i;
        vy[i] = live && t < p.K ? E::get(y[t]) : 0.f;
        vd[i] = live && t < p.K ? E::get(dy[t]) : 0.f;
        s = fmaf(vy[i], vd[i], s);
    }
    s = half_sum(s);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < NV; ++i)
        if (live && l16 + 16 * i < p.K) dx[l16 + 16 * i] = E::put(vy[i] * (vd[i] - s));
}

template <typename T>
__device__ __forceinline__ void softmax_bwd_row(const UnfParams& p, long long row, int lane) {
    using E = Elem<T>;
    const T* y = static_cast<const T*>(p.a) + row * p.K;
    const T* dy = static_cast<const T*>(p.b) + row * p.K;
    T* dx = static_cast<T*>(p.out0) + row * p.K;
    float s = 0.f;
    for (int t = lane; t < p.K; t += 32) s = fmaf(E::get(y[t]), E::get(dy[t]), s);
    s = warp_sum(s);
    __syncwarp();
    for (int t = lane; t < p.K; t += 32) dx[t] = E::put(E::get(y[t]) * (E::get(dy[t]) - s));
    __syncwarp();
}

template <typename T>
__global__ void __launch_bounds__(kThreads) softmax_bwd_kernel(const UnfParams p) {
    const long long w = warp_index();
    if (p.K <= kRegK) {
        if (2 * w < p.rows) softmax_bwd_pair<T>(p, 2 * w, threadIdx.x & 31);
    } else if (w < p.rows) {
        softmax_bwd_row<T>(p, w, threadIdx.x & 31);
    }
}

// The softmax and its gradient over blocks of 8 consecutive rows (bf16, fp16): 8 rows of K weights are
// 16 K bytes, a whole number of 16-byte chunks from an aligned start, so a warp moves its block with
// 16-byte loads and stores through its own slab of shared memory (every read before any write, so
// the output may be an input's tensor) and takes each row with 4 lanes (lane / 4 is the row).  A warp
// whose block would pass the last row takes its rows one at a time instead.  Used for rows longer than
// kRegK, which the kernels above take one per warp: at 8x128x128 / (5, 7, 7) (K = 245) the softmax went
// 0.97 -> 0.58 ms and its gradient 1.05 -> 0.89 ms; at K = 81 two rows per warp stay faster.
constexpr int kSoftRows8 = 8;
constexpr int kSoftMaxK8 = 256;

template <typename T, bool BWD>
__global__ void __launch_bounds__(kThreads) softmax8_kernel(const UnfParams p) {
    using E = Elem<T>;
    extern __shared__ __align__(16) unsigned char slab_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long row0 = warp_index() * kSoftRows8;
    if (row0 >= p.rows) return;
    if (row0 + kSoftRows8 > p.rows) {
        for (long long r = row0; r < p.rows; ++r) {
            if (BWD) softmax_bwd_row<T>(p, r, lane);
            else softmax_row<T>(p, r, lane);
        }
        return;
    }
    const int K = p.K;   // 8 K two-byte weights: K chunks of 16 bytes
    T* sx = reinterpret_cast<T*>(slab_raw) + static_cast<long long>(warp) * kSoftRows8 * K * (BWD ? 2 : 1);
    T* sd = sx + kSoftRows8 * K;   // the gradient's dy block
    const uint4* gx = reinterpret_cast<const uint4*>(static_cast<const T*>(p.a) + row0 * K);
    for (int i = lane; i < K; i += 32) reinterpret_cast<uint4*>(sx)[i] = __ldg(gx + i);
    if (BWD) {
        const uint4* gd = reinterpret_cast<const uint4*>(static_cast<const T*>(p.b) + row0 * K);
        for (int i = lane; i < K; i += 32) reinterpret_cast<uint4*>(sd)[i] = __ldg(gd + i);
    }
    __syncwarp();
    const int r = lane >> 2, q = lane & 3;
    T* xr = sx + r * K;
    if (!BWD) {
        float m = -INFINITY;
        for (int t = q; t < K; t += 4) m = fmaxf(m, E::get(xr[t]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const float ml2 = m * kLog2eF;
        float l = 0.f;
        for (int t = q; t < K; t += 4) l += fast_exp2(fmaf(E::get(xr[t]), kLog2eF, -ml2));
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const float inv = 1.f / l;
        for (int t = q; t < K; t += 4) xr[t] = E::put(fast_exp2(fmaf(E::get(xr[t]), kLog2eF, -ml2)) * inv);
    } else {
        T* dr = sd + r * K;
        float sum = 0.f;
        for (int t = q; t < K; t += 4) sum = fmaf(E::get(xr[t]), E::get(dr[t]), sum);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        for (int t = q; t < K; t += 4) dr[t] = E::put(E::get(xr[t]) * (E::get(dr[t]) - sum));
    }
    __syncwarp();
    uint4* gy = reinterpret_cast<uint4*>(static_cast<T*>(p.out0) + row0 * K);
    const uint4* src = reinterpret_cast<const uint4*>(BWD ? sd : sx);
    for (int i = lane; i < K; i += 32) gy[i] = src[i];
}

// Gradient of the bias table, first stage: block (chunk of tokens) sums dattn over its tokens'
// (query, offset) pairs, for every head, into a shared-memory copy of the tables.  Consecutive
// tokens with the same relative indices of window offset 0 (every interior query along a line) form
// a run.  One thread per (head, window offset) sums its column over the run straight from global
// memory -- a token's rows for all heads are contiguous, so the threads' loads are too -- and adds
// the sum at that offset's table entry.  Distinct (head, offset) pairs of one run hit distinct
// entries, and runs are separated by a barrier.  Fixed order, no atomics: the result does not
// depend on scheduling.
template <typename T>
__global__ void __launch_bounds__(kThreads) rpb_grad_partial_kernel(const UnfParams p, long long tokens, int tpb,
                                                                   float* partial) {
    using E = Elem<T>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int K = p.K, H = p.heads;
    const int S1 = 2 * p.k[1] - 1, S2 = 2 * p.k[2] - 1, S = (2 * p.k[0] - 1) * S1 * S2;
    float* tab = reinterpret_cast<float*>(smem_raw);                        // [heads][S]
    int* rel = reinterpret_cast<int*>(tab + static_cast<size_t>(H) * S);    // [tpb][3]
    const long long tok0 = static_cast<long long>(blockIdx.x) * tpb;
    const int nt = static_cast<int>(min(static_cast<long long>(tpb), tokens - tok0));
    const T* W = static_cast<const T*>(p.a) + tok0 * H * K;
    for (int e = threadIdx.x; e < H * S; e += kThreads) tab[e] = 0.f;
    for (int rr = threadIdx.x; rr < nt; rr += kThreads) {
        const Row r = decode(p, (tok0 + rr) * H);
        for (int a = 0; a < 3; ++a)
            rel[rr * 3 + a] = cidx(p, a, first_nb(p, a, r.x[a])) - cidx(p, a, r.x[a]) + p.k[a] - 1;
    }
    __syncthreads();
    const int pairs = H * K;   // (head, offset) pairs of one token: its H * K contiguous weights
    for (int rr = 0; rr < nt;) {
        const int r0 = rel[rr * 3], r1 = rel[rr * 3 + 1], r2 = rel[rr * 3 + 2];
        int end = rr + 1;
        while (end < nt && rel[end * 3] == r0 && rel[end * 3 + 1] == r1 && rel[end * 3 + 2] == r2) ++end;
        for (int pi = threadIdx.x; pi < pairs; pi += kThreads) {
            const T* col = W + pi;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            int q = rr;
            for (; q + 4 <= end; q += 4) {
                a0 += E::get(col[static_cast<long long>(q) * pairs]);
                a1 += E::get(col[static_cast<long long>(q + 1) * pairs]);
                a2 += E::get(col[static_cast<long long>(q + 2) * pairs]);
                a3 += E::get(col[static_cast<long long>(q + 3) * pairs]);
            }
            for (; q < end; ++q) a0 += E::get(col[static_cast<long long>(q) * pairs]);
            const int h = static_cast<int>(fdiv(static_cast<uint32_t>(pi), p.fd_K)), t = pi - h * K;
            const int t0 = static_cast<int>(fdiv(static_cast<uint32_t>(t), p.fd_k12));
            const int t12 = t - t0 * p.k[1] * p.k[2];
            const int t1 = static_cast<int>(fdiv(static_cast<uint32_t>(t12), p.fd_k2)), t2 = t12 - t1 * p.k[2];
            tab[h * S + ((r0 + t0) * S1 + r1 + t1) * S2 + r2 + t2] += (a0 + a1) + (a2 + a3);
        }
        __syncthreads();
        rr = end;
    }
    float* out = partial + static_cast<long long>(blockIdx.x) * H * S;
    for (int e = threadIdx.x; e < H * S; e += kThreads) out[e] = tab[e];
}

// Second stage: drpb[e] = sum over chunks of partial[chunk][e], one warp per entry e: lane j sums
// chunks j, j + 32, ... in order, then a fixed butterfly adds the lanes.
__global__ void __launch_bounds__(kThreads) rpb_grad_sum_kernel(const float* partial, long long chunks, int entries,
                                                                float* drpb) {
    const int e = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);   // warp-uniform
    if (e >= entries) return;
    const int lane = threadIdx.x & 31;
    float acc = 0.f;
    for (long long c = lane; c < chunks; c += 32) acc += partial[c * entries + e];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) drpb[e] = acc;
}

// Variable windows: attn[row, t] = -inf for every window offset t outside the row's own window of
// size k_a(x_a) along each axis a (the same shifted-window rule, nested inside the full window).
// One warp per token (its rows for every head are contiguous): the kept offsets form a box
// [lo_a, hi_a] per axis, computed once per token, and only offsets outside it are written (nothing
// is read).  A per-block table holds each offset's (t0, t1, t2), so the per-element test needs no
// division.  Sizes are clamped to [1, k_a] and even sizes lowered by one.
constexpr int kMaskTable = 4096;   // offsets covered by the table; larger windows decode per element

template <typename T>
__global__ void __launch_bounds__(kThreads) mask_window_kernel(const UnfParams p, long long tokens) {
    using E = Elem<T>;
    __shared__ uint32_t tdec[kMaskTable];   // t0 << 20 | t1 << 10 | t2
    const int K = p.K, k1 = p.k[1], k2 = p.k[2];
    const bool table = K <= kMaskTable && k1 <= 1024 && k2 <= 1024;   // the packed fields hold 10 bits
    if (table)
        for (int t = threadIdx.x; t < K; t += kThreads)
            tdec[t] = static_cast<uint32_t>(t / (k1 * k2)) << 20 | static_cast<uint32_t>((t / k2) % k1) << 10 |
                      static_cast<uint32_t>(t % k2);
    __syncthreads();
    const long long tok = warp_index();
    if (tok >= tokens) return;   // warp-uniform
    const int lane = threadIdx.x & 31;
    int x[3];
    if (tokens <= 0x7fffffffLL) {   // 32-bit decode
        unsigned u = static_cast<unsigned>(tok);
        x[2] = static_cast<int>(u % static_cast<unsigned>(p.L[2]));
        u /= static_cast<unsigned>(p.L[2]);
        x[1] = static_cast<int>(u % static_cast<unsigned>(p.L[1]));
        u /= static_cast<unsigned>(p.L[1]);
        x[0] = static_cast<int>(u % static_cast<unsigned>(p.L[0]));
    } else {
        long long u = tok;
        x[2] = static_cast<int>(u % p.L[2]);
        u /= p.L[2];
        x[1] = static_cast<int>(u % p.L[1]);
        u /= p.L[1];
        x[0] = static_cast<int>(u % p.L[0]);
    }
    int lo[3], hi[3];
    bool full = true;
    for (int a = 0; a < 3; ++a) {
        lo[a] = 0;
        hi[a] = p.k[a] - 1;
        if (p.vk_off[a] < 0) continue;
        const int k = p.k[a], d = p.d[a], j = cidx(p, a, x[a]), c = x[a] - j * d, Lc = clen(p, a, c);
        int kv = min(max(__ldg(p.vk + p.vk_off[a] + x[a]), 1), k);
        if ((kv & 1) == 0) --kv;
        lo[a] = win_start(j, Lc, kv) - win_start(j, Lc, k);   // offset of the own window in the full one
        hi[a] = lo[a] + kv - 1;
        full = full && kv == k;
    }
    if (full) return;   // nothing to mask
    const T ninf = E::put(-INFINITY);
    T* out = static_cast<T*>(p.out0) + tok * p.heads * K;
    for (int h = 0; h < p.heads; ++h, out += K)
        for (int t = lane; t < K; t += 32) {
            int t0, t1, t2;
            if (table) {
                const uint32_t dd = tdec[t];
                t0 = static_cast<int>(dd >> 20);
                t1 = static_cast<int>((dd >> 10) & 1023u);
                t2 = static_cast<int>(dd & 1023u);
            } else {
                t0 = t / (k1 * k2);
                t1 = (t / k2) % k1;
                t2 = t % k2;
            }
            if (t0 < lo[0] || t0 > hi[0] || t1 < lo[1] || t1 > hi[1] || t2 < lo[2] || t2 > hi[2]) out[t] = ninf;
        }
}

// Tensor-core logits (bf16, fp16): a warp takes 16 consecutive positions of one residue class along
// the innermost axis, for one head.  Those queries share their windows along the outer axes, and
// along the innermost axis their windows lie in one span of at most 15 + k2 class positions.  Per
// window line (t0, t1) the warp multiplies its 16 q rows by the span's key rows with warp-level MMAs
// (m16n8k16, fp32 accumulation) and keeps, for each query, the k2 products of its own window.
// Fragment layouts (PTX m16n8k16, row.col): with g = lane / 4 and q4 = lane % 4, A register i holds
// row g + 8 (i & 1) and columns 2 q4 + 8 (i >> 1) + {0, 1}; B registers hold rows (keys) g of the
// n-tile and columns 2 q4 + {0, 1} (+ 8); C holds rows g and g + 8, columns 2 q4 + {0, 1}.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if (F16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ld32(const void* base, long long elem_off2) {
    return __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(base) + elem_off2));
}

constexpr int kMmaThreads = 128;   // 4 warps: each stages its 16 rows of K weights in shared memory

template <typename T, int D, bool BIAS, bool STAGE>
__global__ void __launch_bounds__(kMmaThreads) dot_mma_kernel(const UnfParams p) {
    using E = Elem<T>;
    constexpr bool F16 = sizeof(T) == 2 && !std::is_same<T, __nv_bfloat16>::value;
    constexpr int KS = D / 16;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const long long unit = (static_cast<long long>(blockIdx.x) * kMmaThreads + threadIdx.x) >> 5;
    if (unit >= p.units) return;   // warp-uniform
    const int lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3;
    int h, s, x1, x0;
    long long b;
    decode_unit(p, unit, h, s, x1, x0, b);
    const int d2 = p.d[2], k2 = p.k[2];
    int c2 = 0, Lc2 = 0;
    for (c2 = 0; c2 < d2; ++c2) {   // the strip's class along the innermost axis
        Lc2 = clen(p, 2, c2);
        const int n = (Lc2 + 15) >> 4;
        if (s < n) break;
        s -= n;
    }
    const int j0 = s * 16, nq = min(16, Lc2 - j0);
    const int ws0 = win_start(j0, Lc2, k2);
    const int span = win_start(j0 + nq - 1, Lc2, k2) - ws0 + k2;   // key positions the strip's windows cover
    // this lane's two query rows (clamped to the last valid one for loads)
    const int m0 = g, m1 = g + 8;
    const int jq0 = j0 + min(m0, nq - 1), jq1 = j0 + min(m1, nq - 1);
    const long long line_tok = (b * p.L[0] + x0) * p.L[1] + x1;
    const long long r0 = (line_tok * p.L[2] + c2 + static_cast<long long>(d2) * jq0) * p.heads + h;
    const long long r1 = (line_tok * p.L[2] + c2 + static_cast<long long>(d2) * jq1) * p.heads + h;
    const int off0 = win_start(jq0, Lc2, k2) - ws0, off1 = win_start(jq1, Lc2, k2) - ws0;
    uint32_t a[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int col = 16 * ks + 2 * q4;
        a[ks][0] = ld32(p.a, r0 * D + col);
        a[ks][1] = ld32(p.a, r1 * D + col);
        a[ks][2] = ld32(p.a, r0 * D + col + 8);
        a[ks][3] = ld32(p.a, r1 * D + col + 8);
    }
    // outer-axis windows (shared by the strip) and, with a bias, the relative indices
    const int f0 = first_nb(p, 0, x0), f1 = first_nb(p, 1, x1);
    const int S1 = 2 * p.k[1] - 1, S2b = 2 * k2 - 1;
    const int rb0 = cidx(p, 0, f0) - cidx(p, 0, x0) + p.k[0] - 1, rb1 = cidx(p, 1, f1) - cidx(p, 1, x1) + p.k[1] - 1;
    const int rbq0 = ws0 + off0 - jq0 + k2 - 1, rbq1 = ws0 + off1 - jq1 + k2 - 1;
    const float* bias = BIAS ? p.rpb + static_cast<long long>(h) * (2 * p.k[0] - 1) * S1 * S2b : nullptr;
    T* out = static_cast<T*>(p.out0);
    T* stage = reinterpret_cast<T*>(smem_raw) + (threadIdx.x >> 5) * 16 * p.K;   // [16 rows][K]
    const bool v0 = m0 < nq, v1 = m1 < nq;
    const int ntiles = (span + 7) >> 3;
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const long long ktok0 = ((b * p.L[0] + f0 + p.d[0] * t0) * p.L[1] + f1 + p.d[1] * t1) * p.L[2] + c2 +
                                    static_cast<long long>(d2) * ws0;   // the span's first key token
            const int tline = (t0 * p.k[1] + t1) * k2;
            const int bline = BIAS ? ((rb0 + t0) * S1 + rb1 + t1) * S2b : 0;
            for (int nt = 0; nt < ntiles; ++nt) {
                const int nk = min(nt * 8 + g, span - 1);   // this lane's key of the n-tile (clamped)
                const long long kr = (ktok0 + static_cast<long long>(d2) * nk) * p.heads + h;
                float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int col = 16 * ks + 2 * q4;
                    mma16816<F16>(c, a[ks], ld32(p.b, kr * D + col), ld32(p.b, kr * D + col + 8));
                }
                // keep each query's own window: span column n -> window offset n - off
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int n = nt * 8 + 2 * q4 + (e & 1);
                    const bool second = e >= 2;
                    const int t2 = n - (second ? off1 : off0);
                    if ((second ? v1 : v0) && t2 >= 0 && t2 < k2) {
                        float val = c[e] * p.scale;
                        if (BIAS) val += __ldg(bias + bline + (second ? rbq1 : rbq0) + t2);
                        if (STAGE)
                            stage[(second ? m1 : m0) * p.K + tline + t2] = E::put(val);
                        else
                            out[(second ? r1 : r0) * p.K + tline + t2] = E::put(val);
                    }
                }
            }
        }
    if (STAGE) {   // every weight of the strip's rows is staged: write each row's K values contiguously
        __syncwarp();
        const long long rbase = (line_tok * p.L[2] + c2 + static_cast<long long>(d2) * j0) * p.heads + h;
        const long long rstep = static_cast<long long>(d2) * p.heads;   // rows between strip positions
        for (int m = 0; m < nq; ++m) {
            T* dst = out + (rbase + m * rstep) * p.K;
            const T* src = stage + m * p.K;
            for (int t = lane; t < p.K; t += 32) dst[t] = src[t];
        }
    }
}

// The strip of a tensor-core warp: 16 consecutive positions of one residue class along the
// innermost axis (nq of them valid), for one head.
struct Strip {
    long long b, line_tok;   // batch; token index of the strip's line without its innermost coordinate
    int x0, x1, h, c2, Lc2, j0, nq, ws0, span;

    __device__ bool init(const UnfParams& p, long long unit) {
        if (unit >= p.units) return false;
        int s;
        decode_unit(p, unit, h, s, x1, x0, b);
        for (c2 = 0; c2 < p.d[2]; ++c2) {
            Lc2 = clen(p, 2, c2);
            const int n = (Lc2 + 15) >> 4;
            if (s < n) break;
            s -= n;
        }
        j0 = s * 16;
        nq = min(16, Lc2 - j0);
        ws0 = win_start(j0, Lc2, p.k[2]);
        span = win_start(j0 + nq - 1, Lc2, p.k[2]) - ws0 + p.k[2];
        line_tok = (b * p.L[0] + x0) * p.L[1] + x1;
        return true;
    }
    // row index of strip position m (clamped to the last valid one)
    __device__ long long row(const UnfParams& p, int m) const {
        return (line_tok * p.L[2] + c2 + static_cast<long long>(p.d[2]) * (j0 + min(m, nq - 1))) * p.heads + h;
    }
    // offset of position m's window in the span
    __device__ int off(const UnfParams& p, int m) const {
        return win_start(j0 + min(m, nq - 1), Lc2, p.k[2]) - ws0;
    }
};

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// 32-bit shared-memory load (volatile: it must not move above the wait for the copy that fills it)
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t pack_b16(uint16_t lo, uint16_t hi) {
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Tensor-core weighted sums (bf16, fp16): out_row = scale * sum_t w[row, t] src_(t-th neighbour).  Per
// window line the warp's 16 rows form a banded A (the span x weights, zero outside each row's window)
// from its staged weight rows, and the span's src rows, staged with a padded stride, give B through
// ldmatrix.trans; m16n8k16 MMAs accumulate [16, D] in fp32.
template <int D>
struct WsumLayout {
    static constexpr int kVStride = D + 8;   // staged src row stride (elements): conflict-free ldmatrix rows
    __host__ __device__ static int span_pad(int k2) { return ((15 + k2) + 15) / 16 * 16; }
    __host__ __device__ static size_t warp_bytes(int K, int k2) {
        return (static_cast<size_t>(16) * K + static_cast<size_t>(span_pad(k2)) * kVStride) * 2;
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(kMmaThreads) wsum_mma_kernel(const UnfParams p) {
    constexpr bool F16 = !std::is_same<T, __nv_bfloat16>::value;
    constexpr int NT = D / 8, VS = WsumLayout<D>::kVStride;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Strip st;
    if (!st.init(p, (static_cast<long long>(blockIdx.x) * kMmaThreads + threadIdx.x) >> 5)) return;
    const int lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3, warp = threadIdx.x >> 5;
    const int K = p.K, k2 = p.k[2], d2 = p.d[2];
    const int spad = WsumLayout<D>::span_pad(k2);
    uint16_t* ws = reinterpret_cast<uint16_t*>(smem_raw + warp * WsumLayout<D>::warp_bytes(K, k2));   // [16][K]
    uint16_t* vs = ws + 16 * K;                                                                      // [spad][VS]
    const uint16_t* W = static_cast<const uint16_t*>(p.a);
    const uint16_t* S = static_cast<const uint16_t*>(p.b);
    // the strip's weight rows (rows past the last valid one read as zero)
    for (int m = 0; m < 16; ++m) {
        const long long r = st.row(p, m);
        for (int t = lane; t < K; t += 32) ws[m * K + t] = m < st.nq ? W[r * K + t] : uint16_t(0);
    }
    const int om0 = st.off(p, g), om1 = st.off(p, g + 8);
    const int f0 = first_nb(p, 0, st.x0), f1 = first_nb(p, 1, st.x1);
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const uint32_t vs_addr = smem_u32(vs);
    const int nks = (st.span + 15) >> 4;   // k-steps this strip needs
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const long long ktok0 = ((st.b * p.L[0] + f0 + p.d[0] * t0) * p.L[1] + f1 + p.d[1] * t1) * p.L[2] +
                                    st.c2 + static_cast<long long>(d2) * st.ws0;
            const int tline = (t0 * p.k[1] + t1) * k2;
            __syncwarp();   // the previous line's B reads are done
            for (int idx = lane; idx < 16 * nks * (D / 8); idx += 32) {
                const int n = idx / (D / 8), c8 = idx % (D / 8);
                uint4 v = make_uint4(0, 0, 0, 0);
                if (n < st.span) v = ld16(S + ((ktok0 + static_cast<long long>(d2) * n) * p.heads + st.h) * D + 8 * c8);
                *reinterpret_cast<uint4*>(vs + n * VS + 8 * c8) = v;
            }
            __syncwarp();
            for (int ks = 0; ks < nks; ++ks) {
                // A: banded weights, a[i] = rows g (+8), span columns 16 ks + 2 q4 (+8) + {0, 1}
                uint32_t a[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int m = g + 8 * (i & 1), om = (i & 1) ? om1 : om0;
                    const int n = 16 * ks + 2 * q4 + 8 * (i >> 1);
                    const int ta = n - om, tb = n + 1 - om;
                    const uint16_t wa = (ta >= 0 && ta < k2) ? ws[m * K + tline + ta] : uint16_t(0);
                    const uint16_t wb = (tb >= 0 && tb < k2) ? ws[m * K + tline + tb] : uint16_t(0);
                    a[i] = pack_b16(wa, wb);
                }
#pragma unroll
                for (int nt = 0; nt < NT; nt += 2) {
                    // four 8x8 tiles: keys [16 ks, +8) and [+8, +16) of channel blocks nt and nt + 1
                    const int mi = lane >> 3, rr = lane & 7;
                    const uint32_t addr =
                        vs_addr + static_cast<uint32_t>(((16 * ks + 8 * (mi & 1) + rr) * VS + 8 * (nt + (mi >> 1))) * 2);
                    uint32_t bfr[4];
                    ldmatrix_x4_trans(bfr, addr);
                    mma16816<F16>(acc[nt], a, bfr[0], bfr[1]);
                    mma16816<F16>(acc[nt + 1], a, bfr[2], bfr[3]);
                }
            }
        }
    // rows g and g + 8, channels 8 nt + 2 q4 + {0, 1}
    T* out = static_cast<T*>(p.out0);
    const long long r0 = st.row(p, g), r1 = st.row(p, g + 8);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int col = 8 * nt + 2 * q4;
        if (g < st.nq)
            *reinterpret_cast<uint32_t*>(out + r0 * D + col) = Elem<T>::pair(acc[nt][0] * p.scale, acc[nt][1] * p.scale);
        if (g + 8 < st.nq)
            *reinterpret_cast<uint32_t*>(out + r1 * D + col) = Elem<T>::pair(acc[nt][2] * p.scale, acc[nt][3] * p.scale);
    }
}

// The weighted sum fed by TMA (bf16, fp16; D <= 64, tensor maps in p).  Per window line (t0, t1) one
// lane copies the span's source rows (srows rows, swizzled as the row width allows) and the strip's 16
// rows of that line's k2 weights (a box of wb offsets from a 16-byte aligned start) into one of three
// stages of the warp's ring; the banded A and ldmatrix.trans B come from the stage as above.  Rows
// past the strip's queries or the span's keys hold real data or zeros: their weights are zero or their
// results are not stored.  Waits are bounded as in the gather below.
template <int D>
struct WsumTmaLayout {
    static constexpr int kStages = 3;
    __host__ __device__ static uint32_t src_bytes(int srows) { return (srows * 2u * D + 1023u) / 1024u * 1024u; }
    __host__ __device__ static uint32_t w_bytes(int wb) { return 32u * static_cast<uint32_t>(wb); }
    __host__ __device__ static uint32_t warp_bytes(int srows, int wb) {
        return (kStages * (src_bytes(srows) + w_bytes(wb)) + 8u * kStages + 1023u) / 1024u * 1024u;
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(kMmaThreads) wsum_tma_kernel(const __grid_constant__ UnfParams p) {
    constexpr bool F16 = !std::is_same<T, __nv_bfloat16>::value;
    constexpr int NT = D / 8, S = WsumTmaLayout<D>::kStages;
    // swizzle of the source rows (2 D bytes each): 16-byte chunk c of row n sits at chunk c ^ ((n >> kSh) & kMask)
    constexpr int kMask = 2 * D / 16 - 1, kSh = D == 64 ? 0 : (D == 32 ? 1 : 2);
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Strip st;
    if (!st.init(p, (static_cast<long long>(blockIdx.x) * kMmaThreads + threadIdx.x) >> 5)) return;
    const int lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3, warp = threadIdx.x >> 5;
    const int K = p.K, k2 = p.k[2], d2 = p.d[2], wb = static_cast<int>(p.wb), srows = static_cast<int>(p.srows);
    const uint32_t kSrc = WsumTmaLayout<D>::src_bytes(srows), wbytes = WsumTmaLayout<D>::w_bytes(wb);
    unsigned char* wbase = smem + warp * WsumTmaLayout<D>::warp_bytes(srows, wb);
    const uint32_t src0 = smem_u32(wbase);
    const uint16_t* wst0 = reinterpret_cast<const uint16_t*>(wbase + S * kSrc);
    uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + S * (kSrc + wbytes));
    const WaitGuard err{p.err, p.wait_ns};
    const int om0 = st.off(p, g), om1 = st.off(p, g + 8);
    const int f0 = first_nb(p, 0, st.x0), f1 = first_nb(p, 1, st.x1);
    const int nl = p.k[0] * p.k[1];  // window lines (t0, t1)
    const int nks = (st.span + 15) >> 4;  // k-steps this strip needs (span <= srows)
    if (lane == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    __syncwarp();
    auto issue = [&](int li) {
        const int t0 = li / p.k[1], t1 = li % p.k[1], s = li % S;
        const int wc = st.h * K + (t0 * p.k[1] + t1) * k2;
        mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(srows) * 2u * D + wbytes);
        tma_load_5d(wbase + s * kSrc, &p.tm_src, &bars[s], st.h * D, st.c2 + d2 * st.ws0, f1 + p.d[1] * t1,
                    f0 + p.d[0] * t0, static_cast<int>(st.b));
        tma_load_5d(wbase + S * kSrc + s * wbytes, &p.tm_w, &bars[s], wc & ~7, st.c2 + d2 * st.j0, st.x1, st.x0,
                    static_cast<int>(st.b));
    };
    if (lane == 0)
        for (int li = 0; li < S && li < nl; ++li) issue(li);
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    int li = 0;
    bool ok = true;
    for (; li < nl; ++li) {
        const int s = li % S;
        if (!__all_sync(0xffffffffu, mbar_test(&bars[s], (li / S) & 1)) &&
            !__all_sync(0xffffffffu, mbar_block(&bars[s], (li / S) & 1, err, kSiteKV))) {
            ok = false;
            break;
        }
        const int wc = st.h * K + li * k2;  // li = t0 k1 + t1: the line's first weight in the row
        const uint16_t* wst = wst0 + s * (wbytes / 2) + (wc & 7);  // query m's weight u at wst[m wb + u]
        const uint32_t vs = src0 + s * kSrc;
        for (int ks = 0; ks < nks; ++ks) {
            // A: banded weights, a[i] = rows g (+8), span columns 16 ks + 2 q4 (+8) + {0, 1}
            uint32_t a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = g + 8 * (i & 1), om = (i & 1) ? om1 : om0;
                const int n = 16 * ks + 2 * q4 + 8 * (i >> 1);
                const int ta = n - om, tb = n + 1 - om;
                const uint16_t wa = (ta >= 0 && ta < k2) ? wst[m * wb + ta] : uint16_t(0);
                const uint16_t wbv = (tb >= 0 && tb < k2) ? wst[m * wb + tb] : uint16_t(0);
                a[i] = pack_b16(wa, wbv);
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt += 2) {
                const int mi = lane >> 3, rr = lane & 7;
                const int n = 16 * ks + 8 * (mi & 1) + rr, c = nt + (mi >> 1);
                const uint32_t addr = vs + static_cast<uint32_t>(n * 2 * D + ((c ^ ((n >> kSh) & kMask)) << 4));
                uint32_t bfr[4];
                ldmatrix_x4_trans(bfr, addr);
                mma16816<F16>(acc[nt], a, bfr[0], bfr[1]);
                mma16816<F16>(acc[nt + 1], a, bfr[2], bfr[3]);
            }
        }
        __syncwarp();  // every lane is done with stage s
        if (lane == 0 && li + S < nl) issue(li + S);
    }
    if (!ok) {
        if (lane == 0)
            for (int l = li; l < nl && l < li + S; ++l) mbar_drain(&bars[l % S], (l / S) & 1, err.limit_ns);
        __syncwarp();
        return;
    }
    T* out = static_cast<T*>(p.out0);
    const long long r0 = st.row(p, g), r1 = st.row(p, g + 8);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int col = 8 * nt + 2 * q4;
        if (g < st.nq)
            *reinterpret_cast<uint32_t*>(out + r0 * D + col) = Elem<T>::pair(acc[nt][0] * p.scale, acc[nt][1] * p.scale);
        if (g + 8 < st.nq)
            *reinterpret_cast<uint32_t*>(out + r1 * D + col) = Elem<T>::pair(acc[nt][2] * p.scale, acc[nt][3] * p.scale);
    }
}

// The logits fed by TMA (bf16, fp16; D <= 64, the key map in p.tm_src): per window line one lane copies
// the span's key rows (srows rows, swizzled as the row width allows) into one of three stages of the
// warp's ring; B fragments are read from the stage through the swizzle.  The strip's weights are
// staged in shared memory ([16][K]) and written row by row at the end.  Waits are bounded.
template <int D>
struct DotTmaLayout {
    static constexpr int kStages = 3;
    __host__ __device__ static uint32_t src_bytes(int srows) { return (srows * 2u * D + 1023u) / 1024u * 1024u; }
    __host__ __device__ static uint32_t warp_bytes(int srows, int K, size_t elem) {
        const uint32_t out = (16u * K * static_cast<uint32_t>(elem) + 15u) / 16u * 16u;
        return (kStages * src_bytes(srows) + out + 8u * kStages + 1023u) / 1024u * 1024u;
    }
};

template <typename T, int D, bool BIAS>
__global__ void __launch_bounds__(kMmaThreads) dot_tma_kernel(const __grid_constant__ UnfParams p) {
    using E = Elem<T>;
    constexpr bool F16 = !std::is_same<T, __nv_bfloat16>::value;
    constexpr int KS = D / 16, S = DotTmaLayout<D>::kStages;
    constexpr int kMask = 2 * D / 16 - 1, kSh = D == 64 ? 0 : (D == 32 ? 1 : 2);
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Strip st;
    if (!st.init(p, (static_cast<long long>(blockIdx.x) * kMmaThreads + threadIdx.x) >> 5)) return;
    const int lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3, warp = threadIdx.x >> 5;
    const int d2 = p.d[2], k2 = p.k[2], srows = static_cast<int>(p.srows);
    const uint32_t kSrc = DotTmaLayout<D>::src_bytes(srows);
    unsigned char* wbase = smem + warp * DotTmaLayout<D>::warp_bytes(srows, p.K, sizeof(T));
    const uint32_t src0 = smem_u32(wbase);
    T* stage = reinterpret_cast<T*>(wbase + S * kSrc);   // [16 rows][K]
    uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + DotTmaLayout<D>::warp_bytes(srows, p.K, sizeof(T)) - 8u * S);
    const WaitGuard err{p.err, p.wait_ns};
    const int m0 = g, m1 = g + 8;
    const long long r0 = st.row(p, m0), r1 = st.row(p, m1);
    const int off0 = st.off(p, m0), off1 = st.off(p, m1);
    const int jq0 = st.j0 + min(m0, st.nq - 1), jq1 = st.j0 + min(m1, st.nq - 1);
    uint32_t a[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int col = 16 * ks + 2 * q4;
        a[ks][0] = ld32(p.a, r0 * D + col);
        a[ks][1] = ld32(p.a, r1 * D + col);
        a[ks][2] = ld32(p.a, r0 * D + col + 8);
        a[ks][3] = ld32(p.a, r1 * D + col + 8);
    }
    const int f0 = first_nb(p, 0, st.x0), f1 = first_nb(p, 1, st.x1);
    const int S1 = 2 * p.k[1] - 1, S2b = 2 * k2 - 1;
    const int rb0 = cidx(p, 0, f0) - cidx(p, 0, st.x0) + p.k[0] - 1, rb1 = cidx(p, 1, f1) - cidx(p, 1, st.x1) + p.k[1] - 1;
    const int rbq0 = st.ws0 + off0 - jq0 + k2 - 1, rbq1 = st.ws0 + off1 - jq1 + k2 - 1;
    const float* bias = BIAS ? p.rpb + static_cast<long long>(st.h) * (2 * p.k[0] - 1) * S1 * S2b : nullptr;
    const bool v0 = m0 < st.nq, v1 = m1 < st.nq;
    const int ntiles = (st.span + 7) >> 3;
    const int nl = p.k[0] * p.k[1];
    if (lane == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    __syncwarp();
    auto issue = [&](int li) {
        const int t0 = li / p.k[1], t1 = li % p.k[1], s = li % S;
        mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(srows) * 2u * D);
        tma_load_5d(wbase + s * kSrc, &p.tm_src, &bars[s], st.h * D, st.c2 + d2 * st.ws0, f1 + p.d[1] * t1,
                    f0 + p.d[0] * t0, static_cast<int>(st.b));
    };
    if (lane == 0)
        for (int li = 0; li < S && li < nl; ++li) issue(li);
    int li = 0;
    bool ok = true;
    for (; li < nl; ++li) {
        const int s = li % S, t0 = li / p.k[1], t1 = li % p.k[1];
        if (!__all_sync(0xffffffffu, mbar_test(&bars[s], (li / S) & 1)) &&
            !__all_sync(0xffffffffu, mbar_block(&bars[s], (li / S) & 1, err, kSiteKV))) {
            ok = false;
            break;
        }
        const uint32_t vs = src0 + s * kSrc;
        const int tline = li * k2;
        const int bline = BIAS ? ((rb0 + t0) * S1 + rb1 + t1) * S2b : 0;
        for (int nt = 0; nt < ntiles; ++nt) {
            const int nk = nt * 8 + g;  // this lane's key row of the n-tile (rows past the span hold real data or zeros)
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                // B: key nk, channels 16 ks + 2 q4 (+ 8): 4 bytes in 16-byte chunks 2 ks and 2 ks + 1
                const uint32_t rowa = vs + static_cast<uint32_t>(nk * 2 * D + 4 * q4);
                const uint32_t sw = static_cast<uint32_t>((nk >> kSh) & kMask);
                const uint32_t b0 = ld_shared_u32(rowa + (((2u * ks) ^ sw) << 4));
                const uint32_t b1 = ld_shared_u32(rowa + (((2u * ks + 1u) ^ sw) << 4));
                mma16816<F16>(c, a[ks], b0, b1);
            }
            // keep each query's own window: span column n -> window offset n - off
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = nt * 8 + 2 * q4 + (e & 1);
                const bool second = e >= 2;
                const int t2 = n - (second ? off1 : off0);
                if ((second ? v1 : v0) && t2 >= 0 && t2 < k2) {
                    float val = c[e] * p.scale;
                    if (BIAS) val += __ldg(bias + bline + (second ? rbq1 : rbq0) + t2);
                    stage[(second ? m1 : m0) * p.K + tline + t2] = E::put(val);
                }
            }
        }
        __syncwarp();  // every lane is done with stage s
        if (lane == 0 && li + S < nl) issue(li + S);
    }
    if (!ok) {
        if (lane == 0)
            for (int l = li; l < nl && l < li + S; ++l) mbar_drain(&bars[l % S], (l / S) & 1, err.limit_ns);
        __syncwarp();
        return;
    }
    __syncwarp();
    T* out = static_cast<T*>(p.out0);
    const long long rbase = st.row(p, 0), rstep = static_cast<long long>(d2) * p.heads;  // rows between strip positions
    for (int m = 0; m < st.nq; ++m) {
        T* dst = out + (rbase + m * rstep) * p.K;
        const T* src = stage + m * p.K;
        for (int t = lane; t < p.K; t += 32) dst[t] = src[t];
    }
}

// Tensor-core gathers over inverse windows (bf16, fp16): out_j = scale * sum over the queries i whose
// windows hold key j of w[i, t(i, j)] src_i, for dK (dattn, q) and dV (attn, dO).  The warp is a
// 16-key strip.  Its keys share their inverse ranges along the outer axes; along the innermost axis
// their queries lie in one span [q_lo, q_hi].  Per query line (i0, i1) the warp stages, for every
// query of the span, the k2 weights of its window line that lies on the strip's key line, and the
// span's src rows; A[m, n] is query n's weight for key m (zero when key m is outside query n's
// window), B the src rows through ldmatrix.trans.  Every key row is written once: no atomics.
template <int D>
struct ScatterLayout {
    static constexpr int kVStride = D + 8;
    __host__ __device__ static int span_pad(int k2) { return (16 + 2 * k2 + 15) / 16 * 16; }
    __host__ __device__ static size_t warp_bytes(int k2) {
        const size_t sp = static_cast<size_t>(span_pad(k2));
        return (sp * k2 + sp * kVStride) * 2 + 16;
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(kMmaThreads) scatter_mma_kernel(const UnfParams p) {
    constexpr bool F16 = !std::is_same<T, __nv_bfloat16>::value;
    constexpr int NT = D / 8, VS = ScatterLayout<D>::kVStride;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Strip st;
    if (!st.init(p, (static_cast<long long>(blockIdx.x) * kMmaThreads + threadIdx.x) >> 5)) return;
    const int lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3, warp = threadIdx.x >> 5;
    const int K = p.K, k2 = p.k[2], d2 = p.d[2], r2 = k2 >> 1;
    const int spad = ScatterLayout<D>::span_pad(k2);
    uint16_t* vs = reinterpret_cast<uint16_t*>(smem_raw + warp * ScatterLayout<D>::warp_bytes(k2));   // [spad][VS]
    uint16_t* wst = vs + spad * VS;                                                                   // [spad][k2]
    const uint16_t* W = static_cast<const uint16_t*>(p.a);
    const uint16_t* S = static_cast<const uint16_t*>(p.b);
    // queries of the strip's keys along the innermost axis (class coordinates)
    const int jl = st.j0 + st.nq - 1, Lc2 = st.Lc2;
    const int q_lo = st.j0 < k2 ? 0 : st.j0 - r2;
    const int q_hi = jl >= Lc2 - k2 ? Lc2 - 1 : jl + r2;
    const int qspan = q_hi - q_lo + 1;   // <= 16 + 2 k2 (the layout's span_pad)
    const int nks = (qspan + 15) >> 4;    // k-steps this strip needs (interior strips: fewer than span_pad / 16)
    // outer axes: the keys' class, class index, class length and query ranges (shared by the strip)
    int cl[2], jk[2], Lc[2], lo[2], hi[2];
    const int xo[2] = {st.x0, st.x1};
    for (int a = 0; a < 2; ++a) {
        const int d = p.d[a], k = p.k[a];
        jk[a] = cidx(p, a, xo[a]);
        cl[a] = xo[a] - jk[a] * d;
        Lc[a] = clen(p, a, cl[a]);
        lo[a] = jk[a] < k ? 0 : jk[a] - (k >> 1);
        hi[a] = jk[a] >= Lc[a] - k ? Lc[a] - 1 : jk[a] + (k >> 1);
    }
    const int jm0 = st.j0 + min(g, st.nq - 1), jm1 = st.j0 + min(g + 8, st.nq - 1);   // this lane's keys
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const uint32_t vs_addr = smem_u32(vs);
    for (int i0 = lo[0]; i0 <= hi[0]; ++i0) {
        const int ta0 = jk[0] - win_start(i0, Lc[0], p.k[0]);
        for (int i1 = lo[1]; i1 <= hi[1]; ++i1) {
            const int wline = (ta0 * p.k[1] + jk[1] - win_start(i1, Lc[1], p.k[1])) * k2;
            const long long qtok0 = ((st.b * p.L[0] + cl[0] + p.d[0] * i0) * p.L[1] + cl[1] + p.d[1] * i1) * p.L[2] +
                                    st.c2 + static_cast<long long>(d2) * q_lo;   // the span's first query token
            __syncwarp();   // the previous line's reads are done
            for (int idx = lane; idx < 16 * nks * (D / 8); idx += 32) {
                const int n = idx / (D / 8), c8 = idx % (D / 8);
                uint4 v = make_uint4(0, 0, 0, 0);
                if (n < qspan) v = ld16(S + ((qtok0 + static_cast<long long>(d2) * n) * p.heads + st.h) * D + 8 * c8);
                *reinterpret_cast<uint4*>(vs + n * VS + 8 * c8) = v;
            }
            for (int idx = lane; idx < qspan * k2; idx += 32) {
                const int n = idx / k2, u = idx - n * k2;
                wst[idx] = W[((qtok0 + static_cast<long long>(d2) * n) * p.heads + st.h) * K + wline + u];
            }
            __syncwarp();
            for (int ks = 0; ks < nks; ++ks) {
                // A[m, n]: query n's weight for key m, a[i] = keys g (+8), queries 16 ks + 2 q4 (+8) + {0, 1}
                uint32_t a[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int jm = (i & 1) ? jm1 : jm0;
                    const int n = 16 * ks + 2 * q4 + 8 * (i >> 1);
                    uint16_t e[2];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int nn = n + h2;
                        const int u = jm - win_start(q_lo + nn, Lc2, k2);
                        e[h2] = (nn < qspan && u >= 0 && u < k2) ? wst[nn * k2 + u] : uint16_t(0);
                    }
                    a[i] = pack_b16(e[0], e[1]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; nt += 2) {
                    const int mi = lane >> 3, rr = lane & 7;
                    const uint32_t addr =
                        vs_addr + static_cast<uint32_t>(((16 * ks + 8 * (mi & 1) + rr) * VS + 8 * (nt + (mi >> 1))) * 2);
                    uint32_t bfr[4];
                    ldmatrix_x4_trans(bfr, addr);
                    mma16816<F16>(acc[nt], a, bfr[0], bfr[1]);
                    mma16816<F16>(acc[nt + 1], a, bfr[2], bfr[3]);
                }
            }
        }
    }
    T* out = static_cast<T*>(p.out0);
    const long long r0 = st.row(p, g), r1 = st.row(p, g + 8);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int col = 8 * nt + 2 * q4;
        if (g < st.nq)
            *reinterpret_cast<uint32_t*>(out + r0 * D + col) = Elem<T>::pair(acc[nt][0] * p.scale, acc[nt][1] * p.scale);
        if (g + 8 < st.nq)
            *reinterpret_cast<uint32_t*>(out + r1 * D + col) = Elem<T>::pair(acc[nt][2] * p.scale, acc[nt][3] * p.scale);
    }
}

// The same gather fed by TMA (bf16, fp16; D <= 64, tensor maps in p).  Per query line, one lane
// copies the span's source rows (srows rows, swizzled as the row width allows) and each span query's window
// weights on that line (a box of wb offsets from a 16-byte aligned start) into one of three stages
// of the warp's ring, so the next two lines load while this one's products run; the banded A and
// ldmatrix.trans B are built from the stage as above (B through the swizzle).  Waits are bounded: on
// expiry the warp records the site, lets its copies in flight land and stops.
template <int D>
struct ScatterTmaLayout {
    static constexpr int kStages = 3;
    // span rows (srows, a multiple of 16) of 2 D bytes, each stage from a 1 KB boundary (swizzle atom)
    __host__ __device__ static uint32_t src_bytes(int srows) { return (srows * 2u * D + 1023u) / 1024u * 1024u; }
    __host__ __device__ static uint32_t w_bytes(int srows, int wb) { return 2u * srows * static_cast<uint32_t>(wb); }
    __host__ __device__ static uint32_t warp_bytes(int srows, int wb) {
        return (kStages * (src_bytes(srows) + w_bytes(srows, wb)) + 8u * kStages + 1023u) / 1024u * 1024u;
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(kMmaThreads) scatter_tma_kernel(const __grid_constant__ UnfParams p) {
    constexpr bool F16 = !std::is_same<T, __nv_bfloat16>::value;
    constexpr int NT = D / 8, S = ScatterTmaLayout<D>::kStages;
    // swizzle of the source rows (2 D bytes each): 16-byte chunk c of row n sits at chunk c ^ ((n >> kSh) & kMask)
    constexpr int kMask = 2 * D / 16 - 1, kSh = D == 64 ? 0 : (D == 32 ? 1 : 2);
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Strip st;
    if (!st.init(p, (static_cast<long long>(blockIdx.x) * kMmaThreads + threadIdx.x) >> 5)) return;
    const int lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3, warp = threadIdx.x >> 5;
    const int K = p.K, k2 = p.k[2], d2 = p.d[2], r2 = k2 >> 1, wb = static_cast<int>(p.wb);
    const int srows = static_cast<int>(p.srows);
    const uint32_t kSrc = ScatterTmaLayout<D>::src_bytes(srows), wbytes = ScatterTmaLayout<D>::w_bytes(srows, wb);
    unsigned char* wbase = smem + warp * ScatterTmaLayout<D>::warp_bytes(srows, wb);
    const uint32_t src0 = smem_u32(wbase);
    const uint16_t* wst0 = reinterpret_cast<const uint16_t*>(wbase + S * kSrc);
    uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + S * (kSrc + wbytes));
    const WaitGuard err{p.err, p.wait_ns};
    // queries of the strip's keys along the innermost axis (class coordinates)
    const int jl = st.j0 + st.nq - 1, Lc2 = st.Lc2;
    const int q_lo = st.j0 < k2 ? 0 : st.j0 - r2;
    const int q_hi = jl >= Lc2 - k2 ? Lc2 - 1 : jl + r2;
    const int qspan = q_hi - q_lo + 1;  // <= srows, the rows of the box (the host takes the largest span)
    const int nks = (qspan + 15) >> 4;
    int cl[2], jk[2], Lc[2], lo[2], hi[2];
    const int xo[2] = {st.x0, st.x1};
    for (int a = 0; a < 2; ++a) {
        const int d = p.d[a], k = p.k[a];
        jk[a] = cidx(p, a, xo[a]);
        cl[a] = xo[a] - jk[a] * d;
        Lc[a] = clen(p, a, cl[a]);
        lo[a] = jk[a] < k ? 0 : jk[a] - (k >> 1);
        hi[a] = jk[a] >= Lc[a] - k ? Lc[a] - 1 : jk[a] + (k >> 1);
    }
    const int n1 = hi[1] - lo[1] + 1, nl = (hi[0] - lo[0] + 1) * n1;  // query lines (i0, i1)
    if (lane == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    __syncwarp();
    // weight offset of line li's window line in the row of heads * K weights
    auto wcol = [&](int li) {
        const int i0 = lo[0] + li / n1, i1 = lo[1] + li % n1;
        const int ta0 = jk[0] - win_start(i0, Lc[0], p.k[0]);
        return st.h * K + (ta0 * p.k[1] + jk[1] - win_start(i1, Lc[1], p.k[1])) * k2;
    };
    auto issue = [&](int li) {
        const int i0 = lo[0] + li / n1, i1 = lo[1] + li % n1, s = li % S;
        const int x = st.c2 + d2 * q_lo, y = cl[1] + p.d[1] * i1, z = cl[0] + p.d[0] * i0;
        mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(srows) * 2u * D + wbytes);
        tma_load_5d(wbase + s * kSrc, &p.tm_src, &bars[s], st.h * D, x, y, z, static_cast<int>(st.b));
        tma_load_5d(wbase + S * kSrc + s * wbytes, &p.tm_w, &bars[s], wcol(li) & ~7, x, y, z, static_cast<int>(st.b));
    };
    if (lane == 0)
        for (int li = 0; li < S && li < nl; ++li) issue(li);
    const int jm0 = st.j0 + min(g, st.nq - 1), jm1 = st.j0 + min(g + 8, st.nq - 1);  // this lane's keys
    // the stage index of each of this lane's A elements (the same on every line): element h2 of a[i] at
    // k-step ks is query n's weight for key jm, at n wb + u (u = jm - n's window start), or 0xffff
    // (zero) outside query n's window or the span; two 16-bit entries per word
    constexpr int kMaxKs = 4;  // srows <= 64
    uint32_t aoff[kMaxKs][4];
#pragma unroll
    for (int ks = 0; ks < kMaxKs; ++ks)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int jm = (i & 1) ? jm1 : jm0;
            uint32_t w2 = 0;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int nn = 16 * ks + 2 * q4 + 8 * (i >> 1) + h2;
                const int u = jm - win_start(q_lo + nn, Lc2, k2);
                const uint32_t o = (nn < qspan && u >= 0 && u < k2) ? static_cast<uint32_t>(nn * wb + u) : 0xffffu;
                w2 |= o << (16 * h2);
            }
            aoff[ks][i] = w2;
        }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    int li = 0;
    bool ok = true;
    for (; li < nl; ++li) {
        const int s = li % S;
        if (!__all_sync(0xffffffffu, mbar_test(&bars[s], (li / S) & 1)) &&
            !__all_sync(0xffffffffu, mbar_block(&bars[s], (li / S) & 1, err, kSiteKV))) {
            ok = false;
            break;
        }
        const int wc = wcol(li);
        const uint16_t* wst = wst0 + s * (wbytes / 2) + (wc & 7);  // query n's weight u at wst[n wb + u]
        const uint32_t vs = src0 + s * kSrc;
#pragma unroll
        for (int ks = 0; ks < kMaxKs; ++ks) {
            if (ks >= nks) break;
            // A[m, n]: query n's weight for key m, a[i] = keys g (+8), queries 16 ks + 2 q4 (+8) + {0, 1}
            uint32_t a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t o0 = aoff[ks][i] & 0xffffu, o1 = aoff[ks][i] >> 16;
                a[i] = pack_b16(o0 != 0xffffu ? wst[o0] : uint16_t(0), o1 != 0xffffu ? wst[o1] : uint16_t(0));
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt += 2) {
                const int mi = lane >> 3, rr = lane & 7;
                const int n = 16 * ks + 8 * (mi & 1) + rr, c = nt + (mi >> 1);
                const uint32_t addr = vs + static_cast<uint32_t>(n * 2 * D + ((c ^ ((n >> kSh) & kMask)) << 4));
                uint32_t bfr[4];
                ldmatrix_x4_trans(bfr, addr);
                mma16816<F16>(acc[nt], a, bfr[0], bfr[1]);
                mma16816<F16>(acc[nt + 1], a, bfr[2], bfr[3]);
            }
        }
        __syncwarp();  // every lane is done with stage s
        if (lane == 0 && li + S < nl) issue(li + S);
    }
    if (!ok) {
        // the copies issued for lines li .. min(li + S, nl) - 1 land before the warp's shared memory is left
        if (lane == 0)
            for (int l = li; l < nl && l < li + S; ++l) mbar_drain(&bars[l % S], (l / S) & 1, err.limit_ns);
        __syncwarp();
        return;
    }
    T* out = static_cast<T*>(p.out0);
    const long long r0 = st.row(p, g), r1 = st.row(p, g + 8);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int col = 8 * nt + 2 * q4;
        if (g < st.nq)
            *reinterpret_cast<uint32_t*>(out + r0 * D + col) = Elem<T>::pair(acc[nt][0] * p.scale, acc[nt][1] * p.scale);
        if (g + 8 < st.nq)
            *reinterpret_cast<uint32_t*>(out + r1 * D + col) = Elem<T>::pair(acc[nt][2] * p.scale, acc[nt][3] * p.scale);
    }
}

int launch_blocks(long long threads_needed) { return static_cast<int>((threads_needed + kThreads - 1) / kThreads); }

enum Op { kDot, kWsum, kScatter };

template <typename T, int D>
int launch_op_td(Op op, const UnfParams& p, cudaStream_t s) {
    using Ln = Lanes<T, D>;
    if (p.rows == 0) return 0;
    const dim3 grid(launch_blocks(p.rows * Ln::CPH)), block(kThreads);
    switch (op) {
        case kDot:
            if constexpr (sizeof(T) == 2 && D <= 64) {   // bf16, fp16 fed by TMA (the key map set by the host)
                const size_t smem =
                    (kMmaThreads / 32) * DotTmaLayout<D>::warp_bytes(static_cast<int>(p.srows), p.K, sizeof(T)) + 1024;
                if (p.tma && smem <= 200 * 1024) {
                    const long long batch = p.rows / (static_cast<long long>(p.L[0]) * p.L[1] * p.L[2] * p.heads);
                    const long long units = batch * p.L[0] * p.L[1] * p.strips2 * p.heads;
                    const dim3 g2(static_cast<unsigned>((units * 32 + kMmaThreads - 1) / kMmaThreads)), b2(kMmaThreads);
                    auto run = [&](auto kernel) {
                        if (smem > 48 * 1024)
                            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
                        kernel<<<g2, b2, smem, s>>>(p);
                    };
                    if (p.rpb) run(dot_tma_kernel<T, D, true>);
                    else run(dot_tma_kernel<T, D, false>);
                    return static_cast<int>(cudaGetLastError());
                }
            }
            if constexpr (sizeof(T) == 2) {   // bf16, fp16: tensor-core logits, one warp per 16-position strip
                const long long batch = p.rows / (static_cast<long long>(p.L[0]) * p.L[1] * p.L[2] * p.heads);
                const long long units = batch * p.L[0] * p.L[1] * p.strips2 * p.heads;
                const dim3 g2(static_cast<unsigned>((units * 32 + kMmaThreads - 1) / kMmaThreads)), b2(kMmaThreads);
                const size_t smem = static_cast<size_t>(kMmaThreads / 32) * 16 * p.K * sizeof(T);
                auto run = [&](auto kernel, size_t bytes) {
                    if (bytes > 48 * 1024)
                        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
                    kernel<<<g2, b2, bytes, s>>>(p);
                };
                if (smem <= 200 * 1024) {   // stage the rows; past that, write each weight directly
                    if (p.rpb) run(dot_mma_kernel<T, D, true, true>, smem);
                    else run(dot_mma_kernel<T, D, false, true>, smem);
                } else {
                    if (p.rpb) run(dot_mma_kernel<T, D, true, false>, 0);
                    else run(dot_mma_kernel<T, D, false, false>, 0);
                }
            } else {
                if (p.rpb)
                    dot_kernel<T, D, true><<<grid, block, Ln::kStageBytes, s>>>(p);
                else
                    dot_kernel<T, D, false><<<grid, block, Ln::kStageBytes, s>>>(p);
            }
            break;
        case kWsum: {
            bool done = false;
            if constexpr (sizeof(T) == 2 && D <= 64) {   // bf16, fp16 fed by TMA (tensor maps set by the host)
                const size_t smem =
                    (kMmaThreads / 32) * WsumTmaLayout<D>::warp_bytes(static_cast<int>(p.srows), static_cast<int>(p.wb)) + 1024;
                if (p.tma && smem <= 200 * 1024) {
                    const long long batch = p.rows / (static_cast<long long>(p.L[0]) * p.L[1] * p.L[2] * p.heads);
                    const long long units = batch * p.L[0] * p.L[1] * p.strips2 * p.heads;
                    const dim3 g2(static_cast<unsigned>((units * 32 + kMmaThreads - 1) / kMmaThreads)), b2(kMmaThreads);
                    if (smem > 48 * 1024)
                        cudaFuncSetAttribute(wsum_tma_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
                    wsum_tma_kernel<T, D><<<g2, b2, smem, s>>>(p);
                    done = true;
                }
            }
            if constexpr (sizeof(T) == 2) {   // bf16, fp16: tensor-core weighted sums
                const size_t smem = (kMmaThreads / 32) * WsumLayout<D>::warp_bytes(p.K, p.k[2]);
                if (!done && smem <= 200 * 1024) {
                    const long long batch = p.rows / (static_cast<long long>(p.L[0]) * p.L[1] * p.L[2] * p.heads);
                    const long long units = batch * p.L[0] * p.L[1] * p.strips2 * p.heads;
                    const dim3 g2(static_cast<unsigned>((units * 32 + kMmaThreads - 1) / kMmaThreads)), b2(kMmaThreads);
                    if (smem > 48 * 1024)
                        cudaFuncSetAttribute(wsum_mma_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
                    wsum_mma_kernel<T, D><<<g2, b2, smem, s>>>(p);
                    done = true;
                }
            }
            if (!done) wsum_kernel<T, D><<<grid, block, Ln::kStageBytes, s>>>(p);
            break;
        }
        case kScatter: {
            bool done = false;
            if constexpr (sizeof(T) == 2 && D <= 64) {   // bf16, fp16 fed by TMA (tensor maps set by the host)
                const size_t smem =
                    (kMmaThreads / 32) * ScatterTmaLayout<D>::warp_bytes(static_cast<int>(p.srows), static_cast<int>(p.wb)) + 1024;
                if (p.tma && smem <= 200 * 1024) {
                    const long long batch = p.rows / (static_cast<long long>(p.L[0]) * p.L[1] * p.L[2] * p.heads);
                    const long long units = batch * p.L[0] * p.L[1] * p.strips2 * p.heads;
                    const dim3 g2(static_cast<unsigned>((units * 32 + kMmaThreads - 1) / kMmaThreads)), b2(kMmaThreads);
                    if (smem > 48 * 1024)
                        cudaFuncSetAttribute(scatter_tma_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
                    scatter_tma_kernel<T, D><<<g2, b2, smem, s>>>(p);
                    done = true;
                }
            }
            if constexpr (sizeof(T) == 2) {   // bf16, fp16: tensor-core gathers over inverse windows
                const size_t smem = (kMmaThreads / 32) * ScatterLayout<D>::warp_bytes(p.k[2]);
                if (!done && smem <= 200 * 1024) {
                    const long long batch = p.rows / (static_cast<long long>(p.L[0]) * p.L[1] * p.L[2] * p.heads);
                    const long long units = batch * p.L[0] * p.L[1] * p.strips2 * p.heads;
                    const dim3 g2(static_cast<unsigned>((units * 32 + kMmaThreads - 1) / kMmaThreads)), b2(kMmaThreads);
                    if (smem > 48 * 1024)
                        cudaFuncSetAttribute(scatter_mma_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
                    scatter_mma_kernel<T, D><<<g2, b2, smem, s>>>(p);
                    done = true;
                }
            }
            if (!done) scatter_kernel<T, D><<<grid, block, 0, s>>>(p);
            break;
        }
    }
    return static_cast<int>(cudaGetLastError());
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
    if constexpr (sizeof(T) == 2) {
        const uintptr_t al = reinterpret_cast<uintptr_t>(p.a) | reinterpret_cast<uintptr_t>(p.out0) |
                             (bwd ? reinterpret_cast<uintptr_t>(p.b) : 0u);
        if (p.K > kRegK && p.K <= kSoftMaxK8 && (al & 15u) == 0) {
            const long long warps = (p.rows + kSoftRows8 - 1) / kSoftRows8;
            const dim3 grid(launch_blocks(warps * 32)), block(kThreads);
            const int smem = (kThreads / 32) * kSoftRows8 * p.K * 2 * (bwd ? 2 : 1);
            auto run = [&](auto kernel) {
                if (smem > 48 * 1024) cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                kernel<<<grid, block, smem, s>>>(p);
            };
            if (bwd) run(softmax8_kernel<T, true>);
            else run(softmax8_kernel<T, false>);
            return static_cast<int>(cudaGetLastError());
        }
    }
    const long long warps = p.K <= kRegK ? (p.rows + 1) / 2 : p.rows;  // rows of at most kRegK weights in pairs
    const dim3 grid(launch_blocks(warps * 32)), block(kThreads);
    if (bwd)
        softmax_bwd_kernel<T><<<grid, block, 0, s>>>(p);
    else
        softmax_kernel<T><<<grid, block, 0, s>>>(p);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_unfused_qk(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kDot, p, elem, s); }
int launch_unfused_av(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kWsum, p, elem, s); }
int launch_unfused_gather(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kWsum, p, elem, s); }
int launch_unfused_scatter(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kScatter, p, elem, s); }
int launch_unfused_dattn(const UnfParams& p, int elem, cudaStream_t s) { return launch_op(kDot, p, elem, s); }
// Tokens per block of the first stage (the partial sums are one set of tables per block): small
// enough that even a 512x512 problem gives every SM several blocks to overlap their load latency.
int rpb_grad_tokens_per_block(int K) { return K <= 1024 ? 256 : 64; }

size_t rpb_grad_workspace_bytes(long long tokens, int heads, int K, int table) {
    const long long chunks = (tokens + rpb_grad_tokens_per_block(K) - 1) / rpb_grad_tokens_per_block(K);
    return static_cast<size_t>(chunks) * heads * table * sizeof(float);
}

int launch_unfused_rpb_grad(const UnfParams& p, int elem, long long tokens, float* partial, float* drpb,
                            cudaStream_t s) {
    const int tpb = rpb_grad_tokens_per_block(p.K);
    const long long chunks = (tokens + tpb - 1) / tpb;
    const int table = (2 * p.k[0] - 1) * (2 * p.k[1] - 1) * (2 * p.k[2] - 1);
    const int entries = p.heads * table;
    if (tokens == 0) return static_cast<int>(cudaMemsetAsync(drpb, 0, sizeof(float) * entries, s));
    const size_t smem = static_cast<size_t>(p.heads) * table * sizeof(float) + static_cast<size_t>(tpb) * 3 * sizeof(int);
    if (smem > 227 * 1024) return static_cast<int>(cudaErrorInvalidValue);   // heads x table too large
    const dim3 grid(static_cast<unsigned>(chunks));
    auto run = [&](auto kernel) {
        if (smem > 48 * 1024)   // many heads or very large windows: more than the default
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        kernel<<<grid, kThreads, smem, s>>>(p, tokens, tpb, partial);
    };
    if (elem == 0)
        run(rpb_grad_partial_kernel<__nv_bfloat16>);
    else if (elem == 2)
        run(rpb_grad_partial_kernel<__half>);
    else
        run(rpb_grad_partial_kernel<float>);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return static_cast<int>(e);
    rpb_grad_sum_kernel<<<launch_blocks(static_cast<long long>(entries) * 32), kThreads, 0, s>>>(partial, chunks,
                                                                                                 entries, drpb);
    return static_cast<int>(cudaGetLastError());
}

int launch_unfused_mask_window(const UnfParams& p, int elem, cudaStream_t s) {
    if (p.rows == 0) return 0;
    const long long tokens = p.rows / p.heads;
    const dim3 grid(launch_blocks(tokens * 32)), block(kThreads);
    if (elem == 0)
        mask_window_kernel<__nv_bfloat16><<<grid, block, 0, s>>>(p, tokens);
    else if (elem == 2)
        mask_window_kernel<__half><<<grid, block, 0, s>>>(p, tokens);
    else
        mask_window_kernel<float><<<grid, block, 0, s>>>(p, tokens);
    return static_cast<int>(cudaGetLastError());
}

int launch_unfused_softmax(const UnfParams& p, int elem, bool bwd, cudaStream_t s) {
    if (elem == 0) return launch_softmax_t<__nv_bfloat16>(bwd, p, s);
    if (elem == 2) return launch_softmax_t<__half>(bwd, p, s);
    return launch_softmax_t<float>(bwd, p, s);
}

}  // namespace na
