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
// Lane layout: a row of D fp32 values is D/4 chunks of 16 bytes, spread over the row's consecutive
// lanes (each lane holds kCPL of them, interleaved).  Neighbouring rows (heads, then tokens) sit next
// to each other in memory, so every row load of a warp is coalesced.  Dot products over D are a
// lane's chunks plus a butterfly over the row's lanes (shuffles restricted to those lanes where rows'
// loops differ in length, so they never wait on each other).
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
    if (p.rows32) {
        const uint32_t u = static_cast<uint32_t>(row);
        const uint32_t bt = fdiv(u, p.fd_heads);
        r.h = static_cast<int>(u - bt * p.fd_heads.d);
        const uint32_t b = fdiv(bt, p.fd_N);
        uint32_t t = bt - b * p.fd_N.d;
        r.b = b;
        r.tok = t;
        for (int a = 2; a >= 0; --a) {
            const uint32_t q = fdiv(t, p.fd_L[a]);
            r.x[a] = static_cast<int>(t - q * p.fd_L[a].d);
            t = q;
        }
        return r;
    }
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
    const int d = p.d[a], j = static_cast<int>(fdiv(static_cast<uint32_t>(i), p.fd_d[a])), c = i - j * d;
    const int Lc = static_cast<int>(fdiv(static_cast<uint32_t>(p.L[a] - c + d - 1), p.fd_d[a]));
    return c + d * win_start(j, Lc, p.k[a]);
}

// Chunks of 16 bytes per lane: a lane holds L of its row's D / 4 chunks, the row's lanes interleaved
// (lane c owns chunks c, c + CPH, ...), so each load instruction of a row is still contiguous.  More
// chunks per lane mean more FMAs per butterfly round but more registers; measured at 1024x1024 9x9
// fp32, one chunk per lane suits the forward and dQ, two suit dK/dV.
template <int D, int L>
struct Chunks {
    static constexpr int CPL = L < D / 4 ? L : D / 4;   // chunks per lane
    static constexpr int CPH = D / 4 / CPL;             // lanes per row
    float4 v[CPL];
};
constexpr int kCplF = 1, kCplQ = 1, kCplKV = 2;   // forward, dQ, dK/dV

// The lanes of one row: CPH lanes per row (so a warp holds 32 / CPH rows).  Lanes past the last row repeat
// it and store nothing.  UNIFORM: every row of the warp runs the same loop (forward, dQ), so the
// butterflies may name the whole warp; otherwise they name only the row's lanes.
template <int D, bool UNIFORM, int L>
struct RowLanes {
    static constexpr int CPH = Chunks<D, L>::CPH;
    int c, rl;
    unsigned mask;     // the lanes that take part in a butterfly
    long long row;
    bool store;

    __device__ bool init(long long rows) {
        const int lane = threadIdx.x & 31;
        c = lane % CPH;
        rl = lane / CPH;
        mask = (UNIFORM || CPH == 32) ? 0xffffffffu : ((CPH >= 32 ? 0u : (1u << CPH)) - 1u) << (rl * CPH);
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

// The lane's first chunk of a row (row-major [rows, D] fp32); its others follow every CPH chunks.
template <int D>
__device__ __forceinline__ const float4* chunk_ptr(const void* base, long long row, int c) {
    return reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * D) + c;
}

template <int D, int L>
__device__ __forceinline__ void load_chunks(Chunks<D, L>& x, const float4* p) {
#pragma unroll
    for (int i = 0; i < Chunks<D, L>::CPL; ++i) x.v[i] = __ldg(p + i * Chunks<D, L>::CPH);
}

template <int D, int L>
__device__ __forceinline__ float dot_chunks(const Chunks<D, L>& a, const Chunks<D, L>& b) {
    float s = dot4(a.v[0], b.v[0]);
#pragma unroll
    for (int i = 1; i < Chunks<D, L>::CPL; ++i) s += dot4(a.v[i], b.v[i]);
    return s;
}

template <int D, int L>
__device__ __forceinline__ void axpy_chunks(Chunks<D, L>& acc, float s, const Chunks<D, L>& x) {
#pragma unroll
    for (int i = 0; i < Chunks<D, L>::CPL; ++i) axpy4(acc.v[i], s, x.v[i]);
}

template <int D, int L>
__device__ __forceinline__ void scale_chunks(Chunks<D, L>& acc, float s) {
#pragma unroll
    for (int i = 0; i < Chunks<D, L>::CPL; ++i) scale4(acc.v[i], s);
}

template <int D, int L>
__device__ __forceinline__ void zero_chunks(Chunks<D, L>& acc) {
#pragma unroll
    for (int i = 0; i < Chunks<D, L>::CPL; ++i) acc.v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

template <int D, int L>
__device__ __forceinline__ void store_chunks(void* base, long long row, int c, const Chunks<D, L>& x) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + row * D) + c;
#pragma unroll
    for (int i = 0; i < Chunks<D, L>::CPL; ++i) p[i * Chunks<D, L>::CPH] = x.v[i];
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

// Keys (queries) per group: their loads issue together (and the forward rescales once per group).
// Larger groups keep more loads in flight per warp but cost registers, hence resident warps;
// measured at 1024x1024 9x9 fp32: one for the forward and dK/dV, two for dQ.
constexpr int kGF = 1;
constexpr int kGB = 2;
constexpr int kGKV = 1;

// Forward: online softmax over the window in log2 units (the scale carries log2 e), one rescale
// per group of keys; LSE is stored in natural-log units.
template <int D>
__global__ void __launch_bounds__(kFmaThreads) fwd_fma_kernel(const FmaParams p) {
    const long long rows = static_cast<long long>(p.B) * p.N * p.heads;
    RowLanes<D, true, kCplF> ln;
    if (!ln.init(rows)) return;
    Chunks<D, kCplF> qc;
    load_chunks<D, kCplF>(qc, chunk_ptr<D>(p.q, ln.row, ln.c));
    FmaWindow win;
    win.start(p, decode_row(p, ln.row));
    const int kstep4 = p.d[2] * p.heads * (D / 4);   // float4s between consecutive keys of a line
    const float sl2 = p.scale * kLog2e;
    Chunks<D, kCplF> acc;
    zero_chunks<D, kCplF>(acc);
    float m = -INFINITY, l = 0.f;
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const long long r0 = win.line_row(p, t0, t1);
            const float4* kl = chunk_ptr<D>(p.key, r0, ln.c);
            const float4* vl = chunk_ptr<D>(p.value, r0, ln.c);
            for (int t2 = 0; t2 < p.k[2]; t2 += kGF) {
                const int n = min(kGF, p.k[2] - t2);
                Chunks<D, kCplF> kc[kGF], vc[kGF];
#pragma unroll
                for (int g = 0; g < kGF; ++g) {
                    const long long o = static_cast<long long>(t2 + min(g, n - 1)) * kstep4;   // a valid key in every slot
                    load_chunks<D, kCplF>(kc[g], kl + o);
                    load_chunks<D, kCplF>(vc[g], vl + o);
                }
                float sg[kGF];
                float gm = -INFINITY;
#pragma unroll
                for (int g = 0; g < kGF; ++g) {
                    const float sv = sl2 * ln.sum(dot_chunks<D, kCplF>(qc, kc[g]));
                    sg[g] = g < n ? sv : -INFINITY;
                    gm = fmaxf(gm, sg[g]);
                }
                const float mn = fmaxf(m, gm);
                const float corr = fast_exp2(m - mn);   // 0 on the first group (m = -inf)
                l *= corr;
                scale_chunks<D, kCplF>(acc, corr);
#pragma unroll
                for (int g = 0; g < kGF; ++g) {
                    const float pe = fast_exp2(sg[g] - mn);   // 0 for the empty slots
                    l += pe;
                    axpy_chunks<D, kCplF>(acc, pe, vc[g]);
                }
                m = mn;
            }
        }
    if (ln.store) {
        scale_chunks<D, kCplF>(acc, 1.f / l);
        store_chunks<D, kCplF>(p.out0, ln.row, ln.c, acc);
        if (ln.c == 0) static_cast<float*>(p.out1)[ln.row] = (m + __log2f(l)) * kLn2;
    }
}

// dQ = scale * sum_j dS_ij k_j with P = exp(scale q.k - LSE), dS = P (dO.v - Delta).
template <int D>
__global__ void __launch_bounds__(kFmaThreads) dq_fma_kernel(const FmaParams p) {
    const long long rows = static_cast<long long>(p.B) * p.N * p.heads;
    RowLanes<D, true, kCplQ> ln;
    if (!ln.init(rows)) return;
    Chunks<D, kCplQ> qc, gc;
    load_chunks<D, kCplQ>(qc, chunk_ptr<D>(p.q, ln.row, ln.c));
    load_chunks<D, kCplQ>(gc, chunk_ptr<D>(p.dO, ln.row, ln.c));
    const float nl2 = -p.lse[ln.row] * kLog2e, dlt = p.delta[ln.row];
    const float sl2 = p.scale * kLog2e;
    FmaWindow win;
    win.start(p, decode_row(p, ln.row));
    const int kstep4 = p.d[2] * p.heads * (D / 4);
    Chunks<D, kCplQ> acc;
    zero_chunks<D, kCplQ>(acc);
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const long long r0 = win.line_row(p, t0, t1);
            const float4* kl = chunk_ptr<D>(p.key, r0, ln.c);
            const float4* vl = chunk_ptr<D>(p.value, r0, ln.c);
            for (int t2 = 0; t2 < p.k[2]; t2 += kGB) {
                const int n = min(kGB, p.k[2] - t2);
                Chunks<D, kCplQ> kc[kGB], vc[kGB];
#pragma unroll
                for (int g = 0; g < kGB; ++g) {
                    const long long o = static_cast<long long>(t2 + min(g, n - 1)) * kstep4;
                    load_chunks<D, kCplQ>(kc[g], kl + o);
                    load_chunks<D, kCplQ>(vc[g], vl + o);
                }
#pragma unroll
                for (int g = 0; g < kGB; ++g) {
                    const float s = ln.sum(dot_chunks<D, kCplQ>(qc, kc[g]));
                    const float dp = ln.sum(dot_chunks<D, kCplQ>(gc, vc[g]));
                    const float ds = g < n ? fast_exp2(fmaf(sl2, s, nl2)) * (dp - dlt) : 0.f;
                    axpy_chunks<D, kCplQ>(acc, ds, kc[g]);
                }
            }
        }
    if (ln.store) {
        scale_chunks<D, kCplQ>(acc, p.scale);
        store_chunks<D, kCplQ>(p.out0, ln.row, ln.c, acc);
    }
}

// Query quads.  A group of G = D/4 lanes (one 16-byte chunk of a row each) takes four consecutive
// class positions of one residue class along the innermost axis, one head: their windows share
// every line and, along the innermost axis, span at most k2 + 3 positions, so each key chunk a lane
// loads serves four queries.  Heads are the fastest index, so a warp's groups load neighbouring rows.
// The four partial dot products of a key are finished by a reduce-scatter over the group (two
// exchange steps) and butterflies over the rest: afterwards the lanes c with c / (G/4) = r hold the
// score of query r.
constexpr int kQuad = 4;

struct Quad {
    long long tok0;   // token of class position 0 on the quad's line: ((b L0 + x0) L1 + x1) L2 + c2
    long long b;
    int x0, x1, c2, h, j0, nq, lc2;

    __device__ bool init(const FmaParams& p, uint32_t u) {
        uint32_t q = fdiv(u, p.fd_heads);
        h = static_cast<int>(u - q * p.fd_heads.d);
        u = q;
        q = fdiv(u, p.fd_qc2);
        const int s = static_cast<int>(u - q * p.fd_qc2.d);
        u = q;
        q = fdiv(u, p.fd_d[2]);
        c2 = static_cast<int>(u - q * p.fd_d[2].d);
        u = q;
        q = fdiv(u, p.fd_L[1]);
        x1 = static_cast<int>(u - q * p.fd_L[1].d);
        u = q;
        q = fdiv(u, p.fd_L[0]);
        x0 = static_cast<int>(u - q * p.fd_L[0].d);
        b = q;
        lc2 = static_cast<int>(fdiv(static_cast<uint32_t>(p.L[2] - c2 + p.d[2] - 1), p.fd_d[2]));
        j0 = kQuad * s;
        if (j0 >= lc2) return false;   // past the end of a shorter class
        nq = min(kQuad, lc2 - j0);
        tok0 = ((b * p.L[0] + x0) * p.L[1] + x1) * p.L[2] + c2;
        return true;
    }
    // class position of query r (the last valid one for r >= nq)
    __device__ int j(int r) const { return j0 + min(r, nq - 1); }
    __device__ long long row(const FmaParams& p, int r) const {
        return (tok0 + static_cast<long long>(p.d[2]) * j(r)) * p.heads + h;
    }
};

template <int G>
struct QuadLanes {
    int c, base;      // lane within the group; the group's first lane
    unsigned mask;    // the group's lanes
    __device__ QuadLanes() {
        const int lane = threadIdx.x & 31;
        c = lane & (G - 1);
        base = lane & ~(G - 1);
        mask = G == 32 ? 0xffffffffu : ((1u << G) - 1u) << base;
    }
    __device__ int rq() const { return c / (G / 4); }   // the query whose score this lane ends with
    __device__ bool owner() const { return (c & (G / 4 - 1)) == 0; }
    // the four partial sums of the lane -> the full sum of query rq() over the group
    __device__ float reduce(const float (&v)[kQuad]) const {
        const bool hi = (c & (G / 2)) != 0;
        const float a0 = (hi ? v[2] : v[0]) + __shfl_xor_sync(mask, hi ? v[0] : v[2], G / 2);
        const float a1 = (hi ? v[3] : v[1]) + __shfl_xor_sync(mask, hi ? v[1] : v[3], G / 2);
        const bool lo = (c & (G / 4)) != 0;
        float x = (lo ? a1 : a0) + __shfl_xor_sync(mask, lo ? a0 : a1, G / 4);
#pragma unroll
        for (int m = G / 8; m >= 1; m >>= 1) x += __shfl_xor_sync(mask, x, m);
        return x;
    }
    // query r's value, from one of its lanes
    __device__ float from(float v, int r) const { return __shfl_sync(mask, v, base + r * (G / 4)); }
};

// Forward over query quads: the online softmax takes the keys of a line in blocks of four (one max
// and one rescale of the four accumulators per block).  Every query's window starts in the first
// block of its first line (consecutive class positions start their windows at most one position
// apart), so the running max is finite after that block.
template <int D>
__global__ void __launch_bounds__(kFmaThreads) fwd_fma_quad_kernel(const FmaParams p) {
    constexpr int G = D / 4;
    const QuadLanes<G> ql;
    const long long unit = (static_cast<long long>(blockIdx.x) * kFmaThreads + threadIdx.x) / G;
    Quad qd;
    if (unit >= p.quads || !qd.init(p, static_cast<uint32_t>(unit))) return;   // the whole group
    const int k2 = p.k[2], rq = ql.rq();
    float4 qv[kQuad], acc[kQuad];
    int ws[kQuad];
#pragma unroll
    for (int r = 0; r < kQuad; ++r) {
        qv[r] = __ldg(chunk_ptr<D>(p.q, qd.row(p, r), ql.c));
        acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        ws[r] = win_start(qd.j(r), qd.lc2, k2);
    }
    const int u0 = ws[0], span = ws[kQuad - 1] - u0 + k2;
    const int lo = (rq == 0 ? ws[0] : rq == 1 ? ws[1] : rq == 2 ? ws[2] : ws[3]) - u0, hi = lo + k2;
    const int f0 = first_nb(p, 0, qd.x0), f1 = first_nb(p, 1, qd.x1);
    const int kstep4 = p.d[2] * p.heads * G;   // float4s between consecutive class positions
    const float sl2 = p.scale * kLog2e;
    float m = -INFINITY, l = 0.f;
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const long long tok = ((qd.b * p.L[0] + f0 + p.d[0] * t0) * p.L[1] + f1 + p.d[1] * t1) * p.L[2] + qd.c2 +
                                  static_cast<long long>(p.d[2]) * u0;
            const float4* kl = chunk_ptr<D>(p.key, tok * p.heads + qd.h, ql.c);
            const float4* vl = chunk_ptr<D>(p.value, tok * p.heads + qd.h, ql.c);
            for (int u = 0; u < span; u += 4) {
                float4 kc[4], vc[4];
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    const int o = min(u + kb, span - 1) * kstep4;   // a key inside the span in every slot
                    kc[kb] = __ldg(kl + o);
                    vc[kb] = __ldg(vl + o);
                }
                float sb[4];
                float bm = -INFINITY;
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    float pd[kQuad];
#pragma unroll
                    for (int r = 0; r < kQuad; ++r) pd[r] = dot4(qv[r], kc[kb]);
                    const float sv = sl2 * ql.reduce(pd);
                    sb[kb] = (u + kb >= lo && u + kb < hi) ? sv : -INFINITY;
                    bm = fmaxf(bm, sb[kb]);
                }
                const float mn = fmaxf(m, bm);
                const float corr = fast_exp2(m - mn);   // 0 on the first block (m = -inf)
                l *= corr;
                m = mn;
#pragma unroll
                for (int r = 0; r < kQuad; ++r) scale4(acc[r], ql.from(corr, r));
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    const float pe = fast_exp2(sb[kb] - mn);   // 0 outside the window
                    l += pe;
#pragma unroll
                    for (int r = 0; r < kQuad; ++r) axpy4(acc[r], ql.from(pe, r), vc[kb]);
                }
            }
        }
#pragma unroll
    for (int r = 0; r < kQuad; ++r) {
        const float lr = ql.from(l, r);
        if (r < qd.nq) {
            scale4(acc[r], 1.f / lr);
            *(reinterpret_cast<float4*>(static_cast<float*>(p.out0) + qd.row(p, r) * D) + ql.c) = acc[r];
        }
    }
    if (ql.owner() && rq < qd.nq) static_cast<float*>(p.out1)[qd.row(p, rq)] = (m + __log2f(l)) * kLn2;
}

// dQ over query quads: per key, the four queries' scores and dO . v, then each query's
// dS = P (dO . v - Delta) with P = exp(scale q . k - LSE), and dQ_r += dS_r k.
template <int D>
__global__ void __launch_bounds__(kFmaThreads) dq_fma_quad_kernel(const FmaParams p) {
    constexpr int G = D / 4;
    const QuadLanes<G> ql;
    const long long unit = (static_cast<long long>(blockIdx.x) * kFmaThreads + threadIdx.x) / G;
    Quad qd;
    if (unit >= p.quads || !qd.init(p, static_cast<uint32_t>(unit))) return;   // the whole group
    const int k2 = p.k[2], rq = ql.rq();
    float4 qv[kQuad], gv[kQuad], acc[kQuad];
    int ws[kQuad];
#pragma unroll
    for (int r = 0; r < kQuad; ++r) {
        const long long row = qd.row(p, r);
        qv[r] = __ldg(chunk_ptr<D>(p.q, row, ql.c));
        gv[r] = __ldg(chunk_ptr<D>(p.dO, row, ql.c));
        acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        ws[r] = win_start(qd.j(r), qd.lc2, k2);
    }
    const long long myrow = qd.row(p, rq);
    const float nl2 = -p.lse[myrow] * kLog2e, dlt = p.delta[myrow];
    const int u0 = ws[0], span = ws[kQuad - 1] - u0 + k2;
    const int lo = (rq == 0 ? ws[0] : rq == 1 ? ws[1] : rq == 2 ? ws[2] : ws[3]) - u0, hi = lo + k2;
    const int f0 = first_nb(p, 0, qd.x0), f1 = first_nb(p, 1, qd.x1);
    const int kstep4 = p.d[2] * p.heads * G;
    const float sl2 = p.scale * kLog2e;
    for (int t0 = 0; t0 < p.k[0]; ++t0)
        for (int t1 = 0; t1 < p.k[1]; ++t1) {
            const long long tok = ((qd.b * p.L[0] + f0 + p.d[0] * t0) * p.L[1] + f1 + p.d[1] * t1) * p.L[2] + qd.c2 +
                                  static_cast<long long>(p.d[2]) * u0;
            const float4* kl = chunk_ptr<D>(p.key, tok * p.heads + qd.h, ql.c);
            const float4* vl = chunk_ptr<D>(p.value, tok * p.heads + qd.h, ql.c);
            for (int u = 0; u < span; u += 2) {
                float4 kc[2], vc[2];
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    const int o = min(u + kb, span - 1) * kstep4;
                    kc[kb] = __ldg(kl + o);
                    vc[kb] = __ldg(vl + o);
                }
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    float ps[kQuad], pp[kQuad];
#pragma unroll
                    for (int r = 0; r < kQuad; ++r) {
                        ps[r] = dot4(qv[r], kc[kb]);
                        pp[r] = dot4(gv[r], vc[kb]);
                    }
                    const float sv = ql.reduce(ps), dp = ql.reduce(pp);
                    const bool in = u + kb >= lo && u + kb < hi;
                    const float ds = in ? fast_exp2(fmaf(sl2, sv, nl2)) * (dp - dlt) : 0.f;
#pragma unroll
                    for (int r = 0; r < kQuad; ++r) axpy4(acc[r], ql.from(ds, r), kc[kb]);
                }
            }
        }
#pragma unroll
    for (int r = 0; r < kQuad; ++r)
        if (r < qd.nq) {
            scale4(acc[r], p.scale);
            *(reinterpret_cast<float4*>(static_cast<float*>(p.out0) + qd.row(p, r) * D) + ql.c) = acc[r];
        }
}

// dK, dV: one row's lanes per key, gathering over the queries whose windows hold the key.  Per axis
// those queries form the class-index interval [i_lo, i_hi]: i_lo = 0 if j < k else j - k/2, and
// i_hi = Lc - 1 if j >= Lc - k else j + k/2 (the border keys are seen by more queries).
// Three blocks per SM (at most 85 registers) with the query loop kept rolled: the compiler's
// unrolled loop held 125 registers, two blocks per SM.  Measured at 1024x1024 9x9 fp32: 12.7 ->
// 12.0 ms (rolled alone, 102 registers and still two blocks: 14.3 ms; the cap alone: 12.7 ms).
template <int D>
__global__ void __launch_bounds__(kFmaThreads, 3) dkdv_fma_kernel(const FmaParams p) {
    const long long rows = static_cast<long long>(p.B) * p.N * p.heads;
    RowLanes<D, false, kCplKV> ln;
    if (!ln.init(rows)) return;
    const RowIdx r = decode_row(p, ln.row);
    int lo[3], hi[3], cl[3];
    for (int a = 0; a < 3; ++a) {
        const int d = p.d[a], j = static_cast<int>(fdiv(static_cast<uint32_t>(r.x[a]), p.fd_d[a])), c = r.x[a] - j * d;
        const int Lc = static_cast<int>(fdiv(static_cast<uint32_t>(p.L[a] - c + d - 1), p.fd_d[a])), ka = p.k[a];
        lo[a] = j < ka ? 0 : j - ka / 2;
        hi[a] = j >= Lc - ka ? Lc - 1 : j + ka / 2;
        cl[a] = c;
    }
    Chunks<D, kCplKV> kc, vc;
    load_chunks<D, kCplKV>(kc, chunk_ptr<D>(p.key, ln.row, ln.c));
    load_chunks<D, kCplKV>(vc, chunk_ptr<D>(p.value, ln.row, ln.c));
    const float sl2 = p.scale * kLog2e;
    Chunks<D, kCplKV> dk, dv;
    zero_chunks<D, kCplKV>(dk);
    zero_chunks<D, kCplKV>(dv);
    const int qstep = p.d[2] * p.heads;
    for (int i0 = lo[0]; i0 <= hi[0]; ++i0)
        for (int i1 = lo[1]; i1 <= hi[1]; ++i1) {
            const long long tok =
                ((r.b * p.L[0] + cl[0] + p.d[0] * i0) * p.L[1] + cl[1] + p.d[1] * i1) * p.L[2] + cl[2];
            const long long qr0 = tok * p.heads + r.h;   // query row of class index 0 along axis 2
            const float4* ql = chunk_ptr<D>(p.q, qr0, ln.c);
            const float4* gl = chunk_ptr<D>(p.dO, qr0, ln.c);
            const float* lsl = p.lse + qr0;
            const float* dll = p.delta + qr0;
#pragma unroll 1
            for (int i2 = lo[2]; i2 <= hi[2]; i2 += kGKV) {
                const int n = min(kGKV, hi[2] - i2 + 1);
                Chunks<D, kCplKV> qc[kGKV], gc[kGKV];
                float ls[kGKV], dl[kGKV];
#pragma unroll
                for (int g = 0; g < kGKV; ++g) {
                    const int ii = i2 + min(g, n - 1);   // a valid query in every slot
                    const long long oq = static_cast<long long>(ii) * qstep;
                    load_chunks<D, kCplKV>(qc[g], ql + oq * (D / 4));
                    load_chunks<D, kCplKV>(gc[g], gl + oq * (D / 4));
                    ls[g] = __ldg(lsl + oq);
                    dl[g] = __ldg(dll + oq);
                }
#pragma unroll
                for (int g = 0; g < kGKV; ++g) {
                    const float s = ln.sum(dot_chunks<D, kCplKV>(kc, qc[g]));
                    const float dp = ln.sum(dot_chunks<D, kCplKV>(vc, gc[g]));
                    const float pe = g < n ? fast_exp2(fmaf(sl2, s, -ls[g] * kLog2e)) : 0.f;
                    axpy_chunks<D, kCplKV>(dv, pe, gc[g]);
                    axpy_chunks<D, kCplKV>(dk, pe * (dp - dl[g]), qc[g]);
                }
            }
        }
    if (ln.store) {
        scale_chunks<D, kCplKV>(dk, p.scale);
        store_chunks<D, kCplKV>(p.out0, ln.row, ln.c, dk);
        store_chunks<D, kCplKV>(p.out1, ln.row, ln.c, dv);
    }
}

// dK, dV over key quads: four consecutive class positions of one head along the innermost axis.
// Along the outer axes the four keys share their inverse intervals; along the innermost axis their
// intervals [lo_r, hi_r] overlap and cover one contiguous run of queries, which the group walks once,
// each loaded query row serving all four keys.  Two queries per step; capped at 128 registers (two
// blocks per SM): measured at 1024x1024 9x9 fp32, 9.9 ms against 12.4 ms uncapped (156 registers,
// one block) and 10.6 ms with one query per step.  The run is k2 + 3 queries long where each key
// needs k2, so the row kernel stays for k2 < 7 (at 16x256x256 / (3, 5, 5) both take 11.6 ms).
template <int D>
__global__ void __launch_bounds__(kFmaThreads, 2) dkdv_fma_quad_kernel(const FmaParams p) {
    constexpr int G = D / 4;
    const QuadLanes<G> ql;
    const long long unit = (static_cast<long long>(blockIdx.x) * kFmaThreads + threadIdx.x) / G;
    Quad qd;
    if (unit >= p.quads || !qd.init(p, static_cast<uint32_t>(unit))) return;   // the whole group
    const int rk = ql.rq();
    float4 kv[kQuad], vv[kQuad], dk[kQuad], dv[kQuad];
#pragma unroll
    for (int r = 0; r < kQuad; ++r) {
        const long long row = qd.row(p, r);
        kv[r] = __ldg(chunk_ptr<D>(p.key, row, ql.c));
        vv[r] = __ldg(chunk_ptr<D>(p.value, row, ql.c));
        dk[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        dv[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // inverse intervals: i_lo = 0 if j < k else j - k/2; i_hi = Lc - 1 if j >= Lc - k else j + k/2
    int lo[2], hi[2], cl[2];
    const int xa[2] = {qd.x0, qd.x1};
    for (int a = 0; a < 2; ++a) {
        const int d = p.d[a], j = static_cast<int>(fdiv(static_cast<uint32_t>(xa[a]), p.fd_d[a])), c = xa[a] - j * d;
        const int Lc = static_cast<int>(fdiv(static_cast<uint32_t>(p.L[a] - c + d - 1), p.fd_d[a])), ka = p.k[a];
        lo[a] = j < ka ? 0 : j - ka / 2;
        hi[a] = j >= Lc - ka ? Lc - 1 : j + ka / 2;
        cl[a] = c;
    }
    const int k2 = p.k[2], lc2 = qd.lc2;
    const int jk = qd.j(rk), j0 = qd.j(0), j3 = qd.j(kQuad - 1);
    const int mylo = jk < k2 ? 0 : jk - k2 / 2, myhi = jk >= lc2 - k2 ? lc2 - 1 : jk + k2 / 2;
    const int ulo = j0 < k2 ? 0 : j0 - k2 / 2, uhi = j3 >= lc2 - k2 ? lc2 - 1 : j3 + k2 / 2;
    const float sl2 = p.scale * kLog2e;
    const int qstep = p.d[2] * p.heads;   // rows between consecutive class positions
    for (int i0 = lo[0]; i0 <= hi[0]; ++i0)
        for (int i1 = lo[1]; i1 <= hi[1]; ++i1) {
            const long long tok = ((qd.b * p.L[0] + cl[0] + p.d[0] * i0) * p.L[1] + cl[1] + p.d[1] * i1) * p.L[2] + qd.c2;
            const long long qr0 = tok * p.heads + qd.h;   // query row of class position 0 along the innermost axis
            const float4* qlp = chunk_ptr<D>(p.q, qr0, ql.c);
            const float4* glp = chunk_ptr<D>(p.dO, qr0, ql.c);
            for (int i2 = ulo; i2 <= uhi; i2 += 2) {
                float4 qc[2], gc[2];
                float ls[2], dl[2];
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const long long oq = static_cast<long long>(min(i2 + g, uhi)) * qstep;   // a query of the run in every slot
                    qc[g] = __ldg(qlp + oq * G);
                    gc[g] = __ldg(glp + oq * G);
                    ls[g] = __ldg(p.lse + qr0 + oq);
                    dl[g] = __ldg(p.delta + qr0 + oq);
                }
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    float ps[kQuad], pp[kQuad];
#pragma unroll
                    for (int r = 0; r < kQuad; ++r) {
                        ps[r] = dot4(kv[r], qc[g]);
                        pp[r] = dot4(vv[r], gc[g]);
                    }
                    const float sv = ql.reduce(ps), dp = ql.reduce(pp);
                    const bool in = i2 + g >= mylo && i2 + g <= myhi;   // (i2 + g <= uhi follows)
                    const float pe = in ? fast_exp2(fmaf(sl2, sv, -ls[g] * kLog2e)) : 0.f;
                    const float ds = pe * (dp - dl[g]);
#pragma unroll
                    for (int r = 0; r < kQuad; ++r) {
                        axpy4(dv[r], ql.from(pe, r), gc[g]);
                        axpy4(dk[r], ql.from(ds, r), qc[g]);
                    }
                }
            }
        }
#pragma unroll
    for (int r = 0; r < kQuad; ++r)
        if (r < qd.nq) {
            const long long row = qd.row(p, r);
            scale4(dk[r], p.scale);
            *(reinterpret_cast<float4*>(static_cast<float*>(p.out0) + row * D) + ql.c) = dk[r];
            *(reinterpret_cast<float4*>(static_cast<float*>(p.out1) + row * D) + ql.c) = dv[r];
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


template <int D, int L, typename F>
int launch_rows(F kernel, const FmaParams& p, cudaStream_t s) {
    const long long total = static_cast<long long>(p.B) * p.N * p.heads;
    if (total == 0) return 0;
    const long long blocks = (total * Chunks<D, L>::CPH + kFmaThreads - 1) / kFmaThreads;
    kernel<<<dim3(static_cast<unsigned>(blocks)), dim3(kFmaThreads), 0, s>>>(p);
    return static_cast<int>(cudaGetLastError());
}

// Query-quad kernels where the quad index fits the 32-bit decode.
template <int D, typename F>
int launch_quads(F kernel, const FmaParams& p, cudaStream_t s) {
    if (p.quads == 0) return 0;
    const long long blocks = (p.quads * (D / 4) + kFmaThreads - 1) / kFmaThreads;
    kernel<<<dim3(static_cast<unsigned>(blocks)), dim3(kFmaThreads), 0, s>>>(p);
    return static_cast<int>(cudaGetLastError());
}

bool quads_ok(const FmaParams& p) { return p.quads < (1LL << 32); }

}  // namespace

int launch_fwd_fma(const FmaParams& p, cudaStream_t s) {
    if (quads_ok(p)) switch (p.D) {
            case 16: return launch_quads<16>(fwd_fma_quad_kernel<16>, p, s);
            case 32: return launch_quads<32>(fwd_fma_quad_kernel<32>, p, s);
            case 64: return launch_quads<64>(fwd_fma_quad_kernel<64>, p, s);
            case 128: return launch_quads<128>(fwd_fma_quad_kernel<128>, p, s);
            default: return static_cast<int>(cudaErrorInvalidValue);
        }
    switch (p.D) {
        case 16: return launch_rows<16, kCplF>(fwd_fma_kernel<16>, p, s);
        case 32: return launch_rows<32, kCplF>(fwd_fma_kernel<32>, p, s);
        case 64: return launch_rows<64, kCplF>(fwd_fma_kernel<64>, p, s);
        case 128: return launch_rows<128, kCplF>(fwd_fma_kernel<128>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dq_fma(const FmaParams& p, cudaStream_t s) {
    if (quads_ok(p)) switch (p.D) {
            case 16: return launch_quads<16>(dq_fma_quad_kernel<16>, p, s);
            case 32: return launch_quads<32>(dq_fma_quad_kernel<32>, p, s);
            case 64: return launch_quads<64>(dq_fma_quad_kernel<64>, p, s);
            case 128: return launch_quads<128>(dq_fma_quad_kernel<128>, p, s);
            default: return static_cast<int>(cudaErrorInvalidValue);
        }
    switch (p.D) {
        case 16: return launch_rows<16, kCplQ>(dq_fma_kernel<16>, p, s);
        case 32: return launch_rows<32, kCplQ>(dq_fma_kernel<32>, p, s);
        case 64: return launch_rows<64, kCplQ>(dq_fma_kernel<64>, p, s);
        case 128: return launch_rows<128, kCplQ>(dq_fma_kernel<128>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dkdv_fma(const FmaParams& p, cudaStream_t s) {
    if (quads_ok(p) && p.k[2] >= 7) switch (p.D) {
            case 16: return launch_quads<16>(dkdv_fma_quad_kernel<16>, p, s);
            case 32: return launch_quads<32>(dkdv_fma_quad_kernel<32>, p, s);
            case 64: return launch_quads<64>(dkdv_fma_quad_kernel<64>, p, s);
            case 128: return launch_quads<128>(dkdv_fma_quad_kernel<128>, p, s);
            default: return static_cast<int>(cudaErrorInvalidValue);
        }
    switch (p.D) {
        case 16: return launch_rows<16, kCplKV>(dkdv_fma_kernel<16>, p, s);
        case 32: return launch_rows<32, kCplKV>(dkdv_fma_kernel<32>, p, s);
        case 64: return launch_rows<64, kCplKV>(dkdv_fma_kernel<64>, p, s);
        case 128: return launch_rows<128, kCplKV>(dkdv_fma_kernel<128>, p, s);
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
