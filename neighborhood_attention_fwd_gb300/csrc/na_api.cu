// na_api.cu -- the C ABI of libna (include/na.h): argument validation, embedding of 1/2/3-D
// problems as 3 axes, the static tile planner of the tensor-core kernels, TMA tensor-map encoding,
// the per-device status word and the launches.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/na.h"
#include "na_device.cuh"
#include "na_internal.h"

namespace na {
uint32_t tc_smem_bytes(int which, const TilePlan& pl, int D);
int tc_tmem_cols(int which, int D);
int tc_max_nc(int which, int D, int sbufs);
}

namespace {

using na::Geom;
using na::TilePlan;

// Per-device status word written by kernels whose bounded waits ran out.
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};
std::mutex g_mu;

// Fixed Delta scratch for na_bwd_noalloc: NA_NOALLOC_MAX_ROWS fp32 values (32 MiB), reserved on every
// device that loads this library for as long as the process lives.  Host code must not use the
// symbol as a device address; the address is looked up per device with cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_delta[NA_NOALLOC_MAX_ROWS];
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_delta on the current device (looked up on the first call per device).
na_status noalloc_scratch(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
        float* p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_delta) != cudaSuccess || !p)
            return NA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return NA_OK;
}

na_status status_ptr(unsigned** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return NA_ERR_CUDA;
        g_status_ptr[dev] = static_cast<unsigned*>(p);
    }
    *out = g_status_ptr[dev];
    return NA_OK;
}

// Wait limit and test hook of the tensor-core kernels' launches (na_debug_wait_hook).
std::atomic<unsigned long long> g_wait_ns{na::dev::kWaitLimitNs};
std::atomic<uint32_t> g_withhold{0};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

na_status get_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return NA_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return NA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return NA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Validate sizes and embed the problem as 3 axes (outermost first).
na_status make_geom(int B, int ndim, const int* spatial, int heads, int D, const int* kernel, const int* dilation,
                    Geom& g) {
    if (ndim < 1 || ndim > 3 || !spatial || !kernel || !dilation || B < 1 || heads < 1 || D < 1)
        return NA_ERR_INVALID_ARG;
    g.B = B;
    g.heads = heads;
    g.D = D;
    const int off = 3 - ndim;
    for (int a = 0; a < 3; ++a) {
        g.L[a] = 1;
        g.k[a] = 1;
        g.d[a] = 1;
    }
    long long tokens = 1;
    for (int a = 0; a < ndim; ++a) {
        const int L = spatial[a], k = kernel[a], d = dilation[a];
        if (L < 1 || k < 1 || (k % 2) == 0 || d < 1 || L / d < k) return NA_ERR_INVALID_ARG;
        g.L[off + a] = L;
        g.k[off + a] = k;
        g.d[off + a] = d;
        tokens *= L;
    }
    const long long elems = tokens * B * heads * static_cast<long long>(D);
    if (tokens > (1LL << 31) || elems > (1LL << 40)) return NA_ERR_UNSUPPORTED;
    return NA_OK;
}

long long tokens_of(const Geom& g) { return static_cast<long long>(g.L[0]) * g.L[1] * g.L[2]; }

// ---------------------------------------------------------------------------------------------
// Tile planner of the tensor-core kernels
// ---------------------------------------------------------------------------------------------

struct PlanKey {
    int which, D, B, heads, L[3], k[3], d[3];
    bool operator<(const PlanKey& o) const {
        return std::tie(which, D, B, heads, L[0], L[1], L[2], k[0], k[1], k[2], d[0], d[1], d[2]) <
               std::tie(o.which, o.D, o.B, o.heads, o.L[0], o.L[1], o.L[2], o.k[0], o.k[1], o.k[2], o.d[0], o.d[1],
                        o.d[2]);
    }
};

std::map<PlanKey, TilePlan> g_plans;

// Chunks a CTA whose tile starts at class index t0 actually processes along one outer axis, as the
// kernels compute it (window or inverse-window range, halo box clamped into the class).
int chunks_along(int which, int t0, int T, int Lc, int k, int H, int G, int nchk) {
    const int last = std::min(t0 + T, Lc) - 1;
    int lo, hi;
    auto ws = [&](int j) { return std::max(0, std::min(j - k / 2, Lc - k)); };
    if (which != 2) {
        lo = ws(t0);
        hi = ws(last) + k - 1;
    } else {
        lo = t0 < k ? 0 : t0 - k / 2;
        hi = last >= Lc - k ? Lc - 1 : last + k / 2;
    }
    const int h0 = std::min(lo, std::max(0, Lc - H));
    return std::min(nchk, ceil_div(hi - h0 + 1, G));
}

// Largest halo extent (class positions) any tile of T positions needs along an axis, over every
// residue class and tile position: the window range [s(first), s(last) + k) for the forward and
// dQ, the inverse range [i_lo(first), i_hi(last)] for dK/dV (a key near a border is seen by up
// to k/2 extra queries on that side, and a tile can touch both borders of a short axis).
int max_halo(int which, int T, int L, int k, int d) {
    int best = 1;
    for (int c = 0; c < d && c < L; ++c) {
        const int Lc = (L - c + d - 1) / d;
        for (int t0 = 0; t0 < Lc; t0 += T) {
            const int last = std::min(t0 + T, Lc) - 1;
            int lo, hi;
            if (which != 2) {
                lo = std::max(0, std::min(t0 - k / 2, Lc - k));
                hi = std::max(0, std::min(last - k / 2, Lc - k)) + k - 1;
            } else {
                lo = t0 < k ? 0 : t0 - k / 2;
                hi = last >= Lc - k ? Lc - 1 : last + k / 2;
            }
            best = std::max(best, hi - lo + 1);
        }
    }
    return best;
}

// Modelled cycles of one interior tile (every row's window unclamped) under a candidate plan.
// The softmax term replays what the kernels do: per chunk each warp (32 consecutive rows) reads
// the run of 16-column groups that holds its rows' windows (forward: one warp per row quarter;
// backward: two warps share a quarter's groups).  Chunks of a tile overlap on the tensor core and
// the copy engine, so the tile costs the largest of softmax, MMA and chunk-copy time.
double tile_cost(int which, const Geom& g, const TilePlan& pl, int n_mma, int per_sm) {
    int ulo[4][3], uhi[4][3];
    for (int w = 0; w < 4; ++w)
        for (int a = 0; a < 3; ++a) {
            ulo[w][a] = 1 << 30;
            uhi[w][a] = -(1 << 30);
        }
    for (int row = 0; row < 128; ++row) {
        const int tq[3] = {row / (pl.T[1] * pl.T[2]), (row / pl.T[2]) % pl.T[1], row % pl.T[2]};
        for (int a = 0; a < 3; ++a) {
            const int len = 2 * (g.k[a] / 2) + 1;  // window or inverse window of an interior row
            ulo[row / 32][a] = std::min(ulo[row / 32][a], tq[a]);
            uhi[row / 32][a] = std::max(uhi[row / 32][a], tq[a] + len);
        }
    }
    int nc[3];
    for (int a = 0; a < 3; ++a) nc[a] = std::min(pl.nchk[a], ceil_div(pl.T[a] + 2 * (g.k[a] / 2), pl.G[a]));
    double soft = 0;
    const int C = nc[0] * nc[1] * nc[2];
    for (int c0 = 0; c0 < nc[0]; ++c0)
        for (int c1 = 0; c1 < nc[1]; ++c1)
            for (int c2 = 0; c2 < nc[2]; ++c2) {
                const int o[3] = {c0 * pl.G[0], c1 * pl.G[1], c2 * pl.G[2]};
                int mx = 0, sum = 0;
                for (int w = 0; w < 4; ++w) {
                    int lo[3], hi[3];
                    bool empty = false;
                    for (int a = 0; a < 3; ++a) {
                        lo[a] = std::max(ulo[w][a] - o[a], 0);
                        hi[a] = std::min(uhi[w][a] - o[a], pl.G[a]);
                        if (lo[a] >= hi[a]) empty = true;
                    }
                    int n = 0;
                    if (!empty) {
                        const int clo = (lo[0] * pl.G[1] + lo[1]) * pl.G[2] + lo[2];
                        const int chi = ((hi[0] - 1) * pl.G[1] + hi[1] - 1) * pl.G[2] + hi[2];
                        n = (chi + 15) / 16 - clo / 16;
                    }
                    mx = std::max(mx, n);
                    sum += n;
                }
                soft += 0.75 * mx + 0.0625 * sum;  // warps wait for the slowest one within a chunk or two
            }
    const double per_group = which == 0 ? 150.0 : 90.0;  // cycles per 16-column group and warp
    const double soft_cyc = soft * per_group + 300.0 * C;
    int nbias = 0;
    for (int a = 0; a < 3; ++a) nbias += pl.H[a] > 1 ? ceil_div(pl.G[a], 16) : 0;
    const double mma_cyc = C * (n_mma * 2.0 * 128 * pl.NC * g.D + nbias * 2.0 * 128 * pl.NC * 16) / 6144.0;
    const double copy_cyc = C * 4.0 * pl.NC * g.D / 40.0;
    double t = std::max(soft_cyc, std::max(mma_cyc, copy_cyc)) + 300.0;
    if (which == 0 && per_sm < 2) t *= 1.7;  // the forward relies on two CTAs per SM to hide latency
    return t;
}

na_status plan_tc(int which, const Geom& g, TilePlan& out) {
    const PlanKey key{which, g.D, g.B, g.heads, {g.L[0], g.L[1], g.L[2]}, {g.k[0], g.k[1], g.k[2]},
                      {g.d[0], g.d[1], g.d[2]}};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            out = it->second;
            return NA_OK;
        }
    }
    const int D = g.D;
    const int tmem_cols = na::tc_tmem_cols(which, D);
    int Lcm[3];
    for (int a = 0; a < 3; ++a) Lcm[a] = ceil_div(g.L[a], g.d[a]);
    const int n_score = which == 0 ? 1 : 2, n_update = which == 2 ? 2 : 1;

    // the cheapest plan whose chunks hold at most ncmax rows
    auto search = [&](int ncmax, TilePlan& bp) {
    bool found = false;
    double best = 0;
    for (int T2 = 8; T2 <= 128; T2 *= 2)
        for (int T1 = 1; T1 * T2 <= 128; T1 *= 2) {
            const int T0 = 128 / (T1 * T2);
            const int T[3] = {T0, T1, T2};
            bool skip = false;
            for (int a = 0; a < 3; ++a) {
                if (T[a] * g.d[a] > 256) skip = true;        // TMA box limit (rows past an axis end are just idle)
            }
            if (skip) continue;
            int Hx[3];
            for (int a = 0; a < 3; ++a) {
                Hx[a] = max_halo(which, T[a], g.L[a], g.k[a], g.d[a]);
                if (Hx[a] >= (1 << 25)) skip = true;  // the kernels' chunk-count reciprocal is exact below 2^26
            }
            if (skip) continue;
            double tiles = 1;
            for (int a = 0; a < 3; ++a) tiles *= ceil_div(Lcm[a], T[a]);
            const int gmax0 = Hx[0] > 1 ? std::min(Hx[0], 32) : 1, gmax1 = Hx[1] > 1 ? std::min(Hx[1], 32) : 1;
            for (int G2 = 1; G2 <= std::min(Hx[2], 32); ++G2) {
                if (G2 * g.d[2] > 256) continue;
                for (int G1 = 1; G1 <= gmax1; ++G1)
                    for (int G0 = 1; G0 <= gmax0; ++G0) {
                        const int NC = G0 * G1 * G2;
                        if (NC > ncmax || NC % 16 != 0) continue;
                        if (G0 * g.d[0] > 256 || G1 * g.d[1] > 256) continue;
                        TilePlan cand{};
                        const int G[3] = {G0, G1, G2};
                        for (int a = 0; a < 3; ++a) {
                            cand.T[a] = T[a];
                            cand.ntile[a] = ceil_div(Lcm[a], T[a]);
                            cand.H[a] = Hx[a];
                            cand.G[a] = G[a];
                            cand.nchk[a] = ceil_div(Hx[a], G[a]);
                        }
                        cand.NC = NC;
                        const int need = static_cast<int>(na::tc_smem_bytes(which, cand, D));
                        if (need > 227 * 1024) continue;
                        const int per_sm = std::max(1, std::min(512 / tmem_cols, (228 * 1024) / (need + 1024)));
                        const double cost =
                            tile_cost(which, g, cand, n_score + n_update, per_sm) * tiles;
                        if (!found || cost < best) {
                            found = true;
                            best = cost;
                            bp = cand;
                        }
                    }
            }
        }
    return found;
    };
    TilePlan bp{};
    if (!search(na::tc_max_nc(which, D, 2), bp)) return NA_ERR_UNSUPPORTED;
    bp.sbufs = 2;
    // A forward whose tiles walk ten or more chunks is bound by each score buffer's chain (the P V
    // product of a chunk, then the score product of the chunk two later into the same buffer), not by
    // the per-chunk costs: it takes three 64-column buffers instead (measured at 8x128x128 / (5, 7, 7),
    // 10 chunks of 96 columns: 0.97 -> 0.80 ms; at 4-7 chunks per tile three buffers were 27-49% slower).
    if (which == 0 && D <= 32 && bp.nchk[0] * bp.nchk[1] * bp.nchk[2] >= 10) {
        TilePlan b3{};
        if (search(na::tc_max_nc(which, D, 3), b3)) {
            bp = b3;
            bp.sbufs = 3;
        }
    }
    bp.tmem_cols = tmem_cols;
    // Shared memory: the layout, padded so that no more than 512 / tmem_cols CTAs fit on an SM
    // (their TMEM allocations then never wait on each other), and checked so that that many do fit.
    const int need = static_cast<int>(na::tc_smem_bytes(which, bp, D));
    int per_sm = 512 / tmem_cols;
    while (per_sm > 1 && per_sm * (need + 1024) > 228 * 1024) --per_sm;
    int smem = need;
    const int floor_bytes = (228 * 1024) / (per_sm + 1) - 1024 + 1;
    if (smem < floor_bytes) smem = floor_bytes;
    if (smem > 227 * 1024) return NA_ERR_UNSUPPORTED;
    bp.per_sm = per_sm;
    bp.smem_bytes = smem;
    long long ctas = static_cast<long long>(g.B) * g.heads;
    for (int a = 0; a < 3; ++a) ctas *= static_cast<long long>(bp.ntile[a]) * g.d[a];
    if (ctas > 0x7fffffffLL) return NA_ERR_UNSUPPORTED;
    bp.ctas = ctas;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_plans[key] = bp;
    }
    out = bp;
    return NA_OK;
}

// Tensor map over a [B, L0, L1, L2, heads, D] bf16 tensor whose box is `e` class positions per axis
// (element stride = dilation) and D channels of one head; at D = 128 the box is 64 channels (one
// 128-byte swizzle row) and the kernels load the two halves of a head with two copies.
na_status encode_map(CUtensorMap* m, const void* base, const Geom& g, const int e[3], bool f16) {
    const cuuint64_t es = 2;
    const cuuint64_t hd = static_cast<cuuint64_t>(g.heads) * g.D;
    cuuint64_t dims[5] = {hd, static_cast<cuuint64_t>(g.L[2]), static_cast<cuuint64_t>(g.L[1]),
                          static_cast<cuuint64_t>(g.L[0]), static_cast<cuuint64_t>(g.B)};
    cuuint64_t strides[4] = {hd * es, hd * es * g.L[2], hd * es * g.L[2] * g.L[1], hd * es * g.L[2] * g.L[1] * g.L[0]};
    const int dbox = g.D > 64 ? 64 : g.D;
    cuuint32_t box[5] = {static_cast<cuuint32_t>(dbox), static_cast<cuuint32_t>(e[2] * g.d[2]),
                         static_cast<cuuint32_t>(e[1] * g.d[1]), static_cast<cuuint32_t>(e[0] * g.d[0]), 1};
    cuuint32_t estr[5] = {1, static_cast<cuuint32_t>(g.d[2]), static_cast<cuuint32_t>(g.d[1]),
                          static_cast<cuuint32_t>(g.d[0]), 1};
    for (int i = 0; i < 5; ++i)
        if (box[i] < 1 || box[i] > 256 || estr[i] > 8) return NA_ERR_UNSUPPORTED;
    const int rowb = dbox * 2;
    const CUtensorMapSwizzle sw = rowb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                              : (rowb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    const CUresult r = g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NA_OK : NA_ERR_CUDA;
}

na_status tc_common(int which, const Geom& g, float scale, na::TcParams& p) {
    if (g.D != 16 && g.D != 32 && g.D != 64 && g.D != 128) return NA_ERR_UNSUPPORTED;
    for (int a = 0; a < 3; ++a)
        if (g.d[a] > 8) return NA_ERR_UNSUPPORTED;
    std::memset(&p, 0, sizeof p);
    na_status st = plan_tc(which, g, p.plan);
    if (st != NA_OK) return st;
    if ((st = get_encoder()) != NA_OK) return st;
    for (int a = 0; a < 3; ++a) {
        p.L[a] = g.L[a];
        p.k[a] = g.k[a];
        p.d[a] = g.d[a];
    }
    p.B = g.B;
    p.heads = g.heads;
    p.D = g.D;
    p.scale = scale;
    // a negative scale is folded into the S product (negated A operand); a zero scale becomes a
    // tiny positive one (uniform weights up to ~1e-28 relative) so that masked scores stay -inf
    p.neg = scale < 0.f ? 1u : 0u;
    p.scale_log2 = std::max(std::fabs(scale), 1e-30f) * 1.44269504088896340736f;
    p.wait_ns = g_wait_ns.load();
    p.withhold = g_withhold.load();
    for (int a = 0; a < 3; ++a) {
        for (int c = 0; c < 8; ++c) p.Lc_tab[a][c] = c < g.d[a] ? (g.L[a] - c + g.d[a] - 1) / g.d[a] : 0;
        p.rcpG[a] = p.plan.G[a] == 1 ? 0u : static_cast<uint32_t>((1ull << 32) / static_cast<uint64_t>(p.plan.G[a]) + 1u);
    }
    const int rad[8] = {g.heads, p.plan.ntile[2], p.plan.ntile[1], p.plan.ntile[0], g.d[2], g.d[1], g.d[0], g.B};
    for (int i = 0; i < 8; ++i) p.rad[i] = static_cast<uint32_t>(rad[i]);
    return status_ptr(&p.err);
}

na_status cuda_status(int e) { return e == 0 ? NA_OK : NA_ERR_CUDA; }

na_status check_ptrs(std::initializer_list<const void*> ps) {
    for (const void* p : ps)
        if (!p) return NA_ERR_INVALID_ARG;
    for (const void* p : ps)
        if (!aligned16(p)) return NA_ERR_ALIGNMENT;
    return NA_OK;
}

na::FmaParams fma_params(const Geom& g, float scale) {
    na::FmaParams p{};
    for (int a = 0; a < 3; ++a) {
        p.L[a] = g.L[a];
        p.k[a] = g.k[a];
        p.d[a] = g.d[a];
    }
    p.B = g.B;
    p.heads = g.heads;
    p.D = g.D;
    p.N = tokens_of(g);
    p.scale = scale;
    p.rows32 = static_cast<long long>(g.B) * p.N * g.heads < (1LL << 32) ? 1u : 0u;
    p.fd_heads = na::make_fastdiv(static_cast<uint32_t>(g.heads));
    p.fd_N = na::make_fastdiv(static_cast<uint32_t>(p.N));
    for (int a = 0; a < 3; ++a) {
        p.fd_L[a] = na::make_fastdiv(static_cast<uint32_t>(g.L[a]));
        p.fd_d[a] = na::make_fastdiv(static_cast<uint32_t>(g.d[a]));
    }
    const int lc2 = (g.L[2] + g.d[2] - 1) / g.d[2];   // class 0 is the longest
    p.qc2 = (lc2 + 3) / 4;
    p.fd_qc2 = na::make_fastdiv(static_cast<uint32_t>(p.qc2));
    p.quads = static_cast<long long>(g.B) * g.L[0] * g.L[1] * g.d[2] * p.qc2 * g.heads;
    return p;
}

na_status check_dtype(na_dtype dt, const Geom& g) {
    if (dt == NA_FP32) return (g.D == 16 || g.D == 32 || g.D == 64 || g.D == 128) ? NA_OK : NA_ERR_UNSUPPORTED;
    if (dt == NA_BF16 || dt == NA_FP16) return NA_OK;
    return NA_ERR_INVALID_ARG;
}


// Validation and parameters shared by the unfused operations.
int elem_of(na_dtype dt) { return dt == NA_BF16 ? 0 : (dt == NA_FP16 ? 2 : 1); }

na_status unfused_params(int B, int ndim, const int* spatial, int heads, int D, const int* kernel,
                         const int* dilation, float scale, na_dtype dtype, bool need_d, na::UnfParams& p) {
    int ones[3] = {1, 1, 1};
    Geom g;
    na_status st = make_geom(B, ndim, spatial, heads, need_d ? D : 16, kernel, dilation ? dilation : ones, g);
    if (st != NA_OK) return st;
    if (!std::isfinite(scale)) return NA_ERR_INVALID_ARG;
    if (dtype != NA_BF16 && dtype != NA_FP16 && dtype != NA_FP32) return NA_ERR_INVALID_ARG;
    if (need_d && D != 16 && D != 32 && D != 64 && D != 128) return NA_ERR_UNSUPPORTED;
    std::memset(&p, 0, sizeof p);
    p.K = 1;
    for (int a = 0; a < 3; ++a) {
        p.L[a] = g.L[a];
        p.k[a] = g.k[a];
        p.d[a] = g.d[a];
        p.K *= g.k[a];
    }
    p.heads = heads;
    p.D = D;
    p.rows = tokens_of(g) * B * heads;
    p.scale = scale;
    for (int c = 0; c < g.d[2]; ++c) p.strips2 += ((g.L[2] - c + g.d[2] - 1) / g.d[2] + 15) / 16;
    p.units = static_cast<long long>(B) * g.L[0] * g.L[1] * p.strips2 * heads;
    p.small = p.rows < (1LL << 32) && p.units < (1LL << 32) ? 1u : 0u;
    p.fd_heads = na::make_fastdiv(static_cast<uint32_t>(heads));
    p.fd_strips2 = na::make_fastdiv(static_cast<uint32_t>(p.strips2));
    for (int a = 0; a < 3; ++a) {
        p.fd_L[a] = na::make_fastdiv(static_cast<uint32_t>(g.L[a]));
        p.fd_d[a] = na::make_fastdiv(static_cast<uint32_t>(g.d[a]));
    }
    p.fd_K = na::make_fastdiv(static_cast<uint32_t>(p.K));
    p.fd_k2 = na::make_fastdiv(static_cast<uint32_t>(g.k[2]));
    p.fd_k12 = na::make_fastdiv(static_cast<uint32_t>(g.k[1] * g.k[2]));
    return NA_OK;
}

// Tensor maps of the TMA-fed weighted sums: with `inverse`, the inverse-window gathers (na_qk_bwd's dK,
// na_av_bwd's dV; src is q or dO), else the window sums (na_av's O, na_qk_bwd's dQ; src is v or k); w
// the weights.  Left off (p.tma = 0, the kernels without TMA run) where TMA cannot describe the
// tensors: D > 64 (a source row wider than the 128-byte swizzle), dilation > 8 (the element stride),
// a weights row of heads * K elements that is not a multiple of 16 bytes, misaligned pointers, or
// spans longer than 64 positions.
void unfused_tma_maps(na::UnfParams& p, int B, const void* src, const void* w, na_dtype dtype, bool inverse) {
    p.tma = 0;
    // w null: only the source map (the logits kernels write the weights instead of reading them)
    if (dtype == NA_FP32 || p.D > 64 || (w && (static_cast<long long>(p.heads) * p.K) % 8 != 0)) return;
    for (int a = 0; a < 3; ++a)
        if (p.d[a] > 8) return;
    // source rows copied per line: the largest span over every 16-position strip of every class along the
    // innermost axis: of the keys in its queries' windows (at most 15 + k2), or of the queries whose
    // windows hold its keys (clamped windows at either border widen that up to about 2 k2 + 14)
    const int k2 = p.k[2], r2 = k2 / 2;
    int span = 1;
    for (int c = 0; c < p.d[2]; ++c) {
        const int Lc = (p.L[2] - c + p.d[2] - 1) / p.d[2];
        for (int j0 = 0; j0 < Lc; j0 += 16) {
            const int jl = std::min(j0 + 15, Lc - 1);
            int lo, hi;
            if (inverse) {
                lo = j0 < k2 ? 0 : j0 - r2;
                hi = jl >= Lc - k2 ? Lc - 1 : jl + r2;
            } else {
                lo = std::max(0, std::min(j0 - r2, Lc - k2));
                hi = std::max(0, std::min(jl - r2, Lc - k2)) + k2 - 1;
            }
            span = std::max(span, hi - lo + 1);
        }
    }
    const int srows = (span + 15) / 16 * 16, wrows = inverse ? srows : 16;
    if (srows > 64 || srows * p.d[2] > 256) return;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(w)) & 15u) return;
    const int wb = (k2 + 7 + 7) / 8 * 8;  // >= k2 + 7 offsets from a 16-byte aligned start
    if (wb > 256 || get_encoder() != NA_OK || status_ptr(&p.err) != NA_OK) return;
    const CUtensorMapDataType ty = dtype == NA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t es = 2;
    auto enc = [&](CUtensorMap* m, const void* base, cuuint64_t row, cuuint32_t inner, int rows, CUtensorMapSwizzle sw) {
        cuuint64_t dims[5] = {row, static_cast<cuuint64_t>(p.L[2]), static_cast<cuuint64_t>(p.L[1]),
                              static_cast<cuuint64_t>(p.L[0]), static_cast<cuuint64_t>(B)};
        cuuint64_t strides[4] = {row * es, row * es * p.L[2], row * es * p.L[2] * p.L[1],
                                 row * es * p.L[2] * p.L[1] * p.L[0]};
        cuuint32_t box[5] = {inner, static_cast<cuuint32_t>(rows * p.d[2]), 1, 1, 1};
        cuuint32_t estr[5] = {1, static_cast<cuuint32_t>(p.d[2]), 1, 1, 1};
        return g_encode(m, ty, 5, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    const CUtensorMapSwizzle sw = p.D == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                            : (p.D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    if (!enc(&p.tm_src, src, static_cast<cuuint64_t>(p.heads) * p.D, static_cast<cuuint32_t>(p.D), srows, sw)) return;
    if (w && !enc(&p.tm_w, w, static_cast<cuuint64_t>(p.heads) * p.K, static_cast<cuuint32_t>(wb), wrows,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
        return;
    p.wb = static_cast<uint32_t>(wb);
    p.srows = static_cast<uint32_t>(srows);
    p.wrows = static_cast<uint32_t>(wrows);
    p.wait_ns = g_wait_ns.load();
    p.tma = 1;
}
}  // namespace

extern "C" {

na_status na_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int ndim, const int* spatial,
                 int heads, int D, const int* kernel, const int* dilation, float scale, na_dtype dtype, void* stream) {
    Geom g;
    na_status st = make_geom(B, ndim, spatial, heads, D, kernel, dilation, g);
    if (st != NA_OK) return st;
    if (!std::isfinite(scale)) return NA_ERR_INVALID_ARG;
    if ((st = check_dtype(dtype, g)) != NA_OK) return st;
    if ((st = check_ptrs({q, k, v, o, lse})) != NA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == NA_FP32) {
        na::FmaParams p = fma_params(g, scale);
        p.q = q;
        p.key = k;
        p.value = v;
        p.out0 = o;
        p.out1 = lse;
        return cuda_status(na::launch_fwd_fma(p, s));
    }
    na::TcParams p;
    if ((st = tc_common(0, g, scale, p)) != NA_OK) return st;
    p.f16 = dtype == NA_FP16 ? 1u : 0u;
    const TilePlan& pl = p.plan;
    const int chunk[3] = {pl.G[0], pl.G[1], pl.G[2]};
    if ((st = encode_map(&p.tm[0], q, g, pl.T, p.f16 != 0)) != NA_OK) return st;
    if ((st = encode_map(&p.tm[1], k, g, chunk, p.f16 != 0)) != NA_OK) return st;
    if ((st = encode_map(&p.tm[2], v, g, chunk, p.f16 != 0)) != NA_OK) return st;
    p.out0 = static_cast<uint16_t*>(o);
    p.lse_out = lse;
    return cuda_status(na::launch_fwd_tc(p, s));
}

size_t na_bwd_workspace_size(int B, int ndim, const int* spatial, int heads) {
    if (ndim < 1 || ndim > 3 || !spatial || B < 1 || heads < 1) return 0;
    long long n = static_cast<long long>(B) * heads;
    for (int a = 0; a < ndim; ++a) {
        if (spatial[a] < 1) return 0;
        n *= spatial[a];
    }
    return static_cast<size_t>((n * 4 + 255) / 256 * 256);
}

na_status na_bwd_delta(const void* o, const void* dO, float* delta, int B, int ndim, const int* spatial, int heads,
                       int D, na_dtype dtype, void* stream) {
    const int ones[3] = {1, 1, 1};
    Geom g;
    na_status st = make_geom(B, ndim, spatial, heads, D, ones, ones, g);
    if (st != NA_OK) return st;
    if ((st = check_dtype(dtype, g)) != NA_OK) return st;
    if (dtype != NA_FP32 && (D % 8 != 0 || D > 256)) return NA_ERR_UNSUPPORTED;
    if ((st = check_ptrs({o, dO, delta})) != NA_OK) return st;
    na::FmaParams p = fma_params(g, 1.f);
    p.o = o;
    p.dO = dO;
    p.out0 = delta;
    return cuda_status(na::launch_delta(p, dtype == NA_BF16 ? 0 : (dtype == NA_FP16 ? 2 : 1), static_cast<cudaStream_t>(stream)));
}

na_status na_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse, const float* delta,
                    void* dQ, int B, int ndim, const int* spatial, int heads, int D, const int* kernel,
                    const int* dilation, float scale, na_dtype dtype, void* stream) {
    Geom g;
    na_status st = make_geom(B, ndim, spatial, heads, D, kernel, dilation, g);
    if (st != NA_OK) return st;
    if (!std::isfinite(scale)) return NA_ERR_INVALID_ARG;
    if ((st = check_dtype(dtype, g)) != NA_OK) return st;
    if ((st = check_ptrs({q, k, v, dO, lse, delta, dQ})) != NA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == NA_FP32) {
        na::FmaParams p = fma_params(g, scale);
        p.q = q;
        p.key = k;
        p.value = v;
        p.dO = dO;
        p.lse = lse;
        p.delta = delta;
        p.out0 = dQ;
        return cuda_status(na::launch_dq_fma(p, s));
    }
    na::TcParams p;
    if ((st = tc_common(1, g, scale, p)) != NA_OK) return st;
    p.f16 = dtype == NA_FP16 ? 1u : 0u;
    const TilePlan& pl = p.plan;
    const int chunk[3] = {pl.G[0], pl.G[1], pl.G[2]};
    if ((st = encode_map(&p.tm[0], q, g, pl.T, p.f16 != 0)) != NA_OK) return st;
    if ((st = encode_map(&p.tm[1], dO, g, pl.T, p.f16 != 0)) != NA_OK) return st;
    if ((st = encode_map(&p.tm[2], k, g, chunk, p.f16 != 0)) != NA_OK) return st;
    if ((st = encode_map(&p.tm[3], v, g, chunk, p.f16 != 0)) != NA_OK) return st;
    p.out0 = static_cast<uint16_t*>(dQ);
    p.lse = lse;
    p.delta = delta;
    return cuda_status(na::launch_dq_tc(p, s));
}

na_status na_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                      const float* delta, void* dK, void* dV, int B, int ndim, const int* spatial, int heads, int D,
                      const int* kernel, const int* dilation, float scale, na_dtype dtype, void* stream) {
    Geom g;
    na_status st = make_geom(B, ndim, spatial, heads, D, kernel, dilation, g);
    if (st != NA_OK) return st;
    if (!std::isfinite(scale)) return NA_ERR_INVALID_ARG;
    if ((st = check_dtype(dtype, g)) != NA_OK) return st;
    if ((st = check_ptrs({q, k, v, dO, lse, delta, dK, dV})) != NA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == NA_FP32) {
        na::FmaParams p = fma_params(g, scale);
        p.q = q;
        p.key = k;
        p.value = v;
        p.dO = dO;
        p.lse = lse;
        p.delta = delta;
        p.out0 = dK;
        p.out1 = dV;
        return cuda_status(na::launch_dkdv_fma(p, s));
    }
    na::TcParams p;
    if ((st = tc_common(2, g, scale, p)) != NA_OK) return st;
    p.f16 = dtype == NA_FP16 ? 1u : 0u;
    const TilePlan& pl = p.plan;
    const int chunk[3] = {pl.G[0], pl.G[1], pl.G[2]};
    if ((st = encode_map(&p.tm[0], k, g, pl.T, p.f16 != 0)) != NA_OK) return st;
    if ((st = encode_map(&p.tm[1], v, g, pl.T, p.f16 != 0)) != NA_OK) return st;
    if ((st = encode_map(&p.tm[2], q, g, chunk, p.f16 != 0)) != NA_OK) return st;
    if ((st = encode_map(&p.tm[3], dO, g, chunk, p.f16 != 0)) != NA_OK) return st;
    p.out0 = static_cast<uint16_t*>(dK);
    p.out1 = static_cast<uint16_t*>(dV);
    p.lse = lse;
    p.delta = delta;
    return cuda_status(na::launch_dkdv_tc(p, s));
}

na_status na_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dQ,
                 void* dK, void* dV, int B, int ndim, const int* spatial, int heads, int D, const int* kernel,
                 const int* dilation, float scale, na_dtype dtype, void* workspace, size_t workspace_bytes,
                 void* stream) {
    Geom g;
    na_status st = make_geom(B, ndim, spatial, heads, D, kernel, dilation, g);
    if (st != NA_OK) return st;
    if (!std::isfinite(scale)) return NA_ERR_INVALID_ARG;
    if ((st = check_dtype(dtype, g)) != NA_OK) return st;
    if ((st = check_ptrs({q, k, v, o, dO, lse, dQ, dK, dV})) != NA_OK) return st;
    if (dtype != NA_FP32) {  // reject unsupported problems before anything is enqueued
        na::TcParams probe;
        if ((st = tc_common(1, g, scale, probe)) != NA_OK) return st;
        if ((st = tc_common(2, g, scale, probe)) != NA_OK) return st;
    }
    const size_t need = na_bwd_workspace_size(B, ndim, spatial, heads);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* ws = workspace;
    bool owned = false;
    if (ws) {
        if (workspace_bytes < need) return NA_ERR_WORKSPACE;
        if (!aligned16(ws)) return NA_ERR_ALIGNMENT;
    } else {
        if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return NA_ERR_WORKSPACE;
        owned = true;
    }
    float* delta = static_cast<float*>(ws);
    st = na_bwd_delta(o, dO, delta, B, ndim, spatial, heads, D, dtype, stream);
    if (st == NA_OK)
        st = na_bwd_dq(q, k, v, dO, lse, delta, dQ, B, ndim, spatial, heads, D, kernel, dilation, scale, dtype, stream);
    if (st == NA_OK)
        st = na_bwd_dkdv(q, k, v, dO, lse, delta, dK, dV, B, ndim, spatial, heads, D, kernel, dilation, scale, dtype,
                         stream);
    if (owned && cudaFreeAsync(ws, s) != cudaSuccess && st == NA_OK) st = NA_ERR_CUDA;
    return st;
}

na_status na_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dQ, void* dK, void* dV, int B, int ndim, const int* spatial,
                         int heads, int D, const int* kernel, const int* dilation, float scale, na_dtype dtype,
                         void* stream) {
    Geom g;
    na_status st = make_geom(B, ndim, spatial, heads, D, kernel, dilation, g);
    if (st != NA_OK) return st;
    // Size limit first, before any CUDA call: the Delta rows must fit the static scratch.
    const long long rows = tokens_of(g) * g.B * g.heads;
    if (rows > static_cast<long long>(NA_NOALLOC_MAX_ROWS)) return NA_ERR_WORKSPACE;
    if (!std::isfinite(scale)) return NA_ERR_INVALID_ARG;
    if ((st = check_dtype(dtype, g)) != NA_OK) return st;
    if ((st = check_ptrs({q, k, v, o, dO, lse, dQ, dK, dV})) != NA_OK) return st;
    if (dtype != NA_FP32) {
        na::TcParams probe;
        if ((st = tc_common(1, g, scale, probe)) != NA_OK) return st;
        if ((st = tc_common(2, g, scale, probe)) != NA_OK) return st;
    }
    float* delta = nullptr;
    if ((st = noalloc_scratch(&delta)) != NA_OK) return st;
    // Every row of delta is rewritten by the Delta step before dQ and dK/dV read it, so the
    // previous call's contents never leak into this one and nothing has to be cleared.
    st = na_bwd_delta(o, dO, delta, B, ndim, spatial, heads, D, dtype, stream);
    if (st == NA_OK)
        st = na_bwd_dq(q, k, v, dO, lse, delta, dQ, B, ndim, spatial, heads, D, kernel, dilation, scale, dtype, stream);
    if (st == NA_OK)
        st = na_bwd_dkdv(q, k, v, dO, lse, delta, dK, dV, B, ndim, spatial, heads, D, kernel, dilation, scale, dtype,
                         stream);
    return st;
}

na_status na_device_status(void* stream, uint32_t* raw) {
    unsigned* ptr = nullptr;
    na_status st = status_ptr(&ptr);
    if (st != NA_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return NA_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, ptr, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return NA_ERR_CUDA;
    if (word != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(ptr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return NA_ERR_CUDA;
    }
    if (raw) *raw = word;
    return word ? NA_ERR_TIMEOUT : NA_OK;
}

na_status na_debug_wait_hook(unsigned long long limit_ns, int withhold) {
    if (withhold != 0 && withhold != 1) return NA_ERR_INVALID_ARG;
    if (limit_ns != 0 && (limit_ns < 100000ull || limit_ns > 10000000000ull)) return NA_ERR_INVALID_ARG;
    g_wait_ns.store(limit_ns == 0 ? na::dev::kWaitLimitNs : limit_ns);
    g_withhold.store(static_cast<uint32_t>(withhold));
    return NA_OK;
}

const char* na_strerror(na_status s) {
    switch (s) {
        case NA_OK: return "success";
        case NA_ERR_INVALID_ARG: return "invalid argument";
        case NA_ERR_UNSUPPORTED: return "unsupported problem for this dtype";
        case NA_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
        case NA_ERR_CUDA: return "CUDA error";
        case NA_ERR_TIMEOUT: return "a device-side wait timed out";
        case NA_ERR_WORKSPACE: return "workspace too small or not allocatable";
        default: return "unknown status";
    }
}

na_status na_plan_info(int which, int B, int ndim, const int* spatial, int heads, int D, const int* kernel,
                       const int* dilation, int64_t* out) {
    if (!out || which < 0 || which > 2) return NA_ERR_INVALID_ARG;
    Geom g;
    na_status st = make_geom(B, ndim, spatial, heads, D, kernel, dilation, g);
    if (st != NA_OK) return st;
    if (D != 16 && D != 32 && D != 64 && D != 128) return NA_ERR_UNSUPPORTED;
    TilePlan pl;
    if ((st = plan_tc(which, g, pl)) != NA_OK) return st;
    // chunks summed over every CTA (depends on the tile position along the two outer axes and class)
    long long total_chunks = 0;
    for (int c0 = 0; c0 < g.d[0]; ++c0)
        for (int c1 = 0; c1 < g.d[1]; ++c1) {
            const int Lc0 = (g.L[0] - c0 + g.d[0] - 1) / g.d[0], Lc1 = (g.L[1] - c1 + g.d[1] - 1) / g.d[1];
            long long n0 = 0, n1 = 0;
            for (int t = 0; t * pl.T[0] < Lc0; ++t)
                n0 += chunks_along(which, t * pl.T[0], pl.T[0], Lc0, g.k[0], pl.H[0], pl.G[0], pl.nchk[0]);
            for (int t = 0; t * pl.T[1] < Lc1; ++t)
                n1 += chunks_along(which, t * pl.T[1], pl.T[1], Lc1, g.k[1], pl.H[1], pl.G[1], pl.nchk[1]);
            long long n2 = 0;  // chunks along axis 2 summed over its tiles and classes
            for (int c2 = 0; c2 < g.d[2]; ++c2) {
                const int Lc2 = (g.L[2] - c2 + g.d[2] - 1) / g.d[2];
                for (int t = 0; t * pl.T[2] < Lc2; ++t)
                    n2 += chunks_along(which, t * pl.T[2], pl.T[2], Lc2, g.k[2], pl.H[2], pl.G[2], pl.nchk[2]);
            }
            total_chunks += n0 * n1 * n2;
        }
    total_chunks *= static_cast<long long>(g.B) * g.heads;
    const int n_mma = which == 0 ? 2 : (which == 1 ? 3 : 4);
    out[0] = pl.T[0];
    out[1] = pl.T[1];
    out[2] = pl.T[2];
    out[3] = pl.H[0];
    out[4] = pl.H[1];
    out[5] = pl.H[2];
    out[6] = pl.G[0];
    out[7] = pl.G[1];
    out[8] = pl.G[2];
    out[9] = pl.NC;
    out[10] = static_cast<int64_t>(pl.nchk[0]) * pl.nchk[1] * pl.nchk[2];
    out[11] = pl.ctas;
    out[12] = total_chunks * n_mma * 2LL * 128 * pl.NC * D;  // MMA FLOPs issued by all CTAs
    out[13] = pl.tmem_cols;
    out[14] = pl.smem_bytes;
    out[15] = total_chunks;
    return NA_OK;
}

// ---------------------------------------------------------------------------------------------
// Unfused operations
// ---------------------------------------------------------------------------------------------

na_status na_qk(const void* q, const void* k, const float* rpb, void* attn, int B, int ndim, const int* spatial,
                int heads, int D, const int* kernel, const int* dilation, float scale, na_dtype dtype, void* stream) {
    na::UnfParams p;
    na_status st = unfused_params(B, ndim, spatial, heads, D, kernel, dilation, scale, dtype, true, p);
    if (st != NA_OK) return st;
    if ((st = check_ptrs({q, k, attn})) != NA_OK) return st;
    if (rpb && (reinterpret_cast<uintptr_t>(rpb) & 3u)) return NA_ERR_ALIGNMENT;
    p.a = q;
    p.b = k;
    p.out0 = attn;
    p.rpb = rpb;
    unfused_tma_maps(p, B, k, nullptr, dtype, false);
    return cuda_status(na::launch_unfused_qk(p, elem_of(dtype), static_cast<cudaStream_t>(stream)));
}

na_status na_av(const void* attn, const void* v, void* o, int B, int ndim, const int* spatial, int heads, int D,
                const int* kernel, const int* dilation, na_dtype dtype, void* stream) {
    na::UnfParams p;
    na_status st = unfused_params(B, ndim, spatial, heads, D, kernel, dilation, 1.f, dtype, true, p);
    if (st != NA_OK) return st;
    if ((st = check_ptrs({attn, v, o})) != NA_OK) return st;
    p.a = attn;
    p.b = v;
    p.out0 = o;
    unfused_tma_maps(p, B, v, attn, dtype, false);
    return cuda_status(na::launch_unfused_av(p, elem_of(dtype), static_cast<cudaStream_t>(stream)));
}

na_status na_softmax(const void* x, void* y, int B, int ndim, const int* spatial, int heads, const int* kernel,
                     na_dtype dtype, void* stream) {
    na::UnfParams p;
    na_status st = unfused_params(B, ndim, spatial, heads, 0, kernel, nullptr, 1.f, dtype, false, p);
    if (st != NA_OK) return st;
    if ((st = check_ptrs({x, y})) != NA_OK) return st;
    p.a = x;
    p.out0 = y;
    return cuda_status(na::launch_unfused_softmax(p, elem_of(dtype), false, static_cast<cudaStream_t>(stream)));
}

na_status na_softmax_bwd(const void* y, const void* dy, void* dx, int B, int ndim, const int* spatial, int heads,
                         const int* kernel, na_dtype dtype, void* stream) {
    na::UnfParams p;
    na_status st = unfused_params(B, ndim, spatial, heads, 0, kernel, nullptr, 1.f, dtype, false, p);
    if (st != NA_OK) return st;
    if ((st = check_ptrs({y, dy, dx})) != NA_OK) return st;
    p.a = y;
    p.b = dy;
    p.out0 = dx;
    return cuda_status(na::launch_unfused_softmax(p, elem_of(dtype), true, static_cast<cudaStream_t>(stream)));
}

na_status na_qk_bwd(const void* dattn, const void* q, const void* k, void* dq, void* dk, int B, int ndim,
                    const int* spatial, int heads, int D, const int* kernel, const int* dilation, float scale,
                    na_dtype dtype, void* stream) {
    na::UnfParams p;
    na_status st = unfused_params(B, ndim, spatial, heads, D, kernel, dilation, scale, dtype, true, p);
    if (st != NA_OK) return st;
    if ((st = check_ptrs({dattn, q, k, dq, dk})) != NA_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    p.a = dattn;
    p.b = k;
    p.out0 = dq;
    unfused_tma_maps(p, B, k, dattn, dtype, false);
    if ((st = cuda_status(na::launch_unfused_gather(p, elem_of(dtype), s))) != NA_OK) return st;
    p.b = q;
    p.out0 = dk;
    unfused_tma_maps(p, B, q, dattn, dtype, true);
    return cuda_status(na::launch_unfused_scatter(p, elem_of(dtype), s));
}

na_status na_av_bwd(const void* dO, const void* attn, const void* v, void* dattn, void* dv, int B, int ndim,
                    const int* spatial, int heads, int D, const int* kernel, const int* dilation, na_dtype dtype,
                    void* stream) {
    na::UnfParams p;
    na_status st = unfused_params(B, ndim, spatial, heads, D, kernel, dilation, 1.f, dtype, true, p);
    if (st != NA_OK) return st;
    if ((st = check_ptrs({dO, attn, v, dattn, dv})) != NA_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    p.a = dO;
    p.b = v;
    p.out0 = dattn;
    unfused_tma_maps(p, B, v, nullptr, dtype, false);
    if ((st = cuda_status(na::launch_unfused_dattn(p, elem_of(dtype), s))) != NA_OK) return st;
    p.a = attn;
    p.b = dO;
    p.out0 = dv;
    unfused_tma_maps(p, B, dO, attn, dtype, true);
    return cuda_status(na::launch_unfused_scatter(p, elem_of(dtype), s));
}

na_status na_mask_window(void* attn, const int* sizes, int B, int ndim, const int* spatial, int heads,
                         const int* kernel, const int* dilation, na_dtype dtype, void* stream) {
    na::UnfParams p;
    na_status st = unfused_params(B, ndim, spatial, heads, 0, kernel, dilation, 1.f, dtype, false, p);
    if (st != NA_OK) return st;
    if ((st = check_ptrs({attn})) != NA_OK) return st;
    if (!sizes) return NA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(sizes) & 3u) return NA_ERR_ALIGNMENT;
    // embedded 3D: the real axes are the last ndim; their sizes follow one another in `sizes`
    int off = 0;
    for (int a = 0; a < 3; ++a) {
        if (a < 3 - ndim) {
            p.vk_off[a] = -1;
        } else {
            p.vk_off[a] = off;
            off += spatial[a - (3 - ndim)];
        }
    }
    p.vk = sizes;
    p.out0 = attn;
    return cuda_status(na::launch_unfused_mask_window(p, elem_of(dtype), static_cast<cudaStream_t>(stream)));
}

size_t na_rpb_grad_workspace_size(int B, int ndim, const int* spatial, int heads, const int* kernel) {
    int ones[3] = {1, 1, 1};
    Geom g;
    if (make_geom(B, ndim, spatial, heads, 16, kernel, ones, g) != NA_OK) return 0;
    const int K = g.k[0] * g.k[1] * g.k[2];
    const int table = (2 * g.k[0] - 1) * (2 * g.k[1] - 1) * (2 * g.k[2] - 1);
    const size_t bytes = na::rpb_grad_workspace_bytes(tokens_of(g) * g.B, g.heads, K, table);
    return (bytes + 255) / 256 * 256;
}

na_status na_rpb_grad(const void* dattn, float* drpb, int B, int ndim, const int* spatial, int heads,
                      const int* kernel, const int* dilation, na_dtype dtype, void* workspace, size_t workspace_bytes,
                      void* stream) {
    na::UnfParams p;
    na_status st = unfused_params(B, ndim, spatial, heads, 0, kernel, dilation, 1.f, dtype, false, p);
    if (st != NA_OK) return st;
    if ((st = check_ptrs({dattn, drpb})) != NA_OK) return st;
    // every head's table must fit one block's shared memory, with the per-token indices
    const long long table = static_cast<long long>(2 * p.k[0] - 1) * (2 * p.k[1] - 1) * (2 * p.k[2] - 1);
    if (static_cast<long long>(heads) * table * 4 + 256LL * 12 > 227LL * 1024) return NA_ERR_UNSUPPORTED;
    const size_t need = na_rpb_grad_workspace_size(B, ndim, spatial, heads, kernel);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* ws = workspace;
    bool owned = false;
    if (ws) {
        if (workspace_bytes < need) return NA_ERR_WORKSPACE;
        if (!aligned16(ws)) return NA_ERR_ALIGNMENT;
    } else {
        if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return NA_ERR_WORKSPACE;
        owned = true;
    }
    p.a = dattn;
    st = cuda_status(na::launch_unfused_rpb_grad(p, elem_of(dtype), p.rows / p.heads, static_cast<float*>(ws), drpb, s));
    if (owned && cudaFreeAsync(ws, s) != cudaSuccess && st == NA_OK) st = NA_ERR_CUDA;
    return st;
}

}  // extern "C"
