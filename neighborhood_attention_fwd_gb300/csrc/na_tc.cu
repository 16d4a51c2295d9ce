// na_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels of libna for bf16 tensors on sm_103a:
// the query-tile forward, the dQ pass over query tiles and the atomic-free dK/dV pass over key
// tiles.
//
// The operation is neighborhood attention as read from NATTEN issue #161 ("Backward pass is very
// slow towards much tokens and large kernels"): each query attends a per-axis window of k keys of
// its residue class (dilation d), shifted at the borders, and the Cartesian product over axes.
// The maintainer's explanation there -- tiled kernels gain their speed by skipping key tiles that
// are fully masked, and pay for the partially masked ones with software predication in 2D/3D --
// is the cost this design attacks:
//   * a CTA owns 128 rows (a box of queries, or keys) of one (batch, head, residue class);
//   * the keys (or queries) any row of the tile can touch form a box, the halo; TMA stages it in
//     chunks (boxes of the halo with element stride = dilation), so nothing outside it is read;
//   * S = Q K^T and the products with P run on tcgen05 (bf16 in, fp32 accumulators in TMEM);
//   * each softmax warp owns 32 TMEM lanes (32 rows) and visits only the halo rows that hold a key
//     of at least one of its rows (the warp's union), in 8-column blocks, applying the exact
//     per-row window with integer tests; everything outside is written to P as zero.
//
// Thread roles (160 threads): warps 0-3 softmax / epilogue, warp 4 lane 0 issues TMA and MMA.
#include <cmath>

#include "na_device.cuh"
#include "na_internal.h"

namespace na {
using namespace dev;

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: keep a stale running max until it is 2^8 off

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Shared-memory layout (offsets from a 1024-byte aligned base).
//   which 0 (fwd) : tileA = Q,            ck/cv = K/V chunks, p0 = P
//   which 1 (dQ)  : tileA = Q, tileB = dO, ck/cv = K/V chunks, p0 = dS
//   which 2 (dKdV): tileA = K, tileB = V,  ck/cv = Q/dO chunks, p0 = P^T, p1 = dS^T, aux = LSE/Delta
struct TcLayout {
    uint32_t tileA, tileB, ck[kSlots], cv[kSlots], p0, p1, aux, bars, total;
};

__host__ __device__ inline TcLayout tc_layout(int which, const TilePlan& pl, int D) {
    const uint32_t tile = 128u * D * 2u;
    const uint32_t chunk = static_cast<uint32_t>(pl.NC) * D * 2u;
    const uint32_t pbytes = static_cast<uint32_t>((pl.NC + 31) / 32) * 8192u;
    TcLayout L{};
    uint32_t o = 0;
    L.tileA = o;
    o += align_up(tile, 1024);
    L.tileB = o;
    if (which != 0) o += align_up(tile, 1024);
    for (int s = 0; s < kSlots; ++s) {
        L.ck[s] = o;
        o += align_up(chunk, 1024);
        L.cv[s] = o;
        o += align_up(chunk, 1024);
    }
    L.p0 = o;
    o += align_up(pbytes, 1024);
    L.p1 = o;
    L.aux = o;
    if (which == 2) {
        o += align_up(pbytes, 1024);
        L.aux = o;
        o += align_up(2u * 2u * 256u * 4u, 1024);
    }
    L.bars = o;
    o += 256;
    L.total = o;
    return L;
}

enum Bar { kBarTile = 0, kBarCk = 1, kBarCv = 3, kBarEmpty = 5, kBarS = 7, kBarP = 8, kBarMM = 9, kBarFin = 10 };

// Per-CTA decode of (head, tile, residue class, batch) and the halo it needs.
struct Cta {
    int h, b;
    int cls[3], Lc[3], t0[3], h0[3], need[3];
    int ncy, ncz, C;
};

__device__ __forceinline__ int inv_lo(int j, int k) { return j < k ? 0 : j - (k >> 1); }
__device__ __forceinline__ int inv_hi(int j, int Lc, int k) { return j >= Lc - k ? Lc - 1 : j + (k >> 1); }

__device__ bool decode_cta(const TcParams& p, int which, Cta& c) {
    const TilePlan& pl = p.plan;
    long long x = blockIdx.x;
    c.h = static_cast<int>(x % p.heads);
    x /= p.heads;
    int t[3];
    for (int a = 2; a >= 0; --a) {
        t[a] = static_cast<int>(x % pl.ntile[a]);
        x /= pl.ntile[a];
    }
    for (int a = 2; a >= 0; --a) {
        c.cls[a] = static_cast<int>(x % p.d[a]);
        x /= p.d[a];
    }
    c.b = static_cast<int>(x);
    bool any = true;
    for (int a = 0; a < 3; ++a) {
        c.Lc[a] = class_len(p.L[a], p.d[a], c.cls[a]);
        c.t0[a] = t[a] * pl.T[a];
        if (c.t0[a] >= c.Lc[a]) any = false;
    }
    if (!any) return false;
    for (int a = 0; a < 3; ++a) {
        const int last = min(c.t0[a] + pl.T[a], c.Lc[a]) - 1;
        int lo, hi;
        if (which != 2) {
            lo = win_start(c.t0[a], c.Lc[a], p.k[a]);
            hi = win_start(last, c.Lc[a], p.k[a]) + p.k[a] - 1;
        } else {
            lo = inv_lo(c.t0[a], p.k[a]);
            hi = inv_hi(last, c.Lc[a], p.k[a]);
        }
        c.h0[a] = min(lo, max(0, c.Lc[a] - pl.H[a]));
        c.need[a] = hi - c.h0[a] + 1;
    }
    c.ncy = min(pl.nchk[0], (c.need[0] + pl.G[0] - 1) / pl.G[0]);
    c.ncz = min(pl.nchk[1], (c.need[1] + pl.G[1] - 1) / pl.G[1]);
    c.C = c.ncy * c.ncz;
    return true;
}

// Per-row geometry: for each axis the halo-coordinate range [lo, lo + len) of keys (fwd, dQ:
// the query's window) or queries (dK/dV: the queries whose windows hold the key) of this row.
struct RowGeom {
    int lo[3], len[3];
    bool valid;
    long long token;  // flat token index (b * N + spatial), valid rows only
};

__device__ RowGeom row_geom(const TcParams& p, int which, const Cta& c, int row) {
    const TilePlan& pl = p.plan;
    RowGeom g;
    int tq[3];
    tq[2] = row % pl.T[2];
    tq[1] = (row / pl.T[2]) % pl.T[1];
    tq[0] = row / (pl.T[2] * pl.T[1]);
    g.valid = true;
    long long tok = c.b;
    for (int a = 0; a < 3; ++a) {
        const int j = c.t0[a] + tq[a];
        if (j >= c.Lc[a]) g.valid = false;
        const int jc = min(j, c.Lc[a] - 1);
        if (which != 2) {
            g.lo[a] = win_start(jc, c.Lc[a], p.k[a]) - c.h0[a];
            g.len[a] = p.k[a];
        } else {
            g.lo[a] = inv_lo(jc, p.k[a]) - c.h0[a];
            g.len[a] = inv_hi(jc, c.Lc[a], p.k[a]) - inv_lo(jc, p.k[a]) + 1;
        }
        tok = tok * p.L[a] + (c.cls[a] + p.d[a] * jc);
    }
    if (!g.valid && which != 0)
        for (int a = 0; a < 3; ++a) g.len[a] = 0;  // no keys: P row is all zero
    g.token = tok;
    return g;
}

// Warp union of the rows' ranges: rows [ulo, uhi) per axis (empty if no row of the warp is live).
struct Union {
    int lo[3], hi[3];
};

__device__ Union warp_union(const RowGeom& g) {
    Union u;
    const bool live = g.len[0] > 0 && g.len[1] > 0 && g.len[2] > 0;
    for (int a = 0; a < 3; ++a) {
        u.lo[a] = warp_min(live ? g.lo[a] : 0x3fffffff);
        u.hi[a] = warp_max(live ? g.lo[a] + g.len[a] : -0x3fffffff);
    }
    return u;
}

// 8-bit mask of the live keys of block `bb` (halo columns 8bb..8bb+7 of the innermost axis) in a
// segment whose outer-axis test gave `rowok`.
__device__ __forceinline__ uint32_t block_mask(const RowGeom& g, bool rowok, int bb) {
    return rowok ? range_bits8(g.lo[2] - 8 * bb, g.lo[2] + g.len[2] - 8 * bb) : 0u;
}

__device__ __forceinline__ bool seg_rowok(const RowGeom& g, int y, int z) {
    return static_cast<unsigned>(y - g.lo[0]) < static_cast<unsigned>(g.len[0]) &&
           static_cast<unsigned>(z - g.lo[1]) < static_cast<unsigned>(g.len[1]);
}

// Byte offset of the 16-byte group holding columns [kcol, kcol+8) of row `row` in a K-major
// operand stored as 32-column atoms (128 rows x 64 B, 64-byte swizzle).
__device__ __forceinline__ uint32_t atom_off(int row, int kcol) {
    return static_cast<uint32_t>(kcol >> 5) * 8192u +
           swz(static_cast<uint32_t>(row) * 64u + static_cast<uint32_t>((kcol & 31) >> 3) * 16u, 3u);
}

// ---------------------------------------------------------------------------------------------
// Producer helpers (one thread)
// ---------------------------------------------------------------------------------------------

struct Producer {
    const TcParams& p;
    const Cta& c;
    uint8_t* smem;
    TcLayout lay;
    uint64_t* bars;
    int D;

    // Load the row tile of tensor map `m` at the CTA's tile origin into `dst`.
    __device__ void load_tile(int m, uint32_t dst, uint64_t* bar) const {
        tma_load_5d(smem + dst, &p.tm[m], bar, c.h * D, c.cls[2] + p.d[2] * c.t0[2], c.cls[1] + p.d[1] * c.t0[1],
                    c.cls[0] + p.d[0] * c.t0[0], c.b);
    }
    // Load chunk `ci` of tensor map `m` (halo box (G0, G1, H2) at (cy*G0, cz*G1, 0)).
    __device__ void load_chunk(int m, int ci, uint32_t dst, uint64_t* bar) const {
        const int cy = ci / c.ncz, cz = ci % c.ncz;
        const int y0 = c.h0[0] + cy * p.plan.G[0], z0 = c.h0[1] + cz * p.plan.G[1];
        tma_load_5d(smem + dst, &p.tm[m], bar, c.h * D, c.cls[2] + p.d[2] * c.h0[2], c.cls[1] + p.d[1] * z0,
                    c.cls[0] + p.d[0] * y0, c.b);
    }
    // D_tmem = A_tile(128 x D) * B_chunk(NC x D)^T, both K-major.
    __device__ void mma_rows_x_chunk(uint32_t d_tmem, uint32_t a_off, uint32_t b_off) const {
        const uint32_t rowb = D * 2u, lay_ = swizzle_layout(D * 2), sbo = 8u * rowb;
        const uint32_t idesc = idesc_bf16(128, p.plan.NC, false, false);
        const uint32_t a = smem_u32(smem + a_off), b = smem_u32(smem + b_off);
        for (int kk = 0; kk < D / 16; ++kk)
            umma_bf16(d_tmem, sdesc(a + kk * 32u, 16u, sbo, lay_), sdesc(b + kk * 32u, 16u, sbo, lay_), idesc,
                      kk > 0);
    }
    // D_tmem (+)= P(128 x NC, 32-column atoms) * B_chunk(NC x D), B MN-major.
    __device__ void mma_p_x_chunk(uint32_t d_tmem, uint32_t p_off, uint32_t b_off, bool accumulate) const {
        const uint32_t rowb = D * 2u, lay_ = swizzle_layout(D * 2), sbo = 8u * rowb;
        const uint32_t idesc = idesc_bf16(128, D, false, true);
        const uint32_t a = smem_u32(smem + p_off), b = smem_u32(smem + b_off);
        for (int kk = 0; kk < p.plan.NC / 16; ++kk) {
            const uint64_t ad = sdesc(a + (kk >> 1) * 8192u + (kk & 1) * 32u, 16u, 512u, 4u);
            const uint64_t bd = sdesc(b + kk * 16u * rowb, 16u * rowb, sbo, lay_);
            umma_bf16(d_tmem, ad, bd, idesc, (accumulate || kk > 0) ? 1u : 0u);
        }
    }
};

// Shared prologue: barriers, TMEM allocation.  Returns the TMEM base address.
__device__ uint32_t tc_setup(uint64_t* bars, uint32_t tmem_cols) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 12);
    if (warp == 4) {
        if (lane == 0) {
            mbar_init(&bars[kBarTile], 1);
            for (int s = 0; s < kSlots; ++s) {
                mbar_init(&bars[kBarCk + s], 1);
                mbar_init(&bars[kBarCv + s], 1);
                mbar_init(&bars[kBarEmpty + s], 1);
            }
            mbar_init(&bars[kBarS], 1);
            mbar_init(&bars[kBarP], kSoftmaxWarps);
            mbar_init(&bars[kBarMM], 1);
            mbar_init(&bars[kBarFin], 1);
            fence_barrier_init();
        }
        __syncwarp();
        tmem_alloc(slot, tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    return *slot;
}

__device__ void tc_teardown(uint64_t* bars, uint32_t tmem, uint32_t tmem_cols, unsigned* err) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 4 && lane == 0) {
        umma_commit(&bars[kBarFin]);  // completes once every MMA of this thread is done
        mbar_wait(&bars[kBarFin], 0, err, kSiteFinal);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// The producer schedule shared by the three kernels.
//   tile tensors: tmA -> tileA (+ tmB -> tileB if two_tiles), both on kBarTile
//   chunk tensors: tmCk -> ck[s] (kBarCk+s), tmCv -> cv[s] (kBarCv+s)
//   per chunk c: first MMAs ("score"), commit kBarS; wait kBarP (softmax wrote P/dS);
//   second MMAs ("update"), commit kBarMM and kBarEmpty+slot; refill the slot.
template <typename ScoreFn, typename UpdateFn>
__device__ void produce(const Producer& pr, int tmA, int tmB, bool two_tiles, int tmCk, int tmCv, bool score_needs_cv,
                        ScoreFn score, UpdateFn update, unsigned* err) {
    uint64_t* bars = pr.bars;
    const int C = pr.c.C;
    const uint32_t tile_bytes = 128u * pr.D * 2u;
    const uint32_t chunk_bytes = static_cast<uint32_t>(pr.p.plan.NC) * pr.D * 2u;
    mbar_arrive_expect_tx(&bars[kBarTile], two_tiles ? 2u * tile_bytes : tile_bytes);
    pr.load_tile(tmA, pr.lay.tileA, &bars[kBarTile]);
    if (two_tiles) pr.load_tile(tmB, pr.lay.tileB, &bars[kBarTile]);
    auto load = [&](int ci, int s) {
        mbar_arrive_expect_tx(&bars[kBarCk + s], chunk_bytes);
        pr.load_chunk(tmCk, ci, pr.lay.ck[s], &bars[kBarCk + s]);
        mbar_arrive_expect_tx(&bars[kBarCv + s], chunk_bytes);
        pr.load_chunk(tmCv, ci, pr.lay.cv[s], &bars[kBarCv + s]);
    };
    for (int ci = 0; ci < min(kSlots, C); ++ci) load(ci, ci);

    bool ok = mbar_wait(&bars[kBarTile], 0, err, kSiteQ);
    ok = ok && mbar_wait(&bars[kBarCk], 0, err, kSiteKV);
    if (score_needs_cv) ok = ok && mbar_wait(&bars[kBarCv], 0, err, kSiteKV);
    if (!ok) return;
    tc_fence_after();
    score(0);
    umma_commit(&bars[kBarS]);
    for (int ci = 0; ci < C; ++ci) {
        const int s = ci % kSlots;
        const uint32_t ph = (ci / kSlots) & 1;
        ok = mbar_wait(&bars[kBarP], ci & 1, err, kSiteP);
        ok = ok && mbar_wait(&bars[kBarCv + s], ph, err, kSiteKV);
        if (!ok) return;
        tc_fence_after();
        update(ci, s);
        umma_commit(&bars[kBarMM]);
        umma_commit(&bars[kBarEmpty + s]);
        if (ci + 1 < C) {
            const int s1 = (ci + 1) % kSlots;
            const uint32_t ph1 = ((ci + 1) / kSlots) & 1;
            ok = mbar_wait(&bars[kBarCk + s1], ph1, err, kSiteKV);
            if (score_needs_cv) ok = ok && mbar_wait(&bars[kBarCv + s1], ph1, err, kSiteKV);
            if (!ok) return;
            tc_fence_after();
            score(s1);
            umma_commit(&bars[kBarS]);
        }
        if (ci + kSlots < C) {
            if (!mbar_wait(&bars[kBarEmpty + s], ph, err, kSiteEmpty)) return;
            load(ci + kSlots, s);
        }
    }
}

// Bounded wait by every lane of a warp; the result is made warp-uniform so that the following
// .sync.aligned tcgen05 instructions never run divergent.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned* err, unsigned site) {
    const bool ok = mbar_wait(bar, parity, err, site);
    return __all_sync(0xffffffffu, ok);
}

// Chunk ci's box in halo coordinates: rows y in [y0, y0 + G0), z in [z0, z0 + G1).
struct ChunkBox {
    int y0, z0, ya, yb, za, zb;  // [ya, yb) x [za, zb): the part of the warp union inside the chunk
};

__device__ __forceinline__ ChunkBox chunk_box(const TilePlan& pl, const Cta& c, const Union& u, int ci) {
    ChunkBox b;
    b.y0 = (ci / c.ncz) * pl.G[0];
    b.z0 = (ci % c.ncz) * pl.G[1];
    b.ya = max(u.lo[0], b.y0);
    b.yb = min(u.hi[0], b.y0 + pl.G[0]);
    b.za = max(u.lo[1], b.z0);
    b.zb = min(u.hi[1], b.z0 + pl.G[1]);
    return b;
}

// Write the 128-row tile staged in `stage` (row-major [128][D] bf16 with the tensor map's swizzle)
// back with TMA.  Called by all 128 softmax threads.
__device__ void store_tile(const TcParams& p, const Cta& c, int m, uint8_t* stage, int D) {
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (threadIdx.x == 0 && ld_volatile(p.err) == 0u) {
        tma_store_5d(&p.tm[m], stage, c.h * D, c.cls[2] + p.d[2] * c.t0[2], c.cls[1] + p.d[1] * c.t0[1],
                     c.cls[0] + p.d[0] * c.t0[0], c.b);
        tma_store_commit();
        tma_store_wait_all();
    }
}

// Read this thread's accumulator row (D fp32 columns at tcol), scale it and stage it as bf16.
template <int D>
__device__ void stage_row(uint32_t taddr, float mul, uint8_t* stage, int row) {
    const uint32_t base = smem_u32(stage), mask = swizzle_mask(D * 2);
#pragma unroll
    for (int cc = 0; cc < D; cc += 8) {
        uint32_t r[8];
        tmem_ld8(taddr + cc, r);
        tmem_ld_wait(r);
        const uint32_t w0 = pack_bf16x2(__uint_as_float(r[0]) * mul, __uint_as_float(r[1]) * mul);
        const uint32_t w1 = pack_bf16x2(__uint_as_float(r[2]) * mul, __uint_as_float(r[3]) * mul);
        const uint32_t w2 = pack_bf16x2(__uint_as_float(r[4]) * mul, __uint_as_float(r[5]) * mul);
        const uint32_t w3 = pack_bf16x2(__uint_as_float(r[6]) * mul, __uint_as_float(r[7]) * mul);
        st_shared_v4(base + swz(static_cast<uint32_t>(row) * (D * 2) + cc * 2, mask), w0, w1, w2, w3);
    }
}

// ---------------------------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const TilePlan& pl = p.plan;
    const TcLayout lay = tc_layout(0, pl, D);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
    Cta c;
    if (!decode_cta(p, 0, c)) return;
    const uint32_t tmem = tc_setup(bars, pl.tmem_cols);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned* err = p.err;
    const uint32_t tS = tmem, tO = tmem + static_cast<uint32_t>(pl.tmem_cols - D);

    if (warp == 4) {
        if (lane == 0) {
            Producer pr{p, c, smem, lay, bars, D};
            auto score = [&](int s) { pr.mma_rows_x_chunk(tS, lay.tileA, lay.ck[s]); };
            auto update = [&](int ci, int s) { pr.mma_p_x_chunk(tO, lay.p0, lay.cv[s], ci > 0); };
            produce(pr, 0, 0, false, 1, 2, false, score, update, err);
        }
        __syncwarp();
    } else {
        const int row = warp * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const RowGeom g = row_geom(p, 0, c, row);
        const Union u = warp_union(g);
        const int blo = max(0, u.lo[2]) >> 3, bhi = min(pl.H[2], u.hi[2] + 7) >> 3;
        const int nb = pl.H[2] >> 3;
        const float sl2 = p.scale_log2;
        const uint32_t sP = smem_u32(smem + lay.p0);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int ci = 0; ci < c.C && ok; ++ci) {
            ok = warp_wait(&bars[kBarS], ci & 1, err, kSiteS);
            if (!ok) break;
            tc_fence_after();
            const ChunkBox cb = chunk_box(pl, c, u, ci);
            // pass 1: masked row max over the warp's part of the chunk (log2 units)
            float cmax = -INFINITY;
            for (int y = cb.ya; y < cb.yb; ++y)
                for (int z = cb.za; z < cb.zb; ++z) {
                    const bool rowok = seg_rowok(g, y, z);
                    const int seg = ((y - cb.y0) * pl.G[1] + (z - cb.z0)) * pl.H[2];
                    for (int bb = blo; bb < bhi; ++bb) {
                        uint32_t r[8];
                        tmem_ld8(tS + lane_base + seg + bb * 8, r);
                        tmem_ld_wait(r);
                        const uint32_t m8 = block_mask(g, rowok, bb);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (m8 & (1u << e)) cmax = fmaxf(cmax, __uint_as_float(r[e]) * sl2);
                    }
                }
            const float mnew = fmaxf(m, cmax);
            const bool rescale = (m != -INFINITY) && (mnew > m + kRescaleThreshold);
            const float alpha = rescale ? fast_exp2(m - mnew) : 1.f;
            if (m == -INFINITY || rescale) m = mnew;
            // P (single buffer) and O are free once the previous chunk's PV product is done
            if (ci > 0) {
                ok = warp_wait(&bars[kBarMM], (ci - 1) & 1, err, kSitePV);
                if (!ok) break;
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int cc = 0; cc < D; cc += 8) {
                    uint32_t r[8];
                    tmem_ld8(tO + lane_base + cc, r);
                    tmem_ld_wait(r);
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                    tmem_st8(tO + lane_base + cc, r);
                }
                tmem_st_wait();
                l *= alpha;
            }
            // pass 2: P = exp2(x - m) on live keys, zero elsewhere
            for (int y = cb.y0; y < cb.y0 + pl.G[0]; ++y)
                for (int z = cb.z0; z < cb.z0 + pl.G[1]; ++z) {
                    const bool segact = y >= cb.ya && y < cb.yb && z >= cb.za && z < cb.zb;
                    const bool rowok = seg_rowok(g, y, z);
                    const int seg = ((y - cb.y0) * pl.G[1] + (z - cb.z0)) * pl.H[2];
                    for (int bb = 0; bb < nb; ++bb) {
                        uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
                        if (segact && bb >= blo && bb < bhi) {
                            uint32_t r[8];
                            tmem_ld8(tS + lane_base + seg + bb * 8, r);
                            tmem_ld_wait(r);
                            const uint32_t m8 = block_mask(g, rowok, bb);
                            float pe[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                pe[e] = (m8 & (1u << e)) ? fast_exp2(fmaf(__uint_as_float(r[e]), sl2, -m)) : 0.f;
                                l += pe[e];
                            }
                            w0 = pack_bf16x2(pe[0], pe[1]);
                            w1 = pack_bf16x2(pe[2], pe[3]);
                            w2 = pack_bf16x2(pe[4], pe[5]);
                            w3 = pack_bf16x2(pe[6], pe[7]);
                        }
                        st_shared_v4(sP + atom_off(row, seg + bb * 8), w0, w1, w2, w3);
                    }
                }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kBarP]);
        }
        // epilogue: O / l -> bf16 -> TMA store; LSE = (m + log2 l) * ln 2
        if (ok) ok = warp_wait(&bars[kBarMM], (c.C - 1) & 1, err, kSitePV);
        if (ok) {
            tc_fence_after();
            stage_row<D>(tO + lane_base, 1.f / l, smem + lay.tileA, row);
            if (g.valid) p.lse_out[g.token * p.heads + c.h] = (m + __log2f(l)) * kLn2;
        }
        store_tile(p, c, 3, smem + lay.tileA, D);
    }
    tc_teardown(bars, tmem, pl.tmem_cols, err);
}

// ---------------------------------------------------------------------------------------------
// dQ
// ---------------------------------------------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(kThreads, 1) dq_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const TilePlan& pl = p.plan;
    const TcLayout lay = tc_layout(1, pl, D);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
    Cta c;
    if (!decode_cta(p, 1, c)) return;
    const uint32_t tmem = tc_setup(bars, pl.tmem_cols);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned* err = p.err;
    const uint32_t tS = tmem, tP = tmem + static_cast<uint32_t>(pl.NC),
                   tQ = tmem + static_cast<uint32_t>(pl.tmem_cols - D);

    if (warp == 4) {
        if (lane == 0) {
            Producer pr{p, c, smem, lay, bars, D};
            auto score = [&](int s) {
                pr.mma_rows_x_chunk(tS, lay.tileA, lay.ck[s]);  // S  = Q K^T
                pr.mma_rows_x_chunk(tP, lay.tileB, lay.cv[s]);  // dP = dO V^T
            };
            auto update = [&](int ci, int s) { pr.mma_p_x_chunk(tQ, lay.p0, lay.ck[s], ci > 0); };  // dQ += dS K
            produce(pr, 0, 1, true, 2, 3, true, score, update, err);
        }
        __syncwarp();
    } else {
        const int row = warp * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const RowGeom g = row_geom(p, 1, c, row);
        const Union u = warp_union(g);
        const int blo = max(0, u.lo[2]) >> 3, bhi = min(pl.H[2], u.hi[2] + 7) >> 3;
        const int nb = pl.H[2] >> 3;
        const float sl2 = p.scale_log2;
        float lse2 = 0.f, dlt = 0.f;
        if (g.valid) {
            lse2 = p.lse[g.token * p.heads + c.h] * kLog2e;
            dlt = p.delta[g.token * p.heads + c.h];
        }
        const uint32_t sDS = smem_u32(smem + lay.p0);
        bool ok = true;
        for (int ci = 0; ci < c.C && ok; ++ci) {
            ok = warp_wait(&bars[kBarS], ci & 1, err, kSiteS);
            if (ok && ci > 0) ok = warp_wait(&bars[kBarMM], (ci - 1) & 1, err, kSitePV);
            if (!ok) break;
            tc_fence_after();
            const ChunkBox cb = chunk_box(pl, c, u, ci);
            for (int y = cb.y0; y < cb.y0 + pl.G[0]; ++y)
                for (int z = cb.z0; z < cb.z0 + pl.G[1]; ++z) {
                    const bool segact = y >= cb.ya && y < cb.yb && z >= cb.za && z < cb.zb;
                    const bool rowok = seg_rowok(g, y, z);
                    const int seg = ((y - cb.y0) * pl.G[1] + (z - cb.z0)) * pl.H[2];
                    for (int bb = 0; bb < nb; ++bb) {
                        uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
                        if (segact && bb >= blo && bb < bhi) {
                            uint32_t rs[8], rp[8];
                            tmem_ld8(tS + lane_base + seg + bb * 8, rs);
                            tmem_ld8(tP + lane_base + seg + bb * 8, rp);
                            tmem_ld_wait2(rs, rp);
                            const uint32_t m8 = block_mask(g, rowok, bb);
                            float ds[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float pe =
                                    (m8 & (1u << e)) ? fast_exp2(fmaf(__uint_as_float(rs[e]), sl2, -lse2)) : 0.f;
                                ds[e] = pe * (__uint_as_float(rp[e]) - dlt);
                            }
                            w0 = pack_bf16x2(ds[0], ds[1]);
                            w1 = pack_bf16x2(ds[2], ds[3]);
                            w2 = pack_bf16x2(ds[4], ds[5]);
                            w3 = pack_bf16x2(ds[6], ds[7]);
                        }
                        st_shared_v4(sDS + atom_off(row, seg + bb * 8), w0, w1, w2, w3);
                    }
                }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kBarP]);
        }
        if (ok) ok = warp_wait(&bars[kBarMM], (c.C - 1) & 1, err, kSitePV);
        if (ok) {
            tc_fence_after();
            stage_row<D>(tQ + lane_base, p.scale, smem + lay.tileA, row);
        }
        store_tile(p, c, 4, smem + lay.tileA, D);
    }
    tc_teardown(bars, tmem, pl.tmem_cols, err);
}

// ---------------------------------------------------------------------------------------------
// dK / dV
// ---------------------------------------------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(kThreads, 1) dkdv_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const TilePlan& pl = p.plan;
    const TcLayout lay = tc_layout(2, pl, D);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
    Cta c;
    if (!decode_cta(p, 2, c)) return;
    const uint32_t tmem = tc_setup(bars, pl.tmem_cols);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned* err = p.err;
    const uint32_t tS = tmem, tP = tmem + static_cast<uint32_t>(pl.NC),
                   tV = tmem + static_cast<uint32_t>(pl.tmem_cols - 2 * D),
                   tK = tmem + static_cast<uint32_t>(pl.tmem_cols - D);

    if (warp == 4) {
        if (lane == 0) {
            Producer pr{p, c, smem, lay, bars, D};
            auto score = [&](int s) {
                pr.mma_rows_x_chunk(tS, lay.tileA, lay.ck[s]);  // S^T  = K Q^T
                pr.mma_rows_x_chunk(tP, lay.tileB, lay.cv[s]);  // dP^T = V dO^T
            };
            auto update = [&](int ci, int s) {
                pr.mma_p_x_chunk(tV, lay.p0, lay.cv[s], ci > 0);  // dV += P^T dO
                pr.mma_p_x_chunk(tK, lay.p1, lay.ck[s], ci > 0);  // dK += dS^T Q
            };
            produce(pr, 0, 1, true, 2, 3, true, score, update, err);
        }
        __syncwarp();
    } else {
        const int row = warp * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const RowGeom g = row_geom(p, 2, c, row);
        const Union u = warp_union(g);
        const int blo = max(0, u.lo[2]) >> 3, bhi = min(pl.H[2], u.hi[2] + 7) >> 3;
        const int nb = pl.H[2] >> 3;
        const float sl2 = p.scale_log2;
        const uint32_t sPT = smem_u32(smem + lay.p0), sDST = smem_u32(smem + lay.p1);
        float* aux = reinterpret_cast<float*>(smem + lay.aux);  // [2 buffers][lse2 | delta][256]
        const int tid = threadIdx.x;
        bool ok = true;
        // Every warp runs every iteration (the named barrier below needs all four), doing no
        // work once a wait has given up.
        for (int ci = 0; ci < c.C; ++ci) {
            // per-column LSE (log2 units) and Delta of this chunk's queries
            float* l2 = aux + (ci & 1) * 512;
            float* dl = l2 + 256;
            const int cy = ci / c.ncz, cz = ci % c.ncz;
            for (int col = tid; col < pl.NC; col += 128) {
                const int x2 = col % pl.H[2], x1 = (col / pl.H[2]) % pl.G[1], x0 = col / (pl.H[2] * pl.G[1]);
                const int j0 = c.h0[0] + cy * pl.G[0] + x0, j1 = c.h0[1] + cz * pl.G[1] + x1, j2 = c.h0[2] + x2;
                float lv = INFINITY, dv = 0.f;
                if (j0 < c.Lc[0] && j1 < c.Lc[1] && j2 < c.Lc[2]) {
                    const long long tok = ((static_cast<long long>(c.b) * p.L[0] + (c.cls[0] + p.d[0] * j0)) * p.L[1] +
                                           (c.cls[1] + p.d[1] * j1)) * p.L[2] + (c.cls[2] + p.d[2] * j2);
                    lv = p.lse[tok * p.heads + c.h] * kLog2e;
                    dv = p.delta[tok * p.heads + c.h];
                }
                l2[col] = lv;
                dl[col] = dv;
            }
            named_bar_sync(1, 128);
            if (ok) ok = warp_wait(&bars[kBarS], ci & 1, err, kSiteS);
            if (ok && ci > 0) ok = warp_wait(&bars[kBarMM], (ci - 1) & 1, err, kSitePV);
            if (!ok) continue;
            tc_fence_after();
            const ChunkBox cb = chunk_box(pl, c, u, ci);
            for (int y = cb.y0; y < cb.y0 + pl.G[0]; ++y)
                for (int z = cb.z0; z < cb.z0 + pl.G[1]; ++z) {
                    const bool segact = y >= cb.ya && y < cb.yb && z >= cb.za && z < cb.zb;
                    const bool rowok = seg_rowok(g, y, z);
                    const int seg = ((y - cb.y0) * pl.G[1] + (z - cb.z0)) * pl.H[2];
                    for (int bb = 0; bb < nb; ++bb) {
                        uint32_t p0 = 0, p1 = 0, p2 = 0, p3 = 0, d0 = 0, d1 = 0, d2 = 0, d3 = 0;
                        if (segact && bb >= blo && bb < bhi) {
                            uint32_t rs[8], rp[8];
                            tmem_ld8(tS + lane_base + seg + bb * 8, rs);
                            tmem_ld8(tP + lane_base + seg + bb * 8, rp);
                            tmem_ld_wait2(rs, rp);
                            const uint32_t m8 = block_mask(g, rowok, bb);
                            const int col0 = seg + bb * 8;
                            float pe[8], ds[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                pe[e] = (m8 & (1u << e)) ? fast_exp2(fmaf(__uint_as_float(rs[e]), sl2, -l2[col0 + e]))
                                                         : 0.f;
                                ds[e] = pe[e] * (__uint_as_float(rp[e]) - dl[col0 + e]);
                            }
                            p0 = pack_bf16x2(pe[0], pe[1]);
                            p1 = pack_bf16x2(pe[2], pe[3]);
                            p2 = pack_bf16x2(pe[4], pe[5]);
                            p3 = pack_bf16x2(pe[6], pe[7]);
                            d0 = pack_bf16x2(ds[0], ds[1]);
                            d1 = pack_bf16x2(ds[2], ds[3]);
                            d2 = pack_bf16x2(ds[4], ds[5]);
                            d3 = pack_bf16x2(ds[6], ds[7]);
                        }
                        const uint32_t off = atom_off(row, seg + bb * 8);
                        st_shared_v4(sPT + off, p0, p1, p2, p3);
                        st_shared_v4(sDST + off, d0, d1, d2, d3);
                    }
                }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kBarP]);
        }
        if (ok) ok = warp_wait(&bars[kBarMM], (c.C - 1) & 1, err, kSitePV);
        if (ok) {
            tc_fence_after();
            stage_row<D>(tV + lane_base, 1.f, smem + lay.tileB, row);
        }
        store_tile(p, c, 5, smem + lay.tileB, D);
        if (ok) stage_row<D>(tK + lane_base, p.scale, smem + lay.tileA, row);
        store_tile(p, c, 4, smem + lay.tileA, D);
    }
    tc_teardown(bars, tmem, pl.tmem_cols, err);
}

template <typename K>
int launch(K kernel, const TcParams& p, cudaStream_t stream) {
    const int smem = p.plan.smem_bytes;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (p.plan.ctas <= 0) return 0;
    kernel<<<dim3(static_cast<unsigned>(p.plan.ctas)), dim3(kThreads), smem, stream>>>(p);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

uint32_t tc_smem_bytes(int which, const TilePlan& pl, int D) { return tc_layout(which, pl, D).total + 1024u; }

int launch_fwd_tc(const TcParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch(fwd_tc_kernel<16>, p, s);
        case 32: return launch(fwd_tc_kernel<32>, p, s);
        case 64: return launch(fwd_tc_kernel<64>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dq_tc(const TcParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch(dq_tc_kernel<16>, p, s);
        case 32: return launch(dq_tc_kernel<32>, p, s);
        case 64: return launch(dq_tc_kernel<64>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dkdv_tc(const TcParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch(dkdv_tc_kernel<16>, p, s);
        case 32: return launch(dkdv_tc_kernel<32>, p, s);
        case 64: return launch(dkdv_tc_kernel<64>, p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace na
