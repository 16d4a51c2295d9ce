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
//   * a tile is 128 rows (a box of queries, or keys) of one (batch, head, residue class);
//   * the keys (or queries) any row of the tile can touch form a box, the halo; TMA stages it in
//     chunks (boxes of the halo with element stride = dilation), so nothing outside it is read;
//   * S = Q K^T and the products with P run on tcgen05 (bf16 in, fp32 accumulators in TMEM);
//   * a chunk is G0 x G1 segments of NB 8-column blocks; each softmax warp owns 32 TMEM lanes
//     (32 rows) and touches only the blocks that hold a key of at least one of its rows; the
//     exact per-row window is applied from bit masks (one bit per segment, one byte per block
//     column), so the predication costs a few integer ops per 8 logits.
//
// Pipeline (persistent CTAs, each looping over tiles):
//   producer warp : TMA of the tile tensors (2-slot ring) and of halo chunks (kStages-slot ring)
//   MMA warp      : per chunk the "score" products into a double-buffered TMEM accumulator, then
//                   the previous chunk's "update" products into a double-buffered tile accumulator
//   softmax warps : per chunk read scores from TMEM, write P (or dS) to a double-buffered smem
//                   operand; per tile read the accumulator and store it with TMA.
// Every mbarrier wait is bounded (see na_device.cuh); a wait that gives up records the site in the
// status word and the CTA stops issuing work.
#include <cmath>

#include "na_device.cuh"
#include "na_internal.h"

namespace na {
using namespace dev;

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: keep a stale running max until it is 2^8 off
constexpr int kStages = 3;                  // halo chunk ring depth
constexpr int kMaxBlocks = 14;              // 8-column blocks per chunk (NC <= 112)

__host__ __device__ constexpr int nwg_of(int which) { return which == 0 ? 1 : 2; }
__host__ __device__ constexpr int threads_of(int which) { return 32 * (4 * nwg_of(which) + 2); }

// Most 8-column blocks one forward chunk can hold for head dim D (TMEM: 2 * NC + 2 * D <= 256).
__host__ __device__ constexpr int fwd_max_blocks(int D) {
    return ((256 - 2 * D) / 2) / 8 < 12 ? ((256 - 2 * D) / 2) / 8 : 12;
}

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Shared-memory layout (offsets from a 1024-byte aligned base).
//   which 0 (fwd) : tile ring [2] x {Q};     chunk ring [kStages] x {K, V};  P[2];           staging {O}
//   which 1 (dQ)  : tile ring [2] x {Q, dO}; chunk ring [kStages] x {K, V};  dS[2];          staging {dQ}
//   which 2 (dKdV): tile ring [2] x {K, V};  chunk ring [kStages] x {Q, dO}; P^T[2], dS^T[2]; staging {dK, dV}
//                   plus per chunk slot the LSE (log2 units) and Delta of its queries.
struct TcLayout {
    uint32_t tile0, tile_slot, tile_t;     // tile ring: tile0 + slot * tile_slot + tensor * tile_t
    uint32_t chunk0, chunk_slot, chunk_t;  // chunk ring
    uint32_t p0, p_buf, p_op;              // P / dS operands
    uint32_t aux0, aux_slot;               // dK/dV per-column LSE (log2) and Delta
    uint32_t stage0, stage_t;              // epilogue staging
    uint32_t bars, total;
    __host__ __device__ uint32_t tile(uint32_t slot, uint32_t t) const { return tile0 + slot * tile_slot + t * tile_t; }
    __host__ __device__ uint32_t chunk(uint32_t slot, uint32_t t) const {
        return chunk0 + slot * chunk_slot + t * chunk_t;
    }
    __host__ __device__ uint32_t p(uint32_t buf, uint32_t op) const { return p0 + buf * p_buf + op * p_op; }
    __host__ __device__ uint32_t aux(uint32_t slot) const { return aux0 + slot * aux_slot; }
    __host__ __device__ uint32_t stage(uint32_t t) const { return stage0 + t * stage_t; }
};

__host__ __device__ inline TcLayout tc_layout(int which, const TilePlan& pl, int D) {
    const uint32_t tile = align_up(128u * D * 2u, 1024);
    const uint32_t chunk = align_up(static_cast<uint32_t>(pl.NC) * D * 2u, 1024);
    const uint32_t pbytes = static_cast<uint32_t>((pl.NC + 31) / 32) * 8192u;
    const uint32_t ntile = which == 0 ? 1 : 2, nop = which == 2 ? 2 : 1, nstage = which == 2 ? 2 : 1;
    const uint32_t auxb = which == 2 ? align_up(2u * 4u * static_cast<uint32_t>(pl.NC), 1024) : 0u;
    TcLayout L{};
    uint32_t o = 0;
    L.tile0 = o;
    L.tile_t = tile;
    L.tile_slot = ntile * tile;
    o += 2 * L.tile_slot;
    L.chunk0 = o;
    L.chunk_t = chunk;
    L.chunk_slot = 2 * chunk;
    o += kStages * L.chunk_slot;
    L.p0 = o;
    L.p_op = pbytes;
    L.p_buf = nop * pbytes;
    o += 2 * L.p_buf;
    L.aux0 = o;
    L.aux_slot = auxb;
    o += kStages * auxb;
    L.stage0 = o;
    L.stage_t = tile;
    o += nstage * tile;
    L.bars = o;
    o += 512;
    L.total = o;
    return L;
}

// mbarrier indices
enum Bar {
    kQFull = 0, kQEmpty = 2, kKVFull = 4, kKVEmpty = 4 + kStages, kSFull = 4 + 2 * kStages,
    kSEmpty = kSFull + 2, kPFull = kSEmpty + 2, kPEmpty = kPFull + 2, kOFull = kPEmpty + 2, kOEmpty = kOFull + 2,
    kStFree = kOEmpty + 2, kStFull = kStFree + 1, kFin = kStFull + 1, kNumBars = kFin + 1
};

// ---------------------------------------------------------------------------------------------
// Tile stream and tile geometry
// ---------------------------------------------------------------------------------------------

// Position in the mixed-radix tile index (digits: head, tile2, tile1, tile0, class2, class1,
// class0, batch).  A persistent CTA starts at blockIdx.x and steps by the grid size, adding the
// grid size's digits with carries instead of dividing.
struct TileIter {
    uint32_t dig[8];
    uint32_t lin;
};

__device__ __forceinline__ TileIter tile_iter_begin(const TcParams& p) {
    TileIter it;
    uint32_t x = blockIdx.x;
    it.lin = x;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        it.dig[i] = x % p.rad[i];
        x /= p.rad[i];
    }
    return it;
}

__device__ __forceinline__ void tile_iter_next(const TcParams& p, TileIter& it) {
    uint32_t carry = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t v = it.dig[i] + p.step[i] + carry;
        carry = v >= p.rad[i] ? 1u : 0u;
        it.dig[i] = carry ? v - p.rad[i] : v;
    }
    it.lin += gridDim.x;
}

// Per-tile decode of (head, tile, residue class, batch) and the halo it needs.
struct Cta {
    int h, b;
    int cls[3], Lc[3], t0[3], h0[3];
    int nc[3], C;  // chunks actually needed along each axis, and in total
};

__device__ __forceinline__ int inv_lo(int j, int k) { return j < k ? 0 : j - (k >> 1); }
__device__ __forceinline__ int inv_hi(int j, int Lc, int k) { return j >= Lc - k ? Lc - 1 : j + (k >> 1); }

__device__ __forceinline__ bool decode_tile(const TcParams& p, int which, const TileIter& it, Cta& c) {
    const TilePlan& pl = p.plan;
    c.h = static_cast<int>(it.dig[0]);
    c.cls[2] = static_cast<int>(it.dig[4]);
    c.cls[1] = static_cast<int>(it.dig[5]);
    c.cls[0] = static_cast<int>(it.dig[6]);
    c.b = static_cast<int>(it.dig[7]);
    const int t[3] = {static_cast<int>(it.dig[3]), static_cast<int>(it.dig[2]), static_cast<int>(it.dig[1])};
    bool any = true;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        c.Lc[a] = class_len(p.L[a], p.d[a], c.cls[a]);
        c.t0[a] = t[a] * pl.T[a];
        if (c.t0[a] >= c.Lc[a]) any = false;
    }
    if (!any) return false;
    c.C = 1;
#pragma unroll
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
        c.nc[a] = min(pl.nchk[a], (hi - c.h0[a] + pl.G[a]) / pl.G[a]);
        c.C *= c.nc[a];
    }
    return true;
}

// Next non-empty tile of this persistent CTA.  `started` is false before the first call.
__device__ __forceinline__ bool next_tile(const TcParams& p, int which, TileIter& it, bool& started, Cta& c) {
    const uint32_t n = static_cast<uint32_t>(p.plan.ctas);
    if (started) tile_iter_next(p, it);
    started = true;
    while (it.lin < n) {
        if (decode_tile(p, which, it, c)) return true;
        tile_iter_next(p, it);
    }
    return false;
}

// Chunk ci's origin in halo coordinates (chunk grid order: axis 0 slowest, axis 2 fastest).
__device__ __forceinline__ void chunk_origin(const TilePlan& pl, const Cta& c, int ci, int& y0, int& z0, int& x0) {
    const int cx = ci % c.nc[2], r = ci / c.nc[2];
    const int cz = r % c.nc[1], cy = r / c.nc[1];
    y0 = cy * pl.G[0];
    z0 = cz * pl.G[1];
    x0 = cx * pl.G[2];
}

// Per-row geometry: for each axis the halo-coordinate range [lo, lo + len) of keys (fwd, dQ: the
// query's window) or queries (dK/dV: the queries whose windows hold the key) of this row.
struct RowGeom {
    int lo[3], len[3];
    bool valid;
    long long token;  // flat token index (b * N + spatial), valid rows only
};

__device__ __forceinline__ RowGeom row_geom(const TcParams& p, int which, const Cta& c, int row) {
    const TilePlan& pl = p.plan;
    RowGeom g;
    // tile extents are powers of two
    const int s2 = __ffs(pl.T[2]) - 1, s1 = __ffs(pl.T[1]) - 1;
    const int tq[3] = {row >> (s2 + s1), (row >> s2) & (pl.T[1] - 1), row & (pl.T[2] - 1)};
    g.valid = true;
    long long tok = c.b;
#pragma unroll
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
    if (!g.valid && which != 0) {
#pragma unroll
        for (int a = 0; a < 3; ++a) g.len[a] = 0;  // no keys: the P row is all zero
    }
    g.token = tok;
    return g;
}

// Warp union of the rows' ranges along each axis (empty when no row of the warp is live).
struct WarpUnion {
    int lo[3], hi[3];
};

__device__ __forceinline__ WarpUnion warp_union(const RowGeom& g) {
    WarpUnion u;
    const bool live = g.len[0] > 0 && g.len[1] > 0 && g.len[2] > 0;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        u.lo[a] = warp_min(live ? g.lo[a] : 0x3fffffff);
        u.hi[a] = warp_max(live ? g.lo[a] + g.len[a] : -0x3fffffff);
    }
    return u;
}

// Bits [lo, hi) of a 32-bit word, lo and hi clamped to [0, 32].
__device__ __forceinline__ uint32_t range_bits32(int lo, int hi) {
    lo = max(0, min(32, lo));
    hi = max(0, min(32, hi));
    const uint32_t up_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
    const uint32_t up_lo = lo >= 32 ? 0xffffffffu : ((1u << lo) - 1u);
    return up_hi & ~up_lo;
}

// Segment bits of a chunk (segment s = (y - y0) * G1 + (z - z0)) whose (y, z) lies in
// [ylo, yhi) x [zlo, zhi).
__device__ __forceinline__ uint32_t segment_bits(const TilePlan& pl, int y0, int z0, int ylo, int yhi, int zlo,
                                                 int zhi) {
    const uint32_t zb = range_bits32(zlo - z0, zhi - z0) & range_bits32(0, pl.G[1]);
    uint32_t bits = 0;
    for (int y = max(ylo, y0); y < min(yhi, y0 + pl.G[0]); ++y) bits |= zb << ((y - y0) * pl.G[1]);
    return bits;
}

// Per-chunk masks.  act: bit i = block i of the chunk intersects the warp union (warp-uniform).
// rowseg: bit s = segment s lies inside this row's window along axes 0 and 1.
// m8: byte bb = this row's live columns of block bb (block columns 8bb .. 8bb+7 of a segment).
struct ChunkMasks {
    uint32_t act, rowseg, m8;
};

// Chunk cursor: origin (halo coordinates) of the current chunk, stepped in chunk-grid order
// (axis 0 slowest, axis 2 fastest) without divisions.
struct ChunkCursor {
    int y0, z0, x0;
};
__device__ __forceinline__ void cursor_next(const TilePlan& pl, const Cta& c, ChunkCursor& k) {
    k.x0 += pl.G[2];
    if (k.x0 >= c.nc[2] * pl.G[2]) {
        k.x0 = 0;
        k.z0 += pl.G[1];
        if (k.z0 >= c.nc[1] * pl.G[1]) {
            k.z0 = 0;
            k.y0 += pl.G[0];
        }
    }
}

template <int NB>
__device__ __forceinline__ ChunkMasks chunk_masks(const TilePlan& pl, const ChunkCursor& k, const WarpUnion& u,
                                                  const RowGeom& g, bool live) {
    constexpr int kSeg = (kMaxBlocks + NB - 1) / NB;
    ChunkMasks m;
    const uint32_t useg = segment_bits(pl, k.y0, k.z0, u.lo[0], u.hi[0], u.lo[1], u.hi[1]);
    // blocks of a segment that intersect the warp's column union
    const int xa = u.lo[2] - k.x0, xb = u.hi[2] - k.x0;
    const uint32_t ublk = xb > xa ? range_bits32(xa >> 3, (xb + 7) >> 3) & ((1u << NB) - 1u) : 0u;
    m.act = 0;
#pragma unroll
    for (int s = 0; s < kSeg; ++s) m.act |= ((useg >> s) & 1u) ? (ublk << (s * NB)) : 0u;
    m.rowseg = live ? segment_bits(pl, k.y0, k.z0, g.lo[0], g.lo[0] + g.len[0], g.lo[1], g.lo[1] + g.len[1]) : 0u;
    m.m8 = 0;
#pragma unroll
    for (int bb = 0; bb < NB; ++bb)
        m.m8 |= range_bits8(g.lo[2] - k.x0 - 8 * bb, g.lo[2] + g.len[2] - k.x0 - 8 * bb) << (8 * bb);
    return m;
}

// Live-column byte of block i (runtime) of the chunk for this row.
template <int NB>
__device__ __forceinline__ uint32_t block_live(const ChunkMasks& m, int i) {
    const int seg = i / NB, bb = i - seg * NB;
    return ((m.rowseg >> seg) & 1u) ? (m.m8 >> (8 * bb)) & 0xffu : 0u;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned* err, unsigned site) {
    const bool ok = mbar_wait(bar, parity, err, site);
    return __all_sync(0xffffffffu, ok);
}

// Byte offset of block i (columns 8i .. 8i+7) of this row in a K-major operand stored as 32-column
// atoms (128 rows x 64 B, 64-byte swizzle): rowbase = row * 64, sw = (row >> 1) & 3.
__device__ __forceinline__ uint32_t p_off(uint32_t rowbase, uint32_t sw, int i) {
    return static_cast<uint32_t>(i >> 2) * 8192u + rowbase + (((static_cast<uint32_t>(i) & 3u) ^ sw) << 4);
}

// Packed fp32x2 arithmetic (one instruction for two values).
__device__ __forceinline__ uint64_t f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_of(uint64_t r) {
    float a, b;
    f2_split(r, a, b);
    return pack_bf16x2(a, b);
}

// Scores of one block with the masked columns replaced by -inf.
__device__ __forceinline__ void mask_block(uint32_t (&v)[8], uint32_t live) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (!(live & (1u << e))) v[e] = 0xff800000u;  // -inf
}

// ---------------------------------------------------------------------------------------------
// Producer warp: TMA of tile tensors and halo chunks; for dK/dV also the per-column LSE / Delta.
// ---------------------------------------------------------------------------------------------

template <int D>
__device__ void producer_loop(const TcParams& p, int which, uint8_t* smem, const TcLayout& lay, uint64_t* bars) {
    const int lane = threadIdx.x & 31;
    unsigned* err = p.err;
    const TilePlan& pl = p.plan;
    const uint32_t tile_bytes = 128u * D * 2u, chunk_bytes = static_cast<uint32_t>(pl.NC) * D * 2u;
    const int ntile = which == 0 ? 1 : 2;
    const int tmCk = which == 0 ? 1 : 2, tmCv = which == 0 ? 2 : 3;
    TileIter it = tile_iter_begin(p);
    bool started = false;
    Cta c;
    uint32_t j = 0, g = 0;
    bool ok = true;
    while (ok && next_tile(p, which, it, started, c)) {
        const uint32_t qs = j & 1;
        if (j >= 2) ok = warp_wait(&bars[kQEmpty + qs], ((j >> 1) - 1) & 1, err, kSiteQ);
        if (!ok) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[kQFull + qs], ntile * tile_bytes);
            for (int tt = 0; tt < ntile; ++tt)
                tma_load_5d(smem + lay.tile(qs, tt), &p.tm[tt], &bars[kQFull + qs], c.h * D,
                            c.cls[2] + p.d[2] * c.t0[2], c.cls[1] + p.d[1] * c.t0[1], c.cls[0] + p.d[0] * c.t0[0],
                            c.b);
        }
        ChunkCursor cur{0, 0, 0};
        for (int ci = 0; ci < c.C; ++ci, ++g, cursor_next(pl, c, cur)) {
            const uint32_t s = g % kStages;
            if (g >= kStages) ok = warp_wait(&bars[kKVEmpty + s], ((g / kStages) - 1) & 1, err, kSiteEmpty);
            if (!ok) break;
            const int y0 = c.h0[0] + cur.y0, z0 = c.h0[1] + cur.z0, x0 = c.h0[2] + cur.x0;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[kKVFull + s], 2u * chunk_bytes);
                tma_load_5d(smem + lay.chunk(s, 0), &p.tm[tmCk], &bars[kKVFull + s], c.h * D,
                            c.cls[2] + p.d[2] * x0, c.cls[1] + p.d[1] * z0, c.cls[0] + p.d[0] * y0, c.b);
                tma_load_5d(smem + lay.chunk(s, 1), &p.tm[tmCv], &bars[kKVFull + s], c.h * D,
                            c.cls[2] + p.d[2] * x0, c.cls[1] + p.d[1] * z0, c.cls[0] + p.d[0] * y0, c.b);
            }
            if (which == 2) {
                // LSE (log2 units) and Delta of the chunk's queries; +inf LSE outside the class
                float* l2 = reinterpret_cast<float*>(smem + lay.aux(s));
                float* dl = l2 + pl.NC;
                for (int col = lane; col < pl.NC; col += 32) {
                    const int x2 = col % pl.G[2], x1 = (col / pl.G[2]) % pl.G[1], xx0 = col / (pl.G[2] * pl.G[1]);
                    const int j0 = y0 + xx0, j1 = z0 + x1, j2 = x0 + x2;
                    float lv = INFINITY, dv = 0.f;
                    if (j0 < c.Lc[0] && j1 < c.Lc[1] && j2 < c.Lc[2]) {
                        const long long tok =
                            ((static_cast<long long>(c.b) * p.L[0] + (c.cls[0] + p.d[0] * j0)) * p.L[1] +
                             (c.cls[1] + p.d[1] * j1)) * p.L[2] + (c.cls[2] + p.d[2] * j2);
                        lv = __ldg(p.lse + tok * p.heads + c.h) * kLog2e;
                        dv = __ldg(p.delta + tok * p.heads + c.h);
                    }
                    l2[col] = lv;
                    dl[col] = dv;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kKVFull + s]);
            }
        }
        ++j;
    }
}

// ---------------------------------------------------------------------------------------------
// MMA warp (lane 0): score products per chunk, update products of the previous chunk.
// ---------------------------------------------------------------------------------------------

template <int D>
struct MmaIssuer {
    const TcParams& p;
    uint8_t* smem;

    // D_tmem = A_tile(128 x D) * B_chunk(NC x D)^T, both K-major; A negated when `neg`.
    __device__ void rows_x_chunk(uint32_t d_tmem, uint32_t a_off, uint32_t b_off, bool neg) const {
        const uint32_t rowb = D * 2u, lay_ = swizzle_layout(D * 2), sbo = 8u * rowb;
        const uint32_t idesc = idesc_bf16(128, p.plan.NC, false, false) | (neg ? (1u << 13) : 0u);
        const uint32_t a = smem_u32(smem + a_off), b = smem_u32(smem + b_off);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            umma_bf16(d_tmem, sdesc(a + kk * 32u, 16u, sbo, lay_), sdesc(b + kk * 32u, 16u, sbo, lay_), idesc,
                      kk > 0);
    }
    // D_tmem (+)= P(128 x NC, 32-column atoms) * B_chunk(NC x D), B MN-major.
    __device__ void p_x_chunk(uint32_t d_tmem, uint32_t p_off, uint32_t b_off, bool accumulate) const {
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

// TMEM column bases.  fwd (256 columns): S[b] at b*NC, O[b] at 256 - (2 - b) * D.
// dQ (512): S[b] at b*NC, dP[b] at (2 + b)*NC, dQ[b] at 512 - (2 - b) * D.
// dKdV (512): S[b] at b*NC, dP[b] at (2 + b)*NC, dV[b] at 512 - (4 - 2b) * D, dK[b] = dV[b] + D.
__device__ __forceinline__ uint32_t tm_s(const TilePlan& pl, uint32_t b) { return b * pl.NC; }
__device__ __forceinline__ uint32_t tm_dp(const TilePlan& pl, uint32_t b) { return (2 + b) * pl.NC; }
template <int D>
__device__ __forceinline__ uint32_t tm_acc(int which, uint32_t b) {
    return which == 0 ? 256u - (2u - b) * D : (which == 1 ? 512u - (2u - b) * D : 512u - (4u - 2u * b) * D);
}

struct PendingUpdate {
    uint32_t g, s, j;
    int ci, C;
    bool valid;
};

template <int D>
__device__ void mma_loop(const TcParams& p, int which, uint8_t* smem, const TcLayout& lay, uint64_t* bars,
                         uint32_t tmem) {
    unsigned* err = p.err;
    const TilePlan& pl = p.plan;
    MmaIssuer<D> mi{p, smem};
    const bool neg = p.neg != 0;
    TileIter it = tile_iter_begin(p);
    bool started = false;
    Cta c;
    uint32_t j = 0, g = 0;
    PendingUpdate pend{0, 0, 0, 0, 0, false};
    bool ok = true;
    auto update = [&](const PendingUpdate& pd) -> bool {
        const uint32_t pb = pd.g & 1, ob = pd.j & 1;
        if (!mbar_wait(&bars[kPFull + pb], (pd.g >> 1) & 1, err, kSiteP)) return false;
        if (pd.ci == 0 && pd.j >= 2 && !mbar_wait(&bars[kOEmpty + ob], ((pd.j >> 1) - 1) & 1, err, kSitePV))
            return false;
        tc_fence_after();
        const uint32_t acc = tmem + tm_acc<D>(which, ob);
        if (which == 0) {
            mi.p_x_chunk(acc, lay.p(pb, 0), lay.chunk(pd.s, 1), pd.ci > 0);  // O += P V
        } else if (which == 1) {
            mi.p_x_chunk(acc, lay.p(pb, 0), lay.chunk(pd.s, 0), pd.ci > 0);  // dQ += dS K
        } else {
            mi.p_x_chunk(acc, lay.p(pb, 0), lay.chunk(pd.s, 1), pd.ci > 0);      // dV += P^T dO
            mi.p_x_chunk(acc + D, lay.p(pb, 1), lay.chunk(pd.s, 0), pd.ci > 0);  // dK += dS^T Q
        }
        umma_commit(&bars[kPEmpty + pb]);
        umma_commit(&bars[kKVEmpty + pd.s]);
        if (pd.ci == pd.C - 1) umma_commit(&bars[kOFull + ob]);
        return true;
    };
    while (ok && next_tile(p, which, it, started, c)) {
        const uint32_t qs = j & 1;
        if (!mbar_wait(&bars[kQFull + qs], (j >> 1) & 1, err, kSiteQ)) break;
        for (int ci = 0; ci < c.C && ok; ++ci, ++g) {
            const uint32_t s = g % kStages, sb = g & 1;
            ok = mbar_wait(&bars[kKVFull + s], (g / kStages) & 1, err, kSiteKV);
            if (ok && g >= 2) ok = mbar_wait(&bars[kSEmpty + sb], ((g >> 1) - 1) & 1, err, kSiteS);
            if (!ok) break;
            tc_fence_after();
            mi.rows_x_chunk(tmem + tm_s(pl, sb), lay.tile(qs, 0), lay.chunk(s, 0), neg);  // S (or S^T)
            if (which != 0) mi.rows_x_chunk(tmem + tm_dp(pl, sb), lay.tile(qs, 1), lay.chunk(s, 1), false);  // dP
            umma_commit(&bars[kSFull + sb]);
            if (ci == c.C - 1) umma_commit(&bars[kQEmpty + qs]);
            if (pend.valid) ok = update(pend);
            pend = PendingUpdate{g, s, j, ci, c.C, true};
        }
        ++j;
    }
    if (ok && pend.valid) update(pend);
}

// ---------------------------------------------------------------------------------------------
// Epilogue helpers
// ---------------------------------------------------------------------------------------------

// Stage columns [c0, c1) of this thread's accumulator row (fp32 at taddr) as bf16 in the tile
// layout of the tensor map (row-major [128][D], swizzle = row width).
template <int D>
__device__ __forceinline__ void stage_cols(uint32_t taddr, float mul, uint8_t* stage, int row, int c0, int c1) {
    const uint32_t base = smem_u32(stage), mask = swizzle_mask(D * 2);
#pragma unroll
    for (int cc = 0; cc < D; cc += 8) {
        if (cc < c0 || cc >= c1) continue;
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

__device__ __forceinline__ void tile_store(const TcParams& p, const Cta& c, int m, uint8_t* stage, int D) {
    tma_store_5d(&p.tm[m], stage, c.h * D, c.cls[2] + p.d[2] * c.t0[2], c.cls[1] + p.d[1] * c.t0[1],
                 c.cls[0] + p.d[0] * c.t0[0], c.b);
}

// ---------------------------------------------------------------------------------------------
// Forward softmax warps (4 warps, 128 rows)
// ---------------------------------------------------------------------------------------------

// Zero the P groups of the blocks in `mask` (blocks of the chunk no row of this warp needs).
__device__ __forceinline__ void zero_blocks(uint32_t sP, uint32_t rowbase, uint32_t sw, uint32_t mask) {
    while (mask) {
        const int i = __ffs(mask) - 1;
        mask &= mask - 1;
        st_shared_v4(sP + p_off(rowbase, sw, i), 0u, 0u, 0u, 0u);
    }
}

template <int D, int NB>
__device__ void fwd_softmax_loop(const TcParams& p, uint8_t* smem, const TcLayout& lay, uint64_t* bars,
                                 uint32_t tmem) {
    constexpr int kMB = fwd_max_blocks(D);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, row = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    unsigned* err = p.err;
    const TilePlan& pl = p.plan;
    const uint32_t all_blocks = (1u << (pl.NC >> 3)) - 1u;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    const uint32_t rowbase = static_cast<uint32_t>(row) * 64u, sw = (static_cast<uint32_t>(row) >> 1) & 3u;
    TileIter it = tile_iter_begin(p);
    bool started = false;
    Cta c;
    uint32_t j = 0, g = 0;
    bool ok = true;
    while (ok && next_tile(p, 0, it, started, c)) {
        const RowGeom geo = row_geom(p, 0, c, row);
        const WarpUnion u = warp_union(geo);
        const bool live = geo.len[0] > 0 && geo.len[1] > 0 && geo.len[2] > 0;
        const uint32_t ob = j & 1;
        const uint32_t tO = tmem + tm_acc<D>(0, ob);
        float m = -INFINITY;
        uint64_t lsum[4] = {0ull, 0ull, 0ull, 0ull};  // four packed partial sums (independent chains)
        ChunkCursor cur{0, 0, 0};
        for (int ci = 0; ci < c.C; ++ci, ++g, cursor_next(pl, c, cur)) {
            const uint32_t sb = g & 1;
            const uint32_t tS = tmem + tm_s(pl, sb) + lane_base;
            const ChunkMasks cm = chunk_masks<NB>(pl, cur, u, geo, live);
            const uint32_t act = cm.act & all_blocks;
            ok = warp_wait(&bars[kSFull + sb], (g >> 1) & 1, err, kSiteS);
            if (!ok) break;
            tc_fence_after();
            // the active blocks of the chunk, compacted into registers, one wait
            uint32_t val[kMB][8];
            int idx[kMB];
            const int nact = __popc(act);
            {
                uint32_t rem = act;
#pragma unroll
                for (int q = 0; q < kMB; ++q) {
                    idx[q] = rem ? __ffs(rem) - 1 : 0;
                    if (rem) {
                        tmem_ld8(tS + 8 * idx[q], val[q]);
                        rem &= rem - 1;
                    }
                }
            }
            tmem_ld_wait_all();
            // mask, then the chunk row max with one accumulator per column position
            float mx[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll
            for (int q = 0; q < kMB; ++q)
                if (q < nact) {
                    reg_fence8(val[q]);
                    mask_block(val[q], block_live<NB>(cm, idx[q]));
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], __uint_as_float(val[q][e]));
                }
            const float cmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            // running max (log2 units; the scale's sign is folded into the S product)
            const float cm2 = cmax * sl2;  // -inf when no live key
            const float mnew = fmaxf(m, cm2);
            const bool rescale = (m != -INFINITY) && (mnew > m + kRescaleThreshold);
            const float alpha = rescale ? fast_exp2(m - mnew) : 1.f;
            if (m == -INFINITY || rescale) m = mnew;
            if (__any_sync(0xffffffffu, rescale)) {
                // O holds the products of chunks g-1, g-2, ...: wait for the last one
                ok = warp_wait(&bars[kPEmpty + ((g - 1) & 1)], ((g - 1) >> 1) & 1, err, kSitePV);
                if (!ok) break;
                tc_fence_after();
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
                const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
                for (int t = 0; t < 4; ++t) lsum[t] = f2_mul(lsum[t], a2);
            }
            // P buffer sb is free once the product of chunk g-2 is done
            if (g >= 2) {
                ok = warp_wait(&bars[kPEmpty + sb], ((g >> 1) - 1) & 1, err, kSitePV);
                if (!ok) break;
            }
            const uint32_t sP = smem_u32(smem + lay.p(sb, 0));
            const float nm = m == -INFINITY ? 0.f : -m;  // masked scores are -inf: exp2 gives 0
            const uint64_t nm2 = f2(nm, nm);
#pragma unroll
            for (int q = 0; q < kMB; ++q)
                if (q < nact) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const uint64_t x =
                            f2_fma(f2(__uint_as_float(val[q][e]), __uint_as_float(val[q][e + 1])), sl2x2, nm2);
                        float xa, xb;
                        f2_split(x, xa, xb);
                        const uint64_t pe = f2(fast_exp2(xa), fast_exp2(xb));
                        lsum[e >> 1] = f2_add(lsum[e >> 1], pe);
                        w[e >> 1] = bf16x2_of(pe);
                    }
                    st_shared_v4(sP + p_off(rowbase, sw, idx[q]), w[0], w[1], w[2], w[3]);
                }
            zero_blocks(sP, rowbase, sw, all_blocks & ~act);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[kSEmpty + sb]);
                mbar_arrive(&bars[kPFull + sb]);
            }
        }
        if (!ok) break;
        // epilogue: O / l -> bf16 -> TMA store; LSE = (m + log2 l) * ln 2
        const uint64_t ls = f2_add(f2_add(lsum[0], lsum[1]), f2_add(lsum[2], lsum[3]));
        float la, lb;
        f2_split(ls, la, lb);
        const float l = la + lb;
        ok = warp_wait(&bars[kOFull + ob], (j >> 1) & 1, err, kSitePV);
        if (!ok) break;
        tc_fence_after();
        // the staging buffer is free once the previous tile's store has read it
        if (threadIdx.x == 0) {
            tma_store_wait_read();
            mbar_arrive(&bars[kStFree]);
        }
        ok = warp_wait(&bars[kStFree], j & 1, err, kSiteSt);
        if (!ok) break;
        stage_cols<D>(tO + lane_base, 1.f / l, smem + lay.stage(0), row, 0, D);
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&bars[kOEmpty + ob]);
            mbar_arrive(&bars[kStFull]);
        }
        if (geo.valid) p.lse_out[geo.token * p.heads + c.h] = (m + __log2f(l)) * kLn2;
        if (threadIdx.x == 0) {
            ok = mbar_wait(&bars[kStFull], j & 1, err, kSiteSt);
            if (ok) {
                tile_store(p, c, 3, smem + lay.stage(0), D);
                tma_store_commit();
            }
        }
        ok = __all_sync(0xffffffffu, ok);
        ++j;
    }
    if (threadIdx.x == 0) tma_store_wait_all();
}

// ---------------------------------------------------------------------------------------------
// Backward softmax warps (8 warps: two warpgroups split each chunk's active blocks)
// ---------------------------------------------------------------------------------------------

template <int D, int WHICH, int NB>
__device__ void bwd_softmax_loop(const TcParams& p, uint8_t* smem, const TcLayout& lay, uint64_t* bars,
                                 uint32_t tmem) {
    constexpr int kMB = 4;  // blocks per warpgroup held in registers at once (more passes if it has more)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wq = warp & 3, wg = warp >> 2;  // lane quarter, warpgroup
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    unsigned* err = p.err;
    const TilePlan& pl = p.plan;
    const uint32_t all_blocks = (1u << (pl.NC >> 3)) - 1u;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    const uint32_t rowbase = static_cast<uint32_t>(row) * 64u, sw = (static_cast<uint32_t>(row) >> 1) & 3u;
    TileIter it = tile_iter_begin(p);
    bool started = false;
    Cta c;
    uint32_t j = 0, g = 0;
    bool ok = true;
    while (ok && next_tile(p, WHICH, it, started, c)) {
        const RowGeom geo = row_geom(p, WHICH, c, row);
        const WarpUnion u = warp_union(geo);
        const bool live = geo.len[0] > 0 && geo.len[1] > 0 && geo.len[2] > 0;
        const uint32_t ob = j & 1;
        float lse2 = 0.f, dlt = 0.f;
        if (WHICH == 1 && geo.valid) {
            lse2 = __ldg(p.lse + geo.token * p.heads + c.h) * kLog2e;
            dlt = __ldg(p.delta + geo.token * p.heads + c.h);
        }
        const uint64_t nl2 = f2(-lse2, -lse2), dl2 = f2(dlt, dlt);
        ChunkCursor cur{0, 0, 0};
        for (int ci = 0; ci < c.C; ++ci, ++g, cursor_next(pl, c, cur)) {
            const uint32_t sb = g & 1, s = g % kStages;
            const uint32_t tS = tmem + tm_s(pl, sb) + lane_base, tP = tmem + tm_dp(pl, sb) + lane_base;
            const ChunkMasks cm = chunk_masks<NB>(pl, cur, u, geo, live);
            // active blocks alternate between the two warpgroups; each zeroes its share of the rest
            uint32_t act = cm.act & all_blocks, mine = 0, rest = 0;
            {
                uint32_t r = act;
                int k = 0;
                while (r) {
                    const uint32_t bit = r & (0u - r);
                    if ((k & 1) == wg) mine |= bit;
                    r ^= bit;
                    ++k;
                }
                const uint32_t idle = all_blocks & ~act;
                rest = idle & (wg == 0 ? 0x55555555u : 0xaaaaaaaau);
            }
            ok = warp_wait(&bars[kSFull + sb], (g >> 1) & 1, err, kSiteS);
            if (ok && g >= 2) ok = warp_wait(&bars[kPEmpty + sb], ((g >> 1) - 1) & 1, err, kSitePV);
            if (!ok) break;
            tc_fence_after();
            const uint32_t sP0 = smem_u32(smem + lay.p(sb, 0)), sP1 = smem_u32(smem + lay.p(sb, 1));
            const float* l2 = reinterpret_cast<const float*>(smem + lay.aux(s));
            const float* dl = l2 + pl.NC;
            while (mine) {
                uint32_t rs[kMB][8], rp[kMB][8];
                int idx[kMB];
                const int n = min(__popc(mine), kMB);
#pragma unroll
                for (int q = 0; q < kMB; ++q) {
                    idx[q] = mine ? __ffs(mine) - 1 : 0;
                    if (q < n) {
                        tmem_ld8(tS + 8 * idx[q], rs[q]);
                        tmem_ld8(tP + 8 * idx[q], rp[q]);
                        mine &= mine - 1;
                    }
                }
                tmem_ld_wait_all();
#pragma unroll
                for (int q = 0; q < kMB; ++q)
                    if (q < n) {
                        const int i = idx[q];
                        reg_fence8(rs[q]);
                        reg_fence8(rp[q]);
                        mask_block(rs[q], block_live<NB>(cm, i));
                        uint32_t a[4], b[4];
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            uint64_t nlc = nl2, dlc = dl2;
                            if (WHICH == 2) {
                                const float2 lv = *reinterpret_cast<const float2*>(l2 + 8 * i + e);
                                const float2 dv = *reinterpret_cast<const float2*>(dl + 8 * i + e);
                                nlc = f2(-lv.x, -lv.y);
                                dlc = f2(dv.x, dv.y);
                            }
                            const uint64_t x =
                                f2_fma(f2(__uint_as_float(rs[q][e]), __uint_as_float(rs[q][e + 1])), sl2x2, nlc);
                            float xa, xb;
                            f2_split(x, xa, xb);
                            const uint64_t pe = f2(fast_exp2(xa), fast_exp2(xb));
                            const uint64_t dp = f2(__uint_as_float(rp[q][e]), __uint_as_float(rp[q][e + 1]));
                            const uint64_t ds = f2_mul(pe, f2_sub(dp, dlc));
                            b[e >> 1] = bf16x2_of(ds);
                            if (WHICH == 2) a[e >> 1] = bf16x2_of(pe);
                        }
                        const uint32_t off = p_off(rowbase, sw, i);
                        if (WHICH == 2) {
                            st_shared_v4(sP0 + off, a[0], a[1], a[2], a[3]);  // P^T
                            st_shared_v4(sP1 + off, b[0], b[1], b[2], b[3]);  // dS^T
                        } else {
                            st_shared_v4(sP0 + off, b[0], b[1], b[2], b[3]);  // dS
                        }
                    }
            }
            zero_blocks(sP0, rowbase, sw, rest);
            if (WHICH == 2) zero_blocks(sP1, rowbase, sw, rest);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[kSEmpty + sb]);
                mbar_arrive(&bars[kPFull + sb]);
            }
        }
        if (!ok) break;
        // epilogue: each warpgroup stages half of the D columns of its quarter's rows
        ok = warp_wait(&bars[kOFull + ob], (j >> 1) & 1, err, kSitePV);
        if (!ok) break;
        tc_fence_after();
        if (threadIdx.x == 0) {
            tma_store_wait_read();
            mbar_arrive(&bars[kStFree]);
        }
        ok = warp_wait(&bars[kStFree], j & 1, err, kSiteSt);
        if (!ok) break;
        const uint32_t acc = tmem + tm_acc<D>(WHICH, ob) + lane_base;
        const int c0 = wg * (D / 2), c1 = c0 + D / 2;
        if (WHICH == 1) {
            stage_cols<D>(acc, p.scale, smem + lay.stage(0), row, c0, c1);  // dQ
        } else {
            stage_cols<D>(acc, 1.f, smem + lay.stage(1), row, c0, c1);          // dV
            stage_cols<D>(acc + D, p.scale, smem + lay.stage(0), row, c0, c1);  // dK
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&bars[kOEmpty + ob]);
            mbar_arrive(&bars[kStFull]);
        }
        if (threadIdx.x == 0) {
            ok = mbar_wait(&bars[kStFull], j & 1, err, kSiteSt);
            if (ok) {
                if (WHICH == 1) {
                    tile_store(p, c, 4, smem + lay.stage(0), D);
                } else {
                    tile_store(p, c, 4, smem + lay.stage(0), D);  // dK
                    tile_store(p, c, 5, smem + lay.stage(1), D);  // dV
                }
                tma_store_commit();
            }
        }
        ok = __all_sync(0xffffffffu, ok);
        ++j;
    }
    if (threadIdx.x == 0) tma_store_wait_all();
}

// ---------------------------------------------------------------------------------------------
// Kernels
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

template <int WHICH>
__device__ __forceinline__ void init_barriers(uint64_t* bars) {
    constexpr uint32_t kSoft = 4 * nwg_of(WHICH);
    for (int i = 0; i < 2; ++i) {
        mbar_init(&bars[kQFull + i], 1);
        mbar_init(&bars[kQEmpty + i], 1);
        mbar_init(&bars[kSFull + i], 1);
        mbar_init(&bars[kSEmpty + i], kSoft);
        mbar_init(&bars[kPFull + i], kSoft);
        mbar_init(&bars[kPEmpty + i], 1);
        mbar_init(&bars[kOFull + i], 1);
        mbar_init(&bars[kOEmpty + i], kSoft);
    }
    for (int s = 0; s < kStages; ++s) {
        mbar_init(&bars[kKVFull + s], WHICH == 2 ? 2 : 1);
        mbar_init(&bars[kKVEmpty + s], 1);
    }
    mbar_init(&bars[kStFree], 1);
    mbar_init(&bars[kStFull], kSoft);
    mbar_init(&bars[kFin], 1);
    fence_barrier_init();
}

template <int D, int WHICH, int NB>
__global__ void __launch_bounds__(threads_of(WHICH), WHICH == 0 ? 2 : 1) tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    const TilePlan& pl = p.plan;
    const TcLayout lay = tc_layout(WHICH, pl, D);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    constexpr int kSoftWarps = 4 * nwg_of(WHICH);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tmem_cols = WHICH == 0 ? 256u : 512u;

    if (warp == kSoftWarps) {
        if (lane == 0) {
            init_barriers<WHICH>(bars);
            for (int m = 0; m < 6; ++m) tma_prefetch_desc(&p.tm[m]);
        }
        __syncwarp();
    }
    if (warp == kSoftWarps + 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kSoftWarps) {
        producer_loop<D>(p, WHICH, smem, lay, bars);
    } else if (warp == kSoftWarps + 1) {
        if (lane == 0) mma_loop<D>(p, WHICH, smem, lay, bars, tmem);
        __syncwarp();
    } else if (WHICH == 0) {
        fwd_softmax_loop<D, NB>(p, smem, lay, bars, tmem);
    } else {
        bwd_softmax_loop<D, WHICH, NB>(p, smem, lay, bars, tmem);
    }

    // teardown: every MMA of this CTA done before TMEM is freed
    if (warp == kSoftWarps + 1 && lane == 0) {
        umma_commit(&bars[kFin]);
        mbar_wait(&bars[kFin], 0, p.err, kSiteFinal);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kSoftWarps + 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

template <int D, int WHICH, int NB>
int launch_tc_nb(const TcParams& p0, cudaStream_t stream) {
    const int smem = p0.plan.smem_bytes;
    auto kernel = tc_kernel<D, WHICH, NB>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (p0.plan.ctas <= 0) return 0;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return static_cast<int>(e);
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return static_cast<int>(e);
    const long long per_sm = p0.plan.per_sm;
    const long long grid = p0.plan.ctas < per_sm * sms ? p0.plan.ctas : per_sm * sms;
    // the grid size written in the tile index's mixed radix
    TcParams p = p0;
    uint32_t x = static_cast<uint32_t>(grid);
    for (int i = 0; i < 8; ++i) {
        p.step[i] = x % p.rad[i];
        x /= p.rad[i];
    }
    kernel<<<dim3(static_cast<unsigned>(grid)), dim3(threads_of(WHICH)), smem, stream>>>(p);
    return static_cast<int>(cudaGetLastError());
}

template <int D, int WHICH>
int launch_tc(const TcParams& p, cudaStream_t stream) {
    switch (p.plan.NB) {
        case 1: return launch_tc_nb<D, WHICH, 1>(p, stream);
        case 2: return launch_tc_nb<D, WHICH, 2>(p, stream);
        case 3: return launch_tc_nb<D, WHICH, 3>(p, stream);
        case 4: return launch_tc_nb<D, WHICH, 4>(p, stream);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace

uint32_t tc_smem_bytes(int which, const TilePlan& pl, int D) { return tc_layout(which, pl, D).total + 1024u; }

int tc_tmem_cols(int which) { return which == 0 ? 256 : 512; }

int tc_max_nc(int which, int D) {
    // double-buffered score accumulators plus double-buffered tile accumulators
    const int cols = tc_tmem_cols(which);
    const int nc = which == 0 ? 8 * fwd_max_blocks(D) : (which == 1 ? (cols - 2 * D) / 4 : (cols - 4 * D) / 4);
    return (nc < 8 * kMaxBlocks ? nc : 8 * kMaxBlocks) / 16 * 16;
}

int launch_fwd_tc(const TcParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_tc<16, 0>(p, s);
        case 32: return launch_tc<32, 0>(p, s);
        case 64: return launch_tc<64, 0>(p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dq_tc(const TcParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_tc<16, 1>(p, s);
        case 32: return launch_tc<32, 1>(p, s);
        case 64: return launch_tc<64, 1>(p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

int launch_dkdv_tc(const TcParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_tc<16, 2>(p, s);
        case 32: return launch_tc<32, 2>(p, s);
        case 64: return launch_tc<64, 2>(p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace na
