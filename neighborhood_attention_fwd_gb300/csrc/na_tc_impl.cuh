// na_tc_impl.cuh -- tensor-core (tcgen05 / TMEM / TMA) kernels of libna for bf16 or fp16 tensors on
// sm_103a: the query-tile forward, the dQ pass over query tiles and the atomic-free dK/dV pass over
// key tiles.  Included by na_tc.cu (bf16 instantiations) and na_tc_f16.cu (fp16 instantiations).
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
//   * the window mask costs the softmax nothing: it is one more tensor-core product per chunk
//     and axis, S += A_bias B_bias^T, where B_bias holds the one-hot local coordinate of every
//     chunk column and A_bias, per row, 0 inside the row's window and -2^100 outside.  A_bias
//     depends on the tile only through its position relative to the borders, so it is built once
//     and rebuilt only along the axes whose border situation changes;
//   * each softmax warp owns 32 TMEM lanes (32 rows) and reads, per chunk, only the contiguous run
//     of 16-column groups that holds the keys of its rows' windows; the rest of its P rows is zero.
//
// Pipeline (persistent CTAs, each looping over tiles):
//   producer warp : TMA of the tile tensors (2-slot ring) and of halo chunks (stage ring); the
//                   window-bias operand when a tile's border situation differs from the last one
//   MMA warp      : per chunk the "score" products (and the bias products) into a double-buffered
//                   TMEM accumulator, then the previous chunk's "update" products into a
//                   double-buffered tile accumulator
//   softmax warps : per chunk read scores from TMEM and write P (forward: into the same TMEM
//                   buffer, over the scores; backward: dS, or P^T and dS^T, to a double-buffered
//                   smem operand); per tile read the accumulator and store it.
// Every mbarrier wait is bounded (see na_device.cuh); a wait that gives up records the site in the
// status word and the CTA stops issuing work.
#pragma once
#include <cmath>
#include <cuda_fp16.h>

#include "na_device.cuh"
#include "na_internal.h"

namespace na {
using namespace dev;

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: keep a stale running max until it is 2^8 off
constexpr int kMaxStages = 5;
// Decoded tile records in flight: the producer decodes every tile once and publishes it; the other
// roles read it instead of decoding it themselves (a decode costs a warp hundreds of cycles, and at a
// tile boundary it sits on the critical path of the MMA issuers and the softmax warps).
constexpr uint32_t kTileRing = 4;

// Halo chunk ring depth.  The chunk ring must cover the P pipeline plus the copy latency: at
// D <= 32 five stages for dQ, four for dK/dV (two P operands per chunk) and three for the forward,
// whose two P operands are its two TMEM score buffers (P is written over the scores); two at
// D >= 64.  (A fourth forward stage measured the same; a fifth dQ stage: 3D 16x256^2 dQ 2.19 -> 2.09 ms.)
__host__ __device__ constexpr int stages_of(int which, int D) { return D <= 32 ? (which == 0 ? 3 : (which == 1 ? 5 : 4)) : 2; }
// Backward chunk ownership: the two warpgroups take alternate chunks (warpgroup w the chunks g with
// g mod 2 == w), each covering its quarter's whole run, so the per-chunk work of waits, run geometry
// and hand-offs is paid once per chunk and quarter.  Chunk g uses P buffer g mod pbufs: dQ two per
// warpgroup, dK/dV (two P operands per buffer) one per warpgroup.
__host__ __device__ constexpr bool alt_of(int which) { return which != 0; }
__host__ __device__ constexpr int pbufs_of(int which) { return which == 1 ? 4 : 2; }
// Score buffers in TMEM: two, or (the forward at D <= 32, when its plan asks for it) three.  Three
// 64-column chunks and the two accumulators fill the forward's 256 columns; the score product into a
// buffer then waits for the P V product of the chunk three back instead of two back.  The forward's P
// buffers are its score buffers.
// D = 128: every tensor of D channels is held as two halves of 64 channels (128-byte rows, the
// 128-byte swizzle's width), each laid out exactly like a D = 64 operand; the products over D run
// once per half.
__host__ __device__ constexpr int dhalf_of(int D) { return D > 64 ? 64 : D; }
// Tile-ring slots and tile-accumulator buffers.  At D = 128 the backward's tiles (two tensors of
// 32 KB) leave shared memory for one tile slot, and dK/dV's accumulators (2 x 128 columns) fill half
// of TMEM, so they are single-buffered and each tile's epilogue runs as soon as its chunks are done.
__host__ __device__ constexpr int tslots_of(int which, int D) { return which != 0 && D > 64 ? 1 : 2; }
__host__ __device__ constexpr int abufs_of(int which, int D) { return which == 2 && D > 64 ? 1 : 2; }
// TMEM columns per CTA: the forward takes 256 (two CTAs per SM) up to D = 64.
__host__ __device__ constexpr int tmem_cols_of(int which, int D) { return which == 0 && D <= 64 ? 256 : 512; }
constexpr int kMaxPBufs = 4;
// Softmax warpgroups: the forward's four warps own one TMEM lane quarter each; in the backward
// kBwdGroups warpgroups share every quarter's groups, warpgroup w taking groups w, w + kBwdGroups, ...
constexpr int kBwdGroups = 2;
static_assert(kBwdGroups >= 2, "the backward epilogue stores half of the D columns per warpgroup 0 and 1");
static_assert(kBwdGroups == 2, "alternate chunks pair two warpgroups");
// Warps that read and release each chunk's scores and write its P operand.
__host__ __device__ constexpr int chunk_warps_of(int which) { return which == 0 || alt_of(which) ? 4 : 4 * kBwdGroups; }
// Distance between the groups one warp takes within a run.
__host__ __device__ constexpr int group_stride_of(int which) { return alt_of(which) ? 1 : kBwdGroups; }
__host__ __device__ constexpr int nwg_of(int which) { return which == 0 ? 1 : kBwdGroups; }
// Warps that issue update products (O, dQ; or dV and dK), one per accumulator, beside the warp issuing
// score products.  A single lane waits tens of cycles on each tcgen05.mma it issues, and it shares its
// SM sub-partition with softmax warps, so products into independent accumulators are issued by
// different warps.
__host__ __device__ constexpr int nupd_of(int which) { return which == 2 ? 2 : 1; }
// The forward adds one idle warp so that its control warps fill the second warpgroup: the two
// warpgroups then take different register budgets (setmaxnreg), the softmax warps the larger.
__host__ __device__ constexpr int threads_of(int which) {
    return 32 * (4 * nwg_of(which) + 2 + nupd_of(which) + (which == 0 ? 1 : 0));
}
// Forward register budgets per thread: softmax warpgroup and control warpgroup.  Two CTAs of 256
// threads launch with 128 registers each; the two budgets sum to twice that.
constexpr uint32_t kFwdSoftRegs = 160, kFwdCtrlRegs = 96;
static_assert(kFwdSoftRegs + kFwdCtrlRegs == 2 * 128, "the forward's split must fit its launch registers");

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Window-bias operands.  Along every axis whose halo is longer than one position, a chunk column's
// local coordinate (< G[a] <= 32) is one-hot encoded in nbg[a] 16-column groups of the constant
// operand B; the per-tile operand A holds, for every row, chunk index along the axis and group,
// 0 where the coordinate is inside the row's window and -2^100 elsewhere.  Both are K-major
// 16-column blocks with 32-byte swizzle: A groups of 128 rows (4 KB), B groups of NC rows.
struct BiasGeom {
    int nbg[3];    // groups per chunk along each axis (0: the axis needs no mask)
    int abase[3];  // first A group of each axis (A group = abase + chunk index * nbg + group)
    int bbase[3];  // first B group of each axis
    int na, nb;    // A groups, B groups
};

__host__ __device__ inline BiasGeom bias_geom(const TilePlan& pl) {
    BiasGeom b{};
    for (int a = 0; a < 3; ++a) {
        b.nbg[a] = pl.H[a] > 1 ? (pl.G[a] + 15) / 16 : 0;
        b.abase[a] = b.na;
        b.bbase[a] = b.nb;
        b.na += pl.nchk[a] * b.nbg[a];
        b.nb += b.nbg[a];
    }
    return b;
}

// Element types: bf16 or fp16 operands (the same 2-byte layouts), fp32 accumulation.  The window
// bias needs 1.0 and a large finite negative value in the operand type.
__host__ __device__ constexpr uint32_t elem_one(bool f16) { return f16 ? 0x3C00u : 0x3F80u; }  // 1.0
__host__ __device__ constexpr uint32_t elem_neg(bool f16) { return f16 ? 0xFBFFu : 0xF180u; }  // -65504 / -2^100
// A chunk maximum below this means "no live key": masked scores are at most the bias plus the
// largest live |score|, so fp16 operands support |scale q.k| < 3.2e4.
template <bool F16>
__host__ __device__ constexpr float masked_below() { return F16 ? -3.2e4f : -1.0e29f; }

// Shared-memory layout (offsets from a 1024-byte aligned base).
//   which 0 (fwd) : tile ring [2] x {Q};     chunk ring [S] x {K, V}   (P is written to TMEM)
//   which 1 (dQ)  : tile ring [2] x {Q, dO}; chunk ring [S] x {K, V};  dS[2]
//   which 2 (dKdV): tile ring [2] x {K, V};  chunk ring [S] x {Q, dO}; P^T[2], dS^T[2];
//                   per softmax warpgroup two buffers of the -LSE (log2 units) and Delta of the
//                   queries of its current chunk
//   all: window-bias operands A (per tile) and B (constant).
struct TcLayout {
    uint32_t tile0, tile_slot, tile_t;     // tile ring: tile0 + slot * tile_slot + tensor * tile_t
    uint32_t tile_h, chunk_h;              // offset of the second 64-channel half of a tile / chunk tensor (D = 128)
    uint32_t chunk0, chunk_slot, chunk_t;  // chunk ring
    uint32_t p0, p_buf, p_op;              // P / dS operands
    uint32_t abias, bbias, bgroup;         // window-bias operands; bgroup = bytes of one B group
    uint32_t aux0, aux_slot;               // dK/dV: -LSE (log2) and Delta, buffer 2 wg + b
    uint32_t tinfo;                        // ring of decoded tile records (kTileRing x 128 bytes)
    uint32_t bars, total;
    __host__ __device__ uint32_t tile(uint32_t slot, uint32_t t) const { return tile0 + slot * tile_slot + t * tile_t; }
    __host__ __device__ uint32_t chunk(uint32_t slot, uint32_t t) const {
        return chunk0 + slot * chunk_slot + t * chunk_t;
    }
    __host__ __device__ uint32_t p(uint32_t buf, uint32_t op) const { return p0 + buf * p_buf + op * p_op; }
    __host__ __device__ uint32_t aux(uint32_t slot) const { return aux0 + slot * aux_slot; }
};

__host__ __device__ inline TcLayout tc_layout(int which, const TilePlan& pl, int D) {
    const uint32_t tile = align_up(128u * D * 2u, 1024);
    const uint32_t chunk = align_up(static_cast<uint32_t>(pl.NC) * D * 2u, 1024);
    const uint32_t pbytes = static_cast<uint32_t>((pl.NC + 31) / 32) * 8192u;
    const uint32_t ntile = which == 0 ? 1 : 2, nop = which == 2 ? 2 : 1;
    const BiasGeom bg = bias_geom(pl);
    TcLayout L{};
    uint32_t o = 0;
    L.tile0 = o;
    L.tile_t = tile;
    L.tile_slot = ntile * tile;
    L.tile_h = 128u * static_cast<uint32_t>(dhalf_of(D)) * 2u;
    L.chunk_h = static_cast<uint32_t>(pl.NC) * static_cast<uint32_t>(dhalf_of(D)) * 2u;
    o += static_cast<uint32_t>(tslots_of(which, D)) * L.tile_slot;
    L.chunk0 = o;
    L.chunk_t = chunk;
    L.chunk_slot = 2 * chunk;
    o += stages_of(which, D) * L.chunk_slot;
    L.p0 = o;
    L.p_op = pbytes;
    L.p_buf = nop * pbytes;
    if (which != 0) o += pbufs_of(which) * L.p_buf;  // the forward's P lives in TMEM, over its scores
    L.abias = o;
    o += static_cast<uint32_t>(bg.na) * 4096u;
    L.bbias = o;
    L.bgroup = static_cast<uint32_t>(pl.NC) * 32u;
    o += align_up(static_cast<uint32_t>(bg.nb) * L.bgroup, 1024);
    L.aux0 = o;
    L.aux_slot = which == 2 ? align_up(8u * static_cast<uint32_t>(pl.NC), 128) : 0u;
    o += align_up(2u * kBwdGroups * L.aux_slot, 1024);
    L.tinfo = o;
    o += kTileRing * 128u;
    L.bars = o;
    o += 512;
    L.total = o;
    return L;
}

// mbarrier indices
enum Bar {
    kQFull = 0, kQEmpty = 2, kKVFull = 4, kKVEmpty = 4 + kMaxStages, kSFull = 4 + 2 * kMaxStages,
    kSEmpty = kSFull + 2, kPFull = kSEmpty + 2, kPEmpty = kPFull + kMaxPBufs, kOFull = kPEmpty + kMaxPBufs,
    kOEmpty = kOFull + 2, kTFull = kOEmpty + 2, kTEmpty = kTFull + kTileRing,
    kFin = kTEmpty + kTileRing, kAuxSync = kFin + 1, kNumBars = kAuxSync + kBwdGroups
};
// The forward's third score buffer (three-buffer plans) has its score-full barrier at kSFull + 2, the
// first score-empty slot: the forward releases its buffers through the P V product's barrier and
// never uses the score-empty ones.

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
struct alignas(16) Cta {
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
        c.Lc[a] = p.Lc_tab[a][c.cls[a]];
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
        // chunks from the halo start to the last needed position: (hi - h0) / G + 1
        const uint32_t x = static_cast<uint32_t>(hi - c.h0[a] + pl.G[a]);
        c.nc[a] = min(pl.nchk[a], static_cast<int>(pl.G[a] == 1 ? x : __umulhi(x, p.rcpG[a])));
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

// Border situation of a tile along one axis: 0 when every row is inside the class, every row's
// window (or inverse window) is the unclamped one and the halo starts at the window of the tile's
// first row -- then the rows' ranges relative to the halo are the same for every such tile --
// otherwise a code of (t0, Lc), which fixes them.
__device__ __forceinline__ uint64_t axis_sig(int which, int t0, int T, int Lc, int k, int H) {
    const int r = k >> 1;
    bool in = t0 + T <= Lc && t0 - r <= Lc - H;
    if (which != 2) {
        in = in && t0 >= r && t0 + T - 1 <= Lc - 1 - r;
    } else {
        in = in && t0 >= k && t0 + T - 1 < Lc - k;
    }
    return in ? 0ull : ((static_cast<uint64_t>(static_cast<uint32_t>(Lc)) << 32) | static_cast<uint32_t>(t0 + 1));
}

// Per-row geometry: for each axis the halo-coordinate range [lo, lo + len) of keys (fwd, dQ: the
// query's window) or queries (dK/dV: the queries whose windows hold the key) of this row.  For dQ
// and dK/dV a row past the end of an axis has len = 0 along that axis (its P row is zero); the
// range along an axis depends on that axis alone.
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
        const bool in = j < c.Lc[a];
        if (!in) g.valid = false;
        const int jc = min(j, c.Lc[a] - 1);
        if (which != 2) {
            g.lo[a] = win_start(jc, c.Lc[a], p.k[a]) - c.h0[a];
            g.len[a] = p.k[a];
        } else {
            g.lo[a] = inv_lo(jc, p.k[a]) - c.h0[a];
            g.len[a] = inv_hi(jc, c.Lc[a], p.k[a]) - inv_lo(jc, p.k[a]) + 1;
        }
        if (!in && which != 0) g.len[a] = 0;
        tok = tok * p.L[a] + (c.cls[a] + p.d[a] * jc);
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

// Chunk cursor: chunk indices along each axis and the chunk origin in halo coordinates, stepped in
// chunk-grid order (axis 0 slowest, axis 2 fastest) without divisions.
struct ChunkCursor {
    int ix[3];
    int o[3];
};
__device__ __forceinline__ ChunkCursor cursor_begin() { return ChunkCursor{{0, 0, 0}, {0, 0, 0}}; }
__device__ __forceinline__ void cursor_next(const TilePlan& pl, const Cta& c, ChunkCursor& k) {
    ++k.ix[2];
    k.o[2] += pl.G[2];
    if (k.ix[2] >= c.nc[2]) {
        k.ix[2] = 0;
        k.o[2] = 0;
        ++k.ix[1];
        k.o[1] += pl.G[1];
        if (k.ix[1] >= c.nc[1]) {
            k.ix[1] = 0;
            k.o[1] = 0;
            ++k.ix[0];
            k.o[0] += pl.G[0];
        }
    }
}

// Steps a cursor N chunks on.
template <int N>
__device__ __forceinline__ void cursor_steps(const TilePlan& pl, const Cta& c, ChunkCursor& k) {
#pragma unroll
    for (int i = 0; i < N; ++i) cursor_next(pl, c, k);
}

// The run of 16-column groups [glo, glo + n) of a chunk that holds every key (column) inside the
// union of a warp's windows.  Chunk column = (y * G1 + z) * G2 + x for local coordinates (y, z, x).
__device__ __forceinline__ void chunk_range(const TilePlan& pl, const ChunkCursor& k, const WarpUnion& u, int& glo,
                                            int& n) {
    int lo[3], hi[3];
    bool empty = false;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        lo[a] = max(u.lo[a] - k.o[a], 0);
        hi[a] = min(u.hi[a] - k.o[a], pl.G[a]);
        if (lo[a] >= hi[a]) empty = true;
    }
    if (empty) {
        glo = 0;
        n = 0;
        return;
    }
    const int clo = (lo[0] * pl.G[1] + lo[1]) * pl.G[2] + lo[2];
    const int chi = ((hi[0] - 1) * pl.G[1] + hi[1] - 1) * pl.G[2] + hi[2];
    glo = clo >> 4;
    n = ((chi + 15) >> 4) - glo;
}

// bf16 pair for bits (2w, 2w+1) of `bits`: `v` where the bit is set, 0 elsewhere.
__device__ __forceinline__ uint32_t bf16_pair(uint32_t bits, int w, uint32_t v) {
    const uint32_t two = (bits >> (2 * w)) & 3u;
    return ((two & 1u) | ((two & 2u) << 15)) * v;
}

// Row r of a K-major 16-column bf16 block with 32-byte swizzle (32-byte rows, base 256-byte
// aligned): element t = `v` where bit t of `bits` is set, 0 elsewhere.
__device__ __forceinline__ void st_row32(uint32_t blk, int r, uint32_t bits, uint32_t v) {
    const uint32_t row = blk + static_cast<uint32_t>(r) * 32u;
    const uint32_t sw = (static_cast<uint32_t>(r) >> 2) & 1u;
    st_shared_v4(row + (sw << 4), bf16_pair(bits, 0, v), bf16_pair(bits, 1, v), bf16_pair(bits, 2, v),
                 bf16_pair(bits, 3, v));
    st_shared_v4(row + ((sw ^ 1u) << 4), bf16_pair(bits, 4, v), bf16_pair(bits, 5, v), bf16_pair(bits, 6, v),
                 bf16_pair(bits, 7, v));
}

// Whole-warp wait.  The common case, a phase that is already complete, takes one test and one vote.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitGuard& err, unsigned site) {
    if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
    const bool ok = mbar_block(bar, parity, err, site);
    return __all_sync(0xffffffffu, ok);
}

// Tile record j of this CTA from the producer's ring.  `warp`: the whole warp waits and reads (lane 0
// releases the slot), else a single lane does.  Returns false after the last tile, or when a wait
// gives up (then `ok` is false).
__device__ __forceinline__ bool fetch_tile(uint8_t* smem, const TcLayout& lay, uint64_t* bars, uint32_t j,
                                           const WaitGuard& err, bool warp, Cta& c, bool& ok) {
    const uint32_t ts = j % kTileRing, par = (j / kTileRing) & 1u;
    ok = warp ? warp_wait(&bars[kTFull + ts], par, err, kSiteQ) : mbar_wait(&bars[kTFull + ts], par, err, kSiteQ);
    if (!ok) return false;
    c = *reinterpret_cast<const Cta*>(smem + lay.tinfo + ts * 128u);
    if (warp) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&bars[kTEmpty + ts]);
    } else {
        mbar_arrive(&bars[kTEmpty + ts]);
    }
    return c.C > 0;
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
// Two fp32 values rounded to the operand type, packed (first value in the low half).
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (F16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        return pack_bf16x2(lo, hi);
    }
}
template <bool F16>
__device__ __forceinline__ uint32_t x2_of(uint64_t r) {
    float a, b;
    f2_split(r, a, b);
    return pack2<F16>(a, b);
}

// Instruction descriptor of kind::f16 with fp32 D and bf16 (f16 = false) or fp16 A and B.
__device__ __forceinline__ uint32_t idesc_mma(int M, int N, bool a_mn, bool b_mn, bool f16) {
    const uint32_t d = idesc_bf16(M, N, a_mn, b_mn);
    return f16 ? (d & ~((7u << 7) | (7u << 10))) : d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 32 lanes x 16 consecutive columns of 32 bits (one row per lane), and the register fence that
// keeps uses of them below the tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}

// ---------------------------------------------------------------------------------------------
// Window-bias operands (built by the producer warp)
// ---------------------------------------------------------------------------------------------

// Constant operand B: per chunk column its local coordinate along each masked axis, one-hot.
__device__ void build_bias_b(const TilePlan& pl, const BiasGeom& bg, uint32_t bbias, uint32_t bgroup, int lane,
                             bool f16) {
    for (int key = lane; key < pl.NC; key += 32) {
        const int loc[3] = {key / (pl.G[2] * pl.G[1]), (key / pl.G[2]) % pl.G[1], key % pl.G[2]};
        for (int a = 0; a < 3; ++a)
            for (int q = 0; q < bg.nbg[a]; ++q) {
                const int t = loc[a] - 16 * q;
                const uint32_t bits = (t >= 0 && t < 16) ? (1u << t) : 0u;
                st_row32(bbias + static_cast<uint32_t>(bg.bbase[a] + q) * bgroup, key, bits, elem_one(f16));
            }
    }
}

// Per-tile operand A along the axes in `axes`: for each row, chunk index and group, -2^100 at the
// coordinates outside the row's range along that axis.
__device__ void build_bias_a(const TcParams& p, int which, const Cta& c, const BiasGeom& bg, uint32_t abias,
                             int lane, uint32_t axes) {
    const uint32_t neg = elem_neg(p.f16 != 0);
    const TilePlan& pl = p.plan;
    for (int q = 0; q < 4; ++q) {
        const int r = lane + 32 * q;
        const RowGeom rg = row_geom(p, which, c, r);
        for (int a = 0; a < 3; ++a) {
            if (!((axes >> a) & 1u)) continue;
            for (int ch = 0; ch < pl.nchk[a]; ++ch)
                for (int qq = 0; qq < bg.nbg[a]; ++qq) {
                    const int o = ch * pl.G[a] + 16 * qq;
                    const uint32_t nv = ~range_bits32(rg.lo[a] - o, rg.lo[a] + rg.len[a] - o);
                    const uint32_t grp = static_cast<uint32_t>(bg.abase[a] + ch * bg.nbg[a] + qq);
                    st_row32(abias + grp * 4096u, r, nv, neg);
                }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Producer warp: TMA of tile tensors and halo chunks; the window-bias operands; for dK/dV also the
// per-column LSE / Delta of each chunk.
// ---------------------------------------------------------------------------------------------

// dK/dV: the -LSE and Delta of one chunk column (the queries of a chunk are its columns).  The
// softmax warpgroup that owns a chunk loads them, one column per thread (column 32 wq + lane), and
// shares them through shared memory.  Column t's element offset from the chunk origin is fixed for
// the launch (ce); a chunk adds its origin and a tile its halo origin and head.
struct AuxCol {
    long long ce;      // element offset of the column from the chunk origin
    long long ax[3];   // element step of one class position along each axis
    int loc[3];        // local coordinates of the column in the chunk
    bool col;          // t < NC
    float l, dl;       // loaded values (valid when `in`)
    bool in;           // the column is inside the class
};

__device__ __forceinline__ void aux_init(const TcParams& p, AuxCol& a, int t) {
    const TilePlan& pl = p.plan;
    const long long st[3] = {static_cast<long long>(p.L[1]) * p.L[2], p.L[2], 1};
#pragma unroll
    for (int i = 0; i < 3; ++i) a.ax[i] = st[i] * p.d[i] * p.heads;
    a.col = t < pl.NC;
    const int cc = min(t, pl.NC - 1);
    a.loc[0] = cc / (pl.G[2] * pl.G[1]);
    a.loc[1] = (cc / pl.G[2]) % pl.G[1];
    a.loc[2] = cc % pl.G[2];
    a.ce = a.loc[0] * a.ax[0] + a.loc[1] * a.ax[1] + a.loc[2] * a.ax[2];
}

// Element index of the tile's halo origin (head c.h).
__device__ __forceinline__ long long aux_tile_base(const TcParams& p, const Cta& c) {
    return (((static_cast<long long>(c.b) * p.L[0] + (c.cls[0] + p.d[0] * c.h0[0])) * p.L[1] +
             (c.cls[1] + p.d[1] * c.h0[1])) * p.L[2] + (c.cls[2] + p.d[2] * c.h0[2])) * p.heads + c.h;
}

// Issue the loads of the column's LSE and Delta for the chunk at cursor k of tile c (base tb).
__device__ __forceinline__ void aux_load(const TcParams& p, const Cta& c, long long tb, const ChunkCursor& k,
                                         AuxCol& a) {
    a.in = a.col && a.loc[0] < c.Lc[0] - c.h0[0] - k.o[0] && a.loc[1] < c.Lc[1] - c.h0[1] - k.o[1] &&
           a.loc[2] < c.Lc[2] - c.h0[2] - k.o[2];
    if (a.in) {
        const long long e = tb + k.o[0] * a.ax[0] + k.o[1] * a.ax[1] + k.o[2] * a.ax[2] + a.ce;
        a.l = __ldg(p.lse + e);
        a.dl = __ldg(p.delta + e);
    }
}

// Publish tile record j (c), or the end record (c == nullptr), once every reader of record
// j - kTileRing has released its slot.
__device__ __forceinline__ bool publish_tile(uint8_t* smem, const TcLayout& lay, uint64_t* bars, uint32_t j,
                                             const WaitGuard& err, int lane, const Cta* c) {
    const uint32_t ts = j % kTileRing;
    if (j >= kTileRing && !warp_wait(&bars[kTEmpty + ts], ((j / kTileRing) - 1) & 1u, err, kSiteQ)) return false;
    if (lane == 0) {
        Cta* dst = reinterpret_cast<Cta*>(smem + lay.tinfo + ts * 128u);
        if (c) {
            *dst = *c;
        } else {
            dst->C = 0;
        }
        mbar_arrive(&bars[kTFull + ts]);
    }
    __syncwarp();
    return true;
}

template <int D, int WHICH>
__device__ void producer_loop(const TcParams& p, uint8_t* smem, const TcLayout& lay, uint64_t* bars) {
    constexpr int kS = stages_of(WHICH, D);
    constexpr uint32_t kTS = tslots_of(WHICH, D);
    constexpr int kDH = dhalf_of(D);
    constexpr int ntile = WHICH == 0 ? 1 : 2;
    constexpr int tmCk = WHICH == 0 ? 1 : 2, tmCv = WHICH == 0 ? 2 : 3;
    const int lane = threadIdx.x & 31;
    const WaitGuard err{p.err, p.wait_ns};
    const TilePlan& pl = p.plan;
    const BiasGeom bg = bias_geom(pl);
    const uint32_t tile_bytes = 128u * D * 2u, chunk_bytes = static_cast<uint32_t>(pl.NC) * D * 2u;
    const uint32_t abias = smem_u32(smem + lay.abias);

    build_bias_b(pl, bg, smem_u32(smem + lay.bbias), lay.bgroup, lane, p.f16 != 0);
    fence_proxy_async_smem();
    uint32_t built = 0;  // axes whose part of A holds the geometry of sig[]
    uint64_t sig[3] = {0, 0, 0};
    TileIter it = tile_iter_begin(p);
    bool started = false;
    Cta c;
    uint32_t j = 0, g = 0;
    bool ok = true;
    while (ok && next_tile(p, WHICH, it, started, c)) {
        if (!(ok = publish_tile(smem, lay, bars, j, err, lane, &c))) break;
        const uint32_t qs = j % kTS;
        if (j >= kTS) ok = warp_wait(&bars[kQEmpty + qs], ((j / kTS) - 1) & 1, err, kSiteQ);
        if (!ok) break;
        // the bias operand A: rebuilt along the axes whose border situation changed, once every
        // score product of the previous tile (its last reader) is done
        uint32_t stale = 0;
        uint64_t ns[3];
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            ns[a] = axis_sig(WHICH, c.t0[a], pl.T[a], c.Lc[a], p.k[a], pl.H[a]);
            if (bg.nbg[a] > 0 && (!((built >> a) & 1u) || ns[a] != sig[a])) stale |= 1u << a;
        }
        if (stale) {
            if (j >= 1) ok = warp_wait(&bars[kQEmpty + (j - 1) % kTS], ((j - 1) / kTS) & 1, err, kSiteQ);
            if (!ok) break;
            build_bias_a(p, WHICH, c, bg, abias, lane, stale);
            fence_proxy_async_smem();
#pragma unroll
            for (int a = 0; a < 3; ++a) sig[a] = ns[a];
            built |= stale;
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[kQFull + qs], ntile * tile_bytes);
            for (int tt = 0; tt < ntile; ++tt)
#pragma unroll
                for (int hh = 0; hh < D / kDH; ++hh)
                    tma_load_5d(smem + lay.tile(qs, tt) + hh * lay.tile_h, &p.tm[tt], &bars[kQFull + qs],
                                c.h * D + hh * kDH, c.cls[2] + p.d[2] * c.t0[2], c.cls[1] + p.d[1] * c.t0[1],
                                c.cls[0] + p.d[0] * c.t0[0], c.b);
        }
        ChunkCursor cur = cursor_begin();
        for (int ci = 0; ci < c.C; ++ci, ++g) {
            const uint32_t s = g % kS;
            if (g >= kS) ok = warp_wait(&bars[kKVEmpty + s], ((g / kS) - 1) & 1, err, kSiteEmpty);
            if (!ok) break;
            const int y0 = c.h0[0] + cur.o[0], z0 = c.h0[1] + cur.o[1], x0 = c.h0[2] + cur.o[2];
            // test hook: CTA 0 never fills its first chunk (no copy, no arrival), so the waits on it
            // run out after the launch's limit
            const bool withheld = p.withhold != 0u && blockIdx.x == 0 && g == 0;
            if (lane == 0 && !withheld) {
                mbar_arrive_expect_tx(&bars[kKVFull + s], 2u * chunk_bytes);
#pragma unroll
                for (int hh = 0; hh < D / kDH; ++hh) {
                    tma_load_5d(smem + lay.chunk(s, 0) + hh * lay.chunk_h, &p.tm[tmCk], &bars[kKVFull + s],
                                c.h * D + hh * kDH, c.cls[2] + p.d[2] * x0, c.cls[1] + p.d[1] * z0,
                                c.cls[0] + p.d[0] * y0, c.b);
                    tma_load_5d(smem + lay.chunk(s, 1) + hh * lay.chunk_h, &p.tm[tmCv], &bars[kKVFull + s],
                                c.h * D + hh * kDH, c.cls[2] + p.d[2] * x0, c.cls[1] + p.d[1] * z0,
                                c.cls[0] + p.d[0] * y0, c.b);
                }
            }
            cursor_next(pl, c, cur);
        }
        ++j;
    }
    if (ok) publish_tile(smem, lay, bars, j, err, lane, nullptr);
    // Copies already issued must land before the CTA exits and its shared memory is reused (after an
    // error the consumers stop early): wait for the last fill of every chunk slot and tile slot.
    if (lane == 0) {
        for (uint32_t k = 0; k < static_cast<uint32_t>(kS); ++k) {
            if (g <= k) continue;
            const uint32_t last = g - 1 - ((g - 1 - k) % kS);  // the last fill of slot k
            if (!(p.withhold != 0u && blockIdx.x == 0 && last == 0)) mbar_drain(&bars[kKVFull + k], (last / kS) & 1, err.limit_ns);
        }
        for (uint32_t k = 0; k < kTS; ++k) {
            if (j <= k) continue;
            const uint32_t last = j - 1 - ((j - 1 - k) % kTS);
            mbar_drain(&bars[kQFull + k], (last / kTS) & 1, err.limit_ns);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------------------------
// Issuing lanes: one for the score products of every chunk, one per update accumulator.
// ---------------------------------------------------------------------------------------------

// Issues the tensor-core products.  An issuing lane shares its SM sub-partition with softmax warps, so
// every instruction it spends per MMA counts: descriptors are built once with start address 0 and
// offset per operand (the start-address field is the low 14 bits of the descriptor and holds
// address >> 4; shared addresses are below 256 KB), and the instruction descriptors are constant.
template <int D>
struct MmaIssuer {
    uint32_t sbase;                        // shared address of the layout base
    uint64_t dk, dp, dmn, dbias;           // descriptor bases: K-major rows of D, P atoms, MN-major rows of D, bias blocks
    uint32_t idesc_s, idesc_sn, idesc_u;   // scores (N = NC), negated scores, updates (N = D)
    uint32_t nkk;                          // NC / 16
    uint32_t tile_h, chunk_h;              // second 64-channel half of a tile / chunk tensor (D = 128)
    uint32_t abias, bbias, bgroup;
    int nbg[3], abase[3], bbase[3];

    __device__ static __forceinline__ uint64_t at(uint64_t base, uint32_t addr) { return base + (addr >> 4); }

    __device__ void init(const TcParams& p, uint8_t* smem, const TcLayout& lay) {
        constexpr int kDH = dhalf_of(D);
        const uint32_t rowb = kDH * 2u, lay_ = swizzle_layout(kDH * 2), sbo = 8u * rowb;
        sbase = smem_u32(smem);
        dk = sdesc(0u, 16u, sbo, lay_);
        dp = sdesc(0u, 16u, 512u, 4u);
        dmn = sdesc(0u, 16u * rowb, sbo, lay_);
        dbias = sdesc(0u, 16u, 256u, 6u);
        idesc_s = idesc_mma(128, p.plan.NC, false, false, p.f16 != 0);
        idesc_sn = idesc_s | (1u << 13);
        idesc_u = idesc_mma(128, kDH, false, true, p.f16 != 0);
        nkk = static_cast<uint32_t>(p.plan.NC) / 16u;
        tile_h = lay.tile_h;
        chunk_h = lay.chunk_h;
        abias = sbase + lay.abias;
        bbias = sbase + lay.bbias;
        bgroup = lay.bgroup;
        const BiasGeom bg = bias_geom(p.plan);
        for (int a = 0; a < 3; ++a) {
            nbg[a] = bg.nbg[a];
            abase[a] = bg.abase[a];
            bbase[a] = bg.bbase[a];
        }
    }

    // D_tmem = A_tile(128 x D) * B_chunk(NC x D)^T, both K-major; A negated when `neg`.  K-step kk
    // reads 16 channels of half kk / (64 / 16) (D = 128) at 32 bytes per step within the half.
    __device__ __forceinline__ void rows_x_chunk(uint32_t d_tmem, uint32_t a_off, uint32_t b_off, bool neg) const {
        constexpr int kPerHalf = dhalf_of(D) / 16;
        const uint32_t a = sbase + a_off, b = sbase + b_off, id = neg ? idesc_sn : idesc_s;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t hh = static_cast<uint32_t>(kk / kPerHalf), r = static_cast<uint32_t>(kk % kPerHalf) * 32u;
            umma_bf16(d_tmem, at(dk, a + hh * tile_h + r), at(dk, b + hh * chunk_h + r), id, kk > 0);
        }
    }
    // D_tmem += A_bias(chunk) * B_bias^T along every masked axis: the window mask.
    __device__ __forceinline__ void add_bias(uint32_t d_tmem, const ChunkCursor& k) const {
#pragma unroll
        for (int ax = 0; ax < 3; ++ax) {
            if (nbg[ax] == 0) continue;
            const uint32_t ga = abias + static_cast<uint32_t>(abase[ax] + k.ix[ax] * nbg[ax]) * 4096u;
            const uint32_t gb = bbias + static_cast<uint32_t>(bbase[ax]) * bgroup;
            umma_bf16(d_tmem, at(dbias, ga), at(dbias, gb), idesc_s, 1u);
            if (nbg[ax] > 1) umma_bf16(d_tmem, at(dbias, ga + 4096u), at(dbias, gb + bgroup), idesc_s, 1u);
        }
    }
    // D_tmem (+)= P(128 x NC) * B_chunk(NC x D), B MN-major, with P read from TMEM: 16-bit pairs packed
    // in NC / 2 columns from a_tmem, so k-step kk (chunk columns 16 kk .. 16 kk + 15) starts at column
    // a_tmem + 8 kk; at D = 128 one product per channel half.
    __device__ __forceinline__ void pt_x_chunk(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_off, bool accumulate) const {
        constexpr int kDH = dhalf_of(D);
#pragma unroll
        for (int hh = 0; hh < D / kDH; ++hh) {
            uint32_t b = sbase + b_off + static_cast<uint32_t>(hh) * chunk_h;
            for (uint32_t kk = 0; kk < nkk; ++kk) {
                umma_ts(d_tmem + hh * kDH, a_tmem + 8u * kk, at(dmn, b), idesc_u, (accumulate || kk > 0) ? 1u : 0u);
                b += 16u * kDH * 2u;
            }
        }
    }
    // D_tmem (+)= P(128 x NC, 32-column atoms) * B_chunk(NC x D), B MN-major; at D = 128 one product
    // of N = 64 per channel half, into accumulator columns [64 h, 64 h + 64).
    __device__ __forceinline__ void p_x_chunk(uint32_t d_tmem, uint32_t p_off, uint32_t b_off, bool accumulate) const {
        constexpr int kDH = dhalf_of(D);
#pragma unroll
        for (int hh = 0; hh < D / kDH; ++hh) {
            uint32_t a = sbase + p_off, b = sbase + b_off + static_cast<uint32_t>(hh) * chunk_h;
            for (uint32_t kk = 0; kk < nkk; ++kk) {
                umma_bf16(d_tmem + hh * kDH, at(dp, a), at(dmn, b), idesc_u, (accumulate || kk > 0) ? 1u : 0u);
                a += (kk & 1u) ? 8192u - 32u : 32u;
                b += 16u * kDH * 2u;
            }
        }
    }
};

// TMEM column bases.  fwd (256 columns): S[b] at b*NC (b < 3 at D <= 32), O[b] at 256 - (2 - b) * D.
// dQ (512): S[b] at b*NC, dP[b] at (2 + b)*NC, dQ[b] at 512 - (2 - b) * D.
// dKdV (512): S[b] at b*NC, dP[b] at (2 + b)*NC, dV[b] at 512 - (4 - 2b) * D, dK[b] = dV[b] + D.
__device__ __forceinline__ uint32_t tm_s(const TilePlan& pl, uint32_t b) { return b * pl.NC; }
__device__ __forceinline__ uint32_t tm_dp(const TilePlan& pl, uint32_t b) { return (2 + b) * pl.NC; }
template <int D>
__device__ __forceinline__ uint32_t tm_acc(int which, uint32_t b) {
    const uint32_t cols = static_cast<uint32_t>(tmem_cols_of(which, D));
    return which == 2 ? cols - (2u * abufs_of(2, D) - 2u * b) * D : cols - (2u - b) * D;
}

// Forward: the update products O += P V of every chunk, issued by one lane as soon as the chunk's P is
// written (and, for a tile's first chunk, its accumulator buffer has been read out).
template <int D, int SB>
__device__ void pv_loop(const TcParams& p, uint8_t* smem, const TcLayout& lay, uint64_t* bars, uint32_t tmem) {
    constexpr uint32_t kS = stages_of(0, D);
    const WaitGuard err{p.err, p.wait_ns};
    MmaIssuer<D> mi;
    mi.init(p, smem, lay);
    Cta c;
    uint32_t j = 0, g = 0;
    bool ok = true;
    while (ok && fetch_tile(smem, lay, bars, j, err, false, c, ok)) {
        const uint32_t ob = j & 1u;
        for (int ci = 0; ci < c.C; ++ci, ++g) {
            constexpr uint32_t kSB = SB;
            const uint32_t pb = g % kSB, s = g % kS;
            ok = mbar_spin(&bars[kPFull + pb], (g / kSB) & 1u, err, kSiteP);
            if (ok && ci == 0 && j >= 2) ok = mbar_spin(&bars[kOEmpty + ob], ((j >> 1) - 1) & 1u, err, kSitePV);
            if (!ok) break;
            tc_fence_after();
            mi.pt_x_chunk(tmem + tm_acc<D>(0, ob), tmem + tm_s(p.plan, pb), lay.chunk(s, 1), ci > 0);  // O += P V
            umma_commit(&bars[kPEmpty + pb]);
            umma_commit(&bars[kKVEmpty + s]);
            if (ci == c.C - 1) umma_commit(&bars[kOFull + ob]);
        }
        ++j;
    }
}

// The score products of every chunk, issued by one lane: S (or S^T) and the window bias, and in the
// backward dP (or dP^T).  The forward's score buffer also holds that chunk's P, so it is free once the
// product P V of the chunk two back is done; the backward's softmax releases it after reading.
template <int D, int WHICH, int SB>
__device__ void score_loop(const TcParams& p, uint8_t* smem, const TcLayout& lay, uint64_t* bars, uint32_t tmem) {
    constexpr uint32_t kS = stages_of(WHICH, D);
    const WaitGuard err{p.err, p.wait_ns};
    const TilePlan& pl = p.plan;
    MmaIssuer<D> mi;
    mi.init(p, smem, lay);
    const bool neg = p.neg != 0;
    Cta c;
    uint32_t j = 0, g = 0;
    bool ok = true;
    constexpr uint32_t kTS = tslots_of(WHICH, D);
    while (ok && fetch_tile(smem, lay, bars, j, err, false, c, ok)) {
        const uint32_t qs = j % kTS;
        if (!mbar_wait(&bars[kQFull + qs], (j / kTS) & 1, err, kSiteQ)) break;
        ChunkCursor cur = cursor_begin();
        for (int ci = 0; ci < c.C; ++ci, ++g, cursor_next(pl, c, cur)) {
            constexpr uint32_t kSB = SB;
            const uint32_t s = g % kS, sb = g % kSB;
            ok = mbar_spin(&bars[kKVFull + s], (g / kS) & 1, err, kSiteKV);
            if (ok && g >= kSB)
                ok = mbar_spin(&bars[(WHICH == 0 ? kPEmpty : kSEmpty) + sb], ((g / kSB) - 1) & 1, err, kSiteS);
            if (!ok) break;
            tc_fence_after();
            mi.rows_x_chunk(tmem + tm_s(pl, sb), lay.tile(qs, 0), lay.chunk(s, 0), neg);  // S or S^T
            mi.add_bias(tmem + tm_s(pl, sb), cur);                                          // + window bias
            if (WHICH != 0) mi.rows_x_chunk(tmem + tm_dp(pl, sb), lay.tile(qs, 1), lay.chunk(s, 1), false);  // dP or dP^T
            umma_commit(&bars[kSFull + sb]);
            if (ci == c.C - 1) umma_commit(&bars[kQEmpty + qs]);
        }
        ++j;
    }
}

// Backward: one update accumulator's products of every chunk, issued by one lane.  `u` selects the
// product: dQ += dS K (dQ kernel); dV += P^T dO (u = 0) or dK += dS^T Q (u = 1) (dK/dV kernel).
// Each issuer arrives once on the chunk-slot, P-buffer and accumulator barriers (their counts are
// the number of issuers).  The chunk slot is also read by the score products, which are complete
// before the P operand (written after their results were read) exists.
template <int D, int WHICH>
__device__ void update_loop(const TcParams& p, uint8_t* smem, const TcLayout& lay, uint64_t* bars, uint32_t tmem,
                            int u) {
    constexpr uint32_t kS = stages_of(WHICH, D);
    constexpr uint32_t kPB = pbufs_of(WHICH);
    const WaitGuard err{p.err, p.wait_ns};
    MmaIssuer<D> mi;
    mi.init(p, smem, lay);
    Cta c;
    uint32_t j = 0, g = 0;
    bool ok = true;
    const uint32_t op_p = WHICH == 2 ? static_cast<uint32_t>(u) : 0u;              // P^T or dS^T
    const uint32_t op_b = WHICH == 1 ? 0u : (u == 0 ? 1u : 0u);                    // K; dO or Q
    const uint32_t acc_off = WHICH == 2 && u == 1 ? static_cast<uint32_t>(D) : 0u;  // dK beside dV
    constexpr uint32_t kAB = abufs_of(WHICH, D);
    while (ok && fetch_tile(smem, lay, bars, j, err, false, c, ok)) {
        const uint32_t ob = j % kAB;
        const uint32_t acc = tmem + tm_acc<D>(WHICH, ob) + acc_off;
        for (int ci = 0; ci < c.C; ++ci, ++g) {
            const uint32_t s = g % kS, pb = g % kPB;
            ok = mbar_spin(&bars[kPFull + pb], (g / kPB) & 1, err, kSiteP);
            if (ok && ci == 0 && j >= kAB) ok = mbar_spin(&bars[kOEmpty + ob], ((j / kAB) - 1) & 1, err, kSitePV);
            if (!ok) break;
            tc_fence_after();
            mi.p_x_chunk(acc, lay.p(pb, op_p), lay.chunk(s, op_b), ci > 0);
            umma_commit(&bars[kPEmpty + pb]);
            umma_commit(&bars[kKVEmpty + s]);
            if (ci == c.C - 1) umma_commit(&bars[kOFull + ob]);
        }
        ++j;
    }
}

// ---------------------------------------------------------------------------------------------
// Epilogue helpers
// ---------------------------------------------------------------------------------------------

// Store columns [c0, c1) of this thread's accumulator row (fp32 at taddr), times `mul`, as bf16
// to dst (the row's first element in global memory).
template <int NCOL, bool F16>
__device__ __forceinline__ void store_row(uint32_t taddr, float mul, uint16_t* dst, bool valid) {
    static_assert(NCOL % 8 == 0 && NCOL <= 64, "row slice of 8..64 columns");
    uint32_t r[NCOL / 8][8];
#pragma unroll
    for (int i = 0; i < NCOL / 8; ++i) tmem_ld8(taddr + 8 * i, r[i]);
    tmem_ld_wait_all();
#pragma unroll
    for (int i = 0; i < NCOL / 8; ++i) reg_fence8(r[i]);
    if (valid) {
#pragma unroll
        for (int i = 0; i < NCOL / 8; ++i) {
            uint4 w;
            w.x = pack2<F16>(__uint_as_float(r[i][0]) * mul, __uint_as_float(r[i][1]) * mul);
            w.y = pack2<F16>(__uint_as_float(r[i][2]) * mul, __uint_as_float(r[i][3]) * mul);
            w.z = pack2<F16>(__uint_as_float(r[i][4]) * mul, __uint_as_float(r[i][5]) * mul);
            w.w = pack2<F16>(__uint_as_float(r[i][6]) * mul, __uint_as_float(r[i][7]) * mul);
            *reinterpret_cast<uint4*>(dst + 8 * i) = w;
        }
    }
}

// Zero 16-column group gi of this row in a P operand.
__device__ __forceinline__ void zero_group(uint32_t sP, uint32_t rowbase, uint32_t sw, int gi) {
    st_shared_v4(sP + p_off(rowbase, sw, 2 * gi), 0u, 0u, 0u, 0u);
    st_shared_v4(sP + p_off(rowbase, sw, 2 * gi + 1), 0u, 0u, 0u, 0u);
}

// ---------------------------------------------------------------------------------------------
// Forward softmax warps (4 warps, 128 rows)
// ---------------------------------------------------------------------------------------------

struct FwdCtx {
    uint64_t* bars;
    WaitGuard err;
    uint32_t tS0, tS_step;  // this warp's lanes of score buffer 0, and the offset of buffer 1
    uint32_t tO;            // this warp's lanes of the tile accumulator
    int ngroups;            // 16-column groups per chunk
    float sl2;
    uint64_t sl2x2;
    int lane;
};

// Groups [glo, glo + n) as a bit mask.
__device__ __forceinline__ uint32_t run_mask(int glo, int n) { return ((1u << n) - 1u) << glo; }

// A packed pair of the operand type back to fp32 (first element from the low half).
template <bool F16>
__device__ __forceinline__ void unpack2(uint32_t v, float& lo, float& hi) {
    if constexpr (F16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
        lo = f.x;
        hi = f.y;
    } else {
        lo = __uint_as_float(v << 16);
        hi = __uint_as_float(v & 0xffff0000u);
    }
}

// One part of a warp's run: groups [gb, gb + cnt) (cnt <= N) of the chunk's score buffer tS.  Their
// scores are read and the running max is updated; when it moves by more than 2^8, O, the partial sums and the
// chunk's groups [gb - gdone, gb) already written as P are rescaled.  Then P = exp2(S sl2 - m) is
// written over the scores as packed 16-bit pairs: group gi's P takes columns 8 gi .. 8 gi + 7 of
// the buffer, which held the scores of group gi / 2, read before this write (or outside the run).
template <int D, int N, bool F16, int SB>
__device__ __forceinline__ bool fwd_part(const FwdCtx& x, uint32_t g, uint32_t tS, int gb, int cnt, int gdone,
                                         float& m, uint64_t (&lsum)[4]) {
    uint32_t v[N][16];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if (i < cnt) {
            tmem_ld16(tS + 16u * (gb + i), v[i]);
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[i][e] = __float_as_uint(-INFINITY);
        }
    }
    tmem_ld_wait_all();
#pragma unroll
    for (int i = 0; i < N; ++i) reg_fence16(v[i]);
    // row max of the part (masked scores carry the -2^100 window bias), four independent chains
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < N; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            mx[e] = fmax3(mx[e], fmaxf(__uint_as_float(v[i][4 * e]), __uint_as_float(v[i][4 * e + 1])),
                          fmaxf(__uint_as_float(v[i][4 * e + 2]), __uint_as_float(v[i][4 * e + 3])));
    const float cmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    // running max (log2 units; the scale's sign is folded into the S product)
    const float cm2 = cmax > masked_below<F16>() ? cmax * x.sl2 : -INFINITY;  // no live key: -inf
    const float mnew = fmaxf(m, cm2);
    const bool rescale = (m != -INFINITY) && (mnew > m + kRescaleThreshold);
    const float alpha = rescale ? fast_exp2(m - mnew) : 1.f;
    if (m == -INFINITY || rescale) m = mnew;
    if (__any_sync(0xffffffffu, rescale)) {
        // O holds the products of chunks g-1, g-2, ...: wait for the last one (before a tile's first
        // chunk that is the previous tile's, harmless; for g = 0 the parity test passes at once)
        constexpr uint32_t kSB = SB;
        if (!warp_wait(&x.bars[kPEmpty + (g - 1) % kSB], ((g - 1) / kSB) & 1u, x.err, kSitePV)) return false;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D; cc += 8) {
            uint32_t r[8];
            tmem_ld8(x.tO + cc, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st8(x.tO + cc, r);
        }
        if (gdone > 0) tmem_st_wait();  // the P groups of this chunk's first part are written
        for (int gi = gb - gdone; gi < gb; ++gi) {
            uint32_t r[8];
            tmem_ld8(tS + 8u * gi, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float lo, hi;
                unpack2<F16>(r[e], lo, hi);
                r[e] = pack2<F16>(lo * alpha, hi * alpha);
            }
            tmem_st8(tS + 8u * gi, r);
        }
        tmem_st_wait();
        const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
        for (int t = 0; t < 4; ++t) lsum[t] = f2_mul(lsum[t], a2);
    }
    const float nm = m == -INFINITY ? 0.f : -m;  // masked scores are -inf: exp2 gives 0
    const uint64_t nm2 = f2(nm, nm);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if (i >= cnt) break;
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            const uint64_t t = f2_fma(f2(__uint_as_float(v[i][e]), __uint_as_float(v[i][e + 1])), x.sl2x2, nm2);
            float ta, tb;
            f2_split(t, ta, tb);
            const uint64_t pe = f2(fast_exp2(ta), fast_exp2(tb));
            lsum[(e >> 1) & 3] = f2_add(lsum[(e >> 1) & 3], pe);
            w[e >> 1] = x2_of<F16>(pe);
        }
        tmem_st8(tS + 8u * (gb + i), w);
    }
    return true;
}

// One chunk of the online softmax for a warp whose keys lie in groups [glo, glo + n) (n <= 6):
// runs of up to four groups in one part, longer runs in two parts of at most three (register
// budget).  Groups outside the run hold scores, not P, so they are zeroed once every score of the
// run has been read; then the P operand (its score buffer) is released to the P V lane.
template <int D, bool F16, int SB>
__device__ __forceinline__ bool fwd_chunk(const FwdCtx& x, uint32_t g, int glo, int n, float& m,
                                          uint64_t (&lsum)[4]) {
    constexpr uint32_t kSB = SB;
    const uint32_t tS = x.tS0 + (g % kSB) * x.tS_step;
    bool ok = true;
    // runs of one to three groups share the three-group part (its count is a run-time argument), so
    // the softmax warps' hot code holds two part bodies instead of four: smaller code for the
    // instruction cache, which the five roles of a CTA share
    switch (n) {
        case 0: break;
        case 1:
        case 2:
        case 3: ok = fwd_part<D, 3, F16, SB>(x, g, tS, glo, n, 0, m, lsum); break;
        case 4: ok = fwd_part<D, 4, F16, SB>(x, g, tS, glo, 4, 0, m, lsum); break;
        default:
            // groups [glo, glo + 3), then [glo + 3, glo + n); one loop body keeps register use at
            // that of a single part
#pragma unroll 1
            for (int part = 0; part < 2 && ok; ++part)
                ok = fwd_part<D, 3, F16, SB>(x, g, tS, glo + 3 * part, part == 0 ? 3 : n - 3, 3 * part, m, lsum);
            break;
    }
    if (!ok) return false;
    for (int gi = 0; gi < x.ngroups; ++gi)
        if (gi < glo || gi >= glo + n) tmem_st8_zero(tS + 8u * gi);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (x.lane == 0) mbar_arrive(&x.bars[kPFull + g % kSB]);
    return true;
}

// A tile whose rows still have to be written: O / l -> bf16 and LSE = (m + log2 l) * ln 2.
struct FwdEpilogue {
    bool live, valid;
    float m, l;
    long long orow;  // row index into [B * tokens * heads]
    uint32_t ob, j;  // accumulator buffer and tile ordinal
};

template <int D, bool F16>
__device__ __forceinline__ bool fwd_epilogue(const TcParams& p, const FwdCtx& x, const FwdEpilogue& e,
                                             uint32_t tmem_lanes) {
    if (!warp_wait(&x.bars[kOFull + e.ob], (e.j >> 1) & 1, x.err, kSitePV)) return false;
    tc_fence_after();
#pragma unroll
    for (int hh = 0; hh < D / dhalf_of(D); ++hh)
        store_row<dhalf_of(D), F16>(tmem_lanes + tm_acc<D>(0, e.ob) + hh * dhalf_of(D), 1.f / e.l,
                                    p.out0 + e.orow * D + hh * dhalf_of(D), e.valid);
    tc_fence_before();
    __syncwarp();
    if (x.lane == 0) mbar_arrive(&x.bars[kOEmpty + e.ob]);
    if (e.valid) p.lse_out[e.orow] = (e.m + __log2f(e.l)) * kLn2;
    return true;
}

template <int D, bool F16, int SB>
__device__ void fwd_softmax_loop(const TcParams& p, uint8_t* smem, const TcLayout& lay, uint64_t* bars,
                                 uint32_t tmem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, row = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const TilePlan& pl = p.plan;
    FwdCtx x;
    x.bars = bars;
    x.err = WaitGuard{p.err, p.wait_ns};
    x.tS0 = tmem + tm_s(pl, 0) + lane_base;
    x.tS_step = tm_s(pl, 1) - tm_s(pl, 0);
    x.ngroups = pl.NC >> 4;
    x.sl2 = p.scale_log2;
    x.sl2x2 = f2(x.sl2, x.sl2);
    x.lane = lane;
    FwdEpilogue ep{false, false, 0.f, 0.f, 0, 0, 0};
    Cta c;
    uint32_t j = 0, g = 0;
    bool ok = true;
    for (;;) {
        // one pass per tile, and one more after the last to store its rows (a single epilogue site)
        const bool more = fetch_tile(smem, lay, bars, j, x.err, true, c, ok);
        if (!ok) break;
        FwdEpilogue next{false, false, 0.f, 0.f, 0, 0, 0};
        if (more) {
            const RowGeom geo = row_geom(p, 0, c, row);
            const WarpUnion wu = warp_union(geo);
            const uint32_t ob = j & 1;
            x.tO = tmem + tm_acc<D>(0, ob) + lane_base;
            float m = -INFINITY;
            uint64_t lsum[4] = {0ull, 0ull, 0ull, 0ull};  // four packed partial sums (independent chains)
            ChunkCursor cur = cursor_begin();
            for (int ci = 0; ci < c.C; ++ci, ++g, cursor_next(pl, c, cur)) {
                ok = warp_wait(&bars[kSFull + g % SB], (g / SB) & 1, x.err, kSiteS);
                if (!ok) break;
                tc_fence_after();
                int glo, n;
                chunk_range(pl, cur, wu, glo, n);
                ok = fwd_chunk<D, F16, SB>(x, g, glo, n, m, lsum);
                if (!ok) break;
            }
            if (!ok) break;
            const uint64_t ls = f2_add(f2_add(lsum[0], lsum[1]), f2_add(lsum[2], lsum[3]));
            float la, lb;
            f2_split(ls, la, lb);
            next = FwdEpilogue{true, geo.valid, m, la + lb, geo.token * p.heads + c.h, ob, j};
        }
        // the previous tile's epilogue, deferred until this tile's chunks are done so that a warp
        // does not idle at the end of a tile while the slowest warp finishes it
        if (ep.live && !(ok = fwd_epilogue<D, F16>(p, x, ep, tmem + lane_base))) break;
        ep = next;
        if (!more) break;
        ++j;
    }
}

// ---------------------------------------------------------------------------------------------
// Backward softmax warps (8 warps: two warpgroups share each chunk's groups, alternating)
// ---------------------------------------------------------------------------------------------

struct BwdCtx {
    uint32_t tS, tP;     // this warp's lanes of the current score / dP buffers
    uint32_t sP0, sP1;   // P-side operands of the current buffer (dQ: dS; dK/dV: P^T, dS^T)
    uint32_t rowbase, sw;
    const float* l2;     // dK/dV: -LSE (log2 units) of the chunk columns
    const float* dl;     // dK/dV: Delta of the chunk columns
    uint64_t nl2, dl2;   // dQ: -LSE (log2 units) and Delta of this row, packed twice
    uint64_t sl2x2;
};

// This warp's K (<= 2) groups g0, g0 + kBwdGroups of the chunk: their scores and dP values are read, the
// score buffer is released when these are the warp's last groups of the chunk (so the next chunk's
// products can start), then P = exp2(S sl2 - LSE2) and dS = P (dP - Delta) are formed and stored.
template <int WHICH, int K, bool F16>
__device__ __forceinline__ void bwd_groups(const BwdCtx& x, int g0, uint64_t* sempty, bool release, int lane) {
    uint32_t rs[K > 0 ? K : 1][16], rp[K > 0 ? K : 1][16];
#pragma unroll
    for (int i = 0; i < K; ++i) {
        tmem_ld16(x.tS + 16u * (g0 + group_stride_of(WHICH) * i), rs[i]);
        tmem_ld16(x.tP + 16u * (g0 + group_stride_of(WHICH) * i), rp[i]);
    }
    if (K > 0) {
        tmem_ld_wait_all();
#pragma unroll
        for (int i = 0; i < K; ++i) {
            reg_fence16(rs[i]);
            reg_fence16(rp[i]);
        }
    }
    if (release) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sempty);
    }
#pragma unroll
    for (int i = 0; i < K; ++i) {
        const int gi = g0 + group_stride_of(WHICH) * i;
        uint32_t a[8], b[8];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            uint64_t nlc[2] = {x.nl2, x.nl2}, dlc[2] = {x.dl2, x.dl2};
            if (WHICH == 2) {
                const float4 lv = *reinterpret_cast<const float4*>(x.l2 + 16 * gi + e);
                const float4 dv = *reinterpret_cast<const float4*>(x.dl + 16 * gi + e);
                nlc[0] = f2(lv.x, lv.y);
                nlc[1] = f2(lv.z, lv.w);
                dlc[0] = f2(dv.x, dv.y);
                dlc[1] = f2(dv.z, dv.w);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int ee = e + 2 * h;
                const uint64_t t =
                    f2_fma(f2(__uint_as_float(rs[i][ee]), __uint_as_float(rs[i][ee + 1])), x.sl2x2, nlc[h]);
                float ta, tb;
                f2_split(t, ta, tb);
                const uint64_t pe = f2(fast_exp2(ta), fast_exp2(tb));
                const uint64_t dp = f2(__uint_as_float(rp[i][ee]), __uint_as_float(rp[i][ee + 1]));
                const uint64_t ds = f2_mul(pe, f2_sub(dp, dlc[h]));
                b[ee >> 1] = x2_of<F16>(ds);
                if (WHICH == 2) a[ee >> 1] = x2_of<F16>(pe);
            }
        }
        const uint32_t o0 = p_off(x.rowbase, x.sw, 2 * gi), o1 = p_off(x.rowbase, x.sw, 2 * gi + 1);
        if (WHICH == 2) {
            st_shared_v4(x.sP0 + o0, a[0], a[1], a[2], a[3]);  // P^T
            st_shared_v4(x.sP0 + o1, a[4], a[5], a[6], a[7]);
            st_shared_v4(x.sP1 + o0, b[0], b[1], b[2], b[3]);  // dS^T
            st_shared_v4(x.sP1 + o1, b[4], b[5], b[6], b[7]);
        } else {
            st_shared_v4(x.sP0 + o0, b[0], b[1], b[2], b[3]);  // dS
            st_shared_v4(x.sP0 + o1, b[4], b[5], b[6], b[7]);
        }
    }
}

// Groups g with g mod kBwdGroups == w, as a 32-bit mask.
__host__ __device__ constexpr uint32_t group_mask(int w) {
    uint32_t m = 0u;
    for (int g = w; g < 32; g += kBwdGroups) m |= 1u << g;
    return m;
}

// A tile whose rows still have to be written; each warpgroup writes half of the D columns of its
// quarter's rows (dQ, or dV and dK).
struct BwdEpilogue {
    bool live, valid;
    long long orow;
    uint32_t ob, j;
};

template <int D, int WHICH, bool F16>
__device__ __forceinline__ bool bwd_epilogue(const TcParams& p, uint64_t* bars, const BwdEpilogue& e,
                                             uint32_t tmem_lanes, int wg, int lane) {
    constexpr uint32_t kAB = abufs_of(WHICH, D);
    if (!warp_wait(&bars[kOFull + e.ob], (e.j / kAB) & 1, WaitGuard{p.err, p.wait_ns}, kSitePV)) return false;
    tc_fence_after();
    const uint32_t acc = tmem_lanes + tm_acc<D>(WHICH, e.ob);
    const int c0 = wg * (D / 2);
    if (wg < 2) {   // two warpgroups store half of the D columns each; any others only release
        if (WHICH == 1) {
            store_row<D / 2, F16>(acc + c0, p.scale, p.out0 + e.orow * D + c0, e.valid);  // dQ
        } else {
            store_row<D / 2, F16>(acc + c0, 1.f, p.out1 + e.orow * D + c0, e.valid);          // dV
            store_row<D / 2, F16>(acc + D + c0, p.scale, p.out0 + e.orow * D + c0, e.valid);  // dK
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[kOEmpty + e.ob]);
    return true;
}

template <int D, int WHICH, bool F16>
__device__ void bwd_softmax_loop(const TcParams& p, uint8_t* smem, const TcLayout& lay, uint64_t* bars,
                                 uint32_t tmem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool kAlt = alt_of(WHICH);
    const int wq = warp & 3, wg = warp >> 2;  // lane quarter, warpgroup
    const uint32_t gmask = group_mask(wg);    // this warpgroup's groups
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const WaitGuard err{p.err, p.wait_ns};
    const TilePlan& pl = p.plan;
    const int ngroups = pl.NC >> 4;
    BwdCtx x;
    x.rowbase = static_cast<uint32_t>(row) * 64u;
    x.sw = (static_cast<uint32_t>(row) >> 1) & 3u;
    x.sl2x2 = f2(p.scale_log2, p.scale_log2);
    x.l2 = nullptr;
    x.dl = nullptr;
    // dK/dV: this thread's column of each chunk its warpgroup owns (loaded while the warp waits for
    // the chunk's scores, then shared within the warpgroup)
    static_assert(WHICH != 2 || alt_of(2), "the column exchange assumes alternate chunks");
    AuxCol ac{};
    long long tb = 0;
    bool pre = false;  // ac already holds this chunk's values
    if (WHICH == 2) aux_init(p, ac, row);
    uint32_t nz0 = run_mask(0, ngroups), nz1 = nz0, nz2 = nz0;  // groups of the quarter's rows that may be nonzero
    BwdEpilogue ep{false, false, 0, 0, 0};
    Cta c;
    uint32_t j = 0, g = 0;
    bool ok = true;
    for (;;) {
        // one pass per tile, and one more after the last to store its rows: the epilogue has a single
        // call site (the kernels' hot code has to stay small for the instruction cache)
        const bool more = fetch_tile(smem, lay, bars, j, err, true, c, ok);
        if (!ok) break;
        BwdEpilogue next{false, false, 0, 0, 0};
        if (more) {
            const RowGeom geo = row_geom(p, WHICH, c, row);
            const WarpUnion wu = warp_union(geo);
            const uint32_t ob = j % abufs_of(WHICH, D);
            if (WHICH == 2) tb = aux_tile_base(p, c);
            float lse2 = 0.f, dlt = 0.f;
            if (WHICH == 1 && geo.valid) {
                lse2 = __ldg(p.lse + geo.token * p.heads + c.h) * kLog2e;
                dlt = __ldg(p.delta + geo.token * p.heads + c.h);
            }
            x.nl2 = f2(-lse2, -lse2);
            x.dl2 = f2(dlt, dlt);
            ChunkCursor cur = cursor_begin();
            // dQ visits only the warpgroup's chunks (its first of the tile, then every other one); dK/dV
            // steps through every chunk and skips the other warpgroup's
            constexpr bool kJump = kAlt && WHICH == 1;
            constexpr int kStep = kJump ? 2 : 1;
            const uint32_t gend = g + static_cast<uint32_t>(c.C);
            int ci = 0;
            if (kJump && (g & 1u) != static_cast<uint32_t>(wg)) {
                ++ci;
                ++g;
                cursor_next(pl, c, cur);
            }
            for (; ci < c.C; ci += kStep, g += kStep, cursor_steps<kStep>(pl, c, cur)) {
                constexpr uint32_t kPB = pbufs_of(WHICH);
                const uint32_t sb = g & 1, pb = g % kPB;
                if (!kJump && kAlt && (g & 1u) != static_cast<uint32_t>(wg)) continue;   // the other warpgroup's chunk
                // dK/dV: the column's values, unless the previous chunk of the warpgroup prefetched them
                if (WHICH == 2 && !pre) aux_load(p, c, tb, cur, ac);
                ok = warp_wait(&bars[kSFull + sb], (g >> 1) & 1, err, kSiteS);
                if (!ok) break;
                tc_fence_after();
                if (WHICH == 2) {
                    // the warpgroup's k-th chunk: its columns' -LSE (log2 units; none outside the class)
                    // and Delta into buffer k mod 2; a buffer is rewritten only after every warp has
                    // passed the exchange of the chunk in between, so after its last read
                    const uint32_t k = g >> 1, buf = lay.aux(2u * static_cast<uint32_t>(wg) + (k & 1u));
                    const uint32_t l2 = smem_u32(smem + buf), dl = l2 + 4u * static_cast<uint32_t>(pl.NC);
                    if (ac.col) {
                        st_shared_f32(l2 + 4u * static_cast<uint32_t>(row), ac.in ? -ac.l * kLog2e : -INFINITY);
                        st_shared_f32(dl + 4u * static_cast<uint32_t>(row), ac.in ? ac.dl : 0.f);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[kAuxSync + wg]);
                    x.l2 = reinterpret_cast<const float*>(smem + buf);
                    // the warpgroup's next chunk of this tile (g + 2): its loads are in flight while this
                    // chunk is processed
                    pre = ci + 2 < c.C;
                    if (pre) {
                        ChunkCursor nx = cur;
                        cursor_next(pl, c, nx);
                        cursor_next(pl, c, nx);
                        aux_load(p, c, tb, nx, ac);
                    }
                    x.dl = x.l2 + pl.NC;
                }
                int glo, n;
                chunk_range(pl, cur, wu, glo, n);
                // this warpgroup's groups of the run: glo + wg, glo + wg + kBwdGroups, ...; the groups of
                // the quarter's last run in this buffer that the new run does not cover are zeroed, split
                // between the warpgroups by group index modulo kBwdGroups
                const int mine = kAlt ? n : (n > wg ? (n - wg + kBwdGroups - 1) / kBwdGroups : 0);
                const uint32_t run = n > 0 ? run_mask(glo, n) : 0u;
                const uint32_t slot = kAlt ? pb >> 1 : pb;   // this warp's record of the buffer's last run
                const uint32_t nzq = slot == 0 ? nz0 : (slot == 1 ? nz1 : nz2);
                const uint32_t stale = nzq & ~run & (kAlt ? 0xffffffffu : gmask);
                if (slot == 0) nz0 = run; else if (slot == 1) nz1 = run; else nz2 = run;
                if (mine == 0 && stale == 0) {
                    // nothing to write: the score buffer is released at once, but the arrival on the P
                    // operand waits for the products of chunk g - kPB, like every other arrival.  With two
                    // P buffers (dK/dV) an idle warp can otherwise reach chunk g + 2 while a slower warp
                    // still writes chunk g, and its arrival would complete chunk g's phase early.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[kSEmpty + sb]);
                    if (g >= kPB && !(ok = warp_wait(&bars[kPEmpty + pb], ((g / kPB) - 1) & 1, err, kSitePV))) break;
                    if (lane == 0) mbar_arrive(&bars[kPFull + pb]);
                    // dK/dV: every warp passes the exchange before it writes the warpgroup's next buffer
                    if (WHICH == 2 && !(ok = warp_wait(&bars[kAuxSync + wg], (g >> 1) & 1u, err, kSiteKV))) break;
                    continue;
                }
                if (g >= kPB) ok = warp_wait(&bars[kPEmpty + pb], ((g / kPB) - 1) & 1, err, kSitePV);
                // dK/dV: every warp of the warpgroup has written its column of the exchange buffer
                if (WHICH == 2 && ok) ok = warp_wait(&bars[kAuxSync + wg], (g >> 1) & 1u, err, kSiteKV);
                if (!ok) break;
                x.tS = tmem + tm_s(pl, sb) + lane_base;
                x.tP = tmem + tm_dp(pl, sb) + lane_base;
                x.sP0 = smem_u32(smem + lay.p(pb, 0));
                x.sP1 = smem_u32(smem + lay.p(pb, 1));
                const int first = glo + (kAlt ? 0 : wg);   // this warp's first group of the run
                if (mine == 0) bwd_groups<WHICH, 0, F16>(x, first, &bars[kSEmpty + sb], true, lane);
                for (int k = 0; k < mine; k += 2) {
                    const bool last = k + 2 >= mine;
                    if (k + 1 < mine)
                        bwd_groups<WHICH, 2, F16>(x, first + group_stride_of(WHICH) * k, &bars[kSEmpty + sb], last, lane);
                    else
                        bwd_groups<WHICH, 1, F16>(x, first + group_stride_of(WHICH) * k, &bars[kSEmpty + sb], last, lane);
                }
                for (uint32_t z = stale; z; z &= z - 1) {
                    zero_group(x.sP0, x.rowbase, x.sw, __ffs(z) - 1);
                    if (WHICH == 2) zero_group(x.sP1, x.rowbase, x.sw, __ffs(z) - 1);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kPFull + pb]);
            }
            if (!ok) break;
            if (kJump) g = gend;
            next = BwdEpilogue{true, geo.valid, geo.token * p.heads + c.h, ob, j};
        }
        // the previous tile's epilogue, deferred until this tile's chunks are done; with a single
        // accumulator buffer the next tile's first products wait for it, so it runs at once
        if (abufs_of(WHICH, D) == 1) ep = next;
        if (ep.live && !(ok = bwd_epilogue<D, WHICH, F16>(p, bars, ep, tmem + lane_base, wg, lane))) break;
        ep = abufs_of(WHICH, D) == 1 ? BwdEpilogue{false, false, 0, 0, 0} : next;
        if (!more) break;
        ++j;
    }
}

// ---------------------------------------------------------------------------------------------
// Kernels
// ---------------------------------------------------------------------------------------------

// The dynamic shared base rounded up to 1024 bytes, as an offset from the __shared__ array itself, so
// that pointers derived from it keep the shared address space (a round trip through an integer would
// make every access through them a generic one).
__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
    return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

template <int D, int WHICH, int SB>
__device__ __forceinline__ void init_barriers(uint64_t* bars) {
    constexpr uint32_t kSoft = 4 * nwg_of(WHICH);
    constexpr uint32_t kChunkWarps = chunk_warps_of(WHICH);
    for (int i = 0; i < 2; ++i) {
        mbar_init(&bars[kQFull + i], 1);
        mbar_init(&bars[kQEmpty + i], 1);
        mbar_init(&bars[kSFull + i], 1);
        if (SB == 2) mbar_init(&bars[kSEmpty + i], kChunkWarps);  // (three buffers: slot 0 is the third score-full)
        mbar_init(&bars[kOFull + i], nupd_of(WHICH) > 0 ? nupd_of(WHICH) : 1);
        mbar_init(&bars[kOEmpty + i], kSoft);
    }
    for (int i = 0; i < (WHICH == 0 ? SB : pbufs_of(WHICH)); ++i) {
        mbar_init(&bars[kPFull + i], kChunkWarps);
        mbar_init(&bars[kPEmpty + i], nupd_of(WHICH) > 0 ? nupd_of(WHICH) : 1);
    }
    for (int s = 0; s < stages_of(WHICH, D); ++s) {
        mbar_init(&bars[kKVFull + s], 1);  // the producer's arrive with the TMA byte count
        mbar_init(&bars[kKVEmpty + s], nupd_of(WHICH) > 0 ? nupd_of(WHICH) : 1);
    }
    for (uint32_t t = 0; t < kTileRing; ++t) {
        mbar_init(&bars[kTFull + t], 1);
        mbar_init(&bars[kTEmpty + t], kSoft + 1 + nupd_of(WHICH));  // softmax warps, score lane, update lanes
    }
    mbar_init(&bars[kFin], 1 + nupd_of(WHICH));
    if (WHICH == 2)
        for (int w = 0; w < kBwdGroups; ++w) mbar_init(&bars[kAuxSync + w], 4);  // the warpgroup's warps
    if (SB == 3) mbar_init(&bars[kSFull + 2], 1);                               // the forward's third score buffer
    fence_barrier_init();
}

template <int D, int WHICH, bool F16, int SB>
__global__ void __launch_bounds__(threads_of(WHICH), WHICH == 0 ? 2 : 1) tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    const TilePlan& pl = p.plan;
    const TcLayout lay = tc_layout(WHICH, pl, D);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    constexpr int kSoftWarps = 4 * nwg_of(WHICH);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tmem_cols = static_cast<uint32_t>(tmem_cols_of(WHICH, D));

    if (warp == kSoftWarps) {
        if (lane == 0) {
            init_barriers<D, WHICH, SB>(bars);
            for (int m = 0; m < 4; ++m) tma_prefetch_desc(&p.tm[m]);
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
    if constexpr (WHICH == 0) {
        // each warpgroup's budget is set in the branch that runs its code
        if (warp < kSoftWarps) {
            reg_alloc<kFwdSoftRegs>();
            fwd_softmax_loop<D, F16, SB>(p, smem, lay, bars, tmem);
        } else {
            reg_dealloc<kFwdCtrlRegs>();
            if (warp == kSoftWarps) {
                producer_loop<D, WHICH>(p, smem, lay, bars);
            } else if (warp == kSoftWarps + 1) {
                if (lane == 0) score_loop<D, WHICH, SB>(p, smem, lay, bars, tmem);
                __syncwarp();
            } else if (warp == kSoftWarps + 2) {
                if (lane == 0) pv_loop<D, SB>(p, smem, lay, bars, tmem);
                __syncwarp();
            }
        }
    } else {
        if (warp == kSoftWarps) {
            producer_loop<D, WHICH>(p, smem, lay, bars);
        } else if (warp == kSoftWarps + 1) {
            if (lane == 0) score_loop<D, WHICH, SB>(p, smem, lay, bars, tmem);
            __syncwarp();
        } else if (warp >= kSoftWarps + 2) {
            if (lane == 0) update_loop<D, WHICH>(p, smem, lay, bars, tmem, warp - (kSoftWarps + 2));
            __syncwarp();
        } else {
            bwd_softmax_loop<D, WHICH, F16>(p, smem, lay, bars, tmem);
        }
    }

    // teardown: every TMEM access of the softmax warps and every MMA of this CTA done before TMEM is
    // freed (each issuing lane commits once)
    if (warp < kSoftWarps) {
        tmem_st_wait();
        tmem_ld_wait_all();
    }
    if (warp >= kSoftWarps + 1 && warp < kSoftWarps + 2 + nupd_of(WHICH) && lane == 0) {  // every issuing lane
        umma_commit(&bars[kFin]);
        mbar_wait(&bars[kFin], 0, WaitGuard{p.err, p.wait_ns}, kSiteFinal);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kSoftWarps + 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

template <int D, int WHICH, bool F16, int SB>
int launch_tc_sb(const TcParams& p0, cudaStream_t stream) {
    const int smem = p0.plan.smem_bytes;
    auto kernel = tc_kernel<D, WHICH, F16, SB>;
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

// The forward at D <= 32 comes in two forms, with two or three score buffers, as its plan says; the
// three-buffer kernels are instantiated in a translation unit of their own (na_tc_sb3.cu).
template <int D, int WHICH, bool F16>
int launch_tc(const TcParams& p, cudaStream_t stream) {
    if constexpr (WHICH == 0 && D <= 32) {
        if (p.plan.sbufs == 3) return launch_fwd_tc_sb3(p, stream);
    }
    return launch_tc_sb<D, WHICH, F16, 2>(p, stream);
}

}  // namespace
}  // namespace na
