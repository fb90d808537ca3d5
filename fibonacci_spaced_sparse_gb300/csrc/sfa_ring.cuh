// sfa_ring.cuh -- the tile map and the shared-memory load ring of the
// tensor-core kernels of libsfa (forward and backward), private to the CUDA
// library.
//
// A CTA owns tiles of TQ consecutive queries of one sequence and one
// key/value head.  For such a tile the keys it reads are the window block
// (rows i0 - W .. i0 + TQ - 1) and, per rung of distance d = alpha f, the one
// contiguous block of rows i0 - floor(d) - 1 .. i0 + TQ - 1 - floor(d): the
// offsets are shared by every query ("Attended set", section 2 of
// "Depth-Staggered Fibonacci Spacing for Sparse Attention", arXiv 2606.28560).
// One producer lane moves these blocks of Khat and V with tiled TMA boxes into
// an mbarrier ring: one query slot (the tile's query rows), one window slot
// (with the RoPE rows of the tile's queries) and NGS group slots of RPG rungs
// each; the consumer warps release slots with one arrival each.  Every wait is bounded: a wait that gives up sets the
// CTA's abort flag and SFA_DEVSTAT_WAIT_TIMEOUT in the status word.
//
// A parameter struct PP used with these templates provides: kmap_w, vmap_w
// (window boxes of win_rows rows), kmap_r[RPG], vmap_r[RPG] (rung boxes),
// a (LayerArgs), rope, status, ntq, ntiles, step_g, step_tq, step_b, win_rows,
// win_region, kQMaps (static, >= 1) tile maps qmaps[] of per-query
// [B][T][8][64] tensors that the query slot carries, and kWinRope (static):
// whether the window slot also carries the RoPE rows of the tile's queries
// (then also tabmap, the map of encode_table over the RoPE table).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "sfa_internal.cuh"
#include "sfa_mma.cuh"

namespace sfa {
namespace ring {

using namespace mma;

constexpr int TQ = 28;                 // queries per tile
constexpr int RPG = 4;                 // rungs per group (one M tile of a query pair)
constexpr int NGS = 2;                 // group slots
constexpr int RUNG_ROWS = TQ + 1;      // rows a rung block needs
constexpr int RUNG_BOX = RUNG_ROWS + 2 * (RPG - 1);
constexpr int ROWB = 128;              // bytes of one 64-element bf16 row
constexpr int TABB = kPairs * 8;       // bytes of one RoPE table row (32 x (cos, sin))
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kNoRung = 1 << 30;       // ceiling of a rung no query of the tile uses

constexpr unsigned round1k(unsigned x) { return (x + 1023u) & ~1023u; }
// A group slot holds the Khat regions of rung positions 0..RPG-1, then their V
// regions.  Position p's box has RUNG_ROWS + 2p rows; each region starts on a
// 1024-byte boundary (the period of the 128-byte swizzle).
constexpr unsigned rung_region_bytes(int p) { return round1k((RUNG_ROWS + 2 * p) * ROWB); }
constexpr unsigned rung_region_off(int p) { return p == 0 ? 0u : rung_region_off(p - 1) + rung_region_bytes(p - 1); }
constexpr unsigned kVOff = rung_region_off(RPG);            // V region of p = Khat region of p + kVOff
// The same offsets in closed form (TQ = 28: 4, 4, 5, 5 KB regions), for
// run-time positions.
__host__ __device__ constexpr unsigned rung_off(int p) { return (unsigned)p * 4096u + (p >= 3 ? 1024u : 0u); }
static_assert(rung_off(0) == rung_region_off(0) && rung_off(1) == rung_region_off(1) &&
                  rung_off(2) == rung_region_off(2) && rung_off(3) == rung_region_off(3),
              "rung region offsets");
constexpr unsigned kGroupSlotBytes = 2 * kVOff;
constexpr unsigned kHeaderBytes = 1024;                     // barriers, flag, rung table
constexpr unsigned kQTileBytes = TQ * kG * ROWB;            // one [TQ][4 heads][64] bf16 query tile

// -------------------------------------------------------------- tile map

// Tile t = (b * ntq + tq) * Hkv + g covers queries i0 = tq * TQ .. of
// sequence b, key/value head g.  A CTA takes tiles blockIdx.x, + gridDim.x, ...
struct Tile {
    int b, g, tq, i0;
};

template <class PP>
__device__ __forceinline__ Tile decode(const PP& P, int t) {
    Tile x;
    x.g = t % kHkv;
    const int rest = t / kHkv;
    x.tq = rest % P.ntq;
    x.b = rest / P.ntq;
    x.i0 = x.tq * TQ;
    return x;
}

// The tile gridDim.x further on.
template <class PP>
__device__ __forceinline__ Tile next_tile(const PP& P, const Tile& x) {
    Tile y;
    y.g = x.g + P.step_g;
    const int cg = y.g >= kHkv;
    y.g -= cg ? kHkv : 0;
    y.tq = x.tq + P.step_tq + cg;
    const int ct = y.tq >= P.ntq;
    y.tq -= ct ? P.ntq : 0;
    y.b = x.b + P.step_b + ct;
    y.i0 = y.tq * TQ;
    return y;
}

// ---------------------------------------------------------- smem layout

struct SRung {
    int n;
    float t;
    int c;
};

struct TC {
    float t;
    int c;
};

struct Smem {
    uint32_t bars;      // full_w, empty_w, full_g[NGS], empty_g[NGS], full_q, empty_q
    uint32_t qslot;     // the query slot
    uint32_t win;       // the window slot
    uint32_t rung;      // NGS group slots
    uint32_t obuf;      // the consumer warps' output staging buffers
    int* abort_flag;
    int* kt;            // rungs usable by the window slot's tile
    const SRung* r;     // the kept rungs, by increasing distance
    uint32_t tc;        // shared address of TC[nr] (t and ceil of each kept rung)
};

__device__ __forceinline__ uint32_t bar_full_w(const Smem& s) { return s.bars; }
__device__ __forceinline__ uint32_t bar_empty_w(const Smem& s) { return s.bars + 8; }
__device__ __forceinline__ uint32_t bar_full_g(const Smem& s, int i) { return s.bars + 16 + 8 * i; }
__device__ __forceinline__ uint32_t bar_empty_g(const Smem& s, int i) { return s.bars + 16 + 8 * (NGS + i); }
__device__ __forceinline__ uint32_t bar_full_q(const Smem& s) { return s.bars + 16 + 16 * NGS; }
__device__ __forceinline__ uint32_t bar_empty_q(const Smem& s) { return s.bars + 24 + 16 * NGS; }
constexpr int kBarBytes = 32 + 16 * NGS;
constexpr int kFlagOffset = kBarBytes;
constexpr int kKtOffset = kFlagOffset + 4;
constexpr int kRungTableOffset = 256;
constexpr int kTcOffset = kRungTableOffset + SFA_MAX_RUNGS * 12;  // {t, ceil} per rung, 8 bytes
static_assert(kKtOffset + 4 <= kRungTableOffset, "header overflow");
static_assert(rung_region_off(1) == 4096 && kVOff == 18432, "rung region layout");
static_assert(kTcOffset + SFA_MAX_RUNGS * 8 <= (int)kHeaderBytes, "header overflow");

// Rungs are sorted by ceil(d): those usable by some query of the tile form a prefix.
__device__ __forceinline__ int active_rungs(const Smem& S, int nr, int i0) {
    int n = 0;
    while (n < nr && S.r[n].c <= i0 + TQ - 1) ++n;
    return n;
}

// ------------------------------------------------------------ producer

// Window block of tile x (and its RoPE rows) into the window slot; returns
// the number of rungs the tile uses (published to the consumers in S.kt).
template <class PP>
__device__ __forceinline__ bool load_window(const PP& P, const Smem& S, const Tile& x, int& wcount,
                                            int& kt) {
    if (!mbar_wait(bar_empty_w(S), (wcount & 1) ^ 1, S.abort_flag)) return false;
    const int nq = min(TQ, P.a.T - x.i0);
    const uint32_t tab_bytes = (PP::kWinRope && P.rope) ? (uint32_t)TQ * TABB : 0u;
    kt = active_rungs(S, P.a.nr, x.i0);
    *S.kt = kt;  // published by the arrive below
    const uint32_t full = bar_full_w(S);
    mbar_arrive_expect_tx(full, 2u * P.win_rows * ROWB + tab_bytes);
    tma_load_4d(S.win, &P.kmap_w, 0, x.g, x.i0 - P.a.W, x.b, full);
    tma_load_4d(S.win + P.win_region, &P.vmap_w, 0, x.g, x.i0 - P.a.W, x.b, full);
    // RoPE rows of the tile's query positions (read by the consumers' Q
    // rotation), in the layout of tab_chunk; rows past T are zero filled
    if (tab_bytes) tma_load_4d(S.win + 2 * P.win_region, &P.tabmap, 0, 0, x.i0, 0, full);
    ++wcount;
    return true;
}

// The per-query tensors of tile x (rows (query, head) of the key/value head's
// 4 query heads, PP::kQMaps of them) into the query slot.  The consumers free
// that slot as soon as they have read it at the start of a tile, so the next
// tile's query rows load while the current tile is computed.
template <class PP>
__device__ __forceinline__ bool load_q(const PP& P, const Smem& S, const Tile& x, int& qcount) {
    if (!mbar_wait(bar_empty_q(S), (qcount & 1) ^ 1, S.abort_flag)) return false;
    const uint32_t full = bar_full_q(S);
    mbar_arrive_expect_tx(full, PP::kQMaps * kQTileBytes);
    for (int m = 0; m < PP::kQMaps; ++m)
        tma_load_4d(S.qslot + m * kQTileBytes, &P.qmaps[m], 0, x.g * kG, x.i0, x.b, full);
    ++qcount;
    return true;
}

// Rung group k0 .. k0 + 3 of tile x into the next group slot.
template <class PP>
__device__ __forceinline__ bool load_group(const PP& P, const Smem& S, const Tile& x, int k0, int kt,
                                           int& gcount) {
    const int slot = gcount & (NGS - 1);
    if (!mbar_wait(bar_empty_g(S, slot), ((gcount / NGS) & 1) ^ 1, S.abort_flag)) return false;
    const int np = min(RPG, kt - k0);
    const uint32_t base = S.rung + slot * kGroupSlotBytes;
    const uint32_t full = bar_full_g(S, slot);
    uint32_t bytes = 0;
    for (int p = 0; p < np; ++p) bytes += 2u * (RUNG_ROWS + 2 * p) * ROWB;
    mbar_arrive_expect_tx(full, bytes);
    for (int p = 0; p < np; ++p) {
        const int row0 = x.i0 - S.r[k0 + p].n - 1 - 2 * p;
        const uint32_t dst = base + rung_off(p);
        tma_load_4d(dst, &P.kmap_r[p], 0, x.g, row0, x.b, full);
        tma_load_4d(dst + kVOff, &P.vmap_r[p], 0, x.g, row0, x.b, full);
    }
    ++gcount;
    return true;
}

// Load order: window(t), its first two rung groups, window(t + 1) (the
// consumers free the window slot before their rung phase, so the next
// window is in flight while they work on the rungs), the rest of t's groups,
// and so on.
template <class PP>
__device__ void producer(const PP& P, const Smem& S) {
    int wcount = 0, gcount = 0, qcount = 0;
    // Khat is written by the launch before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    Tile x = decode(P, blockIdx.x);
    int kt = 0;
    if (blockIdx.x < P.ntiles && !load_q(P, S, x, qcount)) goto fail;
    if (blockIdx.x < P.ntiles && !load_window(P, S, x, wcount, kt)) goto fail;
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x) {
        const Tile nx = next_tile(P, x);
        const bool more = t + (int)gridDim.x < P.ntiles;
        const int ng = (kt + RPG - 1) / RPG;
        const int split = min(2, ng);
        int nkt = 0;
        for (int gi = 0; gi < ng; ++gi) {
            if (gi == split && more && (!load_q(P, S, nx, qcount) || !load_window(P, S, nx, wcount, nkt)))
                goto fail;
            if (!load_group(P, S, x, gi * RPG, kt, gcount)) goto fail;
        }
        if (split == ng && more && (!load_q(P, S, nx, qcount) || !load_window(P, S, nx, wcount, nkt))) goto fail;
        x = nx;
        kt = nkt;
    }
    return;
fail:
    *S.abort_flag = 1;
    if (P.status) atomicOr(P.status, SFA_DEVSTAT_WAIT_TIMEOUT);
    // no copy of this CTA may land after it exits: wait (bounded) for every
    // slot's last announced phase
    if (qcount > 0) (void)mbar_wait(bar_full_q(S), (qcount - 1) & 1, nullptr);
    if (wcount > 0) (void)mbar_wait(bar_full_w(S), (wcount - 1) & 1, nullptr);
    for (int n = max(0, gcount - NGS); n < gcount; ++n)
        (void)mbar_wait(bar_full_g(S, n & (NGS - 1)), (n / NGS) & 1, nullptr);
}

// Warp-uniform bounded wait (every lane polls, the warp leaves together).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
    const unsigned long long t0 = now_ns();
    for (unsigned it = 0;; ++it) {
        if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
        if (__any_sync(kFull, *abort_flag != 0)) return false;
        if ((it & 15) == 15 && __any_sync(kFull, now_ns() - t0 > kWaitNs)) return false;
        __nanosleep(32);
    }
}

__device__ __forceinline__ TC lds_tc(uint32_t addr) {
    TC v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=f"(v.t), "=r"(v.c) : "r"(addr));
    return v;
}

// Byte offset, in the window slot's RoPE rows, of 16-byte chunk c (pairs
// 2 c, 2 c + 1) of tile row p.  A row is two 128-byte lines L = 2 p + c / 8
// loaded under the 128-byte swizzle (the region is 1024-byte aligned), which
// stores chunk c % 8 of line L at chunk (c % 8) ^ (L % 8): the lanes of a warp
// that read the same chunk of neighbouring rows then hit different banks.
__device__ __forceinline__ uint32_t tab_chunk(int p, int c) {
    const int line = 2 * p + (c >> 3);
    return (uint32_t)(line * 128 + ((((c & 7) ^ line) & 7) << 4));
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// RoPE of two rotation pairs held as bf16 pairs x = (x_m, x_m+1) (dimensions
// m, m + 1) and y (their partners + D/2), c = (cos_m, sin_m, cos_m+1,
// sin_m+1): the rotated x and y halves, packed to bf16.  Explicit roundings
// (the product rounded to fp32, one fused multiply-add, round to nearest
// bf16), so that every kernel that rotates queries or keys produces the same
// bits.
__device__ __forceinline__ uint32_t rope_x(float2 x, float2 y, float4 c) {
    return pack_bf16(__fmaf_rn(x.x, c.x, __fmul_rn(-y.x, c.y)), __fmaf_rn(x.y, c.z, __fmul_rn(-y.y, c.w)));
}
__device__ __forceinline__ uint32_t rope_y(float2 x, float2 y, float4 c) {
    return pack_bf16(__fmaf_rn(y.x, c.x, __fmul_rn(x.x, c.y)), __fmaf_rn(y.y, c.z, __fmul_rn(x.y, c.w)));
}

__device__ __forceinline__ uint4 lds_u4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int w) {
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

__device__ __forceinline__ uint32_t swz_row(int r, int hi) {
    return (uint32_t)(r * ROWB) + (uint32_t)(((hi ^ r) & 7) << 4);
}

// Offset of the row that this lane gives to ldmatrix for rung position p of
// unit u: M row (e, kind) of rung p is block row u + e + kind, stored 2p rows
// into its box.
__device__ __forceinline__ uint32_t rung_row(int p, int u, int e, int kind, int hi, bool v) {
    return rung_off(p) + (v ? kVOff : 0u) + swz_row(u + e + kind + 2 * p, hi);
}


// Carves the dynamic shared memory of a ring kernel (1024 spare bytes reach
// the 1024-byte alignment of the swizzled regions), copies the kept rungs into
// the header and initialises the barriers: full barriers take one arrival
// (the producer's expect_tx) plus the copied bytes, empty barriers one
// arrival per consumer warp (ncw of them).  Ends with a CTA barrier.
__device__ __forceinline__ Smem ring_setup(const LayerArgs& a, int ncw, unsigned qslot_bytes,
                                           unsigned win_slot_bytes, unsigned char* smem_raw) {
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    unsigned char* hdr = smem_raw + (base - raw_base);
    Smem S;
    S.bars = base;
    S.abort_flag = reinterpret_cast<int*>(hdr + kFlagOffset);
    S.kt = reinterpret_cast<int*>(hdr + kKtOffset);
    SRung* table = reinterpret_cast<SRung*>(hdr + kRungTableOffset);
    S.r = table;
    S.qslot = base + kHeaderBytes;
    S.win = S.qslot + qslot_bytes;
    S.rung = S.win + win_slot_bytes;
    S.obuf = S.rung + NGS * kGroupSlotBytes;
    S.tc = base + kTcOffset;
    if (threadIdx.x < a.nr) {
        const Rung rg = a.r[threadIdx.x];
        table[threadIdx.x] = SRung{rg.n, rg.t, rg.c};
        reinterpret_cast<TC*>(hdr + kTcOffset)[threadIdx.x] = TC{rg.t, rg.c};
    }
    if (threadIdx.x == 0) {
        mbar_init(bar_full_w(S), 1);
        mbar_init(bar_empty_w(S), ncw);
        for (int i = 0; i < NGS; ++i) {
            mbar_init(bar_full_g(S, i), 1);
            mbar_init(bar_empty_g(S, i), ncw);
        }
        mbar_init(bar_full_q(S), 1);
        mbar_init(bar_empty_q(S), ncw);
        *S.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    return S;
}

// ------------------------------------------------------------- host side

// Number of SMs of device dev (looked up once).
inline int sm_count(int dev, cudaError_t* err) {
    static int sms[64];
    int& n = sms[dev & 63];
    if (n == 0) {
        const cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) {
            *err = e;
            n = 0;
            return 0;
        }
    }
    *err = cudaSuccess;
    return n;
}

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 4-D map over a [B][T][8][64] bf16 tensor (innermost first: d, head, t, b),
// box of `queries` queries x 4 heads, 128-byte swizzle, zero fill outside.
inline bool encode_heads(CUtensorMap* m, const void* base, int B, int T, int queries) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kHq, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)kHq * kD * 2, (cuuint64_t)T * kHq * kD * 2};
    const cuuint32_t box[4] = {(cuuint32_t)kD, (cuuint32_t)kG, (cuuint32_t)queries, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over O [B][T][8][64] bf16 (innermost first: d, head, t, b), box of
// 2 queries x 4 heads, 128-byte swizzle (the staging buffer's layout).
inline bool encode_out(CUtensorMap* m, void* base, int B, int T) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kHq, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)kHq * kD * 2, (cuuint64_t)T * kHq * kD * 2};
    const cuuint32_t box[4] = {(cuuint32_t)kD, (cuuint32_t)kG, 2u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over a [B][T][Hkv][64] bf16 tensor (innermost first: d, g, t, b),
// box of `rows` rows of one head, 128-byte swizzle, zero fill outside.
inline bool encode_rows(CUtensorMap* m, const void* base, int B, int T, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kHkv, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)kHkv * kD * 2,
                                   (cuuint64_t)T * kHkv * kD * 2};
    const cuuint32_t box[4] = {(cuuint32_t)kD, 1u, (cuuint32_t)rows, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map over the RoPE table's first T positions, each 32 (cos, sin) pairs of
// fp32 seen as two 128-byte lines of 32 floats (innermost first: float,
// line, position, 1), box of TQ positions, 128-byte swizzle: the layout that
// tab_chunk addresses.
inline bool encode_table(CUtensorMap* m, const float2* rope, int T) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {32u, 2u, (cuuint64_t)T, 1u};
    const cuuint64_t strides[3] = {128u, (cuuint64_t)TABB, (cuuint64_t)T * TABB};
    const cuuint32_t box[4] = {32u, 2u, (cuuint32_t)TQ, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float2*>(rope), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ring
}  // namespace sfa
