// sfa_fwd_mma.cu -- bf16 forward on the tensor cores (mma.sync m16n8k16,
// fp32 accumulation), the fast path of sfa_forward.
//
// The method is the attention of "Depth-Staggered Fibonacci Spacing for Sparse
// Attention" (arXiv 2606.28560), section 2 "Attended set": query i attends the
// window distances 0..W and one interpolated row per rung at d = alpha f; the
// offsets are shared by every query, so for a tile of consecutive queries each
// rung is ONE contiguous block of key/value rows (a shift, not a gather list).
//
// Two launches:
//  1. rope_k_kernel: Khat = RoPE(K) at the true positions, bf16, into the
//     caller's workspace (every key row is rotated once, then re-read from L2
//     by every tile that needs it).
//  2. fwd_mma_kernel, persistent, (1 producer + 7 consumer) warps per CTA.
//     A CTA owns a tile of TQ = 28 consecutive queries of one sequence b and
//     one key/value head g (4 query heads).  The producer (one lane) loads,
//     with tiled TMA boxes, the window block (rows i0 - W .. i0 + TQ - 1) and,
//     per rung k, the block of rows i0 - n_k - 1 .. i0 + TQ - 1 - n_k of Khat
//     and V into an mbarrier ring of shared-memory slots (rows outside the
//     sequence arrive as zeros), plus the RoPE rows of the tile's queries.
//     Each consumer warp owns two query pairs.  For a pair (i, i + 1) the
//     scores are formed "keys on M": S^T = Khat_rows (16 x 64) . Qhat^T
//     (64 x 8), N = 2 queries x 4 heads.  Five rungs share one 16-row M tile
//     (rows i - n - 1, i - n, i - n + 1 per rung); the lerp acts on the
//     scores, s = (1 - t) s(row i - n) + t s(row i - n - 1), which equals the
//     score of the interpolated key by linearity, and the probability p is
//     split back onto the two rows as p (1 - t) and p t, so P^T V_rows forms
//     the interpolated value.  One online softmax (base 2, lazy rescale: the
//     running max is raised only when a score exceeds it by more than 2^8)
//     runs over window and rung entries; O^T accumulates in registers and is
//     transposed with movmatrix on the way out.
//
// Shared memory: each tensor region of a slot is 1024-byte aligned and filled
// by TMA with the 128-byte swizzle (16-byte chunk c of region row r stored at
// chunk c ^ (r & 7)).  The box of rung position p of an M tile starts
// (3p mod 8) rows early, so the rows the consumers read from different rungs
// of one tile fall in different swizzle phases and every ldmatrix (8 rows)
// touches 8 different bank groups.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "sfa_internal.cuh"
#include "sfa_mma.cuh"

namespace sfa {

namespace {

using namespace mma;

constexpr int TQ = 28;                 // queries per tile
constexpr int NCW = 7;                 // consumer warps (2 query pairs each)
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int NRS = 8;                 // rung slots
constexpr int NWS = 1;                 // window slots (free again after the window phase)
constexpr int MAXPH = 7;               // largest box offset of a rung position
constexpr int RUNG_ROWS = TQ + 1;      // rows a rung block needs
constexpr int RUNG_BOX = RUNG_ROWS + MAXPH;
constexpr int ROWB = 128;              // bytes of one 64-element bf16 row
constexpr int TABB = kPairs * 8;       // bytes of one RoPE table row (32 x (cos, sin))
constexpr int RUNGS_PER_TILE = 5;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.0f;          // raise the running max past this margin

constexpr unsigned round1k(unsigned x) { return (x + 1023u) & ~1023u; }
constexpr unsigned kRungRegion = round1k(RUNG_BOX * ROWB);  // one tensor of a rung slot
constexpr unsigned kRungSlotBytes = 2 * kRungRegion;        // Khat region, then V region
constexpr unsigned kHeaderBytes = 1024;                     // barriers, flag, rung table
constexpr unsigned kObufBytes = 2 * 8 * ROWB;                // per consumer warp: O of 2 query pairs

struct FwdParams {
    CUtensorMap kmap_w;      // Khat, box of win_rows rows
    CUtensorMap vmap_w;      // V, box of win_rows rows
    CUtensorMap kmap_r[5];   // Khat, box of RUNG_ROWS + rung_phase(p) rows, rung position p
    CUtensorMap vmap_r[5];   // V, same boxes
    CUtensorMap omap;        // O [B][T][8][64], box of 2 queries x 4 heads, 128-byte swizzle
    LayerArgs a;
    const __nv_bfloat16* q;
    const float2* rope;      // nullptr: Q is used as given
    __nv_bfloat16* o;
    float* lse;
    unsigned* status;
    int ntq;                 // query tiles per sequence
    int ntiles;              // B * ntq * Hkv
    int win_rows;            // TQ + W
    int nwt;                 // window M tiles of a query quad (W + 4 rows)
    unsigned win_region;     // bytes of one tensor region of a window slot
    unsigned win_slot_bytes; // Khat + V regions and the tile's RoPE rows
};

__device__ __forceinline__ int rung_phase(int p) { return (3 * p) & 7; }

// -------------------------------------------------------------- tile map

struct Tile {
    int b, g, i0;
};

__device__ __forceinline__ Tile decode(const FwdParams& P, int t) {
    Tile x;
    x.g = t % kHkv;
    const int rest = t / kHkv;
    x.i0 = (rest % P.ntq) * TQ;
    x.b = rest / P.ntq;
    return x;
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
    uint32_t bars;      // full_w[NWS], empty_w[NWS], full_r[NRS], empty_r[NRS]
    uint32_t win;       // NWS window slots
    uint32_t rung;      // NRS rung slots
    uint32_t obuf;      // NCW output staging buffers
    int* abort_flag;
    int* kt;            // per window slot: rungs usable by the slot's tile
    const SRung* r;     // the kept rungs, by increasing distance
    uint32_t tc;        // shared address of TC[nr] (t and ceil of each kept rung)
};

__device__ __forceinline__ uint32_t bar_full_w(const Smem& s, int i) { return s.bars + 8 * i; }
__device__ __forceinline__ uint32_t bar_empty_w(const Smem& s, int i) { return s.bars + 8 * (NWS + i); }
__device__ __forceinline__ uint32_t bar_full_r(const Smem& s, int i) { return s.bars + 8 * (2 * NWS + i); }
__device__ __forceinline__ uint32_t bar_empty_r(const Smem& s, int i) {
    return s.bars + 8 * (2 * NWS + NRS + i);
}
constexpr int kBarBytes = 8 * 2 * (NWS + NRS);
constexpr int kFlagOffset = kBarBytes;
constexpr int kKtOffset = kFlagOffset + 4;   // per window slot: rungs usable by its tile
constexpr int kRungTableOffset = 256;
constexpr int kTcOffset = kRungTableOffset + SFA_MAX_RUNGS * 12;  // {t, ceil} per rung, 8 bytes
static_assert(kKtOffset + 4 * NWS <= kRungTableOffset, "header overflow");
static_assert(kTcOffset + SFA_MAX_RUNGS * 8 <= (int)kHeaderBytes, "header overflow");

// Rungs are sorted by ceil(d): those usable by some query of the tile form a prefix.
__device__ __forceinline__ int active_rungs(const Smem& S, int nr, int i0) {
    int n = 0;
    while (n < nr && S.r[n].c <= i0 + TQ - 1) ++n;
    return n;
}

// ------------------------------------------------------------ producer

__device__ void producer(const FwdParams& P, const Smem& S) {
    int wcount = 0, rcount = 0;
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x) {
        const Tile x = decode(P, t);
        {
            const int slot = wcount % NWS;
            if (!mbar_wait(bar_empty_w(S, slot), ((wcount / NWS) & 1) ^ 1, S.abort_flag)) goto fail;
            const uint32_t base = S.win + slot * P.win_slot_bytes;
            const uint32_t full = bar_full_w(S, slot);
            const int nq = min(TQ, P.a.T - x.i0);
            const uint32_t tab_bytes = P.rope ? (uint32_t)nq * TABB : 0u;
            S.kt[slot] = active_rungs(S, P.a.nr, x.i0);  // published by the arrive below
            mbar_arrive_expect_tx(full, 2u * P.win_rows * ROWB + tab_bytes);
            tma_load_4d(base, &P.kmap_w, 0, x.g, x.i0 - P.a.W, x.b, full);
            tma_load_4d(base + P.win_region, &P.vmap_w, 0, x.g, x.i0 - P.a.W, x.b, full);
            // RoPE rows of the tile's query positions (read by the consumers' Q rotation)
            if (P.rope)
                bulk_g2s(base + 2 * P.win_region, P.rope + (size_t)x.i0 * kPairs, tab_bytes, full);
            ++wcount;
        }
        {
            const int kt = S.kt[(wcount - 1) % NWS];
            for (int k = 0; k < kt; ++k) {
                const int slot = rcount & (NRS - 1);
                if (!mbar_wait(bar_empty_r(S, slot), ((rcount / NRS) & 1) ^ 1, S.abort_flag)) goto fail;
                const uint32_t base = S.rung + slot * kRungSlotBytes;
                const uint32_t full = bar_full_r(S, slot);
                const int pos = k % RUNGS_PER_TILE;
                const int ph = rung_phase(pos);
                const int row0 = x.i0 - S.r[k].n - 1 - ph;
                mbar_arrive_expect_tx(full, 2u * (RUNG_ROWS + ph) * ROWB);
                tma_load_4d(base, &P.kmap_r[pos], 0, x.g, row0, x.b, full);
                tma_load_4d(base + kRungRegion, &P.vmap_r[pos], 0, x.g, row0, x.b, full);
                ++rcount;
            }
        }
    }
    return;
fail:
    *S.abort_flag = 1;
    if (P.status) atomicOr(P.status, SFA_DEVSTAT_WAIT_TIMEOUT);
    // no copy of this CTA may land after it exits: wait (bounded) for every
    // slot's last announced phase
    for (int n = max(0, wcount - NWS); n < wcount; ++n)
        (void)mbar_wait(bar_full_w(S, n % NWS), (n / NWS) & 1, nullptr);
    for (int n = max(0, rcount - NRS); n < rcount; ++n)
        (void)mbar_wait(bar_full_r(S, n % NRS), (n / NRS) & 1, nullptr);
}

// ------------------------------------------------------------ consumers

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

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// One query pair (i, i + 1) of one key/value head: the B fragments of
// Qhat^T (scaled into log2 units), the O^T accumulators and softmax state of
// this thread's two columns (query tig/2, heads 2(tig&1) and 2(tig&1)+1).
struct Unit {
    uint32_t qf[4][2];
    float o[4][4];
    float m[2];
    float th[2];   // m + lazy margin: a score above it raises the running max
    float l[2];
};

// Per-thread constants of the fragment layouts (fixed for the whole kernel:
// the warp always owns the query pairs at tile offsets u0 and u0 + 2).
// Addresses are byte offsets inside a slot region, with the 128-byte swizzle
// of ldmatrix k-step (or m tile) 0 folded in: step s reads at offset ^ (s << 5).
struct Lane {
    int g8, q;          // fragment row group; query of this thread's C columns
    int pk, pv;         // rung position of the rows this lane feeds to ldmatrix (5: pad)
    int p_lo, p_hi;     // rung position of this thread's C rows g8 and g8 + 8
    bool b_lo, b_hi;    // that row is row b of query q's interpolation
    unsigned wmask;     // window: bit (8 wt + 4 k + e) = row is a window distance of
                        // quad query 2k + q (before the sequence-start check)
    uint32_t kr[2], krp[2];   // rung tiles, unit k: Khat row offset (rung row / pad row)
    uint32_t vr[2], vrp[2];   // rung tiles, unit k: V row offset (rung row / pad row)
    uint32_t wk, wv;          // window tile 0: Khat and V row offsets
    uint32_t ob[2];           // output staging: stmatrix row address offsets (jj = 0, 1)
};

__device__ __forceinline__ uint32_t swz_row(int r, int hi) {
    return (uint32_t)(r * ROWB) + (uint32_t)(((hi ^ r) & 7) << 4);
}

__device__ __forceinline__ Lane make_lane(int lane, int u0, int W, int win_rows) {
    Lane L;
    L.g8 = lane >> 2;
    L.q = (lane & 3) >> 1;
    const int hk = lane >> 4, hv = (lane >> 3) & 1;
    const int rk = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int rv = (lane & 7) + ((lane >> 4) << 3);
    L.pk = rk < 15 ? rk / 3 : 5;
    L.pv = rv < 15 ? rv / 3 : 5;
    const int ok = rk < 15 ? rk - 3 * L.pk + rung_phase(L.pk) : 0;
    const int ov = rv < 15 ? rv - 3 * L.pv + rung_phase(L.pv) : 0;
    for (int k = 0; k < 2; ++k) {
        const int u = u0 + 2 * k;
        // pad row: a row TMA wrote for rung 0 (box rows 0..RUNG_ROWS-1) in the
        // swizzle phase u + 7 that no other row of the tile uses
        const int pad = (u + 7 <= RUNG_ROWS - 1) ? u + 7 : u - 1;
        L.kr[k] = swz_row(u + ok, hk);
        L.krp[k] = swz_row(pad, hk);
        L.vr[k] = swz_row(u + ov, hv);
        L.vrp[k] = swz_row(pad, hv);
    }
    L.wk = swz_row(min(u0 + rk, win_rows - 1), hk);
    L.wv = swz_row(min(u0 + rv, win_rows - 1), hv);
    const int rlo = L.g8, rhi = L.g8 + 8;
    L.p_lo = rlo / 3;
    L.p_hi = rhi < 15 ? rhi / 3 : 5;
    L.b_lo = (rlo - 3 * L.p_lo) == L.q;
    L.b_hi = rhi < 15 && (rhi - 3 * L.p_hi) == L.q;
    L.wmask = 0u;
    for (int wt = 0; wt < 3; ++wt)
        for (int k = 0; k < 2; ++k)
            for (int e = 0; e < 4; ++e) {
                const int R = 16 * wt + L.g8 + ((e >> 1) << 3);
                const int qq = 2 * k + L.q;
                if (R >= qq && R <= W + qq) L.wmask |= 1u << (8 * wt + 4 * k + e);
            }
    // stmatrix: stored matrix mi = lane >> 3 of call jj is (m tile 2 jj + mi/2,
    // half mi & 1); this lane gives its row (lane & 7) = output row (query, head)
    const int row = lane & 7, mi = lane >> 3;
    for (int jj = 0; jj < 2; ++jj) {
        const int chunk = 2 * (2 * jj + (mi >> 1)) + (mi & 1);
        L.ob[jj] = (uint32_t)(row * ROWB) + (uint32_t)(((chunk ^ row) & 7) << 4);
    }
    return L;
}

// Raw Q of this thread's B-fragment column (query i0 + u + g8/4, head
// g*4 + g8%4): dimensions 16 s + 8 h + 2 tig + {0, 1}.
__device__ __forceinline__ void fetch_q(const FwdParams& P, const Tile& x, int u, int lane,
                                        uint32_t raw[4][2]) {
    const int g8 = lane >> 2, tig = lane & 3;
    const int iq = min(x.i0 + u + (g8 >> 2), P.a.T - 1);  // rows past the end are not stored
    const __nv_bfloat16* qp =
        P.q + (((size_t)x.b * P.a.T + iq) * kHq + x.g * kG + (g8 & 3)) * kD + 2 * tig;
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
        raw[s2][0] = __ldg(reinterpret_cast<const unsigned*>(qp + 16 * s2));
        raw[s2][1] = __ldg(reinterpret_cast<const unsigned*>(qp + 16 * s2 + 8));
    }
}

// Rotate (RoPE rows of the tile in shared memory at `tab`, nq of them) and
// scale the raw Q into B fragments; reset the accumulators.
__device__ __forceinline__ void start_unit(const FwdParams& P, uint32_t tab, int nq, int u, int lane,
                                           const uint32_t raw[4][2], Unit& U) {
    const int g8 = lane >> 2, tig = lane & 3;
    const float sl2 = P.a.scale * kLog2e;
    const uint32_t trow = tab + (uint32_t)(min(u + (g8 >> 2), nq - 1) * TABB + 2 * tig * 8);
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // dims m = 16 s + 8 h + 2 tig + {0, 1} and their partners m + 32
            float4 cs = make_float4(sl2, 0.f, sl2, 0.f);
            if (P.rope) {
                cs = lds_f4(trow + (uint32_t)((16 * s2 + 8 * h) * 8));
                cs.x *= sl2;
                cs.y *= sl2;
                cs.z *= sl2;
                cs.w *= sl2;
            }
            const float2 xv = unpack_bf16(raw[s2][h]);
            const float2 yv = unpack_bf16(raw[s2 + 2][h]);
            U.qf[s2][h] = pack_bf16(xv.x * cs.x - yv.x * cs.y, xv.y * cs.z - yv.y * cs.w);
            U.qf[s2 + 2][h] = pack_bf16(yv.x * cs.x + xv.x * cs.y, yv.y * cs.z + xv.y * cs.w);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) U.o[j][e] = 0.f;
}

// The next tile's raw Q is fetched while this tile is computed.

// Softmax of the first window entries of a row: the running max becomes the
// column max of s (reduced over the 8 threads holding the column).
__device__ __forceinline__ void softmax_first(Unit& U, const float s[4], float p[4]) {
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int w = 4; w <= 16; w <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, w));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, w));
    }
    U.m[0] = mx0;
    U.m[1] = mx1;
    U.th[0] = mx0 + kLazy;
    U.th[1] = mx1 + kLazy;
    // a column without entries yet keeps m = -inf; its p are 0
    const float m0 = mx0 == -INFINITY ? 0.f : mx0, m1 = mx1 == -INFINITY ? 0.f : mx1;
    p[0] = fast_exp2(s[0] - m0);
    p[1] = fast_exp2(s[1] - m1);
    p[2] = fast_exp2(s[2] - m0);
    p[3] = fast_exp2(s[3] - m1);
    U.l[0] = p[0] + p[2];
    U.l[1] = p[1] + p[3];
}

// Raise the running max of this thread's two columns to the column max of s
// and rescale O^T and l.
__device__ __forceinline__ void raise_max(Unit& U, const float s[4]) {
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int w = 4; w <= 16; w <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, w));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, w));
    }
    const float n0 = fmaxf(U.m[0], mx0), n1 = fmaxf(U.m[1], mx1);
    const float c0 = (U.m[0] == -INFINITY) ? (n0 == -INFINITY ? 1.f : 0.f) : fast_exp2(U.m[0] - n0);
    const float c1 = (U.m[1] == -INFINITY) ? (n1 == -INFINITY ? 1.f : 0.f) : fast_exp2(U.m[1] - n1);
    U.m[0] = n0;
    U.m[1] = n1;
    U.th[0] = n0 + kLazy;
    U.th[1] = n1 + kLazy;
    U.l[0] *= c0;
    U.l[1] *= c1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        U.o[j][0] *= c0;
        U.o[j][2] *= c0;
        U.o[j][1] *= c1;
        U.o[j][3] *= c1;
    }
}

// Online-softmax step (lazy: the running max moves only when a score of the
// warp exceeds it by more than 2^8).  Returns the probabilities in p.
__device__ __forceinline__ void softmax_step(Unit& U, const float s[4], float p[4]) {
    const bool need = (s[0] > U.th[0]) || (s[2] > U.th[0]) || (s[1] > U.th[1]) || (s[3] > U.th[1]);
    if (__any_sync(kFull, need)) raise_max(U, s);
    const float m0 = U.m[0] == -INFINITY ? 0.f : U.m[0];
    const float m1 = U.m[1] == -INFINITY ? 0.f : U.m[1];
    p[0] = fast_exp2(s[0] - m0);
    p[1] = fast_exp2(s[1] - m1);
    p[2] = fast_exp2(s[2] - m0);
    p[3] = fast_exp2(s[3] - m1);
    U.l[0] += p[0] + p[2];
    U.l[1] += p[1] + p[3];
}

// Window M tile wt of the warp's query quad at tile offset u0 (positions
// i0 + u0 .. + 3): region rows u0 + R, R = 16 wt .. 16 wt + 15, hold
// positions i0 + u0 - W + R; unit k holds queries 2k, 2k + 1 of the quad.
__device__ __forceinline__ void window_tile(const FwdParams& P, uint32_t slot, int u0, int i0, int wt,
                                            const Lane& L, Unit* U) {
    const int lane = threadIdx.x & 31;
    uint32_t kro = L.wk, vro = L.wv;
    if (wt > 0) {
        const int maxr = P.win_rows - 1;
        kro = swz_row(min(u0 + 16 * wt + (lane & 7) + (((lane >> 3) & 1) << 3), maxr), lane >> 4);
        vro = swz_row(min(u0 + 16 * wt + (lane & 7) + ((lane >> 4) << 3), maxr), (lane >> 3) & 1);
    }
    float c[2][4];
#pragma unroll
    for (int k = 0; k < 2; ++k) c[k][0] = c[k][1] = c[k][2] = c[k][3] = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(slot + (kro ^ (uint32_t)(s2 << 5)), a0, a1, a2, a3);
#pragma unroll
        for (int k = 0; k < 2; ++k) mma16816(c[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
    }
    // window distances of each (row, query); near the sequence start, rows
    // below lo hold positions before it
    unsigned mask = L.wmask >> (8 * wt);
    const int lo = P.a.W - (i0 + u0) - 16 * wt;
    if (lo > 0) {
        if (L.g8 < lo) mask &= ~0x33u;          // rows g8 (e = 0, 1) of both units
        if (L.g8 + 8 < lo) mask &= ~0xccu;      // rows g8 + 8 (e = 2, 3)
    }
    uint32_t b[2][2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float sv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sv[e] = (mask >> (4 * k + e)) & 1u ? c[k][e] : -INFINITY;
        float p[4];
        if (wt == 0)
            softmax_first(U[k], sv, p);
        else
            softmax_step(U[k], sv, p);
        b[k][0] = movm_t(pack_bf16(p[0], p[1]));
        b[k][1] = movm_t(pack_bf16(p[2], p[3]));
    }
    const uint32_t vbase = slot + P.win_region;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vbase + (vro ^ (uint32_t)(j << 5)), a0, a1, a2, a3);
#pragma unroll
        for (int k = 0; k < 2; ++k) mma16816(U[k].o[j], a0, a1, a2, a3, b[k][0], b[k][1]);
    }
}

// Rung M tiles of the warp's two query pairs (tile offsets u0 and u0 + 2,
// positions i0 + u0 ..): np rungs (tile positions 0..np-1 = rungs k0..), rung
// p in ring slot (rc + p) mod NRS, its block row u + e (e = 0, 1, 2: rows
// i - n - 1 + e) stored rung_phase(p) rows into the slot.  The pad row 15
// and rows of absent rungs read a row of rung 0's slot in the swizzle phase
// no other row of the tile uses.  The two pairs are interleaved.
__device__ __forceinline__ void rung_tiles(const Smem& S, int rc, int np, int k0, int nr, int u0, int i0,
                                           const Lane& L, Unit* U) {
    const int lane = threadIdx.x & 31;
    const int g8 = L.g8;
    const bool kin = L.pk < np, vin = L.pv < np;
    const uint32_t kslot = S.rung + (uint32_t)(((rc + (kin ? L.pk : 0)) & (NRS - 1)) * kRungSlotBytes);
    const uint32_t vslot =
        S.rung + kRungRegion + (uint32_t)(((rc + (vin ? L.pv : 0)) & (NRS - 1)) * kRungSlotBytes);
    uint32_t krow[2], vrow[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        krow[k] = kslot + (kin ? L.kr[k] : L.krp[k]);
        vrow[k] = vslot + (vin ? L.vr[k] : L.vrp[k]);
    }
    // S^T = Khat_rows . Qhat^T, two accumulation chains per pair
    float c[2][4], d[2][4];
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[k][e] = d[k][e] = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(krow[k] ^ (uint32_t)(s2 << 5), a0, a1, a2, a3);
            mma16816((s2 & 1) ? d[k] : c[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
        }
    }
    // t and ceil of the rungs of this thread's rows (same for both pairs)
    const TC rlo = lds_tc(S.tc + (uint32_t)(min(k0 + L.p_lo, nr - 1) * 8));
    const TC rhi = lds_tc(S.tc + (uint32_t)(min(k0 + L.p_hi, nr - 1) * 8));
    const bool use_lo = L.b_lo && L.p_lo < np, use_hi = L.b_hi && L.p_hi < np;
    const float tl = rlo.t, th = rhi.t;
    uint32_t b[2][2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = i0 + u0 + 2 * k;
        float cc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) cc[e] = c[k][e] + d[k][e];
        // value of the next M row (row a of an interpolation whose row b is this one)
        const float nx0 = shfl(g8 == 0 ? cc[2] : cc[0], (lane + 4) & 31);
        const float nx1 = shfl(g8 == 0 ? cc[3] : cc[1], (lane + 4) & 31);
        const float nx2 = shfl(cc[2], (lane + 4) & 31);
        const float nx3 = shfl(cc[3], (lane + 4) & 31);
        const bool ul = use_lo && (i + L.q >= rlo.c);
        const bool uh = use_hi && (i + L.q >= rhi.c);
        float sv[4];
        sv[0] = ul ? fmaf(tl, cc[0] - nx0, nx0) : -INFINITY;
        sv[1] = ul ? fmaf(tl, cc[1] - nx1, nx1) : -INFINITY;
        sv[2] = uh ? fmaf(th, cc[2] - nx2, nx2) : -INFINITY;
        sv[3] = uh ? fmaf(th, cc[3] - nx3, nx3) : -INFINITY;
        float p[4];
        softmax_step(U[k], sv, p);
        // p t stays on row b (this row); p (1 - t) moves to row a (the next row)
        const float pt0 = p[0] * tl, pt1 = p[1] * tl, pt2 = p[2] * th, pt3 = p[3] * th;
        const float pa0 = p[0] - pt0, pa1 = p[1] - pt1, pa2 = p[2] - pt2, pa3 = p[3] - pt3;
        const float r0 = shfl(pa0, (lane + 28) & 31);
        const float r1 = shfl(pa1, (lane + 28) & 31);
        const float r2 = shfl(g8 == 7 ? pa0 : pa2, (lane + 28) & 31);
        const float r3 = shfl(g8 == 7 ? pa1 : pa3, (lane + 28) & 31);
        b[k][0] = movm_t(pack_bf16(g8 == 0 ? pt0 : pt0 + r0, g8 == 0 ? pt1 : pt1 + r1));
        b[k][1] = movm_t(pack_bf16(pt2 + r2, pt3 + r3));
    }
    // O^T += V_rows^T . P^T
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vrow[k] ^ (uint32_t)(j << 5), a0, a1, a2, a3);
            mma16816(U[k].o[j], a0, a1, a2, a3, b[k][0], b[k][1]);
        }
    }
}

// Normalise O^T and stage it, transposed, in this warp's output buffer (rows
// (query, head) of the pair, 128-byte swizzle) for the TMA store; the
// log-sum-exp goes straight out.
__device__ __forceinline__ void store_unit(const FwdParams& P, const Tile& x, int u, int k, uint32_t obuf,
                                           const Lane& L, int lane, Unit& U) {
    const int g8 = lane >> 2, tig = lane & 3;
    float l0 = U.l[0], l1 = U.l[1];
#pragma unroll
    for (int w = 4; w <= 16; w <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, w);
        l1 += __shfl_xor_sync(kFull, l1, w);
    }
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const uint32_t buf = obuf + (uint32_t)(k * 8 * ROWB);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
        stsm_x4_t(buf + L.ob[jj], pack_bf16(U.o[2 * jj][0] * inv0, U.o[2 * jj][1] * inv1),
                  pack_bf16(U.o[2 * jj][2] * inv0, U.o[2 * jj][3] * inv1),
                  pack_bf16(U.o[2 * jj + 1][0] * inv0, U.o[2 * jj + 1][1] * inv1),
                  pack_bf16(U.o[2 * jj + 1][2] * inv0, U.o[2 * jj + 1][3] * inv1));
    if (P.lse && g8 == 0) {
        const int iq2 = x.i0 + u + (tig >> 1);
        if (iq2 < P.a.T) {
            const float2 v = make_float2((U.m[0] + __log2f(l0)) * kLn2, (U.m[1] + __log2f(l1)) * kLn2);
            *reinterpret_cast<float2*>(P.lse + ((size_t)x.b * P.a.T + iq2) * kHq + x.g * kG +
                                       2 * (tig & 1)) = v;
        }
    }
}

__device__ void consumer(const FwdParams& P, const Smem& S, int warp, int lane) {
    int wcount = 0, rcount = 0;
    const int u0 = 4 * warp;  // query pairs at tile offsets u0 and u0 + 2
    const Lane L = make_lane(lane, u0, P.a.W, P.win_rows);
    const uint32_t obuf = S.obuf + (uint32_t)(warp * kObufBytes);
    const int nr = max(P.a.nr, 1);
    uint32_t raw[2][4][2];
    Tile x = decode(P, blockIdx.x);
    if (blockIdx.x < P.ntiles) {
#pragma unroll
        for (int k = 0; k < 2; ++k) fetch_q(P, x, u0 + 2 * k, lane, raw[k]);
    }
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x) {
        Unit U[2];
        int kt;
        {
            if (!warp_wait(bar_full_w(S, 0), wcount & 1, S.abort_flag)) goto fail;
            const uint32_t base = S.win;
            const int nq = min(TQ, P.a.T - x.i0);
#pragma unroll
            for (int k = 0; k < 2; ++k) start_unit(P, base + 2 * P.win_region, nq, u0 + 2 * k, lane, raw[k], U[k]);
            for (int wt = 0; wt < P.nwt; ++wt) window_tile(P, base, u0, x.i0, wt, L, U);
            kt = S.kt[0];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty_w(S, 0));
            ++wcount;
        }
        // the next tile's Q is in flight while this tile's rungs are computed
        const Tile nx = decode(P, t + gridDim.x);
        if (t + (int)gridDim.x < P.ntiles) {
#pragma unroll
            for (int k = 0; k < 2; ++k) fetch_q(P, nx, u0 + 2 * k, lane, raw[k]);
        }
        for (int k0 = 0; k0 < kt; k0 += RUNGS_PER_TILE) {
            const int np = min(RUNGS_PER_TILE, kt - k0);
            for (int p = 0; p < np; ++p) {
                const int n = rcount + p;
                if (!warp_wait(bar_full_r(S, n & (NRS - 1)), (n / NRS) & 1, S.abort_flag)) goto fail;
            }
            rung_tiles(S, rcount, np, k0, nr, u0, x.i0, L, U);
            __syncwarp();
            if (lane < np) mbar_arrive(bar_empty_r(S, (rcount + lane) & (NRS - 1)));
            rcount += np;
        }
        // the previous tile's stores must have read this warp's buffer
        if (lane == 0) bulk_wait_read();
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; ++k) store_unit(P, x, u0 + 2 * k, k, obuf, L, lane, U[k]);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < 2; ++k)
                if (x.i0 + u0 + 2 * k < P.a.T)
                    tma_store_4d(&P.omap, obuf + (uint32_t)(k * 8 * ROWB), 0, x.g * kG, x.i0 + u0 + 2 * k, x.b);
            bulk_commit();
        }
        x = nx;
    }
    if (lane == 0) bulk_wait_all();
    return;
fail:
    if (lane == 0) {
        *S.abort_flag = 1;
        if (P.status) atomicOr(P.status, SFA_DEVSTAT_WAIT_TIMEOUT);
        bulk_wait_all();
    }
}

__global__ void __maxnreg__(128) fwd_mma_kernel(const __grid_constant__ FwdParams P) {
    extern __shared__ unsigned char smem_raw[];
    // the dynamic allocation carries 1024 spare bytes to reach 1024 alignment
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    unsigned char* hdr = smem_raw + (base - raw_base);
    Smem S;
    S.bars = base;
    S.abort_flag = reinterpret_cast<int*>(hdr + kFlagOffset);
    S.kt = reinterpret_cast<int*>(hdr + kKtOffset);
    SRung* table = reinterpret_cast<SRung*>(hdr + kRungTableOffset);
    S.r = table;
    S.win = base + kHeaderBytes;
    S.rung = S.win + NWS * P.win_slot_bytes;
    S.obuf = S.rung + NRS * kRungSlotBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    S.tc = base + kTcOffset;
    if (threadIdx.x < P.a.nr) {
        const Rung rg = P.a.r[threadIdx.x];
        table[threadIdx.x] = SRung{rg.n, rg.t, rg.c};
        reinterpret_cast<TC*>(hdr + kTcOffset)[threadIdx.x] = TC{rg.t, rg.c};
    }
    if (threadIdx.x == 0) {
        // full: one arrival (the producer's expect_tx) plus the copied bytes;
        // empty: one arrival per consumer warp
        for (int i = 0; i < NWS; ++i) {
            mbar_init(bar_full_w(S, i), 1);
            mbar_init(bar_empty_w(S, i), NCW);
        }
        for (int i = 0; i < NRS; ++i) {
            mbar_init(bar_full_r(S, i), 1);
            mbar_init(bar_empty_r(S, i), NCW);
        }
        *S.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == NCW) {
        if (lane == 0) producer(P, S);
    } else {
        consumer(P, S, warp, lane);
    }
}

// -------------------------------------------------- RoPE on the keys

// Khat[b][j][g][:] = R(j) K[b][j][g][:] in bf16; one thread per (row, c):
// dimensions 8c..8c+7 and their partners 8c+32..8c+39.
__global__ void __launch_bounds__(256) rope_k_kernel(const __nv_bfloat16* __restrict__ k,
                                                     const float2* __restrict__ rope,
                                                     __nv_bfloat16* __restrict__ khat,
                                                     long long rows, int T) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long row = idx >> 2;
    if (row >= rows) return;
    const int c = (int)(idx & 3);
    const int j = (int)((row / kHkv) % T);
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(k + row * kD + 8 * c));
    const uint4 yv = __ldg(reinterpret_cast<const uint4*>(k + row * kD + kPairs + 8 * c));
    const float4* cs = reinterpret_cast<const float4*>(rope + (size_t)j * kPairs + 8 * c);
    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t ys[4] = {yv.x, yv.y, yv.z, yv.w};
    uint32_t xo[4], yo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float4 t = __ldg(cs + e);  // pairs m = 8c + 2e, 8c + 2e + 1
        const float2 x = unpack_bf16(xs[e]), y = unpack_bf16(ys[e]);
        xo[e] = pack_bf16(x.x * t.x - y.x * t.y, x.y * t.z - y.y * t.w);
        yo[e] = pack_bf16(y.x * t.x + x.x * t.y, y.y * t.z + x.y * t.w);
    }
    *reinterpret_cast<uint4*>(khat + row * kD + 8 * c) = make_uint4(xo[0], xo[1], xo[2], xo[3]);
    *reinterpret_cast<uint4*>(khat + row * kD + kPairs + 8 * c) = make_uint4(yo[0], yo[1], yo[2], yo[3]);
}

// ------------------------------------------------------------- host side

struct DeviceInfo {
    int sms = 0;
    size_t configured_smem = 0;
};

DeviceInfo& device_info(int dev) {
    static DeviceInfo info[64];
    return info[dev & 63];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 4-D map over a [B][T][Hkv][64] bf16 tensor (innermost first: d, g, t, b),
// box of `rows` rows of one head, 128-byte swizzle, zero fill outside.
// 4-D map over O [B][T][8][64] bf16 (innermost first: d, head, t, b), box of
// 2 queries x 4 heads, 128-byte swizzle (the staging buffer's layout).
bool encode_out(CUtensorMap* m, void* base, int B, int T) {
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

bool encode_rows(CUtensorMap* m, const void* base, int B, int T, int rows) {
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

}  // namespace

bool fwd_mma_supported(const LayerArgs& a) { return a.W <= 30; }

size_t fwd_mma_workspace(const LayerArgs& a, bool rope) {
    return rope ? (size_t)a.B * a.T * kHkv * kD * sizeof(__nv_bfloat16) : 0;
}

cudaError_t launch_fwd_mma(const LayerArgs& a, const void* q, const void* k, const void* v,
                           const float2* rope, void* o, float* lse, void* ws, unsigned* status,
                           cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    DeviceInfo& info = device_info(dev);
    if (info.sms == 0) {
        e = cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    FwdParams P;
    std::memset(&P, 0, sizeof(P));
    P.a = a;
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.o = static_cast<__nv_bfloat16*>(o);
    P.lse = lse;
    P.status = status;
    P.rope = rope;
    P.ntq = (a.T + TQ - 1) / TQ;
    P.ntiles = a.B * P.ntq * kHkv;
    P.win_rows = TQ + a.W;
    P.nwt = (a.W + 4 + 15) / 16;
    P.win_region = round1k((unsigned)P.win_rows * ROWB);
    P.win_slot_bytes = 2 * P.win_region + round1k(TQ * TABB);
    const void* khat = k;
    if (rope) {
        const long long rows = (long long)a.B * a.T * kHkv;
        const long long threads = rows * 4;
        rope_k_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(k), rope, static_cast<__nv_bfloat16*>(ws), rows, a.T);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
        khat = ws;
    }
    if (!encode_rows(&P.kmap_w, khat, a.B, a.T, P.win_rows) ||
        !encode_rows(&P.vmap_w, v, a.B, a.T, P.win_rows))
        return cudaErrorInvalidValue;
    if (!encode_out(&P.omap, o, a.B, a.T)) return cudaErrorInvalidValue;
    for (int p = 0; p < RUNGS_PER_TILE; ++p) {
        const int rows = RUNG_ROWS + ((3 * p) & 7);
        if (!encode_rows(&P.kmap_r[p], khat, a.B, a.T, rows) || !encode_rows(&P.vmap_r[p], v, a.B, a.T, rows))
            return cudaErrorInvalidValue;
    }
    const size_t smem = 1024 + kHeaderBytes + NWS * (size_t)P.win_slot_bytes + NRS * (size_t)kRungSlotBytes +
                        NCW * (size_t)kObufBytes;
    if (info.configured_smem < smem) {
        e = cudaFuncSetAttribute(fwd_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(fwd_mma_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        info.configured_smem = smem;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fwd_mma_kernel, NTHREADS, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    long long grid = (long long)info.sms * per_sm;
    if (grid > P.ntiles) grid = P.ntiles;
    fwd_mma_kernel<<<(unsigned)grid, NTHREADS, smem, s>>>(P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    count_launch();
    return cudaSuccess;
}

}  // namespace sfa
