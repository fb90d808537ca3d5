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
//     caller's workspace, with the 64 dimensions of a row stored in the order
//     the score MMA consumes them (see kdim_of below), so that every thread
//     of the main kernel loads its query fragment with two 16-byte loads.
//  2. fwd_mma_kernel, persistent, (1 producer + 7 consumer) warps per CTA.
//     A CTA owns a tile of TQ = 28 consecutive queries of one sequence b and
//     one key/value head g (4 query heads).  The producer (one lane) loads,
//     with tiled TMA boxes, the window block (rows i0 - W .. i0 + TQ - 1) and,
//     per group of four rungs, the four blocks of rows i0 - n_k - 1 ..
//     i0 + TQ - 1 - n_k of Khat and V into an mbarrier ring of shared-memory
//     slots (rows outside the sequence arrive as zeros), plus the RoPE rows of
//     the tile's queries.
//     Each consumer warp owns two query pairs.  For a pair (i, i + 1) the
//     scores are formed "keys on M": S^T = Khat_rows (16 x 64) . Qhat^T
//     (64 x 8), N = 2 queries x 4 heads.
//     Window: the 16 rows i - W .. i + 3 of a query quad form one M tile.
//     Rungs: one M tile holds four rungs; its row r < 8 is row b = i + e - n - 1
//     and row r + 8 is row a = i + e - n of rung r mod 4 for query e = r / 4
//     of the pair.  A thread's two accumulator rows are therefore the two rows
//     of one interpolation, so the lerp on the scores, s = (1 - t) s_a + t s_b
//     (the score of the interpolated key, by linearity), and the split of the
//     probability back onto the rows, p (1 - t) and p t (so that P^T V_rows
//     forms the interpolated value), stay inside the thread.
//     One online softmax (base 2, lazy rescale: the running max is raised
//     only when a score exceeds it by more than 2^8) runs over window and
//     rung entries; O^T accumulates in registers and is transposed with
//     stmatrix into a staging buffer that the warp writes out with
//     coalesced 16-byte stores.
//     In a multi-layer call each consumer warp also rotates, tile by tile,
//     the next layer's keys at its four positions (the window slot already
//     holds their RoPE rows), so that no later layer needs launch 1.
//
// Shared memory: each tensor region of a slot is 1024-byte aligned and filled
// by TMA with the 128-byte swizzle (16-byte chunk c of region row r stored at
// chunk c ^ (r & 7)).  The box of rung position p of a group starts 2p rows
// early, so the eight rows that one ldmatrix phase reads from the four rungs
// fall in eight different swizzle phases (no bank conflicts).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "sfa_internal.cuh"
#include "sfa_mma.cuh"
#include "sfa_ring.cuh"

namespace sfa {

namespace {

using namespace mma;
using namespace ring;

constexpr float kLazy = 8.0f;          // raise the running max past this margin
constexpr float kMinMax = -1e30f;      // floor of the running max (no entry yet)
constexpr int NCW = 7;                     // consumer warps (two query pairs each)
constexpr int NTHREADS = (NCW + 1) * 32;   // + the producer warp
constexpr unsigned kObufBytes = 8 * ROWB;  // per consumer warp: O of one query pair (2 queries x 4 heads)

struct FwdParams {
    static constexpr int kQMaps = 1;  // the query slot carries the tile's Q
    static constexpr bool kWinRope = true;  // the window slot carries the tile's RoPE rows
    CUtensorMap qmaps[kQMaps];        // Q [B][T][8][64], box of TQ queries x 4 heads
    CUtensorMap kmap_w;        // Khat, box of win_rows rows
    CUtensorMap vmap_w;        // V, box of win_rows rows
    CUtensorMap kmap_r[RPG];   // Khat, box of RUNG_ROWS + 2p rows, rung position p
    CUtensorMap vmap_r[RPG];   // V, same boxes
    CUtensorMap tabmap;        // RoPE table rows of a tile (with RoPE)
    LayerArgs a;
    const __nv_bfloat16* q;
    const float2* rope;        // nullptr: Q and K are used as given
    __nv_bfloat16* o;
    float* lse;
    unsigned* status;
    const __nv_bfloat16* k_next;  // keys of the next layer (multi-layer forward) or nullptr
    __nv_bfloat16* khat_next;     // where their rotated copy goes
    float sl2;                 // softmax scale x log2(e)
    float inv_sl2;
    int ntq;                   // query tiles per sequence
    int ntiles;                // B * ntq * Hkv
    int step_g, step_tq, step_b;  // gridDim.x as (sequences, query tiles, heads)
    int win_rows;              // TQ + W
    int nwt;                   // window M tiles of a query quad (W + 4 rows)
    unsigned win_region;       // bytes of one tensor region of the window slot
    unsigned win_slot_bytes;   // Khat + V regions and the tile's RoPE rows
};

// ------------------------------------------------------- dimension order
//
// The score MMA of k-step s takes, in thread (row group, tig), the key and
// query dimensions at positions 16 s + 8 h + 2 tig + j (h, j in {0, 1}) of the
// row as stored.  Khat rows are stored permuted so that position 8 c + 2 tig
// + j (16-byte chunk c) holds dimension kdim_of(c, tig, j): a thread then
// needs the query dimensions 8 tig .. 8 tig + 7 and their RoPE partners
// 32 + 8 tig .. 32 + 8 tig + 7, two contiguous 16-byte pieces, and the two
// members of each rotation pair sit in the same thread.
__host__ __device__ constexpr int kdim_of(int c, int tig, int j) {
    return c < 4 ? 8 * tig + 2 * c + j : 32 + 8 * tig + 2 * (c - 4) + j;
}

// ------------------------------------------------------------ consumers

// One query pair (i, i + 1) of one key/value head: the B fragments of
// Qhat^T, the O^T accumulators and softmax state of this thread's two
// columns (query tig/2, heads 2(tig&1) and 2(tig&1)+1).  Scores stay in the
// units of q.k; m is the running max in log2 units (score x scale x log2 e),
// th the raw score above which m must be raised.  Column pairs use the
// packed two-lane fp32 instructions.
struct Unit {
    uint32_t qf[4][2];
    float o[4][4];
    float2 nm;    // minus the running max, log2 units
    float th[2];
    float2 l;
};


// Per-thread constants of the fragment layouts (fixed for the whole kernel:
// the warp always owns the query pairs at tile offsets u0 and u0 + 2).
// Addresses are byte offsets inside a slot, with the 128-byte swizzle of
// ldmatrix k-step (or m tile) 0 folded in: step s reads at offset ^ (s << 5).
struct Lane {
    int g8, q;          // fragment row group; query of this thread's C columns
    bool useful;        // this thread's rung rows belong to its column query
    unsigned wmask;     // window: bit (8 wt + 4 k + e) = row is a window distance of
                        // quad query 2k + q (before the sequence-start check)
    uint32_t kr[2];     // rung tile of unit k: Khat row offset in a group slot
    uint32_t vr[2];     // rung tile of unit k: V row offset in a group slot
    uint32_t ki, vi;    // integer-offset rung tile (rows a of the quad): Khat / V row offsets
    uint32_t wk, wv;    // window tile 0: Khat and V row offsets
    uint32_t ob[2];     // output staging: stmatrix row address offsets (jj = 0, 1)
};

__device__ __forceinline__ Lane make_lane(int lane, int u0, int W, int win_rows) {
    Lane L;
    L.g8 = lane >> 2;
    L.q = (lane & 3) >> 1;
    L.useful = (L.g8 >> 2) == L.q;
    // ldmatrix row of this lane: K (x4): row (lane & 7) + 8 ((lane >> 3) & 1),
    // k half lane >> 4; V (x4.trans): row (lane & 7) + 8 (lane >> 4), half
    // (lane >> 3) & 1.  M row r is rung r & 3, query (r >> 2) & 1, kind r >> 3.
    const int p = lane & 3, e = (lane >> 2) & 1;
    for (int k = 0; k < 2; ++k) {
        const int u = u0 + 2 * k;
        L.kr[k] = rung_row(p, u, e, (lane >> 3) & 1, lane >> 4, false);
        L.vr[k] = rung_row(p, u, e, lane >> 4, (lane >> 3) & 1, true);
    }
    const int rk = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int rv = (lane & 7) + ((lane >> 4) << 3);
    // integer offsets: M row r is rung r & 3, query e = r >> 2 of the quad, row a
    L.ki = rung_row(rk & 3, u0, rk >> 2, 1, lane >> 4, false);
    L.vi = rung_row(rv & 3, u0, rv >> 2, 1, (lane >> 3) & 1, true);
    L.wk = swz_row(min(u0 + rk, win_rows - 1), lane >> 4);
    L.wv = swz_row(min(u0 + rv, win_rows - 1), (lane >> 3) & 1);
    L.wmask = 0u;
    for (int wt = 0; wt < 3; ++wt)
        for (int k = 0; k < 2; ++k)
            for (int e2 = 0; e2 < 4; ++e2) {
                const int R = 16 * wt + L.g8 + ((e2 >> 1) << 3);
                const int qq = 2 * k + L.q;
                if (R >= qq && R <= W + qq) L.wmask |= 1u << (8 * wt + 4 * k + e2);
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

// Q of this thread's B-fragment column (query u + g8/4, head g8 % 4 = row
// r = 4u + g8 of the Q tile in the query slot, 128-byte swizzle: 16-byte
// chunk c at c ^ (r & 7), and r & 7 = g8) rotated by the RoPE rows of the
// tile (nq of them) into B fragments.  With RoPE the thread reads dimensions
// 8 tig .. 8 tig + 7 (chunk tig) and their partners + 32 (chunk 4 + tig);
// without, the positions of the stored order directly (word w of fragment
// half h' = chunk 4 h' + w, word tig).  The first window tile starts the O^T
// accumulators.
__device__ __forceinline__ void start_unit(const FwdParams& P, const Smem& S, int nq, int u, int lane, Unit& U) {
    const int g8 = lane >> 2, tig = lane & 3;
    const uint32_t slot = S.win;
    const uint32_t qrow = S.qslot + (uint32_t)((4 * u + g8) * ROWB);
    if (P.rope) {
        const uint4 x4 = lds_u4(qrow + (uint32_t)((tig ^ g8) << 4));
        const uint4 y4 = lds_u4(qrow + (uint32_t)(((4 + tig) ^ g8) << 4));
        // table chunks 4 tig + w of the row: w flips the low bits of the
        // swizzled chunk only
        const uint32_t trow = slot + 2 * P.win_region + tab_chunk(min(u + (g8 >> 2), nq - 1), 4 * tig);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            // pairs m = 8 tig + 2 w + {0, 1}: (cos, sin) of both
            const float4 cs = lds_f4(trow ^ (uint32_t)(w << 4));
            const float2 xv = unpack_bf16(u4_get(x4, w));
            const float2 yv = unpack_bf16(u4_get(y4, w));
            U.qf[w >> 1][w & 1] = rope_x(xv, yv, cs);
            U.qf[2 + (w >> 1)][w & 1] = rope_y(xv, yv, cs);
        }
    } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            U.qf[w >> 1][w & 1] = lds_u32(qrow + (uint32_t)(((w ^ g8) << 4) + 4 * tig));
            U.qf[2 + (w >> 1)][w & 1] = lds_u32(qrow + (uint32_t)((((4 + w) ^ g8) << 4) + 4 * tig));
        }
    }
}

// Column max of this thread's two columns over the 8 threads holding them.
__device__ __forceinline__ void col_max(float& mx0, float& mx1) {
#pragma unroll
    for (int w = 4; w <= 16; w <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, w));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, w));
    }
}

// Softmax of the first window entries of a row: the running max becomes the
// column max (floored: a column without entries keeps p = 0).
__device__ __forceinline__ void softmax_first(const FwdParams& P, Unit& U, const float s[4], float p[4]) {
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
    col_max(mx0, mx1);
    const float m0 = fmaxf(mx0 * P.sl2, kMinMax), m1 = fmaxf(mx1 * P.sl2, kMinMax);
    U.nm = f2(-m0, -m1);
    U.th[0] = (m0 + kLazy) * P.inv_sl2;
    U.th[1] = (m1 + kLazy) * P.inv_sl2;
    const float2 sl = f2(P.sl2, P.sl2);
    const float2 x01 = __ffma2_rn(f2(s[0], s[1]), sl, U.nm);
    const float2 x23 = __ffma2_rn(f2(s[2], s[3]), sl, U.nm);
    p[0] = fast_exp2(x01.x);
    p[1] = fast_exp2(x01.y);
    p[2] = fast_exp2(x23.x);
    p[3] = fast_exp2(x23.y);
    U.l = __fadd2_rn(f2(p[0], p[1]), f2(p[2], p[3]));
}

// Raise the running max of this thread's two columns to include the column
// maxima mx0, mx1 (raw, before the reduction) and rescale O^T and l.
__device__ __forceinline__ void raise_max(const FwdParams& P, Unit& U, float mx0, float mx1) {
    col_max(mx0, mx1);
    const float n0 = fmaxf(-U.nm.x, mx0 * P.sl2), n1 = fmaxf(-U.nm.y, mx1 * P.sl2);
    const float2 c = f2(fast_exp2(-U.nm.x - n0), fast_exp2(-U.nm.y - n1));
    U.nm = f2(-n0, -n1);
    U.th[0] = (n0 + kLazy) * P.inv_sl2;
    U.th[1] = (n1 + kLazy) * P.inv_sl2;
    U.l = __fmul2_rn(U.l, c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 a = __fmul2_rn(f2(U.o[j][0], U.o[j][1]), c);
        const float2 b = __fmul2_rn(f2(U.o[j][2], U.o[j][3]), c);
        U.o[j][0] = a.x;
        U.o[j][1] = a.y;
        U.o[j][2] = b.x;
        U.o[j][3] = b.y;
    }
}

// Online-softmax step over four entries (two rows x two columns).
__device__ __forceinline__ void softmax_step4(const FwdParams& P, Unit& U, const float s[4], float p[4]) {
    const bool need = (s[0] > U.th[0]) || (s[2] > U.th[0]) || (s[1] > U.th[1]) || (s[3] > U.th[1]);
    if (__any_sync(kFull, need)) raise_max(P, U, fmaxf(s[0], s[2]), fmaxf(s[1], s[3]));
    const float2 sl = f2(P.sl2, P.sl2);
    const float2 x01 = __ffma2_rn(f2(s[0], s[1]), sl, U.nm);
    const float2 x23 = __ffma2_rn(f2(s[2], s[3]), sl, U.nm);
    p[0] = fast_exp2(x01.x);
    p[1] = fast_exp2(x01.y);
    p[2] = fast_exp2(x23.x);
    p[3] = fast_exp2(x23.y);
    U.l = __fadd2_rn(U.l, __fadd2_rn(f2(p[0], p[1]), f2(p[2], p[3])));
}

// Online-softmax step over one entry per column.
__device__ __forceinline__ float2 softmax_step2(const FwdParams& P, Unit& U, float2 sv) {
    if (__any_sync(kFull, (sv.x > U.th[0]) || (sv.y > U.th[1]))) raise_max(P, U, sv.x, sv.y);
    const float2 x = __ffma2_rn(sv, f2(P.sl2, P.sl2), U.nm);
    const float2 p = f2(fast_exp2(x.x), fast_exp2(x.y));
    U.l = __fadd2_rn(U.l, p);
    return p;
}

// Window M tile wt of the warp's query quad at tile offset u0 (positions
// i0 + u0 .. + 3): region rows u0 + R, R = 16 wt .. 16 wt + 15, hold
// positions i0 + u0 - W + R; unit k holds queries 2k, 2k + 1 of the quad.
template <bool kFirst>
__device__ __forceinline__ void window_tile(const FwdParams& P, uint32_t slot, int u0, int i0, int wt,
                                            const Lane& L, Unit* U) {
    const int lane = threadIdx.x & 31;
    uint32_t kro = L.wk, vro = L.wv;
    if (!kFirst) {
        const int maxr = P.win_rows - 1;
        kro = swz_row(min(u0 + 16 * wt + (lane & 7) + (((lane >> 3) & 1) << 3), maxr), lane >> 4);
        vro = swz_row(min(u0 + 16 * wt + (lane & 7) + ((lane >> 4) << 3), maxr), (lane >> 3) & 1);
    }
    float c[2][4];
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(slot + (kro ^ (uint32_t)(s2 << 5)), a0, a1, a2, a3);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (s2 == 0)
                mma16816_z(c[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
            else
                mma16816(c[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
        }
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
        if (kFirst)
            softmax_first(P, U[k], sv, p);
        else
            softmax_step4(P, U[k], sv, p);
        b[k][0] = movm_t(pack_bf16(p[0], p[1]));
        b[k][1] = movm_t(pack_bf16(p[2], p[3]));
    }
    const uint32_t vbase = slot + P.win_region;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vbase + (vro ^ (uint32_t)(j << 5)), a0, a1, a2, a3);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (kFirst)
                mma16816_z(U[k].o[j], a0, a1, a2, a3, b[k][0], b[k][1]);
            else
                mma16816(U[k].o[j], a0, a1, a2, a3, b[k][0], b[k][1]);
        }
    }
}

// Rung M tile of the warp's two query pairs (tile offsets u0 and u0 + 2,
// positions i = i0 + u0 ..) for the np rungs k0 .. k0 + np - 1 of the group in
// slot `gslot`.  Rows of absent rung positions (np < 4) read rung 0's block;
// their entries are masked.
__device__ __forceinline__ void rung_tile(const FwdParams& P, const Smem& S, uint32_t gslot, int k0, int np,
                                          int nr, int u0, int i, const Lane& L, Unit* U) {
    const int lane = threadIdx.x & 31;
    uint32_t krow[2], vrow[2];
    if (np == RPG) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            krow[k] = gslot + L.kr[k];
            vrow[k] = gslot + L.vr[k];
        }
    } else {
        const int p = (lane & 3) < np ? (lane & 3) : 0, e = (lane >> 2) & 1;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            krow[k] = gslot + rung_row(p, u0 + 2 * k, e, (lane >> 3) & 1, lane >> 4, false);
            vrow[k] = gslot + rung_row(p, u0 + 2 * k, e, lane >> 4, (lane >> 3) & 1, true);
        }
    }
    // S^T = Khat_rows . Qhat^T
    float c[2][4];
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(krow[k] ^ (uint32_t)(s2 << 5), a0, a1, a2, a3);
            if (s2 == 0)
                mma16816_z(c[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
            else
                mma16816(c[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
        }
    }
    // this thread's rows: row b (c0, c1) and row a (c2, c3) of rung k0 + p
    // for query q of the pair; a rung is used from i - ceil(d) >= 0 on
    const int p = L.g8 & 3;
    const TC tc = lds_tc(S.tc + (uint32_t)(min(k0 + p, nr - 1) * 8));
    const int ceil_d = (L.useful && p < np) ? tc.c : kNoRung;
    const float2 t = f2(tc.t, tc.t), omt = f2(1.f - tc.t, 1.f - tc.t);
    uint32_t b[2][2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool ok = i + 2 * k + L.q >= ceil_d;
        // (1 - t) s_a + t s_b
        float2 sv = __ffma2_rn(t, f2(c[k][0], c[k][1]), __fmul2_rn(omt, f2(c[k][2], c[k][3])));
        sv.x = ok ? sv.x : -INFINITY;
        sv.y = ok ? sv.y : -INFINITY;
        const float2 p = softmax_step2(P, U[k], sv);
        // p t on row b, p (1 - t) on row a
        const float2 pb = __fmul2_rn(p, t), pa = __fmul2_rn(p, omt);
        b[k][0] = movm_t(pack_bf16(pb.x, pb.y));
        b[k][1] = movm_t(pack_bf16(pa.x, pa.y));
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

// The rung M tile when every kept rung has an integer distance (t = 0, so
// only row a = i - n of a rung is read): row r of the tile is row a of rung
// k0 + (r & 3) for query e = r >> 2 of the quad, and one tile serves both
// pairs -- pair 0 (queries 0, 1) reads rows 0..7, pair 1 rows 8..15, so a
// thread's useful scores are c0, c1 of pair 0 and c2, c3 of pair 1, and the
// value products run as m16n8k8 on the matching half of the rows.
__device__ __forceinline__ void rung_tile_int(const FwdParams& P, const Smem& S, uint32_t gslot, int k0, int np,
                                              int nr, int u0, int i, const Lane& L, Unit* U) {
    const int lane = threadIdx.x & 31;
    uint32_t krow = gslot + L.ki, vrow = gslot + L.vi;
    if (np < RPG) {
        // rows of absent rung positions read rung 0's block; their entries are masked
        const int rk = (lane & 7) + (((lane >> 3) & 1) << 3), rv = (lane & 7) + ((lane >> 4) << 3);
        const int pk = (rk & 3) < np ? (rk & 3) : 0, pv = (rv & 3) < np ? (rv & 3) : 0;
        krow = gslot + rung_row(pk, u0, rk >> 2, 1, lane >> 4, false);
        vrow = gslot + rung_row(pv, u0, rv >> 2, 1, (lane >> 3) & 1, true);
    }
    // S^T = Khat_rows . Qhat^T for both pairs, one A fragment
    float c[2][4];
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(krow ^ (uint32_t)(s2 << 5), a0, a1, a2, a3);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (s2 == 0)
                mma16816_z(c[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
            else
                mma16816(c[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
        }
    }
    const int p = L.g8 & 3;
    const TC tc = lds_tc(S.tc + (uint32_t)(min(k0 + p, nr - 1) * 8));
    const int ceil_d = (L.useful && p < np) ? tc.c : kNoRung;
    uint32_t b[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool ok = i + 2 * k + L.q >= ceil_d;
        float2 sv = k == 0 ? f2(c[0][0], c[0][1]) : f2(c[1][2], c[1][3]);
        sv.x = ok ? sv.x : -INFINITY;
        sv.y = ok ? sv.y : -INFINITY;
        const float2 pe = softmax_step2(P, U[k], sv);
        b[k] = movm_t(pack_bf16(pe.x, pe.y));
    }
    // O^T += V_rows^T . P^T: pair 0 on rows 0..7, pair 1 on rows 8..15
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vrow ^ (uint32_t)(j << 5), a0, a1, a2, a3);
        mma1688(U[0].o[j], a0, a1, b[0]);
        mma1688(U[1].o[j], a2, a3, b[1]);
    }
}

// Normalise O^T of the pair at tile offset u and stage it, transposed, in
// this warp's output buffer (rows (query, head), 16-byte chunk c of row r at
// c ^ r); the warp then reads it back so that each 16-byte store covers one
// query's four heads, 512 contiguous bytes of O.  The log-sum-exp goes
// straight out.
__device__ __forceinline__ void store_unit(const FwdParams& P, const Tile& x, int u, uint32_t obuf, const Lane& L,
                                           int lane, Unit& U) {
    const int g8 = lane >> 2, tig = lane & 3;
    float2 l = U.l;
#pragma unroll
    for (int w = 4; w <= 16; w <<= 1)
        l = __fadd2_rn(l, f2(__shfl_xor_sync(kFull, l.x, w), __shfl_xor_sync(kFull, l.y, w)));
    // l >= 1: the entry at the running max contributes exactly 1
    const float2 inv = f2(fast_rcp(l.x), fast_rcp(l.y));
    uint32_t r[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 a = __fmul2_rn(f2(U.o[j][0], U.o[j][1]), inv);
        const float2 b = __fmul2_rn(f2(U.o[j][2], U.o[j][3]), inv);
        r[j][0] = pack_bf16(a.x, a.y);
        r[j][1] = pack_bf16(b.x, b.y);
    }
    __syncwarp();  // the previous pair's rows have been read back
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
        stsm_x4_t(obuf + L.ob[jj], r[2 * jj][0], r[2 * jj][1], r[2 * jj + 1][0], r[2 * jj + 1][1]);
    __syncwarp();
    {
        const int cc = lane & 7;
        uint4* dst = reinterpret_cast<uint4*>(P.o + (((size_t)x.b * P.a.T + x.i0 + u) * kHq + x.g * kG) * kD);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int rr = 4 * e + (lane >> 3);  // row (query e, head lane / 8)
            if (x.i0 + u + e < P.a.T)
                dst[(size_t)e * (kHq * kD / 8) + (lane >> 3) * (kD / 8) + cc] =
                    lds_u4(obuf + (uint32_t)rr * ROWB + (uint32_t)(((cc ^ rr) & 7) << 4));
        }
    }
    if (P.lse) {
        // lanes g8 = 0 hold the sums of query u + tig / 2, heads 2 (tig & 1) + {0, 1}
        const int iq2 = x.i0 + u + (tig >> 1);
        const float2 v = make_float2((__log2f(l.x) - U.nm.x) * kLn2, (__log2f(l.y) - U.nm.y) * kLn2);
        float* dst = P.lse + ((size_t)x.b * P.a.T + iq2) * kHq + x.g * kG + 2 * (tig & 1);
        if (g8 == 0 && iq2 < P.a.T) *reinterpret_cast<float2*>(dst) = v;
    }
}

// The next layer's RoPE pass (multi-layer forward), done inside the main
// loop: the consumer warp that owns tile offsets u0 .. u0 + 3 rotates rows
// i0 + u0 .. i0 + u0 + 3 of K_next (the tile's kv head) into Khat_next, in the
// kdim_of order, with the RoPE rows of those positions that the window slot
// already holds.  Tiles cover every (sequence, position, kv head) once, so
// every row is written once.  Lane = (row r, stored chunk c, half h): it
// rotates the pairs m = 8 tig + 2c + {0, 1}, tig = 2h, 2h + 1 -- words
// 4 tig + c (x) and 16 + 4 tig + c (y) of the input row -- and writes words
// tig = 2h, 2h + 1 of stored chunks c (x) and 4 + c (y).
struct NextRows {
    uint32_t xw[2], yw[2];
    bool ok;
};

__device__ __forceinline__ size_t next_row(const FwdParams& P, const Tile& x, int pos) {
    return ((size_t)x.b * P.a.T + pos) * kHkv + x.g;
}

__device__ __forceinline__ void load_next_rows(const FwdParams& P, const Tile& x, int u0, int lane, NextRows& N) {
    const int r = lane >> 3, c = (lane >> 1) & 3, h = lane & 1;
    const int pos = x.i0 + u0 + r;
    N.ok = pos < P.a.T;
    const unsigned* kw = reinterpret_cast<const unsigned*>(P.k_next + next_row(P, x, N.ok ? pos : x.i0) * kD);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        N.xw[j] = __ldg(kw + 4 * (2 * h + j) + c);
        N.yw[j] = __ldg(kw + 16 + 4 * (2 * h + j) + c);
    }
}

__device__ __forceinline__ void store_next_rows(const FwdParams& P, const Smem& S, const Tile& x, int u0, int lane,
                                                const NextRows& N) {
    const int r = lane >> 3, c = (lane >> 1) & 3, h = lane & 1;
    // table chunks 8 h + 4 j + c of row u0 + r: j flips bit 2 of the swizzled chunk
    const uint32_t trow = S.win + 2 * P.win_region + tab_chunk(u0 + r, 8 * h + c);
    uint32_t xo[2], yo[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float4 cs = lds_f4(trow ^ (uint32_t)(j << 6));
        const float2 xv = unpack_bf16(N.xw[j]), yv = unpack_bf16(N.yw[j]);
        xo[j] = rope_x(xv, yv, cs);
        yo[j] = rope_y(xv, yv, cs);
    }
    if (N.ok) {
        unsigned char* out = reinterpret_cast<unsigned char*>(P.khat_next + next_row(P, x, x.i0 + u0 + r) * kD);
        *reinterpret_cast<uint2*>(out + 16 * c + 8 * h) = make_uint2(xo[0], xo[1]);
        *reinterpret_cast<uint2*>(out + 64 + 16 * c + 8 * h) = make_uint2(yo[0], yo[1]);
    }
}

template <bool kInt>
__device__ void consumer(const FwdParams& P, const Smem& S, int warp, int lane) {
    int wcount = 0, gcount = 0, qcount = 0;
    const int u0 = 4 * warp;  // query pairs at tile offsets u0 and u0 + 2
    const Lane L = make_lane(lane, u0, P.a.W, P.win_rows);
    const uint32_t obuf = S.obuf + (uint32_t)(warp * kObufBytes);
    const int nr = max(P.a.nr, 1);
    // Khat_next was read by the launch before this one
    if (P.k_next) asm volatile("griddepcontrol.wait;" ::: "memory");
    Tile x = decode(P, blockIdx.x);
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x) {
        Unit U[2];
        int kt;
        {
            if (!warp_wait(bar_full_q(S), qcount & 1, S.abort_flag)) goto fail;
            if (!warp_wait(bar_full_w(S), wcount & 1, S.abort_flag)) goto fail;
            const int nq = min(TQ, P.a.T - x.i0);
#pragma unroll
            for (int k = 0; k < 2; ++k) start_unit(P, S, nq, u0 + 2 * k, lane, U[k]);
            __syncwarp();
            mbar_arrive_if(bar_empty_q(S), lane == 0);
            ++qcount;
            NextRows N;
            if (P.k_next) load_next_rows(P, x, u0, lane, N);
            window_tile<true>(P, S.win, u0, x.i0, 0, L, U);
            for (int wt = 1; wt < P.nwt; ++wt) window_tile<false>(P, S.win, u0, x.i0, wt, L, U);
            if (P.k_next) store_next_rows(P, S, x, u0, lane, N);
            kt = *S.kt;
            __syncwarp();
            mbar_arrive_if(bar_empty_w(S), lane == 0);
            ++wcount;
        }
        for (int k0 = 0; k0 < kt; k0 += RPG) {
            const int slot = gcount & (NGS - 1);
            if (!warp_wait(bar_full_g(S, slot), (gcount / NGS) & 1, S.abort_flag)) goto fail;
            if (kInt)
                rung_tile_int(P, S, S.rung + (uint32_t)slot * kGroupSlotBytes, k0, min(RPG, kt - k0), nr, u0,
                              x.i0 + u0, L, U);
            else
                rung_tile(P, S, S.rung + (uint32_t)slot * kGroupSlotBytes, k0, min(RPG, kt - k0), nr, u0,
                          x.i0 + u0, L, U);
            __syncwarp();
            mbar_arrive_if(bar_empty_g(S, slot), lane == 0);
            ++gcount;
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) store_unit(P, x, u0 + 2 * k, obuf, L, lane, U[k]);
        x = next_tile(P, x);
    }
    return;
fail:
    if (lane == 0) {
        *S.abort_flag = 1;
        if (P.status) atomicOr(P.status, SFA_DEVSTAT_WAIT_TIMEOUT);
    }
}

// kInt: every kept rung has an integer distance (the interpolation weight of
// row b is zero everywhere), so the rung tiles read rows a only.
template <bool kInt>
__global__ void __maxnreg__(128) fwd_mma_kernel(const __grid_constant__ FwdParams P) {
    extern __shared__ unsigned char smem_raw[];
    const Smem S = ring_setup(P.a, NCW, FwdParams::kQMaps * kQTileBytes, P.win_slot_bytes, smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the next launch (the next layer) may start its prologue; it waits for
    // this grid before it touches memory
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == NCW) {
        if (lane == 0) producer(P, S);
    } else {
        consumer<kInt>(P, S, warp, lane);
    }
}

// -------------------------------------------------- RoPE on the keys

// Khat[b][j][g][:] = R(j) K[b][j][g][:] in bf16, in the stored dimension
// order of kdim_of.  Four threads per row: thread a rotates the pairs
// m = 8a .. 8a + 7 (dimensions 8a .. 8a + 7 and their partners + 32, two
// 16-byte loads), which land in word a of every stored chunk; the four
// threads exchange words through shared memory so that thread a writes whole
// chunks a and 4 + a (two 16-byte stores).
constexpr int kRopeThreads = 256;
constexpr int kRopePitch = ROWB + 16;  // bytes per staged row: 4-byte stores of a phase hit distinct banks

__global__ void __launch_bounds__(kRopeThreads) rope_k_kernel(const __nv_bfloat16* __restrict__ k,
                                                              const float2* __restrict__ rope,
                                                              __nv_bfloat16* __restrict__ khat,
                                                              unsigned rows, unsigned T) {
    // the forward kernel may start its prologue now; it waits for this grid
    // to finish before it reads Khat
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ __align__(16) unsigned char stage[kRopeThreads / 4 * kRopePitch];
    const unsigned lrow = threadIdx.x >> 2, a = threadIdx.x & 3;
    const unsigned row = blockIdx.x * (kRopeThreads / 4) + lrow;
    const bool live = row < rows;
    unsigned char* srow = stage + lrow * kRopePitch;
    if (live) {
        const unsigned j = (row / kHkv) % T;
        const __nv_bfloat16* kr = k + (size_t)row * kD;
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(kr + 8 * a));
        const uint4 yv = __ldg(reinterpret_cast<const uint4*>(kr + 32 + 8 * a));
        const float4* cs = reinterpret_cast<const float4*>(rope + (size_t)j * kPairs + 8 * a);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            // pairs m = 8a + 2c + {0, 1}: stored at chunk c (x) and 4 + c (y), word a
            const float4 t = __ldg(cs + c);
            const float2 x = unpack_bf16(u4_get(xv, c));
            const float2 y = unpack_bf16(u4_get(yv, c));
            const uint32_t xo = rope_x(x, y, t);
            const uint32_t yo = rope_y(x, y, t);
            *reinterpret_cast<uint32_t*>(srow + 16 * c + 4 * a) = xo;
            *reinterpret_cast<uint32_t*>(srow + 64 + 16 * c + 4 * a) = yo;
        }
    }
    __syncwarp();
    if (live) {
        __nv_bfloat16* out = khat + (size_t)row * kD;
        *reinterpret_cast<uint4*>(out + 8 * a) = *reinterpret_cast<const uint4*>(srow + 16 * a);
        *reinterpret_cast<uint4*>(out + 32 + 8 * a) = *reinterpret_cast<const uint4*>(srow + 64 + 16 * a);
    }
}

static_assert(kdim_of(1, 2, 1) == 8 * 2 + 2 * 1 + 1 && kdim_of(5, 3, 0) == 32 + 24 + 2, "dimension order");

// ------------------------------------------------------------- host side

}  // namespace

bool fwd_mma_supported(const LayerArgs& a) { return a.W <= 30; }

size_t fwd_mma_workspace(const LayerArgs& a, bool rope) {
    return rope ? (size_t)a.B * a.T * kHkv * kD * sizeof(__nv_bfloat16) : 0;
}

// The attention launch of one layer: khat holds the rotated keys (or the raw
// keys without RoPE); with k_next set its consumer warps also rotate the next
// layer's keys into khat_next, tile by tile.  `pdl`: the launch directly
// follows a RoPE pass or an attention launch of this library and may overlap
// its prologue (programmatic dependent launch).
cudaError_t launch_fwd_attention(const LayerArgs& a, const void* q, const void* khat, const void* v,
                                 const float2* rope, void* o, float* lse, const void* k_next, void* khat_next,
                                 unsigned* status, bool pdl, cudaStream_t s) {
    if (fwd_tc_supported(a)) return launch_fwd_tc(a, q, khat, v, rope, o, lse, k_next, khat_next, status, pdl, s);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = sm_count(dev, &e);
    if (e != cudaSuccess) return e;
    static CtxSetting configured_smem[2][64];  // per variant and device: dynamic shared memory already allowed
    FwdParams P;
    std::memset(&P, 0, sizeof(P));
    P.a = a;
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.o = static_cast<__nv_bfloat16*>(o);
    P.lse = lse;
    P.status = status;
    P.rope = rope;
    P.k_next = rope ? static_cast<const __nv_bfloat16*>(k_next) : nullptr;
    P.khat_next = static_cast<__nv_bfloat16*>(khat_next);
    P.sl2 = a.scale * kLog2e;
    P.inv_sl2 = 1.0f / P.sl2;
    P.ntq = (a.T + TQ - 1) / TQ;
    P.ntiles = a.B * P.ntq * kHkv;
    P.win_rows = TQ + a.W;
    P.nwt = (a.W + 4 + 15) / 16;
    P.win_region = round1k((unsigned)P.win_rows * ROWB);
    P.win_slot_bytes = 2 * P.win_region + round1k(TQ * TABB);
    if (!encode_rows(&P.kmap_w, khat, a.B, a.T, P.win_rows) ||
        !encode_rows(&P.vmap_w, v, a.B, a.T, P.win_rows))
        return cudaErrorInvalidValue;
    if (!encode_heads(&P.qmaps[0], q, a.B, a.T, TQ))
        return cudaErrorInvalidValue;
    if (rope && !encode_table(&P.tabmap, rope, a.T)) return cudaErrorInvalidValue;
    for (int p = 0; p < RPG; ++p) {
        const int rows = RUNG_ROWS + 2 * p;
        if (!encode_rows(&P.kmap_r[p], khat, a.B, a.T, rows) || !encode_rows(&P.vmap_r[p], v, a.B, a.T, rows))
            return cudaErrorInvalidValue;
    }
    bool integer_offsets = true;
    for (int r = 0; r < a.nr; ++r) integer_offsets = integer_offsets && a.r[r].t == 0.f;
    const auto kernel = integer_offsets ? fwd_mma_kernel<true> : fwd_mma_kernel<false>;
    const int kidx = integer_offsets ? 1 : 0;
    const size_t smem = 1024 + kHeaderBytes + FwdParams::kQMaps * (size_t)kQTileBytes + (size_t)P.win_slot_bytes +
                        NGS * (size_t)kGroupSlotBytes + NCW * (size_t)kObufBytes;
    if (!ctx_setting_holds(configured_smem[kidx][dev & 63], smem)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        ctx_setting_done(configured_smem[kidx][dev & 63], smem);
    }
    // CTAs per SM for this shared-memory size (looked up once per device and
    // size, so that no runtime query runs while a stream is being captured)
    static int occ_per_sm[2][64];
    static size_t occ_smem[2][64];
    if (occ_smem[kidx][dev & 63] != smem) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, NTHREADS, smem);
        if (e != cudaSuccess) return e;
        occ_per_sm[kidx][dev & 63] = n;
        occ_smem[kidx][dev & 63] = smem;
    }
    int per_sm = occ_per_sm[kidx][dev & 63];
    if (per_sm < 1) per_sm = 1;
    long long grid = (long long)sms * per_sm;
    if (grid > P.ntiles) grid = P.ntiles;
    P.step_g = (int)(grid % kHkv);
    P.step_tq = (int)((grid / kHkv) % P.ntq);
    P.step_b = (int)((grid / kHkv) / P.ntq);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kernel, P);
    if (e != cudaSuccess) return e;
    count_launch();
    return cudaSuccess;
}

cudaError_t launch_rope_k(const LayerArgs& a, const void* k, const float2* rope, void* khat, cudaStream_t s) {
    const unsigned rows = (unsigned)a.B * (unsigned)a.T * kHkv;  // < 2^32: B T < 2^31
    const unsigned per_block = kRopeThreads / 4;
    rope_k_kernel<<<(rows + per_block - 1) / per_block, kRopeThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(k), rope, static_cast<__nv_bfloat16*>(khat), rows, (unsigned)a.T);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
}

cudaError_t launch_fwd_mma(const LayerArgs& a, const void* q, const void* k, const void* v,
                           const float2* rope, void* o, float* lse, void* ws, unsigned* status,
                           cudaStream_t s) {
    if (rope) {
        const cudaError_t e = launch_rope_k(a, k, rope, ws, s);
        if (e != cudaSuccess) return e;
    }
    return launch_fwd_attention(a, q, rope ? ws : k, v, rope, o, lse, nullptr, nullptr, status,
                                rope != nullptr, s);
}

}  // namespace sfa
