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
//  2. fwd_mma_kernel, persistent, (1 producer + 8 consumer) warps per CTA.
//     A CTA owns a tile of TQ = 32 consecutive queries of one sequence b and
//     one key/value head g (4 query heads).  The producer warp streams, with
//     cp.async (zero fill before the sequence start and past its end), the
//     window block (rows i0 - W .. i0 + TQ - 1) and, per rung k, the block of
//     rows i0 - n_k - 1 .. i0 + TQ - 1 - n_k of Khat and V into an mbarrier
//     ring of shared-memory slots.  Each consumer warp owns two query pairs.
//     For a pair (i, i + 1) the scores are formed "keys on M": S^T = Khat_rows
//     (16 x 64) . Qhat^T (64 x 8), N = 2 queries x 4 heads.  Five rungs share
//     one 16-row M tile (rows i - n - 1, i - n, i - n + 1 per rung); the lerp
//     acts on the scores, s = (1 - t) s(row i - n) + t s(row i - n - 1), which
//     equals the score of the interpolated key by linearity, and the
//     probability p is split back onto the two rows as p (1 - t) and p t, so
//     P^T V_rows forms the interpolated value.  One online softmax (base 2,
//     lazy rescale: the running max is raised only when a score exceeds it by
//     more than 2^8) runs over window and rung entries; O^T accumulates in
//     registers and is transposed with movmatrix on the way out.
//
// Shared-memory rows are 128 bytes (64 bf16).  Chunk c (16 bytes) of slot row
// r lives at chunk c ^ ((r + phase) & 7); each rung of an M tile gets phase
// 3 x (its position in the tile) so the 8 rows of every ldmatrix land in 8
// different bank groups.
#include "sfa_internal.cuh"
#include "sfa_mma.cuh"

namespace sfa {

namespace {

constexpr int TQ = 28;                 // queries per tile
constexpr int NCW = 7;                 // consumer warps (2 query pairs each)
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int NRS = 8;                 // rung slots
constexpr int NWS = 2;                 // window slots
constexpr int RUNG_ROWS = TQ + 1;
constexpr int ROWB = 128;              // bytes of one 64-element bf16 row
constexpr int PITCH = 144;             // shared-memory row pitch (128 + 16)
constexpr int TABB = kPairs * 8;       // bytes of one RoPE table row (32 x (cos, sin))
constexpr int RUNGS_PER_TILE = 5;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.0f;          // raise the running max past this margin

struct FwdParams {
    LayerArgs a;
    const __nv_bfloat16* q;
    const __nv_bfloat16* khat;
    const __nv_bfloat16* v;
    const float2* rope;      // nullptr: Q is used as given
    __nv_bfloat16* o;
    float* lse;
    unsigned* status;
    int ntq;                 // query tiles per sequence
    int ntiles;              // B * ntq * Hkv
    int win_rows;            // TQ + W
    int nwt;                 // window M tiles (1 or 2)
    unsigned win_slot_bytes; // Khat + V rows and the tile's RoPE rows
};

using namespace mma;

// Rung position p of an M tile stores its rows 16 (3p mod 8) bytes into its
// slot; with the 144-byte pitch, chunk c of row r then sits in bank group
// (3p + r + c) mod 8, so the 8 rows of every ldmatrix hit 8 bank groups.
__device__ __forceinline__ uint32_t phase_off(int p) { return (uint32_t)(((3 * p) & 7) << 4); }

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

// Rungs are sorted by ceil(d): those usable by some query of the tile form a prefix.
__device__ __forceinline__ int active_rungs(const LayerArgs& a, int i0) {
    int n = 0;
    while (n < a.nr && a.r[n].c <= i0 + TQ - 1) ++n;
    return n;
}

// ---------------------------------------------------------- smem layout

struct Smem {
    uint32_t bars;      // full_w[NWS], empty_w[NWS], full_r[NRS], empty_r[NRS]
    uint32_t win;       // NWS window slots
    uint32_t rung;      // NRS rung slots
    int* abort_flag;
};

__device__ __forceinline__ uint32_t bar_full_w(const Smem& s, int i) { return s.bars + 8 * i; }
__device__ __forceinline__ uint32_t bar_empty_w(const Smem& s, int i) { return s.bars + 8 * (NWS + i); }
__device__ __forceinline__ uint32_t bar_full_r(const Smem& s, int i) { return s.bars + 8 * (2 * NWS + i); }
__device__ __forceinline__ uint32_t bar_empty_r(const Smem& s, int i) {
    return s.bars + 8 * (2 * NWS + NRS + i);
}
constexpr int kBarBytes = 8 * 2 * (NWS + NRS);
constexpr int kHeaderBytes = 256;  // barriers + abort flag, 128-aligned slots follow
// Khat rows then V rows at PITCH, after the rung's phase offset (<= 112 bytes)
constexpr unsigned kRungSlotBytes = ((2u * RUNG_ROWS * PITCH + 112u) + 127u) & ~127u;

// ------------------------------------------------------------ producer

// Rows row0 .. row0 + rows - 1 of Khat and V (head g of sequence b) into a
// slot at `dst` (Khat rows, then V rows, PITCH apart): one bulk copy per valid
// row, rows outside [0, T) zero filled by the warp.  Lane 0 announces the
// bytes on the full barrier first.
__device__ __forceinline__ void stage_rows(const FwdParams& P, uint32_t dst, int rows, int b, int g,
                                           int row0, uint32_t bar, uint32_t extra_bytes, int lane) {
    const int T = P.a.T;
    const int lo = min(rows, max(0, -row0));                 // valid rows [lo, hi)
    const int hi = max(lo, min(rows, T - row0));
    // zero rows outside the sequence: 8 stores of 16 bytes per row and tensor
    const int nzero = rows - max(0, hi - lo);
    for (int z = lane; z < nzero * 16; z += 32) {
        const int zr = z >> 4, part = z & 15;
        const int r = zr < lo ? zr : hi + (zr - lo);
        const int tensor = part >> 3, chunk = part & 7;
        st_zero16(dst + (uint32_t)((tensor * rows + r) * PITCH + chunk * 16));
    }
    __syncwarp();
    const uint32_t bytes = (uint32_t)max(0, hi - lo) * 2u * ROWB + extra_bytes;
    if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
    __syncwarp();
    for (int e = lane; e < 2 * max(0, hi - lo); e += 32) {
        const int tensor = e & 1;
        const int r = lo + (e >> 1);
        const size_t off = (((size_t)b * T + row0 + r) * kHkv + g) * kD;
        bulk_g2s(dst + (uint32_t)((tensor * rows + r) * PITCH), (tensor ? P.v : P.khat) + off, ROWB, bar);
    }
}

__device__ void producer(const FwdParams& P, const Smem& S, int lane) {
    int wcount = 0, rcount = 0;
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x) {
        const Tile x = decode(P, t);
        {
            const int slot = wcount % NWS;
            const uint32_t par = ((wcount / NWS) & 1) ^ 1;
            bool ok = mbar_wait(bar_empty_w(S, slot), par, S.abort_flag);
            if (!__all_sync(kFull, ok)) goto fail;
            const uint32_t base = S.win + slot * P.win_slot_bytes;
            // RoPE rows of the tile's query positions (read by the consumers' Q rotation)
            const int nq = min(TQ, P.a.T - x.i0);
            const uint32_t tab_bytes = P.rope ? (uint32_t)nq * TABB : 0u;
            stage_rows(P, base, P.win_rows, x.b, x.g, x.i0 - P.a.W, bar_full_w(S, slot), tab_bytes,
                       lane);
            if (P.rope && lane == 0)
                bulk_g2s(base + (uint32_t)(2 * P.win_rows * PITCH), P.rope + (size_t)x.i0 * kPairs,
                         tab_bytes, bar_full_w(S, slot));
            ++wcount;
        }
        {
            const int kt = active_rungs(P.a, x.i0);
            for (int k = 0; k < kt; ++k) {
                const int slot = rcount % NRS;
                const uint32_t par = ((rcount / NRS) & 1) ^ 1;
                bool ok = mbar_wait(bar_empty_r(S, slot), par, S.abort_flag);
                if (!__all_sync(kFull, ok)) goto fail;
                stage_rows(P, S.rung + slot * kRungSlotBytes + phase_off(k % RUNGS_PER_TILE), RUNG_ROWS,
                           x.b, x.g, x.i0 - P.a.r[k].n - 1, bar_full_r(S, slot), 0u, lane);
                ++rcount;
            }
        }
    }
    return;
fail:
    if (lane == 0) {
        *S.abort_flag = 1;
        if (P.status) atomicOr(P.status, SFA_DEVSTAT_WAIT_TIMEOUT);
    }
    // no copy of this CTA may land after it exits: wait (bounded) for every
    // slot's last announced phase
    if (lane == 0) {
        for (int n = max(0, wcount - NWS); n < wcount; ++n)
            (void)mbar_wait(bar_full_w(S, n % NWS), (n / NWS) & 1, nullptr);
        for (int n = max(0, rcount - NRS); n < rcount; ++n)
            (void)mbar_wait(bar_full_r(S, n % NRS), (n / NRS) & 1, nullptr);
    }
}

// ------------------------------------------------------------ consumers

// One query pair (i, i + 1) of one key/value head: the B fragments of
// Qhat^T (scaled into log2 units), the O^T accumulators and softmax state of
// this thread's two columns (query tig/2, heads 2(tig&1) and 2(tig&1)+1).
struct Unit {
    uint32_t qf[4][2];
    float o[4][4];
    float m[2];
    float l[2];
};

// Raw Q of this thread's B-fragment column (query i0 + u + g8/4, head
// g*4 + g8%4): dimensions 16 s + 8 h + 2 tig + {0, 1}.
__device__ __forceinline__ void fetch_q(const FwdParams& P, const Tile& x, int u, int lane,
                                        uint32_t raw[4][2]) {
    const int g8 = lane >> 2, tig = lane & 3;
    const int iq = x.i0 + u + (g8 >> 2);
    if (iq < P.a.T) {
        const __nv_bfloat16* qp =
            P.q + (((size_t)x.b * P.a.T + iq) * kHq + x.g * kG + (g8 & 3)) * kD + 2 * tig;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            raw[s][0] = __ldg(reinterpret_cast<const unsigned*>(qp + 16 * s));
            raw[s][1] = __ldg(reinterpret_cast<const unsigned*>(qp + 16 * s + 8));
        }
    } else {
#pragma unroll
        for (int s = 0; s < 4; ++s) raw[s][0] = raw[s][1] = 0u;
    }
}

// Rotate (RoPE rows of the tile in shared memory at `tab`) and scale the raw
// Q into B fragments; reset the accumulators.
__device__ __forceinline__ void start_unit(const FwdParams& P, uint32_t tab, int i0, int u, int lane,
                                           const uint32_t raw[4][2], Unit& U) {
    const int g8 = lane >> 2, tig = lane & 3;
    const float sl2 = P.a.scale * kLog2e;
    // RoPE rows are staged only for positions < T
    const bool rot = P.rope && (i0 + u + (g8 >> 2) < P.a.T);
    const uint32_t trow = tab + (uint32_t)((u + (g8 >> 2)) * TABB + 2 * tig * 8);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // dims m = 16 s + 8 h + 2 tig + {0, 1} and their partners m + 32
            float4 cs = make_float4(1.f, 0.f, 1.f, 0.f);
            if (rot) {
                asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                             : "=f"(cs.x), "=f"(cs.y), "=f"(cs.z), "=f"(cs.w)
                             : "r"(trow + (uint32_t)((16 * s + 8 * h) * 8)));
            }
            const float2 xv = unpack_bf16(raw[s][h]);
            const float2 yv = unpack_bf16(raw[s + 2][h]);
            const float x0 = (xv.x * cs.x - yv.x * cs.y) * sl2;
            const float y0 = (yv.x * cs.x + xv.x * cs.y) * sl2;
            const float x1 = (xv.y * cs.z - yv.y * cs.w) * sl2;
            const float y1 = (yv.y * cs.z + xv.y * cs.w) * sl2;
            U.qf[s][h] = pack_bf16(x0, x1);
            U.qf[s + 2][h] = pack_bf16(y0, y1);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) U.o[j][e] = 0.f;
    U.m[0] = U.m[1] = -INFINITY;
    U.l[0] = U.l[1] = 0.f;
}

// S^T (16 rows x 8 columns) = Khat rows . Qhat^T; `kaddr` is this lane's
// ldmatrix row (row (lane & 7) + 8 ((lane >> 3) & 1) of the tile).
__device__ __forceinline__ void scores(uint32_t kaddr, const Unit& U, float c[4]) {
    c[0] = c[1] = c[2] = c[3] = 0.f;
    const uint32_t hi = (uint32_t)(((threadIdx.x & 31) >> 4) << 4);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kaddr + 32 * s + hi, a0, a1, a2, a3);
        mma16816(c, a0, a1, a2, a3, U.qf[s][0], U.qf[s][1]);
    }
}

// O^T += V_rows^T . P^T, P^T given as bf16 B fragments b0 (rows 0-7), b1
// (rows 8-15); `vaddr` is this lane's ldmatrix row (row (lane & 7) + 8 (lane >> 4)).
__device__ __forceinline__ void accumulate(uint32_t vaddr, uint32_t b0, uint32_t b1, Unit& U) {
    const uint32_t hi = (uint32_t)((((threadIdx.x & 31) >> 3) & 1) << 4);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vaddr + 32 * j + hi, a0, a1, a2, a3);
        mma16816(U.o[j], a0, a1, a2, a3, b0, b1);
    }
}

// Online-softmax step for this thread's 4 candidate scores (rows lo/hi x 2
// columns, -inf where absent): raises the running max lazily, returns the
// probabilities in p.
__device__ __forceinline__ void softmax_step(Unit& U, const float s[4], float p[4]) {
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int w = 4; w <= 16; w <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, w));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, w));
    }
    const bool need = (mx0 > U.m[0] + kLazy) || (mx1 > U.m[1] + kLazy);
    if (__any_sync(kFull, need)) {
        const float n0 = fmaxf(U.m[0], mx0), n1 = fmaxf(U.m[1], mx1);
        const float c0 = (U.m[0] == -INFINITY) ? (n0 == -INFINITY ? 1.f : 0.f) : fast_exp2(U.m[0] - n0);
        const float c1 = (U.m[1] == -INFINITY) ? (n1 == -INFINITY ? 1.f : 0.f) : fast_exp2(U.m[1] - n1);
        U.m[0] = n0;
        U.m[1] = n1;
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
    p[0] = s[0] == -INFINITY ? 0.f : fast_exp2(s[0] - U.m[0]);
    p[1] = s[1] == -INFINITY ? 0.f : fast_exp2(s[1] - U.m[1]);
    p[2] = s[2] == -INFINITY ? 0.f : fast_exp2(s[2] - U.m[0]);
    p[3] = s[3] == -INFINITY ? 0.f : fast_exp2(s[3] - U.m[1]);
    U.l[0] += p[0] + p[2];
    U.l[1] += p[1] + p[3];
}

// Window M tile wt of a query pair at tile offset u (query positions i, i + 1):
// slot rows u + R, R = 16 wt .. 16 wt + 15, hold positions i - W + R.
__device__ __forceinline__ void window_tile(const FwdParams& P, uint32_t slot, int u, int i, int wt,
                                            int lane, Unit& U) {
    const int g8 = lane >> 2, tig = lane & 3, q = tig >> 1;
    const int W = P.a.W;
    const int maxr = P.win_rows - 1;
    const int rk = min(u + 16 * wt + (lane & 7) + (((lane >> 3) & 1) << 3), maxr);
    const int rv = min(u + 16 * wt + (lane & 7) + ((lane >> 4) << 3), maxr);
    float c[4];
    scores(slot + (uint32_t)(rk * PITCH), U, c);
    float s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int R = 16 * wt + g8 + ((e >> 1) << 3);  // M row of this value
        const bool ok = (R >= q) && (R <= W + q) && (i - W + R >= 0);
        s[e] = ok ? c[e] : -INFINITY;
    }
    float p[4];
    softmax_step(U, s, p);
    const uint32_t b0 = movm_t(pack_bf16(p[0], p[1]));
    const uint32_t b1 = movm_t(pack_bf16(p[2], p[3]));
    accumulate(slot + (uint32_t)((P.win_rows + rv) * PITCH), b0, b1, U);
}

// Shared-memory address of M row R of a rung tile holding np rungs
// (R = 3 p + e): rung p's slot row u + e.  The pad row 15 and the rows of
// absent rungs read a row of rung 0 whose bank group is the one left free.
__device__ __forceinline__ uint32_t rung_row(int R, int np, int u, uint32_t ring, int rc) {
    const int p = R / 3;
    if (R < 15 && p < np) {
        const int r = u + (R - 3 * p);
        return ring + ((rc + p) % NRS) * kRungSlotBytes + phase_off(p) + (uint32_t)(r * PITCH);
    }
    const int r = (u + 7 <= TQ) ? u + 7 : u - 1;
    return ring + (rc % NRS) * kRungSlotBytes + (uint32_t)(r * PITCH);
}

__device__ __forceinline__ void rung_tile(const FwdParams& P, uint32_t ring, int rc, int np, int k0,
                                          int u, int i, int lane, Unit& U) {
    const int g8 = lane >> 2, tig = lane & 3, q = tig >> 1;
    const uint32_t kaddr = rung_row((lane & 7) + (((lane >> 3) & 1) << 3), np, u, ring, rc);
    const uint32_t vaddr =
        rung_row((lane & 7) + ((lane >> 4) << 3), np, u, ring, rc) + (uint32_t)(RUNG_ROWS * PITCH);
    float c[4];
    scores(kaddr, U, c);
    // value of the next M row (row a of an interpolation whose row b is this one)
    const float nx0 = shfl(g8 == 0 ? c[2] : c[0], (lane + 4) & 31);
    const float nx1 = shfl(g8 == 0 ? c[3] : c[1], (lane + 4) & 31);
    const float nx2 = shfl(c[2], (lane + 4) & 31);
    const float nx3 = shfl(c[3], (lane + 4) & 31);
    const float nx[4] = {nx0, nx1, nx2, nx3};
    float s[4], tw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // h = 0: M row g8, h = 1: M row g8 + 8
        const int R = g8 + 8 * h;
        const int p = R / 3, e = R - 3 * p;
        bool useful = (R < 15) && (p < np) && (e == q);
        float t = 0.f;
        if (useful) {
            const Rung rg = P.a.r[k0 + p];
            t = rg.t;
            useful = (i + q >= rg.c);
        }
        tw[h] = t;
        s[2 * h + 0] = useful ? (1.f - t) * nx[2 * h + 0] + t * c[2 * h + 0] : -INFINITY;
        s[2 * h + 1] = useful ? (1.f - t) * nx[2 * h + 1] + t * c[2 * h + 1] : -INFINITY;
    }
    float p[4];
    softmax_step(U, s, p);
    // p t stays on row b (this row); p (1 - t) moves to row a (the next row)
    float pa[4], pt[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float t = tw[e >> 1];
        pa[e] = p[e] * (1.f - t);
        pt[e] = p[e] * t;
    }
    const float r0 = shfl(pa[0], (lane + 28) & 31);
    const float r1 = shfl(pa[1], (lane + 28) & 31);
    const float r2 = shfl(g8 == 7 ? pa[0] : pa[2], (lane + 28) & 31);
    const float r3 = shfl(g8 == 7 ? pa[1] : pa[3], (lane + 28) & 31);
    const float lo0 = pt[0] + (g8 == 0 ? 0.f : r0);
    const float lo1 = pt[1] + (g8 == 0 ? 0.f : r1);
    const float hi0 = pt[2] + r2;
    const float hi1 = pt[3] + r3;
    const uint32_t b0 = movm_t(pack_bf16(lo0, lo1));
    const uint32_t b1 = movm_t(pack_bf16(hi0, hi1));
    accumulate(vaddr, b0, b1, U);
}

__device__ __forceinline__ void store_unit(const FwdParams& P, const Tile& x, int u, int lane,
                                           Unit& U) {
    const int g8 = lane >> 2, tig = lane & 3;
    float l0 = U.l[0], l1 = U.l[1];
#pragma unroll
    for (int w = 4; w <= 16; w <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, w);
        l1 += __shfl_xor_sync(kFull, l1, w);
    }
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    // column g8 of the transposed fragments: query i0 + u + g8/4, head g*4 + g8%4
    const int iq = x.i0 + u + (g8 >> 2);
    const bool in = iq < P.a.T;
    __nv_bfloat16* op = P.o + (((size_t)x.b * P.a.T + (in ? iq : 0)) * kHq + x.g * kG + (g8 & 3)) * kD +
                        2 * tig;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = movm_t(pack_bf16(U.o[j][0] * inv0, U.o[j][1] * inv1));
        const uint32_t hi = movm_t(pack_bf16(U.o[j][2] * inv0, U.o[j][3] * inv1));
        if (in) {
            *reinterpret_cast<uint32_t*>(op + 16 * j) = lo;
            *reinterpret_cast<uint32_t*>(op + 16 * j + 8) = hi;
        }
    }
    if (P.lse && g8 == 0) {
        const int q = tig >> 1;
        const int iq2 = x.i0 + u + q;
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
    uint32_t raw[2][4][2];
    if (blockIdx.x < P.ntiles) {
        const Tile x = decode(P, blockIdx.x);
#pragma unroll
        for (int k = 0; k < 2; ++k) fetch_q(P, x, u0 + 2 * k, lane, raw[k]);
    }
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x) {
        const Tile x = decode(P, t);
        Unit U[2];
        {
            const int slot = wcount % NWS;
            bool ok = mbar_wait(bar_full_w(S, slot), (wcount / NWS) & 1, S.abort_flag);
            if (!__all_sync(kFull, ok)) goto fail;
            const uint32_t base = S.win + slot * P.win_slot_bytes;
#pragma unroll
            for (int k = 0; k < 2; ++k)
                start_unit(P, base + (uint32_t)(2 * P.win_rows * PITCH), x.i0, u0 + 2 * k, lane, raw[k],
                           U[k]);
            // the next tile's Q is in flight while this tile is computed
            if (t + (int)gridDim.x < P.ntiles) {
                const Tile nx = decode(P, t + gridDim.x);
#pragma unroll
                for (int k = 0; k < 2; ++k) fetch_q(P, nx, u0 + 2 * k, lane, raw[k]);
            }
            for (int wt = 0; wt < P.nwt; ++wt)
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    window_tile(P, base, u0 + 2 * k, x.i0 + u0 + 2 * k, wt, lane, U[k]);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty_w(S, slot));
            ++wcount;
        }
        {
            const int kt = active_rungs(P.a, x.i0);
            for (int k0 = 0; k0 < kt; k0 += RUNGS_PER_TILE) {
                const int np = min(RUNGS_PER_TILE, kt - k0);
                bool ok = true;
                for (int p = 0; p < np; ++p) {
                    const int n = rcount + p;
                    ok = ok && mbar_wait(bar_full_r(S, n % NRS), (n / NRS) & 1, S.abort_flag);
                }
                if (!__all_sync(kFull, ok)) goto fail;
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    rung_tile(P, S.rung, rcount, np, k0, u0 + 2 * k, x.i0 + u0 + 2 * k, lane, U[k]);
                __syncwarp();
                if (lane == 0)
                    for (int p = 0; p < np; ++p) mbar_arrive(bar_empty_r(S, (rcount + p) % NRS));
                rcount += np;
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) store_unit(P, x, u0 + 2 * k, lane, U[k]);
    }
    return;
fail:
    if (lane == 0) {
        *S.abort_flag = 1;
        if (P.status) atomicOr(P.status, SFA_DEVSTAT_WAIT_TIMEOUT);
    }
}

__global__ void __maxnreg__(128) fwd_mma_kernel(const __grid_constant__ FwdParams P) {
    extern __shared__ __align__(128) unsigned char smem[];
    Smem S;
    S.bars = smem_u32(smem);
    S.abort_flag = reinterpret_cast<int*>(smem + kBarBytes);
    S.win = smem_u32(smem) + kHeaderBytes;
    S.rung = S.win + NWS * P.win_slot_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    if (warp == NCW)
        producer(P, S, lane);
    else
        consumer(P, S, warp, lane);
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

struct DeviceInfo {
    int sms = 0;
    size_t configured_smem = 0;
};

DeviceInfo& device_info(int dev) {
    static DeviceInfo info[64];
    return info[dev & 63];
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
    P.a = a;
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.v = static_cast<const __nv_bfloat16*>(v);
    P.o = static_cast<__nv_bfloat16*>(o);
    P.lse = lse;
    P.status = status;
    P.rope = rope;
    P.ntq = (a.T + TQ - 1) / TQ;
    P.ntiles = a.B * P.ntq * kHkv;
    P.win_rows = TQ + a.W;
    P.nwt = (a.W + 2 + 15) / 16;
    P.win_slot_bytes = (unsigned)(((2 * P.win_rows * PITCH + TQ * TABB) + 127) & ~127);
    if (rope) {
        const long long rows = (long long)a.B * a.T * kHkv;
        const long long threads = rows * 4;
        rope_k_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(k), rope, static_cast<__nv_bfloat16*>(ws), rows, a.T);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
        P.khat = static_cast<const __nv_bfloat16*>(ws);
    } else {
        P.khat = static_cast<const __nv_bfloat16*>(k);
    }
    const size_t smem = kHeaderBytes + NWS * (size_t)P.win_slot_bytes + NRS * (size_t)kRungSlotBytes;
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
