// sfa_bwd_mma.cu -- bf16 backward on the tensor cores (mma.sync, fp32
// accumulation), the fast path of sfa_backward.
//
// Gradients of the attention of "Depth-Staggered Fibonacci Spacing for Sparse
// Attention" (arXiv 2606.28560), section 2 "Attended set" and
// "Implementation notes": for query i, head h and every entry e of its key
// list (window rows, and per rung the interpolation of rows a = i - n (weight
// 1 - t) and b = i - n - 1 (weight t)), with the forward's log-sum-exp and
// D = dO . O,
//   p = exp(s - lse), dp = dO . vtilde, ds = p (dp - D),
//   dqhat += scale ds ktilde,  dkhat[row] += w scale ds qhat,  dv[row] += w p dO,
//   dL/dt += scale ds (qhat . khat_b - qhat . khat_a) + p (dO . v_b - dO . v_a),
// dL/dalpha = sum_k f_k dL/dt_k, dL/dtheta = dL/dalpha (alpha - 0.5)(1.5 - alpha).
//
// Three launches, the last two as programmatic dependents of the one before:
//  1. bwd_prep_kernel: zeroes the fp32 dKhat / dV accumulators and writes
//     Khat = RoPE(K) (bf16, natural dimension order) into the workspace (the
//     rotation is skipped when the inputs come rotated).
//  2. bwd_mma_kernel: persistent, the forward's tile map and load ring (one
//     producer lane, seven consumer warps, a warp owns a quad of queries as
//     two pairs).  Per M tile ("keys on M", as in the forward) it recomputes
//     S^T = Khat_rows . Qhat^T and dP^T = V_rows . dO^T, forms p and ds, and
//       dQhat^T += Khat_rows^T . dS^T        (registers, one tile at a time)
//       dKhat_rows = dS . Qhat, dV_rows = P . dO   (m16n8k8 / m16n8k16)
//     The interpolation weights split ds and p onto rows a and b inside the
//     thread, exactly as in the forward.  A window M tile's 16 rows (already
//     summed over the warp's four queries by the MMA) are staged in shared
//     memory and added to the fp32 accumulators by four TMA tensor reductions
//     (cp.reduce.async.bulk.tensor .add); rung rows that several M rows of a
//     warp share (row a of query i is row b of query i + 1) are summed in
//     registers and go to the accumulators with red.global.add.v2.  dQ is
//     rotated back (R(i)^T) and stored through shared memory by TMA; dL/dt is
//     summed per warp in shared memory and per CTA into the workspace.
//  3. bwd_finish_mma_kernel: dK = R(j)^T dKhat and dV to the caller's dtype,
//     and the fixed-order (fp64) reduction of dL/dalpha and dL/dtheta.
#include <cstring>

#include "sfa_internal.cuh"
#include "sfa_mma.cuh"
#include "sfa_ring.cuh"

namespace sfa {

namespace {

using namespace mma;
using namespace ring;

constexpr int NCW = 7;                         // consumer warps (a quad of queries each)
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr unsigned kObufBytes = 2 * 8 * ROWB;  // per consumer warp: dQ of 2 query pairs
constexpr unsigned kDtBytes = NCW * SFA_MAX_RUNGS * 4;
constexpr int kMaxGrid = 1024;                 // CTAs of the persistent kernel (dL/dt partials)
constexpr int kPrepThreads = 256;
constexpr int kFinishThreads = 256;

struct BwdParams {
    static constexpr int kQMaps = 3;  // the query slot carries the tile's Q, dO and O
    static constexpr bool kWinRope = true;
    CUtensorMap qmaps[kQMaps];
    CUtensorMap kmap_w;
    CUtensorMap vmap_w;
    CUtensorMap kmap_r[RPG];
    CUtensorMap vmap_r[RPG];
    CUtensorMap tabmap;        // RoPE table rows of a tile (with RoPE)
    CUtensorMap dkred, dvred;  // fp32 accumulators [B][T][2][64], box 32 dims x 16 rows, 128-byte swizzle
    LayerArgs a;
    const __nv_bfloat16* q;
    const __nv_bfloat16* o;
    const __nv_bfloat16* dO;
    __nv_bfloat16* dq;
    const float* lse;
    const float2* rope;        // nullptr: inputs are used as given
    float* dk_acc;             // [B][T][Hkv][D] fp32, rotated frame
    float* dv_acc;
    long long dv_off;          // dv_acc - dk_acc (floats)
    float* dt_part;            // [gridDim.x][SFA_MAX_RUNGS]
    unsigned* status;
    float sl2;                 // scale x log2(e)
    float scale;
    int ntq, ntiles;
    int step_g, step_tq, step_b;
    int win_rows, nwt;
    unsigned win_region, win_slot_bytes;
};

// ------------------------------------------------------------ consumers

// One query pair of the warp's quad: B fragments of Qhat^T and dO^T in the
// natural dimension order (k-step s, half h: dimensions 16 s + 8 h + 2 tig +
// {0, 1} of column g8), the dQhat^T accumulators, and the per-column
// constants of this thread's two C columns (query tig / 2, heads 2 (tig & 1)
// + {0, 1}).
struct BUnit {
    uint32_t qf[4][2];
    uint32_t df[4][2];
    uint32_t qm[8];     // Qhat as the B operand of dKhat_rows (8-dimension chunk c)
    uint32_t dm[8];     // dO as the B operand of dV_rows
    float dq[4][4];
    float2 lse2;        // log-sum-exp x log2(e)
    float2 D;           // dO . O
    bool qok;           // this thread's C-column query lies inside the sequence
};

struct BLane {
    int g8, q;
    bool useful;        // this thread's rung rows belong to its column query
    bool is_a;          // lanes 0..15: query e = 0 of each pair
    unsigned wmask;
    uint32_t kn[2];     // rung tile of unit k: non-transposed row offsets (Khat; + kVOff: V)
    uint32_t kt[2];     // rung tile of unit k: transposed row offsets (Khat)
    uint32_t wk, wt;    // window tile 0: non-transposed / transposed row offsets
    uint32_t ob[2];
};

__device__ __forceinline__ BLane make_blane(int lane, int u0, int W, int win_rows) {
    BLane L;
    L.g8 = lane >> 2;
    L.q = (lane & 3) >> 1;
    L.useful = (L.g8 >> 2) == L.q;
    L.is_a = lane < 16;
    const int p = lane & 3, e = (lane >> 2) & 1;
    for (int k = 0; k < 2; ++k) {
        const int u = u0 + 2 * k;
        L.kn[k] = rung_row(p, u, e, (lane >> 3) & 1, lane >> 4, false);
        L.kt[k] = rung_row(p, u, e, lane >> 4, (lane >> 3) & 1, false);
    }
    const int rk = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int rv = (lane & 7) + ((lane >> 4) << 3);
    L.wk = swz_row(min(u0 + rk, win_rows - 1), lane >> 4);
    L.wt = swz_row(min(u0 + rv, win_rows - 1), (lane >> 3) & 1);
    L.wmask = 0u;
    for (int wt = 0; wt < 3; ++wt)
        for (int k = 0; k < 2; ++k)
            for (int e2 = 0; e2 < 4; ++e2) {
                const int R = 16 * wt + L.g8 + ((e2 >> 1) << 3);
                const int qq = 2 * k + L.q;
                if (R >= qq && R <= W + qq) L.wmask |= 1u << (8 * wt + 4 * k + e2);
            }
    const int row = lane & 7, mi = lane >> 3;
    for (int jj = 0; jj < 2; ++jj) {
        const int chunk = 2 * (2 * jj + (mi >> 1)) + (mi & 1);
        L.ob[jj] = (uint32_t)(row * ROWB) + (uint32_t)(((chunk ^ row) & 7) << 4);
    }
    return L;
}

// acc[0..1] += (a, b) when ok (predicated inside the instruction, no branch).
__device__ __forceinline__ void red_v2(float* p, float a, float b, bool ok) {
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.b32 q, %3, 0;\n @q red.global.add.v2.f32 [%0], {%1, %2};\n}\n" ::"l"(p),
        "f"(a), "f"(b), "r"((int)ok)
        : "memory");
}

__device__ __forceinline__ void tma_reduce_add_4d(const void* tmap, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            tmap),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void sts64(uint32_t a, float x, float y) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}

// Address of acc[b][row][g][2 tig] (row_base = b T Hkv + g), and whether the
// row lies inside the sequence.
__device__ __forceinline__ float* acc_row(float* acc, size_t row_base, int row, int T, int tig, bool& ok) {
    ok = ok && row >= 0 && row < T;
    return acc + (row_base + (size_t)(ok ? row : 0) * kHkv) * kD + 2 * tig;
}

__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ float2 shfl2_xor(float2 v, int m) {
    return f2(__shfl_xor_sync(kFull, v.x, m), __shfl_xor_sync(kFull, v.y, m));
}

// D = A (16 x 8 bf16, row) * B (8 x 8 bf16, col), fp32 (no accumulator input).
__device__ __forceinline__ void mma1688_z(float d[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
        "{%7,%7,%7,%7};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0), "f"(0.0f));
}

// The natural-order B-fragment words of row r of a swizzled query tile
// (addr = row start + 4 tig): word (s, h) = dimensions 16 s + 8 h + 2 tig +
// {0, 1}, in 16-byte chunk 2 s + h stored at chunk (2 s + h) ^ (r & 7).
__device__ __forceinline__ void load_frag_s(uint32_t addr, int r, uint32_t w[4][2]) {
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            asm volatile("ld.shared.b32 %0, [%1];"
                         : "=r"(w[s][h])
                         : "r"(addr + (uint32_t)((((2 * s + h) ^ (r & 7)) << 4))));
}

// Start of a tile for unit k (query pair at tile offset u): Qhat^T, dO^T and
// their dK/dV forms, D and the log-sum-exp of this thread's C columns.
__device__ __forceinline__ void start_bunit(const BwdParams& P, const Smem& S, const Tile& x, int nq, int u,
                                            int lane, BUnit& U) {
    const uint32_t slot = S.win;
    const int g8 = lane >> 2, tig = lane & 3;
    const int T = P.a.T;
    const uint32_t tab = slot + 2 * P.win_region;
    // B-fragment column: query u + g8/4, head g8 % 4 = row 4 u + g8 of the
    // query tiles (128-byte swizzle)
    uint32_t ow[4][2];
    const uint32_t qrow = S.qslot + (uint32_t)((4 * u + g8) * ROWB) + 4u * tig;
    load_frag_s(qrow, 4 * u + g8, U.qf);
    load_frag_s(qrow + kQTileBytes, 4 * u + g8, U.df);
    load_frag_s(qrow + 2 * kQTileBytes, 4 * u + g8, ow);
    // C columns: query u + tig/2, heads 2 (tig & 1) + {0, 1}
    const int ic = x.i0 + u + (tig >> 1);
    U.qok = ic < T;
    const float* lp = P.lse + ((size_t)x.b * T + min(ic, T - 1)) * kHq + x.g * kG + 2 * (tig & 1);
    U.lse2 = f2(__ldg(lp) * kLog2e, __ldg(lp + 1) * kLog2e);
    // D of column g8 over this thread's 16 dimensions, then the quad of tig
    float dpart = 0.f;
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float2 a = unpack_bf16(U.df[s][h]), b = unpack_bf16(ow[s][h]);
            dpart = fmaf(a.x, b.x, fmaf(a.y, b.y, dpart));
        }
    dpart += __shfl_xor_sync(kFull, dpart, 1);
    dpart += __shfl_xor_sync(kFull, dpart, 2);
    U.D = f2(__shfl_sync(kFull, dpart, 4 * (2 * tig)), __shfl_sync(kFull, dpart, 4 * (2 * tig + 1)));
    if (P.rope) {
        // rotation pairs (m, m + 32): words (s, h) and (s + 2, h) of the thread
        const int pr = min(u + (g8 >> 2), nq - 1);
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // pairs m, m + 1: table chunk m / 2 = 8 s + 4 h + tig of row pr
                // (h flips bit 2 of the swizzled chunk)
                const int m = 16 * s + 8 * h + 2 * tig;
                const float4 cs = lds_f4((tab + tab_chunk(pr, 8 * s + tig)) ^ (uint32_t)(h << 6));
                const float2 xv = unpack_bf16(U.qf[s][h]), yv = unpack_bf16(U.qf[s + 2][h]);
                U.qf[s][h] = rope_x(xv, yv, cs);
                U.qf[s + 2][h] = rope_y(xv, yv, cs);
            }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        U.qm[c] = movm_t(U.qf[c >> 1][c & 1]);
        U.dm[c] = movm_t(U.df[c >> 1][c & 1]);
    }
}

// Window M tile wt of the quad at tile offset u0 (rows u0 + 16 wt .. of the
// window block, positions i0 + u0 - W + R).
template <bool kFirst>
__device__ __forceinline__ void bwd_window_tile(const BwdParams& P, uint32_t slot, const Tile& x, int u0, int wt,
                                                const BLane& L, BUnit* U, uint32_t stg) {
    const int lane = threadIdx.x & 31;
    const int i0 = x.i0;
    uint32_t kro = L.wk, tro = L.wt;
    if (!kFirst) {
        const int maxr = P.win_rows - 1;
        kro = swz_row(min(u0 + 16 * wt + (lane & 7) + (((lane >> 3) & 1) << 3), maxr), lane >> 4);
        tro = swz_row(min(u0 + 16 * wt + (lane & 7) + ((lane >> 4) << 3), maxr), (lane >> 3) & 1);
    }
    const uint32_t vslot = slot + P.win_region;
    float cs[2][4], cp[2][4];
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
        uint32_t a0, a1, a2, a3, v0, v1, v2, v3;
        ldsm_x4(slot + (kro ^ (uint32_t)(s2 << 5)), a0, a1, a2, a3);
        ldsm_x4(vslot + (kro ^ (uint32_t)(s2 << 5)), v0, v1, v2, v3);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (s2 == 0) {
                mma16816_z(cs[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
                mma16816_z(cp[k], v0, v1, v2, v3, U[k].df[s2][0], U[k].df[s2][1]);
            } else {
                mma16816(cs[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
                mma16816(cp[k], v0, v1, v2, v3, U[k].df[s2][0], U[k].df[s2][1]);
            }
        }
    }
    unsigned mask = L.wmask >> (8 * wt);
    const int lo = P.a.W - (i0 + u0) - 16 * wt;
    if (lo > 0) {
        if (L.g8 < lo) mask &= ~0x33u;
        if (L.g8 + 8 < lo) mask &= ~0xccu;
    }
    uint32_t bq[2][2], ad[2][2], ap[2][2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float pv[4], dsv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool ok = ((mask >> (4 * k + e)) & 1u) && U[k].qok;
            const float l2 = (e & 1) ? U[k].lse2.y : U[k].lse2.x;
            const float Dv = (e & 1) ? U[k].D.y : U[k].D.x;
            const float pe = ok ? fast_exp2(fmaf(cs[k][e], P.sl2, -l2)) : 0.f;
            pv[e] = pe;
            dsv[e] = pe * (cp[k][e] - Dv) * P.scale;
        }
        ad[k][0] = pack_bf16(dsv[0], dsv[1]);
        ad[k][1] = pack_bf16(dsv[2], dsv[3]);
        ap[k][0] = pack_bf16(pv[0], pv[1]);
        ap[k][1] = pack_bf16(pv[2], pv[3]);
        bq[k][0] = movm_t(ad[k][0]);
        bq[k][1] = movm_t(ad[k][1]);
    }
    // dQhat^T += Khat_rows^T . dS^T
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(slot + (tro ^ (uint32_t)(j << 5)), a0, a1, a2, a3);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (kFirst)
                mma16816_z(U[k].dq[j], a0, a1, a2, a3, bq[k][0], bq[k][1]);
            else
                mma16816(U[k].dq[j], a0, a1, a2, a3, bq[k][0], bq[k][1]);
        }
    }
    // dKhat_rows = dS . Qhat and dV_rows = P . dO over both pairs (k = 16
    // columns), this thread's rows g8 and g8 + 8, dimensions 8 c + 2 tig + {0, 1}
    const int tig = lane & 3;
    const int rstart = i0 + u0 - P.a.W + 16 * wt;
    if (rstart >= 0) {
        // stage the 16 rows (dK, dV; two halves of 32 dimensions each, 128-byte
        // swizzle) and add them with four tensor reductions; rows past T are
        // clipped by the map, rows outside the quad's window carry zeros.  A
        // reduction may not start before row 0, so tiles at the sequence
        // start take the per-thread path below.
        if (lane == 0) bulk_wait_read();
        __syncwarp();
        const int r0s = L.g8, r1s = L.g8 + 8;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float dk[4], dv[4];
            mma16816_z(dk, ad[0][0], ad[0][1], ad[1][0], ad[1][1], U[0].qm[c], U[1].qm[c]);
            mma16816_z(dv, ap[0][0], ap[0][1], ap[1][0], ap[1][1], U[0].dm[c], U[1].dm[c]);
            const int half = c >> 2, ch = 2 * (c & 3) + (tig >> 1);
            const uint32_t w = (uint32_t)((2 * tig) & 3) * 4u;
            const uint32_t a0 = stg + (uint32_t)((half * 16 + r0s) * 128 + (((ch ^ r0s) & 7) << 4)) + w;
            const uint32_t a1 = stg + (uint32_t)((half * 16 + r1s) * 128 + (((ch ^ r1s) & 7) << 4)) + w;
            sts64(a0, dk[0], dk[1]);
            sts64(a1, dk[2], dk[3]);
            sts64(a0 + 4096u, dv[0], dv[1]);
            sts64(a1 + 4096u, dv[2], dv[3]);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
            tma_reduce_add_4d(&P.dkred, stg, 0, x.g, rstart, x.b);
            tma_reduce_add_4d(&P.dkred, stg + 2048u, 32, x.g, rstart, x.b);
            tma_reduce_add_4d(&P.dvred, stg + 4096u, 0, x.g, rstart, x.b);
            tma_reduce_add_4d(&P.dvred, stg + 6144u, 32, x.g, rstart, x.b);
            bulk_commit();
        }
        return;
    }
    const int r0 = rstart + L.g8;
    bool use0 = 16 * wt + L.g8 <= P.a.W + 3, use1 = 16 * wt + L.g8 + 8 <= P.a.W + 3;
    const size_t rb = (size_t)x.b * P.a.T * kHkv + x.g;
    float* p0 = acc_row(P.dk_acc, rb, r0, P.a.T, tig, use0);
    float* p1 = acc_row(P.dk_acc, rb, r0 + 8, P.a.T, tig, use1);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float dk[4], dv[4];
        mma16816_z(dk, ad[0][0], ad[0][1], ad[1][0], ad[1][1], U[0].qm[c], U[1].qm[c]);
        mma16816_z(dv, ap[0][0], ap[0][1], ap[1][0], ap[1][1], U[0].dm[c], U[1].dm[c]);
        red_v2(p0 + 8 * c, dk[0], dk[1], use0);
        red_v2(p0 + P.dv_off + 8 * c, dv[0], dv[1], use0);
        red_v2(p1 + 8 * c, dk[2], dk[3], use1);
        red_v2(p1 + P.dv_off + 8 * c, dv[2], dv[3], use1);
    }
}

// Rung M tiles of the quad (pairs at tile offsets u0, u0 + 2) for the np
// rungs k0 .. k0 + np - 1 of the group in slot gslot.
__device__ __forceinline__ void bwd_rung_tile(const BwdParams& P, const Smem& S, uint32_t gslot, const Tile& x,
                                              int k0, int np, int nr, int u0, const BLane& L, BUnit* U,
                                              float* dt_w) {
    const int lane = threadIdx.x & 31;
    const int tig = lane & 3;
    uint32_t kn[2], kt[2];
    if (np == RPG) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            kn[k] = gslot + L.kn[k];
            kt[k] = gslot + L.kt[k];
        }
    } else {
        const int p = (lane & 3) < np ? (lane & 3) : 0, e = (lane >> 2) & 1;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            kn[k] = gslot + rung_row(p, u0 + 2 * k, e, (lane >> 3) & 1, lane >> 4, false);
            kt[k] = gslot + rung_row(p, u0 + 2 * k, e, lane >> 4, (lane >> 3) & 1, false);
        }
    }
    // S^T = Khat_rows . Qhat^T, dP^T = V_rows . dO^T
    float cs[2][4], cp[2][4];
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t a0, a1, a2, a3, v0, v1, v2, v3;
            ldsm_x4(kn[k] ^ (uint32_t)(s2 << 5), a0, a1, a2, a3);
            ldsm_x4((kn[k] + kVOff) ^ (uint32_t)(s2 << 5), v0, v1, v2, v3);
            if (s2 == 0) {
                mma16816_z(cs[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
                mma16816_z(cp[k], v0, v1, v2, v3, U[k].df[s2][0], U[k].df[s2][1]);
            } else {
                mma16816(cs[k], a0, a1, a2, a3, U[k].qf[s2][0], U[k].qf[s2][1]);
                mma16816(cp[k], v0, v1, v2, v3, U[k].df[s2][0], U[k].df[s2][1]);
            }
        }
    }
    // rows b (c0, c1) and a (c2, c3) of rung k0 + p for query q of each pair
    const int p = L.g8 & 3;
    const TC tc = lds_tc(S.tc + (uint32_t)(min(k0 + p, nr - 1) * 8));
    const bool rung_ok = L.useful && p < np;
    const float t = tc.t, omt = 1.f - tc.t;
    uint32_t bq[2][2], ad[2][2], ap[2][2];
    float dt = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = x.i0 + u0 + 2 * k + L.q;
        const bool ok = rung_ok && U[k].qok && i >= tc.c;
        const float2 sb = f2(cs[k][0], cs[k][1]), sa = f2(cs[k][2], cs[k][3]);
        const float2 db = f2(cp[k][0], cp[k][1]), da = f2(cp[k][2], cp[k][3]);
        const float2 sv = __ffma2_rn(f2(t, t), sb, f2mul(f2(omt, omt), sa));
        const float2 dpv = __ffma2_rn(f2(t, t), db, f2mul(f2(omt, omt), da));
        const float2 pe = ok ? f2(fast_exp2(fmaf(sv.x, P.sl2, -U[k].lse2.x)),
                                  fast_exp2(fmaf(sv.y, P.sl2, -U[k].lse2.y)))
                             : f2(0.f, 0.f);
        const float2 ds = f2mul(f2mul(pe, f2(dpv.x - U[k].D.x, dpv.y - U[k].D.y)), f2(P.scale, P.scale));
        // dL/dt: ds (s_b - s_a) (raw scores, scale folded into ds) + p (dp_b - dp_a);
        // at t = 0 the derivative is one-sided and zero while row b = i - n - 1
        // lies before the sequence start (i = ceil(d) = n)
        const float2 g = __ffma2_rn(ds, f2(sb.x - sa.x, sb.y - sa.y), f2mul(pe, f2(db.x - da.x, db.y - da.y)));
        if (t > 0.f || i > tc.c) dt += g.x + g.y;
        ad[k][0] = pack_bf16(ds.x * t, ds.y * t);        // row b
        ad[k][1] = pack_bf16(ds.x * omt, ds.y * omt);    // row a
        ap[k][0] = pack_bf16(pe.x * t, pe.y * t);
        ap[k][1] = pack_bf16(pe.x * omt, pe.y * omt);
        bq[k][0] = movm_t(ad[k][0]);
        bq[k][1] = movm_t(ad[k][1]);
    }
    // dL/dt of rung k0 + p: the threads g8 in {p, p + 4}, every tig
    dt += __shfl_xor_sync(kFull, dt, 1);
    dt += __shfl_xor_sync(kFull, dt, 2);
    dt += __shfl_xor_sync(kFull, dt, 16);
    if (lane < 16 && tig == 0 && p < np) dt_w[k0 + p] += dt;
    // dQhat^T += Khat_rows^T . dS^T
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(kt[k] ^ (uint32_t)(j << 5), a0, a1, a2, a3);
            mma16816(U[k].dq[j], a0, a1, a2, a3, bq[k][0], bq[k][1]);
        }
    }
    // dKhat_rows = dS . Qhat, dV_rows = P . dO.  Rows base + m, m = 2k + e +
    // kind: lanes 0..15 (e = 0) hold m = 0, 1 (pair 0) and 2, 3 (pair 1),
    // lanes 16..31 hold m = 1, 2 and 3, 4; the shared rows are summed across
    // the two halves of the warp before the reduction.
    const int base = x.i0 + u0 - S.r[min(k0 + p, nr - 1)].n - 1;
    const size_t rb = (size_t)x.b * P.a.T * kHkv + x.g;
    const bool A = L.is_a;
    bool okx = p < np, oky = p < np, okz = p < np && A;
    float* px = acc_row(P.dk_acc, rb, base + (A ? 0 : 3), P.a.T, tig, okx);
    float* py = acc_row(P.dk_acc, rb, base + (A ? 1 : 4), P.a.T, tig, oky);
    float* pz = acc_row(P.dk_acc, rb, base + 2, P.a.T, tig, okz);
#pragma unroll
    for (int tensor = 0; tensor < 2; ++tensor) {
        const long long off = tensor == 0 ? 0 : P.dv_off;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float m0[4], m1[4];
            if (tensor == 0) {
                mma1688_z(m0, ad[0][0], ad[0][1], U[0].qm[c]);
                mma1688_z(m1, ad[1][0], ad[1][1], U[1].qm[c]);
            } else {
                mma1688_z(m0, ap[0][0], ap[0][1], U[0].dm[c]);
                mma1688_z(m1, ap[1][0], ap[1][1], U[1].dm[c]);
            }
            const float2 u0b = f2(m0[0], m0[1]), u0a = f2(m0[2], m0[3]);
            const float2 u1b = f2(m1[0], m1[1]), u1a = f2(m1[2], m1[3]);
            const float2 r1 = shfl2_xor(A ? u1a : u0b, 16);
            const float2 r2 = shfl2_xor(u0a, 16);
            const float2 vx = A ? u0b : f2add(u1b, r1);
            const float2 vy = A ? f2add(u0a, r1) : u1a;
            const float2 vz = f2add(u1b, r2);
            red_v2(px + off + 8 * c, vx.x, vx.y, okx);
            red_v2(py + off + 8 * c, vy.x, vy.y, oky);
            red_v2(pz + off + 8 * c, vz.x, vz.y, okz);
        }
    }
}

// dQ = R(i)^T dQhat of unit k, staged transposed in this warp's buffer for
// the warp's coalesced 16-byte stores.
__device__ __forceinline__ void store_dq(const BwdParams& P, const Tile& x, int u, int k, uint32_t obuf,
                                         const BLane& L, int lane, BUnit& U) {
    const int g8 = lane >> 2, tig = lane & 3;
    if (P.rope) {
        const int iq = min(x.i0 + u + (tig >> 1), P.a.T - 1);
        const float2* tr = P.rope + (size_t)iq * kPairs;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // dimensions m = 16 j + 8 h + g8 (element 2 h, 2 h + 1) and m + 32 (m tile j + 2)
                const float2 cs = __ldg(tr + 16 * j + 8 * h + g8);
                const float x0 = U.dq[j][2 * h], x1 = U.dq[j][2 * h + 1];
                const float y0 = U.dq[j + 2][2 * h], y1 = U.dq[j + 2][2 * h + 1];
                U.dq[j][2 * h] = cs.x * x0 + cs.y * y0;
                U.dq[j][2 * h + 1] = cs.x * x1 + cs.y * y1;
                U.dq[j + 2][2 * h] = cs.x * y0 - cs.y * x0;
                U.dq[j + 2][2 * h + 1] = cs.x * y1 - cs.y * x1;
            }
    }
    const uint32_t buf = obuf + (uint32_t)(k * 8 * ROWB);
    uint32_t r[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        r[j][0] = pack_bf16(U.dq[j][0], U.dq[j][1]);
        r[j][1] = pack_bf16(U.dq[j][2], U.dq[j][3]);
    }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
        stsm_x4_t(buf + L.ob[jj], r[2 * jj][0], r[2 * jj][1], r[2 * jj + 1][0], r[2 * jj + 1][1]);
}

__device__ void bwd_consumer(const BwdParams& P, const Smem& S, int warp, int lane, float* dt_w, uint32_t stg) {
    int wcount = 0, gcount = 0, qcount = 0;
    const int u0 = 4 * warp;
    const BLane L = make_blane(lane, u0, P.a.W, P.win_rows);
    const uint32_t obuf = S.obuf + (uint32_t)(warp * kObufBytes);
    const int nr = max(P.a.nr, 1);
    // the accumulators are zeroed by the launch before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    Tile x = decode(P, blockIdx.x);
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x) {
        BUnit U[2];
        int kt;
        {
            if (!warp_wait(bar_full_q(S), qcount & 1, S.abort_flag)) goto fail;
            if (!warp_wait(bar_full_w(S), wcount & 1, S.abort_flag)) goto fail;
            const int nq = min(TQ, P.a.T - x.i0);
#pragma unroll
            for (int k = 0; k < 2; ++k) start_bunit(P, S, x, nq, u0 + 2 * k, lane, U[k]);
            __syncwarp();
            mbar_arrive_if(bar_empty_q(S), lane == 0);
            ++qcount;
            bwd_window_tile<true>(P, S.win, x, u0, 0, L, U, stg);
            for (int wt = 1; wt < P.nwt; ++wt) bwd_window_tile<false>(P, S.win, x, u0, wt, L, U, stg);
            kt = *S.kt;
            __syncwarp();
            mbar_arrive_if(bar_empty_w(S), lane == 0);
            ++wcount;
        }
        const Tile nx = next_tile(P, x);
        for (int k0 = 0; k0 < kt; k0 += RPG) {
            const int slot = gcount & (NGS - 1);
            if (!warp_wait(bar_full_g(S, slot), (gcount / NGS) & 1, S.abort_flag)) goto fail;
            bwd_rung_tile(P, S, S.rung + (uint32_t)slot * kGroupSlotBytes, x, k0, min(RPG, kt - k0), nr, u0, L,
                          U, dt_w);
            __syncwarp();
            mbar_arrive_if(bar_empty_g(S, slot), lane == 0);
            ++gcount;
        }
        __syncwarp();  // the previous tile's rows have been read back
#pragma unroll
        for (int k = 0; k < 2; ++k) store_dq(P, x, u0 + 2 * k, k, obuf, L, lane, U[k]);
        __syncwarp();
        {
            // read back so that each 16-byte store covers one query's four
            // heads, 512 contiguous bytes of dQ
            const int cc = lane & 7, h = lane >> 3;
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int iq = x.i0 + u0 + 2 * k + e, rr = 4 * e + h;
                    uint4* dst = reinterpret_cast<uint4*>(P.dq + (((size_t)x.b * P.a.T + iq) * kHq + x.g * kG + h) * kD);
                    if (iq < P.a.T)
                        dst[cc] = lds_u4(obuf + (uint32_t)(k * 8 * ROWB) + (uint32_t)rr * ROWB +
                                         (uint32_t)(((cc ^ rr) & 7) << 4));
                }
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

__global__ void __launch_bounds__(NTHREADS, 1) bwd_mma_kernel(const __grid_constant__ BwdParams P) {
    extern __shared__ unsigned char smem_raw[];
    // the finish kernel may be scheduled now; it waits for this grid before it
    // reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const Smem S = ring_setup(P.a, NCW, BwdParams::kQMaps * kQTileBytes, P.win_slot_bytes, smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // per consumer warp dL/dt sums, after the output staging buffers
    float* dt_all = reinterpret_cast<float*>(smem_raw + (S.obuf + NCW * kObufBytes - smem_u32(smem_raw)));
    for (int i = threadIdx.x; i < NCW * SFA_MAX_RUNGS; i += blockDim.x) dt_all[i] = 0.f;
    // per consumer warp 8 KB of window-reduction staging: dK then dV, each two
    // halves of 32 dimensions x 16 rows in the 128-byte swizzle of the
    // reduction maps (1024-byte aligned)
    const uint32_t stg0 = (smem_u32(dt_all + NCW * SFA_MAX_RUNGS) + 1023u) & ~1023u;
    __syncthreads();
    if (warp == NCW) {
        if (lane == 0) producer(P, S);
    } else {
        bwd_consumer(P, S, warp, lane, dt_all + warp * SFA_MAX_RUNGS, stg0 + (uint32_t)warp * 8192u);
    }
    __syncthreads();
    if (threadIdx.x < SFA_MAX_RUNGS) {
        float s = 0.f;
        for (int w = 0; w < NCW; ++w) s += dt_all[w * SFA_MAX_RUNGS + threadIdx.x];
        P.dt_part[(size_t)blockIdx.x * SFA_MAX_RUNGS + threadIdx.x] = s;
    }
}

// ------------------------------------------------------ prep and finish

// Zeroes the fp32 dK-hat and dV accumulators and, with a RoPE table, writes
// Khat = RoPE(K) in the natural dimension order.  Thread idx of the 4 rows
// threads zeroes the 16-byte words idx + n * 4 rows (n = 0..3) of each
// accumulator (a warp's stores cover 512 contiguous bytes); for the rotation
// four threads take a row (b, j, g), thread a the pairs 8a .. 8a + 7.
__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(const __nv_bfloat16* __restrict__ k,
                                                                const float2* __restrict__ rope,
                                                                __nv_bfloat16* __restrict__ khat,
                                                                float* __restrict__ dk_acc,
                                                                float* __restrict__ dv_acc, unsigned rows,
                                                                unsigned T) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const unsigned idx = blockIdx.x * kPrepThreads + threadIdx.x;
    const unsigned row = idx >> 2, a = idx & 3;
    if (row >= rows) return;
    {
        const size_t nthreads = (size_t)rows * 4;
        float4* zk = reinterpret_cast<float4*>(dk_acc) + idx;
        float4* zv = reinterpret_cast<float4*>(dv_acc) + idx;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            zk[n * nthreads] = z;
            zv[n * nthreads] = z;
        }
    }
    if (!rope) return;
    const unsigned j = (row / kHkv) % T;
    const __nv_bfloat16* kr = k + (size_t)row * kD;
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(kr + 8 * a));
    const uint4 yv = __ldg(reinterpret_cast<const uint4*>(kr + 32 + 8 * a));
    const float4* cs = reinterpret_cast<const float4*>(rope + (size_t)j * kPairs + 8 * a);
    uint32_t xo[4], yo[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float4 t = __ldg(cs + c);
        const float2 x = unpack_bf16(u4_get(xv, c));
        const float2 y = unpack_bf16(u4_get(yv, c));
        xo[c] = rope_x(x, y, t);
        yo[c] = rope_y(x, y, t);
    }
    __nv_bfloat16* out = khat + (size_t)row * kD;
    *reinterpret_cast<uint4*>(out + 8 * a) = make_uint4(xo[0], xo[1], xo[2], xo[3]);
    *reinterpret_cast<uint4*>(out + 32 + 8 * a) = make_uint4(yo[0], yo[1], yo[2], yo[3]);
}

// dK = R(j)^T dKhat and dV, bf16, eight threads per row (pairs 4q .. 4q + 3).
// Block 0 reduces dL/dt over the CTA partials instead: warp w takes the rungs
// w, w + 8, ..., lanes sum strided partials in fp64 and a fixed-order
// butterfly finishes each rung, so the result does not depend on timing.
__global__ void __launch_bounds__(kFinishThreads) bwd_finish_mma_kernel(
    const LayerArgs a, const float* __restrict__ dk_acc, const float* __restrict__ dv_acc,
    const float2* __restrict__ rope, __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
    const float* __restrict__ dt_part, int nparts, float* __restrict__ dalpha, float* __restrict__ dtheta,
    unsigned rows) {
    // launched as a dependent of the main kernel: its results must be complete
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (blockIdx.x == 0) {
        __shared__ double per_rung[SFA_MAX_RUNGS];
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int r = warp; r < SFA_MAX_RUNGS; r += kFinishThreads / 32) {
            double s = 0.0;
            if (r < a.nr)
                for (int p = lane; p < nparts; p += 32) s += (double)dt_part[(size_t)p * SFA_MAX_RUNGS + r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
            if (lane == 0) per_rung[r] = r < a.nr ? (double)a.r[r].f * s : 0.0;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            double total = 0.0;
            for (int r = 0; r < a.nr; ++r) total += per_rung[r];
            const double al = (double)a.alpha;
            *dalpha = (float)total;
            *dtheta = (float)(total * (al - 0.5) * (1.5 - al));
        }
        return;
    }
    // eight threads per row: thread q takes dimensions 4q .. 4q + 3 and their
    // rotation partners 32 + 4q .. 32 + 4q + 3 (a warp's loads cover 128
    // contiguous bytes of a row half, its stores 64)
    const size_t idx = (size_t)(blockIdx.x - 1) * kFinishThreads + threadIdx.x;
    const size_t row = idx >> 3;
    const int q = (int)(idx & 7);
    if (row >= rows) return;
    const size_t base = row * kD + 4 * q;
    float4 x = *reinterpret_cast<const float4*>(dk_acc + base);
    float4 y = *reinterpret_cast<const float4*>(dk_acc + base + 32);
    const float4 vx = *reinterpret_cast<const float4*>(dv_acc + base);
    const float4 vy = *reinterpret_cast<const float4*>(dv_acc + base + 32);
    if (rope) {
        const unsigned j = (unsigned)((row / kHkv) % (unsigned)a.T);
        const float4* cs = reinterpret_cast<const float4*>(rope + (size_t)j * kPairs + 4 * q);
        // pairs 4q, 4q + 1 in t0 and 4q + 2, 4q + 3 in t1: (cos, sin) each
        const float4 t0 = __ldg(cs), t1 = __ldg(cs + 1);
        const float4 x0 = x, y0 = y;
        x = make_float4(t0.x * x0.x + t0.y * y0.x, t0.z * x0.y + t0.w * y0.y, t1.x * x0.z + t1.y * y0.z,
                        t1.z * x0.w + t1.w * y0.w);
        y = make_float4(t0.x * y0.x - t0.y * x0.x, t0.z * y0.y - t0.w * x0.y, t1.x * y0.z - t1.y * x0.z,
                        t1.z * y0.w - t1.w * x0.w);
    }
    *reinterpret_cast<uint2*>(dk + base) = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
    *reinterpret_cast<uint2*>(dk + base + 32) = make_uint2(pack_bf16(y.x, y.y), pack_bf16(y.z, y.w));
    *reinterpret_cast<uint2*>(dv + base) = make_uint2(pack_bf16(vx.x, vx.y), pack_bf16(vx.z, vx.w));
    *reinterpret_cast<uint2*>(dv + base + 32) = make_uint2(pack_bf16(vy.x, vy.y), pack_bf16(vy.z, vy.w));
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct BwdWorkspace {
    __nv_bfloat16* khat;  // only with RoPE
    float* dk_acc;
    float* dv_acc;
    float* dt_part;
};

BwdWorkspace carve(const LayerArgs& a, bool rope, void* base) {
    const size_t nkv = (size_t)a.B * a.T * kHkv * kD;
    char* p = static_cast<char*>(base);
    BwdWorkspace w;
    w.khat = nullptr;
    if (rope) {
        w.khat = reinterpret_cast<__nv_bfloat16*>(p);
        p += align256(nkv * sizeof(__nv_bfloat16));
    }
    w.dk_acc = reinterpret_cast<float*>(p);
    p += align256(nkv * sizeof(float));
    w.dv_acc = reinterpret_cast<float*>(p);
    p += align256(nkv * sizeof(float));
    w.dt_part = reinterpret_cast<float*>(p);
    return w;
}

}  // namespace

bool bwd_mma_supported(const LayerArgs& a) { return a.W <= 30; }

size_t bwd_mma_workspace(const LayerArgs& a, bool rope) {
    const size_t nkv = (size_t)a.B * a.T * kHkv * kD;
    return (rope ? align256(nkv * sizeof(__nv_bfloat16)) : 0) + 2 * align256(nkv * sizeof(float)) +
           align256((size_t)kMaxGrid * SFA_MAX_RUNGS * sizeof(float));
}

// 4-D map over an fp32 accumulator [B][T][2][64] (innermost first: d, head, t,
// b), box of 32 dimensions x 1 head x 16 positions, 128-byte swizzle: the
// target of the window tensor reductions.
static bool encode_red(CUtensorMap* m, const float* base, int B, int T) {
    auto fn = ring::encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kHkv, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 4, (cuuint64_t)kHkv * kD * 4, (cuuint64_t)T * kHkv * kD * 4};
    const cuuint32_t box[4] = {32u, 1u, 16u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_bwd_mma(const LayerArgs& a, const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, const float2* rope, void* dq, void* dk, void* dv,
                           float* dalpha, float* dtheta, void* ws, unsigned* status, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = sm_count(dev, &e);
    if (e != cudaSuccess) return e;
    const BwdWorkspace w = carve(a, rope != nullptr, ws);
    const unsigned rows = (unsigned)a.B * (unsigned)a.T * kHkv;
    {
        // zeroes the accumulators (and rotates K with RoPE on)
        const unsigned blocks = (rows * 4 + kPrepThreads - 1) / kPrepThreads;
        bwd_prep_kernel<<<blocks, kPrepThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(k), rope, w.khat,
                                                        w.dk_acc, w.dv_acc, rows, (unsigned)a.T);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
    }
    const void* khat = rope ? static_cast<const void*>(w.khat) : k;
    BwdParams P;
    std::memset(&P, 0, sizeof(P));
    P.a = a;
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.dq = static_cast<__nv_bfloat16*>(dq);
    P.o = static_cast<const __nv_bfloat16*>(o);
    P.dO = static_cast<const __nv_bfloat16*>(dO);
    P.lse = lse;
    P.rope = rope;
    P.dk_acc = w.dk_acc;
    P.dv_acc = w.dv_acc;
    P.dv_off = w.dv_acc - w.dk_acc;
    P.dt_part = w.dt_part;
    P.status = status;
    P.sl2 = a.scale * kLog2e;
    P.scale = a.scale;
    P.ntq = (a.T + TQ - 1) / TQ;
    P.ntiles = a.B * P.ntq * kHkv;
    P.win_rows = TQ + a.W;
    P.nwt = (a.W + 4 + 15) / 16;
    P.win_region = round1k((unsigned)P.win_rows * ROWB);
    P.win_slot_bytes = 2 * P.win_region + round1k(TQ * TABB);
    if (!encode_rows(&P.kmap_w, khat, a.B, a.T, P.win_rows) || !encode_rows(&P.vmap_w, v, a.B, a.T, P.win_rows) ||
        !encode_red(&P.dkred, P.dk_acc, a.B, a.T) || !encode_red(&P.dvred, P.dv_acc, a.B, a.T) ||
        !encode_heads(&P.qmaps[0], q, a.B, a.T, TQ) ||
        !encode_heads(&P.qmaps[1], dO, a.B, a.T, TQ) || !encode_heads(&P.qmaps[2], o, a.B, a.T, TQ))
        return cudaErrorInvalidValue;
    if (rope && !encode_table(&P.tabmap, rope, a.T)) return cudaErrorInvalidValue;
    for (int p = 0; p < RPG; ++p) {
        const int r = RUNG_ROWS + 2 * p;
        if (!encode_rows(&P.kmap_r[p], khat, a.B, a.T, r) || !encode_rows(&P.vmap_r[p], v, a.B, a.T, r))
            return cudaErrorInvalidValue;
    }
    const size_t smem = 1024 + kHeaderBytes + BwdParams::kQMaps * (size_t)kQTileBytes + (size_t)P.win_slot_bytes +
                        NGS * (size_t)kGroupSlotBytes + NCW * (size_t)kObufBytes + kDtBytes + 1024 + NCW * 8192;
    static CtxSetting configured_smem[64];
    if (!ctx_setting_holds(configured_smem[dev & 63], smem)) {
        e = cudaFuncSetAttribute(bwd_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        ctx_setting_done(configured_smem[dev & 63], smem);
    }
    // CTAs per SM for this shared-memory size (looked up once per device and
    // size, so that no runtime query runs while a stream is being captured)
    static int occ_per_sm[64];
    static size_t occ_smem[64];
    if (occ_smem[dev & 63] != smem) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bwd_mma_kernel, NTHREADS, smem);
        if (e != cudaSuccess) return e;
        occ_per_sm[dev & 63] = n;
        occ_smem[dev & 63] = smem;
    }
    int per_sm = occ_per_sm[dev & 63];
    if (per_sm < 1) per_sm = 1;
    long long grid = (long long)sms * per_sm;
    if (grid > P.ntiles) grid = P.ntiles;
    if (grid > kMaxGrid) grid = kMaxGrid;
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
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, bwd_mma_kernel, P);
    if (e != cudaSuccess) return e;
    count_launch();
    {
        const unsigned row_blocks = (unsigned)(((size_t)rows * 8 + kFinishThreads - 1) / kFinishThreads);
        cudaLaunchConfig_t fc = {};
        fc.gridDim = dim3(row_blocks + 1);
        fc.blockDim = dim3(kFinishThreads);
        fc.dynamicSmemBytes = 0;
        fc.stream = s;
        fc.attrs = attr;
        fc.numAttrs = 1;
        e = cudaLaunchKernelEx(&fc, bwd_finish_mma_kernel, a, (const float*)w.dk_acc, (const float*)w.dv_acc,
                               rope, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv),
                               (const float*)w.dt_part, (int)grid, dalpha, dtheta, rows);
        if (e != cudaSuccess) return e;
        count_launch();
    }
    return cudaSuccess;
}

}  // namespace sfa
