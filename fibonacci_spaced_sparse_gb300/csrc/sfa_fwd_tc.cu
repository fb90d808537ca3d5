// sfa_fwd_tc.cu -- the bf16 forward on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for windows W <= 16.
//
// The method is the attention of "Depth-Staggered Fibonacci Spacing for Sparse
// Attention" (arXiv 2606.28560), section 2 "Attended set": query i attends the
// window distances 0..W and one interpolated row per rung at d = alpha f,
// between rows i - floor(d) (weight 1 - t) and i - floor(d) - 1 (weight t);
// the offsets are shared by every query, so for a tile of consecutive queries
// each rung is ONE contiguous block of key/value rows.
//
// Two CTAs per SM, each persistent over tiles of TQ = 31 consecutive queries
// of one sequence b and one key/value head g; each holds 256 TMEM columns.
// The tile's 31 x 4 (query, head) rows are the M = 128 rows of every MMA (row
// 4 e + h, TMEM lane = row; rows 124..127 are padding).  Per tile:
//   scores   S_win = Qhat . Khat_win^T  (N = 48 key rows i0 - W .. i0 - W + 47)
//            and, per group of up to 2 rungs, S_grp = Qhat . [Khat_k]^T over
//            the group's blocks (32 rows i0 - n_k - 1 .. i0 - n_k + 30 each,
//            contiguous in shared memory: one MMA of N = 32 x rungs per K step);
//   softmax  one thread per (query, head) row reads its window band (with
//            group 0) and, per rung, the two columns of its rows b and a,
//            forms the lerped rung score (1 - t) s_a + t s_b (the score of the
//            interpolated key, by linearity), keeps an online maximum over the
//            groups (the output is rescaled in TMEM when a later group raises
//            it by more than 2^8) and writes the probabilities back over the
//            scores as bf16 pairs: the window band as computed, a rung's p
//            split onto its two rows as p t and p (1 - t), zeros elsewhere, so
//            that P_k . V_k forms the interpolated value row;
//   output   O += P . V (A from TMEM, V row-major as an MN-major operand from
//            shared memory), fp32 in TMEM; the softmax warps normalise their
//            rows by 1 / l and store them (staged in shared memory, written
//            out 512 contiguous bytes per store).
// Rung groups alternate between two TMEM areas (groups counted over the
// CTA's tiles), so the scores of the group after next are computed while the
// softmax warps work on the next one, and the two CTAs of an SM interleave on
// its tensor cores.
//
// Warp roles (8 warps): 0 loads the rung groups with TMA (keys and values,
// two buffers each); 1 issues the MMAs (the whole warp runs the sequence,
// one elected lane issues) and owns the TMEM allocation; 2-5 run the softmax
// and the output (warp w serves TMEM lanes 32 (w % 4) ..); 6-7 rotate the
// queries of each tile in shared memory (RoPE, two (query, head) rows per
// thread, into the stored dimension order of Khat) and, in a multi-layer
// call, the next layer's keys at the tile's positions; their thread 0 loads
// the queries and the window block of the next tile (two buffers each).  The
// waits sleep in the barrier (mbarrier.try_wait with a suspend-time hint).
// Every wait is bounded: a wait that gives up sets the CTA's abort flag and
// SFA_DEVSTAT_WAIT_TIMEOUT, every role then stops, the MMA warp waits for its
// last MMAs and the loading threads for their last copies before the CTA
// frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>

#include "sfa_internal.cuh"
#include "sfa_mma.cuh"
#include "sfa_ring.cuh"
#include "sfa_tc.cuh"

namespace sfa {

namespace {

using namespace mma;
using ring::kLn2;
using ring::kLog2e;
using ring::ROWB;
using ring::TABB;

constexpr int TQ = 31;            // queries per tile (x 4 heads = 124 of the 128 MMA rows)
constexpr int MROWS = 128;
constexpr int NWIN = 48;          // window block rows, N of the window scores
constexpr int NRB = 32;           // rung block rows
constexpr int GR = 2;             // rungs per group (N = 64)
constexpr int MAXW = 16;          // TQ + W rows must fit the window block
constexpr int NTHREADS = 256;     // 8 warps
constexpr int kPrepWarp0 = 6;     // warps 6, 7; 2..5 run the softmax
constexpr int kPrepThreads = 64;
constexpr float kLazy = 8.0f;     // a later group raises the row maximum only past this margin (log2 units)

constexpr int NQB = 2;            // Q buffers: the loads run one tile ahead
constexpr int NKV = 2;            // rung-group key buffers
constexpr int NV = 3;             // rung-group value buffers: a group's values load as soon as the
                                  // P V three groups back has read its buffer, early enough not
                                  // to hold up its own P V (with two, that reload showed)
constexpr uint32_t kQBytes = MROWS * ROWB;          // one Q buffer (rows 124..127 stay zero)
constexpr uint32_t kQBox = TQ * kG * ROWB;          // bytes one Q box moves (zero filled past T)
constexpr uint32_t kWinTensor = NWIN * ROWB;        // 6 KB: Khat, then V
constexpr uint32_t kRungBytes = NRB * ROWB;         // 4 KB
constexpr uint32_t kGroupBytes = GR * kRungBytes;   // 8 KB
constexpr uint32_t kStageBytes = 32 * ROWB / 2;     // one softmax warp's 32 output rows, half a row each

// TMEM columns of a CTA
constexpr uint32_t kColW = 0;     // window scores (48), then its probabilities (24 bf16 pairs)
constexpr uint32_t kColR = 48;    // two group areas of 64: scores (32 per rung), probabilities in
                                  // the first 16 of each
constexpr uint32_t kColO = 176;   // O (64)
constexpr uint32_t kTmemCols = 256;
static_assert(kColR + 2 * NRB * GR <= kColO && kColO + kD <= kTmemCols, "TMEM columns");

constexpr uint32_t kIdescWin = tc::idesc_bf16(MROWS, NWIN, false);
constexpr uint32_t kIdescPV = tc::idesc_bf16(MROWS, kD, true);

// shared memory (from a 1024-byte aligned base): the header, the Q buffers,
// the window block, the rung-group key and value blocks, the output staging
// of the four softmax warps
constexpr uint32_t kHdrBytes = 1024;
constexpr uint32_t kOffQ = kHdrBytes;
constexpr uint32_t kOffWin = kOffQ + NQB * kQBytes;
constexpr uint32_t kOffKg = kOffWin + 4 * kWinTensor;     // [NKV]; the window blocks are [2]
constexpr uint32_t kOffVg = kOffKg + NKV * kGroupBytes;   // [NV]
constexpr uint32_t kOffStage = kOffVg + NV * kGroupBytes;
constexpr uint32_t kSmemUsed = kOffStage + 4 * kStageBytes;
constexpr size_t kSmemBytes = 1024 + (size_t)kSmemUsed;
static_assert(kOffQ % 1024 == 0 && kOffWin % 1024 == 0 && kOffKg % 1024 == 0 && kOffVg % 1024 == 0 &&
                  kOffStage % 1024 == 0 && kWinTensor % 1024 == 0 && kStageBytes % 1024 == 0,
              "operand tiles on the 1024-byte swizzle period");
// two CTAs per SM: 2 x (this + the 1 KB the SM reserves per CTA) <= 228 KB
static_assert(2 * (kSmemBytes + 1024) <= 233472, "shared memory of two CTAs per SM");

// header: barriers, then the shared words, then the rung table
enum : uint32_t {
    B_QFULL = 0, B_QREADY = 8 * NQB, B_QEMPTY = 16 * NQB, B_WFULL = 24 * NQB, B_WEMPTY = B_WFULL + 16,
    B_KFULL = B_WEMPTY + 16, B_VFULL = B_KFULL + 8 * NKV,
    B_VEMPTY = B_VFULL + 8 * NV, B_SFULL = B_VEMPTY + 8 * NV, B_PFULL = B_SFULL + 16, B_OFULL = B_PFULL + 16,
    B_OFREE = B_OFULL + 8, B_DONE = B_OFREE + 8, H_TMEM = B_DONE + 8, H_ABORT = H_TMEM + 4, H_RUNGS = 256
};
static_assert(H_ABORT + 4 <= H_RUNGS && H_RUNGS + SFA_MAX_RUNGS * 12 <= kHdrBytes, "header layout");

struct TcParams {
    CUtensorMap qmap;          // Q [B][T][8][64], box 64 x 4 heads x TQ queries
    CUtensorMap kwmap, vwmap;  // Khat / V [B][T][2][64], box NWIN rows of one head
    CUtensorMap krmap, vrmap;  // box NRB rows
    LayerArgs a;
    const float2* rope;        // nullptr: Q and K are used as given
    __nv_bfloat16* o;
    float* lse;
    unsigned* status;
    const __nv_bfloat16* k_next;  // keys of the next layer (multi-layer forward) or nullptr
    __nv_bfloat16* khat_next;
    float sl2;                 // softmax scale x log2 e
    int ntq, ntiles;
};

struct Tile {
    int b, g, i0;
    int kt;   // rungs some query of the tile uses
    int ng;   // groups: ceil(kt / 2), at least 1 (group 0 also carries the window)
};

struct SR {
    int n;
    float t;
    int c;
};

struct Sm {
    uint32_t base;         // shared address of the header
    unsigned char* hdr;    // generic pointer to the header
    __device__ uint32_t bar(uint32_t off, int i = 0) const { return base + off + 8u * (uint32_t)i; }
    __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(hdr + H_ABORT); }
    __device__ const SR* rungs() const { return reinterpret_cast<const SR*>(hdr + H_RUNGS); }
    __device__ uint32_t q(int i) const { return base + kOffQ + (uint32_t)i * kQBytes; }
    __device__ uint32_t win(int i) const { return base + kOffWin + (uint32_t)i * 2 * kWinTensor; }
    __device__ uint32_t kg(int i) const { return base + kOffKg + (uint32_t)i * kGroupBytes; }
    __device__ uint32_t vg(int i) const { return base + kOffVg + (uint32_t)i * kGroupBytes; }
    __device__ uint32_t stage(int q) const { return base + kOffStage + (uint32_t)q * kStageBytes; }
};

// Tile n of this CTA: blockIdx.x + n gridDim.x, ordered (b, query tile, g).
__device__ __forceinline__ bool tile_of(const TcParams& P, const Sm& S, int n, Tile& x) {
    const long long t = (long long)blockIdx.x + (long long)n * gridDim.x;
    if (t >= P.ntiles) return false;
    x.g = (int)(t % kHkv);
    const int rest = (int)(t / kHkv);
    x.i0 = (rest % P.ntq) * TQ;
    x.b = rest / P.ntq;
    // kept rungs are sorted by distance, so by ceiling: those that some query of
    // the tile uses (i0 + TQ - 1 >= ceil d) form a prefix
    const SR* r = S.rungs();
    int kt = 0;
    while (kt < P.a.nr && r[kt].c <= x.i0 + TQ - 1) ++kt;
    x.kt = kt;
    x.ng = max((kt + GR - 1) / GR, 1);
    return true;
}

__device__ __forceinline__ int group_rungs(const Tile& x, int grp) { return max(0, min(GR, x.kt - GR * grp)); }

__device__ __forceinline__ void give_up(const TcParams& P, const Sm& S) {
    *S.abort_flag() = 1;
    if (P.status) atomicOr(P.status, SFA_DEVSTAT_WAIT_TIMEOUT);
}

// ------------------------------------------------------------- loader

__device__ __forceinline__ void load_q(const TcParams& P, const Sm& S, int qb, const Tile& x) {
    const uint32_t full = S.bar(B_QFULL, qb);
    mbar_arrive_expect_tx(full, kQBox);
    tma_load_4d(S.q(qb), &P.qmap, 0, x.g * kG, x.i0, x.b, full);
}

// The rung blocks of group grp of tile x (key or value rows) into `dst`; a
// group without rungs (the window alone) completes its phase at once.
__device__ __forceinline__ void load_group(const TcParams& P, const Sm& S, const CUtensorMap* map, uint32_t dst,
                                           uint32_t full, const Tile& x, int grp) {
    const int nr = group_rungs(x, grp);
    const SR* r = S.rungs();
    mbar_arrive_expect_tx(full, (uint32_t)nr * kRungBytes);
    for (int k = 0; k < nr; ++k)
        tma_load_4d(dst + (uint32_t)k * kRungBytes, map, 0, x.g, x.i0 - r[GR * grp + k].n - 1, x.b, full);
}

// One lane: the rung groups of every tile (keys, values).  Every load waits
// for its buffer to be released, and a release depends only on loads issued
// earlier in this order (and on the window and query loads, which do not wait
// for any group load), so the order cannot deadlock.
__device__ void loader(const TcParams& P, const Sm& S) {
    volatile int* abort_flag = S.abort_flag();
    // Khat is written by the launch before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int kl = 0, vl = 0;  // group loads issued so far
    Tile x;
    bool failed = false;
    for (int n = 0; !failed && tile_of(P, S, n, x); ++n) {
        // group G (counted over the CTA's tiles) uses key buffer G % NKV and value buffer G % NV
        for (int grp = 0; grp < x.ng; ++grp) {
            const int kb = kl % NKV;
            // the key buffer is free once the scores that read it are complete
            // (key buffer kb and score area kb go together: NKV = 2); their
            // next phase needs the keys this lane has yet to load
            if (!mbar_wait_sleep(S.bar(B_SFULL, kb), (uint32_t)((kl / NKV) & 1) ^ 1u, abort_flag)) {
                failed = true;
                break;
            }
            load_group(P, S, &P.krmap, S.kg(kb), S.bar(B_KFULL, kb), x, grp);
            ++kl;
            const int vb = vl % NV;
            if (!mbar_wait_sleep(S.bar(B_VEMPTY, vb), (uint32_t)((vl / NV) & 1) ^ 1u, abort_flag)) {
                failed = true;
                break;
            }
            load_group(P, S, &P.vrmap, S.vg(vb), S.bar(B_VFULL, vb), x, grp);
            ++vl;
        }
    }
    if (failed) {
        give_up(P, S);
        // no copy of this CTA may land after it exits: wait (bounded) for the
        // last announced phase of every buffer (at most one copy per buffer is
        // ever in flight)
        for (int m = max(0, kl - NKV); m < kl; ++m)
            (void)mbar_wait_sleep(S.bar(B_KFULL, m % NKV), (m / NKV) & 1, nullptr);
        for (int m = max(0, vl - NV); m < vl; ++m)
            (void)mbar_wait_sleep(S.bar(B_VFULL, m % NV), (m / NV) & 1, nullptr);
    }
}

// ------------------------------------------------------------- MMA issue

// Scores of group G (counted over the CTA's tiles; group grp of tile x):
// S_G = Qhat . [Khat_k]^T into group area G % 2, keys from buffer G % 2.
__device__ __forceinline__ bool issue_scores(const Sm& S, uint32_t tmem, uint32_t qa, const Tile& x, int grp, int G,
                                             volatile int* abort_flag) {
    const int b = G & 1, kb = G % NKV;
    if (!warp_wait_sleep(S.bar(B_KFULL, kb), (G / NKV) & 1, abort_flag)) return false;
    tc::fence_after();
    const int nr = group_rungs(x, grp);
    if (nr > 0) {
        const uint32_t idesc = tc::idesc_bf16(MROWS, NRB * nr, false);
        const uint32_t d = tmem + kColR + (uint32_t)(b * NRB * GR);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            tc::mma_ss_warp(d, tc::desc_kmajor(qa + 32 * ks), tc::desc_kmajor(S.kg(kb) + 32 * ks), idesc, ks > 0);
    }
    tc::commit_warp(S.bar(B_SFULL, b));
    return true;
}

// The whole warp (one elected lane issues).  Groups alternate between two TMEM areas, so the scores of group
// G + 2 are issued right after O += P V of group G, while the softmax warps
// work on group G + 1.  Per tile: the window scores with the scores of its
// first two groups, then per group its P V (with the window's for group 0)
// and the scores of the group two on.  The tensor core runs the MMAs of one
// thread in issue order, so scores that overwrite an area follow the P V
// that read its probabilities, and a commit after them also covers it.
__device__ void mma_issuer(const TcParams& P, const Sm& S, uint32_t tmem) {
    volatile int* abort_flag = S.abort_flag();
    int G0 = 0;  // first group of the tile
    Tile x;
    bool ok = true;
    // a tile's descriptor takes a few dependent shared-memory reads (the
    // kept rungs it uses) and two divisions: the next one is worked out
    // while the tensor core runs the current tile's first scores, not at the
    // tile boundary, where its latency would hold back the next scores
    bool have = tile_of(P, S, 0, x);
    for (int n = 0; ok && have; ++n) {
        const int qb = n % NQB;
        const uint32_t qa = S.q(qb);
        if (!warp_wait_sleep(S.bar(B_QREADY, qb), (n / NQB) & 1, abort_flag) ||
            !warp_wait_sleep(S.bar(B_WFULL, n & 1), (n >> 1) & 1, abort_flag)) {
            ok = false;
            break;
        }
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            tc::mma_ss_warp(tmem + kColW, tc::desc_kmajor(qa + 32 * ks), tc::desc_kmajor(S.win(n & 1) + 32 * ks), kIdescWin,
                       ks > 0);
        const int first = min(2, x.ng);
        for (int j = 0; j < first && ok; ++j) ok = issue_scores(S, tmem, qa, x, j, G0 + j, abort_flag);
        if (!ok) break;
        if (x.ng <= 2) tc::commit_warp(S.bar(B_QEMPTY, qb));
        Tile xn;
        const bool more = tile_of(P, S, n + 1, xn);
        for (int grp = 0; grp < x.ng; ++grp) {
            const int G = G0 + grp, b = G & 1, vb = G % NV;
            if (!warp_wait_sleep(S.bar(B_PFULL, b), (G >> 1) & 1, abort_flag) ||
                (grp == 0 && !warp_wait_sleep(S.bar(B_OFREE), (n & 1) ^ 1, abort_flag)) ||
                !warp_wait_sleep(S.bar(B_VFULL, vb), (G / NV) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc::fence_after();
            const uint32_t d = tmem + kColO;
            if (grp == 0) {
#pragma unroll
                for (int ks = 0; ks < NWIN / 16; ++ks)
                    tc::mma_ts_warp(d, tmem + kColW + 8 * ks, tc::desc_mnmajor(S.win(n & 1) + kWinTensor + 2048 * ks),
                               kIdescPV, ks > 0);
                tc::commit_warp(S.bar(B_WEMPTY, n & 1));
            }
            const int nr = group_rungs(x, grp);
            const uint32_t area = tmem + kColR + (uint32_t)(b * NRB * GR);
            for (int k = 0; k < nr; ++k)
#pragma unroll
                for (int ks = 0; ks < NRB / 16; ++ks)
                    tc::mma_ts_warp(d, area + NRB * k + 8 * ks, tc::desc_mnmajor(S.vg(vb) + kRungBytes * k + 2048 * ks),
                               kIdescPV, 1);
            tc::commit_warp(S.bar(B_VEMPTY, vb));
            if (grp + 2 < x.ng) {
                if (!issue_scores(S, tmem, qa, x, grp + 2, G + 2, abort_flag)) {
                    ok = false;
                    break;
                }
                if (grp + 3 >= x.ng) tc::commit_warp(S.bar(B_QEMPTY, qb));
            }
        }
        if (ok) tc::commit_warp(S.bar(B_OFULL));
        G0 += x.ng;
        x = xn;
        have = more;
    }
    if (!ok && (threadIdx.x & 31) == 0) give_up(P, S);
    // TMEM is freed only after every MMA issued has completed
    tc::commit_warp(S.bar(B_DONE));
    (void)warp_wait_sleep(S.bar(B_DONE), 0, nullptr);
}

// ------------------------------------------------------------- queries and next keys

// Qhat of row r (query e = r / 4, head r % 4) of a Q buffer, rotated in place
// at position i0 + e and written in the stored dimension order of Khat: the
// pair (8c + 2w + hh, + 32) of natural chunks c and 4 + c goes to word c of
// stored chunks w and 4 + w (kdim_of in sfa_fwd_mma.cu), so that every score
// is the same dot product as with the natural order.
// The (cos, sin) rows come from the RoPE table in global memory (L1 and L2
// serve them: the four heads of a query read the same row).
__device__ __forceinline__ void rotate_q_row(uint32_t qbuf, const float4* tab, int r) {
    const uint32_t row = qbuf + (uint32_t)r * ROWB;
    const float4* trow = tab + (r >> 2) * (TABB / 16);
    const int sw = r & 7;
    uint4 in[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) in[c] = ring::lds_u4(row + (uint32_t)((c ^ sw) << 4));
    uint32_t xo[4][4], yo[4][4];  // [stored chunk w][word c]
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float4 cs = __ldg(trow + 4 * c + w);
            const float2 xv = unpack_bf16(ring::u4_get(in[c], w)), yv = unpack_bf16(ring::u4_get(in[4 + c], w));
            xo[w][c] = ring::rope_x(xv, yv, cs);
            yo[w][c] = ring::rope_y(xv, yv, cs);
        }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (uint32_t)((w ^ sw) << 4)),
                     "r"(xo[w][0]), "r"(xo[w][1]), "r"(xo[w][2]), "r"(xo[w][3])
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (uint32_t)(((4 + w) ^ sw) << 4)),
                     "r"(yo[w][0]), "r"(yo[w][1]), "r"(yo[w][2]), "r"(yo[w][3])
                     : "memory");
    }
}

// The next layer's keys at the tile's positions (multi-layer forward): item
// id = 4 u + a rotates pairs 8a .. 8a + 7 of K_next[b][i0 + u][g] with the
// tile's RoPE rows, writing word a of every stored chunk of Khat_next (the
// stored order above).
__device__ __forceinline__ void rotate_next_keys(const TcParams& P, const float4* tab, const Tile& x, int id) {
    const int u = id >> 2, a = id & 3;
    const int pos = x.i0 + u;
    if (u >= TQ || pos >= P.a.T) return;
    const size_t rowi = ((size_t)x.b * P.a.T + pos) * kHkv + x.g;
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(P.k_next + rowi * kD + 8 * a));
    const uint4 yv = __ldg(reinterpret_cast<const uint4*>(P.k_next + rowi * kD + 32 + 8 * a));
    const float4* trow = tab + u * (TABB / 16) + 4 * a;
    uint32_t* out = reinterpret_cast<uint32_t*>(P.khat_next + rowi * kD);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float4 cs = __ldg(trow + w);
        const float2 xf = unpack_bf16(ring::u4_get(xv, w)), yf = unpack_bf16(ring::u4_get(yv, w));
        out[4 * w + a] = ring::rope_x(xf, yf, cs);
        out[16 + 4 * w + a] = ring::rope_y(xf, yf, cs);
    }
}

// The window block of tile x (Khat rows, then V rows) into window buffer wb.
__device__ __forceinline__ void load_window(const TcParams& P, const Sm& S, int wb, const Tile& x) {
    const uint32_t full = S.bar(B_WFULL, wb);
    mbar_arrive_expect_tx(full, 2 * kWinTensor);
    tma_load_4d(S.win(wb), &P.kwmap, 0, x.g, x.i0 - P.a.W, x.b, full);
    tma_load_4d(S.win(wb) + kWinTensor, &P.vwmap, 0, x.g, x.i0 - P.a.W, x.b, full);
}

// Warps 6, 7: thread pt (0..63) rotates rows pt and pt + 64 of every tile's
// queries and next-key items pt and pt + 64.  Thread 0 also loads the
// queries and the window block of each tile: those of tile n + 1 once the
// queries of tile n are rotated, as soon as their buffers are released (the
// last scores and the window P V of tile n - 1); neither wait depends on a
// load issued later.
__device__ void prep(const TcParams& P, const Sm& S, int pt, int lane) {
    volatile int* abort_flag = S.abort_flag();
    // Khat (read by the window loads) is written by the launch before this
    // one, which may also still read Khat_next
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int ql = 0, wl = 0;  // query and window loads issued (thread 0)
    bool failed = false;
    Tile x, xn;
    if (pt == 0 && tile_of(P, S, 0, x)) {
        load_q(P, S, 0, x);
        load_window(P, S, 0, x);
        ql = wl = 1;
    }
    for (int n = 0; !failed && tile_of(P, S, n, x); ++n) {
        const int qb = n % NQB;
        if (!warp_wait_sleep(S.bar(B_QFULL, qb), (n / NQB) & 1, abort_flag)) {
            failed = true;
            break;
        }
        if (P.rope) {
            // the table rows of the tile's positions i0 ..
            const float4* tab = reinterpret_cast<const float4*>(P.rope + (size_t)x.i0 * kPairs);
            const int rows = kG * min(TQ, P.a.T - x.i0);
#pragma unroll 1
            for (int r = pt; r < rows; r += kPrepThreads) rotate_q_row(S.q(qb), tab, r);
            if (P.k_next)
#pragma unroll 1
                for (int id = pt; id < 4 * TQ; id += kPrepThreads) rotate_next_keys(P, tab, x, id);
            fence_proxy_async();
        }
        __syncwarp();
        mbar_arrive_if(S.bar(B_QREADY, qb), lane == 0);
        if (pt == 0 && tile_of(P, S, n + 1, xn)) {
            const int nb = ql % NQB, wb = wl & 1;
            if (!mbar_wait_sleep(S.bar(B_QEMPTY, nb), (uint32_t)((ql / NQB) & 1) ^ 1u, abort_flag)) {
                failed = true;
            } else {
                load_q(P, S, nb, xn);
                ++ql;
                if (!mbar_wait_sleep(S.bar(B_WEMPTY, wb), (uint32_t)((wl >> 1) & 1) ^ 1u, abort_flag)) {
                    failed = true;
                } else {
                    load_window(P, S, wb, xn);
                    ++wl;
                }
            }
        }
        failed = __any_sync(0xffffffffu, failed);
    }
    if (failed) {
        if (lane == 0) give_up(P, S);
        if (pt == 0) {
            // no copy of this CTA may land after it exits
            for (int m = max(0, ql - NQB); m < ql; ++m)
                (void)mbar_wait_sleep(S.bar(B_QFULL, m % NQB), (m / NQB) & 1, nullptr);
            for (int m = max(0, wl - 2); m < wl; ++m)
                (void)mbar_wait_sleep(S.bar(B_WFULL, m & 1), (m >> 1) & 1, nullptr);
        }
    }
}

// ------------------------------------------------------------- softmax and output

// Zero columns [4 b, 4 b + 4) of this warp's lanes.
__device__ __forceinline__ void zero_block(uint32_t lane_base, uint32_t b) {
    tc::st_x4(lane_base + 4 * b, 0u, 0u, 0u, 0u);
}

// One tile of the warp's 32 rows (query e = 8 q + lane / 4, head lane % 4).
// kWide: windows W > 12 (up to 16), whose band spans 24 columns of the warp's
// window scores; otherwise 20.
template <bool kWide>
__device__ bool softmax_tile(const TcParams& P, const Sm& S, uint32_t tmem, int n, const Tile& x, int q,
                             int lane, int& sc, Tile& xn, bool& more) {
    volatile int* abort_flag = S.abort_flag();
    const int r = 32 * q + lane;           // MMA row = 4 e + h
    const int e = r >> 2, h = r & 3;       // query offset in the tile, head
    const int jj = lane >> 2;              // e - 8 q: the row's offset inside the warp's columns
    const uint32_t lb = tmem + ((uint32_t)(32 * q) << 16);
    const float sl2 = P.sl2;
    const int i = x.i0 + e;
    const bool row_ok = e < TQ && i < P.a.T;
    const SR* rt = S.rungs();
    // this lane's rung rows b = key 8 q + jj and a = key 8 q + jj + 1 fall in
    // the bf16 pairs 4 q + i1 (and 4 q + i1 + 1 when jj is odd)
    const int i1 = jj >> 1;
    const bool odd = jj & 1;
    float nm = 0.f;   // minus the running maximum, log2 units (0 on rows that do not exist)
    float l = 0.f;
    for (int grp = 0; grp < x.ng; ++grp, ++sc) {
        // group G = sc (counted over the CTA's tiles) in area G % 2
        const int G = sc, b = G & 1;
        if (!warp_wait_sleep(S.bar(B_SFULL, b), (G >> 1) & 1, abort_flag)) return false;
        tc::fence_after();
        const int nr = group_rungs(x, grp);
        const uint32_t area = lb + kColR + (uint32_t)(b * NRB * GR);
        // the scores this warp needs from TMEM, in one round trip: per rung
        // the 9 columns 8 q .. 8 q + 8 of its block, with group 0 the 24
        // window columns 8 q .. 8 q + 23
        uint32_t ra[GR][8], rb[GR];
        constexpr int NWC = kWide ? 24 : 20;  // window columns 8 q .. 8 q + NWC - 1
        uint32_t w16[16], wt[NWC - 16];
#pragma unroll
        for (int k = 0; k < GR; ++k)
            if (k < nr) {
                tc::ld_x8(area + NRB * k + 8 * q, ra[k]);
                tc::ld_x1(area + NRB * k + 8 * q + 8, rb[k]);
            }
        if (grp == 0) {
            tc::ld_x16(lb + kColW + 8 * q, w16);
            if constexpr (kWide)
                tc::ld_x8(lb + kColW + 8 * q + 16, wt);
            else
                tc::ld_x4(lb + kColW + 8 * q + 16, wt);
        }
        tc::wait_ld();
        float sr[GR];
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < GR; ++k) {
            sr[k] = -INFINITY;
            if (k >= nr) continue;
            tc::hold(ra[k]);
            tc::hold(rb[k]);
            // columns jj and jj + 1 by a three-level select on jj
            float x4[5], y2[3];
#pragma unroll
            for (int u = 0; u < 5; ++u) {
                const uint32_t lo = ra[k][u];
                const uint32_t hi = u + 4 < 8 ? ra[k][(u + 4) & 7] : rb[k];
                x4[u] = __uint_as_float((jj & 4) ? hi : lo);
            }
#pragma unroll
            for (int u = 0; u < 3; ++u) y2[u] = (jj & 2) ? x4[u + 2] : x4[u];
            const float sb = (jj & 1) ? y2[1] : y2[0];
            const float sa = (jj & 1) ? y2[2] : y2[1];
            const SR rk = rt[GR * grp + k];
            const float v = __fmaf_rn(rk.t, sb, __fmul_rn(1.f - rk.t, sa));
            sr[k] = (row_ok && i >= rk.c) ? v : -INFINITY;
            m = fmaxf(m, sr[k]);
        }
        // The P V of group G - 2, which read this area's probabilities, is
        // complete: the scores just waited for were committed after it.  The
        // P V of group G - 1 is waited for only before a rescale of O, on the
        // release of its value buffer; that barrier's next phase (group
        // G + 2) cannot begin before this warp hands over group G, so the
        // parity wait is unambiguous however many phases went by unobserved.
        if (grp == 0) {
            tc::hold(w16);
            tc::hold(wt);
            // window band: block column c (position i0 - W + c) of this lane is
            // c = 8 q + u, u < NWC; the row's entries are u = jj .. jj + W at
            // positions >= 0 (jj + W < NWC)
            float w[NWC];
            const int lo = max(jj, P.a.W - x.i0 - 8 * q);
            const int hi = row_ok ? jj + P.a.W : -1;
#pragma unroll
            for (int u = 0; u < NWC; ++u) {
                const float v = __uint_as_float(u < 16 ? w16[u] : wt[(u - 16) % (NWC - 16)]);
                w[u] = (u >= lo && u <= hi) ? v : -INFINITY;
                m = fmaxf(m, w[u]);
            }
            nm = row_ok ? -m * sl2 : 0.f;
            uint32_t pw[12];
#pragma unroll
            for (int u = 0; u < 12; ++u) {
                if (2 * u < NWC) {
                    const float p0 = fast_exp2(__fmaf_rn(w[2 * u], sl2, nm));
                    const float p1 = fast_exp2(__fmaf_rn(w[2 * u + 1], sl2, nm));
                    l += p0 + p1;
                    pw[u] = pack_bf16(p0, p1);
                } else {
                    pw[u] = 0u;  // columns past the band
                }
            }
            // window probabilities: bf16 pairs 4 q .. 4 q + 11 of the 24 the
            // window P V reads, zeros in the other three blocks of four
            const uint32_t p8[8] = {pw[0], pw[1], pw[2], pw[3], pw[4], pw[5], pw[6], pw[7]};
            tc::st_x8(lb + kColW + 4 * q, p8);
            tc::st_x4(lb + kColW + 4 * q + 8, pw[8], pw[9], pw[10], pw[11]);
#pragma unroll
            for (int s = 0; s < 3; ++s) zero_block(lb + kColW, (uint32_t)((q + 3 + s) % 6));
        } else {
            // raise the row maximum only when the group beats it by 2^8; the
            // output so far (once the P V of the group before has completed)
            // and the sum are rescaled
            const bool need = row_ok && __fmaf_rn(m, sl2, nm) > kLazy;
            if (__any_sync(kFull, need)) {
                if (!warp_wait_sleep(S.bar(B_VEMPTY, (G - 1) % NV), ((G - 1) / NV) & 1, abort_flag)) return false;
                tc::fence_after();
                const float nm_new = need ? -m * sl2 : nm;
                const float c = fast_exp2(nm_new - nm);
                l *= c;
                nm = nm_new;
                // in chunks of 8 columns: this rare path must not raise the
                // register count of the common one
#pragma unroll 1
                for (int c8 = 0; c8 < kD; c8 += 8) {
                    uint32_t o[8];
                    tc::ld_x8(lb + kColO + c8, o);
                    tc::wait_ld();
                    tc::hold(o);
#pragma unroll
                    for (int d = 0; d < 8; ++d) o[d] = __float_as_uint(__uint_as_float(o[d]) * c);
                    tc::st_x8(lb + kColO + c8, o);
                }
            }
        }
        // rung probabilities over their scores: p t on row b, p (1 - t) on
        // row a, as bf16 pairs 4 q .. 4 q + 4 of the rung's 16; the other
        // pairs zero
#pragma unroll
        for (int k = 0; k < GR; ++k) {
            if (k >= nr) break;
            const float p = fast_exp2(__fmaf_rn(sr[k], sl2, nm));
            l += p;
            const float tk = rt[GR * grp + k].t;
            const float pb = p * tk, pa = p * (1.f - tk);
            const uint32_t v1 = odd ? pack_bf16(0.f, pb) : pack_bf16(pb, pa);
            const uint32_t v2 = odd ? pack_bf16(pa, 0.f) : 0u;
            uint32_t wv[5];
#pragma unroll
            for (int u = 0; u < 5; ++u) wv[u] = u == i1 ? v1 : (u == i1 + 1 ? v2 : 0u);
            const uint32_t col = area + NRB * k;
            tc::st_x4(col + 4 * q, wv[0], wv[1], wv[2], wv[3]);
            // pair 4 q + 4 (only rows of query 8 q + 7, which exists for q < 3)
            tc::st_x4(col + 4 * ((q + 1) & 3), q < 3 ? wv[4] : 0u, 0u, 0u, 0u);
            zero_block(col, (uint32_t)((q + 2) & 3));
            zero_block(col, (uint32_t)((q + 3) & 3));
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        mbar_arrive_if(S.bar(B_PFULL, b), lane == 0);
    }
    // the next tile's descriptor, while the tile's last P V runs
    more = tile_of(P, S, n + 1, xn);
    // the output: every P V of the tile has completed.  Each lane packs its row
    if (!warp_wait_sleep(S.bar(B_OFULL), n & 1, abort_flag)) return false;
    tc::fence_after();
    // Each half of the rows (32 columns, 64 bytes) is read, normalised,
    // packed, staged and stored before the next half is read, so that few
    // registers are live and the staging buffer holds half rows: 16-byte
    // chunk c of row r at c ^ ((r / 2) % 4), which keeps both the staging
    // writes (a lane per row) and the read-back (four lanes per row) free of
    // bank conflicts.  The warp's 32 rows are 8 queries x 4 heads; a store
    // covers the 64-byte halves of 8 rows (2 queries x 4 heads).
    const uint32_t stage = S.stage(q);
    {
        // row sums are >= 1 on rows that exist (the entry at the maximum contributes 1)
        const float inv = l > 0.f ? fast_rcp(l) : 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            tc::ld_x32(lb + kColO + 32 * half, o);
            tc::wait_ld();
            tc::hold(o);
            if (half == 1) {
                // every column of O has been read: hand it back
                tc::fence_before();
                __syncwarp();
                mbar_arrive_if(S.bar(B_OFREE), lane == 0);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    w[u] = pack_bf16(__uint_as_float(o[8 * c + 2 * u]) * inv,
                                     __uint_as_float(o[8 * c + 2 * u + 1]) * inv);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (uint32_t)lane * (ROWB / 2) +
                                                                              (uint32_t)((c ^ ((lane >> 1) & 3)) << 4)),
                             "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
            }
            __syncwarp();
            const int nq = min(8, P.a.T - (x.i0 + 8 * q));     // queries of the block inside the sequence
            const int nrows = (q == 3 ? min(nq, TQ - 24) : nq) * kG;
            uint4* dst =
                reinterpret_cast<uint4*>(P.o + (((size_t)x.b * P.a.T + x.i0 + 8 * q) * kHq + x.g * kG) * kD);
            const int cc = lane & 3;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int rr = 8 * k + (lane >> 2);
                if (rr < nrows)
                    dst[(size_t)(rr >> 2) * (kHq * kD / 8) + (rr & 3) * 8 + 4 * half + cc] = ring::lds_u4(
                        stage + (uint32_t)rr * (ROWB / 2) + (uint32_t)((cc ^ ((rr >> 1) & 3)) << 4));
            }
            __syncwarp();  // the half has been read back before the next is staged
        }
    }
    if (P.lse && row_ok) P.lse[((size_t)x.b * P.a.T + i) * kHq + x.g * kG + h] = (__log2f(l) - nm) * kLn2;
    return true;
}

template <bool kWide>
__device__ void softmax(const TcParams& P, const Sm& S, uint32_t tmem, int q, int lane) {
    int sc = 0;
    Tile x;
    bool have = tile_of(P, S, 0, x);
    for (int n = 0; have; ++n) {
        Tile xn;
        bool more = false;
        if (!softmax_tile<kWide>(P, S, tmem, n, x, q, lane, sc, xn, more)) {
            if (lane == 0) give_up(P, S);
            break;
        }
        x = xn;
        have = more;
    }
}

template <bool kWide>
__global__ void __launch_bounds__(NTHREADS, 2) fwd_tc_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Sm S;
    S.base = (raw + 1023u) & ~1023u;
    S.hdr = smem_raw + (S.base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x < P.a.nr) {
        const Rung rg = P.a.r[threadIdx.x];
        reinterpret_cast<SR*>(S.hdr + H_RUNGS)[threadIdx.x] = SR{rg.n, rg.t, rg.c};
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NQB; ++i) {
            mbar_init(S.bar(B_QFULL, i), 1);
            mbar_init(S.bar(B_QREADY, i), kPrepThreads / 32);
            mbar_init(S.bar(B_QEMPTY, i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(S.bar(B_WFULL, i), 1);
            mbar_init(S.bar(B_WEMPTY, i), 1);
        }
        for (int i = 0; i < NKV; ++i) {
            mbar_init(S.bar(B_KFULL, i), 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(S.bar(B_VFULL, i), 1);
            mbar_init(S.bar(B_VEMPTY, i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(S.bar(B_SFULL, i), 1);
            mbar_init(S.bar(B_PFULL, i), 4);
        }
        mbar_init(S.bar(B_OFULL), 1);
        mbar_init(S.bar(B_OFREE), 4);
        mbar_init(S.bar(B_DONE), 1);
        *S.abort_flag() = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // rows 124..127 of the Q buffers (no query) stay zero
    if (threadIdx.x < 32 * NQB) {
        const int qb = threadIdx.x >> 5;
        const uint32_t a = S.q(qb) + (uint32_t)(TQ * kG) * ROWB + 16u * (threadIdx.x & 31);
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
    }
    fence_proxy_async();
    if (warp == 1) tc::alloc(S.base + H_TMEM, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(S.hdr + H_TMEM);
    // the next launch (the next layer) may start its prologue; it waits for
    // this grid before it touches memory
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 0) {
        if (lane == 0) loader(P, S);
    } else if (warp == 1) {
        mma_issuer(P, S, tmem);
    } else if (warp < kPrepWarp0) {
        softmax<kWide>(P, S, tmem, warp & 3, lane);
    } else {
        prep(P, S, (int)threadIdx.x - 32 * kPrepWarp0, lane);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// The mma.sync kernel (sfa_fwd_mma.cu) is the default: measured on GB300 it
// is faster for this attention (a model-shape layer, B = 32, T = 1024, W = 12,
// in a 16-layer call: 32 us against 45 us here).  Each softmax group of this
// kernel is a chain of a TMEM load, dependent selects and exponentials and
// TMEM stores on one warp per lane quarter (about 0.45 us per group of two
// rungs), and the tile's groups follow one another, so two tiles per SM do
// not fill the tensor cores (about 14 % busy).
// SFA_FORWARD_KERNEL=tc in the environment (read at every call) selects this
// kernel for windows W <= 16.
bool fwd_tc_supported(const LayerArgs& a) {
    if (a.W > MAXW) return false;
    const char* e = std::getenv("SFA_FORWARD_KERNEL");
    return e && std::strcmp(e, "tc") == 0;
}

cudaError_t launch_fwd_tc(const LayerArgs& a, const void* q, const void* khat, const void* v, const float2* rope,
                          void* o, float* lse, const void* k_next, void* khat_next, unsigned* status, bool pdl,
                          cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = ring::sm_count(dev, &e);
    if (e != cudaSuccess) return e;
    TcParams P;
    std::memset(&P, 0, sizeof(P));
    P.a = a;
    P.rope = rope;
    P.lse = lse;
    P.status = status;
    P.k_next = rope ? static_cast<const __nv_bfloat16*>(k_next) : nullptr;
    P.khat_next = static_cast<__nv_bfloat16*>(khat_next);
    P.sl2 = a.scale * kLog2e;
    P.ntq = (a.T + TQ - 1) / TQ;
    P.ntiles = a.B * P.ntq * kHkv;
    P.o = static_cast<__nv_bfloat16*>(o);
    if (!ring::encode_heads(&P.qmap, q, a.B, a.T, TQ) || !ring::encode_rows(&P.kwmap, khat, a.B, a.T, NWIN) ||
        !ring::encode_rows(&P.vwmap, v, a.B, a.T, NWIN) || !ring::encode_rows(&P.krmap, khat, a.B, a.T, NRB) ||
        !ring::encode_rows(&P.vrmap, v, a.B, a.T, NRB))
        return cudaErrorInvalidValue;
    const bool wide = a.W > 12;
    auto kernel = wide ? fwd_tc_kernel<true> : fwd_tc_kernel<false>;
    static CtxSetting configured[2][64];  // per variant and device
    if (!ctx_setting_holds(configured[wide][dev & 63], kSmemBytes)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        ctx_setting_done(configured[wide][dev & 63], kSmemBytes);
    }
    const int grid = P.ntiles < 2 * sms ? P.ntiles : 2 * sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = kSmemBytes;
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

}  // namespace sfa
