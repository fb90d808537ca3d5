// sfa_fwd_tc.cu -- the bf16 forward on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for windows W <= 16: an
// alternative to the mma.sync kernel of sfa_fwd_mma.cu, selected with
// SFA_FORWARD_KERNEL=tc (see fwd_tc_supported for why it is not the default).
//
// The method is the attention of "Depth-Staggered Fibonacci Spacing for Sparse
// Attention" (arXiv 2606.28560), section 2 "Attended set": query i attends the
// window distances 0..W and one interpolated row per rung at d = alpha f,
// between rows i - floor(d) (weight 1 - t) and i - floor(d) - 1 (weight t);
// the offsets are shared by every query, so for a tile of consecutive queries
// each rung is ONE contiguous block of key/value rows.
//
// A persistent CTA (one per SM: it holds all 512 TMEM columns) walks tiles of
// TQ = 31 consecutive queries of one sequence b and one key/value head g; the
// tile's 31 x 4 (query, head) rows are the M = 128 rows of every MMA (row
// 4 e + h, TMEM lane = row; rows 124..127 are padding).  The CTA keeps two
// tiles in flight, one in each half of TMEM (a "slot" of 256 columns), so
// that the tensor cores work on one tile while the softmax warps of the
// other read and write theirs.  Per tile, in a slot:
//   scores   S_win = Qhat . Khat_win^T  (N = 48 key rows i0 - W .. i0 - W + 47)
//            and, for each group of up to 4 rungs, S_grp = Qhat . [Khat_k]^T
//            over the group's blocks (32 rows i0 - n_k - 1 .. i0 - n_k + 30
//            each, contiguous in shared memory: one MMA of N = 32 x rungs per
//            K step);
//   softmax  one thread per (query, head) row reads its window band and, per
//            rung, the two columns of its rows b and a (the row's query
//            offset selects them from a 16-column load), forms the lerped
//            rung score (1 - t) s_a + t s_b (the score of the interpolated
//            key, by linearity), keeps an online maximum over the groups (the
//            output is rescaled in TMEM when a later group raises it by more
//            than 2^8), and writes the probabilities back into TMEM as bf16
//            over the scores: the window band as computed, a rung's p split
//            onto its two rows as p t and p (1 - t), zeros elsewhere, so that
//            P_k . V_k forms the interpolated value row;
//   output   O += P_win . V_win and P_grp . V_grp (A from TMEM, V row-major
//            as an MN-major operand from shared memory), fp32 in TMEM; the
//            softmax warps then normalise their rows by 1 / l and store them
//            through shared memory with TMA.
// Warp roles (12 warps): 0 loads with TMA for both slots (Q and the RoPE rows
// of a tile, its window block of Khat and V, per rung group the key blocks and
// the value blocks), polling their buffers without blocking so that neither
// slot waits behind the other; 1 and 2 issue the MMAs of slot 0 and slot 1
// (one lane each; warp 1 also allocates TMEM); 3 rotates the queries of both
// slots in shared memory (RoPE, in the stored dimension order of Khat) and the
// next layer's keys (multi-layer forward); 4-7 and 8-11 run the softmax and
// the output of slot 0 and 1 (warp w serves TMEM lanes 32 (w % 4) ..).  Every wait is bounded: a wait that gives up sets the CTA's abort
// flag and SFA_DEVSTAT_WAIT_TIMEOUT, and every role then stops; the MMA lane
// waits for its last MMAs and the loader for its last copies before the CTA
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

constexpr int TQ = 31;           // queries per tile (x 4 heads = 124 of the 128 MMA rows)
constexpr int MROWS = 128;
constexpr int NWIN = 48;         // window block rows, N of the window scores
constexpr int NRB = 32;          // rung block rows
constexpr int GR = 4;            // rungs per group (N = 128)
constexpr int MAXW = 16;         // TQ + W rows must fit the window block
constexpr int NTHREADS = 384;    // 12 warps
constexpr int kSoftWarp0 = 4;    // warps 4..7: slot 0, 8..11: slot 1
constexpr float kLazy = 8.0f;    // a later group raises the row maximum only past this margin (log2 units)

constexpr uint32_t kQBytes = MROWS * ROWB;          // one Q buffer (rows 124..127 stay zero)
constexpr uint32_t kQBox = TQ * kG * ROWB;          // bytes one Q box moves (zero filled past T)
constexpr uint32_t kTabBytes = 8192;                // RoPE rows of a tile's positions (31 x 256)
constexpr uint32_t kWinTensor = NWIN * ROWB;        // 6 KB: Khat, then V
constexpr uint32_t kRungBytes = NRB * ROWB;         // 4 KB
constexpr uint32_t kGroupBytes = GR * kRungBytes;   // 16 KB
constexpr uint32_t kStageBytes = 16 * ROWB;         // half an output warp's rows (4 queries)

// TMEM columns of a slot (slot X starts at column 256 X)
constexpr uint32_t kSlotCols = 256;
constexpr uint32_t kColW = 0;     // window scores (48), then its probabilities (24 bf16 pairs)
constexpr uint32_t kColR = 48;    // group scores (32 per rung), probabilities in the first 16 of each
constexpr uint32_t kColO = 176;   // O (64)
constexpr uint32_t kTmemCols = 512;
static_assert(kColR + NRB * GR <= kColO && kColO + kD <= kSlotCols, "slot columns");

constexpr uint32_t kIdescWin = tc::idesc_bf16(MROWS, NWIN, false);
constexpr uint32_t kIdescPV = tc::idesc_bf16(MROWS, kD, true);

// shared memory: the header, the output staging of the 8 softmax warps, then
// each slot's buffers
constexpr uint32_t kHdrBytes = 1024;
constexpr uint32_t kOffStage = kHdrBytes;
constexpr uint32_t kOffSlots = kOffStage + 8 * kStageBytes;
constexpr uint32_t kSQ = 0;                               // [2] Q buffers
constexpr uint32_t kSTab = kSQ + 2 * kQBytes;             // RoPE rows
constexpr uint32_t kSWin = kSTab + kTabBytes;             // window Khat, then V
constexpr uint32_t kSKg = kSWin + 2 * kWinTensor;         // [2] rung-group key blocks
constexpr uint32_t kSVg = kSKg + 2 * kGroupBytes;         // rung-group value blocks
constexpr uint32_t kSlotBytes = kSVg + kGroupBytes;
constexpr size_t kSmemBytes = 1024 + (size_t)kOffSlots + 2 * (size_t)kSlotBytes;
static_assert(kOffSlots % 1024 == 0 && kSlotBytes % 1024 == 0 && kSTab % 1024 == 0 && kSWin % 1024 == 0 &&
                  kSKg % 1024 == 0 && kSVg % 1024 == 0 && kWinTensor % 1024 == 0,
              "operand tiles on the 1024-byte swizzle period");
static_assert(kSmemBytes <= 232448, "shared memory of one CTA");

// header: per-slot barriers (192 bytes each), then the shared words, then the rung table
enum : uint32_t {
    B_QFULL = 0, B_QREADY = 16, B_QEMPTY = 32, B_TABEMPTY = 48, B_WFULL = 56, B_WEMPTY = 64, B_KFULL = 72,
    B_KEMPTY = 88, B_VFULL = 104, B_VEMPTY = 112, B_SFULL = 120, B_PFULL = 128, B_OFULL = 136, B_OFREE = 144,
    kSlotBarBytes = 192,
    H_DONE = 2 * kSlotBarBytes, H_TMEM = H_DONE + 16, H_ABORT = H_TMEM + 4, H_RUNGS = 512
};
static_assert(H_ABORT + 4 <= H_RUNGS && H_RUNGS + SFA_MAX_RUNGS * 12 <= kHdrBytes, "header layout");

struct TcParams {
    CUtensorMap qmap;          // Q [B][T][8][64], box 64 x 4 heads x TQ queries
    CUtensorMap omap4;         // O, box 64 x 4 heads x 4 queries (stores)
    CUtensorMap omap3;         // O, box 64 x 4 heads x 3 queries (the tile's last 3)
    CUtensorMap kwmap, vwmap;  // Khat / V [B][T][2][64], box NWIN rows of one head
    CUtensorMap krmap, vrmap;  // box NRB rows
    LayerArgs a;
    const float2* rope;        // nullptr: Q and K are used as given
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
    int ng;   // rung groups (ceil(kt / 4))
};

struct SR {
    int n;
    float t;
    int c;
};

struct Sm {
    uint32_t base;         // shared address of the header
    unsigned char* hdr;    // generic pointer to the header
    __device__ uint32_t bar(int X, uint32_t off, int i = 0) const {
        return base + (uint32_t)X * kSlotBarBytes + off + 8u * (uint32_t)i;
    }
    __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(hdr + H_ABORT); }
    __device__ const SR* rungs() const { return reinterpret_cast<const SR*>(hdr + H_RUNGS); }
    __device__ uint32_t slot(int X) const { return base + kOffSlots + (uint32_t)X * kSlotBytes; }
    __device__ uint32_t q(int X, int i) const { return slot(X) + kSQ + (uint32_t)i * kQBytes; }
    __device__ uint32_t tab(int X) const { return slot(X) + kSTab; }
    __device__ uint32_t win(int X) const { return slot(X) + kSWin; }
    __device__ uint32_t kg(int X, int i) const { return slot(X) + kSKg + (uint32_t)i * kGroupBytes; }
    __device__ uint32_t vg(int X) const { return slot(X) + kSVg; }
    __device__ uint32_t stage(int X, int q) const { return base + kOffStage + (uint32_t)(4 * X + q) * kStageBytes; }
};

// Tile n of slot X: the CTA's tiles blockIdx.x + j gridDim.x, j = 2 n + X.
__device__ __forceinline__ bool tile_of(const TcParams& P, const Sm& S, int X, int n, Tile& x) {
    const long long t = (long long)blockIdx.x + (long long)(2 * n + X) * gridDim.x;
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
    x.ng = (kt + GR - 1) / GR;
    return true;
}

__device__ __forceinline__ int group_rungs(const Tile& x, int grp) { return min(GR, x.kt - GR * grp); }

__device__ __forceinline__ void give_up(const TcParams& P, const Sm& S) {
    *S.abort_flag() = 1;
    if (P.status) atomicOr(P.status, SFA_DEVSTAT_WAIT_TIMEOUT);
}

// ------------------------------------------------------------- loader

// One slot's loads in three streams, each in tile order: the Q (and RoPE
// rows) of every tile; the window block and the rung-group key blocks of every
// tile; the rung-group value blocks of every tile.  A stream issues its next
// load as soon as the buffer it fills is free, so no load waits behind
// another stream's.
struct Stream {
    int n;       // tile
    int grp;     // rung group within the tile (-1: the window, key stream)
    bool done;
    Tile x;
};

struct LoadState {
    Stream q, k, v;
    int qn, wl, kgc, vgc;  // Q, window, group key and group value loads so far
};

__device__ __forceinline__ void load_q(const TcParams& P, const Sm& S, int X, int n, const Tile& x) {
    const int qb = n & 1;
    const int nq = min(TQ, P.a.T - x.i0);
    const uint32_t tab_bytes = P.rope ? (uint32_t)nq * TABB : 0u;
    const uint32_t full = S.bar(X, B_QFULL, qb);
    mbar_arrive_expect_tx(full, kQBox + tab_bytes);
    tma_load_4d(S.q(X, qb), &P.qmap, 0, x.g * kG, x.i0, x.b, full);
    if (tab_bytes) bulk_g2s(S.tab(X), P.rope + (size_t)x.i0 * kPairs, tab_bytes, full);
}

// The rung blocks of group grp of tile x (key or value rows) into `dst`.
__device__ __forceinline__ void load_group(const TcParams& P, const Sm& S, const CUtensorMap* map, uint32_t dst,
                                           uint32_t full, const Tile& x, int grp) {
    const int nr = group_rungs(x, grp);
    const SR* r = S.rungs();
    mbar_arrive_expect_tx(full, (uint32_t)nr * kRungBytes);
    for (int k = 0; k < nr; ++k)
        tma_load_4d(dst + (uint32_t)k * kRungBytes, map, 0, x.g, x.i0 - r[GR * grp + k].n - 1, x.b, full);
}

// Issues the slot's next loads while their buffers are free; true if any.
__device__ bool loader_step(const TcParams& P, const Sm& S, int X, LoadState& L) {
    bool any = false;
    // Q and RoPE rows
    while (!L.q.done) {
        const int n = L.q.n;
        if (!mbar_test(S.bar(X, B_QEMPTY, n & 1), ((n >> 1) & 1) ^ 1) || !mbar_test(S.bar(X, B_TABEMPTY), (n & 1) ^ 1))
            break;
        load_q(P, S, X, n, L.q.x);
        ++L.qn;
        L.q.done = !tile_of(P, S, X, ++L.q.n, L.q.x);
        any = true;
    }
    // window blocks and rung-group key blocks
    while (!L.k.done) {
        const Tile& x = L.k.x;
        if (L.k.grp < 0) {
            if (!mbar_test(S.bar(X, B_WEMPTY), (L.k.n & 1) ^ 1)) break;
            const uint32_t full = S.bar(X, B_WFULL);
            mbar_arrive_expect_tx(full, 2 * kWinTensor);
            tma_load_4d(S.win(X), &P.kwmap, 0, x.g, x.i0 - P.a.W, x.b, full);
            tma_load_4d(S.win(X) + kWinTensor, &P.vwmap, 0, x.g, x.i0 - P.a.W, x.b, full);
            ++L.wl;
            L.k.grp = 0;
        } else if (L.k.grp < x.ng) {
            const int kb = L.kgc & 1;
            if (!mbar_test(S.bar(X, B_KEMPTY, kb), ((L.kgc >> 1) & 1) ^ 1)) break;
            load_group(P, S, &P.krmap, S.kg(X, kb), S.bar(X, B_KFULL, kb), x, L.k.grp);
            ++L.kgc;
            ++L.k.grp;
        }
        if (L.k.grp >= 0 && L.k.grp >= x.ng) {
            L.k.grp = -1;
            L.k.done = !tile_of(P, S, X, ++L.k.n, L.k.x);
        }
        any = true;
    }
    // rung-group value blocks
    while (!L.v.done) {
        const Tile& x = L.v.x;
        if (L.v.grp < x.ng) {
            if (!mbar_test(S.bar(X, B_VEMPTY), (L.vgc & 1) ^ 1)) break;
            load_group(P, S, &P.vrmap, S.vg(X), S.bar(X, B_VFULL), x, L.v.grp);
            ++L.vgc;
            ++L.v.grp;
            any = true;
        }
        if (L.v.grp >= x.ng) {
            L.v.grp = 0;
            L.v.done = !tile_of(P, S, X, ++L.v.n, L.v.x);
        }
    }
    return any;
}

__device__ void loader(const TcParams& P, const Sm& S) {
    volatile int* abort_flag = S.abort_flag();
    // Khat is written by the launch before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    LoadState L[2];
    for (int X = 0; X < 2; ++X) {
        L[X] = LoadState{};
        L[X].q.done = !tile_of(P, S, X, 0, L[X].q.x);
        L[X].k = L[X].q;
        L[X].k.grp = -1;
        L[X].v = L[X].q;
    }
    unsigned long long t_last = now_ns();
    for (;;) {
        const bool p0 = loader_step(P, S, 0, L[0]);
        const bool p1 = loader_step(P, S, 1, L[1]);
        bool all = true;
        for (int X = 0; X < 2; ++X) all = all && L[X].q.done && L[X].k.done && L[X].v.done;
        if (all) return;
        if (p0 || p1) {
            t_last = now_ns();
            continue;
        }
        if (*abort_flag) break;
        if (now_ns() - t_last > kWaitNs) {
            give_up(P, S);
            break;
        }
    }
    // no copy of this CTA may land after it exits: wait (bounded) for the last
    // announced phase of every buffer
    for (int X = 0; X < 2; ++X) {
        const LoadState& l = L[X];
        for (int m = max(0, l.qn - 2); m < l.qn; ++m) (void)mbar_wait(S.bar(X, B_QFULL, m & 1), (m >> 1) & 1, nullptr);
        if (l.wl > 0) (void)mbar_wait(S.bar(X, B_WFULL), (l.wl - 1) & 1, nullptr);
        for (int m = max(0, l.kgc - 2); m < l.kgc; ++m)
            (void)mbar_wait(S.bar(X, B_KFULL, m & 1), (m >> 1) & 1, nullptr);
        if (l.vgc > 0) (void)mbar_wait(S.bar(X, B_VFULL), (l.vgc - 1) & 1, nullptr);
    }
}

// ------------------------------------------------------------- MMA issue

// One slot's MMA sequence per tile: [scores of the window and group 0],
// [O += P V of the window and group 0], then per further group [its scores],
// [O += its P V].  Each op issues once its operands are ready; the tensor core
// runs the MMAs of one thread in issue order, so a group's scores, which
// overwrite the probabilities of the group before, follow that group's P V.
struct MmaState {
    int n;        // tile
    int grp;
    int op;       // 0 window + group 0 scores, 1 P V of group grp, 2 scores of group grp
    bool done;
    Tile x;
    int kgc, vgc, pc;  // group key / value buffers consumed; probability phases consumed
};

__device__ bool mma_step(const TcParams& P, const Sm& S, int X, uint32_t tmem, MmaState& M) {
    if (M.done) return false;
    const Tile& x = M.x;
    const uint32_t tb = tmem + (uint32_t)X * kSlotCols;
    const int qb = M.n & 1;
    if (M.op == 0 || M.op == 2) {
        const bool first = M.op == 0;
        if (first && (!mbar_test(S.bar(X, B_QREADY, qb), (M.n >> 1) & 1) ||
                      !mbar_test(S.bar(X, B_WFULL), M.n & 1)))
            return false;
        const bool rungs = M.grp < x.ng;
        if (rungs && !mbar_test(S.bar(X, B_KFULL, M.kgc & 1), (M.kgc >> 1) & 1)) return false;
        tc::fence_after();
        const uint32_t qa = S.q(X, qb);
        if (first) {
            const uint32_t kw = S.win(X);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_ss(tb + kColW, tc::desc_kmajor(qa + 32 * ks), tc::desc_kmajor(kw + 32 * ks), kIdescWin,
                           ks > 0);
        }
        if (rungs) {
            const uint32_t kb = S.kg(X, M.kgc & 1);
            const uint32_t idesc = tc::idesc_bf16(MROWS, NRB * group_rungs(x, M.grp), false);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_ss(tb + kColR, tc::desc_kmajor(qa + 32 * ks), tc::desc_kmajor(kb + 32 * ks), idesc, ks > 0);
            tc::commit(S.bar(X, B_SFULL));
            tc::commit(S.bar(X, B_KEMPTY, M.kgc & 1));
            ++M.kgc;
        } else {
            tc::commit(S.bar(X, B_SFULL));
        }
        // the last scores of the tile: its Q buffer is free
        if (M.grp + 1 >= x.ng) tc::commit(S.bar(X, B_QEMPTY, qb));
        M.op = 1;
        return true;
    }
    // O += P V of group grp (and the window with group 0)
    const bool first = M.grp == 0;
    const bool rungs = M.grp < x.ng;
    if (!mbar_test(S.bar(X, B_PFULL), M.pc & 1)) return false;
    if (first && !mbar_test(S.bar(X, B_OFREE), (M.n & 1) ^ 1)) return false;
    if (rungs && !mbar_test(S.bar(X, B_VFULL), M.vgc & 1)) return false;
    tc::fence_after();
    const uint32_t d = tb + kColO;
    if (first) {
        const uint32_t vw = S.win(X) + kWinTensor;
#pragma unroll
        for (int ks = 0; ks < NWIN / 16; ++ks)
            tc::mma_ts(d, tb + kColW + 8 * ks, tc::desc_mnmajor(vw + 2048 * ks), kIdescPV, ks > 0);
        tc::commit(S.bar(X, B_WEMPTY));
    }
    if (rungs) {
        const int nr = group_rungs(x, M.grp);
        const uint32_t vb = S.vg(X);
        for (int k = 0; k < nr; ++k)
#pragma unroll
            for (int ks = 0; ks < NRB / 16; ++ks)
                tc::mma_ts(d, tb + kColR + NRB * k + 8 * ks, tc::desc_mnmajor(vb + kRungBytes * k + 2048 * ks),
                           kIdescPV, 1);
        tc::commit(S.bar(X, B_VEMPTY));
        ++M.vgc;
    }
    ++M.pc;
    if (M.grp + 1 >= max(x.ng, 1)) {
        tc::commit(S.bar(X, B_OFULL));
        ++M.n;
        M.grp = 0;
        M.op = 0;
        if (!tile_of(P, S, X, M.n, M.x)) M.done = true;
    } else {
        ++M.grp;
        M.op = 2;
    }
    return true;
}

// The MMAs of slot X come from one thread of their own: a thread issues one
// tcgen05.mma about every 200 cycles whatever its size, so the two slots'
// MMAs issue side by side.
__device__ void mma_issuer(const TcParams& P, const Sm& S, uint32_t tmem, int X) {
    volatile int* abort_flag = S.abort_flag();
    MmaState M = MmaState{};
    M.done = !tile_of(P, S, X, 0, M.x);
    unsigned long long t_last = now_ns();
    while (!M.done) {
        if (mma_step(P, S, X, tmem, M)) {
            t_last = now_ns();
            continue;
        }
        if (*abort_flag) break;
        if (now_ns() - t_last > kWaitNs) {
            give_up(P, S);
            break;
        }
    }
    // TMEM is freed only after every MMA issued has completed
    tc::commit(S.base + H_DONE + 8 * X);
    (void)mbar_wait(S.base + H_DONE + 8 * X, 0, nullptr);
}

// Warp 3: the queries of both slots' tiles (and the next layer's keys), in
// the order the slots need them.
// ------------------------------------------------------------- queries and next keys

// Qhat of row r (query e = r / 4, head r % 4) of a Q buffer, rotated in place
// at position i0 + e and written in the stored dimension order of Khat: the
// pair (8c + 2w + hh, + 32) of natural chunks c and 4 + c goes to word c of
// stored chunks w and 4 + w (kdim_of in sfa_fwd_mma.cu), so that every score
// is the same dot product as with the natural order.
__device__ __forceinline__ void rotate_q_row(uint32_t qbuf, uint32_t tab, int r) {
    const uint32_t row = qbuf + (uint32_t)r * ROWB;
    const uint32_t trow = tab + (uint32_t)(r >> 2) * TABB;
    const int sw = r & 7;
    uint4 in[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) in[c] = ring::lds_u4(row + (uint32_t)((c ^ sw) << 4));
    uint32_t xo[4][4], yo[4][4];  // [stored chunk w][word c]
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float4 cs = ring::lds_f4(trow + (uint32_t)(64 * c + 16 * w));
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
__device__ __forceinline__ void rotate_next_keys(const TcParams& P, uint32_t tab, const Tile& x, int id) {
    const int u = id >> 2, a = id & 3;
    const int pos = x.i0 + u;
    if (u >= TQ || pos >= P.a.T) return;
    const size_t rowi = ((size_t)x.b * P.a.T + pos) * kHkv + x.g;
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(P.k_next + rowi * kD + 8 * a));
    const uint4 yv = __ldg(reinterpret_cast<const uint4*>(P.k_next + rowi * kD + 32 + 8 * a));
    const uint32_t trow = tab + (uint32_t)u * TABB + 64u * (uint32_t)a;
    uint32_t* out = reinterpret_cast<uint32_t*>(P.khat_next + rowi * kD);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float4 cs = ring::lds_f4(trow + 16u * (uint32_t)w);
        const float2 xf = unpack_bf16(ring::u4_get(xv, w)), yf = unpack_bf16(ring::u4_get(yv, w));
        out[4 * w + a] = ring::rope_x(xf, yf, cs);
        out[16 + 4 * w + a] = ring::rope_y(xf, yf, cs);
    }
}

__device__ void prep(const TcParams& P, const Sm& S, int lane) {
    volatile int* abort_flag = S.abort_flag();
    // Khat_next may still be read by the launch before this one
    if (P.k_next) asm volatile("griddepcontrol.wait;" ::: "memory");
    Tile x;
    for (int j = 0;; ++j) {
        const int X = j & 1, n = j >> 1;
        if (!tile_of(P, S, X, n, x)) break;
        const int qb = n & 1;
        if (!ring::warp_wait(S.bar(X, B_QFULL, qb), (n >> 1) & 1, abort_flag)) {
            if (lane == 0) give_up(P, S);
            return;
        }
        if (P.rope) {
            const int rows = kG * min(TQ, P.a.T - x.i0);
#pragma unroll 1
            for (int r = lane; r < rows; r += 32) rotate_q_row(S.q(X, qb), S.tab(X), r);
            if (P.k_next)
#pragma unroll 1
                for (int id = lane; id < 4 * TQ; id += 32) rotate_next_keys(P, S.tab(X), x, id);
            fence_proxy_async();
        }
        __syncwarp();
        mbar_arrive_if(S.bar(X, B_QREADY, qb), lane == 0);
        mbar_arrive_if(S.bar(X, B_TABEMPTY), lane == 0);
    }
}

// ------------------------------------------------------------- softmax and output

// Probabilities of a rung for this lane's row, as the 8 bf16 pairs of local K
// 0..15 (the warp's columns 8q .. 8q + 15 of the rung block): p t on row b =
// local jj, p (1 - t) on row a = jj + 1, zero elsewhere.
__device__ __forceinline__ void rung_p_words(float pb, float pa, int jj, uint32_t (&w)[8]) {
    const bool odd = jj & 1;
    const uint32_t v1 = odd ? pack_bf16(0.f, pb) : pack_bf16(pb, pa);
    const uint32_t v2 = pack_bf16(pa, 0.f);
    const int i1 = jj >> 1, i2 = odd ? i1 + 1 : -1;
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = i == i1 ? v1 : (i == i2 ? v2 : 0u);
}

// Zero the 32-bit columns [c0, c1) of this warp's lanes (c0, c1 multiples of 4).
__device__ __forceinline__ void zero_cols(uint32_t lane_base, uint32_t c0, uint32_t c1) {
    for (uint32_t c = c0; c < c1; c += 4) tc::st_x4(lane_base + c, 0u, 0u, 0u, 0u);
}

// Rows of the warp's lanes: the lerped scores of the nr rungs of a group
// (local columns jj and jj + 1 of each 16-column load are rows b and a), two
// rungs per TMEM load round.
__device__ __forceinline__ void group_scores(const Sm& S, uint32_t lb, int q, int jj, int k0, int nr, int i,
                                             bool row_ok, float (&sr)[GR], float& m) {
    const SR* rt = S.rungs();
#pragma unroll
    for (int k2 = 0; k2 < GR; k2 += 2) {
        uint32_t a[2][16];
#pragma unroll
        for (int k = 0; k < 2; ++k)
            if (k2 + k < nr) tc::ld_x16(lb + kColR + NRB * (k2 + k) + 8 * q, a[k]);
        tc::wait_ld();
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            sr[k2 + k] = -INFINITY;
            if (k2 + k >= nr) continue;
            // a[k][jj], a[k][jj + 1] by a three-level select on jj
            float x4[5], y2[3];
#pragma unroll
            for (int u = 0; u < 5; ++u) x4[u] = __uint_as_float((jj & 4) ? a[k][u + 4] : a[k][u]);
#pragma unroll
            for (int u = 0; u < 3; ++u) y2[u] = (jj & 2) ? x4[u + 2] : x4[u];
            const float sb = (jj & 1) ? y2[1] : y2[0];
            const float sa = (jj & 1) ? y2[2] : y2[1];
            const SR rk = rt[k0 + k2 + k];
            const float v = __fmaf_rn(rk.t, sb, __fmul_rn(1.f - rk.t, sa));
            sr[k2 + k] = (row_ok && i >= rk.c) ? v : -INFINITY;
            m = fmaxf(m, sr[k2 + k]);
        }
    }
}

// Probabilities of a group's rungs into TMEM over their scores; returns their sum.
__device__ __forceinline__ float group_probs(const Sm& S, uint32_t lb, int q, int jj, int k0, int nr,
                                             const float (&sr)[GR], float sl2, float nm) {
    const SR* rt = S.rungs();
    float l = 0.f;
#pragma unroll
    for (int k = 0; k < GR; ++k) {
        if (k >= nr) break;
        const float p = fast_exp2(__fmaf_rn(sr[k], sl2, nm));
        l += p;
        const float tk = rt[k0 + k].t;
        uint32_t pk[8];
        rung_p_words(p * tk, p * (1.f - tk), jj, pk);
        const uint32_t col = lb + kColR + NRB * k;
        tc::st_x8(col + 4 * q, pk);
        zero_cols(col, 0, 4 * q);
        zero_cols(col, 4 * q + 8, 16);
    }
    return l;
}

__device__ bool softmax_tile(const TcParams& P, const Sm& S, uint32_t tmem, int X, int n, const Tile& x, int q,
                             int lane, int& sc) {
    volatile int* abort_flag = S.abort_flag();
    const int r = 32 * q + lane;           // MMA row = 4 e + h
    const int e = r >> 2, h = r & 3;       // query offset in the tile, head
    const int jj = lane >> 2;              // e - 8 q: the row's offset inside the warp's columns
    const uint32_t lb = tmem + (uint32_t)X * kSlotCols + ((uint32_t)(32 * q) << 16);
    const float sl2 = P.sl2;
    const int i = x.i0 + e;
    const bool row_ok = e < TQ && i < P.a.T;
    float nm = 0.f;   // minus the running maximum, log2 units (0 on rows that do not exist)
    float l = 0.f;
    const int ngo = max(x.ng, 1);
    for (int grp = 0; grp < ngo; ++grp) {
        if (!ring::warp_wait(S.bar(X, B_SFULL), sc & 1, abort_flag)) return false;
        ++sc;
        tc::fence_after();
        const int nr = grp < x.ng ? group_rungs(x, grp) : 0;
        float sr[GR];
        if (grp == 0) {
            float m = -INFINITY;
            group_scores(S, lb, q, jj, 0, nr, i, row_ok, sr, m);
            // window band: block column c (position i0 - W + c) of this lane is
            // c = 8 q + u, u = 0..23; the row's entries are u = jj .. jj + W at
            // positions >= 0
            float w[24];
            {
                uint32_t a16[16], a8[8];
                tc::ld_x16(lb + kColW + 8 * q, a16);
                tc::ld_x8(lb + kColW + 8 * q + 16, a8);
                tc::wait_ld();
                const int lo = max(jj, P.a.W - x.i0 - 8 * q);
                const int hi = row_ok ? jj + P.a.W : -1;
#pragma unroll
                for (int u = 0; u < 24; ++u) {
                    const float v = __uint_as_float(u < 16 ? a16[u] : a8[u - 16]);
                    w[u] = (u >= lo && u <= hi) ? v : -INFINITY;
                }
            }
#pragma unroll
            for (int u = 0; u < 24; ++u) m = fmaxf(m, w[u]);
            nm = row_ok ? -m * sl2 : 0.f;
            uint32_t pw[12];
#pragma unroll
            for (int u = 0; u < 12; ++u) {
                const float p0 = fast_exp2(__fmaf_rn(w[2 * u], sl2, nm));
                const float p1 = fast_exp2(__fmaf_rn(w[2 * u + 1], sl2, nm));
                l += p0 + p1;
                pw[u] = pack_bf16(p0, p1);
            }
            // window probabilities: bf16 pairs at columns kColW + 4 q + u / 2,
            // zeros in the rest of the 24 columns the window P V reads
            const uint32_t w8[8] = {pw[0], pw[1], pw[2], pw[3], pw[4], pw[5], pw[6], pw[7]};
            tc::st_x8(lb + kColW + 4 * q, w8);
            tc::st_x4(lb + kColW + 4 * q + 8, pw[8], pw[9], pw[10], pw[11]);
            zero_cols(lb + kColW, 0, 4 * q);
            zero_cols(lb + kColW, 4 * q + 12, 24);
        } else {
            float m = -INFINITY;
            group_scores(S, lb, q, jj, GR * grp, nr, i, row_ok, sr, m);
            // raise the row maximum only when the group beats it by 2^8; the
            // output so far (every P V before this group's scores has completed)
            // and the sum are rescaled
            const bool need = row_ok && __fmaf_rn(m, sl2, nm) > kLazy;
            if (__any_sync(kFull, need)) {
                const float nm_new = need ? -m * sl2 : nm;
                const float c = fast_exp2(nm_new - nm);
                l *= c;
                nm = nm_new;
                uint32_t o[32];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tc::ld_x32(lb + kColO + 32 * half, o);
                    tc::wait_ld();
#pragma unroll
                    for (int d = 0; d < 32; ++d) o[d] = __float_as_uint(__uint_as_float(o[d]) * c);
                    tc::st_x32(lb + kColO + 32 * half, o);
                }
            }
        }
        l += group_probs(S, lb, q, jj, GR * grp, nr, sr, sl2, nm);
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        mbar_arrive_if(S.bar(X, B_PFULL), lane == 0);
    }
    // the output: every P V of the tile has completed.  Each lane packs its
    // row; the warp's rows go out in two halves of 4 queries (16 rows), each
    // staged in the 128-byte swizzle of the store box for one TMA store
    if (!ring::warp_wait(S.bar(X, B_OFULL), n & 1, abort_flag)) return false;
    tc::fence_after();
    uint32_t pk[32];
    {
        uint32_t o0[32], o1[32];
        tc::ld_x32(lb + kColO, o0);
        tc::ld_x32(lb + kColO + 32, o1);
        tc::wait_ld();
        // row sums are >= 1 on rows that exist (the entry at the maximum contributes 1)
        const float inv = l > 0.f ? fast_rcp(l) : 0.f;
#pragma unroll
        for (int d = 0; d < 16; ++d) {
            pk[d] = pack_bf16(__uint_as_float(o0[2 * d]) * inv, __uint_as_float(o0[2 * d + 1]) * inv);
            pk[16 + d] = pack_bf16(__uint_as_float(o1[2 * d]) * inv, __uint_as_float(o1[2 * d + 1]) * inv);
        }
    }
    tc::fence_before();
    __syncwarp();
    mbar_arrive_if(S.bar(X, B_OFREE), lane == 0);
    const uint32_t stage = S.stage(X, q);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        if (lane == 0) bulk_wait_read();
        __syncwarp();
        if ((lane >> 4) == half) {
            const int row = lane & 15;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (uint32_t)row * ROWB +
                                                                              (uint32_t)((c ^ (row & 7)) << 4)),
                             "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                             : "memory");
            fence_proxy_async();
        }
        __syncwarp();
        const int qi = x.i0 + 8 * q + 4 * half;
        if (lane == 0 && qi < P.a.T) {
            tma_store_4d((q == 3 && half == 1) ? (const void*)&P.omap3 : (const void*)&P.omap4, stage, 0, x.g * kG,
                         qi, x.b);
            bulk_commit();
        }
    }
    if (P.lse && row_ok) P.lse[((size_t)x.b * P.a.T + i) * kHq + x.g * kG + h] = (__log2f(l) - nm) * kLn2;
    return true;
}

__device__ void softmax(const TcParams& P, const Sm& S, uint32_t tmem, int X, int q, int lane) {
    int sc = 0;
    Tile x;
    for (int n = 0; tile_of(P, S, X, n, x); ++n)
        if (!softmax_tile(P, S, tmem, X, n, x, q, lane, sc)) {
            if (lane == 0) give_up(P, S);
            break;
        }
    if (lane == 0) bulk_wait_all();
}

__global__ void __launch_bounds__(NTHREADS, 1) fwd_tc_kernel(const __grid_constant__ TcParams P) {
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
        for (int X = 0; X < 2; ++X) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(S.bar(X, B_QFULL, i), 1);
                mbar_init(S.bar(X, B_QREADY, i), 1);
                mbar_init(S.bar(X, B_QEMPTY, i), 1);
                mbar_init(S.bar(X, B_KFULL, i), 1);
                mbar_init(S.bar(X, B_KEMPTY, i), 1);
            }
            mbar_init(S.bar(X, B_TABEMPTY), 1);
            mbar_init(S.bar(X, B_WFULL), 1);
            mbar_init(S.bar(X, B_WEMPTY), 1);
            mbar_init(S.bar(X, B_VFULL), 1);
            mbar_init(S.bar(X, B_VEMPTY), 1);
            mbar_init(S.bar(X, B_SFULL), 1);
            mbar_init(S.bar(X, B_PFULL), 4);
            mbar_init(S.bar(X, B_OFULL), 1);
            mbar_init(S.bar(X, B_OFREE), 4);
        }
        mbar_init(S.base + H_DONE, 1);
        mbar_init(S.base + H_DONE + 8, 1);
        *S.abort_flag() = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // rows 124..127 of the four Q buffers (no query) stay zero
    if (threadIdx.x < 128) {
        const int X = threadIdx.x >> 6, qb = (threadIdx.x >> 5) & 1;
        const uint32_t a = S.q(X, qb) + (uint32_t)(TQ * kG) * ROWB + 16u * (threadIdx.x & 31);
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
    } else if (warp < 3) {
        if (lane == 0) mma_issuer(P, S, tmem, warp - 1);
    } else if (warp < kSoftWarp0) {
        prep(P, S, lane);
    } else {
        softmax(P, S, tmem, (warp - kSoftWarp0) >> 2, warp & 3, lane);
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
// is faster for this attention (a model-shape layer, B = 32, T = 1024, W = 12:
// 37 us against 86 us here).  A tcgen05.mma issued by one thread takes about
// 200 cycles whatever its N (up to 256), and a tile needs about 29 of them
// (12 score and 17 output MMAs: K = 16 each, N = 48 .. 128), so the MMA issue
// of the two slots, and the TMEM round trips of the one-thread-per-row
// softmax, bound this kernel well above the mma.sync one.
// SFA_FORWARD_KERNEL=tc in the environment (read at every call) selects it.
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
    if (!ring::encode_heads(&P.qmap, q, a.B, a.T, TQ) || !ring::encode_heads(&P.omap4, o, a.B, a.T, 4) ||
        !ring::encode_heads(&P.omap3, o, a.B, a.T, 3) || !ring::encode_rows(&P.kwmap, khat, a.B, a.T, NWIN) ||
        !ring::encode_rows(&P.vwmap, v, a.B, a.T, NWIN) || !ring::encode_rows(&P.krmap, khat, a.B, a.T, NRB) ||
        !ring::encode_rows(&P.vrmap, v, a.B, a.T, NRB))
        return cudaErrorInvalidValue;
    static CtxSetting configured[64];
    if (!ctx_setting_holds(configured[dev & 63], kSmemBytes)) {
        e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        ctx_setting_done(configured[dev & 63], kSmemBytes);
    }
    const int grid = P.ntiles < sms ? P.ntiles : sms;
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
    e = cudaLaunchKernelEx(&cfg, fwd_tc_kernel, P);
    if (e != cudaSuccess) return e;
    count_launch();
    return cudaSuccess;
}

}  // namespace sfa
