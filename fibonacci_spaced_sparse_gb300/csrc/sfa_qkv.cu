// sfa_qkv.cu -- the front end of an attention layer: the QKV projection
// [Q | K | V] = X . Wqkv^T on the 5th-generation tensor cores, with RoPE
// applied to Q and K in the epilogue, writing the bf16 tensors the sparse
// attention reads.
//
// "Depth-Staggered Fibonacci Spacing for Sparse Attention" (arXiv 2606.28560),
// section 2 "Attended set": RoPE (theta = 1e4) is applied to queries and keys
// at their true positions before any key row is gathered; section 3 "Model
// and training": d_model 512, 8 query heads and 2 key/value heads of
// dimension 64, so Wqkv has (8 + 2 + 2) x 64 = 768 rows.  With RoPE done here
// the attention runs on the rotated tensors with its own rotation off.
//
// A persistent CTA per SM walks tiles of BM = 128 tokens x BN = 256 output
// features (four heads) over the whole d_model:
//   warp 0 (one lane): TMA loads of the X and Wqkv k-blocks (64 columns,
//                      128-byte swizzle) into a four-stage mbarrier ring;
//   warp 1:            allocates 512 TMEM columns (two accumulators of 256);
//                      one lane issues tcgen05.mma (M = 128, N = 256, K = 16,
//                      bf16 -> fp32) into the accumulator of the tile, releases
//                      each stage with tcgen05.commit and hands the finished
//                      accumulator to the epilogue;
//   warps 2..5:        the epilogue: each thread owns one token row (TMEM lane),
//                      reads a head's 64 columns with tcgen05.ld, rotates the
//                      pairs (m, m + 32) by the angle of the token's position
//                      (from the fp64-built table of sfa_rope_table), writes the
//                      bf16 head row into a 128-byte-swizzled staging buffer and
//                      a TMA store moves the warp's 32 rows out; the
//                      accumulator is handed back as soon as it has been read.
// With two accumulators the MMAs of the next tile run while the epilogue
// drains the current one.  Every wait is bounded; a timeout sets
// SFA_DEVSTAT_WAIT_TIMEOUT and the CTA stops.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "sfa_internal.cuh"
#include "sfa_mma.cuh"
#include "sfa_ring.cuh"
#include "sfa_tc.cuh"

namespace sfa {

namespace {

using namespace mma;

constexpr int BM = 128;                 // tokens per tile (TMEM lanes)
constexpr int BN = 256;                 // output features per tile (TMEM columns)
constexpr int BK = 64;                  // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;  // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;           // 6 warps: producer, MMA, 4 epilogue
constexpr int kEpiWarps = 4;
constexpr int kQkvRows = kHq * kD + 2 * kHkv * kD;  // 768 output features
constexpr int kNTiles = kQkvRows / BN;              // 3
constexpr uint32_t kTmemCols = 2 * BN;              // two accumulators
constexpr uint32_t kStoreBytes = 32 * kD * 2;       // one warp's 32 rows of one head (4 KB)
// header: full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], the TMEM
// address, the abort flag
constexpr uint32_t kHdrBytes = 1024;
constexpr uint32_t kBarFull = 0, kBarEmpty = 8 * STAGES, kBarTmemFull = 16 * STAGES,
                   kBarTmemEmpty = 16 * STAGES + 16, kTmemSlot = 16 * STAGES + 32, kAbort = 16 * STAGES + 40;
constexpr size_t kSmemBytes =
    1024 + kHdrBytes + STAGES * (size_t)kStageBytes + kEpiWarps * 2 * (size_t)kStoreBytes;

static_assert(kQkvRows % BN == 0, "the projection splits into whole tiles");
static_assert(BN % kD == 0 && (kHq * kD) % BN == 0, "tiles hold whole heads; Q tiles hold only Q heads");
static_assert(kAbort + 4 <= kHdrBytes, "header");
static_assert(kSmemBytes <= 232448, "shared memory of one CTA");

struct QkvParams {
    CUtensorMap xmap;   // X [M][dm] bf16, box 64 x 128, 128-byte swizzle
    CUtensorMap wmap;   // Wqkv [768][dm] bf16, box 64 x 256, 128-byte swizzle
    CUtensorMap qmap;   // Qhat as [M][512], box 64 x 32, 128-byte swizzle (stores)
    CUtensorMap kmap;   // Khat as [M][128]
    CUtensorMap vmap;   // V as [M][128]
    const float2* rope; // [T][32] (cos, sin) or nullptr (no rotation)
    unsigned* status;
    int M, T, nkb;      // tokens, positions per sequence, k-blocks (dm / 64)
    int tiles;          // ceil(M / BM) * kNTiles
};

// ------------------------------------------------------------ tcgen05

// MMA of one k-step: M = 128 tokens, N = 256 features, both operands K-major
// bf16 tiles in the 128-byte swizzle (sfa_tc.cuh); a K step of 16 elements
// advances each descriptor's start address by 32 bytes.
constexpr uint32_t kIdesc = tc::idesc_bf16(BM, BN, false);

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}

// Wait until at most one committed bulk store of this thread still reads
// its shared-memory source.
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

__device__ __forceinline__ void sts_u4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(kThreads, 1) qkv_rope_kernel(const __grid_constant__ QkvParams P) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* hdr = smem_raw + (base - raw);
    const uint32_t bar_full = base + kBarFull, bar_empty = base + kBarEmpty;
    const uint32_t bar_tfull = base + kBarTmemFull, bar_tempty = base + kBarTmemEmpty;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(hdr + kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(hdr + kAbort);
    const uint32_t stages = base + kHdrBytes;
    const uint32_t stores = stages + STAGES * kStageBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);
            mbar_init(bar_tempty + 8 * b, kEpiWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tc::alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // k-blocks of every tile of this CTA, in order, through the ring
            int kbg = 0;
            for (int t = blockIdx.x; t < P.tiles && *abort_flag == 0; t += gridDim.x) {
                const int m0 = (t / kNTiles) * BM, n0 = (t % kNTiles) * BN;
                for (int kb = 0; kb < P.nkb; ++kb, ++kbg) {
                    const int s = kbg % STAGES;
                    if (!mbar_wait(bar_empty + 8 * s, ((uint32_t)(kbg / STAGES) & 1u) ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        break;
                    }
                    const uint32_t a = stages + (uint32_t)s * kStageBytes;
                    mbar_arrive_expect_tx(bar_full + 8 * s, kStageBytes);
                    tma_load_2d(a, &P.xmap, kb * BK, m0, bar_full + 8 * s);
                    tma_load_2d(a + kABytes, &P.wmap, kb * BK, n0, bar_full + 8 * s);
                }
            }
            // Nothing may land in this CTA's shared memory after it leaves: wait
            // for the MMA's release of the last use of every stage (its
            // tcgen05.commit arrival), or, once a wait has failed, for the
            // copies themselves.
            const bool clean = *abort_flag == 0;
            for (int n = max(0, kbg - STAGES); n < kbg; ++n) {
                const uint32_t ph = (uint32_t)(n / STAGES) & 1u;
                if (!clean || !mbar_wait(bar_empty + 8 * (n % STAGES), ph, nullptr))
                    (void)mbar_wait(bar_full + 8 * (n % STAGES), ph, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int kbg = 0, j = 0;
            for (int t = blockIdx.x; t < P.tiles; t += gridDim.x, ++j) {
                const int buf = j & 1;
                // the epilogue has read this accumulator's previous tile
                if (!mbar_wait(bar_tempty + 8 * buf, ((uint32_t)(j >> 1) & 1u) ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                tc::fence_after();
                const uint32_t acc = tmem + (uint32_t)(buf * BN);
                bool ok = true;
                for (int kb = 0; kb < P.nkb; ++kb, ++kbg) {
                    const int s = kbg % STAGES;
                    if (!mbar_wait(bar_full + 8 * s, (uint32_t)(kbg / STAGES) & 1u, abort_flag)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t a = stages + (uint32_t)s * kStageBytes;
                    const uint64_t ad = tc::desc_kmajor(a), bd = tc::desc_kmajor(a + kABytes);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        tc::mma_ss(acc, ad + (uint64_t)(k * UMMA_K * 2 / 16), bd + (uint64_t)(k * UMMA_K * 2 / 16),
                                   kIdesc, (kb | k) != 0);
                    tc::commit(bar_empty + 8 * s);  // the stage is free once these have read it
                }
                // the accumulator is complete once every MMA above has
                tc::commit(bar_tfull + 8 * buf);
                if (!ok) break;
            }
        }
        __syncwarp();
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (its rows)
        const int wq = warp & 3, lb = 32 * wq;
        const uint32_t sbuf = stores + (uint32_t)(wq * 2) * kStoreBytes;
        int j = 0, nst = 0;
        for (int t = blockIdx.x; t < P.tiles; t += gridDim.x, ++j) {
            const int buf = j & 1;
            if (!mbar_wait(bar_tfull + 8 * buf, (uint32_t)(j >> 1) & 1u, abort_flag)) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            if (*abort_flag) break;
            tc::fence_after();
            const int m0 = (t / kNTiles) * BM, n0 = (t % kNTiles) * BN;
            const int row = lb + lane, m = m0 + row;
            const int pos = m < P.M ? m % P.T : 0;
            // the (cos, sin) row of this token's position, read once for all
            // rotated heads of the tile (every tile holds at least one)
            float4 cs[kPairs / 2];
            if (P.rope) {
                const float4* tr = reinterpret_cast<const float4*>(P.rope + (size_t)pos * kPairs);
#pragma unroll
                for (int j2 = 0; j2 < kPairs / 2; ++j2) cs[j2] = __ldg(tr + j2);
            }
#pragma unroll 1
            for (int h = 0; h < BN / kD; ++h) {
                uint32_t xu[32], yu[32];
                const uint32_t ta = tmem + ((uint32_t)lb << 16) + (uint32_t)(buf * BN + h * kD);
                tc::ld_x32(ta, xu);
                tc::ld_x32(ta + kPairs, yu);
                tc::wait_ld();
                float x[32], y[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    x[j] = __uint_as_float(xu[j]);
                    y[j] = __uint_as_float(yu[j]);
                }
                if (h == BN / kD - 1) {
                    // every column of this accumulator has been read: hand it back
                    tc::fence_before();
                    __syncwarp();
                    mbar_arrive_if(bar_tempty + 8 * buf, lane == 0);
                }
                const int hh = (n0 + h * kD) / kD;  // Q heads 0..7, K heads 8..9, V heads 10..11
                const CUtensorMap* map;
                int col;
                bool rot = P.rope != nullptr;
                if (hh < kHq) {
                    map = &P.qmap;
                    col = hh * kD;
                } else if (hh < kHq + kHkv) {
                    map = &P.kmap;
                    col = (hh - kHq) * kD;
                } else {
                    map = &P.vmap;
                    col = (hh - kHq - kHkv) * kD;
                    rot = false;
                }
                if (rot) {
#pragma unroll
                    for (int j2 = 0; j2 < kPairs / 2; ++j2) {
                        const float4 c = cs[j2];  // pairs 2 j2, 2 j2 + 1
                        const float x0 = x[2 * j2], y0 = y[2 * j2], x1 = x[2 * j2 + 1], y1 = y[2 * j2 + 1];
                        x[2 * j2] = __fmaf_rn(x0, c.x, __fmul_rn(-y0, c.y));
                        y[2 * j2] = __fmaf_rn(y0, c.x, __fmul_rn(x0, c.y));
                        x[2 * j2 + 1] = __fmaf_rn(x1, c.z, __fmul_rn(-y1, c.w));
                        y[2 * j2 + 1] = __fmaf_rn(y1, c.z, __fmul_rn(x1, c.w));
                    }
                }
                // stage the warp's 32 rows (row = lane, 128 bytes, 16-byte chunk c
                // at c ^ (lane & 7): the 128-byte swizzle of the store map)
                const uint32_t sb = sbuf + (uint32_t)(nst & 1) * kStoreBytes;
                if (lane == 0) bulk_wait_read1();  // the store that last used this buffer has read it
                __syncwarp();
                const uint32_t rb = sb + (uint32_t)lane * 128u;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    sts_u4(rb + (uint32_t)(((c ^ lane) & 7) << 4), pack_bf16(x[8 * c], x[8 * c + 1]),
                           pack_bf16(x[8 * c + 2], x[8 * c + 3]), pack_bf16(x[8 * c + 4], x[8 * c + 5]),
                           pack_bf16(x[8 * c + 6], x[8 * c + 7]));
                    sts_u4(rb + (uint32_t)((((4 + c) ^ lane) & 7) << 4), pack_bf16(y[8 * c], y[8 * c + 1]),
                           pack_bf16(y[8 * c + 2], y[8 * c + 3]), pack_bf16(y[8 * c + 4], y[8 * c + 5]),
                           pack_bf16(y[8 * c + 6], y[8 * c + 7]));
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0 && m0 + lb < P.M) {
                    tma_store_2d(map, sb, col, m0 + lb);  // rows past M are not written
                    bulk_commit();
                }
                ++nst;
            }
        }
        if (lane == 0) bulk_wait_all();
        if (*abort_flag && lane == 0 && warp == 2 && P.status) atomicOr(P.status, SFA_DEVSTAT_WAIT_TIMEOUT);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
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

// 2-D map over a row-major bf16 matrix [rows][cols], box of 64 columns x
// box_rows rows, 128-byte swizzle, zero fill outside (loads) / clipped (stores).
bool encode_matrix(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
    auto fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_qkv_rope(int M, int T, int dm, const void* x, const void* w, const float2* rope, void* q,
                            void* k, void* v, unsigned* status, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    QkvParams P;
    std::memset(&P, 0, sizeof(P));
    if (!encode_matrix(&P.xmap, x, M, dm, BM) || !encode_matrix(&P.wmap, w, kQkvRows, dm, BN) ||
        !encode_matrix(&P.qmap, q, M, kHq * kD, 32) || !encode_matrix(&P.kmap, k, M, kHkv * kD, 32) ||
        !encode_matrix(&P.vmap, v, M, kHkv * kD, 32))
        return cudaErrorInvalidValue;
    P.rope = rope;
    P.status = status;
    P.M = M;
    P.T = T;
    P.nkb = dm / BK;
    P.tiles = ((M + BM - 1) / BM) * kNTiles;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = ring::sm_count(dev, &e);
    if (e != cudaSuccess) return e;
    static CtxSetting configured[64];
    if (!ctx_setting_holds(configured[dev & 63], kSmemBytes)) {
        e = cudaFuncSetAttribute(qkv_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        ctx_setting_done(configured[dev & 63], kSmemBytes);
    }
    const int grid = P.tiles < sms ? P.tiles : sms;
    qkv_rope_kernel<<<grid, kThreads, kSmemBytes, s>>>(P);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace sfa
