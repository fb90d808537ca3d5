// sfa_decode.cu -- single-token decode over a key/value cache: for every
// sequence b one new query at position i = pos[b] attends the cache rows of
// its key list ("Attended set", section 2 of "Depth-Staggered Fibonacci
// Spacing for Sparse Attention": the window distances 0..W and one
// interpolated row per rung, rows i - n (weight 1 - t) and i - n - 1
// (weight t), masked while i - ceil(d) < 0): the inference workload behind the
// paper's latency comparison of the interpolated gather (section 3 "Run
// matrix", section 4.3 "The learned scalar is ineffective").
//
// One CTA of kSplit warps per (sequence b, key/value head g); warp w takes
// the batches w, w + kSplit, ... of 8 consecutive entries of the key list
// (at most W + 1 + K entries, a rung entry reading two rows).  Lane m holds
// the RoPE pair of dimensions (m, m + 32) of the four query heads that share
// head g, so RoPE is a per-lane 2x2 rotation of the query at position i and
// of each cached key at its own position.  A warp loads its two dimensions of
// key and value for all 8 rows of a batch before consuming it, so the cache
// loads of a batch are in flight together; scores of the four heads are
// reduced across the warp (fixed order) and each warp keeps an online softmax
// (base 2).  The kSplit partial states are then merged in shared memory in a
// fixed order (the split of the flash-decoding kind).  Rows past pos[b] are
// never read.
#include "sfa_internal.cuh"

namespace sfa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kBatch = 8;         // entries gathered per batch
constexpr int kSplit = 4;         // warps per (sequence, key/value head)

// One entry of the key list: rows ra (weight wa) and rb (weight wb; rb < 0:
// no second row).
struct Entry {
    int ra, rb;
    float wa, wb;
};

// Entry e of query i: window distances first, then the rungs that apply.
__device__ __forceinline__ Entry entry_of(const LayerArgs& a, int i, int e, int nwin, const int* rung_list) {
    Entry x;
    if (e < nwin) {
        x.ra = i - e;
        x.rb = -1;
        x.wa = 1.f;
        x.wb = 0.f;
    } else {
        const Rung R = a.r[rung_list[e - nwin]];
        x.ra = i - R.n;
        x.rb = R.t > 0.f ? x.ra - 1 : -1;
        x.wa = 1.f - R.t;
        x.wb = R.t;
    }
    return x;
}

template <typename T>
__global__ void __launch_bounds__(kSplit * 32)
decode_kernel(const LayerArgs a, int Tc, const T* __restrict__ q, const T* __restrict__ kc,
              const T* __restrict__ vc, const int* __restrict__ pos, const float2* __restrict__ rope,
              T* __restrict__ o, float* __restrict__ lse, unsigned* __restrict__ status) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = blockIdx.x % kHkv, b = blockIdx.x / kHkv;
    // the next launch may be scheduled now; this one reads its inputs only
    // once the launch before it has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int i = __ldg(pos + b);
    const size_t qbase = ((size_t)b * kHq + g * kG) * kD + lane;
    if (i < 0 || i >= Tc) {
        // a position outside the cache: report it, read nothing, output zeros
        if (warp == 0) {
            if (lane == 0 && status) atomicOr(status, SFA_DEVSTAT_BAD_INDEX);
#pragma unroll
            for (int h = 0; h < kG; ++h) {
                o[qbase + h * kD] = from_f32<T>(0.f);
                o[qbase + h * kD + kPairs] = from_f32<T>(0.f);
            }
            if (lse && lane < kG) lse[(size_t)b * kHq + g * kG + lane] = 0.f;
        }
        return;  // the whole CTA leaves together
    }
    // rungs used by query i, in the order of the kept list
    __shared__ int rung_list[SFA_MAX_RUNGS];
    __shared__ float m_s[kSplit][kG], l_s[kSplit][kG];
    __shared__ float2 acc_s[kSplit][kG][32];
    int nrung = 0;
    for (int r = 0; r < a.nr; ++r)
        if (i - a.r[r].c >= 0) {
            if (threadIdx.x == 0) rung_list[nrung] = r;
            ++nrung;
        }
    __syncthreads();
    const int nwin = min(a.W, i) + 1;
    const int nent = nwin + nrung;

    const float2 csi = rope_cs(rope, i, lane);
    float qh0[kG], qh1[kG], m[kG], l[kG], acc0[kG], acc1[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
        const float x0 = to_f32(q[qbase + h * kD]), x1 = to_f32(q[qbase + h * kD + kPairs]);
        qh0[h] = x0 * csi.x - x1 * csi.y;
        qh1[h] = x1 * csi.x + x0 * csi.y;
        m[h] = -INFINITY;
        l[h] = 0.f;
        acc0[h] = acc1[h] = 0.f;
    }
    const float sl2 = a.scale * kLog2e;
    auto row_off = [&](int j) { return (((size_t)b * Tc + j) * kHkv + g) * kD + lane; };
    // rotated key pair and value pair of cache row j
    auto load = [&](int j, float& k0, float& k1, float& v0, float& v1) {
        const size_t off = row_off(j);
        const float x0 = to_f32(kc[off]), x1 = to_f32(kc[off + kPairs]);
        const float2 cs = rope_cs(rope, j, lane);
        k0 = x0 * cs.x - x1 * cs.y;
        k1 = x1 * cs.x + x0 * cs.y;
        v0 = to_f32(vc[off]);
        v1 = to_f32(vc[off + kPairs]);
    };

    for (int e0 = warp * kBatch; e0 < nent; e0 += kSplit * kBatch) {
        float kt0[kBatch], kt1[kBatch], vt0[kBatch], vt1[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            kt0[u] = kt1[u] = vt0[u] = vt1[u] = 0.f;
            if (e0 + u < nent) {
                const Entry x = entry_of(a, i, e0 + u, nwin, rung_list);
                float ka0, ka1, va0, va1;
                load(x.ra, ka0, ka1, va0, va1);
                kt0[u] = x.wa * ka0;
                kt1[u] = x.wa * ka1;
                vt0[u] = x.wa * va0;
                vt1[u] = x.wa * va1;
                if (x.rb >= 0) {
                    float kb0, kb1, vb0, vb1;
                    load(x.rb, kb0, kb1, vb0, vb1);
                    kt0[u] += x.wb * kb0;
                    kt1[u] += x.wb * kb1;
                    vt0[u] += x.wb * vb0;
                    vt1[u] += x.wb * vb1;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (e0 + u >= nent) break;
            float s[kG];
#pragma unroll
            for (int h = 0; h < kG; ++h) s[h] = qh0[h] * kt0[u] + qh1[h] * kt1[u];
            warp_sum4(s);
#pragma unroll
            for (int h = 0; h < kG; ++h) {
                const float s2 = s[h] * sl2;
                const float mn = fmaxf(m[h], s2);
                const float corr = exp2f(m[h] - mn);
                const float pe = exp2f(s2 - mn);
                l[h] = l[h] * corr + pe;
                acc0[h] = acc0[h] * corr + pe * vt0[u];
                acc1[h] = acc1[h] * corr + pe * vt1[u];
                m[h] = mn;
            }
        }
    }
    // merge the kSplit partial states (a warp without entries has m = -inf, l = 0)
#pragma unroll
    for (int h = 0; h < kG; ++h) {
        if (lane == 0) {
            m_s[warp][h] = m[h];
            l_s[warp][h] = l[h];
        }
        acc_s[warp][h][lane] = make_float2(acc0[h], acc1[h]);
    }
    __syncthreads();
    if (warp != 0) return;
#pragma unroll
    for (int h = 0; h < kG; ++h) {
        float mm = m_s[0][h];
        for (int w = 1; w < kSplit; ++w) mm = fmaxf(mm, m_s[w][h]);
        float ll = 0.f, a0 = 0.f, a1 = 0.f;
        for (int w = 0; w < kSplit; ++w) {
            const float c = l_s[w][h] > 0.f ? exp2f(m_s[w][h] - mm) : 0.f;
            ll += l_s[w][h] * c;
            const float2 av = acc_s[w][h][lane];
            a0 += av.x * c;
            a1 += av.y * c;
        }
        const float inv = 1.f / ll;
        o[qbase + h * kD] = from_f32<T>(a0 * inv);
        o[qbase + h * kD + kPairs] = from_f32<T>(a1 * inv);
        if (lse && lane == h) lse[(size_t)b * kHq + g * kG + h] = (mm + log2f(ll)) * kLn2;
    }
}

// ---------------------------------------------------------- bf16, W <= 16
//
// The key list of a query has at most W + 1 + K <= 32 entries here, so one
// CTA of four warps holds all of them at once: lane = (entry e of the warp's
// eight, 16-dimension chunk c).  Chunk c is the RoPE pairs m = 8c .. 8c + 7,
// i.e. dimensions 8c .. 8c + 7 and their partners 32 + 8c .. 32 + 8c + 7, two
// 16-byte pieces of a row, and the (cos, sin) of those pairs are 64
// contiguous bytes of the table row, so every load of a cache row is a
// 16-byte load and all of an entry's rows are in flight together.  A score is
// the sum of four lanes' partial dot products (two shuffles).  Each warp keeps
// the softmax state of its eight entries (their maximum, the exponentials and
// their sum against it); the value products of the 32 entries go through
// shared memory (entry stride padded so that the 16-byte writes of a warp hit
// distinct banks), and after the one block barrier every output is each
// warp's sum merged with the weights 2^(m_warp - m) of the four warps'
// maxima.  Each lane rotates the query chunk it scores with itself.
constexpr int kFastEntries = 32;
constexpr int kFastThreads = 128;
constexpr int kRedStride = 4 * kD + 4;  // floats per entry in the value-product buffer

__device__ __forceinline__ float2 bf2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// The raw words of chunk c of one entry row: Khat dimensions 8c .. 8c + 7 and
// their partners + 32, the same of V, and the (cos, sin) of those pairs.
// Fetched for every row of an entry before any of them is used, so that all
// of an entry's loads are in flight together.
struct RawRow {
    uint4 kx, ky, vx, vy;
    float4 cs[4];
};

__device__ __forceinline__ void fetch_row(const __nv_bfloat16* __restrict__ base,
                                          const __nv_bfloat16* __restrict__ vbase,
                                          const float2* __restrict__ rope, int pos, int c, RawRow& R) {
    R.kx = __ldg(reinterpret_cast<const uint4*>(base) + c);
    R.ky = __ldg(reinterpret_cast<const uint4*>(base) + 4 + c);
    R.vx = __ldg(reinterpret_cast<const uint4*>(vbase) + c);
    R.vy = __ldg(reinterpret_cast<const uint4*>(vbase) + 4 + c);
    if (rope) {
        const float4* t = reinterpret_cast<const float4*>(rope + (size_t)pos * kPairs + 8 * c);
#pragma unroll
        for (int j = 0; j < 4; ++j) R.cs[j] = __ldg(t + j);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) R.cs[j] = make_float4(1.f, 0.f, 1.f, 0.f);
    }
}

// Rotated (x, y) halves of the 8 pairs of a fetched row, and its values, fp32.
__device__ __forceinline__ void unpack_row(const RawRow& R, float (&x)[8], float (&y)[8], float (&v)[16]) {
    const uint32_t kxw[4] = {R.kx.x, R.kx.y, R.kx.z, R.kx.w}, kyw[4] = {R.ky.x, R.ky.y, R.ky.z, R.ky.w};
    const uint32_t vxw[4] = {R.vx.x, R.vx.y, R.vx.z, R.vx.w}, vyw[4] = {R.vy.x, R.vy.y, R.vy.z, R.vy.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 a = bf2(kxw[j]), b = bf2(kyw[j]);
        // pairs 2j, 2j + 1 of the chunk: (cos, sin) in cs[j].xy and cs[j].zw
        x[2 * j] = a.x * R.cs[j].x - b.x * R.cs[j].y;
        y[2 * j] = b.x * R.cs[j].x + a.x * R.cs[j].y;
        x[2 * j + 1] = a.y * R.cs[j].z - b.y * R.cs[j].w;
        y[2 * j + 1] = b.y * R.cs[j].z + a.y * R.cs[j].w;
        const float2 p = bf2(vxw[j]), q = bf2(vyw[j]);
        v[2 * j] = p.x;
        v[2 * j + 1] = p.y;
        v[8 + 2 * j] = q.x;
        v[8 + 2 * j + 1] = q.y;
    }
}

// Rows of entry e of a query at position i (ra < 0: no entry; rb < 0: no
// second row), as the kernel below assigns them.
__device__ __forceinline__ void entry_rows(const LayerArgs& a, int i, int e, int& ra, int& rb) {
    const int nwin = min(a.W, i) + 1;
    ra = rb = -1;
    if (e < nwin) {
        ra = i - e;
        return;
    }
    int k = e - nwin;
    for (int r = 0; r < a.nr; ++r)
        if (a.r[r].c <= i && k-- == 0) {
            ra = i - a.r[r].n;
            rb = a.r[r].t > 0.f ? ra - 1 : -1;
            return;
        }
}

// One 128-byte line of K and one of V of cache row j (head g) into L2.
__device__ __forceinline__ void prefetch_row(const __nv_bfloat16* kc, const __nv_bfloat16* vc, int b, int Tc, int g,
                                             int j) {
    const size_t off = (((size_t)b * Tc + j) * kHkv + g) * kD;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(kc + off));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(vc + off));
}

__global__ void __launch_bounds__(kFastThreads) decode_fast_kernel(
    const LayerArgs a, int Tc, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
    const __nv_bfloat16* __restrict__ vc, const int* __restrict__ pos, const float2* __restrict__ rope,
    __nv_bfloat16* __restrict__ o, float* __restrict__ lse, unsigned* __restrict__ status) {
    __shared__ __align__(16) float red[kFastEntries * kRedStride];  // p v per entry
    __shared__ float mw[4][kG], lw[4][kG];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x % kHkv, b = blockIdx.x / kHkv;
    const size_t qbase = ((size_t)b * kHq + g * kG) * kD;
    const int c = lane & 3, e = warp * 8 + (lane >> 2);
    // the next launch may be scheduled now; this one reads its inputs only
    // once the launch before it has completed.  While it waits, it asks L2 for
    // the cache rows of its entry at the position it reads now (clamped into
    // the cache): if the launch before rewrites the position, only these
    // prefetches go to other rows, and every value used is read after the wait
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (c == 0) {
        const int ip = min(max(*reinterpret_cast<const volatile int*>(pos + b), 0), Tc - 1);
        int ra, rb;
        entry_rows(a, ip, e, ra, rb);
        if (ra >= 0) prefetch_row(kc, vc, b, Tc, g, ra);
        if (rb >= 0) prefetch_row(kc, vc, b, Tc, g, rb);
    }
    if (threadIdx.x < kG) asm volatile("prefetch.global.L2 [%0];" ::"l"(q + qbase + threadIdx.x * kD));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the query's chunk c of every head (dimensions 8c .. 8c + 7 and their
    // partners), loaded together with the position; each lane rotates the
    // chunk it scores with itself, so no shared copy and no barrier is needed
    uint4 qxw[kG], qyw[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
        qxw[h] = __ldg(reinterpret_cast<const uint4*>(q + qbase + h * kD) + c);
        qyw[h] = __ldg(reinterpret_cast<const uint4*>(q + qbase + h * kD) + 4 + c);
    }
    const int i = __ldg(pos + b);
    if (i < 0 || i >= Tc) {
        // a position outside the cache: report it, read nothing, output zeros
        if (tid == 0 && status) atomicOr(status, SFA_DEVSTAT_BAD_INDEX);
        o[qbase + 2 * tid] = __float2bfloat16_rn(0.f);
        o[qbase + 2 * tid + 1] = __float2bfloat16_rn(0.f);
        if (lse && tid < kG) lse[(size_t)b * kHq + g * kG + tid] = 0.f;
        return;  // the whole CTA leaves together
    }
    // this lane's entry: window distances 0..min(W, i), then the rungs with
    // ceil(d) <= i (a prefix of the kept list, which is sorted by distance)
    const int nwin = min(a.W, i) + 1;
    int nact = 0;
    for (int r = 0; r < a.nr; ++r) nact += (a.r[r].c <= i) ? 1 : 0;
    const bool live = e < nwin + nact;
    int ra = i, rb = -1;
    float wa = 1.f, wb = 0.f;
    if (live && e >= nwin) {
        const Rung R = a.r[e - nwin];
        ra = i - R.n;
        rb = R.t > 0.f ? ra - 1 : -1;
        wa = 1.f - R.t;
        wb = R.t;
    } else if (live) {
        ra = i - e;
    }
    // every load of the entry's rows and of the query's (cos, sin) goes out
    // before any of them is used
    RawRow A, Bw;
    {
        const size_t off = (((size_t)b * Tc + ra) * kHkv + g) * kD;
        fetch_row(kc + off, vc + off, rope, ra, c, A);
    }
    if (rb >= 0) {
        const size_t off = (((size_t)b * Tc + rb) * kHkv + g) * kD;
        fetch_row(kc + off, vc + off, rope, rb, c, Bw);
    }
    float4 qcs[4];
    if (rope) {
        const float4* t = reinterpret_cast<const float4*>(rope + (size_t)i * kPairs + 8 * c);
#pragma unroll
        for (int j = 0; j < 4; ++j) qcs[j] = __ldg(t + j);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) qcs[j] = make_float4(1.f, 0.f, 1.f, 0.f);
    }
    float kx[8], ky[8], vv[16];
    unpack_row(A, kx, ky, vv);
    if (rb >= 0) {
        float bx[8], by[8], bv[16];
        unpack_row(Bw, bx, by, bv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            kx[j] = wa * kx[j] + wb * bx[j];
            ky[j] = wa * ky[j] + wb * by[j];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) vv[j] = wa * vv[j] + wb * bv[j];
    }
    const float sl2 = a.scale * kLog2e;
    float s[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
        const uint32_t xw[4] = {qxw[h].x, qxw[h].y, qxw[h].z, qxw[h].w};
        const uint32_t yw[4] = {qyw[h].x, qyw[h].y, qyw[h].z, qyw[h].w};
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // pairs 2j, 2j + 1 of the chunk, rotated at the query's position
            const float2 x = bf2(xw[j]), y = bf2(yw[j]);
            const float qx0 = x.x * qcs[j].x - y.x * qcs[j].y, qy0 = y.x * qcs[j].x + x.x * qcs[j].y;
            const float qx1 = x.y * qcs[j].z - y.y * qcs[j].w, qy1 = y.y * qcs[j].z + x.y * qcs[j].w;
            acc += qx0 * kx[2 * j] + qx1 * kx[2 * j + 1] + qy0 * ky[2 * j] + qy1 * ky[2 * j + 1];
        }
        acc += __shfl_xor_sync(kFull, acc, 1);
        acc += __shfl_xor_sync(kFull, acc, 2);
        s[h] = live ? acc * sl2 : -INFINITY;
    }
    // softmax state per warp (its eight entries): the warp's maximum, and the
    // exponentials and their sum against it; the four warps' states are
    // merged at the end (a warp whose entries are all past the list has
    // maximum -inf and weight 0; warp 0 holds entry 0, the query's own row,
    // which is always live)
    float p[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
        float m = s[h];
#pragma unroll
        for (int w = 4; w <= 16; w <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, w));
        p[h] = live ? exp2f(s[h] - m) : 0.f;
        float l = p[h];
#pragma unroll
        for (int w = 4; w <= 16; w <<= 1) l += __shfl_xor_sync(kFull, l, w);
        if (lane == 0) {
            mw[warp][h] = m;
            lw[warp][h] = l;
        }
    }
    // p v of this entry, chunk c, into the reduction buffer
    float* rr = red + e * kRedStride;
#pragma unroll
    for (int h = 0; h < kG; ++h) {
        float4* dx = reinterpret_cast<float4*>(rr + h * kD + 8 * c);
        float4* dy = reinterpret_cast<float4*>(rr + h * kD + kPairs + 8 * c);
        dx[0] = make_float4(p[h] * vv[0], p[h] * vv[1], p[h] * vv[2], p[h] * vv[3]);
        dx[1] = make_float4(p[h] * vv[4], p[h] * vv[5], p[h] * vv[6], p[h] * vv[7]);
        dy[0] = make_float4(p[h] * vv[8], p[h] * vv[9], p[h] * vv[10], p[h] * vv[11]);
        dy[1] = make_float4(p[h] * vv[12], p[h] * vv[13], p[h] * vv[14], p[h] * vv[15]);
    }
    __syncthreads();
    // thread (h, d): outputs d and d + 32 of head h -- each warp's entries
    // summed in order, the four sums merged with weights 2^(m_w - M)
    {
        const int h = tid >> 5, d = tid & 31;
        const float M = fmaxf(fmaxf(mw[0][h], mw[1][h]), fmaxf(mw[2][h], mw[3][h]));
        float o0 = 0.f, o1 = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float cw = mw[w][h] == -INFINITY ? 0.f : exp2f(mw[w][h] - M);
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int en = 8 * w; en < 8 * w + 8; ++en) {
                a0 += red[en * kRedStride + h * kD + d];
                a1 += red[en * kRedStride + h * kD + kPairs + d];
            }
            o0 = fmaf(cw, a0, o0);
            o1 = fmaf(cw, a1, o1);
            L = fmaf(cw, lw[w][h], L);
        }
        const float inv = 1.f / L;
        o[qbase + h * kD + d] = __float2bfloat16_rn(o0 * inv);
        o[qbase + h * kD + kPairs + d] = __float2bfloat16_rn(o1 * inv);
        if (lse && d == 0) lse[(size_t)b * kHq + g * kG + h] = (M + log2f(L)) * kLn2;
    }
}

}  // namespace

cudaError_t launch_decode(const LayerArgs& a, int Tc, sfa_dtype dt, const void* q, const void* kc,
                          const void* vc, const int* pos, const float2* rope, void* o, float* lse,
                          unsigned* status, cudaStream_t s) {
    // programmatic dependent launch: the CTAs of this launch may be scheduled
    // while the launch before it drains (they wait for it before any read),
    // which hides the gap between back-to-back decode calls
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * kHkv));
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (dt == SFA_BF16 && a.W + 1 + a.nr <= kFastEntries) {
        cfg.blockDim = dim3(kFastThreads);
        e = cudaLaunchKernelEx(&cfg, decode_fast_kernel, a, Tc, (const __nv_bfloat16*)q, (const __nv_bfloat16*)kc,
                               (const __nv_bfloat16*)vc, pos, rope, (__nv_bfloat16*)o, lse, status);
    } else if (dt == SFA_F32) {
        cfg.blockDim = dim3(kSplit * 32);
        e = cudaLaunchKernelEx(&cfg, decode_kernel<float>, a, Tc, (const float*)q, (const float*)kc,
                               (const float*)vc, pos, rope, (float*)o, lse, status);
    } else {
        cfg.blockDim = dim3(kSplit * 32);
        e = cudaLaunchKernelEx(&cfg, decode_kernel<__nv_bfloat16>, a, Tc, (const __nv_bfloat16*)q,
                               (const __nv_bfloat16*)kc, (const __nv_bfloat16*)vc, pos, rope, (__nv_bfloat16*)o,
                               lse, status);
    }
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace sfa
