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

}  // namespace

cudaError_t launch_decode(const LayerArgs& a, int Tc, sfa_dtype dt, const void* q, const void* kc,
                          const void* vc, const int* pos, const float2* rope, void* o, float* lse,
                          unsigned* status, cudaStream_t s) {
    const int blocks = a.B * kHkv;
    if (dt == SFA_F32)
        decode_kernel<float><<<blocks, kSplit * 32, 0, s>>>(a, Tc, (const float*)q, (const float*)kc,
                                                            (const float*)vc, pos, rope, (float*)o, lse,
                                                            status);
    else
        decode_kernel<__nv_bfloat16><<<blocks, kSplit * 32, 0, s>>>(
            a, Tc, (const __nv_bfloat16*)q, (const __nv_bfloat16*)kc, (const __nv_bfloat16*)vc, pos, rope,
            (__nv_bfloat16*)o, lse, status);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace sfa
