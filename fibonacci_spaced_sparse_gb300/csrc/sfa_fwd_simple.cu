// sfa_fwd_simple.cu -- reference-grade forward kernel, one warp per
// (sequence b, query i, key/value head g), fp32 arithmetic for every dtype.
// Serves the fp32 path and any shape the tensor-core kernel does not take.
//
// Lane m holds the RoPE pair of dimensions (m, m + 32) of the four query heads
// that share key/value head g, so RoPE is a per-lane 2x2 rotation.  The key
// list of query i is walked in order: the window distances 0..W, then every
// kept rung (section 2 "Attended set" of "Depth-Staggered Fibonacci Spacing
// for Sparse Attention"): rows i - n (weight 1 - t) and i - n - 1 (weight t),
// masked while i - ceil(d) < 0.  Keys are rotated at their own positions
// before the interpolation.  One online softmax (base 2) runs over all entries.
#include "sfa_internal.cuh"

namespace sfa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T>
struct RowLoader {
    const T* __restrict__ k;
    const T* __restrict__ v;
    const float2* __restrict__ rope;
    int T_;
    int b, g, lane;

    __device__ __forceinline__ size_t off(int j) const {
        return (((size_t)b * T_ + j) * kHkv + g) * kD + lane;
    }
    // Rotated key pair and value pair of row j.
    __device__ __forceinline__ void load(int j, float& k0, float& k1, float& v0, float& v1) const {
        const size_t o = off(j);
        const float x0 = to_f32(k[o]), x1 = to_f32(k[o + kPairs]);
        const float2 cs = rope_cs(rope, j, lane);
        k0 = x0 * cs.x - x1 * cs.y;
        k1 = x1 * cs.x + x0 * cs.y;
        v0 = to_f32(v[o]);
        v1 = to_f32(v[o + kPairs]);
    }
};

template <typename T>
__global__ void __launch_bounds__(256)
fwd_simple_kernel(const LayerArgs a, const T* __restrict__ q, const T* __restrict__ k,
                  const T* __restrict__ v, const float2* __restrict__ rope, T* __restrict__ o,
                  float* __restrict__ lse) {
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw >= (long long)a.B * a.T * kHkv) return;  // whole warp leaves together
    const int g = (int)(gw % kHkv);
    const int i = (int)((gw / kHkv) % a.T);
    const int b = (int)(gw / ((long long)kHkv * a.T));

    const size_t qbase = (((size_t)b * a.T + i) * kHq + g * kG) * kD + lane;
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
    RowLoader<T> rows{k, v, rope, a.T, b, g, lane};

    auto consume = [&](float kt0, float kt1, float vt0, float vt1) {
        float s[kG];
#pragma unroll
        for (int h = 0; h < kG; ++h) s[h] = qh0[h] * kt0 + qh1[h] * kt1;
        warp_sum4(s);
#pragma unroll
        for (int h = 0; h < kG; ++h) {
            const float s2 = s[h] * sl2;
            const float mn = fmaxf(m[h], s2);
            const float corr = exp2f(m[h] - mn);
            const float pe = exp2f(s2 - mn);
            l[h] = l[h] * corr + pe;
            acc0[h] = acc0[h] * corr + pe * vt0;
            acc1[h] = acc1[h] * corr + pe * vt1;
            m[h] = mn;
        }
    };

    // window: distances 0..W
    const int wmax = min(a.W, i);
    for (int delta = 0; delta <= wmax; ++delta) {
        float k0, k1, v0, v1;
        rows.load(i - delta, k0, k1, v0, v1);
        consume(k0, k1, v0, v1);
    }
    // rungs
    for (int r = 0; r < a.nr; ++r) {
        const Rung R = a.r[r];
        if (i - R.c < 0) continue;
        const int ra = i - R.n;
        float ka0, ka1, va0, va1;
        rows.load(ra, ka0, ka1, va0, va1);
        if (R.t > 0.f) {
            float kb0, kb1, vb0, vb1;
            rows.load(ra - 1, kb0, kb1, vb0, vb1);
            const float wa = 1.f - R.t, wb = R.t;
            consume(wa * ka0 + wb * kb0, wa * ka1 + wb * kb1, wa * va0 + wb * vb0,
                    wa * va1 + wb * vb1);
        } else {
            consume(ka0, ka1, va0, va1);
        }
    }

#pragma unroll
    for (int h = 0; h < kG; ++h) {
        const float inv = 1.f / l[h];
        o[qbase + h * kD] = from_f32<T>(acc0[h] * inv);
        o[qbase + h * kD + kPairs] = from_f32<T>(acc1[h] * inv);
    }
    if (lse && lane < kG) {
        // lane h writes head h (values are warp-uniform)
        float mm = m[0], ll = l[0];
#pragma unroll
        for (int h = 1; h < kG; ++h)
            if (lane == h) { mm = m[h]; ll = l[h]; }
        lse[((size_t)b * a.T + i) * kHq + g * kG + lane] = (mm + log2f(ll)) * kLn2;
    }
}

}  // namespace

cudaError_t launch_fwd_simple(const LayerArgs& a, sfa_dtype dt, const void* q, const void* k,
                              const void* v, const float2* rope, void* o, float* lse,
                              cudaStream_t s) {
    const long long warps = (long long)a.B * a.T * kHkv;
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    if (dt == SFA_F32)
        fwd_simple_kernel<float><<<(unsigned)blocks, threads, 0, s>>>(
            a, (const float*)q, (const float*)k, (const float*)v, rope, (float*)o, lse);
    else
        fwd_simple_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, s>>>(
            a, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, rope,
            (__nv_bfloat16*)o, lse);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace sfa
