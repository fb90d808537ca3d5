// sfa_bwd_simple.cu -- backward of the sparse attention, one warp per
// (sequence b, query i, key/value head g), fp32 arithmetic for every dtype.
//
// For every entry e of query i's key list (window rows and interpolated rung
// rows, section 2 "Attended set" of "Depth-Staggered Fibonacci Spacing for
// Sparse Attention") and query head h, with the forward's log-sum-exp:
//   p = exp(s - lse), dp = dO . vtilde, ds = p (dp - dO . o)
//   dqhat += scale ds ktilde
//   dkhat[row a] += (1 - t) scale ds qhat, dkhat[row b] += t scale ds qhat
//   dv[row a]    += (1 - t) p dO,          dv[row b]    += t p dO
//   dL/dt       += scale ds qhat . (khat_b - khat_a) + p dO . (v_b - v_a)
// The interpolation fraction t is what carries the gradient to alpha
// (section 2 "Implementation notes"); dd/dalpha = f, so
// dL/dalpha = sum_k f_k dL/dt_k and, with alpha = 0.5 + sigmoid(theta),
// dL/dtheta = dL/dalpha (alpha - 0.5)(1.5 - alpha) ("Per-layer scalar").
//
// Three launches: zero the fp32 accumulators, the main kernel (dQ directly,
// dK/dV by fp32 atomics in the rotated frame, dL/dt per block), and a finish
// kernel that undoes RoPE on dK, converts dK/dV, and reduces dL/dalpha in a
// fixed order (fp64).
#include "sfa_internal.cuh"

namespace sfa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct Workspace {
    float* dk;     // [B][T][Hkv][D] rotated-frame key gradient
    float* dv;     // [B][T][Hkv][D]
    float* dt;     // [blocks][SFA_MAX_RUNGS]
    long long blocks;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Workspace carve(const LayerArgs& a, void* base) {
    Workspace w;
    const size_t nkv = (size_t)a.B * a.T * kHkv * kD;
    w.blocks = ((long long)a.B * a.T * kHkv + kWarps - 1) / kWarps;
    char* p = static_cast<char*>(base);
    w.dk = reinterpret_cast<float*>(p);
    p += align256(nkv * sizeof(float));
    w.dv = reinterpret_cast<float*>(p);
    p += align256(nkv * sizeof(float));
    w.dt = reinterpret_cast<float*>(p);
    return w;
}

__global__ void zero_kernel(float4* __restrict__ x, long long n4) {
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n4;
         e += (long long)gridDim.x * blockDim.x)
        x[e] = make_float4(0.f, 0.f, 0.f, 0.f);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_simple_kernel(const LayerArgs a, const T* __restrict__ q, const T* __restrict__ k,
                  const T* __restrict__ v, const T* __restrict__ o, const T* __restrict__ dO,
                  const float* __restrict__ lse, const float2* __restrict__ rope,
                  T* __restrict__ dq, float* __restrict__ dk_acc, float* __restrict__ dv_acc,
                  float* __restrict__ dt_part) {
    __shared__ float dt_s[kWarps][SFA_MAX_RUNGS];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    dt_s[warp][lane] = 0.f;
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    if (gw < (long long)a.B * a.T * kHkv) {
        const int g = (int)(gw % kHkv);
        const int i = (int)((gw / kHkv) % a.T);
        const int b = (int)(gw / ((long long)kHkv * a.T));
        const size_t qbase = (((size_t)b * a.T + i) * kHq + g * kG) * kD + lane;
        const size_t lbase = ((size_t)b * a.T + i) * kHq + g * kG;
        const float2 csi = rope_cs(rope, i, lane);
        float qh0[kG], qh1[kG], do0[kG], do1[kG], Dh[kG], lse2[kG], dq0[kG], dq1[kG];
#pragma unroll
        for (int h = 0; h < kG; ++h) {
            const float x0 = to_f32(q[qbase + h * kD]), x1 = to_f32(q[qbase + h * kD + kPairs]);
            qh0[h] = x0 * csi.x - x1 * csi.y;
            qh1[h] = x1 * csi.x + x0 * csi.y;
            do0[h] = to_f32(dO[qbase + h * kD]);
            do1[h] = to_f32(dO[qbase + h * kD + kPairs]);
            Dh[h] = do0[h] * to_f32(o[qbase + h * kD]) + do1[h] * to_f32(o[qbase + h * kD + kPairs]);
            lse2[h] = lse[lbase + h] * kLog2e;
            dq0[h] = dq1[h] = 0.f;
        }
        warp_sum4(Dh);
        const float sl2 = a.scale * kLog2e;

        auto kv_off = [&](int j) { return (((size_t)b * a.T + j) * kHkv + g) * kD + lane; };
        auto load = [&](int j, float& k0, float& k1, float& v0, float& v1) {
            const size_t off = kv_off(j);
            const float x0 = to_f32(k[off]), x1 = to_f32(k[off + kPairs]);
            const float2 cs = rope_cs(rope, j, lane);
            k0 = x0 * cs.x - x1 * cs.y;
            k1 = x1 * cs.x + x0 * cs.y;
            v0 = to_f32(v[off]);
            v1 = to_f32(v[off + kPairs]);
        };

        // One entry: weight wa on row ra and wb on row rb (rb < 0: absent).
        // slot >= 0 marks a rung (accumulates dL/dt into dt_s[warp][slot]).
        auto entry = [&](int ra, float wa, int rb, float wb, int slot) {
            float ka0, ka1, va0, va1, kb0 = 0.f, kb1 = 0.f, vb0 = 0.f, vb1 = 0.f;
            load(ra, ka0, ka1, va0, va1);
            if (rb >= 0) load(rb, kb0, kb1, vb0, vb1);
            const float kt0 = wa * ka0 + wb * kb0, kt1 = wa * ka1 + wb * kb1;
            const float vt0 = wa * va0 + wb * vb0, vt1 = wa * va1 + wb * vb1;
            float s[kG], dp[kG];
#pragma unroll
            for (int h = 0; h < kG; ++h) {
                s[h] = qh0[h] * kt0 + qh1[h] * kt1;
                dp[h] = do0[h] * vt0 + do1[h] * vt1;
            }
            warp_sum4(s);
            warp_sum4(dp);
            float gk0 = 0.f, gk1 = 0.f, gv0 = 0.f, gv1 = 0.f;
#pragma unroll
            for (int h = 0; h < kG; ++h) {
                const float p = exp2f(s[h] * sl2 - lse2[h]);
                const float ds = p * (dp[h] - Dh[h]) * a.scale;
                dq0[h] += ds * kt0;
                dq1[h] += ds * kt1;
                gk0 += ds * qh0[h];
                gk1 += ds * qh1[h];
                gv0 += p * do0[h];
                gv1 += p * do1[h];
            }
            const size_t oa = kv_off(ra);
            atomicAdd(dk_acc + oa, wa * gk0);
            atomicAdd(dk_acc + oa + kPairs, wa * gk1);
            atomicAdd(dv_acc + oa, wa * gv0);
            atomicAdd(dv_acc + oa + kPairs, wa * gv1);
            if (rb >= 0 && wb != 0.f) {
                const size_t ob = kv_off(rb);
                atomicAdd(dk_acc + ob, wb * gk0);
                atomicAdd(dk_acc + ob + kPairs, wb * gk1);
                atomicAdd(dv_acc + ob, wb * gv0);
                atomicAdd(dv_acc + ob + kPairs, wb * gv1);
            }
            if (slot >= 0 && rb >= 0) {
                const float part = gk0 * (kb0 - ka0) + gk1 * (kb1 - ka1) + gv0 * (vb0 - va0) +
                                   gv1 * (vb1 - va1);
                const float tot = warp_sum(part);
                if (lane == 0) dt_s[warp][slot] += tot;
            }
        };

        const int wmax = min(a.W, i);
        for (int delta = 0; delta <= wmax; ++delta) entry(i - delta, 1.f, -1, 0.f, -1);
        for (int r = 0; r < a.nr; ++r) {
            const Rung R = a.r[r];
            if (i - R.c < 0) continue;
            const int ra = i - R.n;
            entry(ra, 1.f - R.t, ra - 1 >= 0 ? ra - 1 : -1, R.t, r);
        }
#pragma unroll
        for (int h = 0; h < kG; ++h) {
            // dQ = R(i)^T dqhat
            dq[qbase + h * kD] = from_f32<T>(dq0[h] * csi.x + dq1[h] * csi.y);
            dq[qbase + h * kD + kPairs] = from_f32<T>(dq1[h] * csi.x - dq0[h] * csi.y);
        }
    }
    __syncthreads();
    if (threadIdx.x < SFA_MAX_RUNGS) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += dt_s[w][threadIdx.x];
        dt_part[(size_t)blockIdx.x * SFA_MAX_RUNGS + threadIdx.x] = s;
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
bwd_finish_kernel(const LayerArgs a, const float* __restrict__ dk_acc,
                  const float* __restrict__ dv_acc, const float2* __restrict__ rope,
                  T* __restrict__ dk, T* __restrict__ dv, const float* __restrict__ dt_part,
                  long long nparts, float* __restrict__ dalpha, float* __restrict__ dtheta) {
    const long long npairs = (long long)a.B * a.T * kHkv * kPairs;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < npairs;
         e += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(e % kPairs);
        const long long row = e / kPairs;  // (b, j, g)
        const int j = (int)((row / kHkv) % a.T);
        const size_t base = (size_t)row * kD + m;
        const float x0 = dk_acc[base], x1 = dk_acc[base + kPairs];
        const float2 cs = rope_cs(rope, j, m);
        dk[base] = from_f32<T>(x0 * cs.x + x1 * cs.y);
        dk[base + kPairs] = from_f32<T>(x1 * cs.x - x0 * cs.y);
        dv[base] = from_f32<T>(dv_acc[base]);
        dv[base + kPairs] = from_f32<T>(dv_acc[base + kPairs]);
    }
    if (blockIdx.x != 0) return;
    __shared__ double red[256];
    double total = 0.0;  // meaningful in thread 0
    for (int r = 0; r < a.nr; ++r) {
        double s = 0.0;
        for (long long p = threadIdx.x; p < nparts; p += blockDim.x)
            s += (double)dt_part[(size_t)p * SFA_MAX_RUNGS + r];
        red[threadIdx.x] = s;
        __syncthreads();
        for (int w = blockDim.x / 2; w > 0; w >>= 1) {
            if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
            __syncthreads();
        }
        if (threadIdx.x == 0) total += (double)a.r[r].f * red[0];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double al = (double)a.alpha;
        *dalpha = (float)total;
        *dtheta = (float)(total * (al - 0.5) * (1.5 - al));
    }
}

}  // namespace

size_t bwd_simple_workspace(const LayerArgs& a) {
    const size_t nkv = (size_t)a.B * a.T * kHkv * kD;
    const long long blocks = ((long long)a.B * a.T * kHkv + kWarps - 1) / kWarps;
    return align256(nkv * sizeof(float)) * 2 + align256((size_t)blocks * SFA_MAX_RUNGS * sizeof(float));
}

cudaError_t launch_bwd_simple(const LayerArgs& a, sfa_dtype dt, const void* q, const void* k,
                              const void* v, const void* o, const void* dO, const float* lse,
                              const float2* rope, void* dq, void* dk, void* dv, float* dalpha,
                              float* dtheta, void* ws, cudaStream_t s) {
    Workspace w = carve(a, ws);
    const size_t nkv = (size_t)a.B * a.T * kHkv * kD;
    // the two accumulators are contiguous (nkv floats is a multiple of 64)
    const long long n4 = (long long)(reinterpret_cast<char*>(w.dt) - reinterpret_cast<char*>(w.dk)) / 16;
    (void)nkv;
    zero_kernel<<<1216, 256, 0, s>>>(reinterpret_cast<float4*>(w.dk), n4);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
    const unsigned blocks = (unsigned)w.blocks;
    const long long npairs = (long long)a.B * a.T * kHkv * kPairs;
    long long fblocks = (npairs + 255) / 256;
    if (fblocks > 152 * 16) fblocks = 152 * 16;
    if (dt == SFA_F32) {
        bwd_simple_kernel<float><<<blocks, kThreads, 0, s>>>(
            a, (const float*)q, (const float*)k, (const float*)v, (const float*)o,
            (const float*)dO, lse, rope, (float*)dq, w.dk, w.dv, w.dt);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
        bwd_finish_kernel<float><<<(unsigned)fblocks, 256, 0, s>>>(
            a, w.dk, w.dv, rope, (float*)dk, (float*)dv, w.dt, w.blocks, dalpha, dtheta);
    } else {
        using bf = __nv_bfloat16;
        bwd_simple_kernel<bf><<<blocks, kThreads, 0, s>>>(
            a, (const bf*)q, (const bf*)k, (const bf*)v, (const bf*)o, (const bf*)dO, lse, rope,
            (bf*)dq, w.dk, w.dv, w.dt);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
        bwd_finish_kernel<bf><<<(unsigned)fblocks, 256, 0, s>>>(
            a, w.dk, w.dv, rope, (bf*)dk, (bf*)dv, w.dt, w.blocks, dalpha, dtheta);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    count_launch();
    return cudaSuccess;
}

}  // namespace sfa
