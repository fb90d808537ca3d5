// sfa_internal.cuh -- launch arguments and device helpers shared by the
// kernels of libsfa.  Private to the CUDA library (not installed, not part of
// the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sfa.h"

namespace sfa {

// Fixed attention shape of the paper (section 3 "Model and training"): 8 query
// heads sharing 2 key/value heads, head dimension 64.
constexpr int kHq = 8;
constexpr int kHkv = 2;
constexpr int kG = kHq / kHkv;  // query heads per key/value head
constexpr int kD = 64;
constexpr int kPairs = kD / 2;  // RoPE pairs (m, m + 32)

// One rung as the kernels use it: the distance d = alpha * f lies strictly
// beyond the window, floor(d) = n, t = d - n, ceil(d) = c (c = n when t = 0).
struct Rung {
    int n;
    float t;
    int c;
    float f;    // base offset, the derivative d d / d alpha
    int index;  // position in the caller's table
};

struct LayerArgs {
    int B, T, W;
    int nr;          // rungs kept (d > W and not masked for every query), by increasing d
    float scale;     // softmax scale
    float alpha;
    Rung r[SFA_MAX_RUNGS];
};

// Host: count of kernel launches made by the library.
void count_launch();

// Host: a key of the CUDA context current on the calling thread, unique for
// the life of the process (a context created after another one was destroyed,
// or by a device reset, never gets the old key); 0 when no context is current
// or the driver cannot say.  Set-up that lives in a context (kernel attributes,
// device addresses of library symbols) is recorded with this key and redone
// when the key differs.
unsigned long long context_key();

// Host: set-up of one kernel attribute value done in one context, per device.
struct CtxSetting {
    unsigned long long key;  // context_key() when it was done (0: never)
    size_t value;
};

// True when `s` records `value` or more, set in the context current now.
inline bool ctx_setting_holds(const CtxSetting& s, size_t value) {
    const unsigned long long k = context_key();
    return k != 0 && s.key == k && s.value >= value;
}

inline void ctx_setting_done(CtxSetting& s, size_t value) {
    s.value = value;
    s.key = context_key();
}

// SFA_TEST_FAULT=launch in the environment: entry points fail with
// SFA_ERR_CUDA after their argument checks, before they launch anything.
bool fault_injected();

// Launchers (each returns the launch error, if any).
cudaError_t launch_rope_table(float2* table, int T, int D, double theta, cudaStream_t s);

cudaError_t launch_fwd_simple(const LayerArgs& a, sfa_dtype dt, const void* q, const void* k,
                              const void* v, const float2* rope, void* o, float* lse,
                              cudaStream_t s);

bool fwd_mma_supported(const LayerArgs& a);
size_t fwd_mma_workspace(const LayerArgs& a, bool rope);
cudaError_t launch_fwd_mma(const LayerArgs& a, const void* q, const void* k, const void* v,
                           const float2* rope, void* o, float* lse, void* ws, unsigned* status,
                           cudaStream_t s);
cudaError_t launch_rope_k(const LayerArgs& a, const void* k, const float2* rope, void* khat, cudaStream_t s);
cudaError_t launch_fwd_attention(const LayerArgs& a, const void* q, const void* khat, const void* v,
                                 const float2* rope, void* o, float* lse, const void* k_next, void* khat_next,
                                 unsigned* status, bool pdl, cudaStream_t s);

// The tcgen05 forward (windows W <= 16, at most 10 kept rungs); the same
// arguments as launch_fwd_attention.
bool fwd_tc_supported(const LayerArgs& a);
cudaError_t launch_fwd_tc(const LayerArgs& a, const void* q, const void* khat, const void* v, const float2* rope,
                          void* o, float* lse, const void* k_next, void* khat_next, unsigned* status, bool pdl,
                          cudaStream_t s);

bool bwd_mma_supported(const LayerArgs& a);
size_t bwd_mma_workspace(const LayerArgs& a, bool rope);
cudaError_t launch_bwd_mma(const LayerArgs& a, const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, const float2* rope, void* dq, void* dk, void* dv,
                           float* dalpha, float* dtheta, void* ws, unsigned* status, cudaStream_t s);

cudaError_t launch_decode(const LayerArgs& a, int Tc, sfa_dtype dt, const void* q, const void* kc,
                          const void* vc, const int* pos, const float2* rope, void* o, float* lse,
                          unsigned* status, cudaStream_t s);

cudaError_t launch_qkv_rope(int M, int T, int dm, const void* x, const void* w, const float2* rope, void* q,
                            void* k, void* v, unsigned* status, cudaStream_t s);

cudaError_t launch_wait_selftest(unsigned* status, cudaStream_t s);

size_t bwd_simple_workspace(const LayerArgs& a);
cudaError_t launch_bwd_simple(const LayerArgs& a, sfa_dtype dt, const void* q, const void* k,
                              const void* v, const void* o, const void* dO, const float* lse,
                              const float2* rope, void* dq, void* dk, void* dv, float* dalpha,
                              float* dtheta, void* ws, cudaStream_t s);

// ------------------------------------------------------------ device helpers

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

constexpr unsigned kFull = 0xffffffffu;

// Sum over the 32 lanes of four per-lane values (one per query head of a
// key/value group); every lane receives all four sums.  Fixed order, so the
// result is deterministic.
__device__ __forceinline__ void warp_sum4(float v[4]) {
    const int lane = threadIdx.x & 31;
    const bool up16 = lane & 16;
    float keep0 = up16 ? v[2] : v[0], keep1 = up16 ? v[3] : v[1];
    const float send0 = up16 ? v[0] : v[2], send1 = up16 ? v[1] : v[3];
    keep0 += __shfl_xor_sync(kFull, send0, 16);
    keep1 += __shfl_xor_sync(kFull, send1, 16);
    const bool up8 = lane & 8;
    float keep = up8 ? keep1 : keep0;
    const float send = up8 ? keep0 : keep1;
    keep += __shfl_xor_sync(kFull, send, 8);
    keep += __shfl_xor_sync(kFull, keep, 4);
    keep += __shfl_xor_sync(kFull, keep, 2);
    keep += __shfl_xor_sync(kFull, keep, 1);
    v[0] = __shfl_sync(kFull, keep, 0);
    v[1] = __shfl_sync(kFull, keep, 8);
    v[2] = __shfl_sync(kFull, keep, 16);
    v[3] = __shfl_sync(kFull, keep, 24);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// (cos, sin) of pair m at position pos, identity without a table.
__device__ __forceinline__ float2 rope_cs(const float2* __restrict__ rope, int pos, int m) {
    return rope ? __ldg(rope + (size_t)pos * kPairs + m) : make_float2(1.f, 0.f);
}

}  // namespace sfa
