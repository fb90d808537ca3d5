// sfa_api.cu -- the C ABI of libsfa (declared in include/sfa.h): argument
// validation, the per-layer rung preparation, and kernel dispatch.
//
// Method: "Depth-Staggered Fibonacci Spacing for Sparse Attention"
// (arXiv 2606.28560), section 2 "Method" -- the attended set (window 0..W plus
// rungs at d_k = alpha f_k read by interpolation) and the per-layer scalar
// alpha = 0.5 + sigmoid(theta).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda.h>

#include "sfa.h"
#include "sfa_internal.cuh"

namespace sfa {

static std::atomic<unsigned long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

void* driver_entry(const char* name, int version) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return fn;
}

}  // namespace

// The driver's context id (cuCtxGetId, unique for the life of the process),
// plus one so that a valid id never reads as "no context".
unsigned long long context_key() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static const GetCurrent get_current = reinterpret_cast<GetCurrent>(driver_entry("cuCtxGetCurrent", 4000));
    static const GetId get_id = reinterpret_cast<GetId>(driver_entry("cuCtxGetId", 12000));
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    if (get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id + 1;
}

// Test hook: SFA_TEST_FAULT=launch in the environment (read once) makes every
// entry point fail with SFA_ERR_CUDA after its argument checks, before it
// touches the GPU, so that callers' error paths can be exercised without a
// device fault.
bool fault_injected() {
    static const bool on = [] {
        const char* e = std::getenv("SFA_TEST_FAULT");
        return e && std::strcmp(e, "launch") == 0;
    }();
    return on;
}

}  // namespace sfa

using sfa::LayerArgs;
using sfa::Rung;

namespace {

constexpr int kMaxT = 1 << 24;  // positions stay exact in fp32
// B * T cap: every tile, row and thread index of the kernels stays far inside
// 32 bits, and Q and O alone at this size (512 GiB in bf16) exceed the memory
// of one GPU, so no shape that fits is turned away.
constexpr long long kMaxTokens = 1LL << 28;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape and value checks shared by every entry point.
sfa_status validate(const sfa_params* p) {
    if (!p) return SFA_ERR_INVALID_ARG;
    if (p->B < 0 || p->T < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0 || p->W < 0)
        return SFA_ERR_INVALID_ARG;
    if (p->K < 0 || p->K > SFA_MAX_RUNGS || (p->K > 0 && !p->rungs)) return SFA_ERR_INVALID_ARG;
    for (int k = 0; k < p->K; ++k)
        if (!std::isfinite(p->rungs[k]) || !(p->rungs[k] > 0.f)) return SFA_ERR_INVALID_ARG;
    if (!std::isfinite(p->alpha) || !(p->alpha > 0.f)) return SFA_ERR_INVALID_ARG;
    if (!std::isfinite(p->rope_theta) || !std::isfinite(p->scale) || p->scale < 0.f)
        return SFA_ERR_INVALID_ARG;
    if (p->dtype != SFA_F32 && p->dtype != SFA_BF16) return SFA_ERR_INVALID_ARG;
    if (p->round_offsets != 0 && p->round_offsets != 1) return SFA_ERR_INVALID_ARG;
    if (p->Hq != sfa::kHq || p->Hkv != sfa::kHkv || p->D != sfa::kD) return SFA_ERR_UNSUPPORTED;
    if (p->T > kMaxT || (long long)p->B * p->T > kMaxTokens) return SFA_ERR_UNSUPPORTED;
    return SFA_OK;
}

// Rung preparation ("Attended set"): d = fl32(alpha) * fl32(f) rounded to
// nearest; rungs with d <= W are dropped (inside the window); rungs whose
// ceil(d) exceeds T - 1 are masked for every query and are left out too.  The
// kept rungs are ordered by increasing distance.
int rung_plan(const sfa_params* p, Rung* out) {
    int n = 0;
    for (int k = 0; k < p->K; ++k) {
        volatile float d = p->alpha * p->rungs[k];
        // rounded mode: the nearest integer, halves up (computed in double on
        // the fp32 product)
        const float dv = p->round_offsets ? (float)std::floor((double)d + 0.5) : (float)d;
        if (!(dv > (float)p->W)) continue;
        if (dv >= (float)p->T) continue;  // ceil(d) >= T: masked for all i < T
        const float fl = std::floor(dv);
        const float ce = std::ceil(dv);
        if ((int)ce > p->T - 1) continue;
        Rung r;
        r.n = (int)fl;
        r.t = dv - fl;  // exact: fl and dv share the exponent range
        r.c = (int)ce;
        r.f = p->round_offsets ? 0.f : p->rungs[k];  // d d / d alpha (zero once rounded)
        r.index = k;
        // insertion by increasing distance (stable): the rungs a query tile can
        // use are then a prefix of the list
        int pos = n++;
        while (pos > 0 && (out[pos - 1].n > r.n || (out[pos - 1].n == r.n && out[pos - 1].t > r.t))) {
            out[pos] = out[pos - 1];
            --pos;
        }
        out[pos] = r;
    }
    return n;
}

void fill_args(const sfa_params* p, LayerArgs* a) {
    std::memset(a, 0, sizeof(*a));
    a->B = p->B;
    a->T = p->T;
    a->W = p->W;
    a->scale = p->scale > 0.f ? p->scale : 1.0f / std::sqrt((float)p->D);
    a->alpha = p->alpha;
    a->nr = rung_plan(p, a->r);
}

const float2* rope_ptr(const sfa_params* p, const float* table) {
    return p->rope_theta > 0.f ? reinterpret_cast<const float2*>(table) : nullptr;
}

// The bf16 forward runs on the tensor-core kernel; fp32, and windows wider
// than that kernel takes, run on the fp32-arithmetic kernel.
// SFA_FORWARD_KERNEL=simple in the environment selects the fp32-arithmetic
// kernel for bf16 too (read once), to compare the two on the same inputs.
bool use_mma(const sfa_params* p, const LayerArgs& a) {
    static const bool force_simple = [] {
        const char* e = std::getenv("SFA_FORWARD_KERNEL");
        return e && std::strcmp(e, "simple") == 0;
    }();
    return p->dtype == SFA_BF16 && sfa::fwd_mma_supported(a) && !force_simple;
}

// The bf16 backward runs on the tensor-core kernels for windows the forward
// kernel also takes; SFA_BACKWARD_KERNEL=simple selects the fp32-arithmetic
// kernel (read once), to compare the two on the same inputs.
bool use_bwd_mma(const sfa_params* p, const LayerArgs& a) {
    static const bool force_simple = [] {
        const char* e = std::getenv("SFA_BACKWARD_KERNEL");
        return e && std::strcmp(e, "simple") == 0;
    }();
    return p->dtype == SFA_BF16 && sfa::bwd_mma_supported(a) && !force_simple;
}

sfa_status launched(cudaError_t e) {
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

// Checks of one forward call's tensors (shared by the single- and
// multi-layer entry points).
sfa_status check_forward_ptrs(const sfa_params* p, const void* Q, const void* K, const void* V,
                                     const float* rope_table, const void* O, const float* lse) {
    if (!Q || !K || !V || !O || !aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
        return SFA_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SFA_ERR_INVALID_ARG;
    if (p->rope_theta > 0.f && (!rope_table || !aligned16(rope_table))) return SFA_ERR_INVALID_ARG;
    return SFA_OK;
}

size_t align256_host(size_t x) { return (x + 255) & ~(size_t)255; }

// The multi-layer forward runs the attention launches back to back and lets
// each one rotate the next layer's keys (two rotated-key buffers in turn)
// when every layer takes the bf16 tensor-core path with RoPE.
bool layers_batched(const sfa_params* p, int L, const int* windows) {
    for (int l = 0; l < L; ++l) {
        sfa_params pl = *p;
        if (windows) pl.W = windows[l];
        LayerArgs a;
        fill_args(&pl, &a);
        if (!use_mma(&pl, a)) return false;
    }
    return p->rope_theta > 0.f;
}

}  // namespace

extern "C" {

SFA_API int sfa_version(void) { return (1 << 16) | 0; }

SFA_API const char* sfa_strerror(sfa_status s) {
    switch (s) {
        case SFA_OK: return "ok";
        case SFA_ERR_INVALID_ARG: return "invalid argument";
        case SFA_ERR_UNSUPPORTED: return "unsupported shape (Hq=8, Hkv=2, D=64 only)";
        case SFA_ERR_CUDA: return "CUDA launch or runtime error";
        case SFA_ERR_DEVICE_STATUS: return "a kernel reported a device-side error";
    }
    return "unknown status";
}

SFA_API unsigned long long sfa_launch_count(void) {
    return sfa::g_launches.load(std::memory_order_relaxed);
}

SFA_API float sfa_alpha_from_theta(float theta) {
    const double th = (double)theta;
    return (float)(0.5 + 1.0 / (1.0 + std::exp(-th)));
}

SFA_API sfa_status sfa_alpha_schedule(sfa_schedule kind, int L, int S, const float* theta,
                                      float* alpha_out) {
    if (L <= 0 || !alpha_out) return SFA_ERR_INVALID_ARG;
    switch (kind) {
        case SFA_SCHEDULE_FIXED:
            for (int l = 0; l < L; ++l) alpha_out[l] = 1.0f;
            return SFA_OK;
        case SFA_SCHEDULE_LEARNED:
            if (!theta) return SFA_ERR_INVALID_ARG;
            for (int l = 0; l < L; ++l) {
                if (!std::isfinite(theta[l])) return SFA_ERR_INVALID_ARG;
                alpha_out[l] = sfa_alpha_from_theta(theta[l]);
            }
            return SFA_OK;
        case SFA_SCHEDULE_LINEAR:
        case SFA_SCHEDULE_COPRIME: {
            if (L < 2) return SFA_ERR_INVALID_ARG;
            int stride = 1;
            if (kind == SFA_SCHEDULE_COPRIME) {
                if (S <= 0) return SFA_ERR_INVALID_ARG;
                int a = S % L, b = L;
                while (a) { int t = b % a; b = a; a = t; }
                if (b != 1) return SFA_ERR_INVALID_ARG;  // gcd(S, L) must be 1
                stride = S;
            }
            for (int l = 0; l < L; ++l) {
                const long long slot = ((long long)stride * l) % L;
                alpha_out[l] = (float)(0.5 + (double)slot / (double)(L - 1));
            }
            return SFA_OK;
        }
    }
    return SFA_ERR_INVALID_ARG;
}

SFA_API sfa_status sfa_rung_plan(const sfa_params* p, int* n_active, int* index, int* n_floor,
                                 float* frac, int* n_ceil) {
    sfa_status st = validate(p);
    if (st != SFA_OK) return st;
    if (!n_active) return SFA_ERR_INVALID_ARG;
    Rung r[SFA_MAX_RUNGS];
    const int n = rung_plan(p, r);
    *n_active = n;
    for (int i = 0; i < n; ++i) {
        if (index) index[i] = r[i].index;
        if (n_floor) n_floor[i] = r[i].n;
        if (frac) frac[i] = r[i].t;
        if (n_ceil) n_ceil[i] = r[i].c;
    }
    return SFA_OK;
}

SFA_API size_t sfa_rope_table_floats(int T, int D) {
    if (T <= 0 || D <= 0 || (D & 1)) return 0;
    return (size_t)T * (size_t)D;
}

SFA_API sfa_status sfa_rope_table(float* table, int T, int D, float rope_theta,
                                  cudaStream_t stream) {
    if (!table || !aligned16(table) || T < 0 || D <= 0 || (D & 1) || T > kMaxT ||
        !std::isfinite(rope_theta) || !(rope_theta > 0.f))
        return SFA_ERR_INVALID_ARG;
    if (T == 0) return SFA_OK;
    if (sfa::fault_injected()) return SFA_ERR_CUDA;
    return launched(sfa::launch_rope_table(reinterpret_cast<float2*>(table), T, D,
                                           (double)rope_theta, stream));
}

SFA_API size_t sfa_forward_workspace_size(const sfa_params* p) {
    if (validate(p) != SFA_OK) return 0;
    LayerArgs a;
    fill_args(p, &a);
    return use_mma(p, a) ? sfa::fwd_mma_workspace(a, p->rope_theta > 0.f) : 0;
}

SFA_API sfa_status sfa_forward(const sfa_params* p, const void* Q, const void* K, const void* V,
                               const float* rope_table, void* O, float* lse, void* workspace,
                               size_t workspace_bytes, unsigned int* status, cudaStream_t stream) {
    sfa_status st = validate(p);
    if (st != SFA_OK) return st;
    if (p->B == 0 || p->T == 0) return SFA_OK;
    if ((st = check_forward_ptrs(p, Q, K, V, rope_table, O, lse)) != SFA_OK) return st;
    LayerArgs a;
    fill_args(p, &a);
    if (use_mma(p, a)) {
        const size_t need = sfa::fwd_mma_workspace(a, p->rope_theta > 0.f);
        if (need && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
                     workspace_bytes < need))
            return SFA_ERR_INVALID_ARG;
        if (sfa::fault_injected()) return SFA_ERR_CUDA;
        return launched(sfa::launch_fwd_mma(a, Q, K, V, rope_ptr(p, rope_table), O, lse, workspace,
                                            status, stream));
    }
    if (sfa::fault_injected()) return SFA_ERR_CUDA;
    return launched(sfa::launch_fwd_simple(a, p->dtype, Q, K, V, rope_ptr(p, rope_table), O, lse,
                                           stream));
}

SFA_API size_t sfa_forward_layers_workspace_size(const sfa_params* p, int L, const int* windows) {
    if (validate(p) != SFA_OK || L <= 0) return 0;
    size_t need = 0;
    for (int l = 0; l < L; ++l) {
        sfa_params pl = *p;
        if (windows) pl.W = windows[l];
        if (pl.W < 0) return 0;
        const size_t n = sfa_forward_workspace_size(&pl);
        if (n > need) need = n;
    }
    // two rotated-key buffers, used in turn
    return layers_batched(p, L, windows) ? 2 * align256_host(need) : need;
}

SFA_API sfa_status sfa_forward_layers(const sfa_params* p, int L, const float* alphas, const int* windows,
                                      const void* const* Q, const void* const* K, const void* const* V,
                                      const float* rope_table, void* const* O, float* const* lse,
                                      void* workspace, size_t workspace_bytes, unsigned int* status,
                                      cudaStream_t stream) {
    sfa_status st = validate(p);
    if (st != SFA_OK) return st;
    if (L <= 0 || !alphas || !Q || !K || !V || !O) return SFA_ERR_INVALID_ARG;
    for (int l = 0; l < L; ++l) {
        sfa_params pl = *p;
        pl.alpha = alphas[l];
        if (windows) pl.W = windows[l];
        if ((st = validate(&pl)) != SFA_OK) return st;
        if (p->B > 0 && p->T > 0 &&
            (st = check_forward_ptrs(&pl, Q[l], K[l], V[l], rope_table, O[l], lse ? lse[l] : nullptr)) != SFA_OK)
            return st;
    }
    if (p->B == 0 || p->T == 0) return SFA_OK;
    const size_t need = sfa_forward_layers_workspace_size(p, L, windows);
    if (need && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need))
        return SFA_ERR_INVALID_ARG;
    if (sfa::fault_injected()) return SFA_ERR_CUDA;
    if (!layers_batched(p, L, windows)) {
        for (int l = 0; l < L; ++l) {
            sfa_params pl = *p;
            pl.alpha = alphas[l];
            if (windows) pl.W = windows[l];
            st = sfa_forward(&pl, Q[l], K[l], V[l], rope_table, O[l], lse ? lse[l] : nullptr, workspace,
                             workspace_bytes, status, stream);
            if (st != SFA_OK) return st;
        }
        return SFA_OK;
    }
    const size_t khat_bytes = need / 2;
    char* ws[2] = {static_cast<char*>(workspace), static_cast<char*>(workspace) + khat_bytes};
    const float2* rope = reinterpret_cast<const float2*>(rope_table);
    LayerArgs a;
    {
        sfa_params pl = *p;
        pl.alpha = alphas[0];
        if (windows) pl.W = windows[0];
        fill_args(&pl, &a);
        if ((st = launched(sfa::launch_rope_k(a, K[0], rope, ws[0], stream))) != SFA_OK) return st;
    }
    for (int l = 0; l < L; ++l) {
        sfa_params pl = *p;
        pl.alpha = alphas[l];
        if (windows) pl.W = windows[l];
        fill_args(&pl, &a);
        const bool more = l + 1 < L;
        st = launched(sfa::launch_fwd_attention(a, Q[l], ws[l & 1], V[l], rope, O[l], lse ? lse[l] : nullptr,
                                                more ? K[l + 1] : nullptr, more ? ws[(l + 1) & 1] : nullptr,
                                                status, true, stream));
        if (st != SFA_OK) return st;
    }
    return SFA_OK;
}

SFA_API sfa_status sfa_decode(const sfa_params* p, const void* Q, const void* Kc, const void* Vc,
                              const int* positions, const float* rope_table, void* O, float* lse,
                              unsigned int* status, cudaStream_t stream) {
    sfa_status st = validate(p);
    if (st != SFA_OK) return st;
    if (p->B == 0) return SFA_OK;
    if (p->T == 0) return SFA_ERR_INVALID_ARG;  // an empty cache holds no position
    if ((st = check_forward_ptrs(p, Q, Kc, Vc, rope_table, O, lse)) != SFA_OK) return st;
    if (!positions || (reinterpret_cast<uintptr_t>(positions) & 3u)) return SFA_ERR_INVALID_ARG;
    LayerArgs a;
    fill_args(p, &a);
    if (sfa::fault_injected()) return SFA_ERR_CUDA;
    return launched(sfa::launch_decode(a, p->T, p->dtype, Q, Kc, Vc, positions, rope_ptr(p, rope_table), O,
                                       lse, status, stream));
}

SFA_API sfa_status sfa_qkv_rope(const sfa_params* p, int d_model, const void* X, const void* Wqkv,
                                const float* rope_table, void* Qhat, void* Khat, void* V,
                                unsigned int* status, cudaStream_t stream) {
    sfa_status st = validate(p);
    if (st != SFA_OK) return st;
    if (p->dtype != SFA_BF16) return SFA_ERR_UNSUPPORTED;
    if (d_model < 64 || d_model > 16384 || d_model % 64 != 0) return SFA_ERR_INVALID_ARG;
    const long long M = (long long)p->B * p->T;
    if (M == 0) return SFA_OK;
    if (!X || !Wqkv || !Qhat || !Khat || !V || !aligned16(X) || !aligned16(Wqkv) || !aligned16(Qhat) ||
        !aligned16(Khat) || !aligned16(V))
        return SFA_ERR_INVALID_ARG;
    if (p->rope_theta > 0.f && (!rope_table || !aligned16(rope_table))) return SFA_ERR_INVALID_ARG;
    if (sfa::fault_injected()) return SFA_ERR_CUDA;
    return launched(sfa::launch_qkv_rope((int)M, p->T, d_model, X, Wqkv, rope_ptr(p, rope_table), Qhat, Khat,
                                         V, status, stream));
}

SFA_API sfa_status sfa_selftest_wait_timeout(unsigned int* status, cudaStream_t stream) {
    if (!status || (reinterpret_cast<uintptr_t>(status) & 3u)) return SFA_ERR_INVALID_ARG;
    if (sfa::fault_injected()) return SFA_ERR_CUDA;
    return launched(sfa::launch_wait_selftest(status, stream));
}

SFA_API size_t sfa_backward_workspace_size(const sfa_params* p) {
    if (validate(p) != SFA_OK) return 0;
    LayerArgs a;
    fill_args(p, &a);
    return use_bwd_mma(p, a) ? sfa::bwd_mma_workspace(a, p->rope_theta > 0.f) : sfa::bwd_simple_workspace(a);
}

SFA_API sfa_status sfa_backward(const sfa_params* p, const void* Q, const void* K, const void* V,
                                const void* O, const void* dO, const float* lse,
                                const float* rope_table, void* dQ, void* dK, void* dV,
                                float* dalpha, float* dtheta, void* workspace,
                                size_t workspace_bytes, unsigned int* status,
                                cudaStream_t stream) {
    sfa_status st = validate(p);
    if (st != SFA_OK) return st;
    if (!dalpha || !dtheta || (reinterpret_cast<uintptr_t>(dalpha) & 3u) ||
        (reinterpret_cast<uintptr_t>(dtheta) & 3u))
        return SFA_ERR_INVALID_ARG;
    LayerArgs a;
    fill_args(p, &a);
    if (p->B == 0 || p->T == 0) {
        if (sfa::fault_injected()) return SFA_ERR_CUDA;
        if (cudaMemsetAsync(dalpha, 0, sizeof(float), stream) != cudaSuccess ||
            cudaMemsetAsync(dtheta, 0, sizeof(float), stream) != cudaSuccess)
            return launched(cudaGetLastError());
        return SFA_OK;
    }
    const void* ptrs[] = {Q, K, V, O, dO, dQ, dK, dV};
    for (const void* q : ptrs)
        if (!q || !aligned16(q)) return SFA_ERR_INVALID_ARG;
    if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return SFA_ERR_INVALID_ARG;
    if (p->rope_theta > 0.f && (!rope_table || !aligned16(rope_table))) return SFA_ERR_INVALID_ARG;
    const bool mma = use_bwd_mma(p, a);
    const size_t need = mma ? sfa::bwd_mma_workspace(a, p->rope_theta > 0.f) : sfa::bwd_simple_workspace(a);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return SFA_ERR_INVALID_ARG;
    if (sfa::fault_injected()) return SFA_ERR_CUDA;
    if (mma)
        return launched(sfa::launch_bwd_mma(a, Q, K, V, O, dO, lse, rope_ptr(p, rope_table), dQ, dK, dV,
                                            dalpha, dtheta, workspace, status, stream));
    return launched(sfa::launch_bwd_simple(a, p->dtype, Q, K, V, O, dO, lse, rope_ptr(p, rope_table),
                                           dQ, dK, dV, dalpha, dtheta, workspace, stream));
}

SFA_API sfa_status sfa_read_status(const unsigned int* status, unsigned int* host_word,
                                   cudaStream_t stream) {
    if (!status) return SFA_ERR_INVALID_ARG;
    if (sfa::fault_injected()) return SFA_ERR_CUDA;
    unsigned int w = 0;
    if (cudaMemcpyAsync(&w, status, sizeof(w), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    if (host_word) *host_word = w;
    return w ? SFA_ERR_DEVICE_STATUS : SFA_OK;
}

}  // extern "C"
