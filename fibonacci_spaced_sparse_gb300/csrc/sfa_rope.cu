// sfa_rope.cu -- the RoPE table: (cos, sin) of pos * theta^(-2m/D) for every
// position and pair, angles and trigonometry in double, stored as float pairs.
// RoPE at the true positions, before the gather: section 2 "Attended set" of
// "Depth-Staggered Fibonacci Spacing for Sparse Attention"; base theta = 1e4
// in section 3 "Model and training".
#include "sfa_internal.cuh"

namespace sfa {

__global__ void rope_table_kernel(float2* __restrict__ table, int T, int half, int D, double theta) {
    const long long n = (long long)T * half;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const int pos = (int)(e / half);
        const int m = (int)(e % half);
        const double w = pow(theta, -2.0 * (double)m / (double)D);
        double s, c;
        sincos((double)pos * w, &s, &c);
        table[e] = make_float2((float)c, (float)s);
    }
}

cudaError_t launch_rope_table(float2* table, int T, int D, double theta, cudaStream_t s) {
    const int half = D / 2;
    const long long n = (long long)T * half;
    const int threads = 256;
    long long blocks = (n + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    rope_table_kernel<<<(unsigned)blocks, threads, 0, s>>>(table, T, half, D, theta);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace sfa
