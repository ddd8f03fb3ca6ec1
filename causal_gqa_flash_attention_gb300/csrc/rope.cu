// rope.cu -- RoPE cos/sin table (the rotation of "NanoEuler: C와 CUDA로 밑바닥부터
// 구축한 GPT-2 규모의 LLM", 기술 사양, RoPE bullet): for position t and pair i the
// angle is t * theta^(-2i/D).  The angle is formed and reduced in fp64 (at t = 16384
// an fp32 angle would already be off by ~1e-3 rad) and stored as fp32.
#include "kernels.h"
#include "ptx.cuh"

namespace ne {

// ld >= half pairs per table row: pairs i >= half (the zero-padded head columns of a
// head_dim run on a wider kernel) get angle 0, i.e. (cos, sin) = (1, 0).
__global__ void rope_table_kernel(float* __restrict__ cos_out, float* __restrict__ sin_out,
                                  float2* __restrict__ interleaved, int T, int half, int ld, double theta,
                                  double inv_half) {
    griddep_launch_dependents();
    griddep_wait();   // an earlier kernel may still read a table this call overwrites
    const long long n = (long long)T * ld;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
         idx += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(idx / ld);
        const int i = (int)(idx % ld);
        double s = 0.0, c = 1.0;
        if (i < half) {
            // theta^(-2i/D) = theta^(-i/half)
            const double w = pow(theta, -(double)i * inv_half);
            sincos((double)t * w, &s, &c);
        }
        if (cos_out) cos_out[idx] = (float)c;
        if (sin_out) sin_out[idx] = (float)s;
        if (interleaved) interleaved[idx] = make_float2((float)c, (float)s);
    }
}

cudaError_t launch_rope_table(float* cos_out, float* sin_out, float2* interleaved, int T, int D,
                              double theta, cudaStream_t st, int ld) {
    const int half = D / 2;
    if (ld < half) ld = half;
    const long long n = (long long)T * ld;
    if (n == 0) return cudaSuccess;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    return launch_k(rope_table_kernel, dim3(blocks), dim3(256), 0, st, cos_out, sin_out, interleaved, T, half, ld,
                    theta, 1.0 / (double)half);
}

// A kernel whose only bounded wait can never complete: nothing arrives on its
// barrier.  It exercises the timeout path (error word + early exit) on demand.
__global__ void selftest_wait_kernel(int* err, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    WaitCtx w{err, &abort_flag, timeout_ns};
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, w, SITE_SELFTEST);
    __syncthreads();
}

cudaError_t launch_selftest_wait(int* err, unsigned long long timeout_ns, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace ne
