// FP32 fused multiply-add throughput probe: the denominator of the gate's
// roofline where the gate is bound by fp32 arithmetic (e >= 16 experts: 2*m*e
// flop per token against 2*m bytes of x).  Not part of the layer.
//
// Every thread runs 8 independent two-wide accumulator chains, scalar fmaf
// pairs or packed fp32x2 fused multiply-adds (the gate's kernels use both),
// so the loop is issue-bound, not latency-bound.  acc <- acc * a + b with
// a = 1 - 2^-10 keeps every value finite and normal.
#include "common.cuh"

namespace moe {
namespace {

constexpr int PROBE_THREADS = 256;
constexpr int PROBE_CHAINS = 8;

template <bool PACKED>
__global__ void __launch_bounds__(PROBE_THREADS)
fma_probe_kernel(float *out, int iters, float a, float b) {
    float2 acc[PROBE_CHAINS];
#pragma unroll
    for (int i = 0; i < PROBE_CHAINS; i++)
        acc[i] = make_float2((float)(threadIdx.x + i), (float)(blockIdx.x + i));
    const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
    for (int it = 0; it < iters; it++) {
#pragma unroll
        for (int i = 0; i < PROBE_CHAINS; i++) {
            if (PACKED)
                acc[i] = __ffma2_rn(acc[i], a2, b2);
            else
                acc[i] = make_float2(__fmaf_rn(acc[i].x, a, b), __fmaf_rn(acc[i].y, a, b));
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < PROBE_CHAINS; i++) s += acc[i].x + acc[i].y;
    if (s == -1.0f) out[0] = s;   // keeps the chains live; never true for these values
}

}  // namespace

moe_status probe_fp32_fma_launch(int packed, int blocks, int iters, float *out,
                                 cudaStream_t stream) {
    const float a = 1.0f - 1.0f / 1024.0f, b = 1.0f / 1024.0f;
    if (packed)
        fma_probe_kernel<true><<<blocks, PROBE_THREADS, 0, stream>>>(out, iters, a, b);
    else
        fma_probe_kernel<false><<<blocks, PROBE_THREADS, 0, stream>>>(out, iters, a, b);
    note_launch();
    return launch_status();
}

}  // namespace moe
