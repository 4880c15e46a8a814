// e4m3 row quantisation for the low-precision experts.
//
// Method: the Tutel profile names FP8 (and blockwise FP8) among its inference
// formats without a block size; here every row of an operand carries one fp32
// scale, scale = amax / 448 (448 = the largest finite e4m3 magnitude), and
// each value is x / scale rounded to the nearest e4m3 code, ties to even,
// saturating at +-448.
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int QR_WARPS = 8;

// One warp per row: amax over the row (max is exact, so the lanes' maxima
// combine in any order), scale = amax / 448 in IEEE fp32 division (1 for an
// all-zero row), then every value divided by the scale (IEEE) and converted
// with the nearest-even, saturating e4m3x2 conversion.  With counts, rows of
// batch b past min(counts[b], *c_dev) are skipped.
__global__ void __launch_bounds__(QR_WARPS * 32)
quantize_rows_kernel(const __nv_bfloat16 *__restrict__ src, int64_t batches, int64_t rpb, int cols,
                     const int32_t *__restrict__ counts, const int32_t *__restrict__ c_dev,
                     uint8_t *__restrict__ q, float *__restrict__ scale, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = cols / 8;   // 16-byte chunks of a bf16 row (8 codes each)
    const int64_t total = batches * rpb;
    const int64_t c_eff = counts ? min((int64_t)*c_dev, rpb) : rpb;
    for (int64_t row = (int64_t)blockIdx.x * QR_WARPS + warp; row < total;
         row += (int64_t)gridDim.x * QR_WARPS) {
        if (counts) {
            const int64_t b = row / rpb, r = row - b * rpb;
            if (r >= min((int64_t)max(counts[b], 0), c_eff)) continue;   // uniform over the warp
        }
        const __nv_bfloat16 *xr = src + row * cols;
        float amax = 0.0f;
        for (int c = lane; c < nch; c += 32) {
            float f[8];
            Elt<__nv_bfloat16>::unpack(ld_v16(xr + 8 * c), f);
#pragma unroll
            for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(f[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        if (lane == 0) scale[row] = s;
        uint8_t *qr = q + row * cols;
        for (int c = lane; c < nch; c += 32) {
            float f[8];
            Elt<__nv_bfloat16>::unpack(ld_v16(xr + 8 * c), f);
            uint32_t w[2];
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const uint32_t lo = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(f[4 * i], s), __fdiv_rn(f[4 * i + 1], s)), __NV_SATFINITE,
                    __NV_E4M3);
                const uint32_t hi = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(f[4 * i + 2], s), __fdiv_rn(f[4 * i + 3], s)),
                    __NV_SATFINITE, __NV_E4M3);
                w[i] = (lo & 0xFFFFu) | (hi << 16);
            }
            *reinterpret_cast<uint2 *>(qr + 8 * c) = make_uint2(w[0], w[1]);
        }
    }
}

}  // namespace

moe_status quantize_rows_fp8_launch(const void *src, int64_t batches, int64_t rows_per_batch,
                                    int cols, const int32_t *counts, const int32_t *c_dev,
                                    void *q, float *scale, int32_t *st, cudaStream_t stream) {
    if (batches < 1 || rows_per_batch < 1 || cols < 16 || cols % 16) return MOE_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int64_t rows = batches * rows_per_batch;
    int64_t grid = (rows + QR_WARPS - 1) / QR_WARPS;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
    if (grid > cap) grid = cap;
    return launch_pdl(quantize_rows_kernel, dim3((unsigned)grid), dim3(QR_WARPS * 32), 0, stream,
                      (const __nv_bfloat16 *)src, batches, rows_per_batch, cols, counts, c_dev,
                      (uint8_t *)q, scale, st);
}

}  // namespace moe
