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

// The same arithmetic with the row held in registers: W warps share a row
// (W in 1, 2, 4, 8: rows of up to 32 * W * QR_CPL 16-byte chunks), each lane loads all of its
// QR_CPL 16-byte chunks before using any (one DRAM pass, many loads in
// flight), the W warps' maxima meet in shared memory, and the codes are
// made from the registers.
constexpr int QR_CPL = 8;   // 16-byte chunks per lane

template <int W>
__global__ void __launch_bounds__(QR_WARPS * 32)
quantize_rows_reg_kernel(const __nv_bfloat16 *__restrict__ src, int64_t batches, int64_t rpb, int cols,
                         const int32_t *__restrict__ counts, const int32_t *__restrict__ c_dev,
                         uint8_t *__restrict__ q, float *__restrict__ scale, int32_t *status) {
    static_assert(QR_WARPS % W == 0, "warps per row");
    constexpr int RPC = QR_WARPS / W;   // rows per CTA and pass
    __shared__ float part[QR_WARPS];
    pdl_enter();
    if (status_bad(status)) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = warp % W, rsel = warp / W;
    const int nch = cols / 8;
    const int64_t total = batches * rpb;
    const int64_t c_eff = counts ? min((int64_t)*c_dev, rpb) : rpb;
    // the loop bound is the same in every thread of the CTA (barriers inside)
    for (int64_t row0 = (int64_t)blockIdx.x * RPC; row0 < total; row0 += (int64_t)gridDim.x * RPC) {
        const int64_t row = row0 + rsel;
        bool active = row < total;
        if (active && counts) {
            const int64_t b = row / rpb, r = row - b * rpb;
            active = r < min((int64_t)max(counts[b], 0), c_eff);
        }
        const __nv_bfloat16 *xr = src + row * cols;
        V16 v[QR_CPL];
        float amax = 0.0f;
        if (active) {
#pragma unroll
            for (int i = 0; i < QR_CPL; i++) {
                const int c = (i * W + sub) * 32 + lane;
                if (c < nch) v[i] = ld_v16(xr + 8 * c);
            }
#pragma unroll
            for (int i = 0; i < QR_CPL; i++) {
                const int c = (i * W + sub) * 32 + lane;
                if (c < nch) {
                    float f[8];
                    Elt<__nv_bfloat16>::unpack(v[i], f);
#pragma unroll
                    for (int j = 0; j < 8; j++) amax = fmaxf(amax, fabsf(f[j]));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (W > 1) {
            if (lane == 0) part[warp] = amax;
            __syncthreads();
#pragma unroll
            for (int w = 0; w < W; w++) amax = fmaxf(amax, part[rsel * W + w]);
            __syncthreads();   // part is rewritten in the next pass
        }
        if (!active) continue;
        const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        if (sub == 0 && lane == 0) scale[row] = s;
        uint8_t *qr = q + row * cols;
#pragma unroll
        for (int i = 0; i < QR_CPL; i++) {
            const int c = (i * W + sub) * 32 + lane;
            if (c >= nch) continue;
            float f[8];
            Elt<__nv_bfloat16>::unpack(v[i], f);
            uint32_t w2[2];
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const uint32_t lo = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(f[4 * k], s), __fdiv_rn(f[4 * k + 1], s)), __NV_SATFINITE,
                    __NV_E4M3);
                const uint32_t hi = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(f[4 * k + 2], s), __fdiv_rn(f[4 * k + 3], s)),
                    __NV_SATFINITE, __NV_E4M3);
                w2[k] = (lo & 0xFFFFu) | (hi << 16);
            }
            *reinterpret_cast<uint2 *>(qr + 8 * c) = make_uint2(w2[0], w2[1]);
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
    // rows up to 8 warps x 32 lanes x QR_CPL chunks: held in registers
    const int nch = cols / 8;
    const int w = nch <= 32 * QR_CPL ? 1 : nch <= 64 * QR_CPL ? 2 : nch <= 128 * QR_CPL ? 4
                : nch <= 256 * QR_CPL ? 8 : 0;
    const int64_t per_cta = w ? QR_WARPS / w : QR_WARPS;
    int64_t grid = (rows + per_cta - 1) / per_cta;
    // one resident wave (the kernels stride over the rows)
    static int resident[9] = {0};
    const int slot = w;   // 0 (loop form), 1, 2, 4, 8
    if (!resident[slot]) {
        int nb = 0;
        cudaError_t err =
            w == 1   ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, quantize_rows_reg_kernel<1>, QR_WARPS * 32, 0)
            : w == 2 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, quantize_rows_reg_kernel<2>, QR_WARPS * 32, 0)
            : w == 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, quantize_rows_reg_kernel<4>, QR_WARPS * 32, 0)
            : w == 8 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, quantize_rows_reg_kernel<8>, QR_WARPS * 32, 0)
                     : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, quantize_rows_kernel, QR_WARPS * 32, 0);
        if (err != cudaSuccess || nb < 1) return MOE_ERR_CUDA;
        resident[slot] = nb;
    }
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * resident[slot];
    if (grid > cap) grid = cap;
    const dim3 g((unsigned)grid), blk(QR_WARPS * 32);
    const auto *x = (const __nv_bfloat16 *)src;
    uint8_t *qq = (uint8_t *)q;
    switch (w) {
        case 1: return launch_pdl(quantize_rows_reg_kernel<1>, g, blk, 0, stream, x, batches,
                                  rows_per_batch, cols, counts, c_dev, qq, scale, st);
        case 2: return launch_pdl(quantize_rows_reg_kernel<2>, g, blk, 0, stream, x, batches,
                                  rows_per_batch, cols, counts, c_dev, qq, scale, st);
        case 4: return launch_pdl(quantize_rows_reg_kernel<4>, g, blk, 0, stream, x, batches,
                                  rows_per_batch, cols, counts, c_dev, qq, scale, st);
        case 8: return launch_pdl(quantize_rows_reg_kernel<8>, g, blk, 0, stream, x, batches,
                                  rows_per_batch, cols, counts, c_dev, qq, scale, st);
        default: return launch_pdl(quantize_rows_kernel, g, blk, 0, stream, x, batches,
                                   rows_per_batch, cols, counts, c_dev, qq, scale, st);
    }
}

}  // namespace moe
