// Gate backward: from the gate values' gradient to the logits, the gate
// weight, its bias and x.
//
// Method: the Tutel profile's gate_type {'type': 'top'}: gates are the softmax
// probabilities of the k selected experts, renormalised over them when
// MOE_FLAG_NORMALIZE_GATES is set.  Top-k selection is piecewise constant, so
// gradients flow only through the softmax:
//   A = sum_r dg_r g_r;
//   renormalised:  dl_{i_r} = g_r (dg_r - A), other experts 0 (a softmax over
//                  the selected logits alone);
//   raw softmax:   dl_j = -p_j A + sum_{r: i_r = j} dg_r g_r, p = softmax(l).
// Then through l = x Wg + b: d_wg = x^T dl, d_bias = sum_t dl, d_x = dl Wg^T.
// All in fp32; every output is one sequential fp32 sum (deterministic).
#include "common.cuh"

namespace moe {
namespace {

template <typename XT> __device__ __forceinline__ float ldx(const XT *p);
template <> __device__ __forceinline__ float ldx<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ldx<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

// ---------------------------------------------------------------- d_logits
// One warp per token: lane r < k holds route r; for the raw softmax the lanes
// split the experts and recompute the token's logits.
constexpr int DL_WARPS = 8;
constexpr int DL_MAXQ = 8;   // experts per lane (e <= 256)

template <typename XT>
__global__ void __launch_bounds__(DL_WARPS * 32)
gate_bwd_dl_kernel(const XT *__restrict__ x, const float *__restrict__ wg,
                   const float *__restrict__ bias, int64_t s, int m, int e, int k, int normalize,
                   const int32_t *__restrict__ idx, const float *__restrict__ gates,
                   const float *__restrict__ d_gates, float *__restrict__ d_logits,
                   int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * DL_WARPS + (threadIdx.x >> 5);
    if (t >= s) return;
    int my_j = -1;
    float my_g = 0.0f, my_dg = 0.0f;
    if (lane < k) {
        my_j = idx[(int64_t)lane * s + t];
        my_g = gates[(int64_t)lane * s + t];
        my_dg = d_gates[(int64_t)lane * s + t];
        if ((unsigned)my_j >= (unsigned)e) {
            set_status(status, MOE_ERR_INVALID_ARG);
            my_j = -1;
        }
    }
    float a = my_dg * my_g;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    float *row = d_logits + t * e;
    if (normalize) {
        for (int j = lane; j < e; j += 32) row[j] = 0.0f;
        __syncwarp();
        if (my_j >= 0) row[my_j] = my_g * (my_dg - a);
        return;
    }
    // raw softmax: logits of this token, lane owns experts lane, lane+32, ...
    float l[DL_MAXQ];
#pragma unroll
    for (int q = 0; q < DL_MAXQ; q++) l[q] = 0.0f;
    const XT *xr = x + t * m;
    for (int i = 0; i < m; i++) {
        const float xi = ldx(xr + i);
        const float *wr = wg + (int64_t)i * e;
#pragma unroll
        for (int q = 0; q < DL_MAXQ; q++) {
            const int j = lane + 32 * q;
            if (j < e) l[q] = fmaf(xi, wr[j], l[q]);
        }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < DL_MAXQ; q++) {
        const int j = lane + 32 * q;
        if (j < e) {
            if (bias) l[q] = l[q] + bias[j];
            mx = fmaxf(mx, l[q]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float z = 0.0f;
#pragma unroll
    for (int q = 0; q < DL_MAXQ; q++)
        if (lane + 32 * q < e) z += expf(l[q] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
#pragma unroll
    for (int q = 0; q < DL_MAXQ; q++) {
        const int j = lane + 32 * q;
        if (j < e) row[j] = -(expf(l[q] - mx) / z) * a;
    }
    __syncwarp();
    // routes of the selected experts, in route order (k <= 32 lanes)
    for (int r = 0; r < k; r++) {
        const int j = __shfl_sync(0xffffffffu, my_j, r);
        const float gd = __shfl_sync(0xffffffffu, my_dg * my_g, r);
        if (lane == 0 && j >= 0) row[j] += gd;
        __syncwarp();
    }
}

// ------------------------------------------------------------- d_wg, d_bias
// d_wg[i, j] = sum_t x[t, i] dl[t, j]: a CTA owns 32 features x 8 experts and
// walks the tokens in order, 32 at a time through shared memory; thread (ty,
// tx) accumulates output (i0 + tx, j0 + ty).  The CTAs with i0 == 0 also sum
// d_bias for their experts.
constexpr int WG_TI = 32, WG_TJ = 8, WG_TT = 32;

template <typename XT>
__global__ void __launch_bounds__(WG_TI * WG_TJ)
gate_bwd_dwg_kernel(const XT *__restrict__ x, const float *__restrict__ dl, int64_t s, int m,
                    int e, float *__restrict__ d_wg, float *__restrict__ d_bias, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    __shared__ float xs[WG_TT][WG_TI + 1];
    __shared__ float ds[WG_TT][WG_TJ + 1];
    const int tx = threadIdx.x % WG_TI, ty = threadIdx.x / WG_TI;
    const int i0 = blockIdx.x * WG_TI, j0 = blockIdx.y * WG_TJ;
    const int i = i0 + tx, j = j0 + ty;
    float acc = 0.0f, accb = 0.0f;
    for (int64_t t0 = 0; t0 < s; t0 += WG_TT) {
        __syncthreads();
        for (int q = threadIdx.x; q < WG_TT * WG_TI; q += WG_TI * WG_TJ) {
            const int tt = q / WG_TI, ii = q % WG_TI;
            xs[tt][ii] = (t0 + tt < s && i0 + ii < m) ? ldx(x + (t0 + tt) * m + i0 + ii) : 0.0f;
        }
        for (int q = threadIdx.x; q < WG_TT * WG_TJ; q += WG_TI * WG_TJ) {
            const int tt = q / WG_TJ, jj = q % WG_TJ;
            ds[tt][jj] = (t0 + tt < s && j0 + jj < e) ? dl[(t0 + tt) * e + j0 + jj] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int tt = 0; tt < WG_TT; tt++) {
            acc = fmaf(xs[tt][tx], ds[tt][ty], acc);
            accb += ds[tt][ty];
        }
    }
    if (d_wg && i < m && j < e) d_wg[(int64_t)i * e + j] = acc;
    if (d_bias && blockIdx.x == 0 && tx == 0 && j < e) d_bias[j] = accb;
}

// --------------------------------------------------------------------- d_x
// d_x[t, i] = sum_j dl[t, j] wg[i, j]: a CTA owns 32 features (their weight
// rows staged in shared memory, rows padded by one word) and DX_TOK tokens;
// lane = feature, warp = token.
constexpr int DX_WARPS = 8, DX_TOK = 64;

__global__ void __launch_bounds__(DX_WARPS * 32)
gate_bwd_dx_kernel(const float *__restrict__ dl, const float *__restrict__ wg, int64_t s, int m,
                   int e, float *__restrict__ d_x, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    extern __shared__ float wgs[];   // [32][e + 1]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i0 = blockIdx.x * 32;
    for (int q = threadIdx.x; q < 32 * e; q += DX_WARPS * 32) {
        const int ii = q / e, j = q % e;
        wgs[ii * (e + 1) + j] = i0 + ii < m ? wg[(int64_t)(i0 + ii) * e + j] : 0.0f;
    }
    __syncthreads();
    const float *wr = wgs + lane * (e + 1);
    const int64_t tb = (int64_t)blockIdx.y * DX_TOK;
    for (int tt = warp; tt < DX_TOK; tt += DX_WARPS) {
        const int64_t t = tb + tt;
        if (t >= s) break;
        const float *dr = dl + t * e;
        float acc = 0.0f;
        for (int j = 0; j < e; j++) acc = fmaf(dr[j], wr[j], acc);
        if (i0 + lane < m) d_x[t * m + i0 + lane] = acc;
    }
}

template <typename XT>
moe_status gate_bwd_typed(const void *x, const float *wg, const float *bias, int64_t s, int m,
                          int e, int k, int normalize, const int32_t *idx, const float *gates,
                          const float *d_gates, float *d_logits, float *d_wg, float *d_bias,
                          float *d_x, int32_t *st, cudaStream_t stream) {
    const int64_t g1 = (s + DL_WARPS - 1) / DL_WARPS;
    if (g1 > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
    moe_status r = launch_pdl(gate_bwd_dl_kernel<XT>, dim3((unsigned)g1), dim3(DL_WARPS * 32), 0,
                              stream, (const XT *)x, wg, bias, s, m, e, k, normalize, idx, gates,
                              d_gates, d_logits, st);
    if (r != MOE_OK) return r;
    if (d_wg || d_bias) {
        // d_bias alone runs only the first feature block's CTAs
        const unsigned gx = d_wg ? (unsigned)((m + WG_TI - 1) / WG_TI) : 1u;
        r = launch_pdl(gate_bwd_dwg_kernel<XT>, dim3(gx, (unsigned)((e + WG_TJ - 1) / WG_TJ)),
                       dim3(WG_TI * WG_TJ), 0, stream, (const XT *)x, (const float *)d_logits, s,
                       m, e, d_wg, d_bias, st);
        if (r != MOE_OK) return r;
    }
    if (d_x) {
        const size_t smem = (size_t)32 * (e + 1) * sizeof(float);
        auto kern = gate_bwd_dx_kernel;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
            return MOE_ERR_CUDA;
        const int64_t gy = (s + DX_TOK - 1) / DX_TOK;
        if (gy > 65535) return MOE_ERR_UNSUPPORTED;
        r = launch_pdl(kern, dim3((unsigned)((m + 31) / 32), (unsigned)gy), dim3(DX_WARPS * 32),
                       smem, stream, (const float *)d_logits, wg, s, m, e, d_x, st);
    }
    return r;
}

}  // namespace

moe_status gate_bwd_launch(const void *x, moe_dtype xdt, const float *wg, const float *bias,
                           int64_t s, int m, int e, int k, unsigned flags, const int32_t *idx,
                           const float *gates, const float *d_gates, float *d_logits, float *d_wg,
                           float *d_bias, float *d_x, int32_t *st, cudaStream_t stream) {
    const int normalize = (flags & MOE_FLAG_NORMALIZE_GATES) ? 1 : 0;
    if (xdt == MOE_BF16)
        return gate_bwd_typed<__nv_bfloat16>(x, wg, bias, s, m, e, k, normalize, idx, gates,
                                             d_gates, d_logits, d_wg, d_bias, d_x, st, stream);
    return gate_bwd_typed<float>(x, wg, bias, s, m, e, k, normalize, idx, gates, d_gates,
                                 d_logits, d_wg, d_bias, d_x, st, stream);
}

}  // namespace moe
