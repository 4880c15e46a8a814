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
// All in fp32 and deterministic: every output is an fp32 sum in a fixed order
// (d_wg and d_bias: per token group in token order, then a fixed tree).
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
// d_wg[i, j] = sum_t x[t, i] dl[t, j] and d_bias[j] = sum_t dl[t, j].  A CTA
// owns WG_F features and WG_EB experts for every token.  Thread (g, q) holds
// the four features i0 + 4q .. i0 + 4q + 3 (one 16- or 8-byte load; rows are
// multiples of four features) and sums the tokens g, g + WG_G, g + 2 WG_G, ...
// with WG_U of them in flight.  The CTA then adds its WG_G token groups'
// partials in a fixed tree (xor shuffles inside a warp, the warps in order),
// so every result is independent of scheduling.  The CTAs of the first
// feature block also sum d_bias.
constexpr int WG_Q = 2, WG_F = 4 * WG_Q, WG_EB = 8, WG_U = 4;
constexpr int WG_THREADS = 512, WG_G = WG_THREADS / WG_Q, WG_WARPS = WG_THREADS / 32;

__device__ __forceinline__ void ld_x4(const float *p, float (&v)[4]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void ld_x4(const __nv_bfloat16 *p, float (&v)[4]) {
    // bf16 -> fp32 is exact: the 16 bits become the high half of the word
    const uint2 a = *reinterpret_cast<const uint2 *>(p);
    v[0] = __uint_as_float(a.x << 16); v[1] = __uint_as_float(a.x & 0xffff0000u);
    v[2] = __uint_as_float(a.y << 16); v[3] = __uint_as_float(a.y & 0xffff0000u);
}

// the n (0, 4 or 8 when VEC) experts of one d_logits row from p; zeros past n
template <bool VEC>
__device__ __forceinline__ void ld_dl8(const float *p, int n, float (&v)[WG_EB]) {
    if (VEC) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (n >= 4) a = *reinterpret_cast<const float4 *>(p);
        if (n >= 8) b = *reinterpret_cast<const float4 *>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int jj = 0; jj < WG_EB; jj++) v[jj] = jj < n ? p[jj] : 0.0f;
    }
}

template <typename XT, bool DVEC>
__global__ void __launch_bounds__(WG_THREADS)
gate_bwd_dwg_kernel(const XT *__restrict__ x, const float *__restrict__ dl, int64_t s, int m,
                    int e, float *__restrict__ d_wg, float *__restrict__ d_bias, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    __shared__ float red[WG_WARPS][WG_F * WG_EB];
    __shared__ float redb[WG_WARPS][WG_EB];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int q = threadIdx.x % WG_Q, g = threadIdx.x / WG_Q;
    const int i0 = blockIdx.x * WG_F, i = i0 + 4 * q;
    const int j0 = blockIdx.y * WG_EB, nj = min(WG_EB, e - j0);
    const bool want_wg = d_wg != nullptr;                  // uniform over the CTA
    const bool want_b = d_bias != nullptr && blockIdx.x == 0;
    const bool load_x = want_wg && i < m;
    float acc[4][WG_EB], accb[WG_EB];
#pragma unroll
    for (int jj = 0; jj < WG_EB; jj++) {
        accb[jj] = 0.0f;
#pragma unroll
        for (int f = 0; f < 4; f++) acc[f][jj] = 0.0f;
    }
    for (int64_t t0 = g; t0 < s; t0 += (int64_t)WG_G * WG_U) {
        float xv[WG_U][4], dv[WG_U][WG_EB];
#pragma unroll
        for (int u = 0; u < WG_U; u++) {
            const int64_t t = t0 + (int64_t)u * WG_G;
            const bool in = t < s;
            ld_dl8<DVEC>(dl + (in ? t : 0) * e + j0, in ? nj : 0, dv[u]);
            if (in && load_x) {
                ld_x4(x + t * m + i, xv[u]);
            } else {
#pragma unroll
                for (int f = 0; f < 4; f++) xv[u][f] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < WG_U; u++)
#pragma unroll
            for (int jj = 0; jj < WG_EB; jj++) {
#pragma unroll
                for (int f = 0; f < 4; f++) acc[f][jj] = fmaf(xv[u][f], dv[u][jj], acc[f][jj]);
                accb[jj] += dv[u][jj];
            }
    }
    // lanes with the same q: xor over the token-group bits of the lane index
    if (want_wg) {
#pragma unroll
        for (int f = 0; f < 4; f++)
#pragma unroll
            for (int jj = 0; jj < WG_EB; jj++) {
                float v = acc[f][jj];
#pragma unroll
                for (int o = WG_Q; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[f][jj] = v;
            }
        if (lane < WG_Q) {
#pragma unroll
            for (int f = 0; f < 4; f++)
#pragma unroll
                for (int jj = 0; jj < WG_EB; jj++) red[warp][(4 * lane + f) * WG_EB + jj] = acc[f][jj];
        }
    }
    if (want_b) {
#pragma unroll
        for (int jj = 0; jj < WG_EB; jj++) {
            float v = accb[jj];
#pragma unroll
            for (int o = WG_Q; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) redb[warp][jj] = v;
        }
    }
    __syncthreads();
    const int o = threadIdx.x;
    if (want_wg && o < WG_F * WG_EB) {
        const int ii = i0 + o / WG_EB, jj = o % WG_EB;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < WG_WARPS; w++) sum += red[w][o];
        if (ii < m && jj < nj) d_wg[(int64_t)ii * e + j0 + jj] = sum;
    }
    if (want_b && o >= WG_F * WG_EB && o < WG_F * WG_EB + WG_EB) {
        const int jj = o - WG_F * WG_EB;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < WG_WARPS; w++) sum += redb[w][jj];
        if (jj < nj) d_bias[j0 + jj] = sum;
    }
}

// --------------------------------------------------------------------- d_x
// d_x[t, i] = sum_j dl[t, j] wg[i, j], summed over j in order.  A CTA owns
// DX_TOK tokens and DX_F features, whose weights it stages transposed in
// shared memory (wgs[j][i], rows padded to DX_LD words); lane l of a warp
// computes features 4l .. 4l + 3 (one float4 store) for DX_U tokens at once.
constexpr int DX_WARPS = 8, DX_U = 4, DX_TOK = DX_WARPS * DX_U, DX_F = 128, DX_LD = DX_F + 4;

template <bool DVEC>
__global__ void __launch_bounds__(DX_WARPS * 32)
gate_bwd_dx_kernel(const float *__restrict__ dl, const float *__restrict__ wg, int64_t s, int m,
                   int e, float *__restrict__ d_x, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    extern __shared__ float4 wgs4[];   // [e][DX_LD] floats
    float *wgs = reinterpret_cast<float *>(wgs4);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i0 = blockIdx.y * DX_F;
    for (int q = threadIdx.x; q < DX_F * e; q += DX_WARPS * 32) {
        const int ii = q / e, j = q % e;
        wgs[j * DX_LD + ii] = i0 + ii < m ? wg[(int64_t)(i0 + ii) * e + j] : 0.0f;
    }
    __syncthreads();
    const int i = i0 + 4 * lane;
    const int64_t tb = (int64_t)blockIdx.x * DX_TOK + warp;   // tokens tb + u DX_WARPS
    float acc[DX_U][4];
#pragma unroll
    for (int u = 0; u < DX_U; u++)
#pragma unroll
        for (int f = 0; f < 4; f++) acc[u][f] = 0.0f;
    for (int j0 = 0; j0 < e; j0 += WG_EB) {
        const int nj = min(WG_EB, e - j0);
        float dv[DX_U][WG_EB];
#pragma unroll
        for (int u = 0; u < DX_U; u++) {
            const int64_t t = tb + (int64_t)u * DX_WARPS;
            const bool in = t < s;
            ld_dl8<DVEC>(dl + (in ? t : 0) * e + j0, in ? nj : 0, dv[u]);
        }
#pragma unroll
        for (int jj = 0; jj < WG_EB; jj++) {
            if (jj < nj) {
                const float4 w = *reinterpret_cast<const float4 *>(wgs + (j0 + jj) * DX_LD + 4 * lane);
#pragma unroll
                for (int u = 0; u < DX_U; u++) {
                    acc[u][0] = fmaf(dv[u][jj], w.x, acc[u][0]);
                    acc[u][1] = fmaf(dv[u][jj], w.y, acc[u][1]);
                    acc[u][2] = fmaf(dv[u][jj], w.z, acc[u][2]);
                    acc[u][3] = fmaf(dv[u][jj], w.w, acc[u][3]);
                }
            }
        }
    }
    if (i < m) {
#pragma unroll
        for (int u = 0; u < DX_U; u++) {
            const int64_t t = tb + (int64_t)u * DX_WARPS;
            if (t < s)
                *reinterpret_cast<float4 *>(d_x + t * m + i) =
                    make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
        }
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
        // d_bias alone runs only the first feature block's CTAs; d_logits rows
        // load as float4 when they stay 16-byte aligned
        const unsigned gx = d_wg ? (unsigned)((m + WG_F - 1) / WG_F) : 1u;
        const dim3 grid(gx, (unsigned)((e + WG_EB - 1) / WG_EB));
        const bool vec = e % 4 == 0 && aligned16(d_logits);
        r = vec ? launch_pdl(gate_bwd_dwg_kernel<XT, true>, grid, dim3(WG_THREADS), 0, stream,
                             (const XT *)x, (const float *)d_logits, s, m, e, d_wg, d_bias, st)
                : launch_pdl(gate_bwd_dwg_kernel<XT, false>, grid, dim3(WG_THREADS), 0, stream,
                             (const XT *)x, (const float *)d_logits, s, m, e, d_wg, d_bias, st);
        if (r != MOE_OK) return r;
    }
    if (d_x) {
        // rows of four features (rows are multiples of four); tokens on grid x
        const size_t smem = (size_t)e * DX_LD * sizeof(float);
        const bool vec = e % 4 == 0 && aligned16(d_logits);
        auto kern = vec ? gate_bwd_dx_kernel<true> : gate_bwd_dx_kernel<false>;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
            return MOE_ERR_CUDA;
        const int64_t gx = (s + DX_TOK - 1) / DX_TOK;
        if (gx > 0x7fffffff || (m + DX_F - 1) / DX_F > 65535) return MOE_ERR_UNSUPPORTED;
        r = launch_pdl(kern, dim3((unsigned)gx, (unsigned)((m + DX_F - 1) / DX_F)),
                       dim3(DX_WARPS * 32), smem, stream, (const float *)d_logits, wg, s, m, e,
                       d_x, st);
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
