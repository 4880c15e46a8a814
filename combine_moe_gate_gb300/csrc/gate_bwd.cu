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

// Coefficient of a route under renormalised gates: d_logits[t, idx_r] =
// g_r (dg_r - A), rounded step by step (no contraction), so that every kernel
// that recomputes it gets the same bits.
__device__ __forceinline__ float route_coef(float g, float dg, float a) {
    return __fmul_rn(g, __fsub_rn(dg, a));
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
    // A in route order (the route-sparse kernels recompute it the same way)
    const float p = __fmul_rn(my_dg, my_g);
    float a = 0.0f;
    for (int r = 0; r < k; r++) a = __fadd_rn(a, __shfl_sync(0xffffffffu, p, r));
    float *row = d_logits + t * e;
    if (normalize) {
        for (int j = lane; j < e; j += 32) row[j] = 0.0f;
        __syncwarp();
        if (my_j >= 0) row[my_j] = route_coef(my_g, my_dg, a);
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
// d_wg = x^T dl is a contraction over the tokens with few outputs (m x e), so
// the tokens are split: a cluster of WG_CL CTAs owns WG_F features x WG_E
// experts and each of its WG_CL * WG_WARPS warps takes one contiguous slice of
// the tokens.  A warp streams its slice through a private ring in shared
// memory (cp.async; WG_NS stages of WG_T tokens, each holding the x rows'
// WG_F features and the d_logits rows' WG_E experts), and lane
// (fg, eg) = (lane % 8, lane / 8) accumulates its 8 features times experts
// 4 eg .. 4 eg + 3 over its tokens in order.  The partial sums are then added
// in a fixed order -- the warps of a CTA in order, then the CTAs of the
// cluster in rank order through distributed shared memory -- so d_wg does not
// depend on scheduling.  The clusters of feature block 0 also sum d_bias.
constexpr int WG_F = 64, WG_E = 16, WG_T = 8, WG_NS = 4, WG_WARPS = 8, WG_CL = 8;
constexpr int WG_OUT = WG_F * WG_E;           // outputs of a cluster
constexpr int WG_SLICES = WG_CL * WG_WARPS;   // token slices of a cluster

template <typename XT> struct WgCfg {
    static constexpr int V = 16 / (int)sizeof(XT);            // features of a 16-byte chunk
    static constexpr int XCH = WG_F / V;                      // chunks of a stage's x row
    static constexpr int CPL = 8 / V;                         // a lane's chunks: fg + 8 c
    static constexpr int XB = WG_T * WG_F * (int)sizeof(XT);  // x bytes of a stage
    static constexpr int SB = XB + WG_T * WG_E * 4;           // bytes of a stage
    static constexpr int SMEM = WG_WARPS * WG_NS * SB;
    static_assert(SMEM >= WG_WARPS * WG_OUT * 4, "the rings hold the warps' partials");
    static_assert((WG_T * XCH) % 32 == 0 && WG_T * WG_E == 4 * 32, "whole chunks per lane");
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The float at `p` (this CTA's shared memory) in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(const float *p, uint32_t rank) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(p), r;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
    return v;
}

// One stage of a warp's ring: tokens t0 .. t0 + WG_T - 1 (those >= t1 and
// features / experts past the end read as zero).
template <typename XT, bool DVEC>
__device__ __forceinline__ void wg_issue(unsigned char *stage, const XT *x, const float *dl,
                                         int64_t t0, int64_t t1, int m, int e, int f0, int j0,
                                         int lane) {
    using C = WgCfg<XT>;
#pragma unroll
    for (int q0 = 0; q0 < WG_T * C::XCH; q0 += 32) {
        const int q = q0 + lane, r = q / C::XCH, ch = q % C::XCH;
        const int64_t t = t0 + r;
        const int f = f0 + ch * C::V;
        const bool ok = t < t1 && f < m;
        cp_async16(stage + q * 16, ok ? (const void *)(x + t * m + f) : (const void *)x, ok);
    }
    float *ds = reinterpret_cast<float *>(stage + C::XB);
    if (DVEC) {
        // WG_T rows of WG_E / 4 chunks: one chunk per lane
        const int r = lane / (WG_E / 4), ch = lane % (WG_E / 4);
        const int64_t t = t0 + r;
        const int j = j0 + 4 * ch;
        const bool ok = t < t1 && j < e;
        cp_async16(ds + 4 * lane, ok ? (const void *)(dl + t * e + j) : (const void *)dl, ok);
    } else {
#pragma unroll
        for (int q0 = 0; q0 < WG_T * WG_E; q0 += 32) {
            const int q = q0 + lane, r = q / WG_E, jj = q % WG_E;
            const int64_t t = t0 + r;
            const int j = j0 + jj;
            const bool ok = t < t1 && j < e;
            cp_async4(ds + q, ok ? (const void *)(dl + t * e + j) : (const void *)dl, ok);
        }
    }
}

// One ring stage into lane (fg, eg)'s sums; SUMB: also d_bias's.
template <typename XT, bool SUMB>
__device__ __forceinline__ void wg_stage(const unsigned char *st, int fg, int eg,
                                         float2 (&acc)[4][4], float (&accb)[4]) {
    using C = WgCfg<XT>;
    const float *ds = reinterpret_cast<const float *>(st + C::XB);
#pragma unroll
    for (int r = 0; r < WG_T; r++) {
        float2 xp[4];   // feature pairs, exactly widened
#pragma unroll
        for (int c = 0; c < C::CPL; c++) {
            const V16 v = *reinterpret_cast<const V16 *>(st + (r * C::XCH + fg + 8 * c) * 16);
            if constexpr (sizeof(XT) == 2) {
#pragma unroll
                for (int i = 0; i < 4; i++) xp[i] = make_float2(bf16lo(v.w[i]), bf16hi(v.w[i]));
            } else {
                xp[2 * c] = make_float2(__uint_as_float(v.w[0]), __uint_as_float(v.w[1]));
                xp[2 * c + 1] = make_float2(__uint_as_float(v.w[2]), __uint_as_float(v.w[3]));
            }
        }
        const float4 d4 = *reinterpret_cast<const float4 *>(ds + r * WG_E + 4 * eg);
        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            const float2 d2 = make_float2(dv[jj], dv[jj]);
#pragma unroll
            for (int p = 0; p < 4; p++) acc[p][jj] = __ffma2_rn(xp[p], d2, acc[p][jj]);
        }
        if (SUMB) {
#pragma unroll
            for (int jj = 0; jj < 4; jj++) accb[jj] += dv[jj];
        }
    }
}

// Grid: n_fb * n_eb clusters of WG_CL CTAs along x, cluster (fb, eb) at
// blockIdx.x / WG_CL = fb * n_eb + eb.  No CTA leaves early (the cluster
// barriers need all of them): after an error the CTAs skip the work and the
// stores instead.
template <typename XT, bool DVEC>
__global__ void __launch_bounds__(WG_WARPS * 32, 2)
gate_bwd_dwg_kernel(const XT *__restrict__ x, const float *__restrict__ dl, int64_t s, int m,
                    int e, int n_eb, float *__restrict__ d_wg, float *__restrict__ d_bias,
                    int32_t *status) {
    using C = WgCfg<XT>;
    extern __shared__ float4 wg_smem4[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(wg_smem4);
    __shared__ float part[WG_OUT];   // this CTA's sums, read by the whole cluster
    __shared__ float part_b[WG_E];
    __shared__ float red_b[WG_WARPS][WG_E];
    pdl_enter();
    const bool bad = __syncthreads_or(status_bad(status)) != 0;   // uniform over the CTA
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int fg = lane & 7, eg = lane >> 3;
    const uint32_t rank = cluster_rank();
    const int cid = blockIdx.x / WG_CL, fb = cid / n_eb, eb = cid % n_eb;
    const int f0 = fb * WG_F, j0 = eb * WG_E;
    const bool sum_b = d_bias != nullptr && fb == 0;   // uniform over the cluster

    // this warp's token slice, a whole number of stages long
    const int64_t len = ((s + WG_SLICES - 1) / WG_SLICES + WG_T - 1) / WG_T * WG_T;
    const int64_t t_lo = min(s, (int64_t)(rank * WG_WARPS + warp) * len);
    const int64_t t_hi = min(s, t_lo + len);
    const int nst = bad ? 0 : (int)((t_hi - t_lo + WG_T - 1) / WG_T);
    unsigned char *ring = smem + warp * (WG_NS * C::SB);

    // acc[p][jj]: the lane's features 2p and 2p + 1 times expert 4 eg + jj
    float2 acc[4][4];
    float accb[4];
#pragma unroll
    for (int jj = 0; jj < 4; jj++) {
        accb[jj] = 0.0f;
#pragma unroll
        for (int p = 0; p < 4; p++) acc[p][jj] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int p = 0; p < WG_NS - 1; p++) {
        if (p < nst)
            wg_issue<XT, DVEC>(ring + p * C::SB, x, dl, t_lo + p * WG_T, t_hi, m, e, f0, j0, lane);
        cp_async_commit();
    }
    for (int it = 0; it < nst; it++) {
        cp_async_wait<WG_NS - 2>();   // stage `it` landed (this lane's copies) ...
        __syncwarp();                 // ... and every lane's; stage it - 1 is free
        const int nx = it + WG_NS - 1;
        if (nx < nst)
            wg_issue<XT, DVEC>(ring + (nx % WG_NS) * C::SB, x, dl, t_lo + (int64_t)nx * WG_T,
                               t_hi, m, e, f0, j0, lane);
        cp_async_commit();
        const unsigned char *st = ring + (it % WG_NS) * C::SB;
        if (sum_b)
            wg_stage<XT, true>(st, fg, eg, acc, accb);
        else
            wg_stage<XT, false>(st, fg, eg, acc, accb);
    }
    cp_async_wait<0>();
    __syncthreads();   // every warp is done with its ring: it takes the partials now

    float *red = reinterpret_cast<float *>(smem);   // [WG_WARPS][WG_OUT]
#pragma unroll
    for (int f = 0; f < 8; f++) {
        const int fl = (fg + 8 * (f / C::V)) * C::V + f % C::V;
        const int p = f / 2;
        *reinterpret_cast<float4 *>(red + warp * WG_OUT + fl * WG_E + 4 * eg) =
            (f & 1) ? make_float4(acc[p][0].y, acc[p][1].y, acc[p][2].y, acc[p][3].y)
                    : make_float4(acc[p][0].x, acc[p][1].x, acc[p][2].x, acc[p][3].x);
    }
    if (sum_b && fg == 0)
        *reinterpret_cast<float4 *>(&red_b[warp][4 * eg]) =
            make_float4(accb[0], accb[1], accb[2], accb[3]);
    __syncthreads();
#pragma unroll
    for (int u = 0; u < WG_OUT / (WG_WARPS * 32); u++) {
        const int o = threadIdx.x + u * WG_WARPS * 32;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < WG_WARPS; w++) sum += red[w * WG_OUT + o];
        part[o] = sum;
    }
    if (sum_b && threadIdx.x < WG_E) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < WG_WARPS; w++) sum += red_b[w][threadIdx.x];
        part_b[threadIdx.x] = sum;
    }
    cluster_sync();   // every CTA's sums are in place
    // CTA `rank` adds its share of the outputs over the cluster, ranks in order
    constexpr int PER = WG_OUT / WG_CL;
    if (threadIdx.x < PER) {
        const int o = (int)rank * PER + threadIdx.x;
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < WG_CL; q++) sum += ld_cluster_f32(&part[o], (uint32_t)q);
        const int fi = f0 + o / WG_E, j = j0 + o % WG_E;
        if (d_wg != nullptr && !bad && fi < m && j < e) d_wg[(int64_t)fi * e + j] = sum;
    }
    if (sum_b && rank == 0 && threadIdx.x < WG_E) {
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < WG_CL; q++) sum += ld_cluster_f32(&part_b[threadIdx.x], (uint32_t)q);
        const int j = j0 + threadIdx.x;
        if (!bad && j < e) d_bias[j] = sum;
    }
    cluster_sync();   // no CTA leaves while the others read its shared memory
}

// --------------------------------------------------------------------- d_x
// d_x = dl wg^T, summed over the experts in order.  Work items are (feature
// block of DX_F features, tile of DX_WARPS * U tokens), feature block major;
// each CTA of a persistent grid takes one contiguous run of them.  It stages
// the gate weights of its current feature block in shared memory, transposed
// (wgs[j][i], DX_LD words a row), and copies each tile's d_logits transposed
// as well (dlt[j][t], TP words a row) with cp.async, double-buffered: the next
// tile lands while this one computes.  Rows e .. ep - 1 of both are zero.
// Lane l computes features 4l .. 4l + 3 of its warp's U tokens with packed
// fp32x2 FMAs over token pairs (a float4 store per token).
constexpr int DX_WARPS = 8, DX_F = 128, DX_LD = DX_F + 4;

inline int dx_u(int e) { return e <= 64 ? 8 : 4; }
__host__ __device__ constexpr int dx_tp(int u) { return DX_WARPS * u + 4; }
inline size_t dx_smem(int e, int u) {
    const size_t ep = (size_t)((e + 3) & ~3);
    return ep * DX_LD * 4 + 2 * ep * dx_tp(u) * 4;
}

template <int U>
__global__ void __launch_bounds__(DX_WARPS * 32, 2)
gate_bwd_dx_kernel(const float *__restrict__ dl, const float *__restrict__ wg, int64_t s, int m,
                   int e, int64_t n_tiles, int64_t n_items, float *__restrict__ d_x,
                   int32_t *status) {
    constexpr int TT = DX_WARPS * U, TP = dx_tp(U);
    static_assert(U % 4 == 0, "whole float4 token groups");
    extern __shared__ float4 dx_smem4[];
    const int ep = (e + 3) & ~3;
    float *wgs = reinterpret_cast<float *>(dx_smem4);   // [ep][DX_LD]
    float *dlt = wgs + ep * DX_LD;                      // 2 x [ep][TP]
    pdl_enter();
    if (__syncthreads_or(status_bad(status))) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t lo = n_items * blockIdx.x / gridDim.x;
    const int64_t hi = n_items * (blockIdx.x + 1) / gridDim.x;

    // tile `tile`'s d_logits rows into buffer b, transposed
    auto issue = [&](int64_t tile, int b) {
        float *dst = dlt + b * ep * TP;
        const int64_t t0 = tile * TT;
        for (int r = warp; r < TT; r += DX_WARPS) {
            const bool in = t0 + r < s;
            const float *src = dl + (in ? t0 + r : 0) * e;
            for (int j = lane; j < ep; j += 32) {
                const bool ok = in && j < e;
                cp_async4(dst + j * TP + r, ok ? (const void *)(src + j) : (const void *)dl, ok);
            }
        }
    };

    int64_t fb = lo / n_tiles, tile = lo - fb * n_tiles, cur_fb = -1;
    if (lo < hi) issue(tile, 0);
    cp_async_commit();
    int b = 0;
    for (int64_t item = lo; item < hi; item++, b ^= 1) {
        const int i0 = (int)fb * DX_F;
        if (fb != cur_fb) {
            // this feature block's weights (the previous tile's readers are done)
            for (int ii = warp; ii < DX_F; ii += DX_WARPS) {
                const bool in = i0 + ii < m;
                const float *src = wg + (int64_t)(in ? i0 + ii : 0) * e;
                for (int j = lane; j < ep; j += 32) {
                    const bool ok = in && j < e;
                    cp_async4(wgs + j * DX_LD + ii, ok ? (const void *)(src + j) : (const void *)wg,
                              ok);
                }
            }
            cp_async_commit();
            cp_async_wait<0>();
            cur_fb = fb;
        }
        const int64_t next_tile = tile + 1 == n_tiles ? 0 : tile + 1;
        if (item + 1 < hi) issue(next_tile, b ^ 1);
        cp_async_commit();
        cp_async_wait<1>();   // this tile (and the weights) landed for this thread ...
        __syncthreads();      // ... and for every thread
        const float *dr = dlt + b * ep * TP + warp * U;
        float2 acc[U / 2][4];   // tokens 2p, 2p + 1 of the warp's U, feature 4 lane + f
#pragma unroll
        for (int p = 0; p < U / 2; p++)
#pragma unroll
            for (int f = 0; f < 4; f++) acc[p][f] = make_float2(0.0f, 0.0f);
#pragma unroll 4
        for (int j = 0; j < ep; j++) {
            float2 dp[U / 2];
#pragma unroll
            for (int q = 0; q < U / 4; q++) {
                const float4 d = *reinterpret_cast<const float4 *>(dr + j * TP + 4 * q);
                dp[2 * q] = make_float2(d.x, d.y);
                dp[2 * q + 1] = make_float2(d.z, d.w);
            }
            const float4 w = *reinterpret_cast<const float4 *>(wgs + j * DX_LD + 4 * lane);
            const float2 w2[4] = {make_float2(w.x, w.x), make_float2(w.y, w.y),
                                  make_float2(w.z, w.z), make_float2(w.w, w.w)};
#pragma unroll
            for (int p = 0; p < U / 2; p++)
#pragma unroll
                for (int f = 0; f < 4; f++) acc[p][f] = __ffma2_rn(dp[p], w2[f], acc[p][f]);
        }
        const int i = i0 + 4 * lane;
        const int64_t tb = tile * TT + warp * U;
        if (i < m) {
#pragma unroll
            for (int p = 0; p < U / 2; p++) {
                if (tb + 2 * p < s)
                    *reinterpret_cast<float4 *>(d_x + (tb + 2 * p) * m + i) =
                        make_float4(acc[p][0].x, acc[p][1].x, acc[p][2].x, acc[p][3].x);
                if (tb + 2 * p + 1 < s)
                    *reinterpret_cast<float4 *>(d_x + (tb + 2 * p + 1) * m + i) =
                        make_float4(acc[p][0].y, acc[p][1].y, acc[p][2].y, acc[p][3].y);
            }
        }
        tile = next_tile;
        if (tile == 0) fb++;
        __syncthreads();   // buffer b and the weights are free again
    }
}

// ------------------------------------------------ renormalised gates: routes
// With MOE_FLAG_NORMALIZE_GATES a token's d_logits row is zero except at its
// k routes' experts, where it holds c_r = g_r (dg_r - A).  d_x and d_wg then
// need only those entries:
//   d_x[t, :]  = sum over the routes r of t, in route order, of c_r wg[:, idx_r]
//   d_wg[:, j] = sum over the tokens t routed to j, in token order, of c x[t, :]
//   d_bias[j]  = the same sum of c alone.
// The kernels below recompute c_r from (idx, gates, d_gates) with the
// d_logits kernel's arithmetic (route_coef, A in route order), so they use
// exactly the values d_logits holds.  A route whose expert index is invalid
// (the d_logits kernel flags it) contributes nothing.

// One token's A and route coefficients from staged route rows: rows r of
// idx, gates and d_gates at ri[r * ld], rg[r * ld], rd[r * ld].
__device__ __forceinline__ float route_a(const float *rg, const float *rd, int k, int ld) {
    float a = 0.0f;
    for (int r = 0; r < k; r++) a = __fadd_rn(a, __fmul_rn(rd[r * ld], rg[r * ld]));
    return a;
}

// d_x: a CTA owns one block of DR_F features, whose gate weights it stages
// transposed (wgs[j][i]), and a contiguous token range, which its warps take
// DR_CT tokens at a time, round robin, each on its own.  A warp copies its
// chunks' route rows (idx, gates, d_gates) with cp.async into a private ring
// of DR_NS buffers, lane t turns token t's routes into pairs (byte offset of
// the expert's weight row, coefficient), route major, and lane l computes
// features 4l .. 4l + 3 of DR_U tokens at a time (a float4 store per token).
// No barrier after the weights are staged.  The kernel reads nothing the
// d_wg kernel before it writes, so it runs alongside it (see pdl_trigger).
constexpr int DR_WARPS = 8, DR_CT = 32, DR_NS = 3, DR_U = 8, DR_F = 128, DR_LD = DR_F + 4;

// per warp: DR_NS x route rows [3 k][DR_CT], then pairs [k][DR_CT]
__host__ __device__ inline size_t dr_rows_bytes(int k) { return (size_t)3 * k * DR_CT * 4; }
__host__ __device__ inline size_t dr_warp_bytes(int k) {
    return DR_NS * dr_rows_bytes(k) + (size_t)DR_CT * k * 8;
}
inline size_t dr_smem(int e, int k) { return (size_t)e * DR_LD * 4 + DR_WARPS * dr_warp_bytes(k); }

__global__ void __launch_bounds__(DR_WARPS * 32, 3)
gate_bwd_dx_routes_kernel(const int32_t *__restrict__ idx, const float *__restrict__ gates,
                          const float *__restrict__ d_gates, const float *__restrict__ wg,
                          int64_t s, int m, int e, int k, int64_t chunk_per_cta,
                          float *__restrict__ d_x, int32_t *status) {
    extern __shared__ float4 dr_smem4[];
    float *wgs = reinterpret_cast<float *>(dr_smem4);   // [e][DR_LD]
    pdl_trigger();
    if (__syncthreads_or(status_bad(status))) {
        pdl_wait();
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i0 = blockIdx.y * DR_F;
    {
        // wgs[j][ii] = wg[i0 + ii, j]: thread q takes feature q % DR_F of experts q / DR_F, ...
        const int ii = threadIdx.x % DR_F;
        const bool in = i0 + ii < m;
        const float *src = wg + (int64_t)(in ? i0 + ii : 0) * e;
        for (int j = threadIdx.x / DR_F; j < e; j += DR_WARPS * 32 / DR_F)
            cp_async4(wgs + j * DR_LD + ii, in ? (const void *)(src + j) : (const void *)wg, in);
    }
    cp_async_commit();
    unsigned char *wbuf = reinterpret_cast<unsigned char *>(wgs + e * DR_LD) +
                          (size_t)warp * dr_warp_bytes(k);
    int2 *pairs = reinterpret_cast<int2 *>(wbuf + DR_NS * dr_rows_bytes(k));   // [k][DR_CT]
    // this warp's chunks: c0 + warp, c0 + warp + DR_WARPS, ... < c1
    const int64_t n_chunks = (s + DR_CT - 1) / DR_CT;
    const int64_t c0 = min(n_chunks, (int64_t)blockIdx.x * chunk_per_cta);
    const int64_t c1 = min(n_chunks, c0 + chunk_per_cta);
    const int nc = c0 + warp < c1 ? (int)((c1 - c0 - warp + DR_WARPS - 1) / DR_WARPS) : 0;

    auto issue = [&](int n) {
        float *dst = reinterpret_cast<float *>(wbuf + (n % DR_NS) * dr_rows_bytes(k));
        const int64_t t = (c0 + warp + (int64_t)n * DR_WARPS) * DR_CT + lane;
        const bool ok = t < s;
        for (int a = 0; a < 3; a++) {
            const float *src = (a == 0 ? reinterpret_cast<const float *>(idx)
                                       : a == 1 ? gates : d_gates) + t;
            for (int r = 0; r < k; r++)
                cp_async4(dst + (a * k + r) * DR_CT + lane,
                          ok ? (const void *)(src + (int64_t)r * s) : (const void *)gates, ok);
        }
    };

#pragma unroll
    for (int n = 0; n < DR_NS - 1; n++) {
        if (n < nc) issue(n);
        cp_async_commit();
    }
    cp_async_wait<DR_NS - 1>();   // the weights (this thread's copies) ...
    __syncthreads();              // ... and everyone's
    const int i = i0 + 4 * lane;
    const unsigned char *wl = reinterpret_cast<const unsigned char *>(wgs + 4 * lane);
    for (int n = 0; n < nc; n++) {
        if (n + DR_NS - 1 < nc) issue(n + DR_NS - 1);
        cp_async_commit();
        cp_async_wait<DR_NS - 1>();
        __syncwarp();
        {
            const float *rb = reinterpret_cast<const float *>(wbuf + (n % DR_NS) * dr_rows_bytes(k));
            const float a = route_a(rb + k * DR_CT + lane, rb + 2 * k * DR_CT + lane, k, DR_CT);
            for (int r = 0; r < k; r++) {
                const int j = __float_as_int(rb[r * DR_CT + lane]);
                const float cf = route_coef(rb[(k + r) * DR_CT + lane], rb[(2 * k + r) * DR_CT + lane], a);
                const bool ok = (unsigned)j < (unsigned)e;
                pairs[r * DR_CT + lane] =
                    make_int2(ok ? j * DR_LD * 4 : 0, __float_as_int(ok ? cf : 0.0f));
            }
        }
        __syncwarp();
        const int64_t tc = (c0 + warp + (int64_t)n * DR_WARPS) * DR_CT;
#pragma unroll 1
        for (int p = 0; p < DR_CT / DR_U; p++) {
            float4 acc[DR_U];
#pragma unroll
            for (int u = 0; u < DR_U; u++) acc[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int r = 0; r < k; r++) {
                const int4 *pr = reinterpret_cast<const int4 *>(pairs + r * DR_CT + p * DR_U);
#pragma unroll
                for (int h = 0; h < DR_U / 2; h++) {
                    const int4 q = pr[h];   // two tokens' pairs
#pragma unroll
                    for (int v = 0; v < 2; v++) {
                        const int off = v ? q.z : q.x;
                        const float cf = __int_as_float(v ? q.w : q.y);
                        const float4 w = *reinterpret_cast<const float4 *>(wl + off);
                        float4 &o = acc[2 * h + v];
                        o.x = fmaf(cf, w.x, o.x);
                        o.y = fmaf(cf, w.y, o.y);
                        o.z = fmaf(cf, w.z, o.z);
                        o.w = fmaf(cf, w.w, o.w);
                    }
                }
            }
            const int64_t tb = tc + p * DR_U;
            if (i < m) {
                float *o = d_x + tb * m + i;
                const int nu = (int)min((int64_t)DR_U, s - tb);
#pragma unroll
                for (int u = 0; u < DR_U; u++, o += m)
                    if (u < nu) *reinterpret_cast<float4 *>(o) = acc[u];
            }
        }
        __syncwarp();   // the pairs are rewritten for the next chunk
    }
    pdl_wait();   // complete only after the kernel before it
}

// Resident CTAs of `kern` on this device (cached per kernel and device).
template <typename K>
int resident_ctas(K kern, int threads, size_t smem) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sms * per_sm;
}

template <typename XT, bool DVEC>
moe_status launch_dwg(const XT *x, const float *dl, int64_t s, int m, int e, float *d_wg,
                      float *d_bias, int32_t *st, cudaStream_t stream) {
    using C = WgCfg<XT>;
    auto kern = gate_bwd_dwg_kernel<XT, DVEC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    // d_bias alone needs only feature block 0
    const int64_t n_fb = d_wg ? (m + WG_F - 1) / WG_F : 1;
    const int n_eb = (e + WG_E - 1) / WG_E;
    const int64_t ctas = n_fb * n_eb * WG_CL;
    if (ctas > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
    return launch_cluster_pdl(kern, dim3((unsigned)ctas), dim3(WG_WARPS * 32), (size_t)C::SMEM,
                              WG_CL, stream, x, dl, s, m, e, n_eb, d_wg, d_bias, st);
}

template <int U>
moe_status launch_dx(const float *dl, const float *wg, int64_t s, int m, int e, float *d_x,
                     int32_t *st, cudaStream_t stream) {
    auto kern = gate_bwd_dx_kernel<U>;
    const size_t smem = dx_smem(e, U);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    const int64_t n_tiles = (s + DX_WARPS * U - 1) / (DX_WARPS * U);
    const int64_t n_items = n_tiles * ((m + DX_F - 1) / DX_F);
    const int res = resident_ctas(kern, DX_WARPS * 32, smem);
    if (res <= 0) return MOE_ERR_CUDA;
    const int64_t grid = n_items < res ? n_items : res;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(DX_WARPS * 32), smem, stream, dl, wg, s, m,
                      e, n_tiles, n_items, d_x, st);
}

moe_status launch_dx_routes(const int32_t *idx, const float *gates, const float *d_gates,
                            const float *wg, int64_t s, int m, int e, int k, float *d_x,
                            int32_t *st, cudaStream_t stream) {
    auto kern = gate_bwd_dx_routes_kernel;
    const size_t smem = dr_smem(e, k);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    const int64_t n_fb = (m + DR_F - 1) / DR_F;
    if (n_fb > 65535) return MOE_ERR_UNSUPPORTED;
    const int res = resident_ctas(kern, DR_WARPS * 32, smem);
    if (res <= 0) return MOE_ERR_CUDA;
    // token ranges per feature block: the resident CTAs shared out, at least
    // one chunk of DR_CT tokens per warp
    const int64_t n_chunks = (s + DR_CT - 1) / DR_CT;
    int64_t g = res / n_fb;
    if (g < 1) g = 1;
    int64_t per = (n_chunks + g - 1) / g;
    if (per < DR_WARPS) per = DR_WARPS;
    g = (n_chunks + per - 1) / per;
    if (g > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
    return launch_pdl(kern, dim3((unsigned)g, (unsigned)n_fb), dim3(DR_WARPS * 32), smem, stream,
                      idx, gates, d_gates, wg, s, m, e, k, per, d_x, st);
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
    // d_logits rows load in 16-byte chunks when they stay 16-byte aligned
    const bool vec = e % 4 == 0 && aligned16(d_logits);
    if (d_wg || d_bias) {
        r = vec ? launch_dwg<XT, true>((const XT *)x, d_logits, s, m, e, d_wg, d_bias, st, stream)
                : launch_dwg<XT, false>((const XT *)x, d_logits, s, m, e, d_wg, d_bias, st, stream);
        if (r != MOE_OK) return r;
    }
    if (d_x && normalize && dr_smem(e, k) <= 227 * 1024) {
        // d_logits is k-sparse: d_x from the routes
        r = launch_dx_routes(idx, gates, d_gates, wg, s, m, e, k, d_x, st, stream);
    } else if (d_x) {
        r = dx_u(e) == 8 ? launch_dx<8>(d_logits, wg, s, m, e, d_x, st, stream)
                         : launch_dx<4>(d_logits, wg, s, m, e, d_x, st, stream);
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
