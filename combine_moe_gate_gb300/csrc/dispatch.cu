// Index-based encode / decode and their backward.
//
// Method: the DeepSpeed-MoE vs Tutel blog, section 3.5 (fast encode/decode:
// act only on the k non-zero entries of the token-to-expert map, O(T*k*D)
// instead of the O(T*E*C*D) einsum; K0 = encode backward = combine forward,
// K1 = encode forward = combine backward, K2 = the cross term) and DeepSpeed
// PR #8195 change 3 (dispatch and combine become a gather each; combine
// accumulates in fp32).
//
// One warp per (token, row slice of up to 2 KB).  Lanes r < k hold route r's (expert, slot,
// gate); the warp streams its slice of the token's row in 16-byte chunks (8 bf16
// / 4 fp32 per lane per access).  Every row access is a full coalesced 512-byte
// warp transaction.  Combine accumulates each element in
// fp32 in ascending route order, as the C ABI specifies, so results are
// deterministic and independent of the launch shape.
#include "common.cuh"

namespace moe {
namespace {

constexpr int DNT = 256;  // threads per CTA (8 token-warps)
constexpr int SL = 128;   // 16-byte chunks of a row per warp in encode: 4 per lane

struct Routes {
    unsigned kept;   // bit r: route r of this token is kept
    int64_t row;     // lane r: element offset of route r's slot row
    float g;         // lane r: route r's gate
};

// Route entries of token t as stored (lane r < k holds route r's), not yet
// checked; a separate step so that the next item's entries can be in flight
// while the current item's rows move.
struct RawRoute {
    int ex, l;
    float g;
};

// Position of a work item it = row * parts + part that steps by a fixed stride:
// one division at the start, none in the loop.
struct ItemIter {
    int64_t row, drow;
    int part, dpart, parts;
    __device__ __forceinline__ ItemIter(int64_t it, int64_t stride, int parts_) : parts(parts_) {
        row = it / parts_;
        part = (int)(it - row * parts_);
        drow = stride / parts_;
        dpart = (int)(stride - drow * parts_);
    }
    __device__ __forceinline__ void next() {
        row += drow;
        part += dpart;
        if (part >= parts) {
            part -= parts;
            row++;
        }
    }
};

// (row, part) of work item it = row * parts + part: a 32-bit division when
// every item index fits (`small`, uniform over the grid), else a 64-bit one.
__device__ __forceinline__ void split_item(int64_t it, int parts, bool small, int64_t &row,
                                           int &part) {
    if (small) {
        const uint32_t u = (uint32_t)it, r = u / (uint32_t)parts;
        row = r;
        part = (int)(u - r * (uint32_t)parts);
    } else {
        row = it / parts;
        part = (int)(it - row * parts);
    }
}

__device__ __forceinline__ RawRoute fetch_route(const int32_t *idx, const int32_t *loc,
                                                const float *gates, int64_t s, int64_t t, int k) {
    const int lane = threadIdx.x & 31;
    RawRoute q{-1, -1, 0.0f};
    if (lane < k && t < s) {
        q.ex = idx[(int64_t)lane * s + t];
        q.l = loc[(int64_t)lane * s + t];
        if (gates) q.g = gates[(int64_t)lane * s + t];
    }
    return q;
}

__device__ __forceinline__ Routes decide_routes(const RawRoute &q, int m, int e, int k, int c_eff,
                                                int64_t c_max, int32_t *status, int lo = 0,
                                                int hi = 0x7fffffff) {
    const int lane = threadIdx.x & 31;
    Routes R{0u, 0, 0.0f};
    bool kept = false;
    if (lane < k) {
        if ((unsigned)q.ex >= (unsigned)e || q.l < 0) {
            set_status(status, MOE_ERR_INVALID_ARG);
        } else if (q.l < c_eff && q.l >= lo && q.l < hi) {
            kept = true;
            R.row = ((int64_t)q.ex * c_max + q.l) * m;
            R.g = q.g;
        }
    }
    R.kept = __ballot_sync(0xffffffffu, kept);
    return R;
}

__device__ __forceinline__ Routes load_routes(const int32_t *idx, const int32_t *loc,
                                              const float *gates, int64_t s, int64_t t, int m,
                                              int e, int k, int c_eff, int64_t c_max,
                                              int32_t *status, int lo = 0, int hi = 0x7fffffff) {
    return decide_routes(fetch_route(idx, loc, gates, s, t, k), m, e, k, c_eff, c_max, status, lo,
                         hi);
}

__device__ __forceinline__ int read_c(const int32_t *c_dev, int64_t c_max) {
    int c = *c_dev;
    return (int)min((int64_t)c, c_max);
}

// ---------------------------------------------------------------- encode (K1)
// Work item = (token, slice of SL 16-byte chunks of its row): one warp per item,
// so a token row is spread over several warps and every warp needs a single
// row round trip (the slice is loaded together with the route entries).
template <typename T>
__global__ void __launch_bounds__(DNT, 4)
encode_kernel(const T *__restrict__ x, const int32_t *__restrict__ idx,
              const int32_t *__restrict__ loc, const int32_t *__restrict__ c_dev, int64_t s,
              int m, int e, int k, int64_t c_max, T *__restrict__ buf, int32_t *status, int lo,
              int hi) {
    pdl_enter();
    if (status_bad(status)) return;
    const int c_eff = read_c(c_dev, c_max);
    const int lane = threadIdx.x & 31;
    const int nch = m / Elt<T>::VEC;
    const int nsl = (nch + SL - 1) / SL;
    const int64_t items = s * nsl;
    const int64_t nw = (int64_t)gridDim.x * (DNT / 32);
    const int64_t it0 = blockIdx.x * (DNT / 32) + (threadIdx.x >> 5);
    ItemIter pos(it0, nw, nsl);
    for (int64_t it = it0; it < items; it += nw, pos.next()) {
        const int64_t t = pos.row;
        const int c0 = pos.part * SL + lane;
        const V16 *src = reinterpret_cast<const V16 *>(x + t * m);
        V16 v[SL / 32];
#pragma unroll
        for (int u = 0; u < SL / 32; u++)
            if (c0 + 32 * u < nch) v[u] = ld_stream(src + c0 + 32 * u);
        Routes R = load_routes(idx, loc, nullptr, s, t, m, e, k, c_eff, c_max, status, lo, hi);
        for (unsigned km = R.kept; km; km &= km - 1) {
            const int r = __ffs(km) - 1;
            const int64_t row = __shfl_sync(0xffffffffu, R.row, r);
            V16 *dst = reinterpret_cast<V16 *>(buf + row);
#pragma unroll
            for (int u = 0; u < SL / 32; u++)
                if (c0 + 32 * u < nch) st_v16(dst + c0 + 32 * u, v[u]);
        }
    }
}

// Zero rows min(counts[j], c) .. c-1 of every expert j (one warp per row).
template <typename T>
__global__ void __launch_bounds__(DNT)
zero_fill_kernel(const int32_t *__restrict__ counts, const int32_t *__restrict__ c_dev, int e,
                 int64_t c_max, int m, T *__restrict__ buf, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    const int c_eff = read_c(c_dev, c_max);
    const int j = blockIdx.y;
    const int kept = min(counts[j], c_eff);
    const int lane = threadIdx.x & 31;
    const int nch = m / Elt<T>::VEC;
    V16 z;
    z.w[0] = z.w[1] = z.w[2] = z.w[3] = 0u;
    for (int64_t row = kept + (int64_t)blockIdx.x * (DNT / 32) + (threadIdx.x >> 5); row < c_eff;
         row += (int64_t)gridDim.x * (DNT / 32)) {
        V16 *dst = reinterpret_cast<V16 *>(buf + ((int64_t)j * c_max + row) * m);
        for (int q = lane; q < nch; q += 32) st_v16(dst + q, z);
    }
}

// ------------------------------------------------ combine: decode (K0) and
// encode backward (K0 with unit weights)
// U: 16-byte chunks per lane (slice = 32*U chunks).  RGK: routes whose row
// loads are in flight together.  ONE: every route fits in one group (k <= RGK),
// so each chunk is finished (all routes, ascending) before the next one and
// only VEC accumulators are live.
template <typename T, bool WEIGHTED, int U, int RGK, bool ONE>
__global__ void __launch_bounds__(DNT, 4)
combine_kernel(const T *__restrict__ src, const int32_t *__restrict__ idx,
               const int32_t *__restrict__ loc, const float *__restrict__ gates,
               const int32_t *__restrict__ c_dev, int64_t s, int m, int e, int k, int64_t c_max,
               T *__restrict__ y, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    constexpr int VEC = Elt<T>::VEC, SLU = 32 * U;
    const int c_eff = read_c(c_dev, c_max);
    const int lane = threadIdx.x & 31;
    const int nch = m / VEC;
    const int nsl = (nch + SLU - 1) / SLU;
    const int64_t items = s * nsl;
    const int64_t nw = (int64_t)gridDim.x * (DNT / 32);
    int64_t it = blockIdx.x * (DNT / 32) + (threadIdx.x >> 5);
    const bool small = items + nw <= 0x7fffffff;
    int64_t t;
    int part;
    split_item(it, nsl, small, t, part);
    RawRoute nxt = fetch_route(idx, loc, WEIGHTED ? gates : nullptr, s, t, k);
    for (; it < items; it += nw) {
        split_item(it, nsl, small, t, part);
        const int c0 = part * SLU + lane;
        const RawRoute cur = nxt;
        // the next item's route entries travel while this item's rows move
        {
            int64_t tn;
            int pn;
            split_item(it + nw, nsl, small, tn, pn);
            nxt = fetch_route(idx, loc, WEIGHTED ? gates : nullptr, s, tn, k);
        }
        Routes R = decide_routes(cur, m, e, k, c_eff, c_max, status);
        V16 *dst = reinterpret_cast<V16 *>(y + t * m);
        float acc[ONE ? 1 : U][VEC];
        if (!ONE) {
#pragma unroll
            for (int u = 0; u < (ONE ? 1 : U); u++)
#pragma unroll
                for (int i = 0; i < VEC; i++) acc[u][i] = 0.0f;
        }
        // routes in ascending order, RGK at a time: every row load of a group is
        // in flight before the group's fused multiply-adds
        for (int rg = 0; rg < k; rg += RGK) {
            const unsigned gm = (R.kept >> rg) & ((1u << RGK) - 1u);
            if (!ONE && !gm) continue;
            V16 v[RGK][U];
            float g[RGK];
#pragma unroll
            for (int rr = 0; rr < RGK; rr++) {
                g[rr] = 0.0f;
                if ((gm >> rr) & 1u) {
                    const int64_t row = __shfl_sync(0xffffffffu, R.row, rg + rr);
                    g[rr] = WEIGHTED ? __shfl_sync(0xffffffffu, R.g, rg + rr) : 1.0f;
                    const V16 *sp = reinterpret_cast<const V16 *>(src + row);
#pragma unroll
                    for (int u = 0; u < U; u++)
                        if (c0 + 32 * u < nch) v[rr][u] = ld_stream(sp + c0 + 32 * u);
                }
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                float a1[VEC];
                float *a = ONE ? a1 : acc[ONE ? 0 : u];
                if (ONE) {
#pragma unroll
                    for (int i = 0; i < VEC; i++) a1[i] = 0.0f;
                }
#pragma unroll
                for (int rr = 0; rr < RGK; rr++) {
                    if (!((gm >> rr) & 1u)) continue;
                    float f[VEC];
                    Elt<T>::unpack(v[rr][u], f);
#pragma unroll
                    for (int i = 0; i < VEC; i++)
                        a[i] = WEIGHTED ? __fmaf_rn(g[rr], f[i], a[i]) : __fadd_rn(a[i], f[i]);
                }
                if (ONE && c0 + 32 * u < nch) st_v16_cs(dst + c0 + 32 * u, Elt<T>::pack(a1));
            }
            if (ONE) break;
        }
        if (!ONE) {
#pragma unroll
            for (int u = 0; u < (ONE ? 1 : U); u++)
                if (c0 + 32 * u < nch) st_v16_cs(dst + c0 + 32 * u, Elt<T>::pack(acc[u]));
        }
    }
}

// g * d (fp32 times a bf16 value) correctly rounded to bf16, one rounding of
// the exact product, by round to odd: the product truncated to fp32 with its
// last bit set when it was inexact keeps 16 bits beyond bf16's precision, so
// rounding that to bf16 (nearest even) rounds the exact product once.  err is
// the exact remainder g*d - p (at most 8 significant bits).  Infinities and
// NaNs keep their bits.
__device__ __forceinline__ float mul_round_odd(float g, float d) {
    const float p = __fmul_rz(g, d);
    const float err = __fmaf_rn(g, d, -p);
    uint32_t u = __float_as_uint(p);
    if (err != 0.0f && (u & 0x7F800000u) != 0x7F800000u) u |= 1u;
    return __uint_as_float(u);
}

// Two of them, packed (lo in the low half).
__device__ __forceinline__ uint32_t mul_round_bf16x2(float g, float lo, float hi) {
    const __nv_bfloat162 r = __floats2bfloat162_rn(mul_round_odd(g, lo), mul_round_odd(g, hi));
    return *reinterpret_cast<const uint32_t *>(&r);
}

template <typename T> struct ScaleRound;
template <> struct ScaleRound<float> {
    __device__ __forceinline__ static V16 apply(float g, const V16 &d) {
        V16 o;
#pragma unroll
        for (int i = 0; i < 4; i++) o.w[i] = __float_as_uint(__fmul_rn(g, __uint_as_float(d.w[i])));
        return o;
    }
};
template <> struct ScaleRound<__nv_bfloat16> {
    __device__ __forceinline__ static V16 apply(float g, const V16 &d) {
        V16 o;
#pragma unroll
        for (int i = 0; i < 4; i++) o.w[i] = mul_round_bf16x2(g, bf16lo(d.w[i]), bf16hi(d.w[i]));
        return o;
    }
};

// -------------------------------------------- decode backward (K1 bwd + K2)
// One warp per (token, route) pair, token-major (a token's routes are
// neighbouring items, so its dY row is re-read from cache): dG of the route is
// a dot product over the whole row kept in one warp, so its summation order is
// fixed (each lane sums its chunks in row order, then an xor butterfly), and
// dE = g*dY is stored as the row goes by.  The row is walked in stretches of
// 32*DU chunks, the next stretch's dY and expert-output chunks loaded before
// the current one is used; the next item's route entry is fetched while this
// item's rows move.
constexpr int DU = 2;   // 16-byte chunks per lane per stretch

struct DbStretch {
    V16 dv[DU];
    V16 ov[DU];
};

__device__ __forceinline__ void db_load(DbStretch &b, const V16 *dyp, const V16 *op, int q0,
                                        int nch) {
#pragma unroll
    for (int u = 0; u < DU; u++)
        if (q0 + 32 * u < nch) {
            b.dv[u] = ld_v16(dyp + q0 + 32 * u);   // kept in cache for the token's other routes
            b.ov[u] = ld_stream(op + q0 + 32 * u);
        }
}

template <typename T>
__global__ void __launch_bounds__(DNT, 4)
decode_bwd_kernel(const T *__restrict__ dy, const T *__restrict__ out,
                  const int32_t *__restrict__ idx, const int32_t *__restrict__ loc,
                  const float *__restrict__ gates, const int32_t *__restrict__ c_dev, int64_t s,
                  int m, int e, int k, int64_t c_max, T *__restrict__ d_out,
                  float *__restrict__ d_gates, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    constexpr int VEC = Elt<T>::VEC;
    constexpr int SW = 32 * DU;   // chunks per stretch
    const int c_eff = read_c(c_dev, c_max);
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (DNT / 32);
    const int nch = m / VEC;
    const int64_t items = s * k;
    // item q = (token q / k, route q % k); lane 0 fetches the route's entry
    const bool small = items + nw <= 0x7fffffff;
    auto fetch = [&](int64_t q, int &ex, int &l, float &g) {
        ex = -1; l = -1; g = 0.0f;
        if (lane == 0 && q < items) {
            int64_t tq;
            int rq;
            split_item(q, k, small, tq, rq);
            const int64_t off = (int64_t)rq * s + tq;
            ex = idx[off];
            l = loc[off];
            g = gates[off];
        }
    };
    int64_t q = blockIdx.x * (DNT / 32) + (threadIdx.x >> 5);
    int nex, nl;
    float ng;
    fetch(q, nex, nl, ng);
    for (; q < items; q += nw) {
        int64_t t;
        int r;
        split_item(q, k, small, t, r);
        int ex = __shfl_sync(0xffffffffu, nex, 0), l = __shfl_sync(0xffffffffu, nl, 0);
        const float g = __shfl_sync(0xffffffffu, ng, 0);
        fetch(q + nw, nex, nl, ng);   // the next item's entry travels meanwhile
        if ((unsigned)ex >= (unsigned)e || l < 0) {
            if (lane == 0) set_status(status, MOE_ERR_INVALID_ARG);
            continue;
        }
        if (l >= c_eff) {   // dropped: no gradient
            if (lane == 0) d_gates[(int64_t)r * s + t] = 0.0f;
            continue;
        }
        const int64_t row = ((int64_t)ex * c_max + l) * m;
        const V16 *dyp = reinterpret_cast<const V16 *>(dy + t * m);
        const V16 *op = reinterpret_cast<const V16 *>(out + row);
        V16 *dp = reinterpret_cast<V16 *>(d_out + row);
        float part = 0.0f;
        auto use = [&](const DbStretch &b, int q0) {
#pragma unroll
            for (int u = 0; u < DU; u++)
                if (q0 + 32 * u < nch) {
                    float a[VEC], bb[VEC];
                    Elt<T>::unpack(b.dv[u], a);
                    Elt<T>::unpack(b.ov[u], bb);
#pragma unroll
                    for (int i = 0; i < VEC; i++) part = __fmaf_rn(a[i], bb[i], part);
                    st_v16(dp + q0 + 32 * u, ScaleRound<T>::apply(g, b.dv[u]));
                }
        };
        // two named stretch buffers, the loop unrolled by two
        DbStretch b0, b1;
        db_load(b0, dyp, op, lane, nch);
        for (int base = 0; base < nch; base += 2 * SW) {
            if (base + SW < nch) db_load(b1, dyp, op, base + SW + lane, nch);
            use(b0, base + lane);
            if (base + 2 * SW < nch) db_load(b0, dyp, op, base + 2 * SW + lane, nch);
            if (base + SW < nch) use(b1, base + SW + lane);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) d_gates[(int64_t)r * s + t] = part;
    }
}

int sm_count_cached() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 148;
    }
    return cached[dev];
}

// CTAs for `items` one-warp work items: one item per warp, but never more CTAs
// than are resident at once (4 per SM at the kernels' <= 64 registers), so no
// partial second wave; larger batches loop inside each warp.
int grid_for_items(int64_t items) {
    int64_t want = (items + (DNT / 32) - 1) / (DNT / 32);
    int64_t cap = (int64_t)sm_count_cached() * 4;
    return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}


int64_t row_slices(int m, moe_dtype dt) {
    const int nch = m / (dt == MOE_BF16 ? 8 : 4);
    return (nch + SL - 1) / SL;
}

}  // namespace

moe_status encode_launch(const void *x, moe_dtype dt, const int32_t *idx, const int32_t *loc,
                         const int32_t *counts, const int32_t *c_dev, int64_t s, int m, int e,
                         int k, int64_t c_max, unsigned flags, void *buf, int32_t *st,
                         cudaStream_t stream, int lo, int hi) {
    const int grid = grid_for_items(s * row_slices(m, dt));
    moe_status r;
    if (dt == MOE_BF16)
        r = launch_pdl(encode_kernel<__nv_bfloat16>, dim3(grid), dim3(DNT), 0, stream,
                       (const __nv_bfloat16 *)x, idx, loc, c_dev, s, m, e, k, c_max,
                       (__nv_bfloat16 *)buf, st, lo, hi);
    else
        r = launch_pdl(encode_kernel<float>, dim3(grid), dim3(DNT), 0, stream, (const float *)x, idx,
                       loc, c_dev, s, m, e, k, c_max, (float *)buf, st, lo, hi);
    if (r != MOE_OK) return r;
    if (flags & MOE_FLAG_ZERO_FILL) {
        int64_t gx = (c_max + (DNT / 32) - 1) / (DNT / 32);
        dim3 g((unsigned)(gx < 1024 ? gx : 1024), (unsigned)e);
        if (dt == MOE_BF16)
            r = launch_pdl(zero_fill_kernel<__nv_bfloat16>, g, dim3(DNT), 0, stream, counts, c_dev, e,
                           c_max, m, (__nv_bfloat16 *)buf, st);
        else
            r = launch_pdl(zero_fill_kernel<float>, g, dim3(DNT), 0, stream, counts, c_dev, e, c_max,
                           m, (float *)buf, st);
        if (r != MOE_OK) return r;
    }
    return MOE_OK;
}

template <typename T, bool W>
moe_status combine_typed(const void *src, const int32_t *idx, const int32_t *loc, const float *gates,
                         const int32_t *c_dev, int64_t s, int m, int e, int k, int64_t c_max,
                         void *y, int32_t *st, cudaStream_t stream) {
    constexpr int VEC = Elt<T>::VEC;
    const int nch = m / VEC;
    const dim3 b(DNT);
    const T *sp = (const T *)src;
    T *yp = (T *)y;
    if (k <= 2) {  // all routes in one group: 4 chunks per lane, 8 live accumulators
        const int64_t items = s * ((nch + 127) / 128);
        return launch_pdl(combine_kernel<T, W, 4, 2, true>, dim3(grid_for_items(items)), b, 0, stream,
                          sp, idx, loc, gates, c_dev, s, m, e, k, c_max, yp, st);
    }
    if (k <= 4) {  // all routes in one group: 2 chunks per lane, 8 live accumulators
        const int64_t items = s * ((nch + 63) / 64);
        return launch_pdl(combine_kernel<T, W, 2, 4, true>, dim3(grid_for_items(items)), b, 0, stream,
                          sp, idx, loc, gates, c_dev, s, m, e, k, c_max, yp, st);
    }
    const int64_t items = s * ((nch + 63) / 64);
    return launch_pdl(combine_kernel<T, W, 2, 4, false>, dim3(grid_for_items(items)), b, 0, stream,
                      sp, idx, loc, gates, c_dev, s, m, e, k, c_max, yp, st);
}

moe_status combine_launch(const void *src, moe_dtype dt, const int32_t *idx, const int32_t *loc,
                          const float *gates, const int32_t *c_dev, int64_t s, int m, int e, int k,
                          int64_t c_max, void *y, int32_t *st, cudaStream_t stream) {
    const bool w = gates != nullptr;
    if (dt == MOE_BF16)
        return w ? combine_typed<__nv_bfloat16, true>(src, idx, loc, gates, c_dev, s, m, e, k, c_max, y, st, stream)
                 : combine_typed<__nv_bfloat16, false>(src, idx, loc, gates, c_dev, s, m, e, k, c_max, y, st, stream);
    return w ? combine_typed<float, true>(src, idx, loc, gates, c_dev, s, m, e, k, c_max, y, st, stream)
             : combine_typed<float, false>(src, idx, loc, gates, c_dev, s, m, e, k, c_max, y, st, stream);
}

moe_status decode_bwd_launch(const void *dy, const void *out, moe_dtype dt, const int32_t *idx,
                             const int32_t *loc, const float *gates, const int32_t *counts,
                             const int32_t *c_dev, int64_t s, int m, int e, int k, int64_t c_max,
                             unsigned flags, void *d_out, float *d_gates, int32_t *st,
                             cudaStream_t stream) {
    if (flags & MOE_FLAG_ZERO_FILL) {
        int64_t gx = (c_max + (DNT / 32) - 1) / (DNT / 32);
        dim3 g((unsigned)(gx < 1024 ? gx : 1024), (unsigned)e);
        moe_status r;
        if (dt == MOE_BF16)
            r = launch_pdl(zero_fill_kernel<__nv_bfloat16>, g, dim3(DNT), 0, stream, counts, c_dev, e,
                           c_max, m, (__nv_bfloat16 *)d_out, st);
        else
            r = launch_pdl(zero_fill_kernel<float>, g, dim3(DNT), 0, stream, counts, c_dev, e, c_max,
                           m, (float *)d_out, st);
        if (r != MOE_OK) return r;
    }
    const int grid = grid_for_items(s * k);
    if (dt == MOE_BF16)
        return launch_pdl(decode_bwd_kernel<__nv_bfloat16>, dim3(grid), dim3(DNT), 0, stream,
                          (const __nv_bfloat16 *)dy, (const __nv_bfloat16 *)out, idx, loc, gates,
                          c_dev, s, m, e, k, c_max, (__nv_bfloat16 *)d_out, d_gates, st);
    return launch_pdl(decode_bwd_kernel<float>, dim3(grid), dim3(DNT), 0, stream, (const float *)dy,
                      (const float *)out, idx, loc, gates, c_dev, s, m, e, k, c_max, (float *)d_out,
                      d_gates, st);
}

}  // namespace moe
