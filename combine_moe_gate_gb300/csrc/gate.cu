// Fused gate: fp32 logits -> softmax -> top-k, one CTA per tile of tokens.
//
// Method: the Tutel profile's gate_type {'type': 'top', 'k': k} (top-k softmax
// gate) and the DeepSpeed-MoE vs Tutel blog, section 1.4 (top-k fused into one
// kernel that emits a dense token-to-expert table instead of a one-hot mask).
//
// Logit order (fixed so routing is reproducible bit for bit; fp32 with one
// rounding per fused multiply-add, then one fp32 add of the bias):
//   e <= 32: the features are cut into chunks of one 16-byte load (8 bf16 or 4
//     fp32 elements); chunk c belongs to lane c mod 32, each lane accumulates
//     its features from +0 in ascending index, and the 32 lane sums are
//     combined by an xor butterfly (o = 16, 8, 4, 2, 1; the logit is lane 0's).
//     gate_lane_kernel is exactly that: lane l of a warp owns chunk l of every
//     512-byte slice of the feature axis.
//   e > 32: one accumulator per logit from +0 in ascending feature index.
//     gate_seq_kernel is a persistent register-blocked SIMT GEMM: warps own
//     expert groups, lanes own tokens, and each accumulator walks the features
//     in order.  (The lane-blocked order needs 32 live partial sums per logit;
//     with all e experts of a token in one CTA, as the fused top-k needs, that
//     leaves a CTA only a handful of tokens for large e.)
// Tensor cores are not used: their internal accumulation order is unspecified
// and would make routing irreproducible.
#include "common.cuh"

namespace moe {
namespace {

// Feature u (compile-time) of a 16-byte chunk, widened exactly to fp32.
template <typename XT, int U>
__device__ __forceinline__ float chunk_elem(const V16 &v) {
    if constexpr (sizeof(XT) == 2)
        return (U & 1) ? bf16hi(v.w[U >> 1]) : bf16lo(v.w[U >> 1]);
    else
        return __uint_as_float(v.w[U]);
}

// e > 32: a persistent CTA of NW warps computes chunks of TOKC tokens x all
// EP experts, chunk after chunk.  The warps form WT token groups x WE expert
// groups: warp (wt, we) owns experts [we*EW, (we+1)*EW) of the chunk's tokens
// wt*32*TT + lane + 32*j (j < TT).  Per K tile of KT features the CTA stages
// the chunk's x rows as they lie in memory (16 bytes = VEC features of one
// token per load) and the tile's weight rows [KT][EP] in fp32; per feature, a
// warp's weight loads are the same address in every lane (a broadcast), so
// shared-memory traffic stays well below what the fp32 pipe consumes.  Two
// experts' chains advance per packed fp32x2 fused multiply-add (each lane of
// the pair rounds exactly as fmaf), so issue slots are left for the loads.
// Every accumulator walks the features in ascending order.  After a chunk's
// last tile the logits (+ bias) go to shared memory -- into the stage just
// consumed when they fit there, which the next refill only reaches after the
// next barrier -- and one warp per token does softmax and top-k, while the
// next chunk's tiles are already in flight.
template <int EP_, int EW_, int TT_, int NW_, int KT_, int ST_, typename XT>
struct SeqCfg {
    static constexpr int EP = EP_;                       // experts per CTA (e padded)
    static constexpr int EW = EW_;                       // experts per warp
    static constexpr int TT = TT_;                       // tokens per lane
    static constexpr int NW = NW_;                       // warps per CTA
    static constexpr int KT = KT_;                       // features per K tile
    static constexpr int ST = ST_;                       // pipeline stages
    static constexpr int NT = NW * 32;
    static constexpr int WE = EP / EW;                   // warps along experts
    static constexpr int WT = NW / WE;                   // warps along tokens
    static constexpr int TOKC = WT * 32 * TT;            // tokens per chunk
    static constexpr int VEC = Elt<XT>::VEC;             // features per 16-byte x load
    static constexpr int XCH = KT / VEC;                 // 16-byte chunks per x row and tile
    static constexpr int XROW = KT * Elt<XT>::BYTES + 16;  // padded x row (bytes)
    static constexpr int X_BYTES = TOKC * XROW;
    static constexpr int W_BYTES = KT * EP * 4;
    static constexpr int STAGE = X_BYTES + W_BYTES;
    static constexpr int LGS = EP + 1;                   // logits row stride (floats)
    static constexpr int LG_BYTES = TOKC * LGS * 4;
    static constexpr bool LG_IN_STAGE = LG_BYTES <= STAGE;
    static constexpr int SMEM = ST * STAGE + (LG_IN_STAGE ? 0 : LG_BYTES);
    static_assert(EP % EW == 0 && NW % WE == 0 && EW % 4 == 0 && EP > 32, "experts per warp");
    static_assert(KT % VEC == 0 && X_BYTES % 16 == 0 && W_BYTES % 16 == 0 && ST >= 2, "stages");
};

// Stage one K tile of one chunk: x rows [t0, t0 + TOKC) x features [k0, k0 + KT)
// and weight rows [k0, k0 + KT) (zero past s, m and e).
template <class C, typename XT>
__device__ __forceinline__ void seq_load(unsigned char *st, const XT *x, const float *wg, int64_t s,
                                         int m, int e, int64_t t0, int k0, bool wg16) {
    for (int q = threadIdx.x; q < C::TOKC * C::XCH; q += C::NT) {
        const int row = q / C::XCH, ch = q % C::XCH;
        const int64_t t = t0 + row;
        const int f = k0 + ch * C::VEC;
        const bool ok = t < s && f < m;
        cp_async16(st + row * C::XROW + ch * 16, ok ? (const void *)(x + t * m + f) : (const void *)x,
                   ok);
    }
    float *ws = reinterpret_cast<float *>(st + C::X_BYTES);
    if (wg16) {
        for (int q = threadIdx.x; q < C::KT * (C::EP / 4); q += C::NT) {
            const int kk = q / (C::EP / 4), j = (q % (C::EP / 4)) * 4;
            const bool ok = k0 + kk < m && j < e;
            cp_async16(ws + kk * C::EP + j, ok ? (const void *)(wg + (int64_t)(k0 + kk) * e + j)
                                               : (const void *)wg, ok);
        }
    } else {
        for (int q = threadIdx.x; q < C::KT * C::EP; q += C::NT) {
            const int kk = q / C::EP, j = q % C::EP;
            const bool ok = k0 + kk < m && j < e;
            cp_async4(ws + kk * C::EP + j, ok ? (const void *)(wg + (int64_t)(k0 + kk) * e + j)
                                              : (const void *)wg, ok);
        }
    }
    cp_async_commit();
}

// One feature U (compile-time) of the lane's x chunks: acc[j][i..i+1] +=
// x[token j][f] * w[f][expert i..i+1] for every token j and expert pair.
template <class C, typename XT, int U>
__device__ __forceinline__ void seq_feature(float2 (&acc)[C::TT][C::EW / 2], const V16 (&xv)[C::TT],
                                            const float *wf) {
    float2 w2[C::EW / 2];
#pragma unroll
    for (int q = 0; q < C::EW / 4; q++) {
        const float4 w4 = reinterpret_cast<const float4 *>(wf)[q];   // same address in every lane
        w2[2 * q] = make_float2(w4.x, w4.y);
        w2[2 * q + 1] = make_float2(w4.z, w4.w);
    }
#pragma unroll
    for (int j = 0; j < C::TT; j++) {
        const float xf = chunk_elem<XT, U>(xv[j]);
        const float2 x2 = make_float2(xf, xf);
#pragma unroll
        for (int i = 0; i < C::EW / 2; i++) acc[j][i] = __ffma2_rn(x2, w2[i], acc[j][i]);
    }
}

template <class C, typename XT, int U>
__device__ __forceinline__ void seq_group(float2 (&acc)[C::TT][C::EW / 2], const V16 (&xv)[C::TT],
                                          const float *wg_tile) {
    if constexpr (U < C::VEC) {
        seq_feature<C, XT, U>(acc, xv, wg_tile + U * C::EP);
        seq_group<C, XT, U + 1>(acc, xv, wg_tile);
    }
}

// Softmax over the e logits of one token and top-k (ties -> lower index), one
// warp; lane r < k writes route r.
__device__ __forceinline__ void softmax_topk_warp(const float *row, int e, int k, int normalize,
                                                  int64_t t, int64_t s, int32_t *idx, float *gates,
                                                  int qe) {
    const int lane = threadIdx.x & 31;
    constexpr int QMAX = 8;                      // e <= 256
    float v[QMAX];
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < QMAX; q++) {
        const int ex = lane + 32 * q;
        v[q] = (q < qe && ex < e) ? row[ex] : -INFINITY;
        mx = fmaxf(mx, v[q]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float z = 0.0f;
#pragma unroll
    for (int q = 0; q < QMAX; q++)
        if (q < qe && lane + 32 * q < e) z += expf(v[q] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    unsigned taken = 0;  // bit q: expert lane+32q already selected
    float my_v = 0.0f;   // lane r keeps route r's logit and expert
    int my_j = 0;
    for (int r = 0; r < k; r++) {
        float bv = -INFINITY;
        int bj = 0x7fffffff;
#pragma unroll
        for (int q = 0; q < QMAX; q++) {
            const int ex = lane + 32 * q;
            const bool cand = q < qe && ex < e && !((taken >> q) & 1u);
            if (cand && (v[q] > bv || (v[q] == bv && ex < bj))) { bv = v[q]; bj = ex; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
            if (ov > bv || (ov == bv && oj < bj)) { bv = ov; bj = oj; }
        }
        if ((bj & 31) == lane) taken |= 1u << (bj >> 5);
        if (lane == r) { my_v = bv; my_j = bj; }
    }
    const float p = lane < k ? expf(my_v - mx) : 0.0f;
    float g;
    if (normalize) {
        float sel = p;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sel += __shfl_xor_sync(0xffffffffu, sel, o);
        g = p / sel;
    } else {
        g = p / z;
    }
    if (lane < k) {
        idx[(int64_t)lane * s + t] = my_j;
        gates[(int64_t)lane * s + t] = g;
    }
}

template <class C, typename XT>
__global__ void __launch_bounds__(C::NT)
gate_seq_kernel(const XT *__restrict__ x, const float *__restrict__ wg,
                const float *__restrict__ bias, int64_t s, int m, int e, int k, int normalize,
                int32_t *__restrict__ idx, float *__restrict__ gates, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    extern __shared__ __align__(16) unsigned char smem_seq[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int we = warp % C::WE, wt = warp / C::WE;   // expert group, token group
    const int tok0 = wt * 32 * C::TT + lane;          // the lane's first token in a chunk
    const bool wg16 = (e % 4) == 0;   // rows of wg start on 16-byte boundaries
    const int ntiles = (m + C::KT - 1) / C::KT;
    const int64_t nchunks = (s + C::TOKC - 1) / C::TOKC;
    const int64_t my_chunks =
        blockIdx.x < nchunks ? (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t total = my_chunks * ntiles;   // (chunk, tile) steps of this CTA, flattened
    // the step being issued (ST - 1 ahead of the one computed): chunk, tile, stage
    int64_t ichunk = blockIdx.x;
    int ikt = 0, ist = 0;
    auto issue_next = [&]() {
        seq_load<C, XT>(smem_seq + ist * C::STAGE, x, wg, s, m, e, ichunk * C::TOKC, ikt * C::KT,
                        wg16);
        ist = ist + 1 == C::ST ? 0 : ist + 1;
        if (++ikt == ntiles) {
            ikt = 0;
            ichunk += gridDim.x;
        }
    };
#pragma unroll
    for (int p = 0; p < C::ST - 1; p++) {
        if (p < total) issue_next();
        else cp_async_commit();
    }
    float2 acc[C::TT][C::EW / 2];
    const int qe = (e + 31) / 32;
    int kt = 0, st_q = 0;
    int64_t chunk = blockIdx.x;   // the computed step's chunk
    for (int64_t q = 0; q < total; q++) {
        cp_async_wait<C::ST - 2>();
        __syncthreads();   // step q landed; step q-1 (and the previous softmax) fully read
        if (q + C::ST - 1 < total) issue_next();
        else cp_async_commit();
        if (kt == 0) {
#pragma unroll
            for (int j = 0; j < C::TT; j++)
#pragma unroll
                for (int i = 0; i < C::EW / 2; i++) acc[j][i] = make_float2(0.0f, 0.0f);
        }
        unsigned char *st = smem_seq + st_q * C::STAGE;
        const float *wtile = reinterpret_cast<const float *>(st + C::X_BYTES) + we * C::EW;
        const int ngroups = min(C::KT, m - kt * C::KT) / C::VEC;   // m is a multiple of VEC
#pragma unroll 1
        for (int g = 0; g < ngroups; g++) {
            V16 xv[C::TT];
#pragma unroll
            for (int j = 0; j < C::TT; j++)
                xv[j] = *reinterpret_cast<const V16 *>(st + (tok0 + 32 * j) * C::XROW + g * 16);
            seq_group<C, XT, 0>(acc, xv, wtile + g * C::VEC * C::EP);
        }
        if (kt == ntiles - 1) {
            // the chunk's logits (+ bias: one fp32 add after the chain), in the
            // stage just read once every warp is done with it
            float *lg = reinterpret_cast<float *>(C::LG_IN_STAGE ? st : smem_seq + C::ST * C::STAGE);
            if (C::LG_IN_STAGE) __syncthreads();
#pragma unroll
            for (int j = 0; j < C::TT; j++)
#pragma unroll
                for (int i = 0; i < C::EW / 2; i++) {
                    const int ex = we * C::EW + 2 * i;
                    float a = acc[j][i].x, b = acc[j][i].y;
                    if (bias) {
                        if (ex < e) a = a + bias[ex];
                        if (ex + 1 < e) b = b + bias[ex + 1];
                    }
                    lg[(tok0 + 32 * j) * C::LGS + ex] = a;
                    lg[(tok0 + 32 * j) * C::LGS + ex + 1] = b;
                }
            __syncthreads();
            const int64_t t0 = chunk * C::TOKC;
            for (int tl = warp; tl < C::TOKC; tl += C::NW) {
                const int64_t t = t0 + tl;
                if (t >= s) break;
                softmax_topk_warp(lg + tl * C::LGS, e, k, normalize, t, s, idx, gates, qe);
            }
        }
        st_q = st_q + 1 == C::ST ? 0 : st_q + 1;
        if (++kt == ntiles) {
            kt = 0;
            chunk += gridDim.x;
        }
    }
    cp_async_wait<0>();
}

// ---------------------------------------------------------------- small e
// e <= 32: the lane-blocked logit order.  Each K tile is a 512-byte slice of
// the feature axis, i.e. 32 chunks of one 16-byte load (V = 8 bf16 or 4 fp32
// features); lane l of every warp owns chunk l of every tile, so over the tiles
// it visits exactly the chunks c with c mod 32 = l, in ascending order.  A warp
// computes T = 64 / EP tokens x all EP experts (64 accumulators per lane); its
// lanes' x loads cover 512 contiguous bytes of a token row, and the K tile's
// weight block is staged as [chunk][feature][expert] with each chunk's block
// padded by 16 bytes, so the lanes' 16-byte weight loads fall on distinct
// banks.  x rows and weight blocks stream through an SK-deep cp.async ring.
// After the last tile an xor butterfly over the lanes finishes every logit,
// and one lane per token does softmax and top-k.
constexpr int SK = 4;    // K tiles in flight
constexpr int LNW = 4;   // warps per CTA

template <int EP, typename XT>
struct LaneCfg {
    static constexpr int V = 16 / (int)sizeof(XT);   // features per chunk (one 16-byte load)
    static constexpr int KS = 32 * V;                // features per K tile
    static constexpr int T = 64 / EP;                // tokens per warp
    static constexpr int TC = LNW * T;               // tokens per CTA
    static constexpr int XROWB = 512 + 16;           // x tile row (bytes, padded)
    static constexpr int XB = TC * XROWB;            // x tile bytes
    static constexpr int WCH = V * EP + 4;           // floats per chunk block of the weight tile
    static constexpr int WB = 32 * WCH * 4;          // weight tile bytes
    static constexpr int STAGE = XB + WB;
    static constexpr int SMEM = SK * STAGE;
    static_assert(EP >= 4 && EP <= 32 && 64 % EP == 0, "experts per CTA");
    static_assert(XB % 16 == 0 && WB % 16 == 0, "16-byte stages");
};

template <typename XT, int EP, int T, int U>
__device__ __forceinline__ void lane_fma_feature(float (&acc)[T][EP], const V16 (&xv)[T],
                                                 const float *wu) {
    float w[EP];
#pragma unroll
    for (int q = 0; q < EP / 4; q++) {
        const float4 w4 = reinterpret_cast<const float4 *>(wu)[q];
        w[4 * q] = w4.x; w[4 * q + 1] = w4.y; w[4 * q + 2] = w4.z; w[4 * q + 3] = w4.w;
    }
#pragma unroll
    for (int tt = 0; tt < T; tt++) {
        const float xf = chunk_elem<XT, U>(xv[tt]);
#pragma unroll
        for (int jj = 0; jj < EP; jj++) acc[tt][jj] = fmaf(xf, w[jj], acc[tt][jj]);
    }
}

// The same with packed fp32x2 FMAs over expert pairs (each half rounds exactly
// as fmaf, so the sums are the same bits): acc[tt][i] holds experts 2i, 2i + 1.
template <typename XT, int EP, int T, int U>
__device__ __forceinline__ void lane_fma2_feature(float2 (&acc)[T][EP / 2], const V16 (&xv)[T],
                                                  const float *wu) {
    float2 w[EP / 2];
#pragma unroll
    for (int q = 0; q < EP / 4; q++) {
        const float4 w4 = reinterpret_cast<const float4 *>(wu)[q];
        w[2 * q] = make_float2(w4.x, w4.y);
        w[2 * q + 1] = make_float2(w4.z, w4.w);
    }
#pragma unroll
    for (int tt = 0; tt < T; tt++) {
        const float xf = chunk_elem<XT, U>(xv[tt]);
        const float2 x2 = make_float2(xf, xf);
#pragma unroll
        for (int i = 0; i < EP / 2; i++) acc[tt][i] = __ffma2_rn(x2, w[i], acc[tt][i]);
    }
}

template <typename XT, int EP, int T, int U, int V>
__device__ __forceinline__ void lane_fma2_chunk(float2 (&acc)[T][EP / 2], const V16 (&xv)[T],
                                                const float *wc) {
    if constexpr (U < V) {
        lane_fma2_feature<XT, EP, T, U>(acc, xv, wc + U * EP);
        lane_fma2_chunk<XT, EP, T, U + 1, V>(acc, xv, wc);
    }
}

template <typename XT, int EP, int T, int U, int V>
__device__ __forceinline__ void lane_fma_chunk(float (&acc)[T][EP], const V16 (&xv)[T],
                                               const float *wc) {
    if constexpr (U < V) {
        lane_fma_feature<XT, EP, T, U>(acc, xv, wc + U * EP);
        lane_fma_chunk<XT, EP, T, U + 1, V>(acc, xv, wc);
    }
}

template <int EP, typename XT>
__global__ void __launch_bounds__(LNW * 32)
gate_lane_kernel(const XT *__restrict__ x, const float *__restrict__ wg,
                 const float *__restrict__ bias, int64_t s, int m, int e, int k, int normalize,
                 int32_t *__restrict__ idx, float *__restrict__ gates, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    using C = LaneCfg<EP, XT>;
    constexpr int V = C::V, T = C::T, NT = LNW * 32;
    extern __shared__ __align__(16) unsigned char smem_lane[];
    const int64_t t0 = (int64_t)blockIdx.x * C::TC;
    const int ntiles = (m + C::KS - 1) / C::KS;
    const int nch = m / V;                               // m is a multiple of V
    const bool wvec = e == EP;                           // whole 16-byte weight rows
    auto load_tile = [&](int tile) {
        unsigned char *st = smem_lane + (tile % SK) * C::STAGE;
        for (int q = threadIdx.x; q < C::TC * 32; q += NT) {   // x: the CTA's rows, 32 chunks
            const int row = q >> 5, ch = q & 31;
            const int64_t t = t0 + row;
            const int f = tile * C::KS + ch * V;
            const bool ok = t < s && f < m;
            cp_async16(st + row * C::XROWB + ch * 16,
                       ok ? (const void *)(x + t * m + f) : (const void *)x, ok);
        }
        float *wt = reinterpret_cast<float *>(st + C::XB);
        if (wvec) {   // weight rows of EP floats, 16 bytes at a time
            for (int q = threadIdx.x; q < C::KS * (EP / 4); q += NT) {
                const int g = q % (EP / 4), r = q / (EP / 4);   // r = chunk * V + feature
                const int ch = r / V, u = r - ch * V;
                const int f = tile * C::KS + r;
                const bool ok = f < m;
                cp_async16(wt + ch * C::WCH + u * EP + g * 4,
                           ok ? (const void *)(wg + (int64_t)f * e + g * 4) : (const void *)wg, ok);
            }
        } else {      // e < EP: one float at a time, zero for experts >= e
            for (int q = threadIdx.x; q < C::KS * EP; q += NT) {
                const int jj = q % EP, r = q / EP;
                const int ch = r / V, u = r - ch * V;
                const int f = tile * C::KS + r;
                const bool ok = f < m && jj < e;
                cp_async4(wt + ch * C::WCH + u * EP + jj,
                          ok ? (const void *)(wg + (int64_t)f * e + jj) : (const void *)wg, ok);
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int p = 0; p < SK - 1; p++) {
        if (p < ntiles) load_tile(p);
        else cp_async_commit();
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc[T][EP];
#pragma unroll
    for (int tt = 0; tt < T; tt++)
#pragma unroll
        for (int jj = 0; jj < EP; jj++) acc[tt][jj] = 0.0f;
    for (int it = 0; it < ntiles; it++) {
        cp_async_wait<SK - 2>();
        __syncthreads();   // tile `it` landed; tile it-1 fully read
        if (it + SK - 1 < ntiles) load_tile(it + SK - 1);
        else cp_async_commit();
        if (it * 32 + lane < nch) {   // this lane's chunk of the tile holds features
            const unsigned char *st = smem_lane + (it % SK) * C::STAGE;
            V16 xv[T];
#pragma unroll
            for (int tt = 0; tt < T; tt++)
                xv[tt] = *reinterpret_cast<const V16 *>(st + (warp * T + tt) * C::XROWB + lane * 16);
            const float *wc = reinterpret_cast<const float *>(st + C::XB) + lane * C::WCH;
            lane_fma_chunk<XT, EP, T, 0, V>(acc, xv, wc);
        }
    }
    cp_async_wait<0>();
    // xor butterfly over the lanes: every lane ends with every full logit
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int tt = 0; tt < T; tt++)
#pragma unroll
            for (int jj = 0; jj < EP; jj++)
                acc[tt][jj] = acc[tt][jj] + __shfl_xor_sync(0xffffffffu, acc[tt][jj], o);
    if (lane >= T) return;
    const int64_t t = t0 + warp * T + lane;
    if (t >= s) return;
    // lane tt takes token tt's row (a static selection keeps it in registers)
    float row[EP];
#pragma unroll
    for (int jj = 0; jj < EP; jj++) row[jj] = acc[0][jj];
#pragma unroll
    for (int tt = 1; tt < T; tt++)
        if (lane == tt) {
#pragma unroll
            for (int jj = 0; jj < EP; jj++) row[jj] = acc[tt][jj];
        }
    float mx = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < EP; jj++)
        if (jj < e) {
            if (bias) row[jj] = row[jj] + bias[jj];
            mx = fmaxf(mx, row[jj]);
        }
    float z = 0.0f;
#pragma unroll
    for (int jj = 0; jj < EP; jj++)
        if (jj < e) z += expf(row[jj] - mx);
    // top-k: k rounds of arg-max over the experts not yet taken (ties -> lower
    // index); the first pass sums the selected probabilities, the second repeats
    // the same selection and writes it
    float sel = 0.0f;
    for (int pass = 0; pass < 2; pass++) {
        uint32_t taken = 0;
        for (int r = 0; r < k; r++) {
            int bj = -1;
            float bv = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < EP; jj++) {
                if (jj < e && !(taken & (1u << jj)) && (bj < 0 || row[jj] > bv)) {
                    bv = row[jj];
                    bj = jj;
                }
            }
            taken |= 1u << bj;
            const float p = expf(bv - mx);
            if (pass == 0) {
                sel += p;
            } else {
                idx[(int64_t)r * s + t] = bj;
                gates[(int64_t)r * s + t] = p / (normalize ? sel : z);
            }
        }
    }
}

// The same lane-blocked order with the whole gate weight resident in shared
// memory (when it fits): a persistent CTA loads Wg once, staged as
// [tile][chunk][feature][expert] with every chunk block padded by 16 bytes,
// and takes one contiguous range of the T-token groups, dealt to its warps in
// turn.  Each lane streams its own 16-byte x chunks through a private RD-deep
// cp.async ring in shared memory (a lane only ever reads what it copied
// itself, so no lane waits on another).  The lane sums are combined by a
// reduce-scatter form of the xor butterfly: at offset o a lane keeps the half
// of its values selected by lane bit o and adds the partner's copy of that
// half, so every logit is the same sum v[l] + v[l ^ o] at every level as in
// the full butterfly, with a fifth of the shuffles; lane l ends with the
// flattened (token, expert) values 2l and 2l + 1, so token tt's EP logits sit
// in the EP / 2 lanes from tt * EP / 2 on, which then do its softmax and
// top-k together with shuffles inside that lane segment.
constexpr int RW_MAX = 16;                // warps per CTA (at most)
// fewer warps (more registers a lane) the more tokens a warp holds
template <int EP> constexpr int res_warps_max() { return EP >= 32 ? RW_MAX : EP == 16 ? 12 : 8; }
constexpr int RD = 3;                     // K tiles of x in flight per warp
constexpr size_t RES_SMEM_MAX = 220 * 1024;

template <int EP, typename XT>
struct ResCfg {
    static constexpr int V = 16 / (int)sizeof(XT);
    static constexpr int KS = 32 * V;
    static constexpr int T = 64 / EP;
    static constexpr int WCH = V * EP + 4;           // floats per chunk block (16-byte pad)
    static constexpr int TILE_FLOATS = 32 * WCH;
    static constexpr int RING_BYTES = RD * T * 32 * 16;   // per warp
    static size_t smem(int m, int nw) {
        return (size_t)((m + KS - 1) / KS) * TILE_FLOATS * 4 + (size_t)nw * RING_BYTES;
    }
};

// Reduce-scatter step: n values -> n/2, lane bit `o` picks the kept half.
template <int N, int O>
__device__ __forceinline__ void rs_step(float (&v)[64], int lane) {
    const bool hi = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; i++) {
        const float keep = hi ? v[N / 2 + i] : v[i];
        const float give = hi ? v[i] : v[N / 2 + i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, give, O);
    }
}

// Softmax and top-k of one token whose logits a and b (experts j0, j0 + 1)
// are spread over a segment of S = EP / 2 lanes: max and sum by xor shuffles
// inside the segment, then k rounds of segment arg-max over the experts not
// yet taken (ties -> lower index).  Route r is written by the segment's lane
// r mod S; its gate divides by the selected probabilities summed in route
// order (renormalised) or by the softmax sum.
template <int S>
__device__ __forceinline__ void segment_topk(float a, float b, int j0, int e, int k, int normalize,
                                             int64_t t, int64_t s, int32_t *idx, float *gates,
                                             int lane) {
    const bool va = j0 < e, vb = j0 + 1 < e;
    float mx = fmaxf(va ? a : -INFINITY, vb ? b : -INFINITY);
#pragma unroll
    for (int o = S / 2; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float z = (va ? expf(a - mx) : 0.0f) + (vb ? expf(b - mx) : 0.0f);
#pragma unroll
    for (int o = S / 2; o >= 1; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const int ls = lane % S;
    bool ta = !va, tb = !vb;   // taken (or not an expert)
    float sel = 0.0f, rp0 = 0.0f, rp1 = 0.0f;
    int rj0 = 0, rj1 = 0;
    for (int r = 0; r < k; r++) {
        float cv = -INFINITY;
        int cj = 0x7fffffff;
        if (!ta) { cv = a; cj = j0; }
        if (!tb && (cj == 0x7fffffff || b > cv)) { cv = b; cj = j0 + 1; }
#pragma unroll
        for (int o = S / 2; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, cv, o);
            const int oj = __shfl_xor_sync(0xffffffffu, cj, o);
            if (oj != 0x7fffffff && (cj == 0x7fffffff || ov > cv || (ov == cv && oj < cj))) {
                cv = ov;
                cj = oj;
            }
        }
        ta = ta || cj == j0;
        tb = tb || cj == j0 + 1;
        const float p = expf(cv - mx);
        sel += p;
        if (r == ls) { rj0 = cj; rp0 = p; }
        if (r == ls + S) { rj1 = cj; rp1 = p; }
    }
    if (t >= s) return;
    const float den = normalize ? sel : z;
    if (ls < k) {
        idx[(int64_t)ls * s + t] = rj0;
        gates[(int64_t)ls * s + t] = rp0 / den;
    }
    if (ls + S < k) {
        idx[(int64_t)(ls + S) * s + t] = rj1;
        gates[(int64_t)(ls + S) * s + t] = rp1 / den;
    }
}

template <int EP, typename XT>
__global__ void __launch_bounds__(res_warps_max<EP>() * 32, 1)
gate_lane_res_kernel(const XT *__restrict__ x, const float *__restrict__ wg,
                     const float *__restrict__ bias, int64_t s, int m, int e, int k, int normalize,
                     int32_t *__restrict__ idx, float *__restrict__ gates, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    using C = ResCfg<EP, XT>;
    constexpr int V = C::V, T = C::T;
    const int nw = blockDim.x >> 5, nt = blockDim.x;
    extern __shared__ __align__(16) unsigned char smem_res[];
    float *wres = reinterpret_cast<float *>(smem_res);
    const int ntiles = (m + C::KS - 1) / C::KS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t w_bytes = (size_t)ntiles * C::TILE_FLOATS * 4;
    unsigned char *ring = smem_res + w_bytes + (size_t)warp * C::RING_BYTES;
    const int nch = m / V;                                       // m is a multiple of V
    // the whole weight, zero past m features and e experts
    if (e == EP) {
        for (int q = threadIdx.x; q < ntiles * C::KS * (EP / 4); q += nt) {
            const int g = q % (EP / 4), r = q / (EP / 4);          // r = feature
            const int tile = r / C::KS, rr = r - tile * C::KS, ch = rr / V, u = rr - ch * V;
            const bool ok = r < m;
            cp_async16(wres + (size_t)tile * C::TILE_FLOATS + ch * C::WCH + u * EP + g * 4,
                       ok ? (const void *)(wg + (int64_t)r * e + g * 4) : (const void *)wg, ok);
        }
    } else {
        for (int q = threadIdx.x; q < ntiles * C::KS * EP; q += nt) {
            const int jj = q % EP, r = q / EP;
            const int tile = r / C::KS, rr = r - tile * C::KS, ch = rr / V, u = rr - ch * V;
            const bool ok = r < m && jj < e;
            cp_async4(wres + (size_t)tile * C::TILE_FLOATS + ch * C::WCH + u * EP + jj,
                      ok ? (const void *)(wg + (int64_t)r * e + jj) : (const void *)wg, ok);
        }
    }
    cp_async_commit();   // the oldest group: waited for below, after the x prologue
    // this CTA's contiguous range of groups, warp w takes lo + w, lo + w + nw, ...
    const int64_t groups = (s + T - 1) / T;
    const int64_t lo = groups * blockIdx.x / gridDim.x, hi = groups * (blockIdx.x + 1) / gridDim.x;
    const int64_t my_groups = lo + warp < hi ? (hi - lo - warp + nw - 1) / nw : 0;
    const int64_t total = my_groups * ntiles;   // (group, tile) steps of this warp, flattened
    const int64_t gstride_t = (int64_t)nw * T;  // tokens between this warp's groups
    // this lane's x chunks of one step: its chunk of tile `it`, every token of
    // the group starting at token t0, into ring slot `slot`
    auto issue = [&](int64_t t0, int it, int slot_i) {
        const int ch = it * 32 + lane;
        unsigned char *slot = ring + slot_i * (T * 32 * 16);
#pragma unroll
        for (int tt = 0; tt < T; tt++) {
            const bool ok = t0 + tt < s && ch < nch;
            cp_async16(slot + (tt * 32 + lane) * 16,
                       ok ? (const void *)(x + (t0 + tt) * m + (int64_t)ch * V) : (const void *)x, ok);
        }
        cp_async_commit();
    };
    // the step being issued (RD - 1 ahead of the one computed): token, tile, slot
    int64_t it0 = (lo + warp) * T;
    int itile = 0, islot = 0;
    auto issue_next = [&]() {
        issue(it0, itile, islot);
        islot = islot + 1 == RD ? 0 : islot + 1;
        if (++itile == ntiles) {
            itile = 0;
            it0 += gstride_t;
        }
    };
#pragma unroll
    for (int p = 0; p < RD - 1; p++) {
        if (p < total) issue_next();
        else cp_async_commit();
    }
    cp_async_wait<RD - 1>();   // the weight (this thread's copies) ...
    __syncthreads();           // ... and every thread's
    float2 acc[T][EP / 2];
    int tile = 0, slot_q = 0;
    int64_t t0 = (lo + warp) * T;   // the computed step's group
    for (int64_t q = 0; q < total; q++) {
        if (q + RD - 1 < total) issue_next();
        else cp_async_commit();
        cp_async_wait<RD - 1>();   // this lane's copies of step q have landed
        if (tile == 0) {
#pragma unroll
            for (int tt = 0; tt < T; tt++)
#pragma unroll
                for (int i = 0; i < EP / 2; i++) acc[tt][i] = make_float2(0.0f, 0.0f);
        }
        if (tile * 32 + lane < nch) {   // this lane's chunk of the tile holds features
            const unsigned char *slot = ring + slot_q * (T * 32 * 16);
            V16 cur[T];
#pragma unroll
            for (int tt = 0; tt < T; tt++)
                cur[tt] = *reinterpret_cast<const V16 *>(slot + (tt * 32 + lane) * 16);
            lane_fma2_chunk<XT, EP, T, 0, V>(acc, cur,
                                             wres + (size_t)tile * C::TILE_FLOATS + lane * C::WCH);
        }
        slot_q = slot_q + 1 == RD ? 0 : slot_q + 1;
        if (++tile != ntiles) continue;
        tile = 0;
        // reduce-scatter over the lanes: lane l ends with flattened values 2l, 2l+1
        float v[64];
#pragma unroll
        for (int tt = 0; tt < T; tt++)
#pragma unroll
            for (int i = 0; i < EP / 2; i++) {
                v[tt * EP + 2 * i] = acc[tt][i].x;
                v[tt * EP + 2 * i + 1] = acc[tt][i].y;
            }
        rs_step<64, 16>(v, lane);
        rs_step<32, 8>(v, lane);
        rs_step<16, 4>(v, lane);
        rs_step<8, 2>(v, lane);
        rs_step<4, 1>(v, lane);
        const int j0 = (2 * lane) % EP;
        float a = v[0], b = v[1];
        if (bias) {   // one fp32 add after the chain
            if (j0 < e) a = a + bias[j0];
            if (j0 + 1 < e) b = b + bias[j0 + 1];
        }
        segment_topk<EP / 2>(a, b, j0, e, k, normalize, t0 + (2 * lane) / EP, s, idx, gates, lane);
        t0 += gstride_t;
    }
    cp_async_wait<0>();
}

template <int EP, typename XT>
moe_status launch_lane(const void *x, const float *wg, const float *bias, int64_t s, int m, int e,
                       int k, int normalize, int32_t *idx, float *gates, int32_t *st,
                       cudaStream_t stream) {
    // the gate weight resident in shared memory when it fits
    {
        using R = ResCfg<EP, XT>;
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (sms < 1) sms = 1;
        const int64_t groups = (s + R::T - 1) / R::T;
        // warps per CTA: enough to spread the groups over every SM, at most RW_MAX
        int64_t nw = (groups + sms - 1) / sms;
        nw = nw < 1 ? 1 : (nw > res_warps_max<EP>() ? res_warps_max<EP>() : nw);
        // fewer warps when their rings would not fit beside the weight
        while (nw > 4 && R::smem(m, (int)nw) > RES_SMEM_MAX) nw--;
        const size_t res_smem = R::smem(m, (int)nw);
        if (res_smem <= RES_SMEM_MAX) {
            auto kern = gate_lane_res_kernel<EP, XT>;
            static int smem_set[64] = {0};
            if (dev >= 0 && dev < 64 && !smem_set[dev]) {
                if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)RES_SMEM_MAX) != cudaSuccess)
                    return MOE_ERR_CUDA;
                smem_set[dev] = 1;
            }
            const int64_t want = (groups + nw - 1) / nw;
            const int64_t grid = want < sms ? want : sms;
            return launch_pdl(kern, dim3((unsigned)grid), dim3((unsigned)(nw * 32)), res_smem, stream,
                              (const XT *)x, wg, bias, s, m, e, k, normalize, idx, gates, st);
        }
    }
    using C = LaneCfg<EP, XT>;
    auto kern = gate_lane_kernel<EP, XT>;
    if (C::SMEM > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    const int64_t grid = (s + C::TC - 1) / C::TC;
    if (grid > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(LNW * 32), C::SMEM, stream, (const XT *)x, wg,
                      bias, s, m, e, k, normalize, idx, gates, st);
}

template <class C, typename XT>
moe_status launch_seq(const void *x, const float *wg, const float *bias, int64_t s, int m, int e,
                      int k, int normalize, int32_t *idx, float *gates, int32_t *st,
                      cudaStream_t stream) {
    auto kern = gate_seq_kernel<C, XT>;
    static int slots[64] = {0};   // resident CTAs per device (persistent grid)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    int nslot = dev >= 0 && dev < 64 ? slots[dev] : 0;
    if (!nslot) {
        if (C::SMEM > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
                cudaSuccess)
            return MOE_ERR_CUDA;
        int per_sm = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::NT, C::SMEM) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        nslot = (per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
        if (dev >= 0 && dev < 64) slots[dev] = nslot;
    }
    const int64_t nchunks = (s + C::TOKC - 1) / C::TOKC;
    const int64_t grid = nchunks < nslot ? nchunks : nslot;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(C::NT), C::SMEM, stream, (const XT *)x, wg,
                      bias, s, m, e, k, normalize, idx, gates, st);
}

template <typename XT>
moe_status gate_dispatch(const void *x, const float *wg, const float *bias, int64_t s, int m, int e,
                         int k, int normalize, int32_t *idx, float *gates, int32_t *st,
                         cudaStream_t stream) {
#define MOE_GATE_CASE(EPV, EWV, TTV, NWV, KTV, STV)                                          \
    if (e <= EPV)                                                                           \
        return launch_seq<SeqCfg<EPV, EWV, TTV, NWV, KTV, STV, XT>, XT>(                    \
            x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    // e <= 32: lane-blocked order, all experts of a token in one warp
    if (e <= 4) return launch_lane<4, XT>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    if (e <= 8) return launch_lane<8, XT>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    if (e <= 16) return launch_lane<16, XT>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    if (e <= 32) return launch_lane<32, XT>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    // e > 32: fp32-FMA bound, sequential order; experts per warp x tokens per lane
    MOE_GATE_CASE(64, 16, 2, 4, 64, 3)
    MOE_GATE_CASE(128, 16, 2, 8, 64, 3)
    MOE_GATE_CASE(256, 32, 4, 8, 32, 2)
#undef MOE_GATE_CASE
    return MOE_ERR_UNSUPPORTED;
}

}  // namespace

moe_status gate_topk_launch(const void *x, moe_dtype xdt, const float *wg, const float *bias,
                            int64_t s, int m, int e, int k, unsigned flags, int32_t *idx,
                            float *gates, int32_t *st, cudaStream_t stream) {
    int normalize = (flags & MOE_FLAG_NORMALIZE_GATES) ? 1 : 0;
    if (xdt == MOE_BF16)
        return gate_dispatch<__nv_bfloat16>(x, wg, bias, s, m, e, k, normalize, idx, gates, st,
                                            stream);
    return gate_dispatch<float>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
}

}  // namespace moe
