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
//     gate_topk_kernel is a register-blocked SIMT GEMM: every thread owns TT
//     tokens x TE experts, and each accumulator walks the features in order.
//     (The lane-blocked order needs 32 live partial sums per logit; with all e
//     experts of a token in one CTA, as the fused top-k needs, that leaves a
//     CTA only a handful of tokens for large e.)
// Tensor cores are not used: their internal accumulation order is unspecified
// and would make routing irreproducible.
#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem, bool valid) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    int n = valid ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// N consecutive floats from shared memory; 16-byte loads when N % 4 == 0
// (callers pass 16-byte aligned addresses in that case).
template <int N>
__device__ __forceinline__ void lds_vec(float *dst, const float *src) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N / 4; i++) {
            float4 v = reinterpret_cast<const float4 *>(src)[i];
            dst[4 * i] = v.x; dst[4 * i + 1] = v.y; dst[4 * i + 2] = v.z; dst[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; i++) dst[i] = src[i];
    }
}

template <int EP_, int TE_, int TT_, int NT_, int KT_, int ST_, typename XT>
struct GateCfg {
    static constexpr int KT = KT_;               // features per shared-memory tile
    static constexpr int STAGES = ST_;           // cp.async pipeline depth
    static constexpr int EP = EP_;               // experts per CTA (e padded)
    static constexpr int TE = TE_;               // experts per thread
    static constexpr int TT = TT_;               // tokens per thread
    static constexpr int NT = NT_;               // threads per CTA
    static constexpr int EX = EP / TE;           // threads along experts
    static constexpr int TY = NT / EX;           // threads along tokens
    static constexpr int TOKC = TY * TT;         // tokens per CTA
    static constexpr int VEC = Elt<XT>::VEC;     // x elements per 16-byte chunk
    static constexpr int XCH = KT / VEC;         // 16-byte chunks per token row per tile
    static constexpr int XROW = KT * Elt<XT>::BYTES + 16;  // padded raw row (bytes)
    static constexpr int XFS = TOKC + 4;         // fp32 x tile row stride (floats)
    static constexpr int LGS = EP + 1;           // logits tile row stride
    // shared memory (bytes): raw x ring, fp32 x tile, Wg ring
    static constexpr int RAW_BYTES = STAGES * TOKC * XROW;
    static constexpr int XF_BYTES = KT * XFS * 4;
    static constexpr int WS_BYTES = STAGES * KT * EP * 4;
    static constexpr int MAIN_BYTES = RAW_BYTES + XF_BYTES + WS_BYTES;
    static constexpr int LG_BYTES = TOKC * LGS * 4;
    static constexpr int SMEM = MAIN_BYTES > LG_BYTES ? MAIN_BYTES : LG_BYTES;
    static_assert(EP % TE == 0 && NT % EX == 0 && TE % 4 == 0 && STAGES >= 2, "layout");
    static_assert(EP > 32, "e <= 32 uses the lane-blocked kernel (its logit order)");
};

template <class C, typename XT>
__device__ __forceinline__ void load_tile(unsigned char *raw, float *ws, const XT *x, const float *wg,
                                          int64_t s, int m, int e, int64_t t0, int k0, bool wg16) {
    const int tid = threadIdx.x;
    // x: TOKC rows x XCH chunks of 16 bytes
    for (int q = tid; q < C::TOKC * C::XCH; q += C::NT) {
        int row = q / C::XCH, ch = q % C::XCH;
        int64_t t = t0 + row;
        int f = k0 + ch * C::VEC;
        bool ok = t < s && f < m;
        const XT *src = ok ? x + t * m + f : x;
        cp_async16(raw + row * C::XROW + ch * 16, src, ok);
    }
    // Wg: KT rows x EP columns (zero beyond m rows / e columns)
    constexpr int KT = C::KT;
    if (wg16) {
        for (int q = tid; q < KT * (C::EP / 4); q += C::NT) {
            int kk = q / (C::EP / 4), j = (q % (C::EP / 4)) * 4;
            bool ok = k0 + kk < m && j < e;
            const float *src = ok ? wg + (int64_t)(k0 + kk) * e + j : wg;
            cp_async16(ws + kk * C::EP + j, src, ok);
        }
    } else {
        for (int q = tid; q < KT * C::EP; q += C::NT) {
            int kk = q / C::EP, j = q % C::EP;
            bool ok = k0 + kk < m && j < e;
            const float *src = ok ? wg + (int64_t)(k0 + kk) * e + j : wg;
            cp_async4(ws + kk * C::EP + j, src, ok);
        }
    }
    cp_async_commit();
}

template <class C, typename XT>
__global__ void __launch_bounds__(C::NT)
gate_topk_kernel(const XT *__restrict__ x, const float *__restrict__ wg,
                 const float *__restrict__ bias, int64_t s, int m, int e, int k, int normalize,
                 int32_t *__restrict__ idx, float *__restrict__ gates, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char *raw = smem;                                   // [STAGES][TOKC][XROW]
    float *xf = (float *)(smem + C::RAW_BYTES);                  // [KT][XFS]
    float *ws = (float *)(smem + C::RAW_BYTES + C::XF_BYTES);    // [STAGES][KT][EP]

    const int tid = threadIdx.x;
    const int tx = tid % C::EX, ty = tid / C::EX;
    const int64_t t0 = (int64_t)blockIdx.x * C::TOKC;
    const bool wg16 = (e % 4) == 0;  // rows of wg start on 16-byte boundaries

    float acc[C::TT][C::TE];
#pragma unroll
    for (int j = 0; j < C::TT; j++)
#pragma unroll
        for (int i = 0; i < C::TE; i++) acc[j][i] = 0.0f;

    constexpr int KT = C::KT, ST = C::STAGES;
    const int ntiles = (m + KT - 1) / KT;
    // prologue: tiles 0 .. ST-2 in flight (one commit group per tile, empty groups past the end)
#pragma unroll
    for (int p = 0; p < ST - 1; p++) {
        if (p < ntiles)
            load_tile<C, XT>(raw + p * C::TOKC * C::XROW, ws + p * KT * C::EP, x, wg, s, m, e, t0,
                             p * KT, wg16);
        else
            cp_async_commit();
    }
    for (int it = 0; it < ntiles; it++) {
        const int cur = it % ST;
        cp_async_wait<ST - 2>();
        __syncthreads();  // tile `it` landed; everyone finished reading tile it-1 and xf
        {
            const int nx = it + ST - 1, nb = nx % ST;
            if (nx < ntiles)
                load_tile<C, XT>(raw + nb * C::TOKC * C::XROW, ws + nb * KT * C::EP, x, wg, s, m, e,
                                 t0, nx * KT, wg16);
            else
                cp_async_commit();
        }
        // widen the raw x tile to fp32, transposed to [feature][token]
        const unsigned char *rc = raw + cur * C::TOKC * C::XROW;
        for (int q = tid; q < C::TOKC * C::XCH; q += C::NT) {
            int row = q % C::TOKC, ch = q / C::TOKC;
            V16 v = *(const V16 *)(rc + row * C::XROW + ch * 16);
            float f[C::VEC];
            Elt<XT>::unpack(v, f);
#pragma unroll
            for (int u = 0; u < C::VEC; u++) xf[(ch * C::VEC + u) * C::XFS + row] = f[u];
        }
        __syncthreads();
        const float *wc = ws + cur * KT * C::EP;
        const int klim = min(KT, m - it * KT);
        if (klim == KT) {
#pragma unroll 4
            for (int kk = 0; kk < KT; kk++) {
                float xv[C::TT], wv[C::TE];
                lds_vec<C::TT>(xv, xf + kk * C::XFS + ty * C::TT);
                lds_vec<C::TE>(wv, wc + kk * C::EP + tx * C::TE);
#pragma unroll
                for (int j = 0; j < C::TT; j++)
#pragma unroll
                    for (int i = 0; i < C::TE; i++) acc[j][i] = fmaf(xv[j], wv[i], acc[j][i]);
            }
        } else {
            for (int kk = 0; kk < klim; kk++) {
                float xv[C::TT], wv[C::TE];
                lds_vec<C::TT>(xv, xf + kk * C::XFS + ty * C::TT);
                lds_vec<C::TE>(wv, wc + kk * C::EP + tx * C::TE);
#pragma unroll
                for (int j = 0; j < C::TT; j++)
#pragma unroll
                    for (int i = 0; i < C::TE; i++) acc[j][i] = fmaf(xv[j], wv[i], acc[j][i]);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // all reads of the tiles done before the logits overwrite them

    float *lg = (float *)smem;  // [TOKC][LGS]
#pragma unroll
    for (int j = 0; j < C::TT; j++)
#pragma unroll
        for (int i = 0; i < C::TE; i++) {
            int ex = tx * C::TE + i;
            float v = acc[j][i];
            if (bias && ex < e) v = v + bias[ex];
            lg[(ty * C::TT + j) * C::LGS + ex] = v;
        }
    __syncthreads();

    {
        // softmax + top-k: one warp per token
        constexpr int NW = C::NT / 32;
        constexpr int QE = (C::EP + 31) / 32;  // experts per lane
        const int lane = tid & 31, warp = tid >> 5;
        for (int tl = warp; tl < C::TOKC; tl += NW) {
            const int64_t t = t0 + tl;
            if (t >= s) break;
            float v[QE];
            float mx = -INFINITY;
#pragma unroll
            for (int q = 0; q < QE; q++) {
                int ex = lane + 32 * q;
                v[q] = ex < e ? lg[tl * C::LGS + ex] : -INFINITY;
                mx = fmaxf(mx, v[q]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float z = 0.0f;
#pragma unroll
            for (int q = 0; q < QE; q++)
                if (lane + 32 * q < e) z += expf(v[q] - mx);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);

            unsigned taken = 0;  // bit q: expert lane+32q already selected
            float my_v = 0.0f;   // lane r keeps route r's logit and expert
            int my_j = 0;
            for (int r = 0; r < k; r++) {
                float bv = -INFINITY;
                int bj = 0x7fffffff;
#pragma unroll
                for (int q = 0; q < QE; q++) {
                    int ex = lane + 32 * q;
                    bool cand = ex < e && !((taken >> q) & 1u);
                    if (cand && (v[q] > bv || (v[q] == bv && ex < bj))) { bv = v[q]; bj = ex; }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    int oj = __shfl_xor_sync(0xffffffffu, bj, o);
                    if (ov > bv || (ov == bv && oj < bj)) { bv = ov; bj = oj; }
                }
                if ((bj & 31) == lane) taken |= 1u << (bj >> 5);
                if (lane == r) { my_v = bv; my_j = bj; }
            }
            float p = lane < k ? expf(my_v - mx) : 0.0f;
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
    }
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

// Feature u (compile-time) of a 16-byte chunk, widened exactly to fp32.
template <typename XT, int U>
__device__ __forceinline__ float chunk_elem(const V16 &v) {
    if constexpr (sizeof(XT) == 2)
        return (U & 1) ? bf16hi(v.w[U >> 1]) : bf16lo(v.w[U >> 1]);
    else
        return __uint_as_float(v.w[U]);
}

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

template <int EP, typename XT>
moe_status launch_lane(const void *x, const float *wg, const float *bias, int64_t s, int m, int e,
                       int k, int normalize, int32_t *idx, float *gates, int32_t *st,
                       cudaStream_t stream) {
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
moe_status launch_cfg(const void *x, const float *wg, const float *bias, int64_t s, int m, int e,
                      int k, int normalize, int32_t *idx, float *gates, int32_t *st,
                      cudaStream_t stream) {
    auto kern = gate_topk_kernel<C, XT>;
    if (C::SMEM > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
    }
    int64_t grid = (s + C::TOKC - 1) / C::TOKC;
    if (grid > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(C::NT), C::SMEM, stream, (const XT *)x, wg,
                      bias, s, m, e, k, normalize, idx, gates, st);
}

template <typename XT>
moe_status gate_dispatch(const void *x, const float *wg, const float *bias, int64_t s, int m, int e,
                         int k, int normalize, int32_t *idx, float *gates, int32_t *st,
                         cudaStream_t stream) {
#define MOE_GATE_CASE(EPV, TEV, TTV, NTV, KTV, STV)                                        \
    if (e <= EPV)                                                                           \
        return launch_cfg<GateCfg<EPV, TEV, TTV, NTV, KTV, STV, XT>, XT>(                   \
            x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    // e <= 32: lane-blocked order, all experts of a token in one warp
    if (e <= 4) return launch_lane<4, XT>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    if (e <= 8) return launch_lane<8, XT>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    if (e <= 16) return launch_lane<16, XT>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    if (e <= 32) return launch_lane<32, XT>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    // e > 32: fp32-FMA bound -> register-blocked 8x8 micro-tiles, sequential order
    MOE_GATE_CASE(64, 8, 8, 128, 32, 3)
    MOE_GATE_CASE(128, 8, 8, 256, 32, 2)
    MOE_GATE_CASE(256, 8, 8, 256, 32, 2)
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
