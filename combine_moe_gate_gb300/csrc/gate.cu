// Fused gate: fp32 logits -> softmax -> top-k, one CTA per tile of tokens.
//
// Method: the Tutel profile's gate_type {'type': 'top', 'k': k} (top-k softmax
// gate) and the DeepSpeed-MoE vs Tutel blog, section 1.4 (top-k fused into one
// kernel that emits a dense token-to-expert table instead of a one-hot mask).
//
// Logit order (fixed so routing is reproducible bit for bit): each logit has a
// single fp32 accumulator starting at +0, updated with a fused multiply-add in
// ascending feature index; the bias is then added once in fp32.  The kernel is
// a register-blocked SIMT GEMM: every thread owns TT tokens x TE experts, and
// each of its accumulators walks the features in ascending order, which is
// exactly that contract.  Tensor cores are not used: their internal
// accumulation order is unspecified and would make routing irreproducible.
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

    if constexpr (C::EP <= 32) {
        // softmax + top-k, one thread per token: the token's <= 32 logits are read
        // from the tile; selection scans experts in ascending index with a strict
        // comparison, so equal logits go to the lower index.
        for (int tl = tid; tl < C::TOKC; tl += C::NT) {
            const int64_t t = t0 + tl;
            if (t >= s) break;
            float v[C::EP];
            float mx = -INFINITY;
#pragma unroll
            for (int q = 0; q < C::EP; q++) {
                v[q] = q < e ? lg[tl * C::LGS + q] : -INFINITY;
                mx = fmaxf(mx, v[q]);
            }
            float z = 0.0f;
#pragma unroll
            for (int q = 0; q < C::EP; q++)
                if (q < e) z += expf(v[q] - mx);
            unsigned taken = 0;
            float psel = 0.0f;
            float pr[C::EP];
#pragma unroll
            for (int r = 0; r < C::EP; r++) {
                if (r >= k) break;
                float bv = -INFINITY;
                int bj = 0;
                bool found = false;
#pragma unroll
                for (int q = 0; q < C::EP; q++) {
                    bool cand = q < e && !((taken >> q) & 1u);
                    if (cand && (!found || v[q] > bv)) { bv = v[q]; bj = q; found = true; }
                }
                taken |= 1u << bj;
                pr[r] = expf(bv - mx);
                psel += pr[r];
                idx[(int64_t)r * s + t] = bj;
            }
            const float den = normalize ? psel : z;
#pragma unroll
            for (int r = 0; r < C::EP; r++) {
                if (r >= k) break;
                gates[(int64_t)r * s + t] = pr[r] / den;
            }
        }
        return;
    } else {
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
// One thread per (token, expert) for e <= 32: the logit's single accumulator
// walks the features in ascending order (the contract above) with no blocking,
// so the batch runs as s*e independent chains.  The gate weight [m][e] is copied
// whole into shared memory (the e threads of a token read consecutive words);
// x reaches shared memory through a SK-deep cp.async ring of tiles of the CTA's
// TPB tokens, so that a whole ring of x (not just a few registers per thread) is
// in flight against HBM latency; the threads of a token read its features with
// broadcast loads.  Softmax and top-k run on the EP lanes of each token with
// segmented shuffles.  (KS below: features per tile, 512 bytes of each row.)
constexpr int SK = 4;    // x tiles in flight

template <int EP, typename XT>
struct SmallCfg {
    static constexpr int KS = 512 / (int)sizeof(XT);             // features per x tile (512 B rows)
    static constexpr int TPB = (256 / 32) * (32 / EP);           // tokens per CTA
    static constexpr int XROWB = 512 + 16;                       // padded x tile row (bytes)
    static constexpr int XBYTES = SK * TPB * XROWB;              // x ring
    static_assert(XBYTES <= 140 * 1024, "x ring");
};

template <int EP, typename XT>
__global__ void __launch_bounds__(256)
gate_small_kernel(const XT *__restrict__ x, const float *__restrict__ wg,
                  const float *__restrict__ bias, int64_t s, int m, int e, int k, int normalize,
                  int32_t *__restrict__ idx, float *__restrict__ gates, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    using SC = SmallCfg<EP, XT>;
    constexpr int VEC = Elt<XT>::VEC, KS = SC::KS;
    constexpr int CPR = KS / VEC;   // 16-byte chunks per token row per tile
    extern __shared__ __align__(16) unsigned char smem_small[];
    unsigned char *xs = smem_small;                          // [SK][TPB][XROWB]
    float *wt = reinterpret_cast<float *>(smem_small + SC::XBYTES);  // [m][e]
    const int64_t t0 = (int64_t)blockIdx.x * SC::TPB;
    const int ntiles = (m + KS - 1) / KS;
    auto load_x = [&](int tile) {
        unsigned char *dst = xs + (tile % SK) * SC::TPB * SC::XROWB;
        for (int q = threadIdx.x; q < SC::TPB * CPR; q += 256) {
            const int row = q / CPR, ch = q % CPR;
            const int64_t t = t0 + row;
            const int f = tile * KS + ch * VEC;
            const bool ok = t < s && f < m;
            cp_async16(dst + row * SC::XROWB + ch * 16, ok ? (const void *)(x + t * m + f) : (const void *)x,
                       ok);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int p = 0; p < SK - 1; p++) {
        if (p < ntiles) load_x(p);
        else cp_async_commit();
    }
    {   // the gate weight, [m][e] as in global memory, copied in one go
        const int total = m * e;
        if ((e & 3) == 0) {
            for (int q = threadIdx.x * 4; q < total; q += 256 * 4)
                cp_async16(wt + q, wg + q, true);
        } else {
            for (int q = threadIdx.x; q < total; q += 256) cp_async4(wt + q, wg + q, true);
        }
        cp_async_commit();
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int TPW = 32 / EP;
    const int j = lane % EP;
    const int tl = warp * TPW + lane / EP;       // token within the CTA
    const int64_t t = t0 + tl;
    const bool live = t < s;
    const float *wr = wt + (j < e ? j : 0);
    float acc = 0.0f;
    for (int it = 0; it < ntiles; it++) {
        if (it == 0) cp_async_wait<0>();   // the weight (committed after the x prologue) and tile 0
        else cp_async_wait<SK - 2>();
        __syncthreads();   // tile `it` landed (and the weight staged); tile it-1 fully read
        if (it + SK - 1 < ntiles) load_x(it + SK - 1);
        else cp_async_commit();
        const unsigned char *xr = xs + (it % SK) * SC::TPB * SC::XROWB + tl * SC::XROWB;
        const int nfeat = min(KS, m - it * KS);
        const float *w = wr + (int64_t)it * KS * e;
        for (int c = 0; c < nfeat / VEC; c++) {
            float f[VEC];
            Elt<XT>::unpack(*reinterpret_cast<const V16 *>(xr + c * 16), f);
#pragma unroll
            for (int u = 0; u < VEC; u++) acc = fmaf(f[u], w[(c * VEC + u) * e], acc);
        }
    }
    cp_async_wait<0>();
    float v = -INFINITY;
    if (j < e) v = bias ? acc + bias[j] : acc;
    // segmented (EP lanes per token) softmax statistics
    float mx = v;
#pragma unroll
    for (int o = EP / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float z = j < e ? expf(v - mx) : 0.0f;
#pragma unroll
    for (int o = EP / 2; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    // top-k: k rounds of segmented arg-max (ties -> lower expert index)
    bool taken = j >= e;
    float my_v = 0.0f;
    int my_j = 0;
    for (int r = 0; r < k; r++) {
        float bv = taken ? -INFINITY : v;
        int bj = taken ? 0x7fffffff : j;
#pragma unroll
        for (int o = EP / 2; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
            if (ov > bv || (ov == bv && oj < bj)) { bv = ov; bj = oj; }
        }
        if (bj == j) taken = true;
        if (j == r) { my_v = bv; my_j = bj; }
    }
    const float p = j < k ? expf(my_v - mx) : 0.0f;
    float sel = p;
#pragma unroll
    for (int o = EP / 2; o > 0; o >>= 1) sel += __shfl_xor_sync(0xffffffffu, sel, o);
    if (live && j < k) {
        idx[(int64_t)j * s + t] = my_j;
        gates[(int64_t)j * s + t] = p / (normalize ? sel : z);
    }
}

template <int EP, typename XT>
moe_status launch_small(const void *x, const float *wg, const float *bias, int64_t s, int m, int e,
                        int k, int normalize, int32_t *idx, float *gates, int32_t *st,
                        cudaStream_t stream) {
    auto kern = gate_small_kernel<EP, XT>;
    const size_t smem = SmallCfg<EP, XT>::XBYTES + (size_t)m * e * sizeof(float);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    constexpr int TPB = SmallCfg<EP, XT>::TPB;
    const int64_t grid = (s + TPB - 1) / TPB;
    if (grid > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(256), smem, stream, (const XT *)x, wg, bias, s,
                      m, e, k, normalize, idx, gates, st);
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

// Shared memory the small-e kernel may use for the transposed gate weight.
constexpr size_t SMALL_E_SMEM_MAX = 64 * 1024;

template <typename XT>
moe_status gate_dispatch(const void *x, const float *wg, const float *bias, int64_t s, int m, int e,
                         int k, int normalize, int32_t *idx, float *gates, int32_t *st,
                         cudaStream_t stream) {
#define MOE_GATE_CASE(EPV, TEV, TTV, NTV, KTV, STV)                                        \
    if (e <= EPV)                                                                           \
        return launch_cfg<GateCfg<EPV, TEV, TTV, NTV, KTV, STV, XT>, XT>(                   \
            x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    // small e whose transposed weight fits in shared memory: one chain per thread
#define MOE_GATE_SMALL(EPV)                                                                  \
    if (e <= EPV && (size_t)m * e * sizeof(float) <= SMALL_E_SMEM_MAX)                       \
        return launch_small<EPV, XT>(x, wg, bias, s, m, e, k, normalize, idx, gates, st, stream);
    MOE_GATE_SMALL(4)
    MOE_GATE_SMALL(8)
    MOE_GATE_SMALL(16)
    MOE_GATE_SMALL(32)
#undef MOE_GATE_SMALL
    // otherwise: HBM/latency bound -> few tokens per CTA, long tiles, deep pipeline;
    // large e: fp32-FMA bound -> register-blocked 8x8 micro-tiles
    MOE_GATE_CASE(4, 4, 1, 64, 128, 4)
    MOE_GATE_CASE(8, 4, 1, 64, 128, 4)
    MOE_GATE_CASE(16, 4, 1, 128, 128, 3)
    MOE_GATE_CASE(32, 8, 1, 128, 64, 4)
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
