// SIMT helper kernels of the expert-FFN backward: zero-padded transposes (so
// that every product runs on the forward's K-major grouped GEMM), the
// activation derivative, and bias-gradient column sums.
//
// Method: the Tutel profile's experts {'type': 'ffn', hidden_size_per_expert,
// has_fc1_bias, has_fc2_bias}, differentiated: with pre = x w1^T + b1 and
// hid = act(pre), d_pre = (d_out w2) * act'(pre); SwiGLU (hid = silu(a) b)
// splits it into d_a = d_hid b silu'(a) and d_b = d_hid silu(a).
#include "ffn_bwd.cuh"

namespace moe {
namespace {

// ------------------------------------------------------------- transposes
// A CTA moves a 64 x 64 tile: 16-byte loads of source rows into shared
// memory, then each thread gathers 8 elements of a source column and stores
// them as one 16-byte piece of a destination row.  Row lengths, pitches and
// offsets are multiples of 8 elements (16 bytes).  In shared memory the
// 16-byte chunks of tile row r are permuted by chunk ^ ((r / 8) % 8), so the
// column gathers of eight lanes, from rows 8 apart, fall in eight different
// banks.
constexpr int TP = 64, TP_THREADS = 256;
constexpr int PAD_TO = 64;         // K block of the weight-gradient GEMMs
constexpr int TP_GRID_X = 16;      // CTAs per (column block, batch) striding over row blocks

__device__ __forceinline__ int tp_col(int r, int c) {   // shared column of tile element (r, c)
    return ((((c >> 3) ^ (r >> 3)) & 7) << 3) | (c & 7);
}

__global__ void __launch_bounds__(TP_THREADS)
transpose_pad_kernel(const uint16_t *__restrict__ src, int64_t src_batch, int64_t src_pitch,
                     uint16_t *__restrict__ dst, int64_t dst_batch, int64_t dst_pitch, int rows,
                     int cols, int dst_cols, const int32_t *__restrict__ counts,
                     const int32_t *__restrict__ skip, const int32_t *__restrict__ c_dev,
                     int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    __shared__ __align__(16) uint16_t tile[TP][TP];
    const int b = blockIdx.z;
    if (skip && min(skip[b], *c_dev) <= 0) return;   // block-uniform
    const int c0 = blockIdx.y * TP;
    int kept = rows;
    if (counts) kept = max(0, min(min(counts[b], *c_dev), rows));
    // zeros are written up to the next multiple of PAD_TO past the kept rows
    // (the consumer reads no further); the CTAs of a batch stride over the row
    // blocks up to there (the grid is sized for c_max rows, most of which are
    // usually not kept)
    const int pad_end = counts ? min(dst_cols, (kept + PAD_TO - 1) / PAD_TO * PAD_TO) : dst_cols;
    const uint16_t *sb = src + (int64_t)b * src_batch;
    uint16_t *db = dst + (int64_t)b * dst_batch;
    for (int r0 = blockIdx.x * TP; r0 < pad_end; r0 += gridDim.x * TP) {
        __syncthreads();   // the previous block's gathers are done with the tile
        for (int i = threadIdx.x; i < TP * (TP / 8); i += TP_THREADS) {
            const int r = i >> 3, c = (i & 7) * 8;
            V16 v;
            v.w[0] = v.w[1] = v.w[2] = v.w[3] = 0u;
            if (r0 + r < kept && c0 + c < cols) v = ld_stream(sb + (int64_t)(r0 + r) * src_pitch + c0 + c);
            *reinterpret_cast<V16 *>(&tile[r][tp_col(r, c)]) = v;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < TP * (TP / 8); i += TP_THREADS) {
            const int c = i >> 3, r = (i & 7) * 8;   // destination row c0 + c, columns r0 + r ..
            if (c0 + c >= cols || r0 + r >= pad_end) continue;
            V16 v;
#pragma unroll
            for (int u = 0; u < 4; u++)
                v.w[u] = (uint32_t)tile[r + 2 * u][tp_col(r + 2 * u, c)] |
                         ((uint32_t)tile[r + 2 * u + 1][tp_col(r + 2 * u + 1, c)] << 16);
            st_v16(db + (int64_t)(c0 + c) * dst_pitch + r0 + r, v);
        }
    }
}

// ---------------------------------------------------- activation backward
constexpr int AB_THREADS = 256;
constexpr int AB_ROWS = 16;   // rows of one expert per CTA
constexpr int AB_U = 4;       // 16-byte chunks per thread in flight together
constexpr int AB_GRID_X = 32; // CTAs per expert

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float exp2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Two floats to packed bf16 (nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&r);
}

// GELU'(z) = Phi(z) + z phi(z), Phi(z) = 0.5 (1 + erf(z / sqrt 2)), phi the
// normal density.  Phi as in the forward GELU: erfc(x) = (1 + a1 x + ... +
// a6 x^6)^-16 for x = |z| / sqrt 2 (Abramowitz & Stegun, Handbook of
// Mathematical Functions, 7.1.28, |error| <= 3e-7), Phi = 1 - erfc / 2 for
// z >= 0 and erfc / 2 below, so the negative tail does not cancel; phi(z) =
// 2^(-z^2 log2(e) / 2) / sqrt(2 pi).  Approximate reciprocal and power of two
// (relative error ~2^-22), far below the bf16 rounding that follows.
__device__ __forceinline__ float gelu_grad(float z) {
    const float x = fabsf(z) * 0.70710678118654752f;
    float p = fmaf(x, 0.0000430638f, 0.0002765672f);
    p = fmaf(x, p, 0.0001520143f);
    p = fmaf(x, p, 0.0092705272f);
    p = fmaf(x, p, 0.0422820123f);
    p = fmaf(x, p, 0.0705230784f);
    p = fmaf(x, p, 1.0f);
    p = p * p;
    p = p * p;
    p = p * p;
    p = p * p;   // overflows to inf for large x, where erfc -> 0
    const float half_erfc = 0.5f * rcp_approx(p);
    const float cdf = z >= 0.0f ? 1.0f - half_erfc : half_erfc;
    // -log2(e) / 2 and 1 / sqrt(2 pi)
    const float dens = exp2_approx((z * z) * -0.72134752044448170f);
    return fmaf(z * 0.3989422804014327f, dens, cdf);
}

template <int ACT>
__device__ __forceinline__ void act_bwd_chunk(const V16 &pa, const V16 &pb, const V16 &dh,
                                              __nv_bfloat16 *dst, int h) {
    float a[8], g[8], o[8];
    Elt<__nv_bfloat16>::unpack(pa, a);
    Elt<__nv_bfloat16>::unpack(dh, g);
    if constexpr (ACT == MOE_ACT_SWIGLU) {
        float b[8], ob[8];
        Elt<__nv_bfloat16>::unpack(pb, b);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float sg = 1.0f / (1.0f + expf(-a[i]));
            o[i] = g[i] * b[i] * sg * (1.0f + a[i] * (1.0f - sg));   // d_a
            ob[i] = g[i] * a[i] * sg;                                // d_b
        }
        st_v16(dst, Elt<__nv_bfloat16>::pack(o));
        st_v16(dst + h, Elt<__nv_bfloat16>::pack(ob));
    } else {
#pragma unroll
        for (int i = 0; i < 8; i++)
            o[i] = g[i] * (ACT == MOE_ACT_RELU ? (a[i] > 0.0f ? 1.0f : 0.0f) : gelu_grad(a[i]));
        V16 v;
#pragma unroll
        for (int i = 0; i < 4; i++) v.w[i] = pack2_bf16(o[2 * i], o[2 * i + 1]);
        st_v16(dst, v);
    }
}

template <int ACT>
__global__ void __launch_bounds__(AB_THREADS)
act_bwd_kernel(const __nv_bfloat16 *__restrict__ pa, const __nv_bfloat16 *__restrict__ pb,
               const __nv_bfloat16 *__restrict__ dh, int e, int64_t c_max, int h,
               const int32_t *__restrict__ counts, const int32_t *__restrict__ c_dev,
               __nv_bfloat16 *__restrict__ d_pre, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    constexpr bool swiglu = ACT == MOE_ACT_SWIGLU;
    const int j = blockIdx.y;
    const int64_t kept = min((int64_t)min(counts[j], *c_dev), c_max);
    const int hv = h / 8;                                  // 16-byte chunks per row
    const int64_t h2 = swiglu ? 2 * (int64_t)h : (int64_t)h;
    // the CTAs of an expert stride over its kept rows, AB_ROWS at a time
    for (int64_t r0 = (int64_t)blockIdx.x * AB_ROWS; r0 < kept;
         r0 += (int64_t)gridDim.x * AB_ROWS) {
        const int nrow = (int)min((int64_t)AB_ROWS, kept - r0);
        const int n = nrow * hv;   // chunks of this row block (AB_ROWS * h / 8 fits an int)
        const int64_t row0 = (int64_t)j * c_max + r0;
        for (int q0 = threadIdx.x; q0 < n; q0 += AB_THREADS * AB_U) {
            V16 va[AB_U], vb[AB_U], vg[AB_U];
            int rr[AB_U], cc[AB_U];   // row in the block, chunk in the row
            // every load of the batch in flight before any arithmetic
#pragma unroll
            for (int u = 0; u < AB_U; u++) {
                const int q = q0 + u * AB_THREADS;
                rr[u] = q / hv;
                cc[u] = q - rr[u] * hv;
                if (q < n) {
                    const int64_t off = (row0 + rr[u]) * h + cc[u] * 8;
                    va[u] = ld_stream(pa + off);
                    vg[u] = ld_stream(dh + off);
                    if (swiglu) vb[u] = ld_stream(pb + off);
                }
            }
#pragma unroll
            for (int u = 0; u < AB_U; u++) {
                if (q0 + u * AB_THREADS < n)
                    act_bwd_chunk<ACT>(va[u], vb[u], vg[u], d_pre + (row0 + rr[u]) * h2 + cc[u] * 8,
                                       h);
            }
        }
    }
}

// --------------------------------------------------------- column sums
// A CTA owns CS_COLS columns of one expert, lane l columns 8l .. 8l + 7 (one
// 16-byte load a row); its 16 warps take every 16th kept row, CS_U rows in
// flight, and the partials are added in warp order.
constexpr int CS_WARPS = 16, CS_COLS = 256, CS_U = 4;

struct ColsumOp {
    const __nv_bfloat16 *src;
    int cols;
    int64_t pitch;
    void *out;   // bf16, or fp32 when the launch says so
};
struct ColsumOps {
    ColsumOp op[2];
};
static_assert(CS_COLS == 32 * 8 && CS_WARPS * 32 >= CS_COLS, "8 columns a lane, a thread a column");

__global__ void __launch_bounds__(CS_WARPS * 32)
colsum_kernel(ColsumOps ops, int64_t c_max, const int32_t *__restrict__ counts,
              const int32_t *__restrict__ c_dev, int out_f32, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    __shared__ float part[CS_WARPS][CS_COLS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j = blockIdx.y;
    // the column blocks of op 0, then those of op 1
    const int nb0 = (ops.op[0].cols + CS_COLS - 1) / CS_COLS;
    const ColsumOp &o = ops.op[(int)blockIdx.x < nb0 ? 0 : 1];
    const int bx = (int)blockIdx.x < nb0 ? (int)blockIdx.x : (int)blockIdx.x - nb0;
    const __nv_bfloat16 *__restrict__ src = o.src;
    const int cols = o.cols;
    const int64_t pitch = o.pitch;
    const int c0 = bx * CS_COLS + 8 * lane;
    const int64_t kept = max(0, min(min(counts[j], *c_dev), (int)min(c_max, (int64_t)0x7fffffff)));
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] = 0.0f;
    if (c0 < cols) {
        const __nv_bfloat16 *sp = src + (int64_t)j * c_max * pitch + c0;
        for (int64_t r0 = warp; r0 < kept; r0 += (int64_t)CS_WARPS * CS_U) {
            V16 v[CS_U];
#pragma unroll
            for (int u = 0; u < CS_U; u++) {
                const int64_t r = r0 + (int64_t)u * CS_WARPS;
                if (r < kept) v[u] = ld_stream(sp + r * pitch);
            }
#pragma unroll
            for (int u = 0; u < CS_U; u++) {
                if (r0 + (int64_t)u * CS_WARPS < kept) {
                    float f[8];
                    Elt<__nv_bfloat16>::unpack(v[u], f);
#pragma unroll
                    for (int i = 0; i < 8; i++) acc[i] += f[i];
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; i++) part[warp][8 * lane + i] = acc[i];
    __syncthreads();
    // threads 0 .. CS_COLS - 1 finish one column each
    const int col = bx * CS_COLS + threadIdx.x;
    if (threadIdx.x < CS_COLS && col < cols) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < CS_WARPS; w++) sum += part[w][threadIdx.x];
        if (out_f32) static_cast<float *>(o.out)[(int64_t)j * cols + col] = sum;
        else static_cast<__nv_bfloat16 *>(o.out)[(int64_t)j * cols + col] = __float2bfloat16_rn(sum);
    }
}

}  // namespace

moe_status transpose_pad_launch(const __nv_bfloat16 *src, int64_t src_batch, int64_t src_pitch,
                                __nv_bfloat16 *dst, int64_t dst_batch, int64_t dst_pitch,
                                int batches, int rows, int cols, int dst_cols,
                                const int32_t *counts, const int32_t *skip, const int32_t *c_dev,
                                int32_t *status, cudaStream_t stream) {
    if (batches < 1 || batches > 65535 || rows < 0 || cols < 1 || dst_cols < rows ||
        cols % 8 || dst_cols % 8 || src_pitch % 8 || dst_pitch % 8 || src_batch % 8 ||
        dst_batch % 8 || !aligned16(src) || !aligned16(dst))
        return MOE_ERR_INVALID_ARG;
    const int rblocks = (dst_cols + TP - 1) / TP;
    const dim3 grid((unsigned)(rblocks < TP_GRID_X ? rblocks : TP_GRID_X),
                    (unsigned)((cols + TP - 1) / TP), (unsigned)batches);
    if (grid.y > 65535) return MOE_ERR_UNSUPPORTED;
    return launch_pdl(transpose_pad_kernel, grid, dim3(TP_THREADS), 0, stream,
                      (const uint16_t *)src, src_batch, src_pitch, (uint16_t *)dst, dst_batch,
                      dst_pitch, rows, cols, dst_cols, counts, skip, c_dev, status);
}

moe_status act_bwd_launch(const __nv_bfloat16 *pa, const __nv_bfloat16 *pb,
                          const __nv_bfloat16 *d_hid, moe_act act, int e, int64_t c_max, int h,
                          const int32_t *counts, const int32_t *c_dev, __nv_bfloat16 *d_pre,
                          int32_t *status, cudaStream_t stream) {
    if (h % 8 != 0 || e < 1 || e > 65535) return MOE_ERR_INVALID_ARG;
    int64_t gx = (c_max + AB_ROWS - 1) / AB_ROWS;
    if (gx > AB_GRID_X) gx = AB_GRID_X;   // CTAs per expert; they stride over the kept rows
    const dim3 grid((unsigned)gx, (unsigned)e);
    if (act == MOE_ACT_SWIGLU)
        return launch_pdl(act_bwd_kernel<MOE_ACT_SWIGLU>, grid, dim3(AB_THREADS), 0, stream, pa, pb,
                          d_hid, e, c_max, h, counts, c_dev, d_pre, status);
    if (act == MOE_ACT_RELU)
        return launch_pdl(act_bwd_kernel<MOE_ACT_RELU>, grid, dim3(AB_THREADS), 0, stream, pa, pb,
                          d_hid, e, c_max, h, counts, c_dev, d_pre, status);
    return launch_pdl(act_bwd_kernel<MOE_ACT_GELU>, grid, dim3(AB_THREADS), 0, stream, pa, pb, d_hid,
                      e, c_max, h, counts, c_dev, d_pre, status);
}

// ------------------------------------------------------------ tail rows
namespace {

constexpr int TR_WARPS = 8;   // one warp per row, 64 / TR_WARPS CTAs per expert and operand

__global__ void __launch_bounds__(TR_WARPS * 32)
tail_rows_kernel(TailOps ops, int64_t c_max, const int32_t *__restrict__ counts,
                 const int32_t *__restrict__ c_dev, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    const TailOp &o = ops.op[blockIdx.z];
    const __nv_bfloat16 *__restrict__ src = o.src;
    __nv_bfloat16 *__restrict__ dst = o.dst;
    const int64_t src_pitch = o.pitch;
    const int cols = o.cols;
    const int j = blockIdx.y;
    const int64_t kept = min((int64_t)max(counts[j], 0), min((int64_t)*c_dev, c_max));
    const int nvalid = (int)(kept & 63);
    if (nvalid == 0) return;
    const int r = blockIdx.x * TR_WARPS + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const __nv_bfloat16 *srow = src + ((int64_t)j * c_max + (kept - nvalid) + r) * src_pitch;
    __nv_bfloat16 *drow = dst + ((int64_t)j * 64 + r) * cols;
    for (int c = lane * 8; c < cols; c += 32 * 8) {
        V16 v{};
        if (r < nvalid) v = ld_v16(srow + c);
        st_v16(drow + c, v);
    }
}

}  // namespace

moe_status tail_rows_launch(const TailOps &ops, int nops, int64_t c_max, int e,
                            const int32_t *counts, const int32_t *c_dev, int32_t *status,
                            cudaStream_t stream) {
    if (nops < 1 || nops > TAIL_MAX_OPS || e < 1 || e > 65535 || c_max < 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < nops; i++) {
        const TailOp &o = ops.op[i];
        if (o.cols < 8 || o.cols % 8 || o.pitch % 8 || !aligned16(o.src) || !aligned16(o.dst))
            return MOE_ERR_INVALID_ARG;
    }
    return launch_pdl(tail_rows_kernel, dim3(64 / TR_WARPS, (unsigned)e, (unsigned)nops),
                      dim3(TR_WARPS * 32), 0, stream, ops, c_max, counts, c_dev, status);
}

// ------------------------------------------------------- zero empty experts
namespace {

constexpr int ZE_THREADS = 256, ZE_BLOCKS = 64;   // CTAs per (expert, matrix)

__global__ void __launch_bounds__(ZE_THREADS)
zero_empty_experts_kernel(ZeroOps ops, int64_t c_max, const int32_t *__restrict__ counts,
                          const int32_t *__restrict__ c_dev, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    const int j = blockIdx.y;
    const int64_t kept = min((int64_t)max(counts[j], 0), min((int64_t)*c_dev, c_max));
    if (kept > 0) return;
    const ZeroOp &o = ops.op[blockIdx.z];
    V16 *dst = reinterpret_cast<V16 *>(static_cast<char *>(o.ptr) + (int64_t)j * o.bytes);
    const int64_t n = o.bytes / 16;
    V16 z{};
    for (int64_t i = (int64_t)blockIdx.x * ZE_THREADS + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * ZE_THREADS)
        st_v16(dst + i, z);
}

}  // namespace

moe_status zero_empty_experts_launch(const ZeroOps &ops, int nops, int64_t c_max, int e,
                                     const int32_t *counts, const int32_t *c_dev, int32_t *status,
                                     cudaStream_t stream) {
    if (nops < 1 || nops > 3 || e < 1 || e > 65535 || c_max < 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < nops; i++)
        if (!ops.op[i].ptr || ops.op[i].bytes < 16 || ops.op[i].bytes % 16 || !aligned16(ops.op[i].ptr))
            return MOE_ERR_INVALID_ARG;
    return launch_pdl(zero_empty_experts_kernel, dim3(ZE_BLOCKS, (unsigned)e, (unsigned)nops),
                      dim3(ZE_THREADS), 0, stream, ops, c_max, counts, c_dev, status);
}

moe_status colsum_launch(const __nv_bfloat16 *src, int e, int64_t c_max, int cols,
                         int64_t src_pitch, const int32_t *counts, const int32_t *c_dev,
                         void *out, int32_t *status, cudaStream_t stream, bool out_f32,
                         const __nv_bfloat16 *src2, int cols2, int64_t src2_pitch, void *out2) {
    // rows of whole 16-byte chunks
    if (e < 1 || e > 65535 || cols < 1 || cols % 8 || src_pitch % 8 || !aligned16(src))
        return MOE_ERR_INVALID_ARG;
    if (src2 && (cols2 < 1 || cols2 % 8 || src2_pitch % 8 || !aligned16(src2)))
        return MOE_ERR_INVALID_ARG;
    ColsumOps ops{};
    ops.op[0] = ColsumOp{src, cols, src_pitch, out};
    ops.op[1] = src2 ? ColsumOp{src2, cols2, src2_pitch, out2} : ColsumOp{src, 0, src_pitch, out};
    const int nb = (cols + CS_COLS - 1) / CS_COLS + (src2 ? (cols2 + CS_COLS - 1) / CS_COLS : 0);
    return launch_pdl(colsum_kernel, dim3((unsigned)nb, (unsigned)e), dim3(CS_WARPS * 32), 0, stream,
                      ops, c_max, counts, c_dev, out_f32 ? 1 : 0, status);
}

}  // namespace moe
