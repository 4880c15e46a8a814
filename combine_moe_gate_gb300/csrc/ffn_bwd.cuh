// Launchers of the SIMT helper kernels of the expert-FFN backward (ffn_bwd.cu);
// the tensor-core products are the forward's grouped GEMM (ffn_tc.cu).
#pragma once
#include "common.cuh"

namespace moe {

// dst[b][c][r] = src[b][r][c] for r < kept_b, 0 for kept_b <= r < dst_cols,
// over c < cols and b < batches, bf16.  kept_b = min(counts[b], *c_dev, rows)
// when counts is given (then the zeros stop at the next multiple of 64 past
// kept_b: the grouped GEMM's K blocks read no further), else rows.  Batches b with min(skip[b], *c_dev) <= 0
// are left untouched when skip is given.  Row pitches are in elements; the
// batch strides too.
moe_status transpose_pad_launch(const __nv_bfloat16 *src, int64_t src_batch, int64_t src_pitch,
                                __nv_bfloat16 *dst, int64_t dst_batch, int64_t dst_pitch,
                                int batches, int rows, int cols, int dst_cols,
                                const int32_t *counts, const int32_t *skip, const int32_t *c_dev,
                                int32_t *status, cudaStream_t stream);

// Activation backward over the kept rows of each expert, bf16 in and out:
//   ReLU / GELU: d_pre[r, u] = d_hid[r, u] * act'(pa[r, u]);
//   SwiGLU:      d_pre[r, u]     = d_hid * pb * silu'(pa)   (u < h),
//                d_pre[r, h + u] = d_hid * silu(pa).
// pa, pb, d_hid [e, c_max, h]; d_pre [e, c_max, h] or [e, c_max, 2h].
moe_status act_bwd_launch(const __nv_bfloat16 *pa, const __nv_bfloat16 *pb,
                          const __nv_bfloat16 *d_hid, moe_act act, int e, int64_t c_max, int h,
                          const int32_t *counts, const int32_t *c_dev, __nv_bfloat16 *d_pre,
                          int32_t *status, cudaStream_t stream);

// out[b][c] = sum over the kept rows r of src[b][r][c] (fp32 sum in a fixed
// order, one rounding to bf16); src rows of `cols` columns at row pitch
// src_pitch, batch stride c_max * src_pitch.  With src2, the same for a
// second matrix (cols2, src2_pitch, out2) in the same launch.  out_f32: the
// sums are stored in fp32 (not rounded to bf16).
moe_status colsum_launch(const __nv_bfloat16 *src, int e, int64_t c_max, int cols,
                         int64_t src_pitch, const int32_t *counts, const int32_t *c_dev,
                         void *out, int32_t *status, cudaStream_t stream, bool out_f32 = false,
                         const __nv_bfloat16 *src2 = nullptr, int cols2 = 0,
                         int64_t src2_pitch = 0, void *out2 = nullptr);

// The partly kept last 64-row block of every expert, for the MN-major weight
// gradients, for up to TAIL_MAX_OPS operands in one launch: with kept_b =
// min(counts[b], *c_dev, c_max) and r0 = kept_b rounded down to a multiple of
// 64, dst[b][r] = src[b][r0 + r] for r < kept_b - r0 and 0 for the rest of
// the 64 rows; experts whose kept rows end on a block boundary are left
// untouched (nothing reads them).  src rows of `cols` columns at row pitch
// `pitch`, c_max rows per expert; dst [e, 64, cols] dense.
constexpr int TAIL_MAX_OPS = 4;
struct TailOp {
    const __nv_bfloat16 *src;
    int64_t pitch;
    int cols;
    __nv_bfloat16 *dst;
};
struct TailOps {
    TailOp op[TAIL_MAX_OPS];
};
moe_status tail_rows_launch(const TailOps &ops, int nops, int64_t c_max, int e,
                            const int32_t *counts, const int32_t *c_dev, int32_t *status,
                            cudaStream_t stream);

// Zero the `bytes` of slab b (of up to 3 matrices [e, ...], slab b of matrix i
// at op[i].ptr + b * op[i].bytes) for every expert b without kept rows
// (min(counts[b], *c_dev, c_max) == 0); other slabs untouched.  16-byte
// stores; bytes a multiple of 16, pointers 16-byte aligned.
struct ZeroOp {
    void *ptr;
    int64_t bytes;
};
struct ZeroOps {
    ZeroOp op[3];
};
moe_status zero_empty_experts_launch(const ZeroOps &ops, int nops, int64_t c_max, int e,
                                     const int32_t *counts, const int32_t *c_dev, int32_t *status,
                                     cudaStream_t stream);

}  // namespace moe
