/*
 * moe_gate.h -- C ABI of the single-GPU top-k Mixture-of-Experts layer hot path
 * (gate -> capacity/locations -> encode -> expert FFN -> decode, plus the
 * backward of encode and decode), built for NVIDIA GB300 (sm_103a).
 *
 * Sources restated (web pages, cited by title and section):
 *   [Tutel]  "Tutel" project profile: key-configuration table (MOELayer
 *            gate_type {'type': 'top', 'k', 'capacity_factor'}, experts
 *            {'type': 'ffn', hidden_size_per_expert, has_fc1_bias,
 *            has_fc2_bias}) and the FAQ on capacity_factor.
 *   [Blog]   "MoE training systems: DeepSpeed-MoE vs Tutel", section 1.4
 *            (dense token-to-expert mapping table; fused top-k + cumsum +
 *            scatter; data-layout transform instead of einsum) and section 3.5
 *            (fast encode/decode kernels K0, K1, K2; dynamic capacity factor).
 *   [PR8195] DeepSpeed PR #8195 (follow-up to #8174): change 1 (per-route
 *            int32 index/location/gate, capacity resolved once without a
 *            device-to-host sync), change 2 (the [e, c, m] vs flat [e*c, m]
 *            buffer hazard), change 3 (index dispatch, fp32 combine).
 *
 * Conventions shared by every call:
 *   - Every pointer argument is caller-owned memory.  Device pointers must be
 *     16-byte aligned.  Tensors are dense row-major with the shapes given.
 *     Outputs overlap neither the inputs nor each other.
 *   - No call allocates, frees or synchronises.  Work is enqueued on `stream`
 *     (a cudaStream_t passed as void*; NULL = the legacy default stream).
 *   - Routing tables are route-major [k, s]: entry (r, t) is at r*s + t.
 *     Route r of token t is its r-th best expert.
 *   - Expert buffers are physically [e, c_max, m] (row stride c_max*m per
 *     expert).  The logical [e, c, m] view is rows 0..c-1 of each expert.
 *     c_max is fixed by the caller; the data-dependent c lives in device
 *     memory (`c_dev`) and is never read back by the library.
 *   - A route is kept iff loc < c.  Dropped routes keep their un-clipped loc.
 *   - dev_status: caller-owned device int32, zeroed by the caller.  A kernel
 *     that detects a data-dependent error (c > c_max, an index out of range,
 *     a bounded wait that gave up) stores the first error code there.  Every
 *     kernel reads it on entry and does nothing if it is non-zero.  The caller
 *     reads it after its own synchronisation.
 *   - Host-side validation is synchronous: a bad shape, NULL or misaligned
 *     pointer returns MOE_ERR_INVALID_ARG and nothing is launched.  A launch
 *     failure returns MOE_ERR_CUDA.
 *   - Shapes: s >= 1, 1 <= k <= min(e, 32), 1 <= e <= 1024, m, h >= 1.
 *     Rows must be 16-byte multiples: m and h multiples of 8 (bf16) or 4 (fp32).
 */
#ifndef MOE_GATE_H
#define MOE_GATE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* bad shape / pointer (host) or bad index (device) */
    MOE_ERR_UNSUPPORTED = 2,  /* valid but not implemented combination */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
    MOE_ERR_CAPACITY = 4,     /* device: capacity c exceeds c_max */
    MOE_ERR_TIMEOUT = 5       /* device: a bounded wait gave up */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
    MOE_ACT_RELU = 0,   /* y = relu(x W1^T + b1) W2^T + b2 */
    MOE_ACT_GELU = 1,   /* y = gelu_erf(x W1^T + b1) W2^T + b2 */
    MOE_ACT_SWIGLU = 2  /* y = (silu(x W1^T) * (x W3^T)) W2^T, no biases */
} moe_act;

#define MOE_FLAG_NORMALIZE_GATES 1u /* divide the k selected gates by their sum */
#define MOE_FLAG_ZERO_FILL 2u       /* zero the unoccupied rows 0..c-1 of each expert */

/*
 * Gate ([Tutel] gate_type 'top'; [Blog] 1.4 fused top-k).
 *   logits[t, j] = fp32 dot(x[t, :], wg[:, j]) + bias[j], fused multiply-adds
 *   (one rounding each) in a fixed order, then one fp32 add of the bias:
 *     e <= 32: the features are cut into chunks of one 16-byte load (8 bf16 or
 *       4 fp32 elements); chunk c goes to lane c mod 32; each of the 32 lanes
 *       accumulates its features from +0 in ascending index; the lane sums are
 *       combined by an xor butterfly (o = 16, 8, 4, 2, 1: v[l] + v[l xor o]),
 *       and the logit is lane 0's value.
 *     e > 32: one accumulator from +0 in ascending feature index.
 *   This fixed order makes idx reproducible bit for bit.
 *   idx[r, t]: expert at position r when experts are ordered by (logit
 *   descending, index ascending).  gates[r, t]: softmax probability of that
 *   expert over all e logits; with MOE_FLAG_NORMALIZE_GATES divided by the sum
 *   of the k selected probabilities.
 * x [s, m] in `xdt`; wg [m, e] fp32; bias [e] fp32 or NULL.
 * idx [k, s] int32 and gates [k, s] fp32 are written.  e <= 256 here.
 */
moe_status moe_gate_topk(const void *x, moe_dtype xdt, const float *wg, const float *bias,
                         int64_t s, int m, int e, int k, unsigned flags,
                         int32_t *idx, float *gates, int32_t *dev_status, void *stream);

/*
 * Capacity bound on the host ([Tutel] FAQ capacity_factor; [Blog] 3.5).
 *   f > 0: exactly c = ceil(f*k*s/e)  (evaluated exactly on the float value f);
 *   f = 0: s  (the largest c the no-drop rule can produce);
 *   f < 0: min(ceil(-f*k*s/e), s).
 * A c_max at least this large never triggers MOE_ERR_CAPACITY.
 */
int64_t moe_capacity_bound(float capacity_factor, int64_t s, int e, int k);

/* Bytes of device workspace moe_capacity_locations needs. */
size_t moe_capacity_workspace_size(int64_t s, int e, int k);

/*
 * Capacity and slot locations ([Blog] 1.4 cumsum; [Blog] 3.5 dynamic capacity).
 *   counts[j] = number of routes that chose expert j (before any drop).
 *   c = ceil(f*k*s/e) for f > 0; max_j counts[j] for f = 0;
 *       min(ceil(-f*k*s/e), max_j counts[j]) for f < 0.   Written to c_dev[0].
 *   loc[r, t] = number of routes ahead of (r, t) in route-priority order
 *   (all tokens' route 0 in token order, then route 1, ...) that chose the
 *   same expert.  Kept iff loc < c.
 *   c > c_max stores MOE_ERR_CAPACITY in dev_status (loc/counts still valid).
 * idx [k, s] int32 in; loc [k, s] int32, counts [e] int32, c_dev [1] int32 out.
 * workspace: device memory of moe_capacity_workspace_size() bytes, contents
 * ignored on entry (scratch).
 */
moe_status moe_capacity_locations(const int32_t *idx, int64_t s, int e, int k,
                                  float capacity_factor, int64_t c_max,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t *loc, int32_t *counts, int32_t *c_dev,
                                  int32_t *dev_status, void *stream);

/*
 * moe_capacity_locations without a workspace argument: the same results from
 * the same kernels, with their scratch in a fixed array inside the library.
 * The pages have no counterpart; this entry point exists for callers that
 * cannot allocate device memory themselves -- for example a plugin running
 * inside an inference engine that owns the device's whole memory pool, or a
 * latency-critical path where cudaMalloc's implicit device synchronisation is
 * not acceptable.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Scratch limit: MOE_CAPACITY_NOALLOC_SCRATCH_BYTES (1 MiB), held
 *     on every GPU that loads the library until the process exits.  Shapes
 *     whose moe_capacity_workspace_size() exceeds it return
 *     MOE_ERR_UNSUPPORTED with nothing launched.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and keeps it for that device's CUDA context; after
 *     cudaDeviceReset the next call looks it up again.  Make the first call on
 *     each device (and the first after a reset) before any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (different
 *     streams without ordering between them) race and give wrong locations.
 *     Calls ordered on one stream are safe; nothing needs clearing in between.
 */
moe_status moe_capacity_locations_noalloc(const int32_t *idx, int64_t s, int e, int k,
                                          float capacity_factor, int64_t c_max, int32_t *loc,
                                          int32_t *counts, int32_t *c_dev, int32_t *dev_status,
                                          void *stream);

/* Bytes of the fixed scratch array moe_capacity_locations_noalloc uses. */
#define MOE_CAPACITY_NOALLOC_SCRATCH_BYTES (1u << 20)

/*
 * Fast encode ([Blog] 3.5, kernel K1 forward; [PR8195] change 3).
 *   buf[idx[r,t], loc[r,t], :] = x[t, :] for every kept route (unweighted copy).
 *   With MOE_FLAG_ZERO_FILL, rows min(counts[j], c)..c-1 of every expert j are
 *   set to zero as well (counts required then, else it may be NULL).  Other
 *   rows of buf are left untouched.
 * x [s, m]; buf [e, c_max, m], both in `dt`.
 */
moe_status moe_encode(const void *x, moe_dtype dt, const int32_t *idx, const int32_t *loc,
                      const int32_t *counts, const int32_t *c_dev, int64_t s, int m, int e,
                      int k, int64_t c_max, unsigned flags, void *buf, int32_t *dev_status,
                      void *stream);

/* Bytes of device workspace moe_expert_ffn needs (the hidden activations). */
size_t moe_expert_ffn_workspace_size(moe_dtype dt, moe_act act, int e, int64_t c_max, int m,
                                     int h);

/*
 * Per-expert FFN ([Tutel] experts 'ffn'; [Blog] 3.5 batched expert matmul over
 * (E, C, D)).  For every expert j and row i < min(counts[j], c):
 *   hid = act(buf[j,i,:] W1[j]^T + b1[j])        (ReLU / GELU, exact erf form)
 *   hid = silu(buf[j,i,:] W1[j]^T) * (buf[j,i,:] W3[j]^T)      (SwiGLU)
 *   out[j,i,:] = hid W2[j]^T + b2[j]
 * Accumulation in fp32; the hidden activation is rounded to `dt` before the
 * second product; each output is rounded once to `dt`.  Rows >= the kept
 * count are not written.
 * buf, out [e, c_max, m]; w1, w3 [e, h, m]; w2 [e, m, h]; b1 [e, h]; b2 [e, m];
 * all in `dt`.  b1/b2 may be NULL (no bias); w3 only for SwiGLU, which takes
 * no biases.  workspace: moe_expert_ffn_workspace_size() bytes, scratch.
 * bf16 runs on the tensor cores (tcgen05, fp32 accumulation in TMEM); fp32
 * runs on the SIMT cores with fp32 fused multiply-add.
 */
moe_status moe_expert_ffn(const void *buf, moe_dtype dt, const int32_t *counts,
                          const int32_t *c_dev, const void *w1, const void *b1, const void *w3,
                          const void *w2, const void *b2, moe_act act, int e, int64_t c_max,
                          int m, int h, void *workspace, size_t workspace_bytes, void *out,
                          int32_t *dev_status, void *stream);

/*
 * moe_expert_ffn for training (bf16): the same outputs, and fc1 also stores
 * what moe_expert_ffn_bwd_saved needs instead of recomputing it, for the kept
 * rows (other rows not written), rounded once to bf16 from the fp32 sums:
 *   ReLU / GELU: the pre-activation buf W1^T + b1, pre [e, c_max, h];
 *   SwiGLU:      a = buf W1^T and b = buf W3^T, pre [e, c_max, 2h] (a, then b).
 * Errors: as moe_expert_ffn; MOE_ERR_INVALID_ARG for a NULL or misaligned
 * pre; MOE_ERR_UNSUPPORTED for fp32.
 */
moe_status moe_expert_ffn_train(const void *buf, moe_dtype dt, const int32_t *counts,
                                const int32_t *c_dev, const void *w1, const void *b1,
                                const void *w3, const void *w2, const void *b2, moe_act act, int e,
                                int64_t c_max, int m, int h, void *workspace,
                                size_t workspace_bytes, void *out, void *pre, int32_t *dev_status,
                                void *stream);

/*
 * Fast decode ([Blog] 3.5, K0 forward; [PR8195] change 3, fp32 combine).
 *   y[t, :] = sum over kept routes r of gates[r,t] * out[idx[r,t], loc[r,t], :],
 *   accumulated in fp32 with fused multiply-add in ascending r from +0 and
 *   rounded once to `dt`.  Tokens with every route dropped get 0.
 * out [e, c_max, m], y [s, m] in `dt`; gates [k, s] fp32.
 */
moe_status moe_decode(const void *out, moe_dtype dt, const int32_t *idx, const int32_t *loc,
                      const float *gates, const int32_t *c_dev, int64_t s, int m, int e, int k,
                      int64_t c_max, void *y, int32_t *dev_status, void *stream);

/*
 * Backward of decode ([Blog] 3.5: K1 is combine's backward, K2 the cross term).
 *   d_out[idx, loc, :] = gates[r,t] * dy[t, :]  (exact product rounded once)
 *   d_gates[r, t] = sum_i dy[t,i] * out[idx, loc, i]  (fp32), 0 if dropped.
 *   With MOE_FLAG_ZERO_FILL (counts required) unoccupied rows < c of d_out
 *   are zeroed; otherwise they are left untouched.
 * dy [s, m], out and d_out [e, c_max, m] in `dt`; gates, d_gates [k, s] fp32.
 */
moe_status moe_decode_bwd(const void *dy, const void *out, moe_dtype dt, const int32_t *idx,
                          const int32_t *loc, const float *gates, const int32_t *counts,
                          const int32_t *c_dev, int64_t s, int m, int e, int k, int64_t c_max,
                          unsigned flags, void *d_out, float *d_gates, int32_t *dev_status,
                          void *stream);

/*
 * Backward of encode ([Blog] 3.5: K0 with unit weights).
 *   dx[t, :] = sum over kept routes of d_buf[idx, loc, :], fp32 accumulation
 *   in ascending r from +0, rounded once to `dt`.  All-dropped tokens get 0.
 * d_buf [e, c_max, m], dx [s, m] in `dt`.
 */
moe_status moe_encode_bwd(const void *d_buf, moe_dtype dt, const int32_t *idx,
                          const int32_t *loc, const int32_t *c_dev, int64_t s, int m, int e,
                          int k, int64_t c_max, void *dx, int32_t *dev_status, void *stream);

/* Bytes of device workspace moe_expert_ffn_bwd needs (0 if unsupported). */
size_t moe_expert_ffn_bwd_workspace_size(moe_dtype dt, moe_act act, int e, int64_t c_max, int m,
                                         int h);

/*
 * Per-expert FFN backward (the gradient of moe_expert_ffn; the pages give
 * only the forward experts 'ffn' of [Tutel]).  For L = sum over kept rows of
 * <d_out, out>, with every kept row i < min(counts[j], c) of expert j:
 *   pre = buf W1^T + b1 (recomputed), d_hid = d_out W2,
 *   d_pre = d_hid * act'(pre)   (SwiGLU: d_a = d_hid * b * silu'(a),
 *                                d_b = d_hid * silu(a), a = buf W1^T, b = buf W3^T),
 *   d_buf = d_pre W1 (+ d_b W3), d_w2 = d_out^T hid, d_b2 = sum d_out,
 *   d_w1 = d_pre^T buf (d_a for SwiGLU), d_w3 = d_b^T buf, d_b1 = sum d_pre.
 * Inputs: buf [e, c_max, m] and hid [e, c_max, h] as moe_expert_ffn read and
 * wrote them (hid is its workspace after the call); w1, w3 [e, h, m];
 * w2 [e, m, h]; b1 [e, h] or NULL; d_out [e, c_max, m]; counts, c_dev as for
 * the forward.  Outputs in `dt`: d_buf [e, c_max, m] (rows past the kept
 * count not written), d_w1, d_w3 [e, h, m], d_w2 [e, m, h], d_b1 [e, h],
 * d_b2 [e, m].  d_w3 is SwiGLU's only, which takes no biases; d_b1 / d_b2 may
 * be NULL.  workspace: moe_expert_ffn_bwd_workspace_size() bytes, scratch.
 * bf16 only (MOE_ERR_UNSUPPORTED for fp32): every product is the forward's
 * tensor-core grouped GEMM (fp32 accumulation in TMEM); d_hid and d_pre (and
 * SwiGLU's recomputed a and b) are rounded to bf16 between the products, the
 * ReLU / GELU pre-activation is recomputed in fp32 inside the product that
 * forms d_pre.
 */
moe_status moe_expert_ffn_bwd(const void *buf, const void *hid, moe_dtype dt,
                              const int32_t *counts, const int32_t *c_dev, const void *w1,
                              const void *b1, const void *w3, const void *w2, moe_act act, int e,
                              int64_t c_max, int m, int h, const void *d_out, void *workspace,
                              size_t workspace_bytes, void *d_buf, void *d_w1, void *d_w3,
                              void *d_w2, void *d_b1, void *d_b2, int32_t *dev_status,
                              void *stream);

/*
 * moe_expert_ffn_bwd with what moe_expert_ffn_train kept (pre): d_pre is
 * formed in the epilogue of the product d_out W2, so d_hid is neither rounded
 * nor stored and nothing is recomputed:
 *   ReLU / GELU: d_pre = (d_out W2) * act'(pre), pre [e, c_max, h];
 *   SwiGLU:      [d_a | d_b] = (d_out W2) * [b silu'(a) | silu(a)],
 *                pre = [a | b] [e, c_max, 2h].
 * The other outputs as moe_expert_ffn_bwd (w3 and d_w3 for SwiGLU only, NULL
 * otherwise; d_b1 / d_b2 for ReLU / GELU only, or NULL).  d_w1, d_w3, d_w2,
 * d_b1, d_b2 in `wgrad_dt`: MOE_BF16, or MOE_F32 for gradients kept in fp32
 * (the products' fp32 sums stored unrounded, as an optimiser with fp32 master
 * weights wants them); d_buf in `dt`.  workspace:
 * moe_expert_ffn_bwd_workspace_size() bytes.  Errors: as moe_expert_ffn_bwd;
 * MOE_ERR_INVALID_ARG for a NULL or misaligned pre or another wgrad_dt.
 */
moe_status moe_expert_ffn_bwd_saved(const void *buf, const void *hid, const void *pre,
                                    moe_dtype dt, const int32_t *counts, const int32_t *c_dev,
                                    const void *w1, const void *w3, const void *w2, moe_act act,
                                    int e, int64_t c_max, int m, int h, const void *d_out,
                                    void *workspace, size_t workspace_bytes, void *d_buf,
                                    moe_dtype wgrad_dt, void *d_w1, void *d_w3, void *d_w2,
                                    void *d_b1, void *d_b2, int32_t *dev_status, void *stream);

/*
 * Gate backward ([Tutel] gate_type 'top': the gates are softmax probabilities
 * of the k selected experts, renormalised over them with
 * MOE_FLAG_NORMALIZE_GATES).  Top-k selection is piecewise constant, so the
 * gradient flows through the softmax only.  With A = sum_r dg[r,t] g[r,t]:
 *   renormalised:  d_logits[t, idx[r,t]] = g (dg - A), other experts 0;
 *   raw softmax:   d_logits[t, j] = -p_j A + sum over routes r to j of dg g,
 *                  p = softmax of the logits (recomputed here from x, wg, bias);
 *   d_wg = x^T d_logits [m, e],  d_bias = sum over t of d_logits [e],
 *   d_x = d_logits wg^T [s, m].
 * Inputs: x [s, m] in `xdt`; wg [m, e] fp32; bias [e] fp32 or NULL (used only
 * to recompute the logits of the raw softmax); idx, gates [k, s] as the gate
 * wrote them; d_gates [k, s] fp32 (e.g. moe_decode_bwd's).  Outputs, all fp32
 * and deterministic: d_logits [s, e] (required), d_wg [m, e], d_bias [e],
 * d_x [s, m] (each may be NULL).  Fixed summation orders: A sums the routes in
 * route order; d_wg and d_bias sum each of 64 contiguous token slices in token
 * order, then the slices in order; d_x sums, per token, the experts in order
 * (raw softmax) or its k routes in route order (renormalised gates, where the
 * other experts' d_logits are zero).  e <= 256 here.
 * This entry point extends the pages' forward gate to its backward.
 */
moe_status moe_gate_bwd(const void *x, moe_dtype xdt, const float *wg, const float *bias,
                        int64_t s, int m, int e, int k, unsigned flags, const int32_t *idx,
                        const float *gates, const float *d_gates, float *d_logits, float *d_wg,
                        float *d_bias, float *d_x, int32_t *dev_status, void *stream);

/*
 * Low-precision experts ([Tutel] profile, notes and highlights: FP8 among its
 * inference formats, "blockwise FP8" without a block size).  Here an operand
 * is e4m3 (OCP FP8 E4M3: 4 exponent bits, bias 7, 3 mantissa bits, largest
 * finite 448) with one fp32 scale per row, so the scales apply once, after
 * the contraction:
 *   q[r, i] = e4m3(x[r, i] / scale[r]),  scale[r] = amax_i |x[r, i]| / 448
 * (fp32 divisions, nearest-even, saturating at +-448; scale 1 for a zero row).
 *
 * moe_quantize_rows_fp8: src [batches, rows_per_batch, cols] bf16 -> q (same
 * shape, one byte per code) and scale [batches, rows_per_batch] fp32.  With
 * counts [batches] and c_dev (both or neither), only the rows r <
 * min(counts[b], *c_dev, rows_per_batch) of batch b are written (the kept
 * rows of an expert buffer); else every row (e.g. weights [e, rows, cols]).
 * cols a multiple of 16.  Deterministic; the codes match an exact-arithmetic
 * reference bit for bit.  This entry point extends the pages' expert FFN to
 * the FP8 format.
 */
moe_status moe_quantize_rows_fp8(const void *src, int64_t batches, int64_t rows_per_batch,
                                 int cols, const int32_t *counts, const int32_t *c_dev, void *q,
                                 float *scale, int32_t *dev_status, void *stream);

/* Bytes of device workspace moe_expert_ffn_fp8 needs (0: bad shape). */
size_t moe_expert_ffn_fp8_workspace_size(int e, int64_t c_max, int m, int h);

/*
 * The expert FFN (ReLU / GELU) on e4m3 operands: buf_q [e, c_max, m] with
 * buf_scale [e, c_max] (moe_quantize_rows_fp8 of the encoded buffer's kept
 * rows), w1_q [e, h, m] with w1_scale [e, h], w2_q [e, m, h] with w2_scale
 * [e, m] (weights quantised per output channel), b1 [e, h], b2 [e, m] bf16 or
 * NULL.  For the kept rows of every expert:
 *   hid = bf16(act(s_x s_w1 (x_q . w1_q^T) + b1));  hid quantised per row;
 *   out = bf16(s_h s_w2 (hid_q . w2_q^T) + b2)
 * with fp32 accumulation (tcgen05 kind::f8f6f4 on CTA pairs).  out [e, c_max,
 * m] bf16.  m and h multiples of 16.  Workspace (moe_expert_ffn_fp8_workspace
 * _size() bytes): the bf16 hidden [e, c_max, h] at offset 0, its codes [e,
 * c_max, h] and its scales [e, c_max] fp32 after it, each starting on a
 * 256-byte boundary; a caller may read them after the call.  SwiGLU returns
 * MOE_ERR_UNSUPPORTED.  This entry point extends the pages' expert FFN to the
 * FP8 format.
 */
moe_status moe_expert_ffn_fp8(const void *buf_q, const float *buf_scale, const int32_t *counts,
                              const int32_t *c_dev, const void *w1_q, const float *w1_scale,
                              const void *b1, const void *w2_q, const float *w2_scale,
                              const void *b2, moe_act act, int e, int64_t c_max, int m, int h,
                              void *workspace, size_t workspace_bytes, void *out,
                              int32_t *dev_status, void *stream);

/* Bytes of device workspace moe_layer_forward needs. */
size_t moe_layer_workspace_size(moe_dtype dt, moe_act act, int64_t s, int m, int e, int k,
                                int64_t c_max, int h);

/*
 * The whole forward layer in one call: moe_gate_topk, moe_capacity_locations,
 * moe_encode, moe_expert_ffn and moe_decode enqueued back to back on `stream`
 * with no host synchronisation.  Intermediate tensors the caller may inspect
 * (idx, gates, loc, counts, c_dev, buf, out) are caller-owned outputs; the
 * rest lives in `workspace` (moe_layer_workspace_size() bytes).
 */
moe_status moe_layer_forward(const void *x, moe_dtype dt, const float *wg, const float *gate_bias,
                             const void *w1, const void *b1, const void *w3, const void *w2,
                             const void *b2, moe_act act, int64_t s, int m, int e, int k, int h,
                             float capacity_factor, int64_t c_max, unsigned flags,
                             int32_t *idx, float *gates, int32_t *loc, int32_t *counts,
                             int32_t *c_dev, void *buf, void *out, void *y,
                             void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, void *stream);

/*
 * moe_layer_forward with the layer's input taken from host memory and its
 * output returned to host memory, for a caller whose tokens live on the host:
 * x_host [s, m] is copied into the device buffer x, the layer runs as in
 * moe_layer_forward, and y is copied to y_host [s, m], all three enqueued on
 * `stream` (cudaMemcpyAsync: with pinned host memory the copies are
 * asynchronous; with pageable memory the runtime may block the calling thread
 * until they are done).  Arguments after x are those of moe_layer_forward.
 * The caller synchronises the stream before reading y_host.
 */
moe_status moe_layer_forward_host(const void *x_host, void *y_host, const void *x, moe_dtype dt,
                                  const float *wg, const float *gate_bias, const void *w1,
                                  const void *b1, const void *w3, const void *w2, const void *b2,
                                  moe_act act, int64_t s, int m, int e, int k, int h,
                                  float capacity_factor, int64_t c_max, unsigned flags,
                                  int32_t *idx, float *gates, int32_t *loc, int32_t *counts,
                                  int32_t *c_dev, void *buf, void *out, void *y, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * moe_layer_forward with the capacity dimension cut into `chunks` pieces so
 * that encoding one piece overlaps the expert FFN of the previous one (the
 * one-GPU form of the adaptive pipelining in [Blog] 3.4, which overlaps
 * all-to-all with expert computation by splitting the capacity dimension):
 * gate and capacity run on `stream`; slot rows [i*q, (i+1)*q) of every expert
 * (q = c_max / chunks rounded up to 256 rows) are encoded on `aux_stream` and
 * run through the FFN on `stream` once their encode is done; decode follows
 * on `stream` (a token's routes may fall in different pieces).  Results are
 * bit-identical to moe_layer_forward.  events: 1 + chunks cudaEvent_t handles
 * (passed as void*) created by the caller, used for the cross-stream order;
 * aux_stream may equal stream (no overlap).  bf16 only (fp32, or chunks = 1:
 * the single pass).  1 <= chunks <= 64.  The caller synchronises `stream`.
 */
moe_status moe_layer_forward_pipelined(const void *x, moe_dtype dt, const float *wg,
                                       const float *gate_bias, const void *w1, const void *b1,
                                       const void *w3, const void *w2, const void *b2, moe_act act,
                                       int64_t s, int m, int e, int k, int h, float capacity_factor,
                                       int64_t c_max, unsigned flags, int32_t *idx, float *gates,
                                       int32_t *loc, int32_t *counts, int32_t *c_dev, void *buf,
                                       void *out, void *y, void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, int chunks, void *stream,
                                       void *aux_stream, void *const *events);

/*
 * Measurement helper, not part of the layer: launches `blocks` CTAs of 256
 * threads, each thread running 8 independent two-wide chains of `iters` fp32
 * fused multiply-adds (packed fp32x2 FMA when `packed`, else scalar pairs),
 * i.e. blocks * 256 * iters * 32 flop.  Timed by the caller with events, it
 * gives this GPU's fp32 FMA throughput, the roofline of a gate whose logits
 * (2*m*e flop per token) outweigh its HBM bytes.  out: one device float the
 * kernel may write (never for these values).
 */
moe_status moe_probe_fp32_fma(int packed, int blocks, int iters, float *out, void *stream);

/* Human-readable name of a status code (static string). */
const char *moe_status_str(moe_status st);

/* Number of kernels this library has launched in this process (monotonic). */
uint64_t moe_launch_count(void);

/*
 * Error-path test hook, not for production use.  The next n launches of the
 * tensor-core grouped GEMM in this process (moe_expert_ffn, _fp8, _bwd and the
 * layer calls all use it; fc1 and fc2 are one launch each) issue no operand
 * copies, so the MMA issuer's bounded wait on its first stage runs out after
 * about one second: the launch sets MOE_ERR_TIMEOUT in the call's status
 * word, drains, releases its tensor memory and returns, and every later
 * kernel that reads that status word writes nothing.  The context stays
 * usable.  n = 0 cancels pending stalls.  The count is process-wide: calls
 * made meanwhile from other threads may take the stalls.
 * Errors: MOE_ERR_INVALID_ARG for n < 0.
 */
moe_status moe_debug_stall_gemms(int32_t n);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GATE_H */
