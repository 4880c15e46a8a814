// C ABI entry points: synchronous argument checks, then kernel launches.
#include <atomic>

#include "common.cuh"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::atomic<int32_t> g_gemm_stalls{0};
bool take_gemm_stall() {
    int32_t n = g_gemm_stalls.load(std::memory_order_relaxed);
    while (n > 0 && !g_gemm_stalls.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) {
    }
    return n > 0;
}

// kernels (one translation unit each)
moe_status gate_topk_launch(const void *x, moe_dtype xdt, const float *wg, const float *bias,
                            int64_t s, int m, int e, int k, unsigned flags, int32_t *idx,
                            float *gates, int32_t *st, cudaStream_t stream);
moe_status gate_bwd_launch(const void *x, moe_dtype xdt, const float *wg, const float *bias,
                           int64_t s, int m, int e, int k, unsigned flags, const int32_t *idx,
                           const float *gates, const float *d_gates, float *d_logits, float *d_wg,
                           float *d_bias, float *d_x, int32_t *st, cudaStream_t stream);
int64_t capacity_bound_host(float f, int64_t s, int e, int k);
size_t capacity_workspace_bytes(int64_t s, int e, int k);
moe_status capacity_launch(const int32_t *idx, int64_t s, int e, int k, float f, int64_t c_max,
                           void *ws, int32_t *loc, int32_t *counts, int32_t *c_dev, int32_t *st,
                           cudaStream_t stream);
moe_status encode_launch(const void *x, moe_dtype dt, const int32_t *idx, const int32_t *loc,
                         const int32_t *counts, const int32_t *c_dev, int64_t s, int m, int e,
                         int k, int64_t c_max, unsigned flags, void *buf, int32_t *st,
                         cudaStream_t stream, int lo, int hi);
moe_status combine_launch(const void *src, moe_dtype dt, const int32_t *idx, const int32_t *loc,
                          const float *gates, const int32_t *c_dev, int64_t s, int m, int e, int k,
                          int64_t c_max, void *y, int32_t *st, cudaStream_t stream);
moe_status decode_bwd_launch(const void *dy, const void *out, moe_dtype dt, const int32_t *idx,
                             const int32_t *loc, const float *gates, const int32_t *counts,
                             const int32_t *c_dev, int64_t s, int m, int e, int k, int64_t c_max,
                             unsigned flags, void *d_out, float *d_gates, int32_t *st,
                             cudaStream_t stream);
moe_status capacity_noalloc_launch(const int32_t *idx, int64_t s, int e, int k, float f,
                                   int64_t c_max, int32_t *loc, int32_t *counts, int32_t *c_dev,
                                   int32_t *st, cudaStream_t stream);
moe_status probe_fp32_fma_launch(int packed, int blocks, int iters, float *out,
                                 cudaStream_t stream);
bool ffn_tc_supported(int e, int64_t c_max, int m, int h);
moe_status ffn_tc_launch(const void *buf, const int32_t *counts, const int32_t *c_dev,
                         const void *w1, const void *b1, const void *w3, const void *w2,
                         const void *b2, moe_act act, int e, int64_t c_max, int m, int h,
                         void *hid, void *out, int32_t *st, cudaStream_t stream, int row_lo,
                         int row_hi, void *pre = nullptr);
size_t ffn_tc_bwd_workspace_bytes(moe_act act, int e, int64_t c_max, int m, int h);
moe_status quantize_rows_fp8_launch(const void *src, int64_t batches, int64_t rows_per_batch,
                                    int cols, const int32_t *counts, const int32_t *c_dev,
                                    void *q, float *scale, int32_t *st, cudaStream_t stream);
moe_status ffn_tc_fp8_launch(const void *buf_q, const float *buf_scale, const int32_t *counts,
                             const int32_t *c_dev, const void *w1_q, const float *w1_scale,
                             const void *b1, const void *w2_q, const float *w2_scale,
                             const void *b2, moe_act act, int e, int64_t c_max, int m, int h,
                             void *hid, void *hid_q, float *hid_scale, void *out, int32_t *st,
                             cudaStream_t stream);
moe_status ffn_tc_bwd_launch(const void *buf, const void *hid, const int32_t *counts,
                             const int32_t *c_dev, const void *w1, const void *b1, const void *w3,
                             const void *w2, moe_act act, int e, int64_t c_max, int m, int h,
                             const void *d_out, void *ws, void *d_buf, void *d_w1, void *d_w3,
                             void *d_w2, void *d_b1, void *d_b2, int32_t *st, cudaStream_t stream,
                             const void *pre = nullptr, bool wgrad_f32 = false);
moe_status ffn_simt_launch(const void *buf, moe_dtype dt, const int32_t *counts,
                           const int32_t *c_dev, const void *w1, const void *b1, const void *w3,
                           const void *w2, const void *b2, moe_act act, int e, int64_t c_max,
                           int m, int h, void *hid, void *out, int32_t *st, cudaStream_t stream);

}  // namespace moe

using namespace moe;

namespace {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;

inline bool ok16(const void *p) { return p != nullptr && aligned16(p); }
inline bool ok4(const void *p) { return p != nullptr && ((uintptr_t)p & 3u) == 0; }
inline bool opt16(const void *p) { return p == nullptr || aligned16(p); }
inline bool valid_dt(moe_dtype dt) { return dt == MOE_F32 || dt == MOE_BF16; }
inline int vec_of(moe_dtype dt) { return dt == MOE_BF16 ? 8 : 4; }
inline size_t esize(moe_dtype dt) { return dt == MOE_BF16 ? 2 : 4; }
inline size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }

bool routing_shape_ok(int64_t s, int e, int k) {
    return s >= 1 && s <= (int64_t)1 << 30 && e >= 1 && e <= kMaxE && k >= 1 && k <= e &&
           k <= kMaxK && s * (int64_t)k < ((int64_t)1 << 31);
}

bool rows_ok(moe_dtype dt, int m) { return valid_dt(dt) && m >= 1 && m % vec_of(dt) == 0; }

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char *moe_status_str(moe_status st) {
    switch (st) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported combination";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_CAPACITY: return "capacity exceeds c_max";
        case MOE_ERR_TIMEOUT: return "bounded wait timed out";
    }
    return "unknown status";
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status moe_debug_stall_gemms(int32_t n) {
    if (n < 0) return MOE_ERR_INVALID_ARG;
    g_gemm_stalls.store(n, std::memory_order_relaxed);
    return MOE_OK;
}

moe_status moe_gate_topk(const void *x, moe_dtype xdt, const float *wg, const float *bias,
                         int64_t s, int m, int e, int k, unsigned flags, int32_t *idx,
                         float *gates, int32_t *dev_status, void *stream) {
    if (!routing_shape_ok(s, e, k) || !rows_ok(xdt, m) || !ok16(x) || !ok16(wg) || !opt16(bias) ||
        !ok4(idx) || !ok4(gates) || !ok4(dev_status) || (flags & ~3u))
        return MOE_ERR_INVALID_ARG;
    if (e > 256) return MOE_ERR_UNSUPPORTED;
    return gate_topk_launch(x, xdt, wg, bias, s, m, e, k, flags, idx, gates, dev_status,
                            as_stream(stream));
}

moe_status moe_gate_bwd(const void *x, moe_dtype xdt, const float *wg, const float *bias,
                        int64_t s, int m, int e, int k, unsigned flags, const int32_t *idx,
                        const float *gates, const float *d_gates, float *d_logits, float *d_wg,
                        float *d_bias, float *d_x, int32_t *dev_status, void *stream) {
    if (!routing_shape_ok(s, e, k) || !rows_ok(xdt, m) || !ok16(x) || !ok16(wg) ||
        !opt16(bias) || !ok4(idx) || !ok4(gates) || !ok4(d_gates) || !ok4(d_logits) ||
        !opt16(d_wg) || !opt16(d_bias) || !opt16(d_x) || !ok4(dev_status) || (flags & ~3u))
        return MOE_ERR_INVALID_ARG;
    if (e > 256) return MOE_ERR_UNSUPPORTED;
    return gate_bwd_launch(x, xdt, wg, bias, s, m, e, k, flags, idx, gates, d_gates, d_logits,
                           d_wg, d_bias, d_x, dev_status, as_stream(stream));
}

int64_t moe_capacity_bound(float capacity_factor, int64_t s, int e, int k) {
    if (!routing_shape_ok(s, e, k) || capacity_factor != capacity_factor) return -1;
    return capacity_bound_host(capacity_factor, s, e, k);
}

size_t moe_capacity_workspace_size(int64_t s, int e, int k) {
    if (!routing_shape_ok(s, e, k)) return 0;
    return capacity_workspace_bytes(s, e, k);
}

moe_status moe_capacity_locations(const int32_t *idx, int64_t s, int e, int k,
                                  float capacity_factor, int64_t c_max, void *workspace,
                                  size_t workspace_bytes, int32_t *loc, int32_t *counts,
                                  int32_t *c_dev, int32_t *dev_status, void *stream) {
    if (!routing_shape_ok(s, e, k) || c_max < 1 || c_max > 0x7fffffff ||
        capacity_factor != capacity_factor || !ok4(idx) || !ok4(loc) || !ok4(counts) ||
        !ok4(c_dev) || !ok4(dev_status) || !ok16(workspace) ||
        workspace_bytes < capacity_workspace_bytes(s, e, k))
        return MOE_ERR_INVALID_ARG;
    return capacity_launch(idx, s, e, k, capacity_factor, c_max, workspace, loc, counts, c_dev,
                           dev_status, as_stream(stream));
}

moe_status moe_capacity_locations_noalloc(const int32_t *idx, int64_t s, int e, int k,
                                          float capacity_factor, int64_t c_max, int32_t *loc,
                                          int32_t *counts, int32_t *c_dev, int32_t *dev_status,
                                          void *stream) {
    if (!routing_shape_ok(s, e, k) || c_max < 1 || c_max > 0x7fffffff ||
        capacity_factor != capacity_factor || !ok4(idx) || !ok4(loc) || !ok4(counts) ||
        !ok4(c_dev) || !ok4(dev_status))
        return MOE_ERR_INVALID_ARG;
    return capacity_noalloc_launch(idx, s, e, k, capacity_factor, c_max, loc, counts, c_dev,
                                   dev_status, as_stream(stream));
}

moe_status moe_encode(const void *x, moe_dtype dt, const int32_t *idx, const int32_t *loc,
                      const int32_t *counts, const int32_t *c_dev, int64_t s, int m, int e, int k,
                      int64_t c_max, unsigned flags, void *buf, int32_t *dev_status,
                      void *stream) {
    if (!routing_shape_ok(s, e, k) || !rows_ok(dt, m) || c_max < 1 || c_max > 0x7fffffff ||
        !ok16(x) || !ok4(idx) || !ok4(loc) || !ok4(c_dev) || !ok16(buf) || !ok4(dev_status) ||
        (flags & ~3u) || ((flags & MOE_FLAG_ZERO_FILL) && !ok4(counts)))
        return MOE_ERR_INVALID_ARG;
    return encode_launch(x, dt, idx, loc, counts, c_dev, s, m, e, k, c_max, flags, buf, dev_status,
                         as_stream(stream), 0, 0x7fffffff);
}

size_t moe_expert_ffn_workspace_size(moe_dtype dt, moe_act act, int e, int64_t c_max, int m,
                                     int h) {
    (void)act;
    (void)m;
    if (!valid_dt(dt) || e < 1 || c_max < 1 || h < 1) return 0;
    return up256((size_t)e * (size_t)c_max * (size_t)h * esize(dt));
}

static moe_status expert_ffn(const void *buf, moe_dtype dt, const int32_t *counts,
                             const int32_t *c_dev, const void *w1, const void *b1, const void *w3,
                             const void *w2, const void *b2, moe_act act, int e, int64_t c_max,
                             int m, int h, void *workspace, size_t workspace_bytes, void *out,
                             void *pre, int32_t *dev_status, void *stream) {
    if (!rows_ok(dt, m) || !rows_ok(dt, h) || e < 1 || e > kMaxE || c_max < 1 ||
        c_max > 0x7fffffff || !ok16(buf) || !ok4(counts) || !ok4(c_dev) || !ok16(w1) ||
        !ok16(w2) || !opt16(b1) || !opt16(b2) || !ok16(out) || !ok4(dev_status) ||
        !ok16(workspace) ||
        workspace_bytes < moe_expert_ffn_workspace_size(dt, act, e, c_max, m, h))
        return MOE_ERR_INVALID_ARG;
    if (act != MOE_ACT_RELU && act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU)
        return MOE_ERR_INVALID_ARG;
    if (act == MOE_ACT_SWIGLU && (!ok16(w3) || b1 != nullptr || b2 != nullptr))
        return MOE_ERR_INVALID_ARG;
    if (pre && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (pre && !ok16(pre)) return MOE_ERR_INVALID_ARG;
    if (dt == MOE_BF16) {
        if (!ffn_tc_supported(e, c_max, m, h)) return MOE_ERR_UNSUPPORTED;
        return ffn_tc_launch(buf, counts, c_dev, w1, b1, w3, w2, b2, act, e, c_max, m, h,
                             workspace, out, dev_status, as_stream(stream), 0, 0, pre);
    }
    return ffn_simt_launch(buf, dt, counts, c_dev, w1, b1, w3, w2, b2, act, e, c_max, m, h,
                           workspace, out, dev_status, as_stream(stream));
}

moe_status moe_expert_ffn(const void *buf, moe_dtype dt, const int32_t *counts,
                          const int32_t *c_dev, const void *w1, const void *b1, const void *w3,
                          const void *w2, const void *b2, moe_act act, int e, int64_t c_max, int m,
                          int h, void *workspace, size_t workspace_bytes, void *out,
                          int32_t *dev_status, void *stream) {
    return expert_ffn(buf, dt, counts, c_dev, w1, b1, w3, w2, b2, act, e, c_max, m, h, workspace,
                      workspace_bytes, out, nullptr, dev_status, stream);
}

moe_status moe_expert_ffn_train(const void *buf, moe_dtype dt, const int32_t *counts,
                                const int32_t *c_dev, const void *w1, const void *b1,
                                const void *w3, const void *w2, const void *b2, moe_act act, int e,
                                int64_t c_max, int m, int h, void *workspace,
                                size_t workspace_bytes, void *out, void *pre, int32_t *dev_status,
                                void *stream) {
    if (!pre) return MOE_ERR_INVALID_ARG;
    return expert_ffn(buf, dt, counts, c_dev, w1, b1, w3, w2, b2, act, e, c_max, m, h, workspace,
                      workspace_bytes, out, pre, dev_status, stream);
}

moe_status moe_decode(const void *out, moe_dtype dt, const int32_t *idx, const int32_t *loc,
                      const float *gates, const int32_t *c_dev, int64_t s, int m, int e, int k,
                      int64_t c_max, void *y, int32_t *dev_status, void *stream) {
    if (!routing_shape_ok(s, e, k) || !rows_ok(dt, m) || c_max < 1 || c_max > 0x7fffffff ||
        !ok16(out) || !ok4(idx) || !ok4(loc) || !ok4(gates) || !ok4(c_dev) || !ok16(y) ||
        !ok4(dev_status))
        return MOE_ERR_INVALID_ARG;
    return combine_launch(out, dt, idx, loc, gates, c_dev, s, m, e, k, c_max, y, dev_status,
                          as_stream(stream));
}

moe_status moe_decode_bwd(const void *dy, const void *out, moe_dtype dt, const int32_t *idx,
                          const int32_t *loc, const float *gates, const int32_t *counts,
                          const int32_t *c_dev, int64_t s, int m, int e, int k, int64_t c_max,
                          unsigned flags, void *d_out, float *d_gates, int32_t *dev_status,
                          void *stream) {
    if (!routing_shape_ok(s, e, k) || !rows_ok(dt, m) || c_max < 1 || c_max > 0x7fffffff ||
        !ok16(dy) || !ok16(out) || !ok4(idx) || !ok4(loc) || !ok4(gates) || !ok4(c_dev) ||
        !ok16(d_out) || !ok4(d_gates) || !ok4(dev_status) || (flags & ~3u) ||
        ((flags & MOE_FLAG_ZERO_FILL) && !ok4(counts)))
        return MOE_ERR_INVALID_ARG;
    return decode_bwd_launch(dy, out, dt, idx, loc, gates, counts, c_dev, s, m, e, k, c_max, flags,
                             d_out, d_gates, dev_status, as_stream(stream));
}

moe_status moe_encode_bwd(const void *d_buf, moe_dtype dt, const int32_t *idx, const int32_t *loc,
                          const int32_t *c_dev, int64_t s, int m, int e, int k, int64_t c_max,
                          void *dx, int32_t *dev_status, void *stream) {
    if (!routing_shape_ok(s, e, k) || !rows_ok(dt, m) || c_max < 1 || c_max > 0x7fffffff ||
        !ok16(d_buf) || !ok4(idx) || !ok4(loc) || !ok4(c_dev) || !ok16(dx) || !ok4(dev_status))
        return MOE_ERR_INVALID_ARG;
    return combine_launch(d_buf, dt, idx, loc, nullptr, c_dev, s, m, e, k, c_max, dx, dev_status,
                          as_stream(stream));
}

size_t moe_expert_ffn_bwd_workspace_size(moe_dtype dt, moe_act act, int e, int64_t c_max, int m,
                                         int h) {
    if (dt != MOE_BF16 || e < 1 || e > kMaxE || c_max < 1 || m < 1 || h < 1) return 0;
    if (act != MOE_ACT_RELU && act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU) return 0;
    return ffn_tc_bwd_workspace_bytes(act, e, c_max, m, h);
}

static moe_status expert_ffn_bwd(const void *buf, const void *hid, const void *pre, moe_dtype dt,
                                 const int32_t *counts, const int32_t *c_dev, const void *w1,
                                 const void *b1, const void *w3, const void *w2, moe_act act, int e,
                                 int64_t c_max, int m, int h, const void *d_out, void *workspace,
                                 size_t workspace_bytes, void *d_buf, moe_dtype wgrad_dt,
                                 void *d_w1, void *d_w3, void *d_w2, void *d_b1, void *d_b2,
                                 int32_t *dev_status, void *stream) {
    if (wgrad_dt != MOE_BF16 && wgrad_dt != MOE_F32) return MOE_ERR_INVALID_ARG;
    if (!rows_ok(dt, m) || !rows_ok(dt, h) || e < 1 || e > kMaxE || c_max < 1 ||
        c_max > 0x7fffffff || !ok16(buf) || !ok16(hid) || !ok4(counts) || !ok4(c_dev) ||
        !ok16(w1) || !ok16(w2) || !opt16(b1) || !ok16(d_out) || !ok16(workspace) ||
        !ok16(d_buf) || !ok16(d_w1) || !ok16(d_w2) || !opt16(d_b1) || !opt16(d_b2) ||
        !ok4(dev_status))
        return MOE_ERR_INVALID_ARG;
    if (act != MOE_ACT_RELU && act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU)
        return MOE_ERR_INVALID_ARG;
    if (act == MOE_ACT_SWIGLU &&
        (!ok16(w3) || !ok16(d_w3) || b1 != nullptr || d_b1 != nullptr || d_b2 != nullptr))
        return MOE_ERR_INVALID_ARG;
    if (dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < moe_expert_ffn_bwd_workspace_size(dt, act, e, c_max, m, h))
        return MOE_ERR_INVALID_ARG;
    const int64_t h2 = act == MOE_ACT_SWIGLU ? 2 * (int64_t)h : h;
    // every operand of the products within the grouped GEMM's index range
    if (!ffn_tc_supported(e, c_max, m, h) || !ffn_tc_supported(e, h2, m, h) ||
        (int64_t)e * h2 >= ((int64_t)1 << 31) || (int64_t)e * ((c_max + 7) / 8 * 8) >= ((int64_t)1 << 31))
        return MOE_ERR_UNSUPPORTED;
    if (pre && !ok16(pre)) return MOE_ERR_INVALID_ARG;
    return ffn_tc_bwd_launch(buf, hid, counts, c_dev, w1, b1, w3, w2, act, e, c_max, m, h, d_out,
                             workspace, d_buf, d_w1, d_w3, d_w2, d_b1, d_b2, dev_status,
                             as_stream(stream), pre, wgrad_dt == MOE_F32);
}

moe_status moe_expert_ffn_bwd(const void *buf, const void *hid, moe_dtype dt,
                              const int32_t *counts, const int32_t *c_dev, const void *w1,
                              const void *b1, const void *w3, const void *w2, moe_act act, int e,
                              int64_t c_max, int m, int h, const void *d_out, void *workspace,
                              size_t workspace_bytes, void *d_buf, void *d_w1, void *d_w3,
                              void *d_w2, void *d_b1, void *d_b2, int32_t *dev_status,
                              void *stream) {
    return expert_ffn_bwd(buf, hid, nullptr, dt, counts, c_dev, w1, b1, w3, w2, act, e, c_max, m, h,
                          d_out, workspace, workspace_bytes, d_buf, dt, d_w1, d_w3, d_w2, d_b1, d_b2,
                          dev_status, stream);
}

moe_status moe_expert_ffn_bwd_saved(const void *buf, const void *hid, const void *pre,
                                    moe_dtype dt, const int32_t *counts, const int32_t *c_dev,
                                    const void *w1, const void *w3, const void *w2, moe_act act,
                                    int e, int64_t c_max, int m, int h, const void *d_out,
                                    void *workspace, size_t workspace_bytes, void *d_buf,
                                    moe_dtype wgrad_dt, void *d_w1, void *d_w3, void *d_w2,
                                    void *d_b1, void *d_b2, int32_t *dev_status, void *stream) {
    if (!pre) return MOE_ERR_INVALID_ARG;
    return expert_ffn_bwd(buf, hid, pre, dt, counts, c_dev, w1, nullptr, w3, w2, act, e, c_max, m, h,
                          d_out, workspace, workspace_bytes, d_buf, wgrad_dt, d_w1, d_w3, d_w2, d_b1,
                          d_b2, dev_status, stream);
}

size_t moe_layer_workspace_size(moe_dtype dt, moe_act act, int64_t s, int m, int e, int k,
                                int64_t c_max, int h) {
    size_t a = moe_capacity_workspace_size(s, e, k);
    size_t b = moe_expert_ffn_workspace_size(dt, act, e, c_max, m, h);
    if (a == 0 || b == 0) return 0;
    return up256(a) + up256(b);
}

moe_status moe_layer_forward(const void *x, moe_dtype dt, const float *wg, const float *gate_bias,
                             const void *w1, const void *b1, const void *w3, const void *w2,
                             const void *b2, moe_act act, int64_t s, int m, int e, int k, int h,
                             float capacity_factor, int64_t c_max, unsigned flags, int32_t *idx,
                             float *gates, int32_t *loc, int32_t *counts, int32_t *c_dev,
                             void *buf, void *out, void *y, void *workspace,
                             size_t workspace_bytes, int32_t *dev_status, void *stream) {
    size_t need = moe_layer_workspace_size(dt, act, s, m, e, k, c_max, h);
    if (need == 0 || workspace_bytes < need || !ok16(workspace)) return MOE_ERR_INVALID_ARG;
    size_t cap_b = up256(moe_capacity_workspace_size(s, e, k));
    char *ws = (char *)workspace;
    moe_status st;
    st = moe_gate_topk(x, dt, wg, gate_bias, s, m, e, k, flags & MOE_FLAG_NORMALIZE_GATES, idx,
                       gates, dev_status, stream);
    if (st != MOE_OK) return st;
    st = moe_capacity_locations(idx, s, e, k, capacity_factor, c_max, ws, cap_b, loc, counts, c_dev,
                                dev_status, stream);
    if (st != MOE_OK) return st;
    st = moe_encode(x, dt, idx, loc, counts, c_dev, s, m, e, k, c_max, flags & MOE_FLAG_ZERO_FILL,
                    buf, dev_status, stream);
    if (st != MOE_OK) return st;
    st = moe_expert_ffn(buf, dt, counts, c_dev, w1, b1, w3, w2, b2, act, e, c_max, m, h,
                        ws + cap_b, workspace_bytes - cap_b, out, dev_status, stream);
    if (st != MOE_OK) return st;
    return moe_decode(out, dt, idx, loc, gates, c_dev, s, m, e, k, c_max, y, dev_status, stream);
}

moe_status moe_layer_forward_host(const void *x_host, void *y_host, const void *x, moe_dtype dt,
                                  const float *wg, const float *gate_bias, const void *w1,
                                  const void *b1, const void *w3, const void *w2, const void *b2,
                                  moe_act act, int64_t s, int m, int e, int k, int h,
                                  float capacity_factor, int64_t c_max, unsigned flags,
                                  int32_t *idx, float *gates, int32_t *loc, int32_t *counts,
                                  int32_t *c_dev, void *buf, void *out, void *y, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status, void *stream) {
    if (x_host == nullptr || y_host == nullptr || !valid_dt(dt) || s < 1 || m < 1 || !ok16(x) ||
        !ok16(y))
        return MOE_ERR_INVALID_ARG;
    if (moe_layer_workspace_size(dt, act, s, m, e, k, c_max, h) == 0) return MOE_ERR_INVALID_ARG;
    const size_t bytes = (size_t)s * (size_t)m * esize(dt);
    cudaStream_t st = as_stream(stream);
    if (cudaMemcpyAsync(const_cast<void *>(x), x_host, bytes, cudaMemcpyHostToDevice, st) !=
        cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    moe_status r = moe_layer_forward(x, dt, wg, gate_bias, w1, b1, w3, w2, b2, act, s, m, e, k, h,
                                     capacity_factor, c_max, flags, idx, gates, loc, counts,
                                     c_dev, buf, out, y, workspace, workspace_bytes, dev_status,
                                     stream);
    if (r != MOE_OK) return r;
    if (cudaMemcpyAsync(y_host, y, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status moe_layer_forward_pipelined(const void *x, moe_dtype dt, const float *wg,
                                       const float *gate_bias, const void *w1, const void *b1,
                                       const void *w3, const void *w2, const void *b2, moe_act act,
                                       int64_t s, int m, int e, int k, int h, float capacity_factor,
                                       int64_t c_max, unsigned flags, int32_t *idx, float *gates,
                                       int32_t *loc, int32_t *counts, int32_t *c_dev, void *buf,
                                       void *out, void *y, void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, int chunks, void *stream,
                                       void *aux_stream, void *const *events) {
    if (chunks < 1 || chunks > 64 || events == nullptr) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i <= chunks; i++)
        if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
    if (dt != MOE_BF16 || chunks == 1)
        return moe_layer_forward(x, dt, wg, gate_bias, w1, b1, w3, w2, b2, act, s, m, e, k, h,
                                 capacity_factor, c_max, flags, idx, gates, loc, counts, c_dev, buf,
                                 out, y, workspace, workspace_bytes, dev_status, stream);
    size_t need = moe_layer_workspace_size(dt, act, s, m, e, k, c_max, h);
    if (need == 0 || workspace_bytes < need || !ok16(workspace)) return MOE_ERR_INVALID_ARG;
    // every stage's own checks, by the calls below, before anything is launched
    if (!routing_shape_ok(s, e, k) || !rows_ok(dt, m) || !rows_ok(dt, h) || c_max < 1 ||
        c_max > 0x7fffffff || !ok16(x) || !ok16(wg) || !opt16(gate_bias) || !ok4(idx) ||
        !ok4(gates) || !ok4(loc) || !ok4(counts) || !ok4(c_dev) || !ok16(buf) || !ok16(out) ||
        !ok16(y) || !ok4(dev_status) || !ok16(w1) || !ok16(w2) || !opt16(b1) || !opt16(b2) ||
        (flags & ~3u) || (act != MOE_ACT_RELU && act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU) ||
        (act == MOE_ACT_SWIGLU && (!ok16(w3) || b1 != nullptr || b2 != nullptr)))
        return MOE_ERR_INVALID_ARG;
    if (e > 256 || !ffn_tc_supported(e, c_max, m, h)) return MOE_ERR_UNSUPPORTED;
    const size_t cap_b = up256(moe_capacity_workspace_size(s, e, k));
    char *ws = (char *)workspace;
    cudaStream_t st = as_stream(stream), aux = as_stream(aux_stream);
    cudaEvent_t *ev = (cudaEvent_t *)events;
    moe_status r;
    r = moe_gate_topk(x, dt, wg, gate_bias, s, m, e, k, flags & MOE_FLAG_NORMALIZE_GATES, idx, gates,
                      dev_status, stream);
    if (r != MOE_OK) return r;
    r = moe_capacity_locations(idx, s, e, k, capacity_factor, c_max, ws, cap_b, loc, counts, c_dev,
                               dev_status, stream);
    if (r != MOE_OK) return r;
    if (cudaEventRecord(ev[0], st) != cudaSuccess || cudaStreamWaitEvent(aux, ev[0], 0) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    // slot chunks [lo, hi) of the expert buffer, in whole 256-row FFN tiles
    const int64_t step = ((c_max + chunks - 1) / chunks + 255) / 256 * 256;
    for (int i = 0; i < chunks; i++) {
        const int64_t lo = (int64_t)i * step, hi = lo + step;
        if (lo >= c_max) break;
        const int ihi = hi >= c_max ? 0x7fffffff : (int)hi;
        // encode of chunk i on the side stream (zero fill, if asked, with the first)
        r = encode_launch(x, dt, idx, loc, counts, c_dev, s, m, e, k, c_max,
                          i == 0 ? (flags & MOE_FLAG_ZERO_FILL) : 0u, buf, dev_status, aux, (int)lo,
                          ihi);
        if (r != MOE_OK) return r;
        if (cudaEventRecord(ev[1 + i], aux) != cudaSuccess ||
            cudaStreamWaitEvent(st, ev[1 + i], 0) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        // the FFN of chunk i on the main stream, while chunk i+1 is encoded
        r = ffn_tc_launch(buf, counts, c_dev, w1, b1, w3, w2, b2, act, e, c_max, m, h, ws + cap_b,
                          out, dev_status, st, (int)lo, hi >= c_max ? 0 : (int)hi);
        if (r != MOE_OK) return r;
    }
    return moe_decode(out, dt, idx, loc, gates, c_dev, s, m, e, k, c_max, y, dev_status, stream);
}

size_t moe_expert_ffn_fp8_workspace_size(int e, int64_t c_max, int m, int h) {
    if (e < 1 || e > kMaxE || c_max < 1 || m < 16 || h < 16 || m % 16 || h % 16) return 0;
    const int64_t rows = (int64_t)e * c_max;
    return up256((size_t)rows * h * 2) + up256((size_t)rows * h) + up256((size_t)rows * 4);
}

moe_status moe_quantize_rows_fp8(const void *src, int64_t batches, int64_t rows_per_batch,
                                 int cols, const int32_t *counts, const int32_t *c_dev, void *q,
                                 float *scale, int32_t *dev_status, void *stream) {
    if (batches < 1 || batches > 0x7fffffff || rows_per_batch < 1 || cols < 16 || cols % 16 ||
        batches * rows_per_batch > ((int64_t)1 << 40) || !ok16(src) || !ok16(q) || !ok4(scale) ||
        !ok4(dev_status) || (counts == nullptr) != (c_dev == nullptr) ||
        (counts && (!ok4(counts) || !ok4(c_dev))))
        return MOE_ERR_INVALID_ARG;
    return quantize_rows_fp8_launch(src, batches, rows_per_batch, cols, counts, c_dev, q, scale,
                                    dev_status, as_stream(stream));
}

moe_status moe_expert_ffn_fp8(const void *buf_q, const float *buf_scale, const int32_t *counts,
                              const int32_t *c_dev, const void *w1_q, const float *w1_scale,
                              const void *b1, const void *w2_q, const float *w2_scale,
                              const void *b2, moe_act act, int e, int64_t c_max, int m, int h,
                              void *workspace, size_t workspace_bytes, void *out,
                              int32_t *dev_status, void *stream) {
    const size_t need = moe_expert_ffn_fp8_workspace_size(e, c_max, m, h);
    if (need == 0 || c_max > 0x7fffffff || !ok16(buf_q) || !ok4(buf_scale) || !ok4(counts) ||
        !ok4(c_dev) || !ok16(w1_q) || !ok16(w1_scale) || !opt16(b1) || !ok16(w2_q) ||
        !ok16(w2_scale) || !opt16(b2) || !ok16(workspace) || workspace_bytes < need ||
        !ok16(out) || !ok4(dev_status))
        return MOE_ERR_INVALID_ARG;
    if (act != MOE_ACT_RELU && act != MOE_ACT_GELU) return MOE_ERR_UNSUPPORTED;
    if (!ffn_tc_supported(e, c_max, m, h)) return MOE_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)e * c_max;
    char *w = (char *)workspace;
    void *hid = w;
    void *hid_q = w + up256((size_t)rows * h * 2);
    float *hid_scale = (float *)(w + up256((size_t)rows * h * 2) + up256((size_t)rows * h));
    return ffn_tc_fp8_launch(buf_q, buf_scale, counts, c_dev, w1_q, w1_scale, b1, w2_q, w2_scale, b2,
                             act, e, c_max, m, h, hid, hid_q, hid_scale, out, dev_status,
                             as_stream(stream));
}

moe_status moe_probe_fp32_fma(int packed, int blocks, int iters, float *out, void *stream) {
    if (blocks < 1 || iters < 1 || !ok4(out)) return MOE_ERR_INVALID_ARG;
    return probe_fp32_fma_launch(packed, blocks, iters, out, as_stream(stream));
}

}  // extern "C"
