// Expert FFN on the SIMT cores (fp32 layers only).
//
// Method: the Tutel profile's experts {'type': 'ffn', hidden_size_per_expert,
// has_fc1_bias, has_fc2_bias} and the DeepSpeed-MoE vs Tutel blog, section 3.5
// (experts run as a batched matmul over the (E, C, D) buffer).  Each launch is
// a grouped GEMM C[j] = A[j] B[j]^T over experts j, restricted to the first
// min(counts[j], c) rows of A[j]; both operands are K-contiguous.  fp32 layers
// stay on fp32 fused multiply-adds so that results meet an fp32 tolerance
// (tf32 tensor cores would not).
#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = 32, BN = 64, BK = 32, SNT = 256;  // 8 outputs per thread

enum Epi { EPI_ACT = 0, EPI_SWIGLU = 1, EPI_OUT = 2 };

__device__ __forceinline__ float gelu_erf(float a) { return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f)); }
__device__ __forceinline__ float silu(float a) { return a / (1.0f + expf(-a)); }

template <typename T> __device__ __forceinline__ float ldf(const T *p);
template <> __device__ __forceinline__ float ldf<float>(const float *p) { return *p; }
template <typename T> __device__ __forceinline__ T stf(float v);
template <> __device__ __forceinline__ float stf<float>(float v) { return v; }

// A: [e, c_max, K] rows; B, B3: [e, N, K]; bias [e, N]; C: [e, c_max, N].
template <typename T, int EPI>
__global__ void __launch_bounds__(SNT)
simt_group_gemm(const T *__restrict__ A, const T *__restrict__ B, const T *__restrict__ B3,
                const T *__restrict__ bias, const int32_t *__restrict__ counts,
                const int32_t *__restrict__ c_dev, int64_t c_max, int N, int K, int act,
                T *__restrict__ C, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    const int j = blockIdx.z;
    const int c_eff = (int)min((int64_t)*c_dev, c_max);
    const int rows = min(counts[j], c_eff);
    const int r0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    if (r0 >= rows) return;
    __shared__ float As[BK][BM + 1];
    __shared__ float Bs[BK][BN + 1];
    __shared__ float B3s[EPI == EPI_SWIGLU ? BK : 1][BN + 1];
    const int tid = threadIdx.x;
    const int tn = tid % (BN / 4), tm = tid / (BN / 4);  // 16 x 16 threads: 2 rows x 4 cols each
    float acc[2][4] = {}, acc3[2][4] = {};
    const T *Aj = A + (int64_t)j * c_max * K;
    const T *Bj = B + (int64_t)j * N * K;
    const T *B3j = EPI == EPI_SWIGLU ? B3 + (int64_t)j * N * K : nullptr;
    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int q = tid; q < BM * BK; q += SNT) {
            int r = q / BK, kk = q % BK;
            As[kk][r] = (r0 + r < rows && k0 + kk < K) ? ldf(Aj + (int64_t)(r0 + r) * K + k0 + kk) : 0.0f;
        }
        for (int q = tid; q < BN * BK; q += SNT) {
            int n = q / BK, kk = q % BK;
            bool ok = n0 + n < N && k0 + kk < K;
            Bs[kk][n] = ok ? ldf(Bj + (int64_t)(n0 + n) * K + k0 + kk) : 0.0f;
            if (EPI == EPI_SWIGLU) B3s[kk][n] = ok ? ldf(B3j + (int64_t)(n0 + n) * K + k0 + kk) : 0.0f;
        }
        __syncthreads();
        const int klim = min(BK, K - k0);
        for (int kk = 0; kk < klim; kk++) {
#pragma unroll
            for (int a = 0; a < 2; a++) {
                float av = As[kk][tm * 2 + a];
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    acc[a][b] = fmaf(av, Bs[kk][tn * 4 + b], acc[a][b]);
                    if (EPI == EPI_SWIGLU) acc3[a][b] = fmaf(av, B3s[kk][tn * 4 + b], acc3[a][b]);
                }
            }
        }
        __syncthreads();
    }
    T *Cj = C + (int64_t)j * c_max * N;
#pragma unroll
    for (int a = 0; a < 2; a++) {
        int r = r0 + tm * 2 + a;
        if (r >= rows) continue;
#pragma unroll
        for (int b = 0; b < 4; b++) {
            int n = n0 + tn * 4 + b;
            if (n >= N) continue;
            float v = acc[a][b];
            if (EPI == EPI_SWIGLU) {
                v = silu(v) * acc3[a][b];
            } else {
                if (bias) v += ldf(bias + (int64_t)j * N + n);
                if (EPI == EPI_ACT) v = act == MOE_ACT_RELU ? fmaxf(v, 0.0f) : gelu_erf(v);
            }
            Cj[(int64_t)r * N + n] = stf<T>(v);
        }
    }
}

template <typename T>
moe_status run(const void *buf, const int32_t *counts, const int32_t *c_dev, const void *w1,
               const void *b1, const void *w3, const void *w2, const void *b2, moe_act act, int e,
               int64_t c_max, int m, int h, void *hid, void *out, int32_t *st, cudaStream_t stream) {
    int64_t gy = (c_max + BM - 1) / BM;
    if (gy > 65535 || e > 65535) return MOE_ERR_UNSUPPORTED;
    dim3 g1((h + BN - 1) / BN, (unsigned)gy, e);
    const T *none = nullptr;
    moe_status r;
    if (act == MOE_ACT_SWIGLU)
        r = launch_pdl(simt_group_gemm<T, EPI_SWIGLU>, g1, dim3(SNT), 0, stream, (const T *)buf,
                       (const T *)w1, (const T *)w3, none, counts, c_dev, c_max, h, m, (int)act,
                       (T *)hid, st);
    else
        r = launch_pdl(simt_group_gemm<T, EPI_ACT>, g1, dim3(SNT), 0, stream, (const T *)buf,
                       (const T *)w1, none, (const T *)b1, counts, c_dev, c_max, h, m, (int)act,
                       (T *)hid, st);
    if (r != MOE_OK) return r;
    dim3 g2((m + BN - 1) / BN, (unsigned)gy, e);
    return launch_pdl(simt_group_gemm<T, EPI_OUT>, g2, dim3(SNT), 0, stream, (const T *)hid,
                      (const T *)w2, none, (const T *)b2, counts, c_dev, c_max, m, h, (int)act,
                      (T *)out, st);
}

}  // namespace

moe_status ffn_simt_launch(const void *buf, moe_dtype dt, const int32_t *counts,
                           const int32_t *c_dev, const void *w1, const void *b1, const void *w3,
                           const void *w2, const void *b2, moe_act act, int e, int64_t c_max,
                           int m, int h, void *hid, void *out, int32_t *st, cudaStream_t stream) {
    if (dt != MOE_F32) return MOE_ERR_UNSUPPORTED;  // bf16 layers run on the tensor cores
    return run<float>(buf, counts, c_dev, w1, b1, w3, w2, b2, act, e, c_max, m, h, hid, out, st,
                      stream);
}

}  // namespace moe
