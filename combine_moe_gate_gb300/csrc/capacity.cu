// Capacity and slot locations.
//
// Method: the DeepSpeed-MoE vs Tutel blog, section 1.4 (slot assignment is a
// cumsum over the token-to-expert table, parallelised as a scan) and section
// 3.5 (dynamic capacity factor: fixed / adaptive no-drop / capped adaptive),
// with the Tutel profile's FAQ on capacity_factor.  Priority order: all
// tokens' route 0 in token order, then route 1, and so on; the location of a
// route is its rank among the routes that chose the same expert, so the flat
// route-major table [k, s] is ranked in its natural order.
//
// Small tables (up to 16384 routes, e <= 256) take one launch of up to 16 CTAs
// (cap_small_kernel); otherwise two launches, no inter-CTA waiting:
//   1. cap_hist: CTA b counts the experts of its chunk of CH routes -> hist[b][e].
//   2. cap_assign: CTA b sums hist[0..b-1][j] for its base offsets, ranks its
//      chunk stably (warps take consecutive segments; inside a warp
//      __match_any_sync groups equal experts and popc of the lower lanes gives
//      the rank), then adds the per-warp prefix.  CTA 0 also forms counts[],
//      the capacity c and the overflow check.
#include <cuda.h>

#include <mutex>
#include <utility>

#include "common.cuh"

namespace moe {
namespace {

constexpr int CAP_NT = 256;            // threads per CTA
constexpr int CAP_NW = CAP_NT / 32;    // warps per CTA
constexpr int CAP_CH = 4096;           // routes per chunk (per CTA)
constexpr int CAP_SEG = CAP_CH / CAP_NW;  // routes per warp
constexpr int CAP_ROUNDS = CAP_SEG / 32;

__global__ void __launch_bounds__(CAP_NT)
cap_hist_kernel(const int32_t *__restrict__ idx, int64_t n, int e, int32_t *__restrict__ hist,
                int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    extern __shared__ int32_t h[];
    for (int j = threadIdx.x; j < e; j += CAP_NT) h[j] = 0;
    __syncthreads();
    const int64_t base = (int64_t)blockIdx.x * CAP_CH;
    constexpr int PER = CAP_CH / CAP_NT;
    int v[PER];
#pragma unroll
    for (int i = 0; i < PER; i++) {  // all loads in flight before any atomic
        int64_t j = base + threadIdx.x + (int64_t)i * CAP_NT;
        v[i] = j < n ? __ldg(idx + j) : -2;
    }
#pragma unroll
    for (int i = 0; i < PER; i++) {
        if ((unsigned)v[i] < (unsigned)e) atomicAdd(&h[v[i]], 1);
        else if (v[i] != -2) set_status(status, MOE_ERR_INVALID_ARG);
    }
    __syncthreads();
    for (int j = threadIdx.x; j < e; j += CAP_NT) hist[(int64_t)blockIdx.x * e + j] = h[j];
}

// c_fixed >= 0: capacity fixed on the host (capacity_factor > 0).
// Otherwise c = min(c_cap, max_j counts[j]) (c_cap = INT_MAX for factor 0).
__global__ void __launch_bounds__(CAP_NT)
cap_assign_kernel(const int32_t *__restrict__ idx, int64_t n, int e, int nblk,
                  const int32_t *__restrict__ hist, int c_fixed, int c_cap, int64_t c_max,
                  int32_t *__restrict__ loc, int32_t *__restrict__ counts,
                  int32_t *__restrict__ c_dev, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    extern __shared__ int32_t sm[];
    int32_t *wcnt = sm;                 // [NW][e]: per-warp counts, then per-warp offsets
    int32_t *base = sm + CAP_NW * e;    // [e]
    __shared__ int32_t s_max;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_max = 0;
    for (int j = tid; j < CAP_NW * e; j += CAP_NT) wcnt[j] = 0;
    for (int j = tid; j < e; j += CAP_NT) {
        int32_t b = 0;
        for (int q = 0; q < (int)blockIdx.x; q++) b += hist[(int64_t)q * e + j];
        base[j] = b;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int j = tid; j < e; j += CAP_NT) {
            int32_t tot = 0;
            for (int q = 0; q < nblk; q++) tot += hist[(int64_t)q * e + j];
            counts[j] = tot;
            atomicMax(&s_max, tot);
        }
        __syncthreads();
        if (tid == 0) {
            int c = c_fixed >= 0 ? c_fixed : min(c_cap, s_max);
            c_dev[0] = c;
            if ((int64_t)c > c_max) set_status(status, MOE_ERR_CAPACITY);
        }
    }

    // stable rank inside this warp's segment
    const int64_t seg0 = (int64_t)blockIdx.x * CAP_CH + (int64_t)warp * CAP_SEG;
    int32_t rank[CAP_ROUNDS];
    int32_t val[CAP_ROUNDS];
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int rd = 0; rd < CAP_ROUNDS; rd++) {  // all loads in flight first
        int64_t j = seg0 + rd * 32 + lane;
        int v = j < n ? __ldg(idx + j) : -1;
        val[rd] = (unsigned)v < (unsigned)e ? v : -1;
    }
#pragma unroll
    for (int rd = 0; rd < CAP_ROUNDS; rd++) {
        const int v = val[rd];
        unsigned peers = __match_any_sync(0xffffffffu, v);
        int prev = v >= 0 ? wcnt[warp * e + v] : 0;
        __syncwarp();
        if (v >= 0 && (peers & lt) == 0) wcnt[warp * e + v] = prev + __popc(peers);
        __syncwarp();
        rank[rd] = prev + __popc(peers & lt);
    }
    __syncthreads();
    // exclusive prefix over warps, seeded with the chunk's base offset
    for (int j = tid; j < e; j += CAP_NT) {
        int32_t run = base[j];
        for (int w = 0; w < CAP_NW; w++) {
            int32_t t = wcnt[w * e + j];
            wcnt[w * e + j] = run;
            run += t;
        }
    }
    __syncthreads();
#pragma unroll
    for (int rd = 0; rd < CAP_ROUNDS; rd++) {
        int64_t j = seg0 + rd * 32 + lane;
        if (j < n && val[rd] >= 0) loc[j] = wcnt[warp * e + val[rd]] + rank[rd];
    }
}

// Small route tables (n <= 16 chunks of CAPS_CH routes, e <= 256): one launch
// of ceil(n / CAPS_CH) CTAs with no inter-CTA waiting.  CTA b histograms the
// routes of all earlier chunks itself (redundant, but at most 15 chunks) for
// its base offsets, then ranks its own chunk stably as cap_assign does.  The
// last CTA, which has seen every route, writes counts[], c and the overflow
// status.
constexpr int CAPS_NT = 1024, CAPS_NW = CAPS_NT / 32, CAPS_CH = 1024, CAPS_MAXE = 256;
constexpr int CAPS_ROUNDS = CAPS_CH / CAPS_NT;   // routes per thread (own chunk)
constexpr int CAPS_MAXBLK = 16;

__global__ void __launch_bounds__(CAPS_NT)
cap_small_kernel(const int32_t *__restrict__ idx, int64_t n, int e, int c_fixed, int c_cap,
                 int64_t c_max, int32_t *__restrict__ loc, int32_t *__restrict__ counts,
                 int32_t *__restrict__ c_dev, int32_t *status) {
    pdl_enter();
    if (status_bad(status)) return;
    __shared__ int32_t base[CAPS_MAXE];
    __shared__ int32_t wcnt[CAPS_NW][CAPS_MAXE];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int q = tid; q < CAPS_MAXE; q += CAPS_NT) base[q] = 0;
    for (int q = tid; q < CAPS_NW * CAPS_MAXE; q += CAPS_NT) (&wcnt[0][0])[q] = 0;
    // own chunk: warp w takes routes [w*32*R, (w+1)*32*R) of it, R = CAPS_ROUNDS rounds of 32
    const int64_t seg0 = (int64_t)blockIdx.x * CAPS_CH + warp * 32 * CAPS_ROUNDS;
    int32_t val[CAPS_ROUNDS], rank[CAPS_ROUNDS];
#pragma unroll
    for (int rd = 0; rd < CAPS_ROUNDS; rd++) {
        const int64_t j = seg0 + rd * 32 + lane;
        const int v = j < n ? __ldg(idx + j) : -1;
        if (j < n && (unsigned)v >= (unsigned)e) set_status(status, MOE_ERR_INVALID_ARG);
        val[rd] = (unsigned)v < (unsigned)e ? v : -1;
    }
    __syncthreads();
    // earlier chunks: warp-aggregated histogram into base[]
    const int64_t pre = (int64_t)blockIdx.x * CAPS_CH;
    for (int64_t q0 = 0; q0 < pre; q0 += CAPS_NT * 8) {
        int v8[8];
#pragma unroll
        for (int b = 0; b < 8; b++) {
            const int64_t q = q0 + b * CAPS_NT + tid;
            const int v = q < pre ? __ldg(idx + q) : -1;
            v8[b] = (unsigned)v < (unsigned)e ? v : -1;
        }
#pragma unroll
        for (int b = 0; b < 8; b++) {
            const unsigned peers = __match_any_sync(0xffffffffu, v8[b]);
            if (v8[b] >= 0 && (peers & ((1u << lane) - 1u)) == 0)
                atomicAdd(&base[v8[b]], __popc(peers));
        }
    }
    // own chunk: stable ranks inside each warp's segment
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int rd = 0; rd < CAPS_ROUNDS; rd++) {
        const int v = val[rd];
        const unsigned peers = __match_any_sync(0xffffffffu, v);
        const int prev = v >= 0 ? wcnt[warp][v] : 0;
        __syncwarp();
        if (v >= 0 && (peers & lt) == 0) wcnt[warp][v] = prev + __popc(peers);
        __syncwarp();
        rank[rd] = prev + __popc(peers & lt);
    }
    __syncthreads();
    const bool last = blockIdx.x == gridDim.x - 1;
    __shared__ int32_t s_max;
    if (tid == 0) s_max = 0;
    __syncthreads();
    for (int x = tid; x < e; x += CAPS_NT) {
        int32_t run = base[x];
        for (int w = 0; w < CAPS_NW; w++) {
            const int32_t c = wcnt[w][x];
            wcnt[w][x] = run;
            run += c;
        }
        if (last) {
            counts[x] = run;
            atomicMax(&s_max, run);
        }
    }
    __syncthreads();
    if (last && tid == 0) {
        const int c = c_fixed >= 0 ? c_fixed : min(c_cap, s_max);
        c_dev[0] = c;
        if ((int64_t)c > c_max) set_status(status, MOE_ERR_CAPACITY);
    }
#pragma unroll
    for (int rd = 0; rd < CAPS_ROUNDS; rd++) {
        const int64_t j = seg0 + rd * 32 + lane;
        if (j < n && val[rd] >= 0) loc[j] = wcnt[warp][val[rd]] + rank[rd];
    }
}

int64_t ceil_div_exact(double x, int e) {
    int64_t c = (int64_t)ceil(x / (double)e);
    while (c > 0 && (double)(c - 1) * (double)e >= x) c--;
    while ((double)c * (double)e < x) c++;
    return c;
}

}  // namespace

int64_t capacity_bound_host(float f, int64_t s, int e, int k) {
    if (f > 0.0f) return ceil_div_exact((double)f * (double)k * (double)s, e);
    if (f == 0.0f) return s;
    int64_t b = ceil_div_exact(-(double)f * (double)k * (double)s, e);
    return b < s ? b : s;
}

size_t capacity_workspace_bytes(int64_t s, int e, int k) {
    int64_t n = s * (int64_t)k;
    int64_t nblk = (n + CAP_CH - 1) / CAP_CH;
    size_t b = (size_t)nblk * (size_t)e * sizeof(int32_t);
    return (b + 255) & ~(size_t)255;
}

moe_status capacity_launch(const int32_t *idx, int64_t s, int e, int k, float f, int64_t c_max,
                           void *ws, int32_t *loc, int32_t *counts, int32_t *c_dev, int32_t *st,
                           cudaStream_t stream) {
    const int64_t n = s * (int64_t)k;
    const int64_t nblk = (n + CAP_CH - 1) / CAP_CH;
    if (nblk > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
    int c_fixed = -1, c_cap = 0x7fffffff;
    if (f > 0.0f) {
        int64_t c = capacity_bound_host(f, s, e, k);
        c_fixed = (int)(c < 0x7fffffff ? c : 0x7fffffff);
    } else if (f < 0.0f) {
        int64_t c = capacity_bound_host(f, s, e, k);
        c_cap = (int)c;
    }
    if (e <= CAPS_MAXE && n <= (int64_t)CAPS_CH * CAPS_MAXBLK) {
        const unsigned nb = (unsigned)((n + CAPS_CH - 1) / CAPS_CH);
        return launch_pdl(cap_small_kernel, dim3(nb), dim3(CAPS_NT), 0, stream, idx, n, e, c_fixed,
                          c_cap, c_max, loc, counts, c_dev, st);
    }
    int32_t *hist = (int32_t *)ws;
    if (launch_pdl(cap_hist_kernel, dim3((unsigned)nblk), dim3(CAP_NT), e * sizeof(int32_t), stream,
                   idx, n, e, hist, st) != MOE_OK)
        return MOE_ERR_CUDA;
    size_t smem = (size_t)(CAP_NW + 1) * e * sizeof(int32_t);
    auto kern = cap_assign_kernel;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_pdl(kern, dim3((unsigned)nblk), dim3(CAP_NT), smem, stream, idx, n, e, (int)nblk,
                      hist, c_fixed, c_cap, c_max, loc, counts, c_dev, st);
}

// ------------------------------------------------------ no-allocation variant
//
// Scratch for moe_capacity_locations_noalloc: a fixed array in the library's
// own device memory, so callers that cannot allocate device memory still get
// the two-kernel capacity path.  Every GPU that loads the library holds these
// 1 MiB until the process exits.  All calls share the array: calls whose
// kernels overlap on the GPU (different streams, no ordering) race on it.
// The histogram kernel writes every entry the assign kernel reads, so nothing
// has to be cleared between calls.
constexpr size_t NOALLOC_SCRATCH_BYTES = MOE_CAPACITY_NOALLOC_SCRATCH_BYTES;
static_assert(NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");
static __device__ __align__(256) int32_t g_cap_scratch[NOALLOC_SCRATCH_BYTES / sizeof(int32_t)];

namespace {

// Identity of the CUDA context current on this thread (cuCtxGetId: unique for
// the life of the process, so a context created after cudaDeviceReset gets a
// new one).  The driver entry points are fetched through the runtime; false
// if either is unavailable or no context is current.
bool current_context_id(unsigned long long *id) {
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static const auto fns = [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault,
                                             &qa) != cudaSuccess ||
            qa != cudaDriverEntryPointSuccess)
            a = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
                cudaSuccess ||
            qb != cudaDriverEntryPointSuccess)
            b = nullptr;
        cudaGetLastError();
        return std::make_pair(reinterpret_cast<GetCurrent>(a), reinterpret_cast<GetId>(b));
    }();
    CUcontext ctx = nullptr;
    if (!fns.first || !fns.second || fns.first(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return fns.second(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_cap_scratch on the current device.  In host code the
// symbol name is only a host-side stand-in, so the address is looked up with
// the device current: once per device and context (the cache is keyed on the
// context's identity, so a reset device, whose module is loaded again into a
// new context, gets a fresh lookup), or on every call when the context's
// identity cannot be read.
int32_t *cap_scratch_on_current_device() {
    static std::mutex mu;
    static int32_t *addr[64] = {nullptr};
    static unsigned long long ctx_of[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    unsigned long long id = 0;
    if (addr[dev] && current_context_id(&id) && id == ctx_of[dev]) return addr[dev];
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_cap_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return nullptr;
    }
    // the lookup makes the device's primary context current if none was
    if (current_context_id(&id)) {
        addr[dev] = static_cast<int32_t *>(p);
        ctx_of[dev] = id;
    } else {
        addr[dev] = nullptr;
    }
    return static_cast<int32_t *>(p);
}

}  // namespace

moe_status capacity_noalloc_launch(const int32_t *idx, int64_t s, int e, int k, float f,
                                   int64_t c_max, int32_t *loc, int32_t *counts, int32_t *c_dev,
                                   int32_t *st, cudaStream_t stream) {
    if (capacity_workspace_bytes(s, e, k) > NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
    int32_t *scratch = cap_scratch_on_current_device();
    if (!scratch) return MOE_ERR_CUDA;
    return capacity_launch(idx, s, e, k, f, c_max, scratch, loc, counts, c_dev, st, stream);
}

}  // namespace moe
