// Shared device/host helpers of the MoE layer kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_gate.h"

namespace moe {

// ---------------------------------------------------------------- launches

// Count of kernels launched by this library (exported by moe_launch_count).
void note_launch();

// True (and one fewer pending) while moe_debug_stall_gemms has stalls pending:
// the tensor-core GEMM launch being prepared then issues no operand copies.
bool take_gemm_stall();

inline moe_status launch_status() {
    cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while its predecessor in the stream drains; it must call
// pdl_enter() before touching anything the predecessor writes.
template <typename... KArgs, typename... Args>
moe_status launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    note_launch();
    if (err != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

// launch_pdl for a kernel launched in clusters of `cl` CTAs along x
// (gridDim.x a multiple of cl).
template <typename... KArgs, typename... Args>
moe_status launch_cluster_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, int cl,
                              cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    note_launch();
    if (err != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

// Wait until the previous kernel in the stream has completed and its writes
// are visible (no-op when launched without programmatic serialization), then
// let the next kernel start its own launch early.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The two halves of pdl_enter, for a kernel that reads nothing its
// predecessor writes: it lets its successor launch at once, runs alongside
// its predecessor, and waits for it (pdl_wait) before it exits, so that its
// own completion still implies its predecessor's.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------ device status

// First error wins; later errors are dropped.
__device__ __forceinline__ void set_status(int32_t *st, int32_t code) {
    if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ bool status_bad(const int32_t *st) {
    return st && *(volatile const int32_t *)st != 0;
}

// ----------------------------------------------------------------- vectors

struct alignas(16) V16 { uint32_t w[4]; };  // 16 bytes: 8 bf16 or 4 fp32

__device__ __forceinline__ V16 ld_stream(const void *p) {
    V16 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]) : "l"(p));
    return v;
}

__device__ __forceinline__ V16 ld_v16(const void *p) {
    V16 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v16(void *p, const V16 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]) : "memory");
}

// Streaming store (evict-first): for outputs nobody reads back soon.
__device__ __forceinline__ void st_v16_cs(void *p, const V16 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]) : "memory");
}

// Asynchronous global -> shared copies (cp.async): `valid` false copies
// nothing and zero-fills the destination (gmem must still be a valid address).
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
// This thread's copies of all but the newest N committed groups have landed.
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// bf16 <-> fp32.  Widening is exact (bit shift).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16 bits, round to nearest even (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint32_t f2bf(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    return f2bf(lo) | (f2bf(hi) << 16);
}

// Element-type traits: 16-byte chunk = VEC elements.
template <typename T> struct Elt;
template <> struct Elt<float> {
    static constexpr int VEC = 4;
    static constexpr int BYTES = 4;
    __device__ __forceinline__ static void unpack(const V16 &v, float *f) {
#pragma unroll
        for (int i = 0; i < 4; i++) f[i] = __uint_as_float(v.w[i]);
    }
    __device__ __forceinline__ static V16 pack(const float *f) {
        V16 v;
#pragma unroll
        for (int i = 0; i < 4; i++) v.w[i] = __float_as_uint(f[i]);
        return v;
    }
};
template <> struct Elt<__nv_bfloat16> {
    static constexpr int VEC = 8;
    static constexpr int BYTES = 2;
    __device__ __forceinline__ static void unpack(const V16 &v, float *f) {
#pragma unroll
        for (int i = 0; i < 4; i++) { f[2 * i] = bf16lo(v.w[i]); f[2 * i + 1] = bf16hi(v.w[i]); }
    }
    __device__ __forceinline__ static V16 pack(const float *f) {
        V16 v;
#pragma unroll
        for (int i = 0; i < 4; i++) v.w[i] = pack_bf16(f[2 * i], f[2 * i + 1]);
        return v;
    }
};

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace moe
