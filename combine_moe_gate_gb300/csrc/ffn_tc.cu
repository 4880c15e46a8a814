// Expert FFN and its backward on the 5th-generation tensor cores (bf16 and e4m3 layers).
//
// Method: the Tutel profile's experts {'type': 'ffn', hidden_size_per_expert,
// has_fc1_bias, has_fc2_bias} and the DeepSpeed-MoE vs Tutel blog, section 3.5
// (experts run as one batched matmul over the (E, C, D) expert buffer, whose
// shape does not depend on the routing).  Here that batched matmul is a
// grouped GEMM over experts j, restricted on the device to the first
// min(counts[j], c) rows of expert j: no host synchronisation is needed to
// learn the ragged row counts.
//
//   fc1:  hid[j] = act(buf[j] W1[j]^T + b1[j])        (SwiGLU: silu(buf W1^T) * (buf W3^T))
//   fc2:  out[j] = hid[j] W2[j]^T + b2[j]
//
// One persistent kernel per GEMM on CTA pairs (clusters of 2), one CTA per SM
// (~218 KB of shared memory, 416 threads):
//   warps 0, 10, 11, 12  TMA producers: each stage's A and B tiles arrive as
//               four boxes (128-byte swizzle) into a ring guarded by full/empty
//               mbarriers; a pair's copies complete on the even CTA's barriers;
//   warp 1      allocates all 512 TMEM columns in both CTAs; in the even CTA
//               one lane issues the 2-SM tcgen05.mma (M = 256 over the pair,
//               N = 256; kind::f16 for bf16, kind::f8f6f4 for e4m3) and
//               tcgen05.commit to release stages and publish accumulators;
//   warps 2-9   epilogue: tcgen05.ld 32 lanes x 32 columns, then the mode's
//               arithmetic in fp32 (bias, activation, e4m3 scales, or an
//               activation derivative), one rounding, and TMA stores of 32 x 32
//               bf16 (or 32 x 16 fp32) boxes staged in shared memory.
// Tiles are 256 x 256 with two accumulators (a tile's epilogue overlaps the
// next tile's main loop) or 256 x 512 with one (TN = 2: two N = 256 MMAs
// share each A tile).  Operands are K-major, or MN-major (row-major [K, N]
// weights and activations read in place, for the backward products), and a
// per-expert-K mode contracts each expert over its own kept rows (the weight
// gradients).  Every wait is bounded: after ~1 s a role sets MOE_ERR_TIMEOUT,
// raises a CTA-wide abort flag and leaves its loop; the CTA then drains its
// outstanding copies and MMAs (bounded) and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int UM = 128;                 // UMMA M (rows of one MMA)
constexpr int BN = 256;                 // UMMA N (rows of B per tile)
constexpr int UK = 16;                  // K of one tcgen05.mma kind::f16
constexpr int EPI_WARPS = 8;
// Warps: 0 producer (A, first half of its rows), 1 MMA, 2..9 epilogue, then
// producers (B first half), (A second half), (B second half).  Every stage's
// operands arrive as four boxes of half the rows, in flight side by side, so
// a stage lands sooner than as two boxes.
constexpr int PROD_WARP0 = 2 + EPI_WARPS;
constexpr int NUM_THREADS = (PROD_WARP0 + 3) * 32;
constexpr uint32_t TMEM_COLS = 512;     // all of TMEM
constexpr int MAX_E = 1024;
constexpr unsigned long long WAIT_NS = 1000000000ull;  // 1 s per wait
constexpr int SMEM_RING = 192 * 1024;   // operand ring per CTA

// EPI_BIAS_BMN: the bias epilogue with B read MN-major, straight from a
// row-major [K, N] tensor (the weights of the data-gradient products).
// EPI_WGRAD_MN: the weight-gradient products out[j] = A[j]^T B[j] with both
// operands read MN-major from row-major activations [e * b_rows, M or N]
// (b_rows rows per expert): expert j contracts over its first k_counts[j]
// rows; a last K block that is only partly kept is read from the tail maps
// instead ([e * BK, M or N]: those rows copied, zeros after them), so no
// row past an expert's kept rows is ever read.
// EPI_DGELU / EPI_DRELU: the activation backward fused into the recomputed
// pre-activation: out = d_hid * act'(acc + bias) with d_hid (GemmArgs::aux)
// laid out like out; the pre-activation itself is never stored.
// EPI_GELU_SAVE / EPI_RELU_SAVE: fc1 that also stores the pre-activation
// acc + bias (bf16) to GemmArgs::aux_out, laid out like out.
// EPI_DGELU_BMN / EPI_DRELU_BMN: d_hid = acc (B MN-major) times act'(pre)
// with the saved pre-activation (GemmArgs::aux) laid out like out.
// EPI_WGRAD_MN_F32: EPI_WGRAD_MN writing fp32 to GemmArgs::out_f32.
// EPI_SWIGLU_SAVE: the SwiGLU fc1 that also stores a = buf W1^T and
// b = buf W3^T (bf16) to GemmArgs::aux_out, rows of 2 * n_out: a, then b.
// EPI_DSWIGLU_BMN: d_hid = acc (B MN-major) and the saved [a | b] rows
// (GemmArgs::aux, 2 * n_out a row) give d_a = d_hid * b * silu'(a) into out
// and d_b = d_hid * silu(a) into out + n_out, out rows of GemmArgs::out_pitch.
enum Epi { EPI_GELU = 0, EPI_RELU = 1, EPI_SWIGLU = 2, EPI_BIAS = 3, EPI_BIAS_BMN = 4,
           EPI_WGRAD_MN = 5, EPI_DGELU = 6, EPI_DRELU = 7, EPI_GELU_SAVE = 8, EPI_RELU_SAVE = 9,
           EPI_DGELU_BMN = 10, EPI_DRELU_BMN = 11, EPI_WGRAD_MN_F32 = 12, EPI_SWIGLU_SAVE = 13,
           EPI_DSWIGLU_BMN = 14 };
// The SwiGLU fc1 modes (W1 and W3 rows paired in one N = 256 MMA).
__host__ __device__ constexpr bool is_swiglu(int epi) { return epi == EPI_SWIGLU || epi == EPI_SWIGLU_SAVE; }

// Tile shape.  TM = 1: 128 x 256 tiles, two 256-column accumulators in TMEM so
// the epilogue of one tile overlaps the main loop of the next.  TM = 2:
// 256 x 256 tiles as two M=128 MMAs sharing every B tile (a third fewer operand
// bytes per FLOP), one 512-column accumulator.  CL = 2 (with TM = 1): a CTA pair
// (cluster of 2) computes a 256 x 256 tile with the 2-SM MMA (M = 256): each
// CTA loads its 128 rows of A and one half of the B tile, so each SM moves the
// TM = 2 operand bytes per FLOP while keeping two accumulators for overlap.
// TN = 2 (with CL = 2, TM = 1): the pair tile is 256 x 512
// as two N = 256 MMAs sharing each A tile, one 512-column accumulator per CTA;
// each SM then fills 48 KB of operands per 1024 MMA cycles instead of 32 KB per
// 512 (the fill of shared memory, not L2, is what bounds the ring).
// BK is the K depth of one pipeline stage: 64 bf16 (one 128-byte swizzle row)
// or 32 (64-byte swizzle); the smaller stage doubles the number of stages in
// the same shared memory, i.e. more operand bytes in flight to cover L2/HBM
// latency.
template <int TM, int BK_, int CL_ = 1, int TN_ = 1, int EB_ = 2>
struct Tiling {
    static constexpr int EB = EB_;                        // bytes per operand element (2 bf16, 1 e4m3)
    static constexpr int TN = TN_;                        // N = 256 MMAs per K step (pairs)
    static constexpr int CL = CL_;                        // CTAs per cluster: 1 or 2
    static constexpr bool PAIR = CL > 1;                  // 2-SM MMA on CTA pairs
    static constexpr int BK = BK_;
    static constexpr int ROWB = BK * EB;                  // bytes per operand row
    static constexpr int A_ROWS = UM * TM;                // rows of A per CTA and stage
    static constexpr int B_ROWS = PAIR ? TN * BN / 2 : BN;  // rows of B per CTA and stage
    static constexpr int BMT = A_ROWS * (PAIR ? 2 : 1);   // rows of A per tile
    static constexpr int A_BOX_ROWS = A_ROWS / 2;                    // rows of one A copy
    static constexpr int B_BOX_ROWS = B_ROWS / 2;                    // rows of one B copy
    static constexpr int A_BYTES = A_ROWS * ROWB;
    static constexpr int B_BYTES = B_ROWS * ROWB;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = SMEM_RING / STAGE_BYTES;
    static constexpr int NACC = TM == 1 && TN == 1 ? 2 : 1;  // accumulator buffers
    static constexpr int ACC_COLS = BN * TM * TN;         // TMEM columns per buffer
    static_assert(ROWB == 128 || ROWB == 64, "BK");
    static_assert(CL == 1 || CL == 2, "cluster size");
    static_assert(!PAIR || TM == 1, "pair tiles use one M=256 MMA");
    static_assert(TN == 1 || (TN == 2 && CL == 2), "512-column tiles on plain CTA pairs");
    static_assert(STAGES >= 3 && STAGES <= 8, "stages");
};

// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(UM >> 4) << 24);
// The same for the 2-SM MMA: M = 256 over the CTA pair (128 rows per CTA).
constexpr uint32_t IDESC_PAIR = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((2 * UM) >> 4) << 24);
// ... with B MN-major (bit 16); with A and B MN-major (bits 15 and 16).
constexpr uint32_t IDESC_PAIR_BMN = IDESC_PAIR | (1u << 16);
constexpr uint32_t IDESC_PAIR_MN = IDESC_PAIR | (1u << 15) | (1u << 16);
// kind::f8f6f4 with A and B e4m3 (format 0), D fp32, both K-major; the 2-SM
// MMA, K = 32 elements (32 bytes, as kind::f16's 16 elements).
constexpr uint32_t IDESC_PAIR_F8 = (1u << 4) | ((uint32_t)(BN >> 3) << 17) |
                                   ((uint32_t)((2 * UM) >> 4) << 24);

template <int STAGES>
struct Ctl {  // control block in shared memory
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
    int32_t total_tiles;
    int32_t tile_start[MAX_E + 1];
};

// Output staging per epilogue warp: 32 rows x 32 bf16 (64-byte swizzle),
// written by the warp and stored to global memory by TMA.
constexpr int STG_WARP_BYTES = 2048;

template <class TL>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)TL::STAGES * TL::STAGE_BYTES + (size_t)EPI_WARPS * STG_WARP_BYTES +
           sizeof(Ctl<TL::STAGES>);
}

struct GemmArgs {
    const int32_t *counts;
    const int32_t *c_dev;
    int32_t *status;
    const __nv_bfloat16 *bias;  // [e, n_out] or nullptr
    __nv_bfloat16 *out;         // [e, c_max, n_out]
    int64_t c_max;
    int e;
    int K;             // contraction length
    int n_out;         // output columns per expert
    int b_rows;        // rows of each B tensor map per expert
    // Contraction per expert (weight gradients): when set, every expert has
    // c_max output rows (counts / c_dev unused) and expert j contracts over
    // its first min(k_counts[j], *k_cdev, K) K columns only; the operands must
    // be zero from there to the next multiple of BK.  An expert with none
    // gets a zero output tile and no MMA.
    const int32_t *k_counts;
    const int32_t *k_cdev;
    // Row range (forward only): expert rows [row_lo, row_hi) of the kept rows
    // are computed (row_hi = 0: no upper end); rows are addressed from row_lo.
    int row_lo;
    int row_hi;
    // e4m3 operands: the fp32 scale of every A row ([e * c_max]) and of every
    // B row, i.e. output column ([e * n_out]); the epilogue forms
    // acc * (a_scale * b_scale) + bias.  NULL for bf16.
    const float *a_scale;
    const float *b_scale;
    // EPI_DGELU / EPI_DRELU: d_hid [e * c_max, n_out], the rows of out;
    // EPI_DGELU_BMN / EPI_DRELU_BMN: the saved pre-activation, likewise.
    const __nv_bfloat16 *aux;
    // EPI_GELU_SAVE / EPI_RELU_SAVE: where the pre-activation goes, likewise.
    __nv_bfloat16 *aux_out;
    // EPI_WGRAD_MN_F32: the result in fp32 [e * c_max, n_out] (out unused).
    float *out_f32;
    // Elements between rows of out (0: n_out).
    int64_t out_pitch;
    // MN-major B stacked along K from two maps (SwiGLU's [W1; W3]): K rows from
    // k_split on come from tmB3, k_split rows earlier (0: tmB only).
    int32_t k_split;
    // Per-expert K: experts without K rows get no tiles (nothing written).
    int32_t skip_empty;
    // Error-path test: the producers issue no copies, so the MMA issuer's
    // bounded wait on the first stage runs out (MOE_ERR_TIMEOUT).
    int32_t stall;
};

// ------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t su32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}

// CL: acquire at cluster scope (arrivals and copies from the peer CTA of a pair).
template <bool CL = false>
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    if (CL)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(su32(b)), "r"(parity)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(su32(b)), "r"(parity)
            : "memory");
    return ok != 0;
}

// Bounded wait for the phase with `parity` to complete.  Returns false if the
// CTA is aborting or the wait ran past WAIT_NS (then the abort is raised).
template <bool CL = false>
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, int32_t *abort_flag,
                                       int32_t *status) {
    if (mbar_try<CL>(b, parity)) return true;
    unsigned long long t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try<CL>(b, parity)) return true;
        if ((it & 31u) == 0) {
            if (*(volatile int32_t *)abort_flag) return false;
            if (gtimer() - t0 > WAIT_NS) {
                *(volatile int32_t *)abort_flag = 1;
                set_status(status, MOE_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(su32(bar))
        : "memory");
}

// TMA store of a box from this CTA's shared memory (bulk async-group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y, const void *src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     (uint64_t)map),
                 "r"(x), "r"(y), "r"(su32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's store groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until all of this thread's store groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint8_t *p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(su32(p)), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// One lane's 32 output columns (pk: 16 packed bf16 pairs, column order) of a
// warp's 32 consecutive rows starting at global row grow0, columns gcol...
// When all 32 rows are kept: through the warp's staging buffer (row = lane,
// 16-byte chunk c of a 64-byte row at c ^ ((row >> 1) & 3), the 64-byte
// swizzle pattern) and one TMA store, which clips columns >= n_out.
// Otherwise direct stores of this lane's row if it is kept.
__device__ __forceinline__ void epi_store32(const CUtensorMap *map, uint8_t *stg,
                                            const uint32_t (&pk)[16], bool all_kept, bool kept,
                                            int lane, int64_t grow0, int gcol, int n_out,
                                            __nv_bfloat16 *orow) {
    if (all_kept) {
        if (gcol >= n_out) return;  // warp-uniform
        if (lane == 0) bulk_wait_read<0>();  // the previous store has read the buffer
        __syncwarp();
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int c = 0; c < 4; c++)
            st_shared_v4(stg + lane * 64 + ((c ^ sw) << 4), pk[c * 4 + 0], pk[c * 4 + 1],
                         pk[c * 4 + 2], pk[c * 4 + 3]);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(map, gcol, (int)grow0, stg);
            bulk_commit();
        }
    } else if (kept) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (gcol + q * 8 < n_out) {
                V16 o;
                o.w[0] = pk[q * 4 + 0]; o.w[1] = pk[q * 4 + 1];
                o.w[2] = pk[q * 4 + 2]; o.w[3] = pk[q * 4 + 3];
                st_v16(orow + gcol + q * 8, o);
            }
        }
    }
}

// The same for 16 fp32 columns (64-byte rows: the same staging pattern and
// swizzle), with a 16 x 32 fp32 output map; the fallback stores this lane's
// row directly.
__device__ __forceinline__ void epi_store16f(const CUtensorMap *map, uint8_t *stg, const float *v,
                                             bool all_kept, bool kept, int lane, int64_t grow0,
                                             int gcol, int n_out, float *frow) {
    if (all_kept) {
        if (gcol >= n_out) return;  // warp-uniform
        if (lane == 0) bulk_wait_read<0>();  // the previous store has read the buffer
        __syncwarp();
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int c = 0; c < 4; c++)
            st_shared_v4(stg + lane * 64 + ((c ^ sw) << 4), __float_as_uint(v[4 * c]),
                         __float_as_uint(v[4 * c + 1]), __float_as_uint(v[4 * c + 2]),
                         __float_as_uint(v[4 * c + 3]));
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(map, gcol, (int)grow0, stg);
            bulk_commit();
        }
    } else if (kept) {
#pragma unroll
        for (int q = 0; q < 4; q++)
            if (gcol + 4 * q < n_out)
                *reinterpret_cast<float4 *>(frow + gcol + 4 * q) =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
}

// ------------------------------------------------------- CTA-pair helpers
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier of either CTA of the pair.  Release at CTA scope (the
// default): what the waiter needs ordered are this thread's completed
// tcgen05.ld (by tcgen05.fence::before_thread_sync), not its global stores; a
// cluster-scope release would wait for those stores as well.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the swizzled layout
// TMA writes: 8-row atoms of ROWB-byte rows (128 B: swizzle mode 2, 64 B:
// mode 4, bits 61-63), atoms ROWB*8 bytes apart (stride byte offset); the
// leading-byte offset is unused for these layouts; bits 46-48 = 0b001.
template <int ROWB>
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    constexpr uint64_t mode = ROWB == 128 ? 2 : 4;
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)((ROWB * 8) >> 4) << 32) | ((uint64_t)1 << 46) | (mode << 61);
}

// Shared-memory matrix descriptor of an MN-major operand in the 128-byte
// swizzled layout TMA writes for boxes of 64 elements along M/N by BK rows
// along K: 8-row groups along K 1024 bytes apart (stride byte offset), the
// 64-element blocks along M/N `lbo` bytes apart (leading byte offset).
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr, uint32_t lbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(IDESC), "r"(accumulate)
        : "memory");
}

// 2-SM MMA, issued by the pair's first CTA: A and B descriptors name the same
// shared-memory offsets in both CTAs; each CTA's TMEM receives its 128 rows.
template <uint32_t ID = IDESC_PAIR>
__device__ __forceinline__ void umma_pair(uint32_t tmem_d, uint64_t a, uint64_t b,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(ID), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_pair_f8(uint32_t tmem_d, uint64_t a, uint64_t b,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(IDESC_PAIR_F8), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            su32(bar))
        : "memory");
}

// Arrive on the mbarrier at this offset in every CTA of `mask` (cluster CTA
// ranks) once the pair MMAs issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(su32(bar)),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Wait for this thread's outstanding tcgen05.ld.  The registers of a load are
// tied to the wait so that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
          "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
          "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
          "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
        :
        : "memory");
}

// Ties further registers to an already completed wait (emits nothing).
__device__ __forceinline__ void tmem_tie(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}

// GELU, exact erf form: a * Phi(a) with Phi(a) = 0.5 (1 + erf(a / sqrt 2)),
// evaluated as 1 - erfc/2 for a >= 0 and erfc(|a| / sqrt 2) / 2 for a < 0 so
// that the negative tail does not cancel.  erfc(x) for x >= 0 by Abramowitz &
// Stegun, Handbook of Mathematical Functions, formula 7.1.28 (Hastings):
// erf(x) = 1 - (1 + a1 x + ... + a6 x^6)^-16 with |error| <= 3e-7, so
// erfc(x) = (1 + a1 x + ... + a6 x^6)^-16: one reciprocal and no exponential,
// which keeps the fc1 epilogue cheap; |GELU error| <= 5e-7, three orders of
// magnitude below the bf16 rounding that follows.  Two values at a time with
// packed fp32x2 arithmetic; the 16th power overflows to inf for large x, where
// erfc -> 0.
__device__ __forceinline__ float2 gelu_erf2(float2 a) {
    const float2 x = __fmul2_rn(make_float2(fabsf(a.x), fabsf(a.y)),
                                make_float2(0.70710678118654752f, 0.70710678118654752f));
    float2 p = __ffma2_rn(x, make_float2(0.0000430638f, 0.0000430638f),
                          make_float2(0.0002765672f, 0.0002765672f));
    p = __ffma2_rn(x, p, make_float2(0.0001520143f, 0.0001520143f));
    p = __ffma2_rn(x, p, make_float2(0.0092705272f, 0.0092705272f));
    p = __ffma2_rn(x, p, make_float2(0.0422820123f, 0.0422820123f));
    p = __ffma2_rn(x, p, make_float2(0.0705230784f, 0.0705230784f));
    p = __ffma2_rn(x, p, make_float2(1.0f, 1.0f));
    float2 q = __fmul2_rn(p, p);
    q = __fmul2_rn(q, q);
    q = __fmul2_rn(q, q);
    q = __fmul2_rn(q, q);
    float2 r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(q.x));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(q.y));
    r = __fmul2_rn(r, make_float2(0.5f, 0.5f));
    const float2 phi = make_float2(a.x >= 0.0f ? 1.0f - r.x : r.x, a.y >= 0.0f ? 1.0f - r.y : r.y);
    return __fmul2_rn(a, phi);
}

// GELU'(z) = Phi(z) + z phi(z), two values at a time: Phi as in gelu_erf2
// (A&S 7.1.28 erfc, 1 - erfc/2 above zero, erfc/2 below); phi(z) =
// 2^(-z^2 log2(e) / 2) / sqrt(2 pi) with the approximate power of two
// (relative error ~2^-22, far below the bf16 rounding that follows).
__device__ __forceinline__ float2 gelu_grad2(float2 z) {
    const float2 x = __fmul2_rn(make_float2(fabsf(z.x), fabsf(z.y)),
                                make_float2(0.70710678118654752f, 0.70710678118654752f));
    float2 p = __ffma2_rn(x, make_float2(0.0000430638f, 0.0000430638f),
                          make_float2(0.0002765672f, 0.0002765672f));
    p = __ffma2_rn(x, p, make_float2(0.0001520143f, 0.0001520143f));
    p = __ffma2_rn(x, p, make_float2(0.0092705272f, 0.0092705272f));
    p = __ffma2_rn(x, p, make_float2(0.0422820123f, 0.0422820123f));
    p = __ffma2_rn(x, p, make_float2(0.0705230784f, 0.0705230784f));
    p = __ffma2_rn(x, p, make_float2(1.0f, 1.0f));
    float2 q = __fmul2_rn(p, p);
    q = __fmul2_rn(q, q);
    q = __fmul2_rn(q, q);
    q = __fmul2_rn(q, q);
    float2 r, d;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(q.x));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(q.y));
    r = __fmul2_rn(r, make_float2(0.5f, 0.5f));
    const float2 cdf = make_float2(z.x >= 0.0f ? 1.0f - r.x : r.x, z.y >= 0.0f ? 1.0f - r.y : r.y);
    const float2 t = __fmul2_rn(__fmul2_rn(z, z), make_float2(-0.72134752044448170f, -0.72134752044448170f));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(d.x) : "f"(t.x));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(d.y) : "f"(t.y));
    return __ffma2_rn(__fmul2_rn(z, make_float2(0.3989422804014327f, 0.3989422804014327f)), d, cdf);
}

__device__ __forceinline__ float silu(float a) { return a / (1.0f + expf(-a)); }

// Tile t -> (expert j, m-tile, n-tile); m-tile varies fastest.  rows: the
// expert's output rows; nk: its K blocks.  kept_rows[] holds the output rows
// per expert, or (uniform_rows > 0: every expert has that many output rows)
// the K columns per expert.
struct Tile { int j, mt, nt, rows, nk; };

__device__ __forceinline__ Tile decode_tile(const int32_t *tile_start, int e, int t, int bmt,
                                            const int32_t *kept_rows, int uniform_rows,
                                            int nk_all, int bk) {
    int lo = 0, hi = e;  // largest j with tile_start[j] <= t
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    Tile T;
    T.j = lo;
    int local = t - tile_start[lo];
    T.rows = uniform_rows > 0 ? uniform_rows : kept_rows[lo];
    T.nk = uniform_rows > 0 ? (kept_rows[lo] + bk - 1) / bk : nk_all;
    int mtiles = (T.rows + bmt - 1) / bmt;
    T.nt = local / mtiles;
    T.mt = local % mtiles;
    return T;
}

template <int EPI, int TM, int BK, int CL, int TN, int EB = 2>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_group_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmO,
              const __grid_constant__ CUtensorMap tmAt, const __grid_constant__ CUtensorMap tmBt,
              const GemmArgs args) {
    using TL = Tiling<TM, BK, CL, TN, EB>;
    static_assert(TN == 1 || !is_swiglu(EPI), "SwiGLU tiles pair W1 and W3 in one N = 256 MMA");
    constexpr bool F8 = EB == 1;   // e4m3 operands (kind::f8f6f4), scaled epilogue
    static_assert(!F8 || (CL == 2 && !is_swiglu(EPI) && EPI != EPI_BIAS_BMN), "e4m3 pair tiles");
    constexpr bool F32OUT = EPI == EPI_WGRAD_MN_F32;   // fp32 result, stored from registers
    constexpr bool AMN = EPI == EPI_WGRAD_MN || F32OUT;   // A MN-major as well, tail blocks from tmAt / tmBt
    constexpr bool DACT = EPI == EPI_DGELU || EPI == EPI_DRELU;   // activation backward epilogue
    constexpr bool DSWI = EPI == EPI_DSWIGLU_BMN;   // SwiGLU derivative of a saved [a | b]
    constexpr bool DACTP = EPI == EPI_DGELU_BMN || EPI == EPI_DRELU_BMN || DSWI;   // act' of a saved pre
    constexpr bool DGELU = EPI == EPI_DGELU || EPI == EPI_DGELU_BMN;
    constexpr bool SAVE = EPI == EPI_GELU_SAVE || EPI == EPI_RELU_SAVE;   // fc1 keeping its pre-activation
    constexpr bool GELU = EPI == EPI_GELU || EPI == EPI_GELU_SAVE;
    constexpr bool RELU = EPI == EPI_RELU || EPI == EPI_RELU_SAVE;
    constexpr bool BMN = EPI == EPI_BIAS_BMN || AMN || DACTP;   // B MN-major: [K, N] rows, 64-column boxes
    static_assert(!BMN || (CL == 2 && BK == 64), "MN-major operands on pair tiles");
    constexpr bool PAIR = TL::PAIR;
    constexpr int STAGES = TL::STAGES, BMT = TL::BMT, A_BYTES = TL::A_BYTES;
    constexpr int B_BYTES = TL::B_BYTES, ROWB = TL::ROWB;
    __shared__ int32_t s_bad;
    pdl_enter();
    if (threadIdx.x == 0) s_bad = status_bad(args.status) ? 1 : 0;
    __syncthreads();
    // A single CTA may leave now (nothing allocated yet); a cluster decides
    // together after its first cluster barrier.
    if (!PAIR && s_bad) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint8_t *stg_all = smem + STAGES * TL::STAGE_BYTES;  // output staging
    Ctl<STAGES> *ctl = (Ctl<STAGES> *)(stg_all + EPI_WARPS * STG_WARP_BYTES);
    __shared__ int32_t kept_rows[MAX_E];
    __shared__ __align__(16) float epi_bias[EPI_WARPS][256];  // per epilogue warp

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = args.e;
    // Pairs: the even CTA of each pair issues the pair's MMAs; tiles are
    // dealt out per cluster.
    const uint32_t rank = PAIR ? cluster_rank() : 0;
    const uint32_t prank = rank & 1u;    // rank within the pair
    const uint32_t lead = rank & ~1u;    // the pair's MMA-issuing CTA
    const int tile0 = (int)(blockIdx.x / CL);
    const int tile_step = (int)(gridDim.x / CL);
    constexpr int NOUT_TILE = is_swiglu(EPI) ? BN / 2 : BN * TN;  // output columns per tile
    const int ntn = (args.n_out + NOUT_TILE - 1) / NOUT_TILE;
    const int nk = (args.K + BK - 1) / BK;
    const bool kmode = args.k_counts != nullptr;           // K per expert
    const int urows = kmode ? (int)args.c_max : 0;

    // ---- setup: per-expert row counts and tile prefix (warp 0), barriers,
    // TMEM allocation (warp 1)
    if (warp == 0) {
        const int c_eff = kmode ? 0 : (int)min((int64_t)*args.c_dev, args.c_max);
        const int k_eff = kmode ? (int)min((int64_t)*args.k_cdev, (int64_t)args.K) : 0;
        int run = 0;
        for (int base = 0; base < e; base += 32) {
            int j = base + lane;
            int rows = j >= e ? 0 : kmode ? urows : min(max(args.counts[j], 0), c_eff);
            if (!kmode && j < e) {   // the kept rows inside [row_lo, row_hi)
                const int hi = args.row_hi > 0 ? min(rows, args.row_hi) : rows;
                rows = max(0, hi - args.row_lo);
            }
            if (j < e) kept_rows[j] = kmode ? min(max(args.k_counts[j], 0), k_eff) : rows;
            // per-expert K: an expert without any K rows gets no tiles when asked
            // (its zero output is written elsewhere)
            if (kmode && args.skip_empty && j < e && kept_rows[j] == 0) rows = 0;
            const int own = ((rows + BMT - 1) / BMT) * ntn;
            int v = own;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (j < e) ctl->tile_start[j] = run + v - own;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) {
            ctl->tile_start[e] = run;
            ctl->total_tiles = run;
            ctl->abort = 0;
            // full: one arrival (with its transaction bytes, for a pair those of
            // both CTAs) from each of the four producers of the MMA-issuing CTA
            // empty: released by the MMAs of every pair whose copies write the stage
            for (int s = 0; s < STAGES; s++) { mbar_init(&ctl->full[s], 4); mbar_init(&ctl->empty[s], 1); }
            for (int a = 0; a < 2; a++) {
                mbar_init(&ctl->tfull[a], 1);
                mbar_init(&ctl->tempty[a], PAIR ? 2 * EPI_WARPS : EPI_WARPS);
            }
            mbar_init(&ctl->drain, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    } else if (warp == 1) {
        if (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             su32(&ctl->tmem_base)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             su32(&ctl->tmem_base)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    if (PAIR) cluster_sync();  // every CTA's barriers initialised, TMEM allocated
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    int total = ctl->total_tiles;
    if (PAIR) {
        int any_bad = 0;
        for (uint32_t r = 0; r < (uint32_t)CL; r++) {
            int b;
            asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(b) : "r"(map_to_rank(su32(&s_bad), r)));
            any_bad |= b;
        }
        if (any_bad) total = 0;  // the same decision in every CTA of the cluster
    }
    int32_t *abort_flag = &ctl->abort;

    if (warp == 0 || warp >= PROD_WARP0) {
        // ----------------------------------------------------- TMA producers
        // Four issuing threads in different warps: prod 0/2 load the two row
        // halves of each stage's A tile, 1/3 those of its B tile (lane 0 of each
        // issues).  In a pair both CTAs load their own halves; the copies
        // complete on the pair-leading CTA's full barriers, whose producers
        // announce the bytes of both.
        const int prod = warp == 0 ? 0 : warp - PROD_WARP0 + 1;
        const bool is_a = (prod & 1) == 0;
        const int hh = prod >> 1;   // row half of this producer's boxes
        constexpr int A_BOX_BYTES = TL::A_BOX_ROWS * ROWB, B_BOX_BYTES = TL::B_BOX_ROWS * ROWB;
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        for (int t = tile0; t < total && !args.stall; t += tile_step) {
            Tile T = decode_tile(ctl->tile_start, e, t, BMT, kept_rows, urows, nk, BK);
            // A: this CTA's 128 rows, half of them per producer
            const int a_row = (int)((int64_t)T.j * args.c_max + args.row_lo + (int64_t)T.mt * BMT +
                                    (int64_t)prank * TL::A_ROWS + (int64_t)hh * TL::A_BOX_ROWS);
            // B rows of this CTA: its half of the (each) N = 256 sub-tile; with
            // TN = 2 producer hh loads N sub-tile hh
            const int b_row = T.j * args.b_rows + T.nt * NOUT_TILE +
                              (TN == 2 ? hh * BN + (int)prank * (BN / 2)
                                       : (PAIR && !is_swiglu(EPI) ? (int)prank * TL::B_ROWS : 0) +
                                             hh * TL::B_BOX_ROWS);
            // MN-major weight gradients: a last K block only partly kept
            // comes from the tail maps (rows j * BK ..)
            const bool part_tail = AMN && (kept_rows[T.j] % BK) != 0;
            for (int kb = 0; kb < T.nk; kb++) {
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait<PAIR>(&ctl->empty[stage], phase ^ 1u, abort_flag, args.status);
                    const bool tail = part_tail && kb == T.nk - 1;
                    const int k_row = tail ? T.j * BK : T.j * args.b_rows + kb * BK;
                    if (ok && PAIR && AMN) {
                        const uint32_t fb = map_to_rank(su32(&ctl->full[stage]), lead);
                        if (is_a) {
                            // this CTA's 128 output rows = A columns, block hh of 64
                            if (prank == 0) mbar_expect_tx(&ctl->full[stage], 2 * A_BOX_BYTES);
                            tma_load_2d_pair(sA + stage * A_BYTES + hh * A_BOX_BYTES,
                                             tail ? &tmAt : &tmA,
                                             T.mt * BMT + (int)prank * TL::A_ROWS + hh * 64, k_row, fb);
                        } else {
                            if (prank == 0) mbar_expect_tx(&ctl->full[stage], 2 * B_BOX_BYTES);
                            const int n_col = b_row - T.j * args.b_rows;
#pragma unroll
                            for (int i = 0; i < TN; i++)   // TN boxes of 64 columns
                                tma_load_2d_pair(sB + stage * B_BYTES + hh * B_BOX_BYTES +
                                                     i * (B_BOX_BYTES / TN),
                                                 tail ? &tmBt : &tmB, n_col + 64 * i, k_row, fb);
                        }
                    } else if (ok && PAIR) {
                        const uint32_t fb = map_to_rank(su32(&ctl->full[stage]), lead);
                        if (is_a) {
                            if (prank == 0) mbar_expect_tx(&ctl->full[stage], 2 * A_BOX_BYTES);
                            tma_load_2d_pair(sA + stage * A_BYTES + hh * A_BOX_BYTES, &tmA, kb * BK,
                                             a_row, fb);
                        } else if (BMN) {
                            // this CTA's 128 columns of N sub-tile hh, K rows kb*BK ..:
                            // two boxes of 64 columns (b_row - j * b_rows is the column)
                            if (prank == 0) mbar_expect_tx(&ctl->full[stage], 2 * B_BOX_BYTES);
                            const int n_col = b_row - T.j * args.b_rows;
                            const bool second = args.k_split > 0 && kb * BK >= args.k_split;
#pragma unroll
                            for (int i = 0; i < TN; i++)   // TN boxes of 64 columns
                                tma_load_2d_pair(sB + stage * B_BYTES + hh * B_BOX_BYTES +
                                                     i * (B_BOX_BYTES / TN),
                                                 second ? &tmB3 : &tmB, n_col + 64 * i,
                                                 second ? k_row - args.k_split : k_row, fb);
                        } else {
                            // SwiGLU: the first CTA's half of B is W1, the second's W3
                            if (prank == 0) mbar_expect_tx(&ctl->full[stage], 2 * B_BOX_BYTES);
                            tma_load_2d_pair(sB + stage * B_BYTES + hh * B_BOX_BYTES,
                                             is_swiglu(EPI) && prank ? &tmB3 : &tmB, kb * BK, b_row, fb);
                        }
                    } else if (ok && is_a) {
                        mbar_expect_tx(&ctl->full[stage], A_BOX_BYTES);
                        tma_load_2d(sA + stage * A_BYTES + hh * A_BOX_BYTES, &tmA, kb * BK, a_row,
                                    &ctl->full[stage]);
                    } else if (ok && is_swiglu(EPI)) {
                        // W1 rows in the first half of the B tile, W3 rows in the second
                        mbar_expect_tx(&ctl->full[stage], B_BOX_BYTES);
                        tma_load_2d(sB + stage * B_BYTES + hh * B_BOX_BYTES, hh ? &tmB3 : &tmB, kb * BK,
                                    b_row - hh * TL::B_BOX_ROWS, &ctl->full[stage]);
                    } else if (ok) {
                        mbar_expect_tx(&ctl->full[stage], B_BOX_BYTES);
                        tma_load_2d(sB + stage * B_BYTES + hh * B_BOX_BYTES, &tmB, kb * BK, b_row,
                                    &ctl->full[stage]);
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) goto producer_done;
                issued++;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    producer_done:
        // wait (bounded) for this thread's copies still in flight before the CTA
        // can exit (a pair's second CTA cannot observe the first CTA's barriers:
        // its copies are covered by the MMAs that consume them, or on an abort
        // by the delay before the final cluster barrier)
        if (lane == 0 && (!PAIR || prank == 0)) {
            for (int i = max(0, issued - STAGES); i < issued; i++) {
                int s = i % STAGES;
                uint32_t ph = (uint32_t)((i / STAGES) & 1);
                unsigned long long t0 = gtimer();
                while (!mbar_try<PAIR>(&ctl->full[s], ph) && gtimer() - t0 < WAIT_NS) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (!PAIR || prank == 0) {
            // both CTAs of the pair
            const uint16_t pair_mask = (uint16_t)3u;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int t = tile0; t < total; t += tile_step) {
                const int tnk = kmode ? decode_tile(ctl->tile_start, e, t, BMT, kept_rows, urows, nk, BK).nk : nk;
                if (!mbar_wait<PAIR>(&ctl->tempty[acc], acc_phase ^ 1u, abort_flag, args.status)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * TL::ACC_COLS);
                bool ok = true;
                for (int kb = 0; kb < tnk; kb++) {
                    if (!mbar_wait<PAIR>(&ctl->full[stage], phase, abort_flag, args.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = su32(sA + stage * A_BYTES);
                    const uint32_t b0 = su32(sB + stage * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < ROWB / 32; kk++) {   // one MMA per 32 bytes of K
                        if (F8) {
#pragma unroll
                            for (int tn = 0; tn < TN; tn++)
                                umma_pair_f8(d + (uint32_t)(tn * BN), sdesc<ROWB>(a0 + kk * 32),
                                             sdesc<ROWB>(b0 + tn * (B_BYTES / TN) + kk * 32),
                                             (kb | kk) != 0);
                        } else if (AMN) {
                            // A and B: K rows of 128 bytes, kk * UK rows in; A's two
                            // 64-column blocks A_BYTES / 2 apart, B's as below
#pragma unroll
                            for (int tn = 0; tn < TN; tn++)
                                umma_pair<IDESC_PAIR_MN>(
                                    d + (uint32_t)(tn * BN), sdesc_mn(a0 + kk * UK * 128, A_BYTES / 2),
                                    sdesc_mn(b0 + tn * (B_BYTES / TN) + kk * UK * 128,
                                             B_BYTES / TN / 2),
                                    (kb | kk) != 0);
                        } else if (BMN) {
                            // B: K rows of 128 bytes, kk * UK rows in; blocks of 64
                            // columns (B_BYTES / TN / 2 bytes) apart
#pragma unroll
                            for (int tn = 0; tn < TN; tn++)
                                umma_pair<IDESC_PAIR_BMN>(
                                    d + (uint32_t)(tn * BN), sdesc<ROWB>(a0 + kk * UK * 2),
                                    sdesc_mn(b0 + tn * (B_BYTES / TN) + kk * UK * 128,
                                             B_BYTES / TN / 2),
                                    (kb | kk) != 0);
                        } else if (PAIR) {
#pragma unroll
                            for (int tn = 0; tn < TN; tn++)  // N sub-tiles share the A tile
                                umma_pair(d + (uint32_t)(tn * BN), sdesc<ROWB>(a0 + kk * UK * 2),
                                          sdesc<ROWB>(b0 + tn * (B_BYTES / TN) + kk * UK * 2),
                                          (kb | kk) != 0);
                        } else {
#pragma unroll
                            for (int hm = 0; hm < TM; hm++)  // M halves share the B tile
                                umma(d + (uint32_t)(hm * BN),
                                     sdesc<ROWB>(a0 + hm * UM * ROWB + kk * UK * 2),
                                     sdesc<ROWB>(b0 + kk * UK * 2), (kb | kk) != 0);
                        }
                    }
                    // stage reusable (in both CTAs of a pair) once these MMAs read it
                    if (PAIR) umma_commit_pair(&ctl->empty[stage], pair_mask);
                    else umma_commit(&ctl->empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                // accumulator ready when all MMAs finish (a tile without K
                // blocks is published at once; its epilogue writes zeros)
                if (PAIR) umma_commit_pair(&ctl->tfull[acc], pair_mask);
                else umma_commit(&ctl->tfull[acc]);
                if (++acc == TL::NACC) { acc = 0; acc_phase ^= 1u; }
            }
            // all MMAs issued by this thread complete before TMEM is released
            if (PAIR) umma_commit_pair(&ctl->drain, pair_mask);
            else umma_commit(&ctl->drain);
        }
        unsigned long long t0 = gtimer();
        while (!mbar_try<PAIR>(&ctl->drain, 0) && gtimer() - t0 < WAIT_NS) {
        }
    } else if (warp >= 2 && warp < PROD_WARP0) {
        // ------------------------------------------------------------- epilogue
        // TM = 1: warp (sub, half) owns rows sub*32.. and half of the columns.
        // TM = 2: warp (sub, half) owns rows half*128 + sub*32.. and all columns.
        // A pair's second CTA holds rows 128..255 of the tile.
        const int ew = warp - 2;
        const int sub = warp & 3;             // TMEM lane quarter this warp may access
        const int half = ew >> 2;
        const int row_in_tile = (int)prank * UM + (TM == 2 ? half * UM : 0) + sub * 32 + lane;
        constexpr int COLS = TM == 2 ? NOUT_TILE : NOUT_TILE / 2;  // output columns per warp
        const int col0 = TM == 2 ? 0 : half * COLS;                // first output column
        uint8_t *stg = stg_all + ew * STG_WARP_BYTES;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = tile0; t < total; t += tile_step) {
            Tile T = decode_tile(ctl->tile_start, e, t, BMT, kept_rows, urows, nk, BK);
            if (!mbar_wait<PAIR>(&ctl->tfull[acc], acc_phase, abort_flag, args.status)) break;
            tc_fence_after();
            const int row = T.mt * BMT + row_in_tile;
            const bool valid = row < T.rows;
            const bool all_kept = row - lane + 31 < T.rows;  // the warp's 32 rows
            const int64_t grow0 = (int64_t)T.j * args.c_max + args.row_lo + row - lane;
            __nv_bfloat16 *orow =
                args.out + ((int64_t)T.j * args.c_max + args.row_lo + row) *
                               (args.out_pitch ? args.out_pitch : (int64_t)args.n_out);
            const __nv_bfloat16 *brow = args.bias ? args.bias + (int64_t)T.j * args.n_out : nullptr;
            const uint32_t tbase = tmem + ((uint32_t)(sub * 32) << 16) +
                                   (uint32_t)(acc * TL::ACC_COLS + (TM == 2 ? half * BN : 0));
            if (is_swiglu(EPI)) {
#pragma unroll 1
                for (int c0 = 0; c0 < COLS; c0 += 32) {
                    const int ocol = col0 + c0;               // column within the tile's output
                    const int gcol = T.nt * NOUT_TILE + ocol; // column within the expert
                    uint32_t r[32], u[32];
                    if (T.nk > 0) {
                        tmem_ld32(tbase + (uint32_t)ocol, r);
                        tmem_ld32(tbase + (uint32_t)(BN / 2 + ocol), u);
                        tmem_wait_ld(r);
                        tmem_tie(u);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i++) r[i] = u[i] = 0u;   // empty contraction
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        pk[i] = pack_bf16(silu(__uint_as_float(r[2 * i])) * __uint_as_float(u[2 * i]),
                                          silu(__uint_as_float(r[2 * i + 1])) *
                                              __uint_as_float(u[2 * i + 1]));
                    epi_store32(&tmO, stg, pk, all_kept, valid, lane, grow0, gcol, args.n_out,
                                orow);
                    if (EPI == EPI_SWIGLU_SAVE && valid) {   // this lane's row of a, then of b
                        __nv_bfloat16 *arow = args.aux_out + ((int64_t)T.j * args.c_max + args.row_lo +
                                                              row) * (2 * (int64_t)args.n_out);
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            if (gcol + 8 * q < args.n_out) {
                                V16 oa, ob;
#pragma unroll
                                for (int i = 0; i < 4; i++) {
                                    oa.w[i] = pack_bf16(__uint_as_float(r[8 * q + 2 * i]),
                                                        __uint_as_float(r[8 * q + 2 * i + 1]));
                                    ob.w[i] = pack_bf16(__uint_as_float(u[8 * q + 2 * i]),
                                                        __uint_as_float(u[8 * q + 2 * i + 1]));
                                }
                                st_v16(arow + gcol + 8 * q, oa);
                                st_v16(arow + args.n_out + gcol + 8 * q, ob);
                            }
                        }
                    }
                }
            } else {
                // this warp's bias columns, widened to fp32 in shared memory once per tile
                float *bsl = epi_bias[ew];
                if (lane * 8 < COLS) {
                    const int g8 = T.nt * NOUT_TILE + col0 + lane * 8;
                    float b8[8];
                    if (brow && g8 < args.n_out) {
                        Elt<__nv_bfloat16>::unpack(*reinterpret_cast<const V16 *>(brow + g8), b8);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; i++) b8[i] = 0.0f;
                    }
                    reinterpret_cast<float4 *>(bsl + lane * 8)[0] = make_float4(b8[0], b8[1], b8[2], b8[3]);
                    reinterpret_cast<float4 *>(bsl + lane * 8)[1] = make_float4(b8[4], b8[5], b8[6], b8[7]);
                }
                __syncwarp();
                // e4m3: this lane's row scale (its output row)
                const float sa = F8 && valid ? args.a_scale[grow0 + lane] : 0.0f;
                const __nv_bfloat16 *drow =
                    DACT || DACTP
                        ? args.aux + ((int64_t)T.j * args.c_max + args.row_lo + row) *
                                         ((DSWI ? 2 : 1) * (int64_t)args.n_out)
                        : nullptr;
                __nv_bfloat16 *prow =
                    SAVE ? args.aux_out + ((int64_t)T.j * args.c_max + args.row_lo + row) * (int64_t)args.n_out
                         : nullptr;
                const float *bsc = F8 ? args.b_scale + (int64_t)T.j * args.n_out : nullptr;
#pragma unroll 1
                for (int c0 = 0; c0 < COLS; c0 += 64) {
                    uint32_t r[2][32];
                    if (T.nk > 0) {
                        tmem_ld32(tbase + (uint32_t)(col0 + c0), r[0]);
                        tmem_ld32(tbase + (uint32_t)(col0 + c0 + 32), r[1]);
                        tmem_wait_ld(r[0]);
                        tmem_tie(r[1]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i++) r[0][i] = r[1][i] = 0u;   // empty contraction
                    }
#pragma unroll
                    for (int h2 = 0; h2 < 2; h2++) {
                        const int gcol = T.nt * NOUT_TILE + col0 + c0 + 32 * h2;
                        uint32_t pk[16];
                        float of[32];   // weight gradients in fp32: this row's 32 columns
                        uint32_t dv[16];   // activation backward: this row's d_hid or pre (SwiGLU: a), 32 columns
                        uint32_t db[16];   // SwiGLU backward: this row's b, 32 columns
                        if (DACT || DACTP) {
#pragma unroll
                            for (int q = 0; q < 4; q++) {
                                V16 v{}, w{};
                                if (valid && gcol + q * 8 < args.n_out) {
                                    v = ld_v16(drow + gcol + q * 8);
                                    if (DSWI) w = ld_v16(drow + args.n_out + gcol + q * 8);
                                }
#pragma unroll
                                for (int i = 0; i < 4; i++) {
                                    dv[q * 4 + i] = v.w[i];
                                    db[q * 4 + i] = w.w[i];
                                }
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            uint32_t pp[4];   // fc1 keeping its pre-activation: 8 packed columns
                            uint32_t pb[4];   // SwiGLU backward: d_b, 8 packed columns
                            const float4 *bp = reinterpret_cast<const float4 *>(bsl + c0 + 32 * h2 + q * 8);
                            const float4 bl = bp[0], bh = bp[1];
                            const float2 bb[4] = {make_float2(bl.x, bl.y), make_float2(bl.z, bl.w),
                                                  make_float2(bh.x, bh.y), make_float2(bh.z, bh.w)};
                            float sc[8];   // e4m3: a_scale * b_scale of the 8 columns
                            if (F8) {
                                const int g8 = gcol + q * 8;
                                float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
                                if (g8 < args.n_out) {   // n_out is a multiple of 16
                                    lo = reinterpret_cast<const float4 *>(bsc + g8)[0];
                                    hi = reinterpret_cast<const float4 *>(bsc + g8)[1];
                                }
                                sc[0] = sa * lo.x; sc[1] = sa * lo.y; sc[2] = sa * lo.z; sc[3] = sa * lo.w;
                                sc[4] = sa * hi.x; sc[5] = sa * hi.y; sc[6] = sa * hi.z; sc[7] = sa * hi.w;
                            }
#pragma unroll
                            for (int i = 0; i < 4; i++) {
                                const float2 acc2 = make_float2(__uint_as_float(r[h2][q * 8 + 2 * i]),
                                                                __uint_as_float(r[h2][q * 8 + 2 * i + 1]));
                                float2 a = F8 ? __ffma2_rn(acc2, make_float2(sc[2 * i], sc[2 * i + 1]), bb[i])
                                              : __fadd2_rn(acc2, bb[i]);
                                if (SAVE) pp[i] = pack_bf16(a.x, a.y);
                                if (GELU) a = gelu_erf2(a);
                                else if (RELU) a = make_float2(fmaxf(a.x, 0.0f), fmaxf(a.y, 0.0f));
                                if constexpr (DSWI) {
                                    // a = d_hid; the saved a and b of these two columns
                                    const float2 av = make_float2(__uint_as_float(dv[q * 4 + i] << 16),
                                                                  __uint_as_float(dv[q * 4 + i] & 0xFFFF0000u));
                                    const float2 bv = make_float2(__uint_as_float(db[q * 4 + i] << 16),
                                                                  __uint_as_float(db[q * 4 + i] & 0xFFFF0000u));
                                    const float sx = 1.0f / (1.0f + expf(-av.x));
                                    const float sy = 1.0f / (1.0f + expf(-av.y));
                                    pb[i] = pack_bf16(a.x * av.x * sx, a.y * av.y * sy);   // d_b
                                    a = make_float2(a.x * bv.x * sx * (1.0f + av.x * (1.0f - sx)),
                                                    a.y * bv.y * sy * (1.0f + av.y * (1.0f - sy)));   // d_a
                                } else if (DACT || DACTP) {
                                    // DACT: aux is d_hid, a the pre-activation; DACTP: aux is
                                    // the saved pre-activation, a = d_hid
                                    const uint32_t u2 = dv[q * 4 + i];
                                    const float2 u = make_float2(__uint_as_float(u2 << 16),
                                                                 __uint_as_float(u2 & 0xFFFF0000u));
                                    const float2 z = DACT ? a : u, g = DACT ? u : a;
                                    const float2 da = DGELU ? gelu_grad2(z)
                                                            : make_float2(z.x > 0.0f ? 1.0f : 0.0f,
                                                                          z.y > 0.0f ? 1.0f : 0.0f);
                                    a = __fmul2_rn(g, da);
                                }
                                if constexpr (F32OUT) {
                                    of[q * 8 + 2 * i] = a.x;
                                    of[q * 8 + 2 * i + 1] = a.y;
                                } else {
                                    pk[q * 4 + i] = pack_bf16(a.x, a.y);
                                }
                            }
                            if (SAVE && valid && gcol + q * 8 < args.n_out) {
                                // this lane's row of the pre-activation, 8 columns
                                V16 o;
                                o.w[0] = pp[0]; o.w[1] = pp[1]; o.w[2] = pp[2]; o.w[3] = pp[3];
                                st_v16(prow + gcol + q * 8, o);
                            }
                            if constexpr (DSWI) {
                                if (valid && gcol + q * 8 < args.n_out) {
                                    // d_b: the second half of this lane's output row, 8 columns
                                    V16 o;
                                    o.w[0] = pb[0]; o.w[1] = pb[1]; o.w[2] = pb[2]; o.w[3] = pb[3];
                                    st_v16(orow + args.n_out + gcol + q * 8, o);
                                }
                            }
                        }
                        if constexpr (F32OUT) {   // fp32 weight gradients: two 16-column boxes
                            float *frow = args.out_f32 + (grow0 + lane) * (int64_t)args.n_out;
                            epi_store16f(&tmO, stg, of, all_kept, valid, lane, grow0, gcol, args.n_out,
                                         frow);
                            epi_store16f(&tmO, stg, of + 16, all_kept, valid, lane, grow0, gcol + 16,
                                         args.n_out, frow);
                        } else {
                            epi_store32(&tmO, stg, pk, all_kept, valid, lane, grow0, gcol,
                                        args.n_out, orow);
                        }
                    }
                }
                __syncwarp();   // slice reused for the next tile
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // a pair's accumulators are reused by the first CTA's MMAs
                if (PAIR) mbar_arrive_cluster(map_to_rank(su32(&ctl->tempty[acc]), lead));
                else mbar_arrive(&ctl->tempty[acc]);
            }
            if (++acc == TL::NACC) { acc = 0; acc_phase ^= 1u; }
        }
        if (lane == 0) bulk_wait_all();  // output stores complete before the CTA exits
        __syncwarp();
    }

    tc_fence_before();
    if (PAIR) {
        // After an abort, copies issued by either CTA may still be landing in
        // its shared memory: give them time (they finish within microseconds)
        // before the pair leaves.
        if (*(volatile int32_t *)abort_flag) {
            unsigned long long t0 = gtimer();
            while (gtimer() - t0 < 1000000ull) {
            }
        }
        cluster_sync();  // no MMA, copy or remote arrival of the pair in flight
        if (warp == 1) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(TMEM_COLS)
                         : "memory");
        }
    } else {
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(TMEM_COLS)
                         : "memory");
        }
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box box_rows x bk
// (bk = 64: 128-byte swizzle; bk = 32: 64-byte swizzle, also the epilogue's
// output staging; bk = 16: 32-byte swizzle).
bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              int bk, uint64_t pitch = 0) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {(pitch ? pitch : cols) * 2};   // row pitch in bytes
    cuuint32_t box[2] = {(cuuint32_t)bk, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    bk == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                    : bk == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                               : CU_TENSOR_MAP_SWIZZLE_32B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// An fp32 output map over a row-major [rows, cols] matrix, boxes of 32 rows
// x 16 columns (64-byte swizzle, the epilogue's staging pattern).
bool make_map_f32_out(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same over an e4m3 (byte) matrix, box box_rows x 128 (128-byte swizzle).
bool make_map_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 148;
    }
    return cached[dev];
}

// Resident clusters of `cl` CTAs of a kernel with this configuration (the
// GPCs bound how many clusters of ~200 KB-shared-memory CTAs fit at once).
template <typename K>
int max_clusters(K kern, size_t smem, int cl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void *)kern, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return sm_count() / cl;
    }
    return n;
}

template <int EPI, int TM, int BK, int CL, int TN, int EB = 2>
moe_status launch_gemm(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &b3,
                       const CUtensorMap &o, const GemmArgs &args_in, cudaStream_t stream,
                       const CUtensorMap *a_tail = nullptr, const CUtensorMap *b_tail = nullptr) {
    using TL = Tiling<TM, BK, CL, TN, EB>;
    GemmArgs args = args_in;
    args.stall = take_gemm_stall() ? 1 : 0;
    auto kern = tc_group_gemm<EPI, TM, BK, CL, TN, EB>;
    constexpr size_t SMEM = smem_bytes<TL>();
    static int units[64] = {0};  // resident CTAs (CL = 1) or clusters, per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    int nunits = dev >= 0 && dev < 64 ? units[dev] : 0;
    if (!nunits) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        nunits = CL > 1 ? max_clusters(kern, SMEM, CL) : sm_count();
        if (dev >= 0 && dev < 64) units[dev] = nunits;
    }
    constexpr int NOUT_TILE = is_swiglu(EPI) ? BN / 2 : BN * TN;
    const int64_t ntn = (args.n_out + NOUT_TILE - 1) / NOUT_TILE;
    int64_t upper = (int64_t)args.e * ((args.c_max + TL::BMT - 1) / TL::BMT) * ntn;
    int64_t grid = upper < nunits ? upper : nunits;
    if (grid < 1) grid = 1;
    if (CL == 1)
        return launch_pdl(kern, dim3((unsigned)grid), dim3(NUM_THREADS), SMEM, stream, a, b, b3, o,
                          a_tail ? *a_tail : a, b_tail ? *b_tail : b, args);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(CL * grid));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kern, a, b, b3, o, a_tail ? *a_tail : a,
                                         b_tail ? *b_tail : b, args);
    note_launch();
    if (err != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

}  // namespace

bool ffn_tc_supported(int e, int64_t c_max, int m, int h) {
    return e >= 1 && e <= MAX_E && (int64_t)e * c_max < ((int64_t)1 << 31) &&
           (int64_t)e * h * 2 < ((int64_t)1 << 31) && (int64_t)e * m < ((int64_t)1 << 31) &&
           m % 8 == 0 && h % 8 == 0;
}

moe_status ffn_tc_launch(const void *buf, const int32_t *counts, const int32_t *c_dev,
                         const void *w1, const void *b1, const void *w3, const void *w2,
                         const void *b2, moe_act act, int e, int64_t c_max, int m, int h,
                         void *hid, void *out, int32_t *st, cudaStream_t stream, int row_lo,
                         int row_hi, void *pre) {
    // fc1: 256-row tiles on CTA pairs (2-SM MMA), two accumulators per CTA so
    // its activation epilogue overlaps the next tile's main loop.
    // fc2 (bias-only epilogue, long K, about one tile per pair): 256 x 512
    // tiles on CTA pairs.
    constexpr int TM1 = 1, BK1 = 64, TM2 = 1, BK2 = 64;
    constexpr int CL1 = 2, CL2 = 2, TN2 = 2;
    using T1 = Tiling<TM1, BK1, CL1>;
    using T2 = Tiling<TM2, BK2, CL2, TN2>;
    CUtensorMap mA1, mB1, mB3, mA2, mB2, mO1, mO2;
    const bool swiglu = act == MOE_ACT_SWIGLU;
    // one CTA's B box: a pair CTA's half tile, or a 1-SM SwiGLU tile's W1/W3 half
    // one producer's B box: half of a CTA's B rows (1-SM SwiGLU: the W1 or W3 half)
    const uint32_t b1_box = T1::B_BOX_ROWS;
    if (!make_map(&mA1, buf, (uint64_t)e * c_max, (uint64_t)m, T1::A_BOX_ROWS, BK1) ||
        !make_map(&mB1, w1, (uint64_t)e * h, (uint64_t)m, b1_box, BK1) ||
        !make_map(&mB3, swiglu ? w3 : w1, (uint64_t)e * h, (uint64_t)m, b1_box, BK1) ||
        !make_map(&mA2, hid, (uint64_t)e * c_max, (uint64_t)h, T2::A_BOX_ROWS, BK2) ||
        !make_map(&mB2, w2, (uint64_t)e * m, (uint64_t)h, T2::B_BOX_ROWS, BK2) ||
        !make_map(&mO1, hid, (uint64_t)e * c_max, (uint64_t)h, 32, 32) ||
        !make_map(&mO2, out, (uint64_t)e * c_max, (uint64_t)m, 32, 32))
        return MOE_ERR_CUDA;
    GemmArgs g1{counts, c_dev, st, (const __nv_bfloat16 *)b1, (__nv_bfloat16 *)hid, c_max, e, m, h, h,
                nullptr, nullptr, row_lo, row_hi};
    g1.aux_out = (__nv_bfloat16 *)pre;   // training: fc1 also keeps its pre-activation
    moe_status r;
    if (swiglu) {
        r = pre ? launch_gemm<EPI_SWIGLU_SAVE, TM1, BK1, CL1, 1>(mA1, mB1, mB3, mO1, g1, stream)
                : launch_gemm<EPI_SWIGLU, TM1, BK1, CL1, 1>(mA1, mB1, mB3, mO1, g1, stream);
    } else if (act == MOE_ACT_GELU) {
        r = pre ? launch_gemm<EPI_GELU_SAVE, TM1, BK1, CL1, 1>(mA1, mB1, mB1, mO1, g1, stream)
                : launch_gemm<EPI_GELU, TM1, BK1, CL1, 1>(mA1, mB1, mB1, mO1, g1, stream);
    } else {
        r = pre ? launch_gemm<EPI_RELU_SAVE, TM1, BK1, CL1, 1>(mA1, mB1, mB1, mO1, g1, stream)
                : launch_gemm<EPI_RELU, TM1, BK1, CL1, 1>(mA1, mB1, mB1, mO1, g1, stream);
    }
    if (r != MOE_OK) return r;
    GemmArgs g2{counts, c_dev, st, (const __nv_bfloat16 *)b2, (__nv_bfloat16 *)out, c_max, e, h, m, m,
                nullptr, nullptr, row_lo, row_hi};
    return launch_gemm<EPI_BIAS, TM2, BK2, CL2, TN2>(mA2, mB2, mB2, mO2, g2, stream);
}

// ------------------------------------------------------------ e4m3 forward
moe_status quantize_rows_fp8_launch(const void *src, int64_t batches, int64_t rows_per_batch,
                                    int cols, const int32_t *counts, const int32_t *c_dev,
                                    void *q, float *scale, int32_t *st, cudaStream_t stream);

// The expert FFN on e4m3 operands with one fp32 scale per row: fc1 on the
// quantised rows and W1 (the same pair tiles as bf16, 128-element K blocks,
// kind::f8f6f4), the scales, bias and activation in the epilogue, bf16 hidden;
// the hidden rows quantised; fc2 likewise into bf16 out, on 256 x 256 pair
// tiles with two accumulators (with 128-element K blocks the main loop is
// short enough for the epilogue to show; measured 4% faster than 256 x 512
// on 8 experts, the same on 64).  ReLU / GELU only.
moe_status ffn_tc_fp8_launch(const void *buf_q, const float *buf_scale, const int32_t *counts,
                             const int32_t *c_dev, const void *w1_q, const float *w1_scale,
                             const void *b1, const void *w2_q, const float *w2_scale,
                             const void *b2, moe_act act, int e, int64_t c_max, int m, int h,
                             void *hid, void *hid_q, float *hid_scale, void *out, int32_t *st,
                             cudaStream_t stream) {
    constexpr int BKF = 128;   // e4m3 elements per K block (128 bytes)
    using T1 = Tiling<1, BKF, 2, 1, 1>;
    using T2 = Tiling<1, BKF, 2, 1, 1>;
    CUtensorMap mA1, mB1, mO1, mA2, mB2, mO2;
    if (!make_map_u8(&mA1, buf_q, (uint64_t)e * c_max, (uint64_t)m, T1::A_BOX_ROWS) ||
        !make_map_u8(&mB1, w1_q, (uint64_t)e * h, (uint64_t)m, T1::B_BOX_ROWS) ||
        !make_map(&mO1, hid, (uint64_t)e * c_max, (uint64_t)h, 32, 32) ||
        !make_map_u8(&mA2, hid_q, (uint64_t)e * c_max, (uint64_t)h, T2::A_BOX_ROWS) ||
        !make_map_u8(&mB2, w2_q, (uint64_t)e * m, (uint64_t)h, T2::B_BOX_ROWS) ||
        !make_map(&mO2, out, (uint64_t)e * c_max, (uint64_t)m, 32, 32))
        return MOE_ERR_CUDA;
    GemmArgs g1{counts, c_dev, st, (const __nv_bfloat16 *)b1, (__nv_bfloat16 *)hid, c_max, e, m, h, h,
                nullptr, nullptr, 0, 0, buf_scale, w1_scale};
    moe_status r = act == MOE_ACT_GELU
                       ? launch_gemm<EPI_GELU, 1, BKF, 2, 1, 1>(mA1, mB1, mB1, mO1, g1, stream)
                       : launch_gemm<EPI_RELU, 1, BKF, 2, 1, 1>(mA1, mB1, mB1, mO1, g1, stream);
    if (r != MOE_OK) return r;
    r = quantize_rows_fp8_launch(hid, e, c_max, h, counts, c_dev, hid_q, hid_scale, st, stream);
    if (r != MOE_OK) return r;
    GemmArgs g2{counts, c_dev, st, (const __nv_bfloat16 *)b2, (__nv_bfloat16 *)out, c_max, e, h, m, m,
                nullptr, nullptr, 0, 0, hid_scale, w2_scale};
    return launch_gemm<EPI_BIAS, 1, BKF, 2, 1, 1>(mA2, mB2, mB2, mO2, g2, stream);
}

}  // namespace moe

// The expert-FFN backward, appended after the forward (the code above is
// the forward GEMM unchanged).
#include "ffn_bwd.cuh"

namespace moe {

// ---------------------------------------------------------------- backward
// The expert-FFN backward as products on 256 x 256 pair tiles with two
// accumulators (each tile's epilogue overlaps the next tile's main loop, and
// a backward product has twice the tiles of a 256 x 512 tiling, so its last
// wave over the SM pairs is less empty), with the SIMT tail copies, bias sums
// and (SwiGLU) activation derivative in between:
//   d_hid = d_out w2                  (B = w2 read MN-major in place);
//   d_pre = d_hid * act'(buf w1^T + b1), the pre-activation recomputed in
//                                      the product's epilogue (SwiGLU: a =
//                                      buf w1^T and b = buf w3^T recomputed
//                                      and stored, then [d_a | d_b]); with
//                                      the forward's saved pre-activation,
//                                      d_pre = (d_out w2) * act'(pre) in one
//                                      product's epilogue instead;
//   d_buf = d_pre w1                  (B = w1 MN-major in place; SwiGLU:
//                                      [d_a | d_b] [w1; w3], both read MN-major
//                                      in place when h is a multiple of 64,
//                                      else against one K-major copy);
//   d_w2 = d_out^T hid, d_w1 = d_pre^T buf (d_w3 = d_b^T buf): the kept rows
//   are the contraction, each expert over its own (an expert with none gets
//   zeros), both operands read MN-major in place and each expert's partly
//   kept last 64-row block from a zero-padded copy;
//   d_b1, d_b2: column sums of d_pre, d_out over the kept rows.
namespace {

constexpr int64_t up256i(int64_t b) { return (b + 255) & ~(int64_t)255; }

struct BwdLayout {
    int64_t pa, pb, dh, dpre, wT, tDo, tHid, tDp, tBuf, total;
};

BwdLayout bwd_layout(moe_act act, int e, int64_t c_max, int m, int h) {
    const bool swiglu = act == MOE_ACT_SWIGLU;
    const int64_t E = e, H2 = swiglu ? 2 * (int64_t)h : h;
    BwdLayout L{};
    int64_t o = 0;
    auto take = [&](int64_t bytes) { const int64_t at = o; o += up256i(bytes); return at; };
    L.pa = take(swiglu ? E * c_max * h * 2 : 0);   // SwiGLU's recomputed a and b
    L.pb = take(swiglu ? E * c_max * h * 2 : 0);
    L.dh = take(E * c_max * h * 2);
    L.dpre = take(E * c_max * H2 * 2);
    L.wT = take(swiglu ? E * m * H2 * 2 : 0);   // [W1 | W3] transposed (SwiGLU only)
    // the partly kept last 64-row block of each expert's d_out, hid, d_pre, buf
    L.tDo = take(E * 64 * m * 2);
    L.tHid = take(E * 64 * h * 2);
    L.tDp = take(E * 64 * H2 * 2);
    L.tBuf = take(E * 64 * m * 2);
    L.total = o;
    return L;
}

// out[j] = A[j] B[j]^T (+ bias[j]) over the rows min(counts[j], *c_dev, c_max)
// of every expert j: A [e * c_max, K], B [e * b_rows, K], out [e, c_max, n_out].
moe_status gemm_bias(const void *a, const void *b, int b_rows, void *out, const void *bias,
                     const int32_t *counts, const int32_t *c_dev, int e, int64_t c_max, int K,
                     int n_out, int32_t *st, cudaStream_t stream) {
    using T2 = Tiling<1, 64, 2, 1>;
    CUtensorMap mA, mB, mO;
    if (!make_map(&mA, a, (uint64_t)e * c_max, (uint64_t)K, T2::A_BOX_ROWS, 64) ||
        !make_map(&mB, b, (uint64_t)e * b_rows, (uint64_t)K, T2::B_BOX_ROWS, 64) ||
        !make_map(&mO, out, (uint64_t)e * c_max, (uint64_t)n_out, 32, 32))
        return MOE_ERR_CUDA;
    GemmArgs g{counts, c_dev, st, (const __nv_bfloat16 *)bias, (__nv_bfloat16 *)out, c_max, e, K,
               n_out, b_rows, nullptr, nullptr, 0, 0};
    return launch_gemm<EPI_BIAS, 1, 64, 2, 1>(mA, mB, mB, mO, g, stream);
}

// The same with B MN-major: out[j] = A[j] B[j] with B [e * K, n_out] row-major
// (K rows per expert; rows past an expert's K meet zero columns of A).
moe_status gemm_bias_bmn(const void *a, const void *b, void *out, const int32_t *counts,
                         const int32_t *c_dev, int e, int64_t c_max, int K, int n_out, int32_t *st,
                         cudaStream_t stream) {
    using T2 = Tiling<1, 64, 2, 1>;
    CUtensorMap mA, mB, mO;
    if (!make_map(&mA, a, (uint64_t)e * c_max, (uint64_t)K, T2::A_BOX_ROWS, 64) ||
        !make_map(&mB, b, (uint64_t)e * K, (uint64_t)n_out, 64, 64) ||
        !make_map(&mO, out, (uint64_t)e * c_max, (uint64_t)n_out, 32, 32))
        return MOE_ERR_CUDA;
    GemmArgs g{counts, c_dev, st, nullptr, (__nv_bfloat16 *)out, c_max, e, K, n_out, K, nullptr,
               nullptr, 0, 0};
    return launch_gemm<EPI_BIAS_BMN, 1, 64, 2, 1>(mA, mB, mB, mO, g, stream);
}

// SwiGLU's d_buf = [d_a | d_b] [w1; w3]: A [e * c_max, 2h], B read MN-major
// from w1 for the first h K rows and from w3 for the next h (h a multiple of
// the 64-row K block, so no block straddles the two).
moe_status gemm_bias_bmn2(const void *a, const void *b1, const void *b3, void *out,
                          const int32_t *counts, const int32_t *c_dev, int e, int64_t c_max, int h,
                          int n_out, int32_t *st, cudaStream_t stream) {
    using T2 = Tiling<1, 64, 2, 1>;
    CUtensorMap mA, mB, mB3, mO;
    if (!make_map(&mA, a, (uint64_t)e * c_max, 2 * (uint64_t)h, T2::A_BOX_ROWS, 64) ||
        !make_map(&mB, b1, (uint64_t)e * h, (uint64_t)n_out, 64, 64) ||
        !make_map(&mB3, b3, (uint64_t)e * h, (uint64_t)n_out, 64, 64) ||
        !make_map(&mO, out, (uint64_t)e * c_max, (uint64_t)n_out, 32, 32))
        return MOE_ERR_CUDA;
    GemmArgs g{counts, c_dev, st, nullptr, (__nv_bfloat16 *)out, c_max, e, 2 * h, n_out, h, nullptr,
               nullptr, 0, 0};
    g.k_split = h;
    return launch_gemm<EPI_BIAS_BMN, 1, 64, 2, 1>(mA, mB, mB3, mO, g, stream);
}

// d_pre = d_hid * act'(buf w1^T + b1) over the kept rows (ReLU / GELU): the
// pre-activation recomputed on the fc1 tiling and differentiated in the
// epilogue, never stored.
moe_status gemm_dact(const void *buf, const void *w1, const void *b1, const void *d_hid, moe_act act,
                     void *d_pre, const int32_t *counts, const int32_t *c_dev, int e, int64_t c_max,
                     int m, int h, int32_t *st, cudaStream_t stream) {
    using T1 = Tiling<1, 64, 2, 1>;
    CUtensorMap mA, mB, mO;
    if (!make_map(&mA, buf, (uint64_t)e * c_max, (uint64_t)m, T1::A_BOX_ROWS, 64) ||
        !make_map(&mB, w1, (uint64_t)e * h, (uint64_t)m, T1::B_BOX_ROWS, 64) ||
        !make_map(&mO, d_pre, (uint64_t)e * c_max, (uint64_t)h, 32, 32))
        return MOE_ERR_CUDA;
    GemmArgs g{counts, c_dev, st, (const __nv_bfloat16 *)b1, (__nv_bfloat16 *)d_pre, c_max, e, m, h, h,
               nullptr, nullptr, 0, 0, nullptr, nullptr, (const __nv_bfloat16 *)d_hid};
    return act == MOE_ACT_GELU ? launch_gemm<EPI_DGELU, 1, 64, 2, 1>(mA, mB, mB, mO, g, stream)
                               : launch_gemm<EPI_DRELU, 1, 64, 2, 1>(mA, mB, mB, mO, g, stream);
}

// d_pre = (d_out w2) * act'(pre) over the kept rows (ReLU / GELU) with the
// forward's saved pre-activation: the data-gradient product reads w2
// MN-major and its epilogue applies the derivative; d_hid is never stored.
moe_status gemm_dact_bmn(const void *d_out, const void *w2, const void *pre, moe_act act, void *d_pre,
                         const int32_t *counts, const int32_t *c_dev, int e, int64_t c_max, int m,
                         int h, int32_t *st, cudaStream_t stream) {
    // 256 x 256 pair tiles with two accumulators: the derivative epilogue
    // (a load of the pre-activation and the GELU derivative per element)
    // overlaps the next tile's main loop
    using T2 = Tiling<1, 64, 2, 1>;
    CUtensorMap mA, mB, mO;
    if (!make_map(&mA, d_out, (uint64_t)e * c_max, (uint64_t)m, T2::A_BOX_ROWS, 64) ||
        !make_map(&mB, w2, (uint64_t)e * m, (uint64_t)h, 64, 64) ||
        !make_map(&mO, d_pre, (uint64_t)e * c_max, (uint64_t)h, 32, 32))
        return MOE_ERR_CUDA;
    GemmArgs g{counts, c_dev, st, nullptr, (__nv_bfloat16 *)d_pre, c_max, e, m, h, m, nullptr,
               nullptr, 0, 0, nullptr, nullptr, (const __nv_bfloat16 *)pre};
    return act == MOE_ACT_GELU ? launch_gemm<EPI_DGELU_BMN, 1, 64, 2, 1>(mA, mB, mB, mO, g, stream)
                               : launch_gemm<EPI_DRELU_BMN, 1, 64, 2, 1>(mA, mB, mB, mO, g, stream);
}

// SwiGLU with the forward's saved [a | b] rows: d_hid = d_out w2 (w2 read
// MN-major) and, in the epilogue, d_pre = [d_hid * b * silu'(a) | d_hid *
// silu(a)] ([e, c_max, 2h]); d_hid is never stored.
moe_status gemm_dswiglu_bmn(const void *d_out, const void *w2, const void *ab, void *d_pre,
                            const int32_t *counts, const int32_t *c_dev, int e, int64_t c_max, int m,
                            int h, int32_t *st, cudaStream_t stream) {
    using T2 = Tiling<1, 64, 2, 1>;
    CUtensorMap mA, mB, mO;
    if (!make_map(&mA, d_out, (uint64_t)e * c_max, (uint64_t)m, T2::A_BOX_ROWS, 64) ||
        !make_map(&mB, w2, (uint64_t)e * m, (uint64_t)h, 64, 64) ||
        // d_a: the first h columns of each 2h-wide row (the map's extent clips a
        // box at h, so d_b's columns are never written by it)
        !make_map(&mO, d_pre, (uint64_t)e * c_max, (uint64_t)h, 32, 32, 2 * (uint64_t)h))
        return MOE_ERR_CUDA;
    GemmArgs g{counts, c_dev, st, nullptr, (__nv_bfloat16 *)d_pre, c_max, e, m, h, m, nullptr,
               nullptr, 0, 0, nullptr, nullptr, (const __nv_bfloat16 *)ab};
    g.out_pitch = 2 * (int64_t)h;
    return launch_gemm<EPI_DSWIGLU_BMN, 1, 64, 2, 1>(mA, mB, mB, mO, g, stream);
}

// Weight gradients out[j] = A[j]^T B[j] over the first min(counts[j], *c_dev,
// c_max) rows of expert j, both operands read MN-major in place: A rows of
// a_cols columns at pitch a_pitch, B rows of b_cols at pitch b_pitch, c_max
// rows per expert; a_tail / b_tail [e, 64, *] (pitches a_tpitch / b_tpitch)
// hold each expert's partly kept last 64-row block (tail_rows_launch);
// out [e, a_cols, b_cols], bf16, or fp32 when out_f32.  Experts without kept
// rows are not written (their zero gradients come from
// zero_empty_experts_launch).
moe_status gemm_wgrad_mn(const void *a, int64_t a_pitch, int a_cols, const void *a_tail,
                         int64_t a_tpitch, const void *b, int64_t b_pitch, int b_cols,
                         const void *b_tail, int64_t b_tpitch, void *out, const int32_t *counts,
                         const int32_t *c_dev, int e, int64_t c_max, int32_t *st, cudaStream_t stream,
                         bool out_f32 = false) {
    CUtensorMap mA, mAt, mB, mBt, mO;
    if (!make_map(&mA, a, (uint64_t)e * c_max, (uint64_t)a_cols, 64, 64, (uint64_t)a_pitch) ||
        !make_map(&mAt, a_tail, (uint64_t)e * 64, (uint64_t)a_cols, 64, 64, (uint64_t)a_tpitch) ||
        !make_map(&mB, b, (uint64_t)e * c_max, (uint64_t)b_cols, 64, 64, (uint64_t)b_pitch) ||
        !make_map(&mBt, b_tail, (uint64_t)e * 64, (uint64_t)b_cols, 64, 64, (uint64_t)b_tpitch) ||
        !(out_f32 ? make_map_f32_out(&mO, out, (uint64_t)e * a_cols, (uint64_t)b_cols)
                  : make_map(&mO, out, (uint64_t)e * a_cols, (uint64_t)b_cols, 32, 32)))
        return MOE_ERR_CUDA;
    GemmArgs g{nullptr, nullptr, st, nullptr, (__nv_bfloat16 *)out, a_cols, e, (int)c_max, b_cols,
               (int)c_max, counts, c_dev, 0, 0};
    g.skip_empty = 1;   // the zero gradients of experts without kept rows: zero_empty_experts_launch
    if (out_f32) {   // fp32 boxes of 32 rows x 16 columns
        g.out_f32 = (float *)out;
        return launch_gemm<EPI_WGRAD_MN_F32, 1, 64, 2, 1>(mA, mB, mB, mO, g, stream, &mAt, &mBt);
    }
    return launch_gemm<EPI_WGRAD_MN, 1, 64, 2, 1>(mA, mB, mB, mO, g, stream, &mAt, &mBt);
}

}  // namespace

size_t ffn_tc_bwd_workspace_bytes(moe_act act, int e, int64_t c_max, int m, int h) {
    return (size_t)bwd_layout(act, e, c_max, m, h).total;
}

moe_status ffn_tc_bwd_launch(const void *buf, const void *hid, const int32_t *counts,
                             const int32_t *c_dev, const void *w1, const void *b1, const void *w3,
                             const void *w2, moe_act act, int e, int64_t c_max, int m, int h,
                             const void *d_out, void *ws, void *d_buf, void *d_w1, void *d_w3,
                             void *d_w2, void *d_b1, void *d_b2, int32_t *st, cudaStream_t stream,
                             const void *pre, bool wgrad_f32) {
    using bf = __nv_bfloat16;
    const bool swiglu = act == MOE_ACT_SWIGLU;
    const BwdLayout L = bwd_layout(act, e, c_max, m, h);
    const int64_t H2 = swiglu ? 2 * (int64_t)h : h;
    if (c_max > 0x7fffffff || H2 > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
    char *w = (char *)ws;
    bf *pa = (bf *)(w + L.pa), *pb = (bf *)(w + L.pb), *dh = (bf *)(w + L.dh);
    bf *dpre = (bf *)(w + L.dpre), *wT = (bf *)(w + L.wT);
    bf *tDo = (bf *)(w + L.tDo), *tHid = (bf *)(w + L.tHid), *tDp = (bf *)(w + L.tDp);
    bf *tBuf = (bf *)(w + L.tBuf);
    moe_status r;
#define MOE_TRY(x) \
    do {           \
        r = (x);   \
        if (r != MOE_OK) return r; \
    } while (0)
    // the data-gradient products read W2 (and W1 for ReLU / GELU) MN-major in
    // place; SwiGLU's [W1 | W3] contraction reads one K-major transposed copy
    // (experts without kept rows are skipped: no tile of theirs reads them)
    const bool swiglu_mn = swiglu && h % 64 == 0;   // [W1; W3] read MN-major in place
    if (swiglu && !swiglu_mn) {
        MOE_TRY(transpose_pad_launch((const bf *)w1, (int64_t)h * m, m, wT, (int64_t)m * H2, H2, e,
                                     h, m, h, nullptr, counts, c_dev, st, stream));
        MOE_TRY(transpose_pad_launch((const bf *)w3, (int64_t)h * m, m, wT + h, (int64_t)m * H2, H2,
                                     e, h, m, h, nullptr, counts, c_dev, st, stream));
    }
    // d_hid; then d_pre (ReLU / GELU: the pre-activation recomputed and
    // differentiated in one product; SwiGLU: a and b recomputed, then the
    // activation backward); then d_buf
    if (pre && swiglu) {
        // the forward's saved [a | b]: one product, d_hid never stored
        MOE_TRY(gemm_dswiglu_bmn(d_out, w2, pre, dpre, counts, c_dev, e, c_max, m, h, st, stream));
    } else if (pre) {
        // the forward's saved pre-activation: one product, d_hid never stored
        MOE_TRY(gemm_dact_bmn(d_out, w2, pre, act, dpre, counts, c_dev, e, c_max, m, h, st, stream));
    } else if (swiglu) {
        MOE_TRY(gemm_bias_bmn(d_out, w2, dh, counts, c_dev, e, c_max, m, h, st, stream));
        MOE_TRY(gemm_bias(buf, w1, h, pa, nullptr, counts, c_dev, e, c_max, m, h, st, stream));
        MOE_TRY(gemm_bias(buf, w3, h, pb, nullptr, counts, c_dev, e, c_max, m, h, st, stream));
        MOE_TRY(act_bwd_launch(pa, pb, dh, act, e, c_max, h, counts, c_dev, dpre, st, stream));
    } else {
        MOE_TRY(gemm_bias_bmn(d_out, w2, dh, counts, c_dev, e, c_max, m, h, st, stream));
        MOE_TRY(gemm_dact(buf, w1, b1, dh, act, dpre, counts, c_dev, e, c_max, m, h, st, stream));
    }
    if (swiglu_mn)
        MOE_TRY(gemm_bias_bmn2(dpre, w1, w3, d_buf, counts, c_dev, e, c_max, h, m, st, stream));
    else if (swiglu)
        MOE_TRY(gemm_bias(dpre, wT, m, d_buf, nullptr, counts, c_dev, e, c_max, (int)H2, m, st, stream));
    else
        MOE_TRY(gemm_bias_bmn(dpre, w1, d_buf, counts, c_dev, e, c_max, h, m, st, stream));
    // weight gradients: the kept rows are the contraction, each expert over
    // its own; both operands are read MN-major in place, the partly kept last
    // 64-row block of each expert from a zero-padded copy
    {
        TailOps tails{};
        tails.op[0] = TailOp{(const bf *)d_out, m, m, tDo};
        tails.op[1] = TailOp{(const bf *)hid, h, h, tHid};
        tails.op[2] = TailOp{dpre, H2, (int)H2, tDp};
        tails.op[3] = TailOp{(const bf *)buf, m, m, tBuf};
        MOE_TRY(tail_rows_launch(tails, 4, c_max, e, counts, c_dev, st, stream));
        // the weight gradients of experts without kept rows are zero: plain
        // stores at the HBM rate instead of the products' zero tiles
        const int64_t gb = wgrad_f32 ? 4 : 2;
        ZeroOps zo{};
        zo.op[0] = ZeroOp{d_w1, (int64_t)h * m * gb};
        zo.op[1] = ZeroOp{d_w2, (int64_t)m * h * gb};
        zo.op[2] = ZeroOp{d_w3, (int64_t)h * m * gb};
        MOE_TRY(zero_empty_experts_launch(zo, swiglu ? 3 : 2, c_max, e, counts, c_dev, st, stream));
    }
    MOE_TRY(gemm_wgrad_mn(d_out, m, m, tDo, m, hid, h, h, tHid, h, d_w2, counts, c_dev, e, c_max, st,
                          stream, wgrad_f32));
    MOE_TRY(gemm_wgrad_mn(dpre, H2, h, tDp, H2, buf, m, m, tBuf, m, d_w1, counts, c_dev, e, c_max,
                          st, stream, wgrad_f32));
    if (swiglu)
        MOE_TRY(gemm_wgrad_mn(dpre + h, H2, h, tDp + h, H2, buf, m, m, tBuf, m, d_w3, counts, c_dev,
                              e, c_max, st, stream, wgrad_f32));
    // bias gradients (ReLU / GELU experts), both in one launch
    if (!swiglu && d_b1 && d_b2)
        MOE_TRY(colsum_launch(dpre, e, c_max, h, h, counts, c_dev, d_b1, st, stream, wgrad_f32,
                              (const bf *)d_out, m, m, d_b2));
    else if (!swiglu && d_b1)
        MOE_TRY(colsum_launch(dpre, e, c_max, h, h, counts, c_dev, d_b1, st, stream, wgrad_f32));
    else if (!swiglu && d_b2)
        MOE_TRY(colsum_launch((const bf *)d_out, e, c_max, m, m, counts, c_dev, d_b2, st, stream,
                              wgrad_f32));
#undef MOE_TRY
    return MOE_OK;
}

}  // namespace moe
