// common.cuh -- device helpers shared by the libmoefp8 kernels (sm_103a only).
//
// Number formats follow the readings stated in include/moefp8.h: OCP e4m3fn codes produced by
// the hardware round-to-nearest-even, saturating convert; BF16 round to nearest even; the
// per-128-group scale max(amax, 1e-10)/448 (UE8M0: rounded up to a power of two); quantised
// values by IEEE division.  The SiLU exponential is one fixed fp32 algorithm written with
// explicit round-to-nearest intrinsics so that no contraction or fast-math substitution can
// change a bit: Cody & Waite reduction by ln 2 (W. J. Cody, W. Waite, "Software Manual for the
// Elementary Functions", 1980) and the degree-7 Taylor polynomial of e^r in Horner form.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moefp8.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libmoefp8 is built for sm_103a only"
#endif

namespace moe {

// ---------------------------------------------------------------------------------------------
// host side: error text, per-device status word, SM count
// ---------------------------------------------------------------------------------------------
void set_error(const char* fmt, ...);
void clear_error();
int* device_status_ptr();     // device address of the current device's status word (or null)
int sm_count();               // SMs of the current device
bool device_is_sm103();
// Raises a kernel's dynamic shared-memory limit to at least `bytes` (cached per device).
bool ensure_smem(const void* func, int bytes);

// Launch helpers shared by the translation units (implemented next to their kernels).
int launch_act_quant(moe_act act, const void* in, moe_dtype in_dtype, int in_splits, int in_rows,
                     int rows, int N, float clamp_limit, moe_scale_fmt fmt,
                     const int32_t* row_expert, const int32_t* expert_map, int E,
                     const int32_t* row_map, int row_div, int out_rows, uint8_t* out_q,
                     float* out_s, moe_quant_strategy strategy, bool pdl, cudaStream_t stream,
                     bool map_early = false, const int32_t* slot_route = nullptr,
                     const int32_t* n_blocks = nullptr, int bm = 0, const int32_t* n_rows = nullptr,
                     bool early_release = false);
// Per-token input quantisation scattered to the route slots (the layer's first stage).
int launch_input_quant_tokens(const void* x, int M, int H, int k, const int32_t* route_slot,
                              int slots, uint8_t* xq, float* xs, moe_scale_fmt fmt, bool pdl,
                              cudaStream_t stream, const int32_t* pad_offset = nullptr,
                              const int32_t* pad_count = nullptr, int32_t* pad_sorted = nullptr,
                              int pad_E = 0, bool late_release = false);
int launch_route_prepare(const int32_t* topk_ids, int M, int k, int E, const int32_t* expert_map,
                         int E_local, int block_m, moe_route_path path, int32_t* sorted_idx,
                         int32_t* block_expert, int32_t* num_blocks, int32_t* expert_count,
                         int32_t* expert_offset, int32_t* route_slot, void* workspace,
                         size_t ws_bytes, bool pdl, cudaStream_t stream,
                         uint32_t* zero_ptr = nullptr, int zero_n = 0, bool skip_pads = false,
                         int32_t* kept_slot = nullptr, int32_t* n_kept = nullptr);
// Whether AUTO route preparation takes its compacting single-CTA path (which alone writes the
// kept-slot list and count).
bool route_compacts(int R, int E, int E_local, bool map);
size_t route_workspace_bytes(int R, int E_local, int block_m);
bool route_single_cta(int R, int E_local, moe_route_path path);
// The weighted top-k sum done in the down GEMM's epilogue (see GemmArgs in grouped_gemm.cu).
struct EpilogueReduce {
    void* out;            // [M, N_out] bf16
    unsigned* cnt;        // [M, N_out/128] arrival counters, zero before the launch
    const float* w;       // [M, k]
    const int32_t* slot;  // route_slot [M*k]
    int k, M;
};
int launch_grouped_gemm(moe_proj proj, const uint8_t* a_q, const float* a_s, int a_rows, int K,
                        const uint8_t* w_q, const float* w_s, int E_local, int N_out,
                        moe_weight_layout w_layout, const int32_t* sorted_idx, const int32_t* block_expert,
                        const int32_t* num_blocks, int B_cap, int block_m, void* out,
                        moe_dtype out_dtype, int out_rows, int splits, bool pdl,
                        cudaStream_t stream, bool wait_first = false,
                        const int32_t* self_ids = nullptr, const int32_t* self_map = nullptr,
                        int self_R = 0, int self_E = 0, const EpilogueReduce* red = nullptr,
                        unsigned long long* sched = nullptr);
// Largest route count for which the gate/up GEMM derives its block table itself.
constexpr int kSelfRouteMaxRoutes = 32;
// Largest route count route preparation sorts in one warp (AUTO path).
constexpr int kRouteWarpMaxRoutes = 32;
int launch_moe_reduce(const void* z, const float* topk_w, const int32_t* topk_ids,
                      const int32_t* expert_map, int M, int k, int E, int E_local, int H, void* out,
                      bool pdl, cudaStream_t stream);
constexpr int kReduceMaxTopk = 32;  // top-k limit of the separate reduce kernel (a route per lane)

// The fused layer kernel (everything after route preparation in one persistent launch).
struct FusedLaunch {
    const void* x;                 // [M, H] bf16
    const int32_t* topk_ids;       // [M, k]
    const float* topk_w;           // [M, k]
    const int32_t* expert_map;     // [E] or null
    int M, k, E, E_local, H, N, bm, B_cap, slots;
    const uint8_t* wgu_q;
    const float* wgu_s;
    const uint8_t* wd_q;
    const float* wd_s;
    moe_weight_layout w_layout;
    int act;
    float clamp_limit;
    int fmt;
    const int32_t* sorted_idx;     // route preparation outputs
    const int32_t* block_expert;
    const int32_t* num_blocks;
    const int32_t* route_slot;
    uint8_t* xq;                   // [slots, H]
    float* xsT;                    // [H/128, slots]
    float* gu;                     // fused_partial_bytes(...)
    uint8_t* aq;                   // [slots, N]
    float* asT;                    // [N/128, slots]
    void* z;                       // [M*k, H] bf16
    void* out;                     // [M, H] bf16
    unsigned* sync;                // fused_counter_words(B_cap) words, zeroed by route preparation
};
int launch_fused_layer(const FusedLaunch& f, cudaStream_t stream);
size_t fused_partial_bytes(int B_cap, int bm, int H, int N, int G);
int fused_counter_words(int B_cap);

// 2-D TMA map over a row-major [rows, cols] byte matrix: box 128 columns x box_rows rows,
// 128-byte swizzle (the K-major operand layout the MMA descriptors expect).
bool make_tma_map_u8(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sets up a launch config with programmatic dependent launch when `pdl` is set: the kernel may
// begin while its predecessor on the stream finishes; it waits (griddepcontrol.wait) before
// touching anything the predecessor writes.
struct Launch {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    Launch(dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl) {
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 0;
        if (pdl) {
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.numAttrs = 1;
        }
    }
};

// ---------------------------------------------------------------------------------------------
// device side
// ---------------------------------------------------------------------------------------------
// Wait for the grid this launch depends on (no-op without programmatic dependent launch).
__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next launch on the stream to start its prologue.
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16 bits, round to nearest even (NaN stays NaN).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return ((u >> 16) & 0x8000u) | 0x7FC0u;
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}
__device__ __forceinline__ float bf16_round_f32(float x) {
    return __uint_as_float(f32_to_bf16_bits(x) << 16);
}

// Two fp32 -> two e4m3 codes (RNE, saturating); `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float pow2_int(int n) {  // n in [-126, 127]
    return __uint_as_float(static_cast<uint32_t>(n + 127) << 23);
}

// e^x in fp32 (see the file header for the algorithm).
__device__ __forceinline__ float exp_f32(float x) {
    if (isnan(x)) return x;
    if (x > 89.0f) return __uint_as_float(0x7F800000u);
    if (x < -104.0f) return 0.0f;
    const float kLog2e = (float)1.44269504088896340736;
    const float kLn2Hi = (float)0.69314718055994530942;
    const float kLn2Lo = (float)(0.69314718055994530942 - (double)(float)0.69314718055994530942);
    float n = rintf(__fmul_rn(x, kLog2e));
    float r = __fmaf_rn(-n, kLn2Hi, x);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = (float)(1.0 / 5040.0);
    p = __fmaf_rn(p, r, (float)(1.0 / 720.0));
    p = __fmaf_rn(p, r, (float)(1.0 / 120.0));
    p = __fmaf_rn(p, r, (float)(1.0 / 24.0));
    p = __fmaf_rn(p, r, (float)(1.0 / 6.0));
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    int ni = static_cast<int>(n);
    int n1 = ni / 2, n2 = ni - n1;
    return __fmul_rn(__fmul_rn(p, pow2_int(n1)), pow2_int(n2));
}

// a = bf16(SiLU(g) * u) after the optional clamp; returned as the fp32 value of that bf16.
template <int ACT>
__device__ __forceinline__ float silu_mul_bf16(float g, float u, float L) {
    if (ACT == MOE_ACT_SILU_MUL) { g = fminf(fmaxf(g, -L), L); u = fminf(fmaxf(u, -L), L); }
    if (ACT == MOE_ACT_SILU_MUL_GATE_UPPER) { g = fminf(g, L); u = fminf(fmaxf(u, -L), L); }
    float e = exp_f32(-g);
    float s = __fdiv_rn(g, __fadd_rn(1.0f, e));
    return bf16_round_f32(__fmul_rn(s, u));
}

// The same SiLU*mul as silu_mul_bf16<act>, with the activation chosen at run time and the code
// kept out of line: one copy, for paths that run once per kernel, where instruction fetch and
// not arithmetic dominates.  Identical arithmetic, operation for operation.
static __device__ __noinline__ float silu_mul_bf16_rt(float g, float u, float L, int act) {
    if (act == MOE_ACT_SILU_MUL) g = fmaxf(g, -L);
    g = fminf(g, L);
    u = fminf(fmaxf(u, -L), L);
    const float e = exp_f32(-g);
    const float s = __fdiv_rn(g, __fadd_rn(1.0f, e));
    return bf16_round_f32(__fmul_rn(s, u));
}

// Group scale from the group's amax.
__device__ __forceinline__ float group_scale(float amax, int fmt) {
    float s = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
    if (fmt == MOE_SCALE_UE8M0) {
        uint32_t b = __float_as_uint(s);
        uint32_t e = (b >> 23) & 0xFFu;
        if (b & 0x7FFFFFu) e += 1u;
        s = __uint_as_float(e << 23);
    }
    return s;
}

// a / s as the quantiser needs it: IEEE division for fp32 scales; for power-of-two scales the
// product with the exact reciprocal is the same correctly rounded value.
__device__ __forceinline__ float quant_div(float a, float s, float inv_pow2, int fmt) {
    return fmt == MOE_SCALE_UE8M0 ? __fmul_rn(a, inv_pow2) : __fdiv_rn(a, s);
}
__device__ __forceinline__ float pow2_reciprocal(float s) {  // s = 2^e, e in [-126, 126]
    uint32_t e = (__float_as_uint(s) >> 23) & 0xFFu;
    return __uint_as_float((254u - e) << 23);
}

// Half-warp quantisation of one 128-wide group: lane l of the half-warp holds the 8 values at
// columns 8l..8l+7 (already materialised as BF16 values in fp32).  Every lane of the warp must
// call this (the amax reduction uses full-mask xor shuffles that stay inside each half-warp).
// Active lanes get their 8 E4M3 codes packed in *codes and the group scale in *scale.
__device__ __forceinline__ void quant_group_codes(const float* a, bool active, int fmt,
                                                  uint2* codes, float* scale) {
    float amax = 0.0f;
    if (active) {
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(a[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 8));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    if (active) {
        const float s = group_scale(amax, fmt);
        const float inv = fmt == MOE_SCALE_UE8M0 ? pow2_reciprocal(s) : 0.0f;
        uint32_t c0 = cvt_e4m3x2(quant_div(a[0], s, inv, fmt), quant_div(a[1], s, inv, fmt));
        uint32_t c1 = cvt_e4m3x2(quant_div(a[2], s, inv, fmt), quant_div(a[3], s, inv, fmt));
        uint32_t c2 = cvt_e4m3x2(quant_div(a[4], s, inv, fmt), quant_div(a[5], s, inv, fmt));
        uint32_t c3 = cvt_e4m3x2(quant_div(a[6], s, inv, fmt), quant_div(a[7], s, inv, fmt));
        *codes = make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
        *scale = s;
    }
}

// Two E4M3 codes of a / s (the quantiser of quant_group_codes), out of line.
static __device__ __noinline__ uint32_t quant_pair_rt(float a0, float a1, float s, float inv, int fmt) {
    return cvt_e4m3x2(quant_div(a0, s, inv, fmt), quant_div(a1, s, inv, fmt));
}

// quant_group_codes with its per-value work out of line (same arithmetic and results).
__device__ __forceinline__ void quant_group_codes_compact(const float* a, bool active, int fmt,
                                                          uint2* codes, float* scale) {
    float amax = 0.0f;
    if (active) {
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(a[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 8));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    if (active) {
        const float s = group_scale(amax, fmt);
        const float inv = fmt == MOE_SCALE_UE8M0 ? pow2_reciprocal(s) : 0.0f;
        const uint32_t c0 = quant_pair_rt(a[0], a[1], s, inv, fmt);
        const uint32_t c1 = quant_pair_rt(a[2], a[3], s, inv, fmt);
        const uint32_t c2 = quant_pair_rt(a[4], a[5], s, inv, fmt);
        const uint32_t c3 = quant_pair_rt(a[6], a[7], s, inv, fmt);
        *codes = make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
        *scale = s;
    }
}

// ---------------------------------------------------------------------------------------------
// mbarrier / TMA / tcgen05 wrappers (PTX ISA, sm_100-family instructions)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Arrive without release semantics: for a consumer that only signals it has finished READING a
// buffer (its loads have completed -- their values are in registers), so the arrive need not
// wait for the thread's earlier global stores to become visible.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after `limit` ns (global timer; ~2 s by default) or as soon as another
// role of the CTA has given up (*abort != 0); on a timeout it records MOE_DEV_TIMEOUT in the
// status word.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
static __device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                       int* status, uint64_t limit = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit) {
                if (status) atomicOr(status, MOE_DEV_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// Inline fast path: one try_wait, then the bounded slow path.
__device__ __forceinline__ bool mbar_wait_fast(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait(bar, parity, abort, status);
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled TMA load into shared memory, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 -> fp32, one CTA.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every previously issued tcgen05.mma of this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Instruction descriptor, kind::f8f6f4: D fp32, A and B E4M3, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f8_f32(int M, int N) {
    return (1u << 4)                                   // D format: f32
           | (0u << 7) | (0u << 10)                    // A, B format: E4M3
           | (0u << 15) | (0u << 16)                   // A, B K-major
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}
// Shared-memory matrix descriptor: K-major operand written by TMA with 128-byte swizzle, rows
// of 128 bytes, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu)
           | (static_cast<uint64_t>(16 >> 4) << 16)     // leading byte offset (unused here)
           | (static_cast<uint64_t>(1024 >> 4) << 32)   // stride byte offset: next 8 rows
           | (1ull << 46)                               // descriptor version (sm_100 family)
           | (2ull << 61);                              // swizzle: 128 B
}

// 32 lanes x 32 columns of fp32 from tensor memory, waited on in the same statement.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace moe
