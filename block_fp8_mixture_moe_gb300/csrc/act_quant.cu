// act_quant.cu -- fused (optionally clamped) SiLU-and-mul + per-128-group dynamic E4M3
// quantisation, and the input quantisation (identity activation) that feeds the W8A8 gate/up
// GEMM.
//
// Method: vLLM PR #53875 "Fuse clamped MoE activation and UE8M0 FP8 block quantization",
// section "Purpose" (clamp, BF16 SiLU and gated multiplication, dynamic E4M3 block
// quantisation with optional UE8M0 scales, optional filtering of invalid or non-local rows);
// lmdeploy PR #4956 "Perf/pytorch block fp8 moe decode", section "Fused SwiGLU and FP8
// quantization" (no BF16 intermediate in memory; bitwise equal to the two-kernel path).
//
// Layout of the work: one half-warp (16 lanes) owns one 128-wide quant group; every lane loads
// 8 BF16 gate values and 8 BF16 up values with one 16-byte load each (or 2x16-byte loads per
// split for fp32 split-K partials), materialises the 8 BF16 activations in registers, and the
// group amax is a 4-step xor-shuffle reduction inside the half-warp.  Each lane then stores its
// 8 E4M3 codes as one 8-byte store (128 contiguous bytes per group) and lane 0 of the half-warp
// stores the group scale.  A warp always processes a pair of groups, so both halves run the
// same loop and the full-mask shuffles never see a divergent partner.
//
// Two launch shapes (the pages' two strategies): PER_GROUP -- one warp per group pair, no loop,
// for launch-bound decode shapes without a filter; PERSISTENT -- a grid of as many CTAs as are
// resident at once that strides over the group pairs, for filtered (expert-parallel) inputs,
// row maps and large outputs.
#include "common.cuh"

#include <algorithm>

namespace moe {
namespace {

struct AQArgs {
    const void* in;
    long long split_stride;  // elements between fp32 split partials
    int in_rows;
    int rows, N, G, W;
    float L;
    int fmt;
    const int32_t* row_expert;
    const int32_t* expert_map;
    int E;
    const int32_t* row_map;
    int row_div;
    int out_rows;
    uint8_t* out_q;
    float* out_s;
    int in_splits;
    int map_early;  // row_map was written two or more launches back: read it before the wait
    int map_smem;   // stage expert_map ([E] ints) in shared memory (persistent launches)
    // slot rows: row w is produced iff slot_route[w] >= 0 (input and output row w), and only
    // rows below n_blocks[0] * bm exist (n_blocks read on the device)
    const int32_t* slot_route;
    const int32_t* n_blocks;
    int bm;
    // nullable: the number of work rows, read on the device (rows is then an upper bound)
    const int32_t* n_rows;
    int* status;
    // release the next launch before this kernel's dependency wait (see launch_act_quant)
    int early_release;
};

// Loads 8 consecutive inputs as fp32 values of their BF16 materialisation.
template <bool F32IN>
__device__ __forceinline__ void load8(const AQArgs& p, long long off, float* v) {
    if (!F32IN) {
        uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.in) + off));
        v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
        v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
    } else {
        // split-K partials: summed in split order in fp32, then rounded to BF16 once
        const float* base = static_cast<const float*>(p.in) + off;
        float4 a = __ldg(reinterpret_cast<const float4*>(base));
        float4 b = __ldg(reinterpret_cast<const float4*>(base) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        // splits 1.. in groups of four: the eight loads of a group are issued together, the
        // additions still run strictly in split order
        int s = 1;
        for (; s + 3 < p.in_splits; s += 4) {
            float4 c[4], d[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float* q = base + (s + t) * p.split_stride;
                c[t] = __ldg(reinterpret_cast<const float4*>(q));
                d[t] = __ldg(reinterpret_cast<const float4*>(q) + 1);
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                v[0] = __fadd_rn(v[0], c[t].x); v[1] = __fadd_rn(v[1], c[t].y);
                v[2] = __fadd_rn(v[2], c[t].z); v[3] = __fadd_rn(v[3], c[t].w);
                v[4] = __fadd_rn(v[4], d[t].x); v[5] = __fadd_rn(v[5], d[t].y);
                v[6] = __fadd_rn(v[6], d[t].z); v[7] = __fadd_rn(v[7], d[t].w);
            }
        }
        for (; s < p.in_splits; ++s) {
            const float* q = base + s * p.split_stride;
            float4 c = __ldg(reinterpret_cast<const float4*>(q));
            float4 d = __ldg(reinterpret_cast<const float4*>(q) + 1);
            v[0] = __fadd_rn(v[0], c.x); v[1] = __fadd_rn(v[1], c.y);
            v[2] = __fadd_rn(v[2], c.z); v[3] = __fadd_rn(v[3], c.w);
            v[4] = __fadd_rn(v[4], d.x); v[5] = __fadd_rn(v[5], d.y);
            v[6] = __fadd_rn(v[6], d.z); v[7] = __fadd_rn(v[7], d.w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = bf16_round_f32(v[i]);
    }
}

// The gate and up inputs of one lane (8 values each).  For fp32 split-K partials the loads of
// up to KG splits of both operands are in flight together, so a row with S splits costs
// ceil(S / KG) dependent round trips to memory; the additions still run strictly in split
// order, starting from split 0.  KG follows the split count: the registers of the in-flight
// loads bound how many warps an SM holds, and this kernel is latency-bound.
template <bool F32IN, int KG>
__device__ __forceinline__ void load_gate_up(const AQArgs& p, long long off_g, long long off_u,
                                             float* g, float* u) {
    if (!F32IN) {
        load8<false>(p, off_g, g);
        load8<false>(p, off_u, u);
        return;
    }
    constexpr int kGroup = KG;
    const float* bg = static_cast<const float*>(p.in) + off_g;
    const float* bu = static_cast<const float*>(p.in) + off_u;
    for (int s0 = 0; s0 < p.in_splits; s0 += kGroup) {
        float4 cg[kGroup][2], cu[kGroup][2];
#pragma unroll
        for (int t = 0; t < kGroup; ++t) {
            if (s0 + t < p.in_splits) {
                const long long so = static_cast<long long>(s0 + t) * p.split_stride;
                const float4* qg = reinterpret_cast<const float4*>(bg + so);
                const float4* qu = reinterpret_cast<const float4*>(bu + so);
                cg[t][0] = __ldg(qg); cg[t][1] = __ldg(qg + 1);
                cu[t][0] = __ldg(qu); cu[t][1] = __ldg(qu + 1);
            }
        }
#pragma unroll
        for (int t = 0; t < kGroup; ++t) {
            if (s0 + t < p.in_splits) {
                const float vg[8] = {cg[t][0].x, cg[t][0].y, cg[t][0].z, cg[t][0].w,
                                     cg[t][1].x, cg[t][1].y, cg[t][1].z, cg[t][1].w};
                const float vu[8] = {cu[t][0].x, cu[t][0].y, cu[t][0].z, cu[t][0].w,
                                     cu[t][1].x, cu[t][1].y, cu[t][1].z, cu[t][1].w};
                if (s0 + t == 0) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) { g[i] = vg[i]; u[i] = vu[i]; }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) { g[i] = __fadd_rn(g[i], vg[i]); u[i] = __fadd_rn(u[i], vu[i]); }
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) { g[i] = bf16_round_f32(g[i]); u[i] = bf16_round_f32(u[i]); }
}

// Decides whether work row `w` is produced, and its input and output rows.  `pre` is the row's
// entry of its first selector (row_expert if given, else row_map) when it was loaded ahead
// (-2: not loaded); smap is the expert map staged in shared memory (or null).
__device__ __forceinline__ bool row_source(const AQArgs& p, int w, int* in_row, int* out_row,
                                           int pre = -2, const int* smap = nullptr) {
    int src = w, dst = w;
    if (p.slot_route && __ldcg(p.slot_route + w) < 0) return false;
    if (p.row_expert) {
        const int id = pre != -2 ? pre : __ldg(p.row_expert + w);
        if (id < 0 || id >= p.E) return false;
        if (p.expert_map && (smap ? smap[id] : __ldg(p.expert_map + id)) < 0) return false;
    }
    if (p.row_map) {
        const int m = (pre != -2 && !p.row_expert) ? pre : __ldg(p.row_map + w);
        if (m < 0) return false;
        dst = m;
        src = p.row_div > 0 ? w / p.row_div : m;
    }
    if (src >= p.in_rows || dst >= p.out_rows) {
        if (p.status) atomicOr(p.status, MOE_DEV_BAD_INDEX);
        return false;
    }
    *in_row = src;
    *out_row = dst;
    return true;
}

// The gate and up inputs of one lane, 4 values each (the layer's few-item shape below): BF16
// (one 8-byte load per operand), or fp32 split-K partials with the same loads in flight
// together and additions in split order as load_gate_up.
template <bool F32IN, int KG>
__device__ __forceinline__ void load_gate_up4(const AQArgs& p, long long off_g, long long off_u,
                                              float* g, float* u) {
    if constexpr (!F32IN) {
        const uint2 wg = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.in) + off_g));
        const uint2 wu = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.in) + off_u));
        g[0] = bf16_lo(wg.x); g[1] = bf16_hi(wg.x); g[2] = bf16_lo(wg.y); g[3] = bf16_hi(wg.y);
        u[0] = bf16_lo(wu.x); u[1] = bf16_hi(wu.x); u[2] = bf16_lo(wu.y); u[3] = bf16_hi(wu.y);
        return;
    }
    const float* bg = static_cast<const float*>(p.in) + off_g;
    const float* bu = static_cast<const float*>(p.in) + off_u;
    for (int s0 = 0; s0 < p.in_splits; s0 += KG) {
        float4 cg[KG], cu[KG];
#pragma unroll
        for (int t = 0; t < KG; ++t) {
            if (s0 + t < p.in_splits) {
                const long long so = static_cast<long long>(s0 + t) * p.split_stride;
                cg[t] = __ldg(reinterpret_cast<const float4*>(bg + so));
                cu[t] = __ldg(reinterpret_cast<const float4*>(bu + so));
            }
        }
#pragma unroll
        for (int t = 0; t < KG; ++t) {
            if (s0 + t < p.in_splits) {
                const float vg[4] = {cg[t].x, cg[t].y, cg[t].z, cg[t].w};
                const float vu[4] = {cu[t].x, cu[t].y, cu[t].z, cu[t].w};
                if (s0 + t == 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) { g[i] = vg[i]; u[i] = vu[i]; }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) { g[i] = __fadd_rn(g[i], vg[i]); u[i] = __fadd_rn(u[i], vu[i]); }
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) { g[i] = bf16_round_f32(g[i]); u[i] = bf16_round_f32(u[i]); }
}

// quant_group_codes for a group spread over a whole warp, 4 values a lane (same scale rule and
// quantiser); the 4 codes of a lane come back in one word, lowest column in the low byte.
__device__ __forceinline__ void quant_group_codes4(const float* a, bool active, int fmt,
                                                   uint32_t* codes, float* scale) {
    float amax = 0.0f;
    if (active) {
#pragma unroll
        for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(a[i]));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
    if (active) {
        const float s = group_scale(amax, fmt);
        const float inv = fmt == MOE_SCALE_UE8M0 ? pow2_reciprocal(s) : 0.0f;
        const uint32_t c0 = cvt_e4m3x2(quant_div(a[0], s, inv, fmt), quant_div(a[1], s, inv, fmt));
        const uint32_t c1 = cvt_e4m3x2(quant_div(a[2], s, inv, fmt), quant_div(a[3], s, inv, fmt));
        *codes = c0 | (c1 << 16);
        *scale = s;
    }
}

template <int ACT, bool F32IN, int KG, bool INL>
__device__ __forceinline__ void quant_pair(const AQArgs& p, long long pair, int lane, int pre = -2,
                                           const int* smap = nullptr) {
    const int half = lane >> 4, l = lane & 15;
    const long long item = pair * 2 + half;
    bool active = item < static_cast<long long>(p.rows) * p.G;
    int row = 0, g = 0, in_row = 0;
    // slot rows with no other filter or map: the slot's route entry is loaded together with
    // the slot's inputs (one round trip, not two), and a pad slot's values are dropped after
    const bool slot_walk = p.slot_route && !p.row_expert && !p.row_map;
    int route = 0;
    if (active) {
        const int w = static_cast<int>(static_cast<unsigned>(item) / static_cast<unsigned>(p.G));
        g = static_cast<int>(item - static_cast<long long>(w) * p.G);
        if (slot_walk) {
            in_row = row = w;
            if (w >= p.in_rows || w >= p.out_rows) {
                if (p.status) atomicOr(p.status, MOE_DEV_BAD_INDEX);
                active = false;
            } else {
                route = __ldcg(p.slot_route + w);
            }
        } else {
            active = row_source(p, w, &in_row, &row, pre, smap);
        }
    }
    float a[8];
    if (active) {
        const long long col = static_cast<long long>(g) * 128 + l * 8;
        const long long rbase = static_cast<long long>(in_row) * p.W;
        float gv[8], uv[8];
        if (ACT == MOE_ACT_IDENTITY)
            load8<F32IN>(p, rbase + col, a);
        else
            load_gate_up<F32IN, KG>(p, rbase + col, rbase + p.N + col, gv, uv);
        if (slot_walk && route < 0) active = false;  // a pad slot
        // INL: inline, so the 8 values' dependent chains (exp, IEEE divide) interleave;
        // else one out-of-line copy (same arithmetic), less code for many warps to fetch
        if constexpr (ACT != MOE_ACT_IDENTITY) {
            if (active) {
                if constexpr (INL) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = silu_mul_bf16<ACT>(gv[i], uv[i], p.L);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = silu_mul_bf16_rt(gv[i], uv[i], p.L, ACT);
                }
            }
        }
    }
    const long long o = static_cast<long long>(row) * p.N + static_cast<long long>(g) * 128 + l * 8;
    uint2 codes;
    float sc;
    if constexpr (INL)
        quant_group_codes(a, active, p.fmt, &codes, &sc);
    else
        quant_group_codes_compact(a, active, p.fmt, &codes, &sc);
    if (active) {
        *reinterpret_cast<uint2*>(p.out_q + o) = codes;
        if (l == 0) p.out_s[static_cast<long long>(row) * p.G + g] = sc;
    }
}

// One (row, 128-column group) item with a whole warp, 4 values a lane: the work row and its
// selector as in quant_pair, SiLU*mul inlined.  Per lane it is half of quant_pair's chain of
// loads, SiLU and quantisation, which shortens the layer's act-quant where one warp per SM does
// the work (decode batches); where the SMs are full of warps (expert-parallel and prefill
// shapes) the per-item overhead over 4 values instead of 8 makes it slower, so the launcher
// takes it only for few items.
template <int ACT, bool F32IN, int KG>
__device__ __forceinline__ void quant_item4(const AQArgs& p, long long item, int lane, int pre,
                                            const int* smap) {
    bool active = item < static_cast<long long>(p.rows) * p.G;
    int row = 0, g = 0, in_row = 0;
    const bool slot_walk = p.slot_route && !p.row_expert && !p.row_map;
    int route = 0;
    if (active) {
        const int w = static_cast<int>(static_cast<unsigned>(item) / static_cast<unsigned>(p.G));
        g = static_cast<int>(item - static_cast<long long>(w) * p.G);
        if (slot_walk) {
            in_row = row = w;
            if (w >= p.in_rows || w >= p.out_rows) {
                if (p.status) atomicOr(p.status, MOE_DEV_BAD_INDEX);
                active = false;
            } else {
                route = __ldcg(p.slot_route + w);
            }
        } else {
            active = row_source(p, w, &in_row, &row, pre, smap);
        }
    }
    float a[4];
    if (active) {
        const long long col = static_cast<long long>(g) * 128 + lane * 4;
        const long long rbase = static_cast<long long>(in_row) * p.W;
        float gv[4], uv[4];
        load_gate_up4<F32IN, KG>(p, rbase + col, rbase + p.N + col, gv, uv);
        if (slot_walk && route < 0) active = false;  // a pad slot
        if (active) {
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = silu_mul_bf16<ACT>(gv[i], uv[i], p.L);
        }
    }
    uint32_t codes;
    float sc;
    quant_group_codes4(a, active, p.fmt, &codes, &sc);
    if (active) {
        const long long o = static_cast<long long>(row) * p.N + static_cast<long long>(g) * 128 + lane * 4;
        *reinterpret_cast<uint32_t*>(p.out_q + o) = codes;
        if (lane == 0) p.out_s[static_cast<long long>(row) * p.G + g] = sc;
    }
}

// W4: one group per warp (quant_item4) instead of one per half-warp (quant_pair).
template <int ACT, bool F32IN, bool PERSISTENT, int KG, bool INL, bool W4 = false>
__global__ void __launch_bounds__(256) k_act_quant(AQArgs p) {
    extern __shared__ int aq_smap[];  // the expert map, when p.map_smem
    const int lane = threadIdx.x & 31;
    const long long warps_per_block = blockDim.x >> 5;
    if (p.n_blocks) {
        // slot rows of the blocks that exist (the route preparation ran two or more launches
        // back, so its count is read before the wait)
        const long long nb = max(0, __ldcg(p.n_blocks));
        p.rows = static_cast<int>(min(static_cast<long long>(p.rows), nb * p.bm));
    }
    if (p.n_rows) {
        // written by route preparation two or more launches back, so read before the wait
        p.rows = min(p.rows, max(0, __ldcg(p.n_rows)));
    }
    // a warp's work unit: a pair of groups, or one group with W4
    const long long items = static_cast<long long>(p.rows) * p.G;
    const long long pairs = W4 ? items : (items + 1) / 2;
    long long pair = static_cast<long long>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
    // a row's first selector: its expert id (a caller input) or its row-map entry
    const int32_t* sel = p.row_expert ? p.row_expert : p.row_map;
    auto sel_of = [&](long long pr) -> int {
        const long long item = W4 ? pr : pr * 2 + (lane >> 4);
        return (pr < pairs && item < items) ? __ldcg(sel + static_cast<unsigned>(item) / static_cast<unsigned>(p.G)) : -1;
    };
    // the first pair's selector before the wait, when it is an input or was written two or
    // more launches back; with an expert filter the (caller's) expert map is staged in shared
    // memory, so a row's filter costs one global load
    int pre = -2;
    if (sel && (p.row_expert || p.map_early) && pair < pairs) pre = sel_of(pair);
    const int* smap = nullptr;
    if (PERSISTENT && p.map_smem) {
        for (int i = threadIdx.x; i < p.E; i += blockDim.x) aq_smap[i] = __ldg(p.expert_map + i);
        __syncthreads();
        smap = aq_smap;
    }
    if (p.early_release) grid_dep_launch();
    grid_dep_wait();
    if (!p.early_release) grid_dep_launch();
    if (!PERSISTENT) {
        if (pair < pairs) quant_pair<ACT, F32IN, KG, INL>(p, pair, lane, pre);
        return;
    }
    const long long stride = static_cast<long long>(gridDim.x) * warps_per_block;
    // each pair's selector is loaded one pair ahead, so a pair whose row is dropped (most of
    // them at expert-parallel shapes) costs no round trip of its own
    const bool ahead = sel != nullptr;
    int cur = pre;
    if (ahead && cur == -2) cur = sel_of(pair);
    for (; pair < pairs; pair += stride) {
        const int nxt = ahead ? sel_of(pair + stride) : -2;
        if constexpr (W4)
            quant_item4<ACT, F32IN, KG>(p, pair, lane, ahead ? cur : -2, smap);
        else
            quant_pair<ACT, F32IN, KG, INL>(p, pair, lane, ahead ? cur : -2, smap);
        cur = nxt;
    }
}

// Input quantisation of the layer, once per token: every (token, 128-column group) is quantised
// and its codes and scale are stored to the expert-sorted slot of each kept route of the token
// (route_slot), giving exactly the rows the per-route gather of k_act_quant gives.  The token
// rows are the caller's input, so a warp loads and quantises its first kHold items before
// waiting for route preparation; only the stores wait for the routing.
// Pairs of 128-groups each warp of the input quantisation quantises before the routing wait.
constexpr int kInputHold = 2;

// PADS: the kernel also writes the -1 pads of sorted_idx that route preparation left out (a
// separate instantiation: the code alone, never taken, cost the small decode layers ~0.5 us).
template <bool PADS>
__global__ void __launch_bounds__(256) k_input_quant_tokens(const uint16_t* __restrict__ x, int M,
                                                            int H, int k, const int32_t* route_slot,
                                                            int slots, uint8_t* xq, float* xs,
                                                            int fmt, int* status,
                                                            const int32_t* pad_off,
                                                            const int32_t* pad_cnt,
                                                            int32_t* pad_sorted, int pad_E,
                                                            int late_release) {
    constexpr int kHold = kInputHold;
    const int lane = threadIdx.x & 31, half = lane >> 4, l = lane & 15;
    const int G = H / 128;
    const long long groups = static_cast<long long>(M) * G;
    const long long pairs = (groups + 1) / 2;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long w0 = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    auto quant = [&](long long pr, int& t, int& g, uint2& codes, float& sc) -> bool {
        const long long item = pr * 2 + half;
        const bool active = pr < pairs && item < groups;
        float a[8];
        t = 0; g = 0;
        if (active) {
            t = static_cast<int>(item / G);
            g = static_cast<int>(item - static_cast<long long>(t) * G);
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<long long>(t) * H + g * 128 + l * 8));
            a[0] = bf16_lo(v.x); a[1] = bf16_hi(v.x); a[2] = bf16_lo(v.y); a[3] = bf16_hi(v.y);
            a[4] = bf16_lo(v.z); a[5] = bf16_hi(v.z); a[6] = bf16_lo(v.w); a[7] = bf16_hi(v.w);
        }
        quant_group_codes_compact(a, active, fmt, &codes, &sc);
        return active;
    };
    auto scatter = [&](int t, int g, uint2 codes, float sc) {
        for (int j0 = 0; j0 < k; j0 += 8) {
            int ms[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                ms[jj] = j0 + jj < k ? __ldcg(route_slot + static_cast<long long>(t) * k + j0 + jj) : -1;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                int m = ms[jj];
                if (m >= slots) { if (status) atomicOr(status, MOE_DEV_BAD_INDEX); m = -1; }
                if (m < 0) continue;
                *reinterpret_cast<uint2*>(xq + static_cast<long long>(m) * H + g * 128 + l * 8) = codes;
                if (l == 0) xs[static_cast<long long>(m) * G + g] = sc;
            }
        }
    };
    // The next launch (the gate/up GEMM) is released at once, or with late_release only after
    // this kernel's routing wait: route preparation is then complete, and the GEMM reads its
    // tables as soon as it starts, waiting for this kernel only before its activation tiles.
    if (!late_release) grid_dep_launch();
    uint2 hc[kHold];
    float hs[kHold];
    int ht[kHold], hg[kHold];
    bool ha[kHold];
#pragma unroll
    for (int i = 0; i < kHold; ++i) ha[i] = quant(w0 + i * warps, ht[i], hg[i], hc[i], hs[i]);
    grid_dep_wait();
    if (late_release) grid_dep_launch();
#pragma unroll
    for (int i = 0; i < kHold; ++i)
        if (ha[i]) scatter(ht[i], hg[i], hc[i], hs[i]);
    if constexpr (PADS) {
        // the -1 pads of sorted_idx that route preparation left out: one warp per expert, the
        // slots after its count up to the next expert's start, then every slot past the blocks
        for (long long e = w0; e < pad_E; e += warps) {
            const int lo = __ldcg(pad_off + e) + __ldcg(pad_cnt + e), hi = __ldcg(pad_off + e + 1);
            for (int sl = lo + lane; sl < hi; sl += 32) pad_sorted[sl] = -1;
        }
        for (long long sl = __ldcg(pad_off + pad_E) + w0 * 32 + lane; sl < slots; sl += warps * 32)
            pad_sorted[sl] = -1;
    }
    for (long long pr = w0 + kHold * warps; pr < pairs; pr += warps) {
        int t, g;
        uint2 codes;
        float sc;
        if (quant(pr, t, g, codes, sc)) scatter(t, g, codes, sc);
    }
}

// The unfused first half: BF16 SiLU*mul written to memory, 8 outputs per thread.  Rows whose
// expert the filter drops (row_expert / expert_map, as in k_act_quant) are skipped.
template <int ACT>
__global__ void __launch_bounds__(256) k_silu_and_mul(const uint16_t* in, int rows, int N,
                                                      float L, const int32_t* row_expert,
                                                      const int32_t* expert_map, int E,
                                                      uint16_t* out) {
    grid_dep_wait();
    grid_dep_launch();
    const long long chunks = static_cast<long long>(rows) * (N / 8);
    for (long long c = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; c < chunks;
         c += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = c / (N / 8);
        const long long col = (c - row * (N / 8)) * 8;
        if (row_expert) {
            const int id = __ldg(row_expert + row);
            if (id < 0 || id >= E) continue;
            if (expert_map && __ldg(expert_map + id) < 0) continue;
        }
        uint4 gw = __ldg(reinterpret_cast<const uint4*>(in + row * 2 * N + col));
        uint4 uw = __ldg(reinterpret_cast<const uint4*>(in + row * 2 * N + N + col));
        const uint32_t gg[4] = {gw.x, gw.y, gw.z, gw.w};
        const uint32_t uu[4] = {uw.x, uw.y, uw.z, uw.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float a0 = silu_mul_bf16<ACT>(bf16_lo(gg[i]), bf16_lo(uu[i]), L);
            float a1 = silu_mul_bf16<ACT>(bf16_hi(gg[i]), bf16_hi(uu[i]), L);
            o[i] = (__float_as_uint(a0) >> 16) | (__float_as_uint(a1) & 0xFFFF0000u);
        }
        *reinterpret_cast<uint4*>(out + row * N + col) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// `units`: work units of the kernel, group pairs, or groups with W4 (persistent only).
template <int ACT, bool F32IN, int KG, bool INL, bool W4 = false>
int launch_aq_grid(const AQArgs& p, long long units, bool persistent, bool pdl, cudaStream_t stream) {
    // Few units (decode batches): one-warp CTAs, one unit each.  A grouped-GEMM CTA (11 warps of
    // ~144 registers, spread over the SM's four schedulers and their register files) leaves room
    // beside it for one more warp, not two, so a one-warp CTA becomes resident next to a running
    // GEMM CTA.  The act-quant is then in place before the gate/up GEMM ends, and no down-GEMM CTA
    // waits for an act-quant CTA to leave its SM.  Measured on GB300 against two-warp CTAs (which
    // started only as GEMM CTAs left): decode M=2 to 8 ~1.8 us faster, M=16 and 32 ~0.8 us.
    const int threads = persistent && units <= (W4 ? 4LL : 2LL) * sm_count() ? 32 : 256, wpb = threads / 32;
    long long blocks = (units + wpb - 1) / wpb;
    const size_t smem = persistent && p.map_smem ? static_cast<size_t>(p.E) * 4 : 0;
    if (persistent) {
        // as many CTAs as are resident at once, so the grid runs in one wave
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_act_quant<ACT, F32IN, true, KG, INL, W4>, threads,
                                                          smem) != cudaSuccess || occ < 1)
            occ = 1;
        long long cap = static_cast<long long>(sm_count()) * occ;
        if (blocks > cap) blocks = cap;
    }
    if (blocks > 0x7FFFFFFFLL) { set_error("act_quant: too many groups"); return MOE_ERR_ARG; }
    Launch L(dim3(static_cast<unsigned>(blocks)), dim3(threads), smem, stream, pdl);
    cudaError_t e;
    if constexpr (W4)
        e = cudaLaunchKernelEx(&L.cfg, k_act_quant<ACT, F32IN, true, KG, INL, true>, p);
    else
        e = persistent ? cudaLaunchKernelEx(&L.cfg, k_act_quant<ACT, F32IN, true, KG, INL>, p)
                       : cudaLaunchKernelEx(&L.cfg, k_act_quant<ACT, F32IN, false, KG, INL>, p);
    if (e != cudaSuccess) {
        set_error("act_quant launch: %s", cudaGetErrorString(e));
        return MOE_ERR_LAUNCH;
    }
    return MOE_OK;
}

// Up to kInlinePairs group pairs the SiLU*mul and quantiser run inline; above, out of line.
// Measured on GB300 (graph-replayed layers): inline 34.9 vs 36.3 us at decode M = 1 and 161.1
// vs 161.9 us at M = 32, within noise at M = 256, and 115.8 vs 116.6 us at the expert-parallel
// shape (T = 1024, N = 2048), where the kernel is issue-bound and the calls cost instructions.
constexpr long long kInlinePairs = 1LL << 40;

template <int ACT, bool F32IN, int KG>
int launch_aq_kg(const AQArgs& p, bool persistent, bool pdl, cudaStream_t stream) {
    const long long pairs = (static_cast<long long>(p.rows) * p.G + 1) / 2;
    if (pairs == 0) return MOE_OK;
    // the kernel divides group indices in 32 bits (a 64-bit division is a long software
    // sequence on the path from the dependency wait to a pair's loads)
    if (static_cast<long long>(p.rows) * p.G >= (1LL << 31)) {
        set_error("act_quant: rows * N / 128 must be below 2^31");
        return MOE_ERR_ARG;
    }
    if constexpr (ACT != MOE_ACT_IDENTITY && KG <= 4) {
        // Few groups (decode batches), of split partials or of the BF16 value of one split: one
        // group per warp (quant_item4).  Measured on GB300 against group pairs (split partials),
        // graph-replayed layer, interleaved A/B: decode
        // M=1 33.4 -> 32.7 us, M=16 113.2 -> 112.0, M=32 161.9 -> 160.8.  With 8 splits (M=2 to 8,
        // which took 6 to 8 before the layer capped the split count at 4) it measured no faster,
        // and with many groups (expert-parallel, prefill) 2-2.5 us slower.  On the BF16 value of
        // one split (decode M=4, 5 and 10): M=4 -0.3 us, M=5 -1.0, M=10 -0.9.  Up to 8 groups
        // per SM instead of 4: M=48 -0.7 us, M=64 -0.55; up to 16 instead of 8: M=96 -0.55,
        // M=128 -0.3.
        const long long items = static_cast<long long>(p.rows) * p.G;
        if (persistent && items <= 16LL * sm_count())
            return launch_aq_grid<ACT, F32IN, KG, true, true>(p, items, persistent, pdl, stream);
    }
    if constexpr (ACT != MOE_ACT_IDENTITY) {
        if (pairs <= kInlinePairs) return launch_aq_grid<ACT, F32IN, KG, true>(p, pairs, persistent, pdl, stream);
    }
    return launch_aq_grid<ACT, F32IN, KG, false>(p, pairs, persistent, pdl, stream);
}

template <int ACT, bool F32IN>
int launch_aq(const AQArgs& p, bool persistent, bool pdl, cudaStream_t stream) {
    if constexpr (!F32IN) {
        return launch_aq_kg<ACT, F32IN, 1>(p, persistent, pdl, stream);
    } else {
        if (p.in_splits <= 1) return launch_aq_kg<ACT, F32IN, 1>(p, persistent, pdl, stream);
        if (p.in_splits <= 4) return launch_aq_kg<ACT, F32IN, 4>(p, persistent, pdl, stream);
        return launch_aq_kg<ACT, F32IN, 8>(p, persistent, pdl, stream);
    }
}

}  // namespace

int launch_act_quant(moe_act act, const void* in, moe_dtype in_dtype, int in_splits, int in_rows,
                     int rows, int N, float clamp_limit, moe_scale_fmt fmt,
                     const int32_t* row_expert, const int32_t* expert_map, int E,
                     const int32_t* row_map, int row_div, int out_rows, uint8_t* out_q,
                     float* out_s, moe_quant_strategy strategy, bool pdl, cudaStream_t stream,
                     bool map_early, const int32_t* slot_route, const int32_t* n_blocks, int bm,
                     const int32_t* n_rows, bool early_release) {
    if (!in || !out_q || !out_s) { set_error("silu_mul_quant_fp8: null pointer"); return MOE_ERR_ARG; }
    if (!aligned16(in) || !aligned16(out_q) || (reinterpret_cast<uintptr_t>(out_s) & 3u)) {
        set_error("silu_mul_quant_fp8: in/out_q must be 16-byte aligned, out_s 4-byte aligned");
        return MOE_ERR_ARG;
    }
    if (rows < 0 || in_rows < 0 || out_rows < 0 || N <= 0 || N % 128) {
        set_error("silu_mul_quant_fp8: need rows, in_rows, out_rows >= 0 and N a positive multiple of 128 (N=%d)", N);
        return MOE_ERR_ARG;
    }
    if (act != MOE_ACT_IDENTITY && act != MOE_ACT_SILU_MUL && act != MOE_ACT_SILU_MUL_GATE_UPPER) {
        set_error("silu_mul_quant_fp8: unknown act %d", static_cast<int>(act));
        return MOE_ERR_ARG;
    }
    if (fmt != MOE_SCALE_F32 && fmt != MOE_SCALE_UE8M0) { set_error("silu_mul_quant_fp8: bad fmt"); return MOE_ERR_ARG; }
    if (in_dtype != MOE_DTYPE_BF16 && in_dtype != MOE_DTYPE_F32) { set_error("silu_mul_quant_fp8: bad in_dtype"); return MOE_ERR_ARG; }
    if (in_splits < 1 || (in_dtype == MOE_DTYPE_BF16 && in_splits != 1)) {
        set_error("silu_mul_quant_fp8: in_splits must be 1 for BF16 input and >= 1 for fp32");
        return MOE_ERR_ARG;
    }
    if (!row_map && (rows > in_rows || rows > out_rows)) {
        set_error("silu_mul_quant_fp8: rows exceeds in_rows or out_rows without a row map");
        return MOE_ERR_ARG;
    }
    if (row_map && row_div < 0) { set_error("silu_mul_quant_fp8: row_div < 0"); return MOE_ERR_ARG; }
    if (row_expert && E <= 0) { set_error("silu_mul_quant_fp8: row_expert needs E > 0"); return MOE_ERR_ARG; }
    if (expert_map && !row_expert) { set_error("silu_mul_quant_fp8: expert_map needs row_expert"); return MOE_ERR_ARG; }
    AQArgs p{};
    p.in = in;
    p.W = act == MOE_ACT_IDENTITY ? N : 2 * N;
    p.split_stride = static_cast<long long>(in_rows) * p.W;
    p.in_rows = in_rows;
    p.in_splits = in_splits;
    p.rows = rows;
    p.N = N;
    p.G = N / 128;
    p.L = clamp_limit;
    p.fmt = fmt;
    p.row_expert = row_expert;
    p.expert_map = expert_map;
    p.E = E;
    p.row_map = row_map;
    p.row_div = row_div;
    p.out_rows = out_rows;
    p.out_q = out_q;
    p.out_s = out_s;
    p.map_early = map_early ? 1 : 0;
    // an expert filter's map, staged in shared memory by persistent launches (up to 8192 ids)
    p.map_smem = (row_expert && expert_map && E <= 8192) ? 1 : 0;
    if (n_blocks && (!slot_route || bm <= 0 || row_map)) {
        set_error("silu_mul_quant_fp8: slot rows need slot_route, bm > 0 and no row map");
        return MOE_ERR_ARG;
    }
    p.slot_route = slot_route;
    p.n_blocks = n_blocks;
    p.bm = bm;
    p.n_rows = n_rows;
    p.early_release = early_release ? 1 : 0;
    p.status = device_status_ptr();
    bool persistent;
    if (strategy == MOE_QUANT_PER_GROUP) persistent = false;
    else if (strategy == MOE_QUANT_PERSISTENT) persistent = true;
    else persistent = row_expert || row_map || static_cast<long long>(rows) * N >= (1LL << 20);
    const bool f32 = in_dtype == MOE_DTYPE_F32;
    switch (act) {
        case MOE_ACT_IDENTITY:
            return f32 ? launch_aq<MOE_ACT_IDENTITY, true>(p, persistent, pdl, stream)
                       : launch_aq<MOE_ACT_IDENTITY, false>(p, persistent, pdl, stream);
        case MOE_ACT_SILU_MUL:
            return f32 ? launch_aq<MOE_ACT_SILU_MUL, true>(p, persistent, pdl, stream)
                       : launch_aq<MOE_ACT_SILU_MUL, false>(p, persistent, pdl, stream);
        default:
            return f32 ? launch_aq<MOE_ACT_SILU_MUL_GATE_UPPER, true>(p, persistent, pdl, stream)
                       : launch_aq<MOE_ACT_SILU_MUL_GATE_UPPER, false>(p, persistent, pdl, stream);
    }
}

int launch_input_quant_tokens(const void* x, int M, int H, int k, const int32_t* route_slot,
                              int slots, uint8_t* xq, float* xs, moe_scale_fmt fmt, bool pdl,
                              cudaStream_t stream, const int32_t* pad_offset,
                              const int32_t* pad_count, int32_t* pad_sorted, int pad_E,
                              bool late_release) {
    const long long pairs = (static_cast<long long>(M) * (H / 128) + 1) / 2;
    if (pairs == 0) return MOE_OK;
    // One pair per warp, at most two CTAs per SM, so the next kernel's CTAs fit beside them.
    // When that grid cannot hold every pair before the routing wait (two per warp), up to four
    // CTAs per SM instead: the pairs left for after the wait were on the critical path
    // (expert-parallel T=1024 117.0 -> 114.2 us, prefill 741.6 -> 739.4, decode M=256 255.9 ->
    // 254.4; interleaved A/B).
    const long long sms = sm_count();
    long long blocks = std::min<long long>((pairs + 7) / 8, sms * 2);
    if (blocks * 8 * kInputHold < pairs) blocks = std::min<long long>((pairs + 15) / 16, sms * 4);
    Launch L(dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl);
    cudaError_t e = pad_sorted
        ? cudaLaunchKernelEx(&L.cfg, k_input_quant_tokens<true>, static_cast<const uint16_t*>(x), M, H, k,
                             route_slot, slots, xq, xs, static_cast<int>(fmt), device_status_ptr(),
                             pad_offset, pad_count, pad_sorted, pad_E, late_release ? 1 : 0)
        : cudaLaunchKernelEx(&L.cfg, k_input_quant_tokens<false>, static_cast<const uint16_t*>(x), M, H, k,
                             route_slot, slots, xq, xs, static_cast<int>(fmt), device_status_ptr(),
                             pad_offset, pad_count, pad_sorted, pad_E, late_release ? 1 : 0);
    if (e != cudaSuccess) { set_error("input quant launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}

}  // namespace moe

extern "C" int silu_and_mul_bf16(moe_act act, const void* in, int rows, int N, float clamp_limit,
                                 const int32_t* row_expert, const int32_t* expert_map, int E,
                                 void* out, cudaStream_t stream) {
    using namespace moe;
    clear_error();
    if (!device_is_sm103()) { set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    if (!in || !out || !aligned16(in) || !aligned16(out)) { set_error("silu_and_mul_bf16: null or misaligned pointer"); return MOE_ERR_ARG; }
    if (rows < 0 || N <= 0 || N % 8) { set_error("silu_and_mul_bf16: bad shape"); return MOE_ERR_ARG; }
    if (row_expert && E <= 0) { set_error("silu_and_mul_bf16: row_expert needs E > 0"); return MOE_ERR_ARG; }
    if (expert_map && !row_expert) { set_error("silu_and_mul_bf16: expert_map needs row_expert"); return MOE_ERR_ARG; }
    if (act != MOE_ACT_SILU_MUL && act != MOE_ACT_SILU_MUL_GATE_UPPER) { set_error("silu_and_mul_bf16: act must be a SiLU*mul"); return MOE_ERR_ARG; }
    const long long chunks = static_cast<long long>(rows) * (N / 8);
    if (chunks == 0) return MOE_OK;
    long long blocks = (chunks + 255) / 256;
    long long cap = static_cast<long long>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    Launch L(dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, false);
    cudaError_t e = act == MOE_ACT_SILU_MUL
        ? cudaLaunchKernelEx(&L.cfg, k_silu_and_mul<MOE_ACT_SILU_MUL>, static_cast<const uint16_t*>(in), rows, N,
                             clamp_limit, row_expert, expert_map, E, static_cast<uint16_t*>(out))
        : cudaLaunchKernelEx(&L.cfg, k_silu_and_mul<MOE_ACT_SILU_MUL_GATE_UPPER>, static_cast<const uint16_t*>(in), rows, N,
                             clamp_limit, row_expert, expert_map, E, static_cast<uint16_t*>(out));
    if (e != cudaSuccess) { set_error("silu_and_mul_bf16 launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}

extern "C" int silu_mul_quant_fp8(moe_act act, const void* in, moe_dtype in_dtype, int in_splits,
                                  int in_rows, int rows, int N, float clamp_limit,
                                  moe_scale_fmt fmt, const int32_t* row_expert,
                                  const int32_t* expert_map, int E, const int32_t* row_map,
                                  int row_div, int out_rows, uint8_t* out_q, float* out_s,
                                  moe_quant_strategy strategy, cudaStream_t stream) {
    moe::clear_error();
    if (!moe::device_is_sm103()) { moe::set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    return moe::launch_act_quant(act, in, in_dtype, in_splits, in_rows, rows, N, clamp_limit, fmt,
                                 row_expert, expert_map, E, row_map, row_div, out_rows, out_q,
                                 out_s, strategy, false, stream);
}
