// moe_reduce.cu -- weighted top-k sum of the per-route expert outputs back to one BF16 row per
// token.
//
// Method: lmdeploy PR #4228 "Moe Reduce kernel" (Copilot overview): the routing weights are no
// longer applied inside the MoE GEMM; a dedicated reduction multiplies each route's output by
// its weight and sums the top-k routes of a token.  Accumulation is fp32 (the page's review
// thread on fp32_acc); the terms are added in top-k order with one fused multiply-add each, so
// the result does not depend on the launch shape.
//
// One warp produces 256 consecutive outputs of one token, 8 per lane.  Lane j < k holds route
// j's id, weight and keep flag, so the kept routes form a warp-uniform bit mask that the warp
// walks in top-k order: no shared memory, no barrier, no per-route predicate.  For each group
// of up to eight kept routes a lane issues its 16-byte loads of 8 BF16 values together, then the
// fused multiply-adds run in route order.  HBM traffic is the kept routes' rows once plus the
// output once.  A grid of one wave walks the (token, 256-column chunk) items; the first item's
// ids, weights and expert-map entries are caller inputs, read before the wait for the previous
// kernel.  top-k is at most 32 (one route per lane).
#include "common.cuh"

#include <algorithm>

namespace moe {
namespace {

constexpr int kMaxTopk = kReduceMaxTopk;
constexpr int kThreads = 256;
constexpr int kGroup = 8;  // kept routes whose loads are in flight together (top-8 in one round)
static_assert(kMaxTopk <= 32, "one route per lane");

// The kept routes of token t as a bit mask (bit j: route j is kept); *wl = this lane's weight.
__device__ __forceinline__ unsigned token_routes(const int32_t* __restrict__ ids,
                                                 const float* __restrict__ w,
                                                 const int32_t* __restrict__ map, int t, int k,
                                                 int E, int E_local, int lane, float* wl) {
    bool keep = false;
    *wl = 0.0f;
    if (lane < k) {
        const long long r = static_cast<long long>(t) * k + lane;
        const int id = __ldg(ids + r);
        *wl = __ldg(w + r);
        keep = id >= 0 && id < E;
        if (keep && map) {
            // the route-preparation rule: a map entry outside [0, E_local) gives the route no
            // slot, so its z row was never written and it adds nothing here either
            const int le = __ldg(map + id);
            keep = le >= 0 && le < E_local;
        }
    }
    return __ballot_sync(0xFFFFFFFFu, keep);
}

__global__ void __launch_bounds__(kThreads) k_moe_reduce(const uint16_t* __restrict__ z,
                                                         const float* __restrict__ w,
                                                         const int32_t* __restrict__ ids,
                                                         const int32_t* __restrict__ map, int M,
                                                         int k, int E, int E_local, int H,
                                                         uint16_t* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int chunks = (H + 255) / 256;
    const long long items = static_cast<long long>(M) * chunks;
    const int wpb = blockDim.x >> 5;
    const long long stride = static_cast<long long>(gridDim.x) * wpb;
    long long it = static_cast<long long>(blockIdx.x) * wpb + (threadIdx.x >> 5);
    grid_dep_launch();
    float wl = 0.0f;
    unsigned keep = 0;
    int t = -1;
    if (it < items) {
        t = static_cast<int>(static_cast<unsigned>(it) / static_cast<unsigned>(chunks));
        keep = token_routes(ids, w, map, t, k, E, E_local, lane, &wl);
    }
    grid_dep_wait();  // the expert outputs z are the previous kernel's
    for (; it < items; it += stride) {
        const int tt = static_cast<int>(static_cast<unsigned>(it) / static_cast<unsigned>(chunks));
        if (tt != t) {
            t = tt;
            keep = token_routes(ids, w, map, t, k, E, E_local, lane, &wl);
        }
        const int col = static_cast<int>(it - static_cast<long long>(t) * chunks) * 256 + lane * 8;
        const bool act = col < H;
        const uint16_t* zt = z + static_cast<long long>(t) * k * H + col;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        unsigned rest = keep;
        while (rest) {
            int jg[kGroup];
            uint4 vg[kGroup];
            int n = 0;
#pragma unroll
            for (int q = 0; q < kGroup; ++q) {
                jg[q] = rest ? __ffs(rest) - 1 : 0;
                if (rest) { rest &= rest - 1; ++n; }
            }
#pragma unroll
            for (int q = 0; q < kGroup; ++q)
                if (q < n && act)
                    vg[q] = __ldcg(reinterpret_cast<const uint4*>(zt + static_cast<long long>(jg[q]) * H));
#pragma unroll
            for (int q = 0; q < kGroup; ++q) {
                if (q < n) {
                    const float wj = __shfl_sync(0xFFFFFFFFu, wl, jg[q]);
                    if (act) {
                        const uint4 v = vg[q];
                        acc[0] = __fmaf_rn(wj, bf16_lo(v.x), acc[0]);
                        acc[1] = __fmaf_rn(wj, bf16_hi(v.x), acc[1]);
                        acc[2] = __fmaf_rn(wj, bf16_lo(v.y), acc[2]);
                        acc[3] = __fmaf_rn(wj, bf16_hi(v.y), acc[3]);
                        acc[4] = __fmaf_rn(wj, bf16_lo(v.z), acc[4]);
                        acc[5] = __fmaf_rn(wj, bf16_hi(v.z), acc[5]);
                        acc[6] = __fmaf_rn(wj, bf16_lo(v.w), acc[6]);
                        acc[7] = __fmaf_rn(wj, bf16_hi(v.w), acc[7]);
                    }
                }
            }
        }
        if (act) {
            uint4 o;
            o.x = f32_to_bf16_bits(acc[0]) | (f32_to_bf16_bits(acc[1]) << 16);
            o.y = f32_to_bf16_bits(acc[2]) | (f32_to_bf16_bits(acc[3]) << 16);
            o.z = f32_to_bf16_bits(acc[4]) | (f32_to_bf16_bits(acc[5]) << 16);
            o.w = f32_to_bf16_bits(acc[6]) | (f32_to_bf16_bits(acc[7]) << 16);
            *reinterpret_cast<uint4*>(out + static_cast<long long>(t) * H + col) = o;
        }
    }
}

}  // namespace

int launch_moe_reduce(const void* z, const float* topk_w, const int32_t* topk_ids,
                      const int32_t* expert_map, int M, int k, int E, int E_local, int H, void* out,
                      bool pdl, cudaStream_t stream) {
    if (M < 0 || k <= 0 || E <= 0 || E_local <= 0 || H <= 0 || H % 8) {
        set_error("moe_reduce: bad shape (need k, E, E_local > 0 and H a multiple of 8)");
        return MOE_ERR_ARG;
    }
    if (!expert_map && E_local != E) {
        set_error("moe_reduce: without an expert map E_local must equal E (%d vs %d)", E_local, E);
        return MOE_ERR_EXPERT_SLICE;
    }
    if (k > kMaxTopk) { set_error("moe_reduce: top-k above %d is not supported", kMaxTopk); return MOE_ERR_ARG; }
    const long long items = static_cast<long long>(M) * ((H + 255) / 256);
    if (items == 0) return MOE_OK;
    // item indices are divided in 32 bits in the kernel
    if (items >= (1LL << 31)) { set_error("moe_reduce: M * H / 256 must be below 2^31"); return MOE_ERR_ARG; }
    if (!z || !topk_w || !topk_ids || !out) { set_error("moe_reduce: null pointer"); return MOE_ERR_ARG; }
    if (!aligned16(z) || !aligned16(out)) { set_error("moe_reduce: z and out must be 16-byte aligned"); return MOE_ERR_ARG; }
    // Few items (decode batches of a few tokens): one item per warp in CTAs of two warps, one
    // CTA per SM -- small enough in registers to become resident beside a grouped-GEMM CTA, so
    // the CTAs launched early by programmatic dependent launch wait on the SMs while the down
    // GEMM finishes.  Otherwise one wave of full CTAs, as many as are resident at once.
    const int sms = sm_count();
    int threads = kThreads;
    long long blocks;
    if (items <= 2LL * sms) {
        threads = 64;
        blocks = (items + 1) / 2;
    } else {
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_moe_reduce, kThreads, 0) != cudaSuccess || occ < 1)
            occ = 1;
        const long long need = (items + kThreads / 32 - 1) / (kThreads / 32);
        blocks = std::min<long long>(need, static_cast<long long>(sms) * occ);
    }
    Launch L(dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, pdl);
    cudaError_t e = cudaLaunchKernelEx(&L.cfg, k_moe_reduce, static_cast<const uint16_t*>(z),
                                       topk_w, topk_ids, expert_map, M, k, E, E_local, H,
                                       static_cast<uint16_t*>(out));
    if (e != cudaSuccess) { set_error("moe_reduce launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}

}  // namespace moe

extern "C" int moe_reduce(const void* z, const float* topk_w, const int32_t* topk_ids,
                          const int32_t* expert_map, int M, int k, int E, int E_local, int H,
                          void* out, cudaStream_t stream) {
    moe::clear_error();
    if (!moe::device_is_sm103()) { moe::set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    return moe::launch_moe_reduce(z, topk_w, topk_ids, expert_map, M, k, E, E_local, H, out, false,
                                  stream);
}

extern "C" int moe_kernel_binary_version(void) {
    cudaFuncAttributes a{};
    if (cudaFuncGetAttributes(&a, reinterpret_cast<const void*>(moe::k_moe_reduce)) != cudaSuccess) {
        cudaGetLastError();  // no device: clear the error, answer -1
        return -1;
    }
    return a.binaryVersion;
}
