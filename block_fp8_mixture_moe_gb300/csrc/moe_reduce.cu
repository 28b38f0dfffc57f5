// moe_reduce.cu -- weighted top-k sum of the per-route expert outputs back to one BF16 row per
// token.
//
// Method: lmdeploy PR #4228 "Moe Reduce kernel" (Copilot overview): the routing weights are no
// longer applied inside the MoE GEMM; a dedicated reduction multiplies each route's output by
// its weight and sums the top-k routes of a token.  Accumulation is fp32 (the page's review
// thread on fp32_acc); the terms are added in top-k order with one fused multiply-add each, so
// the result does not depend on the launch shape.
//
// One thread produces 8 consecutive outputs of one token: per kept route one 16-byte load of 8
// BF16 values (a warp reads 512 contiguous bytes), 8 FMAs, and one 16-byte store at the end.
// HBM traffic is the kept routes' rows once plus the output once.
#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) k_moe_reduce(const uint16_t* __restrict__ z,
                                                    const float* __restrict__ w,
                                                    const int32_t* __restrict__ ids,
                                                    const int32_t* __restrict__ map, int M, int k,
                                                    int E, int H, uint16_t* __restrict__ out) {
    grid_dep_wait();
    grid_dep_launch();
    const int cpt = H / 8;  // 8-wide chunks per token
    const long long total = static_cast<long long>(M) * cpt;
    for (long long c = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; c < total;
         c += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(c / cpt);
        const int col = static_cast<int>(c - static_cast<long long>(t) * cpt) * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const int id = __ldg(ids + static_cast<long long>(t) * k + j);
            if (id < 0 || id >= E) continue;
            if (map && __ldg(map + id) < 0) continue;
            const float wj = __ldg(w + static_cast<long long>(t) * k + j);
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                z + (static_cast<long long>(t) * k + j) * H + col));
            acc[0] = __fmaf_rn(wj, bf16_lo(v.x), acc[0]);
            acc[1] = __fmaf_rn(wj, bf16_hi(v.x), acc[1]);
            acc[2] = __fmaf_rn(wj, bf16_lo(v.y), acc[2]);
            acc[3] = __fmaf_rn(wj, bf16_hi(v.y), acc[3]);
            acc[4] = __fmaf_rn(wj, bf16_lo(v.z), acc[4]);
            acc[5] = __fmaf_rn(wj, bf16_hi(v.z), acc[5]);
            acc[6] = __fmaf_rn(wj, bf16_lo(v.w), acc[6]);
            acc[7] = __fmaf_rn(wj, bf16_hi(v.w), acc[7]);
        }
        uint4 o;
        o.x = f32_to_bf16_bits(acc[0]) | (f32_to_bf16_bits(acc[1]) << 16);
        o.y = f32_to_bf16_bits(acc[2]) | (f32_to_bf16_bits(acc[3]) << 16);
        o.z = f32_to_bf16_bits(acc[4]) | (f32_to_bf16_bits(acc[5]) << 16);
        o.w = f32_to_bf16_bits(acc[6]) | (f32_to_bf16_bits(acc[7]) << 16);
        *reinterpret_cast<uint4*>(out + static_cast<long long>(t) * H + col) = o;
    }
}

}  // namespace

int launch_moe_reduce(const void* z, const float* topk_w, const int32_t* topk_ids,
                      const int32_t* expert_map, int M, int k, int E, int H, void* out, bool pdl,
                      cudaStream_t stream) {
    if (M < 0 || k <= 0 || E <= 0 || H <= 0 || H % 8) { set_error("moe_reduce: bad shape (H multiple of 8)"); return MOE_ERR_ARG; }
    const long long total = static_cast<long long>(M) * (H / 8);
    if (total == 0) return MOE_OK;
    if (!z || !topk_w || !topk_ids || !out) { set_error("moe_reduce: null pointer"); return MOE_ERR_ARG; }
    if (!aligned16(z) || !aligned16(out)) { set_error("moe_reduce: z and out must be 16-byte aligned"); return MOE_ERR_ARG; }
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    Launch L(dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl);
    cudaError_t e = cudaLaunchKernelEx(&L.cfg, k_moe_reduce, static_cast<const uint16_t*>(z),
                                       topk_w, topk_ids, expert_map, M, k, E, H,
                                       static_cast<uint16_t*>(out));
    if (e != cudaSuccess) { set_error("moe_reduce launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}

}  // namespace moe

extern "C" int moe_reduce(const void* z, const float* topk_w, const int32_t* topk_ids,
                          const int32_t* expert_map, int M, int k, int E, int H, void* out,
                          cudaStream_t stream) {
    moe::clear_error();
    if (!moe::device_is_sm103()) { moe::set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    return moe::launch_moe_reduce(z, topk_w, topk_ids, expert_map, M, k, E, H, out, false, stream);
}
