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
// HBM traffic is the kept routes' rows once plus the output once.  top-k is at most 16.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kMaxTopk = kReduceMaxTopk;

// One CTA per (token, 1024-column slice): the token's top-k ids, weights and keep flags are
// read once into shared memory; each thread then issues all its route loads back to back
// before the fused multiply-adds, so the loads overlap instead of running one after another.
__global__ void __launch_bounds__(128) k_moe_reduce(const uint16_t* __restrict__ z,
                                                    const float* __restrict__ w,
                                                    const int32_t* __restrict__ ids,
                                                    const int32_t* __restrict__ map, int M, int k,
                                                    int E, int E_local, int H,
                                                    uint16_t* __restrict__ out) {
    __shared__ float s_w[kMaxTopk];
    __shared__ int s_keep[kMaxTopk];
    grid_dep_launch();
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        const int j = threadIdx.x;
        const int id = __ldg(ids + static_cast<long long>(t) * k + j);
        bool keep = id >= 0 && id < E;
        if (keep && map) {
            // the route-preparation rule: a map entry outside [0, E_local) gives the route no
            // slot, so its z row was never written and it adds nothing here either
            const int le = __ldg(map + id);
            keep = le >= 0 && le < E_local;
        }
        s_keep[j] = keep ? 1 : 0;
        s_w[j] = __ldg(w + static_cast<long long>(t) * k + j);
    }
    // ids, weights and the expert map are the caller's inputs, not the previous kernel's
    // outputs: they are read above; the expert outputs z are read after the wait
    grid_dep_wait();
    __syncthreads();
    const int col = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
    if (col >= H) return;
    uint4 v[kMaxTopk];
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j)
        if (j < k && s_keep[j])
            v[j] = __ldcg(reinterpret_cast<const uint4*>(z + (static_cast<long long>(t) * k + j) * H + col));
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) {
        if (j < k && s_keep[j]) {
            const float wj = s_w[j];
            acc[0] = __fmaf_rn(wj, bf16_lo(v[j].x), acc[0]);
            acc[1] = __fmaf_rn(wj, bf16_hi(v[j].x), acc[1]);
            acc[2] = __fmaf_rn(wj, bf16_lo(v[j].y), acc[2]);
            acc[3] = __fmaf_rn(wj, bf16_hi(v[j].y), acc[3]);
            acc[4] = __fmaf_rn(wj, bf16_lo(v[j].z), acc[4]);
            acc[5] = __fmaf_rn(wj, bf16_hi(v[j].z), acc[5]);
            acc[6] = __fmaf_rn(wj, bf16_lo(v[j].w), acc[6]);
            acc[7] = __fmaf_rn(wj, bf16_hi(v[j].w), acc[7]);
        }
    }
    uint4 o;
    o.x = f32_to_bf16_bits(acc[0]) | (f32_to_bf16_bits(acc[1]) << 16);
    o.y = f32_to_bf16_bits(acc[2]) | (f32_to_bf16_bits(acc[3]) << 16);
    o.z = f32_to_bf16_bits(acc[4]) | (f32_to_bf16_bits(acc[5]) << 16);
    o.w = f32_to_bf16_bits(acc[6]) | (f32_to_bf16_bits(acc[7]) << 16);
    *reinterpret_cast<uint4*>(out + static_cast<long long>(t) * H + col) = o;
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
    const long long total = static_cast<long long>(M) * (H / 8);
    if (total == 0) return MOE_OK;
    if (!z || !topk_w || !topk_ids || !out) { set_error("moe_reduce: null pointer"); return MOE_ERR_ARG; }
    if (!aligned16(z) || !aligned16(out)) { set_error("moe_reduce: z and out must be 16-byte aligned"); return MOE_ERR_ARG; }
    if (k > kMaxTopk) { set_error("moe_reduce: top-k above %d is not supported", kMaxTopk); return MOE_ERR_ARG; }
    const int slices = (H / 8 + 127) / 128;
    Launch L(dim3(static_cast<unsigned>(M), static_cast<unsigned>(slices)), dim3(128), 0, stream, pdl);
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
