// api.cu -- host side of libmoefp8: error text, the per-device status word, device checks, and
// the whole-layer entry point that chains the stages on one stream.
//
// Layer order (lmdeploy PR #4956 "Perf/pytorch block fp8 moe decode", section "Fused SwiGLU
// and FP8 quantization": gate/up GEMM -> fused SiLU-and-mul + quant -> down GEMM; lmdeploy PR
// #4228 "Moe Reduce kernel": weighted top-k sum).  The fused path launches route preparation
// and then one persistent kernel for steps 2-6 (fused_layer.cu); the staged path launches them
// one by one:
//   1. moe_route_prepare            topk_ids -> expert-sorted slots, compact blocks, route_slot
//   2. input quantisation           x rows quantised once per token, stored to the route slots
//   3. grouped GEMM (GATE_UP)       fp32 split-K partials per slot
//   4. silu_mul_quant_fp8(SILU_MUL) partials summed, BF16 materialised in registers, E4M3
//   5. grouped GEMM (DOWN)          BF16 rows scattered back to route order
//   6. moe_reduce                   weighted sum per token
// Steps 2-6 are launched with programmatic dependent launch so each kernel's prologue overlaps
// the previous kernel's tail; every kernel waits for its predecessor before reading its output.
#include "common.cuh"

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

namespace moe {

namespace {
thread_local char g_err[512] = {0};
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
int g_is_sm103[kMaxDevices] = {0};  // 0 unknown, 1 yes, 2 no
int* g_status_ptr[kMaxDevices] = {nullptr};
std::mutex g_dev_mutex;

__device__ int g_status_word;  // one per device that loads the library

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

void init_device(int d) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_is_sm103[d]) return;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, d) != cudaSuccess) { g_is_sm103[d] = 2; return; }
    g_sm_count[d] = prop.multiProcessorCount;
    g_is_sm103[d] = (prop.major == 10 && prop.minor == 3) ? 1 : 2;
    void* p = nullptr;
    if (g_is_sm103[d] == 1 && cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess)
        g_status_ptr[d] = static_cast<int*>(p);
}
}  // namespace

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}
void clear_error() { g_err[0] = 0; }

bool device_is_sm103() {
    int d = current_device();
    if (d < 0 || d >= kMaxDevices) return false;
    if (!g_is_sm103[d]) init_device(d);
    return g_is_sm103[d] == 1;
}

int sm_count() {
    int d = current_device();
    if (d < 0 || d >= kMaxDevices) return 1;
    if (!g_is_sm103[d]) init_device(d);
    return g_sm_count[d] > 0 ? g_sm_count[d] : 1;
}

int* device_status_ptr() {
    int d = current_device();
    if (d < 0 || d >= kMaxDevices) return nullptr;
    if (!g_is_sm103[d]) init_device(d);
    return g_status_ptr[d];
}

bool ensure_smem(const void* func, int bytes) {
    // cudaFuncSetAttribute once per (device, kernel, size), outside any stream capture
    struct Entry { int dev; const void* f; int bytes; };
    static Entry table[256];
    static int n = 0;
    int d = current_device();
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    for (int i = 0; i < n; ++i)
        if (table[i].dev == d && table[i].f == func && table[i].bytes >= bytes) return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    for (int i = 0; i < n; ++i)
        if (table[i].dev == d && table[i].f == func) { table[i].bytes = bytes; return true; }
    if (n < 256) table[n++] = Entry{d, func, bytes};
    return true;
}

// ---------------------------------------------------------------------------------------------
// layer plan: block_m, split count and workspace layout
// ---------------------------------------------------------------------------------------------
namespace {

int forward_block_m(int M, int k, int E_local, int H, int N) {
    (void)k; (void)E_local; (void)H; (void)N;
    // Measured on GB300 with the graph-replayed layer: 16-token blocks are fastest up to
    // M = 256 (each active expert's weights are streamed once per block, and fewer pad rows mean
    // less promotion work); above, 32-token blocks beat 64 at both the expert-parallel shape
    // (M=1024, 6 of 256 experts per token, 32 local) and the Zipf prefill (M=512, E=512).
    if (M <= 256) return 16;
    return 32;
}

// Expected number of blocks under uniform routing, used only to size the split-K of the
// gate/up GEMM (any value is correct; the grid reads num_blocks on the device).
double expected_blocks(int M, int k, int E, int E_local, int bm) {
    const double p_pick = std::min(1.0, static_cast<double>(k) / std::max(1, E));
    const double active = E_local * (1.0 - std::pow(1.0 - p_pick, M));
    const double kept = static_cast<double>(M) * k * E_local / std::max(1, E);
    return std::max(1.0, std::max(active, kept / bm));
}

// Split-K of the gate/up GEMM: the smallest split whose round-robin schedule is within a few
// percent of the best achievable balance over the SMs.  At most 4 splits: the activation kernel
// then takes its one-group-per-warp form and releases the down GEMM early, and with one split
// the GEMM stores BF16.  Measured on GB300 against at most 8 (graph-replayed layer, interleaved
// A/B, three rounds): decode M=2 (7 -> 2 splits) -0.3 us, M=4 (6 -> 1) -1.15, M=8 (7 -> 3)
// -2.35.  Above 8 splits nothing measured faster at any decode size.
int gate_up_splits(int M, int k, int E, int E_local, int H, int N, int bm, int sms) {
    const int KB = H / 128;
    const double units1 = expected_blocks(M, k, E, E_local, bm) * (2 * N / 128);
    int best = 1;
    double best_cost = 1e300;
    const int smax = std::min(KB, 4);
    for (int s = 1; s <= smax; ++s) {
        const double units = units1 * s;
        const double waves = std::ceil(units / sms);
        const double per_unit = std::ceil(static_cast<double>(KB) / s) + 0.5;  // + unit overhead
        const double cost = waves * per_unit;
        if (cost < best_cost * 0.97) { best_cost = cost; best = s; }
    }
    return best;
}

// The grouped GEMMs' dynamic-tail counters: one 64-bit counter per projection in one
// 256-byte region.
constexpr size_t kSchedBytes = 256;

// A GEMM takes the dynamic tail when its expected weight stream is at least this many bytes per
// SM.  Measured on GB300 (graph-replayed layer, interleaved A/B): the Zipf prefill shape (about
// 21 and 10 MB per SM for gate/up and down, block_m 32) went from 780 to 741 us.  Before the
// tail's chunks were taken late (kDynLookahead in the GEMM), every decode and expert-parallel
// GEMM lost with it; the self-routed gate/up GEMM would also have to wait for its predecessor
// before the tail (decode M=1: 33.4 -> 41.4 us with it).
constexpr double kDynTailMinBytesPerSm = 8.0 * 1024 * 1024;
// With late chunks, block_m 16 (the decode GEMMs' 16-token blocks) from 2.5 MiB per SM: both
// GEMMs at decode M=64 -3.4 us, M=128 -8.6, M=256 -7.2; the gate/up GEMM of M=32 (3.8 MiB)
// unchanged, of M=16 (2.35 MiB) +4 us with it, so it stays below the threshold.
constexpr double kDynTailMinBytesPerSmBm16 = 2.5 * 1024 * 1024;

// Whether a GEMM of N_out x K weights per expert takes the dynamic tail (see
// kDynTailMinBytesPerSm): its expected active-expert weight bytes per SM.
bool dyn_tail(int M, int k, int E, int E_local, int N_out, int K, int bm, int sms) {
    if (bm > 32) return false;  // built for the plan's block sizes, 16 and 32
    const double bytes = expected_blocks(M, k, E, E_local, bm) * (N_out / 128) * (K / 128) * 128.0 * 128.0;
    const double min_bytes = bm <= 16 ? kDynTailMinBytesPerSmBm16 : kDynTailMinBytesPerSm;
    return bytes / std::max(1, sms) >= min_bytes;
}

// One workspace layout serves both forward paths: the token-scale and partial-sum regions are
// sized for the larger of the two uses (the fused kernel stores its token scales K-block major
// and its gate/up partial sums per stream-K piece).  The counters: the fused kernel's, the
// GEMMs' dynamic-tail counters and the epilogue-reduce counters.
struct Plan {
    int bm, B_cap, slots, R, splits;
    size_t off_sorted, off_bexp, off_nb, off_cnt, off_off, off_rslot, off_rws, off_xq, off_xs,
        off_gu, off_aq, off_as, off_z, off_sync, off_sched, off_rcnt, off_kslot, off_nkept, total;
};

Plan make_plan(int M, int k, int E, int E_local, int H, int N, int block_m, int sms) {
    Plan P{};
    P.bm = block_m > 0 ? block_m : forward_block_m(M, k, E_local, H, N);
    P.R = M * k;
    P.B_cap = (P.R + P.bm - 1) / P.bm + std::min(E_local, P.R);
    P.slots = P.B_cap * P.bm;
    P.splits = gate_up_splits(M, k, E, E_local, H, N, P.bm, sms);
    // With the dynamic tail on the gate/up GEMM at block_m 16, one split leaves units of a whole
    // K range (896 KB at H=7168, ~19 us of one SM's stream), too coarse for the tail to even out
    // the SMs' end times; two halve them.  Above ~1024 routes the extra fp32 partials cost more.
    // Measured on GB300 (interleaved A/B, three rounds): decode M=64 -2.1 us, M=96 and 128 -0.1
    // to -0.4; M=256 +1.0 with two splits; three or four splits slower at every decode size.
    if (P.splits == 1 && P.bm <= 16 && P.R <= 1024 && H >= 256 &&
        dyn_tail(M, k, E, E_local, 2 * N, H, P.bm, sms))
        P.splits = 2;
    size_t o = 0;
    auto take = [&o](size_t bytes) { size_t at = o; o += align256(bytes); return at; };
    P.off_sorted = take(sizeof(int32_t) * P.slots);
    P.off_bexp = take(sizeof(int32_t) * P.B_cap);
    P.off_nb = take(sizeof(int32_t));
    P.off_cnt = take(sizeof(int32_t) * E_local);
    P.off_off = take(sizeof(int32_t) * (E_local + 1));
    P.off_rslot = take(sizeof(int32_t) * P.R);
    P.off_rws = take(route_workspace_bytes(P.R, E_local, P.bm));
    P.off_xq = take(static_cast<size_t>(P.slots) * H);
    P.off_xs = take(sizeof(float) * static_cast<size_t>(P.slots) * (H / 128));
    P.off_gu = take(std::max(sizeof(float) * static_cast<size_t>(P.splits) * P.slots * 2 * N,
                             fused_partial_bytes(P.B_cap, P.bm, H, N, sms)));
    P.off_aq = take(static_cast<size_t>(P.slots) * N);
    P.off_as = take(sizeof(float) * static_cast<size_t>(P.slots) * (N / 128));
    P.off_z = take(sizeof(uint16_t) * static_cast<size_t>(P.R) * H);
    P.off_sync = take(sizeof(unsigned) * static_cast<size_t>(fused_counter_words(P.B_cap)));
    // the GEMMs' dynamic-tail counters (gate/up, down), directly followed by the epilogue-reduce
    // counters, so that route preparation zeroes both as one range
    P.off_sched = take(kSchedBytes);
    P.off_rcnt = take(sizeof(unsigned) * static_cast<size_t>(M) * (H / 128));
    P.off_kslot = take(sizeof(int32_t) * P.R);  // slots of the kept routes (compacting route prep)
    P.off_nkept = take(sizeof(int32_t));
    P.total = o;
    return P;
}

// AUTO forward path: the one measured faster on GB300 for the shape (graph-replayed layer on
// the decode shapes M = 1..256 and the expert-parallel shape): the staged launches at every
// measured size.  The fused persistent kernel and the reduce in the down GEMM's epilogue were
// slower everywhere (e.g. M = 32: 177 and 250 us against 162 us staged).
moe_forward_path auto_path(int M, int k, int E, int E_local, int H, int N) {
    (void)M; (void)E; (void)E_local; (void)H; (void)N;
    // top-k above the separate reduce kernel's limit: only the fused path takes it
    if (k > kReduceMaxTopk) return MOE_FORWARD_FUSED;
    return MOE_FORWARD_STAGED;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" const char* moe_last_error_string(void) { return g_err; }

extern "C" int moe_device_supported(void) { return device_is_sm103() ? 1 : 0; }

extern "C" int moe_pointer_device_accessible(const void* p) {
    if (!p) return 0;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // an unregistered host pointer: clear the error, answer no
        return 0;
    }
    switch (a.type) {
        case cudaMemoryTypeDevice: return a.device == current_device() ? 1 : 0;
        case cudaMemoryTypeManaged: return 1;
        // pinned host memory: usable in kernels only where the device sees it at the same address
        case cudaMemoryTypeHost: return a.devicePointer == p ? 1 : 0;
        default: return 0;
    }
}

extern "C" int moe_get_device_status(int* status, int reset) {
    clear_error();
    if (!status) { set_error("moe_get_device_status: null status"); return MOE_ERR_ARG; }
    *status = 0;
    int* p = device_status_ptr();
    if (!p) { set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    cudaError_t e = cudaMemcpy(status, p, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && reset) e = cudaMemset(p, 0, sizeof(int));
    if (e != cudaSuccess) { set_error("moe_get_device_status: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}

extern "C" int moe_forward_block_m(int M, int k, int E_local, int H, int N) {
    return forward_block_m(M, k, E_local, H, N);
}

extern "C" int moe_blockfp8_plan_for_sms(int M, int k, int E, int E_local, int H, int N,
                                         int block_m, int sms, int* out_block_m, int* out_B_cap,
                                         int* out_splits, int* out_dyn_gate_up,
                                         int* out_dyn_down) {
    clear_error();
    if (sms <= 0 || M < 0 || k <= 0 || E <= 0 || E_local <= 0 || H <= 0 || N <= 0 || H % 128 ||
        N % 128 || (block_m != 0 && block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128)) {
        set_error("moe_blockfp8_plan: bad sizes or SM count");
        return MOE_ERR_ARG;
    }
    const Plan P = make_plan(M, k, E, E_local, H, N, block_m, sms);
    if (out_block_m) *out_block_m = P.bm;
    if (out_B_cap) *out_B_cap = P.B_cap;
    if (out_splits) *out_splits = P.splits;
    if (out_dyn_gate_up) *out_dyn_gate_up = dyn_tail(M, k, E, E_local, 2 * N, H, P.bm, sms) ? 1 : 0;
    if (out_dyn_down) *out_dyn_down = dyn_tail(M, k, E, E_local, H, N, P.bm, sms) ? 1 : 0;
    return MOE_OK;
}

extern "C" int moe_blockfp8_plan(int M, int k, int E, int E_local, int H, int N, int block_m,
                                 int* out_block_m, int* out_B_cap, int* out_splits) {
    return moe_blockfp8_plan_for_sms(M, k, E, E_local, H, N, block_m, sm_count(), out_block_m,
                                     out_B_cap, out_splits, nullptr, nullptr);
}

extern "C" int moe_blockfp8_dynamic_tail(int M, int k, int E, int E_local, int H, int N, int block_m,
                                         int* gate_up, int* down) {
    if (!gate_up || !down) {
        clear_error();
        set_error("moe_blockfp8_dynamic_tail: null outputs");
        return MOE_ERR_ARG;
    }
    return moe_blockfp8_plan_for_sms(M, k, E, E_local, H, N, block_m, sm_count(), nullptr, nullptr,
                                     nullptr, gate_up, down);
}

extern "C" size_t moe_blockfp8_workspace_bytes(int M, int k, int E, int E_local, int H, int N,
                                               int block_m) {
    if (M < 0 || k <= 0 || E <= 0 || E_local <= 0 || H <= 0 || N <= 0) return 0;
    return make_plan(M, k, E, E_local, H, N, block_m, sm_count()).total;
}

extern "C" int moe_blockfp8_forward(const void* x, const int32_t* topk_ids, const float* topk_w,
                                    int M, int k, int E, const int32_t* expert_map, int E_local,
                                    int H, int N, const uint8_t* wgu_q, const float* wgu_s,
                                    const uint8_t* wd_q, const float* wd_s,
                                    moe_weight_layout w_layout, moe_act act,
                                    float clamp_limit, moe_scale_fmt act_fmt, int block_m,
                                    moe_forward_path path, void* out, void* workspace,
                                    size_t ws_bytes, cudaStream_t stream) {
    clear_error();
    if (!device_is_sm103()) { set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    if (!wgu_q || !wgu_s || !wd_q || !wd_s || (M > 0 && (!x || !topk_ids || !topk_w || !out))) {
        set_error("moe_blockfp8_forward: null pointer");
        return MOE_ERR_ARG;
    }
    if (M < 0 || k <= 0 || E <= 0 || E_local <= 0 || H <= 0 || N <= 0 || H % 128 || N % 128) {
        set_error("moe_blockfp8_forward: need M >= 0, k, E, E_local > 0 and H, N multiples of 128");
        return MOE_ERR_ARG;
    }
    if (k > E) { set_error("moe_blockfp8_forward: k > E"); return MOE_ERR_ARG; }
    // the staged path's separate reduce kernel takes at most kReduceMaxTopk routes per token;
    // AUTO sends larger top-k to the fused path (no limit), an explicit STAGED is refused here,
    // before anything is enqueued
    if (k > kReduceMaxTopk && (path == MOE_FORWARD_STAGED || path == MOE_FORWARD_STAGED_EPILOGUE_REDUCE)) {
        set_error("moe_blockfp8_forward: the staged path takes top-k <= %d (got %d); use FUSED or AUTO",
                  kReduceMaxTopk, k);
        return MOE_ERR_ARG;
    }
    if (act != MOE_ACT_SILU_MUL && act != MOE_ACT_SILU_MUL_GATE_UPPER) {
        set_error("moe_blockfp8_forward: act must be SILU_MUL or SILU_MUL_GATE_UPPER");
        return MOE_ERR_ARG;
    }
    if (block_m != 0 && block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128) {
        set_error("moe_blockfp8_forward: block_m must be 0 (auto), 16, 32, 64 or 128");
        return MOE_ERR_ARG;
    }
    if (path != MOE_FORWARD_AUTO && path != MOE_FORWARD_FUSED && path != MOE_FORWARD_STAGED &&
        path != MOE_FORWARD_STAGED_EPILOGUE_REDUCE) {
        set_error("moe_blockfp8_forward: unknown path %d", static_cast<int>(path));
        return MOE_ERR_ARG;
    }
    if (M > 0 && (!aligned16(x) || !aligned16(wgu_q) || !aligned16(wd_q) || !aligned16(out) ||
                  !aligned16(wgu_s) || !aligned16(wd_s))) {
        set_error("moe_blockfp8_forward: x, out and the weight tensors must be 16-byte aligned");
        return MOE_ERR_ARG;
    }
    if (!expert_map && E_local != E) {
        set_error("moe_blockfp8_forward: without an expert map E_local must equal E");
        return MOE_ERR_EXPERT_SLICE;
    }
    if (static_cast<long long>(M) * k > (1LL << 24)) { set_error("moe_blockfp8_forward: too many routes"); return MOE_ERR_ARG; }
    const Plan P = make_plan(M, k, E, E_local, H, N, block_m, sm_count());
    if (!workspace || ws_bytes < P.total || (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
        set_error("moe_blockfp8_forward: need %zu bytes of 256-byte aligned workspace (got %zu)", P.total, ws_bytes);
        return MOE_ERR_WORKSPACE;
    }
    if (M == 0) return MOE_OK;
    char* ws = static_cast<char*>(workspace);
    int32_t* sorted_idx = reinterpret_cast<int32_t*>(ws + P.off_sorted);
    int32_t* block_expert = reinterpret_cast<int32_t*>(ws + P.off_bexp);
    int32_t* num_blocks = reinterpret_cast<int32_t*>(ws + P.off_nb);
    int32_t* counts = reinterpret_cast<int32_t*>(ws + P.off_cnt);
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + P.off_off);
    int32_t* route_slot = reinterpret_cast<int32_t*>(ws + P.off_rslot);
    uint8_t* xq = reinterpret_cast<uint8_t*>(ws + P.off_xq);
    float* xs = reinterpret_cast<float*>(ws + P.off_xs);
    float* gu = reinterpret_cast<float*>(ws + P.off_gu);
    uint8_t* aq = reinterpret_cast<uint8_t*>(ws + P.off_aq);
    float* as = reinterpret_cast<float*>(ws + P.off_as);
    void* z = ws + P.off_z;
    const size_t rws_bytes = P.off_xq - P.off_rws;
    if (path == MOE_FORWARD_AUTO) path = auto_path(M, k, E, E_local, H, N);
    const bool fused = path == MOE_FORWARD_FUSED;
    // the weighted sum in the down GEMM's epilogue (block_m <= 32; otherwise the reduce kernel)
    const bool epi_reduce = path == MOE_FORWARD_STAGED_EPILOGUE_REDUCE && P.bm <= 32;
    unsigned* rcnt = reinterpret_cast<unsigned*>(ws + P.off_rcnt);
    unsigned* sync = reinterpret_cast<unsigned*>(ws + P.off_sync);
    unsigned long long* sched = reinterpret_cast<unsigned long long*>(ws + P.off_sched);
    // Route preparation in one CTA (more than a warp's routes) leaves the -1 pads of sorted_idx
    // to the input quantisation, which runs on every SM; every reader of sorted_idx comes after
    // it.  Measured on GB300 (interleaved A/B): prefill 733.5 -> 728.3 us, decode M=32 161.7 ->
    // 161.0, smaller sizes unchanged (the one-warp path still writes its own pads).
    const bool defer_pads = P.R > kRouteWarpMaxRoutes;
    // With an expert map, route preparation's compacting path lists the kept routes' slots, and
    // the activation kernel walks exactly those rows: at the expert-parallel shape 739 rows
    // instead of the blocks' 1056 slots, a third of them pads whose loads went for nothing.
    const bool kept_walk = route_compacts(P.R, E, E_local, expert_map != nullptr);
    int32_t* kept_slot = reinterpret_cast<int32_t*>(ws + P.off_kslot);
    int32_t* n_kept = reinterpret_cast<int32_t*>(ws + P.off_nkept);
    const bool dyn_gu = dyn_tail(M, k, E, E_local, 2 * N, H, P.bm, sm_count());
    const bool dyn_dn = dyn_tail(M, k, E, E_local, H, N, P.bm, sm_count());

    int rc;
    if (fused) {
        rc = launch_route_prepare(topk_ids, M, k, E, expert_map, E_local, P.bm, MOE_ROUTE_AUTO,
                                  sorted_idx, block_expert, num_blocks, counts, offsets,
                                  route_slot, ws + P.off_rws, rws_bytes, false, stream, sync,
                                  fused_counter_words(P.B_cap));
        if (rc) return rc;
        FusedLaunch f{};
        f.x = x; f.topk_ids = topk_ids; f.topk_w = topk_w; f.expert_map = expert_map;
        f.M = M; f.k = k; f.E = E; f.E_local = E_local; f.H = H; f.N = N; f.bm = P.bm;
        f.B_cap = P.B_cap; f.slots = P.slots;
        f.wgu_q = wgu_q; f.wgu_s = wgu_s; f.wd_q = wd_q; f.wd_s = wd_s; f.w_layout = w_layout;
        f.act = act; f.clamp_limit = clamp_limit; f.fmt = act_fmt;
        f.sorted_idx = sorted_idx; f.block_expert = block_expert; f.num_blocks = num_blocks;
        f.route_slot = route_slot;
        f.xq = xq; f.xsT = xs; f.gu = gu; f.aq = aq; f.asT = as; f.z = z; f.out = out;
        f.sync = sync;
        return launch_fused_layer(f, stream);
    }
    rc = launch_route_prepare(topk_ids, M, k, E, expert_map, E_local, P.bm, MOE_ROUTE_AUTO,
                              sorted_idx, block_expert, num_blocks, counts, offsets, route_slot,
                              ws + P.off_rws, rws_bytes, false, stream,
                              reinterpret_cast<uint32_t*>(sched),
                              static_cast<int>(kSchedBytes / 4) + (epi_reduce ? M * (H / 128) : 0),
                              defer_pads, kept_walk ? kept_slot : nullptr, kept_walk ? n_kept : nullptr);
    if (rc) return rc;
    // A few routes (decode batches of 1-4 tokens at top-8): the gate/up GEMM sorts them itself
    // from topk_ids, so its weight stream starts while routing and input quantisation still run;
    // the input quantisation releases it at once.  Otherwise the input quantisation releases the
    // GEMM only after its own routing wait, and the GEMM reads route preparation's tables as soon
    // as it starts.  Measured on GB300 against releasing at once with the GEMM waiting for the
    // whole input quantisation first: decode M=8 -1.3 us, M=64 and 256 -1.3/-1.4, M=16 and 32
    // -0.75/-0.4, expert-parallel T=1024 -0.95, prefill -1.3, T=100 unchanged.
    const bool self_route = P.R <= kSelfRouteMaxRoutes && P.bm <= 32;
    rc = launch_input_quant_tokens(x, M, H, k, route_slot, P.slots, xq, xs, act_fmt, true, stream,
                                   defer_pads ? offsets : nullptr, counts,
                                   defer_pads ? sorted_idx : nullptr, E_local, !self_route);
    if (rc) return rc;
    // The gate/up output: fp32 split partials, or with a single split the BF16 value the
    // act-quant would round it to (the same round-to-nearest-even), at half the bytes written and
    // read.  Measured on GB300: prefill 710.1 -> 704.1 us, decode M=128 and 256 -0.4 us.
    const moe_dtype gu_dtype = P.splits == 1 ? MOE_DTYPE_BF16 : MOE_DTYPE_F32;
    if (self_route)
        rc = launch_grouped_gemm(MOE_PROJ_GATE_UP, xq, xs, P.slots, H, wgu_q, wgu_s, E_local, 2 * N,
                                 w_layout, sorted_idx, block_expert, num_blocks, P.B_cap, P.bm, gu,
                                 gu_dtype, P.slots, P.splits, true, stream, /*wait_first=*/false,
                                 topk_ids, expert_map, P.R, E, nullptr, dyn_gu ? sched : nullptr);
    else
        rc = launch_grouped_gemm(MOE_PROJ_GATE_UP, xq, xs, P.slots, H, wgu_q, wgu_s, E_local, 2 * N,
                                 w_layout, sorted_idx, block_expert, num_blocks, P.B_cap, P.bm, gu,
                                 gu_dtype, P.slots, P.splits, true, stream, /*wait_first=*/false,
                                 nullptr, nullptr, 0, 0, nullptr, dyn_gu ? sched : nullptr);
    if (rc) return rc;
    // act-quant walks the routes (through route_slot) or, when the blocks hold fewer slots than
    // there are routes (an expert map that keeps few of them), the slots of the blocks that exist
    const bool slot_rows = expected_blocks(M, k, E, E_local, P.bm) * P.bm < P.R;
    // With at most 4 gate/up splits the act-quant releases the down GEMM before its own wait:
    // the down GEMM's CTAs then take SMs as gate/up CTAs leave and prefetch their weights while
    // the act-quant runs.  Everything the down GEMM reads before its wait (routing, weights) was
    // written before the gate/up GEMM was launched.  Measured on GB300 (interleaved A/B): decode
    // M=16 -2.4 us, M=32 -2.85, M=64 and 256 -0.45/-0.25; with 7 splits (M=8) +1.75, not taken.
    const bool aq_early = P.splits <= 4;
    if (kept_walk)
        rc = launch_act_quant(act, gu, gu_dtype, P.splits, P.slots, P.R, N, clamp_limit, act_fmt,
                              nullptr, nullptr, 0, kept_slot, 0, P.slots, aq, as, MOE_QUANT_PERSISTENT,
                              true, stream, /*map_early=*/true, nullptr, nullptr, 0, n_kept, aq_early);
    else if (slot_rows)
        rc = launch_act_quant(act, gu, gu_dtype, P.splits, P.slots, P.slots, N, clamp_limit, act_fmt,
                              nullptr, nullptr, 0, nullptr, 0, P.slots, aq, as, MOE_QUANT_PERSISTENT,
                              true, stream, false, sorted_idx, num_blocks, P.bm, nullptr, aq_early);
    else
        rc = launch_act_quant(act, gu, gu_dtype, P.splits, P.slots, P.R, N, clamp_limit, act_fmt,
                              nullptr, nullptr, 0, route_slot, 0, P.slots, aq, as,
                              MOE_QUANT_PERSISTENT, true, stream, /*map_early=*/true, nullptr, nullptr,
                              0, nullptr, aq_early);
    if (rc) return rc;
    if (epi_reduce) {
        const EpilogueReduce red{out, rcnt, topk_w, route_slot, k, M};
        return launch_grouped_gemm(MOE_PROJ_DOWN, aq, as, P.slots, N, wd_q, wd_s, E_local, H, w_layout,
                                   sorted_idx, block_expert, num_blocks, P.B_cap, P.bm, z,
                                   MOE_DTYPE_BF16, P.R, 1, true, stream, false, nullptr, nullptr, 0, 0,
                                   &red, dyn_dn ? sched + 1 : nullptr);
    }
    rc = launch_grouped_gemm(MOE_PROJ_DOWN, aq, as, P.slots, N, wd_q, wd_s, E_local, H, w_layout,
                             sorted_idx,
                             block_expert, num_blocks, P.B_cap, P.bm, z, MOE_DTYPE_BF16, P.R, 1,
                             true, stream, false, nullptr, nullptr, 0, 0, nullptr,
                             dyn_dn ? sched + 1 : nullptr);
    if (rc) return rc;
    return launch_moe_reduce(z, topk_w, topk_ids, expert_map, M, k, E, E_local, H, out, true, stream);
}

extern "C" int moe_blockfp8_workspace_layout(int M, int k, int E, int E_local, int H, int N,
                                             int block_m, size_t* offsets) {
    clear_error();
    if (!offsets || M < 0 || k <= 0 || E <= 0 || E_local <= 0 || H <= 0 || N <= 0 || H % 128 ||
        N % 128 || (block_m != 0 && block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128)) {
        set_error("moe_blockfp8_workspace_layout: bad sizes or null offsets");
        return MOE_ERR_ARG;
    }
    const Plan P = make_plan(M, k, E, E_local, H, N, block_m, sm_count());
    offsets[MOE_WS_SORTED_IDX] = P.off_sorted;
    offsets[MOE_WS_BLOCK_EXPERT] = P.off_bexp;
    offsets[MOE_WS_NUM_BLOCKS] = P.off_nb;
    offsets[MOE_WS_EXPERT_COUNT] = P.off_cnt;
    offsets[MOE_WS_EXPERT_OFFSET] = P.off_off;
    offsets[MOE_WS_ROUTE_SLOT] = P.off_rslot;
    offsets[MOE_WS_XQ] = P.off_xq;
    offsets[MOE_WS_XS] = P.off_xs;
    offsets[MOE_WS_GU] = P.off_gu;
    offsets[MOE_WS_AQ] = P.off_aq;
    offsets[MOE_WS_AS] = P.off_as;
    offsets[MOE_WS_Z] = P.off_z;
    return MOE_OK;
}

extern "C" int moe_forward_path_for(int M, int k, int E, int E_local, int H, int N) {
    return auto_path(M, k, E, E_local, H, N);
}
