// fused_layer.cu -- the block-FP8 MoE layer after route preparation as ONE persistent kernel:
// input quantisation -> gate/up grouped GEMM -> fused SiLU*mul + quantisation -> down grouped
// GEMM -> weighted top-k reduce, with the expert weights streaming through the tensor-core
// pipeline from the first to the last phase.
//
// Method (the same arithmetic as the stage-by-stage entry points): lmdeploy PR #4956
// "Perf/pytorch block fp8 moe decode" -- "Active-expert block scheduling" (work only for expert
// blocks that received tokens) and "Fused SwiGLU and FP8 quantization" (no BF16 intermediate in
// memory); lmdeploy PR #4857 "optimize compact blocked FP8 MoE and route preparation" --
// compact blocks, transposed MMA for small block_m; vLLM PR #53875 "Fuse clamped MoE activation
// and UE8M0 FP8 block quantization" -- clamp, UE8M0 scales, W8A8 block shape [128, 128];
// lmdeploy PR #4228 "Moe Reduce kernel" -- weighted top-k sum, fp32 accumulation in top-k order.
//
// Why one kernel: at decode sizes the layer streams tens to hundreds of MB of expert weights,
// and five separate launches each pay a ramp-up and a tail during which HBM idles.  Here the
// grid (one CTA per SM, all co-resident) moves through the phases below, separated by counters
// in global memory (two grid-wide ones, per-block ones in between), and only the ACTIVATION
// side of each GEMM waits on a counter: the weight tiles of the next GEMM are loaded by TMA
// while the previous phase is still finishing.
//
//   P0  every CTA quantises a slice of the x rows (per-128 E4M3 + scale, once per token) and
//       stores them to the expert-sorted slots of the token's routes; grid counter 0.
//   P1  gate/up GEMM.  Its K-blocks are dealt to the CTAs stream-K fashion: the flattened
//       (unit, K-block) space is cut into equal contiguous ranges, so a unit (block, 128-row
//       tile) can be split between neighbouring CTAs; piece p of a unit writes its fp32 partial
//       sum to partial slot p and counts itself in its block's counter (blk_done).
//   P2  fused act-quant: every CTA takes the slots of a contiguous range of blocks (so mostly
//       the blocks whose gate/up pieces it has just produced); an item (slot, group) waits only
//       for its own block's pieces, adds them in K order, rounds to BF16, optionally clamps,
//       a = bf16(SiLU(g)*u), per-128 E4M3 + scale.  The item that completes a block appends
//       it to the ready list.
//   P3  down GEMM over (block, 128-row tile) units, BF16 rows scattered to route order.  The
//       units are handed out dynamically, in the order the blocks became ready, from a global
//       counter: an SM that finished its gate/up work early starts on the down work at once,
//       and SMs that stream slower take fewer units; grid counter 3 when all are stored.
//   P4  every CTA (all its threads) reduces a slice of the tokens: out = bf16(sum_j w_j z_j)
//       in top-k order.
//
// Warp roles (256 threads): warp 0 lane 0 TMA weight producer; warp 7 lane 0 TMA activation
// producer (the only producer that waits on counters); warp 1 lane 0 MMA issuer; warps 2-5
// epilogue and the P0/P2 work; warp 6 metadata (descriptor ring); P4 uses all warps.  A
// pipeline stage holds two K-blocks; its full barrier completes when both producers have
// arrived and all bytes landed.  Every wait is bounded: on a timeout the CTA records
// MOE_DEV_TIMEOUT, stops publishing (the other CTAs then time out too) and leaves.
#include "common.cuh"

#include <algorithm>

namespace moe {
namespace {

struct FusedArgs {
    // routing, complete before this kernel reads it
    const int32_t* sorted_idx;
    const int32_t* block_expert;
    const int32_t* num_blocks;
    const int32_t* route_slot;
    const int32_t* topk_ids;
    const float* topk_w;
    const int32_t* expert_map;
    int B_cap, M, k, E, E_local, R, slots;
    // sizes: gate/up K = H (KB1 blocks), 2N outputs (NT1 tiles); down K = N (KB2), H (NT2)
    int H, N, KB1, NT1, KB2, NT2;
    const uint16_t* x;    // [M, H] bf16
    float* xsT;           // [KB1, slots] token scales of the quantised input (K-block major)
    const float* wgu_s;   // [E_local, NT1, KB1]
    float* gu;            // [pieces, nblk * BM, 2N] fp32 partial sums
    uint8_t* xq;          // [slots, H] E4M3 (through the activation map of P1)
    uint8_t* aq;          // [slots, N] E4M3 (through the activation map of P3)
    float* asT;           // [KB2, slots]
    const float* wd_s;    // [E_local, NT2, KB2]
    uint16_t* z;          // [R, H] bf16, route order
    uint16_t* out;        // [M, H] bf16
    float L;
    int act, fmt, w_tiled;
    unsigned* sync;       // [4]: 0 input quantised (grid), 1 ready blocks, 2 down units handed
                          // out, 3 down done (grid)
    unsigned* blk_done;   // [B_cap] gate/up tile pieces stored per block (x4 epilogue warps)
    unsigned* blk_ready;  // [B_cap] act-quant items (slot, group) done per block, pads included
    unsigned* ready_list; // [B_cap] 1 + block id, in the order the blocks became ready
    int* status;
    // limit of the counter waits (ns), and a test hook: block stall_block's act-quant items wait
    // for one gate/up piece more than exist, so that wait can only run out (-1: none)
    unsigned long long wait_limit_ns;
    int stall_block;
};

template <int BM>
struct FCfg {
    static constexpr int kWBytes = 128 * 128;
    static constexpr int kABytes = BM * 128;
    static constexpr int kKps = 2;
    static constexpr int kStage = kKps * (kWBytes + kABytes);
    static constexpr int kStages = BM <= 16 ? 6 : BM <= 32 ? 5 : BM <= 64 ? 4 : 3;
    static constexpr int kTSlots = BM <= 64 ? 4 : 2;
    static constexpr int kSlotCols = kKps * BM;
    static constexpr int kCols = kTSlots * kSlotCols <= 32 ? 32 : kTSlots * kSlotCols <= 64 ? 64
                               : kTSlots * kSlotCols <= 128 ? 128 : kTSlots * kSlotCols <= 256 ? 256 : 512;
    static constexpr int kCK = 32;                     // K-blocks per descriptor
    static constexpr int kSwMax = 64;                  // weight-block scales per descriptor
    static constexpr int kRing = 8;
    // header ints: e, b, nt0, ntl, piece, kb0, nck, flags, 4 unused
    static constexpr int kDescHdr = 12;
    static constexpr int kDescInts = kDescHdr + BM + kSwMax;
    static constexpr int kDescBytes = ((kDescInts * 4) + 15) / 16 * 16;
    static constexpr int kBarBytes = 1024;
    static constexpr int kSmem = kStages * kStage + kRing * kDescBytes + kBarBytes + 1024;
    static constexpr int kThreads = 256;
    static_assert(kStage % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(kCK % kKps == 0, "descriptors hold whole stages");
    static_assert((kDescHdr * 4) % 16 == 0, "descriptor rows stay 16-byte aligned");
    static_assert(kSmem <= 232448, "shared memory per CTA");
};

// descriptor flags
constexpr int kFirst = 1, kLast = 2, kEnd = 4, kDown = 8, kMarker = 16;
constexpr int kEpiBar = 1;  // named barrier of the 128 epilogue threads

struct FDesc {
    int* hdr;
    int* rows;
    float* sw;
};

template <int BM>
__device__ __forceinline__ FDesc fdesc_at(uint8_t* ring, int slot) {
    using C = FCfg<BM>;
    int* base = reinterpret_cast<int*>(ring + slot * C::kDescBytes);
    return FDesc{base, base + C::kDescHdr, reinterpret_cast<float*>(base + C::kDescHdr + BM)};
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Orders generic-proxy global accesses with async-proxy (TMA) ones.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Named barrier of the epilogue group; the non-aligned form, because one lane of the group may
// arrive from a divergent path (a counter wait).
__device__ __forceinline__ void epi_sync() {
    asm volatile("barrier.sync %0, 128;" ::"n"(kEpiBar) : "memory");
}

// Waits (bounded, like mbar_wait, after `limit` ns) until the counter reaches `target`.
__device__ __noinline__ bool wait_counter(const unsigned* ctr, unsigned target, volatile int* abort,
                                          int* status, unsigned long long limit) {
    if (ld_acquire_gpu(ctr) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(32);
        if (ld_acquire_gpu(ctr) >= target) return true;
        if ((i & 15u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit) {
                if (status) atomicOr(status, MOE_DEV_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// The epilogue group finishes a phase: every thread's writes are done (named barrier), one
// thread publishes them (fence + counter increment) and waits until every CTA has done the
// same; the second named barrier releases the group.  Every epilogue thread executes both
// barriers, also after an abort, so the group never waits on a thread that left.
__device__ __forceinline__ void epi_phase_barrier(unsigned* ctr, unsigned G, int etid,
                                                  volatile int* abort, int* status,
                                                  unsigned long long limit) {
    epi_sync();
    if (etid == 0 && !*abort) {
        __threadfence();
        atomicAdd(ctr, 1u);
        wait_counter(ctr, G, abort, status, limit);
    }
    epi_sync();
}

// The gate/up K-blocks (W of them) are dealt to the first G1 = min(G, W) CTAs in the ranges
// [W*c/G1, W*(c+1)/G1): every such range holds at least one K-block, so the pieces of a unit
// come from consecutive CTAs with no empty range between them.  cta_of(x) is the CTA whose
// range holds position x.
__device__ __forceinline__ int cta_of(long long x, long long W, int G1) {
    return static_cast<int>(((x + 1) * G1 - 1) / W);
}

// Gate/up tile pieces of block b (its blk_done counter reaches 4x this).
__device__ __forceinline__ unsigned block_pieces(int b, int NT1, int KB1, long long W1, int G1) {
    unsigned n = 0;
    for (int nt = 0; nt < NT1; ++nt) {
        const long long u0 = (static_cast<long long>(b) * NT1 + nt) * KB1;
        n += static_cast<unsigned>(cta_of(u0 + KB1 - 1, W1, G1) - cta_of(u0, W1, G1) + 1);
    }
    return n;
}

template <int BM>
__global__ void __launch_bounds__(256, 1)
    k_moe_fused(const __grid_constant__ CUtensorMap tmap_w1, const __grid_constant__ CUtensorMap tmap_a1,
                const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_a2,
                FusedArgs p) {
    using C = FCfg<BM>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ring = smem + C::kStages * C::kStage;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + C::kRing * C::kDescBytes);
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* tempty = tfull + C::kTSlots;
    uint64_t* dfull = tempty + C::kTSlots;
    uint64_t* dempty = dfull + C::kRing;
    uint64_t* mma_done = dempty + C::kRing;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* w_taken = reinterpret_cast<volatile int*>(tmem_slot + 2);  // descriptors the weight producer took

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) { mbar_init(full + i, 2); mbar_init(empty + i, 1); }
        for (int i = 0; i < C::kTSlots; ++i) { mbar_init(tfull + i, 1); mbar_init(tempty + i, 128); }
        for (int i = 0; i < C::kRing; ++i) { mbar_init(dfull + i, 32); mbar_init(dempty + i, 131); }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        *w_taken = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_w1);
        tma_prefetch_desc(&tmap_w2);
    }
    if (warp == 7 && lane == 0) {
        tma_prefetch_desc(&tmap_a1);
        tma_prefetch_desc(&tmap_a2);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(tmem_slot, C::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // Route preparation (the launch this one depends on) is complete once a thread has passed
    // grid_dep_wait(); its outputs are read through L2 (ld.global.cg), the caller's inputs
    // through the read-only path.  The epilogue warps first load and quantise the input rows,
    // which do not depend on the routing, and wait inside P0; every other warp waits here.
    grid_dep_launch();
    const bool epi_warp = warp >= 2 && warp <= 5;
    if (!epi_warp) grid_dep_wait();
    int nblk = 0;
    long long W1 = 0;  // gate/up K-block work
    int G1 = 1;        // CTAs with gate/up work
    int rows1 = 0;     // rows of a partial-sum slot
    auto read_plan = [&]() {
        nblk = max(0, min(__ldcg(p.num_blocks), p.B_cap));
        W1 = static_cast<long long>(nblk) * p.NT1 * p.KB1;
        G1 = static_cast<int>(max(1LL, min(static_cast<long long>(G), W1)));
        rows1 = nblk * BM;
    };
    if (!epi_warp) read_plan();

    if (warp == 6) {
        // ---------------- metadata warp ----------------
        int slot = 0;
        uint32_t ph = 0;
        bool ok = true;
        int cur_b = -1, e = -1, nkept = 0;
        long long base_desc = 0;  // descriptors written so far (all phases, markers included)
        int rows[(BM + 31) / 32];
        // Writes one descriptor (tiles nt0..nt0+ntl-1 of block b, K-blocks [c0, c0+nck)).
        auto emit = [&](int down, int b, int nt0, int ntl, int piece, int c0, int nck, int flags) {
            const float* ws = down ? p.wd_s : p.wgu_s;
            const int NT = down ? p.NT2 : p.NT1, KB = down ? p.KB2 : p.KB1;
            float sw_v[C::kSwMax / 32];
            const int n_sw = ntl * nck;
#pragma unroll
            for (int q = 0; q < C::kSwMax / 32; ++q) {
                const int i = q * 32 + lane;
                const int t = i / nck, kk = i - t * nck;
                sw_v[q] = i < n_sw ? __ldg(ws + (static_cast<long long>(e) * NT + nt0 + t) * KB + c0 + kk) : 0.0f;
            }
            ok = mbar_wait_fast(dempty + slot, ph ^ 1u, abort_flag, p.status);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; return; }
            FDesc d = fdesc_at<BM>(ring, slot);
            if (lane == 0) {
                d.hdr[0] = e; d.hdr[1] = b; d.hdr[2] = nt0; d.hdr[3] = ntl; d.hdr[4] = piece;
                d.hdr[5] = c0; d.hdr[6] = nck; d.hdr[7] = flags | (down ? kDown : 0);
            }
#pragma unroll
            for (int t = 0; t < (BM + 31) / 32; ++t)
                if (t * 32 + lane < BM) d.rows[t * 32 + lane] = rows[t];
#pragma unroll
            for (int q = 0; q < C::kSwMax / 32; ++q) {
                const int i = q * 32 + lane;
                if (i < n_sw) d.sw[i] = sw_v[q];
            }
            mbar_arrive(dfull + slot);
            if (++slot == C::kRing) { slot = 0; ph ^= 1u; }
            ++base_desc;
        };
        // Control descriptor (phase marker or end).
        auto emit_ctl = [&](int flags) {
            ok = mbar_wait_fast(dempty + slot, ph ^ 1u, abort_flag, p.status);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; return; }
            if (lane == 0) fdesc_at<BM>(ring, slot).hdr[7] = flags;
            mbar_arrive(dfull + slot);
            if (++slot == C::kRing) { slot = 0; ph ^= 1u; }
            ++base_desc;
        };
        // Loads block b's expert and output rows (down: route ids; gate/up: slot ids).
        auto load_block = [&](int b, int down) {
            int r_raw[(BM + 31) / 32];
#pragma unroll
            for (int t = 0; t < (BM + 31) / 32; ++t) {
                const int j = t * 32 + lane;
                r_raw[t] = j < BM ? __ldcg(p.sorted_idx + b * BM + j) : -1;
            }
            const int e_raw = __ldcg(p.block_expert + b);
            e = (e_raw >= 0 && e_raw < p.E_local) ? e_raw : -1;
#pragma unroll
            for (int t = 0; t < (BM + 31) / 32; ++t) {
                const int j = t * 32 + lane;
                int row = -1;
                if (j < BM && e >= 0) {
                    const int slot_j = b * BM + j;
                    const int r = r_raw[t];
                    row = r < 0 ? -1 : (down ? r : slot_j);
                    if (row >= (down ? p.R : p.slots)) {
                        if (p.status) atomicOr(p.status, MOE_DEV_BAD_INDEX);
                        row = -1;
                    }
                }
                rows[t] = row;
            }
            nkept = 0;
#pragma unroll
            for (int t = 0; t < (BM + 31) / 32; ++t) nkept += __popc(__ballot_sync(0xFFFFFFFFu, rows[t] >= 0));
            cur_b = b;
        };

        // ---- gate/up: stream-K over the K-blocks of all (block, tile) units ----
        {
            long long x = cta < G1 ? W1 * cta / G1 : W1;
            const long long x_hi = cta < G1 ? W1 * (cta + 1) / G1 : W1;
            long long u = x / p.KB1;
            int kb = static_cast<int>(x - u * p.KB1);
            int b = static_cast<int>(u / p.NT1), nt = static_cast<int>(u - static_cast<long long>(b) * p.NT1);
            while (x < x_hi && ok) {
                if (b != cur_b) load_block(b, 0);
                const int piece_end = static_cast<int>(min(static_cast<long long>(p.KB1), kb + (x_hi - x)));
                if (kb == 0 && piece_end == p.KB1 && p.KB1 <= C::kCK) {
                    // whole units from here: one descriptor for a run of tiles of this block
                    const int run = static_cast<int>(min(static_cast<long long>(p.NT1 - nt), (x_hi - x) / p.KB1));
                    const int ntl = min(run, C::kSwMax / p.KB1);
                    if (e >= 0) emit(0, b, nt, ntl, 0, 0, p.KB1, kFirst | kLast);
                    x += static_cast<long long>(ntl) * p.KB1;
                    nt += ntl;
                } else {
                    const int piece = cta - cta_of(u * p.KB1, W1, G1);
                    for (int c0 = kb; c0 < piece_end && ok && e >= 0; c0 += C::kCK) {
                        const int nck = min(C::kCK, piece_end - c0);
                        emit(0, b, nt, 1, piece, c0, nck,
                             (c0 == kb ? kFirst : 0) | (c0 + nck == piece_end ? kLast : 0));
                    }
                    x += piece_end - kb;
                    if (piece_end == p.KB1) { kb = 0; ++nt; } else { kb = piece_end; }
                }
                if (nt == p.NT1) { nt = 0; ++b; }
                u = static_cast<long long>(b) * p.NT1 + nt;
            }
        }
        if (ok) emit_ctl(kMarker);
        // ---- down: (block, tile) units handed out dynamically ----
        // Units are numbered (ready-list position, tile); a grab takes kGrab consecutive units.
        // A grab is made only when at most kAhead descriptors wait for the weight producer (on
        // top of the stages it has in flight), so a CTA holds about as much down work as its
        // pipeline needs to stay busy, and no more.
        if (ok) {
            constexpr int kAhead = 2;
            cur_b = -1;
            const long long units = static_cast<long long>(nblk) * p.NT2;
            int bi_cur = -1, b_ready = -1;
            long long seen = 0;  // the hand-out counter as last seen by this CTA
            for (;;) {
                {
                    // bounded wait until the weight producer has taken all but kAhead descriptors
                    const uint64_t t0 = globaltimer_ns();
                    bool late = false;
                    while (static_cast<long long>(*w_taken) + kAhead < base_desc) {
                        if (*abort_flag) { late = true; break; }
                        if (globaltimer_ns() - t0 > p.wait_limit_ns) {
                            if (lane == 0) {
                                if (p.status) atomicOr(p.status, MOE_DEV_TIMEOUT);
                                *abort_flag = 1;
                            }
                            late = true;
                            break;
                        }
                        __nanosleep(64);
                    }
                    if (__any_sync(0xFFFFFFFFu, late)) { ok = false; break; }
                }
                // grab size: up to 8 units while much work is left, down to 1 near the end
                const int grab = static_cast<int>(max(1LL, min(8LL, (units - seen) / (4LL * G))));
                long long g0 = 0;
                if (lane == 0) g0 = static_cast<long long>(atomicAdd(p.sync + 2, static_cast<unsigned>(grab)));
                g0 = __shfl_sync(0xFFFFFFFFu, g0, 0);
                seen = g0 + grab;
                if (g0 >= units) break;
                const long long g1 = min(units, g0 + grab);
                for (long long u = g0; u < g1 && ok;) {
                    const int bi = static_cast<int>(u / p.NT2);
                    const int nt = static_cast<int>(u - static_cast<long long>(bi) * p.NT2);
                    if (bi != bi_cur) {
                        // the block at ready-list position bi (bounded wait, acquire)
                        bool okw = true;
                        unsigned v = 0;
                        if (lane == 0) {
                            okw = wait_counter(p.ready_list + bi, 1u, abort_flag, p.status, p.wait_limit_ns);
                            v = ld_acquire_gpu(p.ready_list + bi);
                        }
                        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
                        v = __shfl_sync(0xFFFFFFFFu, v, 0);
                        if (!okw) { ok = false; break; }
                        b_ready = static_cast<int>(v) - 1;
                        bi_cur = bi;
                    }
                    const int b = b_ready;
                    if (b < 0 || b >= nblk) { if (lane == 0 && p.status) atomicOr(p.status, MOE_DEV_BAD_INDEX); ok = false; break; }
                    if (b != cur_b) load_block(b, 1);
                    const int run = static_cast<int>(min(static_cast<long long>(p.NT2 - nt), g1 - u));
                    int adv = run;
                    if (p.KB2 <= C::kCK) {
                        const int ntl = min(run, C::kSwMax / p.KB2);
                        if (e >= 0) emit(1, b, nt, ntl, 0, 0, p.KB2, kFirst | kLast);
                        adv = ntl;
                    } else {
                        for (int c0 = 0; c0 < p.KB2 && ok && e >= 0; c0 += C::kCK) {
                            const int nck = min(C::kCK, p.KB2 - c0);
                            emit(1, b, nt, 1, 0, c0, nck, (c0 == 0 ? kFirst : 0) | (c0 + nck == p.KB2 ? kLast : 0));
                        }
                        adv = 1;
                    }
                    u += adv;
                }
                if (!ok) break;
            }
        }
        if (ok) emit_ctl(kEnd);
    } else if (warp == 0 || warp == 7) {
        // ---------------- TMA producers: warp 0 weights, warp 7 activations ----------------
        if (lane == 0) {
            const bool wprod = warp == 0;
            const uint64_t pol = wprod ? l2_policy_evict_first() : l2_policy_evict_last();
            int s = 0, slot = 0;
            uint32_t ph = 0, dph = 0;
            long long issued = 0;
            bool ok = true;
            int ready_b = -1;
            if (!wprod) {
                // the quantised input rows of every CTA must be in memory before they are read
                ok = wait_counter(p.sync + 0, G, abort_flag, p.status, p.wait_limit_ns);
                fence_proxy_async_global();
            }
            while (ok) {
                if (!mbar_wait_fast(dfull + slot, dph, abort_flag, p.status)) break;
                const FDesc d = fdesc_at<BM>(ring, slot);
                const int flags = d.hdr[7];
                if (flags & kEnd) break;
                if (flags & kMarker) {
                    mbar_arrive(dempty + slot);
                    if (++slot == C::kRing) { slot = 0; dph ^= 1u; }
                    if (wprod) *w_taken = *w_taken + 1;
                    continue;
                }
                const int down = flags & kDown;
                const int e = d.hdr[0], b = d.hdr[1], nt0 = d.hdr[2], ntl = d.hdr[3];
                const int c0 = d.hdr[5], nck = d.hdr[6];
                mbar_arrive(dempty + slot);
                if (++slot == C::kRing) { slot = 0; dph ^= 1u; }
                if (wprod) *w_taken = *w_taken + 1;
                if (!wprod && down && b != ready_b) {
                    // The block's quantised activations were published before it entered the
                    // ready list; the metadata warp acquired that entry before writing this
                    // descriptor, and the descriptor hand-off orders this thread after it.  The
                    // proxy fence orders those generic-proxy writes before the TMA reads.
                    fence_proxy_async_global();
                    ready_b = b;
                }
                const CUtensorMap* map = wprod ? (down ? &tmap_w2 : &tmap_w1) : (down ? &tmap_a2 : &tmap_a1);
                const int NT = down ? p.NT2 : p.NT1, KB = down ? p.KB2 : p.KB1;
                const int Nout = down ? p.H : 2 * p.N;
                const uint32_t bytes = wprod ? C::kWBytes : C::kABytes;
                for (int t = 0; t < ntl && ok; ++t) {
                    const int nt = nt0 + t;
                    const long long wrow = p.w_tiled ? (static_cast<long long>(e) * NT + nt) * KB * 128
                                                     : static_cast<long long>(e) * Nout + nt * 128;
                    for (int kb = c0; kb < c0 + nck; kb += C::kKps) {
                        const int nk = min(C::kKps, c0 + nck - kb);
                        if (!mbar_wait_fast(empty + s, ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
                        uint8_t* st = smem + s * C::kStage;
                        mbar_arrive_expect_tx(full + s, static_cast<uint32_t>(nk) * bytes);
                        for (int j = 0; j < nk; ++j) {
                            if (wprod) {
                                if (p.w_tiled)
                                    tma_load_2d(st + j * C::kWBytes, map, full + s, 0,
                                                static_cast<int>(wrow + (kb + j) * 128), pol);
                                else
                                    tma_load_2d(st + j * C::kWBytes, map, full + s, (kb + j) * 128,
                                                static_cast<int>(wrow), pol);
                            } else {
                                tma_load_2d(st + C::kKps * C::kWBytes + j * C::kABytes, map, full + s,
                                            (kb + j) * 128, b * BM, pol);
                            }
                        }
                        ++issued;
                        if (++s == C::kStages) { s = 0; ph ^= 1u; }
                    }
                }
            }
            if (*abort_flag) {
                // never leave a TMA write in flight: wait (bounded) for the last load of every
                // stage.  A stage completes only when both producers have arrived, and the other
                // producer may have left on the abort first; its own loads land within
                // microseconds, so the kernel's wait limit bounds this wait
                for (int i = 0; i < C::kStages; ++i) {
                    if (issued <= i) break;
                    const long long n_i = (issued - 1 - i) / C::kStages + 1;
                    volatile int no_abort = 0;
                    mbar_wait(full + i, static_cast<uint32_t>((n_i - 1) & 1), &no_abort, p.status,
                              p.wait_limit_ns);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f8_f32(128, BM);
            int s = 0, ts = 0, slot = 0;
            uint32_t ph = 0, tph = 0, dph = 0;
            bool ok = true;
            while (ok) {
                if (!mbar_wait_fast(dfull + slot, dph, abort_flag, p.status)) break;
                const FDesc d = fdesc_at<BM>(ring, slot);
                const int flags = d.hdr[7];
                if (flags & kEnd) break;
                const int ntl = d.hdr[3], nck = d.hdr[6];
                mbar_arrive(dempty + slot);
                if (++slot == C::kRing) { slot = 0; dph ^= 1u; }
                if (flags & kMarker) continue;
                for (int t = 0; t < ntl && ok; ++t) {
                    for (int kk = 0; kk < nck; kk += C::kKps) {
                        const int nk = min(C::kKps, nck - kk);
                        if (!mbar_wait_fast(tempty + ts, tph ^ 1u, abort_flag, p.status)) { ok = false; break; }
                        if (!mbar_wait_fast(full + s, ph, abort_flag, p.status)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t wa = smem_u32(smem + s * C::kStage);
                        const uint32_t aa = wa + C::kKps * C::kWBytes;
                        const uint32_t dt = tmem_base + static_cast<uint32_t>(ts * C::kSlotCols);
                        for (int j = 0; j < nk; ++j) {
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                mma_f8(dt + j * BM, smem_desc_sw128(wa + j * C::kWBytes + ks * 32),
                                       smem_desc_sw128(aa + j * C::kABytes + ks * 32), idesc, ks > 0 ? 1u : 0u);
                        }
                        mma_commit(empty + s);
                        mma_commit(tfull + ts);
                        if (++s == C::kStages) { s = 0; ph ^= 1u; }
                        if (++ts == C::kTSlots) { ts = 0; tph ^= 1u; }
                    }
                }
            }
            mma_commit(mma_done);
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort, p.status, p.wait_limit_ns);
        }
    } else {
        // ---------------- epilogue group (warps 2..5) ----------------
        const int etid = threadIdx.x - 64;          // 0..127
        const int ewarp = etid >> 5;
        const int q = warp & 3;                     // tensor-memory lane quarter of this warp
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        const int r_in_tile = q * 32 + lane;
        const int half = lane >> 4, l = lane & 15;

        // ---- P0: input quantisation of this CTA's slice of (token, group) items ----
        // Each token row is quantised once and its codes and scale are stored to the slot of
        // every kept route of the token (the same values the per-route gather produces).  The
        // first kHold pairs of each warp are loaded and quantised before the wait for route
        // preparation (the input does not depend on it); only the stores to the slots follow it.
        {
            constexpr int kHold = 4;
            const long long groups = static_cast<long long>(p.M) * p.KB1;
            const long long pairs = (groups + 1) / 2;
            const long long lo = pairs * cta / G, hi = pairs * (cta + 1) / G;
            auto item_of = [&](long long pr, int& t, int& g) -> bool {
                const long long item = pr * 2 + half;
                if (pr >= hi || item >= groups) return false;
                t = static_cast<int>(item / p.KB1);
                g = static_cast<int>(item - static_cast<long long>(t) * p.KB1);
                return true;
            };
            auto scatter = [&](int t, int g, uint2 codes, float sc) {
                for (int j0 = 0; j0 < p.k; j0 += 8) {
                    int ms[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        ms[jj] = j0 + jj < p.k ? __ldcg(p.route_slot + t * p.k + j0 + jj) : -1;
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        int m = ms[jj];
                        if (m >= p.slots) { if (p.status) atomicOr(p.status, MOE_DEV_BAD_INDEX); m = -1; }
                        if (m < 0) continue;
                        *reinterpret_cast<uint2*>(p.xq + static_cast<long long>(m) * p.H + g * 128 + l * 8) = codes;
                        if (l == 0) p.xsT[static_cast<long long>(g) * p.slots + m] = sc;
                    }
                }
            };
            auto decode8 = [](const uint4& v, float* a) {
                a[0] = bf16_lo(v.x); a[1] = bf16_hi(v.x); a[2] = bf16_lo(v.y); a[3] = bf16_hi(v.y);
                a[4] = bf16_lo(v.z); a[5] = bf16_hi(v.z); a[6] = bf16_lo(v.w); a[7] = bf16_hi(v.w);
            };
            // the held pairs: all loads first, then the quantisation
            uint4 xv[kHold];
            int ht[kHold], hg[kHold];
            bool ha[kHold];
#pragma unroll
            for (int i = 0; i < kHold; ++i) {
                ha[i] = item_of(lo + ewarp + 4LL * i, ht[i], hg[i]);
                if (ha[i]) xv[i] = __ldg(reinterpret_cast<const uint4*>(
                               p.x + static_cast<long long>(ht[i]) * p.H + hg[i] * 128 + l * 8));
            }
            uint2 hc[kHold];
            float hs[kHold];
#pragma unroll
            for (int i = 0; i < kHold; ++i) {
                float a[8];
                if (ha[i]) decode8(xv[i], a);
                quant_group_codes_compact(a, ha[i], p.fmt, &hc[i], &hs[i]);
            }
            grid_dep_wait();  // route preparation is complete from here on
            read_plan();
#pragma unroll
            for (int i = 0; i < kHold; ++i)
                if (ha[i]) scatter(ht[i], hg[i], hc[i], hs[i]);
            for (long long pr = lo + ewarp + 4LL * kHold; pr < hi; pr += 4) {
                int t = 0, g = 0;
                const bool act = item_of(pr, t, g);
                float a[8];
                if (act) decode8(__ldg(reinterpret_cast<const uint4*>(p.x + static_cast<long long>(t) * p.H + g * 128 + l * 8)), a);
                uint2 codes;
                float sc;
                quant_group_codes_compact(a, act, p.fmt, &codes, &sc);
                if (act) scatter(t, g, codes, sc);
            }
            fence_proxy_async_global();  // the quantised rows are read by TMA
        }
        epi_phase_barrier(p.sync + 0, G, etid, abort_flag, p.status, p.wait_limit_ns);

        int ts = 0, slot = 0;
        uint32_t tph = 0, dph = 0;
        float acc[BM];
#pragma unroll
        for (int j = 0; j < BM; ++j) acc[j] = 0.0f;
        // One descriptor of GEMM work: promotion of every K-block's partial sums with the
        // token and weight-block scales, output at the end of each tile's K range.
        auto run_desc = [&](const FDesc& d, int down) -> bool {
            const int b = d.hdr[1], nt0 = d.hdr[2], ntl = d.hdr[3], piece = d.hdr[4];
            const int c0 = d.hdr[5], nck = d.hdr[6], flags = d.hdr[7];
            const float* sT = down ? p.asT : p.xsT;
            // (down: the block's scales were published before the block entered the ready list,
            // which the metadata warp acquired before writing this descriptor)
            for (int t = 0; t < ntl; ++t) {
                if (flags & kFirst) {
#pragma unroll
                    for (int j = 0; j < BM; ++j) acc[j] = 0.0f;
                }
                const float* swt = d.sw + t * nck;
                for (int kk = 0; kk < nck; kk += C::kKps) {
                    const int nk = min(C::kKps, nck - kk);
                    if constexpr (BM == 16) {
                        // token scales of the stage's K-blocks (plain loads: written in this
                        // kernel; issued before the wait so their latency overlaps it)
                        float sa[2][16];
#pragma unroll
                        for (int j2 = 0; j2 < 2; ++j2) {
                            const float4* src = reinterpret_cast<const float4*>(
                                sT + static_cast<long long>(c0 + kk + min(j2, nk - 1)) * p.slots + b * BM);
#pragma unroll
                            for (int j4 = 0; j4 < 4; ++j4) {
                                const float4 v4 = src[j4];
                                sa[j2][j4 * 4 + 0] = v4.x; sa[j2][j4 * 4 + 1] = v4.y;
                                sa[j2][j4 * 4 + 2] = v4.z; sa[j2][j4 * 4 + 3] = v4.w;
                            }
                        }
                        const bool okw = mbar_wait_fast(tfull + ts, tph, abort_flag, p.status);
                        if (!__all_sync(0xFFFFFFFFu, okw)) return false;
                        tc_fence_after();
                        const uint32_t t0 = lane_base + static_cast<uint32_t>(ts * C::kSlotCols);
                        float v[32];
                        tmem_ld32(t0, v);
                        tc_fence_before();
                        mbar_arrive_relaxed(tempty + ts);
#pragma unroll
                        for (int j2 = 0; j2 < 2; ++j2) {
                            if (j2 < nk) {
                                const float sw = swt[kk + j2];
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    acc[j] = __fmaf_rn(v[j2 * 16 + j], __fmul_rn(sa[j2][j], sw), acc[j]);
                            }
                        }
                    } else {
                        const bool okw = mbar_wait_fast(tfull + ts, tph, abort_flag, p.status);
                        if (!__all_sync(0xFFFFFFFFu, okw)) return false;
                        tc_fence_after();
                        const uint32_t t0 = lane_base + static_cast<uint32_t>(ts * C::kSlotCols);
                        for (int j2 = 0; j2 < nk; ++j2) {
                            const float sw = swt[kk + j2];
                            const float* srow = sT + static_cast<long long>(c0 + kk + j2) * p.slots + b * BM;
#pragma unroll
                            for (int c = 0; c < BM / 32; ++c) {
                                float v[32];
                                tmem_ld32(t0 + static_cast<uint32_t>(j2 * BM + c * 32), v);
#pragma unroll
                                for (int i4 = 0; i4 < 8; ++i4) {
                                    const float4 s4 = reinterpret_cast<const float4*>(srow + c * 32)[i4];
                                    const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        const int jj = c * 32 + i4 * 4 + i;
                                        acc[jj] = __fmaf_rn(v[i4 * 4 + i], __fmul_rn(sv[i], sw), acc[jj]);
                                    }
                                }
                            }
                        }
                        tc_fence_before();
                        mbar_arrive_relaxed(tempty + ts);
                    }
                    if (++ts == C::kTSlots) { ts = 0; tph ^= 1u; }
                }
                if (flags & kLast) {
                    const int n = (nt0 + t) * 128 + r_in_tile;
#pragma unroll
                    for (int j0 = 0; j0 < BM; j0 += 16) {
                        int rws[16];
#pragma unroll
                        for (int j4 = 0; j4 < 4; ++j4) {
                            const int4 r4 = reinterpret_cast<const int4*>(d.rows + j0)[j4];
                            rws[j4 * 4 + 0] = r4.x; rws[j4 * 4 + 1] = r4.y;
                            rws[j4 * 4 + 2] = r4.z; rws[j4 * 4 + 3] = r4.w;
                        }
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int row = rws[jj];
                            if (row < 0) continue;
                            if (down)
                                p.z[static_cast<long long>(row) * p.H + n] =
                                    static_cast<uint16_t>(f32_to_bf16_bits(acc[j0 + jj]));
                            else
                                p.gu[(static_cast<long long>(piece) * rows1 + row) * (2 * p.N) + n] = acc[j0 + jj];
                        }
                    }
                    if (!down) {
                        // this warp's 32 columns of the tile piece are stored
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) atomicAdd(p.blk_done + b, 1u);
                    }
                }
            }
            return true;
        };

        // ---- P1: gate/up epilogue ----
        bool ok = !*abort_flag;
        while (ok) {
            ok = mbar_wait_fast(dfull + slot, dph, abort_flag, p.status);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            const FDesc d = fdesc_at<BM>(ring, slot);
            const int flags = d.hdr[7];
            if (!(flags & (kMarker | kEnd))) ok = run_desc(d, 0);
            mbar_arrive_relaxed(dempty + slot);
            if (++slot == C::kRing) { slot = 0; dph ^= 1u; }
            if (flags & (kMarker | kEnd)) break;
        }

        // ---- P2: fused act-quant of the slots of this CTA's range of blocks ----
        // The CTA walks its slots 32 at a time; every warp drops the pad slots of the chunk
        // (ballot over sorted_idx) and the remaining (slot, group) items are dealt to the 8
        // half-warps of the group, so a chunk takes one pass.  An item waits only for the
        // gate/up pieces of its own block.  Every stored item, and warp 0 for the pad items of the
        // chunk, counts itself in its block; the count that completes a block (BM * N/128)
        // appends the block to the ready list.
        if (!*abort_flag) {
            const int GN = p.N / 128;
            const int W = 2 * p.N;
            const unsigned blk_items = static_cast<unsigned>(BM * GN);
            const long long pstride = static_cast<long long>(rows1) * W;
            const long long s_lo = static_cast<long long>(nblk) * cta / G * BM;
            const long long s_hi = static_cast<long long>(nblk) * (cta + 1) / G * BM;
            bool stop = false;
            auto count_in = [&](long long bb, unsigned cnt) {
                const unsigned old = atomicAdd(p.blk_ready + bb, cnt);
                if (old + cnt == blk_items) {
                    // acquire the other items' stores of this block (each was released by a
                    // fence + atomic), then publish the block
                    __threadfence();
                    const unsigned pos = atomicAdd(p.sync + 1, 1u);
                    if (pos < static_cast<unsigned>(nblk))
                        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.ready_list + pos),
                                     "r"(static_cast<unsigned>(bb) + 1u) : "memory");
                }
            };
            for (long long base = s_lo; base < s_hi && !stop; base += 32) {
                const long long m_l = base + lane;
                const bool real = m_l < s_hi && __ldcg(p.sorted_idx + m_l) >= 0;
                const unsigned mask = __ballot_sync(0xFFFFFFFFu, real);
                const int n_items = __popc(mask) * GN;
                for (int it0 = 2 * ewarp; it0 < n_items && !stop; it0 += 8) {
                    const int it = it0 + half;
                    const bool active = it < n_items;
                    int m = static_cast<int>(base), g = 0;
                    if (active) {
                        const int kth = it / GN;
                        g = it - kth * GN;
                        unsigned mm = mask;
                        for (int q2 = 0; q2 < kth; ++q2) mm &= mm - 1;
                        m = static_cast<int>(base) + __ffs(mm) - 1;
                    }
                    const int b = m / BM;
                    {
                        // wait (bounded, the whole warp) until every active item's block is stored
                        const unsigned tgt = active ? 4u * block_pieces(b, p.NT1, p.KB1, W1, G1) +
                                                          (b == p.stall_block ? 1u : 0u) : 0u;
                        const uint64_t t0 = globaltimer_ns();
                        for (;;) {
                            const bool rdy = !active || ld_acquire_gpu(p.blk_done + b) >= tgt;
                            if (__all_sync(0xFFFFFFFFu, rdy)) break;
                            if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
                            if (globaltimer_ns() - t0 > p.wait_limit_ns) {
                                if (lane == 0) {
                                    if (p.status) atomicOr(p.status, MOE_DEV_TIMEOUT);
                                    *abort_flag = 1;
                                }
                                __syncwarp();
                            }
                            __nanosleep(32);
                        }
                        if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) { stop = true; break; }
                    }
                    float a[8];
                    if (active) {
                        // gate tile g and up tile N/128 + g: each unit's pieces added in K order;
                        // the loads of four pieces of both tiles are issued together
                        const long long ug = static_cast<long long>(b) * p.NT1 + g;
                        const long long uu = ug + GN;
                        const int cg = cta_of(ug * p.KB1, W1, G1);
                        const int cu = cta_of(uu * p.KB1, W1, G1);
                        const int npg = cta_of(ug * p.KB1 + p.KB1 - 1, W1, G1) - cg + 1;
                        const int npu = cta_of(uu * p.KB1 + p.KB1 - 1, W1, G1) - cu + 1;
                        const float* srcg = p.gu + static_cast<long long>(m) * W + g * 128 + l * 8;
                        const float* srcu = srcg + p.N;
                        float gv[8], uv[8];
                        const int npmax = max(npg, npu);
                        for (int pc0 = 0; pc0 < npmax; pc0 += 4) {
                            float4 ga[4], gb[4], ua[4], ub[4];
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                if (pc0 + q4 < npg) {
                                    const float* s2 = srcg + (pc0 + q4) * pstride;
                                    ga[q4] = *reinterpret_cast<const float4*>(s2);
                                    gb[q4] = *reinterpret_cast<const float4*>(s2 + 4);
                                }
                                if (pc0 + q4 < npu) {
                                    const float* s2 = srcu + (pc0 + q4) * pstride;
                                    ua[q4] = *reinterpret_cast<const float4*>(s2);
                                    ub[q4] = *reinterpret_cast<const float4*>(s2 + 4);
                                }
                            }
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const int pc = pc0 + q4;
                                if (pc < npg) {
                                    if (pc == 0) {
                                        gv[0] = ga[0].x; gv[1] = ga[0].y; gv[2] = ga[0].z; gv[3] = ga[0].w;
                                        gv[4] = gb[0].x; gv[5] = gb[0].y; gv[6] = gb[0].z; gv[7] = gb[0].w;
                                    } else {
                                        gv[0] = __fadd_rn(gv[0], ga[q4].x); gv[1] = __fadd_rn(gv[1], ga[q4].y);
                                        gv[2] = __fadd_rn(gv[2], ga[q4].z); gv[3] = __fadd_rn(gv[3], ga[q4].w);
                                        gv[4] = __fadd_rn(gv[4], gb[q4].x); gv[5] = __fadd_rn(gv[5], gb[q4].y);
                                        gv[6] = __fadd_rn(gv[6], gb[q4].z); gv[7] = __fadd_rn(gv[7], gb[q4].w);
                                    }
                                }
                                if (pc < npu) {
                                    if (pc == 0) {
                                        uv[0] = ua[0].x; uv[1] = ua[0].y; uv[2] = ua[0].z; uv[3] = ua[0].w;
                                        uv[4] = ub[0].x; uv[5] = ub[0].y; uv[6] = ub[0].z; uv[7] = ub[0].w;
                                    } else {
                                        uv[0] = __fadd_rn(uv[0], ua[q4].x); uv[1] = __fadd_rn(uv[1], ua[q4].y);
                                        uv[2] = __fadd_rn(uv[2], ua[q4].z); uv[3] = __fadd_rn(uv[3], ua[q4].w);
                                        uv[4] = __fadd_rn(uv[4], ub[q4].x); uv[5] = __fadd_rn(uv[5], ub[q4].y);
                                        uv[6] = __fadd_rn(uv[6], ub[q4].z); uv[7] = __fadd_rn(uv[7], ub[q4].w);
                                    }
                                }
                            }
                        }
                        // (out of line: this runs once per item, where instruction fetch dominates)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            a[i] = silu_mul_bf16_rt(bf16_round_f32(gv[i]), bf16_round_f32(uv[i]), p.L, p.act);
                    }
                    {
                        uint2 codes;
                        float sc;
                        quant_group_codes_compact(a, active, p.fmt, &codes, &sc);
                        if (active) {
                            *reinterpret_cast<uint2*>(p.aq + static_cast<long long>(m) * p.N + g * 128 + l * 8) = codes;
                            if (l == 0) p.asT[static_cast<long long>(g) * p.slots + m] = sc;
                        }
                    }
                    fence_proxy_async_global();  // the quantised activations are read by TMA
                    __threadfence();
                    __syncwarp();
                    if (active && l == 0) count_in(b, 1u);
                }
                if (stop) break;
                // pad items of this chunk, counted once (warp 0)
                if (ewarp == 0 && lane == 0) {
                    const long long c_hi = min(base + 32, s_hi);
                    for (long long bb = base / BM; bb * BM < c_hi; ++bb) {
                        const long long lo_s = max(bb * BM, base), hi_s = min((bb + 1) * BM, c_hi);
                        const unsigned slots_in = static_cast<unsigned>(hi_s - lo_s);
                        unsigned reals = 0;
                        for (long long mm = lo_s; mm < hi_s; ++mm) reals += (mask >> (mm - base)) & 1u;
                        const unsigned pads = (slots_in - reals) * GN;
                        if (pads) count_in(bb, pads);
                    }
                }
            }
        }

        // ---- P3: down epilogue ----
        ok = !*abort_flag;
        while (ok) {
            ok = mbar_wait_fast(dfull + slot, dph, abort_flag, p.status);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            const FDesc d = fdesc_at<BM>(ring, slot);
            const int flags = d.hdr[7];
            if (!(flags & (kMarker | kEnd))) ok = run_desc(d, 1);
            mbar_arrive_relaxed(dempty + slot);
            if (++slot == C::kRing) { slot = 0; dph ^= 1u; }
            if (flags & kEnd) break;
        }
    }

    // ---- P4 (all 256 threads): weighted top-k reduce of this CTA's slice of (token,
    // 8 columns) items.  The ids, weights and keep flags of each thread's first item are
    // loaded before the last grid counter, so only the z rows are read after it.
    const int C8 = p.H / 8;
    const long long items4 = static_cast<long long>(p.M) * C8;
    const long long lo4 = items4 * cta / G, hi4 = items4 * (cta + 1) / G;
    int ids8[8];
    float w8[8];
    bool keep8[8];
    auto load_routes = [&](int t, int j0) {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int r = t * p.k + j0 + jj;
            const bool in = j0 + jj < p.k;
            ids8[jj] = in ? __ldg(p.topk_ids + r) : -1;
            w8[jj] = in ? __ldg(p.topk_w + r) : 0.0f;
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int id = ids8[jj];
            bool keep = id >= 0 && id < p.E;
            if (keep && p.expert_map) {
                const int le = __ldg(p.expert_map + id);
                keep = le >= 0 && le < p.E_local;
            }
            keep8[jj] = keep;
        }
    };
    long long it4 = lo4 + threadIdx.x;
    if (it4 < hi4) load_routes(static_cast<int>(it4 / C8), 0);
    if (warp >= 2 && warp <= 5)
        epi_phase_barrier(p.sync + 3, G, static_cast<int>(threadIdx.x) - 64, abort_flag, p.status,
                          p.wait_limit_ns);
    __syncthreads();  // every role is done; the epilogue group has passed the last counter
    if (!*abort_flag) {
        bool first = true;
        for (; it4 < hi4; it4 += blockDim.x) {
            const int t = static_cast<int>(it4 / C8);
            const int col = static_cast<int>(it4 - static_cast<long long>(t) * C8) * 8;
            float accr[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            // routes in groups of eight: ids, weights and rows of a group are loaded together;
            // the multiply-adds run in top-k order
            for (int j0 = 0; j0 < p.k; j0 += 8) {
                if (!(first && j0 == 0)) load_routes(t, j0);
                uint4 v8[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    if (keep8[jj])
                        v8[jj] = *reinterpret_cast<const uint4*>(
                            p.z + static_cast<long long>(t * p.k + j0 + jj) * p.H + col);
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    if (!keep8[jj]) continue;
                    const float wj = w8[jj];
                    const uint4 v = v8[jj];
                    accr[0] = __fmaf_rn(wj, bf16_lo(v.x), accr[0]);
                    accr[1] = __fmaf_rn(wj, bf16_hi(v.x), accr[1]);
                    accr[2] = __fmaf_rn(wj, bf16_lo(v.y), accr[2]);
                    accr[3] = __fmaf_rn(wj, bf16_hi(v.y), accr[3]);
                    accr[4] = __fmaf_rn(wj, bf16_lo(v.z), accr[4]);
                    accr[5] = __fmaf_rn(wj, bf16_hi(v.z), accr[5]);
                    accr[6] = __fmaf_rn(wj, bf16_lo(v.w), accr[6]);
                    accr[7] = __fmaf_rn(wj, bf16_hi(v.w), accr[7]);
                }
            }
            first = false;
            uint4 o;
            o.x = f32_to_bf16_bits(accr[0]) | (f32_to_bf16_bits(accr[1]) << 16);
            o.y = f32_to_bf16_bits(accr[2]) | (f32_to_bf16_bits(accr[3]) << 16);
            o.z = f32_to_bf16_bits(accr[4]) | (f32_to_bf16_bits(accr[5]) << 16);
            o.w = f32_to_bf16_bits(accr[6]) | (f32_to_bf16_bits(accr[7]) << 16);
            *reinterpret_cast<uint4*>(p.out + static_cast<long long>(t) * p.H + col) = o;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, C::kCols);
    }
}

}  // namespace

// Upper bound on the pieces a gate/up unit of KB K-blocks is cut into when W K-blocks are dealt
// to min(G, W) CTAs in equal contiguous ranges (each range then holds at least W / min(G, W)
// K-blocks).
long long fused_max_pieces(long long W, int G, int KB) {
    if (W <= 0) return 1;
    const long long smin = W / std::min<long long>(G, W);
    return std::min<long long>(KB, (KB + smin - 1) / smin + 1);
}

// Bytes of the fused kernel's fp32 partial-sum buffer for any number of active blocks up to
// B_cap: max over nblk of pieces(nblk) * nblk * block_m rows of 2N floats.
size_t fused_partial_bytes(int B_cap, int bm, int H, int N, int G) {
    const int KB1 = H / 128, NT1 = 2 * N / 128;
    size_t best = 0;
    for (int nb = 1; nb <= B_cap; ++nb) {
        const long long W = static_cast<long long>(nb) * NT1 * KB1;
        const size_t rows = static_cast<size_t>(fused_max_pieces(W, G, KB1)) * nb * bm;
        best = std::max(best, rows * 2 * N * sizeof(float));
    }
    return best;
}

// Counter words of the fused kernel: 4 phase counters, then blk_done, blk_ready and the ready
// list per block.
int fused_counter_words(int B_cap) { return 4 + 3 * B_cap; }

namespace {
// Test hook (moe_debug_inject_stall): one-shot settings for the calling thread's next launch.
thread_local int t_stall_block = -1;
thread_local unsigned long long t_stall_limit_ns = 0;

void take_stall_injection(int* block, unsigned long long* limit_ns) {
    if (t_stall_limit_ns) {
        *block = t_stall_block;
        *limit_ns = t_stall_limit_ns;
    }
    t_stall_block = -1;
    t_stall_limit_ns = 0;
}
}  // namespace

int launch_fused_layer(const FusedLaunch& f, cudaStream_t stream) {
    const int bm = f.bm;
    const int G = sm_count();
    CUtensorMap tw1, ta1, tw2, ta2;
    const int KB1 = f.H / 128, NT1 = 2 * f.N / 128, KB2 = f.N / 128, NT2 = f.H / 128;
    const bool tiled = f.w_layout == MOE_WEIGHTS_TILED;
    const long long w1_rows = tiled ? static_cast<long long>(f.E_local) * NT1 * KB1 * 128
                                    : static_cast<long long>(f.E_local) * 2 * f.N;
    const long long w2_rows = tiled ? static_cast<long long>(f.E_local) * NT2 * KB2 * 128
                                    : static_cast<long long>(f.E_local) * f.H;
    if (w1_rows > 0x7FFFFFFFLL || w2_rows > 0x7FFFFFFFLL) { set_error("fused layer: weight tensor too large"); return MOE_ERR_ARG; }
    if (!make_tma_map_u8(&tw1, f.wgu_q, w1_rows, tiled ? 128 : f.H, 128) ||
        !make_tma_map_u8(&ta1, f.xq, f.slots, f.H, bm) ||
        !make_tma_map_u8(&tw2, f.wd_q, w2_rows, tiled ? 128 : f.N, 128) ||
        !make_tma_map_u8(&ta2, f.aq, f.slots, f.N, bm)) {
        set_error("fused layer: tensor-map encode failed");
        return MOE_ERR_LAUNCH;
    }
    FusedArgs a{};
    a.sorted_idx = f.sorted_idx; a.block_expert = f.block_expert; a.num_blocks = f.num_blocks;
    a.route_slot = f.route_slot; a.topk_ids = f.topk_ids; a.topk_w = f.topk_w;
    a.expert_map = f.expert_map; a.B_cap = f.B_cap; a.M = f.M; a.k = f.k; a.E = f.E;
    a.E_local = f.E_local; a.R = f.M * f.k; a.slots = f.slots;
    a.H = f.H; a.N = f.N; a.KB1 = KB1; a.NT1 = NT1; a.KB2 = KB2; a.NT2 = NT2;
    a.x = static_cast<const uint16_t*>(f.x); a.xsT = f.xsT; a.wgu_s = f.wgu_s; a.gu = f.gu;
    a.xq = f.xq; a.aq = f.aq; a.asT = f.asT; a.wd_s = f.wd_s;
    a.z = static_cast<uint16_t*>(f.z); a.out = static_cast<uint16_t*>(f.out);
    a.L = f.clamp_limit; a.act = f.act; a.fmt = f.fmt; a.w_tiled = tiled ? 1 : 0;
    a.sync = f.sync; a.blk_done = f.sync + 4; a.blk_ready = f.sync + 4 + f.B_cap;
    a.ready_list = f.sync + 4 + 2 * f.B_cap;
    a.status = device_status_ptr();
    a.wait_limit_ns = kWaitLimitNs;
    a.stall_block = -1;
    take_stall_injection(&a.stall_block, &a.wait_limit_ns);
    const void* fn;
    int smem;
    switch (bm) {
        case 16: fn = reinterpret_cast<const void*>(k_moe_fused<16>); smem = FCfg<16>::kSmem; break;
        case 32: fn = reinterpret_cast<const void*>(k_moe_fused<32>); smem = FCfg<32>::kSmem; break;
        case 64: fn = reinterpret_cast<const void*>(k_moe_fused<64>); smem = FCfg<64>::kSmem; break;
        default: fn = reinterpret_cast<const void*>(k_moe_fused<128>); smem = FCfg<128>::kSmem; break;
    }
    if (!ensure_smem(fn, smem)) { set_error("fused layer: shared-memory limit %d refused", smem); return MOE_ERR_LAUNCH; }
    Launch L(dim3(static_cast<unsigned>(G)), dim3(FCfg<16>::kThreads), smem, stream, true);
    cudaError_t e;
    switch (bm) {
        case 16: e = cudaLaunchKernelEx(&L.cfg, k_moe_fused<16>, tw1, ta1, tw2, ta2, a); break;
        case 32: e = cudaLaunchKernelEx(&L.cfg, k_moe_fused<32>, tw1, ta1, tw2, ta2, a); break;
        case 64: e = cudaLaunchKernelEx(&L.cfg, k_moe_fused<64>, tw1, ta1, tw2, ta2, a); break;
        default: e = cudaLaunchKernelEx(&L.cfg, k_moe_fused<128>, tw1, ta1, tw2, ta2, a); break;
    }
    if (e != cudaSuccess) { set_error("fused layer launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}

}  // namespace moe

extern "C" int moe_debug_inject_stall(int block, unsigned long long wait_limit_ns) {
    moe::clear_error();
    if (block < 0 || wait_limit_ns == 0 || wait_limit_ns > moe::kWaitLimitNs) {
        moe::set_error("moe_debug_inject_stall: need block >= 0 and 0 < wait_limit_ns <= %llu",
                       static_cast<unsigned long long>(moe::kWaitLimitNs));
        return MOE_ERR_ARG;
    }
    moe::t_stall_block = block;
    moe::t_stall_limit_ns = wait_limit_ns;
    return MOE_OK;
}
