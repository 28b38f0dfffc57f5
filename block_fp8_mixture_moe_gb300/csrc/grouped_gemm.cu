// grouped_gemm.cu -- block-FP8 grouped GEMM over the active expert blocks, on the fifth-
// generation tensor cores (tcgen05, accumulators in tensor memory) with TMA-fed operands.
//
// Method: lmdeploy PR #4956 "Perf/pytorch block fp8 moe decode", section "Active-expert block
// scheduling" (GEMM programs only for expert blocks that received tokens); lmdeploy PR #4857
// "optimize compact blocked FP8 MoE and route preparation", section "Changes" (compact blocks;
// transposed MMA for small block_m); vLLM PR #53875, "Purpose" (W8A8 block shape [128, 128]:
// one fp32 scale per 128x128 weight block and per token per 128 activation columns).
//
// Orientation (transposed / swap-AB): the MMA's M side is 128 weight rows (output features) of
// one expert and its N side is the block's block_m tokens, so a decode block with one or two
// real tokens still runs full-height MMAs and the weight tile is the A operand.  One work unit
// is (block b, 128-row output tile, K split); a persistent grid of one CTA per SM gives each CTA
// a contiguous range of units (consecutive tiles of the same block).  num_blocks is read on the
// device, so no work exists for inactive experts.
//
// Per CTA (352 threads; 224 for block_m = 128; one CTA per SM):
//   warp 6        : metadata.  Walks this CTA's units ahead of everyone else and writes, per
//                   chunk of up to CK K-blocks of a unit, a descriptor into a shared-memory
//                   ring: expert, block, tile, K range, the block's output rows, and the token
//                   and weight-block scales of those K-blocks.  All dependent global loads of
//                   the kernel happen here, off the critical path.
//   warp 0  lane 0: TMA producer.  Per 128-wide K-block it loads the 128x128 E4M3 weight tile
//                   (16 KB) and the block_m x 128 activation tile into one pipeline stage,
//                   both with 128-byte swizzle, completion counted on the stage's mbarrier.
//   warp 1  lane 0: MMA issuer.  Per K-block: 4 tcgen05.mma (K = 32 each) into a fresh fp32
//                   accumulator buffer in tensor memory, then tcgen05.commit frees the smem
//                   stage and signals the accumulator buffer.
//   warps 2-5, 7-10: epilogue / scale promotion, two warpgroups that take alternate units.
//                   Each thread owns one weight row; per K-block it reads its block_m partial
//                   sums (tcgen05.ld, two buffers per wait when block_m = 16), frees the
//                   buffer, and accumulates partial * a_s[token, kb] * w_s[expert, tile, kb] in
//                   fp32 registers with the scales read from the descriptor; at the end of the
//                   unit it writes BF16 or fp32 (split-K partials) outputs to the rows the
//                   descriptor lists.  A unit of the down projection (K = 256) is a single
//                   pipeline stage, so one warpgroup's promotion and stores per unit would take
//                   longer than the unit's weight tile takes to stream; with two warpgroups the
//                   epilogue keeps up with HBM.
// Block scales differ per K-block, so every K-block gets its own accumulator buffer; 4-8
// buffers let the MMA run ahead of the promotion.  Every wait is bounded (see mbar_wait).
#include "common.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

namespace moe {
namespace {

struct GemmArgs {
    const float* a_s;
    int a_rows, K, KB;
    const float* w_s;
    int E_local, N_out, NT;
    const int32_t* sorted_idx;
    const int32_t* block_expert;
    const int32_t* num_blocks;
    int B_cap;
    void* out;
    int out_f32, out_rows, splits, scatter;
    int w_tiled;
    int* status;
    int wait_first;  // wait for the previous launch before anything (its predecessor is not done)
    int pdl;         // launched with programmatic dependent launch (else nothing to wait for)
    // Self-routing (GATE_UP, at most 32 routes, block_m <= 32): the metadata warp derives the
    // block table from the caller's top-k ids itself -- the same stable counting sort as route
    // preparation's one-warp path, so the blocks, slots and rows are identical -- instead of
    // reading route preparation's outputs.  The ids are an input of the layer, not an output of
    // an earlier kernel, so the weight stream starts before routing and input quantisation are
    // done; only the activation tiles and token scales wait for them.
    const int32_t* self_ids;  // [self_R] global expert ids, or null
    const int32_t* self_map;  // nullable [self_E]
    int self_R, self_E;
    // Epilogue reduce (DOWN, block_m <= 32; red_out == nullptr: none): the weighted top-k sum
    // out[t] = bf16(sum_j w[t,j] z[t*k+j]) over the kept routes in top-k order.  After a unit's
    // z rows are stored, each row counts itself in its (token, 128-column tile) counter; the
    // arrival that completes a token's kept routes sums that token's 128 columns, so the order
    // of the fp32 fused multiply-adds is the same whichever CTA does it.  Tokens with no kept
    // route get zero rows.
    uint16_t* red_out;        // [red_M, N_out] bf16
    unsigned* red_cnt;        // [red_M, NT] arrivals, zero at launch
    const float* red_w;       // [red_M, red_k] routing weights
    const int32_t* red_slot;  // [red_M * red_k] route_slot: >= 0 for a kept route
    int red_k, red_M;
    // Dynamic tail (sched == nullptr: none).  The CTAs first walk equal static shares of three
    // quarters of the units, then take the rest sched_chunk units at a time from this counter
    // (zero at launch), so the SMs that stream faster or start later even out at the end.
    unsigned long long* sched;
    int sched_chunk;
};

// Weight bytes of one chunk of the dynamic tail.  Measured on the Zipf prefill layer: 32 and
// 64 KB 760-765 us, 128 KB 741 us, 256 KB 745 us, 512 KB 750 us (its down GEMM's 96 KB units
// then go two to a chunk and a descriptor).
// Measured on GB300 at the Zipf prefill shape (the down GEMM's 96 KB units; the gate/up GEMM's
// 512 KB units always go one to a chunk): chunks of 1 / 2 / 3 / 4 / 5 units gave 757 / 712.9 /
// 713.8 / 710.9 / 720.6 us for the layer, the best at 4 units, which divide its 32-tile blocks.
constexpr long long kSchedChunkBytes = 384 * 1024;
// descriptors of a CTA's queue still unconsumed when it takes its next dynamic chunk: at most
// kDynLookahead(BM) - 1.  Measured at the prefill shape (block_m 32): 2 / 3 / 4 gave 702.5 /
// 701.8 / 701.7 us against 703.6 us when chunks were taken as soon as the ring had room; at
// decode (block_m 16) 2 against 3: M=32 -0.3 us, M=64 -0.5, M=256 -0.6.
__host__ __device__ constexpr int kDynLookahead(int bm) { return bm <= 16 ? 2 : 3; }

template <int BM>
struct Cfg {
    static constexpr int kWBytes = 128 * 128;          // one 128x128 E4M3 weight tile
    static constexpr int kABytes = BM * 128;           // one block_m x 128 activation tile
    static constexpr int kKps = 2;                     // K-blocks per pipeline stage
    static constexpr int kStage = kKps * (kWBytes + kABytes);  // multiple of 1024
    static constexpr int kStages = BM <= 32 ? 5 : BM <= 64 ? 4 : 3;
    // two epilogue warpgroups.  block_m <= 32: they take alternate units, each with its own
    // ring of tensor-memory slots.  block_m >= 64 (column split): both take every unit, each the
    // promotion of half of its block_m token columns, on one shared ring
    static constexpr int kEpiGroups = 2;
    static constexpr int kEpiThreads = 128 * kEpiGroups;
    static constexpr int kThreads = 96 + kEpiThreads;
    static constexpr bool kColSplit = BM >= 64;
    static constexpr int kCpw = kColSplit ? BM / 2 : BM;  // accumulator columns per thread
    static constexpr int kRings = kColSplit ? 1 : 2;
    // tensor-memory slots of kKps accumulators: kTSlotsG per ring.  block_m 16 takes 8, all 512
    // columns: a unit's MMAs then run up to 8 stages ahead of its promotion instead of 4.
    // Measured on GB300 (graph-replayed layer, interleaved A/B): decode M=4 -0.5 us, M=32 -0.4,
    // M=64 -1.0, M=256 -2.2, the rest unchanged.
    static constexpr int kTSlotsG = BM <= 16 ? 8 : BM <= 64 ? 4 : 2;
    static constexpr int kTSlots = kRings * kTSlotsG;
    static constexpr int kTemptyArrivals = kColSplit ? 256 : 128;
    static constexpr int kSlotCols = kKps * BM;
    static constexpr int kCols = kTSlots * kSlotCols <= 32 ? 32 : kTSlots * kSlotCols <= 64 ? 64
                               : kTSlots * kSlotCols <= 128 ? 128 : kTSlots * kSlotCols <= 256 ? 256 : 512;
    // descriptor ring
    static constexpr int kCK = 512 / BM < 2 ? 2 : 512 / BM;  // K-blocks per descriptor
    static constexpr int kSwMax = 64;                  // weight-block scales per descriptor
    static constexpr int kRing = 8;                    // descriptors in flight
    // descriptors published before the previous kernel is done, their token scales deferred:
    // enough to fill every stage with weight tiles, one ring slot kept for the end marker
    static constexpr int kDefer = kStages < kRing - 1 ? kStages : kRing - 1;
    static constexpr int kDescHdr = 8;                 // ints: e, b, nt0, ntl, sp, kb0, nck, flags
    static constexpr int kDescInts = kDescHdr + 2 * BM + kCK * BM + kSwMax;  // hdr, rows, kept, sa, sw
    static constexpr int kDescBytes = ((kDescInts * 4) + 15) / 16 * 16;
    static constexpr int kBarBytes = 1024;
    static constexpr int kSmem = kStages * kStage + kRing * kDescBytes + kBarBytes + 1024;
    static_assert(kStage % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(kTSlots * kSlotCols <= 512, "tensor memory holds 512 fp32 columns");
    static_assert(kCK % kKps == 0, "descriptors hold whole stages");
    static_assert(kCK * BM == 512, "token-scale area of a descriptor is 512 values");
    static_assert(((kDescHdr + 2 * BM) * 4) % 16 == 0, "token scales stay 16-byte aligned");
    static_assert(kSmem <= 232448, "shared memory per CTA");
};

// descriptor flags: the descriptor starts / ends each of its tiles' K range
constexpr int kFirst = 1, kLast = 2, kEnd = 4;

// One descriptor: ntl consecutive output tiles nt0.. of block b (expert e), split sp, over the
// K-blocks [kb0, kb0 + nck).  rows[j]: output row of slot j (-1: pad or dropped);
// sa[kk * BM + j]: token scale of slot j at K-block kb0 + kk; sw[t * nck + kk]: weight-block
// scale of tile nt0 + t at K-block kb0 + kk.  A descriptor with ntl > 1 covers each tile's
// whole K range (kFirst | kLast).  The header is released first (dfull), for the producer and
// the MMA issuer; the rows and scales follow (dsa), for the epilogue.
struct Desc {
    int* hdr;
    int* rows;
    int* kept;  // epilogue reduce: kept routes of the token of row j
    float* sa;
    float* sw;
};

template <int BM>
__device__ __forceinline__ Desc desc_at(uint8_t* ring, int slot) {
    using C = Cfg<BM>;
    int* base = reinterpret_cast<int*>(ring + slot * C::kDescBytes);
    Desc d;
    d.hdr = base;
    d.rows = base + C::kDescHdr;
    d.kept = d.rows + BM;
    d.sa = reinterpret_cast<float*>(d.kept + BM);
    d.sw = d.sa + C::kCK * BM;
    return d;
}

// DYN: the dynamic tail (p.sched) is compiled in.  A separate instantiation, because the code
// alone, never taken, made the small decode layers ~2 us slower (M=1: 35.3 vs 33.3 us).
template <int BM, bool DYN>
__global__ void __launch_bounds__(Cfg<BM>::kThreads, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_a, GemmArgs p) {
    using C = Cfg<BM>;
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
    uint64_t* dsa = dempty + C::kRing;  // the descriptor's token scales are written
    uint64_t* mma_done = dsa + C::kRing;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // set by an epilogue thread once its wait for the previous launch has returned
    volatile int* dep_seen = reinterpret_cast<volatile int*>(tmem_slot + 2);

    // epilogue reduce: per warpgroup, the tokens whose last unit the warpgroup just finished
    // (double-buffered by unit parity) and two barriers of its 128 threads
    __shared__ int red_list[2][2][32];
    __shared__ int red_n[2][2];
    __shared__ __align__(8) uint64_t rbar[4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        red_n[0][0] = red_n[0][1] = red_n[1][0] = red_n[1][1] = 0;
        for (int i = 0; i < 4; ++i) mbar_init(rbar + i, 128);
        for (int i = 0; i < C::kStages; ++i) { mbar_init(full + i, 1); mbar_init(empty + i, 1); }
        for (int i = 0; i < C::kTSlots; ++i) { mbar_init(tfull + i, 1); mbar_init(tempty + i, C::kTemptyArrivals); }
        for (int i = 0; i < C::kRing; ++i) {
            mbar_init(dfull + i, 32);
            mbar_init(dempty + i, C::kEpiThreads + 2);
            mbar_init(dsa + i, 32);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        *dep_seen = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_a);
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

    // With programmatic dependent launch the previous kernel may still be running here.  The
    // routing metadata (route preparation, complete before that kernel began) and the weights
    // do not depend on it, so the metadata warp publishes the descriptor headers and the
    // producer streams the first stages' weight tiles at once; only the activation tiles and
    // token scales, which that kernel writes, wait for it (grid_dep_wait).  With wait_first the
    // previous kernel released this one before the routing it reads was complete: everything
    // waits for it, and the next launch is released only after that wait, so that it may read
    // the routing early too.
    if (p.wait_first) grid_dep_wait();
    // The next launch (the activation kernel) reads route preparation's outputs before it waits.
    // A self-routing launch may begin before route preparation is complete, so it releases the
    // next launch only after a thread of the CTA has waited for its own predecessor (whose
    // completion implies route preparation's); the first release of a CTA counts.
    const bool self_route = p.self_ids != nullptr;
    if (!self_route) grid_dep_launch();

    if (warp == 6) {
        // ---------------- metadata warp ----------------
        // Units are ordered (block, split, tile) with the tile fastest, and this CTA owns the
        // contiguous range [u_lo, u_hi).  The range is walked incrementally: a run of tiles of
        // the same block and split shares its rows and token scales, so one descriptor covers
        // up to kSwMax / (K-blocks per unit) tiles; a unit longer than kCK K-blocks is cut into
        // one descriptor per kCK K-blocks.  All loads of a descriptor are issued before any of
        // its shared-memory stores.
        int nblk = self_route ? 0 : __ldcg(p.num_blocks);
        nblk = max(0, min(nblk, p.B_cap));
        int nt = 0, sp = 0, b = 0;
        long long left = 0;
        // unit u's position: tile fastest, then split, then block
        auto seek = [&](long long u) {
            nt = static_cast<int>(u % p.NT);
            sp = static_cast<int>((u / p.NT) % p.splits);
            b = static_cast<int>(u / (static_cast<long long>(p.NT) * p.splits));
        };
        int slot = 0;
        uint32_t ph = 0;
        bool ok = true;
        bool dep_done = p.wait_first || !p.pdl;
        // Before the previous kernel is done, up to kDefer descriptors are published without
        // their token scales (ring slots pend0 .. pend0 + npend - 1), so that the producer can
        // stream those descriptors' weight tiles meanwhile; the scales follow after the wait.
        int npend = 0, pend0 = 0;
        auto fill_sa = [&](int sl, int bb, int cc0, int nn) {
            const Desc dd = desc_at<BM>(ring, sl);
            // token scales (written by the previous kernel): lane order (slot j, K-block kk)
            // with kk fastest, so the loads of one slot row are contiguous
            float sa_v[C::kCK * BM / 32];
            const int n_sa = nn * BM;
#pragma unroll
            for (int q = 0; q < C::kCK * BM / 32; ++q) {
                const int i = q * 32 + lane;
                const int j = i / nn, kk = i - j * nn;
                sa_v[q] = i < n_sa ? __ldcg(p.a_s + static_cast<long long>(bb * BM + j) * p.KB + cc0 + kk) : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < C::kCK * BM / 32; ++q) {
                const int i = q * 32 + lane;
                const int j = i / nn, kk = i - j * nn;
                if (i < n_sa) dd.sa[kk * BM + j] = sa_v[q];
            }
            mbar_arrive(dsa + sl);  // rows, weight and token scales: the epilogue goes ahead
        };
        auto flush_pending = [&]() {
            __syncwarp();  // lane 0's header stores are read by every lane
            grid_dep_wait();
            if (self_route) grid_dep_launch();
            dep_done = true;
            for (int i = 0; i < npend; ++i) {
                const int sl = pend0 + i < C::kRing ? pend0 + i : pend0 + i - C::kRing;
                const int* hdr = desc_at<BM>(ring, sl).hdr;
                fill_sa(sl, hdr[1], hdr[5], hdr[6]);
            }
            npend = 0;
        };
        int cur_b = -1, e = -1;
        int rows[(BM + 31) / 32], kept[(BM + 31) / 32];
#pragma unroll
        for (int t = 0; t < (BM + 31) / 32; ++t) { rows[t] = -1; kept[t] = 0; }
        // self-routing: lane r holds route r; match-any groups the routes of one expert, so a
        // route's rank in its expert is the number of same-expert lanes below it, and an
        // expert's padded offset is the sum of the padded counts of the active experts below it
        int sr_e = -1, sr_off = 0, sr_pad = 0, sr_cnt = 0;
        bool sr_lead = false;
        if constexpr (BM <= 32) {
            if (self_route) {
                int er = -1;
                if (lane < p.self_R) {
                    const int id = __ldg(p.self_ids + lane);
                    if (id >= 0 && id < p.self_E) {
                        const int le = p.self_map ? __ldg(p.self_map + id) : id;
                        er = (le >= 0 && le < p.E_local) ? le : -1;
                    }
                }
                const unsigned m = __match_any_sync(0xFFFFFFFFu, er);
                unsigned lt;
                asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
                sr_lead = er >= 0 && (m & lt) == 0;
                sr_e = er;
                sr_cnt = __popc(m);
                sr_pad = sr_lead ? (sr_cnt + BM - 1) / BM * BM : 0;
                int total = 0;
                for (int j = 0; j < 32; ++j) {
                    const int ej = __shfl_sync(0xFFFFFFFFu, er, j);
                    const int pj = __shfl_sync(0xFFFFFFFFu, sr_pad, j);
                    total += pj;
                    sr_off += ej < er ? pj : 0;  // pj > 0 only for an active expert's leader
                }
                nblk = min(total / BM, p.B_cap);
            }
        }
        // this CTA's static range: an equal share of the units, or, with the dynamic tail, an
        // equal share of at most three quarters of them in whole blocks; the rest
        // [dyn_base, units) is handed out.  Whole blocks start every CTA's range at tile 0 of a
        // block, so at any moment the CTAs stream the same tile index of their blocks, and the
        // blocks of a hot expert share each weight tile through L2 instead of re-reading it.
        // Measured on GB300 at the Zipf prefill shape (ncu DRAM bytes, one launch each):
        // gate/up 3.01 -> 2.84 GB, down 1.49 -> 1.39 GB; the layer 726 -> 711 us.
        const long long units = static_cast<long long>(nblk) * p.NT * p.splits;
        long long dyn_base = units;
        if (DYN) {
            long long share = units * 3 / (4LL * gridDim.x);
            const long long per_block = static_cast<long long>(p.NT) * p.splits;
            if (share >= per_block) share -= share % per_block;
            dyn_base = share * gridDim.x;
            seek(share * blockIdx.x);
            left = share;
        } else {
            const long long lo = units * blockIdx.x / gridDim.x;
            seek(lo);
            left = units * (blockIdx.x + 1) / gridDim.x - lo;
        }
        long long npub = 0;  // descriptors published
        for (;;) {
            while (left > 0 && ok) {
                if (self_route && b != cur_b) {
                    if constexpr (BM <= 32) {
                        // block b belongs to the active expert whose padded run holds slot b*BM
                        const unsigned own = __ballot_sync(0xFFFFFFFFu, sr_lead && sr_off <= b * BM &&
                                                                            b * BM < sr_off + sr_pad);
                        const int src = own ? __ffs(own) - 1 : 0;
                        const int e_b = __shfl_sync(0xFFFFFFFFu, sr_e, src);
                        const int off_b = __shfl_sync(0xFFFFFFFFu, sr_off, src);
                        const int cnt_b = __shfl_sync(0xFFFFFFFFu, sr_cnt, src);
                        e = own ? e_b : -1;
                        int row = (lane < BM && e >= 0 && b * BM + lane - off_b < cnt_b) ? b * BM + lane : -1;
                        if (row >= p.out_rows) {
                            if (p.status) atomicOr(p.status, MOE_DEV_BAD_INDEX);
                            row = -1;
                        }
                        rows[0] = row;
                    }
                    cur_b = b;
                } else if (b != cur_b) {
                    // the block's expert and its slot rows, loaded together
                    const int e_raw = __ldcg(p.block_expert + b);
                    int rr[(BM + 31) / 32];
    #pragma unroll
                    for (int t = 0; t < (BM + 31) / 32; ++t) {
                        const int j = t * 32 + lane;
                        rr[t] = j < BM ? __ldcg(p.sorted_idx + b * BM + j) : -1;
                    }
                    e = (e_raw >= 0 && e_raw < p.E_local) ? e_raw : -1;
                    if (e >= 0) {
    #pragma unroll
                        for (int t = 0; t < (BM + 31) / 32; ++t) {
                            const int slot_j = b * BM + t * 32 + lane;
                            int row = rr[t] < 0 ? -1 : (p.scatter ? rr[t] : slot_j);
                            if (row >= p.out_rows) {
                                if (p.status) atomicOr(p.status, MOE_DEV_BAD_INDEX);
                                row = -1;
                            }
                            rows[t] = row;
                        }
                        if (p.red_out) {
                            // epilogue reduce: the number of kept routes of each row's token
    #pragma unroll
                            for (int t = 0; t < (BM + 31) / 32; ++t) {
                                int cnt = 0;
                                if (rows[t] >= 0) {
                                    const long long rb = static_cast<long long>(rows[t] / p.red_k) * p.red_k;
                                    for (int j0 = 0; j0 < p.red_k; j0 += 8) {
                                        int sl[8];
    #pragma unroll
                                        for (int jj = 0; jj < 8; ++jj)
                                            sl[jj] = j0 + jj < p.red_k ? __ldcg(p.red_slot + rb + j0 + jj) : -1;
    #pragma unroll
                                        for (int jj = 0; jj < 8; ++jj) cnt += sl[jj] >= 0 ? 1 : 0;
                                    }
                                }
                                kept[t] = cnt;
                            }
                        }
                    }
                    cur_b = b;
                }
                const int run = static_cast<int>(min(static_cast<long long>(p.NT - nt), left));
                int adv = run;
                if (e >= 0) {
                    const int kb0 = sp * p.KB / p.splits, kb1 = (sp + 1) * p.KB / p.splits;
                    const int len = kb1 - kb0;
                    const bool whole = len <= C::kCK;
                    const int ntl = whole ? min(run, C::kSwMax / len) : 1;
                    adv = ntl;
                    for (int c0 = kb0; c0 < kb1 && ok; c0 += C::kCK) {
                        const int nck = min(C::kCK, kb1 - c0);
                        float sw_v[C::kSwMax / 32];
                        const int n_sw = ntl * nck;
    #pragma unroll
                        for (int q = 0; q < C::kSwMax / 32; ++q) {
                            const int i = q * 32 + lane;
                            const int t = i / nck, kk = i - t * nck;
                            sw_v[q] = i < n_sw ? __ldg(p.w_s + (static_cast<long long>(e) * p.NT + nt + t) * p.KB + c0 + kk) : 0.0f;
                        }
                        ok = mbar_wait_fast(dempty + slot, ph ^ 1u, abort_flag, p.status);
                        if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                        Desc d = desc_at<BM>(ring, slot);
                        if (lane == 0) {
                            d.hdr[0] = e; d.hdr[1] = b; d.hdr[2] = nt; d.hdr[3] = ntl; d.hdr[4] = sp;
                            d.hdr[5] = c0; d.hdr[6] = nck;
                            d.hdr[7] = (c0 == kb0 ? kFirst : 0) | (c0 + nck == kb1 ? kLast : 0);
                        }
                        mbar_arrive(dfull + slot);  // the header: the producer and the MMA go ahead
    #pragma unroll
                        for (int t = 0; t < (BM + 31) / 32; ++t)
                            if (t * 32 + lane < BM) { d.rows[t * 32 + lane] = rows[t]; d.kept[t * 32 + lane] = kept[t]; }
    #pragma unroll
                        for (int q = 0; q < C::kSwMax / 32; ++q) {
                            const int i = q * 32 + lane;
                            if (i < n_sw) d.sw[i] = sw_v[q];
                        }
                        if (dep_done) {
                            fill_sa(slot, b, c0, nck);
                        } else {
                            if (npend == 0) pend0 = slot;
                            ++npend;
                        }
                        if (++slot == C::kRing) { slot = 0; ph ^= 1u; }
                        ++npub;
                        if (npend == C::kDefer) flush_pending();
                    }
                }
                // advance by adv units (never past the end of this block and split's tile run)
                nt += adv;
                left -= adv;
                if (nt == p.NT) {
                    nt = 0;
                    if (++sp == p.splits) { sp = 0; ++b; }
                }
            }
            if constexpr (!DYN) break;
            else {
                if (!ok) break;
                // Dynamic tail.  Route preparation zeroes the counter: a launch that has not yet waited
                // for its predecessor (self-routing) does so first.  Each chunk's successor is taken
                // when the chunk starts, so the atomic's round trip overlaps the chunk's descriptors.
                if (!dep_done) flush_pending();
                // A chunk is taken only once the descriptor kDynLookahead(BM) back has been consumed,
                // so that chunks go out near the end of each CTA's queued work.  Taken as soon as
                // the ring had room, every chunk went out within the first ~35 us at decode M=32
                // (the ring holds 8 descriptors, a CTA ~9 units) and nothing was balanced.
                constexpr int kLa = kDynLookahead(BM);
                if (npub >= kLa) {
                    const int j = slot >= kLa ? slot - kLa : slot - kLa + C::kRing;
                    const uint32_t pj = slot >= kLa ? ph : ph ^ 1u;
                    ok = mbar_wait_fast(dempty + j, pj, abort_flag, p.status);
                    if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                }
                unsigned long long v = 0;
                if (lane == 0) v = atomicAdd(p.sched, static_cast<unsigned long long>(p.sched_chunk));
                const long long c = dyn_base + static_cast<long long>(__shfl_sync(0xFFFFFFFFu, v, 0));
                if (c >= units) break;
                seek(c);
                left = min(static_cast<long long>(p.sched_chunk), units - c);
            }
        }
        if (ok) {
            // end marker (before the deferred token scales, so that the producer stops
            // waiting for descriptors and issues its deferred activation tiles)
            ok = mbar_wait_fast(dempty + slot, ph ^ 1u, abort_flag, p.status);
            if (__all_sync(0xFFFFFFFFu, ok)) {
                if (lane == 0) desc_at<BM>(ring, slot).hdr[7] = kEnd;
                mbar_arrive(dfull + slot);
                mbar_arrive(dsa + slot);
            }
            if (npend > 0) flush_pending();
        }
        if (p.red_out && ok) {
            // epilogue reduce: a token with no kept route gets a zero row (no unit sums it)
            for (int tok = blockIdx.x; tok < p.red_M; tok += gridDim.x) {
                const int sl = lane < p.red_k ? __ldcg(p.red_slot + static_cast<long long>(tok) * p.red_k + lane) : -1;
                if (__any_sync(0xFFFFFFFFu, sl >= 0)) continue;
                uint4* o = reinterpret_cast<uint4*>(p.red_out + static_cast<long long>(tok) * p.N_out);
                for (int c = lane; c < p.N_out / 8; c += 32) o[c] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    } else if (warp == 0) {
        // ---------------- TMA producer ----------------
        // Until the previous kernel is done (grid_dep_wait) only the weight tiles are loaded; a
        // stage's activation tiles are recorded and issued right after the wait, which happens
        // when every stage holds weights, or at the end marker.  Each stage expects its full
        // byte count from the start, so its barrier completes only when both halves have
        // landed.
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_a = l2_policy_evict_last();
            int s = 0, slot = 0;
            uint32_t ph = 0, dph = 0;
            long long issued = 0;
            bool ok = true;
            bool dep_done = p.wait_first || !p.pdl;
            int npend = 0;
            int pend_s[C::kStages], pend_kb[C::kStages], pend_nk[C::kStages], pend_b[C::kStages];
            auto load_a = [&](int st_i, int kb, int nk, int b) {
                uint8_t* st = smem + st_i * C::kStage;
                for (int j = 0; j < nk; ++j)
                    tma_load_2d(st + C::kKps * C::kWBytes + j * C::kABytes, &tmap_a, full + st_i,
                                (kb + j) * 128, b * BM, pol_a);
            };
            auto resolve = [&]() {
                grid_dep_wait();
                if (self_route) grid_dep_launch();
                dep_done = true;
                for (int i = 0; i < npend; ++i) load_a(pend_s[i], pend_kb[i], pend_nk[i], pend_b[i]);
                npend = 0;
            };
            while (ok) {
                if (!mbar_wait_fast(dfull + slot, dph, abort_flag, p.status)) break;
                const Desc d = desc_at<BM>(ring, slot);
                const int flags = d.hdr[7];
                if (flags & kEnd) break;
                const int e = d.hdr[0], b = d.hdr[1], nt0 = d.hdr[2], ntl = d.hdr[3];
                const int c0 = d.hdr[5], nck = d.hdr[6];
                mbar_arrive(dempty + slot);
                if (++slot == C::kRing) { slot = 0; dph ^= 1u; }
                for (int t = 0; t < ntl && ok; ++t) {
                    // row-major weights: box (kb*128, e*N_out + nt*128); tiled weights: every
                    // 128x128 tile is one contiguous 16 KB run at row ((e*NT + nt)*KB + kb)*128
                    const int nt = nt0 + t;
                    const long long wrow = p.w_tiled ? (static_cast<long long>(e) * p.NT + nt) * p.KB * 128
                                                     : static_cast<long long>(e) * p.N_out + nt * 128;
                    for (int kb = c0; kb < c0 + nck; kb += C::kKps) {
                        const int nk = min(C::kKps, c0 + nck - kb);
                        if (!mbar_wait_fast(empty + s, ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
                        uint8_t* st = smem + s * C::kStage;
                        mbar_arrive_expect_tx(full + s, static_cast<uint32_t>(nk * (C::kWBytes + C::kABytes)));
                        for (int j = 0; j < nk; ++j) {
                            if (p.w_tiled)
                                tma_load_2d(st + j * C::kWBytes, &tmap_w, full + s, 0,
                                            static_cast<int>(wrow + (kb + j) * 128), pol_w);
                            else
                                tma_load_2d(st + j * C::kWBytes, &tmap_w, full + s, (kb + j) * 128,
                                            static_cast<int>(wrow), pol_w);
                        }
                        if (dep_done) {
                            load_a(s, kb, nk, b);
                        } else {
                            pend_s[npend] = s; pend_kb[npend] = kb; pend_nk[npend] = nk; pend_b[npend] = b;
                            // the wait blocks this thread, so it waits only when every stage
                            // holds weights -- or as soon as the previous launch is known to be
                            // done (an epilogue thread has passed its own wait), so that the
                            // pending activation tiles go out at once instead of queueing behind
                            // the weight tiles of every remaining stage
                            if (++npend == C::kStages || *dep_seen) resolve();
                        }
                        ++issued;
                        if (++s == C::kStages) { s = 0; ph ^= 1u; }
                    }
                }
            }
            if (!dep_done) resolve();  // no stage may stay without its activation tiles
            if (*abort_flag) {
                // never leave a TMA write in flight: wait for the last load of every stage
                for (int i = 0; i < C::kStages; ++i) {
                    if (issued <= i) break;
                    const long long n_i = (issued - 1 - i) / C::kStages + 1;
                    volatile int no_abort = 0;
                    mbar_wait(full + i, static_cast<uint32_t>((n_i - 1) & 1), &no_abort, p.status);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f8_f32(128, BM);
            int s = 0, slot = 0;
            uint32_t ph = 0, dph = 0;
            // one slot ring per epilogue warpgroup; units alternate between the groups
            int ts0 = 0, ts1 = 0, unit = 0, owner = 0;
            uint32_t tph0 = 0, tph1 = 0;
            bool ok = true;
            while (ok) {
                if (!mbar_wait_fast(dfull + slot, dph, abort_flag, p.status)) break;
                const Desc d = desc_at<BM>(ring, slot);
                const int flags = d.hdr[7];
                if (flags & kEnd) break;
                const int ntl = d.hdr[3], nck = d.hdr[6];
                mbar_arrive(dempty + slot);
                if (++slot == C::kRing) { slot = 0; dph ^= 1u; }
                for (int t = 0; t < ntl && ok; ++t) {
                    if (flags & kFirst) owner = C::kRings == 1 ? 0 : ((unit++) & 1);
                    for (int kk = 0; kk < nck; kk += C::kKps) {
                        const int nk = min(C::kKps, nck - kk);
                        const int ts = owner * C::kTSlotsG + (owner ? ts1 : ts0);
                        const uint32_t tph = owner ? tph1 : tph0;
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
                        if (owner) { if (++ts1 == C::kTSlotsG) { ts1 = 0; tph1 ^= 1u; } }
                        else { if (++ts0 == C::kTSlotsG) { ts0 = 0; tph0 ^= 1u; } }
                    }
                }
            }
            // all issued MMAs complete before tensor memory is released
            mma_commit(mma_done);
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort, p.status);
        }
    } else {
        // ---------------- epilogue (warps 2..5 and 7..10) ----------------
        // warp & 3 selects the 32-lane quarter of tensor memory this warp may read.  Both
        // warpgroups walk every descriptor; units (a unit starts at a kFirst tile) alternate
        // between them, and each group reads only its own ring of tensor-memory slots.
        const int q = warp & 3;
        const int wg = warp >= 7 ? 1 : 0;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        const int r_in_tile = q * 32 + lane;
        int ts = 0, slot = 0;
        uint32_t tph = 0, dph = 0;
        const int ts_base = C::kColSplit ? 0 : wg * C::kTSlotsG;
        const int c0 = C::kColSplit ? wg * C::kCpw : 0;  // this thread's first token column
        int unit = 0;
        bool mine = false;
        uint32_t red_par = 0;  // epilogue reduce: phase of this warpgroup's rbar pair
        float acc[C::kCpw];
#pragma unroll
        for (int j = 0; j < C::kCpw; ++j) acc[j] = 0.0f;
        grid_dep_wait();  // (returns at once: the activations it consumes come after it)
        if (warp == 2 && lane == 0) *dep_seen = 1;
        if (self_route) grid_dep_launch();
        for (;;) {
            bool ok = mbar_wait_fast(dsa + slot, dph, abort_flag, p.status);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            const Desc d = desc_at<BM>(ring, slot);
            const int flags = d.hdr[7];
            if (flags & kEnd) break;
            const int nt0 = d.hdr[2], ntl = d.hdr[3], nck = d.hdr[6];
            const int sp = d.hdr[4];
            for (int t = 0; t < ntl; ++t) {
                if (flags & kFirst) mine = C::kColSplit || ((unit++) & 1) == wg;
                if (!mine) continue;
                if (flags & kFirst) {
#pragma unroll
                    for (int j = 0; j < C::kCpw; ++j) acc[j] = 0.0f;
                }
                const float* swt = d.sw + t * nck;
                for (int kk = 0; kk < nck; kk += C::kKps) {
                    const int nk = min(C::kKps, nck - kk);
                    ok = mbar_wait_fast(tfull + ts_base + ts, tph, abort_flag, p.status);
                    if (!__all_sync(0xFFFFFFFFu, ok)) goto epi_done;
                    tc_fence_after();
                    const uint32_t t0 = lane_base + static_cast<uint32_t>((ts_base + ts) * C::kSlotCols);
                    if (BM == 16) {
                        // both K-blocks of the stage: 32 adjacent columns, one load and one wait
                        float v[32];
                        tmem_ld32(t0, v);
                        tc_fence_before();
                        mbar_arrive_relaxed(tempty + ts_base + ts);
#pragma unroll
                        for (int j2 = 0; j2 < 2; ++j2) {
                            if (j2 < nk) {
                                const float sw = swt[kk + j2];
                                const float4* sa = reinterpret_cast<const float4*>(d.sa + (kk + j2) * BM);
#pragma unroll
                                for (int j4 = 0; j4 < BM / 4; ++j4) {
                                    const float4 a4 = sa[j4];
                                    const float sv[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        const int j = j4 * 4 + i;
                                        acc[j] = __fmaf_rn(v[j2 * 16 + j], __fmul_rn(sv[i], sw), acc[j]);
                                    }
                                }
                            }
                        }
                    } else {
                        for (int j2 = 0; j2 < nk; ++j2) {
                            const float sw = swt[kk + j2];
                            const float* sa = d.sa + (kk + j2) * BM + c0;
#pragma unroll
                            for (int c = 0; c < C::kCpw / 32; ++c) {
                                float v[32];
                                tmem_ld32(t0 + static_cast<uint32_t>(j2 * BM + c0 + c * 32), v);
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    acc[c * 32 + i] = __fmaf_rn(v[i], __fmul_rn(sa[c * 32 + i], sw), acc[c * 32 + i]);
                            }
                        }
                        tc_fence_before();
                        mbar_arrive_relaxed(tempty + ts_base + ts);
                    }
                    if (++ts == C::kTSlotsG) { ts = 0; tph ^= 1u; }
                }
                if (flags & kLast) {
                    const int n = (nt0 + t) * 128 + r_in_tile;
                    // row indices are read into registers 16 at a time before the stores, so no
                    // shared-memory load is ordered between global stores through generic pointers
#pragma unroll
                    for (int j0 = 0; j0 < C::kCpw; j0 += 16) {
                        int rws[16];
#pragma unroll
                        for (int j4 = 0; j4 < 4; ++j4) {
                            const int4 r4 = reinterpret_cast<const int4*>(d.rows + c0 + j0)[j4];
                            rws[j4 * 4 + 0] = r4.x; rws[j4 * 4 + 1] = r4.y;
                            rws[j4 * 4 + 2] = r4.z; rws[j4 * 4 + 3] = r4.w;
                        }
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int row = rws[jj];
                            if (row < 0) continue;
                            const int j = j0 + jj;
                            if (p.out_f32) {
                                float* o = static_cast<float*>(p.out);
                                o[(static_cast<long long>(sp) * p.out_rows + row) * p.N_out + n] = acc[j];
                            } else {
                                uint16_t* o = static_cast<uint16_t*>(p.out);
                                o[static_cast<long long>(row) * p.N_out + n] =
                                    static_cast<uint16_t>(f32_to_bf16_bits(acc[j]));
                            }
                        }
                    }
                    if constexpr (!C::kColSplit) {
                        if (p.red_out) {
                            // Epilogue reduce.  All 128 threads arrive on rbar[0] after their z
                            // stores of the unit; row j's thread then publishes them (fence, count)
                            // and, if its arrival completes the token, lists the token; after
                            // rbar[1] the warpgroup sums the listed tokens' columns.  The list is
                            // double-buffered by unit parity; thread 0 clears the other buffer once
                            // every thread has arrived for this unit (so it has finished the last
                            // one).  Every wait is bounded.
                            const int buf = red_par & 1;
                            mbar_arrive(rbar + wg * 2 + 0);
                            bool okr = true;
                            if (r_in_tile < BM) {
                                okr = mbar_wait_fast(rbar + wg * 2 + 0, red_par, abort_flag, p.status);
                                if (okr) {
                                    if (r_in_tile == 0) red_n[wg][buf ^ 1] = 0;
                                    const int row = d.rows[r_in_tile];
                                    if (row >= 0) {
                                        const int tok = row / p.red_k;
                                        __threadfence();
                                        const unsigned old = atomicAdd(p.red_cnt + static_cast<long long>(tok) * p.NT + nt0 + t, 1u);
                                        if (old + 1u == static_cast<unsigned>(d.kept[r_in_tile])) {
                                            __threadfence();  // the token's other rows, stored by other units
                                            red_list[wg][buf][atomicAdd(&red_n[wg][buf], 1)] = tok;
                                        }
                                    }
                                }
                            }
                            mbar_arrive(rbar + wg * 2 + 1);
                            okr = mbar_wait_fast(rbar + wg * 2 + 1, red_par, abort_flag, p.status) && okr;
                            red_par ^= 1u;
                            if (!__all_sync(0xFFFFFFFFu, okr)) goto epi_done;
                            const int nd = red_n[wg][buf];
                            for (int i = 0; i < nd; ++i) {
                                // out[tok, n] = bf16(sum_j w[tok, j] z[tok*k + j, n]) over the
                                // kept routes in top-k order (k_moe_reduce's arithmetic)
                                const int tok = red_list[wg][buf][i];
                                const long long rb = static_cast<long long>(tok) * p.red_k;
                                const uint16_t* z = static_cast<const uint16_t*>(p.out);
                                float sum = 0.0f;
                                for (int j0 = 0; j0 < p.red_k; j0 += 8) {
                                    int sl[8];
                                    float wv[8];
                                    uint16_t zv[8];
#pragma unroll
                                    for (int jj = 0; jj < 8; ++jj) {
                                        const bool in = j0 + jj < p.red_k;
                                        sl[jj] = in ? __ldcg(p.red_slot + rb + j0 + jj) : -1;
                                        wv[jj] = in ? __ldg(p.red_w + rb + j0 + jj) : 0.0f;
                                    }
#pragma unroll
                                    for (int jj = 0; jj < 8; ++jj)
                                        zv[jj] = sl[jj] >= 0 ? __ldcg(z + (rb + j0 + jj) * p.N_out + n) : 0;
#pragma unroll
                                    for (int jj = 0; jj < 8; ++jj)
                                        if (sl[jj] >= 0)
                                            sum = __fmaf_rn(wv[jj], __uint_as_float(static_cast<uint32_t>(zv[jj]) << 16), sum);
                                }
                                p.red_out[static_cast<long long>(tok) * p.N_out + n] =
                                    static_cast<uint16_t>(f32_to_bf16_bits(sum));
                            }
                        }
                    }
                }
            }
            mbar_arrive_relaxed(dempty + slot);
            if (++slot == C::kRing) { slot = 0; dph ^= 1u; }
        }
    epi_done:;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, C::kCols);
    }
}

template <int BM, bool DYN>
int launch_bm(const CUtensorMap& tw, const CUtensorMap& ta, const GemmArgs& p, long long max_units,
              bool pdl, cudaStream_t stream) {
    using C = Cfg<BM>;
    if (!ensure_smem(reinterpret_cast<const void*>(k_grouped_gemm<BM, DYN>), C::kSmem)) {
        set_error("grouped_gemm: shared-memory limit %d refused", C::kSmem);
        return MOE_ERR_LAUNCH;
    }
    long long grid = std::min<long long>(sm_count(), max_units);
    if (grid <= 0) return MOE_OK;
    Launch L(dim3(static_cast<unsigned>(grid)), dim3(C::kThreads), C::kSmem, stream, pdl);
    cudaError_t e = cudaLaunchKernelEx(&L.cfg, k_grouped_gemm<BM, DYN>, tw, ta, p);
    if (e != cudaSuccess) { set_error("grouped_gemm launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

}  // namespace

// 2-D map over a row-major [rows, K] byte matrix (E4M3 codes), box 128 columns x box_rows rows, 128-byte
// swizzle (the layout the MMA descriptors expect).
bool make_tma_map_u8(CUtensorMap* m, const void* base, long long rows, int K, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


int launch_grouped_gemm(moe_proj proj, const uint8_t* a_q, const float* a_s, int a_rows, int K,
                        const uint8_t* w_q, const float* w_s, int E_local, int N_out,
                        moe_weight_layout w_layout, const int32_t* sorted_idx, const int32_t* block_expert,
                        const int32_t* num_blocks, int B_cap, int block_m, void* out,
                        moe_dtype out_dtype, int out_rows, int splits, bool pdl,
                        cudaStream_t stream, bool wait_first, const int32_t* self_ids,
                        const int32_t* self_map, int self_R, int self_E, const EpilogueReduce* red,
                        unsigned long long* sched) {
    if (proj != MOE_PROJ_GATE_UP && proj != MOE_PROJ_DOWN) { set_error("grouped_gemm: bad proj"); return MOE_ERR_ARG; }
    if (!a_q || !a_s || !w_q || !w_s || !sorted_idx || !block_expert || !num_blocks || !out) {
        set_error("grouped_gemm: null pointer");
        return MOE_ERR_ARG;
    }
    if (!aligned16(a_q) || !aligned16(w_q) || !aligned16(out) || !aligned16(a_s) || !aligned16(w_s)) {
        set_error("grouped_gemm: pointers must be 16-byte aligned");
        return MOE_ERR_ARG;
    }
    if (K <= 0 || K % 128 || N_out <= 0 || N_out % 128 || E_local <= 0 || B_cap < 0 || out_rows < 0) {
        set_error("grouped_gemm: K and N_out must be positive multiples of 128 (K=%d N_out=%d)", K, N_out);
        return MOE_ERR_ARG;
    }
    if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128) {
        set_error("grouped_gemm: block_m must be 16, 32, 64 or 128");
        return MOE_ERR_ARG;
    }
    const int KB = K / 128;
    if (out_dtype == MOE_DTYPE_BF16 ? splits != 1 : (splits < 1 || splits > KB)) {
        set_error("grouped_gemm: splits must be 1 for BF16 output and in [1, K/128] for fp32");
        return MOE_ERR_ARG;
    }
    if (static_cast<long long>(a_rows) < static_cast<long long>(B_cap) * block_m) {
        set_error("grouped_gemm: a_rows (%d) < B_cap*block_m", a_rows);
        return MOE_ERR_ARG;
    }
    if (proj == MOE_PROJ_GATE_UP && static_cast<long long>(out_rows) < static_cast<long long>(B_cap) * block_m) {
        set_error("grouped_gemm: GATE_UP writes slot rows; out_rows must be >= B_cap*block_m");
        return MOE_ERR_ARG;
    }
    if (B_cap == 0) return MOE_OK;
    if (w_layout != MOE_WEIGHTS_ROW_MAJOR && w_layout != MOE_WEIGHTS_TILED) {
        set_error("grouped_gemm: unknown weight layout");
        return MOE_ERR_ARG;
    }
    const bool tiled = w_layout == MOE_WEIGHTS_TILED;
    const long long w_rows = tiled ? static_cast<long long>(E_local) * N_out * (K / 128)
                                   : static_cast<long long>(E_local) * N_out;
    if (w_rows > 0x7FFFFFFFLL) { set_error("grouped_gemm: weight tensor too large"); return MOE_ERR_ARG; }
    CUtensorMap tw, ta;
    if (!make_tma_map_u8(&tw, w_q, w_rows, tiled ? 128 : K, 128) ||
        !make_tma_map_u8(&ta, a_q, a_rows, K, block_m)) {
        set_error("grouped_gemm: tensor-map encode failed (driver entry point missing or bad layout)");
        return MOE_ERR_LAUNCH;
    }
    GemmArgs p{};
    p.a_s = a_s;
    p.a_rows = a_rows;
    p.K = K;
    p.KB = KB;
    p.w_s = w_s;
    p.E_local = E_local;
    p.N_out = N_out;
    p.NT = N_out / 128;
    p.sorted_idx = sorted_idx;
    p.block_expert = block_expert;
    p.num_blocks = num_blocks;
    p.B_cap = B_cap;
    p.out = out;
    p.out_f32 = out_dtype == MOE_DTYPE_F32;
    p.out_rows = out_rows;
    p.splits = splits;
    p.scatter = proj == MOE_PROJ_DOWN;
    p.w_tiled = tiled ? 1 : 0;
    p.status = device_status_ptr();
    p.wait_first = wait_first ? 1 : 0;
    p.pdl = pdl ? 1 : 0;
    if (self_ids) {
        if (proj != MOE_PROJ_GATE_UP || block_m > 32 || self_R < 1 || self_R > 32 || self_E < 1 ||
            !pdl || wait_first) {
            set_error("grouped_gemm: self-routing needs GATE_UP, block_m <= 32, 1..32 routes and PDL");
            return MOE_ERR_ARG;
        }
        p.self_ids = self_ids;
        p.self_map = self_map;
        p.self_R = self_R;
        p.self_E = self_E;
    }
    if (red) {
        if (proj != MOE_PROJ_DOWN || block_m > 32 || out_dtype != MOE_DTYPE_BF16 || !red->out ||
            !red->cnt || !red->w || !red->slot || red->k < 1 || red->k > kReduceMaxTopk ||
            red->M < 1 || !aligned16(red->out)) {
            set_error("grouped_gemm: the epilogue reduce needs DOWN, block_m <= 32, BF16 output and k <= %d",
                      kReduceMaxTopk);
            return MOE_ERR_ARG;
        }
        p.red_out = static_cast<uint16_t*>(red->out);
        p.red_cnt = red->cnt;
        p.red_w = red->w;
        p.red_slot = red->slot;
        p.red_k = red->k;
        p.red_M = red->M;
    }
    if (sched && block_m > 32) {
        set_error("grouped_gemm: the dynamic tail is built for block_m 16 and 32");
        return MOE_ERR_ARG;
    }
    if (sched) {
        // dynamic chunks of about kSchedChunkBytes of weights: a short tail, and few enough
        // descriptors that the metadata warp keeps ahead of the producer.  The chunk's unit count
        // divides a block's (tiles x splits), so that no chunk straddles two blocks (each block a
        // chunk touches costs its expert and rows, and a new descriptor run).
        const long long unit_bytes = static_cast<long long>((KB + splits - 1) / splits) * 128 * 128;
        const long long per_block = static_cast<long long>(N_out / 128) * splits;
        long long chunk = std::max(1LL, (kSchedChunkBytes + unit_bytes - 1) / unit_bytes);
        while (chunk > 1 && per_block % chunk != 0) --chunk;
        p.sched = sched;
        p.sched_chunk = static_cast<int>(chunk);
    }
    const long long max_units = static_cast<long long>(B_cap) * p.NT * splits;
    switch (block_m) {
        case 16: return p.sched ? launch_bm<16, true>(tw, ta, p, max_units, pdl, stream)
                                : launch_bm<16, false>(tw, ta, p, max_units, pdl, stream);
        case 32: return p.sched ? launch_bm<32, true>(tw, ta, p, max_units, pdl, stream)
                                : launch_bm<32, false>(tw, ta, p, max_units, pdl, stream);
        case 64: return launch_bm<64, false>(tw, ta, p, max_units, pdl, stream);
        default: return launch_bm<128, false>(tw, ta, p, max_units, pdl, stream);
    }
}

}  // namespace moe

extern "C" int moe_blockfp8_grouped_gemm(moe_proj proj, const uint8_t* a_q, const float* a_s,
                                         int a_rows, int K, const uint8_t* w_q, const float* w_s,
                                         int E_local, int N_out, moe_weight_layout w_layout,
                                         const int32_t* sorted_idx,
                                         const int32_t* block_expert, const int32_t* num_blocks,
                                         int B_cap, int block_m, void* out, moe_dtype out_dtype,
                                         int out_rows, int splits, cudaStream_t stream) {
    moe::clear_error();
    if (!moe::device_is_sm103()) { moe::set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    return moe::launch_grouped_gemm(proj, a_q, a_s, a_rows, K, w_q, w_s, E_local, N_out, w_layout,
                                    sorted_idx,
                                    block_expert, num_blocks, B_cap, block_m, out, out_dtype,
                                    out_rows, splits, false, stream);
}

namespace moe {
namespace {
// 16 bytes per thread: tiled[e][nt][kb][r][c] = src[e][nt*128 + r][kb*128 + c]
__global__ void __launch_bounds__(256) k_pack_weights(const uint4* __restrict__ src, int E, int N_out,
                                                      int K, uint4* __restrict__ dst) {
    const int NT = N_out / 128, KB = K / 128;
    const long long total = static_cast<long long>(E) * N_out * K / 16;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        long long t = i;
        const int c16 = static_cast<int>(t % 8); t /= 8;
        const int r = static_cast<int>(t % 128); t /= 128;
        const int kb = static_cast<int>(t % KB); t /= KB;
        const int nt = static_cast<int>(t % NT); t /= NT;
        const long long e = t;
        const long long from = ((e * N_out + nt * 128 + r) * K + kb * 128) / 16 + c16;
        dst[i] = __ldg(src + from);
    }
}
}  // namespace
}  // namespace moe

extern "C" int moe_blockfp8_pack_weights(const uint8_t* w_q, int E_local, int N_out, int K,
                                         uint8_t* w_tiled, cudaStream_t stream) {
    using namespace moe;
    clear_error();
    if (!device_is_sm103()) { set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    if (!w_q || !w_tiled || !aligned16(w_q) || !aligned16(w_tiled)) {
        set_error("moe_blockfp8_pack_weights: null or misaligned pointer");
        return MOE_ERR_ARG;
    }
    if (E_local <= 0 || N_out <= 0 || K <= 0 || N_out % 128 || K % 128) {
        set_error("moe_blockfp8_pack_weights: N_out and K must be positive multiples of 128");
        return MOE_ERR_ARG;
    }
    const long long total = static_cast<long long>(E_local) * N_out * K / 16;
    long long blocks = std::min<long long>((total + 255) / 256, static_cast<long long>(sm_count()) * 16);
    Launch L(dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, false);
    cudaError_t e = cudaLaunchKernelEx(&L.cfg, k_pack_weights, reinterpret_cast<const uint4*>(w_q),
                                       E_local, N_out, K, reinterpret_cast<uint4*>(w_tiled));
    if (e != cudaSuccess) { set_error("moe_blockfp8_pack_weights launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}
