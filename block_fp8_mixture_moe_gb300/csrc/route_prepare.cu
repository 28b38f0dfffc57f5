// route_prepare.cu -- route preparation: stable counting sort of the top-k routes by local
// expert, block_m-padded compact blocks for the experts that received routes.
//
// Method: lmdeploy PR #4857 "optimize compact blocked FP8 MoE and route preparation", section
// "Changes": one CTA when routes and experts are at most 2,048 (few graph nodes), a scalable
// parallel path otherwise; outputs are the sorted route indices and the compact blocks.  The
// review on that page asks that the local-expert slice and block_m be checked before launch.
//
// Single CTA (8, 16 or 32 warps, by route count).  Every route's local expert goes to shared
// memory.  Warp w owns a contiguous chunk of routes and counts it into its own row of a
// per-warp histogram [warps][E_local] (uint16), one shared-memory atomic per route (counts do
// not depend on the atomics' order).  A column scan over the rows turns the histogram into
// per-warp starting ranks; a block scan over the block_m-padded expert totals gives each
// expert's first slot.  The scatter walks each warp's chunk again, 32 routes at a time:
// __match_any_sync groups the lanes of one expert, and slot = expert start + warp rank + rank
// inside the group, so the order inside an expert is the route order (stable).
//
// Multi CTA.  Kernel 1: each CTA histograms one chunk of routes (shared-memory atomics; counts
// only) into the workspace; the CTA that finishes last (atomic ticket, no waiting) scans the
// chunk histograms per expert, scans the padded totals and writes counts, offsets, the block
// table and the -1 pads.  Kernel 2: each CTA runs the single-CTA warp walk on its own chunk,
// offset by its chunk prefix.  Neither kernel ever waits on another CTA.
#include "common.cuh"

#include <algorithm>
#include <mutex>

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kSingleWarps = 32;
constexpr int kSingleMaxRoutes = 8192;
// the compacting single-CTA variant when its shared memory fits comfortably
constexpr size_t kCompactMaxSmem = 200 * 1024;
constexpr int kSingleMaxExperts = 2048;
constexpr int kMaxExperts = 4096;
constexpr size_t kMultiHistBytes = 96 * 1024;  // per-warp histogram budget of a scatter CTA

struct RouteArgs {
    const int32_t* ids;
    int R, E;
    const int32_t* map;
    int E_loc, bm, B_cap;
    int bm_shift;  // log2(bm): bm is a power of two, so block arithmetic is shifts
    int32_t* sorted_idx;
    int32_t* block_expert;
    int32_t* num_blocks;
    int32_t* count;
    int32_t* offset;   // nullable
    int32_t* route_slot;  // nullable: slot of each route, -1 when dropped
    int* status;
    // multi-CTA workspace
    int32_t* ws_cnt;   // [nchunks][E_loc]: chunk histograms, then chunk prefixes
    int32_t* ws_off;   // [E_loc + 1]: first slot of each expert
    unsigned* ws_done; // ticket counter
    int chunk, nchunks, warps;
    // optional: words the next kernel needs at zero (its phase counters), cleared here
    uint32_t* zero_ptr;
    int zero_n;
    int compact;  // single CTA with an expert map: compact the kept routes first
    // The -1 pads of sorted_idx are left to the next kernel (the layer's input quantisation,
    // spread over every SM): one CTA's scattered pad stores took 1.6 us at 256 experts and
    // 7 us at 512 on the critical path.  The single-CTA and multi-CTA paths only.
    int skip_pads;
    // With the compaction (single CTA, expert map): the slot of each kept route in route order
    // and their number, so that the layer's activation kernel walks the kept routes only
    // (nullable; written only by the compacting path).
    int32_t* kept_slot;
    int32_t* n_kept;
};

// Clears the caller's zero region (grid-stride over the launch).
__device__ __forceinline__ void clear_zero_region(const RouteArgs& p) {
    if (!p.zero_ptr) return;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.zero_n; i += gridDim.x * blockDim.x)
        p.zero_ptr[i] = 0u;
}

__device__ __forceinline__ int local_of(const RouteArgs& p, int r) {
    int id = __ldg(p.ids + r);
    if (id < 0 || id >= p.E) return -1;
    int e = p.map ? __ldg(p.map + id) : id;
    if (e < -1 || e >= p.E_loc) {
        if (p.status) atomicOr(p.status, MOE_DEV_BAD_EXPERT_MAP);
        return -1;
    }
    return e;
}

// loc[r] = the global expert id of route r, for r in [0, R): a thread issues all its loads (up to
// kIdBatch) before its first store.  A loop that stores each load before the next waits for them
// one after another: 3.3 us for the 6 ids a thread loads at 6144 routes.  (At decode sizes, with
// one or two routes a thread, the plain loop measured faster.)
constexpr int kIdBatch = 8;
__device__ __forceinline__ void load_ids_batched(const RouteArgs& p, int* loc) {
    for (int r0 = threadIdx.x; r0 < p.R; r0 += kIdBatch * blockDim.x) {
        int v[kIdBatch];
#pragma unroll
        for (int q = 0; q < kIdBatch; ++q) {
            const int r = r0 + q * blockDim.x;
            v[q] = r < p.R ? __ldg(p.ids + r) : -1;
        }
#pragma unroll
        for (int q = 0; q < kIdBatch; ++q) {
            const int r = r0 + q * blockDim.x;
            if (r < p.R) loc[r] = v[q];
        }
    }
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// In-place exclusive scan of data[0..n) by the whole block; returns the total.  `tmp` holds at
// least 33 ints.
__device__ int block_exclusive_scan(int* data, int n, int* tmp) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += data[i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = nt >> 5;
        int v = lane < nw ? tmp[lane] : 0;
        int s = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(kFull, s, o);
            if (lane >= o) s += u;
        }
        if (lane < nw) tmp[lane] = s - v;  // exclusive warp prefix
        if (lane == 31) tmp[32] = s;       // total
    }
    __syncthreads();
    int run = tmp[warp] + incl - local;
    for (int i = lo; i < hi; ++i) {
        int v = data[i];
        data[i] = run;
        run += v;
    }
    int total = tmp[32];
    __syncthreads();
    return total;
}

// Per-warp histogram of the routes [w*per_warp, min(n, (w+1)*per_warp)) of `loc`.
__device__ __forceinline__ void warp_histogram(const int* loc, int n, int per_warp,
                                               uint16_t* row) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int lo = w * per_warp, hi = min(n, lo + per_warp);
    // One shared-memory atomic per route.  The 16-bit counters are updated through 32-bit
    // atomics on their word (a warp's count stays below 65536, so no carry reaches the
    // neighbour).  Grouping equal experts with __match_any_sync first took 3.5 us at 4096 routes
    // over 512 experts (prefill layer 732.9 -> 730.1 us, decode M=256 254.8 -> 253.1).
    const uintptr_t rbase = reinterpret_cast<uintptr_t>(row);
    for (int r = lo + lane; r < hi; r += 32) {
        const int e = loc[r];
        if (e >= 0) {
            const uintptr_t a = rbase + 2u * static_cast<unsigned>(e);
            atomicAdd(reinterpret_cast<unsigned*>(a & ~static_cast<uintptr_t>(3)), 1u << ((a & 2u) * 8u));
        }
    }
    __syncwarp();
}

// Turns the per-warp histograms [nw][E_loc] into exclusive per-warp starting ranks; stores the
// expert totals in `tot` when it is not null.
__device__ __forceinline__ void column_scan(uint16_t* wcnt, int nw, int E_loc, int* tot) {
    for (int e = threadIdx.x; e < E_loc; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < nw; ++w) {
            int c = wcnt[w * E_loc + e];
            wcnt[w * E_loc + e] = static_cast<uint16_t>(run);
            run += c;
        }
        if (tot) tot[e] = run;
    }
}

// Stable scatter of this CTA's routes (local ids in `loc`, global route id = first + i, or
// ridx[i] for a compacted list of kept routes).
// slot = start[e] + chunk_base(e) + warp rank + rank in the 32-group.
__device__ __forceinline__ void warp_scatter(const RouteArgs& p, const int* loc, int n, int first,
                                             int per_warp, uint16_t* row, const int* start,
                                             const int32_t* chunk_base, const int* ridx = nullptr) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int lo = w * per_warp, hi = min(n, lo + per_warp);
    for (int base = lo; base < hi; base += 32) {
        const int r = base + lane;
        const int e = r < hi ? loc[r] : -1;
        const unsigned m = __match_any_sync(kFull, e);
        const int route = ridx ? (r < hi ? ridx[r] : -1) : first + r;
        if (e >= 0) {
            int slot = start[e] + row[e] + __popc(m & lanemask_lt());
            if (chunk_base) slot += chunk_base[e];
            p.sorted_idx[slot] = route;
            if (p.route_slot) p.route_slot[route] = slot;
            if (ridx && p.kept_slot) p.kept_slot[r] = slot;
        } else if (r < hi && p.route_slot) {
            p.route_slot[route] = -1;
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(m) - 1) row[e] = static_cast<uint16_t>(row[e] + __popc(m));
        __syncwarp();
    }
}

// Writes counts, offsets, num_blocks, the block table and every -1 pad from the expert totals
// `tot` and the padded starts `start` (start[E_loc] = padded total).
__device__ void write_metadata(const RouteArgs& p, const int* tot, const int* start) {
    const int nb = start[p.E_loc] >> p.bm_shift;
    for (int e = threadIdx.x; e < p.E_loc; e += blockDim.x) {
        p.count[e] = tot[e];
        if (p.offset) p.offset[e] = start[e];
        for (int b = start[e] >> p.bm_shift; b < (start[e + 1] >> p.bm_shift); ++b) p.block_expert[b] = e;
        if (!p.skip_pads)
            for (int s = start[e] + tot[e]; s < start[e + 1]; ++s) p.sorted_idx[s] = -1;
    }
    for (int b = nb + threadIdx.x; b < p.B_cap; b += blockDim.x) p.block_expert[b] = -1;
    if (!p.skip_pads)
        for (long long s = (static_cast<long long>(nb) << p.bm_shift) + threadIdx.x;
             s < (static_cast<long long>(p.B_cap) << p.bm_shift); s += blockDim.x)
            p.sorted_idx[s] = -1;
    if (threadIdx.x == 0) {
        *p.num_blocks = nb;
        if (p.offset) p.offset[p.E_loc] = start[p.E_loc];
    }
}

// Shared memory of the single-CTA kernel: loc[R] | start[E_loc+1] | tot[E_loc] | tmp[33] |
// wcnt[warps][E_loc] (uint16), and with an expert map also smap[E] | kloc[R] | kidx[R].
__host__ __device__ inline size_t single_ints(int R, int E_loc) {
    const size_t ints = static_cast<size_t>(R) + (E_loc + 1) + E_loc + 33;
    return (ints + 3) & ~static_cast<size_t>(3);
}
size_t single_smem_bytes(int R, int E, int E_loc, bool map, int warps = kSingleWarps) {
    const size_t base = single_ints(R, E_loc) * 4 + static_cast<size_t>(warps) * E_loc * 2;
    return map ? ((base + 15) & ~static_cast<size_t>(15)) + (static_cast<size_t>(E) + 2 * R) * 4 : base;
}

template <int W>
__global__ void __launch_bounds__(W * 32, 1) k_route_single(RouteArgs p) {
    extern __shared__ __align__(16) int sm[];
    int* loc = sm;
    int* start = loc + p.R;
    int* tot = start + p.E_loc + 1;
    int* tmp = tot + p.E_loc;
    const size_t ints = single_ints(p.R, p.E_loc);
    uint16_t* wcnt = reinterpret_cast<uint16_t*>(sm + ints);
    grid_dep_wait();
    grid_dep_launch();
    clear_zero_region(p);
    int n = p.R;         // routes the sort walks
    const int* key = loc;
    const int* ridx = nullptr;
    if (p.compact) {
        // With an expert map most routes are usually dropped (an expert-parallel slice keeps
        // about 1/8): the map is staged in shared memory next to the ids, so a route's local
        // expert costs no second dependent global load, and the kept routes are compacted in
        // route order (a block scan) before the sort, which then walks only them.
        int* smap = reinterpret_cast<int*>(
            (reinterpret_cast<uintptr_t>(wcnt + W * p.E_loc) + 15) & ~static_cast<uintptr_t>(15));
        int* kloc = smap + p.E;
        int* kidx = kloc + p.R;
        for (int i = threadIdx.x; i < p.E; i += blockDim.x) smap[i] = __ldg(p.map + i);
        load_ids_batched(p, loc);
        for (int i = threadIdx.x; i < W * p.E_loc; i += blockDim.x) wcnt[i] = 0;
        __syncthreads();
        for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
            const int id = loc[r];
            int e = (id < 0 || id >= p.E) ? -1 : smap[id];
            if (e < -1 || e >= p.E_loc) {
                if (p.status) atomicOr(p.status, MOE_DEV_BAD_EXPERT_MAP);
                e = -1;
            }
            loc[r] = e;
            if (e < 0 && p.route_slot) p.route_slot[r] = -1;
        }
        __syncthreads();
        // stable compaction: thread t owns routes [t*per, (t+1)*per)
        const int per = (p.R + blockDim.x - 1) / blockDim.x;
        const int lo = min(p.R, static_cast<int>(threadIdx.x) * per), hi = min(p.R, lo + per);
        int cnt = 0;
        for (int r = lo; r < hi; ++r) cnt += loc[r] >= 0;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) tmp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int nw = blockDim.x >> 5;
            const int v = lane < nw ? tmp[lane] : 0;
            int sc = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(kFull, sc, o);
                if (lane >= o) sc += u;
            }
            if (lane < nw) tmp[lane] = sc - v;
            if (lane == 31) tmp[32] = sc;
        }
        __syncthreads();
        int pos = tmp[warp] + incl - cnt;
        for (int r = lo; r < hi; ++r) {
            if (loc[r] >= 0) { kloc[pos] = loc[r]; kidx[pos] = r; ++pos; }
        }
        n = tmp[32];
        if (threadIdx.x == 0 && p.n_kept) *p.n_kept = n;
        key = kloc;
        ridx = kidx;
        __syncthreads();
    } else {
        for (int r = threadIdx.x; r < p.R; r += blockDim.x) loc[r] = local_of(p, r);
        for (int i = threadIdx.x; i < W * p.E_loc; i += blockDim.x) wcnt[i] = 0;
        __syncthreads();
    }
    const int per_warp = (n + W - 1) / W;
    uint16_t* row = wcnt + (threadIdx.x >> 5) * p.E_loc;
    warp_histogram(key, n, per_warp, row);
    __syncthreads();
    column_scan(wcnt, W, p.E_loc, tot);
    __syncthreads();
    for (int e = threadIdx.x; e < p.E_loc; e += blockDim.x)
        start[e] = ((tot[e] + p.bm - 1) >> p.bm_shift) << p.bm_shift;
    __syncthreads();
    const int total = block_exclusive_scan(start, p.E_loc, tmp);
    if (threadIdx.x == 0) start[p.E_loc] = total;
    __syncthreads();
    write_metadata(p, tot, start);
    warp_scatter(p, key, n, 0, per_warp, row, start, nullptr, ridx);
}

// At most 32 routes: one warp holds a route per lane.  __match_any_sync groups the lanes of
// equal experts, so a route's stable rank in its expert is the number of same-expert lanes
// below it; the groups' leaders form a table of at most 32 active experts (local id, count,
// padded count).  Meanwhile the CTA's other warps write every pad and empty block entry; after
// the one barrier, each expert's count and padded offset are sums over that table, and the
// real entries overwrite the pads.
constexpr int kWarpMaxRoutes = kRouteWarpMaxRoutes;
constexpr int kWarpThreads = 256;

// The one-warp sort's table: the active experts of at most 32 routes (local id, route count,
// padded count), in the order of their leading lanes.
struct WarpTable {
    int e[32], cnt[32], pad[32];
    int n;
};

// Before a CTA barrier: lane r of warp 0 takes route r (its local expert in *e, its stable rank
// among the same-expert lanes in *rank) and fills the table; with `pads`, the CTA's other warps
// meanwhile write every -1 pad of sorted_idx and block_expert.
__device__ __forceinline__ void warp_table_build(const RouteArgs& p, WarpTable& t, bool pads,
                                                 int* e, int* rank) {
    const int tid = threadIdx.x, lane = tid & 31;
    *e = -1;
    *rank = 0;
    if (tid < 32) {
        const int er = lane < p.R ? local_of(p, lane) : -1;
        const unsigned m = __match_any_sync(kFull, er);
        const int rk = __popc(m & lanemask_lt());
        const bool lead = er >= 0 && rk == 0;
        const unsigned leads = __ballot_sync(kFull, lead);
        if (lead) {
            const int i = __popc(leads & lanemask_lt());
            const int c = __popc(m);
            t.e[i] = er;
            t.cnt[i] = c;
            t.pad[i] = ((c + p.bm - 1) >> p.bm_shift) << p.bm_shift;
        }
        if (lane == 0) t.n = __popc(leads);
        *e = er;
        *rank = rk;
    } else if (pads) {
        const int nthr = blockDim.x - 32, u = tid - 32;
        for (long long sl = u; sl < (static_cast<long long>(p.B_cap) << p.bm_shift); sl += nthr) p.sorted_idx[sl] = -1;
        for (int b = u; b < p.B_cap; b += nthr) p.block_expert[b] = -1;
    }
}

// After the barrier: the padded offset of local expert x (the padded counts of the active
// experts below it).
__device__ __forceinline__ int warp_table_offset(const WarpTable& t, int x) {
    int off = 0;
    for (int i = 0; i < t.n; ++i) off += t.e[i] < x ? t.pad[i] : 0;
    return off;
}

// After the barrier: counts, offsets, block table, block count and the real sorted_idx and
// route_slot entries (over the pads written before it).
__device__ __forceinline__ void warp_table_write(const RouteArgs& p, const WarpTable& t, int e, int rank) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int n = t.n;
    for (int x = tid; x < p.E_loc; x += blockDim.x) {
        int c = 0;
        for (int i = 0; i < n; ++i) c = t.e[i] == x ? t.cnt[i] : c;
        p.count[x] = c;
        if (p.offset) p.offset[x] = warp_table_offset(t, x);
    }
    if (tid < n) {
        const int off = warp_table_offset(t, t.e[tid]);
        for (int b = off >> p.bm_shift; b < ((off + t.pad[tid]) >> p.bm_shift); ++b) p.block_expert[b] = t.e[tid];
    }
    if (tid == 0) {
        int total = 0;
        for (int i = 0; i < n; ++i) total += t.pad[i];
        *p.num_blocks = total >> p.bm_shift;
        if (p.offset) p.offset[p.E_loc] = total;
    }
    if (tid < 32 && lane < p.R) {
        const int slot = e >= 0 ? warp_table_offset(t, e) + rank : -1;
        if (e >= 0) p.sorted_idx[slot] = lane;
        if (p.route_slot) p.route_slot[lane] = slot;
    }
}

__global__ void __launch_bounds__(kWarpThreads, 1) k_route_warp(RouteArgs p) {
    __shared__ WarpTable t;
    grid_dep_wait();
    grid_dep_launch();
    clear_zero_region(p);
    int e, rank;
    warp_table_build(p, t, true, &e, &rank);
    __syncthreads();
    warp_table_write(p, t, e, rank);
}

// Multi-CTA kernel 1: chunk histograms; the last CTA to finish builds the metadata.
__global__ void __launch_bounds__(1024) k_route_count(RouteArgs p) {
    extern __shared__ __align__(16) int sm[];
    int* hist = sm;                         // [E_loc]
    int* start = hist + p.E_loc;            // [E_loc + 1]
    int* tmp = start + p.E_loc + 1;         // [33]
    __shared__ int is_last;
    grid_dep_wait();
    grid_dep_launch();
    clear_zero_region(p);
    const int c = blockIdx.x;
    const int lo = c * p.chunk, hi = min(p.R, lo + p.chunk);
    for (int e = threadIdx.x; e < p.E_loc; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    for (int r = lo + threadIdx.x; r < hi; r += blockDim.x) {
        int e = local_of(p, r);
        if (e >= 0) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E_loc; e += blockDim.x)
        p.ws_cnt[static_cast<long long>(c) * p.E_loc + e] = hist[e];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(p.ws_done, 1u) == static_cast<unsigned>(p.nchunks - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // per expert: exclusive prefix over chunks (in place) and the total
    int* tot = hist;
    for (int e = threadIdx.x; e < p.E_loc; e += blockDim.x) {
        int run = 0;
        for (int cc = 0; cc < p.nchunks; ++cc) {
            int32_t* q = p.ws_cnt + static_cast<long long>(cc) * p.E_loc + e;
            int v = __ldcg(q);
            *q = run;
            run += v;
        }
        tot[e] = run;
        start[e] = ((run + p.bm - 1) >> p.bm_shift) << p.bm_shift;
    }
    __syncthreads();
    const int total = block_exclusive_scan(start, p.E_loc, tmp);
    if (threadIdx.x == 0) start[p.E_loc] = total;
    __syncthreads();
    for (int e = threadIdx.x; e <= p.E_loc; e += blockDim.x) p.ws_off[e] = start[e];
    write_metadata(p, tot, start);
    if (threadIdx.x == 0) *p.ws_done = 0u;  // ready for the next call
}

// Multi-CTA kernel 2: the stable warp walk over one chunk.
__global__ void __launch_bounds__(1024) k_route_scatter(RouteArgs p) {
    extern __shared__ __align__(16) int sm[];
    int* loc = sm;                                        // [chunk]
    int* start = loc + p.chunk;                           // [E_loc]
    size_t ints = static_cast<size_t>(p.chunk) + p.E_loc;
    ints = (ints + 3) & ~static_cast<size_t>(3);
    uint16_t* wcnt = reinterpret_cast<uint16_t*>(sm + ints);  // [warps][E_loc]
    grid_dep_wait();
    grid_dep_launch();
    const int c = blockIdx.x;
    const int first = c * p.chunk;
    const int n = min(p.R - first, p.chunk);
    for (int i = threadIdx.x; i < n; i += blockDim.x) loc[i] = local_of(p, first + i);
    for (int e = threadIdx.x; e < p.E_loc; e += blockDim.x) start[e] = __ldcg(p.ws_off + e);
    for (int i = threadIdx.x; i < p.warps * p.E_loc; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    uint16_t* row = wcnt + (threadIdx.x >> 5) * p.E_loc;
    warp_histogram(loc, n, 32, row);
    __syncthreads();
    column_scan(wcnt, p.warps, p.E_loc, nullptr);
    __syncthreads();
    warp_scatter(p, loc, n, first, 32, row, start, p.ws_cnt + static_cast<long long>(c) * p.E_loc);
}

int multi_warps(int E_loc) {
    int w = static_cast<int>(kMultiHistBytes / (static_cast<size_t>(E_loc) * 2));
    return std::max(1, std::min(32, w));
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

bool route_single_cta(int R, int E_local, moe_route_path path) {
    if (path == MOE_ROUTE_SINGLE_CTA) return true;
    if (path == MOE_ROUTE_MULTI_CTA) return false;
    // The pages switch at 2,048 routes and experts; on GB300 the single CTA measured faster than
    // the two multi-CTA launches at 4,096 routes over 512 experts and 6,144 over 32.
    return R <= kSingleMaxRoutes && E_local <= 512;
}

bool route_compacts(int R, int E, int E_local, bool map) {
    return map && R > kWarpMaxRoutes && route_single_cta(R, E_local, MOE_ROUTE_AUTO) &&
           single_smem_bytes(R, E, E_local, true) <= kCompactMaxSmem;
}

size_t route_workspace_bytes(int R, int E_local, int block_m) {
    (void)block_m;
    const int chunk = multi_warps(E_local) * 32;
    const long long nchunks = std::max(1, (R + chunk - 1) / chunk);
    return align256(static_cast<size_t>(nchunks) * E_local * 4) +
           align256(static_cast<size_t>(E_local + 1) * 4) + 256;
}

int launch_route_prepare(const int32_t* topk_ids, int M, int k, int E, const int32_t* expert_map,
                         int E_local, int block_m, moe_route_path path, int32_t* sorted_idx,
                         int32_t* block_expert, int32_t* num_blocks, int32_t* expert_count,
                         int32_t* expert_offset, int32_t* route_slot, void* workspace,
                         size_t ws_bytes, bool pdl, cudaStream_t stream, uint32_t* zero_ptr,
                         int zero_n, bool skip_pads, int32_t* kept_slot, int32_t* n_kept) {
    if (M < 0 || k <= 0 || E <= 0 || E_local <= 0) {
        set_error("moe_route_prepare: need M >= 0, k > 0, E > 0, E_local > 0");
        return MOE_ERR_ARG;
    }
    if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128) {
        set_error("moe_route_prepare: block_m must be 16, 32, 64 or 128 (got %d)", block_m);
        return MOE_ERR_ARG;
    }
    if (k > E) { set_error("moe_route_prepare: top-k %d > E %d", k, E); return MOE_ERR_ARG; }
    if (!expert_map && E_local != E) {
        set_error("moe_route_prepare: without an expert map E_local must equal E (%d vs %d)", E_local, E);
        return MOE_ERR_EXPERT_SLICE;
    }
    if (E_local > kMaxExperts || (!expert_map ? false : E_local > E)) {
        set_error("moe_route_prepare: E_local %d outside [1, min(E, %d)]", E_local, kMaxExperts);
        return MOE_ERR_EXPERT_SLICE;
    }
    if (static_cast<long long>(M) * k > (1LL << 24)) { set_error("moe_route_prepare: too many routes"); return MOE_ERR_ARG; }
    const int R = M * k;
    if (!num_blocks || !expert_count || (R > 0 && (!topk_ids || !sorted_idx || !block_expert))) {
        set_error("moe_route_prepare: null output or input pointer");
        return MOE_ERR_ARG;
    }
    RouteArgs p{};
    p.ids = topk_ids;
    p.R = R;
    p.E = E;
    p.map = expert_map;
    p.E_loc = E_local;
    p.bm = block_m;
    p.bm_shift = block_m == 16 ? 4 : block_m == 32 ? 5 : block_m == 64 ? 6 : 7;
    p.B_cap = (R + block_m - 1) / block_m + std::min(E_local, R);
    p.sorted_idx = sorted_idx;
    p.block_expert = block_expert;
    p.num_blocks = num_blocks;
    p.count = expert_count;
    p.offset = expert_offset;
    p.route_slot = route_slot;
    p.status = device_status_ptr();
    p.zero_ptr = zero_ptr;
    p.zero_n = zero_ptr ? zero_n : 0;
    p.skip_pads = skip_pads ? 1 : 0;
    p.kept_slot = kept_slot;
    p.n_kept = n_kept;
    if (path == MOE_ROUTE_AUTO && R > 0 && R <= kWarpMaxRoutes) {
        // a handful of routes (decode batches of a few tokens): one warp sorts them
        Launch L(dim3(1), dim3(kWarpThreads), 0, stream, pdl);
        cudaError_t e = cudaLaunchKernelEx(&L.cfg, k_route_warp, p);
        if (e != cudaSuccess) { set_error("route warp launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
        return MOE_OK;
    }
    const bool single = route_single_cta(R, E_local, path) && R > 0;
    if (single) {
        if (R > kSingleMaxRoutes || E_local > kSingleMaxExperts) {
            set_error("moe_route_prepare: the single-CTA path takes at most %d routes and %d experts",
                      kSingleMaxRoutes, kSingleMaxExperts);
            return MOE_ERR_ARG;
        }
        // with an expert map, the compacting variant when its shared memory fits comfortably
        p.compact = expert_map && single_smem_bytes(R, E, E_local, true) <= kCompactMaxSmem ? 1 : 0;
        // Fewer warps for fewer routes: the per-warp histograms, their per-expert column scan
        // and every CTA barrier shrink with the warp count.  Measured on GB300 (graph-replayed
        // layer, interleaved A/B) against 32 warps: decode M=8 -0.9 us, M=16 -1.7, M=32 -1.2 with
        // 8 warps up to 256 routes; M=64 -1.2 with 16 up to 512; 4 warps up to 128 routes were
        // slower than 8.
        const int W = R <= 256 ? 8 : R <= 512 ? 16 : kSingleWarps;
        const size_t smem = single_smem_bytes(R, E, E_local, p.compact != 0, W);
        const void* kfn = W == 8 ? reinterpret_cast<const void*>(k_route_single<8>)
                        : W == 16 ? reinterpret_cast<const void*>(k_route_single<16>)
                                  : reinterpret_cast<const void*>(k_route_single<kSingleWarps>);
        if (!ensure_smem(kfn, static_cast<int>(smem))) {
            set_error("route single: shared-memory limit %zu refused", smem);
            return MOE_ERR_LAUNCH;
        }
        Launch L(dim3(1), dim3(W * 32), smem, stream, pdl);
        cudaError_t e = W == 8 ? cudaLaunchKernelEx(&L.cfg, k_route_single<8>, p)
                      : W == 16 ? cudaLaunchKernelEx(&L.cfg, k_route_single<16>, p)
                                : cudaLaunchKernelEx(&L.cfg, k_route_single<kSingleWarps>, p);
        if (e != cudaSuccess) { set_error("route single launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
        return MOE_OK;
    }
    if (R == 0) {
        // nothing to sort: zero counts and offsets, no blocks (B_cap is 0)
        cudaError_t e = cudaMemsetAsync(expert_count, 0, sizeof(int32_t) * E_local, stream);
        if (e == cudaSuccess && expert_offset)
            e = cudaMemsetAsync(expert_offset, 0, sizeof(int32_t) * (E_local + 1), stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(num_blocks, 0, sizeof(int32_t), stream);
        if (e == cudaSuccess && zero_ptr && zero_n > 0)
            e = cudaMemsetAsync(zero_ptr, 0, sizeof(uint32_t) * zero_n, stream);
        if (e != cudaSuccess) { set_error("route memset: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
        return MOE_OK;
    }
    const size_t need = route_workspace_bytes(R, E_local, block_m);
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
        set_error("moe_route_prepare: multi-CTA path needs %zu bytes of 256-byte aligned workspace (got %zu)",
                  need, ws_bytes);
        return MOE_ERR_WORKSPACE;
    }
    p.warps = multi_warps(E_local);
    p.chunk = p.warps * 32;
    p.nchunks = (R + p.chunk - 1) / p.chunk;
    char* ws = static_cast<char*>(workspace);
    p.ws_cnt = reinterpret_cast<int32_t*>(ws);
    ws += align256(static_cast<size_t>(p.nchunks) * E_local * 4);
    p.ws_off = reinterpret_cast<int32_t*>(ws);
    ws += align256(static_cast<size_t>(E_local + 1) * 4);
    p.ws_done = reinterpret_cast<unsigned*>(ws);
    // shared-memory limits first: a refusal returns before anything is enqueued
    const size_t smem1 = (static_cast<size_t>(E_local) * 2 + 1 + 33) * 4;
    const size_t ints2 = ((static_cast<size_t>(p.chunk) + E_local) + 3) & ~static_cast<size_t>(3);
    const size_t smem2 = ints2 * 4 + static_cast<size_t>(p.warps) * E_local * 2;
    if (!ensure_smem(reinterpret_cast<const void*>(k_route_count), static_cast<int>(smem1)) ||
        !ensure_smem(reinterpret_cast<const void*>(k_route_scatter), static_cast<int>(smem2))) {
        set_error("route multi: shared-memory limit refused");
        return MOE_ERR_LAUNCH;
    }
    cudaError_t e = cudaMemsetAsync(p.ws_done, 0, sizeof(unsigned), stream);
    if (e != cudaSuccess) { set_error("route memset: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    {
        Launch L(dim3(p.nchunks), dim3(1024), smem1, stream, false);
        e = cudaLaunchKernelEx(&L.cfg, k_route_count, p);
    }
    if (e == cudaSuccess) {
        Launch L(dim3(p.nchunks), dim3(p.warps * 32), smem2, stream, false);
        e = cudaLaunchKernelEx(&L.cfg, k_route_scatter, p);
    }
    if (e != cudaSuccess) { set_error("route multi launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}

}  // namespace moe

extern "C" int moe_block_capacity(int M, int k, int E_local, int block_m) {
    if (M < 0 || k <= 0 || E_local <= 0 || block_m <= 0) return -1;
    const long long R = static_cast<long long>(M) * k;
    const long long cap = (R + block_m - 1) / block_m + std::min<long long>(E_local, R);
    return cap > 0x7FFFFFFFLL ? -1 : static_cast<int>(cap);
}

extern "C" size_t moe_route_prepare_workspace_bytes(int M, int k, int E_local, int block_m) {
    if (M < 0 || k <= 0 || E_local <= 0) return 0;
    return moe::route_workspace_bytes(M * k, E_local, block_m);
}

extern "C" int moe_route_prepare(const int32_t* topk_ids, int M, int k, int E,
                                 const int32_t* expert_map, int E_local, int block_m,
                                 moe_route_path path, int32_t* sorted_idx, int32_t* block_expert,
                                 int32_t* num_blocks, int32_t* expert_count,
                                 int32_t* expert_offset, int32_t* route_slot, void* workspace,
                                 size_t ws_bytes, cudaStream_t stream) {
    moe::clear_error();
    if (!moe::device_is_sm103()) { moe::set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    return moe::launch_route_prepare(topk_ids, M, k, E, expert_map, E_local, block_m, path,
                                     sorted_idx, block_expert, num_blocks, expert_count,
                                     expert_offset, route_slot, workspace, ws_bytes, false, stream);
}

// ---------------------------------------------------------------------------------------------
// Allocation-free variant of the multi-CTA route preparation.
//
// For callers that cannot allocate device memory or hand the library a workspace: the chunk
// histograms, the per-expert slot offsets and the ticket counter live in one file-scope device
// array instead of the caller's workspace.  Every GPU that loads the library keeps this array
// (266,752 bytes) until the process exits.  Limits: at most kNoAllocMaxRoutes routes (M*k) and
// kNoAllocMaxExperts local experts; larger calls are rejected before anything is enqueued.
// ---------------------------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int kNoAllocMaxRoutes = 65536;
constexpr int kNoAllocMaxExperts = 1024;
constexpr int kNoAllocChunk = 1024;  // 32 warps x 32 routes: the scatter CTA size for <= 1536 experts
constexpr int kNoAllocChunks = kNoAllocMaxRoutes / kNoAllocChunk;
constexpr size_t kNoAllocCntInts = static_cast<size_t>(kNoAllocChunks) * kNoAllocMaxExperts;
constexpr size_t kNoAllocOffInts = 1088;  // >= kNoAllocMaxExperts + 1, keeps 256-byte alignment
constexpr size_t kNoAllocInts = kNoAllocCntInts + kNoAllocOffInts + 64;

static __device__ __align__(256) int32_t g_route_noalloc_scratch[kNoAllocInts];

int32_t* g_noalloc_ptr[64] = {nullptr};
std::mutex g_noalloc_mutex;

// Device address of the scratch array on the current device, looked up once per device.
int32_t* noalloc_scratch() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[d]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_route_noalloc_scratch);
        if (e != cudaSuccess) {
            set_error("moe_route_prepare_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            return nullptr;
        }
        g_noalloc_ptr[d] = static_cast<int32_t*>(p);
    }
    return g_noalloc_ptr[d];
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_prepare_noalloc(const int32_t* topk_ids, int M, int k, int E,
                                         const int32_t* expert_map, int E_local, int block_m,
                                         int32_t* sorted_idx, int32_t* block_expert,
                                         int32_t* num_blocks, int32_t* expert_count,
                                         int32_t* expert_offset, int32_t* route_slot,
                                         cudaStream_t stream) {
    using namespace moe;
    clear_error();
    if (!device_is_sm103()) { set_error("no sm_103 device is current"); return MOE_ERR_UNSUPPORTED; }
    if (M < 0 || k <= 0 || E <= 0 || E_local <= 0) {
        set_error("moe_route_prepare_noalloc: need M >= 0, k > 0, E > 0, E_local > 0");
        return MOE_ERR_ARG;
    }
    if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128) {
        set_error("moe_route_prepare_noalloc: block_m must be 16, 32, 64 or 128 (got %d)", block_m);
        return MOE_ERR_ARG;
    }
    if (!expert_map && E_local != E) {
        set_error("moe_route_prepare_noalloc: without an expert map E_local must equal E (%d vs %d)", E_local, E);
        return MOE_ERR_EXPERT_SLICE;
    }
    if (expert_map && E_local > E) {
        set_error("moe_route_prepare_noalloc: E_local %d > E %d", E_local, E);
        return MOE_ERR_EXPERT_SLICE;
    }
    if (k > E) { set_error("moe_route_prepare_noalloc: top-k %d > E %d", k, E); return MOE_ERR_ARG; }
    const long long R = static_cast<long long>(M) * k;
    if (R > kNoAllocMaxRoutes || E_local > kNoAllocMaxExperts) {
        set_error("moe_route_prepare_noalloc: at most %d routes (M*k) and %d local experts fit its "
                  "fixed scratch (got %lld routes, %d experts); use moe_route_prepare with a workspace",
                  kNoAllocMaxRoutes, kNoAllocMaxExperts, R, E_local);
        return MOE_ERR_ARG;
    }
    if (!num_blocks || !expert_count || (R > 0 && (!topk_ids || !sorted_idx || !block_expert))) {
        set_error("moe_route_prepare_noalloc: null output or input pointer");
        return MOE_ERR_ARG;
    }
    if (R == 0) {
        cudaError_t e = cudaMemsetAsync(expert_count, 0, sizeof(int32_t) * E_local, stream);
        if (e == cudaSuccess && expert_offset)
            e = cudaMemsetAsync(expert_offset, 0, sizeof(int32_t) * (E_local + 1), stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(num_blocks, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess) { set_error("route memset: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
        return MOE_OK;
    }
    int32_t* scratch = noalloc_scratch();
    if (!scratch) return MOE_ERR_LAUNCH;
    RouteArgs p{};
    p.ids = topk_ids;
    p.R = static_cast<int>(R);
    p.E = E;
    p.map = expert_map;
    p.E_loc = E_local;
    p.bm = block_m;
    p.bm_shift = block_m == 16 ? 4 : block_m == 32 ? 5 : block_m == 64 ? 6 : 7;
    p.B_cap = static_cast<int>((R + block_m - 1) / block_m + std::min<long long>(E_local, R));
    p.sorted_idx = sorted_idx;
    p.block_expert = block_expert;
    p.num_blocks = num_blocks;
    p.count = expert_count;
    p.offset = expert_offset;
    p.route_slot = route_slot;
    p.status = device_status_ptr();
    p.warps = kNoAllocChunk / 32;
    p.chunk = kNoAllocChunk;
    p.nchunks = static_cast<int>((R + kNoAllocChunk - 1) / kNoAllocChunk);
    p.ws_cnt = scratch;                                       // [nchunks][E_local]
    p.ws_off = scratch + kNoAllocCntInts;                     // [E_local + 1]
    p.ws_done = reinterpret_cast<unsigned*>(scratch + kNoAllocCntInts + kNoAllocOffInts);
    // shared-memory limits first: a refusal returns before anything is enqueued
    const size_t smem1 = (static_cast<size_t>(E_local) * 2 + 1 + 33) * 4;
    const size_t ints2 = ((static_cast<size_t>(p.chunk) + E_local) + 3) & ~static_cast<size_t>(3);
    const size_t smem2 = ints2 * 4 + static_cast<size_t>(p.warps) * E_local * 2;
    if (!ensure_smem(reinterpret_cast<const void*>(k_route_count), static_cast<int>(smem1)) ||
        !ensure_smem(reinterpret_cast<const void*>(k_route_scatter), static_cast<int>(smem2))) {
        set_error("moe_route_prepare_noalloc: shared-memory limit refused");
        return MOE_ERR_LAUNCH;
    }
    // the ticket counter must start at zero (the array keeps the previous call's contents)
    cudaError_t e = cudaMemsetAsync(p.ws_done, 0, sizeof(unsigned), stream);
    if (e != cudaSuccess) { set_error("route memset: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    {
        Launch L(dim3(p.nchunks), dim3(1024), smem1, stream, false);
        e = cudaLaunchKernelEx(&L.cfg, k_route_count, p);
    }
    if (e == cudaSuccess) {
        Launch L(dim3(p.nchunks), dim3(p.warps * 32), smem2, stream, false);
        e = cudaLaunchKernelEx(&L.cfg, k_route_scatter, p);
    }
    if (e != cudaSuccess) { set_error("moe_route_prepare_noalloc launch: %s", cudaGetErrorString(e)); return MOE_ERR_LAUNCH; }
    return MOE_OK;
}
