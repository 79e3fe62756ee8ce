// smr_align.cu -- moe_align_block_size kernels.
//
// "[ROCm][Kernel] W4A16 MoE prefill: M-aware moe_align block size (1.6x
// TTFT)", Purpose: every touched expert is padded up to a full alignment
// block of A rows; num_tokens_post_padded = sum over touched experts of
// ceil(tokens_e / A) * A. The output order inside an expert is ascending flat
// slot index, so results are deterministic and bit-identical across runs.
//
//  - numel <= kAlignSingleMax: one CTA of 512 threads stages the ids in
//    shared memory and does count, scan, scatter and padding (one launch);
//  - larger inputs, three launches with no inter-CTA waiting, over tiles of
//    >= 1024 slots: per-tile expert counts; for each expert the tiles' starts
//    inside it (a prefix over tiles) and its total; then per tile the padded
//    expert offsets (block scan of the totals), the stable scatter of the
//    tile's slots, and the padding rows and block owners of a share of the
//    experts;
//  - behind the tcgen05 route the counts come from the route's epilogue (one
//    tile per 64 token rows), and the scatter ranks a slot among its
//    expert's slots by the tile rows that hold the expert (each row holds an
//    expert at most once).
#include "smr_device.cuh"
#include "smr_launch.h"

namespace smr {

constexpr int kAlignThreads = 512;
constexpr int kAlignWarps = kAlignThreads / 32;

// The expert the align files slot i under: its id e, or behind an EPLB remap
// the physical replica of logical expert e that token i / width uses,
// map[e * R + (i / width) mod count[e]]. A logical id, replica count or
// physical id out of range gives -1, which the callers skip and flag as a
// bad id.
__device__ __forceinline__ int align_expert_of(const AlignLaunch &a, int e, int i) {
    if (a.map == nullptr) return e;
    if ((unsigned)e >= (unsigned)a.E_log) return -1;
    const int c = __ldg(a.map_count + e);
    if (c < 1 || c > a.map_R) return -1;
    const int p = __ldg(a.map + (int64_t)e * a.map_R + (i / a.width) % c);
    return (unsigned)p < (unsigned)a.E_al ? p : -1;
}

__global__ void __launch_bounds__(kAlignThreads) align_single_kernel(const AlignLaunch a) {
    extern __shared__ __align__(16) int sm[];
    griddep_launch_dependents();  // the next kernel may launch; it waits for this grid
    griddep_wait();  // the ids come from the previous kernel
    uint32_t *err = &reinterpret_cast<WsHeader *>(a.hdr)->error;
    int *ids = sm;  // [kAlignSingleMax] staged ids
    AlignSmem s = align_carve(sm + kAlignSingleMax, a.E_al);
    stage_ids(ids, a.ids, a.numel);
    if (a.map != nullptr) {  // EPLB: file each slot under its physical replica
        for (int i = threadIdx.x; i < a.numel; i += blockDim.x) ids[i] = align_expert_of(a, ids[i], i);
        __syncwarp();
        __syncthreads();
    }
    align_count(ids, a.numel, a.E_al, s, err);
    const int npp = align_offsets(s.cnt, a.E_al, a.A, s);
    align_scatter(ids, a.numel, a.E_al, 0, s, false, a.sorted, a.sorted_cap, err);
    align_fill(a.A, a.E_al, s.cnt, s, a.numel, a.sorted, a.sorted_cap, a.expert_ids, a.expert_cap, err,
               threadIdx.x, blockDim.x);
    if (threadIdx.x == 0) *a.npp = npp;
}

// ---- multi-CTA path: count, scan over tiles, scatter ----------------------

constexpr int kTileThreads = 256;
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kTileSub = kTileWarps * 128;  // slots per sub-chunk of the scatter
constexpr int kMaxExpertsAl = 1025;
static_assert(kAlignMinTile % kTileSub == 0, "tiles are whole sub-chunks");

// 1. Per-tile expert counts (shared-memory histogram), four loads in flight
//    per thread; ids outside [0, E_al) are skipped and flagged.
__global__ void __launch_bounds__(kTileThreads) align_tile_count_kernel(const AlignLaunch a, int tile) {
    extern __shared__ int cnt[];
    uint32_t *err = &reinterpret_cast<WsHeader *>(a.hdr)->error;
    const int tid = threadIdx.x;
    griddep_launch_dependents();
    griddep_wait();  // the ids come from the previous kernel
    for (int e = tid; e < a.E_al; e += kTileThreads) cnt[e] = 0;
    __syncwarp();
    __syncthreads();
    const int beg = blockIdx.x * tile, end = min(beg + tile, a.numel);
    for (int i0 = beg; i0 < end; i0 += 4 * kTileThreads) {
        int v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = __ldcg(a.ids + min(i0 + j * kTileThreads + tid, end - 1));
        if (a.map != nullptr)  // EPLB: count physical replicas
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = align_expert_of(a, v[j], min(i0 + j * kTileThreads + tid, end - 1));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (i0 + j * kTileThreads + tid < end) {
                if ((unsigned)v[j] < (unsigned)a.E_al) atomicAdd(&cnt[v[j]], 1);
                else set_error(err, kErrBadId);
            }
        }
    }
    __syncwarp();
    __syncthreads();
    for (int e = tid; e < a.E_al; e += kTileThreads)
        a.tile_counts[(int64_t)blockIdx.x * a.E_al + e] = cnt[e];
}

// 2. For EPB experts per CTA: every tile's start inside each expert
//    (exclusive prefix over tiles, in tile order) and each expert's total.
//    Thread (expert el, chunk c) adds a contiguous run of tiles; the 32
//    chunk sums of an expert are then scanned by one warp (lane = chunk)
//    with shuffles. Few experts per CTA spread the tile-start stores (256
//    tiles x 513 experts: 525 KB at the large batch) over many SMs: one SM
//    stores only a few bytes per clock.
template <int EPB>
__global__ void __launch_bounds__(EPB * 32) align_tile_scan_kernel(const AlignLaunch a, int ntiles) {
    __shared__ int part[32][EPB + 1];
    __shared__ int tot_s[EPB];
    const int el = threadIdx.x % EPB, c = threadIdx.x / EPB;
    griddep_wait();  // the tile counts come from the previous kernel
    // the next kernel launches only after every CTA got here, so once the
    // previous kernel (and everything before it) has completed: the scatter
    // behind the route reads the route's ids before its own wait
    griddep_launch_dependents();
    const int e = blockIdx.x * EPB + el;
    const int ec = min(e, a.E_al - 1);  // clamped: every load stays in bounds
    const int tpc = (ntiles + 31) / 32;
    const int t0 = min(c * tpc, ntiles), t1 = min(t0 + tpc, ntiles);
    // one batch of 16 loads covers a chunk of up to 16 tiles (up to 512
    // tiles); its values stay in registers for the second pass
    int v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        v[j] = __ldcg(a.tile_counts + (int64_t)min(t0 + j, ntiles - 1) * a.E_al + ec);
    int sum = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) sum += (t0 + j < t1) ? v[j] : 0;
    for (int t = t0 + 16; t < t1; t += 16) {  // longer chunks (more than 512 tiles)
        int w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            w[j] = __ldcg(a.tile_counts + (int64_t)min(t + j, ntiles - 1) * a.E_al + ec);
#pragma unroll
        for (int j = 0; j < 16; ++j) sum += (t + j < t1) ? w[j] : 0;
    }
    part[c][el] = sum;
    __syncthreads();
    {
        // warp w scans expert w's column over the 32 chunks (lane = chunk):
        // exclusive prefix in place, the total aside
        const int w = threadIdx.x >> 5, q = threadIdx.x & 31;
        const int x = part[q][w];
        int inc = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            inc += q >= o ? y : 0;
        }
        part[q][w] = inc - x;
        if (q == 31) tot_s[w] = inc;
    }
    __syncthreads();
    int run = part[c][el];
    const int total = tot_s[el];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (t0 + j < t1 && e < a.E_al) a.tile_base[(int64_t)(t0 + j) * a.E_al + e] = run;
        run += (t0 + j < t1) ? v[j] : 0;
    }
    for (int t = t0 + 16; t < t1; t += 16) {
        int w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            w[j] = __ldcg(a.tile_counts + (int64_t)min(t + j, ntiles - 1) * a.E_al + ec);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (t + j < t1 && e < a.E_al) a.tile_base[(int64_t)(t + j) * a.E_al + e] = run;
            run += (t + j < t1) ? w[j] : 0;
        }
    }
    if (c == 0 && e < a.E_al) a.totals[e] = total;
}
constexpr int kScanExperts = 8;  // experts per scan CTA (256 threads)

// 3. Per tile: padded expert offsets from the totals (block scan, fixed
//    order), then the stable scatter of the tile's slots to
//    off[e] + (tile start in e) + rank inside the tile; each CTA also writes
//    the padding rows and block owners of experts t, t + tiles, ... (one warp
//    per expert, coalesced). The tile is taken in sub-chunks of 1024 slots:
//    warp w owns slots [w*128, w*128 + 128) of a sub-chunk, four per lane,
//    kept in registers with their peer masks between counting and scattering.
__global__ void __launch_bounds__(kTileThreads) align_tile_scatter_kernel(const AlignLaunch a, int tile) {
    extern __shared__ __align__(16) int sm[];
    uint32_t *err = &reinterpret_cast<WsHeader *>(a.hdr)->error;
    const int E_al = a.E_al;
    int *wcnt = sm;                   // [8 warps][E_al] counts, then starts
    int *cum = wcnt + kTileWarps * E_al;  // [E_al] running start of this tile in each expert
    int *tot = cum + E_al;            // [E_al] expert totals
    int *off = tot + E_al;            // [E_al + 1] padded expert offsets
    int *scratch = off + E_al + 1;    // [32]
    const int t = blockIdx.x, ntiles = gridDim.x;
    const int beg = t * tile, n = min(beg + tile, a.numel) - beg;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lt = lanemask_lt();
    griddep_launch_dependents();  // the next kernel may launch; it waits for this grid
    griddep_wait();  // the tile starts and totals come from the previous kernel
    // the first sub-chunk's ids (warp w: slots w*128 + g*32 + lane), this
    // tile's starts and the totals: all loads issued first, one round trip
    auto load_ids = [&](int c0, int (&e4)[4]) {
#pragma unroll
        for (int g = 0; g < 4; ++g) e4[g] = __ldcg(a.ids + beg + min(c0 + warp * 128 + g * 32 + lane, n - 1));
        if (a.map != nullptr)  // EPLB: scatter by physical replica
#pragma unroll
            for (int g = 0; g < 4; ++g)
                e4[g] = align_expert_of(a, e4[g], beg + min(c0 + warp * 128 + g * 32 + lane, n - 1));
    };
    int e4[4];
    load_ids(0, e4);
    constexpr int kPerThread = (kMaxExpertsAl + kTileThreads - 1) / kTileThreads;
    int bse[kPerThread], tt[kPerThread];
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
        const int e = min(threadIdx.x + j * kTileThreads, E_al - 1);
        bse[j] = __ldcg(a.tile_base + (int64_t)t * E_al + e);
        tt[j] = __ldcg(a.totals + e);
    }
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
        const int e = threadIdx.x + j * kTileThreads;
        if (e < E_al) {
            cum[e] = bse[j];
            tot[e] = tt[j];
        }
    }
    __syncwarp();
    __syncthreads();
    AlignSmem s;
    s.off = off;
    s.scratch = scratch;
    const int npp = align_offsets(tot, E_al, a.A, s);
    uint32_t bad = 0;
    for (int c0 = 0; c0 < n; c0 += kTileSub) {
        // the warp's four groups of 32 slots: ids and peer masks
        if (c0 > 0) load_ids(c0, e4);
        uint32_t pm[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int i = c0 + warp * 128 + g * 32 + lane;
            int e = e4[g];
            if (i >= n) e = kNoExpert;
            else if ((unsigned)e >= (unsigned)E_al) {
                set_error(err, kErrBadId);
                e = kNoExpert;
            }
            e4[g] = e;
        }
        for (int q = threadIdx.x; q < kTileWarps * E_al; q += kTileThreads) wcnt[q] = 0;
        __syncwarp();
        __syncthreads();
        int *wc = wcnt + warp * E_al;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            pm[g] = peers_of(e4[g]);
            if (e4[g] != kNoExpert && lane == __ffs(pm[g]) - 1) wc[e4[g]] += __popc(pm[g]);
            __syncwarp();
        }
        __syncthreads();
        // per expert: starts of the warps' runs (after earlier sub-chunks)
        for (int e = threadIdx.x; e < E_al; e += kTileThreads) {
            int run = cum[e];
#pragma unroll
            for (int w = 0; w < kTileWarps; ++w) {
                const int c = wcnt[w * E_al + e];
                wcnt[w * E_al + e] = run;
                run += c;
            }
            cum[e] = run;
        }
        __syncwarp();
        __syncthreads();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int e = e4[g];
            if (e != kNoExpert)
                st_slot(a.sorted, off[e] + wc[e] + __popc(pm[g] & lt), a.sorted_cap,
                        beg + c0 + warp * 128 + g * 32 + lane, bad);
            __syncwarp();
            if (e != kNoExpert && lane == __ffs(pm[g]) - 1) wc[e] += __popc(pm[g]);
            __syncwarp();
        }
        __syncthreads();  // the next sub-chunk clears the counts
    }
    for (int e = t + warp * ntiles; e < E_al; e += kTileWarps * ntiles) {
        const int c = tot[e];
        if (c == 0) continue;  // warp-uniform
        const int o0 = off[e], o1 = off[e + 1];
        for (int b = o0 / a.A + lane; b < o1 / a.A; b += 32) st_slot(a.expert_ids, b, a.expert_cap, e, bad);
        for (int q = o0 + c + lane; q < o1; q += 32) st_slot(a.sorted, q, a.sorted_cap, a.numel, bad);
        __syncwarp();
    }
    report_bad_slots(bad, err);
    if (t == 0 && threadIdx.x == 0) *a.npp = npp;
}

// 3'. Behind the tcgen05 route, whose tiles are kTcCountRows token rows of
//    `width` slots with distinct experts in each row: the rank of a slot
//    among its expert's slots in the tile is the number of earlier rows of
//    the tile that hold the expert, read from a per-expert 64-bit mask of
//    rows (shared-memory atomicOr). Then as above: padded offsets, the
//    scatter to off[e] + (tile start in e) + rank, and the padding rows and
//    block owners of a share of the experts.
constexpr int kRowsMaxSlots = 8;  // slots per thread: kTcCountRows * 32 / kTileThreads
static_assert(kTcCountRows == 64, "two mask words per expert");
static_assert(kTcCountRows * 32 <= kRowsMaxSlots * kTileThreads, "a tile of width 32");
__global__ void __launch_bounds__(kTileThreads) align_rows_scatter_kernel(const AlignLaunch a, int width) {
    extern __shared__ __align__(16) int sm[];
    uint32_t *err = &reinterpret_cast<WsHeader *>(a.hdr)->error;
    const int E_al = a.E_al, tid = threadIdx.x;
    uint32_t *mask = reinterpret_cast<uint32_t *>(sm);  // [E_al][2] the tile's rows holding each expert
    int *base = sm + 2 * E_al;                          // [E_al] this tile's start inside each expert
    int *tot = base + E_al;                             // [E_al] expert totals
    int *off = tot + E_al;                              // [E_al + 1] padded expert offsets
    int *scratch = off + E_al + 1;                      // [32]
    const int t = blockIdx.x, ntiles = gridDim.x, warp = tid >> 5, lane = tid & 31;
    const int tile = kTcCountRows * width;
    const int beg = t * tile, n = min(beg + tile, a.numel) - beg;
    griddep_launch_dependents();  // the next kernel may launch; it waits for this grid
    // The ids are the route's: the scan before this kernel let it launch only
    // after waiting for the route, so they are complete already, and the
    // per-expert row masks are built before waiting for the scan
    int ev[kRowsMaxSlots];
#pragma unroll
    for (int j = 0; j < kRowsMaxSlots; ++j) ev[j] = __ldcg(a.ids + beg + min(tid + j * kTileThreads, n - 1));
    for (int q = tid; q < 2 * E_al; q += kTileThreads) mask[q] = 0u;
    __syncthreads();
    int rw[kRowsMaxSlots];  // the slot's row in the tile, or -1
#pragma unroll
    for (int j = 0; j < kRowsMaxSlots; ++j) {
        const int i = tid + j * kTileThreads;
        const bool in = i < n, ok = in && (unsigned)ev[j] < (unsigned)E_al;
        if (in && !ok) set_error(err, kErrBadId);
        rw[j] = ok ? i / width : -1;
        if (ok) atomicOr(&mask[2 * ev[j] + (rw[j] >> 5)], 1u << (rw[j] & 31));
    }
    griddep_wait();  // the tile starts and totals come from the scan
    constexpr int kPerThread = (kMaxExpertsAl + kTileThreads - 1) / kTileThreads;
    int bse[kPerThread], tt[kPerThread];
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
        const int e = min(tid + j * kTileThreads, E_al - 1);
        bse[j] = __ldcg(a.tile_base + (int64_t)t * E_al + e);
        tt[j] = __ldcg(a.totals + e);
    }
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
        const int e = tid + j * kTileThreads;
        if (e < E_al) {
            base[e] = bse[j];
            tot[e] = tt[j];
        }
    }
    __syncthreads();  // base and tot (read by align_offsets) and the masks are complete
    AlignSmem s;
    s.off = off;
    s.scratch = scratch;
    const int npp = align_offsets(tot, E_al, a.A, s);  // ends with a CTA barrier: the masks are complete
    uint32_t bad = 0;
#pragma unroll
    for (int j = 0; j < kRowsMaxSlots; ++j) {
        if (rw[j] >= 0) {
            const int e = ev[j], r = rw[j];
            const uint32_t m0 = mask[2 * e], m1 = mask[2 * e + 1];
            const int rank = r < 32 ? __popc(m0 & ((1u << r) - 1u))
                                    : __popc(m0) + __popc(m1 & ((1u << (r - 32)) - 1u));
            st_slot(a.sorted, off[e] + base[e] + rank, a.sorted_cap, beg + tid + j * kTileThreads, bad);
        }
    }
    __syncwarp();
    for (int e = t + warp * ntiles; e < E_al; e += kTileWarps * ntiles) {
        const int c = tot[e];
        if (c == 0) continue;  // warp-uniform
        const int o0 = off[e], o1 = off[e + 1];
        for (int b = o0 / a.A + lane; b < o1 / a.A; b += 32) st_slot(a.expert_ids, b, a.expert_cap, e, bad);
        for (int q = o0 + c + lane; q < o1; q += 32) st_slot(a.sorted, q, a.sorted_cap, a.numel, bad);
        __syncwarp();
    }
    report_bad_slots(bad, err);
    if (t == 0 && tid == 0) *a.npp = npp;
}

// Once per kernel and device: the dynamic shared-memory limit and the largest
// shared-memory carveout. Every kernel of the library asks for the same
// carveout, so consecutive launches (route, then align) do not reconfigure
// the SMs' L1/shared split in between.
static cudaError_t configure(const void *kern, int slot, size_t bytes) {
    static std::atomic<bool> done[5][kMaxDevices];
    return once_per_device(done[slot], [kern, bytes](int) {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        return r;
    });
}

// A launch that may overlap the end of the previous kernel in the stream
// (programmatic stream serialization); the kernel waits for it with
// griddep_wait() before reading its output.
template <typename... Args>
static cudaError_t launch_dependent(void (*kern)(Args...), int grid, int block, size_t smem,
                                    cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_align(const AlignLaunch &a, cudaStream_t stream) {
    cudaError_t e;
    if (a.numel <= kAlignSingleMax && a.counted_tile == 0) {
        const size_t smem = (size_t)(kAlignSingleMax + align_smem_words(kAlignWarps, a.E_al)) * 4;
        const size_t smem_max = (size_t)(kAlignSingleMax + align_smem_words(kAlignWarps, 1025)) * 4;
        if ((e = configure((const void *)align_single_kernel, 0, smem_max)) != cudaSuccess) return e;
        return launch_dependent(align_single_kernel, 1, kAlignThreads, smem, stream, a);
    }
    int tile, ntiles;
    if (a.counted_tile > 0) {  // counts written by the route, one tile per route CTA
        tile = a.counted_tile;
        ntiles = (a.numel + tile - 1) / tile;
    } else {
        tile = align_tile_size(a.numel);
        ntiles = align_num_tiles(a.numel);
        if ((e = configure((const void *)align_tile_count_kernel, 2, (size_t)kMaxExpertsAl * 4)) !=
            cudaSuccess)
            return e;
        e = launch_dependent(align_tile_count_kernel, ntiles, kTileThreads, (size_t)a.E_al * 4,
                             stream, a, tile);
        if (e != cudaSuccess) return e;
    }
    if ((e = configure((const void *)align_tile_scan_kernel<kScanExperts>, 3, 0)) != cudaSuccess) return e;
    e = launch_dependent(align_tile_scan_kernel<kScanExperts>, (a.E_al + kScanExperts - 1) / kScanExperts,
                         kScanExperts * 32, 0, stream, a, ntiles);
    if (e != cudaSuccess) return e;
    if (a.counted_tile > 0) {  // route tiles: kTcCountRows rows of counted_tile / kTcCountRows slots
        const size_t smem = (size_t)(5 * a.E_al + 1 + 32) * 4;
        const size_t smem_max = (size_t)(5 * kMaxExpertsAl + 1 + 32) * 4;
        if ((e = configure((const void *)align_rows_scatter_kernel, 4, smem_max)) != cudaSuccess) return e;
        return launch_dependent(align_rows_scatter_kernel, ntiles, kTileThreads, smem, stream, a,
                                a.counted_tile / kTcCountRows);
    }
    const size_t smem = (size_t)((kTileWarps + 3) * a.E_al + 1 + 32) * 4;
    const size_t smem_max = (size_t)((kTileWarps + 3) * kMaxExpertsAl + 1 + 32) * 4;
    if ((e = configure((const void *)align_tile_scatter_kernel, 1, smem_max)) != cudaSuccess) return e;
    return launch_dependent(align_tile_scatter_kernel, ntiles, kTileThreads, smem, stream, a, tile);
}

}  // namespace smr
