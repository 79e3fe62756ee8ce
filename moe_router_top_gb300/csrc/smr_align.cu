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
//  - larger inputs: align_hist_kernel writes per-tile expert counts to the
//    workspace, then align_scatter_kernel (one CTA per tile) derives the
//    global segment offsets from all tile counts (a short fixed-order loop),
//    scatters its tile and writes its share of padding rows and block expert
//    ids (two launches, no inter-CTA waiting).
#include "smr_device.cuh"
#include "smr_launch.h"

namespace smr {

constexpr int kAlignThreads = 512;
constexpr int kAlignWarps = kAlignThreads / 32;

__global__ void __launch_bounds__(kAlignThreads) align_single_kernel(const AlignLaunch a) {
    extern __shared__ __align__(16) int sm[];
    uint32_t *err = &reinterpret_cast<WsHeader *>(a.hdr)->error;
    int *ids = sm;  // [kAlignSingleMax] staged ids
    AlignSmem s = align_carve(sm + kAlignSingleMax, a.E_al);
    stage_ids(ids, a.ids, a.numel);
    align_count(ids, a.numel, a.E_al, s, err);
    const int npp = align_offsets(s.cnt, a.E_al, a.A, s);
    align_scatter(ids, a.numel, a.E_al, 0, s, false, a.sorted);
    align_fill(a.A, a.E_al, s.cnt, s, a.numel, a.sorted, a.expert_ids, threadIdx.x, blockDim.x);
    if (threadIdx.x == 0) *a.npp = npp;
}

__global__ void __launch_bounds__(kAlignThreads) align_hist_kernel(const AlignLaunch a) {
    extern __shared__ int cnt[];
    constexpr int kPer = kAlignTile / kAlignThreads;  // ids per thread
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t *err = &reinterpret_cast<WsHeader *>(a.hdr)->error;
    for (int e = threadIdx.x; e < a.E_al; e += blockDim.x) cnt[e] = 0;
    const int beg = blockIdx.x * kAlignTile, end = min(beg + kAlignTile, a.numel);
    // every load of the tile is issued before the first is used (addresses
    // clamped into the tile, out-of-tile lanes masked afterwards)
    int v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int i = beg + j * kAlignThreads + warp * 32 + lane;
        v[j] = __ldg(a.ids + min(i, end - 1));
    }
    __syncwarp();
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int i = beg + j * kAlignThreads + warp * 32 + lane;
        if (i < end) {
            if ((unsigned)v[j] < (unsigned)a.E_al) atomicAdd(&cnt[v[j]], 1);
            else set_error(err, kErrBadId);
        }
    }
    __syncwarp();
    __syncthreads();
    for (int e = threadIdx.x; e < a.E_al; e += blockDim.x)
        a.tile_counts[(int64_t)blockIdx.x * a.E_al + e] = cnt[e];
}

__global__ void __launch_bounds__(kAlignThreads) align_scatter_kernel(const AlignLaunch a) {
    extern __shared__ __align__(16) int sm[];
    uint32_t *err = &reinterpret_cast<WsHeader *>(a.hdr)->error;
    int *ids = sm;  // [kAlignTile] this tile's ids
    AlignSmem s = align_carve(sm + kAlignTile, a.E_al);
    const int t = blockIdx.x, ntiles = gridDim.x;
    const int beg = t * kAlignTile, n = min(beg + kAlignTile, a.numel) - beg;
    stage_ids(ids, a.ids + beg, n);
    align_count(ids, n, a.E_al, s, err);  // per-warp starts inside this tile
    // global per-expert totals and this tile's offset inside each expert, from
    // all tiles' counts (fixed order; sixteen loads in flight per thread)
    for (int e = threadIdx.x; e < a.E_al; e += blockDim.x) {
        int base = 0, tot = 0;
        for (int u0 = 0; u0 < ntiles; u0 += 16) {
            int c[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)  // clamped addresses: all 16 loads in flight
                c[j] = __ldg(a.tile_counts + (int64_t)min(u0 + j, ntiles - 1) * a.E_al + e);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                c[j] = (u0 + j < ntiles) ? c[j] : 0;
                base += (u0 + j < t) ? c[j] : 0;
                tot += c[j];
            }
        }
        s.base[e] = base;
        s.cnt[e] = tot;
    }
    __syncwarp();
    __syncthreads();
    const int npp = align_offsets(s.cnt, a.E_al, a.A, s);
    align_scatter(ids, n, a.E_al, beg, s, true, a.sorted);
    align_fill(a.A, a.E_al, s.cnt, s, a.numel, a.sorted, a.expert_ids,
               threadIdx.x * ntiles + t, ntiles * blockDim.x);
    if (t == 0 && threadIdx.x == 0) *a.npp = npp;
}

static cudaError_t set_smem(const void *kern, size_t bytes) {
    static bool done[3][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    int slot = kern == (const void *)align_single_kernel ? 0
             : kern == (const void *)align_scatter_kernel ? 1 : 2;
    if (dev < 64 && !done[slot][dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bytes);
        if (e != cudaSuccess) return e;
        done[slot][dev] = true;
    }
    return cudaSuccess;
}

cudaError_t launch_align(const AlignLaunch &a, cudaStream_t stream) {
    const size_t smem = (size_t)(kAlignTile + align_smem_words(kAlignWarps, a.E_al)) * 4;
    const size_t smem_max = (size_t)(kAlignTile + align_smem_words(kAlignWarps, 1025)) * 4;
    cudaError_t e;
    if (a.numel <= kAlignSingleMax) {
        if ((e = set_smem((const void *)align_single_kernel, smem_max)) != cudaSuccess) return e;
        align_single_kernel<<<1, kAlignThreads, smem, stream>>>(a);
        return cudaGetLastError();
    }
    const int ntiles = align_num_tiles(a.numel);
    align_hist_kernel<<<ntiles, kAlignThreads, (size_t)a.E_al * 4, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = set_smem((const void *)align_scatter_kernel, smem_max)) != cudaSuccess) return e;
    align_scatter_kernel<<<ntiles, kAlignThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace smr
