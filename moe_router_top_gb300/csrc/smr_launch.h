// smr_launch.h -- internal launcher interface between the C-ABI layer
// (smr_api.cpp) and the kernel translation units. Host-only types.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace smr {

// Gate rows split across CTAs, last CTA (ticket) does top-k [+ align].
struct SmallRouteLaunch {
    const uint16_t *x;
    int64_t ld;
    const uint16_t *w;
    const uint16_t *ws;
    const float *bias;
    int M, H, E, S, k;
    float scale;
    int32_t *ids;
    float *wts;
    uint16_t *logits_out;
    float *scratch;        // workspace: [M][E+S] fp32 gate logits
    void *hdr;             // workspace header (WsHeader)
    // fused align (sorted == nullptr: route only)
    int A;
    int32_t *sorted;
    int32_t *expert_ids;
    int32_t *npp;
};
constexpr int kSmallMaxM = 16;
// Number of K ranges the gate rows are split into (the CTAs of one cluster);
// the scratch holds M * (E + S) fp32 gate logits.
int small_route_k_ranges(int E, int S, int H);
cudaError_t launch_small_route(const SmallRouteLaunch &a, cudaStream_t stream);
// Fixed scratch in device memory (no allocation): capacity, and its device
// address for the current device (set up on first use per device).
constexpr size_t kStaticScratchBytes = 256 * 1024;
cudaError_t static_scratch(void **ptr);

// tcgen05 GEMM with the top-k fused into the epilogue.
struct TcRouteLaunch {
    const uint16_t *x;
    int64_t ld;
    const uint16_t *w;
    const uint16_t *ws;
    const float *bias;
    int M, H, E, S, k;
    float scale;
    int32_t *ids;
    float *wts;
    uint16_t *logits_out;
    void *hdr;
};
// Returns cudaErrorNotSupported when the shape is outside the tcgen05 path.
bool tc_route_supported(int H, int E, int k, int S);
cudaError_t launch_tc_route(const TcRouteLaunch &a, cudaStream_t stream);

// moe_align_block_size.
struct AlignLaunch {
    const int32_t *ids;
    int numel;
    int E_al;
    int A;
    int32_t *sorted;
    int32_t *expert_ids;
    int32_t *npp;
    void *hdr;
    int32_t *tile_counts;  // workspace for the multi-CTA path
};
constexpr int kAlignSingleMax = 8192;   // numel handled by one CTA
constexpr int kAlignTile = 8192;        // slots per CTA in the multi-CTA path
inline int align_num_tiles(int numel) { return (numel + kAlignTile - 1) / kAlignTile; }
cudaError_t launch_align(const AlignLaunch &a, cudaStream_t stream);

}  // namespace smr
