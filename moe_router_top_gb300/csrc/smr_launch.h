// smr_launch.h -- internal launcher interface between the C-ABI layer
// (smr_api.cpp) and the kernel translation units. Host-only types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace smr {

constexpr int kMaxDevices = 64;

// Per-device one-time set-up (kernel attributes, the fixed scratch array):
// set_up(dev) runs with `dev` current the first time a caller reaches it on
// that device, exactly once even when host threads race (a mutex guards the
// first calls; later calls see the flag without locking). A failure is
// returned and the set-up is tried again by the next call.
template <typename F>
inline cudaError_t once_per_device(std::atomic<bool> (&done)[kMaxDevices], F &&set_up) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = set_up(dev);
    if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
    return e;
}

// Failure-injection hook for tests (smr_test_force_wait_timeout): which
// bounded wait is made to wait for something nothing provides, and its
// limit. Read once per launch into the kernel parameters.
enum StallSite : int { kStallNone = 0, kStallSmallTail = 1, kStallTcMerge = 2 };
struct StallHook {
    int site;
    long long limit;
};
StallHook stall_hook();

// Gate rows split across CTAs; the last row group's leader collects the tagged
// selection keys and does the top-k [+ align].
struct SmallRouteLaunch {
    const uint16_t *x;
    int64_t ld;
    const uint16_t *w;
    const uint16_t *ws;
    const float *bias;
    int M, H, E, S, k;
    float scale;
    int renorm;       // 1: weights renormalised over the top-k; 0: the E-expert softmax's
    int shared_bf16;  // 1: the shared logit is rounded to bf16 before the sigmoid
    int32_t *ids;
    float *wts;
    uint16_t *logits_out;
    unsigned long long *scratch;  // workspace: [M][E] tagged selection keys of the routed logits
    void *hdr;             // workspace header (WsHeader)
    // fused align (sorted == nullptr: route only)
    int A;
    int32_t *sorted;
    int32_t *expert_ids;
    int32_t *npp;
    int64_t sorted_cap, expert_cap;  // output array lengths (every write is checked)
    // failure-injection test hook: the tail polls for a tag no row group
    // writes, giving up after stall_limit reloads
    int stall;
    long long stall_limit;
    // optional: the hidden states as e4m3 codes [M][H] with one fp32 scale
    // per 128 elements [M][H / 128] (H % 128 == 0)
    uint8_t *xq;
    float *xs;
};
constexpr int kSmallMaxM = 16;
// Number of K ranges the gate rows are split into (the CTAs of one cluster);
// the scratch holds the M * E tagged selection keys of the routed logits
// (8 bytes each).
int small_route_k_ranges(int E, int S, int H);
cudaError_t launch_small_route(const SmallRouteLaunch &a, cudaStream_t stream);
// Fixed scratch in device memory (no allocation): capacity, and its device
// address for the current device (set up on first use per device, thread-safe).
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
    int renorm;       // as in SmallRouteLaunch
    int shared_bf16;
    int32_t *ids;
    float *wts;
    uint16_t *logits_out;
    void *hdr;
    // optional (align fused behind the route): expert counts of every
    // kTcCountRows-row tile, [ceil(M / kTcCountRows)][E + S]
    int32_t *tile_counts;
    // failure-injection test hook: the merge of the two column halves waits
    // on a barrier nothing arrives on, giving up after stall_limit SM cycles
    int stall;
    long long stall_limit;
    // logits-only launch (the route for E > 512 or E % 32 != 0): the gate
    // rows [col0, col0 + E) (w, bias already offset to row col0) are
    // computed and written, rounded to bf16 with the bias, into
    // logits_ws[M][ld_logits] at column col0 (columns past E up to the next
    // multiple of 32: -inf); the shared logit (ws != nullptr) into s_out[M].
    // k, ids, wts, logits_out and tile_counts are then unused.
    bool logits_only;
    int col0;
    uint16_t *logits_ws;
    int64_t ld_logits;
    float *s_out;
    // optional: the hidden states as e4m3 codes [M][H] with one fp32 scale
    // per 128 elements [M][H / 128] (H % 128 == 0)
    uint8_t *xq;
    float *xs;
    // optional: the align fused into the route (fa_sorted != nullptr; at
    // most kFusedAlignMax ids): the last CTA to finish aligns them
    int fa_A;
    int32_t *fa_sorted, *fa_eids, *fa_npp;
    int64_t fa_sorted_cap, fa_eids_cap;
};
constexpr int kTcTileRows = 128;   // token rows per CTA of the tcgen05 route
constexpr int kTcCountRows = 64;   // token rows per align tile counted by the route
// Returns cudaErrorNotSupported when the shape is outside the tcgen05 path.
bool tc_route_supported(int H, int E, int k, int S);
cudaError_t launch_tc_route(const TcRouteLaunch &a, cudaStream_t stream);
// Gate columns per logits-only launch, and the workspace row stride (elements)
// of the logits of E experts.
constexpr int kTcRangeCols = 512;
inline int64_t generic_logits_ld(int E) { return (E + 31) / 32 * 32; }

// Top-k + softmax + shared slot of every token row from the logits a
// logits-only route wrote (one warp per row).
struct SelectLaunch {
    const uint16_t *logits;  // [M][ld] bf16 bits, -inf past E
    int64_t ld;
    const float *s;          // [M] shared logit (S == 1)
    int M, E, S, k;
    int renorm, shared_bf16;
    float scale;
    int32_t *ids;
    float *wts;
    uint16_t *logits_out;    // optional [M][E]
};
cudaError_t launch_select(const SelectLaunch &a, cudaStream_t stream);
// A 2-D bf16 tensor map with the 128-byte swizzle (rows of row_bytes; boxes
// of box_inner x box_outer elements); false if it cannot be encoded.
bool make_tma_map_2d(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

// The consumer expert GEMM over the align's output: for every block b of A
// rows of sorted_token_ids below num_tokens_post_padded, expert
// expert_ids[b]'s [N, H] weights against the gathered hidden-state rows;
// out[slot][N] fp32 for every routed slot (padding rows are not written).
struct ExpertGemmLaunch {
    const uint16_t *x;
    int64_t ld;
    int width, H, N, A, num_experts;
    int64_t numel, max_blocks;
    const uint16_t *w;       // [num_experts][N][H]
    const int32_t *sorted, *eids, *npp;
    float *out;
    void *hdr;               // workspace header (sticky error word)
};
cudaError_t launch_expert_gemm(const ExpertGemmLaunch &a, cudaStream_t stream);

// moe_align_block_size.
struct AlignLaunch {
    const int32_t *ids;
    int numel;
    int E_al;
    int A;
    int32_t *sorted;
    int32_t *expert_ids;
    int32_t *npp;
    int64_t sorted_cap, expert_cap;  // output array lengths (every write is checked)
    void *hdr;
    // multi-CTA path (workspace): [tiles][E_al] counts, [tiles][E_al] each
    // tile's start inside every expert, [E_al] expert totals
    int32_t *tile_counts;
    int32_t *tile_base;
    int32_t *totals;
    // > 0: the tile counts were written by the tcgen05 route (tiles of
    // counted_tile slots); the count launch is skipped
    int counted_tile;
    // optional EPLB remap (map == nullptr: none): the id e of slot i (token
    // i / width) becomes map[e * map_R + (i / width) % map_count[e]]; E_al
    // is then the number of physical experts, E_log that of logical ones
    const int32_t *map;
    const int32_t *map_count;
    int map_R, E_log, width;
};
// numel handled by one CTA: above ~2000 slots the three multi-CTA launches
// measured faster (8184 slots: 33 us in one CTA, 12 us in three launches)
constexpr int kAlignSingleMax = 2048;
// route_align behind a tcgen05 route over at most this many slots aligns in
// the route's last CTA (one launch); above it the route's 64-row tile counts
// feed the scan and the rows scatter, whose first round trip runs under the
// scan (measured per call, E = 128, H = 2048: 26.0 against 27.6 us at 360
// slots, 27.4 against 25.9 at 1152, 30.0 against 25.9 at 1800)
constexpr int kFusedAlignMax = 704;
constexpr int kAlignMinTile = 1024;     // slots per CTA in the multi-CTA path, at least
constexpr int kAlignMaxTiles = 2048;    // tiles, at most (larger inputs take larger tiles)
inline int align_tile_size(int64_t numel) {
    int64_t t = (numel + kAlignMaxTiles - 1) / kAlignMaxTiles;
    if (t < kAlignMinTile) t = kAlignMinTile;
    return (int)((t + kAlignMinTile - 1) / kAlignMinTile * kAlignMinTile);
}
inline int align_num_tiles(int64_t numel) {
    const int64_t t = align_tile_size(numel);
    return (int)((numel + t - 1) / t);
}
// Workspace words of the multi-CTA path over `tiles` tiles.
inline int64_t align_scratch_words_tiles(int64_t tiles, int E_al) { return 2 * tiles * E_al + E_al; }
inline int64_t align_scratch_words(int64_t numel, int E_al) {
    return align_scratch_words_tiles(align_num_tiles(numel), E_al);
}
// Launches of launch_align for these inputs.
inline int align_launches(int64_t numel, bool counted) {
    return counted ? 2 : (numel <= kAlignSingleMax ? 1 : 3);
}
cudaError_t launch_align(const AlignLaunch &a, cudaStream_t stream);

}  // namespace smr
