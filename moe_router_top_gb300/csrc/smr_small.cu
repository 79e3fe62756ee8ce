// smr_small.cu -- single-launch route (+ align) for M <= 16 tokens.
//
// What it computes is the one-launch small-M router of "[AMD] One-launch
// small-M MoE router for Qwen3.5 on gfx950", Modifications: the E+S gate rows
// are computed for all M tokens with fp32 accumulation across CTAs; the routed
// logits are rounded to bf16; one CTA then selects the top-k with the lowest
// id winning ties, applies softmax + renormalisation, writes the shared
// slot (E, sigmoid(s) * scale) and, when
// asked, runs moe_align_block_size on the M*(k+S) ids it just produced
// ("[ROCm][Kernel] W4A16 MoE prefill: M-aware moe_align block size",
// Purpose) -- all in one launch.
//
// GB300 design:
//  - the gate stream is HBM-bound (4 MiB at E=512, H=4096). CTA (g, q) owns
//    gate rows [16g, 16g+16) and the q-th of KQ contiguous ranges of 32-wide
//    K slices, so ~130 CTAs (one wave on the SMs) each stream ~32 KB; every
//    thread issues all of its 16-byte loads (gate rows via ld.global.nc, no L1
//    allocation) before the first multiply;
//  - the dot products run on the tensor cores with mma.sync m16n8k16 (bf16 in,
//    fp32 accumulate): 16 gate rows x 8 tokens per instruction. A sum over K
//    does not depend on the order of K, so each thread feeds its own
//    contiguous 8-element chunk straight from its 16-byte loads into the A and
//    B fragments (the same K permutation on both operands), with no shared
//    memory staging;
//  - the KQ CTAs of a row group form a thread-block cluster: each adds its 8
//    warps' partials in a fixed order and stores the sum into a slot in the
//    shared memory of the cluster's first CTA (distributed shared memory),
//    which adds the KQ slots in a fixed order after one cluster barrier and
//    stores the group's final logits -- results are deterministic;
//  - each group leader rounds its logits, stores them as ordered 32-bit
//    selection keys tagged with the call's epoch in one 64-bit word, and
//    writes the shared expert's slot itself; the leader of the last group
//    runs the tail, loading every key word until it carries this call's tag
//    (bounded; no fence, counter or atomic on the hand-off);
//  - the tail is warp-parallel and compact (it runs once per call): one warp
//    per token ranks the keys at or above the k-th largest lane maximum;
//    the align of the few ids places them from per-expert token masks (one
//    block per expert when A >= M) or ranks (expert, position) keys.
#include "smr_device.cuh"
#include "smr_launch.h"

namespace smr {

constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSliceK = 32;           // K elements per slice (two m16n8k16 steps)
constexpr int kMaxSlicesPerWarp = 4;  // slices whose loads are in flight at once
constexpr int kSmallMaxCluster = 8;   // K ranges per row group = CTAs per cluster (portable size)
constexpr int kSmallFrontWords = 4096;  // partials + cluster slots (16 KB), reused by the tail
constexpr int kSmallMaxE = 1024;
// The tail's arrays after the front words: the tokens of each expert (bit m
// for token m, E + S <= 1025 words) and the touched-expert bitmap.
constexpr int kSmallMaskWords = 1028;
constexpr int kSmallBitWords = 36;
// sorted_token_ids staged for one bulk copy (64 KB: npp <= 16384).
constexpr int kSmallSortedWords = 16384;
constexpr int kSmallSmemWords = kSmallFrontWords + kSmallMaskWords + kSmallBitWords + kSmallSortedWords;
static_assert(((kSmallFrontWords + kSmallMaskWords + kSmallBitWords) * 4) % 16 == 0, "16-byte aligned staging");
static_assert(kSmallBitWords % 4 == 0, "bitmap read as uint4");
static_assert(kSmallMaxE + 1 <= kSmallMaskWords && (kSmallMaxE + 32) / 32 <= kSmallBitWords, "mask arrays");
static_assert(kSmallMaxM <= 32, "one bit per token");
static_assert(kSmallWarps * 256 + kSmallMaxCluster * 256 <= kSmallFrontWords, "partials + slots");
// Reloads of a key word that still holds an older tag before the tail gives
// up (each one waits for an L2 round trip: well above a second in all).
constexpr int kSmallPollLimit = 1 << 22;
constexpr int kSmallCandWords = 3072;  // the top-k's per-warp candidate lists, past the align's arrays
static_assert(kSmallMaxM * 32 * 3 + 32 <= kSmallCandWords, "tail arrays");
static_assert(kSmallCandWords + kSmallWarps * 32 <= kSmallFrontWords, "candidate lists");
static_assert(kSmallMaxM * 32 <= 2 * kSmallThreads, "two ranks per thread in the align");

struct SmallParams {
    SmallRouteLaunch a;
    int rows;     // E + S
    int mask_align;  // fused align with A >= M: one block per touched expert
    int KQ;       // K ranges per 16-row group
    int slices;   // ceil(H / 32)
    int per_cta;  // slices per K range
};

// Top-k of one token row in one warp. krow: the token's E selection keys
// (the bf16-rounded logit and the expert id, see make_key) in the low half
// of words whose high half is the call's tag, written by the row groups
// (want: the tag to wait for, at most poll_limit reloads);
// cand_s: 32 words of shared memory owned by this warp.
// Writes ids and weights of the routed slots 0..k-1 to global memory (the
// shared slot k was written by its row group) and the align's
// (expert << 10 | flat slot) keys of all k + S slots to keys_s; with tmask,
// also marks token m in the routed experts' token masks and the
// touched-expert bitmap tbits. The selection itself is warp_topk_keys.
template <int NK>
__device__ __forceinline__ void warp_topk_row(const unsigned long long *krow, uint32_t want,
                                              long long poll_limit, int E, int S,
                                              int k, int renorm, int32_t *ids, float *wts, uint32_t *keys_s,
                                              int flat0,
                                              uint32_t *cand_s, uint32_t *tmask, uint32_t *tbits, int m,
                                              uint32_t *err) {
    const int lane = threadIdx.x & 31;
    // every load issued before the first use; lanes past E read a clamped
    // (valid) element that is masked below. A word carries this call's tag
    // once its row group has stored it: the words still holding another tag
    // than `want` (this call's tag; another one only under the failure-
    // injection hook) are loaded again, at most poll_limit times.
    unsigned long long v[NK];
#pragma unroll
    for (int i = 0; i < NK; ++i) v[i] = ld_relaxed_u64(krow + min(lane + 32 * i, E - 1));
#pragma unroll 1
    for (long long tries = 0;; ++tries) {
        bool ok = true;
#pragma unroll
        for (int i = 0; i < NK; ++i) ok = ok && (uint32_t)(v[i] >> 32) == want;
        if (__all_sync(0xffffffffu, ok)) break;
        if (tries >= poll_limit) {  // warp-uniform: the outputs of this call are not valid
            if (lane == 0) set_error(err, kErrWaitTimeout);
            break;
        }
#pragma unroll
        for (int i = 0; i < NK; ++i)
            if ((uint32_t)(v[i] >> 32) != want) v[i] = ld_relaxed_u64(krow + min(lane + 32 * i, E - 1));
    }
    uint32_t key[NK];
#pragma unroll
    for (int i = 0; i < NK; ++i) key[i] = (lane + 32 * i < E) ? (uint32_t)v[i] : 0u;
    float weight;
    const uint32_t mine = warp_topk_keys<NK>(key, k, renorm, cand_s, weight);
    if (lane < k) {
        const int id = key_id(mine);
        ids[lane] = id;
        wts[lane] = weight;
        keys_s[lane] = ((uint32_t)id << 10) | (uint32_t)(flat0 + lane);  // the align's key
        if (tmask != nullptr) {
            atomicOr(tmask + id, 1u << m);
            atomicOr(tbits + (id >> 5), 1u << (id & 31));
        }
    } else if (S != 0 && lane == k) {
        keys_s[lane] = ((uint32_t)E << 10) | (uint32_t)(flat0 + lane);
    }
    __syncwarp();
}

// moe_align_block_size ("[ROCm][Kernel] W4A16 MoE prefill: M-aware
// moe_align block size", Purpose) for a small batch whose every expert fits
// one block (A >= M: an expert receives at most one id per token), from
// the per-expert token masks and the touched-expert bitmap the top-k filled:
//  - an expert's block is the number of touched experts below it (warp 0
//    scans the popcounts of the <= 36 bitmap words; then one popcount
//    within the expert's word);
//  - an id's place in its block is the number of earlier tokens in its
//    expert's mask (ids of one expert come one per token, so this is the
//    ascending flat order the alignment lists them in);
//  - npp = A * touched experts; every slot of a block past its count holds
//    the sentinel n = M * width.
// The stores of one SM are the bound here (about 7 bytes per clock for
// scattered and 16-byte stores alike), so sorted_token_ids[0, npp) is built
// in shared memory and written by one bulk copy (cp.async.bulk) when it fits
// sbuf and A is a multiple of 4; otherwise the ids and the padding are stored
// directly. sbuf holds the sentinel over [0, min(kSmallSortedWords,
// A * min(E + S, n))) on entry (filled at the kernel's start), which covers
// any npp: the ids are placed into it.
__device__ __forceinline__ void align_masks(const uint32_t *keys_s, int M, int width, int A,
                                            const uint32_t *tmask, const uint32_t *tbits, int *wpre, int *blkcnt,
                                            uint32_t *sbuf, int32_t *sorted, int64_t sorted_cap,
                                            int32_t *expert_ids, int64_t expert_cap, int32_t *npp_out,
                                            uint32_t *err) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // warp 0: touched experts before each bitmap word (an exclusive scan of
    // the words' popcounts; words 32-35 are summed by lane 31) and in all
    if (warp == 0) {
        const int c = __popc(tbits[lane]);
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            inc += lane >= o ? v : 0;
        }
        wpre[lane] = inc - c;
        if (lane == 31) {
            int run = inc;
#pragma unroll
            for (int w = 32; w < kSmallBitWords; ++w) {
                wpre[w] = run;
                run += __popc(tbits[w]);
            }
            wpre[kSmallBitWords] = run;
        }
    }
    __syncwarp();
    __syncthreads();
    const int nblk = wpre[kSmallBitWords];
    const int n = M * width;
    const int npp = nblk * A;
    if (tid == 0) *npp_out = npp;
    const bool bulk = (A & 3) == 0 && (reinterpret_cast<uintptr_t>(sorted) & 15u) == 0 &&
                      npp <= kSmallSortedWords && (int64_t)npp <= sorted_cap;
    uint32_t bad = 0;
#pragma unroll 1
    for (int m = warp; m < M; m += kSmallWarps) {
        if (lane < width) {
            const int i = m * width + lane;
            const int e = (int)(keys_s[i] >> 10), we = e >> 5;
            const uint32_t tm = tmask[e];
            const int j = __popc(tm & ((1u << m) - 1u));
            const int b = wpre[we] + __popc(tbits[we] & ((1u << (e & 31)) - 1u));
            if (bulk) sbuf[b * A + j] = (uint32_t)i;
            else st_slot(sorted, (int64_t)b * A + j, sorted_cap, i, bad);
            if (j == 0) {
                blkcnt[b] = __popc(tm);
                st_slot(expert_ids, b, expert_cap, e, bad);
            }
        }
        __syncwarp();
    }
    if (bulk) {
        // the generic-proxy writes of sbuf become visible to the bulk copy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0 && npp > 0) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                         ::"l"(sorted), "r"(smem_u32(sbuf)), "r"(npp * 4) : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            // the CTA's shared memory must outlive the copy's reads of it
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
        report_bad_slots(bad, err);
        return;
    }
    __syncwarp();
    __syncthreads();
    // direct padding stores: slots j >= the block's count (16-byte stores
    // when A is a multiple of 4, so that four slots never straddle two
    // blocks, and the array is 16-byte aligned)
    const bool pow2 = (A & (A - 1)) == 0;
    const int lgA = __ffs(A) - 1;
    if ((A & 3) == 0 && (reinterpret_cast<uintptr_t>(sorted) & 15u) == 0) {
#pragma unroll 1
        for (int q = tid * 4; q < npp; q += kSmallThreads * 4) {
            const int b = pow2 ? q >> lgA : q / A, j = q - b * A, c = blkcnt[b];
            if (j >= c) {
                st_slot4(sorted, q, sorted_cap, make_int4(n, n, n, n), bad);
            } else if (j + 4 > c) {
                for (int u = c - j; u < 4; ++u) st_slot(sorted, q + u, sorted_cap, n, bad);
            }
        }
    } else {
#pragma unroll 1
        for (int q = tid; q < npp; q += kSmallThreads) {
            const int b = q / A, j = q - b * A;
            if (j >= blkcnt[b]) st_slot(sorted, q, sorted_cap, n, bad);
        }
    }
    report_bad_slots(bad, err);
}

// moe_align_block_size ("[ROCm][Kernel] W4A16 MoE prefill: M-aware
// moe_align block size", Purpose) for the n <= 512 ids of one small batch,
// without a histogram or scan over all experts. keys[i] = (expert << 10) | i
// (written by the top-k; keys[n, n4) = ~0) are unique, and their ascending
// order is the stable expert order the alignment lists ids in, so:
//  1. each id's rank = the number of keys below its key (G = 8, 4, 2 or 1
//     consecutive lanes share one id's count and add it with shuffles), and
//     the sorted keys go to srt[rank];
//  2. every thread takes H ranks (r = tid, tid + 256): a rank starts an
//     expert's run when its expert differs from the previous rank's; the run
//     ends at the next start (ballots of the starts, one 32-bit word per 32
//     ranks); a start carries its run's padded size ceil(cnt / A) * A, whose
//     exclusive prefix over ranks (warp scans plus the totals of the earlier
//     words) is the run's offset in sorted_token_ids; the start writes its
//     blocks' records;
//  3. the CTA writes every slot of the blocks as one flat range, 4 slots per
//     thread and step.
// A single warp's instruction stream, not the amount of work, bounds this at
// these sizes, so every step is spread over all warps.
template <int G>
__device__ __forceinline__ void align_tiny_rank(const uint32_t *keys, int n, int n4, uint32_t *srt) {
    const int tid = threadIdx.x, sub = tid % G, nv = n4 / 4;
#pragma unroll 1
    for (int i0 = 0; i0 < n4; i0 += kSmallThreads / G) {  // one pass when G >= 2
        const int i = i0 + tid / G;
        const uint32_t k = keys[min(i, n4 - 1)];
        int r = 0;
#pragma unroll 4
        for (int j = sub; j < nv; j += G) {
            const uint4 v = reinterpret_cast<const uint4 *>(keys)[j];
            r += (v.x < k) + (v.y < k) + (v.z < k) + (v.w < k);
        }
#pragma unroll
        for (int o = 1; o < G; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
        if (i < n && sub == 0) srt[r] = k;
        __syncwarp();
    }
}

template <int H>
__device__ __forceinline__ void align_tiny(const uint32_t *keys, int n, int A, uint32_t *sm, int32_t *sorted,
                                           int64_t sorted_cap, int32_t *expert_ids,
                                           int64_t expert_cap, int32_t *npp_out, uint32_t *err) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kCap = kSmallMaxM * 32;
    constexpr int NW = kSmallWarps * H;  // 32-rank words
    const int n4 = (n + 3) & ~3;
    uint32_t *srt = sm;                   // [n] keys by rank
    // [nblk] per block: expert (11 bits) | first sorted position << 11 (10
    // bits) | ids in the block << 21 (<= 512)
    uint32_t *binfo = sm + kCap;
    uint32_t *starts = binfo + kCap;                      // [NW] ballots of the run starts
    int *wtot = reinterpret_cast<int *>(starts + 16);     // [NW] padded sizes per word
    if (n4 <= kSmallThreads / 8)
        align_tiny_rank<8>(keys, n, n4, srt);
    else if (n4 <= kSmallThreads / 4)
        align_tiny_rank<4>(keys, n, n4, srt);
    else if (n4 <= kSmallThreads / 2)
        align_tiny_rank<2>(keys, n, n4, srt);
    else
        align_tiny_rank<1>(keys, n, n4, srt);
    __syncthreads();
    const bool pow2 = (A & (A - 1)) == 0;
    const int lgA = __ffs(A) - 1;
    const int nw = (n + 31) >> 5;  // words holding ranks
    uint32_t s[H];
    bool f[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const int r = tid + h * kSmallThreads;
        s[h] = srt[min(r, n - 1)];
        const uint32_t prev = srt[max(min(r, n - 1) - 1, 0)];
        f[h] = r < n && (r == 0 || (s[h] >> 10) != (prev >> 10));
        const uint32_t m = __ballot_sync(0xffffffffu, f[h]);
        if (lane == 0) starts[warp + h * kSmallWarps] = m;
    }
    __syncthreads();
    uint32_t mk[NW];
#pragma unroll
    for (int w = 0; w < NW; w += 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(starts + w);
        mk[w] = v.x; mk[w + 1] = v.y; mk[w + 2] = v.z; mk[w + 3] = v.w;
    }
    int pad[H], cnt[H], inc[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const int wd = warp + h * kSmallWarps, r = tid + h * kSmallThreads;
        // the next run start after rank r: a later bit of this word, else the
        // first start of a later word, else n
        const uint32_t later = lane == 31 ? 0u : starts[wd] & ~((2u << lane) - 1u);
        int nxt = n;
#pragma unroll
        for (int w = NW - 1; w >= 0; --w)
            nxt = (w > wd && w < nw && mk[w] != 0u) ? w * 32 + __ffs(mk[w]) - 1 : nxt;
        nxt = later ? wd * 32 + __ffs(later) - 1 : nxt;
        cnt[h] = nxt - r;
        pad[h] = f[h] ? (pow2 ? ((cnt[h] + A - 1) >> lgA) << lgA : (cnt[h] + A - 1) / A * A) : 0;
        inc[h] = pad[h];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc[h], o);
            inc[h] += lane >= o ? v : 0;
        }
        if (lane == 31) wtot[wd] = inc[h];
    }
    __syncthreads();
    int wt[NW];
#pragma unroll
    for (int w = 0; w < NW; w += 4) {
        const int4 v = *reinterpret_cast<const int4 *>(wtot + w);
        wt[w] = v.x; wt[w + 1] = v.y; wt[w + 2] = v.z; wt[w + 3] = v.w;
    }
    int npp = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) npp += (w < nw) ? wt[w] : 0;
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const int wd = warp + h * kSmallWarps;
        int off = inc[h] - pad[h];
#pragma unroll
        for (int w = 0; w < NW; ++w) off += (w < wd) ? wt[w] : 0;
        if (pad[h]) {
            const int r = tid + h * kSmallThreads;
            const uint32_t e = s[h] >> 10;
            const int b0 = pow2 ? off >> lgA : off / A;
            binfo[b0] = e | ((uint32_t)r << 11) | ((uint32_t)min(A, cnt[h]) << 21);
            for (int u = 1; u * A < pad[h]; ++u)  // an expert with more than A ids
                binfo[b0 + u] = e | ((uint32_t)(r + u * A) << 11) | ((uint32_t)min(A, cnt[h] - u * A) << 21);
        }
    }
    if (tid == 0) *npp_out = npp;
    __syncthreads();
    // the blocks' experts, then every slot of sorted_token_ids: slot u of
    // block b holds the u-th id of its expert's run in the block, or the
    // sentinel n past the run (16-byte stores when A is a multiple of 4 and
    // the array is 16-byte aligned)
    const int nblk = pow2 ? npp >> lgA : npp / A;
    uint32_t bad = 0;
    for (int b = tid; b < nblk; b += kSmallThreads)
        st_slot(expert_ids, b, expert_cap, (int)(binfo[b] & 2047u), bad);
    if ((A & 3) == 0 && (reinterpret_cast<uintptr_t>(sorted) & 15u) == 0) {
#pragma unroll 2
        for (int q = tid * 4; q < npp; q += kSmallThreads * 4) {
            const int b = pow2 ? q >> lgA : q / A, u = q - b * A;
            const uint32_t bi = binfo[b];
            const int bp = (int)((bi >> 11) & 1023u) + u, bc = (int)(bi >> 21) - u;
            int v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = j < bc ? (int)(srt[bp + min(j, bc - 1)] & 1023u) : n;
            st_slot4(sorted, q, sorted_cap, make_int4(v[0], v[1], v[2], v[3]), bad);
        }
    } else {
        for (int q = tid; q < npp; q += kSmallThreads) {
            const int b = q / A, u = q - b * A;
            const uint32_t bi = binfo[b];
            const int bc = (int)(bi >> 21);
            st_slot(sorted, q, sorted_cap,
                    u < bc ? (int)(srt[(int)((bi >> 11) & 1023u) + min(u, bc - 1)] & 1023u) : n, bad);
        }
    }
    report_bad_slots(bad, err);
}

// The hidden states to e4m3 ("Netra Kernel ...", Fusing the activation/
// quantization boundary: one scale per 128 values): the kq-th of KQ CTAs
// takes its share of the 128-element blocks, one warp per (token, block),
// four elements per lane, re-read from L2 (this kernel loaded them already).
// scale = amax / 448 and codes = e4m3(x * (448 / amax)) rounded to nearest
// even and saturated, in fp32; a block of zeros gets scale 0 and zero codes.
__device__ __noinline__ void small_quant_x(const SmallRouteLaunch &p, int kq, int KQ) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = p.H >> 7, b0 = kq * nb / KQ, b1 = (kq + 1) * nb / KQ, per = b1 - b0;
#pragma unroll 1
    for (int j = warp; j < p.M * per; j += kSmallWarps) {
        const int m = j / per, b = b0 + j % per;
        const uint2 v = __ldcg(reinterpret_cast<const uint2 *>(p.x + (int64_t)m * p.ld + b * 128) + lane);
        const float f0 = __uint_as_float(v.x << 16), f1 = __uint_as_float(v.x & 0xFFFF0000u);
        const float f2 = __uint_as_float(v.y << 16), f3 = __uint_as_float(v.y & 0xFFFF0000u);
        // magnitudes are nonnegative floats: their bit patterns order alike
        const float amax = __uint_as_float(__reduce_max_sync(
            0xffffffffu, __float_as_uint(fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3))))));
        uint32_t codes = 0u;
        if (amax > 0.0f) {
            const float inv = 448.0f / amax;
            uint16_t lo, hi;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(f1 * inv), "f"(f0 * inv));
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(f3 * inv), "f"(f2 * inv));
            codes = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        reinterpret_cast<uint32_t *>(p.xq + (int64_t)m * p.H + b * 128)[lane] = codes;
        if (lane == 0) p.xs[(int64_t)m * nb + b] = amax / 448.0f;
    }
}

// NB: blocks of 8 tokens, 1 (M <= 8) or 2 (M <= 16); NK: keys per lane in
// the top-k, 16 (E <= 512) or 32 (E <= 1024) -- one top-k per instance, so
// the tail's code is laid out in the order it runs
template <int NB, int NK>
__global__ void __launch_bounds__(kSmallThreads, 1) small_route_kernel(const SmallParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    const SmallRouteLaunch &p = P.a;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;  // mma fragment coordinates
    const int rows = P.rows;
    const int rg = blockIdx.x / P.KQ;         // row group
    const int kq = (int)cluster_ctarank();    // K range = rank in the group's cluster
    const int row0 = rg * 16;

    // the group leader (rank 0) finishes the group's logits with thread
    // (row r16, token m16); the tail CTA clears its token masks and bitmap
    const int r16 = tid >> 4, m16 = tid & 15;  // 256 threads = 16 rows x 16 tokens
    uint32_t *tmask = reinterpret_cast<uint32_t *>(smem) + kSmallFrontWords;  // [E + S]
    uint32_t *tbits = tmask + kSmallMaskWords;                                 // [ceil((E + S) / 32)]
    WsHeader *hdr = reinterpret_cast<WsHeader *>(p.hdr);
    const bool tail_cta = kq == 0 && rg == (int)(gridDim.x / (unsigned)P.KQ) - 1;
    // the group leader's barrier for the other K ranges' partial sums: set
    // up now, expecting their bytes; every CTA of the cluster arrives at the
    // cluster barrier here and waits on it only before its remote stores
    __shared__ __align__(8) uint64_t s_red_bar;
    __shared__ int s_red_abort;
    if (kq == 0 && tid == 0) {
        s_red_abort = 0;
        mbar_init(smem_u32(&s_red_bar), 1);
        mbar_fence_init();
        mbar_arrive_expect_tx(smem_u32(&s_red_bar), (uint32_t)(P.KQ - 1) * 256u * 4u);
    }
    __syncwarp();
    cluster_arrive();
    if (kq == 0 && tail_cta && P.mask_align) {
        for (int i = tid; i < rows; i += kSmallThreads) tmask[i] = 0u;
        if (tid < kSmallBitWords) tbits[tid] = 0u;
        // the staged sorted_token_ids start as the sentinel n = M * (k + S),
        // over the largest range the align can use: A * min(E + S, n) slots
        const int n = p.M * (p.k + p.S);
        const int fill = (int)min((int64_t)kSmallSortedWords, (int64_t)p.A * min(rows, n));
        uint4 *sb4 = reinterpret_cast<uint4 *>(tbits + kSmallBitWords);
        for (int q = tid; q < (fill + 3) / 4; q += kSmallThreads) sb4[q] = make_uint4(n, n, n, n);
    }

    // ---- 1. gate rows x tokens on the tensor cores ----
    // rows past E+S and tokens past M read a clamped (valid) row; their
    // results are never stored
    const int ra = min(row0 + g, rows - 1), rb = min(row0 + g + 8, rows - 1);
    const uint16_t *wa = (ra < p.E) ? p.w + (int64_t)ra * p.H : p.ws;
    const uint16_t *wb = (rb < p.E) ? p.w + (int64_t)rb * p.H : p.ws;
    const uint16_t *xa = p.x + (int64_t)min(g, p.M - 1) * p.ld;
    const uint16_t *xb = p.x + (int64_t)min(g + 8, p.M - 1) * p.ld;
    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[nb][j] = 0.0f;

    const int s_beg = kq * P.per_cta, s_end = min(s_beg + P.per_cta, P.slices);
    bool waited = false;
    for (int s0 = s_beg + warp; s0 < s_end; s0 += kSmallWarps * kMaxSlicesPerWarp) {
        uint4 va[kMaxSlicesPerWarp], vb[kMaxSlicesPerWarp], x0[kMaxSlicesPerWarp],
            x1[kMaxSlicesPerWarp];
#pragma unroll
        for (int j = 0; j < kMaxSlicesPerWarp; ++j) {
            const int s = s0 + j * kSmallWarps;
            const int kc = min(s * kSliceK + 8 * t, p.H - 8);  // clamped so every load stays in bounds
            va[j] = ld_stream_v4(wa + kc);
            vb[j] = ld_stream_v4(wb + kc);
        }
        // The gate weights are the layer's parameters; the hidden states may
        // come from the previous kernel in the stream: the first batch of gate
        // loads is in flight before waiting for that kernel to complete. The
        // hidden states' lines are only prefetched into L2 before the wait (a
        // hint, no value is read: L2 is coherent, and the loads after the wait
        // go through L2), so that after it they are an L2 hit rather than a
        // DRAM access queued behind the gate stream.
        if (!waited) {
#pragma unroll
            for (int j = 0; j < kMaxSlicesPerWarp; ++j) {
                const int kc = min((s0 + j * kSmallWarps) * kSliceK + 8 * t, p.H - 8);
                asm volatile("prefetch.global.L2 [%0];" ::"l"(xa + kc));
                if (NB > 1) asm volatile("prefetch.global.L2 [%0];" ::"l"(xb + kc));
            }
            griddep_wait();
            waited = true;
        }
#pragma unroll
        for (int j = 0; j < kMaxSlicesPerWarp; ++j) {
            const int s = s0 + j * kSmallWarps;
            const int kc = min(s * kSliceK + 8 * t, p.H - 8);
            x0[j] = __ldcg(reinterpret_cast<const uint4 *>(xa + kc));
            if (NB > 1) x1[j] = __ldcg(reinterpret_cast<const uint4 *>(xb + kc));
        }
#pragma unroll
        for (int j = 0; j < kMaxSlicesPerWarp; ++j) {
            const int s = s0 + j * kSmallWarps;
            if (s >= s_end) continue;  // uniform across the warp (mma.sync is warp-wide)
            if (s * kSliceK + 8 * t >= p.H) {  // this thread's chunk is past H: contributes 0
                va[j] = vb[j] = x0[j] = make_uint4(0u, 0u, 0u, 0u);
                if (NB > 1) x1[j] = x0[j];
            }
            // one slice = two K=16 steps over this thread's elements k0..k0+7:
            // step 0 takes elements 0-3 (as logical k 2t,2t+1 | 2t+8,2t+9),
            // step 1 elements 4-7; A rows g and g+8, B column = token g
            mma_bf16_16816(acc[0], va[j].x, vb[j].x, va[j].y, vb[j].y, x0[j].x, x0[j].y);
            mma_bf16_16816(acc[0], va[j].z, vb[j].z, va[j].w, vb[j].w, x0[j].z, x0[j].w);
            if (NB > 1) {
                mma_bf16_16816(acc[NB - 1], va[j].x, vb[j].x, va[j].y, vb[j].y, x1[j].x, x1[j].y);
                mma_bf16_16816(acc[NB - 1], va[j].z, vb[j].z, va[j].w, vb[j].w, x1[j].z, x1[j].w);
            }
        }
    }

    // everything below reads or writes data the previous kernel may use
    // (bias, workspace, outputs): after its completion (a warp without
    // slices has not waited yet)
    griddep_wait();
    // this call's tag: a 31-bit call count with the top bit set, so that it
    // never equals a cleared word (0) or a nonnegative int32 the align leaves
    // in a shared workspace; the leader of the last row group runs the tail
    float bias_v = 0.0f;
    uint32_t tag = 0u;
    if (kq == 0) {
        tag = ((__ldcg(&hdr->epoch) + 1u) & 0x7FFFFFFFu) | 0x80000000u;
        if (p.bias != nullptr && row0 + r16 < p.E) bias_v = __ldcg(p.bias + row0 + r16);
    }

    // ---- 2. sum the 8 warps, then the cluster's K ranges, in a fixed order ----
    // Shared memory: [0, 8 KB) the warps' partials; [8 KB, 16 KB) the group
    // leader's slots for the cluster's K ranges (written by each CTA of the
    // cluster into the leader's memory); the tail reuses [0, 16 KB); the
    // tail's token masks and bitmap follow at 16 KB.
    float *red = reinterpret_cast<float *>(smem);                 // [8 warps][16 rows][16 tokens]
    float *slots = red + kSmallWarps * 16 * 16;                   // [KQ][16 rows][16 tokens]
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int tok = nb * 8 + 2 * t;
        red[(warp * 16 + g) * 16 + tok] = acc[nb][0];
        red[(warp * 16 + g) * 16 + tok + 1] = acc[nb][1];
        red[(warp * 16 + g + 8) * 16 + tok] = acc[nb][2];
        red[(warp * 16 + g + 8) * 16 + tok + 1] = acc[nb][3];
    }
    __syncwarp();
    __syncthreads();
    {
        // this K range's sum over the warps -> slot kq of the group leader:
        // the leader keeps its own; the others send theirs with st.async,
        // which completes bytes on the leader's barrier, and are done
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kSmallWarps; ++w) v += red[w * 256 + tid];  // tid = row * 16 + token
        cluster_wait();  // the leader's barrier is initialised
        if (kq != 0) {
            st_async_cluster_f32(cluster_addr(smem_u32(slots + kq * 256 + tid), 0u), v,
                                 cluster_addr(smem_u32(&s_red_bar), 0u));
            if (rg == 0 && p.xq != nullptr) small_quant_x(p, kq, P.KQ);
            return;
        }
        slots[tid] = v;  // read back by this thread only
    }
    // the other K ranges' slots have landed (bounded wait; on timeout the
    // error bit is set and the sums are not valid)
    if (!mbar_wait_bounded(smem_u32(&s_red_bar), 0u, &s_red_abort) && tid == 0)
        set_error(&hdr->error, kErrWaitTimeout);
    {
        // the group's final logits: a routed one becomes its selection key
        // (bias added in fp32, then rounded to bf16); the shared expert's
        // slot k = (E, scale * sigmoid(s)) is final here, s not rounded
        float v = 0.0f;
        for (int q = 0; q < P.KQ; ++q) v += slots[q * 256 + tid];
        const int row = row0 + r16;
        if (m16 < p.M && m16 < NB * 8 && row < rows) {
            if (row < p.E) {
                const float zr = round_bf16(v + bias_v);
                st_relaxed_u64(p.scratch + (int64_t)m16 * p.E + row,
                               ((unsigned long long)tag << 32) | make_key(zr, row));
                if (p.logits_out != nullptr)
                    p.logits_out[(int64_t)m16 * p.E + row] = (uint16_t)(__float_as_uint(zr) >> 16);
            } else {
                p.ids[(int64_t)m16 * (p.k + 1) + p.k] = p.E;
                p.wts[(int64_t)m16 * (p.k + 1) + p.k] = p.scale * sigmoid_stable(p.shared_bf16 ? round_bf16(v) : v);
            }
        }
    }
    __syncwarp();
    __syncthreads();
    if (rg == 0 && p.xq != nullptr) small_quant_x(p, 0, P.KQ);  // after this group's keys

    // ---- 3. hand-off: the tail CTA collects the tagged keys ----
    // No fence and no counter: every key word carries the call's tag, so
    // the tail loads each word until it holds this call's tag (the other
    // groups' CTAs have all been launched alongside; they only need SMs).
    if (!tail_cta) return;
    // every other CTA has finished its gate stream (or exited): the next
    // kernel in the stream may launch now (programmatic dependent launch) and
    // stream its own weights during this tail; whatever it reads from this
    // kernel it reads after its own wait
    griddep_launch_dependents();
    __syncwarp();  // a split warp would replay the whole tail once per path

    // ---- 4. tail: top-k + softmax, one warp per token ----
    const int width = p.k + p.S;
    const int n = p.M * width, n4 = (n + 3) & ~3;
    uint32_t *keys_s = reinterpret_cast<uint32_t *>(smem);  // [n4] the align's keys
    uint32_t *cand_s = keys_s + kSmallCandWords;               // [8 warps][32] top-k candidates
    if (P.mask_align && p.S != 0 && tid == 0) {  // the shared expert: every token
        tmask[p.E] = (p.M == 32) ? 0xFFFFFFFFu : (1u << p.M) - 1u;
        atomicOr(tbits + (p.E >> 5), 1u << (p.E & 31));
    }
    // the tag the tail waits for: this call's, or under the failure-
    // injection hook one that no row group writes (the wait then runs out
    // after the hook's limit, sets the error bit and the tail goes on with
    // the words it holds)
    const uint32_t want = p.stall ? (tag + 1u) | 0x80000000u : tag;
    const long long poll_limit = p.stall ? p.stall_limit : kSmallPollLimit;
    for (int m = warp; m < p.M; m += kSmallWarps)
        warp_topk_row<NK>(p.scratch + (int64_t)m * p.E, want, poll_limit, p.E, p.S, p.k, p.renorm,
                          p.ids + (int64_t)m * width,
                          p.wts + (int64_t)m * width, keys_s + m * width, m * width, cand_s + warp * 32,
                          P.mask_align ? tmask : nullptr, tbits, m, &hdr->error);
    if (tid == 0) hdr->epoch = tag;  // read by the next call's CTAs (after this launch ends)
    if (p.sorted == nullptr) return;

    // ---- 5. moe_align_block_size on the M*width ids of this call ----
    __syncwarp();
    __syncthreads();
    if (P.mask_align) {
        int *blkcnt = reinterpret_cast<int *>(keys_s + kSmallMaxM * 32);  // [<= n] ids per block
        int *wpre = blkcnt + kSmallMaxM * 32;                              // [37] blocks before each word
        uint32_t *sbuf = tbits + kSmallBitWords;                           // [kSmallSortedWords]
        align_masks(keys_s, p.M, width, p.A, tmask, tbits, wpre, blkcnt, sbuf, p.sorted, p.sorted_cap,
                    p.expert_ids, p.expert_cap, p.npp, &hdr->error);
        return;
    }
    if (tid < n4 - n) keys_s[n + tid] = 0xFFFFFFFFu;  // padding keys sort last and match nothing
    __syncwarp();
    __syncthreads();
    if (n <= kSmallThreads)
        align_tiny<1>(keys_s, n, p.A, keys_s + kSmallMaxM * 32, p.sorted, p.sorted_cap, p.expert_ids,
                      p.expert_cap, p.npp, &hdr->error);
    else
        align_tiny<2>(keys_s, n, p.A, keys_s + kSmallMaxM * 32, p.sorted, p.sorted_cap, p.expert_ids,
                      p.expert_cap, p.npp, &hdr->error);
}

template <int NB, int NK>
static cudaError_t launch_nb(const SmallParams &P, int grid, size_t smem, cudaStream_t stream) {
    static std::atomic<bool> configured[kMaxDevices];
    cudaError_t e = once_per_device(configured, [smem](int) {
        // the same carveout as every other kernel of the library
        cudaError_t r = cudaFuncSetAttribute(small_route_kernel<NB, NK>,
                                             cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(small_route_kernel<NB, NK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
        return r;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kSmallThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)P.KQ;  // the K ranges of one row group
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start before the previous kernel in the stream completes (it waits
    // for that kernel before reading the hidden states or touching the
    // workspace and outputs)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, small_route_kernel<NB, NK>, P);
}

int small_route_k_ranges(int E, int S, int H) {
    // enough CTAs for one wave on ~150 SMs, at least one slice per warp
    const int groups = (E + S + 15) / 16;
    const int slices = (H + kSliceK - 1) / kSliceK;
    int KQ = 150 / groups;
    if (KQ > kSmallMaxCluster) KQ = kSmallMaxCluster;
    if (KQ < 1) KQ = 1;
    const int max_kq = (slices + kSmallWarps - 1) / kSmallWarps;
    if (KQ > max_kq) KQ = max_kq;
    return KQ;
}

// ---- fixed device scratch for callers that cannot allocate ----------------
//
// Some callers cannot call cudaMalloc on their launch path at all (a host
// that hands out no device allocator, a runtime that forbids allocation once
// its memory pool is sized, code that must not disturb a captured allocation
// pattern). For them the single-launch route+align can run on this
// file-scope array instead of a caller workspace. It lives in every GPU
// that loads the library until the process exits. Host code must not use
// the symbol itself as a pointer (on the host it is only a stand-in), so the
// device address is fetched once per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_route_scratch[kStaticScratchBytes];

cudaError_t static_scratch(void **ptr) {
    static std::atomic<bool> ready[kMaxDevices];
    static std::atomic<void *> addr[kMaxDevices];
    // first use on a device (with it current), once even when host threads
    // race: resolve the address and clear the whole array (header and tagged
    // key words), as a caller clears a workspace before its first use
    cudaError_t e = once_per_device(ready, [](int dev) {
        void *p = nullptr;
        cudaError_t r = cudaGetSymbolAddress(&p, g_route_scratch);
        if (r != cudaSuccess) return r;
        r = cudaMemset(p, 0, kStaticScratchBytes);
        if (r == cudaSuccess) r = cudaDeviceSynchronize();  // cleared before any stream's first launch
        if (r == cudaSuccess) addr[dev].store(p, std::memory_order_relaxed);
        return r;
    });
    if (e != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    *ptr = addr[dev].load(std::memory_order_relaxed);
    return cudaSuccess;
}

cudaError_t launch_small_route(const SmallRouteLaunch &a, cudaStream_t stream) {
    if (a.M <= 0 || a.M > kSmallMaxM) return cudaErrorInvalidValue;
    SmallParams P;
    P.a = a;
    if (P.a.stall_limit <= 0) P.a.stall_limit = kSmallPollLimit;
    P.rows = a.E + a.S;
    P.slices = (a.H + kSliceK - 1) / kSliceK;
    P.KQ = small_route_k_ranges(a.E, a.S, a.H);
    P.mask_align = (a.sorted != nullptr && a.A >= a.M) ? 1 : 0;
    P.per_cta = (P.slices + P.KQ - 1) / P.KQ;
    const int groups = (P.rows + 15) / 16;
    const int grid = groups * P.KQ;
    const size_t smem = (size_t)kSmallSmemWords * 4;
    if (a.E <= 512)
        return a.M <= 8 ? launch_nb<1, 16>(P, grid, smem, stream) : launch_nb<2, 16>(P, grid, smem, stream);
    return a.M <= 8 ? launch_nb<1, 32>(P, grid, smem, stream) : launch_nb<2, 32>(P, grid, smem, stream);
}

}  // namespace smr
