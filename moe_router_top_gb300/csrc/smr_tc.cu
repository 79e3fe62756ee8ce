// smr_tc.cu -- large-M route: tcgen05 gate GEMM with the top-k fused into the
// epilogue.
//
// Computes the same route as the small-M kernel ("[AMD] One-launch small-M
// MoE router for Qwen3.5 on gfx950", Modifications: fp32-accumulated gate
// logits, bf16 rounding of the routed logits, top-k with the lowest id winning
// ties, softmax + renormalisation, shared slot (E, sigmoid(s) * scale)), but
// for many tokens, where the gate GEMM is a dense contraction
// (M=16384: 2*16384*4096*513 = 68.9 GFLOP) and belongs on the tensor cores.
//
// CTA pairs (clusters of 2) own 256-token tiles and use the pair form of the
// 5th-generation tensor-core MMA (tcgen05.mma.cta_group::2, M=256): each CTA
// keeps its 128 token rows of x and HALF of every gate tile in its shared
// memory, and the two SMs' tensor cores share the halves. An M=128 single-SM
// MMA would need every SM to receive the whole gate tile; with it, TMA writes
// plus MMA operand reads reach the SM's shared-memory bandwidth, while the
// pair form halves the gate bytes per SM.
//
// Per CTA, 256 threads (8 warps); warp w issues on scheduler w % 4:
//   warp 0     TMA producer: x tile [128 x 64] and this CTA's half of each
//              N<=256 gate piece [E/2 x 64] per k-block (128-byte swizzle),
//              into a ring of shared-memory stages; loads of both CTAs
//              complete the leader CTA's "full" barrier;
//   warp 3     in the leader CTA, one thread issues the pair MMAs and commits
//              (multicast to both CTAs) to free each stage; warps 0 and 3
//              are alone on their schedulers;
//   warp 1     also allocates TMEM for the pair (E fp32 columns x 128 lanes
//              per CTA);
//   warps 1, 2, 5, 6  meanwhile compute the shared-expert logit of their row
//              from the x tile of each stage (CUDA cores, fp32 per k-block,
//              compensated sum across k-blocks), read once the MMAs are done
//              with the stage and before it is refilled;
//   warps 4, 7 stage the bias and clear the expert counts.
// Epilogue, all 8 warps: warp w reads TMEM lane quarter w%4 (thread = token
// row) and column half w/4 (E/2 experts). Each half selects its own exact
// top-k of bf16-rounded logits in three steps:
//   1. one sweep over TMEM: add the bias, round to bf16 two at a time, keep
//      the rounded row in the (now idle) stage ring, and take the maximum of
//      each unit of 8 (or 4) consecutive columns; T = k-th largest unit
//      maximum (k units hold a logit >= T, so every top-k logit, ties
//      included, is >= T, and only units whose maximum is >= T -- about k of
//      them -- can hold one);
//   2. append the logits >= T of those units to a per-thread shared list
//      with predicated stores (about 1.2k entries on random data);
//   3. order the list as keys in registers (a sorting network up to 16
//      entries; exact k-pass fallback over the half's rounded logits if the
//      list overflows).
// Half 0 posts its top-k to shared memory; half 1 merges the two sorted lists
// (a k-step pointer merge), applies the softmax and writes the row with its
// shared slot. Every mbarrier wait is bounded; on timeout the kernel sets the
// workspace's error bit, skips its outputs and still frees TMEM and leaves
// through the cluster barriers. Warps hand off through mbarriers only.
#include <cudaTypedefs.h>

#include "smr_device.cuh"
#include "smr_launch.h"

namespace smr {

constexpr int kTcBM = 128;            // token rows per CTA (256 per CTA pair)
constexpr int kTcBK = 64;             // k-block: 64 bf16 = 128-byte rows, 128B swizzle
constexpr int kTcSW = kTcBK * 2;
constexpr int kTcThreads = 256;
constexpr int kCandCap = 32;
constexpr int kGroup = 8;             // consecutive columns per group (one 16-byte bf16 group)
// epilogue lists: half 0's candidates (then its top-k), the softmax
// numerators, half 1's candidates, and kGroup slots of room after each list
// for a unit's entries past kCandCap (the numerators are written only after
// the candidates are dead)
constexpr int kEpiListBytes = (3 * kCandCap + kGroup) * kTcBM * 4;
constexpr int kTcSmemLimit = 232448;  // 227 KiB opt-in per CTA

struct TcParams {
    int M, H, E, S, k, width;
    float scale;
    int renorm;       // 1: weights renormalised over the top-k; 0: the E-expert softmax's
    int shared_bf16;  // 1: the shared logit is rounded to bf16 before the sigmoid
    const float *bias;
    const uint16_t *ws;
    const uint16_t *x;  // hidden states (row stride ld), read directly by the shared-logit warps
    int64_t ld;
    int32_t *ids;
    float *wts;
    uint16_t *logits_out;
    uint32_t *err;
    int32_t *tile_counts;  // optional: expert counts of each 64-row tile, [tiles][E + S]
    int stall;             // failure-injection hook: the half merge waits on a barrier
    long long stall_limit; // nothing arrives on, for at most stall_limit SM cycles
    int E_valid;           // gate rows that exist (E is padded to whole swizzle atoms)
    int col0;              // logits-only: first column of this launch in the logit rows
    uint16_t *logits_ws;   // logits-only: [M][ld_logits] bf16
    int64_t ld_logits;
    float *s_out;          // logits-only: [M] shared logit
    uint8_t *xq;           // optional: hidden states as e4m3 codes [M][H]
    float *xs;             // and their scales [M][H / 128]
    int fa_A;              // optional fused align (fa_sorted != nullptr), see TcRouteLaunch
    int32_t *fa_sorted, *fa_eids, *fa_npp;
    int64_t fa_sorted_cap, fa_eids_cap;
    uint32_t *ticket;      // the workspace header's ticket
    int num_kb, stages, n_pieces, piece_n;  // gate pieces of piece_n <= 256 columns
    uint32_t tmem_cols, stage_bytes, misc_off, misc_bias_off, misc_ws_off, misc_hist_off, misc_den_off;
};

// Compensated (two-sum) accumulation of k-block partial sums.
__device__ __forceinline__ void two_sum_acc(float &hi, float &lo, float x) {
    const float t = hi + x;
    const float bp = t - hi;
    const float err = (hi - (t - bp)) + (x - bp);
    hi = t;
    lo += err;
}

// Descending sort of N unsigned keys: Batcher's odd-even merge sort (merges
// of sorted runs of p = 1, 2, 4, ... keys; each merge compares keys k apart
// for k = p, p/2, ..., 1, only within one run pair). The comparator list is
// built at compile time and the network fully unrolled: 63 compare-exchanges
// for N = 16.
template <int N>
struct OddEvenNet {
    int x[N * N], y[N * N], count;
    constexpr OddEvenNet() : x(), y(), count(0) {
        for (int p = 1; p < N; p <<= 1)
            for (int k = p; k >= 1; k >>= 1)
                for (int j = k % p; j + k < N; j += 2 * k)
                    for (int i = 0; i < k; ++i)
                        if (i + j + k < N && (i + j) / (2 * p) == (i + j + k) / (2 * p)) {
                            x[count] = i + j;
                            y[count] = i + j + k;
                            ++count;
                        }
    }
};
template <int N>
__device__ __forceinline__ void sort_desc_oddeven(uint32_t (&a)[N]) {
    constexpr OddEvenNet<N> net{};
#pragma unroll
    for (int c = 0; c < net.count; ++c) {
        const uint32_t hi = max(a[net.x[c]], a[net.y[c]]), lo = min(a[net.x[c]], a[net.y[c]]);
        a[net.x[c]] = hi;
        a[net.y[c]] = lo;
    }
}

// Candidate entry (bf16 bits of the rounded logit in the high half, expert id
// in the low half) -> ordered selection key.
__device__ __forceinline__ uint32_t entry_key(uint32_t entry) {
    // a value >= +0 flips its sign bit, a negative one all its bits; the id
    // becomes 0xFFFF - id either way
    const uint32_t key = entry ^ ((uint32_t)((int32_t)entry >> 31) | 0x8000FFFFu);
    return key + ((key >> 16) == 0x7FFFu ? 0x10000u : 0u);  // a rounded -0 ranks (and ties) as +0
}

// TMEM loads of CW columns (CW = 32 or 16) for one warp's 32 lanes.
template <int CW>
__device__ __forceinline__ void tmem_ld_async(uint32_t taddr, uint32_t (&r)[CW]) {
    if constexpr (CW == 32) tmem_ld32_async(taddr, r); else tmem_ld16_async(taddr, r);
}
template <int CW>
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[CW]) {
    if constexpr (CW == 32) tmem_wait_ld(r); else tmem_wait_ld16(r);
}

// Two fp32 values rounded to bf16 (nearest-even) in one 32-bit word, lo in
// the low half (the lower address in memory).
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// Lane-wise maximum of two bf16 pairs.
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w));
}
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Row stride of the rounded-logit copy in shared memory: an odd multiple of
// 16 bytes, so eight consecutive rows' 16-byte groups fall in distinct banks.
__host__ __device__ constexpr uint32_t dump_row_bytes(int ecols) { return (uint32_t)ecols * 2u + 16u; }

// bf16 pair -> ordered unsigned 16-bit keys (numeric order as unsigned
// order, -0 and +0 both 0x8000): a value >= +0 sets its sign bit, a negative
// one b becomes 2^16 - b. (The negative half's +1 never carries out of it.)
__device__ __forceinline__ uint32_t ordered_bf16x2(uint32_t x) {
    const uint32_t neg = (x >> 15) & 0x00010001u;  // sign bit of each half
    return (x ^ ((neg * 0xFFFFu) | 0x80008000u)) + neg;
}
// Ordered 16-bit key -> the bf16 value as a float.
__device__ __forceinline__ float ordered16_value(uint32_t o) {
    const uint32_t b = (o & 0x8000u) ? (o & 0x7FFFu) : ((0x10000u - o) & 0xFFFFu);
    return __uint_as_float(b << 16);
}
// The larger halves of two bf16 pairs' halves: (max of a's halves, max of b's).
__device__ __forceinline__ uint32_t halves_max_bf16x2(uint32_t a, uint32_t b) {
    return max_bf16x2(__byte_perm(a, b, 0x5410), __byte_perm(a, b, 0x7632));
}

// Lane-wise (16-bit halves) wrapping add and unsigned maximum.
__device__ __forceinline__ uint32_t add_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// A value of rank <= k among the 32 ordered 16-bit keys packed in pw (0 =
// empty): the maximum, then k - 1 steps to the largest key below the current
// one. A step adds 2^16 - m to every half (mod 2^16): keys >= m land in
// [0, 2^16 - m) and keys < m in [2^16 - m, 2^16), in their own order, so one
// maximum over the shifted halves, shifted back, is the next key down; it is
// 0 (an empty half) or >= m when no key below m is left, and m stays. Equal
// keys count once, so the result is at
// most the k-th largest; it stays a valid lower bound for "at least k keys
// are >= it".
__device__ __forceinline__ uint32_t kth_largest_packed(const uint32_t (&pw)[kCandCap / 2], int k) {
    uint32_t m2 = pw[0];
#pragma unroll
    for (int i = 1; i < kCandCap / 2; ++i) m2 = max_u16x2(m2, pw[i]);
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll 1
    for (int r = 1; r < k; ++r) {
        const uint32_t d = (0x10000u - m) & 0xFFFFu, dd = d | (d << 16);
        uint32_t z[kCandCap / 2];
#pragma unroll
        for (int i = 0; i < kCandCap / 2; ++i) z[i] = add_u16x2(pw[i], dd);
#pragma unroll
        for (int w = kCandCap / 4; w >= 1; w >>= 1)  // a tree of maxima
#pragma unroll
            for (int i = 0; i < w; ++i) z[i] = max_u16x2(z[i], z[i + w]);
        const uint32_t z2 = z[0];
        const uint32_t nx = (max(z2 & 0xFFFFu, z2 >> 16) + m) & 0xFFFFu;
        m = (nx != 0u && nx < m) ? nx : m;  // (nx >= m: every key is >= m)
    }
    return m;
}

// A thread's n <= SLOTS candidate entries (list column, stride kTcBM words)
// -> its k largest keys, in order, written back to the same column.
template <int SLOTS>
__device__ __forceinline__ void topk_from_list(uint32_t *col, uint32_t n, int k) {
    uint32_t a[SLOTS];
#pragma unroll
    for (int j = 0; j < SLOTS; ++j) a[j] = (j < (int)n) ? entry_key(col[j * kTcBM]) : 0u;
    if constexpr (SLOTS == 16) {  // the common case: one sorting network
        sort_desc_oddeven(a);
#pragma unroll
        for (int r = 0; r < SLOTS; ++r)
            if (r < k) col[r * kTcBM] = a[r];
        for (int r = SLOTS; r < k; ++r) col[r * kTcBM] = 0u;
    } else {
        // k rounds. Keys are distinct: after the maximum, each round takes
        // the largest key below the previous one as the maximum of a[i] - m
        // (mod 2^32), which puts keys >= m below every key < m, shifted back;
        // the result is >= m (every slot holds a key >= m) or 0 (an empty
        // slot) when no key is left, and then 0 stays. (Rolled: this path's
        // instructions are fetched cold, and a network over both halves of
        // the list measured slower in the whole step.)
        uint32_t m = a[0];
#pragma unroll
        for (int i = 1; i < SLOTS; ++i) m = max(m, a[i]);
        col[0] = m;
#pragma unroll 1
        for (int r = 1; r < k; ++r) {
            uint32_t z = a[0] - m;
#pragma unroll
            for (int i = 1; i < SLOTS; ++i) z = max(z, a[i] - m);
            const uint32_t nxt = z + m;
            m = nxt < m ? nxt : 0u;
            col[r * kTcBM] = m;
        }
    }
}

// Exact fallback for a row whose candidates overflowed the list: k passes
// over the ng groups of its rounded logits in shared memory, each taking the
// largest key below the previous one.
__device__ __noinline__ void topk_from_row(uint32_t drow, int ng, int c_beg, int k, uint32_t *col) {
    uint32_t prev = 0xFFFFFFFFu;
    for (int r = 0; r < k; ++r) {
        uint32_t best = 0u;
        for (int g = 0; g < ng; ++g) {
            const uint4 v = ld_shared_v4(drow + (uint32_t)(g * 16));
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const uint32_t hb = (u & 1) ? (wv[u >> 1] & 0xFFFF0000u) : (wv[u >> 1] << 16);
                const uint32_t k2 = entry_key(hb | (uint32_t)(c_beg + g * kGroup + u));
                best = (k2 < prev && k2 > best) ? k2 : best;
            }
        }
        col[r * kTcBM] = best;
        prev = best;
    }
}

// The largest magnitude of a k-block row's 64 bf16 (eight 16-byte chunks),
// as a packed pair of bf16 maxima.
__device__ __forceinline__ uint32_t absmax_bf16x2(const uint4 (&a)[kTcBK / 8]) {
    uint32_t m = 0u;  // packed bf16 magnitudes: sign bits cleared, then pair maxima
#pragma unroll
    for (int c = 0; c < kTcBK / 8; ++c) {
        m = max_bf16x2(m, max_bf16x2(a[c].x & 0x7FFF7FFFu, a[c].y & 0x7FFF7FFFu));
        m = max_bf16x2(m, max_bf16x2(a[c].z & 0x7FFF7FFFu, a[c].w & 0x7FFF7FFFu));
    }
    return m;
}
// 128 bf16 (two k-blocks' eight 16-byte chunks each, in element order) to
// e4m3: scale = amax / 448, codes = e4m3(x * (448 / amax)) rounded to
// nearest even and saturated (cvt.rn.satfinite), the divisions and the
// product in fp32; a block of zeros gets scale 0 and zero codes. m: the
// packed maxima of both halves (absmax_bf16x2). Writes 128 code bytes
// (8-byte aligned) and the scale.
__device__ __forceinline__ void quant_block_e4m3(const uint4 (&a)[kTcBK / 8], const uint4 (&b)[kTcBK / 8],
                                                 uint32_t m, uint8_t *q, float *scale) {
    const float amax = fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
    if (amax == 0.0f) {  // zero codes (also for -0 elements) and scale 0
#pragma unroll
        for (int i = 0; i < 8; ++i) reinterpret_cast<uint4 *>(q)[i] = make_uint4(0u, 0u, 0u, 0u);
        *scale = 0.0f;
        return;
    }
    const float inv = 448.0f / amax;
    *scale = amax / 448.0f;
    // one 8-element chunk at a time (8 codes, one 8-byte store), so that few
    // products are live at once
#pragma unroll
    for (int c = 0; c < 2 * (kTcBK / 8); ++c) {
        const uint4 v = c < kTcBK / 8 ? a[c] : b[c - kTcBK / 8];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t code[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint16_t lo, hi;
            asm volatile("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo)
                         : "f"(__uint_as_float(w[2 * h] & 0xFFFF0000u) * inv), "f"(__uint_as_float(w[2 * h] << 16) * inv));
            asm volatile("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi)
                         : "f"(__uint_as_float(w[2 * h + 1] & 0xFFFF0000u) * inv),
                           "f"(__uint_as_float(w[2 * h + 1] << 16) * inv));
            code[h] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        reinterpret_cast<uint2 *>(q)[c] = make_uint2(code[0], code[1]);
    }
}

// The align fused into the route for at most kFusedAlignMax ids
// ("[ROCm][Kernel] W4A16 MoE prefill: M-aware moe_align block size",
// Purpose; the shared expert is expert E, appended to the sorted route stream
// as "Netra Kernel ...", Reusing routing work instead of recomputing it, does
// without a separate launch). Every thread publishes its id stores, one
// thread per CTA takes a ticket; the last CTA to finish stages all the ids
// from L2 into its idle stage ring and runs the single-CTA align there, then
// sets the ticket back to zero for the next call (whose route writes nothing
// before this grid has completed).
// s_last: a word of shared memory (kept out of static shared memory, so that
// the kernel's dynamic allocation can take the whole opt-in limit).
__device__ __noinline__ void fused_align_tail(const TcParams &p, uint8_t *smem, volatile int *s_last) {
    __threadfence();  // this thread's ids are visible device-wide before the ticket
    __syncthreads();
    if (threadIdx.x == 0) *s_last = atomicAdd(p.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!*s_last) return;
    __threadfence();  // the other CTAs' ids, published before their tickets
    const int numel = p.M * p.width, E_al = p.E + p.S;
    int *ids = reinterpret_cast<int *>(smem);
    AlignSmem s = align_carve(ids + kAlignSingleMax, E_al);
    stage_ids(ids, p.ids, numel);
    align_count(ids, numel, E_al, s, p.err);
    const int npp = align_offsets(s.cnt, E_al, p.fa_A, s);
    align_scatter(ids, numel, E_al, 0, s, false, p.fa_sorted, p.fa_sorted_cap, p.err);
    align_fill(p.fa_A, E_al, s.cnt, s, numel, p.fa_sorted, p.fa_sorted_cap, p.fa_eids, p.fa_eids_cap, p.err,
               threadIdx.x, blockDim.x);
    if (threadIdx.x == 0) {
        *p.fa_npp = npp;
        *p.ticket = 0u;
    }
}

// Optional logits output: the row's rounded logits from shared memory.
__device__ __noinline__ void copy_row_out(uint32_t drow, uint16_t *dst, int ng) {
    for (int g = 0; g < ng; ++g) reinterpret_cast<uint4 *>(dst)[g] = ld_shared_v4(drow + (uint32_t)(g * 16));
}

template <int CW, bool LO, bool XQ, bool QD>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_route_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const int ST = p.stages;
    uint8_t *misc = smem + p.misc_off;
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);  // leader: both CTAs' loads landed
    uint64_t *mma_done = full + ST;    // both CTAs: the pair MMAs are done with the stage
    uint64_t *empty = mma_done + ST;   // both CTAs, with a shared gate: the shared-logit warps are too
    uint64_t *accum = empty + ST;      // the pair MMAs of the whole K loop are done
    uint64_t *half_done = accum + 1;   // the 4 warps of column half 0 posted their top-k
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(half_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);  // then the fused align's flag
    float *bias_s = reinterpret_cast<float *>(misc + p.misc_bias_off);
    int *hist = reinterpret_cast<int *>(misc + p.misc_hist_off);  // [2][E + S] counts of the CTA's two 64-row tiles
    float *ws_s = reinterpret_cast<float *>(misc + p.misc_ws_off);  // the shared gate row in fp32
    float2 *den_s = reinterpret_cast<float2 *>(misc + p.misc_den_off);  // [128] half 0's (sum, max)
    float *sh_s = reinterpret_cast<float *>(misc + p.misc_den_off + kTcBM * sizeof(float2));  // [128] shared logits

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kTcBM;
    const uint32_t rank = cluster_ctarank();  // 0 = leader of the pair, 1 = peer
    const bool leader = rank == 0;
    const uint16_t pair_mask = 0x3;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&mma_done[s]), 1);  // the MMA commit (multicast to both CTAs)
            mbar_init(smem_u32(&empty[s]), 4);     // the 4 side warps (shared logit, e4m3 x)
        }
        mbar_init(smem_u32(accum), 1);
        mbar_init(smem_u32(half_done), 4);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_w);
    }
    if (warp == 1) {  // one warp in each CTA of the pair allocates for both
        tmem_alloc_pair(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish_pair();
    }
    griddep_launch_dependents();  // the align launches may start; they wait for this grid
    // barriers initialised and TMEM allocated in this CTA; the producer and
    // the MMA issuer start once the peer is there too, while the other warps
    // stage what only later steps read (overlapping the first loads)
    tc_fence_before();
    cluster_arrive();
    // warp roles in the K loop: 0 the TMA producer and 3 the MMA issuer,
    // each alone on its scheduler (warp w runs on scheduler w % 4); 1, 2, 5
    // and 6 the side warps (shared logit, e4m3 hidden states; side rows
    // si * 32 + lane); 4 and 7 stage the bias and clear the expert counts
    const bool is_side = warp == 1 || warp == 2 || warp == 5 || warp == 6;
    const int si = warp < 4 ? warp - 1 : warp - 3;
    if (warp == 4 || warp == 7) {  // bias and expert counts, read in the epilogue
        const int j = (warp == 4 ? 0 : 32) + lane;
        for (int i = j; i < p.E; i += 64) bias_s[i] = (p.bias && i < p.E_valid) ? p.bias[i] : 0.0f;
        for (int i = j; i < 2 * (p.E + p.S); i += 64) hist[i] = 0;
    } else if (is_side && p.S) {
        // the shared gate row in fp32 (converted once here rather than per
        // stage), zero-padded to whole k-blocks
        const int nch = p.H >> 3;
        for (int c = si * 32 + lane; c < p.num_kb * (kTcBK / 8); c += 128) {
            float f[8];
            unpack8(c < nch ? reinterpret_cast<const uint4 *>(p.ws)[c] : make_uint4(0u, 0u, 0u, 0u), f);
            reinterpret_cast<float4 *>(ws_s)[2 * c] = make_float4(f[0], f[1], f[2], f[3]);
            reinterpret_cast<float4 *>(ws_s)[2 * c + 1] = make_float4(f[4], f[5], f[6], f[7]);
        }
        asm volatile("bar.sync 2, 128;" ::: "memory");  // the 4 shared-logit warps read all of it
    }
    cluster_wait();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const bool side = p.S || XQ;  // the side warps read every stage's x tile
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    const int hf = warp >> 2; // column half this warp takes in the epilogue
    const int row = q * 32 + lane;
    const int grow = m0 + row;
    const bool valid = grow < p.M;
    float s_hi = 0.0f, s_lo = 0.0f;  // shared-expert logit of a side warp's row (compensated sum)

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            const uint32_t half = (uint32_t)(p.piece_n / 2);  // gate rows per CTA per piece
            // a tile entirely past M (the padding partner of a pair) loads a
            // valid tile instead; its results are never written
            const int m_load = m0 < p.M ? m0 : 0;
            // the gate pieces of the first stages (layer parameters) are
            // requested before waiting for the previous kernel in the stream
            // (programmatic dependent launch), the hidden states after it;
            // their first stages are only prefetched into L2 before the wait
            // (a hint: no value is read, L2 is coherent and the loads after
            // the wait go through it), so that those loads hit L2
            const int pre = min(ST, p.num_kb);
            for (int kb = 0; kb < pre; ++kb) {
                const uint32_t fb = cluster_addr(smem_u32(&full[kb]), 0u);  // leader's barrier
                if (leader) mbar_arrive_expect_tx(smem_u32(&full[kb]), 2u * p.stage_bytes);
                const uint32_t b_dst = smem_u32(smem + (size_t)kb * p.stage_bytes) + kTcBM * kTcSW;
                for (int pc = 0; pc < p.n_pieces; ++pc)
                    tma_load_2d_pair(b_dst + (uint32_t)pc * half * kTcSW, &tm_w, kb * kTcBK,
                                     pc * p.piece_n + (int)(rank * half), fb);
            }
            for (int kb = 0; kb < pre; ++kb) tma_prefetch_l2_2d(&tm_x, kb * kTcBK, m_load);
            griddep_wait();
            int kb = 0;
            for (; kb < p.num_kb; ++kb) {
                const int s = kb % ST;
                const uint32_t ph = (uint32_t)(kb / ST) & 1u;
                const uint32_t fb = cluster_addr(smem_u32(&full[s]), 0u);  // leader's barrier
                const uint32_t a_dst = smem_u32(smem + (size_t)s * p.stage_bytes);
                if (kb >= pre) {
                    // a stage is refilled once the MMAs (and, with a shared
                    // gate, the shared-logit warps) are done with it
                    if (!mbar_wait_bounded(smem_u32(side ? &empty[s] : &mma_done[s]), ph ^ 1u, abort_flag)) break;
                    if (leader) mbar_arrive_expect_tx(smem_u32(&full[s]), 2u * p.stage_bytes);
                }
                tma_load_2d_pair(a_dst, &tm_x, kb * kTcBK, m_load, fb);
                if (kb >= pre) {
                    const uint32_t b_dst = a_dst + kTcBM * kTcSW;
                    for (int pc = 0; pc < p.n_pieces; ++pc)
                        tma_load_2d_pair(b_dst + (uint32_t)pc * half * kTcSW, &tm_w, kb * kTcBK,
                                         pc * p.piece_n + (int)(rank * half), fb);
                }
            }
            if (kb < p.num_kb) set_error(p.err, kErrWaitTimeout);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------ MMA issuer (leader) ----
        if (leader && lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(2 * kTcBM, p.piece_n);
            const uint32_t half = (uint32_t)(p.piece_n / 2);
            for (int kb = 0; kb < p.num_kb; ++kb) {
                const int s = kb % ST;
                const uint32_t ph = (uint32_t)(kb / ST) & 1u;
                if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag)) {
                    set_error(p.err, kErrWaitTimeout);
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_u32(smem + (size_t)s * p.stage_bytes);
                const uint32_t b_base = a_base + kTcBM * kTcSW;
                // piece-major: a piece's four K=16 steps back to back into its
                // accumulator, then the next piece (alternating the two
                // accumulators step by step ran the pair MMAs ~15% slower:
                // 65.5 against 55.5 us per 16384-token launch)
                for (int pc = 0; pc < p.n_pieces; ++pc) {
#pragma unroll
                    for (int kk = 0; kk < kTcBK / 16; ++kk) {
                        const uint64_t adesc = smem_desc_sw<kTcSW>(a_base + kk * 32);
                        const uint64_t bdesc =
                            smem_desc_sw<kTcSW>(b_base + (uint32_t)pc * half * kTcSW + kk * 32);
                        tc_mma_bf16_pair(tmem + (uint32_t)(pc * p.piece_n), adesc, bdesc, idesc,
                                         (kb | kk) != 0 ? 1u : 0u);
                    }
                }
                tc_commit_pair(smem_u32(&mma_done[s]), pair_mask);
            }
            tc_commit_pair(smem_u32(accum), pair_mask);
        }
        __syncwarp();
    } else if (is_side && side) {
        // ---- side warps 1, 2, 5, 6: shared-expert logit and e4m3 hidden states ----
        // once the MMAs are done with a stage (their commit reaches both
        // CTAs) its x tile is still in place: thread = token row reads the
        // row's 64 elements of the k-block (eight 16-byte chunks, 128-byte
        // swizzle: chunk c sits at c ^ (row & 7)); then
        //  - shared logit: fp32 dot per k-block, compensated sum across them;
        //  - e4m3: the even k-block's elements wait in registers for the odd
        //    one; the 128-element block's largest magnitude gives its scale
        //    amax / 448 and the codes e4m3(x * (448 / amax)), stored with
        //    16-byte stores ("Netra Kernel ...", Fusing the activation/
        //    quantization boundary: E4M3 with one scale per 128 values);
        // each warp then releases the stage
        const int srow = si * 32 + lane, sgrow = m0 + srow;
        const bool svalid = sgrow < p.M;
        const uint32_t swz = (uint32_t)(srow & 7);
        uint4 prev[kTcBK / 8];  // the even k-block's chunks (e4m3 only)
        uint32_t prev_max = 0u; // and their largest magnitudes (packed bf16 pair)
        for (int kb = 0; kb < p.num_kb; ++kb) {
            const int s = kb % ST;
            const uint32_t ph = (uint32_t)(kb / ST) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&mma_done[s]), ph, abort_flag))) {
                set_error(p.err, kErrWaitTimeout);
                break;
            }
            const uint8_t *xrow = smem + (size_t)s * p.stage_bytes + (size_t)srow * kTcSW;
            uint4 xv[kTcBK / 8];
#pragma unroll
            for (int c = 0; c < kTcBK / 8; ++c) xv[c] = *reinterpret_cast<const uint4 *>(xrow + ((c ^ swz) << 4));
            // every loaded value is used below before the stage is released
            // (a release issued while shared-memory loads are still in flight
            // may let the next TMA write overtake them)
            if (p.S) {
                const float4 *wsv = reinterpret_cast<const float4 *>(ws_s) + kb * (kTcBK / 4);
                float part = 0.0f;
#pragma unroll
                for (int c = 0; c < kTcBK / 8; ++c) {
                    float xf[8];
                    unpack8(xv[c], xf);
                    const float4 w0 = wsv[2 * c], w1 = wsv[2 * c + 1];
                    const float wf[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) part = fmaf(xf[e], wf[e], part);
                }
                two_sum_acc(s_hi, s_lo, part);
            }
            if constexpr (XQ) {
                const uint32_t m = absmax_bf16x2(xv);
                if ((kb & 1) == 0) {
#pragma unroll
                    for (int c = 0; c < kTcBK / 8; ++c) prev[c] = xv[c];
                    prev_max = m;
                } else if (svalid) {
                    quant_block_e4m3(prev, xv, max_bf16x2(prev_max, m),
                                     p.xq + (int64_t)sgrow * p.H + (kb >> 1) * 128,
                                     p.xs + (int64_t)sgrow * (p.H >> 7) + (kb >> 1));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }
        __syncwarp();
        if (p.S) sh_s[srow] = s_hi + s_lo;  // read by the merge after the epilogue's first barrier
    }

    // ---------------------------------- epilogue: all 8 warps ----------
    // warp (q, hf) owns TMEM lanes of quarter q (token rows q*32..q*32+31) and
    // expert columns [hf*E/2, (hf+1)*E/2); each half finds its own exact
    // top-k, half 1 merges both lists and writes the row. The epilogue runs
    // once per CTA after other kernels have used the SM, so its instructions
    // are fetched cold and its code size counts next to its instruction
    // count: short rolled loops (k steps to the next key, a pointer merge),
    // with one 16-key sorting network as the only long straight-line part.
    griddep_wait();   // outputs and counts are written only after the previous kernel completed
    __syncthreads();  // the bias and count staging of warps 4 and 7 is visible to every warp
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(accum), 0u, abort_flag));
    tc_fence_after();
    ok = __shfl_sync(0xffffffffu, (ok && !*abort_flag) ? 1 : 0, 0) != 0;  // one decision per warp
    __syncwarp();  // lanes left the bounded wait on different iterations
    if constexpr (LO) {
        // logits only: this launch's columns [col0, col0 + E), the bias added
        // and rounded to bf16 (columns past E_valid: -inf), into the rows of
        // the workspace; the shared logit of the side warps' rows. A select
        // kernel takes the top-k over whole rows afterwards.
        if (ok) {
            const int ecols = p.E / 2, c_beg = hf * ecols;
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c_beg;
            uint16_t *dst = p.logits_ws + (int64_t)(valid ? grow : 0) * p.ld_logits + p.col0 + c_beg;
#pragma unroll 1
            for (int ch = 0; ch < ecols / CW; ++ch) {
                uint32_t r[CW];
                tmem_ld_async<CW>(taddr + (uint32_t)(ch * CW), r);
                tmem_ld_wait<CW>(r);
#pragma unroll
                for (int u = 0; u < CW / kGroup; ++u) {
                    uint32_t wv[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int i = u * kGroup + 2 * t, c = c_beg + ch * CW + i;
                        const float lo = c < p.E_valid ? __uint_as_float(r[i]) + bias_s[c] : -INFINITY;
                        const float hi = c + 1 < p.E_valid ? __uint_as_float(r[i + 1]) + bias_s[c + 1] : -INFINITY;
                        wv[t] = pack_bf16x2_rn(lo, hi);
                    }
                    if (valid)
                        *reinterpret_cast<uint4 *>(dst + ch * CW + u * kGroup) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
            if (hf == 1 && p.S && valid) p.s_out[grow] = sh_s[row];
        } else if (lane == 0) {
            set_error(p.err, kErrWaitTimeout);
        }
    } else {
        const int ecols = p.E / 2;
        const int c_beg = hf * ecols;
        const int nch = ecols / CW;       // CW-column TMEM chunks per half
        const int ng = ecols / kGroup;    // groups of kGroup consecutive columns per half
        // the stage ring is idle once the accumulator is complete. Per half a
        // list column per thread ([32][128] words: group maxima, then candidates,
        // then the half's top-k), softmax numerators of half 1, and each half's
        // rounded logits (row stride rs)
        uint32_t *list = reinterpret_cast<uint32_t *>(smem) + hf * (2 * kCandCap * kTcBM);
        uint32_t *list0 = reinterpret_cast<uint32_t *>(smem);                 // half 0's top-k
        float *numer = reinterpret_cast<float *>(smem) + kCandCap * kTcBM;  // [32][128], between the lists
        const uint32_t rs = dump_row_bytes(ecols);
        const uint32_t drow = smem_u32(smem) + (uint32_t)(kEpiListBytes + (hf * kTcBM + row) * rs);
        float den_half = 0.0f, v_half = 0.0f;  // without renormalisation: this half's denominator
        // threshold units: groups of kGroup columns, or for a half of at most
        // 128 columns quads of 4 (with few groups, k of them would select
        // nearly every group and overflow the candidate list)
        constexpr bool quads = QD;  // (QD only with ecols <= 128)
        const int nu = quads ? ecols / 4 : ng;
        if (ok) {
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c_beg;
            // 1. one sweep over this half's TMEM columns: add the bias, round to
            //    bf16 two at a time, keep the row in shared memory and the maximum
            //    of each group of kGroup columns in the thread's list column
            uint32_t ra[CW], rb[CW];
            // (without a bias the logits are rounded as they are: no bias
            // loads and adds in this issue-bound sweep)
            auto process = [&](uint32_t (&r)[CW], int ch, auto with_bias) {
                const int c = c_beg + ch * CW;
                uint32_t pair = 0u;  // the even group's pair maxima
    #pragma unroll
                for (int u = 0; u < CW / kGroup; ++u) {
                    uint32_t wv[4];
                    if constexpr (decltype(with_bias)::value) {
                        float b[kGroup];
                        const float4 b0 = *reinterpret_cast<const float4 *>(bias_s + c + u * kGroup);
                        const float4 b1 = *reinterpret_cast<const float4 *>(bias_s + c + u * kGroup + 4);
                        b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
                        b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
    #pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int i = u * kGroup + 2 * t;
                            wv[t] = pack_bf16x2_rn(__uint_as_float(r[i]) + b[2 * t],
                                                   __uint_as_float(r[i + 1]) + b[2 * t + 1]);
                        }
                    } else {
    #pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int i = u * kGroup + 2 * t;
                            wv[t] = pack_bf16x2_rn(__uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                        }
                    }
                    const int g = ch * (CW / kGroup) + u;
                    st_shared_v4(drow + (uint32_t)(g * 16), make_uint4(wv[0], wv[1], wv[2], wv[3]));
                    // the unit maxima: bf16 pair maxima, then one conversion to
                    // ordered keys per two units (a -0 maximum ranks as +0)
                    const uint32_t qa = max_bf16x2(wv[0], wv[1]), qb = max_bf16x2(wv[2], wv[3]);
                    if (quads) {  // the group's two quads, one word
                        list[g * kTcBM + row] = ordered_bf16x2(halves_max_bf16x2(qa, qb));
                    } else {      // two groups, one word
                        const uint32_t m = max_bf16x2(qa, qb);  // (even columns' maximum, odd columns')
                        if (u & 1) list[(g >> 1) * kTcBM + row] = ordered_bf16x2(halves_max_bf16x2(pair, m));
                        pair = m;
                    }
                }
            };
            auto sweep = [&](auto with_bias) {
                tmem_ld_async<CW>(taddr, ra);
                tmem_ld_wait<CW>(ra);
                for (int ch = 0; ch < nch; ch += 2) {  // the next chunk's load in flight
                    const bool two = ch + 1 < nch;
                    if (two) tmem_ld_async<CW>(taddr + (uint32_t)((ch + 1) * CW), rb);
                    process(ra, ch, with_bias);
                    if (two) {
                        tmem_ld_wait<CW>(rb);
                        if (ch + 2 < nch) tmem_ld_async<CW>(taddr + (uint32_t)((ch + 2) * CW), ra);
                        process(rb, ch + 1, with_bias);
                        if (ch + 2 < nch) tmem_ld_wait<CW>(ra);
                    }
                }
            };
            if (p.bias != nullptr)
                sweep(std::true_type{});
            else
                sweep(std::false_type{});
            __syncwarp();
            if (__builtin_expect(p.logits_out != nullptr, 0) && valid)
                copy_row_out(drow, p.logits_out + (int64_t)grow * p.E + c_beg, ng);
            // the k-th largest unit maximum T bounds this half's top-k from
            // below (k units hold a logit >= T); only units whose maximum is
            // >= T can hold a logit >= T. Unit maxima are ordered 16-bit keys,
            // two per word, so each of the k steps works on 16 registers.
            uint32_t sel = 0;
            float T = -INFINITY;
            if (p.k <= nu) {
                uint32_t pw[kCandCap / 2];
    #pragma unroll
                for (int i = 0; i < kCandCap / 2; ++i) pw[i] = (2 * i < nu) ? list[i * kTcBM + row] : 0u;
                const uint32_t t16 = kth_largest_packed(pw, p.k);
                T = ordered16_value(t16);
                const uint32_t ts = t16 | (t16 << 16);
    #pragma unroll
                for (int i = 0; i < kCandCap / 2; ++i) {
                    const uint32_t ge = __vcmpgeu2(pw[i], ts);
                    sel |= ((ge & 1u) << (2 * i)) | (((ge >> 16) & 1u) << (2 * i + 1));
                }
                sel &= (nu >= 32) ? 0xFFFFFFFFu : ((1u << nu) - 1u);
            } else {
                sel = (nu >= 32) ? 0xFFFFFFFFu : ((1u << nu) - 1u);  // fewer units than k: all
            }
            __syncwarp();
            // 2. append every logit >= T of the selected units (about k units)
            //    to the list column, over the unit maxima. A unit adds at most
            //    kGroup entries, so while n <= kCandCap it is taken without a
            //    bound check (the kGroup slots past a list are room for it);
            //    n > kCandCap marks an overflow
            constexpr uint32_t nv = quads ? 4u : (uint32_t)kGroup;  // columns per unit
            uint32_t *cand = list + row;
    #pragma unroll 1
            while (__any_sync(0xffffffffu, sel != 0u)) {
                const bool on = sel != 0u && cand <= list + row + kCandCap * kTcBM;
                const int g = sel != 0u ? __ffs(sel) - 1 : 0;  // the unit
                sel &= sel - 1u;
                uint32_t wv[4];
                if (quads) {
                    const uint2 v = ld_shared_v2(drow + (uint32_t)(g * 8));
                    wv[0] = v.x; wv[1] = v.y; wv[2] = 0u; wv[3] = 0u;
                } else {
                    const uint4 v = ld_shared_v4(drow + (uint32_t)(g * 16));
                    wv[0] = v.x; wv[1] = v.y; wv[2] = v.z; wv[3] = v.w;
                }
                const uint32_t col = (uint32_t)(c_beg + g * (int)nv);  // a multiple of nv
    #pragma unroll
                for (int u = 0; u < (int)nv; ++u) {
                    const uint32_t hb = (u & 1) ? (wv[u >> 1] & 0xFFFF0000u) : (wv[u >> 1] << 16);
                    const bool c = on && __uint_as_float(hb) >= T;
                    if (c) *cand = hb | col | (uint32_t)u;
                    cand += c ? kTcBM : 0;
                }
            }
            const uint32_t n = (uint32_t)(cand - (list + row)) / kTcBM;
            __syncwarp();
            // 3. this half's top-k, in order, into the list column: a sorting
            //    network over up to 16 candidate keys, else k rounds of the
            //    largest remaining key. A row whose candidates overflowed the
            //    list takes k passes over its rounded logits.
            if (__all_sync(0xffffffffu, n <= 16u)) {
                topk_from_list<16>(list + row, n, p.k);  // the common case (~0.3% of rows exceed 16)
            } else if (__builtin_expect(__any_sync(0xffffffffu, n > (uint32_t)kCandCap), 0)) {
                if (n > (uint32_t)kCandCap) topk_from_row(drow, ng, c_beg, p.k, list + row);
                else topk_from_list<kCandCap>(list + row, n, p.k);
            } else {
                topk_from_list<kCandCap>(list + row, n, p.k);
            }
            __syncwarp();
            // 4. without renormalisation: this half's share of the E-expert
            //    softmax denominator, every rounded logit's exponential relative
            //    to the half's largest (eight per group as a tree, the groups by a
            //    compensated sum); half 1 rescales both to the row's largest
            if (!p.renorm) {
                v_half = key_value(list[row]);
                float hi = 0.0f, lo = 0.0f;
    #pragma unroll 1
                for (int g = 0; g < ng; ++g) {
                    const uint4 v = ld_shared_v4(drow + (uint32_t)(g * 16));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                    float e[kGroup];
    #pragma unroll
                    for (int u = 0; u < kGroup; ++u)
                        e[u] = expf(__uint_as_float((u & 1) ? (wv[u >> 1] & 0xFFFF0000u) : (wv[u >> 1] << 16)) - v_half);
    #pragma unroll
                    for (int h = kGroup / 2; h >= 1; h >>= 1)
    #pragma unroll
                        for (int u = 0; u < h; ++u) e[u] += e[u + h];
                    two_sum_acc(hi, lo, e[0]);
                }
                den_half = hi + lo;
            }
        }
        if (hf == 0) {
            if (!p.renorm) den_s[row] = make_float2(den_half, v_half);  // posted with the top-k
            __syncwarp();
            // (under the failure-injection hook half 0 does not post: the merge's
            // wait then runs out, which sets the error bit and skips the outputs)
            if (lane == 0 && !p.stall) mbar_arrive(smem_u32(half_done));
        } else {
            // ------------------------------ half 1: merge, softmax, write -----
            const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(half_done), 0u, abort_flag,
                                                                       p.stall ? p.stall_limit : kWaitCycles));
            __syncwarp();
            if (ok && got && valid) {
                int32_t *orow = p.ids + (int64_t)grow * p.width;
                float *wrow = p.wts + (int64_t)grow * p.width;
                int *h = hist + (row / kTcCountRows) * (p.E + p.S);
                const bool count = p.tile_counts != nullptr;
                // both halves' lists are sorted descending: a pointer merge of k
                // steps gives the row's top-k; the softmax numerators go to
                // shared memory, the ids straight out, and (for the align
                // behind the route) each expert's count up by one -- a
                // shared-memory reduction whose result nothing here waits for
                int i = 0, j = 0;
                float vmax = 0.0f, sum = 0.0f;
    #pragma unroll 1
                for (int r = 0; r < p.k; ++r) {
                    const uint32_t x1 = i < p.k ? list[i * kTcBM + row] : 0u;
                    const uint32_t x0 = j < p.k ? list0[j * kTcBM + row] : 0u;
                    const bool take1 = x1 > x0;
                    const uint32_t m = take1 ? x1 : x0;
                    i += take1 ? 1 : 0;
                    j += take1 ? 0 : 1;
                    vmax = (r == 0) ? key_value(m) : vmax;
                    const float ev = expf(key_value(m) - vmax);
                    sum += ev;
                    numer[r * kTcBM + row] = ev;
                    orow[r] = key_id(m);
                    if (count) atomicAdd(&h[key_id(m)], 1);
                }
                float den = sum;
                if (!p.renorm) {  // both halves' denominators at the row's largest logit
                    const float2 d0 = den_s[row];
                    den = den_half * expf(v_half - vmax) + d0.x * expf(d0.y - vmax);
                }
                const float inv = 1.0f / den;  // one division; each weight within 1.5 ulp of ev / den
    #pragma unroll 4
                for (int r = 0; r < p.k; ++r) wrow[r] = numer[r * kTcBM + row] * inv;
                if (p.S) {  // (its count is the tile's number of rows, set below)
                    const float sh = sh_s[row];
                    orow[p.k] = p.E;
                    wrow[p.k] = p.scale * sigmoid_stable(p.shared_bf16 ? round_bf16(sh) : sh);
                }
            }
            __syncwarp();
            if (p.tile_counts) {
                asm volatile("bar.sync 1, 128;" ::: "memory");  // the 4 warps of half 1
                const int E_al = p.E + p.S;
                for (int t = 0; t < kTcTileRows / kTcCountRows; ++t) {  // tiles that hold rows
                    const int r0 = m0 + t * kTcCountRows;
                    if (r0 < p.M) {
                        const int rows_t = min(kTcCountRows, p.M - r0);  // every row has one shared slot
                        for (int e = threadIdx.x - 128; e < E_al; e += 128)
                            p.tile_counts[(int64_t)(blockIdx.x * (kTcTileRows / kTcCountRows) + t) * E_al + e] =
                                (e == p.E) ? rows_t : hist[t * E_al + e];
                    }
                }
            }
            if (!(ok && got)) set_error(p.err, kErrWaitTimeout);
        }
    }
    tc_fence_before();
    // both CTAs' epilogues are done with TMEM and no barrier of either CTA
    // can still be signalled: free the pair's TMEM, then leave
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, p.tmem_cols);
    }
    if constexpr (!LO) {
        if (p.fa_sorted != nullptr) fused_align_tail(p, smem, abort_flag + 1);
    }
}

// ------------------------------------------------------------------ host --

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    // looked up once (a function-local static is initialised exactly once,
    // also when host threads race)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    }();
    return fn;
}

bool make_tma_map_2d(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              kTcSW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                           : (kTcSW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B),
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcPlan {
    TcParams p;
    size_t smem;
    int grid;
};

static bool plan_tc(int M, int H, int E, int k, int S, TcPlan *out) {
    if (E < 32 || E > 512 || E % 32 != 0 || k < 1 || k > 32 || k > E || H < 8 || H % 8 != 0 ||
        H > 16384)
        return false;
    TcParams p{};
    p.H = H;
    p.E = E;
    p.E_valid = E;
    p.S = S;
    p.k = k;
    p.M = M;
    p.width = k + S;
    p.num_kb = (H + kTcBK - 1) / kTcBK;
    // gate pieces of at most 256 columns (one pair MMA each, N <= 256); each
    // CTA holds half of every piece's rows (a multiple of 8: whole swizzle atoms)
    p.n_pieces = (E + 255) / 256;
    p.piece_n = E / p.n_pieces;
    if (p.piece_n % 16 != 0) return false;
    uint32_t cols = 32;
    while (cols < (uint32_t)E) cols <<= 1;
    p.tmem_cols = cols;
    p.stage_bytes = (uint32_t)(kTcBM * kTcSW + (E / 2) * kTcSW);
    // misc: barriers and flags (256 B: 3*stages+2 mbarriers, TMEM slot, abort
    // flag), bias [E] fp32, expert counts [2][E+S] int32, shared gate [H, padded
    // to whole k-blocks] fp32, half 0's softmax denominators [128] (sum, max),
    // the shared logits [128]
    p.misc_bias_off = 256;
    p.misc_hist_off = 256 + (uint32_t)((E * 4 + 15) & ~15);
    p.misc_ws_off = p.misc_hist_off + (uint32_t)((2 * (E + S) * 4 + 15) & ~15);
    p.misc_den_off = p.misc_ws_off + (uint32_t)(S ? (size_t)p.num_kb * kTcBK * 4 : 0);
    const size_t misc = p.misc_den_off + (size_t)kTcBM * (sizeof(float2) + sizeof(float));
    const size_t budget = (size_t)kTcSmemLimit - 1024 - misc;
    int st = (int)(budget / p.stage_bytes);
    if (st > 6) st = 6;
    if (st < 2) return false;
    static_assert(8 * (3 * 6 + 2) + 12 <= 256, "barriers, TMEM slot and two flags fit the misc header");
    // the epilogue (candidate lists, half 0's top-k, both halves' rounded
    // logits) reuses the stage ring; the misc block follows the larger one
    const size_t ring = (size_t)st * p.stage_bytes;
    const size_t epi = (size_t)kEpiListBytes + 2 * (size_t)kTcBM * dump_row_bytes(E / 2);
    const size_t front = ring > epi ? ring : epi;
    if (1024 + front + misc > (size_t)kTcSmemLimit) return false;
    p.stages = st;
    p.misc_off = (uint32_t)front;
    out->p = p;
    out->smem = 1024 + front + misc;
    const int tiles = (M + kTcBM - 1) / kTcBM;
    out->grid = (tiles + 1) / 2 * 2;  // whole CTA pairs; a missing partner tile is all padding
    return true;
}

bool tc_route_supported(int H, int E, int k, int S) {
    TcPlan plan;
    return plan_tc(1, H, E, k, S, &plan);
}

template <int CW, bool LO, bool XQ, bool QD>
static cudaError_t launch_ng(const CUtensorMap &mx, const CUtensorMap &mw, const TcPlan &plan,
                             cudaStream_t stream) {
    static std::atomic<bool> configured[kMaxDevices];
    cudaError_t e = once_per_device(configured, [](int) {
        cudaError_t r = cudaFuncSetAttribute(tc_route_kernel<CW, LO, XQ, QD>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kTcSmemLimit);
        if (r == cudaSuccess)  // the same carveout as every other kernel of the library
            r = cudaFuncSetAttribute(tc_route_kernel<CW, LO, XQ, QD>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        return r;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;  // CTA pairs
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start before the previous kernel in the stream completes (it waits
    // for that kernel before loading hidden states or writing anything)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tc_route_kernel<CW, LO, XQ, QD>, mx, mw, plan.p);
}

cudaError_t launch_tc_route(const TcRouteLaunch &a, cudaStream_t stream) {
    TcPlan plan;
    // a logits-only launch computes its E valid gate rows padded to whole
    // 32-row groups (zero rows past E from the tensor map's fill)
    const int E_pad = a.logits_only ? (a.E + 31) / 32 * 32 : a.E;
    if (!plan_tc(a.M, a.H, E_pad, a.logits_only ? 1 : a.k, a.S, &plan)) return cudaErrorNotSupported;
    TcParams &p = plan.p;
    p.E_valid = a.E;
    p.col0 = a.col0;
    p.logits_ws = a.logits_ws;
    p.ld_logits = a.ld_logits;
    p.s_out = a.s_out;
    p.xq = a.xq;
    p.xs = a.xs;
    p.fa_A = a.fa_A;
    p.fa_sorted = a.fa_sorted;
    p.fa_eids = a.fa_eids;
    p.fa_npp = a.fa_npp;
    p.fa_sorted_cap = a.fa_sorted_cap;
    p.fa_eids_cap = a.fa_eids_cap;
    p.ticket = &reinterpret_cast<WsHeader *>(a.hdr)->ticket;
    // the fused align stages the ids and its arrays in the idle stage ring
    if (a.fa_sorted != nullptr &&
        (a.logits_only || (size_t)p.misc_off < (size_t)(kAlignSingleMax + align_smem_words(kTcThreads / 32,
                                                                                             a.E + a.S)) * 4))
        return cudaErrorNotSupported;
    p.scale = a.scale;
    p.renorm = a.renorm;
    p.shared_bf16 = a.shared_bf16;
    p.bias = a.bias;
    p.x = a.x;
    p.ld = a.ld;
    p.ws = a.ws;
    p.ids = a.ids;
    p.wts = a.wts;
    p.logits_out = a.logits_out;
    p.err = &reinterpret_cast<WsHeader *>(a.hdr)->error;
    p.tile_counts = a.tile_counts;
    p.stall = a.stall;
    p.stall_limit = a.stall_limit > 0 ? a.stall_limit : kWaitCycles;
    CUtensorMap mx, mw;
    if (!make_tma_map_2d(&mx, a.x, (uint64_t)a.H, (uint64_t)a.M, (uint64_t)a.ld * 2, kTcBK, kTcBM))
        return cudaErrorInvalidValue;
    if (!make_tma_map_2d(&mw, a.w, (uint64_t)a.H, (uint64_t)a.E, (uint64_t)a.H * 2, kTcBK,
                  (uint32_t)(p.piece_n / 2)))
        return cudaErrorInvalidValue;
    // 32-column TMEM chunks when each column half is a multiple of 32, else 16
    const bool wide = (E_pad / 2) % 32 == 0;
    // the e4m3 hidden states are a separate instantiation, so that a route
    // without them keeps the plain kernel's registers and code
    // quads (QD) as the threshold units for column halves of at most 128
    const bool qd = !a.logits_only && E_pad / 2 <= 128;
    if (a.xq != nullptr) {
        if (a.logits_only)
            return wide ? launch_ng<32, true, true, false>(mx, mw, plan, stream)
                        : launch_ng<16, true, true, false>(mx, mw, plan, stream);
        if (qd)
            return wide ? launch_ng<32, false, true, true>(mx, mw, plan, stream)
                        : launch_ng<16, false, true, true>(mx, mw, plan, stream);
        return wide ? launch_ng<32, false, true, false>(mx, mw, plan, stream)
                    : launch_ng<16, false, true, false>(mx, mw, plan, stream);
    }
    if (a.logits_only)
        return wide ? launch_ng<32, true, false, false>(mx, mw, plan, stream)
                    : launch_ng<16, true, false, false>(mx, mw, plan, stream);
    if (qd)
        return wide ? launch_ng<32, false, false, true>(mx, mw, plan, stream)
                    : launch_ng<16, false, false, true>(mx, mw, plan, stream);
    return wide ? launch_ng<32, false, false, false>(mx, mw, plan, stream)
                : launch_ng<16, false, false, false>(mx, mw, plan, stream);
}

}  // namespace smr
