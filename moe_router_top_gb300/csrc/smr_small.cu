// smr_small.cu -- single-launch route (+ align) for M <= 16 tokens.
//
// What it computes is the one-launch small-M router of "[AMD] One-launch
// small-M MoE router for Qwen3.5 on gfx950", Modifications: the E+S gate rows
// are computed for all M tokens with fp32 accumulation across CTAs; the last
// CTA to finish (self-resetting ticket, no spin-wait) rounds the routed logits
// to bf16, selects the top-k with the lowest id winning ties, applies softmax +
// renormalisation, writes the shared slot (E, sigmoid(s) * scale) and, when
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
//  - the 8 warps' partial sums are added in a fixed order and stored per K
//    range; the tail adds the KQ ranges in a fixed order, so results are
//    deterministic;
//  - the tail is warp-parallel: one warp per token, each lane holds E/32
//    ordered 32-bit keys sorted in registers, k rounds of one redux.sync max
//    and a register shift pop the winner -- instead of k serial argmax
//    passes over the row.
#include "smr_device.cuh"
#include "smr_launch.h"

namespace smr {

constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSliceK = 32;           // K elements per slice (two m16n8k16 steps)
constexpr int kMaxSlicesPerWarp = 4;  // slices whose loads are in flight at once

struct SmallParams {
    SmallRouteLaunch a;
    int rows;     // E + S
    int KQ;       // K ranges per 16-row group
    int slices;   // ceil(H / 32)
    int per_cta;  // slices per K range
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Sort NK keys descending in registers (bitonic network).
template <int NK>
__device__ __forceinline__ void sort_keys_desc(uint32_t (&a)[NK]) {
#pragma unroll
    for (int size = 2; size <= NK; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < NK; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = ((i & size) == 0);
                    const uint32_t hi = max(a[i], a[j]), lo = min(a[i], a[j]);
                    a[i] = desc ? hi : lo;
                    a[j] = desc ? lo : hi;
                }
            }
        }
    }
}

// Top-k of one token row in one warp. part: fp32 partial logits laid out
// [KQ][M][rows]; this token's first range starts at part, later ranges are
// kq_stride apart. Writes ids and weights of slots 0..k-1 and returns the
// slot's id in lanes j < k (-1 elsewhere).
template <int NK>
__device__ __forceinline__ int warp_topk_row(const float *part, int KQ, int64_t kq_stride, int E,
                                             int k, const float *bias, uint16_t *logits_out,
                                             int32_t *ids, float *wts) {
    const int lane = threadIdx.x & 31;
    float z[NK];
#pragma unroll
    for (int i = 0; i < NK; ++i) z[i] = 0.0f;
    // all partial loads of a pair of ranges are issued before any is used:
    // addresses are clamped into the row, out-of-row lanes are masked below
    int q = 0;
    for (; q + 2 <= KQ; q += 2) {
        float v0[NK], v1[NK];
#pragma unroll
        for (int i = 0; i < NK; ++i) {
            const int e = min(lane + 32 * i, E - 1);
            v0[i] = __ldcg(part + q * kq_stride + e);
            v1[i] = __ldcg(part + (q + 1) * kq_stride + e);
        }
#pragma unroll
        for (int i = 0; i < NK; ++i) z[i] = (z[i] + v0[i]) + v1[i];
    }
    if (q < KQ) {
#pragma unroll
        for (int i = 0; i < NK; ++i) z[i] += __ldcg(part + q * kq_stride + min(lane + 32 * i, E - 1));
    }
    uint32_t key[NK];
#pragma unroll
    for (int i = 0; i < NK; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0u;
        if (e < E) {
            const float zr = round_bf16(bias ? z[i] + __ldg(bias + e) : z[i]);
            key[i] = make_key(zr, e);
            if (logits_out) logits_out[e] = (uint16_t)(__float_as_uint(zr) >> 16);
        }
    }
    sort_keys_desc<NK>(key);
    uint32_t mine = 0u, first = 0u;
    for (int r = 0; r < k; ++r) {
        const uint32_t gmax = __reduce_max_sync(0xffffffffu, key[0]);
        if (r == 0) first = gmax;
        if (lane == r) mine = gmax;
        if (key[0] == gmax) {  // the single lane holding the winner pops it
#pragma unroll
            for (int i = 0; i + 1 < NK; ++i) key[i] = key[i + 1];
            key[NK - 1] = 0u;
        }
    }
    // softmax over the selected logits (renormalised top-k)
    const float vmax = key_value(first);
    const float ev = (lane < k) ? expf(key_value(mine) - vmax) : 0.0f;
    float sum = ev;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    int id = -1;
    if (lane < k) {
        id = key_id(mine);
        ids[lane] = id;
        wts[lane] = ev / sum;
    }
    return id;
}

template <int NB>  // N blocks of 8 tokens: 1 (M <= 8) or 2 (M <= 16)
__global__ void __launch_bounds__(kSmallThreads) small_route_kernel(const SmallParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    const SmallRouteLaunch &p = P.a;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;  // mma fragment coordinates
    const int rows = P.rows;
    const int rg = blockIdx.x / P.KQ, kq = blockIdx.x % P.KQ;
    const int row0 = rg * 16;
    __shared__ int s_last;

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
    for (int s0 = s_beg + warp; s0 < s_end; s0 += kSmallWarps * kMaxSlicesPerWarp) {
        uint4 va[kMaxSlicesPerWarp], vb[kMaxSlicesPerWarp], x0[kMaxSlicesPerWarp],
            x1[kMaxSlicesPerWarp];
#pragma unroll
        for (int j = 0; j < kMaxSlicesPerWarp; ++j) {
            const int s = s0 + j * kSmallWarps;
            const int k0 = s * kSliceK + 8 * t;
            const int kc = min(k0, p.H - 8);  // clamped so every load stays in bounds
            va[j] = ld_stream_v4(wa + kc);
            vb[j] = ld_stream_v4(wb + kc);
            x0[j] = __ldg(reinterpret_cast<const uint4 *>(xa + kc));
            if (NB > 1) x1[j] = __ldg(reinterpret_cast<const uint4 *>(xb + kc));
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

    // ---- 2. sum the 8 warps in a fixed order, store this K range's partials ----
    float *red = reinterpret_cast<float *>(smem);  // [8 warps][16 rows][16 tokens]
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int tok = nb * 8 + 2 * t;
        red[(warp * 16 + g) * 16 + tok] = acc[nb][0];
        red[(warp * 16 + g) * 16 + tok + 1] = acc[nb][1];
        red[(warp * 16 + g + 8) * 16 + tok] = acc[nb][2];
        red[(warp * 16 + g + 8) * 16 + tok + 1] = acc[nb][3];
    }
    __syncthreads();
    {
        const int r = tid >> 4, m = tid & 15;  // 256 threads = 16 rows x 16 tokens
        if (m < p.M && m < NB * 8 && row0 + r < rows) {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kSmallWarps; ++w) v += red[(w * 16 + r) * 16 + m];
            p.scratch[((int64_t)kq * p.M + m) * rows + row0 + r] = v;
            __threadfence();
        }
    }
    __syncthreads();

    // ---- 3. hand-off: the last CTA to arrive runs the tail ----
    WsHeader *hdr = reinterpret_cast<WsHeader *>(p.hdr);
    if (tid == 0) {
        const unsigned tk = atomicAdd(&hdr->ticket, 1u);
        s_last = (tk == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) hdr->ticket = 0u;  // every CTA has arrived: reset for the next call

    // ---- 4. tail: top-k + softmax + shared slot, one warp per token ----
    const int width = p.k + p.S;
    int32_t *ids_s = reinterpret_cast<int32_t *>(smem);  // [M*width]
    int *align_smem = ids_s + kSmallMaxM * 32;
    const int64_t kq_stride = (int64_t)p.M * rows;
    const int nk = (p.E + 31) >> 5;
    __syncthreads();
    for (int m = warp; m < p.M; m += kSmallWarps) {
        const float *zrow = p.scratch + (int64_t)m * rows;
        uint16_t *lrow = p.logits_out ? p.logits_out + (int64_t)m * p.E : nullptr;
        int32_t *irow = p.ids + (int64_t)m * width;
        float *wrow = p.wts + (int64_t)m * width;
        int id;
        if (nk <= 4)
            id = warp_topk_row<4>(zrow, P.KQ, kq_stride, p.E, p.k, p.bias, lrow, irow, wrow);
        else if (nk <= 8)
            id = warp_topk_row<8>(zrow, P.KQ, kq_stride, p.E, p.k, p.bias, lrow, irow, wrow);
        else if (nk <= 16)
            id = warp_topk_row<16>(zrow, P.KQ, kq_stride, p.E, p.k, p.bias, lrow, irow, wrow);
        else
            id = warp_topk_row<32>(zrow, P.KQ, kq_stride, p.E, p.k, p.bias, lrow, irow, wrow);
        if (lane < p.k) ids_s[m * width + lane] = id;
        if (p.S && lane == p.k) {
            float s = 0.0f;
            for (int q = 0; q < P.KQ; ++q) s += __ldcg(zrow + q * kq_stride + p.E);
            irow[p.k] = p.E;
            wrow[p.k] = p.scale * sigmoid_stable(s);
            ids_s[m * width + p.k] = p.E;
        }
    }
    if (p.sorted == nullptr) return;

    // ---- 5. moe_align_block_size on the M*width ids of this call ----
    __syncthreads();
    const int numel = p.M * width;
    AlignSmem as = align_carve(align_smem, rows);
    align_count(ids_s, numel, rows, as, &hdr->error);
    const int npp = align_offsets(as.cnt, rows, p.A, as);
    align_scatter(ids_s, numel, rows, 0, as, false, p.sorted);
    align_fill(p.A, rows, as.cnt, as, numel, p.sorted, p.expert_ids, tid, kSmallThreads);
    if (tid == 0) *p.npp = npp;
}

template <int NB>
static cudaError_t launch_nb(const SmallParams &P, int grid, size_t smem, cudaStream_t stream) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(small_route_kernel<NB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    small_route_kernel<NB><<<grid, kSmallThreads, smem, stream>>>(P);
    return cudaGetLastError();
}

int small_route_k_ranges(int E, int S, int H) {
    // enough CTAs for one wave on ~150 SMs, at least one slice per warp
    const int groups = (E + S + 15) / 16;
    const int slices = (H + kSliceK - 1) / kSliceK;
    int KQ = 150 / groups;
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
    static void *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (addr[dev] == nullptr) {
        // first use on this device (with it current): resolve the address and
        // zero the hand-off counter and error word, which later calls leave
        // at zero themselves
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        e = cudaMemset(p, 0, sizeof(WsHeader));
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_small_route(const SmallRouteLaunch &a, cudaStream_t stream) {
    if (a.M <= 0 || a.M > kSmallMaxM) return cudaErrorInvalidValue;
    SmallParams P;
    P.a = a;
    P.rows = a.E + a.S;
    P.slices = (a.H + kSliceK - 1) / kSliceK;
    P.KQ = small_route_k_ranges(a.E, a.S, a.H);
    P.per_cta = (P.slices + P.KQ - 1) / P.KQ;
    const int groups = (P.rows + 15) / 16;
    const int grid = groups * P.KQ;
    const size_t stage = (size_t)kSmallWarps * 16 * 16 * 4;
    const size_t tail = (size_t)(kSmallMaxM * 32 + align_smem_words(kSmallWarps, P.rows)) * 4;
    const size_t smem = stage > tail ? stage : tail;
    return a.M <= 8 ? launch_nb<1>(P, grid, smem, stream) : launch_nb<2>(P, grid, smem, stream);
}

}  // namespace smr
