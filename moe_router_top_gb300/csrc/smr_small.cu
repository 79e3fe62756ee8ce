// smr_small.cu -- single-launch route (+ align) for M <= 16 tokens.
//
// What it computes is the one-launch small-M router of "[AMD] One-launch
// small-M MoE router for Qwen3.5 on gfx950", Modifications: every CTA
// computes a few of the E+S gate rows for all M tokens with fp32
// accumulation; the last CTA to finish (self-resetting ticket, no spin-wait)
// rounds the routed logits to bf16, selects the top-k with the lowest id
// winning ties, applies softmax + renormalisation, writes the shared slot
// (E, sigmoid(s) * scale) and, when asked, runs moe_align_block_size on the
// M*(k+S) ids it just produced ("[ROCm][Kernel] W4A16 MoE prefill: M-aware
// moe_align block size", Purpose) -- all in one launch.
//
// GB300 design:
//  - the gate stream is HBM-bound (4 MiB at E=512, H=4096): each of the
//    ~129 CTAs (one wave on 152 SMs) issues all of its 16-byte weight loads
//    (ld.global.nc, no L1 allocation) before any arithmetic, so the whole
//    matrix is in flight at once;
//  - the tokens' hidden states go to shared memory with cp.async into
//    thread-private slots (no CTA barrier), each x chunk is reused by all R
//    gate rows of the CTA;
//  - the per-thread partial dot products are reduced with a warp butterfly
//    reduce-scatter (R*MT values, 5 shuffle stages) and a fixed-order sum
//    over the 8 warps, so results are deterministic;
//  - the top-k tail is warp-parallel: one warp per token, the E logits as
//    ordered 32-bit keys spread over 32 lanes, k rounds of one redux.sync
//    max -- instead of k serial argmax passes over the row.
#include "smr_device.cuh"
#include "smr_launch.h"

namespace smr {

constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kCPT = 2;  // 16-byte chunks of a row per thread per pass

struct SmallParams {
    SmallRouteLaunch a;
    int rows;  // E + S
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
}

template <int N>
struct Log2 { static constexpr int value = 1 + Log2<N / 2>::value; };
template <>
struct Log2<1> { static constexpr int value = 0; };

// Top-k of one token row in one warp. logits: fp32 [E] (read through L2);
// writes ids/weights for slots 0..k-1 and returns the slot's id in lane j < k
// (-1 elsewhere).
__device__ __forceinline__ int warp_topk_row(const float *logits, const float *bias, int E, int k,
                                             uint16_t *logits_out, int32_t *ids, float *wts) {
    const int lane = threadIdx.x & 31;
    const int nk = (E + 31) >> 5;
    uint32_t key[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        key[i] = 0u;
        const int e = lane + 32 * i;
        if (i < nk && e < E) {
            float z = __ldcg(logits + e);
            if (bias) z += __ldg(bias + e);
            const float zr = round_bf16(z);
            key[i] = make_key(zr, e);
            if (logits_out) logits_out[e] = (uint16_t)(__float_as_uint(zr) >> 16);
        }
    }
    uint32_t lm = 0u;
#pragma unroll
    for (int i = 0; i < 32; ++i) lm = max(lm, key[i]);
    uint32_t mine = 0u, first = 0u;
    for (int r = 0; r < k; ++r) {
        const uint32_t g = __reduce_max_sync(0xffffffffu, lm);
        if (r == 0) first = g;
        if (lane == r) mine = g;
        if (lm == g) {  // the single lane holding the winner removes it
            lm = 0u;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (key[i] == g) key[i] = 0u;
                lm = max(lm, key[i]);
            }
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

template <int R, int MT>
__global__ void __launch_bounds__(kSmallThreads) small_route_kernel(const SmallParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    const SmallRouteLaunch &p = P.a;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rows = P.rows;
    const int row0 = blockIdx.x * R;
    const int nch = p.H >> 3;
    constexpr int N = R * MT;

    uint4 *xs = reinterpret_cast<uint4 *>(smem);  // [MT][kCPT][256], thread-private slots
    float *red = reinterpret_cast<float *>(smem + MT * kCPT * kSmallThreads * 16);  // [8][N]
    __shared__ int s_last;

    // ---- 1. gate rows x tokens: fp32 partial dot products per thread ----
    float acc[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.0f;

    for (int c0 = 0; c0 < nch; c0 += kSmallThreads * kCPT) {
        uint4 wv[R][kCPT];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = row0 + r;
            const uint16_t *src = (row < p.E) ? p.w + (int64_t)row * p.H : p.ws;
#pragma unroll
            for (int j = 0; j < kCPT; ++j) {
                const int c = c0 + j * kSmallThreads + tid;
                wv[r][j] = (row < rows && c < nch) ? ld_stream_v4(src + (int64_t)c * 8)
                                                   : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < p.M) {
#pragma unroll
                for (int j = 0; j < kCPT; ++j) {
                    const int c = c0 + j * kSmallThreads + tid;
                    if (c < nch)
                        cp_async16(&xs[(m * kCPT + j) * kSmallThreads + tid],
                                   p.x + (int64_t)m * p.ld + (int64_t)c * 8);
                }
            }
        }
        cp_async_wait_all();
#pragma unroll
        for (int j = 0; j < kCPT; ++j) {
            const int c = c0 + j * kSmallThreads + tid;
            if (c < nch) {
                float wf[R][8];
#pragma unroll
                for (int r = 0; r < R; ++r) unpack8(wv[r][j], wf[r]);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < p.M) {
                        float xf[8];
                        unpack8(xs[(m * kCPT + j) * kSmallThreads + tid], xf);
#pragma unroll
                        for (int r = 0; r < R; ++r)
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[r][m] = fmaf(wf[r][e], xf[e], acc[r][m]);
                    }
                }
            }
        }
    }

    // ---- 2. reduce over the CTA: warp butterfly reduce-scatter + 8 warps ----
    float v[N];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) v[r * MT + m] = acc[r][m];
    constexpr int LOGN = Log2<N>::value;
    constexpr int STEPS = LOGN < 5 ? LOGN : 5;
#pragma unroll
    for (int s = 0; s < STEPS; ++s) {
        const int o = 16 >> s;
        const int half = N >> (s + 1);
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    constexpr int KEEP = (N >> STEPS) > 0 ? (N >> STEPS) : 1;  // values per lane now
#pragma unroll
    for (int o = 16 >> STEPS; o >= 1; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    if (N >= 32) {
#pragma unroll
        for (int j = 0; j < KEEP; ++j) red[warp * N + lane * KEEP + j] = v[j];
    } else if ((lane & ((32 >> STEPS) - 1)) == 0) {
        red[warp * N + (lane >> (5 - STEPS))] = v[0];
    }
    __syncthreads();
    if (tid < N) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < kSmallWarps; ++w) t += red[w * N + tid];
        const int r = tid / MT, m = tid % MT, row = row0 + r;
        if (row < rows && m < p.M) p.scratch[(int64_t)m * rows + row] = t;
        __threadfence();
    }
    __syncthreads();

    // ---- 3. hand-off: the last CTA to arrive runs the tail ----
    WsHeader *hdr = reinterpret_cast<WsHeader *>(p.hdr);
    if (tid == 0) {
        const unsigned t = atomicAdd(&hdr->ticket, 1u);
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) hdr->ticket = 0u;  // every CTA has arrived: reset for the next call

    // ---- 4. tail: top-k + softmax + shared slot, one warp per token ----
    const int width = p.k + p.S;
    int32_t *ids_s = reinterpret_cast<int32_t *>(smem);  // [M*width], reuses x staging
    int *align_smem = ids_s + kSmallMaxM * 32;
    __syncthreads();
    for (int m = warp; m < p.M; m += kSmallWarps) {
        const float *zrow = p.scratch + (int64_t)m * rows;
        const int id = warp_topk_row(zrow, p.bias, p.E, p.k,
                                     p.logits_out ? p.logits_out + (int64_t)m * p.E : nullptr,
                                     p.ids + (int64_t)m * width, p.wts + (int64_t)m * width);
        if (lane < p.k) ids_s[m * width + lane] = id;
        if (p.S && lane == p.k) {
            const float s = __ldcg(zrow + p.E);
            p.ids[(int64_t)m * width + p.k] = p.E;
            p.wts[(int64_t)m * width + p.k] = p.scale * sigmoid_stable(s);
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
    align_blocks(npp, p.A, rows, as.cnt, as, numel, p.sorted, p.expert_ids, warp, kSmallWarps);
    if (tid == 0) *p.npp = npp;
}

template <int R, int MT>
static cudaError_t launch_rm(const SmallParams &P, int grid, size_t smem, cudaStream_t stream) {
    auto kern = small_route_kernel<R, MT>;
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             160 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    kern<<<grid, kSmallThreads, smem, stream>>>(P);
    return cudaGetLastError();
}

template <int R>
static cudaError_t launch_r(const SmallParams &P, int MT, int grid, size_t smem,
                            cudaStream_t stream) {
    switch (MT) {
        case 1: return launch_rm<R, 1>(P, grid, smem, stream);
        case 2: return launch_rm<R, 2>(P, grid, smem, stream);
        case 4: return launch_rm<R, 4>(P, grid, smem, stream);
        case 8: return launch_rm<R, 8>(P, grid, smem, stream);
        default: return launch_rm<R, 16>(P, grid, smem, stream);
    }
}

cudaError_t launch_small_route(const SmallRouteLaunch &a, cudaStream_t stream) {
    if (a.M <= 0 || a.M > kSmallMaxM) return cudaErrorInvalidValue;
    SmallParams P;
    P.a = a;
    P.rows = a.E + a.S;
    const int R = P.rows <= 160 ? 1 : (P.rows <= 320 ? 2 : 4);
    int MT = 1;
    while (MT < a.M) MT <<= 1;
    const int grid = (P.rows + R - 1) / R;
    const size_t stage = (size_t)MT * kCPT * kSmallThreads * 16 + (size_t)kSmallWarps * R * MT * 4;
    const size_t tail = (size_t)(kSmallMaxM * 32 + align_smem_words(kSmallWarps, P.rows)) * 4;
    const size_t smem = stage > tail ? stage : tail;
    switch (R) {
        case 1: return launch_r<1>(P, MT, grid, smem, stream);
        case 2: return launch_r<2>(P, MT, grid, smem, stream);
        default: return launch_r<4>(P, MT, grid, smem, stream);
    }
}

}  // namespace smr
