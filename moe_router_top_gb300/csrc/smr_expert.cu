// smr_expert.cu -- the consumer of the align: the expert GEMM over
// sorted_token_ids / expert_ids with the num_tokens_post_padded early exit.
//
// "[ROCm][Kernel] W4A16 MoE prefill: M-aware moe_align block size (1.6x
// TTFT)", Purpose: the fused MoE GEMM takes the aligned rows in blocks of
// BLOCK_SIZE_M = A; block b runs the full K contraction against the weights
// of expert expert_ids[b], and a block at or past num_tokens_post_padded
// returns at once -- so its work is proportional to npp, which is what the
// M-aware alignment tier shrinks. Here with bf16 expert weights and fp32
// outputs, to show that tier end to end.
//
// GB300 design: one CTA (4 warps) per (block, 256- or 128-column tile of N).
//  - the grid covers the whole capacity (the host cannot know npp without a
//    synchronisation); a CTA reads npp and returns if its block starts at or
//    past it;
//  - the A operand is the block's A hidden-state rows, gathered by
//    sorted_token_ids (slot / width = token; padding rows zero-filled) with
//    16-byte cp.async copies written straight into the 128-byte-swizzled
//    K-major layout the tensor core reads, then handed to it with
//    fence.proxy.async; the B operand (the expert's weight tile) by TMA;
//  - tcgen05.mma (M = A, N = 256 or 128, K = 16) issued by one thread into
//    TMEM over a ring of 4 stages; the epilogue reads TMEM back and stores
//    every routed row's fp32 outputs at its slot.
// Every wait is bounded; a wait that gives up sets the workspace's error bit.
#include <cudaTypedefs.h>

#include "smr_device.cuh"
#include "smr_launch.h"

namespace smr {

constexpr int kXgThreads = 128;
constexpr int kXgBK = 64;   // k-block: 64 bf16 = one 128-byte swizzled row
constexpr int kXgStages = 4;

struct XgParams {
    const uint16_t *x;
    int64_t ld;
    int width, H, N, BN, num_experts, num_kb;
    int64_t numel;
    const int32_t *sorted, *eids, *npp;
    float *out;
    uint32_t *err;
    uint32_t stage_bytes, misc_off, tmem_cols;
};

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// A: the block's rows (the MMA's M), 64 or 128.
template <int A>
__global__ void __launch_bounds__(kXgThreads, 1)
expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const XgParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    constexpr int ST = kXgStages;
    constexpr int kCopies = A * (kXgBK / 8) / kXgThreads;  // 16-byte A copies per thread per k-block
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x, nt = blockIdx.y;

    griddep_launch_dependents();
    griddep_wait();  // the align's outputs come from the previous kernel
    const int npp = __ldcg(p.npp);
    if ((int64_t)b * A >= npp) return;  // the early exit: a block past npp does nothing
    const int e = __ldcg(p.eids + b);
    if ((unsigned)e >= (unsigned)p.num_experts) {  // only a corrupted align output gets here
        if (tid == 0) set_error(p.err, kErrBadId);
        return;
    }

    uint8_t *misc = smem + p.misc_off;
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);  // TMA: the expert tile landed
    uint64_t *mma_done = full + ST;                        // the MMAs are done with the stage
    uint64_t *accum = mma_done + ST;                       // every MMA is done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *slot = reinterpret_cast<int *>(misc + 128);       // [A] the block's slots (-1: padding)

    for (int r = tid; r < A; r += kXgThreads) {
        const int i = __ldcg(p.sorted + (int64_t)b * A + r);
        const bool real = (unsigned)i < (unsigned)p.numel;
        if (!real && i != p.numel) set_error(p.err, kErrBadSlot);  // neither a slot nor the sentinel
        slot[r] = real ? i : -1;
    }
    if (tid == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&mma_done[s]), 1);
        }
        mbar_init(smem_u32(accum), 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tm_w);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // this thread's A copies: chunk c (16 bytes) of block row r lands at
    // r * 128 + ((c ^ (r & 7)) << 4), the 128-byte swizzle
    const uint16_t *src[kCopies];
    uint32_t dst_off[kCopies], src_bytes[kCopies];
#pragma unroll
    for (int j = 0; j < kCopies; ++j) {
        const int id = tid + j * kXgThreads, r = id >> 3, c = id & 7;
        const int i = slot[r];
        src[j] = p.x + (int64_t)(i < 0 ? 0 : i / p.width) * p.ld + c * 8;
        src_bytes[j] = i < 0 ? 0u : 16u;  // padding rows read as zeros
        dst_off[j] = (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
    }
    const uint32_t ring = smem_u32(smem);
    const uint32_t b_tile_bytes = (uint32_t)p.BN * 128u;
    auto load_stage = [&](int kb, int s) {
        const uint32_t base = ring + (uint32_t)s * p.stage_bytes;
#pragma unroll
        for (int j = 0; j < kCopies; ++j) cp_async_16(base + dst_off[j], src[j] + kb * kXgBK, src_bytes[j]);
        if (tid == 0) {
            mbar_arrive_expect_tx(smem_u32(&full[s]), b_tile_bytes);
            tma_load_2d(base + A * 128, &tm_w, kb * kXgBK, e * p.N + nt * p.BN, smem_u32(&full[s]));
        }
    };

    const uint32_t idesc = idesc_bf16_f32(A, p.BN);
    const int nkb = p.num_kb;
    int issued = 0;  // k-blocks whose loads were issued
    for (; issued < ST - 1 && issued < nkb; ++issued) {
        load_stage(issued, issued);
        cp_async_commit();
    }
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % ST;
        const int kn = kb + ST - 1;
        bool w_ok = true;
        if (kn < nkb) {
            const int sn = kn % ST;
            // the stage held k-block kn - ST: refilled once its MMAs are done
            if (kn >= ST)
                w_ok = mbar_wait_bounded(smem_u32(&mma_done[sn]), (uint32_t)((kn / ST) - 1) & 1u, abort_flag);
            if (w_ok) {
                load_stage(kn, sn);
                issued = kn + 1;
            }
        }
        cp_async_commit();
        cp_async_wait<ST - 1>();  // this thread's copies of k-block kb have landed
        // the generic-proxy writes of the copies become visible to the tensor
        // core (async proxy), then to the issuing thread; one decision for the
        // whole CTA, so that every thread leaves the loop at the same barrier
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (!__syncthreads_and(w_ok && !*abort_flag)) {
            ok = false;
            break;
        }
        if (tid == 0) {
            if (mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)(kb / ST) & 1u, abort_flag)) {
                tc_fence_after();
                const uint32_t a_base = ring + (uint32_t)s * p.stage_bytes;
                const uint32_t b_base = a_base + A * 128;
#pragma unroll
                for (int kk = 0; kk < kXgBK / 16; ++kk)
                    tc_mma_bf16(tmem, smem_desc_sw<128>(a_base + kk * 32), smem_desc_sw<128>(b_base + kk * 32),
                                idesc, (kb | kk) != 0 ? 1u : 0u);
                tc_commit(smem_u32(&mma_done[s]));
            }
        }
    }
    if (tid == 0) tc_commit(smem_u32(accum));  // after the MMAs issued (if any)
    cp_async_wait<0>();
    // every issued MMA completes before TMEM is read or freed, also after an
    // abort (a wait bounded by time only)
    volatile int never = 0;
    const bool done = mbar_wait_bounded(smem_u32(accum), 0u, &never);
    tc_fence_after();
    ok = __syncthreads_and(ok && done && !*abort_flag);
    if (!ok) {
        // a wait gave up: the outputs of this block are not written; the
        // expert tiles still in flight land before the CTA leaves
        if (tid == 0) {
            set_error(p.err, kErrWaitTimeout);
            for (int kb = issued - ST > 0 ? issued - ST : 0; kb < issued; ++kb) {
                volatile int drain = 0;
                mbar_wait_bounded(smem_u32(&full[kb % ST]), (uint32_t)(kb / ST) & 1u, &drain);
            }
        }
    } else {
        // TMEM -> fp32 rows at their slots. M = 128: block row r is TMEM lane
        // r; M = 64: rows 16q..16q+15 sit in lanes 32q..32q+15 (the M = 64
        // accumulator uses the first 16 lanes of each 32-lane quarter)
        const int r = A == 128 ? warp * 32 + lane : warp * 16 + (lane & 15);
        const int i = (A == 128 || lane < 16) ? slot[r] : -1;
        float *orow = p.out + (int64_t)(i < 0 ? 0 : i) * p.N + nt * p.BN;
#pragma unroll 1
        for (int ch = 0; ch < p.BN / 32; ++ch) {
            uint32_t v[32];
            tmem_ld32_async(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(ch * 32), v);
            tmem_wait_ld(v);
            if (i >= 0) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    reinterpret_cast<float4 *>(orow + ch * 32)[u] =
                        make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                    __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

cudaError_t launch_expert_gemm(const ExpertGemmLaunch &a, cudaStream_t stream) {
    if ((a.A != 64 && a.A != 128) || a.N % 128 != 0 || a.H % kXgBK != 0 || a.max_blocks < 1)
        return cudaErrorNotSupported;
    XgParams p{};
    p.x = a.x;
    p.ld = a.ld;
    p.width = a.width;
    p.H = a.H;
    p.N = a.N;
    p.BN = a.N % 256 == 0 ? 256 : 128;
    p.num_experts = a.num_experts;
    p.num_kb = a.H / kXgBK;
    p.numel = a.numel;
    p.sorted = a.sorted;
    p.eids = a.eids;
    p.npp = a.npp;
    p.out = a.out;
    p.err = &reinterpret_cast<WsHeader *>(a.hdr)->error;
    p.stage_bytes = (uint32_t)(a.A + p.BN) * 128u;
    p.misc_off = (uint32_t)kXgStages * p.stage_bytes;
    p.tmem_cols = (uint32_t)p.BN;
    const size_t smem = 1024 + p.misc_off + 128 + (size_t)a.A * 4;
    CUtensorMap mw;
    if (!make_tma_map_2d(&mw, a.w, (uint64_t)a.H, (uint64_t)a.num_experts * a.N, (uint64_t)a.H * 2, kXgBK,
                         (uint32_t)p.BN))
        return cudaErrorInvalidValue;
    static std::atomic<bool> configured[2][kMaxDevices];
    const void *kern = a.A == 128 ? (const void *)expert_gemm_kernel<128> : (const void *)expert_gemm_kernel<64>;
    cudaError_t e = once_per_device(configured[a.A == 128], [kern](int) {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        return r;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.max_blocks, (unsigned)(a.N / p.BN), 1);
    cfg.blockDim = dim3(kXgThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.A == 128) return cudaLaunchKernelEx(&cfg, expert_gemm_kernel<128>, mw, p);
    return cudaLaunchKernelEx(&cfg, expert_gemm_kernel<64>, mw, p);
}

}  // namespace smr
