// smr_device.cuh -- device helpers shared by the routing kernels (sm_103a).
//
// Contents: workspace header, bf16 rounding and the ordered selection key,
// inline-PTX wrappers (mbarrier, TMA, tcgen05), and the single-CTA
// moe_align_block_size routine used by the fused small-M kernel and by the
// standalone align kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace smr {

// ------------------------------------------------------------ workspace --

// Sticky error bits in the workspace header.
constexpr uint32_t kErrBadId = 1u;        // align saw an id outside [0, E_al)
constexpr uint32_t kErrWaitTimeout = 2u;  // a bounded wait gave up
constexpr uint32_t kErrBadSlot = 4u;      // an align output position fell outside its array (skipped)

// First 256 bytes of every workspace. Zeroed once by the caller; afterwards
// only the error word (set on errors, cleared by the caller), the small
// route's call tag (advanced by every small-M call) and the fused align's
// ticket (back at zero after every call) change.
struct WsHeader {
    uint32_t unused;  // zero
    uint32_t error;   // sticky error bits (kErr*)
    uint32_t epoch;   // small route: tag of the last completed call (top bit set once used)
    uint32_t ticket;  // tcgen05 route with the align fused: CTAs done (back to 0 at the end)
    uint32_t reserved[60];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// ------------------------------------------------------ bf16 and keys ----

// Round an fp32 logit to bf16 (round to nearest even) and return it as fp32.
// -0 is folded into +0 (adding +0.0f under round-to-nearest), so that equal
// values compare and tie-break by id only.
__device__ __forceinline__ float round_bf16(float z) {
    return __bfloat162float(__float2bfloat16_rn(z)) + 0.0f;
}

// Ordered 32-bit selection key of a bf16-valued logit and its expert id:
// the high half maps the bf16 bit pattern to an unsigned order that matches
// the numeric order; the low half is 0xFFFF - id, so among equal values the
// lower id has the larger key. One unsigned max then selects by
// (value desc, id asc) -- the argmax key of "Netra Kernel ...", Sampling:
// make small batches large enough, restated for bf16 logits. Valid keys are
// never 0 (id <= 1024), so 0 marks an empty or removed entry.
__device__ __forceinline__ uint32_t make_key(float zr, int id) {
    uint32_t b = __float_as_uint(zr) >> 16;
    uint32_t ord = (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
    return (ord << 16) | (0xFFFFu - (uint32_t)id);
}
__device__ __forceinline__ int key_id(uint32_t key) { return (int)(0xFFFFu - (key & 0xFFFFu)); }
__device__ __forceinline__ float key_value(uint32_t key) {
    uint32_t ord = key >> 16;
    uint32_t b = (ord & 0x8000u) ? (ord & 0x7FFFu) : (~ord & 0xFFFFu);
    return __uint_as_float(b << 16);
}

// sigmoid(s) = 1 / (1 + exp(-s)), evaluated as exp(s) / (1 + exp(s)) for
// s < 0 so that tiny results keep their (possibly subnormal) value instead of
// flushing through 1 / (1 + inf).
__device__ __forceinline__ float sigmoid_stable(float s) {
    if (s >= 0.0f) return 1.0f / (1.0f + expf(-s));
    const float e = expf(s);
    return e / (1.0f + e);
}

// Unpack 8 bf16 (one 16-byte chunk) to fp32.
__device__ __forceinline__ void unpack8(const uint4 &v, float f[8]) {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xFFFF0000u);
    f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// Streaming 16-byte load of read-only data that is used once (gate weights).
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ void set_error(uint32_t *err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------ mbarrier ---

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}"
                 ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 " selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait: gives up after `limit` SM cycles (by default 2^32, about 2 s
// at the maximum clock) or as soon as *abort becomes non-zero; on giving up
// it sets *abort.
constexpr long long kWaitCycles = 1ll << 32;
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort,
                                                  long long limit = kWaitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            return false;
        }
    }
}

// ------------------------------------------------------------- mma.sync ---

// D += A (16x16, row-major fragments a0-a3) x B (16x8, column-major b0-b1),
// bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ----------------------------------------------------------------- TMA ---

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Cluster-wide barrier (every thread of every CTA in the cluster, converged
// warps), release/acquire ordered.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_sync(), for work placed between them.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// A hint: the box of a 2-D tensor map at {c0, c1} (c0 as for a load: a
// multiple of 16 bytes) into L2; nothing lands in shared memory and no
// value is read.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(c0), "r"(c1)
                 : "memory");
}

// ------------------------------------------------------------- tcgen05 ---

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- single-CTA (cta_group::1) forms (the expert GEMM).
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation, one CTA.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive on an mbarrier of this CTA once all previously issued MMAs of this
// thread have completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}
// TMA 2-D tile load into this CTA's shared memory, completing bytes on an
// mbarrier of this CTA.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar) : "memory");
}

// ---- CTA-pair (cta_group::2) forms: one MMA spans the two CTAs of a
// cluster pair (M = 256, 128 rows per CTA), each CTA holding its own A rows
// and half of the B rows at the same shared-memory offset.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive on the mbarrier at this offset in each CTA of cta_mask once the
// pair MMAs issued so far complete.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"(cta_mask) : "memory");
}
// TMA load into this CTA's shared memory that completes an mbarrier which may
// live in the peer CTA of the pair (bar is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar_cluster) : "memory");
}
// shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start before the previous kernel in the stream has
// finished; griddep_wait() blocks until that kernel has completed and its
// memory is visible (immediately when the launch was not programmatic), so it
// precedes every read of the previous kernel's output. griddep_launch_dependents()
// lets the next such kernel start now.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Relaxed 64-bit accesses at GPU scope (naturally aligned: single-copy
// atomic, so a reader sees either the old or the new word whole).
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// 32-bit store into another CTA's shared memory that completes 4 bytes of
// the transaction count of an mbarrier there (both addresses from
// cluster_addr); no fence and no cluster barrier: the receiver waits on its
// mbarrier.
__device__ __forceinline__ void st_async_cluster_f32(uint32_t addr, float v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 ::"r"(addr), "r"(__float_as_uint(v)), "r"(bar) : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// lane (base lane + i), columns [col, col+32). Asynchronous: the registers
// are valid only after tmem_wait_ld(r), which also ties them to the wait so
// the compiler cannot read them earlier.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
// 32 lanes x 16 consecutive columns (same contract as tmem_ld32_async).
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
          "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
        :: "memory");
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
          "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
          "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
          "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
          "+r"(r[31])
        :: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma: K-major operand whose rows
// are SW bytes long (SW = 128, 64 or 32: 64, 32 or 16 bf16) and swizzled the
// way TMA writes them with the matching swizzle mode; rows are packed, so
// 8-row groups are 8*SW bytes apart. Fields: start address >> 4 (bits 0-13),
// leading byte offset >> 4 (16-29, unused for swizzled K-major), stride byte
// offset >> 4 (32-45), descriptor version 1 (46-47), base offset 0 (49-51;
// tile bases are 1024-byte aligned), layout (61-63): 2 = 128B, 4 = 64B,
// 6 = 32B swizzle. A K step inside the row advances the start address.
template <int SW>
__device__ __forceinline__ uint64_t smem_desc_sw(uint32_t saddr) {
    static_assert(SW == 128 || SW == 64 || SW == 32, "swizzle width");
    constexpr uint64_t layout = SW == 128 ? 2 : (SW == 64 ? 4 : 6);
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)((8u * SW) >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= layout << 61;
    return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator (bits 4-5 = 1),
// A and B bf16 (bits 7-9 and 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

// ------------------------------------------------ warp top-k + softmax --

// Lanes below this one in the warp.
__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}


// Top-k and softmax of one token row held by one warp as NK keys per lane
// (make_key of the bf16-rounded logit and the expert id; 0 = no key), as
// "[AMD] One-launch small-M MoE router for Qwen3.5 on gfx950", Modifications,
// defines them: the k largest rounded logits, the lowest id first among equal
// ones, slots ordered by (value desc, id asc); weights = softmax over the
// selected (renorm = 1) or the softmax over every key read at the selected
// (renorm = 0). Returns the key of slot `lane` (lanes < k) and sets its
// weight. cand_s: 32 words of shared memory owned by the warp. key[] is
// consumed.
//
// Selection by threshold instead of k serial maxima: T = the k-th largest of
// the 32 lane maxima is a lower bound of the k-th largest key (the k lanes
// whose maxima reach T hold k distinct keys >= T), so the top-k are among
// the keys >= T. Those (usually k + a few) are compacted into cand_s by
// ballots, each one ranked against the others in one shuffle pass, and
// stored at its rank. When more than 32 keys reach T (the largest logits
// concentrated in a few lanes), k exact rounds of a warp maximum take over.
template <int NK>
__device__ __forceinline__ uint32_t warp_topk_keys(uint32_t (&key)[NK], int k, int renorm, uint32_t *cand_s,
                                                   float &weight) {
    const int lane = threadIdx.x & 31;
    // this lane's largest key (a tree: depth log2(NK))
    uint32_t lm[NK / 2];
#pragma unroll
    for (int i = 0; i < NK / 2; ++i) lm[i] = max(key[i], key[i + NK / 2]);
#pragma unroll
    for (int h = NK / 4; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) lm[i] = max(lm[i], lm[i + h]);
    const uint32_t lmax = lm[0];
    // without renormalisation the weights divide by the softmax denominator
    // over all E experts: every key's exponential relative to the row's
    // largest logit, summed as a tree (per lane, then across the warp)
    float den_all = 0.0f;
    if (!renorm) {
        const float vtop = key_value(__reduce_max_sync(0xffffffffu, lmax));
        float ex[NK];
#pragma unroll
        for (int i = 0; i < NK; ++i) ex[i] = key[i] ? expf(key_value(key[i]) - vtop) : 0.0f;
#pragma unroll
        for (int h = NK / 2; h >= 1; h >>= 1)
#pragma unroll
            for (int i = 0; i < h; ++i) ex[i] += ex[i + h];
        den_all = ex[0];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) den_all += __shfl_xor_sync(0xffffffffu, den_all, o);
    }
    // T: the lane maximum with exactly k - 1 larger ones. Valid keys are
    // unique and nonzero; a lane without a valid key holds 0 and ranks at or
    // past min(E, 32) >= k, so exactly one lane matches.
    int rl = 0;
#pragma unroll
    for (int d = 1; d < 32; ++d) rl += __shfl_xor_sync(0xffffffffu, lmax, d) > lmax;
    const uint32_t T = __shfl_sync(0xffffffffu, lmax, __ffs(__ballot_sync(0xffffffffu, rl == k - 1)) - 1);
    uint32_t bal[NK];
    int tot = 0;
#pragma unroll
    for (int i = 0; i < NK; ++i) {
        bal[i] = __ballot_sync(0xffffffffu, key[i] >= T);
        tot += __popc(bal[i]);
    }
    uint32_t mine, first;
    if (tot <= 32) {  // warp-uniform
        // compact the candidates, in (i, lane) order, into cand_s[0, tot)
        const uint32_t lt = lanemask_lt();
        int base = 0;
#pragma unroll
        for (int i = 0; i < NK; ++i) {
            if (key[i] >= T) cand_s[base + __popc(bal[i] & lt)] = key[i];
            base += __popc(bal[i]);
        }
        __syncwarp();
        const uint32_t c = lane < tot ? cand_s[lane] : 0u;
        int r = 0;  // candidates above this one (0 never counts: valid keys are nonzero)
#pragma unroll
        for (int d = 1; d < 32; ++d) r += __shfl_xor_sync(0xffffffffu, c, d) > c;
        __syncwarp();
        if (lane < tot && r < k) cand_s[r] = c;  // slot r of the row
        __syncwarp();
        mine = cand_s[lane];  // meaningful for lanes < k
        first = cand_s[0];
        __syncwarp();
    } else {
        // k rounds: each lane's largest key, the warp's largest (redux), and
        // the lane holding it clears it (keys are unique)
        mine = 0u;
        first = 0u;
#pragma unroll 1
        for (int r = 0; r < k; ++r) {
            uint32_t m2[NK / 2];
#pragma unroll
            for (int i = 0; i < NK / 2; ++i) m2[i] = max(key[i], key[i + NK / 2]);
#pragma unroll
            for (int h = NK / 4; h >= 1; h >>= 1)
#pragma unroll
                for (int i = 0; i < h; ++i) m2[i] = max(m2[i], m2[i + h]);
            const uint32_t gmax = __reduce_max_sync(0xffffffffu, m2[0]);
            first = (r == 0) ? gmax : first;
            mine = (lane == r) ? gmax : mine;
#pragma unroll
            for (int i = 0; i < NK; ++i) key[i] = (key[i] == gmax) ? 0u : key[i];
        }
    }
    // softmax over the selected logits (renormalised top-k), or the E-expert
    // softmax at the selected ids; every lane evaluates the exponential, lanes
    // past k drop it. The weight is the exponential times the correctly
    // rounded reciprocal of the denominator (two roundings, within 1.5 ulp of
    // the quotient).
    const float vmax = key_value(first);
    const float ex = expf(key_value(mine) - vmax);
    const float ev = (lane < k) ? ex : 0.0f;
    float sum = ev;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv = __frcp_rn(renorm ? sum : den_all);
    weight = ev * inv;
    return mine;
}

// ------------------------------------------------------ align building blocks --
//
// moe_align_block_size over flat slot indices i = t*width + s ("[ROCm][Kernel]
// W4A16 MoE prefill: M-aware moe_align block size", Purpose): count slots per
// expert, pad each count to a multiple of A, exclusive-scan the padded counts
// into segment offsets, scatter slot indices into their expert's segment in
// ascending order, fill the rest of each segment with the sentinel numel and
// record the expert of every A-row block.
//
// Stability without a sort: each warp owns a contiguous range of slots; a
// first pass counts per (warp, expert), an exclusive prefix over warps gives
// each warp its start inside every expert segment, and a second pass ranks
// equal ids inside each 32-slot step with a ballot-built peer mask + popc.

// Convergence: a CTA barrier does not merge a warp whose lanes reached it on
// different paths (loops with per-lane trip counts, single-lane stores), and
// a warp that stays split replays every later instruction once per path and
// pays a handshake at each shuffle or ballot. Every barrier after divergent
// work is therefore preceded by __syncwarp().
struct AlignSmem {
    int *wcnt;     // [nwarps][E_al] per-warp counts, then per-warp starts
    int *cnt;      // [E_al] counts of this CTA's slots (then reused as totals)
    int *off;      // [E_al + 1] padded segment offsets
    int *base;     // [E_al] extra per-expert offset of this CTA's slots
    int *scratch;  // [32] scan scratch
};

__host__ __device__ constexpr int align_smem_words(int nwarps, int num_experts) {
    return nwarps * num_experts + num_experts + (num_experts + 1) + num_experts + 32;
}

__device__ __forceinline__ AlignSmem align_carve(int *smem, int num_experts) {
    const int nw = blockDim.x >> 5;
    AlignSmem s;
    s.wcnt = smem;
    s.cnt = s.wcnt + nw * num_experts;
    s.off = s.cnt + num_experts;
    s.base = s.off + num_experts + 1;
    s.scratch = s.base + num_experts;
    return s;
}


// Lanes of the warp holding the same value as this lane, for values in
// [0, 2048): eleven ballots, one per bit (a fixed cost, unlike a
// data-dependent match loop). Invalid entries use 2047, never a valid id.
__device__ __forceinline__ uint32_t peers_of(int v) {
    uint32_t m = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < 11; ++b) {
        const bool bit = (v >> b) & 1;
        const uint32_t bal = __ballot_sync(0xffffffffu, bit);
        m &= bit ? bal : ~bal;
    }
    return m;
}
constexpr int kNoExpert = 2047;

// Align output write, checked against the caller's array length: a position
// outside it (only possible from a corrupted workspace) is skipped and noted
// in `bad` (a predicated store, no branch); the caller reports bad once.
__device__ __forceinline__ void st_slot(int32_t *arr, int64_t pos, int64_t cap, int32_t v, uint32_t &bad) {
    const uint32_t ok = (uint64_t)pos < (uint64_t)cap ? 1u : 0u;
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q st.global.b32 [%0], %1;\n}"
                 ::"l"(arr + (ok ? pos : 0)), "r"(v), "r"(ok));
    bad |= ok ^ 1u;
}
// Four consecutive slots [pos, pos + 4) in one 16-byte store (arr + pos must
// be 16-byte aligned); all four are skipped and noted in `bad` unless the
// last is below cap.
__device__ __forceinline__ void st_slot4(int32_t *arr, int64_t pos, int64_t cap, int4 v, uint32_t &bad) {
    const uint32_t ok = (uint64_t)pos + 3u < (uint64_t)cap ? 1u : 0u;
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %5, 0;\n @q st.global.v4.b32 [%0], {%1, %2, %3, %4};\n}"
                 ::"l"(arr + (ok ? pos : 0)), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(ok));
    bad |= ok ^ 1u;
}
// Reports the bad-slot flag of a thread (rarely taken; the warp reconverges).
__device__ __forceinline__ void report_bad_slots(uint32_t bad, uint32_t *err) {
    if (bad) set_error(err, kErrBadSlot);
    __syncwarp();
}

// Slots [warp*L, min((warp+1)*L, n)) belong to warp `warp`; L is a multiple of 32.
__device__ __forceinline__ int align_warp_span(int n) {
    const int nw = blockDim.x >> 5;
    return ((n + nw - 1) / nw + 31) & ~31;
}

// Pass 1: per-warp counts -> s.wcnt, then per-expert exclusive prefix over
// warps (in s.wcnt) and the CTA total (in s.cnt). Ids outside [0, E_al) are
// skipped and flagged.
__device__ __forceinline__ void align_count(const int32_t *ids, int n, int E_al,
                                            const AlignSmem &s, uint32_t *err) {
    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < nw * E_al; i += blockDim.x) s.wcnt[i] = 0;
    __syncwarp();
    __syncthreads();
    const int L = align_warp_span(n);
    const int beg = warp * L, end = min(beg + L, n);
    int *wc = s.wcnt + warp * E_al;
    for (int b = beg; b < end; b += 32) {
        const int i = b + lane;
        int e = (i < end) ? ids[i] : kNoExpert;
        if (i < end && (unsigned)e >= (unsigned)E_al) {
            set_error(err, kErrBadId);
            e = kNoExpert;
        }
        const uint32_t peers = peers_of(e);
        if (e != kNoExpert && lane == __ffs(peers) - 1) wc[e] += __popc(peers);
        __syncwarp();
    }
    __syncwarp();
    __syncthreads();
    for (int e = threadIdx.x; e < E_al; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < nw; ++w) {
            const int c = s.wcnt[w * E_al + e];
            s.wcnt[w * E_al + e] = run;
            run += c;
        }
        s.cnt[e] = run;
    }
    __syncwarp();
    __syncthreads();
}

// Exclusive scan over the CTA of one int per thread; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *scratch, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncwarp();
    __syncthreads();
    if (warp == 0) {
        int t = lane < nw ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        scratch[lane] = t;
    }
    __syncwarp();
    __syncthreads();
    const int excl = x - v + (warp > 0 ? scratch[warp - 1] : 0);
    *total = scratch[nw - 1];
    __syncwarp();
    __syncthreads();
    return excl;
}

// c rounded up to a multiple of A (c >= 0; a mask when A is a power of two).
__device__ __forceinline__ int pad_to_blocks(int c, int A) {
    return (A & (A - 1)) == 0 ? (c + A - 1) & -A : (c + A - 1) / A * A;
}

// Padded segment offsets from per-expert totals tot[]: off[e] = sum over
// e' < e of ceil(tot[e']/A)*A; returns npp = off[E_al]. Each thread scans a
// contiguous run of experts so the order of the sum is fixed.
__device__ __forceinline__ int align_offsets(const int *tot, int E_al, int A, const AlignSmem &s) {
    const int per = (E_al + blockDim.x - 1) / blockDim.x;
    const int e0 = threadIdx.x * per, e1 = min(e0 + per, E_al);
    int local = 0;
    for (int e = e0; e < e1; ++e) local += pad_to_blocks(tot[e], A);
    __syncwarp();
    int total;
    int run = block_exclusive_scan(local, s.scratch, &total);
    for (int e = e0; e < e1; ++e) {
        s.off[e] = run;
        run += pad_to_blocks(tot[e], A);
    }
    if (threadIdx.x == 0) s.off[E_al] = total;
    __syncwarp();
    __syncthreads();
    return total;
}

// Pass 2: stable scatter of this CTA's n slots (flat indices flat0 + i) to
// sorted[off[e] + base[e] + warp start + rank]. Consumes s.wcnt.
__device__ __forceinline__ void align_scatter(const int32_t *ids, int n, int E_al, int flat0,
                                              const AlignSmem &s, bool use_base,
                                              int32_t *sorted, int64_t sorted_cap, uint32_t *err) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = align_warp_span(n);
    const int beg = warp * L, end = min(beg + L, n);
    int *wc = s.wcnt + warp * E_al;
    const uint32_t lt = lanemask_lt();
    uint32_t bad = 0;
    for (int b = beg; b < end; b += 32) {
        const int i = b + lane;
        int e = (i < end) ? ids[i] : kNoExpert;
        if ((unsigned)e >= (unsigned)E_al) e = kNoExpert;
        const uint32_t peers = peers_of(e);
        if (e != kNoExpert) {
            const int pos = s.off[e] + (use_base ? s.base[e] : 0) + wc[e] + __popc(peers & lt);
            st_slot(sorted, pos, sorted_cap, flat0 + i, bad);
        }
        __syncwarp();
        if (e != kNoExpert && lane == __ffs(peers) - 1) wc[e] += __popc(peers);
        __syncwarp();
    }
    report_bad_slots(bad, err);
}

// Padding and block owners, one thread per expert (experts first, first +
// stride, ...): a touched expert e owns blocks [off[e]/A, off[e+1]/A) and its
// rows past its last slot, [off[e] + tot[e], off[e+1]), hold the sentinel.
__device__ __forceinline__ void align_fill(int A, int E_al, const int *tot, const AlignSmem &s,
                                           int sentinel, int32_t *sorted, int64_t sorted_cap,
                                           int32_t *expert_ids, int64_t expert_cap, uint32_t *err,
                                           int first, int stride) {
    uint32_t bad = 0;
    for (int e = first; e < E_al; e += stride) {
        const int c = tot[e];
        if (c == 0) continue;
        const int o0 = s.off[e], o1 = s.off[e + 1];
        for (int b = o0 / A; b < o1 / A; ++b) st_slot(expert_ids, b, expert_cap, e, bad);
        for (int q = o0 + c; q < o1; ++q) st_slot(sorted, q, sorted_cap, sentinel, bad);
    }
    __syncwarp();
    report_bad_slots(bad, err);
}

// Copy n int32 ids from global memory to shared memory with 16-byte loads
// where the source is aligned (all loads in flight before any is used).
__device__ __forceinline__ void stage_ids(int *dst, const int32_t *src, int n) {
    const bool vec = ((reinterpret_cast<uintptr_t>(src) & 15) == 0);
    const int n4 = vec ? (n >> 2) : 0;
    const int4 *s4 = reinterpret_cast<const int4 *>(src);
    int4 *d4 = reinterpret_cast<int4 *>(dst);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) d4[i] = __ldcg(s4 + i);
    for (int i = n4 * 4 + threadIdx.x; i < n; i += blockDim.x) dst[i] = __ldcg(src + i);
    __syncwarp();
    __syncthreads();
}

}  // namespace smr
