/*
 * smr.h -- C ABI of the GB300 (sm_103a) MoE routing front-end.
 *
 * The library computes, for M tokens with hidden size H, E routed experts and
 * an optional shared expert (S = 1):
 *
 *   route  : gate GEMM [M,H] x [E+S,H] (bf16 in, fp32 accumulation), the
 *            routed logits rounded to bf16, top-k with the lowest expert id
 *            winning ties, softmax + renormalisation over the k selected,
 *            and the shared slot k = (E, sigmoid(shared logit) * scale).
 *            "[AMD] One-launch small-M MoE router for Qwen3.5 on gfx950",
 *            Motivation and Modifications.
 *   align  : moe_align_block_size -- per-expert counts, padded prefix sum,
 *            sorted_token_ids, one expert id per block and
 *            num_tokens_post_padded = sum over touched experts of
 *            ceil(tokens_e / A) * A, with the M-aware choice of A.
 *            "[ROCm][Kernel] W4A16 MoE prefill: M-aware moe_align block size
 *            (1.6x TTFT)", Purpose and Scope and safety.
 *
 * Conventions (all entry points):
 *  - Every tensor argument is a DEVICE pointer owned by the caller. The
 *    library never allocates, frees, looks up symbols, touches the file
 *    system or synchronises the host on a launch path; kernels are enqueued
 *    on the caller's stream (a cudaStream_t passed as void*; NULL = legacy
 *    default stream). The same pointers and sizes replay correctly inside a
 *    captured CUDA graph ("Netra Kernel ...", Compile exact contracts, not
 *    model names: fixed pointers, no allocation or host sync on replay).
 *  - Calls outside the supported contract are refused before any launch with
 *    SMR_ERR_INVALID_ARG or SMR_ERR_UNSUPPORTED; smr_last_error() then lists
 *    every reason, so the caller can fall back to another implementation
 *    ("[AMD] One-launch small-M MoE router ...", Modifications: guarded call,
 *    everything else takes the existing path).
 *  - Workspace: a caller-owned device buffer of at least the size the
 *    matching *_workspace_size() returns, 256-byte aligned, ZEROED ONCE by
 *    the caller before its first use (cudaMemsetAsync). Every call leaves
 *    the buffer ready for the next one (counters back at zero, a call tag
 *    that only advances), so it can be reused by later calls and graph
 *    replays without clearing. Calls that share a workspace must not run
 *    concurrently.
 *  - Kernels are launched with programmatic stream serialization: a launch
 *    may start while the preceding kernel on the stream is finishing. It
 *    reads hidden states, ids and the workspace, and writes every output,
 *    only after that kernel has completed (griddepcontrol.wait), and it lets
 *    the next kernel launch early (a next kernel that is not launched
 *    programmatically waits for its completion as usual). The layer's
 *    parameters -- gate_w, shared_w and bias -- may be read before the
 *    preceding kernel has finished: they must not be written by the kernel
 *    immediately preceding a call on the same stream.
 *  - Inputs must be finite. NaN or Inf in hidden states, gate weights or
 *    bias give unspecified (but in-bounds) results.
 */
#ifndef SMR_H_
#define SMR_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SMR_API __attribute__((visibility("default")))
#else
#define SMR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum smr_status {
    SMR_OK = 0,
    SMR_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, too-small capacity */
    SMR_ERR_UNSUPPORTED = 2,  /* valid request outside the implemented contract */
    SMR_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small */
    SMR_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    SMR_ERR_DEVICE = 5        /* no usable sm_103 device is current */
} smr_status;

/* Route problem. Row-major tensors; sizes in elements unless stated. */
typedef struct smr_route_args {
    int32_t M;               /* tokens, >= 0 */
    int32_t H;               /* hidden size, multiple of 8, 8..16384 */
    int32_t E;               /* routed experts, 1..1024 */
    int32_t topk;            /* routed top-k, 1..E, topk + has_shared <= 32 */
    int32_t has_shared;      /* S: 1 = shared expert with id E, 0 = none */
    float shared_scale;      /* multiplies sigmoid(shared logit) */
    int32_t renormalize;     /* 1: weights = softmax renormalised over the top-k (sum 1);
                                0: the softmax over all E routed experts read at the top-k
                                ids (unnormalised top-k weights) */
    const void *hidden;      /* bf16 [M, ld_hidden], 16-byte aligned */
    int64_t ld_hidden;       /* row stride of hidden in elements, >= H, multiple of 8 */
    const void *gate_w;      /* bf16 [E, H] contiguous (nn.Linear layout), 16-byte aligned */
    const void *shared_w;    /* bf16 [1, H], 16-byte aligned; NULL iff has_shared == 0 */
    const float *bias;       /* fp32 [E] added to each routed fp32 logit before the
                                bf16 rounding, or NULL */
    int32_t *topk_ids;       /* out: int32 [M, topk + S]; slots 0..topk-1 in order of
                                (rounded logit desc, id asc); slot topk = E if S */
    float *topk_weights;     /* out: fp32 [M, topk + S] */
    uint16_t *logits_out;    /* optional out: bf16 bits [M, E] of the rounded routed
                                logits (bias included); NULL to skip */
    int32_t shared_logit_bf16; /* 1: round the shared logit to bf16 before the sigmoid
                                  (the shared gate as a bf16 dot product, "Netra Kernel
                                  ...", Reusing routing work instead of recomputing it);
                                  0: use the fp32 logit (only the routed logits are
                                  rounded, "[AMD] One-launch small-M MoE router ...",
                                  Modifications) */
    /* Optional: the hidden states quantised once, in the route's launch, for
     * the expert GEMMs ("Netra Kernel ...", Fusing the activation/quantization
     * boundary: E4M3 with one scale per 128 contiguous values). For every row
     * t and 128-element block b: scale = amax / 448 (amax the block's largest
     * magnitude), codes = E4M3(x * (448 / amax)) rounded to nearest even and
     * saturated at +-448, the divisions and the product in fp32; a block of
     * zeros gets scale 0 and zero codes. Needs H % 128 == 0. NULL to skip. */
    uint8_t *hidden_fp8;     /* out: e4m3 codes [M, H], 16-byte aligned */
    float *hidden_scales;    /* out: fp32 [M, H / 128] */
} smr_route_args;

/* Align problem over a [num_tokens, width] id matrix. */
typedef struct smr_align_args {
    const int32_t *topk_ids;      /* int32 [num_tokens, width], ids in [0, num_experts) */
    int32_t num_tokens;           /* >= 0 */
    int32_t width;                /* slots per token (topk + S), >= 1 */
    int32_t num_experts;          /* E_al = E + S, 1..1024 */
    int32_t routed_topk;          /* k and E used by the M-aware tier (block_size == 0) */
    int32_t routed_experts;
    int32_t block_size;           /* A >= 1, or 0 = smr_select_block_size(num_tokens,
                                     routed_topk, routed_experts) */
    int32_t *sorted_token_ids;    /* out: int32 [sorted_cap]; [0, npp) defined: flat slot
                                     index t*width+s grouped by expert, ascending inside
                                     each expert, padding rows = num_tokens*width */
    int64_t sorted_cap;           /* >= smr_align_capacity(num_tokens*width, num_experts, A) */
    int32_t *expert_ids;          /* out: int32 [expert_cap]; [0, npp/A) defined */
    int64_t expert_cap;           /* >= ceil(smr_align_capacity(...) / A) */
    int32_t *num_tokens_post_padded;  /* out: device int32 [1] = npp */
    /* Optional expert-parallel load-balancing (EPLB) logical->physical remap
     * applied inside the align (the pages' guards refuse such a remap without
     * defining it; this is the library's reading): logical expert e (an id in
     * topk_ids) is held by eplb_count[e] in [1, eplb_max_replicas] physical
     * replicas listed in eplb_map[e * eplb_max_replicas + r]; the slot of
     * token t goes to replica r = t mod eplb_count[e]. Counts, padding, the
     * capacity (numel + num_physical * (A - 1)) and expert_ids are then over
     * the num_physical physical experts; sorted_token_ids still holds flat
     * slot indices. An id, count or physical id out of range is skipped and
     * sets bit 0 of the sticky device error word. eplb_map == NULL: no remap
     * (the other three fields are ignored). Device pointers, read only. */
    const int32_t *eplb_map;      /* int32 [num_experts, eplb_max_replicas] or NULL */
    const int32_t *eplb_count;    /* int32 [num_experts] */
    int32_t eplb_max_replicas;    /* 1..64 */
    int32_t num_physical;         /* 1..1025 */
} smr_align_args;

/* The consumer of the align: the expert GEMM. */
typedef struct smr_expert_gemm_args {
    const void *hidden;            /* bf16 [num_tokens, ld_hidden], 16-byte aligned */
    int64_t ld_hidden;             /* row stride in elements, >= H, multiple of 8 */
    int32_t num_tokens;            /* T >= 0 */
    int32_t width;                 /* slots per token (the align's width), >= 1 */
    int32_t H;                     /* hidden size, multiple of 64, <= 16384 */
    const void *expert_w;          /* bf16 [num_experts, N, H] (each expert's [N, H] rows), 16-byte aligned */
    int32_t num_experts;           /* the align's num_experts (or num_physical), 1..1025 */
    int32_t N;                     /* output columns per expert, multiple of 128, <= 16384 */
    int32_t block_size;            /* A used by the align: 64 or 128 */
    const int32_t *sorted_token_ids;  /* the align's outputs (device) */
    int64_t sorted_cap;            /* its length: the grid covers ceil(sorted_cap / A) blocks */
    const int32_t *expert_ids;
    const int32_t *num_tokens_post_padded;
    float *out;                    /* out: fp32 [num_tokens * width, N], row = flat slot index
                                      t * width + s; 16-byte aligned */
} smr_expert_gemm_args;

/* M-aware alignment tier (host, no device work): 64 if
 * num_tokens * topk < 128 * num_experts (fewer than one full 128-row block of
 * routed rows per expert), else 128. Returns -1 on non-positive topk or
 * num_experts or negative num_tokens. */
SMR_API int32_t smr_select_block_size(int32_t num_tokens, int32_t topk, int32_t num_experts);

/* Worst-case num_tokens_post_padded: numel + num_experts * (A - 1) (the
 * workspace num_slots formula of the alignment page, Scope and safety).
 * Returns -1 on invalid arguments. */
SMR_API int64_t smr_align_capacity(int64_t numel, int32_t num_experts, int32_t block_size);

/* Workspace bytes for one call with these arguments (0 if none is needed);
 * pointers inside args are not read. */
SMR_API size_t smr_route_workspace_size(const smr_route_args *args);
SMR_API size_t smr_align_workspace_size(const smr_align_args *args);
SMR_API size_t smr_route_align_workspace_size(const smr_route_args *route, const smr_align_args *align);

/* Route only: the gate GEMM, bf16 rounding, top-k with the lowest id winning
 * ties, softmax (renormalised over the selected, or not) and the shared slot
 * ("[AMD] One-launch small-M MoE router for Qwen3.5 on gfx950",
 * Modifications). One kernel launch for M <= 16: the gate rows are split
 * across CTAs, and one CTA selects after collecting the row groups'
 * tagged selection keys from the workspace. For M > 16 with E % 32 == 0 and
 * 32 <= E <= 512, one tcgen05 GEMM launch with the top-k fused into its
 * epilogue; any other E (up to 1024) takes ceil(E / 512) tcgen05 launches
 * that write the rounded logits into the workspace, then one select launch
 * (one warp per row). M == 0 launches nothing. Refusals (SMR_ERR_*) are
 * returned before any launch; a failed launch returns SMR_ERR_CUDA. */
SMR_API smr_status smr_route(const smr_route_args *args, void *workspace, size_t workspace_bytes,
                     void *stream);

/* Align only: moe_align_block_size ("[ROCm][Kernel] W4A16 MoE prefill:
 * M-aware moe_align block size (1.6x TTFT)", Purpose). Reads topk_ids,
 * writes sorted_token_ids, expert_ids and num_tokens_post_padded. One launch
 * for num_tokens * width <= 2048, else three (tile counts, tile starts,
 * scatter). An id outside [0, num_experts) is skipped and sets the sticky
 * device error word (see smr_get_device_error). */
SMR_API smr_status smr_align(const smr_align_args *args, void *workspace, size_t workspace_bytes,
                     void *stream);

/* Route then align on the route's output (the two passages above, in the
 * order the pages' serving paths run them). align->topk_ids must equal
 * route->topk_ids, align->num_tokens == route->M, align->width == topk + S,
 * align->num_experts == E + S; routed_topk/routed_experts are taken from the
 * route. For M <= 16 both run in ONE launch; for larger M the tcgen05 route
 * aligns in its last CTA when M * width <= 704 (one launch), else it also
 * writes each 64-row tile's expert counts and two align launches follow.
 * With an EPLB remap the align always runs as its own launches behind the
 * route (1 or 3). */
SMR_API smr_status smr_route_align(const smr_route_args *route, const smr_align_args *align,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Route then align for 1 <= M <= 16 in one launch, like smr_route_align, but
 * with NO workspace argument and no allocation: for callers that cannot
 * allocate device memory on their launch path (no device allocator is
 * available to them, or allocation is forbidden once their memory pool is
 * sized). The scratch is a fixed array of 256 KiB inside the library, kept
 * by every GPU that loads the library until the process exits. (The pages
 * have no counterpart; this is an interface convenience.)
 *  - The first call on a device, with that device current, resolves the
 *    array's device address and clears the array (then synchronises the
 *    device); make that first call outside any stream capture. Later calls
 *    do no set-up.
 *  - Every call on a device shares the one array, which keeps the last
 *    call's contents: calls that overlap on the GPU (different streams
 *    without ordering, or host threads) race and give wrong results.
 *  - Problems whose scratch would exceed the array (see
 *    smr_route_align_workspace_size) and M outside [1, 16] are refused with
 *    SMR_ERR_UNSUPPORTED. Outputs are as for smr_route_align. */
SMR_API smr_status smr_route_align_static(const smr_route_args *route, const smr_align_args *align,
                                          void *stream);

/* The expert GEMM that consumes the align ("[ROCm][Kernel] W4A16 MoE
 * prefill: M-aware moe_align block size (1.6x TTFT)", Purpose), with bf16
 * expert weights: for every block b of A rows of sorted_token_ids with
 * b * A < num_tokens_post_padded, the rows' hidden states (slot / width =
 * token) against expert expert_ids[b]'s [N, H] weights; every routed slot i
 * gets out[i] = hidden[i / width] . W[e]^T (fp32 accumulation and output).
 * Padding rows are computed as zeros and not stored; blocks at or past npp
 * return at once (the early exit whose work the M-aware tier shrinks).
 * One launch of ceil(sorted_cap / A) x N / 256 (or 128) CTAs. The workspace
 * (>= 256 bytes, zeroed once) only carries the sticky error word: bit 0 for
 * an expert id out of range, bit 2 for a sorted entry that is neither a slot
 * nor the sentinel (both from a corrupted align output), bit 1 for a wait
 * that gave up (the block's outputs are then not written). */
SMR_API smr_status smr_expert_gemm(const smr_expert_gemm_args *args, void *workspace, size_t workspace_bytes,
                                   void *stream);

/* Sticky device error word of a workspace: synchronises `stream`, then copies
 * the word to *code_out (0 = no error; bit 0 = an id out of range in align,
 * bit 1 = a bounded wait inside a kernel gave up, bit 2 = an align output
 * position fell outside sorted_cap / expert_cap -- possible only from a
 * corrupted workspace -- and that write was skipped). Not for launch paths. */
SMR_API smr_status smr_get_device_error(const void *workspace, void *stream, int32_t *code_out);

/* Clears the sticky device error word (stream-ordered memset). */
SMR_API smr_status smr_clear_device_error(void *workspace, void *stream);

/* The sticky device error word of smr_route_align_static's fixed scratch
 * array on the current device (same bits and synchronisation as
 * smr_get_device_error), and its clear. The first use on a device sets the
 * array up like the first smr_route_align_static call does. Not for launch
 * paths. */
SMR_API smr_status smr_get_static_device_error(void *stream, int32_t *code_out);
SMR_API smr_status smr_clear_static_device_error(void *stream);

/* TEST HOOK -- failure injection without a GPU fault (vLLM #60833
 * "--monokernel decode", Details: bounded waits that set a sticky failed word
 * instead of hanging). Process-wide; affects launches made after the call.
 *   SMR_STALL_SMALL_TAIL: the small-M tail waits for a call tag that no row
 *     group writes, giving up after `limit` reloads of its key words;
 *   SMR_STALL_TC_MERGE: the tcgen05 route's merge of its two column halves
 *     waits on a barrier nothing arrives on, giving up after `limit` SM
 *     cycles (no copy is in flight there).
 * The wait runs out, bit 1 of the workspace's sticky error word is set, the
 * kernel returns (the tcgen05 route skips its outputs; the small-M tail goes
 * on with the keys it holds) and later calls are unaffected.
 * SMR_STALL_NONE (limit ignored) switches the hook off. Returns
 * SMR_ERR_INVALID_ARG for another site or a limit < 1. */
#define SMR_STALL_NONE 0
#define SMR_STALL_SMALL_TAIL 1
#define SMR_STALL_TC_MERGE 2
SMR_API smr_status smr_test_force_wait_timeout(int32_t site, int64_t limit);

/* Static string for a status; thread-local text of the last refusal (every
 * reason, "; "-separated) or CUDA error on this thread, "" if none. */
SMR_API const char *smr_status_string(smr_status status);
SMR_API const char *smr_last_error(void);

/* Library version, 0xMMmmpp. */
SMR_API int32_t smr_version(void);

/* Number of kernels the most recent successful smr_route / smr_align /
 * smr_route_align call on this thread enqueued (0 after a refusal). */
SMR_API int32_t smr_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SMR_H_ */
