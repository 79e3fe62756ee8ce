// smr_api.cpp -- the C ABI (include/smr.h): argument validation with every
// refusal reason, workspace layout, dispatch to the kernels, error reporting.
//
// Dispatch ("[AMD] One-launch small-M MoE router for Qwen3.5 on gfx950",
// Modifications, for the guarded single launch; "[ROCm][Kernel] W4A16 MoE
// prefill: M-aware moe_align block size", Purpose, for the alignment tier):
//   route_align, M <= 16 : 1 launch  (small route + fused align)
//   route_align, M > 16  : 1 tcgen05 route launch whose last CTA aligns all ids when
//                          there are at most kFusedAlignMax (704), else the route (which
//                          then counts the experts of its rows) + 2 align launches;
//                          with E > 512 or E % 32 != 0: ceil(E / 512) logits-only
//                          tcgen05 launches + 1 select launch + 1 or 3 align launches
//   route        : 1 launch;  align : 1 launch (numel <= kAlignSingleMax, 2048) or 3.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <string>
#include <vector>

#include "smr.h"
#include "smr_launch.h"

namespace {

constexpr size_t kHeaderBytes = 256;
constexpr size_t kWsAlign = 256;
constexpr int kMaxH = 16384;
constexpr int kMaxExperts = 1024;

thread_local std::string g_last_error;
thread_local int g_last_launches = 0;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Reasons {
    std::vector<std::string> invalid, unsupported;
    void bad(const std::string &s) { invalid.push_back(s); }
    void unsup(const std::string &s) { unsupported.push_back(s); }
    bool ok() const { return invalid.empty() && unsupported.empty(); }
    smr_status finish(const char *what) {
        std::string msg;
        for (auto &r : invalid) msg += (msg.empty() ? "" : "; ") + r;
        for (auto &r : unsupported) msg += (msg.empty() ? "" : "; ") + r;
        g_last_error = std::string(what) + ": " + msg;
        g_last_launches = 0;
        return invalid.empty() ? SMR_ERR_UNSUPPORTED : SMR_ERR_INVALID_ARG;
    }
};

smr_status cuda_fail(const char *what, cudaError_t e) {
    g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    g_last_launches = 0;
    return SMR_ERR_CUDA;
}

// The kernels are built for sm_103a only.
smr_status check_device() {
    static std::atomic<int> cached[smr::kMaxDevices];  // 0 unknown, 1 ok, 2 bad
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        g_last_error = std::string("no current CUDA device: ") + cudaGetErrorString(e);
        return SMR_ERR_DEVICE;
    }
    if (dev < smr::kMaxDevices && cached[dev].load(std::memory_order_relaxed) == 1) return SMR_OK;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    const bool ok = (major == 10 && minor == 3);
    if (dev < smr::kMaxDevices) cached[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
    if (!ok) {
        g_last_error = "device " + std::to_string(dev) + " is sm_" + std::to_string(major) +
                       std::to_string(minor) + "; this library is built for sm_103a (GB300)";
        return SMR_ERR_DEVICE;
    }
    return SMR_OK;
}

// Failure-injection hook (smr_test_force_wait_timeout), process-wide.
std::atomic<int> g_stall_site{smr::kStallNone};
std::atomic<long long> g_stall_limit{0};

// --- route ------------------------------------------------------------------

void check_route(const smr_route_args *a, Reasons &r) {
    if (a->M < 0) r.bad("M must be >= 0 (got " + std::to_string(a->M) + ")");
    if (a->H < 8 || a->H > kMaxH || a->H % 8 != 0)
        r.bad("H must be a multiple of 8 in [8, 16384] (got " + std::to_string(a->H) + ")");
    if (a->E < 1 || a->E > kMaxExperts)
        r.bad("E must be in [1, 1024] (got " + std::to_string(a->E) + ")");
    if (a->has_shared != 0 && a->has_shared != 1)
        r.bad("has_shared must be 0 or 1 (got " + std::to_string(a->has_shared) + ")");
    const int S = a->has_shared ? 1 : 0;
    if (a->topk < 1 || a->topk > a->E)
        r.bad("topk must be in [1, E] (got " + std::to_string(a->topk) + ")");
    else if (a->topk + S > 32)
        r.unsup("topk + has_shared must be <= 32 (got " + std::to_string(a->topk + S) + ")");
    if (a->renormalize != 0 && a->renormalize != 1)
        r.bad("renormalize must be 0 or 1 (got " + std::to_string(a->renormalize) + ")");
    if (a->shared_logit_bf16 != 0 && a->shared_logit_bf16 != 1)
        r.bad("shared_logit_bf16 must be 0 or 1 (got " + std::to_string(a->shared_logit_bf16) + ")");
    if (!std::isfinite(a->shared_scale)) r.bad("shared_scale must be finite");
    if (a->M > 0) {
        if (!a->hidden) r.bad("hidden is NULL");
        else if (!aligned(a->hidden, 16)) r.bad("hidden must be 16-byte aligned");
        if (a->ld_hidden < a->H || a->ld_hidden % 8 != 0)
            r.bad("ld_hidden must be >= H and a multiple of 8 (got " + std::to_string(a->ld_hidden) + ")");
        if (!a->gate_w) r.bad("gate_w is NULL");
        else if (!aligned(a->gate_w, 16)) r.bad("gate_w must be 16-byte aligned");
        if (S && !a->shared_w) r.bad("shared_w is NULL but has_shared == 1");
        if (S && a->shared_w && !aligned(a->shared_w, 16)) r.bad("shared_w must be 16-byte aligned");
        if (!S && a->shared_w) r.bad("shared_w must be NULL when has_shared == 0");
        if (a->bias && !aligned(a->bias, 4)) r.bad("bias must be 4-byte aligned");
        if (!a->topk_ids) r.bad("topk_ids is NULL");
        else if (!aligned(a->topk_ids, 4)) r.bad("topk_ids must be 4-byte aligned");
        if (!a->topk_weights) r.bad("topk_weights is NULL");
        else if (!aligned(a->topk_weights, 4)) r.bad("topk_weights must be 4-byte aligned");
        if (a->logits_out && !aligned(a->logits_out, 16)) r.bad("logits_out must be 16-byte aligned");
        if (a->hidden_fp8) {
            if (a->H % 128 != 0) r.bad("hidden_fp8 needs H % 128 == 0 (one scale per 128 values)");
            if (!aligned(a->hidden_fp8, 16)) r.bad("hidden_fp8 must be 16-byte aligned");
            if (!a->hidden_scales) r.bad("hidden_scales is NULL but hidden_fp8 is set");
            else if (!aligned(a->hidden_scales, 4)) r.bad("hidden_scales must be 4-byte aligned");
        }
    }
}

// M > 16 with a gate outside the fused tcgen05 epilogue (E > 512 or E not a
// multiple of 32): logits-only tcgen05 launches, then the select kernel.
bool generic_route(const smr_route_args *a) {
    return a->M > smr::kSmallMaxM && !smr::tc_route_supported(a->H, a->E, a->topk, a->has_shared ? 1 : 0);
}

size_t generic_logits_bytes(const smr_route_args *a) {
    return round_up((size_t)a->M * (size_t)smr::generic_logits_ld(a->E) * 2, kWsAlign);
}

size_t route_scratch_bytes(const smr_route_args *a) {
    if (a->M <= 0) return 0;
    if (a->M <= smr::kSmallMaxM) return round_up((size_t)a->M * (size_t)a->E * 8, kWsAlign);  // tagged keys
    if (generic_route(a))  // bf16 logit rows + shared logits
        return generic_logits_bytes(a) + round_up((size_t)a->M * 4, kWsAlign);
    return 0;
}

// --- align ------------------------------------------------------------------

int effective_block_size(const smr_align_args *a) {
    if (a->block_size > 0) return a->block_size;
    return smr_select_block_size(a->num_tokens, a->routed_topk, a->routed_experts);
}

// The experts the align counts and pads: the physical ones behind an EPLB
// remap, else the ids' own range.
bool has_eplb(const smr_align_args *a) { return a->eplb_map != nullptr; }
int align_experts(const smr_align_args *a) { return has_eplb(a) ? a->num_physical : a->num_experts; }
constexpr int kMaxReplicas = 64;

void check_align(const smr_align_args *a, Reasons &r, bool ids_from_route) {
    if (a->num_tokens < 0) r.bad("num_tokens must be >= 0");
    if (a->width < 1) r.bad("width must be >= 1");
    if (a->num_experts < 1 || a->num_experts > kMaxExperts + 1)
        r.bad("num_experts must be in [1, 1025] (got " + std::to_string(a->num_experts) + ")");
    if (a->block_size < 0 || a->block_size > 4096)
        r.bad("block_size must be 0 (M-aware tier) or in [1, 4096] (got " +
              std::to_string(a->block_size) + ")");
    if (a->block_size == 0 && !ids_from_route && (a->routed_topk < 1 || a->routed_experts < 1))
        r.bad("block_size == 0 needs routed_topk >= 1 and routed_experts >= 1");
    if (has_eplb(a)) {
        if (!a->eplb_count) r.bad("eplb_count is NULL but eplb_map is set");
        if (!aligned(a->eplb_map, 4) || (a->eplb_count && !aligned(a->eplb_count, 4)))
            r.bad("eplb_map and eplb_count must be 4-byte aligned");
        if (a->eplb_max_replicas < 1 || a->eplb_max_replicas > kMaxReplicas)
            r.bad("eplb_max_replicas must be in [1, 64] (got " + std::to_string(a->eplb_max_replicas) + ")");
        if (a->num_physical < 1 || a->num_physical > kMaxExperts + 1)
            r.bad("num_physical must be in [1, 1025] (got " + std::to_string(a->num_physical) + ")");
    }
    if (!r.invalid.empty()) return;
    const int64_t numel = (int64_t)a->num_tokens * a->width;
    if (numel > (int64_t)1 << 30) r.unsup("num_tokens * width must be <= 2^30");
    const int A = effective_block_size(a);
    if (A < 1) {
        r.bad("cannot derive a block size");
        return;
    }
    const int64_t cap = smr_align_capacity(numel, align_experts(a), A);
    if (!ids_from_route) {
        if (numel > 0 && !a->topk_ids) r.bad("topk_ids is NULL");
        else if (a->topk_ids && !aligned(a->topk_ids, 4)) r.bad("topk_ids must be 4-byte aligned");
    }
    if (!a->sorted_token_ids) r.bad("sorted_token_ids is NULL");
    if (!a->expert_ids) r.bad("expert_ids is NULL");
    if (!a->num_tokens_post_padded) r.bad("num_tokens_post_padded is NULL");
    if (a->sorted_cap < cap)
        r.bad("sorted_cap " + std::to_string(a->sorted_cap) + " < required " + std::to_string(cap));
    if (a->expert_cap < (cap + A - 1) / A)
        r.bad("expert_cap " + std::to_string(a->expert_cap) + " < required " +
              std::to_string((cap + A - 1) / A));
    if (cap > INT32_MAX) r.unsup("capacity exceeds int32 indexing");
}

size_t align_scratch_bytes(const smr_align_args *a) {
    const int64_t numel = (int64_t)a->num_tokens * a->width;
    if (numel <= smr::kAlignSingleMax) return 0;
    return round_up((size_t)smr::align_scratch_words(numel, align_experts(a)) * 4, kWsAlign);
}

smr_status check_ws(void *ws, size_t bytes, size_t need, const char *what) {
    if (!ws) {
        g_last_error = std::string(what) + ": workspace is NULL";
        return SMR_ERR_WORKSPACE;
    }
    if (!aligned(ws, kWsAlign)) {
        g_last_error = std::string(what) + ": workspace must be 256-byte aligned";
        return SMR_ERR_WORKSPACE;
    }
    if (bytes < need) {
        g_last_error = std::string(what) + ": workspace has " + std::to_string(bytes) +
                       " bytes, needs " + std::to_string(need);
        return SMR_ERR_WORKSPACE;
    }
    return SMR_OK;
}

// The align behind a tcgen05 route over more than kFusedAlignMax slots takes
// its per-tile expert counts from the route (tiles of 64 token rows), unless
// an EPLB remap changes what is counted.
bool align_counted_by_route(const smr_route_args *r, const smr_align_args *a, int64_t numel) {
    return r->M > smr::kSmallMaxM && numel > smr::kFusedAlignMax && !has_eplb(a) && !generic_route(r);
}
int64_t route_tiles(const smr_route_args *r) {
    return (r->M + smr::kTcCountRows - 1) / smr::kTcCountRows;
}

// counted_tile > 0: tiles of that many slots whose counts the route writes.
smr::AlignLaunch make_align_launch(const smr_align_args *a, const int32_t *ids, void *ws,
                                   size_t align_off, int counted_tile = 0) {
    smr::AlignLaunch L{};
    L.ids = ids;
    L.numel = a->num_tokens * a->width;
    L.E_al = align_experts(a);
    L.A = effective_block_size(a);
    L.map = a->eplb_map;
    L.map_count = a->eplb_count;
    L.map_R = has_eplb(a) ? a->eplb_max_replicas : 1;
    L.E_log = a->num_experts;
    L.width = a->width;
    L.sorted = a->sorted_token_ids;
    L.expert_ids = a->expert_ids;
    L.npp = a->num_tokens_post_padded;
    L.sorted_cap = a->sorted_cap;
    L.expert_cap = a->expert_cap;
    L.hdr = ws;
    L.tile_counts = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + align_off);
    L.counted_tile = counted_tile;
    const int64_t tiles = counted_tile > 0 ? ((int64_t)L.numel + counted_tile - 1) / counted_tile
                                           : smr::align_num_tiles(L.numel);
    const int64_t tw = tiles * L.E_al;
    L.tile_base = L.tile_counts + tw;
    L.totals = L.tile_base + tw;
    return L;
}

smr_status run_route(const smr_route_args *a, void *ws, cudaStream_t stream,
                     const smr_align_args *fused_align, int *launches,
                     int32_t *tile_counts = nullptr) {
    const int S = a->has_shared ? 1 : 0;
    if (a->M <= smr::kSmallMaxM) {
        smr::SmallRouteLaunch L{};
        L.x = static_cast<const uint16_t *>(a->hidden);
        L.ld = a->ld_hidden;
        L.w = static_cast<const uint16_t *>(a->gate_w);
        L.ws = static_cast<const uint16_t *>(a->shared_w);
        L.bias = a->bias;
        L.M = a->M; L.H = a->H; L.E = a->E; L.S = S; L.k = a->topk;
        L.scale = a->shared_scale;
        L.renorm = a->renormalize;
        L.shared_bf16 = a->shared_logit_bf16;
        L.ids = a->topk_ids;
        L.wts = a->topk_weights;
        L.logits_out = a->logits_out;
        L.scratch = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(ws) + kHeaderBytes);
        L.hdr = ws;
        if (fused_align) {
            L.A = effective_block_size(fused_align);
            L.sorted = fused_align->sorted_token_ids;
            L.expert_ids = fused_align->expert_ids;
            L.npp = fused_align->num_tokens_post_padded;
            L.sorted_cap = fused_align->sorted_cap;
            L.expert_cap = fused_align->expert_cap;
        }
        L.xq = a->hidden_fp8;
        L.xs = a->hidden_scales;
        const smr::StallHook hook = smr::stall_hook();
        L.stall = hook.site == smr::kStallSmallTail;
        L.stall_limit = L.stall ? hook.limit : 0;
        cudaError_t e = smr::launch_small_route(L, stream);
        if (e != cudaSuccess) return cuda_fail("small-M route launch", e);
        *launches += 1;
        return SMR_OK;
    }
    if (generic_route(a)) {
        // the logits of every 512-column range of the gate, then the top-k
        // over whole rows
        const int64_t ld = smr::generic_logits_ld(a->E);
        uint16_t *lg = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + kHeaderBytes);
        float *sv = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kHeaderBytes + generic_logits_bytes(a));
        for (int c0 = 0; c0 < a->E; c0 += smr::kTcRangeCols) {
            smr::TcRouteLaunch L{};
            L.x = static_cast<const uint16_t *>(a->hidden);
            L.ld = a->ld_hidden;
            L.w = static_cast<const uint16_t *>(a->gate_w) + (int64_t)c0 * a->H;
            L.ws = (c0 == 0 && S) ? static_cast<const uint16_t *>(a->shared_w) : nullptr;
            L.bias = a->bias ? a->bias + c0 : nullptr;
            L.M = a->M; L.H = a->H; L.E = std::min(smr::kTcRangeCols, a->E - c0);
            L.S = (c0 == 0) ? S : 0; L.k = 1;
            L.hdr = ws;
            L.logits_only = true;
            L.col0 = c0;
            L.logits_ws = lg;
            L.ld_logits = ld;
            L.s_out = sv;
            L.xq = (c0 == 0) ? a->hidden_fp8 : nullptr;  // the first launch quantises x
            L.xs = a->hidden_scales;
            cudaError_t e = smr::launch_tc_route(L, stream);
            if (e != cudaSuccess) return cuda_fail("tcgen05 logits launch", e);
            *launches += 1;
        }
        smr::SelectLaunch L{};
        L.logits = lg;
        L.ld = ld;
        L.s = sv;
        L.M = a->M; L.E = a->E; L.S = S; L.k = a->topk;
        L.renorm = a->renormalize;
        L.shared_bf16 = a->shared_logit_bf16;
        L.scale = a->shared_scale;
        L.ids = a->topk_ids;
        L.wts = a->topk_weights;
        L.logits_out = a->logits_out;
        cudaError_t e = smr::launch_select(L, stream);
        if (e != cudaSuccess) return cuda_fail("select launch", e);
        *launches += 1;
        return SMR_OK;
    }
    smr::TcRouteLaunch L{};
    L.x = static_cast<const uint16_t *>(a->hidden);
    L.ld = a->ld_hidden;
    L.w = static_cast<const uint16_t *>(a->gate_w);
    L.ws = static_cast<const uint16_t *>(a->shared_w);
    L.bias = a->bias;
    L.M = a->M; L.H = a->H; L.E = a->E; L.S = S; L.k = a->topk;
    L.scale = a->shared_scale;
    L.renorm = a->renormalize;
    L.shared_bf16 = a->shared_logit_bf16;
    L.ids = a->topk_ids;
    L.wts = a->topk_weights;
    L.logits_out = a->logits_out;
    L.hdr = ws;
    L.tile_counts = tile_counts;
    L.xq = a->hidden_fp8;
    L.xs = a->hidden_scales;
    if (fused_align) {  // at most kFusedAlignMax ids: the route's last CTA aligns them
        L.fa_A = effective_block_size(fused_align);
        L.fa_sorted = fused_align->sorted_token_ids;
        L.fa_eids = fused_align->expert_ids;
        L.fa_npp = fused_align->num_tokens_post_padded;
        L.fa_sorted_cap = fused_align->sorted_cap;
        L.fa_eids_cap = fused_align->expert_cap;
    }
    const smr::StallHook hook = smr::stall_hook();
    L.stall = hook.site == smr::kStallTcMerge;
    L.stall_limit = L.stall ? hook.limit : 0;
    cudaError_t e = smr::launch_tc_route(L, stream);
    if (e != cudaSuccess) return cuda_fail("tcgen05 route launch", e);
    *launches += 1;
    return SMR_OK;
}

}  // namespace

namespace smr {
StallHook stall_hook() {
    return StallHook{g_stall_site.load(std::memory_order_relaxed), g_stall_limit.load(std::memory_order_relaxed)};
}
}  // namespace smr

extern "C" {

SMR_API int32_t smr_select_block_size(int32_t num_tokens, int32_t topk, int32_t num_experts) {
    if (num_tokens < 0 || topk < 1 || num_experts < 1) return -1;
    return ((int64_t)num_tokens * topk < (int64_t)128 * num_experts) ? 64 : 128;
}

SMR_API int64_t smr_align_capacity(int64_t numel, int32_t num_experts, int32_t block_size) {
    if (numel < 0 || num_experts < 1 || block_size < 1) return -1;
    return numel + (int64_t)num_experts * (block_size - 1);
}

SMR_API size_t smr_route_workspace_size(const smr_route_args *args) {
    if (!args) return 0;
    return kHeaderBytes + route_scratch_bytes(args);
}

SMR_API size_t smr_align_workspace_size(const smr_align_args *args) {
    if (!args) return 0;
    return kHeaderBytes + align_scratch_bytes(args);
}

SMR_API size_t smr_route_align_workspace_size(const smr_route_args *route, const smr_align_args *align) {
    if (!route || !align) return 0;
    smr_align_args al = *align;
    al.num_tokens = route->M;
    al.width = route->topk + (route->has_shared ? 1 : 0);
    al.num_experts = route->E + (route->has_shared ? 1 : 0);
    const int64_t numel = (int64_t)al.num_tokens * al.width;
    if (align_counted_by_route(route, &al, numel))  // tiles of 64 route rows
        return kHeaderBytes + route_scratch_bytes(route) +
               round_up((size_t)smr::align_scratch_words_tiles(route_tiles(route), al.num_experts) * 4,
                        kWsAlign);
    return kHeaderBytes + route_scratch_bytes(route) + align_scratch_bytes(&al);
}

SMR_API smr_status smr_route(const smr_route_args *args, void *workspace, size_t workspace_bytes,
                             void *stream) {
    g_last_launches = 0;
    if (!args) {
        g_last_error = "smr_route: args is NULL";
        return SMR_ERR_INVALID_ARG;
    }
    Reasons r;
    check_route(args, r);
    if (!r.ok()) return r.finish("smr_route");
    if (args->M == 0) return SMR_OK;
    smr_status st = check_ws(workspace, workspace_bytes, smr_route_workspace_size(args), "smr_route");
    if (st != SMR_OK) return st;
    if ((st = check_device()) != SMR_OK) return st;
    int launches = 0;
    st = run_route(args, workspace, static_cast<cudaStream_t>(stream), nullptr, &launches);
    if (st == SMR_OK) g_last_launches = launches;
    return st;
}

SMR_API smr_status smr_align(const smr_align_args *args, void *workspace, size_t workspace_bytes,
                             void *stream) {
    g_last_launches = 0;
    if (!args) {
        g_last_error = "smr_align: args is NULL";
        return SMR_ERR_INVALID_ARG;
    }
    Reasons r;
    check_align(args, r, false);
    if (!r.ok()) return r.finish("smr_align");
    smr_status st = check_ws(workspace, workspace_bytes, smr_align_workspace_size(args), "smr_align");
    if (st != SMR_OK) return st;
    if ((st = check_device()) != SMR_OK) return st;
    smr::AlignLaunch L = make_align_launch(args, args->topk_ids, workspace, kHeaderBytes);
    cudaError_t e = smr::launch_align(L, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("align launch", e);
    g_last_launches = smr::align_launches(L.numel, false);
    return SMR_OK;
}

SMR_API smr_status smr_route_align(const smr_route_args *route, const smr_align_args *align,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    g_last_launches = 0;
    if (!route || !align) {
        g_last_error = "smr_route_align: route or align args is NULL";
        return SMR_ERR_INVALID_ARG;
    }
    Reasons r;
    check_route(route, r);
    const int S = route->has_shared ? 1 : 0;
    smr_align_args al = *align;
    al.routed_topk = route->topk;
    al.routed_experts = route->E;
    if (align->topk_ids != route->topk_ids) r.bad("align.topk_ids must equal route.topk_ids");
    if (align->num_tokens != route->M) r.bad("align.num_tokens must equal route.M");
    if (align->width != route->topk + S) r.bad("align.width must equal route.topk + has_shared");
    if (align->num_experts != route->E + S) r.bad("align.num_experts must equal route.E + has_shared");
    check_align(&al, r, true);
    if (!r.ok()) return r.finish("smr_route_align");
    smr_status st = check_ws(workspace, workspace_bytes, smr_route_align_workspace_size(route, &al),
                             "smr_route_align");
    if (st != SMR_OK) return st;
    if ((st = check_device()) != SMR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    if (route->M >= 1 && route->M <= smr::kSmallMaxM && !has_eplb(&al)) {
        st = run_route(route, workspace, s, &al, &launches);
        if (st == SMR_OK) g_last_launches = launches;
        return st;
    }
    if (route->M > 0 && (int64_t)route->M * al.width <= smr::kFusedAlignMax && !has_eplb(&al) &&
        !generic_route(route)) {
        // mid M: one launch, the align fused into the route's last CTA
        st = run_route(route, workspace, s, &al, &launches);
        if (st == SMR_OK) g_last_launches = launches;
        return st;
    }
    const bool counted = align_counted_by_route(route, &al, (int64_t)route->M * al.width);
    smr::AlignLaunch L = make_align_launch(&al, route->topk_ids, workspace,
                                           kHeaderBytes + route_scratch_bytes(route),
                                           counted ? smr::kTcCountRows * al.width : 0);
    if (route->M > 0) {
        st = run_route(route, workspace, s, nullptr, &launches, counted ? L.tile_counts : nullptr);
        if (st != SMR_OK) return st;
    }
    cudaError_t e = smr::launch_align(L, s);
    if (e != cudaSuccess) return cuda_fail("align launch", e);
    launches += smr::align_launches(L.numel, counted);
    g_last_launches = launches;
    return SMR_OK;
}


SMR_API smr_status smr_route_align_static(const smr_route_args *route, const smr_align_args *align,
                                          void *stream) {
    g_last_launches = 0;
    if (!route || !align) {
        g_last_error = "smr_route_align_static: route or align args is NULL";
        return SMR_ERR_INVALID_ARG;
    }
    Reasons r;
    check_route(route, r);
    const int S = route->has_shared ? 1 : 0;
    smr_align_args al = *align;
    al.routed_topk = route->topk;
    al.routed_experts = route->E;
    if (align->topk_ids != route->topk_ids) r.bad("align.topk_ids must equal route.topk_ids");
    if (align->num_tokens != route->M) r.bad("align.num_tokens must equal route.M");
    if (align->width != route->topk + S) r.bad("align.width must equal route.topk + has_shared");
    if (align->num_experts != route->E + S) r.bad("align.num_experts must equal route.E + has_shared");
    check_align(&al, r, true);
    if (route->M < 1 || route->M > smr::kSmallMaxM)
        r.unsup("the fixed-scratch entry point covers 1 <= M <= 16 (got M=" +
                std::to_string(route->M) + ")");
    if (has_eplb(&al)) r.unsup("the fixed-scratch entry point takes no EPLB remap");
    if (!r.ok()) return r.finish("smr_route_align_static");
    const size_t need = smr_route_align_workspace_size(route, &al);
    if (need > smr::kStaticScratchBytes) {
        r.unsup("needs " + std::to_string(need) + " bytes of scratch, above the fixed " +
                std::to_string(smr::kStaticScratchBytes) + "-byte array");
        return r.finish("smr_route_align_static");
    }
    smr_status st = check_device();
    if (st != SMR_OK) return st;
    void *scratch = nullptr;
    cudaError_t e = smr::static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail("smr_route_align_static: scratch set-up", e);
    int launches = 0;
    st = run_route(route, scratch, static_cast<cudaStream_t>(stream), &al, &launches);
    if (st == SMR_OK) g_last_launches = launches;
    return st;
}

SMR_API smr_status smr_expert_gemm(const smr_expert_gemm_args *a, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    g_last_launches = 0;
    if (!a) {
        g_last_error = "smr_expert_gemm: args is NULL";
        return SMR_ERR_INVALID_ARG;
    }
    Reasons r;
    if (a->num_tokens < 0) r.bad("num_tokens must be >= 0");
    if (a->width < 1) r.bad("width must be >= 1");
    if (a->H < 64 || a->H > kMaxH || a->H % 64 != 0)
        r.bad("H must be a multiple of 64 in [64, 16384] (got " + std::to_string(a->H) + ")");
    if (a->N < 128 || a->N > kMaxH || a->N % 128 != 0)
        r.bad("N must be a multiple of 128 in [128, 16384] (got " + std::to_string(a->N) + ")");
    if (a->num_experts < 1 || a->num_experts > kMaxExperts + 1)
        r.bad("num_experts must be in [1, 1025] (got " + std::to_string(a->num_experts) + ")");
    if (a->block_size != 64 && a->block_size != 128)
        r.unsup("block_size must be 64 or 128 (the MMA's rows; got " + std::to_string(a->block_size) + ")");
    const int64_t numel = (int64_t)a->num_tokens * a->width;
    if (numel > 0) {
        if (!a->hidden || !aligned(a->hidden, 16)) r.bad("hidden must be a 16-byte aligned pointer");
        if (a->ld_hidden < a->H || a->ld_hidden % 8 != 0) r.bad("ld_hidden must be >= H and a multiple of 8");
        if (!a->expert_w || !aligned(a->expert_w, 16)) r.bad("expert_w must be a 16-byte aligned pointer");
        if (!a->sorted_token_ids || !a->expert_ids || !a->num_tokens_post_padded)
            r.bad("sorted_token_ids, expert_ids and num_tokens_post_padded must be set");
        if (!a->out || !aligned(a->out, 16)) r.bad("out must be a 16-byte aligned pointer");
        if (a->sorted_cap < 1) r.bad("sorted_cap must be >= 1");
        if (numel * (int64_t)a->N > ((int64_t)1 << 40)) r.unsup("num_tokens * width * N too large");
    }
    if (!r.ok()) return r.finish("smr_expert_gemm");
    if (numel == 0) return SMR_OK;
    smr_status st = check_ws(workspace, workspace_bytes, kHeaderBytes, "smr_expert_gemm");
    if (st != SMR_OK) return st;
    if ((st = check_device()) != SMR_OK) return st;
    smr::ExpertGemmLaunch L{};
    L.x = static_cast<const uint16_t *>(a->hidden);
    L.ld = a->ld_hidden;
    L.width = a->width;
    L.H = a->H;
    L.N = a->N;
    L.A = a->block_size;
    L.num_experts = a->num_experts;
    L.numel = numel;
    L.max_blocks = (a->sorted_cap + a->block_size - 1) / a->block_size;
    L.w = static_cast<const uint16_t *>(a->expert_w);
    L.sorted = a->sorted_token_ids;
    L.eids = a->expert_ids;
    L.npp = a->num_tokens_post_padded;
    L.out = a->out;
    L.hdr = workspace;
    cudaError_t e = smr::launch_expert_gemm(L, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("expert GEMM launch", e);
    g_last_launches = 1;
    return SMR_OK;
}

SMR_API smr_status smr_get_device_error(const void *workspace, void *stream, int32_t *code_out) {
    if (!workspace || !code_out) {
        g_last_error = "smr_get_device_error: workspace or code_out is NULL";
        return SMR_ERR_INVALID_ARG;
    }
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("smr_get_device_error", e);
    uint32_t word = 0;
    e = cudaMemcpy(&word, static_cast<const uint8_t *>(workspace) + 4, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail("smr_get_device_error", e);
    *code_out = (int32_t)word;
    return SMR_OK;
}

SMR_API smr_status smr_clear_device_error(void *workspace, void *stream) {
    if (!workspace) {
        g_last_error = "smr_clear_device_error: workspace is NULL";
        return SMR_ERR_INVALID_ARG;
    }
    cudaError_t e = cudaMemsetAsync(static_cast<uint8_t *>(workspace) + 4, 0, 4,
                                    static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("smr_clear_device_error", e);
    return SMR_OK;
}

SMR_API smr_status smr_get_static_device_error(void *stream, int32_t *code_out) {
    if (!code_out) {
        g_last_error = "smr_get_static_device_error: code_out is NULL";
        return SMR_ERR_INVALID_ARG;
    }
    smr_status st = check_device();
    if (st != SMR_OK) return st;
    void *scratch = nullptr;
    cudaError_t e = smr::static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail("smr_get_static_device_error: scratch set-up", e);
    return smr_get_device_error(scratch, stream, code_out);
}

SMR_API smr_status smr_clear_static_device_error(void *stream) {
    smr_status st = check_device();
    if (st != SMR_OK) return st;
    void *scratch = nullptr;
    cudaError_t e = smr::static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail("smr_clear_static_device_error: scratch set-up", e);
    return smr_clear_device_error(scratch, stream);
}

SMR_API smr_status smr_test_force_wait_timeout(int32_t site, int64_t limit) {
    if (site < SMR_STALL_NONE || site > SMR_STALL_TC_MERGE || (site != SMR_STALL_NONE && limit < 1)) {
        g_last_error = "smr_test_force_wait_timeout: site must be 0, 1 or 2 and limit >= 1 when set";
        return SMR_ERR_INVALID_ARG;
    }
    g_stall_limit.store(site == SMR_STALL_NONE ? 0 : limit, std::memory_order_relaxed);
    g_stall_site.store(site, std::memory_order_relaxed);
    return SMR_OK;
}

SMR_API const char *smr_status_string(smr_status status) {
    switch (status) {
        case SMR_OK: return "SMR_OK";
        case SMR_ERR_INVALID_ARG: return "SMR_ERR_INVALID_ARG";
        case SMR_ERR_UNSUPPORTED: return "SMR_ERR_UNSUPPORTED";
        case SMR_ERR_WORKSPACE: return "SMR_ERR_WORKSPACE";
        case SMR_ERR_CUDA: return "SMR_ERR_CUDA";
        case SMR_ERR_DEVICE: return "SMR_ERR_DEVICE";
    }
    return "SMR_ERR_UNKNOWN";
}

SMR_API const char *smr_last_error(void) { return g_last_error.c_str(); }

SMR_API int32_t smr_version(void) { return 0x000200; }

SMR_API int32_t smr_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
