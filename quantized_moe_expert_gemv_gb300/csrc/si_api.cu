// si_api.cu -- the C ABI (include/si_moe.h): plans, validation, scratch
// layout and stream-ordered launches.  Nothing here allocates device memory
// or synchronises, except si_moe_read_status and si_moe_forward_decode_host
// (which are documented to).
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "si_internal.h"

using si::DecodeArgs;
using si::DecodeLayout;
using si::Plan;

// One captured host-buffer decode (si_moe_forward_decode_host): the copy of x
// from a page-locked staging buffer into the scratch, the decode's launches,
// and the copies of out and of the status word back into page-locked staging.
// Its key is everything the captured launches bake in.
struct HostGraph {
    si_moe_layer layer{};
    si_moe_route_out ro{};
    bool has_ro = false;
    void *scratch = nullptr;
    int n = 0;
    cudaGraphExec_t exec = nullptr;
    uint8_t *x_pin = nullptr;    // [n][H] bf16
    uint8_t *out_pin = nullptr;  // [n][H] fp32, then the status word
};

struct si_moe_plan_s {
    Plan p;
    std::mutex host_mu;                  // serialises the host-buffer calls on this plan
    std::vector<HostGraph> host_graphs;  // least recently used first
    ~si_moe_plan_s() {
        for (HostGraph &g : host_graphs) {
            if (g.exec) cudaGraphExecDestroy(g.exec);
            if (g.x_pin) cudaFreeHost(g.x_pin);
            if (g.out_pin) cudaFreeHost(g.out_pin);
        }
        cudaGetLastError();
    }
};

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

si_status validate_desc(const si_moe_desc *d) {
    if (!d) return SI_ERR_INVALID_ARG;
    if (d->wtype != SI_WTYPE_Q4_K && d->wtype != SI_WTYPE_Q5_K && d->wtype != SI_WTYPE_NVFP4) return SI_ERR_UNSUPPORTED;
    if ((d->flags & ~SI_FLAG_ACT_INT8) != 0) return SI_ERR_UNSUPPORTED;
    if ((d->flags & SI_FLAG_ACT_INT8) && d->wtype != SI_WTYPE_Q4_K) return SI_ERR_UNSUPPORTED;
    if (d->hidden <= 0 || d->intermediate <= 0 || d->hidden % 256 || d->intermediate % 256)
        return SI_ERR_INVALID_ARG;
    if (d->n_experts < 1 || d->n_experts > SI_MAX_EXPERTS) return SI_ERR_INVALID_ARG;
    if (d->top_k < 1 || d->top_k > d->n_experts || d->top_k > SI_MAX_TOPK) return SI_ERR_INVALID_ARG;
    if (d->max_tokens < 1) return SI_ERR_INVALID_ARG;
    // decode keeps n tokens of activations (fp32) in shared memory
    if ((size_t)SI_MAX_DECODE_TOKENS * d->hidden * 4 * 33 / 32 > 200 * 1024) return SI_ERR_UNSUPPORTED;
    return SI_OK;
}

}  // namespace

namespace si {

DecodeLayout decode_layout(const si_moe_desc &d, int n) {
    DecodeLayout L{};
    size_t o = 0;
    auto take = [&o](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.ctrl = take(kCtrlBytes);
    L.logits = take((size_t)n * d.n_experts * sizeof(float));
    L.ids = take((size_t)n * d.top_k * sizeof(int32_t));
    L.wts = take((size_t)n * d.top_k * sizeof(float));
    L.counts = take((size_t)d.n_experts * sizeof(int32_t));
    L.uniq = take(sizeof(UniqTable));
    L.h = take((size_t)n * d.top_k * d.intermediate * sizeof(float));
    L.xq = take((size_t)n * (d.hidden / 64) * kXqWords * sizeof(uint32_t));
    L.total = o;
    return L;
}

PrefillLayout prefill_layout(const si_moe_desc &d, int n) {
    PrefillLayout L{};
    size_t o = 0;
    auto take = [&o](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    const size_t pairs = (size_t)n * d.top_k;
    const size_t rows = pairs + 32 * (size_t)d.n_experts;
    L.rows = (int64_t)rows;
    L.ctrl = take(kCtrlBytes);
    L.wt = take((size_t)((d.n_experts + 127) / 128 * 128) * d.hidden * sizeof(float));
    L.logits = take((size_t)n * d.n_experts * sizeof(float));
    L.ids = take(pairs * sizeof(int32_t));
    L.wts = take(pairs * sizeof(float));
    L.counts = take((size_t)d.n_experts * sizeof(int32_t));
    L.hist = take((size_t)((n + 31) / 32) * d.n_experts * sizeof(int32_t));
    L.rms = take((size_t)n * sizeof(float));
    L.rrow = take(rows * sizeof(float));
    L.offsets = take(((size_t)d.n_experts + 1) * sizeof(int32_t));
    L.poff = take(((size_t)d.n_experts + 1) * sizeof(int32_t));
    L.perm = take(pairs * sizeof(int32_t));
    L.pperm = take(rows * sizeof(int32_t));
    L.inv = take(pairs * sizeof(int32_t));
    L.xp = take(rows * d.hidden * sizeof(uint16_t));
    L.h = take(rows * d.intermediate * sizeof(uint16_t));
    L.y = take(rows * d.hidden * sizeof(float));
    L.total = o;
    return L;
}

}  // namespace si

extern "C" {

const char *si_status_string(si_status s) {
    switch (s) {
        case SI_OK: return "ok";
        case SI_ERR_INVALID_ARG: return "invalid argument";
        case SI_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case SI_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        case SI_ERR_SCRATCH_TOO_SMALL: return "scratch buffer too small";
        case SI_ERR_CUDA: return "CUDA error";
        case SI_ERR_TIMEOUT: return "device-side wait timed out";
        case SI_ERR_DEVICE: return "device-side check failed";
        case SI_ERR_RANGE: return "value outside the fp16 range of the prefill operands";
    }
    return "unknown status";
}

si_status si_moe_plan(const si_moe_desc *desc, int cuda_device, si_moe_plan_t *out) {
    if (!out) return SI_ERR_INVALID_ARG;
    *out = nullptr;
    const si_status v = validate_desc(desc);
    if (v != SI_OK) return v;
    Plan p{};
    p.desc = *desc;
    p.device = cuda_device;
    if (cudaDeviceGetAttribute(&p.sm_count, cudaDevAttrMultiProcessorCount, cuda_device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p.l2_bytes, cudaDevAttrL2CacheSize, cuda_device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, cuda_device) !=
            cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, cuda_device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, cuda_device);
    if (major != 10 || minor != 3) return SI_ERR_UNSUPPORTED;  // built for sm_103a only
    p.dec = si::decode_layout(*desc, SI_MAX_DECODE_TOKENS);
    // Bounded device-side waits: about one second at GB300 clocks.  A test may
    // shorten the budget through SI_FAULT_WAIT_BUDGET (a non-negative decimal
    // cycle count); unset or malformed leaves the default.
    p.wait_budget = 2000000000LL;
    p.fault_wait = false;
    if (const char *env = std::getenv("SI_FAULT_WAIT_BUDGET")) {
        char *end = nullptr;
        const long long v = std::strtoll(env, &end, 10);
        if (end && end != env && *end == '\0' && v >= 0) {
            p.wait_budget = v;
            p.fault_wait = true;  // and make a wait run out for certain: see kCtrlFaultFlag
        }
    }
    const int cur_dev = [] { int d = 0; cudaGetDevice(&d); return d; }();
    if (cur_dev != cuda_device) cudaSetDevice(cuda_device);
    for (int n = 1; n <= SI_MAX_DECODE_TOKENS; ++n) {
        si::DecodeArgs tmp{};
        p.fused_ok[n] = false;
        if (desc->wtype == SI_WTYPE_Q4_K && si::expert_fused_layout(*desc, n, p.sm_count, p.smem_optin, tmp)) {
            int per_sm = 0;
            if (si::expert_fused_occupancy(desc->hidden / 256, n > 1, tmp.fz_smem, p.smem_optin, &per_sm) == cudaSuccess &&
                per_sm >= 1)
                p.fused_ok[n] = true;
            cudaGetLastError();
        }
    }
    {
        // Largest cluster size whose clusters (one per selected expert and 256-wide
        // block of the intermediate dimension) are all resident at once.
        p.cluster_ok = false;
        p.cluster_size = 0;
        p.cluster_active = 0;
        const int units = desc->top_k * (desc->intermediate / 256);
        for (int C = 8; C >= 2 && !p.cluster_ok; --C) {
            si::DecodeArgs tmp{};
            if (units * C > p.sm_count) continue;
            if (!si::expert_cluster_layout(*desc, C, p.smem_optin, tmp)) continue;
            int clusters = 0;
            if (si::expert_cluster_prepare(desc->hidden / 256, p.smem_optin, tmp.cl_smem, C, &clusters) ==
                    cudaSuccess &&
                clusters >= units) {
                p.cluster_ok = true;
                p.cluster_size = C;
                p.cluster_active = clusters;
            }
            cudaGetLastError();
        }
        // 2..4 tokens of a plain block: clusters over the distinct experts, in waves.  The
        // single-token cluster size if the per-token buffers fit beside its stages, else the
        // smallest larger size that fits (one resident cluster is enough: the units run in
        // waves).  The int8-activation flag applies to single tokens only: batched tokens
        // keep int16 activations.
        p.cluster_mt_ok = false;
        p.cluster_mt_size = 0;
        p.cluster_mt_active = 0;
        if (p.cluster_ok && si::router_one_shape(desc->n_experts, desc->hidden) && desc->top_k <= 8) {
            for (int C = p.cluster_size; C <= 8 && !p.cluster_mt_ok; ++C) {
                si::DecodeArgs tmp{};
                if (!si::expert_cluster_layout(*desc, C, p.smem_optin, tmp, SI_MAX_DECODE_TOKENS)) continue;
                int clusters = 0;
                if (si::expert_cluster_prepare(desc->hidden / 256, p.smem_optin, tmp.cl_smem, C, &clusters, true) ==
                        cudaSuccess &&
                    clusters >= 1) {
                    p.cluster_mt_ok = true;
                    p.cluster_mt_size = C;
                    p.cluster_mt_active = clusters;
                }
                cudaGetLastError();
            }
        }
    }
    p.prefill_ok = si::prefill_prepare(p) == cudaSuccess;
    cudaGetLastError();
    if (cur_dev != cuda_device) cudaSetDevice(cur_dev);
    si_moe_plan_s *h = new (std::nothrow) si_moe_plan_s;
    if (!h) return SI_ERR_INVALID_ARG;
    h->p = p;
    *out = h;
    return SI_OK;
}

void si_moe_plan_destroy(si_moe_plan_t plan) { delete plan; }

// Scratch of si_moe_forward_decode_host: the decode scratch, then the device
// copies of x ([n][H] bf16) and of out ([n][H] fp32), each 256-byte aligned.
struct HostStaging {
    size_t x, out, total;
};
static HostStaging host_staging(const si_moe_desc &d, int n) {
    HostStaging h{};
    h.x = si::decode_layout(d, n).total;
    h.out = align_up(h.x + (size_t)n * d.hidden * sizeof(uint16_t), 256);
    h.total = align_up(h.out + (size_t)n * d.hidden * sizeof(float), 256);
    return h;
}

si_status si_moe_scratch_bytes(si_moe_plan_t plan, int mode, int32_t n_tokens, size_t *bytes) {
    if (!plan || !bytes) return SI_ERR_INVALID_ARG;
    const si_moe_desc &d = plan->p.desc;
    if (mode == SI_MODE_DECODE) {
        if (n_tokens < 1 || n_tokens > SI_MAX_DECODE_TOKENS) return SI_ERR_INVALID_ARG;
        *bytes = si::decode_layout(d, n_tokens).total;
        return SI_OK;
    }
    if (mode == SI_MODE_DECODE_HOST) {
        if (n_tokens < 1 || n_tokens > SI_MAX_DECODE_TOKENS) return SI_ERR_INVALID_ARG;
        *bytes = host_staging(d, n_tokens).total;
        return SI_OK;
    }
    if (mode == SI_MODE_PREFILL) {
        if (n_tokens < 1 || n_tokens > d.max_tokens) return SI_ERR_INVALID_ARG;
        *bytes = si::prefill_layout(d, n_tokens).total;
        return SI_OK;
    }
    return SI_ERR_INVALID_ARG;
}

si_status si_moe_scratch_init(si_moe_plan_t plan, void *scratch, size_t scratch_bytes,
                              si_stream_t stream) {
    if (!plan || !scratch) return SI_ERR_INVALID_ARG;
    if (!aligned(scratch, 16)) return SI_ERR_MISALIGNED;
    if (scratch_bytes < si::kCtrlBytes) return SI_ERR_SCRATCH_TOO_SMALL;
    if (cudaMemsetAsync(scratch, 0, si::kCtrlBytes, (cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    return SI_OK;
}

}  // extern "C"

// NVFP4 layers carry their tensor scales (and have no pre-normed variant);
// Q4_K layers carry none.
static si_status check_weight_scales(const si_moe_desc &d, const si_moe_layer *layer) {
    if (d.wtype == SI_WTYPE_NVFP4) {
        if (!layer->w_scale) return SI_ERR_INVALID_ARG;
        if (!aligned(layer->w_scale, 4)) return SI_ERR_MISALIGNED;
        if (layer->norm_weight) return SI_ERR_UNSUPPORTED;
    } else if (layer->w_scale) {
        return SI_ERR_INVALID_ARG;
    }
    if ((d.flags & SI_FLAG_ACT_INT8) && layer->norm_weight) return SI_ERR_UNSUPPORTED;
    if (d.wtype == SI_WTYPE_Q5_K && layer->norm_weight) return SI_ERR_UNSUPPORTED;  // plain Q5_K blocks only
    return SI_OK;
}

// Every argument check of a decode call except those of the scratch buffer.
si_status si::check_decode_args(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                int32_t n_tokens, const float *out, const si_moe_route_out *ro) {
    if (!plan || !layer || !x_bf16 || !out) return SI_ERR_INVALID_ARG;
    if (!layer->w_gate || !layer->w_up || !layer->w_down || !layer->router_w) return SI_ERR_INVALID_ARG;
    if (n_tokens < 1 || n_tokens > SI_MAX_DECODE_TOKENS) return SI_ERR_INVALID_ARG;
    if (!aligned(layer->w_gate, 16) || !aligned(layer->w_up, 16) || !aligned(layer->w_down, 16) ||
        !aligned(layer->router_w, 16) || !aligned(x_bf16, 16) || !aligned(out, 16) ||
        (layer->router_bias && !aligned(layer->router_bias, 4)) ||
        (layer->norm_weight && !aligned(layer->norm_weight, 16)))
        return SI_ERR_MISALIGNED;
    if (layer->norm_weight && !(layer->norm_eps >= 0.f && layer->norm_eps <= 3.0e38f)) return SI_ERR_INVALID_ARG;
    if (ro && ((ro->topk_ids && !aligned(ro->topk_ids, 4)) || (ro->topk_w && !aligned(ro->topk_w, 4)) ||
               (ro->expert_counts && !aligned(ro->expert_counts, 4)) ||
               (ro->logits && !aligned(ro->logits, 4))))
        return SI_ERR_MISALIGNED;
    const si_status wst = check_weight_scales(plan->p.desc, layer);
    if (wst != SI_OK) return wst;
    return SI_OK;
}

extern "C" {

static si_status forward_decode_impl(si_moe_plan_t plan, const si_moe_layer *layer,
                                     const void *x_bf16, int32_t n_tokens, float *out,
                                     si_moe_route_out *ro, void *scratch, size_t scratch_bytes,
                                     cudaEvent_t const *events, si_stream_t stream) {
    const si_status chk = si::check_decode_args(plan, layer, x_bf16, n_tokens, out, ro);
    if (chk != SI_OK) return chk;
    if (!scratch) return SI_ERR_INVALID_ARG;
    if (!aligned(scratch, 16)) return SI_ERR_MISALIGNED;
    const si_moe_desc &d = plan->p.desc;
    const DecodeLayout L = si::decode_layout(d, n_tokens);
    if (scratch_bytes < L.total) return SI_ERR_SCRATCH_TOO_SMALL;
    uint8_t *sb = static_cast<uint8_t *>(scratch);
    DecodeArgs a{};
    a.wg = static_cast<const uint8_t *>(layer->w_gate);
    a.wu = static_cast<const uint8_t *>(layer->w_up);
    a.wd = static_cast<const uint8_t *>(layer->w_down);
    a.router_w = layer->router_w;
    a.router_bias = layer->router_bias;
    a.norm_w = layer->norm_weight;
    a.norm_eps = layer->norm_weight ? layer->norm_eps : 0.f;
    a.wtype = d.wtype;
    a.wscale = layer->w_scale;
    a.x = static_cast<const uint16_t *>(x_bf16);
    a.out = out;
    a.H = d.hidden;
    a.I = d.intermediate;
    a.E = d.n_experts;
    a.k = d.top_k;
    a.n = n_tokens;
    a.ctrl = reinterpret_cast<int32_t *>(sb + L.ctrl);
    a.logits = reinterpret_cast<float *>(sb + L.logits);
    a.ids = reinterpret_cast<int32_t *>(sb + L.ids);
    a.wts = reinterpret_cast<float *>(sb + L.wts);
    a.counts = reinterpret_cast<int32_t *>(sb + L.counts);
    a.uniq = reinterpret_cast<si::UniqTable *>(sb + L.uniq);
    a.h = reinterpret_cast<float *>(sb + L.h);
    a.xq = reinterpret_cast<uint32_t *>(sb + L.xq);
    if (ro) {
        a.o_ids = ro->topk_ids;
        a.o_w = ro->topk_w;
        a.o_counts = ro->expert_counts;
        a.o_logits = ro->logits;
    }
    if (si::launch_decode(plan->p, a, (cudaStream_t)stream, events) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    return SI_OK;
}

si_status si_moe_forward_decode(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                int32_t n_tokens, float *out, si_moe_route_out *ro, void *scratch,
                                size_t scratch_bytes, si_stream_t stream) {
    return forward_decode_impl(plan, layer, x_bf16, n_tokens, out, ro, scratch, scratch_bytes,
                               nullptr, stream);
}

constexpr size_t kHostGraphs = 4;  // captured host-buffer decodes kept per plan

// Field by field: a caller's struct may hold anything in its padding.
static bool same_host_key(const HostGraph &g, const si_moe_layer *layer, const si_moe_route_out *ro,
                          void *scratch, int n) {
    const si_moe_layer &a = g.layer;
    const bool same_layer = a.w_gate == layer->w_gate && a.w_up == layer->w_up && a.w_down == layer->w_down &&
                            a.router_w == layer->router_w && a.router_bias == layer->router_bias &&
                            a.norm_weight == layer->norm_weight && a.w_scale == layer->w_scale &&
                            (!a.norm_weight || std::memcmp(&a.norm_eps, &layer->norm_eps, sizeof(float)) == 0);
    const bool same_ro = g.has_ro == (ro != nullptr) &&
                         (!ro || (g.ro.topk_ids == ro->topk_ids && g.ro.topk_w == ro->topk_w &&
                                  g.ro.expert_counts == ro->expert_counts &&
                                  g.ro.expert_offsets == ro->expert_offsets && g.ro.perm == ro->perm &&
                                  g.ro.logits == ro->logits));
    return g.n == n && g.scratch == scratch && same_layer && same_ro;
}

static void free_host_graph(HostGraph &g) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.x_pin) cudaFreeHost(g.x_pin);
    if (g.out_pin) cudaFreeHost(g.out_pin);
    g = HostGraph{};
    cudaGetLastError();
}

// Capture one host-buffer decode on a private stream and instantiate it.
static si_status build_host_graph(si_moe_plan_t plan, HostGraph &g) {
    const si_moe_desc &d = plan->p.desc;
    const HostStaging hs = host_staging(d, g.n);
    const size_t x_bytes = (size_t)g.n * d.hidden * sizeof(uint16_t);
    const size_t out_bytes = (size_t)g.n * d.hidden * sizeof(float);
    uint8_t *sb = static_cast<uint8_t *>(g.scratch);
    if (cudaHostAlloc(reinterpret_cast<void **>(&g.x_pin), x_bytes, cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(reinterpret_cast<void **>(&g.out_pin), out_bytes + sizeof(int32_t), cudaHostAllocDefault) !=
            cudaSuccess) {
        free_host_graph(g);
        return SI_ERR_CUDA;
    }
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
        free_host_graph(g);
        return SI_ERR_CUDA;
    }
    si_status st = SI_OK;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        st = SI_ERR_CUDA;
    } else {
        if (cudaMemcpyAsync(sb + hs.x, g.x_pin, x_bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess) st = SI_ERR_CUDA;
        if (st == SI_OK)
            st = forward_decode_impl(plan, &g.layer, sb + hs.x, g.n, reinterpret_cast<float *>(sb + hs.out),
                                     g.has_ro ? &g.ro : nullptr, g.scratch, hs.x, nullptr, cs);
        if (st == SI_OK &&
            (cudaMemcpyAsync(g.out_pin, sb + hs.out, out_bytes, cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
             cudaMemcpyAsync(g.out_pin + out_bytes, g.scratch, sizeof(int32_t), cudaMemcpyDeviceToHost, cs) !=
                 cudaSuccess))
            st = SI_ERR_CUDA;
        cudaGraph_t graph = nullptr;  // the capture is ended whatever happened inside it
        if (cudaStreamEndCapture(cs, &graph) != cudaSuccess && st == SI_OK) st = SI_ERR_CUDA;
        if (st == SI_OK && cudaGraphInstantiate(&g.exec, graph, 0) != cudaSuccess) st = SI_ERR_CUDA;
        if (graph) cudaGraphDestroy(graph);
    }
    cudaStreamDestroy(cs);
    if (st != SI_OK) free_host_graph(g);
    cudaGetLastError();
    return st;
}

si_status si_moe_forward_decode_host(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16_host,
                                     int32_t n_tokens, float *out_host, si_moe_route_out *ro, void *scratch,
                                     size_t scratch_bytes, si_stream_t stream) {
    if (!plan || !x_bf16_host || !out_host || !scratch) return SI_ERR_INVALID_ARG;
    if (n_tokens < 1 || n_tokens > SI_MAX_DECODE_TOKENS) return SI_ERR_INVALID_ARG;
    if (!aligned(scratch, 16)) return SI_ERR_MISALIGNED;
    const si_moe_desc &d = plan->p.desc;
    const HostStaging hs = host_staging(d, n_tokens);
    if (scratch_bytes < hs.total) return SI_ERR_SCRATCH_TOO_SMALL;
    uint8_t *sb = static_cast<uint8_t *>(scratch);
    // every argument error before anything is queued
    const si_status chk = si::check_decode_args(plan, layer, sb + hs.x, n_tokens,
                                                reinterpret_cast<const float *>(sb + hs.out), ro);
    if (chk != SI_OK) return chk;
    const size_t x_bytes = (size_t)n_tokens * d.hidden * sizeof(uint16_t);
    const size_t out_bytes = (size_t)n_tokens * d.hidden * sizeof(float);

    std::lock_guard<std::mutex> lock(plan->host_mu);
    std::vector<HostGraph> &cache = plan->host_graphs;
    size_t at = cache.size();
    for (size_t i = 0; i < cache.size(); ++i)
        if (same_host_key(cache[i], layer, ro, scratch, n_tokens)) at = i;
    if (at == cache.size()) {  // first call with this layer, scratch and token count
        HostGraph g{};
        g.layer = *layer;
        if (ro) g.ro = *ro;
        g.has_ro = ro != nullptr;
        g.scratch = scratch;
        g.n = n_tokens;
        const si_status st = build_host_graph(plan, g);
        if (st != SI_OK) return st;
        if (cache.size() == kHostGraphs) {
            free_host_graph(cache.front());
            cache.erase(cache.begin());
        }
        cache.push_back(g);
        at = cache.size() - 1;
    } else if (at + 1 != cache.size()) {  // most recently used last
        const HostGraph g = cache[at];
        cache.erase(cache.begin() + (long)at);
        cache.push_back(g);
        at = cache.size() - 1;
    }
    HostGraph &g = cache[at];
    std::memcpy(g.x_pin, x_bf16_host, x_bytes);
    if (cudaGraphLaunch(g.exec, (cudaStream_t)stream) != cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    std::memcpy(out_host, g.out_pin, out_bytes);
    int32_t word = 0;
    std::memcpy(&word, g.out_pin + out_bytes, sizeof(word));
    if (word != 0) {  // reported once, as si_moe_read_status does
        if (cudaMemsetAsync(scratch, 0, sizeof(word), (cudaStream_t)stream) != cudaSuccess) {
            cudaGetLastError();
            return SI_ERR_CUDA;
        }
        return (si_status)word;
    }
    return SI_OK;
}

si_status si_debug_decode_events(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                 int32_t n_tokens, float *out, si_moe_route_out *ro, void *scratch,
                                 size_t scratch_bytes, void *const *events, si_stream_t stream) {
    return forward_decode_impl(plan, layer, x_bf16, n_tokens, out, ro, scratch, scratch_bytes,
                               reinterpret_cast<cudaEvent_t const *>(events), stream);
}

static si_status forward_prefill_impl(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                      int32_t n_tokens, float *out, si_moe_route_out *ro, void *scratch,
                                      size_t scratch_bytes, cudaEvent_t const *events, si_stream_t stream) {
    if (!plan || !layer || !x_bf16 || !out || !scratch) return SI_ERR_INVALID_ARG;
    if (!layer->w_gate || !layer->w_up || !layer->w_down || !layer->router_w) return SI_ERR_INVALID_ARG;
    const si_moe_desc &d = plan->p.desc;
    if (n_tokens < 1 || n_tokens > d.max_tokens) return SI_ERR_INVALID_ARG;
    if (!aligned(layer->w_gate, 16) || !aligned(layer->w_up, 16) || !aligned(layer->w_down, 16) ||
        !aligned(layer->router_w, 16) || !aligned(x_bf16, 16) || !aligned(out, 16) ||
        !aligned(scratch, 16) || (layer->router_bias && !aligned(layer->router_bias, 4)) ||
        (layer->norm_weight && !aligned(layer->norm_weight, 16)))
        return SI_ERR_MISALIGNED;
    if (layer->norm_weight && !(layer->norm_eps >= 0.f && layer->norm_eps <= 3.0e38f)) return SI_ERR_INVALID_ARG;
    if (ro && ((ro->topk_ids && !aligned(ro->topk_ids, 4)) || (ro->topk_w && !aligned(ro->topk_w, 4)) ||
               (ro->expert_counts && !aligned(ro->expert_counts, 4)) ||
               (ro->expert_offsets && !aligned(ro->expert_offsets, 4)) || (ro->perm && !aligned(ro->perm, 4)) ||
               (ro->logits && !aligned(ro->logits, 4))))
        return SI_ERR_MISALIGNED;
    const si_status wst = check_weight_scales(d, layer);
    if (wst != SI_OK) return wst;
    if (!plan->p.prefill_ok) return SI_ERR_UNSUPPORTED;
    const si::PrefillLayout L = si::prefill_layout(d, n_tokens);
    if (scratch_bytes < L.total) return SI_ERR_SCRATCH_TOO_SMALL;
    uint8_t *sb = static_cast<uint8_t *>(scratch);
    si::PrefillArgs a{};
    a.wg = static_cast<const uint8_t *>(layer->w_gate);
    a.wu = static_cast<const uint8_t *>(layer->w_up);
    a.wd = static_cast<const uint8_t *>(layer->w_down);
    a.router_w = layer->router_w;
    a.router_bias = layer->router_bias;
    a.norm_w = layer->norm_weight;
    a.norm_eps = layer->norm_weight ? layer->norm_eps : 0.f;
    a.wtype = d.wtype;
    a.wscale = layer->w_scale;
    a.x = static_cast<const uint16_t *>(x_bf16);
    a.out = out;
    a.H = d.hidden;
    a.I = d.intermediate;
    a.E = d.n_experts;
    a.k = d.top_k;
    a.T = n_tokens;
    a.ctrl = reinterpret_cast<int32_t *>(sb + L.ctrl);
    a.logits = reinterpret_cast<float *>(sb + L.logits);
    a.ids = reinterpret_cast<int32_t *>(sb + L.ids);
    a.wts = reinterpret_cast<float *>(sb + L.wts);
    a.counts = reinterpret_cast<int32_t *>(sb + L.counts);
    a.hist = reinterpret_cast<int32_t *>(sb + L.hist);
    a.rms = reinterpret_cast<float *>(sb + L.rms);
    a.rrow = reinterpret_cast<float *>(sb + L.rrow);
    a.offsets = reinterpret_cast<int32_t *>(sb + L.offsets);
    a.rows = L.rows;
    a.wt = reinterpret_cast<float *>(sb + L.wt);
    a.poff = reinterpret_cast<int32_t *>(sb + L.poff);
    a.perm = reinterpret_cast<int32_t *>(sb + L.perm);
    a.pperm = reinterpret_cast<int32_t *>(sb + L.pperm);
    a.inv = reinterpret_cast<int32_t *>(sb + L.inv);
    a.xp = reinterpret_cast<uint16_t *>(sb + L.xp);
    a.h = reinterpret_cast<uint16_t *>(sb + L.h);
    a.y = reinterpret_cast<float *>(sb + L.y);
    if (ro) {
        a.o_ids = ro->topk_ids;
        a.o_w = ro->topk_w;
        a.o_counts = ro->expert_counts;
        a.o_offsets = ro->expert_offsets;
        a.o_perm = ro->perm;
        a.o_logits = ro->logits;
    }
    a.wait_budget = plan->p.wait_budget;
    if (si::launch_prefill(plan->p, a, (cudaStream_t)stream, events) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    return SI_OK;
}

si_status si_moe_forward_prefill(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                 int32_t n_tokens, float *out, si_moe_route_out *ro, void *scratch,
                                 size_t scratch_bytes, si_stream_t stream) {
    return forward_prefill_impl(plan, layer, x_bf16, n_tokens, out, ro, scratch, scratch_bytes, nullptr, stream);
}

si_status si_debug_prefill_events(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                  int32_t n_tokens, float *out, si_moe_route_out *ro, void *scratch,
                                  size_t scratch_bytes, void *const *events, si_stream_t stream) {
    return forward_prefill_impl(plan, layer, x_bf16, n_tokens, out, ro, scratch, scratch_bytes,
                                reinterpret_cast<cudaEvent_t const *>(events), stream);
}

int si_debug_plan_info(si_moe_plan_t plan, int32_t *info, int32_t n) {
    if (!plan || !info || n < 1) return -1;
    const int32_t v[6] = {plan->p.sm_count, plan->p.cluster_ok ? 1 : 0, plan->p.cluster_size,
                          plan->p.cluster_active, plan->p.desc.top_k * (plan->p.desc.intermediate / 256),
                          plan->p.smem_optin};
    for (int q = 0; q < n && q < 6; ++q) info[q] = v[q];
    return n < 6 ? n : 6;
}

int si_debug_decode_fused(si_moe_plan_t plan, int32_t n_tokens) {
    if (!plan || n_tokens < 1 || n_tokens > SI_MAX_DECODE_TOKENS) return -1;
    if (n_tokens == 1 && plan->p.cluster_ok) return 2;
    if (n_tokens > 1 && plan->p.cluster_mt_ok) return 3;
    return plan->p.fused_ok[n_tokens] ? 1 : 0;
}

si_status si_moe_read_status(si_moe_plan_t plan, const void *scratch, si_stream_t stream) {
    if (!plan || !scratch) return SI_ERR_INVALID_ARG;
    if (!aligned(scratch, 16)) return SI_ERR_MISALIGNED;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    int32_t word = 0;
    if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    if (word != 0) {
        if (cudaMemset(const_cast<void *>(scratch), 0, sizeof(word)) != cudaSuccess) {
            cudaGetLastError();
            return SI_ERR_CUDA;
        }
        return (si_status)word;
    }
    return SI_OK;
}

si_status si_debug_q4k_dequant(const void *blocks, int64_t n_blocks, float *out_f32,
                               uint16_t *out_bf16, si_stream_t stream) {
    if (!blocks || n_blocks < 0 || (!out_f32 && !out_bf16)) return SI_ERR_INVALID_ARG;
    if (!aligned(blocks, 16) || (out_f32 && !aligned(out_f32, 16)) || (out_bf16 && !aligned(out_bf16, 16)))
        return SI_ERR_MISALIGNED;
    if (si::launch_debug_dequant(static_cast<const uint8_t *>(blocks), n_blocks, out_f32, out_bf16,
                                 (cudaStream_t)stream) != cudaSuccess)
        return SI_ERR_CUDA;
    return SI_OK;
}

si_status si_debug_q4k_dequant_f16(const void *blocks, int64_t n_blocks, const float *gamma, uint16_t *out_f16,
                                   si_stream_t stream) {
    if (!blocks || n_blocks < 0 || !out_f16) return SI_ERR_INVALID_ARG;
    if (!aligned(blocks, 16) || !aligned(out_f16, 16) || (gamma && !aligned(gamma, 16))) return SI_ERR_MISALIGNED;
    if (si::launch_debug_dequant_f16(static_cast<const uint8_t *>(blocks), n_blocks, gamma, out_f16,
                                     (cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    return SI_OK;
}

si_status si_debug_q5k_dequant_f16(const void *blocks, int64_t n_blocks, const float *gamma, uint16_t *out_f16,
                                   si_stream_t stream) {
    if (!blocks || n_blocks < 0 || !out_f16) return SI_ERR_INVALID_ARG;
    if (!aligned(blocks, 16) || !aligned(out_f16, 16) || (gamma && !aligned(gamma, 16))) return SI_ERR_MISALIGNED;
    if (si::launch_debug_q5k_f16(static_cast<const uint8_t *>(blocks), n_blocks, gamma, out_f16,
                                 (cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    return SI_OK;
}

si_status si_debug_nvfp4_dequant_f16(const void *blocks, int64_t n_blocks, float g, uint16_t *out_f16,
                                     si_stream_t stream) {
    if (!blocks || n_blocks < 0 || !out_f16) return SI_ERR_INVALID_ARG;
    if (!aligned(blocks, 16) || !aligned(out_f16, 16)) return SI_ERR_MISALIGNED;
    if (si::launch_debug_nvfp4_f16(static_cast<const uint8_t *>(blocks), n_blocks, g, out_f16, (cudaStream_t)stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    return SI_OK;
}

si_status si_debug_topk(const float *logits, int32_t n, const si_moe_desc *desc,
                        si_moe_route_out *ro, si_stream_t stream) {
    if (!logits || !desc || !ro) return SI_ERR_INVALID_ARG;
    if (n < 1 || n > SI_MAX_DECODE_TOKENS) return SI_ERR_INVALID_ARG;
    if (desc->n_experts < 1 || desc->n_experts > SI_MAX_EXPERTS || desc->top_k < 1 ||
        desc->top_k > desc->n_experts || desc->top_k > SI_MAX_TOPK)
        return SI_ERR_INVALID_ARG;
    if (!aligned(logits, 4)) return SI_ERR_MISALIGNED;
    if (si::launch_debug_topk(logits, n, desc->n_experts, desc->top_k, ro->topk_ids, ro->topk_w,
                              ro->expert_counts, (cudaStream_t)stream) != cudaSuccess)
        return SI_ERR_CUDA;
    return SI_OK;
}

}  // extern "C"
