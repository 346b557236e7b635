// si_internal.h -- host-side plan, scratch layout and kernel launchers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/si_moe.h"

namespace si {

// Scratch control block (int32 words at the start of every scratch buffer).
enum CtrlWord : int {
    kCtrlStatus = 0,        // first device-side error code (si_status), 0 = none
    kCtrlRouterTicket = 1,  // arrival counter of the router CTAs (self-resetting)
    kCtrlNumUnique = 2,     // distinct experts selected by this decode call
    kCtrlBarCount = 3,      // grid-barrier arrival counter of the fused expert kernel
    kCtrlBarGen = 4,        // grid-barrier generation
    kCtrlFaultFlag = 5,     // never written: the fault-injection wait of the expert kernels waits on it
    kCtrlWords = 64,
};
constexpr size_t kCtrlBytes = kCtrlWords * sizeof(int32_t);
// x quantised per 64-column chunk (NC = H/64 chunks) as one block of 40*NC
// words: first the int16 pairs, chunk c at words 32c.. with its 16-byte unit q
// stored at unit q ^ (c & 7); then 8 words per chunk: the scale, the two
// 32-column sums (fp32 bits), four 16-column integer sums and a pad.
constexpr int kXqWords = 40;
// int8-activation mode: 20*NC words: first the int8 codes, 16 words per chunk,
// chunk c's 16-byte unit q (4 bytes = 4 columns per word) at byte
// 128*(c/2) + 16*((4*(c%2) + q) ^ ((c/2) % 8)); then 4 words per chunk: the
// two 32-column scales and the two 32-column sums (fp32 bits).
constexpr int kXq8Words = 20;
__host__ __device__ constexpr int xq8_unit_byte(int c, int q) { return 128 * (c >> 1) + 16 * ((4 * (c & 1) + q) ^ ((c >> 1) & 7)); }
constexpr int kMaxSlots = SI_MAX_DECODE_TOKENS * SI_MAX_TOPK;  // 64

// Table of the distinct experts of one decode call (all int32).
struct UniqTable {
    int32_t expert[kMaxSlots];                        // ascending expert ids
    int32_t ntok[kMaxSlots];                          // tokens that chose it
    int32_t tok[kMaxSlots][SI_MAX_DECODE_TOKENS];     // which tokens
    int32_t slot[kMaxSlots][SI_MAX_DECODE_TOKENS];    // at which top-k slot
};
static_assert(offsetof(UniqTable, tok) % 16 == 0 && SI_MAX_DECODE_TOKENS == 4,
              "a slot's tokens are read as one 16-byte word");

struct DecodeLayout {
    size_t ctrl, logits, ids, wts, counts, uniq, h, xq, total;
};

struct Plan {
    si_moe_desc desc;
    int device;
    int sm_count;
    int l2_bytes;
    int smem_optin;
    long long wait_budget;  // SM cycles a device-side wait may spin before reporting SI_ERR_TIMEOUT
    bool fault_wait;        // test mode: expert kernels first wait on a flag nothing sets
    bool fused_ok[SI_MAX_DECODE_TOKENS + 1];  // fused expert kernel usable for n tokens
    bool cluster_ok;                          // cluster expert kernel usable for n = 1
    bool cluster_mt_ok;                       // and for 2..4 tokens (units of distinct experts)
    int cluster_mt_size;                      // CTAs per cluster of the multi-token kernel
    int cluster_mt_active;                    // resident clusters of the multi-token kernel
    bool prefill_ok;                          // tensor-core prefill kernels configured
    int cluster_size;                         // CTAs per cluster (all clusters co-resident)
    int cluster_active;                       // clusters of that size the device holds at once
    DecodeLayout dec;  // sized for SI_MAX_DECODE_TOKENS tokens
};

DecodeLayout decode_layout(const si_moe_desc &d, int n_tokens);

// Argument checks of a decode call (everything but the scratch buffer), made
// before any launch.
si_status check_decode_args(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                            int32_t n_tokens, const float *out, const si_moe_route_out *ro);

// Arguments of the decode kernels (device pointers + sizes).
struct DecodeArgs {
    const uint8_t *wg, *wu, *wd;
    const float *router_w, *router_bias;
    const float *norm_w;  // [H] RMSNorm gain of a pre-normed block (out = x + MoE(norm(x))), or null
    float norm_eps;
    int wtype;              // SI_WTYPE_Q4_K or SI_WTYPE_NVFP4
    const float *wscale;    // NVFP4: [E][3] tensor scales of gate, up, down
    const uint16_t *x;  // [n][H] bf16 bits
    float *out;         // [n][H]
    int H, I, E, k, n;
    int32_t *ctrl;
    float *logits;  // [n][E]
    int32_t *ids;   // [n][k]
    float *wts;     // [n][k]
    int32_t *counts;
    UniqTable *uniq;
    float *h;  // [n][k][I]
    uint32_t *xq;  // [n][H/64][kXqWords]: x quantised per 64 columns by the router (cluster paths)
    int32_t *o_ids;
    float *o_w;
    int32_t *o_counts;
    float *o_logits;
    long long wait_budget;
    int fault_wait;  // test mode (SI_FAULT_WAIT_BUDGET set): wait on kCtrlFaultFlag first
    // shared-memory plan of the fused expert kernel (set by expert_fused_layout)
    int fz_off_a, fz_off_b, fz_off_x, fz_off_h, fz_off_hs, fz_off_yw, fz_off_bar;
    int fz_nsa, fz_nsb, fz_rb, fz_stage_b, fz_smem;
    // shared-memory plan of the cluster expert kernel (set by expert_cluster_layout)
    int cl_off_a, cl_off_b, cl_off_h, cl_off_x, cl_off_y, cl_off_bar;
    int cl_nsa, cl_C, cl_tail_rows, cl_nbox, cl_box_stride, cl_smem;
    int cl_ystride;  // floats per token of the down partials
    int cl_mt;       // 2..4 tokens on the cluster kernel: units (distinct expert, block column), in waves
    int cl_active;   // clusters resident at once (MT: the last wave lets the next kernel launch)
    int zero_out;  // router sets out[n][H] to 0, or to x in a pre-normed block (the expert kernel accumulates into it)
    int act8;      // int8-activation mode (SI_FLAG_ACT_INT8) on the single-token cluster path
    int sel_logits;  // single token, cluster expert kernel: the router writes ids in rank order, the
                     // selected logits (not weights) and 0/1 counts; the expert kernel forms the weights
};

// Prefill scratch: routing arrays and the expert-major rows of the two GEMMs.
// Each expert's rows start at a multiple of 32 (padded offsets poff), so the
// 32-row tiles of the GEMM epilogues never reach another expert's rows.
struct PrefillLayout {
    size_t ctrl, wt, logits, ids, wts, counts, hist, offsets, poff, perm, pperm, inv, xp, h, y, rms, rrow, total;
    int64_t rows;  // padded row capacity: T*k + 32*E
};
PrefillLayout prefill_layout(const si_moe_desc &d, int n_tokens);

struct PrefillArgs {
    const uint8_t *wg, *wu, *wd;
    const float *router_w, *router_bias;
    const float *norm_w;  // [H] RMSNorm gain of a pre-normed block (out = x + MoE(norm(x))), or null
    float norm_eps;
    int wtype;              // SI_WTYPE_Q4_K or SI_WTYPE_NVFP4
    const float *wscale;    // NVFP4: [E][3] tensor scales of gate, up, down
    const uint16_t *x;  // [T][H] bf16 bits
    float *out;         // [T][H]
    int H, I, E, k, T;
    int64_t rows;      // padded row capacity of pperm/xp/h/y
    int32_t *ctrl;
    float *wt;         // [H][E] router weights transposed
    float *logits;     // [T][E]
    int32_t *ids;      // [T*k] pair p = t*k + slot
    float *wts;        // [T*k] renormalised routing weights
    int32_t *counts;   // [E]
    int32_t *hist;     // [ceil(T/32)][E] pairs per expert of each 32-token chunk
    float *rms;        // [T] 1 / rms of each token (pre-normed block only)
    float *rrow;       // [rows] 1 / rms of the token of each padded row, 0 on padding (pre-normed block)
    int32_t *offsets;  // [E+1] exclusive scan of counts
    int32_t *poff;     // [E+1] exclusive scan of counts rounded up to 32
    int32_t *perm;     // [T*k] pair ids ordered by expert, then pair id
    int32_t *pperm;    // [rows] pair id of each padded row (-1 = padding)
    int32_t *inv;      // [T*k] padded row of each pair
    uint16_t *xp;      // [rows][H] fp16 bits: x of each padded row's token
    uint16_t *h;       // [rows][I] fp16 bits
    float *y;          // [rows][H] fp32, before the routing weight
    int32_t *o_ids;
    float *o_w;
    int32_t *o_counts, *o_offsets, *o_perm;
    float *o_logits;
    long long wait_budget;
};

cudaError_t launch_prefill(const Plan &p, const PrefillArgs &a, cudaStream_t s,
                           cudaEvent_t const *events = nullptr);
cudaError_t prefill_prepare(const Plan &p);  // kernel attributes (shared memory opt-in)

cudaError_t launch_decode(const Plan &p, const DecodeArgs &a, cudaStream_t s,
                          cudaEvent_t const *events = nullptr);
bool expert_fused_layout(const si_moe_desc &d, int n, int grid, int smem_max, DecodeArgs &a);
cudaError_t launch_expert_fused(const DecodeArgs &a, int grid, cudaStream_t s);
cudaError_t expert_fused_occupancy(int nbh, bool dedup, int smem, int smem_max, int *blocks_per_sm);
bool expert_cluster_layout(const si_moe_desc &d, int C, int smem_max, DecodeArgs &a, int nt = 1);
cudaError_t launch_expert_cluster(const DecodeArgs &a, cudaStream_t s);
bool router_one_shape(int E, int H);  // the column-split router takes this shape
cudaError_t expert_cluster_prepare(int nbh, int smem_max, int smem, int C, int *active_clusters, bool mt = false);
cudaError_t launch_debug_dequant(const uint8_t *blocks, int64_t n_blocks, float *out_f32,
                                 uint16_t *out_bf16, cudaStream_t s);
cudaError_t launch_debug_nvfp4_f16(const uint8_t *blocks, int64_t n_blocks, float g, uint16_t *out, cudaStream_t s);
cudaError_t launch_debug_q5k_f16(const uint8_t *blocks, int64_t n_blocks, const float *gamma, uint16_t *out,
                                 cudaStream_t s);
cudaError_t launch_debug_dequant_f16(const uint8_t *blocks, int64_t n_blocks, const float *gamma, uint16_t *out,
                                     cudaStream_t s);
cudaError_t launch_debug_topk(const float *logits, int n, int E, int k, int32_t *ids, float *w,
                              int32_t *counts, cudaStream_t s);

}  // namespace si
