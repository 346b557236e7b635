// si_expert_cluster.cu -- single-token decode: the selected experts' FFN on
// thread-block clusters, with no grid-wide synchronisation.
//
// sparkinfer README (luciferlive112116), "Layout": kernels/ "fused quantized MoE
// expert FFN", "decode GEMV"; opening section: experts "quantized-resident,
// dequantized on-read, minimizing bytes-per-token"; "Milestone 1": "split-K
// occupancy".
//
// Work unit = (selected expert e = ids[s], 256-wide block column b of its
// intermediate dimension).  One cluster of C CTAs owns a unit:
//   * gate/up: the cluster's CTAs split the unit's 256 intermediate rows; each
//     computes h_r = silu(g_r) * u_r for its rows (activations quantised to
//     int16 per 64-column chunk, dp2a on the 4-bit codes) and writes h_r into
//     the shared memory of every CTA of the cluster (distributed shared memory,
//     asynchronous stores that count their bytes on the receiving CTA's
//     mbarrier);
//   * each CTA waits on its own mbarrier for the unit's 256 h values (cheaper
//     than a release/acquire cluster barrier: measured ~1300 cycles for the
//     stores plus that barrier against ~740 for the asynchronous stores and the
//     local wait);
//   * down: CTA rank c applies Q4_K block b of the down rows
//     [H*c/C, H*(c+1)/C) of expert e to that h slice and adds w_s * y into the
//     output with float reductions (the top-k combine: every output row sums
//     one partial per (slot, block column)).
// The router kernel first sets the output to zero (to x in a pre-normed
// block, whose residual it is).  Weight bytes: gate/up rows by
// 1-D bulk copies, one pair of copies (gate rows, up rows) per group of two
// consumer warps and stage, each group on its own barrier, so that a warp
// starts on its rows as soon as they have landed (the copies are issued in
// group order; waiting for the whole first stage held every warp back by
// about 1.2 us per token); down blocks, 144-byte pieces with a 432-byte row stride,
// by 2-D tensor maps (boxes of 144 bytes x 128 rows, all completing on one
// mbarrier: they are issued after the gate/up rows and land while those are
// computed, and every wait on an mbarrier costs its warp a few hundred
// cycles even when the phase is already complete; the last box of a CTA uses
// a second map whose box height is the remainder).  The barriers'
// transaction counts are posted before the dependency wait, and the producer
// thread reads its unit's expert id and issues every copy right after that
// wait (L2 evict-first).  The kernel lets the next kernel of the stream
// launch at once: that kernel's own dependency wait still covers all of this
// kernel's work.
//
// 2..4 tokens (MT): the same kernel over the distinct experts the tokens
// selected (sparkinfer README, "Milestone 2": redundant weight reads removed).
// A unit is (distinct expert s, block column b), the distinct experts numbered
// in the router's table order (token count descending, then id); its bytes are
// read once and dotted with the x of every
// token that chose expert s (at most 4), and h, the down partials and the
// combine are kept per token.  The router leaves the table of distinct experts
// (expert, tokens, their ranks) and the ranked logits; warp 0 forms the
// routing weights.  Units number U * I/256 (U known only on the device), so
// the grid covers the largest possible count and clusters whose s >= U leave
// at once; the clusters run in waves, with no grid-wide synchronisation.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "si_device.cuh"
#include "si_internal.h"

namespace si {

namespace {
constexpr int kCW = 16;                     // consumer warps (four per SM sub-partition)
constexpr int kClThreads = (kCW + 1) * 32;  // + one producer warp
constexpr int kPairs = 2;                   // gate/up row pairs per warp per stage
constexpr long long kDrain = 4000000000LL;
constexpr int kMaxDownLanes = 8;            // row groups per warp in the down phase: RPC <= 8*kCW*8
constexpr int kBoxRows = 8 * kCW;           // down rows per tensor box = rows of one down iteration
constexpr int kHqTok = 160;                 // words of one token's quantised h: [4][32] + [4][7] (+ pad)
// Copy groups per gate/up stage: the rows of consumer warps [g*kCW/kGrp, (g+1)*kCW/kGrp) arrive by
// their own copies on their own barrier, so each warp starts as soon as its own rows have landed
// (the copies are issued in group order) instead of when the whole stage has.  Measured on the
// layer workload: 9.85 (one barrier per stage), 9.11 (4 groups), 8.68 (8), 9.8 (16) us per token.
constexpr int kGrp = 8;

__device__ __forceinline__ uint4 ld_s128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// Sum of four per-lane partials over a group of GS lanes: on return lane 0 of
// the group holds the total of v0, lane GS/4 of v1, lane GS/2 of v2 and lane
// 3GS/4 of v3.
template <int GS>
__device__ __forceinline__ float quad_sum(float v0, float v1, float v2, float v3, int li) {
    const bool up2 = (li & (GS / 2)) != 0;
    float x = up2 ? v2 : v0, y = up2 ? v3 : v1;
    x += __shfl_xor_sync(0xffffffffu, up2 ? v0 : v2, GS / 2);
    y += __shfl_xor_sync(0xffffffffu, up2 ? v1 : v3, GS / 2);
    const bool up1 = (li & (GS / 4)) != 0;
    float v = up1 ? y : x;
    v += __shfl_xor_sync(0xffffffffu, up1 ? x : y, GS / 4);
#pragma unroll
    for (int off = GS / 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Sum of (g, u) over a group of GS lanes; lane 0 of the group gets the g total,
// lane GS/2 the u total.
template <int GS>
__device__ __forceinline__ float pair_sum(float g, float u, int li) {
    const bool up = (li & (GS / 2)) != 0;
    float v = up ? u : g;
    v += __shfl_xor_sync(0xffffffffu, up ? g : u, GS / 2);
#pragma unroll
    for (int off = GS / 4; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}
}  // namespace

// NVFP4 (WF = 1) instead of Q4_K (WF = 0) weights: the same data movement
// (144-byte super-blocks), a different chunk dot product (si_device.cuh), the
// activations' 16-column integer sums next to their scale, and the matrices'
// tensor scales on the gate and up partials and on the combine weight.
// WF = 2: Q4_K weights in the int8-activation mode (SI_FLAG_ACT_INT8): x (from
// the router) and h are int8 per 32 columns, dotted with dp4a.
// WF = 3: Q5_K weights (176-byte super-blocks: the fifth code bit of every
// weight in 32 qh bytes ahead of the Q4_K-style codes), int16 activations.
template <int NBH, bool NORM, int WF, bool MT>
__global__ void __launch_bounds__(kClThreads, 1)
    k_expert_cluster(const __grid_constant__ CUtensorMap tmap_down, const __grid_constant__ CUtensorMap tmap_tail,
                     DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t sm[];
    constexpr int GS = 4 * NBH;
    constexpr int RPW = 32 / GS;
    constexpr int CH = kCW * RPW * kPairs;  // row pairs per stage
    constexpr bool FP4 = WF == 1, A8 = WF == 2, Q5 = WF == 3;
    constexpr int BB = Q5 ? kQ5BlockBytes : kBlockBytes;  // bytes per super-block
    constexpr int QO = Q5 ? kQ5QsOff : 16;                // offset of the codes in a block
    constexpr int rowg = NBH * BB;
    constexpr int stageA = 2 * CH * rowg;
    __shared__ int s_err;
    __shared__ float s_w;
    __shared__ int s_lastA[8];
    __shared__ int s_lastB;
    __shared__ int s_tok[SI_MAX_DECODE_TOKENS];    // MT: the unit's tokens
    __shared__ float s_wt[SI_MAX_DECODE_TOKENS];   // MT: their routing weights for expert s
    static_assert(!MT || (WF != 2 && !NORM), "the multi-token units take plain Q4_K, NVFP4 or Q5_K blocks");
    // the next kernel's dependency wait still covers this whole grid; MT: see below
    if (!MT) pdl_launch_dependents();

    // parameters used after the dependency wait, read now
    const uint8_t *const wg = pin_ptr(a.wg), *const wu = pin_ptr(a.wu);
    const int32_t *const ids = pin_ptr(a.ids);
    const float *const zsel = pin_ptr(a.wts);  // the selected logits in rank order (see below)
    float *const o_w = pin_ptr(a.o_w);
    const int k = pin_i32(a.k);
    float *const out_g = pin_ptr(a.out);
    int32_t *const ctrl = pin_ptr(a.ctrl);
    const long long budget = (long long)pin_u64((uint64_t)a.wait_budget);
    const int fault_wait = pin_i32(a.fault_wait);
    const int I = pin_i32(a.I), H = pin_i32(a.H);
    const float *const wsc = FP4 ? pin_ptr(a.wscale) : nullptr;  // NVFP4 tensor scales [E][3]
    const uint32_t *const xq_g = pin_ptr(a.xq);  // x quantised by the router (plain block)
    const int n_tok = MT ? pin_i32(a.n) : 1;
    const UniqTable *const uniq = MT ? pin_ptr(a.uniq) : nullptr;
    const int cl_active = MT ? pin_i32(a.cl_active) : 0;
    const int ystride = MT ? pin_i32(a.cl_ystride) : 0;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = (int)cluster_nctarank();
    const int rank = (int)cluster_ctarank();
    const int nbI = I / kQK;
    const int unit = blockIdx.x / C;
    // slot: the top-k slot of the single token, or (MT) the index of the distinct expert
    const int slot = unit / nbI, bcol = unit - slot * nbI;
    const int r_lo = kQK * bcol + (kQK * rank) / C;
    const int n_rp = kQK * bcol + (kQK * (rank + 1)) / C - r_lo;
    const int c_lo = (H * rank) / C;
    const int n_rows = (H * (rank + 1)) / C - c_lo;
    const int nA = (n_rp + CH - 1) / CH;
    const int NSA = pin_i32(a.cl_nsa);
    const int box_stride = pin_i32(a.cl_box_stride), nbox = pin_i32(a.cl_nbox), tail_rows = pin_i32(a.cl_tail_rows);

    uint8_t *stA = sm + pin_i32(a.cl_off_a);
    uint8_t *stB = sm + pin_i32(a.cl_off_b);
    float *hslice = reinterpret_cast<float *>(sm + pin_i32(a.cl_off_h));  // [256] h of the unit
    float *ybuf = reinterpret_cast<float *>(sm + pin_i32(a.cl_off_y));    // [rows] down partials
    uint32_t *const xq_s = reinterpret_cast<uint32_t *>(sm + pin_i32(a.cl_off_x));  // quantised x, later h
    const uint32_t fullA = smem_addr(sm + pin_i32(a.cl_off_bar));  // [NSA][kGrp]
    const uint32_t emptyA = fullA + 8 * NSA * kGrp;
    const uint32_t fullB = emptyA + 8 * NSA;  // all down boxes complete on this one barrier
    const uint32_t hbar = fullB + 8;          // the unit's 256 h values, stored by every CTA of the cluster
    const uint32_t xbar = hbar + 8;           // the router's quantised x (plain block)
    const uint32_t xq_bytes = (uint32_t)(H / 64) * (A8 ? kXq8Words : kXqWords) * 4;
    int32_t *status = ctrl + kCtrlStatus;
    constexpr int CG = CH / kGrp;  // row pairs per copy group
    static_assert(CH % kGrp == 0 && kCW % kGrp == 0, "copy groups split the stage and the warps evenly");
    // row pairs of copy group g in stage j (0 past the stage's last pair)
    auto grp_pairs = [&](int j, int g) { return max(0, min(CG * (g + 1), min(CH, n_rp - CH * j)) - CG * g); };

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmap_down);  // descriptor fetches off the critical path
        prefetch_tensormap(&tmap_tail);
        for (int st = 0; st < NSA; ++st) {
            for (int g = 0; g < kGrp; ++g) mbar_init(fullA + 8 * (st * kGrp + g), 1);
            mbar_init(emptyA + 8 * st, kCW);
            s_lastA[st] = -1;
        }
        mbar_init(fullB, 1);
        mbar_init(hbar, 1);
        mbar_init(xbar, 1);
        s_lastB = -1;
        s_err = 0;
        fence_mbar_init();
        // the byte counts of the first ring pass and of every down box do not
        // depend on the routing: post them now (the producer's arrival)
        for (int j = 0; j < min(nA, NSA); ++j)
            for (int g = 0; g < kGrp; ++g)  // an empty group's barrier completes here
                mbar_arrive_expect_tx(fullA + 8 * (j * kGrp + g), (uint32_t)(2 * grp_pairs(j, g) * rowg));
        // the bytes the box copies deliver: the last box is tail_rows high for every
        // CTA (the largest CTA's remainder), which may exceed this CTA's n_rows
        mbar_arrive_expect_tx(fullB, (uint32_t)(((nbox - 1) * kBoxRows + tail_rows) * BB));
        if (!MT) {  // MT: the counts depend on the routing, posted by the producer after the wait
            mbar_arrive_expect_tx(hbar, (uint32_t)(kQK * 4));  // every h value of the unit, once
            if (!NORM) mbar_arrive_expect_tx(xbar, xq_bytes);
        }
    }
    // A plain block reads x quantised by the router (after the dependency wait, in
    // the consumer warps), so this kernel may be launched before the router has
    // read x.  A pre-normed block quantises x * gamma / rms(x) here, before the
    // dependency wait (the router launches it only after its own wait on the
    // producers of x, so x is final): warp 0 quantises the token's H/64 chunks
    // into shared memory, each a row of 32 words whose 16-byte unit q is stored
    // at unit q ^ (row & 7), so that the lanes that load different rows into
    // registers hit different banks; the norm gain is staged in the (still idle)
    // gate/up stages while warp 0's loads of x are in flight (lanes 0..H/64-1
    // hold all of x).
    const bool xq_lane = NORM && warp == 0 && lane < H / 64;
    uint4 xr[8];
    if (xq_lane) {
        const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + 64 * lane);
#pragma unroll
        for (int q = 0; q < 8; ++q) xr[q] = __ldg(xp + q);
    }
    float4 *const gam_s = reinterpret_cast<float4 *>(stA);  // [H/4]
    if (NORM) {
        for (int i = threadIdx.x; i < H / 4; i += blockDim.x)
            gam_s[i] = __ldg(reinterpret_cast<const float4 *>(a.norm_w) + i);
        __syncthreads();
    }
    if (xq_lane) {
        uint32_t *xq = xq_s;                                   // [H/64][32] words, 16-byte units swizzled
        float *xqf = reinterpret_cast<float *>(xq + H / 2);   // [H/64][7]: scale, Xa, Xb, 4 x 16-column int sums
        float xf[64];
        uint32_t wq[32];
        float sa, sb;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t wv[4] = {xr[q].x, xr[q].y, xr[q].z, xr[q].w};
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                xf[8 * q + 2 * e2] = __uint_as_float(wv[e2] << 16);
                xf[8 * q + 2 * e2 + 1] = __uint_as_float(wv[e2] & 0xffff0000u);
            }
        }
        if (NORM) {
            float ss = 0.f;
#pragma unroll
            for (int q = 0; q < 64; ++q) ss = fmaf(xf[q], xf[q], ss);
            const unsigned mask = H / 64 == 32 ? 0xffffffffu : (1u << (H / 64)) - 1u;
            for (int o = 1; o < H / 64; o <<= 1) ss += __shfl_xor_sync(mask, ss, o);
            const float r = rms_scale(ss, H, a.norm_eps);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 g = gam_s[16 * lane + q];
                xf[4 * q] *= r * g.x;
                xf[4 * q + 1] *= r * g.y;
                xf[4 * q + 2] *= r * g.z;
                xf[4 * q + 3] *= r * g.w;
            }
        }
        const float sc = quantize64(xf, wq, sa, sb);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            reinterpret_cast<uint4 *>(xq + 32 * lane)[q ^ (lane & 7)] =
                make_uint4(wq[4 * q], wq[4 * q + 1], wq[4 * q + 2], wq[4 * q + 3]);
        xqf[7 * lane] = sc;
        xqf[7 * lane + 1] = sa;
        xqf[7 * lane + 2] = sb;
        if (FP4) {
            int XQ[4];
            xq_block_sums(wq, XQ);
#pragma unroll
            for (int b4 = 0; b4 < 4; ++b4) reinterpret_cast<int *>(xqf)[7 * lane + 3 + b4] = XQ[b4];
        }
    }
    // the gate/up stages are written by the copy engine later: order the staging's
    // shared-memory accesses before those asynchronous writes
    if (NORM) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    // peers store into hbar's CTA only after every CTA's barriers are initialised:
    // arrive now (thread 0's init fence is the release), wait before the first store
    cluster_arrive_relaxed();
    pdl_wait();  // routing of this token is complete
    // MT: units past the table of distinct experts have nothing to do (the whole
    // cluster leaves: no copy was issued, no peer stores into it).  The clusters of the
    // last wave let the next kernel launch; the others count as having let it at exit.
    // The unit's table entry is read together with U (independent loads, one round
    // trip; the table has room for every unit's slot).
    int nt = 1, mt_e = 0;
    int4 mt_tok = make_int4(0, 0, 0, 0);
    if (MT) {
        const int U = ctrl[kCtrlNumUnique];
        const int ntv = uniq->ntok[slot];
        mt_e = uniq->expert[slot];
        mt_tok = *reinterpret_cast<const int4 *>(&uniq->tok[slot][0]);
        if (slot >= U) return;
        nt = ntv;
        if (unit >= U * nbI - cl_active) pdl_launch_dependents();
    }
    auto unit_tok = [&mt_tok](int t) { return t == 0 ? mt_tok.x : t == 1 ? mt_tok.y : t == 2 ? mt_tok.z : mt_tok.w; };
    // The router left the k selected experts in rank order with their logits.
    // Only the producer thread needs this unit's expert id, to address its
    // copies: it reads it itself and issues them at once.  The renormalised
    // weight of rank r, exp(z_r - z_0) / sum_j exp(z_j - z_0) (z_0 the
    // largest), is needed only by the final reductions: warp 0 forms all k
    // meanwhile (CTA 0 reports them); the __syncthreads before the reductions
    // publishes it.
    if (MT) {
        if (warp == 0) {
            // pair p = lane (token p / k, rank p % k): exp(z_p - z_0) / sum over the token's k
            // logits (z_0 its largest, at rank 0); then the weights of the unit's tokens
            const int nk = n_tok * k;
            const float z = lane < nk ? zsel[lane] : 0.f;
            const int4 sl = *reinterpret_cast<const int4 *>(&uniq->slot[slot][0]);
            const int base = (lane / k) * k;
            const float ex = expf(z - __shfl_sync(0xffffffffu, z, base));
            float den = 0.f;
            for (int r = 0; r < k; ++r) den += __shfl_sync(0xffffffffu, ex, base + r);
            const float wp = ex / den;
            if (blockIdx.x == 0 && o_w && lane < nk) o_w[lane] = wp;
            const int my_t = lane < nt ? lane : 0;
            const int tk = unit_tok(my_t);
            const int sr = my_t == 0 ? sl.x : my_t == 1 ? sl.y : my_t == 2 ? sl.z : sl.w;
            const float wt = __shfl_sync(0xffffffffu, wp, tk * k + sr);
            if (lane < nt) {
                s_tok[lane] = tk;
                s_wt[lane] = FP4 ? wt * wsc[3 * mt_e + 2] : wt;  // NVFP4: times the down tensor scale
            }
        }
    } else if (warp == 0) {
        const float zr = lane < k ? zsel[lane] : 0.f;
        const float z0 = __shfl_sync(0xffffffffu, zr, 0);
        const float ex = lane < k ? expf(zr - z0) : 0.f;
        float den = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        const float w = ex / den;
        if (lane == slot) s_w = FP4 ? w * wsc[3 * ids[slot] + 2] : w;  // NVFP4: times the down tensor scale
        if (blockIdx.x == 0 && o_w && lane < k) o_w[lane] = w;
    }
    volatile int *verr = &s_err;

    // --------------------------------------------------------- producer
    if (warp == kCW) {
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            // the router's quantised x first (every consumer warp needs it for stage 0),
            // one copy into this CTA's shared memory
            if (MT) {  // x of each of the unit's tokens, in table order
                mbar_arrive_expect_tx(hbar, (uint32_t)(nt * kQK * 4));
                mbar_arrive_expect_tx(xbar, (uint32_t)nt * xq_bytes);
                for (int t = 0; t < nt; ++t)
                    bulk_g2s(smem_addr(xq_s) + t * xq_bytes, xq_g + (size_t)unit_tok(t) * (xq_bytes / 4), xq_bytes,
                             xbar, l2_evict_last_policy());
            } else if (!NORM) {
                bulk_g2s(smem_addr(xq_s), xq_g, xq_bytes, xbar, l2_evict_last_policy());
            }
            const int e = MT ? mt_e : ids[slot];
            auto issueA = [&](int j) -> bool {
                const int st = j % NSA;
                if (j >= NSA) {
                    const uint32_t par = ((j / NSA) - 1) & 1;
                    const long long t0 = clock64();
                    while (!mbar_try_wait(emptyA + 8 * st, par)) {
                        if (*verr || clock64() - t0 > budget) {
                            if (!*verr) set_status(status, SI_ERR_TIMEOUT);
                            *verr = 1;
                            return false;
                        }
                        __nanosleep(20);
                    }
                    for (int g = 0; g < kGrp; ++g)  // later passes: posted here
                        mbar_arrive_expect_tx(fullA + 8 * (st * kGrp + g), (uint32_t)(2 * grp_pairs(j, g) * rowg));
                }
                const int cnt = min(CH, n_rp - CH * j);  // the stage's pairs: gate rows, then as many up rows
                const uint32_t dst = smem_addr(stA + (size_t)st * stageA);
                for (int g = 0; g < kGrp; ++g) {
                    const int pg = grp_pairs(j, g);
                    if (pg == 0) break;
                    const size_t src = ((size_t)e * I + r_lo + CH * j + CG * g) * rowg;
                    const uint32_t bar = fullA + 8 * (st * kGrp + g);
                    bulk_g2s(dst + CG * g * rowg, wg + src, (uint32_t)(pg * rowg), bar, pol);
                    bulk_g2s(dst + (cnt + CG * g) * rowg, wu + src, (uint32_t)(pg * rowg), bar, pol);
                }
                s_lastA[st] = (j / NSA) & 1;
                return true;
            };
            const int first = min(nA, NSA);
            for (int j = 0; j < first; ++j) issueA(j);
            // down blocks of this CTA's rows: boxes of 128 rows x 144 bytes, the last one
            // tail_rows high (its own map); each box completes its own barrier
            for (int bx = 0; bx < nbox; ++bx)
                tma_load_2d(smem_addr(stB + (size_t)bx * box_stride), bx == nbox - 1 ? &tmap_tail : &tmap_down,
                            BB * bcol, e * H + c_lo + bx * kBoxRows, fullB, pol);
            s_lastB = 0;
            for (int j = first; j < nA; ++j)
                if (!issueA(j)) break;
        }
        __syncwarp();
        cluster_wait();
    }

    // --------------------------------------------------------- gate/up
    if (warp < kCW) {
        const int g = lane / GS, li = lane % GS, b = li >> 2, i = li & 3;
        const int chunk = 4 * b + i;
        uint32_t xw[32];
        float xs, Xa, Xb;
        int XQ[4];
        if (NORM) {  // quantised in the prologue
            const uint32_t *xq = xq_s;
            const float *xqf = reinterpret_cast<const float *>(xq + H / 2);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 v = reinterpret_cast<const uint4 *>(xq + 32 * chunk)[q ^ (chunk & 7)];
                xw[4 * q] = v.x, xw[4 * q + 1] = v.y, xw[4 * q + 2] = v.z, xw[4 * q + 3] = v.w;
            }
            xs = xqf[7 * chunk], Xa = xqf[7 * chunk + 1], Xb = xqf[7 * chunk + 2];
#pragma unroll
            for (int b4 = 0; b4 < 4; ++b4) XQ[b4] = FP4 ? reinterpret_cast<const int *>(xqf)[7 * chunk + 3 + b4] : 0;
        } else if (A8) {  // int8 per 32 columns, quantised by the router, copied by the producer
            if (!mbar_wait_warp(xbar, 0, budget)) {
                set_status(status, SI_ERR_TIMEOUT);
                *verr = 1;
            }
            const uint8_t *xq8 = reinterpret_cast<const uint8_t *>(xq_s);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 v = *reinterpret_cast<const uint4 *>(xq8 + xq8_unit_byte(chunk, q));
                xw[4 * q] = v.x, xw[4 * q + 1] = v.y, xw[4 * q + 2] = v.z, xw[4 * q + 3] = v.w;
            }
            const float4 f = reinterpret_cast<const float4 *>(xq_s + 16 * (H / 64))[chunk];
            xs = f.x, XQ[0] = __float_as_int(f.y), Xa = f.z, Xb = f.w;  // da, db (bits), the two sums
            XQ[1] = XQ[2] = XQ[3] = 0;
        }
        // quantised by the router, copied by the producer (MT: token t of the unit at t * xq_bytes)
        auto load_x = [&](int t) {
            const uint32_t *xq = xq_s + (size_t)t * (xq_bytes / 4);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 v = reinterpret_cast<const uint4 *>(xq + 32 * chunk)[q ^ (chunk & 7)];
                xw[4 * q] = v.x, xw[4 * q + 1] = v.y, xw[4 * q + 2] = v.z, xw[4 * q + 3] = v.w;
            }
            const uint4 f = reinterpret_cast<const uint4 *>(xq + H / 2 + 8 * chunk)[0];
            const uint4 f2 = reinterpret_cast<const uint4 *>(xq + H / 2 + 8 * chunk)[1];
            xs = __uint_as_float(f.x), Xa = __uint_as_float(f.y), Xb = __uint_as_float(f.z);
            XQ[0] = (int)f.w, XQ[1] = (int)f2.x, XQ[2] = (int)f2.y, XQ[3] = (int)f2.z;
        };
        if (!NORM && !A8) {
            if (!mbar_wait_warp(xbar, 0, budget)) {
                set_status(status, SI_ERR_TIMEOUT);
                *verr = 1;
            }
            load_x(0);
        }
        auto xwf = [&xw](int p) { return xw[p]; };
        // NVFP4: this unit's expert's gate and up tensor scales
        float tsg = 1.f, tsu = 1.f;
        if (FP4) {
            const int eu = MT ? mt_e : ids[slot];
            tsg = wsc[3 * eu];
            tsu = wsc[3 * eu + 1];
        }
        if (fault_wait) {
            const bool got = wait_flag_bounded(ctrl + kCtrlFaultFlag, budget);
            if (!__all_sync(0xffffffffu, got)) {
                set_status(status, SI_ERR_TIMEOUT);
                *verr = 1;
            }
        }
        cluster_wait();  // every CTA of the cluster has initialised its barriers
        // Every stage is visited and every h value is stored, also after an error
        // (zeros then), so that every CTA's h barrier completes and no CTA exits
        // while a peer may still store into it.  MT: the stages stay resident (no
        // ring reuse), and each of the unit's tokens passes over them in turn.
        for (int t = 0; t < (MT ? nt : 1); ++t) {
        if (MT && t > 0) load_x(t);
        for (int j = 0; j < nA; ++j) {
            const int st = j % NSA;
            bool ok = !__any_sync(0xffffffffu, *verr != 0);
            if (ok && (!MT || t == 0) &&
                !mbar_wait_warp(fullA + 8 * (st * kGrp + warp / (kCW / kGrp)), (j / NSA) & 1, budget)) {
                set_status(status, SI_ERR_TIMEOUT);
                *verr = 1;
                ok = false;
            }
            const uint8_t *stage = stA + (size_t)st * stageA;
            const int cnt = min(CH, n_rp - CH * j);  // row pairs of this stage: gate rows, then as many up rows
            float part[2 * kPairs];
#pragma unroll
            for (int m = 0; m < kPairs; ++m) {
                const int ql = (warp * RPW + g) * kPairs + m;  // row pair within the stage
                part[2 * m] = part[2 * m + 1] = 0.f;
                // a partly filled stage: skip the empty slots (per row group; the last stage
                // holds only its own rows, so nothing may be read past them)
                if (ok && CH * j + ql < n_rp) {
                    const uint8_t *grow = stage + ql * rowg + b * BB;
                    const uint8_t *urow = grow + cnt * rowg;
                    const uint4 hg = ld_s128(grow), qg0 = ld_s128(grow + QO + 32 * i), qg1 = ld_s128(grow + QO + 16 + 32 * i);
                    const uint4 hu = ld_s128(urow), qu0 = ld_s128(urow + QO + 32 * i), qu1 = ld_s128(urow + QO + 16 + 32 * i);
                    if (Q5) {
                        const uint4 hg0 = ld_s128(grow + kQ5QhOff), hg1 = ld_s128(grow + kQ5QhOff + 16);
                        const uint4 hu0 = ld_s128(urow + kQ5QhOff), hu1 = ld_s128(urow + kQ5QhOff + 16);
                        part[2 * m] = chunk_contrib_i(chunk_scales_i(hg, i), chunk_isums5(qg0, qg1, hg0, hg1, i, xwf), xs, Xa, Xb);
                        part[2 * m + 1] = chunk_contrib_i(chunk_scales_i(hu, i), chunk_isums5(qu0, qu1, hu0, hu1, i, xwf), xs, Xa, Xb);
                    } else if (FP4) {
                        part[2 * m] = tsg * chunk_contrib_nvfp4(hg, i, qg0, qg1, xwf, xs, XQ);
                        part[2 * m + 1] = tsu * chunk_contrib_nvfp4(hu, i, qu0, qu1, xwf, xs, XQ);
                    } else if (A8) {
                        const float db = __int_as_float(XQ[0]);
                        part[2 * m] = chunk_contrib_i8(chunk_scales_i(hg, i), chunk_isums8(qg0, qg1, xwf), xs, db, Xa, Xb);
                        part[2 * m + 1] = chunk_contrib_i8(chunk_scales_i(hu, i), chunk_isums8(qu0, qu1, xwf), xs, db, Xa, Xb);
                    } else {
                        part[2 * m] = chunk_contrib_i(chunk_scales_i(hg, i), chunk_isums(qg0, qg1, xwf), xs, Xa, Xb);
                        part[2 * m + 1] = chunk_contrib_i(chunk_scales_i(hu, i), chunk_isums(qu0, qu1, xwf), xs, Xa, Xb);
                    }
                }
            }
            // totals: g0 at group lane 0, u0 at GS/4, g1 at GS/2, u1 at 3GS/4
            const float tot = quad_sum<GS>(part[0], part[1], part[2], part[3], li);
            const float uu = __shfl_down_sync(0xffffffffu, tot, GS / 4);
            float hv = silu(tot) * uu;  // meaningful in group lanes 0 (pair 0) and GS/2 (pair 1)
            // lanes 0..C-1 of the group each store one pair's h into one peer (parallel pushes)
#pragma unroll
            for (int m = 0; m < kPairs; ++m) {
                const float hm = __shfl_sync(0xffffffffu, hv, (lane - li) + m * (GS / 2));
                const int q = CH * j + (warp * RPW + g) * kPairs + m;
                if (q < n_rp)
                    for (int peer = li; peer < C; peer += GS)  // GS may be smaller than C
                        st_async_cluster_u32(hslice + (kQK * t + r_lo + q - kQK * bcol), hbar, (uint32_t)peer,
                                             __float_as_uint(hm));
            }
            __syncwarp();
            if (lane == 0 && (!MT || t == nt - 1)) mbar_arrive(emptyA + 8 * st);
        }
        }
    }

    // every CTA of the cluster has stored its h rows into this CTA
    if (warp < kCW && !mbar_wait_warp_cluster(hbar, 0, budget)) {
        set_status(status, SI_ERR_TIMEOUT);
        *verr = 1;
    }

    // --------------------------------------------------------- down + combine
    const bool skip = __any_sync(0xffffffffu, *verr != 0);
    // reuse of the x region: per token [4][32] words (the same unit swizzle) + [4][7]
    const int ntl = MT ? nt : 1;
    if (warp < kCW && !skip) {
        uint32_t *hq = xq_s + (MT ? kHqTok * (warp >> 2) : 0);
        float *hqf = reinterpret_cast<float *>(hq + 128);
        const float *hsl = hslice + (MT ? kQK * (warp >> 2) : 0);
        if (A8 && warp < 4) {  // int8 per 32 columns, the layout of the router's x (kXq8Words)
            const float2 v = reinterpret_cast<const float2 *>(hsl + 64 * warp)[lane];  // columns 2l, 2l+1
            float d, sum;
            const uint32_t lo = quant_pair8(v.x, v.y, &d, &sum);
            const uint32_t hi = __shfl_down_sync(0xffffffffu, lo, 1);
            if ((lane & 1) == 0) {
                const int w = lane >> 1;
                reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(hq) + xq8_unit_byte(warp, w >> 2))[w & 3] =
                    lo | (hi << 16);
            }
            float *sc = reinterpret_cast<float *>(hq + 16 * 4) + 4 * warp;
            if (lane == 0) sc[0] = d, sc[2] = sum;
            if (lane == 16) sc[1] = d, sc[3] = sum;
        } else if (warp < 4 * ntl) {  // the unit's four 64-column chunks of h: warp 4t+c quantises chunk c of token t
            const int wc = MT ? (warp & 3) : warp;
            const float2 v = reinterpret_cast<const float2 *>(hsl + 64 * wc)[lane];  // columns 2l, 2l+1
            float mx = fmaxf(fabsf(v.x), fabsf(v.y));
            float sum = v.x + v.y;  // lanes 0..15: sub-block a, 16..31: sub-block b
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            const float inv = mx > 0.f ? 32767.0f / mx : 0.f;
            hq[32 * wc + 4 * ((lane >> 2) ^ wc) + (lane & 3)] = pack_q16(v.x, v.y, inv);
            if (lane == 0) {
                hqf[7 * wc] = mx * (1.0f / 32767.0f);
                hqf[7 * wc + 1] = sum;
            }
            if (lane == 16) hqf[7 * wc + 2] = sum;
            if (FP4) {  // integer sums of the quantised h over 16-column blocks (8 lanes each)
                const uint32_t wq2 = pack_q16(v.x, v.y, inv);
                int s2 = (int)(int16_t)(wq2 & 0xffffu) + ((int)wq2 >> 16);
                s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
                s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
                s2 += __shfl_xor_sync(0xffffffffu, s2, 4);
                if ((lane & 7) == 0) reinterpret_cast<int *>(hqf)[7 * wc + 3 + (lane >> 3)] = s2;
            }
        }
    }
    if (warp < kCW) asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");  // consumer warps only
    if (warp < kCW && !skip) {
        const int r8 = lane >> 2, i = lane & 3;
        // box m holds rows [128m, 128m + 128) = the rows of iteration m; every box
        // completes on one barrier (they land while gate/up is computed), rows past
        // n_rows are skipped
        const bool landed = mbar_wait_warp(fullB, 0, budget);
        if (!landed) {
            set_status(status, SI_ERR_TIMEOUT);
            *verr = 1;
        }
        for (int t = 0; t < (landed ? ntl : 0); ++t) {  // MT: each of the unit's tokens in turn
            const uint32_t *hq = xq_s + (MT ? kHqTok * t : 0);
            const float *hqf = reinterpret_cast<const float *>(hq + 128);
            uint32_t hw[32];
            float hs, Ha, Hb, hdb = 0.f;
            int HQ[4];
            if (A8) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(hq) + xq8_unit_byte(i, q));
                    hw[4 * q] = v.x, hw[4 * q + 1] = v.y, hw[4 * q + 2] = v.z, hw[4 * q + 3] = v.w;
                }
                const float4 f = reinterpret_cast<const float4 *>(hq + 16 * 4)[i];
                hs = f.x, hdb = f.y, Ha = f.z, Hb = f.w;
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 v = reinterpret_cast<const uint4 *>(hq + 32 * i)[q ^ i];
                    hw[4 * q] = v.x, hw[4 * q + 1] = v.y, hw[4 * q + 2] = v.z, hw[4 * q + 3] = v.w;
                }
                hs = hqf[7 * i], Ha = hqf[7 * i + 1], Hb = hqf[7 * i + 2];
            }
#pragma unroll
            for (int b4 = 0; b4 < 4; ++b4) HQ[b4] = FP4 ? reinterpret_cast<const int *>(hqf)[7 * i + 3 + b4] : 0;
            auto hwf = [&hw](int p) { return hw[p]; };
            float *yb = ybuf + (MT ? ystride * t : 0);
#pragma unroll 1
            for (int m = 0; m < nbox; ++m) {
                const int lr = kBoxRows * m + 8 * warp + r8;
                float v = 0.f;
                if (lr < n_rows) {
                    const uint8_t *blk = stB + (size_t)m * box_stride + (size_t)(8 * warp + r8) * BB;
                    const uint4 hd = ld_s128(blk), q0 = ld_s128(blk + QO + 32 * i), q1 = ld_s128(blk + QO + 16 + 32 * i);
                    uint4 qh0 = make_uint4(0, 0, 0, 0), qh1 = qh0;
                    if (Q5) qh0 = ld_s128(blk + kQ5QhOff), qh1 = ld_s128(blk + kQ5QhOff + 16);
                    v = Q5   ? chunk_contrib_i(chunk_scales_i(hd, i), chunk_isums5(q0, q1, qh0, qh1, i, hwf), hs, Ha, Hb)
                        : FP4 ? chunk_contrib_nvfp4(hd, i, q0, q1, hwf, hs, HQ)
                        : A8 ? chunk_contrib_i8(chunk_scales_i(hd, i), chunk_isums8(q0, q1, hwf), hs, hdb, Ha, Hb)
                             : chunk_contrib_i(chunk_scales_i(hd, i), chunk_isums(q0, q1, hwf), hs, Ha, Hb);
                }
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                if (i == 0 && lr < n_rows) yb[lr] = v;
            }
        }
    }
    __syncthreads();
    if (!*verr) {
        if (MT) {  // each token's partials, weighted by its routing weight for this expert
            for (int idx = threadIdx.x; idx < ntl * n_rows; idx += blockDim.x) {
                const int t = idx / n_rows, lr = idx - t * n_rows;
                red_add_f32(out_g + (size_t)s_tok[t] * H + c_lo + lr, s_wt[t] * ybuf[ystride * t + lr]);
            }
        } else {
            const float w = s_w;
            float *out = out_g + c_lo;
            for (int lr = threadIdx.x; lr < n_rows; lr += blockDim.x) red_add_f32(out + lr, w * ybuf[lr]);
        }
    } else if (threadIdx.x == 0) {  // no copy may still be writing this CTA's shared memory at exit
        for (int st = 0; st < NSA; ++st)
            if (s_lastA[st] >= 0)
                for (int g = 0; g < kGrp; ++g) mbar_wait_bounded(fullA + 8 * (st * kGrp + g), s_lastA[st], kDrain);
        if (s_lastB >= 0) mbar_wait_bounded(fullB, 0, kDrain);
        if (!NORM) mbar_wait_bounded(xbar, 0, kDrain);  // issued by the producer in every case
        // the peers store every h value, also after an error: let them all land here
        // before this CTA's shared memory goes away
        mbar_wait_bounded_cluster(hbar, 0, kDrain);
    }
}

// ------------------------------------------------------------------ host
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// Cluster size and shared-memory plan for n = 1 (nt = 1), or for units of
// up to nt tokens (the multi-token kernel: x, h and the down partials once
// per token, and the gate/up stages without ring reuse); false if this shape
// needs the other expert kernels.
bool expert_cluster_layout(const si_moe_desc &d, int C, int smem_max, DecodeArgs &a, int nt) {
    const int nbh = d.hidden / kQK;
    if (nbh != 1 && nbh != 2 && nbh != 4 && nbh != 8) return false;
    if (C < 2 || C > 8) return false;
    const int CH = kCW * (32 / (4 * nbh)) * kPairs;
    const int BB = d.wtype == SI_WTYPE_Q5_K ? kQ5BlockBytes : kBlockBytes;
    const int rowg = nbh * BB;
    const int stageA = 2 * CH * rowg;
    const int rp_max = (kQK + C - 1) / C;
    const int nA_max = (rp_max + CH - 1) / CH;
    const int rpc = (d.hidden + C - 1) / C;  // down rows per CTA (max)
    if (rpc > kBoxRows * kMaxDownLanes) return false;
    const int nbox = (rpc + kBoxRows - 1) / kBoxRows;
    const int tail = rpc - (nbox - 1) * kBoxRows;  // 1..128 rows in the last box
    const int box_stride = kBoxRows * BB;  // 18432 = 144 * 128 for Q4_K
    auto al = [](int v) { return (v + 127) / 128 * 128; };
    int NSA = nA_max < 3 ? nA_max : 3;
    if (nt > 1 && nA_max > NSA) return false;  // the tokens pass over the resident stages in turn
    int off = 0;
    a.cl_off_a = off;
    // without ring reuse the last stage holds only the rows that remain
    off += nA_max <= NSA ? (NSA - 1) * stageA + 2 * (rp_max - (NSA - 1) * CH) * rowg : NSA * stageA;
    off = al(off);
    a.cl_off_b = off;
    off += (nbox - 1) * box_stride + al(tail * BB);
    a.cl_off_h = off;
    off += nt * al(kQK * 4);
    a.cl_off_x = off;  // quantised x per token: [H/64][32] words + [H/64][8] (later: quantised h)
    off += nt * al(d.hidden / 64 * kXqWords * 4);
    if (nt * kHqTok > nt * (d.hidden / 64) * kXqWords) return false;  // h per token fits where x was
    a.cl_off_y = off;
    a.cl_ystride = al(rpc * 4) / 4;
    off += nt * al(rpc * 4);
    a.cl_off_bar = off;
    off += 8 * (NSA * kGrp + NSA + 3) + 64;
    if (off + 1024 > smem_max) return false;  // + static shared memory
    a.cl_nsa = NSA;
    a.cl_C = C;
    a.cl_tail_rows = tail;
    a.cl_nbox = nbox;
    a.cl_box_stride = box_stride;
    a.cl_smem = off;
    return true;
}

// Down rows of all experts as a 2-D byte tensor [E*H rows][I/256*144 bytes];
// a box is one 144-byte block column of `rows` consecutive rows.
static bool make_down_tensor_map(const DecodeArgs &a, int rows, CUtensorMap *tm) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int nbi = a.I / kQK;
    const int BB = a.wtype == SI_WTYPE_Q5_K ? kQ5BlockBytes : kBlockBytes;
    cuuint64_t dims[2] = {(cuuint64_t)nbi * BB, (cuuint64_t)a.E * a.H};
    cuuint64_t strides[1] = {(cuuint64_t)nbi * BB};
    cuuint32_t box[2] = {(cuuint32_t)BB, (cuuint32_t)rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.wd), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NBH>
static cudaError_t launch_cluster_t(const DecodeArgs &a, const CUtensorMap &tm, const CUtensorMap &tt,
                                    cudaStream_t s) {
    // MT: room for every distinct expert the call can have (at most n*k, at most E)
    const int units = (a.cl_mt ? (a.n * a.k < a.E ? a.n * a.k : a.E) : a.k) * (a.I / kQK);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units * a.cl_C);
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = a.cl_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = a.cl_C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (a.cl_mt) {
        if (a.wtype == SI_WTYPE_NVFP4) return cudaLaunchKernelEx(&cfg, k_expert_cluster<NBH, false, 1, true>, tm, tt, a);
        if (a.wtype == SI_WTYPE_Q5_K) return cudaLaunchKernelEx(&cfg, k_expert_cluster<NBH, false, 3, true>, tm, tt, a);
        return cudaLaunchKernelEx(&cfg, k_expert_cluster<NBH, false, 0, true>, tm, tt, a);
    }
    if (a.wtype == SI_WTYPE_NVFP4) return cudaLaunchKernelEx(&cfg, k_expert_cluster<NBH, false, 1, false>, tm, tt, a);
    if (a.wtype == SI_WTYPE_Q5_K) return cudaLaunchKernelEx(&cfg, k_expert_cluster<NBH, false, 3, false>, tm, tt, a);
    if (a.act8) return cudaLaunchKernelEx(&cfg, k_expert_cluster<NBH, false, 2, false>, tm, tt, a);
    return a.norm_w ? cudaLaunchKernelEx(&cfg, k_expert_cluster<NBH, true, 0, false>, tm, tt, a)
                    : cudaLaunchKernelEx(&cfg, k_expert_cluster<NBH, false, 0, false>, tm, tt, a);
}

cudaError_t launch_expert_cluster(const DecodeArgs &a, cudaStream_t s) {
    CUtensorMap tm, tt;
    if (!make_down_tensor_map(a, kBoxRows, &tm) || !make_down_tensor_map(a, a.cl_tail_rows, &tt))
        return cudaErrorInvalidValue;
    switch (a.H / kQK) {
        case 1: return launch_cluster_t<1>(a, tm, tt, s);
        case 2: return launch_cluster_t<2>(a, tm, tt, s);
        case 4: return launch_cluster_t<4>(a, tm, tt, s);
        default: return launch_cluster_t<8>(a, tm, tt, s);
    }
}

cudaError_t expert_cluster_prepare(int nbh, int smem_max, int smem, int C, int *active_clusters, bool mt) {
    *active_clusters = 0;
    if (!tensor_map_encoder()) return cudaErrorNotSupported;  // down blocks are fetched by a tensor map
    // single token: plain / pre-normed Q4_K, NVFP4, int8 act, Q5_K; mt: the multi-token kernel
    const void *fs[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
#define SI_CL_VARIANTS(B)                                                                              \
    if (mt) {                                                                                          \
        fs[0] = (const void *)k_expert_cluster<B, false, 0, true>;                                     \
        fs[1] = (const void *)k_expert_cluster<B, false, 1, true>;                                     \
        fs[2] = (const void *)k_expert_cluster<B, false, 3, true>;                                     \
    } else {                                                                                           \
        fs[0] = (const void *)k_expert_cluster<B, false, 0, false>;                                    \
        fs[1] = (const void *)k_expert_cluster<B, true, 0, false>;                                     \
        fs[2] = (const void *)k_expert_cluster<B, false, 1, false>;                                    \
        fs[3] = (const void *)k_expert_cluster<B, false, 2, false>;                                    \
        fs[4] = (const void *)k_expert_cluster<B, false, 3, false>;                                    \
    }
    switch (nbh) {
        case 1: SI_CL_VARIANTS(1) break;
        case 2: SI_CL_VARIANTS(2) break;
        case 4: SI_CL_VARIANTS(4) break;
        default: SI_CL_VARIANTS(8) break;
    }
#undef SI_CL_VARIANTS
    int least = 1 << 30;
    for (const void *f : fs) {  // every variant must fit; the smallest resident count counts
        if (!f) continue;
        cudaFuncAttributes fa;
        cudaError_t err = cudaFuncGetAttributes(&fa, f);
        if (err != cudaSuccess) return err;
        const int dyn_max = smem_max - (int)fa.sharedSizeBytes;
        if (smem > dyn_max) return cudaErrorInvalidValue;
        if ((err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max)) != cudaSuccess)
            return err;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C);
        cfg.blockDim = dim3(kClThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if ((err = cudaOccupancyMaxActiveClusters(&n, f, &cfg)) != cudaSuccess) return err;
        least = n < least ? n : least;
    }
    *active_clusters = least;
    return cudaSuccess;
}

}  // namespace si
