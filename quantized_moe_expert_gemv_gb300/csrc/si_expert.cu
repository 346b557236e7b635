// si_expert.cu -- fused expert kernel of the decode path: for the experts the
// router selected, dequant-on-read gate/up GEMV + SwiGLU, then the down GEMV
// and the weighted top-k combine, in one launch.
//
// sparkinfer README (luciferlive112116), "Layout": kernels/ "fused quantized MoE
// expert FFN", "decode GEMV"; opening section: experts "quantized-resident,
// dequantized on-read, minimizing bytes-per-token"; "Milestone 1": "split-K
// occupancy" (here: every SM streams a slice of every selected expert).
//
// Launch: one CTA per SM (grid = SM count, all CTAs resident), 8 consumer
// warps + 1 producer warp.  Programmatic dependent launch: the CTAs become
// resident while the router kernel runs and wait on griddepcontrol.wait.
//
//  * Work split.  The U*I (expert, intermediate-row) pairs are cut into G equal
//    contiguous ranges, one per CTA; the H output rows likewise.
//  * Producer warp.  As soon as the routing is known it issues TMA bulk copies
//    (cp.async.bulk, L2 evict-first) of every gate/up row pair of its range
//    into a ring of NSA stages (8 row pairs per stage) and of its down rows of
//    every selected expert into a ring of NSB stages, so the whole slice of
//    the token's expert bytes is in flight at once.
//  * Phase A (consumers).  Lane (block b, chunk i) of a row keeps the 64
//    activations of its columns in registers; each row is a 32-lane dot with
//    the Q4_K chunk code sums of si_device.cuh; h = silu(g) * u goes to the
//    scratch buffer.
//  * Grid barrier (bounded).  All of h exists.
//  * Phase B.  Warp w takes experts w, w+8, ...; its h is staged in shared
//    memory; lane (row r, chunk i) dots the prefetched down rows; results are
//    weighted by the routing weight and summed over the top-k slots in slot
//    order (deterministic, no atomics).
#include <cstdint>

#include "si_device.cuh"
#include "si_internal.h"

namespace si {

constexpr int kConsumerWarps = 8;
constexpr int kExpertThreads = (kConsumerWarps + 1) * 32;
constexpr long long kDrainBudget = 4000000000LL;  // cycles to wait for in-flight copies after an error
constexpr int kMaxDownRowsPerLane = 4;            // rows per CTA <= 32
constexpr int kStaticSmemReserve = 4096;            // static shared memory of k_expert (routing table, flags)
constexpr int kPairsPerWarp = 2;                  // gate/up row pairs per warp per stage
constexpr int kHqStride = 20;                     // words per quantised h sub-block in shared memory (16 + pad)

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// Sum of four per-lane partials (v0..v3) over a group of GS lanes.  On
// return, lane 0 of the group holds the total of v0, lane GS/4 of v1, lane
// GS/2 of v2, lane 3GS/4 of v3.
template <int GS>
__device__ __forceinline__ float group_sum_quad(float v0, float v1, float v2, float v3, int li) {
    const bool up2 = (li & (GS / 2)) != 0;
    float a = up2 ? v2 : v0, b = up2 ? v3 : v1;
    a += __shfl_xor_sync(0xffffffffu, up2 ? v0 : v2, GS / 2);
    b += __shfl_xor_sync(0xffffffffu, up2 ? v1 : v3, GS / 2);
    const bool up1 = (li & (GS / 4)) != 0;
    float v = up1 ? b : a;
    v += __shfl_xor_sync(0xffffffffu, up1 ? a : b, GS / 4);
#pragma unroll
    for (int off = GS / 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Sum of two per-lane partials (g, u) over a group of GS lanes.  Returns the
// g total (first) and the u total (second) in every lane of the group.
template <int GS>
__device__ __forceinline__ float2 group_sum_pair(float g, float u, int li) {
    const bool upper = (li & (GS / 2)) != 0;
    float v = upper ? u : g;
    const float o = upper ? g : u;
    v += __shfl_xor_sync(0xffffffffu, o, GS / 2);
#pragma unroll
    for (int off = GS / 4; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const float other = __shfl_xor_sync(0xffffffffu, v, GS / 2);
    return make_float2(upper ? other : v, upper ? v : other);
}

// Per-token quantised activations in shared memory (deduplicated batches):
// words [n][32][H/64] (word p of every 64-column chunk together, so that the
// lanes of a row, one chunk each, read word p from consecutive banks),
// scales [n][H/64], sub-block sums [n][H/32].
struct XQ {
    const uint32_t *w;
    const float *sc;
    const float *sum;
};

// The call's routing (distinct experts, their tokens/slots, the weights),
// copied once into shared memory: the producer and the consumers read it for
// every copy and row, and a global-memory round trip each time would
// serialise the whole kernel.
struct SmemRoute {
    int U;
    int expert[kMaxSlots];
    int ntok[kMaxSlots];
    int tok[kMaxSlots][SI_MAX_DECODE_TOKENS];
    int slot[kMaxSlots][SI_MAX_DECODE_TOKENS];
    float wts[kMaxSlots];  // [n*k] routing weights by pair id
};

struct ExpertWork {
    int p0, p1;  // row pairs [p0, p1) of the flattened (slot, intermediate row) space
    int c0, nrows;
    int nA, nB;
};

// ---------------------------------------------------------------- producer
template <int NBH>
__device__ void produce_A(const DecodeArgs &a, const SmemRoute &rt, const ExpertWork &wk, int j, uint8_t *stA,
                          uint32_t fullA, uint32_t emptyA, int *lastA, volatile int *s_err, uint64_t pol,
                          bool &ok) {
    constexpr int CH = kConsumerWarps * (32 / (4 * NBH)) * kPairsPerWarp;
    constexpr int rowg = NBH * kBlockBytes;
    constexpr int stage_bytes = 2 * CH * rowg;
    const int NSA = a.fz_nsa;
    const int st = j % NSA;
    if (j >= NSA) {
        const uint32_t parity = ((j / NSA) - 1) & 1;
        const long long t0 = clock64();
        while (!mbar_try_wait(emptyA + 8 * st, parity)) {
            if (*s_err || clock64() - t0 > a.wait_budget) {
                if (!*s_err) set_status(a.ctrl + kCtrlStatus, SI_ERR_TIMEOUT);
                *s_err = 1;
                ok = false;
                return;
            }
            __nanosleep(20);
        }
    }
    const int qa = wk.p0 + CH * j;
    const int qb = min(qa + CH, wk.p1);
    const uint32_t full = fullA + 8 * st;
    mbar_arrive_expect_tx(full, (uint32_t)(2 * (qb - qa) * rowg));
    const uint32_t dst_g = smem_addr(stA + (size_t)st * stage_bytes);
    const uint32_t dst_u = dst_g + CH * rowg;
    for (int p = qa; p < qb;) {
        const int s = p / a.I;
        const int r = p - s * a.I;
        const int run_end = min(qb, (s + 1) * a.I);
        const int n = run_end - p;
        const size_t src_off = ((size_t)rt.expert[s] * a.I + r) * rowg;
        const uint32_t off = (uint32_t)((p - qa) * rowg);
        bulk_g2s(dst_g + off, a.wg + src_off, (uint32_t)(n * rowg), full, pol);
        bulk_g2s(dst_u + off, a.wu + src_off, (uint32_t)(n * rowg), full, pol);
        p = run_end;
    }
    lastA[st] = (j / NSA) & 1;
}

__device__ void produce_B(const DecodeArgs &a, const SmemRoute &rt, const ExpertWork &wk, int s, uint8_t *stB,
                          uint32_t fullB, uint32_t emptyB, int *lastB, volatile int *s_err, uint64_t pol,
                          bool &ok) {
    const int NSB = a.fz_nsb;
    const int st = s % NSB;
    if (s >= NSB) {
        const uint32_t parity = ((s / NSB) - 1) & 1;
        const long long t0 = clock64();
        while (!mbar_try_wait(emptyB + 8 * st, parity)) {
            if (*s_err || clock64() - t0 > a.wait_budget) {
                if (!*s_err) set_status(a.ctrl + kCtrlStatus, SI_ERR_TIMEOUT);
                *s_err = 1;
                ok = false;
                return;
            }
            __nanosleep(20);
        }
    }
    const int rowd = (a.I / kQK) * kBlockBytes;
    const uint32_t bytes = (uint32_t)(wk.nrows * rowd);
    const uint32_t full = fullB + 8 * st;
    mbar_arrive_expect_tx(full, bytes);
    const size_t src_off = ((size_t)rt.expert[s] * a.H + wk.c0) * rowd;
    bulk_g2s(smem_addr(stB + (size_t)st * a.fz_stage_b), a.wd + src_off, bytes, full, pol);
    lastB[st] = (s / NSB) & 1;
}

// ------------------------------------------------------------------ kernel
template <int NBH, bool DEDUP, bool NORM>
__global__ void __launch_bounds__(kExpertThreads, 1) k_expert(DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t sm[];
    constexpr int GS = 4 * NBH;   // lanes per gate/up row
    constexpr int RPW = 32 / GS;  // rows per warp pass
    constexpr int CH = kConsumerWarps * RPW * kPairsPerWarp;  // row pairs per stage
    constexpr int rowg = NBH * kBlockBytes;
    constexpr int stageA_bytes = 2 * CH * rowg;
    __shared__ int s_err;
    __shared__ SmemRoute rt;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NSA = a.fz_nsa, NSB = a.fz_nsb;
    uint8_t *stA = sm + a.fz_off_a;
    uint8_t *stB = sm + a.fz_off_b;
    const uint32_t fullA = smem_addr(sm + a.fz_off_bar);
    const uint32_t emptyA = fullA + 8 * NSA;
    const uint32_t fullB = emptyA + 8 * NSA;
    const uint32_t emptyB = fullB + 8 * NSB;
    int *lastA = reinterpret_cast<int *>(sm + a.fz_off_bar + 16 * (NSA + NSB));
    int *lastB = lastA + NSA;
    // dedup phase B: every pair's h row, bulk-copied into the (then idle) phase-A stages
    const uint32_t hbar = smem_addr(sm + a.fz_off_bar + ((20 * (NSA + NSB) + 7) & ~7));
    const bool hstage = DEDUP && (size_t)a.n * a.k * a.I * sizeof(float) <= (size_t)NSA * stageA_bytes;
    __shared__ int s_hcopy;
    int32_t *status = a.ctrl + kCtrlStatus;

    if (threadIdx.x == 0) {
        for (int st = 0; st < NSA; ++st) {
            mbar_init(fullA + 8 * st, 1);
            mbar_init(emptyA + 8 * st, kConsumerWarps);
            lastA[st] = -1;
        }
        for (int st = 0; st < NSB; ++st) {
            mbar_init(fullB + 8 * st, 1);
            mbar_init(emptyB + 8 * st, 1);
            lastB[st] = -1;
        }
        s_err = 0;
        s_hcopy = 0;
        mbar_init(hbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();  // the router kernel (and everything before it) is complete

    {
        const int *src = reinterpret_cast<const int *>(a.uniq);  // UniqTable: expert, ntok, tok, slot
        for (int q = threadIdx.x; q < kMaxSlots * (2 + 2 * SI_MAX_DECODE_TOKENS); q += blockDim.x) {
            const int v = src[q];
            if (q < kMaxSlots) rt.expert[q] = v;
            else if (q < 2 * kMaxSlots) rt.ntok[q - kMaxSlots] = v;
            else if (q < 2 * kMaxSlots + kMaxSlots * SI_MAX_DECODE_TOKENS)
                (&rt.tok[0][0])[q - 2 * kMaxSlots] = v;
            else
                (&rt.slot[0][0])[q - 2 * kMaxSlots - kMaxSlots * SI_MAX_DECODE_TOKENS] = v;
        }
        for (int q = threadIdx.x; q < a.n * a.k; q += blockDim.x) rt.wts[q] = a.wts[q];
        if (threadIdx.x == 0) rt.U = a.ctrl[kCtrlNumUnique];
    }
    __syncthreads();
    const SmemRoute *u = &rt;
    const int U = rt.U;
    ExpertWork wk;
    {
        const long long P = (long long)U * a.I;
        const int G = gridDim.x, bid = blockIdx.x;
        if (DEDUP) {
            // balance the phase-A dot products: row r of distinct expert s costs ntok[s] of
            // them, so CTA b takes the rows whose cumulative cost falls in its 1/G share
            long long W = 0;
            for (int q = 0; q < U; ++q) W += (long long)rt.ntok[q] * a.I;
            auto row_at = [&](long long target) -> int {  // first row pair whose cost start >= target
                long long acc = 0;
                for (int q = 0; q < U; ++q) {
                    const long long c = (long long)rt.ntok[q] * a.I;
                    if (acc + c > target) {
                        const int nt = rt.ntok[q] > 0 ? rt.ntok[q] : 1;
                        return q * a.I + (int)((target - acc + nt - 1) / nt);
                    }
                    acc += c;
                }
                return (int)P;
            };
            wk.p0 = row_at(W * bid / G);
            wk.p1 = row_at(W * (bid + 1) / G);
        } else {
            wk.p0 = (int)(P * bid / G);
            wk.p1 = (int)(P * (bid + 1) / G);
        }
        wk.c0 = (int)((long long)a.H * bid / G);
        wk.nrows = (int)((long long)a.H * (bid + 1) / G) - wk.c0;
        wk.nA = (wk.p1 - wk.p0 + CH - 1) / CH;
        wk.nB = wk.nrows > 0 ? U : 0;
    }
    bool ok = true;
    volatile int *verr = &s_err;

    // ------------------------------------------------ issue (producer warp)
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            const int first = min(wk.nA, NSA);
            for (int j = 0; j < first; ++j)
                produce_A<NBH>(a, rt, wk, j, stA, fullA, emptyA, lastA, verr, pol, ok);
            for (int s = 0; s < min(wk.nB, NSB); ++s)
                produce_B(a, rt, wk, s, stB, fullB, emptyB, lastB, verr, pol, ok);
            for (int j = first; j < wk.nA && ok; ++j)
                produce_A<NBH>(a, rt, wk, j, stA, fullA, emptyA, lastA, verr, pol, ok);
        }
        __syncwarp();
    }

    // ------------------------------------------------ phase A (consumers)
    if (warp < kConsumerWarps) {
        const int g = lane / GS, li = lane % GS, b = li >> 2, i = li & 3;
        const int chunk = 4 * b + i;  // this lane's 64-column chunk of a gate/up row
        uint32_t xw[32];
        float xs = 0.f, Xa = 0.f, Xb = 0.f;
        XQ xq{};
        if (!DEDUP) {
            float xf[64];
            const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + 64 * chunk);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 v = __ldg(xp + q);
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    xf[8 * q + 2 * e2] = __uint_as_float(wv[e2] << 16);
                    xf[8 * q + 2 * e2 + 1] = __uint_as_float(wv[e2] & 0xffff0000u);
                }
            }
            if (NORM) {  // pre-normed block: the GS lanes of a group hold all H/64 chunks of x
                float ss = 0.f;
#pragma unroll
                for (int q = 0; q < 64; ++q) ss = fmaf(xf[q], xf[q], ss);
#pragma unroll
                for (int o = 1; o < GS; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float r = rms_scale(ss, a.H, a.norm_eps);
                const float4 *gp = reinterpret_cast<const float4 *>(a.norm_w + 64 * chunk);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float4 gv = __ldg(gp + q);
                    xf[4 * q] *= r * gv.x;
                    xf[4 * q + 1] *= r * gv.y;
                    xf[4 * q + 2] *= r * gv.z;
                    xf[4 * q + 3] *= r * gv.w;
                }
            }
            xs = quantize64(xf, xw, Xa, Xb);
        } else {
            uint32_t *xqw = reinterpret_cast<uint32_t *>(sm + a.fz_off_x);  // [n][H/2]
            float *xqs = reinterpret_cast<float *>(xqw + (size_t)a.n * a.H / 2);  // [n][H/64]
            float *xqx = xqs + (size_t)a.n * a.H / 64;                          // [n][H/32]
            __shared__ float s_rms[SI_MAX_DECODE_TOKENS];
            if (NORM) {  // pre-normed block: warp t finds 1 / rms of token t
                if (warp < a.n) {
                    float ss = 0.f;
                    for (int c = 2 * lane; c < a.H; c += 64) {
                        const uint32_t v = __ldg(reinterpret_cast<const uint32_t *>(a.x + (size_t)warp * a.H + c));
                        const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
                        ss = fmaf(lo, lo, ss);
                        ss = fmaf(hi, hi, ss);
                    }
                    ss = warp_sum(ss);
                    if (lane == 0) s_rms[warp] = rms_scale(ss, a.H, a.norm_eps);
                }
                asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
            }
            for (int c = threadIdx.x; c < a.n * a.H / 64; c += kConsumerWarps * 32) {
                const int t = c / (a.H / 64), cc = c - t * (a.H / 64);
                float xf[64];
                uint32_t wq[32];
                const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + 64 * cc);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 v = __ldg(xp + q);
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        xf[8 * q + 2 * e2] = __uint_as_float(wv[e2] << 16);
                        xf[8 * q + 2 * e2 + 1] = __uint_as_float(wv[e2] & 0xffff0000u);
                    }
                }
                if (NORM) {
                    const float r = s_rms[t];
                    const float4 *gp = reinterpret_cast<const float4 *>(a.norm_w + 64 * cc);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float4 gv = __ldg(gp + q);
                        xf[4 * q] *= r * gv.x;
                        xf[4 * q + 1] *= r * gv.y;
                        xf[4 * q + 2] *= r * gv.z;
                        xf[4 * q + 3] *= r * gv.w;
                    }
                }
                float sa, sb;
                xqs[c] = quantize64(xf, wq, sa, sb);
                xqx[2 * c] = sa;
                xqx[2 * c + 1] = sb;
#pragma unroll
                for (int p = 0; p < 32; ++p) xqw[(size_t)t * a.H / 2 + p * (a.H / 64) + cc] = wq[p];
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
            xq = XQ{xqw, xqs, xqx};
        }

        if (a.fault_wait) {
            const bool got = wait_flag_bounded(a.ctrl + kCtrlFaultFlag, a.wait_budget);
            if (!__all_sync(0xffffffffu, got)) {
                set_status(status, SI_ERR_TIMEOUT);
                *verr = 1;
            }
        }
        for (int j = 0; j < wk.nA && !__any_sync(0xffffffffu, *verr != 0); ++j) {
            const int st = j % NSA;
            const bool landed = mbar_wait_bounded(fullA + 8 * st, (j / NSA) & 1, a.wait_budget);
            if (!__all_sync(0xffffffffu, landed)) {  // one decision per warp
                set_status(status, SI_ERR_TIMEOUT);
                *verr = 1;
                break;
            }
            const uint8_t *stage = stA + (size_t)st * stageA_bytes;
            float part[2 * kPairsPerWarp];   // g, u of each of this warp's row pairs
            int rows[kPairsPerWarp];
            bool act[kPairsPerWarp];
#pragma unroll
            for (int m = 0; m < kPairsPerWarp; ++m) {
                const int ql = (warp * RPW + g) * kPairsPerWarp + m;  // row pair within the stage
                const int q = CH * j + ql;
                act[m] = q < wk.p1 - wk.p0;
                rows[m] = wk.p0 + (act[m] ? q : 0);
                const uint8_t *grow = stage + ql * rowg + b * kBlockBytes;
                const uint8_t *urow = grow + CH * rowg;
                const uint4 hg = lds128(grow), qg0 = lds128(grow + 16 + 32 * i), qg1 = lds128(grow + 32 + 32 * i);
                const uint4 hu = lds128(urow), qu0 = lds128(urow + 16 + 32 * i), qu1 = lds128(urow + 32 + 32 * i);
                const ChunkScalesI cg = chunk_scales_i(hg, i), cu = chunk_scales_i(hu, i);
                if (!DEDUP) {
                    auto xwf = [&xw](int p) { return xw[p]; };
                    part[2 * m] = chunk_contrib_i(cg, chunk_isums(qg0, qg1, xwf), xs, Xa, Xb);
                    part[2 * m + 1] = chunk_contrib_i(cu, chunk_isums(qu0, qu1, xwf), xs, Xa, Xb);
                } else {
                    // every token that chose this row's expert; h lands per (token, slot) pair
                    const int p = rows[m];
                    const int s = p / a.I, r = p - s * a.I;
                    const int nt = act[m] ? u->ntok[s] : 0;
                    const int nt_warp = __reduce_max_sync(0xffffffffu, nt);
                    for (int t = 0; t < nt_warp; ++t) {
                        const int tok = t < nt ? u->tok[s][t] : 0;
                        const uint32_t *wrow = xq.w + (size_t)tok * a.H / 2 + chunk;
                        const int cks = a.H / 64;
                        auto xwf = [wrow, cks](int pp) { return wrow[pp * cks]; };
                        const float sc = xq.sc[tok * (a.H / 64) + chunk];
                        const float xa = xq.sum[tok * (a.H / 32) + 2 * chunk];
                        const float xb = xq.sum[tok * (a.H / 32) + 2 * chunk + 1];
                        const float gp = chunk_contrib_i(cg, chunk_isums(qg0, qg1, xwf), sc, xa, xb);
                        const float up = chunk_contrib_i(cu, chunk_isums(qu0, qu1, xwf), sc, xa, xb);
                        const float2 gu = group_sum_pair<GS>(gp, up, li);
                        if (t < nt && li == 0) {
                            const int pair = u->tok[s][t] * a.k + u->slot[s][t];
                            a.h[(size_t)pair * a.I + r] = silu(gu.x) * gu.y;
                        }
                    }
                }
            }
            if (!DEDUP) {
                static_assert(kPairsPerWarp == 2, "reduction below is written for two row pairs");
                const float tot = group_sum_quad<GS>(part[0], part[1], part[2], part[3], li);
                const float other = __shfl_down_sync(0xffffffffu, tot, GS / 4);  // u of the same pair
                const int m = (li == 0) ? 0 : 1;
                if ((li == 0 || li == GS / 2) && act[m]) {
                    const int p = rows[m];
                    const int s = p / a.I, r = p - s * a.I;
                    a.h[(size_t)u->slot[s][0] * a.I + r] = silu(tot) * other;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(emptyA + 8 * st);
        }
    }

    // ------------------------------------------------ all of h exists
    const bool bar_ok = grid_barrier(a.ctrl + kCtrlBarCount, a.ctrl + kCtrlBarGen, status, a.wait_budget);
    pdl_launch_dependents();
    if (!bar_ok) s_err = 1;

    if (warp == kConsumerWarps) {
        if (lane == 0 && !*verr) {
            const uint64_t pol = l2_evict_first_policy();
            if (hstage) {  // h was written by all CTAs with ordinary stores; the copies read it
                asm volatile("fence.proxy.async;" ::: "memory");
                const uint32_t hrow = (uint32_t)(a.I * sizeof(float));
                mbar_arrive_expect_tx(hbar, (uint32_t)(a.n * a.k) * hrow);
                for (int q = 0; q < a.n * a.k; ++q)
                    bulk_g2s(smem_addr(stA) + (uint32_t)q * hrow, a.h + (size_t)q * a.I, hrow, hbar, pol);
                s_hcopy = 1;
            }
            for (int s = NSB; s < wk.nB && ok; ++s)
                produce_B(a, rt, wk, s, stB, fullB, emptyB, lastB, verr, pol, ok);
        }
        __syncwarp();
    }

    // ------------------------------------------------ phase B (down + combine)
    float *yw = reinterpret_cast<float *>(sm + a.fz_off_yw);  // [n*k][RB]
    const int RB = a.fz_rb;
    const bool skip_b = __any_sync(0xffffffffu, *verr != 0);  // read once per warp
    if (warp < kConsumerWarps && !skip_b) {
        const int nbI = a.I / kQK;
        const int rowd = nbI * kBlockBytes;
        const int nsub = a.I / 32;
        // this warp's quantised copy of one h vector: words [I/32][kHqStride] (16 words of a
        // 32-value sub-block, padded so that neighbouring sub-blocks start in other banks),
        // scales [I/64], sums [I/32]
        uint32_t *hq = reinterpret_cast<uint32_t *>(sm + a.fz_off_h) +
                       (size_t)warp * (a.I / 32 * kHqStride + a.I / 64 + a.I / 32);
        float *hsc = reinterpret_cast<float *>(hq + a.I / 32 * kHqStride);
        float *hsum = hsc + a.I / 64;
        const int r8 = lane >> 2, i = lane & 3;
        bool hready = hstage;
        if (hstage && !__all_sync(0xffffffffu, mbar_wait_warp(hbar, 0, a.wait_budget))) {
            set_status(status, SI_ERR_TIMEOUT);
            *verr = 1;
            hready = false;
        }
        // Chunk s lives in stage s % NSB.  Every stage is owned by one warp, which takes that
        // stage's chunks in issue order, so no warp ever waits on a stage phase that is more
        // than one use ahead of the barrier (mbarrier phases are told apart by parity only).
        for (int s = 0; s < wk.nB; ++s) {
            const int st = s % NSB;
            if (st % kConsumerWarps != warp) continue;
            const bool landed = mbar_wait_bounded(fullB + 8 * st, (s / NSB) & 1, a.wait_budget);
            if (!__all_sync(0xffffffffu, landed)) {
                set_status(status, SI_ERR_TIMEOUT);
                *verr = 1;
                break;
            }
            const uint8_t *rows = stB + (size_t)st * a.fz_stage_b;
            const int nt = u->ntok[s];
            for (int jt = 0; jt < nt; ++jt) {
                const int pair = u->tok[s][jt] * a.k + u->slot[s][jt];
                const float wgt = rt.wts[pair];
                // quantise h of this (token, slot): lane = sub-block, partner lane^1 shares the chunk.
                // A lane reads the eight 16-byte units of its 128-byte sub-block starting at unit
                // sb & 7 (hv[4q..4q+3] = unit (q + sb) & 7), so the lanes of a quarter warp hit
                // different banks; the packed words go back to their own positions.
                for (int sb0 = 0; sb0 < nsub; sb0 += 32) {
                    const int sb = sb0 + lane, rot = sb & 7;
                    float hv[32];
                    float mx = 0.f, sum = 0.f;
                    if (sb < nsub) {
                        if (hready) {
                            const float4 *hp = reinterpret_cast<const float4 *>(stA) + ((size_t)pair * a.I + 32 * sb) / 4;
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 v = hp[(q + rot) & 7];
                                hv[4 * q] = v.x, hv[4 * q + 1] = v.y, hv[4 * q + 2] = v.z, hv[4 * q + 3] = v.w;
                            }
                        } else {
                            const float4 *hp = reinterpret_cast<const float4 *>(a.h + (size_t)pair * a.I + 32 * sb);
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 v = __ldcg(hp + ((q + rot) & 7));
                                hv[4 * q] = v.x, hv[4 * q + 1] = v.y, hv[4 * q + 2] = v.z, hv[4 * q + 3] = v.w;
                            }
                        }
                        float m8[8], s8[8];  // balanced trees: short dependency chains
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            m8[q] = fmaxf(fmaxf(fabsf(hv[4 * q]), fabsf(hv[4 * q + 1])),
                                          fmaxf(fabsf(hv[4 * q + 2]), fabsf(hv[4 * q + 3])));
                            s8[q] = (hv[4 * q] + hv[4 * q + 1]) + (hv[4 * q + 2] + hv[4 * q + 3]);
                        }
#pragma unroll
                        for (int w2 = 4; w2 >= 1; w2 >>= 1) {
#pragma unroll
                            for (int q = 0; q < w2; ++q) {
                                m8[q] = fmaxf(m8[q], m8[q + w2]);
                                s8[q] += s8[q + w2];
                            }
                        }
                        mx = m8[0];
                        sum = s8[0];
                    }
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    if (sb < nsub) {
                        const float inv = mx > 0.f ? 32767.0f / mx : 0.f;
#pragma unroll
                        for (int pp = 0; pp < 16; ++pp) {
                            const int lo = __float2int_rn(hv[2 * pp] * inv);
                            const int hi = __float2int_rn(hv[2 * pp + 1] * inv);
                            hq[kHqStride * sb + 2 * (((pp >> 1) + rot) & 7) + (pp & 1)] =
                                (uint32_t)(lo & 0xffff) | ((uint32_t)hi << 16);
                        }
                        hsum[sb] = sum;
                        if ((sb & 1) == 0) hsc[sb >> 1] = mx * (1.0f / 32767.0f);
                    }
                }
                __syncwarp();
                float acc[kMaxDownRowsPerLane] = {0.f, 0.f, 0.f, 0.f};
                for (int bb = 0; bb < nbI; ++bb) {
                    const int c = 4 * bb + i;
                    uint32_t hw[32];  // sub-blocks 2c and 2c+1
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(hq + kHqStride * (2 * c + (q >> 2)) + 4 * (q & 3));
                        hw[4 * q] = v.x, hw[4 * q + 1] = v.y, hw[4 * q + 2] = v.z, hw[4 * q + 3] = v.w;
                    }
                    const float xs = hsc[c], Ha = hsum[2 * c], Hb = hsum[2 * c + 1];
                    auto xwf = [&hw](int p) { return hw[p]; };
#pragma unroll
                    for (int m = 0; m < kMaxDownRowsPerLane; ++m) {
                        const int lr = r8 + 8 * m;
                        if (lr < wk.nrows) {
                            const uint8_t *blk = rows + (size_t)lr * rowd + bb * kBlockBytes;
                            const uint4 hd = lds128(blk), q0 = lds128(blk + 16 + 32 * i),
                                        q1 = lds128(blk + 32 + 32 * i);
                            acc[m] += chunk_contrib_i(chunk_scales_i(hd, i), chunk_isums(q0, q1, xwf), xs, Ha, Hb);
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < kMaxDownRowsPerLane; ++m) {
                    float v = acc[m];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    const int lr = r8 + 8 * m;
                    if (i == 0 && lr < wk.nrows) yw[(size_t)pair * RB + lr] = wgt * v;
                }
                __syncwarp();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(emptyB + 8 * st);
        }
    }
    __syncthreads();

    if (!*verr) {
        for (int idx = threadIdx.x; idx < a.n * wk.nrows; idx += blockDim.x) {
            const int t = idx / wk.nrows, lr = idx - t * wk.nrows;
            float sacc = 0.f;
            for (int slot = 0; slot < a.k; ++slot) sacc += yw[(size_t)(t * a.k + slot) * RB + lr];
            if (NORM) sacc += bf16_bits_to_f32(a.x[(size_t)t * a.H + wk.c0 + lr]);  // the residual
            a.out[(size_t)t * a.H + wk.c0 + lr] = sacc;
        }
    } else if (threadIdx.x == 0) {
        // An error stopped this CTA early: let its copies in flight land before it exits.
        for (int st = 0; st < NSA; ++st)
            if (lastA[st] >= 0) mbar_wait_bounded(fullA + 8 * st, lastA[st], kDrainBudget);
        for (int st = 0; st < NSB; ++st)
            if (lastB[st] >= 0) mbar_wait_bounded(fullB + 8 * st, lastB[st], kDrainBudget);
        if (s_hcopy) mbar_wait_bounded(hbar, 0, kDrainBudget);
    }
}

// ------------------------------------------------------------------ host side
// Shared-memory plan of the fused kernel for n tokens on `grid` CTAs; returns
// false if this shape needs the generic kernels.
bool expert_fused_layout(const si_moe_desc &d, int n, int grid, int smem_max, DecodeArgs &a) {
    const int nbh = d.hidden / kQK;
    if (nbh != 1 && nbh != 2 && nbh != 4 && nbh != 8) return false;
    const int nbi = d.intermediate / kQK;
    const int RB = (d.hidden + grid - 1) / grid;
    if (RB > 8 * kMaxDownRowsPerLane) return false;
    const int umax = n * d.top_k;
    const int CH = kConsumerWarps * (32 / (4 * nbh)) * kPairsPerWarp;
    const size_t stageA = (size_t)2 * CH * nbh * kBlockBytes;
    const size_t stageB = (size_t)RB * nbi * kBlockBytes;
    const long long P = (long long)umax * d.intermediate;
    const int nA_max = (int)(((P + grid - 1) / grid + CH - 1) / CH);
    const bool dedup = n > 1;
    auto al = [](size_t v) { return (v + 127) / 128 * 128; };
    const size_t x_bytes =
        dedup ? al((size_t)n * (d.hidden / 2 + d.hidden / 64 + d.hidden / 32) * 4) : 0;
    const size_t h_bytes =
        al((size_t)kConsumerWarps * (d.intermediate / 32 * kHqStride + d.intermediate / 64 + d.intermediate / 32) * 4);
    const size_t hs_bytes = 0;
    const size_t yw_bytes = al((size_t)umax * RB * 4);
    // deduplicated batches spend their time computing in phase A (one row serves several tokens),
    // so fewer A stages suffice there and the room goes to down-row stages for phase B
    const int nsa_cap = dedup ? 3 : 4;
    int NSA = nA_max < nsa_cap ? (nA_max < 1 ? 1 : nA_max) : nsa_cap;
    const size_t fixed = x_bytes + h_bytes + hs_bytes + yw_bytes;
    auto bar_bytes = [](int nsa, int nsb) { return (size_t)16 * (nsa + nsb) + (size_t)4 * (nsa + nsb) + 64; };
    const long long sA = (long long)stageA, sB = (long long)stageB;
    auto fits = [&](int nsa, int nsb) {
        const long long need = kStaticSmemReserve + (long long)fixed + (long long)nsa * sA + (long long)nsb * sB +
                               (long long)bar_bytes(nsa, nsb) + 128;
        return need <= (long long)smem_max;
    };
    int NSB = 0;
    while (NSB < umax && fits(NSA, NSB + 1)) ++NSB;
    if (NSB < 1) {
        NSA = 2;
        while (NSB < umax && fits(NSA, NSB + 1)) ++NSB;
        if (NSB < 1) return false;
    }
    // phase B: stage st belongs to consumer warp st % kConsumerWarps, so a multiple of the
    // warp count gives every warp the same number of stages (and of experts)
    if (NSB > kConsumerWarps) NSB -= NSB % kConsumerWarps;
    size_t off = 0;
    a.fz_off_a = (int)off;
    off += NSA * stageA;
    a.fz_off_b = (int)off;
    off += al(NSB * stageB);
    a.fz_off_x = (int)off;
    off += x_bytes;
    a.fz_off_h = (int)off;
    off += h_bytes;
    a.fz_off_hs = (int)off;
    off += hs_bytes;
    a.fz_off_yw = (int)off;
    off += yw_bytes;
    a.fz_off_bar = (int)off;
    off += bar_bytes(NSA, NSB);
    a.fz_nsa = NSA;
    a.fz_nsb = NSB;
    a.fz_rb = RB;
    a.fz_stage_b = (int)stageB;
    a.fz_smem = (int)off;
    return off <= (size_t)smem_max;
}

template <int NBH, bool DEDUP>
static cudaError_t launch_expert_t(const DecodeArgs &a, int grid, cudaStream_t s) {
    // dynamic smem limits raised at plan time; NORM: pre-normed block
    auto kern = a.norm_w ? k_expert<NBH, DEDUP, true> : k_expert<NBH, DEDUP, false>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kExpertThreads);
    cfg.dynamicSmemBytes = a.fz_smem;
    cfg.stream = s;
    // The grid barrier between gate/up and down needs every CTA resident at
    // once: a cooperative launch guarantees that, or fails at launch time.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_expert_fused(const DecodeArgs &a, int grid, cudaStream_t s) {
    const int nbh = a.H / kQK;
    const bool dedup = a.n > 1;
    switch (nbh) {
        case 1: return dedup ? launch_expert_t<1, true>(a, grid, s) : launch_expert_t<1, false>(a, grid, s);
        case 2: return dedup ? launch_expert_t<2, true>(a, grid, s) : launch_expert_t<2, false>(a, grid, s);
        case 4: return dedup ? launch_expert_t<4, true>(a, grid, s) : launch_expert_t<4, false>(a, grid, s);
        default: return dedup ? launch_expert_t<8, true>(a, grid, s) : launch_expert_t<8, false>(a, grid, s);
    }
}

cudaError_t expert_fused_occupancy(int nbh, bool dedup, int smem, int smem_max, int *blocks_per_sm) {
#define SI_FZ_PAIR(B) \
    (dedup ? fs2{(const void *)k_expert<B, true, false>, (const void *)k_expert<B, true, true>} \
           : fs2{(const void *)k_expert<B, false, false>, (const void *)k_expert<B, false, true>})
    struct fs2 {
        const void *f[2];
    };
    fs2 fs{};
    switch (nbh) {
        case 1: fs = SI_FZ_PAIR(1); break;
        case 2: fs = SI_FZ_PAIR(2); break;
        case 4: fs = SI_FZ_PAIR(4); break;
        default: fs = SI_FZ_PAIR(8); break;
    }
#undef SI_FZ_PAIR
    int least = 1 << 30;
    for (const void *f : fs.f) {  // plain and pre-normed block: both must fit
        cudaFuncAttributes fa;
        cudaError_t err = cudaFuncGetAttributes(&fa, f);
        if (err != cudaSuccess) return err;
        // the opt-in limit covers static + dynamic shared memory
        const int dyn_max = smem_max - (int)fa.sharedSizeBytes;
        if (smem > dyn_max) return cudaErrorInvalidValue;
        err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max);
        if (err != cudaSuccess) return err;
        int n = 0;
        if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kExpertThreads, smem)) != cudaSuccess)
            return err;
        least = n < least ? n : least;
    }
    *blocks_per_sm = least;
    return cudaSuccess;
}

}  // namespace si
