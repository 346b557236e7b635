// si_prefill.cu -- grouped prefill: T tokens through the mixture-of-experts FFN.
//
// SP⚡RKINFER README (gittensor-ai-lab), "Benchmark · Qwen3.8-27B", prefill
// paragraph: the Q4_K weights are dequantized into the GEMM operand on every
// prefill pass; sparkinfer-k3 blog post, "v0.2.2": a chunk of tokens shares one
// weight-tile read; sparkinfer README (luciferlive112116), "Layout", moe/:
// on-device counts.
//
// Steps (stream order, no host synchronisation):
//   1. k_prefill_route   logits [T][E] (fp32), top-k per token, renormalised
//                        weights, per-expert pair counts (atomics)
//   2. k_prefill_scan    offsets[E+1] = exclusive scan of the counts
//   3. k_prefill_perm    perm: pair ids t*k+slot ordered by expert, then pair
//                        id (stable); inv: each pair's position in perm
//   4. k_prefill_gemm<0> per (expert, 128 intermediate rows): [gate; up] rows
//                        (M = 256) x the expert's tokens (N <= 384 per pass)
//                        over K = H, then h = fp16(silu(g) * u) in perm order
//   5. k_prefill_gemm<1> per (expert, 256 output rows): down rows x the
//                        expert's h rows over K = I, times the routing weight,
//                        into y (fp32, perm order)
//   6. k_prefill_combine out[t] = sum over slots, in slot order, of w[t][s] * y[inv[t*k+s]]
//
// A pre-normed block (layer norm_weight set: out = x + MoE(x * gamma / rms(x)))
// adds k_prefill_rms (1 / rms of every token) before step 1 and folds gamma
// into the router's W^T and 1 / rms into its logits.  The expert GEMM keeps x
// exact in its fp16 operand: gamma multiplies the dequantized gate/up weights
// (per hidden column, before the rounding to fp16) and 1 / rms multiplies g
// and u per token in the epilogue.  (Rounding the normalised row itself to
// fp16 shares one rounding error per column across all intermediate rows;
// measured against the oracle that alone gave up to 3.8e-3 rel-L2.)  Step 6
// adds x.
//
// The GEMMs run on the 5th-generation tensor cores as CTA pairs: 16-bit
// operands in shared memory (K-major, 128-byte swizzle), fp32 accumulators in
// tensor memory.  Weights (operand A) are Q4_K blocks fetched by tensor-map
// copies and dequantized by eight warps of each CTA: w = d*sc*q - dmin*m,
// exact in fp32, rounded once to fp16 (nearest even).  Tokens (operand B) are
// the expert's rows of a permuted copy of x (or of h), fetched by tensor-map
// copies, each CTA of the pair holding half of them.  One thread of the pair
// issues 256 x N x 16 MMAs; a warpgroup of each CTA reads its 128
// accumulator rows back for the epilogue.
//
// Operand precision: fp16, not bf16.  Rounding the dequantized weights to
// bf16 (8-bit mantissa) moves a token's layer output by up to ~5e-3 relative
// L2 on these weight distributions -- more than the output tolerance --
// while fp16 (11-bit mantissa) stays near 6e-4.  Both are kind::f16 MMAs at
// the same rate.  x (bf16) converts to fp16 exactly in fp16's normal range;
// any value beyond fp16's range (input, weight or h) is reported as
// SI_ERR_RANGE instead of becoming infinite silently.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "si_device.cuh"
#include "si_internal.h"
#include "si_tc.cuh"

namespace si {

// =====================================================================
// 1-3. Routing, counts, offsets, permutation
// =====================================================================
// W^T [H][Ew] (fp32) of the router weights, Ew = E rounded up to 128 (zero
// columns), so a chunk of 32 hidden columns x 128 experts is one [32][128]
// tile for the tensor-map copies of k_prefill_route.
__device__ __forceinline__ int router_ew(int E) { return (E + 127) & ~127; }
__global__ void __launch_bounds__(256) k_prefill_wt(PrefillArgs a) {
    __shared__ float tile[32][33];
    const int c0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int Ew = router_ew(a.E);
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    for (int r = ty; r < 32; r += 8)
        tile[r][tx] = (e0 + r < a.E) ? __ldg(a.router_w + (size_t)(e0 + r) * a.H + c0 + tx) : 0.f;
    __syncthreads();
    // a pre-normed block folds the norm gain into the rows: z = r_t * sum_c (W[e][c] * gamma_c) * x_tc
    for (int r = ty; r < 32; r += 8)
        a.wt[(size_t)(c0 + r) * Ew + e0 + tx] = a.norm_w ? tile[tx][r] * __ldg(a.norm_w + c0 + r) : tile[tx][r];
}

// Pre-normed block: rms[t] = 1 / sqrt(mean(x_t^2) + eps), one warp per token.
__global__ void __launch_bounds__(512) k_prefill_rms(PrefillArgs a) {
    const int t = blockIdx.x * 16 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= a.T) return;
    const uint32_t *xr = reinterpret_cast<const uint32_t *>(a.x + (size_t)t * a.H);
    float ss = 0.f;
    for (int c = lane; c < a.H / 2; c += 32) {
        const uint32_t v = __ldg(xr + c);
        const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) a.rms[t] = rms_scale(ss, a.H, a.norm_eps);
}

namespace {
constexpr int kRtTok = 32;                       // tokens per router CTA
constexpr int kRtExp = 128;                      // experts per pass
constexpr int kRtKs = 64;                        // hidden columns per stage
constexpr int kRtNS = 4;                         // stages
constexpr int kRtThreads = 512;
constexpr int kRtG = kRtThreads / 64;            // K groups of 64 threads (8 tokens x 8 experts each)
constexpr int kRtW = kRtKs * kRtExp * 4;         // 32 KB: W^T rows [64][128] fp32
constexpr int kRtX = kRtKs * kRtTok * 2;         // 4 KB: x [32 tokens][64] bf16 (tensor-map box)
constexpr int kRtOffX = kRtNS * kRtW;
constexpr int kRtOffZ = kRtOffX + kRtNS * kRtX;  // logits [32][SI_MAX_EXPERTS] fp32
constexpr int kRtOffBar = kRtOffZ + kRtTok * SI_MAX_EXPERTS * 4;
constexpr int kRtSmem = kRtOffBar + kRtNS * 8 + 16 + 1024;
static_assert(kRtG * kRtTok * kRtExp * 4 <= kRtNS * kRtW, "the K groups' partial sums fit in the W^T stages");
static_assert(kRtKs % (2 * kRtG) == 0, "stage columns split into column pairs over the K groups");
}  // namespace

// Logits of 32 tokens x all experts in fp32 on the SIMT pipes, W^T streamed by
// tensor-map copies in stages of 64 hidden columns.  The 512 threads form 8
// K groups (columns 8g..8g+7 of every stage); in a group each thread holds
// 8 tokens x 8 experts (packed FMA), so one 16-byte shared load feeds 8 FMAs.
// Each group sums its H/8 columns in hidden order; the 8 group sums are
// added in a fixed order.
// Then one warp per token takes the top-k as k rounds of a warp-wide argmax
// (descending logit, ties to the lower index), the renormalised weights and
// the per-expert pair counts.
__global__ void __launch_bounds__(kRtThreads, 1)
    k_prefill_route(const __grid_constant__ CUtensorMap tm_wt, const __grid_constant__ CUtensorMap tm_x, PrefillArgs a) {
    extern __shared__ uint8_t rt_smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(rt_smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kg = warp >> 1;                        // K group
    const int gi = ((warp & 1) << 5) | lane;         // thread within the group
    const int tb = gi >> 4, eb = gi & 15;            // tokens 8tb..8tb+7, experts 8eb..8eb+7 of the pass
    const int t0 = blockIdx.x * kRtTok;
    const int nst = a.H / kRtKs;
    // every CTA reads all of W^T: CTA b walks the stages from (3b) mod nst, so
    // the CTAs do not all request the same L2 lines at the same moment
    const int rot = (3 * blockIdx.x) % nst;
    const uint32_t full = smem_addr(sm + kRtOffBar);
    float(*s_z)[SI_MAX_EXPERTS] = reinterpret_cast<float(*)[SI_MAX_EXPERTS]>(sm + kRtOffZ);
    __shared__ int s_hist[SI_MAX_EXPERTS];  // pairs of this chunk per expert
    int32_t *status = a.ctrl + kCtrlStatus;
    for (int e = tid; e < a.E; e += kRtThreads) s_hist[e] = 0;
    if (tid == 0) {
        prefetch_tensormap(&tm_wt);
        prefetch_tensormap(&tm_x);
        for (int s = 0; s < kRtNS; ++s) mbar_init(full + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    int step = 0;  // stage copies issued so far (over all expert passes)
    for (int e0 = 0; e0 < a.E; e0 += kRtExp) {
        const int base = step;
        auto issue = [&](int j) {  // stage j of this expert pass into buffer (base + j) % NS
            const int s = (base + j) % kRtNS;
            const int c0 = kRtKs * ((j + rot) % nst);
            mbar_arrive_expect_tx(full + 8 * s, kRtW + kRtX);
            tma_load_2d_plain(smem_addr(sm + s * kRtW), &tm_wt, e0, c0, full + 8 * s);
            tma_load_2d_plain(smem_addr(sm + kRtOffX + s * kRtX), &tm_x, c0, t0, full + 8 * s);  // rows >= T: zeros
        };
        if (tid == 0)
            for (int j = 0; j < min(kRtNS, nst); ++j) issue(j);
        f32x2 acc[8][4];  // [token][expert pair]
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[i][q] = pack2(0.f, 0.f);
        for (int j = 0; j < nst; ++j) {
            const int s = (base + j) % kRtNS;
            if (!mbar_wait_warp(full + 8 * s, ((base + j) / kRtNS) & 1, a.wait_budget)) set_status(status, SI_ERR_TIMEOUT);
            const float *wt = reinterpret_cast<const float *>(sm + s * kRtW);  // [64 columns][128 experts] fp32
            const uint32_t *xs = reinterpret_cast<const uint32_t *>(sm + kRtOffX + s * kRtX);  // [32 tokens][32 column pairs] bf16x2
#pragma unroll 2
            for (int kp = 0; kp < kRtKs / kRtG / 2; ++kp) {
                const int k = (kRtKs / kRtG) * kg + 2 * kp;  // columns k, k + 1 in order
                const float4 w0 = *reinterpret_cast<const float4 *>(wt + k * kRtExp + 8 * eb);
                const float4 w1 = *reinterpret_cast<const float4 *>(wt + k * kRtExp + 8 * eb + 4);
                const float4 v0 = *reinterpret_cast<const float4 *>(wt + (k + 1) * kRtExp + 8 * eb);
                const float4 v1 = *reinterpret_cast<const float4 *>(wt + (k + 1) * kRtExp + 8 * eb + 4);
                const f32x2 wp[4] = {pack2(w0.x, w0.y), pack2(w0.z, w0.w), pack2(w1.x, w1.y), pack2(w1.z, w1.w)};
                const f32x2 vp[4] = {pack2(v0.x, v0.y), pack2(v0.z, v0.w), pack2(v1.x, v1.y), pack2(v1.z, v1.w)};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t xb = xs[(8 * tb + i) * (kRtKs / 2) + (k >> 1)];  // bf16 of columns k, k + 1
                    const float xa = __uint_as_float(xb << 16), xc = __uint_as_float(xb & 0xffff0000u);
                    const f32x2 xx = pack2(xa, xa), xy = pack2(xc, xc);
#pragma unroll
                    for (int q = 0; q < 4; ++q) ffma2(acc[i][q], xx, wp[q]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) ffma2(acc[i][q], xy, vp[q]);
                }
            }
            __syncthreads();  // buffer s (W^T and x) free
            if (tid == 0 && j + kRtNS < nst) issue(j + kRtNS);
        }
        step = base + nst;
        // the 4 K groups' sums through shared memory (the W^T buffers are free), added in group order
        float *part = reinterpret_cast<float *>(sm);  // [kRtG][32 tokens][128 experts]
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<float2 *>(part + (kg * kRtTok + 8 * tb + i) * kRtExp + 8 * eb + 2 * q) = unpack2(acc[i][q]);
        __syncthreads();
        for (int idx = tid; idx < kRtTok * kRtExp; idx += kRtThreads) {
            const int tk = idx / kRtExp, ex = idx % kRtExp, e = e0 + ex;
            if (e < a.E) {
                float z = part[idx];
#pragma unroll
                for (int g = 1; g < kRtG; ++g) z += part[idx + g * kRtTok * kRtExp];
                if (a.norm_w) z *= t0 + tk < a.T ? __ldg(a.rms + t0 + tk) : 0.f;
                s_z[tk][e] = a.router_bias ? z + __ldg(a.router_bias + e) : z;
            }
        }
        __syncthreads();  // the W^T buffers are reused by the next pass
    }
    if (a.o_logits)
        for (int idx = tid; idx < kRtTok * a.E; idx += kRtThreads) {
            const int tk = idx / a.E, e = idx % a.E;
            if (t0 + tk < a.T) a.o_logits[(size_t)(t0 + tk) * a.E + e] = s_z[tk][e];
        }
    // top-k: warp w takes tokens 2w, 2w+1; lane holds experts lane + 32m
    for (int tt = 0; tt < kRtTok / (kRtThreads / 32); ++tt) {
        const int tk = (kRtTok / (kRtThreads / 32)) * warp + tt, t = t0 + tk;
        if (t >= a.T) break;
        uint32_t taken = 0;
        float myv = 0.f;
        int myi = 0;
        for (int r = 0; r < a.k; ++r) {
            float v = -INFINITY;
            int bi = 0x7fffffff;
            for (int m = 0; 32 * m + lane < a.E; ++m) {
                const int e = 32 * m + lane;
                const float ze = s_z[tk][e];
                if (!((taken >> m) & 1u) && (bi == 0x7fffffff || ze > v || (ze == v && e < bi))) v = ze, bi = e;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, v, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > v || (ov == v && oi < bi))) v = ov, bi = oi;
            }
            v = __shfl_sync(0xffffffffu, v, 0);  // one decision for the whole warp
            bi = __shfl_sync(0xffffffffu, bi, 0);
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == r) myv = v, myi = bi;
        }
        // weights exp(z_r - z_0) / sum over the selected, the sum in slot order
        const float z0 = __shfl_sync(0xffffffffu, myv, 0);
        const float ex = expf(myv - z0);
        float den = 0.f;
        for (int r = 0; r < a.k; ++r) den += __shfl_sync(0xffffffffu, ex, r);
        if (lane < a.k) {
            const size_t p = (size_t)t * a.k + lane;
            const float w = ex / den;
            a.ids[p] = myi;
            a.wts[p] = w;
            if (a.o_ids) a.o_ids[p] = myi;
            if (a.o_w) a.o_w[p] = w;
            atomicAdd(a.counts + myi, 1);
            atomicAdd(s_hist + myi, 1);
        }
    }
    __syncthreads();
    for (int e = tid; e < a.E; e += kRtThreads) a.hist[(size_t)blockIdx.x * a.E + e] = s_hist[e];
}

// offsets[e] = counts[0] + ... + counts[e-1], offsets[E] = T*k; poff the same
// over the counts rounded up to multiples of 32.  One CTA.
__global__ void __launch_bounds__(256) k_prefill_scan(PrefillArgs a) {
    __shared__ int s_warp[8][2];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    const int c = e < a.E ? a.counts[e] : 0;
    const int cp = (c + 31) & ~31;
    int incl = c, inclp = cp;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        const int vp = __shfl_up_sync(0xffffffffu, inclp, o);
        if (lane >= o) incl += v, inclp += vp;
    }
    if (lane == 31) s_warp[warp][0] = incl, s_warp[warp][1] = inclp;
    __syncthreads();
    int base = 0, basep = 0;
    for (int w = 0; w < warp; ++w) base += s_warp[w][0], basep += s_warp[w][1];
    if (e < a.E) {
        a.offsets[e] = base + incl - c;
        a.poff[e] = basep + inclp - cp;
        if (a.o_offsets) a.o_offsets[e] = base + incl - c;
        if (a.o_counts) a.o_counts[e] = c;
    }
    if (e == a.E - 1) {
        a.offsets[a.E] = a.T * a.k;
        a.poff[a.E] = basep + inclp;
        if (a.o_offsets) a.o_offsets[a.E] = a.T * a.k;
    }
}

// One CTA per 32-token chunk (its 32k pairs, in pair order): each pair's
// position among its expert's pairs is the expert's offset, plus the pairs
// of that expert in earlier chunks (from the router's per-chunk counts), plus
// those earlier in this chunk (warp match masks and per-warp counts) -- the
// stable order by pair id.  perm[pos] = p, inv[p] = its padded row,
// pperm[row] = p; the CTAs also mark the padding rows (pperm = -1).
__global__ void __launch_bounds__(512) k_prefill_perm(PrefillArgs a) {
    __shared__ int s_base[SI_MAX_EXPERTS];
    __shared__ int s_wcnt[16][SI_MAX_EXPERTS];  // [warp][expert] pairs of this chunk per warp
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, nch = gridDim.x;
    const int np = a.T * a.k;
    const int p = 32 * a.k * c + tid;  // this thread's pair (tid < 32k)
    for (int e = tid; e < a.E; e += blockDim.x) {
        int b = a.offsets[e];
        for (int q = 0; q < c; ++q) b += __ldg(a.hist + (size_t)q * a.E + e);
        s_base[e] = b;
        for (int w = 0; w < 16; ++w) s_wcnt[w][e] = 0;
        // padding rows of the experts this CTA owns
        if (e % nch == c)
            for (int r = a.poff[e] + a.counts[e]; r < a.poff[e + 1]; ++r) a.pperm[r] = -1;
    }
    __syncthreads();
    const bool mine = tid < 32 * a.k && p < np;
    const int e = mine ? __ldg(a.ids + p) : -1 - lane;  // distinct dummies never match a real expert
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const int before = __popc(same & ((1u << lane) - 1u));
    if (mine && before == 0) s_wcnt[warp][e] = __popc(same);
    __syncthreads();
    if (mine) {
        int pos = s_base[e] + before;
        for (int w = 0; w < warp; ++w) pos += s_wcnt[w][e];
        const int j = pos - a.offsets[e];  // rank among the expert's pairs
        const int prow = a.poff[e] + j;
        a.perm[pos] = p;
        if (a.o_perm) a.o_perm[pos] = p;
        a.inv[p] = prow;
        a.pperm[prow] = p;
    }
}

// Padded expert-major token rows for the gate/up GEMM: xp[r] = fp16(x[token of
// pperm[r]]), zero for padding rows; a value beyond fp16's range is reported.
// A pre-normed block keeps x exact here and records each row's 1 / rms in
// rrow[r] for the gate/up epilogue (0 on padding rows).
__global__ void __launch_bounds__(256) k_prefill_xperm(PrefillArgs a) {
    constexpr int kRows = 4;  // rows per CTA iteration, their loads in flight together
    const int nrows = a.poff[a.E];
    const int c8 = a.H / 8;  // 16-byte groups per row
    const int G = gridDim.x;
    for (int r0 = blockIdx.x; r0 < nrows; r0 += kRows * G) {  // rows r0 + u*G, 32-bit indices
        int p[kRows];
#pragma unroll
        for (int u = 0; u < kRows; ++u) p[u] = r0 + u * G < nrows ? __ldg(a.pperm + r0 + u * G) : -1;
        if (a.norm_w && threadIdx.x == 0)  // pre-normed block
#pragma unroll
            for (int u = 0; u < kRows; ++u)
                if (r0 + u * G < nrows) a.rrow[r0 + u * G] = p[u] >= 0 ? __ldg(a.rms + p[u] / a.k) : 0.f;
        for (int c = threadIdx.x; c < c8; c += blockDim.x) {
            uint4 v[kRows];
#pragma unroll
            for (int u = 0; u < kRows; ++u)
                v[u] = p[u] >= 0 ? __ldg(reinterpret_cast<const uint4 *>(a.x + (size_t)(p[u] / a.k) * a.H) + c)
                                 : make_uint4(0u, 0u, 0u, 0u);
            bool big = false;
#pragma unroll
            for (int u = 0; u < kRows; ++u) {
                if (r0 + u * G >= nrows) break;
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                uint32_t h[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
                    big |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
                    const __half2 hh = __floats2half2_rn(lo, hi);
                    h[i] = *reinterpret_cast<const uint32_t *>(&hh);
                }
                __stcg(reinterpret_cast<uint4 *>(a.xp + (size_t)(r0 + u * G) * a.H) + c, make_uint4(h[0], h[1], h[2], h[3]));
            }
            if (big) set_status(a.ctrl + kCtrlStatus, SI_ERR_RANGE);
        }
    }
}

// out[t][c] = sum over slots s = 0..k-1 (in order) of y[inv[t*k+s]][c] (+ x[t][c]
// in a pre-normed block).
__global__ void __launch_bounds__(256) k_prefill_combine(PrefillArgs a) {
    const int c4 = a.H / 4;
    const size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= (size_t)a.T * c4) return;
    const int t = (int)(q / c4), c = (int)(q - (size_t)t * c4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < a.k; ++s) {
        const int pos = __ldg(a.inv + (size_t)t * a.k + s);
        const float w = __ldg(a.wts + (size_t)t * a.k + s);
        const float4 v = __ldg(reinterpret_cast<const float4 *>(a.y + (size_t)pos * a.H) + c);
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
    }
    if (a.norm_w) {  // the residual of a pre-normed block
        const uint2 xv = __ldg(reinterpret_cast<const uint2 *>(a.x + (size_t)t * a.H) + c);
        acc.x += __uint_as_float(xv.x << 16);
        acc.y += __uint_as_float(xv.x & 0xffff0000u);
        acc.z += __uint_as_float(xv.y << 16);
        acc.w += __uint_as_float(xv.y & 0xffff0000u);
    }
    reinterpret_cast<float4 *>(a.out + (size_t)t * a.H)[c] = acc;
}

// =====================================================================
// 4-5. Grouped GEMMs on the tensor cores, one CTA pair per work unit
// =====================================================================
// A work unit is (expert, row tile of 256 A rows); its two CTAs (ranks 0, 1
// of a 2-CTA cluster, on two SMs) each dequantize 128 A rows and load half of
// the expert's token rows, and the even CTA issues M = 256 pair MMAs that
// read both CTAs' shared memory.  Each SM thus receives only half of the
// token operand per K step: the copy engine delivers about 52 bytes per clock
// into one SM from L2, which a single-CTA M = 128 tile with ~256 tokens
// (32 KB of tokens per 64-wide K step) would exceed.
namespace {
constexpr int kGW = 16;                    // warps (see the role map in k_prefill_gemm)
constexpr int kGThreads = kGW * 32;
constexpr int kNS = 4;                     // operand stages (64-wide K steps): A (dequantized) + B (tokens)
constexpr int kNR = 2;                     // raw Q4_K stages (256-wide K blocks)
constexpr int kMaxTok = 384;               // tokens per pass: one chunk of <= 256 or two of <= 192
constexpr int kChunkRows = 96;             // first operand-B row (per CTA) of the second chunk in a stage
constexpr int kNBuf = 2;                   // accumulator buffers of 256 tensor-memory columns
constexpr int kBRows = 192;                // operand-B rows per CTA and stage
constexpr int kATile = 128 * 128;          // 128 weight rows x 64 fp16
constexpr int kBTile = kBRows * 128;       // 192 token rows x 64 fp16
// 128 weight rows x one block; the regions after the raw stages depend on the
// block size (144 bytes for Q4_K and NVFP4, 176 for Q5_K)
__host__ __device__ constexpr int gemm_raw(int bb) { return 128 * bb; }
constexpr int kOffB = kNS * kATile;
constexpr int kOffRaw = kOffB + kNS * kBTile;
constexpr int kStgBuf = 8192;              // MODE 0 epilogue staging buffer: 32 tokens x 64 fp16
__host__ __device__ constexpr int gemm_off_stg(int bb) { return kOffRaw + kNR * gemm_raw(bb); }
__host__ __device__ constexpr int gemm_off_bar(int bb) { return gemm_off_stg(bb) + 2 * kStgBuf; }
constexpr int kNBar = 2 * kNR + 2 * kNS + 2 * kNBuf + 2;
// 16-byte readiness tokens [kNS][8], copied odd -> even CTA
__host__ __device__ constexpr int gemm_off_tok(int bb) { return (gemm_off_bar(bb) + kNBar * 8 + 15) & ~15; }
__host__ __device__ constexpr int gemm_smem(int bb) { return gemm_off_tok(bb) + 16 * 8 * kNS + 16 + 1024; }  // + alignment slack
static_assert(gemm_smem(kQ5BlockBytes) + 64 <= 232448, "shared memory plan exceeds the per-CTA limit");
static_assert(kATile % 1024 == 0 && kOffB % 1024 == 0 && kBTile % 1024 == 0 && (kChunkRows * 128) % 1024 == 0,
              "128-byte-swizzled operand tiles start on 1024-byte boundaries");
static_assert(kOffRaw % 128 == 0 && gemm_raw(kBlockBytes) % 128 == 0 && gemm_raw(kQ5BlockBytes) % 128 == 0 &&
                  gemm_off_stg(kBlockBytes) % 128 == 0 && gemm_off_stg(kQ5BlockBytes) % 128 == 0 && kStgBuf % 128 == 0,
              "tensor-map copy destinations and sources are 128-byte aligned");
static_assert(gemm_off_bar(kBlockBytes) % 8 == 0 && gemm_off_tok(kBlockBytes) % 16 == 0 &&
                  gemm_off_bar(kQ5BlockBytes) % 8 == 0 && gemm_off_tok(kQ5BlockBytes) % 16 == 0,
              "mbarriers 8-byte, bulk-copy tokens 16-byte aligned");
constexpr long long kDrainG = 4000000000LL;
constexpr uint16_t kPairMask = 3;          // both CTAs of the pair

__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Tensor-map load into this CTA's shared memory that completes its bytes on
// an mbarrier of either CTA of the pair (cluster-window address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 2-D tensor store shared -> global (bulk-group completion), its commit and
// the wait until the shared-memory source may be overwritten.
__device__ __forceinline__ void tma_store_2d(const void *tmap, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// The sequence of work every role of both CTAs walks through in the same
// order: units (expert, row tile) strided over the CTA pairs, each in passes
// of <= kMaxTok tokens; a pass is one chunk of n <= 256 tokens or two of
// n <= 192 (n a multiple of 32, so every chunk starts on a 32-row boundary of
// the expert's padded rows and each CTA's half, n/2, is a multiple of 16).
// Chunks are numbered globally in this order; chunk g accumulates in
// tensor-memory buffer g % kNBuf, and chunk c of a pass is issued by MMA
// thread c (see below).
struct Pass {
    int e, tile, prow, sc, nt;  // expert, row tile, first padded row of the expert, first token, tokens
    int nch, n;                 // chunks and tokens per chunk (the last chunk may hold fewer valid tokens)
    int rot;                    // K steps are taken from (kb + rot) % nK: the pairs working on one expert
                                // start at different Q4_K blocks and so read different token columns
};
__device__ __forceinline__ Pass make_pass(int e, int tile, int prow, int sc, int ne, int nK) {
    Pass p;
    p.e = e;
    p.tile = tile;
    p.prow = prow;
    p.sc = sc;
    p.nt = min(kMaxTok, ne - sc);
    p.nch = p.nt <= 256 ? 1 : 2;
    p.n = ((p.nt + p.nch - 1) / p.nch + 31) & ~31;
    p.rot = 4 * (tile % (nK / 4));
    return p;
}
}  // namespace

// Q4_K -> fp16 operand conversion, one thread's share: sub-block 2j + half of
// the 144-byte block blk (32 weights, block columns 64j + 32half .. +31).
// A 4-bit code q at bit p of a word becomes the fp32 value 2^23 + q*2^p by
// or-ing in the exponent of 2^23; fma(dsc*2^-p, that, -dsc*2^(23-p)) then
// equals dsc*q exactly (a 21-bit product), and subtracting dm rounds once:
// the fp32 value w = d*sc*q - dmin*m (the same as fma(dsc, q, -dm)).  With
// GAMMA, w is multiplied in fp32 by gp[l], the gain of column l (a pre-normed
// block's RMSNorm gain).  The result is rounded to fp16 (round-to-nearest-
// even): o[i] holds columns 2i (low half) and 2i+1.  Bytes 0, 1 of a word are
// taken at p = 4*half, 4*half+8; bytes 2, 3 likewise after a 16-bit shift.
// Returns true when a weight of the sub-block (before the gain) lies beyond
// fp16's finite range.  The GEMM's dequantization warps and the test export
// si_debug_q4k_dequant_f16 both run this function.
struct Q4F16Lane {
    uint32_t m0, m8;           // nibble masks at p = 4*half and 4*half + 8
    float tp0, tp8, to0, to8;  // 2^-p and -2^(23-p) for both
};
__device__ __forceinline__ Q4F16Lane q4f16_lane(int half) {
    const int p0 = 4 * half;
    Q4F16Lane c;
    c.m0 = 15u << p0;
    c.m8 = 15u << (p0 + 8);
    c.tp0 = __uint_as_float((127u - p0) << 23);
    c.tp8 = __uint_as_float((119u - p0) << 23);
    c.to0 = -__uint_as_float((150u - p0) << 23);
    c.to8 = -__uint_as_float((142u - p0) << 23);
    return c;
}
// The 32 weights of one sub-block from its code words cw (a code at mask m0
// of a word -- bit position p -- and at m8 -- p + 8 --, and likewise in the
// word's upper half): 2^23 + q*2^p by or-ing in an exponent; with s = -1 when
// d*sc is negative (or -0), else 1, fma(., s*d*sc*2^-p, -s*d*sc*2^(23-p)) =
// s*d*sc*q exactly (+0 for q = 0), and fma(that, s, -dmin*m) rounds once to
// the fp32 weight, with the sign of zero the exact expression d*sc*q - dmin*m
// has; times the gain with GAMMA; rounded to fp16.
template <bool GAMMA>
__device__ __forceinline__ void codes_to_f16(const uint32_t (&cw)[8], uint32_t m0, uint32_t m8, f32x2 C, f32x2 O,
                                             f32x2 S, f32x2 D, const float *gp, uint32_t (&o)[16]) {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t w = cw[t], hi = w >> 16;
        const f32x2 v01 = pack2(__uint_as_float((w & m0) | 0x4B000000u), __uint_as_float((w & m8) | 0x4B000000u));
        const f32x2 v23 = pack2(__uint_as_float((hi & m0) | 0x4B000000u), __uint_as_float((hi & m8) | 0x4B000000u));
        f32x2 r01 = fma2(fma2(v01, C, O), S, D), r23 = fma2(fma2(v23, C, O), S, D);
        if (GAMMA) {
            const float4 g4 = __ldg(reinterpret_cast<const float4 *>(gp) + t);
            r01 = mul2(r01, pack2(g4.x, g4.y));
            r23 = mul2(r23, pack2(g4.z, g4.w));
        }
        const float2 a01 = unpack2(r01), a23 = unpack2(r23);
        o[2 * t] = f16x2_rn(a01.x, a01.y);
        o[2 * t + 1] = f16x2_rn(a23.x, a23.y);
    }
}

template <bool GAMMA>
__device__ __forceinline__ bool q4k_subblock_f16(const Q4F16Lane &c, const uint8_t *blk, int j, int half,
                                                 const float *gp, uint32_t (&o)[16]) {
    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
    const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * j);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * j);
    int sc, m;
    unpack_sc_m(hdr, 2 * j + half, sc, m);
    const float dd = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
    const float dsc = dd * (float)sc, dm = dmin * (float)m;
    const bool bad = fmaxf(fabsf(fmaf(dsc, 15.f, -dm)), fabsf(dm)) > 65504.f;
    const float sg = signbit(dsc) ? -1.f : 1.f, sd = sg * dsc;
    const f32x2 C = pack2(sd * c.tp0, sd * c.tp8), O = pack2(sd * c.to0, sd * c.to8), S = pack2(sg, sg),
                D = pack2(-dm, -dm);
    const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    codes_to_f16<GAMMA>(wv, c.m0, c.m8, C, O, S, D, gp, o);
    return bad;
}

// Q5_K -> fp16 operand conversion, one thread's share: sub-block 2j + half
// (32 weights).  The 5-bit codes are first gathered one per byte (the four
// low bits from qs, the fifth from bit 2j+half of qh), then formed as in
// q4k_subblock_f16 (bytes 0, 1 of a word at p = 0, 8; bytes 2, 3 after a
// 16-bit shift): w = d*sc*q - dmin*m exact in fp32, rounded once to fp16.
// Returns true when a weight (before the gain) lies beyond fp16's range.
template <bool GAMMA>
__device__ __forceinline__ bool q5k_subblock_f16(const uint8_t *blk, int j, int half, const float *gp,
                                                 uint32_t (&o)[16]) {
    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
    const uint4 h0 = *reinterpret_cast<const uint4 *>(blk + kQ5QhOff);
    const uint4 h1 = *reinterpret_cast<const uint4 *>(blk + kQ5QhOff + 16);
    const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + kQ5QsOff + 32 * j);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + kQ5QsOff + 16 + 32 * j);
    int sc, m;
    unpack_sc_m(hdr, 2 * j + half, sc, m);
    const float dd = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
    const float dsc = dd * (float)sc, dm = dmin * (float)m;
    const bool bad = fmaxf(fabsf(fmaf(dsc, 31.f, -dm)), fabsf(dm)) > 65504.f;
    const Q4F16Lane c = q4f16_lane(0);  // 2^-p and -2^(23-p) for p = 0, 8
    const float sg = signbit(dsc) ? -1.f : 1.f, sd = sg * dsc;
    const f32x2 C = pack2(sd * c.tp0, sd * c.tp8), O = pack2(sd * c.to0, sd * c.to8), S = pack2(sg, sg),
                D = pack2(-dm, -dm);
    const uint32_t qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint32_t cw[8];  // one 5-bit code per byte
#pragma unroll
    for (int t = 0; t < 8; ++t) cw[t] = half ? q5_codes_hi(qv[t], hv[t], j) : q5_codes_lo(qv[t], hv[t], j);
    codes_to_f16<GAMMA>(cw, 31u, 31u << 8, C, O, S, D, gp, o);
    return bad;
}

// NVFP4 -> fp16 operand conversion, one thread's share: weights 64j + 32half
// .. +31 of the super-block at blk (scale blocks 4j + 2half and 4j + 2half + 1).
// Each w = e2m1 * e4m3 * g is formed in fp32 -- (T - 12) * (e4m3 / 2) is the
// exact product e2m1 * e4m3, one rounding for g -- and rounded to fp16
// (nearest even); o[i] holds columns 2i (low half) and 2i+1.  Returns true
// when a weight lies beyond fp16's finite range.  The GEMM's dequantization
// warps and the test export si_debug_nvfp4_dequant_f16 both run it.
__device__ __forceinline__ bool nvfp4_half_f16(const uint8_t *blk, int j, int half, float g, uint32_t (&o)[16]) {
    const uint4 c4 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * j + 16 * half);  // 32 codes
    const uint32_t sw = *reinterpret_cast<const uint32_t *>(blk + 4 * j) >> (16 * half);  // their 2 scale bytes
    const float s0 = 0.5f * e4m3_to_f32(sw & 0xffu), s1 = 0.5f * e4m3_to_f32((sw >> 8) & 0xffu);
    const bool bad = fmaxf(fabsf(s0), fabsf(s1)) * 12.f * fabsf(g) > 65504.f;
    const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
    // e2m1 of code n of a word: (T - 12) / 2 in fp32, with the code's sign bit
    // or-ed in so that code 8 is -0 (the value is already negative otherwise)
    auto e2 = [](uint32_t vv, int byte, uint32_t word, int n) {
        const float v = (float)((int)((vv >> (8 * byte)) & 0xffu) - 12);
        return __uint_as_float(__float_as_uint(v) | ((word << (28 - 4 * n)) & 0x80000000u));
    };
#pragma unroll
    for (int t = 0; t < 4; ++t) {  // codes 8t .. 8t+7
        const float sc = t < 2 ? s0 : s1;
        const uint32_t v[2] = {e2m1_t4(cw[t]), e2m1_t4(cw[t] >> 16)};
#pragma unroll
        for (int m = 0; m < 4; ++m) {  // codes 8t + 2m, 8t + 2m + 1
            const uint32_t vv = v[m >> 1] >> (16 * (m & 1));
            const float w0 = __fmul_rn(__fmul_rn(e2(vv, 0, cw[t], 2 * m), sc), g);
            const float w1 = __fmul_rn(__fmul_rn(e2(vv, 1, cw[t], 2 * m + 1), sc), g);
            o[4 * t + m] = f16x2_rn(w0, w1);
        }
    }
    return bad;
}

// MODE 0 (gate/up): unit tile covers intermediate rows tile*128 .. +127;
//   CTA r holds rows tile*128 + 64r + i as A rows 2i (gate) and 2i+1 (up);
//   K = H; B rows = padded token rows of the expert (xp); epilogue
//   h[row][tile*128 + 64r + i] = fp16(silu(g_i) * u_i).
// MODE 1 (down): unit tile covers output rows tile*256 .. +255; CTA r holds
//   rows tile*256 + 128r + i; K = I; B rows = h rows of the expert; epilogue
//   y[row][tile*256 + 128r + i] = acc (the combine applies the routing weight).
// Roles (both CTAs): warp 0 Q4_K block copies, warp 2 operand-B copies of
// this CTA's half of the tokens, warps 4-11 dequantization, warps 12-15
// epilogue of this CTA's 128 accumulator rows; warp 1 allocates tensor
// memory (collectively for the pair) and, in the even CTA, issues the MMAs.
// Warp 3 of the even CTA is a second MMA thread: a two-chunk pass gives one
// chunk to each thread, so that one thread's barrier wait and commit (which
// would leave the tensor cores idle -- an issuing thread keeps only about one
// MMA queued) overlap the other thread's MMAs.  Accumulators are two
// 256-column buffers used round robin: the epilogue of one chunk overlaps
// the MMAs of the next.
// Barriers (same offsets in both CTAs).  One pair of barriers per operand
// stage, so the MMA thread makes one wait and one commit per K step (each
// costs it ~100 cycles, and it has ~128 cycles per 256-column MMA to spare):
// full (even CTA) completes when the even CTA's B producer has armed it, its
// 8 dequant warps have arrived, the B boxes of both CTAs have landed (the odd
// CTA's tensor copies signal the even CTA's barrier) and the odd CTA's 8
// dequant warps have each copied a 16-byte token into the even CTA after
// fencing their A tile -- copy-engine signals, so no thread stalls on a
// release at cluster scope (several hundred ns under this kernel's memory
// traffic); empty (both CTAs, both MMA threads) and d_full are completed by
// the multicast MMA commits; d_empty (even CTA) by both CTAs' epilogue
// warps; raw_* are local.
// WF = 1: NVFP4 weights (the same 144-byte blocks; nvfp4_half_f16 instead of
// q4k_subblock_f16, times the expert matrix's tensor scale).
template <int MODE, bool NORM, int WF>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGThreads, 1)
    k_prefill_gemm(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                   const __grid_constant__ CUtensorMap tm_b64, const __grid_constant__ CUtensorMap tm_b16,
                   const __grid_constant__ CUtensorMap tm_h, PrefillArgs a) {
    extern __shared__ uint8_t g_smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(g_smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int BB = WF == 3 ? kQ5BlockBytes : kBlockBytes;  // bytes per weight block (WF 3: Q5_K)
    constexpr int kRaw = gemm_raw(BB), kOffStg = gemm_off_stg(BB), kOffBar = gemm_off_bar(BB),
                  kOffTok = gemm_off_tok(BB);
    __shared__ uint32_t s_taddr;
    __shared__ int s_err;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int tiles = MODE == 0 ? a.I / 128 : a.H / 256;
    const int nU = a.E * tiles;
    const int K = MODE == 0 ? a.H : a.I;
    const int nK = K / 64;
    const long long budget = a.wait_budget;
    int32_t *status = a.ctrl + kCtrlStatus;

    const uint32_t bar0 = smem_addr(sm + kOffBar);
    const uint32_t raw_full = bar0, raw_empty = bar0 + 8 * kNR;
    const uint32_t full = bar0 + 16 * kNR, empty = full + 8 * kNS;
    const uint32_t d_full = empty + 8 * kNS, d_empty = d_full + 8 * kNBuf, fin = d_empty + 8 * kNBuf;  // fin: [2]
    volatile int *verr = &s_err;

    if (threadIdx.x == 0) {
        s_err = 0;
        prefetch_tensormap(&tm_a0);
        if (MODE == 0) prefetch_tensormap(&tm_a1);
        prefetch_tensormap(&tm_b64);
        prefetch_tensormap(&tm_b16);
        if (MODE == 0) prefetch_tensormap(&tm_h);
        for (int r = 0; r < kNR; ++r) {
            mbar_init(raw_full + 8 * r, 1);
            mbar_init(raw_empty + 8 * r, 8);
        }
        for (int s = 0; s < kNS; ++s) {
            mbar_init(full + 8 * s, 1 + 8);  // the B producer's arming + the even CTA's 8 dequant warps
            mbar_init(empty + 8 * s, 2);     // one commit from each MMA thread
        }
        for (int b = 0; b < kNBuf; ++b) {
            mbar_init(d_full + 8 * b, 1);
            mbar_init(d_empty + 8 * b, 8);  // 4 epilogue warps of each CTA
        }
        mbar_init(fin, 1);
        mbar_init(fin + 8, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc_pair(smem_addr(&s_taddr), 512);
        tc::tmem_relinquish_pair();
    }
    tc::fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
    tc::fence_after_sync();
    const uint32_t taddr = s_taddr;

    // Work units (expert, row tile) go to the pairs round by round in a snake
    // order over the experts sorted by descending pair count (ties: lower id):
    // the last, partial round gets the cheapest units and every pair a mix of
    // large and small ones.  Both CTAs of a pair derive the same order.
    __shared__ int s_cnt[SI_MAX_EXPERTS], s_order[SI_MAX_EXPERTS];
    for (int t = threadIdx.x; t < a.E; t += blockDim.x) s_cnt[t] = __ldg(a.counts + t);
    __syncthreads();
    for (int t = threadIdx.x; t < a.E; t += blockDim.x) {
        const int ct = s_cnt[t];
        int rk = 0;
        for (int j = 0; j < a.E; ++j) rk += (s_cnt[j] > ct) | ((s_cnt[j] == ct) & (j < t));
        s_order[rk] = t;
    }
    __syncthreads();

    // every role walks the same passes
    auto for_each_pass = [&](auto &&body) {
        for (int rr = 0; rr * npairs < nU && !*verr; ++rr) {
            const int u = rr * npairs + ((rr & 1) ? npairs - 1 - pair : pair);
            if (u >= nU) continue;
            const int e = s_order[u / tiles], tile = u - (u / tiles) * tiles;
            const int ne = __ldg(a.counts + e), prow = __ldg(a.poff + e);
            for (int sc = 0; sc < ne && !*verr; sc += kMaxTok) body(make_pass(e, tile, prow, sc, ne, nK));
        }
    };
    auto fail = [&]() {
        if (!*verr) set_status(status, SI_ERR_TIMEOUT);
        *verr = 1;
    };

    if (warp == 0) {
        // ------------------------------------------------ Q4_K weight blocks of this CTA's 128 rows
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();  // each Q4_K block is read by one CTA
            int rstep = 0;
            for_each_pass([&](const Pass &ps) {
                for (int bi = 0; bi < nK / 4; ++bi, ++rstep) {
                    const int blk = ((4 * bi + ps.rot) % nK) >> 2;
                    const int r = rstep % kNR;
                    if (rstep >= kNR && !mbar_wait_spin(raw_empty + 8 * r, ((rstep / kNR) - 1) & 1, budget)) {
                        fail();
                        return;
                    }
                    const uint32_t dst = smem_addr(sm + kOffRaw + r * kRaw);
                    mbar_arrive_expect_tx(raw_full + 8 * r, 128 * BB);
                    if (MODE == 0) {
                        const int y = ps.e * a.I + ps.tile * 128 + 64 * rank;
                        tma_load_2d(dst, &tm_a0, BB * blk, y, raw_full + 8 * r, pol);
                        tma_load_2d(dst + 64 * BB, &tm_a1, BB * blk, y, raw_full + 8 * r, pol);
                    } else {
                        tma_load_2d(dst, &tm_a0, BB * blk, ps.e * a.H + ps.tile * 256 + 128 * rank,
                                    raw_full + 8 * r, pol);
                    }
                }
            });
            // drain: every issued block has landed before the CTA exits
            for (int q = (rstep > kNR ? rstep - kNR : 0); q < rstep; ++q)
                mbar_wait_bounded(raw_full + 8 * (q % kNR), (q / kNR) & 1, kDrainG);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ this CTA's half of every chunk's token rows
        if (lane == 0) {
            const uint32_t lead_full = mapa_shared(full, 0);
            int step = 0;
            for_each_pass([&](const Pass &ps) {
                const int hr = ps.n >> 1;  // rows per chunk half (multiple of 16, <= 128; <= 96 with two chunks)
                for (int kb = 0; kb < nK; ++kb, ++step) {
                    const int s = step % kNS;
                    if (step >= kNS && !mbar_wait_spin_cluster(empty + 8 * s, ((step / kNS) - 1) & 1, budget)) {
                        fail();
                        return;
                    }
                    const uint32_t bt = smem_addr(sm + kOffB + s * kBTile);
                    // even CTA: both CTAs' boxes and the odd CTA's 8 A-tile tokens
                    if (rank == 0) mbar_arrive_expect_tx(full + 8 * s, (uint32_t)(2 * ps.nch * hr * 128 + 8 * 16));
                    const int x = 64 * ((kb + ps.rot) % nK);
                    for (int c = 0; c < ps.nch; ++c) {
                        const uint32_t dst = bt + c * kChunkRows * 128;
                        const int row = ps.prow + ps.sc + c * ps.n + rank * hr;
                        int q = 0;
                        for (; q + 64 <= hr; q += 64) tma_load_2d_pair(dst + q * 128, &tm_b64, x, row + q, lead_full + 8 * s);
                        for (; q < hr; q += 16) tma_load_2d_pair(dst + q * 128, &tm_b16, x, row + q, lead_full + 8 * s);
                    }
                }
            });
            if (rank == 0)  // the even CTA's full covers the copies of both CTAs
                for (int q = (step > kNS ? step - kNS : 0); q < step; ++q)
                    mbar_wait_bounded_cluster(full + 8 * (q % kNS), (q / kNS) & 1, kDrainG);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------ pair MMA issue (even CTA: warps 1 and 3, one thread each)
        if (lane == 0 && rank == 0) {
            const int me = warp >> 1;  // MMA thread 0 or 1: issues chunk c == me of each pass
            const uint64_t desc_base = tc::sdesc_sw128(smem_addr(sm));
            int step = 0, g0 = 0;  // g0: global index of the pass's first chunk
            bool issued = false;
            for_each_pass([&](const Pass &ps) {
                for (int c = me; c < ps.nch; c += 2) {  // this thread's buffers of the pass are drained
                    const int g = g0 + c;
                    if (g >= kNBuf &&
                        !mbar_wait_spin_cluster(d_empty + 8 * (g % kNBuf), ((g / kNBuf) - 1) & 1, budget)) {
                        fail();
                        return;
                    }
                }
                tc::fence_after_sync();
                const uint32_t idesc = tc::idesc_f16_f32(256, ps.n);
                for (int kb = 0; kb < nK; ++kb, ++step) {
                    const int s = step % kNS;
                    if (!mbar_wait_spin_cluster(full + 8 * s, (step / kNS) & 1, budget)) {
                        fail();
                        return;
                    }
                    tc::fence_after_sync();  // the dequant warps fenced their A-tile writes to the async proxy
                    // descriptors: stage bases (1024-byte aligned) >> 4 in the address field
                    const uint64_t ad = desc_base + (uint64_t)((s * kATile) >> 4);
                    const uint64_t bd = desc_base + (uint64_t)((kOffB + s * kBTile) >> 4);
                    for (int c = me; c < ps.nch; c += 2)
                        tc::mma_pair_k64(taddr + 256 * ((g0 + c) % kNBuf), ad, bd + (uint64_t)((c * kChunkRows * 128) >> 4),
                                         idesc, kb > 0);
                    tc::mma_pair_commit_mc(empty + 8 * s, kPairMask);  // also when this thread had no chunk
                    issued = true;
                }
                for (int c = me; c < ps.nch; c += 2) tc::mma_pair_commit_mc(d_full + 8 * ((g0 + c) % kNBuf), kPairMask);
                g0 += ps.nch;
            });
            if (issued) {  // every MMA has completed before either CTA releases its memory
                tc::mma_pair_commit_mc(fin + 8 * me, 1);
                mbar_wait_bounded(fin + 8 * me, 0, kDrainG);
            }
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------ dequant (warps 4-11) of this CTA's 128 rows
        const int d = threadIdx.x - 128;  // 0..255
        const float *const gam = (MODE == 0 && NORM) ? a.norm_w : nullptr;  // pre-normed block: RMSNorm gain
        const int row = d >> 1, half = d & 1;
        // MODE 0: A row 2i = gate row i, 2i+1 = up row i (raw rows: gate 0-63, up 64-127)
        const int raw_row = MODE == 0 ? ((row & 1) ? 64 + (row >> 1) : (row >> 1)) : row;
        const Q4F16Lane lc = q4f16_lane(half);  // the codes of this thread are bits 4*half.. of each byte
        const uint32_t tok = smem_addr(sm + kOffTok), lead_tok = mapa_shared(tok, 0);
        const uint32_t lead_full = mapa_shared(full, 0);
        int astep = 0, rstep = 0;
        for_each_pass([&](const Pass &ps) {
            for (int kb = 0; kb < nK; ++kb, ++astep) {
                const int j = kb & 3;  // the rotation is whole Q4_K blocks, so chunk j of a block is kb & 3
                const int r = rstep % kNR;
                if (j == 0 && !mbar_wait_warp_spin(raw_full + 8 * r, (rstep / kNR) & 1, budget)) {
                    fail();
                    return;
                }
                const int s = astep % kNS;
                if (astep >= kNS && !mbar_wait_warp_spin_cluster(empty + 8 * s, ((astep / kNS) - 1) & 1, budget)) {
                    fail();
                    return;
                }
                const uint8_t *blk = sm + kOffRaw + r * kRaw + raw_row * BB;
                uint32_t o[16];
                // pre-normed block: the gate/up weights of hidden column c times gamma_c (the
                // token's 1 / rms is applied to g and u in the epilogue), so x stays exact
                const float *gp = (MODE == 0 && NORM) ? gam + 64 * ((kb + ps.rot) % nK) + 32 * half : nullptr;
                if (WF == 1) {
                    const float g = a.wscale[3 * ps.e + (MODE == 1 ? 2 : (raw_row >= 64 ? 1 : 0))];
                    if (nvfp4_half_f16(blk, j, half, g, o)) set_status(status, SI_ERR_RANGE);
                } else if (WF == 3) {
                    if (q5k_subblock_f16<MODE == 0 && NORM>(blk, j, half, gp, o)) set_status(status, SI_ERR_RANGE);
                } else if (q4k_subblock_f16<MODE == 0 && NORM>(lc, blk, j, half, gp, o)) {
                    set_status(status, SI_ERR_RANGE);
                }
                uint8_t *at = sm + s * kATile + row * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = (4 * half + c) ^ (row & 7);
                    *reinterpret_cast<uint4 *>(at + chunk * 16) =
                        make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0) {
                        mbar_arrive(full + 8 * s);
                    } else {
                        const uint32_t slot = 16 * (8 * s + (warp - 4));
                        asm volatile(
                            "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], 16, "
                            "[%2];" ::"r"(lead_tok + slot),
                            "r"(tok + slot), "r"(lead_full + 8 * s)
                            : "memory");
                    }
                }
                if (j == 3) {
                    if (lane == 0) mbar_arrive(raw_empty + 8 * r);
                    ++rstep;
                }
            }
        });
    } else if (warp >= 12) {
        // ------------------------------------------------ epilogue (warps 12-15) of this CTA's accumulator rows
        // MODE 0: h goes through two 8 KB staging buffers and tensor-map stores
        // of 32 tokens x 64 fp16 (128-byte rows; a buffer is rewritten once the
        // store issued from it two stores earlier has read it).  MODE 1: y is
        // stored straight from registers -- for one token the 32 lanes of a warp
        // hold 32 consecutive output columns, 128 contiguous bytes.
        const int ew = warp - 12;  // tensor-memory lanes 32*ew ..
        const float *const rrow = (MODE == 0 && NORM) ? a.rrow : nullptr;  // pre-normed block: 1 / rms per row
        const bool lead = threadIdx.x == 12 * 32;
        const uint32_t lead_d_empty = mapa_shared(d_empty, 0);
        int chunk = 0, nst = 0;  // chunk: global index
        auto stage_begin = [&]() -> uint8_t * {
            if (lead && nst >= 2) bulk_wait_read1();
            asm volatile("bar.sync 4, 128;" ::: "memory");
            return sm + kOffStg + (nst & 1) * kStgBuf;
        };
        auto stage_end = [&](uint8_t *buf, int x, int y) {
            tc::fence_proxy_async_smem();
            asm volatile("bar.sync 4, 128;" ::: "memory");
            if (lead) {
                tma_store_2d(&tm_h, x, y, smem_addr(buf));
                bulk_commit();
            }
            ++nst;
        };
        for_each_pass([&](const Pass &ps) {
            for (int c = 0; c < ps.nch; ++c, ++chunk) {
                const int b = chunk % kNBuf;
                const int nv = min(ps.n, ps.nt - c * ps.n);  // valid tokens of this chunk
                const int rowc = ps.prow + ps.sc + c * ps.n;  // padded row of the chunk's first token
                if (!mbar_wait_warp_spin_cluster(d_full + 8 * b, (chunk / kNBuf) & 1, budget)) {
                    fail();
                    return;
                }
                tc::fence_after_sync();
                if (MODE == 1) {
                    // y = accumulators, straight from registers; the tensor-memory load of the
                    // next 32 columns is in flight while this group is stored
                    const uint32_t tcol = taddr + ((uint32_t)(32 * ew) << 16) + 256 * b;
                    float *yc = a.y + (size_t)rowc * a.H + ps.tile * 256 + 128 * rank + 32 * ew + lane;
                    uint32_t v[2][32];
                    tc::tmem_ld32(tcol, v[0]);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        const int col0 = 32 * g;
                        if (col0 >= nv) break;
                        if (g < 7 && col0 + 32 < nv) tc::tmem_ld32(tcol + col0 + 32, v[(g + 1) & 1]);
                        const int nq = min(32, nv - col0);
#pragma unroll
                        for (int q = 0; q < 32; ++q)
                            if (q < nq) __stcs(yc + (size_t)(col0 + q) * a.H, __uint_as_float(v[g & 1][q]));
                        tc::tmem_wait_ld();
                    }
                }
                for (int col0 = 0; MODE == 0 && col0 < nv; col0 += 32) {
                    uint32_t v[32];
                    tc::tmem_ld32(taddr + ((uint32_t)(32 * ew) << 16) + 256 * b + col0, v);
                    tc::tmem_wait_ld();
                    const int row0 = rowc + col0;  // padded row of token col0
                    if (MODE == 0) {
                        // lanes 2i / 2i+1 hold g / u of intermediate row i for 32 tokens; the even
                        // lane forms h for tokens 0-15, the odd lane for 16-31.  Rows past the
                        // chunk's tokens land in the expert's own padding (32-row aligned).
                        uint16_t *hs = reinterpret_cast<uint16_t *>(stage_begin());  // [32 tokens][64] fp16
                        const int up = lane & 1;
                        const int il = 16 * ew + (lane >> 1);
                        float hv[16];
                        bool big = false;
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const float send = __uint_as_float(up ? v[q] : v[q + 16]);
                            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                            // pre-normed block: g and u of this token times its 1 / rms
                            const float rq = rrow ? __ldg(rrow + row0 + q + 16 * up) : 1.f;
                            const float gg = (up ? recv : __uint_as_float(v[q])) * rq;
                            const float uu = (up ? __uint_as_float(v[q + 16]) : recv) * rq;
                            hv[q] = __fdividef(gg, 1.0f + __expf(-gg)) * uu;
                            // columns past the chunk's tokens hold stale accumulators: not checked
                            big |= (col0 + q + 16 * up < nv) & (fabsf(hv[q]) > 65504.f);
                        }
#pragma unroll
                        for (int q = 0; q < 16; ++q) hs[(q + 16 * up) * 64 + il] = __half_as_ushort(__float2half_rn(hv[q]));
                        if (big) set_status(status, SI_ERR_RANGE);
                        stage_end(reinterpret_cast<uint8_t *>(hs), ps.tile * 128 + 64 * rank, row0);
                    }
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0) mbar_arrive(d_empty + 8 * b);
                    else mbar_arrive_cluster(lead_d_empty + 8 * b);
                }
            }
        });
        if (MODE == 0 && lead) bulk_wait0();
    }
    // Both CTAs stay until every pair MMA has completed (the even CTA waited
    // for them) and every remote arrival has been made; then the pair releases
    // its tensor memory together.
    tc::fence_before_sync();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc_pair(taddr, 512);
    }
}

// Test export: the GEMM operand conversion above on n_blocks blocks, one
// thread per sub-block; out[256b + c] = fp16 of column c of block b.
__global__ void __launch_bounds__(256) k_debug_dequant_f16(const uint8_t *blocks, int64_t n_blocks,
                                                           const float *gamma, uint16_t *out) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_blocks * 8) return;
    const int64_t b = t >> 3;
    const int j = (int)(t & 7) >> 1, half = (int)(t & 1);
    const Q4F16Lane lc = q4f16_lane(half);
    const uint8_t *blk = blocks + b * kBlockBytes;
    uint32_t o[16];
    if (gamma)
        q4k_subblock_f16<true>(lc, blk, j, half, gamma + 256 * b + 64 * j + 32 * half, o);
    else
        q4k_subblock_f16<false>(lc, blk, j, half, nullptr, o);
    uint4 *dst = reinterpret_cast<uint4 *>(out + 256 * b + 64 * j + 32 * half);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}

__global__ void __launch_bounds__(256) k_debug_nvfp4_f16(const uint8_t *blocks, int64_t n_blocks, float g,
                                                         uint16_t *out) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_blocks * 8) return;
    const int64_t b = t >> 3;
    const int j = (int)(t & 7) >> 1, half = (int)(t & 1);
    uint32_t o[16];
    nvfp4_half_f16(blocks + b * kBlockBytes, j, half, g, o);
    uint4 *dst = reinterpret_cast<uint4 *>(out + 256 * b + 64 * j + 32 * half);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}

// Test export: the Q5_K operand conversion, as k_debug_dequant_f16.
__global__ void __launch_bounds__(256) k_debug_q5k_f16(const uint8_t *blocks, int64_t n_blocks, const float *gamma,
                                                       uint16_t *out) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_blocks * 8) return;
    const int64_t b = t >> 3;
    const int j = (int)(t & 7) >> 1, half = (int)(t & 1);
    const uint8_t *blk = blocks + b * kQ5BlockBytes;
    uint32_t o[16];
    if (gamma)
        q5k_subblock_f16<true>(blk, j, half, gamma + 256 * b + 64 * j + 32 * half, o);
    else
        q5k_subblock_f16<false>(blk, j, half, nullptr, o);
    uint4 *dst = reinterpret_cast<uint4 *>(out + 256 * b + 64 * j + 32 * half);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}

cudaError_t launch_debug_q5k_f16(const uint8_t *blocks, int64_t n_blocks, const float *gamma, uint16_t *out,
                                 cudaStream_t s) {
    if (n_blocks == 0) return cudaSuccess;
    const int64_t threads = n_blocks * 8;
    k_debug_q5k_f16<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(blocks, n_blocks, gamma, out);
    return cudaGetLastError();
}

cudaError_t launch_debug_nvfp4_f16(const uint8_t *blocks, int64_t n_blocks, float g, uint16_t *out, cudaStream_t s) {
    if (n_blocks == 0) return cudaSuccess;
    const int64_t threads = n_blocks * 8;
    k_debug_nvfp4_f16<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(blocks, n_blocks, g, out);
    return cudaGetLastError();
}

cudaError_t launch_debug_dequant_f16(const uint8_t *blocks, int64_t n_blocks, const float *gamma, uint16_t *out,
                                     cudaStream_t s) {
    if (n_blocks == 0) return cudaSuccess;
    const int64_t threads = n_blocks * 8;
    k_debug_dequant_f16<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(blocks, n_blocks, gamma, out);
    return cudaGetLastError();
}

// =====================================================================
// host
// =====================================================================
static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// A block-quantised matrix of all experts as a 2-D byte tensor
// [rows][blocks_per_row * bb] (bb = 144 for Q4_K and NVFP4, 176 for Q5_K); a box
// is one bb-byte block column of `box_rows` consecutive rows.
static bool q4k_map(const uint8_t *base, int64_t rows, int blocks_per_row, int box_rows, int bb, CUtensorMap *tm) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)blocks_per_row * bb, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)blocks_per_row * bb};
    cuuint32_t box[2] = {(cuuint32_t)bb, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major matrix [rows][cols] of fp16 (esize 2) or fp32 (esize 4); box of
// box_cols x box_rows; 128-byte swizzle for tensor-core operand tiles.
static bool mat_map(const void *base, int64_t rows, int cols, int esize, int box_cols, int box_rows, bool sw128,
                    CUtensorMap *tm) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(tm, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t prefill_prepare(const Plan &p) {
    (void)p;
    if (!encoder()) return cudaErrorNotSupported;
    cudaError_t err = cudaFuncSetAttribute(k_prefill_route, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
    if (err != cudaSuccess) return err;
    const void *fs[8] = {(const void *)k_prefill_gemm<0, false, 0>, (const void *)k_prefill_gemm<0, true, 0>,
                         (const void *)k_prefill_gemm<1, false, 0>, (const void *)k_prefill_gemm<0, false, 1>,
                         (const void *)k_prefill_gemm<1, false, 1>, (const void *)k_prefill_gemm<0, false, 3>,
                         (const void *)k_prefill_gemm<1, false, 3>, nullptr};
    for (const void *f : fs)
        if (f && (err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             gemm_smem(f == fs[5] || f == fs[6] ? kQ5BlockBytes : kBlockBytes))) !=
                     cudaSuccess)
            return err;
    return cudaSuccess;
}

// Records events[i] on s (as an external event node while s is being captured).
static cudaError_t mark(cudaEvent_t const *events, int i, cudaStream_t s) {
    if (!events || !events[i]) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t err = cudaStreamIsCapturing(s, &cs);
    if (err != cudaSuccess) return err;
    return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(events[i], s, cudaEventRecordExternal)
                                               : cudaEventRecord(events[i], s);
}

cudaError_t launch_prefill(const Plan &p, const PrefillArgs &a, cudaStream_t s, cudaEvent_t const *events) {
    cudaError_t err;
    if ((err = mark(events, 0, s)) != cudaSuccess) return err;
    if ((err = cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * a.E, s)) != cudaSuccess) return err;
    const int Ew = (a.E + 127) & ~127;
    k_prefill_wt<<<dim3(a.H / 32, Ew / 32), 256, 0, s>>>(a);
    if (a.norm_w) k_prefill_rms<<<(a.T + 15) / 16, 512, 0, s>>>(a);
    {
        CUtensorMap twt;
        CUtensorMap tx;  // x [T][H] bf16 bits (16-bit elements; the copy does not convert)
        if (!mat_map(a.wt, a.H, Ew, 4, kRtExp, kRtKs, false, &twt) || !mat_map(a.x, a.T, a.H, 2, kRtKs, kRtTok, false, &tx))
            return cudaErrorInvalidValue;
        const int grid = (a.T + kRtTok - 1) / kRtTok;
        k_prefill_route<<<grid, kRtThreads, kRtSmem, s>>>(twt, tx, a);
    }
    k_prefill_scan<<<1, 256, 0, s>>>(a);
    k_prefill_perm<<<(a.T + 31) / 32, 512, 0, s>>>(a);

    k_prefill_xperm<<<8 * p.sm_count, 256, 0, s>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if ((err = mark(events, 1, s)) != cudaSuccess) return err;

    // operand B: token rows in boxes of 64 and of 16 rows (a CTA's half of a chunk is 64*a + 16*b rows)
    CUtensorMap tg, tu, td, txp64, txp16, th64, th16, ths;
    const int bb = a.wtype == SI_WTYPE_Q5_K ? kQ5BlockBytes : kBlockBytes;
    if (!q4k_map(a.wg, (int64_t)a.E * a.I, a.H / kQK, 64, bb, &tg) ||
        !q4k_map(a.wu, (int64_t)a.E * a.I, a.H / kQK, 64, bb, &tu) ||
        !q4k_map(a.wd, (int64_t)a.E * a.H, a.I / kQK, 128, bb, &td) ||
        !mat_map(a.xp, a.rows, a.H, 2, 64, 64, true, &txp64) || !mat_map(a.xp, a.rows, a.H, 2, 64, 16, true, &txp16) ||
        !mat_map(a.h, a.rows, a.I, 2, 64, 64, true, &th64) || !mat_map(a.h, a.rows, a.I, 2, 64, 16, true, &th16) ||
        !mat_map(a.h, a.rows, a.I, 2, 64, 32, false, &ths))
        return cudaErrorInvalidValue;
    // one CTA pair (2-CTA cluster, declared on the kernel) per two SMs
    const int grid = 2 * (p.sm_count / 2);
    const bool q5 = a.wtype == SI_WTYPE_Q5_K;  // (the API takes Q5_K in plain blocks only)
    if (a.norm_w)  // pre-normed block: gamma folded into the weights, 1 / rms into the epilogue
        k_prefill_gemm<0, true, 0><<<grid, kGThreads, gemm_smem(kBlockBytes), s>>>(tg, tu, txp64, txp16, ths, a);
    else if (q5)
        k_prefill_gemm<0, false, 3><<<grid, kGThreads, gemm_smem(kQ5BlockBytes), s>>>(tg, tu, txp64, txp16, ths, a);
    else if (a.wtype == SI_WTYPE_NVFP4)
        k_prefill_gemm<0, false, 1><<<grid, kGThreads, gemm_smem(kBlockBytes), s>>>(tg, tu, txp64, txp16, ths, a);
    else
        k_prefill_gemm<0, false, 0><<<grid, kGThreads, gemm_smem(kBlockBytes), s>>>(tg, tu, txp64, txp16, ths, a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if ((err = mark(events, 2, s)) != cudaSuccess) return err;
    if (q5)
        k_prefill_gemm<1, false, 3><<<grid, kGThreads, gemm_smem(kQ5BlockBytes), s>>>(td, td, th64, th16, ths, a);
    else if (a.wtype == SI_WTYPE_NVFP4)
        k_prefill_gemm<1, false, 1><<<grid, kGThreads, gemm_smem(kBlockBytes), s>>>(td, td, th64, th16, ths, a);
    else
        k_prefill_gemm<1, false, 0><<<grid, kGThreads, gemm_smem(kBlockBytes), s>>>(td, td, th64, th16, ths, a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if ((err = mark(events, 3, s)) != cudaSuccess) return err;
    const size_t n4 = (size_t)a.T * (a.H / 4);
    k_prefill_combine<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    return mark(events, 4, s);
}

}  // namespace si
