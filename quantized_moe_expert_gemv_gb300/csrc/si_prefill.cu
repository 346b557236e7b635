// si_prefill.cu -- grouped prefill: T tokens through the mixture-of-experts FFN.
//
// SP⚡RKINFER README (gittensor-ai-lab), "Benchmark · Qwen3.6-35B-A3B", prefill
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
//   4. k_prefill_gemm<0> per (expert, 64 intermediate rows): [gate; up] rows
//                        (M = 128) x the expert's tokens (N <= 512 per pass)
//                        over K = H, then h = fp16(silu(g) * u) in perm order
//   5. k_prefill_gemm<1> per (expert, 128 output rows): down rows x the
//                        expert's h rows over K = I, times the routing weight,
//                        into y (fp32, perm order)
//   6. k_prefill_combine out[t] = sum over slots, in slot order, of y[inv[t*k+s]]
//
// The GEMMs run on the 5th-generation tensor cores: 16-bit operands in shared
// memory (K-major, 128-byte swizzle), fp32 accumulators in tensor memory.
// Weights (operand A) are Q4_K blocks fetched by tensor-map copies and
// dequantized by eight warps: w = d*sc*q - dmin*m, exact in fp32, rounded once
// to fp16 (nearest even).  Tokens (operand B) are gathered row by row with
// 16-byte asynchronous copies.  One MMA thread issues 128 x N x 16 MMAs; a
// warpgroup reads the accumulators back for the epilogue.
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
#include <cuda_fp16.h>

#include <cstdint>

#include "si_device.cuh"
#include "si_internal.h"
#include "si_tc.cuh"

namespace si {

// =====================================================================
// 1-3. Routing, counts, offsets, permutation
// =====================================================================
namespace {
constexpr int kRtTok = 32;      // tokens per router CTA
constexpr int kRtExp = 128;     // experts per pass of the router tile
constexpr int kRtKc = 32;       // hidden columns per staged chunk
constexpr int kRtThreads = 256;
constexpr int kRtXBytes = kRtKc * kRtTok * 4;
constexpr int kRtWBytes = kRtExp * (kRtKc + 1) * 4;
constexpr int kRtSmem = kRtXBytes + kRtWBytes + kRtTok * SI_MAX_EXPERTS * 4;  // 53,760
}  // namespace

// Logits of 32 tokens x all experts (fp32 FMA, hidden order), then per token
// (one warp each) the top-k by k rounds of a warp-wide maximum (ties to the
// lower index), the renormalised weights and the per-expert pair counts.
__global__ void __launch_bounds__(kRtThreads) k_prefill_route(PrefillArgs a) {
    extern __shared__ __align__(16) uint8_t rt_smem[];
    float(*s_x)[kRtTok] = reinterpret_cast<float(*)[kRtTok]>(rt_smem);                            // [kRtKc][kRtTok]
    float(*s_w)[kRtKc + 1] = reinterpret_cast<float(*)[kRtKc + 1]>(rt_smem + kRtXBytes);          // [kRtExp][kRtKc+1]
    float(*s_z)[SI_MAX_EXPERTS] = reinterpret_cast<float(*)[SI_MAX_EXPERTS]>(rt_smem + kRtXBytes + kRtWBytes);
    const int t0 = blockIdx.x * kRtTok;
    const int tid = threadIdx.x, te = tid & 31, tt = tid >> 5;  // experts te + 32i, tokens 4tt..4tt+3
    for (int e0 = 0; e0 < a.E; e0 += kRtExp) {
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        for (int c0 = 0; c0 < a.H; c0 += kRtKc) {
            for (int q = tid; q < kRtExp * kRtKc; q += kRtThreads) {
                const int r = q / kRtKc, c = q - r * kRtKc;
                s_w[r][c] = (e0 + r < a.E) ? __ldg(a.router_w + (size_t)(e0 + r) * a.H + c0 + c) : 0.f;
            }
            for (int q = tid; q < kRtTok * kRtKc; q += kRtThreads) {
                const int tk = q / kRtKc, c = q - tk * kRtKc;
                const int t = t0 + tk;
                const float xv = t < a.T ? __uint_as_float((uint32_t)__ldg(a.x + (size_t)t * a.H + c0 + c) << 16) : 0.f;
                s_x[c][tk] = xv;
                if (e0 == 0 && t < a.T) {  // fp16 copy of x for the tensor-core GEMM
                    if (fabsf(xv) > 65504.f) set_status(a.ctrl + kCtrlStatus, SI_ERR_RANGE);
                    a.xh[(size_t)t * a.H + c0 + c] = __half_as_ushort(__float2half_rn(xv));
                }
            }
            __syncthreads();
#pragma unroll 8
            for (int c = 0; c < kRtKc; ++c) {
                const float4 xv = *reinterpret_cast<const float4 *>(&s_x[c][4 * tt]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float w = s_w[te + 32 * i][c];
                    acc[i][0] = fmaf(w, xv.x, acc[i][0]);
                    acc[i][1] = fmaf(w, xv.y, acc[i][1]);
                    acc[i][2] = fmaf(w, xv.z, acc[i][2]);
                    acc[i][3] = fmaf(w, xv.w, acc[i][3]);
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = e0 + te + 32 * i;
            if (e < a.E) {
                const float b = a.router_bias ? __ldg(a.router_bias + e) : 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) s_z[4 * tt + j][e] = a.router_bias ? acc[i][j] + b : acc[i][j];
            }
        }
    }
    __syncthreads();
    // top-k: warp w takes tokens w, w+8, w+16, w+24
    const int lane = tid & 31, warp = tid >> 5;
    const int per = (a.E + 31) >> 5;
    for (int tk = warp; tk < kRtTok; tk += kRtThreads / 32) {
        const int t = t0 + tk;
        if (t >= a.T) break;
        const float *z = s_z[tk];
        if (a.o_logits)
            for (int e = lane; e < a.E; e += 32) a.o_logits[(size_t)t * a.E + e] = z[e];
        // lane l holds experts per*l .. per*l+per-1 as order-preserving keys (0 = taken)
        uint32_t key[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = per * lane + q;
            uint32_t u = 0;
            if (q < per && e < a.E) {
                const uint32_t b = __float_as_uint(z[e] + 0.0f);
                u = max((b & 0x80000000u) ? ~b : (b | 0x80000000u), 1u);
            }
            key[q] = u;
        }
        int my_id = 0;
        float my_z = 0.f;
        for (int r = 0; r < a.k; ++r) {
            uint32_t best = 0;
            int bq = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (key[q] > best) best = key[q], bq = q;
            const uint32_t top = __reduce_max_sync(0xffffffffu, best);
            const int win = __ffs(__ballot_sync(0xffffffffu, best == top)) - 1;
            const int wq = __shfl_sync(0xffffffffu, bq, win);
            if (lane == win) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q == wq) key[q] = 0u;
            }
            if (lane == r) {
                my_id = per * win + wq;
                my_z = z[my_id];
            }
        }
        const float z0 = __shfl_sync(0xffffffffu, my_z, 0);
        const float ex = lane < a.k ? expf(my_z - z0) : 0.f;
        float den = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (lane < a.k) {
            const size_t p = (size_t)t * a.k + lane;
            const float w = ex / den;
            a.ids[p] = my_id;
            a.wts[p] = w;
            if (a.o_ids) a.o_ids[p] = my_id;
            if (a.o_w) a.o_w[p] = w;
            atomicAdd(a.counts + my_id, 1);
        }
    }
}

// offsets[e] = counts[0] + ... + counts[e-1]; offsets[E] = T*k.  One CTA.
__global__ void __launch_bounds__(256) k_prefill_scan(PrefillArgs a) {
    __shared__ int s_warp[8];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    const int c = e < a.E ? a.counts[e] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_warp[w];
    if (e < a.E) {
        a.offsets[e] = base + incl - c;
        if (a.o_offsets) a.o_offsets[e] = base + incl - c;
        if (a.o_counts) a.o_counts[e] = c;
    }
    if (e == 0) {
        a.offsets[a.E] = a.T * a.k;
        if (a.o_offsets) a.o_offsets[a.E] = a.T * a.k;
    }
}

// One CTA per expert: an ordered stream compaction of the pair ids that chose
// it (pair order), written at offsets[e].
__global__ void __launch_bounds__(1024) k_prefill_perm(PrefillArgs a) {
    __shared__ int s_warp[32];
    __shared__ int s_base;
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int off = a.offsets[e];
    const int np = a.T * a.k;
    if (tid == 0) s_base = 0;
    __syncthreads();
    for (int p0 = 0; p0 < np; p0 += 1024) {
        const int p = p0 + tid;
        const bool mine = p < np && __ldg(a.ids + p) == e;
        const uint32_t bal = __ballot_sync(0xffffffffu, mine);
        if (lane == 0) s_warp[warp] = __popc(bal);
        __syncthreads();
        int before = s_base;
        for (int w = 0; w < warp; ++w) before += s_warp[w];
        if (mine) {
            const int pos = off + before + __popc(bal & ((1u << lane) - 1u));
            a.perm[pos] = p;
            a.inv[p] = pos;
            if (a.o_perm) a.o_perm[pos] = p;
        }
        __syncthreads();
        if (tid == 0) {
            int tot = 0;
            for (int w = 0; w < 32; ++w) tot += s_warp[w];
            s_base += tot;
        }
        __syncthreads();
    }
}

// out[t][c] = sum over slots s = 0..k-1 (in order) of y[inv[t*k+s]][c].
__global__ void __launch_bounds__(256) k_prefill_combine(PrefillArgs a) {
    const int c4 = a.H / 4;
    const size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= (size_t)a.T * c4) return;
    const int t = (int)(q / c4), c = (int)(q - (size_t)t * c4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < a.k; ++s) {
        const int pos = __ldg(a.inv + (size_t)t * a.k + s);
        const float4 v = __ldg(reinterpret_cast<const float4 *>(a.y + (size_t)pos * a.H) + c);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    reinterpret_cast<float4 *>(a.out + (size_t)t * a.H)[c] = acc;
}

// =====================================================================
// 4-5. Grouped GEMMs on the tensor cores
// =====================================================================
namespace {
constexpr int kGW = 12;                    // warps: 0-1 gather, 2 weight copies, 3 MMA, 4-11 dequant (4-7 epilogue)
constexpr int kGThreads = kGW * 32;
constexpr int kNS = 2;                     // operand stages (64-wide K steps)
constexpr int kNR = 2;                     // raw Q4_K stages (256-wide K blocks)
constexpr int kMaxTok = 512;               // tokens per pass: two 256-column accumulators
constexpr int kATile = 128 * 128;          // 128 weight rows x 64 fp16
constexpr int kBTile = kMaxTok * 128;      // up to 512 token rows x 64 fp16
constexpr int kStage = kATile + kBTile;
constexpr int kRaw = 128 * kBlockBytes;    // 128 weight rows x one Q4_K block
constexpr int kXch = 64 * 33 * 4;          // gate/up epilogue exchange: 64 rows x 32 tokens (+pad)
constexpr int kOffRaw = kNS * kStage;
constexpr int kOffXch = kOffRaw + kNR * kRaw;
constexpr int kOffRows = kOffXch + kXch;   // [kMaxTok] int64 source element offsets (-1 = pad)
constexpr int kOffBar = kOffRows + kMaxTok * 8;
constexpr int kNBar = 2 * kNR + 3 * kNS + 2 + 1;
constexpr int kGemmSmem = kOffBar + kNBar * 8 + 16 + 1024;  // + alignment slack
constexpr long long kDrainG = 4000000000LL;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// The sequence of work every role walks through in the same order: units
// (expert, row tile) strided over the grid, each in passes of <= 512 tokens.
struct Pass {
    int e, tile, off, sc, nt;  // expert, row tile, first pair position, first token of the pass, tokens
};
}  // namespace

// MODE 0 (gate/up): A rows 0-63 = gate rows tile*64.., rows 64-127 = up rows;
//   K = H; B row r = token of pair perm[off + sc + r]; epilogue writes
//   h[off + sc + r][tile*64 + i] = fp16(silu(g_i) * u_i).
// MODE 1 (down): A rows = down rows tile*128..; K = I; B row r = h row
//   off + sc + r; epilogue writes y[pos][tile*128 + i] = w_pair * acc.
template <int MODE>
__global__ void __launch_bounds__(kGThreads, 1)
    k_prefill_gemm(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                   PrefillArgs a) {
    extern __shared__ uint8_t g_smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(g_smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint32_t s_taddr;
    __shared__ int s_err;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = MODE == 0 ? a.I / 64 : a.H / 128;
    const int nU = a.E * tiles;
    const int K = MODE == 0 ? a.H : a.I;
    const int nK = K / 64;
    const long long budget = a.wait_budget;
    int32_t *status = a.ctrl + kCtrlStatus;

    const uint32_t bar0 = smem_addr(sm + kOffBar);
    const uint32_t raw_full = bar0, raw_empty = bar0 + 8 * kNR;
    const uint32_t full_a = bar0 + 16 * kNR, full_b = full_a + 8 * kNS, empty = full_b + 8 * kNS;
    const uint32_t d_full = empty + 8 * kNS, d_empty = d_full + 8, fin = d_empty + 8;
    int64_t *rows = reinterpret_cast<int64_t *>(sm + kOffRows);
    volatile int *verr = &s_err;

    if (threadIdx.x == 0) {
        s_err = 0;
        prefetch_tensormap(&tm_a0);
        if (MODE == 0) prefetch_tensormap(&tm_a1);
        for (int r = 0; r < kNR; ++r) {
            mbar_init(raw_full + 8 * r, 1);
            mbar_init(raw_empty + 8 * r, 8);
        }
        for (int s = 0; s < kNS; ++s) {
            mbar_init(full_a + 8 * s, 8);
            mbar_init(full_b + 8 * s, 64);
            mbar_init(empty + 8 * s, 1);
        }
        mbar_init(d_full, 1);
        mbar_init(d_empty, 4);
        mbar_init(fin, 1);
        fence_mbar_init();
    }
    if (warp == 3) {
        tc::tmem_alloc(smem_addr(&s_taddr), 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = s_taddr;

    // every role walks the same passes
    auto for_each_pass = [&](auto &&body) {
        for (int u = blockIdx.x; u < nU && !*verr; u += gridDim.x) {
            const int e = u / tiles, tile = u - e * tiles;
            const int ne = __ldg(a.counts + e), off = __ldg(a.offsets + e);
            for (int sc = 0; sc < ne && !*verr; sc += kMaxTok) body(Pass{e, tile, off, sc, min(kMaxTok, ne - sc)});
        }
    };
    auto fail = [&]() {
        if (!*verr) set_status(status, SI_ERR_TIMEOUT);
        *verr = 1;
    };

    if (warp < 2) {
        // ------------------------------------------------ gather: token rows -> B tiles
        // Gather warp w owns token rows [256w, 256w + 256) of a pass: it builds
        // their source offsets and copies them, 8 lanes per 128-byte row.
        const int r_lo = 256 * warp;
        const int sub = lane >> 3, c = lane & 7;
        int step = 0;
        for_each_pass([&](const Pass &ps) {
            const int ntp = (ps.nt + 15) & ~15;
            const int r_hi = min(ntp, r_lo + 256);
            __syncwarp();
            for (int r = r_lo + lane; r < r_hi; r += 32) {
                int64_t src = -1;
                if (r < ps.nt) {
                    const int pos = ps.off + ps.sc + r;
                    src = MODE == 0 ? (int64_t)(__ldg(a.perm + pos) / a.k) * a.H : (int64_t)pos * a.I;
                }
                rows[r] = src;
            }
            __syncwarp();
            const uint16_t *base = MODE == 0 ? a.xh : a.h;
            for (int kb = 0; kb < nK; ++kb, ++step) {
                const int s = step % kNS;
                if (step >= kNS && !mbar_wait_warp(empty + 8 * s, ((step / kNS) - 1) & 1, budget)) {
                    fail();
                    return;
                }
                const uint32_t bt = smem_addr(sm + s * kStage + kATile);
                for (int r = r_lo + sub; r < r_hi; r += 4) {
                    const int64_t src = rows[r];
                    const uint32_t dst = bt + r * 128 + ((c ^ (r & 7)) << 4);
                    cp_async16(dst, base + (src >= 0 ? src + kb * 64 + c * 8 : 0), src >= 0);
                }
                cp_async_arrive_noinc(full_b + 8 * s);
            }
        });
        cp_async_wait_all();
    } else if (warp == 2) {
        // ------------------------------------------------ Q4_K weight blocks (tensor-map copies)
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int rstep = 0;
            for_each_pass([&](const Pass &ps) {
                for (int blk = 0; blk < nK / 4; ++blk, ++rstep) {
                    const int r = rstep % kNR;
                    if (rstep >= kNR && !mbar_wait_bounded(raw_empty + 8 * r, ((rstep / kNR) - 1) & 1, budget)) {
                        fail();
                        return;
                    }
                    const uint32_t dst = smem_addr(sm + kOffRaw + r * kRaw);
                    mbar_arrive_expect_tx(raw_full + 8 * r, kRaw);
                    if (MODE == 0) {
                        const int y = ps.e * a.I + ps.tile * 64;
                        tma_load_2d(dst, &tm_a0, kBlockBytes * blk, y, raw_full + 8 * r, pol);
                        tma_load_2d(dst + 64 * kBlockBytes, &tm_a1, kBlockBytes * blk, y, raw_full + 8 * r, pol);
                    } else {
                        tma_load_2d(dst, &tm_a0, kBlockBytes * blk, ps.e * a.H + ps.tile * 128, raw_full + 8 * r,
                                    pol);
                    }
                }
            });
            // drain: every issued block must have landed before the CTA exits
            for (int q = (rstep > kNR ? rstep - kNR : 0); q < rstep; ++q)
                mbar_wait_bounded(raw_full + 8 * (q % kNR), (q / kNR) & 1, kDrainG);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            int step = 0, npass = 0;
            bool issued = false;
            for_each_pass([&](const Pass &ps) {
                if (npass > 0 && !mbar_wait_bounded(d_empty, (npass - 1) & 1, budget)) {
                    fail();
                    return;
                }
                tc::fence_after_sync();
                const int nch = (ps.nt + 255) >> 8;
                for (int kb = 0; kb < nK; ++kb, ++step) {
                    const int s = step % kNS;
                    const uint32_t par = (step / kNS) & 1;
                    if (!mbar_wait_bounded(full_a + 8 * s, par, budget) || !mbar_wait_bounded(full_b + 8 * s, par, budget)) {
                        fail();
                        return;
                    }
                    tc::fence_proxy_async_smem();  // gathered rows were written through the generic proxy
                    tc::fence_after_sync();
                    const uint32_t at = smem_addr(sm + s * kStage);
                    for (int c = 0; c < nch; ++c) {
                        const int nc = min(256, ps.nt - 256 * c);
                        const uint32_t idesc = tc::idesc_f16_f32(128, (nc + 15) & ~15);
                        const uint32_t bt = at + kATile + c * 256 * 128;
                        for (int j = 0; j < 4; ++j)
                            tc::mma_f16kind(taddr + 256 * c, tc::sdesc_sw128(at + 32 * j), tc::sdesc_sw128(bt + 32 * j),
                                         idesc, kb > 0 || j > 0);
                    }
                    tc::mma_commit(empty + 8 * s);
                    issued = true;
                }
                tc::mma_commit(d_full);
                ++npass;
            });
            if (issued) {  // every MMA has completed before the tensor memory is released
                tc::mma_commit(fin);
                mbar_wait_bounded(fin, 0, kDrainG);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ dequant (warps 4-11), epilogue (warps 4-7)
        const int d = threadIdx.x - 128;  // 0..255
        const int row = d >> 1, half = d & 1;
        const int ew = warp - 4;          // epilogue warp 0..3 (tensor-memory lanes 32*ew..)
        float *xch = reinterpret_cast<float *>(sm + kOffXch);
        int astep = 0, rstep = 0, npass = 0;
        for_each_pass([&](const Pass &ps) {
            for (int kb = 0; kb < nK; ++kb, ++astep) {
                const int j = kb & 3;
                const int r = rstep % kNR;
                if (j == 0 && !mbar_wait_warp(raw_full + 8 * r, (rstep / kNR) & 1, budget)) {
                    fail();
                    return;
                }
                const int s = astep % kNS;
                if (astep >= kNS && !mbar_wait_warp(empty + 8 * s, ((astep / kNS) - 1) & 1, budget)) {
                    fail();
                    return;
                }
                const uint8_t *blk = sm + kOffRaw + r * kRaw + row * kBlockBytes;
                const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
                const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * j);
                const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * j);
                int sc, m;
                unpack_sc_m(hdr, 2 * j + half, sc, m);
                const float dd = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
                const float dsc = dd * (float)sc, dm = dmin * (float)m;
                if (fmaxf(fabsf(fmaf(dsc, 15.f, -dm)), fabsf(dm)) > 65504.f) set_status(status, SI_ERR_RANGE);
                const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                const int sh = 4 * half;
                uint32_t o[16];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const uint32_t b = wv[t] >> sh;
                    const float f0 = fmaf(dsc, (float)(b & 15u), -dm);
                    const float f1 = fmaf(dsc, (float)((b >> 8) & 15u), -dm);
                    const float f2 = fmaf(dsc, (float)((b >> 16) & 15u), -dm);
                    const float f3 = fmaf(dsc, (float)((b >> 24) & 15u), -dm);
                    o[2 * t] = f16x2_rn(f0, f1);
                    o[2 * t + 1] = f16x2_rn(f2, f3);
                }
                uint8_t *at = sm + s * kStage + row * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = (4 * half + c) ^ (row & 7);
                    *reinterpret_cast<uint4 *>(at + chunk * 16) =
                        make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_a + 8 * s);
                if (j == 3) {
                    if (lane == 0) mbar_arrive(raw_empty + 8 * r);
                    ++rstep;
                }
            }
            if (ew < 4) {
                // -------------------------------------------- epilogue
                if (!mbar_wait_warp(d_full, npass & 1, budget)) {
                    fail();
                    return;
                }
                tc::fence_after_sync();
                const int nch = (ps.nt + 255) >> 8;
                for (int c = 0; c < nch; ++c) {
                    const int nc = min(256, ps.nt - 256 * c);
                    for (int col0 = 0; col0 < nc; col0 += 32) {
                        uint32_t v[32];
                        tc::tmem_ld32(taddr + ((uint32_t)(32 * ew) << 16) + 256 * c + col0, v);
                        tc::tmem_wait_ld();
                        if (MODE == 0) {
                            if (ew >= 2)  // up rows: hand them to the gate-row threads
                                for (int q = 0; q < 32; ++q) xch[(32 * (ew - 2) + lane) * 33 + q] = __uint_as_float(v[q]);
                            asm volatile("bar.sync 3, 128;" ::: "memory");
                            if (ew < 2) {
                                const int i = ps.tile * 64 + 32 * ew + lane;
                                for (int q = 0; q < 32 && col0 + q < nc; ++q) {
                                    const float gg = __uint_as_float(v[q]);
                                    const float uu = xch[(32 * ew + lane) * 33 + q];
                                    const float hv = silu(gg) * uu;
                                    const size_t pos = (size_t)ps.off + ps.sc + 256 * c + col0 + q;
                                    if (fabsf(hv) > 65504.f) set_status(status, SI_ERR_RANGE);
                                    a.h[pos * a.I + i] = __half_as_ushort(__float2half_rn(hv));
                                }
                            }
                            asm volatile("bar.sync 3, 128;" ::: "memory");
                        } else {
                            const int f = ps.tile * 128 + 32 * ew + lane;
                            const int pos0 = ps.off + ps.sc + 256 * c + col0;
                            float wl = 0.f;  // routing weight of token col0 + lane
                            if (col0 + lane < nc) wl = __ldg(a.wts + __ldg(a.perm + pos0 + lane));
                            for (int q = 0; q < 32; ++q) {
                                const float wq = __shfl_sync(0xffffffffu, wl, q);
                                if (col0 + q < nc) a.y[(size_t)(pos0 + q) * a.H + f] = wq * __uint_as_float(v[q]);
                            }
                        }
                    }
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(d_empty);
            }
            ++npass;
        });
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 3) {
        tc::fence_after_sync();
        tc::tmem_dealloc(taddr, 512);
    }
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

// Q4_K matrix of all experts as a 2-D byte tensor [rows][blocks_per_row * 144];
// a box is one 144-byte block column of `box_rows` consecutive rows.
static bool q4k_map(const uint8_t *base, int64_t rows, int blocks_per_row, int box_rows, CUtensorMap *tm) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)blocks_per_row * kBlockBytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)blocks_per_row * kBlockBytes};
    cuuint32_t box[2] = {(cuuint32_t)kBlockBytes, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t prefill_prepare(const Plan &p) {
    (void)p;
    if (!encoder()) return cudaErrorNotSupported;
    cudaError_t err = cudaFuncSetAttribute(k_prefill_route, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(k_prefill_gemm<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (err != cudaSuccess) return err;
    return cudaFuncSetAttribute(k_prefill_gemm<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
}

static cudaError_t mark(cudaEvent_t const *events, int i, cudaStream_t s) {
    if (!events || !events[i]) return cudaSuccess;
    return cudaEventRecordWithFlags(events[i], s, cudaEventRecordExternal);
}

cudaError_t launch_prefill(const Plan &p, const PrefillArgs &a, cudaStream_t s, cudaEvent_t const *events) {
    cudaError_t err;
    if ((err = mark(events, 0, s)) != cudaSuccess) return err;
    if ((err = cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * a.E, s)) != cudaSuccess) return err;
    k_prefill_route<<<(a.T + kRtTok - 1) / kRtTok, kRtThreads, kRtSmem, s>>>(a);
    k_prefill_scan<<<1, 256, 0, s>>>(a);
    k_prefill_perm<<<a.E, 1024, 0, s>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if ((err = mark(events, 1, s)) != cudaSuccess) return err;

    CUtensorMap tg, tu, td;
    if (!q4k_map(a.wg, (int64_t)a.E * a.I, a.H / kQK, 64, &tg) || !q4k_map(a.wu, (int64_t)a.E * a.I, a.H / kQK, 64, &tu) ||
        !q4k_map(a.wd, (int64_t)a.E * a.H, a.I / kQK, 128, &td))
        return cudaErrorInvalidValue;
    const int grid = p.sm_count;
    k_prefill_gemm<0><<<grid, kGThreads, kGemmSmem, s>>>(tg, tu, a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if ((err = mark(events, 2, s)) != cudaSuccess) return err;
    k_prefill_gemm<1><<<grid, kGThreads, kGemmSmem, s>>>(td, td, a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if ((err = mark(events, 3, s)) != cudaSuccess) return err;
    const size_t n4 = (size_t)a.T * (a.H / 4);
    k_prefill_combine<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    return mark(events, 4, s);
}

}  // namespace si
