// si_decode.cu -- bs=1 (and n<=4 deduplicated) decode through a Q4_K MoE FFN.
//
// Three stream-ordered kernels per layer, no host synchronisation
// (sparkinfer README, "Layout": moe/ "sync-free MoE router + expert dispatch
// (on-device counts, CUDA-graph-ready)"; kernels/ "decode GEMV", "fused
// quantized MoE expert FFN"):
//   1. k_router_topk : router GEMV z = W_r x (+bias); the last CTA to arrive
//                      takes softmax, top-k, renormalised weights, per-expert
//                      counts and the table of distinct experts.
//   2. k_gateup      : for every (distinct expert, intermediate row) the gate
//                      and up rows are dequantized on read and dotted with x of
//                      each token that chose the expert; h = silu(g) * u.
//   3. k_down        : every output row c dots the down rows of the selected
//                      experts with their h and sums them weighted by the
//                      routing weights (fixed order, no atomics).
#include <cstdint>

#include "si_device.cuh"
#include "si_internal.h"

namespace si {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// --------------------------------------------------------------- router
__device__ __forceinline__ float dot8_bf16(const float4 &w0, const float4 &w1, const uint4 &xv, float s) {
    s = fmaf(w0.x, __uint_as_float(xv.x << 16), s);
    s = fmaf(w0.y, __uint_as_float(xv.x & 0xffff0000u), s);
    s = fmaf(w0.z, __uint_as_float(xv.y << 16), s);
    s = fmaf(w0.w, __uint_as_float(xv.y & 0xffff0000u), s);
    s = fmaf(w1.x, __uint_as_float(xv.z << 16), s);
    s = fmaf(w1.y, __uint_as_float(xv.z & 0xffff0000u), s);
    s = fmaf(w1.z, __uint_as_float(xv.w << 16), s);
    s = fmaf(w1.w, __uint_as_float(xv.w & 0xffff0000u), s);
    return s;
}

// Sum of squares of the 8 bf16 values of xv, added to s.
__device__ __forceinline__ float sumsq8_bf16(const uint4 &xv, float s) {
    const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float lo = __uint_as_float(w[q] << 16), hi = __uint_as_float(w[q] & 0xffff0000u);
        s = fmaf(lo, lo, s);
        s = fmaf(hi, hi, s);
    }
    return s;
}

// Chunk c (64 columns) of one token's x, held by a warp as bf16 pairs (lane l:
// word wv = columns 2l, 2l+1), quantised into the cluster expert kernel's
// activation record at xq (NC = H/64 chunks): int16 pairs, xq = rint(x / s),
// s = max|x| / 32767, with the two 32-column sums and the four 16-column sums
// of xq; or, in the int8-activation mode, int8 per 32 columns with their
// scales and sums (layouts: kXqWords, kXq8Words).
__device__ __forceinline__ void router_quant_chunk(uint32_t wv, int c, int NC, uint32_t *xq_p, int lane, bool act8) {
    const float v0 = __uint_as_float(wv << 16), v1 = __uint_as_float(wv & 0xffff0000u);
    if (act8) {
        float d, sum;
        const uint32_t lo = quant_pair8(v0, v1, &d, &sum);
        const uint32_t hi = __shfl_down_sync(0xffffffffu, lo, 1);
        if ((lane & 1) == 0) {  // word lane/2 = columns 2*lane .. 2*lane+3
            const int w = lane >> 1;
            reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(xq_p) + xq8_unit_byte(c, w >> 2))[w & 3] =
                lo | (hi << 16);
        }
        float *sc = reinterpret_cast<float *>(xq_p + 16 * NC + 4 * c);
        if (lane == 0) sc[0] = d, sc[2] = sum;
        if (lane == 16) sc[1] = d, sc[3] = sum;
        return;
    }
    float mx = fmaxf(fabsf(v0), fabsf(v1));
    float sum = v0 + v1;  // lanes 0..15: the first 32 columns, 16..31: the second
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv = mx > 0.f ? 32767.0f / mx : 0.f;
    const uint32_t q = pack_q16(v0, v1, inv);
    int s2 = (int)(int16_t)(q & 0xffffu) + ((int)q >> 16);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 4);
    xq_p[32 * c + 4 * ((lane >> 2) ^ (c & 7)) + (lane & 3)] = q;
    uint32_t *dst = xq_p + 32 * NC + 8 * c;
    if (lane == 0) {
        dst[0] = __float_as_uint(mx * (1.0f / 32767.0f));
        dst[1] = __float_as_uint(sum);
    }
    if (lane == 16) dst[2] = __float_as_uint(sum);
    if ((lane & 7) == 0) dst[3 + (lane >> 3)] = (uint32_t)s2;
}

// Router + top-k, one thread-block cluster (or one CTA for small E).  NORM (a
// pre-normed block): the router rows are scaled by the RMSNorm gain in
// registers and each warp scales its logit by the token's 1 / rms.  Warp
// w of CTA c owns expert e = c*WPC + w.  NJ > 0: H == 256*NJ and the
// expert's router row is loaded into registers before the programmatic-
// dependent-launch wait (router weights do not depend on the token, so this
// overlaps the previous kernel's tail).  NJ == 0: any H, loaded after the wait.
// Logits are gathered into CTA 0 through distributed shared memory
// (asynchronous stores that count their bytes on the receiving CTA's
// mbarrier, which that CTA waits on: cheaper than a release/acquire cluster
// barrier); CTA 0 takes softmax, top-k, renormalised weights, per-expert
// counts and the table of distinct experts (deterministic: ascending expert
// id, tokens in pair order).  One token feeding the cluster expert kernel
// (sel_logits): every CTA receives every logit, each warp ranks its own
// expert and stores the selected ones at their rank; the expert kernel forms
// the weights.  A plain block also quantises x for that kernel.
template <int NJ, bool NORM>
__global__ void __launch_bounds__(NJ > 0 ? 512 : 1024) k_router_topk(DecodeArgs a) {
    __shared__ float s_z[SI_MAX_DECODE_TOKENS][SI_MAX_EXPERTS];
    __shared__ int s_ids[SI_MAX_DECODE_TOKENS][SI_MAX_TOPK];
    __shared__ float s_w[SI_MAX_DECODE_TOKENS][SI_MAX_TOPK];
    __shared__ int s_counts[SI_MAX_EXPERTS];
    __shared__ int s_pos[SI_MAX_EXPERTS];
    __shared__ int s_U;
    __shared__ __align__(8) uint64_t s_zbar;  // completes when this CTA has received its logits
    __shared__ uint4 s_x[NJ > 0 ? SI_MAX_DECODE_TOKENS * 32 * NJ : 1];  // x [n][H] bf16 (NJ > 0)
    // parameters used after the dependency wait, read now
    const uint16_t *const xg_p = pin_ptr(a.x);
    float *const out_p = pin_ptr(a.out);
    const float *const bias_p = pin_ptr(a.router_bias);
    const float *const gam_p = NORM ? pin_ptr(a.norm_w) : nullptr;  // pre-normed block: RMSNorm gain
    const float norm_eps = a.norm_eps;
    float *const ologits_p = pin_ptr(a.o_logits);
    int32_t *const ids_p = pin_ptr(a.ids);
    float *const wts_p = pin_ptr(a.wts);
    int32_t *const oids_p = pin_ptr(a.o_ids);
    float *const ow_p = pin_ptr(a.o_w);
    int32_t *const counts_p = pin_ptr(a.counts);
    int32_t *const ocounts_p = pin_ptr(a.o_counts);
    uint32_t *const xq_p = pin_ptr(a.xq);
    const int n = pin_i32(a.n), H = pin_i32(a.H), E = pin_i32(a.E), k = pin_i32(a.k);
    const int zero_out = pin_i32(a.zero_out), sel_logits = pin_i32(a.sel_logits);
    // One plain token for the cluster expert kernel (shapes the column-split router does
    // not take): that kernel's work before its own dependency wait reads nothing this
    // call produces (x is quantised here), so it may be launched at once and be resident
    // when this grid completes.
    const bool early_dependents = !NORM && sel_logits;
    if (early_dependents) pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpc = blockDim.x >> 5;
    const int e = blockIdx.x * wpc + warp;
    const float *wrow = a.router_w + (size_t)min(e, E - 1) * H;
    float4 wr[2 * (NJ > 0 ? NJ : 1)];
    if (NJ > 0) {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            wr[2 * j] = __ldg(reinterpret_cast<const float4 *>(wrow + 256 * j + 8 * lane));
            wr[2 * j + 1] = __ldg(reinterpret_cast<const float4 *>(wrow + 256 * j + 8 * lane + 4));
        }
    }
    if (NJ > 0 && gam_p) {  // pre-normed block: z = r * sum_c (W[e][c] * gamma_c) * x_c
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gam_p + 256 * j + 8 * lane));
            const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gam_p + 256 * j + 8 * lane + 4));
            wr[2 * j] = make_float4(wr[2 * j].x * g0.x, wr[2 * j].y * g0.y, wr[2 * j].z * g0.z, wr[2 * j].w * g0.w);
            wr[2 * j + 1] = make_float4(wr[2 * j + 1].x * g1.x, wr[2 * j + 1].y * g1.y, wr[2 * j + 1].z * g1.z,
                                        wr[2 * j + 1].w * g1.w);
        }
    }
    if (NJ > 0) {  // the router rows must be in registers before the wait, not fetched after it
#pragma unroll
        for (int j = 0; j < 2 * NJ; ++j)
            asm volatile("" ::"f"(wr[j].x), "f"(wr[j].y), "f"(wr[j].z), "f"(wr[j].w));
    }
    // Warm L2 with x (a prefetch returns no data: if an earlier kernel is still
    // writing x, L2 stays coherent and the loads below happen after the wait).
    if (blockIdx.x == 0 && threadIdx.x < (n * H * 2) / 128) prefetch_l2(reinterpret_cast<const uint8_t *>(xg_p) + 128 * threadIdx.x);
    const bool zsa = gridDim.x > 1;  // a cluster: logits by asynchronous stores
    if (zsa) {
        if (threadIdx.x == 0) {
            mbar_init(smem_addr(&s_zbar), 1);
            fence_mbar_init();
            // a single token: every CTA receives all n*E logits; several: CTA 0 alone
            if (sel_logits || cluster_ctarank() == 0) mbar_arrive_expect_tx(smem_addr(&s_zbar), (uint32_t)(n * E * 4));
        }
        __syncthreads();
        cluster_arrive_relaxed();
    }
    pdl_wait();  // x and the scratch are ready (previous kernels complete)
    if (!early_dependents) pdl_launch_dependents();  // the expert kernel may become resident now (x is final)
    if (NJ > 0) {             // x once per CTA into shared memory (every warp reads all of it)
        const uint4 *xg = reinterpret_cast<const uint4 *>(xg_p);
        for (int q = threadIdx.x; q < n * 32 * NJ; q += blockDim.x) s_x[q] = __ldg(xg + q);
    }
    if (zero_out && !(NORM && NJ > 0)) {  // the cluster expert kernel accumulates the top-k combine into out
        const int nthr = gridDim.x * blockDim.x;
        for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < n * H; q += nthr)
            out_p[q] = NORM ? bf16_bits_to_f32(__ldg(xg_p + q)) : 0.f;  // the residual, or nothing
    }
    if (NJ > 0) __syncthreads();
    if (zero_out && NORM && NJ > 0) {  // the residual, from the copy of x in shared memory
        const uint16_t *xs16 = reinterpret_cast<const uint16_t *>(s_x);
        const int nthr = gridDim.x * blockDim.x;
        for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < n * H; q += nthr) out_p[q] = bf16_bits_to_f32(xs16[q]);
    }
    if (e < E) {
        float acc[SI_MAX_DECODE_TOKENS] = {0.f, 0.f, 0.f, 0.f};
        float ss[SI_MAX_DECODE_TOKENS] = {0.f, 0.f, 0.f, 0.f};  // sum of squares of x (pre-normed block)
        if (NJ > 0 && gam_p) {
#pragma unroll
            for (int t = 0; t < SI_MAX_DECODE_TOKENS; ++t) {
                if (t < n) {
#pragma unroll
                    for (int j = 0; j < NJ; ++j) ss[t] = sumsq8_bf16(s_x[32 * (NJ * t + j) + lane], ss[t]);
                }
            }
        }
        if (NJ > 0) {
            // one partial per 256-column slice (independent chains), then a binary tree
#pragma unroll
            for (int t = 0; t < SI_MAX_DECODE_TOKENS; ++t) {
                if (t < n) {
                    float pj[NJ > 0 ? NJ : 1];
#pragma unroll
                    for (int j = 0; j < NJ; ++j)
                        pj[j] = dot8_bf16(wr[2 * j], wr[2 * j + 1], s_x[32 * (NJ * t + j) + lane], 0.f);
#pragma unroll
                    for (int w2 = 1; w2 < NJ; w2 <<= 1) {
#pragma unroll
                        for (int j = 0; j + w2 < NJ; j += 2 * w2) pj[j] += pj[j + w2];
                    }
                    acc[t] = pj[0];
                }
            }
        } else {
            for (int c = 8 * lane; c < H; c += 256) {
                float4 w0 = __ldg(reinterpret_cast<const float4 *>(wrow + c));
                float4 w1 = __ldg(reinterpret_cast<const float4 *>(wrow + c + 4));
                if (gam_p) {
                    const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gam_p + c));
                    const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gam_p + c + 4));
                    w0 = make_float4(w0.x * g0.x, w0.y * g0.y, w0.z * g0.z, w0.w * g0.w);
                    w1 = make_float4(w1.x * g1.x, w1.y * g1.y, w1.z * g1.z, w1.w * g1.w);
                }
#pragma unroll
                for (int t = 0; t < SI_MAX_DECODE_TOKENS; ++t) {
                    if (t < n) {
                        const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(xg_p + (size_t)t * H + c));
                        acc[t] = dot8_bf16(w0, w1, xv, acc[t]);
                        if (gam_p) ss[t] = sumsq8_bf16(xv, ss[t]);
                    }
                }
            }
        }
        if (zsa) cluster_wait();  // every CTA's barrier is initialised
#pragma unroll
        for (int t = 0; t < SI_MAX_DECODE_TOKENS; ++t) {
            if (t < n) {
                float z = warp_sum(acc[t]);
                if (gam_p) z *= rms_scale(warp_sum(ss[t]), H, norm_eps);
                if (bias_p) z += __ldg(bias_p + e);
                if (sel_logits) {  // every CTA of the cluster gets every logit (lane c -> CTA c)
                    if (lane < (int)gridDim.x) {
                        if (zsa) st_async_cluster_u32(&s_z[t][e], smem_addr(&s_zbar), (uint32_t)lane, __float_as_uint(z));
                        else s_z[t][e] = z;
                    }
                } else if (lane == 0) {
                    if (zsa) st_async_cluster_u32(&s_z[t][e], smem_addr(&s_zbar), 0, __float_as_uint(z));
                    else s_z[t][e] = z;
                }
                if (lane == 0 && ologits_p) ologits_p[t * E + e] = z;
            }
        }
    }
    // One plain token for the cluster expert kernel: quantise x per 64-column chunk
    // into the scratch (int16 pairs, xq = rint(x / s), s = max|x| / 32767; the two
    // 32-column sums; the four 16-column sums of xq), one warp per chunk, in the
    // layout the expert kernel copies into its shared memory as it is.
    if (early_dependents) {
        const uint32_t *xw32 = NJ > 0 ? reinterpret_cast<const uint32_t *>(s_x) : reinterpret_cast<const uint32_t *>(xg_p);
        const int NC = H / 64;
        const bool act8 = pin_i32(a.act8) != 0;
        for (int c = blockIdx.x + gridDim.x * warp; c < n * NC; c += gridDim.x * wpc) {
            const int t = c / NC, cc = c - t * NC;
            router_quant_chunk(xw32[(size_t)t * (H / 2) + 32 * cc + lane], cc, NC, xq_p + (size_t)t * NC * kXqWords,
                               lane, act8);
        }
    }
    if (zsa) {
        if (e >= E) cluster_wait();  // warps without an expert still take the cluster barrier
        if (sel_logits || cluster_ctarank() == 0) {
            if (!mbar_wait_warp_cluster(smem_addr(&s_zbar), 0, a.wait_budget)) set_status(a.ctrl + kCtrlStatus, SI_ERR_TIMEOUT);
        }
    } else {
        __syncthreads();
    }

    // ---- one token feeding the cluster expert kernel: every warp ranks its own
    // expert against all E logits (the number of logits that beat it: greater,
    // or equal with a lower index -- descending order, ties to the lower index)
    // and, if selected, stores it at its rank with its logit.
    if (sel_logits) {
        if (e < E) {
            const float ze = s_z[0][e];
            int c = 0;
#pragma unroll
            for (int q = 0; q < SI_MAX_EXPERTS / 32; ++q) {
                const int j = lane + 32 * q;
                if (j < E) {
                    const float zj = s_z[0][j];
                    c += (zj > ze) | ((zj == ze) & (j < e));
                }
            }
            const int r = __reduce_add_sync(0xffffffffu, c);
            if (lane == 0) {
                if (r < k) {
                    ids_p[r] = e;
                    wts_p[r] = ze;  // the expert kernel turns these into renormalised weights
                    if (oids_p) oids_p[r] = e;
                }
                counts_p[e] = r < k ? 1 : 0;
                if (ocounts_p) ocounts_p[e] = r < k ? 1 : 0;
            }
        }
        return;
    }
    if (gridDim.x > 1 && cluster_ctarank() != 0) return;

    // ---- CTA 0: top-k of every token, then counts and the distinct-expert table
    const int nk = n * k;
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_counts[i] = 0;
    cta_topk_ranks(s_z, n, E, k, s_ids, s_w);
    __syncthreads();
    if (warp < n) {
        warp_renorm(s_w[warp], k);
        for (int i = lane; i < k; i += 32) {
            ids_p[warp * k + i] = s_ids[warp][i];
            wts_p[warp * k + i] = s_w[warp][i];
            if (oids_p) oids_p[warp * k + i] = s_ids[warp][i];
            if (ow_p) ow_p[warp * k + i] = s_w[warp][i];
        }
    }
    __syncthreads();
    for (int p = threadIdx.x; p < nk; p += blockDim.x) atomicAdd(&s_counts[s_ids[p / k][p % k]], 1);
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of "selected" flags over the E experts (8 per lane)
        int flag[8], run = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int ex = 8 * lane + q;
            flag[q] = (ex < E && s_counts[ex] > 0) ? 1 : 0;
            run += flag[q];
        }
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int pos = incl - run;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int ex = 8 * lane + q;
            if (ex < E) s_pos[ex] = pos;
            pos += flag[q];
        }
        if (lane == 31) s_U = incl;
    }
    __syncthreads();
    UniqTable *u = a.uniq;
    for (int ex = threadIdx.x; ex < E; ex += blockDim.x) {
        const int c = s_counts[ex];
        if (c > 0) {
            u->expert[s_pos[ex]] = ex;
            u->ntok[s_pos[ex]] = c;
        }
        counts_p[ex] = c;
        if (ocounts_p) ocounts_p[ex] = c;
    }
    for (int p = threadIdx.x; p < nk; p += blockDim.x) {
        const int t = p / k, i = p - t * k;
        const int ex = s_ids[t][i];
        int j = 0;  // rank among the pairs that chose ex (pair-id order)
        for (int q = 0; q < p; ++q) j += (s_ids[q / k][q % k] == ex);
        u->tok[s_pos[ex]][j] = t;
        u->slot[s_pos[ex]][j] = i;
    }
    if (threadIdx.x == 0) a.ctrl[kCtrlNumUnique] = s_U;
}

// ---------------------------------------------------------------- gate/up
template <int NT>
__device__ __forceinline__ void gateup_rowpair(const DecodeArgs &a, const float *xs,
                                               const float *Xs, const UniqTable *u, int s, int r,
                                               int lane) {
    const int e = u->expert[s];
    const int nbH = a.H / kQK;
    const bool q5 = a.wtype == SI_WTYPE_Q5_K;
    const int BB = q5 ? kQ5BlockBytes : kBlockBytes, qoff = q5 ? kQ5QsOff : 16;
    const size_t row_bytes = (size_t)nbH * BB;
    const uint8_t *gbase = a.wg + ((size_t)e * a.I + r) * row_bytes;
    const uint8_t *ubase = a.wu + ((size_t)e * a.I + r) * row_bytes;
    int tok[NT], slot[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        tok[t] = u->tok[s][t];
        slot[t] = u->slot[s][t];
    }
    float g[NT], uu[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) g[t] = uu[t] = 0.f;
    for (int it = lane; it < 4 * nbH; it += 32) {
        const int b = it >> 2, i = it & 3;
        const uint8_t *bg = gbase + b * BB;
        const uint8_t *bu = ubase + b * BB;
        const uint4 hg = ldg_nc_v4(bg), qg0 = ldg_nc_v4(bg + qoff + 32 * i),
                    qg1 = ldg_nc_v4(bg + qoff + 16 + 32 * i);
        const uint4 hu = ldg_nc_v4(bu), qu0 = ldg_nc_v4(bu + qoff + 32 * i),
                    qu1 = ldg_nc_v4(bu + qoff + 16 + 32 * i);
        uint4 hg0 = make_uint4(0, 0, 0, 0), hg1 = hg0, hu0 = hg0, hu1 = hg0;  // Q5_K: the qh bytes
        if (q5) {
            hg0 = ldg_nc_v4(bg + kQ5QhOff), hg1 = ldg_nc_v4(bg + kQ5QhOff + 16);
            hu0 = ldg_nc_v4(bu + kQ5QhOff), hu1 = ldg_nc_v4(bu + kQ5QhOff + 16);
        }
        const bool fp4 = a.wtype == SI_WTYPE_NVFP4;
        const SubScales sg = chunk_scales(hg, i), su = chunk_scales(hu, i);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float *xa = xs + (size_t)tok[t] * a.H + kQK * b + 64 * i;
            const f32x2 *pa = reinterpret_cast<const f32x2 *>(xa);
            const f32x2 *pb = reinterpret_cast<const f32x2 *>(xa + 32);
            auto xa2 = [pa](int p) { return pa[p]; };
            auto xb2 = [pb](int p) { return pb[p]; };
            const float Xa = Xs[tok[t] * (a.H / 32) + 8 * b + 2 * i];
            const float Xb = Xs[tok[t] * (a.H / 32) + 8 * b + 2 * i + 1];
            if (fp4) {  // NVFP4: the tensor scales are applied to the row sums below
                g[t] += chunk_contrib_nvfp4_f32(hg, i, qg0, qg1, xa2, xb2);
                uu[t] += chunk_contrib_nvfp4_f32(hu, i, qu0, qu1, xa2, xb2);
            } else if (q5) {
                g[t] += chunk_contrib(sg, chunk_code_sums5(qg0, qg1, hg0, hg1, i, xa2, xb2), Xa, Xb);
                uu[t] += chunk_contrib(su, chunk_code_sums5(qu0, qu1, hu0, hu1, i, xa2, xb2), Xa, Xb);
            } else {
                g[t] += chunk_contrib(sg, chunk_code_sums(qg0, qg1, xa2, xb2), Xa, Xb);
                uu[t] += chunk_contrib(su, chunk_code_sums(qu0, qu1, xa2, xb2), Xa, Xb);
            }
        }
    }
    const float tsg = a.wtype == SI_WTYPE_NVFP4 ? a.wscale[3 * e] : 1.f;
    const float tsu = a.wtype == SI_WTYPE_NVFP4 ? a.wscale[3 * e + 1] : 1.f;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const float gs = tsg * warp_sum(g[t]);
        const float us = tsu * warp_sum(uu[t]);
        if (lane == 0) a.h[((size_t)tok[t] * a.k + slot[t]) * a.I + r] = silu(gs) * us;
    }
}

__global__ void __launch_bounds__(kThreads) k_gateup_generic(DecodeArgs a) {
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;               // [n][H]
    float *Xs = smem + a.n * a.H;   // [n][H/32] sub-block sums
    const int nH = a.n * a.H;
    for (int i = threadIdx.x; i < nH; i += kThreads) xs[i] = bf16_bits_to_f32(a.x[i]);
    __syncthreads();
    if (a.norm_w) {  // pre-normed block: the experts see x * gamma / rms(x)
        __shared__ float s_r[SI_MAX_DECODE_TOKENS];
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (warp < a.n) {
            float ss = 0.f;
            for (int c = lane; c < a.H; c += 32) ss = fmaf(xs[warp * a.H + c], xs[warp * a.H + c], ss);
            ss = warp_sum(ss);
            if (lane == 0) s_r[warp] = rms_scale(ss, a.H, a.norm_eps);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nH; i += kThreads) xs[i] = xs[i] * s_r[i / a.H] * __ldg(a.norm_w + i % a.H);
        __syncthreads();
    }
    for (int i = threadIdx.x; i < nH / 32; i += kThreads) {
        float s = 0.f;
        for (int l = 0; l < 32; ++l) s += xs[32 * i + l];
        Xs[i] = s;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const UniqTable *u = a.uniq;
    const int U = a.ctrl[kCtrlNumUnique];
    const int total = U * a.I;
    for (int p = blockIdx.x * kWarps + warp; p < total; p += gridDim.x * kWarps) {
        const int s = p / a.I, r = p - s * a.I;
        switch (u->ntok[s]) {
            case 1: gateup_rowpair<1>(a, xs, Xs, u, s, r, lane); break;
            case 2: gateup_rowpair<2>(a, xs, Xs, u, s, r, lane); break;
            case 3: gateup_rowpair<3>(a, xs, Xs, u, s, r, lane); break;
            default: gateup_rowpair<4>(a, xs, Xs, u, s, r, lane); break;
        }
    }
}

// ------------------------------------------------------------------- down
template <int GS>
__global__ void __launch_bounds__(kThreads) k_down_generic(DecodeArgs a) {
    extern __shared__ __align__(16) float smem[];
    float *Hs = smem;  // [n*k][I/32] sub-block sums of h
    const int nIs = a.I / 32;
    for (int i = threadIdx.x; i < a.n * a.k * nIs; i += kThreads) {
        const float4 *hp = reinterpret_cast<const float4 *>(a.h + (size_t)32 * i);
        float s = 0.f;
#pragma unroll
        for (int l = 0; l < 8; ++l) {
            const float4 v = __ldg(hp + l);
            s += v.x + v.y + v.z + v.w;
        }
        Hs[i] = s;
    }
    __syncthreads();
    constexpr int kGroups = 32 / GS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gl = lane % GS;
    const int c = (blockIdx.x * kWarps + warp) * kGroups + lane / GS;
    if ((blockIdx.x * kWarps + warp) * kGroups >= a.H) return;  // whole warp idle
    const int nbI = a.I / kQK;
    const bool q5 = a.wtype == SI_WTYPE_Q5_K;
    const int BB = q5 ? kQ5BlockBytes : kBlockBytes, qoff = q5 ? kQ5QsOff : 16;
    const size_t row_bytes = (size_t)nbI * BB;
    const UniqTable *u = a.uniq;
    const int U = a.ctrl[kCtrlNumUnique];
    float acc[SI_MAX_DECODE_TOKENS] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < U; ++s) {
        const int e = u->expert[s];
        const int nt = u->ntok[s];
        const uint8_t *row = a.wd + ((size_t)e * a.H + c) * row_bytes;
        int sl[SI_MAX_DECODE_TOKENS];
#pragma unroll
        for (int t = 0; t < SI_MAX_DECODE_TOKENS; ++t)
            sl[t] = (t < nt) ? u->tok[s][t] * a.k + u->slot[s][t] : 0;
        float y[SI_MAX_DECODE_TOKENS] = {0.f, 0.f, 0.f, 0.f};
        for (int it = gl; it < 4 * nbI; it += GS) {
            const int b = it >> 2, i = it & 3;
            const uint8_t *blk = row + b * BB;
            const uint4 hd = ldg_nc_v4(blk), q0 = ldg_nc_v4(blk + qoff + 32 * i),
                        q1 = ldg_nc_v4(blk + qoff + 16 + 32 * i);
            uint4 qh0 = make_uint4(0, 0, 0, 0), qh1 = qh0;  // Q5_K: the qh bytes
            if (q5) qh0 = ldg_nc_v4(blk + kQ5QhOff), qh1 = ldg_nc_v4(blk + kQ5QhOff + 16);
            const SubScales sc = chunk_scales(hd, i);
            const bool fp4 = a.wtype == SI_WTYPE_NVFP4;
#pragma unroll
            for (int t = 0; t < SI_MAX_DECODE_TOKENS; ++t) {
                if (t < nt) {
                    const float *ha = a.h + (size_t)sl[t] * a.I + kQK * b + 64 * i;
                    const f32x2 *pa = reinterpret_cast<const f32x2 *>(ha);
                    const f32x2 *pb = reinterpret_cast<const f32x2 *>(ha + 32);
                    auto xa2 = [pa](int p) { return __ldg(pa + p); };
                    auto xb2 = [pb](int p) { return __ldg(pb + p); };
                    const float Xa = Hs[sl[t] * nIs + 8 * b + 2 * i];
                    const float Xb = Hs[sl[t] * nIs + 8 * b + 2 * i + 1];
                    y[t] += fp4  ? chunk_contrib_nvfp4_f32(hd, i, q0, q1, xa2, xb2)
                            : q5 ? chunk_contrib(sc, chunk_code_sums5(q0, q1, qh0, qh1, i, xa2, xb2), Xa, Xb)
                                 : chunk_contrib(sc, chunk_code_sums(q0, q1, xa2, xb2), Xa, Xb);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < SI_MAX_DECODE_TOKENS; ++t) {
            if (t < nt) {
                const float ys = (a.wtype == SI_WTYPE_NVFP4 ? a.wscale[3 * e + 2] : 1.f) * group_sum<GS>(y[t]);
                const int tk = u->tok[s][t];
                const float w = a.wts[sl[t]];
#pragma unroll
                for (int q = 0; q < SI_MAX_DECODE_TOKENS; ++q)
                    if (q == tk) acc[q] = fmaf(w, ys, acc[q]);
            }
        }
    }
    if (gl == 0 && c < a.H) {
#pragma unroll
        for (int t = 0; t < SI_MAX_DECODE_TOKENS; ++t)
            if (t < a.n)  // plus the residual x in a pre-normed block
                a.out[(size_t)t * a.H + c] = a.norm_w ? acc[t] + bf16_bits_to_f32(a.x[(size_t)t * a.H + c]) : acc[t];
    }
}

// --------------------------------------------------------------- launcher
static int pow2_at_least(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
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

// One CTA for up to 32 experts, else an 8-CTA cluster (portable size).
static int router_cluster_size(int E) { return E <= 32 ? 1 : 8; }

template <int NJ>
static cudaError_t launch_router_t(const DecodeArgs &a, cudaStream_t s) {
    const int C = router_cluster_size(a.E);
    const int wpc = (a.E + C - 1) / C;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(32 * wpc);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return a.norm_w ? cudaLaunchKernelEx(&cfg, k_router_topk<NJ, true>, a)
                    : cudaLaunchKernelEx(&cfg, k_router_topk<NJ, false>, a);
}

// Router + top-k of n <= 4 plain tokens for a cluster expert kernel, on an
// 8-CTA cluster, WPC experts per CTA (E == 8*WPC) and CPT columns per thread
// (H == 32*WPC*CPT).  Thread t of CTA c holds, in registers loaded before the
// dependency wait, the router weights of the CTA's WPC experts at columns
// CPT*t .. CPT*t+CPT-1, so that x is read once per CTA (CPT columns per
// thread and token, no shared copy) instead of once per expert.  For each
// token each thread forms WPC partial sums; a reduce-scatter across the warp's
// lanes (log2(WPC) halving shuffle steps) leaves each expert's warp sum in
// 32/WPC lanes, and the warps' sums are added in shared memory (fixed order).
// Then every CTA receives every logit by asynchronous stores, and each warp
// ranks its own expert for every token (descending logits, ties to the lower
// index) and stores it at its rank, with its logit, where it is selected; the
// expert kernel forms the renormalised weights from these.  Several tokens:
// each CTA also sends, for each token count c, the bits of its experts that c
// tokens chose to every CTA (a second asynchronous exchange), so that each
// selected expert's warp knows its index among the distinct experts and
// writes its entry of the table (expert, tokens that chose it with their
// ranks); CTA 0 writes their number.  The table lists the experts by token
// count, descending, then by id: the expert kernel's units of the experts
// several tokens chose take longest, and so start in its first wave.
// x is quantised for the expert kernel, which is launched at once.
template <int WPC, int CPT, int NT>
__global__ void __launch_bounds__(32 * WPC) k_router_one(DecodeArgs a) {
    // NT: 1 (one token) or SI_MAX_DECODE_TOKENS (n = 2..NT tokens)
    __shared__ float s_z[NT][SI_MAX_EXPERTS];
    __shared__ float s_part[NT][WPC][WPC];  // [token][warp][local expert]
    __shared__ __align__(8) uint64_t s_zbar;
    __shared__ __align__(8) uint64_t s_selbar;  // several tokens: every CTA's selection bits have arrived
    __shared__ uint32_t s_sel[8][NT];           // [CTA][c-1] bit w: the CTA's expert w was chosen by c tokens
    __shared__ uint32_t s_mysel[NT];
    const uint16_t *const xg_p = pin_ptr(a.x);
    float *const out_p = pin_ptr(a.out);
    const float *const bias_p = pin_ptr(a.router_bias);
    float *const ologits_p = pin_ptr(a.o_logits);
    int32_t *const ids_p = pin_ptr(a.ids);
    float *const wts_p = pin_ptr(a.wts);
    int32_t *const oids_p = pin_ptr(a.o_ids);
    int32_t *const counts_p = pin_ptr(a.counts);
    int32_t *const ocounts_p = pin_ptr(a.o_counts);
    uint32_t *const xq_p = pin_ptr(a.xq);
    const int H = pin_i32(a.H), E = pin_i32(a.E), k = pin_i32(a.k), n = NT == 1 ? 1 : pin_i32(a.n);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = (int)gridDim.x;
    const int e0 = blockIdx.x * WPC;  // this CTA's experts
    pdl_launch_dependents();  // the cluster expert kernel reads nothing of this call before its own wait
    float w[WPC][CPT];
#pragma unroll
    for (int q = 0; q < WPC; ++q) {
        const float *row = a.router_w + (size_t)(e0 + q) * H + CPT * threadIdx.x;
        if (CPT == 2) {
            const float2 v = __ldg(reinterpret_cast<const float2 *>(row));
            w[q][0] = v.x, w[q][1] = v.y;
        } else {
#pragma unroll
            for (int c4 = 0; c4 < CPT / 4; ++c4) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(row) + c4);
                w[q][4 * c4] = v.x, w[q][4 * c4 + 1] = v.y, w[q][4 * c4 + 2] = v.z, w[q][4 * c4 + 3] = v.w;
            }
        }
    }
#pragma unroll
    for (int q = 0; q < WPC; ++q)  // the weights are in registers before the wait, not fetched after it
#pragma unroll
        for (int c = 0; c < CPT; ++c) asm volatile("" ::"f"(w[q][c]));
    if (blockIdx.x == 0 && threadIdx.x < (n * H * 2) / 128)
        prefetch_l2(reinterpret_cast<const uint8_t *>(xg_p) + 128 * threadIdx.x);
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&s_zbar), 1);
        if (NT > 1) mbar_init(smem_addr(&s_selbar), 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(smem_addr(&s_zbar), (uint32_t)(n * E * 4));  // every logit, once
        if (NT > 1) mbar_arrive_expect_tx(smem_addr(&s_selbar), (uint32_t)(C * NT * 4));
        for (int c = 0; c < NT; ++c) s_mysel[c] = 0;
    }
    __syncthreads();
    cluster_arrive_relaxed();
    pdl_wait();  // x and the scratch are ready (previous kernels complete)
    // the chunk of x this warp quantises for the expert kernel (at most one: n*H/64 <= 8*WPC), loaded
    // together with the columns of the dot products
    const int NC = H / 64;
    const int qc = blockIdx.x + C * warp;
    const uint32_t qword = qc < n * NC ? __ldg(reinterpret_cast<const uint32_t *>(xg_p) + 32 * qc + lane) : 0u;
    uint32_t xw[NT][CPT / 2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (t < n) {
            const uint16_t *xp = xg_p + (size_t)t * H + CPT * threadIdx.x;
            if (CPT == 2) xw[t][0] = __ldg(reinterpret_cast<const uint32_t *>(xp));
            else if (CPT == 4) {
                const uint2 v = __ldg(reinterpret_cast<const uint2 *>(xp));
                xw[t][0] = v.x, xw[t][1 % (CPT / 2)] = v.y;
            } else {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xp));
                xw[t][0] = v.x, xw[t][1 % (CPT / 2)] = v.y, xw[t][2 % (CPT / 2)] = v.z, xw[t][3 % (CPT / 2)] = v.w;
            }
        }
    }
    for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < n * H; q += C * blockDim.x) out_p[q] = 0.f;  // the combine accumulates
    constexpr int kGroup = 32 / WPC;  // lanes that share one expert after the halving steps
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (t < n) {
            float xf[CPT];
#pragma unroll
            for (int c = 0; c < CPT / 2; ++c) {
                xf[2 * c] = __uint_as_float(xw[t][c] << 16);
                xf[2 * c + 1] = __uint_as_float(xw[t][c] & 0xffff0000u);
            }
            float v[WPC];
#pragma unroll
            for (int q = 0; q < WPC; ++q) {
                float acc = w[q][0] * xf[0];
#pragma unroll
                for (int c = 1; c < CPT; ++c) acc = fmaf(w[q][c], xf[c], acc);
                v[q] = acc;
            }
            // reduce-scatter across the lanes: step s halves the experts a lane keeps
#pragma unroll
            for (int s = 0; (1 << s) < WPC; ++s) {
                const int half = WPC >> (s + 1), mask = 16 >> s;
                const bool up = (lane & mask) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float keep = up ? v[i + half] : v[i], send = up ? v[i] : v[i + half];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                }
            }
#pragma unroll
            for (int m = kGroup / 2; m > 0; m >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
            if (lane % kGroup == 0) s_part[t][warp][lane / kGroup] = v[0];
        }
    }
    __syncthreads();
    cluster_wait();  // every CTA's mbarrier is initialised (all arrived long ago)
    const int e = e0 + warp;
#pragma unroll
    for (int t = 0; t < NT; ++t) {  // warp q: the logits of expert e0 + q, the sums of the WPC warps' partials
        if (t < n) {
            float z = lane < WPC ? s_part[t][lane][warp] : 0.f;
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) z += __shfl_xor_sync(0xffffffffu, z, m);
            if (bias_p) z += __ldg(bias_p + e);
            if (lane < C) st_async_cluster_u32(&s_z[t][e], smem_addr(&s_zbar), (uint32_t)lane, __float_as_uint(z));
            if (lane == 0 && ologits_p) ologits_p[t * E + e] = z;
        }
    }
    // x quantised per 64-column chunk for the expert kernel (token t at word t * NC * kXqWords); the
    // first chunk of each warp was loaded above, further ones (n*H/64 > 8*WPC) are loaded here
    for (int c = qc; c < n * NC; c += C * WPC) {
        const int t = c / NC, cc = c - t * NC;
        const uint32_t wv = c == qc ? qword : __ldg(reinterpret_cast<const uint32_t *>(xg_p) + 32 * c + lane);
        router_quant_chunk(wv, cc, NC, xq_p + (size_t)t * NC * kXqWords, lane, pin_i32(a.act8) != 0);
    }
    if (!mbar_wait_warp_cluster(smem_addr(&s_zbar), 0, a.wait_budget)) set_status(a.ctrl + kCtrlStatus, SI_ERR_TIMEOUT);
    // warp q ranks expert e0 + q against all E logits of each token (greater, or equal
    // with a lower index, beats it) and stores it at its rank where it is selected
    int chosen = 0;
    int rk[NT];  // this expert's rank for each token
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        rk[t] = k;
        if (t < n) {
            const float ze = s_z[t][e];
            int cnt = 0;
#pragma unroll
            for (int q = 0; q < SI_MAX_EXPERTS / 32; ++q) {
                const int j = lane + 32 * q;
                if (j < E) {
                    const float zj = s_z[t][j];
                    cnt += (zj > ze) | ((zj == ze) & (j < e));
                }
            }
            const int r = __reduce_add_sync(0xffffffffu, cnt);
            rk[t] = r;
            if (r < k) {
                ++chosen;
                if (lane == 0) {
                    ids_p[t * k + r] = e;
                    wts_p[t * k + r] = ze;  // the expert kernel turns these into renormalised weights
                    if (oids_p) oids_p[t * k + r] = e;
                }
            }
        }
    }
    if (lane == 0) {
        counts_p[e] = chosen;
        if (ocounts_p) ocounts_p[e] = chosen;
    }
    if (NT > 1) {  // the table of distinct experts
        if (lane == 0 && chosen) atomicOr(&s_mysel[chosen - 1], 1u << warp);
        __syncthreads();
        if (warp == 0 && lane < C)
#pragma unroll
            for (int c = 0; c < NT; ++c)
                st_async_cluster_u32(&s_sel[blockIdx.x][c], smem_addr(&s_selbar), (uint32_t)lane, s_mysel[c]);
        // every warp waits (the CTA may leave only once every peer's store has landed)
        if (!mbar_wait_warp_cluster(smem_addr(&s_selbar), 0, a.wait_budget)) {
            set_status(a.ctrl + kCtrlStatus, SI_ERR_TIMEOUT);
            return;
        }
        // index: experts chosen by more tokens, then those chosen as often with a smaller id
        int U = 0, below = 0;
        for (int cta = 0; cta < C; ++cta) {
#pragma unroll
            for (int c = 0; c < NT; ++c) {
                const int pc = __popc(s_sel[cta][c]);
                U += pc;
                below += (c + 1 > chosen || (c + 1 == chosen && cta < (int)blockIdx.x)) ? pc : 0;
            }
        }
        if (chosen) below += __popc(s_sel[blockIdx.x][chosen - 1] & ((1u << warp) - 1u));
        if (chosen && lane == 0) {
            UniqTable *u = a.uniq;
            u->expert[below] = e;
            u->ntok[below] = chosen;
            int j = 0;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (t < n && rk[t] < k) {
                    u->tok[below][j] = t;
                    u->slot[below][j] = rk[t];
                    ++j;
                }
            }
        }
        if (blockIdx.x == 0 && threadIdx.x == 0) a.ctrl[kCtrlNumUnique] = U;
    }
}

template <int WPC, int CPT>
static cudaError_t launch_router_one(const DecodeArgs &a, cudaStream_t s) {
    auto kern = a.n == 1 ? k_router_one<WPC, CPT, 1> : k_router_one<WPC, CPT, SI_MAX_DECODE_TOKENS>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(8);
    cfg.blockDim = dim3(32 * WPC);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 8;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Shapes the column-split router takes (E = 8 * WPC experts, H = 32 * WPC * CPT).
bool router_one_shape(int E, int H) {
    return (E == 128 && (H == 2048 || H == 1024)) || (E == 64 && (H == 2048 || H == 1024));
}

static cudaError_t launch_router(const DecodeArgs &a, cudaStream_t s) {
    // plain tokens for a cluster expert kernel: the column-split router
    if ((a.sel_logits || a.cl_mt) && !a.norm_w && router_one_shape(a.E, a.H)) {
        const int wpc = a.E / 8;
        if (wpc == 16 && a.H == 512 * 4) return launch_router_one<16, 4>(a, s);
        if (wpc == 16 && a.H == 512 * 2) return launch_router_one<16, 2>(a, s);
        if (wpc == 8 && a.H == 256 * 8) return launch_router_one<8, 8>(a, s);
        if (wpc == 8 && a.H == 256 * 4) return launch_router_one<8, 4>(a, s);
    }
    // register prefetch of the router rows: 2*NJ float4 per lane; with 1024
    // threads per CTA (E > 128) keep the register footprint small instead
    if ((a.E + router_cluster_size(a.E) - 1) / router_cluster_size(a.E) > 16) return launch_router_t<0>(a, s);
    switch (a.H / kQK) {
        case 1: return launch_router_t<1>(a, s);
        case 2: return launch_router_t<2>(a, s);
        case 3: return launch_router_t<3>(a, s);
        case 4: return launch_router_t<4>(a, s);
        case 5: return launch_router_t<5>(a, s);
        case 6: return launch_router_t<6>(a, s);
        case 7: return launch_router_t<7>(a, s);
        case 8: return launch_router_t<8>(a, s);
        default: return launch_router_t<0>(a, s);
    }
}

cudaError_t launch_decode(const Plan &p, const DecodeArgs &a_in, cudaStream_t s,
                          cudaEvent_t const *events) {
    DecodeArgs a = a_in;
    a.wait_budget = p.wait_budget;
    a.fault_wait = p.fault_wait ? 1 : 0;
    const bool cluster =
        a.n == 1 && p.cluster_ok && expert_cluster_layout(p.desc, p.cluster_size, p.smem_optin, a);
    // 2..4 tokens of a plain block: the cluster kernel over the distinct experts
    // (its table of distinct experts is formed from the column-split router's ranked ids)
    const bool mt = a.n > 1 && p.cluster_mt_ok && !a.norm_w && router_one_shape(a.E, a.H) && a.n * a.k <= 32 &&
                    expert_cluster_layout(p.desc, p.cluster_mt_size, p.smem_optin, a, a.n);
    a.cl_mt = mt ? 1 : 0;
    a.cl_active = p.cluster_mt_active;
    a.zero_out = cluster || mt ? 1 : 0;
    a.sel_logits = cluster ? 1 : 0;
    a.act8 = cluster && (p.desc.flags & SI_FLAG_ACT_INT8) ? 1 : 0;  // the other decode paths keep their precision
    cudaError_t err = mark(events, 0, s);
    if (err != cudaSuccess) return err;
    err = launch_router(a, s);
    if (err != cudaSuccess) return err;
    if ((err = mark(events, 1, s)) != cudaSuccess) return err;

    if (cluster || mt) {
        err = launch_expert_cluster(a, s);
        if (err != cudaSuccess) return err;
        if ((err = mark(events, 2, s)) != cudaSuccess) return err;
        return mark(events, 3, s);
    }
    if (p.fused_ok[a.n] && expert_fused_layout(p.desc, a.n, p.sm_count, p.smem_optin, a)) {
        err = launch_expert_fused(a, p.sm_count, s);
        if (err != cudaSuccess) return err;
        if ((err = mark(events, 2, s)) != cudaSuccess) return err;
        return mark(events, 3, s);
    }

    const size_t gu_smem = (size_t)a.n * a.H * sizeof(float) + (size_t)a.n * (a.H / 32) * sizeof(float);
    if (gu_smem > 48 * 1024) {
        err = cudaFuncSetAttribute(k_gateup_generic, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gu_smem);
        if (err != cudaSuccess) return err;
    }
    const int slots = a.n * a.k;
    const int gu_blocks = (slots * a.I + kWarps - 1) / kWarps;
    k_gateup_generic<<<gu_blocks, kThreads, gu_smem, s>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if ((err = mark(events, 2, s)) != cudaSuccess) return err;

    const size_t dn_smem = (size_t)slots * (a.I / 32) * sizeof(float);
    const int gs = pow2_at_least(4 * (a.I / kQK) < 32 ? 4 * (a.I / kQK) : 32);
    const int rows_per_block = kWarps * (32 / gs);
    const int dn_blocks = (a.H + rows_per_block - 1) / rows_per_block;
    switch (gs) {
        case 4: k_down_generic<4><<<dn_blocks, kThreads, dn_smem, s>>>(a); break;
        case 8: k_down_generic<8><<<dn_blocks, kThreads, dn_smem, s>>>(a); break;
        case 16: k_down_generic<16><<<dn_blocks, kThreads, dn_smem, s>>>(a); break;
        default: k_down_generic<32><<<dn_blocks, kThreads, dn_smem, s>>>(a); break;
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    return mark(events, 3, s);
}

}  // namespace si
