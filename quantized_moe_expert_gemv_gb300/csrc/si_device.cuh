// si_device.cuh -- device-side building blocks shared by the sm_103a kernels.
//
// Q4_K (GGUF) super-block: 144 bytes per 256 weights,
//   bytes 0-1 d (fp16), 2-3 dmin (fp16), 4-15 scales[12], 16-143 qs[128].
// Sub-block j (32 weights) has a 6-bit scale sc_j and min m_j:
//   j < 4 : sc = scales[j] & 63,                           m = scales[j+4] & 63
//   j >= 4: sc = (scales[j+4] & 15) | ((scales[j-4]>>6)<<4), m = (scales[j+4]>>4) | ((scales[j]>>6)<<4)
// qs is four 32-byte chunks; byte l of chunk i holds weight l of sub-block 2i
// in its low nibble and weight l of sub-block 2i+1 in its high nibble.
// Weight = d*sc*q - dmin*m.  (sparkinfer README, "Layout": "GGUF dequant",
// "fused quantized MoE expert FFN"; experts are "dequantized on-read".)
//
// The GEMV kernels never materialise a weight.  For one 32-byte chunk
// (sub-blocks a = 2i and b = 2i+1) against activations x they use
//   sum_l w_l x_l = d*sc_a*(S_a) + d*sc_b*(S_b) - dmin*(m_a*X_a + m_b*X_b)
// with S = sum q*x and X = sum x over the sub-block.  Each 4-bit code q is
// turned into the fp32 value 128 + q by placing it in the mantissa of 128.0
// (one byte permute, exact), so the loop accumulates F = sum (128+q)*x and
// S = F - 128*X.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace si {

constexpr int kQK = 256;          // weights per super-block
constexpr int kBlockBytes = 144;  // bytes per super-block

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// ------------------------------------------------------- packed fp32 pairs
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 unpack2(f32x2 v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
// acc += a * b on both lanes of the pair (one packed FMA, sm_100-family).
__device__ __forceinline__ void ffma2(f32x2 &acc, f32x2 a, f32x2 b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// 128 + q for the 4-bit code in byte `B` of a word whose bytes are < 16.
template <int B>
__device__ __forceinline__ float code_plus_128(uint32_t nibble_bytes) {
    // result bytes (hi..lo): 0x43, byte B of the word, 0x00, 0x00  ->  128 + q
    return __uint_as_float(__byte_perm(nibble_bytes, 0x43u, (4 << 12) | (B << 8) | (5 << 4) | 5));
}

// ------------------------------------------------------- scale/min unpack
struct SubScales {
    float dsc_a, dsc_b;   // d*sc for sub-blocks 2i and 2i+1 (exact in fp32)
    float dm_a, dm_b;     // dmin*m for the same (exact in fp32)
};

// hdr = the first 16 bytes of a block: {d|dmin<<16, scales[0..3], [4..7], [8..11]}
__device__ __forceinline__ void unpack_sc_m(const uint4 &hdr, int j, int &sc, int &m) {
    if (j < 4) {
        sc = (hdr.y >> (8 * j)) & 63;
        m = (hdr.z >> (8 * j)) & 63;
    } else {
        const int s = 8 * (j - 4);
        const uint32_t c = (hdr.w >> s) & 0xffu;       // scales[j+4]
        sc = (c & 15) | (((hdr.y >> (s + 6)) & 3) << 4);  // top bits of scales[j-4]
        m = (c >> 4) | (((hdr.z >> (s + 6)) & 3) << 4);   // top bits of scales[j]
    }
}

__device__ __forceinline__ SubScales chunk_scales(const uint4 &hdr, int i) {
    const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
    int sca, ma, scb, mb;
    unpack_sc_m(hdr, 2 * i, sca, ma);
    unpack_sc_m(hdr, 2 * i + 1, scb, mb);
    SubScales s;
    s.dsc_a = d * (float)sca;
    s.dsc_b = d * (float)scb;
    s.dm_a = dmin * (float)ma;
    s.dm_b = dmin * (float)mb;
    return s;
}

// F_a = sum_l (128 + q_lo(l)) * xa[l], F_b = sum_l (128 + q_hi(l)) * xb[l]
// over the 32 bytes of one chunk (q0, q1 = its two 16-byte halves).
// xa, xb: 32 activations each, as pairs (xa2[t] = {x[2t], x[2t+1]}).
struct ChunkSums {
    float Fa, Fb;
};

template <typename XA, typename XB>
__device__ __forceinline__ ChunkSums chunk_code_sums(const uint4 &q0, const uint4 &q1, XA xa2,
                                                     XB xb2) {
    f32x2 acc_a = 0ull, acc_b = 0ull;  // (+0.0f, +0.0f)
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t lo = w[t] & 0x0f0f0f0fu;
        const uint32_t hi = (w[t] >> 4) & 0x0f0f0f0fu;
        ffma2(acc_a, pack2(code_plus_128<0>(lo), code_plus_128<1>(lo)), xa2(2 * t));
        ffma2(acc_a, pack2(code_plus_128<2>(lo), code_plus_128<3>(lo)), xa2(2 * t + 1));
        ffma2(acc_b, pack2(code_plus_128<0>(hi), code_plus_128<1>(hi)), xb2(2 * t));
        ffma2(acc_b, pack2(code_plus_128<2>(hi), code_plus_128<3>(hi)), xb2(2 * t + 1));
    }
    const float2 a = unpack2(acc_a), b = unpack2(acc_b);
    return ChunkSums{a.x + a.y, b.x + b.y};
}

// Contribution of one chunk to a row dot product, given the code sums and
// the sub-block activation sums Xa, Xb.
__device__ __forceinline__ float chunk_contrib(const SubScales &s, const ChunkSums &f, float Xa,
                                               float Xb) {
    float r = s.dsc_a * (f.Fa - 128.0f * Xa);
    r = fmaf(s.dsc_b, f.Fb - 128.0f * Xb, r);
    r = fmaf(-s.dm_a, Xa, r);
    r = fmaf(-s.dm_b, Xb, r);
    return r;
}

// --------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int GS>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = GS / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// ------------------------------------------------------------------ top-k
// One warp selects the k largest of z[0..E) (E <= 256, k <= 16), descending,
// equal values -> lower index first, and the renormalised softmax weights
// w_i = exp(z_i - z_0) / sum_j exp(z_j - z_0) over the selected logits
// (equal to the full softmax renormalised over the selection).  All lanes
// return the same ids/weights.
__device__ __forceinline__ void warp_topk(const float *z, int E, int k, int *ids, float *wts) {
    const int lane = threadIdx.x & 31;
    float v[8];
    bool live[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int idx = lane + 32 * j;
        live[j] = idx < E;
        v[j] = live[j] ? z[idx] : 0.0f;
    }
    float zsel[16];
    for (int i = 0; i < k; ++i) {
        float bv = 0.0f;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int idx = lane + 32 * j;
            if (live[j] && (bi == 0x7fffffff || v[j] > bv)) {
                bv = v[j];
                bi = idx;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            const bool take = (oi != 0x7fffffff) &&
                              (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
            if (take) {
                bv = ov;
                bi = oi;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (lane + 32 * j == bi) live[j] = false;
        ids[i] = bi;
        zsel[i] = bv;
    }
    float denom = 0.0f;
    for (int i = 0; i < k; ++i) denom += expf(zsel[i] - zsel[0]);
    for (int i = 0; i < k; ++i) wts[i] = expf(zsel[i] - zsel[0]) / denom;
}

}  // namespace si

// =====================================================================
// Asynchronous copies, mbarriers, programmatic dependent launch, bounded
// waits (sm_90+ PTX, used on sm_103a).
// =====================================================================
namespace si {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// L2 policy for streamed expert weights: evict first, so one token's
// experts do not displace activations/router weights (and do not make a
// later token's reads look like HBM reads when they are L2 hits).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk global -> shared copy (TMA, non-tensor); completes `bytes` of the
// transaction count of mbarrier `bar`.  dst/src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Record the first device-side error of a call (0 = none).
__device__ __forceinline__ void set_status(int32_t *status, int code) { atomicCAS(status, 0, code); }

// Wait for phase `parity` of an mbarrier for at most `budget` SM cycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long budget) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > budget) return false;
        __nanosleep(20);
    }
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier over all CTAs of a launch whose CTAs are all resident
// (grid <= resident capacity).  ctr/gen are two words of the scratch control
// block: the last arriver resets the counter and bumps the generation.
// Called by every thread of the CTA; returns false (and records
// SI_ERR_TIMEOUT) if the other CTAs did not arrive within `budget` cycles.
__device__ __forceinline__ bool grid_barrier(int32_t *ctr, int32_t *gen, int32_t *status,
                                             long long budget) {
    __shared__ int s_ok;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int g0 = ld_acquire_gpu(gen);
        int ok = 1;
        if (atomicAdd(ctr, 1) == (int)gridDim.x - 1) {
            *ctr = 0;
            __threadfence();
            atomicAdd(gen, 1);
        } else {
            const long long t0 = clock64();
            while (ld_acquire_gpu(gen) == g0) {
                if (clock64() - t0 > budget) {
                    ok = 0;
                    set_status(status, 6 /* SI_ERR_TIMEOUT */);
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

}  // namespace si
