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
constexpr int kBlockBytes = 144;  // bytes per super-block (Q4_K, NVFP4)
// Q5_K (GGUF's K-quant with 5-bit codes): 176 bytes per 256 weights -- d,
// dmin and the 12 scale/min bytes as in Q4_K (bytes 0-15), qh[32] (bytes
// 16-47: bit j of qh[l] is the value-16 bit of weight l of sub-block j) and
// qs[128] (bytes 48-175, arranged as Q4_K's).
constexpr int kQ5BlockBytes = 176;
constexpr int kQ5QhOff = 16, kQ5QsOff = 48;

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

// RMSNorm scale of a row of H values from its sum of squares:
// 1 / sqrt(sumsq / H + eps) (IEEE square root and division).
__device__ __forceinline__ float rms_scale(float sumsq, int H, float eps) {
    return 1.0f / sqrtf(sumsq / (float)H + eps);
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

// Q5_K: the 5-bit codes of sub-blocks 2i (lo) and 2i+1 (hi) for the four
// weights of word t of a chunk's qs (w) and qh (qhw) bytes, one code per byte.
__device__ __forceinline__ uint32_t q5_codes_lo(uint32_t w, uint32_t qhw, int i) {
    return (w & 0x0f0f0f0fu) | (((qhw >> (2 * i)) & 0x01010101u) << 4);
}
__device__ __forceinline__ uint32_t q5_codes_hi(uint32_t w, uint32_t qhw, int i) {
    return ((w >> 4) & 0x0f0f0f0fu) | (((qhw >> (2 * i + 1)) & 0x01010101u) << 4);
}

// chunk_code_sums for Q5_K codes (qh0, qh1: the block's 32 qh bytes).
template <typename XA, typename XB>
__device__ __forceinline__ ChunkSums chunk_code_sums5(const uint4 &q0, const uint4 &q1, const uint4 &qh0,
                                                      const uint4 &qh1, int i, XA xa2, XB xb2) {
    f32x2 acc_a = 0ull, acc_b = 0ull;
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t h[8] = {qh0.x, qh0.y, qh0.z, qh0.w, qh1.x, qh1.y, qh1.z, qh1.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t lo = q5_codes_lo(w[t], h[t], i), hi = q5_codes_hi(w[t], h[t], i);
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

// L2 policy for small data every CTA reads (keep it in L2).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
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

// A value passed through a register move the compiler may neither move nor
// re-derive: pins a kernel-parameter read to this point of the program.  A
// graph launch's parameter buffer is not in the constant caches when the
// kernel starts, so parameters needed after the dependency wait are read
// before it, where the miss overlaps the wait.
__device__ __forceinline__ uint64_t pin_u64(uint64_t v) {
    uint64_t r;
    asm volatile("mov.b64 %0, %1;" : "=l"(r) : "l"(v));
    return r;
}
__device__ __forceinline__ int pin_i32(int v) {
    int r;
    asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v));
    return r;
}
template <typename T>
__device__ __forceinline__ T *pin_ptr(T *p) {
    return reinterpret_cast<T *>(pin_u64(reinterpret_cast<uint64_t>(p)));
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

// The same wait without sleeping between polls (for a thread on the critical
// path, e.g. the one issuing tensor-core MMAs); the clock is read every 64
// polls.
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity, long long budget) {
    const long long t0 = clock64();
    for (int n = 0;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63) == 63 && clock64() - t0 > budget) return false;
    }
}

// The same wait for a whole warp: every lane polls, so that each lane's own
// try_wait is the acquire of the copied bytes (one instruction for the warp;
// letting lane 0 poll alone and then repeating the wait on every lane
// measured slower).  Warp-uniform result.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, long long budget) {
    const bool ok = mbar_wait_bounded(bar, parity, budget);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Fault-injection wait (test mode only): wait for `*flag != 0` -- a word
// nothing writes -- for at most `budget` cycles; returns false when the wait
// runs out, which it always does.
__device__ __forceinline__ bool wait_flag_bounded(const int32_t *flag, long long budget) {
    const long long t0 = clock64();
    while (ld_acquire_gpu(flag) == 0) {
        if (clock64() - t0 > budget) return false;
        __nanosleep(32);
    }
    return true;
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

// =====================================================================
// Thread-block clusters: distributed shared memory and the cluster barrier.
// =====================================================================
namespace si {

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Store v into shared memory of CTA `rank` of this cluster, at the address that
// `local` has in this CTA.
__device__ __forceinline__ void st_cluster_f32(const void *local, uint32_t rank, float v) {
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(raddr), "f"(v) : "memory");
}
// Store the 32-bit v into shared memory of CTA `rank` of this cluster, at the
// address that `local` has in this CTA, and count its 4 bytes against the
// transaction count of that CTA's mbarrier at the address `bar` has here.  A
// thread that sees the barrier's phase complete also sees the stored value.
__device__ __forceinline__ void st_async_cluster_u32(const void *local, uint32_t bar, uint32_t rank, uint32_t v) {
    uint32_t raddr, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(bar), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr), "r"(v),
                 "r"(rbar)
                 : "memory");
}
// Split cluster barrier: every thread of every CTA of the cluster arrives
// (relaxed: order earlier writes with a fence first, e.g. fence_mbar_init)
// and later waits (acquire).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// All threads of all CTAs of the cluster; release/acquire orders DSMEM stores.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address in the cluster window of the shared-memory word that has address
// `local` in this CTA, as seen in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
// Arrive (release at cluster scope) on an mbarrier given by its cluster-window
// address, in this CTA or another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// try_wait with acquire at cluster scope: for phases completed by arrivals of
// other CTAs of the cluster.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_spin_cluster(uint32_t bar, uint32_t parity, long long budget) {
    const long long t0 = clock64();
    for (int n = 0;; ++n) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((n & 63) == 63 && clock64() - t0 > budget) return false;
    }
}
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity, long long budget) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (clock64() - t0 > budget) return false;
        __nanosleep(20);
    }
}
// Whole warp, no sleep between polls (each try_wait already suspends the
// thread for a while in hardware): for waits on the critical path of a
// pipeline, where a sleep granule would show up as a bubble.
__device__ __forceinline__ bool mbar_wait_warp_spin(uint32_t bar, uint32_t parity, long long budget) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_spin(bar, parity, budget);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) ok = mbar_wait_spin(bar, parity, budget);
    return __all_sync(0xffffffffu, ok);
}
// Every lane of the warp waits (bounded, sleeping between polls) with
// cluster-scope acquire: for barriers completed by other CTAs' st.async.
__device__ __forceinline__ bool mbar_wait_warp_cluster(uint32_t bar, uint32_t parity, long long budget) {
    bool ok = mbar_try_wait_cluster(bar, parity);
    if (!ok) {
        const long long t0 = clock64();
        while (!(ok = mbar_try_wait_cluster(bar, parity)) && clock64() - t0 <= budget) __nanosleep(20);
    }
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool mbar_wait_warp_spin_cluster(uint32_t bar, uint32_t parity, long long budget) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_spin_cluster(bar, parity, budget);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) ok = mbar_wait_spin_cluster(bar, parity, budget);
    return __all_sync(0xffffffffu, ok);
}

}  // namespace si

// =====================================================================
// int16-activation chunk dot products (dp2a).
//
// A chunk is 64 consecutive input columns: sub-blocks 2i (a) and 2i+1 (b) of
// one Q4_K block.  Its activations are held as 32 words of signed 16-bit
// pairs (word p = columns 2p | 2p+1 << 16), xq = rint(x / s) with
// s = max|x| / 32767 over the chunk, so |xq| <= 32767 and the quantisation
// error is at most s/2 per column (relative ~1.5e-5 of the chunk's largest
// activation).  Dot products with the 4-bit codes are then exact int32 sums
// (dp2a: two 16x8-bit products per instruction); the sub-block sums of the
// unquantised activations, X_a and X_b, carry the min term exactly:
//   sum_l w_l x_l ~= d*s*(sc_a*I_a + sc_b*I_b) - dmin*(m_a*X_a + m_b*X_b)
// with I = sum q*xq.  Bounds: |I| <= 32*15*32767 < 2^24 and
// |sc_a*I_a + sc_b*I_b| <= 2*63*15728160 < 2^31.
// (The pages' decode kernels use "on-read dp4a MMVQ" with 8-bit
// activations; 16-bit activations keep the error far below the tolerance.)
// =====================================================================
namespace si {

__device__ __forceinline__ int dp2a_lo(uint32_t xpair, uint32_t bytes, int acc) {
    asm("dp2a.lo.s32.u32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xpair), "r"(bytes));
    return acc;
}
__device__ __forceinline__ int dp2a_hi(uint32_t xpair, uint32_t bytes, int acc) {
    asm("dp2a.hi.s32.u32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xpair), "r"(bytes));
    return acc;
}

// round(a*inv) and round(b*inv) (|.| <= 32767) as one word of int16 pairs:
// adding 1.5*2^23 puts the rounded integer in the low mantissa bits
// (round-to-nearest-even by the addition), two's complement included.
__device__ __forceinline__ uint32_t pack_q16(float a, float b, float inv) {
    const uint32_t ua = __float_as_uint(fmaf(a, inv, 12582912.0f));
    const uint32_t ub = __float_as_uint(fmaf(b, inv, 12582912.0f));
    return __byte_perm(ua, ub, 0x5410);
}

// Quantise 64 activations (pairs) into 32 int16-pair words; returns the scale.
__device__ __forceinline__ float quantize64(const float (&x)[64], uint32_t (&w)[32], float &Xa, float &Xb) {
    // max |x| and the two sub-block sums as balanced trees (short dependency chains)
    float m[32], sa[16], sb[16];
#pragma unroll
    for (int l = 0; l < 32; ++l) m[l] = fmaxf(fabsf(x[2 * l]), fabsf(x[2 * l + 1]));
#pragma unroll
    for (int l = 0; l < 16; ++l) {
        sa[l] = x[2 * l] + x[2 * l + 1];
        sb[l] = x[32 + 2 * l] + x[32 + 2 * l + 1];
    }
#pragma unroll
    for (int w2 = 16; w2 >= 1; w2 >>= 1) {
#pragma unroll
        for (int l = 0; l < w2; ++l) m[l] = fmaxf(m[l], m[l + w2]);
    }
#pragma unroll
    for (int w2 = 8; w2 >= 1; w2 >>= 1) {
#pragma unroll
        for (int l = 0; l < w2; ++l) {
            sa[l] += sa[l + w2];
            sb[l] += sb[l + w2];
        }
    }
    const float mx = m[0];
    Xa = sa[0];
    Xb = sb[0];
    const float inv = mx > 0.f ? 32767.0f / mx : 0.f;
#pragma unroll
    for (int p = 0; p < 32; ++p) w[p] = pack_q16(x[2 * p], x[2 * p + 1], inv);
    return mx * (1.0f / 32767.0f);
}

// I_a = sum_l q_lo(l)*xq[l], I_b = sum_l q_hi(l)*xq[32+l] over one 32-byte
// chunk (q0, q1); xw(p) returns activation word p (p < 32).
template <typename XW>
__device__ __forceinline__ int2 chunk_isums(const uint4 &q0, const uint4 &q1, XW xw) {
    int a0 = 0, a1 = 0, b0 = 0, b1 = 0;
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t lo = w[t] & 0x0f0f0f0fu;  // codes of sub-block a, weights 4t..4t+3
        const uint32_t hi = w[t] & 0xf0f0f0f0u;  // 16 x codes of sub-block b
        a0 = dp2a_lo(xw(2 * t), lo, a0);
        a1 = dp2a_hi(xw(2 * t + 1), lo, a1);
        b0 = dp2a_lo(xw(16 + 2 * t), hi, b0);
        b1 = dp2a_hi(xw(16 + 2 * t + 1), hi, b1);
    }
    return make_int2(a0 + a1, (b0 + b1) >> 4);  // b sums are exact multiples of 16
}

// chunk_isums for Q5_K codes (qh0, qh1: the block's 32 qh bytes; i the chunk).
template <typename XW>
__device__ __forceinline__ int2 chunk_isums5(const uint4 &q0, const uint4 &q1, const uint4 &qh0, const uint4 &qh1,
                                            int i, XW xw) {
    int a0 = 0, a1 = 0, b0 = 0, b1 = 0;
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t h[8] = {qh0.x, qh0.y, qh0.z, qh0.w, qh1.x, qh1.y, qh1.z, qh1.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t lo = q5_codes_lo(w[t], h[t], i), hi = q5_codes_hi(w[t], h[t], i);
        a0 = dp2a_lo(xw(2 * t), lo, a0);
        a1 = dp2a_hi(xw(2 * t + 1), lo, a1);
        b0 = dp2a_lo(xw(16 + 2 * t), hi, b0);
        b1 = dp2a_hi(xw(16 + 2 * t + 1), hi, b1);
    }
    return make_int2(a0 + a1, b0 + b1);
}

struct ChunkScalesI {
    float d, dmin;
    int sca, scb, ma, mb;
};

// Scales and mins of sub-blocks 2i and 2i+1 without branching on i (i varies
// across the lanes of a warp).  The pair's bytes sit at bit offset 16*(i&1):
//   i < 2 : sc = bytes of scales[0..3] & 63,  m = bytes of scales[4..7] & 63
//   i >= 2: sc = (scales[8..11] & 15) | (top 2 bits of scales[0..3]) << 4
//           m  = (scales[8..11] >> 4) | (top 2 bits of scales[4..7]) << 4
__device__ __forceinline__ ChunkScalesI chunk_scales_i(const uint4 &hdr, int i) {
    ChunkScalesI s;
    s.d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
    s.dmin = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
    const int sh = 16 * (i & 1);
    const bool low = i < 2;
    const uint32_t Y = hdr.y >> sh, Z = hdr.z >> sh, W = hdr.w >> sh;
    const uint32_t hiY = (Y >> 2) & 0x3030u, hiZ = (Z >> 2) & 0x3030u;
    const uint32_t scp = low ? (Y & 0x3f3fu) : ((W & 0x0f0fu) | hiY);
    const uint32_t mp = low ? (Z & 0x3f3fu) : (((W >> 4) & 0x0f0fu) | hiZ);
    s.sca = scp & 0xffu;
    s.scb = (scp >> 8) & 0xffu;
    s.ma = mp & 0xffu;
    s.mb = (mp >> 8) & 0xffu;
    return s;
}

// int8-activation mode.  Unsigned bytes (a) times signed bytes (b), summed into c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// I_a = sum_l q_lo(l)*xa[l], I_b = sum_l q_hi(l)*xb[l] over one 32-byte chunk
// (q0, q1) against int8 activations: xw(t) holds columns 4t..4t+3 of
// sub-block a (t < 8) and of sub-block b (t >= 8, columns 32+4(t-8)..).
template <typename XW>
__device__ __forceinline__ int2 chunk_isums8(const uint4 &q0, const uint4 &q1, XW xw) {
    int a0 = 0, a1 = 0, b0 = 0, b1 = 0;
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int t = 0; t < 8; t += 2) {
        a0 = dp4a_us(w[t] & 0x0f0f0f0fu, xw(t), a0);
        b0 = dp4a_us(w[t] & 0xf0f0f0f0u, xw(8 + t), b0);  // 16 x the codes of sub-block b
        a1 = dp4a_us(w[t + 1] & 0x0f0f0f0fu, xw(t + 1), a1);
        b1 = dp4a_us(w[t + 1] & 0xf0f0f0f0u, xw(9 + t), b1);
    }
    return make_int2(a0 + a1, (b0 + b1) >> 4);  // b sums are exact multiples of 16
}

// d*(sc_a*da*I_a + sc_b*db*I_b) - dmin*(m_a*Xa + m_b*Xb): the scale term on the
// int8 activations (scales da, db), the min term on the exact sums Xa, Xb.
__device__ __forceinline__ float chunk_contrib_i8(const ChunkScalesI &c, int2 I, float da, float db, float Xa,
                                                  float Xb) {
    const float s = fmaf((float)c.sca * da, (float)I.x, (float)c.scb * db * (float)I.y);
    return fmaf(c.d, s, -c.dmin * fmaf((float)c.ma, Xa, (float)c.mb * Xb));
}

// One 64-column chunk held by a warp as lane pairs (lane l: columns 2l, 2l+1)
// quantised per 32 columns to int8: q = rint(v * 127/mx) (the product rounded
// once), scale mx * (1/127).  Returns this lane's two codes as the low 16 bits
// (column 2l in the low byte); on return lane 0 holds (scale, sum) of columns
// 0..31 and lane 16 of columns 32..63 in *d, *s.
__device__ __forceinline__ uint32_t quant_pair8(float v0, float v1, float *d, float *s) {
    float mx = fmaxf(fabsf(v0), fabsf(v1));
    float sum = v0 + v1;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {  // within each half of the warp (one 32-column block each)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    }
    const float inv = mx > 0.f ? 127.0f / mx : 0.f;
    const int q0 = (int)(__float_as_uint(fmaf(v0, inv, 12582912.0f)) & 0xffu);  // low byte of 1.5*2^23 + round(v*inv)
    const int q1 = (int)(__float_as_uint(fmaf(v1, inv, 12582912.0f)) & 0xffu);
    *d = mx * (1.0f / 127.0f);
    *s = sum;
    return (uint32_t)(q0 | (q1 << 8));
}

__device__ __forceinline__ float chunk_contrib_i(const ChunkScalesI &c, int2 I, float xs, float Xa, float Xb) {
    const int sc = c.sca * I.x + c.scb * I.y;
    const float mm = fmaf((float)c.ma, Xa, (float)c.mb * Xb);
    return fmaf(c.d * xs, (float)sc, -c.dmin * mm);
}

// =====================================================================
// NVFP4 super-blocks (144 bytes per 256 weights): bytes 0-15 the FP8 E4M3
// scales of weights 16j .. 16j+15, bytes 16-143 the E2M1 codes (byte 16 + l:
// weight 2l in its low nibble, 2l+1 in its high nibble); weight = e2m1 *
// e4m3 * g, g the matrix's fp32 tensor scale.  E2M1 code c: bit 3 sign,
// bits 2-1 exponent (bias 1), bit 0 mantissa: magnitudes 0, 0.5, 1, 1.5, 2,
// 3, 4, 6.  (sparkinfer README, "Milestone 2": NVFP4 experts; the CuTe-DSL
// README's moe row: W4A16, bf16 activations with inline FP4 weight dequant.)
// The GEMV takes each code through the integer T(c) = 12 + 2*e2m1(c) in
// [0, 24] and the same int16 activations as the Q4_K path:
//   sum_l e2m1_l x_l ~= s/2 * (sum_l T_l xq_l - 12 * sum_l xq_l)
// per 16-weight block, exact in int32; the block's E4M3 scale, the
// activation scale s and the tensor scale multiply the block sums.
// =====================================================================
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// T of the four codes in the low 16 bits of `codes` (code k -> byte k).  A
// byte permute selects from an 8-entry table by the low three bits of each
// code; with the code's bit 3 set it returns the sign of the selected byte
// instead (0: every entry is below 128).  So one permute gives T for the
// positive codes and 0 for the negative ones, the other (bit 3 flipped) the
// reverse, and the two are or-ed.
__device__ __forceinline__ uint32_t e2m1_t4(uint32_t codes) {
    // positive codes m = 0..7: 12 + 2*{0, .5, 1, 1.5, 2, 3, 4, 6}; negative: 12 - 2*...
    return prmt(0x0F0E0D0Cu, 0x18141210u, codes) | prmt(0x090A0B0Cu, 0x00040608u, codes ^ 0x8888u);
}

// FP8 E4M3 byte (bit 7 sign, bits 6-3 exponent E with bias 7, bits 2-0
// mantissa M) -> fp32, exactly: E > 0: 2^(E-7) * (1 + M/8); E == 0: M * 2^-9.
// (S.1111.111 is NaN in E4M3; block scales never hold it.)
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const uint32_t E = (b >> 3) & 15u, M = b & 7u;
    const float v = E ? __uint_as_float(((E + 120u) << 23) | (M << 20)) : (float)M * 0.001953125f;
    return __uint_as_float(__float_as_uint(v) | ((b & 0x80u) << 24));
}

// Integer sums of the int16 activations of one 64-column chunk (32 words)
// over its four 16-column blocks.
__device__ __forceinline__ void xq_block_sums(const uint32_t (&w)[32], int (&XQ)[4]) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        int s = 0;
#pragma unroll
        for (int p = 8 * b; p < 8 * b + 8; ++p) s += (int)(int16_t)(w[p] & 0xffffu) + ((int)w[p] >> 16);
        XQ[b] = s;
    }
}

// Contribution of chunk i (64 weights: scale blocks 4i .. 4i+3, codes q0, q1)
// of an NVFP4 super-block with header hdr (its 16 scale bytes) to a row dot
// product with int16 activations xw(p) of scale xs and block sums XQ, before
// the tensor scale.
template <typename XW>
__device__ __forceinline__ float chunk_contrib_nvfp4(const uint4 &hdr, int i, const uint4 &q0, const uint4 &q1, XW xw,
                                                     float xs, const int (&XQ)[4]) {
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    int blk[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        int a0 = 0, a1 = 0;
#pragma unroll
        for (int t = 2 * b; t < 2 * b + 2; ++t) {
            const uint32_t lo = e2m1_t4(w[t]), hi = e2m1_t4(w[t] >> 16);  // weights 8t..8t+3, 8t+4..8t+7
            a0 = dp2a_lo(xw(4 * t), lo, a0);
            a1 = dp2a_hi(xw(4 * t + 1), lo, a1);
            a0 = dp2a_lo(xw(4 * t + 2), hi, a0);
            a1 = dp2a_hi(xw(4 * t + 3), hi, a1);
        }
        blk[b] = a0 + a1 - 12 * XQ[b];
    }
    // the four scale bytes of this chunk are 32-bit word i of the header (i varies across lanes)
    const uint32_t sw = i == 0 ? hdr.x : (i == 1 ? hdr.y : (i == 2 ? hdr.z : hdr.w));
    float r = e4m3_to_f32(sw & 0xffu) * (float)blk[0];
    r = fmaf(e4m3_to_f32((sw >> 8) & 0xffu), (float)blk[1], r);
    r = fmaf(e4m3_to_f32((sw >> 16) & 0xffu), (float)blk[2], r);
    r = fmaf(e4m3_to_f32(sw >> 24), (float)blk[3], r);
    return 0.5f * xs * r;
}

// The same chunk with fp32 activations: xa2(p) = {x[2p], x[2p+1]} for the
// chunk's weights 0..31 and xb2(p) for 32..63 (p = 0..15); before the tensor
// scale.  (The generic kernels keep the activations in fp32.)
template <typename XA, typename XB>
__device__ __forceinline__ float chunk_contrib_nvfp4_f32(const uint4 &hdr, int i, const uint4 &q0, const uint4 &q1,
                                                         XA xa2, XB xb2) {
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t sw = i == 0 ? hdr.x : (i == 1 ? hdr.y : (i == 2 ? hdr.z : hdr.w));
    float r = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float acc = 0.f;
#pragma unroll
        for (int t = 2 * b; t < 2 * b + 2; ++t) {
            const uint32_t v[2] = {e2m1_t4(w[t]), e2m1_t4(w[t] >> 16)};  // weights 8t..8t+3, 8t+4..8t+7
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                    const int p = 4 * t + 2 * hh + pr;  // activation pair of weights 2p, 2p+1 of the chunk
                    const f32x2 xp = p < 16 ? xa2(p) : xb2(p - 16);
                    const float2 x2 = unpack2(xp);
                    acc = fmaf((float)((int)((v[hh] >> (16 * pr)) & 0xffu) - 12), x2.x, acc);
                    acc = fmaf((float)((int)((v[hh] >> (16 * pr + 8)) & 0xffu) - 12), x2.y, acc);
                }
            }
        }
        r = fmaf(e4m3_to_f32((sw >> (8 * b)) & 0xffu), acc, r);
    }
    return 0.5f * r;
}

// Top-k of n rows of logits z[t][0..E) by ranks, using all threads of a CTA:
// the rank of z[t][e] is the number of logits that beat it (greater, or equal
// with a lower index); the experts of rank < k are the selection, stored at
// their rank (descending order, ties -> lower index).  ids/zsel are
// [n][SI_MAX_TOPK] in shared memory; zsel receives the selected logits.
// When the CTA has spare threads, tpi threads share one logit's comparisons
// and add their counts with shuffles.  Needs a __syncthreads before (z
// complete) and after (results complete).
__device__ __forceinline__ int rank_part(const float *zr, int E, int e, float ze, int j0, int step) {
    int rank = 0;
#pragma unroll 4
    for (int j = j0; j < E; j += step) {
        const float zj = zr[j];
        rank += (zj > ze) | ((zj == ze) & (j < e));
    }
    return rank;
}

__device__ __forceinline__ void cta_topk_ranks(const float (*z)[256], int n, int E, int k, int (*ids)[16],
                                               float (*zsel)[16]) {
    const int items = n * E;
    int tpi = 1;
    while (tpi < 32 && items * tpi * 2 <= (int)blockDim.x) tpi <<= 1;
    if (tpi == 1) {
        for (int q = threadIdx.x; q < items; q += blockDim.x) {
            const int t = q / E, e = q - t * E;
            const float ze = z[t][e];
            const int rank = rank_part(z[t], E, e, ze, 0, 1);
            if (rank < k) {
                ids[t][rank] = e;
                zsel[t][rank] = ze;
            }
        }
    } else {
        // one pass; every thread takes part in the shuffles (items * tpi <= blockDim)
        const int q = threadIdx.x;
        const int item = min(q / tpi, items - 1), part = q & (tpi - 1);
        const int t = item / E, e = item - t * E;
        const float ze = z[t][e];
        int rank = rank_part(z[t], E, e, ze, part, tpi);
        for (int o = tpi >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (q / tpi < items && part == 0 && rank < k) {
            ids[t][rank] = e;
            zsel[t][rank] = ze;
        }
    }
}

// Renormalised softmax weights of one token's selected logits (one warp):
// w_i = exp(z_i - z_0) / sum_j exp(z_j - z_0), z_0 the largest.  In place.
__device__ __forceinline__ void warp_renorm(float *zw, int k) {
    const int lane = threadIdx.x & 31;
    const float z0 = zw[0];
    const float ex = lane < k ? expf(zw[lane] - z0) : 0.f;
    float den = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    __syncwarp();
    if (lane < k) zw[lane] = ex / den;
    __syncwarp();
}

}  // namespace si

// =====================================================================
// Tiled TMA (tensor-map) loads and float reductions into global memory.
// =====================================================================
namespace si {

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// 2-D tiled tensor load of one box into shared memory (dst 128-byte aligned),
// completing bytes on mbarrier `bar`; x = innermost coordinate (elements).
__device__ __forceinline__ void prefetch_tensormap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// The same without an L2 cache hint.
__device__ __forceinline__ void tma_load_2d_plain(uint32_t dst, const void *tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void red_add_f32(float *p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

}  // namespace si
