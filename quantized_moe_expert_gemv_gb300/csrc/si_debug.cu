// si_debug.cu -- test exports: explicit Q4_K dequantization and stand-alone top-k.
//
// The dequant kernel writes every weight of the Q4_K blocks as the value the
// format defines, w = d*sc*q - dmin*m: d*sc and dmin*m are exact in fp32
// (at most 17 significant bits), d*sc*q is exact (at most 21 bits), so one
// fused multiply-add rounds the exact difference once.  The bf16 copy is the
// round-to-nearest-even of that fp32 value (the operand rounding the grouped
// prefill applies).
#include <cstdint>

#include "si_device.cuh"
#include "si_internal.h"

namespace si {

__global__ void __launch_bounds__(256) k_debug_dequant(const uint8_t *blocks, int64_t n_blocks,
                                                       float *out_f32, uint16_t *out_bf16) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (block, sub-block)
    if (gid >= n_blocks * 8) return;
    const int64_t blk_idx = gid >> 3;
    const int j = (int)(gid & 7);
    const uint8_t *blk = blocks + blk_idx * kBlockBytes;
    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
    const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
    int sc, m;
    unpack_sc_m(hdr, j, sc, m);
    const float dsc = d * (float)sc, dm = dmin * (float)m;
    const uint8_t *qs = blk + 16 + 32 * (j >> 1);
    const int shift = (j & 1) ? 4 : 0;
    const int64_t base = blk_idx * kQK + 32 * j;
    for (int l = 0; l < 32; ++l) {
        const int q = (qs[l] >> shift) & 15;
        const float w = fmaf(dsc, (float)q, -dm);
        if (out_f32) out_f32[base + l] = w;
        if (out_bf16) out_bf16[base + l] = __bfloat16_as_ushort(__float2bfloat16_rn(w));
    }
}

cudaError_t launch_debug_dequant(const uint8_t *blocks, int64_t n_blocks, float *out_f32,
                                 uint16_t *out_bf16, cudaStream_t s) {
    if (n_blocks <= 0) return cudaSuccess;
    const int64_t threads = n_blocks * 8;
    const int64_t grid = (threads + 255) / 256;
    k_debug_dequant<<<(unsigned)grid, 256, 0, s>>>(blocks, n_blocks, out_f32, out_bf16);
    return cudaGetLastError();
}

__global__ void __launch_bounds__(128) k_debug_topk(const float *logits, int n, int E, int k,
                                                    int32_t *ids, float *w, int32_t *counts) {
    __shared__ float s_z[SI_MAX_DECODE_TOKENS][SI_MAX_EXPERTS];
    __shared__ int s_ids[SI_MAX_DECODE_TOKENS][SI_MAX_TOPK];
    __shared__ float s_w[SI_MAX_DECODE_TOKENS][SI_MAX_TOPK];
    __shared__ int s_counts[SI_MAX_EXPERTS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < n * E; i += blockDim.x) s_z[i / E][i % E] = logits[i];
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_counts[i] = 0;
    __syncthreads();
    cta_topk_ranks(s_z, n, E, k, s_ids, s_w);
    __syncthreads();
    if (warp < n) {
        warp_renorm(s_w[warp], k);
        for (int i = lane; i < k; i += 32) {
            if (ids) ids[warp * k + i] = s_ids[warp][i];
            if (w) w[warp * k + i] = s_w[warp][i];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int t = 0; t < n; ++t)
            for (int i = 0; i < k; ++i) s_counts[s_ids[t][i]] += 1;
    __syncthreads();
    if (counts)
        for (int i = threadIdx.x; i < E; i += blockDim.x) counts[i] = s_counts[i];
}

cudaError_t launch_debug_topk(const float *logits, int n, int E, int k, int32_t *ids, float *w,
                              int32_t *counts, cudaStream_t s) {
    k_debug_topk<<<1, 128, 0, s>>>(logits, n, E, k, ids, w, counts);
    return cudaGetLastError();
}

}  // namespace si
