// si_noalloc.cu -- single-token/small-batch decode for callers that cannot
// allocate device memory.
//
// Some callers of this library have no way to call cudaMalloc: a plug-in
// running inside a host framework whose memory pool owns all device memory
// and hands it no allocator, or a latency-critical decode loop where an
// allocation would synchronise the device and stall the pipeline.  For them
// si_moe_forward_decode_noalloc runs the same decode kernels as
// si_moe_forward_decode, with the scratch taken from one fixed array below
// instead of a caller buffer.  The caller still passes weights, inputs and
// outputs.  The array is part of the module image: every GPU that loads this
// library holds SI_STATIC_SCRATCH_BYTES of it until the process exits.
#include <mutex>

#include "si_internal.h"

namespace {

// The scratch of every si_moe_forward_decode_noalloc call on a device.  Zero
// at module load; word 0 (the device status) keeps the first device-side
// error until si_moe_read_status_noalloc reads and clears it.
static __device__ __align__(256) unsigned char g_static_scratch[SI_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};  // device address of g_static_scratch, per device

// In host code g_static_scratch names a host-side stand-in, not device
// memory; the kernels need the device address, looked up once per device
// with that device current (the first call on the device).  A
// cudaDeviceReset destroys the module and with it this address: the entry
// points below are not usable on a device after it has been reset.
si_status scratch_address(void **addr) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    if (device < 0 || device >= kMaxDevices) return SI_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[device]) {
        void *p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, g_static_scratch);
        if (err != cudaSuccess || !p) {
            cudaGetLastError();
            return SI_ERR_CUDA;
        }
        g_scratch_addr[device] = p;
    }
    *addr = g_scratch_addr[device];
    return SI_OK;
}

}  // namespace

extern "C" si_status si_moe_forward_decode_noalloc(si_moe_plan_t plan, const si_moe_layer *layer,
                                                   const void *x_bf16, int32_t n_tokens, float *out,
                                                   si_moe_route_out *route_out, si_stream_t stream) {
    // every argument error is returned before anything touches the array
    const si_status chk = si::check_decode_args(plan, layer, x_bf16, n_tokens, out, route_out);
    if (chk != SI_OK) return chk;
    size_t need = 0;
    const si_status st = si_moe_scratch_bytes(plan, SI_MODE_DECODE, n_tokens, &need);
    if (st != SI_OK) return st;
    if (need > SI_STATIC_SCRATCH_BYTES) return SI_ERR_SCRATCH_TOO_SMALL;  // shape too large for the array
    void *scratch = nullptr;
    const si_status sa = scratch_address(&scratch);
    if (sa != SI_OK) return sa;
    // The array keeps the previous call's contents; the arrival counters of
    // the control block must start at zero, so clear them in stream order.
    // The status word (word 0) is left alone: it holds an earlier call's
    // device-side error until si_moe_read_status_noalloc reads it.
    if (cudaMemsetAsync(static_cast<unsigned char *>(scratch) + sizeof(int32_t), 0,
                        si::kCtrlBytes - sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return SI_ERR_CUDA;
    }
    return si_moe_forward_decode(plan, layer, x_bf16, n_tokens, out, route_out, scratch,
                                 SI_STATIC_SCRATCH_BYTES, stream);
}

extern "C" si_status si_moe_read_status_noalloc(si_stream_t stream) {
    void *scratch = nullptr;
    const si_status sa = scratch_address(&scratch);
    if (sa != SI_OK) return sa;
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
        if (cudaMemset(scratch, 0, sizeof(word)) != cudaSuccess) {
            cudaGetLastError();
            return SI_ERR_CUDA;
        }
        return (si_status)word;
    }
    return SI_OK;
}
