// tq_static.cu -- decode attention for callers that cannot allocate device
// memory.
//
// Some callers may not call cudaMalloc once they are running: serving loops
// that pre-reserve all device memory at start-up and forbid later allocation
// (cudaMalloc can synchronize the device and fragment a tightly budgeted
// pool), or hosts whose device memory belongs to another framework's
// allocator and that cannot hand out a workspace of their own.  For them,
// tq_decode_attention_static runs the same decode-attention kernels as
// tq_decode_attention, but its scratch (plan, rotated queries, split-K
// partials) lives in the fixed-size device array below.  With the CUDA
// runtime's default lazy module loading, a device commits the array's memory
// when this file's module is first loaded there, i.e. at the first static
// call (or static error-flag read) on that device; it then holds it until the
// process exits.
#include <mutex>

#include <cuda_runtime.h>

#include "tq_internal.h"

namespace {

// The scratch area: TQ_STATIC_WORKSPACE_BYTES bytes per device, 256-byte aligned.
static __device__ __align__(256) unsigned char g_static_workspace[TQ_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_addr[kMaxDevices] = {};

}  // namespace

// Device address of the array on the current device, looked up once per device.
// In host code `g_static_workspace` names a host-side stand-in, not device
// memory, so the address must come from cudaGetSymbolAddress with the device
// current.
tq_status tqk::static_workspace(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tqk::record_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess) return tqk::record_cuda_error(e);
        if (p == nullptr) return TQ_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return TQ_OK;
}

// tq_decode_attention checks q, out and their alignment first, then builds and
// validates the plan, and returns TQ_ERR_SIZE before uploading or launching
// anything when the plan needs more scratch than the array holds: the same
// error codes, in the same order, as a call with a caller workspace of
// TQ_STATIC_WORKSPACE_BYTES.
extern "C" tq_status tq_decode_attention_static(const tq_layer_view *layers, int n_layers, int batch,
                                                int n_heads, int q_heads, int head_dim, const float *qjl_S,
                                                int jl_dim, const void *q, float *out, void *stream) {
    if (!q || !out) return TQ_ERR_ARG;
    void *ws = nullptr;
    const tq_status st = tqk::static_workspace(&ws);
    if (st != TQ_OK) return st;
    return tq_decode_attention(layers, n_layers, batch, n_heads, q_heads, head_dim, qjl_S, jl_dim, q, out, ws,
                               static_cast<size_t>(TQ_STATIC_WORKSPACE_BYTES), stream);
}
