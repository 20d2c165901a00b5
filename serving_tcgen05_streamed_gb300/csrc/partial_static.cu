// partial_static.cu -- packed_kv_attention_partial with its carried state in
// a fixed area of device memory that the library owns, for callers that can
// allocate no device memory of their own.
//
// Some callers cannot call cudaMalloc: code that runs inside a host that owns
// all device memory (an inference server's or a framework's pool, a plugin
// slot with a fixed memory budget) and hands it no workspace, and code on a
// path where cudaMalloc is not allowed because it may synchronise the
// device.  For them this entry point keeps the key-chunk attention's state
// (o_acc and lse_acc) in the array below instead of in caller buffers; the
// caller still passes Q, the key chunk and the output.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace kvq {
namespace {

// The state area: KVQ_STATIC_STATE_BYTES of device memory, allocated when the
// library is loaded on a device and held until the process exits.  In host
// code the name stands for a host-side shadow, never for the device address:
// the address comes from cudaGetSymbolAddress below.
constexpr size_t kStateFloats = KVQ_STATIC_STATE_BYTES / sizeof(float);
__device__ __align__(256) float g_static_state[kStateFloats];

std::mutex g_state_mu;
void *g_state_ptr[64] = {nullptr};  // device address of g_static_state, per device

// Device address of the state area on the current device, resolved once per
// device (with that device current) on its first use.
int state_address(float **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_state_mu);
    if (!g_state_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_state);
        if (e != cudaSuccess || !p) return report_cuda(e == cudaSuccess ? cudaErrorInvalidSymbol : e, "state address");
        g_state_ptr[dev] = p;
    }
    *out = static_cast<float *>(g_state_ptr[dev]);
    return KVQ_OK;
}

}  // namespace
}  // namespace kvq

extern "C" int packed_kv_attention_partial_static(const void *q, int64_t n_q, const kvq_range *ranges, int n_ranges,
                                                  int hidden, int group, float sm_scale, int flags, int out_fp32,
                                                  void *out, kvq_stream_t stream) {
    using namespace kvq;
    if (n_q < 1 || hidden < 128 || hidden % 128) return KVQ_ERR_ARG;
    const uint64_t need = static_cast<uint64_t>(n_q) * static_cast<uint64_t>(hidden + hidden / 128) * sizeof(float);
    if (need > KVQ_STATIC_STATE_BYTES) return KVQ_ERR_TOO_LARGE;
    float *base = nullptr;
    const int st = state_address(&base);
    if (st) return st;
    // o_acc [n_q][hidden] then lse_acc [n_q][heads]; n_q * hidden * 4 bytes keeps lse_acc 16-byte aligned
    float *o_acc = base;
    float *lse_acc = base + static_cast<size_t>(n_q) * static_cast<size_t>(hidden);
    return packed_kv_attention_partial(q, n_q, ranges, n_ranges, hidden, group, sm_scale, flags, o_acc, lse_acc,
                                       out_fp32, out, stream);
}
