// Allocation-free variant of mdn_chunk_fwd.
//
// mdn_chunk_fwd needs device scratch (the per-chunk prepared blocks and the
// chunk offsets of packed sequences) that its caller allocates.  Some callers
// cannot allocate device memory at the point where they run the prefill: an
// inference server that reserves all device memory when it starts and forbids
// allocation afterwards (cudaMalloc can synchronise the device and take an
// unbounded time), or plugin code that has no handle to its host's allocator.
// For them, mdn_chunk_fwd_static_ws runs the same kernels on a scratch array
// that lives in this library's own device memory.
//
// The array below is a file-scope __device__ variable.  Its name in host code
// is only a host-side stand-in, not a device address: the device address is
// fetched with cudaGetSymbolAddress, once per device, with that device
// current, on the first call made on that device.  Under lazy module loading
// that first lookup is also where this file's module is loaded and the array
// gets its device memory, so the first call on each device must come before
// the caller reserves the device's memory (and before any stream capture).
// Every call on a device shares the array and it keeps the previous call's
// contents; nothing in it needs to start at zero, because every byte a call
// reads was written earlier in the same call.
#include <stdint.h>

#include <atomic>

#include "mdn_internal.cuh"

static __device__ __align__(256) unsigned char g_mdn_static_ws[MDN_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;
// Device address of g_mdn_static_ws, per device.  Relaxed ordering is
// enough: the cached value is the same pointer whichever thread looks it up
// (a second lookup is harmless) and it guards no other data.
std::atomic<void *> g_static_ws_addr[kMaxDevices];

}  // namespace

extern "C" mdn_status mdn_chunk_fwd_static_ws(
    const void *q, const void *k, const void *v, const float *alpha, const float *mu,
    const float *eta, const float *beta, const float *S0, const float *M0, void *o,
    float *S_T, float *M_T, const int32_t *cu_seqlens, int n_seq, int B, int T, int H,
    int dk, int dv, mdn_dtype dtype, int chunk, void *stream) {
    // the same shape, pointer and device checks as mdn_chunk_fwd, first, so
    // that every error it would report comes back here unchanged
    int *status = nullptr;
    const mdn_status st = mdn::chunk_fwd_check(q, k, v, alpha, mu, eta, beta, S0, M0, o, S_T,
                                               M_T, nullptr, nullptr, nullptr, cu_seqlens, n_seq,
                                               B, T, H, dk, dv, dtype, chunk, &status);
    if (st != MDN_OK) return st;
    const long T_total = (long)B * (long)T;
    const size_t need = mdn_chunk_fwd_workspace_size(n_seq, (int)T_total, H, dk, dv, dtype);
    if (need > (size_t)MDN_STATIC_WORKSPACE_BYTES) return MDN_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return MDN_ERR_UNSUPPORTED;
    void *ws = g_static_ws_addr[dev].load(std::memory_order_relaxed);
    if (ws == nullptr) {
        if (cudaGetSymbolAddress(&ws, g_mdn_static_ws) != cudaSuccess || ws == nullptr) {
            cudaGetLastError();
            return MDN_ERR_CUDA;
        }
        g_static_ws_addr[dev].store(ws, std::memory_order_relaxed);
    }
    return mdn_chunk_fwd(q, k, v, alpha, mu, eta, beta, S0, M0, o, S_T, M_T, cu_seqlens, n_seq,
                         B, T, H, dk, dv, dtype, chunk, ws,
                         (size_t)MDN_STATIC_WORKSPACE_BYTES, stream);
}
