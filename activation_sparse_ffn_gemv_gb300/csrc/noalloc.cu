// noalloc.cu -- sffn_decode_noalloc: the decode path with its scratch memory in
// a fixed array that lives inside the library, for callers that cannot hand the
// library a workspace (see include/sffn.h).
//
// The scratch is a file-scope __device__ array.  Host code must never pass the
// array's name to a kernel: on the host that name is only a stand-in symbol, not
// a device address.  The device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SFFN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
void *g_scratch_addr[kMaxDev];
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call for that device).  Returns nullptr on failure.
void *scratch_address(int dev) {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" sffn_status sffn_decode_noalloc(const void *x, int B, const sffn_ffn_weights *w, int mode, int score,
                                           float param, void *out, int32_t *active_idx, int32_t *n_active,
                                           sffn_stream_t stream) {
    // sffn_decode's own validation (it returns before launching anything when
    // the workspace pointer is null, so check the arguments the same way here).
    if (!x || !w || !out || !active_idx || !n_active) return SFFN_ERR_INVALID_ARG;
    size_t need = sffn_workspace_size(0, B, w);
    if (need == 0) return (B < 1 || B > 8) ? SFFN_ERR_SHAPE : SFFN_ERR_INVALID_ARG;
    if (need > (size_t)SFFN_NOALLOC_SCRATCH_BYTES) return SFFN_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SFFN_ERR_CUDA;
    void *ws = scratch_address(dev);
    if (!ws) return SFFN_ERR_CUDA;
    // The array keeps whatever the previous call left; the decode kernels write
    // every scratch word before reading it, except the control block (error word,
    // epoch, finish count, chunk flags), which is cleared here so that each call
    // starts clean.
    if (cudaMemsetAsync(ws, 0, sffn::kControlBytes, (cudaStream_t)stream) != cudaSuccess) return SFFN_ERR_CUDA;
    return sffn_decode(x, B, w, mode, score, param, out, active_idx, n_active, ws,
                       (size_t)SFFN_NOALLOC_SCRATCH_BYTES, stream);
}
