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
void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
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
    // the same argument checks as sffn_decode, in the same order, before the
    // shared array is touched
    sffn_status st = sffn::validate_decode_call(x, B, w, mode, score, param, out, active_idx, n_active);
    if (st != SFFN_OK) return st;
    if (sffn::make_decode_plan(B, w->d_model, w->d_ff).total > (size_t)SFFN_NOALLOC_SCRATCH_BYTES)
        return SFFN_ERR_WORKSPACE;
    void *ws = scratch_address();
    if (!ws) return SFFN_ERR_CUDA;
    // The array keeps whatever the previous call left.  The decode kernels write
    // every scratch word before they read it, except the control block: its
    // grid-barrier counters (arrivals, and the arrivals before the current call)
    // are reset here so that each call starts from a consistent pair even after
    // an earlier call gave up at the barrier.  The error word is left alone: it
    // keeps the first recorded error until sffn_decode_noalloc_read_error reads
    // and clears it.
    cudaError_t e = cudaMemsetAsync(static_cast<char *>(ws) + sffn::kCtlBar, 0, sffn::kControlBytes - sffn::kCtlBar,
                                    (cudaStream_t)stream);
    if (e != cudaSuccess) return SFFN_ERR_CUDA;
    return sffn_decode(x, B, w, mode, score, param, out, active_idx, n_active, ws,
                       (size_t)SFFN_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" sffn_status sffn_decode_noalloc_read_error(int32_t *code, sffn_stream_t stream) {
    if (!code) return SFFN_ERR_INVALID_ARG;
    void *ws = scratch_address();
    if (!ws) return SFFN_ERR_CUDA;
    return sffn_read_device_error(ws, code, stream);
}
