// fa_bwd_noalloc.cu -- the backward pass for callers that cannot allocate
// device memory.
//
// fa_bwd needs a caller-provided workspace (the D vector and the fp32 dQ
// accumulator).  Some callers cannot obtain one: code running where
// cudaMalloc is not allowed or not wanted -- for example inside a host
// callback, a custom allocator's own hooks, a plugin that receives only
// tensor pointers from its host framework, or a process whose memory pool is
// fixed up front.  For them this entry point uses a fixed scratch buffer that
// lives in the library itself (a file-scope device array), so a call
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
//
// The buffer is FA_BWD_NOALLOC_SCRATCH_BYTES long (include/fa.h).  Every
// device that loads this part of the library holds it until the process
// exits.  All calls on a device share it, so two calls whose kernels overlap
// on the GPU (different streams, no ordering between them) race on it.  Each
// call overwrites D and zeroes the dQ accumulator before using them, so the
// contents left by an earlier call never leak into a later one.
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include <cuda_runtime.h>

namespace {

constexpr size_t kScratchBytes = FA_BWD_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol, never a usable address: the device address is obtained with
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_lock;

// Device address of g_bwd_scratch on the current device; looked up once per
// device (on the first call made with that device current) and cached.
void *scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_lock);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" fa_status_t fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                      const float *lse, const void *dO, void *dq, void *dk, void *dv, int B,
                                      int Hq, int Hkv, int N, int d, int causal, float scale, fa_dtype_t dtype,
                                      void *stream) {
    // Size check first: a problem too large for the built-in buffer is
    // refused before anything touches the GPU.
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    const size_t need = fa_bwd_workspace_bytes(B, Hq, N, d);
    if (need == 0) return FA_ERR_INVALID_ARG;
    if (need > kScratchBytes) return FA_ERR_WORKSPACE;
    void *scratch = scratch_address();
    if (!scratch) return FA_ERR_CUDA;
    // Same validation and kernels as fa_bwd, with the built-in buffer as the
    // workspace.
    return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype, scratch,
                  kScratchBytes, stream);
}
