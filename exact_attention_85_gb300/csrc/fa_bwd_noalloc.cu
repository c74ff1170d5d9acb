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
// The buffer is FA_BWD_NOALLOC_SCRATCH_BYTES long (include/fa.h).  It belongs
// to this translation unit's own module, which the CUDA runtime loads -- and
// so commits the buffer's device memory -- when the module is first used (the
// first call on a device, under the default lazy module loading) or when the
// library is loaded (CUDA_MODULE_LOADING=EAGER).  From then on the device
// holds it until the process exits.  All calls on a device share it, so two
// calls whose kernels overlap on the GPU (different streams, no ordering
// between them) race on it.  Each call overwrites D and zeroes the dQ
// accumulator before using them, so the contents left by an earlier call
// never leak into a later one.
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "host_util.h"

namespace {

constexpr size_t kScratchBytes = FA_BWD_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol, never a usable address: the device address is obtained with
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
    void *ctx;  // context the address was looked up in
    void *addr;
};
ScratchSlot g_slot[kMaxDevices];
std::mutex g_scratch_lock;

// Device address of g_bwd_scratch on the current device.  Set-up happens on
// the first call made with the device current: cudaGetSymbolAddress (which
// loads this module if it is not loaded yet) with its return code checked.
// The address is cached per device together with the context it was found
// in, and looked up again if the device's current context changes (after a
// cudaDeviceReset the old address no longer exists).
void *scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void *ctx = fa::current_context();  // null before the runtime has made one current
    std::lock_guard<std::mutex> lk(g_scratch_lock);
    ScratchSlot &s = g_slot[dev];
    if (s.addr != nullptr && ctx != nullptr && s.ctx == ctx) return s.addr;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return nullptr;
    if (ctx == nullptr) ctx = fa::current_context();  // the lookup made the context current
    if (ctx == nullptr) return nullptr;
    s.ctx = ctx;
    s.addr = p;
    return p;
}

}  // namespace

extern "C" fa_status_t fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                      const float *lse, const void *dO, void *dq, void *dk, void *dv, int B,
                                      int Hq, int Hkv, int N, int d, int causal, float scale, fa_dtype_t dtype,
                                      void *stream) {
    // fa_bwd checks the workspace last, after every other argument, and
    // launches nothing before that check: asked without a workspace it
    // answers FA_ERR_WORKSPACE exactly when everything else is valid.  So
    // invalid arguments are classified here exactly as fa_bwd classifies them.
    const fa_status_t st = fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype,
                                  nullptr, 0, stream);
    if (st != FA_ERR_WORKSPACE) return st;
    // a problem too large for the built-in buffer is refused before anything
    // touches the GPU
    if (fa_bwd_workspace_bytes(B, Hq, N, d) > kScratchBytes) return FA_ERR_WORKSPACE;
    void *scratch = scratch_address();
    if (!scratch) return FA_ERR_CUDA;
    // the same kernels as fa_bwd, with the built-in buffer as the workspace
    return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype, scratch, kScratchBytes,
                  stream);
}
