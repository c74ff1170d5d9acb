// fa_api.cu -- the extern "C" boundary of libfa.so: argument validation,
// the per-device status word, TMA descriptor encoding and dispatch to the
// kernel launchers.  Declarations and their contracts are in include/fa.h.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "host_util.h"
#include "ptx.cuh"

// Optional NVTX ranges around every entry point that launches work (built
// with -DFA_NVTX, e.g. FA_NVTX=1 for build.py): a profiler timeline then
// shows each call by name.  Off by default; header-only, nothing to link.
#ifdef FA_NVTX
#include <nvtx3/nvToolsExt.h>
namespace {
struct FaRange {
    explicit FaRange(const char *name) { nvtxRangePushA(name); }
    ~FaRange() { nvtxRangePop(); }
};
}  // namespace
#define FA_RANGE(name) FaRange fa_range_(name)
#else
#define FA_RANGE(name) ((void)0)
#endif

namespace fa {

// Two status words per device that loads the library (module-scope device
// variable, status.cuh): timeouts, then the other conditions.  Kernels
// receive the address of the first as a parameter.
__device__ unsigned int g_status_word[2];

namespace {

constexpr int kMaxDevices = 64;
struct StatusSlot {
    void *ctx;  // context the address was looked up in
    unsigned int *addr;
};
StatusSlot g_status_slot[kMaxDevices];
std::mutex g_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
    std::lock_guard<std::mutex> lk(g_mutex);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

__global__ void selftest_wait_kernel(unsigned int *status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // nothing ever arrives on this barrier
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, (volatile int *)&abort_flag, status, 0xFFFF, limit_ns);
    __syncthreads();
}

}  // namespace

bool make_tmap_3d_box(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes, uint64_t dim0,
                      uint64_t dim1, uint64_t dim2, uint32_t box0, uint32_t box1, uint32_t box2,
                      CUtensorMapSwizzle swizzle) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {dim0, dim1, dim2};
    cuuint64_t strides[2] = {dim0 * elem_bytes, dim0 * dim1 * elem_bytes};
    cuuint32_t box[3] = {box0, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    std::memset(map, 0, sizeof(*map));
    CUresult r = enc(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes, uint64_t dim0,
                  uint64_t dim1, uint64_t dim2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle) {
    return make_tmap_3d_box(map, base, dtype, elem_bytes, dim0, dim1, dim2, box0, box1, 1, swizzle);
}

bool make_tmap_tiles(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int d, const SeqLayout &lay,
                     int heads, uint32_t rows) {
    if (lay.varlen)  // [total][heads][d]: coordinates (column, head, token)
        return make_tmap_3d_box(map, base, dtype, 2, d, heads, lay.total, 64, 1, rows, CU_TENSOR_MAP_SWIZZLE_128B);
    // [B * heads][N][d]: coordinates (column, row, plane)
    return make_tmap_3d_box(map, base, dtype, 2, d, lay.N, (uint64_t)lay.B * heads, 64, rows, 1,
                            CU_TENSOR_MAP_SWIZZLE_128B);
}

void *current_context() {
    static CtxGetCurrentFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<CtxGetCurrentFn>(nullptr);
        return reinterpret_cast<CtxGetCurrentFn>(f);
    }();
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

unsigned int *device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void *ctx = current_context();  // null before the runtime has made one current
    std::lock_guard<std::mutex> lk(g_mutex);
    StatusSlot &s = g_status_slot[dev];
    if (s.addr != nullptr && ctx != nullptr && s.ctx == ctx) return s.addr;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess || p == nullptr) return nullptr;
    if (ctx == nullptr) ctx = current_context();  // the lookup made the context current
    if (ctx == nullptr) return nullptr;
    s.ctx = ctx;
    s.addr = static_cast<unsigned int *>(p);
    return s.addr;
}

cudaError_t launch_selftest_wait(int timeout_us, cudaStream_t st) {
    unsigned int *status = device_status_ptr();
    if (!status) return cudaErrorUnknown;
    selftest_wait_kernel<<<1, 32, 0, st>>>(status, (unsigned long long)timeout_us * 1000ull);
    return cudaGetLastError();
}

}  // namespace fa

// ------------------------------------------------------------------ C ABI

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// rows: rows of one head's tensors, B * N dense or `total` packed (a packed
// batch holds far fewer rows than B * max_seqlen when its lengths differ)
fa_status_t check_shape(int B, int Hq, int Hkv, int N, int d, float scale, long long rows) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    // rows and (batch x head) planes are counted in 32 bits; element offsets
    // are 64-bit everywhere, so a tensor may hold more than 2^31 elements
    if (rows > 0x7FFFFFFFll || (long long)B * Hq > 0x7FFFFFFFll) return FA_ERR_UNSUPPORTED;
    // 1-D grid of (Q tiles x heads x batch) CTAs
    if ((long long)((N + 127) / 128) * B * Hq > 0x7FFFFFFFll) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

fa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Shared validation and launch of the forward entry points (window 0: none).
fa_status_t fwd_common(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv,
                       int N, int d, int causal, int window, float scale, fa_dtype_t dtype, void *stream,
                       const fa::SeqLayout *packed = nullptr, bool o_f32 = false, bool persistent = false) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    fa_status_t s = check_shape(B, Hq, Hkv, N, d, scale, packed ? packed->total : (long long)B * N);
    if (s != FA_OK) return s;
    fa::SeqLayout lay{0, B, N, B * N, nullptr};
    if (packed) lay = *packed;
    fa::FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, dtype == FA_BF16, window, lay, o_f32};
    if (persistent) return from_cuda(fa::launch_fwd_persist(a, static_cast<cudaStream_t>(stream)));
    return from_cuda(fa::launch_fwd(a, static_cast<cudaStream_t>(stream)));
}

// Shared validation and launch of the backward entry points: two_pass picks
// the deterministic variant, whose workspace holds D only.
fa_status_t bwd_common(const void *q, const void *k, const void *v, const void *o, const float *lse,
                       const void *dO, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N, int d,
                       int causal, int window, float scale, fa_dtype_t dtype, bool two_pass, void *workspace,
                       size_t workspace_bytes, void *stream, const fa::SeqLayout *packed = nullptr) {
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
    for (const void *p : ptrs)
        if (!aligned16(p)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    fa_status_t s = check_shape(B, Hq, Hkv, N, d, scale, packed ? packed->total : (long long)B * N);
    if (s != FA_OK) return s;
    fa::SeqLayout lay{0, B, N, B * N, nullptr};
    if (packed) lay = *packed;
    const size_t rows = (size_t)lay.total * Hq;
    const size_t need = two_pass ? round256(rows * sizeof(float))
                                 : round256(rows * sizeof(float)) + round256(rows * (size_t)d * sizeof(float));
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FA_ERR_WORKSPACE;
    float *D = static_cast<float *>(workspace);
    float *dq_acc =
        two_pass ? nullptr
                 : reinterpret_cast<float *>(static_cast<char *>(workspace) + round256(rows * sizeof(float)));
    fa::BwdArgs a{q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype == FA_BF16,
                  window, lay, D, dq_acc};
    return from_cuda(fa::launch_bwd(a, static_cast<cudaStream_t>(stream), two_pass));
}

}  // namespace

extern "C" {

const char *fa_status_string(fa_status_t s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    }
    return "FA_ERR_UNKNOWN";
}

fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv,
                   int N, int d, int causal, float scale, fa_dtype_t dtype, void *stream) {
    FA_RANGE("fa_fwd");
    return fwd_common(q, k, v, o, lse, B, Hq, Hkv, N, d, causal ? 1 : 0, 0, scale, dtype, stream);
}

fa_status_t fa_fwd_persistent(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                              int Hkv, int N, int d, int causal, float scale, fa_dtype_t dtype, void *stream) {
    FA_RANGE("fa_fwd_persistent");
    if (reinterpret_cast<uintptr_t>(o) & 31u) return FA_ERR_INVALID_ARG;  // O rows are stored 32 bytes at a time
    return fwd_common(q, k, v, o, lse, B, Hq, Hkv, N, d, causal ? 1 : 0, 0, scale, dtype, stream, nullptr, false,
                      true);
}

fa_status_t fa_fwd_f32_out(const void *q, const void *k, const void *v, float *o_f32, float *lse, int B, int Hq,
                           int Hkv, int N, int d, int causal, float scale, fa_dtype_t dtype, void *stream) {
    FA_RANGE("fa_fwd_f32_out");
    return fwd_common(q, k, v, o_f32, lse, B, Hq, Hkv, N, d, causal ? 1 : 0, 0, scale, dtype, stream, nullptr,
                      true);
}

fa_status_t fa_fwd_local(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                         int Hkv, int N, int d, int window, float scale, fa_dtype_t dtype, void *stream) {
    FA_RANGE("fa_fwd_local");
    if (window < 1) return FA_ERR_INVALID_ARG;
    return fwd_common(q, k, v, o, lse, B, Hq, Hkv, N, d, 1, window, scale, dtype, stream);
}

size_t fa_bwd_workspace_bytes(int B, int Hq, int N, int d) {
    if (B < 1 || Hq < 1 || N < 1 || d < 1) return 0;
    const size_t rows = (size_t)B * Hq * N;
    return round256(rows * sizeof(float)) + round256(rows * (size_t)d * sizeof(float));
}

size_t fa_bwd_two_pass_workspace_bytes(int B, int Hq, int N, int d) {
    if (B < 1 || Hq < 1 || N < 1 || d < 1) return 0;
    return round256((size_t)B * Hq * N * sizeof(float));
}

fa_status_t fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
                   void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                   fa_dtype_t dtype, void *workspace, size_t workspace_bytes, void *stream) {
    FA_RANGE("fa_bwd");
    return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d, causal ? 1 : 0, 0, scale, dtype, false,
                      workspace, workspace_bytes, stream);
}

fa_status_t fa_bwd_two_pass(const void *q, const void *k, const void *v, const void *o, const float *lse,
                            const void *dO, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N, int d,
                            int causal, float scale, fa_dtype_t dtype, void *workspace, size_t workspace_bytes,
                            void *stream) {
    FA_RANGE("fa_bwd_two_pass");
    return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d, causal ? 1 : 0, 0, scale, dtype, true,
                      workspace, workspace_bytes, stream);
}

fa_status_t fa_bwd_local(const void *q, const void *k, const void *v, const void *o, const float *lse,
                         const void *dO, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N, int d,
                         int window, float scale, fa_dtype_t dtype, int deterministic, void *workspace,
                         size_t workspace_bytes, void *stream) {
    FA_RANGE("fa_bwd_local");
    if (window < 1) return FA_ERR_INVALID_ARG;
    return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d, 1, window, scale, dtype,
                      deterministic != 0, workspace, workspace_bytes, stream);
}

namespace {
// Checks shared by the packed (variable-length) entry points.
fa_status_t check_varlen(const int *cu_seqlens, int B, int max_seqlen, int total, int Hq, int Hkv, int d,
                         int causal, int window) {
    if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FA_ERR_INVALID_ARG;
    if (B < 1 || max_seqlen < 1 || total < 1 || Hq < 1 || Hkv < 1) return FA_ERR_INVALID_ARG;
    if (window < 0 || (window > 0 && !causal)) return FA_ERR_INVALID_ARG;
    return FA_OK;  // sizes: check_shape, with the packed total as the row count
}
}  // namespace

fa_status_t fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse, const int *cu_seqlens,
                          int B, int max_seqlen, int total, int Hq, int Hkv, int d, int causal, int window,
                          float scale, fa_dtype_t dtype, void *stream) {
    FA_RANGE("fa_fwd_varlen");
    fa_status_t s = check_varlen(cu_seqlens, B, max_seqlen, total, Hq, Hkv, d, causal, window);
    if (s != FA_OK) return s;
    const fa::SeqLayout lay{1, B, max_seqlen, total, cu_seqlens};
    return fwd_common(q, k, v, o, lse, B, Hq, Hkv, max_seqlen, d, causal ? 1 : 0, window, scale, dtype, stream,
                      &lay);
}

size_t fa_bwd_varlen_workspace_bytes(int total, int Hq, int d, int deterministic) {
    if (total < 1 || Hq < 1 || d < 1) return 0;
    const size_t rows = (size_t)total * Hq;
    return round256(rows * sizeof(float)) + (deterministic ? 0 : round256(rows * (size_t)d * sizeof(float)));
}

fa_status_t fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                          const void *dO, void *dq, void *dk, void *dv, const int *cu_seqlens, int B,
                          int max_seqlen, int total, int Hq, int Hkv, int d, int causal, int window, float scale,
                          fa_dtype_t dtype, int deterministic, void *workspace, size_t workspace_bytes,
                          void *stream) {
    FA_RANGE("fa_bwd_varlen");
    fa_status_t s = check_varlen(cu_seqlens, B, max_seqlen, total, Hq, Hkv, d, causal, window);
    if (s != FA_OK) return s;
    const fa::SeqLayout lay{1, B, max_seqlen, total, cu_seqlens};
    return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, max_seqlen, d, causal ? 1 : 0, window, scale,
                      dtype, deterministic != 0, workspace, workspace_bytes, stream, &lay);
}

size_t fa_hadamard_quant_workspace_bytes(long rows, int d) {
    (void)rows;
    (void)d;
    return 256;
}

fa_status_t fa_hadamard_quant_fp8(const void *x_bf16, const float *signs, void *x_e4m3, float *descale, long rows,
                                  int d, void *workspace, size_t workspace_bytes, void *stream) {
    FA_RANGE("fa_hadamard_quant_fp8");
    if (!x_bf16 || !x_e4m3 || !descale || rows < 1) return FA_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(x_e4m3) || (signs && !aligned16(signs))) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < fa_hadamard_quant_workspace_bytes(rows, d) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FA_ERR_WORKSPACE;
    fa::QuantArgs a{x_bf16, signs, x_e4m3, descale, rows, d, static_cast<float *>(workspace)};
    return from_cuda(fa::launch_hadamard_quant(a, static_cast<cudaStream_t>(stream)));
}

fa_status_t fa_fwd_fp8(const void *q8, const void *k8, const void *v8, const float *q_descale,
                       const float *k_descale, const float *v_descale, void *o_bf16, float *lse, int B, int Hq,
                       int Hkv, int N, int d, int causal, float scale, void *stream) {
    FA_RANGE("fa_fwd_fp8");
    if (!q8 || !k8 || !v8 || !q_descale || !k_descale || !v_descale || !o_bf16 || !lse) return FA_ERR_INVALID_ARG;
    const void *ptrs[] = {q8, k8, v8, o_bf16, lse};
    for (const void *p : ptrs)
        if (!aligned16(p)) return FA_ERR_INVALID_ARG;
    fa_status_t s = check_shape(B, Hq, Hkv, N, d, scale, (long long)B * N);
    if (s != FA_OK) return s;
    if (d != 128) return FA_ERR_UNSUPPORTED;  // one 128-byte swizzle atom per e4m3 row
    fa::Fp8FwdArgs a{q8, k8, v8, q_descale, k_descale, v_descale, o_bf16, lse, B, Hq, Hkv, N, d,
                     causal ? 1 : 0, scale};
    return from_cuda(fa::launch_fwd_fp8(a, static_cast<cudaStream_t>(stream)));
}

fa_status_t fa_get_device_status(void *stream) {
    unsigned int *p = fa::device_status_ptr();
    if (!p) return FA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int host[2] = {0u, 0u};
    if (cudaMemcpyAsync(host, p, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, sizeof(host), st) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
    if (host[0] & fa::kStatusTimeout) return FA_ERR_TIMEOUT;
    if (host[1] & fa::kStatusBadLaunch) return FA_ERR_CUDA;
    return (host[1] & fa::kStatusBadArgs) ? FA_ERR_INVALID_ARG : FA_OK;
}

long long fa_probe_exp2(float *sink, int blocks, int iters, void *stream) {
    FA_RANGE("fa_probe_exp2");
    if (!sink || !aligned16(sink) || blocks < 1 || blocks > 65535 || iters < 1 || iters > (1 << 24)) return -1;
    long long exps = 0;
    if (fa::launch_ex2_rate(sink, blocks, iters, &exps, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return -1;
    return exps;
}

fa_status_t fa_selftest_bounded_wait(int timeout_us, void *stream) {
    FA_RANGE("fa_selftest_bounded_wait");
    if (timeout_us < 1 || timeout_us > 1000000) return FA_ERR_INVALID_ARG;
    return from_cuda(fa::launch_selftest_wait(timeout_us, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
