// host_util.h -- host-side helpers shared by the launchers: TMA descriptor
// encoding and the launch-argument structs.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Encodes a 3-D tiled TMA descriptor over a dense [dim2][dim1][dim0] tensor
// (dim0 contiguous) with a box of box0 x box1 x 1 elements.  Returns false if
// the driver entry point is unavailable or the encoding is rejected.
bool make_tmap_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t dim0, uint64_t dim1, uint64_t dim2, uint32_t box0, uint32_t box1,
                  CUtensorMapSwizzle swizzle);

// Row layout of the sequences of one call.
//   dense  (varlen = 0): B sequences of N rows; a tensor with H heads is
//                        [B][H][N][d] and LSE / D are [B][H][N].
//   packed (varlen = 1): B sequences of cu_seqlens[b+1] - cu_seqlens[b] rows
//                        (at most N = max_seqlen) stored back to back,
//                        token-major: [total][H][d]; LSE / D are [H][total].
struct SeqLayout {
    int varlen;
    int B, N;               // sequences, rows per sequence (varlen: the maximum)
    int total;              // varlen: rows of all sequences (cu_seqlens[B])
    const int *cu_seqlens;  // varlen: device [B + 1] prefix sums of the lengths
};

// 3-D tiled TMA descriptor with an explicit three-dimensional box.
bool make_tmap_3d_box(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                      uint64_t dim0, uint64_t dim1, uint64_t dim2, uint32_t box0, uint32_t box1, uint32_t box2,
                      CUtensorMapSwizzle swizzle);

// TMA descriptor for 64-column x `rows`-row boxes of the 16-bit tensor with
// `heads` heads in layout `lay` (128-byte swizzle).  Dense: coordinates
// (column, row, plane); packed: (column, head, token).
bool make_tmap_tiles(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int d, const SeqLayout &lay,
                     int heads, uint32_t rows);

// Device address of this library's status words (status.cuh) on the current device
// (looked up once per device and context, cached).
unsigned int *device_status_ptr();

// The CUDA context current on the calling thread (driver handle), or null if
// none is current or the driver entry point is unavailable.  Addresses of
// device symbols are cached per (device, context): after a cudaDeviceReset
// the device's next primary context is a new one and the lookup is redone.
void *current_context();

struct FwdArgs {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int B, Hq, Hkv, N, d, causal;
    float scale;
    bool bf16;
    int window;  // 0: none; > 0: causal sliding window of that many keys
    SeqLayout lay;
    bool o_f32;  // O written as fp32 (debug output), else in the input type
};

struct BwdArgs {
    const void *q, *k, *v, *o, *dO;
    const float *lse;
    void *dq, *dk, *dv;
    int B, Hq, Hkv, N, d, causal;
    float scale;
    bool bf16;
    int window;    // 0: none; > 0: causal sliding window of that many keys
    SeqLayout lay;
    float *D;      // [B][Hq][N] (packed: [Hq][total])
    float *dq_acc; // [B][Hq][N][d]; unused (may be null) by the two-pass backward
};

struct Fp8FwdArgs {
    const void *q8, *k8, *v8;
    const float *q_descale, *k_descale, *v_descale;
    void *o;
    float *lse;
    int B, Hq, Hkv, N, d, causal;
    float scale;
};

struct QuantArgs {
    const void *x;
    const float *signs;
    void *x8;
    float *descale;
    long rows;
    int d;
    float *amax;  // workspace cell
};

cudaError_t launch_fwd(const FwdArgs &a, cudaStream_t st);
// The persistent forward (dense layout, no window, 16-bit output only).
cudaError_t launch_fwd_persist(const FwdArgs &a, cudaStream_t st);
cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t st, bool two_pass);
// The persistent main kernel of the backward (dense layout, atomic dQ, dK and
// dV 32-byte aligned): the step between fa_bwd's D preprocessing and its dQ
// conversion.
cudaError_t launch_bwd_persist_main(const BwdArgs &a, cudaStream_t st);
cudaError_t launch_fwd_fp8(const Fp8FwdArgs &a, cudaStream_t st);
cudaError_t launch_hadamard_quant(const QuantArgs &a, cudaStream_t st);
cudaError_t launch_selftest_wait(int timeout_us, cudaStream_t st);
cudaError_t launch_ex2_rate(float *sink, int blocks, int iters, long long *exps, cudaStream_t st);

}  // namespace fa
