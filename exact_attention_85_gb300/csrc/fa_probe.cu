// fa_probe.cu -- measurement aid: the throughput of the exp2 instruction the
// softmax uses (ex2.approx.ftz.f32, executed by the special-function unit).
//
// The FA3 summary ("Overlapping GEMM and softmax asynchronously") notes that
// the exponential runs on a separate, much slower unit than the matrix
// multiply-add, so that at head dimension 128 it can take half as long as
// the matmuls.  Dividing the exps of one attention call by the rate measured
// here gives the time the call would take if it were bound by exp2 alone.
//
// Every thread runs eight independent chains x <- 2^x - 1.5.  For x in
// [-1, -0.5] the next value lies in [-1, -0.79], so the chains stay bounded
// and never meet a special value; the only other work is one add per exp.
#include "host_util.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kProbeThreads = 256;
constexpr int kChains = 8;

__global__ void __launch_bounds__(kProbeThreads) ex2_rate_kernel(float *sink, int iters) {
    float x[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = -0.5f - 0.0625f * i;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) x[i] = ex2_approx(x[i]) - 1.5f;
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += x[i];
    sink[(size_t)blockIdx.x * kProbeThreads + threadIdx.x] = s;
}

}  // namespace

cudaError_t launch_ex2_rate(float *sink, int blocks, int iters, long long *exps, cudaStream_t st) {
    ex2_rate_kernel<<<blocks, kProbeThreads, 0, st>>>(sink, iters);
    *exps = (long long)blocks * kProbeThreads * kChains * iters;
    return cudaGetLastError();
}

}  // namespace fa
