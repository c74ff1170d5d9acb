#include "host_util.h"
namespace fa {
cudaError_t launch_fwd_fp8(const Fp8FwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_hadamard_quant(const QuantArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}
