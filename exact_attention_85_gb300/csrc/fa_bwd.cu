#include "host_util.h"
namespace fa {
cudaError_t launch_bwd(const BwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}
