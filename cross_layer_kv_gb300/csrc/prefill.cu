#include "fkv_kernels.h"
namespace fkv {
cudaError_t prefill_launch(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}
