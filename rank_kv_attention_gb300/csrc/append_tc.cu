// Tensor-core (tcgen05) append projection: not yet enabled; the generic
// append path is used for every shape.
#include "append_kernels.cuh"

namespace lrkv {

bool tc_append_supported(int, int, int, int, int) { return false; }

cudaError_t launch_append_tc(const AppendArgsT<__nv_bfloat16> &) { return cudaErrorNotSupported; }

}  // namespace lrkv
