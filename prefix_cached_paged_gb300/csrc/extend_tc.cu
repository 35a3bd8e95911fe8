// placeholder until the tcgen05 kernel lands: route to the CUDA-core kernel
#include "extend_common.h"
namespace rc {
int launch_extend_tc(const rc_extend_args* a, int* status, cudaStream_t s) {
  return launch_extend_simt(a, status, s);
}
}  // namespace rc
