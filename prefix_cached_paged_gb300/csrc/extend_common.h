// Launchers of the extend-attention kernels (validated arguments in, RC status out).
#pragma once
#include <cuda_runtime.h>

#include "rc.h"

namespace rc {
int launch_extend_simt(const rc_extend_args* a, int* status, cudaStream_t s);
int launch_extend_tc(const rc_extend_args* a, int* status, cudaStream_t s);
}  // namespace rc
