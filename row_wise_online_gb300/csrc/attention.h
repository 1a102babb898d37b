// attention.h -- launch interface of the attention forward kernel (kernel_attention.cu).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "launch.h"

namespace rwo {

// Attention forward (tcgen05): q [BH][Sq][d], k and v [BH][Sk][d], o [BH][Sq][d], bf16 (dtype 1)
// or fp16 (dtype 2), d = 64 or 128.
bool attention_fits(int64_t d, int dtype);
cudaError_t launch_attention(const void* q, const void* k, const void* v, void* o, float* lse, int64_t BH, int64_t Sq,
                             int64_t Sk, int64_t d, float scale, bool causal, int dtype, cudaStream_t stream,
                             const DeviceInfo& dev);

}  // namespace rwo
