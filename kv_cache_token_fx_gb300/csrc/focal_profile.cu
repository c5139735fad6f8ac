// Focal-layer selection by warm-up profiling (FastOCR, Focal-Guided Pruning: "Focal Layer
// Selection"): during a short warm-up every layer attends over the whole cache, and the share of its
// attention that falls on the image tokens is recorded; the layers with the highest share become the
// focal layers.
//
// The share per (b, KV head) comes from the focal call's importance scores over the image tokens:
// those scores are the group's R softmax rows summed, so their sum divided by R is the mean image
// share of the group's rows.  One CTA per row reduces n scores in a fixed order (deterministic).
#include <stdint.h>

#include "fx_internal.h"

namespace fx {
namespace {

constexpr int kMassThreads = 256;

__global__ void __launch_bounds__(kMassThreads) focal_mass_kernel(const float* scores, int n, float inv_r,
                                                                  int accumulate, float* mass)
{
    griddep_wait();   // the scores come from the kernel just before
    griddep_launch();
    const int row = blockIdx.x;
    const float* s = scores + (int64_t)row * n;
    float acc = 0.f;
    for (int j = threadIdx.x; j < n; j += kMassThreads) acc += s[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ float sw[kMassThreads / 32];
    if ((threadIdx.x & 31) == 0) sw[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < kMassThreads / 32; ++w) t += sw[w];
        mass[row] = (accumulate ? mass[row] : 0.f) + t * inv_r;
    }
}

}  // namespace

cudaError_t launch_focal_mass(const float* scores, int rows, int n, float inv_r, int accumulate, float* mass,
                              bool pdl, cudaStream_t s)
{
    return launch_kernel(focal_mass_kernel, dim3(rows), dim3(kMassThreads), 0, s, pdl, 0u, scores, n, inv_r,
                         accumulate, mass);
}

}  // namespace fx
