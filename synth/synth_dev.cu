/*
 * synth_dev.cu -- device side of the synthetic input generator (see synth.h).
 *
 * Fills large device buffers (the history K/V of a workload, tens of GB) in
 * place so that nothing that size crosses the host link.  Produces exactly
 * the values synth_fill_normal produces on the host.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

__global__ void synth_fill_normal_kernel(float* __restrict__ dst, uint64_t count,
                                         uint64_t key, uint64_t index0) {
    uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += stride)
        dst[i] = synth_normal(key, index0 + i);
}

extern "C" int synth_dev_fill_normal(float* dst, uint64_t count, uint64_t seed,
                                     uint64_t stream, uint64_t index0,
                                     void* cuda_stream) {
    if (count == 0) return 0;
    if (!dst) return (int)cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    uint64_t want = (count + 255) / 256;
    uint64_t cap = (uint64_t)sms * 8;
    unsigned grid = (unsigned)(want < cap ? want : cap);
    synth_fill_normal_kernel<<<grid, 256, 0, (cudaStream_t)cuda_stream>>>(
        dst, count, synth_key(seed, stream), index0);
    return (int)cudaGetLastError();
}
