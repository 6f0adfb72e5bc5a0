/*
 * synth_cuda.cu -- device implementation of the generator defined in synth.h.
 * Same integer arithmetic as synth_host.c; the two fp32 operations use the
 * explicit round-to-nearest intrinsics so the compiler cannot fuse them.
 * Exposed through a small C ABI (libsynth_cuda.so), used only by harnesses
 * that need synthetic tensors directly in device memory.
 */
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint32_t sum16x4(uint64_t r) {
    return (uint32_t)(r & 0xffff) + (uint32_t)((r >> 16) & 0xffff) + (uint32_t)((r >> 32) & 0xffff) +
           (uint32_t)(r >> 48);
}

__device__ __forceinline__ uint16_t bf16_rne(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

__global__ void fill_kernel(uint16_t* __restrict__ out, uint64_t n, uint64_t key, uint64_t index0, float c,
                            float mean) {
    const uint64_t gamma = 0x9e3779b97f4a7c15ULL;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
         i += (uint64_t)gridDim.x * blockDim.x) {
        uint64_t j = 3 * (index0 + i);
        uint32_t s = sum16x4(mix64(key + (j + 1) * gamma)) + sum16x4(mix64(key + (j + 2) * gamma)) +
                     sum16x4(mix64(key + (j + 3) * gamma));
        float v = __fmul_rn((float)((int32_t)s - 393210), c);
        if (mean != 0.0f) v = __fadd_rn(v, mean);
        out[i] = bf16_rne(v);
    }
}

uint64_t host_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

}  // namespace

extern "C" {

/* Fill dev_out[0..n) (device memory, bf16 bit patterns) with elements
 * index0 .. index0+n-1 of tensor `tensor_id`; asynchronous on `stream`.
 * Returns 0 or the CUDA error code of the launch. */
int synth_fill_bf16_cuda(uint16_t* dev_out, uint64_t n, uint64_t seed, uint64_t tensor_id, float sigma,
                         float mean, uint64_t index0, void* stream) {
    if (n == 0) return 0;
    uint64_t key = host_mix64(host_mix64(seed) ^ tensor_id);
    float c = (float)((double)sigma / 65535.0);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    uint64_t blocks = (n + 255) / 256;
    uint64_t cap = (uint64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(dev_out, n, key, index0, c, mean);
    return (int)cudaGetLastError();
}
}
