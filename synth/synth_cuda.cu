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

// FP8 E4M3 code of f, round to nearest even, saturating (the definition in
// synth.h; integer rounding of the fp32 bits, no library conversion)
__device__ __forceinline__ uint8_t e4m3_rne(float f) {
    const uint32_t u = __float_as_uint(f);
    const uint32_t sign = (u >> 24) & 0x80u, a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return 0x7f;
    if (a >= 0x43e80000u) return (uint8_t)(sign | 0x7eu);
    if (a >= 0x3c800000u) {
        const uint32_t r = a + 0x7ffffu + ((a >> 20) & 1u);
        return (uint8_t)(sign | ((((r >> 23) - 127u + 7u)) << 3) | ((r >> 20) & 7u));
    }
    const float x = __fmul_rn(__uint_as_float(a), 512.0f);
    uint32_t n = (uint32_t)x;
    const float fr = __fsub_rn(x, (float)n);
    if (fr > 0.5f || (fr == 0.5f && (n & 1u))) ++n;
    return (uint8_t)(sign | n);
}

__global__ void fill_e4m3_kernel(uint8_t* __restrict__ out, uint64_t n, uint64_t key, uint64_t index0, float c) {
    const uint64_t gamma = 0x9e3779b97f4a7c15ULL;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
         i += (uint64_t)gridDim.x * blockDim.x) {
        uint64_t j = 3 * (index0 + i);
        uint32_t s = sum16x4(mix64(key + (j + 1) * gamma)) + sum16x4(mix64(key + (j + 2) * gamma)) +
                     sum16x4(mix64(key + (j + 3) * gamma));
        out[i] = e4m3_rne(__fmul_rn((float)((int32_t)s - 393210), c));
    }
}

__global__ void fill_e8m0_kernel(uint8_t* __restrict__ out, uint64_t n, uint64_t key, uint64_t index0) {
    const uint64_t gamma = 0x9e3779b97f4a7c15ULL;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
         i += (uint64_t)gridDim.x * blockDim.x)
        out[i] = (uint8_t)(117u + (uint32_t)(mix64(key + (index0 + i + 1) * gamma) & 1u));
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

static unsigned grid_for(uint64_t n) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    uint64_t blocks = (n + 255) / 256, cap = (uint64_t)sms * 16;
    return (unsigned)(blocks > cap ? cap : blocks);
}

/* E4M3 codes (sigma 16 draws) of elements index0 .. index0+n-1 of tensor
 * `tensor_id` into dev_out; asynchronous on `stream`. */
int synth_fill_e4m3_cuda(uint8_t* dev_out, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t index0,
                         void* stream) {
    if (n == 0) return 0;
    const uint64_t key = host_mix64(host_mix64(seed) ^ tensor_id);
    const float c = (float)((double)16.0f / 65535.0);
    fill_e4m3_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(dev_out, n, key, index0, c);
    return (int)cudaGetLastError();
}

/* E8M0 scale bytes of blocks index0 .. index0+n-1 of scale tensor `tensor_id`. */
int synth_fill_e8m0_cuda(uint8_t* dev_out, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t index0,
                         void* stream) {
    if (n == 0) return 0;
    const uint64_t key = host_mix64(host_mix64(seed) ^ tensor_id);
    fill_e8m0_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(dev_out, n, key, index0);
    return (int)cudaGetLastError();
}
}
