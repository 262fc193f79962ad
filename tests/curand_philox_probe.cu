// curand_philox_probe.cu -- test infrastructure only.
//
// Philox4x32-10 outputs computed by cuRAND's device API (the header-defined
// curand_Philox4x32_10(counter, key)), for pinning the CPU oracle's generator
// against an implementation that is not this project's.  The tests compile
// this file with nvcc on the GPU machine and call the one entry point below
// through ctypes; nothing in the library or the oracle uses it.
#include <cuda_runtime.h>
#include <curand_philox4x32_x.h>
#include <stdint.h>

__global__ void philox_probe_kernel(const uint4* __restrict__ ctr, const uint2* __restrict__ key,
                                    uint4* __restrict__ out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = curand_Philox4x32_10(ctr[i], key[i]);
}

// out[4 i .. 4 i + 3] = Philox4x32-10(counter = ctr[4 i .. 4 i + 3], key = key[2 i .. 2 i + 1]),
// host arrays; returns the first CUDA error code (0 = success).
extern "C" int curand_philox4x32_10_batch(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int n) {
    if (n <= 0) return 0;
    uint4 *dc = nullptr, *dout = nullptr;
    uint2* dk = nullptr;
    cudaError_t e = cudaMalloc(&dc, sizeof(uint4) * (size_t)n);
    if (e == cudaSuccess) e = cudaMalloc(&dk, sizeof(uint2) * (size_t)n);
    if (e == cudaSuccess) e = cudaMalloc(&dout, sizeof(uint4) * (size_t)n);
    if (e == cudaSuccess) e = cudaMemcpy(dc, ctr, sizeof(uint4) * (size_t)n, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(dk, key, sizeof(uint2) * (size_t)n, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
        philox_probe_kernel<<<(n + 255) / 256, 256>>>(dc, dk, dout, n);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(out, dout, sizeof(uint4) * (size_t)n, cudaMemcpyDeviceToHost);
    cudaFree(dc);
    cudaFree(dk);
    cudaFree(dout);
    return (int)e;
}
