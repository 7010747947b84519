// Test-only kernel: compares the library's division helper (reciprocal + Markstein
// correction), and for power-of-two divisors the single multiply by the exact reciprocal,
// with CUDA's correctly rounded division, bit for bit, over dividend ranges given by their bit
// patterns and divisors 1..pmax.  Built and loaded by the GPU tests.
#include <cstdint>
#include <cuda_runtime.h>

#include "spl_device.cuh"

namespace {

__global__ void k_div_check(const float* rps, uint32_t bits_lo, uint32_t count,
                            unsigned long long* bad, uint32_t* first_bad) {
    const int P = blockIdx.y + 1;
    const float d = static_cast<float>(P);
    const float rd = rps[blockIdx.y];
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += gridDim.x * blockDim.x) {
        const uint32_t b = bits_lo + i;
        const float x = __uint_as_float(b);
        const float q = spl::div_rn(x, d, rd);
        const float r = __fdiv_rn(x, d);
        bool same = __float_as_uint(q) == __float_as_uint(r) || (q != q && r != r);
        if ((P & (P - 1)) == 0) {   // the decode's path for P = 2^k: one multiply by 2^-k
            const float m = __fmul_rn(x, rd);
            same = same && (__float_as_uint(m) == __float_as_uint(r) || (m != m && r != r));
        }
        if (!same) {
            atomicAdd(bad, 1ull);
            atomicCAS(first_bad, 0xffffffffu, b);
        }
    }
}

}  // namespace

// Returns 0 and writes the mismatch count (and the first mismatching dividend's bits, or
// 0xffffffff) for dividends with bit patterns [bits_lo, bits_lo + count) and every divisor
// 1..pmax; returns the CUDA error code on failure.
extern "C" int div_check(int pmax, uint32_t bits_lo, uint32_t count,
                         unsigned long long* mismatches, uint32_t* first_bad) {
    float h_rp[256];
    if (pmax < 1 || pmax > 256) return -1;
    for (int p = 1; p <= pmax; ++p) h_rp[p - 1] = 1.0f / static_cast<float>(p);
    float* d_rp = nullptr;
    unsigned long long* d_bad = nullptr;
    uint32_t* d_first = nullptr;
    cudaError_t e = cudaMalloc(&d_rp, sizeof h_rp);
    if (e == cudaSuccess) e = cudaMalloc(&d_bad, sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMalloc(&d_first, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemcpy(d_rp, h_rp, sizeof h_rp, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(d_bad, 0, sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemset(d_first, 0xff, sizeof(uint32_t));
    if (e == cudaSuccess) {
        k_div_check<<<dim3(1024, pmax), 256>>>(d_rp, bits_lo, count, d_bad, d_first);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(mismatches, d_bad, sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(first_bad, d_first, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    cudaFree(d_rp);
    cudaFree(d_bad);
    cudaFree(d_first);
    return static_cast<int>(e);
}
