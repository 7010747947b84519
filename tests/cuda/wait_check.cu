// Test-only kernels for the bounded mbarrier wait used by the codec's kernels: one waits on a
// phase that no copy will ever complete (a transaction count nothing pays off) and must give
// up after the limit; the other waits on a phase that completes and must return at once.
// Nothing is copied, so nothing is in flight when the CTA exits.
#include <cstdint>
#include <cuda_runtime.h>

#include "spl_device.cuh"

namespace {

__global__ void k_wait(int complete, uint32_t* ok, unsigned long long* ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        spl::mbar_init(&bar, 1);
        if (complete) spl::mbar_arrive(&bar);      // the only expected arrival: phase done
        else spl::mbar_expect_tx(&bar, 16);        // arrival + 16 bytes that never come
    }
    __syncthreads();
    const uint64_t t0 = spl::global_ns();
    const bool done = spl::mbar_wait(&bar, 0u);
    const uint64_t t1 = spl::global_ns();
    if (threadIdx.x == 0) {
        *ok = done ? 1u : 0u;
        *ns = t1 - t0;
    }
}

}  // namespace

// Runs one 32-thread CTA; returns the CUDA error code (0 on success).
extern "C" int wait_check(int complete, uint32_t* ok_host, unsigned long long* ns_host) {
    uint32_t* d_ok = nullptr;
    unsigned long long* d_ns = nullptr;
    cudaError_t e = cudaMalloc(&d_ok, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMalloc(&d_ns, sizeof(unsigned long long));
    if (e == cudaSuccess) {
        k_wait<<<1, 32>>>(complete, d_ok, d_ns);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(ok_host, d_ok, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(ns_host, d_ns, sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(d_ok);
    cudaFree(d_ns);
    return static_cast<int>(e);
}
