// A bounded mbarrier wait that runs out: the library's mbar_wait_bounded on
// a barrier that nothing arrives at returns false after its poll limit, the
// kernel reports RS_DEV_PIPE_TIMEOUT in the status word and returns, and the
// context stays usable.  Also prints the cycles a wait of a given number of
// polls took, so the test can check what the kernels' limit amounts to.
//
// Build: nvcc -gencode arch=compute_103a,code=sm_103a -std=c++17 wait_timeout.cu
// Output: one line per limit "polls status cycles", then "after ok" once a
// second kernel has run and synchronised on the same context.
#include <cstdio>
#include <cuda_runtime.h>

#include "../../recurrent_state_gb300/csrc/rs_device.cuh"

namespace {

constexpr int kStatusTimeout = 8;  // RS_DEV_PIPE_TIMEOUT

__global__ void wait_nothing_arrives(int32_t *status, uint32_t limit, long long *cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) rs::mbar_init(&bar, 1);  // one arrival expected, none ever made
    rs::fence_mbar_init();
    __syncthreads();
    const long long t0 = clock64();
    const bool done = rs::mbar_wait_bounded(&bar, 0u, limit);
    const long long t1 = clock64();
    if (!done) atomicOr(status, kStatusTimeout);
    if (threadIdx.x == 0) *cycles = t1 - t0;
}

__global__ void add_one(int32_t *x) { atomicAdd(x, 1); }

bool check(cudaError_t e, const char *what) {
    if (e != cudaSuccess) {
        std::printf("error %s: %s\n", what, cudaGetErrorString(e));
        return false;
    }
    return true;
}

}  // namespace

int main() {
    int32_t *status = nullptr;
    long long *cycles = nullptr;
    if (!check(cudaMalloc(&status, sizeof(int32_t)), "malloc") ||
        !check(cudaMalloc(&cycles, sizeof(long long)), "malloc"))
        return 1;
    const uint32_t limits[] = {1u << 10, 1u << 14};
    for (uint32_t limit : limits) {
        if (!check(cudaMemset(status, 0, sizeof(int32_t)), "memset")) return 1;
        wait_nothing_arrives<<<1, 32>>>(status, limit, cycles);
        if (!check(cudaGetLastError(), "launch") || !check(cudaDeviceSynchronize(), "sync")) return 1;
        int32_t st = 0;
        long long cy = 0;
        if (!check(cudaMemcpy(&st, status, sizeof st, cudaMemcpyDeviceToHost), "copy") ||
            !check(cudaMemcpy(&cy, cycles, sizeof cy, cudaMemcpyDeviceToHost), "copy"))
            return 1;
        std::printf("%u %d %lld\n", limit, st, cy);
    }
    if (!check(cudaMemset(status, 0, sizeof(int32_t)), "memset")) return 1;
    add_one<<<4, 32>>>(status);
    if (!check(cudaGetLastError(), "launch") || !check(cudaDeviceSynchronize(), "sync")) return 1;
    int32_t n = 0;
    if (!check(cudaMemcpy(&n, status, sizeof n, cudaMemcpyDeviceToHost), "copy")) return 1;
    std::printf("after %s\n", n == 128 ? "ok" : "wrong");
    int clock_khz = 0;
    cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, 0);
    std::printf("clock_khz %d\n", clock_khz);
    cudaFree(status);
    cudaFree(cycles);
    return 0;
}
