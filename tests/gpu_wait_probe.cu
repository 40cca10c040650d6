// Test driver for the library's bounded mbarrier wait (pa_device.cuh): a
// wait on a phase that nothing completes must give up after its time limit
// and raise PA_ERRBIT_WAIT_TIMEOUT, leaving the context usable; a wait on a
// completed phase returns at once.  Built by tests/test_gpu_wait_timeout.py.
#include "pa_device.cuh"

using namespace pa;

__global__ void wait_probe_kernel(int32_t* flag, unsigned long long* elapsed_ns, int arrive,
                                  unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (arrive) mbar_arrive(&bar);
        const uint64_t t0 = global_timer_ns();
        const bool ok = mbar_wait_bounded(&bar, 0u, limit_ns);
        *elapsed_ns = global_timer_ns() - t0;
        if (!ok) raise_flag(flag, PA_ERRBIT_WAIT_TIMEOUT);
    }
}

extern "C" int wait_probe(int32_t* flag, unsigned long long* elapsed_ns, int arrive, unsigned long long limit_ns) {
    wait_probe_kernel<<<1, 32>>>(flag, elapsed_ns, arrive, limit_ns);
    return static_cast<int>(cudaDeviceSynchronize());
}
