// selftest.cu -- a check that the device-side waits are bounded.
//
// Every wait in the forward's kernels (mbarrier phases of the TMA/MMA
// pipelines, the shrink-done counter) gives up after a bounded number of
// rounds and records kStatusTimeout in the workspace status word instead of
// spinning forever.  This kernel runs one such wait on something nothing will
// ever satisfy, so a test can see the wait end, read MOELORA_ETIMEOUT through
// moe_lora_get_status, and go on using the same context.
#include "common.cuh"
#include "kernels.cuh"
#include "tma.cuh"

namespace moelora {

namespace {

__global__ void k_selftest_wait(int kind, WsHeader* hdr) {
    __shared__ uint64_t bar;
    int* counter = &hdr->reserved[0];
    if (threadIdx.x == 0) {
        hdr->status = 0;
        *counter = 0;
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    __threadfence();
    // kind 0: phase 0 of a barrier that expects one arrival nobody makes;
    // kind 1: a counter nobody increments
    const bool ok = kind == 0 ? mbar_wait(&bar, 0) : wait_count(counter, 1) != 0;
    if (!ok) atomicOr(&hdr->status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(int kind, void* workspace, cudaStream_t stream) {
    k_selftest_wait<<<1, 32, 0, stream>>>(kind, static_cast<WsHeader*>(workspace));
    return cudaGetLastError();
}

}  // namespace moelora
