// spv_selftest.cu -- self-test of the bounded waits and of the error word.
//
// Every spin of the library's kernels (the tree walk's cluster barrier, the
// streaming ring's mbarriers) gives up after a bounded number of polls,
// records SPV_ERR_TIMEOUT in the workspace's error word and returns, so the
// CUDA context stays usable.  This kernel runs the same bounded flag wait on
// a header word that nothing ever sets, so the give-up path and its report
// can be checked on a GPU without a fault.
#include "spv_internal.h"
#include "spv_stream.cuh"

namespace spv {

// Header word 1 of the workspace: cleared here and never set by anyone.
__global__ void selftest_wait_kernel(unsigned *words, unsigned polls)
{
    if (threadIdx.x != 0) return;
    atomicExch(&words[1], 0u);
    __threadfence();
    wait_flag_ge(&words[1], 1u, polls, &words[0]);
}

cudaError_t launch_selftest_wait(void *ws, unsigned polls, cudaStream_t st)
{
    selftest_wait_kernel<<<1, 32, 0, st>>>(static_cast<unsigned *>(ws), polls);
    return cudaGetLastError();
}

}  // namespace spv
