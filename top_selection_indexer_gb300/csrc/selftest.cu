// Self-test of the failure path: a bounded device-side wait that runs out.
//
// Every tensor-core kernel waits on mbarriers through tc::mbar_wait, whose clock budget
// turns a wait that never completes into the device error word (and an abort flag for the
// other roles) instead of a hang.  This kernel exercises exactly that helper: one thread
// waits on a barrier that nothing will complete; after the budget the helper sets the error
// word and the kernel returns.  Nothing faults, traps or spins without bound.
#include "tc_common.cuh"

namespace tsi {
namespace {

__global__ void __launch_bounds__(32) tsi_wait_timeout_probe_kernel(unsigned* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);  // one arrival expected; none will come
    abort_flag = 0;
    tc::fence_barrier_init();
    tc::mbar_wait(&bar, 0, &abort_flag, err);  // runs out after tc::kWaitCycles
}

}  // namespace

cudaError_t launch_wait_timeout_probe(unsigned* err, cudaStream_t st) {
    tsi_wait_timeout_probe_kernel<<<1, 32, 0, st>>>(err);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace tsi
