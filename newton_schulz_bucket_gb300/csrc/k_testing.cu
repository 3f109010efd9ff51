// Test hook kernel for failure detection without a GPU fault: one bounded
// mbarrier wait (the same helper the tcgen05 GEMM waits with) on a barrier
// that one thread completes, or that nothing completes.  In the second case
// the wait gives up after `limit` cycles, sets bit 16 of the error word and
// the kernel ends normally.
#include "common.cuh"
#include "mbarrier.cuh"

namespace muon {

namespace {

__global__ void k_wait_probe(int* err, long long limit, int arrive) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  if (threadIdx.x == 0) {
    mbar_init(a, 1);
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 1 && arrive) mbar_arrive(a);
  if (threadIdx.x == 0) mbar_wait(a, 0, &abort_flag, err, 16, limit);
}

}  // namespace

cudaError_t launch_wait_probe(int* err, long long limit, int arrive, cudaStream_t s) {
  k_wait_probe<<<1, 32, 0, s>>>(err, limit, arrive);
  return cudaGetLastError();
}

}  // namespace muon
