// Instantiations of the standalone flush, the read-copy quantizer and the
// conventional read-update-write comparison kernel.
#include "rssm_launch.cuh"

namespace rssm {
cudaError_t launch_flush(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype, int rf) {
  return dtype == 0 ? dispatch_n<kFlush, float>(p, grid, smem, st, N, rf)
                    : dispatch_n<kFlush, __nv_bfloat16>(p, grid, smem, st, N, rf);
}
cudaError_t launch_quant(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int rf) {
  if (rf == kRfNone) return cudaErrorInvalidValue;
  return dispatch_n<kQuant, float>(p, grid, smem, st, N, rf);
}
// Self-test of the bounded waits: one warp waits on an mbarrier that nothing
// completes. The wait gives up after its time limit, sets the timeout bit of
// the error word and returns; the context stays usable.
__global__ void wait_selftest_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  mbar_wait(smem_u32(&bar), 0, reinterpret_cast<volatile int*>(&abort_flag), err);
}
cudaError_t launch_wait_selftest(uint32_t* err, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err);
  return cudaGetLastError();
}
cudaError_t launch_conv(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype) {
  return dtype == 0 ? dispatch_n<kConv, float>(p, grid, smem, st, N, kRfNone)
                    : dispatch_n<kConv, __nv_bfloat16>(p, grid, smem, st, N, kRfNone);
}
}  // namespace rssm
