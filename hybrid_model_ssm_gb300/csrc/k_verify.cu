// Instantiations of the speculative-verify kernel, plus the commit kernel.
#include "rssm_launch.cuh"

namespace rssm {
// Commit: count[b] += accepted[b] for 0 <= accepted[b] <= T (one thread per sequence).
__global__ void commit_kernel(int B, int T, int R, const int32_t* __restrict__ accepted, int32_t* count,
                              uint32_t* err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int a = accepted[b];
  const int c = count[b];
  if (a < 0 || a > T || c + a > R) {
    atomicOr(err, kErrAccept);
    return;
  }
  count[b] = c + a;
}

cudaError_t launch_verify(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype, int rf) {
  if (rf == kDelta) return launch_delta(kVerify, p, grid, smem, st, N, dtype);
  return dtype == 0 ? dispatch_n<kVerify, float>(p, grid, smem, st, N, rf)
                    : dispatch_n<kVerify, __nv_bfloat16>(p, grid, smem, st, N, rf);
}
cudaError_t launch_commit(int B, int T, int R, const int32_t* accepted, int32_t* count, uint32_t* err,
                          cudaStream_t st) {
  const int threads = 256;
  commit_kernel<<<(B + threads - 1) / threads, threads, 0, st>>>(B, T, R, accepted, count, err);
  return cudaGetLastError();
}
}  // namespace rssm
