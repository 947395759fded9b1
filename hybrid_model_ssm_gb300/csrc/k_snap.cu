// Instantiations of the conventional speculative verify used as the in-run
// comparison: every draft advances the full state and writes a snapshot of it
// (one state read and T state writes per round); commit moves a per-sequence
// slot index to the accepted snapshot.
#include "rssm_launch.cuh"

namespace rssm {
// cur[b] <- (cur[b] + accepted[b]) mod nslot for 0 <= accepted[b] <= T (one thread per sequence).
__global__ void snap_commit_kernel(int B, int T, int nslot, const int32_t* __restrict__ accepted, int32_t* cur,
                                   uint32_t* err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int a = accepted[b];
  const int c = cur[b];
  if (a < 0 || a > T || c < 0 || c >= nslot) {
    atomicOr(err, kErrAccept);
    return;
  }
  cur[b] = (c + a) % nslot;
}

cudaError_t launch_snap(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype) {
  return dtype == 0 ? dispatch_n<kSnap, float>(p, grid, smem, st, N, kRfNone)
                    : dispatch_n<kSnap, __nv_bfloat16>(p, grid, smem, st, N, kRfNone);
}
cudaError_t launch_snap_commit(int B, int T, int nslot, const int32_t* accepted, int32_t* cur, uint32_t* err,
                               cudaStream_t st) {
  const int threads = 256;
  snap_commit_kernel<<<(B + threads - 1) / threads, threads, 0, st>>>(B, T, nslot, accepted, cur, err);
  return cudaGetLastError();
}
}  // namespace rssm
