// Instantiations of the head kernel for gated delta-rule layers (FP32
// checkpoint, N in {64, 128}): the decode step, the speculative verify, the
// standalone flush and the conventional read-update-write step used for comparison.
#include "rssm_launch.cuh"

namespace rssm {
template <int MODE, typename TIn>
static cudaError_t delta_n(const Params& p, int grid, size_t smem, cudaStream_t st, int N) {
  if (N == 64) return launch_one<MODE, 64, TIn, kDelta>(p, grid, smem, st);
  if (N == 128) return launch_one<MODE, 128, TIn, kDelta>(p, grid, smem, st);
  return cudaErrorInvalidValue;
}
cudaError_t launch_delta(int mode, const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype) {
  if (mode == kDecode) return dtype == 0 ? delta_n<kDecode, float>(p, grid, smem, st, N)
                                         : delta_n<kDecode, __nv_bfloat16>(p, grid, smem, st, N);
  if (mode == kFlush) return dtype == 0 ? delta_n<kFlush, float>(p, grid, smem, st, N)
                                        : delta_n<kFlush, __nv_bfloat16>(p, grid, smem, st, N);
  if (mode == kVerify) return dtype == 0 ? delta_n<kVerify, float>(p, grid, smem, st, N)
                                         : delta_n<kVerify, __nv_bfloat16>(p, grid, smem, st, N);
  if (mode == kConv) return dtype == 0 ? delta_n<kConv, float>(p, grid, smem, st, N)
                                       : delta_n<kConv, __nv_bfloat16>(p, grid, smem, st, N);
  return cudaErrorInvalidValue;
}
}  // namespace rssm
