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
cudaError_t launch_conv(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype) {
  return dtype == 0 ? dispatch_n<kConv, float>(p, grid, smem, st, N, kRfNone)
                    : dispatch_n<kConv, __nv_bfloat16>(p, grid, smem, st, N, kRfNone);
}
}  // namespace rssm
