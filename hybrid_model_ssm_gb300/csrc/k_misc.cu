// Instantiations of the standalone flush, the read-copy quantizer and the
// conventional read-update-write comparison kernel.
#include "rssm_launch.cuh"

namespace rssm {
cudaError_t launch_flush(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype, int rf) {
  if (rf == kDelta) return launch_delta(kFlush, p, grid, smem, st, N, dtype);
  return dtype == 0 ? dispatch_n<kFlush, float>(p, grid, smem, st, N, rf)
                    : dispatch_n<kFlush, __nv_bfloat16>(p, grid, smem, st, N, rf);
}
// The sequences a standalone flush folds (count >= min_count, 0 < count <= R),
// in increasing order, into flist[0 .. *fcount). One block.
__global__ void flush_list_kernel(const int32_t* count, int B, int R, int min_count, int32_t* flist,
                                  int32_t* fcount) {
  __shared__ int warp_n[32];
  __shared__ int base;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) base = 0;
  __syncthreads();
  for (int b0 = 0; b0 < B; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    bool f = false;
    if (b < B) {
      const int c = count[b];
      f = c >= min_count && c > 0 && c <= R;
    }
    const unsigned m = __ballot_sync(kFull, f);
    if (lane == 0) warp_n[w] = __popc(m);
    __syncthreads();
    int off = base;
    for (int i = 0; i < w; ++i) off += warp_n[i];
    if (f) flist[off + __popc(m & ((1u << lane) - 1u))] = b;
    __syncthreads();
    if (threadIdx.x == 0) {
      int t = 0;
      for (int i = 0; i < nw; ++i) t += warp_n[i];
      base += t;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *fcount = base;
}

cudaError_t launch_flush_list(const int32_t* count, int B, int R, int min_count, int32_t* flist, int32_t* fcount,
                              cudaStream_t st) {
  flush_list_kernel<<<1, 1024, 0, st>>>(count, B, R, min_count, flist, fcount);
  return cudaGetLastError();
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
// Test support: the checkpoint store's binary32 -> binary16 rounding applied to
// x[0..n), element i taking word (i % 4) of the generator call for element
// group (base + i) / 4 at the given epoch (base a multiple of 4).
__global__ void sround_test_kernel(const float* __restrict__ x, uint16_t* __restrict__ y, long long n, long long base,
                                   uint32_t epoch, unsigned long long seed, int sr) {
  const long long g4 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (g4 >= n) return;
  float xv[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) xv[e] = (g4 + e < n) ? x[g4 + e] : 0.f;
  const float4 a = make_float4(xv[0], xv[1], xv[2], xv[3]);
  // the fold's store, in either mode
  const uint2 h = sr ? sr_f16x4(a, sr_words((size_t)(base + g4), epoch, seed))
                     : make_uint2(rn_f16x2_sat(a.x, a.y), rn_f16x2_sat(a.z, a.w));
  const uint32_t h01 = h.x, h23 = h.y;
  const uint16_t hv[4] = {(uint16_t)h01, (uint16_t)(h01 >> 16), (uint16_t)h23, (uint16_t)(h23 >> 16)};
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (g4 + e < n) y[g4 + e] = hv[e];
}
cudaError_t launch_sround_test(const float* x, uint16_t* y, long long n, long long base, uint32_t epoch,
                               unsigned long long seed, int sr, cudaStream_t st) {
  const long long groups = (n + 3) / 4;
  const int threads = 256;
  sround_test_kernel<<<(unsigned)((groups + threads - 1) / threads), threads, 0, st>>>(x, y, n, base, epoch, seed, sr);
  return cudaGetLastError();
}
}  // namespace rssm
