// rssm_launch.cuh - host-side dispatch from runtime sizes to kernel instantiations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "rssm_device.cuh"

namespace rssm {

constexpr int kSmemMax = 227 * 1024;  // largest dynamic shared memory per CTA on sm_103a

template <int MODE, int N, typename TIn, int RF>
cudaError_t launch_one(const Params& p, int grid, size_t smem, cudaStream_t st) {
  auto kern = head_kernel<MODE, N, TIn, RF>;
  static bool attr_set = false;  // one GPU per process: set the opt-in size once
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // programmatic dependent launch: the kernel waits for the previous grid before
  // its first global access, so it may be scheduled while that grid drains
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// N in {16,32,64,128}; dtype 0 = f32, 1 = bf16; rf 0/1/2/3 (1, 2 and 3 only for N >= 64;
// 3, the FP16 checkpoint, for decode, verify and flush).
template <int MODE, typename TIn>
cudaError_t dispatch_n(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int rf) {
  if (rf == kRfNone) {
    if constexpr (MODE != kQuant) {
      switch (N) {
        case 16: return launch_one<MODE, 16, TIn, kRfNone>(p, grid, smem, st);
        case 32: return launch_one<MODE, 32, TIn, kRfNone>(p, grid, smem, st);
        case 64: return launch_one<MODE, 64, TIn, kRfNone>(p, grid, smem, st);
        case 128: return launch_one<MODE, 128, TIn, kRfNone>(p, grid, smem, st);
      }
    }
  } else if constexpr (MODE == kDecode || MODE == kFlush || MODE == kQuant) {
    if (rf == kRfE4m3) {
      if (N == 64) return launch_one<MODE, 64, TIn, kRfE4m3>(p, grid, smem, st);
      if (N == 128) return launch_one<MODE, 128, TIn, kRfE4m3>(p, grid, smem, st);
    } else if (rf == kRfE2m1) {
      if (N == 64) return launch_one<MODE, 64, TIn, kRfE2m1>(p, grid, smem, st);
      if (N == 128) return launch_one<MODE, 128, TIn, kRfE2m1>(p, grid, smem, st);
    }
  }
  if constexpr (MODE == kDecode || MODE == kVerify || MODE == kFlush) {
    if (rf == kCkF16) {
      if (N == 64) return launch_one<MODE, 64, TIn, kCkF16>(p, grid, smem, st);
      if (N == 128) return launch_one<MODE, 128, TIn, kCkF16>(p, grid, smem, st);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype, int rf);
// The warp-per-head non-flush step (rf = kRfE4m3, kRfE2m1 or kCkF16; N in {64, 128}):
// CTAs of `warps` warps with their stages (rssm_nonflush.cuh) in `smem` bytes.
struct NfStage;
cudaError_t launch_nonflush(const Params& p, const NfStage& sg, int grid, int warps, size_t smem, cudaStream_t st,
                            int N, int dtype, int rf);
// Gated delta-rule layers (rf = kDelta): mode kDecode, kVerify, kFlush or kConv, N in {64, 128}.
cudaError_t launch_delta(int mode, const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype);
cudaError_t launch_verify(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype, int rf);
cudaError_t launch_sround_test(const float* x, uint16_t* y, long long n, long long base, uint32_t epoch,
                               unsigned long long seed, int sr, cudaStream_t st);
cudaError_t launch_flush(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype, int rf);
// The standalone flush's list of folding sequences (one block), before launch_flush.
cudaError_t launch_flush_list(const int32_t* count, int B, int R, int min_count, int32_t* flist, int32_t* fcount,
                              cudaStream_t st);
cudaError_t launch_quant(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int rf);
cudaError_t launch_conv(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype);
cudaError_t launch_wait_selftest(uint32_t* err, cudaStream_t st);
cudaError_t launch_commit(int B, int T, int R, const int32_t* accepted, int32_t* count, uint32_t* err,
                          cudaStream_t st);
cudaError_t launch_snap(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype);
cudaError_t launch_snap_commit(int B, int T, int nslot, const int32_t* accepted, int32_t* cur, uint32_t* err,
                               cudaStream_t st);
struct TcParams;
// Tensor-core verify (bf16 inputs, FP32 checkpoint): N in {64, 128}, P in {32, 64, 128}.
cudaError_t launch_verify_tc(const TcParams& p, const CUtensorMap& tmap, int grid, size_t smem, cudaStream_t st,
                             int N, int P);

}  // namespace rssm
