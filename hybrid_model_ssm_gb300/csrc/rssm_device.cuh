// rssm_device.cuh - device code of the ReplaySSM decode library (sm_103a).
//
// One kernel template serves every mode. Each CTA owns a contiguous range of
// (sequence, head) pairs. One producer warp streams the 32 KiB FP32
// checkpoint tile of each head (or its read copy) into a ring of shared-memory
// stages with bulk TMA copies (cp.async.bulk + mbarrier transaction counts).
// Eight consumer warps compute from the staged tile while the next tiles
// are in flight. The small per-group data (the buffered keys K, the queries,
// the dot products k_j^T q) sits in shared memory. The per-head decays and
// coefficients stay in registers and are exchanged with warp shuffles.
//
// Math (aikraft.ru, "ReplaySSM: Революция в декодировании гибридных моделей",
// §01 recurrence, §03 unrolled window, §05 output-only evaluation;
// ai.cheesepanini.fun, "知识卡片：ReplaySSM——重新思考混合模型解码的状态存储",
// 方法/产品要点):
//   non-flush:  o = g_{1:h} (S_ckpt q) + sum_j g_{j+1:h} (k_j^T q) v_j
//   flush:      S_new = g_{1:h} S_ckpt + sum_j (g_{j+1:h} v_j) k_j^T,  o = S_new q
//   verify:     O = S_ckpt Q D + V (W ⊙ (K^T Q))
// with g_{a:b} the product of the decays alpha_a..alpha_b (empty product 1).
//
// Every wait is bounded. A wait that runs out sets an error bit, and the CTA
// then drains its outstanding copies (also bounded) and returns.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace rssm {

constexpr int kNCW = 8;                    // consumer warps per CTA
constexpr int kThreads = (kNCW + 1) * 32;  // + one producer warp
constexpr int kKR = 8;                     // FP32-tile row-instructions per warp per pass
constexpr int kTQ = 4;                     // verify queries per pass over the tile
constexpr int kTMax = 8;                   // largest draft count
constexpr int kRMax = 32;                  // largest ring (records per head)
constexpr int kMaxStages = 8;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s
constexpr unsigned kFull = 0xffffffffu;

enum Mode : int { kDecode = 0, kVerify = 1, kFlush = 2, kQuant = 3, kConv = 4 };
enum Rf : int { kRfNone = 0, kRfE4m3 = 1, kRfE2m1 = 2 };
enum Err : uint32_t { kErrCapacity = 1u, kErrAccept = 2u, kErrTimeout = 4u };

struct Params {
  int B, H, P, N, G, L, R, Rp, HPG, T, min_count;
  float* ckpt;         // [B,H,P,N] checkpoint, or the full state for kConv
  uint8_t* copy;       // read copy: head_stride bytes per (b,h), or null
  int head_stride, bsc_off, rsc_off;
  float* ring_a;       // [B,H,Rp] decays
  void* ring_v;        // [B,H,R,P] values (input dtype)
  void* ring_k;        // [B,G,R,N] keys (input dtype)
  int32_t* start;      // [B]
  int32_t* count;      // [B]
  int32_t* ticket;     // [B], zero between launches
  uint32_t* err;       // error word
  const float* alpha;  // decode/conv [B,H]; verify [B,T,H]
  const void* v;       // decode/conv [B,H,P]; verify [B,T,H,P]
  const void* k;       // decode/conv [B,G,N]; verify [B,T,G,N]
  const void* q;       // decode/conv [B,G,N]; verify [B,T,G,N]
  float* o;            // decode/conv [B,H,P]; verify [B,T,H,P]
  int stages, stage_bytes;
  int kt_off, qt_off, skq_off, wsc_off, wsc_floats, bar_off;  // shared-memory carve (bytes / floats)
};

// ----------------------------------------------------------------- input types
template <typename T> struct In;
template <> struct In<float> {
  using raw = uint32_t;
  static __device__ __forceinline__ float ld(const void* p, size_t i) { return reinterpret_cast<const float*>(p)[i]; }
};
template <> struct In<__nv_bfloat16> {
  using raw = uint16_t;
  static __device__ __forceinline__ float ld(const void* p, size_t i) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  }
};
template <typename T>
__device__ __forceinline__ void copy_raw(void* dst, size_t di, const void* src, size_t si) {
  using R = typename In<T>::raw;
  reinterpret_cast<R*>(dst)[di] = reinterpret_cast<const R*>(src)[si];
}

// ------------------------------------------------------------ PTX primitives
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bulk copy global -> shared, completing `bytes` transactions on `bar`.
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bounded wait on an mbarrier phase. Returns false (after flagging the CTA and
// the device error word) when the wait runs out or another thread aborted.
static __device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t* err) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > kWaitLimitNs) break;
    }
  }
  *abort_flag = 1;
  atomicOr(err, kErrTimeout);
  return false;
}

// ------------------------------------------------------------ FP8/FP4 codes
// cvt packs the value converted from the first source into the upper half.
__device__ __forceinline__ uint32_t enc_e4m3x4(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}
__device__ __forceinline__ uint32_t enc_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(x));
  return r & 0xffu;
}
// Four E2M1 codes -> 16 bits, element 0 in the lowest nibble.
__device__ __forceinline__ uint32_t enc_e2m1x4(float x0, float x1, float x2, float x3) {
  uint16_t r;
  asm("{ .reg .b8 b0, b1; cvt.rn.satfinite.e2m1x2.f32 b0, %1, %2; cvt.rn.satfinite.e2m1x2.f32 b1, %3, %4;"
      " mov.b16 %0, {b0, b1}; }"
      : "=h"(r)
      : "f"(x1), "f"(x0), "f"(x3), "f"(x2));
  return r;
}
// Four E4M3 codes (bytes of w, element 0 lowest) -> four floats.
__device__ __forceinline__ void dec_e4m3x4(uint32_t w, float* out) {
  uint32_t h01, h23;
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.rn.f16x2.e4m3x2 %0, lo; cvt.rn.f16x2.e4m3x2 %1, hi; }"
      : "=r"(h01), "=r"(h23)
      : "r"(w));
  const float2 a = __half22float2(*reinterpret_cast<__half2*>(&h01));
  const float2 b = __half22float2(*reinterpret_cast<__half2*>(&h23));
  out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
}
__device__ __forceinline__ float dec_e4m3(uint32_t code) {
  float t[4];
  dec_e4m3x4(code & 0xffu, t);
  return t[0];
}
// Eight E2M1 codes (nibbles of w, element 0 lowest) -> eight floats.
__device__ __forceinline__ void dec_e2m1x8(uint32_t w, float* out) {
  uint32_t h[4];
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
      " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
      " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h[i]));
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

// ------------------------------------------------------------ warp reductions
// Transposed reduction: K values per lane are summed over the lanes that differ
// in the bits of mask M and below. Each step hands half of the values to the
// partner lane, so K values cost K-1 shuffles instead of K*log2(lanes).
// On return lane L holds max(1, K/(2M)) sums; value i is original index off+i.
template <int K, int M>
struct TRed {
  static __device__ __forceinline__ void run(float* v, int lane, int& off) {
    if constexpr (K > 1) {
      constexpr int H2 = K / 2;
      const bool up = (lane & M) != 0;
#pragma unroll
      for (int i = 0; i < H2; ++i) {
        const float send = up ? v[i] : v[i + H2];
        const float keep = up ? v[i + H2] : v[i];
        v[i] = keep + __shfl_xor_sync(kFull, send, M);
      }
      if (up) off += H2;
      TRed<H2, M / 2>::run(v, lane, off);
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], M);
      TRed<1, M / 2>::run(v, lane, off);
    }
  }
};
template <int K>
struct TRed<K, 0> {
  static __device__ __forceinline__ void run(float*, int, int&) {}
};

template <int LPR>
__device__ __forceinline__ float seg_max(float x) {
#pragma unroll
  for (int m = LPR / 2; m >= 1; m >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, m));
  return x;
}
template <int D>
__device__ __forceinline__ float low_sum(float x) {
#pragma unroll
  for (int m = 1; m < D; m <<= 1) x += __shfl_xor_sync(kFull, x, m);
  return x;
}
// incl[lane] = prod_{i >= lane} x_i over the warp.
__device__ __forceinline__ float suffix_prod(float x, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const float y = __shfl_down_sync(kFull, x, d);
    if (lane + d < 32) x *= y;
  }
  return x;
}

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// ------------------------------------------------------------ quantize a row slice
// Lane holds 4 consecutive elements (x) of a row covered by LPR lanes.
// Writes its codes, and the scales when it owns them, into the head's read copy.
template <int RF, int LPR>
__device__ __forceinline__ void quantize_store(const float4 x, bool live_row, int row, int col4, int N,
                                               uint8_t* head_copy, int bsc_off, int rsc_off) {
  float a = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
  a = seg_max<LPR>(a);  // row amax (all lanes of the row)
  const bool live = a > 7.888609052210118e-31f;  // 2^-100
  if constexpr (RF == kRfE4m3) {
    const float inv = live ? __fdiv_rn(448.f, a) : 0.f;
    const float s = live ? __fdiv_rn(a, 448.f) : 0.f;
    const uint32_t c = enc_e4m3x4(__fmul_rn(x.x, inv), __fmul_rn(x.y, inv), __fmul_rn(x.z, inv), __fmul_rn(x.w, inv));
    if (live_row) {
      *reinterpret_cast<uint32_t*>(head_copy + (size_t)row * N + col4 * 4) = c;
      if (col4 == 0) *reinterpret_cast<float*>(head_copy + rsc_off + row * 4) = s;
    }
  } else {
    const float s_r = live ? __fdiv_rn(a, 2688.f) : 0.f;
    const float d6 = __fmul_rn(6.f, s_r);
    float ab = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
    ab = fmaxf(ab, __shfl_xor_sync(kFull, ab, 1));
    ab = fmaxf(ab, __shfl_xor_sync(kFull, ab, 2));  // 16-element block = 4 lanes
    const float ratio = d6 > 0.f ? __fdiv_rn(ab, d6) : 0.f;
    const uint32_t sb = enc_e4m3(ratio);
    const float d = __fmul_rn(dec_e4m3(sb), s_r);
    const float r = d > 0.f ? __fdiv_rn(1.f, d) : 0.f;
    const uint32_t c = enc_e2m1x4(__fmul_rn(x.x, r), __fmul_rn(x.y, r), __fmul_rn(x.z, r), __fmul_rn(x.w, r));
    if (live_row) {
      *reinterpret_cast<uint16_t*>(head_copy + (size_t)row * (N / 2) + col4 * 2) = (uint16_t)c;
      if ((col4 & 3) == 0) head_copy[bsc_off + row * (N / 16) + (col4 >> 2)] = (uint8_t)sb;
      if (col4 == 0) *reinterpret_cast<float*>(head_copy + rsc_off + row * 4) = s_r;
    }
  }
}

// ============================================================================
// The head kernel.
// ============================================================================
template <int MODE, int N, typename TIn, int RF>
__global__ void __launch_bounds__(kThreads, 1) head_kernel(const Params p) {
  constexpr int LPR = N / 4;    // lanes per FP32 row (4 columns per lane)
  constexpr int RPI = 32 / LPR;  // rows per warp instruction
  static_assert(LPR >= 1 && LPR <= 32 && (32 % LPR) == 0, "N must be 4..128, power of two");
  constexpr bool kAppendMode = (MODE == kDecode || MODE == kVerify);

  extern __shared__ __align__(128) uint8_t smem[];
  float* Kt = reinterpret_cast<float*>(smem + p.kt_off);    // [J][N] keys of the current group
  float* Qt = reinterpret_cast<float*>(smem + p.qt_off);    // [nq][N] queries of the current group
  float* sKQ = reinterpret_cast<float*>(smem + p.skq_off);  // [nq][R] k_j^T q_tau
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  // bars: full[stages], empty[stages], group, end; then the abort flag
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kMaxStages + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total = (long long)p.B * p.H;
  const long long h0 = (long long)blockIdx.x * total / gridDim.x;
  const long long h1 = (long long)(blockIdx.x + 1) * total / gridDim.x;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
  const uint32_t grp_bar = smem_u32(bars + 2 * kMaxStages), end_bar = smem_u32(bars + 2 * kMaxStages + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kNCW);
    }
    mbar_init(grp_bar, kNCW * 32);
    mbar_init(end_bar, kThreads);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // Per-sequence decision shared by producer and consumers (both read the same
  // count[b]; no thread writes pointers before every CTA of b is done).
  //   returns records J to use (>=0) and whether the head tile is loaded.
  auto seq_plan = [&](int b, int& c, int& st, bool& load, bool& flush, bool& bad) {
    c = 0; st = 0; flush = false; bad = false; load = true;
    if constexpr (MODE == kConv || MODE == kQuant) return;
    c = p.count[b];
    st = p.start[b];
    if constexpr (MODE == kDecode) {
      bad = (c + 1 > p.R) || c < 0;
      flush = !bad && (c + 1 >= p.L);
      load = !bad;
    } else if constexpr (MODE == kVerify) {
      bad = (c + p.T > p.R) || c < 0;
      load = !bad;
    } else {  // kFlush
      flush = (c >= p.min_count) && (c > 0) && (c <= p.R);
      load = flush;
    }
  };

  if (warp == kNCW) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int li = 0, cur_b = -1, c = 0, st = 0;
      bool load = false, flush = false, bad = false;
      bool ok = true;
      const uint32_t f32_bytes = (uint32_t)p.P * N * 4;
      for (long long gh = h0; gh < h1 && ok; ++gh) {
        const int b = (int)(gh / p.H);
        if (b != cur_b) {
          cur_b = b;
          seq_plan(b, c, st, load, flush, bad);
        }
        if (!load) continue;
        const int s = li % p.stages, use = li / p.stages;
        if (use > 0 && !mbar_wait(empty0 + 8 * s, (use - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        const bool from_copy = (RF != kRfNone) && (MODE == kDecode) && !flush;
        const void* src = from_copy ? (const void*)(p.copy + (size_t)gh * p.head_stride)
                                    : (const void*)(p.ckpt + (size_t)gh * p.P * N);
        const uint32_t bytes = from_copy ? (uint32_t)p.head_stride : f32_bytes;
        const uint32_t dst = smem_u32(smem + (size_t)s * p.stage_bytes);
        mbar_arrive_tx(full0 + 8 * s, bytes);
        tma_load_1d(dst, src, bytes, full0 + 8 * s);
        ++li;
      }
      if (!ok) {  // drain the copies still in flight (bounded), then leave
        for (int i = (li > p.stages ? li - p.stages : 0); i < li; ++i) {
          volatile int dummy = 0;
          mbar_wait(full0 + 8 * (i % p.stages), (i / p.stages) & 1, &dummy, p.err);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int ct = threadIdx.x;  // 0..255
    const int col4 = lane % LPR, rsub = lane / LPR;
    float* wsc = reinterpret_cast<float*>(smem + p.wsc_off) + warp * p.wsc_floats;  // per-warp scratch
    int li = 0, gphase = 0;
    long long cur_gg = -1;
    int cur_b = -1, c = 0, st = 0, J = 0;
    bool load = false, flush = false, bad = false;
    float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int CPL = (RF == kRfE2m1) ? 32 : 16;  // copy-tile columns per lane
    constexpr int LPRc = (N / CPL) > 0 ? (N / CPL) : 1;
    constexpr int RPIc = 32 / LPRc;
    constexpr int KRc = (kKR * 4 / CPL) > 0 ? (kKR * 4 / CPL) : 1;
    float qc[(RF != kRfNone && MODE == kDecode) ? CPL : 1];
    const int nq = (MODE == kVerify) ? p.T : 1;
    const int rows_pass = kNCW * kKR * RPI;
    const int npass = (p.P + rows_pass - 1) / rows_pass;

    auto group_sync = [&]() -> bool {
      mbar_arrive(grp_bar);
      const bool r = mbar_wait(grp_bar, gphase, abort_flag, p.err);
      gphase ^= 1;
      return r;
    };

    bool ok = true;
    for (long long gh = h0; gh < h1 && ok; ++gh) {
      const int b = (int)(gh / p.H), hh = (int)(gh % p.H), g = hh / p.HPG;
      const long long gg = (long long)b * p.G + g;
      if (b != cur_b) {
        cur_b = b;
        seq_plan(b, c, st, load, flush, bad);
        if (bad && ct == 0) atomicOr(p.err, kErrCapacity);
        if constexpr (MODE == kDecode) J = c + 1;
        else if constexpr (MODE == kVerify) J = c + p.T;
        else if constexpr (MODE == kFlush) J = c;
        else if constexpr (MODE == kConv) J = 1;
        else J = 0;
        cur_gg = -1;
      }
      if (!load) continue;
      if (gg != cur_gg) {
        // ------------------------------------------------ group set-up
        cur_gg = gg;
        if (!group_sync()) { ok = false; break; }
        const size_t kbase = (size_t)(b * p.G + g) * p.R;  // ring row of this group
        const bool first_cta_of_group = ((long long)b * p.H + (long long)g * p.HPG) >= h0;
        for (int idx = ct; idx < J * N; idx += kNCW * 32) {
          const int j = idx / N, n = idx % N;
          float val;
          if constexpr (MODE == kConv) {
            val = In<TIn>::ld(p.k, (size_t)(b * p.G + g) * N + n);
          } else if (j < c) {
            val = In<TIn>::ld(p.ring_k, (kbase + (st + j) % p.R) * N + n);
          } else if constexpr (MODE == kDecode) {
            val = In<TIn>::ld(p.k, (size_t)(b * p.G + g) * N + n);
            if (first_cta_of_group && !flush) copy_raw<TIn>(p.ring_k, (kbase + (st + j) % p.R) * N + n, p.k, (size_t)(b * p.G + g) * N + n);
          } else if constexpr (MODE == kVerify) {
            const size_t si = ((size_t)(b * p.T + (j - c)) * p.G + g) * N + n;
            val = In<TIn>::ld(p.k, si);
            if (first_cta_of_group) copy_raw<TIn>(p.ring_k, (kbase + (st + j) % p.R) * N + n, p.k, si);
          } else {
            val = 0.f;
          }
          Kt[idx] = val;
        }
        if constexpr (MODE == kDecode || MODE == kConv || MODE == kVerify) {
          for (int idx = ct; idx < nq * N; idx += kNCW * 32) {
            const int t = idx / N, n = idx % N;
            const size_t si = (MODE == kVerify) ? ((size_t)(b * p.T + t) * p.G + g) * N + n : (size_t)(b * p.G + g) * N + n;
            Qt[idx] = In<TIn>::ld(p.q, si);
          }
        }
        if (!group_sync()) { ok = false; break; }
        if constexpr (MODE == kDecode || MODE == kVerify) {
          // k_j^T q_tau for all pairs: 8 threads per pair, strided over N
          const int npair = J * nq;
          for (int base = 0; base < npair * 8; base += kNCW * 32) {
            const int idx = base + ct;
            const int pr = idx >> 3, sub = idx & 7;
            float acc = 0.f;
            if (pr < npair) {
              const int t = pr / J, j = pr % J;
              for (int n = sub; n < N; n += 8) acc = fmaf(Kt[j * N + n], Qt[t * N + n], acc);
            }
            acc += __shfl_xor_sync(kFull, acc, 4);
            acc += __shfl_xor_sync(kFull, acc, 2);
            acc += __shfl_xor_sync(kFull, acc, 1);
            if (pr < npair && sub == 0) sKQ[(pr / J) * p.R + (pr % J)] = acc;
          }
          if (!group_sync()) { ok = false; break; }
        }
        if constexpr (MODE == kDecode || MODE == kConv) q4 = lds4(Qt + col4 * 4);
        if constexpr (RF != kRfNone && MODE == kDecode) {
#pragma unroll
          for (int i = 0; i < CPL; ++i) qc[i] = Qt[(lane % LPRc) * CPL + i];
        }
      }

      // ---------------------------------------------------- wait for the tile
      const int s = li % p.stages;
      if (!mbar_wait(full0 + 8 * s, (li / p.stages) & 1, abort_flag, p.err)) { ok = false; break; }
      const uint8_t* tile = smem + (size_t)s * p.stage_bytes;
      const float* tf = reinterpret_cast<const float*>(tile);
      const size_t hrow = (size_t)b * p.H + hh;  // (b, h) index

      // record accessors: decays a(j), values v(j,row) for record j (0-based)
      auto rec_v = [&](int j, int row) -> float {
        if constexpr (MODE == kConv) return In<TIn>::ld(p.v, hrow * p.P + row);
        if (j < c) return In<TIn>::ld(p.ring_v, (hrow * p.R + (st + j) % p.R) * p.P + row);
        if constexpr (MODE == kVerify) return In<TIn>::ld(p.v, ((size_t)(b * p.T + (j - c)) * p.H + hh) * p.P + row);
        return In<TIn>::ld(p.v, hrow * p.P + row);
      };
      float aj = 1.f;  // lane j holds alpha_{j+1}
      if (lane < J) {
        if constexpr (MODE == kConv) aj = p.alpha[hrow];
        else if (lane < c) aj = p.ring_a[hrow * p.Rp + (st + lane) % p.R];
        else if constexpr (MODE == kVerify) aj = p.alpha[((size_t)b * p.T + (lane - c)) * p.H + hh];
        else aj = p.alpha[hrow];
      }

      // ---------------------------------------------------- appends
      if constexpr (kAppendMode) {
        const bool do_append = (MODE == kVerify) || !flush;
        if (do_append) {
          const int na = (MODE == kVerify) ? p.T : 1;
          for (int idx = ct; idx < na * p.P; idx += kNCW * 32) {
            const int t = idx / p.P, row = idx % p.P;
            const size_t dst = (hrow * p.R + (st + c + t) % p.R) * p.P + row;
            const size_t src = (MODE == kVerify) ? ((size_t)(b * p.T + t) * p.H + hh) * p.P + row : hrow * p.P + row;
            copy_raw<TIn>(p.ring_v, dst, p.v, src);
          }
          if (ct < na) {
            const size_t src = (MODE == kVerify) ? ((size_t)b * p.T + ct) * p.H + hh : hrow;
            p.ring_a[hrow * p.Rp + (st + c + ct) % p.R] = p.alpha[src];
          }
        }
      }

      const bool fold = (MODE == kConv) || (MODE == kQuant) || (MODE == kFlush) || (MODE == kDecode && flush);
      if constexpr (MODE == kVerify) {
        // ================================================ verify (T queries)
        // per query tau: x_j = alpha_j for j < c+tau+1 else 1
        float* cw = wsc;                 // [kTMax][kRMax] coefficients
        float* gw = wsc + kTMax * kRMax;  // [kTMax] g_{1:c+tau+1}
        for (int t = 0; t < p.T; ++t) {
          const int ht = c + t + 1;
          const float x = (lane < ht) ? aj : 1.f;
          const float incl = suffix_prod(x, lane);
          const float nxt = __shfl_down_sync(kFull, incl, 1);
          const float w = (lane < 31) ? nxt : 1.f;
          cw[t * kRMax + lane] = (lane < ht) ? w * sKQ[t * p.R + lane] : 0.f;
          if (lane == 0) gw[t] = incl;
        }
        __syncwarp();
        for (int pass = 0; pass < npass; ++pass) {
          const int rbase = (pass * kNCW + warp) * kKR;
          for (int t0 = 0; t0 < p.T; t0 += kTQ) {
            float4 qv[kTQ];
#pragma unroll
            for (int t = 0; t < kTQ; ++t) qv[t] = (t0 + t < p.T) ? lds4(Qt + (t0 + t) * N + col4 * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
            float part[kKR * kTQ];
#pragma unroll
            for (int kk = 0; kk < kKR; ++kk) {
              const int row = (rbase + kk) * RPI + rsub;
              const float4 sv = (row < p.P) ? lds4(tf + ((size_t)row * LPR + col4) * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int t = 0; t < kTQ; ++t) part[kk * kTQ + t] = dot4(sv, qv[t]);
            }
            int off = 0;
            TRed<kKR * kTQ, LPR / 2>::run(part, lane, off);
            constexpr int KF = (kKR * kTQ / LPR) > 0 ? (kKR * kTQ / LPR) : 1;
            constexpr int D = (LPR / (kKR * kTQ)) > 0 ? (LPR / (kKR * kTQ)) : 1;
            const int dup = lane & (D - 1);
#pragma unroll
            for (int i = 0; i < KF; ++i) {
              const int kk = (off + i) / kTQ, t = t0 + (off + i) % kTQ;
              const int row = (rbase + kk) * RPI + rsub;
              const bool valid = row < p.P && t < p.T;
              float ov = 0.f;
              if (valid) {
                for (int j = dup; j < J; j += D) ov = fmaf(cw[t * kRMax + j], rec_v(j, row), ov);
              }
              ov = low_sum<D>(ov);
              if (dup == 0 && valid) p.o[(((size_t)b * p.T + t) * p.H + hh) * p.P + row] = fmaf(gw[t], part[i], ov);
            }
          }
        }
        __syncwarp();
      } else if (fold) {
        // ================================================ fold path
        // S_new = g_{1:J} S + sum_j (g_{j+1:J} v_j) k_j^T ; store ; o = S_new q
        const float incl = suffix_prod(aj, lane);
        const float nxt = __shfl_down_sync(kFull, incl, 1);
        const float wj = (lane < 31) ? nxt : 1.f;  // lane j: g_{j+2:J}, the weight of record j+1
        const float gam = __shfl_sync(kFull, incl, 0);
        for (int pass = 0; pass < npass; ++pass) {
          const int rbase = (pass * kNCW + warp) * kKR;  // first row-instruction of this warp
          // u[(j*RPI + rs)*KR + k] = w_j * v_j[row]
          const int nu = J * RPI * kKR;
          for (int base = 0; base < nu; base += 32) {
            const int idx = base + lane;
            const int j = min(idx / (RPI * kKR), J > 0 ? J - 1 : 0);
            const float wsel = __shfl_sync(kFull, wj, j);
            if (idx < nu) {
              const int rem = idx % (RPI * kKR), rs = rem / kKR, kk = rem % kKR;
              const int row = (rbase + kk) * RPI + rs;
              wsc[idx] = (row < p.P) ? wsel * rec_v(j, row) : 0.f;
            }
          }
          __syncwarp();
          float4 acc[kKR];
#pragma unroll
          for (int kk = 0; kk < kKR; ++kk) {
            const int row = (rbase + kk) * RPI + rsub;
            if (row < p.P) {
              const float4 sv = lds4(tf + ((size_t)row * LPR + col4) * 4);
              acc[kk] = make_float4(gam * sv.x, gam * sv.y, gam * sv.z, gam * sv.w);
            } else {
              acc[kk] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
          for (int j = 0; j < J; ++j) {
            const float4 kv = lds4(Kt + j * N + col4 * 4);
            const float* uj = wsc + (j * RPI + rsub) * kKR;
            const float4 u0 = lds4(uj), u1 = lds4(uj + 4);
            const float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int kk = 0; kk < kKR; ++kk) {
              acc[kk].x = fmaf(uu[kk], kv.x, acc[kk].x);
              acc[kk].y = fmaf(uu[kk], kv.y, acc[kk].y);
              acc[kk].z = fmaf(uu[kk], kv.z, acc[kk].z);
              acc[kk].w = fmaf(uu[kk], kv.w, acc[kk].w);
            }
          }
          // store the new checkpoint (or state) and refresh the read copy
#pragma unroll
          for (int kk = 0; kk < kKR; ++kk) {
            const int row = (rbase + kk) * RPI + rsub;
            const bool live_row = row < p.P;
            if constexpr (MODE != kQuant) {
              if (live_row) *reinterpret_cast<float4*>(p.ckpt + (hrow * p.P + row) * N + col4 * 4) = acc[kk];
            }
            if constexpr (RF != kRfNone && MODE != kConv) {
              // rows beyond P still join the shuffles with zeros
              quantize_store<RF, LPR>(acc[kk], live_row, row, col4, N, p.copy + hrow * p.head_stride, p.bsc_off,
                                      p.rsc_off);
            }
          }
          if constexpr (MODE == kDecode || MODE == kConv) {
            float part[kKR];
#pragma unroll
            for (int kk = 0; kk < kKR; ++kk) part[kk] = dot4(acc[kk], q4);
            int off = 0;
            TRed<kKR, LPR / 2>::run(part, lane, off);
            constexpr int KF = (kKR / LPR) > 0 ? (kKR / LPR) : 1;
            constexpr int D = (LPR / kKR) > 0 ? (LPR / kKR) : 1;
#pragma unroll
            for (int i = 0; i < KF; ++i) {
              const int row = (rbase + off + i) * RPI + rsub;
              if ((lane & (D - 1)) == 0 && row < p.P) p.o[hrow * p.P + row] = part[i];
            }
          }
          __syncwarp();
        }
      } else if constexpr (MODE == kDecode) {
        // ================================================ non-flush decode
        const float incl = suffix_prod(aj, lane);
        const float nxt = __shfl_down_sync(kFull, incl, 1);
        const float w = (lane < 31) ? nxt : 1.f;
        const float gam = __shfl_sync(kFull, incl, 0);
        const float cj = (lane < J) ? w * sKQ[lane] : 0.f;  // g_{j+2:J} * k_{j+1}^T q
        for (int pass = 0; pass < npass; ++pass) {
          if constexpr (RF == kRfNone) {
            const int rbase = (pass * kNCW + warp) * kKR;
            float part[kKR];
#pragma unroll
            for (int kk = 0; kk < kKR; ++kk) {
              const int row = (rbase + kk) * RPI + rsub;
              part[kk] = (row < p.P) ? dot4(lds4(tf + ((size_t)row * LPR + col4) * 4), q4) : 0.f;
            }
            int off = 0;
            TRed<kKR, LPR / 2>::run(part, lane, off);
            constexpr int KF = (kKR / LPR) > 0 ? (kKR / LPR) : 1;
            constexpr int D = (LPR / kKR) > 0 ? (LPR / kKR) : 1;
            const int dup = lane & (D - 1);
#pragma unroll
            for (int i = 0; i < KF; ++i) {
              const int row = (rbase + off + i) * RPI + rsub;
              float ov = 0.f;
              for (int j = 0; j < J; ++j) {
                const float cjj = __shfl_sync(kFull, cj, j);
                if ((j & (D - 1)) == dup && row < p.P) ov = fmaf(cjj, rec_v(j, row), ov);
              }
              ov = low_sum<D>(ov);
              if (dup == 0 && row < p.P) p.o[hrow * p.P + row] = fmaf(gam, part[i], ov);
            }
          } else {
            // read copy: lanes own CPL consecutive codes of a row
            const int rows0 = (pass * kNCW + warp) * kKR * RPI;  // first row of this warp
            const int colc = lane % LPRc, rsc = lane / LPRc;
            const float* rscale = reinterpret_cast<const float*>(tile + p.rsc_off);
            float part[KRc];
#pragma unroll
            for (int kk = 0; kk < KRc; ++kk) {
              const int row = rows0 + kk * RPIc + rsc;
              float acc = 0.f;
              if (row < p.P) {
                if constexpr (RF == kRfE4m3) {
                  const uint4 cw = *reinterpret_cast<const uint4*>(tile + (size_t)row * N + colc * 16);
                  const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                  for (int qd = 0; qd < 4; ++qd) {
                    float f[4];
                    dec_e4m3x4(ws[qd], f);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc = fmaf(f[e], qc[qd * 4 + e], acc);
                  }
                } else {
                  const uint4 cw = *reinterpret_cast<const uint4*>(tile + (size_t)row * (N / 2) + colc * 16);
                  const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
                  const uint8_t* bsp = tile + p.bsc_off + row * (N / 16) + colc * 2;
                  float blk[2] = {0.f, 0.f};
#pragma unroll
                  for (int qd = 0; qd < 4; ++qd) {
                    float f[8];
                    dec_e2m1x8(ws[qd], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) blk[qd >> 1] = fmaf(f[e], qc[qd * 8 + e], blk[qd >> 1]);
                  }
                  acc = fmaf(dec_e4m3(bsp[0]), blk[0], dec_e4m3(bsp[1]) * blk[1]);
                }
                acc *= rscale[row];
              }
              part[kk] = acc;
            }
            int off = 0;
            TRed<KRc, LPRc / 2>::run(part, lane, off);
            constexpr int KF = (KRc / LPRc) > 0 ? (KRc / LPRc) : 1;
            constexpr int D = (LPRc / KRc) > 0 ? (LPRc / KRc) : 1;
            const int dup = lane & (D - 1);
#pragma unroll
            for (int i = 0; i < KF; ++i) {
              const int row = rows0 + (off + i) * RPIc + rsc;
              float ov = 0.f;
              for (int j = 0; j < J; ++j) {
                const float cjj = __shfl_sync(kFull, cj, j);
                if ((j & (D - 1)) == dup && row < p.P) ov = fmaf(cjj, rec_v(j, row), ov);
              }
              ov = low_sum<D>(ov);
              if (dup == 0 && row < p.P) p.o[hrow * p.P + row] = fmaf(gam, part[i], ov);
            }
          }
        }
      }

      // ---------------------------------------------------- release the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
      ++li;
    }
  }

  // ------------------------------------------------------------------ epilogue
  // Pointer updates: once every CTA covering a sequence has finished reading its
  // pointers, the last one (ticket) advances them. Never a spin wait.
  mbar_arrive(end_bar);
  if (threadIdx.x == 0) {
    const bool done = mbar_wait(end_bar, 0, abort_flag, p.err) && !*abort_flag;
    if (done && (MODE == kDecode || MODE == kFlush) && h1 > h0) {
      const int b_first = (int)(h0 / p.H), b_last = (int)((h1 - 1) / p.H);
      for (int b = b_first; b <= b_last; ++b) {
        const long long lo = max(h0, (long long)b * p.H), hi = min(h1, (long long)(b + 1) * p.H);
        const int n_b = (int)(hi - lo);
        int c, st;
        bool load, flush, bad;
        seq_plan(b, c, st, load, flush, bad);
        if (MODE == kFlush && !flush) continue;
        if (MODE == kDecode && bad) continue;
        __threadfence();
        const int prev = atomicAdd(p.ticket + b, n_b);
        if (prev + n_b == p.H) {
          __threadfence();
          if (MODE == kDecode) {
            if (flush) {
              p.start[b] = (st + c + 1) % p.R;
              p.count[b] = 0;
            } else {
              p.count[b] = c + 1;
            }
          } else {
            p.start[b] = (st + c) % p.R;
            p.count[b] = 0;
          }
          p.ticket[b] = 0;
        }
      }
    }
  }
}

}  // namespace rssm
