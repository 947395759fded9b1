// rssm_device.cuh - device code of the ReplaySSM decode library (sm_103a).
//
// One kernel template serves every mode. Each CTA owns a contiguous range of
// (sequence, head) pairs. A producer warp feeds a ring of shared-memory
// stages. For each head, one bulk TMA copy (cp.async.bulk + mbarrier
// transaction count) brings the 32 KiB FP32 checkpoint tile, or its read copy.
// The producer lanes also gather that head's buffered records in record order
// with cp.async: the decays alpha_j and the value rows v_j. For each group of
// H/G heads, they gather the buffered keys k_j and the queries into a
// double-buffered group area. Eight consumer warps therefore read only
// shared memory, and the next stages stay in flight while they compute.
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

constexpr int kNDW = 8;                    // dot warps per CTA (stream the checkpoint tile)
constexpr int kNCoef = 2;                  // warps computing the per-head decay terms (alternate heads)
static_assert((kNCoef & (kNCoef - 1)) == 0, "coefficient warps: a power of two");
constexpr int kTileWarp = kNDW;            // warp that issues the bulk tile copies
constexpr int kCoef0 = kNDW + 1;           // first coefficient warp
constexpr int kGatherWarp = kNDW + 1 + kNCoef;  // warp that gathers the records, keys and queries
constexpr int kThreads = (kNDW + 2 + kNCoef) * 32;
constexpr int kMaxSlots = 32;              // largest record-slot ring
constexpr int kKR = 8;                     // FP32-tile row-instructions per warp per pass (multiple of 4)
static_assert(kKR % 4 == 0, "rows per warp must be a multiple of 4");
constexpr int kTQ = 4;                     // verify queries per pass over the tile
constexpr int kTMax = 8;                   // largest draft count
constexpr int kRMax = 32;                  // largest ring (records per head)
constexpr int kMaxStages = 16;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s
// The warp-per-head non-flush step (rssm_nonflush.cuh): at most this many warps per CTA,
// one CTA per SM (the warps' shared-memory stages decide how many fit).
constexpr int kNfMaxWarps = 16;
constexpr int kNfMaxThreads = kNfMaxWarps * 32;
constexpr unsigned kFull = 0xffffffffu;

enum Mode : int { kDecode = 0, kVerify = 1, kFlush = 2, kQuant = 3, kConv = 4, kSnap = 5 };
// Storage formats of the head tile: the FP32 checkpoint (kRfNone), an E4M3 or
// E2M1 read copy next to it, or an FP16 checkpoint (kCkF16: no read copy).
// kDelta: an FP32 checkpoint of a gated delta-rule layer (the same tiles; the
// ring keeps each record's pseudo-value w instead of v).
enum Rf : int { kRfNone = 0, kRfE4m3 = 1, kRfE2m1 = 2, kCkF16 = 3, kDelta = 4 };
enum Err : uint32_t { kErrCapacity = 1u, kErrAccept = 2u, kErrTimeout = 4u, kErrPlan = 8u };

// One partition of a CTA's shared memory into tile stages and record slots.
struct Layout {
  int stages, stage_bytes, slots, slot_bytes, slot_off, sv_off, sc_off;
  int nv_off;   // delta-rule layers: the new record's v row
  int dgroups;  // dot-warp groups (1, 2, 4 or 8): group d takes every dgroups-th head, so that many are in flight
};

struct Params {
  int B, H, P, N, G, L, R, Rp, HPG, T, min_count;
  float* ckpt;         // [B,H,P,N] checkpoint; the full state for kConv; kSnap: [nslot][B,H,P,N] state slots
  uint8_t* copy;       // read copy: head_stride bytes per (b,h), or null
  int head_stride, bsc_off, rsc_off;
  float* ring_a;       // [B,H,Rp] decays
  void* ring_v;        // [B,H,R,P] values (input dtype); delta-rule layers: pseudo-values w (fp32)
  void* ring_k;        // [B,G,R,N] keys (input dtype)
  int32_t* start;      // [B]
  int32_t* count;      // [B]
  int32_t* ticket;     // [B], zero between launches
  int32_t* epoch;      // [B] flushes so far (FP16 checkpoint: part of the rounding counter)
  const int32_t* flist;   // kFlush: the flushing sequences in order, or null (every sequence)
  const int32_t* fcount;  // kFlush: their number
  unsigned long long seed;  // FP16 checkpoint: generator key
  int sr;              // FP16 checkpoint: 1 stochastic rounding, 0 round to nearest
  int skip_nonflush;   // kDecode: leave non-flush sequences to the warp-per-head kernel (pointers still advance)
  const int32_t* cur;  // kSnap: [B] slot holding each sequence's state
  int nslot;           // kSnap: state slots (T_max + 1)
  uint32_t* err;       // error word
  const float* alpha;  // decode/conv [B,H]; verify [B,T,H]
  const float* beta;   // delta-rule decode [B,H]
  const void* v;       // decode/conv [B,H,P]; verify [B,T,H,P]
  const void* k;       // decode/conv [B,G,N]; verify [B,T,G,N]
  const void* q;       // decode/conv [B,G,N]; verify [B,T,G,N]
  float* o;            // decode/conv [B,H,P]; verify [B,T,H,P]
  // Shared memory (bytes). From offset 0, one of two layouts:
  //   `stages` tile stages: the head tile (P x N fp32, or the read copy);
  //   `slots` record slots: [alpha_j (kRMax fp32) | v_j rows | coefficients],
  //   coefficients: g (or g_t) at 0..15, then the value term [P], the scaled
  //   values [R][P] of a fold, or the verify weights [kTMax][kRMax].
  // lay[0] fits every head; lay[1] (decode) only non-flush heads: tiles of the
  // read copy, at most L - 1 records and no fold, so more heads are in flight.
  // A CTA takes lay[1] when none of its sequences flushes in this launch.
  // Behind both: two group areas of [k_j rows (R x N) | queries (kTMax x N)],
  // the coefficient-warp scratch and the barriers.
  Layout lay[2];
  int nf_ok;  // lay[1] is valid
  int gb_off, gb_bytes, gq_off;
  int wsc_off, bar_off;  // coefficient-warp scratch (kTMax x kRMax fp32), barriers
  int dsc_off;           // delta-rule verify: per dot warp [32 rows][8] row sums
};

// ----------------------------------------------------------------- input types
// Loads of v/k/q elements (fp32 or bf16) as fp32 from shared memory.
template <typename T> struct In;
template <> struct In<float> {
  static constexpr int kBytes = 4;
  static __device__ __forceinline__ float lds(const uint8_t* base, int i) {
    return reinterpret_cast<const float*>(base)[i];
  }
  static __device__ __forceinline__ float4 lds4(const uint8_t* base, int i) {  // i multiple of 4
    return *reinterpret_cast<const float4*>(base + 4 * i);
  }
  static __device__ __forceinline__ float2 lds2(const uint8_t* base, int i) {  // i even
    return *reinterpret_cast<const float2*>(base + 4 * i);
  }
};
template <> struct In<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static __device__ __forceinline__ float lds(const uint8_t* base, int i) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
  }
  static __device__ __forceinline__ float4 lds4(const uint8_t* base, int i) {  // i multiple of 4
    const uint2 w = *reinterpret_cast<const uint2*>(base + 2 * i);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  static __device__ __forceinline__ float2 lds2(const uint8_t* base, int i) {  // i even
    const uint32_t w = *reinterpret_cast<const uint32_t*>(base + 2 * i);
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
};

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
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(n) : "memory");
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

// Bulk store shared -> global (the ring appends), tracked by the thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The shared-memory sources of this thread's bulk stores have been read.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// This thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Small asynchronous copies global -> shared (the record gathers).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once all earlier cp.async of this thread have landed (counted in the init count).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bounded wait on an mbarrier phase. Returns false (after flagging the CTA and
// the device error word) when the wait runs out or another thread aborted.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                   uint32_t* err) {
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
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t* err) {
  return mbar_try(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, err);
}

// (sequence, head, group) of consecutive flattened heads, advanced without divisions.
struct HeadIter {
  int b, hh, g, gpos;
  __device__ __forceinline__ void init(long long h0, int H, int HPG) {
    b = (int)(h0 / H);
    hh = (int)(h0 - (long long)b * H);
    g = hh / HPG;
    gpos = hh - g * HPG;
  }
  __device__ __forceinline__ void next(int H, int HPG) {
    ++hh;
    if (++gpos == HPG) { gpos = 0; ++g; }
    if (hh == H) { hh = 0; g = 0; gpos = 0; ++b; }
  }
};

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
// The same transposed scheme for a maximum.
template <int K, int M>
struct TMax {
  static __device__ __forceinline__ void run(float* v, int lane, int& off) {
    if constexpr (K > 1) {
      constexpr int H2 = K / 2;
      const bool up = (lane & M) != 0;
#pragma unroll
      for (int i = 0; i < H2; ++i) {
        const float send = up ? v[i] : v[i + H2];
        const float keep = up ? v[i + H2] : v[i];
        v[i] = fmaxf(keep, __shfl_xor_sync(kFull, send, M));
      }
      if (up) off += H2;
      TMax<H2, M / 2>::run(v, lane, off);
    } else {
      v[0] = fmaxf(v[0], __shfl_xor_sync(kFull, v[0], M));
      TMax<1, M / 2>::run(v, lane, off);
    }
  }
};
template <int K>
struct TMax<K, 0> {
  static __device__ __forceinline__ void run(float*, int, int&) {}
};

// Sum over the warp, returned to every lane.
__device__ __forceinline__ float warp_allsum(float x) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(kFull, x, m);
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

// Ring slot of record j (0-based) for a buffer starting at slot st < R, with j < R.
__device__ __forceinline__ int ring_slot(int st, int j, int R) {
  const int x = st + j;
  return x >= R ? x - R : x;
}
__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
// Packed pairs of fp32 for fma.rn.f32x2 (two independent IEEE fmas per instruction).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
// the first element of a pair sits in the low 32 bits
__device__ __forceinline__ float lo2(f32x2 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(f32x2 v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// ------------------------------------------------------------ quantize a warp's rows
// The warp holds KR rows; row kk is covered by LPR lanes with 4 consecutive
// elements (x[kk]) each. Writes the rows' codes and scales into the head's read
// copy. The row and block maxima use transposed reductions, so each scale is
// computed once, by the lane that ends up holding its maximum, and broadcast.
__device__ __forceinline__ float absmax4(const float4 x) {
  return fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
}
template <int RF, int LPR, int KR>
__device__ __forceinline__ void quantize_rows(const float4 (&x)[KR], int lane, int row0, int row_step, int P, int N,
                                              uint8_t* head_copy, int bsc_off, int rsc_off) {
  static_assert(KR <= LPR && (LPR % KR) == 0 && KR >= 4, "row maxima need KR <= LPR");
  constexpr int LPK = LPR / KR;  // lanes that end up holding one row's maximum
  const int col4 = lane % LPR;
  const int seg = lane - col4;   // first lane of this lane's row segment
  // row k of the warp is row0 + k * row_step (rows at or beyond P hold zeros)
  float a[KR];
#pragma unroll
  for (int kk = 0; kk < KR; ++kk) a[kk] = absmax4(x[kk]);
  int off = 0;
  TMax<KR, LPR / 2>::run(a, lane, off);  // lane: the maximum of row `off`
  const float am = a[0];
  const bool live = am > 7.888609052210118e-31f;  // 2^-100
  const bool owner = (lane & (LPK - 1)) == 0;
  const int orow = row0 + off * row_step;
  if constexpr (RF == kRfE4m3) {
    const float inv_own = live ? __fdiv_rn(448.f, am) : 0.f;
    if (owner && orow < P) *reinterpret_cast<float*>(head_copy + rsc_off + orow * 4) = live ? __fdiv_rn(am, 448.f) : 0.f;
#pragma unroll
    for (int kk = 0; kk < KR; ++kk) {
      const float inv = __shfl_sync(kFull, inv_own, seg + kk * LPK);
      const uint32_t c = enc_e4m3x4(__fmul_rn(x[kk].x, inv), __fmul_rn(x[kk].y, inv), __fmul_rn(x[kk].z, inv),
                                    __fmul_rn(x[kk].w, inv));
      const int row = row0 + kk * row_step;
      if (row < P) *reinterpret_cast<uint32_t*>(head_copy + (size_t)row * N + col4 * 4) = c;
    }
  } else {
    const float sr_own = live ? __fdiv_rn(am, 2688.f) : 0.f;
    if (owner && orow < P) *reinterpret_cast<float*>(head_copy + rsc_off + orow * 4) = sr_own;
    float sr[KR];
#pragma unroll
    for (int kk = 0; kk < KR; ++kk) sr[kk] = __shfl_sync(kFull, sr_own, seg + kk * LPK);
    // 16-element blocks are 4 lanes: transposed maximum over them
    constexpr int VB = KR / 4;  // rows per lane after it
    float bm[KR];
#pragma unroll
    for (int kk = 0; kk < KR; ++kk) bm[kk] = absmax4(x[kk]);
    int boff = 0;
    TMax<KR, 2>::run(bm, lane, boff);  // lane: block maxima of rows boff .. boff + VB - 1
    float r[VB];
#pragma unroll
    for (int i = 0; i < VB; ++i) {
      float s_r = sr[0];
#pragma unroll
      for (int kk = 1; kk < KR; ++kk) s_r = (kk == boff + i) ? sr[kk] : s_r;
      const float d6 = __fmul_rn(6.f, s_r);
      const float ratio = d6 > 0.f ? __fdiv_rn(bm[i], d6) : 0.f;
      const uint32_t sb = enc_e4m3(ratio);
      const float d = __fmul_rn(dec_e4m3(sb), s_r);
      r[i] = d > 0.f ? __fdiv_rn(1.f, d) : 0.f;
      const int row = row0 + (boff + i) * row_step;
      if (row < P) head_copy[bsc_off + row * (N / 16) + (col4 >> 2)] = (uint8_t)sb;
    }
#pragma unroll
    for (int kk = 0; kk < KR; ++kk) {
      const float rk = __shfl_sync(kFull, r[kk % VB], (lane & ~3) + kk / VB);
      const uint32_t c = enc_e2m1x4(__fmul_rn(x[kk].x, rk), __fmul_rn(x[kk].y, rk), __fmul_rn(x[kk].z, rk),
                                    __fmul_rn(x[kk].w, rk));
      const int row = row0 + kk * row_step;
      if (row < P) *reinterpret_cast<uint16_t*>(head_copy + (size_t)row * (N / 2) + col4 * 2) = (uint16_t)c;
    }
  }
}

// ------------------------------------------------------------ FP16 checkpoint
// Philox4x32 with 10 rounds (Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11): per round the 64-bit products of c0 and
// c2 with the two multipliers are split into halves and mixed with c1, c3 and
// the key; the key advances by the Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const unsigned long long m0 = (unsigned long long)0xD2511F53u * c.x;  // one widening multiply each
    const unsigned long long m1 = (unsigned long long)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(m1 >> 32) ^ c.y ^ k.x, (uint32_t)m1, (uint32_t)(m0 >> 32) ^ c.w ^ k.y, (uint32_t)m0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}
// The generator words of the group of four checkpoint elements starting at
// element e (a multiple of 4) at a flush epoch: counter (e / 4 low and high
// words, epoch, 0), key the seed.
__device__ __forceinline__ uint4 sr_words(size_t e, uint32_t epoch, unsigned long long seed) {
  const unsigned long long grp = (unsigned long long)e >> 2;
  return philox4x32_10(make_uint4((uint32_t)grp, (uint32_t)(grp >> 32), epoch, 0u),
                       make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
}
// binary32 -> binary16 bits by stochastic rounding with the 32-bit word r: with
// lo = |x| rounded toward zero and hi the next binary16 away from zero, hi is
// taken when r < floor(frac 2^32), frac = (|x| - lo) / (hi - lo). The result
// saturates to +-65504 and keeps the sign; NaN gives 0x7E00.
// Branch-free on the bit pattern. With e the biased exponent and m the significand
// with its leading one, Z = floor(m 2^(32 - s)), s = clamp(126 - e, 13, 63), is |x|
// in units of the binary16 spacing at |x| (2^-24 below 2^-14, 2^(e - 137) above)
// as a 32.32 fixed-point number, its low word floor(frac 2^32). Adding 2^32 - 1 - r
// carries into the high word exactly when r < that fraction word, and the high word
// plus (max(e, 113) - 113) 2^10 is the binary16 magnitude. For e = 0 (zero, binary32
// subnormals) the shift of 63 leaves Z = 0, so the leading one added to m is harmless.
__device__ __forceinline__ uint32_t sr_f16_bits(float x, uint32_t r) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t au = u & 0x7FFFFFFFu;
  const uint32_t e = au >> 23;
  const uint32_t m = (au & 0x7FFFFFu) | 0x800000u;
  const int sh = min(max(126 - (int)e, 13), 63);
  const unsigned long long Z = ((unsigned long long)m << 32) >> sh;
  uint32_t mag = (uint32_t)((Z + (unsigned long long)(~r)) >> 32) + ((max(e, 113u) - 113u) << 10);
  mag = min(mag, 0x7BFFu) | ((u >> 16) & 0x8000u);
  return au > 0x7F800000u ? 0x7E00u : mag;
}
// Four values and the four words of one generator call -> two binary16x2 words.
__device__ __forceinline__ uint2 sr_f16x4(const float4& a, const uint4& w) {
  return make_uint2(sr_f16_bits(a.x, w.x) | (sr_f16_bits(a.y, w.y) << 16),
                    sr_f16_bits(a.z, w.z) | (sr_f16_bits(a.w, w.w) << 16));
}
// Two binary32 values -> binary16x2 (lo in the low half), round to nearest even,
// saturating to +-65504 (the round-to-nearest store, two elements per instruction).
__device__ __forceinline__ uint32_t rn_f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Four consecutive checkpoint elements as float4, from an FP32 or FP16 tile.
template <bool F16>
__device__ __forceinline__ float4 ld_tile4(const uint8_t* tile, size_t e) {
  if constexpr (F16) {
    const uint2 u = *reinterpret_cast<const uint2*>(tile + e * 2);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  } else {
    return *reinterpret_cast<const float4*>(tile + e * 4);
  }
}

// ============================================================================
// The head kernel.
// ============================================================================
// Records are numbered j = 0..J-1 in arrival order after the checkpoint:
// committed records j < c live in the ring at slot (start + j) mod R; the
// decode step's own record is j = c; verify drafts are j = c..c+T-1.
//
// Warp roles, all walking the CTA's heads in the same order:
//   tile warp     bulk TMA of each head tile into a ring of `stages` tile stages
//   gather warp   cp.async of alpha_j and v_j into a deeper ring of `slots`
//                 record slots, and of k_j and the queries into two group areas;
//                 it runs ahead of the tiles so record latency stays hidden
//   coefficients  per head: the decay scan g_{j+1:h}, and the value term
//                 sum_j c_j v_j (non-flush), the scaled values g v_j (fold) or
//                 the verify weights, published in the record slot; the appends
//   dot warps     stream the tile: rows . q, the reduction, the output (and the
//                 fold's rank-J update, store and read-copy refresh)
template <int MODE, int N, typename TIn, int RF>
__global__ void __launch_bounds__(kThreads, 1) head_kernel(const Params p) {
  constexpr int LPR = N / 4;     // lanes per FP32 row (4 columns per lane)
  constexpr int RPI = 32 / LPR;  // rows per warp instruction
  static_assert(LPR >= 1 && LPR <= 32 && (32 % LPR) == 0, "N must be 4..128, power of two");
  constexpr int ES = In<TIn>::kBytes;
  constexpr bool kAppendMode = (MODE == kDecode || MODE == kVerify);
  constexpr bool kGroupData = (MODE != kQuant);
  constexpr bool kQuery = (MODE == kDecode || MODE == kVerify || MODE == kConv || MODE == kSnap);
  constexpr bool kDrafts = (MODE == kVerify || MODE == kSnap);  // inputs carry a draft axis [B,T,...]
  constexpr bool kCopyRF = (RF == kRfE4m3 || RF == kRfE2m1);    // a low-precision read copy exists
  constexpr bool kF16 = (RF == kCkF16);                          // the checkpoint itself is FP16
  constexpr int CKES = kF16 ? 2 : 4;                             // checkpoint bytes per element
  constexpr bool kDel = (RF == kDelta);                          // gated delta-rule layer
  // decode: the tile lane brings each head's new record into its slot (the gather
  // lane, far ahead, the buffered ones); other modes: the gather lane brings all
  constexpr bool kTileNew = (MODE == kDecode);
  constexpr int kSbOff = (kRMax + kTMax) * 4;                    // delta: slot offset of the write strengths
  constexpr int kCoefOff = 16;  // floats before the per-row coefficients

  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  // bars: tfull[kMaxStages], tempty[kMaxStages], sfull[kMaxSlots], scoef[kMaxSlots],
  //       sempty[kMaxSlots], gfull[2], gempty[2], end; then the abort flag
  const uint32_t tfull0 = smem_u32(bars), tempty0 = smem_u32(bars + kMaxStages);
  const uint32_t sfull0 = smem_u32(bars + 2 * kMaxStages), scoef0 = sfull0 + 8 * kMaxSlots;
  const uint32_t sempty0 = scoef0 + 8 * kMaxSlots;
  const uint32_t gfull0 = sempty0 + 8 * kMaxSlots, gempty0 = gfull0 + 16;
  const uint32_t end_bar = gempty0 + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kMaxStages + 3 * kMaxSlots + 5);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Launched as a programmatic dependent of the previous kernel in the stream:
  // the next launch may be scheduled now, and nothing here touches global
  // memory before the previous grid has completed.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // kFlush with a list: heads are numbered over the listed sequences only
  const bool listed = (MODE == kFlush) && p.flist != nullptr;
  const long long total = listed ? (long long)min(max(*p.fcount, 0), p.B) * p.H : (long long)p.B * p.H;
  auto seq_of = [&](int vb) -> int { return listed ? p.flist[vb] : vb; };
  const long long h0 = (long long)blockIdx.x * total / gridDim.x;
  const long long h1 = (long long)(blockIdx.x + 1) * total / gridDim.x;
  const int nq = kDrafts ? p.T : 1;

  // Layout: the non-flush one unless one of this CTA's sequences flushes now.
  // Every thread decides alike from the same counts, which no CTA changes
  // before all CTAs of the sequence are done with them.
  bool lean = false;
  if constexpr (MODE == kDecode) {
    if (h1 > h0 && (p.nf_ok || p.skip_nonflush)) {
      bool need = false;
      const int b_first = (int)(h0 / p.H), b_last = (int)((h1 - 1) / p.H);
      for (int b = b_first + lane; b <= b_last; b += 32) {
        const int c = p.count[b];
        need |= (c >= 0 && c + 1 <= p.R && c + 1 >= p.L);
      }
      const bool none = !__any_sync(kFull, need);  // no sequence of this CTA flushes now
      lean = p.nf_ok && none;
      if (p.skip_nonflush && none) {
        // Nothing to fold (the warp-per-head kernel took the outputs and appends):
        // warp 0's lanes only advance the pointers, with the same tickets as below.
        if (warp == 0) {
          for (int b = b_first + lane; b <= b_last; b += 32) {
            const int c = p.count[b];
            if (c < 0 || c + 1 > p.R) {
              atomicOr(p.err, kErrCapacity);
              continue;
            }
            const long long lo = max(h0, (long long)b * p.H), hi = min(h1, (long long)(b + 1) * p.H);
            const int n_b = (int)(hi - lo);
            __threadfence();
            const int prev = atomicAdd(p.ticket + b, n_b);
            if (prev + n_b == p.H) {
              __threadfence();
              p.count[b] = c + 1;
              p.ticket[b] = 0;
            }
          }
        }
        return;
      }
    }
  }
  Layout lay;  // field by field, so that no copy goes through local memory
  lay.stages = lean ? p.lay[1].stages : p.lay[0].stages;
  lay.stage_bytes = lean ? p.lay[1].stage_bytes : p.lay[0].stage_bytes;
  lay.slots = lean ? p.lay[1].slots : p.lay[0].slots;
  lay.slot_bytes = lean ? p.lay[1].slot_bytes : p.lay[0].slot_bytes;
  lay.slot_off = lean ? p.lay[1].slot_off : p.lay[0].slot_off;
  lay.sv_off = lean ? p.lay[1].sv_off : p.lay[0].sv_off;
  lay.sc_off = lean ? p.lay[1].sc_off : p.lay[0].sc_off;
  lay.nv_off = lean ? p.lay[1].nv_off : p.lay[0].nv_off;
  lay.dgroups = lean ? p.lay[1].dgroups : p.lay[0].dgroups;

  // The parity waits need every ring to be a multiple of the consumers that take
  // its entries in turn (see the host plan). Refuse any other plan.
  if (lay.dgroups < 1 || (lay.dgroups & (lay.dgroups - 1)) != 0 || lay.stages < lay.dgroups ||
      lay.stages > kMaxStages || lay.slots > kMaxSlots ||
      lay.stages % lay.dgroups != 0 || lay.slots % kNCoef != 0 || lay.slots % lay.dgroups != 0 ||
      kNDW % lay.dgroups != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrPlan);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < lay.stages; ++s) {
      mbar_init(tfull0 + 8 * s, 1);
      mbar_init(tempty0 + 8 * s, kNDW / lay.dgroups);  // the warps of the head's dot group
    }
    for (int s = 0; s < lay.slots; ++s) {
      // the gather lane's bytes, the new records' bytes and their cp.async decays
      mbar_init(sfull0 + 8 * s, kTileNew ? 3 : 2);
      mbar_init(scoef0 + 8 * s, 1);
      mbar_init(sempty0 + 8 * s, kNDW / lay.dgroups + 1);  // the head's dot group + its coefficient warp
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(gfull0 + 8 * s, 1);  // lane 0's key and query bytes
      mbar_init(gempty0 + 8 * s, kNDW + kNCoef);
    }
    mbar_init(end_bar, kThreads);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // Per-sequence plan, identical in every role: all read the same count[b], and
  // nobody writes pointers before every CTA of b has finished.
  auto seq_plan = [&](int b, int& c, int& st, bool& load, bool& flush, bool& bad) {
    c = 0; st = 0; flush = false; bad = false; load = true;
    if constexpr (MODE == kConv || MODE == kQuant) {
      flush = true;
      return;
    }
    if constexpr (MODE == kSnap) {  // no ring: the T drafts are all new records; st = state slot
      st = p.cur[b];
      bad = st < 0 || st >= p.nslot;
      load = !bad;
      return;
    }
    c = p.count[b];
    st = p.start[b];
    if constexpr (MODE == kDecode) {
      bad = (c + 1 > p.R) || c < 0;
      flush = !bad && (c + 1 >= p.L);
      load = !bad && (flush || !p.skip_nonflush);
    } else if constexpr (MODE == kVerify) {
      bad = (c + p.T > p.R) || c < 0;
      load = !bad;
    } else {  // kFlush
      flush = (c >= p.min_count) && (c > 0) && (c <= p.R);
      load = flush;
    }
  };
  auto records = [&](int c) -> int {
    if constexpr (MODE == kDecode) return c + 1;
    else if constexpr (MODE == kVerify) return c + p.T;
    else if constexpr (MODE == kFlush) return c;
    else if constexpr (MODE == kConv) return 1;
    else if constexpr (MODE == kSnap) return p.T;
    else return 0;
  };

  // Move a head loop past the rest of the current sequence (virtual index it.b):
  // the loop's increment then lands on the next sequence's first head.
  auto skip_seq = [&](long long& gh, HeadIter& it) {
    gh = min(h1, (long long)(it.b + 1) * p.H) - 1;
    it.init(gh, p.H, p.HPG);
  };

  // Ring positions (index, phase parity) of the tile stages and record slots.
  int ts = 0, tph = 0, rs = 0, rph = 0;
  auto tile_next = [&]() {
    if (++ts == lay.stages) { ts = 0; tph ^= 1; }
  };
  auto slot_next = [&]() {
    if (++rs == lay.slots) { rs = 0; rph ^= 1; }
  };

  bool ok = true;
  if (warp == kTileWarp) {
    // ====================================================================== tile warp
    // In decode it also brings each head's new record (from the call's inputs)
    // into the head's record slot: the value row by bulk copy, the decay (and
    // write strength) by 4-byte cp.async.
    if (lane == 0) {
      int li = 0, cur_b = -1, c = 0, st = 0;
      bool load = false, flush = false, bad = false;
      const uint32_t rbytes = (uint32_t)p.P * ES;
      HeadIter it;
      it.init(h0, p.H, p.HPG);
      for (long long gh = h0; gh < h1; ++gh, it.next(p.H, p.HPG)) {
        const int b = seq_of(it.b), hh = it.hh;
        if (b != cur_b) {
          cur_b = b;
          seq_plan(b, c, st, load, flush, bad);
        }
        if (!load) {  // past the rest of this sequence in one step
          skip_seq(gh, it);
          continue;
        }
        if constexpr (kTileNew) {
          if (li >= lay.slots && !mbar_wait(sempty0 + 8 * rs, rph ^ 1, abort_flag, p.err)) { ok = false; break; }
          const int nnew = records(c) - c;
          const uint32_t sbar = sfull0 + 8 * rs;
          const uint32_t sdst = smem_u32(smem + lay.slot_off + (size_t)rs * lay.slot_bytes);
          mbar_arrive_tx(sbar, (uint32_t)nnew * rbytes);
          for (int t = 0; t < nnew; ++t) {
            const size_t nrow = kDrafts ? ((size_t)b * p.T + t) * p.H + hh : (size_t)b * p.H + hh;
            cp_async4(sdst + 4 * (kRMax + t), p.alpha + nrow);
            if constexpr (kDel) cp_async4(sdst + kSbOff + 4 * (kRMax + t), p.beta + nrow);
            const uint32_t vdst = kDel ? sdst + lay.nv_off + t * rbytes : sdst + lay.sv_off + (c + t) * rbytes;
            tma_load_1d(vdst, reinterpret_cast<const uint8_t*>(p.v) + nrow * rbytes, rbytes, sbar);
          }
          cp_async_arrive(sbar);  // completes with this lane's decay copies
          slot_next();
        }
        if (li >= lay.stages && !mbar_wait(tempty0 + 8 * ts, tph ^ 1, abort_flag, p.err)) { ok = false; break; }
        const bool from_copy = kCopyRF && (MODE == kDecode) && !flush;
        const size_t hrow = (size_t)b * p.H + it.hh;
        size_t srow = hrow;  // kSnap: the head's row in the sequence's current state slot
        if constexpr (MODE == kSnap) srow += (size_t)st * ((size_t)p.B * p.H);
        const void* src = from_copy ? (const void*)(p.copy + hrow * p.head_stride)
                                    : (const void*)(reinterpret_cast<const uint8_t*>(p.ckpt) + srow * p.P * N * CKES);
        const uint32_t bytes = from_copy ? (uint32_t)p.head_stride : (uint32_t)(p.P * N * CKES);
        mbar_arrive_tx(tfull0 + 8 * ts, bytes);
        tma_load_1d(smem_u32(smem + (size_t)ts * lay.stage_bytes), src, bytes, tfull0 + 8 * ts);
        tile_next();
        ++li;
      }
      cp_async_wait_all();
      if (!ok) {  // drain the bulk copies still in flight (bounded), then leave
        volatile int dummy = 0;
        for (int k = 0; k < lay.stages && k < li; ++k) {
          const int i = li - 1 - k;
          mbar_wait(tfull0 + 8 * (i % lay.stages), (i / lay.stages) & 1, &dummy, p.err);
        }
        for (int k = 0; kTileNew && k <= lay.stages && k <= li; ++k) {  // its latest record-slot fills
          const int i = li - k;
          mbar_wait(sfull0 + 8 * (i % lay.slots), (i / lay.slots) & 1, &dummy, p.err);
        }
      }
    }
  } else if (warp == kGatherWarp) {
    // ====================================================================== gather (one lane)
    // Per group: the keys and queries into a group area; per head: the records
    // into a slot. Committed records sit in the ring at slots st .. st + c - 1
    // (mod R), so their key rows, value rows and decays are at most two
    // contiguous runs each; every run is one bulk copy. New records come from
    // the call's inputs: one bulk copy per row and a 4-byte cp.async per decay
    // (in decode the tile lane brings the new record's value row and decay).
    if (lane == 0) {
      int li = 0, gi = 0, cur_b = -1, c = 0, st = 0, J = 0;
      long long cur_gg = -1;
      bool load = false, flush = false, bad = false;
      const uint32_t rbytes = (uint32_t)p.P * ES, kbytes = (uint32_t)N * ES;
      HeadIter it;
      it.init(h0, p.H, p.HPG);
      for (long long gh = h0; gh < h1; ++gh, it.next(p.H, p.HPG)) {
        const int b = seq_of(it.b), hh = it.hh, g = it.g;
        const long long gg = (long long)b * p.G + g;
        const size_t hrow = (size_t)b * p.H + hh;
        if (b != cur_b) {
          cur_b = b;
          seq_plan(b, c, st, load, flush, bad);
          if (bad) atomicOr(p.err, kErrCapacity);
          J = records(c);
          cur_gg = -1;
        }
        if (!load) {  // past the rest of this sequence in one step
          skip_seq(gh, it);
          continue;
        }
        const int nnew = J - c;  // records that come from the call's inputs
        if constexpr (kGroupData) {
          if (gg != cur_gg) {
            cur_gg = gg;
            const int gs = gi & 1, guse = gi >> 1;
            if (guse > 0 && !mbar_wait(gempty0 + 8 * gs, (guse - 1) & 1, abort_flag, p.err)) { ok = false; break; }
            const uint32_t gbar = gfull0 + 8 * gs;
            const uint32_t gdst = smem_u32(smem + p.gb_off + gs * p.gb_bytes);
            const size_t grow = (size_t)b * p.G + g;
            mbar_arrive_tx(gbar, (uint32_t)(J + (kQuery ? nq : 0)) * kbytes);
            if (c > 0) {
              const int n1 = min(c, p.R - st);
              const uint8_t* rk = reinterpret_cast<const uint8_t*>(p.ring_k) + grow * p.R * kbytes;
              tma_load_1d(gdst, rk + (size_t)st * kbytes, (uint32_t)n1 * kbytes, gbar);
              if (c > n1) tma_load_1d(gdst + n1 * kbytes, rk, (uint32_t)(c - n1) * kbytes, gbar);
            }
            for (int t = 0; t < nnew; ++t) {
              const size_t krow = kDrafts ? ((size_t)b * p.T + t) * p.G + g : grow;
              tma_load_1d(gdst + (c + t) * kbytes, reinterpret_cast<const uint8_t*>(p.k) + krow * kbytes, kbytes, gbar);
            }
            if constexpr (kQuery) {
              for (int t = 0; t < nq; ++t) {
                const size_t qrow = kDrafts ? ((size_t)b * p.T + t) * p.G + g : grow;
                tma_load_1d(gdst + p.gq_off + t * kbytes, reinterpret_cast<const uint8_t*>(p.q) + qrow * kbytes,
                            kbytes, gbar);
              }
            }
            ++gi;
          }
        }
        if (li >= lay.slots && !mbar_wait(sempty0 + 8 * rs, rph ^ 1, abort_flag, p.err)) { ok = false; break; }
        const uint32_t sbar = sfull0 + 8 * rs;
        const uint32_t sdst = smem_u32(smem + lay.slot_off + (size_t)rs * lay.slot_bytes);
        // slot: decays at [ring slot] (committed) and kRMax + t (new, from the tile
        // lane); value rows in record order (delta-rule layers: the buffered
        // records' pseudo-values (fp32), the new record's v row at nv_off)
        const uint32_t vb = kDel ? (uint32_t)p.P * 4 : rbytes;  // bytes of a buffered value row
        mbar_arrive_tx(sbar, (uint32_t)c * vb + (kTileNew ? 0u : (uint32_t)nnew * rbytes) + (c > 0 ? (uint32_t)p.Rp * 4 : 0u));
        if (c > 0) {
          tma_load_1d(sdst, p.ring_a + hrow * p.Rp, (uint32_t)p.Rp * 4, sbar);
          const int n1 = min(c, p.R - st);
          const uint8_t* rv = reinterpret_cast<const uint8_t*>(p.ring_v) + hrow * p.R * vb;
          tma_load_1d(sdst + lay.sv_off, rv + (size_t)st * vb, (uint32_t)n1 * vb, sbar);
          if (c > n1) tma_load_1d(sdst + lay.sv_off + n1 * vb, rv, (uint32_t)(c - n1) * vb, sbar);
        }
        if constexpr (!kTileNew) {
          for (int t = 0; t < nnew; ++t) {
            const size_t nrow = kDrafts ? ((size_t)b * p.T + t) * p.H + hh : hrow;
            cp_async4(sdst + 4 * (kRMax + t), p.alpha + nrow);
            if constexpr (kDel) cp_async4(sdst + kSbOff + 4 * (kRMax + t), p.beta + nrow);
            const uint32_t vdst = kDel ? sdst + lay.nv_off + t * rbytes : sdst + lay.sv_off + (c + t) * rbytes;
            tma_load_1d(vdst, reinterpret_cast<const uint8_t*>(p.v) + nrow * rbytes, rbytes, sbar);
          }
          cp_async_arrive(sbar);  // completes with this lane's decay copies
        }
        slot_next();
        ++li;
      }
      cp_async_wait_all();
      if (!ok) {  // wait (bounded) for the copies still in flight, then leave
        volatile int dummy = 0;
        for (int k = 0; k < lay.slots && k < li; ++k) {
          const int i = li - 1 - k;
          mbar_wait(sfull0 + 8 * (i % lay.slots), (i / lay.slots) & 1, &dummy, p.err);
        }
        for (int k = 0; k < 2 && k < gi; ++k) {
          const int i = gi - 1 - k;
          mbar_wait(gfull0 + 8 * (i & 1), (i >> 1) & 1, &dummy, p.err);
        }
      }
    }
  } else if (warp >= kCoef0 && warp < kCoef0 + kNCoef) {
    // ====================================================================== coefficients
    const int cwi = warp - kCoef0;  // this warp takes the loaded heads with index = cwi (mod kNCoef)
    // scratch: [kTMax][kRMax] verify weights; delta: a row of couplings [kRMax]
    float* skq_w = reinterpret_cast<float*>(smem + p.wsc_off) + cwi * kTMax * kRMax;
    int lh = 0, gi = 0, cur_b = -1, c = 0, st = 0, J = 0;
    long long cur_gg = -1;
    bool load = false, flush = false, bad = false;
    float sj = 0.f;  // decode: lane j holds k_j^T q
    float mj = 0.f;  // delta: lane j < c holds k_j^T k_c (the new record's key)
    const uint8_t* cK = smem + p.gb_off;  // the current group area: keys, then queries
    HeadIter it;
    it.init(h0, p.H, p.HPG);
    for (long long gh = h0; gh < h1 && ok; ++gh, it.next(p.H, p.HPG)) {
      const int b = seq_of(it.b), g = it.g;
      const long long gg = (long long)b * p.G + g;
      const size_t hrow = (size_t)b * p.H + it.hh;
      if (b != cur_b) {
        cur_b = b;
        seq_plan(b, c, st, load, flush, bad);
        J = records(c);
        cur_gg = -1;
      }
      if (!load) {  // past the rest of this sequence in one step
        skip_seq(gh, it);
        continue;
      }
      if constexpr (kGroupData) {
        if (gg != cur_gg) {
          cur_gg = gg;
          if (gi > 0) {
            bulk_wait_read();  // key appends from the previous group area have read it
            __syncwarp();
            if (lane == 0) mbar_arrive(gempty0 + 8 * ((gi - 1) & 1));
          }
          const int gs = gi & 1;
          if (!__all_sync(kFull, mbar_wait(gfull0 + 8 * gs, (gi >> 1) & 1, abort_flag, p.err))) { ok = false; break; }
          const uint8_t* gK = smem + p.gb_off + gs * p.gb_bytes;
          const uint8_t* gQ = gK + p.gq_off;
          cK = gK;
          if constexpr (MODE == kDecode || MODE == kVerify) {
            // k_j^T q_t: one pair per lane, N/4 chunks visited from a lane-dependent start
            const int npair = J * nq;
            for (int pr = lane; pr < ((npair + 31) & ~31); pr += 32) {
              float acc = 0.f;
              const int t = (nq == 1) ? 0 : pr / J;
              const int j = pr - t * J;
              if (pr < npair) {
#pragma unroll 8
                for (int i = 0; i < N / 4; ++i) {
                  const int c4 = (i + lane) & (N / 4 - 1);
                  acc += dot4(In<TIn>::lds4(gK, j * N + 4 * c4), In<TIn>::lds4(gQ, t * N + 4 * c4));
                }
              }
              if constexpr (MODE == kDecode) {
                sj = acc;  // npair = J <= 32: one pass, lane j holds k_j^T q
              } else {
                if (pr < npair) skq_w[t * kRMax + j] = acc;
              }
            }
            __syncwarp();
          }
          if constexpr (kDel && MODE == kVerify) {
            // k_j^T k_{c+t}: every record's key against each draft key, rows T..2T-1 of the scratch
            const int npk = J * nq;
            for (int pr = lane; pr < npk; pr += 32) {
              const int t = pr / J, j = pr - t * J;
              float acc = 0.f;
#pragma unroll 8
              for (int i = 0; i < N / 4; ++i) {
                const int c4 = (i + lane) & (N / 4 - 1);
                acc += dot4(In<TIn>::lds4(gK, j * N + 4 * c4), In<TIn>::lds4(gK, (c + t) * N + 4 * c4));
              }
              skq_w[(nq + t) * kRMax + j] = acc;
            }
            __syncwarp();
          }
          if constexpr (kDel && (MODE == kDecode || MODE == kConv)) {  // lane j < c: k_j^T k_c, the new key against the buffered ones
            float acc = 0.f;
            if (lane < c) {
#pragma unroll 8
              for (int t = 0; t < N / 4; ++t) {
                const int c4 = (t + lane) & (N / 4 - 1);
                acc += dot4(In<TIn>::lds4(gK, lane * N + 4 * c4), In<TIn>::lds4(gK, c * N + 4 * c4));
              }
            }
            mj = acc;
          }
          if constexpr (kAppendMode) {  // the group's first head (if this CTA owns it) appends the new keys
            const long long gfirst = (long long)b * p.H + (long long)g * p.HPG;
            const int na = (MODE == kVerify) ? p.T : (flush ? 0 : 1);
            if (cwi == 0 && gfirst >= h0 && lane < na) {  // lane t: one bulk store per new key row
              const size_t grow = (size_t)b * p.G + g;
              const int t = lane;
              bulk_store(reinterpret_cast<uint8_t*>(p.ring_k) + (grow * p.R + ring_slot(st, c + t, p.R)) * N * ES,
                         smem_u32(gK + (c + t) * N * ES), N * ES);
              bulk_commit();
            }
          }
          ++gi;
        }
      }
      if ((lh++ % kNCoef) != cwi) {  // another coefficient warp takes this head
        slot_next();
        continue;
      }
      if (!__all_sync(kFull, mbar_wait(sfull0 + 8 * rs, rph, abort_flag, p.err))) { ok = false; break; }
      uint8_t* slot = smem + lay.slot_off + (size_t)rs * lay.slot_bytes;
      const float* sa = reinterpret_cast<const float*>(slot);  // decays: [ring slot] committed, [kRMax + t] new
      const uint8_t* sv = slot + lay.sv_off;                      // v_j rows, record order
      float* sc = reinterpret_cast<float*>(slot + lay.sc_off);    // coefficients
      // lane j holds alpha of record j
      const float aj = (lane < c) ? sa[ring_slot(st, lane, p.R)] : (lane < J) ? sa[kRMax + lane - c] : 1.f;
      if constexpr (MODE == kVerify && kDel) {
        // Gated delta rule, T drafts after c committed records (draft t is record c + t):
        //   y_t = P_t (S k_{c+t}) + sum_{i<c} D_it (k_i^T k_{c+t}) w_i + sum_{s<t} E_ts w'_s
        //   w'_t = beta_t (v_t - alpha_{c+t} y_t)
        //   o_t = G_t (S q_t) + sum_{i<c} W_it (k_i^T q_t) w_i + sum_{s<=t} F_ts w'_s
        // with P_t = alpha_0 .. alpha_{c+t-1}, G_t = alpha_0 .. alpha_{c+t}, D_it and W_it the
        // decays strictly after record i up to c+t-1 and c+t, E_ts = (alpha_{c+s+1} .. alpha_{c+t-1})
        // (k_{c+s}^T k_{c+t}) and F_ts = (alpha_{c+s+1} .. alpha_{c+t}) (k_{c+s}^T q_t).
        // sc: [t] G_t, [T + t] P_t; [16 + v kRMax + i] the committed weights of vector v
        // (v < T: query t with W_it; v >= T: draft key v - T with D_it); then E [t][4], F [t][4].
        const float sfx = suffix_prod((lane < c) ? aj : 1.f, lane);  // alpha_lane .. alpha_{c-1}
        const float dn = __shfl_down_sync(kFull, sfx, 1);
        const float dpart = (lane < 31) ? dn : 1.f;                  // alpha_{lane+1} .. alpha_{c-1}
        const float call = __shfl_sync(kFull, sfx, 0);                // alpha_0 .. alpha_{c-1}
        float pre = 1.f;                                               // alpha_c .. alpha_{c+t-1}
        for (int t = 0; t < p.T; ++t) {
          const float inc = pre * sa[kRMax + t];
          if (lane == 0) {
            sc[t] = call * inc;
            sc[p.T + t] = call * pre;
          }
          const bool com = lane < c;
          sc[kCoefOff + t * kRMax + lane] = com ? dpart * inc * skq_w[t * kRMax + lane] : 0.f;
          sc[kCoefOff + (p.T + t) * kRMax + lane] = com ? dpart * pre * skq_w[(p.T + t) * kRMax + lane] : 0.f;
          pre = inc;
        }
        if (lane < 16) {  // (t, s) = (lane / 4, lane % 4)
          const int t = lane >> 2, s = lane & 3;
          float e = 0.f, f = 0.f;
          if (t < p.T && s <= t) {
            float pe = 1.f;
            for (int u = s + 1; u < t; ++u) pe *= sa[kRMax + u];
            if (s < t) e = pe * skq_w[(p.T + t) * kRMax + c + s];
            f = (s < t ? pe * sa[kRMax + t] : 1.f) * skq_w[t * kRMax + c + s];
          }
          sc[kCoefOff + kTMax * kRMax + lane] = e;
          sc[kCoefOff + kTMax * kRMax + 16 + lane] = f;
        }
      } else if constexpr (MODE == kVerify) {
        // Per query t (records 0 .. c + t): g_{1:c+t+1} into sc[t] and the record
        // weights g_{j+2:c+t+1} (k_j^T q_t) into sc[kCoefOff + t kRMax + j]. One scan
        // covers the committed records; the drafts' decays enter as per-lane running
        // products: record l's weight for query t is
        // (alpha_{l+1} .. alpha_{c-1}) (alpha_{max(l+1,c)} .. alpha_{c+t}).
        const float sfx = suffix_prod((lane < c) ? aj : 1.f, lane);  // alpha_lane .. alpha_{c-1}
        const float dn = __shfl_down_sync(kFull, sfx, 1);
        const float dpart = (lane < 31) ? dn : 1.f;                  // alpha_{lane+1} .. alpha_{c-1}
        const float call = __shfl_sync(kFull, sfx, 0);                // alpha_0 .. alpha_{c-1}
        const int s0 = max(lane + 1 - c, 0);                           // first draft after record lane
        float np = 1.f, nall = 1.f;                                    // drafts s0 .. t; drafts 0 .. t
        for (int t = 0; t < p.T; ++t) {
          const float at = sa[kRMax + t];
          nall *= at;
          if (t >= s0) np *= at;
          const int ht = c + t + 1;
          sc[kCoefOff + t * kRMax + lane] = (lane < ht) ? dpart * np * skq_w[t * kRMax + lane] : 0.f;
          if (lane == 0) sc[t] = call * nall;
        }
      } else if constexpr (kDel) {
        // Gated delta rule through pseudo-values. After records 0..J-1 the state is
        //   gamma S + sum_i W_i w_i k_i^T,  gamma = alpha_0 .. alpha_{J-1}, W_i = alpha_{i+1} .. alpha_{J-1},
        // where the ring keeps w_i = beta_i (v_i - alpha_i y_i), y_i = (state before record i) k_i.
        // The new record c gets y_c = P_c (S k_c) + sum_{i<c} D_ic (k_i^T k_c) w_i with
        // P_c = alpha_0 .. alpha_{c-1} and D_ic = alpha_{i+1} .. alpha_{c-1} (the dot warps
        // hold S), and the output is o = gamma S q + sum_i W_i (k_i^T q) w_i.
        // sc: [0] gamma, [2] P_c, [3] alpha_c, [4] beta_c, [5] k_c^T q,
        //     [16 + i] W_i k_i^T q and [16 + kRMax + i] D_ic k_i^T k_c (i < c), and for a
        //     fold [16 + 2 kRMax + i P + p] W_i w_i[p] (buffered records; the dot warps add record c)
        const int cn = (MODE == kFlush) ? J : c;  // records from the ring
        const float sfx = suffix_prod((lane < cn) ? aj : 1.f, lane);  // alpha_lane .. alpha_{cn-1}
        const float dn = __shfl_down_sync(kFull, sfx, 1);
        const float dex = (lane < 31) ? dn : 1.f;  // alpha_{lane+1} .. alpha_{cn-1}
        const float anew = (MODE == kFlush) ? 1.f : __shfl_sync(kFull, aj, cn);
        const float wsuf = dex * anew;             // W_lane for lane < cn
        const float pc = __shfl_sync(kFull, sfx, 0);
        const float sqc = __shfl_sync(kFull, sj, cn);
        if (lane == 0) {
          sc[0] = pc * anew;
          sc[2] = pc;
          sc[3] = anew;
          sc[4] = (MODE == kFlush) ? 0.f : reinterpret_cast<const float*>(slot + kSbOff)[kRMax];
          sc[5] = sqc;
        }
        sc[kCoefOff + lane] = (lane < cn) ? wsuf * sj : 0.f;
        sc[kCoefOff + kRMax + lane] = (lane < cn) ? dex * mj : 0.f;
        if (flush) {  // the fold's scaled pseudo-values of the buffered records
          const float* sw = reinterpret_cast<const float*>(sv);
          float* su = sc + kCoefOff + 2 * kRMax;
          for (int j = 0; j < cn; ++j) {
            const float wj = __shfl_sync(kFull, wsuf, j);
            for (int r = 2 * lane; r < p.P; r += 64) {
              const float2 w2 = *reinterpret_cast<const float2*>(sw + j * p.P + r);
              *reinterpret_cast<float2*>(su + j * p.P + r) = make_float2(wj * w2.x, wj * w2.y);
            }
          }
        }
      } else if constexpr (MODE != kSnap) {
        const float incl = suffix_prod(aj, lane);
        const float nxt = __shfl_down_sync(kFull, incl, 1);
        const float wj = (lane < 31) ? nxt : 1.f;  // lane j: weight g_{j+2:J} of record j
        if (lane == 0) sc[0] = incl;               // g_{1:J}
        if (flush) {
          // fold: scaled values u_j[p] = g_{j+2:J} v_j[p]; lane handles row pairs 2*lane + 64 m
#pragma unroll 4
          for (int j = 0; j < J; ++j) {
            const float wjj = __shfl_sync(kFull, wj, j);
            for (int r = 2 * lane; r < p.P; r += 64) {
              const float2 v2 = In<TIn>::lds2(sv, j * p.P + r);
              *reinterpret_cast<float2*>(sc + kCoefOff + j * p.P + r) = make_float2(wjj * v2.x, wjj * v2.y);
            }
          }
        } else if constexpr (MODE == kDecode) {
          // non-flush: the record weights c_j = g_{j+2:J} (k_j^T q); the dot warps
          // add sum_j c_j v_j[p] inside their row reductions
          sc[kCoefOff + lane] = (lane < J) ? wj * sj : 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(scoef0 + 8 * rs);  // coefficients published
      if constexpr (kAppendMode) {  // the new decays and value rows go to the ring
        // (delta-rule layers: the dot warps append the pseudo-value row instead)
        const int na = (MODE == kVerify) ? p.T : (flush ? 0 : 1);
        if (lane < na) p.ring_a[hrow * p.Rp + ring_slot(st, c + lane, p.R)] = sa[kRMax + lane];
        if constexpr (MODE == kVerify && !kDel) {
          // the T value rows: one bulk store per contiguous ring run (at most two),
          // issued by one lane; the slot is released once the copies have read it
          if (lane == 0 && na > 0) {
            const int s1 = ring_slot(st, c, p.R);
            const int n1 = min(na, p.R - s1);
            uint8_t* rv = reinterpret_cast<uint8_t*>(p.ring_v) + hrow * p.R * p.P * ES;
            bulk_store(rv + (size_t)s1 * p.P * ES, smem_u32(sv + c * p.P * ES), n1 * p.P * ES);
            if (na > n1) bulk_store(rv, smem_u32(sv + (c + n1) * p.P * ES), (na - n1) * p.P * ES);
            bulk_commit();
            bulk_wait_read();
          }
        } else if constexpr (!kDel) {
          const int chp = p.P * ES / 16;
          for (int t = 0; t < na; ++t) {  // 16-byte stores spread over the lanes
            uint8_t* dst = reinterpret_cast<uint8_t*>(p.ring_v) + (hrow * p.R + ring_slot(st, c + t, p.R)) * p.P * ES;
            for (int ch = lane; ch < chp; ch += 32)
              *reinterpret_cast<uint4*>(dst + ch * 16) = *reinterpret_cast<const uint4*>(sv + (c + t) * p.P * ES + ch * 16);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sempty0 + 8 * rs);  // this warp is done with the slot
      slot_next();
    }
    bulk_wait_all();  // every append has reached global memory before the warp leaves
  } else {
    // ====================================================================== dot warps
    const int col4 = lane % LPR, rsub = lane / LPR;
    int gi = 0, cur_b = -1, c = 0, st = 0, J = 0;
    long long cur_gg = -1;
    bool load = false, flush = false, bad = false;
    int ep = 0;  // FP16 checkpoint: the sequence's flush epoch (rounding counter)
    const uint8_t* gK = smem + p.gb_off;
    const uint8_t* gQ = gK + p.gq_off;
    float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int CPL = (RF == kRfE2m1) ? 32 : 16;  // copy-tile columns per lane
    constexpr int LPRc = (N / CPL) > 0 ? (N / CPL) : 1;
    constexpr int RPIc = 32 / LPRc;
    constexpr int KRc = (kKR * 4 / CPL) > 0 ? (kKR * 4 / CPL) : 1;
    float qc[(kCopyRF && MODE == kDecode) ? CPL : 1];
    // FP32 non-flush rows (N >= 64): LP16 lanes per row, 16 columns per lane as
    // 4 chunks of 4 interleaved over the row's lanes (each quarter warp reads
    // 128 contiguous bytes: no bank conflicts); q16 holds the matching q values.
    constexpr bool kWideRows = ((RF == kRfNone || kF16 || kDel) && MODE == kDecode && N >= 64);
    constexpr int LP16 = kWideRows ? N / 16 : 1;
    float q16[kWideRows ? 16 : 1];
    float k16[kDel ? 16 : 1];  // delta-rule layers: the new record's key, same columns as q16
    const int wpg = kNDW / lay.dgroups;                 // warps per dot group
    const int dgrp = warp / wpg, wr = warp - dgrp * wpg;  // this warp's group and rank in it
    const int rows_pass = wpg * kKR * RPI;
    const int npass = (p.P + rows_pass - 1) / rows_pass;
    int lh = 0;  // loaded heads seen
    HeadIter it;
    it.init(h0, p.H, p.HPG);
    for (long long gh = h0; gh < h1 && ok; ++gh, it.next(p.H, p.HPG)) {
      const int b = seq_of(it.b), hh = it.hh, g = it.g;
      const long long gg = (long long)b * p.G + g;
      const size_t hrow = (size_t)b * p.H + hh;
      if (b != cur_b) {
        cur_b = b;
        seq_plan(b, c, st, load, flush, bad);
        J = records(c);
        cur_gg = -1;
        if constexpr (kF16) ep = p.epoch[b];
      }
      if (!load) {  // past the rest of this sequence in one step
        skip_seq(gh, it);
        continue;
      }
      if constexpr (kGroupData) {
        if (gg != cur_gg) {
          cur_gg = gg;
          if (gi > 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(gempty0 + 8 * ((gi - 1) & 1));
          }
          const int gs = gi & 1;
          if (!__all_sync(kFull, mbar_wait(gfull0 + 8 * gs, (gi >> 1) & 1, abort_flag, p.err))) { ok = false; break; }
          gK = smem + p.gb_off + gs * p.gb_bytes;
          gQ = gK + p.gq_off;
          if constexpr (MODE == kDecode || MODE == kConv) q4 = In<TIn>::lds4(gQ, col4 * 4);
          if constexpr (kWideRows && !kF16) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const float4 qq = In<TIn>::lds4(gQ, (c4 * LP16 + lane % LP16) * 4);
              q16[4 * c4] = qq.x; q16[4 * c4 + 1] = qq.y; q16[4 * c4 + 2] = qq.z; q16[4 * c4 + 3] = qq.w;
              if constexpr (kDel) {
                const float4 kq = In<TIn>::lds4(gK, c * N + (c4 * LP16 + lane % LP16) * 4);
                k16[4 * c4] = kq.x; k16[4 * c4 + 1] = kq.y; k16[4 * c4 + 2] = kq.z; k16[4 * c4 + 3] = kq.w;
              }
            }
          }
          if constexpr (kWideRows && kF16) {  // two chunks of 8 halves per lane
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
              for (int hq = 0; hq < 2; ++hq) {
                const float4 qq = In<TIn>::lds4(gQ, (c * LP16 + lane % LP16) * 8 + 4 * hq);
                q16[8 * c + 4 * hq] = qq.x; q16[8 * c + 4 * hq + 1] = qq.y;
                q16[8 * c + 4 * hq + 2] = qq.z; q16[8 * c + 4 * hq + 3] = qq.w;
              }
            }
          }
          if constexpr (kCopyRF && MODE == kDecode) {
#pragma unroll
            for (int i = 0; i < CPL; ++i) qc[i] = In<TIn>::lds(gQ, (lane % LPRc) * CPL + i);
          }
          ++gi;
        }
      }
      if ((lh++ & (lay.dgroups - 1)) != dgrp) {  // another dot group takes this head (dgroups: power of two)
        tile_next();
        slot_next();
        continue;
      }
      // the coefficient warp arrives only after the record gathers landed, so
      // its barrier also covers alpha_j and v_j
      const bool got = mbar_wait(tfull0 + 8 * ts, tph, abort_flag, p.err) &&
                       mbar_wait(scoef0 + 8 * rs, rph, abort_flag, p.err);
      if (!__all_sync(kFull, got)) { ok = false; break; }
      const uint8_t* tile = smem + (size_t)ts * lay.stage_bytes;
      const float* tf = reinterpret_cast<const float*>(tile);
      const uint8_t* slot = smem + lay.slot_off + (size_t)rs * lay.slot_bytes;
      const uint8_t* sv = slot + lay.sv_off;
      const float* sc = reinterpret_cast<const float*>(slot + lay.sc_off);

      if constexpr (MODE == kVerify) {
        // ================================================ verify (T queries)
        // o[t][row] = g_{1:c+t+1} (S q_t)[row] + sum_j w_tj v_j[row]. The lanes of a
        // row split the records (lane k of the row takes j = k, k + lanes, ...) and
        // add their share to the scaled dot before the row reduction, so the value
        // term costs no shuffles. w_tj = 0 for records that query t does not see.
        const float* cw = sc + kCoefOff;  // [kTMax][kRMax]
        if constexpr (kDel) {
          // Gated delta rule. Per row, 2T sums as the outer-product verify forms them,
          // over the vectors q_0 .. q_{T-1}, k_c .. k_{c+T-1} (scales and committed
          // weights from the coefficient warps), kept in a per-warp scratch of 32 rows;
          // then, one lane per row for 32 rows at a time, the chain over the drafts that
          // forms each draft's pseudo-value w'_t (appended to the ring) and its output.
          constexpr int LPV = N / 16, RPW = 32 / LPV, KWV = 2, JI = kRMax / LPV, ROWS = KWV * RPW;
          constexpr int MB = 32 / ROWS;  // row groups per chain batch
          constexpr int SROW = 8;        // scratch floats per row: 2T <= 8
          static_assert(MB * ROWS == 32, "a chain batch is 32 rows");
          const int cl = lane % LPV, rw = lane / LPV;
          const int nvec = 2 * p.T;
          float* dsc = reinterpret_cast<float*>(smem + p.dsc_off) + warp * 32 * SROW;
          const float* sw = reinterpret_cast<const float*>(sv);  // committed pseudo-values [c][P]
          const float* ef = cw + kTMax * kRMax;                  // E [t][4], then F [t][4]
          const float* sa = reinterpret_cast<const float*>(slot);
          const float* sbeta = reinterpret_cast<const float*>(slot + kSbOff);
          int m = 0;  // row group of this warp
          for (int r0 = wr * ROWS; r0 < p.P; r0 += wpg * ROWS, ++m) {
            const int mb = m % MB;
            for (int t0 = 0; t0 < nvec; t0 += kTQ) {
              f32x2 qv[kTQ][8];
              float g[kTQ];
              float wv[JI][kTQ];
#pragma unroll
              for (int tt = 0; tt < kTQ; ++tt) {
                const int v = t0 + tt;
                const bool tv = v < nvec;
                const uint8_t* vec = v < p.T ? gQ + (size_t)v * N * ES : gK + (size_t)(c + v - p.T) * N * ES;
                g[tt] = tv ? sc[v] : 0.f;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                  const float4 qq = tv ? In<TIn>::lds4(vec, (cc * LPV + cl) * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
                  qv[tt][2 * cc] = pk2(qq.x, qq.y);
                  qv[tt][2 * cc + 1] = pk2(qq.z, qq.w);
                }
#pragma unroll
                for (int i = 0; i < JI; ++i) {
                  const int j = cl + LPV * i;
                  wv[i][tt] = (tv && j < c) ? cw[v * kRMax + j] : 0.f;
                }
              }
              float part[KWV * kTQ];
#pragma unroll
              for (int kk = 0; kk < KWV; ++kk) {
                const int row = r0 + kk * RPW + rw;
                float a[kTQ];
#pragma unroll
                for (int tt = 0; tt < kTQ; ++tt) a[tt] = 0.f;
                if (row < p.P) {
                  const float* rp = tf + (size_t)row * N;
                  f32x2 a2[kTQ];
#pragma unroll
                  for (int tt = 0; tt < kTQ; ++tt) a2[tt] = 0ull;
#pragma unroll
                  for (int cc = 0; cc < 4; ++cc) {
                    const ulonglong2 x = *reinterpret_cast<const ulonglong2*>(rp + (cc * LPV + cl) * 4);
#pragma unroll
                    for (int tt = 0; tt < kTQ; ++tt) {
                      a2[tt] = fma2(x.x, qv[tt][2 * cc], a2[tt]);
                      a2[tt] = fma2(x.y, qv[tt][2 * cc + 1], a2[tt]);
                    }
                  }
#pragma unroll
                  for (int tt = 0; tt < kTQ; ++tt) a[tt] = g[tt] * (lo2(a2[tt]) + hi2(a2[tt]));
#pragma unroll
                  for (int i = 0; i < JI; ++i) {
                    const int j = cl + LPV * i;
                    if (j < c) {
                      const float wj = sw[j * p.P + row];
#pragma unroll
                      for (int tt = 0; tt < kTQ; ++tt) a[tt] = fmaf(wv[i][tt], wj, a[tt]);
                    }
                  }
                }
#pragma unroll
                for (int tt = 0; tt < kTQ; ++tt) part[kk * kTQ + tt] = a[tt];
              }
              int off = 0;
              TRed<KWV * kTQ, LPV / 2>::run(part, lane, off);
              constexpr int KF = (KWV * kTQ / LPV) > 0 ? (KWV * kTQ / LPV) : 1;
              constexpr int D = (LPV / (KWV * kTQ)) > 0 ? (LPV / (KWV * kTQ)) : 1;
#pragma unroll
              for (int i = 0; i < KF; ++i) {
                const int kk = (off + i) / kTQ, v = t0 + (off + i) % kTQ;
                if ((cl & (D - 1)) == 0 && v < nvec) dsc[(mb * ROWS + kk * RPW + rw) * SROW + v] = part[i];
              }
            }
            if (mb != MB - 1 && r0 + wpg * ROWS < p.P) continue;  // the batch is not full yet
            __syncwarp();
            const int row = r0 - (mb - lane / ROWS) * (wpg * ROWS) + lane % ROWS;  // lane's row in the batch
            if (lane < (mb + 1) * ROWS && row < p.P) {
              const float* rs = dsc + lane * SROW;
              const uint8_t* nv = slot + lay.nv_off;
              float wd[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                wd[t] = 0.f;
                if (t < p.T) {
                  float y = rs[p.T + t];
#pragma unroll
                  for (int s2 = 0; s2 < t; ++s2) y = fmaf(ef[t * 4 + s2], wd[s2], y);
                  wd[t] = sbeta[kRMax + t] * fmaf(-sa[kRMax + t], y, In<TIn>::lds(nv, t * p.P + row));
                  float o = rs[t];
#pragma unroll
                  for (int s2 = 0; s2 <= t; ++s2) o = fmaf(ef[16 + t * 4 + s2], wd[s2], o);
                  p.o[(((size_t)b * p.T + t) * p.H + hh) * p.P + row] = o;
                  reinterpret_cast<float*>(p.ring_v)[(hrow * p.R + ring_slot(st, c + t, p.R)) * p.P + row] = wd[t];
                }
              }
            }
            __syncwarp();
          }
        } else if constexpr (N >= 64 && !kF16) {
          // LPV lanes per row, 16 columns per lane in 4 interleaved chunks (as the
          // wide non-flush rows); KWV row instructions x kTQ queries per pass.
          constexpr int LPV = N / 16, RPW = 32 / LPV, KWV = 2, JI = kRMax / LPV;
          const int cl = lane % LPV, rw = lane / LPV;
          for (int t0 = 0; t0 < p.T; t0 += kTQ) {
            f32x2 qv[kTQ][8];  // the lane's 16 query columns as 8 column pairs
            float g[kTQ];
            float wv[JI][kTQ];  // this lane's record weights
#pragma unroll
            for (int tt = 0; tt < kTQ; ++tt) {
              const bool tv = t0 + tt < p.T;
              g[tt] = tv ? sc[t0 + tt] : 0.f;
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const float4 qq = tv ? In<TIn>::lds4(gQ, (t0 + tt) * N + (cc * LPV + cl) * 4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                qv[tt][2 * cc] = pk2(qq.x, qq.y);
                qv[tt][2 * cc + 1] = pk2(qq.z, qq.w);
              }
#pragma unroll
              for (int i = 0; i < JI; ++i) {
                const int j = cl + LPV * i;
                wv[i][tt] = (tv && j < J) ? cw[(t0 + tt) * kRMax + j] : 0.f;
              }
            }
            for (int r0 = wr * KWV * RPW; r0 < p.P; r0 += wpg * KWV * RPW) {
              float part[KWV * kTQ];
#pragma unroll
              for (int kk = 0; kk < KWV; ++kk) {
                const int row = r0 + kk * RPW + rw;
                float a[kTQ];
#pragma unroll
                for (int tt = 0; tt < kTQ; ++tt) a[tt] = 0.f;
                if (row < p.P) {
                  const float* rp = tf + (size_t)row * N;
                  f32x2 a2[kTQ];  // column-pair partial sums, packed fp32x2 FMAs
#pragma unroll
                  for (int tt = 0; tt < kTQ; ++tt) a2[tt] = 0ull;
#pragma unroll
                  for (int cc = 0; cc < 4; ++cc) {
                    const ulonglong2 x = *reinterpret_cast<const ulonglong2*>(rp + (cc * LPV + cl) * 4);
#pragma unroll
                    for (int tt = 0; tt < kTQ; ++tt) {
                      a2[tt] = fma2(x.x, qv[tt][2 * cc], a2[tt]);
                      a2[tt] = fma2(x.y, qv[tt][2 * cc + 1], a2[tt]);
                    }
                  }
#pragma unroll
                  for (int tt = 0; tt < kTQ; ++tt) a[tt] = g[tt] * (lo2(a2[tt]) + hi2(a2[tt]));
#pragma unroll
                  for (int i = 0; i < JI; ++i) {
                    const int j = cl + LPV * i;
                    if (j < J) {
                      const float vj = In<TIn>::lds(sv, j * p.P + row);
#pragma unroll
                      for (int tt = 0; tt < kTQ; ++tt) a[tt] = fmaf(wv[i][tt], vj, a[tt]);
                    }
                  }
                }
#pragma unroll
                for (int tt = 0; tt < kTQ; ++tt) part[kk * kTQ + tt] = a[tt];
              }
              int off = 0;
              TRed<KWV * kTQ, LPV / 2>::run(part, lane, off);
              constexpr int KF = (KWV * kTQ / LPV) > 0 ? (KWV * kTQ / LPV) : 1;
              constexpr int D = (LPV / (KWV * kTQ)) > 0 ? (LPV / (KWV * kTQ)) : 1;
#pragma unroll
              for (int i = 0; i < KF; ++i) {
                const int kk = (off + i) / kTQ, t = t0 + (off + i) % kTQ;
                const int row = r0 + kk * RPW + rw;
                if ((cl & (D - 1)) == 0 && row < p.P && t < p.T)
                  p.o[(((size_t)b * p.T + t) * p.H + hh) * p.P + row] = part[i];
              }
            }
          }
        } else {
          for (int pass = 0; pass < npass; ++pass) {
            const int rbase = (pass * wpg + wr) * kKR;
            for (int t0 = 0; t0 < p.T; t0 += kTQ) {
              float4 qv[kTQ];
              float g[kTQ];
#pragma unroll
              for (int t = 0; t < kTQ; ++t) {
                qv[t] = (t0 + t < p.T) ? In<TIn>::lds4(gQ, (t0 + t) * N + col4 * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
                g[t] = (t0 + t < p.T) ? sc[t0 + t] : 0.f;
              }
              float part[kKR * kTQ];
#pragma unroll
              for (int kk = 0; kk < kKR; ++kk) {
                const int row = (rbase + kk) * RPI + rsub;
                const float4 x4 =
                    (row < p.P) ? ld_tile4<kF16>(tile, (size_t)row * N + col4 * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int t = 0; t < kTQ; ++t) part[kk * kTQ + t] = g[t] * dot4(x4, qv[t]);
                if (row < p.P) {
                  for (int j = col4; j < J; j += LPR) {  // this lane's share of the records
                    const float vj = In<TIn>::lds(sv, j * p.P + row);
#pragma unroll
                    for (int t = 0; t < kTQ; ++t)
                      if (t0 + t < p.T) part[kk * kTQ + t] = fmaf(cw[(t0 + t) * kRMax + j], vj, part[kk * kTQ + t]);
                  }
                }
              }
              int off = 0;
              TRed<kKR * kTQ, LPR / 2>::run(part, lane, off);
              constexpr int KF = (kKR * kTQ / LPR) > 0 ? (kKR * kTQ / LPR) : 1;
              constexpr int D = (LPR / (kKR * kTQ)) > 0 ? (LPR / (kKR * kTQ)) : 1;
#pragma unroll
              for (int i = 0; i < KF; ++i) {
                const int kk = (off + i) / kTQ, t = t0 + (off + i) % kTQ;
                const int row = (rbase + kk) * RPI + rsub;
                if ((lane & (D - 1)) == 0 && row < p.P && t < p.T)
                  p.o[(((size_t)b * p.T + t) * p.H + hh) * p.P + row] = part[i];
              }
            }
          }
        }
      } else if constexpr (MODE == kSnap) {
        // ================================================ conventional verify with snapshots
        // x <- a_t x + v_t[row] k_t ; o_t = x q_t ; x -> state slot (st + 1 + t) mod nslot,
        // for t = 0 .. T-1: one read of the state, T writes.
        const float* sa = reinterpret_cast<const float*>(slot);  // new records' decays at kRMax + t
        for (int pass = 0; pass < npass; ++pass) {
          const int rbase = (pass * wpg + wr) * kKR;
          if (rbase * RPI >= p.P) break;  // warp-uniform: no rows left for this warp
          float4 x[kKR];
#pragma unroll
          for (int kk = 0; kk < kKR; ++kk) {
            const int row = (rbase + kk) * RPI + rsub;
            x[kk] = (row < p.P) ? lds4(tf + ((size_t)row * LPR + col4) * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          for (int t = 0; t < p.T; ++t) {
            const float at = sa[kRMax + t];
            const float4 kt = In<TIn>::lds4(gK, t * N + col4 * 4);
            const float4 qt = In<TIn>::lds4(gQ, t * N + col4 * 4);
            const int slot_t = (st + 1 + t) % p.nslot;
            float* dst = p.ckpt + ((size_t)slot_t * p.B * p.H + hrow) * p.P * N;
            float part[kKR];
#pragma unroll
            for (int kk = 0; kk < kKR; ++kk) {
              const int row = (rbase + kk) * RPI + rsub;
              const float vt = (row < p.P) ? In<TIn>::lds(sv, t * p.P + row) : 0.f;
              x[kk].x = fmaf(vt, kt.x, at * x[kk].x);
              x[kk].y = fmaf(vt, kt.y, at * x[kk].y);
              x[kk].z = fmaf(vt, kt.z, at * x[kk].z);
              x[kk].w = fmaf(vt, kt.w, at * x[kk].w);
              if (row < p.P) *reinterpret_cast<float4*>(dst + (size_t)row * N + col4 * 4) = x[kk];
              part[kk] = dot4(x[kk], qt);
            }
            int off = 0;
            TRed<kKR, LPR / 2>::run(part, lane, off);
            constexpr int KF = (kKR / LPR) > 0 ? (kKR / LPR) : 1;
            constexpr int D = (LPR / kKR) > 0 ? (LPR / kKR) : 1;
#pragma unroll
            for (int i = 0; i < KF; ++i) {
              const int row = (rbase + off + i) * RPI + rsub;
              if ((lane & (D - 1)) == 0 && row < p.P) p.o[(((size_t)b * p.T + t) * p.H + hh) * p.P + row] = part[i];
            }
          }
        }
      } else if (flush) {
        // ================================================ fold path
        // S_new = g_{1:J} S + sum_j u_j k_j^T with u_j = g_{j+2:J} v_j ; store ; o = S_new q
        // Delta rule: the same update with the scaled pseudo-values W_i w_i; the new
        // record's w_c (decode, conventional step) is formed first for this warp's rows.
        const float gam = sc[0];
        float* su = const_cast<float*>(sc) + (kDel ? kCoefOff + 2 * kRMax : kCoefOff);  // [J][P]
        for (int pass = 0; pass < npass; ++pass) {
          const int rbase = (pass * wpg + wr) * kKR;
          if (rbase * RPI >= p.P) break;  // warp-uniform: no rows left for this warp
          const float* ub = su + rbase * RPI;  // values of the warp's rows: ub[j * P + local row]
          if constexpr (kDel && MODE != kFlush) {
            // w_c = beta_c (v_c - alpha_c (P_c S k_c + sum_{i<c} D_ic k_i^T k_c w_i)) per row;
            // the row sums S k_c are reduced transposed (lane seg + kk D ends with row kk's)
            static_assert(LPR >= kKR, "delta-rule fold: a row spans at least kKR lanes");
            constexpr int D = LPR / kKR;
            const float4 kc4 = In<TIn>::lds4(gK, c * N + col4 * 4);
            float part[kKR];
#pragma unroll
            for (int kk = 0; kk < kKR; ++kk) {
              const int row = (rbase + kk) * RPI + rsub;
              part[kk] = (row < p.P) ? dot4(ld_tile4<false>(tile, (size_t)row * N + col4 * 4), kc4) : 0.f;
            }
            int off = 0;
            TRed<kKR, LPR / 2>::run(part, lane, off);
            const int row = (rbase + off) * RPI + rsub;
            // the D lanes holding a row split the buffered records (lane d: i = d, d + D, ...)
            const int d = lane & (D - 1);
            float y = (d == 0) ? sc[2] * part[0] : 0.f;
            if (row < p.P) {
              const float* sw = reinterpret_cast<const float*>(sv);
              const float* dk = sc + kCoefOff + kRMax;
              for (int i = d; i < c; i += D) y = fmaf(dk[i], sw[i * p.P + row], y);
            }
#pragma unroll
            for (int m = 1; m < D; m <<= 1) y += __shfl_xor_sync(kFull, y, m);
            if (d == 0 && row < p.P) {
              const float vn = In<TIn>::lds(slot + lay.nv_off, row);
              su[c * p.P + row] = sc[4] * fmaf(-sc[3], y, vn);  // W_c = 1
            }
            __syncwarp();
          }
          float4 acc[kKR];
          if constexpr (RPI == 1) {
            // The warp's 8 rows are consecutive and all valid (P is a multiple of 8).
            // Accumulate row pairs with packed fp32x2 fmas: A[kp][col] = {row 2kp, row 2kp+1}.
            f32x2 A[kKR / 2][4];
#pragma unroll
            for (int kp = 0; kp < kKR / 2; ++kp) {
              const float4 x0 = ld_tile4<kF16>(tile, (size_t)(rbase + 2 * kp) * N + col4 * 4);
              const float4 x1 = ld_tile4<kF16>(tile, (size_t)(rbase + 2 * kp + 1) * N + col4 * 4);
              A[kp][0] = pk2(gam * x0.x, gam * x1.x);
              A[kp][1] = pk2(gam * x0.y, gam * x1.y);
              A[kp][2] = pk2(gam * x0.z, gam * x1.z);
              A[kp][3] = pk2(gam * x0.w, gam * x1.w);
            }
#pragma unroll 4
            for (int j = 0; j < J; ++j) {
              const float4 kv = In<TIn>::lds4(gK, j * N + col4 * 4);
              const f32x2 kx = pk2(kv.x, kv.x), ky = pk2(kv.y, kv.y), kz = pk2(kv.z, kv.z), kw = pk2(kv.w, kv.w);
              f32x2 U[kKR / 2];
#pragma unroll
              for (int qd = 0; qd < kKR / 4; ++qd) {
                const ulonglong2 uq = *reinterpret_cast<const ulonglong2*>(ub + j * p.P + 4 * qd);
                U[2 * qd] = uq.x;
                U[2 * qd + 1] = uq.y;
              }
#pragma unroll
              for (int kp = 0; kp < kKR / 2; ++kp) {
                A[kp][0] = fma2(U[kp], kx, A[kp][0]);
                A[kp][1] = fma2(U[kp], ky, A[kp][1]);
                A[kp][2] = fma2(U[kp], kz, A[kp][2]);
                A[kp][3] = fma2(U[kp], kw, A[kp][3]);
              }
            }
#pragma unroll
            for (int kp = 0; kp < kKR / 2; ++kp) {
              acc[2 * kp] = make_float4(lo2(A[kp][0]), lo2(A[kp][1]), lo2(A[kp][2]), lo2(A[kp][3]));
              acc[2 * kp + 1] = make_float4(hi2(A[kp][0]), hi2(A[kp][1]), hi2(A[kp][2]), hi2(A[kp][3]));
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < kKR; ++kk) {
              const int row = (rbase + kk) * RPI + rsub;
              if (row < p.P) {
                const float4 x = ld_tile4<kF16>(tile, (size_t)row * N + col4 * 4);
                acc[kk] = make_float4(gam * x.x, gam * x.y, gam * x.z, gam * x.w);
              } else {
                acc[kk] = make_float4(0.f, 0.f, 0.f, 0.f);
              }
            }
            for (int j = 0; j < J; ++j) {
              const float4 kv = In<TIn>::lds4(gK, j * N + col4 * 4);
              float uu[kKR];
#pragma unroll
              for (int kk = 0; kk < kKR; ++kk) {
                const int row = (rbase + kk) * RPI + rsub;
                uu[kk] = (row < p.P) ? ub[j * p.P + kk * RPI + rsub] : 0.f;
              }
#pragma unroll
              for (int kk = 0; kk < kKR; ++kk) {
                acc[kk].x = fmaf(uu[kk], kv.x, acc[kk].x);
                acc[kk].y = fmaf(uu[kk], kv.y, acc[kk].y);
                acc[kk].z = fmaf(uu[kk], kv.z, acc[kk].z);
                acc[kk].w = fmaf(uu[kk], kv.w, acc[kk].w);
              }
            }
          }
          if constexpr (MODE != kQuant && kF16) {
            uint8_t* ck = reinterpret_cast<uint8_t*>(p.ckpt);
            if (p.sr) {
#pragma unroll
              for (int kk = 0; kk < kKR; ++kk) {
                const int row = (rbase + kk) * RPI + rsub;
                const size_t e = (hrow * p.P + row) * N + col4 * 4;  // first of the four elements
                const uint2 h = sr_f16x4(acc[kk], sr_words(e, (uint32_t)ep, p.seed));
                if (row < p.P) *reinterpret_cast<uint2*>(ck + e * 2) = h;
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < kKR; ++kk) {
                const int row = (rbase + kk) * RPI + rsub;
                if (row < p.P)
                  *reinterpret_cast<uint2*>(ck + ((hrow * p.P + row) * N + col4 * 4) * 2) =
                      make_uint2(rn_f16x2_sat(acc[kk].x, acc[kk].y), rn_f16x2_sat(acc[kk].z, acc[kk].w));
              }
            }
          } else if constexpr (MODE != kQuant) {
#pragma unroll
            for (int kk = 0; kk < kKR; ++kk) {
              const int row = (rbase + kk) * RPI + rsub;
              if (row < p.P) *reinterpret_cast<float4*>(p.ckpt + (hrow * p.P + row) * N + col4 * 4) = acc[kk];
            }
          }
          if constexpr (kCopyRF && MODE != kConv) {
            quantize_rows<RF, LPR, kKR>(acc, lane, rbase * RPI + rsub, RPI, p.P, N, p.copy + hrow * p.head_stride,
                                        p.bsc_off, p.rsc_off);
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
        }
      } else if constexpr (MODE == kDecode) {
        // ================================================ non-flush decode: o = g (S q) + value term
        // o[row] = g (S q)[row] + sum_j c_j v_j[row]: the lanes of a row split the
        // records (lane k of the row takes j = k, k + lanes, ...) and add their
        // share to the scaled dot before the row reduction.
        const float gam = sc[0];
        const float* scj = sc + kCoefOff;  // [kRMax] record weights, 0 past J
        if constexpr (kDel) {
          // Delta rule: per row, A = gamma (S q) + sum_{i<c} W_i s_i w_i and
          // B = P_c (S k_c) + sum_{i<c} D_ic M_ic w_i; then the new record's pseudo-value
          // w_c = beta_c (v_c - alpha_c B) goes to the ring and o = A + s_c w_c.
          // Rows as in the FP32 non-flush path; lane k of a row takes records k, k + LP16, ...
          constexpr int RPW = 32 / LP16, KW = 4;
          constexpr int JI = kRMax / LP16;
          const int cl = lane % LP16, rw = lane / LP16;
          float cwv[JI], dwv[JI];
#pragma unroll
          for (int i = 0; i < JI; ++i) {
            cwv[i] = scj[cl + LP16 * i];
            dwv[i] = sc[kCoefOff + kRMax + cl + LP16 * i];
          }
          const float pcv = sc[2], acv = sc[3], bcv = sc[4], sqc = sc[5];
          const float* sw = reinterpret_cast<const float*>(sv);
          const uint8_t* nv = slot + lay.nv_off;
          float* wring = reinterpret_cast<float*>(p.ring_v) + (hrow * p.R + ring_slot(st, c, p.R)) * p.P;
          for (int r0 = wr * KW * RPW; r0 < p.P; r0 += wpg * KW * RPW) {
            float part[2 * KW];
#pragma unroll
            for (int kk = 0; kk < KW; ++kk) {
              const int row = r0 + kk * RPW + rw;
              float ra = 0.f, rb = 0.f;
              if (row < p.P) {
                const float* rp = tf + (size_t)row * N;
                float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                  const float4 x = lds4(rp + (c4 * LP16 + cl) * 4);
                  a0 = fmaf(x.x, q16[4 * c4], a0); a1 = fmaf(x.y, q16[4 * c4 + 1], a1);
                  a0 = fmaf(x.z, q16[4 * c4 + 2], a0); a1 = fmaf(x.w, q16[4 * c4 + 3], a1);
                  b0 = fmaf(x.x, k16[4 * c4], b0); b1 = fmaf(x.y, k16[4 * c4 + 1], b1);
                  b0 = fmaf(x.z, k16[4 * c4 + 2], b0); b1 = fmaf(x.w, k16[4 * c4 + 3], b1);
                }
                ra = gam * (a0 + a1);
                rb = pcv * (b0 + b1);
#pragma unroll
                for (int i = 0; i < JI; ++i) {
                  const int j = cl + LP16 * i;
                  if (j < c) {
                    const float wv = sw[j * p.P + row];
                    ra = fmaf(cwv[i], wv, ra);
                    rb = fmaf(dwv[i], wv, rb);
                  }
                }
              }
              part[2 * kk] = ra;
              part[2 * kk + 1] = rb;
            }
            int off = 0;
            TRed<2 * KW, LP16 / 2>::run(part, lane, off);  // lane: value off (and off + 1 if LP16 < 2 KW)
            float va, vb;
            bool wo, ww;  // this lane writes the output / the pseudo-value
            if constexpr (LP16 < 2 * KW) {  // both values of row off / 2 in this lane
              va = part[0]; vb = part[1];
              wo = ww = true;
            } else {  // one value per lane: lanes off and off ^ 1 hold a row's pair
              const float other = __shfl_xor_sync(kFull, part[0], 1);
              const bool isa = (off & 1) == 0;
              va = isa ? part[0] : other;
              vb = isa ? other : part[0];
              wo = isa; ww = !isa;
            }
            const int row = r0 + (off >> 1) * RPW + rw;
            if (row < p.P) {
              const float w = bcv * fmaf(-acv, vb, In<TIn>::lds(nv, row));
              if (wo) p.o[hrow * p.P + row] = fmaf(sqc, w, va);
              if (ww) wring[row] = w;
            }
          }
        } else if constexpr (kWideRows) {
          constexpr int RPW = 32 / LP16, KW = 4;  // rows per warp instruction, row instructions per pass
          constexpr int JI = kRMax / LP16;
          const int cl = lane % LP16, rw = lane / LP16;
          float cwv[JI];
#pragma unroll
          for (int i = 0; i < JI; ++i) cwv[i] = scj[cl + LP16 * i];
          for (int r0 = wr * KW * RPW; r0 < p.P; r0 += wpg * KW * RPW) {
            float part[KW];
#pragma unroll
            for (int kk = 0; kk < KW; ++kk) {
              const int row = r0 + kk * RPW + rw;
              float a0 = 0.f, a1 = 0.f;
              if (row < p.P) {
                if constexpr (kF16) {  // two 16-byte chunks of 8 halves
#pragma unroll
                  for (int c = 0; c < 2; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4*>(tile + ((size_t)row * N + (c * LP16 + cl) * 8) * 2);
                    const uint32_t hw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[e]));
                      a0 = fmaf(f.x, q16[8 * c + 2 * e], a0);
                      a1 = fmaf(f.y, q16[8 * c + 2 * e + 1], a1);
                    }
                  }
                } else {
                  const float* rp = tf + (size_t)row * N;
#pragma unroll
                  for (int c = 0; c < 4; ++c) {
                    const float4 x = lds4(rp + (c * LP16 + cl) * 4);
                    a0 = fmaf(x.x, q16[4 * c], a0);
                    a1 = fmaf(x.y, q16[4 * c + 1], a1);
                    a0 = fmaf(x.z, q16[4 * c + 2], a0);
                    a1 = fmaf(x.w, q16[4 * c + 3], a1);
                  }
                }
                a0 = gam * (a0 + a1);
#pragma unroll
                for (int i = 0; i < JI; ++i) {
                  const int j = cl + LP16 * i;
                  if (j < J) a0 = fmaf(cwv[i], In<TIn>::lds(sv, j * p.P + row), a0);
                }
              }
              part[kk] = a0;
            }
            int off = 0;
            TRed<KW, LP16 / 2>::run(part, lane, off);  // lane: row r0 + off * RPW + rw
            constexpr int D = (LP16 / KW) > 0 ? (LP16 / KW) : 1;  // lanes holding the same row
            const int row = r0 + off * RPW + rw;
            if ((cl & (D - 1)) == 0 && row < p.P) p.o[hrow * p.P + row] = part[0];
          }
        } else
        for (int pass = 0; pass < npass; ++pass) {
          if constexpr (!kCopyRF) {
            const int rbase = (pass * wpg + wr) * kKR;
            float part[kKR];
#pragma unroll
            for (int kk = 0; kk < kKR; ++kk) {
              const int row = (rbase + kk) * RPI + rsub;
              float a = 0.f;
              if (row < p.P) {
                a = gam * dot4(ld_tile4<kF16>(tile, (size_t)row * N + col4 * 4), q4);
                for (int j = col4; j < J; j += LPR) a = fmaf(scj[j], In<TIn>::lds(sv, j * p.P + row), a);
              }
              part[kk] = a;
            }
            int off = 0;
            TRed<kKR, LPR / 2>::run(part, lane, off);
            constexpr int KF = (kKR / LPR) > 0 ? (kKR / LPR) : 1;
            constexpr int D = (LPR / kKR) > 0 ? (LPR / kKR) : 1;
#pragma unroll
            for (int i = 0; i < KF; ++i) {
              const int row = (rbase + off + i) * RPI + rsub;
              if ((lane & (D - 1)) == 0 && row < p.P) p.o[hrow * p.P + row] = part[i];
            }
          } else {
            // read copy: lanes own CPL consecutive codes of a row
            const int rows0 = (pass * wpg + wr) * kKR * RPI;  // first row of this warp
            const int colc = lane % LPRc, rsc = lane / LPRc;
            const float* rscale = reinterpret_cast<const float*>(tile + p.rsc_off);
            constexpr int JIc = kRMax / LPRc;  // this lane's records: j = colc + LPRc i
            float part[KRc];
#pragma unroll
            for (int kk = 0; kk < KRc; ++kk) {
              const int row = rows0 + kk * RPIc + rsc;
              float acc = 0.f;
              if (row < p.P) {
                float val = 0.f;  // this lane's share of sum_j c_j v_j[row], loads issued first
#pragma unroll
                for (int i = 0; i < JIc; ++i) {
                  const int j = colc + LPRc * i;
                  if (j < J) val = fmaf(scj[j], In<TIn>::lds(sv, j * p.P + row), val);
                }
                if constexpr (RF == kRfE4m3) {
                  const uint4 cwd = *reinterpret_cast<const uint4*>(tile + (size_t)row * N + colc * 16);
                  const uint32_t ws[4] = {cwd.x, cwd.y, cwd.z, cwd.w};
#pragma unroll
                  for (int qd = 0; qd < 4; ++qd) {
                    float f[4];
                    dec_e4m3x4(ws[qd], f);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc = fmaf(f[e], qc[qd * 4 + e], acc);
                  }
                } else {
                  const uint4 cwd = *reinterpret_cast<const uint4*>(tile + (size_t)row * (N / 2) + colc * 16);
                  const uint32_t ws[4] = {cwd.x, cwd.y, cwd.z, cwd.w};
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
                acc = fmaf(acc, gam * rscale[row], val);
              }
              part[kk] = acc;
            }
            int off = 0;
            TRed<KRc, LPRc / 2>::run(part, lane, off);
            constexpr int KF = (KRc / LPRc) > 0 ? (KRc / LPRc) : 1;
            constexpr int D = (LPRc / KRc) > 0 ? (LPRc / KRc) : 1;
#pragma unroll
            for (int i = 0; i < KF; ++i) {
              const int row = rows0 + (off + i) * RPIc + rsc;
              if ((lane & (D - 1)) == 0 && row < p.P) p.o[hrow * p.P + row] = part[i];
            }
          }
        }
      }

      // ---------------------------------------------------- release the stage and the slot
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(tempty0 + 8 * ts);
        mbar_arrive(sempty0 + 8 * rs);
      }
      tile_next();
      slot_next();
    }
  }

  // ------------------------------------------------------------------ epilogue
  // Pointer updates: once every CTA covering a sequence has finished reading its
  // pointers, the last one (ticket) advances them. Never a spin wait. Warp 0's
  // lanes take the CTA's sequences in parallel (their fences and tickets overlap).
  mbar_arrive(end_bar);
  if (warp == 0) {
    bool done = false;
    if (lane == 0) done = mbar_wait(end_bar, 0, abort_flag, p.err) && !*abort_flag;
    done = __shfl_sync(kFull, done, 0);
    if (done && (MODE == kDecode || MODE == kFlush) && h1 > h0) {
      const int b_first = (int)(h0 / p.H), b_last = (int)((h1 - 1) / p.H);
      for (int vb = b_first + lane; vb <= b_last; vb += 32) {
        const long long lo = max(h0, (long long)vb * p.H), hi = min(h1, (long long)(vb + 1) * p.H);
        const int n_b = (int)(hi - lo);
        const int b = seq_of(vb);
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
          if constexpr (kF16) {
            if (MODE == kFlush || flush) p.epoch[b] += 1;
          }
          p.ticket[b] = 0;
        }
      }
    }
  }
}

}  // namespace rssm
