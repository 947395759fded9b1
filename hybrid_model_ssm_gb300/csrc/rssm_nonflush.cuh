// rssm_nonflush.cuh - the non-flush decode step for small head tiles (an E4M3 or
// E2M1 read copy, or an FP16 checkpoint): one warp per head, each warp with its
// own double-buffered stages and nothing shared between the warps.
//
// The output-only step (aikraft.ru, "ReplaySSM: Революция в декодировании
// гибридных моделей", §03 unrolled window, §05 output-only evaluation, §06 split
// precision) is
//   o = g_{1:J} (S q) + sum_j g_{j+2:J} (k_j^T q) v_j        (records j = 0 .. J-1)
// with S read from the head's small tile (the read copy, or the FP16 checkpoint).
// The pipelined head kernel pays a fixed cost per head (mbarrier round trips
// between its roles, one gather lane) that a 4.9-16 KiB tile cannot hide. Here
// each warp walks a contiguous run of heads on its own. One lane copies the next
// head's tile and decays into the warp's other tile stage with bulk copies (an
// mbarrier per stage counts their bytes) while the warp computes the current
// head; the value rows, needed only at the end of a head, have one stage that
// is refilled for the next head as soon as the current head's value term is
// done. Every head costs one overlapped round trip however many records it holds. The keys' dots with the query are computed
// once per group, from registers. Every wait is bounded, as in the head kernel.
//
// Sequences that flush in this step, and sequences whose ring would overflow,
// are skipped. The head kernel, launched right after with skip_nonflush set,
// folds the flushing sequences, flags the overflowing ones and advances every
// sequence's pointers, so both launches read the same counts.
#pragma once

#include "rssm_device.cuh"

namespace rssm {

constexpr int kNfBatch = 8;  // tile chunks per lane between row reductions

// Per-warp shared memory of the warp-per-head step: three mbarriers (two tile
// stages, one value stage), the tile dots (P floats), two tile stages of
// [tile | the ring's decays (Rp)], and one value stage of the head's value rows
// in record order (at most L - 1: a sequence with L - 1 buffered records folds).
struct NfStage {
  int tile_bytes, a_off, tbytes, vbytes, rsum_bytes;
};
__host__ __device__ inline NfStage nf_stage(int tile_bytes, int L, int Rp, int P, int in_bytes) {
  NfStage g;
  g.tile_bytes = tile_bytes;
  g.a_off = (tile_bytes + 15) / 16 * 16;
  g.tbytes = (g.a_off + Rp * 4 + 127) / 128 * 128;
  const int vrows = L > 1 ? L - 1 : 1;
  g.vbytes = (vrows * P * in_bytes + 127) / 128 * 128;
  g.rsum_bytes = (P * 4 + 127) / 128 * 128;
  return g;
}
// Order this thread's earlier generic-proxy accesses to shared memory before its
// later bulk copies into it.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
constexpr int kNfCtaBytes = 128;  // the CTA's abort flag, padded
constexpr int kNfBarBytes = 32;   // a warp's three stage barriers, padded (stages stay 16-byte aligned)
__host__ __device__ inline int nf_warp_bytes(const NfStage& g) {
  return kNfBarBytes + g.rsum_bytes + 2 * g.tbytes + g.vbytes;
}

// A head tile as rows of 16-byte chunks: CW columns per chunk, CPR chunks per row.
template <int N, int RF>
struct NfTile {
  static constexpr int CW = RF == kRfE4m3 ? 16 : RF == kRfE2m1 ? 32 : 8;
  static constexpr int CPR = N / CW;
  static_assert(CPR >= 2 && CPR <= 32 && (32 % CPR) == 0, "tile chunks per row");
};

// n consecutive input elements (n * bytes = 4, 8 or 16) as raw words and as floats.
template <typename TIn, int n>
struct Raw {
  static constexpr int kWords = n * In<TIn>::kBytes / 4;
  uint32_t w[kWords];
  __device__ __forceinline__ void load(const uint8_t* base, int i) {
    const uint8_t* a = base + (size_t)i * In<TIn>::kBytes;
    if constexpr (kWords == 4) {
      const uint4 u = *reinterpret_cast<const uint4*>(a);
      w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else if constexpr (kWords == 2) {
      const uint2 u = *reinterpret_cast<const uint2*>(a);
      w[0] = u.x; w[1] = u.y;
    } else {
      w[0] = *reinterpret_cast<const uint32_t*>(a);
    }
  }
  __device__ __forceinline__ void store(uint8_t* base, int i) const {
    uint8_t* a = base + (size_t)i * In<TIn>::kBytes;
    if constexpr (kWords == 4) {
      *reinterpret_cast<uint4*>(a) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (kWords == 2) {
      *reinterpret_cast<uint2*>(a) = make_uint2(w[0], w[1]);
    } else {
      *reinterpret_cast<uint32_t*>(a) = w[0];
    }
  }
  __device__ __forceinline__ float get(int e) const {
    if constexpr (In<TIn>::kBytes == 4) {
      return __uint_as_float(w[e]);
    } else {
      const uint32_t x = w[e >> 1];
      return __uint_as_float((e & 1) ? (x & 0xFFFF0000u) : (x << 16));  // bf16 -> fp32 is exact
    }
  }
};

// The two E4M3 block scales of a 32-column chunk (bytes 0 and 1 of bs) as floats,
// with one conversion (E4M3 values are exact in binary16 and in binary32).
__device__ __forceinline__ float2 dec_e4m3x2(uint32_t bs) {
  uint32_t h;
  asm("{ .reg .b16 lo; cvt.u16.u32 lo, %1; cvt.rn.f16x2.e4m3x2 %0, lo; }" : "=r"(h) : "r"(bs));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// c + a.lo b.lo + a.hi b.hi for binary16 pairs a and b, accumulated in FP32: each
// fma.rn.f32.f16 multiplies two exact binary16 values (an exact product in FP32)
// and rounds once, the same as an FP32 fma of the two values.
__device__ __forceinline__ float fma_h2(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;"
      " fma.rn.f32.f16 %0, al, bl, %3; fma.rn.f32.f16 %0, ah, bh, %0; }"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

// The chunk's dot with the query at its columns, the query given as binary16
// pairs qh (the group's query times an exact power of two): E4M3 and E2M1 codes
// convert to binary16 exactly, and FP16 tiles are binary16 already.
template <int RF>
__device__ __forceinline__ float chunk_dot_h(const uint4 u, const uint32_t* qh, uint32_t bs) {
  const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
  if constexpr (RF == kRfE4m3) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      uint32_t h01, h23;
      asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.rn.f16x2.e4m3x2 %0, lo; cvt.rn.f16x2.e4m3x2 %1, hi; }"
          : "=r"(h01), "=r"(h23)
          : "r"(ws[qd]));
      a0 = fma_h2(h01, qh[2 * qd], a0);
      a1 = fma_h2(h23, qh[2 * qd + 1], a1);
    }
    return a0 + a1;
  } else if constexpr (RF == kRfE2m1) {
    float blk[2] = {0.f, 0.f};
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      uint32_t h[4];
      asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
          " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
          " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
          : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
          : "r"(ws[qd]));
#pragma unroll
      for (int e = 0; e < 4; ++e) blk[qd >> 1] = fma_h2(h[e], qh[qd * 4 + e], blk[qd >> 1]);
    }
    const float2 sc = dec_e4m3x2(bs);
    return fmaf(sc.x, blk[0], sc.y * blk[1]);
  } else {  // FP16 checkpoint: eight halves
    float a0 = fma_h2(ws[0], qh[0], 0.f);
    float a1 = fma_h2(ws[1], qh[1], 0.f);
    a0 = fma_h2(ws[2], qh[2], a0);
    a1 = fma_h2(ws[3], qh[3], a1);
    return a0 + a1;
  }
}

// The chunk's dot with the query at its columns (E2M1: with its two block scales
// in bs, one E4M3 code per 16 columns; the row scale is applied later).
template <int RF>
__device__ __forceinline__ float chunk_dot(const uint4 u, const float* qt, uint32_t bs) {
  const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
  if constexpr (RF == kRfE4m3) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      float f[4];
      dec_e4m3x4(ws[qd], f);
      a0 = fmaf(f[0], qt[4 * qd], a0);
      a1 = fmaf(f[1], qt[4 * qd + 1], a1);
      a0 = fmaf(f[2], qt[4 * qd + 2], a0);
      a1 = fmaf(f[3], qt[4 * qd + 3], a1);
    }
    return a0 + a1;
  } else if constexpr (RF == kRfE2m1) {
    float blk[2] = {0.f, 0.f};
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      float f[8];
      dec_e2m1x8(ws[qd], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) blk[qd >> 1] = fmaf(f[e], qt[qd * 8 + e], blk[qd >> 1]);
    }
    const float2 sc = dec_e4m3x2(bs);
    return fmaf(sc.x, blk[0], sc.y * blk[1]);
  } else {  // FP16 checkpoint: eight halves
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ws[e]));
      a0 = fmaf(f.x, qt[2 * e], a0);
      a1 = fmaf(f.y, qt[2 * e + 1], a1);
    }
    return a0 + a1;
  }
}

// A head the warp computes: its sequence, head and group, and the sequence's pointers.
struct NfHead {
  int b, hh, g, gpos, c, st;
};

template <int N, typename TIn, int RF>
__global__ void __launch_bounds__(kNfMaxThreads, 1) nonflush_kernel(const Params p, const NfStage sg) {
  using Tile = NfTile<N, RF>;
  constexpr int CW = Tile::CW, CPR = Tile::CPR, RPI = 32 / CPR;
  constexpr int ES = In<TIn>::kBytes;
  constexpr int NPL = N / 32;  // key and query columns per lane in the key dots
  static_assert(NPL == 2 || NPL == 4, "N in {64, 128}");
  constexpr int KB = kNfBatch;
  constexpr int D = (CPR > KB) ? CPR / KB : 1;  // lanes left holding the same row sum
  // bf16 inputs: the tile dot takes binary16 operands (the query scaled by 2^s per
  // group, exact) with FP32 accumulation; f32 inputs keep FP32 operands
  constexpr bool kHalf = (ES == 2);
  extern __shared__ __align__(128) uint8_t nf_smem[];

  // Programmatic dependent launch: the head kernel that follows may be scheduled
  // as this grid drains; it waits for this grid's completion before its first
  // global access. Nothing here touches global memory before the previous grid
  // (the last step's kernels) has completed.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const long long nw = (long long)gridDim.x * nwarps;
  const long long gw = (long long)blockIdx.x * nwarps + warp;
  const long long total = (long long)p.B * p.H;
  const long long h0 = gw * total / nw, h1 = (gw + 1) * total / nw;
  // dynamic shared memory: the CTA's abort flag (set when a wait of any warp runs
  // out), then each warp's area
  volatile int* abort_flag = reinterpret_cast<volatile int*>(nf_smem);
  if (threadIdx.x == 0) *abort_flag = 0;
  uint8_t* wbase = nf_smem + kNfCtaBytes + (size_t)warp * nf_warp_bytes(sg);
  const uint32_t bar0 = smem_u32(wbase);  // tile stage b's barrier at bar0 + 8 b, the value stage's at bar0 + 16
  const uint32_t vbar = bar0 + 16;
  float* rsum = reinterpret_cast<float*>(wbase + kNfBarBytes);
  uint8_t* const tstage = wbase + kNfBarBytes + sg.rsum_bytes;  // tile stage b at tstage + b tbytes
  const uint8_t* const sv = tstage + 2 * sg.tbytes;             // the value stage
  if (lane == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    mbar_init(vbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int vrow = p.P * ES;  // bytes of a value row

  // The next head to compute, skipping sequences that flush in this step or
  // would overflow their ring (the head kernel takes those).
  HeadIter it;
  it.init(h0, p.H, p.HPG);
  long long gh = h0;
  int sb = -1, sc = 0, sst = 0;
  bool sskip = true;
  auto find = [&](NfHead& r) -> bool {
    for (; gh < h1; ++gh, it.next(p.H, p.HPG)) {
      if (it.b != sb) {
        sb = it.b;
        sc = p.count[sb];
        sst = p.start[sb];
        sskip = sc < 0 || sc + 1 > p.R || sc + 1 >= p.L;
      }
      if (!sskip) {
        r.b = it.b; r.hh = it.hh; r.g = it.g; r.gpos = it.gpos; r.c = sc; r.st = sst;
        ++gh;
        it.next(p.H, p.HPG);
        return true;
      }
    }
    return false;
  };
  // Bulk-copy a head's tile and the ring's decays into tile stage `buf`; every lane
  // returns the step's own decay (read now, used one head later).
  auto issue_tile = [&](const NfHead& r, int buf) -> float {
    const size_t hrow = (size_t)r.b * p.H + r.hh;
    if (lane == 0) {
      const uint32_t dst = smem_u32(tstage + (size_t)buf * sg.tbytes), bar = bar0 + 8u * buf;
      const uint8_t* tile = (RF == kCkF16) ? reinterpret_cast<const uint8_t*>(p.ckpt) + hrow * (size_t)p.P * N * 2
                                           : p.copy + hrow * (size_t)p.head_stride;
      fence_proxy_async_shared();  // the warp's earlier reads of this stage come first
      mbar_arrive_tx(bar, (uint32_t)(sg.tile_bytes + p.Rp * 4));
      tma_load_1d(dst, tile, (uint32_t)sg.tile_bytes, bar);
      tma_load_1d(dst + sg.a_off, p.ring_a + hrow * p.Rp, (uint32_t)(p.Rp * 4), bar);
    }
    return p.alpha[hrow];
  };
  // Bulk-copy a head's value rows into the value stage, in record order: the
  // committed ones are at most two contiguous ring runs, then the step's own.
  auto issue_values = [&](const NfHead& r) {
    if (lane == 0) {
      const size_t hrow = (size_t)r.b * p.H + r.hh;
      const uint32_t dst = smem_u32(sv);
      const uint8_t* rv = reinterpret_cast<const uint8_t*>(p.ring_v) + hrow * p.R * (size_t)vrow;
      fence_proxy_async_shared();
      mbar_arrive_tx(vbar, (uint32_t)((r.c + 1) * vrow));
      if (r.c > 0) {
        const int n1 = min(r.c, p.R - r.st);
        tma_load_1d(dst, rv + (size_t)r.st * vrow, (uint32_t)(n1 * vrow), vbar);
        if (r.c > n1) tma_load_1d(dst + n1 * vrow, rv, (uint32_t)((r.c - n1) * vrow), vbar);
      }
      tma_load_1d(dst + r.c * vrow, reinterpret_cast<const uint8_t*>(p.v) + hrow * (size_t)vrow, (uint32_t)vrow,
                  vbar);
    }
  };
  // Wait (bounded) for a barrier's next phase. On failure, lane 0 waits (bounded)
  // for every copy still in flight into this warp's stages (bits of `pend`: tile
  // stages 0 and 1, the value stage) and keeps the pointers of the sequences of
  // the heads not done, and the warp leaves.
  uint32_t phase = 0;  // bit i: the parity barrier i (tile 0, tile 1, values) completes next
  uint32_t pend = 0;   // bit i: a copy issued on barrier i not yet waited for
  auto wait_or_leave = [&](int i, int b_first) -> bool {
    const uint32_t bar = bar0 + 8u * i;
    if (__all_sync(kFull, mbar_wait(bar, (phase >> i) & 1u, abort_flag, p.err))) {
      phase ^= 1u << i;
      pend &= ~(1u << i);
      return true;
    }
    if (lane == 0) {
      volatile int dummy = 0;
      for (int j = 0; j < 3; ++j)
        if ((pend >> j) & 1u) mbar_wait(bar0 + 8u * j, (phase >> j) & 1u, &dummy, p.err);
      // The heads from here on get no output or append. Their sequences keep their
      // pointers, as after an aborted head-kernel CTA: the head kernel advances a
      // sequence only when its ticket reaches H, and rssm_clear_error resets tickets.
      const int b_last = (int)((h1 - 1) / p.H);
      for (int b = b_first; b <= b_last; ++b) atomicAdd(p.ticket + b, -(1 << 20));
    }
    __syncwarp();
    return false;
  };

  long long cur_g = -1;
  float sj = 0.f;  // lane j < J: k_j^T q of the current group
  float qt[kHalf ? 1 : CW];         // the query at this lane's tile columns (f32 inputs)
  uint32_t qh[kHalf ? CW / 2 : 1];  // the same, times 2^s, as binary16 pairs (bf16 inputs)
  float qs_lo = 1.f, qs_hi = 1.f;   // 2^-s in two exact factors (bf16 inputs)
  NfHead cur, nxt;
  bool have = find(cur);
  float acur = 1.f;  // the current head's own decay
  if (have) {
    acur = issue_tile(cur, 0);
    issue_values(cur);
    pend = 1u | 4u;
  }
  int buf = 0;
  while (have) {
    const bool more = find(nxt);
    float anxt = 1.f;
    if (more) {
      anxt = issue_tile(nxt, buf ^ 1);
      pend |= 1u << (buf ^ 1);
    }
    const int c = cur.c, st = cur.st, J = c + 1;
    const size_t grow = (size_t)cur.b * p.G + cur.g;
    const size_t hrow = (size_t)cur.b * p.H + cur.hh;
    const int snew = ring_slot(st, c, p.R);  // the ring slot of the step's own record

    if ((long long)grow != cur_g) {
      // ------------------------------------------------ per group: the query and k_j^T q
      cur_g = (long long)grow;
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(p.q) + grow * N * ES;
      Raw<TIn, NPL> qk;
      qk.load(qrow, lane * NPL);
      if constexpr (kHalf) {
        // 2^s puts max|q| in [2^14, 2^15): every bf16 element within 2^-17 of the
        // maximum is exact in binary16 after scaling. s is split into two factors
        // so that each power of two is a normal float.
        float qm = 0.f;
#pragma unroll
        for (int e = 0; e < NPL; ++e) qm = fmaxf(qm, fabsf(qk.get(e)));
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) qm = fmaxf(qm, __shfl_xor_sync(kFull, qm, m));
        const int ex = (int)((__float_as_uint(qm) >> 23) & 0xFFu) - 127;  // floor(log2 max), -127 for 0 or tiny
        const int sh = 14 - ex;            // -113 .. 141
        const int s1 = sh / 2, s2 = sh - s1;  // each in -57 .. 71: normal powers of two
        const float m1 = __uint_as_float((uint32_t)(127 + s1) << 23), m2 = __uint_as_float((uint32_t)(127 + s2) << 23);
        qs_lo = __uint_as_float((uint32_t)(127 - s1) << 23);
        qs_hi = __uint_as_float((uint32_t)(127 - s2) << 23);
#pragma unroll
        for (int i = 0; i < CW; i += 4) {
          Raw<TIn, 4> q4;
          q4.load(qrow, (lane % CPR) * CW + i);
          qh[i / 2] = rn_f16x2_sat(q4.get(0) * m1 * m2, q4.get(1) * m1 * m2);
          qh[i / 2 + 1] = rn_f16x2_sat(q4.get(2) * m1 * m2, q4.get(3) * m1 * m2);
        }
      } else {
#pragma unroll
        for (int i = 0; i < CW; i += 4) {
          Raw<TIn, 4> q4;
          q4.load(qrow, (lane % CPR) * CW + i);
#pragma unroll
          for (int e = 0; e < 4; ++e) qt[i + e] = q4.get(e);
        }
      }
      Raw<TIn, NPL> kn;  // the step's own key
      kn.load(reinterpret_cast<const uint8_t*>(p.k) + grow * N * ES, lane * NPL);
      const uint8_t* rk = reinterpret_cast<const uint8_t*>(p.ring_k) + grow * p.R * N * ES;
      sj = 0.f;
      for (int j0 = 0; j0 < J; j0 += 8) {  // eight key rows in flight
        float d[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = j0 + u;
          Raw<TIn, NPL> kj = kn;
          if (j < c) kj.load(rk + (size_t)ring_slot(st, j, p.R) * N * ES, lane * NPL);
          d[u] = 0.f;
#pragma unroll
          for (int e = 0; e < NPL; ++e) d[u] = fmaf(kj.get(e), qk.get(e), d[u]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float t = warp_allsum(d[u]);
          if (lane == j0 + u) sj = t;
        }
      }
      // the group's first head appends the new key
      if (cur.gpos == 0) kn.store(reinterpret_cast<uint8_t*>(p.ring_k) + (grow * p.R + snew) * N * ES, lane * NPL);
    }

    // this head's tile and decays have landed (the next head's may still be in flight)
    if (!wait_or_leave(buf, cur.b)) return;
    const uint8_t* stg = tstage + (size_t)buf * sg.tbytes;
    const float* sa = reinterpret_cast<const float*>(stg + sg.a_off);

    // -------------------------------------------------- decays and record weights
    // lane j: alpha_j (committed records in ring order, then the step's own), 1 past J
    float aj = 1.f;
    if (lane < c) aj = sa[ring_slot(st, lane, p.R)];
    else if (lane == c) aj = acur;
    const float incl = suffix_prod(aj, lane);           // g_{lane+1:J}
    const float nxa = __shfl_down_sync(kFull, incl, 1);
    const float cj = (lane < J) ? ((lane < 31) ? nxa : 1.f) * sj : 0.f;  // g_{j+2:J} k_j^T q
    const float gam = __shfl_sync(kFull, incl, 0);      // g_{1:J}
    if (lane == c) p.ring_a[hrow * p.Rp + snew] = aj;

    // -------------------------------------------------- the tile: rows . q
    const int nch = p.P * CPR;  // 16-byte chunks; chunk ch is row ch / CPR, columns (ch % CPR) CW ..
    for (int c0 = 0; c0 < nch; c0 += 32 * KB) {
      float part[KB];
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        const int ch = c0 + i * 32 + lane;
        part[i] = 0.f;
        if (ch < nch) {
          const uint4 u = *reinterpret_cast<const uint4*>(stg + (size_t)ch * 16);
          uint32_t bs = 0u;
          if constexpr (RF == kRfE2m1)
            bs = *reinterpret_cast<const uint16_t*>(stg + p.bsc_off + (ch / CPR) * (N / 16) + (ch % CPR) * 2);
          if constexpr (kHalf) part[i] = chunk_dot_h<RF>(u, qh, bs);
          else part[i] = chunk_dot<RF>(u, qt, bs);
        }
      }
      int off = 0;
      TRed<KB, CPR / 2>::run(part, lane, off);  // over the CPR lanes of a row
      constexpr int KF = (KB / CPR) > 0 ? KB / CPR : 1;
#pragma unroll
      for (int i = 0; i < KF; ++i) {
        const int row = (c0 / CPR) + (off + i) * RPI + lane / CPR;
        if ((lane & (D - 1)) == 0 && row < p.P) rsum[row] = part[i];
      }
    }
    __syncwarp();

    // -------------------------------------------------- o = g (S q) + sum_j c_j v_j, row pairs
    if (!wait_or_leave(2, cur.b)) return;  // this head's value rows
    const float* rscale = reinterpret_cast<const float*>(stg + p.rsc_off);
    for (int r0 = 0; r0 < p.P; r0 += 64) {
      const int r = r0 + 2 * lane;
      const bool live = r < p.P;  // P is a multiple of 8: rows r and r + 1 together
      float v0 = 0.f, v1 = 0.f;
#pragma unroll 4
      for (int j = 0; j < J; ++j) {
        const float w = __shfl_sync(kFull, cj, j);
        if (live) {
          Raw<TIn, 2> vv;
          vv.load(sv + (size_t)j * vrow, r);
          v0 = fmaf(w, vv.get(0), v0);
          v1 = fmaf(w, vv.get(1), v1);
        }
      }
      if (live) {
        float t0 = rsum[r], t1 = rsum[r + 1];
        if constexpr (kHalf) {  // undo the query's scale (exact unless the sum underflows)
          t0 = (t0 * qs_lo) * qs_hi;
          t1 = (t1 * qs_lo) * qs_hi;
        }
        if constexpr (RF != kCkF16) {
          t0 *= rscale[r];
          t1 *= rscale[r + 1];
        }
        *reinterpret_cast<float2*>(p.o + hrow * p.P + r) = make_float2(fmaf(gam, t0, v0), fmaf(gam, t1, v1));
        Raw<TIn, 2> vc;  // the step's own value pair goes to the ring
        vc.load(sv + (size_t)c * vrow, r);
        vc.store(reinterpret_cast<uint8_t*>(p.ring_v) + (hrow * p.R + snew) * (size_t)vrow, r);
      }
    }
    __syncwarp();  // the stages and the row sums are rewritten by later heads
    if (more) {  // the value stage is free: the next head's rows
      issue_values(nxt);
      pend |= 4u;
    }
    cur = nxt;
    acur = anxt;
    have = more;
    buf ^= 1;
  }
}

}  // namespace rssm
