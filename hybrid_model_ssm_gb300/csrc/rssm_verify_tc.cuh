// rssm_verify_tc.cuh - speculative verify on the 5th-generation tensor cores.
//
// Verify evaluates, for T draft queries at once (ai.cheesepanini.fun,
// "知识卡片：ReplaySSM——重新思考混合模型解码的状态存储", 方法/产品要点, verify form;
// aikraft.ru, "ReplaySSM: Революция в декодировании гибридных моделей", §05):
//     O = S_ckpt Q D + V (W ⊙ (K^T Q))
// The checkpoint product S_ckpt Q is a dense contraction (P x N times N x T per
// head), and for large T it is more than the CUDA cores keep up with at the
// speed the checkpoint streams in. Here it runs as kind::tf32 MMAs with the
// accumulator in tensor memory. TF32 alone keeps 10 mantissa bits, too few for
// a 1e-4 tolerance, so the checkpoint is split S = hi + lo, hi = S with its low
// 13 mantissa bits cleared (exact in TF32), lo = S - hi (exact in fp32, and its
// own TF32 rounding costs only 2^-21 of S). bf16 queries are exact in TF32.
// The product is hi Q + lo Q: hi is the tile as it sits in shared memory (a
// kind::tf32 operand's low 13 mantissa bits are ignored), lo from tensor memory.
//
// An item is 128 checkpoint rows: 128/P consecutive heads of one group, which
// share their queries, so one M = 128 MMA serves them. Warp roles:
//   TMA lane      tensor copies of each item's tile, one 16 KiB K-block (32
//                 columns of 128 rows, 128-byte swizzled) per stage
//   gather lane   per group: committed and draft keys, draft queries; per item:
//                 the committed decays and value rows and the draft value rows
//   MMA warp      allocates tensor memory; one lane issues the MMAs of each
//                 K-block (4 from hi in shared memory, 4 from lo in tensor
//                 memory) into the item's accumulator
//   coefficients  per group: K^T Q and the queries as the B operand (fp32,
//                 swizzled); per item: the decay products g_t and the record
//                 weights, the appends of draft decays and keys
//   row warps     two sets of eight, taking alternate items (each set owns one
//                 tensor-memory buffer, and its items' tile stages and record
//                 slots), so that two items' chains overlap. Thread = checkpoint
//                 row: form each K-block's lo = S - hi (into tensor memory; the
//                 MMAs read hi from the tile as stored); after the MMAs, the epilogue
//                 o[t] = g_t (S q_t) + sum_j w_tj v_j[row], the output store and
//                 the appends of the draft value rows
// Every wait is bounded (the same waits as the head kernel); a CTA that gives
// up drains its copies and MMAs and frees its tensor memory before it returns.
#pragma once

#include <cuda.h>

#include "rssm_device.cuh"
#include "rssm_tc.cuh"

namespace rssm {

constexpr int kTcT = 16;                 // queries per MMA (N dimension): drafts, zero padded
constexpr int kTcRows = 128;             // checkpoint rows per item (MMA M)
constexpr int kTcKB = 32;                // fp32 columns per K-block (128 bytes)
constexpr int kTcStageBytes = kTcRows * kTcKB * 4;  // 16 KiB
constexpr int kTcMaxStages = 12;
constexpr int kTcMaxSlots = 8;
constexpr int kTcSets = 2;               // row-warp sets, taking alternate items
constexpr int kTcSetWarps = 8;           // row warps of a set: two per tensor-memory lane quarter
constexpr int kTcRowWarps = kTcSets * kTcSetWarps;
constexpr int kTcTmaWarp = kTcRowWarps, kTcGatherWarp = kTcRowWarps + 1, kTcMmaWarp = kTcRowWarps + 2;
constexpr int kTcCoef0 = kTcRowWarps + 3;
constexpr int kTcCoefWarps = 2;
constexpr int kTcThreads = (kTcCoef0 + kTcCoefWarps) * 32;
constexpr uint32_t kTcCols = 512;        // tensor memory: two buffers of 256 columns
constexpr int kTcCoefFloats = kTcT + kTcT * kRMax;  // per head: g_t, then weights [T][kRMax]

struct TcParams {
  int B, H, G, L, R, Rp, HPG, T;
  const float* alpha;          // [B,T,H]
  const __nv_bfloat16* v;      // [B,T,H,P]
  const __nv_bfloat16* k;      // [B,T,G,N]
  const __nv_bfloat16* q;      // [B,T,G,N]
  float* o;                    // [B,T,H,P]
  float* ring_a;               // [B,H,Rp]
  __nv_bfloat16* ring_v;       // [B,H,R,P]
  __nv_bfloat16* ring_k;       // [B,G,R,N]
  const int32_t* start;
  const int32_t* count;
  uint32_t* err;
  // shared memory (bytes from the 1024-aligned base): stages at 0, then
  int stages, slots;
  int qop_off, qop_bytes;      // two B operands [kTcT x N] fp32, swizzled
  int slot_off, slot_bytes;    // slots: committed decays | committed v | draft v | coefficients
  int sv_off, sd_off, sc_off;  //   (offsets inside a slot)
  int gb_off, gb_bytes, gq_off;  // two group areas: keys [R x N] | queries [kTcT x N] (bf16)
  int wsc_off, bar_off;
};

template <int N, int P>
__global__ void __launch_bounds__(kTcThreads, 1)
    verify_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tmap) {
  constexpr int IH = kTcRows / P;   // heads per item
  constexpr int NKB = N / kTcKB;    // K-blocks per item
  static_assert(IH >= 1 && IH * P == kTcRows && NKB >= 1, "an item is 128 rows of whole heads");
  constexpr uint32_t kIdesc = tc::idesc_tf32(kTcRows, kTcT);
  constexpr int ES = 2;  // bf16 inputs

  extern __shared__ __align__(128) uint8_t tc_smem[];  // 1024-byte alignment is checked below
  uint8_t* const smem = tc_smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  // tfull, tempty, sdone [kTcMaxStages]; sfull, scoef, sempty [kTcMaxSlots]; dfull[2],
  // gfull[2], gempty[2], qfull[2], qempty[2], kqdone[2], drain; then the abort flag
  // and the tensor-memory base address
  const uint32_t tfull0 = smem_u32(bars), tempty0 = tfull0 + 8 * kTcMaxStages, sdone0 = tempty0 + 8 * kTcMaxStages;
  const uint32_t sfull0 = sdone0 + 8 * kTcMaxStages, scoef0 = sfull0 + 8 * kTcMaxSlots;
  const uint32_t sempty0 = scoef0 + 8 * kTcMaxSlots, dfull0 = sempty0 + 8 * kTcMaxSlots;
  const uint32_t gfull0 = dfull0 + 16, gempty0 = gfull0 + 16, qfull0 = gempty0 + 16, qempty0 = qfull0 + 16;
  const uint32_t kqdone0 = qempty0 + 16, drain_bar = kqdone0 + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * kTcMaxStages + 3 * kTcMaxSlots + 13);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kTcMaxStages + 3 * kTcMaxSlots + 14);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int HI = p.H / IH;  // items per sequence
  const long long total = (long long)p.B * HI;
  const long long i0 = (long long)blockIdx.x * total / gridDim.x;
  const long long i1 = (long long)(blockIdx.x + 1) * total / gridDim.x;

  // The swizzled operands need a 1024-byte aligned base. Every tile stage and
  // record slot must belong to one row-warp set for good (its items come every
  // other item), so that a set never waits on an entry the other set still holds:
  // stages a multiple of kTcSets K-blocks per item, slots a multiple of kTcSets.
  // Refuse any other plan.
  if ((smem_u32(smem) & 1023u) != 0 || p.stages < kTcSets * NKB || (p.stages % (kTcSets * NKB)) != 0 ||
      p.stages > kTcMaxStages || p.slots < 2 || p.slots > kTcMaxSlots || (p.slots % kTcCoefWarps) != 0 ||
      (p.slots % kTcSets) != 0 || p.T < 1 || p.T > kTcT) {
    if (threadIdx.x == 0) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      atomicOr(p.err, kErrPlan);
    }
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(tfull0 + 8 * s, 1);
      mbar_init(tempty0 + 8 * s, 1);             // the MMA commit
      mbar_init(sdone0 + 8 * s, 4);              // the four row warps (one per lane quarter) of its K-block
    }
    for (int s = 0; s < p.slots; ++s) {
      mbar_init(sfull0 + 8 * s, 1);
      mbar_init(scoef0 + 8 * s, 1);
      mbar_init(sempty0 + 8 * s, kTcSetWarps);  // the row warps of the item's set
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(dfull0 + 8 * s, 1);
      mbar_init(gfull0 + 8 * s, 1);
      mbar_init(gempty0 + 8 * s, kTcCoefWarps);
      mbar_init(qfull0 + 8 * s, 1);
      mbar_init(qempty0 + 8 * s, 1);
      mbar_init(kqdone0 + 8 * s, kTcCoefWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kTcMmaWarp) tc::tmem_alloc(smem_u32(tmem_slot), kTcCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  // nothing below touches global memory before the previous grid has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");

  auto item_of = [&](long long it, int& b, int& hh0, int& g) {
    b = (int)(it / HI);
    hh0 = (int)(it - (long long)b * HI) * IH;
    g = hh0 / p.HPG;
  };
  // per sequence: committed records c, ring start st; a sequence whose drafts
  // would overflow its ring is skipped by every role alike
  auto seq_plan = [&](int b, int& c, int& st, bool& load) {
    c = p.count[b];
    st = p.start[b];
    load = c >= 0 && c + p.T <= p.R;
  };
  uint8_t* const qop0 = smem + p.qop_off;

  bool ok = true;
  if (warp == kTcTmaWarp) {
    // ====================================================================== TMA lane
    if (lane == 0) {
      tc::tmap_prefetch(&tmap);
      int li = 0, cur_b = -1, c = 0, st = 0;
      bool load = false;
      for (long long it = i0; it < i1; ++it) {
        int b, hh0, g;
        item_of(it, b, hh0, g);
        if (b != cur_b) { cur_b = b; seq_plan(b, c, st, load); }
        if (!load) continue;
        for (int kb = 0; kb < NKB; ++kb, ++li) {
          const int s = li % p.stages;
          if (li >= p.stages && !mbar_wait(tempty0 + 8 * s, ((li / p.stages) - 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t bar = tfull0 + 8 * s;
          mbar_arrive_tx(bar, kTcStageBytes);
          const uint32_t dst = smem_u32(smem + (size_t)s * kTcStageBytes);
#pragma unroll
          for (int j = 0; j < IH; ++j)
            tc::tma_load_2d(dst + j * P * 128, &tmap, kb * kTcKB, (int)(((long long)b * p.H + hh0 + j) * P), bar);
        }
        if (!ok) break;
      }
      if (!ok) {  // wait (bounded) for the tile copies still in flight
        volatile int dummy = 0;
        for (int k2 = 0; k2 < p.stages && k2 < li; ++k2) {
          const int i = li - 1 - k2;
          mbar_wait(tfull0 + 8 * (i % p.stages), (i / p.stages) & 1, &dummy, p.err);
        }
      }
    }
  } else if (warp == kTcGatherWarp) {
    // ====================================================================== gather lane
    if (lane == 0) {
      int li = 0, gi = 0, cur_b = -1, c = 0, st = 0;
      long long cur_gg = -1;
      bool load = false;
      const uint32_t rbytes = (uint32_t)P * ES, kbytes = (uint32_t)N * ES;
      for (long long it = i0; it < i1; ++it) {
        int b, hh0, g;
        item_of(it, b, hh0, g);
        if (b != cur_b) {
          cur_b = b;
          seq_plan(b, c, st, load);
          if (!load) atomicOr(p.err, kErrCapacity);
          cur_gg = -1;
        }
        if (!load) continue;
        const long long gg = (long long)b * p.G + g;
        if (gg != cur_gg) {
          cur_gg = gg;
          const int gs = gi & 1;
          if (gi >= 2 && !mbar_wait(gempty0 + 8 * gs, ((gi >> 1) - 1) & 1, abort_flag, p.err)) { ok = false; break; }
          const uint32_t gbar = gfull0 + 8 * gs;
          const uint32_t gdst = smem_u32(smem + p.gb_off + gs * p.gb_bytes);
          mbar_arrive_tx(gbar, (uint32_t)(c + 2 * p.T) * kbytes);
          const uint8_t* rk = reinterpret_cast<const uint8_t*>(p.ring_k) + (size_t)gg * p.R * kbytes;
          if (c > 0) {
            const int n1 = min(c, p.R - st);
            tma_load_1d(gdst, rk + (size_t)st * kbytes, (uint32_t)n1 * kbytes, gbar);
            if (c > n1) tma_load_1d(gdst + n1 * kbytes, rk, (uint32_t)(c - n1) * kbytes, gbar);
          }
          for (int t = 0; t < p.T; ++t) {
            const size_t row = ((size_t)b * p.T + t) * p.G + g;
            tma_load_1d(gdst + (c + t) * kbytes, reinterpret_cast<const uint8_t*>(p.k) + row * kbytes, kbytes, gbar);
            tma_load_1d(gdst + p.gq_off + t * kbytes, reinterpret_cast<const uint8_t*>(p.q) + row * kbytes, kbytes,
                        gbar);
          }
          ++gi;
        }
        const int sl = li % p.slots;
        if (li >= p.slots && !mbar_wait(sempty0 + 8 * sl, ((li / p.slots) - 1) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t sbar = sfull0 + 8 * sl;
        const uint32_t sdst = smem_u32(smem + p.slot_off + (size_t)sl * p.slot_bytes);
        const size_t hrow0 = (size_t)b * p.H + hh0;
        mbar_arrive_tx(sbar, (c > 0 ? (uint32_t)(IH * p.Rp * 4) : 0u) + (uint32_t)(IH * c) * rbytes +
                                 (uint32_t)(p.T * IH) * rbytes);
        if (c > 0) {
          tma_load_1d(sdst, p.ring_a + hrow0 * p.Rp, (uint32_t)(IH * p.Rp * 4), sbar);
          const int n1 = min(c, p.R - st);
          for (int j = 0; j < IH; ++j) {
            const uint8_t* rv = reinterpret_cast<const uint8_t*>(p.ring_v) + (hrow0 + j) * p.R * rbytes;
            const uint32_t d = sdst + p.sv_off + (uint32_t)(j * (p.R - p.T)) * rbytes;
            tma_load_1d(d, rv + (size_t)st * rbytes, (uint32_t)n1 * rbytes, sbar);
            if (c > n1) tma_load_1d(d + n1 * rbytes, rv, (uint32_t)(c - n1) * rbytes, sbar);
          }
        }
        for (int t = 0; t < p.T; ++t) {  // the item's IH heads are contiguous in the draft rows
          const size_t row = ((size_t)b * p.T + t) * p.H + hh0;
          tma_load_1d(sdst + p.sd_off + (uint32_t)(t * IH) * rbytes,
                      reinterpret_cast<const uint8_t*>(p.v) + row * rbytes, (uint32_t)IH * rbytes, sbar);
        }
        ++li;
      }
      if (!ok) {  // wait (bounded) for the copies still in flight
        volatile int dummy = 0;
        for (int k2 = 0; k2 < p.slots && k2 < li; ++k2) {
          const int i = li - 1 - k2;
          mbar_wait(sfull0 + 8 * (i % p.slots), (i / p.slots) & 1, &dummy, p.err);
        }
        for (int k2 = 0; k2 < 2 && k2 < gi; ++k2) {
          const int i = gi - 1 - k2;
          mbar_wait(gfull0 + 8 * (i & 1), (i >> 1) & 1, &dummy, p.err);
        }
      }
    }
  } else if (warp == kTcMmaWarp) {
    // ====================================================================== MMA lane
    if (lane == 0) {
      int li = 0, ii = 0, gi = 0, cur_b = -1, c = 0, st = 0;
      long long cur_gg = -1;
      bool load = false;
      uint32_t qaddr = 0;
      for (long long it = i0; it < i1 && ok; ++it) {
        int b, hh0, g;
        item_of(it, b, hh0, g);
        if (b != cur_b) { cur_b = b; seq_plan(b, c, st, load); cur_gg = -1; }
        if (!load) continue;
        const long long gg = (long long)b * p.G + g;
        if (gg != cur_gg) {
          cur_gg = gg;
          if (gi > 0) tc::mma_commit(qempty0 + 8 * ((gi - 1) & 1));  // the last group's operand, once read
          const int gs = gi & 1;
          if (!mbar_wait(qfull0 + 8 * gs, (gi >> 1) & 1, abort_flag, p.err)) { ok = false; break; }
          tc::fence_after_sync();
          qaddr = smem_u32(qop0 + gs * p.qop_bytes);
          ++gi;
        }
        const uint32_t buf = (uint32_t)(ii & 1) * 256u;
        const uint32_t d = tbase + buf + 128u, lo0 = tbase + buf;
        for (int kb = 0; kb < NKB; ++kb, ++li) {
          const int s = li % p.stages;
          if (!mbar_wait(sdone0 + 8 * s, (li / p.stages) & 1, abort_flag, p.err)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t a0 = smem_u32(smem + (size_t)s * kTcStageBytes);
          const uint32_t b0 = qaddr + kb * 2048;
#pragma unroll
          for (int k = 0; k < kTcKB / 8; ++k)
            tc::mma_ss(d, tc::sdesc_sw128(a0 + 32 * k), tc::sdesc_sw128(b0 + 32 * k), kIdesc, kb > 0 || k > 0);
#pragma unroll
          for (int k = 0; k < kTcKB / 8; ++k)
            tc::mma_ts(d, lo0 + kb * kTcKB + 8 * k, tc::sdesc_sw128(b0 + 32 * k), kIdesc, true);
          tc::mma_commit(tempty0 + 8 * s);  // the stage is free once these MMAs have read it
        }
        if (!ok) break;
        tc::mma_commit(dfull0 + 8 * (ii & 1));
        ++ii;
      }
      // every MMA of this CTA has completed before the tensor memory is freed
      tc::mma_commit(drain_bar);
      volatile int dummy = 0;
      mbar_wait(drain_bar, 0, &dummy, p.err);
    }
  } else if (warp >= kTcCoef0) {
    // ====================================================================== coefficient warps
    const int cwi = warp - kTcCoef0;
    float* const skq0 = reinterpret_cast<float*>(smem + p.wsc_off);  // [2 groups][t][j] k_j^T q_t, shared
    const float* skq = skq0;
    int li = 0, gi = 0, cur_b = -1, c = 0, st = 0;
    long long cur_gg = -1;
    bool load = false;
    for (long long it = i0; it < i1 && ok; ++it) {
      int b, hh0, g;
      item_of(it, b, hh0, g);
      if (b != cur_b) { cur_b = b; seq_plan(b, c, st, load); cur_gg = -1; }
      if (!load) continue;
      const long long gg = (long long)b * p.G + g;
      const int J = c + p.T;
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
        if (cwi == 0) {
          // first the queries as the MMA's B operand: fp32 (exact from bf16), [kTcT x N], K-major swizzled
          if (gi >= 2 && !__all_sync(kFull, mbar_wait(qempty0 + 8 * gs, ((gi >> 1) - 1) & 1, abort_flag, p.err))) {
            ok = false;
            break;
          }
          uint8_t* qop = qop0 + gs * p.qop_bytes;
          for (int idx = lane; idx < kTcT * N; idx += 32) {
            const int t = idx / N, n = idx - t * N;
            const float x = t < p.T ? In<__nv_bfloat16>::lds(gQ, t * N + n) : 0.f;
            *reinterpret_cast<float*>(qop + (n / kTcKB) * 2048 + tc::swz128(t, n % kTcKB)) = x;
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(qfull0 + 8 * gs);
          // the group's first item appends the draft keys (the CTA that owns it)
          const long long gfirst = ((long long)b * p.H + (long long)g * p.HPG) / IH;
          if (gfirst >= i0 && lane < p.T) {
            bulk_store(reinterpret_cast<uint8_t*>(p.ring_k) + ((size_t)gg * p.R + ring_slot(st, c + lane, p.R)) * N * ES,
                       smem_u32(gK + (c + lane) * N * ES), N * ES);
            bulk_commit();
          }
        }
        // k_j^T q_t, the two warps taking alternate (j, t) pairs, N/4 chunks from a lane-dependent start
        float* kq = skq0 + gs * kTcT * kRMax;
        const int npair = J * p.T;
        for (int pr = cwi * 32 + lane; pr < npair; pr += 32 * kTcCoefWarps) {
          const int t = pr / J, j = pr - t * J;
          float acc = 0.f;
#pragma unroll 8
          for (int i = 0; i < N / 4; ++i) {
            const int c4 = (i + lane) & (N / 4 - 1);
            acc += dot4(In<__nv_bfloat16>::lds4(gK, j * N + 4 * c4), In<__nv_bfloat16>::lds4(gQ, t * N + 4 * c4));
          }
          kq[t * kRMax + j] = acc;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(kqdone0 + 8 * gs);
        if (!__all_sync(kFull, mbar_wait(kqdone0 + 8 * gs, (gi >> 1) & 1, abort_flag, p.err))) { ok = false; break; }
        skq = kq;
        ++gi;
      }
      const int sl = li % p.slots;
      const int use = li / p.slots;
      ++li;
      if (((li - 1) % kTcCoefWarps) != cwi) continue;  // the other coefficient warp takes this item
      if (!__all_sync(kFull, mbar_wait(sfull0 + 8 * sl, use & 1, abort_flag, p.err))) { ok = false; break; }
      uint8_t* slot = smem + p.slot_off + (size_t)sl * p.slot_bytes;
      for (int j = 0; j < IH; ++j) {
        const size_t hrow = (size_t)b * p.H + hh0 + j;
        const float* sa = reinterpret_cast<const float*>(slot) + j * p.Rp;  // committed decays, ring order
        float* sc = reinterpret_cast<float*>(slot + p.sc_off) + j * kTcCoefFloats;
        const float aj = (lane < c) ? sa[ring_slot(st, lane, p.R)] : 1.f;
        const float ad = (lane < p.T) ? p.alpha[((size_t)b * p.T + lane) * p.H + hh0 + j] : 1.f;  // draft decays
        // query t sees records 0 .. c + t: the weight of record l is
        // (alpha_{l+1} .. alpha_{c-1}) (alpha_{max(l+1,c)} .. alpha_{c+t}) (k_l^T q_t),
        // and the checkpoint term is scaled by alpha_0 .. alpha_{c+t}
        const float sfx = suffix_prod((lane < c) ? aj : 1.f, lane);
        const float dn = __shfl_down_sync(kFull, sfx, 1);
        const float dpart = (lane < 31) ? dn : 1.f;
        const float call = __shfl_sync(kFull, sfx, 0);
        const int s0 = max(lane + 1 - c, 0);
        float np = 1.f, nall = 1.f;
        for (int t = 0; t < p.T; ++t) {
          const float at = __shfl_sync(kFull, ad, t);
          nall *= at;
          if (t >= s0) np *= at;
          sc[kTcT + t * kRMax + lane] = (lane < c + t + 1) ? dpart * np * skq[t * kRMax + lane] : 0.f;
          if (lane == 0) sc[t] = call * nall;
        }
        if (lane < p.T) p.ring_a[hrow * p.Rp + ring_slot(st, c + lane, p.R)] = ad;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(scoef0 + 8 * sl);
    }
    bulk_wait_all();
  } else {
    // ====================================================================== row warps
    const int set = warp / kTcSetWarps, sw = warp - set * kTcSetWarps;  // this warp's set and rank in it
    const int quarter = sw & 3, half = sw >> 2;
    const int row = 32 * quarter + lane;         // checkpoint row of the item (tensor-memory lane)
    const int hj = row / P, pr = row - hj * P;   // head within the item, row within the head
    const uint32_t tl = (uint32_t)(32 * quarter) << 16;
    int li = 0, ii = 0, si = 0, cur_b = -1, c = 0, st = 0;
    bool load = false;
    // the item waiting for its epilogue
    bool pend = false;
    int pb = 0, phh = 0, pc = 0, pst = 0, pii = 0, psl = 0, puse = 0;

    auto epilogue = [&]() -> bool {
      const uint32_t buf = (uint32_t)(pii & 1) * 256u;
      if (!__all_sync(kFull, mbar_wait(dfull0 + 8 * (pii & 1), (pii >> 1) & 1, abort_flag, p.err))) return false;
      tc::fence_after_sync();
      uint32_t dv[8];
      tc::tmem_ld8(tbase + tl + buf + 128u + 8u * half, dv);
      tc::tmem_ld_wait();
      if (!__all_sync(kFull, mbar_wait(scoef0 + 8 * psl, puse & 1, abort_flag, p.err))) return false;
      const uint8_t* slot = smem + p.slot_off + (size_t)psl * p.slot_bytes;
      const float* sc = reinterpret_cast<const float*>(slot + p.sc_off) + hj * kTcCoefFloats;
      const uint8_t* svh = slot + p.sv_off + (size_t)hj * (p.R - p.T) * P * ES;  // committed rows of my head
      const uint8_t* sdr = slot + p.sd_off + (size_t)hj * P * ES;                 // my head's draft rows
      const int J = pc + p.T;
      const int t0 = 8 * half;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = sc[t0 + i] * __uint_as_float(dv[i]);
      // value term: records in fours, each weight row of a query read as float4
      // (the weights past c + t are zero, and records past J read as zero)
      for (int j0 = 0; j0 < J; j0 += 4) {
        float v4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jj = j0 + u;
          v4[u] = jj >= J ? 0.f
                  : jj < pc ? In<__nv_bfloat16>::lds(svh, jj * P + pr)
                            : In<__nv_bfloat16>::lds(sdr, (jj - pc) * IH * P + pr);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 w = *reinterpret_cast<const float4*>(sc + kTcT + (t0 + i) * kRMax + j0);
          acc[i] = fmaf(w.x, v4[0], fmaf(w.y, v4[1], fmaf(w.z, v4[2], fmaf(w.w, v4[3], acc[i]))));
        }
      }
      const size_t hh = (size_t)phh + hj;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = t0 + i;
        if (t < p.T) p.o[(((size_t)pb * p.T + t) * p.H + hh) * P + pr] = acc[i];
      }
      if (half == 0) {  // append the draft value rows of my row
        const size_t hrow = (size_t)pb * p.H + hh;
        const __nv_bfloat16* dr = reinterpret_cast<const __nv_bfloat16*>(sdr);
        for (int t = 0; t < p.T; ++t)
          p.ring_v[(hrow * p.R + ring_slot(pst, pc + t, p.R)) * P + pr] = dr[t * IH * P + pr];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sempty0 + 8 * psl);
      return true;
    };

    for (long long it = i0; it < i1 && ok; ++it) {
      int b, hh0, g;
      item_of(it, b, hh0, g);
      if (b != cur_b) { cur_b = b; seq_plan(b, c, st, load); }
      if (!load) continue;
      if ((ii % kTcSets) != set) {  // the other set's item: count its stages, buffer and slot
        li += NKB;
        ++ii;
        ++si;
        continue;
      }
      // ---- the set's previous item's epilogue first: its MMAs have completed once its
      // accumulator is read (the wait inside), so this item's split may overwrite the
      // buffer's lo columns and this item's MMAs its accumulator. The other set's
      // work fills the SM meanwhile.
      if (pend && !epilogue()) { ok = false; break; }
      pend = false;
      // ---- split: lo = S - hi into this item's tensor-memory buffer. The
      // four warps of a half take K-blocks half, half + 2, ...: whole 128-byte rows,
      // one 32-column store to tensor memory each, one fence sequence per item.
      const uint32_t lo0 = tbase + tl + (uint32_t)(ii & 1) * 256u;
      for (int kb = half; kb < NKB; kb += 2) {
        const int lk = li + kb, s = lk % p.stages;
        if (!__all_sync(kFull, mbar_wait(tfull0 + 8 * s, (lk / p.stages) & 1, abort_flag, p.err))) { ok = false; break; }
        uint8_t* tile = smem + (size_t)s * kTcStageBytes + row * 128;
        uint32_t lo[32];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          // kind::tf32 reads an fp32 operand's sign, exponent and top 10 mantissa bits
          // and ignores the low 13: the MMA of the tile as stored is the MMA of hi
          const uint4 x = *reinterpret_cast<const uint4*>(tile + ((ch ^ (row & 7)) << 4));
          const uint4 h = make_uint4(x.x & 0xFFFFE000u, x.y & 0xFFFFE000u, x.z & 0xFFFFE000u, x.w & 0xFFFFE000u);
          lo[4 * ch + 0] = __float_as_uint(__uint_as_float(x.x) - __uint_as_float(h.x));
          lo[4 * ch + 1] = __float_as_uint(__uint_as_float(x.y) - __uint_as_float(h.y));
          lo[4 * ch + 2] = __float_as_uint(__uint_as_float(x.z) - __uint_as_float(h.z));
          lo[4 * ch + 3] = __float_as_uint(__uint_as_float(x.w) - __uint_as_float(h.w));
        }
        tc::tmem_st32(lo0 + kb * kTcKB, lo);
      }
      if (!ok) break;
      tc::tmem_st_wait();
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0)
        for (int kb = half; kb < NKB; kb += 2) mbar_arrive(sdone0 + 8 * ((li + kb) % p.stages));
      li += NKB;
      pend = true;
      pb = b; phh = hh0; pc = c; pst = st; pii = ii; psl = si % p.slots; puse = si / p.slots;
      ++ii;
      ++si;
    }
    if (ok && pend && !epilogue()) ok = false;
  }

  // ------------------------------------------------------------------ teardown
  // Every role has left its loop with nothing in flight (bounded drains above);
  // the MMA warp frees the tensor memory once all threads are here.
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, kTcCols);
  }
}

}  // namespace rssm
