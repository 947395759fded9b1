// rssm_api.cu - the C ABI of librssm.so (declared in include/rssm.h).
//
// Host side only: it validates arguments, derives buffer layouts and launch
// shapes, and enqueues kernels on the caller's stream. It never allocates
// device memory. Errors are returned as rssm_status. The message is kept per
// thread for rssm_last_error().
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "../../include/rssm.h"
#include "rssm_launch.cuh"
#include "rssm_nonflush.cuh"
#include "rssm_verify_tc.cuh"

namespace {

thread_local std::string g_msg = "no error";

rssm_status fail(rssm_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_msg = buf;
  return s;
}

rssm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RSSM_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Delta-rule layers verify at most this many drafts (2 T vectors per row).
constexpr int kDeltaTMax = 4;

// Tensor-core verify: used by default from this many drafts up (more than the
// CUDA-core verify takes); below it the CUDA-core verify measures faster.
constexpr int kTcAutoMinT = 9;

struct Geom {
  int R = 0, Rp = 0, esize = 0, ck_es = 4, rf = 0;  // ck_es: checkpoint bytes per element; rf: tile format
  bool tc_ok = false;  // the tensor-core verify serves this configuration
  size_t v_off = 0, k_off = 0, ring_bytes = 0;
  size_t off_count = 0, off_ticket = 0, off_err = 0, off_epoch = 0, off_flist = 0, off_fcount = 0, ptr_bytes = 0;
  size_t head_stride = 0, bsc_off = 0, rsc_off = 0, copy_bytes = 0;
};

// Validate a configuration and derive the buffer layouts.
rssm_status derive(const rssm_config* c, Geom* g) {
  if (!c) return fail(RSSM_EINVAL, "config is NULL");
  if (c->B < 1 || c->H < 1 || c->P < 1 || c->N < 1 || c->G < 1 || c->L < 1 || c->T_max < 1)
    return fail(RSSM_EINVAL, "sizes must be positive (B=%d H=%d P=%d N=%d G=%d L=%d T_max=%d)", c->B, c->H,
                c->P, c->N, c->G, c->L, c->T_max);
  if (c->H % c->G) return fail(RSSM_EINVAL, "H=%d is not a multiple of G=%d", c->H, c->G);
  if (c->in_dtype != RSSM_F32 && c->in_dtype != RSSM_BF16) return fail(RSSM_EINVAL, "in_dtype %d", c->in_dtype);
  if (c->read_fmt < RSSM_READ_NONE || c->read_fmt > RSSM_READ_E2M1_B16)
    return fail(RSSM_EINVAL, "read_fmt %d", c->read_fmt);
  if (c->N != 16 && c->N != 32 && c->N != 64 && c->N != 128)
    return fail(RSSM_EUNSUPPORTED, "N=%d (supported: 16, 32, 64, 128)", c->N);
  if (c->P % 8) return fail(RSSM_EUNSUPPORTED, "P=%d must be a multiple of 8", c->P);
  if ((size_t)c->P * c->N * 4 > 64 * 1024) return fail(RSSM_EUNSUPPORTED, "P*N*4 > 64 KiB");
  if (c->P > 128) return fail(RSSM_EUNSUPPORTED, "P=%d > 128", c->P);
  // The tensor-core verify: bf16 inputs, an FP32 checkpoint of the outer-product
  // recurrence, N in {64, 128}, and 128 checkpoint rows holding whole heads of one group.
  g->tc_ok = c->in_dtype == RSSM_BF16 && c->ckpt_fmt == RSSM_CKPT_F32 && c->recurrence == RSSM_GATED_OUTER &&
             (c->N == 64 || c->N == 128) && (c->P == 32 || c->P == 64 || c->P == 128) && c->G > 0 &&
             c->H % c->G == 0 && (c->H / c->G) % (128 / c->P) == 0;
  if (c->T_max > rssm::kTcT) return fail(RSSM_EUNSUPPORTED, "T_max=%d > %d", c->T_max, rssm::kTcT);
  if (c->T_max > rssm::kTMax && !g->tc_ok)
    return fail(RSSM_EUNSUPPORTED,
                "T_max=%d > %d needs the tensor-core verify (bf16 inputs, FP32 checkpoint, outer-product recurrence, "
                "N in {64, 128}, P in {32, 64, 128}, H/G a multiple of 128/P)",
                c->T_max, rssm::kTMax);
  const int R = c->L + c->T_max - 1;
  if (R > rssm::kRMax) return fail(RSSM_EUNSUPPORTED, "R = L + T_max - 1 = %d > %d", R, rssm::kRMax);
  if (c->read_fmt != RSSM_READ_NONE && c->N < 64)
    return fail(RSSM_EUNSUPPORTED, "read copies need N in {64, 128}");
  if (c->ckpt_fmt < RSSM_CKPT_F32 || c->ckpt_fmt > RSSM_CKPT_F16_RN) return fail(RSSM_EINVAL, "ckpt_fmt %d", c->ckpt_fmt);
  if (c->ckpt_fmt != RSSM_CKPT_F32 && (c->N < 64 || c->read_fmt != RSSM_READ_NONE))
    return fail(RSSM_EUNSUPPORTED, "an FP16 checkpoint needs N in {64, 128} and no read copy");
  if (c->recurrence != RSSM_GATED_OUTER && c->recurrence != RSSM_GATED_DELTA)
    return fail(RSSM_EINVAL, "recurrence %d", c->recurrence);
  if (c->recurrence == RSSM_GATED_DELTA &&
      (c->N < 64 || c->read_fmt != RSSM_READ_NONE || c->ckpt_fmt != RSSM_CKPT_F32 || c->T_max > kDeltaTMax))
    return fail(RSSM_EUNSUPPORTED,
                "a delta-rule layer needs N in {64, 128}, an FP32 checkpoint, no read copy and T_max <= %d", kDeltaTMax);
  if ((long long)c->B * c->H > (1ll << 30)) return fail(RSSM_EUNSUPPORTED, "B*H too large");
  g->R = R;
  g->Rp = (R + 3) / 4 * 4;
  g->esize = c->in_dtype == RSSM_F32 ? 4 : 2;
  g->ck_es = c->ckpt_fmt == RSSM_CKPT_F32 ? 4 : 2;
  g->rf = c->recurrence == RSSM_GATED_DELTA ? (int)rssm::kDelta
         : c->ckpt_fmt != RSSM_CKPT_F32    ? (int)rssm::kCkF16
                                           : c->read_fmt;
  const size_t B = c->B, H = c->H, P = c->P, N = c->N, G = c->G;
  const size_t a_bytes = B * H * g->Rp * 4;
  // delta layers keep each record's pseudo-value w (fp32) where the others keep v
  const size_t w_es = c->recurrence == RSSM_GATED_DELTA ? 4 : (size_t)g->esize;
  g->v_off = align_up(a_bytes, 256);
  g->k_off = align_up(g->v_off + B * H * R * P * w_es, 256);
  g->ring_bytes = align_up(g->k_off + B * G * R * N * g->esize, 256);
  const size_t pb = align_up(B * 4, 256);
  g->off_count = pb;
  g->off_ticket = 2 * pb;
  g->off_err = 3 * pb;
  g->off_epoch = 3 * pb + 256;
  g->off_flist = 4 * pb + 256;   // the standalone flush's list of folding sequences
  g->off_fcount = 5 * pb + 256;  // and their number
  g->ptr_bytes = 5 * pb + 512;
  if (c->read_fmt == RSSM_READ_E4M3_ROW) {
    g->bsc_off = P * N;
    g->rsc_off = P * N;
    g->head_stride = align_up(P * N + 4 * P, 16);
  } else if (c->read_fmt == RSSM_READ_E2M1_B16) {
    g->bsc_off = P * N / 2;
    g->rsc_off = align_up(g->bsc_off + P * N / 16, 16);
    g->head_stride = align_up(g->rsc_off + 4 * P, 16);
  }
  g->copy_bytes = B * H * g->head_stride;
  return RSSM_OK;
}

struct Plan {
  int stages = 0;
  size_t smem = 0;
  rssm::Params p{};
};

// Shared-memory plan of a head-kernel launch: the group areas, scratch and
// barriers at the top of the CTA's shared memory, and below them two layouts of
// tile stages and record slots (see rssm::Params). lay[0] fits every head.
// lay[1], offered to decode steps, holds only non-flush heads: its stages hold
// the tile that non-flush steps read (the read copy when there is one) and its
// slots at most L - 1 records and no fold coefficients, so more heads fit.
enum class LayoutKind { kGeneral, kNonFlush, kVerify };

rssm_status plan_layout(const rssm_config* c, const Geom& g, LayoutKind kind, size_t budget, rssm::Layout* L) {
  using namespace rssm;
  auto a128 = [](size_t x) { return align_up(x, 128); };
  const bool nf = kind == LayoutKind::kNonFlush;
  const size_t P = c->P, N = c->N, es = (size_t)g.esize, R = g.R;
  const size_t tile = a128(nf && g.head_stride ? g.head_stride : P * N * (size_t)g.ck_es);
  const size_t vrows = nf ? (size_t)c->L : R;
  // decays: kRMax ring slots, then kTMax new records; delta layers keep the new
  // records' write strengths the same way right after them, their buffered
  // pseudo-values (fp32) as the value rows and the new record's v row after those
  const bool delta = g.rf == rssm::kDelta;
  const size_t sv_off = (size_t)(kRMax + kTMax) * 4 * (delta ? 2 : 1);
  const size_t nv_off = sv_off + vrows * P * (delta ? 4 : es);
  const size_t sc_off = align_up(nv_off + (delta ? (size_t)c->T_max * P * es : 0), 16);
  // coefficients: 16 scalars, then the record weights [kRMax] (non-flush),
  // [kTMax][kRMax] (verify), or the fold's scaled values [R][P] (general, which
  // also serves non-flush heads). Delta layers: 16 scalars, the output weights
  // and the new record's couplings [kRMax] each, then (general) the fold's
  // scaled values [R][P].
  // Delta-rule verify: 16 scalars, the committed weights [kTMax][kRMax] of 2T vectors,
  // then the drafts' couplings E and F [4][4] each.
  const size_t sc_floats = delta ? (kind == LayoutKind::kVerify ? 16 + (size_t)kTMax * kRMax + 32
                                                                : 16 + 2 * (size_t)kRMax + (nf ? 0 : R * P))
                         : nf    ? 16 + std::max(P, (size_t)kRMax)
                              : kind == LayoutKind::kVerify ? 16 + (size_t)kTMax * kRMax
                                                            : 16 + std::max({(size_t)kRMax, R * P, (size_t)c->T_max * P});
  const size_t slot = a128(sc_off + sc_floats * 4);
  if (2 * tile + 2 * slot > budget) return fail(RSSM_EUNSUPPORTED, "tile too large for shared memory");
  const int stages = (int)std::max<size_t>(2, std::min<size_t>(kMaxStages, budget / (tile + 3 * slot)));
  const int slots = (int)std::max<size_t>(2, std::min<size_t>(kMaxSlots, (budget - stages * tile) / slot));
  // Dot groups: as many heads in flight as keeps two tile stages per group.
  int dgroups = 1;
  while (dgroups < 8 && stages >= 4 * dgroups && slots >= 4 * dgroups) dgroups *= 2;
  // verify heads are compute-heavier (T queries): one stage per dot group measured best
  if (kind == LayoutKind::kVerify)
    while (dgroups < 8 && stages >= 2 * dgroups && slots >= 4 * dgroups) dgroups *= 2;
  while (dgroups > 1 && (stages < dgroups || slots < dgroups)) dgroups /= 2;
  // Every ring's length must be a multiple of the number of consumers that take
  // its entries in turn. Then the previous use of an entry belongs to the same
  // consumer and has completed, and an mbarrier parity wait cannot be satisfied
  // by the previous phase.
  const int stages_used = stages - stages % dgroups;
  const int slot_mult = std::max(kNCoef, dgroups);  // both are powers of two
  const int slots_used = slots - slots % slot_mult;
  if (stages_used < 2 || slots_used < slot_mult) return fail(RSSM_EUNSUPPORTED, "shared memory too small for the rings");
  L->dgroups = dgroups;
  L->stages = stages_used;
  L->stage_bytes = (int)tile;
  L->slots = slots_used;
  L->slot_bytes = (int)slot;
  L->slot_off = (int)((size_t)stages_used * tile);
  L->sv_off = (int)sv_off;
  L->nv_off = (int)nv_off;
  L->sc_off = (int)sc_off;
  if ((size_t)L->slot_off + (size_t)slots_used * slot > budget) return fail(RSSM_EUNSUPPORTED, "shared memory plan too large");
  return RSSM_OK;
}

// kind: kGeneral (flush, quantize, conventional), kNonFlush (decode: the general
// layout plus the non-flush one), kVerify (verify: no fold area).
rssm_status plan_smem(const rssm_config* c, const Geom& g, Plan* pl, LayoutKind kind = LayoutKind::kGeneral) {
  using namespace rssm;
  auto a128 = [](size_t x) { return align_up(x, 128); };
  const size_t N = c->N, es = (size_t)g.esize, R = g.R;
  const size_t gq_off = R * N * es;
  const size_t gb = a128(gq_off + (size_t)kTMax * N * es);
  const size_t wsc = a128((size_t)kNCoef * kTMax * kRMax * 4);
  // delta-rule verify: per dot warp, 32 rows of 2T <= 8 sums
  const size_t dsc = (g.rf == kDelta && kind == LayoutKind::kVerify) ? (size_t)kNDW * 32 * 8 * 4 : 0;
  const size_t bars = a128((2 * kMaxStages + 3 * kMaxSlots + 6) * 8);
  const size_t fixed = 2 * gb + wsc + dsc + bars;
  if (fixed >= (size_t)kSmemMax) return fail(RSSM_EUNSUPPORTED, "group areas too large for shared memory");
  const size_t budget = ((size_t)kSmemMax - fixed) / 128 * 128;
  rssm::Params& p = pl->p;
  rssm_status s = plan_layout(c, g, kind == LayoutKind::kVerify ? LayoutKind::kVerify : LayoutKind::kGeneral, budget,
                              &p.lay[0]);
  if (s != RSSM_OK) return s;
  p.lay[1] = p.lay[0];
  p.nf_ok = 0;
  if (kind == LayoutKind::kNonFlush && c->L >= 2 &&
      plan_layout(c, g, LayoutKind::kNonFlush, budget, &p.lay[1]) == RSSM_OK)
    p.nf_ok = 1;
  size_t off = budget;
  p.gb_off = (int)off; off += 2 * gb;
  p.gb_bytes = (int)gb;
  p.gq_off = (int)gq_off;
  p.wsc_off = (int)off; off += wsc;
  p.dsc_off = (int)off; off += dsc;
  p.bar_off = (int)off; off += bars;
  if (off > (size_t)kSmemMax) return fail(RSSM_EUNSUPPORTED, "shared memory plan too large");
  pl->stages = p.lay[0].stages;
  pl->smem = off;
  return RSSM_OK;
}

// Shared-memory plan of the tensor-core verify for T drafts: 16 KiB K-block
// stages from the 1024-aligned base, two B operands, record slots, two group
// areas, the coefficient scratch and the barriers.
rssm_status plan_tc(const rssm_config* c, const Geom& g, int T, rssm::TcParams* tp, size_t* smem) {
  using namespace rssm;
  auto a128 = [](size_t x) { return align_up(x, 128); };
  const size_t N = c->N, P = c->P, R = g.R, Rp = g.Rp, IH = 128 / P, NKB = N / kTcKB;
  if (T < 1 || T > kTcT || (size_t)T > R) return fail(RSSM_EINVAL, "T=%d for the tensor-core verify", T);
  const size_t qop = NKB * 2048;
  const size_t sv = IH * Rp * 4;
  const size_t sd = sv + IH * (R - T) * P * 2;
  const size_t scf = sd + (size_t)T * IH * P * 2;
  const size_t slot = a128(scf + IH * (size_t)kTcCoefFloats * 4);
  const size_t gq = R * N * 2;
  const size_t gb = a128(gq + (size_t)kTcT * N * 2);
  const size_t wsc = (size_t)kTcCoefWarps * kTcT * kRMax * 4;
  const size_t bars = a128((3 * (size_t)kTcMaxStages + 3 * (size_t)kTcMaxSlots + 15) * 8);
  const size_t fixed = 2 * qop + 2 * gb + wsc + bars;
  if (fixed + NKB * (size_t)kTcStageBytes + 2 * slot > (size_t)kSmemMax)
    return fail(RSSM_EUNSUPPORTED, "the tensor-core verify does not fit shared memory");
  const size_t budget = (size_t)kSmemMax - fixed;
  size_t slots = 4;
  size_t stages = std::min<size_t>(kTcMaxStages, budget >= slots * slot ? (budget - slots * slot) / kTcStageBytes : 0);
  if (stages < (size_t)kTcSets * NKB) {
    slots = 2;
    stages = std::min<size_t>(kTcMaxStages, (budget - slots * slot) / kTcStageBytes);
  }
  // each row-warp set keeps its own stages: a multiple of kTcSets items' K-blocks
  stages -= stages % ((size_t)kTcSets * NKB);
  if (stages < (size_t)kTcSets * NKB)
    return fail(RSSM_EUNSUPPORTED, "the tensor-core verify does not fit shared memory");
  tp->stages = (int)stages;
  tp->slots = (int)slots;
  size_t off = stages * kTcStageBytes;
  tp->qop_off = (int)off; tp->qop_bytes = (int)qop; off += 2 * qop;
  tp->slot_off = (int)off; tp->slot_bytes = (int)slot; off += slots * slot;
  tp->sv_off = (int)sv; tp->sd_off = (int)sd; tp->sc_off = (int)scf;
  tp->gb_off = (int)off; tp->gb_bytes = (int)gb; tp->gq_off = (int)gq; off += 2 * gb;
  tp->wsc_off = (int)off; off += wsc;
  off = align_up(off, 16);
  tp->bar_off = (int)off; off += bars;
  if (off > (size_t)kSmemMax) return fail(RSSM_EUNSUPPORTED, "tensor-core verify plan too large");
  // more than half of the shared memory: one CTA per SM, so a CTA never waits
  // for tensor memory held by another CTA of the same kernel
  *smem = std::max<size_t>(off, (size_t)kSmemMax / 2 + 1024);
  return RSSM_OK;
}

// derive() plus a check that every launch of a handle with this configuration
// fits one CTA's shared memory, so that an unplaceable size is refused when the
// buffers are sized and the handle is made, not at its first launch.
rssm_status derive_placed(const rssm_config* c, Geom* g) {
  rssm_status s = derive(c, g);
  if (s != RSSM_OK) return s;
  Plan pl;
  s = plan_smem(c, *g, &pl);
  if (s == RSSM_OK && c->T_max > 1) s = plan_smem(c, *g, &pl, LayoutKind::kVerify);
  if (s == RSSM_OK && c->T_max > 1 && g->tc_ok) {
    rssm::TcParams tp{};
    size_t smem = 0;
    s = plan_tc(c, *g, c->T_max, &tp, &smem);
  }
  if (s != RSSM_OK)
    return fail(s, "P=%d N=%d R=%d with %s inputs does not fit one CTA's shared memory (%s)", c->P, c->N, g->R,
                c->in_dtype == RSSM_F32 ? "f32" : "bf16", g_msg.c_str());
  return RSSM_OK;
}

int sm_count() {
  thread_local int cached_dev = -1, cached = 0;  // per thread: no shared mutable state
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached = n;
    cached_dev = dev;
  }
  return cached;
}

}  // namespace

struct rssm_ctx {
  CUtensorMap tmap;  // the checkpoint as rows of N fp32, 32 x P boxes, 128-byte swizzle (tensor-core verify)
  rssm_config cfg;
  Geom g;
  void* ckpt;  // fp32 or fp16 [B,H,P,N]
  uint8_t* ring;
  uint8_t* ptrs;
  uint8_t* copy;
  int last_T;         // draft count of the last verify, 0 when none is pending
  int verify_kernel;  // 0 automatic, 1 CUDA cores, 2 tensor cores
  int decode_kernel;  // 0 automatic, 1 the pipelined head kernel only, 2 warp-per-head non-flush step first
  Plan dplan;         // the decode launch plan with the handle's buffers filled in (made once, at creation)
};

namespace {

void fill_common(const rssm_ctx* h, rssm::Params* p) {
  const rssm_config& c = h->cfg;
  p->B = c.B; p->H = c.H; p->P = c.P; p->N = c.N; p->G = c.G; p->L = c.L;
  p->R = h->g.R; p->Rp = h->g.Rp; p->HPG = c.H / c.G; p->T = 1; p->min_count = 1;
  p->ckpt = static_cast<float*>(h->ckpt);  // the kernels read fp16 checkpoints through byte offsets
  p->copy = h->copy;
  p->head_stride = (int)h->g.head_stride;
  p->bsc_off = (int)h->g.bsc_off;
  p->rsc_off = (int)h->g.rsc_off;
  p->ring_a = reinterpret_cast<float*>(h->ring);
  p->ring_v = h->ring + h->g.v_off;
  p->ring_k = h->ring + h->g.k_off;
  p->start = reinterpret_cast<int32_t*>(h->ptrs);
  p->count = reinterpret_cast<int32_t*>(h->ptrs + h->g.off_count);
  p->ticket = reinterpret_cast<int32_t*>(h->ptrs + h->g.off_ticket);
  p->err = reinterpret_cast<uint32_t*>(h->ptrs + h->g.off_err);
  p->epoch = reinterpret_cast<int32_t*>(h->ptrs + h->g.off_epoch);
  p->seed = c.seed;
  p->sr = c.ckpt_fmt == RSSM_CKPT_F16_SR ? 1 : 0;
}

int persistent_grid(long long heads) {
  const int sms = sm_count();
  return (int)std::max(1ll, std::min<long long>(heads, sms > 0 ? sms : 1));
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// The checkpoint [B,H,P,N] fp32 as a 2-D tensor of B*H*P rows of N elements,
// read in boxes of 32 columns x P rows (one head's K-block) with the 128-byte swizzle.
rssm_status make_ckpt_tensor_map(const rssm_config* c, void* ckpt, CUtensorMap* out) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(RSSM_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {(cuuint64_t)c->N, (cuuint64_t)c->B * c->H * c->P};
  const cuuint64_t strides[1] = {(cuuint64_t)c->N * 4};
  const cuuint32_t box[2] = {32, (cuuint32_t)c->P};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ckpt, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RSSM_ECUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return RSSM_OK;
}

// Which verify kernel a launch of T drafts takes: 2 tensor cores, 1 CUDA cores.
int verify_kernel_for(const rssm_ctx* h, int T) {
  if (!h->g.tc_ok || h->g.rf == rssm::kDelta) return 1;
  if (h->verify_kernel == 1 && T <= rssm::kTMax) return 1;
  if (h->verify_kernel == 2) return 2;
  return (T >= kTcAutoMinT || T > rssm::kTMax) ? 2 : 1;
}

// The warp-per-head non-flush step serves the small head tiles: an E4M3 or E2M1
// read copy, or an FP16 checkpoint (N in {64, 128}, outer-product recurrence).
bool nonflush_applies_fmt(const Geom& g) {
  return g.rf == rssm::kRfE4m3 || g.rf == rssm::kRfE2m1 || g.rf == rssm::kCkF16;
}

// The per-warp stages of the warp-per-head step, and how many warps fit a CTA.
rssm::NfStage nonflush_stage(const rssm_config& c, const Geom& g) {
  const int tile = g.rf == rssm::kCkF16 ? c.P * c.N * 2 : (int)g.head_stride;
  return rssm::nf_stage(tile, c.L, g.Rp, c.P, g.esize);
}
int nonflush_warps(const rssm::NfStage& sg) {
  return std::min(rssm::kNfMaxWarps, (rssm::kSmemMax - rssm::kNfCtaBytes) / rssm::nf_warp_bytes(sg));
}
size_t nonflush_smem(const rssm::NfStage& sg, int warps) {
  return rssm::kNfCtaBytes + (size_t)warps * rssm::nf_warp_bytes(sg);
}

bool nonflush_applies(const rssm_config& c, const Geom& g) {
  return nonflush_applies_fmt(g) && nonflush_warps(nonflush_stage(c, g)) >= 1;
}

// Which decode kernels a step launches: 2 the warp-per-head non-flush step and
// then the head kernel for the flushing sequences, 1 the head kernel alone.
int decode_kernel_for(const rssm_ctx* h) {
  if (!nonflush_applies(h->cfg, h->g) || h->decode_kernel == 1) return 1;
  if (h->decode_kernel == 2) return 2;
  // automatic: the read copies; an FP16 checkpoint's 16 KiB tiles fit too few
  // warps per SM, and the head kernel alone measures as fast there
  return h->g.rf == rssm::kCkF16 ? 1 : 2;
}

// Enqueue one decode step with the parameters in p (pointers, inputs, ticket block set).
cudaError_t launch_decode_step(const rssm_ctx* h, rssm::Params& p, size_t smem, cudaStream_t st) {
  const long long heads = (long long)h->cfg.B * h->cfg.H;
  if (decode_kernel_for(h) == 2) {
    const rssm::NfStage sg = nonflush_stage(h->cfg, h->g);
    const int warps = nonflush_warps(sg);
    const long long want = (heads + warps - 1) / warps;
    const int grid = (int)std::max(1ll, std::min<long long>(want, (long long)std::max(1, sm_count())));
    const cudaError_t e =
        rssm::launch_nonflush(p, sg, grid, warps, nonflush_smem(sg, warps), st, h->cfg.N, h->cfg.in_dtype, h->g.rf);
    if (e != cudaSuccess) return e;
    p.skip_nonflush = 1;
  }
  return rssm::launch_decode(p, persistent_grid(heads), smem, st, h->cfg.N, h->cfg.in_dtype, h->g.rf);
}

}  // namespace

extern "C" {

const char* rssm_last_error(void) { return g_msg.c_str(); }

rssm_status rssm_workspace_size(const rssm_config* cfg, size_t* ring_bytes, size_t* ptr_bytes,
                                size_t* read_copy_bytes) {
  Geom g;
  const rssm_status s = derive_placed(cfg, &g);
  if (s != RSSM_OK) return s;
  if (ring_bytes) *ring_bytes = g.ring_bytes;
  if (ptr_bytes) *ptr_bytes = g.ptr_bytes;
  if (read_copy_bytes) *read_copy_bytes = g.copy_bytes;
  return RSSM_OK;
}

rssm_status rssm_ring_offsets(const rssm_config* cfg, size_t* v_off, size_t* k_off) {
  Geom g;
  const rssm_status s = derive_placed(cfg, &g);
  if (s != RSSM_OK) return s;
  if (v_off) *v_off = g.v_off;
  if (k_off) *k_off = g.k_off;
  return RSSM_OK;
}

rssm_status rssm_read_copy_layout(const rssm_config* cfg, size_t* head_stride, size_t* bscale_off,
                                  size_t* rscale_off) {
  Geom g;
  const rssm_status s = derive_placed(cfg, &g);
  if (s != RSSM_OK) return s;
  if (cfg->read_fmt == RSSM_READ_NONE) return fail(RSSM_EINVAL, "configuration has no read copy");
  if (head_stride) *head_stride = g.head_stride;
  if (bscale_off) *bscale_off = g.bsc_off;
  if (rscale_off) *rscale_off = g.rsc_off;
  return RSSM_OK;
}

rssm_status rssm_launch_plan(const rssm_config* cfg, int32_t kind, rssm_launch_plan_info* out) {
  if (!out) return fail(RSSM_EINVAL, "out is NULL");
  if (kind < 0 || kind > 4)
    return fail(RSSM_EINVAL, "kind=%d (0 flush, 1 decode, 2 verify, 3 tensor-core verify, 4 warp-per-head step)",
                kind);
  Geom g;
  rssm_status s = derive(cfg, &g);
  if (s != RSSM_OK) return s;
  if (kind == 4) {
    if (!nonflush_applies_fmt(g))
      return fail(RSSM_EUNSUPPORTED, "the warp-per-head non-flush step serves read copies and FP16 checkpoints");
    const rssm::NfStage sg = nonflush_stage(*cfg, g);
    const int warps = nonflush_warps(sg);
    if (warps < 1) return fail(RSSM_EUNSUPPORTED, "one warp's stages do not fit a CTA's shared memory");
    *out = rssm_launch_plan_info{};
    out->smem_bytes = (int64_t)nonflush_smem(sg, warps);
    out->stages[0] = 2;
    out->stage_bytes[0] = sg.tbytes;
    out->slots[0] = 1;
    out->slot_bytes[0] = sg.vbytes;
    out->dgroups[0] = warps;
    return RSSM_OK;
  }
  if (kind >= 2 && cfg->T_max < 2) return fail(RSSM_EINVAL, "verify launches need T_max > 1");
  if (kind == 3 && cfg->recurrence != RSSM_GATED_OUTER)
    return fail(RSSM_EINVAL, "the tensor-core verify serves the outer-product recurrence");
  if (kind == 3) {
    if (!g.tc_ok) return fail(RSSM_EUNSUPPORTED, "this configuration has no tensor-core verify");
    rssm::TcParams tp{};
    size_t smem = 0;
    s = plan_tc(cfg, g, cfg->T_max, &tp, &smem);
    if (s != RSSM_OK) return s;
    *out = rssm_launch_plan_info{};
    out->smem_bytes = (int64_t)smem;
    out->stages[0] = tp.stages;
    out->stage_bytes[0] = rssm::kTcStageBytes;
    out->slots[0] = tp.slots;
    out->slot_bytes[0] = tp.slot_bytes;
    out->dgroups[0] = 0;
    return RSSM_OK;
  }
  if (kind == 2 && cfg->T_max > rssm::kTMax)
    return fail(RSSM_EUNSUPPORTED, "the CUDA-core verify takes at most %d drafts", rssm::kTMax);
  const LayoutKind lk = kind == 0 ? LayoutKind::kGeneral : kind == 1 ? LayoutKind::kNonFlush : LayoutKind::kVerify;
  Plan pl;
  s = plan_smem(cfg, g, &pl, lk);
  if (s != RSSM_OK) return s;
  *out = rssm_launch_plan_info{};
  out->smem_bytes = (int64_t)pl.smem;
  out->nonflush_layout = pl.p.nf_ok;
  for (int i = 0; i < 2; ++i) {
    const rssm::Layout& L = pl.p.lay[i];
    out->stages[i] = L.stages;
    out->stage_bytes[i] = L.stage_bytes;
    out->slots[i] = L.slots;
    out->slot_bytes[i] = L.slot_bytes;
    out->dgroups[i] = L.dgroups;
  }
  return RSSM_OK;
}

rssm_status rssm_create(const rssm_config* cfg, void* ckpt, void* ring, void* ptrs, void* read_copy,
                        void* stream, rssm_handle* out) {
  if (!out) return fail(RSSM_EINVAL, "out is NULL");
  *out = nullptr;
  Geom g;
  rssm_status s = derive_placed(cfg, &g);
  if (s != RSSM_OK) return s;
  if (!ckpt || !ring || !ptrs) return fail(RSSM_EINVAL, "ckpt, ring and ptrs must be non-NULL");
  if (!aligned16(ckpt) || !aligned16(ring) || !aligned16(ptrs))
    return fail(RSSM_EINVAL, "ckpt, ring and ptrs must be 16-byte aligned");
  if (cfg->read_fmt != RSSM_READ_NONE && (!read_copy || !aligned16(read_copy)))
    return fail(RSSM_EINVAL, "read_copy must be a non-NULL 16-byte aligned buffer for this read format");
  rssm_ctx* h = new (std::nothrow) rssm_ctx;
  if (!h) return fail(RSSM_EINVAL, "out of host memory");
  h->cfg = *cfg;
  h->g = g;
  h->ckpt = ckpt;  // fp32 or fp16
  h->ring = static_cast<uint8_t*>(ring);
  h->ptrs = static_cast<uint8_t*>(ptrs);
  h->copy = cfg->read_fmt != RSSM_READ_NONE ? static_cast<uint8_t*>(read_copy) : nullptr;
  h->last_T = 0;
  h->verify_kernel = 0;
  h->decode_kernel = 0;
  s = plan_smem(cfg, g, &h->dplan, LayoutKind::kNonFlush);
  if (s != RSSM_OK) {
    delete h;
    return s;
  }
  fill_common(h, &h->dplan.p);
  std::memset(&h->tmap, 0, sizeof(h->tmap));
  if (g.tc_ok && cfg->T_max > 1) {
    s = make_ckpt_tensor_map(cfg, ckpt, &h->tmap);
    if (s != RSSM_OK) {
      delete h;
      return s;
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ptrs, 0, g.ptr_bytes, st);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "cudaMemsetAsync(ptrs)");
  }
  if (h->copy) {
    Plan pl;
    s = plan_smem(cfg, g, &pl);
    if (s != RSSM_OK) {
      delete h;
      return s;
    }
    fill_common(h, &pl.p);
    const long long heads = (long long)cfg->B * cfg->H;
    e = rssm::launch_quant(pl.p, persistent_grid(heads), pl.smem, st, cfg->N, cfg->read_fmt);
    if (e != cudaSuccess) {
      delete h;
      return cuda_fail(e, "read-copy quantize launch");
    }
  }
  *out = h;
  return RSSM_OK;
}

namespace {
rssm_status decode_impl(rssm_handle h, const float* alpha, const float* beta, const void* v, const void* k,
                        const void* q, float* o, void* stream);
}

rssm_status rssm_decode_step(rssm_handle h, const float* alpha, const void* v, const void* k, const void* q,
                             float* o, void* stream) {
  if (h && h->cfg.recurrence == RSSM_GATED_DELTA)
    return fail(RSSM_EINVAL, "a delta-rule layer decodes with rssm_decode_step_delta");
  return decode_impl(h, alpha, nullptr, v, k, q, o, stream);
}

rssm_status rssm_decode_step_delta(rssm_handle h, const float* alpha, const float* beta, const void* v,
                                   const void* k, const void* q, float* o, void* stream) {
  if (h && h->cfg.recurrence != RSSM_GATED_DELTA)
    return fail(RSSM_EINVAL, "rssm_decode_step_delta needs a delta-rule layer");
  if (!beta || !aligned16(beta)) return fail(RSSM_EINVAL, "beta must be a 16-byte aligned device pointer");
  return decode_impl(h, alpha, beta, v, k, q, o, stream);
}

namespace {
rssm_status decode_impl(rssm_handle h, const float* alpha, const float* beta, const void* v, const void* k,
                        const void* q, float* o, void* stream) {
  if (!h) return fail(RSSM_EINVAL, "handle is NULL");
  if (!alpha || !v || !k || !q || !o) return fail(RSSM_EINVAL, "NULL tensor");
  if (!aligned16(alpha) || !aligned16(v) || !aligned16(k) || !aligned16(q) || !aligned16(o))
    return fail(RSSM_EINVAL, "tensors must be 16-byte aligned");
  Plan pl = h->dplan;  // planned at creation; only the inputs change per step
  pl.p.alpha = alpha; pl.p.beta = beta; pl.p.v = v; pl.p.k = k; pl.p.q = q; pl.p.o = o;
  const cudaError_t e = launch_decode_step(h, pl.p, pl.smem, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  h->last_T = 0;
  return RSSM_OK;
}
}  // namespace

namespace {
rssm_status verify_impl(rssm_handle h, int32_t T, const float* alpha, const float* beta, const void* v,
                        const void* k, const void* q, float* o, void* stream);
}

rssm_status rssm_verify(rssm_handle h, int32_t T, const float* alpha, const void* v, const void* k, const void* q,
                        float* o, void* stream) {
  if (h && h->cfg.recurrence == RSSM_GATED_DELTA)
    return fail(RSSM_EINVAL, "a delta-rule layer verifies with rssm_verify_delta");
  return verify_impl(h, T, alpha, nullptr, v, k, q, o, stream);
}

rssm_status rssm_verify_delta(rssm_handle h, int32_t T, const float* alpha, const float* beta, const void* v,
                              const void* k, const void* q, float* o, void* stream) {
  if (h && h->cfg.recurrence != RSSM_GATED_DELTA)
    return fail(RSSM_EINVAL, "rssm_verify_delta needs a delta-rule layer");
  if (!beta || !aligned16(beta)) return fail(RSSM_EINVAL, "beta must be a 16-byte aligned device pointer");
  return verify_impl(h, T, alpha, beta, v, k, q, o, stream);
}

namespace {
rssm_status verify_impl(rssm_handle h, int32_t T, const float* alpha, const float* beta, const void* v,
                        const void* k, const void* q, float* o, void* stream) {
  if (!h) return fail(RSSM_EINVAL, "handle is NULL");
  if (T < 1 || T > h->cfg.T_max) return fail(RSSM_EINVAL, "T=%d outside 1..T_max=%d", T, h->cfg.T_max);
  if (!alpha || !v || !k || !q || !o) return fail(RSSM_EINVAL, "NULL tensor");
  if (!aligned16(alpha) || !aligned16(v) || !aligned16(k) || !aligned16(q) || !aligned16(o))
    return fail(RSSM_EINVAL, "tensors must be 16-byte aligned");
  if (verify_kernel_for(h, T) == 2) {
    rssm::TcParams tp{};
    size_t smem = 0;
    const rssm_status s = plan_tc(&h->cfg, h->g, T, &tp, &smem);
    if (s != RSSM_OK) return s;
    const rssm_config& c = h->cfg;
    tp.B = c.B; tp.H = c.H; tp.G = c.G; tp.L = c.L; tp.R = h->g.R; tp.Rp = h->g.Rp; tp.HPG = c.H / c.G; tp.T = T;
    tp.alpha = alpha;
    tp.v = static_cast<const __nv_bfloat16*>(v);
    tp.k = static_cast<const __nv_bfloat16*>(k);
    tp.q = static_cast<const __nv_bfloat16*>(q);
    tp.o = o;
    tp.ring_a = reinterpret_cast<float*>(h->ring);
    tp.ring_v = reinterpret_cast<__nv_bfloat16*>(h->ring + h->g.v_off);
    tp.ring_k = reinterpret_cast<__nv_bfloat16*>(h->ring + h->g.k_off);
    tp.start = reinterpret_cast<const int32_t*>(h->ptrs);
    tp.count = reinterpret_cast<const int32_t*>(h->ptrs + h->g.off_count);
    tp.err = reinterpret_cast<uint32_t*>(h->ptrs + h->g.off_err);
    const long long items = (long long)c.B * c.H / (128 / c.P);
    const cudaError_t e = rssm::launch_verify_tc(tp, h->tmap, persistent_grid(items), smem,
                                                 static_cast<cudaStream_t>(stream), c.N, c.P);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core verify launch");
    h->last_T = T;
    return RSSM_OK;
  }
  if (T > rssm::kTMax) return fail(RSSM_EUNSUPPORTED, "T=%d > %d needs the tensor-core verify", T, rssm::kTMax);
  Plan pl;
  const rssm_status s = plan_smem(&h->cfg, h->g, &pl, LayoutKind::kVerify);
  if (s != RSSM_OK) return s;
  fill_common(h, &pl.p);
  pl.p.T = T;
  pl.p.alpha = alpha; pl.p.beta = beta; pl.p.v = v; pl.p.k = k; pl.p.q = q; pl.p.o = o;
  const long long heads = (long long)h->cfg.B * h->cfg.H;
  // verify reads the checkpoint itself, never a read copy
  const int vrf = h->g.rf == rssm::kCkF16 || h->g.rf == rssm::kDelta ? h->g.rf : (int)rssm::kRfNone;
  const cudaError_t e = rssm::launch_verify(pl.p, persistent_grid(heads), pl.smem, static_cast<cudaStream_t>(stream),
                                            h->cfg.N, h->cfg.in_dtype, vrf);
  if (e != cudaSuccess) return cuda_fail(e, "verify launch");
  h->last_T = T;
  return RSSM_OK;
}
}  // namespace

rssm_status rssm_set_verify_kernel(rssm_handle h, int32_t kind) {
  if (!h) return fail(RSSM_EINVAL, "handle is NULL");
  if (kind < 0 || kind > 2) return fail(RSSM_EINVAL, "kind=%d (0 automatic, 1 CUDA cores, 2 tensor cores)", kind);
  if (kind == 2 && !h->g.tc_ok)
    return fail(RSSM_EUNSUPPORTED, "this configuration has no tensor-core verify");
  if (kind == 2 && h->cfg.T_max < 2) return fail(RSSM_EUNSUPPORTED, "T_max = 1: no verify");
  h->verify_kernel = kind;
  return RSSM_OK;
}

rssm_status rssm_get_verify_kernel(rssm_handle h, int32_t T, int32_t* kind) {
  if (!h || !kind) return fail(RSSM_EINVAL, "NULL argument");
  if (T < 1 || T > h->cfg.T_max) return fail(RSSM_EINVAL, "T=%d outside 1..T_max=%d", T, h->cfg.T_max);
  *kind = verify_kernel_for(h, T);
  return RSSM_OK;
}

rssm_status rssm_set_decode_kernel(rssm_handle h, int32_t kind) {
  if (!h) return fail(RSSM_EINVAL, "handle is NULL");
  if (kind < 0 || kind > 2)
    return fail(RSSM_EINVAL, "kind=%d (0 automatic, 1 head kernel only, 2 warp-per-head non-flush step)", kind);
  if (kind == 2 && !nonflush_applies(h->cfg, h->g))
    return fail(RSSM_EUNSUPPORTED, "the warp-per-head non-flush step serves read copies and FP16 checkpoints");
  h->decode_kernel = kind;
  return RSSM_OK;
}

rssm_status rssm_get_decode_kernel(rssm_handle h, int32_t* kind) {
  if (!h || !kind) return fail(RSSM_EINVAL, "NULL argument");
  *kind = decode_kernel_for(h);
  return RSSM_OK;
}

rssm_status rssm_commit(rssm_handle h, const int32_t* accepted, void* stream) {
  if (!h) return fail(RSSM_EINVAL, "handle is NULL");
  if (!accepted) return fail(RSSM_EINVAL, "accepted is NULL");
  if (h->last_T < 1) return fail(RSSM_EINVAL, "commit without a pending verify");
  rssm::Params p{};
  fill_common(h, &p);
  const cudaError_t e = rssm::launch_commit(h->cfg.B, h->last_T, h->g.R, accepted, p.count, p.err,
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "commit launch");
  h->last_T = 0;
  return RSSM_OK;
}

rssm_status rssm_flush(rssm_handle h, int32_t min_count, void* stream) {
  if (!h) return fail(RSSM_EINVAL, "handle is NULL");
  if (min_count < 1) return fail(RSSM_EINVAL, "min_count=%d must be >= 1", min_count);
  Plan pl;
  const rssm_status s = plan_smem(&h->cfg, h->g, &pl);
  if (s != RSSM_OK) return s;
  fill_common(h, &pl.p);
  pl.p.min_count = min_count;
  // A one-block kernel lists the folding sequences; the persistent kernel then
  // spreads exactly their heads over the SMs.
  int32_t* flist = reinterpret_cast<int32_t*>(h->ptrs + h->g.off_flist);
  int32_t* fcount = reinterpret_cast<int32_t*>(h->ptrs + h->g.off_fcount);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = rssm::launch_flush_list(pl.p.count, h->cfg.B, h->g.R, min_count, flist, fcount, st);
  if (e != cudaSuccess) return cuda_fail(e, "flush list launch");
  pl.p.flist = flist;
  pl.p.fcount = fcount;
  e = rssm::launch_flush(pl.p, persistent_grid((long long)h->cfg.B * h->cfg.H), pl.smem, st, h->cfg.N,
                         h->cfg.in_dtype, h->g.rf);
  if (e != cudaSuccess) return cuda_fail(e, "flush launch");
  h->last_T = 0;
  return RSSM_OK;
}

rssm_status rssm_read_pointers(rssm_handle h, int32_t* start_host, int32_t* count_host, uint32_t* err_host,
                               void* stream) {
  if (!h) return fail(RSSM_EINVAL, "handle is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t nb = (size_t)h->cfg.B * 4;
  uint32_t err = 0;
  cudaError_t e = cudaSuccess;
  if (start_host && e == cudaSuccess) e = cudaMemcpyAsync(start_host, h->ptrs, nb, cudaMemcpyDeviceToHost, st);
  if (count_host && e == cudaSuccess)
    e = cudaMemcpyAsync(count_host, h->ptrs + h->g.off_count, nb, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&err, h->ptrs + h->g.off_err, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "read pointers");
  if (err_host) *err_host = err;
  if (err & rssm::kErrPlan) return fail(RSSM_EUNSUPPORTED, "a kernel refused its launch plan (error word 0x%x)", err);
  if (err & rssm::kErrTimeout) return fail(RSSM_ETIMEOUT, "a bounded wait inside a kernel expired (error word 0x%x)", err);
  if (err & (rssm::kErrCapacity | rssm::kErrAccept))
    return fail(RSSM_ECAPACITY, "ring overflow or bad accepted length (error word 0x%x)", err);
  return RSSM_OK;
}

rssm_status rssm_clear_error(rssm_handle h, void* stream) {
  if (!h) return fail(RSSM_EINVAL, "handle is NULL");
  // A launch that gave up on a wait leaves the per-sequence tickets of its
  // sequences part-counted (the aborted CTA never adds its share), so the
  // tickets are reset together with the error word.
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(h->ptrs + h->g.off_ticket, 0, (size_t)h->cfg.B * sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->ptrs + h->g.off_err, 0, 4, st);
  if (e != cudaSuccess) return cuda_fail(e, "clear error");
  return RSSM_OK;
}

rssm_status rssm_selftest_bounded_wait(uint32_t* err_word, void* stream) {
  if (!err_word) return fail(RSSM_EINVAL, "err_word is NULL");
  const cudaError_t e = rssm::launch_wait_selftest(err_word, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "bounded-wait self-test launch");
  return RSSM_OK;
}

rssm_status rssm_destroy(rssm_handle h) {
  delete h;
  return RSSM_OK;
}

namespace {
rssm_status conventional_impl(const rssm_config* cfg, float* state, const float* alpha, const float* beta,
                              const void* v, const void* k, const void* q, float* o, void* stream) {
  Geom g;
  rssm_status s = derive(cfg, &g);
  if (s != RSSM_OK) return s;
  const bool delta = cfg->recurrence == RSSM_GATED_DELTA;
  if (delta != (beta != nullptr))
    return fail(RSSM_EINVAL, delta ? "a delta-rule layer steps with rssm_conventional_step_delta"
                                   : "rssm_conventional_step_delta needs a delta-rule configuration");
  g.ck_es = 4;  // the comparison keeps an fp32 state
  g.rf = delta ? rssm::kDelta : rssm::kRfNone;
  if (!state || !alpha || !v || !k || !q || !o) return fail(RSSM_EINVAL, "NULL tensor");
  if (!aligned16(state) || !aligned16(alpha) || !aligned16(v) || !aligned16(k) || !aligned16(q) || !aligned16(o) ||
      (beta && !aligned16(beta)))
    return fail(RSSM_EINVAL, "tensors must be 16-byte aligned");
  Plan pl;
  s = plan_smem(cfg, g, &pl);
  if (s != RSSM_OK) return s;
  rssm::Params& p = pl.p;
  p.B = cfg->B; p.H = cfg->H; p.P = cfg->P; p.N = cfg->N; p.G = cfg->G; p.L = cfg->L;
  p.R = g.R; p.Rp = g.Rp; p.HPG = cfg->H / cfg->G; p.T = 1; p.min_count = 1;
  p.ckpt = state;
  p.alpha = alpha; p.beta = beta; p.v = v; p.k = k; p.q = q; p.o = o;
  const long long heads = (long long)cfg->B * cfg->H;
  const cudaError_t e =
      delta ? rssm::launch_delta(rssm::kConv, p, persistent_grid(heads), pl.smem, static_cast<cudaStream_t>(stream),
                                 cfg->N, cfg->in_dtype)
            : rssm::launch_conv(p, persistent_grid(heads), pl.smem, static_cast<cudaStream_t>(stream), cfg->N,
                                cfg->in_dtype);
  if (e != cudaSuccess) return cuda_fail(e, "conventional launch");
  return RSSM_OK;
}
}  // namespace

rssm_status rssm_conventional_step(const rssm_config* cfg, float* state, const float* alpha, const void* v,
                                   const void* k, const void* q, float* o, void* stream) {
  return conventional_impl(cfg, state, alpha, nullptr, v, k, q, o, stream);
}

rssm_status rssm_conventional_step_delta(const rssm_config* cfg, float* state, const float* alpha, const float* beta,
                                         const void* v, const void* k, const void* q, float* o, void* stream) {
  if (!beta) return fail(RSSM_EINVAL, "NULL beta");
  return conventional_impl(cfg, state, alpha, beta, v, k, q, o, stream);
}

rssm_status rssm_conventional_verify(const rssm_config* cfg, float* states, const int32_t* cur, int32_t T,
                                     const float* alpha, const void* v, const void* k, const void* q, float* o,
                                     uint32_t* err_word, void* stream) {
  Geom g;
  rssm_status s = derive(cfg, &g);
  if (s != RSSM_OK) return s;
  g.ck_es = 4;  // the comparison keeps fp32 states
  g.rf = rssm::kRfNone;
  if (cfg->recurrence != RSSM_GATED_OUTER) return fail(RSSM_EUNSUPPORTED, "the snapshot comparator is outer-product only");
  if (T < 1 || T > cfg->T_max) return fail(RSSM_EINVAL, "T=%d outside 1..T_max=%d", T, cfg->T_max);
  if (T > rssm::kTMax) return fail(RSSM_EUNSUPPORTED, "the snapshot comparator takes at most %d drafts", rssm::kTMax);
  if (!states || !cur || !alpha || !v || !k || !q || !o || !err_word) return fail(RSSM_EINVAL, "NULL pointer");
  if (!aligned16(states) || !aligned16(alpha) || !aligned16(v) || !aligned16(k) || !aligned16(q) || !aligned16(o))
    return fail(RSSM_EINVAL, "tensors must be 16-byte aligned");
  Plan pl;
  s = plan_smem(cfg, g, &pl, LayoutKind::kVerify);
  if (s != RSSM_OK) return s;
  rssm::Params& p = pl.p;
  p.B = cfg->B; p.H = cfg->H; p.P = cfg->P; p.N = cfg->N; p.G = cfg->G; p.L = cfg->L;
  p.R = g.R; p.Rp = g.Rp; p.HPG = cfg->H / cfg->G; p.T = T; p.min_count = 1;
  p.ckpt = states;
  p.cur = cur;
  p.nslot = cfg->T_max + 1;
  p.err = err_word;
  p.alpha = alpha; p.v = v; p.k = k; p.q = q; p.o = o;
  const long long heads = (long long)cfg->B * cfg->H;
  const cudaError_t e = rssm::launch_snap(p, persistent_grid(heads), pl.smem, static_cast<cudaStream_t>(stream),
                                          cfg->N, cfg->in_dtype);
  if (e != cudaSuccess) return cuda_fail(e, "conventional verify launch");
  return RSSM_OK;
}

rssm_status rssm_conventional_commit(const rssm_config* cfg, int32_t* cur, const int32_t* accepted, int32_t T,
                                     uint32_t* err_word, void* stream) {
  Geom g;
  const rssm_status s = derive(cfg, &g);
  if (s != RSSM_OK) return s;
  if (T < 1 || T > cfg->T_max) return fail(RSSM_EINVAL, "T=%d outside 1..T_max=%d", T, cfg->T_max);
  if (!cur || !accepted || !err_word) return fail(RSSM_EINVAL, "NULL pointer");
  const cudaError_t e = rssm::launch_snap_commit(cfg->B, T, cfg->T_max + 1, accepted, cur, err_word,
                                                 static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "conventional commit launch");
  return RSSM_OK;
}

rssm_status rssm_round_f16(const float* x, uint16_t* y, int64_t n, int64_t base, uint32_t epoch, uint64_t seed,
                           int32_t sr, void* stream) {
  if (n < 0 || base < 0 || (base & 3) != 0) return fail(RSSM_EINVAL, "n=%lld base=%lld", (long long)n, (long long)base);
  if (n == 0) return RSSM_OK;
  if (!x || !y) return fail(RSSM_EINVAL, "NULL pointer");
  const cudaError_t e = rssm::launch_sround_test(x, y, n, base, epoch, seed, sr, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "round launch");
  return RSSM_OK;
}

// ---------------------------------------------------------------------------
// Decode step with library-owned scratch.
//
// Some callers cannot hand the library any more device memory once decoding
// has started: engines that carve one fixed arena at start-up, code that runs
// while another component owns the device allocator, or paths that are being
// captured into a CUDA graph, where cudaMalloc is not allowed. The decode
// kernel needs one piece of scratch, the per-sequence ticket counters that
// tell the last CTA of a sequence to advance its pointers. This variant keeps
// those counters in a static device array of this file instead of the
// caller's pointer block, so it allocates nothing.
// ---------------------------------------------------------------------------
namespace {
constexpr int kStaticTicketSeqs = 8192;  // 32 KiB held by every GPU that loads the library
__device__ __align__(256) int32_t g_static_tickets[kStaticTicketSeqs];
constexpr int kMaxDevices = 64;
int32_t* g_static_ticket_addr[kMaxDevices] = {};  // device address of the array, per device
std::mutex g_static_ticket_mu;
}  // namespace

rssm_status rssm_decode_step_static_scratch(rssm_handle h, const float* alpha, const void* v, const void* k,
                                            const void* q, float* o, void* stream) {
  if (!h) return fail(RSSM_EINVAL, "handle is NULL");
  if (h->cfg.recurrence == RSSM_GATED_DELTA)
    return fail(RSSM_EUNSUPPORTED, "the static-scratch step serves the outer-product recurrence");
  if (!alpha || !v || !k || !q || !o) return fail(RSSM_EINVAL, "NULL tensor");
  if (!aligned16(alpha) || !aligned16(v) || !aligned16(k) || !aligned16(q) || !aligned16(o))
    return fail(RSSM_EINVAL, "tensors must be 16-byte aligned");
  if (h->cfg.B > kStaticTicketSeqs)
    return fail(RSSM_EUNSUPPORTED, "B=%d exceeds the %d sequences of the library-owned scratch", h->cfg.B,
                kStaticTicketSeqs);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(RSSM_EUNSUPPORTED, "device %d beyond %d", dev, kMaxDevices);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  int32_t* tickets = nullptr;
  {
    // The host-side name of the array is not a device address: ask the runtime
    // for the real one, with the device current. Outside a stream capture this
    // is done on every call, so a context that was reset and reloaded the
    // module gets its new address. Inside a capture the address found by an
    // earlier call on this device is used.
    std::lock_guard<std::mutex> lock(g_static_ticket_mu);
    if (cap == cudaStreamCaptureStatusNone) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_static_tickets);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static tickets)");
      g_static_ticket_addr[dev] = static_cast<int32_t*>(ptr);
    } else if (!g_static_ticket_addr[dev]) {
      return fail(RSSM_EINVAL, "the first static-scratch call on device %d must come before any stream capture", dev);
    }
    tickets = g_static_ticket_addr[dev];
  }
  Plan pl = h->dplan;
  pl.p.ticket = tickets;
  pl.p.alpha = alpha; pl.p.v = v; pl.p.k = k; pl.p.q = q; pl.p.o = o;
  // The array keeps the last call's contents; the tickets must start at zero.
  e = cudaMemsetAsync(tickets, 0, (size_t)h->cfg.B * sizeof(int32_t), st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static tickets)");
  e = launch_decode_step(h, pl.p, pl.smem, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch (static scratch)");
  h->last_T = 0;
  return RSSM_OK;
}

}  // extern "C"
