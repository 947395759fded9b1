/*
 * rssm.h - C ABI of the ReplaySSM decode library (librssm.so), sm_103a.
 *
 * The library implements decoding for the gated outer-product SSM recurrence
 *     S_t = alpha_t S_{t-1} + v_t k_t^T,   o_t = S_t q_t
 * (aikraft.ru, "ReplaySSM: Революция в декодировании гибридных моделей", §01,
 * recurrence). The state of each (sequence, value head) is an FP32 checkpoint
 * plus a ring buffer of the records (alpha_j, v_j, k_j) that arrived since the
 * checkpoint (same page §03; ai.cheesepanini.fun,
 * "知识卡片：ReplaySSM——重新思考混合模型解码的状态存储", 方法/产品要点, core
 * representation). k and q are shared by the H/G consecutive value heads of a
 * group.
 *
 * Conventions for every call:
 *  - All tensors are caller-owned device memory in row-major layout with the
 *    last index contiguous. Base pointers must be 16-byte aligned. No call
 *    allocates device memory: the caller provides every buffer, and the
 *    library's one piece of device memory of its own is the static ticket
 *    array of rssm_decode_step_static_scratch. The only run-time allocation is
 *    the small host handle.
 *  - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *    void*; NULL means the legacy default stream). The one exception is
 *    rssm_read_pointers, which synchronizes the stream.
 *  - Argument errors (shapes, alignment, NULL pointers, unsupported sizes) are
 *    detected on the host before anything is enqueued. They return a status,
 *    and rssm_last_error() describes them.
 *  - Per-sequence errors found on the device (ring overflow, a bad accepted
 *    length, a wait that ran out of time) set bits in a device error word and
 *    skip the affected sequence. Other sequences proceed. rssm_read_pointers
 *    reports the word.
 *  - No C++ exception crosses this boundary. A handle is not thread safe: use
 *    one stream per handle at a time.
 *
 * A second recurrence, the gated delta rule of Gated DeltaNet layers, is
 * selected per handle by rssm_config.recurrence (see rssm_recurrence).
 *
 * Supported sizes: N in {16, 32, 64, 128}; P a multiple of 8, at most 128;
 * H a multiple of G; R = L + T_max - 1 <= 32; T_max <= 8, or T_max <= 16 for
 * configurations that the tensor-core verify serves (bf16 inputs, an FP32
 * checkpoint of the outer-product recurrence, N in {64, 128}, P in {32, 64,
 * 128} and H/G a multiple of 128/P; see rssm_set_verify_kernel). Read copies and
 * FP16 checkpoints need N in {64, 128}. A delta-rule layer needs N in
 * {64, 128}, an FP32 checkpoint, no read copy and T_max = 1. Every launch
 * keeps two checkpoint tiles, two record slots and two groups' keys and
 * queries in one CTA's shared memory; the one corner of the grid above where
 * they do not fit is f32 inputs with P = N = 128 and R >= 30 (a delta-rule
 * layer: L >= 29). rssm_workspace_size, rssm_ring_offsets,
 * rssm_read_copy_layout and rssm_create return RSSM_EUNSUPPORTED for every
 * size they cannot place.
 */
#ifndef RSSM_H_
#define RSSM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RSSM_OK = 0,
  RSSM_EINVAL = 1,        /* bad argument (shape, pointer, alignment, value) */
  RSSM_ECAPACITY = 2,     /* device error word: ring overflow or bad accepted length */
  RSSM_ECUDA = 3,         /* a CUDA runtime call failed */
  RSSM_EUNSUPPORTED = 4,  /* valid but unsupported size or format */
  RSSM_ETIMEOUT = 5       /* device error word: a bounded wait inside a kernel expired */
} rssm_status;

typedef enum { RSSM_F32 = 0, RSSM_BF16 = 1 } rssm_dtype;

/* Low-precision read copy of the checkpoint, refreshed at every flush and read
 * by non-flush decode steps. The recurrence always stays in FP32 (aikraft.ru
 * page §06; sitech.ge, "NVIDIA و Dao AI Lab يقدّمان ReplaySSM…", section
 * "الحد من خطأ التكميم"). Byte layout per (sequence, head): see
 * rssm_read_copy_layout. */
typedef enum {
  RSSM_READ_NONE = 0,
  RSSM_READ_E4M3_ROW = 1,  /* E4M3 codes, one fp32 scale per row of N */
  RSSM_READ_E2M1_B16 = 2   /* E2M1 codes (2 per byte, low nibble first), one E4M3
                              scale per 16 elements along N, one fp32 scale per row */
} rssm_read_fmt;

/* Problem sizes. B sequences, H value heads, P head dim of v and o, N state dim
 * of k and q, G groups, L flush window, T_max largest draft count of a verify
 * (1 for plain decoding). The ring has R = L + T_max - 1 slots per head.
 * in_dtype is the storage type of v, k and q (rssm_dtype); alpha, the
 * checkpoint and all outputs are fp32. read_fmt is an rssm_read_fmt. */
typedef enum {
  RSSM_CKPT_F32 = 0,    /* FP32 checkpoint (default) */
  RSSM_CKPT_F16_SR = 1, /* FP16 checkpoint, each fold stored with stochastic rounding */
  RSSM_CKPT_F16_RN = 2  /* FP16 checkpoint, stored rounded to nearest (comparison) */
} rssm_ckpt_fmt;

/* The layer's recurrence. RSSM_GATED_OUTER (default): S_t = alpha_t S_{t-1} +
 * v_t k_t^T (Mamba-2-style heads, aikraft.ru page §01). RSSM_GATED_DELTA: the
 * gated delta rule S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 * of Gated DeltaNet layers, which the pages name as using the same replay form
 * (ai.cheesepanini.fun page, 方法/产品要点). Its ring keeps, in place of v_j,
 * each record's pseudo-value w_j = beta_j (v_j - alpha_j y_j), y_j the state
 * just before record j applied to k_j. After records 0..J-1 the state is then
 * g S_ckpt + sum_j W_j w_j k_j^T (g the product of all J decays, W_j that of
 * the decays after j): the outer-product replay form with v replaced by w. The
 * step that appends record c forms y_c = P_c S_ckpt k_c + sum_{i<c} D_ic
 * (k_i^T k_c) w_i (P_c the decays before c, D_ic those strictly between i and
 * c) while it reads the checkpoint anyway. Delta layers decode with
 * rssm_decode_step_delta and verify with rssm_verify_delta; they need ckpt_fmt
 * F32, read_fmt NONE, T_max <= 4 and N in {64, 128}. */
typedef enum { RSSM_GATED_OUTER = 0, RSSM_GATED_DELTA = 1 } rssm_recurrence;

typedef struct {
  int32_t B, H, P, N, G, L, T_max;
  int32_t in_dtype;
  int32_t read_fmt;
  int32_t ckpt_fmt;   /* rssm_ckpt_fmt; FP16 needs N in {64, 128} and read_fmt NONE */
  uint64_t seed;      /* FP16 stochastic rounding: generator key */
  int32_t recurrence; /* rssm_recurrence */
} rssm_config;

typedef struct rssm_ctx* rssm_handle;

/* Byte sizes of the three caller-allocated buffers that rssm_create binds
 * (no counterpart in the pages: they hold the pages' checkpoint-plus-window
 * representation, aikraft.ru page §03, in this library's layout).
 *  ring_bytes: the record ring, made of
 *      alpha [B,H,Rp] fp32 (Rp = R rounded up to 4) at offset 0,
 *      V     [B,H,R,P] in_dtype at offset v_off (delta layers: the
 *            pseudo-values w [B,H,R,P] fp32),
 *      K     [B,G,R,N] in_dtype at offset k_off (see rssm_ring_offsets).
 *  ptr_bytes: pointer block of int32 start[B], count[B], ticket[B], one
 *      uint32 error word (256 bytes), int32 epoch[B] (flushes per sequence),
 *      then int32 flist[B] and one int32 (256 bytes), the standalone flush's
 *      list of folding sequences; each array 256-byte aligned.
 *  read_copy_bytes: B*H*head_stride for a read copy, else 0.
 * Any output pointer may be NULL. Returns RSSM_EINVAL or RSSM_EUNSUPPORTED for
 * a bad configuration. */
rssm_status rssm_workspace_size(const rssm_config* cfg, size_t* ring_bytes, size_t* ptr_bytes,
                                size_t* read_copy_bytes);

/* Byte offsets of the V and K arrays inside the ring buffer (both 256-aligned;
 * a layout query with no counterpart in the pages). */
rssm_status rssm_ring_offsets(const rssm_config* cfg, size_t* v_off, size_t* k_off);

/* Read-copy layout (the read copy of aikraft.ru page §06; the byte layout is
 * this library's). Each (sequence, head) owns head_stride bytes at
 * (b*H + h)*head_stride. Inside it:
 *   codes at 0: [P][N] bytes (E4M3) or [P][N/2] bytes (E2M1, element 2i in the low nibble);
 *   block scales at bscale_off: [P][N/16] E4M3 bytes (E2M1 only);
 *   row scales at rscale_off: [P] fp32.
 * Quantizer (both formats), with rn32 IEEE round-to-nearest-even binary32 and
 * the FP8/FP4 conversions rounding to nearest even with saturation:
 *   E4M3: a = max|x| over the row; a <= 2^-100 gives an all-zero row;
 *         inv = rn32(448/a), s = rn32(a/448), code = E4M3(rn32(x*inv)).
 *   E2M1: s_r = rn32(a/2688), d6 = rn32(6*s_r); per block of 16:
 *         sb = E4M3(rn32(max|x|_blk / d6)), d = rn32(value(sb)*s_r),
 *         r = d > 0 ? rn32(1/d) : 0, code = E2M1(rn32(x*r)).
 * Returns RSSM_EINVAL when cfg has no read copy. */
rssm_status rssm_read_copy_layout(const rssm_config* cfg, size_t* head_stride, size_t* bscale_off,
                                  size_t* rscale_off);

/* Shared-memory plan of the head kernel's launches for a configuration (no
 * counterpart in the paper: introspection of this library's launch shapes).
 * Host only; makes no CUDA call. Every launch runs one CTA per SM with the
 * layouts below:
 *   kind 0: flush and read-copy refresh (layout 0 only);
 *   kind 1: decode (layout 0 for any head, layout 1 for steps in which none of
 *           a CTA's sequences folds; nonflush_layout = 0 when only layout 0 fits);
 *   kind 2: verify on the CUDA cores (layout 0 only; needs 1 < T_max <= 8;
 *           a delta-rule configuration gives the plan of rssm_verify_delta);
 *   kind 3: verify on the tensor cores at T = T_max (needs T_max > 1 and a
 *           configuration it serves): stages[0] K-block stages of
 *           stage_bytes[0] = 16 KiB (32 checkpoint columns of 128 rows),
 *           slots[0] record slots of slot_bytes[0], dgroups[0] = 0;
 *   kind 4: the warp-per-head non-flush decode step (read copies and FP16
 *           checkpoints; RSSM_EUNSUPPORTED otherwise): dgroups[0] warps per
 *           CTA, each with stages[0] = 2 tile stages of stage_bytes[0] (the
 *           head's tile, then the ring's decays at the next 16-byte boundary)
 *           and slots[0] = 1 value stage of slot_bytes[0] (the L - 1 value
 *           rows a non-flush step can read); smem_bytes adds the CTA's abort
 *           flag and each warp's barriers and row sums.
 * Per layout: checkpoint tile stages (stage_bytes each), record slots
 * (slot_bytes each) and the number of dot-warp groups, i.e. heads in flight.
 * Both ring lengths are multiples of the number of consumers that take their
 * entries in turn (stages of dgroups, slots of max(2, dgroups)). smem_bytes is
 * the dynamic shared memory of the launch, at most 227 KiB. Returns
 * RSSM_EINVAL for a bad kind or configuration, RSSM_EUNSUPPORTED when the
 * sizes cannot be placed. */
typedef struct {
  int64_t smem_bytes;
  int32_t nonflush_layout;
  int32_t stages[2], stage_bytes[2], slots[2], slot_bytes[2], dgroups[2];
} rssm_launch_plan_info;
rssm_status rssm_launch_plan(const rssm_config* cfg, int32_t kind, rssm_launch_plan_info* out);

/* Bind a decoding context to caller memory.
 *  ckpt      [B,H,P,N] device: the initial state, fp32, or fp16 (binary16) when
 *            ckpt_fmt is an FP16 format. It becomes the checkpoint and is
 *            updated in place at every flush. An FP16 checkpoint is folded in
 *            FP32 and stored back rounded (aikraft.ru page §06: an FP16
 *            recurrent checkpoint with stochastic rounding stays close to FP32):
 *            stochastically with RSSM_CKPT_F16_SR, using Philox4x32-10 keyed by
 *            cfg->seed, counter (element index / 4, the sequence's epoch, 0);
 *            the value x rounds up to the next binary16 away from zero iff the
 *            word is below floor(frac * 2^32), frac being x's position between
 *            its binary16 neighbours; saturates to +-65504. The flush step's
 *            own output uses the unrounded FP32 state.
 *  ring      device buffer of ring_bytes; contents need not be initialised.
 *  ptrs      device buffer of ptr_bytes; zeroed here (start = count = 0).
 *  read_copy device buffer of read_copy_bytes, or NULL when read_fmt is NONE;
 *            filled here by quantizing ckpt.
 * The buffers must stay valid until rssm_destroy. Enqueues a memset and,
 * with a read copy, one kernel on the stream. *out receives the handle. */
rssm_status rssm_create(const rssm_config* cfg, void* ckpt, void* ring, void* ptrs, void* read_copy,
                        void* stream, rssm_handle* out);

/* One decode step for all B sequences (aikraft.ru page §03, "non-flush" and
 * "flush" steps). Inputs: alpha [B,H] fp32, v [B,H,P], k [B,G,N], q [B,G,N] in
 * in_dtype. Output o [B,H,P] fp32.
 * Per sequence with c committed records the step appends its record as record
 * h = c+1. If h < L it computes only the output, from the checkpoint (or
 * its read copy) and the ring (same page §05, output-only evaluation):
 *     o = gamma_{1:h} (S_ckpt q) + sum_j gamma_{j+1:h} (k_j^T q) v_j
 * and writes no state. If h >= L it folds all h records into the checkpoint,
 * writes it once (and refreshes the read copy), outputs o = S_new q, and
 * clears the buffer (start += h mod R, count = 0). A sequence with h > R sets
 * RSSM_ECAPACITY in the error word and is left untouched.
 * With an E4M3 or E2M1 read copy the step is two kernels by default
 * (rssm_set_decode_kernel; an FP16 checkpoint may choose them too): a
 * warp-per-head kernel computes the non-flush sequences' outputs and appends
 * their records, then the head kernel folds the flushing sequences and advances
 * every sequence's pointers. Other configurations launch the head kernel alone. */
rssm_status rssm_decode_step(rssm_handle h, const float* alpha, const void* v, const void* k,
                             const void* q, float* o, void* stream);

/* Choose the kernels of this handle's decode steps (library control, no
 * counterpart in the pages): 0 automatic (the default: 2 with a read copy, else
 * 1), 1 the head kernel alone, 2 the warp-per-head non-flush kernel before it.
 * RSSM_EUNSUPPORTED for 2 unless the handle has an E4M3 or E2M1 read copy or an
 * FP16 checkpoint.
 * Both give the same outputs and state up to FP32 summation order. Host only. */
rssm_status rssm_set_decode_kernel(rssm_handle h, int32_t kind);

/* The decode kernels of this handle's steps into *kind: 1 the head kernel alone,
 * 2 the warp-per-head non-flush kernel and then the head kernel. Host only. */
rssm_status rssm_get_decode_kernel(rssm_handle h, int32_t* kind);

/* Speculative verify of T <= T_max drafts (aikraft.ru page §05;
 * ai.cheesepanini.fun card, 方法/产品要点, verify formula). Inputs: alpha
 * [B,T,H] fp32, v [B,T,H,P], k [B,T,G,N], q [B,T,G,N]. Output o [B,T,H,P] fp32.
 * The T draft records are appended after the c committed ones. Pointers do
 * not move. Each draft's output uses the checkpoint once for all T queries:
 *     O = S_ckpt Q D + V (W ⊙ (K^T Q)),  D = diag(gamma_{1:c+tau}),
 *     W[j,tau] = gamma_{j+1:c+tau} for j <= c+tau, else 0.
 * Verify reads the checkpoint itself (FP32, or FP16 with an FP16 ckpt_fmt),
 * never the read copy. A sequence with c + T > R sets RSSM_ECAPACITY and is
 * skipped. T outside 1..T_max returns RSSM_EINVAL; so does a delta-rule handle
 * (it verifies with rssm_verify_delta).
 * Two kernels compute it (rssm_set_verify_kernel chooses; by default the
 * CUDA-core one up to 8 drafts and the tensor-core one above, where it applies):
 *  - CUDA cores: FP32 FMAs over the checkpoint tile, T <= 8.
 *  - Tensor cores: S_ckpt Q as kind::tf32 MMAs (tcgen05, accumulator in tensor
 *    memory) with the checkpoint split into hi (its top 11 significant bits,
 *    exact in TF32) and lo = S - hi, each multiplied by the exact bf16 queries:
 *    about 5e-7 relative error against the FP32 product, T <= 16. The value
 *    term V (W ⊙ K^T Q) stays on the CUDA cores in FP32. */
rssm_status rssm_verify(rssm_handle h, int32_t T, const float* alpha, const void* v, const void* k,
                        const void* q, float* o, void* stream);

/* Speculative verify of T <= T_max (<= 4) drafts of a gated delta-rule layer
 * (the pages' output-only verify, ai.cheesepanini.fun page, 方法/产品要点, which
 * its 待核实 list says Gated DeltaNet can use; the form is derived under
 * rssm_recurrence). rssm_verify's arguments plus beta [B,T,H] fp32, the drafts'
 * write strengths (16-byte aligned). Draft t is record c + t after the c
 * committed records. Per row, with P_t the decays before record c + t, G_t
 * those up to and including it, the committed records' pseudo-values w_i from
 * the ring and the drafts' own w'_s formed here:
 *     y_t  = P_t S_ckpt k_{c+t} + sum_{i<c} (decays after i, before c+t) (k_i^T k_{c+t}) w_i
 *            + sum_{s<t} (decays after c+s, before c+t) (k_{c+s}^T k_{c+t}) w'_s
 *     w'_t = beta_t (v_t - alpha_{c+t} y_t)
 *     o_t  = G_t S_ckpt q_t + sum_{i<c} (decays after i, to c+t) (k_i^T q_t) w_i
 *            + sum_{s<=t} (decays after c+s, to c+t) (k_{c+s}^T q_t) w'_s
 * The checkpoint is read once for the 2T vectors. Each w'_t is appended to the
 * ring (with alpha and k), and a later rssm_commit keeps the accepted prefix:
 * an accepted draft's w' depends only on the state before it, so it is the
 * pseudo-value a decode step would have written. Pointers do not move. A
 * sequence with c + T > R sets RSSM_ECAPACITY and is skipped. RSSM_EINVAL on a
 * handle of the other recurrence or for T outside 1..T_max. */
rssm_status rssm_verify_delta(rssm_handle h, int32_t T, const float* alpha, const float* beta, const void* v,
                              const void* k, const void* q, float* o, void* stream);

/* Choose the kernel of this handle's verify launches (library control, no
 * counterpart in the pages): 0 automatic (the default), 1 the CUDA cores (for
 * T <= 8; more drafts still take the tensor cores), 2 the tensor cores.
 * RSSM_EUNSUPPORTED for 2 on a configuration the tensor-core verify does not
 * serve (see the supported sizes above) or with T_max = 1. Host only. */
rssm_status rssm_set_verify_kernel(rssm_handle h, int32_t kind);

/* The kernel (1 CUDA cores, 2 tensor cores) that a verify of T drafts on this
 * handle launches, into *kind (host only; RSSM_EINVAL for T outside 1..T_max). */
rssm_status rssm_get_verify_kernel(rssm_handle h, int32_t T, int32_t* kind);

/* Commit the accepted prefix of the last verify: count[b] += accepted[b]
 * (aikraft.ru page §05; records past the pointer are ignored and later
 * overwritten). accepted [B] int32 device, each in 0..T of the last verify.
 * A value outside that range sets RSSM_ECAPACITY and leaves the sequence
 * unchanged. Nothing else moves. Returns RSSM_EINVAL when no verify is pending
 * (none since the handle was made, it was committed already, or a decode step
 * or flush came after it). */
rssm_status rssm_commit(rssm_handle h, const int32_t* accepted, void* stream);

/* Fold every sequence that holds count >= min_count records (min_count >= 1)
 * into its checkpoint, write it once, refresh the read copy, and clear its
 * buffer (aikraft.ru page §03, the flush step; the pages do not say where the
 * flush goes in speculative decoding, and this library places it after the
 * commit). Pass min_count = L after a commit. Other sequences are not touched.
 * Two launches on `stream`: a one-block kernel lists the folding sequences in
 * the pointer block, then the fold runs over exactly their heads. */
rssm_status rssm_flush(rssm_handle h, int32_t min_count, void* stream);

/* Copy start[B], count[B] (int32) and the error word to host memory,
 * synchronizing the stream first (library plumbing; no counterpart in the
 * pages). Any output may be NULL. Error word bits:
 * 1 ring overflow, 2 bad accepted length, 4 a bounded wait expired, 8 a kernel
 * refused its launch plan. Returns RSSM_OK, RSSM_EUNSUPPORTED (bit 8),
 * RSSM_ETIMEOUT (bit 4) or RSSM_ECAPACITY (bits 1|2). */
rssm_status rssm_read_pointers(rssm_handle h, int32_t* start_host, int32_t* count_host,
                               uint32_t* err_host, void* stream);

/* Clear the device error word and reset the per-sequence ticket counters of the
 * pointer block (asynchronous, two memsets on `stream`; library plumbing, no
 * counterpart in the pages). A launch whose bounded wait expired (bit 4) can
 * leave the tickets of its sequences part-counted, so that their pointers stay
 * where they were (in a two-kernel decode step, the sequences whose heads the
 * warp-per-head kernel did not finish as well); call this before the next
 * decode step or flush on the handle, with no launch of the handle in flight. */
rssm_status rssm_clear_error(rssm_handle h, void* stream);

/* Self-test of the kernels' bounded waits (no counterpart in the paper). It
 * launches one warp that waits on an mbarrier nothing completes. After the
 * wait limit (about 1 s) the warp gives up, ORs the timeout bit (4) into
 * *err_word (a device uint32 the caller owns) and returns. No trap, no
 * fault: the context stays usable. Asynchronous on `stream`. */
rssm_status rssm_selftest_bounded_wait(uint32_t* err_word, void* stream);

/* Release the host handle. Caller memory is not touched (no counterpart in the pages). */
rssm_status rssm_destroy(rssm_handle h);

/* Message of the last error on the calling thread, never NULL (no counterpart in the pages). */
const char* rssm_last_error(void);

/* Decode step that allocates nothing (no counterpart in the paper: a library
 * convenience). Same arguments, results and error behaviour as
 * rssm_decode_step. The decode kernel's only scratch, one ticket counter per
 * sequence, lives in a static device array of the library (8192 sequences,
 * 32 KiB, held by every GPU that loads the library until the process exits)
 * instead of the caller's pointer block. It is for callers that cannot provide
 * more device memory once decoding runs: a fixed arena planned at start-up, an
 * allocator owned by another component, or a stream being captured.
 *  - B above 8192 returns RSSM_EUNSUPPORTED.
 *  - Each call outside a stream capture looks up the array's device address
 *    with the device current (cudaGetSymbolAddress); a call inside a capture
 *    reuses the address an earlier call found on that device. So make the
 *    first call on a device before any stream capture (a capture without one
 *    returns RSSM_EINVAL).
 *  - Each call clears the counters it uses with cudaMemsetAsync on `stream`.
 *    It calls no cudaMalloc or cudaFree.
 *  - Every call shares the one array: calls that overlap on the GPU (other
 *    streams, other handles) race on it. Serialize them on one stream. */
rssm_status rssm_decode_step_static_scratch(rssm_handle h, const float* alpha, const void* v, const void* k,
                                            const void* q, float* o, void* stream);

/* One decode step of a gated delta-rule layer (recurrence RSSM_GATED_DELTA;
 * the replay form that ai.cheesepanini.fun page's 待核实 list says Gated
 * DeltaNet can use, derived under rssm_recurrence): rssm_decode_step plus
 * beta [B,H] fp32 (16-byte aligned), the write strength of each head's record. Non-flush steps read the checkpoint once, append the
 * record's pseudo-value and compute the output (the form above); the step
 * whose append brings the count to L folds all records and writes the
 * checkpoint once. RSSM_EINVAL on a handle of the other recurrence (and
 * rssm_decode_step refuses delta handles). */
rssm_status rssm_decode_step_delta(rssm_handle h, const float* alpha, const float* beta, const void* v,
                                   const void* k, const void* q, float* o, void* stream);

/* Comparison kernel (not part of the replay path): the conventional fused
 * read-update-write step S <- alpha S + v k^T, o = S q on a full state
 * [B,H,P,N] fp32, read and written every step (aikraft.ru page §01). cfg's
 * L, T_max and read_fmt are ignored; a delta-rule cfg is RSSM_EINVAL. */
rssm_status rssm_conventional_step(const rssm_config* cfg, float* state, const float* alpha,
                                   const void* v, const void* k, const void* q, float* o,
                                   void* stream);

/* Comparison kernel for gated delta-rule layers (the recurrence read under
 * rssm_recurrence for the Gated DeltaNet layers that aikraft.ru page's
 * introduction names): the conventional step of that recurrence, S <- alpha S (I - beta k k^T) + beta v k^T, o = S q, reading and
 * writing the full fp32 state every step. cfg->recurrence must be
 * RSSM_GATED_DELTA (and rssm_conventional_step refuses such a cfg); beta [B,H]
 * fp32, 16-byte aligned; the other arguments as for rssm_conventional_step. */
rssm_status rssm_conventional_step_delta(const rssm_config* cfg, float* state, const float* alpha,
                                         const float* beta, const void* v, const void* k, const void* q,
                                         float* o, void* stream);

/* Comparison kernels (not part of the replay path): conventional speculative
 * verify with per-draft state snapshots, the rollback scheme the replay design
 * replaces (aikraft.ru page §02 and §05; sitech.ge page, traffic and rollback
 * section). Each sequence's state lives in one of nslot = T_max + 1 slots.
 *
 * rssm_conventional_verify: for t = 0 .. T-1, S <- alpha_t S + v_t k_t^T,
 * o[b,t] = S q_t, and S is written to slot (cur[b] + 1 + t) mod nslot. The state
 * is read once and written T times; slot cur[b] is left as it was.
 *  - states: [nslot][B,H,P,N] fp32, device, caller-owned, 16-byte aligned.
 *  - cur: [B] int32 device, the slot of each sequence's state (caller
 *    initialises it, e.g. to 0). A value outside 0..nslot-1 skips the sequence
 *    and sets bit 1 in *err_word.
 *  - alpha [B,T,H] fp32; v [B,T,H,P], k and q [B,T,G,N] in cfg->in_dtype;
 *    o [B,T,H,P] fp32 (the layouts of rssm_verify).
 *  - err_word: one uint32 in device memory (bit 1 as above).
 *  - 1 <= T <= cfg->T_max, else RSSM_EINVAL. cfg->L and read_fmt are ignored;
 *    a delta-rule cfg is RSSM_EUNSUPPORTED.
 * rssm_conventional_commit: cur[b] <- (cur[b] + accepted[b]) mod nslot, which
 * selects the snapshot after the accepted drafts (accepted[b] = 0 keeps the
 * state). accepted[b] outside 0..T, or cur[b] outside 0..nslot-1, leaves the
 * sequence alone and sets bit 2 in *err_word. Both calls are asynchronous on
 * `stream`. */
rssm_status rssm_conventional_verify(const rssm_config* cfg, float* states, const int32_t* cur, int32_t T,
                                     const float* alpha, const void* v, const void* k, const void* q,
                                     float* o, uint32_t* err_word, void* stream);
rssm_status rssm_conventional_commit(const rssm_config* cfg, int32_t* cur, const int32_t* accepted, int32_t T,
                                     uint32_t* err_word, void* stream);

/* Test support (no counterpart in the pages): the FP16 checkpoint store's
 * rounding applied to x[0..n) fp32 device -> y[0..n) binary16 bits device,
 * element i rounding with word (i mod 4) of the generator call for element
 * group (base + i) / 4 at `epoch` with key `seed`; sr = 1 stochastic, 0 nearest.
 * base must be a multiple of 4 and n >= 0, else RSSM_EINVAL. Asynchronous. */
rssm_status rssm_round_f16(const float* x, uint16_t* y, int64_t n, int64_t base, uint32_t epoch, uint64_t seed,
                           int32_t sr, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RSSM_H_ */
