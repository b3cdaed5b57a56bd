/*
 * bq.h - C ABI of the GB300 DBuffer step (libbq.so).
 *
 * The library implements, for ONE GPU, the per-device hot path of veScale-FSDP
 * ("veScale-FSDP: Flexible and High-Performance FSDP at Scale"): a RaggedShard
 * layout planner that packs the tensors of one fully_shard unit into a DBuffer of
 * V equal local shards, and the step over a device's shards of that buffer - the
 * fused pre-communication pack of gradients, block-wise 8-bit Adam, block-wise FP8
 * requantisation of the updated parameters - plus Muon's Newton-Schulz
 * orthogonalisation of whole matrices.  V devices are simulated as layout only:
 * the caller chooses which local shards [dev_lo, dev_hi) one call processes.
 *
 * Conventions (every entry point):
 *   - returns int: BQ_OK (0) or a negative BQ_E* code; nothing aborts, traps or
 *     throws across the ABI; bq_last_error() gives a message for the calling
 *     thread's last failure.
 *   - the CALLER owns every device buffer and stream; the library owns only the
 *     host objects it returns (bq_layout, bq_shard) and frees them on *_free.
 *   - device work is asynchronous on the given stream (a cudaStream_t passed as
 *     bq_stream_t; NULL = legacy default stream); launch failures come back as
 *     BQ_ECUDA.  Kernels do no device-wide synchronisation and no allocation.
 *   - device pointers must be 16-byte aligned (BQ_EALIGN otherwise).
 *   - element buffers of a shard range cover the global DBuffer offsets
 *     [dev_lo*S, dev_hi*S): element at global offset x lives at index x - dev_lo*S.
 *     Scale buffers cover the slots of devices [dev_lo, dev_hi): slot z lives at
 *     index z - slot_base(dev_lo) (slot bases are in the exported table).
 */
#ifndef BQ_H
#define BQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bq_stream_t; /* == cudaStream_t */

enum {
  BQ_OK = 0,
  BQ_EINVAL = -1,      /* bad argument or descriptor */
  BQ_EINFEASIBLE = -2, /* no layout satisfies the constraints */
  BQ_EALIGN = -3,      /* misaligned pointer, stride or layout offset */
  BQ_ECUDA = -4,       /* CUDA runtime / launch error */
  BQ_ENOSPC = -5,      /* caller buffer or workspace too small */
  BQ_EDEVICE = -6      /* no usable device / unsupported architecture */
};

/* Adam block geometry of a tensor. */
enum {
  BQ_ADAM_FLAT256 = 0, /* 256 consecutive elements (last block may be short) */
  BQ_ADAM_TILE128 = 1, /* 128x128 tiles of the 2-D view (1-D tensors: 128 elements) */
  BQ_OPT_MUON = 2,     /* 2-D tensor updated by Muon (bq_muon_*): no Adam blocks, no FP8 */
  BQ_ADAM_TILE32 = 3   /* 32x32 tiles of the 2-D view (1-D: 32 elements), 32-row granularity, no FP8 */
};

/* One RaggedShard tensor: row-major 2-D view rows x cols (1-D: rows = 1), atomic
 * block g in elements (a device boundary may only fall at a multiple of g from
 * the tensor start), Adam block geometry, and whether it has 128x128 FP8 tiles. */
typedef struct {
  int64_t rows, cols, g;
  int32_t adam_kind;
  int32_t fp8;
} bq_tensor_desc;

/* Planner options.  alpha: collective alignment of S (elements); start_align:
 * alignment of every tensor start (elements; the step kernels need a multiple of
 * 8); order: the tensors' placement order in the buffer (the walkthrough's paper
 * section 5 names three tried): 0 = as given (the default the pages use), 1 =
 * atomic block size g, largest first, 2 = shape (rows, then columns), largest
 * first; ties keep the given order.  BQ_EINVAL for any other value. */
typedef struct {
  int64_t alpha;
  int64_t start_align;
  int32_t order;
  int32_t reserved;
} bq_plan_opts;

typedef struct bq_layout bq_layout; /* planned DBuffer layout (host object) */
typedef struct bq_shard bq_shard;   /* layout + device tables for [dev_lo, dev_hi) */

typedef struct {
  int64_t V, S, N;
  int64_t n_intervals, n_mslots, n_fslots;
  int64_t total_elems;   /* sum of tensor sizes */
  int64_t padding_elems; /* V*S - total_elems */
  int64_t export_len;    /* int64 entries written by bq_layout_export */
  int64_t case3_prefix;  /* length of the winning Case-3 prefix */
} bq_layout_info;

/* fp32 Adam hyper-parameters of one step; omb1 = 1-b1, omb2 = 1-b2 and the
 * reciprocal bias corrections rbc1 = 1/(1-b1^t), rbc2 = 1/(1-b2^t).  Fill it
 * with bq_adam_hparams. */
typedef struct {
  float lr, b1, b2, eps, omb1, omb2, rbc1, rbc2;
} bq_adam_hp;

/* One Newton-Schulz problem: bf16 row-major x (rows x cols, row pitch ld_x
 * elements) -> bf16 y (same shape, pitch ld_y).  x and y may alias. */
typedef struct {
  const void* x;
  void* y;
  int64_t rows, cols, ld_x, ld_y;
} bq_mat;

const char* bq_strerror(int code);
const char* bq_last_error(void);
int bq_version(void);

/* ------------------------------------------------------------------ planner
 * bq_plan - lay out n tensors over V devices.
 * Defined by: veScale-FSDP planning problem and heuristic (feynmanwiki
 * walkthrough, paper section 5: equal local shards of size S, contiguous
 * non-overlapping tensors with padding only between them, device boundaries only
 * at multiples of g from a tensor's start, minimise S; default tensor order, DP
 * feasibility per S, binary search over multiples of an LCM alignment, Case-3
 * prefixes of the size-sorted tensors).
 * t: host array of n descriptors (read only).  On success *out receives a new
 * layout owned by the caller (free with bq_layout_free).  Errors: BQ_EINVAL for
 * a bad descriptor (g not a multiple of the Adam block / FP8 band it must keep
 * whole, or a 2-D FP8 / tile tensor with cols % 8 != 0), BQ_EINFEASIBLE never in
 * practice (S = sum n + N*start_align always fits). */
int bq_plan(const bq_tensor_desc* t, int n, int V, const bq_plan_opts* opts, bq_layout** out);
void bq_layout_free(bq_layout* layout);
int bq_layout_query(const bq_layout* layout, bq_layout_info* info);

/* bq_layout_export - flat int64 table (host buffer buf of n entries):
 *   header    [magic 0x4251, version 1, V, S, N, NI, n_mslots, n_fslots]
 *   tensors   N  x [start, numel, rows, cols, g, adam_kind, fp8]
 *   intervals NI x [dev, tensor, t_off, len, local_off, mslot, fslot]
 *   devices   (V+1) x [first interval, mslot base, fslot base]
 * Intervals are in device order, tensors in buffer order within a device; slots
 * are numbered per device in interval order, inside an interval in tensor-flat
 * order (256-element blocks) or band-major / column-tile-minor order (128x128
 * tiles, 1-D: 128-element tiles).  fslot = -1 for tensors without FP8.
 * BQ_ENOSPC if n < export_len. */
int bq_layout_export(const bq_layout* layout, int64_t* buf, size_t n);

/* ------------------------------------------------------------------ device tables
 * bq_layout_upload - derive the work tables of local shards [dev_lo, dev_hi) and
 * copy them into the caller's device workspace dev_ws (ws_bytes, query with
 * bq_layout_upload_bytes) on stream.  *out receives a host bq_shard (free with
 * bq_shard_free) that the step calls take; the workspace must stay alive and
 * unmodified while the shard is used (besides the tables it holds the shard's
 * device error word, read by bq_shard_check, so every shard needs its own
 * workspace).  BQ_EALIGN if an interval's local offset is not a multiple of 8
 * elements (plan with start_align % 8 == 0). */
int bq_layout_upload_bytes(const bq_layout* layout, int dev_lo, int dev_hi, size_t* bytes);
int bq_layout_upload(const bq_layout* layout, int dev_lo, int dev_hi, void* dev_ws, size_t ws_bytes,
                     bq_stream_t stream, bq_shard** out);
void bq_shard_free(bq_shard* shard);

/* ------------------------------------------------------------------ groups of shard ranges
 * A group steps the local shards of several layouts at once - e.g. every
 * fully_shard unit of a model's slice on one rank - with one launch per kernel
 * family instead of one per unit.  Defined by: DBuffer's group-level fused
 * operations (feynmanwiki walkthrough, paper section 5, DBuffer paragraphs:
 * one fused launch over the whole buffer instead of per-tensor launches),
 * carried from one DBuffer to a list of them.
 * Member u = local shards [dev_lo, dev_hi) of `layout`.  Its place in the
 * group's buffers (bq_group_place):
 *   element buffers (gradient DBuffer, master, m, v, FP8 staging): the member's
 *     element x (as in a single upload of that range) lives at elem_base + x;
 *     elem_base is a multiple of 256 and the gaps between members are padding
 *     (zeroed by bq_pack, untouched by the other calls);
 *   Adam / FP8 scale buffers: the member's slot z at mslot_base / fslot_base + z;
 *   per-tensor pointer and lr arrays (bq_pack, bq_muon_*): the member's tensor i
 *     at entry tensor_base + i.
 * info->elems, mslots, fslots, tensors: the group's buffer lengths.
 * bq_group_upload builds and checks every member's tables, concatenates them
 * with those offsets into the caller's device workspace (ws_bytes from
 * bq_group_upload_bytes; one synchronised copy) and returns a bq_shard that
 * bq_pack, bq_step_adam8, bq_quant_fp8, bq_dequant_fp8, bq_muon_momentum,
 * bq_muon_apply and bq_shard_check accept like any other (its "range" is the
 * whole group).  The layouts may be freed after the upload (the tables are
 * copied).  The same layout may appear in several members (identical units).
 * Errors: BQ_EINVAL (n < 1, a NULL layout, a bad range, or a group above 2^40
 * elements / 2^31 slots or tensors), BQ_EALIGN (as bq_layout_upload),
 * BQ_ENOSPC (workspace too small), BQ_ECUDA. */
typedef struct {
  const bq_layout* layout;
  int32_t dev_lo, dev_hi;
} bq_member;

typedef struct {
  int64_t elem_base, mslot_base, fslot_base, tensor_base;
} bq_member_place;

typedef struct {
  int64_t elems, mslots, fslots, tensors;
} bq_group_info;

int bq_group_place(const bq_member* members, int n, bq_member_place* place, bq_group_info* info);
int bq_group_upload_bytes(const bq_member* members, int n, size_t* bytes);
int bq_group_upload(const bq_member* members, int n, void* dev_ws, size_t ws_bytes, bq_stream_t stream,
                    bq_shard** out);

/* bq_shard_check - synchronise `stream` and read the shard's device error word
 * (kept in its workspace): the 2-D Adam kernel's producer / consumer waits give
 * up after about a second, record where (1, 2: the copy producer; 3: a compute
 * warp) and let the kernel exit; 8 records a 128x128-tile region larger than a
 * tile (a corrupted table: its excess is not updated).  BQ_OK if the word is
 * clear; otherwise the word is cleared and BQ_ECUDA returned (also on a CUDA
 * error).
 * Defined by no passage of the pages: a failure-reporting aid of this library. */
int bq_shard_check(const bq_shard* shard, bq_stream_t stream);

/* bq_wait_selftest - exercise the failure path of the kernels' bounded waits:
 * one GPU thread waits on an mbarrier that nothing arrives at, through the same
 * wait loop as the step kernels but with a limit of about a millisecond, gives
 * up, writes 7 to the device int *dev_status (1 would mean the wait completed)
 * and returns; the context stays usable.  Asynchronous on stream.  No passage of
 * the pages defines it: a failure-detection aid of this library. */
int bq_wait_selftest(int* dev_status, bq_stream_t stream);

/* ------------------------------------------------------------------ step
 * bq_pack - group-level fused pre-communication add / scale / zero / copy.
 * Defined by: DBuffer's fused pre-communication ops (bud-325 summary, Key claims
 * and Method; feynmanwiki walkthrough, paper section 5, DBuffer paragraphs).
 * For every element j of every interval (dev, i, t_off, len, local_off) in range:
 *   y = f32(grad_i[t_off + j]) * scale; if accumulate: y = f32(dbuf[pos]) + y;
 *   dbuf[pos] = bf16_rne(y)  (pos = (dev-dev_lo)*S + local_off + j)
 * and every padding element of the range is set to +0.
 * grad_ptrs: DEVICE array of N device pointers, grad_ptrs[i] = address of element
 * 0 of tensor i (bf16); only the owned elements are read, so a pointer may be a
 * virtual base below an allocation that holds just the owned range.
 * dbuf_grad: bf16, (dev_hi-dev_lo)*S elements. */
int bq_pack(const bq_shard* shard, const void* const* grad_ptrs, void* dbuf_grad, float scale, int accumulate,
            bq_stream_t stream);

/* bq_step_adam8 - block-wise 8-bit Adam on the local shards, optionally fused with
 * the FP8 requantisation of the updated parameters.
 * Defined by: 8-bit Adam with per-block quantised state kept device-local by
 * RaggedShard granularity (bud-325 summary, Key claims; feynmanwiki walkthrough,
 * paper section 6.3) and block-wise FP8 (DeepSeek-V3 style, bud-325 TL;DR).
 * Per element, each an IEEE fp32 op rounded to nearest; fma = one rounding:
 *   g=f32(grad); m=qm*sm; v=qv*sv; m'=fma(b1,m,omb1*g); v'=fma(b2,v,omb2*(g*g));
 *   u=(m'*rbc1)/(sqrt(v'*rbc2)+eps); p'=fma(-lr,u,p)
 * per Adam block: sm'=max|m'|/127, qm'=clamp(rint(m'*(127/max|m'|)),-127,127)
 *   with the product rounded once, directly to an integer; sv'=max v'/255,
 *   qv'=clamp(rint(v'*(255/max v')),0,255) likewise (each reciprocal is one fp32
 *   division per block; if it overflows, rint(fp32(m'/sm')) resp. v'/sv');
 *   a block whose scale is 0 gets zero codes.
 * per FP8 tile (if fp8_out != NULL): s=max|p'|/448, code=e4m3_rne_satfinite(
 *   fp32(p'*(448/max|p'|))) (p'/s if the reciprocal overflows); scale 0 -> +-0.
 * grad: bf16 packed buffer; master fp32, m int8, v uint8, fp8_out uint8 - all
 * (dev_hi-dev_lo)*S elements, updated in place (padding untouched); m_scale,
 * v_scale: fp32 per Adam slot; fp8_scale: fp32 per FP8 slot (a scale buffer may
 * be NULL when the range has no slot of its kind).  hp: host pointer.
 * Resources: the 2-D kernels take 64 or 128 tensor-memory columns per CTA for
 * their lifetime (at most 384 of an SM's 512); a CTA whose columns are held by
 * a co-resident kernel (e.g. a tensor-core GEMM on another stream) waits until
 * that kernel's CTA exits.  The first call on a set of (grad, master, m, v)
 * buffers writes tensor maps of those buffers into the shard's workspace,
 * ordered on `stream`, and later calls on the same buffers read through them; a
 * call made while `stream` is being captured into a graph reads the same data
 * block by block instead, so a replay never depends on the maps.  A shard
 * serves one stream at a time. */
int bq_step_adam8(const bq_shard* shard, const void* grad, float* master, int8_t* m, uint8_t* v, float* m_scale,
                  float* v_scale, const bq_adam_hp* hp, uint8_t* fp8_out, float* fp8_scale, bq_stream_t stream);

/* bq_adam_hparams - the hyper-parameters of step t (t >= 1) of bq_step_adam8.
 * Defined by: Adam's bias-corrected moment estimates (the 8-bit Adam of the
 * feynmanwiki walkthrough, paper section 6.3, keeps Adam's update and quantises
 * only the state).  lr, b1, b2, eps are taken as given (double) and rounded once
 * to fp32; omb1 = 1-b1, omb2 = 1-b2, rbc1 = 1/(1-b1^t), rbc2 = 1/(1-b2^t) are
 * evaluated in fp64 (b^t by the C library's pow) and rounded once to fp32.
 * Host only; out: caller's struct.  BQ_EINVAL: out NULL, t < 1, b1 or b2 outside
 * [0, 1), or a non-finite / negative lr or eps. */
int bq_adam_hparams(double lr, double b1, double b2, double eps, int64_t t, bq_adam_hp* out);

/* bq_quant_fp8 - standalone FP8 requantisation of master into fp8_out / fp8_scale
 * (same tile rule as above). */
int bq_quant_fp8(const bq_shard* shard, const float* master, uint8_t* fp8_out, float* fp8_scale,
                 bq_stream_t stream);

/* ------------------------------------------------------------------ Muon
 * bq_muon_ns - Newton-Schulz orthogonalisation of `batch` whole matrices.
 * Defined by: Muon's matrix-sign preconditioner run at one root on the complete
 * 2-D matrix (feynmanwiki walkthrough, paper section 6.3).  Per matrix (a tall
 * one is iterated as its transpose and written back transposed):
 *   X = x / (||x||_F + eps); repeat steps: A = X X^T; B = b A + c A A; X = a X + B X
 * on tcgen05 tensor cores: bf16 operands, fp32 accumulation, bf16 storage of
 * X, A, B between products, fp32 Frobenius norm.
 * mats: host array; ws: device workspace of ws_bytes, 256-byte aligned (bf16
 * scratch for X, A, B, fp32 partial norms and an error word).
 * bq_muon_ns_workspace gives the size that lets the matrices of a batch run
 * concurrently: each gets its own region and the library forks them onto its
 * own side streams (three per device, created on the first such call, never
 * destroyed) from `stream` and joins them back into it, so the idle SMs of one
 * matrix's products run another's (an ordinary fork and join of events, which
 * also works inside a stream capture; one batch at a time enqueues on a
 * device's side streams).  Any ws_bytes of at least the largest single
 * matrix's need also works: the matrices then run one after another on
 * `stream` and reuse one region.  The results are the same either way.
 * Resources: every CTA of the products holds all 512 tensor-memory columns of
 * its SM while it runs (the B X product runs on clusters of two CTAs that hold
 * the columns of both their SMs); a CTA whose columns are held by a co-resident
 * kernel waits until that kernel's CTA exits.
 * Errors: BQ_EINVAL (bad descriptor, rows or cols above 2^20), BQ_EALIGN,
 * BQ_ENOSPC, BQ_EDEVICE (driver entry point for tensor maps unavailable). */
int bq_muon_ns_workspace(int batch, const bq_mat* mats, size_t* bytes);
int bq_muon_ns(int batch, const bq_mat* mats, int steps, float a, float b, float c, float eps, void* ws,
               size_t ws_bytes, bq_stream_t stream);

/* bq_muon_ns_check - synchronise `stream` and read the workspace's device error
 * word: every wait inside the tensor-core kernels gives up after about two
 * seconds, records where, and lets the kernel exit cleanly.  The word is
 * cleared once at the start of each bq_muon_ns call and keeps the first site
 * recorded for any matrix of that call's batch.  BQ_OK if no wait timed out
 * during the last bq_muon_ns on this workspace, BQ_ECUDA otherwise (or on a
 * CUDA error).  ws == NULL reads the static scratch of the current device
 * instead, i.e. the word of the last bq_muon_ns_noalloc call on it. */
int bq_muon_ns_check(const void* ws, size_t ws_bytes, bq_stream_t stream);

/* bq_dequant_fp8 - the bf16 view of the FP8 buffer after the AllGather.
 * Defined by: block-wise FP8 training in the DeepSeek-V3 style (bud-325 summary,
 * TL;DR and Key claims): the gathered E4M3 parameters serve the compute as code
 * x tile scale.  Reading: each code decoded exactly, times its tile's fp32 scale
 * in fp32 (one rounding), rounded to bf16 (nearest even).
 * fp8 / fp8_scale: the staging buffer and tile scales of local shards
 * [dev_lo, dev_hi) as bq_step_adam8 / bq_quant_fp8 write them; out_bf16: bf16
 * buffer with the DBuffer layout of the range; only elements of FP8 tiles are
 * written.  Asynchronous on stream.  BQ_EALIGN: fp8 or out_bf16 not 16-byte
 * aligned, fp8_scale not 4-byte aligned. */
int bq_dequant_fp8(const bq_shard* shard, const uint8_t* fp8, const float* fp8_scale, void* out_bf16,
                   bq_stream_t stream);

/* ------------------------------------------------------------------ the Muon step around Newton-Schulz
 * Defined by: the Muon experiment of the walkthrough (paper section 6.3).  For
 * every 2-D weight the optimizer takes its gradient, applies the momentum update,
 * keeps the original placement, picks a load-balanced root where the full matrix
 * materialises, runs Newton-Schulz there and sends the result back to be applied
 * to the weight.  The pages give no formula; the readings implemented:
 *   momentum  M <- fma(mu, M, G), fp32, one rounding (heavy-ball momentum)
 *   NS input  bf16(M) (nearest even), the whole matrix in row-major order
 *   apply     W <- fma(-lr, O, W), fp32, O the bf16 Newton-Schulz output
 * Tensors planned with adam_kind = BQ_OPT_MUON take this path; bq_step_adam8
 * leaves them untouched.  On one GPU with every shard of the range resident the
 * root's gather and the send-back are the device-local copies these calls make;
 * across GPUs they would be exchanges between ranks (not built here). */

/* bq_muon_roots - root device (0..V-1) of every Muon tensor, -1 for the others,
 * into roots[0..N).  Rule (a reading; the pages name none): longest-processing-
 * time greedy on the nominal Newton-Schulz step cost 4 m^2 n + 2 m^3 (m, n the
 * smaller and larger dimension): largest first (ties: lower tensor index), each
 * to the device with the least cost assigned so far (ties: lower device index).
 * Host only.  BQ_ENOSPC if n < N. */
int bq_muon_roots(const bq_layout* layout, int32_t* roots, size_t n);

/* bq_muon_momentum - momentum update of every Muon tensor piece in the shard's
 * range: grad is the bf16 gradient DBuffer of local shards [dev_lo, dev_hi)
 * (after pack), mom the fp32 momentum buffer with the same layout (updated in
 * place; elements of other tensors and padding untouched).  gather_ptrs is a
 * DEVICE array of N pointers: entry i is the bf16 row-major rows x cols buffer of
 * Muon tensor i that receives bf16(M) at each owned tensor offset (the root's
 * Newton-Schulz input), or NULL to skip tensor i; entries of non-Muon tensors are
 * never read.  Asynchronous on stream.  BQ_EALIGN: grad, mom not 16-byte or
 * gather_ptrs not 8-byte aligned. */
int bq_muon_momentum(const bq_shard* shard, const void* grad, float* mom, float mu, void* const* gather_ptrs,
                     bq_stream_t stream);

/* bq_muon_apply - W <- fma(-lr[i], O_i, W) over every Muon tensor piece in the
 * shard's range: master is the fp32 master DBuffer of the range (updated in
 * place), update_ptrs a DEVICE array of N pointers to the bf16 row-major
 * Newton-Schulz outputs O_i (NULL: skip tensor i), lr a DEVICE array of N fp32
 * step sizes (any shape factor folded in by the caller).  Asynchronous on
 * stream.  BQ_EALIGN: master not 16-byte, update_ptrs not 8-byte, lr not 4-byte
 * aligned. */
int bq_muon_apply(const bq_shard* shard, float* master, const void* const* update_ptrs, const float* lr,
                  bq_stream_t stream);

/* bq_muon_ns_noalloc - bq_muon_ns for callers that cannot allocate device memory
 * when the step runs (a runtime that reserves all GPU memory up front and
 * forbids later cudaMalloc, a plug-in whose host framework owns the allocator,
 * a code path that must not allocate for latency reasons).  The paper has no
 * counterpart: this is an interface convenience of this library.
 * The caller passes inputs and outputs as for bq_muon_ns; the scratch is a fixed
 * 32 MiB array inside the library's device image (every GPU that loads the
 * library holds it until the process exits), so nothing is allocated and no
 * workspace is passed.  The matrices run one after another on `stream` (no side
 * streams), reusing the scratch; a batch with a matrix needing more than 32 MiB
 * is rejected with BQ_ENOSPC before any work is queued (for example, a 1024 x
 * 4096 matrix fits; a 2048 x 2048 one does not).
 * The first call on each device looks up the scratch array's device address
 * with that device current; make that first call before any stream capture.
 * All calls share the one array and each call overwrites it: calls that can
 * overlap on the GPU (different streams without ordering between them) race,
 * so order them.  The device error word lives in the shared scratch too: read
 * it with bq_muon_ns_check(NULL, 0, stream) after the call (same device
 * current).  The address looked up on the first call is kept for the process;
 * after a cudaDeviceReset it may be stale. */
int bq_muon_ns_noalloc(int batch, const bq_mat* mats, int steps, float a, float b, float c, float eps,
                       bq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BQ_H */
