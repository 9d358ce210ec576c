/*
 * ulysses.h — C ABI of the single-GPU Ulysses sequence-parallel attention path.
 *
 * What the calls compute (page "Ulysses Sequence Parallelism for million-token
 * context training", section "How Ulysses sequence parallelism works"):
 *   step 1  every rank holds a contiguous chunk of S/P tokens with all heads
 *           (the "sequence layout" below);
 *   step 3  an all-to-all leaves every rank with all S positions for its subset
 *           of heads  -> ulysses_seq2head;
 *   step 4  local dense attention over the whole sequence for those heads
 *           -> ulysses_attn_fwd / ulysses_attn_bwd;
 *   step 5  a second all-to-all restores the sequence-sharded form
 *           -> ulysses_head2seq.
 * The P ranks are P partitions of one device buffer, so each all-to-all is an
 * on-device permutation.  UPipe head chunking (page "Ulysses Sequence
 * Parallelism" commentary, section on contexts beyond a million tokens:
 * process only some heads at a time) is the `head_chunk` / `stage` pair.
 *
 * Layouts (row-major, element size 2 bytes for BF16, 4 for FP32):
 *   sequence layout  X_seq [B][S][H][D]      rank r owns tokens [r*S/P, (r+1)*S/P)
 *   head layout      X_head[B][n][S][D]      n = heads of the selected stage
 *   permutation      X_head[b][h'][t][d] = X_seq[b][t][h0 + h'][d]
 *   where rank r owns heads [r*H/P, (r+1)*H/P) and stage s = r*(hq/C) + c
 *   starts at h0 = r*hq + c*C (hq = H/P, C = head_chunk).  stage = -1 selects
 *   every head of every rank (n = H, h0 = 0).
 *
 * GQA: q head h (index inside the buffer) reads kv head h / G, G = H_q/H_kv.
 * A stage owns C q heads and C/G kv heads, so C % G == 0 is required.
 *
 * Masks (AutoSP paper, section 2.A step 4, index recomputation; TRL SFTTrainer
 * packing): `cu_seqlens` holds num_docs+1 int32 GLOBAL token offsets rising
 * from 0 to S (device pointer; NULL = one document).  Row i attends key j iff
 * both lie in the same document and (causal ? j <= i : true).
 *
 * Ownership and execution: every pointer argument is a DEVICE pointer that the
 * caller allocates and frees (the library allocates no device memory).  All
 * calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 * the legacy default stream) and return a status code; the message for the
 * last failure on the calling thread is ulysses_last_error().
 *
 * Errors: ULYSSES_ERR_INVALID for shapes the method rejects (S % P != 0,
 * H % P != 0 — the pages' "num_heads >= sp_size, divisible" constraint —,
 * hq % C != 0, C % G != 0, bad stage, NULL pointers, in-place re-layout);
 * ULYSSES_ERR_UNSUPPORTED for valid but unimplemented cases (D not in {64,128},
 * B > 1 together with cu_seqlens); ULYSSES_ERR_CUDA when a launch fails;
 * ULYSSES_ERR_TIMEOUT (from ulysses_check) when a kernel gave up a bounded wait.
 * cu_seqlens contents are validated on the device: a non-monotone table or
 * one that does not end at S sets the device error word (read by
 * ulysses_check) and the attention kernels then write nothing meaningful.
 */
#ifndef ULYSSES_H
#define ULYSSES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ULYSSES_OK = 0,
  ULYSSES_ERR_INVALID = 1,
  ULYSSES_ERR_UNSUPPORTED = 2,
  ULYSSES_ERR_CUDA = 3,
  ULYSSES_ERR_TIMEOUT = 4,
  ULYSSES_ERR_BAD_SEQLENS = 5,
  ULYSSES_ERR_BOUNDS = 6
};

enum { ULYSSES_BF16 = 0, ULYSSES_FP32 = 1 };

/* Kernel selection for diagnostics: AUTO picks the tcgen05 kernels for BF16
 * with D = 128 and the fp32 SIMT kernels otherwise; SIMT forces the latter. */
enum { ULYSSES_KERNEL_AUTO = 0, ULYSSES_KERNEL_SIMT = 1 };

/* ---------------------------------------------------------------------------
 * The layer with the all-to-alls folded into the attention kernels: on one
 * device the head view of the sequence layout is a strided view, so the
 * kernels read Q/K/V/O/dO through sequence-layout TMA tensor maps and write
 * O, dQ (tensor reduce-adds), dK and dV straight into the sequence layout; no
 * head-layout copies and no re-layout launches.  Arguments and results as
 * ulysses_layer_fwd / ulysses_layer_bwd (same UPipe stage loop), restricted to
 * B == 1, bf16, S >= 128, D = 128 for the backward (64 or 128 forward), and no
 * kv-head replication; otherwise ULYSSES_ERR_UNSUPPORTED.  The backward's
 * workspace (ulysses_layer_fused_workspace bytes) holds the stage's D_i terms.
 * Results equal the unfused layer's (dQ up to the order of its fp32 additions). */
size_t ulysses_layer_fused_workspace(int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                                     int dtype);
int ulysses_layer_fwd_fused(const void* q_seq, const void* k_seq, const void* v_seq, void* o_seq, float* lse,
                            int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                            const int32_t* cu_seqlens, int num_docs, int causal, float scale, int dtype,
                            void* stream);
int ulysses_layer_bwd_fused(const void* q_seq, const void* k_seq, const void* v_seq, const void* o_seq,
                            const void* do_seq, const float* lse, float* dq_seq, float* dk_seq, float* dv_seq,
                            int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                            const int32_t* cu_seqlens, int num_docs, int causal, float scale, int dtype,
                            void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Projections with the re-layout fused in (steps 2 and 6: on one device the
 * all-to-alls around the projections become addressing).  bf16 operands, fp32
 * accumulation, bf16 results; tcgen05 GEMM.
 *
 * ulysses_qkv_proj:  [Q | K | V] = X W_qkv^T, written straight into head layout.
 *   x         [S][hidden]                       (the tokens' hidden states)
 *   w_qkv     [(H_q + 2 H_kv) D][hidden]        (row f = weights of output feature f;
 *             features ordered Q heads, K heads, V heads, D per head)
 *   qkv_head  [H_q + 2 H_kv][S][D] written: the head layout of all ranks, i.e.
 *             what ulysses_seq2head (stage -1) gives for the projected Q, K, V.
 *   Needs D in {64, 128}, hidden % 64 == 0, (H_q + 2 H_kv) D % 256 == 0.
 * ulysses_out_proj:  Y = O W_o^T, reading O straight out of head layout.
 *   o_head    [H_q][S][D]  (O_seq[s][h D + d] = o_head[h][s][d])
 *   w_o       [hidden][H_q D]
 *   y         [S][hidden] written.
 *   Needs D in {64, 128}, hidden % 256 == 0.
 * All pointers device, 16-byte aligned; asynchronous on `stream`. */
int ulysses_qkv_proj(const void* x, const void* w_qkv, void* qkv_head, int64_t S, int hidden, int H_q,
                     int H_kv, int D, void* stream);
int ulysses_out_proj(const void* o_head, const void* w_o, void* y, int64_t S, int H_q, int D, int hidden,
                     void* stream);

/* ---------------------------------------------------------------------------
 * Ring-attention variant (the scheme the pages compare Ulysses with): each
 * rank keeps its query chunk and meets the KV chunks one ring step at a time.
 *
 * ulysses_lse_merge folds one step's partial attention into a running result:
 *   first != 0:  o_acc = o_part,  lse_acc = lse_part
 *   otherwise:   LSE = log(e^{lse_acc} + e^{lse_part}),
 *                o_acc = e^{lse_acc - LSE} o_acc + e^{lse_part - LSE} o_part,
 *                lse_acc = LSE   (rows with no key in either stay empty)
 *   o_acc [rows][D] fp32 and lse_acc [rows] fp32 are read and written;
 *   o_part [rows][D] in `dtype` and lse_part [rows] fp32 are read.
 *   D must be a multiple of 32.
 * ulysses_cast_f32 writes n fp32 values as `dtype` (the merged O's output).
 * ulysses_add_f32 adds n fp32 values into dst (summing the steps' dQ/dK/dV).
 * All pointers are device pointers; asynchronous on `stream`. */
int ulysses_lse_merge(float* o_acc, float* lse_acc, const void* o_part, const float* lse_part,
                      int64_t rows, int D, int dtype, int first, void* stream);
int ulysses_cast_f32(void* dst, const float* src, int64_t n, int dtype, void* stream);
int ulysses_add_f32(float* dst, const float* src, int64_t n, void* stream);

/* Ring variant of the whole layer, run natively (B == 1).  P virtual ranks;
 * rank r keeps query chunk r (tokens [r L, (r+1) L), L = S / P) and meets KV
 * chunk c = (r - t) mod P at ring step t.  Under a causal mask the chunks
 * wholly in the future (c > r) are skipped, the diagonal step (c = r) is
 * causal and the others are full; the steps' (O, LSE) are merged with
 * ulysses_lse_merge's rule.  The backward runs every step with the merged LSE
 * and O; the steps' partial dQ, dK, dV are summed in sequence layout.
 *   q_seq/o_seq/do_seq [S][H_q][D], k_seq/v_seq [S][H_kv][D] in dtype;
 *   lse  [P][H_q][L] fp32, chunk-major (written by fwd, read by bwd);
 *   dq_seq [S][H_q][D], dk_seq/dv_seq [S][H_kv][D] fp32 (written by bwd);
 *   workspace >= ulysses_ring_workspace() bytes, 256-byte aligned (the same
 *   size serves both directions).
 * S % P must be 0; H_q % H_kv == 0; D in {64, 128}. */
size_t ulysses_ring_workspace(int64_t S, int H_q, int H_kv, int D, int P, int dtype);
int ulysses_ring_fwd(const void* q_seq, const void* k_seq, const void* v_seq, void* o_seq, float* lse,
                     int64_t S, int H_q, int H_kv, int D, int P, int causal, float scale, int dtype,
                     void* workspace, size_t ws_bytes, void* stream);
int ulysses_ring_bwd(const void* q_seq, const void* k_seq, const void* v_seq, const void* o_seq,
                     const void* do_seq, const float* lse, float* dq_seq, float* dk_seq, float* dv_seq,
                     int64_t S, int H_q, int H_kv, int D, int P, int causal, float scale, int dtype,
                     void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Padding to a multiple of the sequence-parallel degree (the pages' TRL
 * section sets pad_to_multiple_of to the SP size).
 * ulysses_pad_seq: x [B][S][H][D] -> x_pad [B][S_pad][H][D], the tokens
 *   t >= S set to zero.  S_pad >= S; H*D*elt a multiple of 16 bytes; x and
 *   x_pad must not overlap.
 * ulysses_pad_cu_seqlens: cu_pad = the real documents' offsets (cu_seqlens,
 *   num_docs + 1 entries, or [0, S] when cu_seqlens is NULL), followed by S_pad
 *   when S_pad > S: the pad tokens form a document of their own, so no real
 *   token attends to them or is attended by them.  cu_pad holds num_docs + 2
 *   int32 (num_docs = 1 without a table); the padded table has one document
 *   more than the real one when S_pad > S.  All pointers device pointers. */
int ulysses_pad_seq(const void* x, void* x_pad, int64_t S, int64_t S_pad, int B, int H, int D, int dtype,
                    void* stream);
int ulysses_pad_cu_seqlens(const int32_t* cu_seqlens, int num_docs, int32_t* cu_pad, int64_t S, int64_t S_pad,
                           void* stream);

/* Self-test of the failure path shared by every kernel: launches one CTA that
 * waits on an mbarrier nothing arrives on, bounded by limit_ns (0 < limit_ns
 * <= 2e9).  The wait gives up, the kernel records ULYSSES_ERR_TIMEOUT in the
 * device error word and exits; ulysses_check then reports it and clears the
 * word.  No GPU fault or hang is involved: the context stays usable.
 * Returns ULYSSES_ERR_INVALID for an out-of-range limit. */
int ulysses_selftest_wait_timeout(int64_t limit_ns, void* stream);

/* ---------------------------------------------------------------------------
 * All-to-all #1 (step 3): sequence layout -> head layout of one stage.
 *   x_seq   [B][S][H][D], read only.
 *   x_head  [B][n][S][D], written (n = head_chunk, or H when stage = -1).
 *   H       heads of THIS tensor (H_q for Q/O/dO, H_kv for K/V).
 *   head_chunk  heads of this tensor per stage per rank (C for Q, C/G for K/V);
 *           ignored when stage = -1.
 *   dtype   ULYSSES_BF16 or ULYSSES_FP32 (only the element size matters: the
 *           copy is bit-exact).
 * x_seq and x_head must not overlap.  Both must be 16-byte aligned.
 * ------------------------------------------------------------------------- */
int ulysses_seq2head(const void* x_seq, void* x_head, int64_t S, int B, int H, int D, int P,
                     int head_chunk, int stage, int dtype, void* stream);

/* All-to-all #2 (step 5): head layout of one stage -> its heads of the
 * sequence layout.  Arguments as ulysses_seq2head; only the selected stage's
 * heads of x_seq are written. */
int ulysses_head2seq(const void* x_head, void* x_seq, int64_t S, int B, int H, int D, int P,
                     int head_chunk, int stage, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * Batched re-layout: several tensors of one stage in one launch (for example
 * Q, K and V before a stage's forward, or dQ, dK and dV after its backward),
 * so that the small K/V tensors share the launch and the tail of the large
 * one.  Each item is one ulysses_seq2head / ulysses_head2seq call:
 *   src, dst     as x_seq / x_head (seq2head) or x_head / x_seq (head2seq)
 *   H, head_chunk, stage   as in the single calls
 *   add          head2seq with ULYSSES_FP32 only: add into dst (as
 *                ulysses_head2seq_add); must be 0 for seq2head
 * All items share S, B, D, P and dtype; at most 6 items.  No item's
 * destination may overlap any item's source (ULYSSES_ERR_INVALID).  The item
 * array is read on the host during the call. */
typedef struct {
  const void* src;
  void* dst;
  int H;
  int head_chunk;
  int stage;
  int add;
} ulysses_relayout_item;

int ulysses_seq2head_n(const ulysses_relayout_item* items, int n_items, int64_t S, int B, int D, int P,
                       int dtype, void* stream);
int ulysses_head2seq_n(const ulysses_relayout_item* items, int n_items, int64_t S, int B, int D, int P,
                       int dtype, void* stream);

/* As ulysses_head2seq, but adds the head rows into x_seq instead of writing
 * them (dtype must be ULYSSES_FP32).  Used for the gradients of a replicated
 * kv head: every rank holding a copy contributes a partial dK/dV.
 *
 * KV-head replication (the sequence-parallel degree exceeding the kv head
 * count, H < P with P % H == 0): rank r holds kv head r / (P / H), as when the
 * heads are repeated P / H times before the all-to-all.  In this mode `stage`
 * names the rank (0 <= stage < P), n = 1 and head_chunk is not used, for
 * ulysses_seq2head, ulysses_head2seq and ulysses_head2seq_add alike.  The
 * attention calls accept H_kv < P (P % H_kv == 0, H_q % P == 0); a stage's kv
 * buffer then holds that single head. */
int ulysses_head2seq_add(const void* x_head, void* x_seq, int64_t S, int B, int H, int D, int P,
                         int head_chunk, int stage, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * Local attention forward (step 4) on head-layout buffers of one stage.
 *   q_h  [B][Cq][S][D],  k_h, v_h [B][Cq/G][S][D]   (Cq = head_chunk, or H_q
 *        when stage = -1), dtype BF16 or FP32.
 *   o_h  [B][Cq][S][D] written in the input dtype: O_i = sum_j softmax(s_i)_j v_j
 *   lse  [B][Cq][S] fp32 written: natural-log logsumexp of the scaled scores.
 *   scale  score scale; <= 0 selects 1/sqrt(D).
 * All of q_h/k_h/v_h/o_h must be 16-byte aligned.
 * ------------------------------------------------------------------------- */
int ulysses_attn_fwd(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse,
                     int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk, int stage,
                     const int32_t* cu_seqlens, int num_docs, int causal, float scale, int dtype,
                     void* stream);

/* Bytes of device workspace ulysses_attn_bwd needs (the per-row
 * D_i = dO_i . O_i terms, fp32, plus alignment). */
size_t ulysses_attn_bwd_workspace(int64_t S, int B, int H_q, int H_kv, int D, int P,
                                  int head_chunk, int stage, int dtype);

/* ---------------------------------------------------------------------------
 * Local attention backward on head-layout buffers of one stage (the adjoint of
 * step 4; the adjoint of each all-to-all is the other one).
 *   inputs  q_h, k_h, v_h, o_h (forward output), do_h [B][Cq][S][D], lse (from
 *           the forward), all as in ulysses_attn_fwd.
 *   outputs dq_h [B][Cq][S][D], dk_h, dv_h [B][Cq/G][S][D], all fp32,
 *           overwritten.  dK/dV are summed over the G q heads of each kv head.
 *   workspace  device scratch of at least ulysses_attn_bwd_workspace() bytes,
 *           256-byte aligned, owned by the caller; contents need no init.
 * ------------------------------------------------------------------------- */
int ulysses_attn_bwd(const void* q_h, const void* k_h, const void* v_h, const void* o_h,
                     const void* do_h, const float* lse, float* dq_h, float* dk_h, float* dv_h,
                     void* workspace, size_t ws_bytes, int64_t S, int B, int H_q, int H_kv, int D,
                     int P, int head_chunk, int stage, const int32_t* cu_seqlens, int num_docs,
                     int causal, float scale, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * ulysses_attn_bwd without a workspace argument (no counterpart in the pages:
 * this is an interface convenience).  For callers that cannot allocate device
 * memory themselves: plugins running inside a host framework that owns every
 * device allocation, loops where a cudaMalloc (which may synchronise the
 * device) is not acceptable, or processes under a hard memory cap.
 *   Arguments, layouts, outputs and errors are those of ulysses_attn_bwd; the
 *   D_i scratch comes from a 16 MiB array built into the library (every GPU
 *   that loads the library holds it until the process exits).
 *   Limit: B * (heads in the stage) * S <= 4,194,304 rows; larger shapes are
 *   rejected with ULYSSES_ERR_UNSUPPORTED (use ulysses_attn_bwd).
 *   The library itself allocates nothing here (no cudaMalloc/cudaFree).
 *   Every call looks up the array's device address for the calling thread's
 *   current device (a host-side lookup; the first one on a device may load
 *   the library's device code, so make the first call on each device before
 *   any stream capture).
 *   All calls share the one array: calls that overlap on the GPU (different
 *   streams, or host threads without ordering) race on it and must be
 *   serialised by the caller.  The array keeps the last call's D_i values;
 *   every call rewrites the rows it uses before reading them.
 * ------------------------------------------------------------------------- */
int ulysses_attn_bwd_noalloc(const void* q_h, const void* k_h, const void* v_h, const void* o_h,
                             const void* do_h, const float* lse, float* dq_h, float* dk_h, float* dv_h,
                             int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                             int stage, const int32_t* cu_seqlens, int num_docs, int causal,
                             float scale, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * Whole layer (steps 3-5, forward or backward) with the UPipe stage loop run
 * natively: for every rank r and chunk c, seq2head of the stage's Q/K/V
 * (and O/dO), attention, head2seq of the results.  Head-layout buffers of one
 * stage live in `workspace` and are reused by the next stage, which bounds the
 * attention-side scratch by the chunk size.
 *   q_seq/o_seq/do_seq [B][S][H_q][D], k_seq/v_seq [B][S][H_kv][D] (dtype)
 *   lse  [B][H_q][S] fp32 (global head order), written by fwd, read by bwd
 *   dq_seq [B][S][H_q][D], dk_seq/dv_seq [B][S][H_kv][D], fp32, written by bwd
 *   workspace  >= ulysses_layer_workspace() bytes, 256-byte aligned.
 * ------------------------------------------------------------------------- */
size_t ulysses_layer_workspace(int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                               int dtype);

int ulysses_layer_fwd(const void* q_seq, const void* k_seq, const void* v_seq, void* o_seq,
                      float* lse, int64_t S, int B, int H_q, int H_kv, int D, int P,
                      int head_chunk, const int32_t* cu_seqlens, int num_docs, int causal,
                      float scale, int dtype, void* workspace, size_t ws_bytes, void* stream);

int ulysses_layer_bwd(const void* q_seq, const void* k_seq, const void* v_seq, const void* o_seq,
                      const void* do_seq, const float* lse, float* dq_seq, float* dk_seq,
                      float* dv_seq, int64_t S, int B, int H_q, int H_kv, int D, int P,
                      int head_chunk, const int32_t* cu_seqlens, int num_docs, int causal,
                      float scale, int dtype, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Status and diagnostics.
 * ulysses_check: synchronises `stream`, then reads and clears the device
 *   error word that kernels set when a bounded wait expires (returns
 *   ULYSSES_ERR_TIMEOUT) or when cu_seqlens is malformed
 *   (ULYSSES_ERR_BAD_SEQLENS).  Returns ULYSSES_ERR_CUDA if the stream
 *   reports a CUDA error.
 * ulysses_last_error: message of the last failure on this thread ("" if none).
 * ulysses_set_kernel: ULYSSES_KERNEL_AUTO or ULYSSES_KERNEL_SIMT (process wide).
 * ulysses_launch_count: number of kernels this library has launched so far in
 *   this process (host-side counter).
 * ulysses_checked_build: 1 for the bounds-checked build of the library
 *   (compiled with -DULYSSES_CHECKS), 0 otherwise.  In the checked build every
 *   kernel checks its global-memory indexes against the sizes of the buffers
 *   it was given; a failed check skips the access and ulysses_check returns
 *   ULYSSES_ERR_BOUNDS.  The normal build compiles the checks away.
 * ------------------------------------------------------------------------- */
int ulysses_check(void* stream);
const char* ulysses_last_error(void);
int ulysses_set_kernel(int which);
long long ulysses_launch_count(void);
int ulysses_checked_build(void);

#ifdef __cplusplus
}
#endif

#endif /* ULYSSES_H */
