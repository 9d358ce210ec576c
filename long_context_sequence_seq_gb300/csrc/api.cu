// C ABI: argument validation, kernel dispatch and the UPipe stage driver.
//
// Validation follows the constraints the pages state for Ulysses: the
// sequence must split evenly over the ranks (pad_to_multiple_of == sp_size in
// the TRL SFTTrainer section and the "sequence divisibility" best practice),
// and every rank must own whole heads ("num_heads >= sp_size" in the Ulysses
// vs Ring table; heads divisible by the SP size in the DeepSpeed-Ulysses
// commentary).  UPipe chunks must hold whole kv heads under GQA.
#include <atomic>
#include <cstdarg>
#include <mutex>
#include <cstdio>
#include <cstring>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace ulysses {

// One NVTX range per UPipe stage of the layer drivers, so a profiler that
// records NVTX (ncu --nvtx) can attribute kernels to stages; without an
// attached tool the push and pop are no-ops.
struct StageRange {
  StageRange(const char* what, int s) {
    char name[48];
    snprintf(name, sizeof(name), "ulysses %s stage %d", what, s);
    nvtxRangePushA(name);
  }
  ~StageRange() { nvtxRangePop(); }
  StageRange(const StageRange&) = delete;
  StageRange& operator=(const StageRange&) = delete;
};

static thread_local char g_msg[512];
static std::atomic<long long> g_launches{0};
static std::atomic<int> g_kernel_choice{ULYSSES_KERNEL_AUTO};

void count_launch(int n) { g_launches.fetch_add(n); }

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(ULYSSES_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return ULYSSES_OK;
}

int opt_in_smem(PerDeviceOnce<>& once, const void* func, int bytes, const char* what) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(ULYSSES_ERR_CUDA, "%s: cudaGetDevice: %s", what, cudaGetErrorString(e));
  const int rc = once.run(dev, [&]() -> int {
    cudaError_t r = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (r != cudaSuccess)
      return set_error(ULYSSES_ERR_CUDA, "%s: shared-memory opt-in of %d bytes on device %d: %s", what, bytes, dev,
                       cudaGetErrorString(r));
    return ULYSSES_OK;
  }, -1);
  if (rc == -1) return set_error(ULYSSES_ERR_UNSUPPORTED, "%s: device %d beyond the library's 64-device table", what, dev);
  return rc;
}

// Error-word readers, one per translation unit that raises device errors.
unsigned read_error_api(cudaStream_t st);
unsigned read_error_attn_tc_fwd(cudaStream_t st);
unsigned read_error_attn_tc_bwd(cudaStream_t st);
unsigned read_error_proj_gemm(cudaStream_t st);
ULYSSES_ERROR_READER(read_error_api)

// cu_seqlens check: cu[0] == 0, cu[nd] == S, non-decreasing.
__global__ void check_seqlens_kernel(const int32_t* __restrict__ cu, int nd, int64_t S) {
  for (int i = threadIdx.x + blockIdx.x * blockDim.x; i <= nd; i += blockDim.x * gridDim.x) {
    int32_t c = cu[i];
    bool bad = (i == 0 && c != 0) || (i == nd && (int64_t)c != S) || (i > 0 && c < cu[i - 1]);
    if (bad) raise_error(kErrSeqlens);
  }
}

int launch_check_seqlens(const int32_t* cu, int nd, int64_t S, cudaStream_t st) {
  check_seqlens_kernel<<<1, 256, 0, st>>>(cu, nd, S);
  count_launch();
  return check_launch("check_seqlens");
}

int launch_tc_fwd(const AttnArgs& a, cudaStream_t st);  // attn_tc_fwd.cu
int launch_tc_bwd(const AttnArgs& a, cudaStream_t st);  // attn_tc_bwd.cu
bool tc_fwd_supported(const AttnArgs& a);
bool tc_bwd_supported(const AttnArgs& a);

}  // namespace ulysses

using namespace ulysses;

namespace {

int elt_size(int dtype) { return dtype == ULYSSES_BF16 ? 2 : (dtype == ULYSSES_FP32 ? 4 : 0); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Heads of a stage: n heads starting at h0.
int stage_span(int H, int P, int C, int stage, int* n, int* h0) {
  if (P > 0 && H > 0 && H < P && P % H == 0) {
    // kv-head replication (H_kv < P): rank r holds head r / (P / H); `stage`
    // names the rank and head_chunk is not used
    if (stage < 0 || stage >= P)
      return set_error(ULYSSES_ERR_INVALID, "with H=%d < P=%d, stage names a rank in [0,%d), got %d", H, P, P, stage);
    *n = 1;
    *h0 = stage / (P / H);
    return ULYSSES_OK;
  }
  if (P <= 0 || H <= 0 || H % P)
    return set_error(ULYSSES_ERR_INVALID, "H=%d must be a positive multiple of P=%d, or divide P", H, P);
  if (stage == -1) { *n = H; *h0 = 0; return ULYSSES_OK; }
  const int hq = H / P;
  if (C <= 0 || hq % C)
    return set_error(ULYSSES_ERR_INVALID, "head_chunk=%d must divide H/P=%d", C, hq);
  const int per_rank = hq / C;
  if (stage < 0 || stage >= P * per_rank)
    return set_error(ULYSSES_ERR_INVALID, "stage=%d out of range [0,%d)", stage, P * per_rank);
  *n = C;
  *h0 = (stage / per_rank) * hq + (stage % per_rank) * C;
  return ULYSSES_OK;
}

// Validates one re-layout tensor and fills its job (heads moved, first head).
int relayout_job(bool to_head, const void* src, void* dst, int64_t S, int B, int H, int D, int P, int C,
                 int stage, int dtype, bool add, RelayoutJob* job) {
  const int elt = elt_size(dtype);
  if (!elt) return set_error(ULYSSES_ERR_INVALID, "unknown dtype %d", dtype);
  if (add && (to_head || dtype != ULYSSES_FP32))
    return set_error(ULYSSES_ERR_UNSUPPORTED, "accumulating re-layout is head->seq, fp32 only");
  if (S < 0 || B <= 0 || D <= 0) return set_error(ULYSSES_ERR_INVALID, "bad sizes S=%lld B=%d D=%d", (long long)S, B, D);
  if (P <= 0 || S % P) return set_error(ULYSSES_ERR_INVALID, "S=%lld not divisible by P=%d", (long long)S, P);
  if ((D * elt) % 16)
    return set_error(ULYSSES_ERR_UNSUPPORTED, "D*elt=%d must be a multiple of 16 bytes", D * elt);
  int n = 0, h0 = 0;
  int rc = stage_span(H, P, C, stage, &n, &h0);
  if (rc) return rc;
  *job = RelayoutJob{src, dst, H, n, h0, add ? 1 : 0, 0};
  if (S == 0) return ULYSSES_OK;
  if (!src || !dst) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (!aligned16(src) || !aligned16(dst)) return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  return ULYSSES_OK;
}

// Byte ranges of a job's source and destination.
void job_ranges(bool to_head, const RelayoutJob& j, int64_t S, int B, int D, int elt, const char** a, size_t* la,
                const char** b, size_t* lb) {
  const size_t seq_bytes = (size_t)B * S * j.H * D * elt, head_bytes = (size_t)B * j.n * S * D * elt;
  *a = (const char*)j.src; *la = to_head ? seq_bytes : head_bytes;
  *b = (const char*)j.dst; *lb = to_head ? head_bytes : seq_bytes;
}

bool overlap(const char* a, size_t la, const char* b, size_t lb) { return a < b + lb && b < a + la; }

// A batch of re-layouts of one launch: every item's destination must be
// disjoint from every item's source (the launch has no order among them).
int relayout_n(bool to_head, const ulysses_relayout_item* items, int n_items, int64_t S, int B, int D, int P,
               int dtype, void* stream) {
  if (n_items < 0 || n_items > kMaxRelayoutJobs)
    return set_error(ULYSSES_ERR_INVALID, "n_items=%d must be in [0, %d]", n_items, kMaxRelayoutJobs);
  if (n_items > 0 && !items) return set_error(ULYSSES_ERR_INVALID, "NULL item list");
  RelayoutBatch bt{};
  for (int i = 0; i < n_items; ++i) {
    const ulysses_relayout_item& it = items[i];
    int rc = relayout_job(to_head, it.src, it.dst, S, B, it.H, D, P, it.head_chunk, it.stage, dtype,
                          it.add != 0, &bt.job[i]);
    if (rc) return rc;
  }
  if (S == 0 || n_items == 0) return ULYSSES_OK;
  const int elt = elt_size(dtype);
  for (int i = 0; i < n_items; ++i)
    for (int k = 0; k < n_items; ++k) {
      const char *ai, *bi, *ak, *bk;
      size_t lai, lbi, lak, lbk;
      job_ranges(to_head, bt.job[i], S, B, D, elt, &ai, &lai, &bi, &lbi);
      job_ranges(to_head, bt.job[k], S, B, D, elt, &ak, &lak, &bk, &lbk);
      if (overlap(bi, lbi, ak, lak))
        return set_error(ULYSSES_ERR_INVALID, "re-layout cannot run in place (destination %d overlaps source %d)", i, k);
    }
  bt.njobs = n_items;
  bt.S = S;
  bt.B = B;
  bt.V = D * elt / 16;
  return launch_relayout_batch(to_head, bt, (cudaStream_t)stream);
}

int relayout(bool to_head, const void* src, void* dst, int64_t S, int B, int H, int D, int P,
             int C, int stage, int dtype, void* stream, bool add = false) {
  ulysses_relayout_item it{src, dst, H, C, stage, add ? 1 : 0};
  return relayout_n(to_head, &it, 1, S, B, D, P, dtype, stream);
}

// Shape validation shared by attention calls; fills a (without pointers).
int attn_shape(AttnArgs& a, int64_t S, int B, int H_q, int H_kv, int D, int P, int C, int stage,
               const int32_t* cu, int nd, int causal, float scale, int dtype) {
  memset(&a, 0, sizeof(a));
  if (!elt_size(dtype)) return set_error(ULYSSES_ERR_INVALID, "unknown dtype %d", dtype);
  if (S < 0 || B <= 0) return set_error(ULYSSES_ERR_INVALID, "bad sizes S=%lld B=%d", (long long)S, B);
  if (H_q <= 0 || H_kv <= 0 || H_q % H_kv)
    return set_error(ULYSSES_ERR_INVALID, "H_q=%d must be a multiple of H_kv=%d", H_q, H_kv);
  if (P <= 0 || S % P) return set_error(ULYSSES_ERR_INVALID, "S=%lld not divisible by P=%d", (long long)S, P);
  const bool rep_kv = H_kv < P;   // kv-head replication: rank r uses kv head r / (P / H_kv)
  if (H_q % P || (rep_kv ? P % H_kv : H_kv % P))
    return set_error(ULYSSES_ERR_INVALID,
                     "heads (H_q=%d, H_kv=%d) must divide evenly over P=%d (or H_kv divide P)", H_q, H_kv, P);
  int nq = 0, h0 = 0;
  int rc = stage_span(H_q, P, C, stage, &nq, &h0);
  if (rc) return rc;
  // a stage's kv buffer holds whole kv heads; with replication it holds the
  // one kv head all of the rank's q heads use
  const int G = rep_kv ? nq : H_q / H_kv;
  if (nq % G) return set_error(ULYSSES_ERR_INVALID, "head_chunk=%d must hold whole kv heads (G=%d)", nq, G);
  if (D != 64 && D != 128) return set_error(ULYSSES_ERR_UNSUPPORTED, "head dim %d not in {64,128}", D);
  if (cu && B > 1) return set_error(ULYSSES_ERR_UNSUPPORTED, "cu_seqlens needs B == 1");
  if (cu && nd <= 0) return set_error(ULYSSES_ERR_INVALID, "num_docs must be >= 1 with cu_seqlens");
  if (S > ((int64_t)1 << 31) - 1) return set_error(ULYSSES_ERR_UNSUPPORTED, "S must fit int32 token offsets");
  a.S = S; a.nq = nq; a.n_q = B * nq; a.G = G; a.D = D;
  a.lse_bstride = (int64_t)nq * S;
  a.cu = cu; a.nd = cu ? nd : 0; a.causal = causal ? 1 : 0;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  a.dtype = dtype;
  return ULYSSES_OK;
}

bool use_tc_fwd(const AttnArgs& a) {
  return g_kernel_choice.load() == ULYSSES_KERNEL_AUTO && tc_fwd_supported(a);
}
bool use_tc_bwd(const AttnArgs& a) {
  return g_kernel_choice.load() == ULYSSES_KERNEL_AUTO && tc_bwd_supported(a);
}

int run_fwd(AttnArgs& a, cudaStream_t st) {
  if (a.S == 0) return ULYSSES_OK;
  if (a.cu) { int rc = launch_check_seqlens(a.cu, a.nd, a.S, st); if (rc) return rc; }
  return use_tc_fwd(a) ? launch_tc_fwd(a, st) : launch_simt_fwd(a, st);
}

int run_bwd(AttnArgs& a, cudaStream_t st) {
  if (a.S == 0) return ULYSSES_OK;
  if (a.cu) { int rc = launch_check_seqlens(a.cu, a.nd, a.S, st); if (rc) return rc; }
  return use_tc_bwd(a) ? launch_tc_bwd(a, st) : launch_simt_bwd(a, st);
}

size_t delta_bytes(int64_t S, int B, int nq) { return align256((size_t)B * nq * S * sizeof(float)); }

// Stage argument of a layer stage's K/V re-layout: the q stage itself, or,
// with kv-head replication (H_kv < P), the rank the stage belongs to.
int kv_stage(int H_kv, int P, int s, int stages) {
  return H_kv < P ? s / (stages / P) : s;
}
// With replication: is stage s the first of the stages sharing its kv head?
// (rank r uses kv head r / (P / H_kv); stages run in rank order)
bool kv_first_stage(int H_kv, int P, int s, int stages) {
  const int per_rank = stages / P, r = s / per_rank, R = P / H_kv;
  return r % R == 0 && s % per_rank == 0;
}

struct LayerWs {
  char *qh, *kh, *vh, *oh, *doh; float *dqh, *dkh, *dvh, *delta; size_t total;
};

LayerWs layer_ws(char* base, int64_t S, int B, int Cq, int Ckv, int D, int elt) {
  LayerWs w{};
  size_t off = 0;
  auto take = [&](size_t bytes) { char* p = base ? base + off : nullptr; off += align256(bytes); return p; };
  const size_t q_b = (size_t)B * Cq * S * D, kv_b = (size_t)B * Ckv * S * D;
  w.qh = take(q_b * elt); w.kh = take(kv_b * elt); w.vh = take(kv_b * elt);
  w.oh = take(q_b * elt); w.doh = take(q_b * elt);
  w.dqh = (float*)take(q_b * 4); w.dkh = (float*)take(kv_b * 4); w.dvh = (float*)take(kv_b * 4);
  w.delta = (float*)take((size_t)B * Cq * S * 4);
  w.total = off;
  return w;
}

// ---------------------------------------------------------------------------
// Scratch for ulysses_attn_bwd_noalloc: the backward's per-row D_i terms live
// in this file-scope device array instead of a caller-provided workspace.
// Every device that loads the library holds it (16 MiB) until the process
// exits.  In host code the symbol is only a stand-in, so its device address is
// looked up with the calling device current, on every call: the lookup is a
// host-side table read once the library's device code is loaded, and it stays
// right if the device's context is reset between calls.
constexpr size_t kNoAllocDeltaFloats = size_t(1) << 22;   // 4,194,304 rows
static __device__ __align__(256) float g_noalloc_delta[kNoAllocDeltaFloats];

int noalloc_scratch(float** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_delta);
  if (e != cudaSuccess || p == nullptr)
    return set_error(ULYSSES_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  *out = static_cast<float*>(p);
  return ULYSSES_OK;
}

}  // namespace

extern "C" {

// One CTA waits on an mbarrier that nothing arrives on: the bounded wait used
// by every kernel gives up after limit_ns, records ULYSSES_ERR_TIMEOUT in the
// device error word and the kernel exits.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  tc::mbar_wait(&bar, 0, &abort_flag, limit_ns);
}

int ulysses_selftest_wait_timeout(int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > (int64_t)kWaitLimitNs)
    return set_error(ULYSSES_ERR_INVALID, "limit_ns must be in (0, %llu]", (unsigned long long)kWaitLimitNs);
  selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_ns);
  count_launch();
  return check_launch("selftest_wait");
}

// ---------------------------------------------------------------------------
// The layer with the all-to-alls folded into the attention kernels'
// addressing (sequence-layout tensor maps and stores): no head-layout copies.
static int fused_check(AttnArgs& a, int B, int H_kv, int P, bool bwd) {
  if (B != 1) return set_error(ULYSSES_ERR_UNSUPPORTED, "fused layer: B must be 1");
  if (H_kv < P) return set_error(ULYSSES_ERR_UNSUPPORTED, "fused layer: kv-head replication not supported");
  if (a.dtype != ULYSSES_BF16 || (bwd && a.D != 128) || a.S < 128)
    return set_error(ULYSSES_ERR_UNSUPPORTED, "fused layer: bf16, S >= 128%s", bwd ? ", D = 128" : "");
  return ULYSSES_OK;
}

size_t ulysses_layer_fused_workspace(int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                                     int dtype) {
  AttnArgs a;
  if (attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, 0, nullptr, 0, 1, 0.f, dtype)) return 0;
  return align256(delta_bytes(S, B, a.nq));
}

int ulysses_layer_fwd_fused(const void* q_seq, const void* k_seq, const void* v_seq, void* o_seq, float* lse,
                            int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                            const int32_t* cu_seqlens, int num_docs, int causal, float scale, int dtype,
                            void* stream) {
  AttnArgs a;
  int rc = attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, 0, cu_seqlens, num_docs, causal, scale, dtype);
  if (rc) return rc;
  if (S == 0) return ULYSSES_OK;
  if ((rc = fused_check(a, B, H_kv, P, false))) return rc;
  if (!q_seq || !k_seq || !v_seq || !o_seq || !lse) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (!aligned16(q_seq) || !aligned16(k_seq) || !aligned16(v_seq) || !aligned16(o_seq))
    return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const int C = a.nq, stages = P * (H_q / P / C);
  const size_t e = (size_t)D * 2;   // bytes per head of a row
  if (cu_seqlens) { rc = launch_check_seqlens(cu_seqlens, num_docs, S, st); if (rc) return rc; }
  for (int s = 0; s < stages; ++s) {
    StageRange range("fused fwd", s);
    int n = 0, h0 = 0;
    stage_span(H_q, P, C, s, &n, &h0);
    AttnArgs sa = a;
    sa.seq = 1; sa.hq_tot = H_q; sa.hkv_tot = H_kv;
    sa.q = (const char*)q_seq + h0 * e;
    sa.k = (const char*)k_seq + (h0 / a.G) * e;
    sa.v = (const char*)v_seq + (h0 / a.G) * e;
    sa.o_out = (char*)o_seq + h0 * e;
    sa.lse = lse + (size_t)h0 * S;
    sa.lse_bstride = (int64_t)H_q * S;
    if ((rc = launch_tc_fwd(sa, st))) return rc;
  }
  return ULYSSES_OK;
}

int ulysses_layer_bwd_fused(const void* q_seq, const void* k_seq, const void* v_seq, const void* o_seq,
                            const void* do_seq, const float* lse, float* dq_seq, float* dk_seq, float* dv_seq,
                            int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                            const int32_t* cu_seqlens, int num_docs, int causal, float scale, int dtype,
                            void* workspace, size_t ws_bytes, void* stream) {
  AttnArgs a;
  int rc = attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, 0, cu_seqlens, num_docs, causal, scale, dtype);
  if (rc) return rc;
  if (S == 0) return ULYSSES_OK;
  if ((rc = fused_check(a, B, H_kv, P, true))) return rc;
  if (!q_seq || !k_seq || !v_seq || !o_seq || !do_seq || !lse || !dq_seq || !dk_seq || !dv_seq || !workspace)
    return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (!aligned16(q_seq) || !aligned16(k_seq) || !aligned16(v_seq) || !aligned16(o_seq) || !aligned16(do_seq) ||
      !aligned16(dq_seq) || !aligned16(dk_seq) || !aligned16(dv_seq))
    return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  if (ws_bytes < delta_bytes(S, B, a.nq))
    return set_error(ULYSSES_ERR_INVALID, "workspace too small: %zu < %zu", ws_bytes, delta_bytes(S, B, a.nq));
  cudaStream_t st = (cudaStream_t)stream;
  const int C = a.nq, stages = P * (H_q / P / C);
  const size_t e = (size_t)D * 2, ef = (size_t)D;   // bf16 bytes / fp32 elements per head of a row
  if (cu_seqlens) { rc = launch_check_seqlens(cu_seqlens, num_docs, S, st); if (rc) return rc; }
  for (int s = 0; s < stages; ++s) {
    StageRange range("fused bwd", s);
    int n = 0, h0 = 0;
    stage_span(H_q, P, C, s, &n, &h0);
    const int kh0 = h0 / a.G;
    AttnArgs sa = a;
    sa.seq = 1; sa.hq_tot = H_q; sa.hkv_tot = H_kv;
    sa.q = (const char*)q_seq + h0 * e;
    sa.k = (const char*)k_seq + kh0 * e;
    sa.v = (const char*)v_seq + kh0 * e;
    sa.o = (const char*)o_seq + h0 * e;
    sa.dO = (const char*)do_seq + h0 * e;
    sa.lse_in = lse + (size_t)h0 * S;
    sa.lse_bstride = (int64_t)H_q * S;
    sa.dq = dq_seq + h0 * ef;
    sa.dk = dk_seq + kh0 * ef;
    sa.dv = dv_seq + kh0 * ef;
    sa.delta = (float*)workspace;
    if ((rc = launch_tc_bwd(sa, st))) return rc;
  }
  return ULYSSES_OK;
}

int ulysses_qkv_proj(const void* x, const void* w_qkv, void* qkv_head, int64_t S, int hidden, int H_q,
                     int H_kv, int D, void* stream) {
  if (S < 0 || hidden <= 0 || H_q <= 0 || H_kv <= 0) return set_error(ULYSSES_ERR_INVALID, "bad sizes");
  if (D != 64 && D != 128) return set_error(ULYSSES_ERR_UNSUPPORTED, "head dim %d not in {64,128}", D);
  if (hidden % 64) return set_error(ULYSSES_ERR_UNSUPPORTED, "hidden=%d must be a multiple of 64", hidden);
  if (((H_q + 2 * H_kv) * D) % 256)
    return set_error(ULYSSES_ERR_UNSUPPORTED, "(H_q + 2 H_kv) D = %d must be a multiple of 256", (H_q + 2 * H_kv) * D);
  if (S == 0) return ULYSSES_OK;
  if (!x || !w_qkv || !qkv_head) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(qkv_head))
    return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  return launch_qkv_proj(x, w_qkv, qkv_head, S, hidden, H_q + 2 * H_kv, D, (cudaStream_t)stream);
}

int ulysses_out_proj(const void* o_head, const void* w_o, void* y, int64_t S, int H_q, int D, int hidden,
                     void* stream) {
  if (S < 0 || hidden <= 0 || H_q <= 0) return set_error(ULYSSES_ERR_INVALID, "bad sizes");
  if (D != 64 && D != 128) return set_error(ULYSSES_ERR_UNSUPPORTED, "head dim %d not in {64,128}", D);
  if (hidden % 256) return set_error(ULYSSES_ERR_UNSUPPORTED, "hidden=%d must be a multiple of 256", hidden);
  if (S == 0) return ULYSSES_OK;
  if (!o_head || !w_o || !y) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (!aligned16(o_head) || !aligned16(w_o) || !aligned16(y))
    return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  return launch_out_proj(o_head, w_o, y, S, H_q, D, hidden, (cudaStream_t)stream);
}

int ulysses_lse_merge(float* o_acc, float* lse_acc, const void* o_part, const float* lse_part,
                      int64_t rows, int D, int dtype, int first, void* stream) {
  if (!elt_size(dtype)) return set_error(ULYSSES_ERR_INVALID, "unknown dtype %d", dtype);
  if (rows < 0 || D <= 0 || D % 32) return set_error(ULYSSES_ERR_INVALID, "bad sizes rows=%lld D=%d", (long long)rows, D);
  if (rows == 0) return ULYSSES_OK;
  if (!o_acc || !lse_acc || !o_part || !lse_part) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  return launch_lse_merge(o_acc, lse_acc, o_part, lse_part, rows, D, dtype, first ? 1 : 0, (cudaStream_t)stream);
}

int ulysses_cast_f32(void* dst, const float* src, int64_t n, int dtype, void* stream) {
  if (!elt_size(dtype)) return set_error(ULYSSES_ERR_INVALID, "unknown dtype %d", dtype);
  if (n < 0) return set_error(ULYSSES_ERR_INVALID, "bad size %lld", (long long)n);
  if (n == 0) return ULYSSES_OK;
  if (!dst || !src) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  return launch_cast_f32(dst, src, n, dtype, (cudaStream_t)stream);
}

int ulysses_add_f32(float* dst, const float* src, int64_t n, void* stream) {
  if (n < 0) return set_error(ULYSSES_ERR_INVALID, "bad size %lld", (long long)n);
  if (n == 0) return ULYSSES_OK;
  if (!dst || !src) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  return launch_add_f32(dst, src, n, (cudaStream_t)stream);
}

int ulysses_seq2head(const void* x_seq, void* x_head, int64_t S, int B, int H, int D, int P,
                     int head_chunk, int stage, int dtype, void* stream) {
  return relayout(true, x_seq, x_head, S, B, H, D, P, head_chunk, stage, dtype, stream);
}

int ulysses_head2seq(const void* x_head, void* x_seq, int64_t S, int B, int H, int D, int P,
                     int head_chunk, int stage, int dtype, void* stream) {
  return relayout(false, x_head, x_seq, S, B, H, D, P, head_chunk, stage, dtype, stream);
}

int ulysses_seq2head_n(const ulysses_relayout_item* items, int n_items, int64_t S, int B, int D, int P,
                       int dtype, void* stream) {
  for (int i = 0; i < n_items && items; ++i)
    if (items[i].add) return set_error(ULYSSES_ERR_UNSUPPORTED, "accumulating re-layout is head->seq, fp32 only");
  return relayout_n(true, items, n_items, S, B, D, P, dtype, stream);
}

int ulysses_head2seq_n(const ulysses_relayout_item* items, int n_items, int64_t S, int B, int D, int P,
                       int dtype, void* stream) {
  return relayout_n(false, items, n_items, S, B, D, P, dtype, stream);
}

int ulysses_head2seq_add(const void* x_head, void* x_seq, int64_t S, int B, int H, int D, int P,
                         int head_chunk, int stage, int dtype, void* stream) {
  return relayout(false, x_head, x_seq, S, B, H, D, P, head_chunk, stage, dtype, stream, true);
}

int ulysses_attn_fwd(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse,
                     int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk, int stage,
                     const int32_t* cu_seqlens, int num_docs, int causal, float scale, int dtype,
                     void* stream) {
  AttnArgs a;
  int rc = attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, stage, cu_seqlens, num_docs, causal,
                      scale, dtype);
  if (rc) return rc;
  if (S == 0) return ULYSSES_OK;
  if (!q_h || !k_h || !v_h || !o_h || !lse) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (!aligned16(q_h) || !aligned16(k_h) || !aligned16(v_h) || !aligned16(o_h))
    return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  a.q = q_h; a.k = k_h; a.v = v_h; a.o_out = o_h; a.lse = lse;
  return run_fwd(a, (cudaStream_t)stream);
}

size_t ulysses_attn_bwd_workspace(int64_t S, int B, int H_q, int H_kv, int D, int P,
                                  int head_chunk, int stage, int dtype) {
  AttnArgs a;
  if (attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, stage, nullptr, 0, 1, 0.f, dtype)) return 0;
  return delta_bytes(S, B, a.nq);
}

int ulysses_attn_bwd(const void* q_h, const void* k_h, const void* v_h, const void* o_h,
                     const void* do_h, const float* lse, float* dq_h, float* dk_h, float* dv_h,
                     void* workspace, size_t ws_bytes, int64_t S, int B, int H_q, int H_kv, int D,
                     int P, int head_chunk, int stage, const int32_t* cu_seqlens, int num_docs,
                     int causal, float scale, int dtype, void* stream) {
  AttnArgs a;
  int rc = attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, stage, cu_seqlens, num_docs, causal,
                      scale, dtype);
  if (rc) return rc;
  if (S == 0) return ULYSSES_OK;
  if (!q_h || !k_h || !v_h || !o_h || !do_h || !lse || !dq_h || !dk_h || !dv_h || !workspace)
    return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (ws_bytes < delta_bytes(S, B, a.nq))
    return set_error(ULYSSES_ERR_INVALID, "workspace too small: %zu < %zu", ws_bytes, delta_bytes(S, B, a.nq));
  if (!aligned16(q_h) || !aligned16(k_h) || !aligned16(v_h) || !aligned16(o_h) || !aligned16(do_h) ||
      !aligned16(dq_h) || !aligned16(dk_h) || !aligned16(dv_h) || !aligned16(workspace))
    return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  a.q = q_h; a.k = k_h; a.v = v_h; a.o = o_h; a.dO = do_h; a.lse_in = lse;
  a.dq = dq_h; a.dk = dk_h; a.dv = dv_h; a.delta = (float*)workspace;
  return run_bwd(a, (cudaStream_t)stream);
}

int ulysses_attn_bwd_noalloc(const void* q_h, const void* k_h, const void* v_h, const void* o_h,
                             const void* do_h, const float* lse, float* dq_h, float* dk_h, float* dv_h,
                             int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                             int stage, const int32_t* cu_seqlens, int num_docs, int causal,
                             float scale, int dtype, void* stream) {
  AttnArgs a;
  int rc = attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, stage, cu_seqlens, num_docs, causal,
                      scale, dtype);
  if (rc) return rc;
  if (S == 0) return ULYSSES_OK;
  const size_t rows = (size_t)B * a.nq * S;
  if (rows > kNoAllocDeltaFloats)
    return set_error(ULYSSES_ERR_UNSUPPORTED,
                     "attn_bwd_noalloc: B*heads*S = %zu rows exceeds the built-in scratch of %zu rows; "
                     "use ulysses_attn_bwd with a workspace",
                     rows, kNoAllocDeltaFloats);
  if (!q_h || !k_h || !v_h || !o_h || !do_h || !lse || !dq_h || !dk_h || !dv_h)
    return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (!aligned16(q_h) || !aligned16(k_h) || !aligned16(v_h) || !aligned16(o_h) || !aligned16(do_h) ||
      !aligned16(dq_h) || !aligned16(dk_h) || !aligned16(dv_h))
    return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  float* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  a.q = q_h; a.k = k_h; a.v = v_h; a.o = o_h; a.dO = do_h; a.lse_in = lse;
  a.dq = dq_h; a.dk = dk_h; a.dv = dv_h; a.delta = scratch;
  return run_bwd(a, (cudaStream_t)stream);
}

size_t ulysses_layer_workspace(int64_t S, int B, int H_q, int H_kv, int D, int P, int head_chunk,
                               int dtype) {
  AttnArgs a;
  if (attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, 0, nullptr, 0, 1, 0.f, dtype)) return 0;
  return layer_ws(nullptr, S, B, a.nq, a.nq / a.G, D, elt_size(dtype)).total;
}

int ulysses_layer_fwd(const void* q_seq, const void* k_seq, const void* v_seq, void* o_seq,
                      float* lse, int64_t S, int B, int H_q, int H_kv, int D, int P,
                      int head_chunk, const int32_t* cu_seqlens, int num_docs, int causal,
                      float scale, int dtype, void* workspace, size_t ws_bytes, void* stream) {
  AttnArgs a;
  int rc = attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, 0, cu_seqlens, num_docs, causal,
                      scale, dtype);
  if (rc) return rc;
  if (S == 0) return ULYSSES_OK;
  if (!q_seq || !k_seq || !v_seq || !o_seq || !lse || !workspace) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  const int elt = elt_size(dtype), C = a.nq, Ckv = C / a.G;
  LayerWs w = layer_ws((char*)workspace, S, B, C, Ckv, D, elt);
  if (ws_bytes < w.total) return set_error(ULYSSES_ERR_INVALID, "workspace too small: %zu < %zu", ws_bytes, w.total);
  if (((uintptr_t)workspace & 255u) != 0) return set_error(ULYSSES_ERR_INVALID, "workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const int stages = P * (H_q / P / C);
  if (cu_seqlens) { rc = launch_check_seqlens(cu_seqlens, num_docs, S, st); if (rc) return rc; }
  for (int s = 0; s < stages; ++s) {
    StageRange range("fwd", s);
    int n = 0, h0 = 0;
    stage_span(H_q, P, C, s, &n, &h0);
    const int ks = kv_stage(H_kv, P, s, stages);
    const ulysses_relayout_item gather[3] = {{q_seq, w.qh, H_q, C, s, 0},
                                             {k_seq, w.kh, H_kv, Ckv, ks, 0},
                                             {v_seq, w.vh, H_kv, Ckv, ks, 0}};
    if ((rc = relayout_n(true, gather, 3, S, B, D, P, dtype, stream))) return rc;
    AttnArgs sa = a;
    sa.q = w.qh; sa.k = w.kh; sa.v = w.vh; sa.o_out = w.oh;
    sa.lse = lse + (size_t)h0 * S;
    sa.lse_bstride = (int64_t)H_q * S;
    rc = use_tc_fwd(sa) ? launch_tc_fwd(sa, st) : launch_simt_fwd(sa, st);
    if (rc) return rc;
    if ((rc = relayout(false, w.oh, o_seq, S, B, H_q, D, P, C, s, dtype, stream))) return rc;
  }
  return ULYSSES_OK;
}

int ulysses_layer_bwd(const void* q_seq, const void* k_seq, const void* v_seq, const void* o_seq,
                      const void* do_seq, const float* lse, float* dq_seq, float* dk_seq,
                      float* dv_seq, int64_t S, int B, int H_q, int H_kv, int D, int P,
                      int head_chunk, const int32_t* cu_seqlens, int num_docs, int causal,
                      float scale, int dtype, void* workspace, size_t ws_bytes, void* stream) {
  AttnArgs a;
  int rc = attn_shape(a, S, B, H_q, H_kv, D, P, head_chunk, 0, cu_seqlens, num_docs, causal,
                      scale, dtype);
  if (rc) return rc;
  if (S == 0) return ULYSSES_OK;
  if (!q_seq || !k_seq || !v_seq || !o_seq || !do_seq || !lse || !dq_seq || !dk_seq || !dv_seq || !workspace)
    return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  const int elt = elt_size(dtype), C = a.nq, Ckv = C / a.G;
  LayerWs w = layer_ws((char*)workspace, S, B, C, Ckv, D, elt);
  if (ws_bytes < w.total) return set_error(ULYSSES_ERR_INVALID, "workspace too small: %zu < %zu", ws_bytes, w.total);
  if (((uintptr_t)workspace & 255u) != 0) return set_error(ULYSSES_ERR_INVALID, "workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const int stages = P * (H_q / P / C);
  if (cu_seqlens) { rc = launch_check_seqlens(cu_seqlens, num_docs, S, st); if (rc) return rc; }
  for (int s = 0; s < stages; ++s) {
    StageRange range("bwd", s);
    int n = 0, h0 = 0;
    stage_span(H_q, P, C, s, &n, &h0);
    const int ks = kv_stage(H_kv, P, s, stages);
    const ulysses_relayout_item gather[5] = {{q_seq, w.qh, H_q, C, s, 0},
                                             {k_seq, w.kh, H_kv, Ckv, ks, 0},
                                             {v_seq, w.vh, H_kv, Ckv, ks, 0},
                                             {o_seq, w.oh, H_q, C, s, 0},
                                             {do_seq, w.doh, H_q, C, s, 0}};
    if ((rc = relayout_n(true, gather, 5, S, B, D, P, dtype, stream))) return rc;
    AttnArgs sa = a;
    sa.q = w.qh; sa.k = w.kh; sa.v = w.vh; sa.o = w.oh; sa.dO = w.doh;
    sa.lse_in = lse + (size_t)h0 * S;
    sa.lse_bstride = (int64_t)H_q * S;
    sa.dq = w.dqh; sa.dk = w.dkh; sa.dv = w.dvh; sa.delta = w.delta;
    rc = use_tc_bwd(sa) ? launch_tc_bwd(sa, st) : launch_simt_bwd(sa, st);
    if (rc) return rc;
    // with kv-head replication every stage holds a partial dK/dV of its kv
    // head: the head's first stage writes it, the later ones add to it
    const int add = (H_kv < P && !kv_first_stage(H_kv, P, s, stages)) ? 1 : 0;
    const ulysses_relayout_item scatter[3] = {{w.dqh, dq_seq, H_q, C, s, 0},
                                              {w.dkh, dk_seq, H_kv, Ckv, ks, add},
                                              {w.dvh, dv_seq, H_kv, Ckv, ks, add}};
    if ((rc = relayout_n(false, scatter, 3, S, B, D, P, ULYSSES_FP32, stream))) return rc;
  }
  return ULYSSES_OK;
}

}  // extern "C"

namespace {
// ---------------------------------------------------------------------------
// Ring-attention variant driven natively: rank r keeps query chunk r and meets
// KV chunk (r - t) mod P at ring step t.
struct RingWs {
  char *qh, *kh, *vh, *oh, *doh;
  float *o_acc, *lse_part, *dqh, *dkh, *dvh, *delta;
  size_t total;
};

RingWs ring_ws(char* base, int64_t L, int Hq, int Hkv, int D, int elt) {
  RingWs w{};
  size_t off = 0;
  auto take = [&](size_t bytes) { char* p = base ? base + off : nullptr; off += align256(bytes); return p; };
  const size_t q_n = (size_t)Hq * L * D, kv_n = (size_t)Hkv * L * D;
  w.qh = take(q_n * elt); w.kh = take(kv_n * elt); w.vh = take(kv_n * elt);
  w.oh = take(q_n * elt); w.doh = take(q_n * elt);
  w.o_acc = (float*)take(q_n * 4); w.lse_part = (float*)take((size_t)Hq * L * 4);
  w.dqh = (float*)take(q_n * 4); w.dkh = (float*)take(kv_n * 4); w.dvh = (float*)take(kv_n * 4);
  w.delta = (float*)take((size_t)Hq * L * 4);
  w.total = off;
  return w;
}

int ring_shape(AttnArgs& a, int64_t S, int H_q, int H_kv, int D, int P, int causal, float scale, int dtype) {
  if (P <= 0 || S < 0 || S % P) return set_error(ULYSSES_ERR_INVALID, "S=%lld not divisible by P=%d", (long long)S, P);
  return attn_shape(a, S / P, 1, H_q, H_kv, D, 1, 0, -1, nullptr, 0, causal, scale, dtype);
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Padding to a multiple of P (pad_to_multiple_of in the TRL section).
int ulysses_pad_seq(const void* x, void* x_pad, int64_t S, int64_t S_pad, int B, int H, int D, int dtype,
                    void* stream) {
  const int elt = elt_size(dtype);
  if (!elt) return set_error(ULYSSES_ERR_INVALID, "unknown dtype %d", dtype);
  if (S < 0 || S_pad < S || B <= 0 || H <= 0 || D <= 0)
    return set_error(ULYSSES_ERR_INVALID, "bad sizes S=%lld S_pad=%lld B=%d H=%d D=%d", (long long)S,
                     (long long)S_pad, B, H, D);
  const int64_t row = (int64_t)H * D * elt;
  if (row % 16) return set_error(ULYSSES_ERR_UNSUPPORTED, "H*D*elt=%lld must be a multiple of 16 bytes", (long long)row);
  if (S_pad == 0) return ULYSSES_OK;
  if (!x_pad || (S > 0 && !x)) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (!aligned16(x_pad) || (S > 0 && !aligned16(x))) return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  if (S > 0 && overlap((const char*)x, (size_t)B * S * row, (const char*)x_pad, (size_t)B * S_pad * row))
    return set_error(ULYSSES_ERR_INVALID, "padding cannot run in place");
  return launch_pad_seq(x, x_pad, S, S_pad, B, row, (cudaStream_t)stream);
}

int ulysses_pad_cu_seqlens(const int32_t* cu_seqlens, int num_docs, int32_t* cu_pad, int64_t S, int64_t S_pad,
                           void* stream) {
  if (S < 0 || S_pad < S || S_pad > ((int64_t)1 << 31) - 1)
    return set_error(ULYSSES_ERR_INVALID, "bad sizes S=%lld S_pad=%lld", (long long)S, (long long)S_pad);
  if (cu_seqlens && num_docs <= 0) return set_error(ULYSSES_ERR_INVALID, "num_docs must be >= 1 with cu_seqlens");
  if (!cu_pad) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  return launch_pad_cu(cu_seqlens, cu_seqlens ? num_docs : 1, cu_pad, S, S_pad, (cudaStream_t)stream);
}

size_t ulysses_ring_workspace(int64_t S, int H_q, int H_kv, int D, int P, int dtype) {
  AttnArgs a;
  if (ring_shape(a, S, H_q, H_kv, D, P, 1, 0.f, dtype)) return 0;
  return ring_ws(nullptr, S / P, H_q, H_kv, D, elt_size(dtype)).total;
}

int ulysses_ring_fwd(const void* q_seq, const void* k_seq, const void* v_seq, void* o_seq, float* lse,
                     int64_t S, int H_q, int H_kv, int D, int P, int causal, float scale, int dtype,
                     void* workspace, size_t ws_bytes, void* stream) {
  AttnArgs a;
  int rc = ring_shape(a, S, H_q, H_kv, D, P, causal, scale, dtype);
  if (rc) return rc;
  if (S == 0) return ULYSSES_OK;
  if (!q_seq || !k_seq || !v_seq || !o_seq || !lse || !workspace) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  const int elt = elt_size(dtype);
  const int64_t L = S / P;
  RingWs w = ring_ws((char*)workspace, L, H_q, H_kv, D, elt);
  if (ws_bytes < w.total) return set_error(ULYSSES_ERR_INVALID, "workspace too small: %zu < %zu", ws_bytes, w.total);
  if (((uintptr_t)workspace & 255u) != 0) return set_error(ULYSSES_ERR_INVALID, "workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const size_t q_chunk = (size_t)L * H_q * D * elt, kv_chunk = (size_t)L * H_kv * D * elt;
  for (int r = 0; r < P; ++r) {
    StageRange range("ring fwd rank", r);
    if ((rc = relayout(true, (const char*)q_seq + r * q_chunk, w.qh, L, 1, H_q, D, 1, 0, -1, dtype, stream)))
      return rc;
    float* lse_r = lse + (size_t)r * H_q * L;
    int first = 1;
    for (int t = 0; t < P; ++t) {
      const int c = (r - t + P) % P;
      if (causal && c > r) continue;                 // a chunk wholly in the future
      const ulysses_relayout_item kv[2] = {{(const char*)k_seq + c * kv_chunk, w.kh, H_kv, 0, -1, 0},
                                           {(const char*)v_seq + c * kv_chunk, w.vh, H_kv, 0, -1, 0}};
      if ((rc = relayout_n(true, kv, 2, L, 1, D, 1, dtype, stream))) return rc;
      AttnArgs sa = a;
      sa.causal = (causal && c == r) ? 1 : 0;       // the diagonal step is causal, the others full
      sa.q = w.qh; sa.k = w.kh; sa.v = w.vh; sa.o_out = w.oh; sa.lse = w.lse_part;
      if ((rc = run_fwd(sa, st))) return rc;
      if ((rc = launch_lse_merge(w.o_acc, lse_r, w.oh, w.lse_part, (int64_t)H_q * L, D, dtype, first, st)))
        return rc;
      first = 0;
    }
    if ((rc = launch_cast_f32(w.oh, w.o_acc, (int64_t)H_q * L * D, dtype, st))) return rc;
    if ((rc = relayout(false, w.oh, (char*)o_seq + r * q_chunk, L, 1, H_q, D, 1, 0, -1, dtype, stream))) return rc;
  }
  return ULYSSES_OK;
}

int ulysses_ring_bwd(const void* q_seq, const void* k_seq, const void* v_seq, const void* o_seq,
                     const void* do_seq, const float* lse, float* dq_seq, float* dk_seq, float* dv_seq,
                     int64_t S, int H_q, int H_kv, int D, int P, int causal, float scale, int dtype,
                     void* workspace, size_t ws_bytes, void* stream) {
  AttnArgs a;
  int rc = ring_shape(a, S, H_q, H_kv, D, P, causal, scale, dtype);
  if (rc) return rc;
  if (S == 0) return ULYSSES_OK;
  if (!q_seq || !k_seq || !v_seq || !o_seq || !do_seq || !lse || !dq_seq || !dk_seq || !dv_seq || !workspace)
    return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (P > 4096) return set_error(ULYSSES_ERR_UNSUPPORTED, "P=%d above 4096 ring ranks", P);
  const int elt = elt_size(dtype);
  const int64_t L = S / P;
  RingWs w = ring_ws((char*)workspace, L, H_q, H_kv, D, elt);
  if (ws_bytes < w.total) return set_error(ULYSSES_ERR_INVALID, "workspace too small: %zu < %zu", ws_bytes, w.total);
  if (((uintptr_t)workspace & 255u) != 0) return set_error(ULYSSES_ERR_INVALID, "workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const size_t q_chunk = (size_t)L * H_q * D * elt, kv_chunk = (size_t)L * H_kv * D * elt;
  const size_t qf_chunk = (size_t)L * H_q * D, kvf_chunk = (size_t)L * H_kv * D;   // fp32 elements
  std::vector<char> kv_seen(P, 0);
  for (int r = 0; r < P; ++r) {
    StageRange range("ring bwd rank", r);
    const ulysses_relayout_item qod[3] = {{(const char*)q_seq + r * q_chunk, w.qh, H_q, 0, -1, 0},
                                          {(const char*)o_seq + r * q_chunk, w.oh, H_q, 0, -1, 0},
                                          {(const char*)do_seq + r * q_chunk, w.doh, H_q, 0, -1, 0}};
    if ((rc = relayout_n(true, qod, 3, L, 1, D, 1, dtype, stream))) return rc;
    bool q_seen = false;
    for (int t = 0; t < P; ++t) {
      const int c = (r - t + P) % P;
      if (causal && c > r) continue;
      const ulysses_relayout_item kv[2] = {{(const char*)k_seq + c * kv_chunk, w.kh, H_kv, 0, -1, 0},
                                           {(const char*)v_seq + c * kv_chunk, w.vh, H_kv, 0, -1, 0}};
      if ((rc = relayout_n(true, kv, 2, L, 1, D, 1, dtype, stream))) return rc;
      AttnArgs sa = a;
      sa.causal = (causal && c == r) ? 1 : 0;
      sa.q = w.qh; sa.k = w.kh; sa.v = w.vh; sa.o = w.oh; sa.dO = w.doh;
      sa.lse_in = lse + (size_t)r * H_q * L;        // the merged LSE of query chunk r
      sa.dq = w.dqh; sa.dk = w.dkh; sa.dv = w.dvh; sa.delta = w.delta;
      if ((rc = run_bwd(sa, st))) return rc;
      // the step's partial gradients: the first one of a chunk writes, the rest add
      const ulysses_relayout_item g[3] = {{w.dqh, dq_seq + r * qf_chunk, H_q, 0, -1, q_seen ? 1 : 0},
                                          {w.dkh, dk_seq + c * kvf_chunk, H_kv, 0, -1, kv_seen[c] ? 1 : 0},
                                          {w.dvh, dv_seq + c * kvf_chunk, H_kv, 0, -1, kv_seen[c] ? 1 : 0}};
      if ((rc = relayout_n(false, g, 3, L, 1, D, 1, ULYSSES_FP32, stream))) return rc;
      q_seen = true;
      kv_seen[c] = 1;
    }
  }
  return ULYSSES_OK;
}

int ulysses_check(void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return set_error(ULYSSES_ERR_CUDA, "stream error: %s", cudaGetErrorString(e));
  unsigned w = read_error_api(st) | read_error_attn_tc_fwd(st) | read_error_attn_tc_bwd(st) |
               read_error_proj_gemm(st);
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(ULYSSES_ERR_CUDA, "error-word read failed: %s", cudaGetErrorString(e));
  if (w & kErrTimeout) return set_error(ULYSSES_ERR_TIMEOUT, "a kernel gave up a bounded wait");
  if (w & kErrSeqlens) return set_error(ULYSSES_ERR_BAD_SEQLENS, "cu_seqlens must rise from 0 to S");
  if (w & kErrBounds) return set_error(ULYSSES_ERR_BOUNDS, "a kernel index fell outside its buffer (checked build)");
  return ULYSSES_OK;
}

const char* ulysses_last_error(void) { return g_msg; }

int ulysses_set_kernel(int which) {
  if (which != ULYSSES_KERNEL_AUTO && which != ULYSSES_KERNEL_SIMT)
    return set_error(ULYSSES_ERR_INVALID, "unknown kernel choice %d", which);
  g_kernel_choice.store(which);
  return ULYSSES_OK;
}

long long ulysses_launch_count(void) { return g_launches.load(); }

int ulysses_checked_build(void) {
#ifdef ULYSSES_CHECKS
  return 1;
#else
  return 0;
#endif
}

}  // extern "C"
