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

int relayout(bool to_head, const void* src, void* dst, int64_t S, int B, int H, int D, int P,
             int C, int stage, int dtype, void* stream, bool add = false) {
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
  if (S == 0) return ULYSSES_OK;
  if (!src || !dst) return set_error(ULYSSES_ERR_INVALID, "NULL buffer");
  if (!aligned16(src) || !aligned16(dst)) return set_error(ULYSSES_ERR_INVALID, "buffers must be 16-byte aligned");
  const size_t seq_bytes = (size_t)B * S * H * D * elt, head_bytes = (size_t)B * n * S * D * elt;
  const char* a = (const char*)src; const char* b = (const char*)dst;
  size_t la = to_head ? seq_bytes : head_bytes, lb = to_head ? head_bytes : seq_bytes;
  if (a < b + lb && b < a + la) return set_error(ULYSSES_ERR_INVALID, "re-layout cannot run in place");
  return launch_relayout(to_head, src, dst, S, B, H, D, n, h0, elt, (cudaStream_t)stream, add);
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
// looked up once per device (with that device current) and passed to kernels.
constexpr size_t kNoAllocDeltaFloats = size_t(1) << 22;   // 4,194,304 rows
static __device__ __align__(256) float g_noalloc_delta[kNoAllocDeltaFloats];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(ULYSSES_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_error(ULYSSES_ERR_UNSUPPORTED, "device %d beyond %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_delta);
    if (e != cudaSuccess || p == nullptr)
      return set_error(ULYSSES_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
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
    if ((rc = relayout(true, q_seq, w.qh, S, B, H_q, D, P, C, s, dtype, stream))) return rc;
    if ((rc = relayout(true, k_seq, w.kh, S, B, H_kv, D, P, Ckv, ks, dtype, stream))) return rc;
    if ((rc = relayout(true, v_seq, w.vh, S, B, H_kv, D, P, Ckv, ks, dtype, stream))) return rc;
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
    if ((rc = relayout(true, q_seq, w.qh, S, B, H_q, D, P, C, s, dtype, stream))) return rc;
    if ((rc = relayout(true, k_seq, w.kh, S, B, H_kv, D, P, Ckv, ks, dtype, stream))) return rc;
    if ((rc = relayout(true, v_seq, w.vh, S, B, H_kv, D, P, Ckv, ks, dtype, stream))) return rc;
    if ((rc = relayout(true, o_seq, w.oh, S, B, H_q, D, P, C, s, dtype, stream))) return rc;
    if ((rc = relayout(true, do_seq, w.doh, S, B, H_q, D, P, C, s, dtype, stream))) return rc;
    AttnArgs sa = a;
    sa.q = w.qh; sa.k = w.kh; sa.v = w.vh; sa.o = w.oh; sa.dO = w.doh;
    sa.lse_in = lse + (size_t)h0 * S;
    sa.lse_bstride = (int64_t)H_q * S;
    sa.dq = w.dqh; sa.dk = w.dkh; sa.dv = w.dvh; sa.delta = w.delta;
    rc = use_tc_bwd(sa) ? launch_tc_bwd(sa, st) : launch_simt_bwd(sa, st);
    if (rc) return rc;
    if ((rc = relayout(false, w.dqh, dq_seq, S, B, H_q, D, P, C, s, ULYSSES_FP32, stream))) return rc;
    // with kv-head replication every stage holds a partial dK/dV of its kv
    // head: the head's first stage writes it, the later ones add to it
    const bool add = H_kv < P && !kv_first_stage(H_kv, P, s, stages);
    if ((rc = relayout(false, w.dkh, dk_seq, S, B, H_kv, D, P, Ckv, ks, ULYSSES_FP32, stream, add))) return rc;
    if ((rc = relayout(false, w.dvh, dv_seq, S, B, H_kv, D, P, Ckv, ks, ULYSSES_FP32, stream, add))) return rc;
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

}  // extern "C"
