// Internal launcher interfaces shared by the CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "device_once.h"

namespace ulysses {

// Arguments of one attention launch on head-layout buffers (batch folded into
// the head index: buffer q head n in [0, n_q) reads kv head n / G).
struct AttnArgs {
  const void* q; const void* k; const void* v; const void* o; const void* dO;
  void* o_out;          // forward output O (input dtype)
  float* lse;           // forward output LSE
  const float* lse_in;  // backward input LSE
  float* dq; float* dk; float* dv;
  float* delta;         // backward scratch D_i, [n_q][S]
  int64_t S;
  int n_q;              // q heads in the buffer across the batch (B * nq)
  int nq;               // q heads per batch entry in the buffer
  int G; int D;
  int64_t lse_bstride;  // LSE element stride between batch entries
  const int32_t* cu; int nd; int causal; float scale; int dtype;
  // seq != 0: q/k/v/o/dO and dq/dk/dv point at the stage's first head inside
  // sequence-layout tensors [S][hq_tot or hkv_tot][D] (B == 1) instead of
  // head-layout buffers: the re-layout is folded into the kernels' addressing
  int seq; int hq_tot; int hkv_tot;
};

// Opts `func` in to `bytes` of dynamic shared memory on the current device,
// once per device (the runtime records the attribute per device); reports
// ULYSSES_ERR_CUDA with a message when the runtime refuses.  api.cu.
int opt_in_smem(PerDeviceOnce<>& once, const void* func, int bytes, const char* what);

// One tensor of a batched re-layout launch (relayout.cu): moves n heads
// starting at h0 of a sequence-layout tensor with H heads to or from a
// head-layout buffer; `add` (scatter, fp32 only) adds instead of writing.
// x0 is filled in by the launcher.
constexpr int kMaxRelayoutJobs = 6;
struct RelayoutJob {
  const void* src; void* dst;
  int H, n, h0, add;
  int x0;
};
// Tensors of one launch share S, B and the row size V (16-byte words per
// D-vector).
struct RelayoutBatch {
  RelayoutJob job[kMaxRelayoutJobs];
  int njobs;
  int B;
  int V;
  int64_t S;
};
int launch_relayout_batch(bool to_head, RelayoutBatch& bt, cudaStream_t stream);
int launch_relayout(bool to_head, const void* src, void* dst, int64_t S, int B, int H, int D,
                    int n, int h0, int elt, cudaStream_t stream, bool add = false);
int launch_simt_fwd(const AttnArgs& a, cudaStream_t st);
int launch_simt_bwd(const AttnArgs& a, cudaStream_t st);
int launch_delta(const AttnArgs& a, cudaStream_t st);
int launch_check_seqlens(const int32_t* cu, int nd, int64_t S, cudaStream_t st);
int launch_lse_merge(float* o_acc, float* lse_acc, const void* o_part, const float* lse_part, int64_t rows,
                     int D, int dtype, int first, cudaStream_t st);                       // ring.cu
int launch_cast_f32(void* dst, const float* src, int64_t n, int dtype, cudaStream_t st);  // ring.cu
int launch_add_f32(float* dst, const float* src, int64_t n, cudaStream_t st);             // ring.cu
int launch_pad_seq(const void* x, void* x_pad, int64_t S, int64_t S_pad, int B, int64_t row_bytes,
                   cudaStream_t st);                                                      // pad.cu
int launch_pad_cu(const int32_t* cu, int nd, int32_t* out, int64_t S, int64_t S_pad, cudaStream_t st);  // pad.cu
int launch_qkv_proj(const void* x, const void* w, void* qkv_head, int64_t S, int hidden, int n_heads, int D,
                    cudaStream_t st);                                                     // proj_gemm.cu
int launch_out_proj(const void* o_head, const void* w, void* y, int64_t S, int H_q, int D, int hidden,
                    cudaStream_t st);                                                     // proj_gemm.cu

}  // namespace ulysses
