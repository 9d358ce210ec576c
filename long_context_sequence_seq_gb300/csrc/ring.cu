// Pieces of the ring-attention variant ("Ulysses vs Ring" comparison of the
// Ulysses sequence parallelism pages): every rank keeps its query chunk and
// sees the KV chunks one ring step at a time, so the partial results of the
// steps are merged with their log-sum-exp weights:
//   LSE = log(e^{LSE_a} + e^{LSE_b}),  O = e^{LSE_a - LSE} O_a + e^{LSE_b - LSE} O_b
// and the backward's partial dQ/dK/dV of the steps are summed.  The
// attention blocks themselves run in the K2/K4 kernels.  These kernels are
// HBM streams: one pass over the rows they touch.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ulysses {

namespace {

// One warp per row; D / 32 elements per lane.
template <typename T>
__global__ void __launch_bounds__(256) lse_merge_kernel(float* __restrict__ o_acc, float* __restrict__ lse_acc,
                                                        const T* __restrict__ o_part,
                                                        const float* __restrict__ lse_part, int64_t rows,
                                                        int D, int first) {
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float lb = lse_part[row];
  float wa = 0.f, wb = 1.f, l = lb;
  if (!first) {
    const float la = lse_acc[row];
    const float m = fmaxf(la, lb);
    if (m == -INFINITY) {            // neither step saw a key: keep the empty row
      wa = 0.f; wb = 0.f; l = -INFINITY;
    } else {
      const float ea = expf(la - m), eb = expf(lb - m);
      l = m + logf(ea + eb);
      wa = ea / (ea + eb);
      wb = eb / (ea + eb);
    }
  } else if (lb == -INFINITY) {
    wb = 0.f;
  }
  float* oa = o_acc + row * D;
  const T* ob = o_part + row * D;
  for (int d = lane; d < D; d += 32) {
    const float b = (float)ob[d];
    oa[d] = first ? wb * b : wa * oa[d] + wb * b;
  }
  if (lane == 0) lse_acc[row] = l;
}

template <typename T>
__global__ void __launch_bounds__(256) cast_kernel(T* __restrict__ dst, const float* __restrict__ src, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = (T)src[i];
}

__global__ void __launch_bounds__(256) add_kernel(float* __restrict__ dst, const float* __restrict__ src, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] += src[i];
}

unsigned grid_for(int64_t n) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (n + 255) / 256, cap = (int64_t)sms * 8;
  return (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

int launch_lse_merge(float* o_acc, float* lse_acc, const void* o_part, const float* lse_part, int64_t rows,
                     int D, int dtype, int first, cudaStream_t st) {
  if (rows == 0) return ULYSSES_OK;
  const unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
  if (dtype == ULYSSES_BF16)
    lse_merge_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(o_acc, lse_acc, (const __nv_bfloat16*)o_part,
                                                              lse_part, rows, D, first);
  else
    lse_merge_kernel<float><<<blocks, 256, 0, st>>>(o_acc, lse_acc, (const float*)o_part, lse_part, rows, D,
                                                     first);
  count_launch();
  return check_launch("lse_merge");
}

int launch_cast_f32(void* dst, const float* src, int64_t n, int dtype, cudaStream_t st) {
  if (n == 0) return ULYSSES_OK;
  if (dtype == ULYSSES_BF16)
    cast_kernel<__nv_bfloat16><<<grid_for(n), 256, 0, st>>>((__nv_bfloat16*)dst, src, n);
  else
    cast_kernel<float><<<grid_for(n), 256, 0, st>>>((float*)dst, src, n);
  count_launch();
  return check_launch("cast_f32");
}

int launch_add_f32(float* dst, const float* src, int64_t n, cudaStream_t st) {
  if (n == 0) return ULYSSES_OK;
  add_kernel<<<grid_for(n), 256, 0, st>>>(dst, src, n);
  count_launch();
  return check_launch("add_f32");
}

}  // namespace ulysses
