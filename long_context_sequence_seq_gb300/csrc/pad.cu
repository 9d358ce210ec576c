// Padding the sequence to a multiple of the sequence-parallel degree.
//
// The pages' TRL section sets pad_to_multiple_of to the SP size so that the
// sequence splits evenly over the ranks (the sequence-divisibility best
// practice).  Padding here appends zero tokens and gives them a document of
// their own in cu_seqlens, so no real token attends to a pad token or is
// attended by one, and the real tokens' results equal those of the unpadded
// sequence.  Both kernels are plain HBM streams (the copy moves 16-byte
// words; the cu_seqlens kernel writes num_docs + 2 integers).
#include "common.cuh"
#include "internal.h"

namespace ulysses {

namespace {

// x_pad[b][t][:] = t < S ? x[b][t][:] : 0, rows of W 16-byte words.
__global__ void __launch_bounds__(256) pad_seq_kernel(const int4* __restrict__ src, int4* __restrict__ dst,
                                                      int64_t S, int64_t S_pad, int64_t W, int64_t total) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t w = i % W, row = i / W;          // row = b * S_pad + t
    const int64_t t = row % S_pad, b = row / S_pad;
    const int64_t si = (b * S + t) * W + w;
    dst[i] = (t < S && in_bounds(si, (total / S_pad) * S * W)) ? src[si] : make_int4(0, 0, 0, 0);
  }
}

// cu_pad[0..nd] = the real documents (one document [0, S] without a table),
// cu_pad[nd + 1] = S_pad when there is padding.
__global__ void pad_cu_kernel(const int32_t* __restrict__ cu, int nd, int32_t* __restrict__ out, int64_t S,
                              int64_t S_pad) {
  for (int i = threadIdx.x + blockIdx.x * blockDim.x; i <= nd + 1; i += blockDim.x * gridDim.x) {
    if (i <= nd) out[i] = cu ? cu[i] : (i == 0 ? 0 : (int32_t)S);
    else if (S_pad > S) out[i] = (int32_t)S_pad;
  }
}

}  // namespace

int launch_pad_seq(const void* x, void* x_pad, int64_t S, int64_t S_pad, int B, int64_t row_bytes,
                   cudaStream_t st) {
  const int64_t W = row_bytes / 16, total = (int64_t)B * S_pad * W;
  if (total == 0) return ULYSSES_OK;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (total + 255) / 256, cap = (int64_t)sms * 8;
  pad_seq_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, st>>>((const int4*)x, (int4*)x_pad, S, S_pad, W,
                                                                       total);
  count_launch();
  return check_launch("pad_seq");
}

int launch_pad_cu(const int32_t* cu, int nd, int32_t* out, int64_t S, int64_t S_pad, cudaStream_t st) {
  pad_cu_kernel<<<1, 256, 0, st>>>(cu, nd, out, S, S_pad);
  count_launch();
  return check_launch("pad_cu_seqlens");
}

}  // namespace ulysses
