// K1: the two all-to-alls of Ulysses sequence parallelism as on-device
// permutations ("How Ulysses sequence parallelism works", steps 3 and 5).
//
//   seq layout  X_seq [B][S][H][D]  (P stacked rank chunks of S/P tokens)
//   head layout X_head[B][n][S][D]  (the stage's n heads, every position)
//   X_head[b][h'][t][:] = X_seq[b][t][h0 + h'][:]
// The scatter also has an accumulating form (fp32), X_seq += X_head, which
// sums the partial dK/dV of stages that share a replicated kv head.
//
// The unit moved is one D-vector (128-512 bytes), copied as 16-byte words, so
// both the read and the write side are fully coalesced.  The kernel is a pure
// HBM stream: 2 * bytes moved per call, no arithmetic.  Bit-exact by
// construction (raw 16-byte words, any element type).
#include "common.cuh"

namespace ulysses {

// Each thread moves kUnroll 16-byte words per iteration of a grid-stride loop.
constexpr int kUnroll = 4;

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// to_head = true:  seq -> head (gather)   to_head = false: head -> seq (scatter)
// kAdd (scatter only): add the fp32 head rows into the sequence rows
template <bool kToHead, bool kAdd = false>
__global__ void __launch_bounds__(256) relayout_kernel(const int4* __restrict__ src,
                                                       int4* __restrict__ dst, int64_t S,
                                                       int n, int H, int h0, int vec_per_row,
                                                       int64_t total_vecs) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // index o enumerates the head layout [B][n][S][V] (V = 16-byte words per row)
  for (; base < total_vecs; base += stride * kUnroll) {
    int4 val[kUnroll];
    int64_t seq_idx[kUnroll], head_idx[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      int64_t o = base + (int64_t)u * stride;
      head_idx[u] = o;
      if (o < total_vecs) {
        int64_t v = o % vec_per_row;
        int64_t row = o / vec_per_row;        // ((b*n + hh)*S + t)
        int64_t t = row % S;
        int64_t bh = row / S;
        int64_t hh = bh % n;
        int64_t b = bh / n;
        seq_idx[u] = (((b * S + t) * H) + h0 + hh) * vec_per_row + v;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (head_idx[u] < total_vecs)
        val[u] = ld_stream(src + (kToHead ? seq_idx[u] : head_idx[u]));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (head_idx[u] < total_vecs) {
        if (kAdd) {
          int4* p = dst + seq_idx[u];
          const int4 o = *p;
          val[u] = make_int4(__float_as_int(__int_as_float(o.x) + __int_as_float(val[u].x)),
                             __float_as_int(__int_as_float(o.y) + __int_as_float(val[u].y)),
                             __float_as_int(__int_as_float(o.z) + __int_as_float(val[u].z)),
                             __float_as_int(__int_as_float(o.w) + __int_as_float(val[u].w)));
          *p = val[u];
        } else {
          dst[kToHead ? head_idx[u] : seq_idx[u]] = val[u];
        }
      }
    }
  }
}

int launch_relayout(bool to_head, const void* src, void* dst, int64_t S, int B, int H, int D,
                    int n, int h0, int elt, cudaStream_t stream, bool add) {
  const int row_bytes = D * elt;
  const int vec_per_row = row_bytes / 16;
  const int64_t total = (int64_t)B * n * S * vec_per_row;
  if (total == 0) return ULYSSES_OK;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  int64_t want = (total + (int64_t)threads * kUnroll - 1) / ((int64_t)threads * kUnroll);
  int64_t cap = (int64_t)sms * 8;  // 8 CTAs of 256 threads per SM: full occupancy
  int blocks = (int)(want < cap ? want : cap);
  if (to_head)
    relayout_kernel<true><<<blocks, threads, 0, stream>>>(
        (const int4*)src, (int4*)dst, S, n, H, h0, vec_per_row, total);
  else if (add)
    relayout_kernel<false, true><<<blocks, threads, 0, stream>>>(
        (const int4*)src, (int4*)dst, S, n, H, h0, vec_per_row, total);
  else
    relayout_kernel<false><<<blocks, threads, 0, stream>>>(
        (const int4*)src, (int4*)dst, S, n, H, h0, vec_per_row, total);
  count_launch();
  return check_launch("relayout");
}

}  // namespace ulysses
