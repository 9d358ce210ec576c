// K1: the two all-to-alls of Ulysses sequence parallelism as on-device
// permutations ("How Ulysses sequence parallelism works", steps 3 and 5).
//
//   seq layout  X_seq [B][S][H][D]  (P stacked rank chunks of S/P tokens)
//   head layout X_head[B][n][S][D]  (the stage's n heads, every position)
//   X_head[b][h'][t][:] = X_seq[b][t][h0 + h'][:]
// The scatter also has an accumulating form (fp32), X_seq += X_head, which
// sums the partial dK/dV of stages that share a replicated kv head.
//
// One launch moves a batch of up to kMaxJobs tensors of one stage (Q, K and V
// of a forward stage; Q, K, V, O and dO of a backward stage; dQ, dK and dV),
// so the small K/V tensors do not pay a launch and a tail of their own.  The
// grid is two-dimensional: blockIdx.x = (tensor, batch entry, head), fastest,
// so CTAs that run together read neighbouring heads of the same tokens;
// blockIdx.y = a block of tokens.  A thread block is (words of a row) x (rows):
// the unit moved is one D-vector (128-512 bytes) as 16-byte words, so both
// sides are coalesced, and no division runs per word (one per CTA).  The
// kernel is a pure HBM stream: 2 * bytes moved per call, no arithmetic.
// Bit-exact by construction (raw 16-byte words, any element type).
#include "common.cuh"
#include "internal.h"

namespace ulysses {

namespace {

constexpr int kRows = 4;          // rows per thread per token block (loads in flight)
constexpr int kThreads = 256;

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ int4 add_f32x4(int4 a, int4 b) {
  return make_int4(__float_as_int(__int_as_float(a.x) + __int_as_float(b.x)),
                   __float_as_int(__int_as_float(a.y) + __int_as_float(b.y)),
                   __float_as_int(__int_as_float(a.z) + __int_as_float(b.z)),
                   __float_as_int(__int_as_float(a.w) + __int_as_float(b.w)));
}

// to_head = true:  seq -> head (gather)   to_head = false: head -> seq (scatter)
template <bool kToHead>
__global__ void __launch_bounds__(kThreads) relayout_kernel(const __grid_constant__ RelayoutBatch bt) {
  // the job (tensor) of this CTA: the last one whose first column is <= x
  const int x = blockIdx.x;
  int j = 0;
#pragma unroll
  for (int k = 1; k < kMaxRelayoutJobs; ++k)
    if (k < bt.njobs && x >= bt.job[k].x0) j = k;
  const RelayoutJob& jb = bt.job[j];
  const int bh = x - jb.x0;                 // b * n + hh
  const int b = bh / jb.n, hh = bh - b * jb.n;
  const int V = bt.V;
  const int64_t S = bt.S;
  const int4* __restrict__ src = reinterpret_cast<const int4*>(jb.src);
  int4* __restrict__ dst = reinterpret_cast<int4*>(jb.dst);
  // word offsets of token 0 of this (b, head) on both sides, and the step
  // between consecutive tokens
  const int64_t head_base = (int64_t)bh * S * V;
  const int64_t seq_base = ((int64_t)b * S * jb.H + jb.h0 + hh) * V;
  const int64_t seq_step = (int64_t)jb.H * V;
  const int64_t head_total = (int64_t)bt.B * jb.n * S * V, seq_total = (int64_t)bt.B * S * jb.H * V;
  const int64_t src_total = kToHead ? seq_total : head_total, dst_total = kToHead ? head_total : seq_total;
  const int rows_per_blk = blockDim.y * kRows;
  for (int64_t tb = blockIdx.y; tb * rows_per_blk < S; tb += gridDim.y) {
    const int64_t t0 = tb * rows_per_blk + threadIdx.y;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
      int4 val[kRows];
      bool ok[kRows];
#pragma unroll
      for (int u = 0; u < kRows; ++u) {
        const int64_t t = t0 + (int64_t)u * blockDim.y;
        const int64_t si = (kToHead ? seq_base + t * seq_step : head_base + t * V) + v;
        const int64_t di = (kToHead ? head_base + t * V : seq_base + t * seq_step) + v;
        ok[u] = t < S && in_bounds(si, src_total) && in_bounds(di, dst_total);
        if (ok[u]) val[u] = ld_stream(src + si);
      }
#pragma unroll
      for (int u = 0; u < kRows; ++u) {
        if (ok[u]) {
          const int64_t t = t0 + (int64_t)u * blockDim.y;
          int4* p = dst + (kToHead ? head_base + t * V : seq_base + t * seq_step) + v;
          if (!kToHead && jb.add) *p = add_f32x4(*p, val[u]);
          else *p = val[u];
        }
      }
    }
  }
}

}  // namespace

int launch_relayout_batch(bool to_head, RelayoutBatch& bt, cudaStream_t stream) {
  if (bt.njobs <= 0 || bt.S == 0) return ULYSSES_OK;
  int cols = 0;
  for (int k = 0; k < bt.njobs; ++k) {
    bt.job[k].x0 = cols;
    cols += bt.B * bt.job[k].n;
  }
  const int bx = bt.V < kThreads ? bt.V : kThreads;
  const int by = kThreads / bx;
  const int64_t n_tb = (bt.S + (int64_t)by * kRows - 1) / ((int64_t)by * kRows);
  dim3 block((unsigned)bx, (unsigned)by);
  dim3 grid((unsigned)cols, (unsigned)(n_tb < 65535 ? n_tb : 65535));
  if (to_head)
    relayout_kernel<true><<<grid, block, 0, stream>>>(bt);
  else
    relayout_kernel<false><<<grid, block, 0, stream>>>(bt);
  count_launch();
  return check_launch("relayout");
}

int launch_relayout(bool to_head, const void* src, void* dst, int64_t S, int B, int H, int D,
                    int n, int h0, int elt, cudaStream_t stream, bool add) {
  RelayoutBatch bt{};
  bt.njobs = 1;
  bt.S = S;
  bt.B = B;
  bt.V = D * elt / 16;
  bt.job[0] = RelayoutJob{src, dst, H, n, h0, add ? 1 : 0, 0};
  return launch_relayout_batch(to_head, bt, stream);
}

}  // namespace ulysses
