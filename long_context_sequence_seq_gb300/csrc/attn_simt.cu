// K5: fp32 SIMT attention forward/backward (and K3, the D_i pre-pass).
//
// Exact masked softmax attention ("How Ulysses sequence parallelism works",
// step 4) computed with fp32 FMAs and fp32 expf: the path for fp32 inputs,
// whose 1e-4 bound the bf16/tf32 tensor-core formats cannot meet, and for head
// dims the tcgen05 kernels do not cover.  Online softmax over 32-key chunks:
//   m' = max(m, max_j s_ij),  l' = l e^{m-m'} + sum_j e^{s_ij-m'},
//   acc' = acc e^{m-m'} + sum_j e^{s_ij-m'} v_j,   O_i = acc/l, LSE_i = m + ln l.
// Backward recomputes P_ij = exp(s_ij - LSE_i) and forms
//   dP_ij = dO_i.v_j, dS_ij = P_ij (dP_ij - D_i), D_i = dO_i.O_i,
//   dQ_i = scale sum_j dS_ij k_j, dK_j = scale sum_i dS_ij q_i, dV_j = sum_i P_ij dO_i
// in a query-major kernel (dQ) and a key-major kernel (dK, dV, looping over
// the G query heads of the kv head), so no atomics are needed.
//
// Batch is folded into the head index: buffer head n in [0, B*nq) reads kv
// head n / G (the kv buffer holds B*nq/G heads).
#include "common.cuh"
#include "internal.h"

namespace ulysses {

namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;  // 16
constexpr int kChunk = 32;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Load rows [r0, r0+rows) of a [S][D] matrix into shared fp32 [rows][ld], zero past S.
template <typename T, int D>
__device__ __forceinline__ void load_rows(float* dst, int ld, const T* __restrict__ src, int64_t S,
                                          int64_t r0, int rows) {
  for (int e = threadIdx.x; e < rows * D; e += blockDim.x) {
    int r = e / D, d = e % D;
    int64_t gr = r0 + r;
    dst[r * ld + d] = (gr >= 0 && gr < S) ? to_f32<T>(src[gr * D + d]) : 0.f;
  }
}

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) simt_fwd_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ o,
    float* __restrict__ lse, int64_t S, int nq, int G, int64_t lse_bstride,
    const int32_t* __restrict__ cu, int nd, int causal, float scale) {
  constexpr int DW = D / 32;
  extern __shared__ float smem[];
  float(*Qs)[D] = reinterpret_cast<float(*)[D]>(smem);
  float(*Ks)[D + 1] = reinterpret_cast<float(*)[D + 1]>(smem + kRowsPerCta * D);
  float(*Vs)[D + 1] = reinterpret_cast<float(*)[D + 1]>(smem + kRowsPerCta * D + kChunk * (D + 1));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n = blockIdx.y;
  const int64_t kvh = n / G;
  const T* qh = q + n * S * D;
  const T* kh = k + kvh * S * D;
  const T* vh = v + kvh * S * D;
  const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta;
  const int64_t last = min(row0 + kRowsPerCta, S) - 1;

  int64_t lo[kRowsPerWarp], hi[kRowsPerWarp];
  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DW];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    int64_t i = row0 + warp * kRowsPerWarp + r;
    if (i < S) key_range(cu, nd, S, causal, i, lo[r], hi[r]); else { lo[r] = 0; hi[r] = 0; }
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int dd = 0; dd < DW; ++dd) acc[r][dd] = 0.f;
  }
  int64_t kmin, kmax, tmp;
  key_range(cu, nd, S, causal, row0, kmin, tmp);
  key_range(cu, nd, S, causal, last, tmp, kmax);

  load_rows<T, D>(&Qs[0][0], D, qh, S, row0, kRowsPerCta);
  for (int64_t c0 = kmin; c0 < kmax; c0 += kChunk) {
    __syncthreads();
    load_rows<T, D>(&Ks[0][0], D + 1, kh, S, c0, kChunk);
    load_rows<T, D>(&Vs[0][0], D + 1, vh, S, c0, kChunk);
    __syncthreads();
    const int64_t j = c0 + lane;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      if (c0 >= hi[r] || c0 + kChunk <= lo[r]) continue;  // warp-uniform
      const float* qr = Qs[warp * kRowsPerWarp + r];
      float s = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) s = fmaf(qr[d], Ks[lane][d], s);
      s *= scale;
      const bool ok = (j >= lo[r]) && (j < hi[r]);
      s = ok ? s : -INFINITY;
      const float mc = warp_max(s);
      if (mc == -INFINITY) continue;
      const float mn = fmaxf(m[r], mc);
      const float alpha = (m[r] == -INFINITY) ? 0.f : expf(m[r] - mn);
      const float p = ok ? expf(s - mn) : 0.f;
      l[r] = l[r] * alpha + warp_sum(p);
#pragma unroll
      for (int dd = 0; dd < DW; ++dd) acc[r][dd] *= alpha;
      for (int jj = 0; jj < kChunk; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int dd = 0; dd < DW; ++dd) acc[r][dd] = fmaf(pj, Vs[jj][lane + 32 * dd], acc[r][dd]);
      }
      m[r] = mn;
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    int64_t i = row0 + warp * kRowsPerWarp + r;
    if (i >= S) continue;
    const float inv = 1.f / l[r];
#pragma unroll
    for (int dd = 0; dd < DW; ++dd) {
      const int64_t oi = (n * S + i) * D + lane + 32 * dd;
      if (in_bounds(oi, (int64_t)gridDim.y * S * D)) o[oi] = from_f32<T>(acc[r][dd] * inv);
    }
    const int64_t li = lse_index(n, nq, lse_bstride, S, i);
    if (lane == 0 && in_bounds(li, ((int64_t)gridDim.y + nq - 1) / nq * lse_bstride)) lse[li] = m[r] + logf(l[r]);
  }
}

// K3: D_i = sum_d dO_id O_id  (fp32), one warp per row.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const T* __restrict__ o,
                                                        const T* __restrict__ dO,
                                                        float* __restrict__ delta, int64_t rows) {
  const int lane = threadIdx.x & 31;
  int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  float s = 0.f;
#pragma unroll
  if (in_bounds(row * D + D - 1, rows * D))
    for (int d = lane; d < D; d += 32) s = fmaf(to_f32<T>(o[row * D + d]), to_f32<T>(dO[row * D + d]), s);
  s = warp_sum(s);
  if (lane == 0) delta[row] = s;
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) simt_bwd_dq_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const T* __restrict__ dO, const float* __restrict__ lse, const float* __restrict__ delta,
    float* __restrict__ dq, int64_t S, int nq, int G, int64_t lse_bstride,
    const int32_t* __restrict__ cu, int nd, int causal, float scale) {
  constexpr int DW = D / 32;
  extern __shared__ float smem[];
  float(*Qs)[D] = reinterpret_cast<float(*)[D]>(smem);
  float(*dOs)[D] = reinterpret_cast<float(*)[D]>(smem + kRowsPerCta * D);
  float(*Ks)[D + 1] = reinterpret_cast<float(*)[D + 1]>(smem + 2 * kRowsPerCta * D);
  float(*Vs)[D + 1] =
      reinterpret_cast<float(*)[D + 1]>(smem + 2 * kRowsPerCta * D + kChunk * (D + 1));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n = blockIdx.y;
  const int64_t kvh = n / G;
  const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta;
  const int64_t last = min(row0 + kRowsPerCta, S) - 1;
  int64_t lo[kRowsPerWarp], hi[kRowsPerWarp];
  float L[kRowsPerWarp], Dl[kRowsPerWarp], acc[kRowsPerWarp][DW];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    int64_t i = row0 + warp * kRowsPerWarp + r;
    if (i < S) {
      key_range(cu, nd, S, causal, i, lo[r], hi[r]);
      const int64_t li = lse_index(n, nq, lse_bstride, S, i), di = n * S + i;
      L[r] = in_bounds(li, ((int64_t)gridDim.y + nq - 1) / nq * lse_bstride) ? lse[li] : 0.f;
      Dl[r] = in_bounds(di, (int64_t)gridDim.y * S) ? delta[di] : 0.f;
    } else { lo[r] = 0; hi[r] = 0; L[r] = 0.f; Dl[r] = 0.f; }
#pragma unroll
    for (int dd = 0; dd < DW; ++dd) acc[r][dd] = 0.f;
  }
  int64_t kmin, kmax, tmp;
  key_range(cu, nd, S, causal, row0, kmin, tmp);
  key_range(cu, nd, S, causal, last, tmp, kmax);
  load_rows<T, D>(&Qs[0][0], D, q + n * S * D, S, row0, kRowsPerCta);
  load_rows<T, D>(&dOs[0][0], D, dO + n * S * D, S, row0, kRowsPerCta);
  for (int64_t c0 = kmin; c0 < kmax; c0 += kChunk) {
    __syncthreads();
    load_rows<T, D>(&Ks[0][0], D + 1, k + kvh * S * D, S, c0, kChunk);
    load_rows<T, D>(&Vs[0][0], D + 1, v + kvh * S * D, S, c0, kChunk);
    __syncthreads();
    const int64_t j = c0 + lane;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      if (c0 >= hi[r] || c0 + kChunk <= lo[r]) continue;
      const float* qr = Qs[warp * kRowsPerWarp + r];
      const float* dr = dOs[warp * kRowsPerWarp + r];
      float s = 0.f, dp = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) {
        s = fmaf(qr[d], Ks[lane][d], s);
        dp = fmaf(dr[d], Vs[lane][d], dp);
      }
      const bool ok = (j >= lo[r]) && (j < hi[r]);
      const float p = ok ? expf(s * scale - L[r]) : 0.f;
      const float ds = p * (dp - Dl[r]);
      for (int jj = 0; jj < kChunk; ++jj) {
        const float dj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
        for (int dd = 0; dd < DW; ++dd) acc[r][dd] = fmaf(dj, Ks[jj][lane + 32 * dd], acc[r][dd]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    int64_t i = row0 + warp * kRowsPerWarp + r;
    if (i >= S) continue;
#pragma unroll
    for (int dd = 0; dd < DW; ++dd) {
      const int64_t qi = (n * S + i) * D + lane + 32 * dd;
      if (in_bounds(qi, (int64_t)gridDim.y * S * D)) dq[qi] = acc[r][dd] * scale;
    }
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) simt_bwd_dkdv_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const T* __restrict__ dO, const float* __restrict__ lse, const float* __restrict__ delta,
    float* __restrict__ dk, float* __restrict__ dv, int64_t S, int nq, int G, int64_t lse_bstride,
    const int32_t* __restrict__ cu, int nd, int causal, float scale) {
  constexpr int DW = D / 32;
  extern __shared__ float smem[];
  float(*Kr)[D] = reinterpret_cast<float(*)[D]>(smem);
  float(*Vr)[D] = reinterpret_cast<float(*)[D]>(smem + kRowsPerCta * D);
  float(*Qs)[D + 1] = reinterpret_cast<float(*)[D + 1]>(smem + 2 * kRowsPerCta * D);
  float(*dOs)[D + 1] =
      reinterpret_cast<float(*)[D + 1]>(smem + 2 * kRowsPerCta * D + kChunk * (D + 1));
  float* Ls = smem + 2 * kRowsPerCta * D + 2 * kChunk * (D + 1);
  float* Ds = Ls + kChunk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t kvh = blockIdx.y;
  const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta;
  const int64_t last = min(row0 + kRowsPerCta, S) - 1;
  int64_t lo[kRowsPerWarp], hi[kRowsPerWarp];
  float ak[kRowsPerWarp][DW], av[kRowsPerWarp][DW];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    int64_t j = row0 + warp * kRowsPerWarp + r;
    if (j < S) query_range(cu, nd, S, causal, j, lo[r], hi[r]); else { lo[r] = 0; hi[r] = 0; }
#pragma unroll
    for (int dd = 0; dd < DW; ++dd) { ak[r][dd] = 0.f; av[r][dd] = 0.f; }
  }
  int64_t qmin, qmax, tmp;
  query_range(cu, nd, S, causal, row0, qmin, tmp);
  query_range(cu, nd, S, causal, last, tmp, qmax);
  load_rows<T, D>(&Kr[0][0], D, k + kvh * S * D, S, row0, kRowsPerCta);
  load_rows<T, D>(&Vr[0][0], D, v + kvh * S * D, S, row0, kRowsPerCta);
  for (int g = 0; g < G; ++g) {
    const int64_t n = kvh * G + g;
    for (int64_t c0 = qmin; c0 < qmax; c0 += kChunk) {
      __syncthreads();
      load_rows<T, D>(&Qs[0][0], D + 1, q + n * S * D, S, c0, kChunk);
      load_rows<T, D>(&dOs[0][0], D + 1, dO + n * S * D, S, c0, kChunk);
      if (threadIdx.x < kChunk) {
        int64_t i = c0 + threadIdx.x;
        const int64_t li = lse_index(n, nq, lse_bstride, S, i), di = n * S + i;
        const int64_t n_q = (int64_t)gridDim.y * G;   // this kernel's grid runs over kv heads
        Ls[threadIdx.x] = (i < S && in_bounds(li, (n_q + nq - 1) / nq * lse_bstride)) ? lse[li] : 0.f;
        Ds[threadIdx.x] = (i < S && in_bounds(di, n_q * S)) ? delta[di] : 0.f;
      }
      __syncthreads();
      const int64_t i = c0 + lane;
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        if (c0 >= hi[r] || c0 + kChunk <= lo[r]) continue;
        const float* kr = Kr[warp * kRowsPerWarp + r];
        const float* vr = Vr[warp * kRowsPerWarp + r];
        float s = 0.f, dp = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; ++d) {
          s = fmaf(Qs[lane][d], kr[d], s);
          dp = fmaf(dOs[lane][d], vr[d], dp);
        }
        const bool ok = (i >= lo[r]) && (i < hi[r]);
        const float p = ok ? expf(s * scale - Ls[lane]) : 0.f;
        const float ds = p * (dp - Ds[lane]);
        for (int ii = 0; ii < kChunk; ++ii) {
          const float pi = __shfl_sync(0xffffffffu, p, ii);
          const float di = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
          for (int dd = 0; dd < DW; ++dd) {
            av[r][dd] = fmaf(pi, dOs[ii][lane + 32 * dd], av[r][dd]);
            ak[r][dd] = fmaf(di, Qs[ii][lane + 32 * dd], ak[r][dd]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    int64_t j = row0 + warp * kRowsPerWarp + r;
    if (j >= S) continue;
#pragma unroll
    for (int dd = 0; dd < DW; ++dd) {
      const int64_t ki = (kvh * S + j) * D + lane + 32 * dd;
      if (!in_bounds(ki, (int64_t)gridDim.y * S * D)) continue;
      dk[ki] = ak[r][dd] * scale;
      dv[ki] = av[r][dd];
    }
  }
}

// ---------------------------------------------------------------------------
// Launchers (called by api.cu after validation)
// ---------------------------------------------------------------------------



template <int D>
constexpr size_t fwd_smem() { return sizeof(float) * (kRowsPerCta * D + 2 * kChunk * (D + 1)); }
template <int D>
constexpr size_t bwd_smem() {
  return sizeof(float) * (2 * kRowsPerCta * D + 2 * kChunk * (D + 1) + 2 * kChunk);
}

template <typename K>
static void allow_smem(K kernel, size_t bytes) {
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int D>
static int simt_fwd_t(const AttnArgs& a, cudaStream_t st) {
  dim3 grid((unsigned)((a.S + kRowsPerCta - 1) / kRowsPerCta), (unsigned)a.n_q);
  allow_smem(simt_fwd_kernel<T, D>, fwd_smem<D>());
  simt_fwd_kernel<T, D><<<grid, kWarps * 32, fwd_smem<D>(), st>>>(
      (const T*)a.q, (const T*)a.k, (const T*)a.v, (T*)a.o_out, a.lse, a.S, a.nq, a.G,
      a.lse_bstride, a.cu, a.nd, a.causal, a.scale);
  count_launch();
  return check_launch("simt_fwd");
}

template <typename T, int D>
static int delta_t(const AttnArgs& a, cudaStream_t st) {
  int64_t rows = (int64_t)a.n_q * a.S;
  unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
  bwd_delta_kernel<T, D><<<blocks, 256, 0, st>>>((const T*)a.o, (const T*)a.dO, a.delta, rows);
  count_launch();
  return check_launch("bwd_delta");
}

template <typename T, int D>
static int simt_bwd_t(const AttnArgs& a, cudaStream_t st) {
  int rc = delta_t<T, D>(a, st);
  if (rc) return rc;
  dim3 gq((unsigned)((a.S + kRowsPerCta - 1) / kRowsPerCta), (unsigned)a.n_q);
  allow_smem(simt_bwd_dq_kernel<T, D>, bwd_smem<D>());
  simt_bwd_dq_kernel<T, D><<<gq, kWarps * 32, bwd_smem<D>(), st>>>(
      (const T*)a.q, (const T*)a.k, (const T*)a.v, (const T*)a.dO, a.lse_in, a.delta, a.dq, a.S,
      a.nq, a.G, a.lse_bstride, a.cu, a.nd, a.causal, a.scale);
  count_launch();
  if ((rc = check_launch("simt_bwd_dq"))) return rc;
  dim3 gk((unsigned)((a.S + kRowsPerCta - 1) / kRowsPerCta), (unsigned)(a.n_q / a.G));
  allow_smem(simt_bwd_dkdv_kernel<T, D>, bwd_smem<D>());
  simt_bwd_dkdv_kernel<T, D><<<gk, kWarps * 32, bwd_smem<D>(), st>>>(
      (const T*)a.q, (const T*)a.k, (const T*)a.v, (const T*)a.dO, a.lse_in, a.delta, a.dk, a.dv,
      a.S, a.nq, a.G, a.lse_bstride, a.cu, a.nd, a.causal, a.scale);
  count_launch();
  return check_launch("simt_bwd_dkdv");
}

int launch_simt_fwd(const AttnArgs& a, cudaStream_t st) {
  if (a.dtype == ULYSSES_FP32)
    return a.D == 64 ? simt_fwd_t<float, 64>(a, st) : simt_fwd_t<float, 128>(a, st);
  return a.D == 64 ? simt_fwd_t<__nv_bfloat16, 64>(a, st) : simt_fwd_t<__nv_bfloat16, 128>(a, st);
}

int launch_delta(const AttnArgs& a, cudaStream_t st) {
  if (a.dtype == ULYSSES_FP32)
    return a.D == 64 ? delta_t<float, 64>(a, st) : delta_t<float, 128>(a, st);
  return a.D == 64 ? delta_t<__nv_bfloat16, 64>(a, st) : delta_t<__nv_bfloat16, 128>(a, st);
}

int launch_simt_bwd(const AttnArgs& a, cudaStream_t st) {
  if (a.dtype == ULYSSES_FP32)
    return a.D == 64 ? simt_bwd_t<float, 64>(a, st) : simt_bwd_t<float, 128>(a, st);
  return a.D == 64 ? simt_bwd_t<__nv_bfloat16, 64>(a, st) : simt_bwd_t<__nv_bfloat16, 128>(a, st);
}

}  // namespace ulysses
