// Shared device helpers: error word, bounded waits, launch bookkeeping.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ulysses.h"

namespace ulysses {

// Device error word bits (read and cleared by ulysses_check).
enum : unsigned {
  kErrTimeout = 1u,     // a bounded wait gave up
  kErrSeqlens = 2u,     // cu_seqlens not monotone from 0 to S
  kErrBounds = 4u,      // checked build: an index fell outside its buffer
};

// One error word per translation unit (no relocatable device code is needed);
// api.cu reads and clears every unit's word through its reader function.
static __device__ unsigned g_error_word;

#define ULYSSES_ERROR_READER(fn)                                                   \
  unsigned fn(cudaStream_t st) {                                                   \
    unsigned v = 0, zero = 0;                                                      \
    cudaMemcpyFromSymbolAsync(&v, g_error_word, sizeof(v), 0,                      \
                              cudaMemcpyDeviceToHost, st);                         \
    cudaMemcpyToSymbolAsync(g_error_word, &zero, sizeof(zero), 0,                  \
                            cudaMemcpyHostToDevice, st);                           \
    cudaStreamSynchronize(st);                                                     \
    return v;                                                                      \
  }

// Host-side helpers implemented in api.cu.
void count_launch(int n = 1);
int set_error(int code, const char* fmt, ...);
int check_launch(const char* what);

__device__ __forceinline__ void raise_error(unsigned bits) { atomicOr(&g_error_word, bits); }

// Bounds check of a global-memory index against its buffer's element count.
// Built with -DULYSSES_CHECKS (the checked library), a failing check records
// kErrBounds in the error word and the caller skips the access, so an index
// bug is reported by ulysses_check instead of reading or writing outside the
// buffer.  In the normal build it is constant true and costs nothing.
#ifdef ULYSSES_CHECKS
__device__ __forceinline__ bool in_bounds(int64_t i, int64_t n) {
  if (i >= 0 && i < n) return true;
  raise_error(kErrBounds);
  return false;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(int64_t, int64_t) { return true; }
#endif

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound for any single spin-wait inside a kernel.  Every legitimate
// wait in these kernels is microseconds long; two seconds means something is
// wrong and the kernel bails out instead of hanging the device.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Document of token t: largest d with cu[d] <= t (binary search, cu has nd+1 entries).
__device__ __forceinline__ int doc_of(const int32_t* __restrict__ cu, int nd, int64_t t) {
  int lo = 0, hi = nd - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// LSE element of buffer head n (batch folded into n), token t.
__device__ __forceinline__ int64_t lse_index(int64_t n, int nq, int64_t lse_bstride, int64_t S,
                                             int64_t t) {
  return (n / nq) * lse_bstride + (n % nq) * S + t;
}

// Key range [lo, hi) of query row i.
__device__ __forceinline__ void key_range(const int32_t* __restrict__ cu, int nd, int64_t S,
                                          int causal, int64_t i, int64_t& lo, int64_t& hi) {
  int64_t ds = 0, de = S;
  if (cu != nullptr) {
    int d = doc_of(cu, nd, i);
    ds = __ldg(cu + d);
    de = __ldg(cu + d + 1);
  }
  // clamp so that a malformed table (flagged separately) cannot drive
  // loops or loads outside [0, S)
  lo = ds < 0 ? 0 : (ds > S ? S : ds);
  hi = causal ? i + 1 : (de < 0 ? 0 : (de > S ? S : de));
  if (hi < lo) hi = lo;
}

// Query range [lo, hi) of rows that attend key j (the transpose of key_range).
__device__ __forceinline__ void query_range(const int32_t* __restrict__ cu, int nd, int64_t S,
                                            int causal, int64_t j, int64_t& lo, int64_t& hi) {
  int64_t ds = 0, de = S;
  if (cu != nullptr) {
    int d = doc_of(cu, nd, j);
    ds = __ldg(cu + d);
    de = __ldg(cu + d + 1);
  }
  lo = causal ? j : (ds < 0 ? 0 : (ds > S ? S : ds));
  hi = de < 0 ? 0 : (de > S ? S : de);
  if (hi < lo) hi = lo;
}

}  // namespace ulysses
