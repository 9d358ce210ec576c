// Projections with the re-layout fused into the GEMM (steps 2 and 6 of "How
// Ulysses sequence parallelism works"): on one device the all-to-alls around
// the projections become addressing, so
//   QKV projection  C = X W_qkv^T   writes its tiles straight into head layout
//                   [H_q + 2 H_kv][S][D] (Q heads, then K heads, then V heads);
//   out projection  Y = O W_o^T     reads O straight out of head layout
//                   [H_q][S][D] (a 3D TMA map gathers the K dimension across
//                   heads), writing Y row-major [S][hidden].
// bf16 operands, fp32 accumulation in TMEM, bf16 results.
//
// Persistent tcgen05 GEMM: one CTA per SM walks output tiles of 128 x 256
// (n fastest, so the CTAs working at one time share A row blocks in L2).
//   warp 0      TMA producer: A (128 x 64) and B (256 x 64) k-chunks into a
//               4-stage ring (48 KB a stage)
//   warp 1      TMEM owner; issues tcgen05.mma M=128 N=256 K=16 warp-wide
//               (one elected lane), accumulating a tile in one of two
//               256-column TMEM buffers
//   warps 4-7   epilogue: TMEM lane quarter = 32 rows of the tile; reads the
//               256 columns in 32-column chunks, rounds to bf16, stores; the
//               next tile's MMAs run meanwhile in the other buffer
// All waits are bounded (the library's mbarrier wait).
#include <cuda_bf16.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace ulysses {

ULYSSES_ERROR_READER(read_error_proj_gemm)

namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int NST = 4;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;

struct GemmLayout {
  static constexpr int kTileA = BM * BK * 2;     // 16 KB, swizzle-128B
  static constexpr int kTileB = BN * BK * 2;     // 32 KB
  static constexpr int kStage = kTileA + kTileB;
  static constexpr int kBar = NST * kStage;
  // full[NST], empty[NST], acc_full[2], acc_empty[2], drain
  static constexpr int kNumBar = 2 * NST + 4 + 1;
  static constexpr int kMisc = kBar + kNumBar * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

// A: head layout (k = head * D + d) when a_head_dim > 0, else row-major.
// C: head layout [N / c_head_dim][M][c_head_dim] when c_head_dim > 0, else
// row-major [M][N].
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   __nv_bfloat16* __restrict__ out, int64_t M, int N, int K, int a_head_dim,
                   int c_head_dim) {
  using L = GemmLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* full = bars;
  uint64_t* empty = full + NST;
  uint64_t* acc_full = empty + NST;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = N / BN;
  const int64_t m_tiles = (M + BM - 1) / BM;
  const int64_t total = m_tiles * n_tiles;
  const int kchunks = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 4); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmA);
    tma_prefetch(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int64_t g = 0;   // k-chunks issued so far by this CTA
      bool go = true;
      for (int64_t t = blockIdx.x; go && t < total; t += gridDim.x) {
        const int m0 = (int)((t / n_tiles) * BM), n0 = (int)((t % n_tiles) * BN);
        for (int kc = 0; kc < kchunks; ++kc, ++g) {
          const int s = (int)(g % NST);
          if (!mbar_wait(&empty[s], ((uint32_t)(g / NST) & 1u) ^ 1u, abort_flag)) { go = false; break; }
          uint8_t* st = smem + s * L::kStage;
          mbar_expect_tx(&full[s], L::kStage);
          const int k0 = kc * BK;
          if (a_head_dim > 0)
            tma_load_3d(st, &tmA, k0 % a_head_dim, m0, k0 / a_head_dim, &full[s]);
          else
            tma_load_3d(st, &tmA, k0, m0, 0, &full[s]);
          tma_load_3d(st + L::kTileA, &tmB, k0, n0, 0, &full[s]);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16(BM, BN, false, false);
    bool ok = true;
    int64_t g = 0;
    int i = 0;
    for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x, ++i) {
      const uint32_t b = (uint32_t)(i & 1);
      // the epilogue has read this accumulator's previous tile
      if (!mbar_wait_warp(&acc_empty[b], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      for (int kc = 0; kc < kchunks; ++kc, ++g) {
        const int s = (int)(g % NST);
        if (!mbar_wait_warp(&full[s], (uint32_t)(g / NST) & 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t ad = sdesc_sw128(smem_u32(smem + s * L::kStage), 16, 1024);
        const uint64_t bd = sdesc_sw128(smem_u32(smem + s * L::kStage + L::kTileA), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ss_w(tbase + b * BN, sdesc_add(ad, kk * 32), sdesc_add(bd, kk * 32), idesc,
                   (kc > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(&empty[s]);
      }
      if (!ok) break;
      mma_commit_w(&acc_full[b]);
    }
    mma_commit_w(drain);
    mbar_wait(drain, 0, nullptr);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    int i = 0;
    for (int64_t t = blockIdx.x; t < total; t += gridDim.x, ++i) {
      const uint32_t b = (uint32_t)(i & 1);
      if (!mbar_wait_warp(&acc_full[b], (uint32_t)(i >> 1) & 1u, abort_flag)) break;
      tc_fence_after();
      const int64_t m = (t / n_tiles) * BM + wq * 32 + lane;
      const int n0 = (int)((t % n_tiles) * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + b * BN + c * 32, v);
        tmem_ld_wait();
        reg_fence(v);
        if (c == BN / 32 - 1) {
          // every column of this accumulator is in registers: free it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
        const int n = n0 + c * 32;
        __nv_bfloat16* dst = c_head_dim > 0
            ? out + ((int64_t)(n / c_head_dim) * M + m) * c_head_dim + (n % c_head_dim)
            : out + m * (int64_t)N + n;
        if (m < M && in_bounds((dst - out) + 31, M * (int64_t)N)) {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_uint4(pack_bf16(__uint_as_float(v[8 * e]), __uint_as_float(v[8 * e + 1])),
                               pack_bf16(__uint_as_float(v[8 * e + 2]), __uint_as_float(v[8 * e + 3])),
                               pack_bf16(__uint_as_float(v[8 * e + 4]), __uint_as_float(v[8 * e + 5])),
                               pack_bf16(__uint_as_float(v[8 * e + 6]), __uint_as_float(v[8 * e + 7])));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

int launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, void* out, int64_t M, int N, int K, int a_head_dim,
                int c_head_dim, cudaStream_t st) {
  const int smem = GemmLayout::kAlloc;
  static PerDeviceOnce<> smem_once;
  int rc = opt_in_smem(smem_once, (const void*)tc_gemm_kernel, smem, "tc_gemm");
  if (rc) return rc;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t total = (M + BM - 1) / BM * (N / BN);
  const unsigned grid = (unsigned)(total < sms ? total : sms);
  tc_gemm_kernel<<<grid, kThreads, smem, st>>>(ta, tb, (__nv_bfloat16*)out, M, N, K, a_head_dim, c_head_dim);
  count_launch();
  return check_launch("tc_gemm");
}

}  // namespace

int launch_qkv_proj(const void* x, const void* w, void* qkv_head, int64_t S, int hidden, int n_heads, int D,
                    cudaStream_t st) {
  CUtensorMap ta, tb;
  int rc;
  const int N = n_heads * D;
  if ((rc = make_tmap_bf16_3d(&ta, x, S, 1, hidden, BM))) return rc;      // [S][hidden]
  if ((rc = make_tmap_bf16_3d(&tb, w, N, 1, hidden, BN))) return rc;      // [N][hidden]
  return launch_gemm(ta, tb, qkv_head, S, N, hidden, 0, D, st);
}

int launch_out_proj(const void* o_head, const void* w, void* y, int64_t S, int H_q, int D, int hidden,
                    cudaStream_t st) {
  CUtensorMap ta, tb;
  int rc;
  if ((rc = make_tmap_bf16_3d(&ta, o_head, S, H_q, D, BM))) return rc;   // [H_q][S][D]
  if ((rc = make_tmap_bf16_3d(&tb, w, hidden, 1, H_q * D, BN))) return rc;   // [hidden][H_q D]
  return launch_gemm(ta, tb, y, S, hidden, H_q * D, D, 0, st);
}

}  // namespace ulysses
