// K3 + K4: attention backward for sm_103a (bf16 inputs, fp32 gradients).
//
// The adjoint of step 4 of "How Ulysses sequence parallelism works" (local
// dense attention): with P recomputed from the saved logsumexp,
//   P_ij = exp(s_ij - LSE_i),  dV_j = sum_i P_ij dO_i,  dP_ij = dO_i.v_j,
//   D_i = dO_i.O_i,  dS_ij = P_ij (dP_ij - D_i),
//   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
// dK/dV summed over the G query heads of each kv head.
//
// K3 (bwd_pre_kernel): D_i for every row and dQ := 0 (dQ is accumulated with
// fp32 reductions by K4).
//
// K4 (tc_bwd_kernel): one CTA per (kv head, 128-key block); it owns dK/dV of
// its block (accumulated in TMEM, no atomics) and walks the G query heads and
// every 64-row query block that can see its keys.  Transposed formulation,
// so the key index is the TMEM lane:
//   S^T  = K Q_i^T            (M=128 keys, N=64 queries, K=D; A = K from smem)
//   dP^T = V dO_i^T           (A = V, copied into TMEM once per CTA)
//   softmax warps: P^T = exp2(S^T*scale*log2e - LSE_i*log2e), masked, stored
//                  back to TMEM as bf16; dS^T = P^T (dP^T - D_i) to shared
//                  memory (swizzled, [key][query]).
//   dV  += P^T dO_i            (A = P^T from TMEM, B = dO_i, MN-major)
//   dK  += dS^T Q_i            (A = dS^T from shared memory, K-major; B = Q_i, MN-major)
//   dQ_i^T = K^T dS^T          (M = D, N = 64 queries; A = K, MN-major;
//                               B = dS^T from shared memory, MN-major)
// Keeping V in TMEM makes dP^T an A-from-TMEM MMA (the shared-memory operand
// reads bound the N = 64 shared-memory form) and frees V's 32 KB of shared
// memory for a fifth Q/dO stage.
// Four readout warps then read dQ_i^T out of TMEM (lane = feature d) and
// write scale * dQ_i as [query][feature] fp32 rows into the tile's consumed
// Q/dO stage buffers; a flusher warp adds them into dQ with TMA bulk
// reduce-adds (cp.reduce.async.bulk) and then releases the stage.
//
// What bounds it: neither the tensor pipe nor shared memory saturates (at a
// 16K stage: tensor pipe 51% of active cycles, shared-memory banks 27% read /
// 11% write); the MMAs of a tile take ~1540 clk at full rate against ~2540
// clk per tile.  An event trace of one CTA at S = 64K shows the period equal
// to a Q/dO stage's lifetime over the five stages: a stage is held from its
// TMA load (~3000 clk to arrive: the same TMA unit carries the dQ reductions)
// through the tile's MMAs and gradient work to the flusher's reductions of
// the dQ rows staged in it (~2100 clk for 32 KB).  Timing-only variants that
// skip work: no dQ reductions +7%, half of them +5%, no Q/dO loads +5%, no
// P/dS arithmetic +5%.
//
// Warp roles (512 threads): 0 TMA producer (lane 0) and LSE/D_i loader (all
// lanes), 1 TMEM owner and score-MMA issuer, 2 gradient-MMA issuer (both
// issue warp-wide, one elected lane issues), 3 dQ flusher, 4-7 dQ^T readout
// (one per TMEM lane quarter), 8-15 gradient warps: two per lane quarter,
// each taking 32 of the tile's 64 queries (thread = key row).  Warpgroups 0-1
// run on 112 registers per thread and give the rest to the gradient
// warpgroups (144).  TMEM columns: dV [0,128), dK [128,256), two S^T/P^T
// buffers [256,384) that also receive each tile's dQ^T, one dP^T buffer
// [384,448) and V [448,512) (bf16, two features per column).
#include <type_traits>

#include "internal.h"
#include "tc_ptx.cuh"

namespace ulysses {

ULYSSES_ERROR_READER(read_error_attn_tc_bwd)

namespace {

using namespace tc;

constexpr int BN = 128;     // keys per CTA
constexpr int BMQ = 64;     // queries per inner tile
constexpr int D = 128;
constexpr int NSTAGE = 5;   // Q/dO/LSE/D_i ring (a consumed stage also stages its dQ tile)
constexpr int kThreads = 512;
constexpr int kReadWarps = 4;   // warps 4..7: dQ^T readout, one per TMEM lane quarter
constexpr int kGradWarps = 8;   // warps 8..15: two per TMEM lane quarter, one per 32-query half
// Register budgets: warpgroups 0-1 give registers back, 2-3 (gradient) take
// them: 2 * 128 * kRegsLow + 2 * 128 * kRegsHigh = 128 (launch) * 512 threads.
constexpr uint32_t kRegsLow = 112, kRegsHigh = 144;
static_assert(2 * 128 * kRegsLow + 2 * 128 * kRegsHigh == 128 * kThreads, "register split");
constexpr uint32_t kTmemCols = 512;
// TMEM: dV, dK accumulators; two S^T/P^T buffers (each later reused for the
// tile's dQ^T); one dP^T buffer; V as the A operand of dP^T.
constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384, kColV = 448;
constexpr float kLog2e = 1.4426950408889634f;

// TMEM column of bf16 K-step kk (16 queries) of a packed P^T / dS^T tile: each
// 32-query half is packed into the first 16 columns of its own 32 fp32
// columns, so neither half overwrites scores the other half still reads.
__device__ __forceinline__ uint32_t packed_col(int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); }

struct BwdLayout {
  static constexpr int kChunkKV = BN * 128;          // 64 features x 128 keys
  static constexpr int kChunkQ = BMQ * 128;          // 64 features x 64 queries
  static constexpr int kTileKV = kChunkKV * (D / 64);
  static constexpr int kTileQ = kChunkQ * (D / 64);
  static constexpr int kTileDS = BN * BMQ * 2;       // [128 keys][64 queries] bf16
  static constexpr int kK = 0;
  static constexpr int kQ = kK + kTileKV;                    // NSTAGE tiles
  static constexpr int kDO = kQ + NSTAGE * kTileQ;            // NSTAGE tiles
  static constexpr int kDS = kDO + NSTAGE * kTileQ;           // one dS^T tile
  static constexpr int kStat = kDS + kTileDS;                 // NSTAGE x {LSE2[64], D[64]}
  static constexpr int kBar = kStat + NSTAGE * 2 * BMQ * 4;
  // kv_full, q_full[NSTAGE], q_empty[NSTAGE], s_full[2], ds_full[2], dsm_free,
  // dq_full[2], dq_empty, fin, drain, stg_full[NSTAGE], dk_done[NSTAGE],
  // v_full, dp_free, p_full[2]
  static constexpr int kNumBar = 1 + 4 * NSTAGE + 7 + 3 + 4 + 1 + 1;
  static constexpr int kMisc = kBar + kNumBar * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};
static_assert(BwdLayout::kAlloc <= 232448, "shared memory budget");

__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      float* __restrict__ delta,
                                                      float* __restrict__ dq, int64_t rows, int64_t S,
                                                      int seq, int hq_tot) {
  const int lane = threadIdx.x & 31;
  const int64_t hr = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;   // head-major row
  if (hr >= rows) return;
  // where the row lives: head layout [n][S][D], or sequence layout [S][hq_tot][D]
  const int64_t row = seq ? (hr % S) * hq_tot + hr / S : hr;
  if (!in_bounds(row * D + D - 1, (seq ? (int64_t)hq_tot * S : rows) * D)) return;
  // 128 features = 32 lanes x 4
  const uint2 ov = *reinterpret_cast<const uint2*>(o + row * D + lane * 4);
  const uint2 dv = *reinterpret_cast<const uint2*>(dO + row * D + lane * 4);
  const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
  const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float2 a = __bfloat1622float2(o2[e]), b = __bfloat1622float2(d2[e]);
    s = fmaf(a.x, b.x, s);
    s = fmaf(a.y, b.y, s);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) delta[hr] = s;
  *reinterpret_cast<float4*>(dq + row * D + lane * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Work of a key block: the 64-query tiles that see its keys (the same range
// the kernel walks).
__device__ __forceinline__ int key_block_work(int kb, const int32_t* __restrict__ cu, int nd, int64_t S,
                                              int causal) {
  const int64_t k0 = (int64_t)kb * BN;
  const int64_t last_key = (k0 + BN < S ? k0 + BN : S) - 1;
  int64_t q_lo, q_hi, tmp;
  query_range(cu, nd, S, causal, k0, q_lo, tmp);
  query_range(cu, nd, S, causal, last_key, tmp, q_hi);
  q_lo = (q_lo / BMQ) * BMQ;
  return q_hi > q_lo ? (int)((q_hi - q_lo + BMQ - 1) / BMQ) : 0;
}

// Block-wide sum of a per-thread count in [0, 16) through __syncthreads_count
// on its bits (every thread of the CTA must call it).
__device__ __forceinline__ int block_count16(int c) {
  return __syncthreads_count(c & 1) + 2 * __syncthreads_count(c & 2) + 4 * __syncthreads_count(c & 4) +
         8 * __syncthreads_count(c & 8);
}

// With packed documents the work of a key block depends on its document, so
// key blocks in index order leave a heavy block of a late document to start
// near the end of the grid.  Rank r of the grid gets instead the r-th key
// block in decreasing work (ties: lower block first), the longest-processing-
// time order a list scheduler such as the block scheduler handles best.  Every
// CTA selects its own block: it evaluates the work of all nkb blocks (kLptPer
// per thread), finds by bisection the work value t of rank r (the least t
// with fewer than r + 1 blocks above it), then the block among those of work
// t.  All threads of the CTA call it; `scratch` holds 33 words.
constexpr int kLptPer = 8;
constexpr int kLptMaxBlocks = kLptPer * kThreads;
__device__ int lpt_key_block(int r, int nkb, const int32_t* __restrict__ cu, int nd, int64_t S, int causal,
                             int* scratch) {
  int wk[kLptPer];
  int wmax = 0;
#pragma unroll
  for (int i = 0; i < kLptPer; ++i) {
    const int kb = (int)threadIdx.x + i * kThreads;
    wk[i] = kb < nkb ? key_block_work(kb, cu, nd, S, causal) : -1;
    wmax = wk[i] > wmax ? wk[i] : wmax;
  }
  auto count_above = [&](int t) {
    int c = 0;
#pragma unroll
    for (int i = 0; i < kLptPer; ++i) c += wk[i] > t ? 1 : 0;
    return block_count16(c);
  };
  // the largest work in the CTA: bisection bound (every thread takes part)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int o = 16; o > 0; o >>= 1) wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
  if (lane == 0) scratch[warp] = wmax;
  __syncthreads();
  int hi = 0;
  for (int w = 0; w < kThreads / 32; ++w) hi = max(hi, scratch[w]);
  __syncthreads();
  int lo = 0;   // count_above(hi) == 0 <= r
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (count_above(mid) <= r) hi = mid; else lo = mid + 1;
  }
  int idx = r - count_above(lo);   // rank among the blocks of work lo, in index order
  int result = -1;
#pragma unroll
  for (int i = 0; i < kLptPer; ++i) {
    if (result >= 0) continue;   // uniform over the CTA
    const bool m = wk[i] == lo;
    const int ci = __syncthreads_count(m);
    if (idx < ci) {
      // exclusive prefix of m over thread index (block index order in chunk i)
      const unsigned bal = __ballot_sync(0xffffffffu, m);
      if (lane == 0) scratch[warp] = __popc(bal);
      __syncthreads();
      int before = __popc(bal & ((1u << lane) - 1u));
      for (int w = 0; w < warp; ++w) before += scratch[w];
      if (m && before == idx) scratch[32] = (int)threadIdx.x + i * kThreads;
      __syncthreads();
      result = scratch[32];
    } else {
      idx -= ci;
    }
  }
  fence_async_smem();   // the scratch words are overwritten by TMA later
  __syncthreads();
  return result < 0 ? 0 : result;
}

// Pipeline, it = tile, b = it & 1.  Score issuer (warp 1), running ahead:
//   S^T_it, dP^T_it -> s_full[b]   (needs Q/dO of it, the readout of dQ^T_{it-2}
//                                    which lived in S buffer b, and every
//                                    gradient warp done reading dP^T_{it-1})
// Gradient issuer (warp 2):
//   wait p_full[b]   dV += P^T_it dO_it
//   wait ds_full[b]  dQ^T_it = K^T dS^T_it (into S buffer b) -> dq_full[b]
//                    dK += dS^T_it Q_it                     -> dsm_free, dk_done[stage]
// so the tensor pipe runs tile it's gradient MMAs and later tiles' score MMAs
// while the gradient warps work.  dQ^T goes before dK so that its readout
// (which frees S buffer b for the scores of it+2) overlaps dK; the readout
// then waits for dk_done before it reuses the tile's Q buffer.  Barriers the
// score issuer waits on are per buffer (dq_empty[b]) or cannot run a phase
// ahead of it (dp_free, q_full need its own earlier MMAs), so parity waits
// are unambiguous; the per-stage dk_done cannot run two phases ahead of the
// readout: dK of the stage's next tile needs the stage refilled, which needs
// this readout.
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const float* __restrict__ lse, const float* __restrict__ delta,
                  float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
                  int64_t S, int nq, int G, int64_t lse_bstride, const int32_t* __restrict__ cu,
                  int nd, int causal, float scale, const __grid_constant__ CUtensorMap tmDQ, int seq,
                  int hkv_tot, const __nv_bfloat16* __restrict__ vptr) {
  using L = BwdLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem + L::kK;
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sDO = smem + L::kDO;
  uint8_t* sDS = smem + L::kDS;
  float* sStat = reinterpret_cast<float*>(smem + L::kStat);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + NSTAGE;
  uint64_t* s_full = q_empty + NSTAGE;
  uint64_t* ds_full = s_full + 2;
  uint64_t* dsm_free = ds_full + 2;
  uint64_t* dq_full = dsm_free + 1;
  uint64_t* dq_empty = dq_full + 2;       // [2] readout of the dQ^T in S buffer b done
  uint64_t* fin = dq_empty + 2;
  uint64_t* drain = fin + 1;
  uint64_t* stg_full = drain + 1;     // dQ tile of a stage written to its Q/dO buffers
  uint64_t* dk_done = stg_full + NSTAGE;   // dK of a stage's tile done: its Q buffer is free
  uint64_t* v_full = dk_done + NSTAGE;     // V copied into TMEM
  uint64_t* dp_free = v_full + 1;          // every gradient warp has read the tile's dP^T
  uint64_t* p_full = dp_free + 1;          // [2] P^T of the tile written to TMEM
  uint64_t* drain_s = p_full + 2;          // the score issuer's MMAs have all completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.x;                          // kv head in the buffer
  // key block: in index order (already decreasing work without documents),
  // or in decreasing work for packed documents; the Q stage area is free
  // scratch until the first TMA load
  const int kb = (cu != nullptr && gridDim.y <= kLptMaxBlocks)
                     ? lpt_key_block((int)blockIdx.y, (int)gridDim.y, cu, nd, S, causal,
                                     reinterpret_cast<int*>(sQ))
                     : (int)blockIdx.y;
  const int64_t k0 = (int64_t)kb * BN;                 // first key of the block

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&q_full[s], 2);
      mbar_init(&q_empty[s], 1);
      mbar_init(&stg_full[s], kReadWarps);
      mbar_init(&dk_done[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&ds_full[b], kGradWarps);
      mbar_init(&dq_full[b], 1);
    }
    mbar_init(&dq_empty[0], kReadWarps);
    mbar_init(&dq_empty[1], kReadWarps);
    mbar_init(dsm_free, 1);
    mbar_init(fin, 1);
    mbar_init(drain, 1);
    mbar_init(v_full, kReadWarps);
    mbar_init(dp_free, kGradWarps);
    mbar_init(&p_full[0], kGradWarps);
    mbar_init(&p_full[1], kGradWarps);
    mbar_init(drain_s, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmQ); tma_prefetch(&tmK); tma_prefetch(&tmDO);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  if (warp < 8) regs_dec<kRegsLow>(); else regs_inc<kRegsHigh>();

  // Query rows that can see this key block: [q_lo, q_hi), q_lo rounded down
  // to the query tile so every tile starts on a 64-row boundary.
  const int64_t last_key = (k0 + BN < S ? k0 + BN : S) - 1;
  int64_t q_lo, q_hi, tmp;
  query_range(cu, nd, S, causal, k0, q_lo, tmp);
  query_range(cu, nd, S, causal, last_key, tmp, q_hi);
  q_lo = (q_lo / BMQ) * BMQ;
  const int n_qb = q_hi > q_lo ? (int)((q_hi - q_lo + BMQ - 1) / BMQ) : 0;
  const int n_it = n_qb * G;   // iteration it -> q head g = it / n_qb, block qb = it % n_qb

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer + LSE / D_i loader
    // Lane 0 issues the TMA loads; every lane then loads two rows' LSE and
    // D_i terms of the tile into the stage's stats (the second arrival on
    // q_full).
    if (lane == 0) {
      mbar_expect_tx(kv_full, L::kTileKV);
      for (int c = 0; c < D / 64; ++c) {
        // head layout: (feature, row, head); sequence layout: (feature, head, row)
        tma_load_3d(sK + c * L::kChunkKV, &tmK, c * 64, seq ? kvh : (int)k0, seq ? (int)k0 : kvh, kv_full);
      }
    }
    __syncwarp();
    for (int it = 0; it < n_it; ++it) {
      const int st = it % NSTAGE;
      const uint32_t round = it / NSTAGE;
      if (!mbar_wait_warp(&q_empty[st], (round & 1) ^ 1, abort_flag)) break;
      const int n = kvh * G + it / n_qb;
      const int64_t q0 = q_lo + (int64_t)(it % n_qb) * BMQ;
      if (lane == 0) {
        mbar_expect_tx(&q_full[st], 2 * L::kTileQ);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(sQ + st * L::kTileQ + c * L::kChunkQ, &tmQ, c * 64, seq ? n : (int)q0, seq ? (int)q0 : n,
                      &q_full[st]);
          tma_load_3d(sDO + st * L::kTileQ + c * L::kChunkQ, &tmDO, c * 64, seq ? n : (int)q0, seq ? (int)q0 : n,
                      &q_full[st]);
        }
      }
      float* stat = sStat + st * 2 * BMQ;
#pragma unroll
      for (int r = lane; r < BMQ; r += 32) {
        const int64_t i = q0 + r;
        const int64_t li = lse_index(n, nq, lse_bstride, S, i), di = (int64_t)n * S + i;
        const int64_t n_q = (int64_t)gridDim.x * G;
        stat[r] = (i < S && in_bounds(li, (n_q + nq - 1) / nq * lse_bstride)) ? lse[li] * kLog2e : 0.f;
        stat[BMQ + r] = (i < S && in_bounds(di, n_q * S)) ? delta[di] : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[st]);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues S^T and dP^T of every tile as soon as its stage, its S
    // buffer and the dP^T buffer are free, running ahead of the gradient
    // warps; warp 2 issues the gradient MMAs of each tile (dV once P^T is in
    // TMEM, dQ^T and dK once dS^T is in shared memory).  MMAs of different
    // warps are not ordered with respect to each other: every cross-warp
    // dependency goes through an mbarrier (s_full, p_full, ds_full, dq_full
    // -> readout -> dq_empty, dp_free, dsm_free).
    constexpr uint32_t id_s = idesc_bf16(BN, BMQ, false, false);    // S^T, dP^T
    constexpr uint32_t id_g = idesc_bf16(BN, D, false, true);       // dV, dK
    constexpr uint32_t id_q = idesc_bf16(D, BMQ, true, true);       // dQ^T
    const uint32_t k_addr = smem_u32(sK);
    const uint64_t kd_k = sdesc_sw128(k_addr, 16, 1024);           // K, K-major
    const uint64_t kd_mn = sdesc_sw128(k_addr, L::kChunkKV, 1024);  // K^T, MN-major
    const uint64_t dsd_k = sdesc_sw128(smem_u32(sDS), 16, 1024);    // dS^T as the K-major A of dK
    auto issue_scores = [&](int it) -> bool {
      const int st = it % NSTAGE;
      const uint32_t round = it / NSTAGE;
      if (!mbar_wait_warp(&q_full[st], round & 1, abort_flag)) return false;
      // S buffer of this parity held dQ^T_{it-2}: its readout must be done
      if (it >= 2 && !mbar_wait_warp(&dq_empty[it & 1], ((it - 2) >> 1) & 1, abort_flag)) return false;
      // the single dP^T buffer: every gradient warp has read dP^T_{it-1}
      if (it >= 1 && !mbar_wait_warp(dp_free, (it - 1) & 1, abort_flag)) return false;
      tc_fence_after();
      {
        const uint64_t qd = sdesc_sw128(smem_u32(sQ + st * L::kTileQ), 16, 1024);
        const uint64_t dod = sdesc_sw128(smem_u32(sDO + st * L::kTileQ), 16, 1024);
        const uint32_t b = (uint32_t)(it & 1);
        // S^T and dP^T are independent accumulators: interleave them per K step
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off_kv = (kk >> 2) * L::kChunkKV + (kk & 3) * 32;
          const uint32_t off_q = (kk >> 2) * L::kChunkQ + (kk & 3) * 32;
          mma_ss_w(tbase + kColS + b * BMQ, sdesc_add(kd_k, off_kv), sdesc_add(qd, off_q), id_s, kk > 0 ? 1u : 0u);
          // A = V from TMEM: 16 features of every key = 8 columns
          mma_ts_w(tbase + kColDP, tbase + kColV + kk * 8, sdesc_add(dod, off_q), id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&s_full[b]);
      }
      __syncwarp();
      return true;
    };
    if (warp == 1) {
      bool ok = mbar_wait_warp(kv_full, 0, abort_flag) && mbar_wait_warp(v_full, 0, abort_flag);
      for (int it = 0; ok && it < n_it; ++it) ok = issue_scores(it);
      mma_commit_w(drain_s);
      mbar_wait(drain_s, 0, nullptr);
    } else {
      bool ok = mbar_wait_warp(kv_full, 0, abort_flag);
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it % NSTAGE;
        const uint32_t b = (uint32_t)(it & 1);
        if (!mbar_wait_warp(&p_full[b], (it >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        {
          // B = dO_it / Q_it as MN-major: 16 queries per step (2048 B), 64-feature
          // chunks L::kChunkQ apart.
          const uint64_t dod = sdesc_sw128(smem_u32(sDO + st * L::kTileQ), L::kChunkQ, 1024);
          const uint64_t qd = sdesc_sw128(smem_u32(sQ + st * L::kTileQ), L::kChunkQ, 1024);
          const uint64_t dsd = sdesc_sw128(smem_u32(sDS), 8192, 1024);
          // dV first (it reads P^T from S buffer b), then dQ^T into S buffer b, then
          // dK: the dQ^T readout overlaps dK, so the next scores into buffer b
          // wait less.  dK reads the dS^T tile in shared memory (K-major A).
  #pragma unroll
          for (int kk = 0; kk < BMQ / 16; ++kk)
            mma_ts_w(tbase + kColDV, tbase + kColS + b * BMQ + packed_col(kk), sdesc_add(dod, kk * 2048), id_g,
                     (it > 0 || kk > 0) ? 1u : 0u);
          // dQ^T and dK read the dS^T tile in shared memory
          if (!mbar_wait_warp(&ds_full[b], (it >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          // dQ^T = K^T dS^T into S buffer b: A = K (MN-major, 64-feature chunks
          // L::kChunkKV apart), B = dS^T ([key][query] rows of 128 B); 16 keys per step.
  #pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ss_w(tbase + kColS + b * BMQ, sdesc_add(kd_mn, kk * 2048), sdesc_add(dsd, kk * 2048), id_q,
                     kk > 0 ? 1u : 0u);
          mma_commit_w(&dq_full[b]);
  #pragma unroll
          for (int kk = 0; kk < BMQ / 16; ++kk)
            mma_ss_w(tbase + kColDK, sdesc_add(dsd_k, kk * 32), sdesc_add(qd, kk * 2048), id_g,
                     (it > 0 || kk > 0) ? 1u : 0u);
          mma_commit_w(dsm_free);
          mma_commit_w(&dk_done[st]);
        }
        __syncwarp();
      }
      mma_commit_w(fin);
      mma_commit_w(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ dQ flusher
    // Tile x's dQ rows sit in its (consumed) Q buffer (rows 0-31) and dO
    // buffer (rows 32-63); add them into dQ with bulk reductions, then hand
    // the stage back to the producer once the reads are done.
    if (lane == 0) {
      for (int x = 0; x < n_it; ++x) {
        const int st = x % NSTAGE;
        if (!mbar_wait(&stg_full[st], (x / NSTAGE) & 1, abort_flag)) break;
        const int n = kvh * G + x / n_qb;
        const int64_t q0 = q_lo + (int64_t)(x % n_qb) * BMQ;
        const int64_t rows = S - q0 < BMQ ? S - q0 : BMQ;
        const int64_t n_q = (int64_t)gridDim.x * G;
        if (!in_bounds(q0, S) || (!seq && !in_bounds(((int64_t)n * S + q0 + rows) * D - 1, n_q * S * D))) {
          // checked build only: skip the reduce, keep the pipeline going
        } else if (seq) {
          // rows of one head are H_q D apart in the sequence layout: tensor
          // reduce-adds of 32-row boxes (rows past S are dropped)
          tma_reduce_add_3d(&tmDQ, sQ + st * L::kTileQ, 0, n, (int)q0);
          if (rows > 32) tma_reduce_add_3d(&tmDQ, sDO + st * L::kTileQ, 0, n, (int)q0 + 32);
        } else {
          float* dst = dq + ((int64_t)n * S + q0) * D;
          // 8-row (4 KB) pieces: with more, smaller reductions in flight the
          // tile's dQ reaches L2 sooner than as two 16 KB pieces (measured)
#pragma unroll 1
          for (int r0 = 0; r0 < rows; r0 += 8) {
            const int64_t nr = rows - r0 < 8 ? rows - r0 : 8;
            const uint8_t* src = (r0 < 32 ? sQ : sDO) + st * L::kTileQ + (r0 & 31) * D * 4;
            bulk_reduce_add_f32(dst + (int64_t)r0 * D, src, (uint32_t)(nr * D * 4));
          }
        }
        bulk_commit();
        bulk_wait_read0();
        mbar_arrive(&q_empty[st]);
      }
      bulk_wait0();   // every dQ reduce has landed before the CTA retires
    }
    __syncwarp();
  } else if (warp < 4 + kReadWarps) {
    // ------------------------------------------------------------ dQ^T readout
    // Warp 4 + wq: TMEM lane quarter wq = features [32wq, 32wq+32).  dQ^T of
    // tile x (in S buffer x & 1) -> scale * dQ as [query][feature] fp32 rows in
    // tile x's consumed Q buffer (queries 0-31) and dO buffer (queries 32-63);
    // the flusher warp adds them into dQ.  Running beside the gradient warps,
    // this frees the S buffer for the next scores as early as possible.
    const int wq = warp & 3;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int d = wq * 32 + lane;
    {
      // V of this CTA's keys into TMEM columns [kColV, kColV + 64): thread =
      // key row (TMEM lane), column c = features 2c, 2c+1 (the row's bytes as
      // 32-bit words); rows past S are zero
      const int64_t jv = k0 + wq * 32 + lane;
      const int64_t vrow = seq ? jv * hkv_tot + kvh : (int64_t)kvh * S + jv;
      const bool have = jv < S && in_bounds(vrow * D + D - 1, (seq ? (int64_t)hkv_tot : (int64_t)gridDim.x) * S * D);
      const uint4* src = reinterpret_cast<const uint4*>(vptr + (have ? vrow : 0) * D);
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {     // 64 features (32 columns) at a time
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 a = have ? src[8 * half + e] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * e] = a.x; w[4 * e + 1] = a.y; w[4 * e + 2] = a.z; w[4 * e + 3] = a.w;
        }
        tmem_st32(tbase + lane_off + kColV + half * 32, w);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(v_full);
    }
    for (int x = 0; x < n_it; ++x) {
      const uint32_t bx = (uint32_t)(x & 1);
      const int sx = x % NSTAGE;
      if (!mbar_wait_warp(&dq_full[bx], (x >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32(tbase + lane_off + kColS + bx * BMQ, r0);
      tmem_ld32(tbase + lane_off + kColS + bx * BMQ + 32, r1);
      tmem_ld_wait();
      reg_fence(r0);
      reg_fence(r1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dq_empty[bx]);
      float* c0 = reinterpret_cast<float*>(sQ + sx * L::kTileQ) + d;
      float* c1 = reinterpret_cast<float*>(sDO + sx * L::kTileQ) + d;
      // queries 32-63 into the dO buffer (dV, which read it, is done) ...
#pragma unroll
      for (int c = 0; c < 32; ++c) c1[c * D] = __uint_as_float(r1[c]) * scale;
      // ... queries 0-31 into the Q buffer once dK has read it
      if (!mbar_wait_warp(&dk_done[sx], (x / NSTAGE) & 1, abort_flag)) break;
#pragma unroll
      for (int c = 0; c < 32; ++c) c0[c * D] = __uint_as_float(r0[c]) * scale;
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&stg_full[sx]);
    }
  } else {
    // ------------------------------------------------------------ gradient warps
    // Warp (8 + 4h + wq): TMEM lane quarter wq, query half h (columns
    // [32h, 32h+32) of the 64-query tile).  Thread = key row jr for P^T/dS^T
    // (TMEM lane wq*32 + lane).
    const int wq = warp & 3;
    const int h = (warp - 8) >> 2;
    const int jr = wq * 32 + lane;
    const int64_t j = k0 + jr;
    int64_t qlo = 0, qhi = 0;
    if (j < S) query_range(cu, nd, S, causal, j, qlo, qhi);
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float sl2 = scale * kLog2e;
    bool ok = true;

    for (int it = 0; it < n_it; ++it) {
      const int st = it % NSTAGE;
      const uint32_t round = it / NSTAGE;
      const uint32_t b = (uint32_t)(it & 1);
      const int64_t q0 = q_lo + (int64_t)(it % n_qb) * BMQ + h * 32;   // this half's first query
      if (!mbar_wait_warp(&q_full[st], round & 1, abort_flag)) { ok = false; break; }
      if (!mbar_wait_warp(&s_full[b], (it >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const float* stat = sStat + st * 2 * BMQ + h * 32;
      // this row's queries as columns [clo, chi) of the half
      const int64_t dlo = qlo - q0, dhi = qhi - q0;
      const int clo = dlo <= 0 ? 0 : (dlo >= 32 ? 32 : (int)dlo);
      const int chi = dhi <= 0 ? 0 : (dhi >= 32 ? 32 : (int)dhi);
      uint32_t sv[32], pv[32];
      tmem_ld32(tbase + lane_off + kColS + b * BMQ + h * 32, sv);
      tmem_ld32(tbase + lane_off + kColDP + h * 32, pv);
      tmem_ld_wait();
      reg_fence(sv);
      reg_fence(pv);
      // dP^T is in registers: the next tile's dP^T may overwrite its buffer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dp_free);
      uint32_t pp[16], dd[16];
      // P^T = 2^(s * scale * log2 e - LSE_i log2 e), dS^T = P^T (dP^T - D_i).
      // The mask test sits outside the loop so each version is one basic block
      // and the compiler can put all LSE / D_i loads in flight at once.
      auto grad_cols = [&](auto masked) {
#pragma unroll
        for (int col = 0; col < 32; col += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(stat + col);
          const float4 d4 = *reinterpret_cast<const float4*>(stat + BMQ + col);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
          const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
          float p[4], g[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            p[u] = ex2(fmaf(__uint_as_float(sv[col + u]), sl2, -lv[u]));
            if (decltype(masked)::value) p[u] = (col + u >= clo && col + u < chi) ? p[u] : 0.f;
            g[u] = p[u] * (__uint_as_float(pv[col + u]) - dl[u]);
          }
          pp[col >> 1] = pack_bf16(p[0], p[1]);
          pp[(col >> 1) + 1] = pack_bf16(p[2], p[3]);
          dd[col >> 1] = pack_bf16(g[0], g[1]);
          dd[(col >> 1) + 1] = pack_bf16(g[2], g[3]);
        }
      };
      if (clo == 0 && chi == 32)
        grad_cols(std::false_type{});
      else
        grad_cols(std::true_type{});
      // bf16 pairs: 16 columns per half, inside the half's own 32 columns
      tmem_st16(tbase + lane_off + kColS + b * BMQ + h * 32, pp);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
      // the dS^T tile in shared memory was last read by dQ^T_{it-1} and dK_{it-1}
      if (it >= 1 && !mbar_wait_warp(dsm_free, (it - 1) & 1, abort_flag)) { ok = false; break; }
      uint8_t* row = sDS + jr * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int lc = h * 4 + c;                 // logical 16-byte chunk of the 128-byte row
        uint4 w = make_uint4(dd[4 * c], dd[4 * c + 1], dd[4 * c + 2], dd[4 * c + 3]);
        *reinterpret_cast<uint4*>(row + ((lc ^ (jr & 7)) << 4)) = w;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full[b]);
    }
    // epilogue: half 0 writes dV, half 1 writes scale * dK of this key block
    if (ok && n_it > 0 && mbar_wait_warp(fin, 0, abort_flag)) {
      tc_fence_after();
      float* dst = (h == 0 ? dv : dk) + (seq ? (int64_t)j * hkv_tot + kvh : (int64_t)kvh * S + j) * D;
      const float mul = h == 0 ? 1.f : scale;
      const uint32_t col0 = h == 0 ? kColDV : kColDK;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tbase + lane_off + col0 + c * 32, r);
        tmem_ld_wait();
        reg_fence(r);
        const int64_t kv_elems = (seq ? (int64_t)hkv_tot : (int64_t)gridDim.x) * S * D;
        if (j < S && in_bounds((dst - (h == 0 ? dv : dk)) + c * 32 + 31, kv_elems)) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + c * 32 + e) =
                make_float4(__uint_as_float(r[e]) * mul, __uint_as_float(r[e + 1]) * mul,
                            __uint_as_float(r[e + 2]) * mul, __uint_as_float(r[e + 3]) * mul);
        }
      }
    } else if (n_it == 0 && j < S) {
      // no query sees these keys: zero gradients
      float* dst = (h == 0 ? dv : dk) + (seq ? (int64_t)j * hkv_tot + kvh : (int64_t)kvh * S + j) * D;
      for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

bool tc_bwd_supported(const AttnArgs& a) {
  return a.dtype == ULYSSES_BF16 && a.D == 128 && a.S >= BN && (a.S + BN - 1) / BN <= 65535;
}

int launch_tc_bwd(const AttnArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.n_q * a.S;
  bwd_pre_kernel<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(
      (const __nv_bfloat16*)a.o, (const __nv_bfloat16*)a.dO, a.delta, a.dq, rows, a.S, a.seq, a.hq_tot);
  count_launch();
  int rc = check_launch("bwd_pre");
  if (rc) return rc;
  CUtensorMap tq, tk, tv, tdo, tdq;
  const int n_kv = a.n_q / a.G;
  if (a.seq) {
    if ((rc = make_tmap_bf16_seq(&tq, a.q, a.S, a.n_q, a.hq_tot, D, BMQ))) return rc;
    if ((rc = make_tmap_bf16_seq(&tdo, a.dO, a.S, a.n_q, a.hq_tot, D, BMQ))) return rc;
    if ((rc = make_tmap_bf16_seq(&tk, a.k, a.S, n_kv, a.hkv_tot, D, BN))) return rc;
    if ((rc = make_tmap_bf16_seq(&tv, a.v, a.S, n_kv, a.hkv_tot, D, BN))) return rc;
    if ((rc = make_tmap_f32_seq(&tdq, a.dq, a.S, a.n_q, a.hq_tot, D, 32))) return rc;
  } else {
    if ((rc = make_tmap_bf16_3d(&tq, a.q, a.S, a.n_q, D, BMQ))) return rc;
    if ((rc = make_tmap_bf16_3d(&tdo, a.dO, a.S, a.n_q, D, BMQ))) return rc;
    if ((rc = make_tmap_bf16_3d(&tk, a.k, a.S, n_kv, D, BN))) return rc;
    if ((rc = make_tmap_bf16_3d(&tv, a.v, a.S, n_kv, D, BN))) return rc;
    tdq = tq;   // not read in the head layout
  }
  const int smem = BwdLayout::kAlloc;
  static PerDeviceOnce<> smem_once;
  if ((rc = opt_in_smem(smem_once, (const void*)tc_bwd_kernel, smem, "tc_bwd"))) return rc;
  dim3 grid((unsigned)n_kv, (unsigned)((a.S + BN - 1) / BN));
  tc_bwd_kernel<<<grid, kThreads, smem, st>>>(tq, tk, tv, tdo, a.lse_in, a.delta, a.dq, a.dk, a.dv,
                                              a.S, a.nq, a.G, a.lse_bstride, a.cu, a.nd, a.causal,
                                              a.scale, tdq, a.seq, a.hkv_tot, (const __nv_bfloat16*)a.v);
  count_launch();
  return check_launch("tc_bwd");
}

}  // namespace ulysses
