// K2: causal / document-masked GQA attention forward for sm_103a.
//
// Computes step 4 of "How Ulysses sequence parallelism works" (local dense
// attention over all S positions for the rank's heads) as exact softmax
// attention with an online softmax (the FlashAttention family the page names
// for long sequences: O(n) memory, O(n^2) FLOPs):
//   s_ij = scale q_i.k_j (masked to the row's key range), in log2 units
//   m'   = max(m, max_j s_ij),  l' = l 2^{m-m'} + sum_j 2^{s_ij-m'}
//   O'   = O 2^{m-m'} + sum_j 2^{s_ij-m'} v_j,   O_i = O/l,  LSE_i = (m + log2 l) ln 2
//
// One CTA per (q head, 128-row query tile); warp roles:
//   warp 0      TMA producer: Q once, then K_j into a 3-slot K ring and V_j
//               into a 3-slot V ring, K one tile ahead (K0 K1 V0 K2 V1 ...)
//   warp 1      TMEM owner; issues S_j = Q K_j^T (tcgen05.mma SS, fp32 in TMEM)
//   warp 2      issues O += P_j V_j (tcgen05.mma, A = P from TMEM as bf16)
//   warps 4-7   softmax: one thread per query row (TMEM lane), reads S_j with
//               tcgen05.ld, masks, exponentiates (ex2), writes P_j over S_j as
//               bf16, rescales O in TMEM when the running max has grown by more
//               than 2^8, and runs the epilogue (O/l to global memory, LSE).
// The MMA warps run their issue code warp-wide and let one elected lane issue
// (a lane-0 branch makes the issuing thread, not the tensor pipe, the limit).
// S is triple-buffered in TMEM, so QK_{j+1} and QK_{j+2} can run on the tensor
// pipe while the softmax works on tile j, and PV_j overlaps softmax j+1.
//
// Two CTAs of q heads that share a kv head (same query tile) form a cluster:
// they read the same K/V tiles, so each CTA loads half of a tile's rows and
// multicasts them into both CTAs' slot, and a slot is refilled once both
// CTAs' QK_j (K) or PV_j (V) have completed (commits multicast to both empty
// barriers).  This halves the K/V reads from L2 and keeps the pair on the
// same keys, which matters once K/V outgrow L2 (million-token stages).
// Clusters of four would quarter them, but only 36 such clusters fit on the
// GPU at once (144 of 152 SMs), which costs more than it saves.
//
// TMEM columns (512 allocated): S/P buffers [0,128), [128,256), [256,384);
// O accumulator [384, 384+D).
// Shared memory: Q tile (D/64 swizzle-128B chunks of 128 rows) + the K ring
// and the V ring, three 128 x D tiles each (224 KB in all for D = 128).
//
// Masks: row i sees keys [lo_i, hi_i) = [start of its document, i+1) (causal)
// or the whole document; a CTA walks keys from its first row's document start
// up to its last row's bound, masking element-wise only in tiles that cross a
// row's bound.  Later query tiles have more key tiles, so the grid is ordered
// heaviest-first (longest-processing-time order) for the causal case.
#include "internal.h"
#include "tc_ptx.cuh"

namespace ulysses {

ULYSSES_ERROR_READER(read_error_attn_tc_fwd)

namespace {

using namespace tc;

constexpr int BM = 128;      // query rows per CTA
constexpr int BN = 128;      // keys per tile
constexpr int NRING = 3;     // slots in each of the K ring and the V ring
constexpr int NSLOT = 2 * NRING;
constexpr int NSBUF = 3;     // S/P buffers in TMEM (QK runs two tiles ahead)
constexpr uint32_t kColO = NSBUF * BN;   // O accumulator columns [kColO, kColO + D)
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;   // lazy-rescale threshold (log2 units)

template <int D>
struct FwdLayout {
  static constexpr int kChunkQ = BM * 128;            // one 64-column swizzled chunk of Q
  static constexpr int kChunkKV = BN * 128;           // one 64-column chunk of a K/V tile
  static constexpr int kTileQ = kChunkQ * (D / 64);
  static constexpr int kTileKV = kChunkKV * (D / 64);
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + kTileQ;
  static constexpr int kBar = kKV + NSLOT * kTileKV;
  // q_full, k_full/v_full[NRING], k_empty/v_empty[NRING], s_full[NSBUF], p_full[NSBUF], drain[2],
  // v_free[NRING]
  static constexpr int kNumBar = 1 + 4 * NRING + 2 * NSBUF + 2 + NRING;
  static constexpr int kMisc = kBar + kNumBar * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;        // slack for 1024-byte alignment
};

template <int D, int CL>
__global__ void __launch_bounds__(kThreads, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ out,
                  float* __restrict__ lse, int64_t S, int nq, int G, int64_t lse_bstride,
                  const int32_t* __restrict__ cu, int nd, int causal, float sl2, int seq, int hq_tot) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sKV = smem + L::kKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NRING;
  uint64_t* k_empty = v_full + NRING;
  // v_empty[j % NRING] completes when PV_j has run: it frees V_j's slot and
  // also tells the softmax that O holds PV_j (so it may rescale or read O)
  uint64_t* v_empty = k_empty + NRING;
  uint64_t* s_full = v_empty + NRING;
  uint64_t* p_full = s_full + NSBUF;
  uint64_t* drain = p_full + NSBUF;
  // with a cluster: v_free[j % NRING] completes when PV_j has run in every CTA
  // of the cluster (the V slot may be refilled); k_empty counts every CTA's QK_j
  uint64_t* v_free = drain + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x;                            // q head in the buffer
  const int qt = gridDim.y - 1 - blockIdx.y;           // heaviest tiles first
  const int64_t q0 = (int64_t)qt * BM;
  const int kvh = n / G;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2 * NRING; ++s) mbar_init(&k_full[s], 1);          // k/v full
    for (int s = 0; s < NRING; ++s) mbar_init(&k_empty[s], CL);             // every CTA's QK_j
    for (int s = 0; s < NRING; ++s) mbar_init(&v_empty[s], 1);              // this CTA's PV_j
    for (int s = 0; s < NRING; ++s) mbar_init(&v_free[s], CL);              // every CTA's PV_j
    for (int b = 0; b < NSBUF; ++b) { mbar_init(&s_full[b], 1); mbar_init(&p_full[b], 4); }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmQ);
    tma_prefetch(&tmK);
    tma_prefetch(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // the cluster's barriers are initialised before any CTA loads into or
  // arrives on another's
  if constexpr (CL > 1) cluster_sync();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t crank = CL > 1 ? cluster_ctarank() : 0u;
  constexpr uint16_t kMask = (uint16_t)((1u << CL) - 1u);

  // Key tiles of this CTA: [kv_lo, kv_hi) in steps of BN.
  const int64_t last_row = (q0 + BM < S ? q0 + BM : S) - 1;
  int64_t kv_lo, kv_hi, tmp;
  key_range(cu, nd, S, causal, q0, kv_lo, tmp);
  key_range(cu, nd, S, causal, last_row, tmp, kv_hi);
  const int n_kv = kv_hi > kv_lo ? (int)((kv_hi - kv_lo + BN - 1) / BN) : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_expect_tx(q_full, L::kTileQ);
      // head layout: (feature, row, head); sequence layout: (feature, head, row)
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sQ + c * L::kChunkQ, &tmQ, c * 64, seq ? n : (int)q0, seq ? (int)q0 : n, q_full);
      // K tiles into the K ring (slot freed by QK_j), V tiles into the V ring
      // (freed by PV_j); K runs one tile ahead: K0 K1 V0 K2 V1 ...
      bool go = true;
      for (int t = 0; go && t <= n_kv; ++t)
        for (int kv = 0; kv < 2; ++kv) {
          const int j = kv ? t - 1 : t;
          if (j < 0 || j >= n_kv) continue;
          const int r = j % NRING;
          uint64_t* empty = kv ? (CL > 1 ? &v_free[r] : &v_empty[r]) : &k_empty[r];
          uint64_t* full = kv ? &v_full[r] : &k_full[r];
          if (!mbar_wait(empty, ((uint32_t)(j / NRING) & 1u) ^ 1u, abort_flag)) { go = false; break; }
          mbar_expect_tx(full, L::kTileKV);
          const int k0 = (int)(kv_lo + (int64_t)j * BN);
          uint8_t* dst = sKV + (kv * NRING + r) * L::kTileKV;
          if constexpr (CL > 1) {
            // this CTA's share of the tile: rows [crank BN/CL, (crank+1) BN/CL),
            // multicast into the same slot of every CTA of the cluster
            const int kr = k0 + (int)crank * (BN / CL);
            uint8_t* part = dst + crank * (BN / CL) * 128;
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d_mc(part + c * L::kChunkKV, kv ? &tmV : &tmK, c * 64, seq ? kvh : kr, seq ? kr : kvh, full,
                             kMask);
          } else {
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(dst + c * L::kChunkKV, kv ? &tmV : &tmK, c * 64, seq ? kvh : k0, seq ? k0 : kvh, full);
          }
        }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Two issuing warps keep the tensor pipe fed: warp 1 issues S_j = Q K_j^T,
    // warp 2 issues O += P_j V_j.  The whole warp runs the issue code
    // (warp-uniform operands); the *_w helpers let one elected lane issue.
    // MMAs of different warps are not ordered with respect to each other, so
    // every cross-warp dependency goes through an mbarrier:
    //   QK_j   waits K_j loaded, and (j >= NSBUF) v_empty of PV_{j-NSBUF}: the
    //          S/P buffer it overwrites has been read by that PV;
    //   PV_j   waits P_j written (p_full) and V_j loaded; PV_j after PV_{j-1}
    //          on O is ordered by issue order within warp 2.
    // S is NSBUF-buffered, so QK runs up to NSBUF - 1 tiles ahead of the softmax.
    bool ok = mbar_wait_warp(q_full, 0, abort_flag);
    if (warp == 1) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, false, false);
      const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int slot = j % NRING;
        if (j >= NSBUF &&
            !mbar_wait_warp(&v_empty[(j - NSBUF) % NRING], ((j - NSBUF) / NRING) & 1, abort_flag)) {
          ok = false;
          break;
        }
        if (!mbar_wait_warp(&k_full[slot], (j / NRING) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kdesc = sdesc_sw128(smem_u32(sKV + slot * L::kTileKV), 16, 1024);
        const uint32_t d_tmem = tbase + (uint32_t)(j % NSBUF) * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major: 16 features = 32 bytes along the swizzled row, 64-feature chunks apart
          const uint32_t off = (kk >> 2) * L::kChunkQ + (kk & 3) * 32;
          const uint32_t offk = (kk >> 2) * L::kChunkKV + (kk & 3) * 32;
          mma_ss_w(d_tmem, sdesc_add(qdesc, off), sdesc_add(kdesc, offk), idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&s_full[j % NSBUF]);
        if constexpr (CL > 1) mma_commit_mc_w(&k_empty[slot], kMask);
        else mma_commit_w(&k_empty[slot]);
      }
      // drain: nothing of ours may still be in flight at teardown
      mma_commit_w(&drain[0]);
      mbar_wait(&drain[0], 0, nullptr);
    } else {
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, false, true);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int r = j % NRING;
        if (!mbar_wait_warp(&p_full[j % NSBUF], (j / NSBUF) & 1, abort_flag)) { ok = false; break; }
        if (!mbar_wait_warp(&v_full[r], (j / NRING) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        // V as the MN-major B operand: 16 keys = two 8-row groups (1024 B apart),
        // 64-wide D chunks L::kChunkKV apart.
        const uint64_t vdesc = sdesc_sw128(smem_u32(sKV + (NRING + r) * L::kTileKV), L::kChunkKV, 1024);
        const uint32_t p_tmem = tbase + (uint32_t)(j % NSBUF) * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts_w(tbase + kColO, p_tmem + kk * 8, sdesc_add(vdesc, kk * 2048), idesc_pv,
                   (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(&v_empty[r]);
        if constexpr (CL > 1) mma_commit_mc_w(&v_free[r], kMask);
      }
      mma_commit_w(&drain[1]);
      mbar_wait(&drain[1], 0, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int64_t i = q0 + r;
    const bool valid = i < S;
    int64_t lo = 0, hi = 0;
    if (valid) key_range(cu, nd, S, causal, i, lo, hi);
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!mbar_wait_warp(&s_full[j % NSBUF], (j / NSBUF) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sbuf = tbase + lane_off + (uint32_t)(j % NSBUF) * BN;
      uint32_t sv[BN / 32][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(sbuf + c * 32, sv[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) reg_fence(sv[c]);
      // the row's keys as columns [clo, chi) of this tile
      const int64_t k0 = kv_lo + (int64_t)j * BN;
      const int64_t dlo = lo - k0, dhi = hi - k0;
      const int clo = dlo <= 0 ? 0 : (dlo >= BN ? BN : (int)dlo);
      const int chi = dhi <= 0 ? 0 : (dhi >= BN ? BN : (int)dhi);
      if (!(clo == 0 && chi == BN)) {     // the tile crosses this row's key bounds
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = c * 32 + e;
            if (col < clo || col >= chi) sv[c][e] = __float_as_uint(-INFINITY);
          }
      }
      // row max over the tile: three-input max, four independent partial maxima
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float& q = mx[(e >> 3) & 3];
          q = max3f(q, __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
          q = max3f(q, __uint_as_float(sv[c][e + 2]), __uint_as_float(sv[c][e + 3]));
          q = max3f(q, __uint_as_float(sv[c][e + 4]), __uint_as_float(sv[c][e + 5]));
          q = max3f(q, __uint_as_float(sv[c][e + 6]), __uint_as_float(sv[c][e + 7]));
        }
      const float mt = fmaxf(max3f(mx[0], mx[1], mx[2]), mx[3]);
      // lazy rescale: keep the running max until a row's max grows by more
      // than 2^kRescaleLog2 (it is only a stabiliser: O = acc / l and
      // LSE = (m + log2 l) ln 2 stay exact for any m, and P stays <= 2^8)
      const float m_cand = fmaxf(m, mt * sl2);
      const bool upd = m_cand > m + kRescaleLog2;       // also true when m is still -inf
      const float m_next = upd ? m_cand : m;
      const float m_use = (m_next == -INFINITY) ? 0.f : m_next;
      const float alpha = upd ? ex2(m - m_use) : 1.f;
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[BN / 64][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float a0, a1;
          fma2f(a0, a1, __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]), sl2, -m_use);
          const float p0 = ex2(a0), p1 = ex2(a1);
          rs[(e >> 1) & 3] += p0 + p1;
          pk[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_bf16(p0, p1);
        }
      l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) tmem_st32(sbuf + c * 32, pk[c]);
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O must hold PV_{j-1} before this warp rescales its rows.  A warp
        // that keeps its max does not touch O and need not wait: PV_j comes
        // after PV_{j-1} in issue order, and PV_j waits for every warp's P_j.
        // The wait cannot alias an older phase: PV_{j-1+NRING} needs this
        // warp's P for tile j-1+NRING.
        if (!mbar_wait_warp(&v_empty[(j - 1) % NRING], ((j - 1) / NRING) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tbase + lane_off + kColO + c * 32, ov);
          tmem_ld_wait();
          reg_fence(ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(tbase + lane_off + kColO + c * 32, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[j % NSBUF]);
      m = m_next;
    }
    if (ok && n_kv > 0 && mbar_wait_warp(&v_empty[(n_kv - 1) % NRING], ((n_kv - 1) / NRING) & 1, abort_flag)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tbase + lane_off + kColO + c * 32, ov);
        tmem_ld_wait();
        reg_fence(ov);
        const int64_t row = seq ? (int64_t)i * hq_tot + n : (int64_t)n * S + i;
        if (valid && in_bounds(row * D + c * 32 + 31, (seq ? (int64_t)hq_tot : (int64_t)gridDim.x) * S * D)) {
          uint4* dst = reinterpret_cast<uint4*>(out + row * D + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(ov[8 * e + 0]) * inv, __uint_as_float(ov[8 * e + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(ov[8 * e + 2]) * inv, __uint_as_float(ov[8 * e + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(ov[8 * e + 4]) * inv, __uint_as_float(ov[8 * e + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(ov[8 * e + 6]) * inv, __uint_as_float(ov[8 * e + 7]) * inv);
            dst[e] = w;
          }
        }
      }
      const int64_t li = lse_index(n, nq, lse_bstride, S, i);
      if (valid && in_bounds(li, ((int64_t)gridDim.x + nq - 1) / nq * lse_bstride)) lse[li] = (m + __log2f(l)) * kLn2;
    }
  }
  // warps 2-3 have no role in this version

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  // no CTA retires while another of its cluster may still address it
  if constexpr (CL > 1) cluster_sync();
}

// Cluster size: two CTAs of q heads that share a kv head (same query tile)
// share each K/V tile, each loading half of its rows and multicasting them to
// the other; one CTA without GQA.
inline int fwd_cluster(int G) { return G % 2 == 0 ? 2 : 1; }

template <int D, int CL>
int launch_fwd_dc(const AttnArgs& a, cudaStream_t st) {
  CUtensorMap tq, tk, tv;
  const int n_kv = a.n_q / a.G;
  int rc;
  if (a.seq) {
    if ((rc = make_tmap_bf16_seq(&tq, a.q, a.S, a.n_q, a.hq_tot, D, BM))) return rc;
    if ((rc = make_tmap_bf16_seq(&tk, a.k, a.S, n_kv, a.hkv_tot, D, BN / CL))) return rc;
    if ((rc = make_tmap_bf16_seq(&tv, a.v, a.S, n_kv, a.hkv_tot, D, BN / CL))) return rc;
  } else {
    if ((rc = make_tmap_bf16_3d(&tq, a.q, a.S, a.n_q, D, BM))) return rc;
    if ((rc = make_tmap_bf16_3d(&tk, a.k, a.S, n_kv, D, BN / CL))) return rc;
    if ((rc = make_tmap_bf16_3d(&tv, a.v, a.S, n_kv, D, BN / CL))) return rc;
  }
  const int smem = FwdLayout<D>::kAlloc;
  static PerDeviceOnce<> smem_once;   // one per (head dim, cluster size) instance
  if ((rc = opt_in_smem(smem_once, (const void*)tc_fwd_kernel<D, CL>, smem, "tc_fwd"))) return rc;
  const int64_t n_qt = (a.S + BM - 1) / BM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_q, (unsigned)n_qt);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, tc_fwd_kernel<D, CL>, tq, tk, tv, (__nv_bfloat16*)a.o_out, a.lse,
                                           a.S, a.nq, a.G, a.lse_bstride, a.cu, a.nd, a.causal, a.scale * kLog2e,
                                           a.seq, a.hq_tot);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();   // the error is reported here, not left for the next call
    return set_error(ULYSSES_ERR_CUDA, "tc_fwd: cluster launch failed: %s", cudaGetErrorString(e));
  }
  count_launch();
  return check_launch("tc_fwd");
}

template <int D>
int launch_fwd_d(const AttnArgs& a, cudaStream_t st) {
  // the grid's x (q heads of the buffer) holds whole kv groups, so a cluster
  // along x never spans two kv heads
  return fwd_cluster(a.G) == 2 ? launch_fwd_dc<D, 2>(a, st) : launch_fwd_dc<D, 1>(a, st);
}

}  // namespace

bool tc_fwd_supported(const AttnArgs& a) {
  return a.dtype == ULYSSES_BF16 && (a.D == 64 || a.D == 128) && a.S >= BM &&
         (a.S + BM - 1) / BM <= 65535;
}

int launch_tc_fwd(const AttnArgs& a, cudaStream_t st) {
  return a.D == 128 ? launch_fwd_d<128>(a, st) : launch_fwd_d<64>(a, st);
}

}  // namespace ulysses
