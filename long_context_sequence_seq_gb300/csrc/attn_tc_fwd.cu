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
//   warp 0      TMA producer: Q once, then K_j / V_j tiles into a 4-slot ring
//   warp 1      TMEM owner and MMA issuer (one elected lane):
//                 S_j = Q K_j^T      (tcgen05.mma, SS, fp32 accumulate in TMEM)
//                 O  += P_j V_j      (tcgen05.mma, A = P from TMEM as bf16)
//   warps 4-7   softmax: one thread per query row (TMEM lane), reads S_j with
//               tcgen05.ld, masks, exponentiates (ex2), writes P_j over S_j as
//               bf16, rescales O in TMEM when the running max grows, and runs
//               the epilogue (O/l to global memory, LSE).
// S is double-buffered in TMEM, so Q K_{j+1}^T runs on the tensor pipe while
// the softmax warps work on tile j.
//
// TMEM columns (512 allocated): S/P buffer 0 [0,128), buffer 1 [128,256),
// O accumulator [256, 256+D).
// Shared memory: Q tile (D/64 swizzle-128B chunks of 128 rows) + a ring of
// four 128 x D tiles holding K and V in load order K0 V0 K1 V1 ...
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
constexpr int NSLOT = 4;     // K/V ring slots
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdLayout {
  static constexpr int kChunkQ = BM * 128;            // one 64-column swizzled chunk of Q
  static constexpr int kChunkKV = BN * 128;           // one 64-column chunk of a K/V tile
  static constexpr int kTileQ = kChunkQ * (D / 64);
  static constexpr int kTileKV = kChunkKV * (D / 64);
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + kTileQ;
  static constexpr int kBar = kKV + NSLOT * kTileKV;
  // q_full, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2], o_done, drain
  static constexpr int kNumBar = 1 + 2 * NSLOT + 2 + 2 + 1 + 1;
  static constexpr int kMisc = kBar + kNumBar * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;        // slack for 1024-byte alignment
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ out,
                  float* __restrict__ lse, int64_t S, int nq, int G, int64_t lse_bstride,
                  const int32_t* __restrict__ cu, int nd, int causal, float sl2) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sKV = smem + L::kKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + NSLOT;
  uint64_t* s_full = kv_empty + NSLOT;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x;                            // q head in the buffer
  const int qt = gridDim.y - 1 - blockIdx.y;           // heaviest tiles first
  const int64_t q0 = (int64_t)qt * BM;
  const int kvh = n / G;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NSLOT; ++s) { mbar_init(&kv_full[s], 1); mbar_init(&kv_empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&s_full[b], 1); mbar_init(&p_full[b], 4); }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
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
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

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
      for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * L::kChunkQ, &tmQ, c * 64, (int)q0, n, q_full);
      for (int idx = 0; idx < 2 * n_kv; ++idx) {
        const int j = idx >> 1, slot = idx % NSLOT;
        const uint32_t round = idx / NSLOT;
        if (!mbar_wait(&kv_empty[slot], (round & 1) ^ 1, abort_flag)) break;
        mbar_expect_tx(&kv_full[slot], L::kTileKV);
        const int k0 = (int)(kv_lo + (int64_t)j * BN);
        uint8_t* dst = sKV + slot * L::kTileKV;
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(dst + c * L::kChunkKV, (idx & 1) ? &tmV : &tmK, c * 64, k0, kvh, &kv_full[slot]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16(BM, D, false, true);
    const uint32_t q_addr = smem_u32(sQ);
    bool ok = mbar_wait(q_full, 0, abort_flag);

    const uint64_t qdesc = sdesc_sw128(q_addr, 16, 1024);
    auto issue_qk = [&](int j) -> bool {
      const int idx = 2 * j, slot = idx % NSLOT;
      const uint32_t round = idx / NSLOT;
      if (!mbar_wait(&kv_full[slot], round & 1, abort_flag)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t kdesc = sdesc_sw128(smem_u32(sKV + slot * L::kTileKV), 16, 1024);
        const uint32_t d_tmem = tbase + (uint32_t)(j & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major: 16 features = 32 bytes along the swizzled row, 64-feature chunks apart
          const uint32_t off = (kk >> 2) * L::kChunkQ + (kk & 3) * 32;
          const uint32_t offk = (kk >> 2) * L::kChunkKV + (kk & 3) * 32;
          mma_ss(d_tmem, sdesc_add(qdesc, off), sdesc_add(kdesc, offk), idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[j & 1]);
        mma_commit(&kv_empty[slot]);
      }
      __syncwarp();
      return true;
    };

    if (ok && n_kv > 0) ok = issue_qk(0);
    for (int j = 0; ok && j < n_kv; ++j) {
      if (j + 1 < n_kv && !issue_qk(j + 1)) { ok = false; break; }
      if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag)) { ok = false; break; }
      const int idx = 2 * j + 1, slot = idx % NSLOT;
      const uint32_t round = idx / NSLOT;
      if (!mbar_wait(&kv_full[slot], round & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
        // V as the MN-major B operand: 16 keys = two 8-row groups (1024 B apart),
        // 64-wide D chunks L::kChunkKV apart.
        const uint64_t vdesc = sdesc_sw128(smem_u32(sKV + slot * L::kTileKV), L::kChunkKV, 1024);
        const uint32_t p_tmem = tbase + (uint32_t)(j & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tbase + 256, p_tmem + kk * 8, sdesc_add(vdesc, kk * 2048), idesc_pv,
                 (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(o_done);
        mma_commit(&kv_empty[slot]);
      }
      __syncwarp();
    }
    // drain: nothing of ours may still be in flight at teardown
    if (lane == 0) mma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, nullptr);
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
      if (!mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sbuf = tbase + lane_off + (uint32_t)(j & 1) * BN;
      uint32_t sv[BN / 32][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(sbuf + c * 32, sv[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) reg_fence(sv[c]);
      const int64_t k0 = kv_lo + (int64_t)j * BN;
      float mt = -INFINITY;
      if (k0 >= lo && k0 + BN <= hi) {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) mt = fmaxf(mt, __uint_as_float(sv[c][e]));
      } else {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int64_t kj = k0 + c * 32 + e;
            const float x = (kj >= lo && kj < hi) ? __uint_as_float(sv[c][e]) : -INFINITY;
            sv[c][e] = __float_as_uint(x);
            mt = fmaxf(mt, x);
          }
      }
      const float m_new = fmaxf(m, mt * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m - m_use);
      float rs = 0.f;
      uint32_t pk[BN / 64][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(sv[c][e]), sl2, -m_use));
          const float p1 = ex2(fmaf(__uint_as_float(sv[c][e + 1]), sl2, -m_use));
          rs += p0 + p1;
          pk[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_bf16(p0, p1);
        }
      l = l * alpha + rs;
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) tmem_st32(sbuf + c * 32, pk[c]);
      if (j > 0) {
        // O must hold PV_{j-1} before it is rescaled for tile j
        if (!mbar_wait(o_done, (j - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tbase + lane_off + 256 + c * 32, ov);
            tmem_ld_wait();
            reg_fence(ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tbase + lane_off + 256 + c * 32, ov);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[j & 1]);
      m = m_new;
    }
    if (ok && n_kv > 0 && mbar_wait(o_done, (n_kv - 1) & 1, abort_flag)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tbase + lane_off + 256 + c * 32, ov);
        tmem_ld_wait();
        reg_fence(ov);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out + ((int64_t)n * S + i) * D + c * 32);
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
      if (valid) lse[lse_index(n, nq, lse_bstride, S, i)] = (m + __log2f(l)) * kLn2;
    }
  }
  // warps 2-3 have no role in this version

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <int D>
int launch_fwd_d(const AttnArgs& a, cudaStream_t st) {
  CUtensorMap tq, tk, tv;
  const int n_kv = a.n_q / a.G;
  int rc;
  if ((rc = make_tmap_bf16_3d(&tq, a.q, a.S, a.n_q, D, BM))) return rc;
  if ((rc = make_tmap_bf16_3d(&tk, a.k, a.S, n_kv, D, BN))) return rc;
  if ((rc = make_tmap_bf16_3d(&tv, a.v, a.S, n_kv, D, BN))) return rc;
  const int smem = FwdLayout<D>::kAlloc;
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(tc_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    attr_set = true;
  }
  const int64_t n_qt = (a.S + BM - 1) / BM;
  dim3 grid((unsigned)a.n_q, (unsigned)n_qt);
  tc_fwd_kernel<D><<<grid, kThreads, smem, st>>>(tq, tk, tv, (__nv_bfloat16*)a.o_out, a.lse, a.S,
                                                 a.nq, a.G, a.lse_bstride, a.cu, a.nd, a.causal,
                                                 a.scale * kLog2e);
  count_launch();
  return check_launch("tc_fwd");
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
