// Deterministic dQ of the backward pass on sm_103a.
//
// One CTA owns 128 query rows of one (batch or sequence, head) and walks the key tiles those
// rows can see, in order:
//   S   = Q K_j^T,   dP = dO V_j^T                 (tcgen05, fp32 in TMEM)
//   P   = exp2(S c2 - LSE2),   dS = P (dP - Delta)  (compute warps, thread = query row)
//   dQ += dS K_j                                   (tcgen05, fp32 accumulator in TMEM)
// and stores dQ = sm_scale * acc once. Every element of dQ is a sum in a fixed order, with no
// atomics, so the result is the same on every run. The key-tile kernel of the backward pass
// runs without its dQ products in this mode (dK and dV are accumulated per key tile in TMEM
// and are deterministic there too); the price is that S and dP are computed twice.
//
// Warp roles (320 threads): warps 0..7 two compute warpgroups that split the 128 key columns
// of each step (thread = query row = TMEM lane); warp 8 TMA producer (Q, dO once, K/V ring);
// warp 9 MMA issuer (whole warp walks the schedule, one elected lane issues). S/dP of step
// j+1 are issued as soon as the compute warps have loaded those of step j. TMEM: S (128
// columns), dP (128), dQ (D). dS goes through shared memory as the K-major A operand.
#include <atomic>

#include "attn_common.cuh"
#include "attn_launch.h"

namespace attn_sm103 {

template <int D>
struct DqCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int NST = (D == 128) ? 2 : 3;  // K/V stages
  static constexpr int NDS = (D == 128) ? 1 : 2;  // dS buffers (shared memory budget)
  static constexpr int TILE = 128 * D * 2;        // one 128-row Q, dO, K or V tile
  static constexpr int DS_BYTES = BM * BN * 2;
  static constexpr int OFF_Q = 0, OFF_DO = TILE, OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_DS = OFF_V + NST * TILE;
  static constexpr int SMEM_BYTES = OFF_DS + NDS * DS_BYTES + 1024;
  static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DQ = 256, TMEM_COLS = 512;
  static constexpr int NTHREADS = 320;
  static constexpr int WARP_PRODUCER = 8, WARP_MMA = 9;
};

template <int NST, int NDS>
struct DqBars {
  uint64_t q_full;
  uint64_t k_full[NST], v_full[NST], kv_empty[NST];
  uint64_t s_full, s_free;
  uint64_t ds_full[NDS], ds_empty[NDS];
  uint64_t dq_full, mma_drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint8_t* align1024d(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, bool F16>
__global__ void __launch_bounds__(320, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdDqParams p) {
  using C = DqCfg<D>;
  constexpr int BM = C::BM, BN = C::BN, NST = C::NST, NDS = C::NDS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ DqBars<NST, NDS> bars;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 1-D grid over (unit, head) pairs x query blocks (grid_pos)
  const GridPos gp = grid_pos((int)blockIdx.x, p.tiles, (int)(gridDim.x / p.tiles), p.group);
  const int h = gp.zh % p.H, z = gp.zh / p.H;
  const int n_blk = p.tiles;
  const int m_blk = p.causal ? n_blk - 1 - gp.rank : gp.rank;  // causal: heaviest block first

  SeqView sv;
  if (!decode_seq(p.seq, z, threadIdx.x == 0 ? p.status : nullptr, sv)) return;
  const int q_lo = m_blk * BM;
  if (q_lo >= sv.len_q) return;
  const int q_hi = min(q_lo + BM, sv.len_q);
  int n_kt = (sv.len_k + BN - 1) / BN;
  if (p.causal) n_kt = min(n_kt, (q_hi - 1) / BN + 1);  // top-left: keys up to the last row
  const int64_t zh = (int64_t)sv.batch * p.H + h;

  if (n_kt <= 0) {  // no visible keys: dQ = 0 on the valid rows
    if (threadIdx.x < BM) {
      const int row = q_lo + threadIdx.x;
      if (row < sv.len_q) {
        uint16_t* dr = p.dq + sv.batch * p.dq_sb + h * p.dq_sh + (sv.row0_q + row) * p.dq_ss;
        for (int d = 0; d < p.d_out; d += 8) *reinterpret_cast<uint4*>(dr + d) = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }

  uint8_t* smem = align1024d(smem_raw);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
  const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
  const uint32_t sDS = smem_u32(smem + C::OFF_DS);

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(smem_u32(&bars.q_full), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars.s_full), 1);
    mbar_init(smem_u32(&bars.s_free), 256);
    for (int b = 0; b < NDS; ++b) {
      mbar_init(smem_u32(&bars.ds_full[b]), 256);
      mbar_init(smem_u32(&bars.ds_empty[b]), 1);
    }
    mbar_init(smem_u32(&bars.dq_full), 1);
    mbar_init(smem_u32(&bars.mma_drain), 1);
    mbar_fence_init();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(smem_u32(&bars.tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort = &bars.abort;

  if (warp == C::WARP_PRODUCER) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_do);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
      const uint32_t qb = smem_u32(&bars.q_full);
      mbar_arrive_expect_tx(qb, 2 * C::TILE);
#pragma unroll
      for (int s = 0; s < D / 64; ++s) {
        tma_load_4d(sQ + s * BM * 128, &p.tm_q, qb, s * 64, sv.row0_q + q_lo, h, sv.batch);
        tma_load_4d(sDO + s * BM * 128, &p.tm_do, qb, s * 64, sv.row0_q + q_lo, h, sv.batch);
      }
      int last_j[NST];  // last key tile loaded into each stage (-1: none)
#pragma unroll
      for (int st = 0; st < NST; ++st) last_j[st] = -1;
      for (int j = 0; j < n_kt; ++j) {
        const int st = j % NST;
        if (j >= NST &&
            !mbar_wait(smem_u32(&bars.kv_empty[st]), ((j / NST) - 1) & 1, abort, kWaitTimeoutNs))
          break;
        last_j[st] = j;
        const int krow = sv.row0_k + j * BN;
        const uint32_t kb = smem_u32(&bars.k_full[st]), vb = smem_u32(&bars.v_full[st]);
        mbar_arrive_expect_tx(kb, C::TILE);
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_4d(sK + st * C::TILE + s * BN * 128, &p.tm_k, kb, s * 64, krow, h, sv.batch);
        mbar_arrive_expect_tx(vb, C::TILE);
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_4d(sV + st * C::TILE + s * BN * 128, &p.tm_v, vb, s * 64, krow, h, sv.batch);
      }
      if (*abort) {  // the consumers gave up: let the copies in flight land before exiting
        mbar_wait_drain(qb, 0, kWaitTimeoutNs);
#pragma unroll
        for (int st = 0; st < NST; ++st)
          if (last_j[st] >= 0) {
            mbar_wait_drain(smem_u32(&bars.k_full[st]), (last_j[st] / NST) & 1, kWaitTimeoutNs);
            mbar_wait_drain(smem_u32(&bars.v_full[st]), (last_j[st] / NST) & 1, kWaitTimeoutNs);
          }
      }
    }
  } else if (warp == C::WARP_MMA) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = idesc_f32acc(128, BN, false, false, F16);  // S, dP (M = queries)
    constexpr uint32_t idQ = idesc_f32acc(128, D, false, true, F16);    // dQ: B = K, MN-major
    const uint32_t tS = tmem + C::COL_S, tDP = tmem + C::COL_DP, tDQ = tmem + C::COL_DQ;
    const uint64_t q_kd = desc_kmajor(sQ, BM, 0), do_kd = desc_kmajor(sDO, BM, 0);
    const uint64_t k_kd = desc_kmajor(sK, BN, 0), v_kd = desc_kmajor(sV, BN, 0);
    const uint64_t k_mn = desc_mnmajor(sK, BN, 0);
    const uint64_t ds_kd = desc_kmajor(sDS, BM, 0);
    constexpr uint32_t TSTEP = C::TILE >> 4, DSSTEP = C::DS_BYTES >> 4;
    auto issue_sdp = [&](int j) -> bool {
      const int st = j % NST;
      if (!mbar_wait(smem_u32(&bars.k_full[st]), (j / NST) & 1, abort, kWaitTimeoutNs) ||
          !mbar_wait(smem_u32(&bars.v_full[st]), (j / NST) & 1, abort, kWaitTimeoutNs))
        return false;
      tc_fence_after();
      const uint32_t ko = st * TSTEP;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma_ss_w(tS, q_kd + kmajor_step(BM, kk), k_kd + ko + kmajor_step(BN, kk), idS, kk > 0);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma_ss_w(tDP, do_kd + kmajor_step(BM, kk), v_kd + ko + kmajor_step(BN, kk), idS, kk > 0);
      umma_commit_w(smem_u32(&bars.s_full));
      return true;
    };
    bool ok = mbar_wait(smem_u32(&bars.q_full), 0, abort, kWaitTimeoutNs) && issue_sdp(0);
    for (int j = 0; ok && j < n_kt; ++j) {
      const int st = j % NST, b = j % NDS;
      if (j + 1 < n_kt) {
        // S and dP of step j are in registers of the compute warps: overwrite them
        if (!mbar_wait(smem_u32(&bars.s_free), j & 1, abort, kWaitTimeoutNs)) break;
        if (!issue_sdp(j + 1)) break;
      }
      if (!mbar_wait(smem_u32(&bars.ds_full[b]), (j / NDS) & 1, abort, kWaitTimeoutNs)) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk)
        umma_ss_w(tDQ, ds_kd + b * DSSTEP + kmajor_step(BM, kk), k_mn + st * TSTEP + mnmajor_step(kk),
                  idQ, (j > 0 || kk > 0));
      umma_commit_w(smem_u32(&bars.ds_empty[b]));
      umma_commit_w(smem_u32(&bars.kv_empty[st]));  // K_j (and V_j, read by dP(j)) done
    }
    if (ok) umma_commit_w(smem_u32(&bars.dq_full));
    // every product this warp issued has completed before tensor memory is released
    umma_commit_w(smem_u32(&bars.mma_drain));
    mbar_wait_drain(smem_u32(&bars.mma_drain), 0, kWaitTimeoutNs);
  } else {
    // ------------------------------------------------------------------ dS compute, epilogue
    const int g = warp >> 2;                 // warpgroup: key columns [64 g, 64 g + 64)
    const int r = (warp & 3) * 32 + lane;    // query row in the block = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int q = q_lo + r;
    const bool row_ok = q < sv.len_q;
    const int64_t grow = sv.row0_q + q;
    const float c2 = p.scale_log2;
    float nlse2 = 0.f, ndl = 0.f;
    if (row_ok) {
      nlse2 = -p.lse[sv.batch * p.l_sb + h * p.l_sh + grow * p.l_ss] * 1.4426950408889634f;
      ndl = -p.delta[zh * p.rows_q + grow];
    }
    const int c_base = g * 64;
    bool ok = true;
    for (int j = 0; ok && j < n_kt; ++j) {
      const int b = j % NDS;
      if (!mbar_wait(smem_u32(&bars.s_full), j & 1, abort, kWaitTimeoutNs)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv_all[64], dpv_all[64];
      ATTN_TMEM_LD4_X32(tmem + C::COL_S + lane_off + c_base, tmem + C::COL_S + lane_off + c_base + 32,
                        tmem + C::COL_DP + lane_off + c_base,
                        tmem + C::COL_DP + lane_off + c_base + 32,
                        reinterpret_cast<uint32_t*>(sv_all), reinterpret_cast<uint32_t*>(sv_all + 32),
                        reinterpret_cast<uint32_t*>(dpv_all),
                        reinterpret_cast<uint32_t*>(dpv_all + 32));
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.s_free));
      const int k0 = j * BN + c_base;  // key index of this thread's first column
      // element masks only where the tile crosses the key length, the diagonal or the rows
      const bool need_mask = !row_ok || (k0 + 64 > sv.len_k) || (p.causal && k0 + 63 > q_lo);
      const int kmax = !row_ok ? -1 : (p.causal ? min(q, sv.len_k - 1) : sv.len_k - 1);
      uint8_t* gDS = smem + C::OFF_DS + b * C::DS_BYTES;
      const uint64_t c2x2 = f2_pack(c2, c2), nl2 = f2_pack(nlse2, nlse2), nd2 = f2_pack(ndl, ndl);
      uint32_t pd[32];  // dS of this thread's 64 columns, packed in pairs
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const float* s = sv_all + ch * 32;
        const float* dp = dpv_all + ch * 32;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0, x1, y0, y1, d0, d1;
          f2_unpack(f2_fma(f2_pack(s[e], s[e + 1]), c2x2, nl2), x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          f2_unpack(f2_add(f2_pack(dp[e], dp[e + 1]), nd2), y0, y1);
          f2_unpack(f2_mul(f2_pack(p0, p1), f2_pack(y0, y1)), d0, d1);
          if (need_mask) {
            const int kk = k0 + ch * 32 + e;
            d0 = (kk <= kmax) ? d0 : 0.f;
            d1 = (kk + 1 <= kmax) ? d1 : 0.f;
          }
          pd[ch * 16 + e / 2] = pack2<F16>(d0, d1);
        }
      }
      // the dS buffer was last read by the dQ MMA NDS steps ago
      if (j >= NDS &&
          !mbar_wait(smem_u32(&bars.ds_empty[b]), ((j / NDS) - 1) & 1, abort, kWaitTimeoutNs)) {
        ok = false;
        break;
      }
      // row r of the K-major dS tile: slab g holds keys [64 g, 64 g + 64)
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const uint32_t off = sw128_offset(r, c_base + c8 * 8, BM);
        *reinterpret_cast<uint4*>(gDS + off) =
            make_uint4(pd[c8 * 4 + 0], pd[c8 * 4 + 1], pd[c8 * 4 + 2], pd[c8 * 4 + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars.ds_full[b]));
    }
    // ---- epilogue: dQ = sm_scale * acc; warpgroup g writes columns [g D/2, (g+1) D/2)
    if (ok) ok = mbar_wait(smem_u32(&bars.dq_full), 0, abort, kWaitTimeoutNs);
    tc_fence_after();
    if (ok) {
      uint16_t* dr = p.dq + sv.batch * p.dq_sb + h * p.dq_sh + grow * p.dq_ss;
      const float sc = p.sm_scale;
#pragma unroll
      for (int c = g * (D / 2); c < (g + 1) * (D / 2); c += 32) {
        uint32_t a[32];
        ATTN_TMEM_LD_X32(tmem + C::COL_DQ + lane_off + c, a);
        if (row_ok && c < p.d_out) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 v;
            v.x = pack2<F16>(__uint_as_float(a[e]) * sc, __uint_as_float(a[e + 1]) * sc);
            v.y = pack2<F16>(__uint_as_float(a[e + 2]) * sc, __uint_as_float(a[e + 3]) * sc);
            v.z = pack2<F16>(__uint_as_float(a[e + 4]) * sc, __uint_as_float(a[e + 5]) * sc);
            v.w = pack2<F16>(__uint_as_float(a[e + 6]) * sc, __uint_as_float(a[e + 7]) * sc);
            *reinterpret_cast<uint4*>(dr + c + e) = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && bars.abort && p.status != nullptr) atomicCAS(p.status, 0, kStatusTimeout);
}

template <int D, bool F16>
static cudaError_t launch_dq_impl(const BwdDqParams& p, dim3 grid, cudaStream_t stream) {
  using C = DqCfg<D>;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  attn_bwd_dq_kernel<D, F16><<<grid, C::NTHREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdDqParams& p, int D, bool f16, dim3 grid, cudaStream_t stream) {
  if (D == 128)
    return f16 ? launch_dq_impl<128, true>(p, grid, stream) : launch_dq_impl<128, false>(p, grid, stream);
  return f16 ? launch_dq_impl<64, true>(p, grid, stream) : launch_dq_impl<64, false>(p, grid, stream);
}

// Query rows per CTA of the deterministic dQ kernel (Q / dO tensor maps use this box).
int bwd_dq_block_m() { return 128; }

}  // namespace attn_sm103
