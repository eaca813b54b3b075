// Forward pass of fused scaled-dot-product attention on sm_103a.
//
// One CTA computes one 128-row query tile of one (batch or sequence, head):
//   S_j = Q K_j^T                       tcgen05 MMA, fp32 accumulator in TMEM
//   online softmax over S_j              one thread per query row (TMEM lane), exp2 domain
//   O  += P_j V_j                        tcgen05 MMA, P_j read from TMEM (written over S_j)
// then O / l (bf16) and LSE = (m + log2 l) ln 2 are stored. Forward keeps LSE so that the
// backward pass can rebuild P (the stash / recompute split of the nvFuser SDPA page).
//
// Warp roles (256 threads):
//   warp 0      TMA producer: Q once, then K_j / V_j into an NST-deep ring of stages
//   warp 1      TMEM allocator and MMA issuer (one elected thread)
//   warps 4..7  softmax + O correction + epilogue; thread r owns query row r
// TMEM (512 columns): S buffers at columns 0 and 128 (double buffered, so Q K_{j+1}^T runs
// while row statistics of S_j are computed), O at column 256.
//
// Online softmax in base 2 with a lazy rescale: the reference maximum m only moves when
// a row maximum exceeds it by more than 8 (p <= 2^8); O and l are rescaled by 2^(m_old -
// m_new) only then. The final O / l is the same quantity whatever m was used.
//
// Tile schedule: key tiles past the sequence's key length, and (causal, top-left) key
// tiles entirely above the diagonal are never loaded; element masks are applied only on
// tiles that straddle the diagonal or the key length. Query tiles at or past the sequence's
// query length exit before doing anything (AOTriton padded-varlen prologue).
#include "attn_common.cuh"
#include "attn_launch.h"

namespace attn_sm103 {

template <int D>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int NST = (D == 128) ? 2 : 4;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + NST * KV_BYTES;
  static constexpr int SMEM_BYTES = OFF_V + NST * KV_BYTES + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
};

template <int NST>
struct FwdBars {
  uint64_t q_full;
  uint64_t k_full[NST], v_full[NST], kv_empty[NST];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D>
__global__ void __launch_bounds__(256, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int BM = C::BM, BN = C::BN, NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdBars<NST> bars;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, z = blockIdx.z;
  const int m_tile = p.causal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;

  SeqView sv;
  if (!decode_seq(p.seq, z, threadIdx.x == 0 ? p.status : nullptr, sv)) return;
  if (m_tile * BM >= sv.len_q) return;  // past this sequence's queries

  const int q_lo = m_tile * BM;
  const int q_hi = min(q_lo + BM, sv.len_q);  // exclusive
  int n_tiles = (sv.len_k + BN - 1) / BN;
  if (p.causal) n_tiles = min(n_tiles, (q_hi - 1) / BN + 1);

  if (n_tiles <= 0) {  // no visible keys: O = 0, LSE = -inf on the valid rows
    if (warp >= 4) {
      const int row = q_lo + (threadIdx.x - 128);
      if (row < sv.len_q) {
        const int64_t grow = sv.row0_q + row;
        __nv_bfloat16* orow = p.o + sv.batch * p.o_sb + h * p.o_sh + grow * p.o_ss;
        for (int d = 0; d < D; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
        p.lse[sv.batch * p.l_sb + h * p.l_sh + grow * p.l_ss] = -INFINITY;
      }
    }
    return;
  }

  uint8_t* smem = align1024(smem_raw);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q);
  const uint32_t sK = smem_u32(smem + C::OFF_K);
  const uint32_t sV = smem_u32(smem + C::OFF_V);

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(smem_u32(&bars.q_full), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.kv_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars.s_full[b]), 1);
      mbar_init(smem_u32(&bars.p_full[b]), 128);
    }
    mbar_init(smem_u32(&bars.o_done), 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars.tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort = &bars.abort;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
      const uint32_t qb = smem_u32(&bars.q_full);
      mbar_arrive_expect_tx(qb, C::Q_BYTES);
#pragma unroll
      for (int s = 0; s < D / 64; ++s)
        tma_load_4d(sQ + s * BM * 128, &p.tm_q, qb, s * 64, sv.row0_q + q_lo, h, sv.batch);
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % NST;
        if (j >= NST &&
            !mbar_wait(smem_u32(&bars.kv_empty[st]), ((j / NST) - 1) & 1, abort, kWaitTimeoutNs))
          break;
        const int krow = sv.row0_k + j * BN;
        const uint32_t kb = smem_u32(&bars.k_full[st]);
        mbar_arrive_expect_tx(kb, C::KV_BYTES);
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_4d(sK + st * C::KV_BYTES + s * BN * 128, &p.tm_k, kb, s * 64, krow, h, sv.batch);
        const uint32_t vb = smem_u32(&bars.v_full[st]);
        mbar_arrive_expect_tx(vb, C::KV_BYTES);
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_4d(sV + st * C::KV_BYTES + s * BN * 128, &p.tm_v, vb, s * 64, krow, h, sv.batch);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, BN, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
      const uint32_t tS[2] = {tmem + C::COL_S0, tmem + C::COL_S1};
      const uint32_t tO = tmem + C::COL_O;
      bool ok = mbar_wait(smem_u32(&bars.q_full), 0, abort, kWaitTimeoutNs);
      auto issue_s = [&](int j) -> bool {
        const int st = j % NST;
        if (!mbar_wait(smem_u32(&bars.k_full[st]), (j / NST) & 1, abort, kWaitTimeoutNs))
          return false;
        tc_fence_after();
        const uint32_t kbase = sK + st * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tS[j & 1], desc_kmajor(sQ, BM, kk), desc_kmajor(kbase, BN, kk), idS, kk > 0);
        umma_commit(smem_u32(&bars.s_full[j & 1]));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles && !issue_s(j + 1)) break;
        const int st = j % NST;
        if (!mbar_wait(smem_u32(&bars.p_full[j & 1]), (j >> 1) & 1, abort, kWaitTimeoutNs)) break;
        if (!mbar_wait(smem_u32(&bars.v_full[st]), (j / NST) & 1, abort, kWaitTimeoutNs)) break;
        tc_fence_after();
        const uint32_t vbase = sV + st * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ts(tO, tS[j & 1] + kk * 8, desc_mnmajor(vbase, BN, kk), idO, (j > 0 || kk > 0));
        umma_commit(smem_u32(&bars.kv_empty[st]));
        umma_commit(smem_u32(&bars.o_done));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    const int r = threadIdx.x - 128;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int row = q_lo + r;  // local query index
    const float c2 = p.scale_log2;
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1;
      if (!mbar_wait(smem_u32(&bars.s_full[b]), (j >> 1) & 1, abort, kWaitTimeoutNs)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tSb = tmem + (b ? C::COL_S1 : C::COL_S0) + lane_off;
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t* u = reinterpret_cast<uint32_t*>(&s[c * 32]);
        ATTN_TMEM_LD_X32(tSb + c * 32, u);
      }
      const int k0 = j * BN;
      if (k0 + BN > sv.len_k || (p.causal && k0 + BN - 1 > q_lo)) {
        const int kmax = p.causal ? min(row, sv.len_k - 1) : sv.len_k - 1;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (k0 + c > kmax) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < BN; ++c) mx = fmaxf(mx, s[c]);
      const float mx2 = mx * c2;
      float m_new = m_use, scale = 1.f;
      if (mx2 > m_use + 8.f) {
        m_new = mx2;
        scale = ex2_approx(m_use - m_new);
      }
      const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float p0 = ex2_approx(fmaf(s[2 * c], c2, neg_m));
        const float p1 = ex2_approx(fmaf(s[2 * c + 1], c2, neg_m));
        rs0 += p0;
        rs1 += p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * scale + (rs0 + rs1);
      m_use = m_new;
      if (j > 0) {
        if (!mbar_wait(smem_u32(&bars.o_done), (j - 1) & 1, abort, kWaitTimeoutNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, scale != 1.f)) {
          const uint32_t tOr = tmem + C::COL_O + lane_off;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            ATTN_TMEM_LD_X32(tOr + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * scale);
            ATTN_TMEM_ST_X32(tOr + c * 32, o);
          }
        }
      }
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) ATTN_TMEM_ST_X16(tSb + c * 16, (&pk[c * 16]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.p_full[b]));
    }
    if (ok) ok = mbar_wait(smem_u32(&bars.o_done), (n_tiles - 1) & 1, abort, kWaitTimeoutNs);
    tc_fence_after();
    if (ok) {
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const bool valid = row < sv.len_q;
      const int64_t grow = sv.row0_q + row;
      __nv_bfloat16* orow = p.o + sv.batch * p.o_sb + h * p.o_sh + grow * p.o_ss;
      const uint32_t tOr = tmem + C::COL_O + lane_off;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        ATTN_TMEM_LD_X32(tOr + c * 32, o);
        if (valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[e + 0]) * inv_l, __uint_as_float(o[e + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv_l, __uint_as_float(o[e + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv_l, __uint_as_float(o[e + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv_l, __uint_as_float(o[e + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c * 32 + e) = v;
          }
        }
      }
      if (valid)
        p.lse[sv.batch * p.l_sb + h * p.l_sh + grow * p.l_ss] =
            (l > 0.f) ? (m_use + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && bars.abort && p.status != nullptr) atomicCAS(p.status, 0, kStatusTimeout);
}

template <int D>
static cudaError_t launch_fwd_impl(const FwdParams& p, dim3 grid, cudaStream_t stream) {
  using C = FwdCfg<D>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  attn_fwd_kernel<D><<<grid, 256, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const FwdParams& p, int D, dim3 grid, cudaStream_t stream) {
  return D == 128 ? launch_fwd_impl<128>(p, grid, stream) : launch_fwd_impl<64>(p, grid, stream);
}

int fwd_block_m() { return 128; }

}  // namespace attn_sm103
