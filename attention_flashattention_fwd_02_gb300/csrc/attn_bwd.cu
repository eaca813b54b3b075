// Backward pass of fused scaled-dot-product attention on sm_103a: three kernels.
//
//  1. attn_bwd_pre_kernel    Delta_i = sum_d dO_id O_id (fp32) and zeroing of the fp32 dQ
//                            accumulator rows. Memory-bound.
//  2. attn_bwd_main_kernel   one CTA per 128-key tile (K_n, V_n loaded once), looping over
//                            the query tiles that can see those keys:
//                              S^T  = K_n Q_m^T           (tcgen05, TMEM)
//                              dP^T = V_n dO_m^T          (tcgen05, TMEM)
//                              P^T  = exp2(S^T c2 - LSE2), dS^T = P^T (dP^T - Delta)
//                              dV  += P^T dO_m            (tcgen05, TMEM accumulator)
//                              dK  += dS^T Q_m            (tcgen05, TMEM accumulator)
//                              dQ_m partial = dS K_n      (tcgen05, TMEM) -> TMA reduce-add
//                            then dK * sm_scale and dV are written. P is rebuilt from the
//                            LSE that the forward pass stashed.
//  3. attn_bwd_post_kernel   dQ = sm_scale * accumulator, rounded to the element type.
//
// Main-kernel warp roles: warps 0..7 are two compute warpgroups that split the query
// columns of each key row (thread row j = TMEM lane j) to form P^T (written to TMEM, where it
// is the A operand of the dV MMA) and dS^T (written to shared memory for the dK and dQ MMAs),
// and at the end write dK / dV. Warp 8 is the TMA producer; warp 9 allocates TMEM and issues
// the MMAs. Each step's dQ partial goes from TMEM into the global fp32 accumulator through
// shared-memory staging and TMA reduce-adds: at d_head 128 (512 threads) warps 12..15 do this
// (each the 32 TMEM lanes it can reach) while the compute warps already work on the next
// step, and warp 11 has no role; at d_head 64 (320 threads; the compute warps hold a step's
// 128 score columns in registers, and a CTA of more warps would leave each fewer than that
// needs) every compute warp drains its own 32 x 32 block after forming the next step's P and
// dS. With a bias, warp 10 loads each step's bias tile into shared memory by TMA (352
// threads at d_head 64). Tile sizes: 128 keys per CTA; 64 query rows per step when d_head = 128 (dQ is
// formed transposed, K_n^T dS^T, so that every MMA has M = 128), 128 when d_head = 64.
#include <atomic>

#include "attn_common.cuh"
#include "attn_launch.h"

namespace attn_sm103 {

__device__ __forceinline__ uint8_t* align1024b(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

constexpr float kLog2e = 1.4426950408889634f;

// =========================================================================== preprocess
// One group of W/8 threads per row, W = the head size rounded up to a power of two: each
// thread reads 8 elements (16 bytes) of O and dO; threads past the head size (p.D) add zero.
template <int W, bool F16>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const __grid_constant__ BwdPreParams p) {
  constexpr int TPR = W / 8;             // threads per row
  constexpr int ROWS = 256 / TPR;        // rows per block
  const int h = blockIdx.y, z = blockIdx.z;
  SeqView sv;
  if (!decode_seq(p.seq, z, threadIdx.x == 0 ? p.status : nullptr, sv)) return;
  const int r = blockIdx.x * ROWS + threadIdx.x / TPR;
  const int part = threadIdx.x % TPR;
  if (blockIdx.x * ROWS >= sv.len_q) return;
  float acc = 0.f;
  const bool valid = r < sv.len_q;
  const bool cols = part * 8 < p.D;
  const int64_t grow = sv.row0_q + r;
  if (valid && cols) {
    const uint4 a = *reinterpret_cast<const uint4*>(p.o + sv.batch * p.o_sb + h * p.o_sh +
                                                    grow * p.o_ss + part * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(p.dout + sv.batch * p.do_sb + h * p.do_sh +
                                                    grow * p.do_ss + part * 8);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa = unpack2<F16>(aw[e]);
      const float2 fb = unpack2<F16>(bw[e]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (valid) {
    const int64_t idx = ((int64_t)sv.batch * p.H + h) * p.rows + grow;
    if (part == 0) p.delta[idx] = acc;
  }
  if (valid && cols && p.dq_acc != nullptr) {
    const int64_t idx = ((int64_t)sv.batch * p.H + h) * p.rows + grow;
    float4* dst = reinterpret_cast<float4*>(p.dq_acc + idx * p.D + part * 8);
    dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Power-of-two thread-group width covering head size D.
static int pow2_width(int D) { return D <= 32 ? 32 : D <= 64 ? 64 : D <= 128 ? 128 : 256; }

cudaError_t launch_bwd_preprocess(const BwdPreParams& p, cudaStream_t stream) {
  const int W = pow2_width(p.D);
  const int rows_per_block = 256 / (W / 8);
  const int max_len = p.seq.mode == kCompact ? p.seq.max_q : p.seq.Sq;
  dim3 grid((max_len + rows_per_block - 1) / rows_per_block, p.H, p.units);
  if (grid.x == 0 || grid.z == 0) return cudaSuccess;
  if (W == 256) {
    if (p.f16) attn_bwd_pre_kernel<256, true><<<grid, 256, 0, stream>>>(p);
    else attn_bwd_pre_kernel<256, false><<<grid, 256, 0, stream>>>(p);
  } else if (W == 128) {
    if (p.f16) attn_bwd_pre_kernel<128, true><<<grid, 256, 0, stream>>>(p);
    else attn_bwd_pre_kernel<128, false><<<grid, 256, 0, stream>>>(p);
  } else if (W == 64) {
    if (p.f16) attn_bwd_pre_kernel<64, true><<<grid, 256, 0, stream>>>(p);
    else attn_bwd_pre_kernel<64, false><<<grid, 256, 0, stream>>>(p);
  } else {
    if (p.f16) attn_bwd_pre_kernel<32, true><<<grid, 256, 0, stream>>>(p);
    else attn_bwd_pre_kernel<32, false><<<grid, 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

// =========================================================================== dQ epilogue
template <int W, bool F16>
__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const __grid_constant__ BwdPostParams p) {
  constexpr int TPR = W / 8;
  constexpr int ROWS = 256 / TPR;
  const int h = blockIdx.y, z = blockIdx.z;
  SeqView sv;
  if (!decode_seq(p.seq, z, nullptr, sv)) return;
  const int r = blockIdx.x * ROWS + threadIdx.x / TPR;
  const int part = threadIdx.x % TPR;
  if (r >= sv.len_q || part * 8 >= p.D) return;
  const int64_t grow = sv.row0_q + r;
  const int64_t idx = ((int64_t)sv.batch * p.H + h) * p.rows + grow;
  const float4* src = reinterpret_cast<const float4*>(p.dq_acc + idx * p.D + part * 8);
  const float4 a = src[0], b = src[1];
  uint4 v;
  v.x = pack2<F16>(a.x * p.sm_scale, a.y * p.sm_scale);
  v.y = pack2<F16>(a.z * p.sm_scale, a.w * p.sm_scale);
  v.z = pack2<F16>(b.x * p.sm_scale, b.y * p.sm_scale);
  v.w = pack2<F16>(b.z * p.sm_scale, b.w * p.sm_scale);
  *reinterpret_cast<uint4*>(p.dq + sv.batch * p.dq_sb + h * p.dq_sh + grow * p.dq_ss + part * 8) = v;
}

cudaError_t launch_bwd_dq_epilogue(const BwdPostParams& p, cudaStream_t stream) {
  const int W = pow2_width(p.D);
  const int rows_per_block = 256 / (W / 8);
  const int max_len = p.seq.mode == kCompact ? p.seq.max_q : p.seq.Sq;
  dim3 grid((max_len + rows_per_block - 1) / rows_per_block, p.H, p.units);
  if (grid.x == 0 || grid.z == 0) return cudaSuccess;
  if (W == 256) {
    if (p.f16) attn_bwd_post_kernel<256, true><<<grid, 256, 0, stream>>>(p);
    else attn_bwd_post_kernel<256, false><<<grid, 256, 0, stream>>>(p);
  } else if (W == 128) {
    if (p.f16) attn_bwd_post_kernel<128, true><<<grid, 256, 0, stream>>>(p);
    else attn_bwd_post_kernel<128, false><<<grid, 256, 0, stream>>>(p);
  } else if (W == 64) {
    if (p.f16) attn_bwd_post_kernel<64, true><<<grid, 256, 0, stream>>>(p);
    else attn_bwd_post_kernel<64, false><<<grid, 256, 0, stream>>>(p);
  } else {
    if (p.f16) attn_bwd_post_kernel<32, true><<<grid, 256, 0, stream>>>(p);
    else attn_bwd_post_kernel<32, false><<<grid, 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

// =========================================================================== dbias epilogue
// The gradient of a bias shared by several units or heads: dbias = the fp32 sums the
// key-tile kernel added up, rounded to the element type, over the bias's whole shape (zero
// wherever no sequence reached). One block per row, threads over its keys.
template <bool F16>
__global__ void __launch_bounds__(256) attn_dbias_post_kernel(const __grid_constant__ DbiasPostParams p) {
  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
    const int64_t b = row / ((int64_t)p.Hb * p.Sq), hq = row % ((int64_t)p.Hb * p.Sq);
    const int64_t hh = hq / p.Sq, q = hq % p.Sq;
    const float* src = p.acc + row * p.Sk;
    uint16_t* dst = p.dbias + b * p.db_sb + hh * p.db_sh + q * p.db_ss;
    for (int k = threadIdx.x; k < p.Sk; k += blockDim.x)
      dst[k] = (uint16_t)(pack2<F16>(src[k], 0.f) & 0xffffu);
  }
}

cudaError_t launch_dbias_epilogue(const DbiasPostParams& p, cudaStream_t stream) {
  if (p.rows == 0 || p.Sk == 0) return cudaSuccess;
  const unsigned grid = (unsigned)(p.rows < 65536 * 16 ? p.rows : 65536 * 16);
  if (p.f16) attn_dbias_post_kernel<true><<<grid, 256, 0, stream>>>(p);
  else attn_dbias_post_kernel<false><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// =========================================================================== main kernel
template <int D, bool BIAS = false>
struct BwdCfg {
  // d_head 256: dK and dV of 128 keys would take all 512 TMEM columns, so a CTA accumulates
  // dK, dV and the dQ partial for one half of d (DH = 128 columns) and recomputes S^T and dP^T
  // over all 256 columns (its sibling CTA, with the other half, computes them too).
  static constexpr bool DSPLIT = (D == 256);
  static constexpr int DH = DSPLIT ? D / 2 : D;     // d columns a CTA accumulates
  static constexpr int BN = 128;                    // keys per CTA (MMA M for S^T, dP^T, dK, dV)
  static constexpr int BM = DSPLIT ? 32 : (D == 128) ? 64 : 128;  // query rows per step
  static constexpr bool DQ_T = (D >= 128);          // dQ^T = K^T dS^T (M = DH) vs dQ = dS K (M = BM)
  // dS is stored transposed, [key][query] in 128-byte swizzled slabs of 64 queries, except at
  // d_head 256, whose 32-query steps are too short for such rows: there it is stored
  // [query][key] (slabs of 64 keys), the MN-major A operand of dK and the K-major B of dQ^T.
  static constexpr bool DS_QMAJOR = DSPLIT;
  static constexpr int NCWG = DSPLIT ? 1 : 2;       // compute warpgroups (HALF columns each)
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int DS_BYTES = BN * BM * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  // Q / dO / LSE / Delta stages: two at d_head 256, and in the d_head 64 bias kernel, whose
  // bias tile slot takes the third stage's room
  static constexpr int QST = (DSPLIT || (D == 64 && BIAS)) ? 2 : 3;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;        // QST stages
  static constexpr int OFF_DO = OFF_Q + QST * Q_BYTES;  // QST stages
  static constexpr int OFF_DS = OFF_DO + QST * Q_BYTES; // 2 buffers
  // dQ drain: a warpgroup of its own at d_head 128 and 256, each warp staging BM / 32 blocks
  // of 32 x 32 fp32 in an area of its own; at d_head 64 the compute warps, each staging its
  // 32 x 32 block in rows of the dS^T buffer it has just released (only that warp writes those
  // rows again, two steps later, after waiting for the reduce to read them).
  static constexpr bool DQ_WARPS = DQ_T;
  static constexpr int DQ_BLOCKS = BM / 32;             // 32 x 32 blocks per drain warp
  // d_head 64 and 128 with a bias: a warp of its own (warp 10) loads each step's bias tile
  // (BM query rows x 128 keys, two 64-key slabs with the 128-byte swizzle) into a slot of
  // shared memory by TMA. The room comes at d_head 128 from the drain warps, which then stage
  // one 32 x 32 block at a time (4 KB each), at d_head 64 from a third Q / dO stage.
  static constexpr bool BIAS_TMA = BIAS && (D <= 128);
  static constexpr int WARP_BIAS = 10;
  static constexpr int STG_BLOCKS = BIAS_TMA ? 1 : DQ_BLOCKS;  // blocks a drain warp stages at once
  static constexpr int OFF_STG = OFF_DS + 2 * DS_BYTES;
  static constexpr int STG_BYTES = DQ_WARPS ? 4 * STG_BLOCKS * 4096 : 0;
  // d_head 64: the score products also subtract LSE / sm_scale and Delta, through one more
  // K = 16 step that multiplies a tile of ones by those values (each split into three bf16
  // parts), so the compute warps read neither per column. The K = 16 operand tiles (32 bytes
  // per row) are packed as the 32-byte column groups of two 128-row SW128 slabs: group 0 the
  // ones, groups 1..QST the LSE rows of the Q stages, groups 4..3+QST the Delta rows.
  static constexpr bool AUG = (D == 64);
  static constexpr int OFF_AUG = OFF_STG + STG_BYTES;
  static constexpr int AUG_BYTES = AUG ? 2 * BN * 128 : 0;
  static_assert(!AUG || (BM == BN && QST <= 3), "augmented operand packing");
  static constexpr int LSE_ST = AUG ? 1 : QST;  // stages of the per-column LSE / Delta arrays
  static constexpr int OFF_BIAS = OFF_AUG + AUG_BYTES;
  static constexpr int BIAS_BYTES = BIAS_TMA ? BM * BN * 2 : 0;
  static constexpr int SMEM_BYTES = OFF_BIAS + BIAS_BYTES + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB per CTA)");
  // TMEM columns: dK, dV accumulators (DH each); S^T, dP^T of the current step; the dQ
  // partial; and P^T (16-bit, two values per column) as the A operand of the dV MMA.
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_DK = 0, COL_DV = DH, COL_S = 2 * DH, COL_DP = 2 * DH + BM;
  static constexpr uint32_t COL_DQ = 2 * DH + 2 * BM;
  static constexpr uint32_t COL_P = COL_DQ + (DQ_T ? BM : D);
  static_assert(COL_P + BM / 2 <= TMEM_COLS, "TMEM layout does not fit");
  // d_head 128: dS^T also goes to the last 32 TMEM columns (16-bit, like P^T) and is the A
  // operand of dK from there, which takes its 16 KB a step off the shared-memory reads (the
  // step is bound by them); shared memory keeps dS^T for dQ. Elsewhere TMEM has no room
  // (d_head 64) or dS is stored query-major for 32-query steps (d_head 256).
  static constexpr bool DS_TMEM = (D == 128);
  static constexpr uint32_t COL_DST = COL_P + BM / 2;
  static_assert(!DS_TMEM || COL_DST + BM / 2 <= TMEM_COLS, "TMEM layout does not fit");
  // Warps. d_head 64: 0..7 compute, 8 producer, 9 MMA (320 threads; with a bias also 10,
  // the bias tile loader: 352). d_head 128: 0..7 compute, 8 producer, 9 MMA, 10 the bias
  // tile loader of the bias kernel (else no role), 11 no role, 12..15 dQ drain (512 threads
  // leave 128 registers a thread, which these roles fit in). d_head 256: 0..3 compute, 4..7
  // dQ drain, 8 producer, 9 MMA (320 threads). A drain warp reaches the TMEM lanes of its
  // index mod 4.
  static constexpr int NTHREADS = (D == 128) ? 512 : (BIAS_TMA ? 352 : 320);
  static constexpr int WARP_PRODUCER = 8, WARP_MMA = 9, WARP_DRAIN0 = DSPLIT ? 4 : 12;
  static constexpr int NCOMPUTE = 128 * NCWG;        // compute threads
  // Epilogue: a compute warp stores its 32 keys x CW columns of dK and of dV through shared
  // memory with TMA stores; the K and V tiles' space is free by then and holds the 2 x 4 NCWG
  // warp areas. A warp's area holds CW / EPI_SC slabs of 32 rows (keys) x EPI_SC columns (64
  // or 128 bytes a row) whose 16-byte chunks are swizzled like the TMA's 64- or 128-byte
  // modes, so that a warp's 16-byte stores (one row a lane) spread over all banks. Tiles
  // reaching past the sequence leave with row stores.
  static constexpr bool EPI_TMA = true;
  static constexpr int CW = DH / NCWG;
  static constexpr int EPI_W_BYTES = 32 * CW * 2;
  static constexpr int EPI_SC = CW < 64 ? CW : 64;
  static constexpr int EPI_SLAB_BYTES = 32 * EPI_SC * 2;
  static_assert(2 * 4 * NCWG * EPI_W_BYTES <= 2 * KV_BYTES, "epilogue staging");
};

template <int BM, int QST, int LSE_ST>
struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[QST], q_empty[QST];
  uint64_t s_full, s_free, p_full, p_empty;
  uint64_t ds_full[2];
  uint64_t dq_full, dq_empty, dkdv_full;
  uint64_t bias_full, bias_empty;  // d_head 128 bias kernels: the step's bias tile in its slot
  uint64_t mma_drain;  // completion of the MMA warp's last products
  uint32_t tmem_base;
  int abort;
  alignas(16) float nlse2[LSE_ST][BM];   // -LSE * log2(e) of the step's query rows
  alignas(16) float ndelta[LSE_ST][BM];  // -Delta
};

// BIAS: an additive bias enters the rebuilt scores. Each compute thread (one key row) reads
// its key's column of the bias for the step's query rows straight from global memory (a warp
// reads 32 consecutive keys of one query row per load); every unit (batch, or sequence of a
// compact batch) finds its block at offset 0 of its own slice of the bias's first dimension.
// With p.dbias set, dS is written to the same places; with p.dbias_acc set (a bias shared by
// several units or heads), dS is added in fp32 to an accumulator of the bias's shape.
template <int D, bool F16, bool BIAS = false>
__global__ void __launch_bounds__(BwdCfg<D, BIAS>::NTHREADS, 1)
    attn_bwd_main_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D, BIAS>;
  static_assert(!BIAS || D <= 128, "no bias kernel at d_head 256");
  constexpr int BN = C::BN, BM = C::BM, DH = C::DH;
  constexpr int HALF = BM / C::NCWG;  // score columns per compute warpgroup
  extern __shared__ uint8_t smem_raw[];
  constexpr int QST = C::QST;
  __shared__ BwdBars<BM, QST, C::LSE_ST> bars;
  static_assert(C::SMEM_BYTES + sizeof(BwdBars<BM, QST, C::LSE_ST>) <= 232448,
                "static and dynamic shared memory (227 KB per CTA)");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 1-D grid over (unit, head) pairs x key tiles (grid_pos; key tile 0, the heaviest of a
  // causal grid, first); at d_head 256 each key tile has two CTAs, one per half of d
  // (index 2 tile + half)
  const GridPos gp = grid_pos((int)blockIdx.x, p.tiles, (int)(gridDim.x / p.tiles), p.group);
  const int h = gp.zh % p.H, z = gp.zh / p.H;
  const int kt = gp.rank;
  const int n_tile = C::DSPLIT ? kt >> 1 : kt;
  const int dh = C::DSPLIT ? kt & 1 : 0;  // the half of d this CTA accumulates

  SeqView sv;
  if (!decode_seq(p.seq, z, threadIdx.x == 0 ? p.status : nullptr, sv)) return;
  const int k_lo = n_tile * BN;
  if (k_lo >= sv.len_k) return;
  const int m_begin = p.causal ? k_lo / BM : 0;
  const int m_end = (sv.len_q + BM - 1) / BM;
  const int n_steps = max(0, m_end - m_begin);
  const int64_t zh = (int64_t)sv.batch * p.H + h;
  // Query tile of step it. Without a causal mask every key tile visits all query tiles; the
  // starting tile is rotated by the key-tile index so that the CTAs of one head do not add
  // into the same dQ rows at the same time.
  const int rot = p.causal ? 0 : (n_steps > 0 ? n_tile % n_steps : 0);
  auto q_tile = [&](int it) {
    const int r = it + rot;
    return m_begin + (r >= n_steps ? r - n_steps : r);
  };

  if (n_steps == 0) {  // no query sees these keys: dK = dV = 0
    if (threadIdx.x < BN) {
      const int key = k_lo + threadIdx.x;
      if (key < sv.len_k) {
        const int64_t grow = sv.row0_k + key;
        uint16_t* kr = p.dk + sv.batch * p.dk_sb + h * p.dk_sh + grow * p.dk_ss;
        uint16_t* vr = p.dv + sv.batch * p.dv_sb + h * p.dv_sh + grow * p.dv_ss;
        for (int d = dh * DH; d < min(dh * DH + DH, p.d_out); d += 8) {
          *reinterpret_cast<uint4*>(kr + d) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vr + d) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    return;
  }

  uint8_t* smem = align1024b(smem_raw);
  const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
  const uint32_t sDS = smem_u32(smem + C::OFF_DS);
  const uint32_t sAUG = smem_u32(smem + C::OFF_AUG);

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(smem_u32(&bars.kv_full), 1);
    for (int s = 0; s < QST; ++s) {
      mbar_init(smem_u32(&bars.q_full[s]), 33);  // producer lane 0 (tx) + 32 lanes (LSE/Delta)
      mbar_init(smem_u32(&bars.q_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(smem_u32(&bars.ds_full[s]), C::NCOMPUTE);
    mbar_init(smem_u32(&bars.s_full), 1);
    mbar_init(smem_u32(&bars.s_free), C::NCOMPUTE);
    mbar_init(smem_u32(&bars.p_full), C::NCOMPUTE);
    mbar_init(smem_u32(&bars.p_empty), 1);
    mbar_init(smem_u32(&bars.dq_full), 1);
    mbar_init(smem_u32(&bars.dq_empty), C::DQ_WARPS ? 128 : 256);  // the draining warps
    mbar_init(smem_u32(&bars.dkdv_full), 1);
    mbar_init(smem_u32(&bars.mma_drain), 1);
    mbar_init(smem_u32(&bars.bias_full), 1);
    mbar_init(smem_u32(&bars.bias_empty), C::NCOMPUTE);
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
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
      tma_prefetch_map(&p.tm_do);
      const uint32_t kvb = smem_u32(&bars.kv_full);
      mbar_arrive_expect_tx(kvb, 2 * C::KV_BYTES);
#pragma unroll
      for (int s = 0; s < D / 64; ++s) {
        tma_load_4d(sK + s * BN * 128, &p.tm_k, kvb, s * 64, sv.row0_k + k_lo, h, sv.batch);
        tma_load_4d(sV + s * BN * 128, &p.tm_v, kvb, s * 64, sv.row0_k + k_lo, h, sv.batch);
      }
    }
    // Row r of 32-byte column group grp of the augmented operands: (a, b, c, 0, ..., 0) as bf16.
    auto aug_row = [&](int grp, int r, float a, float b, float c) {
      uint8_t* row = smem + C::OFF_AUG + (grp >> 2) * (BN * 128) + r * 128;
      const int c0 = 2 * (grp & 3);
      *reinterpret_cast<uint4*>(row + 16 * (c0 ^ (r & 7))) =
          make_uint4(pack_bf16x2(a, b), pack_bf16x2(c, 0.f), 0u, 0u);
      *reinterpret_cast<uint4*>(row + 16 * ((c0 + 1) ^ (r & 7))) = make_uint4(0u, 0u, 0u, 0u);
    };
    // v as the sum of three bf16 values (about 24 significant bits)
    auto aug_split = [&](int grp, int r, float v) {
      const float hi = __bfloat162float(__float2bfloat16_rn(v));
      const float r1 = v - hi;
      const float mid = __bfloat162float(__float2bfloat16_rn(r1));
      aug_row(grp, r, hi, mid, r1 - mid);
    };
    if (C::AUG)  // the ones tile, made visible to the MMAs by the first step's q_full arrival
      for (int r = lane; r < BN; r += 32) aug_row(0, r, 1.f, 1.f, 1.f);
    int last_it[QST];  // last step loaded into each stage (-1: none)
#pragma unroll
    for (int st = 0; st < QST; ++st) last_it[st] = -1;
    // LSE and Delta of a step's query rows (this lane's rows lane + 32 i; 0 off the
    // sequence), loaded one step ahead: the loads of step it + 1 are issued right after the
    // copies of step it, and nothing uses the values before they are written to shared
    // memory (the LSE's scaling by log2(e) too), so their latency hides behind the copies and
    // the next wait instead of holding up the copies (at a CTA's start that was two global
    // round trips before its first Q / dO copy)
    constexpr int NL = (BM + 31) / 32;
    float nl2[NL], ndl[NL];
    auto fetch_rows = [&](int itf, float* l2o, float* dlo) {
      const int q_lo_f = q_tile(itf) * BM;
#pragma unroll
      for (int u = 0; u < NL; ++u) {
        const int q = q_lo_f + lane + 32 * u;
        l2o[u] = 0.f;
        dlo[u] = 0.f;
        if (lane + 32 * u < BM && q < sv.len_q) {
          const int64_t grow = sv.row0_q + q;
          l2o[u] = p.lse[sv.batch * p.l_sb + h * p.l_sh + grow * p.l_ss];
          dlo[u] = p.delta[zh * p.rows_q + grow];
        }
      }
    };
    if (n_steps > 0) fetch_rows(0, nl2, ndl);
    for (int it = 0; it < n_steps; ++it) {
      const int st = it % QST;
      float cl2[NL], cdl[NL];  // this step's rows
#pragma unroll
      for (int u = 0; u < NL; ++u) {
        cl2[u] = nl2[u];
        cdl[u] = ndl[u];
      }
      if (it == p.withhold_step) {  // failure-detection test: this stage never fills
        if (it + 1 < n_steps) fetch_rows(it + 1, nl2, ndl);
        continue;
      }
      if (it >= QST &&
          !mbar_wait(smem_u32(&bars.q_empty[st]), ((it / QST) - 1) & 1, abort, p.timeout_ns))
        break;
      last_it[st] = it;
      const int q_lo = q_tile(it) * BM;
      const uint32_t qb = smem_u32(&bars.q_full[st]);
      if (lane == 0) {
        mbar_arrive_expect_tx(qb, 2 * C::Q_BYTES);
#pragma unroll
        for (int s = 0; s < D / 64; ++s) {
          tma_load_4d(sQ + st * C::Q_BYTES + s * BM * 128, &p.tm_q, qb, s * 64, sv.row0_q + q_lo, h,
                      sv.batch);
          tma_load_4d(sDO + st * C::Q_BYTES + s * BM * 128, &p.tm_do, qb, s * 64, sv.row0_q + q_lo,
                      h, sv.batch);
        }
      }
      if (it + 1 < n_steps) fetch_rows(it + 1, nl2, ndl);
#pragma unroll
      for (int u = 0; u < NL; ++u) {
        const int i = lane + 32 * u;
        if (i >= BM) break;
        const float l2 = cl2[u] * kLog2e, dl = cdl[u];
        if constexpr (C::AUG) {
          // c2 (S + a) = c2 S - LSE log2(e) with a = -LSE / sm_scale
          aug_split(1 + st, i, -l2 / p.scale_log2);
          aug_split(4 + st, i, -dl);
        } else {
          bars.nlse2[st][i] = -l2;
          bars.ndelta[st][i] = -dl;
        }
      }
      if (C::AUG) fence_proxy_async_smem();  // the rows are read by the MMAs (async proxy)
      mbar_arrive(qb);
    }
    // The K / V tile of the CTA one SM count further in launch order (likely the next to
    // start on a freed SM) into L2: its first copies then come from L2
    if (lane == 0 && !*abort) {
      uint32_t nsm;
      asm volatile("mov.u32 %0, %%nsmid;" : "=r"(nsm));
      const int nb = (int)blockIdx.x + (int)nsm;
      if (nb < (int)gridDim.x) {
        const GridPos gq = grid_pos(nb, p.tiles, (int)(gridDim.x / p.tiles), p.group);
        const int hq = gq.zh % p.H, zq = gq.zh / p.H;
        const int kq = (C::DSPLIT ? gq.rank >> 1 : gq.rank) * BN;
        SeqView sq;
        if (decode_seq(p.seq, zq, nullptr, sq) && kq < sq.len_k) {
#pragma unroll
          for (int s = 0; s < D / 64; ++s) {
            tma_prefetch_l2_4d(&p.tm_k, s * 64, sq.row0_k + kq, hq, sq.batch);
            tma_prefetch_l2_4d(&p.tm_v, s * 64, sq.row0_k + kq, hq, sq.batch);
          }
        }
      }
    }
    if (lane == 0 && *abort) {  // the consumers gave up: let the copies in flight land
      mbar_wait_drain(smem_u32(&bars.kv_full), 0, p.timeout_ns);
#pragma unroll
      for (int st = 0; st < QST; ++st)
        if (last_it[st] >= 0)
          mbar_wait_drain(smem_u32(&bars.q_full[st]), (last_it[st] / QST) & 1, p.timeout_ns);
    }
  } else if (warp == C::WARP_MMA) {
    // ------------------------------------------------------------------ MMA issuer
    // Issue order per step: S/dP(it+1) as soon as the compute warpgroups have loaded S^T and
    // dP^T of step it (so the next step's scores are ready when their P/dS math ends), then
    // dV(it) [P from TMEM], dK(it), dQ(it). The whole warp walks the schedule, so that every
    // descriptor is warp-uniform; one elected lane issues.
    {
      constexpr uint32_t idS = idesc_f32acc(128, BM, false, false, F16);  // S^T, dP^T
      constexpr uint32_t idG = idesc_f32acc(128, DH, false, true, F16);   // dV (A from TMEM)
      constexpr uint32_t idK = idesc_f32acc(128, DH, C::DS_QMAJOR, true, F16);  // dK
      constexpr uint32_t idQ = C::DQ_T ? idesc_f32acc(128, BM, true, !C::DS_QMAJOR, F16)  // dQ^T
                                       : idesc_f32acc(128, D, true, true, F16);  // dQ
      const uint32_t tS = tmem + C::COL_S, tDP = tmem + C::COL_DP, tP = tmem + C::COL_P;
      const uint32_t tDK = tmem + C::COL_DK, tDV = tmem + C::COL_DV, tDQ = tmem + C::COL_DQ;
      const uint64_t k_kd = desc_kmajor(sK, BN, 0), v_kd = desc_kmajor(sV, BN, 0);
      // the half of d this CTA accumulates starts at 64-column slab dh * DH / 64
      const uint32_t dslab = (uint32_t)(dh * (DH / 64));
      const uint64_t k_mn = desc_mnmajor(sK + dslab * BN * 128, BN, 0);
      const uint64_t q_kd = desc_kmajor(sQ, BM, 0), do_kd = desc_kmajor(sDO, BM, 0);
      const uint64_t q_mn = desc_mnmajor(sQ + dslab * BM * 128, BM, 0);
      const uint64_t do_mn = desc_mnmajor(sDO + dslab * BM * 128, BM, 0);
      // dS^T as the A operand of dK and the B operand of dQ: [key][query] slabs (K-major A,
      // MN-major B), or [query][key] slabs (MN-major A, K-major B)
      const uint64_t ds_a = C::DS_QMAJOR ? desc_mnmajor(sDS, BM, 0) : desc_kmajor(sDS, BN, 0);
      const uint64_t ds_b = C::DS_QMAJOR ? desc_kmajor(sDS, BM, 0) : desc_mnmajor(sDS, BN, 0);
      const uint64_t aug_kd = desc_kmajor(sAUG, BN, 0);
      constexpr uint32_t QSTEP = C::Q_BYTES >> 4, DSSTEP = C::DS_BYTES >> 4;
      auto issue_sdp = [&](int it) -> bool {
        const int st = it % QST;
        if (!mbar_wait(smem_u32(&bars.q_full[st]), (it / QST) & 1, abort, p.timeout_ns))
          return false;
        tc_fence_after();
        const uint32_t qo = st * QSTEP;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_w(tS, k_kd + kmajor_step(BN, kk), q_kd + qo + kmajor_step(BM, kk), idS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_w(tDP, v_kd + kmajor_step(BN, kk), do_kd + qo + kmajor_step(BM, kk), idS,
                    kk > 0);
        if constexpr (C::AUG) {  // S^T - LSE / sm_scale and dP^T - Delta (always bf16 operands)
          constexpr uint32_t idA = idesc_f32acc(128, BM, false, false, false);
          umma_ss_w(tS, aug_kd, aug_kd + kmajor_step(BN, 1 + st), idA, 1);
          umma_ss_w(tDP, aug_kd, aug_kd + kmajor_step(BN, 4 + st), idA, 1);
        }
        umma_commit_w(smem_u32(&bars.s_full));
        return true;
      };
      bool ok = mbar_wait(smem_u32(&bars.kv_full), 0, abort, p.timeout_ns) && issue_sdp(0);
      for (int it = 0; ok && it < n_steps; ++it) {
        const int st = it % QST, bs = it & 1;
        const uint32_t qo = st * QSTEP, dso = bs * DSSTEP;
        if (it + 1 < n_steps) {
          // S^T / dP^T of step it are in registers of the compute warpgroups: overwrite them
          if (!mbar_wait(smem_u32(&bars.s_free), it & 1, abort, p.timeout_ns)) break;
          if (!issue_sdp(it + 1)) break;
        }
        if (!mbar_wait(smem_u32(&bars.p_full), it & 1, abort, p.timeout_ns)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          umma_ts_w(tDV, tP + kk * 8, do_mn + qo + mnmajor_step(kk), idG, (it > 0 || kk > 0));
        if (!C::DS_TMEM)
          umma_commit_w(smem_u32(&bars.p_empty));  // P^T of step it read: the next P may land
        if (!mbar_wait(smem_u32(&bars.ds_full[bs]), (it >> 1) & 1, abort, p.timeout_ns)) break;
        tc_fence_after();
        if constexpr (C::DS_TMEM) {
          // dK = dS^T Q with dS^T from tensor memory; then P^T and dS^T of step it are read
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            umma_ts_w(tDK, tmem + C::COL_DST + kk * 8, q_mn + qo + mnmajor_step(kk), idK,
                      (it > 0 || kk > 0));
          umma_commit_w(smem_u32(&bars.p_empty));
        } else {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            umma_ss_w(tDK,
                      ds_a + dso + (C::DS_QMAJOR ? mnmajor_step(kk) : kmajor_step(BN, kk)),
                      q_mn + qo + mnmajor_step(kk), idK, (it > 0 || kk > 0));
        }
        if (p.with_dq) {
          if (it > 0 &&
              !mbar_wait(smem_u32(&bars.dq_empty), (it - 1) & 1, abort, p.timeout_ns))
            break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            if (C::DQ_T)
              umma_ss_w(tDQ, k_mn + mnmajor_step(kk),
                        ds_b + dso + (C::DS_QMAJOR ? kmajor_step(BM, kk) : mnmajor_step(kk)),
                        idQ, kk > 0);
            else
              umma_ss_w(tDQ, ds_b + dso + mnmajor_step(kk), k_mn + mnmajor_step(kk), idQ, kk > 0);
          }
        }
        umma_commit_w(smem_u32(&bars.q_empty[st]));
        // dq_full after dK as well as dQ: at d_head 64 the drain stages dQ in the dS^T buffer
        // that dK reads
        if (p.with_dq) umma_commit_w(smem_u32(&bars.dq_full));
      }
      umma_commit_w(smem_u32(&bars.dkdv_full));
      // every product this warp issued has completed before tensor memory is released
      umma_commit_w(smem_u32(&bars.mma_drain));
      mbar_wait_drain(smem_u32(&bars.mma_drain), 0, p.timeout_ns);
  }
  } else if (C::BIAS_TMA && warp == C::WARP_BIAS) {
    // ------------------------------------------------------------------ bias tile loader
    // Step it's bias tile (its BM query rows x this CTA's 128 keys, at the bias's own local
    // coordinates; a size-1 batch or head dimension is read at index 0) into the one slot,
    // once the compute warps have read the previous step's (bias_empty). Keys past the
    // bias's extent read as zeros; rows and keys past the sequence are masked by the compute
    // warps whatever they hold.
    if (lane == 0) {
      tma_prefetch_map(&p.tm_bias);
      const int hb = p.b_sh == 0 ? 0 : h, bb = p.b_sb == 0 ? 0 : z;
      const uint32_t bf = smem_u32(&bars.bias_full);
      int loaded = 0;
      for (int it = 0; it < n_steps; ++it) {
        if (it > 0 && !mbar_wait(smem_u32(&bars.bias_empty), (it - 1) & 1, abort, p.timeout_ns))
          break;
        mbar_arrive_expect_tx(bf, C::BIAS_BYTES);
#pragma unroll
        for (int s = 0; s < 2; ++s)
          tma_load_4d(smem_u32(smem + C::OFF_BIAS + s * BM * 128), &p.tm_bias, bf, k_lo + s * 64,
                      q_tile(it) * BM, hb, bb);
        ++loaded;
      }
      if (*abort && loaded > 0)  // the consumers gave up: let the last copy land
        mbar_wait_drain(bf, (loaded - 1) & 1, p.timeout_ns);
    }
  } else if (warp < 4 * C::NCWG) {
    // ------------------------------------------------------------------ P^T / dS^T compute
    // NCWG warpgroups; warpgroup g owns score columns [g*HALF, (g+1)*HALF) of every key row.
    const int g = warp >> 2;
    const int j = (warp & 3) * 32 + lane;  // key row in tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int key = k_lo + j;
    const bool key_ok = key < sv.len_k;
    const float c2 = p.scale_log2;
    const int c_base = g * HALF;
    // d_head 64: drains warpgroup g's 32 columns of the dQ partial of step itd (lanes are
    // query rows, columns d). The warp stages its 32 x 32 fp32 block in rows [32 (warp & 3),
    // +32) of warpgroup g's slab of the dS^T buffer of step itd (128-byte swizzle; the dK / dQ
    // products of that step are complete, and only this warp writes these rows again, two
    // steps later, after waiting for this reduce to read them) and adds it to the fp32
    // accumulator with one TMA tensor reduce-add issued by its lane 0. Query rows past the
    // sequence hold exact zeros (their dS was masked), so whole blocks can be added.
    auto drain_dq = [&](int itd) -> bool {
      if (!mbar_wait(smem_u32(&bars.dq_full), itd & 1, abort, p.timeout_ns)) return false;
      tc_fence_after();
      float v[32];
      ATTN_TMEM_LD_X32(tmem + C::COL_DQ + lane_off + g * 32, reinterpret_cast<uint32_t*>(v));
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.dq_empty));
      uint8_t* stage = smem + C::OFF_DS + (itd & 1) * C::DS_BYTES + g * (C::DS_BYTES / 2) +
                       (warp & 3) * 4096;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(stage + lane * 128 + 16 * (c ^ (lane & 7))) =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      // a block wholly in the zero padding past the head size adds nothing: skip it
      if (lane == 0 && g * 32 < p.d_out) {
        tma_reduce_add_2d(&p.tm_dq, smem_u32(stage), g * 32,
                          (int)(zh * p.rows_q + sv.row0_q + q_tile(itd) * BM + (warp & 3) * 32));
        bulk_commit_group();
      }
      return true;
    };
    bool ok = true;
    for (int it = 0; it < n_steps; ++it) {
      const int st = it % QST, bs = it & 1;
      const int q_lo = q_tile(it) * BM;
      if (!mbar_wait(smem_u32(&bars.s_full), it & 1, abort, p.timeout_ns) ||
          !mbar_wait(smem_u32(&bars.q_full[st]), (it / QST) & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool need_mask = (q_lo + BM > sv.len_q) || (k_lo + BN > sv.len_k) ||
                             (p.causal && k_lo + BN - 1 > q_lo);
      const int q_min = p.causal ? key : 0;  // top-left causal: query q sees key iff q >= key
      // The dS^T buffer of this step was last read by the dK / dQ products of step it - 2,
      // which completed before s_full(it) (the MMA warp commits s_full(it) after issuing
      // them).
      uint8_t* gDS = smem + C::OFF_DS + bs * C::DS_BYTES;
      if (!C::DQ_WARPS && p.with_dq && it >= 2) {
        // this warp's rows of the buffer staged dQ two steps ago: wait for that reduce
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
      }
      // All of this warpgroup's S^T and dP^T columns are fetched behind one wait.
      float sv_all[HALF], dpv_all[HALF];
      if constexpr (HALF == 64) {
        ATTN_TMEM_LD4_X32(tmem + C::COL_S + lane_off + c_base, tmem + C::COL_S + lane_off + c_base + 32,
                          tmem + C::COL_DP + lane_off + c_base,
                          tmem + C::COL_DP + lane_off + c_base + 32,
                          reinterpret_cast<uint32_t*>(sv_all), reinterpret_cast<uint32_t*>(sv_all + 32),
                          reinterpret_cast<uint32_t*>(dpv_all),
                          reinterpret_cast<uint32_t*>(dpv_all + 32));
      } else {
        ATTN_TMEM_LD2_X32(tmem + C::COL_S + lane_off + c_base, tmem + C::COL_DP + lane_off + c_base,
                          reinterpret_cast<uint32_t*>(sv_all), reinterpret_cast<uint32_t*>(dpv_all));
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.s_free));  // the MMA warp may compute the next S^T / dP^T
      // P^T (and at d_head 128 dS^T) of the previous step must have been read by its dV (dK)
      // MMA before this step's lands
      if (it > 0 && !mbar_wait(smem_u32(&bars.p_empty), (it - 1) & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (C::BIAS_TMA && !mbar_wait(smem_u32(&bars.bias_full), it & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int ch = 0; ch < HALF / 32; ++ch) {
        const int c0 = c_base + ch * 32;
        const float* s = sv_all + ch * 32;
        const float* dp = dpv_all + ch * 32;
        uint32_t pp[16], pd[16];
        const uint64_t c2x2 = f2_pack(c2, c2);
        // bias log2(e) of this key and the chunk's 32 query rows (0 off the sequence)
        float bl[BIAS ? 32 : 1];
        if constexpr (BIAS) {
          uint16_t raw[32];
          if constexpr (C::BIAS_TMA) {
            // from the staged tile: this key's column, the chunk's 32 rows (a warp reads 64
            // contiguous bytes of one row at a time)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              raw[e] = *reinterpret_cast<const uint16_t*>(smem + C::OFF_BIAS +
                                                          sw128_offset(c0 + e, j, BM));
            if (ch == HALF / 32 - 1) mbar_arrive(smem_u32(&bars.bias_empty));  // slot read
          } else {
            const uint16_t* bcol = p.bias + z * p.b_sb + h * p.b_sh + key;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int qq = q_lo + c0 + e;
              raw[e] = (key_ok && qq < sv.len_q) ? bcol[(int64_t)qq * p.b_ss] : (uint16_t)0;
            }
          }
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 b = unpack2<F16>((uint32_t)raw[e] | ((uint32_t)raw[e + 1] << 16));
            bl[e] = b.x * 1.4426950408889634f;
            bl[e + 1] = b.y * 1.4426950408889634f;
          }
        }
#pragma unroll
        for (int e4 = 0; e4 < 32; e4 += 4) {
          float pv[4], ds[4], x[4];
          if constexpr (C::AUG && BIAS) {
            // S and dP arrive with LSE / sm_scale and Delta already subtracted; add the bias
            f2_unpack(f2_fma(f2_pack(s[e4], s[e4 + 1]), c2x2, f2_pack(bl[e4], bl[e4 + 1])), x[0],
                      x[1]);
            f2_unpack(f2_fma(f2_pack(s[e4 + 2], s[e4 + 3]), c2x2, f2_pack(bl[e4 + 2], bl[e4 + 3])),
                      x[2], x[3]);
#pragma unroll
            for (int u = 0; u < 4; ++u) pv[u] = ex2_approx(x[u]);
            f2_unpack(f2_mul(f2_pack(pv[0], pv[1]), f2_pack(dp[e4], dp[e4 + 1])), ds[0], ds[1]);
            f2_unpack(f2_mul(f2_pack(pv[2], pv[3]), f2_pack(dp[e4 + 2], dp[e4 + 3])), ds[2], ds[3]);
          } else if constexpr (C::AUG) {
            // S and dP arrive with LSE / sm_scale and Delta already subtracted
            f2_unpack(f2_mul(f2_pack(s[e4], s[e4 + 1]), c2x2), x[0], x[1]);
            f2_unpack(f2_mul(f2_pack(s[e4 + 2], s[e4 + 3]), c2x2), x[2], x[3]);
#pragma unroll
            for (int u = 0; u < 4; ++u) pv[u] = ex2_approx(x[u]);
            f2_unpack(f2_mul(f2_pack(pv[0], pv[1]), f2_pack(dp[e4], dp[e4 + 1])), ds[0], ds[1]);
            f2_unpack(f2_mul(f2_pack(pv[2], pv[3]), f2_pack(dp[e4 + 2], dp[e4 + 3])), ds[2], ds[3]);
          } else {
            const float4 l4 = *reinterpret_cast<const float4*>(&bars.nlse2[st][c0 + e4]);
            const float4 d4 = *reinterpret_cast<const float4*>(&bars.ndelta[st][c0 + e4]);
            float y[4];
            // P = 2^(S c2 [+ bias log2(e)] - LSE2); dS = P (dP - Delta): paired fp32
            // instructions
            uint64_t a01 = f2_pack(l4.x, l4.y), a23 = f2_pack(l4.z, l4.w);
            if constexpr (BIAS) {
              a01 = f2_add(a01, f2_pack(bl[e4], bl[e4 + 1]));
              a23 = f2_add(a23, f2_pack(bl[e4 + 2], bl[e4 + 3]));
            }
            f2_unpack(f2_fma(f2_pack(s[e4], s[e4 + 1]), c2x2, a01), x[0], x[1]);
            f2_unpack(f2_fma(f2_pack(s[e4 + 2], s[e4 + 3]), c2x2, a23), x[2], x[3]);
#pragma unroll
            for (int u = 0; u < 4; ++u) pv[u] = ex2_approx(x[u]);
            f2_unpack(f2_add(f2_pack(dp[e4], dp[e4 + 1]), f2_pack(d4.x, d4.y)), y[0], y[1]);
            f2_unpack(f2_add(f2_pack(dp[e4 + 2], dp[e4 + 3]), f2_pack(d4.z, d4.w)), y[2], y[3]);
            f2_unpack(f2_mul(f2_pack(pv[0], pv[1]), f2_pack(y[0], y[1])), ds[0], ds[1]);
            f2_unpack(f2_mul(f2_pack(pv[2], pv[3]), f2_pack(y[2], y[3])), ds[2], ds[3]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (need_mask) {
              const int qq = q_lo + c0 + e4 + u;
              const bool valid = key_ok && qq < sv.len_q && qq >= q_min;
              pv[u] = valid ? pv[u] : 0.f;
              ds[u] = valid ? ds[u] : 0.f;
            }
          }
          if constexpr (BIAS) {
            if (p.dbias_acc != nullptr && key_ok) {  // a shared bias: sum dS in fp32
              float* acol = p.dbias_acc + z * p.dba_sb + h * p.dba_sh + key;
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int qq = q_lo + c0 + e4 + u;
                if (qq < sv.len_q && qq >= q_min) atomicAdd(acol + (int64_t)qq * p.dba_ss, ds[u]);
              }
            }
          }
          pp[e4 / 2] = pack2<F16>(pv[0], pv[1]);
          pp[e4 / 2 + 1] = pack2<F16>(pv[2], pv[3]);
          pd[e4 / 2] = pack2<F16>(ds[0], ds[1]);
          pd[e4 / 2 + 1] = pack2<F16>(ds[2], ds[3]);
        }
        if constexpr (BIAS) {
          if (p.dbias != nullptr && key_ok) {  // dbias = dS (rounded like the dS operand)
            uint16_t* dcol = p.dbias + z * p.db_sb + h * p.db_sh + key;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int qq = q_lo + c0 + e;
              if (qq < sv.len_q)
                dcol[(int64_t)qq * p.db_ss] = (uint16_t)(pd[e / 2] >> ((e & 1) * 16));
            }
          }
        }
        ATTN_TMEM_ST_X16(tmem + C::COL_P + lane_off + c0 / 2, pp);
        if constexpr (C::DS_TMEM) ATTN_TMEM_ST_X16(tmem + C::COL_DST + lane_off + c0 / 2, pd);
        if constexpr (C::DS_QMAJOR) {
          // [query][key]: one 16-bit element per query row; the warp's 32 keys of one row
          // are 64 contiguous bytes (one wavefront)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            *reinterpret_cast<uint16_t*>(gDS + sw128_offset(c0 + e, j, BM)) =
                (uint16_t)(pd[e >> 1] >> ((e & 1) * 16));
        } else {
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            const uint32_t off = sw128_offset(j, c0 + c8 * 8, BN);
            *reinterpret_cast<uint4*>(gDS + off) =
                make_uint4(pd[c8 * 4 + 0], pd[c8 * 4 + 1], pd[c8 * 4 + 2], pd[c8 * 4 + 3]);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.p_full));
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars.ds_full[bs]));
      // d_head 64: dQ partial of the previous step (its MMA ran while this step's P/dS were
      // formed)
      if (!C::DQ_WARPS && p.with_dq && it > 0 && !drain_dq(it - 1)) {
        ok = false;
        break;
      }
    }
    if (!C::DQ_WARPS && p.with_dq && ok && n_steps > 0) ok = drain_dq(n_steps - 1);
    if (!C::DQ_WARPS && lane == 0) bulk_wait_group0();  // this warp's reduces are complete
    // ---- epilogue: dK = sm_scale * acc, dV = acc; the CTA holds columns [dh DH, +DH) of
    // them, warpgroup g writes its share [g DH / NCWG, +DH / NCWG) of those
    if (ok) ok = mbar_wait(smem_u32(&bars.dkdv_full), 0, abort, p.timeout_ns);
    tc_fence_after();
    // A key tile inside its sequence leaves through shared memory: each warp writes its 32
    // keys of dK and dV (its warpgroup's columns) as rows of the swizzled slabs of its own
    // areas, in the space of the K and V tiles (every product that read them has completed:
    // dkdv_full), and one lane stores each slab with a TMA copy. A tile reaching past the
    // sequence's end is stored row by row (a copy would also write the keys past the end).
    constexpr int CW = C::CW;
    if (C::EPI_TMA && ok && k_lo + BN <= sv.len_k) {
      const float sc = p.sm_scale;
      const uint32_t ak = smem_u32(smem + C::OFF_K + warp * C::EPI_W_BYTES);
      const uint32_t av = ak + 4 * C::NCWG * C::EPI_W_BYTES;
#pragma unroll
      for (int c = 0; c < CW; c += 32) {
        uint32_t a[32], b[32];
        ATTN_TMEM_LD2_X32(tmem + C::COL_DK + lane_off + g * CW + c,
                          tmem + C::COL_DV + lane_off + g * CW + c, a, b);
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 vk, vv;
          vk.x = pack2<F16>(__uint_as_float(a[e]) * sc, __uint_as_float(a[e + 1]) * sc);
          vk.y = pack2<F16>(__uint_as_float(a[e + 2]) * sc, __uint_as_float(a[e + 3]) * sc);
          vk.z = pack2<F16>(__uint_as_float(a[e + 4]) * sc, __uint_as_float(a[e + 5]) * sc);
          vk.w = pack2<F16>(__uint_as_float(a[e + 6]) * sc, __uint_as_float(a[e + 7]) * sc);
          vv.x = pack2<F16>(__uint_as_float(b[e]), __uint_as_float(b[e + 1]));
          vv.y = pack2<F16>(__uint_as_float(b[e + 2]), __uint_as_float(b[e + 3]));
          vv.z = pack2<F16>(__uint_as_float(b[e + 4]), __uint_as_float(b[e + 5]));
          vv.w = pack2<F16>(__uint_as_float(b[e + 6]), __uint_as_float(b[e + 7]));
          const int col = c + e, j = (col % C::EPI_SC) / 8;
          const int pj = C::EPI_SC == 64 ? (j ^ (lane & 7)) : (j ^ ((lane >> 1) & 3));
          const uint32_t off =
              (col / C::EPI_SC) * C::EPI_SLAB_BYTES + lane * (C::EPI_SC * 2) + pj * 16;
          st_shared_v4(ak + off, vk);
          st_shared_v4(av + off, vv);
        }
      }
      fence_proxy_async_smem();  // the areas, written by this warp, to the copy engine
      __syncwarp();
      if (lane == 0) {
        const int row = sv.row0_k + k_lo + (warp & 3) * 32;
#pragma unroll
        for (int s = 0; s < CW / C::EPI_SC; ++s) {
          tma_store_4d(&p.tm_dk, ak + s * C::EPI_SLAB_BYTES, dh * DH + g * CW + s * C::EPI_SC, row,
                       h, sv.batch);
          tma_store_4d(&p.tm_dv, av + s * C::EPI_SLAB_BYTES, dh * DH + g * CW + s * C::EPI_SC, row,
                       h, sv.batch);
        }
        bulk_commit_group();
        bulk_wait_group0();  // complete before the CTA exits
      }
    } else if (ok) {
      const int64_t grow = sv.row0_k + key;
      uint16_t* kr = p.dk + sv.batch * p.dk_sb + h * p.dk_sh + grow * p.dk_ss + dh * DH;
      uint16_t* vr = p.dv + sv.batch * p.dv_sb + h * p.dv_sh + grow * p.dv_ss + dh * DH;
      const float sc = p.sm_scale;
#pragma unroll
      for (int c = g * CW; c < (g + 1) * CW; c += 32) {
        uint32_t a[32], b[32];
        ATTN_TMEM_LD2_X32(tmem + C::COL_DK + lane_off + c, tmem + C::COL_DV + lane_off + c, a, b);
        if (key_ok && dh * DH + c < p.d_out) {  // columns past the head size are zero padding
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 vk, vv;
            vk.x = pack2<F16>(__uint_as_float(a[e]) * sc, __uint_as_float(a[e + 1]) * sc);
            vk.y = pack2<F16>(__uint_as_float(a[e + 2]) * sc, __uint_as_float(a[e + 3]) * sc);
            vk.z = pack2<F16>(__uint_as_float(a[e + 4]) * sc, __uint_as_float(a[e + 5]) * sc);
            vk.w = pack2<F16>(__uint_as_float(a[e + 6]) * sc, __uint_as_float(a[e + 7]) * sc);
            vv.x = pack2<F16>(__uint_as_float(b[e]), __uint_as_float(b[e + 1]));
            vv.y = pack2<F16>(__uint_as_float(b[e + 2]), __uint_as_float(b[e + 3]));
            vv.z = pack2<F16>(__uint_as_float(b[e + 4]), __uint_as_float(b[e + 5]));
            vv.w = pack2<F16>(__uint_as_float(b[e + 6]), __uint_as_float(b[e + 7]));
            *reinterpret_cast<uint4*>(kr + c + e) = vk;
            *reinterpret_cast<uint4*>(vr + c + e) = vv;
          }
        }
      }
    }
  } else if (C::DQ_WARPS && warp >= C::WARP_DRAIN0 && warp < C::WARP_DRAIN0 + 4) {
    // ------------------------------------------------------------------ dQ drain (d_head >= 128)
    // Each drain warp owns the 32 TMEM lanes its warp index reaches (quarter qw) of the dQ^T
    // partial (lanes are d of the CTA's half, the BM columns the step's query rows). It loads
    // them right after the products complete and releases the TMEM columns, stages BM / 32
    // blocks of 32 x 32 fp32 in its own shared-memory area (128-byte swizzle) and adds each to
    // the fp32 accumulator with one TMA reduce-add. Query rows past the sequence hold exact
    // zeros (their dS was masked), so whole blocks can be added; blocks wholly in the zero
    // padding past the head size add nothing and are skipped.
    const int qw = warp & 3;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    bool ok = p.with_dq != 0;
    for (int it = 0; ok && it < n_steps; ++it) {
      if (!mbar_wait(smem_u32(&bars.dq_full), it & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int q_lo = q_tile(it) * BM;
      if constexpr (C::STG_BLOCKS == 1 && C::DQ_BLOCKS > 1) {
        // one 4 KB area a warp: every block of the partial first (the TMEM columns are then
        // free), then block by block, each after the previous reduce-add has read the area
        uint8_t* stage = smem + C::OFF_STG + qw * 4096;
        float v[C::DQ_BLOCKS][32];
#pragma unroll
        for (int b = 0; b < C::DQ_BLOCKS; ++b)
          ATTN_TMEM_LD_X32(tmem + C::COL_DQ + lane_off + 32 * b, reinterpret_cast<uint32_t*>(v[b]));
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.dq_empty));
        const int c0 = dh * DH + qw * 32;
#pragma unroll
        for (int b = 0; b < C::DQ_BLOCKS; ++b) {
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            *reinterpret_cast<float*>(stage + i * 128 + 16 * ((lane >> 2) ^ (i & 7)) +
                                      4 * (lane & 3)) = v[b][i];
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && c0 < p.d_out) {
            tma_reduce_add_2d(&p.tm_dq, smem_u32(stage), c0,
                              (int)(zh * p.rows_q + sv.row0_q + q_lo + b * 32));
            bulk_commit_group();
          }
          __syncwarp();
        }
        continue;
      }
      uint8_t* stage = smem + C::OFF_STG + qw * (C::DQ_BLOCKS * 4096);
      // this warp's previous reduce-adds must have read the area before it is rewritten
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
      // one 32-column block at a time (32 registers of data live)
#pragma unroll
      for (int b = 0; b < C::DQ_BLOCKS; ++b) {
        float v[32];
        ATTN_TMEM_LD_X32(tmem + C::COL_DQ + lane_off + 32 * b, reinterpret_cast<uint32_t*>(v));
        if (b == C::DQ_BLOCKS - 1) {  // the dQ columns are free for the next step's product
          tc_fence_before();
          mbar_arrive(smem_u32(&bars.dq_empty));
        }
        uint8_t* blk = stage + b * 4096;
#pragma unroll
        for (int i = 0; i < 32; ++i)  // row i = query row 32 b + i, column = this lane's d
          *reinterpret_cast<float*>(blk + i * 128 + 16 * ((lane >> 2) ^ (i & 7)) +
                                    4 * (lane & 3)) = v[i];
      }
      fence_proxy_async_smem();
      __syncwarp();
      // blocks: column d = dh DH + 32 qw, query rows 32 b within the step
      const int c0 = dh * DH + qw * 32;
      if (lane == 0 && c0 < p.d_out) {
#pragma unroll
        for (int b = 0; b < C::DQ_BLOCKS; ++b)
          tma_reduce_add_2d(&p.tm_dq, smem_u32(stage + b * 4096), c0,
                            (int)(zh * p.rows_q + sv.row0_q + q_lo + b * 32));
        bulk_commit_group();
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_group0();  // this warp's reduce-adds complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && bars.abort && p.status != nullptr) atomicCAS(p.status, 0, kStatusTimeout);
}

template <int D, bool F16, bool BIAS>
static cudaError_t launch_bwd_main_impl(const BwdParams& p, dim3 grid, cudaStream_t stream) {
  using C = BwdCfg<D, BIAS>;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_main_kernel<D, F16, BIAS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  attn_bwd_main_kernel<D, F16, BIAS><<<grid, C::NTHREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdParams& p, int D, bool f16, bool bias, dim3 grid,
                            cudaStream_t stream) {
  if (bias) {
    if (D == 128)
      return f16 ? launch_bwd_main_impl<128, true, true>(p, grid, stream)
                 : launch_bwd_main_impl<128, false, true>(p, grid, stream);
    return f16 ? launch_bwd_main_impl<64, true, true>(p, grid, stream)
               : launch_bwd_main_impl<64, false, true>(p, grid, stream);
  }
  if (D == 256)
    return f16 ? launch_bwd_main_impl<256, true, false>(p, grid, stream)
               : launch_bwd_main_impl<256, false, false>(p, grid, stream);
  if (D == 128)
    return f16 ? launch_bwd_main_impl<128, true, false>(p, grid, stream)
               : launch_bwd_main_impl<128, false, false>(p, grid, stream);
  return f16 ? launch_bwd_main_impl<64, true, false>(p, grid, stream)
             : launch_bwd_main_impl<64, false, false>(p, grid, stream);
}

int bwd_block_m(int D) {
  return D == 256 ? BwdCfg<256>::BM : D == 128 ? BwdCfg<128>::BM : BwdCfg<64>::BM;
}
int bwd_epilogue_cols(int D) { return D == 256 ? 128 : D / 2; }
int bwd_ctas_per_key_tile(int D) { return D == 256 ? 2 : 1; }
int bwd_block_n() { return 128; }

}  // namespace attn_sm103
