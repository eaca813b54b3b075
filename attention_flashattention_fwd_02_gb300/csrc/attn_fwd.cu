// Forward pass of fused scaled-dot-product attention on sm_103a.
//
// One CTA computes two 128-row query tiles (rows [256 m, 256 m + 256)) of one (batch or
// sequence, head). For every key tile j:
//   S_t = Q_t K_j^T            tcgen05 MMA into TMEM, t = 0, 1
//   online softmax of S_t      one thread per query row (TMEM lane), base-2 exponent
//   O_t += P_t V_j             tcgen05 MMA, P_t read from TMEM where it overwrote S_t
// and at the end O_t / l (16-bit) and LSE = (m + log2 l) ln 2 are stored. Forward keeps LSE
// so that the backward pass can rebuild P (the stash / recompute split of the nvFuser SDPA
// page).
//
// Warp roles (320 threads at d_head 128 and 256, 352 at d_head 64):
//   warps 0..3   softmax, O correction and epilogue of query tile 0 (thread r owns row r)
//   warps 4..7   the same for query tile 1 (d_head 256: warp 4 loads V, 5..7 idle)
//   warp 8       TMA producer: Q_0, Q_1 once, then K_j / V_j into an NST-deep stage ring
//   warp 9       TMEM allocator and MMA issuer (at d_head 64: PV products only)
//   warp 10      d_head 64 only: issuer of the score products S = Q K^T
// Each issuing warp walks its schedule as a whole; one elected lane issues.
// Score buffers rotate: the score tiles S_t(j) are numbered k = 0, 1, ... (S_0(0), S_1(0),
// S_0(1), S_1(1), ...; once one query tile has run out of key tiles, only the other's), and S
// number k lives in TMEM buffer k mod NSB, where its P overwrites it. PV(k) is issued as soon
// as P(k) is published, and S(k + NSB) goes into the buffer PV(k) reads.
//   d_head 128, NSB = 2: one warp issues S(0), S(1), then PV(k), S(k + 2) for every k; the
//     tensor pipe runs them in issue order, so S(k + 2) needs no wait for PV(k). This is the
//     ping-pong of two query tiles.
//   d_head 64, NSB = 3 (TMEM has room for a third 128-column buffer): the products are short
//     and one warp that waits, issues and commits all of them spends more cycles per step
//     than the tensor pipe does, so a second warp issues the score products; S(k) waits until
//     PV(k - NSB) has completed. The next score tile of a query tile is computed while its
//     softmax runs.
// TMEM (512 columns): NSB score buffers of 128 columns, then O_0 and O_1 (D columns each).
//
// d_head 256: O alone takes 256 columns, so a CTA owns one query tile (NQ = 1, 128 rows) and
// two score buffers; Q, one K and one V stage (64 KB each) fill shared memory. K_j is
// released as soon as its score product has completed and V_j once its PV product has, and
// each has a producer warp of its own: K_{j+1} streams in while the softmax of S_j and
// PV_{j-1} run, V_{j+1} while S_{j+2} runs.
//
// Online softmax in base 2 with a lazy rescale: a row's reference maximum m only moves when
// a new row maximum exceeds it by more than 8 (so p <= 2^8); O and l are rescaled by
// 2^(m_old - m_new) only then. The final O / l is the same whatever m was used.
//
// Tile schedule: key tiles at or past the sequence's key length, and (causal, top-left)
// key tiles entirely above a query tile's diagonal, are never loaded or multiplied; element
// masks are applied only on tiles that straddle the diagonal or the key length. Query tiles
// at or past the sequence's query length exit before doing anything (the AOTriton
// padded-varlen kernel prologue returns early the same way).
#include <atomic>

#include "attn_common.cuh"
#include "attn_launch.h"

namespace attn_sm103 {

// BIAS (d_head 64 and 128): the additive bias tile of each score tile (128 query rows x 128
// keys, 16-bit) is staged in shared memory, in slots that belong to one query tile each:
// tile t's bias tiles go to its own slots in its key-tile order, each slot refilled once tile
// t's softmax warps have read its previous tile. At d_head 64 each of the two query tiles has
// one slot (slot t, phase j for key tile j); at d_head 128 a CTA owns one query tile (Q, two
// K/V stages and two bias slots fill shared memory) and that tile has two slots (slot j mod
// 2, phase j / 2). Slots shared by both tiles would let a parity wait pass on the other
// tile's load.
template <int D, bool BIAS = false>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int NQ = (D == 256 || (D == 128 && BIAS)) ? 1 : 2;  // query tiles per CTA
  // d_head 128 with a bias: one query tile, one K and one V stage released separately (as at
  // d_head 256) and four bias slots, so that the bias tiles, read once from DRAM, are loaded
  // four key tiles ahead
  static constexpr bool ONE_KV = (D == 256) || (D == 128 && BIAS);
  // d_head 64 with a bias: two K/V stages instead of four, for two bias slots per query tile
  static constexpr int NST = ONE_KV ? 1 : (D == 128 || BIAS) ? 2 : 4;
  static constexpr bool SPLIT_KV = ONE_KV;   // K and V released and loaded separately
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int NBS = BIAS ? 4 : 0;  // bias slots
  static constexpr int BS_T = BIAS ? NBS / NQ : 1; // bias slots per query tile (1: no bias role)
  static constexpr int B_BYTES = BM * BN * 2;      // one bias slot
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = NQ * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NST * KV_BYTES;
  static constexpr int OFF_B = OFF_V + NST * KV_BYTES;
  // Epilogue staging (where shared memory has room: not with a bias): each softmax warp owns
  // OST_SLABS slabs of 32 rows x 64 columns (4 KB, 128-byte swizzle) that it fills from TMEM
  // and copies out with TMA stores.
  static constexpr int OST_SLABS = (D == 256) ? 2 : 1;
  static constexpr int OST_W_BYTES = OST_SLABS * 4096;
  static constexpr int OFF_OST = OFF_B + NBS * B_BYTES;
  static constexpr bool O_TMA = !BIAS;
  static constexpr int SMEM_BYTES = OFF_OST + (O_TMA ? NQ * 4 * OST_W_BYTES : 0) + 1024;
  // Split grids: one partial-result slot holds O (unnormalised, fp32, as [D / 4][NQ * BM][4]:
  // a warp's 32 rows of 4 columns are 512 contiguous bytes) and the rows' running maximum and
  // sum.
  static constexpr int SLOT_FLOATS = NQ * BM * (D + 2);
  static constexpr int NSB = (D == 64) ? 3 : 2;  // rotating score / P buffers
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O0 = NSB * 128, COL_O1 = NSB * 128 + (NQ == 2 ? D : 0);
  static_assert(COL_O0 + NQ * D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB per CTA)");
  static constexpr bool SPLIT_ISSUE = (NSB == 3);  // separate S and PV issuing warps
  static constexpr int WARP_PRODUCER = 8, WARP_MMA = 9, WARP_SMMA = 10;
  static constexpr int WARP_VPROD = 4;  // V producer (SPLIT_KV only; a tile-1 warp otherwise)
  static_assert(!SPLIT_KV || NQ == 1, "the V producer takes a warp of query tile 1");
  static constexpr int WARP_BIAS = SPLIT_ISSUE ? 11 : 10;  // bias producer (BIAS only)
  static constexpr int NTHREADS = (SPLIT_ISSUE ? 352 : 320) + (BIAS ? 32 : 0);
};

constexpr int NCLC = 4;  // work-stealing response slots

template <int NST, int NSB>
struct FwdBars {
  alignas(16) uint4 clc_resp[NCLC];      // work-stealing responses (cluster launch control)
  uint64_t clc_full[NCLC], clc_empty[NCLC];
  uint64_t tsync;         // the softmax warps meet (a block with one tile past the end; the
                          // parts of a block split over CTAs)
  uint64_t q_full;
  uint64_t q_empty;       // the score products of a block have read Q (persistent grids)
  uint64_t k_full[NST], v_full[NST], kv_empty[NST];
  uint64_t k_empty[NST];  // SPLIT_KV: K stage free (kv_empty then frees the V stage)
  uint64_t s_full[NSB], p_full[NSB], buf_free[NSB];
  uint64_t o_done[2][2];  // PV_t(j) completed: barrier [t][j mod 2] (see the rescale wait)
  uint64_t b_full[4], b_empty[4];  // bias slots (NBS of them used)
  uint64_t mma_drain[2];           // completion of each issuing warp's last products
  uint32_t tmem_base;
  int abort;
  int merge_last;  // split grids: this CTA finished a block's last part and merges its parts
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Issue order of the score tiles of the two query tiles (n0, n1 key tiles each): S number k
// belongs to query tile t_of(k) and key tile j_of(k); k_of is the inverse.
struct ScoreOrder {
  int n_min, t_long, total;
  __device__ ScoreOrder(int n0, int n1)
      : n_min(min(n0, n1)), t_long(n1 > n0 ? 1 : 0), total(n0 + n1) {}
  __device__ __forceinline__ int k_of(int t, int j) const {
    return j < n_min ? 2 * j + t : n_min + j;
  }
  __device__ __forceinline__ int t_of(int k) const { return k < 2 * n_min ? (k & 1) : t_long; }
  __device__ __forceinline__ int j_of(int k) const { return k < 2 * n_min ? (k >> 1) : k - n_min; }
};

// Number of key tiles a query tile [q_lo, q_hi) must visit.
__device__ __forceinline__ int key_tiles(int q_lo, int q_hi, int len_k, int causal, int BN) {
  if (q_hi <= q_lo) return 0;
  int n = (len_k + BN - 1) / BN;
  if (causal) n = min(n, (q_hi - 1) / BN + 1);
  return n;
}

// Work item of a CTA: one query block (NQ tiles of 128 rows) of one (unit, head) pair.
struct FwdItem {
  SeqView sv;
  int z, h, blk_lo;
  int q_lo[2], q_hi[2], n_t[2], n_max;
  int j0;        // first key tile (a split grid's segment of the key range; else 0)
  bool partial;  // the segment is not the whole key range: the epilogue merges partial results
};

template <int D, bool F16, bool BIAS, bool SPLIT>
__global__ void __launch_bounds__((D == 64 ? 352 : 320) + (BIAS ? 32 : 0), 1)
    attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D, BIAS>;
  constexpr int BM = C::BM, BN = C::BN, NST = C::NST, NSB = C::NSB;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdBars<NST, NSB> bars;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work items: (unit, head) pairs x query blocks, numbered in the launch's CTA order
  // (grid_pos); causal blocks are visited from the last (heaviest) one down. A CTA starts with
  // item blockIdx.x and then takes, with work stealing (p.clc: a grid of one CTA per item), the
  // item of a CTA whose launch it cancelled, or else items blockIdx.x + gridDim.x, ... (a
  // grid of fewer CTAs than items). Every role walks the same items; the rings (K/V stages,
  // score buffers, O completions, bias slots) are indexed by running counts over the CTA's
  // items, so a CTA's pipeline runs on from one item into the next: the next block's Q loads
  // once the score products of the block before are done (q_empty). O_t needs no barrier of
  // its own: the next block's first PV_t waits for P_t(0), which tile t's warps publish only
  // after their epilogue has read O_t.
  const int n_items = p.uh * p.tiles;
  // Split grid (p.split): the units (item, key tile) of all items, item-major, are cut into
  // gridDim.x equal ranges, one per CTA; a CTA's items are the ones its range meets, each over
  // the part of the key range inside the range.
  // (computed where used: a first item held in a register from here on measured 2-3 % slower
  // in the unsplit kernels)
  auto u_lo = [&]() { return (int64_t)blockIdx.x * p.n_units / gridDim.x; };
  auto u_hi = [&]() { return ((int64_t)blockIdx.x + 1) * p.n_units / gridDim.x; };
  auto first_item = [&]() { return SPLIT ? (int)(u_lo() / p.nk) : (int)blockIdx.x; };
  // Readers of each work-stealing response (one arrival each on its slot's empty barrier):
  // the MMA and S issuers, the V and bias producers, each softmax warp. The producer, which
  // makes the requests, reads each response before it reuses the slot.
  constexpr int CLC_READERS = 1 + (C::SPLIT_ISSUE ? 1 : 0) + (C::SPLIT_KV ? 1 : 0) +
                              (BIAS ? 1 : 0) + 4 * C::NQ;
  enum { kProducer, kLane, kWarp };
  // The item after `item` for a role, or -1 when there is none (or a wait gave up). ci counts
  // the responses this role has read: response ci sits in slot ci mod NCLC, phase
  // (ci / NCLC) mod 2 of its full barrier.
  auto next_item = [&](int item, int& ci, int who) -> int {
    if (SPLIT) return (int64_t)(item + 1) * p.nk < u_hi() ? item + 1 : -1;
    if (!p.clc) return item + (int)gridDim.x < n_items ? item + (int)gridDim.x : -1;
    const int slot = ci % NCLC;
    const uint32_t full = smem_u32(&bars.clc_full[slot]);
    volatile int* ab = &bars.abort;
    const bool landed = who == kWarp ? mbar_wait_warp(full, (ci / NCLC) & 1, ab, p.timeout_ns)
                                     : mbar_wait(full, (ci / NCLC) & 1, ab, p.timeout_ns);
    if (!landed) return -1;
    const int nx = clc_cancelled_x(smem_u32(&bars.clc_resp[slot]));
    if (who == kWarp) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.clc_empty[slot]));
    } else if (who == kLane) {
      mbar_arrive(smem_u32(&bars.clc_empty[slot]));
    }
    ++ci;
    return nx;
  };
  auto decode_item = [&](int item, FwdItem& w) -> bool {
    const GridPos gp = grid_pos(item, p.tiles, p.uh, p.group);
    w.h = gp.zh % p.H;
    w.z = gp.zh / p.H;
    const int m_blk = p.causal ? p.tiles - 1 - gp.rank : gp.rank;
    if (!decode_seq(p.seq, w.z, threadIdx.x == 0 ? p.status : nullptr, w.sv)) return false;
    w.blk_lo = m_blk * (C::NQ * BM);
    if (w.blk_lo >= w.sv.len_q) return false;  // past this sequence's queries
#pragma unroll
    for (int t = 0; t < 2; ++t) {  // with one query tile per CTA, tile 1 is empty
      w.q_lo[t] = w.blk_lo + t * BM;
      w.q_hi[t] = t < C::NQ ? min(w.q_lo[t] + BM, w.sv.len_q) : w.q_lo[t];
      w.n_t[t] = key_tiles(w.q_lo[t], w.q_hi[t], w.sv.len_k, p.causal, BN);
    }
    w.j0 = 0;
    w.partial = false;
    if (SPLIT) {  // non-causal dense grids: every tile of the block has the nk key tiles
      const int64_t base = (int64_t)item * p.nk;
      const int j_lo = (int)(max(u_lo(), base) - base);
      const int j_hi = (int)(min(u_hi(), base + p.nk) - base);
      w.j0 = j_lo;
      w.partial = j_lo > 0 || j_hi < p.nk;
#pragma unroll
      for (int t = 0; t < 2; ++t) w.n_t[t] = w.n_t[t] > 0 ? j_hi - j_lo : 0;
    }
    w.n_max = max(w.n_t[0], w.n_t[1]);
    return true;
  };

  uint8_t* smem = align1024(smem_raw);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q);
  const uint32_t sK = smem_u32(smem + C::OFF_K);
  const uint32_t sV = smem_u32(smem + C::OFF_V);

  if (threadIdx.x == 0) {
    bars.abort = 0;
    for (int i = 0; i < NCLC; ++i) {
      mbar_init(smem_u32(&bars.clc_full[i]), 1);
      mbar_init(smem_u32(&bars.clc_empty[i]), CLC_READERS);
    }
    mbar_init(smem_u32(&bars.tsync), 4 * C::NQ);
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.q_empty), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.kv_empty[s]), 1);
      mbar_init(smem_u32(&bars.k_empty[s]), 1);
    }
    for (int b = 0; b < NSB; ++b) {
      mbar_init(smem_u32(&bars.s_full[b]), 1);
      mbar_init(smem_u32(&bars.p_full[b]), 128);
      mbar_init(smem_u32(&bars.buf_free[b]), 1);
    }
    for (int r = 0; r < 4; ++r) mbar_init(smem_u32(&bars.o_done[r >> 1][r & 1]), 1);
    for (int t = 0; t < 4; ++t) {
      mbar_init(smem_u32(&bars.b_full[t]), 1);
      mbar_init(smem_u32(&bars.b_empty[t]), 128);
    }
    for (int t = 0; t < 2; ++t) mbar_init(smem_u32(&bars.mma_drain[t]), 1);
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
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
      const uint32_t qb = smem_u32(&bars.q_full);
      int kv_g = 0, q_n = 0;  // key tiles and query blocks loaded so far
      int last_g[NST];        // last key tile (running count) loaded into each stage (-1: none)
#pragma unroll
      for (int st = 0; st < NST; ++st) last_g[st] = -1;
      bool go = true;
      int ci = 0, issued = 0;  // work-stealing responses read, requests made
      for (int item = first_item(); go && item >= 0;
           item = go ? next_item(item, ci, kProducer) : -1) {
        if (p.clc) {
          // request the item after this one now, so that the answer is in when this one ends;
          // the slot is free once every reader has read the response it held before
          const int slot = issued % NCLC, u = issued / NCLC;
          if (u > 0 && !mbar_wait(smem_u32(&bars.clc_empty[slot]), (u - 1) & 1, abort,
                                  p.timeout_ns))
            break;
          mbar_arrive_expect_tx(smem_u32(&bars.clc_full[slot]), 16);
          clc_try_cancel(smem_u32(&bars.clc_resp[slot]), smem_u32(&bars.clc_full[slot]));
          ++issued;
        }
        FwdItem w;
        if (!decode_item(item, w) || w.n_max == 0) continue;
        // the previous block's score products have read Q
        if (q_n > 0 && !mbar_wait(smem_u32(&bars.q_empty), (q_n - 1) & 1, abort, p.timeout_ns))
          break;
        mbar_arrive_expect_tx(qb, C::NQ * C::Q_BYTES);
#pragma unroll
        for (int t = 0; t < C::NQ; ++t)
#pragma unroll
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(sQ + t * C::Q_BYTES + s * BM * 128, &p.tm_q, qb, s * 64,
                        w.sv.row0_q + w.q_lo[t], w.h, w.sv.batch);
        ++q_n;
        for (int j = 0; j < w.n_max; ++j) {
          const int g = kv_g + j, st = g % NST;
          // failure-detection test: no key tile from this one on is loaded (skipping only this
          // one would leave the next wait on its stage aiming at a phase that never completes)
          if (j == p.withhold_tile) {
            go = false;
            break;
          }
          const uint32_t empty =
              C::SPLIT_KV ? smem_u32(&bars.k_empty[st]) : smem_u32(&bars.kv_empty[st]);
          if (g >= NST && !mbar_wait(empty, ((g / NST) - 1) & 1, abort, p.timeout_ns)) {
            go = false;
            break;
          }
          last_g[st] = g;
          const int krow = w.sv.row0_k + ((SPLIT ? w.j0 : 0) + j) * BN;
          const uint32_t kb = smem_u32(&bars.k_full[st]);
          mbar_arrive_expect_tx(kb, C::KV_BYTES);
#pragma unroll
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(sK + st * C::KV_BYTES + s * BN * 128, &p.tm_k, kb, s * 64, krow, w.h,
                        w.sv.batch);
          // the tile that will next fill this stage: into L2 now, so that its load is not a
          // DRAM round trip when the stage frees up
          const bool pf = j + NST < w.n_max && j + NST != p.withhold_tile;
          if (pf) {
#pragma unroll
            for (int s = 0; s < D / 64; ++s)
              tma_prefetch_l2_4d(&p.tm_k, s * 64, krow + NST * BN, w.h, w.sv.batch);
          }
          if (C::SPLIT_KV) continue;  // V has its own producer warp
          const uint32_t vb = smem_u32(&bars.v_full[st]);
          mbar_arrive_expect_tx(vb, C::KV_BYTES);
#pragma unroll
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(sV + st * C::KV_BYTES + s * BN * 128, &p.tm_v, vb, s * 64, krow, w.h,
                        w.sv.batch);
          if (pf) {
#pragma unroll
            for (int s = 0; s < D / 64; ++s)
              tma_prefetch_l2_4d(&p.tm_v, s * 64, krow + NST * BN, w.h, w.sv.batch);
          }
        }
        kv_g += w.n_max;
      }
      // a request whose response was not read: let it land before the CTA exits
      if (issued > ci)
        mbar_wait_drain(smem_u32(&bars.clc_full[(issued - 1) % NCLC]),
                        ((issued - 1) / NCLC) & 1, p.timeout_ns);
      if (*abort) {  // the consumers gave up: let this lane's copies land before exiting
        if (q_n > 0) mbar_wait_drain(qb, (q_n - 1) & 1, p.timeout_ns);
#pragma unroll
        for (int st = 0; st < NST; ++st)
          if (last_g[st] >= 0) {
            mbar_wait_drain(smem_u32(&bars.k_full[st]), (last_g[st] / NST) & 1, p.timeout_ns);
            if (!C::SPLIT_KV)
              mbar_wait_drain(smem_u32(&bars.v_full[st]), (last_g[st] / NST) & 1, p.timeout_ns);
          }
      }
    }
  } else if (C::SPLIT_KV && warp == C::WARP_VPROD) {
    // ------------------------------------------------------------------ V producer (d_head 256)
    if (lane == 0) {
      int kv_g = 0;
      int last_g[NST];
#pragma unroll
      for (int st = 0; st < NST; ++st) last_g[st] = -1;
      bool go = true;
      int ci = 0;
      for (int item = first_item(); go && item >= 0; item = go ? next_item(item, ci, kLane) : -1) {
        FwdItem w;
        if (!decode_item(item, w) || w.n_max == 0) continue;
        for (int j = 0; j < w.n_max; ++j) {
          const int g = kv_g + j, st = g % NST;
          if (j == p.withhold_tile ||
              (g >= NST && !mbar_wait(smem_u32(&bars.kv_empty[st]), ((g / NST) - 1) & 1, abort,
                                      p.timeout_ns))) {
            go = false;
            break;
          }
          last_g[st] = g;
          const uint32_t vb = smem_u32(&bars.v_full[st]);
          mbar_arrive_expect_tx(vb, C::KV_BYTES);
#pragma unroll
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(sV + st * C::KV_BYTES + s * BN * 128, &p.tm_v, vb, s * 64,
                        w.sv.row0_k + ((SPLIT ? w.j0 : 0) + j) * BN, w.h, w.sv.batch);
          if (j + NST < w.n_max && j + NST != p.withhold_tile) {
#pragma unroll
            for (int s = 0; s < D / 64; ++s)
              tma_prefetch_l2_4d(&p.tm_v, s * 64,
                                 w.sv.row0_k + ((SPLIT ? w.j0 : 0) + j + NST) * BN, w.h,
                                 w.sv.batch);
          }
        }
        kv_g += w.n_max;
      }
      if (*abort)
#pragma unroll
        for (int st = 0; st < NST; ++st)
          if (last_g[st] >= 0)
            mbar_wait_drain(smem_u32(&bars.v_full[st]), (last_g[st] / NST) & 1, p.timeout_ns);
    }
  } else if (BIAS && warp == C::WARP_BIAS) {
    // ------------------------------------------------------------------ bias producer
    // bias tiles in score-tile order: key tile j of query tile t (running count b over the
    // tile's key tiles) into slot t * BS_T + b mod BS_T (phase b / BS_T), each slot refilled
    // once tile t's softmax warps have read its previous tile (they wait on nothing this warp
    // does afterwards). A warp of its own, so that its waits never share a warp with the K/V
    // producer's. Every unit (batch, or sequence of a compact batch) finds its bias block at
    // offset 0 of its own slice of the bias's first dimension, so the key coordinate (the
    // innermost, which a TMA copy needs 16-byte aligned) is always a multiple of 64 elements.
    if (lane == 0) {
      tma_prefetch_map(&p.tm_b);
      const uint32_t sB = smem_u32(smem + C::OFF_B);
      int b_g[2] = {0, 0};        // bias tiles of each query tile loaded so far
      int last_ph[4] = {-1, -1, -1, -1};  // last phase loaded into each slot
      bool go = true;
      int ci = 0;
      for (int item = first_item(); go && item >= 0; item = go ? next_item(item, ci, kLane) : -1) {
        FwdItem w;
        if (!decode_item(item, w) || w.n_max == 0) continue;
        const ScoreOrder order(w.n_t[0], w.n_t[1]);
        const int hb = p.bias_h_bcast ? 0 : w.h, bb = p.bias_b_bcast ? 0 : w.z;
        for (int k = 0; k < order.total; ++k) {
          const int t = order.t_of(k), j = order.j_of(k);
          const int gb = b_g[t] + j;
          const int slot = t * C::BS_T + gb % C::BS_T, ph = gb / C::BS_T;
          if (ph >= 1 &&
              !mbar_wait(smem_u32(&bars.b_empty[slot]), (ph - 1) & 1, abort, p.timeout_ns)) {
            go = false;
            break;
          }
          const uint32_t bf = smem_u32(&bars.b_full[slot]);
          mbar_arrive_expect_tx(bf, C::B_BYTES);
#pragma unroll
          for (int s = 0; s < 2; ++s)
            tma_load_4d(sB + slot * C::B_BYTES + s * BM * 128, &p.tm_b, bf, ((SPLIT ? w.j0 : 0) + j) * BN + s * 64,
                        w.q_lo[t], hb, bb);
          last_ph[slot] = ph;
        }
        b_g[0] += w.n_t[0];
        b_g[1] += w.n_t[1];
      }
      if (*abort)  // let the copies in flight land before exiting
#pragma unroll
        for (int sl = 0; sl < C::NBS; ++sl)
          if (last_ph[sl] >= 0)
            mbar_wait_drain(smem_u32(&bars.b_full[sl]), last_ph[sl] & 1, p.timeout_ns);
    }
  } else if (warp == C::WARP_MMA) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idO = idesc_f32acc(128, D, false, true, F16);
    constexpr uint32_t idS = idesc_f32acc(128, BN, false, false, F16);
    const uint64_t v_desc = desc_mnmajor(sV, BN, 0);
    const uint64_t q_desc = desc_kmajor(sQ, BM, 0);
    const uint64_t k_desc = desc_kmajor(sK, BN, 0);
    int kv_g = 0, s_g = 0, q_n = 0;  // key tiles, score tiles, query blocks of earlier items
    int pv_g0 = 0, pv_g1 = 0;        // PV products of query tile 0 / 1 in earlier items
    int k_seen = -1, v_seen = -1;    // key tiles (running count) whose K / V were seen full
    bool ok = true;
    int ci = 0;
    for (int item = first_item(); ok && item >= 0; item = ok ? next_item(item, ci, kWarp) : -1) {
      FwdItem w;
      if (!decode_item(item, w) || w.n_max == 0) continue;
      const ScoreOrder order(w.n_t[0], w.n_t[1]);
      const int total = order.total;
      // S number k of this item into buffer (s_g + k) mod NSB (single-issuer schedule); false
      // when a wait gave up
      auto issue_s = [&](int k) -> bool {
        const int t = order.t_of(k), j = order.j_of(k);
        const int g = kv_g + j, st = g % NST;
        if (g != k_seen) {
          if (!mbar_wait_warp(smem_u32(&bars.k_full[st]), (g / NST) & 1, abort, p.timeout_ns))
            return false;
          k_seen = g;
          tc_fence_after();
        }
        const int bsel = (s_g + k) % NSB;
        const uint32_t tS = tmem + bsel * 128;
        const uint64_t qd = q_desc + (uint32_t)(t * (C::Q_BYTES >> 4));
        const uint64_t kd = k_desc + (uint32_t)(st * (C::KV_BYTES >> 4));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_w(tS, qd + kmajor_step(BM, kk), kd + kmajor_step(BN, kk), idS, kk > 0);
        umma_commit_w(smem_u32(&bars.s_full[bsel]));
        // one query tile: K_j has no other reader once this product has completed
        if (C::SPLIT_KV) umma_commit_w(smem_u32(&bars.k_empty[st]));
        if (k == total - 1) umma_commit_w(smem_u32(&bars.q_empty));  // Q read for the last time
        return true;
      };
      if (!C::SPLIT_ISSUE) {
        ok = mbar_wait_warp(smem_u32(&bars.q_full), q_n & 1, abort, p.timeout_ns);
        for (int k = 0; ok && k < min(NSB, total); ++k) ok = issue_s(k);
      }
      for (int k = 0; ok && k < total; ++k) {
        const int t = order.t_of(k), j = order.j_of(k);
        const int g = kv_g + j, st = g % NST, gs = s_g + k, bsel = gs % NSB;
        if (g != v_seen) {
          if (!mbar_wait_warp(smem_u32(&bars.v_full[st]), (g / NST) & 1, abort, p.timeout_ns)) {
            ok = false;
            break;
          }
          v_seen = g;
        }
        if (!mbar_wait_warp(smem_u32(&bars.p_full[bsel]), (gs / NSB) & 1, abort, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tS = tmem + bsel * 128;
        const uint32_t tO = tmem + (t ? C::COL_O1 : C::COL_O0);
        const uint64_t vd = v_desc + (uint32_t)(st * (C::KV_BYTES >> 4));
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ts_w(tO, tS + kk * 8, vd + mnmajor_step(kk), idO, (j > 0 || kk > 0));
        umma_commit_w(smem_u32(&bars.o_done[t][((t ? pv_g1 : pv_g0) + j) & 1]));
        if (C::SPLIT_ISSUE) umma_commit_w(smem_u32(&bars.buf_free[bsel]));
        // Stage st is free once the last product reading V_j is done; the score products that
        // read K_j finished before their P was published, hence before this PV.
        if (k + 1 == total || order.j_of(k + 1) != j) umma_commit_w(smem_u32(&bars.kv_empty[st]));
        if (!C::SPLIT_ISSUE && k + NSB < total) ok = issue_s(k + NSB);
      }
      s_g += total;
      kv_g += w.n_max;
      ++q_n;
      pv_g0 += w.n_t[0];
      pv_g1 += w.n_t[1];
    }
    // every product this warp issued has completed before tensor memory is released
    umma_commit_w(smem_u32(&bars.mma_drain[0]));
    mbar_wait_drain(smem_u32(&bars.mma_drain[0]), 0, p.timeout_ns);
  } else if (C::SPLIT_ISSUE && warp == C::WARP_SMMA) {
    // ------------------------------------------------------------------ S issuer (d_head 64)
    constexpr uint32_t idS = idesc_f32acc(128, BN, false, false, F16);
    const uint64_t q_desc = desc_kmajor(sQ, BM, 0);
    const uint64_t k_desc = desc_kmajor(sK, BN, 0);
    int kv_g = 0, s_g = 0, q_n = 0;
    int k_seen = -1;  // key tile (running count) whose K stage was last seen full
    bool ok = true;
    int ci = 0;
    for (int item = first_item(); ok && item >= 0; item = ok ? next_item(item, ci, kWarp) : -1) {
      FwdItem w;
      if (!decode_item(item, w) || w.n_max == 0) continue;
      const ScoreOrder order(w.n_t[0], w.n_t[1]);
      const int total = order.total;
      ok = mbar_wait_warp(smem_u32(&bars.q_full), q_n & 1, abort, p.timeout_ns);
      for (int k = 0; ok && k < total; ++k) {
        const int t = order.t_of(k), j = order.j_of(k);
        const int g = kv_g + j, st = g % NST, gs = s_g + k, bsel = gs % NSB;
        // PV(gs - NSB) read this buffer; its release cannot run a phase ahead, since the next
        // release of the buffer needs S(gs), issued below.
        if (gs >= NSB &&
            !mbar_wait_warp(smem_u32(&bars.buf_free[bsel]), ((gs - NSB) / NSB) & 1, abort,
                       p.timeout_ns)) {
          ok = false;
          break;
        }
        if (g != k_seen) {
          if (!mbar_wait_warp(smem_u32(&bars.k_full[st]), (g / NST) & 1, abort, p.timeout_ns)) {
            ok = false;
            break;
          }
          k_seen = g;
        }
        tc_fence_after();
        const uint32_t tS = tmem + bsel * 128;
        const uint64_t qd = q_desc + (uint32_t)(t * (C::Q_BYTES >> 4));
        const uint64_t kd = k_desc + (uint32_t)(st * (C::KV_BYTES >> 4));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_w(tS, qd + kmajor_step(BM, kk), kd + kmajor_step(BN, kk), idS, kk > 0);
        umma_commit_w(smem_u32(&bars.s_full[bsel]));
        if (k == total - 1) umma_commit_w(smem_u32(&bars.q_empty));  // Q read for the last time
      }
      s_g += total;
      kv_g += w.n_max;
      ++q_n;
    }
    umma_commit_w(smem_u32(&bars.mma_drain[1]));
    mbar_wait_drain(smem_u32(&bars.mma_drain[1]), 0, p.timeout_ns);
  } else if (warp < 4 * C::NQ) {
    // ------------------------------------------------------------------ softmax / epilogue
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int r = (warp & 3) * 32 + lane;    // row in tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tOt = tmem + (t ? C::COL_O1 : C::COL_O0) + lane_off;
    const float c2 = p.scale_log2;
    int s_g = 0, pv_g = 0;  // score tiles of earlier items; PVs of this query tile in them
    bool ok = true;
    int ci = 0, n_sync = 0;  // work-stealing responses read; meetings of the softmax warps
    // every softmax warp of the CTA meets here (a bounded wait: a warp that gave up leaves
    // the others free); false when the wait gave up
    auto tile_meet = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.tsync));
      const bool met = mbar_wait_warp(smem_u32(&bars.tsync), n_sync & 1, abort, p.timeout_ns);
      ++n_sync;
      return met;
    };
    for (int item = first_item(); ok && item >= 0; item = ok ? next_item(item, ci, kWarp) : -1) {
      int q_lo, n, len_k, j0;
      bool one_empty;  // a query block with one tile past the sequence's end
      ScoreOrder order(0, 0);
      {
      FwdItem w;
      if (!decode_item(item, w)) continue;
      if (w.n_max == 0) {  // no visible keys: O = 0, LSE = -inf on the valid rows
        const int row = w.blk_lo + (int)threadIdx.x;
        if (row < w.sv.len_q) {
          const int64_t grow = w.sv.row0_q + row;
          uint16_t* orow = p.o + w.sv.batch * p.o_sb + w.h * p.o_sh + grow * p.o_ss;
          for (int d = 0; d < p.d_out; d += 8)
            *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
          p.lse[w.sv.batch * p.l_sb + w.h * p.l_sh + grow * p.l_ss] = -INFINITY;
        }
        continue;
      }
      order = ScoreOrder(w.n_t[0], w.n_t[1]);
      q_lo = t ? w.q_lo[1] : w.q_lo[0];
      n = t ? w.n_t[1] : w.n_t[0];
      len_k = w.sv.len_k;
      j0 = SPLIT ? w.j0 : 0;
      one_empty = C::NQ == 2 && min(w.n_t[0], w.n_t[1]) == 0;
      }
      const int row = q_lo + r;  // local query index
      float m_use = -INFINITY, l = 0.f;
      for (int j = 0; ok && j < n; ++j) {
        const int gs = s_g + order.k_of(t, j), bsel = gs % NSB;
        const uint32_t tSt = tmem + bsel * 128 + lane_off;
        if (!mbar_wait_warp(smem_u32(&bars.s_full[bsel]), (gs / NSB) & 1, abort, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[BN];
        static_assert(BN == 128, "one four-way TMEM load covers the score row");
        ATTN_TMEM_LD4_X32(tSt, tSt + 32, tSt + 64, tSt + 96, reinterpret_cast<uint32_t*>(s),
                          reinterpret_cast<uint32_t*>(s + 32), reinterpret_cast<uint32_t*>(s + 64),
                          reinterpret_cast<uint32_t*>(s + 96));
        if constexpr (BIAS) {
          // s <- s c2 + bias log2(e): the scores in base-2 units, bias included
          const int gb = pv_g + j;  // this tile's key tiles so far (the bias producer's count)
          const int slot = t * C::BS_T + gb % C::BS_T;
          if (!mbar_wait_warp(smem_u32(&bars.b_full[slot]), (gb / C::BS_T) & 1, abort,
                         p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint8_t* brow = smem + C::OFF_B + slot * C::B_BYTES + r * 128;
          const uint64_t c2x2b = f2_pack(c2, c2), l2e = f2_pack(1.4426950408889634f, 1.4426950408889634f);
#pragma unroll
          for (int sl = 0; sl < 2; ++sl)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const uint4 wv4 = *reinterpret_cast<const uint4*>(brow + sl * BM * 128 +
                                                                16 * (ch ^ (r & 7)));
              const uint32_t wv[4] = {wv4.x, wv4.y, wv4.z, wv4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int c = sl * 64 + ch * 8 + 2 * e;
                const float2 bv = unpack2<F16>(wv[e]);
                f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), c2x2b, f2_mul(f2_pack(bv.x, bv.y), l2e)),
                          s[c], s[c + 1]);
              }
            }
          mbar_arrive(smem_u32(&bars.b_empty[slot]));
        }
        // with a bias the scores are already scaled
        const float cs = BIAS ? 1.f : c2;
        const int k0 = (j0 + j) * BN;
        if (k0 + BN > len_k || (p.causal && k0 + BN - 1 > q_lo)) {
          const int kmax = p.causal ? min(row, len_k - 1) : len_k - 1;
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (k0 + c > kmax) s[c] = -INFINITY;
        }
        // row maximum: four independent chains of three-input max
        float mx0 = fmax3(s[0], s[1], s[2]), mx1 = fmax3(s[3], s[4], s[5]);
        float mx2 = fmax3(s[6], s[7], s[8]), mx3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
        for (int c = 12; c + 8 <= BN; c += 8) {
          mx0 = fmax3(mx0, s[c], s[c + 1]);
          mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
          mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
          mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
        }
        mx0 = fmax3(mx0, s[BN - 4], s[BN - 3]);
        mx1 = fmax3(mx1, s[BN - 2], s[BN - 1]);
        const float mxs = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * cs;
        float m_new = m_use, scale = 1.f;
        if (mxs > m_use + 8.f) {
          m_new = mxs;
          scale = ex2_approx(m_use - m_new);
        }
        const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
        // p = 2^(s c2 - m): scale-and-shift and the row sum run on paired fp32 instructions
        const uint64_t c2x2 = f2_pack(cs, cs), negm2 = f2_pack(neg_m, neg_m);
        uint64_t rs0 = 0, rs1 = 0;  // two pairs of partial sums (0.0f bit pattern is 0)
        uint32_t pk[BN / 2];
#pragma unroll
        for (int c = 0; c < BN / 2; c += 2) {
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), c2x2, negm2), x0, x1);
          f2_unpack(f2_fma(f2_pack(s[2 * c + 2], s[2 * c + 3]), c2x2, negm2), x2, x3);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
          rs0 = f2_add(rs0, f2_pack(p0, p1));
          rs1 = f2_add(rs1, f2_pack(p2, p3));
          pk[c] = pack2<F16>(p0, p1);
          pk[c + 1] = pack2<F16>(p2, p3);
        }
        float a0, a1;
        f2_unpack(f2_add(rs0, rs1), a0, a1);
        l = l * scale + (a0 + a1);
        m_use = m_new;
        // O_t is rescaled only when the reference maximum moved; PV_t(j-1) must have finished
        // first. PV_t number i (running count over the CTA's items) completes phase i / 2 of
        // barrier [t][i mod 2], and the parity names the phase exactly: every schedule has
        // completed PV(k - 3), hence PV_t(j - 3), once S_t(j) is in TMEM, and PV_t(j + 1)
        // cannot run before this thread publishes P_t(j).
        if (j > 0 && __any_sync(0xffffffffu, scale != 1.f)) {
          const int gp = pv_g + j - 1;
          if (!mbar_wait_warp(smem_u32(&bars.o_done[t][gp & 1]), (gp >> 1) & 1, abort, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t sc2 = f2_pack(scale, scale);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            ATTN_TMEM_LD_X32(tOt + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float y0, y1;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), sc2),
                        y0, y1);
              o[e] = __float_as_uint(y0);
              o[e + 1] = __float_as_uint(y1);
            }
            ATTN_TMEM_ST_X32(tOt + c * 32, o);
          }
        }
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) ATTN_TMEM_ST_X16(tSt + c * 16, (&pk[c * 16]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.p_full[bsel]));
      }
      // A tile without key tiles in this block waits here until the other tile's warps have
      // seen all of the block's score tiles: its next wait, on the next block's score tile,
      // is then at most one phase ahead of its buffer's barrier (a parity wait is exact only
      // then; skipping the block alone could leave it further behind). Both tiles' warps
      // arrive and wait (a bounded wait: a warpgroup that gave up leaves the other one free).
      if (one_empty) ok = tile_meet() && ok;
      if (n > 0 && ok) {
        // PV_t(n-1) last. Its wait needs PV_t(n-3) complete, which S_t(n-1) in TMEM does not
        // imply where the two issuing warps run one query tile's consecutive score tiles (it
        // implies PV(k - 3) only); PV_t(n-2) first, whose wait needs PV_t(n-4) = PV(<= k - 3).
        // No PV_t follows either (the next block's first PV_t needs this thread's next P), so
        // neither barrier can run a phase ahead.
        if (n > 1) {
          const int gp = pv_g + n - 2;
          ok = mbar_wait_warp(smem_u32(&bars.o_done[t][gp & 1]), (gp >> 1) & 1, abort, p.timeout_ns);
        }
        if (ok) {
          const int gp = pv_g + n - 1;
          ok = mbar_wait_warp(smem_u32(&bars.o_done[t][gp & 1]), (gp >> 1) & 1, abort, p.timeout_ns);
        }
        tc_fence_after();
      }
      if (ok) {
        // the item's addresses, decoded again rather than held through the key loop
        FwdItem w;
        decode_item(item, w);
        const bool valid = row < w.sv.len_q;
        const int64_t grow = w.sv.row0_q + row;
        uint16_t* orow = p.o + w.sv.batch * p.o_sb + w.h * p.o_sh + grow * p.o_ss;
        if (SPLIT && w.partial) {
          // A part of a block split over CTAs: this part's unnormalised O and row statistics
          // go to its slot (one per (block, CTA) pair); the CTA that completes the block's
          // last part merges all parts, in part order, so that the result does not depend on
          // which CTA finishes last.
          constexpr int RB = C::NQ * BM;  // rows of a block
          const int rr = t * BM + r;
          const int64_t U = p.n_units;
          const int G = (int)gridDim.x;
          // CTA whose range holds unit u: the largest c with floor(c U / G) <= u
          auto cta_of = [&](int64_t u) { return (int)(((u + 1) * G - 1) / U); };
          const int c_first = cta_of((int64_t)item * p.nk);
          const int c_last = cta_of((int64_t)(item + 1) * p.nk - 1);
          float* own = p.part + (size_t)(item + blockIdx.x) * C::SLOT_FLOATS;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            if (n > 0) {
              ATTN_TMEM_LD_X32(tOt + c * 32, o);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(own + ((c * 32 + e) / 4 * RB + rr) * 4) =
                  make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                              __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
          }
          own[D * RB + rr] = m_use;
          own[(D + 1) * RB + rr] = l;
          __threadfence();
          ok = tile_meet();  // every row of this part is written
          if (ok && threadIdx.x == 0) {
            const int done = atomicAdd(p.part_cnt + item, 1);
            bars.merge_last = done == c_last - c_first;
            if (done == c_last - c_first) p.part_cnt[item] = 0;  // zero again for the next call
          }
          ok = ok && tile_meet();
          if (ok && bars.merge_last) {
            __threadfence();
            // The merge reads the other parts' slots from L2. Each group of loads below is
            // issued before any of its values is used, so a row waits about one L2 round trip
            // per group rather than one per load: the statistics of eight parts at a time,
            // then per 32-column chunk two parts' values (and maxima) at a time. The parts
            // are summed in part order whichever CTA merges.
            const int me = (int)blockIdx.x;
            auto slot = [&](int c2) { return p.part + (size_t)(item + c2) * C::SLOT_FLOATS; };
            auto weight = [&](float mp, float mx) {  // a part's weight, 2^(m - mx)
              return mp == -INFINITY ? 0.f : ex2_approx(mp - mx);
            };
            float m8[8], l8[8];  // the statistics of the first eight parts
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int c2 = c_first + u;
              const bool in = c2 <= c_last, mine = c2 == me;
              m8[u] = !in ? -INFINITY : mine ? m_use : __ldcg(slot(c2) + D * RB + rr);
              l8[u] = !in ? 0.f : mine ? l : __ldcg(slot(c2) + (D + 1) * RB + rr);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int u = 0; u < 8; ++u) mx = fmaxf(mx, m8[u]);
            for (int g0 = c_first + 8; g0 <= c_last; g0 += 8) {
              float mv[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int c2 = g0 + u;
                mv[u] = c2 > c_last ? -INFINITY : c2 == me ? m_use : __ldcg(slot(c2) + D * RB + rr);
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) mx = fmaxf(mx, mv[u]);
            }
            float lsum = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) lsum += weight(m8[u], mx) * l8[u];
            for (int g0 = c_first + 8; g0 <= c_last; g0 += 8) {
              float mv[8], lv[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int c2 = g0 + u;
                const bool in = c2 <= c_last, mine = c2 == me;
                mv[u] = !in ? -INFINITY : mine ? m_use : __ldcg(slot(c2) + D * RB + rr);
                lv[u] = !in ? 0.f : mine ? l : __ldcg(slot(c2) + (D + 1) * RB + rr);
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) lsum += weight(mv[u], mx) * lv[u];
            }
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              float acc[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) acc[e] = 0.f;
              for (int g0 = c_first; g0 <= c_last; g0 += 2) {
                float4 x[2][8];
                float mp[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int c2 = g0 + u;
                  if (c2 == me) {  // this CTA's part, still in tensor memory
                    mp[u] = m_use;
                    uint32_t o[32];
                    if (n > 0) {
                      ATTN_TMEM_LD_X32(tOt + c * 32, o);
                    } else {
#pragma unroll
                      for (int e = 0; e < 32; ++e) o[e] = 0u;
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                      x[u][e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                            __uint_as_float(o[4 * e + 2]),
                                            __uint_as_float(o[4 * e + 3]));
                  } else if (c2 <= c_last) {
                    const float* sl = slot(c2);
                    mp[u] = __ldcg(sl + D * RB + rr);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                      x[u][e] = __ldcg(reinterpret_cast<const float4*>(sl + ((c * 8 + e) * RB + rr) * 4));
                  } else {
                    mp[u] = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[u][e] = make_float4(0.f, 0.f, 0.f, 0.f);
                  }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const float sc = weight(mp[u], mx);
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    acc[4 * e] += sc * x[u][e].x;
                    acc[4 * e + 1] += sc * x[u][e].y;
                    acc[4 * e + 2] += sc * x[u][e].z;
                    acc[4 * e + 3] += sc * x[u][e].w;
                  }
                }
              }
              if (valid && c * 32 < p.d_out) {
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                  uint4 v;
                  v.x = pack2<F16>(acc[e + 0] * inv, acc[e + 1] * inv);
                  v.y = pack2<F16>(acc[e + 2] * inv, acc[e + 3] * inv);
                  v.z = pack2<F16>(acc[e + 4] * inv, acc[e + 5] * inv);
                  v.w = pack2<F16>(acc[e + 6] * inv, acc[e + 7] * inv);
                  *reinterpret_cast<uint4*>(orow + c * 32 + e) = v;
                }
              }
            }
            if (valid)
              p.lse[w.sv.batch * p.l_sb + w.h * p.l_sh + grow * p.l_ss] =
                  lsum > 0.f ? (mx + __log2f(lsum)) * 0.69314718055994531f : -INFINITY;
          }
        } else {
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        // A query tile wholly inside its sequence leaves through shared memory: each warp
        // writes its 32 rows as 64-column slabs (128-byte swizzle) and one lane copies each
        // slab out with a TMA store, whole 128-byte rows at a time (row-per-thread global
        // stores write 16 bytes into each of 32 rows per instruction). A tile reaching past
        // the sequence's end is stored row by row: a copy would also write the rows past the
        // end (the next sequence's, in a compact batch). The condition is the same for the
        // whole warpgroup.
        const bool staged = C::O_TMA && n > 0 && q_lo + BM <= w.sv.len_q;
        if (staged) {
          uint8_t* region = smem + C::OFF_OST + (t * 4 + (warp & 3)) * C::OST_W_BYTES;
          const int row_w = w.sv.row0_q + q_lo + (warp & 3) * 32;  // first row of this warp
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            const int sub = h % C::OST_SLABS;
            uint32_t o[64];
            ATTN_TMEM_LD2_X32(tOt + 64 * h, tOt + 64 * h + 32, o, (o + 32));
            if (sub == 0) {  // this warp's earlier copies out of the region have read it
              if (lane == 0) bulk_wait_group_read0();
              __syncwarp();
            }
            uint8_t* slab = region + sub * 4096 + lane * 128;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              uint4 v;
              v.x = pack2<F16>(__uint_as_float(o[8 * e + 0]) * inv_l, __uint_as_float(o[8 * e + 1]) * inv_l);
              v.y = pack2<F16>(__uint_as_float(o[8 * e + 2]) * inv_l, __uint_as_float(o[8 * e + 3]) * inv_l);
              v.z = pack2<F16>(__uint_as_float(o[8 * e + 4]) * inv_l, __uint_as_float(o[8 * e + 5]) * inv_l);
              v.w = pack2<F16>(__uint_as_float(o[8 * e + 6]) * inv_l, __uint_as_float(o[8 * e + 7]) * inv_l);
              *reinterpret_cast<uint4*>(slab + ((e ^ (lane & 7)) << 4)) = v;
            }
            if (sub == C::OST_SLABS - 1 || h == D / 64 - 1) {
              fence_proxy_async_smem();  // the slabs, written by this warp, to the copy engine
              __syncwarp();
              if (lane == 0) {
#pragma unroll
                for (int s2 = 0; s2 <= sub; ++s2)
                  tma_store_4d(&p.tm_o, smem_u32(region + s2 * 4096), (h - sub + s2) * 64, row_w,
                               w.h, w.sv.batch);
                bulk_commit_group();
              }
            }
          }
        } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          if (n > 0) {
            ATTN_TMEM_LD_X32(tOt + c * 32, o);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          if (valid && c * 32 < p.d_out) {  // columns past the head size are zero padding
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 v;
              v.x = pack2<F16>(__uint_as_float(o[e + 0]) * inv_l, __uint_as_float(o[e + 1]) * inv_l);
              v.y = pack2<F16>(__uint_as_float(o[e + 2]) * inv_l, __uint_as_float(o[e + 3]) * inv_l);
              v.z = pack2<F16>(__uint_as_float(o[e + 4]) * inv_l, __uint_as_float(o[e + 5]) * inv_l);
              v.w = pack2<F16>(__uint_as_float(o[e + 6]) * inv_l, __uint_as_float(o[e + 7]) * inv_l);
              *reinterpret_cast<uint4*>(orow + c * 32 + e) = v;
            }
          }
        }
        }
        if (valid)
          p.lse[w.sv.batch * p.l_sb + w.h * p.l_sh + grow * p.l_ss] =
              (l > 0.f) ? (m_use + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
      }
      s_g += order.total;
      pv_g += n;
    }
    // the staged epilogue's copies have completed (they read shared memory)
    if (C::O_TMA && lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && bars.abort && p.status != nullptr) atomicCAS(p.status, 0, kStatusTimeout);
}

template <int D, bool F16, bool BIAS, bool SPLIT = false>
static cudaError_t launch_fwd_impl(const FwdParams& p, dim3 grid, cudaStream_t stream) {
  using C = FwdCfg<D, BIAS>;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, F16, BIAS, SPLIT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  attn_fwd_kernel<D, F16, BIAS, SPLIT><<<grid, C::NTHREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

template <bool BIAS>
static cudaError_t launch_fwd_dispatch(const FwdParams& p, int D, bool f16, dim3 grid,
                                       cudaStream_t stream) {
  if (D == 256)
    return f16 ? launch_fwd_impl<256, true, BIAS>(p, grid, stream)
               : launch_fwd_impl<256, false, BIAS>(p, grid, stream);
  if (D == 128)
    return f16 ? launch_fwd_impl<128, true, BIAS>(p, grid, stream)
               : launch_fwd_impl<128, false, BIAS>(p, grid, stream);
  return f16 ? launch_fwd_impl<64, true, BIAS>(p, grid, stream)
             : launch_fwd_impl<64, false, BIAS>(p, grid, stream);
}

cudaError_t launch_attn_fwd(const FwdParams& p, int D, bool f16, bool bias, dim3 grid,
                            cudaStream_t stream) {
  if (bias) {  // the bias kernels exist for the 64- and 128-wide configurations
    if (D == 128)
      return f16 ? launch_fwd_impl<128, true, true>(p, grid, stream)
                 : launch_fwd_impl<128, false, true>(p, grid, stream);
    if (D != 64) return cudaErrorInvalidValue;
    return f16 ? launch_fwd_impl<64, true, true>(p, grid, stream)
               : launch_fwd_impl<64, false, true>(p, grid, stream);
  }
  if (p.split) {  // split grids (no bias): their own instantiations
    if (D == 256)
      return f16 ? launch_fwd_impl<256, true, false, true>(p, grid, stream)
                 : launch_fwd_impl<256, false, false, true>(p, grid, stream);
    if (D == 128)
      return f16 ? launch_fwd_impl<128, true, false, true>(p, grid, stream)
                 : launch_fwd_impl<128, false, false, true>(p, grid, stream);
    return f16 ? launch_fwd_impl<64, true, false, true>(p, grid, stream)
               : launch_fwd_impl<64, false, false, true>(p, grid, stream);
  }
  return launch_fwd_dispatch<false>(p, D, f16, grid, stream);
}

// Query rows per CTA: two 128-row tiles; one at kernel width 256, and at width 128 with a
// bias. The 4-D Q tensor map uses a 128-row box.
int fwd_block_m(int width, bool bias) {
  return (width == 256 || (width == 128 && bias)) ? 128 : 256;
}
int fwd_box_rows() { return 128; }

}  // namespace attn_sm103
