// Kernel parameter blocks and the per-tile sequence decode shared by the forward and
// backward kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103_ptx.cuh"

namespace attn_sm103 {

// Sequence addressing modes.
enum : int { kDense = 0, kPadded = 1, kCompact = 2 };

// Device status codes (same values as attn_status in include/attn.h).
enum : int { kStatusBadSeqlens = 8, kStatusTimeout = 9 };

// A bounded wait gives up after this long (a correct pipeline waits microseconds).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

struct SeqAddr {
  const int* cu_q;  // int32 prefix sums (padded: [B+1], compact: [num_seqs+1]); null = dense
  const int* cu_k;
  int mode;         // kDense / kPadded / kCompact
  int Sq, Sk;       // token extents of the tensors (dense/padded: S; compact: T)
  int max_q, max_k; // grid bounds on per-sequence lengths
};

// Per-(batch or sequence) view: valid lengths, first row in the token axis, batch index of
// the rank-4 tensors. Follows the AOTriton padded-varlen prologue: padded sequences start
// at row 0 of their own batch; compact sequences start at cu[s] of the single batch.
struct SeqView {
  int len_q, len_k, row0_q, row0_k, batch;
};

// Returns false (and reports) when the cu_seqlens of unit z are inconsistent with the
// tensors or the grid; the caller then skips the unit without touching memory.
__device__ __forceinline__ bool decode_seq(const SeqAddr& a, int z, int* status, SeqView& v) {
  if (a.mode == kDense) {
    v.len_q = a.Sq; v.len_k = a.Sk; v.row0_q = 0; v.row0_k = 0; v.batch = z;
    return true;
  }
  const int q0 = __ldg(a.cu_q + z), q1 = __ldg(a.cu_q + z + 1);
  const int k0 = __ldg(a.cu_k + z), k1 = __ldg(a.cu_k + z + 1);
  bool ok = q0 >= 0 && q1 >= q0 && k0 >= 0 && k1 >= k0;
  v.len_q = q1 - q0;
  v.len_k = k1 - k0;
  if (a.mode == kPadded) {
    ok = ok && v.len_q <= a.Sq && v.len_k <= a.Sk;
    v.row0_q = 0; v.row0_k = 0; v.batch = z;
  } else {
    ok = ok && q1 <= a.Sq && k1 <= a.Sk && v.len_q <= a.max_q && v.len_k <= a.max_k;
    v.row0_q = q0; v.row0_k = k0; v.batch = 0;
  }
  if (!ok && status != nullptr) atomicCAS(status, 0, kStatusBadSeqlens);
  return ok;
}

// CTA order of a launch over `tiles` tiles of each of `uh` (unit, head) pairs, 1-D grid in
// launch order: groups of `group` pairs run one after another, and inside a group the tiles go
// by rank (rank 0, the heaviest of a causal grid, first) across the group's pairs. A group
// holds as many pairs as the operands their blocks share keep in L2 (the measured limits of
// attn_tune_table.h); group >= uh is longest-first over the whole grid, group == 1 keeps each
// pair's tiles together. Returns the pair index and the tile rank of block `linear`.
struct GridPos {
  int zh, rank;
};
__device__ __forceinline__ GridPos grid_pos(int linear, int tiles, int uh, int group) {
  const int per = group * tiles;  // blocks of a full group
  const int g = linear / per;
  const int r = linear - g * per;
  const int gs = min(group, uh - g * group);  // pairs in this group (the last may be short)
  return GridPos{g * group + r % gs, r / gs};
}

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;   // 4-D (D, S, H, B) 16-bit, box (64, 128, 1, 1), SW128
  CUtensorMap tm_o;               // O, box (64, 32, 1, 1), SW128: the staged epilogue's stores
  CUtensorMap tm_b;               // bias kernels only: 4-D (Sk, Sq, Hb, Bb), box (64, 128, 1, 1)
  int bias_b_bcast, bias_h_bcast; // bias broadcast over batch / head (size-1 dimension)
  uint16_t* o;                    // bf16 or fp16 elements (the kernel's element type)
  int64_t o_sb, o_sh, o_ss;       // element strides of o (D stride is 1)
  float* lse;
  int64_t l_sb, l_sh, l_ss;
  SeqAddr seq;
  int causal;
  float scale_log2;               // sm_scale * log2(e)
  int* status;                    // device status word, may be null
  uint64_t timeout_ns;            // bound on every pipeline wait
  int withhold_tile;              // test hook: key tile the producer never loads (-1: none)
  int tiles, group;               // query blocks per (unit, head) pair; CTA-order group size
  int uh;                         // (unit, head) pairs: work items = uh * tiles
  int split;                      // 1: non-causal dense grid with fewer blocks than SMs; the
                                  // (block, key tile) units are cut into gridDim.x equal
                                  // ranges, one per CTA, and blocks split over several CTAs
                                  // merge their partial results
  int nk;                         // split: key tiles per block
  int64_t n_units;                // split: blocks x nk
  float* part;                    // split: partial-result slots (one per (block, CTA) pair)
  int* part_cnt;                  // split: parts of each block done (returns to 0)
  int clc;                        // 1: one CTA per item, CTAs steal the items of CTAs not yet
                                  // launched (cluster launch control); 0: CTA c takes items
                                  // c, c + gridDim.x, ...
  int H;                          // heads
  int d_out;                      // head size of the tensors (<= the kernel's D; the TMA
                                  // loads fill the columns past it with zeros)
};

struct BwdPreParams {
  const uint16_t* o;              // 16-bit elements
  const uint16_t* dout;
  int64_t o_sb, o_sh, o_ss, do_sb, do_sh, do_ss;
  float* delta;                   // [B*H or H][rows] fp32, row index = token row
  float* dq_acc;                  // [B*H or H][rows][D] fp32, zeroed here; may be null
  int units, H, rows, D;          // units = B (dense/padded) or num_seqs (compact);
                                  // rows = Sq (dense/padded) or Tq (compact)
  int f16;                        // element type: 0 bf16, 1 fp16
  SeqAddr seq;
  int* status;
};

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // 4-D maps; Q/dO box rows = BM, K/V box rows = BN
  CUtensorMap tm_dq;                    // 2-D fp32 map over the dQ accumulator [rows][D]
                                        // (d_head 64), box (32, 128), 128-byte swizzle
  CUtensorMap tm_bias;                  // bias kernels: 4-D (Sk, Sq, Hb, Bb) over the bias,
                                        // box (64, query rows a step), 128-byte swizzle
  CUtensorMap tm_dk, tm_dv;             // dK, dV: box (a warpgroup's columns, 32 keys), no
                                        // swizzle (the staged epilogue's stores)
  const float* lse;
  int64_t l_sb, l_sh, l_ss;
  const float* delta;             // [z-major][rows] as written by the preprocess kernel
  float* dq_acc;
  uint16_t* dk;
  int64_t dk_sb, dk_sh, dk_ss;
  uint16_t* dv;
  int64_t dv_sb, dv_sh, dv_ss;
  int H, rows_q;                  // rows_q: per-(batch, head) row count of delta / dq_acc
  SeqAddr seq;
  int causal;
  int d_out;                      // head size of the tensors (<= the kernel's D)
  const uint16_t* bias;           // BIAS kernels: bias element (b, h, q, key) at
  int64_t b_sb, b_sh, b_ss;       //   b*b_sb + h*b_sh + q*b_ss + key (0 strides broadcast)
  uint16_t* dbias;                // BIAS kernels, may be null: dS written at the same layout
  int64_t db_sb, db_sh, db_ss;
  float* dbias_acc;               // BIAS kernels, may be null: dS added (fp32) at element
  int64_t dba_sb, dba_sh, dba_ss; //   b*dba_sb + h*dba_sh + q*dba_ss + key (0 strides sum)
  uint64_t timeout_ns;            // bound on every pipeline wait
  int withhold_step;              // test hook: step whose Q / dO the producer never loads (-1)
  int with_dq;                    // 0: no dQ products (the deterministic dQ kernel makes dQ)
  int tiles, group;               // key-tile CTAs per (unit, head) pair; CTA-order group size
  float scale_log2;               // sm_scale * log2(e)
  float sm_scale;
  int* status;
};

struct BwdPostParams {
  const float* dq_acc;
  uint16_t* dq;
  int64_t dq_sb, dq_sh, dq_ss;
  int units, H, rows, D;          // as in BwdPreParams
  int f16;                        // element type: 0 bf16, 1 fp16
  SeqAddr seq;
  float sm_scale;
};

// Rounds the fp32 gradient of a shared bias to the element type.
struct DbiasPostParams {
  const float* acc;               // [rows][Sk] fp32, rows = Bb * Hb * Sq
  uint16_t* dbias;                // (Bb, Hb, Sq, Sk), element strides below (key stride 1)
  int64_t db_sb, db_sh, db_ss;
  int64_t rows;
  int Hb, Sq, Sk;
  int f16;
};

// Deterministic dQ kernel: one CTA per 128 query rows, walking the key tiles in order.
struct BwdDqParams {
  CUtensorMap tm_q, tm_do;        // 4-D 16-bit maps, box (64, 128, 1, 1)
  CUtensorMap tm_k, tm_v;         // box (64, 128, 1, 1)
  const float* lse;
  int64_t l_sb, l_sh, l_ss;
  const float* delta;             // [B*H or H][rows_q] fp32
  uint16_t* dq;
  int64_t dq_sb, dq_sh, dq_ss;
  int H, rows_q;
  SeqAddr seq;
  int causal;
  float scale_log2;               // sm_scale * log2(e)
  float sm_scale;
  int* status;
  int tiles, group;               // query blocks per (unit, head) pair; CTA-order group size
  int d_out;                      // head size of the tensors (<= the kernel's D)
};

}  // namespace attn_sm103
