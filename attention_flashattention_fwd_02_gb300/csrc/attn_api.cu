// C ABI of the attention library (declared in include/attn.h): argument validation,
// workspace layout, TMA tensor-map encoding and kernel launches. Host code only.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/attn.h"
#include "attn_launch.h"
#include "attn_tune_table.h"

using namespace attn_sm103;

namespace {

constexpr int64_t kMaxI32 = 2147483647;

// ----------------------------------------------------------------------------- driver entry
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// The current device must be sm_103 (GB300); cached per device ordinal.
attn_status check_device() {
  static int cache[64] = {0};  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev] == 1 ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) cache[dev] = ok ? 1 : 2;
  return ok ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
}

// Streaming multiprocessors of the current device (cached per device ordinal; 0 on error).
int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

// ----------------------------------------------------------------------------- validation
attn_status check_tensor4(const attn_tensor4* t) {
  if (t == nullptr || t->data == nullptr) return ATTN_ERR_NULL;
  if (t->dtype != ATTN_DTYPE_BF16 && t->dtype != ATTN_DTYPE_F16) return ATTN_ERR_UNSUPPORTED;
  for (int i = 0; i < 4; ++i)
    if (t->size[i] < 0 || t->size[i] > kMaxI32) return ATTN_ERR_SHAPE;
  if (t->stride[3] != 1) return ATTN_ERR_STRIDE;
  for (int i = 0; i < 3; ++i)
    if (t->size[i] > 1 && (t->stride[i] <= 0 || t->stride[i] % 8 != 0)) return ATTN_ERR_STRIDE;
  if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0) return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

attn_status check_tensor3(const attn_tensor3* t) {
  if (t == nullptr || t->data == nullptr) return ATTN_ERR_NULL;
  for (int i = 0; i < 3; ++i) {
    if (t->size[i] < 0 || t->size[i] > kMaxI32) return ATTN_ERR_SHAPE;
    if (t->size[i] > 1 && t->stride[i] <= 0) return ATTN_ERR_STRIDE;
  }
  if (reinterpret_cast<uintptr_t>(t->data) % 4 != 0) return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

bool same_dtype(const attn_tensor4* a, const attn_tensor4* b) { return a->dtype == b->dtype; }

bool same_shape(const attn_tensor4* a, const attn_tensor4* b) {
  for (int i = 0; i < 4; ++i)
    if (a->size[i] != b->size[i]) return false;
  return true;
}

// The problem every entry point reduces to.
struct Problem {
  int mode;          // kDense / kPadded / kCompact
  int B, H, Sq, Sk, D;
  bool f16;          // element type of every rank-4 tensor
  int units;         // grid z: B, or num_seqs for compact
  int max_q, max_k;  // per-unit length bounds (grid extents)
  const int* cu_q;
  const int* cu_k;
};

// Shapes of q (B,H,Sq,D) and k/v (B,H,Sk,D); mode from cu_seqlens / num_seqs.
attn_status make_problem(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                         const int32_t* cu_q, const int32_t* cu_k, int compact, int32_t num_seqs,
                         int32_t max_seqlen_q, int32_t max_seqlen_k, Problem* pr) {
  attn_status s;
  if ((s = check_tensor4(q)) != ATTN_OK) return s;
  if ((s = check_tensor4(k)) != ATTN_OK) return s;
  if ((s = check_tensor4(v)) != ATTN_OK) return s;
  if (!same_shape(k, v)) return ATTN_ERR_SHAPE;
  if (!same_dtype(q, k) || !same_dtype(q, v)) return ATTN_ERR_DTYPE;
  if (q->size[0] != k->size[0] || q->size[1] != k->size[1] || q->size[3] != k->size[3])
    return ATTN_ERR_SHAPE;
  const int64_t D = q->size[3];
  // 256: forward only (the backward stages reject it)
  if (D != 32 && D != 64 && D != 96 && D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;
  if (q->size[1] > 65535) return ATTN_ERR_UNSUPPORTED;  // grid y
  pr->B = (int)q->size[0];
  pr->H = (int)q->size[1];
  pr->Sq = (int)q->size[2];
  pr->Sk = (int)k->size[2];
  pr->D = (int)D;
  pr->f16 = q->dtype == ATTN_DTYPE_F16;
  if (compact) {
    if (q->size[0] != 1) return ATTN_ERR_SHAPE;  // compact varlen takes batch exactly 1
    if (cu_q == nullptr || cu_k == nullptr) return ATTN_ERR_NULL;
    if (num_seqs < 0 || num_seqs > 65535) return ATTN_ERR_SHAPE;
    pr->mode = kCompact;
    pr->units = num_seqs;
    pr->max_q = max_seqlen_q > 0 ? (max_seqlen_q < pr->Sq ? max_seqlen_q : pr->Sq) : pr->Sq;
    pr->max_k = max_seqlen_k > 0 ? (max_seqlen_k < pr->Sk ? max_seqlen_k : pr->Sk) : pr->Sk;
  } else {
    if ((cu_q == nullptr) != (cu_k == nullptr)) return ATTN_ERR_NULL;
    if (pr->B > 65535) return ATTN_ERR_UNSUPPORTED;  // grid z
    pr->mode = cu_q ? kPadded : kDense;
    pr->units = pr->B;
    pr->max_q = pr->Sq;
    pr->max_k = pr->Sk;
  }
  pr->cu_q = cu_q;
  pr->cu_k = cu_k;
  return ATTN_OK;
}

attn_status check_lse(const attn_tensor3* lse, const Problem& pr) {
  attn_status s = check_tensor3(lse);
  if (s != ATTN_OK) return s;
  if (lse->size[0] != pr.B || lse->size[1] != pr.H || lse->size[2] != pr.Sq) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

// An additive bias (Bb, Hb, Sq_b, Sk_b) in q's element type: Bb in {1, units} (units = B,
// or num_seqs for compact varlen), Hb in {1, H}; dense and padded forms take Sq_b = Sq,
// Sk_b = Sk; compact sequences index the block at offset 0 of their own slice, so Sq_b and
// Sk_b must hold the longest sequence (the max_seqlen bounds). d_head up to 128.
attn_status check_bias(const attn_tensor4* bias, const attn_tensor4* q, const attn_tensor4* k,
                       const Problem& pr) {
  if (pr.D > 128) return ATTN_ERR_UNSUPPORTED;
  attn_status s = check_tensor4(bias);
  if (s != ATTN_OK) return s;
  if (!same_dtype(q, bias)) return ATTN_ERR_DTYPE;
  if ((bias->size[0] != 1 && bias->size[0] != pr.units) ||
      (bias->size[1] != 1 && bias->size[1] != pr.H))
    return ATTN_ERR_SHAPE;
  if (pr.mode == kCompact) {
    if (bias->size[2] < pr.max_q || bias->size[3] < pr.max_k) return ATTN_ERR_SHAPE;
  } else if (bias->size[2] != q->size[2] || bias->size[3] != k->size[2]) {
    return ATTN_ERR_SHAPE;
  }
  return ATTN_OK;
}

// A bias with a size-1 batch or head dimension gets its gradient summed in fp32 in the
// workspace, after the status word, Delta and the dQ accumulator.
bool bias_shared(const attn_tensor4* bias) { return bias->size[0] == 1 || bias->size[1] == 1; }

size_t dbias_acc_bytes(const attn_tensor4* bias) {
  return (size_t)bias->size[0] * (size_t)bias->size[1] * (size_t)bias->size[2] *
         (size_t)bias->size[3] * 4;
}

SeqAddr seq_addr(const Problem& pr) {
  SeqAddr a;
  a.cu_q = pr.cu_q;
  a.cu_k = pr.cu_k;
  a.mode = pr.mode;
  a.Sq = pr.Sq;
  a.Sk = pr.Sk;
  a.max_q = pr.max_q;
  a.max_k = pr.max_k;
  return a;
}

// 4-D tensor map over a BHSD view: dims (D, S, H, B) innermost first, box (box_cols, rows, 1,
// 1), swizzle 128, 64 or 0 bytes (a swizzled box's rows are that long). Strides of size-1
// dimensions are never used; they are replaced by a valid dummy so that any view of such a
// dimension is accepted.
attn_status make_map(CUtensorMap* m, const attn_tensor4* t, int box_rows, int box_cols = 64,
                     int swizzle = 128) {
  auto enc = encode_fn();
  if (enc == nullptr) return ATTN_ERR_CUDA;
  const int64_t B = t->size[0], H = t->size[1], S = t->size[2], D = t->size[3];
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)(S > 0 ? S : 1), (cuuint64_t)(H > 0 ? H : 1),
                        (cuuint64_t)(B > 0 ? B : 1)};
  const int64_t ss = (S > 1) ? t->stride[2] : D;
  const int64_t sh = (H > 1) ? t->stride[1] : ss * (S > 0 ? S : 1);
  const int64_t sb = (B > 1) ? t->stride[0] : sh * (H > 0 ? H : 1);
  cuuint64_t strides[3] = {(cuuint64_t)ss * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
  for (int i = 0; i < 3; ++i)
    if (strides[i] % 16 != 0 || strides[i] >= (1ull << 40)) return ATTN_ERR_STRIDE;
  cuuint32_t box[4] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty =
      t->dtype == ATTN_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(m, ty, 4, t->data, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                   : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                   : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 2-D fp32 tensor map over the dQ accumulator viewed as [rows][D]: box (32, 32), 128-byte
// swizzle (32 floats = 128 bytes per box row). Each warp of the backward kernel adds one such
// 32 x 32 block per step.
attn_status make_map_acc(CUtensorMap* m, float* acc, int64_t rows, int64_t D) {
  auto enc = encode_fn();
  if (enc == nullptr) return ATTN_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)D * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, acc, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// Causal tiles differ in work. Dispatched heaviest first across all (unit, head) pairs, they
// leave no tail (a per-head heaviest-first order starts the last head's heaviest tile near
// the end); but the CTAs of one head then spread over the whole launch, and the operands they
// share must stay in L2 (129 MB) between them. So the whole grid runs longest-first when those
// operands fit the kernel's measured limit in attn_tune_table.h, else each pair's blocks run
// together (grid_group). Groups in between were measured too and lost to the per-head order
// in the backward (the per-head operands' L2 reuse outweighs the tail).
// Head sizes 32 and 96 run on the kernels built for 64 and 128: the TMA loads (box 64
// columns wide) fill the columns past the head size with zeros, which add nothing to any
// product, and only the real columns are stored.
int kernel_width(int D) { return D <= 64 ? 64 : D <= 128 ? 128 : 256; }

// Tuning hook: ATTN_GRID_ORDER = "<kernel>:tile", "<kernel>:seq" or "<kernel>:g<N>"
// (comma-separated entries) forces the order of that kernel's causal grids: longest-first
// over the whole grid, each head's blocks together, or groups of N (unit, head) pairs; the
// sweep that writes the table times these orders this way. Returns the forced group size, or
// -1 (uh: the number of (unit, head) pairs).
int grid_order_override(const char* kernel, int uh) {
  const char* v = getenv("ATTN_GRID_ORDER");
  if (v == nullptr) return -1;
  const size_t n = strlen(kernel);
  for (const char* e = v; *e;) {
    if (strncmp(e, kernel, n) == 0 && e[n] == ':') {
      if (strncmp(e + n + 1, "tile", 4) == 0) return uh;
      if (strncmp(e + n + 1, "seq", 3) == 0) return 1;
      if (e[n + 1] == 'g') {
        const int g = atoi(e + n + 2);
        if (g >= 1) return g;
      }
    }
    const char* c = strchr(e, ',');
    if (c == nullptr) break;
    e = c + 1;
  }
  return -1;
}

double tile_major_limit(const char* kernel, int width) {
  for (const GridOrderRule& r : kGridOrderRules)
    if (r.width == width && strcmp(r.kernel, kernel) == 0) return r.max_tile_major_bytes;
  return 0.0;
}

// Group size of the CTA order (grid_pos in attn_common.cuh) for `uh` (unit, head) pairs whose
// blocks share `shared_bytes` over all pairs. kernel: "fwd", "bwd_main", "bwd_main_nodq" or
// "bwd_dq"; width: 64, 128 or 256. Causal grids: all pairs (longest-first over the whole grid)
// when the shared operands fit the kernel's measured L2 limit, else one; non-causal grids,
// whose blocks are equally heavy, keep each pair's blocks together.
int grid_group(const char* kernel, int width, int causal, double shared_bytes, int uh) {
  if (!causal || uh <= 1) return 1;
  const int forced = grid_order_override(kernel, uh);
  if (forced >= 1) return forced < uh ? forced : uh;
  return shared_bytes <= tile_major_limit(kernel, width) ? uh : 1;
}

// The measured split rule for a forward of the given kernel width (no rule: no split).
bool fwd_split_by_table(int width, int64_t n_items, int64_t key_tiles, int sms) {
  for (const FwdSplitRule& r : kFwdSplitRules)
    if (r.width == width)
      return 2 * n_items <= sms && (double)n_items <= r.max_blocks_per_sm * sms &&
             key_tiles >= r.min_key_tiles;
  return false;
}

// Forward grid: one CTA per work item. With more items than SMs the running CTAs steal the
// items of CTAs not yet launched (cluster launch control), so each SM's CTA walks items in the
// grid's order until none are left, its pipeline running on across them. Tuning and test
// hooks: ATTN_FWD_PERSISTENT=0 turns the stealing off; ATTN_FWD_CTAS=<n> launches n CTAs
// (n >= 1), CTA c taking items c, c + n, ... Returns the grid size; *clc is the stealing flag.
int fwd_grid_size(int n_items, int* clc) {
  *clc = 0;
  const char* c = getenv("ATTN_FWD_CTAS");
  if (c != nullptr && atoi(c) >= 1) return atoi(c) < n_items ? atoi(c) : n_items;
  const char* v = getenv("ATTN_FWD_PERSISTENT");
  *clc = (v == nullptr || atoi(v) != 0) && n_items > sm_count();
  return n_items;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace header shared by the forward and backward calls: the status word at offset 0 and,
// at kSplitCntOff, the forward's split-block counters (each back at zero when its call ends;
// no backward kernel writes the header, so one workspace can serve both passes).
constexpr size_t kFwdMinWorkspace = 256;  // the forward's status word (and alignment room)
constexpr size_t kWsHeader = 2048;
constexpr size_t kSplitCntOff = 1024;
constexpr int kSplitMaxBlocks = 256;  // a split grid has fewer blocks than SMs

// Bytes of one partial-result slot of a split forward grid (FwdCfg::SLOT_FLOATS floats).
size_t fwd_split_slot_bytes(int width) {
  return (size_t)fwd_block_m(width, false) * (size_t)(width + 2) * 4;
}
// Workspace a split forward grid over n_items blocks needs (0: none can split): the header
// and one slot per (block, CTA) pair that can hold a part.
size_t fwd_split_ws_bytes(int64_t n_items, int width) {
  if (n_items <= 0 || n_items >= kSplitMaxBlocks) return 0;
  return kWsHeader + (size_t)(n_items + kSplitMaxBlocks) * fwd_split_slot_bytes(width);
}

struct BwdWorkspace {
  size_t delta_off, dq_off, total;
};

BwdWorkspace bwd_layout(int64_t B, int64_t H, int64_t rows, int64_t D) {
  BwdWorkspace w;
  const size_t n = (size_t)(B > 0 ? B : 0) * (size_t)(H > 0 ? H : 0) * (size_t)(rows > 0 ? rows : 0);
  w.delta_off = kWsHeader;
  w.dq_off = w.delta_off + align256(n * 4);
  w.total = w.dq_off + n * (size_t)D * 4;
  return w;
}

bool valid_scale(float s) { return isfinite(s) && s > 0.f; }

// Test hook for the failure-detection path: when the environment variable
// ATTN_TEST_WITHHOLD_KV_TILE holds a key-tile index, the forward producers load no key tile
// from that one on and every wait is bounded by 50 ms, so the kernel gives up, reports
// ATTN_ERR_DEVICE_TIMEOUT in the status word and returns (no trap, no fault).
int withheld_tile_for_test() {
  const char* v = getenv("ATTN_TEST_WITHHOLD_KV_TILE");
  if (v == nullptr || *v == 0) return -1;
  return atoi(v);
}

// Test hook of the backward key-tile kernel: step whose Q / dO tile is never loaded.
int withheld_step_for_test() {
  const char* v = getenv("ATTN_TEST_WITHHOLD_Q_STEP");
  if (v == nullptr || *v == 0) return -1;
  return atoi(v);
}

// ----------------------------------------------------------------------------- forward
attn_status fwd_common(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                       const int32_t* cu_q, const int32_t* cu_k, int compact, int32_t num_seqs,
                       int32_t max_q, int32_t max_k, float sm_scale, int causal,
                       const attn_tensor4* o, const attn_tensor3* lse, void* ws, size_t ws_bytes,
                       void* stream, const attn_tensor4* bias = nullptr) {
  Problem pr;
  attn_status s = make_problem(q, k, v, cu_q, cu_k, compact, num_seqs, max_q, max_k, &pr);
  if (s != ATTN_OK) return s;
  if (bias != nullptr && (s = check_bias(bias, q, k, pr)) != ATTN_OK) return s;
  if ((s = check_tensor4(o)) != ATTN_OK) return s;
  if (!same_shape(q, o)) return ATTN_ERR_SHAPE;
  if (!same_dtype(q, o)) return ATTN_ERR_DTYPE;
  if ((s = check_lse(lse, pr)) != ATTN_OK) return s;
  if (!valid_scale(sm_scale)) return ATTN_ERR_UNSUPPORTED;
  if (ws != nullptr && ws_bytes < kFwdMinWorkspace) return ATTN_ERR_WORKSPACE;
  if (ws != nullptr && reinterpret_cast<uintptr_t>(ws) % 16 != 0) return ATTN_ERR_ALIGN;
  if ((s = check_device()) != ATTN_OK) return s;
  if (pr.units == 0 || pr.max_q == 0 || pr.H == 0) return ATTN_OK;

  FwdParams p;
  memset(&p, 0, sizeof(p));
  const int BM = fwd_block_m(kernel_width(pr.D), bias != nullptr);
  if ((s = make_map(&p.tm_q, q, fwd_box_rows())) != ATTN_OK) return s;
  if ((s = make_map(&p.tm_k, k, 128)) != ATTN_OK) return s;
  if ((s = make_map(&p.tm_v, v, 128)) != ATTN_OK) return s;
  if ((s = make_map(&p.tm_o, o, 32)) != ATTN_OK) return s;
  if (bias != nullptr) {
    if ((s = make_map(&p.tm_b, bias, 128)) != ATTN_OK) return s;
    p.bias_b_bcast = bias->size[0] == 1 && pr.units > 1;
    p.bias_h_bcast = bias->size[1] == 1 && pr.H > 1;
  }
  p.o = reinterpret_cast<uint16_t*>(o->data);
  p.o_sb = o->stride[0];
  p.o_sh = o->stride[1];
  p.o_ss = o->stride[2];
  p.lse = reinterpret_cast<float*>(lse->data);
  p.l_sb = lse->stride[0];
  p.l_sh = lse->stride[1];
  p.l_ss = lse->stride[2];
  p.seq = seq_addr(pr);
  p.causal = causal ? 1 : 0;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.status = reinterpret_cast<int*>(ws);
  p.withhold_tile = withheld_tile_for_test();
  p.timeout_ns = p.withhold_tile >= 0 ? 50000000ull : kWaitTimeoutNs;
  const int n_blk = (pr.max_q + BM - 1) / BM;
  const int uh = pr.units * pr.H;
  p.tiles = n_blk;
  p.H = pr.H;
  p.group = grid_group("fwd", kernel_width(pr.D), p.causal,
                       (double)pr.units * pr.H * pr.max_k * pr.D * 4, uh);
  p.uh = uh;
  if ((int64_t)n_blk * uh > kMaxI32) return ATTN_ERR_UNSUPPORTED;  // 1-D grid
  const int n_items = n_blk * uh;
  dim3 grid((unsigned)fwd_grid_size(n_items, &p.clc));
  // Few blocks (non-causal, dense, no bias): cut the (block, key tile) units into equal
  // ranges, the same number for every block and at most one per SM, given the workspace for
  // the partial results. The measured table (kFwdSplitRules) says when: at most about half as
  // many blocks as SMs (every block then has two parts or more) and key ranges long enough
  // to outweigh the partial results and their merge. ATTN_FWD_SPLIT=0 turns it off, =1
  // splits any grid with fewer blocks than SMs (more than half as many: one range per SM).
  const int sms = sm_count();
  const int64_t nk = ((int64_t)pr.max_k + 127) / 128;
  const size_t split_need = fwd_split_ws_bytes(n_items, kernel_width(pr.D));
  const char* sv = getenv("ATTN_FWD_SPLIT");
  const bool split_on = sv == nullptr ? fwd_split_by_table(kernel_width(pr.D), n_items, nk, sms)
                                      : atoi(sv) != 0;
  if (!causal && bias == nullptr && pr.mode == kDense && sms > n_items && nk >= 2 &&
      split_need > 0 && ws != nullptr && ws_bytes >= split_need && split_on) {
    const int64_t units = (int64_t)n_items * nk;
    // a multiple of the block count: every block splits into the same number of parts and no
    // CTA runs two (measured on GB300: 32 blocks over 128 CTAs 34 us, over 152 CTAs 42 us)
    const int per_block = (int)(nk < sms / n_items ? nk : sms / n_items);
    int G = per_block >= 2 ? n_items * per_block : (units < sms ? (int)units : sms);
    // ATTN_FWD_CTAS=<n> sets the split grid's size too (a sweep hook; each CTA then runs
    // units / n of the work, n at most the slots the workspace holds)
    const char* cs = getenv("ATTN_FWD_CTAS");
    const bool forced = cs != nullptr && atoi(cs) >= 1;
    if (forced) {
      const int64_t n = atoi(cs) < units ? atoi(cs) : units;
      G = (int)(n < kSplitMaxBlocks ? n : kSplitMaxBlocks);
    }
    if (G > n_items || forced) {
      p.split = 1;
      p.nk = (int)nk;
      p.n_units = units;
      p.part_cnt = reinterpret_cast<int*>(static_cast<char*>(ws) + kSplitCntOff);
      p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
      p.clc = 0;
      grid = dim3((unsigned)G);
    }
  }
  p.d_out = pr.D;
  cudaError_t e = launch_attn_fwd(p, kernel_width(pr.D), pr.f16, bias != nullptr, grid,
                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ----------------------------------------------------------------------------- backward
struct BwdArgs {
  const attn_tensor4 *q, *k, *v, *o, *dout, *dq, *dk, *dv;
  const attn_tensor3* lse;
  const attn_tensor4* bias = nullptr;   // optional additive bias (attn_bwd_bias)
  const attn_tensor4* dbias = nullptr;  // optional gradient of the bias
};

// Stages: 1 preprocess, 2 key-tile kernel, 4 dQ epilogue, 8 deterministic dQ kernel. In
// deterministic mode the preprocess leaves the fp32 accumulator alone, the key-tile kernel
// skips its dQ products and the workspace needs only the status word and Delta.
attn_status bwd_stage(int stage_mask, const BwdArgs& a, const Problem& pr, float sm_scale,
                      int causal, void* ws, size_t ws_bytes, void* stream,
                      bool deterministic = false) {
  // d_head 256: the key-tile kernel splits d over two CTAs per key tile; the deterministic
  // dQ kernel has no such split (its dQ accumulator and S, dP would need 512 TMEM columns next
  // to Q, dO, K and V in shared memory)
  if (deterministic && pr.D > 128) return ATTN_ERR_UNSUPPORTED;
  const BwdWorkspace w = bwd_layout(pr.B, pr.H, pr.Sq, pr.D);
  // the fp32 sums of a shared bias's gradient follow the regular workspace
  const bool dbias_sum = a.bias != nullptr && a.dbias != nullptr && bias_shared(a.bias);
  const size_t acc_off = align256(w.total);
  const size_t need = dbias_sum ? acc_off + dbias_acc_bytes(a.bias)
                                : (deterministic ? w.dq_off : w.total);
  if (ws == nullptr || ws_bytes < need) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return ATTN_ERR_ALIGN;
  attn_status s = check_device();
  if (s != ATTN_OK) return s;
  if (pr.units == 0 || pr.H == 0) return ATTN_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  float* delta = reinterpret_cast<float*>(base + w.delta_off);
  float* dq_acc = reinterpret_cast<float*>(base + w.dq_off);
  int* status = reinterpret_cast<int*>(base);
  const SeqAddr sa = seq_addr(pr);

  if (stage_mask & 1) {
    BwdPreParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.o = reinterpret_cast<const uint16_t*>(a.o->data);
    pp.dout = reinterpret_cast<const uint16_t*>(a.dout->data);
    pp.f16 = pr.f16 ? 1 : 0;
    pp.o_sb = a.o->stride[0]; pp.o_sh = a.o->stride[1]; pp.o_ss = a.o->stride[2];
    pp.do_sb = a.dout->stride[0]; pp.do_sh = a.dout->stride[1]; pp.do_ss = a.dout->stride[2];
    pp.delta = delta;
    pp.dq_acc = deterministic ? nullptr : dq_acc;
    pp.units = pr.units; pp.H = pr.H; pp.rows = pr.Sq; pp.D = pr.D;
    pp.seq = sa;
    pp.status = status;
    if (launch_bwd_preprocess(pp, st) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (stage_mask & 2) {
    if (pr.max_k > 0) {
      BwdParams p;
      memset(&p, 0, sizeof(p));
      const int BM = bwd_block_m(kernel_width(pr.D)), BN = bwd_block_n();
      if ((s = make_map(&p.tm_q, a.q, BM)) != ATTN_OK) return s;
      if ((s = make_map(&p.tm_do, a.dout, BM)) != ATTN_OK) return s;
      if ((s = make_map(&p.tm_k, a.k, BN)) != ATTN_OK) return s;
      if ((s = make_map(&p.tm_v, a.v, BN)) != ATTN_OK) return s;
      // the epilogue's dK / dV stores: 32 keys x a slab of at most 64 of a compute
      // warpgroup's columns, swizzled like the staged slab (128 or 64 bytes a row)
      const int cw = std::min(bwd_epilogue_cols(kernel_width(pr.D)), 64);
      if ((s = make_map(&p.tm_dk, a.dk, 32, cw, cw * 2)) != ATTN_OK) return s;
      if ((s = make_map(&p.tm_dv, a.dv, 32, cw, cw * 2)) != ATTN_OK) return s;
      p.with_dq = deterministic ? 0 : 1;
      p.withhold_step = withheld_step_for_test();
      p.timeout_ns = p.withhold_step >= 0 ? 50000000ull : kWaitTimeoutNs;
      if (p.with_dq &&
          (s = make_map_acc(&p.tm_dq, dq_acc, (int64_t)pr.B * pr.H * pr.Sq, pr.D)) != ATTN_OK)
        return s;
      p.lse = reinterpret_cast<const float*>(a.lse->data);
      p.l_sb = a.lse->stride[0]; p.l_sh = a.lse->stride[1]; p.l_ss = a.lse->stride[2];
      p.delta = delta;
      p.dq_acc = dq_acc;
      p.dk = reinterpret_cast<uint16_t*>(a.dk->data);
      p.dk_sb = a.dk->stride[0]; p.dk_sh = a.dk->stride[1]; p.dk_ss = a.dk->stride[2];
      p.dv = reinterpret_cast<uint16_t*>(a.dv->data);
      p.dv_sb = a.dv->stride[0]; p.dv_sh = a.dv->stride[1]; p.dv_ss = a.dv->stride[2];
      p.H = pr.H;
      p.rows_q = pr.Sq;
      p.seq = sa;
      p.causal = causal ? 1 : 0;
      p.scale_log2 = sm_scale * 1.4426950408889634f;
      p.sm_scale = sm_scale;
      p.status = status;
      // key tiles (two CTAs each at d_head 256, one per half of d)
      const int n_tiles = (pr.max_k + BN - 1) / BN * bwd_ctas_per_key_tile(kernel_width(pr.D));
      // the operands every CTA of a head visits: Q, dO (16-bit) and, when this kernel
      // accumulates dQ, the fp32 accumulator
      const int uh = pr.units * pr.H;
      p.tiles = n_tiles;
      p.group = p.with_dq
          ? grid_group("bwd_main", kernel_width(pr.D), p.causal,
                       (double)pr.units * pr.H * pr.max_q * pr.D * 8, uh)
          : grid_group("bwd_main_nodq", kernel_width(pr.D), p.causal,
                       (double)pr.units * pr.H * pr.max_q * pr.D * 4, uh);
      if ((int64_t)n_tiles * uh > kMaxI32) return ATTN_ERR_UNSUPPORTED;  // 1-D grid
      const dim3 grid((unsigned)(n_tiles * uh));
      p.d_out = pr.D;
      if (a.bias != nullptr) {
        // size-1 batch / head dimensions broadcast: stride 0
        p.bias = reinterpret_cast<const uint16_t*>(a.bias->data);
        // the kernel stages each step's bias tile (its query rows x 128 keys) by TMA
        if ((s = make_map(&p.tm_bias, a.bias, bwd_block_m(kernel_width(pr.D)))) != ATTN_OK)
          return s;
        p.b_sb = a.bias->size[0] == 1 ? 0 : a.bias->stride[0];
        p.b_sh = a.bias->size[1] == 1 ? 0 : a.bias->stride[1];
        p.b_ss = a.bias->stride[2];
        if (dbias_sum) {
          // summed in fp32 over the units / heads that share the bias, rounded afterwards
          float* acc = reinterpret_cast<float*>(base + acc_off);
          if (cudaMemsetAsync(acc, 0, dbias_acc_bytes(a.bias), st) != cudaSuccess)
            return ATTN_ERR_CUDA;
          const int64_t Hb = a.bias->size[1], Sqb = a.bias->size[2], Skb = a.bias->size[3];
          p.dbias_acc = acc;
          p.dba_sb = a.bias->size[0] == 1 ? 0 : Hb * Sqb * Skb;
          p.dba_sh = Hb == 1 ? 0 : Sqb * Skb;
          p.dba_ss = Skb;
        } else if (a.dbias != nullptr) {
          p.dbias = reinterpret_cast<uint16_t*>(a.dbias->data);
          p.db_sb = a.dbias->stride[0];
          p.db_sh = a.dbias->stride[1];
          p.db_ss = a.dbias->stride[2];
        }
      }
      if (launch_bwd_main(p, kernel_width(pr.D), pr.f16, a.bias != nullptr, grid, st) !=
          cudaSuccess)
        return ATTN_ERR_CUDA;
    }
    if (dbias_sum) {
      DbiasPostParams dp;
      memset(&dp, 0, sizeof(dp));
      dp.acc = reinterpret_cast<const float*>(base + acc_off);
      dp.dbias = reinterpret_cast<uint16_t*>(a.dbias->data);
      dp.db_sb = a.dbias->stride[0];
      dp.db_sh = a.dbias->stride[1];
      dp.db_ss = a.dbias->stride[2];
      dp.rows = a.bias->size[0] * a.bias->size[1] * a.bias->size[2];
      dp.Hb = (int)a.bias->size[1];
      dp.Sq = (int)a.bias->size[2];
      dp.Sk = (int)a.bias->size[3];
      dp.f16 = pr.f16 ? 1 : 0;
      if (launch_dbias_epilogue(dp, st) != cudaSuccess) return ATTN_ERR_CUDA;
    }
  }
  if (stage_mask & 4) {
    BwdPostParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.dq_acc = dq_acc;
    pp.dq = reinterpret_cast<uint16_t*>(a.dq->data);
    pp.f16 = pr.f16 ? 1 : 0;
    pp.dq_sb = a.dq->stride[0]; pp.dq_sh = a.dq->stride[1]; pp.dq_ss = a.dq->stride[2];
    pp.units = pr.units; pp.H = pr.H; pp.rows = pr.Sq; pp.D = pr.D;
    pp.seq = sa;
    pp.sm_scale = sm_scale;
    if (launch_bwd_dq_epilogue(pp, st) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (stage_mask & 8) {
    BwdDqParams p;
    memset(&p, 0, sizeof(p));
    const int BMq = bwd_dq_block_m();
    if ((s = make_map(&p.tm_q, a.q, BMq)) != ATTN_OK) return s;
    if ((s = make_map(&p.tm_do, a.dout, BMq)) != ATTN_OK) return s;
    if ((s = make_map(&p.tm_k, a.k, 128)) != ATTN_OK) return s;
    if ((s = make_map(&p.tm_v, a.v, 128)) != ATTN_OK) return s;
    p.lse = reinterpret_cast<const float*>(a.lse->data);
    p.l_sb = a.lse->stride[0]; p.l_sh = a.lse->stride[1]; p.l_ss = a.lse->stride[2];
    p.delta = delta;
    p.dq = reinterpret_cast<uint16_t*>(a.dq->data);
    p.dq_sb = a.dq->stride[0]; p.dq_sh = a.dq->stride[1]; p.dq_ss = a.dq->stride[2];
    p.H = pr.H;
    p.rows_q = pr.Sq;
    p.seq = sa;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.sm_scale = sm_scale;
    p.status = status;
    p.d_out = pr.D;
    const int n_blk = (pr.max_q + BMq - 1) / BMq;
    // the operands every CTA of a head visits: K and V
    const int uh = pr.units * pr.H;
    p.tiles = n_blk;
    p.group = grid_group("bwd_dq", kernel_width(pr.D), p.causal,
                         (double)pr.units * pr.H * pr.max_k * pr.D * 4, uh);
    if ((int64_t)n_blk * uh > kMaxI32) return ATTN_ERR_UNSUPPORTED;  // 1-D grid
    const dim3 grid((unsigned)(n_blk * uh));
    if (launch_bwd_dq(p, kernel_width(pr.D), pr.f16, grid, st) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

// Host checks of a backward call's arguments (everything but the workspace); fills *pr.
attn_status bwd_validate(const BwdArgs& a, const int32_t* cu_q, const int32_t* cu_k, int compact,
                         int32_t num_seqs, int32_t max_q, int32_t max_k, float sm_scale,
                         bool deterministic, Problem* pr_out) {
  Problem& pr = *pr_out;
  attn_status s =
      make_problem(a.q, a.k, a.v, cu_q, cu_k, compact, num_seqs, max_q, max_k, &pr);
  if (s != ATTN_OK) return s;
  const attn_tensor4* qshaped[] = {a.o, a.dout, a.dq};
  for (const attn_tensor4* t : qshaped) {
    if ((s = check_tensor4(t)) != ATTN_OK) return s;
    if (!same_shape(a.q, t)) return ATTN_ERR_SHAPE;
    if (!same_dtype(a.q, t)) return ATTN_ERR_DTYPE;
  }
  const attn_tensor4* kshaped[] = {a.dk, a.dv};
  for (const attn_tensor4* t : kshaped) {
    if ((s = check_tensor4(t)) != ATTN_OK) return s;
    if (!same_shape(a.k, t)) return ATTN_ERR_SHAPE;
    if (!same_dtype(a.q, t)) return ATTN_ERR_DTYPE;
  }
  if ((s = check_lse(a.lse, pr)) != ATTN_OK) return s;
  if (!valid_scale(sm_scale)) return ATTN_ERR_UNSUPPORTED;
  if (a.bias != nullptr) {
    // as the biased forward; no deterministic form
    if (deterministic) return ATTN_ERR_UNSUPPORTED;
    if ((s = check_bias(a.bias, a.q, a.k, pr)) != ATTN_OK) return s;
    if (a.dbias != nullptr) {
      if ((s = check_tensor4(a.dbias)) != ATTN_OK) return s;
      if (!same_dtype(a.q, a.dbias)) return ATTN_ERR_DTYPE;
      if (!same_shape(a.bias, a.dbias)) return ATTN_ERR_SHAPE;
    }
  } else if (a.dbias != nullptr) {
    return ATTN_ERR_NULL;
  }
  return ATTN_OK;
}

attn_status bwd_common(const BwdArgs& a, const int32_t* cu_q, const int32_t* cu_k, int compact,
                       int32_t num_seqs, int32_t max_q, int32_t max_k, float sm_scale,
                       int causal, void* ws, size_t ws_bytes, void* stream,
                       bool deterministic = false) {
  Problem pr;
  attn_status s = bwd_validate(a, cu_q, cu_k, compact, num_seqs, max_q, max_k, sm_scale,
                               deterministic, &pr);
  if (s != ATTN_OK) return s;
  if (deterministic) return bwd_stage(1 | 2 | 8, a, pr, sm_scale, causal, ws, ws_bytes, stream, true);
  return bwd_stage(7, a, pr, sm_scale, causal, ws, ws_bytes, stream);
}

}  // namespace

namespace attn_sm103 {

attn_status bwd_check_args(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                           const attn_tensor4* o, const attn_tensor3* lse,
                           const attn_tensor4* dout, const int32_t* cu_seqlens_q,
                           const int32_t* cu_seqlens_k, float sm_scale,
                           const attn_tensor4* dq, const attn_tensor4* dk,
                           const attn_tensor4* dv) {
  BwdArgs a{q, k, v, o, dout, dq, dk, dv, lse};
  Problem pr;
  attn_status s = bwd_validate(a, cu_seqlens_q, cu_seqlens_k, 0, -1, 0, 0, sm_scale, false, &pr);
  if (s != ATTN_OK) return s;
  return check_device();
}

}  // namespace attn_sm103

// =============================================================================== C ABI
extern "C" {

size_t attn_fwd_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t D) {
  if (B <= 0 || H <= 0 || Sq <= 0 || D <= 0) return kFwdMinWorkspace;
  const int width = kernel_width((int)D);
  const int rows = fwd_block_m(width, false);
  const int64_t n_items = B * H * ((Sq + rows - 1) / rows);
  const size_t split = fwd_split_ws_bytes(n_items, width);
  return split > kFwdMinWorkspace ? split : kFwdMinWorkspace;
}

size_t attn_bwd_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t D) {
  return bwd_layout(B, H, Sq, D).total;
}

size_t attn_bwd_bias_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t D,
                                    int64_t Bb, int64_t Hb, int64_t Sq_b, int64_t Sk_b) {
  const size_t base = bwd_layout(B, H, Sq, D).total;
  if (Bb != 1 && Hb != 1) return base;
  const auto nn = [](int64_t x) { return (size_t)(x > 0 ? x : 0); };
  return align256(base) + nn(Bb) * nn(Hb) * nn(Sq_b) * nn(Sk_b) * 4;
}

size_t attn_bwd_deterministic_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t D) {
  return bwd_layout(B, H, Sq, D).dq_off;  // status word and Delta
}

attn_status attn_fwd(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, float sm_scale,
                     int causal, const attn_tensor4* o, const attn_tensor3* lse,
                     void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_common(q, k, v, cu_seqlens_q, cu_seqlens_k, 0, -1, 0, 0, sm_scale, causal, o, lse,
                    workspace, workspace_bytes, stream);
}

attn_status attn_fwd_bias(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                          const attn_tensor4* bias, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_k, float sm_scale, int causal,
                          const attn_tensor4* o, const attn_tensor3* lse, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return fwd_common(q, k, v, cu_seqlens_q, cu_seqlens_k, 0, -1, 0, 0, sm_scale, causal, o, lse,
                    workspace, workspace_bytes, stream, bias);
}

attn_status attn_fwd_compact_varlen_bias(const attn_tensor4* q, const attn_tensor4* k,
                                         const attn_tensor4* v, const attn_tensor4* bias,
                                         const int32_t* cu_seqlens_q,
                                         const int32_t* cu_seqlens_k, int32_t num_seqs,
                                         int32_t max_seqlen_q, int32_t max_seqlen_k,
                                         float sm_scale, int causal, const attn_tensor4* o,
                                         const attn_tensor3* lse, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (bias == nullptr) return ATTN_ERR_NULL;
  return fwd_common(q, k, v, cu_seqlens_q, cu_seqlens_k, 1, num_seqs, max_seqlen_q, max_seqlen_k,
                    sm_scale, causal, o, lse, workspace, workspace_bytes, stream, bias);
}

attn_status attn_fwd_padded_varlen(const attn_tensor4* q, const attn_tensor4* k,
                                   const attn_tensor4* v, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, float sm_scale, int causal,
                                   const attn_tensor4* o, const attn_tensor3* lse,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return ATTN_ERR_NULL;
  return attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, sm_scale, causal, o, lse, workspace,
                  workspace_bytes, stream);
}

attn_status attn_fwd_compact_varlen(const attn_tensor4* q, const attn_tensor4* k,
                                    const attn_tensor4* v, const int32_t* cu_seqlens_q,
                                    const int32_t* cu_seqlens_k, int32_t num_seqs,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k, float sm_scale,
                                    int causal, const attn_tensor4* o, const attn_tensor3* lse,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_common(q, k, v, cu_seqlens_q, cu_seqlens_k, 1, num_seqs, max_seqlen_q, max_seqlen_k,
                    sm_scale, causal, o, lse, workspace, workspace_bytes, stream);
}

attn_status attn_bwd(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                     const attn_tensor4* o, const attn_tensor3* lse, const attn_tensor4* dout,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, float sm_scale,
                     int causal, const attn_tensor4* dq, const attn_tensor4* dk,
                     const attn_tensor4* dv, void* workspace, size_t workspace_bytes,
                     void* stream) {
  BwdArgs a{q, k, v, o, dout, dq, dk, dv, lse};
  return bwd_common(a, cu_seqlens_q, cu_seqlens_k, 0, -1, 0, 0, sm_scale, causal, workspace,
                    workspace_bytes, stream);
}

attn_status attn_bwd_padded_varlen(const attn_tensor4* q, const attn_tensor4* k,
                                   const attn_tensor4* v, const attn_tensor4* o,
                                   const attn_tensor3* lse, const attn_tensor4* dout,
                                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                   float sm_scale, int causal, const attn_tensor4* dq,
                                   const attn_tensor4* dk, const attn_tensor4* dv,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return ATTN_ERR_NULL;
  return attn_bwd(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, sm_scale, causal, dq, dk,
                  dv, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_compact_varlen(const attn_tensor4* q, const attn_tensor4* k,
                                    const attn_tensor4* v, const attn_tensor4* o,
                                    const attn_tensor3* lse, const attn_tensor4* dout,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                    int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                                    float sm_scale, int causal, const attn_tensor4* dq,
                                    const attn_tensor4* dk, const attn_tensor4* dv,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  BwdArgs a{q, k, v, o, dout, dq, dk, dv, lse};
  return bwd_common(a, cu_seqlens_q, cu_seqlens_k, 1, num_seqs, max_seqlen_q, max_seqlen_k,
                    sm_scale, causal, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_bias(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                          const attn_tensor4* o, const attn_tensor3* lse, const attn_tensor4* dout,
                          const attn_tensor4* bias, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_k, float sm_scale, int causal,
                          const attn_tensor4* dq, const attn_tensor4* dk, const attn_tensor4* dv,
                          const attn_tensor4* dbias, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (bias == nullptr) return ATTN_ERR_NULL;
  BwdArgs a{q, k, v, o, dout, dq, dk, dv, lse, bias, dbias};
  return bwd_common(a, cu_seqlens_q, cu_seqlens_k, 0, -1, 0, 0, sm_scale, causal, workspace,
                    workspace_bytes, stream);
}

attn_status attn_bwd_compact_varlen_bias(
    const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v, const attn_tensor4* o,
    const attn_tensor3* lse, const attn_tensor4* dout, const attn_tensor4* bias,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t max_seqlen_q, int32_t max_seqlen_k, float sm_scale, int causal,
    const attn_tensor4* dq, const attn_tensor4* dk, const attn_tensor4* dv,
    const attn_tensor4* dbias, void* workspace, size_t workspace_bytes, void* stream) {
  if (bias == nullptr) return ATTN_ERR_NULL;
  BwdArgs a{q, k, v, o, dout, dq, dk, dv, lse, bias, dbias};
  return bwd_common(a, cu_seqlens_q, cu_seqlens_k, 1, num_seqs, max_seqlen_q, max_seqlen_k,
                    sm_scale, causal, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_deterministic(const attn_tensor4* q, const attn_tensor4* k,
                                   const attn_tensor4* v, const attn_tensor4* o,
                                   const attn_tensor3* lse, const attn_tensor4* dout,
                                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                   float sm_scale, int causal, const attn_tensor4* dq,
                                   const attn_tensor4* dk, const attn_tensor4* dv,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  BwdArgs a{q, k, v, o, dout, dq, dk, dv, lse};
  return bwd_common(a, cu_seqlens_q, cu_seqlens_k, 0, -1, 0, 0, sm_scale, causal, workspace,
                    workspace_bytes, stream, true);
}

attn_status attn_bwd_compact_varlen_deterministic(
    const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v, const attn_tensor4* o,
    const attn_tensor3* lse, const attn_tensor4* dout, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
    float sm_scale, int causal, const attn_tensor4* dq, const attn_tensor4* dk,
    const attn_tensor4* dv, void* workspace, size_t workspace_bytes, void* stream) {
  BwdArgs a{q, k, v, o, dout, dq, dk, dv, lse};
  return bwd_common(a, cu_seqlens_q, cu_seqlens_k, 1, num_seqs, max_seqlen_q, max_seqlen_k,
                    sm_scale, causal, workspace, workspace_bytes, stream, true);
}

attn_status attn_bwd_preprocess(const attn_tensor4* o, const attn_tensor4* dout,
                                const int32_t* cu_seqlens_q, int32_t num_seqs,
                                int32_t max_seqlen_q, void* workspace, size_t workspace_bytes,
                                void* stream) {
  // Shapes come from o; k/v are not needed by this stage, o stands in for them.
  Problem pr;
  const int compact = num_seqs >= 0;
  attn_status s = make_problem(o, o, o, cu_seqlens_q, cu_seqlens_q, compact, num_seqs,
                               max_seqlen_q, max_seqlen_q, &pr);
  if (s != ATTN_OK) return s;
  if ((s = check_tensor4(dout)) != ATTN_OK) return s;
  if (!same_shape(o, dout)) return ATTN_ERR_SHAPE;
  if (!same_dtype(o, dout)) return ATTN_ERR_DTYPE;
  BwdArgs a{o, o, o, o, dout, nullptr, nullptr, nullptr, nullptr};
  return bwd_stage(1, a, pr, 1.f, 0, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_main(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                          const attn_tensor3* lse, const attn_tensor4* dout,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                          int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                          float sm_scale, int causal, const attn_tensor4* dk,
                          const attn_tensor4* dv, void* workspace, size_t workspace_bytes,
                          void* stream) {
  Problem pr;
  const int compact = num_seqs >= 0;
  attn_status s = make_problem(q, k, v, cu_seqlens_q, cu_seqlens_k, compact, num_seqs,
                               max_seqlen_q, max_seqlen_k, &pr);
  if (s != ATTN_OK) return s;
  if ((s = check_tensor4(dout)) != ATTN_OK) return s;
  if (!same_shape(q, dout)) return ATTN_ERR_SHAPE;
  if (!same_dtype(q, dout)) return ATTN_ERR_DTYPE;
  const attn_tensor4* kshaped[] = {dk, dv};
  for (const attn_tensor4* t : kshaped) {
    if ((s = check_tensor4(t)) != ATTN_OK) return s;
    if (!same_shape(k, t)) return ATTN_ERR_SHAPE;
    if (!same_dtype(q, t)) return ATTN_ERR_DTYPE;
  }
  if ((s = check_lse(lse, pr)) != ATTN_OK) return s;
  if (!valid_scale(sm_scale)) return ATTN_ERR_UNSUPPORTED;
  BwdArgs a{q, k, v, q, dout, nullptr, dk, dv, lse};
  return bwd_stage(2, a, pr, sm_scale, causal, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_dq_epilogue(const attn_tensor4* dq, const int32_t* cu_seqlens_q,
                                 int32_t num_seqs, int32_t max_seqlen_q, float sm_scale,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  Problem pr;
  const int compact = num_seqs >= 0;
  attn_status s = make_problem(dq, dq, dq, cu_seqlens_q, cu_seqlens_q, compact, num_seqs,
                               max_seqlen_q, max_seqlen_q, &pr);
  if (s != ATTN_OK) return s;
  if (!valid_scale(sm_scale)) return ATTN_ERR_UNSUPPORTED;
  BwdArgs a{dq, dq, dq, dq, dq, dq, nullptr, nullptr, nullptr};
  return bwd_stage(4, a, pr, sm_scale, 0, workspace, workspace_bytes, stream);
}

attn_status attn_read_device_status(void* workspace, void* stream, int32_t* out) {
  if (workspace == nullptr || out == nullptr) return ATTN_ERR_NULL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(workspace, 0, sizeof(v), st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return ATTN_ERR_CUDA;
  *out = v;
  return ATTN_OK;
}

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "inconsistent tensor sizes";
    case ATTN_ERR_STRIDE: return "unsupported strides (D stride must be 1, others multiples of 8)";
    case ATTN_ERR_ALIGN: return "base pointer not 16-byte aligned";
    case ATTN_ERR_UNSUPPORTED:
      return "unsupported case (d_head, element type, device, sm_scale or size limits)";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA runtime or driver error";
    case ATTN_ERR_DEVICE_BAD_SEQLENS: return "device: inconsistent cu_seqlens (sequence skipped)";
    case ATTN_ERR_DEVICE_TIMEOUT: return "device: pipeline wait timed out";
    case ATTN_ERR_DTYPE: return "tensors of one call have different element types";
  }
  return "unknown status";
}

}  // extern "C"
