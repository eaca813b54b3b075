/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused scaled-dot-product attention library.
 *
 * The operation is FlashAttention-style scaled dot-product attention ("Investigate a new
 * SDPA IR node", nvFuser issue #2278): for every (batch or sequence, head)
 *
 *     S = sm_scale * Q K^T,  P = softmax(S) over the visible keys,  O = P V,
 *     LSE_i = log sum_j exp(S_ij)   (natural log, stored by the forward pass),
 *
 * and the backward pass rebuilds P from LSE to produce dQ, dK, dV of a loss whose gradient
 * with respect to O is dO. The forward pass returns LSE because backward consumes it: the
 * nvFuser page splits the op into a forward node that stashes what backward needs and a
 * backward node that consumes it (SdpaOpFwd / SdpaOpBwd).
 *
 * Layout. Every tensor is rank 4, (B, H, S, D) ("BHSD", the only layout of the AOTriton
 * flash API -- "Add varlen support to AOTriton's Flash Attention", last comment: new layouts
 * get new APIs, not flags). Strides are in ELEMENTS and arbitrary, except that the D stride
 * must be 1, the other strides must be multiples of 8 elements (16 bytes) and base pointers
 * 16-byte aligned (tensor-memory-accelerator requirements). Q, K, V, O, dO, dQ, dK, dV share
 * one 16-bit element type, bf16 or fp16 (attn_tensor4.dtype); arithmetic accumulates in fp32.
 * LSE is fp32 with shape (B, H, Sq). Q/K/V/O share B, H and D; seqlen_q and seqlen_k
 * may differ ("[RFC] Goal for triton.ops.flash_attention" lists a different number of
 * queries and keys as a missing case; the AOTriton issue #12 page states that QKVO share a
 * dtype and shape except for seqlen_q vs seqlen_k). d_head must be 32, 64, 96 or 128 (32
 * and 96 run on the 64- and 128-wide kernels with zero-filled columns; only the real
 * columns of the outputs are written), or 256 in the calls without a bias (the forward with
 * one 128-row query tile per CTA; the backward with two CTAs per key tile, one per half of d);
 * the deterministic backward returns ATTN_ERR_UNSUPPORTED for 256.
 *
 * Masking. causal != 0 applies a top-left aligned mask: query i sees key j iff j <= i,
 * indices local to the sequence. Keys at or past a sequence's length are never seen.
 *
 * Variable length (AOTriton PR #31, "Add varlen support to AOTriton's Flash Attention"):
 *   - compact varlen: the *_compact_varlen calls; tensors are (1, H, T, D) -- a THD tensor
 *     viewed with transpose + unsqueeze -- and sequence s owns rows [cu[s], cu[s+1]).
 *     Batch must be exactly 1 (the page says extra batches are not processed; here they
 *     are an error, never silently ignored).
 *   - padded varlen: attn_fwd / attn_bwd with non-NULL cu_seqlens (or the *_padded_varlen
 *     aliases); batch b is valid on rows [0, cu[b+1]-cu[b]) of its own (B, H, S, D) slice,
 *     i.e. data starts at offset 0 inside each batch, as in the padded-varlen kernel
 *     prologue quoted on that page.
 *   All sequence-length arguments and cu_seqlens entries are int32 (same page, note 3).
 *
 * Output contract. Rows at or past a sequence's length are not written (the kernel
 * prologue on the AOTriton page returns early for them). A sequence with no keys gets
 * O = 0 and LSE = -inf on its valid rows and zero dQ.
 *
 * Ownership and asynchrony. The caller owns every buffer (inputs, outputs, workspace);
 * the library allocates nothing and keeps no per-call state. Pointers passed as "device"
 * must be device memory of the current device. Calls are asynchronous and ordered on the
 * given CUDA stream (a cudaStream_t passed as void*; NULL = legacy default stream).
 *
 * Errors. Argument errors are detected on the host, return a status != ATTN_OK and launch
 * nothing ("no silently incorrect results": the RFC page above warns that the Triton demo
 * can silently return wrong answers on unexpected shapes or strides). Errors only visible
 * on the device (inconsistent cu_seqlens, a pipeline wait that timed out) are written to a
 * status word (int32) at offset 0 of the workspace; read it with attn_read_device_status.
 * The word is sticky: kernels only ever set it, so the caller zeroes it once when the
 * workspace is allocated, and attn_read_device_status clears it after reading. A sequence
 * whose cu_seqlens are inconsistent is skipped, never read out of bounds.
 *
 * Environment. The library reads these variables, none needed in normal use:
 *   ATTN_GRID_ORDER="<kernel>:tile|seq|g<N>[,...]" forces the CTA order of a kernel's causal
 *     grids (kernel = fwd, bwd_main, bwd_main_nodq or bwd_dq; g<N>: groups of N (unit, head)
 *     pairs); otherwise the order comes from a table measured on GB300 (the sweep that
 *     writes the table sets it). Results do not depend on the order.
 *   ATTN_FWD_PERSISTENT=0 turns off the forward's work stealing (with more query blocks
 *     than SMs, running CTAs take over the blocks of CTAs not yet launched);
 *     ATTN_FWD_CTAS=n launches n CTAs, CTA c taking blocks c, c + n, ... Results do not
 *     depend on the grid.
 *   ATTN_FWD_SPLIT=0|1 turns the forward's split grid off, or on for every non-causal dense
 *     grid with fewer query blocks than SMs (default: the table measured on GB300 decides,
 *     by the block count and the key tiles per block). Results agree within rounding (the
 *     parts are merged in a fixed order). A split grid takes its size from ATTN_FWD_CTAS too
 *     (at most 256 CTAs).
 *   ATTN_TEST_WITHHOLD_KV_TILE=j / ATTN_TEST_WITHHOLD_Q_STEP=i (failure-detection tests):
 *     the forward loads no key tile from j on / the backward skips query step i, and every
 *     wait gives up after 50 ms, so the call ends with ATTN_ERR_DEVICE_TIMEOUT in the status
 *     word instead of hanging.
 */
#ifndef ATTN_SM103_ATTN_H_
#define ATTN_SM103_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of the rank-4 tensors. */
typedef enum { ATTN_DTYPE_BF16 = 0, ATTN_DTYPE_F16 = 1 } attn_dtype;

/* A rank-4 (B, H, S, D) tensor view; strides in elements; dtype is an attn_dtype. */
typedef struct {
  void* data;
  int64_t size[4];
  int64_t stride[4];
  int32_t dtype;
} attn_tensor4;

/* A rank-3 (B, H, S) fp32 tensor view (LSE); strides in elements. */
typedef struct {
  void* data;
  int64_t size[3];
  int64_t stride[3];
} attn_tensor3;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL = 1,          /* a required pointer is NULL */
  ATTN_ERR_SHAPE = 2,         /* inconsistent sizes (B, H, D, S), or compact batch != 1 */
  ATTN_ERR_STRIDE = 3,        /* D stride != 1, or a stride not a multiple of 8 elements */
  ATTN_ERR_ALIGN = 4,         /* base pointer not 16-byte aligned */
  ATTN_ERR_UNSUPPORTED = 5,   /* d_head not 32/64/96/128/256 (256: no bias and no
                                 deterministic backward), device not sm_103, or size limits */
  ATTN_ERR_WORKSPACE = 6,     /* workspace NULL or smaller than the *_workspace_size value */
  ATTN_ERR_CUDA = 7,          /* a CUDA runtime/driver call failed (launch, tensor map) */
  ATTN_ERR_DEVICE_BAD_SEQLENS = 8, /* device: cu_seqlens not monotone or past the tensor */
  ATTN_ERR_DEVICE_TIMEOUT = 9, /* device: a bounded pipeline wait gave up */
  ATTN_ERR_DTYPE = 10          /* tensors of one call with different element types */
} attn_status;

/* Workspace bytes for attn_fwd* with Q of shape (B, H, Sq, D) (compact: B = 1, Sq = total
 * query tokens). The forward calls need 256 bytes (the device status word); given this many
 * (zeroed once, like every workspace), a non-causal dense call with at most half as many
 * query blocks (256 rows; 128 at head size 256) as the GPU has SMs and long enough key
 * ranges (a table measured on GB300: at least 16 key tiles of 128 at head sizes up to 128,
 * 32 at 256) splits each block's key range over several CTAs and merges the parts (the
 * blocks' counters at bytes 1024..2047
 * return to zero at the end of every call; after ATTN_ERR_DEVICE_TIMEOUT zero the workspace
 * again). One workspace of max(attn_fwd_workspace_size, attn_bwd_workspace_size) bytes
 * serves both passes: no backward kernel writes bytes 4..2047. */
size_t attn_fwd_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t D);

/* Workspace bytes needed by attn_bwd* (status word, per-row Delta = rowsum(dO * O) in fp32,
 * and an fp32 dQ accumulator of shape (B, H, Sq, D)). */
size_t attn_bwd_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t D);

/*
 * Forward pass, dense (cu_seqlens_q == cu_seqlens_k == NULL) or padded varlen (both
 * non-NULL, int32 device arrays of B+1 prefix sums; only the differences are used).
 *   q: (B, H, Sq, D)          k, v: (B, H, Sk, D)          (bf16 or fp16, one type)
 *   o: (B, H, Sq, D) out      lse: (B, H, Sq) fp32 out (natural-log logsumexp)
 *   workspace: device, >= 256 bytes, attn_fwd_workspace_size bytes for the split grid (may
 *   be NULL with 0 bytes: device errors are then not reported). stream: cudaStream_t.
 */
attn_status attn_fwd(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, float sm_scale,
                     int causal, const attn_tensor4* o, const attn_tensor3* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward pass with an additive attention bias (the bias argument that the AOTriton varlen
 * page reserves, note 1 of "Add varlen support to AOTriton's Flash Attention"):
 * S = sm_scale * Q K^T + bias, then mask and softmax; lse is that of the biased scores.
 * Arguments as in attn_fwd (dense, or padded varlen with cu_seqlens), plus
 *   bias: (Bb, Hb, Sq, Sk) in q's element type, Bb in {1, B} and Hb in {1, H} (size 1
 *         broadcasts; pass size-1 dimensions, not zero strides). D stride 1; the Sq stride
 *         (and the other strides) a multiple of 8 elements, so a row of Sk keys is padded to
 *         a multiple of 8 elements when Sk is not; 16-byte aligned base. Padded varlen uses
 *         the block at offset 0 of each batch, like q.
 * Supported for d_head 32, 64, 96 and 128 (ATTN_ERR_UNSUPPORTED for 256). A NULL bias is
 * the same as attn_fwd. Errors as attn_fwd; ATTN_ERR_SHAPE for a bias whose sizes do not
 * fit. attn_bwd_bias is the matching backward; attn_fwd_compact_varlen_bias the compact
 * form.
 */
attn_status attn_fwd_bias(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                          const attn_tensor4* bias, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_k, float sm_scale, int causal,
                          const attn_tensor4* o, const attn_tensor3* lse, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Compact varlen forward with an additive bias: arguments as in attn_fwd_compact_varlen plus
 *   bias: (Bb, Hb, Sq_b, Sk_b), Bb in {1, num_seqs}, Hb in {1, H}, Sq_b >= max_seqlen_q and
 *         Sk_b >= max_seqlen_k (the sequence-length bounds of the call; pass them). Sequence s
 *         finds its [len_q, len_k] block at offset 0 of slice s of the first dimension (slice
 *         0 when Bb = 1), as a padded batch entry does: the pages reserve the argument without
 *         fixing its layout, and offset-0 blocks keep every tensor-memory-accelerator copy of
 *         the bias on a 16-byte boundary. Strides as for attn_fwd_bias. Errors as
 *         attn_fwd_compact_varlen, ATTN_ERR_SHAPE for a bias whose sizes do not fit.
 */
attn_status attn_fwd_compact_varlen_bias(const attn_tensor4* q, const attn_tensor4* k,
                                         const attn_tensor4* v, const attn_tensor4* bias,
                                         const int32_t* cu_seqlens_q,
                                         const int32_t* cu_seqlens_k, int32_t num_seqs,
                                         int32_t max_seqlen_q, int32_t max_seqlen_k,
                                         float sm_scale, int causal, const attn_tensor4* o,
                                         const attn_tensor3* lse, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * Backward pass matching attn_fwd (same q, k, v, cu_seqlens, sm_scale, causal; o and lse
 * as returned by attn_fwd). dout: (B, H, Sq, D). Writes dq (B, H, Sq, D), dk and dv
 * (B, H, Sk, D), all in q's element type. workspace: device, >= attn_bwd_workspace_size
 * bytes, required.
 * Runs three kernels in stream order: attn_bwd_preprocess, attn_bwd_main and
 * attn_bwd_dq_epilogue below.
 */
attn_status attn_bwd(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                     const attn_tensor4* o, const attn_tensor3* lse, const attn_tensor4* dout,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, float sm_scale,
                     int causal, const attn_tensor4* dq, const attn_tensor4* dk,
                     const attn_tensor4* dv, void* workspace, size_t workspace_bytes,
                     void* stream);

/*
 * Backward pass matching attn_fwd_bias: arguments as in attn_bwd plus the bias given to the
 * forward pass (non-NULL, same limits). dbias, optional (NULL: no bias gradient), has the
 * bias's shape and receives the gradient with respect to the bias:
 *   - a bias whose batch and head dimensions both have more than one entry: dS itself,
 *     rounded to the element
 *     type, written only on the (query, key) tiles the kernel visits -- entries in fully
 *     masked causal tiles and past a sequence's length are left as they are, so pass it
 *     zeroed;
 *   - a bias with a size-1 batch or head dimension: dS summed over the units and heads that
 *     share each entry, in fp32 in the workspace, then rounded; every entry of dbias is
 *     written (zero where no sequence reaches). The workspace must then hold
 *     attn_bwd_bias_workspace_size bytes. The fp32 sums are added in an order that varies
 *     from run to run (last bits only).
 */
attn_status attn_bwd_bias(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                          const attn_tensor4* o, const attn_tensor3* lse, const attn_tensor4* dout,
                          const attn_tensor4* bias, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_k, float sm_scale, int causal,
                          const attn_tensor4* dq, const attn_tensor4* dk, const attn_tensor4* dv,
                          const attn_tensor4* dbias, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * Workspace bytes attn_bwd_bias and attn_bwd_compact_varlen_bias need for a bias of shape
 * (Bb, Hb, Sq_b, Sk_b): attn_bwd_workspace_size(B, H, Sq, D), plus room for the fp32 sums
 * of the bias gradient when Bb or Hb is 1 (used only when a dbias is requested).
 */
size_t attn_bwd_bias_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t D, int64_t Bb,
                                    int64_t Hb, int64_t Sq_b, int64_t Sk_b);

/*
 * Compact varlen backward with an additive bias: arguments as in attn_bwd_compact_varlen plus
 * the bias given to attn_fwd_compact_varlen_bias and an optional dbias of its shape, written
 * as described for attn_bwd_bias (the units are the sequences).
 */
attn_status attn_bwd_compact_varlen_bias(
    const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v, const attn_tensor4* o,
    const attn_tensor3* lse, const attn_tensor4* dout, const attn_tensor4* bias,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t max_seqlen_q, int32_t max_seqlen_k, float sm_scale, int causal,
    const attn_tensor4* dq, const attn_tensor4* dk, const attn_tensor4* dv,
    const attn_tensor4* dbias, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Deterministic backward: same arguments and results as attn_bwd, and the same bits on every
 * run. attn_bwd adds each key tile's dQ contribution into an fp32 accumulator with
 * reductions whose order varies from run to run; here a second kernel owns each block of
 * 128 query rows, walks the key tiles in order and accumulates dQ in tensor memory, while
 * the key-tile kernel computes only dK and dV. S and dP are therefore computed twice (seven
 * products per tile instead of five). workspace: device, >= attn_bwd_workspace_size bytes
 * is always enough; only the status word and Delta are used (the fp32 accumulator is not),
 * so attn_bwd_deterministic_workspace_size bytes suffice. Determinism assumes the same
 * device, inputs and launch configuration.
 */
size_t attn_bwd_deterministic_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t D);
attn_status attn_bwd_deterministic(const attn_tensor4* q, const attn_tensor4* k,
                                   const attn_tensor4* v, const attn_tensor4* o,
                                   const attn_tensor3* lse, const attn_tensor4* dout,
                                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                   float sm_scale, int causal, const attn_tensor4* dq,
                                   const attn_tensor4* dk, const attn_tensor4* dv,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* Compact varlen forward: q, o (1, H, Tq, D); k, v (1, H, Tk, D); lse (1, H, Tq).
 * cu_seqlens_q / cu_seqlens_k: int32 device arrays of num_seqs+1 prefix sums into the
 * token axis. max_seqlen_q / max_seqlen_k: host upper bounds on the sequence lengths, used
 * only to size the grid (pass <= 0 to use Tq / Tk); a length above the bound is reported
 * as ATTN_ERR_DEVICE_BAD_SEQLENS and that sequence is skipped. */
attn_status attn_fwd_compact_varlen(const attn_tensor4* q, const attn_tensor4* k,
                                    const attn_tensor4* v, const int32_t* cu_seqlens_q,
                                    const int32_t* cu_seqlens_k, int32_t num_seqs,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k, float sm_scale,
                                    int causal, const attn_tensor4* o, const attn_tensor3* lse,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Compact varlen backward; arguments as in attn_fwd_compact_varlen and attn_bwd. */
attn_status attn_bwd_compact_varlen(const attn_tensor4* q, const attn_tensor4* k,
                                    const attn_tensor4* v, const attn_tensor4* o,
                                    const attn_tensor3* lse, const attn_tensor4* dout,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                    int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                                    float sm_scale, int causal, const attn_tensor4* dq,
                                    const attn_tensor4* dk, const attn_tensor4* dv,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Deterministic compact varlen backward; arguments as in attn_bwd_compact_varlen, results and
 * workspace as in attn_bwd_deterministic. */
attn_status attn_bwd_compact_varlen_deterministic(
    const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v, const attn_tensor4* o,
    const attn_tensor3* lse, const attn_tensor4* dout, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
    float sm_scale, int causal, const attn_tensor4* dq, const attn_tensor4* dk,
    const attn_tensor4* dv, void* workspace, size_t workspace_bytes, void* stream);

/* Padded varlen under its own name (the AOTriton page plans "attn_?wd_padded_varlen");
 * identical to attn_fwd / attn_bwd except that cu_seqlens must be non-NULL. */
attn_status attn_fwd_padded_varlen(const attn_tensor4* q, const attn_tensor4* k,
                                   const attn_tensor4* v, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, float sm_scale, int causal,
                                   const attn_tensor4* o, const attn_tensor3* lse,
                                   void* workspace, size_t workspace_bytes, void* stream);
attn_status attn_bwd_padded_varlen(const attn_tensor4* q, const attn_tensor4* k,
                                   const attn_tensor4* v, const attn_tensor4* o,
                                   const attn_tensor3* lse, const attn_tensor4* dout,
                                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                   float sm_scale, int causal, const attn_tensor4* dq,
                                   const attn_tensor4* dk, const attn_tensor4* dv,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three stages of attn_bwd / attn_bwd_compact_varlen, callable one by one (timing,
 * profiling). num_seqs < 0 selects the dense / padded form (cu_seqlens NULL = dense),
 * num_seqs >= 0 the compact form. Each validates its own arguments like attn_bwd.
 *  - attn_bwd_preprocess: Delta_i = sum_d dO_id * O_id into the workspace and zeroes the
 *    fp32 dQ accumulator. Memory-bound.
 *  - attn_bwd_main: recomputes P from LSE per key tile, accumulates dK and dV in tensor
 *    memory and writes them, and adds dS K into the dQ accumulator.
 *  - attn_bwd_dq_epilogue: dq = sm_scale * accumulator in dq's element type. Memory-bound.
 */
attn_status attn_bwd_preprocess(const attn_tensor4* o, const attn_tensor4* dout,
                                const int32_t* cu_seqlens_q, int32_t num_seqs,
                                int32_t max_seqlen_q, void* workspace, size_t workspace_bytes,
                                void* stream);
attn_status attn_bwd_main(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                          const attn_tensor3* lse, const attn_tensor4* dout,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                          int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                          float sm_scale, int causal, const attn_tensor4* dk,
                          const attn_tensor4* dv, void* workspace, size_t workspace_bytes,
                          void* stream);
attn_status attn_bwd_dq_epilogue(const attn_tensor4* dq, const int32_t* cu_seqlens_q,
                                 int32_t num_seqs, int32_t max_seqlen_q, float sm_scale,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass for callers that cannot allocate device memory (allocator-free runtimes,
 * plugins that may not allocate while executing, fixed up-front memory budgets). The pages
 * have no counterpart of this entry point; it exists for such callers only.
 * Same arguments and results as attn_bwd (dense or padded varlen), without a workspace:
 * the scratch space (status word, Delta, fp32 dQ accumulator) comes from a fixed array of
 * ATTN_NOALLOC_SCRATCH_BYTES in the library's own device memory, which every GPU that loads
 * the library holds until the process exits. Nothing is allocated. Returns
 * ATTN_ERR_WORKSPACE when attn_bwd_workspace_size(B, H, Sq, D) exceeds that size. The first
 * call on each device looks up the array's device address (with that device current) and
 * should come before any stream capture. All calls share the array: calls whose executions
 * overlap on the GPU race. The array's status word is cleared at the start of every call;
 * attn_noalloc_read_device_status reads the device-side status of the last call.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
attn_status attn_bwd_noalloc(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                             const attn_tensor4* o, const attn_tensor3* lse,
                             const attn_tensor4* dout, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, float sm_scale, int causal,
                             const attn_tensor4* dq, const attn_tensor4* dk,
                             const attn_tensor4* dv, void* stream);
/* The device status word of the no-alloc array (ATTN_OK or an ATTN_ERR_DEVICE_* code of the
 * calls since it was last read), read after synchronising `stream` and cleared, like
 * attn_read_device_status. Returns ATTN_ERR_NULL when out is NULL. */
attn_status attn_noalloc_read_device_status(void* stream, int32_t* out);

/* Reads the device status word at offset 0 of `workspace` after synchronising `stream`
 * (the only blocking call of the library) and clears it. *out receives ATTN_OK or one of
 * the ATTN_ERR_DEVICE_* codes. */
attn_status attn_read_device_status(void* workspace, void* stream, int32_t* out);

/* Static, human-readable name of a status code. */
const char* attn_status_string(attn_status s);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SM103_ATTN_H_ */
