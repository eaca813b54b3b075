// Internal launch entry points between the C ABI (attn_api.cu) and the kernel files.
#pragma once
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "attn_common.cuh"

namespace attn_sm103 {

// Forward: grid = (query blocks, H, B or num_seqs); a block covers fwd_block_m(width, bias)
// query rows (width = kernel width 64, 128 or 256), loaded with a Q tensor map whose box has
// fwd_box_rows() rows.
int fwd_block_m(int width, bool bias);
int fwd_box_rows();
cudaError_t launch_attn_fwd(const FwdParams& p, int D, bool f16, bool bias, dim3 grid,
                            cudaStream_t stream);

// Backward stages.
int bwd_block_m(int D);  // query rows per inner step of the main kernel
int bwd_block_n();       // key rows per CTA of the main kernel
int bwd_ctas_per_key_tile(int D);  // 2 at d_head 256 (one per half of d), else 1
int bwd_epilogue_cols(int D);      // dK / dV columns a compute warpgroup stores
cudaError_t launch_bwd_preprocess(const BwdPreParams& p, cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdParams& p, int D, bool f16, bool bias, dim3 grid,
                            cudaStream_t stream);
cudaError_t launch_bwd_dq_epilogue(const BwdPostParams& p, cudaStream_t stream);
cudaError_t launch_dbias_epilogue(const DbiasPostParams& p, cudaStream_t stream);
// Deterministic dQ: grid = (query blocks, H, units); a block covers bwd_dq_block_m() rows.
int bwd_dq_block_m();
cudaError_t launch_bwd_dq(const BwdDqParams& p, int D, bool f16, dim3 grid, cudaStream_t stream);

// Every host check attn_bwd (dense or padded varlen) makes before it touches the stream, the
// workspace aside: arguments, head size and device. Launches nothing.
attn_status bwd_check_args(const attn_tensor4* q, const attn_tensor4* k, const attn_tensor4* v,
                           const attn_tensor4* o, const attn_tensor3* lse,
                           const attn_tensor4* dout, const int32_t* cu_seqlens_q,
                           const int32_t* cu_seqlens_k, float sm_scale,
                           const attn_tensor4* dq, const attn_tensor4* dk,
                           const attn_tensor4* dv);

}  // namespace attn_sm103
