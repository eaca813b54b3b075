// attn_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point where they
// run the backward pass: code inside an allocator-free runtime, a plugin whose host forbids
// allocation during its execute step, or an embedded caller with a fixed memory budget that
// was committed up front. attn_bwd needs a caller-provided workspace (status word, the
// per-row Delta and the fp32 dQ accumulator); this entry point supplies that workspace from
// a fixed-size array in the library's own device memory instead, so the caller passes only
// inputs and outputs.
//
// The array is a file-scope static __device__ buffer of kNoallocScratchBytes: every GPU that
// loads this library's code holds it until the process exits. Host code cannot use the
// array's name as a device address (it names a host-side shadow), so on the first call on
// each device the device address is looked up with cudaGetSymbolAddress, with that device
// current, and cached; that first call should therefore come before any stream capture.
// Every call shares the one array and it keeps the previous call's contents: the status
// word is cleared at the start of each call and the dQ accumulator is zeroed by the
// backward preprocessing kernel. Calls whose executions overlap on the GPU (different
// streams, or different host threads without ordering) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn.h"

namespace {

constexpr size_t kNoallocScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once per device).
attn_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_bwd_noalloc(const attn_tensor4* q, const attn_tensor4* k,
                                        const attn_tensor4* v, const attn_tensor4* o,
                                        const attn_tensor3* lse, const attn_tensor4* dout,
                                        const int32_t* cu_seqlens_q,
                                        const int32_t* cu_seqlens_k, float sm_scale,
                                        int causal, const attn_tensor4* dq,
                                        const attn_tensor4* dk, const attn_tensor4* dv,
                                        void* stream) {
  if (q == nullptr) return ATTN_ERR_NULL;
  const size_t need = attn_bwd_workspace_size(q->size[0], q->size[1], q->size[2], q->size[3]);
  if (need > kNoallocScratchBytes) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  attn_status s = scratch_address(&scratch);
  if (s != ATTN_OK) return s;
  // The device status word starts at zero for every call (memset, not an allocation).
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return attn_bwd(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, sm_scale, causal, dq, dk,
                  dv, scratch, kNoallocScratchBytes, stream);
}
