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
// array's name as a device address (it names a host-side shadow), so the first call on each
// device looks the device address up with cudaGetSymbolAddress, with that device current,
// and caches it together with the id of the CUDA context it belongs to; that first call should
// therefore come before any stream capture. A call that finds a different context current on
// the device (after cudaDeviceReset, or once the primary context was released and created
// again, the module is loaded anew and the array may have moved) looks the address up again.
// Every call shares the one array and it keeps the previous call's contents: the status
// word is cleared at the start of each call and the dQ accumulator is zeroed by the
// backward preprocessing kernel. Calls whose executions overlap on the GPU (different
// streams, or different host threads without ordering) race on the array.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn.h"
#include "attn_launch.h"

namespace {

constexpr size_t kNoallocScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchEntry {
  void* ptr;
  unsigned long long ctx_id;
};
ScratchEntry g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Id of the calling thread's current CUDA context (driver entry points, looked up once).
// Returns false when no context is current yet or the driver lacks the calls.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's current context (looked up
// once per device and context).
attn_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& e = g_scratch[dev];
  if (e.ptr == nullptr || !have_ctx || e.ctx_id != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return ATTN_ERR_CUDA;
    // the lookup makes the device's primary context current if none was
    if (!current_context_id(&ctx)) return ATTN_ERR_CUDA;
    e.ptr = p;
    e.ctx_id = ctx;
  }
  *out = e.ptr;
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
  // every argument check first, so that a rejected call puts nothing on the stream
  attn_status s = attn_sm103::bwd_check_args(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k,
                                             sm_scale, dq, dk, dv);
  if (s != ATTN_OK) return s;
  const size_t need = attn_bwd_workspace_size(q->size[0], q->size[1], q->size[2], q->size[3]);
  if (need > kNoallocScratchBytes) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((s = scratch_address(&scratch)) != ATTN_OK) return s;
  // The device status word starts at zero for every call (memset, not an allocation).
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return attn_bwd(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, sm_scale, causal, dq, dk,
                  dv, scratch, kNoallocScratchBytes, stream);
}

// The status word of the array (offset 0): read after synchronising the stream, then cleared,
// as attn_read_device_status does for a workspace.
extern "C" attn_status attn_noalloc_read_device_status(void* stream, int32_t* out) {
  if (out == nullptr) return ATTN_ERR_NULL;
  void* scratch = nullptr;
  const attn_status s = scratch_address(&scratch);
  if (s != ATTN_OK) return s;
  return attn_read_device_status(scratch, stream, out);
}
