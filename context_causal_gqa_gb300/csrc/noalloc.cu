// noalloc.cu -- ccg_attn_bwd_noalloc: the backward for callers that cannot
// allocate device memory.
//
// Some callers of this library are handed device pointers for their inputs
// and outputs but own no allocator: a plugin inside a host framework that
// manages every byte of device memory itself, or code that must not call
// cudaMalloc after start-up (latency-critical loops, memory budgets fixed at
// initialisation).  Such callers cannot provide the workspace that
// ccg_attn_bwd needs (the work plan and the Delta = rowsum(O * dO) vector).
// For them, this entry point takes its scratch from a fixed-size array that
// lives in the library's own device image instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kNoAllocScratchBytes of device memory for it until the
// process exits.  Host code cannot use the array's name as a device address
// (in host code it names a host-side stand-in); the device address is
// fetched with cudaGetSymbolAddress, with that device current, on the first
// call made on that device, and again on the first call after the device's
// context changed (a device reset).  That first call should therefore come
// before any stream capture begins.
//
// Every call on a device shares the one array and it keeps the previous
// call's contents: the plan and Delta are fully rewritten by every call
// before they are read, and the internal status word (used when the caller
// passes no status word) is cleared at the start of every call.  Calls whose
// execution overlaps on the GPU (different streams, or different host
// threads without ordering) race on the array and must not be issued.
//
// There is no counterpart of this entry point in the TransformerEngine pull
// request the rest of the library follows.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr size_t kStatusOffset = kNoAllocScratchBytes - 256;  // last 256 bytes: status word

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;

// The cached address of the array on one device, with the CUDA context it
// was looked up in.  A device reset (cudaDeviceReset) or a destroyed and
// re-created primary context reloads the library's device image, which may
// place the array elsewhere: the address is looked up again whenever the
// current context differs from the one it was taken in.
struct ScratchCache {
  CUcontext ctx = nullptr;
  void* ptr = nullptr;
};
ScratchCache g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (the library has
// no link-time dependency on the driver library).
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch array on the current device, looked up with
// that device current on its first use in the current context; nullptr if
// the address could not be obtained.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr) return nullptr;
  CUcontext ctx = nullptr;                       // null before the runtime's first use on this thread
  if (get_ctx(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchCache& c = g_scratch[dev];
  if (ctx != nullptr && c.ptr != nullptr && c.ctx == ctx) return c.ptr;
  // the lookup makes the device's primary context current if none was
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
  c.ctx = ctx;
  c.ptr = p;
  return c.ptr;
}

}  // namespace

extern "C" {

ccg_status ccg_attn_bwd_noalloc(const ccg_attn_desc* desc, const void* q, const void* k, const void* v,
                                const void* o, const void* dout, const float* lse,
                                const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, void* dq,
                                void* dk, void* dv, int32_t* d_status, ccg_stream_t stream) {
  const size_t need = ccg_workspace_size(desc, 1);
  if (need == 0) return desc == nullptr ? CCG_ERR_INVALID_ARG : CCG_ERR_UNSUPPORTED;
  if (need > kStatusOffset) return CCG_ERR_WORKSPACE;   // problem too large for the fixed scratch
  auto* base = static_cast<unsigned char*>(scratch_for_current_device());
  if (base == nullptr) return CCG_ERR_CUDA;
  int32_t* status = d_status;
  if (status == nullptr) {
    status = reinterpret_cast<int32_t*>(base + kStatusOffset);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return CCG_ERR_CUDA;
  }
  return ccg_attn_bwd(desc, q, k, v, o, dout, lse, cu_seqlens, cu_seqlens_padded, dq, dk, dv, base,
                      kStatusOffset, status, stream);
}

}  // extern "C"
