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
// fetched once per device with cudaGetSymbolAddress, with that device
// current, on the first call made on that device.  That first call should
// therefore come before any stream capture begins.
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
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr size_t kStatusOffset = kNoAllocScratchBytes - 256;  // last 256 bytes: status word

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once
// per device); nullptr if the address could not be obtained.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
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
