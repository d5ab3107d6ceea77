// gdp_chunk_fwd_noalloc: the chunked forward with its scratch memory in a
// fixed device array owned by this library, for callers that cannot allocate.
//
// Some callers have no way to obtain device memory for a workspace at the
// point where they run the forward pass: code that executes under a
// pre-planned memory budget where every byte was reserved up front (embedded
// or safety-critical inference runtimes), code called from inside another
// framework's allocator or memory-pool callbacks (where re-entering the
// allocator is not allowed), and latency-critical loops that must never hit a
// cudaMalloc/cudaFree, which can synchronise the device. This entry point
// takes the same inputs and outputs as gdp_chunk_fwd but uses
// `g_noalloc_scratch` below instead of a caller workspace, and never calls
// cudaMalloc, cudaFree or any other allocating routine.
//
// The array lives for the lifetime of the process on every GPU that loads the
// library (kNoallocScratchBytes of device memory each). All calls share it and
// it keeps the previous call's contents; the status word at its start is
// cleared by every call, and the chunk tables (per-sequence records included,
// which a bad cu_seqlens list sets to zero length) are rewritten before any
// kernel reads them, so nothing a call reads depends on an earlier call.
// Calls that overlap on the GPU (on different streams, or from different host
// threads) race on the array and must be serialised by the caller.
//
// The device address is looked up once per device and kept; a cudaDeviceReset
// between calls would leave it stale (the header says so).
#include <mutex>

#include "gdp_internal.cuh"

namespace gdp {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // 32 MiB

// The scratch array. In host code this name is only a host-side stand-in for
// the device symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current). Returns null on failure.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace
}  // namespace gdp

extern "C" gdp_status gdp_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                            const float* beta, const float* g,
                                            const float* initial_state,
                                            const int32_t* cu_seqlens, int N_seq, int B, int T,
                                            int H, int HV, int K, int V, int M, int chunk_size,
                                            float scale, int use_qk_l2norm, gdp_dtype dt,
                                            float* o, float* final_state, cudaStream_t stream) {
  const size_t need =
      gdp_chunk_fwd_workspace_size(B, T, N_seq, H, HV, K, V, M, chunk_size, dt);
  if (need == 0) {
    // invalid or unsupported sizes: let the regular entry point name the error
    return gdp_chunk_fwd(q, k, v, beta, g, initial_state, cu_seqlens, N_seq, B, T, H, HV, K, V,
                         M, chunk_size, scale, use_qk_l2norm, dt, o, final_state, nullptr, 0,
                         stream);
  }
  if (need > gdp::kNoallocScratchBytes) return GDP_ERR_WORKSPACE;
  void* ws = gdp::scratch_address();
  if (!ws) return GDP_ERR_CUDA;
  return gdp_chunk_fwd(q, k, v, beta, g, initial_state, cu_seqlens, N_seq, B, T, H, HV, K, V, M,
                       chunk_size, scale, use_qk_l2norm, dt, o, final_state, ws,
                       gdp::kNoallocScratchBytes, stream);
}
