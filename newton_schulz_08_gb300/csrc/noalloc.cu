// ns5_noalloc: the batched Newton-Schulz call for callers that cannot hand
// the library a workspace.
//
// Some callers are not allowed to allocate device memory: code hosted by a
// framework whose allocator owns the whole GPU and forbids side allocations,
// or code on a latency-critical path where cudaMalloc / cudaFree may
// synchronise the device.  This entry point runs exactly the pipeline of
// ns5() but takes its scratch (partial norms, per-matrix table, the two X
// buffers, A and B) from one file-scope device array of fixed size instead of
// a caller-provided workspace.  It never calls cudaMalloc, cudaFree or any
// allocating routine.
//
// The array lives in device memory of every GPU on which this library's
// device code is loaded, until the process exits.  Its address is looked up
// once per device (cudaGetSymbolAddress, with that device current) on the
// first call made on that device.  All calls share the array and it keeps
// the previous call's contents; the pipeline clears the one thing that must
// start at zero (the status word) and overwrites everything else it reads
// before reading it.  Calls that may overlap on the GPU race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/muon.h"

namespace {

constexpr size_t kScratchBytes = MUON_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).  In host code the array's name is only a
// stand-in, so the address must come from the runtime.
muon_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MUON_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MUON_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MUON_OK;
}

}  // namespace

extern "C" muon_status_t ns5_noalloc(const void* G, int g_dtype, void* O, int batch, int64_t rows,
                                     int64_t cols, int ns_steps, void* stream) {
  if (batch == 0) return MUON_OK;
  if (batch < 0) return MUON_ERR_INVALID_ARG;
  const size_t need = ns5_workspace_size(batch, rows, cols);
  if (need == 0) {
    // invalid or oversized shape: ns5 reports which, before touching anything
    return ns5(G, g_dtype, O, batch, rows, cols, ns_steps, nullptr, 0, stream);
  }
  if (need > kScratchBytes) return MUON_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  const muon_status_t s = scratch_address(&ws);
  if (s != MUON_OK) return s;
  return ns5(G, g_dtype, O, batch, rows, cols, ns_steps, ws, kScratchBytes, stream);
}
