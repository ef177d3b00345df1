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
// device code is loaded, until the process exits.  CUDA loads modules
// lazily, so the array is reserved on a device when the first call made
// there looks up its address; callers that budget device memory should make
// one call at initialisation (and before any stream capture).  The address
// is looked up again on every call (cudaGetSymbolAddress, with the caller's
// device current): after cudaDeviceReset, or under another context, the
// module is loaded again and the array may sit elsewhere, so an address kept
// from an earlier call could point at memory the array no longer owns.  The
// lookup allocates nothing once the module is loaded.  All calls share the
// array and it keeps the previous call's contents; the pipeline clears the
// one thing that must start at zero (the status word) and overwrites
// everything else it reads before reading it.  Calls that may overlap on
// the GPU race on the array.
#include <cuda_runtime.h>

#include "../../include/muon.h"

namespace {

constexpr size_t kScratchBytes = MUON_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array in the current context.  In host code
// the array's name is only a stand-in, so the address must come from the
// runtime.  The device is checked first, so that an unsupported GPU gets
// its own status (and loads nothing).
muon_status_t scratch_address(void** out) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return MUON_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return MUON_ERR_UNSUPPORTED_DEVICE;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();  // leave no sticky-looking error behind for the caller
    return MUON_ERR_CUDA;
  }
  *out = p;
  return MUON_OK;
}

}  // namespace

extern "C" muon_status_t ns5_noalloc(const void* G, int g_dtype, void* O, int batch, int64_t rows,
                                     int64_t cols, int ns_steps, void* stream) {
  if (batch == 0) return MUON_OK;
  if (batch < 0 || !G || !O || (g_dtype != MUON_BF16 && g_dtype != MUON_F32)) return MUON_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(G) & 15u) || (reinterpret_cast<uintptr_t>(O) & 15u)) return MUON_ERR_MISALIGNED;
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

// The status word of the last ns5_noalloc call on the current device: the
// first word of the scratch array, read the way muon_device_status reads a
// workspace's (a copy into a host variable, then the stream is waited for).
extern "C" muon_status_t ns5_noalloc_status(void* stream) {
  void* ws = nullptr;
  const muon_status_t s = scratch_address(&ws);
  if (s != MUON_OK) return s;
  return muon_device_status(ws, stream);
}
