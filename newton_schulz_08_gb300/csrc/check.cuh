// Device-side checks of the debug build (compiled with -DMUON_DEBUG): a
// failed check adds one to this translation unit's failure counter and the
// guarded access is skipped; nothing traps.  In the release build
// MUON_CHECK(cond) is the constant true and `cond` is not evaluated.
//
// Each translation unit has its own counter (the library is built without
// relocatable device code); muon_debug_check_failures (muon_capi.cu) reads
// and clears all of them through the per-unit host functions declared here.
#pragma once

#include <cuda_runtime.h>

#ifdef MUON_DEBUG
namespace muon {
namespace {
__device__ int g_check_failures;
}  // namespace
}  // namespace muon
#define MUON_CHECK(cond) ((cond) ? true : (atomicAdd(&::muon::g_check_failures, 1), false))
// Reads (and clears) this unit's counter; defined once per unit by
// MUON_CHECK_READER(name).
#define MUON_CHECK_READER(name)                                                              \
  cudaError_t name(int* out) {                                                               \
    int v = 0;                                                                               \
    cudaError_t e = cudaMemcpyFromSymbol(&v, ::muon::g_check_failures, sizeof(int));         \
    if (e != cudaSuccess) return e;                                                          \
    const int zero = 0;                                                                      \
    e = cudaMemcpyToSymbol(::muon::g_check_failures, &zero, sizeof(int));                    \
    *out = v;                                                                                \
    return e;                                                                                \
  }
#else
#define MUON_CHECK(cond) true
#define MUON_CHECK_READER(name) \
  cudaError_t name(int* out) {  \
    *out = 0;                   \
    return cudaSuccess;         \
  }
#endif

namespace muon {
cudaError_t check_failures_elementwise(int* out);
cudaError_t check_failures_gemm(int* out);
cudaError_t check_failures_fp8(int* out);
cudaError_t check_failures_adam(int* out);
}  // namespace muon
