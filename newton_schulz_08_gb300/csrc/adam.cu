// Adam step with cautious weight decay for a list of tensors (the
// embedding-type parameters that the Muon step does not cover), in one
// launch per 64 tensors.
//
// Method: the page on the modded-nanogpt record "2026-06-11_RecursiveFromBest"
// (lqnn.cn, news/184262), section "3.3 bigram 与 value-embedding 银行上的
// C-Optim / 谨慎 Adam": Adam on the bigram and value-embedding banks, the
// weight decay applied only where the update and the parameter agree in sign
// (a mask that is true where update * p is positive).  Adam itself is the
// textbook algorithm (bias-corrected moment estimates); the decay is
// decoupled: p <- p - lr * (u + wd * p * mask).
//
// Per element, in float32, each operation one IEEE operation in this order
// (no fused multiply-add, so results do not depend on compiler contraction):
//   m1 = b1*m + (1-b1)*g;  v1 = b2*v + (1-b2)*(g*g)
//   u  = (m1 / bc1) / (sqrt(v1 / bc2) + eps)
//   d  = mask ? wd*p : 0,  mask = (u > 0 && p > 0) || (u < 0 && p < 0)
//        (always wd*p when not cautious)
//   p1 = p - lr*(u + d)
// with (1-b1), (1-b2), bc1 = 1 - b1^t, bc2 = 1 - b2^t formed in double on the
// host and rounded once to float.
//
// HBM-bound: 26 bytes per element with bfloat16 gradients (p, m, v read and
// written, g read).  Blocks of 8192 elements of one tensor; each thread has
// two 4-element vectors of p, m, v and g in flight, loads issued before any
// store; ragged tails take a scalar path.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/muon.h"
#include "check.cuh"

namespace muon {

namespace {

constexpr int kAdamThreads = 256;
constexpr int kAdamVec = 4;                                      // elements per vector
constexpr int kAdamBlockElems = kAdamThreads * kAdamVec * 2 * 4;  // 8192
constexpr int kAdamMaxTensors = 64;                              // per launch

struct AdamTensor {
  float* p;
  const void* g;
  float* m;
  float* v;
  long long numel;
  int g_f32;
  int pad;
};

struct AdamParams {
  AdamTensor t[kAdamMaxTensors];
  int block_begin[kAdamMaxTensors + 1];
  int n;
  float b1, b2, omb1, omb2, bc1, bc2, lr, eps, wd;
  int cautious;
};

__device__ __forceinline__ void adam_elem(float& p, float g, float& m, float& v, const AdamParams& k) {
  const float m1 = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.omb1, g));
  const float v1 = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.omb2, __fmul_rn(g, g)));
  const float u = __fdiv_rn(__fdiv_rn(m1, k.bc1), __fadd_rn(__fsqrt_rn(__fdiv_rn(v1, k.bc2)), k.eps));
  const bool mask = !k.cautious || (u > 0.0f && p > 0.0f) || (u < 0.0f && p < 0.0f);
  const float d = mask ? __fmul_rn(k.wd, p) : 0.0f;
  p = __fsub_rn(p, __fmul_rn(k.lr, __fadd_rn(u, d)));
  m = m1;
  v = v1;
}

__device__ __forceinline__ float load_grad(const void* g, int f32, long long i) {
  return f32 ? static_cast<const float*>(g)[i] : __bfloat162float(static_cast<const __nv_bfloat16*>(g)[i]);
}

__global__ void __launch_bounds__(kAdamThreads) adam_kernel(const __grid_constant__ AdamParams P) {
  // which tensor: largest i with block_begin[i] <= blockIdx.x
  int lo = 0, hi = P.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.block_begin[mid] <= static_cast<int>(blockIdx.x)) lo = mid; else hi = mid - 1;
  }
  const AdamTensor& T = P.t[lo];
  const long long e0 = static_cast<long long>(blockIdx.x - P.block_begin[lo]) * kAdamBlockElems;
  const long long e1 = min(T.numel, e0 + kAdamBlockElems);
  // debug build: the block starts inside its tensor
  if (!MUON_CHECK(e0 >= 0 && e0 < T.numel)) return;
  // whole vectors of this block; the tensor's last partial vector is done
  // element by element
  const long long nvec = (e1 - e0) / kAdamVec;
  for (long long v0 = threadIdx.x; v0 < nvec; v0 += 2 * kAdamThreads) {
    float4 pp[2], mm[2], vv[2];
    float gg[2][4];
    bool have[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const long long vi = v0 + h * kAdamThreads;
      have[h] = vi < nvec;
      if (!have[h]) continue;
      const long long i = e0 + vi * kAdamVec;
      pp[h] = *reinterpret_cast<const float4*>(T.p + i);
      mm[h] = *reinterpret_cast<const float4*>(T.m + i);
      vv[h] = *reinterpret_cast<const float4*>(T.v + i);
      if (T.g_f32) {
        const float4 q = *reinterpret_cast<const float4*>(static_cast<const float*>(T.g) + i);
        gg[h][0] = q.x; gg[h][1] = q.y; gg[h][2] = q.z; gg[h][3] = q.w;
      } else {
        const uint2 q = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(T.g) + i);
        gg[h][0] = __uint_as_float(q.x << 16);
        gg[h][1] = __uint_as_float(q.x & 0xFFFF0000u);
        gg[h][2] = __uint_as_float(q.y << 16);
        gg[h][3] = __uint_as_float(q.y & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!have[h]) continue;
      const long long i = e0 + (v0 + h * kAdamThreads) * kAdamVec;
      adam_elem(pp[h].x, gg[h][0], mm[h].x, vv[h].x, P);
      adam_elem(pp[h].y, gg[h][1], mm[h].y, vv[h].y, P);
      adam_elem(pp[h].z, gg[h][2], mm[h].z, vv[h].z, P);
      adam_elem(pp[h].w, gg[h][3], mm[h].w, vv[h].w, P);
      *reinterpret_cast<float4*>(T.p + i) = pp[h];
      *reinterpret_cast<float4*>(T.m + i) = mm[h];
      *reinterpret_cast<float4*>(T.v + i) = vv[h];
    }
  }
  for (long long i = e0 + nvec * kAdamVec + threadIdx.x; i < e1; i += kAdamThreads) {
    float p = T.p[i], m = T.m[i], v = T.v[i];
    adam_elem(p, load_grad(T.g, T.g_f32, i), m, v, P);
    T.p[i] = p;
    T.m[i] = m;
    T.v[i] = v;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  uintptr_t lo, hi;
};

bool overlap(const Span& a, const Span& b) { return a.lo < b.hi && b.lo < a.hi; }

}  // namespace

}  // namespace muon

namespace muon {
MUON_CHECK_READER(check_failures_adam)
}  // namespace muon

extern "C" muon_status_t adam_step(const adam_tensor_desc* tensors, int n_tensors, float lr, float beta1,
                                   float beta2, float eps, float weight_decay, int step, int cautious,
                                   void* stream) {
  using namespace muon;
  if (n_tensors < 0 || (n_tensors > 0 && !tensors)) return MUON_ERR_INVALID_ARG;
  if (step < 1) return MUON_ERR_INVALID_ARG;
  if (!(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f)) return MUON_ERR_INVALID_ARG;
  if (!std::isfinite(lr) || !std::isfinite(weight_decay) || !(eps >= 0.0f) || !std::isfinite(eps))
    return MUON_ERR_INVALID_ARG;
  std::vector<Span> written, read;
  for (int i = 0; i < n_tensors; ++i) {
    const adam_tensor_desc& d = tensors[i];
    if (!d.param || !d.grad || !d.exp_avg || !d.exp_avg_sq || d.numel <= 0) return MUON_ERR_INVALID_ARG;
    if (d.grad_dtype != MUON_BF16 && d.grad_dtype != MUON_F32) return MUON_ERR_INVALID_ARG;
    if (d.numel > (1LL << 40)) return MUON_ERR_TOO_LARGE;
    if (!aligned16(d.param) || !aligned16(d.grad) || !aligned16(d.exp_avg) || !aligned16(d.exp_avg_sq))
      return MUON_ERR_MISALIGNED;
    const uintptr_t n4 = static_cast<uintptr_t>(d.numel) * 4;
    const uintptr_t ng = static_cast<uintptr_t>(d.numel) * (d.grad_dtype == MUON_F32 ? 4 : 2);
    written.push_back({reinterpret_cast<uintptr_t>(d.param), reinterpret_cast<uintptr_t>(d.param) + n4});
    written.push_back({reinterpret_cast<uintptr_t>(d.exp_avg), reinterpret_cast<uintptr_t>(d.exp_avg) + n4});
    written.push_back(
        {reinterpret_cast<uintptr_t>(d.exp_avg_sq), reinterpret_cast<uintptr_t>(d.exp_avg_sq) + n4});
    read.push_back({reinterpret_cast<uintptr_t>(d.grad), reinterpret_cast<uintptr_t>(d.grad) + ng});
  }
  // grid of each launch (kAdamMaxTensors tensors) within range
  for (int t0 = 0; t0 < n_tensors; t0 += kAdamMaxTensors) {
    long long blocks = 0;
    for (int j = t0; j < n_tensors && j < t0 + kAdamMaxTensors; ++j)
      blocks += (tensors[j].numel + kAdamBlockElems - 1) / kAdamBlockElems;
    if (blocks > 0x7FFFFFFFLL) return MUON_ERR_TOO_LARGE;
  }
  // written ranges overlap neither each other nor any gradient
  for (size_t a = 0; a < written.size(); ++a) {
    for (size_t b = a + 1; b < written.size(); ++b)
      if (overlap(written[a], written[b])) return MUON_ERR_ALIASING;
    for (const Span& r : read)
      if (overlap(written[a], r)) return MUON_ERR_ALIASING;
  }
  if (n_tensors == 0) return MUON_OK;

  AdamParams P;
  P.b1 = beta1;
  P.b2 = beta2;
  P.omb1 = static_cast<float>(1.0 - static_cast<double>(beta1));
  P.omb2 = static_cast<float>(1.0 - static_cast<double>(beta2));
  P.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta1), step));
  P.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta2), step));
  P.lr = lr;
  P.eps = eps;
  P.wd = weight_decay;
  P.cautious = cautious ? 1 : 0;
  if (!(P.bc1 > 0.0f) || !(P.bc2 > 0.0f)) return MUON_ERR_INVALID_ARG;  // beta^t rounds to 1
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int t0 = 0; t0 < n_tensors; t0 += kAdamMaxTensors) {
    const int n = n_tensors - t0 < kAdamMaxTensors ? n_tensors - t0 : kAdamMaxTensors;
    long long blocks = 0;
    for (int j = 0; j < n; ++j) {
      const adam_tensor_desc& d = tensors[t0 + j];
      P.t[j] = {d.param, d.grad, d.exp_avg, d.exp_avg_sq, static_cast<long long>(d.numel),
                d.grad_dtype == MUON_F32 ? 1 : 0, 0};
      P.block_begin[j] = static_cast<int>(blocks);
      blocks += (d.numel + kAdamBlockElems - 1) / kAdamBlockElems;
    }
    P.block_begin[n] = static_cast<int>(blocks);
    P.n = n;
    adam_kernel<<<static_cast<unsigned>(blocks), kAdamThreads, 0, s>>>(P);
    if (cudaGetLastError() != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}
