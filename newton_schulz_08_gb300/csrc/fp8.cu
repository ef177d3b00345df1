// HBM-bound passes of the FP8 scaled product on sm_103a.
//
// Method: page "深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术"
// (reposource.net), section "自定义FP8矩阵乘法实现": the forward casts the
// input and the weight, divided by their scales, to E4M3
// (x.div(x_s).to(float8_e4m3fn)); its backward (subsection "反向传播优化")
// casts the output gradient, divided by grad_s, to E5M2, and multiplies it
// with transposed copies of the E4M3 operands (w_f8.T.contiguous(),
// x_f8.T.contiguous(), grad_f8.T.contiguous()).  The products run on the
// tensor cores (ns_gemm.cu, mode kFp8); these passes prepare and finish them.
//
//   fp8_quantize   forward operands: q = E4M3(bf16(src / scale)), two tensors
//                  per launch, 4 x 8 elements per thread in flight.
//   fp8_transpose  backward operands, 128 x 128 tiles through shared memory:
//                  the gradient's codes E5M2(bf16(g / grad_s)) row-major and
//                  transposed, and transposed copies of the E4M3 x_f8, w_f8.
//   fp8_reduce     a product whose contraction was split: out = bf16(scale *
//                  (part[0] + part[1] + ...)), in that order.
//
// Every quotient is rounded once to bfloat16, as a bf16 tensor's division
// rounds the exact quotient: bf16(x / s) for a bf16 x and a float s.
#include <cuda_fp8.h>

#include "check.cuh"
#include "plan.h"

namespace muon {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void grid_dep() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

cudaError_t launch_pdl(const void* fn, int blocks, void** args, cudaStream_t stream) {
  if (blocks <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// x / s rounded once to bfloat16 by "round to odd" (Boldo and Melquiond,
// "When double rounding is odd", 2005): the fp32 quotient truncated toward
// zero, with its last bit set when the division is inexact, rounds to
// bfloat16 (16 fewer bits) exactly as the exact quotient would.  The
// remainder x - q s of a faithfully rounded quotient is representable, so
// the fused multiply-add gives it exactly.
__device__ __forceinline__ float div_to_bf16_exact(float x, float s) {
  const float q = __fdiv_rz(x, s);
  const float r = fmaf(-q, s, x);
  uint32_t b = __float_as_uint(q);
  if (r != 0.0f && isfinite(q)) b |= 1u;
  return __bfloat162float(__float2bfloat16_rn(__uint_as_float(b)));
}

// The same value, mostly without a division.  q = x * inv (inv = 1/s
// rounded to float) is within 2^-23 relative of x / s, two float ulps: its
// bfloat16 rounding is that of x / s unless a bfloat16 rounding boundary
// (a float whose low 16 bits are 0x8000) lies within those two ulps.  The
// low 16 bits of q tell: within three ulps of such a boundary (about one
// quotient in 10^4) the exact routine above decides.
__device__ __forceinline__ float div_to_bf16(float x, float s, float inv) {
  const float q = x * inv;
  const uint32_t low = __float_as_uint(q) & 0xFFFFu;
  if (isfinite(q) && low - 0x7FFDu > 6u) return __bfloat162float(__float2bfloat16_rn(q));
  return div_to_bf16_exact(x, s);
}

// E4M3 ("fn", no infinities): round to nearest even; past the rounding range
// of the largest finite value 448 (|v| > 464) the result is NaN, and so are
// infinite and NaN inputs.
__device__ __forceinline__ uint32_t to_e4m3(float v) {
  if (!(fabsf(v) <= 464.0f)) return 0x7Fu;
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// E5M2: round to nearest even; from the midpoint between the largest finite
// value 57344 and 2^16 on (|v| >= 61440, where ties round to the even 2^16)
// the result is an infinity of v's sign; NaN stays NaN.
__device__ __forceinline__ uint32_t to_e5m2(float v) {
  const float a = fabsf(v);
  if (a < 61440.0f) return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E5M2));
  if (a != a) return 0x7Fu;
  return signbit(v) ? 0xFCu : 0x7Cu;
}

__device__ __forceinline__ float word_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float word_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two codes (a in the low byte), range-checked: past the finite range the
// single conversions give NaN or infinity.
template <bool E5M2>
__device__ __forceinline__ uint32_t to_fp8x2(float a, float b) {
  if (E5M2) {
    if (fabsf(a) < 61440.0f && fabsf(b) < 61440.0f)
      return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E5M2));
    return to_e5m2(a) | (to_e5m2(b) << 8);
  }
  if (fabsf(a) <= 464.0f && fabsf(b) <= 464.0f)
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
  return to_e4m3(a) | (to_e4m3(b) << 8);
}

// The codes of the pair (x0, x1): code(bf16(x / s)).  Fast path, taken
// when both quotients are well inside the code's finite range (|q| below
// 61000 for E5M2, 460 for E4M3: their bf16 roundings then stay below the
// overflow thresholds 61440 and 464, and the range test also rules out
// infinities and NaN) and away from a bf16 rounding boundary (div_to_bf16):
// one paired bf16 rounding and one paired code conversion.  Otherwise
// each quotient is rounded exactly and range-checked on its own.
template <bool E5M2>
__device__ __forceinline__ uint32_t quantise_pair(float x0, float x1, float s, float inv) {
  constexpr float kLim = E5M2 ? 61000.0f : 460.0f;
  const float q0 = x0 * inv, q1 = x1 * inv;
  const uint32_t l0 = __float_as_uint(q0) & 0xFFFFu, l1 = __float_as_uint(q1) & 0xFFFFu;
  if (fabsf(q0) < kLim && fabsf(q1) < kLim && l0 - 0x7FFDu > 6u && l1 - 0x7FFDu > 6u) {
    const float2 v = __bfloat1622float2(__floats2bfloat162_rn(q0, q1));
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, E5M2 ? __NV_E5M2 : __NV_E4M3));
  }
  return to_fp8x2<E5M2>(div_to_bf16(x0, s, inv), div_to_bf16(x1, s, inv));
}

// Four bf16 pairs (one 16-byte vector) to 8 one-byte codes (two words).
template <bool E5M2>
__device__ __forceinline__ uint2 quantise8(uint4 w, float s, float inv) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int k = 0; k < 4; ++k)
    out[k >> 1] |= quantise_pair<E5M2>(word_lo(ws[k]), word_hi(ws[k]), s, inv) << (16 * (k & 1));
  return make_uint2(out[0], out[1]);
}

}  // namespace

// ---------------------------------------------------------------- forward
// six blocks per SM (40 registers): 36.8 against 38.9 us at 65536 x 768 with five
__global__ void __launch_bounds__(kThreads, 6) fp8_quantize_kernel(const __grid_constant__ Fp8QuantParams P) {
  grid_dep();
  const int t = static_cast<long long>(blockIdx.x) >= P.blocks0 ? 1 : 0;
  const long long b = static_cast<long long>(blockIdx.x) - (t ? P.blocks0 : 0);
  const long long n = P.n[t];
  const float s = P.scale[t], inv = P.inv_scale[t];
  const __nv_bfloat16* src = P.src[t];
  uint8_t* dst = P.dst[t];
  const long long base = b * kQuantPerBlock;
  uint4 w[kQuantVecs];
  long long i0[kQuantVecs];
#pragma unroll
  for (int h = 0; h < kQuantVecs; ++h) {
    i0[h] = base + (static_cast<long long>(h) * kThreads + threadIdx.x) * 8;
    // src 16-byte aligned: a whole vector is in range or the tail handles it
    if (i0[h] + 8 <= n) w[h] = *reinterpret_cast<const uint4*>(src + i0[h]);
  }
#pragma unroll
  for (int h = 0; h < kQuantVecs; ++h) {
    if (i0[h] + 8 <= n) {
      *reinterpret_cast<uint2*>(dst + i0[h]) = quantise8<false>(w[h], s, inv);
    } else {
      for (long long i = i0[h]; i < n; ++i) dst[i] = static_cast<uint8_t>(to_e4m3(div_to_bf16_exact(__bfloat162float(src[i]), s)));
    }
  }
}

cudaError_t launch_fp8_quantize(const Fp8QuantParams& P, int blocks, cudaStream_t stream) {
  void* args[] = {const_cast<Fp8QuantParams*>(&P)};
  return launch_pdl(reinterpret_cast<const void*>(&fp8_quantize_kernel), blocks, args, stream);
}

// --------------------------------------------------------------- backward
// One 128 x 128 tile of a job per block.  Load: 4 passes of 32 rows, 8
// threads per row, 16 columns (32 bytes of bf16 or 16 codes) each; a
// quantising job also writes its 16 codes row-major.  The codes go to a
// shared tile of 128-byte rows whose 4-byte words are swizzled: word w of
// row r sits at w ^ (4 * ((r / 16) % 8)).  Then each thread reads a
// 16-row x 4-column block as 16 words, transposes it as four 4 x 4 byte
// blocks and writes 16 bytes to each of 4 rows of the transposed output.
// In a warp the 4 lanes of a group take 4 adjacent word columns and the 8
// groups the 8 row blocks: the swizzle puts the 32 words of one read in 32
// different banks, and each store writes 4 whole 128-byte output rows.
// five blocks per SM (48 registers, a few spilled): more tiles' loads in flight;
// 189.5 against 204.3 us at 65536 x 3072 with four (six: no faster)
__global__ void __launch_bounds__(kThreads, 5) fp8_transpose_kernel(const __grid_constant__ Fp8TParams P) {
  grid_dep();
  __shared__ __align__(16) uint32_t tile[kFp8Tile * kFp8Tile / 4];
  int j = 0;
  while (j + 1 < P.n_jobs && static_cast<int>(blockIdx.x) >= P.job[j + 1].tile_begin) ++j;
  const Fp8TJob& J = P.job[j];
  const int t = static_cast<int>(blockIdx.x) - J.tile_begin;
  const int r0 = (t / J.tiles_c) * kFp8Tile, c0 = (t % J.tiles_c) * kFp8Tile;
  const int tid = threadIdx.x;
  const int cl = (tid & 7) * 16;  // tile columns cl .. cl + 15
  auto slot = [](int r, int w) { return r * (kFp8Tile / 4) + (w ^ (((r >> 4) & 7) << 2)); };
  // rows and columns are multiples of 16: a 16-element piece is wholly
  // inside the source or wholly outside
  if (J.quant) {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(J.src);
    uint4 v[4][2];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int r = r0 + p * 32 + (tid >> 3), c = c0 + cl;
      if (r < J.rows && c < J.cols) {
        const uint4* q = reinterpret_cast<const uint4*>(src + static_cast<long long>(r) * J.cols + c);
        v[p][0] = q[0];
        v[p][1] = q[1];
      }
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int rl = p * 32 + (tid >> 3);
      const int r = r0 + rl, c = c0 + cl;
      uint2 a = make_uint2(0u, 0u), b = make_uint2(0u, 0u);
      if (r < J.rows && c < J.cols) {
        a = quantise8<true>(v[p][0], J.scale, J.inv_scale);
        b = quantise8<true>(v[p][1], J.scale, J.inv_scale);
        if (MUON_CHECK(c + 16 <= J.cols && (c & 15) == 0))
          *reinterpret_cast<uint4*>(J.dst + static_cast<long long>(r) * J.cols + c) = make_uint4(a.x, a.y, b.x, b.y);
      }
      *reinterpret_cast<uint4*>(&tile[slot(rl, cl >> 2)]) = make_uint4(a.x, a.y, b.x, b.y);
    }
  } else {
    const uint8_t* src = static_cast<const uint8_t*>(J.src);
    uint4 v[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int r = r0 + p * 32 + (tid >> 3), c = c0 + cl;
      v[p] = make_uint4(0u, 0u, 0u, 0u);
      if (r < J.rows && c < J.cols) v[p] = *reinterpret_cast<const uint4*>(src + static_cast<long long>(r) * J.cols + c);
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) *reinterpret_cast<uint4*>(&tile[slot(p * 32 + (tid >> 3), cl >> 2)]) = v[p];
  }
  __syncthreads();
  // transposed: output rows c0 + 4 wc .. + 3 (source columns), source rows
  // r0 + rb .. + 15 as 16 bytes of each
  const int lane = tid & 31;
  const int wc = (tid >> 5) * 4 + (lane & 3);
  const int rb = (lane >> 2) * 16;
  uint32_t o[4][4];  // [output row][word]
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t a[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) a[m] = tile[slot(rb + 4 * k + m, wc)];
    // a[m] byte i = tile[rb + 4k + m][4 wc + i]; output row i, word k, byte m
    const uint32_t t0 = __byte_perm(a[0], a[1], 0x5140), t1 = __byte_perm(a[2], a[3], 0x5140);
    const uint32_t t2 = __byte_perm(a[0], a[1], 0x7362), t3 = __byte_perm(a[2], a[3], 0x7362);
    o[0][k] = __byte_perm(t0, t1, 0x5410);
    o[1][k] = __byte_perm(t0, t1, 0x7632);
    o[2][k] = __byte_perm(t2, t3, 0x5410);
    o[3][k] = __byte_perm(t2, t3, 0x7632);
  }
  const int rr = r0 + rb;
  if (rr < J.rows) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = c0 + 4 * wc + i;
      if (c < J.cols && MUON_CHECK(rr + 16 <= J.rows && (rr & 15) == 0))
        *reinterpret_cast<uint4*>(J.dst_t + static_cast<long long>(c) * J.rows + rr) =
            make_uint4(o[i][0], o[i][1], o[i][2], o[i][3]);
    }
  }
}

cudaError_t launch_fp8_transpose(const Fp8TParams& P, int blocks, cudaStream_t stream) {
  void* args[] = {const_cast<Fp8TParams*>(&P)};
  return launch_pdl(reinterpret_cast<const void*>(&fp8_transpose_kernel), blocks, args, stream);
}

// out = bf16(scale * (part[0] + part[1] + ...)), 4 elements per thread.
__global__ void __launch_bounds__(kThreads) fp8_reduce_kernel(const __grid_constant__ Fp8ReduceParams P) {
  grid_dep();
  const long long i = (static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x) * 4;
  if (i >= P.n) return;
  if (!MUON_CHECK(i + 4 <= P.n)) return;
  float4 acc = *reinterpret_cast<const float4*>(P.part + i);
  for (int s = 1; s < P.splits; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(P.part + static_cast<long long>(s) * P.n + i);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(P.scale * acc.x, P.scale * acc.y);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(P.scale * acc.z, P.scale * acc.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&lo);
  w.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(P.out + i) = w;
}

cudaError_t launch_fp8_reduce(const Fp8ReduceParams& P, int blocks, cudaStream_t stream) {
  void* args[] = {const_cast<Fp8ReduceParams*>(&P)};
  return launch_pdl(reinterpret_cast<const void*>(&fp8_reduce_kernel), blocks, args, stream);
}

MUON_CHECK_READER(check_failures_fp8)

}  // namespace muon
