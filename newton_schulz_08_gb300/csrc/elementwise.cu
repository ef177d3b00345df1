// HBM-bound passes of the Muon step on sm_103a.
//
// Method: page "深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术"
// (reposource.net), section "Muon优化器：动量正交化技术" (step 1: the
// standard momentum update) and section "Newton-Schulz正交化" (X =
// G.bfloat16()).  Readings of what the page leaves out: Nesterov momentum
// buf <- mu*buf + g, u <- g + mu*buf (updated buf); tall matrices (more rows
// than columns) are transposed; X is divided by (||X||_F + 1e-7) before the
// iteration, the norm taken of the bfloat16-rounded X and the quotient
// rounded to bfloat16.
//
// momentum_cast: one pass over (g, buf): buf <- mu*buf + g (in place),
//   u = g + mu*buf, Xraw = bf16(u) written to the workspace (transposed for
//   tall matrices through a shared-memory tile), and one partial sum of
//   Xraw^2 per block (warp shuffles, then a fixed-order block reduction: the
//   result does not depend on scheduling).
// normalise: X0 = bf16(Xraw / (sqrt(sum of the matrix's partials) + 1e-7)),
//   in place; the partials are summed in a fixed order by every block.  With
//   zero Newton-Schulz steps it also applies the update (or writes O).
#include "plan.h"

namespace muon {

namespace {

constexpr int kEwThreads = 256;

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// Sum over the block in a fixed order; valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.0f;
  if (threadIdx.x == 0)
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
  return s;
}

__device__ __forceinline__ float load_g(const void* g, int f32, long long i) {
  return f32 ? static_cast<const float*>(g)[i]
             : __bfloat162float(static_cast<const __nv_bfloat16*>(g)[i]);
}

// u from g and buf; updates buf in place when present.
__device__ __forceinline__ float momentum_u(float g, float* buf, long long i, float mu, int nesterov) {
  if (!buf) return g;
  const float b = fmaf(mu, buf[i], g);
  buf[i] = b;
  return nesterov ? fmaf(mu, b, g) : b;
}

}  // namespace

__global__ void __launch_bounds__(kEwThreads) momentum_cast_kernel(const __grid_constant__ K1Params P) {
  __shared__ float red[kEwThreads / 32];
  __shared__ float tile[64][65];
  // which matrix: largest i with block_begin[i] <= blockIdx.x
  int lo = 0, hi = P.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.block_begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
  }
  const K1Mat& M = P.mats[lo];
  const int b = blockIdx.x - P.block_begin[lo];
  const int R = M.R, C = M.C;
  float ss = 0.0f;

  if (b == 0 && threadIdx.x == 0) {
    MatInfo mi;
    mi.out = M.out;
    mi.R = R;
    mi.C = C;
    mi.tall = M.tall;
    mi.part_off = M.part_off;
    mi.nparts = M.nparts;
    mi.pad = 0;
    P.table[M.table_index] = mi;
  }

  if (!M.tall) {
    // X = u, same layout: rows [r0, r1) of the matrix
    const int r0 = b * M.rows_per_block;
    const int r1 = min(R, r0 + M.rows_per_block);
    const bool vec = (C & 7) == 0;
    if (vec) {
      const int cv = C >> 3;  // 8-element vectors per row
      const long long nvec = static_cast<long long>(r1 - r0) * cv;
      for (long long v = threadIdx.x; v < nvec; v += kEwThreads) {
        const int r = r0 + static_cast<int>(v / cv);
        const int c = static_cast<int>(v % cv) * 8;
        const long long i = static_cast<long long>(r) * C + c;
        float g[8];
        if (M.g_f32) {
          const float4* gp = reinterpret_cast<const float4*>(static_cast<const float*>(M.g) + i);
          const float4 a = gp[0], bq = gp[1];
          g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
          g[4] = bq.x; g[5] = bq.y; g[6] = bq.z; g[7] = bq.w;
        } else {
          const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(M.g) + i);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            g[2 * k] = __uint_as_float(ws[k] << 16);
            g[2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
          }
        }
        float u[8];
        if (M.buf) {
          float4* bp = reinterpret_cast<float4*>(M.buf + i);
          float4 b0 = bp[0], b1 = bp[1];
          float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            bv[k] = fmaf(P.mu, bv[k], g[k]);
            u[k] = P.nesterov ? fmaf(P.mu, bv[k], g[k]) : bv[k];
          }
          bp[0] = make_float4(bv[0], bv[1], bv[2], bv[3]);
          bp[1] = make_float4(bv[4], bv[5], bv[6], bv[7]);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) u[k] = g[k];
        }
        uint32_t packed[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(u[2 * k], u[2 * k + 1]);
          packed[k] = *reinterpret_cast<const uint32_t*>(&h);
          const float x0 = __low2float(h), x1 = __high2float(h);
          ss = fmaf(x0, x0, ss);
          ss = fmaf(x1, x1, ss);
        }
        *reinterpret_cast<uint4*>(M.x + static_cast<long long>(r) * M.ldx + c) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
    } else {
      const long long ne = static_cast<long long>(r1 - r0) * C;
      for (long long e = threadIdx.x; e < ne; e += kEwThreads) {
        const int r = r0 + static_cast<int>(e / C);
        const int c = static_cast<int>(e % C);
        const long long i = static_cast<long long>(r) * C + c;
        const float u = momentum_u(load_g(M.g, M.g_f32, i), M.buf, i, P.mu, P.nesterov);
        const float x = bf16_round(u);
        ss = fmaf(x, x, ss);
        M.x[static_cast<long long>(r) * M.ldx + c] = __float2bfloat16_rn(u);
      }
    }
  } else {
    // tall: X = u^T (C x R).  64 rows of u per block, 64 x 64 tiles through
    // shared memory so that both the reads of u and the writes of X are
    // contiguous across a warp.
    const int r0 = b * 64;
    for (int c0 = 0; c0 < C; c0 += 64) {
      for (int e = threadIdx.x; e < 64 * 64; e += kEwThreads) {
        const int rr = e >> 6, cc = e & 63;
        const int r = r0 + rr, c = c0 + cc;
        float x = 0.0f;
        if (r < R && c < C) {
          const long long i = static_cast<long long>(r) * C + c;
          const float u = momentum_u(load_g(M.g, M.g_f32, i), M.buf, i, P.mu, P.nesterov);
          x = bf16_round(u);
          ss = fmaf(x, x, ss);
        }
        tile[rr][cc] = x;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < 64 * 64; e += kEwThreads) {
        const int cc = e >> 6, rr = e & 63;  // X row = c, X column = r
        const int r = r0 + rr, c = c0 + cc;
        if (r < R && c < C) M.x[static_cast<long long>(c) * M.ldx + r] = __float2bfloat16_rn(tile[rr][cc]);
      }
      __syncthreads();
    }
  }

  const float s = block_sum(ss, red);
  if (threadIdx.x == 0) P.partials[M.part_off + b] = s;
}

__global__ void __launch_bounds__(kEwThreads) normalise_kernel(const __grid_constant__ NormParams P) {
  __shared__ float red[kEwThreads / 32];
  __shared__ float sh_d;
  int c = 0;
  while (c + 1 < P.n_classes && (int)blockIdx.x >= P.cls[c + 1].block_begin) ++c;
  const NormClass& K = P.cls[c];
  const int local = blockIdx.x - K.block_begin;
  const int idx = local / K.blocks_per_mat;
  const int b = local - idx * K.blocks_per_mat;
  const MatInfo mi = P.table[K.mat_begin + idx];

  // the matrix's norm: fixed-order sum of its partials
  float part = 0.0f;
  for (int i = threadIdx.x; i < mi.nparts; i += kEwThreads) part += P.partials[mi.part_off + i];
  const float ss = block_sum(part, red);
  if (threadIdx.x == 0) {
    const float d = sqrtf(ss) + 1e-7f;
    sh_d = d;
    if (b == 0 && !isfinite(d)) atomicOr(P.status, kStatusNonFinite);
  }
  __syncthreads();
  const float d = sh_d;

  __nv_bfloat16* X = K.x + static_cast<long long>(idx) * K.m * K.ldx;
  const int r0 = b * K.rows_per_block;
  const int r1 = min(K.m, r0 + K.rows_per_block);
  const int n = K.n;
  if (P.final_mode == kFinalNone && (n & 7) == 0) {
    const int cv = n >> 3;
    const long long nvec = static_cast<long long>(r1 - r0) * cv;
    for (long long v = threadIdx.x; v < nvec; v += kEwThreads) {
      const int r = r0 + static_cast<int>(v / cv);
      const int cc = static_cast<int>(v % cv) * 8;
      uint4* p = reinterpret_cast<uint4*>(X + static_cast<long long>(r) * K.ldx + cc);
      uint4 w = *p;
      uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = __uint_as_float(ws[k] << 16) / d;
        const float hi = __uint_as_float(ws[k] & 0xFFFF0000u) / d;
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        ws[k] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *p = make_uint4(ws[0], ws[1], ws[2], ws[3]);
    }
  } else {
    const long long ne = static_cast<long long>(r1 - r0) * n;
    for (long long e = threadIdx.x; e < ne; e += kEwThreads) {
      const int r = r0 + static_cast<int>(e / n);
      const int cc = static_cast<int>(e % n);
      __nv_bfloat16* p = X + static_cast<long long>(r) * K.ldx + cc;
      const __nv_bfloat16 x0 = __float2bfloat16_rn(__bfloat162float(*p) / d);
      *p = x0;
      if (P.final_mode != kFinalNone) {
        // X is m x n; the matrix as stored is X (wide) or X^T (tall)
        const long long o = mi.tall ? static_cast<long long>(cc) * K.m + r : static_cast<long long>(r) * n + cc;
        if (P.final_mode == kFinalParam) {
          float* pp = static_cast<float*>(mi.out) + o;
          *pp = fmaf(-P.lr, __bfloat162float(x0), *pp);
        } else {
          static_cast<__nv_bfloat16*>(mi.out)[o] = x0;
        }
      }
    }
  }
}

cudaError_t launch_momentum_cast(const K1Params& P, int blocks, cudaStream_t stream) {
  if (blocks <= 0) return cudaSuccess;
  void* args[] = {const_cast<K1Params*>(&P)};
  return cudaLaunchKernel(reinterpret_cast<const void*>(&momentum_cast_kernel), dim3(blocks),
                          dim3(kEwThreads), args, 0, stream);
}

cudaError_t launch_normalise(const NormParams& P, int blocks, cudaStream_t stream) {
  if (blocks <= 0) return cudaSuccess;
  void* args[] = {const_cast<NormParams*>(&P)};
  return cudaLaunchKernel(reinterpret_cast<const void*>(&normalise_kernel), dim3(blocks),
                          dim3(kEwThreads), args, 0, stream);
}

}  // namespace muon
