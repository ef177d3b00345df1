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
// normalise: X0 = bf16(Xraw * (1 / (sqrt(sum of the matrix's partials) +
//   1e-7))), in place; the partials are summed in a fixed order by every
//   block.
// apply: after the last step, O = X in the stored orientation written
//   (Newton-Schulz alone), or p <- p - lr * O for a Muon step with no
//   iteration (otherwise the last update applies it).
#include "check.cuh"
#include "plan.h"

namespace muon {

namespace {

constexpr int kEwThreads = 256;
constexpr int kNormBatch = 8;  // normalise: 8-element vectors per thread in flight (four blocks per SM)
constexpr int kCastBatch = 8;  // cast-only momentum pass: 8-element vectors per thread in flight
constexpr int kMomBatch = 2;   // momentum pass with bf16 G: 8-element vectors per thread in flight
// Tall momentum pass: the 64 x 64 fp32 shared tile has rows of 66 floats and
// column c of row r stored at c ^ (8 * ((r / 16) % 4)).  A warp's writes (two
// rows, four consecutive columns per lane, the upper half-warp's in rotated
// order) and its reads (column cc of rows rb + 2j, rb a multiple of 16) then
// fall in 32 different banks.
constexpr int kTallPitch = 66;
__device__ __forceinline__ int tall_col(int r, int c) { return c ^ (((r >> 4) & 3) << 3); }

// Programmatic dependent launch: wait for the previous grid's results, then
// let the next grid be scheduled.
__device__ __forceinline__ void ptx_grid_dep_wait() {
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
  cfg.blockDim = dim3(kEwThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

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

__global__ void __launch_bounds__(kEwThreads, 4) momentum_cast_kernel(const __grid_constant__ K1Params P) {
  ptx_grid_dep_wait();
  __shared__ float red[kEwThreads / 32];
  __shared__ float tile[2][64][kTallPitch];
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
  // debug build: the block lies inside its matrix's partial sums
  if (!MUON_CHECK(b >= 0 && b < M.nparts && M.rows_per_block > 0)) return;

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
    if (vec && !M.buf && !M.g_f32) {
      // cast only (bf16 G, no momentum buffer): 2 + 2 bytes per element, so
      // kCastBatch 16-byte vectors per thread are kept in flight
      const int cv = C >> 3;
      const long long nvec = static_cast<long long>(r1 - r0) * cv;
      for (long long v0 = threadIdx.x; v0 < nvec; v0 += kCastBatch * kEwThreads) {
        uint4 w[kCastBatch];
        long long iv[kCastBatch];
#pragma unroll
        for (int h = 0; h < kCastBatch; ++h) {
          const long long v = v0 + h * kEwThreads;
          iv[h] = -1;
          if (v < nvec) {
            const int r = r0 + static_cast<int>(v / cv);
            const int c = static_cast<int>(v % cv) * 8;
            iv[h] = static_cast<long long>(r) * M.ldx + c;
            w[h] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(M.g) +
                                                   static_cast<long long>(r) * C + c);
          }
        }
#pragma unroll
        for (int h = 0; h < kCastBatch; ++h) {
          if (iv[h] < 0) continue;
          const uint32_t ws[4] = {w[h].x, w[h].y, w[h].z, w[h].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float x0 = __uint_as_float(ws[k] << 16), x1 = __uint_as_float(ws[k] & 0xFFFF0000u);
            ss = fmaf(x0, x0, ss);
            ss = fmaf(x1, x1, ss);
          }
          if (MUON_CHECK(iv[h] + 8 <= static_cast<long long>(R) * M.ldx)) *reinterpret_cast<uint4*>(M.x + iv[h]) = w[h];
        }
      }
    } else if (vec && M.buf && !M.g_f32) {
      // momentum and cast, bf16 G: rows [r0, r1) are contiguous in g, buf
      // and X (a wide matrix's X pitch is C when C is a multiple of 8).
      // kMomBatch 8-element vectors per thread, all their loads (16 bytes
      // of g, 32 of buf) issued before any store: 48 bytes per vector
      const long long base = static_cast<long long>(r0) * C;
      const int nvec = (r1 - r0) * (C >> 3);
      const uint4* gv = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(M.g) + base);
      float4* bv4 = reinterpret_cast<float4*>(M.buf + base);
      uint4* xv = reinterpret_cast<uint4*>(M.x + base);
      // debug build: the block's rows lie inside the matrix and X's pitch is C
      if (!MUON_CHECK(M.ldx == C && r1 <= R)) return;
      for (int v0 = threadIdx.x; v0 < nvec; v0 += kMomBatch * kEwThreads) {
        uint4 gw[kMomBatch];
        float4 b0[kMomBatch], b1[kMomBatch];
#pragma unroll
        for (int h = 0; h < kMomBatch; ++h) {
          const int v = v0 + h * kEwThreads;
          if (v < nvec) {
            gw[h] = __ldg(gv + v);
            b0[h] = bv4[2 * v];
            b1[h] = bv4[2 * v + 1];
          }
        }
#pragma unroll
        for (int h = 0; h < kMomBatch; ++h) {
          const int v = v0 + h * kEwThreads;
          if (v >= nvec) continue;
          const uint32_t ws[4] = {gw[h].x, gw[h].y, gw[h].z, gw[h].w};
          float b[8] = {b0[h].x, b0[h].y, b0[h].z, b0[h].w, b1[h].x, b1[h].y, b1[h].z, b1[h].w};
          uint32_t packed[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float g0 = __uint_as_float(ws[k] << 16), g1 = __uint_as_float(ws[k] & 0xFFFF0000u);
            b[2 * k] = fmaf(P.mu, b[2 * k], g0);
            b[2 * k + 1] = fmaf(P.mu, b[2 * k + 1], g1);
            const float u0 = P.nesterov ? fmaf(P.mu, b[2 * k], g0) : b[2 * k];
            const float u1 = P.nesterov ? fmaf(P.mu, b[2 * k + 1], g1) : b[2 * k + 1];
            const __nv_bfloat162 hh = __floats2bfloat162_rn(u0, u1);
            packed[k] = *reinterpret_cast<const uint32_t*>(&hh);
            const float x0 = __low2float(hh), x1 = __high2float(hh);
            ss = fmaf(x0, x0, ss);
            ss = fmaf(x1, x1, ss);
          }
          bv4[2 * v] = make_float4(b[0], b[1], b[2], b[3]);
          bv4[2 * v + 1] = make_float4(b[4], b[5], b[6], b[7]);
          xv[v] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
      }
    } else if (vec) {
      const int cv = C >> 3;  // 8-element vectors per row
      const long long nvec = static_cast<long long>(r1 - r0) * cv;
      // two vectors per thread per iteration, all loads issued before any
      // store so that both are in flight together
      for (long long v0 = threadIdx.x; v0 < nvec; v0 += 2 * kEwThreads) {
        float g[2][8], bv[2][8];
        long long iv[2];
        bool have[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const long long v = v0 + h * kEwThreads;
          have[h] = v < nvec;
          const int r = r0 + static_cast<int>((have[h] ? v : v0) / cv);
          const int c = static_cast<int>((have[h] ? v : v0) % cv) * 8;
          iv[h] = static_cast<long long>(r) * C + c;
          if (!have[h]) continue;
          if (M.g_f32) {
            const float4* gp = reinterpret_cast<const float4*>(static_cast<const float*>(M.g) + iv[h]);
            const float4 a = gp[0], bq = gp[1];
            g[h][0] = a.x; g[h][1] = a.y; g[h][2] = a.z; g[h][3] = a.w;
            g[h][4] = bq.x; g[h][5] = bq.y; g[h][6] = bq.z; g[h][7] = bq.w;
          } else {
            const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(M.g) + iv[h]);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              g[h][2 * k] = __uint_as_float(ws[k] << 16);
              g[h][2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
            }
          }
          if (M.buf) {
            const float4* bp = reinterpret_cast<const float4*>(M.buf + iv[h]);
            const float4 b0 = bp[0], b1 = bp[1];
            bv[h][0] = b0.x; bv[h][1] = b0.y; bv[h][2] = b0.z; bv[h][3] = b0.w;
            bv[h][4] = b1.x; bv[h][5] = b1.y; bv[h][6] = b1.z; bv[h][7] = b1.w;
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!have[h]) continue;
          float u[8];
          if (M.buf) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              bv[h][k] = fmaf(P.mu, bv[h][k], g[h][k]);
              u[k] = P.nesterov ? fmaf(P.mu, bv[h][k], g[h][k]) : bv[h][k];
            }
            float4* bp = reinterpret_cast<float4*>(M.buf + iv[h]);
            bp[0] = make_float4(bv[h][0], bv[h][1], bv[h][2], bv[h][3]);
            bp[1] = make_float4(bv[h][4], bv[h][5], bv[h][6], bv[h][7]);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) u[k] = g[h][k];
          }
          uint32_t packed[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 hh = __floats2bfloat162_rn(u[2 * k], u[2 * k + 1]);
            packed[k] = *reinterpret_cast<const uint32_t*>(&hh);
            const float x0 = __low2float(hh), x1 = __high2float(hh);
            ss = fmaf(x0, x0, ss);
            ss = fmaf(x1, x1, ss);
          }
          const long long r = iv[h] / C, c = iv[h] % C;
          if (MUON_CHECK(iv[h] + 8 <= static_cast<long long>(R) * C && c + 8 <= M.ldx))
            *reinterpret_cast<uint4*>(M.x + r * M.ldx + c) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
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
    // tall: X = u^T (C x R).  A block covers 64 rows x kTallCols columns of
    // u, in 64 x 64 tiles through a double-buffered shared tile, so that both
    // the reads of u and the writes of X are contiguous across a warp.  A
    // thread loads 4 consecutive columns of 4 rows (float4 buf, 8-byte bf16
    // or 16-byte fp32 g) and stores 16 consecutive entries of one X row (two
    // 16-byte stores); the next tile's loads are issued before the current
    // tile is written out.
    const int ncb = (C + kTallCols - 1) / kTallCols;
    const int r0 = (b / ncb) * 64;
    const int cb0 = (b % ncb) * kTallCols;
    const int cb1 = min(C, cb0 + kTallCols);
    const int tid = threadIdx.x;
    const int cl = (tid & 15) * 4;  // tile columns cl .. cl + 3
    const int rq = tid >> 4;        // tile rows rq + 16 k
    auto write_out = [&](int c0, float (*tl)[kTallPitch]) {
      const int cc = tid >> 2;        // X row c0 + cc
      const int rb = (tid & 3) * 16;  // X columns r0 + rb .. + 15
      const int c = c0 + cc;
      if (c < cb1) {
        __nv_bfloat16* xd = M.x + static_cast<long long>(c) * M.ldx + r0 + rb;
        if (r0 + rb + 16 <= R && MUON_CHECK(r0 + rb + 16 <= M.ldx && c < C)) {
          uint32_t w[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const __nv_bfloat162 h =
                __floats2bfloat162_rn(tl[rb + 2 * j][tall_col(rb + 2 * j, cc)], tl[rb + 2 * j + 1][tall_col(rb + 2 * j + 1, cc)]);
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
          }
          reinterpret_cast<uint4*>(xd)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(xd)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
          for (int j = 0; j < 16 && r0 + rb + j < R; ++j) xd[j] = __float2bfloat16_rn(tl[rb + j][tall_col(rb + j, cc)]);
        }
      }
    };
    if ((C & 3) == 0) {
      // g and buf of one tile in registers (g raw: fp32 x 4, or bf16 x 4 in
      // the first two words)
      float4 gq[4], bq[4];
      auto load_tile = [&](int c0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = r0 + rq + 16 * k, c = c0 + cl;
          if (r < R && c < cb1) {
            const long long i = static_cast<long long>(r) * C + c;
            if (M.g_f32) {
              gq[k] = *reinterpret_cast<const float4*>(static_cast<const float*>(M.g) + i);
            } else {
              const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(M.g) + i);
              gq[k].x = __uint_as_float(v.x);
              gq[k].y = __uint_as_float(v.y);
            }
            if (M.buf) bq[k] = *reinterpret_cast<const float4*>(M.buf + i);
          }
        }
      };
      load_tile(cb0);
      int tb = 0;
      for (int c0 = cb0; c0 < cb1; c0 += 64, tb ^= 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rr = rq + 16 * k;
          const int r = r0 + rr, c = c0 + cl;
          float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          if (r < R && c < cb1) {
            float g[4];
            if (M.g_f32) {
              g[0] = gq[k].x; g[1] = gq[k].y; g[2] = gq[k].z; g[3] = gq[k].w;
            } else {
              const uint32_t w0 = __float_as_uint(gq[k].x), w1 = __float_as_uint(gq[k].y);
              g[0] = __uint_as_float(w0 << 16);
              g[1] = __uint_as_float(w0 & 0xFFFF0000u);
              g[2] = __uint_as_float(w1 << 16);
              g[3] = __uint_as_float(w1 & 0xFFFF0000u);
            }
            float u[4];
            if (M.buf) {
              float4 bv = bq[k];
              bv.x = fmaf(P.mu, bv.x, g[0]);
              bv.y = fmaf(P.mu, bv.y, g[1]);
              bv.z = fmaf(P.mu, bv.z, g[2]);
              bv.w = fmaf(P.mu, bv.w, g[3]);
              *reinterpret_cast<float4*>(M.buf + static_cast<long long>(r) * C + c) = bv;
              u[0] = P.nesterov ? fmaf(P.mu, bv.x, g[0]) : bv.x;
              u[1] = P.nesterov ? fmaf(P.mu, bv.y, g[1]) : bv.y;
              u[2] = P.nesterov ? fmaf(P.mu, bv.z, g[2]) : bv.z;
              u[3] = P.nesterov ? fmaf(P.mu, bv.w, g[3]) : bv.w;
            } else {
              u[0] = g[0]; u[1] = g[1]; u[2] = g[2]; u[3] = g[3];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              x[j] = bf16_round(u[j]);
              ss = fmaf(x[j], x[j], ss);
            }
          }
          // the upper half-warp writes its four columns in rotated order
          // (bank-conflict-free with the row pitch and column swizzle)
          const bool rot = (tid & 8) != 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int jr = rot ? (j + 1) & 3 : j;
            const float xv = rot ? x[(j + 1) & 3] : x[j];
            tile[tb][rr][tall_col(rr, cl + jr)] = xv;
          }
        }
        // one barrier per tile: the other buffer was last read before the
        // previous tile's barrier
        __syncthreads();
        if (c0 + 64 < cb1) load_tile(c0 + 64);
        write_out(c0, tile[tb]);
      }
    } else {
      for (int c0 = cb0; c0 < cb1; c0 += 64) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rr = rq + 16 * k;
          const int r = r0 + rr;
          for (int j = 0; j < 4; ++j) {
            const int c = c0 + cl + j;
            float x = 0.0f;
            if (r < R && c < cb1) {
              const long long i = static_cast<long long>(r) * C + c;
              x = bf16_round(momentum_u(load_g(M.g, M.g_f32, i), M.buf, i, P.mu, P.nesterov));
              ss = fmaf(x, x, ss);
            }
            tile[0][rr][tall_col(rr, cl + j)] = x;
          }
        }
        __syncthreads();
        write_out(c0, tile[0]);
        __syncthreads();
      }
    }
  }

  const float s = block_sum(ss, red);
  if (threadIdx.x == 0) P.partials[M.part_off + b] = s;
}

__global__ void __launch_bounds__(kEwThreads, 4) normalise_kernel(const __grid_constant__ NormParams P) {
  ptx_grid_dep_wait();
  __shared__ float red[kEwThreads / 32];
  __shared__ float sh_d;
  int c = 0;
  // blocks run in reverse order of the momentum pass's: the rows that pass
  // wrote last are read first, while they are still in L2 (56.0 -> 52.0 us on
  // the GPT-2 bank)
  const int bid = static_cast<int>(gridDim.x - 1 - blockIdx.x);
  while (c + 1 < P.n_classes && bid >= P.cls[c + 1].block_begin) ++c;
  const NormClass& K = P.cls[c];
  const int local = bid - K.block_begin;
  const int idx = local / K.blocks_per_mat;
  const int b = local - idx * K.blocks_per_mat;
  // debug build: the block's rows lie inside its class and matrix
  if (!MUON_CHECK(idx < K.count && b * K.rows_per_block < K.m)) return;
  const MatInfo mi = P.table[K.mat_begin + idx];

  __nv_bfloat16* X = K.x + static_cast<long long>(idx) * K.m * K.ldx;
  const int r0 = b * K.rows_per_block;
  const int r1 = min(K.m, r0 + K.rows_per_block);
  const int n = K.n;
  const bool vec = (n & 7) == 0;
  const int cv = n >> 3;  // 8-element vectors per row
  const long long nvec = vec ? static_cast<long long>(r1 - r0) * cv : 0;
  // a batch: kNormBatch vectors of 8 per thread, all loads issued before any
  // store; the first batch is loaded before the norm is known, so that the
  // reduction of the partials below overlaps its latency.  With n a multiple
  // of 8 the row pitch is n, so the block's rows [r0, r1) are one contiguous
  // run of nvec vectors.
  (void)cv;
  // debug build: the vector path's rows are contiguous
  if (vec && !MUON_CHECK(K.ldx == n)) return;
  uint4* const xv = reinterpret_cast<uint4*>(X + static_cast<long long>(r0) * n);
  uint4 w[kNormBatch];
  bool have[kNormBatch];
  auto load_batch = [&](long long v0) {
#pragma unroll
    for (int h = 0; h < kNormBatch; ++h) {
      const long long v = v0 + h * kEwThreads;
      have[h] = v < nvec;
      if (have[h]) w[h] = xv[v];
    }
  };
  if (vec) load_batch(threadIdx.x);

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
  // X0 = bf16(x * r), r = 1/d rounded to float: the product is within 1.5
  // float ulp of the quotient x/d (an IEEE division: 0.5 ulp) and costs one
  // instruction instead of a division sequence; after the bf16 rounding the
  // two differ only for quotients within 2^-8 bf16 ulp of a rounding midpoint
  const float inv_d = 1.0f / d;

  if (vec) {
    for (long long v0 = threadIdx.x; v0 < nvec; v0 += kNormBatch * kEwThreads) {
      if (v0 != threadIdx.x) load_batch(v0);
#pragma unroll
      for (int h = 0; h < kNormBatch; ++h) {
        if (!have[h]) continue;
        uint32_t ws[4] = {w[h].x, w[h].y, w[h].z, w[h].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = __uint_as_float(ws[k] << 16) * inv_d;
          const float hi = __uint_as_float(ws[k] & 0xFFFF0000u) * inv_d;
          const __nv_bfloat162 hh = __floats2bfloat162_rn(lo, hi);
          ws[k] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        xv[v0 + h * kEwThreads] = make_uint4(ws[0], ws[1], ws[2], ws[3]);
      }
    }
  } else {
    const long long ne = static_cast<long long>(r1 - r0) * n;
    for (long long e = threadIdx.x; e < ne; e += kEwThreads) {
      const int r = r0 + static_cast<int>(e / n);
      const int cc = static_cast<int>(e % n);
      __nv_bfloat16* p = X + static_cast<long long>(r) * K.ldx + cc;
      *p = __float2bfloat16_rn(__bfloat162float(*p) * inv_d);
    }
  }
}

// apply: O = X_final in the matrix's stored orientation; Newton-Schulz alone
// writes O (bf16), a Muon step with no iteration does p <- p - lr * O (fp32
// FMA; with iterations the last update does it).  One
// 64 x 64 tile of X per block.  Tall matrices (O = X^T) go through a shared
// tile so that both the reads of X and the accesses to p / O are contiguous
// across a warp.
__global__ void __launch_bounds__(kEwThreads) apply_kernel(const __grid_constant__ ApplyParams P) {
  ptx_grid_dep_wait();
  __shared__ float tile[64][65];
  int c = 0;
  while (c + 1 < P.n_classes && (int)blockIdx.x >= P.cls[c + 1].tile_begin) ++c;
  const ApplyClass& K = P.cls[c];
  const int local = blockIdx.x - K.tile_begin;
  const int per_mat = K.tiles_m * K.tiles_n;
  const int idx = local / per_mat;
  const int t = local - idx * per_mat;
  const int r0 = (t / K.tiles_n) * 64;  // X rows
  const int c0 = (t % K.tiles_n) * 64;  // X columns
  const MatInfo mi = P.table[K.mat_begin + idx];
  const __nv_bfloat16* X = K.x + static_cast<long long>(idx) * K.m * K.ldx;
  const int m = K.m, n = K.n;
  // debug build: the tile lies inside its matrix, whose recorded shape is
  // the class's
  if (!MUON_CHECK(idx < K.count && r0 < m && c0 < n && (mi.tall ? mi.C == m && mi.R == n : mi.R == m && mi.C == n)))
    return;
  const int tid = threadIdx.x;
  const bool param = P.final_mode == kFinalParam;
  if (!mi.tall) {
    // stored as X: element (r, c) at r * n + c; a thread handles 8 columns
    // of two rows, both rows' loads issued before the stores
    if ((n & 7) == 0) {
      uint4 w[2];
      float4 pa[2], pb[2];
      long long o[2];
      bool have[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int r = r0 + (tid >> 3) + 32 * k;
        const int cc = c0 + (tid & 7) * 8;
        have[k] = r < m && cc < n;
        o[k] = static_cast<long long>(r) * n + cc;
        if (!have[k]) continue;
        w[k] = *reinterpret_cast<const uint4*>(X + static_cast<long long>(r) * K.ldx + cc);
        if (param) {
          const float4* pp = reinterpret_cast<const float4*>(static_cast<const float*>(mi.out) + o[k]);
          pa[k] = pp[0];
          pb[k] = pp[1];
        }
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (!have[k]) continue;
        if (param) {
          const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
          float4 a = pa[k], b = pb[k];
          a.x = fmaf(-P.lr, __uint_as_float(ws[0] << 16), a.x);
          a.y = fmaf(-P.lr, __uint_as_float(ws[0] & 0xFFFF0000u), a.y);
          a.z = fmaf(-P.lr, __uint_as_float(ws[1] << 16), a.z);
          a.w = fmaf(-P.lr, __uint_as_float(ws[1] & 0xFFFF0000u), a.w);
          b.x = fmaf(-P.lr, __uint_as_float(ws[2] << 16), b.x);
          b.y = fmaf(-P.lr, __uint_as_float(ws[2] & 0xFFFF0000u), b.y);
          b.z = fmaf(-P.lr, __uint_as_float(ws[3] << 16), b.z);
          b.w = fmaf(-P.lr, __uint_as_float(ws[3] & 0xFFFF0000u), b.w);
          float4* pp = reinterpret_cast<float4*>(static_cast<float*>(mi.out) + o[k]);
          pp[0] = a;
          pp[1] = b;
        } else {
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(mi.out) + o[k]) = w[k];
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int r = r0 + (tid >> 3) + 32 * k;
        const int cc = c0 + (tid & 7) * 8;
        if (r >= m || cc >= n) continue;
        const __nv_bfloat16* xs = X + static_cast<long long>(r) * K.ldx + cc;
        const long long o = static_cast<long long>(r) * n + cc;
        for (int j = 0; j < 8 && cc + j < n; ++j) {
          const __nv_bfloat16 x = xs[j];
          if (param) {
            float* pp = static_cast<float*>(mi.out) + o + j;
            *pp = fmaf(-P.lr, __bfloat162float(x), *pp);
          } else {
            static_cast<__nv_bfloat16*>(mi.out)[o + j] = x;
          }
        }
      }
    }
  } else {
    // stored as X^T (n x m): element (c, r) at c * m + r.  X tile in with
    // 16-byte loads, out along p's rows with 4-element vectors.
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int e = tid + kEwThreads * k;
      const int rr = e >> 3, cc = (e & 7) * 8;
      const int r = r0 + rr, col = c0 + cc;
      if (r < m && col + 8 <= n) {
        const uint4 v = *reinterpret_cast<const uint4*>(X + static_cast<long long>(r) * K.ldx + col);
        const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          tile[rr][cc + 2 * j] = __uint_as_float(ws[j] << 16);
          tile[rr][cc + 2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          tile[rr][cc + j] = (r < m && col + j < n) ? __bfloat162float(X[static_cast<long long>(r) * K.ldx + col + j]) : 0.0f;
      }
    }
    __syncthreads();
    if ((m & 3) == 0) {
      float4 pv[4];
      bool have[4];
      long long o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = tid + kEwThreads * k;
        const int jj = e >> 4, rr = (e & 15) * 4;
        const int col = c0 + jj, r = r0 + rr;
        have[k] = col < n && r < m;  // m % 4 == 0: the 4 entries are all in range
        o[k] = static_cast<long long>(col) * m + r;
        if (have[k] && param) pv[k] = *reinterpret_cast<const float4*>(static_cast<const float*>(mi.out) + o[k]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!have[k]) continue;
        const int e = tid + kEwThreads * k;
        const int jj = e >> 4, rr = (e & 15) * 4;
        const float x0 = tile[rr][jj], x1 = tile[rr + 1][jj], x2 = tile[rr + 2][jj], x3 = tile[rr + 3][jj];
        if (param) {
          float4 a = pv[k];
          a.x = fmaf(-P.lr, x0, a.x);
          a.y = fmaf(-P.lr, x1, a.y);
          a.z = fmaf(-P.lr, x2, a.z);
          a.w = fmaf(-P.lr, x3, a.w);
          *reinterpret_cast<float4*>(static_cast<float*>(mi.out) + o[k]) = a;
        } else {
          const __nv_bfloat162 h0 = __floats2bfloat162_rn(x0, x1), h1 = __floats2bfloat162_rn(x2, x3);
          uint2 u;
          u.x = *reinterpret_cast<const uint32_t*>(&h0);
          u.y = *reinterpret_cast<const uint32_t*>(&h1);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(mi.out) + o[k]) = u;
        }
      }
    } else {
      for (int e = tid; e < 64 * 64; e += kEwThreads) {
        const int cc = e >> 6, rr = e & 63;
        const int r = r0 + rr, col = c0 + cc;
        if (r >= m || col >= n) continue;
        const long long o = static_cast<long long>(col) * m + r;
        const float x = tile[rr][cc];
        if (param) {
          float* pp = static_cast<float*>(mi.out) + o;
          *pp = fmaf(-P.lr, x, *pp);
        } else {
          static_cast<__nv_bfloat16*>(mi.out)[o] = __float2bfloat16_rn(x);
        }
      }
    }
  }
}

cudaError_t launch_momentum_cast(const K1Params& P, int blocks, cudaStream_t stream) {
  void* args[] = {const_cast<K1Params*>(&P)};
  return launch_pdl(reinterpret_cast<const void*>(&momentum_cast_kernel), blocks, args, stream);
}

cudaError_t launch_apply(const ApplyParams& P, int blocks, cudaStream_t stream) {
  void* args[] = {const_cast<ApplyParams*>(&P)};
  return launch_pdl(reinterpret_cast<const void*>(&apply_kernel), blocks, args, stream);
}

cudaError_t launch_normalise(const NormParams& P, int blocks, cudaStream_t stream) {
  void* args[] = {const_cast<NormParams*>(&P)};
  return launch_pdl(reinterpret_cast<const void*>(&normalise_kernel), blocks, args, stream);
}

MUON_CHECK_READER(check_failures_elementwise)

}  // namespace muon
