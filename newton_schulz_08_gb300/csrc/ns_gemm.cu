// The three contractions of one quintic Newton-Schulz step, on the sm_103a
// tensor cores (tcgen05 + TMA + TMEM), for every matrix of a bank at once.
//
// Method: page "深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术"
// (reposource.net), section "Newton-Schulz正交化": per step
//     A = X X^T,   B = b A + c A A,   X' = a X + B X,
// with X an m x n bfloat16 matrix (m <= n) and (a, b, c) = (3.4445, -4.7750,
// 2.0315).  Each statement's result is rounded once to bfloat16.
//
//   kGram   : A = X X^T.          Only tiles holding upper-triangle entries are
//             computed; the epilogue writes each entry with r <= c to (r, c)
//             and, mirrored, to (c, r), so A is exactly symmetric.
//   kPoly   : B = b A + c (A A).  A is symmetric, so A A = A A^T and the same
//             upper-triangle Gram structure applies with K = m; the epilogue
//             reads A's tile and fuses b A + c (.).
//   kUpdate : X' = a X + B X.     All tiles of the m x n result; B is the
//             K-major operand, X the MN-major one.  The epilogue reads X's
//             tile and fuses a X + (.).  On the last step it applies the
//             parameter update p <- p - lr O (or writes O), transposing back
//             matrices that were tall.
//
// Kernel structure (one CTA per SM, persistent over a static tile list that
// spans all shape classes of the bank):
//   warp 0     TMA producer: 4-stage ring of (128 x 64) A and (256 x 64) B
//              tiles, 128-byte swizzle, one mbarrier pair per stage.
//   warp 1     TMEM owner and MMA issuer: tcgen05.mma 128 x 256 x 16, fp32
//              accumulators in TMEM, two accumulator buffers (2 x 256 columns)
//              so the epilogue of one tile overlaps the main loop of the next.
//   warps 2-5  epilogue: tcgen05.ld of 32 columns at a time, fused arithmetic,
//              bfloat16 rounding, global stores.
// Every barrier wait is bounded; on expiry the CTA raises the timeout bit of
// the device status word, drains its own in-flight copies and MMAs, frees
// TMEM and returns.
#include "plan.h"
#include "ptx.cuh"

namespace muon {

namespace {

struct Tile {
  int cls, idx, I, J;
};

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const GemmParams& P, int t) {
  int c = 0;
#pragma unroll 1
  while (c + 1 < P.n_classes && t >= P.cls[c + 1].tile_begin) ++c;
  const GemmClass& C = P.cls[c];
  const int local = t - C.tile_begin;
  Tile r;
  r.cls = c;
  r.idx = local / C.tiles_per_mat;
  int q = local - r.idx * C.tiles_per_mat;
  if (MODE == kUpdate) {
    r.I = q % C.tiles_m;
    r.J = q / C.tiles_m;
  } else {
    // column block J holds row blocks 0 .. min(2J+1, tiles_m-1)
    int J = 0;
#pragma unroll 1
    while (true) {
      const int cnt = min(2 * J + 2, C.tiles_m);
      if (q < cnt) break;
      q -= cnt;
      ++J;
    }
    r.I = q;
    r.J = J;
  }
  return r;
}

__device__ __forceinline__ void raise_timeout(const GemmParams& P, volatile int* abort) {
  *abort = 1;
  atomicOr(P.status, kStatusTimeout);
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t u, float& lo, float& hi) {
  lo = __uint_as_float(u << 16);
  hi = __uint_as_float(u & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Load 32 consecutive bf16 (row-major, starting at `src`) as floats.
__device__ __forceinline__ void load_row32(const __nv_bfloat16* src, int valid, float (&v)[32]) {
  if (valid >= 32) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = s[q];
      unpack_bf16x2(w.x, v[8 * q + 0], v[8 * q + 1]);
      unpack_bf16x2(w.y, v[8 * q + 2], v[8 * q + 3]);
      unpack_bf16x2(w.z, v[8 * q + 4], v[8 * q + 5]);
      unpack_bf16x2(w.w, v[8 * q + 6], v[8 * q + 7]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = j < valid ? __bfloat162float(src[j]) : 0.0f;
  }
}

// Store 32 packed bf16 (16 words) to `dst`, first `valid` elements only.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, int valid, const uint32_t (&w)[16]) {
  if (valid >= 32) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) d[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  } else {
    uint16_t* d = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < valid) d[j] = static_cast<uint16_t>((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
  }
}

__device__ __forceinline__ uint16_t word_half(const uint32_t (&w)[16], int j) {
  return static_cast<uint16_t>((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
}

// ------------------------------------------------------------------ epilogues
template <int MODE>
__device__ __forceinline__ void epilogue_chunk(const GemmParams& P, const GemmClass& C,
                                               const Tile& tl, int rg, int c0,
                                               const uint32_t (&acc)[32]) {
  if (MODE == kGram || MODE == kPoly) {
    const int m = C.m;
    if (rg >= m) return;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(acc[j]);
    if (MODE == kPoly) {
      float a[32];
      const __nv_bfloat16* src = C.aux + tl.idx * C.aux_mat_stride + static_cast<long long>(rg) * C.ld_aux + c0;
      load_row32(src, m - c0, a);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = fmaf(P.cb, a[j], P.cc * v[j]);
    }
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
    __nv_bfloat16* out = C.out + tl.idx * C.out_mat_stride;
    // direct: entries with rg <= c
    __nv_bfloat16* drow = out + static_cast<long long>(rg) * C.ld_out + c0;
    if (c0 >= rg) {
      store_row32(drow, m - c0, w);
    } else {
      uint16_t* d = reinterpret_cast<uint16_t*>(drow);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = c0 + j;
        if (c >= rg && c < m) d[j] = word_half(w, j);
      }
    }
    // mirror: entries with rg < c go to (c, rg); a warp writes 32 adjacent rg
    uint16_t* mcol = reinterpret_cast<uint16_t*>(out) + rg;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int c = c0 + j;
      if (c > rg && c < m) mcol[static_cast<long long>(c) * C.ld_out] = word_half(w, j);
    }
  } else {
    const int m = C.m, n = C.n;
    if (rg >= m) return;
    const int valid = n - c0;
    float x[32];
    const __nv_bfloat16* xs = C.aux + tl.idx * C.aux_mat_stride + static_cast<long long>(rg) * C.ld_aux + c0;
    load_row32(xs, valid, x);
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      w[j] = pack_bf16x2(fmaf(P.ca, x[2 * j], __uint_as_float(acc[2 * j])),
                         fmaf(P.ca, x[2 * j + 1], __uint_as_float(acc[2 * j + 1])));
    if (P.store_x) {
      __nv_bfloat16* xd = C.out + tl.idx * C.out_mat_stride + static_cast<long long>(rg) * C.ld_out + c0;
      store_row32(xd, valid, w);
    }
    if (P.final_mode != kFinalNone) {
      const MatInfo mi = P.table[C.mat_begin + tl.idx];
      if (P.final_mode == kFinalParam) {
        float* p = static_cast<float*>(mi.out);
        if (!mi.tall) {
          float* prow = p + static_cast<long long>(rg) * n + c0;
          if (valid >= 32 && (n & 3) == 0) {
            float4* p4 = reinterpret_cast<float4*>(prow);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4 t = p4[q];
              float o0, o1, o2, o3;
              unpack_bf16x2(w[2 * q], o0, o1);
              unpack_bf16x2(w[2 * q + 1], o2, o3);
              t.x = fmaf(-P.lr, o0, t.x);
              t.y = fmaf(-P.lr, o1, t.y);
              t.z = fmaf(-P.lr, o2, t.z);
              t.w = fmaf(-P.lr, o3, t.w);
              p4[q] = t;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (j < valid) {
                float o = __uint_as_float(static_cast<uint32_t>(word_half(w, j)) << 16);
                prow[j] = fmaf(-P.lr, o, prow[j]);
              }
            }
          }
        } else {
          // tall: O = X^T, p is n x m; a warp covers 32 adjacent rg
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < valid) {
              float* pe = p + static_cast<long long>(c0 + j) * m + rg;
              float o = __uint_as_float(static_cast<uint32_t>(word_half(w, j)) << 16);
              *pe = fmaf(-P.lr, o, *pe);
            }
          }
        }
      } else {
        uint16_t* o = static_cast<uint16_t*>(mi.out);
        if (!mi.tall) {
          uint16_t* orow = o + static_cast<long long>(rg) * n + c0;
          if ((n & 7) == 0) {
            store_row32(reinterpret_cast<__nv_bfloat16*>(orow), valid, w);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < valid) orow[j] = word_half(w, j);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < valid) o[static_cast<long long>(c0 + j) * m + rg] = word_half(w, j);
        }
      }
    }
  }
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = bars + 2 * kStages + 2;
  uint64_t* drain = bars + 2 * kStages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never = reinterpret_cast<volatile int*>(tmem_slot + 2);  // stays 0

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_addr(&tfull[a]), 1);
      ptx::mbar_init(ptx::smem_addr(&tempty[a]), 128);
    }
    ptx::mbar_init(ptx::smem_addr(drain), 1);
    *abort = 0;
    *never = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const long long budget = P.wait_budget;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      for (int c = 0; c < P.n_classes; ++c) {
        ptx::prefetch_tmap(&P.cls[c].tmA);
        ptx::prefetch_tmap(&P.cls[c].tmB);
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[kStages];
      bool issued[kStages];
      for (int s = 0; s < kStages; ++s) issued[s] = false, issued_phase[s] = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < P.total_tiles; t += gridDim.x) {
        const Tile tl = decode_tile<MODE>(P, t);
        const GemmClass& C = P.cls[tl.cls];
        const int kblocks = (C.K + kBK - 1) / kBK;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_addr(&empty[stage]), phase ^ 1, budget, abort)) {
            raise_timeout(P, abort);
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_addr(&full[stage]);
          const uint32_t sa = ptx::smem_addr(smem + stage * kStageBytes);
          const uint32_t sb = sa + kStageA;
          ptx::mbar_arrive_expect_tx(fb, kStageBytes);
          ptx::tma_load_3d(sa, &C.tmA, fb, kb * kBK, tl.I * kBM, tl.idx);
          if (MODE == kUpdate) {
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j)
              ptx::tma_load_3d(sb + j * (64 * kBK * 2), &C.tmB, fb, tl.J * kBN + 64 * j, kb * kBK, tl.idx);
          } else {
            ptx::tma_load_3d(sb, &C.tmB, fb, kb * kBK, tl.J * kBN, tl.idx);
            ptx::tma_load_3d(sb + kBM * kBK * 2, &C.tmB, fb, kb * kBK, tl.J * kBN + kBM, tl.idx);
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // let copies already in flight land before the CTA goes away
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) ptx::mbar_wait(ptx::smem_addr(&full[s]), issued_phase[s], budget, never);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && !P.inject_stall) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16(kBM, kBN, 0, MODE == kUpdate ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < P.total_tiles; t += gridDim.x, ++it) {
        const Tile tl = decode_tile<MODE>(P, t);
        const GemmClass& C = P.cls[tl.cls];
        const int kblocks = (C.K + kBK - 1) / kBK;
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!ptx::mbar_wait(ptx::smem_addr(&tempty[acc]), acc_phase ^ 1, budget, abort)) {
          raise_timeout(P, abort);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + acc * kBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_addr(&full[stage]), phase, budget, abort)) {
            raise_timeout(P, abort);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_addr(smem + stage * kStageBytes);
          const uint32_t sb = sa + kStageA;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t adesc = ptx::sdesc_sw128(sa + k * 32, 16, 1024);
            const uint64_t bdesc = MODE == kUpdate ? ptx::sdesc_sw128(sb + k * 2048, 64 * kBK * 2, 1024)
                                                   : ptx::sdesc_sw128(sb + k * 32, 16, 1024);
            ptx::mma_bf16(d, adesc, bdesc, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_addr(&empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_addr(&tfull[acc]));
      }
      // wait until every MMA issued here has completed
      ptx::mma_commit(ptx::smem_addr(drain));
      ptx::mbar_wait(ptx::smem_addr(drain), 0, budget, never);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < P.total_tiles; t += gridDim.x, ++it) {
      const Tile tl = decode_tile<MODE>(P, t);
      const GemmClass& C = P.cls[tl.cls];
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!ptx::mbar_wait(ptx::smem_addr(&tfull[acc]), acc_phase, budget, abort)) {
        raise_timeout(P, abort);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN;
      const int rg = tl.I * kBM + row_in_tile;
      const int warp_row0 = tl.I * kBM + q * 32;
      const int ncols = MODE == kUpdate ? C.n : C.m;
#pragma unroll 1
      for (int ch = 0; ch < kBN / 32; ++ch) {
        const int c0 = tl.J * kBN + ch * 32;
        if (c0 >= ncols) break;  // warp-uniform
        if (MODE != kUpdate && c0 + 31 < warp_row0) continue;  // strictly below the diagonal
        uint32_t r[32];
        __syncwarp();
        ptx::tmem_ld32(tb + ch * 32, r);
        ptx::tmem_ld_wait();
        epilogue_chunk<MODE>(P, C, tl, rg, c0, r);
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_addr(&tempty[acc]));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

template __global__ void ns_gemm_kernel<kGram>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kPoly>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kUpdate>(const __grid_constant__ GemmParams P);

// ------------------------------------------------------------------ launcher
cudaError_t launch_ns_gemm(int mode, const GemmParams& P, int num_sms, cudaStream_t stream) {
  const void* fn = mode == kGram   ? reinterpret_cast<const void*>(&ns_gemm_kernel<kGram>)
                   : mode == kPoly ? reinterpret_cast<const void*>(&ns_gemm_kernel<kPoly>)
                                   : reinterpret_cast<const void*>(&ns_gemm_kernel<kUpdate>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  const int grid = P.total_tiles < num_sms ? P.total_tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  void* args[] = {const_cast<GemmParams*>(&P)};
  return cudaLaunchKernel(fn, dim3(grid), dim3(kGemmThreads), args, kGemmSmem, stream);
}

}  // namespace muon
