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
//             tile and fuses a X + (.).  (The parameter update after the
//             last step is a separate coalesced pass, apply_kernel.)
//
// Kernel structure (one CTA per SM, persistent over a static tile list that
// spans all shape classes of the bank):
//   warp 0     TMA producer: 4-stage ring of (128 x 64) A and (256 x 64) B
//              tiles, 128-byte swizzle, one mbarrier pair per stage.
//   warp 1     TMEM owner and MMA issuer: tcgen05.mma 128 x 256 x 16, fp32
//              accumulators in TMEM, two accumulator buffers (2 x 256 columns)
//              so the epilogue of one tile overlaps the main loop of the next.
//   warps 2-9  epilogue: two warps per TMEM lane quarter, each owning half of
//              the tile's 256 columns; the epilogue input row (A or X) is
//              loaded before the accumulator is ready, then tcgen05.ld of 32
//              columns at a time, fused arithmetic, bf16 rounding, stores.
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
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
// 32 consecutive bf16 of one row as 16 packed words (zeros past `valid`).
__device__ __forceinline__ void load_words32(const __nv_bfloat16* src, int valid, uint32_t (&w)[16]) {
  if (valid >= 32) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = s[q];
      w[4 * q] = v.x;
      w[4 * q + 1] = v.y;
      w[4 * q + 2] = v.z;
      w[4 * q + 3] = v.w;
    }
  } else {
    const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t lo = 2 * j < valid ? s[2 * j] : 0u;
      const uint32_t hi = 2 * j + 1 < valid ? s[2 * j + 1] : 0u;
      w[j] = lo | (hi << 16);
    }
  }
}

__device__ __forceinline__ float word_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float word_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One 32-column chunk of one tile row: `acc` from TMEM, `aux` the row's
// epilogue input (A for the polynomial, X for the update; unused for Gram).
template <int MODE>
__device__ __forceinline__ void epilogue_chunk(const GemmParams& P, const GemmClass& C,
                                               const Tile& tl, int rg, int c0,
                                               const uint32_t (&acc)[32], const uint32_t (&aux)[16]) {
  uint32_t w[16];
  if (MODE == kGram) {
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]));
  } else if (MODE == kPoly) {
    // B = b A + c (A A)
#pragma unroll
    for (int j = 0; j < 16; ++j)
      w[j] = pack_bf16x2(fmaf(P.cb, word_lo(aux[j]), P.cc * __uint_as_float(acc[2 * j])),
                         fmaf(P.cb, word_hi(aux[j]), P.cc * __uint_as_float(acc[2 * j + 1])));
  } else {
    // X' = a X + B X
#pragma unroll
    for (int j = 0; j < 16; ++j)
      w[j] = pack_bf16x2(fmaf(P.ca, word_lo(aux[j]), __uint_as_float(acc[2 * j])),
                         fmaf(P.ca, word_hi(aux[j]), __uint_as_float(acc[2 * j + 1])));
  }
  __nv_bfloat16* out = C.out + tl.idx * C.out_mat_stride;
  if (MODE == kUpdate) {
    store_row32(out + static_cast<long long>(rg) * C.ld_out + c0, C.n - c0, w);
    return;
  }
  const int m = C.m;
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
      ptx::mbar_init(ptx::smem_addr(&tempty[a]), 32 * kEpiWarps);
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
    // Warp w (2..9) reads TMEM lane quarter w % 4 (rows 32q..32q+31 of the
    // tile) and the column half (w - 2) / 4 (chunks 4h .. 4h+3 of 32 columns).
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = q * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < P.total_tiles; t += gridDim.x, ++it) {
      const Tile tl = decode_tile<MODE>(P, t);
      const GemmClass& C = P.cls[tl.cls];
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const int rg = tl.I * kBM + row_in_tile;
      const int warp_row0 = tl.I * kBM + q * 32;
      const int ncols = MODE == kUpdate ? C.n : C.m;
      const int cbase = tl.J * kBN + half * (kBN / 2);
      // this thread's epilogue input for its 128 columns, loaded before the
      // accumulator is ready so that the loads overlap the main loop
      uint32_t aux[4][16];
      if (MODE != kGram) {
        const __nv_bfloat16* arow = C.aux + tl.idx * C.aux_mat_stride + static_cast<long long>(rg) * C.ld_aux;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int c0 = cbase + ch * 32;
          if (rg < C.m && c0 < ncols) {
            load_words32(arow + c0, ncols - c0, aux[ch]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) aux[ch][j] = 0u;
          }
        }
      }
      if (!ptx::mbar_wait(ptx::smem_addr(&tfull[acc]), acc_phase, budget, abort)) {
        raise_timeout(P, abort);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN + half * (kBN / 2);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int c0 = cbase + ch * 32;
        if (c0 >= ncols) break;  // warp-uniform
        if (MODE != kUpdate && c0 + 31 < warp_row0) continue;  // strictly below the diagonal
        uint32_t r[32];
        __syncwarp();
        ptx::tmem_ld32(tb + ch * 32, r);
        ptx::tmem_ld_wait();
        if (rg < C.m) epilogue_chunk<MODE>(P, C, tl, rg, c0, r, aux[ch]);
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
