// The three contractions of one quintic Newton-Schulz step, on the sm_103a
// tensor cores (tcgen05 + TMA + TMEM), for every matrix of a bank at once.
//
// Method: page "深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术"
// (reposource.net), section "Newton-Schulz正交化": per step
//     A = X X^T,   B = b A + c A A,   X' = a X + B X,
// with X an m x n bfloat16 matrix (m <= n) and (a, b, c) = (3.4445, -4.7750,
// 2.0315).  Each statement's result is rounded once to bfloat16.
//
//   kGram   : A = X X^T.          Only the 256 x 256 blocks on and above the
//             diagonal are computed (diagonal blocks whole: the tensor core's
//             sums for (r, c) and (c, r) agree bit for bit, so A is exactly
//             symmetric).  For m up to kSymUpperMaxM only those blocks are
//             stored and the polynomial reads the others transposed; for
//             wider A the epilogue also writes the mirrored entries.
//   kPoly   : B = b A + c (A A).  A is symmetric, so A A = A A^T and the same
//             block-upper structure applies with K = m.  Where A is stored
//             block-upper, operand blocks below the diagonal are loaded from
//             the stored block above it as MN-major operands (one 4-D copy
//             per 128 x 64 half where the width is a multiple of 64), and B
//             is stored block-upper as well; for wider matrices the epilogue
//             also writes the mirrored entries, so B is stored whole.  The
//             epilogue reads A's (upper) tile and fuses b A + c (.).
//   kUpdate : X' = a X + B X.     All tiles of the m x n result; B is the
//             A operand (K-major, or MN-major where a block-upper B is read
//             below its diagonal), X the MN-major B operand.  The epilogue
//             reads X's tile and fuses a X + (.).  In the last step of the
//             Muon step it applies p <- p - lr X' (fp32, in p's own layout)
//             instead of storing X'.
//   kFp8    : out = s (A B^T), the FP8 scaled product of the same page's
//             section "自定义FP8矩阵乘法实现": A (M x K) and B (N x K) in E4M3,
//             both K-major (tcgen05.mma kind::f8f6f4, K blocks of 128
//             one-byte elements, the same 128-byte rows as 64 bf16), s =
//             x_s w_s applied to the fp32 accumulator, bf16 out.
//
// Kernel structure: clusters of two CTAs on neighbouring SMs; each pair
// computes 256 x 256 output tiles with tcgen05.mma.cta_group::2 (M = 256 over
// the pair), persistent over a static tile list that spans all shape classes
// of the bank.  Per CTA:
//   warp 0     TMA producer: 5-stage ring (6 for the Gram, whose epilogue
//              stages no input) of this CTA's halves, (128 x 64) A rows and
//              (128 x 64) B columns, 128-byte swizzle; completion is counted
//              on the leader CTA's full barrier.
//   warp 1     TMEM allocation (both CTAs, 2 x 256 fp32 accumulator columns);
//              in the leader CTA one thread issues the MMAs 256 x 256 x 16
//              (operand major-ness chosen per K block in the polynomial) and
//              commits to the
//              stage / accumulator barriers of both CTAs.
//   warps 2-9  epilogue of this CTA's 128 accumulator rows: two warps per
//              TMEM lane quarter, each owning half of the 256 columns and
//              working alone (its own TMA boxes and input barrier):
//              tcgen05.ld of 32 columns at a time, fused arithmetic, bf16
//              rounding, staged stores; an arrive on the leader's
//              accumulator-empty barrier once its columns are read.
// Each CTA moves 32 KB per 64-deep K block for 2 x 128 x 256 x 64 MACs of
// the pair: a third less operand traffic per FLOP than single-CTA
// 128 x 256 tiles.  Every barrier wait is bounded; on expiry the CTA raises
// the timeout bit of the device status word, lets its copies and MMAs
// drain, frees TMEM and returns.
#include <mutex>

#include "check.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace muon {

namespace {

struct Tile {
  int cls, idx, I, J;
  int split;  // kFp8: slice of the contraction (0 when it is not split)
};

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const GemmParams& P, int t) {
  // A launch may walk its tile list from the end (the planner's choice, for
  // L2 reuse of what the previous launch wrote last).  Every role of a CTA
  // decodes the same sequence, so the order is all that changes.
  if (P.reverse) t = P.total_tiles - 1 - t;
  int c = 0;
#pragma unroll 1
  while (c + 1 < P.n_classes && t >= P.cls[c + 1].tile_begin) ++c;
  const GemmClass& C = P.cls[c];
  const int local = t - C.tile_begin;
  Tile r;
  r.cls = c;
  r.idx = local / C.tiles_per_mat;
  int q = local - r.idx * C.tiles_per_mat;
  r.split = 0;
  if (MODE == kFp8) {
    const int mn = C.tiles_m * C.tiles_n;
    r.split = q / mn;
    q -= r.split * mn;
    r.I = q % C.tiles_m;
    r.J = q / C.tiles_m;
  } else if (MODE == kUpdate) {
    r.I = q % C.tiles_m;
    r.J = q / C.tiles_m;
  } else {
    // square tiles on and above the diagonal: column block J holds row
    // blocks 0 .. J
    int J = 0;
#pragma unroll 1
    while (true) {
      const int cnt = J + 1;
      if (q < cnt) break;
      q -= cnt;
      ++J;
    }
    r.I = q;
    r.J = J;
  }
  return r;
}

// K blocks [*kb0, *kb1) of a tile: the whole contraction, or the tile's
// slice of it when the class splits it (kFp8)
template <int MODE>
__device__ __forceinline__ void k_range(const GemmClass& C, const Tile& tl, int kkb, int* kb0, int* kb1) {
  const int kblocks = (C.K + kkb - 1) / kkb;
  if (MODE == kFp8 && C.ksplit > 1) {
    const int per = (kblocks + C.ksplit - 1) / C.ksplit;
    *kb0 = tl.split * per;
    *kb1 = min(kblocks, *kb0 + per);
  } else {
    *kb0 = 0;
    *kb1 = kblocks;
  }
}

__device__ __forceinline__ void raise_timeout(const GemmParams& P, volatile int* abort) {
  *abort = 1;
  atomicOr(P.status, kStatusTimeout);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float word_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float word_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace

// SYM: 1 for classes whose A and B are stored as their blocks on and above
// the diagonal only (m <= kSymUpperMaxM): the Gram and the polynomial write
// no mirrored entries, the polynomial reads A's blocks below the diagonal
// transposed and the update reads B's.  A compile-time choice, so that the
// other classes run code without any of it.
// APPLY (update only): the Muon step's last update, which applies
// p <- p - lr X' instead of storing X'; also compile-time, so that the other
// updates run without its registers.
template <int MODE, int SYM, int APPLY>
__global__ void __launch_bounds__(kGemmThreads, 1)
    ns_gemm_kernel(const __grid_constant__ typename GemmParamsOf<APPLY>::type P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using Shape = GemmShape<MODE, APPLY>;
  constexpr int kSt = Shape::stages;
  // the Gram and the FP8 product stage no epilogue input; an FP8 K block is
  // 128 one-byte elements (a 128-byte row, as 64 bf16 are)
  constexpr bool kNoAux = MODE == kGram || MODE == kFp8;
  // the Gram stages one 64 x 32 box per warp (32 KB in all); the others stage
  // the warp's two boxes (64 KB)
  constexpr bool kSmallStg = MODE == kGram;
  constexpr int kKB = MODE == kFp8 ? 2 * kBK : kBK;  // elements per K block
  uint8_t* stg = smem + kSt * kStageBytes;  // epilogue staging tile
  uint8_t* pslots = stg + Shape::staging;    // APPLY 2: parameter blocks
  uint64_t* bars = reinterpret_cast<uint64_t*>(pslots + Shape::pslots);
  uint64_t* full = bars;                       // leader: both CTAs' tiles landed
  uint64_t* empty = bars + kSt;            // stage free in this CTA
  uint64_t* tfull = bars + 2 * kSt;        // accumulator ready (this CTA's lanes)
  uint64_t* tempty = bars + 2 * kSt + 2;   // leader: both CTAs drained it
  uint64_t* drain = bars + 2 * kSt + 4;
  uint64_t* aux_full = bars + 2 * kSt + 5; // [kEpiWarps] epilogue input of a warp landed
  uint64_t* pfull = aux_full + kEpiWarps;   // [kEpiWarps][2] APPLY 2: a parameter block landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pfull + 2 * kEpiWarps);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never = reinterpret_cast<volatile int*>(tmem_slot + 2);  // stays 0

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long t_start = clock64();
  long long* prof = P.wait_profile && MODE != kFp8 ? P.wait_profile + (MODE * 256 + static_cast<long long>(blockIdx.x)) * kWaitCounters
                                   : nullptr;
  const uint32_t rank = ptx::cluster_ctarank();  // 0: leader (issues the MMAs)
  const int pair = static_cast<int>(ptx::cluster_id_x());
  const int npairs = static_cast<int>(ptx::nclusters_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_addr(&tfull[a]), 1);
      ptx::mbar_init(ptx::smem_addr(&tempty[a]), 2 * kEpiWarps);
    }
    ptx::mbar_init(ptx::smem_addr(drain), 1);
    for (int w = 0; w < kEpiWarps; ++w) ptx::mbar_init(ptx::smem_addr(&aux_full[w]), 1);
    for (int w = 0; w < 2 * kEpiWarps; ++w) ptx::mbar_init(ptx::smem_addr(&pfull[w]), 1);
    *abort = 0;
    *never = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), 512);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncwarp();
  ptx::cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  ptx::tc_fence_after();
  // the prologue above overlaps the previous kernel's tail; from here on this
  // kernel reads what that kernel wrote
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const uint32_t tmem_base = *tmem_slot;
  const long long budget = P.wait_budget;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      // Both CTAs load their own halves (A rows, B columns) into their own
      // shared memory; completion is counted on the leader's full barrier.
      for (int c = 0; c < P.n_classes; ++c) {
        ptx::prefetch_tmap(&P.cls[c].tmA);
        ptx::prefetch_tmap(&P.cls[c].tmB);
        ptx::prefetch_tmap(&P.cls[c].tmAux);
        ptx::prefetch_tmap(&P.cls[c].tmOut);
        ptx::prefetch_tmap(&P.cls[c].tmT);
        ptx::prefetch_tmap(&P.cls[c].tmT4);
        if (MODE != kUpdate) ptx::prefetch_tmap(&P.cls[c].tmMir);
      }
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int half = static_cast<int>(rank) * (kBM / 2);
      for (int t = pair; ok && t < P.total_tiles; t += npairs) {
        const Tile tl = decode_tile<MODE>(P, t);
        const GemmClass& C = P.cls[tl.cls];
        int kb0, kb1;
        k_range<MODE>(C, tl, kKB, &kb0, &kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          const long long w0 = prof ? clock64() : 0;
          if (!ptx::mbar_wait(ptx::smem_addr(&empty[stage]), phase ^ 1, budget, abort)) {
            raise_timeout(P, abort);
            ok = false;
            break;
          }
          if (prof) prof[kWpProducerEmpty] += clock64() - w0;
          // debug build: every copy's inner coordinate is a whole number of
          // 16-byte units and non-negative (an unaligned one faults)
          if (!MUON_CHECK(kb * kKB >= 0 && (kb * kKB) % 8 == 0 && (tl.I * kBM + half) % 8 == 0 &&
                          (tl.J * kBN + half) % 8 == 0)) {
            raise_timeout(P, abort);
            ok = false;
            break;
          }
          const uint32_t fb = ptx::map_to_rank(ptx::smem_addr(&full[stage]), 0);
          const uint32_t sa = ptx::smem_addr(smem + stage * kStageBytes);
          const uint32_t sb = sa + kStageA;
          if (rank == 0) ptx::mbar_arrive_expect_tx(ptx::smem_addr(&full[stage]), 2 * kStageBytes);
          // A and B are stored as their 256 x 256 blocks on and above the
          // diagonal: an operand block below it is read as the transpose of
          // the stored block (MN-major, two 64 x 64 boxes)
          const int jb = kb * kBK / kBN;  // block column of this k block
          // an MN-major half of A read transposed (128 columns = two 64-column
          // atoms): one 4-D copy where the map exists, else two 3-D copies
          auto load_t = [&](uint32_t dst, int col) {
            if (C.t4) {
              ptx::tma_load_4d_pair(dst, &C.tmT4, fb, 0, kb * kBK, col / 64, tl.idx);
            } else {
#pragma unroll
              for (int j = 0; j < 2; ++j)
                ptx::tma_load_3d_pair(dst + j * (64 * kBK * 2), &C.tmT, fb, col + 64 * j, kb * kBK, tl.idx);
            }
          };
          if ((MODE == kPoly || MODE == kUpdate) && SYM && jb < tl.I) {
            load_t(sa, tl.I * kBM + half);
          } else {
            ptx::tma_load_3d_pair(sa, &C.tmA, fb, kb * kKB, tl.I * kBM + half, tl.idx);
          }
          if (MODE == kUpdate) {
#pragma unroll
            for (int j = 0; j < (kBN / 2) / 64; ++j)
              ptx::tma_load_3d_pair(sb + j * (64 * kBK * 2), &C.tmB, fb, tl.J * kBN + half + 64 * j, kb * kBK,
                                    tl.idx);
          } else if (MODE == kPoly && SYM && jb < tl.J) {
            load_t(sb, tl.J * kBN + half);
          } else {
            ptx::tma_load_3d_pair(sb, &C.tmB, fb, kb * kKB, tl.J * kBN + half, tl.idx);
          }
          if (++stage == kSt) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0 && !P.inject_stall) {
      // ---------------------------------------------------------- MMA issuer
      // instruction descriptors by operand major-ness (A, B): K-major, or
      // MN-major for transposed reads of blocks below the diagonal
      constexpr uint32_t idesc_kk = ptx::idesc_bf16(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_km = ptx::idesc_bf16(kBM, kBN, 0, 1);
      constexpr uint32_t idesc_mk = ptx::idesc_bf16(kBM, kBN, 1, 0);
      constexpr uint32_t idesc_mm = ptx::idesc_bf16(kBM, kBN, 1, 1);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      const long long loop0 = prof ? clock64() : 0;
      for (int t = pair; ok && t < P.total_tiles; t += npairs, ++it) {
        const Tile tl = decode_tile<MODE>(P, t);
        const GemmClass& C = P.cls[tl.cls];
        int kb0, kb1;
        k_range<MODE>(C, tl, kKB, &kb0, &kb1);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        const long long w1 = prof ? clock64() : 0;
        if (!ptx::mbar_wait_cluster(ptx::smem_addr(&tempty[acc]), acc_phase ^ 1, budget, abort)) {
          raise_timeout(P, abort);
          break;
        }
        if (prof) prof[kWpMmaTempty] += clock64() - w1;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + acc * kBN;
        // One K block: its stage's operands are waited for, then its four
        // MMAs issue back to back.  Everything they take is formed before
        // the wait.  A descriptor's low 14 bits are the operand address / 16,
        // so the k-th MMA's descriptor is the first one plus k steps: 32
        // bytes (16 K elements of a 128-byte row) K-major, 2048 bytes (16 rows
        // of 128 bytes) MN-major.  Shared addresses stay below 2^18, so the
        // sum never carries out of the field.
        auto kblock = [&](int st, uint32_t ph, int kb) -> bool {
          const uint32_t sa = ptx::smem_addr(smem + st * kStageBytes);
          const uint32_t sb = sa + kStageA;
          const int jb = kb * kBK / kBN;
          const bool a_mn = (MODE == kPoly || MODE == kUpdate) && SYM && jb < tl.I;
          const bool b_mn = MODE == kUpdate || (MODE == kPoly && SYM && jb < tl.J);
          const uint32_t idesc =
              MODE == kFp8 ? P.idesc_f8 : (a_mn ? (b_mn ? idesc_mm : idesc_mk) : (b_mn ? idesc_km : idesc_kk));
          const uint64_t a0 = a_mn ? ptx::sdesc_sw128(sa, 64 * kBK * 2, 1024) : ptx::sdesc_sw128(sa, 16, 1024);
          const uint64_t b0 = b_mn ? ptx::sdesc_sw128(sb, 64 * kBK * 2, 1024) : ptx::sdesc_sw128(sb, 16, 1024);
          const uint64_t astep = a_mn ? 2048 / 16 : 32 / 16;
          const uint64_t bstep = b_mn ? 2048 / 16 : 32 / 16;
          const uint32_t acc0 = kb != kb0 ? 1u : 0u;
          const long long w2 = prof ? clock64() : 0;
          if (!ptx::mbar_wait(ptx::smem_addr(&full[st]), ph, budget, abort)) return false;
          if (prof) prof[kWpMmaFull] += clock64() - w2;
          ptx::tc_fence_after();
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            if (MODE == kFp8)
              ptx::mma_f8_pair(d, a0 + k * astep, b0 + k * bstep, idesc, k == 0 ? acc0 : 1u);
            else
              ptx::mma_bf16_pair(d, a0 + k * astep, b0 + k * bstep, idesc, k == 0 ? acc0 : 1u);
          }
          return true;
        };
        // Each stage is released as soon as its MMAs are issued (the commit
        // arrives once they have completed).  Releasing stages in pairs after
        // eight MMAs issues the MMAs with fewer pauses, but it holds every
        // first stage of a pair for four more MMAs, and the operand ring then
        // runs dry more often: measured slower on every phase.
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!kblock(stage, phase, kb)) {
            raise_timeout(P, abort);
            ok = false;
            break;
          }
          ptx::mma_commit_pair_mc(ptx::smem_addr(&empty[stage]), 0x3);
          if (++stage == kSt) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_mc(ptx::smem_addr(&tfull[acc]), 0x3);
      }
      // wait until every MMA issued here has completed
      ptx::mma_commit_pair(ptx::smem_addr(drain));
      ptx::mbar_wait(ptx::smem_addr(drain), 0, budget, never);
      if (prof) prof[kWpMmaLoop] += clock64() - loop0;
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // This CTA's TMEM lanes hold rows 128*rank .. 128*rank+127 of the 256-row
    // tile.  Warp w (2..9) reads lane quarter w % 4 (32 rows) and column half
    // (w - 2) / 4 (4 chunks of 32 columns).  The tile's 128 x 256 bf16 block
    // goes through the staging buffer: the epilogue input (A or X) arrives
    // there by TMA, each thread reads its row's 16-byte pieces and writes the
    // result in place.  Every warp works alone: its 32 rows of each of its
    // two 64-column boxes form a TMA box of their own (32 rows of 128 bytes,
    // 1 KB aligned, so the swizzle phase is that of the full box), which
    // lane 0 stores as soon as the warp has written it (the first store
    // overlaps the second box) and reloads for the warp's next tile once the
    // store has read it, on the warp's own input barrier.  No barrier spans
    // warps.
    // The layout is TMA's 128-byte swizzle: boxes of 64 columns, rows of
    // 128 bytes, 16-byte piece j of row r at piece (j ^ (r % 8)).
    const int q = warp & 3;
    const int colhalf = (warp - 2) >> 2;
    const int row_local = q * 32 + lane;  // 0 .. 127 within this CTA's rows
    const bool elected = warp == 2 && lane == 0;  // diagnostics
    uint64_t* my_aux = &aux_full[warp - 2];
    const uint32_t my_rows = static_cast<uint32_t>(q * kEpiRows * 128);  // this warp's rows within a box
    const uint32_t stg_a = ptx::smem_addr(stg);
    const uint32_t tempty_leader[2] = {ptx::map_to_rank(ptx::smem_addr(&tempty[0]), 0),
                                       ptx::map_to_rank(ptx::smem_addr(&tempty[1]), 0)};
    const int rowoff = static_cast<int>(rank) * (kBM / 2);
    auto load_aux = [&](int t) {  // this warp's rows of its two boxes of tile t's epilogue input
      const Tile tn = decode_tile<MODE>(P, t);
      const GemmClass& Cn = P.cls[tn.cls];
      ptx::mbar_arrive_expect_tx(ptx::smem_addr(my_aux), 2 * kEpiRows * 128);
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const int bx = 2 * colhalf + bb;
        ptx::tma_load_3d(stg_a + bx * (kBM / 2) * 128 + my_rows, &Cn.tmAux, ptx::smem_addr(my_aux),
                         tn.J * kBN + 64 * bx, tn.I * kBM + rowoff + q * kEpiRows, tn.idx);
      }
    };
    auto store_box = [&](const GemmClass& C, const Tile& tl, int bx) {
      const int sbx = kSmallStg ? colhalf : bx;
      if (!MUON_CHECK(tl.J * kBN + 64 * bx >= 0 && (tl.J * kBN + 64 * bx) % 8 == 0 && tl.I >= 0)) return;
      ptx::tma_store_3d(&C.tmOut, stg_a + sbx * (kBM / 2) * 128 + my_rows, tl.J * kBN + 64 * bx,
                        tl.I * kBM + rowoff + q * kEpiRows, tl.idx);
      ptx::bulk_commit();
    };
    // p <- p - lr X' for this warp's 32 rows of box bx (64 columns of X'),
    // p stored like X (R = m rows of n): the rounded X' is read back from the
    // staging tile, half a warp per row and 4 columns (16 bytes of p) per
    // lane, all 16 of a lane's loads in flight before its stores
    auto apply_box = [&](const GemmClass& C, const Tile& tl, float* pm, int bx) {
      __syncwarp();
      const uint32_t box = stg_a + bx * ((kBM / 2) * 128);
      const int cl = (lane & 15) * 4;
      const int cg = tl.J * kBN + 64 * bx + cl;
      const bool vec = (C.n & 3) == 0;  // rows 16-byte aligned
      {
        float pv[16][4];
        uint32_t xv[16][2];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int rl = q * kEpiRows + 2 * k + (lane >> 4);
          const int r = tl.I * kBM + rowoff + rl;
          ptx::lds64(box + rl * 128 + (((cl >> 3) ^ (rl & 7)) << 4) + (cl & 7) * 2, xv[k][0], xv[k][1]);
          const float* pp = pm + static_cast<long long>(r) * C.n + cg;
          if (r < C.m && vec && cg < C.n) {
            const float4 f = *reinterpret_cast<const float4*>(pp);
            pv[k][0] = f.x;
            pv[k][1] = f.y;
            pv[k][2] = f.z;
            pv[k][3] = f.w;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) pv[k][e] = (r < C.m && cg + e < C.n) ? pp[e] : 0.0f;
          }
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int rl = q * kEpiRows + 2 * k + (lane >> 4);
          const int r = tl.I * kBM + rowoff + rl;
          float o[4] = {word_lo(xv[k][0]), word_hi(xv[k][0]), word_lo(xv[k][1]), word_hi(xv[k][1])};
#pragma unroll
          for (int e = 0; e < 4; ++e) o[e] = fmaf(-P.lr, o[e], pv[k][e]);
          float* pp = pm + static_cast<long long>(r) * C.n + cg;
          if (r < C.m && vec && cg < C.n) {
            *reinterpret_cast<float4*>(pp) = make_float4(o[0], o[1], o[2], o[3]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (r < C.m && cg + e < C.n) pp[e] = o[e];
          }
        }
      }
    };
    // APPLY 2: the parameter block of chunk ch (32 columns of X') of tile t
    // moves through slot ch % 2 of this warp as one 32 x 32 fp32 TMA box of
    // the matrix's own tensor map (128-byte swizzle; clipped or zero-filled
    // at the matrix edge): p's rows are X' rows (wide and square matrices)
    // or X' columns (tall ones, p = X'^T).  The block of the next chunk (of
    // the next tile after a tile's last chunk) is loaded while a chunk is
    // applied.
    constexpr bool bulkp = MODE == kUpdate && APPLY == 2;
    const uint32_t pslot0 = ptx::smem_addr(pslots) + static_cast<uint32_t>((warp - 2) * 2 * kPSlot);
    uint32_t p_phase[2] = {0u, 0u};
    bool p_pending[2] = {false, false};
    // box coordinates (x: column, y: row of p) of a chunk's block
    auto p_xy = [&](const Tile& tn, int tall, int ch, int* x, int* y) {
      const int r0 = tn.I * kBM + rowoff + q * kEpiRows;
      const int c0 = tn.J * kBN + colhalf * (kBN / 2) + ch * 32;
      *x = tall ? r0 : c0;
      *y = tall ? c0 : r0;
    };
    auto p_map = [&](const GemmClass& Cn, const Tile& tn) -> const CUtensorMap* {
      if constexpr (APPLY == 2) return &P.pmap[Cn.mat_begin + tn.idx];
      return nullptr;
    };
    auto p_load = [&](int t, int ch, int sl) {  // lane 0
      const Tile tn = decode_tile<MODE>(P, t);
      const GemmClass& Cn = P.cls[tn.cls];
      int x, y;
      p_xy(tn, P.table[Cn.mat_begin + tn.idx].tall, ch, &x, &y);
      const uint32_t bar = ptx::smem_addr(&pfull[(warp - 2) * 2 + sl]);
      // debug build: fp32 boxes start on 4-element columns (16 bytes); the
      // block is then skipped and its wait expires (bounded)
      if (!MUON_CHECK(x >= 0 && y >= 0 && x % 4 == 0)) return;
      ptx::mbar_arrive_expect_tx(bar, kPSlot);
      ptx::tma_load_2d(pslot0 + sl * kPSlot, p_map(Cn, tn), bar, x, y);
    };
    if (bulkp && pair < P.total_tiles) {
      if (lane == 0) p_load(pair, 0, 0);
      p_pending[0] = true;
    }
    if (!kNoAux && lane == 0 && pair < P.total_tiles) load_aux(pair);
    uint32_t aux_phase = 0;
    bool ok = true;
    int it = 0;
    for (int t = pair; t < P.total_tiles; t += npairs, ++it) {
      const Tile tl = decode_tile<MODE>(P, t);
      const GemmClass& C = P.cls[tl.cls];
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      // the Muon step's last update: p <- p - lr X' instead of storing X'
      constexpr bool fuse = MODE == kUpdate && APPLY;
      float* pm = nullptr;
      bool ptall = false;
      if (fuse) {
        const MatInfo& mi = P.table[C.mat_begin + tl.idx];
        pm = static_cast<float*>(mi.out);
        ptall = mi.tall != 0;
        // debug build: the parameter recorded for this matrix has the class's shape
        if (!MUON_CHECK(ptall ? (mi.C == C.m && mi.R == C.n) : (mi.R == C.m && mi.C == C.n))) pm = nullptr;
      }
      if (!kNoAux) {
        if (!ptx::mbar_wait(ptx::smem_addr(my_aux), aux_phase, budget, abort)) {
          raise_timeout(P, abort);
          ok = false;
        }
        aux_phase ^= 1;
      }
      const long long w3 = (prof && elected) ? clock64() : 0;
      if (ok && !ptx::mbar_wait(ptx::smem_addr(&tfull[acc]), acc_phase, budget, abort)) {
        raise_timeout(P, abort);
        ok = false;
      }
      // the warp's lanes agree on leaving (warp-level syncs follow)
      if (__any_sync(0xFFFFFFFFu, !ok || *abort)) break;
      const long long w4 = (prof && elected) ? clock64() : 0;
      if (prof && elected) prof[kWpEpiTfull] += w4 - w3;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN + colhalf * (kBN / 2);
      uint32_t w[4][16];  // the rounded tile, kept for the mirrored writes
      // the accumulator's 4 chunks of 32 columns are read one chunk ahead:
      // chunk ch + 1's TMEM load is in flight while chunk ch is processed
      // (except in the register-path parameter update, whose registers are
      // too many to keep a load in flight safely: there each chunk's load is
      // waited for at once)
      constexpr bool kPipeTmem = !(MODE == kUpdate && APPLY == 1);
      uint32_t rbuf[2][32];
      __syncwarp();
      if (kPipeTmem) ptx::tmem_ld32(tb, rbuf[0]);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int c0 = colhalf * (kBN / 2) + ch * 32;  // column within the tile
        // tall p (Muon step's last update): p = X'^T, n rows of m.  For X
        // column c the warp's 32 rows are 32 consecutive floats of p's row c,
        // one coalesced 128-byte access; the chunk's loads are issued before
        // its accumulator columns are read
        float pv[32];
        float* pc = nullptr;
        const int rt = tl.I * kBM + rowoff + row_local;
        const int ct = tl.J * kBN + c0;
        if (MODE == kUpdate && fuse && ptall && !bulkp && pm) {
          pc = pm + static_cast<long long>(ct) * C.m + rt;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            pv[j] = (rt < C.m && ct + j < C.n) ? pc[static_cast<long long>(j) * C.m] : 0.0f;
        }
        uint32_t(&r)[32] = rbuf[ch & 1];
        if (!kPipeTmem) {
          __syncwarp();
          ptx::tmem_ld32(tb + ch * 32, r);
        }
        ptx::tmem_ld_wait(r);
        if (ch == 3) {
          // every column of the accumulator has been read: the MMA warp may
          // reuse it
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_cluster(tempty_leader[acc]);
        } else if (kPipeTmem) {
          __syncwarp();
          ptx::tmem_ld32(tb + (ch + 1) * 32, rbuf[(ch + 1) & 1]);
        }
        // staging box: the tile's 64-column box, or (Gram) the warp's one box
        const int sbx = kSmallStg ? colhalf : (c0 >> 6);
        const uint32_t rowa = stg_a + sbx * ((kBM / 2) * 128) + row_local * 128;
        if (MODE == kFp8 && C.ksplit > 1) {
          // a slice of a split contraction: the fp32 partial sums of these
          // 32 columns (128 bytes per row) fill the warp's 32 x 128-byte
          // slot as one fp32 box, stored to the slice's plane of the
          // partial-sum array once the previous chunk's box has been read
          // (two slots per warp, used in turn: a slot is rewritten once the
          // store two chunks back -- possibly of the previous tile -- has
          // read it)
          const uint32_t fslot = stg_a + (2 * colhalf + (ch & 1)) * ((kBM / 2) * 128);
          if (lane == 0) ptx::bulk_wait_read1();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            ptx::sts128(fslot + row_local * 128 + ((j ^ (row_local & 7)) << 4), r[4 * j], r[4 * j + 1], r[4 * j + 2],
                        r[4 * j + 3]);
          ptx::fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&C.tmAux, fslot + my_rows, tl.J * kBN + c0, tl.I * kBM + rowoff + q * kEpiRows,
                              tl.split);
            ptx::bulk_commit();
          }
          continue;
        }
        if (kSmallStg && ch == 2) {
          // the warp's box still holds its first half until the store has read it
          if (lane == 0) ptx::bulk_wait_read0();
          __syncwarp();
        }
        if (MODE == kFp8 && (ch & 1) == 0) {
          // the FP8 product stages no input, so a tile's stores need not be
          // read before the next tile starts: a box is rewritten once its
          // store from the previous tile has read it (one younger store may
          // still be pending)
          if (lane == 0) ptx::bulk_wait_read1();
          __syncwarp();
        }
        const int j0 = (c0 & 63) >> 3;
        uint32_t ow[16];  // this chunk's 32 rounded values (pairs)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t addr = rowa + ((((j0 + jj) ^ (row_local & 7))) << 4);
          float v[8];
          uint32_t wq[4];
          if (kNoAux) {
            // Gram: the product; FP8: the product times x_s w_s
#pragma unroll
            for (int e = 0; e < 8; ++e)
              v[e] = MODE == kFp8 ? C.scale * __uint_as_float(r[8 * jj + e]) : __uint_as_float(r[8 * jj + e]);
          } else {
            uint32_t x[4];
            ptx::lds128(addr, x[0], x[1], x[2], x[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = word_lo(x[e]), hi = word_hi(x[e]);
              const float a0 = __uint_as_float(r[8 * jj + 2 * e]), a1 = __uint_as_float(r[8 * jj + 2 * e + 1]);
              if (MODE == kPoly) {
                v[2 * e] = fmaf(P.cb, lo, P.cc * a0);      // b A + c (A A)
                v[2 * e + 1] = fmaf(P.cb, hi, P.cc * a1);
              } else {
                v[2 * e] = fmaf(P.ca, lo, a0);             // a X + B X
                v[2 * e + 1] = fmaf(P.ca, hi, a1);
              }
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            wq[e] = ow[4 * jj + e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
            if (MODE != kUpdate) w[ch][4 * jj + e] = wq[e];
          }
          if (!(fuse && ptall)) ptx::sts128(addr, wq[0], wq[1], wq[2], wq[3]);
        }
        if (bulkp) {
          // the other slot (its last store has read it) takes the next
          // chunk's block
          {
            const int nt = ch < 3 ? t : t + npairs;
            if (__all_sync(0xFFFFFFFFu, nt < P.total_tiles && !*abort)) {
              if (lane == 0) {
                ptx::bulk_wait_read0();
                p_load(nt, (ch + 1) & 3, (ch + 1) & 1);
              }
              p_pending[(ch + 1) & 1] = true;
              __syncwarp();
            }
          }
          // p <- p - lr X' on this chunk's block in shared memory, then back
          const int sl = ch & 1;
          const uint32_t slot = pslot0 + sl * kPSlot;
          if (ptx::mbar_wait(ptx::smem_addr(&pfull[(warp - 2) * 2 + sl]), p_phase[sl], budget, abort)) {
            p_phase[sl] ^= 1;
            p_pending[sl] = false;
          } else {
            raise_timeout(P, abort);  // the block may still land: waited for at the end
          }
          __syncwarp();  // (wide) every lane's X' row is staged
          if (!ptall) {
            // 8 lanes per block row, 4 columns (16 bytes of p, 8 of X') each
            const int colin = (c0 & 63) + (lane & 7) * 4;  // column within the 64-column box
            const uint32_t box = stg_a + (c0 >> 6) * ((kBM / 2) * 128);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int br = 4 * k + (lane >> 3);  // block row
              const int rl = q * kEpiRows + br;
              uint32_t x0, x1;
              ptx::lds64(box + rl * 128 + (((colin >> 3) ^ (rl & 7)) << 4) + (colin & 7) * 2, x0, x1);
              float4 pv4;
              const uint32_t pa = slot + br * 128 + (((lane & 7) ^ (br & 7)) << 4);
              ptx::lds128f(pa, pv4);
              pv4.x = fmaf(-P.lr, word_lo(x0), pv4.x);
              pv4.y = fmaf(-P.lr, word_hi(x0), pv4.y);
              pv4.z = fmaf(-P.lr, word_lo(x1), pv4.z);
              pv4.w = fmaf(-P.lr, word_hi(x1), pv4.w);
              ptx::sts128f(pa, pv4);
            }
          } else {
            // block row j is X' column c0 + j; this lane's X' row is its column
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const uint32_t pa = slot + j * 128 + (((lane >> 2) ^ (j & 7)) << 4) + (lane & 3) * 4;
              float pvj;
              ptx::lds32(pa, pvj);
              ptx::sts32(pa, fmaf(-P.lr, (j & 1) ? word_hi(ow[j >> 1]) : word_lo(ow[j >> 1]), pvj));
            }
          }
          ptx::fence_async_smem();
          __syncwarp();
          if (lane == 0 && !*abort) {
            int x, y;
            p_xy(tl, ptall, ch, &x, &y);
            if (MUON_CHECK(x >= 0 && y >= 0 && x % 4 == 0)) ptx::tma_store_2d(p_map(C, tl), slot, x, y);
            ptx::bulk_commit();
          }
        }
        if (MODE == kUpdate && fuse && ptall && !bulkp && pm) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float o = (j & 1) ? word_hi(ow[j >> 1]) : word_lo(ow[j >> 1]);
            if (rt < C.m && ct + j < C.n) pc[static_cast<long long>(j) * C.m] = fmaf(-P.lr, o, pv[j]);
          }
        }
        if (ch & 1) {
          // this warp's rows of box 2*colhalf + ch/2 are written: store them
          // (or apply them to p)
          if (MODE == kUpdate && fuse) {
            if (!ptall && !bulkp && pm) apply_box(C, tl, pm, 2 * colhalf + (ch >> 1));
          } else {
            ptx::fence_async_smem();
            __syncwarp();
            if (lane == 0) store_box(C, tl, 2 * colhalf + (ch >> 1));
          }
        }
      }
      if ((MODE == kPoly || MODE == kGram) && !SYM && tl.I != tl.J) {
        // A and B of wide matrices are stored whole: the mirrored entries
        // (r, c) -> (c, r) of the warp's 32 rows go through its first staging
        // slot transposed, 64 columns at a time: row c of the slot holds the
        // 32 values of column c (64 bytes, unswizzled, one store instruction
        // for the warp), and one TMA box of 64 rows c by 32 columns r takes
        // them out (clipped at the matrix edge)
        const uint32_t slot = stg_a + (MODE == kGram ? colhalf : 2 * colhalf) * ((kBM / 2) * 128) + my_rows;
        const int r0 = tl.I * kBM + rowoff + q * kEpiRows;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (lane == 0) ptx::bulk_wait_read0();  // the slot's last store has read it
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int ch = 2 * h + (c >> 5), j = c & 31;
            ptx::sts16(slot + c * 64 + lane * 2, static_cast<uint16_t>(w[ch][j >> 1] >> (16 * (j & 1))));
          }
          ptx::fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&C.tmMir, slot, r0, tl.J * kBN + colhalf * (kBN / 2) + 64 * h, tl.idx);
            ptx::bulk_commit();
          }
        }
      }
      if (MODE == kUpdate && fuse) {
        // the staging rows were read with ordinary loads: order those reads
        // before the copy of the next input tile overwrites them
        ptx::fence_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        if (MODE != kFp8) ptx::bulk_wait_read0();  // this warp's rows are free again
        if (!kNoAux && t + npairs < P.total_tiles) {
          ptx::fence_async_smem();
          load_aux(t + npairs);
        }
      }
      __syncwarp();
      if (prof && elected) {
        prof[kWpEpiBusy] += clock64() - w4;
        prof[kWpTiles] += 1;
      }
    }
    if (lane == 0) ptx::bulk_wait0();
    if (!kNoAux && lane == 0 && *abort) {
      // an input tile may still be in flight
      ptx::mbar_wait(ptx::smem_addr(my_aux), aux_phase, budget, never);
    }
    if (bulkp && *abort) {
      // so may parameter blocks
#pragma unroll
      for (int sl = 0; sl < 2; ++sl)
        if (p_pending[sl] && lane == 0)
          ptx::mbar_wait(ptx::smem_addr(&pfull[(warp - 2) * 2 + sl]), p_phase[sl], budget, never);
    }
  }

  ptx::tc_fence_before();
  if (*abort) {
    // give copies this CTA issued before giving up time to land
    const long long t0 = clock64();
    while (clock64() - t0 < 200000) {
    }
  }
  __syncwarp();
  ptx::cluster_sync();
  if (prof && threadIdx.x == 0) prof[kWpKernel] += clock64() - t_start;
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, 512);
  }
}

template __global__ void ns_gemm_kernel<kGram, 0, 0>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kGram, 1, 0>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kPoly, 0, 0>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kPoly, 1, 0>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kUpdate, 0, 0>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kUpdate, 0, 1>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kUpdate, 1, 0>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kUpdate, 1, 1>(const __grid_constant__ GemmParams P);
template __global__ void ns_gemm_kernel<kUpdate, 0, 2>(const __grid_constant__ GemmParamsP P);
template __global__ void ns_gemm_kernel<kUpdate, 1, 2>(const __grid_constant__ GemmParamsP P);
template __global__ void ns_gemm_kernel<kFp8, 0, 0>(const __grid_constant__ GemmParams P);

// ------------------------------------------------------------------ launcher
namespace {

// The kernel instantiation of a (mode, variant) and its shared memory.
// Variant bit 0: A (and B) stored block-upper (Gram, polynomial, update);
// variant / 2: the update with the parameter update (1: from registers, 2:
// streamed through shared memory).  FP8: 0.
const void* gemm_fn(int mode, int variant, int* smem) {
  switch (mode) {
    case kGram:
      *smem = GemmShape<kGram>::smem;
      return variant & 1 ? reinterpret_cast<const void*>(&ns_gemm_kernel<kGram, 1, 0>)
                         : reinterpret_cast<const void*>(&ns_gemm_kernel<kGram, 0, 0>);
    case kPoly:
      *smem = GemmShape<kPoly>::smem;
      return variant & 1 ? reinterpret_cast<const void*>(&ns_gemm_kernel<kPoly, 1, 0>)
                         : reinterpret_cast<const void*>(&ns_gemm_kernel<kPoly, 0, 0>);
    case kUpdate:
      *smem = variant >= 4 ? GemmShape<kUpdate, 2>::smem : GemmShape<kUpdate>::smem;
      switch (variant) {
        case 0: return reinterpret_cast<const void*>(&ns_gemm_kernel<kUpdate, 0, 0>);
        case 1: return reinterpret_cast<const void*>(&ns_gemm_kernel<kUpdate, 1, 0>);
        case 2: return reinterpret_cast<const void*>(&ns_gemm_kernel<kUpdate, 0, 1>);
        case 3: return reinterpret_cast<const void*>(&ns_gemm_kernel<kUpdate, 1, 1>);
        case 4: return reinterpret_cast<const void*>(&ns_gemm_kernel<kUpdate, 0, 2>);
        default: return reinterpret_cast<const void*>(&ns_gemm_kernel<kUpdate, 1, 2>);
      }
    default:
      *smem = GemmShape<kFp8>::smem;
      return reinterpret_cast<const void*>(&ns_gemm_kernel<kFp8, 0, 0>);
  }
}

void gemm_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], int smem, cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg = {};
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

constexpr int kMaxGemmDevices = 64;
constexpr int kGemmSlots = 32;  // mode * 8 + variant
std::mutex g_pairs_mu;
int g_max_pairs[kMaxGemmDevices][kGemmSlots] = {};

}  // namespace

// CTA pairs of a (mode, variant) kernel that can be resident at once on the
// current device, at most num_sms / 2.  The first query per device and
// kernel also raises the kernel's dynamic shared-memory limit there; both
// are kept per device.  Enqueues nothing.
cudaError_t ns_gemm_pairs(int mode, int variant, int num_sms, int* pairs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxGemmDevices) return cudaErrorInvalidDevice;
  const int slot = mode * 8 + variant;
  std::lock_guard<std::mutex> lk(g_pairs_mu);
  int& n = g_max_pairs[dev][slot];
  if (n <= 0) {
    int smem = 0;
    const void* fn = gemm_fn(mode, variant, &smem);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    gemm_config(cfg, attr, smem, nullptr);
    cfg.gridDim = dim3(num_sms);
    int q = 0;
    e = cudaOccupancyMaxActiveClusters(&q, fn, &cfg);
    if (e != cudaSuccess) return e;
    n = q > 0 ? q : 1;
  }
  *pairs = n < num_sms / 2 ? n : num_sms / 2;
  return cudaSuccess;
}

// Clusters of two CTAs (one pair per cluster), persistent: `pairs` pairs
// (from ns_gemm_pairs), at most one per tile.
cudaError_t launch_ns_gemm(int mode, int variant, const GemmParams& P, int pairs, cudaStream_t stream) {
  int smem = 0;
  const void* fn = gemm_fn(mode, variant, &smem);
  if (P.total_tiles < pairs) pairs = P.total_tiles;
  if (pairs <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  gemm_config(cfg, attr, smem, stream);
  cfg.gridDim = dim3(2 * pairs);
  cfg.numAttrs = 2;
  void* args[] = {const_cast<GemmParams*>(&P)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

MUON_CHECK_READER(check_failures_gemm)

}  // namespace muon
