// Internal launch-parameter structures shared by the host planner
// (muon_capi.cu) and the kernels (elementwise.cu, ns_gemm.cu).
//
// A bank of matrices is grouped into shape classes (m, n) with m = min(R, C)
// and n = max(R, C): after the momentum pass every matrix of a class is held
// in the workspace as X (m x n, bf16, row-major, row pitch ldx), tall matrices
// already transposed.  The Newton-Schulz kernels iterate over all tiles of
// all classes in one persistent launch per phase.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace muon {

constexpr int kMaxClasses = 8;     // shape classes per launch
constexpr int kK1MaxMats = 96;     // matrices per momentum-pass launch
constexpr int kTallCols = 256;  // momentum pass: a tall matrix's block is 64 rows x 256 columns

// device status word bits (kept in the workspace header)
constexpr int kStatusNonFinite = 1;
constexpr int kStatusTimeout = 2;

enum GemmMode { kGram = 0, kPoly = 1, kUpdate = 2, kFp8 = 3 };  // kFp8: out = s * (A B^T), E4M3 operands
enum FinalMode { kFinalNone = 0, kFinalParam = 1, kFinalOut = 2 };

// One row per matrix of the bank; written by the momentum pass into the
// workspace, read by the normalise pass and the last B*X launch.
struct MatInfo {
  void* out;        // fp32 param (Muon step) or bf16 O (Newton-Schulz only)
  int R, C;         // stored shape
  int tall;         // R > C: X = u^T
  int part_off;     // first partial sum of this matrix
  int nparts;       // number of partial sums
  int pad;
};

// ---------------------------------------------------------------- momentum
struct K1Mat {
  const void* g;      // gradient (or G), R x C, row-major
  float* buf;         // momentum buffer (null: no momentum, u = g)
  void* out;          // recorded in MatInfo
  __nv_bfloat16* x;   // X destination in the workspace
  int R, C, ldx;
  int tall;
  int g_f32;          // 1: g is float32, 0: bfloat16
  int rows_per_block; // wide: rows per block; tall: 64
  int part_off;       // first partial of this matrix
  int nparts;
  int table_index;    // global matrix index in the MatInfo table
  int pad;
};

struct K1Params {
  K1Mat mats[kK1MaxMats];
  int block_begin[kK1MaxMats + 1];
  int n;
  float mu;
  int nesterov;
  float* partials;
  MatInfo* table;
};

// ---------------------------------------------------------------- normalise
struct NormClass {
  __nv_bfloat16* x;   // class region, count x m x ldx
  int count, m, n, ldx;
  int mat_begin;      // first global matrix index of the class
  int rows_per_block;
  int blocks_per_mat;
  int block_begin;
};

struct NormParams {
  NormClass cls[kMaxClasses];
  int n_classes;
  const float* partials;
  const MatInfo* table;
  int* status;
};

// ---------------------------------------------------------------- FP8
// Operands of the FP8 scaled product: q = E4M3(bf16(src / scale)) for two
// contiguous bf16 tensors (x and w), 8 elements per thread.
struct Fp8QuantParams {
  const __nv_bfloat16* src[2];
  uint8_t* dst[2];
  long long n[2];
  float scale[2];
  float inv_scale[2];  // 1 / scale rounded to float (fast path of the quotient)
  long long blocks0;   // blocks of tensor 0; the rest quantise tensor 1
};
constexpr int kQuantVecs = 4;  // 8-element vectors per thread, all in flight
constexpr int kQuantPerBlock = 256 * 8 * kQuantVecs;

// Operands of the FP8 product's backward (page section "自定义FP8矩阵乘法实现",
// "反向传播优化"): per job, a rows x cols source in 128 x 128 tiles, written
// transposed (cols x rows one-byte codes) and, for the gradient, also
// row-major.  A gradient job quantises: code = E5M2(bf16(src / scale)); the
// other jobs copy E4M3 codes.
struct Fp8TJob {
  const void* src;    // rows x cols: bf16 (quant) or one-byte codes
  uint8_t* dst;       // rows x cols codes (quant jobs), else null
  uint8_t* dst_t;     // cols x rows codes
  int rows, cols;     // multiples of 16
  int quant;          // 1: bf16 source quantised to E5M2
  float scale, inv_scale;
  int tiles_c;        // 128-column tiles across
  int tile_begin;     // first block of this job
  int pad;
};
constexpr int kFp8TJobs = 3;
constexpr int kFp8Tile = 128;
struct Fp8TParams {
  Fp8TJob job[kFp8TJobs];
  int n_jobs;
};

// Split-K reduction of an FP8 product: out = bf16(scale * sum over the
// splits of part[split]) in a fixed order.
struct Fp8ReduceParams {
  const float* part;  // splits x n fp32
  __nv_bfloat16* out; // n
  long long n;        // a multiple of 4
  int splits;
  float scale;
};

// ---------------------------------------------------------------- GEMMs
struct GemmClass {
  CUtensorMap tmA;              // operand A (K-major rows, box 64 x 128)
  CUtensorMap tmB;              // operand B (Gram/poly: K-major box 64 x 128;
                                //            update: MN-major box 64 x 64)
  CUtensorMap tmAux;            // epilogue input tile (A or X_t), box 64 x 128
  CUtensorMap tmOut;            // output tile, box 64 x 128
  CUtensorMap tmT;              // poly: A's stored blocks read transposed
                                //   (MN-major, box 64 x 64)
  CUtensorMap tmT4;             // the same as 4-D (64 columns, rows, 64-column
                                //   chunk, matrix): both atoms in one copy
  CUtensorMap tmMir;            // Gram (wide A) / poly: the output's mirrored
                                //   entries, box 32 x 64, unswizzled
  int m, n, count, K;
  int tiles_m, tiles_n, tiles_per_mat;
  int tile_begin;
  int mat_begin;
  int t4;                       // 1: tmT4 is valid (width a multiple of 64)
  int ksplit;                   // kFp8: the contraction is split in this
                                //   many slices, each tile writing fp32
                                //   partial sums through tmAux (1: none)
  float scale;                  // kFp8: the product's scale
};

struct GemmParams {
  GemmClass cls[kMaxClasses];
  int n_classes;
  int total_tiles;
  float ca, cb, cc;             // Newton-Schulz coefficients
  int* status;
  long long wait_budget;        // clock64 cycles per barrier wait
  int inject_stall;             // test hook: MMA warp issues nothing
  uint32_t idesc_f8;            // kFp8: instruction descriptor (operand formats)
  long long* wait_profile;      // diagnostics: kWaitCounters per CTA, or null
  const MatInfo* table;         // update of the Muon step's last iteration:
  float lr;                     //   the matrices' parameters and the rate
  int apply;                    // 1: the epilogue applies p <- p - lr X' (fp32,
                                //   in p's own layout) instead of storing X'
  int reverse;                  // 1: the tile list is walked from its end
};

// The Muon step's last update with the parameters streamed through shared
// memory (APPLY 2): one 2-D fp32 tensor map per matrix of the launch, in
// class order, over the parameter in its own layout (box 32 x 32, 128-byte
// swizzle).  Kernel parameters are limited to 32 KB, which bounds the
// number of matrices; larger banks take the register path.
constexpr int kMaxPMaps = 190;
struct GemmParamsP : GemmParams {
  CUtensorMap pmap[kMaxPMaps];
};
static_assert(sizeof(GemmParamsP) <= 32764, "kernel parameters are limited to 32764 bytes");
template <int APPLY>
struct GemmParamsOf {
  using type = GemmParams;
};
template <>
struct GemmParamsOf<2> {
  using type = GemmParamsP;
};

// diagnostics counters per CTA (clock64 cycles unless noted)
enum WaitCounter {
  kWpProducerEmpty = 0,  // producer waiting for a free stage
  kWpMmaFull,            // MMA issuer waiting for operands
  kWpMmaTempty,          // MMA issuer waiting for a drained accumulator
  kWpEpiTfull,           // epilogue (warp 2) waiting for an accumulator
  kWpEpiBusy,            // epilogue (warp 2) working on tiles
  kWpKernel,             // thread 0: whole kernel
  kWpTiles,              // tiles processed (count)
  kWpMmaLoop,            // MMA issuer: whole loop
  kWaitCounters
};

// ---------------------------------------------------------------- apply
// Final pass: O = X (transposed back for tall matrices); the Muon step
// applies p <- p - lr * O, Newton-Schulz alone writes O.  64 x 64 tiles of X.
struct ApplyClass {
  const __nv_bfloat16* x;  // final X buffer of the class, count x m x ldx
  int count, m, n, ldx;
  int mat_begin;
  int tiles_m, tiles_n;    // 64 x 64 tiles per matrix
  int tile_begin;
};

struct ApplyParams {
  ApplyClass cls[kMaxClasses];
  int n_classes;
  int final_mode;          // kFinalParam or kFinalOut
  float lr;
  const MatInfo* table;
};

// tile sizes of the tcgen05 kernels: a CTA pair computes a kBM x kBN tile,
// each CTA holding half of the A rows and half of the B columns
constexpr int kBM = 256;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 5;
constexpr int kStageA = (kBM / 2) * kBK * 2;  // 16 KB
constexpr int kStageB = (kBN / 2) * kBK * 2;  // 16 KB
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kStageOut = (kBM / 2) * kBN * 2;  // 64 KB epilogue staging

// Shared-memory shape per phase.  A Gram tile has no epilogue input, so its
// staging holds one 64 x 32 box per warp (32 KB, reused for the warp's second
// box once the first has been stored) and the space freed is a sixth operand
// stage; the polynomial and update tiles stage the input next to the output.
// The FP8 product's tiles are short (6 K blocks at K = 768), so its warps
// stage both their boxes at once and it keeps five stages.
// Gram / poly: the largest m for which A is stored as its blocks on and above
// the diagonal only, the polynomial reading the others transposed.  Transposed
// reads walk 64 rows per K block; for wider matrices their lost locality costs
// the polynomial more than the Gram's mirrored writes cost (measured on
// 768-, 1024-, 1600- and 4096-wide banks).
constexpr int kSymUpperMaxM = 768;

//
// The Muon step's last update (APPLY 2) streams the parameters through
// shared memory: every epilogue warp owns two slots of 32 rows x 32 fp32
// (4 KB) for the parameter blocks of its next chunks; the operand ring
// gives up two stages for them (that launch is bound by its 8 bytes of
// parameter traffic per element, not by the MMAs).
constexpr int kEpiWarps = 8;     // two warps per TMEM lane quarter, one per column half
constexpr int kEpiRows = 32;     // rows of an epilogue staging box: one warp's TMEM lane quarter
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr int kPSlot = 32 * 32 * 4;  // one parameter block: 32 rows of 128 bytes
constexpr int kGemmBarBytes = 512;   // mbarriers and flags

template <int MODE, int APPLY = 0>
struct GemmShape {
  static constexpr int stages = MODE == kGram ? kStages + 1 : (APPLY == 2 ? kStages - 2 : kStages);
  static constexpr int staging = MODE == kGram ? kStageOut / 2 : kStageOut;
  static constexpr int pslots = APPLY == 2 ? kEpiWarps * 2 * kPSlot : 0;
  static constexpr int smem = stages * kStageBytes + staging + pslots + 1024 /*align*/ + kGemmBarBytes;
};

}  // namespace muon
