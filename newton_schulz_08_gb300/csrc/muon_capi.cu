// C ABI of libmuon.so (declared in include/muon.h): argument checks, the bank
// planner (shape classes, workspace layout, tile lists), TMA descriptor
// encoding and the launch sequence of one Muon step / one Newton-Schulz call.
//
// Launch sequence (all on the caller's stream, nothing synchronises):
//   memset(status word)
//   momentum_cast      1 launch per 96 matrices: momentum, bf16 cast,
//                      transpose of tall matrices, partial norms
//   normalise          1 launch: X0 = bf16(Xraw / (||Xraw||_F + 1e-7))
//   ns_steps x { Gram, Poly, Update }   1 persistent launch each for the
//                      whole bank (per group of <= 8 shape classes); in the
//                      Muon step the last Update also applies p <- p - lr O
//   apply              Newton-Schulz alone (or a step with no iteration):
//                      1 launch, O = final X transposed back for tall
//                      matrices written (or p <- p - lr O)
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <initializer_list>
#include <list>
#include <memory>
#include <mutex>
#include <vector>

#include "../../include/muon.h"
#include "check.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace muon {

cudaError_t ns_gemm_pairs(int mode, int variant, int num_sms, int* pairs);
cudaError_t launch_ns_gemm(int mode, int variant, const GemmParams& P, int pairs, cudaStream_t stream);
cudaError_t launch_momentum_cast(const K1Params& P, int blocks, cudaStream_t stream);
cudaError_t launch_normalise(const NormParams& P, int blocks, cudaStream_t stream);
cudaError_t launch_apply(const ApplyParams& P, int blocks, cudaStream_t stream);
cudaError_t launch_fp8_quantize(const Fp8QuantParams& P, int blocks, cudaStream_t stream);
cudaError_t launch_fp8_transpose(const Fp8TParams& P, int blocks, cudaStream_t stream);
cudaError_t launch_fp8_reduce(const Fp8ReduceParams& P, int blocks, cudaStream_t stream);

namespace {

// Newton-Schulz coefficients (a, b, c), section "Newton-Schulz正交化".
constexpr float kCoefA = 3.4445f;
constexpr float kCoefB = -4.7750f;
constexpr float kCoefC = 2.0315f;

constexpr size_t kAlign = 1024;
constexpr int kElemsPerBlock = 16384;  // elementwise passes: ~16K elements per block

std::atomic<long long> g_wait_budget{4000000000LL};
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_record_events{0};
std::atomic<long long> g_wait_profile{0};  // device address of the counters, 0: off
std::atomic<int> g_fail_encode{0};         // test hook: every tensor-map encode fails

// Optional CUDA-event brackets around every launch (diagnostics).
// kinds: 0 momentum_cast, 1 normalise, 2 gram, 3 poly, 4 update, 5 apply,
// 6 the Muon step's last update (p <- p - lr O applied in its epilogue),
// 7 fp8_quantize, 8 the FP8 scaled product
struct EventPair {
  cudaEvent_t start, stop;
  int kind;
};
std::mutex g_ev_mu;
std::vector<EventPair> g_ev_pending;
std::vector<EventPair> g_ev_pool;

bool ev_begin(EventPair& e, int kind, cudaStream_t s) {
  if (!g_record_events.load()) return false;
  {
    std::lock_guard<std::mutex> lk(g_ev_mu);
    if (!g_ev_pool.empty()) {
      e = g_ev_pool.back();
      g_ev_pool.pop_back();
    } else {
      if (cudaEventCreate(&e.start) != cudaSuccess) return false;
      if (cudaEventCreate(&e.stop) != cudaSuccess) return false;
    }
  }
  e.kind = kind;
  return cudaEventRecord(e.start, s) == cudaSuccess;
}

void ev_end(EventPair& e, bool active, cudaStream_t s) {
  if (!active) return;
  cudaEventRecord(e.stop, s);
  std::lock_guard<std::mutex> lk(g_ev_mu);
  g_ev_pending.push_back(e);
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// One matrix of a job, whatever the entry point.
struct JobMat {
  const void* g;
  int g_f32;
  float* buf;   // null: no momentum
  void* out;    // param (fp32) or O (bf16)
  long long R, C;
};

struct ClassPlan {
  int m, n, count;
  int ldx, lda;
  size_t x_off[2], a_off, b_off;
  int mat_begin;  // position in class order
  int norm_rpb, norm_blocks;
};

struct Plan {
  std::vector<ClassPlan> cls;
  std::vector<int> order;  // class order -> job index
  std::vector<int> part_off, nparts, k1_rpb;
  size_t parts_off = 0, table_off = 0, total = 0;
  int total_parts = 0;
};

bool build_plan(const std::vector<JobMat>& mats, Plan& P) {
  const int N = static_cast<int>(mats.size());
  std::vector<int> cls_of(N);
  for (int i = 0; i < N; ++i) {
    const long long m = std::min(mats[i].R, mats[i].C), n = std::max(mats[i].R, mats[i].C);
    int c = -1;
    for (size_t k = 0; k < P.cls.size(); ++k)
      if (P.cls[k].m == m && P.cls[k].n == n) c = static_cast<int>(k);
    if (c < 0) {
      ClassPlan cp{};
      cp.m = static_cast<int>(m);
      cp.n = static_cast<int>(n);
      cp.count = 0;
      P.cls.push_back(cp);
      c = static_cast<int>(P.cls.size()) - 1;
    }
    cls_of[i] = c;
    P.cls[c].count++;
  }
  for (size_t c = 0; c < P.cls.size(); ++c) {
    P.cls[c].mat_begin = static_cast<int>(P.order.size());
    for (int i = 0; i < N; ++i)
      if (cls_of[i] == static_cast<int>(c)) P.order.push_back(i);
  }
  // partial sums of the momentum pass
  P.part_off.resize(N);
  P.nparts.resize(N);
  P.k1_rpb.resize(N);
  int parts = 0;
  for (int k = 0; k < N; ++k) {
    const JobMat& M = mats[P.order[k]];
    int rpb, blocks;
    if (M.R > M.C) {
      rpb = 64;
      blocks = static_cast<int>(ceil_div(M.R, 64) * ceil_div(M.C, kTallCols));
    } else {
      rpb = static_cast<int>(std::max<long long>(1, kElemsPerBlock / M.C));
      blocks = static_cast<int>(ceil_div(M.R, rpb));
    }
    P.k1_rpb[k] = rpb;
    P.part_off[k] = parts;
    P.nparts[k] = blocks;
    if (parts > INT_MAX - blocks) return false;
    parts += blocks;
  }
  P.total_parts = parts;
  size_t off = 256;  // header: status word
  P.parts_off = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(parts), kAlign);
  P.table_off = off;
  off = align_up(off + sizeof(MatInfo) * static_cast<size_t>(N), kAlign);
  for (ClassPlan& cp : P.cls) {
    cp.ldx = static_cast<int>(align_up(cp.n, 8));
    cp.lda = static_cast<int>(align_up(cp.m, 8));
    const size_t xb = sizeof(__nv_bfloat16) * static_cast<size_t>(cp.count) * cp.m * cp.ldx;
    const size_t ab = sizeof(__nv_bfloat16) * static_cast<size_t>(cp.count) * cp.m * cp.lda;
    cp.x_off[0] = off;
    off = align_up(off + xb, kAlign);
    cp.x_off[1] = off;
    off = align_up(off + xb, kAlign);
    cp.a_off = off;
    off = align_up(off + ab, kAlign);
    cp.b_off = off;
    off = align_up(off + ab, kAlign);
    cp.norm_rpb = static_cast<int>(std::max(1, kElemsPerBlock / cp.n));
    cp.norm_blocks = static_cast<int>(ceil_div(cp.m, cp.norm_rpb));
  }
  P.total = off;
  return true;
}

// ------------------------------------------------------------------- checks
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;
  bool written;
};

bool ranges_overlap(std::vector<Range>& r) {
  std::sort(r.begin(), r.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
  uintptr_t max_all = 0, max_written = 0;
  for (const Range& x : r) {
    if (x.lo < max_written) return true;
    if (x.written && x.lo < max_all) return true;
    max_all = std::max(max_all, x.hi);
    if (x.written) max_written = std::max(max_written, x.hi);
  }
  return false;
}

muon_status_t check_shapes(long long R, long long C) {
  if (R <= 0 || C <= 0) return MUON_ERR_INVALID_ARG;
  if (R > INT_MAX || C > INT_MAX) return MUON_ERR_TOO_LARGE;
  // per-matrix element counts and tile indices stay within int / TMA limits
  if (R * C > (1LL << 40)) return MUON_ERR_TOO_LARGE;
  const long long m = std::min(R, C);
  if (ceil_div(m, kBM) * ceil_div(std::max(R, C), kBN) > (1LL << 24)) return MUON_ERR_TOO_LARGE;
  return MUON_OK;
}

// ----------------------------------------------------------------- devices
struct DeviceInfo {
  int ok = -1;  // -1 unknown, 0 unsupported, 1 sm_103
  int sms = 0;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

muon_status_t current_device(int& sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (dev < 0 || dev >= 64) return MUON_ERR_UNSUPPORTED_DEVICE;
  DeviceInfo& d = g_dev[dev];
  if (d.ok < 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MUON_ERR_CUDA;
    d.ok = (major == 10 && minor == 3) ? 1 : 0;
    d.sms = n;
  }
  if (d.ok != 1) return MUON_ERR_UNSUPPORTED_DEVICE;
  sms = d.sms;
  return MUON_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 map over `count` matrices of rows x cols (row pitch `pitch`).
bool encode_map(CUtensorMap* map, void* base, int cols, int rows, int count, int pitch, int box_cols,
                int box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = tensor_map_encoder();
  if (!enc || g_fail_encode.load()) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(count)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch) * 2,
                           static_cast<cuuint64_t>(pitch) * 2 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D one-byte map over one rows x cols matrix (row pitch `pitch` bytes),
// 128-byte swizzle: the FP8 operands.
bool encode_map_u8(CUtensorMap* map, void* base, long long cols, long long rows, long long pitch, int box_cols,
                   int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc || g_fail_encode.load()) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch), static_cast<cuuint64_t>(pitch) * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D bf16 map viewing the columns of `count` matrices of rows x cols (row
// pitch `pitch`) as 64-column chunks: dims (64, rows, cols / 64, count),
// box (64, 64, 2, 1).  A copy brings two 64-column swizzle atoms of 64 rows,
// one after the other, as an MN-major operand needs them.  Only for cols a
// multiple of 64 (a chunk never reaches past a row).
bool encode_map4(CUtensorMap* map, void* base, int cols, int rows, int count, int pitch) {
  auto enc = tensor_map_encoder();
  if (!enc || cols % 64 != 0 || g_fail_encode.load()) return false;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64),
                        static_cast<cuuint64_t>(count)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(pitch) * 2, 128,
                           static_cast<cuuint64_t>(pitch) * 2 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[4] = {64, 64, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 map over one rows x cols row-major matrix, box 32 x 32 with
// 128-byte swizzle: a parameter matrix streamed by the last update.
bool encode_map_f32_2d(CUtensorMap* map, void* base, long long cols, long long rows) {
  auto enc = tensor_map_encoder();
  if (!enc || g_fail_encode.load()) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// square kBM x kBN tiles on and above the diagonal
int sym_tiles_per_mat(int m) {
  const int tn = static_cast<int>(ceil_div(m, kBN));
  return tn * (tn + 1) / 2;
}

// ------------------------------------------------------------- prepared call
// Everything a call enqueues, computed before the first enqueue: launch
// parameters with every tensor map encoded, grid sizes, and the order.  The
// per-call scalars (lr, momentum, Nesterov flag) and the diagnostic knobs
// are patched into a copy at enqueue time, so a prepared call depends only
// on the device, the entry point, the pointers and shapes, ns_steps and the
// workspace address.
enum LaunchType { kLMomentum = 0, kLNorm, kLGemm, kLApply };

struct LaunchRec {
  int type;     // LaunchType
  int ev_kind;  // kernel kind for the event brackets
  int grid;     // blocks (elementwise passes) or CTA pairs (GEMMs)
  int mode, variant;
  int index;    // into the typed parameter vector
};

struct Prepared {
  size_t ws_total = 0;
  std::vector<K1Params> k1;
  std::vector<NormParams> norm;
  std::vector<GemmParams> gemm;
  std::vector<GemmParamsP> gemm_p;  // launches that stream the parameters
  std::vector<ApplyParams> apply;
  std::vector<LaunchRec> seq;
};

muon_status_t prepare(const std::vector<JobMat>& mats, const Plan& P, int ns_steps, int final_mode, char* ws,
                      int sms, Prepared& Q) {
  const int N = static_cast<int>(mats.size());
  Q.ws_total = P.total;
  float* partials = reinterpret_cast<float*>(ws + P.parts_off);
  MatInfo* table = reinterpret_cast<MatInfo*>(ws + P.table_off);
  int* status = reinterpret_cast<int*>(ws);

  // momentum + cast (+ transpose) + partial norms
  for (int k0 = 0; k0 < N; k0 += kK1MaxMats) {
    K1Params kp;
    std::memset(&kp, 0, sizeof(kp));
    const int n = std::min(kK1MaxMats, N - k0);
    int blocks = 0;
    for (int j = 0; j < n; ++j) {
      const int k = k0 + j;
      const JobMat& M = mats[P.order[k]];
      int c = 0;
      while (!(k >= P.cls[c].mat_begin && k < P.cls[c].mat_begin + P.cls[c].count)) ++c;
      const ClassPlan& cp = P.cls[c];
      K1Mat& km = kp.mats[j];
      km.g = M.g;
      km.buf = M.buf;
      km.out = M.out;
      km.x = reinterpret_cast<__nv_bfloat16*>(ws + cp.x_off[0]) +
             static_cast<long long>(k - cp.mat_begin) * cp.m * cp.ldx;
      km.R = static_cast<int>(M.R);
      km.C = static_cast<int>(M.C);
      km.ldx = cp.ldx;
      km.tall = M.R > M.C;
      km.g_f32 = M.g_f32;
      km.rows_per_block = P.k1_rpb[k];
      km.part_off = P.part_off[k];
      km.nparts = P.nparts[k];
      km.table_index = k;
      kp.block_begin[j] = blocks;
      blocks += P.nparts[k];
    }
    kp.block_begin[n] = blocks;
    kp.n = n;
    kp.partials = partials;
    kp.table = table;
    Q.seq.push_back({kLMomentum, 0, blocks, 0, 0, static_cast<int>(Q.k1.size())});
    Q.k1.push_back(kp);
  }

  // normalise
  for (size_t c0 = 0; c0 < P.cls.size(); c0 += kMaxClasses) {
    NormParams np;
    std::memset(&np, 0, sizeof(np));
    const int nc = static_cast<int>(std::min<size_t>(kMaxClasses, P.cls.size() - c0));
    int blocks = 0;
    for (int j = 0; j < nc; ++j) {
      const ClassPlan& cp = P.cls[c0 + j];
      NormClass& k = np.cls[j];
      k.x = reinterpret_cast<__nv_bfloat16*>(ws + cp.x_off[0]);
      k.count = cp.count;
      k.m = cp.m;
      k.n = cp.n;
      k.ldx = cp.ldx;
      k.mat_begin = cp.mat_begin;
      k.rows_per_block = cp.norm_rpb;
      k.blocks_per_mat = cp.norm_blocks;
      k.block_begin = blocks;
      blocks += cp.norm_blocks * cp.count;
    }
    np.n_classes = nc;
    np.partials = partials;
    np.table = table;
    np.status = status;
    Q.seq.push_back({kLNorm, 1, blocks, 0, 0, static_cast<int>(Q.norm.size())});
    Q.norm.push_back(np);
  }

  // Newton-Schulz steps
  for (int t = 0; t < ns_steps; ++t) {
    const int src = t & 1, dst = src ^ 1;
    for (size_t c0 = 0; c0 < P.cls.size(); c0 += kMaxClasses) {
      const int nc = static_cast<int>(std::min<size_t>(kMaxClasses, P.cls.size() - c0));
      // classes whose A and B are stored block-upper (m up to kSymUpperMaxM)
      // and the others go to separate kernel instantiations
      for (int mode = kGram; mode <= kUpdate; ++mode) {
        for (int sym = 0; sym <= 1; ++sym) {
          GemmParams gp;
          std::memset(&gp, 0, sizeof(gp));
          int tiles = 0;
          int ng = 0;
          for (int j = 0; j < nc; ++j) {
            const ClassPlan& cp = P.cls[c0 + j];
            if ((cp.m <= kSymUpperMaxM ? 1 : 0) != sym) continue;
            GemmClass& g = gp.cls[ng++];
            void* xs = ws + cp.x_off[src];
            void* xd = ws + cp.x_off[dst];
            void* A = ws + cp.a_off;
            void* B = ws + cp.b_off;
            bool ok = true;
            // operands: A rows (box 64 x 128 per CTA), B rows or X columns, and
            // the symmetric operand's stored blocks read transposed (64 x 64);
            // epilogue: input and output boxes of one warp (64 x 32)
            if (mode == kGram) {
              ok = encode_map(&g.tmA, xs, cp.n, cp.m, cp.count, cp.ldx, kBK, kBM / 2) &&
                   encode_map(&g.tmB, xs, cp.n, cp.m, cp.count, cp.ldx, kBK, kBN / 2) &&
                   encode_map(&g.tmAux, A, cp.m, cp.m, cp.count, cp.lda, 64, kEpiRows) &&
                   encode_map(&g.tmOut, A, cp.m, cp.m, cp.count, cp.lda, 64, kEpiRows) &&
                   encode_map(&g.tmT, A, cp.m, cp.m, cp.count, cp.lda, 64, kBK);
              g.K = cp.n;
            } else if (mode == kPoly) {
              ok = encode_map(&g.tmA, A, cp.m, cp.m, cp.count, cp.lda, kBK, kBM / 2) &&
                   encode_map(&g.tmB, A, cp.m, cp.m, cp.count, cp.lda, kBK, kBN / 2) &&
                   encode_map(&g.tmAux, A, cp.m, cp.m, cp.count, cp.lda, 64, kEpiRows) &&
                   encode_map(&g.tmOut, B, cp.m, cp.m, cp.count, cp.lda, 64, kEpiRows) &&
                   encode_map(&g.tmT, A, cp.m, cp.m, cp.count, cp.lda, 64, kBK);
              g.K = cp.m;
            } else {
              ok = encode_map(&g.tmA, B, cp.m, cp.m, cp.count, cp.lda, kBK, kBM / 2) &&
                   encode_map(&g.tmB, xs, cp.n, cp.m, cp.count, cp.ldx, 64, kBK) &&
                   encode_map(&g.tmAux, xs, cp.n, cp.m, cp.count, cp.ldx, 64, kEpiRows) &&
                   encode_map(&g.tmOut, xd, cp.n, cp.m, cp.count, cp.ldx, 64, kEpiRows) &&
                   encode_map(&g.tmT, B, cp.m, cp.m, cp.count, cp.lda, 64, kBK);
              g.K = cp.m;
            }
            if (!ok) return MUON_ERR_CUDA;
            // poly / update: one-copy transposed reads of A / B where the
            // width allows
            g.t4 = (mode == kPoly || mode == kUpdate) && sym &&
                   encode_map4(&g.tmT4, mode == kPoly ? A : B, cp.m, cp.m, cp.count, cp.lda);
            // mirrored entries of the Gram (wide A) and the polynomial (B)
            if (mode != kUpdate && !encode_map(&g.tmMir, mode == kGram ? A : B, cp.m, cp.m, cp.count, cp.lda, 32,
                                               64, CU_TENSOR_MAP_SWIZZLE_NONE))
              return MUON_ERR_CUDA;
            g.m = cp.m;
            g.n = cp.n;
            g.count = cp.count;
            g.tiles_m = static_cast<int>(ceil_div(cp.m, kBM));
            if (mode == kUpdate) {
              g.tiles_n = static_cast<int>(ceil_div(cp.n, kBN));
              g.tiles_per_mat = g.tiles_m * g.tiles_n;
            } else {
              g.tiles_n = static_cast<int>(ceil_div(cp.m, kBN));
              g.tiles_per_mat = sym_tiles_per_mat(cp.m);
            }
            g.tile_begin = tiles;
            g.mat_begin = cp.mat_begin;
            tiles += g.tiles_per_mat * cp.count;
          }
          if (ng == 0) continue;
          gp.n_classes = ng;
          gp.total_tiles = tiles;
          gp.ca = kCoefA;
          gp.cb = kCoefB;
          gp.cc = kCoefC;
          gp.status = status;
          // the Muon step's last update applies p -= lr X' itself
          gp.table = table;
          gp.apply = mode == kUpdate && final_mode == kFinalParam && t == ns_steps - 1;
          // the Gram and update launches walk their tiles from the end: more of
          // what the previous launch wrote last is still in L2 when it is read
          // (GPT-2 bank: step 1.300 -> 1.289 ms)
          gp.reverse = mode == kGram || mode == kUpdate;
          // the parameters stream through shared memory as TMA boxes of a
          // tensor map per matrix, when the maps fit in the kernel's
          // parameters and every row of every matrix starts 16-byte aligned
          bool streamed = gp.apply && N <= kMaxPMaps;
          for (int j = 0; j < ng; ++j) streamed = streamed && gp.cls[j].m % 4 == 0 && gp.cls[j].n % 4 == 0;
          const int variant = sym + 2 * (gp.apply ? (streamed ? 2 : 1) : 0);
          int pairs = 0;
          if (ns_gemm_pairs(mode, variant, sms, &pairs) != cudaSuccess) return MUON_ERR_CUDA;
          if (streamed) {
            GemmParamsP pp;
            std::memset(&pp, 0, sizeof(pp));
            static_cast<GemmParams&>(pp) = gp;
            for (int k = 0; k < N; ++k) {
              const JobMat& M = mats[P.order[k]];
              if (!encode_map_f32_2d(&pp.pmap[k], M.out, M.C, M.R)) return MUON_ERR_CUDA;
            }
            Q.seq.push_back({kLGemm, 6, pairs, mode, variant, static_cast<int>(Q.gemm_p.size())});
            Q.gemm_p.push_back(pp);
          } else {
            Q.seq.push_back({kLGemm, gp.apply ? 6 : 2 + mode, pairs, mode, variant, static_cast<int>(Q.gemm.size())});
            Q.gemm.push_back(gp);
          }
        }
      }
    }
  }

  // O = final X (transposed back) written, or, with no Newton-Schulz step,
  // p <- p - lr O (the last update has applied it otherwise)
  if (final_mode == kFinalParam && ns_steps > 0) return MUON_OK;
  const int fin = ns_steps & 1;
  for (size_t c0 = 0; c0 < P.cls.size(); c0 += kMaxClasses) {
    ApplyParams ap;
    std::memset(&ap, 0, sizeof(ap));
    const int nc = static_cast<int>(std::min<size_t>(kMaxClasses, P.cls.size() - c0));
    int blocks = 0;
    for (int j = 0; j < nc; ++j) {
      const ClassPlan& cp = P.cls[c0 + j];
      ApplyClass& k = ap.cls[j];
      k.x = reinterpret_cast<const __nv_bfloat16*>(ws + cp.x_off[fin]);
      k.count = cp.count;
      k.m = cp.m;
      k.n = cp.n;
      k.ldx = cp.ldx;
      k.mat_begin = cp.mat_begin;
      k.tiles_m = static_cast<int>(ceil_div(cp.m, 64));
      k.tiles_n = static_cast<int>(ceil_div(cp.n, 64));
      k.tile_begin = blocks;
      blocks += k.tiles_m * k.tiles_n * cp.count;
    }
    ap.n_classes = nc;
    ap.final_mode = final_mode;
    ap.table = table;
    Q.seq.push_back({kLApply, 5, blocks, 0, 0, static_cast<int>(Q.apply.size())});
    Q.apply.push_back(ap);
  }
  return MUON_OK;
}

// Enqueues a prepared call on `stream`: the status word is cleared, then
// every kernel of the sequence is launched with the call's scalars.
muon_status_t enqueue(const Prepared& Q, char* ws, float lr, float mu, int nesterov, cudaStream_t stream) {
  if (cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return MUON_ERR_CUDA;
  const long long budget = g_wait_budget.load();
  const int stall = g_inject_stall.load();
  long long* prof = reinterpret_cast<long long*>(g_wait_profile.load());
  for (const LaunchRec& L : Q.seq) {
    EventPair ev;
    const bool rec = ev_begin(ev, L.ev_kind, stream);
    cudaError_t e = cudaSuccess;
    if (L.type == kLMomentum) {
      K1Params kp = Q.k1[L.index];
      kp.mu = mu;
      kp.nesterov = nesterov;
      e = launch_momentum_cast(kp, L.grid, stream);
    } else if (L.type == kLNorm) {
      e = launch_normalise(Q.norm[L.index], L.grid, stream);
    } else if (L.type == kLGemm && L.variant >= 4) {
      GemmParamsP gp = Q.gemm_p[L.index];
      gp.lr = lr;
      gp.wait_budget = budget;
      gp.inject_stall = stall;
      gp.wait_profile = prof;
      e = launch_ns_gemm(L.mode, L.variant, gp, L.grid, stream);
    } else if (L.type == kLGemm) {
      GemmParams gp = Q.gemm[L.index];
      gp.lr = lr;
      gp.wait_budget = budget;
      gp.inject_stall = stall;
      gp.wait_profile = prof;
      e = launch_ns_gemm(L.mode, L.variant, gp, L.grid, stream);
    } else {
      ApplyParams ap = Q.apply[L.index];
      ap.lr = lr;
      e = launch_apply(ap, L.grid, stream);
    }
    if (e != cudaSuccess) return MUON_ERR_CUDA;
    ev_end(ev, rec, stream);
  }
  return MUON_OK;
}

// Prepared calls, most recently used first, keyed by the device, the entry
// point and its pointer / shape arguments, ns_steps and the workspace
// address (everything a prepared call depends on).  Host memory only.
constexpr size_t kPlanCacheMax = 32;

struct CacheEntry {
  std::vector<uint64_t> key;
  std::shared_ptr<const Prepared> plan;
};

std::mutex g_cache_mu;
std::list<CacheEntry> g_cache;

std::shared_ptr<const Prepared> cache_find(const std::vector<uint64_t>& key) {
  if (g_fail_encode.load()) return nullptr;
  std::lock_guard<std::mutex> lk(g_cache_mu);
  for (auto it = g_cache.begin(); it != g_cache.end(); ++it) {
    if (it->key == key) {
      g_cache.splice(g_cache.begin(), g_cache, it);
      return g_cache.front().plan;
    }
  }
  return nullptr;
}

void cache_insert(std::vector<uint64_t> key, std::shared_ptr<const Prepared> plan) {
  if (g_fail_encode.load()) return;
  std::lock_guard<std::mutex> lk(g_cache_mu);
  for (auto it = g_cache.begin(); it != g_cache.end(); ++it) {
    if (it->key == key) {
      g_cache.erase(it);
      break;
    }
  }
  g_cache.push_front({std::move(key), std::move(plan)});
  while (g_cache.size() > kPlanCacheMax) g_cache.pop_back();
}

muon_status_t check_common(int ns_steps, void* ws, size_t ws_bytes, size_t need) {
  if (ns_steps < 0) return MUON_ERR_INVALID_ARG;
  if (!ws) return MUON_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MUON_ERR_MISALIGNED;
  if (ws_bytes < need) return MUON_ERR_WORKSPACE_TOO_SMALL;
  return MUON_OK;
}

// Full checks and preparation of a call that was not in the cache; the
// result is cached under `key` once everything has succeeded.
muon_status_t plan_call(const std::vector<JobMat>& mats, std::vector<Range>& ranges, int ns_steps, int final_mode,
                        void* ws, size_t ws_bytes, std::vector<uint64_t> key,
                        std::shared_ptr<const Prepared>& out) {
  Plan P;
  if (!build_plan(mats, P)) return MUON_ERR_TOO_LARGE;
  muon_status_t s = check_common(ns_steps, ws, ws_bytes, P.total);
  if (s != MUON_OK) return s;
  ranges.push_back({reinterpret_cast<uintptr_t>(ws), reinterpret_cast<uintptr_t>(ws) + P.total, true});
  if (ranges_overlap(ranges)) return MUON_ERR_ALIASING;
  int sms = 0;
  s = current_device(sms);
  if (s != MUON_OK) return s;
  auto Q = std::make_shared<Prepared>();
  s = prepare(mats, P, ns_steps, final_mode, static_cast<char*>(ws), sms, *Q);
  if (s != MUON_OK) return s;
  out = Q;
  if (!key.empty()) cache_insert(std::move(key), std::move(Q));
  return MUON_OK;
}

// Cache key: device ordinal, entry point, ns_steps, workspace address, then
// the entry point's own arguments.  Without a current device the key stays
// empty and the call is neither looked up nor cached (the full checks then
// report the call's own error first).
void key_head(std::vector<uint64_t>& key, int entry, int ns_steps, const void* ws) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  key.push_back(static_cast<uint64_t>(dev));
  key.push_back(static_cast<uint64_t>(entry));
  key.push_back(static_cast<uint64_t>(static_cast<int64_t>(ns_steps)));
  key.push_back(reinterpret_cast<uint64_t>(ws));
}

size_t plan_size(const std::vector<JobMat>& mats) {
  Plan P;
  if (!build_plan(mats, P)) return 0;
  return P.total;
}

bool collect_muon(const muon_mat_desc* mats, int n, std::vector<JobMat>& out,
                  std::vector<Range>* ranges, muon_status_t& err) {
  err = MUON_OK;
  for (int i = 0; i < n; ++i) {
    const muon_mat_desc& d = mats[i];
    if (!d.param || !d.grad || !d.buf || d.reserved != 0 ||
        (d.grad_dtype != MUON_BF16 && d.grad_dtype != MUON_F32)) {
      err = MUON_ERR_INVALID_ARG;
      return false;
    }
    err = check_shapes(d.rows, d.cols);
    if (err != MUON_OK) return false;
    if (!aligned16(d.param) || !aligned16(d.grad) || !aligned16(d.buf)) {
      err = MUON_ERR_MISALIGNED;
      return false;
    }
    JobMat j;
    j.g = d.grad;
    j.g_f32 = d.grad_dtype == MUON_F32;
    j.buf = d.buf;
    j.out = d.param;
    j.R = d.rows;
    j.C = d.cols;
    out.push_back(j);
    if (ranges) {
      const uintptr_t e = static_cast<uintptr_t>(d.rows * d.cols);
      const uintptr_t gsz = j.g_f32 ? 4 : 2;
      ranges->push_back({reinterpret_cast<uintptr_t>(d.param), reinterpret_cast<uintptr_t>(d.param) + 4 * e, true});
      ranges->push_back({reinterpret_cast<uintptr_t>(d.buf), reinterpret_cast<uintptr_t>(d.buf) + 4 * e, true});
      ranges->push_back({reinterpret_cast<uintptr_t>(d.grad), reinterpret_cast<uintptr_t>(d.grad) + gsz * e, false});
    }
  }
  return true;
}

// 1 / s rounded to float for the quantise passes' fast quotient, or NaN
// when it is not a normal float (the passes then divide exactly).
float fast_inverse(float s) {
  const float inv = static_cast<float>(1.0 / static_cast<double>(s));
  return std::isnormal(inv) ? inv : NAN;
}

// FP8 backward: the contraction over the M rows (grad_w) is split in this
// many slices when its output has few tiles, so that the product fills the
// GPU; a pure function of the shapes (every slice non-empty).
int fp8_bwd_ksplit(long long M, long long N, long long K) {
  const long long tiles = ceil_div(N, kBN) * ceil_div(K, kBM);
  const long long kblocks = ceil_div(M, 2 * kBK);
  if (tiles >= 64) return 1;
  long long s = std::min<long long>({4, ceil_div(72, tiles), kblocks});
  const long long per = ceil_div(kblocks, s);
  return static_cast<int>(ceil_div(kblocks, per));
}

struct Fp8BwdLayout {
  size_t gT, xT, wT, part, total;
  int ksplit;
};

Fp8BwdLayout fp8_bwd_layout(long long M, long long N, long long K) {
  Fp8BwdLayout L;
  L.ksplit = fp8_bwd_ksplit(M, N, K);
  size_t off = 256;  // status word
  L.gT = off;
  off = align_up(off + static_cast<size_t>(N) * M, kAlign);
  L.xT = off;
  off = align_up(off + static_cast<size_t>(K) * M, kAlign);
  L.wT = off;
  off = align_up(off + static_cast<size_t>(K) * N, kAlign);
  L.part = off;
  if (L.ksplit > 1) off = align_up(off + sizeof(float) * L.ksplit * static_cast<size_t>(N) * K, kAlign);
  L.total = off;
  return L;
}

// 3-D fp32 map over `planes` row-major rows x cols planes (the partial sums
// of a split product), 128-byte swizzle, box 32 x 32.
bool encode_map_f32(CUtensorMap* map, void* base, long long cols, long long rows, int planes) {
  auto enc = tensor_map_encoder();
  if (!enc || g_fail_encode.load()) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 4, static_cast<cuuint64_t>(cols) * 4 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(kEpiRows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One class of an FP8 product: out (rows x cols, bf16) = scale * (A . B^T)
// with A rows x k and B cols x k one-byte codes, K-major.
bool fp8_class(GemmClass& g, void* a, void* b, void* out, long long rows, long long cols, long long k, float scale,
               int ksplit, void* part) {
  if (!encode_map_u8(&g.tmA, a, k, rows, k, 2 * kBK, kBM / 2) || !encode_map_u8(&g.tmB, b, k, cols, k, 2 * kBK, kBN / 2) ||
      !encode_map(&g.tmOut, out, static_cast<int>(cols), static_cast<int>(rows), 1, static_cast<int>(cols), 64,
                  kEpiRows))
    return false;
  g.tmAux = g.tmT = g.tmT4 = g.tmMir = g.tmOut;
  if (ksplit > 1 && !encode_map_f32(&g.tmAux, part, cols, rows, ksplit)) return false;
  g.m = static_cast<int>(rows);
  g.n = static_cast<int>(cols);
  g.count = 1;
  g.K = static_cast<int>(k);
  g.tiles_m = static_cast<int>(ceil_div(rows, kBM));
  g.tiles_n = static_cast<int>(ceil_div(cols, kBN));
  g.ksplit = ksplit;
  g.tiles_per_mat = g.tiles_m * g.tiles_n * ksplit;
  g.scale = scale;
  g.mat_begin = 0;
  return true;
}

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" {

size_t muon_workspace_size(const muon_mat_desc* mats, int n_mats) {
  if (n_mats <= 0 || !mats) return 0;
  std::vector<JobMat> v;
  muon_status_t err;
  // shapes only: pointers may still be unset when sizing
  for (int i = 0; i < n_mats; ++i) {
    if (check_shapes(mats[i].rows, mats[i].cols) != MUON_OK) return 0;
    JobMat j{};
    j.R = mats[i].rows;
    j.C = mats[i].cols;
    v.push_back(j);
  }
  (void)err;
  return plan_size(v);
}

muon_status_t muon_step(const muon_mat_desc* mats, int n_mats, float lr, float momentum, int nesterov,
                        int ns_steps, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_mats == 0) return MUON_OK;
  if (n_mats < 0 || !mats) return MUON_ERR_INVALID_ARG;
  if (nesterov != 0 && nesterov != 1) return MUON_ERR_INVALID_ARG;
  if (ns_steps < 0) return MUON_ERR_INVALID_ARG;
  std::vector<uint64_t> key;
  key.reserve(4 + 6 * static_cast<size_t>(n_mats));
  key_head(key, 0, ns_steps, workspace);
  const bool keyed = !key.empty();
  for (int i = 0; keyed && i < n_mats; ++i) {
    const muon_mat_desc& d = mats[i];
    key.push_back(reinterpret_cast<uint64_t>(d.param));
    key.push_back(reinterpret_cast<uint64_t>(d.grad));
    key.push_back(reinterpret_cast<uint64_t>(d.buf));
    key.push_back(static_cast<uint64_t>(d.rows));
    key.push_back(static_cast<uint64_t>(d.cols));
    key.push_back((static_cast<uint64_t>(static_cast<uint32_t>(d.grad_dtype)) << 32) |
                  static_cast<uint32_t>(d.reserved));
  }
  std::shared_ptr<const Prepared> Q = keyed ? cache_find(key) : nullptr;
  if (!Q) {
    std::vector<JobMat> v;
    std::vector<Range> ranges;
    muon_status_t err;
    if (!collect_muon(mats, n_mats, v, &ranges, err)) return err;
    err = plan_call(v, ranges, ns_steps, kFinalParam, workspace, workspace_bytes, std::move(key), Q);
    if (err != MUON_OK) return err;
  }
  if (workspace_bytes < Q->ws_total) return MUON_ERR_WORKSPACE_TOO_SMALL;
  return enqueue(*Q, static_cast<char*>(workspace), lr, momentum, nesterov, static_cast<cudaStream_t>(stream));
}

size_t ns5_workspace_size(int batch, int64_t rows, int64_t cols) {
  if (batch <= 0 || check_shapes(rows, cols) != MUON_OK) return 0;
  std::vector<JobMat> v(batch);
  for (auto& j : v) j.R = rows, j.C = cols;
  return plan_size(v);
}

muon_status_t ns5(const void* G, int g_dtype, void* O, int batch, int64_t rows, int64_t cols,
                  int ns_steps, void* workspace, size_t workspace_bytes, void* stream) {
  if (batch == 0) return MUON_OK;
  if (batch < 0 || !G || !O) return MUON_ERR_INVALID_ARG;
  if (g_dtype != MUON_BF16 && g_dtype != MUON_F32) return MUON_ERR_INVALID_ARG;
  muon_status_t s = check_shapes(rows, cols);
  if (s != MUON_OK) return s;
  if (!aligned16(G) || !aligned16(O)) return MUON_ERR_MISALIGNED;
  if (ns_steps < 0) return MUON_ERR_INVALID_ARG;
  std::vector<uint64_t> key;
  key_head(key, 1, ns_steps, workspace);
  const bool keyed = !key.empty();
  if (keyed)
    for (uint64_t v : {reinterpret_cast<uint64_t>(G), static_cast<uint64_t>(g_dtype), reinterpret_cast<uint64_t>(O),
                       static_cast<uint64_t>(batch), static_cast<uint64_t>(rows), static_cast<uint64_t>(cols)})
      key.push_back(v);
  std::shared_ptr<const Prepared> Q = keyed ? cache_find(key) : nullptr;
  if (!Q) {
    const long long per = rows * cols;
    const size_t gsz = g_dtype == MUON_F32 ? 4 : 2;
    std::vector<JobMat> v(batch);
    for (int i = 0; i < batch; ++i) {
      v[i].g = static_cast<const char*>(G) + gsz * per * i;
      v[i].g_f32 = g_dtype == MUON_F32;
      v[i].buf = nullptr;
      v[i].out = static_cast<char*>(O) + 2 * per * i;
      v[i].R = rows;
      v[i].C = cols;
    }
    std::vector<Range> ranges = {
        {reinterpret_cast<uintptr_t>(G), reinterpret_cast<uintptr_t>(G) + gsz * per * batch, false},
        {reinterpret_cast<uintptr_t>(O), reinterpret_cast<uintptr_t>(O) + 2 * per * batch, true}};
    s = plan_call(v, ranges, ns_steps, kFinalOut, workspace, workspace_bytes, std::move(key), Q);
    if (s != MUON_OK) return s;
  }
  if (workspace_bytes < Q->ws_total) return MUON_ERR_WORKSPACE_TOO_SMALL;
  return enqueue(*Q, static_cast<char*>(workspace), 0.0f, 0.0f, 0, static_cast<cudaStream_t>(stream));
}

size_t ns5_bank_workspace_size(const int64_t* rows, const int64_t* cols, int n_mats) {
  if (n_mats <= 0 || !rows || !cols) return 0;
  std::vector<JobMat> v(n_mats);
  for (int i = 0; i < n_mats; ++i) {
    if (check_shapes(rows[i], cols[i]) != MUON_OK) return 0;
    v[i].R = rows[i];
    v[i].C = cols[i];
  }
  return plan_size(v);
}

muon_status_t ns5_bank(const void* const* G, const int32_t* g_dtype, void* const* O, const int64_t* rows,
                       const int64_t* cols, int n_mats, int ns_steps, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (n_mats == 0) return MUON_OK;
  if (n_mats < 0 || !G || !g_dtype || !O || !rows || !cols) return MUON_ERR_INVALID_ARG;
  if (ns_steps < 0) return MUON_ERR_INVALID_ARG;
  std::vector<uint64_t> key;
  key.reserve(4 + 5 * static_cast<size_t>(n_mats));
  key_head(key, 2, ns_steps, workspace);
  const bool keyed = !key.empty();
  for (int i = 0; keyed && i < n_mats; ++i) {
    key.push_back(reinterpret_cast<uint64_t>(G[i]));
    key.push_back(static_cast<uint64_t>(static_cast<uint32_t>(g_dtype[i])));
    key.push_back(reinterpret_cast<uint64_t>(O[i]));
    key.push_back(static_cast<uint64_t>(rows[i]));
    key.push_back(static_cast<uint64_t>(cols[i]));
  }
  std::shared_ptr<const Prepared> Q = keyed ? cache_find(key) : nullptr;
  if (!Q) {
    std::vector<JobMat> v(n_mats);
    std::vector<Range> ranges;
    for (int i = 0; i < n_mats; ++i) {
      if (!G[i] || !O[i] || (g_dtype[i] != MUON_BF16 && g_dtype[i] != MUON_F32)) return MUON_ERR_INVALID_ARG;
      muon_status_t s = check_shapes(rows[i], cols[i]);
      if (s != MUON_OK) return s;
      if (!aligned16(G[i]) || !aligned16(O[i])) return MUON_ERR_MISALIGNED;
      const uintptr_t e = static_cast<uintptr_t>(rows[i] * cols[i]);
      v[i].g = G[i];
      v[i].g_f32 = g_dtype[i] == MUON_F32;
      v[i].buf = nullptr;
      v[i].out = O[i];
      v[i].R = rows[i];
      v[i].C = cols[i];
      ranges.push_back({reinterpret_cast<uintptr_t>(G[i]),
                        reinterpret_cast<uintptr_t>(G[i]) + (v[i].g_f32 ? 4 : 2) * e, false});
      ranges.push_back({reinterpret_cast<uintptr_t>(O[i]), reinterpret_cast<uintptr_t>(O[i]) + 2 * e, true});
    }
    muon_status_t s = plan_call(v, ranges, ns_steps, kFinalOut, workspace, workspace_bytes, std::move(key), Q);
    if (s != MUON_OK) return s;
  }
  if (workspace_bytes < Q->ws_total) return MUON_ERR_WORKSPACE_TOO_SMALL;
  return enqueue(*Q, static_cast<char*>(workspace), 0.0f, 0.0f, 0, static_cast<cudaStream_t>(stream));
}

muon_status_t muon_device_status(const void* workspace, void* stream) {
  if (!workspace) return MUON_ERR_INVALID_ARG;
  int v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MUON_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MUON_ERR_CUDA;
  if (v & kStatusTimeout) return MUON_ERR_DEVICE_TIMEOUT;
  if (v & kStatusNonFinite) return MUON_WARN_NONFINITE;
  return MUON_OK;
}

const char* muon_status_str(muon_status_t s) {
  switch (s) {
    case MUON_OK: return "ok";
    case MUON_WARN_NONFINITE: return "warning: a matrix had a non-finite norm";
    case MUON_ERR_INVALID_ARG: return "invalid argument";
    case MUON_ERR_MISALIGNED: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case MUON_ERR_ALIASING: return "operands overlap";
    case MUON_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MUON_ERR_CUDA: return "CUDA runtime error";
    case MUON_ERR_DEVICE_TIMEOUT: return "bounded device wait expired";
    case MUON_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (sm_103)";
    case MUON_ERR_TOO_LARGE: return "dimension too large";
    case MUON_ERR_SCRATCH_LIMIT: return "ns5_noalloc: problem needs more than the 64 MiB static scratch";
  }
  return "unknown status";
}

muon_status_t ns5_workspace_layout(int batch, int64_t rows, int64_t cols, muon_ws_layout* out) {
  if (!out || batch <= 0) return MUON_ERR_INVALID_ARG;
  muon_status_t s = check_shapes(rows, cols);
  if (s != MUON_OK) return s;
  std::vector<JobMat> v(batch);
  for (auto& j : v) j.R = rows, j.C = cols;
  Plan P;
  if (!build_plan(v, P)) return MUON_ERR_TOO_LARGE;
  const ClassPlan& c = P.cls[0];
  out->x_offset[0] = c.x_off[0];
  out->x_offset[1] = c.x_off[1];
  out->a_offset = c.a_off;
  out->b_offset = c.b_off;
  out->ldx = c.ldx;
  out->lda = c.lda;
  out->m = c.m;
  out->n = c.n;
  return MUON_OK;
}

int muon_set_debug(const char* key, long long value) {
  if (!key) return -1;
  if (!std::strcmp(key, "wait_budget_cycles")) {
    g_wait_budget.store(value > 0 ? value : 1);
    return 0;
  }
  if (!std::strcmp(key, "inject_stall")) {
    g_inject_stall.store(value ? 1 : 0);
    return 0;
  }
  if (!std::strcmp(key, "wait_profile_buffer")) {
    g_wait_profile.store(value);
    return 0;
  }
  if (!std::strcmp(key, "record_kernel_events")) {
    g_record_events.store(value ? 1 : 0);
    return 0;
  }
  if (!std::strcmp(key, "fail_tensor_map_encode")) {
    g_fail_encode.store(value ? 1 : 0);
    return 0;
  }
  return -1;
}

int muon_debug_check_failures(long long* failures) {
  if (!failures) return -1;
  *failures = 0;
#ifdef MUON_DEBUG
  long long total = 0;
  for (cudaError_t (*f)(int*) : {&check_failures_elementwise, &check_failures_gemm, &check_failures_fp8,
                                 &check_failures_adam}) {
    int v = 0;
    if (f(&v) != cudaSuccess) {
      cudaGetLastError();
      return -2;
    }
    total += v;
  }
  *failures = total;
  return 0;
#else
  return -1;
#endif
}

void muon_plan_cache_clear(void) {
  std::lock_guard<std::mutex> lk(g_cache_mu);
  g_cache.clear();
}

int muon_kernel_times(double* ms, int* launches, int n_kinds) {
  if (!ms || !launches || n_kinds <= 0) return -1;
  for (int k = 0; k < n_kinds; ++k) ms[k] = 0.0, launches[k] = 0;
  std::vector<EventPair> pending;
  {
    std::lock_guard<std::mutex> lk(g_ev_mu);
    pending.swap(g_ev_pending);
  }
  int rc = 0;
  for (EventPair& e : pending) {
    float t = 0.0f;
    if (cudaEventSynchronize(e.stop) != cudaSuccess || cudaEventElapsedTime(&t, e.start, e.stop) != cudaSuccess)
      rc = -1;
    if (e.kind < n_kinds) {
      ms[e.kind] += t;
      launches[e.kind] += 1;
    }
  }
  std::lock_guard<std::mutex> lk(g_ev_mu);
  g_ev_pool.insert(g_ev_pool.end(), pending.begin(), pending.end());
  return rc;
}

// FP8 scaled product (page section "自定义FP8矩阵乘法实现"): x_f8 =
// E4M3(bf16(x / x_s)), w_f8 = E4M3(bf16(w / w_s)), out = bf16(x_s w_s
// (x_f8 . w_f8^T)) with an fp32 accumulator.
muon_status_t fp8_mm(const void* x, const void* w, float x_s, float w_s, void* out, void* x_f8, void* w_f8,
                     int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 0) return MUON_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MUON_OK;
  if (K == 0 || K % 16 != 0 || N % 8 != 0) return MUON_ERR_INVALID_ARG;
  if (!x || !w || !out || !x_f8 || !w_f8 || !workspace) return MUON_ERR_INVALID_ARG;
  if (!(std::isfinite(x_s) && x_s > 0.0f && std::isfinite(w_s) && w_s > 0.0f)) return MUON_ERR_INVALID_ARG;
  if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return MUON_ERR_TOO_LARGE;
  if (M * K > (1LL << 40) || N * K > (1LL << 40) || M * N > (1LL << 40)) return MUON_ERR_TOO_LARGE;
  const long long tm = ceil_div(M, kBM), tn = ceil_div(N, kBN);
  if (tm * tn > (1LL << 24)) return MUON_ERR_TOO_LARGE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(out) || !aligned16(x_f8) || !aligned16(w_f8))
    return MUON_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_ERR_MISALIGNED;
  if (workspace_bytes < 256) return MUON_ERR_WORKSPACE_TOO_SMALL;
  auto at = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
  std::vector<Range> ranges = {{at(x), at(x) + 2 * static_cast<uintptr_t>(M * K), false},
                               {at(w), at(w) + 2 * static_cast<uintptr_t>(N * K), false},
                               {at(out), at(out) + 2 * static_cast<uintptr_t>(M * N), true},
                               {at(x_f8), at(x_f8) + static_cast<uintptr_t>(M * K), true},
                               {at(w_f8), at(w_f8) + static_cast<uintptr_t>(N * K), true},
                               {at(workspace), at(workspace) + 256, true}};
  if (ranges_overlap(ranges)) return MUON_ERR_ALIASING;
  int sms = 0;
  muon_status_t s = current_device(sms);
  if (s != MUON_OK) return s;
  // everything the launches take is prepared before the first enqueue
  GemmParams gp;
  std::memset(&gp, 0, sizeof(gp));
  // the maps other than A, B and out are not read by the FP8 product (only
  // prefetched)
  if (!fp8_class(gp.cls[0], x_f8, w_f8, out, M, N, K,
                 static_cast<float>(static_cast<double>(x_s) * static_cast<double>(w_s)), 1, nullptr))
    return MUON_ERR_CUDA;
  gp.n_classes = 1;
  gp.total_tiles = static_cast<int>(tm * tn);
  gp.idesc_f8 = ptx::idesc_f8(kBM, kBN, ptx::kFmtE4M3, ptx::kFmtE4M3);
  gp.status = static_cast<int*>(workspace);
  gp.wait_budget = g_wait_budget.load();
  gp.inject_stall = g_inject_stall.load();
  int pairs = 0;
  if (ns_gemm_pairs(kFp8, 0, sms, &pairs) != cudaSuccess) return MUON_ERR_CUDA;

  Fp8QuantParams q;
  std::memset(&q, 0, sizeof(q));
  q.src[0] = static_cast<const __nv_bfloat16*>(x);
  q.src[1] = static_cast<const __nv_bfloat16*>(w);
  q.dst[0] = static_cast<uint8_t*>(x_f8);
  q.dst[1] = static_cast<uint8_t*>(w_f8);
  q.n[0] = M * K;
  q.n[1] = N * K;
  q.scale[0] = x_s;
  q.scale[1] = w_s;
  q.inv_scale[0] = fast_inverse(x_s);
  q.inv_scale[1] = fast_inverse(w_s);
  q.blocks0 = ceil_div(M * K, kQuantPerBlock);
  const long long qblocks = q.blocks0 + ceil_div(N * K, kQuantPerBlock);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 256, st) != cudaSuccess) return MUON_ERR_CUDA;
  EventPair evq;
  const bool recq = ev_begin(evq, 7, st);
  if (launch_fp8_quantize(q, static_cast<int>(qblocks), st) != cudaSuccess) return MUON_ERR_CUDA;
  ev_end(evq, recq, st);
  EventPair evg;
  const bool recg = ev_begin(evg, 8, st);
  if (launch_ns_gemm(kFp8, 0, gp, pairs, st) != cudaSuccess) return MUON_ERR_CUDA;
  ev_end(evg, recg, st);
  return MUON_OK;
}

size_t fp8_mm_backward_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0 || M % 16 || N % 16 || K % 16) return 0;
  if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return 0;
  if (M == 0 || N == 0 || K == 0) return 256;
  return fp8_bwd_layout(M, N, K).total;
}

// Backward of the FP8 scaled product (page section "自定义FP8矩阵乘法实现",
// "反向传播优化"): g_f8 = E5M2(bf16(g / grad_s)), grad_x = bf16(grad_s w_s
// (g_f8 . w_f8)), grad_w = bf16(grad_s x_s (g_f8^T . x_f8)), fp32 accumulation.
muon_status_t fp8_mm_backward(const void* g, const void* x_f8, const void* w_f8, float x_s, float w_s, float grad_s,
                              void* grad_x, void* grad_w, void* g_f8, int64_t M, int64_t N, int64_t K,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 0) return MUON_ERR_INVALID_ARG;
  if (M % 16 || N % 16 || K % 16) return MUON_ERR_INVALID_ARG;
  if (!g || !x_f8 || !w_f8 || !grad_x || !grad_w || !g_f8 || !workspace) return MUON_ERR_INVALID_ARG;
  for (float v : {x_s, w_s, grad_s})
    if (!(std::isfinite(v) && v > 0.0f)) return MUON_ERR_INVALID_ARG;
  if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return MUON_ERR_TOO_LARGE;
  if (M * K > (1LL << 40) || N * K > (1LL << 40) || M * N > (1LL << 40)) return MUON_ERR_TOO_LARGE;
  if (ceil_div(M, kBM) * ceil_div(K, kBN) + 4 * ceil_div(N, kBM) * ceil_div(K, kBN) > (1LL << 24))
    return MUON_ERR_TOO_LARGE;
  for (const void* p : std::initializer_list<const void*>{g, x_f8, w_f8, grad_x, grad_w, g_f8})
    if (!aligned16(p)) return MUON_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_ERR_MISALIGNED;
  const bool empty = M == 0 || N == 0 || K == 0;
  const Fp8BwdLayout L = empty ? Fp8BwdLayout{256, 256, 256, 256, 256, 1} : fp8_bwd_layout(M, N, K);
  if (workspace_bytes < L.total) return MUON_ERR_WORKSPACE_TOO_SMALL;
  auto at = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
  const uintptr_t mn = static_cast<uintptr_t>(M * N), mk = static_cast<uintptr_t>(M * K),
                  nk = static_cast<uintptr_t>(N * K);
  std::vector<Range> ranges = {{at(g), at(g) + 2 * mn, false},           {at(x_f8), at(x_f8) + mk, false},
                               {at(w_f8), at(w_f8) + nk, false},         {at(grad_x), at(grad_x) + 2 * mk, true},
                               {at(grad_w), at(grad_w) + 2 * nk, true},  {at(g_f8), at(g_f8) + mn, true},
                               {at(workspace), at(workspace) + L.total, true}};
  if (ranges_overlap(ranges)) return MUON_ERR_ALIASING;
  int sms = 0;
  muon_status_t s = current_device(sms);
  if (s != MUON_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (empty) {
    // an empty contraction: the non-empty gradient is zero
    if (cudaMemsetAsync(workspace, 0, 256, st) != cudaSuccess) return MUON_ERR_CUDA;
    if (mk && cudaMemsetAsync(grad_x, 0, 2 * mk, st) != cudaSuccess) return MUON_ERR_CUDA;
    if (nk && cudaMemsetAsync(grad_w, 0, 2 * nk, st) != cudaSuccess) return MUON_ERR_CUDA;
    return MUON_OK;
  }
  char* ws = static_cast<char*>(workspace);
  uint8_t* gT = reinterpret_cast<uint8_t*>(ws + L.gT);
  uint8_t* xT = reinterpret_cast<uint8_t*>(ws + L.xT);
  uint8_t* wT = reinterpret_cast<uint8_t*>(ws + L.wT);
  float* part = reinterpret_cast<float*>(ws + L.part);

  // everything the launches take is prepared before the first enqueue
  Fp8TParams tp;
  std::memset(&tp, 0, sizeof(tp));
  int tblocks = 0;
  auto job = [&](int j, const void* src, uint8_t* dst, uint8_t* dst_t, long long rows, long long cols, int quant) {
    Fp8TJob& J = tp.job[j];
    J.src = src;
    J.dst = dst;
    J.dst_t = dst_t;
    J.rows = static_cast<int>(rows);
    J.cols = static_cast<int>(cols);
    J.quant = quant;
    J.scale = grad_s;
    J.inv_scale = fast_inverse(grad_s);
    J.tiles_c = static_cast<int>(ceil_div(cols, kFp8Tile));
    J.tile_begin = tblocks;
    tblocks += static_cast<int>(ceil_div(rows, kFp8Tile) * J.tiles_c);
  };
  job(0, g, static_cast<uint8_t*>(g_f8), gT, M, N, 1);
  job(1, x_f8, nullptr, xT, M, K, 0);
  job(2, w_f8, nullptr, wT, N, K, 0);
  tp.n_jobs = 3;

  GemmParams gp;
  std::memset(&gp, 0, sizeof(gp));
  // class 0, grad_w (N x K, contraction over M, the long tiles first);
  // class 1, grad_x (M x K, contraction over N)
  const float sw = static_cast<float>(static_cast<double>(grad_s) * static_cast<double>(x_s));
  const float sx = static_cast<float>(static_cast<double>(grad_s) * static_cast<double>(w_s));
  if (!fp8_class(gp.cls[0], gT, xT, grad_w, N, K, M, sw, L.ksplit, part) ||
      !fp8_class(gp.cls[1], g_f8, wT, grad_x, M, K, N, sx, 1, nullptr))
    return MUON_ERR_CUDA;
  gp.cls[0].tile_begin = 0;
  gp.cls[1].tile_begin = gp.cls[0].tiles_per_mat;
  gp.n_classes = 2;
  gp.total_tiles = gp.cls[0].tiles_per_mat + gp.cls[1].tiles_per_mat;
  gp.idesc_f8 = ptx::idesc_f8(kBM, kBN, ptx::kFmtE5M2, ptx::kFmtE4M3);
  gp.status = static_cast<int*>(workspace);
  gp.wait_budget = g_wait_budget.load();
  gp.inject_stall = g_inject_stall.load();
  int pairs = 0;
  if (ns_gemm_pairs(kFp8, 0, sms, &pairs) != cudaSuccess) return MUON_ERR_CUDA;

  Fp8ReduceParams rp;
  rp.part = part;
  rp.out = static_cast<__nv_bfloat16*>(grad_w);
  rp.n = N * K;
  rp.splits = L.ksplit;
  rp.scale = sw;
  const int rblocks = static_cast<int>(ceil_div(N * K, 4 * 256));

  if (cudaMemsetAsync(workspace, 0, 256, st) != cudaSuccess) return MUON_ERR_CUDA;
  EventPair ev;
  bool rec = ev_begin(ev, 9, st);
  if (launch_fp8_transpose(tp, tblocks, st) != cudaSuccess) return MUON_ERR_CUDA;
  ev_end(ev, rec, st);
  rec = ev_begin(ev, 10, st);
  if (launch_ns_gemm(kFp8, 0, gp, pairs, st) != cudaSuccess) return MUON_ERR_CUDA;
  ev_end(ev, rec, st);
  if (L.ksplit > 1) {
    rec = ev_begin(ev, 11, st);
    if (launch_fp8_reduce(rp, rblocks, st) != cudaSuccess) return MUON_ERR_CUDA;
    ev_end(ev, rec, st);
  }
  return MUON_OK;
}

}  // extern "C"
