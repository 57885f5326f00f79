// Internal interfaces between the C ABI (flce_api.cu) and the kernels.
// Host-side only declarations plus the plain-data parameter blocks passed by
// value to the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "flce_math.cuh"
#include "tc_gemm.cuh"

namespace flce {

// CTAs per tensor-core GEMM tile: 2 = CTA pairs (tcgen05.mma.cta_group::2,
// 256-row tiles), 1 = single CTAs (128-row tiles).
constexpr int kPairCG = 2;
constexpr int kTileRowsTC = kBM * kPairCG;
constexpr int kBLoadRowsTC = kBN / kPairCG;

// Tile of the fp32 (FFMA) kernels: kSimtTileN rows x kSimtTileV vocabulary
// columns; the forward statistics of the fp32 path are per kSimtTileV
// columns (the tensor-core path's per kBN), and its grad_bias partials per
// kSimtTileN rows.
constexpr int kSimtTileV = 128;
constexpr int kSimtTileN = 128;

// Input element types of the tensor-core path (FLCE_BF16, FLCE_F16).
enum TcType { kTcBF16 = 1, kTcF16 = 2 };

struct FwdStatsParams {
  const void* bias;           // [V] in the input type, or null
  const int64_t* targets;     // [N]
  float4* partials;           // [N][n_vt] (m, s, t, argmax)
  float* zsum;                // [N][n_vt] sum of the tile's logits (label smoothing) or null
  float* zt;                  // [N] target logit
  int64_t n_rows;             // rows of the buffers
  const int32_t* n_rows_dyn;  // rows actually present (device count) or null
  int64_t v;
  int64_t n_vt;
  int metrics;                // 1: also the argmax and entropy terms (t); 0: (m, s) only
  LogitXform xf;
  int64_t c0;                 // first column of the launch's vocabulary chunk (multiple of 256)
};

// Bytes of one epilogue warp's staging buffer for the D tensor stores: a
// 32 x 32 box of 16-bit values.
constexpr int kDlogitsStageBytes = 32 * 32 * 2;

// The 4-warp forms of the epilogues with per-element arithmetic (both
// forwards, both dlogits) run lane quarters 0 and 1 through the relay of the
// GEMM kernel: their arithmetic then runs on the schedulers that do not issue
// the TMA loads and the MMAs.
constexpr bool kEpiRelay = true;

struct DlogitsParams {
  CUtensorMap d_map;  // D of the chunk [N][width] (pitch ldd), box {32, 32}, for the stores
  // fp32 operands split into bf16 parts: D is stored as its three bf16 parts,
  // d_map taking hi and these mid and lo (same geometry)
  CUtensorMap d_map_x[2];
  const void* bias;
  const int64_t* targets;
  const float* lse;
  const float* grad_out;
  const int32_t* n_valid;
  const float* dscale;  // device scalar multiplying the stored D, or null (1)
  float* gb_partial;  // [m_tiles][gb_ld] or null
  int64_t gb_ld;
  int64_t n_rows;             // rows of the buffers
  const int32_t* n_rows_dyn;  // rows actually present (device count) or null
  int64_t v;
  int64_t ignore_index;
  int c0;     // first vocabulary column of the chunk
  int width;  // columns in the chunk
  int reduction;
  float label_smoothing;
  float z_loss;
  LogitXform xf;
};

// Fused linear KL divergence: forward statistics per (row, vocabulary tile)
// are (m, s, A, Q): the running max and sum e^{z-m} of z, A = sum q (log
// max(q, eps) - z) and Q = sum q over the tile's columns.
struct FwdKLParams {
  const void* bias;
  const void* q;              // [N][V] teacher probabilities, input type
  int q_vec;                  // 1: rows of q are 16-byte aligned (V % 8 == 0)
  const int32_t* row_map;     // original row of each (compacted) row, or null
  float4* partials;
  int64_t n_rows;
  const int32_t* n_rows_dyn;
  int64_t v;
  int64_t n_vt;
  float eps;
  LogitXform xf;              // scale = 1 / temperature
  int64_t c0;                 // first column of the launch's vocabulary chunk (multiple of 256)
};

struct DlogitsKLParams {
  CUtensorMap d_map;  // as in DlogitsParams
  CUtensorMap d_map_x[2];  // as in DlogitsParams
  const void* bias;
  const void* q;
  int q_vec;
  const int32_t* row_map;
  const int64_t* labels;      // of the (compacted) rows, or null: every row counts
  const float* lse;
  const float* qsum;
  const float* grad_out;      // scalar, or per (compacted) row for reduction none
  const int32_t* n_counted;
  const float* dscale;
  float* gb_partial;
  int64_t gb_ld;
  int64_t n_rows;
  const int32_t* n_rows_dyn;
  int64_t v;
  int64_t ignore_index;
  int c0;
  int width;
  int reduction;              // flce_kl_reduction
  LogitXform xf;
};

struct StoreRowsParams {
  void* out;  // input type, or fp32 when out_f32
  int out_f32;
  const float* out_scale;  // device scalar multiplying the results, or null (1)
  int64_t ld;
  int64_t rows;
  int64_t row0;
  int cols;
};

enum AccMode { kAccStore = 0, kAccAdd = 1, kAccAddOut = 2, kAccStoreOut = 3 };

struct AccRowsParams {
  float* acc;
  void* out;  // input type (fp32 when out_f32)
  int out_f32;
  const float* out_scale;  // device scalar multiplying the results, or null (1)
  int mode;
  int64_t ld;
  int64_t rows;
  const int32_t* rows_dyn;  // rows actually present (device count) or null
  const int32_t* row_map;   // output row of each accumulator row, or null (identity)
  int cols;
};

// ---------------------------------------------------------------- launchers
cudaError_t launch_tc_fwd_kl(int type, const CUtensorMap& tm_hidden_k,
                             const CUtensorMap& tm_weight_k, const GemmGeom& g,
                             const FwdKLParams& p, int epi_warps, int sms, cudaStream_t s);
cudaError_t launch_tc_dlogits_kl(int type, const CUtensorMap& tm_hidden_k,
                                 const CUtensorMap& tm_weight_k, const GemmGeom& g,
                                 const DlogitsKLParams& p, int epi_warps, int sms,
                                 cudaStream_t s);

// `type` is a TcType; every launcher runs the CTA-pair GEMM of that type.
// epi_warps (4 or 8): epilogue warps of the forward GEMMs, see fwd_epi_warps;
// with 8 the statistics are kept per 128 columns (fwd_parts_per_tile).
// The forward statistics GEMM over fp32 operands split into three bf16 parts
// (maps [0] hi, [1] mid, [2] lo; g.passes part pairs); the bias is fp32.
cudaError_t launch_tc_fwd_stats_split(const CUtensorMap (&tm_hidden_k)[3],
                                      const CUtensorMap (&tm_weight_k)[3], const GemmGeom& g,
                                      const FwdStatsParams& p, int epi_warps, int sms,
                                      cudaStream_t s);
cudaError_t launch_tc_fwd_stats(int type, const CUtensorMap& tm_hidden_k,
                                const CUtensorMap& tm_weight_k, const GemmGeom& g,
                                const FwdStatsParams& p, int epi_warps, int sms, cudaStream_t s);
// epi_warps (4 or 8): epilogue warps of the dlogits GEMMs, see dlogits_epi_warps.
cudaError_t launch_tc_dlogits(int type, const CUtensorMap& tm_hidden_k,
                              const CUtensorMap& tm_weight_k, const GemmGeom& g,
                              const DlogitsParams& p, int epi_warps, int sms, cudaStream_t s);

// Epilogue warps for the dlogits GEMMs of a contraction of length h. A
// 256 x 256 pair tile's MMAs take time in proportion to h while its epilogue
// (softmax, D, its store and the grad_bias sums) does not; at short h two
// warps per TMEM lane quarter keep the epilogue under the MMAs.
constexpr int64_t kDlogitsEpi8MaxH = 2048;
inline int dlogits_epi_warps(int64_t h) { return h <= kDlogitsEpi8MaxH ? 8 : 4; }
// The forward GEMMs of both losses follow the same rule; their per-row
// statistics are then kept per 128-column half of a 256-column tile. It gains
// the KL forward, whose epilogue also reads a teacher row chunk per 32
// columns, and costs the cross-entropy forward nothing; one rule for both
// keeps their folds identical, so that a one-hot teacher reproduces the
// cross-entropy bitwise.
inline int fwd_epi_warps(int64_t h) { return h <= kDlogitsEpi8MaxH ? 8 : 4; }
inline int64_t fwd_parts_per_tile(int64_t h) { return fwd_epi_warps(h) / 4; }

// Both gradient GEMMs of one vocabulary chunk in one launch, tiles drawn
// from the device counter `sched` (zero before the launch):
//   grad_hidden: A = D (K-major, tm_d_k), B = weight rows (MN-major), AccRows;
//   grad_weight: A = D^T (MN-major, tm_d_mn), B = hidden (MN-major), StoreRows.
// gh_first puts grad_hidden's tiles first (the longer contraction should).
struct GradsLaunch {
  CUtensorMap tm_d_k, tm_weight_mn, tm_d_mn, tm_hidden_mn;
  GemmGeom g_gh, g_gw;
  AccRowsParams ap;
  StoreRowsParams sp;
  int* sched;
  bool gh_first;
};
cudaError_t launch_tc_grads(int type, const GradsLaunch& l, int sms, cudaStream_t s);

// The backward's GEMMs over fp32 operands split into three bf16 parts (maps
// [0] hi, [1] mid, [2] lo; the geometries carry the part pairs): dlogits
// with an fp32 bias, storing D as three bf16 parts (p.d_map, p.d_map_x), and
// the fused gradient launch.
cudaError_t launch_tc_dlogits_split(const CUtensorMap (&tm_hidden_k)[3],
                                    const CUtensorMap (&tm_weight_k)[3], const GemmGeom& g,
                                    const DlogitsParams& p, int epi_warps, int sms,
                                    cudaStream_t s);
struct GradsSplitLaunch {
  CUtensorMap d_k[3], weight_mn[3], d_mn[3], hidden_mn[3];
  GemmGeom g_gh, g_gw;
  AccRowsParams ap;
  StoreRowsParams sp;
  int* sched;
  bool gh_first;
};
cudaError_t launch_tc_grads_split(const GradsSplitLaunch& l, int sms, cudaStream_t s);
// The fused linear KL divergence's forward and dlogits GEMMs over split
// operands (fp32 bias and teacher probabilities).
cudaError_t launch_tc_fwd_kl_split(const CUtensorMap (&tm_hidden_k)[3],
                                   const CUtensorMap (&tm_weight_k)[3], const GemmGeom& g,
                                   const FwdKLParams& p, int epi_warps, int sms, cudaStream_t s);
cudaError_t launch_tc_dlogits_kl_split(const CUtensorMap (&tm_hidden_k)[3],
                                       const CUtensorMap (&tm_weight_k)[3], const GemmGeom& g,
                                       const DlogitsKLParams& p, int epi_warps, int sms,
                                       cudaStream_t s);

// Bounded-wait self-test: result[0] (one CTA) and result[1..2] (a CTA pair).
cudaError_t launch_wait_selftest(int* err_word, uint64_t budget_ns, int* result, cudaStream_t s);

// KL per-row merge and the scalar loss.
struct MergeKLParams {
  const float4* partials;
  const int64_t* labels;  // of the (compacted) rows, or null
  const int32_t* row_map;
  const int32_t* n_dyn;
  int64_t n, n_vt, ignore_index;
  float* loss_rows;
  float* lse_rows;
  float* qsum_rows;
};
cudaError_t launch_merge_kl(const MergeKLParams& p, cudaStream_t s);

struct FinalizeKLParams {
  const float* loss_rows;
  const int64_t* labels;  // original rows, or null
  int64_t n, v, ignore_index;
  int reduction;          // flce_kl_reduction
  float* loss_out;
  int32_t* n_counted;
};
cudaError_t launch_finalize_kl(const FinalizeKLParams& p, cudaStream_t s);

// fp16 backward: D is stored as D * dscale with dscale = 2^k chosen so that
// |D * dscale| < 16384 (the row upstream gradient times logit_scale bounds
// |D|; fp16's largest finite value is 65504) and entries down to ~1e-8 of
// the largest stay normal; out_scale = 1 / dscale exactly. Writes both to
// `scales` [2].
// `reduction` uses the cross-entropy codes (0 none, 1 sum, 2 mean over
// n_valid); `extra_div` further divides the uniform row gradient (V for the
// KL "mean"). With `row_bound` (KL: per-row sum of q), |D| is bounded by the
// row gradient times logit_scale times max row_bound instead of (1 + 2 |z_loss|
// max |lse|). Rows whose target (label) is ignore_index are skipped; targets
// may be null (every row counts).
cudaError_t launch_dlogits_scale(const float* grad_out, const int32_t* n_valid,
                                 const int64_t* targets, int64_t n, int64_t ignore_index,
                                 int reduction, float logit_scale, float z_loss,
                                 const float* lse_rows, const float* row_bound, float extra_div,
                                 float* scales, cudaStream_t s);

// fp32 (SIMT) path
struct SimtFwdParams {
  const float* hidden;
  const float* weight;
  const float* bias;
  const float* q;  // KL: teacher probabilities [N][V]; null for the cross-entropy
  float eps;
  const int64_t* targets;
  float4* partials;
  float* zsum;
  float* zt;
  int64_t n, h, v, n_vt;
  LogitXform xf;
};
cudaError_t launch_simt_fwd(const SimtFwdParams& p, cudaStream_t s);

struct SimtDlogitsParams {
  const float* hidden;
  const float* weight;
  const float* bias;
  const float* q;     // KL: teacher probabilities [N][V]; null for the cross-entropy
  const float* qsum;  // KL: per-row sum of q
  const int64_t* targets;  // cross-entropy targets, or KL labels (nullable for KL)
  const float* lse;
  const float* grad_out;
  const int32_t* n_valid;
  float* d;  // [N][ldd]
  int64_t ldd;
  float* gb_partial;  // [ceil(N / kSimtTileN)][gb_ld] or null
  int64_t gb_ld;
  int64_t n, h, v, ignore_index;
  int64_t c0, width;
  int reduction;
  float label_smoothing;
  float z_loss;
  LogitXform xf;
};
cudaError_t launch_simt_dlogits(const SimtDlogitsParams& p, cudaStream_t s);

// C[m, n] (+)= sum_k A[m*sam + k*sak] * B[k*sbk + n*sbn], fp32.
cudaError_t launch_simt_gemm(int64_t m, int64_t n, int64_t k, const float* a, int64_t sam,
                             int64_t sak, const float* b, int64_t sbk, int64_t sbn, float* c,
                             int64_t ldc, int accumulate, cudaStream_t s);

// row kernels
struct MergeParams {
  const float4* partials;
  const float* zsum;          // per-tile logit sums (label smoothing) or null
  float label_smoothing;
  float z_loss;
  const float* zt;
  const int64_t* targets;     // of the (possibly compacted) rows
  const int32_t* row_map;     // original row of each compacted row, or null
  const int32_t* n_dyn;       // compacted row count (device) or null
  int64_t n, v, n_vt, ignore_index;
  float* loss_rows;
  float* lse_rows;
  int32_t* correct_ws;     // [N] always written
  float* entropy_ws;       // [N] always written
  int32_t* correct_rows;   // user copy or null
  float* entropy_rows;     // user copy or null
  int32_t* err_word;
};
cudaError_t launch_merge_rows(const MergeParams& p, cudaStream_t s);

struct FinalizeParams {
  const float* loss_rows;
  const int32_t* correct_ws;
  const float* entropy_ws;
  const int64_t* targets;
  int64_t n, ignore_index;
  int reduction;
  float* loss_out;     // null for "none"
  float* metrics_out;  // null to skip
  int32_t* n_valid;
};
cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s);

// out[j] = sum_{r < n_parts} part[r*ld + j] (fixed order), cast to the output
// type (out_type: 0 fp32, 1 bf16, 2 fp16).
// With n_dyn, n_parts = ceil(*n_dyn / rows_per_part) (at most the static one).
cudaError_t launch_bias_reduce(const float* part, int64_t n_parts, int64_t ld, int64_t v,
                               void* out, int out_type, const int32_t* n_dyn,
                               int rows_per_part, cudaStream_t s);

// ---- valid-row compaction (FLCE_SKIP_IGNORED_ROWS)
struct CompactParams {
  const int64_t* targets;
  int64_t n, ignore_index;
  int32_t* row_map;  // [N] out: original row of compacted row j (stable order)
  int32_t* n_kept;   // out: number of kept rows
  // forward only (null in the backward): outputs of the ignored rows
  float* loss_rows;
  float* lse_rows;
  int32_t* correct_ws;
  float* entropy_ws;
  int32_t* correct_rows;
  float* entropy_rows;
  float* qsum_rows;  // KL forward (nullable); correct_ws / entropy_ws are nullable too
};
cudaError_t launch_compact_rows(const CompactParams& p, cudaStream_t s);

struct GatherParams {
  const void* hidden;  // 16-bit elements
  int64_t n, h;
  const int32_t* row_map;
  const int32_t* n_kept;
  int pad_rows;  // rows [n_kept, roundup(n_kept, pad_rows)) are zero-filled
  void* hidden_c;
  const int64_t* targets;
  int64_t* targets_c;
  int64_t ignore_index;
  const float* lse;   // backward: gathered into lse_c (nullable)
  float* lse_c;
  const float* grad_rows;  // backward, reduction none (nullable)
  float* grad_rows_c;
  const float* qsum;  // KL backward: per-row sum of q (nullable)
  float* qsum_c;
};
cudaError_t launch_gather_rows(const GatherParams& p, cudaStream_t s);

// x[0, n) (fp32, 16-byte aligned, n a multiple of 4) -> three bf16 arrays
// with x = hi + mid + lo exactly (the split-bf16 form of fp32 operands).
cudaError_t launch_split3(const float* x, int64_t n, void* hi, void* mid, void* lo, int sms,
                          cudaStream_t s);

// grad_hidden rows of ignored targets := 0 (16-bit elements, [N, h]).
cudaError_t launch_zero_ignored_rows(const int64_t* targets, int64_t n, int64_t ignore_index,
                                     void* out, int64_t h, cudaStream_t s);


}  // namespace flce
