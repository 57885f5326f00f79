// Per-row and scalar kernels of the fused linear cross-entropy:
//   merge_rows  combines the per-(row, vocabulary tile) softmax statistics
//               of a row into lse, loss, argmax-correctness and entropy
//               ("fused-linear-ce" model card, §Algorithm: running
//               log-sum-exp; §Metrics for free: argmax with the running max,
//               entropy with the same rescaling);
//   finalize    the reduced loss, n_valid and the two scalar metrics, in a
//               fixed summation order (bitwise repeatable);
//   bias_reduce grad_bias from per-row-tile column partial sums, fixed order.
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "flce_internal.h"

namespace flce {

namespace {

constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeWarps * 32) merge_rows_kernel(const MergeParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
  if (row >= p.n) return;  // warp-uniform
  const float4* part = p.partials + row * p.n_vt;
  RowStats st;
  st.init();
  for (int64_t u = lane; u < p.n_vt; u += 32) st = merge_stats(st, RowStats::unpack(part[u]));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) st = merge_stats(st, shfl_xor_stats(st, off));
  if (lane != 0) return;
  const float log_s = logf(st.s);
  const float lse = st.m + log_s;
  const float entropy = log_s - st.t / st.s;
  const int64_t t = p.targets[row];
  float loss = 0.0f;
  int correct = 0;
  if (t != p.ignore_index) {
    if (t >= 0 && t < p.v) {
      loss = lse - p.zt[row];
      correct = (static_cast<int64_t>(st.a) == t) ? 1 : 0;
    } else {
      loss = __int_as_float(0x7fc00000);  // NaN
      if (p.err_word) atomicOr(p.err_word, 1 /* FLCE_DEVERR_TARGET_RANGE */);
    }
  }
  p.loss_rows[row] = loss;
  p.lse_rows[row] = lse;
  p.correct_ws[row] = correct;
  p.entropy_ws[row] = entropy;
  if (p.correct_rows) p.correct_rows[row] = correct;
  if (p.entropy_rows) p.entropy_rows[row] = entropy;
}

constexpr int kFinThreads = 1024;

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const FinalizeParams p) {
  __shared__ double s_loss[kFinThreads];
  __shared__ double s_ent[kFinThreads];
  __shared__ long long s_nv[kFinThreads];
  __shared__ long long s_nc[kFinThreads];
  const int tid = threadIdx.x;
  double ls = 0.0, es = 0.0;
  long long nv = 0, nc = 0;
  for (int64_t i = tid; i < p.n; i += kFinThreads) {
    if (p.targets[i] == p.ignore_index) continue;
    ++nv;
    ls += static_cast<double>(p.loss_rows[i]);
    es += static_cast<double>(p.entropy_ws[i]);
    nc += p.correct_ws[i];
  }
  s_loss[tid] = ls;
  s_ent[tid] = es;
  s_nv[tid] = nv;
  s_nc[tid] = nc;
  __syncthreads();
  for (int w = kFinThreads / 2; w >= 1; w >>= 1) {
    if (tid < w) {
      s_loss[tid] += s_loss[tid + w];
      s_ent[tid] += s_ent[tid + w];
      s_nv[tid] += s_nv[tid + w];
      s_nc[tid] += s_nc[tid + w];
    }
    __syncthreads();
  }
  if (tid != 0) return;
  const double n_valid = static_cast<double>(s_nv[0]);
  p.n_valid[0] = static_cast<int32_t>(s_nv[0]);
  if (p.loss_out != nullptr) {
    if (p.reduction == 1) {
      p.loss_out[0] = static_cast<float>(s_loss[0]);
    } else if (p.reduction == 2) {
      p.loss_out[0] = static_cast<float>(s_loss[0] / n_valid);  // 0/0 -> NaN
    }
  }
  if (p.metrics_out != nullptr) {
    p.metrics_out[0] = static_cast<float>(static_cast<double>(s_nc[0]) / n_valid);
    p.metrics_out[1] = static_cast<float>(s_ent[0] / n_valid);
  }
}

__global__ void __launch_bounds__(256)
    bias_reduce_kernel(const float* __restrict__ part, int64_t n_parts, int64_t ld, int64_t v,
                       void* out, int out_bf16) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (j >= v) return;
  float acc = 0.0f;
  for (int64_t r = 0; r < n_parts; ++r) acc += part[r * ld + j];
  if (out_bf16) {
    static_cast<__nv_bfloat16*>(out)[j] = __float2bfloat16_rn(acc);
  } else {
    static_cast<float*>(out)[j] = acc;
  }
}

}  // namespace

cudaError_t launch_merge_rows(const MergeParams& p, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((p.n + kMergeWarps - 1) / kMergeWarps);
  merge_rows_kernel<<<grid, kMergeWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s) {
  finalize_kernel<<<1, kFinThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bias_reduce(const float* part, int64_t n_parts, int64_t ld, int64_t v,
                               void* out, int out_bf16, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((v + 255) / 256);
  bias_reduce_kernel<<<grid, 256, 0, s>>>(part, n_parts, ld, v, out, out_bf16);
  return cudaGetLastError();
}

}  // namespace flce
