// Per-row and scalar kernels of the fused linear cross-entropy:
//   merge_rows  combines the per-(row, vocabulary tile) softmax statistics
//               of a row into lse, loss, argmax-correctness and entropy
//               ("fused-linear-ce" model card, §Algorithm: running
//               log-sum-exp; §Metrics for free: argmax with the running max,
//               entropy with the same rescaling);
//   finalize    the reduced loss, n_valid and the two scalar metrics, in a
//               fixed summation order (bitwise repeatable);
//   bias_reduce grad_bias from per-row-tile column partial sums, fixed order;
//   merge_kl / finalize_kl  the same two steps for the fused linear KL
//               divergence (FusedLinearKLDivLoss pull request, Liger-Kernel
//               #1423, Details: loss = sum q (log q - z) + lse * sum q).
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "flce_internal.h"

namespace flce {

namespace {

constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeWarps * 32) merge_rows_kernel(const MergeParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
  const int64_t n_rows = p.n_dyn != nullptr ? static_cast<int64_t>(*p.n_dyn) : p.n;
  if (row >= n_rows) return;  // warp-uniform
  const float4* part = p.partials + row * p.n_vt;
  RowStats st;
  st.init();
  for (int64_t u = lane; u < p.n_vt; u += 32) st = merge_stats(st, RowStats::unpack(part[u]));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) st = merge_stats(st, shfl_xor_stats(st, off));
  float zsum = 0.0f;  // sum of the row's logits (label smoothing)
  if (p.zsum != nullptr) {
    const float* zp = p.zsum + row * p.n_vt;
    for (int64_t u = lane; u < p.n_vt; u += 32) zsum += zp[u];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) zsum += __shfl_xor_sync(0xffffffffu, zsum, off);
  }
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
      if (p.zsum != nullptr) {
        // cross-entropy against (1 - eps) onehot + eps / V
        const float eps = p.label_smoothing;
        loss = fmaf(1.0f - eps, loss, eps * (lse - zsum / static_cast<float>(p.v)));
      }
      if (p.z_loss != 0.0f) loss = fmaf(p.z_loss * lse, lse, loss);
      correct = (static_cast<int64_t>(st.a) == t) ? 1 : 0;
    } else {
      loss = __int_as_float(0x7fc00000);  // NaN
      if (p.err_word) atomicOr(p.err_word, 1 /* FLCE_DEVERR_TARGET_RANGE */);
    }
  }
  const int64_t orig = p.row_map != nullptr ? static_cast<int64_t>(p.row_map[row]) : row;
  p.loss_rows[orig] = loss;
  p.lse_rows[orig] = lse;
  p.correct_ws[orig] = correct;
  p.entropy_ws[orig] = entropy;
  if (p.correct_rows) p.correct_rows[orig] = correct;
  if (p.entropy_rows) p.entropy_rows[orig] = entropy;
}

constexpr int kFinThreads = 1024;
constexpr int kFinUnroll = 4;

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const FinalizeParams p) {
  __shared__ double s_loss[kFinThreads];
  __shared__ double s_ent[kFinThreads];
  __shared__ long long s_nv[kFinThreads];
  __shared__ long long s_nc[kFinThreads];
  const int tid = threadIdx.x;
  double ls = 0.0, es = 0.0;
  long long nv = 0, nc = 0;
  // Rows tid, tid + kFinThreads, ... in that order. A row's four loads do
  // not wait for its target, and kFinUnroll rows are in flight per thread.
  for (int64_t i0 = tid; i0 < p.n; i0 += kFinUnroll * kFinThreads) {
    int64_t t[kFinUnroll];
    float l[kFinUnroll], e[kFinUnroll];
    int c[kFinUnroll];
#pragma unroll
    for (int u = 0; u < kFinUnroll; ++u) {
      const int64_t i = i0 + u * kFinThreads;
      const bool in = i < p.n;
      t[u] = in ? p.targets[i] : p.ignore_index;
      l[u] = in ? p.loss_rows[i] : 0.0f;
      e[u] = in ? p.entropy_ws[i] : 0.0f;
      c[u] = in ? p.correct_ws[i] : 0;
    }
#pragma unroll
    for (int u = 0; u < kFinUnroll; ++u) {
      if (t[u] == p.ignore_index) continue;
      ++nv;
      ls += static_cast<double>(l[u]);
      es += static_cast<double>(e[u]);
      nc += c[u];
    }
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

// KL: a row's (m, s) merge as softmax statistics; A = sum q (log max(q,
// eps) - z) and Q = sum q are plain sums. loss = A + lse * Q on counted rows.
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kl_kernel(const MergeKLParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
  const int64_t n_rows = p.n_dyn != nullptr ? static_cast<int64_t>(*p.n_dyn) : p.n;
  if (row >= n_rows) return;  // warp-uniform
  const float4* part = p.partials + row * p.n_vt;
  RowStats st;
  st.init();
  float a_sum = 0.0f, q_sum = 0.0f;
  for (int64_t u = lane; u < p.n_vt; u += 32) {
    const float4 v = part[u];
    RowStats x;
    x.m = v.x;
    x.s = v.y;
    x.t = 0.0f;
    x.a = 0;
    st = merge_stats(st, x);
    a_sum += v.z;
    q_sum += v.w;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    st = merge_stats(st, shfl_xor_stats(st, off));
    a_sum += __shfl_xor_sync(0xffffffffu, a_sum, off);
    q_sum += __shfl_xor_sync(0xffffffffu, q_sum, off);
  }
  if (lane != 0) return;
  const float lse = st.m + logf(st.s);
  const bool counted = p.labels == nullptr || p.labels[row] != p.ignore_index;
  const int64_t orig = p.row_map != nullptr ? static_cast<int64_t>(p.row_map[row]) : row;
  p.loss_rows[orig] = counted ? fmaf(lse, q_sum, a_sum) : 0.0f;
  p.lse_rows[orig] = lse;
  p.qsum_rows[orig] = q_sum;
}

__global__ void __launch_bounds__(kFinThreads) finalize_kl_kernel(const FinalizeKLParams p) {
  __shared__ double s_loss[kFinThreads];
  __shared__ long long s_nc[kFinThreads];
  const int tid = threadIdx.x;
  double ls = 0.0;
  long long nc = 0;
  for (int64_t i0 = tid; i0 < p.n; i0 += kFinUnroll * kFinThreads) {
    bool counted[kFinUnroll];
    float l[kFinUnroll];
#pragma unroll
    for (int u = 0; u < kFinUnroll; ++u) {
      const int64_t i = i0 + u * kFinThreads;
      const bool in = i < p.n;
      counted[u] = in && (p.labels == nullptr || p.labels[i] != p.ignore_index);
      l[u] = in ? p.loss_rows[i] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kFinUnroll; ++u) {
      if (!counted[u]) continue;
      ++nc;
      ls += static_cast<double>(l[u]);
    }
  }
  s_loss[tid] = ls;
  s_nc[tid] = nc;
  __syncthreads();
  for (int w = kFinThreads / 2; w >= 1; w >>= 1) {
    if (tid < w) {
      s_loss[tid] += s_loss[tid + w];
      s_nc[tid] += s_nc[tid + w];
    }
    __syncthreads();
  }
  if (tid != 0) return;
  p.n_counted[0] = static_cast<int32_t>(s_nc[0]);
  if (p.loss_out == nullptr) return;
  const double tot = s_loss[0], cnt = static_cast<double>(s_nc[0]);
  if (p.reduction == 1) {
    p.loss_out[0] = static_cast<float>(tot);
  } else if (p.reduction == 2) {
    p.loss_out[0] = static_cast<float>(tot / cnt);  // 0/0 -> NaN
  } else if (p.reduction == 3) {
    p.loss_out[0] = static_cast<float>(tot / (cnt * static_cast<double>(p.v)));
  }
}

__global__ void __launch_bounds__(256)
    bias_reduce_kernel(const float* __restrict__ part, int64_t n_parts, int64_t ld, int64_t v,
                       void* out, int out_type, const int32_t* n_dyn, int rows_per_part) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (j >= v) return;
  if (n_dyn != nullptr) {
    const int64_t parts = (static_cast<int64_t>(*n_dyn) + rows_per_part - 1) / rows_per_part;
    n_parts = parts < n_parts ? parts : n_parts;
  }
  float acc = 0.0f;
  for (int64_t r = 0; r < n_parts; ++r) acc += part[r * ld + j];
  if (out_type == kTcBF16) {
    static_cast<__nv_bfloat16*>(out)[j] = __float2bfloat16_rn(acc);
  } else if (out_type == kTcF16) {
    static_cast<__half*>(out)[j] = __float2half_rn(acc);
  } else {
    static_cast<float*>(out)[j] = acc;
  }
}

// scales[0] = 2^k with |gs * 2^k| in [8192, 16384), scales[1] = 2^-k; gs
// bounds |D|: the largest row upstream gradient (grad_out/n_valid/extra_div,
// grad_out/extra_div, or max |grad_out[i]| over counted rows) times
// |logit_scale| times either (1 + 2 |z_loss| max |lse|) or, with row_bound,
// max row_bound over counted rows. 1 and 1 when gs is zero or not finite.
__device__ __forceinline__ float block_max(float x, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  if (lane == 0) red[warp] = x;
  __syncthreads();
  x = red[lane];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  __syncthreads();
  return x;
}

__global__ void __launch_bounds__(1024)
    dlogits_scale_kernel(const float* grad_out, const int32_t* n_valid, const int64_t* targets,
                         int64_t n, int64_t ignore_index, int reduction, float logit_scale,
                         float z_loss, const float* lse_rows, const float* row_bound,
                         float extra_div, float* scales) {
  __shared__ float red[32];
  const int tid = threadIdx.x;
  float factor = 1.0f;
  if (row_bound != nullptr) {
    float b = 0.0f;
    for (int64_t i = tid; i < n; i += 1024)
      if (targets == nullptr || targets[i] != ignore_index) b = fmaxf(b, fabsf(row_bound[i]));
    factor = block_max(b, red);
  } else if (z_loss != 0.0f) {
    float lm = 0.0f;
    for (int64_t i = tid; i < n; i += 1024)
      if (targets == nullptr || targets[i] != ignore_index) lm = fmaxf(lm, fabsf(lse_rows[i]));
    lm = block_max(lm, red);
    factor = fmaf(2.0f * fabsf(z_loss), lm, 1.0f);
  }
  float g = 0.0f;
  if (reduction == 0) {
    for (int64_t i = tid; i < n; i += 1024)
      if (targets == nullptr || targets[i] != ignore_index) g = fmaxf(g, fabsf(grad_out[i]));
    g = block_max(g, red);
  } else {
    g = fabsf(grad_out[0]) / extra_div;
    if (reduction == 2) g = n_valid[0] > 0 ? g / static_cast<float>(n_valid[0]) : 0.0f;
  }
  if (tid != 0) return;
  const float gs = g * fabsf(logit_scale) * factor;
  float up = 1.0f, down = 1.0f;
  if (gs > 0.0f && isfinite(gs)) {
    int e = 0;
    frexpf(gs, &e);  // gs in [2^(e-1), 2^e)
    up = ldexpf(1.0f, 14 - e);
    down = ldexpf(1.0f, e - 14);
  }
  scales[0] = up;
  scales[1] = down;
}

// Stable compaction of the rows whose target is not ignore_index: one block
// scans the rows in order, 1024 at a time (ballot + warp-total scan), so
// compacted row j is the j-th kept row. Ignored rows get their forward
// outputs here.
constexpr int kCompactThreads = 1024;

__global__ void __launch_bounds__(kCompactThreads) compact_rows_kernel(const CompactParams p) {
  __shared__ int warp_off[32];
  __shared__ int chunk_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int carry = 0;
  // the target of this thread's row in the next pass is loaded one pass ahead
  int64_t t_next = tid < p.n ? p.targets[tid] : p.ignore_index;
  for (int64_t base = 0; base < p.n; base += kCompactThreads) {
    const int64_t i = base + tid;
    const bool in = i < p.n;
    const int64_t t = t_next;
    const int64_t i_next = i + kCompactThreads;
    t_next = i_next < p.n ? p.targets[i_next] : p.ignore_index;
    const bool keep = in && t != p.ignore_index;
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    const int before = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_off[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
      const int v = warp_off[lane];
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      warp_off[lane] = incl - v;
      if (lane == 31) chunk_total = incl;
    }
    __syncthreads();
    if (keep) {
      p.row_map[carry + warp_off[warp] + before] = static_cast<int32_t>(i);
    } else if (in && p.loss_rows != nullptr) {
      const float nan = __int_as_float(0x7fc00000);
      p.loss_rows[i] = 0.0f;
      p.lse_rows[i] = nan;
      if (p.correct_ws) p.correct_ws[i] = 0;
      if (p.entropy_ws) p.entropy_ws[i] = nan;
      if (p.correct_rows) p.correct_rows[i] = 0;
      if (p.entropy_rows) p.entropy_rows[i] = nan;
      if (p.qsum_rows) p.qsum_rows[i] = nan;
    }
    carry += chunk_total;
    __syncthreads();
  }
  if (tid == 0) *p.n_kept = carry;
}

constexpr int kGatherThreads = 256;  // 8 warps: one row per warp
constexpr int kRowsPerBlock = kGatherThreads / 32;
constexpr int kCopyUnroll = 4;  // 16-byte loads in flight per lane

// dst[q] = src[q] (or 0 when src is null) for q < vecs, by one warp.
__device__ __forceinline__ void copy_row(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                         int64_t vecs, int lane) {
  for (int64_t q0 = lane; q0 < vecs; q0 += 32 * kCopyUnroll) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t q = q0 + 32 * u;
      v[u] = (src != nullptr && q < vecs) ? __ldg(src + q) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t q = q0 + 32 * u;
      if (q < vecs) dst[q] = v[u];
    }
  }
}

// Compacted row j <- original row row_map[j]; rows [n_kept, pad) are zero so
// that a contraction over rows reads zeros past the last kept row.
__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const GatherParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  const int64_t kept = *p.n_kept;
  const int64_t pad = (kept + p.pad_rows - 1) / p.pad_rows * p.pad_rows;
  if (j >= pad || j >= p.n) return;
  const int64_t vecs = p.h / 8;  // 8 16-bit elements per 16-byte vector (h % 8 == 0)
  uint4* dst = reinterpret_cast<uint4*>(p.hidden_c) + j * vecs;
  if (j < kept) {
    const int64_t src_row = p.row_map[j];
    copy_row(dst, reinterpret_cast<const uint4*>(p.hidden) + src_row * vecs, vecs, lane);
    if (lane == 0) {
      p.targets_c[j] = p.targets[src_row];
      if (p.lse_c) p.lse_c[j] = p.lse[src_row];
      if (p.grad_rows_c) p.grad_rows_c[j] = p.grad_rows[src_row];
      if (p.qsum_c) p.qsum_c[j] = p.qsum[src_row];
    }
  } else {
    copy_row(dst, nullptr, vecs, lane);
    if (lane == 0) {
      p.targets_c[j] = p.ignore_index;
      if (p.lse_c) p.lse_c[j] = 0.0f;
      if (p.grad_rows_c) p.grad_rows_c[j] = 0.0f;
      if (p.qsum_c) p.qsum_c[j] = 0.0f;
    }
  }
}

// fp32 -> three bf16 parts, x = hi + mid + lo: hi = bf16(x), mid = bf16(x - hi),
// lo = x - hi - mid. Each remainder is exact in fp32 and lo needs at most 8
// significant bits, so the three parts hold x exactly (no underflow in
// bf16, whose exponent range is fp32's). Four elements per thread.
__device__ __forceinline__ void split3_store(const float (&e)[4], uint2* __restrict__ hi,
                                             uint2* __restrict__ mid, uint2* __restrict__ lo,
                                             int64_t i) {
  __nv_bfloat16 h[4], m[4], l[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    h[k] = __float2bfloat16_rn(e[k]);
    const float r1 = e[k] - __bfloat162float(h[k]);
    m[k] = __float2bfloat16_rn(r1);
    l[k] = __float2bfloat16_rn(r1 - __bfloat162float(m[k]));
  }
  auto pack = [](const __nv_bfloat16 (&b)[4]) {
    uint2 w;
    w.x = static_cast<uint32_t>(__bfloat16_as_ushort(b[0])) |
          (static_cast<uint32_t>(__bfloat16_as_ushort(b[1])) << 16);
    w.y = static_cast<uint32_t>(__bfloat16_as_ushort(b[2])) |
          (static_cast<uint32_t>(__bfloat16_as_ushort(b[3])) << 16);
    return w;
  };
  hi[i] = pack(h);
  mid[i] = pack(m);
  lo[i] = pack(l);
}

__global__ void __launch_bounds__(256)
    split3_kernel(const float4* __restrict__ x, int64_t n4, uint2* __restrict__ hi,
                  uint2* __restrict__ mid, uint2* __restrict__ lo) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = __ldg(x + i);
    const float e[4] = {v.x, v.y, v.z, v.w};
    split3_store(e, hi, mid, lo, i);
  }
}

__global__ void __launch_bounds__(256)
    split3_scalar_kernel(const float* __restrict__ x, int64_t n4, uint2* __restrict__ hi,
                         uint2* __restrict__ mid, uint2* __restrict__ lo) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float e[4] = {__ldg(x + 4 * i), __ldg(x + 4 * i + 1), __ldg(x + 4 * i + 2),
                        __ldg(x + 4 * i + 3)};
    split3_store(e, hi, mid, lo, i);
  }
}

__global__ void __launch_bounds__(kGatherThreads)
    zero_ignored_rows_kernel(const int64_t* __restrict__ targets, int64_t n, int64_t ignore_index,
                             void* out, int64_t h) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (i >= n || targets[i] != ignore_index) return;
  copy_row(reinterpret_cast<uint4*>(out) + i * (h / 8), nullptr, h / 8, threadIdx.x & 31);
}

}  // namespace

cudaError_t launch_compact_rows(const CompactParams& p, cudaStream_t s) {
  compact_rows_kernel<<<1, kCompactThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const GatherParams& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((p.n + kRowsPerBlock - 1) / kRowsPerBlock);
  gather_rows_kernel<<<grid, kGatherThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dlogits_scale(const float* grad_out, const int32_t* n_valid,
                                 const int64_t* targets, int64_t n, int64_t ignore_index,
                                 int reduction, float logit_scale, float z_loss,
                                 const float* lse_rows, const float* row_bound, float extra_div,
                                 float* scales, cudaStream_t s) {
  dlogits_scale_kernel<<<1, 1024, 0, s>>>(grad_out, n_valid, targets, n, ignore_index, reduction,
                                          logit_scale, z_loss, lse_rows, row_bound, extra_div,
                                          scales);
  return cudaGetLastError();
}

cudaError_t launch_merge_kl(const MergeKLParams& p, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((p.n + kMergeWarps - 1) / kMergeWarps);
  merge_kl_kernel<<<grid, kMergeWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_finalize_kl(const FinalizeKLParams& p, cudaStream_t s) {
  finalize_kl_kernel<<<1, kFinThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_split3(const float* x, int64_t n, void* hi, void* mid, void* lo,
                          int sms, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int64_t n4 = n / 4;
  int64_t blocks = (n4 + 255) / 256;
  if (blocks > 8 * static_cast<int64_t>(sms)) blocks = 8 * static_cast<int64_t>(sms);
  if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
    split3_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        reinterpret_cast<const float4*>(x), n4, static_cast<uint2*>(hi),
        static_cast<uint2*>(mid), static_cast<uint2*>(lo));
  } else {  // a caller's fp32 array need only be 4-byte aligned
    split3_scalar_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        x, n4, static_cast<uint2*>(hi), static_cast<uint2*>(mid), static_cast<uint2*>(lo));
  }
  return cudaGetLastError();
}

cudaError_t launch_zero_ignored_rows(const int64_t* targets, int64_t n, int64_t ignore_index,
                                     void* out, int64_t h, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((n + kRowsPerBlock - 1) / kRowsPerBlock);
  zero_ignored_rows_kernel<<<grid, kGatherThreads, 0, s>>>(targets, n, ignore_index, out, h);
  return cudaGetLastError();
}

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
                               void* out, int out_type, const int32_t* n_dyn,
                               int rows_per_part, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((v + 255) / 256);
  bias_reduce_kernel<<<grid, 256, 0, s>>>(part, n_parts, ld, v, out, out_type, n_dyn,
                                          rows_per_part);
  return cudaGetLastError();
}

}  // namespace flce
