// fp32 path of the fused linear cross-entropy: plain FFMA kernels.
//
// fp32 inputs need full fp32 products and sums; the bf16 tensor-core path
// would round them. These kernels follow the same plan as the tensor-core
// path ("fused-linear-ce" model card, §Algorithm): a vocabulary-tiled forward
// that folds each logit tile into per-(row, tile) softmax statistics, and a
// backward that recomputes the logits of one vocabulary chunk, forms D =
// g (p - onehot) dz/dlin in fp32 and contracts it with hidden and weight.
// With teacher probabilities q the same two kernels serve the fused linear KL
// divergence (FusedLinearKLDivLoss pull request, Liger-Kernel #1423): the
// forward keeps A = sum q (log max(q, eps) - z) and Q = sum q per tile, the
// backward forms D = g (p Q - q) / T.
#include <cfloat>
#include <cstdint>
#include <cuda_runtime.h>

#include "flce_internal.h"

namespace flce {

namespace {

constexpr int TN = kSimtTileN;  // rows per block
constexpr int TV = kSimtTileV;  // vocabulary columns per block
constexpr int TK = 32;

// acc[i][j] = hidden[row0 + ty*4 + i] . weight[col0 + tx + 32 j] over all H.
__device__ __forceinline__ void logit_tile(const float* __restrict__ hidden,
                                           const float* __restrict__ weight, int64_t n, int64_t h,
                                           int64_t v, int64_t row0, int64_t col0,
                                           float (&as)[TN][TK + 1], float (&bs)[TV][TK + 1],
                                           float (&acc)[4][4]) {
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int64_t k0 = 0; k0 < h; k0 += TK) {
#pragma unroll
    for (int r = 0; r < (TN * TK) / 256; ++r) {
      const int idx = tid + 256 * r, rr = idx / TK, kk = idx % TK;
      const int64_t gr = row0 + rr, gk = k0 + kk;
      as[rr][kk] = (gr < n && gk < h) ? hidden[gr * h + gk] : 0.0f;
    }
#pragma unroll
    for (int r = 0; r < (TV * TK) / 256; ++r) {
      const int idx = tid + 256 * r, cc = idx / TK, kk = idx % TK;
      const int64_t gc = col0 + cc, gk = k0 + kk;
      bs[cc][kk] = (gc < v && gk < h) ? weight[gc * h + gk] : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = as[ty * 4 + i][kk];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = bs[tx + 32 * j][kk];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) simt_fwd_kernel(const SimtFwdParams p) {
  __shared__ float as[TN][TK + 1];
  __shared__ float bs[TV][TK + 1];
  __shared__ float zs[TN][TV + 1];
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * TN;
  const int64_t col0 = static_cast<int64_t>(blockIdx.y) * TV;
  float acc[4][4];
  logit_tile(p.hidden, p.weight, p.n, p.h, p.v, row0, col0, as, bs, acc);
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t c = col0 + tx + 32 * j;
      const float b = (p.bias != nullptr && c < p.v) ? p.bias[c] : 0.0f;
      zs[ty * 4 + i][tx + 32 * j] = p.xf(acc[i][j], b);
    }
  __syncthreads();
  const int warp = ty, lane = tx;
  for (int r = 0; r < 4; ++r) {
    const int rl = warp * 4 + r;
    const int64_t row = row0 + rl;
    if (row >= p.n) break;  // warp-uniform
    RowStats st;
    st.init();
    float zsum = 0.0f;          // cross-entropy: sum z (label smoothing)
    float a_sum = 0.0f;         // KL: sum q (log max(q, eps) - z)
    float q_sum = 0.0f;         // KL: sum q
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int cl = lane + 32 * j;
      const int64_t c = col0 + cl;
      if (c < p.v) {
        const float z = zs[rl][cl];
        if (z > st.m) {
          st.a = static_cast<int>(c);
          st.rebase(z);
        }
        st.add(z);
        zsum += z;
        if (p.q != nullptr) {
          const float q = p.q[row * p.v + c];
          a_sum = fmaf(q, logf(fmaxf(q, p.eps)) - z, a_sum);
          q_sum += q;
        }
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      st = merge_stats(st, shfl_xor_stats(st, off));
      zsum += __shfl_xor_sync(0xffffffffu, zsum, off);
      a_sum += __shfl_xor_sync(0xffffffffu, a_sum, off);
      q_sum += __shfl_xor_sync(0xffffffffu, q_sum, off);
    }
    if (lane == 0) {
      if (p.q != nullptr) {  // KL partials: (m, s, A, Q)
        p.partials[row * p.n_vt + blockIdx.y] = make_float4(st.m, st.s, a_sum, q_sum);
        continue;
      }
      p.partials[row * p.n_vt + blockIdx.y] = st.pack();
      if (p.zsum != nullptr) p.zsum[row * p.n_vt + blockIdx.y] = zsum;
      const int64_t t = p.targets[row];
      if (t >= col0 && t < col0 + TV && t < p.v) p.zt[row] = zs[rl][t - col0];
    }
  }
}

__global__ void __launch_bounds__(256) simt_dlogits_kernel(const SimtDlogitsParams p) {
  __shared__ float as[TN][TK + 1];
  __shared__ float bs[TV][TK + 1];
  __shared__ float ds[TN][TV + 1];
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * TN;
  const int64_t lcol0 = static_cast<int64_t>(blockIdx.y) * TV;  // within the chunk
  const int64_t col0 = p.c0 + lcol0;
  const int64_t vend = p.c0 + p.width;  // end of this chunk (<= V)
  float acc[4][4];
  logit_tile(p.hidden, p.weight, p.n, p.h, vend, row0, col0, as, bs, acc);
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rl = ty * 4 + i;
    const int64_t row = row0 + rl;
    const bool row_ok = row < p.n;
    const bool kl = p.q != nullptr;
    const int64_t t = (row_ok && p.targets != nullptr) ? p.targets[row] : p.ignore_index;
    float g = 0.0f;
    if (kl) {
      const bool counted = row_ok && (p.targets == nullptr || t != p.ignore_index);
      g = kl_row_grad(counted, p.reduction, p.grad_out, p.n_valid, p.v, row);
    } else if (row_ok) {
      g = row_grad(t, p.ignore_index, p.v, p.reduction, p.grad_out, p.n_valid, row);
    }
    const float lse = row_ok ? p.lse[row] : 0.0f;
    const float qs = (kl && row_ok) ? p.qsum[row] : 0.0f;
    const float pz = fmaf(2.0f * p.z_loss, lse, 1.0f);
    const float eps_v = p.label_smoothing / static_cast<float>(p.v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int cl = tx + 32 * j;
      const int64_t c = col0 + cl;
      float d = 0.0f;
      if (row_ok && c < vend) {
        const float b = (p.bias != nullptr) ? p.bias[c] : 0.0f;
        const float z = p.xf(acc[i][j], b);
        const float pr = ex2_approx((z - lse) * kLog2e);
        if (kl) {
          d = fmaf(pr, qs, -p.q[row * p.v + c]);  // p sum q - q
        } else {
          d = fmaf(pr, pz, -eps_v);
          if (c == t) d -= 1.0f - p.label_smoothing;
        }
        d *= g * p.xf.scale * p.xf.dz_du(z);
        p.d[row * p.ldd + (c - p.c0)] = d;
      }
      ds[rl][cl] = d;
    }
  }
  if (p.gb_partial != nullptr) {
    __syncthreads();
    if (tid < TV) {
      const int64_t c = col0 + tid;
      if (c < vend) {
        float sum = 0.0f;
        for (int r = 0; r < TN; ++r) sum += ds[r][tid];
        p.gb_partial[static_cast<int64_t>(blockIdx.x) * p.gb_ld + c] = sum;
      }
    }
  }
}

__global__ void __launch_bounds__(256)
    simt_gemm_kernel(int64_t m, int64_t n, int64_t k, const float* __restrict__ a, int64_t sam,
                     int64_t sak, const float* __restrict__ b, int64_t sbk, int64_t sbn,
                     float* __restrict__ c, int64_t ldc, int accumulate) {
  __shared__ float as[16][65];
  __shared__ float bs[16][65];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * 64;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 64;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int64_t k0 = 0; k0 < k; k0 += 16) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int idx = tid + 256 * r;
      int mm, kk;
      if (sam == 1) {
        mm = idx & 63;
        kk = idx >> 6;
      } else {
        kk = idx & 15;
        mm = idx >> 4;
      }
      const int64_t gm = m0 + mm, gk = k0 + kk;
      as[kk][mm] = (gm < m && gk < k) ? a[gm * sam + gk * sak] : 0.0f;
      int nn, kb;
      if (sbn == 1) {
        nn = idx & 63;
        kb = idx >> 6;
      } else {
        kb = idx & 15;
        nn = idx >> 4;
      }
      const int64_t gn = n0 + nn, gkb = k0 + kb;
      bs[kb][nn] = (gn < n && gkb < k) ? b[gkb * sbk + gn * sbn] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = as[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty + 16 * i;
    if (gm >= m) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gn = n0 + tx + 16 * j;
      if (gn >= n) continue;
      float* dst = c + gm * ldc + gn;
      *dst = accumulate ? (*dst + acc[i][j]) : acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_simt_fwd(const SimtFwdParams& p, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((p.n + TN - 1) / TN),
                  static_cast<unsigned>((p.v + TV - 1) / TV));
  simt_fwd_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_simt_dlogits(const SimtDlogitsParams& p, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((p.n + TN - 1) / TN),
                  static_cast<unsigned>((p.width + TV - 1) / TV));
  simt_dlogits_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_simt_gemm(int64_t m, int64_t n, int64_t k, const float* a, int64_t sam,
                             int64_t sak, const float* b, int64_t sbk, int64_t sbn, float* c,
                             int64_t ldc, int accumulate, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((n + 63) / 64), static_cast<unsigned>((m + 63) / 64));
  simt_gemm_kernel<<<grid, 256, 0, s>>>(m, n, k, a, sam, sak, b, sbk, sbn, c, ldc, accumulate);
  return cudaGetLastError();
}

}  // namespace flce
