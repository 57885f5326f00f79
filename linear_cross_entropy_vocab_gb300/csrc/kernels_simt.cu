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
//
// All four contractions share one register-blocked mainloop: a 128 x 128
// output tile per 256-thread block, 8 x 8 outputs per thread, k-steps of 8
// staged through double-buffered shared memory with the next step's global
// loads in flight during the current step's FMAs (packed f32x2). Each operand is either
// K-major (k contiguous: hidden and weight for the logits, D for grad_hidden)
// or MN-major (the tile's own dimension contiguous: D^T and hidden for
// grad_weight, weight for grad_hidden); both land in shared memory as
// [k][mn] so that every thread reads its 8 rows and 8 columns as two float4
// each. VEC kernels move 16-byte vectors and need 16-byte-aligned bases and
// leading dimensions that are multiples of 4; the others move single floats
// and accept any fp32 layout.
#include <cfloat>
#include <cstdint>
#include <cuda_runtime.h>

#include "flce_internal.h"

namespace flce {

namespace {

constexpr int BM = kSimtTileN;  // rows of the output tile
constexpr int BN = kSimtTileV;  // columns of the output tile
constexpr int BK = 8;           // k per shared-memory stage
constexpr int LDS = BM + 4;     // padded row of a [k][mn] stage (16-byte multiple)
constexpr int kThreads = 256;
static_assert(BM == 128 && BN == 128, "the thread layout below assumes 128 x 128 tiles");

// Element (mn, k) of an operand sits at p[mn * s_mn + k * s_k]; K-major
// operands have s_k == 1, MN-major ones s_mn == 1. Elements outside
// [0, mn_ext) x [0, k_ext) read as zero.
struct Operand {
  const float* p;
  int64_t s_mn, s_k, mn_ext, k_ext;
};

struct Stage {
  float a[BK][LDS];
  float b[BK][LDS];
};

// Each thread moves four elements of a 128 x 8 operand tile.
// K-major (s_k == 1): thread t takes row mn = t / 2 and k = 4 (t % 2) .. +3.
// MN-major (s_mn == 1): thread t takes k = t / 32 and mn = 4 (t % 32) .. +3.
// Element i of the thread at step k0 sits at ptr + k0 * s_k + i (the unit
// stride of either layout) and is read when bit i of `ok` is set and
// k0 + kofs (+ i, K-major) < k_ext; the rest read as zero.
template <bool KMAJ, bool VEC>
struct TileLoader {
  const float* ptr;
  int64_t s_k;  // k stride of an MN-major operand (1 for K-major)
  int kofs;
  unsigned ok;

  __device__ __forceinline__ TileLoader(const Operand& op, int64_t mn0, int tid) {
    if (KMAJ) {
      const int64_t gm = mn0 + (tid >> 1);
      kofs = (tid & 1) * 4;
      s_k = 1;
      ok = gm < op.mn_ext ? 0xfu : 0u;
      ptr = op.p + (ok ? gm * op.s_mn : 0) + kofs;
    } else {
      const int64_t gm = mn0 + (tid & 31) * 4;
      kofs = tid >> 5;
      s_k = op.s_k;
      ok = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i) ok |= (gm + i < op.mn_ext ? 1u : 0u) << i;
      ptr = op.p + (ok ? gm : 0) + kofs * op.s_k;
    }
  }

  __device__ __forceinline__ void load(int64_t k0, int64_t k_ext, float (&r)[4]) const {
    const float* src = ptr + (KMAJ ? k0 : k0 * s_k);
    const int64_t k = k0 + kofs;
    if (VEC && ok == 0xfu && k + (KMAJ ? 3 : 0) < k_ext) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src));
      r[0] = v.x, r[1] = v.y, r[2] = v.z, r[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        r[i] = (((ok >> i) & 1u) && k + (KMAJ ? i : 0) < k_ext) ? __ldg(src + i) : 0.0f;
    }
  }
};

// The K-major store is a transpose: lanes of one warp cover 16 rows at two
// k offsets 4 apart, which the 132-float row pitch puts 16 banks apart.
template <bool KMAJ>
__device__ __forceinline__ void store_tile(float (&s)[BK][LDS], int tid, const float (&r)[4]) {
  if (KMAJ) {
    const int mn = tid >> 1, k = (tid & 1) * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) s[k + i][mn] = r[i];
  } else {
    *reinterpret_cast<float4*>(&s[tid >> 5][(tid & 31) * 4]) = make_float4(r[0], r[1], r[2], r[3]);
  }
}

// Output row (column) of the thread's i-th row (j-th column) in the tile:
// thread (tx, ty) = (t % 16, t / 16) owns rows 4 ty .. +3 and 64 + 4 ty .. +3
// and columns 4 tx .. +3 and 64 + 4 tx .. +3. The 16 threads of one ty are
// one half-warp, so a row's 128 columns reduce with xor shuffles 1 .. 8.
__device__ __forceinline__ int tile_row(int ty, int i) { return (i >> 2) * 64 + ty * 4 + (i & 3); }
__device__ __forceinline__ int tile_col(int tx, int j) { return (j >> 2) * 64 + tx * 4 + (j & 3); }

// acc[i][j] = sum_k A(m0 + tile_row(i), k) B(n0 + tile_col(j), k) over
// k < a.k_ext (== b.k_ext). Ends with a barrier, so the caller may reuse
// `st` as scratch.
template <bool AK, bool BKM, bool VEC>
__device__ __forceinline__ void mainloop(const Operand& a, const Operand& b, int64_t m0,
                                         int64_t n0, Stage (&st)[2], float (&acc)[8][8]) {
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  // Column pairs of the accumulator, updated by packed f32x2 FMAs (two
  // round-to-nearest fp32 FMAs per instruction, so the same sums as fmaf):
  // the FMA pipe then needs half the issue slots, which leaves room for the
  // shared-memory loads and the a-value broadcasts.
  uint64_t acc2[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc2[i][j] = 0ull;
  const int64_t k_ext = a.k_ext;
  const TileLoader<AK, VEC> la(a, m0, tid);
  const TileLoader<BKM, VEC> lb(b, n0, tid);
  float ra[4], rb[4];
  la.load(0, k_ext, ra);
  lb.load(0, k_ext, rb);
  store_tile<AK>(st[0].a, tid, ra);
  store_tile<BKM>(st[0].b, tid, rb);
  __syncthreads();
  int buf = 0;
  for (int64_t k0 = 0; k0 < k_ext; k0 += BK) {
    const bool more = k0 + BK < k_ext;
    if (more) {
      la.load(k0 + BK, k_ext, ra);
      lb.load(k0 + BK, k_ext, rb);
    }
    const Stage& s = st[buf];
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&s.a[kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&s.a[kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&s.b[kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&s.b[kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const uint64_t bp[4] = {f2_pack(b0.x, b0.y), f2_pack(b0.z, b0.w), f2_pack(b1.x, b1.y),
                              f2_pack(b1.z, b1.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint64_t ap = f2_pack(av[i], av[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc2[i][j] = f2_fma(ap, bp[j], acc2[i][j]);
      }
    }
    if (more) {
      store_tile<AK>(st[buf ^ 1].a, tid, ra);
      store_tile<BKM>(st[buf ^ 1].b, tid, rb);
    }
    __syncthreads();
    buf ^= 1;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) f2_unpack(acc2[i][j], acc[i][2 * j], acc[i][2 * j + 1]);
}

// Loads q[row][c .. c + 3] (zeros past v) as one vector when `vec`.
__device__ __forceinline__ void load_q4(const float* __restrict__ qrow, int64_t c, int64_t v,
                                        bool vec, float (&q)[4]) {
  if (vec && c + 3 < v) {
    const float4 x = __ldcs(reinterpret_cast<const float4*>(qrow + c));
    q[0] = x.x, q[1] = x.y, q[2] = x.z, q[3] = x.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = (c + i < v) ? __ldcs(qrow + c + i) : 0.0f;
  }
}

// Forward: one 128-row x 128-column logit tile per block, folded into the
// per-(row, tile) partials. Cross-entropy partials are (m, s, t, argmax)
// plus the tile's logit sum (label smoothing) and the target logit; KL
// partials are (m, s, A, Q).
template <bool VEC>
__global__ void __launch_bounds__(kThreads, 2) simt_fwd_kernel(const SimtFwdParams p, int q_vec) {
  __shared__ __align__(16) Stage st[2];
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * BM;
  const int64_t col0 = static_cast<int64_t>(blockIdx.y) * BN;
  const Operand a{p.hidden, p.h, 1, p.n, p.h};
  const Operand b{p.weight, p.h, 1, p.v, p.h};
  float acc[8][8];
  mainloop<true, true, VEC>(a, b, row0, col0, st, acc);

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const bool kl = p.q != nullptr;
  bool col_ok[8];
  float bias[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t c = col0 + tile_col(tx, j);
    col_ok[j] = c < p.v;
    bias[j] = (p.bias != nullptr && col_ok[j]) ? p.bias[c] : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t row = row0 + tile_row(ty, i);
    const bool row_ok = row < p.n;  // uniform over the half-warp that owns the row
    float z[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) z[j] = p.xf(acc[i][j], bias[j]);
    // The thread's 8 columns ascend with j, so a strict > keeps the lowest
    // index reaching the maximum.
    RowStats rs;
    rs.init();
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (col_ok[j] && z[j] > rs.m) {
        rs.m = z[j];
        rs.a = static_cast<int>(col0 + tile_col(tx, j));
      }
    float zsum = 0.0f, a_sum = 0.0f, q_sum = 0.0f;
    float q[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    if (kl && row_ok) {
      const float* qrow = p.q + row * p.v;
      float q4[4];
      load_q4(qrow, col0 + tile_col(tx, 0), p.v, q_vec != 0, q4);
#pragma unroll
      for (int k = 0; k < 4; ++k) q[k] = q4[k];
      load_q4(qrow, col0 + tile_col(tx, 4), p.v, q_vec != 0, q4);
#pragma unroll
      for (int k = 0; k < 4; ++k) q[4 + k] = q4[k];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!col_ok[j]) continue;
      const float d = z[j] - rs.m;
      const float e = ex2_approx(d * kLog2e);
      rs.s += e;
      rs.t = fmaf(e, d, rs.t);
      zsum += z[j];
      if (kl) {
        a_sum = fmaf(q[j], logf(fmaxf(q[j], p.eps)) - z[j], a_sum);
        q_sum += q[j];
      }
    }
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
      rs = merge_stats(rs, shfl_xor_stats(rs, off));
      zsum += __shfl_xor_sync(0xffffffffu, zsum, off);
      a_sum += __shfl_xor_sync(0xffffffffu, a_sum, off);
      q_sum += __shfl_xor_sync(0xffffffffu, q_sum, off);
    }
    if (!row_ok) continue;
    const int64_t slot = row * p.n_vt + blockIdx.y;
    if (kl) {
      if (tx == 0) p.partials[slot] = make_float4(rs.m, rs.s, a_sum, q_sum);
      continue;
    }
    if (tx == 0) {
      p.partials[slot] = rs.pack();
      if (p.zsum != nullptr) p.zsum[slot] = zsum;
    }
    const int64_t t = p.targets[row];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (col_ok[j] && t == col0 + tile_col(tx, j)) p.zt[row] = z[j];
  }
}

// Backward: recompute one 128 x 128 logit tile of the vocabulary chunk
// [c0, c0 + width), form D and store it; with a bias, also the tile's
// column sums of D over its 128 rows (the grad_bias partial of this row
// block), in a fixed order.
template <bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
    simt_dlogits_kernel(const SimtDlogitsParams p, int q_vec, int d_vec) {
  __shared__ __align__(16) Stage st[2];
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * BM;
  const int64_t col0 = p.c0 + static_cast<int64_t>(blockIdx.y) * BN;
  const int64_t vend = p.c0 + p.width;  // end of this chunk (<= V)
  const Operand a{p.hidden, p.h, 1, p.n, p.h};
  const Operand b{p.weight, p.h, 1, vend, p.h};
  float acc[8][8];
  mainloop<true, true, VEC>(a, b, row0, col0, st, acc);

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const bool kl = p.q != nullptr;
  const float eps_v = p.label_smoothing / static_cast<float>(p.v);
  bool col_ok[8];
  float bias[8], colsum[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t c = col0 + tile_col(tx, j);
    col_ok[j] = c < vend;
    bias[j] = (p.bias != nullptr && col_ok[j]) ? p.bias[c] : 0.0f;
    colsum[j] = 0.0f;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t row = row0 + tile_row(ty, i);
    if (row >= p.n) continue;
    const int64_t t = p.targets != nullptr ? p.targets[row] : p.ignore_index;
    float g;
    if (kl)
      g = kl_row_grad(p.targets == nullptr || t != p.ignore_index, p.reduction, p.grad_out,
                      p.n_valid, p.v, row);
    else
      g = row_grad(t, p.ignore_index, p.v, p.reduction, p.grad_out, p.n_valid, row);
    const float lse = p.lse[row];
    const float qs = kl ? p.qsum[row] : 0.0f;
    const float pz = fmaf(2.0f * p.z_loss, lse, 1.0f);
    float q[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    if (kl) {
      const float* qrow = p.q + row * p.v;
      float q4[4];
      load_q4(qrow, col0 + tile_col(tx, 0), vend, q_vec != 0, q4);
#pragma unroll
      for (int k = 0; k < 4; ++k) q[k] = q4[k];
      load_q4(qrow, col0 + tile_col(tx, 4), vend, q_vec != 0, q4);
#pragma unroll
      for (int k = 0; k < 4; ++k) q[4 + k] = q4[k];
    }
    float d[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t c = col0 + tile_col(tx, j);
      const float z = p.xf(acc[i][j], bias[j]);
      const float pr = ex2_approx((z - lse) * kLog2e);
      float dj;
      if (kl) {
        dj = fmaf(pr, qs, -q[j]);  // p sum q - q
      } else {
        dj = fmaf(pr, pz, -eps_v);
        if (c == t) dj -= 1.0f - p.label_smoothing;
      }
      dj *= g * p.xf.scale * p.xf.dz_du(z);
      d[j] = col_ok[j] ? dj : 0.0f;
      colsum[j] += d[j];
    }
    float* drow = p.d + row * p.ldd - p.c0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t c = col0 + tile_col(tx, 4 * h);
      if (d_vec && c + 3 < vend) {
        *reinterpret_cast<float4*>(drow + c) =
            make_float4(d[4 * h], d[4 * h + 1], d[4 * h + 2], d[4 * h + 3]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (c + k < vend) drow[c + k] = d[4 * h + k];
      }
    }
  }
  if (p.gb_partial == nullptr) return;
  // Column sums: the two ty of a warp by a shuffle, then the 8 warps in
  // order through shared memory (free again after the mainloop's barrier).
#pragma unroll
  for (int j = 0; j < 8; ++j) colsum[j] += __shfl_xor_sync(0xffffffffu, colsum[j], 16);
  float(*red)[BN] = reinterpret_cast<float(*)[BN]>(&st[0]);
  const int warp = tid >> 5;
  if ((tid & 16) == 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j) red[warp][tile_col(tx, j)] = colsum[j];
  }
  __syncthreads();
  if (tid < BN) {
    const int64_t c = col0 + tid;
    if (c < vend) {
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) sum += red[w][tid];
      p.gb_partial[static_cast<int64_t>(blockIdx.x) * p.gb_ld + c] = sum;
    }
  }
}

// C[m][n] (+)= sum_k A(m, k) B(n, k): the grad_weight (A = D^T, B = hidden,
// both MN-major) and grad_hidden (A = D K-major, B = weight MN-major)
// contractions.
template <bool AK, bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
    simt_gemm_kernel(const Operand a, const Operand b, float* __restrict__ c, int64_t ldc,
                     int accumulate, int c_vec) {
  __shared__ __align__(16) Stage st[2];
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;
  float acc[8][8];
  mainloop<AK, false, VEC>(a, b, m0, n0, st, acc);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t gm = m0 + tile_row(ty, i);
    if (gm >= a.mn_ext) continue;
    float* crow = c + gm * ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t gn = n0 + tile_col(tx, 4 * h);
      float* dst = crow + gn;
      if (c_vec && gn + 3 < b.mn_ext) {
        float4 v = make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2],
                               acc[i][4 * h + 3]);
        if (accumulate) {
          const float4 o = *reinterpret_cast<const float4*>(dst);
          v.x += o.x, v.y += o.y, v.z += o.z, v.w += o.w;
        }
        *reinterpret_cast<float4*>(dst) = v;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (gn + k < b.mn_ext) dst[k] = accumulate ? dst[k] + acc[i][4 * h + k] : acc[i][4 * h + k];
      }
    }
  }
}

bool al16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

}  // namespace

cudaError_t launch_simt_fwd(const SimtFwdParams& p, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((p.n + BM - 1) / BM),
                  static_cast<unsigned>((p.v + BN - 1) / BN));
  const bool vec = al16(p.hidden) && al16(p.weight) && p.h % 4 == 0;
  const int q_vec = (p.q != nullptr && al16(p.q) && p.v % 4 == 0) ? 1 : 0;
  if (vec)
    simt_fwd_kernel<true><<<grid, kThreads, 0, s>>>(p, q_vec);
  else
    simt_fwd_kernel<false><<<grid, kThreads, 0, s>>>(p, q_vec);
  return cudaGetLastError();
}

cudaError_t launch_simt_dlogits(const SimtDlogitsParams& p, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((p.n + BM - 1) / BM),
                  static_cast<unsigned>((p.width + BN - 1) / BN));
  const bool vec = al16(p.hidden) && al16(p.weight) && p.h % 4 == 0;
  const int q_vec = (p.q != nullptr && al16(p.q) && p.v % 4 == 0) ? 1 : 0;
  const int d_vec = (al16(p.d) && p.ldd % 4 == 0 && p.c0 % 4 == 0) ? 1 : 0;
  if (vec)
    simt_dlogits_kernel<true><<<grid, kThreads, 0, s>>>(p, q_vec, d_vec);
  else
    simt_dlogits_kernel<false><<<grid, kThreads, 0, s>>>(p, q_vec, d_vec);
  return cudaGetLastError();
}

cudaError_t launch_simt_gemm(int64_t m, int64_t n, int64_t k, const float* a, int64_t sam,
                             int64_t sak, const float* b, int64_t sbk, int64_t sbn, float* c,
                             int64_t ldc, int accumulate, cudaStream_t s) {
  if (sbn != 1 || (sam != 1 && sak != 1)) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>((n + BN - 1) / BN), static_cast<unsigned>((m + BM - 1) / BM));
  const Operand oa{a, sam, sak, m, k};
  const Operand ob{b, sbn, sbk, n, k};
  const bool a_k = sak == 1;
  const int64_t a_ld = a_k ? sam : sak;
  const bool vec = al16(a) && al16(b) && a_ld % 4 == 0 && sbk % 4 == 0;
  const int c_vec = (al16(c) && ldc % 4 == 0) ? 1 : 0;
  if (a_k && vec)
    simt_gemm_kernel<true, true><<<grid, kThreads, 0, s>>>(oa, ob, c, ldc, accumulate, c_vec);
  else if (a_k)
    simt_gemm_kernel<true, false><<<grid, kThreads, 0, s>>>(oa, ob, c, ldc, accumulate, c_vec);
  else if (vec)
    simt_gemm_kernel<false, true><<<grid, kThreads, 0, s>>>(oa, ob, c, ldc, accumulate, c_vec);
  else
    simt_gemm_kernel<false, false><<<grid, kThreads, 0, s>>>(oa, ob, c, ldc, accumulate, c_vec);
  return cudaGetLastError();
}

}  // namespace flce
