// Tensor-core kernels (sm_103a) of the fused linear cross-entropy and of the
// fused linear KL divergence.
//
// Four instances of the persistent tcgen05 GEMM (tc_gemm.cuh), one per
// contraction of the method ("fused-linear-ce" model card, §Algorithm):
//   fwd_stats   logits = hidden @ W^T per 256 x 256 pair tile, folded on the
//               fly into per-(row, vocabulary tile) softmax statistics;
//               nothing of size N x V is written.
//   bwd_dlogits the same logits recomputed for one vocabulary chunk, turned
//               into D = g (p - onehot) dz/dlin and stored in bf16.
//   grad_weight grad_W[chunk] = D^T @ hidden (K = tokens, fp32 in TMEM,
//               written once).
//   grad_hidden grad_h += D @ W[chunk] (K = chunk width), accumulated in an
//               fp32 buffer across chunks; the last chunk writes the input type.
// Each is instantiated for bf16 and for fp16 inputs (tcgen05 kind::f16 takes
// both, with A and B of one type). For fp16, D is stored scaled by a power of
// two so that its small entries stay in fp16's normal range; the two gradient
// GEMMs undo the scale in their epilogues.
//
// The KL divergence (FusedLinearKLDivLoss pull request, Liger-Kernel #1423,
// Details) runs the same four contractions; two epilogues differ:
//   fwd_kl          per (row, tile): the softmax statistics (m, s) and, from
//                   the teacher row, A = sum q (log max(q, eps) - z), Q = sum q;
//   bwd_dlogits_kl  D = g (p Q - q) / T.
// The file also holds the self-test kernel of the bounded waits.
#include <cfloat>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "flce_internal.h"
#include "flce_math.cuh"
#include "tc_gemm.cuh"

namespace flce {

namespace {

// 32 bias values of columns [c, c+32) (fewer when nv < 32; the rest are 0).
// T: the bias element type (16-bit, or float for split fp32 operands).
template <typename T>
__device__ __forceinline__ void load_bias32(const void* bias_v, int64_t c, int nv,
                                            float (&b)[32]) {
  const T* bias = static_cast<const T*>(bias_v);
  if (bias == nullptr) {
#pragma unroll
    for (int k = 0; k < 32; ++k) b[k] = 0.0f;
    return;
  }
  if constexpr (std::is_same_v<T, float>) {
    // the caller's fp32 bias need only be 4-byte aligned
    if (nv == 32 && (reinterpret_cast<uintptr_t>(bias + c) & 15u) == 0) {
      const float4* src = reinterpret_cast<const float4*>(bias + c);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 w = __ldg(src + q);
        b[4 * q] = w.x;
        b[4 * q + 1] = w.y;
        b[4 * q + 2] = w.z;
        b[4 * q + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) b[k] = (k < nv) ? __ldg(bias + c + k) : 0.0f;
    }
    return;
  } else if (nv == 32) {
    const uint4* src = reinterpret_cast<const uint4*>(bias + c);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = __ldg(src + q);
      const uint32_t parts[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        b[q * 8 + 2 * h] = Elem<T>::lo(parts[h]);
        b[q * 8 + 2 * h + 1] = Elem<T>::hi(parts[h]);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) b[k] = (k < nv) ? Elem<T>::to(bias[c + k]) : 0.0f;
  }
}

// 32 values rounded to T and stored with four 16-byte stores (dst 16-byte
// aligned), or element by element when only nv < 32 are in range.
template <typename T>
__device__ __forceinline__ void store32(T* dst, const float (&v)[32], int nv, float scale) {
  if (nv == 32) {
    uint4* dv = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      dv[q] = make_uint4(Elem<T>::pack2(v[q * 8 + 0] * scale, v[q * 8 + 1] * scale),
                         Elem<T>::pack2(v[q * 8 + 2] * scale, v[q * 8 + 3] * scale),
                         Elem<T>::pack2(v[q * 8 + 4] * scale, v[q * 8 + 5] * scale),
                         Elem<T>::pack2(v[q * 8 + 6] * scale, v[q * 8 + 7] * scale));
    }
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (k < nv) dst[k] = Elem<T>::from(v[k] * scale);
  }
}

// 32 fp32 values times scale, with 16-byte stores when dst is 16-byte aligned
// (a caller's fp32 buffer need only be 4-byte aligned), element by element
// otherwise or when only nv < 32 are in range.
__device__ __forceinline__ void store32_f32(float* dst, const float (&v)[32], int nv,
                                            float scale) {
  if (nv == 32 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
    float4* dv = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      dv[q] = make_float4(v[4 * q] * scale, v[4 * q + 1] * scale, v[4 * q + 2] * scale,
                          v[4 * q + 3] * scale);
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (k < nv) dst[k] = v[k] * scale;
  }
}

// Fold 32 logits (the first nv valid) of columns [cb, cb+32) into st. The
// chunk maximum is taken by a tree and the two sums of the chunk by four
// interleaved partial sums, so that the dependent chains are 5 and 8 long
// instead of 32 (the epilogue runs one warp per scheduler, so every step of
// a chain is a stall). ARGMAX: also track the lowest index of the maximum;
// ENTROPY: also keep t = sum e^{z-m} (z-m) (otherwise t is left as it was).
template <bool FULL, bool ARGMAX = true, bool ENTROPY = true>
__device__ __forceinline__ void fold_chunk(RowStats& st, const float (&z)[32], int nv, int cb) {
  float mx[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float lo = (FULL || 2 * k < nv) ? z[2 * k] : -FLT_MAX;
    const float hi = (FULL || 2 * k + 1 < nv) ? z[2 * k + 1] : -FLT_MAX;
    mx[k] = fmaxf(lo, hi);
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
    for (int k = 0; k < w; ++k) mx[k] = fmaxf(mx[k], mx[k + w]);
  }
  const float cm = mx[0];
  if (cm > st.m) {
    if constexpr (ARGMAX) {
      int kf = 0;
#pragma unroll
      for (int k = 31; k >= 0; --k) {
        if ((FULL || k < nv) && z[k] == cm) kf = k;
      }
      st.a = cb + kf;
    }
    st.rebase(cm);
  }
  float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float t4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if constexpr (FULL) {
    // two columns per instruction: d = z - m, e = 2^(d log2 e), s += e,
    // t += e d; the four running sums are two packed pairs
    const uint64_t nm2 = f2_pack(-st.m, -st.m), l2 = f2_pack(kLog2e, kLog2e);
    uint64_t sp[2] = {0, 0}, tp[2] = {0, 0};
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
      const uint64_t d = f2_add(f2_pack(z[k], z[k + 1]), nm2);
      float x0, x1;
      f2_unpack(f2_mul(d, l2), x0, x1);
      const uint64_t e = f2_pack(ex2_approx(x0), ex2_approx(x1));
      sp[(k >> 1) & 1] = f2_add(sp[(k >> 1) & 1], e);
      if constexpr (ENTROPY) tp[(k >> 1) & 1] = f2_fma(e, d, tp[(k >> 1) & 1]);
    }
    f2_unpack(sp[0], s4[0], s4[1]);
    f2_unpack(sp[1], s4[2], s4[3]);
    if constexpr (ENTROPY) {
      f2_unpack(tp[0], t4[0], t4[1]);
      f2_unpack(tp[1], t4[2], t4[3]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      if (k < nv) {
        const float d = z[k] - st.m;
        const float e = ex2_approx(d * kLog2e);
        s4[k & 3] += e;
        if constexpr (ENTROPY) t4[k & 3] = fmaf(e, d, t4[k & 3]);
      }
    }
  }
  st.s += (s4[0] + s4[1]) + (s4[2] + s4[3]);
  if constexpr (ENTROPY) st.t += (t4[0] + t4[1]) + (t4[2] + t4[3]);
}

// Lane l of the warp ends with the sum over the 32 lanes of v[l].
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// 32 entries q[c .. c+32) of one teacher row, fetched one chunk ahead of use.
// issue() starts the loads of a full, 16-byte aligned chunk as streaming
// (evict-first) loads: each teacher entry is read once, so it should not
// displace the weight and hidden tiles that other CTAs re-read from L2. A
// chunk that starts on a 32-byte boundary is read with two 32-byte loads (one
// whole sector each), else with four 16-byte ones. Each lane of a warp reads
// another row, so every load instruction touches 32 sectors: at the mid
// shape the 32-byte form takes 3-4 % off both KL GEMMs. get() unpacks the
// chunk; a partial or unaligned chunk is read there with scalar loads
// instead. Entries past nv (and every entry of an inactive row) are 0.
template <typename T>
struct RowChunk32 {
  static constexpr bool kF32 = std::is_same_v<T, float>;  // fp32 teacher (split operands)
  static constexpr int kVecs = kF32 ? 8 : 4;               // 16-byte vectors of a chunk
  uint4 w[kVecs];
  bool raw;

  __device__ __forceinline__ void issue(const T* row_ptr, int64_t c, int nv, bool vec,
                                        bool active) {
    raw = active && vec && nv == 32;
    if (raw) {
      const uint4* src = reinterpret_cast<const uint4*>(row_ptr + c);
      if ((reinterpret_cast<uintptr_t>(src) & 31u) == 0) {
#pragma unroll
        for (int r = 0; r < kVecs; r += 2) ld_cs_32B(src + r, w[r], w[r + 1]);
      } else {
#pragma unroll
        for (int r = 0; r < kVecs; ++r) w[r] = __ldcs(src + r);
      }
    }
  }

  __device__ __forceinline__ void get(const T* row_ptr, int64_t c, int nv, bool active,
                                      float (&q)[32]) const {
    if (raw) {
      if constexpr (kF32) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          q[4 * r] = __uint_as_float(w[r].x);
          q[4 * r + 1] = __uint_as_float(w[r].y);
          q[4 * r + 2] = __uint_as_float(w[r].z);
          q[4 * r + 3] = __uint_as_float(w[r].w);
        }
      } else {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const uint32_t parts[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            q[r * 8 + 2 * h] = Elem<T>::lo(parts[h]);
            q[r * 8 + 2 * h + 1] = Elem<T>::hi(parts[h]);
          }
        }
      }
    } else if (active) {
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        if constexpr (kF32)
          q[k] = (k < nv) ? row_ptr[c + k] : 0.0f;
        else
          q[k] = (k < nv) ? Elem<T>::to(row_ptr[c + k]) : 0.0f;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) q[k] = 0.0f;
    }
  }
};

// The tail every dlogits epilogue shares, per 32-column chunk `ch`: the 32
// values of D of this warp's 32 rows (times dscale, rounded to T; rows past
// the present ones hold d = 0) go through the warp's 2 KB staging buffer
// (row-major, 64 bytes a row) to a tensor store of one 32 x 32 box at column
// cb, row row0 of the chunk's buffer; the store leaves out rows past the
// buffer and columns past the chunk. When grad_bias partials are wanted,
// this warp's 32 column sums of D over its rows are left in ctl->red.
template <typename T>
__device__ __forceinline__ void emit_dlogits(float (&d)[32], const CUtensorMap* dmap,
                                             int64_t row0, int64_t buf_rows, int cb,
                                             float dscale, bool bias_sums, int ch, int quarter,
                                             int part, int lane, GemmCtl* ctl) {
  uint8_t* buf = ctl->out_stage + (part * 4 + quarter) * kDlogitsStageBytes;
  if (lane == 0) tma_store_wait_read();  // the warp's previous box has left the buffer
  __syncwarp();
  uint4* dst = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    dst[q] = make_uint4(Elem<T>::pack2(d[q * 8 + 0] * dscale, d[q * 8 + 1] * dscale),
                        Elem<T>::pack2(d[q * 8 + 2] * dscale, d[q * 8 + 3] * dscale),
                        Elem<T>::pack2(d[q * 8 + 4] * dscale, d[q * 8 + 5] * dscale),
                        Elem<T>::pack2(d[q * 8 + 6] * dscale, d[q * 8 + 7] * dscale));
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && row0 < buf_rows) {  // no box starts past the buffer's rows
    tma_store_2d(dmap, smem_addr(buf), cb, static_cast<int32_t>(row0));
    tma_store_commit();
  }
  if (bias_sums) ctl->red[quarter][ch][lane] = transpose_reduce32(d, lane);
}

// The same for D stored as its three bf16 parts (fp32 operands split into
// bf16 parts): hi = bf16(d), mid = bf16(d - hi), lo = d - hi - mid (exact), each
// staged in turn through the warp's buffer and stored to dmap (hi) and
// dmap_x[0], dmap_x[1] (mid, lo).
__device__ __forceinline__ void emit_dlogits_split(float (&d)[32], const CUtensorMap* dmap,
                                                   const CUtensorMap* dmap_x, int64_t row0,
                                                   int64_t buf_rows, int cb, bool bias_sums,
                                                   int ch, int quarter, int part, int lane,
                                                   GemmCtl* ctl) {
  uint8_t* buf = ctl->out_stage + (part * 4 + quarter) * kDlogitsStageBytes;
  float r[32];  // what the parts stored so far leave of d
#pragma unroll
  for (int k = 0; k < 32; ++k) r[k] = d[k];
#pragma unroll 1
  for (int q = 0; q < 3; ++q) {
    if (lane == 0) tma_store_wait_read();  // the previous box has left the buffer
    __syncwarp();
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const __nv_bfloat16 a = __float2bfloat16_rn(r[2 * k]);
      const __nv_bfloat16 b = __float2bfloat16_rn(r[2 * k + 1]);
      r[2 * k] -= __bfloat162float(a);
      r[2 * k + 1] -= __bfloat162float(b);
      w[k] = static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
    for (int g = 0; g < 4; ++g) dst[g] = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && row0 < buf_rows) {
      tma_store_2d(q == 0 ? dmap : dmap_x + (q - 1), smem_addr(buf), cb,
                   static_cast<int32_t>(row0));
      tma_store_commit();
    }
  }
  if (bias_sums) ctl->red[quarter][ch][lane] = transpose_reduce32(d, lane);
}

// After the chunks of a tile: grad_bias partials of the tile's columns, the
// sum of the four lane quarters' column sums in a fixed order. With W
// epilogue warps, warp (quarter, part) flushes chunks e * 8/W .. +8/W - 1,
// e = 4 part + quarter. One barrier per tile; the next tile's writes to
// ctl->red come after the epilogue warps' next common barrier (epi_all), so
// none overtakes these reads.
template <int W>
__device__ __forceinline__ void flush_bias_sums(float* gb_partial, int64_t gb_ld, int m_tile,
                                                int c0, int col0, int width, int quarter,
                                                int part, int lane, GemmCtl* ctl) {
  constexpr int kPer = (kBN / 32) / W;
  named_bar_sync(kEpiBar, 32 * W);
  const int first = (4 * part + quarter) * kPer;
#pragma unroll
  for (int ch = first; ch < first + kPer; ++ch) {
    const int col = col0 + ch * 32 + lane;
    if (col < width) {
      const float tot = ((ctl->red[0][ch][lane] + ctl->red[1][ch][lane]) + ctl->red[2][ch][lane]) +
                        ctl->red[3][ch][lane];
      gb_partial[static_cast<int64_t>(m_tile) * gb_ld + c0 + col] = tot;
    }
  }
}

}  // namespace

// ------------------------------------------------------------------ forward
// METRICS: also fold what the metrics need (the argmax and the entropy sum);
// without them the statistics are (m, s) only, and a and t stay at their
// initial values (the per-row correctness and entropy are then not computed).
// W = 8: two warps per TMEM lane quarter, each folding one 128-column half
// of the tile into its own statistics (partials per 128 columns; for short
// contractions, where the epilogue would outlast the MMAs).
// TB: the bias type (T, or float when the operands are fp32 split into bf16
// parts). A launch may cover one vocabulary chunk from column p.c0 (a
// multiple of 256): tiles, partial slots and columns are offset by it.
template <typename T, bool METRICS = true, int W = 4, typename TB = T>
struct EpiFwdStats {
  static constexpr uint32_t kABFormat = Elem<T>::kFormat;
  static constexpr int kEpiWarps = W;
  static constexpr bool kRelay = kEpiRelay && W == 4;
  static constexpr int kChunks = (kBN / 32) * 4 / W;  // 32-column chunks per warp
  using Params = FwdStatsParams;
  __device__ static void tile(const Params& p, int m_tile, int n_tile, AccSrc& acc,
                              int row_in_tile, int /*quarter*/, int part,
                              int /*lane*/,
                              GemmCtl* /*ctl*/) {
    const int64_t n_eff = p.n_rows_dyn != nullptr ? *p.n_rows_dyn : p.n_rows;
    const int64_t row = static_cast<int64_t>(m_tile) * kBM + row_in_tile;
    const bool row_ok = row < n_eff;
    const int64_t t = row_ok ? __ldg(p.targets + row) : INT64_MIN;
    const int64_t tile = p.c0 / kBN + n_tile;  // vocabulary tile of the whole row
    const int64_t col0 = tile * kBN;
    const int64_t slot = tile * (W / 4) + part;  // partials index
    RowStats st;
    st.init();
    float zt = 0.0f;
    float zs = 0.0f;  // sum of this part's logits (used for label smoothing)
    bool has_zt = false;
#pragma unroll 1
    for (int ch = part * kChunks; ch < (part + 1) * kChunks; ++ch) {
      const int64_t cb = col0 + ch * 32;
      if (cb >= p.v) break;
      const int nv = static_cast<int>(p.v - cb < 32 ? p.v - cb : 32);
      float z[32], b[32];
      acc.load(ch, z);
      load_bias32<TB>(p.bias, cb, nv, b);
      p.xf.apply32(z, b);
      if (nv == 32) {
        fold_chunk<true, METRICS, METRICS>(st, z, nv, static_cast<int>(cb));
      } else {
        fold_chunk<false, METRICS, METRICS>(st, z, nv, static_cast<int>(cb));
      }
      if (p.zsum != nullptr) {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (k < nv) zs += z[k];
      }
      const int64_t tk = t - cb;
      if (tk >= 0 && tk < nv) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (k == tk) zt = z[k];
        }
        has_zt = true;
      }
    }
    if (row_ok) {
      p.partials[row * p.n_vt + slot] = st.pack();
      if (p.zsum != nullptr) p.zsum[row * p.n_vt + slot] = zs;
      if (has_zt) p.zt[row] = zt;
    }
  }
};

// ------------------------------------------------------------------ dlogits
// W = 8: two warps per TMEM lane quarter, one per column half of the tile
// (for short contractions, where the epilogue would outlast the MMAs).
// TB: the bias type (T, or float for fp32 operands split into bf16 parts);
// DS: store D as its three bf16 parts (p.d_map, p.d_map_x).
template <typename T, int W = 4, typename TB = T, bool DS = false>
struct EpiDlogits {
  static constexpr uint32_t kABFormat = Elem<T>::kFormat;
  static constexpr int kEpiWarps = W;
  static constexpr bool kRelay = kEpiRelay && W == 4;
  static constexpr int kOutStageBytes = W * kDlogitsStageBytes;  // one buffer per warp
  static constexpr int kChunks = (kBN / 32) * 4 / W;  // 32-column chunks per warp
  using Params = DlogitsParams;
  __device__ static void tile(const Params& p, int m_tile, int n_tile, AccSrc& acc,
                              int row_in_tile, int quarter, int part,
                              int lane, GemmCtl* ctl) {
    const int64_t n_eff = p.n_rows_dyn != nullptr ? *p.n_rows_dyn : p.n_rows;
    const int64_t row = static_cast<int64_t>(m_tile) * kBM + row_in_tile;
    const bool row_ok = row < n_eff;
    const int64_t t = row_ok ? __ldg(p.targets + row) : p.ignore_index;
    const float g = row_ok ? row_grad(t, p.ignore_index, p.v, p.reduction, p.grad_out, p.n_valid, row)
                           : 0.0f;
    const float gs = g * p.xf.scale;
    const float lse_r = row_ok ? __ldg(p.lse + row) : 0.0f;
    const float lse2 = lse_r * kLog2e;
    // D/(g * dz/dlin) = p * (1 + 2 z_loss lse) - (1 - eps) [target] - eps / V
    const float pz = fmaf(2.0f * p.z_loss, lse_r, 1.0f);
    const float eps_v = p.label_smoothing / static_cast<float>(p.v);
    const float on_target = 1.0f - p.label_smoothing;
    const int64_t tl = t - p.c0;  // target column within this chunk
    const int col0 = n_tile * kBN;
    const float dscale = p.dscale != nullptr ? *p.dscale : 1.0f;
    // grad_bias column partials, for tiles holding present rows (uniform per tile)
    const bool bias_sums = p.gb_partial != nullptr && static_cast<int64_t>(m_tile) * kBM < n_eff;
#pragma unroll 1
    for (int ch = part * kChunks; ch < (part + 1) * kChunks; ++ch) {
      const int cb = col0 + ch * 32;
      if (cb >= p.width) break;
      const int nv = p.width - cb < 32 ? p.width - cb : 32;
      float z[32], b[32];
      acc.load(ch, z);
      load_bias32<TB>(p.bias, p.c0 + cb, nv, b);
      float d[32];
      p.xf.apply32(z, b);
      if (!p.xf.has_cap) {
        // two columns per instruction; dz/dlin = logit_scale (in gs)
        const uint64_t l2 = f2_pack(kLog2e, kLog2e), nl2 = f2_pack(-lse2, -lse2);
        const uint64_t pz2 = f2_pack(pz, pz), ne2 = f2_pack(-eps_v, -eps_v);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(z[k], z[k + 1]), l2, nl2), x0, x1);
          f2_unpack(f2_fma(f2_pack(ex2_approx(x0), ex2_approx(x1)), pz2, ne2), d[k], d[k + 1]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          d[k] = fmaf(ex2_approx(fmaf(z[k], kLog2e, -lse2)), pz, -eps_v);
      }
      const int64_t tk = tl - cb;
      if (tk >= 0 && tk < nv) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (k == tk) d[k] -= on_target;
        }
      }
      if (!row_ok) {
#pragma unroll
        for (int k = 0; k < 32; ++k) d[k] = 0.0f;
      } else if (!p.xf.has_cap) {
        const uint64_t g2 = f2_pack(gs, gs);
#pragma unroll
        for (int k = 0; k < 32; k += 2)
          f2_unpack(f2_mul(f2_pack(d[k], d[k + 1]), g2), d[k], d[k + 1]);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) d[k] = d[k] * gs * p.xf.dz_du(z[k]);
      }
      if constexpr (DS)
        emit_dlogits_split(d, &p.d_map, p.d_map_x,
                           static_cast<int64_t>(m_tile) * kBM + quarter * 32, p.n_rows, cb,
                           bias_sums, ch, quarter, part, lane, ctl);
      else
        emit_dlogits<T>(d, &p.d_map, static_cast<int64_t>(m_tile) * kBM + quarter * 32,
                        p.n_rows, cb, dscale, bias_sums, ch, quarter, part, lane, ctl);
    }
    if (bias_sums)
      flush_bias_sums<W>(p.gb_partial, p.gb_ld, m_tile, p.c0, col0, p.width, quarter, part,
                         lane, ctl);
  }
};

// ------------------------------------------------------------ KL forward
// W = 8: two warps per TMEM lane quarter, one per 128-column half, each with
// its own statistics (partials per 128 columns), as in EpiFwdStats.
// TB: the type of the bias and of the teacher probabilities (T, or float for
// fp32 operands split into bf16 parts); p.c0 as in EpiFwdStats.
template <typename T, int W = 4, typename TB = T>
struct EpiFwdKL {
  static constexpr uint32_t kABFormat = Elem<T>::kFormat;
  static constexpr int kEpiWarps = W;
  static constexpr bool kRelay = kEpiRelay && W == 4;
  static constexpr int kChunks = (kBN / 32) * 4 / W;  // 32-column chunks per warp
  using Params = FwdKLParams;
  __device__ static void tile(const Params& p, int m_tile, int n_tile, AccSrc& acc,
                              int row_in_tile, int /*quarter*/, int part,
                              int /*lane*/,
                              GemmCtl* /*ctl*/) {
    const int64_t n_eff = p.n_rows_dyn != nullptr ? *p.n_rows_dyn : p.n_rows;
    const int64_t row = static_cast<int64_t>(m_tile) * kBM + row_in_tile;
    const bool row_ok = row < n_eff;
    const int64_t orig = (row_ok && p.row_map != nullptr) ? p.row_map[row] : row;
    const TB* qrow = static_cast<const TB*>(p.q) + (row_ok ? orig : 0) * p.v;
    const int64_t tile = p.c0 / kBN + n_tile;  // vocabulary tile of the whole row
    const int64_t col0 = tile * kBN;
    const int64_t slot = tile * (W / 4) + part;  // partials index
    RowStats st;
    st.init();
    float a_sum = 0.0f;  // sum q (log max(q, eps) - z)
    float q_sum = 0.0f;  // sum q
    const bool vec = p.q_vec != 0;
    RowChunk32<TB> cur, nxt;
    const int ch_end = (part + 1) * kChunks;
    const int64_t c_first = col0 + part * kChunks * 32;
    if (c_first < p.v)
      cur.issue(qrow, c_first, p.v - c_first < 32 ? static_cast<int>(p.v - c_first) : 32, vec,
                row_ok);
#pragma unroll 1
    for (int ch = part * kChunks; ch < ch_end; ++ch) {
      const int64_t cb = col0 + ch * 32;
      if (cb >= p.v) break;
      const int nv = static_cast<int>(p.v - cb < 32 ? p.v - cb : 32);
      const int64_t cn = cb + 32;  // next chunk of this warp
      if (ch + 1 < ch_end && cn < p.v)
        nxt.issue(qrow, cn, p.v - cn < 32 ? static_cast<int>(p.v - cn) : 32, vec, row_ok);
      float z[32], b[32];
      acc.load(ch, z);
      load_bias32<TB>(p.bias, cb, nv, b);
      p.xf.apply32(z, b);
      if (nv == 32) {
        fold_chunk<true, false, false>(st, z, nv, static_cast<int>(cb));
      } else {
        fold_chunk<false, false, false>(st, z, nv, static_cast<int>(cb));
      }
      if (row_ok) {
        float q[32];
        cur.get(qrow, cb, nv, row_ok, q);  // 0 past nv
        float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f}, q4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          // q = 0 past nv adds exactly 0 (z there is finite: the accumulator
          // holds 0 for columns past V)
          a4[k & 3] = fmaf(q[k], __logf(fmaxf(q[k], p.eps)) - z[k], a4[k & 3]);
          q4[k & 3] += q[k];
        }
        a_sum += (a4[0] + a4[1]) + (a4[2] + a4[3]);
        q_sum += (q4[0] + q4[1]) + (q4[2] + q4[3]);
      }
      cur = nxt;
    }
    if (row_ok) p.partials[row * p.n_vt + slot] = make_float4(st.m, st.s, a_sum, q_sum);
  }
};

// ------------------------------------------------------------ KL dlogits
// D = g (p * sum_k q_k - q) * dz/dlin, with dz/dlin = 1 / temperature.
// TB: as in EpiFwdKL; DS: D stored as its three bf16 parts (see EpiDlogits).
template <typename T, int W = 4, typename TB = T, bool DS = false>
struct EpiDlogitsKL {
  static constexpr uint32_t kABFormat = Elem<T>::kFormat;
  static constexpr int kEpiWarps = W;
  static constexpr bool kRelay = kEpiRelay && W == 4;
  static constexpr int kOutStageBytes = W * kDlogitsStageBytes;
  static constexpr int kChunks = (kBN / 32) * 4 / W;  // 32-column chunks per warp
  using Params = DlogitsKLParams;
  __device__ static void tile(const Params& p, int m_tile, int n_tile, AccSrc& acc,
                              int row_in_tile, int quarter, int part,
                              int lane, GemmCtl* ctl) {
    const int64_t n_eff = p.n_rows_dyn != nullptr ? *p.n_rows_dyn : p.n_rows;
    const int64_t row = static_cast<int64_t>(m_tile) * kBM + row_in_tile;
    const bool row_ok = row < n_eff;
    const bool counted =
        row_ok && (p.labels == nullptr || __ldg(p.labels + row) != p.ignore_index);
    const float gs = kl_row_grad(counted, p.reduction, p.grad_out, p.n_counted, p.v, row) *
                     p.xf.scale;
    const float lse2 = row_ok ? __ldg(p.lse + row) * kLog2e : 0.0f;
    const float qs = row_ok ? __ldg(p.qsum + row) : 0.0f;
    const int64_t orig = (row_ok && p.row_map != nullptr) ? p.row_map[row] : row;
    const TB* qrow = static_cast<const TB*>(p.q) + (row_ok ? orig : 0) * p.v + p.c0;
    const int col0 = n_tile * kBN;
    const float dscale = p.dscale != nullptr ? *p.dscale : 1.0f;
    const bool bias_sums = p.gb_partial != nullptr && static_cast<int64_t>(m_tile) * kBM < n_eff;
    const bool vec = p.q_vec != 0;
    RowChunk32<TB> cur, nxt;
    const int ch_end = (part + 1) * kChunks;
    const int c_first = col0 + part * kChunks * 32;
    if (c_first < p.width)
      cur.issue(qrow, c_first, p.width - c_first < 32 ? p.width - c_first : 32, vec, row_ok);
#pragma unroll 1
    for (int ch = part * kChunks; ch < ch_end; ++ch) {
      const int cb = col0 + ch * 32;
      if (cb >= p.width) break;
      const int nv = p.width - cb < 32 ? p.width - cb : 32;
      const int cn = cb + 32;  // next chunk of this warp
      if (ch + 1 < ch_end && cn < p.width)
        nxt.issue(qrow, cn, p.width - cn < 32 ? p.width - cn : 32, vec, row_ok);
      float z[32], b[32], q[32];
      acc.load(ch, z);
      load_bias32<TB>(p.bias, p.c0 + cb, nv, b);
      cur.get(qrow, cb, nv, row_ok, q);
      float d[32];
      p.xf.apply32(z, b);
      if (!counted) {
#pragma unroll
        for (int k = 0; k < 32; ++k) d[k] = 0.0f;
      } else {
        // two columns per instruction (the KL divergence has no softcap, so
        // dz/dlin = 1/T is in gs)
        const uint64_t l2 = f2_pack(kLog2e, kLog2e), nl2 = f2_pack(-lse2, -lse2);
        const uint64_t qs2 = f2_pack(qs, qs), g2 = f2_pack(gs, gs);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(z[k], z[k + 1]), l2, nl2), x0, x1);
          const uint64_t pq = f2_fma(f2_pack(ex2_approx(x0), ex2_approx(x1)), qs2,
                                     f2_pack(-q[k], -q[k + 1]));
          f2_unpack(f2_mul(pq, g2), d[k], d[k + 1]);
        }
      }
      if constexpr (DS)
        emit_dlogits_split(d, &p.d_map, p.d_map_x,
                           static_cast<int64_t>(m_tile) * kBM + quarter * 32, p.n_rows, cb,
                           bias_sums, ch, quarter, part, lane, ctl);
      else
        emit_dlogits<T>(d, &p.d_map, static_cast<int64_t>(m_tile) * kBM + quarter * 32,
                        p.n_rows, cb, dscale, bias_sums, ch, quarter, part, lane, ctl);
      cur = nxt;
    }
    if (bias_sums)
      flush_bias_sums<W>(p.gb_partial, p.gb_ld, m_tile, p.c0, col0, p.width, quarter, part,
                         lane, ctl);
  }
};

// ------------------------------------------------------------ grad_weight
template <typename T>
struct EpiStoreRows {
  static constexpr uint32_t kABFormat = Elem<T>::kFormat;
  using Params = StoreRowsParams;
  __device__ static void tile(const Params& p, int m_tile, int n_tile, AccSrc& acc,
                              int row_in_tile, int, int, int, GemmCtl*) {
    const int64_t row = static_cast<int64_t>(m_tile) * kBM + row_in_tile;
    const bool row_ok = row < p.rows;
    const float scale = p.out_scale != nullptr ? *p.out_scale : 1.0f;
#pragma unroll 1
    for (int ch = 0; ch < kBN / 32; ++ch) {
      const int cb = n_tile * kBN + ch * 32;
      if (cb >= p.cols) break;
      float z[32];
      acc.load(ch, z);
      if (!row_ok) continue;
      const int nv = p.cols - cb < 32 ? p.cols - cb : 32;
      const int64_t off = (p.row0 + row) * p.ld + cb;
      if (p.out_f32) {
        store32_f32(static_cast<float*>(p.out) + off, z, nv, scale);
      } else {
        store32<T>(static_cast<T*>(p.out) + off, z, nv, scale);
      }
    }
  }
};

// ------------------------------------------------------------ grad_hidden
template <typename T>
struct EpiAccRows {
  static constexpr uint32_t kABFormat = Elem<T>::kFormat;
  using Params = AccRowsParams;
  __device__ static void tile(const Params& p, int m_tile, int n_tile, AccSrc& acc,
                              int row_in_tile, int, int, int, GemmCtl*) {
    const int64_t n_eff = p.rows_dyn != nullptr ? *p.rows_dyn : p.rows;
    const int64_t row = static_cast<int64_t>(m_tile) * kBM + row_in_tile;
    const bool row_ok = row < n_eff;
    // accumulator rows are in the (possibly compacted) row order; the final
    // output goes to row_map[row]
    const int64_t out_row = (row_ok && p.row_map != nullptr) ? p.row_map[row] : row;
    const float scale = p.out_scale != nullptr ? *p.out_scale : 1.0f;
#pragma unroll 1
    for (int ch = 0; ch < kBN / 32; ++ch) {
      const int cb = n_tile * kBN + ch * 32;
      if (cb >= p.cols) break;
      float z[32];
      acc.load(ch, z);
      if (!row_ok) continue;
      const int nv = p.cols - cb < 32 ? p.cols - cb : 32;
      const int64_t off = row * p.ld + cb;
      const int64_t out_off = out_row * p.ld + cb;
      if (p.out_scale != nullptr) {
#pragma unroll
        for (int k = 0; k < 32; ++k) z[k] *= scale;
      }
      if (p.mode == kAccAdd || p.mode == kAccAddOut) {
        const float* src = p.acc + off;
        if (nv == 32) {
          const float4* sv = reinterpret_cast<const float4*>(src);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 a = sv[q];
            z[4 * q] += a.x;
            z[4 * q + 1] += a.y;
            z[4 * q + 2] += a.z;
            z[4 * q + 3] += a.w;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (k < nv) z[k] += src[k];
        }
      }
      if (p.mode == kAccStore || p.mode == kAccAdd) {
        float* dst = p.acc + off;
        if (nv == 32) {
          float4* dv = reinterpret_cast<float4*>(dst);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dv[q] = make_float4(z[4 * q], z[4 * q + 1], z[4 * q + 2], z[4 * q + 3]);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (k < nv) dst[k] = z[k];
        }
      } else if (p.out_f32) {
        store32_f32(static_cast<float*>(p.out) + out_off, z, nv, 1.0f);
      } else {
        store32<T>(static_cast<T*>(p.out) + out_off, z, nv, 1.0f);
      }
    }
  }
};

// ------------------------------------------------------------ wait self-test
// One thread per CTA waits, through the GEMM pipeline's own bounded wait, on
// phase 0 of an mbarrier that nothing arrives on: the wait must give up after
// `budget_ns`, set FLCE_DEVERR_TIMEOUT in *err_word and return false, which
// the thread records in result[blockIdx.x] (0 = gave up, 1 = the phase
// completed). CG = 2 runs in clusters of two CTAs and uses the cluster-scope
// wait of the CTA-pair kernels. No tensor memory, copy or MMA is involved.
template <int CG>
__global__ void __launch_bounds__(32) wait_selftest_kernel(int* err_word, uint64_t budget_ns,
                                                            int* result) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = wait_bar<CG>(smem_addr(&bar), 0u, &abort_flag, err_word, budget_ns);
    result[blockIdx.x] = ok ? 1 : 0;
  }
}

cudaError_t launch_wait_selftest(int* err_word, uint64_t budget_ns, int* result, cudaStream_t s) {
  wait_selftest_kernel<1><<<1, 32, 0, s>>>(err_word, budget_ns, result);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, wait_selftest_kernel<2>, err_word, budget_ns, result + 1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ------------------------------------------------------------------ launchers
namespace {

// Persistent grid: one CTA (CG = 1) or one CTA pair (CG = 2) per resident
// slot, never more than there are tiles (of both segments).
template <int CG, class S0, class S1>
cudaError_t launch_gemm_args(const GemmArgs<S0, S1>& a, int sms, cudaStream_t stream) {
  auto kern = tc_gemm_kernel<CG, S0, S1>;
  constexpr int smem = gemm_smem_bytes<CG, typename S0::Epi, typename S1::Epi>();
  static_assert(smem <= 227 * 1024, "more shared memory than a CTA may have");
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3(gemm_threads<typename S0::Epi>(), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  int units = sms;
  if constexpr (CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int max_clusters[64] = {0};  // resident pairs, per device
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (max_clusters[dev] == 0) {
      cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n < 1) return cudaErrorInvalidConfiguration;
      max_clusters[dev] = n;
    }
    units = max_clusters[dev];
  }
  int64_t total = static_cast<int64_t>(a.g0.m_tiles) * a.g0.n_tiles;
  if constexpr (S1::kPresent) total += static_cast<int64_t>(a.g1.m_tiles) * a.g1.n_tiles;
  const int64_t grid_units = total < units ? total : units;
  if (grid_units < 1) return cudaSuccess;
  cfg.gridDim = dim3(static_cast<unsigned>(grid_units * CG), 1, 1);
  if (a.g0.pdl != 0) {
    // may start while the previous kernel of the stream drains (see GemmGeom::pdl)
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// One GEMM (one segment), statically scheduled unless g.sched is set.
template <int CG, bool A_MN, bool B_MN, class Epi>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const GemmGeom& g,
                        const typename Epi::Params& ep, int sms, cudaStream_t stream) {
  GemmArgs<Seg<A_MN, B_MN, Epi>, NoSeg> a{};
  a.a0 = ta;
  a.b0 = tb;
  a.g0 = g;
  a.ep0 = ep;
  return launch_gemm_args<CG>(a, sms, stream);
}

// One GEMM over split operands: parts[0] of A and B in the segment's own
// maps, parts 1 and 2 (mid, lo) in the extra maps; g.passes / pass_a /
// pass_b say which part pairs the contraction runs over.
template <int CG, bool A_MN, bool B_MN, class Epi>
cudaError_t launch_gemm_split(const CUtensorMap (&ta)[3], const CUtensorMap (&tb)[3],
                              const GemmGeom& g, const typename Epi::Params& ep, int sms,
                              cudaStream_t stream) {
  GemmArgs<Seg<A_MN, B_MN, Epi, true>, NoSeg> a{};
  a.a0 = ta[0];
  a.b0 = tb[0];
  a.x0.a[0] = ta[1];
  a.x0.a[1] = ta[2];
  a.x0.b[0] = tb[1];
  a.x0.b[1] = tb[2];
  a.g0 = g;
  a.ep0 = ep;
  return launch_gemm_args<CG>(a, sms, stream);
}

// grad_hidden (D K-major times W MN-major, accumulated rows) and grad_weight
// (D^T times hidden, both MN-major, stored rows) of one vocabulary chunk in
// one dynamically scheduled launch; the segment with the longer contraction
// goes first so that its tiles are handed out before the shorter ones.
template <typename T>
cudaError_t launch_grads_typed(const GradsLaunch& l, int sms, cudaStream_t s) {
  using GH = Seg<false, true, EpiAccRows<T>>;
  using GW = Seg<true, true, EpiStoreRows<T>>;
  if (l.gh_first) {
    GemmArgs<GH, GW> a{};
    a.a0 = l.tm_d_k;
    a.b0 = l.tm_weight_mn;
    a.g0 = l.g_gh;
    a.ep0 = l.ap;
    a.a1 = l.tm_d_mn;
    a.b1 = l.tm_hidden_mn;
    a.g1 = l.g_gw;
    a.ep1 = l.sp;
    a.g0.sched = l.sched;
    return launch_gemm_args<kPairCG>(a, sms, s);
  }
  GemmArgs<GW, GH> a{};
  a.a0 = l.tm_d_mn;
  a.b0 = l.tm_hidden_mn;
  a.g0 = l.g_gw;
  a.ep0 = l.sp;
  a.a1 = l.tm_d_k;
  a.b1 = l.tm_weight_mn;
  a.g1 = l.g_gh;
  a.ep1 = l.ap;
  a.g0.sched = l.sched;
  return launch_gemm_args<kPairCG>(a, sms, s);
}

}  // namespace

cudaError_t launch_tc_fwd_stats(int type, const CUtensorMap& tm_hidden_k,
                                const CUtensorMap& tm_weight_k, const GemmGeom& g,
                                const FwdStatsParams& p, int epi_warps, int sms, cudaStream_t s) {
  const bool f16 = type == kTcF16;
  if (epi_warps == 8) {
    if (p.metrics)
      return f16 ? launch_gemm<kPairCG, false, false, EpiFwdStats<__half, true, 8>>(
                       tm_hidden_k, tm_weight_k, g, p, sms, s)
                 : launch_gemm<kPairCG, false, false, EpiFwdStats<__nv_bfloat16, true, 8>>(
                       tm_hidden_k, tm_weight_k, g, p, sms, s);
    return f16 ? launch_gemm<kPairCG, false, false, EpiFwdStats<__half, false, 8>>(
                     tm_hidden_k, tm_weight_k, g, p, sms, s)
               : launch_gemm<kPairCG, false, false, EpiFwdStats<__nv_bfloat16, false, 8>>(
                     tm_hidden_k, tm_weight_k, g, p, sms, s);
  }
  if (p.metrics)
    return f16 ? launch_gemm<kPairCG, false, false, EpiFwdStats<__half, true>>(
                     tm_hidden_k, tm_weight_k, g, p, sms, s)
               : launch_gemm<kPairCG, false, false, EpiFwdStats<__nv_bfloat16, true>>(
                     tm_hidden_k, tm_weight_k, g, p, sms, s);
  return f16 ? launch_gemm<kPairCG, false, false, EpiFwdStats<__half, false>>(
                   tm_hidden_k, tm_weight_k, g, p, sms, s)
             : launch_gemm<kPairCG, false, false, EpiFwdStats<__nv_bfloat16, false>>(
                   tm_hidden_k, tm_weight_k, g, p, sms, s);
}

cudaError_t launch_tc_fwd_stats_split(const CUtensorMap (&tm_hidden_k)[3],
                                      const CUtensorMap (&tm_weight_k)[3], const GemmGeom& g,
                                      const FwdStatsParams& p, int epi_warps, int sms,
                                      cudaStream_t s) {
  using B = __nv_bfloat16;
  if (epi_warps == 8) {
    if (p.metrics)
      return launch_gemm_split<kPairCG, false, false, EpiFwdStats<B, true, 8, float>>(
          tm_hidden_k, tm_weight_k, g, p, sms, s);
    return launch_gemm_split<kPairCG, false, false, EpiFwdStats<B, false, 8, float>>(
        tm_hidden_k, tm_weight_k, g, p, sms, s);
  }
  if (p.metrics)
    return launch_gemm_split<kPairCG, false, false, EpiFwdStats<B, true, 4, float>>(
        tm_hidden_k, tm_weight_k, g, p, sms, s);
  return launch_gemm_split<kPairCG, false, false, EpiFwdStats<B, false, 4, float>>(
      tm_hidden_k, tm_weight_k, g, p, sms, s);
}

cudaError_t launch_tc_dlogits(int type, const CUtensorMap& tm_hidden_k,
                              const CUtensorMap& tm_weight_k, const GemmGeom& g,
                              const DlogitsParams& p, int epi_warps, int sms, cudaStream_t s) {
  if (epi_warps == 8) {
    if (type == kTcF16)
      return launch_gemm<kPairCG, false, false, EpiDlogits<__half, 8>>(tm_hidden_k, tm_weight_k,
                                                                        g, p, sms, s);
    return launch_gemm<kPairCG, false, false, EpiDlogits<__nv_bfloat16, 8>>(
        tm_hidden_k, tm_weight_k, g, p, sms, s);
  }
  if (type == kTcF16)
    return launch_gemm<kPairCG, false, false, EpiDlogits<__half>>(tm_hidden_k, tm_weight_k, g, p,
                                                                   sms, s);
  return launch_gemm<kPairCG, false, false, EpiDlogits<__nv_bfloat16>>(tm_hidden_k, tm_weight_k,
                                                                        g, p, sms, s);
}

cudaError_t launch_tc_fwd_kl(int type, const CUtensorMap& tm_hidden_k,
                             const CUtensorMap& tm_weight_k, const GemmGeom& g,
                             const FwdKLParams& p, int epi_warps, int sms, cudaStream_t s) {
  const bool f16 = type == kTcF16;
  if (epi_warps == 8)
    return f16 ? launch_gemm<kPairCG, false, false, EpiFwdKL<__half, 8>>(tm_hidden_k,
                                                                          tm_weight_k, g, p,
                                                                          sms, s)
               : launch_gemm<kPairCG, false, false, EpiFwdKL<__nv_bfloat16, 8>>(
                     tm_hidden_k, tm_weight_k, g, p, sms, s);
  return f16 ? launch_gemm<kPairCG, false, false, EpiFwdKL<__half>>(tm_hidden_k, tm_weight_k, g,
                                                                     p, sms, s)
             : launch_gemm<kPairCG, false, false, EpiFwdKL<__nv_bfloat16>>(tm_hidden_k,
                                                                            tm_weight_k, g, p,
                                                                            sms, s);
}

cudaError_t launch_tc_dlogits_kl(int type, const CUtensorMap& tm_hidden_k,
                                 const CUtensorMap& tm_weight_k, const GemmGeom& g,
                                 const DlogitsKLParams& p, int epi_warps, int sms,
                                 cudaStream_t s) {
  if (epi_warps == 8) {
    if (type == kTcF16)
      return launch_gemm<kPairCG, false, false, EpiDlogitsKL<__half, 8>>(tm_hidden_k, tm_weight_k,
                                                                          g, p, sms, s);
    return launch_gemm<kPairCG, false, false, EpiDlogitsKL<__nv_bfloat16, 8>>(
        tm_hidden_k, tm_weight_k, g, p, sms, s);
  }
  if (type == kTcF16)
    return launch_gemm<kPairCG, false, false, EpiDlogitsKL<__half>>(tm_hidden_k, tm_weight_k, g,
                                                                     p, sms, s);
  return launch_gemm<kPairCG, false, false, EpiDlogitsKL<__nv_bfloat16>>(tm_hidden_k,
                                                                          tm_weight_k, g, p,
                                                                          sms, s);
}

cudaError_t launch_tc_grads(int type, const GradsLaunch& l, int sms, cudaStream_t s) {
  if (type == kTcF16) return launch_grads_typed<__half>(l, sms, s);
  return launch_grads_typed<__nv_bfloat16>(l, sms, s);
}

cudaError_t launch_tc_dlogits_split(const CUtensorMap (&tm_hidden_k)[3],
                                    const CUtensorMap (&tm_weight_k)[3], const GemmGeom& g,
                                    const DlogitsParams& p, int epi_warps, int sms,
                                    cudaStream_t s) {
  using B = __nv_bfloat16;
  if (epi_warps == 8)
    return launch_gemm_split<kPairCG, false, false, EpiDlogits<B, 8, float, true>>(
        tm_hidden_k, tm_weight_k, g, p, sms, s);
  return launch_gemm_split<kPairCG, false, false, EpiDlogits<B, 4, float, true>>(
      tm_hidden_k, tm_weight_k, g, p, sms, s);
}

cudaError_t launch_tc_fwd_kl_split(const CUtensorMap (&tm_hidden_k)[3],
                                   const CUtensorMap (&tm_weight_k)[3], const GemmGeom& g,
                                   const FwdKLParams& p, int epi_warps, int sms, cudaStream_t s) {
  using B = __nv_bfloat16;
  if (epi_warps == 8)
    return launch_gemm_split<kPairCG, false, false, EpiFwdKL<B, 8, float>>(tm_hidden_k,
                                                                           tm_weight_k, g, p,
                                                                           sms, s);
  return launch_gemm_split<kPairCG, false, false, EpiFwdKL<B, 4, float>>(tm_hidden_k,
                                                                         tm_weight_k, g, p,
                                                                         sms, s);
}

cudaError_t launch_tc_dlogits_kl_split(const CUtensorMap (&tm_hidden_k)[3],
                                       const CUtensorMap (&tm_weight_k)[3], const GemmGeom& g,
                                       const DlogitsKLParams& p, int epi_warps, int sms,
                                       cudaStream_t s) {
  using B = __nv_bfloat16;
  if (epi_warps == 8)
    return launch_gemm_split<kPairCG, false, false, EpiDlogitsKL<B, 8, float, true>>(
        tm_hidden_k, tm_weight_k, g, p, sms, s);
  return launch_gemm_split<kPairCG, false, false, EpiDlogitsKL<B, 4, float, true>>(
      tm_hidden_k, tm_weight_k, g, p, sms, s);
}

// The fused gradient launch over split operands (as launch_grads_typed).
cudaError_t launch_tc_grads_split(const GradsSplitLaunch& l, int sms, cudaStream_t s) {
  using B = __nv_bfloat16;
  using GH = Seg<false, true, EpiAccRows<B>, true>;
  using GW = Seg<true, true, EpiStoreRows<B>, true>;
  auto fill_gh = [&](auto& a, auto& maps_a, auto& maps_b, CUtensorMap& ta, CUtensorMap& tb) {
    ta = l.d_k[0];
    tb = l.weight_mn[0];
    maps_a[0] = l.d_k[1];
    maps_a[1] = l.d_k[2];
    maps_b[0] = l.weight_mn[1];
    maps_b[1] = l.weight_mn[2];
    (void)a;
  };
  auto fill_gw = [&](auto& a, auto& maps_a, auto& maps_b, CUtensorMap& ta, CUtensorMap& tb) {
    ta = l.d_mn[0];
    tb = l.hidden_mn[0];
    maps_a[0] = l.d_mn[1];
    maps_a[1] = l.d_mn[2];
    maps_b[0] = l.hidden_mn[1];
    maps_b[1] = l.hidden_mn[2];
    (void)a;
  };
  if (l.gh_first) {
    GemmArgs<GH, GW> a{};
    fill_gh(a, a.x0.a, a.x0.b, a.a0, a.b0);
    fill_gw(a, a.x1.a, a.x1.b, a.a1, a.b1);
    a.g0 = l.g_gh;
    a.ep0 = l.ap;
    a.g1 = l.g_gw;
    a.ep1 = l.sp;
    a.g0.sched = l.sched;
    return launch_gemm_args<kPairCG>(a, sms, s);
  }
  GemmArgs<GW, GH> a{};
  fill_gw(a, a.x0.a, a.x0.b, a.a0, a.b0);
  fill_gh(a, a.x1.a, a.x1.b, a.a1, a.b1);
  a.g0 = l.g_gw;
  a.ep0 = l.sp;
  a.g1 = l.g_gh;
  a.ep1 = l.ap;
  a.g0.sched = l.sched;
  return launch_gemm_args<kPairCG>(a, sms, s);
}

}  // namespace flce
