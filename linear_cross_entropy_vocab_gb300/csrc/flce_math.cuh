// Device math shared by the CUDA kernels of the fused linear cross-entropy
// and KL divergence: the logit transform (bias, logit_scale, softcap), the
// running softmax statistics a vocabulary sweep keeps per row and their
// merge, the upstream gradient of a row, and packed-pair fp32 arithmetic.
//
// "fused-linear-ce" model card (trl-lib), §Algorithm: each logit tile gets
// bias / logit_scale / softcap and is folded into a running log-sum-exp with
// the online-softmax rescaling; §Metrics for free: the argmax rides along with
// the running maximum and the entropy term sum_j p_j z_j uses the same
// rescaling.
//
// Running statistics of a set of logits z_j with maximum m:
//   s = sum_j e^{z_j - m}            (so lse = m + log s)
//   t = sum_j e^{z_j - m} (z_j - m)  (so sum_j p_j z_j = m + t/s, and the
//                                     entropy is lse - m - t/s = log s - t/s)
//   a = lowest index j with z_j = m
// Keeping t relative to the running maximum avoids the cancellation of
// sum_j p_j z_j against lse when the logits are large.
#pragma once

#include <cfloat>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_ptx.cuh"

namespace flce {

constexpr float kLog2e = 1.4426950408889634f;

// tanh from its exponential form tanh(x) = (e^{2x} - 1) / (e^{2x} + 1),
// with |x| clamped to 9 (tanh(9) rounds to 1 in fp32). Absolute error is a
// few 1e-7.
__device__ __forceinline__ float tanh_exp2(float x) {
  x = fminf(fmaxf(x, -9.0f), 9.0f);
  const float e = ex2_approx(x * (2.0f * kLog2e));
  return __fdividef(e - 1.0f, e + 1.0f);
}

// Packed pairs of fp32 values (the .f32x2 arithmetic of sm_100-family GPUs):
// one instruction adds, multiplies or fused-multiply-adds two lanes, each
// rounded as the scalar instruction would round it.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

struct LogitXform {
  float scale;
  float softcap;      // used only if has_cap
  float inv_softcap;  // 1 / softcap
  int has_cap;

  // z = softcap(scale * (acc + b)); b is 0 without a bias.
  __device__ __forceinline__ float operator()(float acc, float b) const {
    const float u = scale * (acc + b);
    if (has_cap) return softcap * tanh_exp2(u * inv_softcap);
    return u;
  }
  // The transform of 32 accumulator values in place, two at a time where
  // there is no softcap (the same roundings as operator()).
  __device__ __forceinline__ void apply32(float (&z)[32], const float (&b)[32]) const {
    if (has_cap) {
#pragma unroll
      for (int k = 0; k < 32; ++k) z[k] = (*this)(z[k], b[k]);
      return;
    }
    const uint64_t s2 = f2_pack(scale, scale);
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
      const uint64_t u = f2_mul(s2, f2_add(f2_pack(z[k], z[k + 1]), f2_pack(b[k], b[k + 1])));
      f2_unpack(u, z[k], z[k + 1]);
    }
  }
  // dz/du at final logit z: 1 - (z/softcap)^2 with a softcap, else 1.
  __device__ __forceinline__ float dz_du(float z) const {
    if (!has_cap) return 1.0f;
    const float q = z * inv_softcap;
    return fmaf(-q, q, 1.0f);
  }
};

// Running statistics of one row over part of the vocabulary.
struct RowStats {
  float m;  // running maximum (starts at -FLT_MAX: finite, so no inf - inf)
  float s;  // sum e^{z - m}
  float t;  // sum e^{z - m} (z - m)
  int a;    // lowest index reaching m

  __device__ __forceinline__ void init() {
    m = -FLT_MAX;
    s = 0.0f;
    t = 0.0f;
    a = 0x7fffffff;
  }

  // Move the reference maximum to m_new >= m.
  __device__ __forceinline__ void rebase(float m_new) {
    const float dm = m - m_new;  // <= 0
    const float alpha = ex2_approx(dm * kLog2e);
    t = alpha * fmaf(s, dm, t);
    s = alpha * s;
    m = m_new;
  }

  // Add one logit (its maximum must already be folded in by rebase).
  __device__ __forceinline__ void add(float z) {
    const float d = z - m;
    const float e = ex2_approx(d * kLog2e);
    s += e;
    t = fmaf(e, d, t);
  }

  __device__ __forceinline__ float4 pack() const {
    return make_float4(m, s, t, __int_as_float(a));
  }
  __device__ __forceinline__ static RowStats unpack(float4 v) {
    RowStats r;
    r.m = v.x;
    r.s = v.y;
    r.t = v.z;
    r.a = __float_as_int(v.w);
    return r;
  }
};

// Merge two partial statistics. Ties of the maximum go to the lower index,
// so the merged argmax is the lowest index reaching the overall maximum
// whatever the merge order.
__device__ __forceinline__ RowStats merge_stats(const RowStats& x, const RowStats& y) {
  RowStats r;
  r.m = fmaxf(x.m, y.m);
  if (y.m > x.m || (y.m == x.m && y.a < x.a)) {
    r.a = y.a;
  } else {
    r.a = x.a;
  }
  const float dx = x.m - r.m, dy = y.m - r.m;
  const float ax = ex2_approx(dx * kLog2e), ay = ex2_approx(dy * kLog2e);
  r.s = ax * x.s + ay * y.s;
  r.t = ax * fmaf(x.s, dx, x.t) + ay * fmaf(y.s, dy, y.t);
  return r;
}

__device__ __forceinline__ RowStats shfl_xor_stats(const RowStats& x, int mask) {
  RowStats r;
  r.m = __shfl_xor_sync(0xffffffffu, x.m, mask);
  r.s = __shfl_xor_sync(0xffffffffu, x.s, mask);
  r.t = __shfl_xor_sync(0xffffffffu, x.t, mask);
  r.a = __shfl_xor_sync(0xffffffffu, x.a, mask);
  return r;
}

// Upstream gradient of row `row`'s loss term: grad_out/n_valid ("mean"),
// grad_out ("sum"), grad_out[row] ("none"); 0 for ignored rows and rows
// whose target is outside [0, V).
__device__ __forceinline__ float row_grad(int64_t t, int64_t ignore_index, int64_t v,
                                          int reduction, const float* grad_out,
                                          const int32_t* n_valid, int64_t row) {
  if (t == ignore_index || t < 0 || t >= v) return 0.0f;
  if (reduction == 0) return grad_out[row];           // none
  if (reduction == 1) return grad_out[0];             // sum
  return grad_out[0] / static_cast<float>(n_valid[0]);  // mean (n_valid >= 1 here)
}

// Upstream gradient of row `row`'s KL term (reduction codes: 0 none, 1 sum,
// 2 batchmean, 3 mean); 0 for rows not counted.
__device__ __forceinline__ float kl_row_grad(bool counted, int reduction, const float* grad_out,
                                             const int32_t* n_counted, int64_t v, int64_t row) {
  if (!counted) return 0.0f;
  if (reduction == 0) return grad_out[row];
  float g = grad_out[0];
  if (reduction >= 2) g /= static_cast<float>(n_counted[0]);  // n_counted >= 1 here
  if (reduction == 3) g /= static_cast<float>(v);
  return g;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The 16-bit input types: conversion and the tcgen05 operand-format code.
template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
  static constexpr uint32_t kFormat = 1;
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    return pack_bf16x2(lo, hi);
  }
  __device__ __forceinline__ static __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
  __device__ __forceinline__ static float lo(uint32_t w) {
    return __low2float(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
  __device__ __forceinline__ static float hi(uint32_t w) {
    return __high2float(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
  __device__ __forceinline__ static float to(__nv_bfloat16 x) { return __bfloat162float(x); }
};

template <>
struct Elem<__half> {
  static constexpr uint32_t kFormat = 0;
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static __half from(float x) { return __float2half_rn(x); }
  __device__ __forceinline__ static float lo(uint32_t w) {
    return __low2float(*reinterpret_cast<const __half2*>(&w));
  }
  __device__ __forceinline__ static float hi(uint32_t w) {
    return __high2float(*reinterpret_cast<const __half2*>(&w));
  }
  __device__ __forceinline__ static float to(__half x) { return __half2float(x); }
};

}  // namespace flce
