// Persistent, warp-specialised tcgen05 GEMM main loop with pluggable
// epilogues, for sm_103a.
//
//   D[tile] = sum_k A[m, k] * B[n, k]      (bf16 in, fp32 accumulate in TMEM)
//
// CG = 1: one CTA computes a 128 x 256 tile (tcgen05.mma.cta_group::1).
// CG = 2: a cluster of two CTAs computes a 256 x 256 tile with
//   tcgen05.mma.cta_group::2 issued by the even CTA: each CTA stages its own
//   128 rows of A and 128 of the 256 rows of B, and receives its 128 rows of
//   D in its own TMEM. Per flop, each SM stages a third less operand data,
//   which leaves room for a deeper (6-stage) copy ring.
//
// Roles of the 192 threads of a CTA (one CTA per SM, persistent over tiles):
//   warp 0   one thread issues TMA tile loads into the stage ring
//   warp 1   allocates tensor memory; one thread (of the even CTA) issues the
//            MMAs and commits them to mbarriers
//   warps 2-5  the epilogue: each thread owns one accumulator row (TMEM
//            lane), pulls its 256 fp32 columns with tcgen05.ld and hands them
//            to the epilogue policy.
// An epilogue may ask for 8 warps (320 threads): warps 2-9, two per TMEM lane
// quarter, each pulling one 128-column half of its rows.
// The 512 TMEM columns hold two 128 x 256 fp32 accumulators per CTA, so the
// epilogue of tile i overlaps the MMAs of tile i+1.
//
// Each operand is K-major (rows of K contiguous elements) or MN-major (K rows
// of contiguous M or N elements); both are staged with 128-byte swizzle:
//   K-major:  one TMA box {64 (K), rows}; 8-row groups 1024 B apart.
//   MN-major: boxes {64 (M/N), 64 (K)} of 8 KB each, side by side along M/N.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda.h>

#include "tc_ptx.cuh"

namespace flce {

constexpr int kBM = 128;  // accumulator rows per CTA = TMEM lanes
constexpr int kBN = 256;  // accumulator columns per buffer
constexpr int kBK = 64;   // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kUK = 16;   // K per tcgen05.mma (kind::f16)
constexpr int kEpiWarps = 4;  // epilogue warps unless the epilogue declares kEpiWarps = 8
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr int kMaxStages = 6;

template <int CG>
struct TileCfg {
  static constexpr int kBNLoad = kBN / CG;  // rows of B staged per CTA
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = kBNLoad * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = CG == 1 ? 4 : 6;
  static constexpr int kTileRows = kBM * CG;  // M rows of one (pair) tile
};

struct GemmCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  float red[4][kBN / 32][32];  // epilogue scratch: per-warp column sums, [quarter][chunk][lane]
};

template <int CG>
constexpr int gemm_smem_bytes() {
  return TileCfg<CG>::kStages * TileCfg<CG>::kStageBytes + 1024 /* alignment slack */ +
         ((static_cast<int>(sizeof(GemmCtl)) + 127) / 128) * 128;
}

// Tile grid and TMA coordinate offsets of one GEMM launch. m_tiles counts
// tiles of TileCfg<CG>::kTileRows rows.
struct GemmGeom {
  int m_tiles, n_tiles, k_iters;
  int m_fastest;  // 1: tile u -> (u % m_tiles, u / m_tiles); 0: n fastest
  int a_mn0, a_k0;  // A: offset along M and along K (elements / rows)
  int b_mn0, b_k0;  // B: offset along N and along K
  // Optional device-side row count: when non-null, the M extent (axis 0) or
  // the K extent (axis 1) is *dyn_rows rows, at most the static extent. It is
  // read at kernel start, so the host needs no synchronisation to learn it.
  const int32_t* dyn_rows;
  int dyn_axis;
  // When > 0, tiles are taken in bands: with m_fastest, bands of `group`
  // M-tiles (all N-tiles of a band before the next band); otherwise bands of
  // `group` N-tiles (all M-tiles of a band before the next). The
  // tiles in flight then share fewer rows of the operand that every tile of
  // the other axis reuses, which keeps it in L2.
  int group;
  int* err_word;
};

__device__ __forceinline__ void tile_coords(const GemmGeom& g, int m_tiles, int u, int& m,
                                            int& n) {
  if (g.m_fastest) {
    if (g.group > 0 && g.group < m_tiles) {
      const int band = g.group * g.n_tiles;
      const int first = (u / band) * g.group;
      const int rows = m_tiles - first < g.group ? m_tiles - first : g.group;
      const int r = u % band;
      m = first + r % rows;
      n = r / rows;
    } else {
      m = u % m_tiles;
      n = u / m_tiles;
    }
  } else {
    if (g.group > 0 && g.group < g.n_tiles) {
      const int band = g.group * m_tiles;
      const int first = (u / band) * g.group;
      const int cols = g.n_tiles - first < g.group ? g.n_tiles - first : g.group;
      const int r = u % band;
      n = first + r % cols;
      m = r / cols;
    } else {
      n = u % g.n_tiles;
      m = u / g.n_tiles;
    }
  }
}

// 32 accumulator columns, or zeros when the contraction was empty (K = 0).
__device__ __forceinline__ void load_acc(uint32_t taddr, float (&v)[32], bool zero) {
  if (zero) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.0f;
  } else {
    tmem_load_32cols(taddr, v);
  }
}

template <int CG, bool MN, int ROWS>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             int mn0, int k0) {
  if constexpr (!MN) {
    if constexpr (CG == 1)
      tma_load_2d(dst, map, bar, k0, mn0);  // box {64 along K, ROWS}
    else
      tma_load_2d_pair(dst, map, bar, k0, mn0);
  } else {
#pragma unroll
    for (int b = 0; b < ROWS / 64; ++b) {  // boxes {64 along M/N, 64 along K}
      if constexpr (CG == 1)
        tma_load_2d(dst + b * 8192, map, bar, mn0 + b * 64, k0);
      else
        tma_load_2d_pair(dst + b * 8192, map, bar, mn0 + b * 64, k0);
    }
  }
}

// Epilogue warps of Epi: Epi::kEpiWarps where it declares one, else 4. With
// 8, warps w and w + 4 share TMEM lane quarter w % 4 and split the tile's
// columns into halves (`part` 0 and 1).
template <class Epi, class = void>
struct EpiWarps {
  static constexpr int value = kEpiWarps;
};
template <class Epi>
struct EpiWarps<Epi, std::void_t<decltype(Epi::kEpiWarps)>> {
  static constexpr int value = Epi::kEpiWarps;
};
// Threads per CTA: the TMA warp, the MMA warp and the epilogue warps.
template <class Epi>
constexpr int gemm_threads() {
  return 64 + 32 * EpiWarps<Epi>::value;
}

// Descriptor of the kk-th K=16 slice of a staged operand.
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
  if constexpr (!MN) {
    return smem_desc_sw128(base + kk * (kUK * 2), 16, 1024);
  } else {
    return smem_desc_sw128(base + kk * (kUK * 128), 8192, 1024);
  }
}

template <int CG>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* err_word, uint64_t budget_ns = kWaitBudgetNs) {
  if constexpr (CG == 1) {
    return mbar_wait(bar, parity, abort_flag, err_word, budget_ns);
  } else {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait_cluster(bar, parity)) return true;
      if ((it & 63u) == 0u) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > budget_ns) {
          *abort_flag = 1;
          if (err_word) atomicOr(err_word, 2 /* FLCE_DEVERR_TIMEOUT */);
          return false;
        }
      }
    }
  }
}

// Bounded wait that ignores the abort flag: used to let copies and MMAs in
// flight finish before the CTA releases its memory.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (globaltimer_ns() - t0 > 1000000000ull) break;
  }
}

// AND of `ok` over the kThreads epilogue threads (named barrier 1).
template <int kThreads>
__device__ __forceinline__ bool epi_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(ok)), "n"(kThreads)
      : "memory");
  return r != 0;
}

// Epi must provide:
//   static constexpr uint32_t kABFormat;  // operand type: 1 bf16, 0 fp16
//   struct Params;
//   static __device__ void tile(const Params&, int m_block, int n_tile,
//                               uint32_t taddr, bool acc_zero, int row_in_tile,
//                               int quarter, int part, int lane, GemmCtl* ctl);
// and may declare static constexpr int kEpiWarps = 8 (see EpiWarps).
// m_block indexes 128-row blocks of M (this CTA's rows are
// m_block*128 + [0, 128)). `taddr` addresses this warp's 32 TMEM lanes at
// column 0 of the tile's accumulator (read it with load_acc(..., acc_zero));
// `part` is this warp's column half with 8 epilogue warps, else 0; the
// epilogue threads may use named barrier 1.
template <int CG, bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(gemm_threads<Epi>(), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const GemmGeom g, const typename Epi::Params ep) {
  using Cfg = TileCfg<CG>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  GemmCtl* ctl = reinterpret_cast<GemmCtl*>(smem_raw + (base - raw) + Cfg::kStages * Cfg::kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int m_tiles = g.m_tiles;
  int k_iters = g.k_iters;
  if (g.dyn_rows != nullptr) {
    const int r = *g.dyn_rows;
    if (g.dyn_axis == 0) {
      const int t = (r + Cfg::kTileRows - 1) / Cfg::kTileRows;
      m_tiles = t < m_tiles ? t : m_tiles;
    } else {
      const int t = (r + kBK - 1) / kBK;
      k_iters = t < k_iters ? t : k_iters;
    }
  }
  const int total = m_tiles * g.n_tiles;
  volatile int* abort_flag = &ctl->abort;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit0 = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = CG == 2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  auto stage_a = [&](int s) { return base + s * Cfg::kStageBytes; };
  auto stage_b = [&](int s) { return base + s * Cfg::kStageBytes + Cfg::kABytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&ctl->acc_full[b]), 1);
      mbar_init(smem_addr(&ctl->acc_empty[b]), EpiWarps<Epi>::value * CG);
    }
    mbar_init(smem_addr(&ctl->mma_done), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) {
    if constexpr (CG == 1) {
      tmem_alloc(smem_addr(&ctl->tmem_base), kTmemCols);
      tmem_relinquish();
    } else {
      tmem_alloc_pair(smem_addr(&ctl->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    }
  }
  tc_fence_before_sync();
  if constexpr (CG == 1) {
    __syncthreads();
  } else {
    cluster_sync();  // the peer's barriers are initialised before any remote use
  }
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;       // bit s: stage s has been loaded at least once
      uint32_t last_phase = 0;  // bit s: phase of the last load into stage s
      bool ok = true;
      for (int u = unit0; u < total && ok; u += units) {
        int m, n;
        tile_coords(g, m_tiles, u, m, n);
        for (int k = 0; k < k_iters; ++k) {
          if (!wait_bar<CG>(smem_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag, g.err_word)) {
            ok = false;
            break;
          }
          const uint32_t full_local = smem_addr(&ctl->full[stage]);
          uint32_t full = full_local;
          if constexpr (CG == 2) full = map_to_rank(full_local, 0);
          if (leader) mbar_arrive_expect_tx(full_local, CG * Cfg::kStageBytes);
          load_operand<CG, A_MN, kBM>(stage_a(stage), &tm_a, full,
                                      g.a_mn0 + m * Cfg::kTileRows + static_cast<int>(rank) * kBM,
                                      g.a_k0 + k * kBK);
          load_operand<CG, B_MN, Cfg::kBNLoad>(
              stage_b(stage), &tm_b, full,
              g.b_mn0 + n * kBN + static_cast<int>(rank) * Cfg::kBNLoad, g.b_k0 + k * kBK);
          armed |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // let every copy already issued land before the CTAs exit
        for (int s = 0; s < Cfg::kStages; ++s) {
          if (armed & (1u << s)) drain_wait(smem_addr(&ctl->full[s]), (last_phase >> s) & 1u);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc =
          idesc_f16kind_f32(kBM * CG, kBN, A_MN ? 1 : 0, B_MN ? 1 : 0, Epi::kABFormat);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int u = unit0; u < total && ok; u += units, ++it) {
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
        if (!wait_bar<CG>(smem_addr(&ctl->acc_empty[buf]), use ^ 1u, abort_flag, g.err_word)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * kBN);
        for (int k = 0; k < k_iters; ++k) {
          if (!wait_bar<CG>(smem_addr(&ctl->full[stage]), phase, abort_flag, g.err_word)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = stage_a(stage), b0 = stage_b(stage);
#pragma unroll
          for (int kk = 0; kk < kBK / kUK; ++kk) {
            const uint32_t acc = (k | kk) != 0 ? 1u : 0u;
            if constexpr (CG == 1)
              umma_bf16(d_tmem, operand_desc<A_MN>(a0, kk), operand_desc<B_MN>(b0, kk), idesc, acc);
            else
              umma_bf16_pair(d_tmem, operand_desc<A_MN>(a0, kk), operand_desc<B_MN>(b0, kk), idesc,
                             acc);
          }
          if constexpr (CG == 1)
            umma_commit(smem_addr(&ctl->empty[stage]));
          else
            umma_commit_pair(smem_addr(&ctl->empty[stage]), 0x3);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (CG == 1)
          umma_commit(smem_addr(&ctl->acc_full[buf]));
        else
          umma_commit_pair(smem_addr(&ctl->acc_full[buf]), 0x3);
      }
      // all MMAs issued by this thread complete before TMEM is released
      if constexpr (CG == 1)
        umma_commit(smem_addr(&ctl->mma_done));
      else
        umma_commit_pair(smem_addr(&ctl->mma_done), 0x3);
      drain_wait(smem_addr(&ctl->mma_done), 0);
    } else if (lane == 0 && CG == 2) {
      // the odd CTA's TMEM is written by the even CTA's MMAs: wait for them
      drain_wait(smem_addr(&ctl->mma_done), 0);
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter+32)
    const int part = (warp - 2) >> 2;  // column half with 8 epilogue warps, else 0
    const int row_in_tile = quarter * 32 + lane;
    uint32_t acc_empty_leader = smem_addr(&ctl->acc_empty[0]);
    if constexpr (CG == 2) acc_empty_leader = map_to_rank(acc_empty_leader, 0);
    int it = 0;
    for (int u = unit0; u < total; u += units, ++it) {
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
      const bool got = wait_bar<CG>(smem_addr(&ctl->acc_full[buf]), use, abort_flag, g.err_word);
      if (!epi_all<32 * EpiWarps<Epi>::value>(got)) break;
      tc_fence_after_sync();
      int m, n;
      tile_coords(g, m_tiles, u, m, n);
      const uint32_t taddr =
          tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * kBN);
      Epi::tile(ep, m * CG + static_cast<int>(rank), n, taddr, k_iters == 0, row_in_tile,
                quarter, part, lane, ctl);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        const uint32_t bar = acc_empty_leader + static_cast<uint32_t>(buf * sizeof(uint64_t));
        if constexpr (CG == 1)
          mbar_arrive(bar);
        else
          mbar_arrive_cluster(bar);
      }
    }
  }

  tc_fence_before_sync();
  __syncwarp();
  if constexpr (CG == 1) {
    __syncthreads();
  } else {
    cluster_sync();
  }
  if (warp == 1) {
    __syncwarp();  // the release is warp-collective
    tc_fence_after_sync();
    if constexpr (CG == 1)
      tmem_dealloc(tmem, kTmemCols);
    else
      tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace flce
