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
// A 4-warp epilogue may ask for a relay (256 threads): a TMEM lane quarter can
// only be read by warps of its own scheduler (warp id mod 4), and schedulers 0
// and 1 also run the TMA and MMA threads, whose issue the epilogue's
// arithmetic delays. So warps 4 and 5 (schedulers 0, 1) only copy quarters 0
// and 1 from TMEM into shared memory, 32 columns at a time, and warps 6 and 7
// (schedulers 2, 3) run the epilogue on those rows; warps 2 and 3 run it on
// quarters 2 and 3 as before.
// The 512 TMEM columns hold two 128 x 256 fp32 accumulators per CTA, so the
// epilogue of tile i overlaps the MMAs of tile i+1.
//
// A launch runs the tiles of one GEMM or of two GEMMs that share nothing but
// the SMs ("segments": each with its own operands, majorness, extents and
// epilogue). Tiles are taken either statically (unit u of U takes tiles u,
// u + U, ...) or dynamically: the even CTA's producer thread draws the next
// tile index from a global counter and hands it to every role of both CTAs
// through a small ring in shared memory, so that a pair that finishes early
// takes more tiles. Dynamic scheduling balances tiles of unequal length (the
// two segments' contractions differ) and fills the last round.
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

constexpr int kSchedSlots = 8;  // tile indices in flight between the roles (dynamic scheduling)

struct GemmCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint64_t sched_full[kSchedSlots];   // slot holds a tile index (count 1: the fetching thread)
  uint64_t sched_empty[kSchedSlots];  // every reading role has taken it (even CTA's barriers)
  int sched_tile[kSchedSlots];        // tile index, or -1: no tiles left
  uint8_t* out_stage;  // the epilogue's staging area for tensor stores (Epi::kOutStageBytes)
  uint32_t tmem_base;
  int abort;
  float red[4][kBN / 32][32];  // epilogue scratch: per-warp column sums, [quarter][chunk][lane]
};

// Shared memory an epilogue stages its tensor stores in: Epi::kOutStageBytes
// where it declares them (a multiple of 1024), else none. The area follows
// the stage ring, 1024-byte aligned.
template <class Epi, class = void>
struct OutStage {
  static constexpr int bytes = 0;
};
template <class Epi>
struct OutStage<Epi, std::void_t<decltype(Epi::kOutStageBytes)>> {
  static constexpr int bytes = Epi::kOutStageBytes;
};

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
  // Dynamic scheduling (read from the first segment's geometry): a device
  // counter, zero before the launch, from which tile indices are drawn; null
  // for static scheduling.
  int* sched;
  // Programmatic dependent launch (first segment's geometry; the launch
  // carries the attribute when non-zero). Every CTA lets the next kernel
  // start at once; kPdlWaitLoads: the producer waits for the previous
  // kernels before its first load; kPdlWaitEpilogue: the epilogue threads
  // wait before their first tile.
  int pdl;
  // Split operands (segments with Seg::kSplit: fp32 inputs as three bf16
  // parts, x = hi + mid + lo): every tile runs its contraction `passes`
  // times over the same K range, pass p reading part pass_a[p] of A and part
  // pass_b[p] of B (0: the segment's own map; 1, 2: its two extra maps), all
  // into the same accumulator.
  int passes;
  uint8_t pass_a[6], pass_b[6];
};
constexpr int kPdlWaitLoads = 1;
constexpr int kPdlWaitEpilogue = 2;

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
// Whether Epi asks for the relay (Epi::kRelay; 4 epilogue warps only).
template <class Epi, class = void>
struct EpiRelay {
  static constexpr bool value = false;
};
template <class Epi>
struct EpiRelay<Epi, std::void_t<decltype(Epi::kRelay)>> {
  static constexpr bool value = Epi::kRelay;
};
// Warps that run epilogue code: the epilogue's own, plus the two relay
// readers.
template <class Epi>
__host__ __device__ constexpr int epi_phys_warps() {
  return EpiWarps<Epi>::value + (EpiRelay<Epi>::value ? 2 : 0);
}
// Threads per CTA: the TMA warp, the MMA warp and the epilogue warps.
template <class Epi>
constexpr int gemm_threads() {
  return 64 + 32 * epi_phys_warps<Epi>();
}

// ---- the relay (see the top of this file)
// Per relayed quarter, two slots of 32 rows x 32 fp32 columns. Row r (the
// lane) holds its 8 16-byte groups at r*128 + 16*(g ^ (r & 7)), so that the
// 16-byte accesses of any 8 consecutive lanes fall in distinct banks.
constexpr int kRelaySlotBytes = 32 * 32 * 4;
constexpr int kRelayBytes = 2 /* quarters */ * 2 /* slots */ * kRelaySlotBytes;
// Named barriers of the hand-off, per relayed quarter q: slot s full
// kRelayBar + 4q + s, slot s empty kRelayBar + 4q + 2 + s (64 threads: the
// reader warp and the computing warp). Barrier 1 is the epilogue-wide one.
constexpr uint32_t kRelayBar = 2;

__device__ __forceinline__ void relay_put(uint8_t* slot, int lane, const float (&v)[32]) {
  float4* row = reinterpret_cast<float4*>(slot + lane * 128);
#pragma unroll
  for (int g = 0; g < 8; ++g)
    row[g ^ (lane & 7)] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
}
__device__ __forceinline__ void relay_get(const uint8_t* slot, int lane, float (&v)[32]) {
  const float4* row = reinterpret_cast<const float4*>(slot + lane * 128);
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const float4 x = row[g ^ (lane & 7)];
    v[4 * g] = x.x;
    v[4 * g + 1] = x.y;
    v[4 * g + 2] = x.z;
    v[4 * g + 3] = x.w;
  }
}

// Where an epilogue warp's accumulator columns come from: its own TMEM lanes,
// or, for the warps that compute on relayed quarters, the two shared-memory
// slots that the quarter's reader fills. Relayed chunks arrive in column
// order; load() may skip chunks but not go back.
struct AccSrc {
  uint32_t taddr;  // this warp's TMEM lanes, column 0 of the tile's accumulator
  bool zero;       // the contraction was empty: every column reads 0
  uint8_t* relay;  // null: read TMEM; else the quarter's two relay slots
  uint32_t bar;    // the quarter's first relay barrier
  int taken;       // relayed chunks taken (or skipped) in this tile

  // 32 columns from column 32 * ch.
  __device__ __forceinline__ void load(int ch, float (&v)[32]) {
    if (zero) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      return;
    }
    if (relay == nullptr) {
      tmem_load_32cols(taddr + static_cast<uint32_t>(ch * 32), v);
      return;
    }
    skip_to(ch);
    const int slot = taken & 1;
    named_bar_sync(bar + slot, 64);
    relay_get(relay + slot * kRelaySlotBytes, threadIdx.x & 31, v);
    named_bar_arrive(bar + 2 + slot, 64);
    ++taken;
  }
  // Release the relayed chunks before ch without reading them.
  __device__ __forceinline__ void skip_to(int ch) {
    if (zero || relay == nullptr) return;
    while (taken < ch) {
      const int slot = taken & 1;
      named_bar_sync(bar + slot, 64);
      named_bar_arrive(bar + 2 + slot, 64);
      ++taken;
    }
  }
};

template <int CG, class E0, class E1>
constexpr int gemm_smem_bytes() {
  constexpr int out = OutStage<E0>::bytes > OutStage<E1>::bytes ? OutStage<E0>::bytes
                                                                 : OutStage<E1>::bytes;
  constexpr int relay = EpiRelay<E0>::value ? kRelayBytes : 0;
  return TileCfg<CG>::kStages * TileCfg<CG>::kStageBytes + 1024 /* alignment slack */ + out +
         relay + ((static_cast<int>(sizeof(GemmCtl)) + 127) / 128) * 128;
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

// Named barrier of the warps that run the epilogue policy (after the relay's).
constexpr uint32_t kEpiBar = kRelayBar + 8;

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

// Tile and contraction extents of one segment, with the device-side row
// count applied.
template <int CG>
__device__ __forceinline__ void seg_extent(const GemmGeom& g, int& m_tiles, int& k_iters) {
  using Cfg = TileCfg<CG>;
  m_tiles = g.m_tiles;
  k_iters = g.k_iters;
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
}

// Stores `v` into the shared variable at shared::cluster address `addr`
// (possibly in the peer CTA).
__device__ __forceinline__ void st_shared_cluster(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Epi must provide:
//   static constexpr uint32_t kABFormat;  // operand type: 1 bf16, 0 fp16
//   struct Params;
//   static __device__ void tile(const Params&, int m_block, int n_tile,
//                               AccSrc& acc, int row_in_tile, int quarter,
//                               int part, int lane, GemmCtl* ctl);
// and may declare static constexpr int kEpiWarps = 8 (see EpiWarps) or, with
// 4 warps, static constexpr bool kRelay = true (see EpiRelay).
// m_block indexes 128-row blocks of M (this CTA's rows are
// m_block*128 + [0, 128)). `acc` gives this warp's 32 accumulator rows, 32
// columns at a time, in increasing column order (acc.load(chunk, v));
// `part` is this warp's column half with 8 epilogue warps, else 0. The
// warps that run tile() may use named barrier kEpiBar (32 * kEpiWarps
// threads).

// One GEMM of a launch: operand majorness, epilogue, and whether its
// operands are split into parts (GemmGeom::passes).
template <bool A_MN_, bool B_MN_, class Epi_, bool SPLIT_ = false>
struct Seg {
  static constexpr bool kPresent = true;
  static constexpr bool A_MN = A_MN_;
  static constexpr bool B_MN = B_MN_;
  static constexpr bool kSplit = SPLIT_;
  using Epi = Epi_;
};

// The absent second segment of a one-GEMM launch.
struct NoEpi {
  static constexpr uint32_t kABFormat = 1;
  struct Params {};
  __device__ static void tile(const Params&, int, int, AccSrc&, int, int, int, int, GemmCtl*) {}
};
struct NoSeg {
  static constexpr bool kPresent = false;
  static constexpr bool A_MN = false;
  static constexpr bool B_MN = false;
  static constexpr bool kSplit = false;
  using Epi = NoEpi;
};

// The extra parts (mid, lo) of a split segment's operands; nothing otherwise.
template <bool SPLIT>
struct SplitMaps {};
template <>
struct SplitMaps<true> {
  CUtensorMap a[2], b[2];
};

// Kernel arguments: tensor maps, geometry and epilogue parameters of both
// segments (the second ones unused for a one-GEMM launch). Tile indices
// [0, tiles of segment 0) are segment 0's, the rest segment 1's.
__device__ __forceinline__ const CUtensorMap* split_a(const SplitMaps<true>& x) { return x.a; }
__device__ __forceinline__ const CUtensorMap* split_b(const SplitMaps<true>& x) { return x.b; }
__device__ __forceinline__ const CUtensorMap* split_a(const SplitMaps<false>&) { return nullptr; }
__device__ __forceinline__ const CUtensorMap* split_b(const SplitMaps<false>&) { return nullptr; }

template <class S0, class S1>
struct GemmArgs {
  CUtensorMap a0, b0, a1, b1;
  GemmGeom g0, g1;
  typename S0::Epi::Params ep0;
  typename S1::Epi::Params ep1;
  SplitMaps<S0::kSplit> x0;
  SplitMaps<S1::kSplit> x1;
};

template <int CG, class S0, class S1>
__global__ void __launch_bounds__(gemm_threads<typename S0::Epi>(), 1)
    tc_gemm_kernel(const __grid_constant__ GemmArgs<S0, S1> args) {
  using Cfg = TileCfg<CG>;
  using E0 = typename S0::Epi;
  using E1 = typename S1::Epi;
  constexpr int W = EpiWarps<E0>::value;   // warps that run the epilogue policy
  constexpr bool kRelay = EpiRelay<E0>::value;
  constexpr int WP = epi_phys_warps<E0>();  // warps in the epilogue branch
  static_assert(!S1::kPresent || EpiWarps<E1>::value == W, "segments differ in epilogue warps");
  static_assert(!S1::kPresent || EpiRelay<E1>::value == kRelay, "segments differ in relay");
  static_assert(!kRelay || W == 4, "the relay serves a 4-warp epilogue");
  static_assert(!S1::kPresent || E1::kABFormat == E0::kABFormat, "segments differ in type");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  constexpr int kOut = OutStage<E0>::bytes > OutStage<E1>::bytes ? OutStage<E0>::bytes
                                                                 : OutStage<E1>::bytes;
  uint8_t* const out_stage = smem_raw + (base - raw) + Cfg::kStages * Cfg::kStageBytes;
  uint8_t* const relay_slots = out_stage + kOut;
  GemmCtl* ctl = reinterpret_cast<GemmCtl*>(relay_slots + (kRelay ? kRelayBytes : 0));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int m_tiles0, k_iters0, m_tiles1 = 0, k_iters1 = 0;
  seg_extent<CG>(args.g0, m_tiles0, k_iters0);
  if constexpr (S1::kPresent) seg_extent<CG>(args.g1, m_tiles1, k_iters1);
  const int total0 = m_tiles0 * args.g0.n_tiles;
  const int total = total0 + (S1::kPresent ? m_tiles1 * args.g1.n_tiles : 0);
  int* const err_word = args.g0.err_word;
  int* const sched = args.g0.sched;
  const bool dynamic = sched != nullptr;
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
      // the warps that read TMEM: W per CTA (with the relay, its two readers
      // stand in for the two warps they serve)
      mbar_init(smem_addr(&ctl->acc_empty[b]), W * CG);
    }
    // readers of a schedule slot: the MMA thread and the epilogue warps of
    // the even CTA, the producer and the epilogue warps of the odd one
    for (int s = 0; s < kSchedSlots; ++s) {
      mbar_init(smem_addr(&ctl->sched_full[s]), 1);
      mbar_init(smem_addr(&ctl->sched_empty[s]), CG * (1 + WP));
    }
    mbar_init(smem_addr(&ctl->mma_done), 1);
    ctl->out_stage = out_stage;
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&args.a0);
    tma_prefetch_desc(&args.b0);
    if constexpr (S1::kPresent) {
      tma_prefetch_desc(&args.a1);
      tma_prefetch_desc(&args.b1);
    }
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
  const int pdl = args.g0.pdl;
  if (pdl != 0 && threadIdx.x == 0) grid_launch_dependents();

  // ---- the tile sequence
  // Static: iteration it takes tile unit0 + it * units. Dynamic: the even
  // CTA's producer draws tickets from `sched` and publishes each (or -1 once
  // they run out) in slot it % kSchedSlots of both CTAs; every other role
  // reads the slot and releases it on the even CTA's sched_empty barrier.
  auto slot_of = [](int it) { return it % kSchedSlots; };
  auto phase_of = [](int it) { return static_cast<uint32_t>(it / kSchedSlots) & 1u; };
  // the even CTA's readers release a slot with a CTA-scope arrive, the odd
  // CTA's with a cluster-scope one on the even CTA's barrier
  auto sched_ack = [&](int slot) {
    const uint32_t bar = smem_addr(&ctl->sched_empty[slot]);
    if (CG == 2 && !leader)
      mbar_arrive_cluster(map_to_rank(bar, 0));
    else
      mbar_arrive(bar);
  };
  // Reader side of iteration it: the tile index (-1: none left); false when
  // the wait gave up.
  auto sched_read = [&](int it, int& u) -> bool {
    const int slot = slot_of(it);
    if (!wait_bar<CG>(smem_addr(&ctl->sched_full[slot]), phase_of(it), abort_flag, err_word))
      return false;
    u = *reinterpret_cast<volatile int*>(&ctl->sched_tile[slot]);
    sched_ack(slot);
    return true;
  };
  // Fetcher side: publish u in slot it % kSchedSlots of both CTAs.
  auto sched_publish = [&](int it, int u) {
    const int slot = slot_of(it);
    const uint32_t tile_addr = smem_addr(&ctl->sched_tile[slot]);
    const uint32_t bar = smem_addr(&ctl->sched_full[slot]);
    *reinterpret_cast<volatile int*>(&ctl->sched_tile[slot]) = u;
    mbar_arrive(bar);  // release (CTA scope): the store comes first
    if constexpr (CG == 2) {
      st_shared_cluster(map_to_rank(tile_addr, 1), u);
      mbar_arrive_cluster(map_to_rank(bar, 1));  // release (cluster scope) to the odd CTA
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;       // bit s: stage s has been loaded at least once
      uint32_t last_phase = 0;  // bit s: phase of the last load into stage s
      bool ok = true;
      // loads of one tile of segment S (tile index ul within the segment)
      // xa, xb: the extra parts of a split segment's operands (else unused);
      // a split segment's tile runs g.passes passes of k_iters stages each
      auto produce = [&](auto seg, const CUtensorMap* ta, const CUtensorMap* tb,
                         const CUtensorMap* xa, const CUtensorMap* xb, const GemmGeom& g,
                         int m_tiles, int k_iters, int ul) -> bool {
        using S = decltype(seg);
        int m, n;
        tile_coords(g, m_tiles, ul, m, n);
        const int k_total = S::kSplit ? g.passes * k_iters : k_iters;
        for (int kt = 0; kt < k_total; ++kt) {
          int k = kt;
          const CUtensorMap* ma = ta;
          const CUtensorMap* mb = tb;
          if constexpr (S::kSplit) {
            const int pass = kt / k_iters;
            k = kt - pass * k_iters;
            if (g.pass_a[pass] != 0) ma = xa + (g.pass_a[pass] - 1);
            if (g.pass_b[pass] != 0) mb = xb + (g.pass_b[pass] - 1);
          }
          if (!wait_bar<CG>(smem_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag, err_word))
            return false;
          const uint32_t full_local = smem_addr(&ctl->full[stage]);
          uint32_t full = full_local;
          if constexpr (CG == 2) full = map_to_rank(full_local, 0);
          if (leader) mbar_arrive_expect_tx(full_local, CG * Cfg::kStageBytes);
          load_operand<CG, S::A_MN, kBM>(stage_a(stage), ma, full,
                                         g.a_mn0 + m * Cfg::kTileRows + static_cast<int>(rank) * kBM,
                                         g.a_k0 + k * kBK);
          load_operand<CG, S::B_MN, Cfg::kBNLoad>(
              stage_b(stage), mb, full,
              g.b_mn0 + n * kBN + static_cast<int>(rank) * Cfg::kBNLoad, g.b_k0 + k * kBK);
          armed |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      };
      if (pdl & kPdlWaitLoads) grid_dependency_wait();
      // Dynamic: the even CTA's producer publishes each tile index one tile
      // ahead of its own loads, so that the odd CTA's producer knows it a
      // whole tile before its copies are due; it keeps one ticket drawn
      // ahead, drawn after the previous publication so that the release
      // does not wait for the atomic.
      int ticket = 0, cur = -1;
      auto publish_next = [&](int it) -> bool {
        if (!wait_bar<CG>(smem_addr(&ctl->sched_empty[slot_of(it)]), phase_of(it) ^ 1u,
                          abort_flag, err_word))
          return false;
        const int u = ticket < total ? ticket : -1;
        sched_publish(it, u);
        if (u >= 0) ticket = atomicAdd(sched, 1);
        return true;
      };
      if (dynamic && leader) {
        ticket = atomicAdd(sched, 1);
        ok = publish_next(0);
        cur = *reinterpret_cast<volatile int*>(&ctl->sched_tile[0]);
      }
      for (int it = 0; ok; ++it) {
        int u;
        if (!dynamic) {
          u = unit0 + it * units;
          if (u >= total) break;
        } else if (leader) {
          u = cur;
          if (u < 0) break;
          if (!publish_next(it + 1)) {
            ok = false;
            break;
          }
          cur = *reinterpret_cast<volatile int*>(&ctl->sched_tile[slot_of(it + 1)]);
        } else {
          if (!sched_read(it, u)) {
            ok = false;
            break;
          }
          if (u < 0) break;
        }
        if (!S1::kPresent || u < total0)
          ok = produce(S0{}, &args.a0, &args.b0, split_a(args.x0), split_b(args.x0), args.g0,
                       m_tiles0, k_iters0, u);
        else
          ok = produce(S1{}, &args.a1, &args.b1, split_a(args.x1), split_b(args.x1), args.g1,
                       m_tiles1, k_iters1, u - total0);
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
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // the MMAs of one tile of segment S into accumulator d_tmem
      auto mma = [&](auto seg, int k_iters, uint32_t d_tmem) -> bool {
        using S = decltype(seg);
        constexpr uint32_t idesc =
            idesc_f16kind_f32(kBM * CG, kBN, S::A_MN ? 1 : 0, S::B_MN ? 1 : 0, E0::kABFormat);
        for (int k = 0; k < k_iters; ++k) {
          if (!wait_bar<CG>(smem_addr(&ctl->full[stage]), phase, abort_flag, err_word))
            return false;
          tc_fence_after_sync();
          const uint32_t a0 = stage_a(stage), b0 = stage_b(stage);
#pragma unroll
          for (int kk = 0; kk < kBK / kUK; ++kk) {
            const uint32_t acc = (k | kk) != 0 ? 1u : 0u;
            if constexpr (CG == 1)
              umma_bf16(d_tmem, operand_desc<S::A_MN>(a0, kk), operand_desc<S::B_MN>(b0, kk),
                        idesc, acc);
            else
              umma_bf16_pair(d_tmem, operand_desc<S::A_MN>(a0, kk),
                             operand_desc<S::B_MN>(b0, kk), idesc, acc);
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
        return true;
      };
      for (int it = 0; ok; ++it) {
        int u;
        if (!dynamic) {
          u = unit0 + it * units;
          if (u >= total) break;
        } else {
          if (!sched_read(it, u)) {
            ok = false;
            break;
          }
          if (u < 0) break;
        }
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
        if (!wait_bar<CG>(smem_addr(&ctl->acc_empty[buf]), use ^ 1u, abort_flag, err_word)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * kBN);
        if (!S1::kPresent || u < total0)
          ok = mma(S0{}, S0::kSplit ? args.g0.passes * k_iters0 : k_iters0, d_tmem);
        else
          ok = mma(S1{}, S1::kSplit ? args.g1.passes * k_iters1 : k_iters1, d_tmem);
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
    // Roles: without the relay, warp w runs the policy on TMEM lane quarter
    // w % 4 (column half (w - 2) / 4). With it (warps 2-7): warps 2, 3 run the
    // policy on quarters 2, 3; warps 4, 5 read quarters 0, 1 into the relay
    // slots; warps 6, 7 run the policy on quarters 0, 1 from those slots.
    const bool reader = kRelay && (warp == 4 || warp == 5);
    const bool relayed = kRelay && warp >= 6;
    const int quarter = relayed ? (warp & 3) - 2 : (warp & 3);  // TMEM lanes [32q, 32q+32)
    const int part = kRelay ? 0 : (warp - 2) >> 2;  // column half with 8 epilogue warps, else 0
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t relay_bar = kRelayBar + 4u * static_cast<uint32_t>(quarter);
    uint8_t* const relay = relay_slots + quarter * 2 * kRelaySlotBytes;
    uint32_t relay_used = 0;  // reader: bit s set once slot s has been filled
    uint32_t acc_empty_leader = smem_addr(&ctl->acc_empty[0]);
    if constexpr (CG == 2) acc_empty_leader = map_to_rank(acc_empty_leader, 0);
    if (pdl & kPdlWaitEpilogue) grid_dependency_wait();
    for (int it = 0;; ++it) {
      int u;
      if (!dynamic) {
        u = unit0 + it * units;
        if (u >= total) break;
      } else {
        // one lane per warp reads the slot; the warps decide together
        int uu = -1;
        bool got_s = true;
        if (lane == 0) got_s = sched_read(it, uu);
        got_s = __shfl_sync(0xffffffffu, got_s ? 1 : 0, 0) != 0;
        uu = __shfl_sync(0xffffffffu, uu, 0);
        if (!epi_all<32 * WP>(got_s)) break;
        u = uu;
        if (u < 0) break;
      }
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
      // the relayed warps take their columns from the slots, not from TMEM
      const bool got =
          relayed || wait_bar<CG>(smem_addr(&ctl->acc_full[buf]), use, abort_flag, err_word);
      if (!epi_all<32 * WP>(got)) break;
      tc_fence_after_sync();
      const uint32_t taddr =
          tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * kBN);
      const bool seg0 = !S1::kPresent || u < total0;
      const bool acc_zero = seg0 ? k_iters0 == 0 : k_iters1 == 0;
      if (reader) {
        // all 8 chunks of the quarter, in column order; the computing warp
        // takes or skips each one
        if (!acc_zero) {
#pragma unroll 1
          for (int ch = 0; ch < kBN / 32; ++ch) {
            float v[32];
            tmem_load_32cols(taddr + static_cast<uint32_t>(ch * 32), v);
            const int slot = ch & 1;
            if (relay_used & (1u << slot)) named_bar_sync(relay_bar + 2 + slot, 64);
            relay_used |= 1u << slot;
            relay_put(relay + slot * kRelaySlotBytes, lane, v);
            named_bar_arrive(relay_bar + slot, 64);
          }
        }
      } else {
        AccSrc acc{taddr, acc_zero, relayed ? relay : nullptr, relay_bar, 0};
        int m, n;
        if (seg0) {
          tile_coords(args.g0, m_tiles0, u, m, n);
          E0::tile(args.ep0, m * CG + static_cast<int>(rank), n, acc, row_in_tile, quarter, part,
                   lane, ctl);
        } else {
          tile_coords(args.g1, m_tiles1, u - total0, m, n);
          E1::tile(args.ep1, m * CG + static_cast<int>(rank), n, acc, row_in_tile, quarter, part,
                   lane, ctl);
        }
        acc.skip_to(kBN / 32);  // chunks the policy did not take
      }
      if (!relayed) {
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
    // a reader waits until its last slots have been taken: every arrival on
    // the relay barriers is then matched
#pragma unroll
    for (int slot = 0; slot < 2; ++slot)
      if (relay_used & (1u << slot)) named_bar_sync(relay_bar + 2 + slot, 64);
    // an epilogue that stages tensor stores issues them from lane 0 of each
    // warp: they complete before the CTA leaves
    if constexpr (kOut > 0) {
      if (lane == 0) tma_store_wait_all();
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
