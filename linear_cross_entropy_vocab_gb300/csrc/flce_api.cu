// C ABI of libflce.so (declared in include/flce.h): argument checks,
// workspace planning, tensor-map encoding and the launch sequences of the
// forward and backward passes of the fused linear cross-entropy and of the
// fused linear KL divergence (which shares the backward sequence), plus the
// fixed-scratch forward, the bounded-wait self-test and the launch profiler.
// No device memory is allocated here and no call synchronises the caller's
// stream.
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "flce.h"
#include "flce_internal.h"

namespace {

using flce::GemmGeom;

thread_local char g_err[512] = {0};

flce_status fail(flce_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

flce_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FLCE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ----------------------------------------------------------- device facts
struct DeviceInfo {
  int known = 0;
  int sms = 0;
  int major = 0, minor = 0;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

// Also makes the current device's primary context current on the calling
// thread (a thread that never made a runtime call, such as an autograd worker,
// may have none, and the tensor-map encoder needs one).
bool device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (cudaSetDevice(dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.known) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return false;
    d.known = 1;
  }
  *out = d;
  return true;
}

// ---------------------------------------------------- tensor-map encoding
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeFn g_encode = nullptr;

EncodeFn encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeFn>(fn);
  });
  return g_encode;
}

thread_local CUtensorMapDataType g_map_type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

// 2-D tensor of 16-bit elements (of type g_map_type: the input type of the
// current call) [outer][inner] with row pitch `pitch_elems`, box
// {box_inner, box_outer}, 128-byte swizzle (the GEMM operands) or none (the
// epilogues' stores), zero fill out of bounds.
// On failure records the driver's result in the thread's error text.
bool make_map(CUtensorMap* map, const char* what, const void* base, int64_t inner,
              int64_t outer, int64_t pitch_elems, uint32_t box_inner, uint32_t box_outer,
              bool swizzle = true) {
  EncodeFn enc = encoder();
  if (!enc) {
    fail(FLCE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_elems) * 2u};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(map, g_map_type, 2, const_cast<void*>(base), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fail(FLCE_ERR_CUDA,
         "cuTensorMapEncodeTiled(%s) failed with CUresult %d (base %p, dims %lld x %lld, "
         "pitch %lld, box %u x %u)",
         what, static_cast<int>(r), base, (long long)inner, (long long)outer,
         (long long)pitch_elems, box_inner, box_outer);
    return false;
  }
  return true;
}

// ------------------------------------------------------------ profiler
// Optional CUDA-event brackets around each launch (flce_profile_*).
struct ProfRecord {
  int role;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
bool g_prof_ready = false;
ProfRecord g_prof[FLCE_PROFILE_MAX_RECORDS];
int g_prof_n = 0;
int32_t g_prof_dropped = 0;
const char* g_role_names[16];
int g_n_roles = 0;

int role_id(const char* name) {
  for (int i = 0; i < g_n_roles; ++i)
    if (std::strcmp(g_role_names[i], name) == 0) return i;
  if (g_n_roles < 16) {
    g_role_names[g_n_roles] = name;
    return g_n_roles++;
  }
  return 15;
}

// Brackets one kernel launch with events on `s` while profiling is enabled.
class ProfScope {
 public:
  ProfScope(const char* role, cudaStream_t s) : s_(s) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return;
    if (g_prof_n >= FLCE_PROFILE_MAX_RECORDS) {
      ++g_prof_dropped;
      return;
    }
    rec_ = &g_prof[g_prof_n++];
    rec_->role = role_id(role);
    cudaEventRecord(rec_->start, s_);
  }
  ~ProfScope() {
    if (rec_ != nullptr) cudaEventRecord(rec_->stop, s_);
  }

 private:
  cudaStream_t s_;
  ProfRecord* rec_ = nullptr;
};

// ------------------------------------------------------------- planning
constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Default backward vocabulary chunking: the dlogits buffer D of one chunk is
// at most 512 MiB and spans at most about a fifth of the vocabulary (V/5
// rounded up to whole 256-column tiles; a vocabulary of fewer than five tiles
// gets one chunk per tile), so that together with grad_weight (V x H),
// grad_hidden and its fp32 accumulator the backward stays below the N x V
// logits of a plain implementation even where H is half of N (the
// 4096-token, 2048-wide, 32000-word head: peak 0.96 x N V 2 bytes).
constexpr int64_t kDefaultDlogitsBudget = int64_t(512) << 20;  // bytes of one dlogits chunk
constexpr int64_t kMinDefaultChunks = 5;

// Tile bands (GemmGeom::group) of the row-tile-fastest GEMMs. With bands of
// 16 pair row tiles (4096 rows) the forward and dlogits kernels re-read
// hidden far less (measured at the Llama-3 head shape: forward DRAM reads
// 6.5 -> 2.7-4.2 GB, dlogits 7.0 -> 3.1-3.4 GB per step); grad_hidden does
// best with 8 (19.7 -> 11.6-13.5 GB). grad_weight runs fastest along H, in
// bands of H tiles (kBandGradWeight below).
// Tile order of the forward GEMM and of the dlogits GEMMs: dynamic (drawn
// from a device counter, as the gradient launches always are) or static.
// Static order lets pairs drift apart in the tile sequence, which widens the
// window of weight tiles in flight; with dynamic order the forward read W
// exactly twice (2.17 GB per launch at the Llama-3 head shape, against
// 2.9-3.1 GB static on the same box), within 0.4 % of the static time. The
// dlogits launches gain less (0.59 -> 0.52 GB) and cost more at the
// 2048-wide head (+2 %), so they stay static.
constexpr bool kDynamicForward = true;
constexpr bool kDynamicDlogits = false;
constexpr int kBandForward = 16;
constexpr int kBandDlogits = 16;
constexpr int kBandGradHidden = 8;
// grad_weight tiles (vocabulary rows x H columns, contraction over the kept
// rows) run in bands of 8 H tiles: hidden's columns of a band stay in L2 while
// D is read once per band. At the Llama-3 head shape this cuts the fused
// gradient launch's DRAM reads from 3.9 to 3.3 GB. Single interleaved steps
// ran 1 % slower, but runs of back-to-back steps, which hold the GPU at its
// power cap, ran 1 % faster: there a step's speed follows its energy, and DRAM
// traffic is part of it.
constexpr int kBandGradWeight = 8;

// Workspace items of valid-row compaction (FLCE_SKIP_IGNORED_ROWS).
struct CompactPlan {
  bool on = false;
  size_t row_map = 0, n_kept = 0, hidden_c = 0, targets_c = 0, lse_c = 0, grad_c = 0,
         qsum_c = 0;
};

struct FwdPlan {
  int64_t n_vt = 0;
  size_t partials = 0, zsum = 0, zt = 0, correct = 0, entropy = 0, sched = 0, total = 0;
  bool has_zsum = false;
  CompactPlan cp;
  // fp32 inputs on the tensor cores: hidden's three bf16 parts, and the
  // parts of one vocabulary chunk of W at a time
  bool split = false;
  int64_t split_chunk = 0;
  size_t split_h = 0, split_w = 0;
};

struct BwdPlan {
  int64_t chunk = 0, n_chunks = 0, gb_parts = 0;
  size_t d = 0, acc = 0, gb = 0, scales = 0, sched = 0, sched_bytes = 0, total = 0;
  bool use_acc = false;
  CompactPlan cp;
  // fp32 inputs on the tensor cores (cross-entropy): D is held as three
  // bf16 parts; hidden's parts, and the parts of the chunk's W rows
  bool split = false;
  size_t split_h = 0, split_w = 0;
};

// bf16 and fp16 inputs run on the tensor cores; fp32 on FFMA kernels.
bool is_tc(const flce_problem* p) { return p->dtype == FLCE_BF16 || p->dtype == FLCE_F16; }

int tc_type(const flce_problem* p) { return p->dtype == FLCE_F16 ? flce::kTcF16 : flce::kTcBF16; }

// fp32 inputs whose rows are a multiple of 16 bytes run on the tensor cores
// with split operands: each value as three bf16 parts (hi + mid + lo, exact),
// each product as six part products (the three dropped ones, mid.lo, lo.mid
// and lo.lo, come to about 2^-23 of it), accumulated in fp32.
constexpr bool kSplitF32 = true;
int64_t split_chunk(const flce_problem* p, bool caller_chunk = true);
// Split operands also need their bf16 parts in the workspace: hidden's, one
// chunk's of W and of D, and the fp32 grad_hidden accumulator. They are used
// only while that stays under 40 % of one fp32 N x V logit matrix, so that a
// step's peak memory (with the fp32 gradients) stays under one; smaller
// problems (a short batch or a small vocabulary) run the FFMA kernels.
bool is_split(const flce_problem* p) {
  if (!kSplitF32 || p->dtype != FLCE_F32 || p->h % 8 != 0 || p->n <= 0) return false;
  const int64_t c = split_chunk(p, false);  // the default chunk: vocab_chunk does not decide
  const double parts = 6.0 * p->n * p->h + 6.0 * (p->n + p->h) * c + 4.0 * p->n * p->h;
  return parts <= 0.4 * 4.0 * p->n * p->v;
}
// Part pairs (A part, B part) of the six passes: hi.hi, hi.mid, mid.hi,
// hi.lo, lo.hi, mid.mid (0 hi, 1 mid, 2 lo).
constexpr uint8_t kSplitPassA[6] = {0, 0, 1, 0, 2, 1};
constexpr uint8_t kSplitPassB[6] = {0, 1, 0, 2, 0, 1};
// Default vocabulary chunk of the split path (forward and backward): a
// chunk's bf16 parts of D (N x c) and of W (c x H), 6 (N + H) c bytes, take at
// most 512 MiB and at most a fifth of one fp32 N x V logit matrix; a multiple
// of 256 columns, at least 256. (vocab_chunk, when set and caller_chunk, is
// taken as given.)
int64_t split_chunk(const flce_problem* p, bool caller_chunk) {
  const int64_t v_round = cdiv(p->v, 256) * 256;
  if (caller_chunk && p->vocab_chunk > 0) {
    const int64_t c = cdiv(p->vocab_chunk, 256) * 256;
    return c < v_round ? c : v_round;
  }
  const int64_t rows = p->n > 0 ? p->n : 1;
  int64_t budget = rows * v_round * 4 / 5;
  if (budget > (int64_t(512) << 20)) budget = int64_t(512) << 20;
  int64_t c = budget / (6 * (rows + p->h)) / 256 * 256;
  if (c < 256) c = 256;
  return c < v_round ? c : v_round;
}

bool skips_ignored(const flce_problem* p) {
  return is_tc(p) && (p->flags & FLCE_SKIP_IGNORED_ROWS) != 0;
}

// Appends the compaction items at `off`; returns the new end.
size_t plan_compaction(const flce_problem* p, bool backward, bool kl, size_t off,
                       CompactPlan* c) {
  c->on = skips_ignored(p);
  if (!c->on) return off;
  const size_t n = static_cast<size_t>(p->n);
  c->row_map = off;
  off = align_up(off + n * 4);
  c->n_kept = off;
  off = align_up(off + 4);
  c->hidden_c = off;
  off = align_up(off + n * static_cast<size_t>(p->h) * 2);
  c->targets_c = off;
  off = align_up(off + n * 8);
  if (backward) {
    c->lse_c = off;
    off = align_up(off + n * 4);
    c->grad_c = off;
    off = align_up(off + n * 4);
    if (kl) {
      c->qsum_c = off;
      off = align_up(off + n * 4);
    }
  }
  return off;
}

flce_status check_problem(const flce_problem* p) {
  if (p == nullptr) return fail(FLCE_ERR_INVALID_ARG, "problem pointer is NULL");
  if (p->n < 0 || p->h < 1 || p->v < 1)
    return fail(FLCE_ERR_INVALID_ARG, "need n >= 0, h >= 1, v >= 1 (got n=%lld h=%lld v=%lld)",
                (long long)p->n, (long long)p->h, (long long)p->v);
  const int64_t lim = int64_t(1) << 30;
  if (p->n >= lim || p->h >= lim || p->v >= lim)
    return fail(FLCE_ERR_UNSUPPORTED, "n, h and v must each be below 2^30");
  if (p->dtype != FLCE_F32 && p->dtype != FLCE_BF16 && p->dtype != FLCE_F16)
    return fail(FLCE_ERR_INVALID_ARG, "dtype must be FLCE_F32, FLCE_BF16 or FLCE_F16");
  if (p->has_bias != 0 && p->has_bias != 1)
    return fail(FLCE_ERR_INVALID_ARG, "has_bias must be 0 or 1");
  if (p->reduction < FLCE_RED_NONE || p->reduction > FLCE_RED_MEAN)
    return fail(FLCE_ERR_INVALID_ARG, "reduction must be none, sum or mean");
  if (p->grad_weight_dtype != FLCE_F32 && p->grad_weight_dtype != p->dtype)
    return fail(FLCE_ERR_INVALID_ARG, "grad_weight_dtype must be FLCE_F32 or the input dtype");
  if (!std::isfinite(p->logit_scale))
    return fail(FLCE_ERR_INVALID_ARG, "logit_scale must be finite");
  if (std::isnan(p->softcap) || std::isinf(p->softcap))
    return fail(FLCE_ERR_INVALID_ARG, "softcap must be finite (<= 0 disables it)");
  if (p->vocab_chunk < 0) return fail(FLCE_ERR_INVALID_ARG, "vocab_chunk must be >= 0");
  if ((p->flags & ~FLCE_SKIP_IGNORED_ROWS) != 0 || p->reserved != 0)
    return fail(FLCE_ERR_INVALID_ARG, "unknown flags or non-zero reserved field");
  if (!(p->label_smoothing >= 0.0f && p->label_smoothing <= 1.0f))
    return fail(FLCE_ERR_INVALID_ARG, "label_smoothing must be in [0, 1]");
  if (!std::isfinite(p->z_loss) || p->z_loss < 0.0f)
    return fail(FLCE_ERR_INVALID_ARG, "z_loss must be finite and >= 0");
  if (is_tc(p) && p->h % 8 != 0)
    return fail(FLCE_ERR_UNSUPPORTED,
                "bf16/fp16 inputs need h %% 8 == 0 (16-byte row pitch); h=%lld", (long long)p->h);
  if (is_tc(p)) {
    const int64_t m_tiles = cdiv(p->n, flce::kBM), n_tiles = cdiv(p->v, flce::kBM);
    if (m_tiles * n_tiles >= (int64_t(1) << 31))
      return fail(FLCE_ERR_UNSUPPORTED, "too many tiles");
  }
  return FLCE_OK;
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Per-row statistics entries of the forward: one per 256-column tile on the
// tensor cores (two, per 128-column half, when the forward runs 8 epilogue
// warps), one per kSimtTileV columns on the fp32 path.
int64_t forward_parts(const flce_problem* p, bool split = false) {
  if (!is_tc(p) && !split) return cdiv(p->v, flce::kSimtTileV);
  return cdiv(p->v, flce::kBN) * flce::fwd_parts_per_tile(p->h);
}

FwdPlan plan_forward(const flce_problem* p) {
  FwdPlan f;
  f.split = is_split(p);
  f.n_vt = forward_parts(p, f.split);
  size_t off = 0;
  f.partials = off;
  off = align_up(off + static_cast<size_t>(p->n) * f.n_vt * 16);
  f.has_zsum = p->label_smoothing != 0.0f;
  f.zsum = off;
  if (f.has_zsum) off = align_up(off + static_cast<size_t>(p->n) * f.n_vt * 4);
  f.zt = off;
  off = align_up(off + static_cast<size_t>(p->n) * 4);
  f.correct = off;
  off = align_up(off + static_cast<size_t>(p->n) * 4);
  f.entropy = off;
  off = align_up(off + static_cast<size_t>(p->n) * 4);
  f.sched = off;  // tile counter of the forward GEMM
  if (is_tc(p)) off = align_up(off + sizeof(int));
  off = plan_compaction(p, false, false, off, &f.cp);
  if (f.split) {
    f.split_chunk = split_chunk(p);
    f.split_h = off;
    off = align_up(off + 3 * static_cast<size_t>(p->n) * p->h * 2);
    f.split_w = off;
    off = align_up(off + 3 * static_cast<size_t>(f.split_chunk) * p->h * 2);
  }
  f.total = off;
  return f;
}

BwdPlan plan_backward(const flce_problem* p, bool kl = false) {
  BwdPlan b;
  b.split = is_split(p);
  const bool tc = is_tc(p) || b.split;  // tile shapes and accumulation of the tensor-core GEMMs
  const int64_t elem = is_tc(p) ? 2 : (b.split ? 6 : 4);  // bytes of one D entry
  const int64_t v_round = cdiv(p->v, 256) * 256;
  int64_t c = p->vocab_chunk;
  if (b.split) {
    c = split_chunk(p);
  } else if (c > 0) {
    c = cdiv(c, 256) * 256;
  } else {
    // balanced chunks: at least kMinDefaultChunks (at most one per tile),
    // more when one would exceed the budget
    const int64_t rows = p->n > 0 ? p->n : 1;
    int64_t nch = cdiv(rows * elem * v_round, kDefaultDlogitsBudget);
    const int64_t tiles = v_round / 256;
    const int64_t floor_chunks = tiles < kMinDefaultChunks ? tiles : kMinDefaultChunks;
    if (nch < floor_chunks) nch = floor_chunks;
    c = cdiv(cdiv(p->v, nch), 256) * 256;
    while (c > 256 && c * rows * elem > kDefaultDlogitsBudget) {
      ++nch;
      c = cdiv(cdiv(p->v, nch), 256) * 256;
    }
  }
  if (c > v_round) c = v_round;
  b.chunk = c;
  b.n_chunks = cdiv(p->v, c);
  b.use_acc = tc && b.n_chunks > 1;
  b.gb_parts = p->has_bias ? cdiv(p->n, tc ? flce::kBM : flce::kSimtTileN) : 0;
  size_t off = 0;
  b.d = off;
  off = align_up(off + static_cast<size_t>(p->n) * c * elem);
  b.acc = off;
  if (b.use_acc) off = align_up(off + static_cast<size_t>(p->n) * p->h * 4);
  b.gb = off;
  if (p->has_bias) off = align_up(off + static_cast<size_t>(b.gb_parts) * p->v * 4);
  b.scales = off;
  if (p->dtype == FLCE_F16) off = align_up(off + 2 * sizeof(float));
  // tile counters of the dynamically scheduled launches, two per chunk
  // (dlogits, gradients), zeroed at the start of every backward call
  b.sched = off;
  if (tc) {
    b.sched_bytes = align_up(static_cast<size_t>(2 * b.n_chunks) * sizeof(int));
    off += b.sched_bytes;
  }
  off = plan_compaction(p, true, kl, off, &b.cp);
  if (b.split) {
    b.split_h = off;
    off = align_up(off + 3 * static_cast<size_t>(p->n) * p->h * 2);
    b.split_w = off;
    off = align_up(off + 3 * static_cast<size_t>(c) * p->h * 2);
  }
  b.total = off;
  return b;
}

flce::LogitXform make_xform(const flce_problem* p) {
  flce::LogitXform xf;
  xf.scale = p->logit_scale;
  xf.has_cap = p->softcap > 0.0f ? 1 : 0;
  xf.softcap = xf.has_cap ? p->softcap : 1.0f;
  xf.inv_softcap = 1.0f / xf.softcap;
  return xf;
}

flce_status check_device(DeviceInfo* dev) {
  if (!device_info(dev)) return fail(FLCE_ERR_CUDA, "cannot query the current CUDA device");
  if (!(dev->major == 10 && dev->minor == 3))
    return fail(FLCE_ERR_UNSUPPORTED,
                "libflce.so is built for sm_103a (GB300); current device is sm_%d%d", dev->major,
                dev->minor);
  return FLCE_OK;
}

flce_status check_workspace(void* ws, size_t have, size_t need) {
  if (have < need)
    return fail(FLCE_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", have,
                need);
  if (need > 0 && (ws == nullptr || !aligned(ws, kAlign)))
    return fail(FLCE_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
  return FLCE_OK;
}

// Problem and pointer checks of the cross-entropy forward (flce_forward and
// flce_forward_noalloc): argument errors are reported before anything else.
flce_status check_forward_args(const flce_problem* p, const void* hidden, const void* weight,
                               const void* bias, const int64_t* targets, const float* loss_rows,
                               const float* lse_rows, const float* loss_out,
                               const int32_t* n_valid) {
  flce_status st = check_problem(p);
  if (st != FLCE_OK) return st;
  const size_t in_align = is_tc(p) ? 16 : 4;
  if (weight == nullptr) return fail(FLCE_ERR_INVALID_ARG, "weight is NULL");
  if (n_valid == nullptr) return fail(FLCE_ERR_INVALID_ARG, "n_valid is NULL");
  if (p->reduction != FLCE_RED_NONE && loss_out == nullptr)
    return fail(FLCE_ERR_INVALID_ARG, "loss_out is NULL (required for sum and mean)");
  if (p->has_bias && bias == nullptr) return fail(FLCE_ERR_INVALID_ARG, "has_bias but bias is NULL");
  if (!p->has_bias && bias != nullptr)
    return fail(FLCE_ERR_INVALID_ARG, "bias given but has_bias is 0");
  if (p->n > 0) {
    if (hidden == nullptr || targets == nullptr || loss_rows == nullptr || lse_rows == nullptr)
      return fail(FLCE_ERR_INVALID_ARG, "hidden, targets, loss_rows and lse_rows are required");
    if (!aligned(hidden, in_align)) return fail(FLCE_ERR_UNSUPPORTED, "hidden is misaligned");
    if (!aligned(targets, 8)) return fail(FLCE_ERR_UNSUPPORTED, "targets is misaligned");
  }
  if (!aligned(weight, in_align)) return fail(FLCE_ERR_UNSUPPORTED, "weight is misaligned");
  if (bias != nullptr && !aligned(bias, in_align))
    return fail(FLCE_ERR_UNSUPPORTED, "bias is misaligned");
  return FLCE_OK;
}

// Valid-row compaction (FLCE_SKIP_IGNORED_ROWS): row_map / n_kept from the
// targets, then the kept rows of hidden (and, through `gp`, of the per-row
// inputs the caller names) gathered into the workspace. `cp` and `gp` carry
// the caller's optional outputs; the common fields are filled here.
flce_status launch_compaction(const flce_problem* p, const CompactPlan& plan, uint8_t* ws,
                              const void* hidden, const int64_t* targets, flce::CompactParams cp,
                              flce::GatherParams gp, cudaStream_t s) {
  int32_t* row_map = reinterpret_cast<int32_t*>(ws + plan.row_map);
  int32_t* n_kept = reinterpret_cast<int32_t*>(ws + plan.n_kept);
  cp.targets = targets;
  cp.n = p->n;
  cp.ignore_index = p->ignore_index;
  cp.row_map = row_map;
  cp.n_kept = n_kept;
  gp.hidden = hidden;
  gp.n = p->n;
  gp.h = p->h;
  gp.row_map = row_map;
  gp.n_kept = n_kept;
  gp.pad_rows = flce::kTileRowsTC;
  gp.hidden_c = ws + plan.hidden_c;
  gp.targets = targets;
  gp.targets_c = reinterpret_cast<int64_t*>(ws + plan.targets_c);
  gp.ignore_index = p->ignore_index;
  cudaError_t e;
  {
    ProfScope ps("compact_rows", s);
    e = flce::launch_compact_rows(cp, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "row compaction kernel");
  {
    ProfScope ps("gather_rows", s);
    e = flce::launch_gather_rows(gp, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "row gather kernel");
  return FLCE_OK;
}

// ------------------------------------------------------------ KL problems
// The KL divergence runs on the cross-entropy's plans and kernels: its
// problem maps to an flce_problem with logit_scale = 1 / temperature, no
// softcap, and the reduction code the shared steps understand (none 0,
// sum 1, batchmean and mean 2: an average over counted rows; "mean" further
// divides by V where it is applied).
flce_status check_kl_problem(const flce_kl_problem* k, flce_problem* ce) {
  if (k == nullptr) return fail(FLCE_ERR_INVALID_ARG, "problem pointer is NULL");
  if (!(k->temperature > 0.0f) || !std::isfinite(k->temperature) ||
      !std::isfinite(1.0f / k->temperature))
    return fail(FLCE_ERR_INVALID_ARG, "temperature must be finite and > 0 (with 1/T finite)");
  if (!(k->eps > 0.0f) || !std::isfinite(k->eps))
    return fail(FLCE_ERR_INVALID_ARG, "eps must be finite and > 0");
  if (k->reduction < FLCE_KL_NONE || k->reduction > FLCE_KL_MEAN)
    return fail(FLCE_ERR_INVALID_ARG, "reduction must be none, sum, batchmean or mean");
  if (k->reserved != 0) return fail(FLCE_ERR_INVALID_ARG, "non-zero reserved field");
  std::memset(ce, 0, sizeof(*ce));
  ce->n = k->n;
  ce->h = k->h;
  ce->v = k->v;
  ce->dtype = k->dtype;
  ce->has_bias = k->has_bias;
  ce->ignore_index = k->ignore_index;
  ce->logit_scale = 1.0f / k->temperature;
  ce->softcap = 0.0f;
  ce->reduction = k->reduction == FLCE_KL_NONE  ? FLCE_RED_NONE
                  : k->reduction == FLCE_KL_SUM ? FLCE_RED_SUM
                                                : FLCE_RED_MEAN;
  ce->grad_weight_dtype = k->grad_weight_dtype;
  ce->vocab_chunk = k->vocab_chunk;
  ce->flags = k->flags;
  return check_problem(ce);
}

struct KLFwdPlan {
  int64_t n_vt = 0;
  size_t partials = 0, sched = 0, total = 0;
  CompactPlan cp;
  bool split = false;  // as in FwdPlan
  int64_t split_chunk = 0;
  size_t split_h = 0, split_w = 0;
};

KLFwdPlan plan_kl_forward(const flce_problem* ce) {
  KLFwdPlan f;
  f.split = is_split(ce);
  f.n_vt = forward_parts(ce, f.split);
  size_t off = align_up(static_cast<size_t>(ce->n) * f.n_vt * 16);
  f.sched = off;  // tile counter of the forward GEMM
  if (is_tc(ce)) off = align_up(off + sizeof(int));
  off = plan_compaction(ce, false, true, off, &f.cp);
  if (f.split) {
    f.split_chunk = split_chunk(ce);
    f.split_h = off;
    off = align_up(off + 3 * static_cast<size_t>(ce->n) * ce->h * 2);
    f.split_w = off;
    off = align_up(off + 3 * static_cast<size_t>(f.split_chunk) * ce->h * 2);
  }
  f.total = off;
  return f;
}

// KL inputs of the shared backward (null for the cross-entropy).
struct KLArgs {
  const void* q;      // teacher probabilities [N][V], input type
  const float* qsum;  // per-row sum of q
  int reduction;      // flce_kl_reduction
};

// The backward of both losses: the cross-entropy (kl == null) and the KL
// divergence (kl != null: D from the teacher probabilities; targets are the
// optional labels). `p` has been checked by the caller.
flce_status backward_impl(const flce_problem* p, const KLArgs* kl, const void* hidden,
                          const void* weight, const void* bias, const int64_t* targets,
                          const float* lse_rows, const int32_t* n_valid, const float* grad_out,
                          void* grad_hidden, void* grad_weight, void* grad_bias,
                          int32_t* err_word, void* workspace, size_t workspace_bytes,
                          void* stream) {
  flce_status st = FLCE_OK;
  const bool bf16 = is_tc(p);  // tensor-core path (bf16 or fp16)
  const size_t in_align = bf16 ? 16 : 4;
  g_map_type = p->dtype == FLCE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (weight == nullptr || grad_weight == nullptr)
    return fail(FLCE_ERR_INVALID_ARG, "weight and grad_weight are required");
  if (p->has_bias && (bias == nullptr || grad_bias == nullptr))
    return fail(FLCE_ERR_INVALID_ARG, "has_bias needs bias and grad_bias");
  if (!p->has_bias && (bias != nullptr || grad_bias != nullptr))
    return fail(FLCE_ERR_INVALID_ARG, "bias/grad_bias given but has_bias is 0");
  if (p->n > 0) {
    if (hidden == nullptr || lse_rows == nullptr || n_valid == nullptr || grad_out == nullptr ||
        grad_hidden == nullptr)
      return fail(FLCE_ERR_INVALID_ARG,
                  "hidden, lse_rows, n_valid, grad_out and grad_hidden are required");
    if (!aligned(hidden, in_align) || !aligned(grad_hidden, in_align))
      return fail(FLCE_ERR_UNSUPPORTED, "hidden or grad_hidden is misaligned");
    if (targets != nullptr && !aligned(targets, 8))
      return fail(FLCE_ERR_UNSUPPORTED, "targets is misaligned");
  }
  if (!aligned(weight, in_align) || !aligned(grad_weight, in_align))
    return fail(FLCE_ERR_UNSUPPORTED, "weight or grad_weight is misaligned");
  if (bias != nullptr && !aligned(bias, in_align))
    return fail(FLCE_ERR_UNSUPPORTED, "bias is misaligned");
  const BwdPlan plan = plan_backward(p, kl != nullptr);
  st = check_workspace(workspace, workspace_bytes, plan.total);
  if (st != FLCE_OK) return st;
  DeviceInfo dev;
  st = check_device(&dev);
  if (st != FLCE_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t gw_elem = p->grad_weight_dtype == FLCE_F32 ? 4 : 2;
  cudaError_t e;
  if (p->n == 0) {
    e = cudaMemsetAsync(grad_weight, 0, static_cast<size_t>(p->v) * p->h * gw_elem, s);
    if (e == cudaSuccess && grad_bias != nullptr)
      e = cudaMemsetAsync(grad_bias, 0, static_cast<size_t>(p->v) * (bf16 ? 2 : 4), s);
    return e == cudaSuccess ? FLCE_OK : cuda_fail(e, "cudaMemsetAsync");
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const flce::LogitXform xf = make_xform(p);
  float* gb_partial = p->has_bias ? reinterpret_cast<float*>(ws + plan.gb) : nullptr;
  // valid-row compaction (rows come from the targets, so none without them)
  const bool compact = plan.cp.on && targets != nullptr;

  if (bf16) {
    void* dbuf = ws + plan.d;
    float* acc = plan.use_acc ? reinterpret_cast<float*>(ws + plan.acc) : nullptr;
    const int type = tc_type(p);
    int* sched = reinterpret_cast<int*>(ws + plan.sched);
    e = cudaMemsetAsync(sched, 0, plan.sched_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (tile counters)");
    // fp16: D is stored times a power of two, undone by the gradient GEMMs
    float* scales = p->dtype == FLCE_F16 ? reinterpret_cast<float*>(ws + plan.scales) : nullptr;
    if (scales != nullptr) {
      ProfScope ps("dlogits_scale", s);
      // KL: |p Q - q| <= Q bounds D per row; "mean" also divides by V
      const float extra_div =
          (kl != nullptr && kl->reduction == FLCE_KL_MEAN) ? static_cast<float>(p->v) : 1.0f;
      e = flce::launch_dlogits_scale(grad_out, n_valid, targets, p->n, p->ignore_index,
                                     p->reduction, p->logit_scale, p->z_loss, lse_rows,
                                     kl != nullptr ? kl->qsum : nullptr, extra_div, scales, s);
      if (e != cudaSuccess) return cuda_fail(e, "dlogits scale kernel");
    }
    // valid-row compaction: rows of hidden, targets, lse, per-row upstream
    // gradients (and KL row sums of q) are gathered; grad_hidden is
    // scattered back
    int32_t* row_map = compact ? reinterpret_cast<int32_t*>(ws + plan.cp.row_map) : nullptr;
    int32_t* n_kept = compact ? reinterpret_cast<int32_t*>(ws + plan.cp.n_kept) : nullptr;
    const void* rows_src = hidden;
    const int64_t* rows_targets = targets;
    const float* rows_lse = lse_rows;
    const float* rows_grad = grad_out;
    const float* rows_qsum = kl != nullptr ? kl->qsum : nullptr;
    if (compact) {
      flce::GatherParams gp{};
      gp.lse = lse_rows;
      gp.lse_c = reinterpret_cast<float*>(ws + plan.cp.lse_c);
      if (p->reduction == FLCE_RED_NONE) {
        gp.grad_rows = grad_out;
        gp.grad_rows_c = reinterpret_cast<float*>(ws + plan.cp.grad_c);
      }
      if (kl != nullptr) {
        gp.qsum = kl->qsum;
        gp.qsum_c = reinterpret_cast<float*>(ws + plan.cp.qsum_c);
      }
      st = launch_compaction(p, plan.cp, ws, hidden, targets, flce::CompactParams{}, gp, s);
      if (st != FLCE_OK) return st;
      {
        ProfScope ps("zero_ignored_rows", s);
        e = flce::launch_zero_ignored_rows(targets, p->n, p->ignore_index, grad_hidden, p->h,
                                           s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "grad_hidden zero kernel");
      rows_src = ws + plan.cp.hidden_c;
      rows_targets = reinterpret_cast<const int64_t*>(ws + plan.cp.targets_c);
      rows_lse = gp.lse_c;
      if (p->reduction == FLCE_RED_NONE) rows_grad = gp.grad_rows_c;
      if (kl != nullptr) rows_qsum = gp.qsum_c;
    }
    CUtensorMap tm_h_k, tm_w_k, tm_h_mn, tm_w_mn;
    if (!make_map(&tm_h_k, "hidden", rows_src, p->h, p->n, p->h, flce::kBK, flce::kBM) ||
        !make_map(&tm_w_k, "weight", weight, p->h, p->v, p->h, flce::kBK, flce::kBLoadRowsTC) ||
        !make_map(&tm_h_mn, "hidden^T", rows_src, p->h, p->n, p->h, 64, flce::kBK) ||
        !make_map(&tm_w_mn, "weight^T", weight, p->h, p->v, p->h, 64, flce::kBK))
      return FLCE_ERR_CUDA;
    const int h_tiles = static_cast<int>(cdiv(p->h, flce::kBN));
    for (int64_t c = 0; c < plan.n_chunks; ++c) {
      const int64_t c0 = c * plan.chunk;
      const int64_t width = (p->v - c0) < plan.chunk ? (p->v - c0) : plan.chunk;
      CUtensorMap tm_d_k, tm_d_mn, tm_d_st;
      if (!make_map(&tm_d_k, "dlogits", dbuf, width, p->n, plan.chunk, flce::kBK, flce::kBM) ||
          !make_map(&tm_d_mn, "dlogits^T", dbuf, width, p->n, plan.chunk, 64, flce::kBK) ||
          !make_map(&tm_d_st, "dlogits store", dbuf, width, p->n, plan.chunk, 32, 32, false))
        return FLCE_ERR_CUDA;

      // 1. recompute the chunk's logits and form D
      GemmGeom g1{};
      g1.m_tiles = static_cast<int>(cdiv(p->n, flce::kTileRowsTC));
      g1.n_tiles = static_cast<int>(cdiv(width, flce::kBN));
      g1.k_iters = static_cast<int>(cdiv(p->h, flce::kBK));
      g1.m_fastest = 1;
      g1.group = kBandDlogits;
      g1.b_mn0 = static_cast<int>(c0);
      g1.dyn_rows = n_kept;
      g1.dyn_axis = 0;
      g1.err_word = err_word;
      // Successive launches overlap: the next kernel's CTAs start on the SMs
      // the previous one has left. dlogits stores D only after the previous
      // chunk's gradient launch, which reads D, has completed; the gradient
      // launch reads D only after this dlogits has completed. Each kernel
      // thus completes after its predecessor, so the fp32 grad_hidden
      // accumulator is updated one chunk after another.
      g1.pdl = flce::kPdlWaitEpilogue;
      if (kDynamicDlogits) g1.sched = sched + plan.n_chunks + c;
      if (kl != nullptr) {
        flce::DlogitsKLParams dp{};
        dp.d_map = tm_d_st;
        dp.bias = bias;
        dp.q = kl->q;
        dp.q_vec = (p->v % 8 == 0 && aligned(kl->q, 16)) ? 1 : 0;
        dp.row_map = row_map;
        dp.labels = rows_targets;
        dp.lse = rows_lse;
        dp.qsum = rows_qsum;
        dp.grad_out = rows_grad;
        dp.n_counted = n_valid;
        dp.dscale = scales;
        dp.gb_partial = gb_partial;
        dp.gb_ld = p->v;
        dp.n_rows = p->n;
        dp.n_rows_dyn = n_kept;
        dp.v = p->v;
        dp.ignore_index = p->ignore_index;
        dp.c0 = static_cast<int>(c0);
        dp.width = static_cast<int>(width);
        dp.reduction = kl->reduction;
        dp.xf = xf;
        ProfScope ps("bwd_dlogits_kl", s);
        e = flce::launch_tc_dlogits_kl(type, tm_h_k, tm_w_k, g1, dp,
                                       flce::dlogits_epi_warps(p->h), dev.sms, s);
      } else {
        flce::DlogitsParams dp{};
        dp.d_map = tm_d_st;
        dp.bias = bias;
        dp.targets = rows_targets;
        dp.lse = rows_lse;
        dp.grad_out = rows_grad;
        dp.n_valid = n_valid;
        dp.dscale = scales;
        dp.gb_partial = gb_partial;
        dp.gb_ld = p->v;
        dp.n_rows = p->n;
        dp.n_rows_dyn = n_kept;
        dp.v = p->v;
        dp.ignore_index = p->ignore_index;
        dp.c0 = static_cast<int>(c0);
        dp.width = static_cast<int>(width);
        dp.reduction = p->reduction;
        dp.label_smoothing = p->label_smoothing;
        dp.z_loss = p->z_loss;
        dp.xf = xf;
        {
          ProfScope ps("bwd_dlogits", s);
          e = flce::launch_tc_dlogits(type, tm_h_k, tm_w_k, g1, dp,
                                      flce::dlogits_epi_warps(p->h), dev.sms, s);
        }
      }
      if (e != cudaSuccess) return cuda_fail(e, "dlogits kernel");

      // 2. and 3., one launch: grad_weight[c0 : c0+width] = D^T @ hidden and
      // grad_hidden (+)= D @ weight[c0 : c0+width]
      flce::GradsLaunch gl{};
      gl.tm_d_k = tm_d_k;
      gl.tm_weight_mn = tm_w_mn;
      gl.tm_d_mn = tm_d_mn;
      gl.tm_hidden_mn = tm_h_mn;
      GemmGeom& g2 = gl.g_gw;
      g2.m_tiles = static_cast<int>(cdiv(width, flce::kTileRowsTC));
      g2.n_tiles = h_tiles;
      g2.k_iters = static_cast<int>(cdiv(p->n, flce::kBK));
      g2.m_fastest = 0;
      g2.group = kBandGradWeight;
      g2.dyn_rows = n_kept;  // the contraction runs over the kept rows
      g2.dyn_axis = 1;
      g2.err_word = err_word;
      flce::StoreRowsParams& sp = gl.sp;
      sp.out = grad_weight;
      sp.out_f32 = p->grad_weight_dtype == FLCE_F32 ? 1 : 0;
      sp.out_scale = scales != nullptr ? scales + 1 : nullptr;
      sp.ld = p->h;
      sp.rows = width;
      sp.row0 = c0;
      sp.cols = static_cast<int>(p->h);
      GemmGeom& g3 = gl.g_gh;
      g3.m_tiles = static_cast<int>(cdiv(p->n, flce::kTileRowsTC));
      g3.n_tiles = h_tiles;
      g3.k_iters = static_cast<int>(cdiv(width, flce::kBK));
      g3.m_fastest = 1;
      g3.group = kBandGradHidden;
      g3.b_k0 = static_cast<int>(c0);
      g3.dyn_rows = n_kept;
      g3.dyn_axis = 0;
      g3.err_word = err_word;
      flce::AccRowsParams& ap = gl.ap;
      ap.acc = acc;
      ap.out = grad_hidden;
      ap.out_scale = scales != nullptr ? scales + 1 : nullptr;
      if (plan.n_chunks == 1)
        ap.mode = flce::kAccStoreOut;
      else if (c == 0)
        ap.mode = flce::kAccStore;
      else if (c == plan.n_chunks - 1)
        ap.mode = flce::kAccAddOut;
      else
        ap.mode = flce::kAccAdd;
      ap.ld = p->h;
      ap.rows = p->n;
      ap.rows_dyn = n_kept;
      ap.row_map = row_map;
      ap.cols = static_cast<int>(p->h);
      gl.sched = sched + c;
      g2.pdl = flce::kPdlWaitLoads | flce::kPdlWaitEpilogue;
      g3.pdl = flce::kPdlWaitLoads | flce::kPdlWaitEpilogue;
      // the longer contraction's tiles are handed out first
      gl.gh_first = g3.k_iters >= g2.k_iters;
      {
        ProfScope ps("bwd_grads", s);
        e = flce::launch_tc_grads(type, gl, dev.sms, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "gradient kernel");
    }
  } else if (plan.split) {
    // fp32 operands as three bf16 parts each (see is_split): hidden once, the
    // chunk's W rows per chunk; D is written and read as three bf16 parts
    uint8_t* hp = ws + plan.split_h;
    uint8_t* wp = ws + plan.split_w;
    uint8_t* dp0 = ws + plan.d;
    const size_t h_part = static_cast<size_t>(p->n) * p->h * 2;
    const size_t w_part = static_cast<size_t>(plan.chunk) * p->h * 2;
    const size_t d_part = static_cast<size_t>(p->n) * plan.chunk * 2;
    float* acc = plan.use_acc ? reinterpret_cast<float*>(ws + plan.acc) : nullptr;
    int* sched = reinterpret_cast<int*>(ws + plan.sched);
    e = cudaMemsetAsync(sched, 0, plan.sched_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (tile counters)");
    {
      ProfScope ps("split_f32", s);
      e = flce::launch_split3(static_cast<const float*>(hidden), p->n * p->h, hp, hp + h_part,
                              hp + 2 * h_part, dev.sms, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "fp32 split kernel");
    CUtensorMap tm_h_k[3], tm_h_mn[3];
    for (int q = 0; q < 3; ++q)
      if (!make_map(&tm_h_k[q], "hidden part", hp + q * h_part, p->h, p->n, p->h, flce::kBK,
                    flce::kBM) ||
          !make_map(&tm_h_mn[q], "hidden part^T", hp + q * h_part, p->h, p->n, p->h, 64,
                    flce::kBK))
        return FLCE_ERR_CUDA;
    const int h_tiles = static_cast<int>(cdiv(p->h, flce::kBN));
    auto set_passes = [](GemmGeom& g) {
      g.passes = 6;
      for (int q = 0; q < 6; ++q) {
        g.pass_a[q] = kSplitPassA[q];
        g.pass_b[q] = kSplitPassB[q];
      }
    };
    for (int64_t c = 0; c < plan.n_chunks; ++c) {
      const int64_t c0 = c * plan.chunk;
      const int64_t width = (p->v - c0) < plan.chunk ? (p->v - c0) : plan.chunk;
      {
        ProfScope ps("split_f32", s);
        e = flce::launch_split3(static_cast<const float*>(weight) + c0 * p->h, width * p->h, wp,
                                wp + w_part, wp + 2 * w_part, dev.sms, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "fp32 split kernel");
      CUtensorMap tm_w_k[3], tm_w_mn[3], tm_d_k[3], tm_d_mn[3], tm_d_st[3];
      for (int q = 0; q < 3; ++q) {
        uint8_t* wq = wp + q * w_part;
        uint8_t* dq = dp0 + q * d_part;
        if (!make_map(&tm_w_k[q], "weight part", wq, p->h, width, p->h, flce::kBK,
                      flce::kBLoadRowsTC) ||
            !make_map(&tm_w_mn[q], "weight part^T", wq, p->h, width, p->h, 64, flce::kBK) ||
            !make_map(&tm_d_k[q], "dlogits part", dq, width, p->n, plan.chunk, flce::kBK,
                      flce::kBM) ||
            !make_map(&tm_d_mn[q], "dlogits part^T", dq, width, p->n, plan.chunk, 64,
                      flce::kBK) ||
            !make_map(&tm_d_st[q], "dlogits part store", dq, width, p->n, plan.chunk, 32, 32,
                      false))
          return FLCE_ERR_CUDA;
      }

      // 1. the chunk's logits and D, stored as three bf16 parts
      GemmGeom g1{};
      g1.m_tiles = static_cast<int>(cdiv(p->n, flce::kTileRowsTC));
      g1.n_tiles = static_cast<int>(cdiv(width, flce::kBN));
      g1.k_iters = static_cast<int>(cdiv(p->h, flce::kBK));
      g1.m_fastest = 1;
      g1.group = kBandDlogits;
      g1.err_word = err_word;
      // the split of this chunk's W rows precedes it: loads wait too
      g1.pdl = flce::kPdlWaitLoads | flce::kPdlWaitEpilogue;
      set_passes(g1);
      flce::DlogitsParams dp{};
      dp.d_map = tm_d_st[0];
      dp.d_map_x[0] = tm_d_st[1];
      dp.d_map_x[1] = tm_d_st[2];
      dp.bias = bias;
      dp.targets = targets;
      dp.lse = lse_rows;
      dp.grad_out = grad_out;
      dp.n_valid = n_valid;
      dp.gb_partial = gb_partial;
      dp.gb_ld = p->v;
      dp.n_rows = p->n;
      dp.v = p->v;
      dp.ignore_index = p->ignore_index;
      dp.c0 = static_cast<int>(c0);
      dp.width = static_cast<int>(width);
      dp.reduction = p->reduction;
      dp.label_smoothing = p->label_smoothing;
      dp.z_loss = p->z_loss;
      dp.xf = xf;
      if (kl != nullptr) {
        flce::DlogitsKLParams dk{};
        dk.d_map = tm_d_st[0];
        dk.d_map_x[0] = tm_d_st[1];
        dk.d_map_x[1] = tm_d_st[2];
        dk.bias = bias;
        dk.q = kl->q;
        dk.q_vec = (p->v % 8 == 0 && aligned(kl->q, 16)) ? 1 : 0;
        dk.labels = targets;
        dk.lse = lse_rows;
        dk.qsum = kl->qsum;
        dk.grad_out = grad_out;
        dk.n_counted = n_valid;
        dk.gb_partial = gb_partial;
        dk.gb_ld = p->v;
        dk.n_rows = p->n;
        dk.v = p->v;
        dk.ignore_index = p->ignore_index;
        dk.c0 = static_cast<int>(c0);
        dk.width = static_cast<int>(width);
        dk.reduction = kl->reduction;
        dk.xf = xf;
        ProfScope ps("bwd_dlogits_kl_split", s);
        e = flce::launch_tc_dlogits_kl_split(tm_h_k, tm_w_k, g1, dk,
                                             flce::dlogits_epi_warps(p->h), dev.sms, s);
      } else {
        ProfScope ps("bwd_dlogits_split", s);
        e = flce::launch_tc_dlogits_split(tm_h_k, tm_w_k, g1, dp, flce::dlogits_epi_warps(p->h),
                                          dev.sms, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "split dlogits kernel");

      // 2. and 3., one launch: grad_weight[c0 : c0+width] = D^T @ hidden and
      // grad_hidden (+)= D @ weight[c0 : c0+width], six part products each
      flce::GradsSplitLaunch gl{};
      for (int q = 0; q < 3; ++q) {
        gl.d_k[q] = tm_d_k[q];
        gl.weight_mn[q] = tm_w_mn[q];
        gl.d_mn[q] = tm_d_mn[q];
        gl.hidden_mn[q] = tm_h_mn[q];
      }
      GemmGeom& g2 = gl.g_gw;
      g2.m_tiles = static_cast<int>(cdiv(width, flce::kTileRowsTC));
      g2.n_tiles = h_tiles;
      g2.k_iters = static_cast<int>(cdiv(p->n, flce::kBK));
      g2.m_fastest = 0;
      g2.group = kBandGradWeight;
      g2.err_word = err_word;
      set_passes(g2);
      flce::StoreRowsParams& sp = gl.sp;
      sp.out = grad_weight;
      sp.out_f32 = p->grad_weight_dtype == FLCE_F32 ? 1 : 0;
      sp.ld = p->h;
      sp.rows = width;
      sp.row0 = c0;
      sp.cols = static_cast<int>(p->h);
      GemmGeom& g3 = gl.g_gh;
      g3.m_tiles = static_cast<int>(cdiv(p->n, flce::kTileRowsTC));
      g3.n_tiles = h_tiles;
      g3.k_iters = static_cast<int>(cdiv(width, flce::kBK));
      g3.m_fastest = 1;
      g3.group = kBandGradHidden;
      g3.err_word = err_word;
      set_passes(g3);
      flce::AccRowsParams& ap = gl.ap;
      ap.acc = acc;
      ap.out = grad_hidden;
      ap.out_f32 = 1;
      if (plan.n_chunks == 1)
        ap.mode = flce::kAccStoreOut;
      else if (c == 0)
        ap.mode = flce::kAccStore;
      else if (c == plan.n_chunks - 1)
        ap.mode = flce::kAccAddOut;
      else
        ap.mode = flce::kAccAdd;
      ap.ld = p->h;
      ap.rows = p->n;
      ap.cols = static_cast<int>(p->h);
      gl.sched = sched + c;
      g2.pdl = flce::kPdlWaitLoads | flce::kPdlWaitEpilogue;
      g3.pdl = flce::kPdlWaitLoads | flce::kPdlWaitEpilogue;
      gl.gh_first = g3.k_iters >= g2.k_iters;
      {
        ProfScope ps("bwd_grads_split", s);
        e = flce::launch_tc_grads_split(gl, dev.sms, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "split gradient kernel");
    }
  } else {
    float* dbuf = reinterpret_cast<float*>(ws + plan.d);
    for (int64_t c = 0; c < plan.n_chunks; ++c) {
      const int64_t c0 = c * plan.chunk;
      const int64_t width = (p->v - c0) < plan.chunk ? (p->v - c0) : plan.chunk;
      flce::SimtDlogitsParams dp{};
      dp.hidden = static_cast<const float*>(hidden);
      dp.weight = static_cast<const float*>(weight);
      dp.bias = static_cast<const float*>(bias);
      dp.q = kl != nullptr ? static_cast<const float*>(kl->q) : nullptr;
      dp.qsum = kl != nullptr ? kl->qsum : nullptr;
      dp.targets = targets;
      dp.lse = lse_rows;
      dp.grad_out = grad_out;
      dp.n_valid = n_valid;
      dp.d = dbuf;
      dp.ldd = plan.chunk;
      dp.gb_partial = gb_partial;
      dp.gb_ld = p->v;
      dp.n = p->n;
      dp.h = p->h;
      dp.v = p->v;
      dp.ignore_index = p->ignore_index;
      dp.c0 = c0;
      dp.width = width;
      dp.reduction = kl != nullptr ? kl->reduction : p->reduction;
      dp.label_smoothing = p->label_smoothing;
      dp.z_loss = p->z_loss;
      dp.xf = xf;
      {
        ProfScope ps("bwd_dlogits_f32", s);
        e = flce::launch_simt_dlogits(dp, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "fp32 dlogits kernel");
      // grad_weight rows [c0, c0+width) = D^T @ hidden
      {
        ProfScope ps("bwd_grad_weight_f32", s);
        e = flce::launch_simt_gemm(width, p->h, p->n, dbuf, 1, plan.chunk,
                                 static_cast<const float*>(hidden), p->h, 1,
                                   static_cast<float*>(grad_weight) + c0 * p->h, p->h, 0, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "fp32 grad_weight kernel");
      // grad_hidden (+)= D @ weight[c0 : c0+width]
      {
        ProfScope ps("bwd_grad_hidden_f32", s);
        e = flce::launch_simt_gemm(p->n, p->h, width, dbuf, plan.chunk, 1,
                                 static_cast<const float*>(weight) + c0 * p->h, p->h, 1,
                                   static_cast<float*>(grad_hidden), p->h, c > 0 ? 1 : 0, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "fp32 grad_hidden kernel");
    }
  }
  if (p->has_bias) {
    ProfScope ps("bwd_bias_reduce", s);
    const int32_t* n_dyn =
        compact ? reinterpret_cast<const int32_t*>(ws + plan.cp.n_kept) : nullptr;
    e = flce::launch_bias_reduce(gb_partial, plan.gb_parts, p->v, p->v, grad_bias,
                                 bf16 ? tc_type(p) : 0, n_dyn, flce::kBM, s);
    if (e != cudaSuccess) return cuda_fail(e, "grad_bias kernel");
  }
  return FLCE_OK;
}


}  // namespace

// ------------------------------------------------- fixed forward scratch
// Scratch for flce_forward_noalloc(). It is one fixed array per GPU that
// loads this library and stays allocated until the process exits, so it is
// kept small: 16 MiB.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char flce_static_scratch[kStaticScratchBytes];

namespace {

// The array's device address, per device, with the id of the context it was
// looked up in: a context that is torn down and re-created (cudaDeviceReset)
// loads the module again, possibly at another address.
struct ScratchAddr {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[64];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
std::once_flag g_ctx_fn_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Unique id of the context current on the calling thread.
bool current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_fn_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of flce_static_scratch on the current device. The host-side
// name of the array is only a stand-in, so the address is looked up with
// cudaGetSymbolAddress with the device current: once per device, and again
// whenever the device's context is not the one the cached address came from.
// The caller has made the device's primary context current (check_device).
flce_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(FLCE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  unsigned long long ctx_id = 0;
  if (!current_context_id(&ctx_id))
    return fail(FLCE_ERR_CUDA, "cannot identify the current CUDA context");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& a = g_scratch_addr[dev];
  if (a.ptr == nullptr || a.ctx_id != ctx_id) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, flce_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(flce_static_scratch)");
    a.ptr = ptr;
    a.ctx_id = ctx_id;
  }
  *out = a.ptr;
  return FLCE_OK;
}

}  // namespace

extern "C" {

const char* flce_status_string(flce_status s) {
  switch (s) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARG: return "FLCE_ERR_INVALID_ARG";
    case FLCE_ERR_UNSUPPORTED: return "FLCE_ERR_UNSUPPORTED";
    case FLCE_ERR_WORKSPACE: return "FLCE_ERR_WORKSPACE";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA";
    case FLCE_ERR_DEVICE_TIMEOUT: return "FLCE_ERR_DEVICE_TIMEOUT";
  }
  return "FLCE_ERR_UNKNOWN";
}

const char* flce_last_error(void) { return g_err; }

flce_status flce_profile_enable(int enable) {
  g_err[0] = 0;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (enable && !g_prof_ready) {
    for (int i = 0; i < FLCE_PROFILE_MAX_RECORDS; ++i) {
      if (cudaEventCreate(&g_prof[i].start) != cudaSuccess ||
          cudaEventCreate(&g_prof[i].stop) != cudaSuccess)
        return fail(FLCE_ERR_CUDA, "cudaEventCreate failed");
    }
    g_prof_ready = true;
  }
  g_prof_on = enable != 0;
  g_prof_n = 0;
  g_prof_dropped = 0;
  return FLCE_OK;
}

int flce_profile_collect(flce_kernel_time* out, int max_entries, int32_t* dropped) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double total[16] = {0};
  int count[16] = {0};
  int order[16];
  int n_used = 0;
  for (int r = 0; r < g_prof_n; ++r) {
    float ms = 0.0f;
    if (cudaEventSynchronize(g_prof[r].stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof[r].start, g_prof[r].stop) != cudaSuccess)
      return -1;
    const int role = g_prof[r].role;
    if (count[role] == 0) order[n_used++] = role;
    ++count[role];
    total[role] += ms;
  }
  int written = 0;
  for (int k = 0; k < n_used && written < max_entries; ++k) {
    const int role = order[k];
    std::memset(out[written].name, 0, FLCE_PROFILE_NAME_LEN);
    std::strncpy(out[written].name, g_role_names[role], FLCE_PROFILE_NAME_LEN - 1);
    out[written].launches = count[role];
    out[written].total_ms = total[role];
    ++written;
  }
  if (dropped) *dropped = g_prof_dropped;
  g_prof_n = 0;
  g_prof_dropped = 0;
  return written;
}

int flce_device_supported(void) {
  DeviceInfo d;
  if (!device_info(&d)) return 0;
  return (d.major == 10 && d.minor == 3) ? 1 : 0;
}

size_t flce_forward_workspace_size(const flce_problem* p) {
  if (check_problem(p) != FLCE_OK) return 0;
  return plan_forward(p).total;
}

size_t flce_backward_workspace_size(const flce_problem* p) {
  if (check_problem(p) != FLCE_OK) return 0;
  return plan_backward(p).total;
}

flce_status flce_forward(const flce_problem* p, const void* hidden, const void* weight,
                         const void* bias, const int64_t* targets, float* loss_rows,
                         float* lse_rows, int32_t* correct_rows, float* entropy_rows,
                         float* loss_out, float* metrics_out, int32_t* n_valid, int32_t* err_word,
                         void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  flce_status st = check_forward_args(p, hidden, weight, bias, targets, loss_rows, lse_rows,
                                      loss_out, n_valid);
  if (st != FLCE_OK) return st;
  const bool bf16 = is_tc(p);  // tensor-core path (bf16 or fp16)
  g_map_type = p->dtype == FLCE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const FwdPlan plan = plan_forward(p);
  st = check_workspace(workspace, workspace_bytes, plan.total);
  if (st != FLCE_OK) return st;
  DeviceInfo dev;
  st = check_device(&dev);
  if (st != FLCE_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float4* partials = reinterpret_cast<float4*>(ws + plan.partials);
  float* zsum = plan.has_zsum ? reinterpret_cast<float*>(ws + plan.zsum) : nullptr;
  float* zt = reinterpret_cast<float*>(ws + plan.zt);
  int32_t* correct_ws = reinterpret_cast<int32_t*>(ws + plan.correct);
  float* entropy_ws = reinterpret_cast<float*>(ws + plan.entropy);
  const flce::LogitXform xf = make_xform(p);
  cudaError_t e;

  if (p->n > 0) {
    // valid-row compaction: the GEMMs read the kept rows from a gathered copy
    const bool compact = plan.cp.on;
    int32_t* row_map = compact ? reinterpret_cast<int32_t*>(ws + plan.cp.row_map) : nullptr;
    int32_t* n_kept = compact ? reinterpret_cast<int32_t*>(ws + plan.cp.n_kept) : nullptr;
    const void* rows_src = hidden;
    const int64_t* rows_targets = targets;
    if (compact) {
      flce::CompactParams cp{};
      cp.loss_rows = loss_rows;
      cp.lse_rows = lse_rows;
      cp.correct_ws = correct_ws;
      cp.entropy_ws = entropy_ws;
      cp.correct_rows = correct_rows;
      cp.entropy_rows = entropy_rows;
      st = launch_compaction(p, plan.cp, ws, hidden, targets, cp, flce::GatherParams{}, s);
      if (st != FLCE_OK) return st;
      rows_src = ws + plan.cp.hidden_c;
      rows_targets = reinterpret_cast<const int64_t*>(ws + plan.cp.targets_c);
    }
    if (bf16) {
      CUtensorMap tm_h, tm_w;
      if (!make_map(&tm_h, "hidden", rows_src, p->h, p->n, p->h, flce::kBK, flce::kBM) ||
          !make_map(&tm_w, "weight", weight, p->h, p->v, p->h, flce::kBK, flce::kBLoadRowsTC))
        return FLCE_ERR_CUDA;
      GemmGeom g{};
      g.m_tiles = static_cast<int>(cdiv(p->n, flce::kTileRowsTC));
      g.n_tiles = static_cast<int>(cdiv(p->v, flce::kBN));
      g.k_iters = static_cast<int>(cdiv(p->h, flce::kBK));
      g.m_fastest = 1;
      g.group = kBandForward;
      g.dyn_rows = n_kept;
      g.dyn_axis = 0;
      g.err_word = err_word;
      if (kDynamicForward) {
        g.sched = reinterpret_cast<int*>(ws + plan.sched);
        e = cudaMemsetAsync(g.sched, 0, sizeof(int), s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (tile counter)");
      }
      flce::FwdStatsParams fp{};
      fp.bias = bias;
      fp.targets = rows_targets;
      fp.partials = partials;
      fp.zsum = zsum;
      fp.zt = zt;
      fp.n_rows = p->n;
      fp.n_rows_dyn = n_kept;
      fp.v = p->v;
      fp.n_vt = plan.n_vt;
      // the argmax and entropy terms only when an output uses them
      fp.metrics = (metrics_out != nullptr || correct_rows != nullptr || entropy_rows != nullptr)
                       ? 1 : 0;
      fp.xf = xf;
      ProfScope ps("fwd_stats", s);
      e = flce::launch_tc_fwd_stats(tc_type(p), tm_h, tm_w, g, fp, flce::fwd_epi_warps(p->h),
                                    dev.sms, s);
      if (e != cudaSuccess) return cuda_fail(e, "forward statistics kernel");
    } else if (plan.split) {
      // fp32 operands as three bf16 parts each: hidden once, W one
      // vocabulary chunk at a time, six part products per tile
      uint8_t* hp = ws + plan.split_h;
      uint8_t* wp = ws + plan.split_w;
      const size_t h_part = static_cast<size_t>(p->n) * p->h * 2;
      const size_t w_part = static_cast<size_t>(plan.split_chunk) * p->h * 2;
      {
        ProfScope ps("split_f32", s);
        e = flce::launch_split3(static_cast<const float*>(hidden), p->n * p->h, hp, hp + h_part,
                                hp + 2 * h_part, dev.sms, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "fp32 split kernel");
      CUtensorMap tm_h[3];
      for (int q = 0; q < 3; ++q)
        if (!make_map(&tm_h[q], "hidden part", hp + q * h_part, p->h, p->n, p->h, flce::kBK,
                      flce::kBM))
          return FLCE_ERR_CUDA;
      for (int64_t c0 = 0; c0 < p->v; c0 += plan.split_chunk) {
        const int64_t width = (p->v - c0) < plan.split_chunk ? (p->v - c0) : plan.split_chunk;
        {
          ProfScope ps("split_f32", s);
          e = flce::launch_split3(static_cast<const float*>(weight) + c0 * p->h, width * p->h,
                                  wp, wp + w_part, wp + 2 * w_part, dev.sms, s);
        }
        if (e != cudaSuccess) return cuda_fail(e, "fp32 split kernel");
        CUtensorMap tm_w[3];
        for (int q = 0; q < 3; ++q)
          if (!make_map(&tm_w[q], "weight part", wp + q * w_part, p->h, width, p->h, flce::kBK,
                        flce::kBLoadRowsTC))
            return FLCE_ERR_CUDA;
        GemmGeom g{};
        g.m_tiles = static_cast<int>(cdiv(p->n, flce::kTileRowsTC));
        g.n_tiles = static_cast<int>(cdiv(width, flce::kBN));
        g.k_iters = static_cast<int>(cdiv(p->h, flce::kBK));
        g.m_fastest = 1;
        g.group = kBandForward;
        g.err_word = err_word;
        g.passes = 6;
        for (int q = 0; q < 6; ++q) {
          g.pass_a[q] = kSplitPassA[q];
          g.pass_b[q] = kSplitPassB[q];
        }
        flce::FwdStatsParams fp{};
        fp.bias = bias;
        fp.targets = targets;
        fp.partials = partials;
        fp.zsum = zsum;
        fp.zt = zt;
        fp.n_rows = p->n;
        fp.v = p->v;
        fp.n_vt = plan.n_vt;
        fp.metrics =
            (metrics_out != nullptr || correct_rows != nullptr || entropy_rows != nullptr) ? 1 : 0;
        fp.xf = xf;
        fp.c0 = c0;
        ProfScope ps("fwd_stats_split", s);
        e = flce::launch_tc_fwd_stats_split(tm_h, tm_w, g, fp, flce::fwd_epi_warps(p->h),
                                            dev.sms, s);
        if (e != cudaSuccess) return cuda_fail(e, "split forward statistics kernel");
      }
    } else {
      flce::SimtFwdParams fp{};
      fp.hidden = static_cast<const float*>(hidden);
      fp.weight = static_cast<const float*>(weight);
      fp.bias = static_cast<const float*>(bias);
      fp.targets = targets;
      fp.partials = partials;
      fp.zsum = zsum;
      fp.zt = zt;
      fp.n = p->n;
      fp.h = p->h;
      fp.v = p->v;
      fp.n_vt = plan.n_vt;
      fp.xf = xf;
      ProfScope ps("fwd_stats_f32", s);
      e = flce::launch_simt_fwd(fp, s);
      if (e != cudaSuccess) return cuda_fail(e, "fp32 forward kernel");
    }
    flce::MergeParams mp{};
    mp.partials = partials;
    mp.zsum = zsum;
    mp.label_smoothing = p->label_smoothing;
    mp.z_loss = p->z_loss;
    mp.zt = zt;
    mp.targets = rows_targets;
    mp.row_map = row_map;
    mp.n_dyn = n_kept;
    mp.n = p->n;
    mp.v = p->v;
    mp.n_vt = plan.n_vt;
    mp.ignore_index = p->ignore_index;
    mp.loss_rows = loss_rows;
    mp.lse_rows = lse_rows;
    mp.correct_ws = correct_ws;
    mp.entropy_ws = entropy_ws;
    mp.correct_rows = correct_rows;
    mp.entropy_rows = entropy_rows;
    mp.err_word = err_word;
    {
      ProfScope ps("merge_rows", s);
      e = flce::launch_merge_rows(mp, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "row merge kernel");
  }
  flce::FinalizeParams fin{};
  fin.loss_rows = loss_rows;
  fin.correct_ws = correct_ws;
  fin.entropy_ws = entropy_ws;
  fin.targets = targets;
  fin.n = p->n;
  fin.ignore_index = p->ignore_index;
  fin.reduction = p->reduction;
  fin.loss_out = p->reduction == FLCE_RED_NONE ? nullptr : loss_out;
  fin.metrics_out = metrics_out;
  fin.n_valid = n_valid;
  {
    ProfScope ps("finalize", s);
    e = flce::launch_finalize(fin, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "finalize kernel");
  return FLCE_OK;
}

flce_status flce_backward(const flce_problem* p, const void* hidden, const void* weight,
                          const void* bias, const int64_t* targets, const float* lse_rows,
                          const int32_t* n_valid, const float* grad_out, void* grad_hidden,
                          void* grad_weight, void* grad_bias, int32_t* err_word, void* workspace,
                          size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  flce_status st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (p->n > 0 && targets == nullptr) return fail(FLCE_ERR_INVALID_ARG, "targets is NULL");
  return backward_impl(p, nullptr, hidden, weight, bias, targets, lse_rows, n_valid, grad_out,
                       grad_hidden, grad_weight, grad_bias, err_word, workspace, workspace_bytes,
                       stream);
}

// ---------------------------------------------------------------- KL
size_t flce_kl_forward_workspace_size(const flce_kl_problem* p) {
  flce_problem ce;
  if (check_kl_problem(p, &ce) != FLCE_OK) return 0;
  return plan_kl_forward(&ce).total;
}

size_t flce_kl_backward_workspace_size(const flce_kl_problem* p) {
  flce_problem ce;
  if (check_kl_problem(p, &ce) != FLCE_OK) return 0;
  return plan_backward(&ce, true).total;
}

flce_status flce_kl_forward(const flce_kl_problem* k, const void* hidden, const void* weight,
                            const void* bias, const void* target_probs, const int64_t* labels,
                            float* loss_rows, float* lse_rows, float* qsum_rows, float* loss_out,
                            int32_t* n_counted, int32_t* err_word, void* workspace,
                            size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  flce_problem ce;
  flce_problem* p = &ce;
  flce_status st = check_kl_problem(k, p);
  if (st != FLCE_OK) return st;
  const bool tc = is_tc(p);
  const size_t in_align = tc ? 16 : 4;
  const size_t elem = tc ? 2 : 4;
  g_map_type = p->dtype == FLCE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (weight == nullptr) return fail(FLCE_ERR_INVALID_ARG, "weight is NULL");
  if (n_counted == nullptr) return fail(FLCE_ERR_INVALID_ARG, "n_counted is NULL");
  if (k->reduction != FLCE_KL_NONE && loss_out == nullptr)
    return fail(FLCE_ERR_INVALID_ARG, "loss_out is NULL (required unless reduction is none)");
  if (p->has_bias && bias == nullptr) return fail(FLCE_ERR_INVALID_ARG, "has_bias but bias is NULL");
  if (!p->has_bias && bias != nullptr)
    return fail(FLCE_ERR_INVALID_ARG, "bias given but has_bias is 0");
  if (p->n > 0) {
    if (hidden == nullptr || target_probs == nullptr || loss_rows == nullptr ||
        lse_rows == nullptr || qsum_rows == nullptr)
      return fail(FLCE_ERR_INVALID_ARG,
                  "hidden, target_probs, loss_rows, lse_rows and qsum_rows are required");
    if (!aligned(hidden, in_align)) return fail(FLCE_ERR_UNSUPPORTED, "hidden is misaligned");
    if (!aligned(target_probs, elem))
      return fail(FLCE_ERR_UNSUPPORTED, "target_probs is misaligned");
    if (labels != nullptr && !aligned(labels, 8))
      return fail(FLCE_ERR_UNSUPPORTED, "labels is misaligned");
  }
  if (!aligned(weight, in_align)) return fail(FLCE_ERR_UNSUPPORTED, "weight is misaligned");
  if (bias != nullptr && !aligned(bias, in_align))
    return fail(FLCE_ERR_UNSUPPORTED, "bias is misaligned");
  const KLFwdPlan plan = plan_kl_forward(p);
  st = check_workspace(workspace, workspace_bytes, plan.total);
  if (st != FLCE_OK) return st;
  DeviceInfo dev;
  st = check_device(&dev);
  if (st != FLCE_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float4* partials = reinterpret_cast<float4*>(ws + plan.partials);
  const flce::LogitXform xf = make_xform(p);
  cudaError_t e;
  if (p->n > 0) {
    const bool compact = plan.cp.on && labels != nullptr;
    int32_t* row_map = compact ? reinterpret_cast<int32_t*>(ws + plan.cp.row_map) : nullptr;
    int32_t* n_kept = compact ? reinterpret_cast<int32_t*>(ws + plan.cp.n_kept) : nullptr;
    const void* rows_src = hidden;
    const int64_t* rows_labels = labels;
    if (compact) {
      flce::CompactParams cp{};
      cp.loss_rows = loss_rows;
      cp.lse_rows = lse_rows;
      cp.qsum_rows = qsum_rows;
      st = launch_compaction(p, plan.cp, ws, hidden, labels, cp, flce::GatherParams{}, s);
      if (st != FLCE_OK) return st;
      rows_src = ws + plan.cp.hidden_c;
      rows_labels = reinterpret_cast<const int64_t*>(ws + plan.cp.targets_c);
    }
    if (tc) {
      CUtensorMap tm_h, tm_w;
      if (!make_map(&tm_h, "hidden", rows_src, p->h, p->n, p->h, flce::kBK, flce::kBM) ||
          !make_map(&tm_w, "weight", weight, p->h, p->v, p->h, flce::kBK, flce::kBLoadRowsTC))
        return FLCE_ERR_CUDA;
      GemmGeom g{};
      g.m_tiles = static_cast<int>(cdiv(p->n, flce::kTileRowsTC));
      g.n_tiles = static_cast<int>(cdiv(p->v, flce::kBN));
      g.k_iters = static_cast<int>(cdiv(p->h, flce::kBK));
      g.m_fastest = 1;
      g.group = kBandForward;
      g.dyn_rows = n_kept;
      g.dyn_axis = 0;
      g.err_word = err_word;
      if (kDynamicForward) {
        g.sched = reinterpret_cast<int*>(ws + plan.sched);
        e = cudaMemsetAsync(g.sched, 0, sizeof(int), s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (tile counter)");
      }
      flce::FwdKLParams fp{};
      fp.bias = bias;
      fp.q = target_probs;
      fp.q_vec = (p->v % 8 == 0 && aligned(target_probs, 16)) ? 1 : 0;
      fp.row_map = row_map;
      fp.partials = partials;
      fp.n_rows = p->n;
      fp.n_rows_dyn = n_kept;
      fp.v = p->v;
      fp.n_vt = plan.n_vt;
      fp.eps = k->eps;
      fp.xf = xf;
      ProfScope ps("fwd_kl", s);
      e = flce::launch_tc_fwd_kl(tc_type(p), tm_h, tm_w, g, fp, flce::fwd_epi_warps(p->h),
                                 dev.sms, s);
      if (e != cudaSuccess) return cuda_fail(e, "KL forward kernel");
    } else if (plan.split) {
      // as the cross-entropy's split forward, with the teacher rows in fp32
      uint8_t* hp = ws + plan.split_h;
      uint8_t* wp = ws + plan.split_w;
      const size_t h_part = static_cast<size_t>(p->n) * p->h * 2;
      const size_t w_part = static_cast<size_t>(plan.split_chunk) * p->h * 2;
      {
        ProfScope ps("split_f32", s);
        e = flce::launch_split3(static_cast<const float*>(hidden), p->n * p->h, hp, hp + h_part,
                                hp + 2 * h_part, dev.sms, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "fp32 split kernel");
      CUtensorMap tm_h[3];
      for (int q = 0; q < 3; ++q)
        if (!make_map(&tm_h[q], "hidden part", hp + q * h_part, p->h, p->n, p->h, flce::kBK,
                      flce::kBM))
          return FLCE_ERR_CUDA;
      for (int64_t c0 = 0; c0 < p->v; c0 += plan.split_chunk) {
        const int64_t width = (p->v - c0) < plan.split_chunk ? (p->v - c0) : plan.split_chunk;
        {
          ProfScope ps("split_f32", s);
          e = flce::launch_split3(static_cast<const float*>(weight) + c0 * p->h, width * p->h,
                                  wp, wp + w_part, wp + 2 * w_part, dev.sms, s);
        }
        if (e != cudaSuccess) return cuda_fail(e, "fp32 split kernel");
        CUtensorMap tm_w[3];
        for (int q = 0; q < 3; ++q)
          if (!make_map(&tm_w[q], "weight part", wp + q * w_part, p->h, width, p->h, flce::kBK,
                        flce::kBLoadRowsTC))
            return FLCE_ERR_CUDA;
        GemmGeom g{};
        g.m_tiles = static_cast<int>(cdiv(p->n, flce::kTileRowsTC));
        g.n_tiles = static_cast<int>(cdiv(width, flce::kBN));
        g.k_iters = static_cast<int>(cdiv(p->h, flce::kBK));
        g.m_fastest = 1;
        g.group = kBandForward;
        g.err_word = err_word;
        g.passes = 6;
        for (int q = 0; q < 6; ++q) {
          g.pass_a[q] = kSplitPassA[q];
          g.pass_b[q] = kSplitPassB[q];
        }
        flce::FwdKLParams fp{};
        fp.bias = bias;
        fp.q = target_probs;
        fp.q_vec = (p->v % 8 == 0 && aligned(target_probs, 16)) ? 1 : 0;
        fp.partials = partials;
        fp.n_rows = p->n;
        fp.v = p->v;
        fp.n_vt = plan.n_vt;
        fp.eps = k->eps;
        fp.xf = xf;
        fp.c0 = c0;
        ProfScope ps("fwd_kl_split", s);
        e = flce::launch_tc_fwd_kl_split(tm_h, tm_w, g, fp, flce::fwd_epi_warps(p->h), dev.sms,
                                         s);
        if (e != cudaSuccess) return cuda_fail(e, "split KL forward kernel");
      }
    } else {
      flce::SimtFwdParams fp{};
      fp.hidden = static_cast<const float*>(hidden);
      fp.weight = static_cast<const float*>(weight);
      fp.bias = static_cast<const float*>(bias);
      fp.q = static_cast<const float*>(target_probs);
      fp.eps = k->eps;
      fp.partials = partials;
      fp.n = p->n;
      fp.h = p->h;
      fp.v = p->v;
      fp.n_vt = plan.n_vt;
      fp.xf = xf;
      ProfScope ps("fwd_kl_f32", s);
      e = flce::launch_simt_fwd(fp, s);
      if (e != cudaSuccess) return cuda_fail(e, "fp32 KL forward kernel");
    }
    flce::MergeKLParams mp{};
    mp.partials = partials;
    mp.labels = rows_labels;
    mp.row_map = row_map;
    mp.n_dyn = n_kept;
    mp.n = p->n;
    mp.n_vt = plan.n_vt;
    mp.ignore_index = p->ignore_index;
    mp.loss_rows = loss_rows;
    mp.lse_rows = lse_rows;
    mp.qsum_rows = qsum_rows;
    {
      ProfScope ps("merge_kl", s);
      e = flce::launch_merge_kl(mp, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "KL row merge kernel");
  }
  flce::FinalizeKLParams fin{};
  fin.loss_rows = loss_rows;
  fin.labels = labels;
  fin.n = p->n;
  fin.v = p->v;
  fin.ignore_index = p->ignore_index;
  fin.reduction = k->reduction;
  fin.loss_out = k->reduction == FLCE_KL_NONE ? nullptr : loss_out;
  fin.n_counted = n_counted;
  {
    ProfScope ps("finalize_kl", s);
    e = flce::launch_finalize_kl(fin, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "KL finalize kernel");
  return FLCE_OK;
}

flce_status flce_kl_backward(const flce_kl_problem* k, const void* hidden, const void* weight,
                             const void* bias, const void* target_probs, const int64_t* labels,
                             const float* lse_rows, const float* qsum_rows,
                             const int32_t* n_counted, const float* grad_out, void* grad_hidden,
                             void* grad_weight, void* grad_bias, int32_t* err_word,
                             void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  flce_problem ce;
  flce_status st = check_kl_problem(k, &ce);
  if (st != FLCE_OK) return st;
  if (ce.n > 0) {
    if (target_probs == nullptr || qsum_rows == nullptr)
      return fail(FLCE_ERR_INVALID_ARG, "target_probs and qsum_rows are required");
    if (!aligned(target_probs, is_tc(&ce) ? 2 : 4))
      return fail(FLCE_ERR_UNSUPPORTED, "target_probs is misaligned");
  }
  const KLArgs kl{target_probs, qsum_rows, k->reduction};
  return backward_impl(&ce, &kl, hidden, weight, bias, labels, lse_rows, n_counted, grad_out,
                       grad_hidden, grad_weight, grad_bias, err_word, workspace, workspace_bytes,
                       stream);
}

flce_status flce_selftest_wait_timeout(int32_t* err_word, int32_t* result, double budget_s,
                                       void* stream) {
  g_err[0] = 0;
  if (err_word == nullptr || result == nullptr)
    return fail(FLCE_ERR_INVALID_ARG, "err_word and result are required");
  if (!(budget_s > 0.0) || budget_s > 1.0)
    return fail(FLCE_ERR_INVALID_ARG, "budget_s must be in (0, 1] seconds");
  DeviceInfo dev;
  flce_status st = check_device(&dev);
  if (st != FLCE_OK) return st;
  const cudaError_t e =
      flce::launch_wait_selftest(err_word, static_cast<uint64_t>(budget_s * 1e9), result,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FLCE_OK : cuda_fail(e, "wait self-test kernel");
}

// Forward pass for callers that cannot provide a workspace: the same kernels
// as flce_forward(), with their scratch taken from flce_static_scratch.
flce_status flce_forward_noalloc(const flce_problem* p, const void* hidden, const void* weight,
                                 const void* bias, const int64_t* targets, float* loss_rows,
                                 float* lse_rows, int32_t* correct_rows, float* entropy_rows,
                                 float* loss_out, float* metrics_out, int32_t* n_valid,
                                 int32_t* err_word, void* stream) {
  g_err[0] = 0;
  flce_status st = check_forward_args(p, hidden, weight, bias, targets, loss_rows, lse_rows,
                                      loss_out, n_valid);
  if (st != FLCE_OK) return st;
  const size_t need = plan_forward(p).total;
  if (need > kStaticScratchBytes)
    return fail(FLCE_ERR_UNSUPPORTED,
                "flce_forward_noalloc: this problem needs %zu bytes of scratch, the fixed "
                "scratch holds %zu (flce_forward_workspace_size must not exceed it); "
                "call flce_forward with a workspace instead",
                need, kStaticScratchBytes);
  // the same device check, in the same order, as flce_forward: an unsupported
  // or absent device gives the same status before the symbol is looked up
  DeviceInfo dev;
  st = check_device(&dev);
  if (st != FLCE_OK) return st;
  void* scratch = nullptr;
  st = static_scratch(&scratch);
  if (st != FLCE_OK) return st;
  // Nothing in the scratch needs to start at zero: every element the kernels
  // read is first written by the same call.
  return flce_forward(p, hidden, weight, bias, targets, loss_rows, lse_rows, correct_rows,
                      entropy_rows, loss_out, metrics_out, n_valid, err_word, scratch,
                      kStaticScratchBytes, stream);
}

}  // extern "C"
