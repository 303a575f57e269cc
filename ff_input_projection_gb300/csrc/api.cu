// C ABI of libfp: argument checks, layout analysis, tensor maps, launches.
//
// fp_forward never synchronises (the Walrus PR #12 "Make fused_ff_qkv
// contiguous" profile counts five implicit device syncs per forward; this path
// adds none). Checks run on the host before any CUDA call, so a rejected call
// has launched nothing.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <vector>

#include "../../include/fp.h"
#include "fp_internal.h"

struct fp_plan {
  int C, F, heads, hd, groups, rope_n_elem;
  int k_transposed;
  int act;
  float rope_base;
  int device;
  int* d_status;     // [2]: sticky device error, tag of an aborted launch
  float2* d_table;   // rotary (cos, sin) table
  float* d_attn;     // partial results of the attention's split tail
  int64_t attn_cap;  // bytes
  int64_t table_cap; // entries
  int64_t table_T;   // T of the default-position table held in d_table (-1: none)
  cudaStream_t table_stream;  // stream that last wrote the table
  cudaEvent_t table_ready;    // recorded after that write
  // backward: the q/k/v gather runs beside the ff-gradient GEMM on this stream,
  // forked from and joined back to the caller's stream by the two events
  cudaStream_t side_stream;
  cudaEvent_t ev_fork, ev_join;
  int last_launches;
  uint64_t wait_limit_ns;
  int inject_stall;
  int group_m;
  int max_ctas;
  int cluster;  // CTAs per cluster on the tensor-core path (1 or 2)
  int bounds_check;  // FP_OPT_BOUNDS_CHECK
  int tile_n;        // FP_OPT_TILE_N
  uint32_t launch_seq;
  // Scratch grown inside a call is allocated in stream order on that call's
  // stream (scratch_stream); scratch_ready is recorded there after the growth,
  // and calls on other streams wait for it. Tables it replaced may still be
  // read by queued work, so they are kept here until fp_destroy or fp_reserve.
  cudaStream_t scratch_stream;
  cudaEvent_t scratch_ready;
  bool scratch_pending;
  std::vector<void*> retired;
  // fp_forward_host: device staging for two chunks in flight, the upload and
  // download streams, and per-slot events (upload done, compute done,
  // download done) plus the fork event recorded on the caller's stream
  void* d_host_stage = nullptr;
  int64_t host_stage_cap = 0;  // bytes
  cudaStream_t up_stream = nullptr, down_stream = nullptr;
  cudaEvent_t ev_host_fork = nullptr;
  cudaEvent_t ev_up[2] = {nullptr, nullptr}, ev_comp[2] = {nullptr, nullptr},
              ev_down[2] = {nullptr, nullptr};
  int host_last = 0;  // slot of the previous host call's last download
};

namespace {

// Launch knobs shared by plans (their defaults) and the no-allocation entry point.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;
constexpr int kDefaultGroupM = 32;   // M-tiles per rasterisation group
constexpr int kDefaultCluster = 2;   // CTA pairs on the tensor-core path

// NVTX range over one entry-point call (visible in Nsight timelines; a no-op
// when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

thread_local char g_err[512];

fp_status fail(fp_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return st;
}

fp_status ok() {
  g_err[0] = '\0';
  return FP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(const Range& a, const Range& b) {
  return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int sm_count(int dev) {
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

// Token axes after dropping unit axes and merging contiguous neighbours.
struct TokAxes {
  int64_t S_in = 1, s_stride = 1;
  int n_outer = 0;
  int64_t outer_size[FP_MAX_DIMS], outer_stride[FP_MAX_DIMS];  // innermost first
  int64_t Bb = 1, T = 1, M = 1;
};

TokAxes analyse_tokens(const fp_layout& L) {
  TokAxes ta;
  int seen = 0;
  for (int a = 0; a < L.ndim; ++a) {
    if (a == L.channel_dim) continue;
    if (seen < L.n_batch_dims) ta.Bb *= L.sizes[a];
    else ta.T *= L.sizes[a];
    ++seen;
  }
  ta.M = ta.Bb * ta.T;
  // innermost-first list of (size, stride) groups
  int64_t gs[FP_MAX_DIMS], gt[FP_MAX_DIMS];
  int ng = 0;
  for (int a = L.ndim - 1; a >= 0; --a) {
    if (a == L.channel_dim || L.sizes[a] == 1) continue;
    if (ng > 0 && L.strides[a] == gt[ng - 1] * gs[ng - 1]) {
      gs[ng - 1] *= L.sizes[a];
    } else {
      gs[ng] = L.sizes[a];
      gt[ng] = L.strides[a];
      ++ng;
    }
  }
  if (ng == 0) {
    gs[0] = 1;
    gt[0] = 1;
    ng = 1;
  }
  ta.S_in = gs[0];
  ta.s_stride = gt[0];
  ta.n_outer = ng - 1;
  for (int i = 1; i < ng; ++i) {
    ta.outer_size[i - 1] = gs[i];
    ta.outer_stride[i - 1] = gt[i];
  }
  return ta;
}

// Make `stream` wait for `ev`. Inside a stream capture an event recorded
// outside the capture is waited on as an external event node, which is legal
// there and orders graph replays after the recorded work.
cudaError_t wait_event(cudaStream_t stream, cudaEvent_t ev) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
  return cudaStreamWaitEvent(stream, ev,
                             cs == cudaStreamCaptureStatusActive ? cudaEventWaitExternal : 0);
}

// Grows the plan's device scratch (status words, rotary table) to hold
// `table_entries` (cos, sin) pairs. Inside a call (`in_stream` true) nothing
// synchronises: the memory comes from cudaMallocAsync and is cleared by
// cudaMemsetAsync on `stream`, scratch_ready is recorded after it, and a table
// it replaces is retired (queued work on any stream may still read it). From
// fp_reserve (`in_stream` false) the growth completes before returning and
// retired tables are freed once the device is idle.
fp_status ensure_device_state(fp_plan* p, int64_t table_entries, cudaStream_t stream,
                              bool in_stream, int64_t attn_bytes = 0) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(FP_ERR_CUDA, "cudaGetDevice failed");
  if (p->d_status && p->device != dev)
    return fail(FP_ERR_INVALID_ARG, "plan was first used on device %d, now on device %d",
                p->device, dev);
  const cudaStream_t s = in_stream ? stream : nullptr;
  bool grew = false;
  if (!p->d_status) {
    void* st = nullptr;
    if (cudaMallocAsync(&st, 2 * sizeof(int), s) != cudaSuccess)
      return fail(FP_ERR_OUT_OF_MEMORY, "status word allocation failed");
    if (cudaMemsetAsync(st, 0, 2 * sizeof(int), s) != cudaSuccess) {
      cudaFreeAsync(st, s);
      return fail(FP_ERR_CUDA, "status word initialisation failed");
    }
    p->d_status = static_cast<int*>(st);
    p->device = dev;
    grew = true;
  }
  if (table_entries > p->table_cap) {
    // at least double, so that a slowly growing T retires little memory
    const int64_t cap = std::max(table_entries, 2 * p->table_cap);
    void* t = nullptr;
    if (cudaMallocAsync(&t, static_cast<size_t>(cap) * sizeof(float2), s) != cudaSuccess)
      return fail(FP_ERR_OUT_OF_MEMORY, "rotary table allocation (%lld entries) failed",
                  static_cast<long long>(cap));
    if (p->d_table) p->retired.push_back(p->d_table);
    p->d_table = static_cast<float2*>(t);
    p->table_cap = cap;
    p->table_T = -1;
    grew = true;
  }
  if (attn_bytes > p->attn_cap) {
    const int64_t cap = std::max(attn_bytes, 2 * p->attn_cap);
    void* a = nullptr;
    if (cudaMallocAsync(&a, static_cast<size_t>(cap), s) != cudaSuccess)
      return fail(FP_ERR_OUT_OF_MEMORY, "attention scratch allocation (%lld bytes) failed",
                  static_cast<long long>(cap));
    if (p->d_attn) p->retired.push_back(p->d_attn);
    p->d_attn = static_cast<float*>(a);
    p->attn_cap = cap;
    grew = true;
  }
  if (!in_stream) {
    if (cudaStreamSynchronize(nullptr) != cudaSuccess)
      return fail(FP_ERR_CUDA, "scratch allocation failed: %s",
                  cudaGetErrorString(cudaGetLastError()));
    if (!p->retired.empty()) {
      cudaDeviceSynchronize();  // nothing queued reads a retired table any more
      for (void* q : p->retired) cudaFreeAsync(q, nullptr);
      p->retired.clear();
    }
    p->scratch_pending = false;
    return FP_OK;
  }
  if (grew) {
    if (!p->scratch_ready &&
        cudaEventCreateWithFlags(&p->scratch_ready, cudaEventDisableTiming) != cudaSuccess)
      return fail(FP_ERR_CUDA, "event creation failed");
    if (cudaEventRecord(p->scratch_ready, stream) != cudaSuccess)
      return fail(FP_ERR_CUDA, "event record failed");
    p->scratch_stream = stream;
    p->scratch_pending = true;
  } else if (p->scratch_pending && stream != p->scratch_stream) {
    // scratch allocated in another stream's order: this stream waits for it
    if (wait_event(stream, p->scratch_ready) != cudaSuccess)
      return fail(FP_ERR_CUDA, "stream wait on the plan's scratch failed");
  }
  return FP_OK;
}

int rope_half_of(const fp_plan* p) {
  if (p->rope_base <= 0.0f || p->heads == 0) return 0;
  return (p->rope_n_elem > 0 ? p->rope_n_elem : p->hd) / 2;
}

int n_total(const fp_plan* p) {
  if (p->groups > 0) return p->F + (p->heads + 2 * p->groups) * p->hd;
  return p->F + 3 * p->heads * p->hd;
}

}  // namespace

namespace {

// Caller arguments of one forward call.
struct Args {
  const void* x;
  const fp_layout* xl;
  const void* W;
  const void* b;
  const int32_t* pos;
  void* out_ff;
  void* out_q;
  void* out_k;
  void* out_v;
};

// Result of the host-side checks: the token map and the kernel to run.
struct Prepared {
  fp_layout L;
  TokAxes ta;
  fp::TokenMap tk;
  int esz = 2, N = 0, rh = 0, bn_eff = 0;
  bool rope = false, tc_path = false, a_mn = false;
};

// Device scratch and launch knobs a launch uses.
struct Scratch {
  int* status;     // [2]
  float2* table;   // >= T * rh entries when rope
  int device;
  int launch_tag;  // >= 1
  uint64_t wait_limit_ns;
  int inject_stall;
  int group_m;
  int max_ctas;
  int cluster;
  int bounds_check;  // 0 off, 1 on, 2 on against half-size extents (test of the check)
  int tile_n;        // 0 automatic, 256 or 192 (tensor-core tiles without rotation)
};

// Every check of a forward call; touches no GPU.
fp_status prepare(const fp_plan& P, const Args& a, Prepared& pr) {
  const fp_plan* p = &P;
  if (!a.xl) return fail(FP_ERR_INVALID_ARG, "x_layout is NULL");
  const fp_layout L = *a.xl;
  pr.L = L;
  if (L.dtype != FP_BF16 && L.dtype != FP_F32) return fail(FP_ERR_INVALID_ARG, "unknown dtype");
  if (L.ndim < 1 || L.ndim > FP_MAX_DIMS) return fail(FP_ERR_INVALID_ARG, "ndim out of range");
  if (L.channel_dim < 0 || L.channel_dim >= L.ndim)
    return fail(FP_ERR_INVALID_ARG, "channel_dim out of range");
  if (L.n_batch_dims < 0 || L.n_batch_dims > L.ndim - 1)
    return fail(FP_ERR_INVALID_ARG, "n_batch_dims out of range");
  for (int d = 0; d < L.ndim; ++d)
    if (L.sizes[d] < 0 || L.strides[d] < 0)
      return fail(FP_ERR_INVALID_ARG, "negative size or stride on axis %d", d);
  if (L.sizes[L.channel_dim] != p->C)
    return fail(FP_ERR_INVALID_ARG, "x has %lld channels, plan has C = %d",
                static_cast<long long>(L.sizes[L.channel_dim]), p->C);
  const int esz = L.dtype == FP_BF16 ? 2 : 4;
  const int N = n_total(p);
  const int nkv = p->groups > 0 ? p->groups : p->heads;
  pr.esz = esz;
  pr.N = N;
  pr.ta = analyse_tokens(L);
  const TokAxes& ta = pr.ta;
  if (ta.M == 0) return FP_OK;
  if (!a.x || !a.W) return fail(FP_ERR_INVALID_ARG, "x and W must be non-NULL");
  if ((p->F > 0) != (a.out_ff != nullptr))
    return fail(FP_ERR_INVALID_ARG, "out_ff must be non-NULL exactly when ff_hidden > 0");
  const bool want_qkv = p->heads > 0;
  if (want_qkv != (a.out_q != nullptr) || want_qkv != (a.out_k != nullptr) ||
      want_qkv != (a.out_v != nullptr))
    return fail(FP_ERR_INVALID_ARG, "out_q/out_k/out_v must be non-NULL exactly when heads > 0");
  const void* ptrs[] = {a.x, a.W, a.b, a.pos, a.out_ff, a.out_q, a.out_k, a.out_v};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(FP_ERR_MISALIGNED, "every pointer must be 16-byte aligned");
  // aliasing: outputs against each other and against every input
  int64_t x_span = 1;
  for (int d = 0; d < L.ndim; ++d) x_span += (L.sizes[d] - 1) * L.strides[d];
  auto rng = [](const void* q, int64_t bytes) {
    uintptr_t lo = reinterpret_cast<uintptr_t>(q);
    return Range{lo, q ? lo + static_cast<uintptr_t>(bytes) : lo};
  };
  const Range ins[] = {rng(a.x, x_span * esz), rng(a.W, static_cast<int64_t>(p->C) * N * esz),
                       rng(a.b, static_cast<int64_t>(N) * esz),
                       rng(a.pos, static_cast<int64_t>(ta.T) * 4)};
  const Range outs[] = {rng(a.out_ff, ta.M * p->F * esz),
                        rng(a.out_q, ta.M * p->heads * p->hd * esz),
                        rng(a.out_k, ta.M * nkv * p->hd * esz),
                        rng(a.out_v, ta.M * nkv * p->hd * esz)};
  for (int i = 0; i < 4; ++i) {
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i], outs[j])) return fail(FP_ERR_INVALID_ARG, "output buffers overlap");
    for (const Range& in : ins)
      if (overlaps(outs[i], in)) return fail(FP_ERR_INVALID_ARG, "an output overlaps an input");
  }
  const int rh = rope_half_of(p);
  const bool rope = rh > 0;
  pr.rh = rh;
  pr.rope = rope;
  fp::TokenMap& tk = pr.tk;
  tk = fp::TokenMap{};
  tk.S_in = ta.S_in;
  tk.s_stride = ta.s_stride;
  tk.c_stride = p->C == 1 ? 1 : L.strides[L.channel_dim];
  tk.n_outer = 1;
  tk.n_outer_dims = ta.n_outer;
  if (tk.n_outer_dims > fp::kMaxOuter)
    return fail(FP_ERR_UNSUPPORTED_LAYOUT, "x has more than %d non-mergeable token axes",
                fp::kMaxOuter);
  for (int i = 0; i < tk.n_outer_dims; ++i) {
    tk.outer_size[i] = ta.outer_size[i];
    tk.outer_stride[i] = ta.outer_stride[i];
    tk.n_outer *= ta.outer_size[i];
  }
  // bf16 runs on the tensor-core kernel when its TMA maps and 16-column
  // epilogue granules can describe the problem; otherwise (and for f32) on the
  // FFMA kernel, which addresses any strides.
  bool a_mn = false;
  bool tc_path = L.dtype == FP_BF16;
  if (tc_path) {
    if (p->F % 16 || (p->heads > 0 && p->hd % 16)) tc_path = false;
    if (rope && rh % 16 && rh > 8) tc_path = false;
    if (tk.n_outer_dims > 3) tc_path = false;
    if (tk.c_stride == 1) a_mn = false;
    else if (tk.s_stride == 1 || tk.S_in == 1) a_mn = true;
    else tc_path = false;
    const int64_t other = a_mn ? tk.c_stride : tk.s_stride;
    const bool other_unused = a_mn ? p->C == 1 : tk.S_in == 1;
    if (!other_unused && (other * esz) % 16) tc_path = false;
    for (int i = 0; i < tk.n_outer_dims; ++i)
      if ((tk.outer_stride[i] * esz) % 16) tc_path = false;
  }
  pr.tc_path = tc_path;
  pr.a_mn = a_mn;
  if (tc_path)
    pr.bn_eff = rope ? (fp::kTcBN / p->hd) * p->hd : fp::kTcBN;
  else
    pr.bn_eff = rope ? (fp::kSimtBN / p->hd) * p->hd : fp::kSimtBN;
  return FP_OK;
}

// Caller-given rotary tables [T, n_rot] (cos and sin, any strides).
struct ExtTable {
  const void* cosv;
  const void* sinv;
  bool bf16;
  int64_t stride_t, stride_i;
};

// Enqueue the rotary table (when build_table, or the import of caller tables
// when ext is given) and the GEMM kernel on `stream`. Uses only the scratch it
// is given; allocates nothing.
fp_status launch(const fp_plan& P, const Prepared& pr, const Args& a, const Scratch& sc,
                 bool build_table, cudaStream_t stream, int* launches,
                 const ExtTable* ext = nullptr) {
  const fp_plan* p = &P;
  const TokAxes& ta = pr.ta;
  const fp::TokenMap& tk = pr.tk;
  const int N = pr.N, esz = pr.esz, rh = pr.rh, bn_eff = pr.bn_eff;
  *launches = 0;
  if (ext) {
    cudaError_t err = fp::launch_rope_import(reinterpret_cast<float4*>(sc.table), ext->cosv,
                                             ext->sinv, ext->bf16, ta.T, rh, ext->stride_t,
                                             ext->stride_i, stream);
    if (err != cudaSuccess)
      return fail(FP_ERR_CUDA, "rotary table import launch: %s", cudaGetErrorString(err));
    ++*launches;
  } else if (build_table) {
    cudaError_t err = fp::launch_rope_table(sc.table, a.pos, ta.T, rh, 2 * rh,
                                            static_cast<double>(p->rope_base), stream);
    if (err != cudaSuccess)
      return fail(FP_ERR_CUDA, "rotary table launch: %s", cudaGetErrorString(err));
    ++*launches;
  }
  fp::Epilogue e{};
  e.M = ta.M;
  e.T = ta.T;
  e.N = N;
  e.F = p->F;
  e.C = p->C;
  e.heads = p->heads;
  e.hd = p->hd;
  e.groups = p->groups;
  e.act = p->act;
  e.rope_half = rh;
  e.rope_cs = pr.rope && !ext ? sc.table : nullptr;
  e.rope_cs4 = ext ? reinterpret_cast<const float4*>(sc.table) : nullptr;
  e.rope_per_lane = ext ? 1 : 0;
  e.bias = a.b;
  e.out_ff = a.out_ff;
  e.out_q = a.out_q;
  e.out_k = a.out_k;
  e.out_v = a.out_v;
  e.status = sc.status;
  e.bn_eff = bn_eff;
  e.k_transposed = p->k_transposed;
  e.ff_ld = p->F;
  e.bounds_check = sc.bounds_check ? 1 : 0;
  {
    const int nkv = p->groups > 0 ? p->groups : p->heads;
    const int64_t ext[4] = {ta.M * p->F, ta.M * p->heads * p->hd, ta.M * nkv * p->hd,
                            ta.M * nkv * p->hd};
    for (int i = 0; i < 4; ++i) e.extent[i] = sc.bounds_check == 2 ? ext[i] / 2 : ext[i];
  }
  const int num_n_tiles = (N + bn_eff - 1) / bn_eff;

  if (pr.tc_path) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
    if (!encode) return fail(FP_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    fp::TcParams tp;
    memset(&tp, 0, sizeof tp);
    // A: 5-D map [inner, second, outer0, outer1, outer2]
    cuuint64_t gdim[5], gstride[4];
    cuuint32_t box[5], estr[5] = {1, 1, 1, 1, 1};
    if (pr.a_mn) {
      gdim[0] = ta.S_in;
      gdim[1] = p->C;
      gstride[0] = static_cast<cuuint64_t>(tk.c_stride) * esz;
      box[0] = 64;
      box[1] = fp::kTcBK;
    } else {
      gdim[0] = p->C;
      gdim[1] = ta.S_in;
      gstride[0] = static_cast<cuuint64_t>(tk.s_stride) * esz;
      box[0] = fp::kTcBK;
      box[1] = fp::kTcBM;
    }
    // a unit-extent second axis may carry any stride: give TMA a valid one
    if (gstride[0] == 0 || gstride[0] % 16) gstride[0] = 16 * ((gdim[0] * esz + 15) / 16);
    cuuint64_t last = gstride[0];
    for (int d = 0; d < 3; ++d) {
      if (d < tk.n_outer_dims) {
        gdim[2 + d] = tk.outer_size[d];
        gstride[1 + d] = static_cast<cuuint64_t>(tk.outer_stride[d]) * esz;
        last = gstride[1 + d];
      } else {
        gdim[2 + d] = 1;
        gstride[1 + d] = last;
      }
      box[2 + d] = 1;
    }
    if (pr.a_mn && ta.S_in % 64 == 0 && tk.n_outer_dims <= 2) {
      // unit token stride, whole 64-token blocks: tokens become (64 inside a
      // block, S_in/64 blocks), and one [2 blocks][64 ch][64 tok] box is a stage
      // (the same shared-memory image as two [64 ch][64 tok] boxes; one TMA
      // instruction instead of two measured 3 % faster on the Walrus shape)
      gdim[0] = 64;
      gdim[1] = p->C;
      gdim[2] = ta.S_in / 64;
      gstride[0] = static_cast<cuuint64_t>(tk.c_stride) * esz;
      gstride[1] = 64ull * esz;
      cuuint64_t prev = gstride[1];
      for (int d = 0; d < 2; ++d) {
        if (d < tk.n_outer_dims) {
          gdim[3 + d] = tk.outer_size[d];
          gstride[2 + d] = static_cast<cuuint64_t>(tk.outer_stride[d]) * esz;
          prev = gstride[2 + d];
        } else {
          gdim[3 + d] = 1;
          gstride[2 + d] = prev;
        }
      }
      if (gstride[0] == 0 || gstride[0] % 16) gstride[0] = 16 * ((64 * esz + 15) / 16);
      box[0] = 64;
      box[1] = fp::kTcBK;
      box[2] = 2;
      box[3] = box[4] = 1;
      tp.a_split = 1;
    }
    CUresult r = encode(&tp.tmap_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(a.x),
                        gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(FP_ERR_UNSUPPORTED_LAYOUT, "tensor map for x rejected (CUresult %d)",
                  static_cast<int>(r));
    cuuint64_t bdim[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(p->C)};
    cuuint64_t bstride[1] = {static_cast<cuuint64_t>(N) * esz};
    cuuint32_t bbox[2] = {64, fp::kTcBK};
    r = encode(&tp.tmap_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W), bdim,
               bstride, bbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(FP_ERR_UNSUPPORTED_LAYOUT, "tensor map for W rejected (CUresult %d)",
                  static_cast<int>(r));
    if (a.b) {
      // bias: one row of N, loaded 64 columns at a time into the bias operand
      cuuint64_t d[2] = {static_cast<cuuint64_t>(N), 1};
      cuuint64_t st[1] = {static_cast<cuuint64_t>(N) * esz};
      cuuint32_t bx[2] = {64, 1};
      r = encode(&tp.tmap_bias, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.b), d, st,
                 bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS)
        return fail(FP_ERR_UNSUPPORTED_LAYOUT, "tensor map for the bias rejected (CUresult %d)",
                    static_cast<int>(r));
    }
    // output maps: when they encode, the epilogue writes whole 32-row blocks by
    // TMA from 32-byte-swizzled staging rows (the 16-byte halves of rows 4-7 of
    // every 8 swapped, so the staging stores are free of bank conflicts)
    {
      const cuuint32_t ostr[3] = {1, 1, 1};
      bool okm = true;
      if (a.out_ff) {
        cuuint64_t d[2] = {static_cast<cuuint64_t>(p->F), static_cast<cuuint64_t>(ta.M)};
        cuuint64_t st[1] = {static_cast<cuuint64_t>(p->F) * esz};
        cuuint32_t bx[2] = {16, 32};
        okm = okm && encode(&tp.tmap_ff, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out_ff, d, st, bx,
                            ostr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        cuuint32_t bx32[2] = {32, 32};  // 64-byte rows, 64-byte swizzle
        okm = okm && encode(&tp.tmap_ff32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out_ff, d, st,
                            bx32, ostr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
      }
      const int nkv = p->groups > 0 ? p->groups : p->heads;
      void* const outs3[3] = {a.out_q, a.out_k, a.out_v};
      CUtensorMap* const maps3[3] = {&tp.tmap_q, &tp.tmap_k, &tp.tmap_v};
      for (int i = 0; i < 3 && p->heads > 0; ++i) {
        if (i == 1 && p->k_transposed) continue;  // pre-transposed k is stored directly
        const int nh = i == 0 ? p->heads : nkv;
        cuuint64_t d[3] = {static_cast<cuuint64_t>(p->hd), static_cast<cuuint64_t>(ta.T),
                           static_cast<cuuint64_t>(ta.Bb * nh)};
        cuuint64_t st[2] = {static_cast<cuuint64_t>(p->hd) * esz,
                            static_cast<cuuint64_t>(ta.T * p->hd) * esz};
        cuuint32_t bx[3] = {16, 32, 1};
        okm = okm && encode(maps3[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, outs3[i], d, st, bx,
                            ostr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
      }
      tp.tma_store = okm && ta.M <= INT32_MAX ? 1 : 0;  // TMA coordinates are 32-bit
    }
    tp.tok = tk;
    tp.epi = e;
    tp.C = p->C;
    tp.num_k_blocks = (p->C + fp::kTcBK - 1) / fp::kTcBK;
    tp.m_tiles_per_slab = (ta.S_in + fp::kTcBM - 1) / fp::kTcBM;
    tp.num_m_tiles = tk.n_outer * tp.m_tiles_per_slab;
    tp.num_n_tiles = num_n_tiles;
    tp.num_tiles = tp.num_m_tiles * num_n_tiles;
    // two CTAs share each W tile when there are M-tiles to pair
    tp.cluster = (sc.cluster == 2 && tp.num_m_tiles >= 2) ? 2 : 1;
    tp.num_units = (tp.num_m_tiles + tp.cluster - 1) / tp.cluster * num_n_tiles;
    tp.bn_mma = fp::kTcBN;
    if (!pr.rope && tp.cluster == 2) {
      // 192-column tiles only where 256-column tiles would compute at least
      // 15 % more columns than N (N = 384: 512 against 384). Measured on the
      // wave-quantised shapes instead (BERT ff, N = 3072 on 384 units of 256),
      // 192 was 5-40 % slower: the operand traffic per FLOP grows by a third
      // and the kernel runs at the rate the loads arrive, not at the wave fill.
      const int64_t m_units = (tp.num_m_tiles + 1) / 2;
      const int64_t c256 = (N + 255) / 256 * 256, c192 = (N + 191) / 192 * 192;
      const bool use192 = sc.tile_n == 192 || (sc.tile_n == 0 && c192 * 100 <= c256 * 85);
      if (use192) {
        tp.bn_mma = 192;
        tp.epi.bn_eff = 192;
        tp.num_n_tiles = (N + 191) / 192;
        tp.num_tiles = tp.num_m_tiles * tp.num_n_tiles;
        tp.num_units = m_units * tp.num_n_tiles;
      }
    }
    if (tp.num_units * tp.cluster > INT32_MAX)
      return fail(FP_ERR_UNSUPPORTED_LAYOUT, "more than 2^31 output tiles");
    tp.group_m = sc.group_m;
    tp.wait_limit_ns = sc.wait_limit_ns;
    tp.inject_stall = sc.inject_stall;
    tp.launch_tag = sc.launch_tag;
    int ctas = sm_count(sc.device);
    if (sc.max_ctas > 0) ctas = std::min(ctas, sc.max_ctas);
    if (static_cast<int64_t>(ctas) > tp.num_units * tp.cluster)
      ctas = static_cast<int>(tp.num_units * tp.cluster);
    cudaError_t err = fp::launch_tc_gemm(tp, pr.a_mn, ctas, stream);
    if (err != cudaSuccess)
      return fail(FP_ERR_CUDA, "tensor-core GEMM launch: %s", cudaGetErrorString(err));
  } else {
    fp::SimtParams sp;
    memset(&sp, 0, sizeof sp);
    sp.x = a.x;
    sp.W = a.W;
    sp.tok = tk;
    sp.epi = e;
    sp.C = p->C;
    sp.m_tiles_per_slab = (ta.S_in + fp::kSimtBM - 1) / fp::kSimtBM;
    sp.num_m_tiles = tk.n_outer * sp.m_tiles_per_slab;
    sp.num_n_tiles = num_n_tiles;
    cudaError_t err = fp::launch_simt_gemm(sp, pr.L.dtype == FP_BF16, stream);
    if (err != cudaSuccess)
      return fail(FP_ERR_CUDA, "FFMA GEMM launch: %s", cudaGetErrorString(err));
  }
  ++*launches;
  return FP_OK;
}

// Device address of the no-allocation entry point's static scratch (defined
// with that entry point at the end of this file).
fp_status noalloc_scratch(int dev, unsigned char** out);

}  // namespace

extern "C" {

const char* fp_status_string(fp_status s) {
  switch (s) {
    case FP_OK: return "ok";
    case FP_ERR_INVALID_ARG: return "invalid argument";
    case FP_ERR_UNSUPPORTED_LAYOUT: return "unsupported activation layout";
    case FP_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case FP_ERR_CUDA: return "CUDA call failed";
    case FP_ERR_OUT_OF_MEMORY: return "device allocation failed";
    case FP_ERR_TIMEOUT: return "device-side wait ran out";
    case FP_ERR_DEVICE_BOUNDS: return "device-side bounds check failed";
  }
  return "unknown status";
}

const char* fp_last_error(void) { return g_err; }

fp_status fp_create_ex(fp_plan** plan, const fp_config* cfg) {
  if (!plan) return fail(FP_ERR_INVALID_ARG, "plan is NULL");
  *plan = nullptr;
  if (!cfg) return fail(FP_ERR_INVALID_ARG, "config is NULL");
  const int C = cfg->C, F = cfg->ff_hidden, heads = cfg->heads, hd = cfg->head_dim;
  const int G = cfg->n_query_groups, ne = cfg->rope_n_elem;
  if (C <= 0) return fail(FP_ERR_INVALID_ARG, "C must be > 0 (got %d)", C);
  if (F < 0) return fail(FP_ERR_INVALID_ARG, "ff_hidden must be >= 0");
  if (heads < 0) return fail(FP_ERR_INVALID_ARG, "heads must be >= 0");
  if (G < 0) return fail(FP_ERR_INVALID_ARG, "n_query_groups must be >= 0");
  if (heads > 0) {
    if (hd <= 0 || hd % 2)
      return fail(FP_ERR_INVALID_ARG, "head_dim must be even and > 0 (got %d)", hd);
    if (static_cast<int64_t>(heads) * hd != C)
      return fail(FP_ERR_INVALID_ARG, "heads * head_dim (%d * %d) must equal C (%d)", heads,
                  hd, C);
    if (F % hd)
      return fail(FP_ERR_INVALID_ARG, "ff_hidden (%d) must be a multiple of head_dim (%d)", F,
                  hd);
    if (G > 0 && heads % G)
      return fail(FP_ERR_INVALID_ARG, "heads (%d) must be a multiple of n_query_groups (%d)",
                  heads, G);
    if (ne < 0 || ne % 2 || ne > hd)
      return fail(FP_ERR_INVALID_ARG, "rope_n_elem must be even and <= head_dim (got %d)", ne);
  } else if (G > 0) {
    return fail(FP_ERR_INVALID_ARG, "n_query_groups needs heads > 0");
  }
  if (F == 0 && heads == 0) return fail(FP_ERR_INVALID_ARG, "nothing to compute");
  if (cfg->act < FP_ACT_NONE || cfg->act > FP_ACT_RELU2)
    return fail(FP_ERR_INVALID_ARG, "unknown act");
  if (cfg->rope_base > 0.0f && heads > 0 && hd > 128)
    return fail(FP_ERR_INVALID_ARG, "rotary embedding needs head_dim <= 128 (got %d)", hd);
  fp_plan* p = new (std::nothrow) fp_plan();
  if (!p) return fail(FP_ERR_OUT_OF_MEMORY, "host allocation failed");
  p->C = C;
  p->F = F;
  p->heads = heads;
  p->hd = heads > 0 ? hd : 0;
  p->groups = heads > 0 ? G : 0;
  p->rope_n_elem = heads > 0 ? ne : 0;
  p->k_transposed = heads > 0 && cfg->k_transposed ? 1 : 0;
  p->act = cfg->act;
  p->rope_base = cfg->rope_base;
  p->device = -1;
  p->d_status = nullptr;
  p->d_table = nullptr;
  p->d_attn = nullptr;
  p->attn_cap = 0;
  p->table_cap = 0;
  p->table_T = -1;
  p->table_stream = nullptr;
  p->table_ready = nullptr;
  p->side_stream = nullptr;
  p->ev_fork = nullptr;
  p->ev_join = nullptr;
  p->last_launches = 0;
  p->wait_limit_ns = kDefaultWaitLimitNs;
  p->inject_stall = 0;
  p->group_m = kDefaultGroupM;
  p->max_ctas = 0;
  p->cluster = kDefaultCluster;
  p->bounds_check = 0;
  p->tile_n = 0;
  p->launch_seq = 0;
  p->scratch_stream = nullptr;
  p->scratch_ready = nullptr;
  p->scratch_pending = false;
  *plan = p;
  return ok();
}

fp_status fp_create(fp_plan** plan, int C, int ff_hidden, int heads, int head_dim, fp_act act,
                    float rope_base) {
  fp_config cfg{C, ff_hidden, heads, head_dim, 0, 0, static_cast<int32_t>(act), rope_base, 0};
  return fp_create_ex(plan, &cfg);
}

void fp_destroy(fp_plan* plan) {
  if (!plan) return;
  if (plan->d_status || plan->d_table || plan->d_attn || plan->d_host_stage || plan->up_stream) {
    int prev = -1;
    cudaGetDevice(&prev);
    if (plan->device >= 0) cudaSetDevice(plan->device);
    // queued work may still use the scratch: free it once the device is idle
    cudaDeviceSynchronize();
    if (plan->d_status) cudaFreeAsync(plan->d_status, nullptr);
    if (plan->d_table) cudaFreeAsync(plan->d_table, nullptr);
    if (plan->d_attn) cudaFreeAsync(plan->d_attn, nullptr);
    if (plan->d_host_stage) cudaFreeAsync(plan->d_host_stage, nullptr);
    for (void* q : plan->retired) cudaFreeAsync(q, nullptr);
    cudaStreamSynchronize(nullptr);
    for (cudaEvent_t e : {plan->ev_host_fork, plan->ev_up[0], plan->ev_up[1], plan->ev_comp[0],
                          plan->ev_comp[1], plan->ev_down[0], plan->ev_down[1]})
      if (e) cudaEventDestroy(e);
    if (plan->up_stream) cudaStreamDestroy(plan->up_stream);
    if (plan->down_stream) cudaStreamDestroy(plan->down_stream);
    if (plan->table_ready) cudaEventDestroy(plan->table_ready);
    if (plan->scratch_ready) cudaEventDestroy(plan->scratch_ready);
    if (plan->ev_fork) cudaEventDestroy(plan->ev_fork);
    if (plan->ev_join) cudaEventDestroy(plan->ev_join);
    if (plan->side_stream) cudaStreamDestroy(plan->side_stream);
    if (prev >= 0) cudaSetDevice(prev);
  }
  delete plan;
}

int fp_last_launch_count(const fp_plan* plan) { return plan ? plan->last_launches : 0; }

fp_status fp_set_option(fp_plan* plan, fp_option opt, int64_t value) {
  if (!plan) return fail(FP_ERR_INVALID_ARG, "plan is NULL");
  switch (opt) {
    case FP_OPT_WAIT_LIMIT_NS:
      if (value <= 0) return fail(FP_ERR_INVALID_ARG, "wait limit must be > 0");
      plan->wait_limit_ns = static_cast<uint64_t>(value);
      return ok();
    case FP_OPT_INJECT_STALL:
      plan->inject_stall = value ? 1 : 0;
      return ok();
    case FP_OPT_GROUP_M:
      if (value < 1 || value > 4096) return fail(FP_ERR_INVALID_ARG, "group_m out of range");
      plan->group_m = static_cast<int>(value);
      return ok();
    case FP_OPT_MAX_CTAS:
      if (value < 0) return fail(FP_ERR_INVALID_ARG, "max_ctas must be >= 0");
      plan->max_ctas = static_cast<int>(value);
      return ok();
    case FP_OPT_CLUSTER:
      if (value != 1 && value != 2) return fail(FP_ERR_INVALID_ARG, "cluster must be 1 or 2");
      plan->cluster = static_cast<int>(value);
      return ok();
    case FP_OPT_TILE_N:
      if (value != 0 && value != 256 && value != 192)
        return fail(FP_ERR_INVALID_ARG, "tile width must be 0, 256 or 192");
      plan->tile_n = static_cast<int>(value);
      return ok();
    case FP_OPT_BOUNDS_CHECK:
      if (value < 0 || value > 2) return fail(FP_ERR_INVALID_ARG, "bounds check must be 0, 1 or 2");
      plan->bounds_check = static_cast<int>(value);
      return ok();
  }
  return fail(FP_ERR_INVALID_ARG, "unknown option %d", static_cast<int>(opt));
}

fp_status fp_reserve(fp_plan* plan, int64_t max_tokens_per_batch) {
  if (!plan) return fail(FP_ERR_INVALID_ARG, "plan is NULL");
  if (max_tokens_per_batch < 0) return fail(FP_ERR_INVALID_ARG, "negative size");
  fp_status st = ensure_device_state(plan, max_tokens_per_batch * rope_half_of(plan), nullptr,
                                     false);
  return st == FP_OK ? ok() : st;
}

fp_status fp_get_device_status(fp_plan* plan, void* stream) {
  int* words = plan ? plan->d_status : nullptr;
  if (!plan) {
    // the no-allocation entry point's status words, on the current device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(FP_ERR_CUDA, "cudaGetDevice failed");
    unsigned char* base = nullptr;
    const fp_status st = noalloc_scratch(dev, &base);
    if (st != FP_OK) return st;
    words = reinterpret_cast<int*>(base);
  }
  if (!words) return ok();
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return fail(FP_ERR_CUDA, "stream synchronisation failed: %s",
                cudaGetErrorString(cudaGetLastError()));
  int h[2] = {0, 0};
  if (cudaMemcpy(h, words, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail(FP_ERR_CUDA, "status read failed");
  if (h[0] != 0) {
    int zero[2] = {0, 0};
    cudaMemcpy(words, zero, sizeof zero, cudaMemcpyHostToDevice);
    return fail(static_cast<fp_status>(h[0]), "device reported: %s",
                fp_status_string(static_cast<fp_status>(h[0])));
  }
  return ok();
}

fp_status fp_forward(fp_plan* p, const void* x, const fp_layout* xl, const void* W, const void* b,
                     const int32_t* pos, void* out_ff, void* out_q, void* out_k, void* out_v,
                     void* stream_v) {
  const NvtxRange range("fp_forward");
  if (!p) return fail(FP_ERR_INVALID_ARG, "plan is NULL");
  const Args a{x, xl, W, b, pos, out_ff, out_q, out_k, out_v};
  Prepared pr;
  fp_status st = prepare(*p, a, pr);
  if (st != FP_OK) return st;
  if (pr.ta.M == 0) {
    p->last_launches = 0;
    return ok();  // no tokens: nothing to do
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  st = ensure_device_state(p, pr.rope ? pr.ta.T * pr.rh : 0, stream, true);
  if (st != FP_OK) return st;
  // The table depends only on (positions, base, rotated width). With the
  // default positions 0..T-1 it is a constant of the plan and of T, so it is
  // built once and reused; caller-given positions rebuild it on every call.
  const bool build_table = pr.rope && (pos != nullptr || p->table_T != pr.ta.T);
  if (pr.rope && !build_table && stream != p->table_stream) {
    // cached table written on another stream: order this call after that write
    if (wait_event(stream, p->table_ready) != cudaSuccess)
      return fail(FP_ERR_CUDA, "stream wait on the rotary table failed");
  }
  p->launch_seq = p->launch_seq % 0x7FFFFFFEu + 1u;
  const Scratch sc{p->d_status, p->d_table, p->device, static_cast<int>(p->launch_seq),
                   p->wait_limit_ns, p->inject_stall, p->group_m, p->max_ctas, p->cluster,
                   p->bounds_check, p->tile_n};
  int launches = 0;
  st = launch(*p, pr, a, sc, build_table, stream, &launches);
  if (st != FP_OK) return st;
  p->inject_stall = 0;
  if (build_table) {
    if (!p->table_ready &&
        cudaEventCreateWithFlags(&p->table_ready, cudaEventDisableTiming) != cudaSuccess)
      return fail(FP_ERR_CUDA, "event creation failed");
    if (cudaEventRecord(p->table_ready, stream) != cudaSuccess)
      return fail(FP_ERR_CUDA, "event record failed");
    p->table_stream = stream;
    p->table_T = pos ? -1 : pr.ta.T;
  }
  p->last_launches = launches;
  return ok();
}

namespace {

// A host pointer the copy engines can reach asynchronously: page-locked host
// memory (cudaHostAlloc or cudaHostRegister).
bool page_locked(const void* q) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
    cudaGetLastError();  // an unregistered pointer is an answer, not an error
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

constexpr int kHostChunks = 4;
constexpr int64_t kStageAlign = 256;

int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// How a host entry point splits x: along axis 0 when x is dense (row-major
// strides over its sizes) and axis 0 is a batch axis, in up to kHostChunks
// chunks of `per_chunk` units; else one chunk of one unit (the whole call).
struct HostChunks {
  bool dense, chunked;
  int64_t numel, span, per_chunk;
  int n_chunks;
};

HostChunks host_chunks(const fp_layout& L) {
  HostChunks h{};
  h.dense = true;
  h.numel = 1;
  for (int d = L.ndim - 1; d >= 0; --d) {
    if (L.sizes[d] > 1 && L.strides[d] != h.numel) h.dense = false;
    h.numel *= L.sizes[d];
  }
  h.chunked = h.dense && L.channel_dim != 0 && L.n_batch_dims >= 1 && L.sizes[0] > 1;
  h.span = h.chunked ? L.sizes[0] : 1;
  h.per_chunk = (h.span + kHostChunks - 1) / kHostChunks;
  h.n_chunks = static_cast<int>((h.span + h.per_chunk - 1) / h.per_chunk);
  return h;
}

// The host entry points' copy streams and events (created on first use) and
// device staging of at least `bytes` (grown in `stream` order; a replaced
// buffer may still be read by queued copies, so it is retired).
fp_status host_pipeline_setup(fp_plan* p, int64_t bytes, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(FP_ERR_CUDA, "cudaGetDevice failed");
  if (p->d_status && p->device != dev)
    return fail(FP_ERR_INVALID_ARG, "plan was first used on device %d, now on device %d",
                p->device, dev);
  if (!p->up_stream) {
    if (cudaStreamCreateWithFlags(&p->up_stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p->down_stream, cudaStreamNonBlocking) != cudaSuccess)
      return fail(FP_ERR_CUDA, "copy stream creation failed");
    for (cudaEvent_t* e : {&p->ev_host_fork, &p->ev_up[0], &p->ev_up[1], &p->ev_comp[0],
                           &p->ev_comp[1], &p->ev_down[0], &p->ev_down[1]})
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess)
        return fail(FP_ERR_CUDA, "event creation failed");
  }
  if (bytes > p->host_stage_cap) {
    void* q = nullptr;
    if (cudaMallocAsync(&q, static_cast<size_t>(bytes), stream) != cudaSuccess)
      return fail(FP_ERR_OUT_OF_MEMORY, "host-call staging allocation (%lld bytes) failed",
                  static_cast<long long>(bytes));
    if (p->d_host_stage) p->retired.push_back(p->d_host_stage);
    p->d_host_stage = q;
    p->host_stage_cap = bytes;
  }
  return FP_OK;
}

// Host calls on one plan run one after another, whichever streams they are
// on: the call starts after the previous call's last download (which follows
// all of that call's uploads and compute), and both copy streams start after
// `stream`'s work so far.
fp_status host_pipeline_fork(fp_plan* p, cudaStream_t stream) {
  if (wait_event(stream, p->ev_down[p->host_last]) != cudaSuccess)
    return fail(FP_ERR_CUDA, "stream wait on the previous host call failed");
  if (cudaEventRecord(p->ev_host_fork, stream) != cudaSuccess ||
      cudaStreamWaitEvent(p->up_stream, p->ev_host_fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->down_stream, p->ev_host_fork, 0) != cudaSuccess)
    return fail(FP_ERR_CUDA, "forking the copy streams failed");
  return FP_OK;
}

// `stream` waits for the last download; the download stream runs in order,
// so its last event covers every chunk.
fp_status host_pipeline_join(fp_plan* p, int n_chunks, cudaStream_t stream) {
  p->host_last = (n_chunks - 1) & 1;
  if (cudaStreamWaitEvent(stream, p->ev_down[p->host_last], 0) != cudaSuccess)
    return fail(FP_ERR_CUDA, "joining the download stream failed");
  return FP_OK;
}

}  // namespace

fp_status fp_forward_host(fp_plan* p, const void* x_host, const fp_layout* xl, const void* W,
                          const void* b, const int32_t* pos, void* ff_h, void* q_h, void* k_h,
                          void* v_h, void* stream_v) {
  const NvtxRange range("fp_forward_host");
  if (!p) return fail(FP_ERR_INVALID_ARG, "plan is NULL");
  if (!xl) return fail(FP_ERR_INVALID_ARG, "x_layout is NULL");
  // shapes, strides and outputs exactly as fp_forward sees them
  {
    const Args full{x_host, xl, W, b, pos, ff_h, q_h, k_h, v_h};
    Prepared pr;
    const fp_status st = prepare(*p, full, pr);
    if (st != FP_OK) return st;
    if (pr.ta.M == 0) {
      p->last_launches = 0;
      return ok();
    }
  }
  void* const outs_h[4] = {ff_h, q_h, k_h, v_h};
  if (!page_locked(x_host)) return fail(FP_ERR_INVALID_ARG, "x_host is not page-locked host memory");
  for (void* q : outs_h)
    if (q && !page_locked(q))
      return fail(FP_ERR_INVALID_ARG, "output buffers must be page-locked host memory");
  const fp_layout L = *xl;
  const int64_t esz = L.dtype == FP_BF16 ? 2 : 4;
  const TokAxes ta = analyse_tokens(L);
  const HostChunks hc = host_chunks(L);
  const bool chunked = hc.chunked;
  const int64_t span = hc.span, per_chunk = hc.per_chunk, numel = hc.numel;
  const int n_chunks = hc.n_chunks;
  // elements of x and of each output per unit of axis 0 (the whole call when not chunked)
  const int nkv = p->groups > 0 ? p->groups : p->heads;
  const int64_t m_unit = ta.M / span;
  int64_t x_unit = 0;
  if (chunked) {
    x_unit = numel / span;
  } else {
    x_unit = 1;  // span of the strided x, in elements
    for (int d = 0; d < L.ndim; ++d) x_unit += (L.sizes[d] - 1) * L.strides[d];
  }
  const int64_t out_unit[4] = {m_unit * p->F, m_unit * p->heads * p->hd, m_unit * nkv * p->hd,
                               m_unit * nkv * p->hd};
  // one staging slot: x, then ff, q, k, v, each 256-byte aligned
  int64_t off[5], slot = 0;
  off[0] = 0;
  slot = align_up(per_chunk * x_unit * esz, kStageAlign);
  for (int i = 0; i < 4; ++i) {
    off[i + 1] = slot;
    slot += outs_h[i] ? align_up(per_chunk * out_unit[i] * esz, kStageAlign) : 0;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  fp_status st0 = host_pipeline_setup(p, 2 * slot, stream);
  if (st0 != FP_OK) return st0;
  unsigned char* const stage = static_cast<unsigned char*>(p->d_host_stage);
  auto chunk_layout = [&](int64_t units) {
    fp_layout c = L;
    if (chunked) c.sizes[0] = units;
    return c;
  };
  auto dev_out = [&](int s, int i) -> void* {
    return outs_h[i] ? stage + s * slot + off[i + 1] : nullptr;
  };
  // every fp_forward check, on the first chunk's staging pointers, before any copy
  {
    const fp_layout c0 = chunk_layout(std::min<int64_t>(per_chunk, span));
    const Args a0{stage, &c0, W, b, pos, dev_out(0, 0), dev_out(0, 1), dev_out(0, 2),
                  dev_out(0, 3)};
    Prepared pr;
    const fp_status st = prepare(*p, a0, pr);
    if (st != FP_OK) return st;
  }
  st0 = host_pipeline_fork(p, stream);
  if (st0 != FP_OK) return st0;
  const unsigned char* const xh = static_cast<const unsigned char*>(x_host);
  int launches = 0;
  for (int c = 0; c < n_chunks; ++c) {
    const int s = c & 1;
    const int64_t u0 = c * per_chunk, units = std::min(per_chunk, span - u0);
    // upload: slot s's x is free once chunk c - 2 has been computed
    if (c >= 2 && cudaStreamWaitEvent(p->up_stream, p->ev_comp[s], 0) != cudaSuccess)
      return fail(FP_ERR_CUDA, "upload stream wait failed");
    if (cudaMemcpyAsync(stage + s * slot, xh + u0 * x_unit * esz,
                        static_cast<size_t>(units * x_unit * esz), cudaMemcpyHostToDevice,
                        p->up_stream) != cudaSuccess ||
        cudaEventRecord(p->ev_up[s], p->up_stream) != cudaSuccess)
      return fail(FP_ERR_CUDA, "upload of chunk %d failed", c);
    // compute: after the upload, and once chunk c - 2's outputs have left slot s
    if (cudaStreamWaitEvent(stream, p->ev_up[s], 0) != cudaSuccess ||
        (c >= 2 && cudaStreamWaitEvent(stream, p->ev_down[s], 0) != cudaSuccess))
      return fail(FP_ERR_CUDA, "compute stream wait failed");
    const fp_layout cl = chunk_layout(units);
    const fp_status st = fp_forward(p, stage + s * slot, &cl, W, b, pos, dev_out(s, 0),
                                    dev_out(s, 1), dev_out(s, 2), dev_out(s, 3), stream);
    if (st != FP_OK) return st;
    launches += p->last_launches;
    if (cudaEventRecord(p->ev_comp[s], stream) != cudaSuccess ||
        cudaStreamWaitEvent(p->down_stream, p->ev_comp[s], 0) != cudaSuccess)
      return fail(FP_ERR_CUDA, "compute event failed");
    // download
    for (int i = 0; i < 4; ++i) {
      if (!outs_h[i]) continue;
      unsigned char* dst = static_cast<unsigned char*>(outs_h[i]) + u0 * out_unit[i] * esz;
      if (cudaMemcpyAsync(dst, dev_out(s, i), static_cast<size_t>(units * out_unit[i] * esz),
                          cudaMemcpyDeviceToHost, p->down_stream) != cudaSuccess)
        return fail(FP_ERR_CUDA, "download of chunk %d failed", c);
    }
    if (cudaEventRecord(p->ev_down[s], p->down_stream) != cudaSuccess)
      return fail(FP_ERR_CUDA, "download event failed");
  }
  st0 = host_pipeline_join(p, n_chunks, stream);
  if (st0 != FP_OK) return st0;
  p->last_launches = launches;
  return ok();
}

fp_status fp_forward_rope_table(fp_plan* p, const void* x, const fp_layout* x_layout,
                                const void* W, const void* b, const void* rope_cos,
                                const void* rope_sin, const fp_rope_table* tl, void* out_ff,
                                void* out_q, void* out_k, void* out_v, void* stream_v) {
  const NvtxRange range("fp_forward_rope_table");
  if (!p) return fail(FP_ERR_INVALID_ARG, "plan is NULL");
  if (rope_half_of(p) == 0) return fail(FP_ERR_INVALID_ARG, "the plan has no rotary embedding");
  if (!rope_cos || !rope_sin || !tl)
    return fail(FP_ERR_INVALID_ARG, "rope_cos, rope_sin and their layout must be non-NULL");
  if (tl->dtype != FP_BF16 && tl->dtype != FP_F32)
    return fail(FP_ERR_INVALID_ARG, "unknown table dtype");
  if (tl->stride_t < 0 || tl->stride_i < 0)
    return fail(FP_ERR_INVALID_ARG, "negative table stride");
  const int tsz = tl->dtype == FP_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(rope_cos) % tsz || reinterpret_cast<uintptr_t>(rope_sin) % tsz)
    return fail(FP_ERR_MISALIGNED, "tables must be aligned to their element size");
  const Args a{x, x_layout, W, b, nullptr, out_ff, out_q, out_k, out_v};
  Prepared pr;
  fp_status st = prepare(*p, a, pr);
  if (st != FP_OK) return st;
  if (pr.ta.M == 0) {
    p->last_launches = 0;
    return ok();
  }
  // outputs may not overlap the tables either
  const int n_rot = 2 * pr.rh;
  const int64_t span = (pr.ta.T - 1) * tl->stride_t + (n_rot - 1) * tl->stride_i + 1;
  auto rng = [](const void* q, int64_t bytes) {
    uintptr_t lo = reinterpret_cast<uintptr_t>(q);
    return Range{lo, q ? lo + static_cast<uintptr_t>(bytes) : lo};
  };
  const int nkv = p->groups > 0 ? p->groups : p->heads;
  const Range tabs[] = {rng(rope_cos, span * tsz), rng(rope_sin, span * tsz)};
  const Range outs[] = {rng(out_ff, pr.ta.M * p->F * pr.esz),
                        rng(out_q, pr.ta.M * p->heads * p->hd * pr.esz),
                        rng(out_k, pr.ta.M * nkv * p->hd * pr.esz),
                        rng(out_v, pr.ta.M * nkv * p->hd * pr.esz)};
  for (const Range& o : outs)
    for (const Range& t : tabs)
      if (overlaps(o, t)) return fail(FP_ERR_INVALID_ARG, "an output overlaps a rotary table");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  // the imported table is one float4 per (position, pair): two float2 entries
  st = ensure_device_state(p, 2 * pr.ta.T * pr.rh, stream, true);
  if (st != FP_OK) return st;
  p->table_T = -1;  // the default-position table (if any) is overwritten
  p->launch_seq = p->launch_seq % 0x7FFFFFFEu + 1u;
  const Scratch sc{p->d_status, p->d_table, p->device, static_cast<int>(p->launch_seq),
                   p->wait_limit_ns, p->inject_stall, p->group_m, p->max_ctas, p->cluster,
                   p->bounds_check, p->tile_n};
  const ExtTable ext{rope_cos, rope_sin, tl->dtype == FP_BF16, tl->stride_t, tl->stride_i};
  int launches = 0;
  st = launch(*p, pr, a, sc, false, stream, &launches, &ext);
  if (st != FP_OK) return st;
  p->inject_stall = 0;
  p->last_launches = launches;
  return ok();
}

// ---------------------------------------------------------------- backward

namespace {

// 5-D map over x (or over dx, which has x's strides): tokens or channels
// innermost, the non-mergeable token axes outermost, as in the forward.
CUresult encode_x_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* m, const void* base,
                      const Prepared& pr, int C, bool tokens_inner, cuuint32_t box0,
                      cuuint32_t box1, CUtensorMapSwizzle sw) {
  const fp::TokenMap& tk = pr.tk;
  const int esz = pr.esz;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t box[5] = {box0, box1, 1, 1, 1}, estr[5] = {1, 1, 1, 1, 1};
  if (tokens_inner) {
    gdim[0] = tk.S_in;
    gdim[1] = C;
    gstride[0] = static_cast<cuuint64_t>(tk.c_stride) * esz;
  } else {
    gdim[0] = C;
    gdim[1] = tk.S_in;
    gstride[0] = static_cast<cuuint64_t>(tk.s_stride) * esz;
  }
  if (gstride[0] == 0 || gstride[0] % 16) gstride[0] = 16 * ((gdim[0] * esz + 15) / 16);
  cuuint64_t last = gstride[0];
  for (int d = 0; d < 3; ++d) {
    if (d < tk.n_outer_dims) {
      gdim[2 + d] = tk.outer_size[d];
      gstride[1 + d] = static_cast<cuuint64_t>(tk.outer_stride[d]) * esz;
      last = gstride[1 + d];
    } else {
      gdim[2 + d] = 1;
      gstride[1 + d] = last;
    }
  }
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), gdim, gstride,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// G ([M, N] bf16, M = n_outer * S_in) seen as [n_outer][S_in][cols], cols <= N.
CUresult encode_g_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* m, const void* G,
                      const Prepared& pr, int N, int cols, cuuint32_t box0, cuuint32_t box1,
                      CUtensorMapSwizzle sw) {
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(pr.tk.S_in),
                        static_cast<cuuint64_t>(pr.tk.n_outer)};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(N) * 2,
                           static_cast<cuuint64_t>(pr.tk.S_in) * N * 2};
  cuuint32_t box[3] = {box0, box1, 1}, estr[3] = {1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(G), gdim, gstride, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_2d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* m, const void* base,
                   CUtensorMapDataType dt, int esz, int64_t inner, int64_t outer, cuuint32_t box0,
                   cuuint32_t box1, CUtensorMapSwizzle sw) {
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(inner) * esz};
  cuuint32_t box[2] = {box0, box1}, estr[2] = {1, 1};
  return encode(m, dt, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

size_t backward_workspace_bytes(int64_t M, int N) {
  return (static_cast<size_t>(M) * static_cast<size_t>(N) * 2 + 255) / 256 * 256;
}

}  // namespace

fp_status fp_backward_workspace_size(const fp_plan* p, const fp_layout* x_layout, size_t* bytes) {
  if (!p || !x_layout || !bytes) return fail(FP_ERR_INVALID_ARG, "NULL argument");
  const fp_layout& L = *x_layout;
  if (L.ndim < 1 || L.ndim > FP_MAX_DIMS || L.channel_dim < 0 || L.channel_dim >= L.ndim)
    return fail(FP_ERR_INVALID_ARG, "bad x_layout");
  for (int d = 0; d < L.ndim; ++d)
    if (L.sizes[d] < 0) return fail(FP_ERR_INVALID_ARG, "negative size");
  const TokAxes ta = analyse_tokens(L);
  *bytes = backward_workspace_bytes(ta.M, n_total(p));
  return ok();
}

// fp_backward's body. `accumulate`: add this call's dW and db into the
// buffers instead of overwriting them (the host entry point's later chunks);
// the kernels add into dW and db in either case, so only the clearing differs.
static fp_status backward_impl(fp_plan* p, const void* x, const fp_layout* xl, const void* W,
                               const void* b, const int32_t* pos, const void* g_ff,
                               const void* g_q, const void* g_k, const void* g_v, void* dx,
                               float* dW, float* db, void* workspace, size_t workspace_bytes,
                               void* stream_v, bool accumulate) {
  const NvtxRange range("fp_backward");
  if (!p) return fail(FP_ERR_INVALID_ARG, "plan is NULL");
  // the upstream gradients have the forward outputs' shapes: reuse its checks
  const Args a{x, xl, W, b, pos, const_cast<void*>(g_ff), const_cast<void*>(g_q),
               const_cast<void*>(g_k), const_cast<void*>(g_v)};
  Prepared pr;
  fp_status st = prepare(*p, a, pr);
  if (st != FP_OK) return st;
  if (xl->dtype != FP_BF16)
    return fail(FP_ERR_UNSUPPORTED_LAYOUT, "the backward takes bf16 activations");
  const int N = pr.N, C = p->C, F = p->F;
  const int64_t M = pr.ta.M;
  if (M > 0 && !pr.tc_path)
    return fail(FP_ERR_UNSUPPORTED_LAYOUT,
                "the backward runs on the tensor-core path only (bf16, head_dim and ff_hidden "
                "multiples of 16, x addressable by TMA)");
  if (!dW || (M > 0 && !dx)) return fail(FP_ERR_INVALID_ARG, "dx and dW are required");
  const void* ptrs[] = {dx, dW, db, workspace};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(FP_ERR_MISALIGNED, "every pointer must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(FP_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  if (M == 0) {
    // no tokens: the gradients of W and b are zero, dx is empty
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    if (!accumulate &&
        (cudaMemsetAsync(dW, 0, static_cast<size_t>(C) * N * sizeof(float), stream) != cudaSuccess ||
         (db && cudaMemsetAsync(db, 0, static_cast<size_t>(N) * sizeof(float), stream) != cudaSuccess)))
      return fail(FP_ERR_CUDA, "clearing dW / db failed");
    p->last_launches = 0;
    return ok();
  }
  if (!workspace || workspace_bytes < backward_workspace_bytes(M, N))
    return fail(FP_ERR_INVALID_ARG, "workspace too small: %zu bytes needed",
                backward_workspace_bytes(M, N));
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  st = ensure_device_state(p, pr.rope ? pr.ta.T * pr.rh : 0, stream, true);
  if (st != FP_OK) return st;
  int launches = 0;
  // rotary table: the forward's, rebuilt under the same rule
  const bool build_table = pr.rope && (pos != nullptr || p->table_T != pr.ta.T);
  if (pr.rope && !build_table && stream != p->table_stream) {
    if (wait_event(stream, p->table_ready) != cudaSuccess)
      return fail(FP_ERR_CUDA, "stream wait on the rotary table failed");
  }
  if (build_table) {
    cudaError_t err = fp::launch_rope_table(p->d_table, pos, pr.ta.T, pr.rh, 2 * pr.rh,
                                            static_cast<double>(p->rope_base), stream);
    if (err != cudaSuccess) return fail(FP_ERR_CUDA, "rotary table launch: %s", cudaGetErrorString(err));
    ++launches;
    if (!p->table_ready &&
        cudaEventCreateWithFlags(&p->table_ready, cudaEventDisableTiming) != cudaSuccess)
      return fail(FP_ERR_CUDA, "event creation failed");
    if (cudaEventRecord(p->table_ready, stream) != cudaSuccess)
      return fail(FP_ERR_CUDA, "event record failed");
    p->table_stream = stream;
    p->table_T = pos ? -1 : pr.ta.T;
  }
  if (!accumulate &&
      (cudaMemsetAsync(dW, 0, static_cast<size_t>(C) * N * sizeof(float), stream) != cudaSuccess ||
       (db && cudaMemsetAsync(db, 0, static_cast<size_t>(N) * sizeof(float), stream) != cudaSuccess)))
    return fail(FP_ERR_CUDA, "clearing dW / db failed");

  p->launch_seq = p->launch_seq % 0x7FFFFFFEu + 1u;
  const int tag = static_cast<int>(p->launch_seq);
  // 1. q|k|v part of G (launched in step 2: beside the ff gradient when that
  // runs on the tensor-core forward kernel, else before it)
  auto launch_gather = [&](cudaStream_t gs) -> fp_status {
    fp::BwdGatherParams gp{};
    gp.g_q = g_q;
    gp.g_k = g_k;
    gp.g_v = g_v;
    gp.G = workspace;
    gp.db = db;
    gp.rope_cs = pr.rope ? p->d_table : nullptr;
    gp.M = M;
    gp.T = pr.ta.T;
    gp.F = F;
    gp.N = N;
    gp.C = C;
    gp.heads = p->heads;
    gp.hd = p->hd;
    gp.groups = p->groups;
    gp.rope_half = pr.rh;
    gp.k_transposed = p->k_transposed;
    cudaError_t err = fp::launch_bwd_gather(gp, gs);
    if (err != cudaSuccess) return fail(FP_ERR_CUDA, "gradient gather launch: %s", cudaGetErrorString(err));
    ++launches;
    return FP_OK;
  };
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
  if (!encode) return fail(FP_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  fp::BwdGemmParams base{};
  base.tok = pr.tk;
  base.group_m = p->group_m;
  base.C = C;
  base.F = F;
  base.N = N;
  base.act = p->act;
  base.status = p->d_status;
  base.wait_limit_ns = p->wait_limit_ns;
  base.launch_tag = tag;
  base.k_splits = 1;
  base.cluster = 1;
  const int mps = static_cast<int>((pr.tk.S_in + fp::kTcBM - 1) / fp::kTcBM);
  const int ctas = p->max_ctas > 0 ? std::min(sm_count(p->device), p->max_ctas) : sm_count(p->device);
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  auto map_fail = [&](const char* what) {
    return fail(FP_ERR_UNSUPPORTED_LAYOUT, "backward: tensor map for %s rejected", what);
  };
  // 2. ff part of G: recompute x W_ff + b_ff, times act' and the upstream gradient.
  // CTA pairs of the forward kernel in its gradient mode when every tile is a
  // whole number of 32-column units; the single-CTA backward kernel otherwise.
  const int64_t fwd_m_tiles = pr.tk.n_outer * mps;
  // (TMA coordinates are 32-bit: the gradient mode's stores need M < 2^31)
  const bool tc_grad = F > 0 && F % 32 == 0 && fwd_m_tiles >= 2 && M <= INT32_MAX;
  // The gather (HBM-bound) and the ff gradient (tensor- and latency-bound)
  // write disjoint columns of G and of db. With both present the ff gradient
  // runs on all but kGatherSMs SMs and the gather on a second stream fills
  // the rest: a gradient CTA holds nearly all of an SM's shared memory, so
  // no gather block lands beside it. The gradient is launched first so its
  // CTAs claim their SMs before the gather's blocks are queued. SMs left to
  // the gather, walrus backward: 12 -> 470 us, 24 -> 465, 36 -> 462, 48 -> 469
  // (471 with the two in sequence).
  constexpr int kGatherSMs = 36;
  const bool fork = tc_grad && p->heads > 0 && ctas >= kGatherSMs + 16;
  if (p->heads > 0 && !fork) {
    st = launch_gather(stream);
    if (st != FP_OK) return st;
  }
  if (fork) {
    if (!p->side_stream &&
        cudaStreamCreateWithFlags(&p->side_stream, cudaStreamNonBlocking) != cudaSuccess)
      return fail(FP_ERR_CUDA, "side stream creation failed");
    if ((!p->ev_fork && cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess) ||
        (!p->ev_join && cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) != cudaSuccess))
      return fail(FP_ERR_CUDA, "event creation failed");
    if (cudaEventRecord(p->ev_fork, stream) != cudaSuccess ||
        cudaStreamWaitEvent(p->side_stream, p->ev_fork, 0) != cudaSuccess)
      return fail(FP_ERR_CUDA, "forking the gather stream failed");
  }
  if (tc_grad) {
    fp::TcParams tp;
    memset(&tp, 0, sizeof tp);
    if (encode_x_map(encode, &tp.tmap_a, x, pr, C, pr.a_mn, 64, pr.a_mn ? 64 : 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return map_fail("x");
    if (encode_2d(encode, &tp.tmap_b, W, BF, 2, N, C, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) !=
        CUDA_SUCCESS)
      return map_fail("W");
    if (b && encode_2d(encode, &tp.tmap_bias, b, BF, 2, N, 1, 64, 1, CU_TENSOR_MAP_SWIZZLE_NONE) !=
                 CUDA_SUCCESS)
      return map_fail("b");
    {  // G's ff columns, [M][F] with row stride N, 32 x 32 boxes
      cuuint64_t d[2] = {static_cast<cuuint64_t>(F), static_cast<cuuint64_t>(M)};
      cuuint64_t st[1] = {static_cast<cuuint64_t>(N) * 2};
      cuuint32_t bx[2] = {32, 32}, es[2] = {1, 1};
      if (encode(&tp.tmap_ff32, BF, 2, workspace, d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return map_fail("G");
    }
    tp.tma_store = 1;
    tp.tok = pr.tk;
    fp::Epilogue& e = tp.epi;
    e.M = M;
    e.T = pr.ta.T;
    e.N = F;  // only the ff columns
    e.F = F;
    e.C = C;
    e.act = p->act;
    e.bias = b;
    e.out_ff = workspace;
    e.ff_ld = N;
    e.g_ff = g_ff;
    e.db = db;
    e.status = p->d_status;
    e.bn_eff = fp::kTcBN;
    tp.C = C;
    tp.num_k_blocks = (C + fp::kTcBK - 1) / fp::kTcBK;
    tp.m_tiles_per_slab = mps;
    tp.num_m_tiles = fwd_m_tiles;
    tp.num_n_tiles = (F + fp::kTcBN - 1) / fp::kTcBN;
    tp.num_tiles = tp.num_m_tiles * tp.num_n_tiles;
    tp.cluster = 2;
    tp.num_units = (tp.num_m_tiles + 1) / 2 * tp.num_n_tiles;
    tp.group_m = p->group_m;
    tp.wait_limit_ns = p->wait_limit_ns;
    tp.inject_stall = p->inject_stall;
    tp.launch_tag = tag;
    cudaError_t err = fp::launch_tc_gemm(tp, pr.a_mn, fork ? (ctas - kGatherSMs) & ~1 : ctas,
                                         stream, true);
    if (err != cudaSuccess) return fail(FP_ERR_CUDA, "backward GEMM launch: %s", cudaGetErrorString(err));
    ++launches;
    if (fork) {
      st = launch_gather(p->side_stream);
      if (st != FP_OK) return st;
      if (cudaEventRecord(p->ev_join, p->side_stream) != cudaSuccess ||
          cudaStreamWaitEvent(stream, p->ev_join, 0) != cudaSuccess)
        return fail(FP_ERR_CUDA, "joining the gather stream failed");
    }
  } else if (F > 0) {
    fp::BwdGemmParams gp = base;
    gp.mode = fp::BWD_GRADFF;
    if (encode_x_map(encode, &gp.tmap_a, x, pr, C, pr.a_mn, 64, pr.a_mn ? 64 : 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return map_fail("x");
    if (encode_2d(encode, &gp.tmap_b, W, BF, 2, N, C, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) !=
        CUDA_SUCCESS)
      return map_fail("W");
    if (encode_g_map(encode, &gp.tmap_out, workspace, pr, N, F, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
      return map_fail("G");
    gp.m_tiles_per_slab = mps;
    gp.num_m_tiles = static_cast<int>(pr.tk.n_outer) * mps;
    gp.num_n_tiles = (F + fp::kTcBN - 1) / fp::kTcBN;
    gp.num_k_blocks = (C + fp::kTcBK - 1) / fp::kTcBK;
    gp.num_units = static_cast<int64_t>(gp.num_m_tiles) * gp.num_n_tiles;
    gp.bias = b;
    gp.g_ff = g_ff;
    gp.db = db;
    cudaError_t err = fp::launch_bwd_gemm(gp, pr.a_mn, ctas, stream);
    if (err != cudaSuccess) return fail(FP_ERR_CUDA, "backward GEMM launch: %s", cudaGetErrorString(err));
    ++launches;
  }
  // CTA pairs for the dx GEMM (the plan's cluster option), whole clusters
  const int bwd_cl = p->cluster == 2 && ctas >= 2 ? 2 : 1;
  // 3. dx = G W^T, stored in x's layout (dx^T = W G^T when tokens are innermost)
  {
    fp::BwdGemmParams gp = base;
    if (encode_x_map(encode, &gp.tmap_out, dx, pr, C, pr.a_mn, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) !=
        CUDA_SUCCESS)
      return map_fail("dx");
    gp.num_k_blocks = (N + fp::kTcBK - 1) / fp::kTcBK;
    if (!pr.a_mn) {
      gp.mode = fp::BWD_DX;
      gp.m_tiles_per_slab = mps;
      gp.num_m_tiles = static_cast<int>(pr.tk.n_outer) * mps;
      gp.num_n_tiles = (C + fp::kTcBN - 1) / fp::kTcBN;
      gp.cluster = gp.num_m_tiles >= 2 ? bwd_cl : 1;
      if (encode_g_map(encode, &gp.tmap_a, workspace, pr, N, N, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return map_fail("G");
      // B: this CTA's share of the tile's 256 channel rows
      if (encode_2d(encode, &gp.tmap_b, W, BF, 2, N, C, 64, fp::kTcBN / gp.cluster,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return map_fail("W");
    } else {
      gp.mode = fp::BWD_DXT;
      gp.num_m_tiles = (C + fp::kTcBM - 1) / fp::kTcBM;
      gp.n_tiles_per_slab = static_cast<int>((pr.tk.S_in + fp::kTcBN - 1) / fp::kTcBN);
      gp.num_n_tiles = static_cast<int>(pr.tk.n_outer) * gp.n_tiles_per_slab;
      gp.cluster = gp.num_m_tiles >= 2 ? bwd_cl : 1;
      if (encode_2d(encode, &gp.tmap_a, W, BF, 2, N, C, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) !=
          CUDA_SUCCESS)
        return map_fail("W");
      // B: this CTA's share of the tile's 256 token rows
      if (encode_g_map(encode, &gp.tmap_b, workspace, pr, N, N, 64, fp::kTcBN / gp.cluster,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return map_fail("G");
    }
    gp.num_units = static_cast<int64_t>((gp.num_m_tiles + gp.cluster - 1) / gp.cluster) *
                   gp.num_n_tiles;
    cudaError_t err = fp::launch_bwd_gemm(gp, false, ctas, stream);
    if (err != cudaSuccess) return fail(FP_ERR_CUDA, "backward GEMM launch: %s", cudaGetErrorString(err));
    ++launches;
  }
  // 4. dW = X^T G (fp32), the token range split across CTAs, partials added by TMA
  {
    fp::BwdGemmParams gp = base;
    gp.mode = fp::BWD_DW;
    if (encode_x_map(encode, &gp.tmap_a, x, pr, C, pr.a_mn, 64, pr.a_mn ? 128 : 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return map_fail("x");
    if (encode_g_map(encode, &gp.tmap_b, workspace, pr, N, N, 64, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return map_fail("G");
    if (encode_2d(encode, &gp.tmap_out, dW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, N, C, 16, 32,
                  CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
      return map_fail("dW");
    gp.num_m_tiles = (C + fp::kTcBM - 1) / fp::kTcBM;
    gp.num_n_tiles = (N + fp::kTcBN - 1) / fp::kTcBN;
    // single CTAs: on CTA pairs this GEMM measured slower (walrus 148 -> 163 us,
    // the LLM shape 630 -> 733 us) while the dx GEMMs gained
    gp.cluster = 1;
    gp.k_blocks_per_slab = static_cast<int>((pr.tk.S_in + fp::kTcBK - 1) / fp::kTcBK);
    const int64_t kb = pr.tk.n_outer * gp.k_blocks_per_slab;
    if (kb > INT32_MAX) return fail(FP_ERR_UNSUPPORTED_LAYOUT, "too many tokens");
    gp.num_k_blocks = static_cast<int>(kb);
    // work items are (row-tile group of `cluster`, column tile, split); a wave
    // is one item per cluster
    const int64_t tiles =
        static_cast<int64_t>((gp.num_m_tiles + gp.cluster - 1) / gp.cluster) * gp.num_n_tiles;
    const int64_t slots = std::max<int64_t>(1, ctas / gp.cluster);
    // k splits: counting up from one item per cluster, the first count whose
    // waves are at least 97 % full (a last, partly idle wave costs a whole
    // one), else the fullest; ties take fewer splits (less reduce-add
    // traffic). Large outputs are not split (each split adds a
    // read-modify-write of dW), and every split keeps at least 16 k-blocks.
    int64_t splits = 1;
    double best_fill = -1.0;
    const int64_t max_splits = tiles >= 4 * slots
                                   ? 1
                                   : std::max<int64_t>(1, std::min<int64_t>(kb / 16, 32));
    for (int64_t sp = std::min(max_splits, std::max<int64_t>(1, (slots + tiles - 1) / tiles));
         sp <= max_splits; ++sp) {
      const int64_t units = tiles * sp;
      const double fill = static_cast<double>(units) /
                          static_cast<double>((units + slots - 1) / slots * slots);
      if (fill > best_fill + 1e-9) {
        best_fill = fill;
        splits = sp;
      }
      if (fill > 0.97) break;
    }
    splits = std::max<int64_t>(1, std::min<int64_t>(splits, kb));
    gp.k_splits = static_cast<int>(splits);
    gp.num_units = tiles * splits;
    cudaError_t err = fp::launch_bwd_gemm(gp, !pr.a_mn, ctas, stream);
    if (err != cudaSuccess) return fail(FP_ERR_CUDA, "backward GEMM launch: %s", cudaGetErrorString(err));
    ++launches;
  }
  p->inject_stall = 0;
  p->last_launches = launches;
  return ok();
}

// ---------------------------------------------------------------- attention over the outputs

fp_status fp_backward(fp_plan* p, const void* x, const fp_layout* xl, const void* W, const void* b,
                      const int32_t* pos, const void* g_ff, const void* g_q, const void* g_k,
                      const void* g_v, void* dx, float* dW, float* db, void* workspace,
                      size_t workspace_bytes, void* stream_v) {
  return backward_impl(p, x, xl, W, b, pos, g_ff, g_q, g_k, g_v, dx, dW, db, workspace,
                       workspace_bytes, stream_v, false);
}

fp_status fp_backward_host(fp_plan* p, const void* x_host, const fp_layout* xl, const void* W,
                           const void* b, const int32_t* pos, const void* gff_h,
                           const void* gq_h, const void* gk_h, const void* gv_h, void* dx_h,
                           float* dW_h, float* db_h, void* stream_v) {
  const NvtxRange range("fp_backward_host");
  if (!p) return fail(FP_ERR_INVALID_ARG, "plan is NULL");
  if (!xl) return fail(FP_ERR_INVALID_ARG, "x_layout is NULL");
  const void* const g_h[4] = {gff_h, gq_h, gk_h, gv_h};
  {
    // the forward's checks on x and the gradients (they have the outputs' shapes)
    const Args full{x_host, xl, W, b, pos, const_cast<void*>(gff_h), const_cast<void*>(gq_h),
                    const_cast<void*>(gk_h), const_cast<void*>(gv_h)};
    Prepared pr;
    const fp_status st = prepare(*p, full, pr);
    if (st != FP_OK) return st;
    if (xl->dtype != FP_BF16)
      return fail(FP_ERR_UNSUPPORTED_LAYOUT, "the backward takes bf16 activations");
    if (pr.ta.M > 0 && !pr.tc_path)
      return fail(FP_ERR_UNSUPPORTED_LAYOUT,
                  "the backward runs on the tensor-core path only (bf16, head_dim and ff_hidden "
                  "multiples of 16, x addressable by TMA)");
  }
  if (!dW_h || !dx_h) return fail(FP_ERR_INVALID_ARG, "dx and dW are required");
  const fp_layout L = *xl;
  const HostChunks hc = host_chunks(L);
  // dx comes back as whole byte ranges: a strided x's gaps would be overwritten
  if (!hc.dense)
    return fail(FP_ERR_UNSUPPORTED_LAYOUT, "fp_backward_host needs a dense (row-major) x");
  const void* const host_ptrs[] = {x_host, gff_h, gq_h, gk_h, gv_h, dx_h, dW_h, db_h};
  for (const void* q : host_ptrs)
    if (q && !page_locked(q))
      return fail(FP_ERR_INVALID_ARG, "host buffers must be page-locked host memory");
  const int64_t esz = 2;
  const TokAxes ta = analyse_tokens(L);
  const int N = n_total(p), C = p->C;
  const bool chunked = hc.chunked;
  const int64_t span = hc.span, per_chunk = hc.per_chunk, numel = hc.numel;
  const int n_chunks = hc.n_chunks;
  const int nkv = p->groups > 0 ? p->groups : p->heads;
  const int64_t m_unit = ta.M / span, x_unit = numel / span;
  const int64_t g_unit[4] = {m_unit * p->F, m_unit * p->heads * p->hd, m_unit * nkv * p->hd,
                             m_unit * nkv * p->hd};
  // one slot: x, g_ff, g_q, g_k, g_v, dx; then, shared by the slots, the G
  // workspace of one chunk, dW and db
  int64_t off[6], slot = 0;
  off[0] = 0;
  slot = align_up(per_chunk * x_unit * esz, kStageAlign);
  for (int i = 0; i < 4; ++i) {
    off[i + 1] = slot;
    slot += g_h[i] ? align_up(per_chunk * g_unit[i] * esz, kStageAlign) : 0;
  }
  off[5] = slot;
  slot += align_up(per_chunk * x_unit * esz, kStageAlign);
  const int64_t ws_bytes =
      align_up(static_cast<int64_t>(backward_workspace_bytes(per_chunk * m_unit, N)), kStageAlign);
  const int64_t dw_bytes = align_up(static_cast<int64_t>(C) * N * 4, kStageAlign);
  const int64_t db_bytes = align_up(static_cast<int64_t>(N) * 4, kStageAlign);
  const int64_t total = 2 * slot + ws_bytes + dw_bytes + db_bytes;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  fp_status st0 = host_pipeline_setup(p, total, stream);
  if (st0 != FP_OK) return st0;
  unsigned char* const stage = static_cast<unsigned char*>(p->d_host_stage);
  void* const ws = stage + 2 * slot;
  float* const dW = reinterpret_cast<float*>(stage + 2 * slot + ws_bytes);
  float* const db = db_h ? reinterpret_cast<float*>(stage + 2 * slot + ws_bytes + dw_bytes) : nullptr;
  auto chunk_layout = [&](int64_t units) {
    fp_layout c = L;
    if (chunked) c.sizes[0] = units;
    return c;
  };
  auto dev_g = [&](int s, int i) -> const void* {
    return g_h[i] ? stage + s * slot + off[i + 1] : nullptr;
  };
  st0 = host_pipeline_fork(p, stream);
  if (st0 != FP_OK) return st0;
  int launches = 0;
  for (int c = 0; c < n_chunks; ++c) {
    const int s = c & 1;
    const int64_t u0 = c * per_chunk, units = std::min(per_chunk, span - u0);
    // upload x and the four gradients; slot s is free once chunk c - 2 is computed
    if (c >= 2 && cudaStreamWaitEvent(p->up_stream, p->ev_comp[s], 0) != cudaSuccess)
      return fail(FP_ERR_CUDA, "upload stream wait failed");
    if (cudaMemcpyAsync(stage + s * slot, static_cast<const unsigned char*>(x_host) + u0 * x_unit * esz,
                        static_cast<size_t>(units * x_unit * esz), cudaMemcpyHostToDevice,
                        p->up_stream) != cudaSuccess)
      return fail(FP_ERR_CUDA, "upload of chunk %d failed", c);
    for (int i = 0; i < 4; ++i) {
      if (!g_h[i]) continue;
      if (cudaMemcpyAsync(const_cast<void*>(dev_g(s, i)),
                          static_cast<const unsigned char*>(g_h[i]) + u0 * g_unit[i] * esz,
                          static_cast<size_t>(units * g_unit[i] * esz), cudaMemcpyHostToDevice,
                          p->up_stream) != cudaSuccess)
        return fail(FP_ERR_CUDA, "upload of chunk %d failed", c);
    }
    if (cudaEventRecord(p->ev_up[s], p->up_stream) != cudaSuccess)
      return fail(FP_ERR_CUDA, "upload event failed");
    // gradients of the chunk; dW and db summed over the chunks
    if (cudaStreamWaitEvent(stream, p->ev_up[s], 0) != cudaSuccess ||
        (c >= 2 && cudaStreamWaitEvent(stream, p->ev_down[s], 0) != cudaSuccess))
      return fail(FP_ERR_CUDA, "compute stream wait failed");
    const fp_layout cl = chunk_layout(units);
    const fp_status st = backward_impl(p, stage + s * slot, &cl, W, b, pos, dev_g(s, 0),
                                       dev_g(s, 1), dev_g(s, 2), dev_g(s, 3),
                                       stage + s * slot + off[5], dW, db, ws,
                                       static_cast<size_t>(ws_bytes), stream, c > 0);
    if (st != FP_OK) return st;
    launches += p->last_launches;
    if (cudaEventRecord(p->ev_comp[s], stream) != cudaSuccess ||
        cudaStreamWaitEvent(p->down_stream, p->ev_comp[s], 0) != cudaSuccess)
      return fail(FP_ERR_CUDA, "compute event failed");
    if (cudaMemcpyAsync(static_cast<unsigned char*>(dx_h) + u0 * x_unit * esz,
                        stage + s * slot + off[5], static_cast<size_t>(units * x_unit * esz),
                        cudaMemcpyDeviceToHost, p->down_stream) != cudaSuccess)
      return fail(FP_ERR_CUDA, "download of chunk %d failed", c);
    if (c == n_chunks - 1 &&
        (cudaMemcpyAsync(dW_h, dW, static_cast<size_t>(C) * N * 4, cudaMemcpyDeviceToHost,
                         p->down_stream) != cudaSuccess ||
         (db_h && cudaMemcpyAsync(db_h, db, static_cast<size_t>(N) * 4, cudaMemcpyDeviceToHost,
                                  p->down_stream) != cudaSuccess)))
      return fail(FP_ERR_CUDA, "download of dW / db failed");
    if (cudaEventRecord(p->ev_down[s], p->down_stream) != cudaSuccess)
      return fail(FP_ERR_CUDA, "download event failed");
  }
  st0 = host_pipeline_join(p, n_chunks, stream);
  if (st0 != FP_OK) return st0;
  p->last_launches = launches;
  return ok();
}

extern "C" fp_status fp_attention(fp_plan* p, const void* q, const void* k, const void* v,
                                  void* out, int64_t batch, int64_t T_q, int64_t T_k, float scale,
                                  void* stream_v) {
  const NvtxRange range("fp_attention");
  if (!p) return fail(FP_ERR_INVALID_ARG, "plan is NULL");
  if (p->heads == 0) return fail(FP_ERR_INVALID_ARG, "the plan has no attention heads");
  if (batch < 0 || T_q < 0 || T_k < 0) return fail(FP_ERR_INVALID_ARG, "negative size");
  const int hd = p->hd, heads = p->heads;
  const int kvh = p->groups > 0 ? p->groups : p->heads;
  if (hd != 64 && hd != 128)
    return fail(FP_ERR_UNSUPPORTED_LAYOUT, "attention takes head_dim 64 or 128 (plan has %d)", hd);
  if (batch == 0 || T_q == 0) return ok();
  if (T_k == 0) return fail(FP_ERR_INVALID_ARG, "attention needs at least one key");
  if (!q || !k || !v || !out) return fail(FP_ERR_INVALID_ARG, "q, k, v and out must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(FP_ERR_MISALIGNED, "every pointer must be 16-byte aligned");
  if (p->k_transposed && T_k % 8)
    return fail(FP_ERR_UNSUPPORTED_LAYOUT,
                "pre-transposed k needs T_k a multiple of 8 (its rows are TMA strides)");
  const int64_t BH = batch * heads, BHkv = batch * kvh;
  if (BH > INT32_MAX || T_q > INT32_MAX || T_k > INT32_MAX ||
      BH * ((T_q + 127) / 128) > INT32_MAX)
    return fail(FP_ERR_UNSUPPORTED_LAYOUT, "attention sizes beyond 32-bit grid coordinates");
  auto rng = [](const void* a, int64_t bytes) {
    uintptr_t lo = reinterpret_cast<uintptr_t>(a);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
  };
  const Range ro = rng(out, BH * T_q * hd * 2);
  if (overlaps(ro, rng(q, BH * T_q * hd * 2)) || overlaps(ro, rng(k, BHkv * T_k * hd * 2)) ||
      overlaps(ro, rng(v, BHkv * T_k * hd * 2)))
    return fail(FP_ERR_INVALID_ARG, "out overlaps an input");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(FP_ERR_CUDA, "cudaGetDevice failed");
  const int64_t q_blocks = BH * ((T_q + 127) / 128);
  const fp::AttnSplit split = fp::attention_split(q_blocks, T_k, hd, sm_count(dev));
  fp_status st = ensure_device_state(p, 0, stream, true, split.part_bytes);
  if (st != FP_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
  if (!encode) return fail(FP_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  fp::AttnParams ap;
  memset(&ap, 0, sizeof ap);
  const cuuint32_t es[3] = {1, 1, 1};
  auto map3 = [&](CUtensorMap* m, const void* base, cuuint64_t d0, cuuint64_t d1, cuuint64_t d2,
                  cuuint32_t b0, cuuint32_t b1) {
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const cuuint32_t box[3] = {b0, b1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  CUresult r = map3(&ap.tmap_q, q, hd, T_q, BH, 64, 128);
  if (r == CUDA_SUCCESS)
    r = p->k_transposed ? map3(&ap.tmap_k, k, T_k, hd, BHkv, 64, 64)
                        : map3(&ap.tmap_k, k, hd, T_k, BHkv, 64, 128);
  if (r == CUDA_SUCCESS) r = map3(&ap.tmap_v, v, hd, T_k, BHkv, 64, 64);
  if (r != CUDA_SUCCESS)
    return fail(FP_ERR_UNSUPPORTED_LAYOUT, "attention tensor map rejected (CUresult %d)",
                static_cast<int>(r));
  ap.out = out;
  ap.Tq = T_q;
  ap.Tk = T_k;
  ap.BH = static_cast<int>(BH);
  ap.hd = hd;
  ap.heads = heads;
  ap.kv_heads = kvh;
  ap.k_transposed = p->k_transposed;
  ap.num_q_blocks = static_cast<int>((T_q + 127) / 128);
  const double sc = scale > 0.0f ? static_cast<double>(scale) : 1.0 / sqrt(static_cast<double>(hd));
  ap.scale_log2e = static_cast<float>(sc * 1.4426950408889634);
  p->launch_seq = p->launch_seq % 0x7FFFFFFEu + 1u;
  ap.status = p->d_status;
  ap.wait_limit_ns = p->wait_limit_ns;
  ap.launch_tag = static_cast<int>(p->launch_seq);
  ap.full = split.full;
  ap.splits = split.splits;
  ap.part = p->d_attn;
  int launches = 0;
  const cudaError_t err = fp::launch_attention(ap, stream, &launches);
  p->last_launches = launches;
  if (err != cudaSuccess)
    return fail(FP_ERR_CUDA, "attention launch: %s", cudaGetErrorString(err));
  return ok();
}

// ---------------------------------------------------------------- no-allocation entry point
//
// fp_forward_noalloc serves callers that must not allocate device memory
// themselves or through this library once they are running: plug-ins of a
// host framework that owns every device byte through its own pool, and
// fixed-budget serving processes that size memory once at start-up and treat
// a later cudaMalloc (which can also stall the device) as a failure. It runs
// the same kernels as fp_forward; their device scratch (status words and the
// rotary table) lives in the static array below instead of in a plan.

}  // extern "C"

namespace {

constexpr int64_t kNoAllocTableEntries = int64_t{1} << 19;  // (cos, sin) pairs: 4 MiB
constexpr int64_t kNoAllocHeaderBytes = 256;                // status words live here

}  // namespace

// [status words (256 B) | rotary table (4 MiB)]. Every GPU that loads this
// library holds it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocHeaderBytes +
                                                                 8 * kNoAllocTableEntries];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// Device address of g_noalloc_scratch on the current device. In host code the
// symbol's name is only a host-side stand-in, so the address is asked of the
// runtime once per device (with that device current) and cached.
fp_status noalloc_scratch(int dev, unsigned char** out) {
  if (dev < 0 || dev >= 64) return fail(FP_ERR_INVALID_ARG, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    cudaError_t err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (err != cudaSuccess || !ptr)
      return fail(FP_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                  cudaGetErrorString(err));
    g_noalloc_addr[dev] = ptr;
  }
  *out = static_cast<unsigned char*>(g_noalloc_addr[dev]);
  return FP_OK;
}

// The rules fp_create_ex applies, for a configuration that gets no plan.
fp_status check_config(const fp_config& c) {
  if (c.C <= 0) return fail(FP_ERR_INVALID_ARG, "C must be > 0 (got %d)", c.C);
  if (c.ff_hidden < 0 || c.heads < 0 || c.n_query_groups < 0)
    return fail(FP_ERR_INVALID_ARG, "ff_hidden, heads and n_query_groups must be >= 0");
  if (c.heads > 0) {
    if (c.head_dim <= 0 || c.head_dim % 2)
      return fail(FP_ERR_INVALID_ARG, "head_dim must be even and > 0 (got %d)", c.head_dim);
    if (static_cast<int64_t>(c.heads) * c.head_dim != c.C)
      return fail(FP_ERR_INVALID_ARG, "heads * head_dim must equal C");
    if (c.ff_hidden % c.head_dim)
      return fail(FP_ERR_INVALID_ARG, "ff_hidden must be a multiple of head_dim");
    if (c.n_query_groups > 0 && c.heads % c.n_query_groups)
      return fail(FP_ERR_INVALID_ARG, "heads must be a multiple of n_query_groups");
    if (c.rope_n_elem < 0 || c.rope_n_elem % 2 || c.rope_n_elem > c.head_dim)
      return fail(FP_ERR_INVALID_ARG, "rope_n_elem must be even and <= head_dim");
    if (c.rope_base > 0.0f && c.head_dim > 128)
      return fail(FP_ERR_INVALID_ARG, "rotary embedding needs head_dim <= 128");
  } else if (c.n_query_groups > 0) {
    return fail(FP_ERR_INVALID_ARG, "n_query_groups needs heads > 0");
  }
  if (c.ff_hidden == 0 && c.heads == 0) return fail(FP_ERR_INVALID_ARG, "nothing to compute");
  if (c.act < FP_ACT_NONE || c.act > FP_ACT_RELU2) return fail(FP_ERR_INVALID_ARG, "unknown act");
  return FP_OK;
}

std::atomic<uint32_t> g_noalloc_seq{0};

}  // namespace

extern "C" fp_status fp_forward_noalloc(const fp_config* config, const void* x,
                                        const fp_layout* x_layout, const void* W, const void* b,
                                        const int32_t* pos, void* out_ff, void* out_q,
                                        void* out_k, void* out_v, void* stream_v) {
  if (!config) return fail(FP_ERR_INVALID_ARG, "config is NULL");
  fp_status st = check_config(*config);
  if (st != FP_OK) return st;
  fp_plan pl{};  // on the stack: no plan object, no device state of its own
  pl.C = config->C;
  pl.F = config->ff_hidden;
  pl.heads = config->heads;
  pl.hd = config->heads > 0 ? config->head_dim : 0;
  pl.groups = config->heads > 0 ? config->n_query_groups : 0;
  pl.rope_n_elem = config->heads > 0 ? config->rope_n_elem : 0;
  pl.k_transposed = config->heads > 0 && config->k_transposed ? 1 : 0;
  pl.act = config->act;
  pl.rope_base = config->rope_base;
  const Args a{x, x_layout, W, b, pos, out_ff, out_q, out_k, out_v};
  Prepared pr;
  st = prepare(pl, a, pr);
  if (st != FP_OK) return st;
  if (pr.ta.M == 0) return ok();
  const int64_t need = pr.rope ? pr.ta.T * pr.rh : 0;
  if (need > kNoAllocTableEntries)
    return fail(FP_ERR_INVALID_ARG,
                "rotary table needs %lld entries (T = %lld positions x %d frequencies); "
                "fp_forward_noalloc holds at most %lld",
                static_cast<long long>(need), static_cast<long long>(pr.ta.T), pr.rh,
                static_cast<long long>(kNoAllocTableEntries));
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(FP_ERR_CUDA, "cudaGetDevice failed");
  unsigned char* base = nullptr;
  st = noalloc_scratch(dev, &base);
  if (st != FP_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  int* status = reinterpret_cast<int*>(base);
  // the array keeps the previous call's contents: the status words must start at zero
  if (cudaMemsetAsync(status, 0, 2 * sizeof(int), stream) != cudaSuccess)
    return fail(FP_ERR_CUDA, "clearing the static status words failed");
  const uint32_t tag = g_noalloc_seq.fetch_add(1) % 0x7FFFFFFEu + 1u;
  const Scratch sc{status, reinterpret_cast<float2*>(base + kNoAllocHeaderBytes), dev,
                   static_cast<int>(tag), kDefaultWaitLimitNs, 0, kDefaultGroupM, 0,
                   kDefaultCluster, 0, 0};
  int launches = 0;
  // the shared table may hold another call's positions: always rebuild it
  st = launch(pl, pr, a, sc, pr.rope, stream, &launches);
  return st == FP_OK ? ok() : st;
}
