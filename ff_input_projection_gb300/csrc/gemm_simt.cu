// Fused projection on the FFMA pipes (TF32 off).
//
// The fp32 leg of the projection: activations and weight stay fp32 and every
// product is an fp32 FFMA, so results do not depend on whether TF32 matmul is
// enabled (the fp32-vs-TF32 ambiguity raised in xformers PR #283 "[perf] Fused
// linear", last comments). x is read in place through its strides, as in
// Walrus PR #12 "Make fused_ff_qkv contiguous" (no permuted copy). The same
// kernel, instantiated for bf16 storage (widened to fp32 on load, rounded once
// at the store), serves bf16 activations whose strides a TMA map cannot
// describe (e.g. an odd spatial extent) or whose block widths are not
// multiples of 16.
//
// Tile: 128 tokens x 128 fused columns, 256 threads with an 8x8 register
// block each (accumulated on packed fp32 pairs) (rows ty*4+{0..3} and
// 64+ty*4+{0..3}, columns likewise). Two main loops:
//  * general (any strides, bf16 or fp32 storage): k-steps of 16,
//    double-buffered in shared memory with a register prefetch of the next
//    k-step;
//  * fp32 with 16-byte-aligned chunks, either unit-stride tokens
//    (channels-first x such as NCHW) or unit-stride channels (row-major x):
//    k-steps of 32 copied global -> shared by cp.async; tiles of 128 or 64
//    columns (4 CTAs of 128 threads per SM), whichever spreads the work more
//    evenly.
// The epilogue stages the fp32 tile in shared memory so a rotary pair (lane i,
// lane i + half) can be read by whichever thread owns either lane, then adds
// bias, applies the activation or the rotation, and writes ff token-major and
// q/k/v head-major with consecutive threads on consecutive lanes. Tiles of the
// second loop without rotation or transposed k skip the staging and store
// 16-byte groups straight from registers.
#include "epilogue.cuh"
#include "fp_internal.h"

namespace fp {

namespace {

constexpr int BM = kSimtBM, BN = kSimtBN, BK = 16, NT = 256;
constexpr int CS_LD = BN + 4;
// epilogue tile + per-row output bases; covers the 2x(A+B) operand buffers
constexpr int kSmemBytes = BM * CS_LD * 4 + 5 * BM * 8;
static_assert(2 * BK * (BM + BN) * 4 <= kSmemBytes, "operand buffers must fit in the epilogue tile");

__device__ __forceinline__ int64_t outer_offset(const TokenMap& tk, int64_t o) {
  int64_t off = 0;
  for (int d = 0; d < tk.n_outer_dims; ++d) {
    int64_t sz = tk.outer_size[d];
    int64_t i = o % sz;
    o /= sz;
    off += i * tk.outer_stride[d];
  }
  return off;
}

// K_MAJOR: unit channel stride, so a thread walks channels (16 consecutive
// channels of one token per k-step); otherwise a thread keeps one token and
// walks channels at their stride (coalesced when tokens are unit-stride).
template <typename T>
__device__ __forceinline__ float ld_elem(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p, int64_t i) {
  return __ldg(p + i);
}
template <>
__device__ __forceinline__ float ld_elem<uint16_t>(const uint16_t* p, int64_t i) {
  return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(p) + i));
}
__device__ __forceinline__ void st_elem(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_elem(uint16_t* p, int64_t i, float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  p[i] = *reinterpret_cast<uint16_t*>(&h);
}

// Epilogue of one tile, kept out of line so the main loop's register
// allocation does not carry it. Cs holds the fp32 accumulator tile [BM][CS_LD]
// followed by room for five [BM] int64 arrays.
// TBN: the tile's column count (the CTA has 2 * TBN threads; the tile's row
// stride in Cs is TBN + 4).
template <typename T, int TBN = BN>
__device__ __noinline__ void simt_epilogue(const SimtParams& p, float* Cs, int64_t o, int64_t s0,
                                           int n0) {
  constexpr int CSLD = TBN + 4, NTE = 2 * TBN;
  const int tid = threadIdx.x;
  const int64_t S_in = p.tok.S_in;
  const int N = p.epi.N;
  const Epilogue& e = p.epi;
  const T* bias = static_cast<const T*>(e.bias);
  const int half = e.rope_half;
  // Per-row output bases, once per tile (rows of a tile are consecutive tokens
  // of one slab): token index into ff, q and k/v buffers, and the position.
  int64_t* row_ff = reinterpret_cast<int64_t*>(Cs + BM * CSLD);  // [BM]
  int64_t* row_q = row_ff + BM;
  int64_t* row_kv = row_q + BM;
  int64_t* row_t = row_kv + BM;
  int64_t* row_kt = row_t + BM;
  const int nkv = e.groups > 0 ? e.groups : e.heads;
  if (tid < BM) {
    const int64_t m = o * S_in + s0 + tid;
    const int64_t bb = m / e.T, t = m - bb * e.T;
    row_ff[tid] = m * e.F;
    row_q[tid] = (bb * e.heads * e.T + t) * e.hd;
    row_kv[tid] = (bb * nkv * e.T + t) * e.hd;
    row_t[tid] = t;
    row_kt[tid] = bb * nkv * e.hd * e.T + t;
  }
  __syncthreads();
  // each thread owns one column of the tile and every other row
  const int c = tid % TBN;
  const int n = n0 + c;
  if (c >= e.bn_eff || n >= N) return;
  const ColInfo ci = decode_col(e, n);
  const float bv = bias ? ld_elem(bias, n) : 0.0f;
  const bool rot = half > 0 && (ci.seg == 1 || ci.seg == 2) && ci.j < 2 * half;
  const bool lo = ci.j < half;
  const int f = lo ? ci.j : ci.j - half;
  const int pc = lo ? c + half : c - half;
  const float pbv = (rot && bias) ? ld_elem(bias, lo ? n + half : n - half) : 0.0f;
  T* const base = static_cast<T*>(out_base(e, ci.seg));
  // pre-transposed k: element (b, head, lane j, token t) at ((b*nkv + head)*hd + j)*T + t
  const bool kt = e.k_transposed && ci.seg == 2;
  const int64_t col_off = ci.seg == 0 ? ci.j
                          : kt        ? (static_cast<int64_t>(ci.head) * e.hd + ci.j) * e.T
                                      : static_cast<int64_t>(ci.head) * e.T * e.hd + ci.j;
  const int64_t* const rb = ci.seg == 0 ? row_ff : ci.seg == 1 ? row_q : kt ? row_kt : row_kv;
  const int64_t tile_rows = S_in - s0;
  // rows in batches of 8: every load of a batch (accumulator, rotation partner,
  // cos/sin) is issued before its stores, so table latency is paid once per batch
  constexpr int kStep = NTE / TBN, kBatch = 8;
  for (int r0 = tid / TBN; r0 < BM; r0 += kStep * kBatch) {
    float v[kBatch], pv[kBatch], cc[kBatch], ss[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int r = r0 + q * kStep;
      const bool in = r < BM && r < tile_rows;
      v[q] = in ? Cs[r * CSLD + c] + bv : 0.0f;
      pv[q] = 0.0f;
      cc[q] = 1.0f;
      ss[q] = 0.0f;
      if (in && rot) {
        pv[q] = Cs[r * CSLD + pc] + pbv;
        if (e.rope_per_lane) {
          const float4 c4 = e.rope_cs4[static_cast<int64_t>(f) * e.T + row_t[r]];
          cc[q] = lo ? c4.x : c4.z;
          ss[q] = lo ? c4.y : c4.w;
        } else {
          const float2 cs = e.rope_cs[static_cast<int64_t>(f) * e.T + row_t[r]];
          cc[q] = cs.x;
          ss[q] = cs.y;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int r = r0 + q * kStep;
      if (r >= BM || r >= tile_rows) break;
      float out = v[q];
      if (ci.seg == 0)
        out = activate(e.act, out);
      else if (rot)
        // rotate-half: lane i gets x_i cos - x_{i+half} sin, lane i+half gets x_{i+half} cos + x_i sin
        out = lo ? out * cc[q] - pv[q] * ss[q] : out * cc[q] + pv[q] * ss[q];
      if (store_in_bounds(e, ci.seg, rb[r] + col_off, 1)) st_elem(base, rb[r] + col_off, out);
    }
  }
}

// T: storage type of x, W, b and the outputs (float, or uint16_t bf16 bits).
template <typename T, bool K_MAJOR>
__global__ void __launch_bounds__(NT, 2) simt_gemm_kernel(const SimtParams p) {
  const T* X = static_cast<const T*>(p.x);
  const T* Wt = static_cast<const T*>(p.W);
  extern __shared__ __align__(16) float smem[];
  float* As = smem;                // [2][BK][BM]
  float* Bs = smem + 2 * BK * BM;  // [2][BK][BN]

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int64_t tile = blockIdx.x;
  const int n_tile = static_cast<int>(tile % p.num_n_tiles);
  const int64_t m_tile = tile / p.num_n_tiles;
  const int64_t o = m_tile / p.m_tiles_per_slab;
  const int64_t s0 = (m_tile - o * p.m_tiles_per_slab) * BM;
  const int n0 = n_tile * p.epi.bn_eff;
  const TokenMap& tk = p.tok;
  const int64_t S_in = tk.S_in;
  const int C = p.C, N = p.epi.N;

  // A element (row m, channel k) of this tile: x[a_base + m*s_stride + k*c_stride]
  //   K_MAJOR:  k = tid % 16 fixed, rows m = tid/16 + 16 i
  //   else:     row m = tid % 128 fixed, channels k = tid/128 + 2 i
  const int a_m0 = K_MAJOR ? tid / BK : tid % BM;
  const int a_k0 = K_MAJOR ? tid % BK : tid / BM;
  const int64_t a_base = outer_offset(tk, o) + (s0 + a_m0) * tk.s_stride;
  const int64_t rows_left = S_in - s0 - a_m0;  // rows with m - a_m0 < rows_left exist

  float a_reg[8], b_reg[8];
  // per-thread operand pointers, advanced by one k-step per call
  const int64_t a_step_i = K_MAJOR ? 16 * tk.s_stride : 2 * tk.c_stride;  // between a thread's 8 loads
  const T* a_ptr = X + a_base + static_cast<int64_t>(a_k0) * tk.c_stride;
  const int b_col = n0 + tid % BN;
  const bool b_col_ok = b_col < N;
  const T* b_ptr = Wt + static_cast<int64_t>(tid / BN) * N + b_col;
  auto load_regs = [&](int k0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int dm = K_MAJOR ? 16 * i : 0;
      const int k = k0 + a_k0 + (K_MAJOR ? 0 : 2 * i);
      a_reg[i] = (dm < rows_left && k < C) ? ld_elem(a_ptr, i * a_step_i) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = k0 + tid / BN + 2 * i;
      b_reg[i] = (b_col_ok && k < C) ? ld_elem(b_ptr, static_cast<int64_t>(2 * i) * N) : 0.0f;
    }
    a_ptr += static_cast<int64_t>(BK) * tk.c_stride;
    b_ptr += static_cast<int64_t>(BK) * N;
  };
  auto store_regs = [&](int buf) {
    float* a = As + buf * BK * BM;
    float* b = Bs + buf * BK * BN;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int m = a_m0 + (K_MAJOR ? 16 * i : 0);
      const int k = a_k0 + (K_MAJOR ? 0 : 2 * i);
      a[k * BM + m] = a_reg[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int idx = tid + i * NT;
      b[(idx / BN) * BN + idx % BN] = b_reg[i];
    }
  };

  // accumulators as packed fp32 pairs along the column index: acc2[i][t] holds
  // columns 2t and 2t+1 of row i. One fma.rn.f32x2 is two IEEE fp32 FMAs (the
  // same results as two scalar ones), so the 8 x 8 outer product of a k-step
  // issues as 32 packed FMAs and 8 splats instead of 64 FMAs: the FMA pipe,
  // not instruction issue, becomes the limit.
  uint64_t acc2[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int t = 0; t < 4; ++t) acc2[i][t] = 0ull;

  const int num_k = (C + BK - 1) / BK;
  load_regs(0);
  store_regs(0);
  __syncthreads();
  for (int kb = 0; kb < num_k; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < num_k) load_regs((kb + 1) * BK);
    const float* a = As + buf * BK * BM;
    const float* b = Bs + buf * BK * BN;
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float4 a0 = *reinterpret_cast<const float4*>(a + kk * BM + ty * 4);
      float4 a1 = *reinterpret_cast<const float4*>(a + kk * BM + 64 + ty * 4);
      float4 b0 = *reinterpret_cast<const float4*>(b + kk * BN + tx * 4);
      float4 b1 = *reinterpret_cast<const float4*>(b + kk * BN + 64 + tx * 4);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const uint64_t bv2[4] = {f2_pack(b0.x, b0.y), f2_pack(b0.z, b0.w), f2_pack(b1.x, b1.y),
                               f2_pack(b1.z, b1.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint64_t ai = f2_splat(av[i]);
#pragma unroll
        for (int t = 0; t < 4; ++t) acc2[i][t] = f2_fma(ai, bv2[t], acc2[i][t]);
      }
    }
    if (kb + 1 < num_k) store_regs(buf ^ 1);
    __syncthreads();
  }

  // ---- epilogue: stage the fp32 tile, then bias / activation / rotation / scatter
  float* Cs = smem;  // [BM][CS_LD]
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int r = (i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4);
    float c[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) f2_unpack(acc2[i][t], c[2 * t], c[2 * t + 1]);
    *reinterpret_cast<float4*>(Cs + r * CS_LD + tx * 4) = make_float4(c[0], c[1], c[2], c[3]);
    *reinterpret_cast<float4*>(Cs + r * CS_LD + 64 + tx * 4) = make_float4(c[4], c[5], c[6], c[7]);
  }
  __syncthreads();

  simt_epilogue<T>(p, Cs, o, s0, n0);
}

// ---- fp32 storage with unit-stride tokens (channels-first x, e.g. NCHW): the
// operand tiles are copied global -> shared by cp.async in 16-byte chunks (4
// tokens of one channel; 4 columns of one weight row), so no thread stages
// operands through registers. Chunks past the last token, channel or column
// are zero-filled by the copy's source size.
//
// Two tile widths, 8x8 register blocks either way (16 row groups x TBN / 8
// column groups of threads):
//  * TBN 128: 256 threads, 2 CTAs per SM, k-steps of 32 with three in flight;
//  * TBN 64: 128 threads, 4 CTAs per SM, k-steps of 32 double-buffered. Twice
//    as many tiles for the same work: the launcher takes it when that spreads
//    the work more evenly over the SMs (a smaller largest per-SM share).
// Row-major x with unit-stride channels (AK, K-major A) takes the same loop
// with A held per token: [BM][SK + 4] (the 4-float pad spreads the rows over
// the banks), copied as 4 channels of one token per chunk. A thread then owns
// rows ty + 16 i, and one 8-byte load per row gives two k-steps.
template <int TBN, bool AK>
struct AsyncTile {
  static constexpr int NT = 2 * TBN;
  static constexpr int SK = 32;
  static constexpr int SKP = SK + 4;  // A row stride when K-major
  static constexpr int STAGES = TBN == 128 ? 3 : 2;
  static constexpr int MIN_BLOCKS = TBN == 128 ? 2 : 4;
  static constexpr int CSLD = TBN + 4;
  static constexpr int A_CHUNKS = SK * BM / 4 / NT;   // 16-byte chunks per thread per stage
  static constexpr int B_CHUNKS = SK * TBN / 4 / NT;
  static constexpr int A_STAGE = AK ? BM * SKP : SK * BM;  // floats
  static constexpr int STAGE_BYTES = STAGES * (A_STAGE + SK * TBN) * 4;
  static constexpr int EPI_BYTES = BM * CSLD * 4 + 5 * BM * 8;
  static constexpr int SMEM = STAGE_BYTES > EPI_BYTES ? STAGE_BYTES : EPI_BYTES;
  static_assert(A_CHUNKS * NT * 4 == SK * BM && B_CHUNKS * NT * 4 == SK * TBN, "chunk split");
};

__device__ __forceinline__ void cp_async16(float* dst, const float* src, int src_bytes) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int TBN, bool AK>
__global__ void __launch_bounds__(AsyncTile<TBN, AK>::NT, AsyncTile<TBN, AK>::MIN_BLOCKS)
    simt_gemm_async_kernel(const SimtParams p) {
  using Cfg = AsyncTile<TBN, AK>;
  constexpr int SK = Cfg::SK, STAGES = Cfg::STAGES, NTH = Cfg::NT, CSLD = Cfg::CSLD;
  constexpr int HALF = TBN / 2;  // a thread's second column group starts here
  const float* X = static_cast<const float*>(p.x);
  const float* Wt = static_cast<const float*>(p.W);
  extern __shared__ __align__(16) float smem[];
  constexpr int SKP = Cfg::SKP;
  float* As = smem;                       // [stage][SK][BM], K-major: [stage][BM][SKP]
  float* Bs = smem + STAGES * Cfg::A_STAGE;  // [stage][SK][TBN]

  const int tid = threadIdx.x;
  const int tx = tid % (TBN / 8), ty = tid / (TBN / 8);
  const int64_t tile = blockIdx.x;
  const int n_tile = static_cast<int>(tile % p.num_n_tiles);
  const int64_t m_tile = tile / p.num_n_tiles;
  const int64_t o = m_tile / p.m_tiles_per_slab;
  const int64_t s0 = (m_tile - o * p.m_tiles_per_slab) * BM;
  const int n0 = n_tile * p.epi.bn_eff;
  const TokenMap& tk = p.tok;
  const int C = p.C, N = p.epi.N;
  // accumulator row i of this thread within the tile
  auto row_of = [&](int i) { return AK ? ty + 16 * i : (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4)); };

  // This thread's chunks per stage. A: chunk c = tid + NTH j covers k-row
  // c / 32 (= ak + (NTH / 32) j) and tokens 4 (c % 32) .. + 3. B likewise with
  // TBN / 4 chunks per k-row.
  constexpr int A_ROW_CH = BM / 4, B_ROW_CH = TBN / 4;
  constexpr int A_DK = NTH / A_ROW_CH, B_DK = NTH / B_ROW_CH;  // k-rows between a thread's chunks
  const int ak = tid / A_ROW_CH, ae = (tid % A_ROW_CH) * 4;
  const int bk = tid / B_ROW_CH, be = (tid % B_ROW_CH) * 4;
  const int64_t rows_left = tk.S_in - s0 - ae;
  const int a_bytes = rows_left >= 4 ? 16 : rows_left > 0 ? static_cast<int>(rows_left) * 4 : 0;
  const int b_bytes = n0 + be < N ? 16 : 0;  // N is a multiple of 4
  const float* a_src = X + outer_offset(tk, o) + s0 + ae + static_cast<int64_t>(ak) * tk.c_stride;
  const float* b_src = Wt + static_cast<int64_t>(bk) * N + n0 + be;
  // K-major A: chunk c = tid + NTH j covers token row c / (SK / 4) (= kr +
  // (NTH * 4 / SK) j) and channels 4 (c % (SK / 4)) .. + 3 of the k-step
  constexpr int K_ROW_CH = SK / 4, K_DR = NTH / K_ROW_CH;
  const int kr = tid / K_ROW_CH, kq = (tid % K_ROW_CH) * 4;
  const float* ak_src = X + outer_offset(tk, o) + (s0 + kr) * tk.s_stride + kq;
  const int64_t ak_step = K_DR * tk.s_stride;     // between a thread's chunks
  const int64_t ak_rows = tk.S_in - s0 - kr;      // its chunk j exists while K_DR j < ak_rows
  auto issue = [&](int kb) {
    const int st = kb % STAGES;
    float* b = Bs + st * SK * TBN + bk * TBN + be;
    const int k0 = kb * SK;
    const int64_t kw = static_cast<int64_t>(k0) * N;
    if constexpr (AK) {
      float* a = As + st * Cfg::A_STAGE + kr * SKP + kq;
      const int k_left = C - k0 - kq;
      const int kbytes = k_left >= 4 ? 16 : k_left > 0 ? 4 * k_left : 0;
      const float* src = ak_src + k0;
#pragma unroll
      for (int j = 0; j < Cfg::A_CHUNKS; ++j) {
        const bool in = K_DR * j < ak_rows && kbytes > 0;
        cp_async16(a + j * K_DR * SKP, in ? src : X, in ? kbytes : 0);
        src += ak_step;
      }
    } else {
      float* a = As + st * SK * BM + ak * BM + ae;
      const int64_t ka = static_cast<int64_t>(k0) * tk.c_stride;
#pragma unroll
      for (int j = 0; j < Cfg::A_CHUNKS; ++j) {
        const bool in = k0 + ak + A_DK * j < C;
        cp_async16(a + j * A_DK * BM,
                   in ? a_src + ka + static_cast<int64_t>(j) * A_DK * tk.c_stride : X,
                   in ? a_bytes : 0);
      }
    }
#pragma unroll
    for (int j = 0; j < Cfg::B_CHUNKS; ++j) {
      const bool in = k0 + bk + B_DK * j < C;
      cp_async16(b + j * B_DK * TBN, in ? b_src + kw + static_cast<int64_t>(j) * B_DK * N : Wt,
                 in ? b_bytes : 0);
    }
  };

  uint64_t acc2[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int t = 0; t < 4; ++t) acc2[i][t] = 0ull;

  const int num_k = (C + SK - 1) / SK;
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < num_k) issue(s);
    cp_async_commit();
  }
  for (int kb = 0; kb < num_k; ++kb) {
    // this thread's copies of step kb have landed; the barrier publishes every
    // thread's and retires step kb - 1, whose stage the next issue refills
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    if (kb + STAGES - 1 < num_k) issue(kb + STAGES - 1);
    cp_async_commit();
    const int st = kb % STAGES;
    const float* a = As + st * Cfg::A_STAGE;
    const float* b = Bs + st * SK * TBN;
    if constexpr (AK) {
      // two k-steps per pass: one 8-byte load per owned row, B for both steps
#pragma unroll 2
      for (int kk = 0; kk < SK; kk += 2) {
        float2 a2[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          a2[i] = *reinterpret_cast<const float2*>(a + row_of(i) * SKP + kk);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float4 b0 = *reinterpret_cast<const float4*>(b + (kk + h) * TBN + tx * 4);
          const float4 b1 = *reinterpret_cast<const float4*>(b + (kk + h) * TBN + HALF + tx * 4);
          const uint64_t bv2[4] = {f2_pack(b0.x, b0.y), f2_pack(b0.z, b0.w), f2_pack(b1.x, b1.y),
                                   f2_pack(b1.z, b1.w)};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint64_t ai = f2_splat(h ? a2[i].y : a2[i].x);
#pragma unroll
            for (int t = 0; t < 4; ++t) acc2[i][t] = f2_fma(ai, bv2[t], acc2[i][t]);
          }
        }
      }
      continue;
    }
    // fragments double-buffered in registers: step kk + 1's loads are issued
    // before step kk's FMAs
    float4 fa[2][2], fb[2][2];
    fa[0][0] = *reinterpret_cast<const float4*>(a + ty * 4);
    fa[0][1] = *reinterpret_cast<const float4*>(a + 64 + ty * 4);
    fb[0][0] = *reinterpret_cast<const float4*>(b + tx * 4);
    fb[0][1] = *reinterpret_cast<const float4*>(b + HALF + tx * 4);
#pragma unroll
    for (int kk = 0; kk < SK; ++kk) {
      const int cur = kk & 1, nxt = cur ^ 1;
      if (kk + 1 < SK) {
        fa[nxt][0] = *reinterpret_cast<const float4*>(a + (kk + 1) * BM + ty * 4);
        fa[nxt][1] = *reinterpret_cast<const float4*>(a + (kk + 1) * BM + 64 + ty * 4);
        fb[nxt][0] = *reinterpret_cast<const float4*>(b + (kk + 1) * TBN + tx * 4);
        fb[nxt][1] = *reinterpret_cast<const float4*>(b + (kk + 1) * TBN + HALF + tx * 4);
      }
      const float4 a0 = fa[cur][0], a1 = fa[cur][1], b0 = fb[cur][0], b1 = fb[cur][1];
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const uint64_t bv2[4] = {f2_pack(b0.x, b0.y), f2_pack(b0.z, b0.w), f2_pack(b1.x, b1.y),
                               f2_pack(b1.z, b1.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint64_t ai = f2_splat(av[i]);
#pragma unroll
        for (int t = 0; t < 4; ++t) acc2[i][t] = f2_fma(ai, bv2[t], acc2[i][t]);
      }
    }
  }
  cp_async_wait<0>();  // only empty groups remain; the epilogue overlays the stages
  __syncthreads();

  const Epilogue& e = p.epi;
  if (e.rope_half == 0 && !e.k_transposed && (e.heads == 0 || e.hd % 4 == 0)) {
    // No rotation pairs and no transposed k: each thread stores its own 8 x 8
    // block from registers, 4 consecutive columns (one head, F and hd being
    // multiples of 4) per 16-byte store. Per-row output bases come from shared
    // memory, once per tile.
    int64_t* row_ff = reinterpret_cast<int64_t*>(smem);  // [BM]
    int64_t* row_q = row_ff + BM;
    int64_t* row_kv = row_q + BM;
    const int nkv = e.groups > 0 ? e.groups : e.heads;
    for (int r = tid; r < BM; r += NTH) {
      const int64_t m = o * tk.S_in + s0 + r;
      const int64_t bb = m / e.T, t = m - bb * e.T;
      row_ff[r] = m * e.F;
      row_q[r] = (bb * e.heads * e.T + t) * e.hd;
      row_kv[r] = (bb * nkv * e.T + t) * e.hd;
    }
    __syncthreads();
    const float* bias = static_cast<const float*>(e.bias);
    const int64_t tile_rows = tk.S_in - s0;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int c0 = h2 * HALF + tx * 4;
      const int n = n0 + c0;
      if (c0 >= e.bn_eff || n >= N) continue;
      const ColInfo ci = decode_col(e, n);
      const float4 bv = bias ? *reinterpret_cast<const float4*>(bias + n) : make_float4(0, 0, 0, 0);
      float* const base = static_cast<float*>(out_base(e, ci.seg));
      const int64_t col_off =
          ci.seg == 0 ? ci.j : static_cast<int64_t>(ci.head) * e.T * e.hd + ci.j;
      const int64_t* const rb = ci.seg == 0 ? row_ff : ci.seg == 1 ? row_q : row_kv;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = row_of(i);
        if (r >= tile_rows) continue;
        float4 v;
        f2_unpack(acc2[i][2 * h2], v.x, v.y);
        f2_unpack(acc2[i][2 * h2 + 1], v.z, v.w);
        v.x += bv.x;
        v.y += bv.y;
        v.z += bv.z;
        v.w += bv.w;
        if (ci.seg == 0) {
          v.x = activate(e.act, v.x);
          v.y = activate(e.act, v.y);
          v.z = activate(e.act, v.z);
          v.w = activate(e.act, v.w);
        }
        const int64_t off = rb[r] + col_off;
        if (store_in_bounds(e, ci.seg, off, 4)) *reinterpret_cast<float4*>(base + off) = v;
      }
    }
    return;
  }

  float* Cs = smem;  // [BM][CSLD]
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = row_of(i);
    float c[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) f2_unpack(acc2[i][t], c[2 * t], c[2 * t + 1]);
    *reinterpret_cast<float4*>(Cs + r * CSLD + tx * 4) = make_float4(c[0], c[1], c[2], c[3]);
    *reinterpret_cast<float4*>(Cs + r * CSLD + HALF + tx * 4) = make_float4(c[4], c[5], c[6], c[7]);
  }
  __syncthreads();

  simt_epilogue<float, TBN>(p, Cs, o, s0, n0);
}

// The cp.async kernel's preconditions: fp32 storage and every chunk 16-byte
// aligned (x and W 16-byte aligned; every outer stride and N multiples of 4
// elements; tiles start at multiples of 128 tokens and columns n0 multiples
// of 4), with either unit-stride tokens and a channel stride that is a
// multiple of 4 (returns 1: MN-major A) or unit-stride channels and a token
// stride that is a multiple of 4 (returns 2: K-major A); else 0.
int async_form(const SimtParams& p) {
  const TokenMap& tk = p.tok;
  if (p.epi.N % 4 != 0 || p.epi.bn_eff % 4 != 0) return 0;
  if (reinterpret_cast<uintptr_t>(p.x) % 16 != 0 || reinterpret_cast<uintptr_t>(p.W) % 16 != 0)
    return 0;
  for (int d = 0; d < tk.n_outer_dims; ++d)
    if (tk.outer_stride[d] % 4 != 0) return 0;
  if (tk.s_stride == 1 && tk.c_stride % 4 == 0) return 1;
  if (tk.c_stride == 1 && tk.s_stride % 4 == 0) return 2;
  return 0;
}

template <int TBN, bool AK>
cudaError_t launch_async_tiles(const SimtParams& p, int dev, cudaStream_t stream) {
  using Cfg = AsyncTile<TBN, AK>;
  static int attr_done[64] = {0};
  if (dev >= 64 || !attr_done[dev]) {
    cudaError_t err = cudaFuncSetAttribute(simt_gemm_async_kernel<TBN, AK>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (err != cudaSuccess) return err;
    if (dev < 64) attr_done[dev] = 1;
  }
  const int64_t tiles = p.num_m_tiles * p.num_n_tiles;
  simt_gemm_async_kernel<TBN, AK><<<static_cast<unsigned>(tiles), Cfg::NT, Cfg::SMEM, stream>>>(p);
  return cudaGetLastError();
}

// Tile width: 64 columns when that lowers the largest per-SM share of the work
// (in 128 x 128 tile units, with tiles dealt evenly over the SMs), else 128.
// Narrow tiles need an N-tile of whole heads under rotation (head_dim <= 64).
template <bool AK>
cudaError_t launch_async(const SimtParams& p, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const Epilogue& e = p.epi;
  const int half = e.rope_half > 0;
  const int bn_narrow = half ? (64 / e.hd) * e.hd : 64;
  if (bn_narrow > 0 && bn_narrow % 4 == 0 && sms > 0) {
    const int64_t n_narrow = (e.N + bn_narrow - 1) / bn_narrow;
    const int64_t wide = p.num_m_tiles * p.num_n_tiles, narrow = p.num_m_tiles * n_narrow;
    const int64_t share_wide = 2 * ((wide + sms - 1) / sms);  // in half-tile units
    const int64_t share_narrow = (narrow + sms - 1) / sms;
    if (share_narrow < share_wide) {
      SimtParams q = p;
      q.epi.bn_eff = bn_narrow;
      q.num_n_tiles = static_cast<int>(n_narrow);
      return launch_async_tiles<64, AK>(q, dev, stream);
    }
  }
  return launch_async_tiles<128, AK>(p, dev, stream);
}

template <typename T, bool K_MAJOR>
cudaError_t launch_one(const SimtParams& p, int64_t tiles, cudaStream_t stream) {
  static int attr_done[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !attr_done[dev]) {
    err = cudaFuncSetAttribute(simt_gemm_kernel<T, K_MAJOR>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    if (dev < 64) attr_done[dev] = 1;
  }
  simt_gemm_kernel<T, K_MAJOR><<<static_cast<unsigned>(tiles), NT, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtParams& p, bool bf16, cudaStream_t stream) {
  int64_t tiles = p.num_m_tiles * p.num_n_tiles;
  if (tiles == 0) return cudaSuccess;
  const bool k_major = p.tok.c_stride == 1;
  const int form = bf16 ? 0 : async_form(p);
  if (form == 1) return launch_async<false>(p, stream);
  if (form == 2) return launch_async<true>(p, stream);
  if (bf16)
    return k_major ? launch_one<uint16_t, true>(p, tiles, stream)
                   : launch_one<uint16_t, false>(p, tiles, stream);
  return k_major ? launch_one<float, true>(p, tiles, stream)
                 : launch_one<float, false>(p, tiles, stream);
}

}  // namespace fp
