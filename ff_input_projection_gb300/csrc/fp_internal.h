// Internal kernel parameter blocks and launchers of libfp (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp {

constexpr int kMaxOuter = 6;

enum : int { ACT_NONE = 0, ACT_GELU_ERF = 1, ACT_GELU_TANH = 2, ACT_SILU = 3, ACT_RELU2 = 4 };
enum : int { ST_OK = 0, ST_TIMEOUT = 6, ST_BOUNDS = 7 };

// Token addressing shared by both GEMM kernels. The non-channel axes of x are
// merged where contiguous; the innermost merged group is `S_in` tokens at
// stride `s_stride`, the others are `n_outer_dims` outer axes. Token
// m = o*S_in + s, o = row-major index over the outer axes. M-tiles never cross
// an outer index, so rows in one tile are `s`-consecutive.
struct TokenMap {
  int64_t S_in;
  int64_t s_stride;
  int64_t c_stride;
  int64_t n_outer;  // product of outer sizes
  int n_outer_dims;
  int64_t outer_size[kMaxOuter];    // innermost first
  int64_t outer_stride[kMaxOuter];  // innermost first
};

// Epilogue description shared by both GEMM kernels.
struct Epilogue {
  int64_t M;  // tokens
  int64_t T;  // tokens per batch element
  int N, F, C, heads, hd, groups;  // groups > 0: grouped-query column order
  int act;
  int rope_half;      // 0: no rotation, else rotated lanes / 2
  // rotary tables, frequency-major: entry (i, t) at i * T + t
  const float2* rope_cs;  // [rope_half][T] (cos, sin) of theta_i, shared by lanes i and i+half
  const float4* rope_cs4; // per-lane tables: [rope_half][T] (cos_i, sin_i, cos_i+h, sin_i+h)
  int rope_per_lane;      // 1: use rope_cs4
  const void* bias;   // [N] or null, dtype of x
  void* out_ff;
  void* out_q;
  void* out_k;
  void* out_v;
  int* status;
  int bn_eff;         // columns of an N-tile that this tile owns
  int k_transposed;   // 1: k is written [B*kv, hd, T]
  int64_t ff_ld;      // row stride of out_ff (F; N when out_ff is the backward's G)
  // backward ff gradient (tensor-core kernel, grad mode): out_ff receives
  // g_ff * act'(x W + b) instead of act(x W + b), its column sums go to db
  const void* g_ff;   // [M, F] upstream gradient, dtype of x
  float* db;          // [N] or null
  // opt-in check of every directly addressed output store (stores by TMA are
  // confined to their tensor map): the element extents of out_ff, out_q,
  // out_k, out_v. A store that would leave its buffer is skipped and recorded
  // as ST_BOUNDS in the status word.
  int bounds_check;
  int64_t extent[4];
};

struct TcParams {
  CUtensorMap tmap_a;
  CUtensorMap tmap_b;
  // output maps for TMA stores: ff [M, F] (2-D), q/k/v [B*heads, T, hd] (3-D)
  // (ff twice: 16-column boxes, and 32-column boxes for tiles inside the ff block)
  CUtensorMap tmap_ff, tmap_ff32, tmap_q, tmap_k, tmap_v;
  // bias [N] as a 1-row 2-D map (64-column boxes), when there is a bias
  CUtensorMap tmap_bias;
  int tma_store;  // 1: the output maps are valid
  // 1: the MN-major x map views each slab's tokens as (64 inside a block,
  // S_in/64 blocks), so one box loads both 64-token chunks of a stage
  int a_split;
  // N of the MMAs: 256, or 192 when tiles of 192 columns fill the waves of CTA
  // pairs better (0 reads as 256). Each CTA of a pair then holds bn_mma / 2
  // columns, from column n0 + rank * bn_mma / 2, in its two 64-column chunks.
  int bn_mma;
  TokenMap tok;
  Epilogue epi;
  int C;
  int num_k_blocks;
  int64_t m_tiles_per_slab;
  int64_t num_m_tiles;
  int num_n_tiles;
  int64_t num_tiles;
  int cluster;        // CTAs per cluster sharing one W tile (1 or 2)
  int64_t num_units;  // work items: (M-tile group of `cluster`, N-tile) pairs
  int group_m;
  uint64_t wait_limit_ns;
  int inject_stall;  // 1: CTA 0 withholds its first operand stage (error-path test)
  int launch_tag;    // >= 1, unique per launch: marks this launch as aborted in status[1]
};

// Backward GEMMs on the tensor cores (gemm_bwd.cu). G is the gradient at the
// pre-activation, pre-rotation fused output, [M, N] bf16 (workspace), viewed
// as [n_outer][S_in][N].
enum : int {
  BWD_GRADFF = 0,  // G[:, :F] = g_ff * act'(x W_ff + b_ff): rows tokens, K = C
  BWD_DX = 1,      // dx = G W^T for token-major x: rows tokens, cols channels, K = N
  BWD_DXT = 2,     // dx^T = W G^T for channels-first x: rows channels, cols tokens, K = N
  BWD_DW = 3,      // dW += X^T G (fp32, split over tokens): rows channels, cols N, K = tokens
};

struct BwdGemmParams {
  CUtensorMap tmap_a, tmap_b, tmap_out;
  TokenMap tok;             // token axes of x (S_in, outer axes)
  int mode;
  int num_m_tiles;          // row tiles (tokens: n_outer * m_tiles_per_slab; channels: C/128)
  int m_tiles_per_slab;     // row tiles per slab when rows are tokens
  int num_n_tiles;          // column tiles (tokens: n_outer * n_tiles_per_slab)
  int n_tiles_per_slab;     // column tiles per slab when columns are tokens
  int num_k_blocks;         // k-blocks of 64 (DW: all token blocks over all slabs)
  int k_blocks_per_slab;    // DW: ceil(S_in / 64)
  int k_splits;             // DW: the token range is split this many ways
  int64_t num_units;        // work items: (row-tile group of `cluster`, column tile, k split)
  int cluster;              // CTAs per cluster sharing one B tile (1; 2 for DX/DXT)
  int group_m;
  int C, F, N, act;
  const void* bias;         // GRADFF: [N] bf16 or null
  const void* g_ff;         // GRADFF: [M, F] bf16
  float* db;                // GRADFF: [N] fp32 column sums, or null
  int* status;
  uint64_t wait_limit_ns;
  int launch_tag;
};

// Gather of the q/k/v gradients into G (inverse rotation), with db column sums.
struct BwdGatherParams {
  const void* g_q;
  const void* g_k;
  const void* g_v;
  void* G;                  // [M, N] bf16
  float* db;                // [N] or null
  const float2* rope_cs;    // [rope_half][T] (cos, sin), frequency-major, or null
  int64_t M, T;
  int F, N, C, heads, hd, groups, rope_half, k_transposed;
};

struct SimtParams {
  const void* x;  // float, or bf16 bits
  const void* W;
  TokenMap tok;
  Epilogue epi;
  int C;
  int64_t m_tiles_per_slab;
  int64_t num_m_tiles;
  int num_n_tiles;
};

// Softmax attention over the projection's outputs (attention.cu): q [BH, Tq, hd],
// k [BHkv, Tk, hd] or pre-transposed [BHkv, hd, Tk], v [BHkv, Tk, hd], out
// [BH, Tq, hd], bf16; BH = batch * heads, BHkv = batch * kv_heads.
struct AttnParams {
  CUtensorMap tmap_q, tmap_k, tmap_v;
  void* out;
  int64_t Tq, Tk;
  int BH, hd, heads, kv_heads, k_transposed;
  int num_q_blocks;     // ceil(Tq / 128)
  float scale_log2e;    // softmax scale times log2(e): exp(s * scale) = 2^(s * scale_log2e)
  int* status;
  uint64_t wait_limit_ns;
  int launch_tag;
  // Query blocks (BH * num_q_blocks of them, in (z, block) order) are split
  // between whole blocks and a split tail: the first `full` run over all keys
  // in one CTA each; each remaining block is spread over `splits` CTAs, one
  // contiguous range of key chunks each, which write unnormalised fp32 partial
  // results to `part` ([tail block][split] slots of 128 x (hd + 2) floats:
  // O rows, then m, then l, m in log2 units) for the merge kernel.
  int full, splits;
  float* part;
};

// How a launch spreads its query blocks over the SMs: the blocks past the
// last whole wave are split along the keys when that fills the wave better.
struct AttnSplit {
  int full, tail, splits;
  int64_t part_bytes;  // partial-result scratch the split tail needs (0 when none)
};
AttnSplit attention_split(int64_t q_blocks, int64_t Tk, int hd, int sms);

// Launchers (defined in the .cu files). Return cudaSuccess or the launch error.
cudaError_t launch_rope_table(float2* cs, const int32_t* pos, int64_t T, int half, int n_elem,
                              double rope_base, cudaStream_t stream);
cudaError_t launch_rope_import(float4* dst, const void* cosv, const void* sinv, bool bf16,
                               int64_t T, int half, int64_t stride_t, int64_t stride_i,
                               cudaStream_t stream);
cudaError_t launch_tc_gemm(const TcParams& p, bool a_mn_major, int num_ctas, cudaStream_t stream,
                           bool grad = false);
cudaError_t launch_simt_gemm(const SimtParams& p, bool bf16, cudaStream_t stream);
cudaError_t launch_bwd_gemm(const BwdGemmParams& p, bool a_mn_major, int num_ctas,
                            cudaStream_t stream);
cudaError_t launch_bwd_gather(const BwdGatherParams& p, cudaStream_t stream);
// One launch, or two when the tail is split (the second merges the partials);
// *launches receives the count.
cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream, int* launches);

constexpr int kTcBM = 128, kTcBN = 256, kTcBK = 64;
constexpr int kSimtBM = 128, kSimtBN = 128;

}  // namespace fp
