// bf16 fused projection on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: Y = x W + b for a strided activation x read in place
// (Walrus PR #12 "Make fused_ff_qkv contiguous": one GEMM over all tokens
// instead of per-token GEMVs, and no permuted copy), then in the epilogue the
// activation on the ff block (xformers PR #283 "[perf] Fused linear": w x + b
// then the activation, fused), the rotate-half rotary embedding on q and k
// (nvFuser issue #1597 "Improve performance on RoPE", rope_one_entry, with no
// slice/cat/neg kernels), and the split into ff [M, F] and head-major
// q/k/v [B*heads, T, head_dim] (memory-efficient-attention issue #7, the
// [batch*heads, tokens, head_dim] layout).
//
// Structure (one persistent CTA per SM, 10 warps; CTA pairs by default):
//   warp 0     TMA producer: loads x and W tiles into a shared ring (5 stages
//              of 32 KB in a pair, 3 of 48 KB alone), and each tile's bias
//              row into a bias operand
//   warp 1     allocates 512 TMEM columns; in the even CTA one thread issues
//              tcgen05.mma (2-SM M=256 or 1-SM M=128; N=256, K=16, bf16 in,
//              fp32 accumulate) and commits completion to mbarriers
//   warps 2-9  epilogue: tcgen05.ld of the fp32 accumulator (one token row
//              per thread), activation / rotation in registers, bf16
//              round-to-nearest-even, TMA tensor stores of 32 x 32 (ff) and
//              32 x 16 (q/k/v) blocks
// The accumulator is double-buffered in TMEM (2 x 256 columns), so the
// epilogue of tile i overlaps the main loop of tile i+1. In its gradient mode
// the same kernel computes the backward's ff part, g_ff * act'(x W + b), with
// column sums into db.
//
// The bias enters through the tensor core: each tile starts with one K=16 MMA
// (accumulate off) whose A operand is a constant atom with 0.5 in k-row 0 and
// zeros elsewhere, and whose B operand holds the tile's bias in k-row 0. Both
// descriptors give the second 8-row k group a stride of 0, so it reads the
// same atom again: every accumulator starts at 0.5 b + 0.5 b = b exactly, and
// the epilogue has no bias loads or adds.
//
// Operand layouts (128-byte swizzle, as written by TMA and read by the MMA):
//   A, row-major x (unit channel stride): K-major, [128 rows][64 ch] per stage.
//   A, channels-first x (unit token stride): MN-major, two [64 ch][64 tok] chunks
//      (one TMA box of [2][64][64] when the slab length is a multiple of 64).
//   B, W [C, N] row-major: MN-major (N contiguous), four [64 ch][64 col] chunks.
//
// Every mbarrier wait is bounded (%globaltimer); a wait that runs out records
// a timeout in the plan's status word, tags the launch as aborted so the other
// roles and CTAs stop too, drains its own in-flight copies and MMAs, frees
// TMEM and returns.
#include "epilogue.cuh"
#include "fp_internal.h"
#include "tc_ptx.cuh"

namespace fp {
namespace {

constexpr int BM = kTcBM, BN = kTcBN, BK = kTcBK;
constexpr int UMMA_K = 16;
// Epilogue warps per SM sub-partition, each reading one TMEM lane quarter.
// Forward: two per quarter (168 registers each) measured faster than three
// (128 registers) on every bf16 workload and one (184) slower: the epilogue
// keeps up with the main loop, and fewer warps put fewer stores in flight
// beside the MMAs. The backward's ff-gradient mode (upstream-gradient loads,
// act', column sums) keeps three: with two it measured 2 % slower.
template <bool GRAD>
struct Warps {
  static constexpr int EPQ = GRAD ? 3 : 2;
  static constexpr int EPI = 4 * EPQ;
  static constexpr int NT = 32 * (2 + EPI);
  static constexpr int REGS = GRAD ? 128 : 168;
  // registers are granted per 4 warps (10 warps count as 12, 14 as 16)
  static_assert(((NT / 32 + 3) / 4 * 4) * 32 * REGS <= 65536, "register budget");
};
constexpr int A_BYTES = BM * BK * 2;             // 16 KB: this CTA's 128 token rows
constexpr int CHUNK_BYTES = 64 * BK * 2;         // one [64 ch][64 elems] MN-major chunk, 8 KB
constexpr int ACC_COLS = BN;                     // fp32 accumulator: one TMEM column per output column
constexpr int TMEM_COLS = 2 * ACC_COLS;          // 512: two accumulators
// bias operands: A, two [8 k][64 m] MN-major atoms (k-row 0 = 0.5); B, one
// [8 k][64 n] atom per 64 W columns held, k-row 0 = the tile's bias
constexpr int BIAS_A_BYTES = 2 * 1024;
// per epilogue warp, two 2 KB buffers staging a [32 rows][32 bf16] block (ff)
// or a [32 rows][16 bf16] block (q/k/v, mixed tiles) for a TMA store
constexpr int STAGING_BYTES_PER_WARP = 2 * 2048;
static_assert(TMEM_COLS == 512, "TMEM holds 512 columns");

// Per cluster size: a single CTA holds all 256 W columns of its tile; a CTA
// pair runs 2-SM MMAs (M = 256), each CTA holding its own 128 token rows and
// its own 128 of the 256 W columns, so a stage is 32 KB instead of 48 KB.
template <int CL, int EPI>
struct Cfg {
  static constexpr int STAGING_BYTES = EPI * STAGING_BYTES_PER_WARP;
  static constexpr int B_COLS = BN / CL;
  static constexpr int B_BYTES = B_COLS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = CL == 2 ? 5 : 3;
  static constexpr int BIAS_B_BYTES = (B_COLS / 64) * 1024;
  // full and empty per stage; two accumulators full/empty; drain; bias full, empty
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 1 + 2;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BIAS_A_BYTES + BIAS_B_BYTES +
                                    STAGING_BYTES + NUM_BARS * 8 + 16;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// ------------------------------------------------------------------ tile helpers

struct TileCoord {
  int64_t o;     // outer slab
  int64_t s0;    // first token of the tile inside the slab
  int n0;        // first fused column
  bool phantom;  // M-tile past the end (odd M-tile count in a CTA pair): compute, store nothing
};

// Work item `unit` -> this CTA's tile. A cluster of CL CTAs takes CL
// consecutive M-tiles with the same N-tile (they share its W tile). Groups of
// group_m M-tiles sweep all N-tiles, M fastest inside a group, so concurrently
// running clusters share W and x tiles in L2.
template <int CL>
__device__ __forceinline__ TileCoord tile_coord(const TcParams& p, int64_t unit64, int rank) {
  // tile counts fit in 31 bits (the host checks), so the index arithmetic is 32-bit
  const uint32_t unit = static_cast<uint32_t>(unit64);
  const uint32_t m_units = (static_cast<uint32_t>(p.num_m_tiles) + CL - 1) / CL;
  const uint32_t gsz = p.group_m >= CL ? static_cast<uint32_t>(p.group_m) / CL : 1u;
  const uint32_t per_group = gsz * static_cast<uint32_t>(p.num_n_tiles);
  const uint32_t g = unit / per_group;
  const uint32_t first = g * gsz;
  const uint32_t left = m_units - first;
  const uint32_t gm = left < gsz ? left : gsz;
  const uint32_t r = unit - g * per_group;
  const uint32_t rn = r / gm;
  const uint32_t m_tile = (first + (r - rn * gm)) * CL + rank;
  TileCoord tc;
  tc.phantom = m_tile >= static_cast<uint32_t>(p.num_m_tiles);
  const uint32_t mt = tc.phantom ? static_cast<uint32_t>(p.num_m_tiles) - 1 : m_tile;
  const uint32_t per_slab = static_cast<uint32_t>(p.m_tiles_per_slab);
  const uint32_t o = mt / per_slab;
  tc.o = o;
  tc.s0 = static_cast<int64_t>(mt - o * per_slab) * BM;
  tc.n0 = static_cast<int>(rn) * p.epi.bn_eff;
  return tc;
}

// 16 bf16 values (two per word) at stride `stride` elements: a head's lane
// column of pre-transposed k.
__device__ __forceinline__ void store16_packed_strided(uint16_t* dst, int64_t stride,
                                                       const uint32_t (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    dst[(2 * i) * stride] = static_cast<uint16_t>(w[i] & 0xFFFFu);
    dst[(2 * i + 1) * stride] = static_cast<uint16_t>(w[i] >> 16);
  }
}

// Rotation of lanes [0, 2*RH) of a head held in one 16-column granule (partial
// rotary, rope_n_elem = 2*RH <= 16): pair (i, i + RH) with (cos, sin) of
// frequency i. cs points at the token's entry of frequency 0 of the
// frequency-major table; frequency i is T entries further.
template <int RH>
__device__ __forceinline__ void rotate_in_granule(float (&v)[16], const float2* __restrict__ cs,
                                                  int64_t T) {
#pragma unroll
  for (int i = 0; i < RH; ++i) {
    const float2 c = __ldg(cs + i * T);
    const float x = v[i], y = v[i + RH];
    v[i] = x * c.x - y * c.y;
    v[i + RH] = y * c.x + x * c.y;
  }
}

// Per-lane tables: lane i uses (cos_i, sin_i), lane i+RH uses (cos_i+RH, sin_i+RH).
template <int RH>
__device__ __forceinline__ void rotate_in_granule4(float (&v)[16], const float4* __restrict__ cs,
                                                   int64_t T) {
#pragma unroll
  for (int i = 0; i < RH; ++i) {
    const float4 c = __ldg(cs + i * T);
    const float x = v[i], y = v[i + RH];
    v[i] = x * c.x - y * c.y;
    v[i + RH] = y * c.z + x * c.w;
  }
}

__device__ __forceinline__ void rotate_small4(float (&v)[16], const float4* cs, int rh, int64_t T) {
  switch (rh) {
    case 1: rotate_in_granule4<1>(v, cs, T); break;
    case 2: rotate_in_granule4<2>(v, cs, T); break;
    case 3: rotate_in_granule4<3>(v, cs, T); break;
    case 4: rotate_in_granule4<4>(v, cs, T); break;
    case 5: rotate_in_granule4<5>(v, cs, T); break;
    case 6: rotate_in_granule4<6>(v, cs, T); break;
    case 7: rotate_in_granule4<7>(v, cs, T); break;
    case 8: rotate_in_granule4<8>(v, cs, T); break;
    default: break;
  }
}

__device__ __forceinline__ void rotate_small(float (&v)[16], const float2* cs, int rh, int64_t T) {
  switch (rh) {
    case 1: rotate_in_granule<1>(v, cs, T); break;
    case 2: rotate_in_granule<2>(v, cs, T); break;
    case 3: rotate_in_granule<3>(v, cs, T); break;
    case 4: rotate_in_granule<4>(v, cs, T); break;
    case 5: rotate_in_granule<5>(v, cs, T); break;
    case 6: rotate_in_granule<6>(v, cs, T); break;
    case 7: rotate_in_granule<7>(v, cs, T); break;
    case 8: rotate_in_granule<8>(v, cs, T); break;
    default: break;
  }
}

// ------------------------------------------------------------------ the kernel

// ACT: the ff-block activation, fixed at compile time so the per-value code
// has no branch on it.
// CL: CTAs per cluster. With CL == 2 the two CTAs (neighbouring M-tiles of one
// N-tile) run as a pair: the even CTA issues 2-SM MMAs (M = 256, N = 256) that
// read each CTA's own 128 token rows and each CTA's own half of the W tile, so
// a CTA streams 32 KB per k-step into shared memory and the tensor core reads
// 32 KB back, against 48 KB each way for a single CTA. The odd CTA's loads
// complete directly on the even CTA's full barriers (the cta_group::2 form of
// the tensor copy), which the even CTA's producer arms for both halves. (A
// relay of the odd CTA's completions through a second thread, or a second
// barrier per stage, each measured 20-100 % slower.)
// One CTA per SM (its shared-memory footprint allows no second one).
// GRAD: the backward's ff gradient instead of the forward: every tile lies in
// the ff block and its output is g_ff * act'(x W + b) (same GEMM, bias in the
// MMA), with column sums into db.
template <bool A_MN_MAJOR, int ACT, int CL, bool GRAD = false>
__global__ void __launch_bounds__(Warps<GRAD>::NT, 1)
    tc_gemm_kernel(const __grid_constant__ TcParams p) {
  constexpr int NT = Warps<GRAD>::NT;
  constexpr int NUM_EPI_WARPS = Warps<GRAD>::EPI;
  constexpr int EPI_PER_QUARTER = Warps<GRAD>::EPQ;
  using G = Cfg<CL, NUM_EPI_WARPS>;
  constexpr int STAGING_BYTES = G::STAGING_BYTES;
  constexpr int STAGES = G::STAGES;
  constexpr int STAGE_BYTES = G::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;  // swizzle atoms need 1 KB alignment
  uint8_t* sptr = smem_raw + (sbase - raw_addr);
  const uint32_t bias_a = sbase + STAGES * STAGE_BYTES;
  const uint32_t bias_b = bias_a + BIAS_A_BYTES;
  const uint32_t staging0 = bias_b + G::BIAS_B_BYTES;
  const uint32_t bar0 = staging0 + STAGING_BYTES;
  // full: the stage landed (in a pair: both CTAs' halves, on the even CTA's
  // barrier); empty: the MMAs read it
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t bar1 = bar0 + 8u * (2 * STAGES);
  auto tfull_bar = [&](int b) { return bar1 + 8u * b; };
  auto tempty_bar = [&](int b) { return bar1 + 8u * (2 + b); };
  const uint32_t drain_bar = bar1 + 8u * 4;
  const uint32_t bias_full = bar1 + 8u * 5;    // the bias row landed (both halves)
  const uint32_t bias_empty = bar1 + 8u * 6;   // the bias MMA has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sptr + STAGES * STAGE_BYTES + BIAS_A_BYTES +
                                                    G::BIAS_B_BYTES + STAGING_BYTES +
                                                    G::NUM_BARS * 8);
  const bool has_bias = p.epi.bias != nullptr;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl wc{p.epi.status, p.wait_limit_ns, p.launch_tag};
  const int rank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t first_unit = blockIdx.x / CL;
  const int64_t unit_step = gridDim.x / CL;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);  // one commit from the MMA thread of the pair
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), CL * NUM_EPI_WARPS);  // every epilogue warp of the pair
    }
    mbar_init(drain_bar, 1);
    mbar_init(bias_full, 1);
    mbar_init(bias_empty, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_b);
  }
  if (has_bias) {
    // bias operands: A atoms hold 0.5 (bf16 0x3F00) in k-row 0, B atoms start
    // at zero (their k-row 0 is overwritten per tile; rows 1-7 stay zero)
    for (int i = threadIdx.x; i < (BIAS_A_BYTES + G::BIAS_B_BYTES) / 16; i += NT) {
      const uint32_t off = static_cast<uint32_t>(i) * 16u;
      const uint32_t v = (off < BIAS_A_BYTES && (off & 1023u) < 128u) ? 0x3F003F00u : 0u;
      st_shared_v4(bias_a + off, v, v, v, v);
    }
    fence_async_shared();  // visible to the tensor core (async proxy)
  }
  if (warp == 1) {
    // a pair allocates collectively: one warp of each CTA, 512 columns in each
    if constexpr (CL == 1) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync();  // peers signal our barriers only after they exist
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_kb = p.num_k_blocks;
  // everything above touches no global memory: it overlaps the previous
  // launch's tail; from here on its results are visible
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (every CTA)
    if (lane == 0) {
      bool inject = (p.inject_stall & 1) && blockIdx.x == 0;
      uint32_t armed_mask = 0, armed_parity = 0;  // per stage: armed, parity of its last arming
      int stage = 0;
      uint32_t phase = 0;
      uint32_t bias_phase = 0;
      bool bias_armed = false, aborted = false;
      const bool peer = CL > 1 && rank != 0;
      // first tile column this CTA holds: its half of the MMA's N
      const int col0 = rank * ((p.bn_mma ? p.bn_mma : BN) / CL);
      for (int64_t u = first_unit; u < p.num_units && !aborted; u += unit_step) {
        const TileCoord tc = tile_coord<CL>(p, u, rank);
        int oc[3];
        outer_coords(p.tok, tc.o, oc);
        if (has_bias) {
          // this CTA's part of the tile's bias row into k-row 0 of its B atoms,
          // once the previous tile's bias MMA has read them (columns past N
          // read as zeros)
          if (!wait_bounded(bias_empty, bias_phase ^ 1u, wc, true)) {
            aborted = true;
            break;
          }
          if (!peer) {
            mbar_arrive_expect_tx(bias_full, CL * G::B_COLS * 2);  // both CTAs' parts
#pragma unroll
            for (int j = 0; j < G::B_COLS / 64; ++j)
              tma_load_2d(bias_b + j * 1024, &p.tmap_bias, bias_full, tc.n0 + 64 * j, 0);
            bias_armed = true;
          } else {
            const uint32_t pb = mapa_shared(bias_full, 0);
#pragma unroll
            for (int j = 0; j < G::B_COLS / 64; ++j)
              tma_load_2d_peer(bias_b + j * 1024, &p.tmap_bias, pb, tc.n0 + col0 + 64 * j, 0);
          }
          bias_phase ^= 1u;
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, wc, true)) {
            aborted = true;
            break;
          }
          const uint32_t a_dst = sbase + stage * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          const int k0 = kb * BK;
          if (peer) {
            // the even CTA armed its full barrier for these bytes too
            const uint32_t fb = mapa_shared(full_bar(stage), 0);
            if (A_MN_MAJOR && p.a_split) {
              tma_load_5d_peer(a_dst, &p.tmap_a, fb, 0, k0, static_cast<int>(tc.s0 >> 6), oc[0],
                               oc[1]);
            } else if (A_MN_MAJOR) {
              tma_load_5d_peer(a_dst, &p.tmap_a, fb, static_cast<int>(tc.s0), k0, oc[0], oc[1],
                               oc[2]);
              tma_load_5d_peer(a_dst + CHUNK_BYTES, &p.tmap_a, fb, static_cast<int>(tc.s0) + 64,
                               k0, oc[0], oc[1], oc[2]);
            } else {
              tma_load_5d_peer(a_dst, &p.tmap_a, fb, k0, static_cast<int>(tc.s0), oc[0], oc[1],
                               oc[2]);
            }
#pragma unroll
            for (int j = 0; j < G::B_COLS / 64; ++j)
              tma_load_2d_peer(b_dst + j * CHUNK_BYTES, &p.tmap_b, fb, tc.n0 + col0 + 64 * j, k0);
          } else {
            if (inject) {
              inject = false;  // withhold this stage: its consumer's wait runs out
            } else {
              const uint32_t fb = full_bar(stage);
              mbar_arrive_expect_tx(fb, CL * STAGE_BYTES);  // both CTAs' halves
              if (A_MN_MAJOR && p.a_split) {
                tma_load_5d(a_dst, &p.tmap_a, fb, 0, k0, static_cast<int>(tc.s0 >> 6), oc[0],
                            oc[1]);
              } else if (A_MN_MAJOR) {
                tma_load_5d(a_dst, &p.tmap_a, fb, static_cast<int>(tc.s0), k0, oc[0], oc[1],
                            oc[2]);
                tma_load_5d(a_dst + CHUNK_BYTES, &p.tmap_a, fb, static_cast<int>(tc.s0) + 64, k0,
                            oc[0], oc[1], oc[2]);
              } else {
                tma_load_5d(a_dst, &p.tmap_a, fb, k0, static_cast<int>(tc.s0), oc[0], oc[1],
                            oc[2]);
              }
#pragma unroll
              for (int j = 0; j < G::B_COLS / 64; ++j)
                tma_load_2d(b_dst + j * CHUNK_BYTES, &p.tmap_b, fb, tc.n0 + 64 * j, k0);
              armed_mask |= 1u << stage;
              armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: this CTA's copies must land before it exits. The even CTA waits
      // on the barriers it armed (an armed phase whose peer half never came
      // runs out after 10 ms: nothing is then in flight). The odd CTA's
      // copies complete on the even CTA's barriers, all of which the even
      // CTA's MMA thread waits for in a normal run; after an abort the odd CTA
      // allows its last copies a bounded grace period instead.
      const WaitCtl dc{wc.status, wc.limit_ns < 10000000ull ? wc.limit_ns : 10000000ull,
                       wc.launch_tag};
      for (int s = 0; s < STAGES; ++s)
        if (armed_mask & (1u << s)) wait_bounded(full_bar(s), (armed_parity >> s) & 1u, dc, false);
      if (bias_armed) wait_bounded(bias_full, bias_phase ^ 1u, dc, false);
      if (peer && aborted) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------ MMA issuer (one thread)
    if (lane == 0) {
      const int bn_mma = p.bn_mma ? p.bn_mma : BN;
      const uint32_t idesc = make_idesc(A_MN_MAJOR, true, BM * CL, bn_mma);
      // bias MMA: both operands MN-major; m (n) chunks 1 KB apart, and a k-group
      // stride of 0 so k-rows 8-15 read the same atom as k-rows 0-7
      const uint32_t idesc_bias = make_idesc(true, true, BM * CL, bn_mma);
      const uint64_t bias_a_desc = sw128_desc(bias_a, 1024, 0);
      const uint64_t bias_b_desc = sw128_desc(bias_b, 1024, 0);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t bias_phase = 0;
      bool issued = false;
      int it = 0;
      for (int64_t u = first_unit; u < p.num_units; u += unit_step, ++it) {
        const int buf = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!wait_bounded(tempty_bar(buf), acc_phase ^ 1u, wc, true)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * ACC_COLS;
        if (has_bias) {
          if (!wait_bounded(bias_full, bias_phase, wc, true)) break;
          tc_fence_after();
          umma_bf16<CL>(d_tmem, bias_a_desc, bias_b_desc, idesc_bias, 0u);  // D = bias
          umma_commit_all<CL>(bias_empty);
          bias_phase ^= 1u;
          issued = true;
        }
        const uint32_t acc0 = has_bias ? 1u : 0u;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, wc, true)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sbase + stage * STAGE_BYTES;
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            // A: MN-major -> 16 channel rows of 128 B per K step, chunks of 64 tokens 8 KB apart;
            //    K-major  -> 32 B per K step inside the 128-B swizzled row, 8-row groups 1 KB apart.
            const uint64_t a_desc = A_MN_MAJOR ? sw128_desc(a_addr + k * 2048, CHUNK_BYTES, 1024)
                                               : sw128_desc(a_addr + k * 32, 16, 1024);
            const uint64_t b_desc = sw128_desc(b_addr + k * 2048, CHUNK_BYTES, 1024);
            umma_bf16<CL>(d_tmem, a_desc, b_desc, idesc, (kb | k) != 0 ? 1u : acc0);
          }
          issued = true;
          umma_commit_all<CL>(empty_bar(stage));  // frees the stage in every CTA of the pair
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_all<CL>(tfull_bar(buf));  // accumulators ready for the epilogues
      }
      if (issued) {
        umma_commit<CL>(drain_bar);  // all MMAs retired before TMEM is freed
        wait_bounded(drain_bar, 0, wc, false);
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue warps
    const Epilogue& e = p.epi;
    const int quarter = warp & 3;                  // TMEM lanes this warp may read
    const int part = (warp - 2) >> 2;              // which of a quarter's work units it takes
    const int row = quarter * 32 + lane;
    const int rh = e.rope_half;
    const int nkv = e.groups > 0 ? e.groups : e.heads;
    const int64_t head_stride = e.T * e.hd;
    const uint32_t staging_warp = staging0 + (warp - 2) * STAGING_BYTES_PER_WARP;
    // the staging rows are 32 B; the output maps use the 32-byte swizzle, which
    // swaps the two 16-byte halves of rows 4-7 of every 8, so the eight rows a
    // quarter-warp stores at once fall in distinct banks
    const uint32_t swz = ((lane >> 2) & 1u) * 16u;
    uint32_t stage_sel = 0;  // alternates this warp's two staging buffers
    // a quarter's warps take its work units round-robin; the count runs
    // on across tiles, so a tile whose unit count is not a multiple of 3 does
    // not always load the same warp
    int turn = 0;
    int it = 0;
    for (int64_t u = first_unit; u < p.num_units; u += unit_step, ++it) {
      const int buf = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const int ok = wait_bounded(tfull_bar(buf), acc_phase, wc, true) ? 1 : 0;
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      const TileCoord tc = tile_coord<CL>(p, u, rank);
      const bool valid = !tc.phantom && tc.s0 + row < p.tok.S_in;
      const int64_t m0 = tc.o * p.tok.S_in + tc.s0;  // the tile's first token
      const int64_t m = m0 + row;
      // batch element and position: one division per tile, a step per row
      int64_t bidx, t;
      if (e.T >= BM) {
        bidx = div_nonneg(m0, e.T);
        t = m0 - bidx * e.T + row;
        if (t >= e.T) {
          t -= e.T;
          ++bidx;
        }
      } else {
        bidx = div_nonneg(m, e.T);
        t = m - bidx * e.T;
      }
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * ACC_COLS;
      const int cols = min(e.bn_eff, e.N - tc.n0);  // columns this tile owns
      // Block stores (the ff tiles' warp-wide copy out of the staging buffer,
      // the TMA stores of head tiles and mixed tiles) write the warp's 32 rows
      // as one block: they must all be valid and, for the head-major buffers,
      // lie in one batch element (tokens t .. t+31). Lane 0 issues the TMA
      // stores with its own coordinates.
      const bool tma_ff = p.tma_store && __all_sync(0xFFFFFFFFu, valid);
      // whole heads of the blocked q|k|v order, rotation absent or in 16-lane
      // groups, k not pre-transposed
      const bool fast_heads = tc.n0 >= e.F && e.groups == 0 && !e.k_transposed &&
                              (rh == 0 || rh >= 16) && (tc.n0 - e.F) % e.hd == 0 &&
                              cols % e.hd == 0;
      auto stage_store = [&](const CUtensorMap* map, int c0, int c1, int c2, bool three_d,
                             const uint32_t (&w)[8]) {
        const uint32_t stg = staging_warp + (stage_sel & 1) * 2048;
        ++stage_sel;
        if (lane == 0) bulk_wait_read_1();  // this buffer's previous store has read it
        __syncwarp();
        st_shared_v4(stg + lane * 32 + swz, w[0], w[1], w[2], w[3]);
        st_shared_v4(stg + lane * 32 + (swz ^ 16u), w[4], w[5], w[6], w[7]);
        fence_async_shared();
        __syncwarp();
        if (lane == 0) {
          if (three_d)
            tma_store_3d(map, stg, c0, c1, c2);
          else
            tma_store_2d(map, stg, c0, c1);
          bulk_commit();
        }
      };
      if (tc.n0 + cols <= e.F && (cols & 31) == 0) {
        // ---- a tile inside the ff block: activation, then [M, F] row-major,
        // 32 columns per work unit (the tile's width is a multiple of 32)
        uint16_t* const ff_row = static_cast<uint16_t*>(e.out_ff) + m * e.ff_ld + tc.n0;
        // 64-byte rows, 64-byte swizzle: 16-byte chunk c of row r sits at c ^ ((r >> 1) & 3)
        const uint32_t sw64 = (lane >> 1) & 3u;
        for (int c = 0; c < cols; c += 32) {
          const bool mine = turn == part;
          turn = turn + 1 == EPI_PER_QUARTER ? 0 : turn + 1;
          if (!mine) continue;
          uint32_t v_u[32];
          tmem_ld32(t_row + c, v_u);
          tmem_wait_ld();
          uint32_t w[16];
          if constexpr (GRAD) {
            // upstream gradient of the lane's token, 32 columns (zero past M)
            float gg[32];
            const uint4* g4 = reinterpret_cast<const uint4*>(
                static_cast<const uint16_t*>(e.g_ff) + m * e.F + tc.n0 + c);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 u = valid ? __ldg(g4 + q) : make_uint4(0, 0, 0, 0);
              const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                gg[8 * q + 2 * i] = __uint_as_float(uw[i] << 16);
                gg[8 * q + 2 * i + 1] = __uint_as_float(uw[i] & 0xFFFF0000u);
              }
            }
            if (ACT == ACT_GELU_ERF) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float d0, d1;
                gelu_erf_deriv2(__uint_as_float(v_u[2 * i]), __uint_as_float(v_u[2 * i + 1]), d0,
                                d1);
                gg[2 * i] *= d0;
                gg[2 * i + 1] *= d1;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) gg[i] *= act_deriv<ACT>(__uint_as_float(v_u[i]));
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(gg[2 * i], gg[2 * i + 1]);
            if (e.db) {
              const float cs = column_sum32(gg, lane);
              atomicAdd(e.db + tc.n0 + c + lane, cs);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = activate2_bf16<ACT>(v_u[2 * i], v_u[2 * i + 1]);
          }
          if (tma_ff) {
            const uint32_t stg = staging_warp + (stage_sel & 1) * 2048;
            ++stage_sel;
            if (lane == 0) bulk_wait_read_1();  // this buffer's previous store has read it
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(stg + lane * 64 + ((q ^ sw64) << 4), w[4 * q], w[4 * q + 1],
                           w[4 * q + 2], w[4 * q + 3]);
            fence_async_shared();
            __syncwarp();
            // read back and stored by the whole warp: four lanes per 64-byte
            // row segment, eight rows per instruction (measured faster than a
            // TMA store of the block: 134.3 -> 129.5 us on a 24576 x 768 x 5376
            // product, the same bits)
            {
              uint16_t* const blk = static_cast<uint16_t*>(e.out_ff) + (m - lane) * e.ff_ld +
                                    tc.n0 + c;
              const int ch = lane & 3;
              if (!e.bounds_check) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int r = (lane >> 2) + 8 * k;
                  const uint4 v = ld_shared_v4(stg + r * 64 + ((ch ^ ((r >> 1) & 3)) << 4));
                  *reinterpret_cast<uint4*>(blk + static_cast<int64_t>(r) * e.ff_ld + ch * 8) = v;
                }
              } else {
                // FP_OPT_BOUNDS_CHECK: each 16-byte piece checked against the extent
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int r = (lane >> 2) + 8 * k;
                  const uint4 v = ld_shared_v4(stg + r * 64 + ((ch ^ ((r >> 1) & 3)) << 4));
                  uint16_t* const dst = blk + static_cast<int64_t>(r) * e.ff_ld + ch * 8;
                  if (store_in_bounds(e, 0, dst - static_cast<uint16_t*>(e.out_ff), 8))
                    *reinterpret_cast<uint4*>(dst) = v;
                }
              }
              __syncwarp();
            }
          } else if (valid && store_in_bounds(e, 0, m * e.ff_ld + tc.n0 + c, 32)) {
            uint4* d4 = reinterpret_cast<uint4*>(ff_row + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              d4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
      } else if (fast_heads && tma_ff &&
                 __shfl_sync(0xFFFFFFFFu, static_cast<int>(t), 31) -
                         __shfl_sync(0xFFFFFFFFu, static_cast<int>(t), 0) == 31) {
        // ---- whole heads of the blocked q|k|v part, every row valid and in one
        // batch element: each 32 x 16 block leaves by TMA at (lane j, token t,
        // b*heads + head); heads are decoded once per head, not per column
        const int w0 = tc.n0 - e.F;
        int seg = w0 / e.C;                       // 0 q, 1 k, 2 v
        int head = (w0 - seg * e.C) / e.hd;
        const int nh_tile = cols / e.hd;
        const int z_b = static_cast<int>(bidx) * e.heads;
        for (int hl = 0; hl < nh_tile; ++hl) {
          const uint32_t t_head = t_row + hl * e.hd;
          const CUtensorMap* map = seg == 0 ? &p.tmap_q : seg == 1 ? &p.tmap_k : &p.tmap_v;
          const int z = z_b + head;
          int j0 = 0;
          if (rh > 0 && seg < 2) {
            // rotated pairs (j, j + rh), 16 lanes at a time
            for (int j = 0; j < rh; j += 16) {
              const bool mine = turn == part;
              turn = turn + 1 == EPI_PER_QUARTER ? 0 : turn + 1;
              if (!mine) continue;
              uint32_t lo_u[16], hi_u[16];
              tmem_ld16(t_head + j, lo_u);
              tmem_ld16(t_head + j + rh, hi_u);
              tmem_wait_ld();
              uint32_t lo_w[8], hi_w[8];
              // frequency-major tables: lane (token t) reads entry (f, t) at f * T + t,
              // so a warp's 32 consecutive tokens read one contiguous run per f
              if (e.rope_per_lane) {
                const float4* t4 = e.rope_cs4 + t + j * e.T;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                  for (int i = 4 * h; i < 4 * h + 4; ++i) {
                    const float4 c0 = __ldg(t4 + (2 * i) * e.T), c1 = __ldg(t4 + (2 * i + 1) * e.T);
                    const float x0 = __uint_as_float(lo_u[2 * i]);
                    const float y0 = __uint_as_float(hi_u[2 * i]);
                    const float x1 = __uint_as_float(lo_u[2 * i + 1]);
                    const float y1 = __uint_as_float(hi_u[2 * i + 1]);
                    lo_w[i] = pack_bf16x2(x0 * c0.x - y0 * c0.y, x1 * c1.x - y1 * c1.y);
                    hi_w[i] = pack_bf16x2(y0 * c0.z + x0 * c0.w, y1 * c1.z + x1 * c1.w);
                  }
                  asm volatile("" ::: "memory");
                }
              } else {
                const float2* csf = e.rope_cs + t + j * e.T;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  // (cos, sin) of frequencies j + 2i and j + 2i + 1
                  const float2 ca = __ldg(csf + (2 * i) * e.T), cb = __ldg(csf + (2 * i + 1) * e.T);
                  const float x0 = __uint_as_float(lo_u[2 * i]), y0 = __uint_as_float(hi_u[2 * i]);
                  const float x1 = __uint_as_float(lo_u[2 * i + 1]);
                  const float y1 = __uint_as_float(hi_u[2 * i + 1]);
                  lo_w[i] = pack_bf16x2(x0 * ca.x - y0 * ca.y, x1 * cb.x - y1 * cb.y);
                  hi_w[i] = pack_bf16x2(y0 * ca.x + x0 * ca.y, y1 * cb.x + x1 * cb.y);
                }
              }
              stage_store(map, j, static_cast<int>(t), z, true, lo_w);
              stage_store(map, j + rh, static_cast<int>(t), z, true, hi_w);
            }
            j0 = 2 * rh;  // lanes past the rotated ones pass through
          }
          for (int j = j0; j < e.hd; j += 16) {
            const bool mine = turn == part;
            turn = turn + 1 == EPI_PER_QUARTER ? 0 : turn + 1;
            if (!mine) continue;
            uint32_t v_u[16];
            tmem_ld16(t_head + j, v_u);
            tmem_wait_ld();
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = pack_bf16x2(__uint_as_float(v_u[2 * i]), __uint_as_float(v_u[2 * i + 1]));
            stage_store(map, j, static_cast<int>(t), z, true, w);
          }
          if (++head == e.heads) {
            head = 0;
            ++seg;
          }
        }
      } else {
        // ---- any other tile that reaches the head-major blocks
        const bool tma_heads =
            tma_ff && __shfl_sync(0xFFFFFFFFu, static_cast<int>(t), 31) -
                              __shfl_sync(0xFFFFFFFFu, static_cast<int>(t), 0) == 31;
        uint16_t* const ff_row = static_cast<uint16_t*>(e.out_ff) + m * e.F;
        uint16_t* const q_row = static_cast<uint16_t*>(e.out_q) + (bidx * e.heads * e.T + t) * e.hd;
        uint16_t* const k_row = static_cast<uint16_t*>(e.out_k) + (bidx * nkv * e.T + t) * e.hd;
        uint16_t* const v_row = static_cast<uint16_t*>(e.out_v) + (bidx * nkv * e.T + t) * e.hd;
        // pre-transposed k: element (b, head, lane j, token t) at ((b*nkv + head)*hd + j)*T + t
        uint16_t* const kt_row = static_cast<uint16_t*>(e.out_k) + bidx * nkv * head_stride + t;
        const float2* const cs_t = e.rope_cs + t;  // entry (0, t) of the frequency-major table
        auto put16 = [&](int seg, int head, int j, uint16_t* dst, const uint32_t (&w)[8]) {
          if (!(seg == 0 ? tma_ff : tma_heads)) {
            if (valid &&
                store_in_bounds(e, seg, dst - static_cast<uint16_t*>(out_base(e, seg)), 16)) {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
              d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
              d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
            return;
          }
          if (seg == 0) {
            stage_store(&p.tmap_ff, j, static_cast<int>(m), 0, false, w);
          } else {
            const int nh = seg == 1 ? e.heads : nkv;
            const CUtensorMap* map = seg == 1 ? &p.tmap_q : seg == 2 ? &p.tmap_k : &p.tmap_v;
            stage_store(map, j, static_cast<int>(t), static_cast<int>(bidx * nh + head), true, w);
          }
        };
        ColCursor cur;
        cursor_init(e, tc.n0, cur);
        for (int c = 0; c < cols; c += 16, cursor_advance16(e, cur)) {
          const ColInfo& ci = cur.ci;
          const bool qk = ci.seg == 1 || ci.seg == 2;
          // rh >= 16: lanes i and i+rh sit in different granules, handled as a pair;
          // rh <= 8: every rotated lane sits in the head's first granule.
          const bool rope = rh >= 16 && qk && ci.j < 2 * rh;
          const bool rope_small = rh > 0 && rh <= 8 && qk && ci.j == 0;
          if (rope && ci.j >= rh) continue;  // the high half is written with its low partner
          const bool mine = turn == part;
          turn = turn + 1 == EPI_PER_QUARTER ? 0 : turn + 1;
          if (!mine) continue;
          uint16_t* const dst =
              ci.seg == 0 ? ff_row + ci.j
                          : (ci.seg == 1 ? q_row : ci.seg == 2 ? k_row : v_row) +
                                ci.head * head_stride + ci.j;
          const bool kt = e.k_transposed && ci.seg == 2;
          uint16_t* const dst_t = kt_row + (static_cast<int64_t>(ci.head) * e.hd + ci.j) * e.T;
          if (rope) {
            uint32_t lo_u[16], hi_u[16];
            tmem_ld16(t_row + c, lo_u);
            tmem_ld16(t_row + c + rh, hi_u);
            tmem_wait_ld();
            uint32_t lo_w[8], hi_w[8];  // results, two bf16 per word
            if (e.rope_per_lane) {
              const float4* t4 = e.rope_cs4 + t + ci.j * e.T;
              // two halves, so that at most eight table entries are in flight
#pragma unroll
              for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int i = 4 * h; i < 4 * h + 4; ++i) {
                  const float4 c0 =
                      valid ? __ldg(t4 + (2 * i) * e.T) : make_float4(0.f, 0.f, 0.f, 0.f);
                  const float4 c1 =
                      valid ? __ldg(t4 + (2 * i + 1) * e.T) : make_float4(0.f, 0.f, 0.f, 0.f);
                  const float x0 = __uint_as_float(lo_u[2 * i]);
                  const float y0 = __uint_as_float(hi_u[2 * i]);
                  const float x1 = __uint_as_float(lo_u[2 * i + 1]);
                  const float y1 = __uint_as_float(hi_u[2 * i + 1]);
                  lo_w[i] = pack_bf16x2(x0 * c0.x - y0 * c0.y, x1 * c1.x - y1 * c1.y);
                  hi_w[i] = pack_bf16x2(y0 * c0.z + x0 * c0.w, y1 * c1.z + x1 * c1.w);
                }
                asm volatile("" ::: "memory");
              }
            } else {
              const float2* csf = cs_t + ci.j * e.T;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                // (cos, sin) of frequencies j + 2i and j + 2i + 1
                const float2 ca = valid ? __ldg(csf + (2 * i) * e.T) : make_float2(0.f, 0.f);
                const float2 cb = valid ? __ldg(csf + (2 * i + 1) * e.T) : make_float2(0.f, 0.f);
                const float x0 = __uint_as_float(lo_u[2 * i]), y0 = __uint_as_float(hi_u[2 * i]);
                const float x1 = __uint_as_float(lo_u[2 * i + 1]);
                const float y1 = __uint_as_float(hi_u[2 * i + 1]);
                lo_w[i] = pack_bf16x2(x0 * ca.x - y0 * ca.y, x1 * cb.x - y1 * cb.y);
                hi_w[i] = pack_bf16x2(y0 * ca.x + x0 * ca.y, y1 * cb.x + x1 * cb.y);
              }
            }
            if (kt) {  // pre-transposed k is stored directly, one lane column at a time
              const int64_t off = dst_t - static_cast<uint16_t*>(e.out_k);
              if (valid && store_in_bounds(e, 2, off, 16, e.T))
                store16_packed_strided(dst_t, e.T, lo_w);
              if (valid && store_in_bounds(e, 2, off + rh * e.T, 16, e.T))
                store16_packed_strided(dst_t + rh * e.T, e.T, hi_w);
            } else {
              put16(ci.seg, ci.head, ci.j, dst, lo_w);
              put16(ci.seg, ci.head, ci.j + rh, dst + rh, hi_w);
            }
          } else {
            uint32_t v_u[16];
            tmem_ld16(t_row + c, v_u);
            tmem_wait_ld();
            uint32_t w[8];
            if (ci.seg == 0) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                w[i] = activate2_bf16<ACT>(v_u[2 * i], v_u[2 * i + 1]);
            } else if (rope_small && valid) {
              float v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(v_u[i]);
              if (e.rope_per_lane)
                rotate_small4(v, e.rope_cs4 + t, rh, e.T);
              else
                rotate_small(v, cs_t, rh, e.T);
#pragma unroll
              for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                w[i] = pack_bf16x2(__uint_as_float(v_u[2 * i]), __uint_as_float(v_u[2 * i + 1]));
            }
            if (kt) {
              if (valid && store_in_bounds(e, 2, dst_t - static_cast<uint16_t*>(e.out_k), 16, e.T))
                store16_packed_strided(dst_t, e.T, w);
            } else {
              put16(ci.seg, ci.head, ci.j, dst, w);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      // release the accumulator: the even CTA's MMA thread waits on every
      // epilogue warp of the pair
      if (lane == 0) {
        if (CL == 1 || rank == 0)
          mbar_arrive(tempty_bar(buf));
        else
          mbar_arrive_remote(mapa_shared(tempty_bar(buf), 0));
      }
    }
    if (lane == 0) bulk_wait_all();  // every TMA store of this warp has completed
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // no CTA leaves while its peer may still write into its shared memory or
  // arrive on its barriers
  if (CL > 1) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (CL == 1)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(TMEM_COLS)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(TMEM_COLS)
                   : "memory");
  }
}

template <bool A_MN, int ACT, int CL, bool GRAD = false>
cudaError_t launch_variant(const TcParams& p, int num_ctas, cudaStream_t stream) {
  auto kernel = tc_gemm_kernel<A_MN, ACT, CL, GRAD>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !attr_done[dev]) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<CL, Warps<GRAD>::EPI>::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    if (dev < 64) attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(Warps<GRAD>::NT, 1, 1);
  cfg.dynamicSmemBytes = Cfg<CL, Warps<GRAD>::EPI>::SMEM_BYTES;
  cfg.stream = stream;
  // programmatic dependent launch: the prologue may overlap the previous
  // launch's tail (the kernel waits on it before touching global memory)
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  if (CL == 1) {
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(num_ctas, 1, 1);
    err = cudaLaunchKernelEx(&cfg, kernel, p);
    return err != cudaSuccess ? err : cudaGetLastError();
  }
  cfg.numAttrs = 2;
  // persistent: as many clusters as can be resident at once (one CTA per SM)
  static int max_clusters[64] = {0};
  if (dev >= 64 || !max_clusters[dev]) {
    cfg.gridDim = dim3(num_ctas, 1, 1);
    cudaLaunchConfig_t q = cfg;  // the query sees the cluster shape only
    q.attrs = attr + 1;
    q.numAttrs = 1;
    int n = 0;
    err = cudaOccupancyMaxActiveClusters(&n, kernel, &q);
    if (err != cudaSuccess) return err;
    if (n < 1) return cudaErrorInvalidConfiguration;
    if (dev < 64) max_clusters[dev] = n;
    else return cudaErrorInvalidDevice;
  }
  int64_t clusters = num_ctas / CL;
  if (clusters > max_clusters[dev]) clusters = max_clusters[dev];
  if (clusters > p.num_units) clusters = p.num_units;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * CL), 1, 1);
  err = cudaLaunchKernelEx(&cfg, kernel, p);
  return err != cudaSuccess ? err : cudaGetLastError();
}

template <bool A_MN, int CL, bool GRAD = false>
cudaError_t launch_act(const TcParams& p, int num_ctas, cudaStream_t stream) {
  switch (p.epi.act) {
    case ACT_GELU_ERF: return launch_variant<A_MN, ACT_GELU_ERF, CL, GRAD>(p, num_ctas, stream);
    case ACT_GELU_TANH: return launch_variant<A_MN, ACT_GELU_TANH, CL, GRAD>(p, num_ctas, stream);
    case ACT_SILU: return launch_variant<A_MN, ACT_SILU, CL, GRAD>(p, num_ctas, stream);
    case ACT_RELU2: return launch_variant<A_MN, ACT_RELU2, CL, GRAD>(p, num_ctas, stream);
    default: return launch_variant<A_MN, ACT_NONE, CL, GRAD>(p, num_ctas, stream);
  }
}

}  // namespace

cudaError_t launch_tc_gemm(const TcParams& p, bool a_mn_major, int num_ctas, cudaStream_t stream,
                           bool grad) {
  if (p.num_units == 0) return cudaSuccess;
  if (grad) {  // CTA pairs only
    if (p.cluster != 2) return cudaErrorInvalidValue;
    return a_mn_major ? launch_act<true, 2, true>(p, num_ctas, stream)
                      : launch_act<false, 2, true>(p, num_ctas, stream);
  }
  if (p.cluster == 2)
    return a_mn_major ? launch_act<true, 2>(p, num_ctas, stream)
                      : launch_act<false, 2>(p, num_ctas, stream);
  return a_mn_major ? launch_act<true, 1>(p, num_ctas, stream)
                    : launch_act<false, 1>(p, num_ctas, stream);
}

}  // namespace fp
