// Backward of the fused projection: the gradients of act/rotate/split(x W + b)
// with respect to x, W and b, given the upstream gradients in the forward's
// output layouts.
//
// The pages ("[perf] Fused linear", xformers PR #283) name the backward only
// as the part of the fused linear left unfused and slow. Here it is the chain
// rule in four device steps, every GEMM on the tensor cores:
//
//   gather   G[:, F:] = the q/k/v gradients gathered from their head-major
//            buffers into token-major rows, q and k rotated back by the
//            transpose of the rotation (bwd_gather_pairs_kernel, or
//            bwd_gather_kernel for the layouts it does not cover; CUDA cores);
//   GRADFF   G[:, :F] = g_ff * act'(x W_ff + b_ff): the pre-activation is
//            recomputed by a forward GEMM whose epilogue multiplies the
//            upstream gradient by the activation's derivative (the forward
//            kernel's gradient mode when F is a multiple of 32, else this
//            file's GEMM kernel);
//   DX/DXT   dx = G W^T. For token-major x the tile rows are tokens; for
//            channels-first x the kernel computes dx^T = W G^T, whose rows are
//            channels and whose columns are contiguous tokens, so either way
//            the result is stored straight into x's own layout by TMA;
//   DW       dW = X^T G in fp32, the token range split across CTAs, partial
//            tiles added into dW by TMA reduce-add (cp.reduce.async.bulk).
// db is the column sum of G, accumulated by the gather kernel and the GRADFF
// epilogue (a 31-shuffle butterfly per warp, one atomic add per column).
//
// The GEMM kernel is a persistent tcgen05 pipeline with two TMEM accumulators:
// warp 0 loads, one thread of warp 1 issues tcgen05.mma, warps 2-9 drain the
// accumulators. It runs on single CTAs (M = 128, N = 256, K = 64 per stage, 4
// stages of 48 KB) or, for DX and DXT, on CTA pairs (2-SM MMAs with M = 256,
// 6 stages of 32 KB per CTA). Every wait is bounded as in the forward kernel.
#include <algorithm>

#include "epilogue.cuh"
#include "fp_internal.h"
#include "tc_ptx.cuh"

namespace fp {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, UMMA_K = 16;
constexpr int NUM_EPI_WARPS = 8;  // 2 per TMEM lane quarter
constexpr int NT = 32 * (2 + NUM_EPI_WARPS);
constexpr int A_BYTES = BM * BK * 2;           // 16 KB: this CTA's 128 rows
constexpr int CHUNK_BYTES = 64 * BK * 2;       // one [64 k][64 mn] MN-major chunk, 8 KB
constexpr int ACC_COLS = BN;
constexpr int TMEM_COLS = 2 * ACC_COLS;
// per epilogue warp, two 2 KB buffers staging [32 rows][64 B] for TMA stores
constexpr int STAGING_BYTES_PER_WARP = 2 * 2048;
constexpr int STAGING_BYTES = NUM_EPI_WARPS * STAGING_BYTES_PER_WARP;

// Per cluster size. A single CTA holds the tile's 128 rows and all 256
// columns of B (48 KB a k-step, 4 stages). A CTA pair runs 2-SM MMAs
// (M = 256): each CTA holds its own 128 rows and its own 128 of the 256 B
// columns, 32 KB a k-step, so the same shared memory keeps 6 k-steps in flight.
template <int CL>
struct BwdCfg {
  static constexpr int B_COLS = BN / CL;
  static constexpr int B_BYTES = B_COLS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = CL == 2 ? 6 : 4;
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
  static constexpr int SMEM_BYTES =
      1024 + STAGES * STAGE_BYTES + STAGING_BYTES + NUM_BARS * 8 + 16;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// The odd CTA of a pair: a 3-D tiled load into its own shared memory whose
// bytes complete on an mbarrier of the even CTA (`bar`, a cluster address).
__device__ __forceinline__ void tma_load_3d_peer(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::
          "l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

// fp32 add of a staged tile into global memory
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int c0,
                                                  int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::
          "l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}

// Tile of one work item.
struct Geo {
  int o, s0;     // token slab and first token of the tile (token rows or columns)
  int r0;        // first row when rows are channels (DXT, DW)
  int c0;        // first column: ff column (GRADFF), channel (DX), fused column (DW)
  int kb0, kb1;  // k-block range
  bool phantom;  // row tile past the end (odd row-tile count in a pair): compute, store nothing
};

// Work item -> this CTA's tile. A cluster of CL CTAs takes CL consecutive row
// tiles with the same column tile (they share its B tile). Groups of group_m
// row tiles sweep the column tiles, rows fastest, so concurrently resident
// CTAs share operand tiles in L2. For DW the k splits of one tile are
// (row-tile groups of CL) * num_n_tiles items apart.
template <int CL>
__device__ __forceinline__ Geo unit_geo(const BwdGemmParams& p, int64_t u64, int rank) {
  const uint32_t u = static_cast<uint32_t>(u64);
  const uint32_t m_units = (static_cast<uint32_t>(p.num_m_tiles) + CL - 1) / CL;
  const uint32_t tiles = m_units * p.num_n_tiles;
  const uint32_t split = u / tiles;
  const uint32_t t = u - split * tiles;
  const uint32_t gsz = p.group_m >= CL ? static_cast<uint32_t>(p.group_m) / CL : 1u;
  const uint32_t per_group = gsz * p.num_n_tiles;
  const uint32_t g = t / per_group;
  const uint32_t first = g * gsz;
  const uint32_t left = m_units - first;
  const uint32_t gm = left < gsz ? left : gsz;
  const uint32_t rr = t - g * per_group;
  const uint32_t n_tile = rr / gm;
  const uint32_t m_raw = (first + (rr - n_tile * gm)) * CL + rank;
  Geo q;
  q.phantom = m_raw >= static_cast<uint32_t>(p.num_m_tiles);
  const uint32_t m_tile = q.phantom ? static_cast<uint32_t>(p.num_m_tiles) - 1 : m_raw;
  q.o = q.s0 = q.r0 = q.c0 = 0;
  q.kb0 = 0;
  q.kb1 = p.num_k_blocks;
  if (p.mode == BWD_GRADFF || p.mode == BWD_DX) {
    const uint32_t mps = static_cast<uint32_t>(p.m_tiles_per_slab);
    q.o = static_cast<int>(m_tile / mps);
    q.s0 = static_cast<int>(m_tile - q.o * mps) * BM;
    q.c0 = static_cast<int>(n_tile) * BN;
  } else if (p.mode == BWD_DXT) {
    const uint32_t nps = static_cast<uint32_t>(p.n_tiles_per_slab);
    q.r0 = static_cast<int>(m_tile) * BM;
    q.o = static_cast<int>(n_tile / nps);
    q.s0 = static_cast<int>(n_tile - q.o * nps) * BN;
  } else {
    q.r0 = static_cast<int>(m_tile) * BM;
    q.c0 = static_cast<int>(n_tile) * BN;
    const int64_t kb = p.num_k_blocks;
    q.kb0 = static_cast<int>(kb * split / p.k_splits);
    q.kb1 = static_cast<int>(kb * (split + 1) / p.k_splits);
  }
  return q;
}

// 32 bf16 values (four 16-byte loads from a 16-byte aligned address), widened to fp32
__device__ __forceinline__ void load32_bf16(const uint16_t* src, float (&f)[32]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = __ldg(s4 + q);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
      f[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

// CL: CTAs per cluster. With CL == 2 the even CTA issues 2-SM MMAs (M = 256)
// reading each CTA's own 128 rows and each CTA's half of the B tile; the odd
// CTA's copies complete on the even CTA's full barriers, which the even CTA's
// producer arms for both halves; commits go to both CTAs' barriers; the odd
// CTA's epilogue releases the accumulator on the even CTA's barrier.
template <int MODE, bool A_MN, bool B_MN, int ACT, int CL>
__global__ void __launch_bounds__(NT, 1) bwd_gemm_kernel(const __grid_constant__ BwdGemmParams p) {
  using G = BwdCfg<CL>;
  constexpr int STAGES = G::STAGES;
  constexpr int STAGE_BYTES = G::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - raw_addr);
  const uint32_t staging0 = sbase + STAGES * STAGE_BYTES;
  const uint32_t bar0 = staging0 + STAGING_BYTES;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sptr + STAGES * STAGE_BYTES + STAGING_BYTES +
                                                    G::NUM_BARS * 8);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl wc{p.status, p.wait_limit_ns, p.launch_tag};
  const int rank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t first_unit = blockIdx.x / CL;
  const int64_t unit_step = gridDim.x / CL;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), CL * NUM_EPI_WARPS);  // every epilogue warp of the pair
    }
    mbar_init(drain_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_b);
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
  if (CL > 1) cluster_sync();  // the peer signals our barriers only after they exist
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // everything above touches no global memory: it overlaps the previous
  // launch's tail; from here on its results are visible
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t armed_mask = 0, armed_parity = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const bool peer = CL > 1 && rank != 0;
      const int bcol = rank * G::B_COLS;  // first of the B tile's columns this CTA holds
      for (int64_t u = first_unit; u < p.num_units && ok; u += unit_step) {
        const Geo g = unit_geo<CL>(p, u, rank);
        int oc[3];
        if (MODE != BWD_DW) outer_coords(p.tok, g.o, oc);
        // DW walks K over tokens: (slab, block in slab) advances incrementally and
        // the slab's outer coordinates are recomputed only when the slab changes
        int ok_slab = 0, kb_in = 0;
        int ock[3] = {0, 0, 0};
        if (MODE == BWD_DW) {
          ok_slab = g.kb0 / p.k_blocks_per_slab;
          kb_in = g.kb0 - ok_slab * p.k_blocks_per_slab;
          outer_coords(p.tok, ok_slab, ock);
        }
        for (int kb = g.kb0; kb < g.kb1; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, wc, true)) {
            ok = false;
            break;
          }
          // the even CTA's full barrier takes both CTAs' bytes
          const uint32_t fb = peer ? mapa_shared(full_bar(stage), 0) : full_bar(stage);
          if (!peer) mbar_arrive_expect_tx(fb, CL * STAGE_BYTES);
          const uint32_t a_dst = sbase + stage * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          const int k0 = kb * BK;
          auto ld2 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1) {
            if (peer)
              tma_load_2d_peer(dst, map, fb, c0, c1);
            else
              tma_load_2d(dst, map, fb, c0, c1);
          };
          auto ld3 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2) {
            if (peer)
              tma_load_3d_peer(dst, map, fb, c0, c1, c2);
            else
              tma_load_3d(dst, map, fb, c0, c1, c2);
          };
          auto ld5 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                         int c4) {
            if (peer)
              tma_load_5d_peer(dst, map, fb, c0, c1, c2, c3, c4);
            else
              tma_load_5d(dst, map, fb, c0, c1, c2, c3, c4);
          };
          if (MODE == BWD_GRADFF) {
            if (A_MN) {
              tma_load_5d(a_dst, &p.tmap_a, fb, g.s0, k0, oc[0], oc[1], oc[2]);
              tma_load_5d(a_dst + CHUNK_BYTES, &p.tmap_a, fb, g.s0 + 64, k0, oc[0], oc[1], oc[2]);
            } else {
              tma_load_5d(a_dst, &p.tmap_a, fb, k0, g.s0, oc[0], oc[1], oc[2]);
            }
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(b_dst + j * CHUNK_BYTES, &p.tmap_b, fb, g.c0 + 64 * j, k0);
          } else if (MODE == BWD_DX) {
            ld3(a_dst, &p.tmap_a, k0, g.s0, g.o);       // G rows (tokens), K = N
            ld2(b_dst, &p.tmap_b, k0, g.c0 + bcol);     // W rows (channels), K = N
          } else if (MODE == BWD_DXT) {
            ld2(a_dst, &p.tmap_a, k0, g.r0);            // W rows (channels)
            ld3(b_dst, &p.tmap_b, k0, g.s0 + bcol, g.o);  // G rows (tokens)
          } else {
            // K = tokens: block kb_in of slab ok_slab
            const int sk = kb_in * BK;
            if (A_MN) {  // token-major x: channels contiguous
              ld5(a_dst, &p.tmap_a, g.r0, sk, ock[0], ock[1], ock[2]);
              ld5(a_dst + CHUNK_BYTES, &p.tmap_a, g.r0 + 64, sk, ock[0], ock[1], ock[2]);
            } else {     // channels-first x: tokens contiguous
              ld5(a_dst, &p.tmap_a, sk, g.r0, ock[0], ock[1], ock[2]);
            }
#pragma unroll
            for (int j = 0; j < G::B_COLS / 64; ++j)
              ld3(b_dst + j * CHUNK_BYTES, &p.tmap_b, g.c0 + bcol + 64 * j, sk, ok_slab);
          }
          if (!peer) {
            armed_mask |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (MODE == BWD_DW && ++kb_in == p.k_blocks_per_slab) {
            kb_in = 0;
            ++ok_slab;
            if (kb + 1 < g.kb1) outer_coords(p.tok, ok_slab, ock);
          }
        }
      }
      // drain: this CTA's copies land before it exits. The even CTA waits on
      // the barriers it armed (an armed phase whose peer half never came runs
      // out after 10 ms: nothing is then in flight). The odd CTA's copies
      // complete on the even CTA's barriers, which the even CTA's MMA thread
      // waits for in a normal run; after an abort the odd CTA allows its last
      // copies a bounded grace period instead.
      const WaitCtl dc{wc.status, wc.limit_ns < 10000000ull ? wc.limit_ns : 10000000ull,
                       wc.launch_tag};
      for (int s = 0; s < STAGES; ++s)
        if (armed_mask & (1u << s)) wait_bounded(full_bar(s), (armed_parity >> s) & 1u, dc, false);
      if (peer && !ok) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------ MMA issuer (the even CTA's)
    if (lane == 0) {
      const uint32_t idesc = make_idesc(A_MN, B_MN, BM * CL, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool issued = false;
      int it = 0;
      for (int64_t u = first_unit; u < p.num_units; u += unit_step, ++it) {
        const Geo g = unit_geo<CL>(p, u, rank);
        const int buf = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!wait_bounded(tempty_bar(buf), acc_phase ^ 1u, wc, true)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * ACC_COLS;
        bool ok = true;
        for (int kb = g.kb0; kb < g.kb1; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, wc, true)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sbase + stage * STAGE_BYTES;
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint64_t a_desc = A_MN ? sw128_desc(a_addr + k * 2048, CHUNK_BYTES, 1024)
                                         : sw128_desc(a_addr + k * 32, 16, 1024);
            const uint64_t b_desc = B_MN ? sw128_desc(b_addr + k * 2048, CHUNK_BYTES, 1024)
                                         : sw128_desc(b_addr + k * 32, 16, 1024);
            umma_bf16<CL>(d_tmem, a_desc, b_desc, idesc, (kb != g.kb0 || k != 0) ? 1u : 0u);
          }
          issued = true;
          umma_commit_all<CL>(empty_bar(stage));  // frees the stage in every CTA of the pair
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_all<CL>(tfull_bar(buf));  // accumulators ready for both CTAs' epilogues
      }
      if (issued) {
        umma_commit<CL>(drain_bar);  // all MMAs retired before TMEM is freed
        wait_bounded(drain_bar, 0, wc, false);
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue warps
    const int quarter = warp & 3;
    const int part = (warp - 2) >> 2;  // 0 or 1: which of every 2 units
    const uint32_t staging_warp = staging0 + (warp - 2) * STAGING_BYTES_PER_WARP;
    const uint32_t sw64 = (lane >> 1) & 3u;  // 64-byte rows, 64-byte swizzle
    uint32_t stage_sel = 0;
    int turn = 0;
    int it = 0;
    // stage a [32 rows][16 words] block (one 64-byte row per lane)
    auto stage_rows = [&](const uint32_t (&w)[16]) -> uint32_t {
      const uint32_t stg = staging_warp + (stage_sel & 1) * 2048;
      ++stage_sel;
      if (lane == 0) bulk_wait_read_1();
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(stg + lane * 64 + ((q ^ sw64) << 4), w[4 * q], w[4 * q + 1], w[4 * q + 2],
                     w[4 * q + 3]);
      fence_async_shared();
      __syncwarp();
      return stg;
    };
    for (int64_t u = first_unit; u < p.num_units; u += unit_step, ++it) {
      const int buf = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const int okw = wait_bounded(tfull_bar(buf), acc_phase, wc, true) ? 1 : 0;
      if (!__all_sync(0xFFFFFFFFu, okw)) break;
      tc_fence_after();
      const Geo g = unit_geo<CL>(p, u, rank);
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * ACC_COLS;
      int oc[3];
      if (MODE != BWD_DW) outer_coords(p.tok, g.o, oc);
      const int row0 = quarter * 32;  // the warp's first row in the tile
      if (MODE == BWD_DW) {
        // fp32 partial tile, 16 columns per unit, added into dW
        for (int c = 0; c < BN; c += 16) {
          const bool mine = turn == part;
          turn ^= 1;
          if (!mine) continue;
          uint32_t v[16];
          tmem_ld16(t_row + c, v);
          tmem_wait_ld();
          // a store never starts past the tensor (loads may; stores are clipped, not skipped)
          if (g.phantom || g.c0 + c >= p.N || g.r0 + row0 >= p.C) continue;
          const uint32_t stg = stage_rows(v);
          if (lane == 0) {
            tma_reduce_add_2d(&p.tmap_out, stg, g.c0 + c, g.r0 + row0);
            bulk_commit();
          }
        }
      } else {
        const int s = g.s0 + row0 + lane;  // GRADFF/DX: this lane's token in its slab
        const bool valid = (MODE == BWD_DXT) || s < p.tok.S_in;
        const int64_t m = static_cast<int64_t>(g.o) * p.tok.S_in + s;
        for (int c = 0; c < BN; c += 32) {
          const bool mine = turn == part;
          turn ^= 1;
          if (!mine) continue;
          uint32_t v[32];
          tmem_ld32(t_row + c, v);
          tmem_wait_ld();
          // a store never starts past the tensor (its far edge is clipped by TMA)
          if (g.phantom) continue;
          if (MODE == BWD_GRADFF && (g.c0 + c >= p.F || g.s0 + row0 >= p.tok.S_in)) continue;
          if (MODE == BWD_DX && (g.c0 + c >= p.C || g.s0 + row0 >= p.tok.S_in)) continue;
          if (MODE == BWD_DXT && (g.s0 + c >= p.tok.S_in || g.r0 + row0 >= p.C)) continue;
          uint32_t w[16];
          if (MODE == BWD_GRADFF) {
            const int n = g.c0 + c;  // first ff column of the unit
            float y[32], gg[32];
            const uint16_t* bias = static_cast<const uint16_t*>(p.bias);
            if (bias && n + 32 <= p.N) {
              load32_bf16(bias + n, y);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                y[i] = (bias && n + i < p.N) ? bf16_bits_to_float(bias[n + i]) : 0.0f;
            }
            const uint16_t* grow = static_cast<const uint16_t*>(p.g_ff) + m * p.F + n;
            if (valid && n + 32 <= p.F) {
              load32_bf16(grow, gg);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                gg[i] = (valid && n + i < p.F) ? bf16_bits_to_float(grow[i]) : 0.0f;
            }
            if (ACT == ACT_GELU_ERF) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float d0, d1;
                gelu_erf_deriv2(__uint_as_float(v[2 * i]) + y[2 * i],
                                __uint_as_float(v[2 * i + 1]) + y[2 * i + 1], d0, d1);
                gg[2 * i] *= d0;
                gg[2 * i + 1] *= d1;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) gg[i] *= act_deriv<ACT>(__uint_as_float(v[i]) + y[i]);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(gg[2 * i], gg[2 * i + 1]);
            if (p.db) {
              const float cs = column_sum32(gg, lane);
              if (n + lane < p.F) atomicAdd(p.db + n + lane, cs);
            }
            const uint32_t stg = stage_rows(w);
            if (lane == 0) {  // [n_outer][S_in][F] view of G's ff columns: clips at S_in, F
              tma_store_3d(&p.tmap_out, stg, n, g.s0 + row0, g.o);
              bulk_commit();
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            const uint32_t stg = stage_rows(w);
            if (lane == 0) {
              if (MODE == BWD_DX)  // x token-major: [channels][tokens] box at (channel, token)
                tma_store_5d(&p.tmap_out, stg, g.c0 + c, g.s0 + row0, oc[0], oc[1], oc[2]);
              else                 // x channels-first: [tokens][channels] box at (token, channel)
                tma_store_5d(&p.tmap_out, stg, g.s0 + c, g.r0 + row0, oc[0], oc[1], oc[2]);
              bulk_commit();
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
    if (lane == 0) bulk_wait_all();
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

template <int MODE, bool A_MN, bool B_MN, int ACT, int CL = 1>
cudaError_t launch_one(const BwdGemmParams& p, int num_ctas, cudaStream_t stream) {
  static_assert(MODE != BWD_GRADFF || CL == 1, "the ff-gradient fallback runs single CTAs");
  auto kernel = bwd_gemm_kernel<MODE, A_MN, B_MN, ACT, CL>;
  constexpr int smem = BwdCfg<CL>::SMEM_BYTES;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !attr_done[dev]) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    if (dev < 64) attr_done[dev] = 1;
  }
  // whole clusters, no more than there are work items (a unit is one cluster's)
  int64_t ctas = num_ctas / CL * CL;
  if (ctas > p.num_units * CL) ctas = p.num_units * CL;
  if (ctas < CL) ctas = CL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL > 1 ? 2 : 1;
  err = cudaLaunchKernelEx(&cfg, kernel, p);
  return err != cudaSuccess ? err : cudaGetLastError();
}

template <bool A_MN>
cudaError_t launch_gradff(const BwdGemmParams& p, int num_ctas, cudaStream_t stream) {
  switch (p.act) {
    case ACT_GELU_ERF: return launch_one<BWD_GRADFF, A_MN, true, ACT_GELU_ERF>(p, num_ctas, stream);
    case ACT_GELU_TANH: return launch_one<BWD_GRADFF, A_MN, true, ACT_GELU_TANH>(p, num_ctas, stream);
    case ACT_SILU: return launch_one<BWD_GRADFF, A_MN, true, ACT_SILU>(p, num_ctas, stream);
    case ACT_RELU2: return launch_one<BWD_GRADFF, A_MN, true, ACT_RELU2>(p, num_ctas, stream);
    default: return launch_one<BWD_GRADFF, A_MN, true, ACT_NONE>(p, num_ctas, stream);
  }
}

// ------------------------------------------------------------------ q/k/v gather

// Two gather kernels, both over blocks of 256 threads in token rows (thread
// row y takes tokens y, y + rows, ...), each block staging its slice of the
// rotary table in shared memory and adding its column sums into db once:
//  - bwd_gather_pairs_kernel (16-byte path): a thread owns 16 columns of one
//    head, the rotation pair (j .. j+7, j+rh .. j+rh+7) or two adjacent
//    unrotated groups, so each token costs it two 16-byte loads and two
//    16-byte stores and no partner is loaded twice;
//  - bwd_gather_kernel (lane by lane): 8 columns per thread, element loads,
//    8 rows of 32 threads, 8 tokens per thread; pre-transposed k, or a
//    rotated half-width that is not a multiple of 8.
// Both issue all of a thread's loads before the table fill and its barrier,
// so the two are in flight together. q and k are rotated back with the transpose
// of the rotation.
constexpr int GATHER_ROWS = 8;     // token rows of threads per block
constexpr int GATHER_PER_ROW = 8;  // tokens per thread
constexpr int GATHER_TOKENS = GATHER_ROWS * GATHER_PER_ROW;

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// The block's slice of the frequency-major rotary table, token-major in
// shared memory (row r = the block's token r, tab_ld entries apart). Thread
// tid of 256 always fills token tid % TOKENS, frequencies tid / TOKENS,
// + 256 / TOKENS, ...: consecutive threads read consecutive tokens of one
// frequency row, and the wrap of the position and the source address are
// worked out once.
template <int TOKENS>
__device__ __forceinline__ void fill_table_slice(float2* tab, int tab_ld, const float2* cs,
                                                 int64_t T, int64_t M, int64_t mblk, int rh,
                                                 int tid) {
  static_assert(256 % TOKENS == 0, "a whole number of frequencies per pass");
  constexpr int FSTEP = 256 / TOKENS;
  const int r = tid % TOKENS;
  if (mblk + r >= M) return;
  int64_t t = mblk % T + r;
  if (t >= T) t = T >= TOKENS ? t - T : t % T;
  const int f0 = tid / TOKENS;
  const float2* src = cs + f0 * T + t;
  float2* dst = tab + r * tab_ld + f0;
  const int64_t sstep = FSTEP * T;
#pragma unroll 4
  for (int f = f0; f < rh; f += FSTEP, src += sstep, dst += FSTEP) *dst = __ldg(src);
}

__global__ void __launch_bounds__(32 * GATHER_ROWS, 2) bwd_gather_kernel(const BwdGatherParams p) {
  __shared__ __align__(16) float part[GATHER_ROWS][32][8];
  // the block's slice of the frequency-major rotary table, token-major here
  // ([64 tokens][rope_half + 2]): filled by runs of consecutive tokens per
  // frequency, read by a warp as different frequencies of one token
  extern __shared__ __align__(16) float2 tab[];
  const int nq = p.N - p.F;
  const int col0 = (blockIdx.x * 32 + threadIdx.x) * 8;  // first of 8 columns
  const bool active = col0 < nq;
  int seg = 3, head = 0, j0 = 0;
  if (active) {
    if (p.groups > 0) {
      const int qpk = p.heads / p.groups;
      const int per = (qpk + 2) * p.hd;
      const int gidx = col0 / per, r = col0 - gidx * per, slot = r / p.hd;
      j0 = r - slot * p.hd;
      if (slot < qpk) {
        seg = 1;
        head = gidx * qpk + slot;
      } else {
        seg = slot == qpk ? 2 : 3;
        head = gidx;
      }
    } else {
      seg = 1 + col0 / p.C;
      const int r = col0 - (seg - 1) * p.C;
      head = r / p.hd;
      j0 = r - head * p.hd;
    }
  }
  const int nkv = p.groups > 0 ? p.groups : p.heads;
  const int rh = p.rope_half;
  const bool rot = rh > 0 && seg < 3 && j0 < 2 * rh;
  const bool kt = seg == 2 && p.k_transposed;
  const uint16_t* src = static_cast<const uint16_t*>(seg == 1 ? p.g_q : seg == 2 ? p.g_k : p.g_v);
  const int nh = seg == 1 ? p.heads : nkv;
  uint16_t* G = static_cast<uint16_t*>(p.G);
  float sum[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) sum[i] = 0.0f;
  const int64_t mblk = static_cast<int64_t>(blockIdx.y) * GATHER_TOKENS;
  const int64_t mb = mblk + threadIdx.y;
  // the thread's tokens mb, mb + ROWS, ...: batch element and position walked
  // from one division
  int64_t roff[GATHER_PER_ROW];  // element offset of the token's row of its head
  int tt[GATHER_PER_ROW];        // position of the token in its batch element
  {
    int64_t bb = mb / p.T;
    int64_t t = mb - bb * p.T;
#pragma unroll
    for (int k = 0; k < GATHER_PER_ROW; ++k) {
      tt[k] = static_cast<int>(t);
      roff[k] = ((bb * nh + head) * p.T + t) * p.hd;
      t += GATHER_ROWS;
      while (t >= p.T) {
        t -= p.T;
        ++bb;
      }
    }
  }
  // table rows are rh + 2 entries apart: 16-byte aligned, and the fill's
  // token-strided stores fall in distinct bank pairs
  const int tab_ld = rh + 2;
  if (rh > 0) {
    fill_table_slice<GATHER_TOKENS>(tab, tab_ld, p.rope_cs, p.T, p.M, mblk, rh,
                                    threadIdx.y * 32 + threadIdx.x);
    __syncthreads();
  }
#pragma unroll
  for (int k = 0; k < GATHER_PER_ROW && active; ++k) {
    const int64_t m = mb + static_cast<int64_t>(k) * GATHER_ROWS;
    if (m >= p.M) continue;
    const int t = tt[k];
    // pre-transposed k is [B*kv, hd, T]
    const int64_t hrow = (m / p.T) * nh + head;
    float g[8], gp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = j0 + i;
      const int jp = j < rh ? j + rh : j - rh;
      const int64_t ij = kt ? (hrow * p.hd + j) * p.T + t : roff[k] + j;
      const int64_t ip = kt ? (hrow * p.hd + jp) * p.T + t : roff[k] + jp;
      g[i] = bf16_bits_to_float(src[ij]);
      gp[i] = (rot && j < 2 * rh) ? bf16_bits_to_float(src[ip]) : 0.0f;
    }
    if (rot) {
      const float2* cs = tab + (threadIdx.y + k * GATHER_ROWS) * tab_ld;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = j0 + i;
        if (j < 2 * rh) {
          const float2 c = cs[j < rh ? j : j - rh];
          g[i] = j < rh ? fmaf(g[i], c.x, gp[i] * c.y) : fmaf(g[i], c.x, -gp[i] * c.y);
        }
      }
    }
    uint4 o;
    o.x = pack_bf16x2(g[0], g[1]);
    o.y = pack_bf16x2(g[2], g[3]);
    o.z = pack_bf16x2(g[4], g[5]);
    o.w = pack_bf16x2(g[6], g[7]);
    *reinterpret_cast<uint4*>(G + m * p.N + p.F + col0) = o;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum[i] += g[i];
  }
  if (!p.db) return;  // uniform across the block
  float4* mine = reinterpret_cast<float4*>(part[threadIdx.y][threadIdx.x]);
  mine[0] = make_float4(sum[0], sum[1], sum[2], sum[3]);
  mine[1] = make_float4(sum[4], sum[5], sum[6], sum[7]);
  __syncthreads();
  if (threadIdx.y == 0 && active) {
    float acc[8] = {};
#pragma unroll
    for (int r = 0; r < GATHER_ROWS; ++r) {
      const float4* q = reinterpret_cast<const float4*>(part[r][threadIdx.x]);
      const float4 a = q[0], b = q[1];
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) atomicAdd(p.db + p.F + col0 + i, acc[i]);
  }
}

// 16-byte path. Every head's hd columns split into hd / 16 items of 16
// columns: for a rotated head (q, k with rh > 0) items 0 .. rh/8 - 1 are the
// rotation pairs (j .. j+7, j+rh .. j+rh+7), j = 8 i, and the rest pairs of
// adjacent groups past the rotated part; for v (or no rotation) every item is
// two adjacent groups. Heads lie side by side in G's q|k|v columns in both
// column orders, so item k covers G columns F + 16 k .. with a per-item offset
// of its second group. Needs hd % 16 == 0, rh % 8 == 0, k not pre-transposed.
// XW items per token row of threads (32 or 16), 256 / XW token rows, TPT
// tokens per thread.
template <int XW, int TPT>
__global__ void __launch_bounds__(256, TPT == 4 ? 3 : 2)
    bwd_gather_pairs_kernel(const BwdGatherParams p) {
  constexpr int ROWS = 256 / XW;
  constexpr int TOKENS = ROWS * TPT;
  // the block's slice of the rotary table ([64 tokens][rope_half + 2]), then
  // (after a barrier) the token rows' column sums [ROWS][XW threads][16]
  extern __shared__ __align__(16) float2 tab[];
  const int hd = p.hd, rh = p.rope_half;
  const int per_head = hd / 16;
  const int n_items = (p.N - p.F) / 16;
  const int item = blockIdx.x * XW + threadIdx.x;
  const bool active = item < n_items;
  const int hall = active ? item / per_head : 0;  // head in G's q|k|v order
  const int i = item - hall * per_head;
  int seg, head;
  if (p.groups > 0) {
    const int qpk = p.heads / p.groups;
    const int g = hall / (qpk + 2), slot = hall - g * (qpk + 2);
    seg = slot < qpk ? 0 : slot == qpk ? 1 : 2;
    head = slot < qpk ? g * qpk + slot : g;
  } else {
    seg = hall / p.heads;
    head = hall - seg * p.heads;
  }
  const int nrot = seg < 2 ? rh / 8 : 0;  // rotation pairs in this head
  const bool rot = i < nrot;
  const int ja = rot ? 8 * i : 16 * nrot + 16 * (i - nrot);  // first group's column
  const int jb = rot ? ja + rh : ja + 8;                     // second group's column
  const uint16_t* src = static_cast<const uint16_t*>(seg == 0 ? p.g_q : seg == 1 ? p.g_k : p.g_v);
  const int nh = seg == 0 ? p.heads : (p.groups > 0 ? p.groups : p.heads);
  uint16_t* const Gcol = static_cast<uint16_t*>(p.G) + p.F + static_cast<int64_t>(hall) * hd;
  const int64_t mblk = static_cast<int64_t>(blockIdx.y) * TOKENS;
  const int64_t mb = mblk + threadIdx.y;
  // all TPT tokens' loads before the table fill: batch element and position
  // walked from one division
  uint4 va[TPT], vb[TPT];
  {
    int64_t bb = mb / p.T;
    int64_t t = mb - bb * p.T;
#pragma unroll
    for (int k = 0; k < TPT; ++k) {
      va[k] = make_uint4(0, 0, 0, 0);
      vb[k] = make_uint4(0, 0, 0, 0);
      if (active && mb + static_cast<int64_t>(k) * ROWS < p.M) {
        const uint16_t* row = src + ((bb * nh + head) * p.T + t) * hd;
        va[k] = *reinterpret_cast<const uint4*>(row + ja);
        vb[k] = *reinterpret_cast<const uint4*>(row + jb);
      }
      t += ROWS;
      while (t >= p.T) {
        t -= p.T;
        ++bb;
      }
    }
  }
  // rows rh + 2 entries apart: 16-byte aligned, and the fill's token-strided
  // stores fall in distinct bank pairs
  const int tab_ld = rh + 2;
  if (rh > 0) {
    fill_table_slice<TOKENS>(tab, tab_ld, p.rope_cs, p.T, p.M, mblk, rh,
                             threadIdx.y * XW + threadIdx.x);
    __syncthreads();
  }
  float sa[8], sb[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) sa[q] = sb[q] = 0.0f;
#pragma unroll
  for (int k = 0; k < TPT; ++k) {
    const int64_t m = mb + static_cast<int64_t>(k) * ROWS;
    if (!active || m >= p.M) continue;
    float a[8], b[8];
    unpack8(va[k], a);
    unpack8(vb[k], b);
    if (rot) {
      // (cos, sin) of frequencies ja .. ja + 7: the transpose of the rotation,
      // a' = a c + b s, b' = b c - a s
      const float4* c4 =
          reinterpret_cast<const float4*>(tab + (threadIdx.y + k * ROWS) * tab_ld + ja);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 c = c4[q];
        const float a0 = a[2 * q], b0 = b[2 * q], a1 = a[2 * q + 1], b1 = b[2 * q + 1];
        a[2 * q] = fmaf(a0, c.x, b0 * c.y);
        b[2 * q] = fmaf(b0, c.x, -a0 * c.y);
        a[2 * q + 1] = fmaf(a1, c.z, b1 * c.w);
        b[2 * q + 1] = fmaf(b1, c.z, -a1 * c.w);
      }
    }
    uint16_t* const grow = Gcol + m * p.N;
    *reinterpret_cast<uint4*>(grow + ja) =
        make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                   pack_bf16x2(a[6], a[7]));
    *reinterpret_cast<uint4*>(grow + jb) =
        make_uint4(pack_bf16x2(b[0], b[1]), pack_bf16x2(b[2], b[3]), pack_bf16x2(b[4], b[5]),
                   pack_bf16x2(b[6], b[7]));
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      sa[q] += a[q];
      sb[q] += b[q];
    }
  }
  if (!p.db) return;  // uniform across the block
  // column sums: the table slice is dead, its space takes the partial sums
  if (rh > 0) __syncthreads();
  float4* part = reinterpret_cast<float4*>(tab);
  float4* mine = part + (threadIdx.y * XW + threadIdx.x) * 4;
  mine[0] = make_float4(sa[0], sa[1], sa[2], sa[3]);
  mine[1] = make_float4(sa[4], sa[5], sa[6], sa[7]);
  mine[2] = make_float4(sb[0], sb[1], sb[2], sb[3]);
  mine[3] = make_float4(sb[4], sb[5], sb[6], sb[7]);
  __syncthreads();
  if (threadIdx.y == 0 && active) {
    float acc[16] = {};
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const float4* q4 = part + (r * XW + threadIdx.x) * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = q4[q];
        acc[4 * q] += v.x;
        acc[4 * q + 1] += v.y;
        acc[4 * q + 2] += v.z;
        acc[4 * q + 3] += v.w;
      }
    }
    float* const dcol = p.db + p.F + static_cast<int64_t>(hall) * hd;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      atomicAdd(dcol + ja + q, acc[q]);
      atomicAdd(dcol + jb + q, acc[8 + q]);
    }
  }
}

}  // namespace

cudaError_t launch_bwd_gemm(const BwdGemmParams& p, bool a_mn_major, int num_ctas,
                            cudaStream_t stream) {
  switch (p.mode) {
    case BWD_GRADFF:
      return a_mn_major ? launch_gradff<true>(p, num_ctas, stream)
                        : launch_gradff<false>(p, num_ctas, stream);
    case BWD_DX:
      return p.cluster == 2 ? launch_one<BWD_DX, false, false, ACT_NONE, 2>(p, num_ctas, stream)
                            : launch_one<BWD_DX, false, false, ACT_NONE, 1>(p, num_ctas, stream);
    case BWD_DXT:
      return p.cluster == 2 ? launch_one<BWD_DXT, false, false, ACT_NONE, 2>(p, num_ctas, stream)
                            : launch_one<BWD_DXT, false, false, ACT_NONE, 1>(p, num_ctas, stream);
    default:
      if (p.cluster == 2)
        return a_mn_major ? launch_one<BWD_DW, true, true, ACT_NONE, 2>(p, num_ctas, stream)
                          : launch_one<BWD_DW, false, true, ACT_NONE, 2>(p, num_ctas, stream);
      return a_mn_major ? launch_one<BWD_DW, true, true, ACT_NONE, 1>(p, num_ctas, stream)
                        : launch_one<BWD_DW, false, true, ACT_NONE, 1>(p, num_ctas, stream);
  }
}

cudaError_t launch_bwd_gather(const BwdGatherParams& p, cudaStream_t stream) {
  const int nq = p.N - p.F;
  if (nq <= 0 || p.M == 0) return cudaSuccess;
  if (!p.k_transposed && p.rope_half % 8 == 0 && p.hd % 16 == 0 && nq % 16 == 0) {
    // 16-byte path: 32 items a row of threads; 16 when there is no rotary
    // table and the count is an odd multiple of 16 (with a table, 16-wide
    // blocks fill twice the table per thread and share it over half the
    // heads: walrus 74 us against 66 us for 32-wide blocks, the last of them
    // half idle); 4 tokens a thread when 8 would leave fewer than 8 blocks per
    // SM, or when the table has 64 or more frequencies (its fill and shared
    // memory grow with the tokens of a block: the LLM shape's gather, rh 64,
    // 91 us at 8 tokens against 79 us at 4; walrus, rh 32, 53 against 80)
    const int n_items = nq / 16;
    const int xw = p.rope_half == 0 && n_items % 32 == 16 ? 16 : 32;
    static int sms = 0;
    if (sms == 0) {
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 152;
    }
    const int64_t x_blocks = (n_items + xw - 1) / xw;
    const int64_t tok8 = (256 / xw) * 8;
    const int tpt =
        x_blocks * ((p.M + tok8 - 1) / tok8) < 8LL * sms || p.rope_half >= 64 ? 4 : 8;
    const int64_t tokens = (256 / xw) * tpt;
    const dim3 grid2(static_cast<unsigned>(x_blocks),
                     static_cast<unsigned>((p.M + tokens - 1) / tokens));
    // shared memory: the table slice, later the 16 column sums of 256 threads
    const size_t tab_bytes =
        p.rope_half > 0 ? static_cast<size_t>(p.rope_half + 2) * tokens * sizeof(float2) : 0;
    const size_t smem = std::max<size_t>(tab_bytes, 256 * 16 * sizeof(float));
    auto go = [&](auto kernel) {
      if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(
            kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
      }
      kernel<<<grid2, dim3(xw, 256 / xw), smem, stream>>>(p);
      return cudaSuccess;
    };
    cudaError_t e;
    if (xw == 32)
      e = tpt == 8 ? go(bwd_gather_pairs_kernel<32, 8>) : go(bwd_gather_pairs_kernel<32, 4>);
    else
      e = tpt == 8 ? go(bwd_gather_pairs_kernel<16, 8>) : go(bwd_gather_pairs_kernel<16, 4>);
    if (e != cudaSuccess) return e;
  } else {
    const dim3 grid((nq / 8 + 31) / 32,
                    static_cast<unsigned>((p.M + GATHER_TOKENS - 1) / GATHER_TOKENS));
    const size_t tab_bytes =
        p.rope_half > 0 ? static_cast<size_t>(p.rope_half + 2) * GATHER_TOKENS * sizeof(float2) : 0;
    if (tab_bytes > 48 * 1024) return cudaErrorInvalidValue;  // rope_half <= 64 (head_dim <= 128)
    bwd_gather_kernel<<<grid, dim3(32, GATHER_ROWS), tab_bytes, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace fp
