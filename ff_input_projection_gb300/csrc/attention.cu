// Softmax attention over the fused projection's q, k, v on the 5th-generation
// tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes, per batch*head index z and query i:
//     out[z, i, :] = sum_t softmax_t(scale * q[z, i, :] . k[z', t, :]) v[z', t, :]
// in the [batch*heads, tokens, head_dim] layout of memory-efficient-attention
// issue #7 ("Improve performance via batched-matmul and fused multiplies"):
// its baddbmm (the scaled scores q k^T, the scale fused into the multiply),
// the softmax over the keys and its bmm with the values, chunked as that page
// chunks them. Each CTA takes one chunk of 128 queries and walks the keys in
// chunks of 128, merging the chunks under the running row maximum; with 128
// keys or fewer there is a single key chunk and nothing to merge (the page's
// fast path). k arrives pre-transposed, [batch*heads, head_dim, tokens] (the
// same page's comments on transposing the key once), or as [batch*heads,
// tokens, head_dim]. z' is the k/v head of query head z: grouped-query
// layouts share one k/v head among heads / kv_heads query heads.
//
// Work: 128-query blocks of one (batch, head) each; the blocks past the last
// whole wave of SMs are split along the keys (up to 16 ranges each, partial
// results merged by a second kernel). The kernel is persistent: one CTA per SM
// (8 warps) walks its units in turn, its pipelines running on across unit
// boundaries.
// Structure:
//   warp 0     TMA producer: a unit's q chunk once, then k and v chunks into
//              rings of 4 stages (head_dim 64) or 2 (head_dim 128)
//   warp 1     score MMAs (one thread): S = q k^T into one of NS TMEM score
//              buffers (M 128, N 128, K head_dim), as far ahead as the buffers
//              allow (a buffer is reused once its previous chunk's P v is done)
//   warp 2     P v MMAs (one thread): O += P v into the unit's TMEM output
//              accumulator (M 128, N head_dim, K 128) with P read from tensor
//              memory. Two issuing threads: one thread issuing both measured
//              about 100 cycles per instruction of these thin shapes
//   warps 4-7  softmax, one query row per thread (TMEM lane = row): scores
//              from TMEM, a reference maximum m and the sum l, P = 2^(s c - m)
//              rounded to bf16 and written back over the chunk's scores in
//              TMEM, two keys per 32-bit column (the A operand of P v: no
//              shared-memory store and no proxy fence on the chain). m is
//              raised only when a chunk's maximum exceeds it by more than 8
//              (log2 units): P then stays below 2^8, and the output
//              accumulator is rescaled in TMEM only at those rare steps. At the
//              end of a unit O / l is rounded to bf16 and stored.
// Shared-memory operands (q, k, v) use the 128-byte swizzle TMA writes and the
// MMA reads.
// Every mbarrier wait is bounded: a wait that runs out records a timeout in
// the status word, tags the launch as aborted, drains its own copies and MMAs
// and returns, so the GPU stays usable.
#include <algorithm>

#include "epilogue.cuh"
#include "fp_internal.h"
#include "tc_ptx.cuh"

namespace fp {
namespace {

// max(a, b, c): one three-input max instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

constexpr int QB = 128;   // queries per CTA: one per softmax thread and TMEM lane
constexpr int KB = 128;   // keys per chunk: the N of S and the K of P v
constexpr int ANT = 256;  // 8 warps
constexpr int ATOM = QB * 128;  // a [128 rows][64 bf16] 128-byte-swizzled atom: 16 KB
constexpr int CHUNK = 64 * 128; // a [64 rows][64 bf16] atom: 8 KB

template <int HD>
struct ACfg {
  // k and v stages: a chunk's loads are requested about one chunk's softmax
  // ahead of their use, less than the L2 latency under load, so the ring is
  // as deep as shared memory allows
  static constexpr int RING = HD == 64 ? 4 : 2;
  static constexpr int Q_BYTES = QB * HD * 2;
  static constexpr int K_BYTES = KB * HD * 2;
  static constexpr int V_BYTES = KB * HD * 2;
  // score buffers in TMEM (each also holds its chunk's P): three for
  // head_dim 64, so the scores can be issued two chunks ahead; two for 128
  static constexpr int NS = HD == 64 ? 3 : 2;
  // q full/empty; k full/empty and v full/empty per stage; s full/empty,
  // p full and P v done per score buffer; output empty per output buffer;
  // a drain per MMA-issuing thread
  static constexpr int NUM_BARS = 2 + 4 * RING + 4 * NS + 2 + 2;
  static_assert(1 + 2 * RING <= 32, "armed-barrier bit masks hold 1 + 2 * RING slots");
  static constexpr int SMEM_BYTES =
      1024 + Q_BYTES + RING * (K_BYTES + V_BYTES) + NUM_BARS * 8 + 16;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  // TMEM: scores in [0, NS * 128), the two output buffers after them
  static constexpr int O_COL = NS * KB;
  static_assert(O_COL + 2 * HD <= 512, "TMEM holds 512 columns");
};

// One work unit: a whole 128-query block (units [0, full)), or one key range
// of a block of the split tail (chunks [j0, j0 + nkb) of its keys, partial
// results into slot `slot`).
struct Unit {
  int z, zkv, q0, j0, nkb, slot;
};

__device__ __forceinline__ Unit unit_of(const AttnParams& p, int u, int nkb_all) {
  Unit w;
  int qb = u;
  w.j0 = 0;
  w.nkb = nkb_all;
  w.slot = -1;
  if (qb >= p.full) {
    const int r = (qb - p.full) / p.splits, sp = qb - p.full - r * p.splits;
    w.j0 = static_cast<int>(static_cast<int64_t>(sp) * nkb_all / p.splits);
    w.nkb = static_cast<int>(static_cast<int64_t>(sp + 1) * nkb_all / p.splits) - w.j0;
    w.slot = r * p.splits + sp;
    qb = p.full + r;
  }
  w.z = qb / p.num_q_blocks;
  w.q0 = (qb - w.z * p.num_q_blocks) * QB;
  const int qpk = p.heads / p.kv_heads;
  w.zkv = (w.z / p.heads) * p.kv_heads + (w.z % p.heads) / qpk;
  return w;
}

// Persistent: one CTA per SM walks units u = blockIdx.x, + gridDim.x, ...
// Every role counts the key chunks it has passed over all its units (g): the
// k/v ring stage and phase, the score and P buffer (g mod NS) and their phases
// (g / NS) follow from it, so the pipelines run on across unit boundaries.
// Unit i of a CTA accumulates into output buffer i & 1, so its MMAs can start
// while the softmax warps still store the output of unit i - 1.
template <int HD, bool KT>
__global__ void __launch_bounds__(ANT, 1) attention_kernel(const __grid_constant__ AttnParams p) {
  using G = ACfg<HD>;
  constexpr int RING = G::RING;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - raw);
  const uint32_t q_s = sbase;
  const uint32_t k_s = q_s + G::Q_BYTES;                   // RING stages
  const uint32_t v_s = k_s + RING * G::K_BYTES;            // RING stages
  const uint32_t bar0 = v_s + RING * G::V_BYTES;
  const uint32_t q_full = bar0;
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (1 + RING + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * RING + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (1 + 3 * RING + s); };
  const uint32_t bar1 = bar0 + 8u * (1 + 4 * RING);
  constexpr int NS = G::NS;
  auto s_full = [&](int b) { return bar1 + 8u * b; };
  auto s_empty = [&](int b) { return bar1 + 8u * (NS + b); };
  // P of the chunk in score buffer b: written once the softmax stored it over
  // the scores, read once P v has completed
  auto p_full = [&](int b) { return bar1 + 8u * (2 * NS + b); };
  auto pv_done = [&](int b) { return bar1 + 8u * (3 * NS + b); };
  const uint32_t drain = bar1 + 8u * (4 * NS);
  const uint32_t q_empty = bar1 + 8u * (4 * NS + 1);  // the unit's score MMAs read q
  auto o_empty = [&](int b) { return bar1 + 8u * (4 * NS + 2 + b); };  // output buffer b stored
  const uint32_t drain_pv = bar1 + 8u * (4 * NS + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sptr + (bar1 + 8u * (4 * NS + 5) - sbase));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl wc{p.status, p.wait_limit_ns, p.launch_tag};
  const int nkb_all = static_cast<int>((p.Tk + KB - 1) / KB);
  const int n_units = p.full + (p.BH * p.num_q_blocks - p.full) * p.splits;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < RING; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int b = 0; b < NS; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_empty(b), 4);  // the four softmax warps
      mbar_init(p_full(b), 4);
      mbar_init(pv_done(b), 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(o_empty(b), 4);
    mbar_init(drain, 1);
    mbar_init(drain_pv, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    prefetch_tmap(&p.tmap_q);
    prefetch_tmap(&p.tmap_k);
    prefetch_tmap(&p.tmap_v);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t armed = 0, armed_par = 0;  // bit per barrier slot: 0 q, 1+s k, 1+RING+s v
      auto arm = [&](int slot, uint32_t par) {
        armed |= 1u << slot;
        armed_par = (armed_par & ~(1u << slot)) | (par << slot);
      };
      bool aborted = false;
      int g = 0, ui = 0;  // chunks and units this CTA has passed
      for (int u = static_cast<int>(blockIdx.x); u < n_units && !aborted;
           u += static_cast<int>(gridDim.x), ++ui) {
        const Unit w = unit_of(p, u, nkb_all);
        // the q buffer is free once the previous unit's score MMAs have read it
        if (ui > 0 && !wait_bounded(q_empty, (ui - 1) & 1, wc, true)) break;
        mbar_arrive_expect_tx(q_full, G::Q_BYTES);
#pragma unroll
        for (int a = 0; a < HD / 64; ++a)
          tma_load_3d(q_s + a * ATOM, &p.tmap_q, q_full, 64 * a, w.q0, w.z);
        arm(0, ui & 1);
        for (int j = 0; j < w.nkb; ++j, ++g) {
          const int s = g % RING;
          const uint32_t ph = (g / RING) & 1;
          const int key0 = (w.j0 + j) * KB;
          if (!wait_bounded(k_empty(s), ph ^ 1u, wc, true)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(k_full(s), G::K_BYTES);
          const uint32_t kd = k_s + s * G::K_BYTES;
          if (KT) {
            // [hd][Tk] rows of the head: chunk (h, n) holds hd rows 64h.. and keys 64n..
#pragma unroll
            for (int h = 0; h < HD / 64; ++h)
#pragma unroll
              for (int n = 0; n < 2; ++n)
                tma_load_3d(kd + (h * 2 + n) * CHUNK, &p.tmap_k, k_full(s), key0 + 64 * n, 64 * h,
                            w.zkv);
          } else {
#pragma unroll
            for (int a = 0; a < HD / 64; ++a)
              tma_load_3d(kd + a * ATOM, &p.tmap_k, k_full(s), 64 * a, key0, w.zkv);
          }
          arm(1 + s, ph);
          if (!wait_bounded(v_empty(s), ph ^ 1u, wc, true)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(v_full(s), G::V_BYTES);
          const uint32_t vd = v_s + s * G::V_BYTES;
          // chunk (h, n) holds keys 64h.. and head lanes 64n..
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int n = 0; n < HD / 64; ++n)
              tma_load_3d(vd + (h * (HD / 64) + n) * CHUNK, &p.tmap_v, v_full(s), 64 * n,
                          key0 + 64 * h, w.zkv);
          arm(1 + RING + s, ph);
        }
      }
      // no copy may still be landing in shared memory when the CTA exits
      const WaitCtl dc{wc.status, wc.limit_ns < 10000000ull ? wc.limit_ns : 10000000ull,
                       wc.launch_tag};
      if (armed & 1u) wait_bounded(q_full, armed_par & 1u, dc, false);
      for (int s = 0; s < RING; ++s) {
        if (armed & (1u << (1 + s))) wait_bounded(k_full(s), (armed_par >> (1 + s)) & 1u, dc, false);
        if (armed & (1u << (1 + RING + s)))
          wait_bounded(v_full(s), (armed_par >> (1 + RING + s)) & 1u, dc, false);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------ MMA issuers: warp 1 the
    // scores, warp 2 the P v products (different TMEM accumulators; each
    // thread's commits track its own MMAs)
    if (lane == 0) {
      const bool scores = warp == 1;
      const uint32_t idesc_s = make_idesc(false, KT, QB, KB);
      const uint32_t idesc_o = make_idesc(false, true, QB, HD);
      bool issued = false, ok = true;
      int g = 0, ui = 0;  // chunks and units this CTA has passed
      for (int u = static_cast<int>(blockIdx.x); ok && u < n_units;
           u += static_cast<int>(gridDim.x), ++ui) {
        const Unit w = unit_of(p, u, nkb_all);
        const int g0 = g;
        if (scores) {
          ok = wait_bounded(q_full, ui & 1, wc, true);
          tc_fence_after();
          for (int j = 0; ok && j < w.nkb; ++j) {
            // S for global chunk gj into score buffer gj mod NS, once the
            // buffer's previous chunk is done with: its scores read by the
            // softmax and its P read by P v
            const int gj = g0 + j;
            const int s = gj % RING, b = gj % NS;
            ok = wait_bounded(k_full(s), (gj / RING) & 1, wc, true) &&
                 wait_bounded(s_empty(b), ((gj / NS) & 1) ^ 1u, wc, true) &&
                 (gj < NS || wait_bounded(pv_done(b), ((gj / NS) - 1) & 1, wc, true));
            if (!ok) break;
            tc_fence_after();
            const uint32_t kd = k_s + s * G::K_BYTES;
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
              const uint64_t a_desc = sw128_desc(q_s + (k / 4) * ATOM + (k % 4) * 32, 16, 1024);
              // pre-transposed k: MN-major B, two 64-key chunks per 64 head lanes;
              // else K-major B, like q
              const uint64_t b_desc = KT ? sw128_desc(kd + (k / 4) * 2 * CHUNK + (k % 4) * 2048, CHUNK, 1024)
                                         : sw128_desc(kd + (k / 4) * ATOM + (k % 4) * 32, 16, 1024);
              umma_bf16<1>(tmem + b * KB, a_desc, b_desc, idesc_s, k > 0 ? 1u : 0u);
            }
            umma_commit<1>(s_full(b));
            umma_commit<1>(k_empty(s));
            if (j == w.nkb - 1) umma_commit<1>(q_empty);  // the unit's last read of q
            issued = true;
          }
        } else {
          // the output buffer is free once the softmax stored the unit two back
          const int ob = ui & 1;
          if (ui >= 2) ok = wait_bounded(o_empty(ob), ((ui >> 1) & 1) ^ 1u, wc, true);
          for (int j = 0; ok && j < w.nkb; ++j) {
            const int gj = g0 + j;
            const int s = gj % RING, pb = gj % NS;
            ok = wait_bounded(p_full(pb), (gj / NS) & 1, wc, true) &&
                 wait_bounded(v_full(s), (gj / RING) & 1, wc, true);
            if (!ok) break;
            tc_fence_after();
            const uint32_t vd = v_s + s * G::V_BYTES;
#pragma unroll
            for (int k = 0; k < KB / 16; ++k) {
              // P from tensor memory: 16 keys are 8 packed columns of the score buffer
              const uint64_t b_desc =
                  sw128_desc(vd + (k / 4) * (HD / 64) * CHUNK + (k % 4) * 2048, CHUNK, 1024);
              umma_bf16_ts(tmem + G::O_COL + ob * HD, tmem + pb * KB + 8 * k, b_desc, idesc_o,
                           (j | k) != 0 ? 1u : 0u);
            }
            umma_commit<1>(pv_done(pb));
            umma_commit<1>(v_empty(s));
            issued = true;
          }
        }
        g = g0 + w.nkb;
      }
      if (issued) {
        // every MMA of this thread retired before TMEM is freed
        const uint32_t dr = scores ? drain : drain_pv;
        umma_commit<1>(dr);
        wait_bounded(dr, 0, wc, false);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax and output
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c = p.scale_log2e;
    bool alive = true;
    int g = 0, ui = 0;  // chunks and units this CTA has passed
    for (int u = static_cast<int>(blockIdx.x); alive && u < n_units;
         u += static_cast<int>(gridDim.x), ++ui) {
    const Unit w = unit_of(p, u, nkb_all);
    const int ob = ui & 1;
    const int g0 = g;
    float m_ref = -INFINITY, l_run = 0.0f;
    for (int j = 0; j < w.nkb; ++j) {
      const int gj = g0 + j;
      const int b = gj % NS;
      if (!__all_sync(0xFFFFFFFFu, wait_bounded(s_full(b), (gj / NS) & 1, wc, true) ? 1 : 0)) {
        alive = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[KB];
#pragma unroll
      for (int q = 0; q < KB / 32; ++q)
        tmem_ld32(t_lane + b * KB + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * q));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty(b));  // the score buffer may be overwritten
      // keys past Tk masked out (only the last chunk can hold any); the maxima
      // are taken on the raw scores (the scale c is positive), eight
      // independent partial maxima and sums keep the dependency chains short
      const int valid = static_cast<int>(p.Tk - static_cast<int64_t>(w.j0 + j) * KB);
      if (valid < KB) {
#pragma unroll
        for (int i = 0; i < KB; ++i)
          if (i >= valid) sv[i] = __float_as_uint(-INFINITY);
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
      for (int i = 0; i < KB; i += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mx[k] = fmax3(mx[k], __uint_as_float(sv[i + k]), __uint_as_float(sv[i + 8 + k]));
      const float m_blk = c * fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                    fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // the reference maximum (log2 units) moves only when this chunk's maximum
      // exceeds it by more than 8 (P <= 2^8); the first chunk sets it
      const bool raise = j == 0 || m_blk > m_ref + 8.0f;
      const float m_new = raise ? fmaxf(m_ref, m_blk) : m_ref;
      const float alpha = raise ? ex2_approx(m_ref - m_new) : 1.0f;  // 0 on the first chunk
      // P = 2^(s c - m) on packed pairs (one fma.f32x2 per two scores), rounded
      // to bf16 for the tensor core; the row sum adds the fp32 values
      uint32_t pw[KB / 2];
      uint64_t ps2[4];  // partial sums on packed pairs
#pragma unroll
      for (int k = 0; k < 4; ++k) ps2[k] = 0ull;
      const uint64_t c2 = f2_splat(c), nm2 = f2_splat(-m_new);
#pragma unroll
      for (int i = 0; i < KB / 2; ++i) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), c2,
                         nm2),
                  x0, x1);
        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
        pw[i] = pack_bf16x2(e0, e1);
        ps2[i & 3] = f2_add(ps2[i & 3], f2_pack(e0, e1));
      }
      float ps[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) f2_unpack(ps2[k], ps[2 * k], ps[2 * k + 1]);
      const float sum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      l_run = l_run * alpha + sum;
      m_ref = m_new;
      // P over the chunk's scores in TMEM (they are in registers by now): column
      // c of a row holds keys 2c and 2c+1, the A operand of P v. The next
      // scores into this buffer are issued only after this chunk's P v.
      tmem_st32(t_lane + b * KB, *reinterpret_cast<const uint32_t(*)[32]>(pw));
      tmem_st32(t_lane + b * KB + 32, *reinterpret_cast<const uint32_t(*)[32]>(pw + 32));
      tmem_wait_st();
      if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
        // a raised maximum: the output accumulated so far is scaled once the
        // previous chunk's P v has landed in it
        if (!__all_sync(0xFFFFFFFFu,
                        wait_bounded(pv_done((gj - 1) % NS), ((gj - 1) / NS) & 1, wc, true) ? 1 : 0)) {
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < HD / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(t_lane + G::O_COL + ob * HD + 32 * q, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(t_lane + G::O_COL + ob * HD + 32 * q, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(b));
    }
    g = g0 + w.nkb;
    if (!alive) break;
    const int gl = g - 1;  // the unit's last chunk
    if (!__all_sync(0xFFFFFFFFu,
                    wait_bounded(pv_done(gl % NS), (gl / NS) & 1, wc, true) ? 1 : 0)) {
      alive = false;
      break;
    }
    {
      tc_fence_after();
      if (w.slot >= 0) {
        // a split: unnormalised O, m and l for the merge (every row, also past Tq)
        float* pp = p.part + static_cast<int64_t>(w.slot) * (QB * (HD + 2));
#pragma unroll
        for (int q = 0; q < HD / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(t_lane + G::O_COL + ob * HD + 32 * q, o);
          tmem_wait_ld();
          float4* d4 = reinterpret_cast<float4*>(pp + row * HD + 32 * q);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            d4[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
        }
        pp[QB * HD + row] = m_ref;
        pp[QB * HD + QB + row] = l_run;
      }
      const float inv = 1.0f / l_run;
      const int64_t qi = w.slot >= 0 ? p.Tq : w.q0 + row;  // a split stores no output itself
      uint16_t* dst = static_cast<uint16_t*>(p.out) + (static_cast<int64_t>(w.z) * p.Tq + qi) * HD;
#pragma unroll
      for (int q = 0; q < HD / 32; ++q) {
        uint32_t o[32];
        tmem_ld32(t_lane + G::O_COL + ob * HD + 32 * q, o);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
        if (qi < p.Tq) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * q);
#pragma unroll
          for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
      // the output buffer may take the unit after next
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty(ob));
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                 : "memory");
  }
}

// Merge of the split tail: per query row, the splits' partial results under
// one maximum, m = max m_s, l = sum 2^(m_s - m) l_s, O = sum 2^(m_s - m) O_s / l,
// rounded to bf16. One CTA per (tail block, 8 output columns), one thread per
// row; every split's loads are issued together (at most kMaxSplits of them).
constexpr int kMaxSplits = 16;

template <int HD>
__global__ void __launch_bounds__(QB) attention_merge_kernel(const AttnParams p) {
  grid_dependency_wait();  // the partial results of the attention launch before it
  grid_launch_dependents();
  const int r = static_cast<int>(blockIdx.x);
  const int c0 = static_cast<int>(blockIdx.y) * 8;
  const int row = static_cast<int>(threadIdx.x);
  const int qb = p.full + r;
  const int z = qb / p.num_q_blocks;
  const int64_t qi = static_cast<int64_t>(qb - z * p.num_q_blocks) * QB + row;
  if (qi >= p.Tq) return;
  constexpr int U = QB * (HD + 2);
  const float* base = p.part + static_cast<int64_t>(r) * p.splits * U;
  float ms[kMaxSplits], ls[kMaxSplits];
#pragma unroll
  for (int sp = 0; sp < kMaxSplits; ++sp) {
    const bool in = sp < p.splits;
    ms[sp] = in ? base[sp * U + QB * HD + row] : -INFINITY;
    ls[sp] = in ? base[sp * U + QB * HD + QB + row] : 0.0f;
  }
  float m = -INFINITY;
#pragma unroll
  for (int sp = 0; sp < kMaxSplits; ++sp) m = fmaxf(m, ms[sp]);
  float l = 0.0f;
#pragma unroll
  for (int sp = 0; sp < kMaxSplits; ++sp) {
    ms[sp] = sp < p.splits ? exp2f(ms[sp] - m) : 0.0f;  // the split's weight
    l += ms[sp] * ls[sp];
  }
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int sp = 0; sp < kMaxSplits; ++sp) {
    if (sp < p.splits) {
      const float4* o4 = reinterpret_cast<const float4*>(base + sp * U + row * HD + c0);
      const float4 a = o4[0], b = o4[1];
      const float w = ms[sp];
      acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
      acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
    }
  }
  const float inv = 1.0f / l;
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                        (static_cast<int64_t>(z) * p.Tq + qi) * HD + c0);
  *dst = make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                    pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
}

template <int HD>
cudaError_t launch_merge(const AttnParams& p, int tail, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tail), HD / 8, 1);
  cfg.blockDim = dim3(QB, 1, 1);
  cfg.stream = stream;
  // launched while the attention runs (it releases its dependents at its
  // start); the kernel waits for the attention's results itself
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, attention_merge_kernel<HD>, p);
  return err != cudaSuccess ? err : cudaGetLastError();
}

template <int HD, bool KT>
cudaError_t launch_attn(const AttnParams& p, cudaStream_t stream) {
  auto kernel = attention_kernel<HD, KT>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !attr_done[dev]) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               ACfg<HD>::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    if (dev < 64) attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  const int64_t q_blocks = static_cast<int64_t>(p.BH) * p.num_q_blocks;
  const int64_t tail = q_blocks - p.full;
  // persistent: at most one CTA per SM, walking the units
  int sms = 0;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const int64_t units = p.full + tail * p.splits;
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(units, std::max(sms, 1))), 1, 1);
  cfg.blockDim = dim3(ANT, 1, 1);
  cfg.dynamicSmemBytes = ACfg<HD>::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kernel, p);
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace

AttnSplit attention_split(int64_t q_blocks, int64_t Tk, int hd, int sms) {
  const int64_t nkb = (Tk + KB - 1) / KB;
  const int64_t tail = sms > 0 ? q_blocks % sms : 0;
  AttnSplit a{static_cast<int>(q_blocks), 0, 1, 0};
  if (tail == 0 || nkb < 2) return a;
  // the tail's blocks spread over the SMs the last wave leaves idle, at least
  // one key chunk per split
  const int64_t splits = std::min<int64_t>(std::min<int64_t>(nkb, sms / tail), kMaxSplits);
  if (splits < 2) return a;
  a.full = static_cast<int>(q_blocks - tail);
  a.tail = static_cast<int>(tail);
  a.splits = static_cast<int>(splits);
  a.part_bytes = tail * splits * QB * (hd + 2) * static_cast<int64_t>(sizeof(float));
  return a;
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream, int* launches) {
  *launches = 0;
  if (p.BH == 0 || p.num_q_blocks == 0) return cudaSuccess;
  cudaError_t err = cudaErrorInvalidValue;
  if (p.hd == 64) err = p.k_transposed ? launch_attn<64, true>(p, stream) : launch_attn<64, false>(p, stream);
  if (p.hd == 128)
    err = p.k_transposed ? launch_attn<128, true>(p, stream) : launch_attn<128, false>(p, stream);
  if (err != cudaSuccess) return err;
  *launches = 1;
  const int tail = p.BH * p.num_q_blocks - p.full;
  if (tail == 0 || p.splits < 2) return cudaSuccess;
  err = p.hd == 64 ? launch_merge<64>(p, tail, stream) : launch_merge<128>(p, tail, stream);
  if (err == cudaSuccess) *launches = 2;
  return err;
}

}  // namespace fp
