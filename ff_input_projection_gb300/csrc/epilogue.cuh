// Epilogue arithmetic shared by the tensor-core and FFMA kernels: column
// decoding into (ff | q | k | v, head, lane), activations and output addressing.
#pragma once

#include <cuda_bf16.h>
#include "fp_internal.h"

namespace fp {

struct ColInfo {
  int seg;   // 0 ff, 1 q, 2 k, 3 v
  int head;  // q head, or k/v head (group) index
  int j;     // lane inside the head (ff: the column)
};

// Fused column n -> block, head and lane. Blocked order [ff | q | k | v]
// (fused_ff_qkv of Walrus PR #12); with groups > 0 the q|k|v part follows the
// split_qkv listing of nvFuser issue #1597: per group, q_per_kv query heads,
// then its key head, then its value head.
__device__ __forceinline__ ColInfo decode_col(const Epilogue& e, int n) {
  ColInfo ci;
  if (n < e.F) {
    ci.seg = 0;
    ci.head = 0;
    ci.j = n;
    return ci;
  }
  int w = n - e.F;
  if (e.groups > 0) {
    int qpk = e.heads / e.groups;
    int per = (qpk + 2) * e.hd;
    int g = w / per, r = w - g * per;
    int slot = r / e.hd;
    ci.j = r - slot * e.hd;
    if (slot < qpk) {
      ci.seg = 1;
      ci.head = g * qpk + slot;
    } else {
      ci.seg = slot == qpk ? 2 : 3;
      ci.head = g;
    }
    return ci;
  }
  int seg = w / e.C, r = w - seg * e.C;
  ci.seg = 1 + seg;
  ci.head = r / e.hd;
  ci.j = r - ci.head * e.hd;
  return ci;
}

// Walks the fused columns 16 at a time (ff_hidden and head_dim are multiples
// of 16 on the tensor-core path), so a tile decodes its first column once and
// then only adds.
struct ColCursor {
  ColInfo ci;
  int grp, slot;  // grouped-query position: group and slot inside [q.. | k | v]
};

__device__ __forceinline__ void cursor_init(const Epilogue& e, int n, ColCursor& c) {
  c.ci = decode_col(e, n);
  c.grp = 0;
  c.slot = 0;
  if (e.groups > 0 && c.ci.seg > 0) {
    const int qpk = e.heads / e.groups;
    if (c.ci.seg == 1) {
      c.grp = c.ci.head / qpk;
      c.slot = c.ci.head - c.grp * qpk;
    } else {
      c.grp = c.ci.head;
      c.slot = c.ci.seg == 2 ? qpk : qpk + 1;
    }
  }
}

__device__ __forceinline__ void cursor_advance16(const Epilogue& e, ColCursor& c) {
  c.ci.j += 16;
  if (c.ci.seg == 0) {
    if (c.ci.j >= e.F) {
      c.ci.seg = 1;
      c.ci.head = 0;
      c.ci.j = 0;
      c.grp = 0;
      c.slot = 0;
    }
    return;
  }
  if (c.ci.j < e.hd) return;
  c.ci.j = 0;
  if (e.groups == 0) {
    if (++c.ci.head == e.heads) {
      c.ci.head = 0;
      ++c.ci.seg;
    }
    return;
  }
  const int qpk = e.heads / e.groups;
  if (++c.slot == qpk + 2) {
    c.slot = 0;
    ++c.grp;
  }
  c.ci.seg = c.slot < qpk ? 1 : (c.slot == qpk ? 2 : 3);
  c.ci.head = c.slot < qpk ? c.grp * qpk + c.slot : c.grp;
}

// Element offset of (token m = b*T + t, column info) in its output buffer.
__device__ __forceinline__ int64_t out_offset(const Epilogue& e, const ColInfo& ci, int64_t m,
                                              int64_t b, int64_t t) {
  if (ci.seg == 0) return m * e.F + ci.j;
  int nh = (ci.seg == 1 || e.groups == 0) ? e.heads : e.groups;
  return ((b * nh + ci.head) * e.T + t) * e.hd + ci.j;
}

__device__ __forceinline__ void* out_base(const Epilogue& e, int seg) {
  return seg == 0 ? e.out_ff : seg == 1 ? e.out_q : seg == 2 ? e.out_k : e.out_v;
}

// Activations of the ff block, in fp32 (the caller's dtype is only the storage).
__device__ __forceinline__ float activate(int act, float y) {
  switch (act) {
    case ACT_GELU_ERF:
      return 0.5f * y * (1.0f + erff(y * 0.70710678118654752f));
    case ACT_GELU_TANH: {
      float u = 0.79788456080286536f * (y + 0.044715f * y * y * y);
      return 0.5f * y * (1.0f + tanhf(u));
    }
    case ACT_SILU:
      return y / (1.0f + expf(-y));
    case ACT_RELU2: {
      const float r = fmaxf(y, 0.0f);
      return r * r;
    }
    default:
      return y;
  }
}

// Hardware approximations (PTX rcp.approx / ex2.approx): about 1 ulp and
// 2^-22 relative error respectively.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Packed fp32 pairs (sm_100 f32x2 arithmetic: two IEEE fp32 operations per
// instruction, the same results as two scalar ones).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_splat(float x) { return f2_pack(x, x); }
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi);

// Activation of two fp32 values, rounded to a bf16 pair (low = y0). Branch-free
// and short, on packed fp32 pairs:
//  - exact-erf GELU with erf from Abramowitz & Stegun, "Handbook of
//    Mathematical Functions" (1964), eq. 7.1.26: for z >= 0,
//    erf(z) = 1 - t P(t) exp(-z^2), t = 1 / (1 + p z),
//    P(t) = a1 + a2 t + a3 t^2 + a4 t^3 + a5 t^4, absolute error <= 1.5e-7.
//    With a = |y| and z = a / sqrt 2 both signs of y reduce to
//    GELU(y) = relu(y) - (a/2) t P(t) exp(-a^2/2);
//    the a in front is clamped at 1e30 so y = +-inf gives inf and 0, not NaN
//    (a NaN still propagates through t);
//  - tanh-GELU as y * sigmoid(2u), u = sqrt(2/pi) (y + 0.044715 y^3);
//  - SiLU y * sigmoid(y).
// Absolute errors stay near 1e-7 of the input scale, far below bf16 rounding.
template <int ACT>
__device__ __forceinline__ uint32_t activate2_bf16(uint32_t u0, uint32_t u1) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float y0 = __uint_as_float(u0), y1 = __uint_as_float(u1);
  if (ACT == ACT_GELU_ERF) {
    const float a0 = fabsf(y0), a1 = fabsf(y1);
    const uint64_t A = f2_pack(a0, a1);
    const uint64_t D = f2_fma(A, f2_splat(0.3275911f * 0.70710678118654752f), f2_splat(1.0f));
    float d0, d1;
    f2_unpack(D, d0, d1);
    const uint64_t T = f2_pack(rcp_approx(d0), rcp_approx(d1));
    // -(1/2) a_k: the sign and the 1/2 of the GELU form folded into P
    uint64_t P = f2_fma(f2_splat(-0.5f * 1.061405429f), T, f2_splat(-0.5f * -1.453152027f));
    P = f2_fma(P, T, f2_splat(-0.5f * 1.421413741f));
    P = f2_fma(P, T, f2_splat(-0.5f * -0.284496736f));
    P = f2_fma(P, T, f2_splat(-0.5f * 0.254829592f));
    const uint64_t AC = f2_pack(fminf(a0, 1e30f), fminf(a1, 1e30f));
    const uint64_t S = f2_mul(f2_mul(P, T), AC);  // -(a/2) t P(t)
    const uint64_t Q = f2_mul(f2_mul(A, f2_splat(-0.5f * kLog2e)), A);  // log2 exp(-a^2/2)
    float q0, q1;
    f2_unpack(Q, q0, q1);
    const uint64_t E = f2_pack(ex2_approx(q0), ex2_approx(q1));
    const uint64_t R = f2_fma(S, E, f2_pack(fmaxf(y0, 0.0f), fmaxf(y1, 0.0f)));
    float r0, r1;
    f2_unpack(R, r0, r1);
    return pack_bf16x2(r0, r1);
  } else if (ACT == ACT_GELU_TANH) {
    // sigmoid(2u) = 1 / (1 + 2^(y (k1 + k3 y^2))), k1 = -2 log2(e) sqrt(2/pi)
    constexpr float k1 = -2.0f * kLog2e * 0.79788456080286536f;
    const uint64_t Y = f2_pack(y0, y1);
    const uint64_t G = f2_mul(f2_fma(f2_mul(Y, Y), f2_splat(k1 * 0.044715f), f2_splat(k1)), Y);
    float g0, g1;
    f2_unpack(G, g0, g1);
    const uint64_t E1 = f2_add(f2_pack(ex2_approx(g0), ex2_approx(g1)), f2_splat(1.0f));
    float e0, e1;
    f2_unpack(E1, e0, e1);
    float r0, r1;
    f2_unpack(f2_mul(Y, f2_pack(rcp_approx(e0), rcp_approx(e1))), r0, r1);
    return pack_bf16x2(r0, r1);
  } else if (ACT == ACT_SILU) {
    const uint64_t Y = f2_pack(y0, y1);
    float g0, g1;
    f2_unpack(f2_mul(Y, f2_splat(-kLog2e)), g0, g1);
    const uint64_t E1 = f2_add(f2_pack(ex2_approx(g0), ex2_approx(g1)), f2_splat(1.0f));
    float e0, e1;
    f2_unpack(E1, e0, e1);
    float r0, r1;
    f2_unpack(f2_mul(Y, f2_pack(rcp_approx(e0), rcp_approx(e1))), r0, r1);
    return pack_bf16x2(r0, r1);
  } else if (ACT == ACT_RELU2) {
    const uint64_t Rl = f2_pack(fmaxf(y0, 0.0f), fmaxf(y1, 0.0f));
    float r0, r1;
    f2_unpack(f2_mul(Rl, Rl), r0, r1);
    return pack_bf16x2(r0, r1);
  }
  return pack_bf16x2(y0, y1);
}

// Derivative of the ff activation (fp32, CUDA's math library).
template <int ACT>
__device__ __forceinline__ float act_deriv(float y) {
  if (ACT == ACT_GELU_ERF) {
    return normcdff(y) + y * 0.39894228040143268f * __expf(-0.5f * y * y);
  } else if (ACT == ACT_GELU_TANH) {
    constexpr float k0 = 0.79788456080286536f, k3 = 0.044715f;
    const float th = tanhf(k0 * fmaf(k3 * y, y * y, y));
    return 0.5f * (1.0f + th) + 0.5f * y * (1.0f - th * th) * k0 * fmaf(3.0f * k3, y * y, 1.0f);
  } else if (ACT == ACT_SILU) {
    const float sg = 1.0f / (1.0f + __expf(-y));
    return sg * fmaf(y, 1.0f - sg, 1.0f);
  } else if (ACT == ACT_RELU2) {
    return y > 0.0f ? 2.0f * y : 0.0f;
  }
  return 1.0f;
}

// GELU'(y) = Phi(y) + y phi(y) for two values on packed fp32 pairs, with the
// same Abramowitz & Stegun 7.1.26 erf as the forward: for a = |y|,
// t = 1 / (1 + p a / sqrt 2), erfc(a / sqrt 2) = t P(t) exp(-a^2/2), so
// Phi(y) = h or 1 - h with h = (1/2) t P(t) e, e = exp(-y^2/2), and
// phi(y) = e / sqrt(2 pi). Absolute error about 1e-7.
__device__ __forceinline__ void gelu_erf_deriv2(float y0, float y1, float& d0, float& d1) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float a0 = fabsf(y0), a1 = fabsf(y1);
  const uint64_t A = f2_pack(a0, a1);
  float q0, q1;
  f2_unpack(f2_fma(A, f2_splat(0.3275911f * 0.70710678118654752f), f2_splat(1.0f)), q0, q1);
  const uint64_t T = f2_pack(rcp_approx(q0), rcp_approx(q1));
  uint64_t P = f2_fma(f2_splat(0.5f * 1.061405429f), T, f2_splat(0.5f * -1.453152027f));
  P = f2_fma(P, T, f2_splat(0.5f * 1.421413741f));
  P = f2_fma(P, T, f2_splat(0.5f * -0.284496736f));
  P = f2_fma(P, T, f2_splat(0.5f * 0.254829592f));
  float e0, e1;
  f2_unpack(f2_mul(f2_mul(A, f2_splat(-0.5f * kLog2e)), A), e0, e1);
  const uint64_t E = f2_pack(ex2_approx(e0), ex2_approx(e1));
  float h0, h1;
  f2_unpack(f2_mul(f2_mul(P, T), E), h0, h1);  // (1/2) erfc(|y| / sqrt 2)
  const uint64_t PHI = f2_pack(y0 >= 0.0f ? 1.0f - h0 : h0, y1 >= 0.0f ? 1.0f - h1 : h1);
  const uint64_t R =
      f2_fma(f2_mul(f2_pack(y0, y1), f2_splat(0.39894228040143268f)), E, PHI);
  f2_unpack(R, d0, d1);
}

// Column sums of a warp's [32 rows][32 columns] block (row = lane): a
// butterfly that halves the columns each lane keeps at every step; after five
// steps lane i holds the sum of column i.
__device__ __forceinline__ float column_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int off = 16 >> step;
    const int n = 32 >> step;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
    }
  }
  return v[0];
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// With bounds checking on: may `n` elements, `stride` apart, starting at
// element `off` of output `seg` (0 ff, 1 q, 2 k, 3 v) be stored? A store that
// would leave the buffer is recorded (ST_BOUNDS) and must be skipped.
__device__ __forceinline__ bool store_in_bounds(const Epilogue& e, int seg, int64_t off,
                                                int64_t n, int64_t stride = 1) {
  if (!e.bounds_check) return true;
  if (off >= 0 && off + (n - 1) * stride < e.extent[seg]) return true;
  record_status(e.status, ST_BOUNDS);
  return false;
}

}  // namespace fp
