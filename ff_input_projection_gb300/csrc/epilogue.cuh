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

// Activations for bf16 outputs, branch-free and short:
//  - exact-erf GELU with erf from Abramowitz & Stegun, "Handbook of
//    Mathematical Functions" (1964), eq. 7.1.26: for z >= 0,
//    erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2),
//    t = 1 / (1 + p z), absolute error <= 1.5e-7;
//    GELU(y) = y/2 (1 + sign(y) erf(|y|/sqrt 2)) = (y + |y| erf(|y|/sqrt 2)) / 2;
//  - tanh-GELU with tanh(u) = 1 - 2 / (1 + exp(2u));
//  - SiLU y / (1 + exp(-y)).
// Absolute errors stay near 1e-7 of the input scale, far below bf16 rounding.
template <int ACT>
__device__ __forceinline__ float activate_bf16out(float y) {
  constexpr float kLog2e = 1.4426950408889634f;
  if (ACT == ACT_GELU_ERF) {
    const float a = fabsf(y);
    const float z = a * 0.70710678118654752f;
    const float t = rcp_approx(fmaf(0.3275911f, z, 1.0f));
    float poly = fmaf(1.061405429f, t, -1.453152027f);
    poly = fmaf(poly, t, 1.421413741f);
    poly = fmaf(poly, t, -0.284496736f);
    poly = fmaf(poly, t, 0.254829592f);
    poly *= t;
    const float ez = ex2_approx(-(z * z) * kLog2e);
    const float erf_z = fmaf(-poly, ez, 1.0f);
    return 0.5f * fmaf(a, erf_z, y);
  } else if (ACT == ACT_GELU_TANH) {
    const float u = 0.79788456080286536f * fmaf(0.044715f * y, y * y, y);
    const float th = fmaf(-2.0f, rcp_approx(1.0f + ex2_approx(2.0f * kLog2e * u)), 1.0f);
    return 0.5f * y * (1.0f + th);
  } else if (ACT == ACT_SILU) {
    return y * rcp_approx(1.0f + ex2_approx(-kLog2e * y));
  } else if (ACT == ACT_RELU2) {
    const float r = fmaxf(y, 0.0f);
    return r * r;
  }
  return y;
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

}  // namespace fp
