// Rotary table kernel: cs[i, t] = (cos, sin)(pos[t] * base^(-2 i / n_elem)).
//
// The rotate-half embedding of nvFuser issue #1597 "Improve performance on
// RoPE" (rope_one_entry listing) takes cos/sin tables [T, rope_n_elem] as
// inputs. Both halves of a head use the same angle theta_i, so one (cos, sin)
// pair per (frequency, position) is stored: n_elem/2 * T float2, frequency-major
// so that the 32 lanes of a warp (32 consecutive tokens) read one contiguous
// run per frequency.
//
// Accuracy: the angle is formed and reduced to [-pi, pi] in fp64 (Cody-Waite
// reduction with 2*pi split into a head and a tail), then cos/sin are taken in
// fp32 on the small reduced angle, so large positions lose no bits to the
// fp32 product pos * inv_freq.
#include "fp_internal.h"

namespace fp {

// One block row per frequency (blockIdx.y = f): the inverse frequency
// base^(-2f/n_elem) is formed once per block in fp64 (FP64 throughput is low
// on this part), each thread then forms and reduces its token's angle.
__global__ void rope_table_kernel(float2* __restrict__ cs, const int32_t* __restrict__ pos,
                                  int64_t T, int n_elem, double log2_base) {
  __shared__ double inv_freq_s;
  const int f = static_cast<int>(blockIdx.y);
  if (threadIdx.x == 0) inv_freq_s = exp2(-(2.0 * f / n_elem) * log2_base);
  __syncthreads();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const double p = pos ? static_cast<double>(pos[t]) : static_cast<double>(t);
  const double a = p * inv_freq_s;
  const double two_pi_hi = 6.283185307179586232;      // nearest double to 2*pi
  const double two_pi_lo = 2.4492935982947064e-16;    // 2*pi - two_pi_hi
  const double k = rint(a * 0.15915494309189533577);  // a / (2*pi), nearest integer
  double r = fma(-k, two_pi_hi, a);
  r = fma(-k, two_pi_lo, r);
  float s, c;
  sincosf(static_cast<float>(r), &s, &c);
  cs[static_cast<int64_t>(f) * T + t] = make_float2(c, s);
}

// Caller-given tables (the rope_one_entry listing's cos/sin inputs, [T, n_rot],
// any strides, bf16 or f32): repacked per rotated pair as (cos_i, sin_i,
// cos_{i+half}, sin_{i+half}) in fp32, so the epilogue reads one float4 per pair;
// frequency-major, [half][T], like the computed table.
__device__ __forceinline__ float load_any(const void* p, bool bf16, int64_t i) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16);
  return static_cast<const float*>(p)[i];
}

__global__ void rope_import_kernel(float4* __restrict__ dst, const void* cosv, const void* sinv,
                                   bool bf16, int64_t T, int half, int64_t st_t, int64_t st_i) {
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= T * half) return;
  const int64_t f = i / T;
  const int64_t t = i - f * T;
  const int64_t lo = t * st_t + f * st_i, hi = t * st_t + (f + half) * st_i;
  dst[i] = make_float4(load_any(cosv, bf16, lo), load_any(sinv, bf16, lo), load_any(cosv, bf16, hi),
                       load_any(sinv, bf16, hi));
}

cudaError_t launch_rope_import(float4* dst, const void* cosv, const void* sinv, bool bf16,
                               int64_t T, int half, int64_t stride_t, int64_t stride_i,
                               cudaStream_t stream) {
  int64_t n = T * half;
  if (n == 0) return cudaSuccess;
  int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  rope_import_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      dst, cosv, sinv, bf16, T, half, stride_t, stride_i);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* cs, const int32_t* pos, int64_t T, int half, int n_elem,
                              double rope_base, cudaStream_t stream) {
  if (T == 0 || half == 0) return cudaSuccess;
  const int threads = 256;
  const dim3 grid(static_cast<unsigned>((T + threads - 1) / threads), static_cast<unsigned>(half));
  rope_table_kernel<<<grid, threads, 0, stream>>>(cs, pos, T, n_elem, log2(rope_base));
  return cudaGetLastError();
}

}  // namespace fp
