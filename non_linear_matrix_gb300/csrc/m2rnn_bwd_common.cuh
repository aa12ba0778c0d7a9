// m2rnn_bwd_common.cuh -- device helpers shared by the backward kernels:
// input conversion, MMA fragment packing, global reductions and the
// recompute step (one forward step of Eqs. (10)-(11) of "M2RNN: Non-Linear
// RNNs with Matrix-Valued States" with the operations of the forward kernel).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace m2rnn {
namespace bwdc {

template <bool F32>
struct InT;
template <>
struct InT<true> {
  using T = float;
};
template <>
struct InT<false> {
  using T = __nv_bfloat16;
};

__device__ __forceinline__ float tof(float x) { return x; }
__device__ __forceinline__ float tof(__nv_bfloat16 x) { return __bfloat162float(x); }

// Sub-interval length (recomputed steps held in registers) of each variant.
template <int V, bool F32>
__host__ __device__ constexpr int sub_len() {
  return (V == 16 && !F32) ? 8 : (V == 32 && F32) ? 2 : 4;
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}
__device__ __forceinline__ void red_add(float* p, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory");
}
__device__ __forceinline__ void sts_u32x4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                          uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// bf16x2 pair of two input values (rounding fp32 inputs to bf16).
template <bool F32>
__device__ __forceinline__ uint32_t pair_bf16(uint32_t addr) {
  if (F32) {
    const float2 x = ptx::lds_f32x2(addr);
    return ptx::pack_bf16x2(x.x, x.y);
  }
  return ptx::lds_u32(addr);
}
// Two consecutive input values as floats.
template <bool F32>
__device__ __forceinline__ float2 pair_f32(uint32_t addr) {
  if (F32) return ptx::lds_f32x2(addr);
  const uint32_t w = ptx::lds_u32(addr);
  return make_float2(ptx::bf16x2_lo(w), ptx::bf16x2_hi(w));
}
template <bool F32>
__device__ __forceinline__ float one_f32(uint32_t addr) {
  if (F32) return ptx::lds_f32(addr);
  return __uint_as_float(ptx::lds_u16(addr) << 16);
}

template <int V>
__device__ __forceinline__ void pack_frag(const float (&H)[V / 8][4], uint32_t (&A)[V / 16][4]) {
#pragma unroll
  for (int ks = 0; ks < V / 16; ++ks) {
    A[ks][0] = ptx::pack_bf16x2(H[2 * ks][0], H[2 * ks][1]);
    A[ks][1] = ptx::pack_bf16x2(H[2 * ks][2], H[2 * ks][3]);
    A[ks][2] = ptx::pack_bf16x2(H[2 * ks + 1][0], H[2 * ks + 1][1]);
    A[ks][3] = ptx::pack_bf16x2(H[2 * ks + 1][2], H[2 * ks + 1][3]);
  }
}
template <int V>
__device__ __forceinline__ void pack_frag_lo(const float (&H)[V / 8][4], const uint32_t (&A)[V / 16][4],
                                             uint32_t (&Al)[V / 16][4]) {
#pragma unroll
  for (int ks = 0; ks < V / 16; ++ks)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int nt = 2 * ks + (i >> 1), r = 2 * (i & 1);
      Al[ks][i] = ptx::pack_bf16x2(H[nt][r] - ptx::bf16x2_lo(A[ks][i]),
                                   H[nt][r + 1] - ptx::bf16x2_hi(A[ks][i]));
    }
}

// One forward step of Eqs. (10)-(11) for this warp's 16 rows, with exactly
// the operations of the forward kernel (so trajectories agree bitwise).
// Updates H, A (and Al on the fp32-input path); returns, per element,
// So = (1 - f)(1 - Z^2) and Eo = H_{t-1} - Z, the quantities the reverse step
// needs.
template <int V, bool F32>
__device__ __forceinline__ void recompute_step(float (&H)[V / 8][4], uint32_t (&A)[V / 16][4],
                                               uint32_t (&Al)[V / 16][4],
                                               const uint32_t (&Bw)[V / 16][V / 8][2],
                                               const uint32_t (&Bwl)[V / 16][V / 8][2], float k0,
                                               float k1, const float2 (&vv)[V / 8], float fg,
                                               float (&So)[V / 8][4], float (&Eo)[V / 8][4]) {
  constexpr int NT = V / 8, KS = V / 16;
  const float2 kk0 = make_float2(k0, k0), kk1 = make_float2(k1, k1);
  const float2 f2 = make_float2(fg, fg), m1 = make_float2(-1.f, -1.f);
  const float omf = 1.f - fg;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float2 lo = __fmul2_rn(kk0, vv[nt]), hi = __fmul2_rn(kk1, vv[nt]);
    acc[nt][0] = lo.x;
    acc[nt][1] = lo.y;
    acc[nt][2] = hi.x;
    acc[nt][3] = hi.y;
  }
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      ptx::mma_bf16_16816(acc[nt], A[ks], Bw[ks][nt][0], Bw[ks][nt][1]);
      if (F32) {
        ptx::mma_bf16_16816(acc[nt], A[ks], Bwl[ks][nt][0], Bwl[ks][nt][1]);
        ptx::mma_bf16_16816(acc[nt], Al[ks], Bw[ks][nt][0], Bw[ks][nt][1]);
      }
    }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float2 z;
      z.x = F32 ? tanhf(acc[nt][2 * h]) : ptx::tanh_approx(acc[nt][2 * h]);
      z.y = F32 ? tanhf(acc[nt][2 * h + 1]) : ptx::tanh_approx(acc[nt][2 * h + 1]);
      const float2 hp = make_float2(H[nt][2 * h], H[nt][2 * h + 1]);
      const float2 d = __ffma2_rn(m1, z, hp);
      const float2 hn = __ffma2_rn(f2, d, z);
      H[nt][2 * h] = hn.x;
      H[nt][2 * h + 1] = hn.y;
      Eo[nt][2 * h] = d.x;  // H_{t-1} - Z
      Eo[nt][2 * h + 1] = d.y;
      So[nt][2 * h] = omf * fmaf(-z.x, z.x, 1.f);
      So[nt][2 * h + 1] = omf * fmaf(-z.y, z.y, 1.f);
    }
  pack_frag<V>(H, A);
  if (F32) pack_frag_lo<V>(H, A, Al);
}

}  // namespace bwdc
}  // namespace m2rnn
