// m2rnn_norm.cu -- the readout epilogue after the recurrence: multiply the
// readout by the output gate g_t and apply RMSNorm over a token's d = N*V
// features (frame "Most of the block can be computed before recurrence" of
// "M2RNN: Non-Linear RNNs with Matrix-Valued States"), and its gradient
// (backup frame "RMSNormTP synchronizes per-token statistics"):
//
//     o = y (.) g,  s = (sum_d o^2 / d + eps)^(-1/2),  out = w (.) o s
//     p = w (.) dout,  r = sum_d p o,  do = s p - r s^3 o / d,
//     dy = do (.) g,  dg = do (.) y,  dw = sum over tokens of dout (.) o s.
//
// The forward kernel's epilogue warp already added sum_d o^2 of every token
// into rstd (fused, per CTA, as it stored y); the forward kernel here only
// scales.  Both kernels are bound by HBM traffic: one warp per token row,
// 16-byte vector loads and stores, grid-stride over rows.  For d <= 512 the
// backward keeps a row in registers between its two passes and its share of
// dw in registers across rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "m2rnn_internal.h"
#include "ptx.cuh"
#include "m2rnn_check.cuh"

namespace m2rnn {
namespace {

constexpr int kWarpsPerCta = 8;

template <bool F32>
struct NormT {
  using T = float;
};
template <>
struct NormT<false> {
  using T = __nv_bfloat16;
};

// 8 consecutive values (16-byte aligned) as fp32.
template <bool F32>
__device__ __forceinline__ void load8(const void* src, float (&o)[8]) {
  if constexpr (F32) {
    const float4 a = __ldg(static_cast<const float4*>(src));
    const float4 c = __ldg(static_cast<const float4*>(src) + 1);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = c.x; o[5] = c.y; o[6] = c.z; o[7] = c.w;
  } else {
    const uint4 u = __ldg(static_cast<const uint4*>(src));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = ptx::bf16x2_lo(w[i]);
      o[2 * i + 1] = ptx::bf16x2_hi(w[i]);
    }
  }
}

template <bool F32>
__device__ __forceinline__ void store8(void* dst, const float (&o)[8]) {
  if constexpr (F32) {
    static_cast<float4*>(dst)[0] = make_float4(o[0], o[1], o[2], o[3]);
    static_cast<float4*>(dst)[1] = make_float4(o[4], o[5], o[6], o[7]);
  } else {
    uint4 u;
    u.x = ptx::pack_bf16x2(o[0], o[1]);
    u.y = ptx::pack_bf16x2(o[2], o[3]);
    u.z = ptx::pack_bf16x2(o[4], o[5]);
    u.w = ptx::pack_bf16x2(o[6], o[7]);
    *static_cast<uint4*>(dst) = u;
  }
}

template <bool F32>
__global__ void __launch_bounds__(32 * kWarpsPerCta) norm_fwd_kernel(const NormParams p) {
  using TIn = typename NormT<F32>::T;
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * kWarpsPerCta;
  const int d = p.d, d8 = d / 8;
  const TIn* y = static_cast<const TIn*>(p.y);
  const TIn* g = static_cast<const TIn*>(p.g);
  const TIn* w = static_cast<const TIn*>(p.w);
  TIn* out = static_cast<TIn*>(p.out);
  for (long long row = static_cast<long long>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
       row < p.rows; row += nwarps) {
    float s = 0.f;
    if (lane == 0) s = rsqrtf(p.rstd[row] / static_cast<float>(d) + p.eps);
    s = __shfl_sync(0xffffffffu, s, 0);
    const size_t base = static_cast<size_t>(row) * d;
    for (int e = lane; e < d8; e += 32) {
      if (!in_range(p.status, base + 8 * e, 8, static_cast<size_t>(p.rows) * d, CHK_NORM_IN) ||
          !in_range(p.status, 8 * e, 8, d, CHK_NORM_IN))
        continue;
      float yy[8], gg[8], ww[8], o[8];
      load8<F32>(y + base + 8 * e, yy);
      load8<F32>(g + base + 8 * e, gg);
      load8<F32>(w + 8 * e, ww);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = ww[i] * (yy[i] * gg[i]) * s;
      store8<F32>(out + base + 8 * e, o);
    }
    if (lane == 0) p.rstd[row] = s;  // the sum of squares was read above
  }
}

template <bool F32>
__global__ void __launch_bounds__(32 * kWarpsPerCta) norm_bwd_kernel(const NormParams p) {
  using TIn = typename NormT<F32>::T;
  extern __shared__ float dw_s[];  // [d]: this CTA's share of dw
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * kWarpsPerCta;
  const int d = p.d, d8 = d / 8;
  const float inv_d = 1.f / static_cast<float>(d);
  const TIn* y = static_cast<const TIn*>(p.y);
  const TIn* g = static_cast<const TIn*>(p.g);
  const TIn* w = static_cast<const TIn*>(p.w);
  const TIn* dout = static_cast<const TIn*>(p.dout);
  TIn* dy = static_cast<TIn*>(p.dy);
  for (int e = threadIdx.x; e < d; e += blockDim.x) dw_s[e] = 0.f;
  __syncthreads();
  for (long long row = static_cast<long long>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
       row < p.rows; row += nwarps) {
    const size_t base = static_cast<size_t>(row) * d;
    const float s = p.rstd[row];
    float r = 0.f;  // sum_d (w dout) (y g)
    for (int e = lane; e < d8; e += 32) {
      if (!in_range(p.status, base + 8 * e, 8, static_cast<size_t>(p.rows) * d, CHK_NORM_IN) ||
          !in_range(p.status, 8 * e, 8, d, CHK_NORM_IN))
        continue;
      float yy[8], gg[8], ww[8], uu[8];
      load8<F32>(y + base + 8 * e, yy);
      load8<F32>(g + base + 8 * e, gg);
      load8<F32>(w + 8 * e, ww);
      load8<F32>(dout + base + 8 * e, uu);
#pragma unroll
      for (int i = 0; i < 8; ++i) r = fmaf(ww[i] * uu[i], yy[i] * gg[i], r);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
    const float c = r * s * s * s * inv_d;
    for (int e = lane; e < d8; e += 32) {  // the row again (L1/L2 resident)
      if (!in_range(p.status, base + 8 * e, 8, static_cast<size_t>(p.rows) * d, CHK_NORM_OUT) ||
          !in_range(p.status, 8 * e, 8, d, CHK_NORM_OUT))
        continue;
      float yy[8], gg[8], ww[8], uu[8], dyo[8], dgo[8];
      load8<F32>(y + base + 8 * e, yy);
      load8<F32>(g + base + 8 * e, gg);
      load8<F32>(w + 8 * e, ww);
      load8<F32>(dout + base + 8 * e, uu);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float o = yy[i] * gg[i];
        const float dov = fmaf(s, ww[i] * uu[i], -c * o);
        dyo[i] = dov * gg[i];
        dgo[i] = dov * yy[i];
        atomicAdd(dw_s + 8 * e + i, uu[i] * o * s);
      }
      store8<F32>(dy + base + 8 * e, dyo);
      store8<true>(p.dg + base + 8 * e, dgo);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < d; e += blockDim.x) atomicAdd(p.dw + e, dw_s[e]);
}

// The same for d <= 512 (at most two 8-column groups per lane): a lane's
// columns are the same in every row, so it keeps the row's values in
// registers between the two passes and its share of dw in registers across
// rows, summing it over the CTA's warps in shared memory once at the end.
// dy and dg are computed by the same operations as above.
template <bool F32>
__global__ void __launch_bounds__(32 * kWarpsPerCta) norm_bwd_kernel_reg(const NormParams p) {
  using TIn = typename NormT<F32>::T;
  constexpr int kG = 2;  // 8-column groups per lane
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * kWarpsPerCta;
  const int d = p.d, d8 = d / 8;
  const float inv_d = 1.f / static_cast<float>(d);
  const TIn* y = static_cast<const TIn*>(p.y);
  const TIn* g = static_cast<const TIn*>(p.g);
  const TIn* w = static_cast<const TIn*>(p.w);
  const TIn* dout = static_cast<const TIn*>(p.dout);
  TIn* dy = static_cast<TIn*>(p.dy);
  float ww[kG][8], dwa[kG][8];
  bool col_ok[kG];
#pragma unroll
  for (int j = 0; j < kG; ++j) {
    const int e = lane + 32 * j;
    col_ok[j] = e < d8 && in_range(p.status, 8 * e, 8, d, CHK_NORM_IN);
#pragma unroll
    for (int i = 0; i < 8; ++i) ww[j][i] = dwa[j][i] = 0.f;
    if (col_ok[j]) load8<F32>(w + 8 * e, ww[j]);
  }
  for (long long row = static_cast<long long>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
       row < p.rows; row += nwarps) {
    const size_t base = static_cast<size_t>(row) * d;
    const float s = p.rstd[row];
    float yy[kG][8], gg[kG][8], uu[kG][8];
    bool ok[kG];
    float r = 0.f;  // sum_d (w dout) (y g)
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      const int e = lane + 32 * j;
      ok[j] = col_ok[j] &&
              in_range(p.status, base + 8 * e, 8, static_cast<size_t>(p.rows) * d, CHK_NORM_IN);
      if (ok[j]) {
        load8<F32>(y + base + 8 * e, yy[j]);
        load8<F32>(g + base + 8 * e, gg[j]);
        load8<F32>(dout + base + 8 * e, uu[j]);
#pragma unroll
        for (int i = 0; i < 8; ++i) r = fmaf(ww[j][i] * uu[j][i], yy[j][i] * gg[j][i], r);
      }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
    const float c = r * s * s * s * inv_d;
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      const int e = lane + 32 * j;
      if (!ok[j] || !in_range(p.status, base + 8 * e, 8, static_cast<size_t>(p.rows) * d,
                              CHK_NORM_OUT))
        continue;
      float dyo[8], dgo[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float o = yy[j][i] * gg[j][i];
        const float dov = fmaf(s, ww[j][i] * uu[j][i], -c * o);
        dyo[i] = dov * gg[j][i];
        dgo[i] = dov * yy[j][i];
        dwa[j][i] += uu[j][i] * o * s;
      }
      store8<F32>(dy + base + 8 * e, dyo);
      store8<true>(p.dg + base + 8 * e, dgo);
    }
  }
  // dw: the CTA's warps first (shared memory), then one global add per column
  __shared__ float dw_s[512];
  for (int e = threadIdx.x; e < d; e += blockDim.x) dw_s[e] = 0.f;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kG; ++j) {
    const int e = lane + 32 * j;
    if (col_ok[j])
#pragma unroll
      for (int i = 0; i < 8; ++i) atomicAdd(dw_s + 8 * e + i, dwa[j][i]);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < d; e += blockDim.x) atomicAdd(p.dw + e, dw_s[e]);
}

unsigned norm_grid(long long rows, int sms, int ctas_per_sm) {
  const long long need = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
  const long long cap = static_cast<long long>(sms) * ctas_per_sm;
  return static_cast<unsigned>(need < cap ? need : cap);
}

}  // namespace

size_t norm_bwd_smem_bytes(int d) { return static_cast<size_t>(d) * sizeof(float); }

cudaError_t launch_norm_fwd(const NormParams& p, bool f32_inputs, int sms, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  if (p.d % 8 != 0) return cudaErrorInvalidValue;
  const unsigned grid = norm_grid(p.rows, sms, 8);
  if (f32_inputs)
    norm_fwd_kernel<true><<<grid, 32 * kWarpsPerCta, 0, stream>>>(p);
  else
    norm_fwd_kernel<false><<<grid, 32 * kWarpsPerCta, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_norm_bwd(const NormParams& p, bool f32_inputs, int sms, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  if (p.d % 8 != 0) return cudaErrorInvalidValue;
  if (p.d <= 512) {  // two 8-column groups per lane at most: registers only
    const unsigned grid = norm_grid(p.rows, sms, 2);  // (126 registers: two CTAs per SM)
    if (f32_inputs)
      norm_bwd_kernel_reg<true><<<grid, 32 * kWarpsPerCta, 0, stream>>>(p);
    else
      norm_bwd_kernel_reg<false><<<grid, 32 * kWarpsPerCta, 0, stream>>>(p);
    return cudaGetLastError();
  }
  const size_t smem = norm_bwd_smem_bytes(p.d);
  auto kern = f32_inputs ? norm_bwd_kernel<true> : norm_bwd_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const unsigned grid = norm_grid(p.rows, sms, 4);
  kern<<<grid, 32 * kWarpsPerCta, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace m2rnn
