// m2rnn_decode.cu -- single-step decode kernel of the M2RNN recurrence: one
// step of Eqs. (10)-(12) of "M2RNN: Non-Linear RNNs with Matrix-Valued States"
// for many sequences, with the state carried in HBM between calls (the
// inference path: one new token per sequence per call).
//
//     H' = f H + (1 - f) tanh(H W + k v^T),    y = H'^T q + w_r (.) v
//
// One CTA per (sequence b, head n), one warp per 32 rows (two 16-row MMA
// tiles, 16 rows when K = 16) of the K x V state.
// A step reads and writes the whole fp32 state (2 K V 4 bytes per head)
// against a few hundred bytes of inputs, so the kernel is bound by HBM
// bandwidth: every state element is loaded once (float2 per lane, whole
// 32-byte sectors), updated in registers and stored once.  The update uses
// the forward kernel's operations in the same order (rank-1 k v^T in fp32
// pairs seeding the accumulator, bf16(H) W on the tensor cores with fp32
// accumulation, tanh, the two-FMA blend), so T decode calls reproduce the
// forward kernel's H_T bitwise.  The readout H'^T q is summed in fp32: lane
// products, shuffles over the 8 row groups of a warp, then a shared-memory
// sum over the warps.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "m2rnn.h"
#include "m2rnn_internal.h"
#include "m2rnn_gate.cuh"
#include "m2rnn_check.cuh"
#include "ptx.cuh"

namespace m2rnn {
namespace {

template <bool F32>
struct DecIn;
template <>
struct DecIn<true> {
  using T = float;
};
template <>
struct DecIn<false> {
  using T = __nv_bfloat16;
};
__device__ __forceinline__ float dtof(float x) { return x; }
__device__ __forceinline__ float dtof(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void dstore(float* p, float x) { *p = x; }
__device__ __forceinline__ void dstore(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <int V, bool F32, int MT, bool GATED>
__global__ void __launch_bounds__(256) decode_kernel(const DecodeParams p) {
  using TIn = typename DecIn<F32>::T;
  constexpr int NT = V / 8, KS = V / 16;
  __shared__ float ysum[8][V];  // per-warp readout partials (at most 8 warps)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int K = p.K, N = p.N, nw = K / (16 * MT);
  const size_t head = blockIdx.x;  // b * N + n
  const int b = static_cast<int>(head / N), n = static_cast<int>(head % N);
  const int row0 = 16 * MT * warp;  // MT 16-row tiles per warp

  // [B,Nq,K]: the row of head n's query/key group (no division when shared)
  const size_t qrow = p.Nq == 1 ? static_cast<size_t>(b)
                                : static_cast<size_t>(b) * p.Nq + n / (N / p.Nq);
  const TIn* q = static_cast<const TIn*>(p.q) + qrow * K;
  const TIn* k = static_cast<const TIn*>(p.k) + qrow * K;
  const TIn* v = static_cast<const TIn*>(p.v) + head * V;
  const TIn* Wn = static_cast<const TIn*>(p.W) + static_cast<size_t>(n) * V * V;
  const TIn* wr = static_cast<const TIn*>(p.w_r) + static_cast<size_t>(n) * V;
  const float* Hin = p.H_in + head * K * V;
  float* Hout = p.H_out + head * K * V;
  // index checks of the checked build (uniform over the CTA, before any barrier)
  const size_t BN = static_cast<size_t>(p.B) * N, s_ext = BN * K * V;
  if (!in_range(p.status, qrow * K, K, static_cast<size_t>(p.B) * p.Nq * K, CHK_DEC_IN) ||
      !in_range(p.status, head * V, V, BN * V, CHK_DEC_IN) ||
      !in_range(p.status, head, 1, BN, CHK_DEC_IN) ||
      !in_range(p.status, static_cast<size_t>(n) * V * V, V * V, static_cast<size_t>(N) * V * V, CHK_DEC_IN) ||
      !in_range(p.status, head * V, V, BN * V, CHK_DEC_Y))
    return;

  // the state first: the loads that decide the kernel's time, all in flight
  // before any use
  float H[MT][NT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int o = (row0 + 16 * m + g + 8 * h) * V + 8 * nt + 2 * c;
        const float2 x = in_range(p.status, head * K * V + o, 2, s_ext, CHK_DEC_STATE)
                             ? __ldcs(reinterpret_cast<const float2*>(Hin + o))
                             : make_float2(0.f, 0.f);
        H[m][nt][2 * h] = x.x;
        H[m][nt][2 * h + 1] = x.y;
      }
  // W as the B operand of H W (k-index l, n-index j), bf16 hi (+ lo for fp32 inputs)
  uint32_t Bw[KS][NT][2], Bwl[KS][NT][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kk = 16 * ks + 8 * h + 2 * c, nn = 8 * nt + g;
        const float w0 = dtof(Wn[kk * V + nn]), w1 = dtof(Wn[(kk + 1) * V + nn]);
        Bw[ks][nt][h] = ptx::pack_bf16x2(w0, w1);
        Bwl[ks][nt][h] = F32 ? ptx::pack_bf16x2(w0 - ptx::bf16x2_lo(Bw[ks][nt][h]),
                                                w1 - ptx::bf16x2_hi(Bw[ks][nt][h]))
                             : 0u;
      }
  float2 vv[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
    vv[nt] = make_float2(dtof(v[8 * nt + 2 * c]), dtof(v[8 * nt + 2 * c + 1]));
  // f, or with the fused input gate exp(-alpha softplus(a + beta)) (the
  // forward kernel's function, so decode steps stay bitwise equal to it)
  const float fg = GATED ? gate_f(dtof(static_cast<const TIn*>(p.a)[head]),
                                    dtof(static_cast<const TIn*>(p.alpha)[n]),
                                    dtof(static_cast<const TIn*>(p.beta)[n]))
                           : dtof(static_cast<const TIn*>(p.f)[head]);
  const float2 f2 = make_float2(fg, fg), m1 = make_float2(-1.f, -1.f);

  float ypart[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) ypart[nt][0] = ypart[nt][1] = 0.f;
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const int r0 = row0 + 16 * m;
    const float k0 = dtof(k[r0 + g]), k1 = dtof(k[r0 + g + 8]);
    const float q0 = dtof(q[r0 + g]), q1 = dtof(q[r0 + g + 8]);
    // bf16 A fragments of H (hi, and lo for fp32 inputs)
    uint32_t A[KS][4], Al[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      A[ks][0] = ptx::pack_bf16x2(H[m][2 * ks][0], H[m][2 * ks][1]);
      A[ks][1] = ptx::pack_bf16x2(H[m][2 * ks][2], H[m][2 * ks][3]);
      A[ks][2] = ptx::pack_bf16x2(H[m][2 * ks + 1][0], H[m][2 * ks + 1][1]);
      A[ks][3] = ptx::pack_bf16x2(H[m][2 * ks + 1][2], H[m][2 * ks + 1][3]);
      if (F32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int nt = 2 * ks + (i >> 1), r = 2 * (i & 1);
          Al[ks][i] = ptx::pack_bf16x2(H[m][nt][r] - ptx::bf16x2_lo(A[ks][i]),
                                       H[m][nt][r + 1] - ptx::bf16x2_hi(A[ks][i]));
        }
      }
    }
    // Z = tanh(H W + k v^T);  H' = Z + f (H - Z)
    const float2 kk0 = make_float2(k0, k0), kk1 = make_float2(k1, k1);
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
    for (int nt = 0; nt < NT; ++nt) {
      float hn[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float2 z;
        z.x = F32 ? tanhf(acc[nt][2 * h]) : ptx::tanh_approx(acc[nt][2 * h]);
        z.y = F32 ? tanhf(acc[nt][2 * h + 1]) : ptx::tanh_approx(acc[nt][2 * h + 1]);
        const float2 d = __ffma2_rn(m1, z, make_float2(H[m][nt][2 * h], H[m][nt][2 * h + 1]));
        const float2 r = __ffma2_rn(f2, d, z);
        hn[2 * h] = r.x;
        hn[2 * h + 1] = r.y;
        const int o = (r0 + g + 8 * h) * V + 8 * nt + 2 * c;
        if (in_range(p.status, head * K * V + o, 2, s_ext, CHK_DEC_STATE))
          __stcs(reinterpret_cast<float2*>(Hout + o), r);
      }
      // this lane's two rows of the readout for columns 8nt + 2c, 8nt + 2c + 1
      ypart[nt][0] += fmaf(hn[0], q0, hn[2] * q1);
      ypart[nt][1] += fmaf(hn[1], q0, hn[3] * q1);
    }
  }
  // sum over the 8 row groups of the warp (lanes with equal c)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float s = ypart[nt][e];
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      s += __shfl_xor_sync(0xffffffffu, s, 8);
      s += __shfl_xor_sync(0xffffffffu, s, 16);
      if (g == 0) ysum[warp][8 * nt + 2 * c + e] = s;
    }
  __syncthreads();
  if (tid < V) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += ysum[w][tid];
    s = fmaf(dtof(wr[tid]), dtof(v[tid]), s);
    dstore(static_cast<TIn*>(p.y) + head * V + tid, s);
  }
}

template <int V, bool F32, bool GATED>
cudaError_t launch_decode_g(const DecodeParams& p, cudaStream_t stream) {
  const size_t heads = static_cast<size_t>(p.B) * p.N;
  if (p.K >= 32)  // two 16-row tiles per warp: twice the state bytes in flight per warp
    decode_kernel<V, F32, 2, GATED><<<static_cast<unsigned>(heads), 32 * (p.K / 32), 0, stream>>>(p);
  else
    decode_kernel<V, F32, 1, GATED><<<static_cast<unsigned>(heads), 32 * (p.K / 16), 0, stream>>>(p);
  return cudaGetLastError();
}

template <int V, bool F32>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  return p.gated ? launch_decode_g<V, F32, true>(p, stream) : launch_decode_g<V, F32, false>(p, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int V, bool f32_inputs, cudaStream_t stream) {
  if (p.K < 16 || p.K > 128 || p.K % 16 != 0) return cudaErrorInvalidValue;
  if (V == 16) return f32_inputs ? launch_decode_t<16, true>(p, stream) : launch_decode_t<16, false>(p, stream);
  if (V == 32) return f32_inputs ? launch_decode_t<32, true>(p, stream) : launch_decode_t<32, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace m2rnn
