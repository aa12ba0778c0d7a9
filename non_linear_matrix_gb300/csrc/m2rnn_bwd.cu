// m2rnn_bwd.cu -- BPTT backward kernel of the M2RNN recurrence.
//
// Chain rule of the backup frame "the recurrent gradient needs both paths"
// in the discussion deck of "M2RNN: Non-Linear RNNs with Matrix-Valued
// States": with u_t = dL/dy_t and C_t the gradient arriving from later steps,
//     R_t = C_t + q_t u_t^T,   D_t = ((1 - f_t) R_t) (.) (1 - Z_t (.) Z_t),
//     C_{t-1} = f_t R_t + D_t W^T,   dL/df_t = <R_t, H_{t-1} - Z_t>_F,
//     dL/dW = sum_t H_{t-1}^T D_t,
// plus the terms Eqs. (10)-(12) give for the other inputs:
//     dk_t = sum_n D_t v_t,  dq_t = sum_n H_t u_t,  dv_t = D_t^T k_t + w_r (.) u_t,
//     dw_r = sum_{b,t} u_t (.) v_t,  dH_0 = C_0.
// (The paper's printed Algorithm 2 drops C_t; the deck's boxed recursion is
// followed.)
//
// The deck's backward caches every state in HBM ("recompute the trajectory,
// cache states in HBM, then run the reverse sweep"); here nothing but the
// checkpoints H_{cC} (every C steps, written by the forward pass) leaves the
// chip.  CTA = one (batch b, head n, slice of 16*WPC rows); warp w owns 16
// rows in mma.sync m16n8k16 accumulator layout.  For each checkpoint interval,
// last first:
//   1. load the interval's inputs into shared memory;
//   2. recompute the interval forward from its checkpoint, keeping a
//      sub-checkpoint every S2 steps (fp32);
//   3. for each sub-interval, last first: recompute its S2 steps keeping,
//      in registers, bf16(H) (as MMA operand fragments), s = (1-f)(1-Z^2)
//      (fp32) and e = H_{t-1} - Z (fp16, |e| <= 2; fp32 on the fp32-input
//      path), what the reverse step needs, then run the
//      reverse steps over it; per-step partials go to shared memory and are
//      flushed with vector reductions (head sums of dq, dk) or stores.
// Sub-checkpoints live in thread-private shared-memory slots laid out
// lane-contiguously (no bank conflicts).  The recomputation performs the
// same operations as the forward kernel, so it reproduces its trajectory.
// Synchronisation is __syncthreads only (no spin waits).
//
// This is the serial variant: the three passes run one after the other in
// each warp.  m2rnn_bwd_pipe.cu holds the pipelined variant used for V = 16;
// this one serves V = 32 and any shape the other does not fit.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "m2rnn.h"
#include "m2rnn_internal.h"
#include "ptx.cuh"
#include "m2rnn_bwd_common.cuh"
#include "m2rnn_gate.cuh"
#include "m2rnn_check.cuh"

namespace m2rnn {
namespace {

using namespace bwdc;

// Shared-memory layout of one CTA (byte offsets).  With interleaving the
// k/v/f inputs and the sub-checkpoints are double-buffered (buffer ci & 1
// holds interval ci); the per-step partials are double-buffered by
// sub-interval in every variant.
struct BwdLayout {
  uint32_t in_q, in_dy;              // [C][RS], [C][V]: the interval being reversed
  uint32_t in_k, in_v, in_f;         // buffer 0: [C][RS], [C][V], [C] fp32
  uint32_t kbuf, vbuf, fbuf;         // byte stride to buffer 1
  uint32_t subck, sbuf;              // [NS1][WPC][NT][32][4] fp32, stride to buffer 1
  uint32_t dwsum;                    // [WPC][V][V] fp32 (end of kernel; aliases subck)
  uint32_t r_dq, r_dk, r_dv, r_df;   // [2][S2][RS], [2][S2][RS], [2][S2][WPC][V], [2][S2][WPC]
  uint32_t total;
};

__host__ __device__ inline uint32_t al(uint32_t x) { return (x + 127u) / 128u * 128u; }

__host__ __device__ inline BwdLayout bwd_layout(int V, int C, int S2, int WPC, int es) {
  // Step buffers hold NS1 * S2 >= C steps: recompute steps past the end of
  // an interval read the padding and their results are discarded.
  const uint32_t RS = 16 * WPC, NT = V / 8, NS1 = (C + S2 - 1) / S2, CP = NS1 * S2;
  const uint32_t nb = 1;
  BwdLayout L;
  uint32_t o = 0;
  L.in_q = o;
  o = al(o + C * RS * es);
  L.in_dy = o;
  o = al(o + C * V * es);
  L.kbuf = al(CP * RS * es);
  L.in_k = o;
  o += nb * L.kbuf;
  L.vbuf = al(CP * V * es);
  L.in_v = o;
  o += nb * L.vbuf;
  L.fbuf = al(CP * 4);
  L.in_f = o;
  o += nb * L.fbuf;
  L.sbuf = NS1 * WPC * NT * 512;
  L.subck = L.dwsum = o;
  const uint32_t dws = WPC * V * V * 4;
  o = al(o + (nb * L.sbuf > dws ? nb * L.sbuf : dws));
  L.r_dq = o;
  o = al(o + 2 * S2 * RS * 4);
  L.r_dk = o;
  o = al(o + 2 * S2 * RS * 4);
  L.r_dv = o;
  o = al(o + 2 * S2 * WPC * V * 4);
  L.r_df = o;
  o = al(o + 2 * S2 * WPC * 4);
  L.total = o;
  return L;
}

template <int V, bool F32, bool GATED>
__global__ void __launch_bounds__(256) bwd_kernel(const BwdParams p) {
  using TIn = typename InT<F32>::T;
  constexpr int es = sizeof(TIn);
  constexpr int NT = V / 8, KS = V / 16;
  constexpr int S2 = sub_len<V, F32>();
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int WPC = p.WPC, RS = 16 * WPC, nthr = 32 * WPC;
  const int K = p.K, T = p.T, N = p.N, C = p.C;
  const int slice = blockIdx.x % p.nslices;
  const int bn = blockIdx.x / p.nslices;
  const int b = bn / N, n = bn % N;
  const int Nq = p.Nq, gq = n / (N / Nq);  // query/key group of head n
  const int row0c = slice * RS;            // first row of this CTA
  const int row0 = row0c + 16 * warp;      // first row of this warp
  const BwdLayout L = bwd_layout(V, C, S2, WPC, es);
  const uint32_t sb = ptx::smem_addr(smem);

  const TIn* q = static_cast<const TIn*>(p.q);
  const TIn* kin = static_cast<const TIn*>(p.k);
  const TIn* vin = static_cast<const TIn*>(p.v);
  // f, or with the fused input gate its input a (same layout and dtype)
  constexpr bool gated = GATED;
  const TIn* fin = static_cast<const TIn*>(gated ? p.a : p.f);
  // array extents in elements (index checks of the checked build)
  const size_t BT = static_cast<size_t>(p.B) * T;
  const size_t qk_ext = BT * Nq * K, v_ext = BT * N * V, f_ext = BT * N;
  const size_t s_ext = static_cast<size_t>(p.B) * N * K * V;  // dH_T, dH0
  const bool n_ok = in_range(p.status, n, 1, N, CHK_BWD_PARAM);
  const float g_alpha = gated && n_ok ? tof(static_cast<const TIn*>(p.alpha)[n]) : 0.f;
  const float g_beta = gated && n_ok ? tof(static_cast<const TIn*>(p.beta)[n]) : 0.f;
  float dalpha_acc = 0.f, dbeta_acc = 0.f;  // gate parameter sums of this thread's steps
  const TIn* dy = static_cast<const TIn*>(p.dy);
  const TIn* Wn = static_cast<const TIn*>(p.W) + static_cast<size_t>(n) * V * V;
  const TIn* wr = static_cast<const TIn*>(p.w_r) + static_cast<size_t>(n) * V;

  // W as the B operand of H W (k = l, n = j) and of D W^T (k = j, n = l).
  uint32_t Bw[KS][NT][2], Bwl[KS][NT][2], Bt[KS][NT][2], Btl[KS][NT][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kk = 16 * ks + 8 * h + 2 * c, nn = 8 * nt + g;
        const float w0 = n_ok ? tof(Wn[kk * V + nn]) : 0.f, w1 = n_ok ? tof(Wn[(kk + 1) * V + nn]) : 0.f;
        Bw[ks][nt][h] = ptx::pack_bf16x2(w0, w1);
        Bwl[ks][nt][h] = F32 ? ptx::pack_bf16x2(w0 - ptx::bf16x2_lo(Bw[ks][nt][h]),
                                                w1 - ptx::bf16x2_hi(Bw[ks][nt][h]))
                             : 0u;
        const float t0 = n_ok ? tof(Wn[nn * V + kk]) : 0.f, t1 = n_ok ? tof(Wn[nn * V + kk + 1]) : 0.f;
        Bt[ks][nt][h] = ptx::pack_bf16x2(t0, t1);
        Btl[ks][nt][h] = F32 ? ptx::pack_bf16x2(t0 - ptx::bf16x2_lo(Bt[ks][nt][h]),
                                                t1 - ptx::bf16x2_hi(Bt[ks][nt][h]))
                             : 0u;
      }

  const size_t sidx = (static_cast<size_t>(b) * N + n) * K * V;  // [K][V] block of (b, n)
  // C (state gradient) for this thread's elements, from dH_T or 0.
  float Cg[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = row0 + g + 8 * (r >> 1), col = 8 * nt + 2 * c + (r & 1);
      const size_t o = sidx + row * V + col;
      Cg[nt][r] = p.dHT && in_range(p.status, o, 1, s_ext, CHK_BWD_DHT) ? p.dHT[o] : 0.f;
    }
  float dW[KS][NT][4];
#pragma unroll
  for (int a = 0; a < KS; ++a)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) dW[a][nt][0] = dW[a][nt][1] = dW[a][nt][2] = dW[a][nt][3] = 0.f;
  float dwr_acc = 0.f;  // this thread's column tid % V of sum_t u (.) v (slice 0)

  // thread-private sub-checkpoint slot (lane-contiguous 16-byte groups)
  const uint32_t lane16 = static_cast<uint32_t>(lane * 16);
  auto subck_slot = [&](int buf, int idx, int nt) -> uint32_t {
    return sb + L.subck + buf * L.sbuf + static_cast<uint32_t>(((idx * WPC + warp) * NT + nt) * 512) +
           lane16;
  };
  const uint32_t kq_row = static_cast<uint32_t>((16 * warp) * es);  // this warp's rows

  // rank-1 inputs of local step s of the interval held in k/v/f buffer buf
  auto step_in = [&](int buf, int s, float& k0, float& k1, float2 (&vv)[NT], float& fg) {
    const uint32_t a = sb + L.in_k + buf * L.kbuf + static_cast<uint32_t>(s * RS * es) + kq_row;
    k0 = one_f32<F32>(a + g * es);
    k1 = one_f32<F32>(a + (g + 8) * es);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      vv[nt] = pair_f32<F32>(sb + L.in_v + buf * L.vbuf +
                             static_cast<uint32_t>((s * V + 8 * nt + 2 * c) * es));
    fg = ptx::lds_f32(sb + L.in_f + buf * L.fbuf + 4 * s);
  };
  // cooperative loads of an interval's inputs (Lc steps from t0)
  auto load_qdy = [&](int t0, int Lc) {
    const size_t bt0 = static_cast<size_t>(b) * T + t0;
    const int qv = RS * es / 16;  // 16-byte vectors per step
    for (int e = tid; e < Lc * qv; e += nthr) {
      const int s = e / qv, x = e - s * qv;
      const size_t so = ((bt0 + s) * Nq + gq) * K + row0c;
      if (!in_range(p.status, so + x * (16 / es), 16 / es, qk_ext, CHK_BWD_IN)) continue;
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(q + so) + x);
      sts_u32x4(sb + L.in_q + static_cast<uint32_t>(s * RS * es + 16 * x), a.x, a.y, a.z, a.w);
    }
    const int vvn = V * es / 16;
    for (int e = tid; e < Lc * vvn; e += nthr) {
      const int s = e / vvn, x = e - s * vvn;
      const size_t so = ((bt0 + s) * N + n) * V;
      if (!in_range(p.status, so + x * (16 / es), 16 / es, v_ext, CHK_BWD_IN)) continue;
      const uint4 d = __ldg(reinterpret_cast<const uint4*>(dy + so) + x);
      sts_u32x4(sb + L.in_dy + static_cast<uint32_t>(s * V * es + 16 * x), d.x, d.y, d.z, d.w);
    }
  };
  auto load_kvf = [&](int t0, int Lc, int buf) {
    const size_t bt0 = static_cast<size_t>(b) * T + t0;
    const uint32_t kb = sb + L.in_k + buf * L.kbuf, vb = sb + L.in_v + buf * L.vbuf;
    const int qv = RS * es / 16;
    for (int e = tid; e < Lc * qv; e += nthr) {
      const int s = e / qv, x = e - s * qv;
      const size_t so = ((bt0 + s) * Nq + gq) * K + row0c;
      if (!in_range(p.status, so + x * (16 / es), 16 / es, qk_ext, CHK_BWD_IN)) continue;
      const uint4 d = __ldg(reinterpret_cast<const uint4*>(kin + so) + x);
      sts_u32x4(kb + static_cast<uint32_t>(s * RS * es + 16 * x), d.x, d.y, d.z, d.w);
    }
    const int vvn = V * es / 16;
    for (int e = tid; e < Lc * vvn; e += nthr) {
      const int s = e / vvn, x = e - s * vvn;
      const size_t so = ((bt0 + s) * N + n) * V;
      if (!in_range(p.status, so + x * (16 / es), 16 / es, v_ext, CHK_BWD_IN)) continue;
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(vin + so) + x);
      sts_u32x4(vb + static_cast<uint32_t>(s * V * es + 16 * x), a.x, a.y, a.z, a.w);
    }
    for (int s = tid; s < Lc; s += nthr) {
      if (!in_range(p.status, (bt0 + s) * N + n, 1, f_ext, CHK_BWD_IN)) continue;
      const float x = tof(fin[(bt0 + s) * N + n]);
      ptx::sts_f32(sb + L.in_f + buf * L.fbuf + 4 * s, gated ? gate_f(x, g_alpha, g_beta) : x);
    }
  };
  // checkpoint H_{ci C} of this thread's elements
  auto load_ckpt = [&](int ci, float (&H)[NT][4]) {
    const size_t ck0 = ((static_cast<size_t>(b) * N + n) * p.nck + ci) * K * V;
    const float* ck = p.ckpt + ck0;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int o = (row0 + g + 8 * h) * V + 8 * nt + 2 * c;
        const float2 x = in_range(p.status, ck0 + o, 2, s_ext * p.nck, CHK_BWD_CKPT)
                             ? *reinterpret_cast<const float2*>(ck + o)
                             : make_float2(0.f, 0.f);
        H[nt][2 * h] = x.x;
        H[nt][2 * h + 1] = x.y;
      }
  };
  // interval recompute, one step at a time: steps [m0, m1) of the interval in
  // buffer buf, storing a sub-checkpoint before every S2-th step
  auto interval_recompute = [&](int buf, int m0, int m1, float (&H)[NT][4], uint32_t (&A)[KS][4],
                                uint32_t (&Al)[KS][4]) {
#pragma unroll 1
    for (int m = m0; m < m1; ++m) {
      if (m % S2 == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          ptx::sts_f32x4(subck_slot(buf, m / S2, nt), H[nt][0], H[nt][1], H[nt][2], H[nt][3]);
      }
      float k0, k1, fg, Sd[NT][4], Ed[NT][4];
      float2 vv[NT];
      step_in(buf, m, k0, k1, vv, fg);
      recompute_step<V, F32>(H, A, Al, Bw, Bwl, k0, k1, vv, fg, Sd, Ed);
    }
  };

  const int nck = p.nck;
  // state of the interval recompute
  float H1[NT][4];
  uint32_t A1[KS][4], Al1[KS][4];

#pragma unroll 1
  for (int ci = nck - 1; ci >= 0; --ci) {
    const int t0 = ci * C;
    const int Lc = min(C, T - t0);
    const int buf = 0;
    // ---- 1. inputs -> shared memory ----
    __syncthreads();
    load_qdy(t0, Lc);
    load_kvf(t0, Lc, 0);
    load_ckpt(ci, H1);
    __syncthreads();
    pack_frag<V>(H1, A1);
    if (F32) pack_frag_lo<V>(H1, A1, Al1);
    // ---- 2. recompute the interval, sub-checkpoint every S2 steps ----
    interval_recompute(0, 0, Lc, H1, A1, Al1);

    // ---- 3. sub-intervals, last first ----
    const int nsub = (Lc + S2 - 1) / S2;
#pragma unroll 1
    for (int j = nsub - 1; j >= 0; --j) {
      const int s0 = j * S2;
      const int Ls = min(S2, Lc - s0);
      const int rb = j & 1;  // partial-results buffer of this sub-interval
      float H[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float4 x = ptx::lds_f32x4(subck_slot(buf, j, nt));
        H[nt][0] = x.x;
        H[nt][1] = x.y;
        H[nt][2] = x.z;
        H[nt][3] = x.w;
      }
      uint32_t A[KS][4], Al[KS][4];
      pack_frag<V>(H, A);
      if (F32) pack_frag_lo<V>(H, A, Al);
      // registers for the sub-interval: bf16(H_{s0+i}) fragments, s and e
      uint32_t Hf[S2 + 1][KS][4];
      float Sreg[S2][NT][4];
      float Ef[F32 ? S2 : 1][NT][4];       // fp32 e (fp32-input path)
      uint32_t Eb[F32 ? 1 : S2][KS][4];    // fp16 e (bf16 path), A-fragment order
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int e = 0; e < 4; ++e) Hf[0][ks][e] = A[ks][e];
      // S2 recompute steps (steps past Ls run on buffer padding and are not
      // used)
#pragma unroll
      for (int i = 0; i < S2; ++i) {
        float k0, k1, fg, Ed[NT][4];
        float2 vv[NT];
        step_in(buf, s0 + i, k0, k1, vv, fg);
        recompute_step<V, F32>(H, A, Al, Bw, Bwl, k0, k1, vv, fg, Sreg[i], Ed);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int e = 0; e < 4; ++e) Hf[i + 1][ks][e] = A[ks][e];
        if constexpr (F32) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) Ef[i][nt][r] = Ed[nt][r];
        } else {
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            Eb[i][ks][0] = ptx::pack_f16x2(Ed[2 * ks][0], Ed[2 * ks][1]);
            Eb[i][ks][1] = ptx::pack_f16x2(Ed[2 * ks][2], Ed[2 * ks][3]);
            Eb[i][ks][2] = ptx::pack_f16x2(Ed[2 * ks + 1][0], Ed[2 * ks + 1][1]);
            Eb[i][ks][3] = ptx::pack_f16x2(Ed[2 * ks + 1][2], Ed[2 * ks + 1][3]);
          }
        }
      }
      // reverse steps S2-1 .. 0 (those below Ls); full sub-intervals take a
      // branch-free instantiation
      auto reverse = [&](auto full_tag) {
        constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
        for (int i = S2 - 1; i >= 0; --i) {
          if (FULL || i < Ls) {
            const int s = s0 + i;
            const uint32_t qrow = sb + L.in_q + static_cast<uint32_t>(s * RS * es) + kq_row;
            const uint32_t krow = sb + L.in_k + buf * L.kbuf + static_cast<uint32_t>(s * RS * es) + kq_row;
            const uint32_t vrow = sb + L.in_v + buf * L.vbuf + static_cast<uint32_t>(s * V * es);
            const uint32_t urow = sb + L.in_dy + static_cast<uint32_t>(s * V * es);
            const float qa = one_f32<F32>(qrow + g * es), qb = one_f32<F32>(qrow + (g + 8) * es);
            const float fg = ptx::lds_f32(sb + L.in_f + buf * L.fbuf + 4 * s);
            float2 u[NT];
            uint32_t ub[KS][2], vb[KS][2], kb[2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              u[nt] = pair_f32<F32>(urow + static_cast<uint32_t>((8 * nt + 2 * c) * es));
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t off = static_cast<uint32_t>((16 * ks + 8 * h + 2 * c) * es);
                ub[ks][h] = pair_bf16<F32>(urow + off);
                vb[ks][h] = pair_bf16<F32>(vrow + off);
              }
            kb[0] = pair_bf16<F32>(krow + 2 * c * es);
            kb[1] = pair_bf16<F32>(krow + (8 + 2 * c) * es);

            // R = C + q u^T;  D = R (.) s;  df partial = <R, e>
            float R[NT][4], D[NT][4];
            float dfp = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              float ev[4];
              if constexpr (F32) {
#pragma unroll
                for (int r = 0; r < 4; ++r) ev[r] = Ef[i][nt][r];
              } else {
                const int ks = nt >> 1, hh = 2 * (nt & 1);
                ev[0] = ptx::f16x2_lo(Eb[i][ks][hh]);
                ev[1] = ptx::f16x2_hi(Eb[i][ks][hh]);
                ev[2] = ptx::f16x2_lo(Eb[i][ks][hh + 1]);
                ev[3] = ptx::f16x2_hi(Eb[i][ks][hh + 1]);
              }
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                const float qr = (r < 2) ? qa : qb;
                const float ur = (r & 1) ? u[nt].y : u[nt].x;
                R[nt][r] = fmaf(qr, ur, Cg[nt][r]);
                D[nt][r] = R[nt][r] * Sreg[i][nt][r];
                dfp = fmaf(R[nt][r], ev[r], dfp);
              }
            }
            uint32_t Dh[KS][4], Dl[KS][4];
            pack_frag<V>(D, Dh);
            pack_frag_lo<V>(D, Dh, Dl);
            // C_{t-1} = f R + D W^T   (D as hi + lo bf16 parts)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int r = 0; r < 4; ++r) Cg[nt][r] = fg * R[nt][r];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                ptx::mma_bf16_16816(Cg[nt], Dh[ks], Bt[ks][nt][0], Bt[ks][nt][1]);
                ptx::mma_bf16_16816(Cg[nt], Dl[ks], Bt[ks][nt][0], Bt[ks][nt][1]);
                if (F32) ptx::mma_bf16_16816(Cg[nt], Dh[ks], Btl[ks][nt][0], Btl[ks][nt][1]);
              }
            // dk rows = D v;  dq rows = H_t u  (columns of B all equal)
            float dk4[4], dq4[4];
            ptx::mma_bf16_16816_zero(dk4, Dh[0], vb[0][0], vb[0][1]);
            ptx::mma_bf16_16816_zero(dq4, Hf[i + 1][0], ub[0][0], ub[0][1]);
#pragma unroll
            for (int ks = 1; ks < KS; ++ks) {
              ptx::mma_bf16_16816(dk4, Dh[ks], vb[ks][0], vb[ks][1]);
              ptx::mma_bf16_16816(dq4, Hf[i + 1][ks], ub[ks][0], ub[ks][1]);
            }
            // transposed fragments of D and H_{t-1}
            uint32_t DT[KS][4], HT[KS][4];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                DT[ks][e] = ptx::movmatrix_trans(Dh[ks][e]);
                HT[ks][e] = ptx::movmatrix_trans(Hf[i][ks][e]);
              }
            // dW += H_{t-1}^T D: m-tile over l (= k-step ml of H), n-tile over j
#pragma unroll
            for (int ml = 0; ml < KS; ++ml) {
              const uint32_t Aa[4] = {HT[ml][0], HT[ml][2], HT[ml][1], HT[ml][3]};
#pragma unroll
              for (int nj = 0; nj < NT; ++nj)
                ptx::mma_bf16_16816(dW[ml][nj], Aa, DT[nj >> 1][2 * (nj & 1)],
                                    DT[nj >> 1][2 * (nj & 1) + 1]);
            }
            // dv (this warp's rows) = D^T k: m-tile over j
            float dv4[KS][4];
#pragma unroll
            for (int mj = 0; mj < KS; ++mj) {
              const uint32_t Aa[4] = {DT[mj][0], DT[mj][2], DT[mj][1], DT[mj][3]};
              ptx::mma_bf16_16816_zero(dv4[mj], Aa, kb[0], kb[1]);
            }
            // warp sum of the df partial
            dfp += __shfl_xor_sync(0xffffffffu, dfp, 1);
            dfp += __shfl_xor_sync(0xffffffffu, dfp, 2);
            dfp += __shfl_xor_sync(0xffffffffu, dfp, 4);
            dfp += __shfl_xor_sync(0xffffffffu, dfp, 8);
            dfp += __shfl_xor_sync(0xffffffffu, dfp, 16);
            const int ri = rb * S2 + i;  // row of the partial-results buffers
            if (c == 0) {
              const uint32_t rq = sb + L.r_dq + static_cast<uint32_t>((ri * RS + 16 * warp + g) * 4);
              const uint32_t rk = sb + L.r_dk + static_cast<uint32_t>((ri * RS + 16 * warp + g) * 4);
              ptx::sts_f32(rq, dq4[0]);
              ptx::sts_f32(rq + 32, dq4[2]);
              ptx::sts_f32(rk, dk4[0]);
              ptx::sts_f32(rk + 32, dk4[2]);
#pragma unroll
              for (int mj = 0; mj < KS; ++mj) {
                const uint32_t rv =
                    sb + L.r_dv + static_cast<uint32_t>(((ri * WPC + warp) * V + 16 * mj + g) * 4);
                ptx::sts_f32(rv, dv4[mj][0]);
                ptx::sts_f32(rv + 32, dv4[mj][2]);
              }
            }
            if (lane == 0)
              ptx::sts_f32(sb + L.r_df + static_cast<uint32_t>((ri * WPC + warp) * 4), dfp);
          }
        }
      };
      if (Ls == S2)
        reverse(std::true_type{});
      else
        reverse(std::false_type{});
      // ---- flush the sub-interval's per-step results (buffer rb) ----
      // One barrier per sub-interval: the next sub-interval writes the other
      // buffer, and the one after that is behind the next barrier.
      __syncthreads();
      {
        const size_t bt = static_cast<size_t>(b) * T + t0 + s0;
        const int r4 = RS / 4;
        const uint32_t rq = sb + L.r_dq + static_cast<uint32_t>(rb * S2 * RS * 4);
        const uint32_t rk = sb + L.r_dk + static_cast<uint32_t>(rb * S2 * RS * 4);
        const uint32_t rv = sb + L.r_dv + static_cast<uint32_t>(rb * S2 * WPC * V * 4);
        const uint32_t rf = sb + L.r_df + static_cast<uint32_t>(rb * S2 * WPC * 4);
        for (int e = tid; e < Ls * r4; e += nthr) {
          const int i = e / r4, x = e - i * r4;
          const float4 a = ptx::lds_f32x4(rq + static_cast<uint32_t>((i * RS + 4 * x) * 4));
          const float4 d = ptx::lds_f32x4(rk + static_cast<uint32_t>((i * RS + 4 * x) * 4));
          const size_t qo = ((bt + i) * Nq + gq) * K + row0c + 4 * x;
          if (!in_range(p.status, qo, 4, qk_ext, CHK_BWD_DQK)) continue;
          red_add_v4(p.dq + qo, a.x, a.y, a.z, a.w);
          red_add_v4(p.dk + qo, d.x, d.y, d.z, d.w);
        }
        for (int e = tid; e < Ls * V; e += nthr) {
          const int i = e / V, jj = e - i * V;
          float acc = 0.f;
          for (int w = 0; w < WPC; ++w)
            acc += ptx::lds_f32(rv + static_cast<uint32_t>(((i * WPC + w) * V + jj) * 4));
          const int s = s0 + i;
          const float uu = one_f32<F32>(sb + L.in_dy + static_cast<uint32_t>((s * V + jj) * es));
          const float vv = one_f32<F32>(sb + L.in_v + buf * L.vbuf + static_cast<uint32_t>((s * V + jj) * es));
          const size_t vo = ((bt + i) * N + n) * V + jj;
          float* dst = p.dv + vo;
          if (!in_range(p.status, vo, 1, v_ext, CHK_BWD_DV) ||
              !in_range(p.status, static_cast<size_t>(n) * V + jj, 1, static_cast<size_t>(N) * V,
                        CHK_BWD_PARAM))
            continue;
          if (p.nslices == 1) {
            *dst = fmaf(tof(wr[jj]), uu, acc);
          } else {
            red_add(dst, slice == 0 ? fmaf(tof(wr[jj]), uu, acc) : acc);
          }
          if (slice == 0) dwr_acc = fmaf(uu, vv, dwr_acc);  // e % V == tid % V throughout
        }
        for (int i = tid; i < Ls; i += nthr) {
          float acc = 0.f;
          for (int w = 0; w < WPC; ++w) acc += ptx::lds_f32(rf + static_cast<uint32_t>((i * WPC + w) * 4));
          if (!in_range(p.status, (bt + i) * N + n, 1, f_ext, CHK_BWD_DF)) continue;
          if (gated) {  // chain rule through the gate: this slice's share of da, dalpha, dbeta
            float gf, gda, gdal;
            gate_f_grads(tof(fin[(bt + i) * N + n]), g_alpha, g_beta, gf, gda, gdal);
            dalpha_acc = fmaf(acc, gdal, dalpha_acc);
            acc *= gda;
            dbeta_acc += acc;
          }
          float* dst = p.df + (bt + i) * N + n;
          if (p.nslices == 1)
            *dst = acc;
          else
            red_add(dst, acc);
        }
      }
    }
    // C now holds dL/dH_{t0}: the gradient of this interval's checkpoint.
    if (p.dckpt != nullptr && ci % p.dck_ratio == 0) {
      const size_t d0 = ((static_cast<size_t>(b) * N + n) * p.dck_n + ci / p.dck_ratio) * K * V;
      float* dst = p.dckpt + d0;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int o = (row0 + g + 8 * h) * V + 8 * nt + 2 * c;
          if (in_range(p.status, d0 + o, 2, s_ext * p.dck_n, CHK_BWD_DCKPT))
            *reinterpret_cast<float2*>(dst + o) = make_float2(Cg[nt][2 * h], Cg[nt][2 * h + 1]);
        }
    }
  }

  // ---- end: dH0, dW, dw_r ----
  if (p.dH0 != nullptr) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const size_t o = sidx + (row0 + g + 8 * h) * V + 8 * nt + 2 * c;
        if (in_range(p.status, o, 2, s_ext, CHK_BWD_DH0))
          *reinterpret_cast<float2*>(p.dH0 + o) = make_float2(Cg[nt][2 * h], Cg[nt][2 * h + 1]);
      }
  }
  // dW: this warp's [V][V] sum -> shared memory (over the sub-checkpoints,
  // no longer read) -> CTA sum -> global
  __syncthreads();
  {
    const uint32_t base = sb + L.dwsum + static_cast<uint32_t>(warp * V * V * 4);
#pragma unroll
    for (int ml = 0; ml < KS; ++ml)
#pragma unroll
      for (int nj = 0; nj < NT; ++nj)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int l = 16 * ml + g + 8 * (r >> 1), jj = 8 * nj + 2 * c + (r & 1);
          ptx::sts_f32(base + static_cast<uint32_t>((l * V + jj) * 4), dW[ml][nj][r]);
        }
  }
  __syncthreads();
  for (int e = tid; e < V * V; e += nthr) {
    float acc = 0.f;
    for (int w = 0; w < WPC; ++w)
      acc += ptx::lds_f32(sb + L.dwsum + static_cast<uint32_t>((w * V * V + e) * 4));
    if (n_ok) red_add(p.dW + static_cast<size_t>(n) * V * V + e, acc);
  }
  // each thread holds the u (.) v sum of column tid % V over the steps it flushed
  if (slice == 0 && n_ok) red_add(p.dw_r + static_cast<size_t>(n) * V + tid % V, dwr_acc);
  if (gated && tid < S2 && n_ok) {  // the threads that flushed df
    red_add(p.dalpha + n, dalpha_acc);
    red_add(p.dbeta + n, dbeta_acc);
  }
}

template <int V, bool F32>
cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t stream) {
  const BwdLayout L = bwd_layout(V, p.C, sub_len<V, F32>(), p.WPC, F32 ? 4 : 2);
  auto kern = p.gated ? bwd_kernel<V, F32, true> : bwd_kernel<V, F32, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(L.total));
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.B) * p.N * p.nslices;
  kern<<<grid, 32 * p.WPC, L.total, stream>>>(p);
  return cudaGetLastError();
}

template <int V, bool F32>
int bwd_ctas_per_sm_t(const BwdParams& p) {
  const BwdLayout L = bwd_layout(V, p.C, sub_len<V, F32>(), p.WPC, F32 ? 4 : 2);
  auto kern = p.gated ? bwd_kernel<V, F32, true> : bwd_kernel<V, F32, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(L.total)) != cudaSuccess)
    return 0;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, 32 * p.WPC, L.total) != cudaSuccess)
    return 0;
  return nb;
}

}  // namespace

int bwd_sub_len(int V, bool f32_inputs) {
  if (V == 16) return f32_inputs ? sub_len<16, true>() : sub_len<16, false>();
  return f32_inputs ? sub_len<32, true>() : sub_len<32, false>();
}

size_t bwd_smem_bytes(int V, int C, int S2, int WPC, bool f32_inputs) {
  return bwd_layout(V, C, S2, WPC, f32_inputs ? 4 : 2).total;
}

int bwd_ctas_per_sm(const BwdParams& p, int V, bool f32_inputs) {
  if (V == 16) return f32_inputs ? bwd_ctas_per_sm_t<16, true>(p) : bwd_ctas_per_sm_t<16, false>(p);
  return f32_inputs ? bwd_ctas_per_sm_t<32, true>(p) : bwd_ctas_per_sm_t<32, false>(p);
}

cudaError_t launch_bwd(const BwdParams& p, int V, bool f32_inputs, cudaStream_t stream) {
  if (p.WPC < 1 || p.WPC > 8 || p.S2 != bwd_sub_len(V, f32_inputs)) return cudaErrorInvalidValue;
  if (V == 16) return f32_inputs ? launch_bwd_t<16, true>(p, stream) : launch_bwd_t<16, false>(p, stream);
  if (V == 32) return f32_inputs ? launch_bwd_t<32, true>(p, stream) : launch_bwd_t<32, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace m2rnn
