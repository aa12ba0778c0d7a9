// m2rnn_bwd_pipe.cu -- pipelined BPTT backward kernel of the M2RNN recurrence
// ("M2RNN: Non-Linear RNNs with Matrix-Valued States", Eqs. (10)-(12); chain
// rule of the discussion deck's backup frame, written out in m2rnn_bwd.cu).
//
// Same two-level recomputation as the kernel in m2rnn_bwd.cu (checkpoints
// every C steps from the forward pass, sub-checkpoints every S2 steps, S2
// recomputed steps held in registers), organised as a pipeline of slots.
// Slot (c, jj) reverses sub-interval j = nsub(c) - 1 - jj of checkpoint
// interval c and, in the same warps, runs steps [jj S2, jj S2 + S2) of the
// recompute of interval c - 1, which writes that interval's sub-checkpoints.
// In one slot each warp
//   1. starts asynchronous copies (cp.async) of the next slot's inputs into
//      a raw staging area;
//   2. recomputes its S2 steps from the sub-checkpoint, keeping bf16(H_t)
//      (MMA fragments), s = (1 - f)(1 - Z^2) and e = H_{t-1} - Z;
//   3. runs the S2 reverse steps, each paired with one step of the recompute
//      of interval c - 1: two independent dependency chains per warp, and the
//      tanh work of that recompute overlaps the reverse sweep;
//   4. after the copies complete and a barrier, reduces the slot's per-step
//      partials (dq, dk, dv, df) to global memory and converts the staged
//      inputs into the other half of a double-buffered input area; a second
//      barrier follows.
// Inputs sit in shared memory in the form the loops consume: (k, k) fp32
// pairs per accumulator row, v and dy pairs in lane order, bf16 pairs for the
// MMA B operands.  All address strides are compile-time constants.
//
// One sub-checkpoint buffer serves both intervals in flight: interval c keeps
// sub-checkpoint m in slot m (c even) or NS1 - 1 - m (c odd).  Slot (c, jj)
// reads slot phys(c, nsub(c) - 1 - jj) before it writes phys(c - 1, jj), which
// is the same slot when nsub(c) = NS1 and one already read otherwise.  The
// slots are thread-private (each thread keeps its own accumulator elements),
// so program order is enough.
//
// Steps past the end of an interval (ragged sub-intervals) are recomputed on
// stale buffer contents and their results are never used.  Synchronisation is
// __syncthreads only; there are no spin waits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "m2rnn.h"
#include "m2rnn_bwd_common.cuh"
#include "m2rnn_gate.cuh"
#include "m2rnn_check.cuh"
#include "m2rnn_internal.h"
#include "ptx.cuh"

namespace m2rnn {
namespace {

using namespace bwdc;

// Shared-memory layout (byte offsets).  Everything but the sub-checkpoint
// region, which comes last, is fixed by (V, S2, WPC, input size).
struct PipeLayout {
  uint32_t buf0;   // two input buffers at buf0 + k * bufsz
  uint32_t bufsz;
  // inside an input buffer: the reversed sub-interval ...
  uint32_t kd;  // [WPC][S2][8 g][4]  fp32 (k_g, k_g, k_g+8, k_g+8)
  uint32_t qd;  // [WPC][S2][8 g][2]  fp32 (q_g, q_g+8)
  uint32_t kb;  // [WPC][S2][4 c][2]  bf16 pairs (k_2c, k_2c+1), (k_8+2c, k_9+2c)
  uint32_t vf;  // [S2][4 c][NT][2]   fp32 (v_8nt+2c, v_8nt+2c+1)
  uint32_t vb;  // [S2][4 c][KS][2]   bf16 pairs (v_16ks+2c, ..), (v_16ks+8+2c, ..)
  uint32_t uf;  // as vf, for dy
  uint32_t ub;  // as vb, for dy
  uint32_t fr;  // [S2] fp32 f
  uint32_t gd, gl;  // [S2] fp32 df/da and df/dalpha of the fused input gate
  // ... and the steps of the interval recomputed alongside
  uint32_t lkd, lvf, lfr;
  uint32_t raw;         // one slot's inputs as copied: q, k, k' [S2][RS], v, dy, v' [S2][V]
                        // (input dtype), then f, f' [S2] (the aligned 32-bit word holding f)
  uint32_t r_dq, r_dk;  // [2][S2][WPC][8 g][2 h] fp32 per-step partials (row 16w + 8h + g)
  uint32_t r_dv;        // [2][S2][WPC][KS][8 g][2 h] fp32 (column 16ks + 8h + g)
  uint32_t r_df;        // [2][S2][WPC] fp32
  uint32_t subck;       // [NS1][WPC][NT][32 lanes][4] fp32; dW partials at the end
};

__host__ __device__ constexpr uint32_t al128(uint32_t x) { return (x + 127u) / 128u * 128u; }

__host__ __device__ constexpr PipeLayout pipe_layout(int V, int S2, int WPC, int es, bool gated) {
  const uint32_t NT = V / 8, KS = V / 16;
  PipeLayout L{};
  uint32_t b = 0;
  L.kd = b;
  b = al128(b + WPC * S2 * 8 * 16);
  L.qd = b;
  b = al128(b + WPC * S2 * 8 * 8);
  L.kb = b;
  b = al128(b + WPC * S2 * 4 * 8);
  L.vf = b;
  b = al128(b + S2 * 4 * NT * 8);
  L.vb = b;
  b = al128(b + S2 * 4 * KS * 8);
  L.uf = b;
  b = al128(b + S2 * 4 * NT * 8);
  L.ub = b;
  b = al128(b + S2 * 4 * KS * 8);
  L.fr = b;
  b = al128(b + S2 * 4);
  L.gd = b;  // (the gate's arrays exist in gated launches only)
  b = gated ? al128(b + S2 * 4) : b;
  L.gl = b;
  b = gated ? al128(b + S2 * 4) : b;
  L.lkd = b;
  b = al128(b + WPC * S2 * 8 * 16);
  L.lvf = b;
  b = al128(b + S2 * 4 * NT * 8);
  L.lfr = b;
  b = al128(b + S2 * 4);
  L.bufsz = b;
  uint32_t o = 0;
  L.buf0 = o;
  o += 2 * b;
  L.raw = o;
  o = al128(o + S2 * 3 * (16 * WPC + V) * es + 2 * S2 * 4);
  L.r_dq = o;
  o = al128(o + 2 * S2 * WPC * 8 * 8);
  L.r_dk = o;
  o = al128(o + 2 * S2 * WPC * 8 * 8);
  L.r_dv = o;
  o = al128(o + 2 * S2 * WPC * KS * 8 * 8);
  L.r_df = o;
  o = al128(o + 2 * S2 * WPC * 4);
  L.subck = o;
  return L;
}
__host__ __device__ constexpr uint32_t pipe_smem_total(int V, int C, int S2, int WPC, int es,
                                                       bool gated) {
  const uint32_t NS1 = (C + S2 - 1) / S2;
  const uint32_t sub = NS1 * WPC * (V / 8) * 512, dws = WPC * V * V * 4;
  return pipe_layout(V, S2, WPC, es, gated).subck + al128(sub > dws ? sub : dws);
}

// One forward step with the forward kernel's operations (rank-1 k v^T in fp32
// pairs seeding the accumulator, H W on the tensor cores, tanh, blend).
// kd = (k_g, k_g, k_g+8, k_g+8).  So = (1 - f)(1 - Z^2), Eo = H_{t-1} - Z.
template <int V, bool F32>
__device__ __forceinline__ void pipe_step(float (&H)[V / 8][4], uint32_t (&A)[V / 16][4],
                                          uint32_t (&Al)[V / 16][4],
                                          const uint32_t (&Bw)[V / 16][V / 8][2],
                                          const uint32_t (&Bwl)[V / 16][V / 8][2], float4 kd,
                                          const float2 (&vv)[V / 8], float fg,
                                          float (&So)[V / 8][4], float (&Eo)[V / 8][4]) {
  constexpr int NT = V / 8, KS = V / 16;
  const float2 kk0 = make_float2(kd.x, kd.y), kk1 = make_float2(kd.z, kd.w);
  const float2 f2 = make_float2(fg, fg), m1 = make_float2(-1.f, -1.f);
  const float2 one2 = make_float2(1.f, 1.f), omf2 = make_float2(1.f - fg, 1.f - fg);
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
      Eo[nt][2 * h] = d.x;
      Eo[nt][2 * h + 1] = d.y;
      const float2 s = __fmul2_rn(omf2, __ffma2_rn(make_float2(-z.x, -z.y), z, one2));
      So[nt][2 * h] = s.x;
      So[nt][2 * h + 1] = s.y;
    }
  pack_frag<V>(H, A);
  if (F32) pack_frag_lo<V>(H, A, Al);
}

// Warp sums of S2 per-lane values with log2(S2) exchange rounds plus a plain
// butterfly: afterwards every lane holds the warp sum of v[step_of_lane].
template <int S2>
__device__ __forceinline__ float reduce_steps(float (&v)[S2], int lane) {
  constexpr int P = S2 == 8 ? 3 : S2 == 4 ? 2 : S2 == 2 ? 1 : 0;
  static_assert((1 << P) == S2, "S2 must be 1, 2, 4 or 8");
#pragma unroll
  for (int r = 0; r < P; ++r) {
    const int m = 16 >> r, half = S2 >> (r + 1);
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = up ? v[k] : v[k + half];
      const float keep = up ? v[k + half] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  float s = v[0];
#pragma unroll
  for (int m = 16 >> P; m >= 1; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
  return s;
}
template <int S2>
__device__ __forceinline__ int step_of_lane(int lane) {
  int idx = 0;
#pragma unroll
  for (int r = 0; r < (S2 == 8 ? 3 : S2 == 4 ? 2 : S2 == 2 ? 1 : 0); ++r)
    if (lane & (16 >> r)) idx += S2 >> (r + 1);
  return idx;
}

template <int V, bool F32, int WPC, bool GATED>
__global__ void __launch_bounds__(32 * WPC) bwd_pipe_kernel(const BwdParams p) {
  using TIn = typename InT<F32>::T;
  constexpr int es = sizeof(TIn);
  constexpr int NT = V / 8, KS = V / 16;
  constexpr int S2 = sub_len<V, F32>();
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  constexpr int RS = 16 * WPC, nthr = 32 * WPC;
  const int K = p.K, T = p.T, N = p.N, C = p.C, nck = p.nck;
  const int NS1 = (C + S2 - 1) / S2;
  const int slice = blockIdx.x % p.nslices;
  const int bn = blockIdx.x / p.nslices;
  const int b = bn / N, n = bn % N;
  const int Nq = p.Nq, gq = n / (N / Nq);  // query/key group of head n
  const int row0c = slice * RS;        // first row of this CTA
  const int row0 = row0c + 16 * warp;  // first row of this warp
  constexpr PipeLayout L = pipe_layout(V, S2, WPC, es, GATED);
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
  float Cg[NT][4];  // dL/dH for this thread's elements, from dH_T or 0
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

  // per-thread byte offsets (step i adds i * the per-step stride)
  const uint32_t o_kd = static_cast<uint32_t>((warp * S2 * 8 + g) * 16);  // + i * 128
  const uint32_t o_qd = static_cast<uint32_t>((warp * S2 * 8 + g) * 8);   // + i * 64
  const uint32_t o_kb = static_cast<uint32_t>((warp * S2 * 4 + c) * 8);   // + i * 32
  const uint32_t o_vf = static_cast<uint32_t>(c * NT * 8);                // + i * 32 NT
  const uint32_t o_vb = static_cast<uint32_t>(c * KS * 8);                // + i * 32 KS
  auto subck_slot = [&](int phys, int nt) -> uint32_t {
    return sb + L.subck + static_cast<uint32_t>(((phys * WPC + warp) * NT + nt) * 512 + lane * 16);
  };
  auto phys = [&](int ci2, int m) { return (ci2 & 1) ? NS1 - 1 - m : m; };
  auto load_ckpt = [&](int ci2, float (&Hc)[NT][4]) {
    const size_t ck0 = ((static_cast<size_t>(b) * N + n) * nck + ci2) * K * V;
    const float* ck = p.ckpt + ck0;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int o = (row0 + g + 8 * h) * V + 8 * nt + 2 * c;
        const float2 x = in_range(p.status, ck0 + o, 2, s_ext * nck, CHK_BWD_CKPT)
                             ? *reinterpret_cast<const float2*>(ck + o)
                             : make_float2(0.f, 0.f);
        Hc[nt][2 * h] = x.x;
        Hc[nt][2 * h + 1] = x.y;
      }
  };

  // ---- inputs of a slot.  R = the reversed sub-interval of interval ci2;
  // L (primed) = steps [jj2 S2, jj2 S2 + S2) of interval ci2 - 1.  They are
  // copied asynchronously (cp.async, 16-byte units in the order
  // [q | k | k' | v | dy | v']) into the raw area, then converted into an
  // input buffer.  Steps past the end of an interval are not copied.
  const int upr = RS * es / 16, upv = V * es / 16;  // 16-byte units per step
  const int nq = S2 * upr, nv = S2 * upv;
  const int U = 3 * nq + 3 * nv;
  const uint32_t raw = sb + L.raw;
  const uint32_t raw_f = raw + static_cast<uint32_t>(S2 * 3 * (RS + V) * es);
  const size_t f_total = static_cast<size_t>(p.B) * T * N;
  struct SlotRange {
    size_t tR, tL;  // first global step (b*T + t) of R and of L
    int nR, nL;     // valid steps of R and of L
  };
  auto slot_range = [&](int ci2, int jj2, bool wantR) {
    SlotRange r;
    r.nR = 0;
    r.tR = 0;
    if (wantR) {
      const int Lc2 = min(C, T - ci2 * C), nsub2 = (Lc2 + S2 - 1) / S2;
      const int s02 = (nsub2 - 1 - jj2) * S2;
      r.tR = static_cast<size_t>(b) * T + ci2 * C + s02;
      r.nR = min(S2, Lc2 - s02);
    }
    r.nL = 0;
    r.tL = 0;
    if (ci2 > 0) {
      const int Lp = min(C, T - (ci2 - 1) * C);
      r.tL = static_cast<size_t>(b) * T + (ci2 - 1) * C + jj2 * S2;
      r.nL = max(0, min(S2, Lp - jj2 * S2));
    }
    return r;
  };
  // Fixed per-thread share of the per-slot staging and flush work (the same
  // in every slot, so it is decoded once here).
  // Copy units: at most three per thread, packed as kind | i << 3 | x << 8
  // (kind 0 q, 1 k, 2 k', 3 v, 4 dy, 5 v'; step i; 16-byte unit x), or -1.
  constexpr int kUnits = 3;  // U = 3 S2 es (WPC + 1) <= 3 * 32 WPC for S2 es = 16
  int ucode[kUnits];
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {
    const int e = tid + u * nthr;
    ucode[u] = -1;
    if (e < U) {
      int r = e, kind = 0;
      if (r >= nq) { r -= nq; kind = 1; }
      if (kind == 1 && r >= nq) { r -= nq; kind = 2; }
      if (kind == 2 && r >= nq) { r -= nq; kind = 3; }
      if (kind == 3 && r >= nv) { r -= nv; kind = 4; }
      if (kind == 4 && r >= nv) { r -= nv; kind = 5; }
      const int per = kind < 3 ? upr : upv;
      ucode[u] = kind | ((r / per) << 3) | ((r % per) << 8);
    }
  }
  // Row item (conversion of q, k, k' and the dq/dk flush): rows r0 .. r0 + 3
  // of step i_r.  Column item (conversion of v, dy, v'): columns j0 .. j0 + 3
  // of step i_c.
  const int rq4 = RS / 4;
  const bool row_ok = tid < S2 * rq4;
  const int i_r = tid / rq4, r0 = 4 * (tid - (tid / rq4) * rq4);
  const int rw = r0 >> 4, rh = (r0 >> 3) & 1, rg = r0 & 7;
  const uint32_t qd_off = static_cast<uint32_t>(((rw * S2 + i_r) * 8 + rg) * 8 + rh * 4);
  const uint32_t kb_off = static_cast<uint32_t>(((rw * S2 + i_r) * 4 + (rg >> 1)) * 8 + rh * 4);
  const uint32_t rsrc = static_cast<uint32_t>((i_r * RS + r0) * es);
  const uint32_t rkind = static_cast<uint32_t>(S2 * RS * es);  // raw bytes per row kind
  const uint32_t fl_off = static_cast<uint32_t>(((i_r * WPC + rw) * 8 + rg) * 8 + rh * 4);
  // column items on warp 1, f on warp 2, df on warp 3 (where they exist)
  constexpr int col_base = WPC >= 2 ? 32 : 0, f_base = WPC >= 3 ? 64 : 0, df_base = WPC >= 4 ? 96 : 0;
  constexpr int vq4 = V / 4;
  const int ct = tid - col_base, ft = tid - f_base, dt = tid - df_base;
  const bool col_ok = ct >= 0 && ct < S2 * vq4;
  const int i_c = ct / vq4, j0c = 4 * (ct % vq4);
  const uint32_t csrc = static_cast<uint32_t>(3 * S2 * RS * es + (i_c * V + j0c) * es);

  auto issue = [&](int ci2, int jj2, bool wantR) {
    const SlotRange sr = slot_range(ci2, jj2, wantR);
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
      const int code = ucode[u];
      if (code < 0) continue;
      const int kind = code & 7, i = (code >> 3) & 31, x = code >> 8;
      const bool isR = kind != 2 && kind != 5;
      if (i >= (isR ? sr.nR : sr.nL)) continue;
      const size_t t = (isR ? sr.tR : sr.tL) + i;
      const size_t so = kind <= 2 ? (t * Nq + gq) * K + row0c : (t * N + n) * V;
      const TIn* src = (kind <= 2 ? (kind == 0 ? q : kin) : (kind == 4 ? dy : vin)) + so;
      if (in_range(p.status, so + x * (16 / es), 16 / es, kind <= 2 ? qk_ext : v_ext, CHK_BWD_IN))
        ptx::cp_async16(raw + static_cast<uint32_t>((tid + u * nthr) * 16),
                        reinterpret_cast<const uint4*>(src) + x);
    }
    if (ft >= 0 && ft < 2 * S2) {  // f of R (ft < S2) and of L: the aligned 32-bit word holding it
      const bool isR = ft < S2;
      const int i = isR ? ft : ft - S2;
      if (i < (isR ? sr.nR : sr.nL)) {
        const size_t idx = ((isR ? sr.tR : sr.tL) + i) * N + n;
        const uint32_t dst = raw_f + 4 * ft;
        if (!in_range(p.status, idx, 1, f_ext, CHK_BWD_IN)) {
          // (checked build: skipped)
        } else if (es == 4 || (idx | 1) < f_total) {
          ptx::cp_async4(dst, fin + (es == 4 ? idx : (idx & ~static_cast<size_t>(1))));
        } else {  // the last element of an odd-length bf16 array: its word would overrun
          const uint32_t bits = __bfloat16_as_ushort(*reinterpret_cast<const __nv_bfloat16*>(fin + idx));
          ptx::sts_u32(dst, bits);  // idx is even here: the low half
        }
      }
    }
    ptx::cp_async_commit();
  };
  auto load4 = [&](uint32_t src, float (&x)[4]) {
    if constexpr (F32) {
      const float4 v4 = ptx::lds_f32x4(src);
      x[0] = v4.x;
      x[1] = v4.y;
      x[2] = v4.z;
      x[3] = v4.w;
    } else {
      const uint2 w = ptx::lds_u32x2(src);
      x[0] = ptx::bf16x2_lo(w.x);
      x[1] = ptx::bf16x2_hi(w.x);
      x[2] = ptx::bf16x2_lo(w.y);
      x[3] = ptx::bf16x2_hi(w.y);
    }
  };
  // raw area -> input buffer bufo.  Invalid steps are converted too (stale
  // contents; their results are never used).
  auto convert = [&](int ci2, int jj2, bool wantR, int bufo) {
    const uint32_t B0 = sb + L.buf0 + static_cast<uint32_t>(bufo) * L.bufsz;
    if (row_ok) {
#pragma unroll
      for (int kind = 0; kind < 3; ++kind) {
        if (!wantR && kind != 2) continue;
        float x[4];
        load4(raw + kind * rkind + rsrc, x);
        if (kind == 0) {
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) ptx::sts_f32(B0 + L.qd + qd_off + e2 * 8, x[e2]);
        } else {
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2)
            ptx::sts_f32x2(B0 + (kind == 1 ? L.kd : L.lkd) + 2 * qd_off + e2 * 16, x[e2], x[e2]);
          if (kind == 1) {
            ptx::sts_u32(B0 + L.kb + kb_off, ptx::pack_bf16x2(x[0], x[1]));
            ptx::sts_u32(B0 + L.kb + kb_off + 8, ptx::pack_bf16x2(x[2], x[3]));
          }
        }
      }
    }
    if (col_ok) {
#pragma unroll
      for (int kind = 3; kind < 6; ++kind) {
        if (!wantR && kind != 5) continue;
        float x[4];
        load4(raw + csrc + static_cast<uint32_t>((kind - 3) * S2 * V * es), x);
        const uint32_t fo = kind == 3 ? L.vf : kind == 4 ? L.uf : L.lvf;
        const uint32_t bo = kind == 3 ? L.vb : L.ub;
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          const int j = j0c + 2 * k2, nt = j >> 3, cc = (j & 7) >> 1, ks = j >> 4, hh = (j >> 3) & 1;
          ptx::sts_f32x2(B0 + fo + static_cast<uint32_t>(((i_c * 4 + cc) * NT + nt) * 8), x[2 * k2],
                         x[2 * k2 + 1]);
          if (kind != 5)
            ptx::sts_u32(B0 + bo + static_cast<uint32_t>(((i_c * 4 + cc) * KS + ks) * 8 + hh * 4),
                         ptx::pack_bf16x2(x[2 * k2], x[2 * k2 + 1]));
        }
      }
    }
    if (ft >= 0 && ft < 2 * S2) {
      const bool isR = ft < S2;
      const int i = isR ? ft : ft - S2;
      if (wantR || !isR) {
        const uint32_t wbits = ptx::lds_u32(raw_f + 4 * ft);
        float fv;
        if constexpr (F32) {
          fv = __uint_as_float(wbits);
        } else {
          const SlotRange sr = slot_range(ci2, jj2, wantR);
          const size_t idx = ((isR ? sr.tR : sr.tL) + i) * N + n;
          fv = (idx & 1) ? ptx::bf16x2_hi(wbits) : ptx::bf16x2_lo(wbits);
        }
        if (gated) {  // fv is a: f and, for reversed steps, its derivatives
          float gf, gda, gdal;
          gate_f_grads(fv, g_alpha, g_beta, gf, gda, gdal);
          fv = gf;
          if (isR) {
            ptx::sts_f32(B0 + L.gd + 4 * i, gda);
            ptx::sts_f32(B0 + L.gl + 4 * i, gdal);
          }
        }
        ptx::sts_f32(B0 + (isR ? L.fr : L.lfr) + 4 * i, fv);
      }
    }
  };

  // state of the recompute of the interval before the reversed one
  float H1[NT][4];
  uint32_t A1[KS][4], Al1[KS][4];
  // one recompute step of that interval from input buffer B0, step mi
  auto l1_step = [&](uint32_t B0, int mi) {
    float Sd[NT][4], Ed[NT][4];
    float2 vv[NT];
    const float4 kd = ptx::lds_f32x4(B0 + L.lkd + o_kd + mi * 128);
#pragma unroll
    for (int nt = 0; nt < NT; nt += 2) {
      const float4 t4 = ptx::lds_f32x4(B0 + L.lvf + o_vf + mi * 32 * NT + nt * 8);
      vv[nt] = make_float2(t4.x, t4.y);
      vv[nt + 1] = make_float2(t4.z, t4.w);
    }
    const float fg = ptx::lds_f32(B0 + L.lfr + 4 * mi);
    pipe_step<V, F32>(H1, A1, Al1, Bw, Bwl, kd, vv, fg, Sd, Ed);
  };
  auto store_subck = [&](int ph, const float (&Hs)[NT][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      ptx::sts_f32x4(subck_slot(ph, nt), Hs[nt][0], Hs[nt][1], Hs[nt][2], Hs[nt][3]);
  };
  // serial recompute of S2-step chunks [j0, j1) of the interval ci2 - 1 (or,
  // with ci2 = nck, of the last interval), inputs through buffer bufi
  auto serial_chunks = [&](int ci2, int j0, int j1, int bufi) {
    const uint32_t B0 = sb + L.buf0 + static_cast<uint32_t>(bufi) * L.bufsz;
#pragma unroll 1
    for (int jc = j0; jc < j1; ++jc) {
      issue(ci2, jc, false);
      ptx::cp_async_wait_all();
      __syncthreads();
      convert(ci2, jc, false, bufi);
      __syncthreads();
      store_subck(phys(ci2 - 1, jc), H1);
#pragma unroll
      for (int mi = 0; mi < S2; ++mi) l1_step(B0, mi);
      __syncthreads();
    }
  };

  // ---- prologue: sub-checkpoints of the last interval, inputs of the first slot
  {
    const int cl = nck - 1, nl = (T - cl * C + S2 - 1) / S2;
    load_ckpt(cl, H1);
    pack_frag<V>(H1, A1);
    if (F32) pack_frag_lo<V>(H1, A1, Al1);
    serial_chunks(nck, 0, nl, 0);
    issue(cl, 0, true);
    ptx::cp_async_wait_all();
    __syncthreads();
    convert(cl, 0, true, 0);
    __syncthreads();
  }

  int ci = nck - 1, jj = 0, Lc = T - ci * C;
  int nsub = (Lc + S2 - 1) / S2;
  int bufi = 0;
#pragma unroll 1
  while (true) {
    const int j = nsub - 1 - jj;
    const int s0 = j * S2;
    const int Ls = min(S2, Lc - s0);
    const bool have_l1 = ci > 0;
    const uint32_t B0 = sb + L.buf0 + static_cast<uint32_t>(bufi) * L.bufsz;
    const int rb = bufi;  // partial-results buffer of this slot
    int nci = ci, njj = jj + 1;
    if (njj == nsub) {
      nci = ci - 1;
      njj = 0;
    }
    if (jj == 0 && have_l1) load_ckpt(ci - 1, H1);  // used after the sub-interval recompute
    if (nci >= 0) issue(nci, njj, true);  // lands in the raw area during this slot

    // ---- 2. recompute the sub-interval from its sub-checkpoint ----
    float H[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float4 x = ptx::lds_f32x4(subck_slot(phys(ci, j), nt));
      H[nt][0] = x.x;
      H[nt][1] = x.y;
      H[nt][2] = x.z;
      H[nt][3] = x.w;
    }
    uint32_t A[KS][4], Al[KS][4];
    pack_frag<V>(H, A);
    if (F32) pack_frag_lo<V>(H, A, Al);
    uint32_t Hf[S2 + 1][KS][4];           // bf16(H_{s0+i}) as MMA A fragments
    float Sreg[S2][NT][4];                // s = (1 - f)(1 - Z^2)
    float Ef[F32 ? S2 : 1][NT][4];        // e = H_{t-1} - Z, fp32 (fp32-input path)
    uint32_t Eb[F32 ? 1 : S2][KS][4];     // e as fp16 pairs in A-fragment order (bf16 path)
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int e = 0; e < 4; ++e) Hf[0][ks][e] = A[ks][e];
#pragma unroll
    for (int i = 0; i < S2; ++i) {
      float Ed[NT][4];
      float2 vv[NT];
      const float4 kd = ptx::lds_f32x4(B0 + L.kd + o_kd + i * 128);
#pragma unroll
      for (int nt = 0; nt < NT; nt += 2) {
        const float4 t4 = ptx::lds_f32x4(B0 + L.vf + o_vf + i * 32 * NT + nt * 8);
        vv[nt] = make_float2(t4.x, t4.y);
        vv[nt + 1] = make_float2(t4.z, t4.w);
      }
      const float fg = ptx::lds_f32(B0 + L.fr + 4 * i);
      pipe_step<V, F32>(H, A, Al, Bw, Bwl, kd, vv, fg, Sreg[i], Ed);
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
    if (jj == 0) {
      pack_frag<V>(H1, A1);
      if (F32) pack_frag_lo<V>(H1, A1, Al1);
    }

    // ---- 3. reverse steps, each paired with a recompute step of ci - 1 ----
    float dfv[S2];
    auto reverse = [&](auto full_tag) {
      constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
      for (int i = S2 - 1; i >= 0; --i) {
        if (i == S2 - 1 && have_l1) store_subck(phys(ci - 1, jj), H1);
        l1_step(B0, S2 - 1 - i);
        dfv[i] = 0.f;
        if (FULL || i < Ls) {
          const float2 qq = ptx::lds_f32x2(B0 + L.qd + o_qd + i * 64);
          const float fg = ptx::lds_f32(B0 + L.fr + 4 * i);
          float2 u[NT];
#pragma unroll
          for (int nt = 0; nt < NT; nt += 2) {
            const float4 t4 = ptx::lds_f32x4(B0 + L.uf + o_vf + i * 32 * NT + nt * 8);
            u[nt] = make_float2(t4.x, t4.y);
            u[nt + 1] = make_float2(t4.z, t4.w);
          }
          uint32_t ub[KS][2], vb[KS][2];
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const uint2 a = ptx::lds_u32x2(B0 + L.ub + o_vb + i * 32 * KS + ks * 8);
            const uint2 d = ptx::lds_u32x2(B0 + L.vb + o_vb + i * 32 * KS + ks * 8);
            ub[ks][0] = a.x;
            ub[ks][1] = a.y;
            vb[ks][0] = d.x;
            vb[ks][1] = d.y;
          }
          const uint2 kb = ptx::lds_u32x2(B0 + L.kb + o_kb + i * 32);

          // R = C + q u^T;  D = R (.) s;  df partial = <R, e>;  C <- f R
          float D[NT][4];
          float2 dfp = make_float2(0.f, 0.f);
          const float2 f2 = make_float2(fg, fg);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float qh = h ? qq.y : qq.x;
              const float2 R =
                  __ffma2_rn(make_float2(qh, qh), u[nt], make_float2(Cg[nt][2 * h], Cg[nt][2 * h + 1]));
              const float2 Dv =
                  __fmul2_rn(R, make_float2(Sreg[i][nt][2 * h], Sreg[i][nt][2 * h + 1]));
              float2 ev;
              if constexpr (F32) {
                ev = make_float2(Ef[i][nt][2 * h], Ef[i][nt][2 * h + 1]);
              } else {
                const uint32_t w = Eb[i][nt >> 1][2 * (nt & 1) + h];
                ev = make_float2(ptx::f16x2_lo(w), ptx::f16x2_hi(w));
              }
              dfp = __ffma2_rn(R, ev, dfp);
              D[nt][2 * h] = Dv.x;
              D[nt][2 * h + 1] = Dv.y;
              const float2 cn = __fmul2_rn(f2, R);
              Cg[nt][2 * h] = cn.x;
              Cg[nt][2 * h + 1] = cn.y;
            }
          dfv[i] = dfp.x + dfp.y;
          // D as bf16 hi + lo parts
          uint32_t Dh[KS][4], Dl[KS][4];
          pack_frag<V>(D, Dh);
#pragma unroll
          for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int nt = 2 * ks + (e >> 1), r = 2 * (e & 1);
              const float2 hi = make_float2(ptx::bf16x2_lo(Dh[ks][e]), ptx::bf16x2_hi(Dh[ks][e]));
              const float2 lo = __fadd2_rn(make_float2(D[nt][r], D[nt][r + 1]), make_float2(-hi.x, -hi.y));
              Dl[ks][e] = ptx::pack_bf16x2(lo.x, lo.y);
            }
          // C_{t-1} = f R + D W^T
#pragma unroll
          for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              ptx::mma_bf16_16816(Cg[nt], Dh[ks], Bt[ks][nt][0], Bt[ks][nt][1]);
              ptx::mma_bf16_16816(Cg[nt], Dl[ks], Bt[ks][nt][0], Bt[ks][nt][1]);
              if (F32) ptx::mma_bf16_16816(Cg[nt], Dh[ks], Btl[ks][nt][0], Btl[ks][nt][1]);
            }
          // dk rows = D v;  dq rows = H_t u  (all columns of B equal)
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
          // dW += H_{t-1}^T D: m-tile over l, n-tile over j
#pragma unroll
          for (int ml = 0; ml < KS; ++ml) {
            const uint32_t Aa[4] = {HT[ml][0], HT[ml][2], HT[ml][1], HT[ml][3]};
#pragma unroll
            for (int nj = 0; nj < NT; ++nj)
              ptx::mma_bf16_16816(dW[ml][nj], Aa, DT[nj >> 1][2 * (nj & 1)], DT[nj >> 1][2 * (nj & 1) + 1]);
          }
          // dv (this warp's rows) = D^T k: m-tile over j
          float dv4[KS][4];
#pragma unroll
          for (int mj = 0; mj < KS; ++mj) {
            const uint32_t Aa[4] = {DT[mj][0], DT[mj][2], DT[mj][1], DT[mj][3]};
            ptx::mma_bf16_16816_zero(dv4[mj], Aa, kb.x, kb.y);
          }
          const uint32_t ro = static_cast<uint32_t>((((rb * S2 + i) * WPC + warp) * 8 + g) * 8);
          ptx::sts_f32x2_if(c == 0, sb + L.r_dq + ro, dq4[0], dq4[2]);
          ptx::sts_f32x2_if(c == 0, sb + L.r_dk + ro, dk4[0], dk4[2]);
#pragma unroll
          for (int mj = 0; mj < KS; ++mj)
            ptx::sts_f32x2_if(
                c == 0,
                sb + L.r_dv + static_cast<uint32_t>(((((rb * S2 + i) * WPC + warp) * KS + mj) * 8 + g) * 8),
                dv4[mj][0], dv4[mj][2]);
        }
      }
    };
    if (Ls == S2)
      reverse(std::true_type{});
    else
      reverse(std::false_type{});
    {  // df of the slot's steps: one exchange-reduction for all S2 steps
      const float tot = reduce_steps<S2>(dfv, lane);
      const int idx = step_of_lane<S2>(lane);
      constexpr int grp = 32 / S2;  // lanes holding the same step
      ptx::sts_f32_if((lane & (grp - 1)) == 0 && idx < Ls,
                      sb + L.r_df + static_cast<uint32_t>(((rb * S2 + idx) * WPC + warp) * 4), tot);
    }
    ptx::cp_async_wait_all();
    __syncthreads();

    // ---- 4. per-step results to global memory; inputs of the next slot ----
    {
      const size_t bt = static_cast<size_t>(b) * T + ci * C + s0;
      const uint32_t rq = sb + L.r_dq + static_cast<uint32_t>(rb * S2 * WPC * 64);
      const uint32_t rk = sb + L.r_dk + static_cast<uint32_t>(rb * S2 * WPC * 64);
      const uint32_t rv = sb + L.r_dv + static_cast<uint32_t>(rb * S2 * WPC * KS * 64);
      const uint32_t rf = sb + L.r_df + static_cast<uint32_t>(rb * S2 * WPC * 4);
      const size_t qo = ((bt + i_r) * Nq + gq) * K + row0c + r0;
      if (row_ok && i_r < Ls && in_range(p.status, qo, 4, qk_ext, CHK_BWD_DQK)) {
        const uint32_t o = fl_off;
        red_add_v4(p.dq + qo, ptx::lds_f32(rq + o), ptx::lds_f32(rq + o + 8),
                   ptx::lds_f32(rq + o + 16), ptx::lds_f32(rq + o + 24));
        red_add_v4(p.dk + qo, ptx::lds_f32(rk + o), ptx::lds_f32(rk + o + 8),
                   ptx::lds_f32(rk + o + 16), ptx::lds_f32(rk + o + 24));
      }
      for (int e = tid; e < Ls * V; e += nthr) {
        const int i = e / V, jc = e - i * V;
        const int mj = jc >> 4, hh = (jc >> 3) & 1, gg = jc & 7;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < WPC; ++w)
          acc += ptx::lds_f32(rv + static_cast<uint32_t>((((i * WPC + w) * KS + mj) * 8 + gg) * 8 + hh * 4));
        const uint32_t fo = static_cast<uint32_t>(((i * 4 + ((jc & 7) >> 1)) * NT + (jc >> 3)) * 8 + (jc & 1) * 4);
        const float uu = ptx::lds_f32(B0 + L.uf + fo);
        const float vv = ptx::lds_f32(B0 + L.vf + fo);
        const size_t vo = ((bt + i) * N + n) * V + jc;
        float* dst = p.dv + vo;
        if (!in_range(p.status, vo, 1, v_ext, CHK_BWD_DV) ||
            !in_range(p.status, static_cast<size_t>(n) * V + jc, 1, static_cast<size_t>(N) * V, CHK_BWD_PARAM))
          continue;
        if (p.nslices == 1)
          *dst = fmaf(tof(wr[jc]), uu, acc);
        else
          red_add(dst, slice == 0 ? fmaf(tof(wr[jc]), uu, acc) : acc);
        if (slice == 0) dwr_acc = fmaf(uu, vv, dwr_acc);  // e % V == tid % V throughout
      }
      if (dt >= 0 && dt < Ls) {
        const int i = dt;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < WPC; ++w) acc += ptx::lds_f32(rf + static_cast<uint32_t>((i * WPC + w) * 4));
        if (gated) {  // chain rule through the gate: this slice's share of da, dalpha, dbeta
          const float gda = ptx::lds_f32(B0 + L.gd + 4 * i);
          dalpha_acc = fmaf(acc, ptx::lds_f32(B0 + L.gl + 4 * i), dalpha_acc);
          acc *= gda;
          dbeta_acc += acc;
        }
        const size_t fo = (bt + i) * N + n;
        float* dst = p.df + fo;
        if (in_range(p.status, fo, 1, f_ext, CHK_BWD_DF)) {
          if (p.nslices == 1)
            *dst = acc;
          else
            red_add(dst, acc);
        }
      }
    }
    if (nci >= 0) convert(nci, njj, true, bufi ^ 1);
    __syncthreads();

    if (jj == nsub - 1) {  // end of interval ci
      // the recompute of ci - 1 past what ran alongside (when this interval
      // is the shorter, ragged last one); buffer bufi is free now
      if (have_l1 && nsub < NS1) serial_chunks(ci, nsub, NS1, bufi);
      // C now holds dL/dH at the interval start: the checkpoint's gradient
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
      if (ci == 0) break;
      --ci;
      jj = 0;
      Lc = C;
      nsub = NS1;
    } else {
      ++jj;
    }
    bufi ^= 1;
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
  // dW: this warp's [V][V] sum -> shared memory (over the sub-checkpoints, no
  // longer read after the last barrier) -> CTA sum -> global
  {
    const uint32_t base = sb + L.subck + static_cast<uint32_t>(warp * V * V * 4);
#pragma unroll
    for (int ml = 0; ml < KS; ++ml)
#pragma unroll
      for (int nj = 0; nj < NT; ++nj)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int l = 16 * ml + g + 8 * (r >> 1), jc = 8 * nj + 2 * c + (r & 1);
          ptx::sts_f32(base + static_cast<uint32_t>((l * V + jc) * 4), dW[ml][nj][r]);
        }
  }
  __syncthreads();
  for (int e = tid; e < V * V; e += nthr) {
    float acc = 0.f;
    for (int w = 0; w < WPC; ++w)
      acc += ptx::lds_f32(sb + L.subck + static_cast<uint32_t>((w * V * V + e) * 4));
    if (n_ok) red_add(p.dW + static_cast<size_t>(n) * V * V + e, acc);
  }
  // each thread holds the u (.) v sum of column tid % V over the steps it flushed
  if (slice == 0 && n_ok) red_add(p.dw_r + static_cast<size_t>(n) * V + tid % V, dwr_acc);
  if (gated && dt >= 0 && dt < S2 && n_ok) {
    red_add(p.dalpha + n, dalpha_acc);
    red_add(p.dbeta + n, dbeta_acc);
  }
}

template <int V, bool F32, int WPC>
cudaError_t launch_pipe_t(const BwdParams& p, cudaStream_t stream) {
  const uint32_t smem = pipe_smem_total(V, p.C, sub_len<V, F32>(), WPC, F32 ? 4 : 2, p.gated);
  auto kern = p.gated ? bwd_pipe_kernel<V, F32, WPC, true> : bwd_pipe_kernel<V, F32, WPC, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.B) * p.N * p.nslices;
  kern<<<grid, 32 * WPC, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int V, bool F32, int WPC>
int pipe_ctas_per_sm_t(const BwdParams& p) {
  const uint32_t smem = pipe_smem_total(V, p.C, sub_len<V, F32>(), WPC, F32 ? 4 : 2, p.gated);
  auto kern = p.gated ? bwd_pipe_kernel<V, F32, WPC, true> : bwd_pipe_kernel<V, F32, WPC, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, 32 * WPC, smem) != cudaSuccess)
    return 0;
  return nb;
}

template <bool F32>
int pipe_ctas_per_sm_w(const BwdParams& p) {
  switch (p.WPC) {
    case 1: return pipe_ctas_per_sm_t<16, F32, 1>(p);
    case 2: return pipe_ctas_per_sm_t<16, F32, 2>(p);
    case 4: return pipe_ctas_per_sm_t<16, F32, 4>(p);
    case 8: return pipe_ctas_per_sm_t<16, F32, 8>(p);
  }
  return 0;
}

template <bool F32>
cudaError_t launch_pipe_w(const BwdParams& p, cudaStream_t stream) {
  switch (p.WPC) {
    case 1: return launch_pipe_t<16, F32, 1>(p, stream);
    case 2: return launch_pipe_t<16, F32, 2>(p, stream);
    case 4: return launch_pipe_t<16, F32, 4>(p, stream);
    case 8: return launch_pipe_t<16, F32, 8>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool bwd_has_pipe(int V) { return V == 16; }

size_t bwd_pipe_smem_bytes(int V, int C, int WPC, bool f32_inputs, bool gated) {
  return pipe_smem_total(V, C, bwd_sub_len(V, f32_inputs), WPC, f32_inputs ? 4 : 2, gated);
}

int bwd_pipe_ctas_per_sm(const BwdParams& p, int V, bool f32_inputs) {
  if (V != 16) return 0;
  return f32_inputs ? pipe_ctas_per_sm_w<true>(p) : pipe_ctas_per_sm_w<false>(p);
}

cudaError_t launch_bwd_pipe(const BwdParams& p, int V, bool f32_inputs, cudaStream_t stream) {
  if (V != 16 || p.S2 != bwd_sub_len(V, f32_inputs)) return cudaErrorInvalidValue;
  return f32_inputs ? launch_pipe_w<true>(p, stream) : launch_pipe_w<false>(p, stream);
}

}  // namespace m2rnn
