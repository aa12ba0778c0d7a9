// m2rnn_fwd.cu -- persistent-state forward kernel of the M2RNN recurrence.
//
// Computes, per (batch b, value head n), Eqs. (10)-(12) of "M2RNN: Non-Linear
// RNNs with Matrix-Valued States" (deck frame "Write, transform, retain, and
// read a matrix state"):
//     Z_t = tanh(H_{t-1} W + k_t v_t^T),  H_t = f_t H_{t-1} + (1-f_t) Z_t,
//     y_t = H_t^T q_t + w_r (.) v_t.
// The deck's frame "Efficient tiles do not remove the sequential dependency"
// keeps H and W on chip and scans time sequentially, parallel over batch and
// heads, with a (K,V) x (V,V) GEMM per step.  Here every row of H evolves on
// its own (W mixes value channels within a row; q only combines rows at
// readout), so rows are the unit of parallelism as well.
//
// CTA = one batch item b and G consecutive heads.  Warp roles:
//   warp 0   producer: bulk copies (cp.async.bulk, no multicast) of q, k, v
//            for TC-step chunks into an NSTAGE-deep shared-memory ring, and
//            f converted to fp32; completion on mbarriers.
//   warp 1   epilogue: sums the per-warp readout partials, adds w_r (.) v_t,
//            converts and stores y (coalesced rows of G*V elements).
//   warps 2+ consumers: WPH warps per head, each holding MT 16-row slices of
//            the fp32 state in registers for all T steps, in the accumulator
//            layout of mma.sync m16n8k16.  Per step and slice:
//              acc  = k v^T           (bf16 path: one MMA whose B operand has
//                                      v_t in row 0 and zeros elsewhere)
//              acc += bf16(H) * W     (mma.sync, W in registers)
//              H    = Z + f (H - Z),  Z = tanh(acc)   (SFU tanh, fp32)
//              A    = bf16(H)         (the next step's A operand)
//              ypart += q^T H         (MMA on movmatrix-transposed A)
// The fp32-input path keeps the same structure but splits H and W into
// bf16 hi + lo parts (three MMAs), forms k v^T in fp32, uses the accurate
// tanhf and an fp32 readout.
// Every mbarrier wait has a time limit; a wait that gives up records
// M2RNN_ERR_TIMEOUT in the device status word and the warp leaves its loop.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "m2rnn_internal.h"
#include "ptx.cuh"

namespace m2rnn {
namespace {

constexpr int TC = 32;                   // time steps per ring chunk
constexpr int NSTAGE = 3;                // depth of the input ring
constexpr int NYSTAGE = 2;               // depth of the readout-partial ring
constexpr int kMaxConsumerWarps = 16;    // per CTA
constexpr int kMaxThreads = 32 * (2 + kMaxConsumerWarps);
// Limit of the producer's final wait for its own bulk copies; independent of
// the caller's wait limit so that a tiny limit never lets a CTA exit while a
// copy into its shared memory is still in flight.
constexpr uint64_t kDrainLimitNs = 1000000000ull;

struct FwdLayout {
  uint32_t q, k, v, f, stage;  // offsets inside one ring stage, stage size
  uint32_t yp_base, yp_stage;  // readout partials [TC][G][WPH][V] fp32
  uint32_t wr;                 // w_r as fp32 [G][V]
  uint32_t bars;               // mbarriers
  uint32_t total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline FwdLayout fwd_layout(int K, int V, int G, int WPH, int es) {
  FwdLayout L;
  uint32_t o = 0;
  L.q = o;
  o = align_up(o + TC * K * es, 128);
  L.k = o;
  o = align_up(o + TC * K * es, 128);
  L.v = o;
  o = align_up(o + TC * G * V * es, 128);
  L.f = o;
  o = align_up(o + TC * G * 4, 128);
  L.stage = o;
  L.yp_base = NSTAGE * L.stage;
  L.yp_stage = align_up(TC * G * WPH * V * 4, 128);
  L.wr = L.yp_base + NYSTAGE * L.yp_stage;
  L.bars = align_up(L.wr + G * V * 4, 128);
  L.total = L.bars + 8 * (2 * NSTAGE + 2 * NYSTAGE);
  return L;
}

// mbarrier addresses
__device__ __forceinline__ uint32_t bar_in_full(uint32_t bars, int s) { return bars + 8 * s; }
__device__ __forceinline__ uint32_t bar_in_empty(uint32_t bars, int s) { return bars + 8 * (NSTAGE + s); }
__device__ __forceinline__ uint32_t bar_yp_full(uint32_t bars, int s) { return bars + 8 * (2 * NSTAGE + s); }
__device__ __forceinline__ uint32_t bar_yp_empty(uint32_t bars, int s) {
  return bars + 8 * (2 * NSTAGE + NYSTAGE + s);
}

template <bool F32>
struct InType;
template <>
struct InType<true> {
  using T = float;
};
template <>
struct InType<false> {
  using T = __nv_bfloat16;
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_as(float* d, float x) { *d = x; }
__device__ __forceinline__ void store_as(__nv_bfloat16* d, float x) { *d = __float2bfloat16_rn(x); }

__device__ __forceinline__ void record_timeout(int* status, int site) {
  if (atomicCAS(&status[0], 0, kStatusTimeout) == 0) atomicExch(&status[1], site);
}

// Every lane waits; the warp proceeds only if all lanes saw the phase
// complete (keeps control flow warp-uniform when a wait gives up).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const bool ok = ptx::mbar_wait(bar, parity, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
template <int V, bool F32>
__device__ void fwd_producer(const FwdParams& p, const FwdLayout& L, unsigned char* smem,
                             uint32_t sbase, int b, int n0, int Geff) {
  using TIn = typename InType<F32>::T;
  constexpr int es = sizeof(TIn);
  const int lane = threadIdx.x & 31;
  const int K = p.K, T = p.T, N = p.N, G = p.G;
  const uint32_t bars = sbase + L.bars;
  const int nchunks = (T + TC - 1) / TC;
  const TIn* q = static_cast<const TIn*>(p.q);
  const TIn* k = static_cast<const TIn*>(p.k);
  const TIn* v = static_cast<const TIn*>(p.v);
  const TIn* f = static_cast<const TIn*>(p.f);
  int armed = 0;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int s = ch % NSTAGE;
    if (!warp_wait(bar_in_empty(bars, s), ((ch / NSTAGE) & 1) ^ 1, p.wait_limit_ns)) {
      if (lane == 0) record_timeout(p.status, SITE_FWD_PRODUCER);
      break;
    }
    const int t0 = ch * TC;
    const int Tc = min(TC, T - t0);
    const uint32_t qk_bytes = static_cast<uint32_t>(Tc * K * es);
    const uint32_t v_bytes = static_cast<uint32_t>(Geff * V * es);
    const uint32_t full = bar_in_full(bars, s);
    if (lane == 0) ptx::mbar_expect_tx(full, 2 * qk_bytes + static_cast<uint32_t>(Tc) * v_bytes);
    __syncwarp();
    const uint32_t st = sbase + static_cast<uint32_t>(s) * L.stage;
    const size_t bt0 = static_cast<size_t>(b) * T + t0;
    if (lane == 0) {
      ptx::bulk_g2s(st + L.q, q + bt0 * K, qk_bytes, full);
      ptx::bulk_g2s(st + L.k, k + bt0 * K, qk_bytes, full);
    }
    for (int tl = lane; tl < Tc; tl += 32)
      ptx::bulk_g2s(st + L.v + static_cast<uint32_t>(tl * G * V * es),
                    v + ((bt0 + tl) * N + n0) * V, v_bytes, full);
    float* fs = reinterpret_cast<float*>(smem + static_cast<size_t>(s) * L.stage + L.f);
    for (int e = lane; e < Tc * Geff; e += 32) {
      const int tl = e / Geff, h = e - tl * Geff;
      fs[tl * G + h] = to_f(f[(bt0 + tl) * N + n0 + h]);
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(full);
    armed = ch + 1;
  }
  // Bulk copies complete on their own; before this warp (possibly the last
  // one alive after a time-out) leaves, wait until none is in flight.
  for (int ch = max(0, armed - NSTAGE); ch < armed; ++ch) {
    if (!warp_wait(bar_in_full(bars, ch % NSTAGE), (ch / NSTAGE) & 1, kDrainLimitNs)) {
      if (lane == 0) record_timeout(p.status, SITE_FWD_DRAIN);
      break;
    }
  }
}

// ---------------------------------------------------------------------------
// epilogue warp
// ---------------------------------------------------------------------------
template <int V, bool F32>
__device__ void fwd_epilogue(const FwdParams& p, const FwdLayout& L, unsigned char* smem,
                             uint32_t sbase, int b, int n0, int Geff) {
  using TIn = typename InType<F32>::T;
  const int lane = threadIdx.x & 31;
  const int T = p.T, N = p.N, G = p.G, WPH = p.WPH;
  const uint32_t bars = sbase + L.bars;
  const int nchunks = (T + TC - 1) / TC;
  float* wr_s = reinterpret_cast<float*>(smem + L.wr);
  const TIn* w_r = static_cast<const TIn*>(p.w_r) + static_cast<size_t>(n0) * V;
  const int GV = Geff * V;
  for (int e = lane; e < GV; e += 32) wr_s[e] = to_f(w_r[e]);
  __syncwarp();
  for (int ch = 0; ch < nchunks; ++ch) {
    const int s = ch % NSTAGE, ys = ch % NYSTAGE;
    if (!warp_wait(bar_in_full(bars, s), (ch / NSTAGE) & 1, p.wait_limit_ns) ||
        !warp_wait(bar_yp_full(bars, ys), (ch / NYSTAGE) & 1, p.wait_limit_ns)) {
      if (lane == 0) record_timeout(p.status, SITE_FWD_EPILOGUE);
      break;
    }
    const int t0 = ch * TC;
    const int Tc = min(TC, T - t0);
    const TIn* vs = reinterpret_cast<const TIn*>(smem + static_cast<size_t>(s) * L.stage + L.v);
    const float* yp = reinterpret_cast<const float*>(smem + L.yp_base + static_cast<size_t>(ys) * L.yp_stage);
    TIn* y = static_cast<TIn*>(p.y) + ((static_cast<size_t>(b) * T + t0) * N + n0) * V;
    for (int tl = 0; tl < Tc; ++tl) {
      for (int r = lane; r < GV; r += 32) {
        const int hl = r / V, j = r - hl * V;
        const float* pp = yp + ((tl * G + hl) * WPH) * V + j;
        float acc = 0.f;
        for (int w = 0; w < WPH; ++w) acc += pp[w * V];
        acc = fmaf(wr_s[r], to_f(vs[tl * G * V + r]), acc);
        store_as(y + static_cast<size_t>(tl) * N * V + r, acc);
      }
    }
    __syncwarp();
    if (lane == 0) {
      ptx::mbar_arrive(bar_in_empty(bars, s));
      ptx::mbar_arrive(bar_yp_empty(bars, ys));
    }
  }
}

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------

// Stores the thread's part of the state (rows row0 + 16*mt + g (+8), columns
// 8*nt + 2c (+1)) to a [K][V] fp32 array.
template <int V, int MT>
__device__ __forceinline__ void store_state(float* dst, const float (&H)[MT][V / 8][4], int row0,
                                            int g, int c) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < V / 8; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = row0 + 16 * mt + g + 8 * h;
        *reinterpret_cast<float2*>(dst + row * V + 8 * nt + 2 * c) =
            make_float2(H[mt][nt][2 * h], H[mt][nt][2 * h + 1]);
      }
}

// Accumulator layout of n-tiles (2ks, 2ks+1) -> A operand of k-step ks.
template <int V>
__device__ __forceinline__ void pack_a(const float (&H)[V / 8][4], uint32_t (&A)[V / 16][4]) {
#pragma unroll
  for (int ks = 0; ks < V / 16; ++ks) {
    A[ks][0] = ptx::pack_bf16x2(H[2 * ks][0], H[2 * ks][1]);
    A[ks][1] = ptx::pack_bf16x2(H[2 * ks][2], H[2 * ks][3]);
    A[ks][2] = ptx::pack_bf16x2(H[2 * ks + 1][0], H[2 * ks + 1][1]);
    A[ks][3] = ptx::pack_bf16x2(H[2 * ks + 1][2], H[2 * ks + 1][3]);
  }
}

// bf16 residual of the packing above: A_lo = bf16(H - float(A_hi)).
template <int V>
__device__ __forceinline__ void pack_a_lo(const float (&H)[V / 8][4], const uint32_t (&A)[V / 16][4],
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

template <int V, int MT, bool F32>
__device__ void fwd_consumer(const FwdParams& p, const FwdLayout& L, unsigned char* smem,
                             uint32_t sbase, int b, int n0, int ci) {
  using TIn = typename InType<F32>::T;
  constexpr int NT = V / 8, KS = V / 16;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int K = p.K, T = p.T, N = p.N, G = p.G, WPH = p.WPH;
  const int hl = ci / WPH, w = ci - hl * WPH;
  const int n = n0 + hl;
  const int row0 = w * 16 * MT;
  const uint32_t bars = sbase + L.bars;

  // W as B operands (k = row l of W, n = column j), bf16 hi (+ lo residual).
  const TIn* Wn = static_cast<const TIn*>(p.W) + static_cast<size_t>(n) * V * V;
  uint32_t Bw[KS][NT][2];
  uint32_t Bwl[KS][NT][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r0 = 16 * ks + 8 * h + 2 * c, col = 8 * nt + g;
        const float w0 = to_f(Wn[r0 * V + col]), w1 = to_f(Wn[(r0 + 1) * V + col]);
        Bw[ks][nt][h] = ptx::pack_bf16x2(w0, w1);
        Bwl[ks][nt][h] = F32 ? ptx::pack_bf16x2(w0 - ptx::bf16x2_lo(Bw[ks][nt][h]),
                                                w1 - ptx::bf16x2_hi(Bw[ks][nt][h]))
                             : 0u;
      }

  // State in registers, fp32.
  float H[MT][NT][4];
  const size_t hoff = (static_cast<size_t>(b) * N + n) * K * V;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = row0 + 16 * mt + g + 8 * (r >> 1), col = 8 * nt + 2 * c + (r & 1);
        H[mt][nt][r] = p.H0 ? p.H0[hoff + row * V + col] : 0.f;
      }
  uint32_t A[MT][KS][4];
  uint32_t Al[MT][KS][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    pack_a<V>(H[mt], A[mt]);
    if (F32) pack_a_lo<V>(H[mt], A[mt], Al[mt]);
  }

  const int nchunks = (T + TC - 1) / TC;
  bool ok = true;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int s = ch % NSTAGE, ys = ch % NYSTAGE;
    if (!warp_wait(bar_in_full(bars, s), (ch / NSTAGE) & 1, p.wait_limit_ns) ||
        !warp_wait(bar_yp_empty(bars, ys), ((ch / NYSTAGE) & 1) ^ 1, p.wait_limit_ns)) {
      ok = false;
      break;
    }
    const int t0 = ch * TC;
    const int Tc = min(TC, T - t0);
    const unsigned char* st = smem + static_cast<size_t>(s) * L.stage;
    const TIn* qs = reinterpret_cast<const TIn*>(st + L.q);
    const TIn* kst = reinterpret_cast<const TIn*>(st + L.k);
    const TIn* vs = reinterpret_cast<const TIn*>(st + L.v);
    const float* fs = reinterpret_cast<const float*>(st + L.f);
    float* yp = reinterpret_cast<float*>(smem + L.yp_base + static_cast<size_t>(ys) * L.yp_stage);
#pragma unroll 1
    for (int tl = 0; tl < Tc; ++tl) {
      const int t = t0 + tl;
      if (p.ckpt != nullptr && t % p.C == 0)
        store_state<V, MT>(p.ckpt + ((static_cast<size_t>(b) * N + n) * p.nck + t / p.C) * K * V, H,
                           row0, g, c);
      const float fg = fs[tl * G + hl];
      const TIn* vrow = vs + (tl * G + hl) * V;
      const TIn* krow = kst + tl * K + row0;
      const TIn* qrow = qs + tl * K + row0;
      float ya[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) ya[nt][0] = ya[nt][1] = ya[nt][2] = ya[nt][3] = 0.f;
      // B operand of the rank-1 write: v_t in row 0, zeros elsewhere.
      uint32_t Bv[NT];
      float vv[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (F32) {
          vv[nt][0] = to_f(vrow[8 * nt + 2 * c]);
          vv[nt][1] = to_f(vrow[8 * nt + 2 * c + 1]);
          Bv[nt] = 0u;
        } else {
          const uint32_t raw = reinterpret_cast<const uint16_t*>(vrow)[8 * nt + g];
          Bv[nt] = (c == 0) ? raw : 0u;
          vv[nt][0] = vv[nt][1] = 0.f;
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        float acc[NT][4];
        if (F32) {
          const float k0 = to_f(krow[16 * mt + g]), k1 = to_f(krow[16 * mt + 8 + g]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            acc[nt][0] = k0 * vv[nt][0];
            acc[nt][1] = k0 * vv[nt][1];
            acc[nt][2] = k1 * vv[nt][0];
            acc[nt][3] = k1 * vv[nt][1];
          }
        } else {
          // A operand with k_i in every column of row i: A * Bv = k v^T.
          const uint32_t k0 = reinterpret_cast<const uint16_t*>(krow)[16 * mt + g];
          const uint32_t k1 = reinterpret_cast<const uint16_t*>(krow)[16 * mt + 8 + g];
          const uint32_t Ak[4] = {k0 | (k0 << 16), k1 | (k1 << 16), k0 | (k0 << 16), k1 | (k1 << 16)};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            ptx::mma_bf16_16816(acc[nt], Ak, Bv[nt], 0u);
          }
        }
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            ptx::mma_bf16_16816(acc[nt], A[mt][ks], Bw[ks][nt][0], Bw[ks][nt][1]);
            if (F32) {
              ptx::mma_bf16_16816(acc[nt], A[mt][ks], Bwl[ks][nt][0], Bwl[ks][nt][1]);
              ptx::mma_bf16_16816(acc[nt], Al[mt][ks], Bw[ks][nt][0], Bw[ks][nt][1]);
            }
          }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float z = F32 ? tanhf(acc[nt][r]) : ptx::tanh_approx(acc[nt][r]);
            H[mt][nt][r] = fmaf(fg, H[mt][nt][r] - z, z);
          }
        pack_a<V>(H[mt], A[mt]);
        if (F32) {
          pack_a_lo<V>(H[mt], A[mt], Al[mt]);
          const float q0 = to_f(qrow[16 * mt + g]), q1 = to_f(qrow[16 * mt + 8 + g]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            ya[nt][0] = fmaf(q0, H[mt][nt][0], fmaf(q1, H[mt][nt][2], ya[nt][0]));
            ya[nt][1] = fmaf(q0, H[mt][nt][1], fmaf(q1, H[mt][nt][3], ya[nt][1]));
          }
        } else {
          // Readout y^T += q^T H on the tensor core: A = q in every row,
          // B = this slice of bf16(H_t) transposed 8x8-blockwise.
          const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow);
          const uint32_t qa0 = q32[8 * mt + c], qa1 = q32[8 * mt + 4 + c];
          const uint32_t Aq[4] = {qa0, qa0, qa1, qa1};
#pragma unroll
          for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
              ptx::mma_bf16_16816(ya[2 * ks + h2], Aq, ptx::movmatrix_trans(A[mt][ks][2 * h2]),
                                  ptx::movmatrix_trans(A[mt][ks][2 * h2 + 1]));
        }
      }
      if (F32) {
        // Sum the fp32 partials over the 8 lanes of each column group.
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float x = ya[nt][e];
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            ya[nt][e] = x;
          }
      }
      if (g == 0) {
        float* dst = yp + ((tl * G + hl) * WPH + w) * V;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          *reinterpret_cast<float2*>(dst + 8 * nt + 2 * c) = make_float2(ya[nt][0], ya[nt][1]);
      }
    }
    __syncwarp();
    if (lane == 0) {
      ptx::mbar_arrive(bar_in_empty(bars, s));
      ptx::mbar_arrive(bar_yp_full(bars, ys));
    }
  }
  if (!ok) {
    if (lane == 0) record_timeout(p.status, SITE_FWD_CONSUMER);
    return;
  }
  if (p.HT != nullptr) store_state<V, MT>(p.HT + hoff, H, row0, g, c);
}

template <int V, int MT, bool F32>
__global__ void __launch_bounds__(kMaxThreads, 1) fwd_kernel(const FwdParams p) {
  using TIn = typename InType<F32>::T;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.x / p.ngroups;
  const int n0 = (blockIdx.x % p.ngroups) * p.G;
  const int Geff = min(p.G, p.N - n0);
  const int ncons = Geff * p.WPH;
  const FwdLayout L = fwd_layout(p.K, V, p.G, p.WPH, sizeof(TIn));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bars = sbase + L.bars;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(bar_in_full(bars, s), 1);
      ptx::mbar_init(bar_in_empty(bars, s), ncons + 1);
    }
    for (int s = 0; s < NYSTAGE; ++s) {
      ptx::mbar_init(bar_yp_full(bars, s), ncons);
      ptx::mbar_init(bar_yp_empty(bars, s), 1);
    }
    ptx::mbar_init_fence();
  }
  __syncthreads();
  if (warp == 0)
    fwd_producer<V, F32>(p, L, smem, sbase, b, n0, Geff);
  else if (warp == 1)
    fwd_epilogue<V, F32>(p, L, smem, sbase, b, n0, Geff);
  else if (warp - 2 < ncons)
    fwd_consumer<V, MT, F32>(p, L, smem, sbase, b, n0, warp - 2);
}

template <int V, int MT, bool F32>
cudaError_t launch_t(const FwdParams& p, cudaStream_t stream) {
  const FwdLayout L = fwd_layout(p.K, V, p.G, p.WPH, F32 ? 4 : 2);
  auto kern = fwd_kernel<V, MT, F32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(L.total));
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.B) * static_cast<unsigned>(p.ngroups);
  kern<<<grid, 32 * (2 + p.G * p.WPH), L.total, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int K, int V, int G, int WPH, bool f32_inputs) {
  return fwd_layout(K, V, G, WPH, f32_inputs ? 4 : 2).total;
}

int fwd_max_consumer_warps() { return kMaxConsumerWarps; }

cudaError_t launch_fwd(const FwdParams& p, int V, bool f32_inputs, int MT, cudaStream_t stream) {
  if (f32_inputs) {
    if (MT != 1) return cudaErrorInvalidValue;
    if (V == 16) return launch_t<16, 1, true>(p, stream);
    if (V == 32) return launch_t<32, 1, true>(p, stream);
    return cudaErrorInvalidValue;
  }
  if (V == 16) {
    if (MT == 1) return launch_t<16, 1, false>(p, stream);
    if (MT == 2) return launch_t<16, 2, false>(p, stream);
    if (MT == 4) return launch_t<16, 4, false>(p, stream);
  } else if (V == 32) {
    if (MT == 1) return launch_t<32, 1, false>(p, stream);
    if (MT == 2) return launch_t<32, 2, false>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace m2rnn
