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
//            for TC-step chunks into an NSTAGE-deep shared-memory ring; once
//            a chunk has landed it writes k as duplicated fp32 pairs (k_i,
//            k_i) and f as (f, f), the operand form of the packed fp32
//            multiplies below, then releases the chunk to the consumers.
//   warps 1 .. NEPI  epilogue (three warps in the dense 8-head CTAs, one
//            elsewhere): sums the per-warp readout partials, adds
//            w_r (.) v_t, converts and stores y (16-byte vector stores).
//            The producer's and epilogue's waits sleep between tries instead
//            of polling: these warps share SMSPs with consumer warps.
//   then     consumers: WPH warps per head, each holding MT 16-row slices of
//            the fp32 state in registers for all T steps, in the accumulator
//            layout of mma.sync m16n8k16.  Per step and slice:
//              acc  = k v^T           (packed fp32 multiplies, exact for
//                                      bf16 inputs)
//              acc += bf16(H) * W     (mma.sync, W in registers)
//              H    = Z + f (H - Z),  Z = tanh(acc)   (SFU tanh; fma.f32x2)
//              A    = bf16(H)         (the next step's A operand)
//              ypart = q^T H          (MMA on movmatrix-transposed A)
//            The rank-1 inputs of step t+1 are read while step t computes.
// MT = 0 selects half slices for latency-bound problems: each warp owns 8
// rows (rows 8..15 of its m16 tile are zero padding), which halves the tanh
// and elementwise work on each warp's serial chain and doubles the warps
// working on a head.
// The fp32-input path keeps the same structure but splits H and W into
// bf16 hi + lo parts (three MMAs), uses the accurate tanhf and an fp32
// readout.
// Every mbarrier wait has a time limit; a wait that gives up records
// M2RNN_ERR_TIMEOUT in the device status word and the warp leaves its loop.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "m2rnn_internal.h"
#include "ptx.cuh"
#include "m2rnn_gate.cuh"
#include "m2rnn_check.cuh"

namespace m2rnn {
namespace {

constexpr int NSTAGE = 3;   // depth of the input ring
constexpr int NYSTAGE = 2;  // depth of the readout-partial ring
// Limit of the producer's final wait for its own bulk copies; independent of
// the caller's wait limit so that a tiny limit never lets a CTA exit while a
// copy into its shared memory is still in flight.
constexpr uint64_t kDrainLimitNs = 1000000000ull;

// Consumer warps per CTA: 16 where an 18-warp CTA's register budget (96 per
// thread) holds the variant without spills, 8 otherwise.
template <int V, int MT, bool F32>
constexpr int max_consumer_warps() {
  return (V == 16 && MT <= 2 && !F32) || (V == 16 && MT == 1) ? 16 : 8;
}

// The rank-1 term k v^T from fp32 (k, k) pairs the producer writes and a
// packed fp32 multiply, or (false) from an MMA of two one-column bf16
// operands.  Pairs for fp32 inputs; for V = 32, where the tensor-core form's
// prefetched products need 32 more registers per thread; and for the dense
// 8-head full-wave launch (GC = 8), where the extra MMAs contend for the
// tensor pipe (measured 1.496 ms against 1.569 ms for one full wave, while
// the sparser launches gain from the MMA form).
template <int V, bool F32, int GC = 0>
__host__ __device__ constexpr bool rank1_pairs() {
  return F32 || V != 16 || GC >= 8;
}

struct FwdLayout {
  uint32_t q, k, v;    // raw bulk-copied inputs (input dtype)
  uint32_t kd, fd;     // k as fp32 pairs [TC][K][2], f as fp32 pairs [TC][G][2]
  uint32_t stage;      // bytes per ring stage
  uint32_t yp_base, yp_stage;  // readout partials [TC][G][WPH][V] fp32
  uint32_t wr;         // w_r as fp32 [G][V]
  uint32_t bars;       // mbarriers
  uint32_t total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// TC: time steps per ring chunk (<= 64).
// pairs: k also as fp32 (k, k) pairs (rank1_pairs).
__host__ __device__ inline FwdLayout fwd_layout(int K, int V, int G, int WPH, int es, int TC,
                                                bool pairs = true) {
  FwdLayout L;
  uint32_t o = 0;
  L.q = o;
  o = align_up(o + TC * K * es, 128);
  L.k = o;
  o = align_up(o + TC * K * es, 128);
  L.v = o;
  o = align_up(o + TC * G * V * es, 128);
  L.kd = o;  // fp32 pairs of k (otherwise the consumers read k as copied)
  o = align_up(o + (pairs ? TC * K * 8 : 0), 128);
  L.fd = o;
  o = align_up(o + TC * G * 8, 128);
  L.stage = o;
  L.yp_base = NSTAGE * L.stage;
  L.yp_stage = align_up(TC * G * WPH * V * 4, 128);
  L.wr = L.yp_base + NYSTAGE * L.yp_stage;
  L.bars = align_up(L.wr + G * V * 4, 128);
  L.total = L.bars + 8 * (3 * NSTAGE + 2 * NYSTAGE);
  return L;
}

// mbarrier addresses
__device__ __forceinline__ uint32_t bar_raw_full(uint32_t bars, int s) { return bars + 8 * s; }
__device__ __forceinline__ uint32_t bar_in_full(uint32_t bars, int s) { return bars + 8 * (NSTAGE + s); }
__device__ __forceinline__ uint32_t bar_in_empty(uint32_t bars, int s) {
  return bars + 8 * (2 * NSTAGE + s);
}
__device__ __forceinline__ uint32_t bar_yp_full(uint32_t bars, int s) { return bars + 8 * (3 * NSTAGE + s); }
__device__ __forceinline__ uint32_t bar_yp_empty(uint32_t bars, int s) {
  return bars + 8 * (3 * NSTAGE + NYSTAGE + s);
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

__device__ __forceinline__ void record_timeout(int* status, int site) {
  if (atomicCAS(&status[0], 0, kStatusTimeout) == 0) atomicExch(&status[1], site);
}

// Every lane waits; the warp proceeds only if all lanes saw the phase
// complete (keeps control flow warp-uniform when a wait gives up).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const bool ok = ptx::mbar_wait(bar, parity, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// The same for the producer's and epilogue's waits: those warps share SMSPs
// with consumer warps and mostly wait, so a waiting lane sleeps between its
// tries rather than taking issue slots to poll.  The rings give these warps
// at least a chunk of slack, several microseconds, against the sleep.
constexpr uint32_t kHelperSleepNs = 256;
__device__ __forceinline__ bool warp_wait_idle(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const bool ok = ptx::mbar_wait_sleep(bar, parity, limit_ns, kHelperSleepNs);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
template <int V, bool F32, bool GATED, bool PAIRS>
__device__ __forceinline__ void fwd_producer(const FwdParams& p, const FwdLayout& L, uint32_t sbase,
                                             int b, int n0, int Geff) {
  using TIn = typename InType<F32>::T;
  constexpr int es = sizeof(TIn);
  const int lane = threadIdx.x & 31;
  const int K = p.K, T = p.T, N = p.N, G = p.G;
  const uint32_t bars = sbase + L.bars;
  const int TC = p.tc;
  const int nchunks = (T + TC - 1) / TC;
  const TIn* q = static_cast<const TIn*>(p.q);
  const TIn* k = static_cast<const TIn*>(p.k);
  const TIn* v = static_cast<const TIn*>(p.v);
  // f, or (GATED) the input gate's a, with alpha and beta per head
  const TIn* f = static_cast<const TIn*>(GATED ? p.a : p.f);
  const TIn* galpha = static_cast<const TIn*>(p.alpha);
  const TIn* gbeta = static_cast<const TIn*>(p.beta);
  // query/key group of this CTA's heads (the host keeps a CTA inside one group)
  const int Nq = p.Nq, gq = n0 / (N / Nq);
  // array extents in elements (index checks of the checked build)
  const size_t qk_ext = static_cast<size_t>(p.B) * T * Nq * K;
  const size_t v_ext = static_cast<size_t>(p.B) * T * N * V, f_ext = static_cast<size_t>(p.B) * T * N;

  // bf16 f (or a) of Geff in {1, 2, 4, 8} heads is read with one vector load
  // per step (aligned: n0 and N are multiples of Geff); the gate's alpha and
  // beta of those heads are read once.
  const bool fvec = !F32 && (Geff == 1 || Geff == 2 || Geff == 4 || Geff == 8) && N % Geff == 0;
  float ga[8], gb[8];
  bool gok[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    gok[h] = GATED && h < Geff && in_range(p.status, n0 + h, 1, N, CHK_FWD_PARAM);
    ga[h] = gok[h] ? to_f(galpha[n0 + h]) : 0.f;
    gb[h] = gok[h] ? to_f(gbeta[n0 + h]) : 0.f;
  }

  // Waits for a free stage, starts the bulk copies of chunk ch and writes
  // its f (or, gated, f computed from a) as fp32 pairs.
  auto issue = [&](int ch) -> bool {
    const int s = ch % NSTAGE;
    if (!warp_wait_idle(bar_in_empty(bars, s), ((ch / NSTAGE) & 1) ^ 1, p.wait_limit_ns)) return false;
    const int t0 = ch * TC;
    const int Tc = min(TC, T - t0);
    const uint32_t qk_bytes = static_cast<uint32_t>(Tc * K * es);
    const uint32_t v_bytes = static_cast<uint32_t>(Geff * V * es);
    const uint32_t raw = bar_raw_full(bars, s);
    if (lane == 0) ptx::mbar_expect_tx(raw, 2 * qk_bytes + static_cast<uint32_t>(Tc) * v_bytes);
    __syncwarp();
    const uint32_t st = sbase + static_cast<uint32_t>(s) * L.stage;
    const size_t bt0 = static_cast<size_t>(b) * T + t0;
    // (a copy the checked build skips still counts its bytes as arrived)
    if (Nq == 1) {  // the chunk's q and k rows are contiguous
      if (lane == 0) {
        if (in_range(p.status, bt0 * K, static_cast<size_t>(Tc) * K, qk_ext, CHK_FWD_QK)) {
          ptx::bulk_g2s(st + L.q, q + bt0 * K, qk_bytes, raw);
          ptx::bulk_g2s(st + L.k, k + bt0 * K, qk_bytes, raw);
        } else {
          ptx::mbar_complete_tx(raw, 2 * qk_bytes);
        }
      }
    } else {  // one row per step: [t][Nq][K], group gq
      const uint32_t row_bytes = static_cast<uint32_t>(K * es);
      for (int tl = lane; tl < Tc; tl += 32) {
        const size_t src = ((bt0 + tl) * Nq + gq) * K;
        if (in_range(p.status, src, K, qk_ext, CHK_FWD_QK)) {
          ptx::bulk_g2s(st + L.q + tl * row_bytes, q + src, row_bytes, raw);
          ptx::bulk_g2s(st + L.k + tl * row_bytes, k + src, row_bytes, raw);
        } else {
          ptx::mbar_complete_tx(raw, 2 * row_bytes);
        }
      }
    }
    for (int tl = lane; tl < Tc; tl += 32) {
      const size_t src = ((bt0 + tl) * N + n0) * V;
      if (in_range(p.status, src, static_cast<size_t>(Geff) * V, v_ext, CHK_FWD_V))
        ptx::bulk_g2s(st + L.v + static_cast<uint32_t>(tl * G * V * es), v + src, v_bytes, raw);
      else
        ptx::mbar_complete_tx(raw, v_bytes);
    }
    // f[b, t0:t0+Tc, n0:n0+Geff] -> fp32 pairs [TC][G][2].
    if (fvec) {  // a step per lane: one 2-, 4-, 8- or 16-byte load of its Geff values
      for (int tl = lane; tl < Tc; tl += 32) {
        const size_t fi = (bt0 + tl) * N + n0;
        uint32_t fw[4] = {0u, 0u, 0u, 0u};
        if (in_range(p.status, fi, Geff, f_ext, CHK_FWD_F)) {
          const void* src = f + fi;
          if (Geff == 8) {
            const uint4 u = *static_cast<const uint4*>(src);
            fw[0] = u.x; fw[1] = u.y; fw[2] = u.z; fw[3] = u.w;
          } else if (Geff == 4) {
            const uint2 u = *static_cast<const uint2*>(src);
            fw[0] = u.x; fw[1] = u.y;
          } else if (Geff == 2) {
            fw[0] = *static_cast<const uint32_t*>(src);
          } else {
            fw[0] = *static_cast<const uint16_t*>(src);
          }
        }
        const uint32_t dst = st + L.fd + static_cast<uint32_t>(tl * G * 8);
#pragma unroll
        for (int h = 0; h < 8; h += 2) {
          if (h >= Geff) break;
          float a = ptx::bf16x2_lo(fw[h / 2]), a1 = ptx::bf16x2_hi(fw[h / 2]);
          if constexpr (GATED) {
            a = gok[h] ? gate_f(a, ga[h], gb[h]) : 0.f;
            a1 = gok[h + 1] ? gate_f(a1, ga[h + 1], gb[h + 1]) : 0.f;
          }
          if (h + 1 < Geff)
            ptx::sts_f32x4(dst + 8 * h, a, a, a1, a1);
          else
            ptx::sts_f32x2(dst + 8 * h, a, a);
        }
      }
    }
    const int nf = fvec ? 0 : Tc * Geff;  // otherwise element by element, loads batched
    for (int base = 0; base < nf; base += 256) {
      float fv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = base + lane + 32 * i;
        const int tl = e / Geff, h = e - tl * Geff;
        const size_t fi = (bt0 + tl) * N + n0 + h;
        const bool use = e < nf && in_range(p.status, fi, 1, f_ext, CHK_FWD_F);
        if constexpr (GATED)
          fv[i] = use && in_range(p.status, n0 + h, 1, N, CHK_FWD_PARAM)
                      ? gate_f(to_f(f[fi]), to_f(galpha[n0 + h]), to_f(gbeta[n0 + h]))
                      : 0.f;
        else
          fv[i] = use ? to_f(f[fi]) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = base + lane + 32 * i;
        const int tl = e / Geff, h = e - tl * Geff;
        if (e < nf) ptx::sts_f32x2(st + L.fd + static_cast<uint32_t>((tl * G + h) * 8), fv[i], fv[i]);
      }
    }
    // The copies' bytes were announced above; this arrival is the barrier's
    // single expected one, so its phase completes once all bytes have landed.
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(raw);
    return true;
  };

  // Waits for chunk ch's copies, writes k as fp32 pairs, releases the chunk.
  auto convert = [&](int ch) -> bool {
    const int s = ch % NSTAGE;
    if (!warp_wait(bar_raw_full(bars, s), (ch / NSTAGE) & 1, p.wait_limit_ns)) return false;
    const int Tc = min(TC, T - ch * TC);
    const uint32_t st = sbase + static_cast<uint32_t>(s) * L.stage;
    const int n8 = PAIRS ? Tc * K / 8 : 0;  // else k is used as copied
    for (int i = lane; i < n8; i += 32) {
      float x[8];
      if (F32) {
        const float4 a = ptx::lds_f32x4(st + L.k + 32 * i), c = ptx::lds_f32x4(st + L.k + 32 * i + 16);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
      } else {
        const uint4 u = ptx::lds_u32x4(st + L.k + 16 * i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x[2 * j] = ptx::bf16x2_lo(w[j]);
          x[2 * j + 1] = ptx::bf16x2_hi(w[j]);
        }
      }
      const uint32_t d = st + L.kd + 64 * i;
#pragma unroll
      for (int j = 0; j < 4; ++j) ptx::sts_f32x4(d + 16 * j, x[2 * j], x[2 * j], x[2 * j + 1], x[2 * j + 1]);
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar_in_full(bars, s));
    return true;
  };

  int issued = 0, converted = 0;
  bool ok = true;
  for (int ch = 0; ch < nchunks; ++ch) {
    if (!(ok = issue(ch))) break;
    issued = ch + 1;
    if (ch >= 1) {
      if (!(ok = convert(ch - 1))) break;
      converted = ch;
    }
  }
  if (ok && nchunks > 0) {
    if ((ok = convert(nchunks - 1))) converted = nchunks;
  }
  if (!ok && lane == 0) record_timeout(p.status, SITE_FWD_PRODUCER);
  // Bulk copies complete on their own; before this warp (possibly the last
  // one alive after a time-out) leaves, wait until none is in flight.
  for (int ch = max(converted, issued - NSTAGE); ch < issued; ++ch) {
    if (!warp_wait(bar_raw_full(bars, ch % NSTAGE), (ch / NSTAGE) & 1, kDrainLimitNs)) {
      if (lane == 0) record_timeout(p.status, SITE_FWD_DRAIN);
      break;
    }
  }
}

// ---------------------------------------------------------------------------
// epilogue warp
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store8(float* y, const float (&o)[8]) {
  float4* d = reinterpret_cast<float4*>(y);
  d[0] = make_float4(o[0], o[1], o[2], o[3]);
  d[1] = make_float4(o[4], o[5], o[6], o[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* y, const float (&o)[8]) {
  uint4 u;
  u.x = ptx::pack_bf16x2(o[0], o[1]);
  u.y = ptx::pack_bf16x2(o[2], o[3]);
  u.z = ptx::pack_bf16x2(o[4], o[5]);
  u.w = ptx::pack_bf16x2(o[6], o[7]);
  *reinterpret_cast<uint4*>(y) = u;
}
// Eight consecutive input-dtype values from shared memory, as floats.
template <bool F32>
__device__ __forceinline__ void load8(uint32_t addr, float (&o)[8]) {
  if (F32) {
    const float4 a = ptx::lds_f32x4(addr), c = ptx::lds_f32x4(addr + 16);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = c.x; o[5] = c.y; o[6] = c.z; o[7] = c.w;
  } else {
    const uint4 u = ptx::lds_u32x4(addr);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = ptx::bf16x2_lo(w[i]);
      o[2 * i + 1] = ptx::bf16x2_hi(w[i]);
    }
  }
}

// 8 consecutive input-dtype values from global memory (16-byte aligned).
template <bool F32>
__device__ __forceinline__ void ldg8(const void* src, float (&o)[8]) {
  if (F32) {
    const float4 a = __ldg(static_cast<const float4*>(src)), c = __ldg(static_cast<const float4*>(src) + 1);
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

// Sums the per-warp readout partials, adds w_r (.) v and stores y.  NORM
// (the readout epilogue): also adds this CTA's share of sum (y (.) g)^2 of
// every token into p.ssq[b, t] (the normalisation kernel finishes the norm).
//
// The epilogue runs on NEPI warps (e = 0 .. NEPI-1) that split each chunk's
// outputs between them, so that no SMSP carries all of it next to its
// consumer warps.
template <int V, bool F32, bool NORM, int NEPI>
__device__ __forceinline__ void fwd_epilogue(const FwdParams& p, const FwdLayout& L, uint32_t sbase,
                                             int b, int n0, int Geff, int e) {
  using TIn = typename InType<F32>::T;
  constexpr int es = sizeof(TIn);
  constexpr int LANES = 32 * NEPI;
  const int lane = threadIdx.x & 31, id = 32 * e + lane;
  const int T = p.T, N = p.N, G = p.G, WPH = p.WPH;
  const uint32_t bars = sbase + L.bars;
  const int TC = p.tc;
  const int nchunks = (T + TC - 1) / TC;
  const TIn* w_r = static_cast<const TIn*>(p.w_r) + static_cast<size_t>(n0) * V;
  const int GV = Geff * V;
  const size_t y_ext = static_cast<size_t>(p.B) * T * N * V;  // y and g (index checks)
  // (each epilogue warp writes the same w_r values; it reads only its own)
  for (int i = lane; i < GV; i += 32)
    if (in_range(p.status, static_cast<size_t>(n0) * V + i, 1, static_cast<size_t>(N) * V, CHK_FWD_PARAM))
      ptx::sts_f32(sbase + L.wr + 4 * i, to_f(w_r[i]));
  __syncwarp();
  const int R8 = GV / 8;  // 8-element groups per time step
  // Where R8 divides the epilogue's lanes, every lane keeps one group (heads
  // hl, columns j..j+7) and walks the steps id / R8, + LANES / R8, ...; its
  // w_r stays in registers.
  const bool fixed = R8 > 0 && R8 <= LANES && LANES % R8 == 0;
  const int gi = fixed ? id % R8 : 0;
  const int fr = gi * 8, fhl = fr / V, fj = fr - fhl * V;
  float2 wrf[4];
  {
    const float4 w0 = ptx::lds_f32x4(sbase + L.wr + 4 * fr);
    const float4 w1 = ptx::lds_f32x4(sbase + L.wr + 4 * fr + 16);
    wrf[0] = make_float2(w0.x, w0.y); wrf[1] = make_float2(w0.z, w0.w);
    wrf[2] = make_float2(w1.x, w1.y); wrf[3] = make_float2(w1.z, w1.w);
  }
  for (int ch = 0; ch < nchunks; ++ch) {
    const int s = ch % NSTAGE, ys = ch % NYSTAGE;
    if (!warp_wait_idle(bar_in_full(bars, s), (ch / NSTAGE) & 1, p.wait_limit_ns) ||
        !warp_wait_idle(bar_yp_full(bars, ys), (ch / NYSTAGE) & 1, p.wait_limit_ns)) {
      if (lane == 0) record_timeout(p.status, SITE_FWD_EPILOGUE);
      break;
    }
    const int t0 = ch * TC;
    const int Tc = min(TC, T - t0);
    const uint32_t vs = sbase + static_cast<uint32_t>(s) * L.stage + L.v;
    const uint32_t yp = sbase + L.yp_base + static_cast<uint32_t>(ys) * L.yp_stage;
    TIn* y = static_cast<TIn*>(p.y) + ((static_cast<size_t>(b) * T + t0) * N + n0) * V;
    const int nidx = p.y != nullptr ? Tc * R8 : 0;  // no y in checkpoint-only runs
    if (fixed && nidx > 0) {
      const int tstep = LANES / R8;
#pragma unroll 1
      for (int tl = id / R8; tl < Tc; tl += tstep) {
        const uint32_t pa = yp + static_cast<uint32_t>((((tl * G + fhl) * WPH) * V + fj) * 4);
        float2 o[4];
        {
          const float4 a = ptx::lds_f32x4(pa), c = ptx::lds_f32x4(pa + 16);
          o[0] = make_float2(a.x, a.y); o[1] = make_float2(a.z, a.w);
          o[2] = make_float2(c.x, c.y); o[3] = make_float2(c.z, c.w);
        }
        for (int w = 1; w < WPH; ++w) {  // the warps' partials, in order
          const float4 a = ptx::lds_f32x4(pa + w * V * 4), c = ptx::lds_f32x4(pa + w * V * 4 + 16);
          o[0] = __fadd2_rn(o[0], make_float2(a.x, a.y));
          o[1] = __fadd2_rn(o[1], make_float2(a.z, a.w));
          o[2] = __fadd2_rn(o[2], make_float2(c.x, c.y));
          o[3] = __fadd2_rn(o[3], make_float2(c.z, c.w));
        }
        float vv[8];
        load8<F32>(vs + static_cast<uint32_t>((tl * G * V + fr) * es), vv);
        float oo[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 r2 = __ffma2_rn(wrf[i], make_float2(vv[2 * i], vv[2 * i + 1]), o[i]);
          oo[2 * i] = r2.x;
          oo[2 * i + 1] = r2.y;
        }
        const size_t yo = ((static_cast<size_t>(b) * T + t0 + tl) * N + n0) * V + fr;
        if (in_range(p.status, yo, 8, y_ext, CHK_FWD_Y)) store8(y + static_cast<size_t>(tl) * N * V + fr, oo);
        if constexpr (NORM) {
          float gg[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (in_range(p.status, yo, 8, y_ext, CHK_FWD_G)) ldg8<F32>(static_cast<const TIn*>(p.g) + yo, gg);
          float part = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float og = oo[i] * gg[i];
            part = fmaf(og, og, part);
          }
          const size_t so = static_cast<size_t>(b) * T + t0 + tl;
          if (in_range(p.status, so, 1, static_cast<size_t>(p.B) * T, CHK_FWD_SSQ)) atomicAdd(p.ssq + so, part);
        }
      }
    }
    for (int idx = fixed ? nidx : id; idx < nidx; idx += LANES) {
      const int tl = idx / R8;
      const int r = (idx - tl * R8) * 8;
      const int hl = r / V, j = r - hl * V;
      float o[8], vv[8];
      const uint32_t pa = yp + static_cast<uint32_t>((((tl * G + hl) * WPH) * V + j) * 4);
      {
        const float4 a = ptx::lds_f32x4(pa), c = ptx::lds_f32x4(pa + 16);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = c.x; o[5] = c.y; o[6] = c.z; o[7] = c.w;
      }
      for (int w = 1; w < WPH; ++w) {
        const float4 a = ptx::lds_f32x4(pa + w * V * 4), c = ptx::lds_f32x4(pa + w * V * 4 + 16);
        o[0] += a.x; o[1] += a.y; o[2] += a.z; o[3] += a.w;
        o[4] += c.x; o[5] += c.y; o[6] += c.z; o[7] += c.w;
      }
      load8<F32>(vs + static_cast<uint32_t>((tl * G * V + r) * es), vv);
      const float4 w0 = ptx::lds_f32x4(sbase + L.wr + 4 * r);
      const float4 w1 = ptx::lds_f32x4(sbase + L.wr + 4 * r + 16);
      const float wr[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = fmaf(wr[i], vv[i], o[i]);
      const size_t yo = ((static_cast<size_t>(b) * T + t0 + tl) * N + n0) * V + r;  // = y + tl N V + r
      if (in_range(p.status, yo, 8, y_ext, CHK_FWD_Y)) store8(y + static_cast<size_t>(tl) * N * V + r, o);
      if constexpr (NORM) {
        float gg[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (in_range(p.status, yo, 8, y_ext, CHK_FWD_G)) ldg8<F32>(static_cast<const TIn*>(p.g) + yo, gg);
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float og = o[i] * gg[i];
          part = fmaf(og, og, part);
        }
        const size_t so = static_cast<size_t>(b) * T + t0 + tl;
        if (in_range(p.status, so, 1, static_cast<size_t>(p.B) * T, CHK_FWD_SSQ)) atomicAdd(p.ssq + so, part);
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
// 8*nt + 2c (+1)) to a [K][V] fp32 array.  dst is element off0 of an array
// of `extent` elements (index checks of the checked build, at `site`).
template <int V, int MT, bool HALF = false>
__device__ __forceinline__ void store_state(float* dst, const float (&H)[MT][V / 8][4], int row0,
                                            int g, int c, int* status, size_t off0, size_t extent,
                                            int site) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < V / 8; ++nt)
#pragma unroll
      for (int h = 0; h < (HALF ? 1 : 2); ++h) {
        const int row = row0 + 16 * mt + g + 8 * h;
        const int o = row * V + 8 * nt + 2 * c;
        if (in_range(status, off0 + o, 2, extent, site))
          *reinterpret_cast<float2*>(dst + o) = make_float2(H[mt][nt][2 * h], H[mt][nt][2 * h + 1]);
      }
}

// Accumulator layout of n-tiles (2ks, 2ks+1) -> A operand of k-step ks
// (rows 8..15 zero for half slices).
template <int V, bool HALF = false>
__device__ __forceinline__ void pack_a(const float (&H)[V / 8][4], uint32_t (&A)[V / 16][4]) {
#pragma unroll
  for (int ks = 0; ks < V / 16; ++ks) {
    A[ks][0] = ptx::pack_bf16x2(H[2 * ks][0], H[2 * ks][1]);
    A[ks][1] = HALF ? 0u : ptx::pack_bf16x2(H[2 * ks][2], H[2 * ks][3]);
    A[ks][2] = ptx::pack_bf16x2(H[2 * ks + 1][0], H[2 * ks + 1][1]);
    A[ks][3] = HALF ? 0u : ptx::pack_bf16x2(H[2 * ks + 1][2], H[2 * ks + 1][3]);
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

// Rank-1 inputs of one step, read one step ahead of their use:
// k as fp32 pairs (k_i, k_i) at rows 16mt+g and 16mt+8+g, and v at columns
// 8nt+2c, 8nt+2c+1 (bf16x2 in the bf16 path, fp32 pair in the fp32 path).
// bf16 path: the rank-1 term as an MMA of two one-column operands, k as
// (k_i, 0) A-operand words at rows 16mt+g and 16mt+8+g and v as (v_j, 0)
// B-operand words at columns 8nt+g, on the lanes with c == 0 (zero on the
// others).
template <int MT, int NT, bool F32>
struct StepIn {
  float2 k0[MT], k1[MT];
  uint32_t vb[NT];
  float2 vf[NT];
  float kv[MT][NT][4];  // bf16 path: k v^T of the step, formed while the previous step runs
};

// kdb: the step's k (fp32 pairs in the fp32 path, raw bf16 otherwise) at
// this warp's first row; vb: its v (raw) at this head.
template <int V, int MT, bool F32, bool HALF, bool PAIRS>
__device__ __forceinline__ void load_step(StepIn<MT, V / 8, F32>& in, uint32_t kdb, uint32_t vb,
                                          int g, int c) {
  if constexpr (PAIRS) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      in.k0[mt] = ptx::lds_f32x2(kdb + 8 * (16 * mt + g));
      in.k1[mt] = HALF ? make_float2(0.f, 0.f) : ptx::lds_f32x2(kdb + 8 * (16 * mt + 8 + g));
    }
#pragma unroll
    for (int nt = 0; nt < V / 8; ++nt) {
      if (F32)
        in.vf[nt] = ptx::lds_f32x2(vb + 4 * (8 * nt + 2 * c));
      else
        in.vb[nt] = ptx::lds_u32(vb + 2 * (8 * nt + 2 * c));
    }
  } else {
    uint32_t vz[V / 8];
#pragma unroll
    for (int nt = 0; nt < V / 8; ++nt) vz[nt] = c == 0 ? ptx::lds_u16(vb + 2 * (8 * nt + g)) : 0u;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const uint32_t Ak[4] = {c == 0 ? ptx::lds_u16(kdb + 2 * (16 * mt + g)) : 0u,
                              (c == 0 && !HALF) ? ptx::lds_u16(kdb + 2 * (16 * mt + 8 + g)) : 0u,
                              0u, 0u};
#pragma unroll
      for (int nt = 0; nt < V / 8; ++nt) ptx::mma_bf16_16816_zero(in.kv[mt][nt], Ak, vz[nt], 0u);
    }
  }
}

// Per-warp constant operands and the running state.
template <int V, int MT>
struct WarpState {
  uint32_t Bw[V / 16][V / 8][2];   // W, bf16 hi
  uint32_t Bwl[V / 16][V / 8][2];  // W, bf16 lo residual (fp32-input path)
  float H[MT][V / 8][4];           // state, fp32
  uint32_t A[MT][V / 16][4];       // bf16(H) as A operand
  uint32_t Al[MT][V / 16][4];      // residual of bf16(H) (fp32-input path)
};

// Readout partial y^T = q^T H of this warp's MT slices on the tensor core
// (bf16 path): A = q in every row, B = the slices of bf16(H) transposed
// 8x8-blockwise; columns 8nt+2c, +1 are stored to ypaddr by lanes g == 0.
template <int V, int MT, bool HALF>
__device__ __forceinline__ void readout_bf16(const uint32_t (&A)[MT][V / 16][4], uint32_t qb,
                                             uint32_t ypaddr, int g, int c) {
  constexpr int NT = V / 8, KS = V / 16;
  float ya[NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const uint32_t q0 = ptx::lds_u32(qb + 2 * (16 * mt + 2 * c));
    const uint32_t q1 = ptx::lds_u32(qb + 2 * (16 * mt + 8 + 2 * c));
    const uint32_t Aq[4] = {q0, q0, q1, q1};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t b0 = ptx::movmatrix_trans(A[mt][ks][2 * h2]);
        const uint32_t b1 = HALF ? 0u : ptx::movmatrix_trans(A[mt][ks][2 * h2 + 1]);
        if (mt == 0)
          ptx::mma_bf16_16816_zero(ya[2 * ks + h2], Aq, b0, b1);
        else
          ptx::mma_bf16_16816(ya[2 * ks + h2], Aq, b0, b1);
      }
  }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) ptx::sts_f32x2(ypaddr + 4 * (8 * nt + 2 * c), ya[nt][0], ya[nt][1]);
  }
}

// Z = tanh(acc); H = Z + f (H - Z) for one 16-row slice; then the next
// step's A operand.  Every forward variant (and the backward's recompute)
// performs these operations in this order, so the state is the same bit for
// bit whichever launch shape computed it.
template <int V, bool F32, bool HALF>
__device__ __forceinline__ void state_update(float (&H)[V / 8][4], const float (&acc)[V / 8][4],
                                             float2 f2, uint32_t (&A)[V / 16][4],
                                             uint32_t (&Al)[V / 16][4]) {
  const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int nt = 0; nt < V / 8; ++nt)
#pragma unroll
    for (int h = 0; h < (HALF ? 1 : 2); ++h) {
      float2 z;
      z.x = F32 ? tanhf(acc[nt][2 * h]) : ptx::tanh_approx(acc[nt][2 * h]);
      z.y = F32 ? tanhf(acc[nt][2 * h + 1]) : ptx::tanh_approx(acc[nt][2 * h + 1]);
      const float2 hp = make_float2(H[nt][2 * h], H[nt][2 * h + 1]);
      const float2 d = __ffma2_rn(m1, z, hp);
      const float2 hn = __ffma2_rn(f2, d, z);
      H[nt][2 * h] = hn.x;
      H[nt][2 * h + 1] = hn.y;
    }
  pack_a<V, HALF>(H, A);
  if (F32) pack_a_lo<V>(H, A, Al);
}

// Whether a step writes the previous step's readout (bf16, one 16-row slice
// per warp: the readout's transposes and MMA then fill the latency of the
// state products) instead of its own (measured slower with two slices per
// warp, where the two slices' chains already overlap).
template <int MT, bool F32>
__host__ __device__ constexpr bool defer_readout() {
  return !F32 && MT == 1;
}

// One recurrence step for this warp's MT slices.  Writes a readout partial
// (columns 8nt+2c, +1, on lanes with g == 0) to ypaddr from q at qb: the
// step's own, or with defer_readout() the previous step's, formed from the
// bf16(H) operand of this step's H W products before they are used (the last
// step of a run then needs readout_bf16 afterwards).  next() reads the next
// step's inputs: first, or with defer_readout() right behind this step's
// H W products, so that its loads and k v^T products do not hold up this
// step's chain in the warp's in-order issue.
template <int V, int MT, bool F32, bool HALF, bool PAIRS, typename Next>
__device__ __forceinline__ void fwd_step(WarpState<V, MT>& S, const StepIn<MT, V / 8, F32>& in,
                                         uint32_t qb, uint32_t fdaddr, uint32_t ypaddr, int g,
                                         int c, Next&& next) {
  constexpr int NT = V / 8, KS = V / 16;
  constexpr bool DEFER = defer_readout<MT, F32>();
  if constexpr (!DEFER) next();
  // q (for the readout) and f are read here; their use is tens of cycles on.
  uint32_t qa[MT][2];
  float qf[MT][2];
  if constexpr (!DEFER) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      if (F32) {
        qf[mt][0] = ptx::lds_f32(qb + 4 * (16 * mt + g));
        qf[mt][1] = ptx::lds_f32(qb + 4 * (16 * mt + 8 + g));
      } else {
        qa[mt][0] = ptx::lds_u32(qb + 2 * (16 * mt + 2 * c));
        qa[mt][1] = ptx::lds_u32(qb + 2 * (16 * mt + 8 + 2 * c));
      }
    }
  }
  const float2 f2 = ptx::lds_f32x2(fdaddr);
  const float2 m1 = make_float2(-1.f, -1.f);
  // acc = k v^T (exact fp32 products: one nonzero product per element in
  // the bf16 path's MMA), then acc += bf16(H) W on the tensor core.
  auto products = [&](int mt, float (&acc)[NT][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if constexpr (PAIRS) {
        const float2 vv =
            F32 ? in.vf[nt] : make_float2(ptx::bf16x2_lo(in.vb[nt]), ptx::bf16x2_hi(in.vb[nt]));
        const float2 lo = __fmul2_rn(in.k0[mt], vv);
        const float2 hi = HALF ? make_float2(0.f, 0.f) : __fmul2_rn(in.k1[mt], vv);
        acc[nt][0] = lo.x;
        acc[nt][1] = lo.y;
        acc[nt][2] = hi.x;
        acc[nt][3] = hi.y;
      } else {
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[nt][r] = in.kv[mt][nt][r];
      }
    }
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        ptx::mma_bf16_16816(acc[nt], S.A[mt][ks], S.Bw[ks][nt][0], S.Bw[ks][nt][1]);
        if (F32) {
          ptx::mma_bf16_16816(acc[nt], S.A[mt][ks], S.Bwl[ks][nt][0], S.Bwl[ks][nt][1]);
          ptx::mma_bf16_16816(acc[nt], S.Al[mt][ks], S.Bw[ks][nt][0], S.Bw[ks][nt][1]);
        }
      }
  };
  // Z = tanh(acc); H = Z + f (H - Z); the next step's A operand
  auto update = [&](int mt, const float (&acc)[NT][4]) {
    state_update<V, F32, HALF>(S.H[mt], acc, f2, S.A[mt], S.Al[mt]);
  };
  if constexpr (DEFER) {
    float acc[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) products(mt, acc[mt]);
    next();
    readout_bf16<V, MT, HALF>(S.A, qb, ypaddr, g, c);  // the previous step's, in the MMAs' shadow
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) update(mt, acc[mt]);
  } else {
    float ya[NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      float acc[NT][4];
      products(mt, acc);
      update(mt, acc);
      if constexpr (F32) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float p0 = fmaf(qf[mt][0], S.H[mt][nt][0], qf[mt][1] * S.H[mt][nt][2]);
          const float p1 = fmaf(qf[mt][0], S.H[mt][nt][1], qf[mt][1] * S.H[mt][nt][3]);
          ya[nt][0] = mt == 0 ? p0 : ya[nt][0] + p0;
          ya[nt][1] = mt == 0 ? p1 : ya[nt][1] + p1;
        }
      } else {
        // Readout y^T += q^T H on the tensor core: A = q in every row,
        // B = this slice of bf16(H_t) transposed 8x8-blockwise.
        const uint32_t Aq[4] = {qa[mt][0], qa[mt][0], qa[mt][1], qa[mt][1]};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const uint32_t b0 = ptx::movmatrix_trans(S.A[mt][ks][2 * h2]);
            const uint32_t b1 = HALF ? 0u : ptx::movmatrix_trans(S.A[mt][ks][2 * h2 + 1]);
            if (mt == 0)
              ptx::mma_bf16_16816_zero(ya[2 * ks + h2], Aq, b0, b1);
            else
              ptx::mma_bf16_16816(ya[2 * ks + h2], Aq, b0, b1);
          }
      }
    }
    if constexpr (F32) {
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
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) ptx::sts_f32x2(ypaddr + 4 * (8 * nt + 2 * c), ya[nt][0], ya[nt][1]);
    }
  }  // !DEFER
}

template <int V, int MT_, bool F32, bool PAIRS>
__device__ __forceinline__ void fwd_consumer(const FwdParams& p, const FwdLayout& L, uint32_t sbase,
                                             int b, int n0, int ci) {
  using TIn = typename InType<F32>::T;
  constexpr bool HALF = MT_ == 0;       // half slices: 8 rows per warp
  constexpr int MT = HALF ? 1 : MT_;
  constexpr int es = sizeof(TIn);
  constexpr int NT = V / 8, KS = V / 16;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int K = p.K, T = p.T, N = p.N, G = p.G, WPH = p.WPH;
  const int hl = ci / WPH, w = ci - hl * WPH;
  const int n = n0 + hl;
  const int row0 = w * (HALF ? 8 : 16 * MT);
  const uint32_t bars = sbase + L.bars;

  WarpState<V, MT> S;
  // W as B operands (k = row l of W, n = column j), bf16 hi (+ lo residual).
  const TIn* Wn = static_cast<const TIn*>(p.W) + static_cast<size_t>(n) * V * V;
  const bool w_ok = in_range(p.status, static_cast<size_t>(n) * V * V, V * V,
                             static_cast<size_t>(N) * V * V, CHK_FWD_PARAM);
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r0 = 16 * ks + 8 * h + 2 * c, col = 8 * nt + g;
        const float w0 = w_ok ? to_f(Wn[r0 * V + col]) : 0.f;
        const float w1 = w_ok ? to_f(Wn[(r0 + 1) * V + col]) : 0.f;
        S.Bw[ks][nt][h] = ptx::pack_bf16x2(w0, w1);
        S.Bwl[ks][nt][h] = F32 ? ptx::pack_bf16x2(w0 - ptx::bf16x2_lo(S.Bw[ks][nt][h]),
                                                  w1 - ptx::bf16x2_hi(S.Bw[ks][nt][h]))
                               : 0u;
      }
  const size_t hoff = (static_cast<size_t>(b) * N + n) * K * V;
  const size_t h_ext = static_cast<size_t>(p.B) * N * K * V;  // H0, H_T (index checks)
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = row0 + 16 * mt + g + 8 * (r >> 1), col = 8 * nt + 2 * c + (r & 1);
        const size_t o = hoff + row * V + col;
        S.H[mt][nt][r] = (p.H0 && (!HALF || r < 2) && in_range(p.status, o, 1, h_ext, CHK_FWD_H0))
                             ? p.H0[o]
                             : 0.f;
      }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    pack_a<V, HALF>(S.H[mt], S.A[mt]);
    if (F32) pack_a_lo<V>(S.H[mt], S.A[mt], S.Al[mt]);
  }

  float* ckpt = p.ckpt ? p.ckpt + (static_cast<size_t>(b) * N + n) * p.nck * K * V : nullptr;
  size_t ck_off = (static_cast<size_t>(b) * N + n) * p.nck * K * V;  // element offset of ckpt
  const size_t ck_ext = static_cast<size_t>(p.B) * N * p.nck * K * V;
  // Absolute step before which the next checkpoint is stored (the state
  // after next_ck steps); beyond T when no checkpoints are written.
  int next_ck = ckpt != nullptr ? 0 : T + 1;
  const int TC = p.tc;
  const int nchunks = (T + TC - 1) / TC;
  // Per-time-step strides of this lane's shared-memory reads.
  const uint32_t q_stride = static_cast<uint32_t>(K * es);
  const uint32_t kd_stride = static_cast<uint32_t>(PAIRS ? K * 8 : K * 2);
  const uint32_t v_stride = static_cast<uint32_t>(G * V * es);
  const uint32_t fd_stride = static_cast<uint32_t>(G * 8);
  const uint32_t yp_stride = static_cast<uint32_t>(G * WPH * V * 4);
  bool ok = true;
  StepIn<MT, NT, F32> in0, in1;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int s = ch % NSTAGE, ys = ch % NYSTAGE;
    if (!warp_wait(bar_in_full(bars, s), (ch / NSTAGE) & 1, p.wait_limit_ns) ||
        !warp_wait(bar_yp_empty(bars, ys), ((ch / NYSTAGE) & 1) ^ 1, p.wait_limit_ns)) {
      ok = false;
      break;
    }
    const int t0 = ch * TC;
    const int Tc = min(TC, T - t0);
    const uint32_t st = sbase + static_cast<uint32_t>(s) * L.stage;
    const uint32_t qb = st + L.q + static_cast<uint32_t>(row0 * es);
    const uint32_t kdb = PAIRS ? st + L.kd + static_cast<uint32_t>(row0 * 8)
                                               : st + L.k + static_cast<uint32_t>(row0 * 2);
    const uint32_t vb = st + L.v + static_cast<uint32_t>(hl * V * es);
    const uint32_t fdb = st + L.fd + static_cast<uint32_t>(hl * 8);
    const uint32_t yb = sbase + L.yp_base + static_cast<uint32_t>(ys) * L.yp_stage +
                        static_cast<uint32_t>(((hl * WPH) + w) * V * 4);
    // The rank-1 inputs of step tl+1 are read while step tl computes (by the
    // next() of each fwd_step below).  The
    // read past the chunk's last step (slot Tc <= TC) stays inside this
    // stage's shared memory and its values are never used.
    load_step<V, MT, F32, HALF, PAIRS>(in0, kdb, vb, g, c);
    int tl = 0;
    while (tl < Tc) {
      if (t0 + tl == next_ck) {
        store_state<V, MT, HALF>(ckpt, S.H, row0, g, c, p.status, ck_off, ck_ext, CHK_FWD_CKPT);
        ckpt += K * V;
        ck_off += static_cast<size_t>(K) * V;
        next_ck += p.C;
      }
      const int seg_end = min(Tc, next_ck - t0);  // no checkpoint inside [tl, seg_end)
      // The readout a step writes: its own, or with defer_readout() the
      // previous step's (at the chunk's first step a placeholder for step 0,
      // overwritten by step 0's readout before the chunk is released).
      auto ro = [](uint32_t u) -> uint32_t {
        return defer_readout<MT, F32>() ? (u > 0 ? u - 1 : 0) : u;
      };
      if constexpr (defer_readout<MT, F32>()) {
        // One-slice warps (these launches take their strides at run time):
        // running addresses, one add per stream and two steps, instead of a
        // multiply-add per address and step.
        uint32_t kp = kdb + static_cast<uint32_t>(tl) * kd_stride;
        uint32_t vp = vb + static_cast<uint32_t>(tl) * v_stride;
        uint32_t fp = fdb + static_cast<uint32_t>(tl) * fd_stride;
        if (tl + 1 < seg_end) {  // first pair: step tl writes the readout slot ro(tl)
          const uint32_t q0 = qb + ro(static_cast<uint32_t>(tl)) * q_stride;
          const uint32_t y0 = yb + ro(static_cast<uint32_t>(tl)) * yp_stride;
          fwd_step<V, MT, F32, HALF, PAIRS>(S, in0, q0, fp, y0, g, c,
              [&] { load_step<V, MT, F32, HALF, PAIRS>(in1, kp + kd_stride, vp + v_stride, g, c); });
          fwd_step<V, MT, F32, HALF, PAIRS>(S, in1, qb + static_cast<uint32_t>(tl) * q_stride,
                                            fp + fd_stride,
                                            yb + static_cast<uint32_t>(tl) * yp_stride, g, c,
              [&] { load_step<V, MT, F32, HALF, PAIRS>(in0, kp + 2 * kd_stride, vp + 2 * v_stride, g, c); });
          tl += 2;
          kp += 2 * kd_stride;
          vp += 2 * v_stride;
          fp += 2 * fd_stride;
        }
        uint32_t qp = qb + static_cast<uint32_t>(tl - 1) * q_stride;  // readout of step tl - 1
        uint32_t ypp = yb + static_cast<uint32_t>(tl - 1) * yp_stride;
#pragma unroll 1
        for (; tl + 1 < seg_end; tl += 2) {
          fwd_step<V, MT, F32, HALF, PAIRS>(S, in0, qp, fp, ypp, g, c,
              [&] { load_step<V, MT, F32, HALF, PAIRS>(in1, kp + kd_stride, vp + v_stride, g, c); });
          fwd_step<V, MT, F32, HALF, PAIRS>(S, in1, qp + q_stride, fp + fd_stride,
                                            ypp + yp_stride, g, c,
              [&] { load_step<V, MT, F32, HALF, PAIRS>(in0, kp + 2 * kd_stride, vp + 2 * v_stride, g, c); });
          kp += 2 * kd_stride;
          vp += 2 * v_stride;
          fp += 2 * fd_stride;
          qp += 2 * q_stride;
          ypp += 2 * yp_stride;
        }
      } else {
#pragma unroll 1
        for (; tl + 1 < seg_end; tl += 2) {
          const uint32_t u0 = static_cast<uint32_t>(tl), u1 = u0 + 1, u2 = u0 + 2;
          fwd_step<V, MT, F32, HALF, PAIRS>(S, in0, qb + ro(u0) * q_stride, fdb + u0 * fd_stride,
                                            yb + ro(u0) * yp_stride, g, c,
              [&] { load_step<V, MT, F32, HALF, PAIRS>(in1, kdb + u1 * kd_stride, vb + u1 * v_stride, g, c); });
          fwd_step<V, MT, F32, HALF, PAIRS>(S, in1, qb + ro(u1) * q_stride, fdb + u1 * fd_stride,
                                            yb + ro(u1) * yp_stride, g, c,
              [&] { load_step<V, MT, F32, HALF, PAIRS>(in0, kdb + u2 * kd_stride, vb + u2 * v_stride, g, c); });
        }
      }
      if (tl < seg_end) {  // odd remainder of the segment
        const uint32_t u0 = static_cast<uint32_t>(tl), u1 = u0 + 1;
        fwd_step<V, MT, F32, HALF, PAIRS>(S, in0, qb + ro(u0) * q_stride, fdb + u0 * fd_stride,
                                          yb + ro(u0) * yp_stride, g, c,
            [&] { load_step<V, MT, F32, HALF, PAIRS>(in1, kdb + u1 * kd_stride, vb + u1 * v_stride, g, c); });
        in0 = in1;
        ++tl;
      }
    }
    if constexpr (defer_readout<MT, F32>()) {  // the chunk's last step's readout
      const uint32_t ul = static_cast<uint32_t>(Tc - 1);
      readout_bf16<V, MT, HALF>(S.A, qb + ul * q_stride, yb + ul * yp_stride, g, c);
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
  if (p.HT != nullptr)
    store_state<V, MT, HALF>(p.HT + hoff, S.H, row0, g, c, p.status, hoff, h_ext, CHK_FWD_HT);
}

// KC, GC (0 = taken from the parameters): K and heads per CTA fixed at
// compile time, so that every shared-memory stride of the step loops is an
// immediate (instances for the common K = 64 launches).
// Epilogue warps per CTA: three in the dense 8-head CTAs (with the producer,
// one helper warp per SMSP), one elsewhere (smaller CTAs share SMs, and
// more warps would cost them occupancy).
template <int GC>
__host__ __device__ constexpr int fwd_epilogue_warps() {
  return GC >= 8 ? 3 : 1;
}

template <int V, int MT, bool F32, bool GATED, bool NORM, int KC = 0, int GC = 0>
__global__ void __launch_bounds__(32 * (1 + fwd_epilogue_warps<GC>() + max_consumer_warps<V, MT, F32>()), 1)
    fwd_kernel(const FwdParams prm) {
  FwdParams p = prm;
  if constexpr (KC > 0) {
    p.K = KC;
    p.WPH = MT == 0 ? KC / 8 : KC / (16 * MT);
  }
  if constexpr (GC > 0) p.G = GC;
  using TIn = typename InType<F32>::T;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.x / p.ngroups;
  const int n0 = (blockIdx.x % p.ngroups) * p.G;
  const int Geff = min(p.G, p.N - n0);
  const int ncons = Geff * p.WPH;
  constexpr bool PAIRS = rank1_pairs<V, F32, GC>();
  constexpr int NEPI = fwd_epilogue_warps<GC>();
  const FwdLayout L = fwd_layout(p.K, V, p.G, p.WPH, sizeof(TIn), p.tc, PAIRS);
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bars = sbase + L.bars;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(bar_raw_full(bars, s), 1);
      ptx::mbar_init(bar_in_full(bars, s), 1);
      ptx::mbar_init(bar_in_empty(bars, s), ncons + NEPI);
    }
    for (int s = 0; s < NYSTAGE; ++s) {
      ptx::mbar_init(bar_yp_full(bars, s), ncons);
      ptx::mbar_init(bar_yp_empty(bars, s), NEPI);
    }
    ptx::mbar_init_fence();
  }
  __syncthreads();
  if (warp == 0) {
    // With fault injection on, the producer issues nothing, so every wait of
    // the other warps runs into its time limit (tests of the time-out path).
    if (p.inject_stall == 0) fwd_producer<V, F32, GATED, PAIRS>(p, L, sbase, b, n0, Geff);
  } else if (warp <= NEPI) {
    fwd_epilogue<V, F32, NORM, NEPI>(p, L, sbase, b, n0, Geff, warp - 1);
  } else if (warp - 1 - NEPI < ncons) {
    fwd_consumer<V, MT, F32, PAIRS>(p, L, sbase, b, n0, warp - 1 - NEPI);
  }
}

// ---------------------------------------------------------------------------
// One-wave kernel.  When a batch has more heads than one wave of the CTAs
// above holds (8 heads of two warps each per SM), they run in two waves and
// each wave pays the latency of every step in full.  This kernel instead
// keeps all heads resident at once: CTA c takes G = ceil(B N / SMs) heads
// [c G, c G + G) of the flattened (b, n) order -- at most two batch items,
// since G <= N -- with one consumer warp per head holding all K rows (KC / 16
// slices of 16) and storing y itself, and one producer warp that stages q, k
// (per batch item), v and f.  bf16 inputs, V = 16, N_q = 1.
// ---------------------------------------------------------------------------
constexpr int kWaveMaxHeads = 14;

struct WaveLayout {
  uint32_t q, k;   // [2][TC][K] bf16, one block per batch item of the CTA
  uint32_t kd;     // [2][TC][K][2] fp32 (k, k) pairs
  uint32_t v;      // [TC][G][V] bf16
  uint32_t fd;     // [TC][G][2] fp32 (f, f) pairs
  uint32_t stage;
  uint32_t wr;     // [G][V] fp32 w_r of the CTA's heads (outside the ring)
  uint32_t bars, total;
};

__host__ __device__ inline WaveLayout wave_layout(int K, int V, int G, int TC) {
  WaveLayout L;
  uint32_t o = 0;
  L.q = o;
  o = align_up(o + 2 * TC * K * 2, 128);
  L.k = o;
  o = align_up(o + 2 * TC * K * 2, 128);
  L.kd = o;
  o = align_up(o + 2 * TC * K * 8, 128);
  L.v = o;
  o = align_up(o + TC * G * V * 2, 128);
  L.fd = o;
  o = align_up(o + TC * G * 8, 128);
  L.stage = o;
  L.wr = NSTAGE * L.stage;
  L.bars = align_up(L.wr + G * V * 4, 128);
  L.total = L.bars + 8 * 3 * NSTAGE;
  return L;
}

// The CTA's heads as up to two runs of consecutive heads: cnt0 heads of
// batch item b0 from head n0 on, then cnt1 heads of batch item b0 + 1 from
// head 0 on.
struct WaveSegs {
  int b0, n0, cnt0, cnt1, nseg, Geff;
  __device__ __forceinline__ int b(int sgi) const { return b0 + sgi; }
  __device__ __forceinline__ int first(int sgi) const { return sgi ? 0 : n0; }
  __device__ __forceinline__ int cnt(int sgi) const { return sgi ? cnt1 : cnt0; }
  __device__ __forceinline__ int offset(int sgi) const { return sgi ? cnt0 : 0; }
};

__device__ __forceinline__ WaveSegs wave_segs(const FwdParams& p) {
  WaveSegs sg;
  const long long h0 = static_cast<long long>(blockIdx.x) * p.G;
  const long long total = static_cast<long long>(p.B) * p.N;
  sg.Geff = static_cast<int>(min(static_cast<long long>(p.G), total - h0));
  sg.b0 = static_cast<int>(h0 / p.N);
  sg.n0 = static_cast<int>(h0 - static_cast<long long>(sg.b0) * p.N);
  sg.cnt0 = min(sg.Geff, p.N - sg.n0);
  sg.cnt1 = sg.Geff - sg.cnt0;
  sg.nseg = sg.cnt1 > 0 ? 2 : 1;
  return sg;
}

template <bool GATED>
__device__ __forceinline__ void wave_producer(const FwdParams& p, const WaveLayout& L, uint32_t sbase,
                                              const WaveSegs& sg) {
  using TIn = __nv_bfloat16;
  constexpr int es = 2, V = 16;
  const int lane = threadIdx.x & 31;
  const int K = p.K, T = p.T, N = p.N, G = p.G, TC = p.tc;
  const uint32_t bars = sbase + L.bars;
  const int nchunks = (T + TC - 1) / TC;
  const TIn* q = static_cast<const TIn*>(p.q);
  const TIn* k = static_cast<const TIn*>(p.k);
  const TIn* v = static_cast<const TIn*>(p.v);
  const TIn* f = static_cast<const TIn*>(GATED ? p.a : p.f);
  const TIn* galpha = static_cast<const TIn*>(p.alpha);
  const TIn* gbeta = static_cast<const TIn*>(p.beta);
  const size_t qk_ext = static_cast<size_t>(p.B) * T * K;
  const size_t v_ext = static_cast<size_t>(p.B) * T * N * V, f_ext = static_cast<size_t>(p.B) * T * N;

  auto issue = [&](int ch) -> bool {
    const int s = ch % NSTAGE;
    if (!warp_wait(bar_in_empty(bars, s), ((ch / NSTAGE) & 1) ^ 1, p.wait_limit_ns)) return false;
    const int t0 = ch * TC;
    const int Tc = min(TC, T - t0);
    const uint32_t qk_bytes = static_cast<uint32_t>(Tc * K * es);
    const uint32_t raw = bar_raw_full(bars, s);
    if (lane == 0)
      ptx::mbar_expect_tx(raw, static_cast<uint32_t>(sg.nseg) * 2 * qk_bytes +
                                   static_cast<uint32_t>(Tc * sg.Geff * V * es));
    __syncwarp();
    const uint32_t st = sbase + static_cast<uint32_t>(s) * L.stage;
    for (int sgi = 0; sgi < sg.nseg; ++sgi) {
      const size_t bt0 = static_cast<size_t>(sg.b(sgi)) * T + t0;
      if (lane == 0) {
        const uint32_t off = static_cast<uint32_t>(sgi * TC * K * es);
        if (in_range(p.status, bt0 * K, static_cast<size_t>(Tc) * K, qk_ext, CHK_FWD_QK)) {
          ptx::bulk_g2s(st + L.q + off, q + bt0 * K, qk_bytes, raw);
          ptx::bulk_g2s(st + L.k + off, k + bt0 * K, qk_bytes, raw);
        } else {
          ptx::mbar_complete_tx(raw, 2 * qk_bytes);
        }
      }
      // this batch item's heads of every step: one contiguous run of v
      const uint32_t v_bytes = static_cast<uint32_t>(sg.cnt(sgi) * V * es);
      const uint32_t v_off = static_cast<uint32_t>(sg.offset(sgi) * V * es);
      for (int tl = lane; tl < Tc; tl += 32) {
        const size_t src = ((bt0 + tl) * N + sg.first(sgi)) * V;
        if (in_range(p.status, src, static_cast<size_t>(sg.cnt(sgi)) * V, v_ext, CHK_FWD_V))
          ptx::bulk_g2s(st + L.v + static_cast<uint32_t>(tl * G * V * es) + v_off, v + src, v_bytes, raw);
        else
          ptx::mbar_complete_tx(raw, v_bytes);
      }
    }
    // f (or, gated, f from a) -> fp32 pairs [TC][G][2]; loads batched
    const int Geff = sg.Geff, nf = Tc * Geff;
    for (int base = 0; base < nf; base += 256) {
      float fv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = base + lane + 32 * i;
        const int tl = e / Geff, h = e - tl * Geff;
        const int sgi = h < sg.cnt0 ? 0 : 1;
        const int n = sgi ? h - sg.cnt0 : sg.n0 + h;
        const size_t fi = (static_cast<size_t>(sg.b(sgi)) * T + t0 + tl) * N + n;
        const bool use = e < nf && in_range(p.status, fi, 1, f_ext, CHK_FWD_F);
        if constexpr (GATED)
          fv[i] = use && in_range(p.status, n, 1, N, CHK_FWD_PARAM)
                      ? gate_f(to_f(f[fi]), to_f(galpha[n]), to_f(gbeta[n]))
                      : 0.f;
        else
          fv[i] = use ? to_f(f[fi]) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = base + lane + 32 * i;
        const int tl = e / Geff, h = e - tl * Geff;
        if (e < nf) ptx::sts_f32x2(st + L.fd + static_cast<uint32_t>((tl * G + h) * 8), fv[i], fv[i]);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(raw);
    return true;
  };

  // k of each batch item as fp32 (k, k) pairs, then the chunk is released
  auto convert = [&](int ch) -> bool {
    const int s = ch % NSTAGE;
    if (!warp_wait(bar_raw_full(bars, s), (ch / NSTAGE) & 1, p.wait_limit_ns)) return false;
    const int Tc = min(TC, T - ch * TC);
    const uint32_t st = sbase + static_cast<uint32_t>(s) * L.stage;
    const int n8 = Tc * K / 8;
    for (int sgi = 0; sgi < sg.nseg; ++sgi) {
      const uint32_t src = st + L.k + static_cast<uint32_t>(sgi * TC * K * es);
      const uint32_t dst = st + L.kd + static_cast<uint32_t>(sgi * TC * K * 8);
      for (int i = lane; i < n8; i += 32) {
        const uint4 u = ptx::lds_u32x4(src + 16 * i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = ptx::bf16x2_lo(w[j]), hi = ptx::bf16x2_hi(w[j]);
          ptx::sts_f32x4(dst + 64 * i + 16 * j, lo, lo, hi, hi);
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar_in_full(bars, s));
    return true;
  };

  int issued = 0, converted = 0;
  bool ok = true;
  for (int ch = 0; ch < nchunks; ++ch) {
    if (!(ok = issue(ch))) break;
    issued = ch + 1;
    if (ch >= 1) {
      if (!(ok = convert(ch - 1))) break;
      converted = ch;
    }
  }
  if (ok && nchunks > 0) {
    if ((ok = convert(nchunks - 1))) converted = nchunks;
  }
  if (!ok && lane == 0) record_timeout(p.status, SITE_FWD_PRODUCER);
  for (int ch = max(converted, issued - NSTAGE); ch < issued; ++ch) {
    if (!warp_wait(bar_raw_full(bars, ch % NSTAGE), (ch / NSTAGE) & 1, kDrainLimitNs)) {
      if (lane == 0) record_timeout(p.status, SITE_FWD_DRAIN);
      break;
    }
  }
}

// One step of the one-wave kernel's consumer warp (all MT slices of one
// head): the rank-1 term from the step's fp32 (k, k) pairs, H W on the
// tensor core, the shared state update, the readout q^T H on the tensor
// core and y = q^T H + w_r (.) v stored as bf16 to ydst (nullptr: none).
// The operations per element are those of fwd_step.
template <int MT>
__device__ __forceinline__ void wave_step(WarpState<16, MT>& S, uint32_t kdb, uint32_t vb,
                                          uint32_t qb, uint32_t fdaddr, uint32_t wraddr,
                                          __nv_bfloat16* ydst, int g, int c) {
  constexpr int NT = 2;
  const float2 f2 = ptx::lds_f32x2(fdaddr);
  uint32_t vraw[NT];
  float2 vv[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    vraw[nt] = ptx::lds_u32(vb + 2 * (8 * nt + 2 * c));
    vv[nt] = make_float2(ptx::bf16x2_lo(vraw[nt]), ptx::bf16x2_hi(vraw[nt]));
  }
  float ya[NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const float2 k0 = ptx::lds_f32x2(kdb + 8 * (16 * mt + g));
    const float2 k1 = ptx::lds_f32x2(kdb + 8 * (16 * mt + 8 + g));
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 lo = __fmul2_rn(k0, vv[nt]);
      const float2 hi = __fmul2_rn(k1, vv[nt]);
      acc[nt][0] = lo.x;
      acc[nt][1] = lo.y;
      acc[nt][2] = hi.x;
      acc[nt][3] = hi.y;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) ptx::mma_bf16_16816(acc[nt], S.A[mt][0], S.Bw[0][nt][0], S.Bw[0][nt][1]);
    state_update<16, false, false>(S.H[mt], acc, f2, S.A[mt], S.Al[mt]);
    const uint32_t q0 = ptx::lds_u32(qb + 2 * (16 * mt + 2 * c));
    const uint32_t q1 = ptx::lds_u32(qb + 2 * (16 * mt + 8 + 2 * c));
    const uint32_t Aq[4] = {q0, q0, q1, q1};
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const uint32_t b0 = ptx::movmatrix_trans(S.A[mt][0][2 * h2]);
      const uint32_t b1 = ptx::movmatrix_trans(S.A[mt][0][2 * h2 + 1]);
      if (mt == 0)
        ptx::mma_bf16_16816_zero(ya[h2], Aq, b0, b1);
      else
        ptx::mma_bf16_16816(ya[h2], Aq, b0, b1);
    }
  }
  if (g == 0 && ydst != nullptr) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 wr2 = ptx::lds_f32x2(wraddr + 4 * (8 * nt + 2 * c));
      const float2 o = __ffma2_rn(wr2, vv[nt], make_float2(ya[nt][0], ya[nt][1]));
      *reinterpret_cast<uint32_t*>(ydst + 8 * nt + 2 * c) = ptx::pack_bf16x2(o.x, o.y);
    }
  }
}

template <int KC>
__device__ __forceinline__ void wave_consumer(const FwdParams& p, const WaveLayout& L, uint32_t sbase,
                                              const WaveSegs& sg, int hl) {
  using TIn = __nv_bfloat16;
  constexpr int V = 16, MT = KC / 16, NT = V / 8, KS = V / 16, es = 2;
  constexpr int K = KC;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int T = p.T, N = p.N, G = p.G, TC = p.tc;
  const int sgi = hl < sg.cnt0 ? 0 : 1;
  const int b = sg.b(sgi), n = sgi ? hl - sg.cnt0 : sg.n0 + hl;
  const uint32_t bars = sbase + L.bars;

  WarpState<V, MT> S;
  const TIn* Wn = static_cast<const TIn*>(p.W) + static_cast<size_t>(n) * V * V;
  const bool w_ok = in_range(p.status, static_cast<size_t>(n) * V * V, V * V,
                             static_cast<size_t>(N) * V * V, CHK_FWD_PARAM);
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r0 = 16 * ks + 8 * h + 2 * c, col = 8 * nt + g;
        const float w0 = w_ok ? to_f(Wn[r0 * V + col]) : 0.f;
        const float w1 = w_ok ? to_f(Wn[(r0 + 1) * V + col]) : 0.f;
        S.Bw[ks][nt][h] = ptx::pack_bf16x2(w0, w1);
        S.Bwl[ks][nt][h] = 0u;
      }
  // w_r of this head as fp32 in this warp's shared-memory slot
  const uint32_t wraddr = sbase + L.wr + static_cast<uint32_t>(hl * V * 4);
  if (lane < V) {
    const size_t o = static_cast<size_t>(n) * V + lane;
    ptx::sts_f32(wraddr + 4 * lane,
                 in_range(p.status, o, 1, static_cast<size_t>(N) * V, CHK_FWD_PARAM)
                     ? to_f(static_cast<const TIn*>(p.w_r)[o])
                     : 0.f);
  }
  __syncwarp();
  const size_t hoff = (static_cast<size_t>(b) * N + n) * K * V;
  const size_t h_ext = static_cast<size_t>(p.B) * N * K * V;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = 16 * mt + g + 8 * (r >> 1), col = 8 * nt + 2 * c + (r & 1);
        const size_t o = hoff + row * V + col;
        S.H[mt][nt][r] = (p.H0 && in_range(p.status, o, 1, h_ext, CHK_FWD_H0)) ? p.H0[o] : 0.f;
      }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) pack_a<V, false>(S.H[mt], S.A[mt]);

  float* ckpt = p.ckpt ? p.ckpt + (static_cast<size_t>(b) * N + n) * p.nck * K * V : nullptr;
  size_t ck_off = (static_cast<size_t>(b) * N + n) * p.nck * K * V;
  const size_t ck_ext = static_cast<size_t>(p.B) * N * p.nck * K * V;
  int next_ck = ckpt != nullptr ? 0 : T + 1;
  // y of this head: row t at y_head + t N V (no y in checkpoint-only runs)
  TIn* y_head = p.y ? static_cast<TIn*>(p.y) + (static_cast<size_t>(b) * T * N + n) * V : nullptr;
#if M2RNN_CHECK
  if (y_head != nullptr &&
      !in_range(p.status, (static_cast<size_t>(b) * T * N + n) * V + static_cast<size_t>(T - 1) * N * V,
                V, static_cast<size_t>(p.B) * T * N * V, CHK_FWD_Y))
    y_head = nullptr;  // (checked build: the head's last row would be out of range)
#endif
  const size_t y_step = static_cast<size_t>(N) * V;
  const int nchunks = (T + TC - 1) / TC;
  constexpr uint32_t q_stride = K * es, kd_stride = K * 8;
  const uint32_t v_stride = static_cast<uint32_t>(G * V * es);
  const uint32_t fd_stride = static_cast<uint32_t>(G * 8);
  bool ok = true;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int s = ch % NSTAGE;
    if (!warp_wait(bar_in_full(bars, s), (ch / NSTAGE) & 1, p.wait_limit_ns)) {
      ok = false;
      break;
    }
    const int t0 = ch * TC;
    const int Tc = min(TC, T - t0);
    const uint32_t st = sbase + static_cast<uint32_t>(s) * L.stage;
    const uint32_t qb = st + L.q + static_cast<uint32_t>(sgi * TC * K * es);
    const uint32_t kdb = st + L.kd + static_cast<uint32_t>(sgi * TC * K * 8);
    const uint32_t vb = st + L.v + static_cast<uint32_t>(hl * V * es);
    const uint32_t fdb = st + L.fd + static_cast<uint32_t>(hl * 8);
    TIn* yt = y_head != nullptr ? y_head + static_cast<size_t>(t0) * y_step : nullptr;
    int tl = 0;
    while (tl < Tc) {
      if (t0 + tl == next_ck) {
        store_state<V, MT, false>(ckpt, S.H, 0, g, c, p.status, ck_off, ck_ext, CHK_FWD_CKPT);
        ckpt += K * V;
        ck_off += static_cast<size_t>(K) * V;
        next_ck += p.C;
      }
      const int seg_end = min(Tc, next_ck - t0);
#pragma unroll 2
      for (; tl < seg_end; ++tl) {
        const uint32_t u = static_cast<uint32_t>(tl);
        wave_step<MT>(S, kdb + u * kd_stride, vb + u * v_stride, qb + u * q_stride, fdb + u * fd_stride,
                      wraddr, yt, g, c);
        if (yt != nullptr) yt += y_step;
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar_in_empty(bars, s));
  }
  if (!ok) {
    if (lane == 0) record_timeout(p.status, SITE_FWD_CONSUMER);
    return;
  }
  if (p.HT != nullptr)
    store_state<V, MT, false>(p.HT + hoff, S.H, 0, g, c, p.status, hoff, h_ext, CHK_FWD_HT);
}

template <bool GATED, int KC>
__global__ void __launch_bounds__(32 * (1 + kWaveMaxHeads), 1) fwd_wave_kernel(const FwdParams prm) {
  FwdParams p = prm;
  p.K = KC;
  p.WPH = 1;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const WaveSegs sg = wave_segs(p);
  const WaveLayout L = wave_layout(KC, 16, p.G, p.tc);
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bars = sbase + L.bars;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(bar_raw_full(bars, s), 1);
      ptx::mbar_init(bar_in_full(bars, s), 1);
      ptx::mbar_init(bar_in_empty(bars, s), sg.Geff);
    }
    ptx::mbar_init_fence();
  }
  __syncthreads();
  if (warp == 0) {
    if (p.inject_stall == 0) wave_producer<GATED>(p, L, sbase, sg);
  } else if (warp - 1 < sg.Geff) {
    wave_consumer<KC>(p, L, sbase, sg, warp - 1);
  }
}

// The kernel instance for p (fused gate, readout epilogue, compile-time K
// and heads per CTA), with the rank1_pairs choice it was compiled with (the
// launch's shared-memory layout depends on it).
template <int V, int MT, bool F32>
struct Selected {
  decltype(&fwd_kernel<V, MT, F32, false, false>) kern;
  bool pairs;
  int nepi = 1;  // epilogue warps
};

template <int V, int MT, bool F32>
Selected<V, MT, F32> select_kernel(const FwdParams& p) {
  // the instances with compile-time K and G (the K = 64 launches of large
  // batches; a G = 1, MT = 1 instance measured slower than the generic one)
  if constexpr (V == 16 && MT == 2 && !F32) {
    if (!p.norm && !p.gated && p.K == 64 && p.WPH == 2) {
      if (p.G == 8)
        return {fwd_kernel<16, 2, false, false, false, 64, 8>, rank1_pairs<16, false, 8>(),
                fwd_epilogue_warps<8>()};
      if (p.G == 2)
        return {fwd_kernel<16, 2, false, false, false, 64, 2>, rank1_pairs<16, false, 2>(),
                fwd_epilogue_warps<2>()};
    }
  }
  constexpr bool pairs = rank1_pairs<V, F32>();
  if (p.norm)
    return {p.gated ? fwd_kernel<V, MT, F32, true, true> : fwd_kernel<V, MT, F32, false, true>,
            pairs};
  return {p.gated ? fwd_kernel<V, MT, F32, true, false> : fwd_kernel<V, MT, F32, false, false>,
          pairs};
}

template <int V, int MT, bool F32>
int ctas_per_sm_t(const FwdParams& p) {
  const auto sel = select_kernel<V, MT, F32>(p);
  const FwdLayout L = fwd_layout(p.K, V, p.G, p.WPH, F32 ? 4 : 2, p.tc, sel.pairs);
  auto kern = sel.kern;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(L.total)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32 * (1 + sel.nepi + p.G * p.WPH),
                                                    L.total) !=
      cudaSuccess)
    return 0;
  return n;
}

template <int V, int MT, bool F32>
cudaError_t launch_t(const FwdParams& p, cudaStream_t stream) {
  const auto sel = select_kernel<V, MT, F32>(p);
  const FwdLayout L = fwd_layout(p.K, V, p.G, p.WPH, F32 ? 4 : 2, p.tc, sel.pairs);
  if (p.tc < 2 || p.tc > 64) return cudaErrorInvalidValue;
  if (p.G * p.WPH > max_consumer_warps<V, MT, F32>()) return cudaErrorInvalidConfiguration;
  auto kern = sel.kern;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(L.total));
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.B) * static_cast<unsigned>(p.ngroups);
  kern<<<grid, 32 * (1 + sel.nepi + p.G * p.WPH), L.total, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int fwd_wave_max_heads() { return kWaveMaxHeads; }

size_t fwd_wave_smem_bytes(int K, int G, int tc) { return wave_layout(K, 16, G, tc).total; }

cudaError_t launch_fwd_wave(const FwdParams& p, cudaStream_t stream) {
  if (p.K != 64 || p.G < 1 || p.G > kWaveMaxHeads || p.G > p.N || p.Nq != 1 || p.norm != 0 ||
      p.tc < 2 || p.tc > 32)
    return cudaErrorInvalidValue;
  const WaveLayout L = wave_layout(64, 16, p.G, p.tc);
  auto kern = p.gated ? fwd_wave_kernel<true, 64> : fwd_wave_kernel<false, 64>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(L.total));
  if (e != cudaSuccess) return e;
  const long long heads = static_cast<long long>(p.B) * p.N;
  const unsigned grid = static_cast<unsigned>((heads + p.G - 1) / p.G);
  kern<<<grid, 32 * (1 + p.G), L.total, stream>>>(p);
  return cudaGetLastError();
}

// (with k's fp32 pairs: an upper bound for the planner)
size_t fwd_smem_bytes(int K, int V, int G, int WPH, bool f32_inputs, int tc) {
  return fwd_layout(K, V, G, WPH, f32_inputs ? 4 : 2, tc, true).total;
}

int fwd_max_consumer_warps(int V, int MT, bool f32_inputs) {
  if (f32_inputs) return V == 16 ? max_consumer_warps<16, 1, true>() : max_consumer_warps<32, 1, true>();
  if (MT == 0) return V == 16 ? max_consumer_warps<16, 0, false>() : max_consumer_warps<32, 0, false>();
  if (V == 16)
    return MT == 1   ? max_consumer_warps<16, 1, false>()
           : MT == 2 ? max_consumer_warps<16, 2, false>()
                     : max_consumer_warps<16, 4, false>();
  return MT == 1 ? max_consumer_warps<32, 1, false>() : max_consumer_warps<32, 2, false>();
}

int fwd_ctas_per_sm(const FwdParams& p, int V, bool f32_inputs, int MT) {
  if (f32_inputs) return V == 16 ? ctas_per_sm_t<16, 1, true>(p) : ctas_per_sm_t<32, 1, true>(p);
  if (MT == 0) return V == 16 ? ctas_per_sm_t<16, 0, false>(p) : ctas_per_sm_t<32, 0, false>(p);
  if (V == 16)
    return MT == 1 ? ctas_per_sm_t<16, 1, false>(p)
           : MT == 2 ? ctas_per_sm_t<16, 2, false>(p) : ctas_per_sm_t<16, 4, false>(p);
  return MT == 1 ? ctas_per_sm_t<32, 1, false>(p) : ctas_per_sm_t<32, 2, false>(p);
}

cudaError_t launch_fwd(const FwdParams& p, int V, bool f32_inputs, int MT, cudaStream_t stream) {
  if (f32_inputs) {
    if (MT != 1) return cudaErrorInvalidValue;
    if (V == 16) return launch_t<16, 1, true>(p, stream);
    if (V == 32) return launch_t<32, 1, true>(p, stream);
    return cudaErrorInvalidValue;
  }
  if (MT == 0) return V == 16 ? launch_t<16, 0, false>(p, stream) : launch_t<32, 0, false>(p, stream);
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
