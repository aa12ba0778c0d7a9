// m2rnn_api.cu -- the extern "C" entry points declared in include/m2rnn.h:
// argument validation, kernel-variant dispatch, the device status word and
// the wait time limit.  Kernels live in m2rnn_fwd.cu / m2rnn_bwd.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "m2rnn.h"
#include "m2rnn_internal.h"
#include "m2rnn_check.cuh"

namespace m2rnn {
int fwd_max_consumer_warps(int V, int MT, bool f32_inputs);
}

namespace {

constexpr long long kDefaultWaitLimitNs = 2000000000LL;
std::atomic<long long> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int> g_fault_injection{0};

// Device status word, one per device image of this library.
__device__ int g_device_status[2];

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
int* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

int status_from_cuda(cudaError_t e) { return e == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA; }

// Per-device set-up: the device address of the status word and the SM count.
int device_info(int* dev_out, int** status_out, int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return M2RNN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return M2RNN_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return M2RNN_ERR_CUDA;
    g_status_ptr[dev] = static_cast<int*>(ptr);
    g_num_sms[dev] = sms;
  }
  *dev_out = dev;
  *status_out = g_status_ptr[dev];
  *sms_out = g_num_sms[dev];
  return M2RNN_OK;
}

// A tensor pointer must be 16-byte aligned device (or managed) memory of the
// current device.
int check_ptr(const void* p, int dev, bool required) {
  if (p == nullptr) return required ? M2RNN_ERR_INVALID_ARG : M2RNN_OK;
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return M2RNN_ERR_MISALIGNED;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return M2RNN_ERR_POINTER;
  }
  if (a.type == cudaMemoryTypeManaged) return M2RNN_OK;
  if (a.type != cudaMemoryTypeDevice || a.device != dev) return M2RNN_ERR_POINTER;
  return M2RNN_OK;
}

// Query/key groups of a shape (0 is read as 1).
int groups(const m2rnn_shape* s) { return s->Nq == 0 ? 1 : s->Nq; }

int check_shape(const m2rnn_shape* s) { return m2rnn::validate_shape(s); }

}  // namespace

namespace m2rnn {
int validate_shape(const m2rnn_shape* s) {
  if (s == nullptr) return M2RNN_ERR_INVALID_ARG;
  if (s->B < 1 || s->N < 1 || s->T < 0 || s->ckpt_every < 0) return M2RNN_ERR_INVALID_ARG;
  if (s->Nq < 0 || s->N % groups(s) != 0) return M2RNN_ERR_INVALID_ARG;
  if (s->in_dtype != M2RNN_F32 && s->in_dtype != M2RNN_BF16) return M2RNN_ERR_INVALID_ARG;
  if (!(s->K == 16 || s->K == 32 || s->K == 64 || s->K == 128)) return M2RNN_ERR_UNSUPPORTED_SHAPE;
  if (!(s->V == 16 || s->V == 32)) return M2RNN_ERR_UNSUPPORTED_SHAPE;
  const double elems = static_cast<double>(s->B) * s->T * s->N * s->V;
  if (elems >= 1099511627776.0) return M2RNN_ERR_UNSUPPORTED_SHAPE;  // 2^40
  if (static_cast<long long>(s->B) * s->N >= (1LL << 31)) return M2RNN_ERR_UNSUPPORTED_SHAPE;
  return M2RNN_OK;
}
}  // namespace m2rnn

namespace {

struct FwdConfig {
  int MT, WPH, G, tc;
};

constexpr size_t kSmemBudget = 220 * 1024;  // per CTA, below the 227 KB limit

// Picks rows-per-warp (MT 16-row slices) and heads per CTA.  At least ~16
// consumer warps per SM are needed to keep the SFU busy; beyond that larger
// slices amortise per-step overhead.  Heads per CTA are chosen so that the
// grid covers the SMs.
FwdConfig choose_fwd(const m2rnn_shape* s, int sms) {
  const bool f32 = s->in_dtype == M2RNN_F32;
  const int mtiles = s->K / 16;
  const long long heads = static_cast<long long>(s->B) * s->N;
  int MT = 1;
  if (!f32) {
    for (int cand : {4, 2}) {
      if (mtiles % cand != 0) continue;
      if (s->V == 32 && cand > 2) continue;
      if (heads * (mtiles / cand) >= 16LL * sms) {
        MT = cand;
        break;
      }
    }
  }
  // Tuning override: M2RNN_FWD_MT=0|1|2|4 forces the rows-per-warp variant
  // (0 = half slices of 8 rows; measured slower than full slices when all
  // of a head's warps share one SM, so never chosen automatically).
  if (const char* e = std::getenv("M2RNN_FWD_MT")) {
    const int m = std::atoi(e);
    const bool fits = m != 0 || s->K / 8 <= m2rnn::fwd_max_consumer_warps(s->V, 0, f32);
    if ((m == 0 || m == 1 || m == 2 || m == 4) && (m == 0 || mtiles % m == 0) &&
        !(f32 && m != 1) && !(s->V == 32 && m == 4) && fits)
      MT = m;
  }
  const int WPH = MT == 0 ? s->K / 8 : mtiles / MT;
  const int maxw = m2rnn::fwd_max_consumer_warps(s->V, MT, f32);
  int best = 1;
  const int hpg = s->N / groups(s);  // a CTA's heads stay inside one q/k group
  for (int G = 1; G <= s->N && G * WPH <= maxw; ++G) {
    if (hpg % G != 0) continue;
    if (m2rnn::fwd_smem_bytes(s->K, s->V, G, WPH, f32, 32) > 200 * 1024) continue;
    const long long ctas = static_cast<long long>(s->B) * (s->N / G);
    if (G == 1 || ctas >= sms) best = G;
  }
  // Tuning override: M2RNN_FWD_G=g forces g heads per CTA where it is valid.
  if (const char* e = std::getenv("M2RNN_FWD_G")) {
    const int g = std::atoi(e);
    if (g >= 1 && g <= s->N && hpg % g == 0 && g * WPH <= maxw &&
        m2rnn::fwd_smem_bytes(s->K, s->V, g, WPH, f32, 8) <= kSmemBudget)
      best = g;
  }
  int tc = 32;  // shorter ring chunks where the layout would not fit
  while (tc > 8 && m2rnn::fwd_smem_bytes(s->K, s->V, best, WPH, f32, tc) > kSmemBudget) tc /= 2;
  return {MT, WPH, best, tc};
}

// Ring chunk length of the main launch.  64 steps where the CTAs still fit
// on the SMs as they do with 32 (every CTA at once, or as many per SM): a
// consumer's waits and hand-offs at chunk boundaries then come half as often.
// M2RNN_FWD_TC=n (2..64) forces it where the layout fits.
int refine_tc(const m2rnn::FwdParams& p, const m2rnn_shape* s, int sms, const FwdConfig& cfg,
              bool f32) {
  if (const char* e = std::getenv("M2RNN_FWD_TC")) {
    const int t = std::atoi(e);
    if (t >= 2 && t <= 64 &&
        m2rnn::fwd_smem_bytes(s->K, s->V, cfg.G, cfg.WPH, f32, t) <= kSmemBudget)
      return t;
  }
  if (cfg.tc != 32 || m2rnn::fwd_smem_bytes(s->K, s->V, cfg.G, cfg.WPH, f32, 64) > kSmemBudget)
    return cfg.tc;
  m2rnn::FwdParams q = p;
  q.tc = 32;
  const int r32 = m2rnn::fwd_ctas_per_sm(q, s->V, f32, cfg.MT);
  q.tc = 64;
  const int r64 = m2rnn::fwd_ctas_per_sm(q, s->V, f32, cfg.MT);
  const long long ctas = static_cast<long long>(s->B) * p.ngroups;
  return r64 > 0 && (r64 >= r32 || static_cast<long long>(r64) * sms >= ctas) ? 64 : 32;
}

struct WavePlan {
  int B1;       // leading batch items run with the main configuration (0 = one launch)
  int tail_G;   // heads per CTA of the launch covering the remaining batch items
  int tail_tc;  // its ring chunk length
};

// Decides whether the batch items beyond whole waves of the main
// configuration should get a launch of their own with fewer heads per CTA,
// spread over all SMs, because that shortens the run.
WavePlan plan_full_waves(const m2rnn_shape* s, int sms, const FwdConfig& cfg,
                         const m2rnn::FwdParams& p, bool f32) {
  const WavePlan none{0, cfg.G, cfg.tc};
  const int R = m2rnn::fwd_ctas_per_sm(p, s->V, f32, cfg.MT);
  if (R <= 0 || s->N % cfg.G != 0) return none;
  const long long wave_heads = static_cast<long long>(sms) * R * cfg.G;
  if (wave_heads % s->N != 0) return none;
  const long long wave_b = wave_heads / s->N;
  const long long heads = static_cast<long long>(s->B) * s->N;
  if (heads <= wave_heads) return none;
  const long long B1 = (s->B / wave_b) * wave_b;
  const long long rem_heads = (s->B - B1) * s->N;
  if (rem_heads == 0) return none;
  // Cost of the remainder in "heads per SM" (time of the slowest SM).
  auto cost = [&](int G, int R_) -> long long {
    const long long ctas = rem_heads / G;
    const long long per_sm = (ctas + sms - 1) / sms;
    return per_sm <= R_ ? per_sm * G : -1;
  };
  long long best = cost(cfg.G, R);
  if (best < 0) best = ((rem_heads / cfg.G + static_cast<long long>(sms) * R - 1) /
                        (static_cast<long long>(sms) * R)) * R * cfg.G;
  int bestG = 0, bestTc = cfg.tc;
  for (int G = cfg.G - 1; G >= 1; --G) {
    if ((s->N / groups(s)) % G != 0) continue;
    // Shorter ring chunks shrink the per-CTA shared memory so that more of
    // the small CTAs fit on an SM.
    for (int tc = 32; tc >= 8; tc /= 2) {
      if (m2rnn::fwd_smem_bytes(s->K, s->V, G, p.WPH, f32, tc) > kSmemBudget) continue;
      m2rnn::FwdParams q = p;
      q.G = G;
      q.tc = tc;
      const int RG = m2rnn::fwd_ctas_per_sm(q, s->V, f32, cfg.MT);
      const long long c = RG > 0 ? cost(G, RG) : -1;
      if (c > 0 && c < best) {
        best = c;
        bestG = G;
        bestTc = tc;
      }
    }
  }
  if (bestG == 0) return none;
  return {static_cast<int>(B1), bestG, bestTc};
}

// The fused input gate's inputs (a [B,T,N], alpha and beta [N]); a null
// Gate pointer means f is given directly.
struct Gate {
  const void* a;
  const void* alpha;
  const void* beta;
};

// The readout epilogue's arguments: forward (g, w, eps; outputs out and
// rstd) and backward (g, w, the forward's y and rstd, the upstream dout;
// outputs dg and dw).  A null pointer to either struct: plain y.
struct NormFwd {
  const void* g;
  const void* w;
  float eps;
  void* out;
  float* rstd;
};
struct NormBwd {
  const void* g;
  const void* w;
  const void* y;
  const float* rstd;
  const void* dout;
  float* dg;
  float* dw;
};

// Parameters with every per-batch pointer advanced by b0 batch items.
m2rnn::FwdParams offset_batch(const m2rnn::FwdParams& p, int b0, const m2rnn_shape* s, int es) {
  m2rnn::FwdParams r = p;
  const size_t B0 = static_cast<size_t>(b0), T = s->T, N = s->N, K = s->K, V = s->V;
  const size_t Nq = static_cast<size_t>(p.Nq);
  r.q = static_cast<const char*>(p.q) + B0 * T * Nq * K * es;
  r.k = static_cast<const char*>(p.k) + B0 * T * Nq * K * es;
  r.v = static_cast<const char*>(p.v) + B0 * T * N * V * es;
  if (p.f) r.f = static_cast<const char*>(p.f) + B0 * T * N * es;
  if (p.a) r.a = static_cast<const char*>(p.a) + B0 * T * N * es;
  if (p.y) r.y = static_cast<char*>(p.y) + B0 * T * N * V * es;  // NULL: checkpoint-only run
  if (p.H0) r.H0 = p.H0 + B0 * N * K * V;
  if (p.HT) r.HT = p.HT + B0 * N * K * V;
  if (p.ckpt) r.ckpt = p.ckpt + B0 * N * static_cast<size_t>(p.nck) * K * V;
  if (p.g) r.g = static_cast<const char*>(p.g) + B0 * T * N * V * es;
  if (p.ssq) r.ssq = p.ssq + B0 * T;
  return r;
}

// Plans and launches the forward pass (pointers already validated).  y may
// be NULL (checkpoint-only runs for the backward pass).
int run_fwd(const m2rnn_shape* s, const void* q, const void* k, const void* v, const void* f,
            const Gate* gate, const void* W, const void* w_r, const float* H0, void* y,
            float* H_T, float* ckpt, cudaStream_t st, int* status, int sms,
            const NormFwd* nf = nullptr) {
  const bool want_ckpt = ckpt != nullptr && s->ckpt_every > 0 && s->T > 0;
  const bool f32 = s->in_dtype == M2RNN_F32;
  const FwdConfig cfg = choose_fwd(s, sms);
  m2rnn::FwdParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.f = f;
  p.W = W;
  p.w_r = w_r;
  p.H0 = H0;
  p.y = y;
  p.HT = H_T;
  p.ckpt = want_ckpt ? ckpt : nullptr;  // NULL: no checkpoints written
  p.B = s->B;
  p.T = s->T;
  p.N = s->N;
  p.K = s->K;
  p.C = want_ckpt ? s->ckpt_every : 0;
  p.nck = static_cast<int>(m2rnn_num_checkpoints(s));
  p.G = cfg.G;
  p.WPH = cfg.WPH;
  p.ngroups = (s->N + cfg.G - 1) / cfg.G;
  p.tc = cfg.tc;
  p.status = status;
  p.wait_limit_ns = static_cast<unsigned long long>(g_wait_limit_ns.load());
  p.inject_stall = g_fault_injection.load();
  p.Nq = groups(s);
  if (gate != nullptr) {
    p.f = nullptr;
    p.a = gate->a;
    p.alpha = gate->alpha;
    p.beta = gate->beta;
    p.gated = 1;
  }
  if (nf != nullptr) {  // the epilogue adds sum (y g)^2 per token into rstd
    p.g = nf->g;
    p.ssq = nf->rstd;
    p.norm = 1;
  }
  p.tc = refine_tc(p, s, sms, cfg, f32);

  // One-wave kernel (opt-in, M2RNN_FWD_WAVE=1): every head resident at once,
  // G = ceil(B N / SMs) heads per CTA over the flattened (b, n) order, one
  // warp per head; M2RNN_FWD_WAVE_G forces G.  Measured slower than the
  // two-launch plan below at B=64, T=4096, N=32 (3.07 against 2.78 ms): one
  // warp's four 16-row tiles follow each other in its in-order instruction
  // stream, and 14 such warps per SM hide less latency than 16 warps of two
  // tiles.  It stays for A/B measurement and is tested like the others.
  if (!f32 && s->V == 16 && s->K == 64 && nf == nullptr && groups(s) == 1) {
    const long long heads = static_cast<long long>(s->B) * s->N;
    int Gw = static_cast<int>((heads + sms - 1) / sms);
    const char* e = std::getenv("M2RNN_FWD_WAVE");
    const bool use = e != nullptr && e[0] == '1';
    if (const char* eg = std::getenv("M2RNN_FWD_WAVE_G")) Gw = std::atoi(eg);
    if (use && Gw >= 1 && Gw <= m2rnn::fwd_wave_max_heads() && Gw <= s->N) {
      m2rnn::FwdParams pw = p;
      pw.G = Gw;
      pw.WPH = 1;
      pw.ngroups = 0;
      int tc = 32;
      while (tc > 8 && m2rnn::fwd_wave_smem_bytes(64, Gw, tc) > kSmemBudget) tc /= 2;
      pw.tc = tc;
      return status_from_cuda(m2rnn::launch_fwd_wave(pw, st));
    }
  }

  // Wave planning.  All CTAs of a launch run equally long, so when the heads
  // fill some whole waves plus a remainder, the remainder's batch items get a
  // second launch with fewer heads per CTA, spread over all SMs.
  // M2RNN_FWD_ONE_LAUNCH=1 disables the split (A/B measurement).
  const char* one = std::getenv("M2RNN_FWD_ONE_LAUNCH");
  const WavePlan plan = (one && one[0] == '1') ? WavePlan{0, cfg.G, cfg.tc}
                                               : plan_full_waves(s, sms, cfg, p, f32);
  const int B1 = plan.B1;
  if (B1 <= 0 || B1 >= s->B)
    return status_from_cuda(m2rnn::launch_fwd(p, s->V, f32, cfg.MT, st));
  m2rnn::FwdParams p1 = p;
  p1.B = B1;
  cudaError_t e = m2rnn::launch_fwd(p1, s->V, f32, cfg.MT, st);
  if (e != cudaSuccess) return M2RNN_ERR_CUDA;
  m2rnn::FwdParams p2 = offset_batch(p, B1, s, f32 ? 4 : 2);
  p2.B = s->B - B1;
  p2.G = plan.tail_G;
  p2.ngroups = (s->N + p2.G - 1) / p2.G;
  p2.tc = plan.tail_tc;
  return status_from_cuda(m2rnn::launch_fwd(p2, s->V, f32, cfg.MT, st));
}

// ---- backward planning ------------------------------------------------------

// Longest checkpoint interval the backward kernel takes directly; longer ones
// are re-checkpointed into the workspace at kBwdDefaultC.
constexpr int kBwdMaxC = 128;

// Interval the backward kernel works with, and whether it needs its own
// checkpoints (in the workspace).  Longer intervals are cut into the largest
// divisor of the interval that the kernel takes, so every caller checkpoint
// stays an interval boundary.
int bwd_interval(const m2rnn_shape* s, bool ckpt_given, bool* own_ckpt) {
  const int C = s->ckpt_every;
  const bool direct = ckpt_given && C <= kBwdMaxC;
  *own_ckpt = !direct;
  if (C <= kBwdMaxC) return C;
  for (int d = kBwdMaxC; d > 1; --d)
    if (C % d == 0) return d;
  return 1;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace bytes of the readout epilogue's dy (input dtype, [B,T,N,V]).
size_t norm_dy_bytes(const m2rnn_shape* s) {
  return align256(static_cast<size_t>(s->B) * s->T * s->N * s->V *
                  (s->in_dtype == M2RNN_F32 ? 4 : 2));
}

// Picks the kernel (pipelined where it exists for V, else serial) and the
// warps per CTA (16 rows each) for the fewest waves; ties go to the
// pipelined kernel, then to more rows per CTA (fewer cross-CTA reductions).
// M2RNN_BWD_KERNEL=0 (serial) or 1 (pipelined) forces the kernel and
// M2RNN_BWD_WPC the warps per CTA.
bool choose_bwd(m2rnn::BwdParams& p, int V, bool f32, int sms) {
  const int mtiles = p.K / 16;
  int kinds[2] = {1, 0}, nkinds = 2;
  if (const char* env = std::getenv("M2RNN_BWD_KERNEL")) {
    kinds[0] = std::atoi(env);
    nkinds = 1;
    if (kinds[0] != 0 && kinds[0] != 1) return false;
  }
  if (!m2rnn::bwd_has_pipe(V)) {
    kinds[0] = 0;
    nkinds = 1;
  }
  int force_w = 0;
  if (const char* env = std::getenv("M2RNN_BWD_WPC")) force_w = std::atoi(env);
  int best_w = 0, best_pipe = 0;
  long long best_waves = 0;
  for (int ki = 0; ki < nkinds; ++ki) {
    const int pipe = kinds[ki];
    for (int w = mtiles < 8 ? mtiles : 8; w >= 1; w /= 2) {
      if (mtiles % w != 0 || (force_w > 0 && w != force_w)) continue;
      const size_t smem = pipe ? m2rnn::bwd_pipe_smem_bytes(V, p.C, w, f32, p.gated != 0)
                               : m2rnn::bwd_smem_bytes(V, p.C, p.S2, w, f32);
      if (smem > kSmemBudget) continue;
      m2rnn::BwdParams q = p;
      q.WPC = w;
      q.nslices = mtiles / w;
      q.pipe = pipe;
      const int R = pipe ? m2rnn::bwd_pipe_ctas_per_sm(q, V, f32) : m2rnn::bwd_ctas_per_sm(q, V, f32);
      if (R <= 0) continue;
      const long long ctas = static_cast<long long>(p.B) * p.N * q.nslices;
      const long long waves =
          (ctas + static_cast<long long>(sms) * R - 1) / (static_cast<long long>(sms) * R);
      if (best_w == 0 || waves < best_waves) {
        best_w = w;
        best_pipe = pipe;
        best_waves = waves;
      }
    }
  }
  if (best_w == 0) return false;
  p.WPC = best_w;
  p.nslices = mtiles / best_w;
  p.pipe = best_pipe;
  return true;
}

// Decode entry: validation, then the decode kernel.  gate = NULL: f is given.
int decode_impl(const m2rnn_shape* s, const void* q, const void* k, const void* v, const void* f,
                const Gate* gate, const void* W, const void* w_r, const float* H_in, float* H_out,
                void* y, void* stream) {
  int rc = check_shape(s);
  if (rc != M2RNN_OK) return rc;
  if (s->T != 1) return M2RNN_ERR_INVALID_ARG;
  int dev, sms;
  int* status;
  rc = device_info(&dev, &status, &sms);
  if (rc != M2RNN_OK) return rc;
  const void* req[] = {q, k, v, gate ? gate->a : f, W, w_r, H_in, H_out, y};
  for (const void* p : req)
    if ((rc = check_ptr(p, dev, true)) != M2RNN_OK) return rc;
  if (gate != nullptr) {
    if ((rc = check_ptr(gate->alpha, dev, true)) != M2RNN_OK) return rc;
    if ((rc = check_ptr(gate->beta, dev, true)) != M2RNN_OK) return rc;
  }
  if (H_out != H_in) {  // distinct state buffers must not overlap
    const size_t bytes = static_cast<size_t>(s->B) * s->N * s->K * s->V * sizeof(float);
    const uintptr_t a = reinterpret_cast<uintptr_t>(H_in), b = reinterpret_cast<uintptr_t>(H_out);
    if (a < b + bytes && b < a + bytes) return M2RNN_ERR_INVALID_ARG;
  }
  m2rnn::DecodeParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.f = f;
  p.W = W;
  p.w_r = w_r;
  p.H_in = H_in;
  p.H_out = H_out;
  p.y = y;
  p.B = s->B;
  p.N = s->N;
  p.K = s->K;
  p.Nq = groups(s);
  p.status = status;
  if (gate != nullptr) {
    p.a = gate->a;
    p.alpha = gate->alpha;
    p.beta = gate->beta;
    p.gated = 1;
  }
  return status_from_cuda(m2rnn::launch_decode(p, s->V, s->in_dtype == M2RNN_F32,
                                               static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int m2rnn_version(void) { return 201; }

int m2rnn_checked(void) { return M2RNN_CHECK ? 1 : 0; }

const char* m2rnn_status_string(int status) {
  switch (status) {
    case M2RNN_OK: return "ok";
    case M2RNN_ERR_INVALID_ARG: return "invalid argument (null required pointer, negative size or bad dtype)";
    case M2RNN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (K must be 16/32/64/128, V 16/32)";
    case M2RNN_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case M2RNN_ERR_POINTER: return "pointer is not device memory of the current device";
    case M2RNN_ERR_WORKSPACE: return "workspace missing or too small";
    case M2RNN_ERR_CUDA: return "CUDA runtime error";
    case M2RNN_ERR_TIMEOUT: return "a kernel wait exceeded its time limit";
    case M2RNN_ERR_BOUNDS: return "a kernel index was outside its array (checked build; access skipped)";
    default: return "unknown status";
  }
}

size_t m2rnn_num_checkpoints(const m2rnn_shape* s) {
  if (s == nullptr || s->ckpt_every <= 0 || s->T <= 0) return 0;
  return static_cast<size_t>((s->T + s->ckpt_every - 1) / s->ckpt_every);
}

int m2rnn_set_wait_limit_ns(long long limit_ns) {
  g_wait_limit_ns.store(limit_ns > 0 ? limit_ns : kDefaultWaitLimitNs);
  return M2RNN_OK;
}

int m2rnn_set_fault_injection(int mode) {
  if (mode != 0 && mode != 1) return M2RNN_ERR_INVALID_ARG;
  g_fault_injection.store(mode);
  return M2RNN_OK;
}

int m2rnn_device_status(int* status, int* detail, int clear, void* stream) {
  if (status == nullptr) return M2RNN_ERR_INVALID_ARG;
  int dev, sms;
  int* sp;
  int rc = device_info(&dev, &sp, &sms);
  if (rc != M2RNN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return M2RNN_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpy(h, sp, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return M2RNN_ERR_CUDA;
  *status = h[0];
  if (detail) *detail = h[1];
  if (clear && cudaMemset(sp, 0, sizeof(h)) != cudaSuccess) return M2RNN_ERR_CUDA;
  return M2RNN_OK;
}

int m2rnn_decode(const m2rnn_shape* s, const void* q, const void* k, const void* v, const void* f,
                 const void* W, const void* w_r, const float* H_in, float* H_out, void* y,
                 void* stream) {
  return decode_impl(s, q, k, v, f, nullptr, W, w_r, H_in, H_out, y, stream);
}

int m2rnn_decode_gated(const m2rnn_shape* s, const void* q, const void* k, const void* v,
                       const void* a, const void* alpha, const void* beta, const void* W,
                       const void* w_r, const float* H_in, float* H_out, void* y, void* stream) {
  const Gate gate{a, alpha, beta};
  return decode_impl(s, q, k, v, nullptr, &gate, W, w_r, H_in, H_out, y, stream);
}

}  // extern "C"

namespace {

// Forward entry: validation, then run_fwd.  gate = NULL: f is given.
int fwd_impl(const m2rnn_shape* s, const void* q, const void* k, const void* v, const void* f,
             const Gate* gate, const void* W, const void* w_r, const float* H0, void* y,
             float* H_T, float* ckpt, void* stream, const NormFwd* nf = nullptr) {
  int rc = check_shape(s);
  if (rc != M2RNN_OK) return rc;
  int dev, sms;
  int* status;
  rc = device_info(&dev, &status, &sms);
  if (rc != M2RNN_OK) return rc;
  const bool want_ckpt = s->ckpt_every > 0 && s->T > 0;
  if ((rc = check_ptr(H0, dev, false)) != M2RNN_OK) return rc;
  if ((rc = check_ptr(H_T, dev, false)) != M2RNN_OK) return rc;
  if (gate != nullptr) {  // per-head gate parameters
    if ((rc = check_ptr(gate->alpha, dev, true)) != M2RNN_OK) return rc;
    if ((rc = check_ptr(gate->beta, dev, true)) != M2RNN_OK) return rc;
  }
  if (nf != nullptr) {
    if (!(nf->eps >= 0.f)) return M2RNN_ERR_INVALID_ARG;  // also rejects NaN
    if ((rc = check_ptr(nf->w, dev, true)) != M2RNN_OK) return rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t state_bytes = static_cast<size_t>(s->B) * s->N * s->K * s->V * sizeof(float);
  if (s->T == 0) {  // empty sequences: the [B,0,...] tensors may have no storage
    if (H_T == nullptr) return M2RNN_OK;
    return status_from_cuda(H0 ? cudaMemcpyAsync(H_T, H0, state_bytes, cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(H_T, 0, state_bytes, st));
  }
  const void* req[] = {q, k, v, gate ? gate->a : f, W, w_r, y};
  for (const void* p : req)
    if ((rc = check_ptr(p, dev, true)) != M2RNN_OK) return rc;
  if ((rc = check_ptr(ckpt, dev, false)) != M2RNN_OK) return rc;
  if (nf == nullptr)
    return run_fwd(s, q, k, v, f, gate, W, w_r, H0, y, H_T, want_ckpt ? ckpt : nullptr, st,
                   status, sms);
  const void* nreq[] = {nf->g, nf->out, nf->rstd};
  for (const void* p : nreq)
    if ((rc = check_ptr(p, dev, true)) != M2RNN_OK) return rc;
  const long long rows = static_cast<long long>(s->B) * s->T;
  if (cudaMemsetAsync(nf->rstd, 0, rows * sizeof(float), st) != cudaSuccess) return M2RNN_ERR_CUDA;
  rc = run_fwd(s, q, k, v, f, gate, W, w_r, H0, y, H_T, want_ckpt ? ckpt : nullptr, st, status,
               sms, nf);
  if (rc != M2RNN_OK) return rc;
  m2rnn::NormParams np;
  np.rows = rows;
  np.d = s->N * s->V;
  np.eps = nf->eps;
  np.y = y;
  np.g = nf->g;
  np.w = nf->w;
  np.rstd = nf->rstd;
  np.out = nf->out;
  np.dout = nullptr;
  np.dy = nullptr;
  np.dg = nullptr;
  np.dw = nullptr;
  np.status = status;
  return status_from_cuda(m2rnn::launch_norm_fwd(np, s->in_dtype == M2RNN_F32, sms, st));
}

// Backward entry.  gate = NULL: f is given and dfa receives dL/df; otherwise
// dfa receives dL/da and dalpha, dbeta the gate parameters' gradients.
int bwd_impl(const m2rnn_shape* s, const void* q, const void* k, const void* v, const void* f,
             const Gate* gate, const void* W, const void* w_r, const float* H0, const float* ckpt,
             const void* dy, const float* dH_T, float* dq, float* dk, float* dv, float* dfa,
             float* dalpha, float* dbeta, float* dW, float* dw_r, float* dH0, float* dckpt,
             void* workspace, size_t ws_bytes, void* stream, const NormBwd* nb = nullptr) {
  int rc = check_shape(s);
  if (rc != M2RNN_OK) return rc;
  if (s->ckpt_every <= 0) return M2RNN_ERR_INVALID_ARG;
  int dev, sms;
  int* status;
  rc = device_info(&dev, &status, &sms);
  if (rc != M2RNN_OK) return rc;
  const void* always[] = {W, w_r, dW, dw_r};
  for (const void* x : always)
    if ((rc = check_ptr(x, dev, true)) != M2RNN_OK) return rc;
  if (gate != nullptr) {
    const void* gp[] = {gate->alpha, gate->beta, dalpha, dbeta};
    for (const void* x : gp)
      if ((rc = check_ptr(x, dev, true)) != M2RNN_OK) return rc;
  }
  const void* optional[] = {H0, dH_T, dH0, dckpt};
  for (const void* x : optional)
    if ((rc = check_ptr(x, dev, false)) != M2RNN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool f32 = s->in_dtype == M2RNN_F32;
  const size_t NV = static_cast<size_t>(s->N) * s->V;
  const size_t state_bytes = static_cast<size_t>(s->B) * s->N * s->K * s->V * sizeof(float);
  if (cudaMemsetAsync(dW, 0, NV * s->V * sizeof(float), st) != cudaSuccess ||
      cudaMemsetAsync(dw_r, 0, NV * sizeof(float), st) != cudaSuccess)
    return M2RNN_ERR_CUDA;
  if (gate != nullptr && (cudaMemsetAsync(dalpha, 0, s->N * sizeof(float), st) != cudaSuccess ||
                          cudaMemsetAsync(dbeta, 0, s->N * sizeof(float), st) != cudaSuccess))
    return M2RNN_ERR_CUDA;
  if (nb != nullptr) {
    if ((rc = check_ptr(nb->w, dev, true)) != M2RNN_OK) return rc;
    if ((rc = check_ptr(nb->dw, dev, true)) != M2RNN_OK) return rc;
    if (cudaMemsetAsync(nb->dw, 0, NV * sizeof(float), st) != cudaSuccess) return M2RNN_ERR_CUDA;
  }
  if (s->T == 0) {  // no steps: dH0 = dH_T
    if (dH0 == nullptr) return M2RNN_OK;
    return status_from_cuda(dH_T ? cudaMemcpyAsync(dH0, dH_T, state_bytes, cudaMemcpyDeviceToDevice, st)
                                 : cudaMemsetAsync(dH0, 0, state_bytes, st));
  }
  if (nb != nullptr) {  // dy from the readout epilogue's gradient, into the workspace
    const void* nreq[] = {nb->g, nb->y, nb->rstd, nb->dout, nb->dg};
    for (const void* x : nreq)
      if ((rc = check_ptr(x, dev, true)) != M2RNN_OK) return rc;
    const size_t dy_bytes = norm_dy_bytes(s);
    if (workspace == nullptr || ws_bytes < dy_bytes) return M2RNN_ERR_WORKSPACE;
    if ((rc = check_ptr(workspace, dev, true)) != M2RNN_OK) return rc;
    m2rnn::NormParams np;
    np.rows = static_cast<long long>(s->B) * s->T;
    np.d = s->N * s->V;
    np.eps = 0.f;
    np.y = nb->y;
    np.g = nb->g;
    np.w = nb->w;
    np.rstd = const_cast<float*>(nb->rstd);  // read only in the backward kernel
    np.out = nullptr;
    np.dout = nb->dout;
    np.dy = workspace;
    np.dg = nb->dg;
    np.dw = nb->dw;
    np.status = status;
    if (m2rnn::launch_norm_bwd(np, f32, sms, st) != cudaSuccess) return M2RNN_ERR_CUDA;
    dy = workspace;
    workspace = static_cast<char*>(workspace) + dy_bytes;
    ws_bytes -= dy_bytes;
  }
  const void* req[] = {q, k, v, gate ? gate->a : f, dy, dq, dk, dv, dfa};
  for (const void* x : req)
    if ((rc = check_ptr(x, dev, true)) != M2RNN_OK) return rc;
  if ((rc = check_ptr(ckpt, dev, false)) != M2RNN_OK) return rc;
  bool own = false;
  const int C = bwd_interval(s, ckpt != nullptr, &own);
  const size_t need = m2rnn_bwd_workspace_size(s, ckpt != nullptr);
  if (need > 0) {
    if (workspace == nullptr || ws_bytes < need) return M2RNN_ERR_WORKSPACE;
    if (nb == nullptr && (rc = check_ptr(workspace, dev, true)) != M2RNN_OK) return rc;
  }
  const float* ck = ckpt;
  if (own) {  // checkpoints at interval C into the workspace (no y written)
    m2rnn_shape sf = *s;
    sf.ckpt_every = C;
    rc = run_fwd(&sf, q, k, v, f, gate, W, w_r, H0, nullptr, nullptr,
                 static_cast<float*>(workspace), st, status, sms);
    if (rc != M2RNN_OK) return rc;
    ck = static_cast<const float*>(workspace);
  }
  m2rnn::BwdParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.f = gate ? nullptr : f;
  p.W = W;
  p.w_r = w_r;
  p.ckpt = ck;
  p.dy = dy;
  p.dHT = dH_T;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.df = dfa;
  p.dW = dW;
  p.dw_r = dw_r;
  p.dH0 = dH0;
  p.dckpt = dckpt;
  p.status = status;
  if (gate != nullptr) {
    p.a = gate->a;
    p.alpha = gate->alpha;
    p.beta = gate->beta;
    p.gated = 1;
    p.dalpha = dalpha;
    p.dbeta = dbeta;
  }
  p.Nq = groups(s);
  p.dck_ratio = s->ckpt_every / C;
  p.dck_n = static_cast<int>(m2rnn_num_checkpoints(s));
  p.B = s->B;
  p.T = s->T;
  p.N = s->N;
  p.K = s->K;
  p.C = C;
  p.nck = (s->T + C - 1) / C;
  p.S2 = m2rnn::bwd_sub_len(s->V, f32);
  p.WPC = 1;
  p.nslices = s->K / 16;
  p.pipe = 0;
  if (!choose_bwd(p, s->V, f32, sms)) return M2RNN_ERR_UNSUPPORTED_SHAPE;
  const size_t BT = static_cast<size_t>(s->B) * s->T;
  const size_t qk_elems = BT * groups(s) * s->K;
  if (cudaMemsetAsync(dq, 0, qk_elems * sizeof(float), st) != cudaSuccess ||
      cudaMemsetAsync(dk, 0, qk_elems * sizeof(float), st) != cudaSuccess)
    return M2RNN_ERR_CUDA;
  if (p.nslices > 1 && (cudaMemsetAsync(dv, 0, BT * NV * sizeof(float), st) != cudaSuccess ||
                        cudaMemsetAsync(dfa, 0, BT * s->N * sizeof(float), st) != cudaSuccess))
    return M2RNN_ERR_CUDA;
  return status_from_cuda(p.pipe ? m2rnn::launch_bwd_pipe(p, s->V, f32, st)
                                : m2rnn::launch_bwd(p, s->V, f32, st));
}

// f or the gate (exactly one of the two forms).
int pick_f(const void* f, const void* a, const void* alpha, const void* beta, Gate* gate,
           const Gate** gp) {
  if (f != nullptr && a == nullptr && alpha == nullptr && beta == nullptr) {
    *gp = nullptr;
    return M2RNN_OK;
  }
  if (f == nullptr && a != nullptr && alpha != nullptr && beta != nullptr) {
    *gate = Gate{a, alpha, beta};
    *gp = gate;
    return M2RNN_OK;
  }
  return M2RNN_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

int m2rnn_fwd(const m2rnn_shape* s, const void* q, const void* k, const void* v, const void* f,
              const void* W, const void* w_r, const float* H0, void* y, float* H_T, float* ckpt,
              void* stream) {
  return fwd_impl(s, q, k, v, f, nullptr, W, w_r, H0, y, H_T, ckpt, stream);
}

int m2rnn_fwd_gated(const m2rnn_shape* s, const void* q, const void* k, const void* v,
                    const void* a, const void* alpha, const void* beta, const void* W,
                    const void* w_r, const float* H0, void* y, float* H_T, float* ckpt,
                    void* stream) {
  const Gate gate{a, alpha, beta};
  return fwd_impl(s, q, k, v, nullptr, &gate, W, w_r, H0, y, H_T, ckpt, stream);
}

size_t m2rnn_bwd_workspace_size(const m2rnn_shape* s, int ckpt_given) {
  if (check_shape(s) != M2RNN_OK || s->ckpt_every <= 0 || s->T == 0) return 0;
  bool own = false;
  const int C = bwd_interval(s, ckpt_given != 0, &own);
  if (!own) return 0;
  const size_t nck = static_cast<size_t>((s->T + C - 1) / C);
  return align256(static_cast<size_t>(s->B) * s->N * nck * s->K * s->V * sizeof(float));
}

int m2rnn_bwd(const m2rnn_shape* s, const void* q, const void* k, const void* v, const void* f,
              const void* W, const void* w_r, const float* H0, const float* ckpt, const void* dy,
              const float* dH_T, float* dq, float* dk, float* dv, float* df, float* dW, float* dw_r,
              float* dH0, float* dckpt, void* workspace, size_t ws_bytes, void* stream) {
  return bwd_impl(s, q, k, v, f, nullptr, W, w_r, H0, ckpt, dy, dH_T, dq, dk, dv, df, nullptr,
                  nullptr, dW, dw_r, dH0, dckpt, workspace, ws_bytes, stream);
}

int m2rnn_bwd_gated(const m2rnn_shape* s, const void* q, const void* k, const void* v,
                    const void* a, const void* alpha, const void* beta, const void* W,
                    const void* w_r, const float* H0, const float* ckpt, const void* dy,
                    const float* dH_T, float* dq, float* dk, float* dv, float* da, float* dalpha,
                    float* dbeta, float* dW, float* dw_r, float* dH0, float* dckpt,
                    void* workspace, size_t ws_bytes, void* stream) {
  const Gate gate{a, alpha, beta};
  return bwd_impl(s, q, k, v, nullptr, &gate, W, w_r, H0, ckpt, dy, dH_T, dq, dk, dv, da, dalpha,
                  dbeta, dW, dw_r, dH0, dckpt, workspace, ws_bytes, stream);
}

int m2rnn_fwd_norm(const m2rnn_shape* s, const void* q, const void* k, const void* v,
                   const void* f, const void* a, const void* alpha, const void* beta,
                   const void* W, const void* w_r, const float* H0, const void* g,
                   const void* w_norm, float eps, void* y, void* out, float* rstd, float* H_T,
                   float* ckpt, void* stream) {
  Gate gate;
  const Gate* gp = nullptr;
  int rc = pick_f(f, a, alpha, beta, &gate, &gp);
  if (rc != M2RNN_OK) return rc;
  const NormFwd nf{g, w_norm, eps, out, rstd};
  return fwd_impl(s, q, k, v, f, gp, W, w_r, H0, y, H_T, ckpt, stream, &nf);
}

size_t m2rnn_bwd_norm_workspace_size(const m2rnn_shape* s, int ckpt_given) {
  if (check_shape(s) != M2RNN_OK || s->ckpt_every <= 0 || s->T == 0) return 0;
  return norm_dy_bytes(s) + m2rnn_bwd_workspace_size(s, ckpt_given);
}

int m2rnn_bwd_norm(const m2rnn_shape* s, const void* q, const void* k, const void* v,
                   const void* f, const void* a, const void* alpha, const void* beta,
                   const void* W, const void* w_r, const float* H0, const float* ckpt,
                   const void* g, const void* w_norm, const void* y, const float* rstd,
                   const void* dout, const float* dH_T, float* dq, float* dk, float* dv,
                   float* df, float* dalpha, float* dbeta, float* dW, float* dw_r, float* dg,
                   float* dw_norm, float* dH0, float* dckpt, void* workspace, size_t ws_bytes,
                   void* stream) {
  Gate gate;
  const Gate* gp = nullptr;
  int rc = pick_f(f, a, alpha, beta, &gate, &gp);
  if (rc != M2RNN_OK) return rc;
  const NormBwd nb{g, w_norm, y, rstd, dout, dg, dw_norm};
  return bwd_impl(s, q, k, v, f, gp, W, w_r, H0, ckpt, nullptr, dH_T, dq, dk, dv, df, dalpha,
                  dbeta, dW, dw_r, dH0, dckpt, workspace, ws_bytes, stream, &nb);
}

}  // extern "C"
