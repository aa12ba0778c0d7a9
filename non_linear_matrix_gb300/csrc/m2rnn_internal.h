// m2rnn_internal.h -- launch parameters shared by the C-ABI layer and the
// kernel translation units (host + device).  Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "m2rnn.h"

namespace m2rnn {

// Host-side validation of a shape (the checks every entry point starts
// with): M2RNN_OK or the status to return.  Makes no CUDA call.
int validate_shape(const m2rnn_shape* s);

// Device status word: [0] = first recorded m2rnn_status (0 = OK),
// [1] = location code of the wait that gave up.
enum WaitSite : int {
  SITE_FWD_PRODUCER = 1,
  SITE_FWD_EPILOGUE = 2,
  SITE_FWD_CONSUMER = 3,
  SITE_FWD_DRAIN = 4,
};

constexpr int kStatusTimeout = -7;  // == M2RNN_ERR_TIMEOUT
constexpr int kStatusBounds = -8;   // == M2RNN_ERR_BOUNDS (checked build only)

// Location codes of the checked build's index checks (status word [1]).
enum CheckSite : int {
  CHK_FWD_QK = 101,     // q, k staging copies
  CHK_FWD_V = 102,      // v staging copies
  CHK_FWD_F = 103,      // f (or the gate's a) loads
  CHK_FWD_Y = 104,      // y stores
  CHK_FWD_G = 105,      // readout epilogue: g loads
  CHK_FWD_SSQ = 106,    // readout epilogue: sum-of-squares atomics
  CHK_FWD_H0 = 107,     // H0 loads
  CHK_FWD_HT = 108,     // H_T stores
  CHK_FWD_CKPT = 109,   // checkpoint stores
  CHK_FWD_PARAM = 110,  // W, w_r, alpha, beta loads
  CHK_BWD_IN = 201,     // q, k, v, dy, f (or a) loads
  CHK_BWD_CKPT = 202,   // checkpoint loads
  CHK_BWD_DQK = 203,    // dq, dk reductions
  CHK_BWD_DV = 204,     // dv stores / reductions
  CHK_BWD_DF = 205,     // df (or da) stores / reductions
  CHK_BWD_DCKPT = 206,  // dckpt stores
  CHK_BWD_DH0 = 207,    // dH0 stores
  CHK_BWD_DPARAM = 208, // dW, dw_r, dalpha, dbeta reductions
  CHK_BWD_DHT = 209,    // dH_T loads
  CHK_BWD_PARAM = 210,  // W, w_r, alpha, beta loads
  CHK_DEC_IN = 301,     // q, k, v, f (or a), W, w_r, alpha, beta loads
  CHK_DEC_STATE = 302,  // state loads and stores
  CHK_DEC_Y = 303,      // y stores
  CHK_NORM_IN = 401,    // y, g, w, dout, rstd loads
  CHK_NORM_OUT = 402,   // out, rstd, dy, dg stores, dw reductions
};

struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* f;
  const void* W;
  const void* w_r;
  const float* H0;  // nullable
  void* y;      // nullable inside the library (checkpoint-only runs)
  float* HT;    // nullable
  float* ckpt;  // nullable
  int B, T, N, K;
  int C;        // checkpoint interval (0 = none)
  int nck;      // checkpoints per (b, n)
  int G;        // heads per CTA
  int WPH;      // consumer warps per head
  int ngroups;  // ceil(N / G)
  int tc;       // time steps per shared-memory ring chunk (2..32)
  int* status;
  unsigned long long wait_limit_ns;
  int inject_stall;  // test hook: 1 = the producer issues nothing
  int Nq = 1;        // query/key groups: q, k are [B,T,Nq,K], head n reads n / (N / Nq)
  // fused input gate (gated = 1): f = exp(-alpha softplus(a + beta)) from
  // a [B,T,N] and alpha, beta [N] (input dtype) instead of f
  const void* a = nullptr;
  const void* alpha = nullptr;
  const void* beta = nullptr;
  int gated = 0;
  // readout epilogue (norm = 1): the epilogue adds sum (y (.) g)^2 of its
  // heads for every token into ssq [B,T] (zeroed by the caller); g is [B,T,N,V]
  const void* g = nullptr;
  float* ssq = nullptr;
  int norm = 0;
};

struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* f;
  const void* W;
  const void* w_r;
  const float* ckpt;  // [B,N,nck,K,V]
  const void* dy;
  const float* dHT;   // nullable
  float* dq;          // accumulated with reductions: zeroed by the caller
  float* dk;          //   "
  float* dv;          // stored (nslices == 1) or accumulated (zeroed)
  float* df;          //   "
  float* dW;          // accumulated (zeroed)
  float* dw_r;        // accumulated (zeroed)
  float* dH0;         // nullable
  float* dckpt;       // nullable: dL/dH at every dck_ratio-th interval start
  int dck_ratio;      // user checkpoint interval / C
  int dck_n;          // user checkpoints per (b, n)
  int B, T, N, K;
  int C;        // checkpoint interval
  int nck;      // checkpoints per (b, n)
  int WPC;      // warps per CTA (16 rows each)
  int nslices;  // K / (16 * WPC)
  int S2;       // sub-interval length of the recomputation (= bwd_sub_len)
  int pipe;     // 1: the pipelined kernel (m2rnn_bwd_pipe.cu, V = 16); 0: the
                // serial one (m2rnn_bwd.cu)
  int Nq = 1;   // query/key groups (q, k, dq, dk are [B,T,Nq,K])
  // fused input gate (gated = 1): f from a, alpha, beta as in FwdParams; df
  // then receives dL/da, and dalpha, dbeta [N] (zeroed by the caller) are
  // accumulated
  const void* a = nullptr;
  const void* alpha = nullptr;
  const void* beta = nullptr;
  int gated = 0;
  float* dalpha = nullptr;
  float* dbeta = nullptr;
  int* status = nullptr;  // device status word (index checks of the checked build)
};

cudaError_t launch_bwd(const BwdParams& p, int V, bool f32_inputs, cudaStream_t stream);
int bwd_ctas_per_sm(const BwdParams& p, int V, bool f32_inputs);
size_t bwd_smem_bytes(int V, int C, int S2, int WPC, bool f32_inputs);

// Pipelined backward kernel.
bool bwd_has_pipe(int V);
size_t bwd_pipe_smem_bytes(int V, int C, int WPC, bool f32_inputs, bool gated);
int bwd_pipe_ctas_per_sm(const BwdParams& p, int V, bool f32_inputs);
cudaError_t launch_bwd_pipe(const BwdParams& p, int V, bool f32_inputs, cudaStream_t stream);
int bwd_sub_len(int V, bool f32_inputs);  // sub-interval length of the variant

// Single-step decode (m2rnn_decode.cu).
struct DecodeParams {
  const void* q;      // [B,Nq,K]
  const void* k;      // [B,Nq,K]
  const void* v;      // [B,N,V]
  const void* f;      // [B,N]
  const void* W;      // [N,V,V]
  const void* w_r;    // [N,V]
  const float* H_in;  // [B,N,K,V]
  float* H_out;       // [B,N,K,V], may equal H_in
  void* y;            // [B,N,V]
  int B, N, K;
  int Nq = 1;         // query/key groups (q, k are [B,Nq,K])
  // fused input gate (gated = 1): f from a [B,N] and alpha, beta [N]
  const void* a = nullptr;
  const void* alpha = nullptr;
  const void* beta = nullptr;
  int gated = 0;
  int* status = nullptr;  // device status word (index checks of the checked build)
};
cudaError_t launch_decode(const DecodeParams& p, int V, bool f32_inputs, cudaStream_t stream);

// Readout epilogue kernels (m2rnn_norm.cu).  Forward: turns the per-token
// sums of squares ssq [T_all] into rstd = (ssq / d + eps)^(-1/2) in place and
// writes out = w (.) y (.) g rstd.  Backward: from dout, y, g, w and rstd,
// writes dy (input dtype) and dg (fp32) and adds sum dout (.) y (.) g rstd into
// dw (fp32, zeroed by the caller).  Tokens are rows of d features.
struct NormParams {
  long long rows;   // B * T
  int d;            // N * V features per token
  float eps;
  const void* y;    // [rows][d] input dtype
  const void* g;    // [rows][d]
  const void* w;    // [d]
  float* rstd;      // [rows] (forward: holds ssq on entry)
  void* out;        // forward: [rows][d] input dtype
  const void* dout; // backward: [rows][d] input dtype
  void* dy;         // backward: [rows][d] input dtype
  float* dg;        // backward: [rows][d]
  float* dw;        // backward: [d]
  int* status = nullptr;  // device status word (index checks of the checked build)
};
cudaError_t launch_norm_fwd(const NormParams& p, bool f32_inputs, int sms, cudaStream_t stream);
cudaError_t launch_norm_bwd(const NormParams& p, bool f32_inputs, int sms, cudaStream_t stream);
size_t norm_bwd_smem_bytes(int d);

// Launches the forward kernel variant for (V, input dtype, MT m-tiles/warp).
cudaError_t launch_fwd(const FwdParams& p, int V, bool f32_inputs, int MT, cudaStream_t stream);

// Resident CTAs per SM of the forward variant for p's G, WPH, K and tc.
int fwd_ctas_per_sm(const FwdParams& p, int V, bool f32_inputs, int MT);

// Dynamic shared memory bytes the forward kernel needs.
size_t fwd_smem_bytes(int K, int V, int G, int WPH, bool f32_inputs, int tc);

// One-wave forward kernel (bf16, K = 64, V = 16, N_q = 1, no readout
// epilogue): p.G heads per CTA over the flattened (b, n) order, G <= N and
// G <= fwd_wave_max_heads(), one warp per head.
int fwd_wave_max_heads();
size_t fwd_wave_smem_bytes(int K, int G, int tc);
cudaError_t launch_fwd_wave(const FwdParams& p, cudaStream_t stream);

}  // namespace m2rnn
