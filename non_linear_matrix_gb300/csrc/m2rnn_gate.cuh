// m2rnn_gate.cuh -- the input gate of the frame "The gate preserves a direct
// path through time" of "M2RNN: Non-Linear RNNs with Matrix-Valued States":
//     f_{t,n} = exp(-alpha_n softplus(a_{t,n} + beta_n)),
// evaluated in fp32 with CUDA's expf / log1pf, and its derivatives
//     df/da = df/dbeta = -alpha f sigmoid(a + beta),   df/dalpha = -softplus(a + beta) f.
// softplus(x) = max(x, 0) + log1p(exp(-|x|)) stays finite for any x.
#pragma once
#include <cuda_runtime.h>

namespace m2rnn {

__device__ __forceinline__ float gate_softplus(float x) {
  return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

__device__ __forceinline__ float gate_f(float a, float alpha, float beta) {
  return expf(-alpha * gate_softplus(a + beta));
}

// f and its derivatives with respect to a (= beta) and alpha.
__device__ __forceinline__ void gate_f_grads(float a, float alpha, float beta, float& f,
                                             float& dfda, float& dfdalpha) {
  const float x = a + beta, sp = gate_softplus(x);
  f = expf(-alpha * sp);
  dfda = -alpha * f / (1.f + expf(-x));  // sigmoid(x) = 1 / (1 + e^-x)
  dfdalpha = -sp * f;
}

}  // namespace m2rnn
