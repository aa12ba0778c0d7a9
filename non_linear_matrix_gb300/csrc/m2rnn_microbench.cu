// m2rnn_microbench.cu -- pipe rates and dependent-chain latencies on sm_103a
// that fix the roofline denominators of the M2RNN kernels.
//
// Built as a stand-alone executable (see non_linear_matrix_gb300/build.py,
// build_microbench()).  Prints one line per measurement:
//   * throughput (results per clock per SM) of tanh.approx in f32, bf16x2 and
//     f16x2, ex2.approx, FFMA, fma.f32x2 and mma.sync m16n8k16 bf16;
//   * latency (clocks) of dependent tanh, FFMA, mma and cvt chains;
//   * one recurrence step of a 16x16 state tile (mma -> tanh -> blend ->
//     bf16 repack), alone (the serial step latency) and with many warps per
//     SM (the throughput the step reaches).
// Every global access is out[gid] / cyc[blockIdx.x] / bw[0..7] with buffers
// sized for the largest launch below.
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#include "ptx.cuh"

#define CK(x)                                                              \
  do {                                                                     \
    cudaError_t e_ = (x);                                                  \
    if (e_ != cudaSuccess) {                                               \
      printf("CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
      return 1;                                                            \
    }                                                                      \
  } while (0)

using namespace m2rnn::ptx;

__device__ __forceinline__ uint32_t tanh_bf2(uint32_t x) {
  uint32_t y;
  asm volatile("tanh.approx.bf16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t tanh_h2(uint32_t x) {
  uint32_t y;
  asm volatile("tanh.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ float ex2_f32(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ffma(float a, float b, float c) {
  float y;
  asm volatile("fma.rn.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t y;
  asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(y) : "l"(a), "l"(b), "l"(c));
  return y;
}
__device__ __forceinline__ float tanh_vol(float x) {
  float y;
  asm volatile("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// OP: 0 tanh.f32, 1 tanh.bf16x2, 2 tanh.f16x2, 3 ex2.f32, 4 ffma, 5 fma.f32x2, 6 mma
template <int OP>
__global__ void thr_kernel(float* out, long long* cyc, const uint32_t* bw, int iters) {
  const int gid = blockIdx.x * blockDim.x + threadIdx.x;
  float x[8];
  uint32_t u[8];
  uint64_t w[8];
  float acc[8][4];
  for (int i = 0; i < 8; ++i) {
    x[i] = 0.001f * (threadIdx.x + i);
    u[i] = 0x3c003c00u + i;
    w[i] = (uint64_t)__float_as_uint(x[i]) | ((uint64_t)__float_as_uint(x[i] + 1.f) << 32);
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  }
  const uint32_t a[4] = {bw[0], bw[1], bw[2], bw[3]};
  const uint32_t b0 = bw[4], b1 = bw[5];
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (OP == 0) x[i] = tanh_vol(x[i]);
      if (OP == 1) u[i] = tanh_bf2(u[i]);
      if (OP == 2) u[i] = tanh_h2(u[i]);
      if (OP == 3) x[i] = ex2_f32(x[i]);
      if (OP == 4) x[i] = ffma(x[i], 0.999f, 0.001f);
      if (OP == 5) w[i] = ffma2(w[i], 0x3f7fbe773f7fbe77ull, 0x3a83126f3a83126full);
      if (OP == 6) mma_bf16_16816(acc[i], a, b0, b1);
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
  for (int i = 0; i < 8; ++i)
    s += x[i] + (float)(u[i] & 0xff) + (float)(w[i] & 0xff) + acc[i][0] + acc[i][3];
  out[gid] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// Dependent chains (one warp).
template <int OP>
__global__ void lat_kernel(float* out, long long* cyc, const uint32_t* bw, int iters) {
  float x = 0.001f * threadIdx.x;
  uint32_t u = 0x3c003c00u;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t a[4] = {bw[0], bw[1], bw[2], bw[3]};
  __syncwarp();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    if (OP == 0) x = tanh_vol(x);
    if (OP == 1) u = tanh_bf2(u);
    if (OP == 4) x = ffma(x, 0.999f, 0.001f);
    if (OP == 6) mma_bf16_16816(acc, a, bw[4], bw[5]);
    if (OP == 7) {
      u = pack_bf16x2(x, x);
      x = bf16x2_lo(u) + 1e-3f;
    }
  }
  __syncwarp();
  const long long t1 = clock64();
  out[threadIdx.x] = x + (float)(u & 0xff) + acc[0];
  if (threadIdx.x == 0) cyc[0] = t1 - t0;
}

// One recurrence step of MT 16x16 tiles held by one warp in mma layout:
// acc = bf16(H) * W; Z = tanh(acc); H = Z + f (H - Z); A = bf16(H).
template <int MT>
__global__ void step_kernel(float* out, long long* cyc, const uint32_t* bw, int iters) {
  const int lane = threadIdx.x & 31;
  float H[MT][8];
  uint32_t A[MT][4];
  for (int m = 0; m < MT; ++m)
    for (int i = 0; i < 8; ++i) H[m][i] = 0.01f * (lane + i + m);
  for (int m = 0; m < MT; ++m)
    for (int i = 0; i < 4; ++i) A[m][i] = pack_bf16x2(H[m][2 * i], H[m][2 * i + 1]);
  const uint32_t B0[2] = {bw[0], bw[1]}, B1[2] = {bw[2], bw[3]};  // distinct n-tiles
  const float f = 0.9f;
  __syncwarp();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
      mma_bf16_16816(acc0, A[m], B0[0], B0[1]);
      mma_bf16_16816(acc1, A[m], B1[0], B1[1]);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float z0 = tanh_approx(acc0[r]), z1 = tanh_approx(acc1[r]);
        H[m][r] = fmaf(f, H[m][r] - z0, z0);
        H[m][4 + r] = fmaf(f, H[m][4 + r] - z1, z1);
      }
      A[m][0] = pack_bf16x2(H[m][0], H[m][1]);
      A[m][1] = pack_bf16x2(H[m][2], H[m][3]);
      A[m][2] = pack_bf16x2(H[m][4], H[m][5]);
      A[m][3] = pack_bf16x2(H[m][6], H[m][7]);
    }
  }
  __syncwarp();
  const long long t1 = clock64();
  float s = 0.f;
  for (int m = 0; m < MT; ++m)
    for (int i = 0; i < 8; ++i) s += H[m][i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

__global__ void clock_probe(long long* c, unsigned long long* g, int spin) {
  unsigned long long g0 = globaltimer_ns();
  const long long c0 = clock64();
  float x = 1.f;
  for (int i = 0; i < spin; ++i) x = ffma(x, 0.9999f, 0.0001f);
  const long long c1 = clock64();
  unsigned long long g1 = globaltimer_ns();
  c[0] = c1 - c0 + (x > 100.f);
  g[0] = g1 - g0;
}

int main() {
  int sms = 0;
  CK(cudaSetDevice(0));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, 0));
  printf("device %s sm_%d%d SMs %d\n", prop.name, prop.major, prop.minor, sms);
  const int max_threads = 1024;
  float* out;
  long long* cyc;
  unsigned long long* gt;
  uint32_t* bw;
  CK(cudaMalloc(&out, sizeof(float) * sms * max_threads));
  CK(cudaMalloc(&cyc, sizeof(long long) * sms));
  CK(cudaMalloc(&gt, sizeof(unsigned long long)));
  CK(cudaMalloc(&bw, sizeof(uint32_t) * 8));
  const uint32_t hbw[8] = {0x3d803d80u, 0x3d803d81u, 0x3d813d80u, 0x3d823d83u,
                           0x3c003c00u, 0x3c013c00u, 0u, 0u};
  CK(cudaMemcpy(bw, hbw, sizeof(hbw), cudaMemcpyHostToDevice));
  static long long hc[4096];
  {
    long long c;
    unsigned long long g;
    clock_probe<<<1, 32>>>(cyc, gt, 20000000);
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(&c, cyc, 8, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&g, gt, 8, cudaMemcpyDeviceToHost));
    printf("clock %.0f MHz (%lld clk in %llu ns)\n", 1e3 * (double)c / (double)g, c, g);
  }
  const char* names[] = {"tanh.approx.f32",  "tanh.approx.bf16x2", "tanh.approx.f16x2",
                         "ex2.approx.f32",   "ffma",               "fma.f32x2",
                         "mma.m16n8k16.bf16 (FMA)"};
  const double per_op[] = {1, 2, 2, 1, 1, 2, 2048};
  const int threads = 512, iters = 4096;
  auto run_thr = [&](int op, auto kern) -> int {
    for (int rep = 0; rep < 2; ++rep) {
      kern<<<sms, threads>>>(out, cyc, bw, iters);
      CK(cudaDeviceSynchronize());
    }
    CK(cudaMemcpy(hc, cyc, sizeof(long long) * sms, cudaMemcpyDeviceToHost));
    long long mx = 0;
    for (int i = 0; i < sms; ++i) mx = hc[i] > mx ? hc[i] : mx;
    const double ops = (op == 6) ? (double)(threads / 32) * 8 * iters * per_op[op]
                                 : (double)threads * 8 * iters * per_op[op];
    printf("throughput %-26s %8.1f results/clk/SM\n", names[op], ops / (double)mx);
    return 0;
  };
  if (run_thr(0, thr_kernel<0>) || run_thr(1, thr_kernel<1>) || run_thr(2, thr_kernel<2>) ||
      run_thr(3, thr_kernel<3>) || run_thr(4, thr_kernel<4>) || run_thr(5, thr_kernel<5>) ||
      run_thr(6, thr_kernel<6>))
    return 1;
  auto run_lat = [&](const char* nm, auto kern) -> int {
    kern<<<1, 32>>>(out, cyc, bw, 1000);
    CK(cudaDeviceSynchronize());
    kern<<<1, 32>>>(out, cyc, bw, 10000);
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(hc, cyc, 8, cudaMemcpyDeviceToHost));
    printf("latency %-24s %6.1f clk\n", nm, hc[0] / 10000.0);
    return 0;
  };
  if (run_lat("tanh.approx.f32", lat_kernel<0>) || run_lat("tanh.approx.bf16x2", lat_kernel<1>) ||
      run_lat("ffma", lat_kernel<4>) || run_lat("mma (accumulate chain)", lat_kernel<6>) ||
      run_lat("cvt bf16x2 + unpack", lat_kernel<7>))
    return 1;
  auto run_step = [&](const char* nm, auto kern, int mt, int blocks, int warps) -> int {
    kern<<<blocks, 32 * warps>>>(out, cyc, bw, 200);
    CK(cudaDeviceSynchronize());
    kern<<<blocks, 32 * warps>>>(out, cyc, bw, 2000);
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(hc, cyc, sizeof(long long) * blocks, cudaMemcpyDeviceToHost));
    long long mx = 0;
    for (int i = 0; i < blocks; ++i) mx = hc[i] > mx ? hc[i] : mx;
    const double per_step = mx / 2000.0;
    const double elems_per_sm = (double)warps * mt * 256 * blocks / sms;
    printf("step %-5s warps/CTA %2d CTAs %4d: %7.1f clk/step, %6.2f state elements/clk/SM\n", nm,
           warps, blocks, per_step, elems_per_sm / per_step);
    return 0;
  };
  if (run_step("MT=1", step_kernel<1>, 1, 1, 1) || run_step("MT=2", step_kernel<2>, 2, 1, 1) ||
      run_step("MT=4", step_kernel<4>, 4, 1, 1) || run_step("MT=4", step_kernel<4>, 4, sms, 4) ||
      run_step("MT=4", step_kernel<4>, 4, sms, 16) || run_step("MT=2", step_kernel<2>, 2, sms, 16) ||
      run_step("MT=1", step_kernel<1>, 1, sms, 16) || run_step("MT=1", step_kernel<1>, 1, sms, 32))
    return 1;
  printf("done\n");
  return 0;
}
