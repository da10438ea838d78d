// Measured FP32 FFMA rate of this GPU: the denominator of the strict-f32
// path's roofline (its GEMMs are FFMA-only, no tensor cores).  A kernel with
// eight independent fused multiply-add chains per thread, two 1024-thread
// blocks per SM in the grid, timed with CUDA events; nothing of the training
// step runs here.
#include <cstdio>

#include "../../include/mg.h"
#include "common.cuh"
#include "kernels.h"

namespace mg {
namespace {

constexpr int kPeakThreads = 1024;
constexpr int kPeakChains = 8;

__global__ void __launch_bounds__(kPeakThreads) ffma_peak_kernel(float* sink, int iters) {
  float a[kPeakChains];
#pragma unroll
  for (int i = 0; i < kPeakChains; ++i) a[i] = 1e-3f * (float)((threadIdx.x + i) & 15);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kPeakChains; ++i) a[i] = fmaf(a[i], 0.9999f, 1e-4f);
  }
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < kPeakChains; ++i) s += a[i];
  if (s == 12345.678f) sink[blockIdx.x] = s;   // keeps the chains live; never true
}

}  // namespace
}  // namespace mg

extern "C" mg_status mg_ffma_peak(double* tflops, double* flop_per_clk_per_sm, mg_stream_t stream) {
  using namespace mg;
  if (!tflops) {
    set_global_error("mg_ffma_peak: tflops must be non-NULL");
    return MG_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  float* sink = nullptr;
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;
  if (e == cudaSuccess) e = cudaMalloc(&sink, (size_t)sms * 2 * sizeof(float));
  if (e == cudaSuccess) e = cudaEventCreate(&ev0);
  if (e == cudaSuccess) e = cudaEventCreate(&ev1);
  const int iters = 1 << 14;
  const int grid = 2 * sms;
  float ms = 0.0f;
  cudaStream_t s = (cudaStream_t)stream;
  if (e == cudaSuccess) {
    ffma_peak_kernel<<<grid, kPeakThreads, 0, s>>>(sink, iters);   // warm-up
    cudaEventRecord(ev0, s);
    ffma_peak_kernel<<<grid, kPeakThreads, 0, s>>>(sink, iters);
    cudaEventRecord(ev1, s);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventSynchronize(ev1);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, ev0, ev1);
  if (ev0) cudaEventDestroy(ev0);
  if (ev1) cudaEventDestroy(ev1);
  if (sink) cudaFree(sink);
  if (e != cudaSuccess) {
    char msg[160];
    snprintf(msg, sizeof msg, "mg_ffma_peak: %s", cudaGetErrorString(e));
    set_global_error(msg);
    return MG_ERR_CUDA;
  }
  const double flop = 2.0 * kPeakChains * (double)iters * kPeakThreads * grid;
  *tflops = flop / (ms * 1e-3) / 1e12;
  if (flop_per_clk_per_sm) {
    // per SM and clock at the device's maximum SM clock (the kernel's blocks
    // do not all overlap on an SM, so per-block cycle counts cannot give it)
    int khz = 0;
    if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess || khz <= 0) {
      cudaGetLastError();
      *flop_per_clk_per_sm = 0.0;
    } else {
      *flop_per_clk_per_sm = *tflops * 1e12 / ((double)sms * khz * 1e3);
    }
  }
  return MG_OK;
}
