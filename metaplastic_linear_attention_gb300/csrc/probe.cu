// Issue-rate probe of the arithmetic units the Palimpsa kernels are bound by.
//
// The chunked forward (pass C) and the backward perform one reciprocal per
// element-token (the readout's M / I, slide 9 / paper App. A.12) on the SFU,
// next to a few FP32 FMAs. Their roofline is therefore the SFU reciprocal rate
// of the GPU, which this probe measures directly: one CTA per SM (its dynamic
// shared memory keeps a second CTA off the SM), 32 warps, every thread running
// 8 independent chains of the instruction under test, timed with the SM's own
// cycle counter. The rate per clock and SM is the CTA's instruction count over
// its elapsed cycles; the host takes the median over the SMs.
#include <algorithm>
#include <vector>

#include "palimpsa.h"
#include "palimpsa_internal.cuh"

namespace palimpsa {
namespace {

constexpr int kProbeThreads = 1024;
constexpr int kProbeChains = 8;
constexpr int kProbeIters = 2048;

template <int OP>
__device__ __forceinline__ float probe_op(float x) {
  float r;
  if constexpr (OP == PALIMPSA_PROBE_RCP) {
    // 1 / (x + 1): an add in front of each reciprocal (as in the kernels, where
    // I is formed just before its reciprocal) keeps the code generator from
    // folding a reciprocal of a reciprocal back into its argument; the add runs
    // on the FP32 pipe, whose rate is eight times the SFU's
    asm volatile("{\n\t.reg .f32 t;\n\tadd.f32 t, %1, 0f3F800000;\n\trcp.approx.ftz.f32 %0, t;\n\t}"
                 : "=f"(r)
                 : "f"(x));
  } else if constexpr (OP == PALIMPSA_PROBE_EX2) {
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(-x));  // 2^-x stays in (0, 1]
  } else if constexpr (OP == PALIMPSA_PROBE_RSQ) {
    asm volatile("{\n\t.reg .f32 t;\n\tadd.f32 t, %1, 0f3F800000;\n\trsqrt.approx.ftz.f32 %0, t;\n\t}"
                 : "=f"(r)
                 : "f"(x));  // 1 / sqrt(x + 1) stays in (0, 1]
  } else if constexpr (OP == PALIMPSA_PROBE_LG2) {
    asm volatile("{\n\t.reg .f32 t;\n\tadd.f32 t, %1, 0f40000000;\n\tlg2.approx.ftz.f32 %0, t;\n\t}"
                 : "=f"(r)
                 : "f"(x));  // log2(x + 2) stays in [1, 2)
  } else {
    asm volatile("fma.rn.f32 %0, %1, 0f3F7FBE77, 0f3A83126F;" : "=f"(r) : "f"(x));  // x * 0.999 + 0.001
  }
  return r;
}

template <int OP>
__global__ void __launch_bounds__(kProbeThreads, 1) palimpsa_probe_kernel(long long* cycles, float* sink) {
  extern __shared__ float keep_alone[];  // sized by the host so that one CTA fills an SM
  float x[kProbeChains];
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c) x[c] = 0.5f + 0.01f * (threadIdx.x & 7) + 0.001f * c;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < kProbeIters; ++it) {
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) x[c] = probe_op<OP>(x[c]);
  }
  __syncthreads();
  const long long t1 = clock64();
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c) acc += x[c];
  if (acc == 12345.f) keep_alone[0] = acc;  // never true; keeps the chains live
  if (acc == 12345.f) sink[blockIdx.x] = keep_alone[0];
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

}  // namespace
}  // namespace palimpsa

using namespace palimpsa;

extern "C" palimpsa_status palimpsa_probe_issue_rate(int op, double* per_clk_per_sm, void* cuda_stream) {
  if (!per_clk_per_sm) return PALIMPSA_ERR_NULL;
  if (op < PALIMPSA_PROBE_RCP || op > PALIMPSA_PROBE_LG2) return PALIMPSA_ERR_UNSUPPORTED;
  int dev = 0, sms = 0, smem_sm = 0, smem_optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return PALIMPSA_ERR_CUDA;
  // more than half of the SM's shared memory: a second CTA cannot join the first
  const int smem = std::min(smem_optin, smem_sm / 2 + 1024);
  auto kern = op == PALIMPSA_PROBE_RCP   ? palimpsa_probe_kernel<PALIMPSA_PROBE_RCP>
              : op == PALIMPSA_PROBE_EX2 ? palimpsa_probe_kernel<PALIMPSA_PROBE_EX2>
              : op == PALIMPSA_PROBE_RSQ ? palimpsa_probe_kernel<PALIMPSA_PROBE_RSQ>
              : op == PALIMPSA_PROBE_LG2 ? palimpsa_probe_kernel<PALIMPSA_PROBE_LG2>
                                         : palimpsa_probe_kernel<PALIMPSA_PROBE_FFMA>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return PALIMPSA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  long long* cycles = nullptr;
  float* sink = nullptr;
  if (cudaMallocAsync(&cycles, sizeof(long long) * sms, s) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  if (cudaMallocAsync(&sink, sizeof(float) * sms, s) != cudaSuccess) {
    cudaFreeAsync(cycles, s);
    return PALIMPSA_ERR_CUDA;
  }
  std::vector<long long> host(sms, 0);
  palimpsa_status st = PALIMPSA_OK;
  for (int rep = 0; rep < 2 && st == PALIMPSA_OK; ++rep) {  // the first launch warms the clocks up
    kern<<<sms, kProbeThreads, smem, s>>>(cycles, sink);
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(host.data(), cycles, sizeof(long long) * sms, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      st = PALIMPSA_ERR_CUDA;
  }
  cudaFreeAsync(cycles, s);
  cudaFreeAsync(sink, s);
  if (st != PALIMPSA_OK) return st;
  std::sort(host.begin(), host.end());
  const double med = (double)host[host.size() / 2];
  if (!(med > 0)) return PALIMPSA_ERR_CUDA;
  *per_clk_per_sm = (double)kProbeThreads * kProbeChains * kProbeIters / med;
  return PALIMPSA_OK;
}
