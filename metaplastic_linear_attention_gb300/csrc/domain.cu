// Domain check of a call's inputs, for the entry points whose kernels do not
// test the preconditions as they read them (the backward and the segment
// summary: their inner loops are register-bound, and a test there measured a
// few percent slower; the state combine, a plain stream over the summaries). One grid-stride pass over the arrays; any violation
// latches PALIMPSA_ERR_DOMAIN into the device status word. Nothing faults and
// nothing else is written.
//
// Preconditions (slide 4 / paper Eq. (2): beta >= 0; slide 5: alpha =
// exp(-A d_t) in (0, 1], so A > 0 and d_t >= 0; a precision is positive: I_prior
// > 0, I0 > 0), all finite.
#include <algorithm>

#include "palimpsa_internal.cuh"

namespace palimpsa {
namespace {

// 16-bit bf16 lanes of a 32-bit word: negative (not -0) or not finite.
__device__ __forceinline__ bool bf16x2_bad(uint32_t w) {
  bool bad = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t x = (w >> (16 * h)) & 0xffffu;
    bad |= ((x & 0x8000u) && (x & 0x7fffu)) || ((x & 0x7f80u) == 0x7f80u);
  }
  return bad;
}

template <bool BF16>
__global__ void __launch_bounds__(256) palimpsa_domain_kernel(DomainArgs a) {
  bool bad = false;
  const size_t stride = (size_t)gridDim.x * blockDim.x, t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  // beta: 16-byte pieces (8 bf16 or 4 fp32), then the tail one value at a time
  const size_t per16 = BF16 ? 8 : 4;
  const size_t n16 = a.n_beta / per16;
  for (size_t i = t0; i < n16; i += stride) {
    const uint4 w = reinterpret_cast<const uint4*>(a.beta)[i];
    if constexpr (BF16) {
      bad |= bf16x2_bad(w.x) || bf16x2_bad(w.y) || bf16x2_bad(w.z) || bf16x2_bad(w.w);
    } else {
      bad |= !(nonneg_finite(__uint_as_float(w.x)) && nonneg_finite(__uint_as_float(w.y)) &&
               nonneg_finite(__uint_as_float(w.z)) && nonneg_finite(__uint_as_float(w.w)));
    }
  }
  for (size_t i = n16 * per16 + t0; i < a.n_beta; i += stride) {
    const float b = BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.beta)[i])
                         : static_cast<const float*>(a.beta)[i];
    bad |= !nonneg_finite(b);
  }
  for (size_t i = t0; i < a.n_dt; i += stride) bad |= !nonneg_finite(a.d_t[i]);
  if (a.I0)
    for (size_t i = t0; i < a.n_state; i += stride) bad |= !pos_finite(a.I0[i]);
  for (size_t i = t0; i < (size_t)a.H; i += stride) bad |= !((!a.A || pos_finite(a.A[i])) && pos_finite(a.I_prior[i]));
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) latch_status(a.status, kStatusDomain);
}

}  // namespace

cudaError_t launch_domain_check(const DomainArgs& a, cudaStream_t s) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t work = a.n_beta / 8 + a.n_dt + a.n_state;
  const unsigned blocks = (unsigned)std::max<size_t>(1, std::min<size_t>((size_t)sms * 4, (work + 255) / 256));
  if (a.bf16) palimpsa_domain_kernel<true><<<blocks, 256, 0, s>>>(a);
  else palimpsa_domain_kernel<false><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace palimpsa
