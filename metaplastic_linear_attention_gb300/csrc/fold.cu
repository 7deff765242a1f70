// Affine fold of segment summaries on sm_103a: the exchange step of a time
// split.
//
// Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
// Attention-Based Models" — slide 9 (App. A.12): in the natural parameters both
// recurrences are affine in the state with the shared scalar decay alpha,
//   M_t = alpha_t M_{t-1} + (beta_t (.) v_t) (x) k_t,
//   Ibar_t = alpha_t Ibar_{t-1} + beta_t (x) k_t^2,
// so a stretch of tokens acts on the state as (M, Ibar) -> Gamma (M, Ibar) +
// (dM, dIbar), with Gamma the product of its alphas and (dM, dIbar) the state
// it produces from zero. Composing stretches in order is this fold.
//
// Two uses: (1) the summary of a long range from the summaries of its
// segments (zero start; out = (dM, dIbar, Gamma)); (2) the state at the start
// of a time shard from the summaries of the shards before it (start = the
// sequence's initial state; out = (mu, I) = (M / I, I_prior + Ibar)).
//
// The fold streams R summaries of 8 d_v d_k bytes per head: it is HBM-bound.
// One thread owns 4 consecutive state elements (16-byte loads and stores).
#include "palimpsa_internal.cuh"

namespace palimpsa {
namespace {

__device__ __forceinline__ float4 fma4(float g, float4 x, float4 d) {
  return make_float4(fmaf(g, x.x, d.x), fmaf(g, x.y, d.y), fmaf(g, x.z, d.z), fmaf(g, x.w, d.w));
}

__global__ void __launch_bounds__(256) palimpsa_fold_kernel(FoldArgs f) {
  const long long quads = f.DVK / 4;
  const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= f.heads * quads) return;
  const long long bh = q / quads;
  const long long e = (q % quads) * 4;
  const size_t off = (size_t)bh * f.DVK + e;
  float4 m = make_float4(0.f, 0.f, 0.f, 0.f), ib = m;
  float Ip = 0.f;
  if (f.to_state) {
    Ip = f.I_prior[bh % f.H];
    const float4 i0 = f.I0 ? *reinterpret_cast<const float4*>(f.I0 + off) : make_float4(Ip, Ip, Ip, Ip);
    const float4 u = f.mu0 ? *reinterpret_cast<const float4*>(f.mu0 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
    m = make_float4(i0.x * u.x, i0.y * u.y, i0.z * u.z, i0.w * u.w);
    ib = make_float4(i0.x - Ip, i0.y - Ip, i0.z - Ip, i0.w - Ip);
  }
  float g_all = 1.f;
  for (int s = 0; s < f.R; ++s) {
    const float g = f.gam[s * f.gam_ss + bh * f.gam_sh];
    const float* base = f.sum + s * f.sum_ss + bh * f.sum_sh;
    m = fma4(g, m, *reinterpret_cast<const float4*>(base + e));
    ib = fma4(g, ib, *reinterpret_cast<const float4*>(base + f.DVK + e));
    g_all *= g;
  }
  const size_t o = (size_t)bh * f.out_sh + e;
  if (f.to_state) {
    const float4 I = make_float4(Ip + ib.x, Ip + ib.y, Ip + ib.z, Ip + ib.w);
    *reinterpret_cast<float4*>(f.out_a + o) = make_float4(m.x / I.x, m.y / I.y, m.z / I.z, m.w / I.w);
    *reinterpret_cast<float4*>(f.out_b + o) = I;
  } else {
    *reinterpret_cast<float4*>(f.out_a + o) = m;
    *reinterpret_cast<float4*>(f.out_b + o) = ib;
    if (e == 0) f.out_gamma[bh] = g_all;
  }
}

}  // namespace

cudaError_t launch_fold(const FoldArgs& f, cudaStream_t s) {
  const long long n = f.heads * (f.DVK / 4);
  if (n == 0) return cudaSuccess;
  palimpsa_fold_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(f);
  return cudaGetLastError();
}

}  // namespace palimpsa
