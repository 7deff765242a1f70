// "Without Meta" comparator: the Palimpsa recurrence with the importance frozen
// at its prior, on sm_103a.
//
// Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
// Attention-Based Models" — slide 10 (the "Without Meta" ablations: Palimpsa-M
// without metaplasticity is Mamba2) and slide 11 (the Mamba2 limit of Eq. 5:
// with I = I_prior the mean follows mu_t = alpha_t mu_{t-1} + (beta_t v_t /
// I_prior) (x) k_t). The readout stays y_t = mu_t q_t (slide 4). Slide 22
// compares Palimpsa's kernel speed with a Simple-GLA kernel of this form.
//
// The kernel shares the forward's staging (bulk-copy ring, bounded waits,
// once-per-CTA conversion) and thread tile (2 rows x d_k / 8 columns, row
// teams of 8 lanes), and keeps only mu in registers. Time split: its state
// m = I_prior mu follows Palimpsa's M recurrence exactly (m_t = alpha m_{t-1} +
// (beta_i v_i) k_j), so the forward's passes A and B give m at every segment
// start and this kernel runs each segment from m / I_prior. Per state element and
// token it costs one FMUL and two FFMA (1.5 packed f32x2 instructions) and no
// reciprocal, against Palimpsa's 3 packed instructions plus one SFU
// reciprocal: the measured ratio is the price of metaplasticity.
#include "fwd_staging.cuh"

namespace palimpsa {
namespace {

using namespace fwd;

constexpr int kRows = 2;  // rows per thread

template <int DK, bool BF16, int RG>
__global__ void __launch_bounds__(RG / (4 * kRows) * 32)
palimpsa_fwd_nometa_kernel(FwdArgs a, int C, int nseg, int seg_len, const float* __restrict__ seg_state) {
  constexpr int R = kRows;
  constexpr int NV = DK / 32;
  constexpr int NTH = RG / (4 * R) * 32;
  constexpr int ES = BF16 ? 2 : 4;
  extern __shared__ __align__(128) unsigned char smem[];

  const int DV = a.d_v;
  const Tile tl = tile_of(a, RG, nseg, seg_len);
  if (tl.bad || tl.seg > tl.last_seg) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cg = lane & (kLanesPerRow - 1);
  const int rt = lane >> 3;
  const int lr0 = (warp * 4 + rt) * R;

  const FwdSmem L(C, DK, DV, RG, ES);
  float* kf = reinterpret_cast<float*>(smem + L.kf);
  float* qf = reinterpret_cast<float*>(smem + L.qf);
  float* wf = reinterpret_cast<float*>(smem + L.bvf);  // beta_i v_i / I_prior per row-token
  float* alf = reinterpret_cast<float*>(smem + L.alf);

  const float A_h = a.A[tl.h];
  const float Ip = a.I_prior[tl.h];
  bool domain_bad = !(pos_finite(A_h) && pos_finite(Ip));
  const float rIp = 1.f / Ip;

  const size_t head_tok = tl.head_tok;
  ChunkPipe<DK, ES> pipe(L, smem, static_cast<const char*>(a.q) + head_tok * DK * ES,
                         static_cast<const char*>(a.k) + head_tok * DK * ES,
                         static_cast<const char*>(a.v) + head_tok * DV * ES,
                         static_cast<const char*>(a.beta) + head_tok * DV * ES, C, tl.tb, tl.tn, DV, false);
  pipe.init(a.withhold_first_copy != 0);

  float2 mu[R][2 * NV];
  const size_t state_base = ((size_t)tl.bh * DV + tl.row0) * DK;
  // segments after the first start from the carried m = I_prior mu
  const float* carried = nullptr;
  if (tl.seg > 0) carried = seg_state + ((size_t)tl.bh * (nseg - 1) + (tl.seg - 1)) * 2 * DV * DK;
  else if (nseg > 1)  // the carry's copy of m_0 = I_prior mu0 (never the caller's mu0, which mu_T may alias)
    carried = seg_state + SplitScratch((long long)a.B * a.H, nseg, (long long)DV * DK).init + (size_t)tl.bh * 2 * DV * DK;
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int s = 0; s < NV; ++s) {
      const size_t off = state_base + (size_t)(lr0 + r) * DK + 32 * s + 4 * cg;
      float4 u;
      if (carried) {
        const float4 m = *reinterpret_cast<const float4*>(carried + (size_t)(tl.row0 + lr0 + r) * DK + 32 * s + 4 * cg);
        u = make_float4(m.x * rIp, m.y * rIp, m.z * rIp, m.w * rIp);
      } else {
        u = a.mu0 ? *reinterpret_cast<const float4*>(a.mu0 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      mu[r][2 * s] = make_float2(u.x, u.y);
      mu[r][2 * s + 1] = make_float2(u.z, u.w);
    }
  }

  float* gy = a.y + (head_tok + tl.tb) * DV + tl.row0 + lr0;
  const float* gd = a.d_t + head_tok + tl.tb;
  // d_t one chunk ahead (thread t holds token t of the next chunk; C <= 32), so its
  // load lands during a chunk of compute
  float d_next = 0.f;
  if (pipe.nch > 0 && (int)threadIdx.x < pipe.tc_of(0)) d_next = gd[pipe.t0_of(0) + threadIdx.x];
  for (int c = 0; c < pipe.nch; ++c) {
    const int t0 = pipe.t0_of(c), tc = pipe.tc_of(c);
    const float d_cur = d_next;
    if (c + 1 < pipe.nch && (int)threadIdx.x < pipe.tc_of(c + 1)) d_next = gd[pipe.t0_of(c + 1) + threadIdx.x];
    if (!pipe.wait(c, a.wait_timeout_ns, a.status)) return;
    const unsigned char* raw = pipe.raw(c);
    convert_keys<DK, BF16, true, NTH>(raw, L, smem, tc, false);
    for (int it = threadIdx.x; it < tc * RG; it += NTH) {
      const int t = it / RG, r = it % RG;
      const size_t e = (size_t)t * DV + tl.row0 + r;
      const float vv = raw_elem<BF16>(raw + L.raw_v, e), bb = raw_elem<BF16>(raw + L.raw_b, e);
      domain_bad |= !nonneg_finite(bb);
      wf[it] = (bb * vv) * rIp;
    }
    for (int t = threadIdx.x; t < tc; t += NTH) {  // one token per thread at most (tc <= 32 <= NTH)
      const float d = d_cur;
      domain_bad |= !nonneg_finite(d);
      alf[t] = expf(-A_h * d);
    }
    __syncthreads();
    pipe.refill(c);

    for (int t = 0; t < tc; ++t) {
      const float2 a2 = f2(alf[t]);
      const float2 w = *reinterpret_cast<const float2*>(wf + t * RG + lr0);
      const float wrow[2] = {w.x, w.y};
      float2 acc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
      for (int s = 0; s < NV; ++s) {
        const int col = 32 * s + 4 * cg;
        const float4 k4 = *reinterpret_cast<const float4*>(kf + t * DK + col);
        const float4 q4 = *reinterpret_cast<const float4*>(qf + t * DK + col);
        const float2 kp[2] = {make_float2(k4.x, k4.y), make_float2(k4.z, k4.w)};
        const float2 qp[2] = {make_float2(q4.x, q4.y), make_float2(q4.z, q4.w)};
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float2& m = mu[r][2 * s + p];
            m = __ffma2_rn(a2, m, __fmul2_rn(f2(wrow[r]), kp[p]));
            acc[r] = __ffma2_rn(m, qp[p], acc[r]);
          }
        }
      }
      float yv[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        yv[r] = acc[r].x + acc[r].y;
#pragma unroll
        for (int m = 1; m < kLanesPerRow; m <<= 1) yv[r] += __shfl_xor_sync(0xffffffffu, yv[r], m);
      }
      // every lane of the row team holds the same sums (a butterfly), so all store them
      *reinterpret_cast<float2*>(gy + (size_t)(t0 + t) * DV) = make_float2(yv[0], yv[1]);
    }
    __syncthreads();  // operands of this chunk fully read before the next conversion
  }

  if (tl.seg == tl.last_seg) {  // the sequence's final state
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int s = 0; s < NV; ++s) {
        const size_t off = state_base + (size_t)(lr0 + r) * DK + 32 * s + 4 * cg;
        const float2 m01 = mu[r][2 * s], m23 = mu[r][2 * s + 1];
        *reinterpret_cast<float4*>(a.mu_T + off) = make_float4(m01.x, m01.y, m23.x, m23.y);
      }
    }
  }
  if (__any_sync(0xffffffffu, domain_bad) && lane == 0) latch_status(a.status, kStatusDomain);
}

template <int DK, bool BF16, int RG>
cudaError_t launch_t(const FwdArgs& a, int C, int nseg, int seg_len, const float* st, cudaStream_t s) {
  const FwdSmem L(C, DK, a.d_v, RG, BF16 ? 2 : 4);
  auto kern = palimpsa_fwd_nometa_kernel<DK, BF16, RG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
  if (e != cudaSuccess) return e;
  const long ctas = (long)a.B * a.H * nseg * (a.d_v / RG);
  kern<<<(unsigned)ctas, RG / (4 * kRows) * 32, L.total, s>>>(a, C, nseg, seg_len, st);
  return cudaGetLastError();
}

template <int DK, bool BF16>
cudaError_t launch_rg(const FwdArgs& a, int RG, int C, int nseg, int seg_len, const float* st, cudaStream_t s) {
  switch (RG) {
    case 64: return launch_t<DK, BF16, 64>(a, C, nseg, seg_len, st, s);
    case 32: return launch_t<DK, BF16, 32>(a, C, nseg, seg_len, st, s);
    case 16: return launch_t<DK, BF16, 16>(a, C, nseg, seg_len, st, s);
    default: return launch_t<DK, BF16, 8>(a, C, nseg, seg_len, st, s);
  }
}

}  // namespace

// The comparator with the forward's time split: the same plan (segments from
// the forward's planner), passes A and B for m = I_prior mu, then this kernel
// over every segment.
cudaError_t launch_forward_without_meta(const FwdArgs& a, cudaStream_t s, ScratchProvider* sp) {
  int dev = 0, max_smem = 227 * 1024;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  int RG = 8;
  for (int c : {64, 32, 16, 8})
    if (a.d_v % c == 0) { RG = c; break; }
  const int es = a.bf16 ? 2 : 4;
  int C = a.chunk < 32 ? a.chunk : 32;
  while (C > 16 && FwdSmem(C, a.d_k, a.d_v, RG, es).total > (size_t)max_smem / 3) C /= 2;
  if (FwdSmem(C, a.d_k, a.d_v, RG, es).total > (size_t)max_smem) return cudaErrorInvalidConfiguration;
  int nseg = 1, seg_len = a.T > 0 ? a.T : 1;
  cudaError_t e = plan_forward(a, &nseg, &seg_len);
  if (e != cudaSuccess) return e;
  float* scratch = nullptr;
  if (nseg > 1) {
    const size_t bytes = SplitScratch((long long)a.B * a.H, nseg, (long long)a.d_v * a.d_k).total * sizeof(float);
    if ((e = sp->acquire(bytes, s, &scratch)) != cudaSuccess) return e;
    e = launch_split_prefix(a, nseg, seg_len, scratch, s);
  }
  if (e == cudaSuccess) {
    if (a.d_k == 128)
      e = a.bf16 ? launch_rg<128, true>(a, RG, C, nseg, seg_len, scratch, s)
                 : launch_rg<128, false>(a, RG, C, nseg, seg_len, scratch, s);
    else
      e = a.bf16 ? launch_rg<64, true>(a, RG, C, nseg, seg_len, scratch, s)
                 : launch_rg<64, false>(a, RG, C, nseg, seg_len, scratch, s);
  }
  if (scratch) {
    const cudaError_t e2 = sp->release(scratch, s);
    if (e == cudaSuccess) e = e2;
  }
  return e;
}

}  // namespace palimpsa
