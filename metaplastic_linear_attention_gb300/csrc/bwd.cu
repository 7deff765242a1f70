// Backward of the Palimpsa recurrence on sm_103a: gradients of a loss with
// respect to every input of the chunked forward, given dL/dy (and optionally
// dL/dmu_T, dL/dI_T).
//
// Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
// Attention-Based Models" — the forward is Eq. (5) with the readout of Eq. (2)
// (slides 4, 7) in the natural parameters of slide 9; the pages train through
// this recurrence ("Backpropagation trains the projections and gates that
// generate those updates", slide 4) with a chunked-scan kernel (slide 9).
//
// Per value row i and key column j, with r_t = 1 / I_t and mu_t = M_t r_t:
//   forward   I_t = alpha_t I_{t-1} + (1 - alpha_t) I_prior + beta_i k_j^2
//             M_t = alpha_t M_{t-1} + (beta_i v_i) k_j,      y_i = sum_j mu_t q_j
//   adjoints  gM_t = alpha_{t+1} gM_{t+1} + dy_i q_j r_t
//             gI_t = alpha_{t+1} gI_{t+1} - dy_i q_j mu_t r_t
//   grads     dq_j   += sum_i dy_i mu_t                dk_j += sum_i gM bv_i + 2 gI beta_i k_j
//             d(bv)_i = sum_j gM k_j  -> dv_i = d(bv)_i beta_i,  dbeta_i = d(bv)_i v_i + sum_j gI k_j^2
//             dalpha_t = sum_ij gM_t M_{t-1} + gI_t (I_{t-1} - I_prior)
//             dd_t = -A alpha_t dalpha_t,  dA += -d_t alpha_t dalpha_t,  dI_prior += (1 - alpha_t) sum_ij gI_t
//   start     (t = T) gM = dmu_T r_T, gI = dI_T - dmu_T mu_T r_T;  (t = 0) dmu0 = gM_0 I0, dI0 = gI_0 + gM_0 mu0.
//
// Numerics: the state is never stepped backwards (I_{t-1} = (I_t - c_t) /
// alpha_t cancels badly when alpha is small). A forward sweep stores a
// checkpoint every 64 tokens; each 64-token segment is re-run forward to keep
// its 8-token window starts in shared memory; each window is re-run forward
// into registers and then swept backwards. Every state used is thus computed
// in the forward direction, exactly as the forward kernel computes it.
//
// Layout: one CTA per (head, 8 value rows), one warp per row, a lane owns
// d_k / 32 consecutive key columns. Sums over columns are warp shuffles; sums
// over rows (dq, dk, dalpha) go through shared memory and then, across the
// d_v / 8 CTAs of a head, into fp32 atomics on outputs the library zeroes first.
#include "palimpsa_internal.cuh"

namespace palimpsa {
namespace {

constexpr int kRowsPerCta = 8;   // one warp per value row
constexpr int kSeg = 64;         // checkpoint spacing (tokens)
constexpr int kWin = 8;          // window re-run into registers (tokens)

template <bool BF16, int NC>
__device__ __forceinline__ void load_cols(const void* base, size_t idx, float (&x)[NC]) {
  if constexpr (BF16) {
    const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(base) + idx;
    if constexpr (NC == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    } else {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
      x[0] = bf16_lo(u); x[1] = bf16_hi(u);
    }
  } else {
    const float* p = static_cast<const float*>(base) + idx;
#pragma unroll
    for (int e = 0; e < NC; ++e) x[e] = p[e];
  }
}

template <bool BF16>
__device__ __forceinline__ float load1(const void* base, size_t idx) {
  if constexpr (BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
  else return static_cast<const float*>(base)[idx];
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// Per-token scalars of the forward update for one value row.
struct TokRow {
  float alpha, om, b, v, bv;
};

// alpha_t and (1 - alpha_t) I_prior come from the segment's table in shared
// memory (index t - ts), computed once per CTA.
template <bool BF16>
__device__ __forceinline__ TokRow tok_row(const BwdArgs& a, size_t head_tok, int t, size_t row_idx,
                                          const float* seg_al, const float* seg_om, int ts) {
  TokRow r;
  r.alpha = seg_al[t - ts];
  r.om = seg_om[t - ts];
  r.b = load1<BF16>(a.beta, (head_tok + t) * a.d_v + row_idx);
  r.v = load1<BF16>(a.v, (head_tok + t) * a.d_v + row_idx);
  r.bv = r.b * r.v;
  return r;
}

// All threads: the gate of tokens [ts, te) into the segment tables; ends with a
// CTA barrier (callers must reach it together).
__device__ __forceinline__ void fill_gates(const float* d_t, size_t head_tok, int ts, int te, float A_h, float Ip,
                                           float* seg_al, float* seg_om) {
  __syncthreads();  // previous users of the tables are done
  for (int u = threadIdx.x; u < te - ts; u += blockDim.x) {
    const float x = -A_h * d_t[head_tok + ts + u];
    seg_al[u] = expf(x);
    seg_om[u] = -expm1f(x) * Ip;  // (1 - alpha) I_prior without cancellation
  }
  __syncthreads();
}

// One forward step of a lane's NC state elements (the forward kernel's update).
template <int NC>
__device__ __forceinline__ void fwd_step(float (&M)[NC], float (&I)[NC], const float (&k)[NC], const TokRow& tr) {
#pragma unroll
  for (int e = 0; e < NC; ++e) {
    I[e] = fmaf(tr.alpha, I[e], fmaf(tr.b, k[e] * k[e], tr.om));
    M[e] = fmaf(tr.alpha, M[e], tr.bv * k[e]);
  }
}

template <int DK, bool BF16>
__global__ void __launch_bounds__(kRowsPerCta * 32)
palimpsa_bwd_kernel(BwdArgs a, float* __restrict__ ckpt) {
  constexpr int NC = DK / 32;
  constexpr int NW = kSeg / kWin;
  // dynamic shared memory: window starts [row][window][col] for M and I, the
  // row-reduction buffers [token parity][dq | dk][row][col], and [parity][row] dalpha
  extern __shared__ __align__(16) float bsm[];
  auto win_M = reinterpret_cast<float (*)[NW][DK]>(bsm);
  auto win_I = reinterpret_cast<float (*)[NW][DK]>(bsm + kRowsPerCta * NW * DK);
  auto red = reinterpret_cast<float (*)[2][kRowsPerCta][DK]>(bsm + 2 * kRowsPerCta * NW * DK);
  auto red_a = reinterpret_cast<float (*)[kRowsPerCta]>(bsm + 2 * kRowsPerCta * NW * DK + 4 * kRowsPerCta * DK);
  float* seg_al = bsm + 2 * kRowsPerCta * NW * DK + 4 * kRowsPerCta * DK + 2 * kRowsPerCta;
  float* seg_om = seg_al + kSeg;

  const int DV = a.d_v, T = a.T;
  const int groups = DV / kRowsPerCta;
  const long bh = blockIdx.x / groups;
  const int row0 = (blockIdx.x % groups) * kRowsPerCta;
  const int h = (int)(bh % a.H);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int i = row0 + w;             // this warp's value row
  const int c0 = lane * NC;           // this lane's first key column
  const size_t head_tok = (size_t)bh * T;
  const float A_h = a.A[h], Ip = a.I_prior[h];
  const int nseg = (T + kSeg - 1) / kSeg;
  float* my_ckpt = ckpt + (size_t)blockIdx.x * nseg * kRowsPerCta * DK * 2;

  // ---- initial state
  float M[NC], I[NC], mu0v[NC], I0v[NC];
  const size_t soff = ((size_t)bh * DV + i) * DK + c0;
#pragma unroll
  for (int e = 0; e < NC; ++e) {
    I0v[e] = a.I0 ? a.I0[soff + e] : Ip;
    mu0v[e] = a.mu0 ? a.mu0[soff + e] : 0.f;
    I[e] = I0v[e];
    M[e] = I0v[e] * mu0v[e];
  }

  // ---- phase 1: forward sweep, checkpoint at every segment start
  for (int s = 0; s < nseg; ++s) {
    float* cp = my_ckpt + ((size_t)s * kRowsPerCta + w) * DK * 2;
#pragma unroll
    for (int e = 0; e < NC; ++e) { cp[c0 + e] = M[e]; cp[DK + c0 + e] = I[e]; }
    const int t_end = min(T, (s + 1) * kSeg);
    fill_gates(a.d_t, head_tok, s * kSeg, t_end, A_h, Ip, seg_al, seg_om);
    for (int t = s * kSeg; t < t_end; ++t) {
      float k[NC];
      load_cols<BF16, NC>(a.k, (head_tok + t) * DK + c0, k);
      fwd_step<NC>(M, I, k, tok_row<BF16>(a, head_tok, t, i, seg_al, seg_om, s * kSeg));
    }
  }

  // ---- adjoints at t = T from the final-state gradients
  float gM[NC], gI[NC];
#pragma unroll
  for (int e = 0; e < NC; ++e) {
    const float dmu = a.dmu_T ? a.dmu_T[soff + e] : 0.f;
    const float dI = a.dI_T ? a.dI_T[soff + e] : 0.f;
    const float r = 1.f / I[e];
    gM[e] = dmu * r;
    gI[e] = dI - dmu * (M[e] * r) * r;
  }
  float dIp_acc = 0.f, dA_acc = 0.f;
  int par = 0;

  // ---- phase 2: segments in reverse
  for (int s = nseg - 1; s >= 0; --s) {
    const int ts = s * kSeg, te = min(T, ts + kSeg);
    fill_gates(a.d_t, head_tok, ts, te, A_h, Ip, seg_al, seg_om);
    const float* cp = my_ckpt + ((size_t)s * kRowsPerCta + w) * DK * 2;
#pragma unroll
    for (int e = 0; e < NC; ++e) { M[e] = cp[c0 + e]; I[e] = cp[DK + c0 + e]; }
    // re-run the segment, keeping the state at each window start (this warp's row only)
    for (int t = ts; t < te; ++t) {
      if ((t - ts) % kWin == 0) {
        const int wi = (t - ts) / kWin;
#pragma unroll
        for (int e = 0; e < NC; ++e) { win_M[w][wi][c0 + e] = M[e]; win_I[w][wi][c0 + e] = I[e]; }
      }
      float k[NC];
      load_cols<BF16, NC>(a.k, (head_tok + t) * DK + c0, k);
      fwd_step<NC>(M, I, k, tok_row<BF16>(a, head_tok, t, i, seg_al, seg_om, ts));
    }
    __syncwarp();
    const int nwin = (te - ts + kWin - 1) / kWin;
    for (int wi = nwin - 1; wi >= 0; --wi) {
      const int tw = ts + wi * kWin, n = min(kWin, te - tw);
      // re-run the window into registers: state before token tw + u is (Ms[u], Is[u])
      float Ms[kWin + 1][NC], Is[kWin + 1][NC];
#pragma unroll
      for (int e = 0; e < NC; ++e) { Ms[0][e] = win_M[w][wi][c0 + e]; Is[0][e] = win_I[w][wi][c0 + e]; }
#pragma unroll
      for (int u = 0; u < kWin; ++u) {
        if (u < n) {
          float k[NC];
          load_cols<BF16, NC>(a.k, (head_tok + tw + u) * DK + c0, k);
          const TokRow tr = tok_row<BF16>(a, head_tok, tw + u, i, seg_al, seg_om, ts);
#pragma unroll
          for (int e = 0; e < NC; ++e) {
            Is[u + 1][e] = fmaf(tr.alpha, Is[u][e], fmaf(tr.b, k[e] * k[e], tr.om));
            Ms[u + 1][e] = fmaf(tr.alpha, Ms[u][e], tr.bv * k[e]);
          }
        }
      }
      // sweep the window backwards
#pragma unroll
      for (int u = kWin - 1; u >= 0; --u) {
        if (u < n) {
          const int t = tw + u;
          float k[NC], q[NC];
          load_cols<BF16, NC>(a.k, (head_tok + t) * DK + c0, k);
          load_cols<BF16, NC>(a.q, (head_tok + t) * DK + c0, q);
          const TokRow tr = tok_row<BF16>(a, head_tok, t, i, seg_al, seg_om, ts);
          const float dyi = a.dy[(head_tok + t) * DV + i];
          float s_bv = 0.f, s_b = 0.f, s_al = 0.f, s_gi = 0.f;
          const float om_w = tr.om / Ip;  // 1 - alpha_t
          float dq_p[NC], dk_p[NC];
#pragma unroll
          for (int e = 0; e < NC; ++e) {
            const float r = rcp_approx(Is[u + 1][e]);
            const float mu = Ms[u + 1][e] * r;
            const float dmu = dyi * q[e];
            gM[e] = fmaf(dmu, r, gM[e]);
            gI[e] = fmaf(-dmu * mu, r, gI[e]);
            dq_p[e] = dyi * mu;
            s_bv = fmaf(gM[e], k[e], s_bv);
            s_b = fmaf(gI[e], k[e] * k[e], s_b);
            dk_p[e] = fmaf(gM[e], tr.bv, 2.f * gI[e] * tr.b * k[e]);
            s_al = fmaf(gM[e], Ms[u][e], fmaf(gI[e], Is[u][e] - Ip, s_al));
            s_gi += gI[e];
          }
          s_bv = warp_sum(s_bv);
          s_b = warp_sum(s_b);
          s_al = warp_sum(s_al);
          dIp_acc = fmaf(om_w, s_gi, dIp_acc);  // per lane; reduced over the warp at the end
          if (lane == 0) {
            const size_t o = (head_tok + t) * DV + i;
            a.dv[o] = s_bv * tr.b;
            a.dbeta[o] = fmaf(s_bv, tr.v, s_b);
            red_a[par][w] = s_al;
          }
#pragma unroll
          for (int e = 0; e < NC; ++e) { red[par][0][w][c0 + e] = dq_p[e]; red[par][1][w][c0 + e] = dk_p[e]; }
          __syncthreads();
          for (int it = threadIdx.x; it < 2 * DK; it += kRowsPerCta * 32) {
            const int which = it / DK, j = it % DK;
            float sum = 0.f;
#pragma unroll
            for (int rr = 0; rr < kRowsPerCta; ++rr) sum += red[par][which][rr][j];
            atomicAdd((which ? a.dk : a.dq) + (head_tok + t) * DK + j, sum);
          }
          if (threadIdx.x == 0) {
            float dal = 0.f;
#pragma unroll
            for (int rr = 0; rr < kRowsPerCta; ++rr) dal += red_a[par][rr];
            const float dt = a.d_t[head_tok + t];
            atomicAdd(a.dd_t + head_tok + t, -A_h * tr.alpha * dal);
            dA_acc = fmaf(-dt * tr.alpha, dal, dA_acc);
          }
          par ^= 1;
          // carry the adjoints to t - 1
#pragma unroll
          for (int e = 0; e < NC; ++e) { gM[e] *= tr.alpha; gI[e] *= tr.alpha; }
        }
      }
    }
    __syncwarp();
  }

  // ---- initial-state gradients: M_0 = I0 (.) mu0, I_0 = I0
  float s_ip0 = 0.f;
#pragma unroll
  for (int e = 0; e < NC; ++e) {
    const float dI0 = gI[e] + gM[e] * mu0v[e];
    if (a.dmu0) a.dmu0[soff + e] = gM[e] * I0v[e];
    if (a.dI0) a.dI0[soff + e] = dI0;
    s_ip0 += dI0;
  }
  // With I0 absent the initial precision is I_prior itself.
  if (!a.I0) dIp_acc += s_ip0;
  dIp_acc = warp_sum(dIp_acc);
  if (lane == 0) atomicAdd(a.dI_prior + h, dIp_acc);
  if (threadIdx.x == 0) atomicAdd(a.dA + h, dA_acc);
}

}  // namespace

size_t backward_scratch_bytes(const BwdArgs& a) {
  const size_t ctas = (size_t)a.B * a.H * (a.d_v / kRowsPerCta);
  const size_t nseg = (size_t)(a.T + kSeg - 1) / kSeg;
  return ctas * nseg * kRowsPerCta * a.d_k * 2 * sizeof(float);
}

template <int DK, bool BF16>
cudaError_t launch_t(const BwdArgs& a, float* scratch, cudaStream_t s) {
  const unsigned ctas = (unsigned)((long)a.B * a.H * (a.d_v / kRowsPerCta));
  const size_t smem =
      (2 * kRowsPerCta * (kSeg / kWin) * DK + 4 * kRowsPerCta * DK + 2 * kRowsPerCta + 2 * kSeg) * sizeof(float);
  auto kern = palimpsa_bwd_kernel<DK, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<ctas, kRowsPerCta * 32, smem, s>>>(a, scratch);
  return cudaGetLastError();
}

cudaError_t launch_backward(const BwdArgs& a, float* scratch, cudaStream_t s) {
  if (a.d_k == 128) return a.bf16 ? launch_t<128, true>(a, scratch, s) : launch_t<128, false>(a, scratch, s);
  return a.bf16 ? launch_t<64, true>(a, scratch, s) : launch_t<64, false>(a, scratch, s);
}

}  // namespace palimpsa
