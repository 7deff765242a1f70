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
// checkpoint every 32 tokens; each 32-token segment is re-run forward to keep
// its 8-token window starts in shared memory; each window is re-run forward
// into registers and then swept backwards. Every state used is thus computed
// in the forward direction, exactly as the forward kernel computes it.
//
// Layout: one CTA per (head, 8 value rows), one warp per row, a lane owns
// d_k / 32 consecutive key columns. Sums over columns are warp shuffles; sums
// over rows (dq, dk, dalpha) go through shared memory and then, across the
// d_v / 8 CTAs of a head, into fp32 atomics on outputs the library zeroes first.
//
// Staging: every operand a segment needs (q, k and the CTA's 8 rows of v, beta,
// dy, plus d_t) is copied into shared memory once per CTA with cp.async, into
// a double buffer: the next segment's copies are in flight while the current
// one computes (forwards in the first sweep, backwards in the second; the
// last segment staged by the first sweep is reused by the second). The token
// loops then read only shared memory: k and q as one 8- or 16-byte vector per
// lane, the row and gate scalars as broadcasts.
#include "palimpsa_internal.cuh"

namespace palimpsa {
namespace {

constexpr int kRowsPerCta = 8;     // one warp per value row
constexpr int kThreads = kRowsPerCta * 32;
constexpr int kSeg = 32;           // checkpoint spacing and staging unit (tokens)
constexpr int kWin = 8;            // window re-run into registers (tokens)
constexpr int kNW = kSeg / kWin;   // windows per segment

__host__ __device__ constexpr size_t al16(size_t x) { return (x + 15) / 16 * 16; }

// Shared-memory carve-up (byte offsets; every piece 16-byte aligned).
struct BwdSmem {
  size_t k, q, v, b, dy, dt, stage;   // one staged segment (offsets inside a stage)
  size_t win, red, red_a, al, om, total;

  __host__ __device__ BwdSmem(int DK, int ES) {
    size_t o = 0;
    k = o;  o = al16(o + (size_t)kSeg * DK * ES);
    q = o;  o = al16(o + (size_t)kSeg * DK * ES);
    v = o;  o = al16(o + (size_t)kSeg * kRowsPerCta * ES);
    b = o;  o = al16(o + (size_t)kSeg * kRowsPerCta * ES);
    dy = o; o = al16(o + (size_t)kSeg * kRowsPerCta * 4);
    dt = o; o = al16(o + (size_t)kSeg * 4);
    stage = (o + 127) / 128 * 128;
    o = 2 * stage;
    win = o;   o += (size_t)2 * kRowsPerCta * kNW * DK * 4;   // window starts [M | I][row][window][col]
    red = o;   o += (size_t)2 * 2 * kRowsPerCta * DK * 4;     // [parity][dq | dk][row][col]
    red_a = o; o += (size_t)2 * kRowsPerCta * 4;              // [parity][row] dalpha
    al = o;    o += (size_t)kSeg * 4;                         // alpha of the segment's tokens
    om = o;    o += (size_t)kSeg * 4;                         // (1 - alpha) I_prior
    total = (o + 127) / 128 * 128;
  }
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most one group of this thread is still in flight.
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// All threads: issue the copies of tokens [ts, ts + tn) of one head into a stage.
// Addresses: a token of q or k is d_k * ES bytes (a multiple of 16); the CTA's
// 8 rows of v or beta are 8 * ES contiguous bytes at row0 * ES (row0 is a
// multiple of 8), and of dy 32 bytes; d_t goes 4 bytes at a time.
template <int DK, int ES>
__device__ __forceinline__ void stage_segment(unsigned char* st, const BwdSmem& L, const BwdArgs& a, size_t head_tok,
                                              int row0, int ts, int tn) {
  const int DV = a.d_v;
  const size_t tok0 = head_tok + ts;
  const int kq = tn * DK * ES / 16;
  const char* gk = static_cast<const char*>(a.k) + tok0 * DK * ES;
  const char* gq = static_cast<const char*>(a.q) + tok0 * DK * ES;
  for (int i = threadIdx.x; i < kq; i += kThreads) {
    cp_async16(st + L.k + 16 * (size_t)i, gk + 16 * (size_t)i);
    cp_async16(st + L.q + 16 * (size_t)i, gq + 16 * (size_t)i);
  }
  constexpr int RP = kRowsPerCta * ES / 16;   // 16-byte pieces of one token's rows (v, beta)
  for (int i = threadIdx.x; i < tn * RP; i += kThreads) {
    const int u = i / RP, pc = i % RP;
    const size_t g = ((tok0 + u) * DV + row0) * ES + 16 * pc;
    cp_async16(st + L.v + (size_t)u * kRowsPerCta * ES + 16 * pc, static_cast<const char*>(a.v) + g);
    cp_async16(st + L.b + (size_t)u * kRowsPerCta * ES + 16 * pc, static_cast<const char*>(a.beta) + g);
  }
  constexpr int DP = kRowsPerCta * 4 / 16;    // pieces of one token's dy rows
  for (int i = threadIdx.x; i < tn * DP; i += kThreads) {
    const int u = i / DP, pc = i % DP;
    cp_async16(st + L.dy + (size_t)u * kRowsPerCta * 4 + 16 * pc,
               reinterpret_cast<const char*>(a.dy + (tok0 + u) * DV + row0) + 16 * pc);
  }
  for (int i = threadIdx.x; i < tn; i += kThreads) cp_async4(st + L.dt + 4 * (size_t)i, a.d_t + tok0 + i);
}

// This lane's NC key columns of token u of a staged q or k.
template <bool BF16, int NC>
__device__ __forceinline__ void cols(const unsigned char* base, int DK, int u, int c0, float (&x)[NC]) {
  if constexpr (BF16) {
    const __nv_bfloat16* p = reinterpret_cast<const __nv_bfloat16*>(base) + (size_t)u * DK + c0;
    if constexpr (NC == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      x[0] = bf16_lo(w); x[1] = bf16_hi(w);
    }
  } else {
    const float* p = reinterpret_cast<const float*>(base) + (size_t)u * DK + c0;
    if constexpr (NC == 4) {
      const float4 w = *reinterpret_cast<const float4*>(p);
      x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
    } else {
      const float2 w = *reinterpret_cast<const float2*>(p);
      x[0] = w.x; x[1] = w.y;
    }
  }
}

// Row w's value of token u of a staged v or beta (all lanes read one word).
template <bool BF16>
__device__ __forceinline__ float row_val(const unsigned char* base, int u, int w) {
  if constexpr (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[u * kRowsPerCta + w]);
  else return reinterpret_cast<const float*>(base)[u * kRowsPerCta + w];
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

template <bool BF16>
__device__ __forceinline__ TokRow tok_row(const unsigned char* st, const BwdSmem& L, const float* al,
                                          const float* om, int u, int w) {
  TokRow r;
  r.alpha = al[u];
  r.om = om[u];
  r.b = row_val<BF16>(st + L.b, u, w);
  r.v = row_val<BF16>(st + L.v, u, w);
  r.bv = r.b * r.v;
  return r;
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

// All threads: alpha and (1 - alpha) I_prior of the staged segment's tokens into
// the gate tables (callers order this with barriers on both sides).
__device__ __forceinline__ void fill_gates(const unsigned char* st, const BwdSmem& L, int tn, float A_h, float Ip,
                                           float* al, float* om) {
  const float* dt = reinterpret_cast<const float*>(st + L.dt);
  for (int u = threadIdx.x; u < tn; u += kThreads) {
    const float x = -A_h * dt[u];
    al[u] = expf(x);
    om[u] = -expm1f(x) * Ip;  // (1 - alpha) I_prior without cancellation
  }
}

template <int DK, bool BF16>
__global__ void __launch_bounds__(kThreads)
palimpsa_bwd_kernel(BwdArgs a, float* __restrict__ ckpt) {
  constexpr int NC = DK / 32;
  constexpr int ES = BF16 ? 2 : 4;
  extern __shared__ __align__(128) unsigned char bsm[];
  const BwdSmem L(DK, ES);
  auto win_M = reinterpret_cast<float (*)[kNW][DK]>(bsm + L.win);
  auto win_I = reinterpret_cast<float (*)[kNW][DK]>(bsm + L.win + (size_t)kRowsPerCta * kNW * DK * 4);
  auto red = reinterpret_cast<float (*)[2][kRowsPerCta][DK]>(bsm + L.red);
  auto red_a = reinterpret_cast<float (*)[kRowsPerCta]>(bsm + L.red_a);
  float* al = reinterpret_cast<float*>(bsm + L.al);
  float* om = reinterpret_cast<float*>(bsm + L.om);

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

  // ---- phase 1: forward sweep, checkpoint at every segment start; segment
  // s + 1 is being copied in while segment s computes.
  if (nseg > 0) stage_segment<DK, ES>(bsm, L, a, head_tok, row0, 0, min(kSeg, T));
  cp_async_commit();
  for (int s = 0; s < nseg; ++s) {
    const int ts = s * kSeg, tn = min(kSeg, T - ts);
    if (s + 1 < nseg)
      stage_segment<DK, ES>(bsm + (size_t)((s + 1) & 1) * L.stage, L, a, head_tok, row0, ts + kSeg,
                            min(kSeg, T - ts - kSeg));
    cp_async_commit();
    cp_async_wait_1();
    __syncthreads();  // segment s staged by every thread
    const unsigned char* st = bsm + (size_t)(s & 1) * L.stage;
    fill_gates(st, L, tn, A_h, Ip, al, om);
    float* cp = my_ckpt + ((size_t)s * kRowsPerCta + w) * DK * 2;
#pragma unroll
    for (int e = 0; e < NC; ++e) { cp[c0 + e] = M[e]; cp[DK + c0 + e] = I[e]; }
    __syncthreads();  // gates ready
    for (int u = 0; u < tn; ++u) {
      float k[NC];
      cols<BF16, NC>(st + L.k, DK, u, c0, k);
      fwd_step<NC>(M, I, k, tok_row<BF16>(st, L, al, om, u, w));
    }
    __syncthreads();  // this stage and the gate tables are free again
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

  // ---- phase 2: segments in reverse; segment s - 1 is being copied in while
  // segment s computes (the last segment is still staged from phase 1).
  for (int s = nseg - 1; s >= 0; --s) {
    const int ts = s * kSeg, tn = min(kSeg, T - ts);
    if (s > 0) stage_segment<DK, ES>(bsm + (size_t)((s - 1) & 1) * L.stage, L, a, head_tok, row0, ts - kSeg, kSeg);
    cp_async_commit();
    cp_async_wait_1();
    __syncthreads();  // segment s staged by every thread
    const unsigned char* st = bsm + (size_t)(s & 1) * L.stage;
    const float* dts = reinterpret_cast<const float*>(st + L.dt);
    const float* dys = reinterpret_cast<const float*>(st + L.dy);
    fill_gates(st, L, tn, A_h, Ip, al, om);
    const float* cp = my_ckpt + ((size_t)s * kRowsPerCta + w) * DK * 2;
#pragma unroll
    for (int e = 0; e < NC; ++e) { M[e] = cp[c0 + e]; I[e] = cp[DK + c0 + e]; }
    __syncthreads();  // gates ready
    // re-run the segment, keeping the state at each window start (this warp's row only)
    for (int u = 0; u < tn; ++u) {
      if (u % kWin == 0) {
#pragma unroll
        for (int e = 0; e < NC; ++e) { win_M[w][u / kWin][c0 + e] = M[e]; win_I[w][u / kWin][c0 + e] = I[e]; }
      }
      float k[NC];
      cols<BF16, NC>(st + L.k, DK, u, c0, k);
      fwd_step<NC>(M, I, k, tok_row<BF16>(st, L, al, om, u, w));
    }
    __syncwarp();
    const int nwin = (tn + kWin - 1) / kWin;
    for (int wi = nwin - 1; wi >= 0; --wi) {
      const int uw = wi * kWin, n = min(kWin, tn - uw);
      // re-run the window into registers: state before token uw + uu is (Ms[uu], Is[uu])
      float Ms[kWin + 1][NC], Is[kWin + 1][NC];
#pragma unroll
      for (int e = 0; e < NC; ++e) { Ms[0][e] = win_M[w][wi][c0 + e]; Is[0][e] = win_I[w][wi][c0 + e]; }
#pragma unroll
      for (int uu = 0; uu < kWin; ++uu) {
        if (uu < n) {
          float k[NC];
          cols<BF16, NC>(st + L.k, DK, uw + uu, c0, k);
          const TokRow tr = tok_row<BF16>(st, L, al, om, uw + uu, w);
#pragma unroll
          for (int e = 0; e < NC; ++e) {
            Is[uu + 1][e] = fmaf(tr.alpha, Is[uu][e], fmaf(tr.b, k[e] * k[e], tr.om));
            Ms[uu + 1][e] = fmaf(tr.alpha, Ms[uu][e], tr.bv * k[e]);
          }
        }
      }
      // sweep the window backwards
#pragma unroll
      for (int uu = kWin - 1; uu >= 0; --uu) {
        if (uu < n) {
          const int u = uw + uu, t = ts + u;
          float k[NC], q[NC];
          cols<BF16, NC>(st + L.k, DK, u, c0, k);
          cols<BF16, NC>(st + L.q, DK, u, c0, q);
          const TokRow tr = tok_row<BF16>(st, L, al, om, u, w);
          const float dyi = dys[u * kRowsPerCta + w];
          float s_bv = 0.f, s_b = 0.f, s_al = 0.f, s_gi = 0.f;
          const float om_w = tr.om / Ip;  // 1 - alpha_t
          float dq_p[NC], dk_p[NC];
#pragma unroll
          for (int e = 0; e < NC; ++e) {
            const float r = rcp_approx(Is[uu + 1][e]);
            const float mu = Ms[uu + 1][e] * r;
            const float dmu = dyi * q[e];
            gM[e] = fmaf(dmu, r, gM[e]);
            gI[e] = fmaf(-dmu * mu, r, gI[e]);
            dq_p[e] = dyi * mu;
            s_bv = fmaf(gM[e], k[e], s_bv);
            s_b = fmaf(gI[e], k[e] * k[e], s_b);
            dk_p[e] = fmaf(gM[e], tr.bv, 2.f * gI[e] * tr.b * k[e]);
            s_al = fmaf(gM[e], Ms[uu][e], fmaf(gI[e], Is[uu][e] - Ip, s_al));
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
          for (int it = threadIdx.x; it < 2 * DK; it += kThreads) {
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
            atomicAdd(a.dd_t + head_tok + t, -A_h * tr.alpha * dal);
            dA_acc = fmaf(-dts[u] * tr.alpha, dal, dA_acc);
          }
          par ^= 1;
          // carry the adjoints to t - 1
#pragma unroll
          for (int e = 0; e < NC; ++e) { gM[e] *= tr.alpha; gI[e] *= tr.alpha; }
        }
      }
    }
    __syncthreads();  // this stage, the window starts and the gate tables are free again
  }
  asm volatile("cp.async.wait_all;" ::: "memory");

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
  const size_t smem = BwdSmem(DK, BF16 ? 2 : 4).total;
  auto kern = palimpsa_bwd_kernel<DK, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<ctas, kThreads, smem, s>>>(a, scratch);
  return cudaGetLastError();
}

cudaError_t launch_backward(const BwdArgs& a, float* scratch, cudaStream_t s) {
  if (a.d_k == 128) return a.bf16 ? launch_t<128, true>(a, scratch, s) : launch_t<128, false>(a, scratch, s);
  return a.bf16 ? launch_t<64, true>(a, scratch, s) : launch_t<64, false>(a, scratch, s);
}

}  // namespace palimpsa
