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
//             dalpha_t = sum_ij gM_t M_{t-1} + gI_t (I_{t-1} - I_prior), taken as
//             alpha_t dalpha_t = sum_ij gM_t (M_t - bv_i k_j) + gI_t (I_t - I_prior - beta_i k_j^2)
//               = F_t - R_t,  F_t = sum_ij gM_t M_t + gI_t (I_t - I_prior),
//                             R_t = sum_i (bv_i d(bv)_i + beta_i sum_j gI k_j^2)   (row sums the kernel forms anyway);
//             F itself needs no per-element work at most tokens: with gM_{t-1} = alpha_t gM_t + dy q r,
//             gI_{t-1} = alpha_t gI_t - dy q mu r, the readout's two contributions to F_{t-1} cancel
//             ((dy q r) M - (dy q mu r) I = 0), leaving the scalar recursion
//               F_{t-1} = alpha_t dalpha_t - I_prior J_{t-1},  J_t = sum_ij (-dy_i q_j mu_ij r_ij)
//             (J is summed from the injections themselves, not as a difference of two sums of gI,
//             which would cancel when memory is long), so F is formed element by element only at
//             the last token of each 8-token window and carried through the window by this
//             recursion (over at most 7 tokens, so rounding cannot build up);
//             dd_t = -A (alpha_t dalpha_t),  dA += -d_t (alpha_t dalpha_t),  dI_prior += (1 - alpha_t) sum_ij gI_t
//   start     (t = T) gM = dmu_T r_T, gI = dI_T - dmu_T mu_T r_T;  (t = 0) dmu0 = gM_0 I0, dI0 = gI_0 + gM_0 mu0.
//
// Numerics: the state is never stepped backwards (I_{t-1} = (I_t - c_t) /
// alpha_t cancels badly when alpha is small). A forward sweep stores a
// checkpoint every 32 tokens (or the forward wrote them); each 32-token
// segment is re-run forward to keep its 8-token window starts in shared
// memory; each window is re-run forward into registers and then swept
// backwards. Every state used is computed in the forward direction, exactly as
// the forward kernel computes it.
//
// Layout: one CTA of 4 warps per (head, 8 value rows). A lane owns two value
// rows (lane bits 4, 3 pick the row pair) and d_k / 32 consecutive key columns
// (lane bits 2..0 and the warp pick them), so the per-token loads, the column
// sums over rows and the row sums over columns are shared by twice the
// elements of a one-row lane. Column sums (dq, dk) are summed over two of the
// warp's four row pairs with one reduce-scatter level and go to fp32 atomics,
// where the other two pairs and the d_v / 8 CTAs of a head add into the same
// dq, dk (the library zeroes them first; one level fewer measured faster). Row
// sums (d(bv), sum gI k^2) finish over the 8 column lanes with shuffles and
// over the 4 warps through shared memory once per 8-token window; each lane's
// part of J (the sum of its gI injections) goes to shared memory as it is and
// is summed over the CTA's 128 lanes once per window. Then one warp turns the
// window's per-token sums into the alpha gradients with the F recursion above
// (a suffix sum over the window's tokens), while the other warps go on to the
// next window.
//
// Staging: every operand a segment needs (q, k and the CTA's 8 rows of v, beta,
// dy, plus d_t) is copied into shared memory once per CTA with cp.async, into
// a double buffer: the next segment's copies are in flight while the current
// one computes (forwards in the first sweep, backwards in the second; the
// last segment staged by the first sweep is reused by the second). The token
// loops then read only shared memory.
#include "palimpsa_internal.cuh"

namespace palimpsa {
namespace {

constexpr int kRowsPerCta = 8;     // value rows per CTA: 4 row pairs
constexpr int kWarps = 4;          // warps split the key columns
constexpr int kThreads = kWarps * 32;
constexpr int kSeg = 32;           // checkpoint spacing and staging unit (tokens)
constexpr int kWin = 8;            // window re-run into registers (tokens)
constexpr int kNW = kSeg / kWin;   // windows per segment

__host__ __device__ constexpr size_t al16(size_t x) { return (x + 15) / 16 * 16; }

// Shared-memory carve-up (byte offsets; every piece 16-byte aligned).
struct BwdSmem {
  size_t k, q, v, b, dy, dt, stage;   // one staged segment (offsets inside a stage)
  size_t kf, qf, win, rowp, adap, rb, rbv, gate, sgt, rmi, fw, total;

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
    // fp32 copies of the current segment's k and q (bf16 inputs; fp32 inputs are read in place)
    kf = o;    o += ES == 2 ? (size_t)kSeg * DK * 4 : 0;
    qf = o;    o += ES == 2 ? (size_t)kSeg * DK * 4 : 0;
    win = o;   o += (size_t)2 * kRowsPerCta * kNW * DK * 4;   // window starts [window][M | I][row][pair][thread]
    rowp = o;  o += (size_t)kWarps * kWin * kRowsPerCta * 2 * 4;  // row-sum partials [warp][token][row][2]
    adap = o;  o += (size_t)kWin * kThreads * 4;              // J partials [token][thread]
    rb = o;    o += (size_t)kSeg * kRowsPerCta * 4;           // beta_i of the segment's tokens [token][row]
    rbv = o;   o += (size_t)kSeg * kRowsPerCta * 4;           // beta_i v_i
    gate = o;  o += (size_t)kSeg * 16;                        // [token](alpha, (1 - alpha) I_prior, 1 - alpha, 0)
    sgt = o;   o += (size_t)kWin * 4;                         // the window's J per token (CTA)
    rmi = o;   o += (size_t)kWin * 4;                         // the window's sum_i (bv_i d(bv)_i + beta_i sum_j gI k^2)
    fw = o;    o += (size_t)2 * kWarps * 4;                   // F at the window's last token, per warp, two windows
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
// Without q_dy (the forward sweep's segments, except its last, which the
// adjoint sweep reuses) q and dy are not copied.
template <int DK, int ES>
__device__ __forceinline__ void stage_segment(unsigned char* st, const BwdSmem& L, const BwdArgs& a, size_t head_tok,
                                              int row0, int ts, int tn, bool q_dy = true) {
  const int DV = a.d_v;
  const size_t tok0 = head_tok + ts;
  const int kq = tn * DK * ES / 16;
  const char* gk = static_cast<const char*>(a.k) + tok0 * DK * ES;
  const char* gq = static_cast<const char*>(a.q) + tok0 * DK * ES;
  for (int i = threadIdx.x; i < kq; i += kThreads) {
    cp_async16(st + L.k + 16 * (size_t)i, gk + 16 * (size_t)i);
    if (q_dy) cp_async16(st + L.q + 16 * (size_t)i, gq + 16 * (size_t)i);
  }
  constexpr int RP = kRowsPerCta * ES / 16;   // 16-byte pieces of one token's rows (v, beta)
  for (int i = threadIdx.x; i < tn * RP; i += kThreads) {
    const int u = i / RP, pc = i % RP;
    const size_t g = ((tok0 + u) * DV + row0) * ES + 16 * pc;
    cp_async16(st + L.v + (size_t)u * kRowsPerCta * ES + 16 * pc, static_cast<const char*>(a.v) + g);
    cp_async16(st + L.b + (size_t)u * kRowsPerCta * ES + 16 * pc, static_cast<const char*>(a.beta) + g);
  }
  constexpr int DP = kRowsPerCta * 4 / 16;    // pieces of one token's dy rows
  for (int i = threadIdx.x; q_dy && i < tn * DP; i += kThreads) {
    const int u = i / DP, pc = i % DP;
    cp_async16(st + L.dy + (size_t)u * kRowsPerCta * 4 + 16 * pc,
               reinterpret_cast<const char*>(a.dy + (tok0 + u) * DV + row0) + 16 * pc);
  }
  for (int i = threadIdx.x; i < tn; i += kThreads) cp_async4(st + L.dt + 4 * (size_t)i, a.d_t + tok0 + i);
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

__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }

// One level of a reduce-scatter over the two lanes that differ in lane bit
// `m`: of its first N partials a lane keeps the half its side owns (bit set:
// the upper half) and adds the partner's copy of that half. After the levels
// for bits 16 and 8 (in that order) a lane of row pair g holds partials
// g * V / 4 .. g * V / 4 + V / 4 - 1 of the original V, summed over the warp's
// four row pairs.
template <int V, int N>
__device__ __forceinline__ void rs_level(float (&x)[V], int lane, int m) {
  const bool hi = (lane & m) != 0;
#pragma unroll
  for (int v = 0; v < N / 2; ++v) {
    const float send = hi ? x[v] : x[v + N / 2];
    const float keep = hi ? x[v + N / 2] : x[v];
    x[v] = keep + __shfl_xor_sync(0xffffffffu, send, m);
  }
}

// All threads, once per staged segment: the gate table (alpha, (1 - alpha)
// I_prior, 1 - alpha per token, one 16-byte load), the row tables (beta_i, beta_i v_i of the CTA's 8 rows)
// and, for bf16 inputs, fp32 copies of k and (WITH_Q: the adjoint sweep reads it) q.
// Callers order this with barriers on both sides.
template <int DK, bool BF16, bool WITH_Q = true>
__device__ __forceinline__ void prepare_segment(const unsigned char* st, unsigned char* bsm, const BwdSmem& L, int tn,
                                                float A_h, float Ip) {
  const float* dt = reinterpret_cast<const float*>(st + L.dt);
  float4* gate = reinterpret_cast<float4*>(bsm + L.gate);
  for (int u = threadIdx.x; u < tn; u += kThreads) {
    const float x = -A_h * dt[u];
    const float one_minus = -expm1f(x);  // 1 - alpha without cancellation
    gate[u] = make_float4(expf(x), one_minus * Ip, one_minus, 0.f);
  }
  float* rb = reinterpret_cast<float*>(bsm + L.rb);
  float* rbv = reinterpret_cast<float*>(bsm + L.rbv);
  for (int x = threadIdx.x; x < tn * kRowsPerCta; x += kThreads) {
    const float b = row_val<BF16>(st + L.b, x / kRowsPerCta, x % kRowsPerCta);
    rb[x] = b;
    rbv[x] = b * row_val<BF16>(st + L.v, x / kRowsPerCta, x % kRowsPerCta);
  }
  if constexpr (BF16) {
    // 4 bf16 values (8 bytes) in, one float4 out per item: consecutive threads store
    // consecutive 16 bytes, so the stores are free of bank conflicts
    const int n4 = tn * DK / 4;
    auto convert = [&](const int x) {
#pragma unroll
      for (int which = 0; which < (WITH_Q ? 2 : 1); ++which) {
        const uint2 w = reinterpret_cast<const uint2*>(st + (which ? L.q : L.k))[x];
        reinterpret_cast<float4*>(bsm + (which ? L.qf : L.kf))[x] =
            make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
      }
    };
    if (tn == kSeg) {  // a whole segment: a fixed count per thread, unrolled so the loads go out together
#pragma unroll
      for (int i = 0; i < kSeg * DK / 4 / kThreads; ++i) convert(threadIdx.x + i * kThreads);
    } else {
      for (int x = threadIdx.x; x < n4; x += kThreads) convert(x);
    }
  }
}

// This lane's 2 NP key columns of token u of the fp32 k or q, as NP pairs.
template <int NP>
__device__ __forceinline__ void lane_pairs(const float* base, int DK, int u, int c0, float2 (&x)[NP]) {
  const float* p = base + (size_t)u * DK + c0;
  if constexpr (NP == 2) {
    const float4 w = *reinterpret_cast<const float4*>(p);
    x[0] = make_float2(w.x, w.y);
    x[1] = make_float2(w.z, w.w);
  } else {
    x[0] = *reinterpret_cast<const float2*>(p);
  }
}

// Per-token scalars of the forward update for the lane's two value rows.
struct Tok2 {
  float alpha, om, oma;
  float2 b, bv;  // beta_i and beta_i v_i of rows 2g, 2g + 1
};

__device__ __forceinline__ Tok2 tok2(const unsigned char* bsm, const BwdSmem& L, int u, int g) {
  Tok2 t;
  const float4 gv = reinterpret_cast<const float4*>(bsm + L.gate)[u];
  t.alpha = gv.x;
  t.om = gv.y;
  t.oma = gv.z;
  t.b = reinterpret_cast<const float2*>(bsm + L.rb)[(u * kRowsPerCta) / 2 + g];
  t.bv = reinterpret_cast<const float2*>(bsm + L.rbv)[(u * kRowsPerCta) / 2 + g];
  return t;
}

// One forward step of the lane's two rows (the forward kernel's update, packed):
//   I = alpha I + (beta_i k_j^2 + (1 - alpha) I_prior),  M = alpha M + (beta_i v_i) k_j.
template <int NP>
__device__ __forceinline__ void step_rows(float2 (&M)[2][NP], float2 (&I)[2][NP], const float2 (&k)[NP],
                                          const Tok2& t) {
  const float2 a2 = f2(t.alpha), om2 = f2(t.om);
  float2 kk[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) kk[p] = __fmul2_rn(k[p], k[p]);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float2 b2 = f2(r ? t.b.y : t.b.x), bv2 = f2(r ? t.bv.y : t.bv.x);
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      I[r][p] = __ffma2_rn(a2, I[r][p], __ffma2_rn(b2, kk[p], om2));
      M[r][p] = __ffma2_rn(a2, M[r][p], __fmul2_rn(bv2, k[p]));
    }
  }
}

// Adjoints at t = T of the lane's elements, from the final state (M, I):
// gM = dmu_T / I, gI = dI_T - dmu_T mu_T / I. soff is row 2g's offset; row
// 2g + 1 follows d_k floats later.
template <int NP>
__device__ __forceinline__ void init_adjoints(const BwdArgs& a, size_t soff, int DK, const float2 (&M)[2][NP],
                                              const float2 (&I)[2][NP], float2 (&gM)[2][NP], float2 (&gI)[2][NP]) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const size_t o = soff + (size_t)r * DK + 2 * p;
      const float2 dmu = a.dmu_T ? *reinterpret_cast<const float2*>(a.dmu_T + o) : f2(0.f);
      const float2 dI = a.dI_T ? *reinterpret_cast<const float2*>(a.dI_T + o) : f2(0.f);
      const float2 rr = make_float2(1.f / I[r][p].x, 1.f / I[r][p].y);
      gM[r][p] = __fmul2_rn(dmu, rr);
      gI[r][p] = make_float2(dI.x - dmu.x * (M[r][p].x * rr.x) * rr.x, dI.y - dmu.y * (M[r][p].y * rr.y) * rr.y);
    }
  }
}

// The lane's elements of a row-major array at (row 2g, column c0): two rows,
// `rs` floats apart, of NP pairs each.
template <int NP>
__device__ __forceinline__ void load_rows(const float* base, size_t rs, float2 (&x)[2][NP]) {
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int p = 0; p < NP; ++p) x[r][p] = *reinterpret_cast<const float2*>(base + r * rs + 2 * p);
}
template <int NP>
__device__ __forceinline__ void store_rows(float* base, size_t rs, const float2 (&x)[2][NP]) {
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int p = 0; p < NP; ++p) *reinterpret_cast<float2*>(base + r * rs + 2 * p) = x[r][p];
}

template <int DK, bool BF16, bool PACKED>
__global__ void __launch_bounds__(kThreads, 2)
palimpsa_bwd_kernel(BwdArgs a, float* __restrict__ ckpt) {
  constexpr int C = DK / 32;          // key columns per lane
  constexpr int NP = C / 2;           // column pairs per lane and row
  constexpr int CWARP = DK / kWarps;  // key columns per warp
  constexpr int ES = BF16 ? 2 : 4;
  static_assert(CWARP == 8 * C, "eight column lanes per warp");
  extern __shared__ __align__(128) unsigned char bsm[];
  const BwdSmem L(DK, ES);
  // window starts, lane-linear (only the owning lane reads them back): [window][M | I][row][pair][thread]
  float2* winS = reinterpret_cast<float2*>(bsm + L.win);
  auto win_at = [&](int wi, int mi, int r, int p) -> float2& {
    return winS[(((wi * 2 + mi) * 2 + r) * NP + p) * kThreads + threadIdx.x];
  };
  auto rowp = reinterpret_cast<float (*)[kWin][kRowsPerCta][2]>(bsm + L.rowp);
  auto adap = reinterpret_cast<float (*)[kThreads]>(bsm + L.adap);
  float* sgt_w = reinterpret_cast<float*>(bsm + L.sgt);
  float* rmi_w = reinterpret_cast<float*>(bsm + L.rmi);
  float* fwin = reinterpret_cast<float*>(bsm + L.fw);
  const float* rb_t = reinterpret_cast<const float*>(bsm + L.rb);
  const float* rbv_t = reinterpret_cast<const float*>(bsm + L.rbv);

  const int DV = a.d_v;
  const int groups = DV / kRowsPerCta;
  const long bh = blockIdx.x / groups;
  const int row0 = (blockIdx.x % groups) * kRowsPerCta;
  const int h = (int)(bh % a.H);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 3;                    // this lane's row pair: CTA rows 2g, 2g + 1
  const int c0 = w * CWARP + (lane & 7) * C;  // this lane's first key column
  // this head's sequence: all T tokens, or a packed sequence's own range,
  // checked before anything is read (a bad one is reported and skipped)
  int T = a.T;
  size_t head_tok = (size_t)bh * a.T;
  // checkpoints [slot][value row][M | I], from the forward or written by phase 1
  long long ck_slot0 = bh * (long long)((a.T + kSeg - 1) / kSeg);
  if constexpr (PACKED) {
    const long n = bh / a.H;
    const int s0 = a.cu_seqlens[n], s1 = a.cu_seqlens[n + 1];
    if (!(s0 >= 0 && s1 >= s0 && (long long)s1 <= a.total_T && s1 - s0 <= a.T)) {
      if (threadIdx.x == 0 && a.status) latch_status(a.status, kStatusDomain);
      return;
    }
    T = s1 - s0;
    head_tok = (size_t)h * (size_t)a.total_T + (size_t)s0;
    ck_slot0 = packed_checkpoint_slot0(h, n, s0, a.total_T, a.B);
  }
  const float A_h = a.A[h], Ip = a.I_prior[h];
  const int nseg = (T + kSeg - 1) / kSeg;
  static_assert(kSeg == kCheckpointTokens, "backward segments are the training checkpoints");
  const size_t ck_head = (size_t)ck_slot0 * DV * 2 * DK;
  const size_t ck_lane = (size_t)(row0 + 2 * g) * 2 * DK + c0;   // the lane's first element in a checkpoint
  float* ck_out = ckpt ? ckpt + ck_head + ck_lane : nullptr;  // null when the forward's checkpoints are used
  const float* ck_in = (a.ckpt_in ? a.ckpt_in : ckpt) + ck_head + ck_lane;
  const size_t ck_step = (size_t)DV * 2 * DK;                  // one checkpoint of the head
  const size_t soff = ((size_t)bh * DV + row0 + 2 * g) * DK + c0;  // the lane's first state element

  // ---- initial state
  float2 M[2][NP], I[2][NP];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const size_t o = soff + (size_t)r * DK + 2 * p;
      const float2 i0 = a.I0 ? *reinterpret_cast<const float2*>(a.I0 + o) : f2(Ip);
      const float2 m0 = a.mu0 ? *reinterpret_cast<const float2*>(a.mu0 + o) : f2(0.f);
      I[r][p] = i0;
      M[r][p] = __fmul2_rn(i0, m0);
    }
  }

  // ---- phase 1: forward sweep, checkpoint at every segment start; segment
  // s + 1 is being copied in while segment s computes. Skipped when the forward
  // wrote the checkpoints: then only the last segment is staged for phase 2.
  if (a.ckpt_in) {
    if (nseg > 0)
      stage_segment<DK, ES>(bsm + (size_t)((nseg - 1) & 1) * L.stage, L, a, head_tok, row0, (nseg - 1) * kSeg,
                            T - (nseg - 1) * kSeg);
    cp_async_commit();
  } else {
    if (nseg > 0) stage_segment<DK, ES>(bsm, L, a, head_tok, row0, 0, min(kSeg, T), nseg == 1);
    cp_async_commit();
    for (int s = 0; s < nseg; ++s) {
      const int ts = s * kSeg, tn = min(kSeg, T - ts);
      if (s + 1 < nseg)
        stage_segment<DK, ES>(bsm + (size_t)((s + 1) & 1) * L.stage, L, a, head_tok, row0, ts + kSeg,
                              min(kSeg, T - ts - kSeg), s + 1 == nseg - 1);
      cp_async_commit();
      cp_async_wait_1();
      __syncthreads();  // segment s staged by every thread
      const unsigned char* st = bsm + (size_t)(s & 1) * L.stage;
      prepare_segment<DK, BF16, false>(st, bsm, L, tn, A_h, Ip);  // the forward sweep reads no q
      const float* kf = reinterpret_cast<const float*>(BF16 ? bsm + L.kf : st + L.k);
      float* cp = ck_out + (size_t)s * ck_step;
      store_rows<NP>(cp, 2 * DK, M);
      store_rows<NP>(cp + DK, 2 * DK, I);
      __syncthreads();  // gates ready
      const int whole = tn / kWin * kWin;  // 8 tokens at a time without a per-token branch
      for (int u0 = 0; u0 < whole; u0 += kWin) {
#pragma unroll
        for (int uu = 0; uu < kWin; ++uu) {
          float2 k[NP];
          lane_pairs<NP>(kf, DK, u0 + uu, c0, k);
          step_rows<NP>(M, I, k, tok2(bsm, L, u0 + uu, g));
        }
      }
      for (int u = whole; u < tn; ++u) {
        float2 k[NP];
        lane_pairs<NP>(kf, DK, u, c0, k);
        step_rows<NP>(M, I, k, tok2(bsm, L, u, g));
      }
      __syncthreads();  // this stage and the tables are free again
    }
  }

  // The adjoints start at t = T from the final-state gradients: set from the
  // final state, which the re-run of the last segment reaches (or the initial
  // state when T = 0).
  float2 gM[2][NP], gI[2][NP];
  if (nseg == 0) init_adjoints<NP>(a, soff, DK, M, I, gM, gI);
  float dIp_acc = 0.f, dA_acc = 0.f;
  float acar = 1.f;  // alpha of the token after the one being swept (1 past the end)

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
    const float2* dys = reinterpret_cast<const float2*>(st + L.dy);
    prepare_segment<DK, BF16>(st, bsm, L, tn, A_h, Ip);
    const float* kf = reinterpret_cast<const float*>(BF16 ? bsm + L.kf : st + L.k);
    const float* qf = reinterpret_cast<const float*>(BF16 ? bsm + L.qf : st + L.q);
    load_rows<NP>(ck_in + (size_t)s * ck_step, 2 * DK, M);
    load_rows<NP>(ck_in + (size_t)s * ck_step + DK, 2 * DK, I);
    __syncthreads();  // gates ready
    // re-run the segment, keeping the state at each window start (this lane's elements only).
    // Only the sequence's last segment goes on to its end, where the adjoints start; the others
    // stop at their last window's start, which the window re-run below carries on from.
    const int nwin = (tn + kWin - 1) / kWin;
    const int last_start = (nwin - 1) * kWin;
    const int stop = s == nseg - 1 ? tn : last_start;
    auto keep_start = [&](const int wi) {
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          win_at(wi, 0, r, p) = M[r][p];
          win_at(wi, 1, r, p) = I[r][p];
        }
    };
    // whole windows with their tokens unrolled (no per-token branch), then the
    // sequence's last, partial window when the re-run goes on to the end
    const int whole = stop / kWin;
    for (int wr = 0; wr < whole; ++wr) {
      keep_start(wr);
#pragma unroll
      for (int uu = 0; uu < kWin; ++uu) {
        float2 k[NP];
        lane_pairs<NP>(kf, DK, wr * kWin + uu, c0, k);
        step_rows<NP>(M, I, k, tok2(bsm, L, wr * kWin + uu, g));
      }
    }
    for (int u = whole * kWin; u < stop; ++u) {
      if (u % kWin == 0) keep_start(u / kWin);
      float2 k[NP];
      lane_pairs<NP>(kf, DK, u, c0, k);
      step_rows<NP>(M, I, k, tok2(bsm, L, u, g));
    }
    if (stop == last_start) keep_start(nwin - 1);
    if (s == nseg - 1) init_adjoints<NP>(a, soff, DK, M, I, gM, gI);  // M, I: the final state
    for (int wi = nwin - 1; wi >= 0; --wi) {
      const int uw = wi * kWin, n = min(kWin, tn - uw);
      // re-run the window into registers: (Ms[uu], Is[uu]) is the state after token uw + uu
      float2 Ms[kWin][2][NP], Is[kWin][2][NP];
      auto rerun = [&](const int uu) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            Ms[uu][r][p] = uu ? Ms[uu - 1][r][p] : win_at(wi, 0, r, p);
            Is[uu][r][p] = uu ? Is[uu - 1][r][p] : win_at(wi, 1, r, p);
          }
        float2 k[NP];
        lane_pairs<NP>(kf, DK, uw + uu, c0, k);
        step_rows<NP>(Ms[uu], Is[uu], k, tok2(bsm, L, uw + uu, g));
      };
      // one token of the backward sweep: the adjoints are carried from the token
      // after (times its alpha, acar) and take token uw + uu's readout, in one
      // FMA each; then its gradient sums are formed and handed on. Accumulators
      // start from their first product. At the window's last token (the first
      // swept) the lane also forms its part of F (see the header).
      auto sweep = [&](const int uu, const bool window_end) {
        const int u = uw + uu;
        float2 k[NP], q[NP], kk[NP], dqa[NP], dkM[NP], dkI[NP];
        lane_pairs<NP>(kf, DK, u, c0, k);
        lane_pairs<NP>(qf, DK, u, c0, q);
        const Tok2 tr = tok2(bsm, L, u, g);
        const float2 dyp = dys[(u * kRowsPerCta) / 2 + g];
        const float2 ac2 = f2(acar);
#pragma unroll
        for (int p = 0; p < NP; ++p) kk[p] = __fmul2_rn(k[p], k[p]);
        float2 rM[2], rI[2], sgi[2], ji[2], fp = f2(0.f);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float2 ndy2 = f2(-(r ? dyp.y : dyp.x));
          const float2 bv2 = f2(r ? tr.bv.y : tr.bv.x), b2 = f2(r ? tr.b.y : tr.b.x);
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            const float2 Ic = Is[uu][r][p], Mc = Ms[uu][r][p];
            const float2 nr = make_float2(rcp_approx(-Ic.x), rcp_approx(-Ic.y));  // -1 / I
            const float2 mun = __fmul2_rn(Mc, nr);                                 // -mu
            dqa[p] = r ? __ffma2_rn(ndy2, mun, dqa[p]) : __fmul2_rn(ndy2, mun);   // + dy_i mu
            const float2 injM = __fmul2_rn(ndy2, __fmul2_rn(q[p], nr));            // + dy q / I
            gM[r][p] = __ffma2_rn(ac2, gM[r][p], injM);
            const float2 injI = __fmul2_rn(injM, mun);                             // - dy q mu / I
            gI[r][p] = __ffma2_rn(ac2, gI[r][p], injI);
            dkM[p] = r ? __ffma2_rn(gM[r][p], bv2, dkM[p]) : __fmul2_rn(gM[r][p], bv2);
            dkI[p] = r ? __ffma2_rn(gI[r][p], b2, dkI[p]) : __fmul2_rn(gI[r][p], b2);
            rM[r] = p ? __ffma2_rn(gM[r][p], k[p], rM[r]) : __fmul2_rn(gM[r][p], k[p]);
            rI[r] = p ? __ffma2_rn(gI[r][p], kk[p], rI[r]) : __fmul2_rn(gI[r][p], kk[p]);
            sgi[r] = p ? __fadd2_rn(sgi[r], gI[r][p]) : gI[r][p];
            ji[r] = p ? __fadd2_rn(ji[r], injI) : injI;
            if (window_end) fp = __ffma2_rn(gM[r][p], Mc, __ffma2_rn(gI[r][p], Ic, fp));
          }
        }
        // columns: dq_j and dk_j = sum gM bv + 2 k_j sum gI beta over the lane's
        // rows, then over the warp's 4 row pairs; one fp32 atomic per kept pair
        float cs[2 * C];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          const float2 dk2 = __ffma2_rn(__fadd2_rn(k[p], k[p]), dkI[p], dkM[p]);
          cs[2 * p] = dqa[p].x;
          cs[2 * p + 1] = dqa[p].y;
          cs[C + 2 * p] = dk2.x;
          cs[C + 2 * p + 1] = dk2.y;
        }
        // one reduce-scatter level over the row pairs g and g ^ 2 (lane bit 4): a lane keeps its
        // columns' dq sums (bit clear) or dk sums (bit set); the pairs g and g ^ 1 then meet
        // in the fp32 atomics
        rs_level<2 * C, 2 * C>(cs, lane, 16);
        {
          float* dst = ((lane & 16) ? a.dk : a.dq) + (head_tok + ts + u) * DK + c0;
#pragma unroll
          for (int p = 0; p < NP; ++p)
            atomicAdd(reinterpret_cast<float2*>(dst + 2 * p), make_float2(cs[2 * p], cs[2 * p + 1]));
        }
        // rows: d(bv)_i and sum_j gI k_j^2 over the lane's columns, then over the
        // warp's 8 column lanes; sum gI and J over the lane's elements
        float rv[4] = {rM[0].x + rM[0].y, rM[1].x + rM[1].y, rI[0].x + rI[0].y, rI[1].x + rI[1].y};
        const float sg = (sgi[0].x + sgi[0].y) + (sgi[1].x + sgi[1].y);
        const float jl = (ji[0].x + ji[0].y) + (ji[1].x + ji[1].y);
        dIp_acc = fmaf(tr.oma, sg, dIp_acc);  // (1 - alpha) sum gI; reduced at the end
        rs_level<4, 4>(rv, lane, 4);
        rs_level<4, 2>(rv, lane, 2);
        rv[0] += __shfl_xor_sync(0xffffffffu, rv[0], 1);
        if ((lane & 1) == 0) {
          const int o = (lane >> 1) & 3;   // row 2g + (o & 1); d(bv) for o < 2, else sum gI k^2
          rowp[w][uu][2 * g + (o & 1)][o >> 1] = rv[0];
        }
        adap[uu][threadIdx.x] = jl;  // summed once per window
        if (window_end) {  // this warp's part of F at the window's last token
          const float f = warp_sum((fp.x + fp.y) - Ip * sg);
          if (lane == 0) fwin[(wi & 1) * kWarps + w] = f;
        }
        acar = tr.alpha;  // carries the adjoints to the token before
      };
      // full windows without per-token guards, so that neighbouring tokens interleave
      if (n == kWin) {
#pragma unroll
        for (int uu = 0; uu < kWin; ++uu) rerun(uu);
#pragma unroll
        for (int uu = kWin - 1; uu >= 0; --uu) sweep(uu, uu == kWin - 1);
      } else {
#pragma unroll
        for (int uu = 0; uu < kWin; ++uu)
          if (uu < n) rerun(uu);
#pragma unroll
        for (int uu = kWin - 1; uu >= 0; --uu)
          if (uu < n) sweep(uu, uu == n - 1);
      }
      __syncthreads();
      if (threadIdx.x < kWin * kRowsPerCta) {
        // warps 0, 1: the window's row sums: dv, dbeta per (token, row), and per token
        // R = sum_i (bv_i d(bv)_i + beta_i sum_j gI k_j^2) over the CTA's rows (8 lanes a token)
        const int uu = threadIdx.x / kRowsPerCta, r = threadIdx.x % kRowsPerCta, u = uw + uu;
        float rr = 0.f;
        if (uu < n) {
          float s_bv = 0.f, s_b = 0.f;
#pragma unroll
          for (int ww = 0; ww < kWarps; ++ww) {
            const float2 pr = *reinterpret_cast<const float2*>(&rowp[ww][uu][r][0]);
            s_bv += pr.x;
            s_b += pr.y;
          }
          const size_t o = (head_tok + ts + u) * DV + row0 + r;
          a.dv[o] = s_bv * row_val<BF16>(st + L.b, u, r);
          a.dbeta[o] = fmaf(s_bv, row_val<BF16>(st + L.v, u, r), s_b);
          const int x = u * kRowsPerCta + r;
          rr = fmaf(rbv_t[x], s_bv, rb_t[x] * s_b);
        }
#pragma unroll
        for (int m = 4; m >= 1; m >>= 1) rr += __shfl_xor_sync(0xffffffffu, rr, m);
        if (r == 0) rmi_w[uu] = rr;
      } else {
        // warps 2, 3: the window's J per token: its 128 lane partials, 8 threads a token
        const int t2 = threadIdx.x - kWin * kRowsPerCta, uu = t2 >> 3, part = t2 & 7;
        float sgs = 0.f;
        if (uu < n) {  // float4 c * 8 + part: the 8 threads of a token read 128 consecutive bytes
          const float4* src = reinterpret_cast<const float4*>(&adap[uu][0]);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 v4 = src[c * 8 + part];
            sgs += (v4.x + v4.y) + (v4.z + v4.w);
          }
        }
#pragma unroll
        for (int m = 4; m >= 1; m >>= 1) sgs += __shfl_xor_sync(0xffffffffu, sgs, m);
        if (part == 0) sgt_w[uu] = sgs;
      }
      __syncthreads();  // the row partials are free for the next window; R, G and F are in place
      if (w == 0) {
        // alpha_t dL/dalpha_t = F_t - R_t, with F_{t-1} = F_t - X_t, X_t = R_t + I_prior J_{t-1}:
        // lane uu < n takes token uw + uu; F_t = F(window end) - (X summed over the window's later tokens)
        float X = 0.f, rr = 0.f;
        if (lane < n) {
          rr = rmi_w[lane];
          if (lane > 0) X = fmaf(Ip, sgt_w[lane - 1], rr);
        }
        float suf = X;  // inclusive suffix sum over lanes (lanes >= n hold 0)
#pragma unroll
        for (int m = 1; m < kWin; m <<= 1) {
          const float o = __shfl_down_sync(0xffffffffu, suf, m);
          if (lane + m < 32) suf += o;
        }
        const float* fw = fwin + (wi & 1) * kWarps;
        const float Fend = (fw[0] + fw[1]) + (fw[2] + fw[3]);
        if (lane < n) {
          const float ad = (Fend - (suf - X)) - rr;
          const int u = uw + lane;
          atomicAdd(a.dd_t + head_tok + ts + u, -A_h * ad);
          dA_acc = fmaf(-dts[u], ad, dA_acc);
        }
      }
    }
    __syncthreads();  // this stage, the window starts and the gate tables are free again
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  // the adjoints at t = 0: carried past the first token
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      gM[r][p] = __fmul2_rn(gM[r][p], f2(acar));
      gI[r][p] = __fmul2_rn(gI[r][p], f2(acar));
    }

  // ---- initial-state gradients: M_0 = I0 (.) mu0, I_0 = I0
  float s_ip0 = 0.f;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const size_t o = soff + (size_t)r * DK + 2 * p;
      const float2 i0 = a.I0 ? *reinterpret_cast<const float2*>(a.I0 + o) : f2(Ip);
      const float2 m0 = a.mu0 ? *reinterpret_cast<const float2*>(a.mu0 + o) : f2(0.f);
      const float2 dI0 = __ffma2_rn(gM[r][p], m0, gI[r][p]);
      if (a.dmu0) *reinterpret_cast<float2*>(a.dmu0 + o) = __fmul2_rn(gM[r][p], i0);
      if (a.dI0) *reinterpret_cast<float2*>(a.dI0 + o) = dI0;
      s_ip0 += dI0.x + dI0.y;
    }
  }
  // With I0 absent the initial precision is I_prior itself.
  if (!a.I0) dIp_acc += s_ip0;
  dIp_acc = warp_sum(dIp_acc);
  if (lane == 0) atomicAdd(a.dI_prior + h, dIp_acc);
  dA_acc = warp_sum(dA_acc);  // lanes of warp 0 hold the dA partials of their token slots
  if (lane == 0) atomicAdd(a.dA + h, dA_acc);
}

}  // namespace

size_t backward_scratch_bytes(const BwdArgs& a) {
  if (a.ckpt_in) return 0;  // the forward's checkpoints replace phase 1
  if (a.cu_seqlens)
    return (size_t)a.H * packed_checkpoint_slots(a.total_T, a.B) * a.d_v * 2 * a.d_k * sizeof(float);
  return checkpoint_floats((long long)a.B * a.H, a.T, a.d_k, a.d_v) * sizeof(float);
}

template <int DK, bool BF16, bool PACKED>
cudaError_t launch_t(const BwdArgs& a, float* scratch, cudaStream_t s) {
  const unsigned ctas = (unsigned)((long)a.B * a.H * (a.d_v / kRowsPerCta));
  const size_t smem = BwdSmem(DK, BF16 ? 2 : 4).total;
  auto kern = palimpsa_bwd_kernel<DK, BF16, PACKED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<ctas, kThreads, smem, s>>>(a, scratch);
  return cudaGetLastError();
}

template <bool PACKED>
cudaError_t launch_layout(const BwdArgs& a, float* scratch, cudaStream_t s) {
  if (a.d_k == 128)
    return a.bf16 ? launch_t<128, true, PACKED>(a, scratch, s) : launch_t<128, false, PACKED>(a, scratch, s);
  return a.bf16 ? launch_t<64, true, PACKED>(a, scratch, s) : launch_t<64, false, PACKED>(a, scratch, s);
}

cudaError_t launch_backward(const BwdArgs& a, float* scratch, cudaStream_t s) {
  return a.cu_seqlens ? launch_layout<true>(a, scratch, s) : launch_layout<false>(a, scratch, s);
}

}  // namespace palimpsa
