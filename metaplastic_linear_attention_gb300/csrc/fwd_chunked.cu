// Chunked forward of the Palimpsa recurrence on sm_103a.
//
// Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
// Attention-Based Models" — slide 7 (paper Eq. 5) for the update, slide 4
// (Eq. 2) for the readout, slide 9 (App. A.12) for the natural parameters
// M = I (.) mu, Ibar = I - I_prior and the chunked scan: chunks are processed
// in parallel and the state is carried from one to the next.
//
// Design (GB300-first, not the pages' Triton kernel):
// * The state of one value row i is 2 x d_k fp32 numbers (M_ij and I_ij). A CTA
//   owns RG rows of one head for a whole segment of the sequence and keeps
//   their state in registers: nothing of the state touches HBM between the
//   first read and the final write.
// * Time split (few heads): the sequence is cut into S segments. Pass A writes
//   each segment's summary (Gamma = prod alpha, and the decayed sums of the
//   segment's writes into M and Ibar); pass B carries the true state across
//   segment boundaries (state_{s+1} = Gamma_s state_s + summary_s, the affine
//   scan of slide 9); pass C runs the recurrence with the readout from each
//   segment's true initial state. With S = 1 only pass C runs.
// * Staging: thread 0 stages each chunk of C tokens with four bulk async copies
//   (cp.async.bulk, completion counted on an mbarrier with expect_tx) into a
//   2-deep raw ring; all warps then convert a landed chunk, once per CTA, into
//   fp32 operands shared by every row. Every wait is bounded.
// * Compute thread tile (pass C): R rows x (d_k / 8) columns. The 8 lanes of a
//   "row team" split the key dimension; lane cg owns the float4 column blocks
//   32 s + 4 cg, so a warp's reads of k, k^2 and q are 128-byte wavefronts that
//   all four row teams share (broadcast).
// * Per state element and token pass C computes
//       c = beta_i k_j^2 + (1 - alpha) I_prior      (FFMA)
//       I = alpha I + c                             (FFMA)
//       M = alpha M + (beta_i v_i) k_j              (FMUL + FFMA)
//       y_i += (M * rcp(I)) q_j                     (MUFU.RCP, FMUL + FFMA)
//   as packed f32x2 instructions over adjacent key columns; it is bound by the
//   SFU reciprocal (16 per clock per SM on GB300). Pass A needs two FFMA per
//   element and token (no reciprocal, no readout).
// * y_{t,i} is reduced over the row team with three butterfly shuffles and
//   stored straight to global memory.
// * Fused prologue (palimpsa_forward_fused): the conversion stage of passes A
//   and C also applies the layer's activations - softplus to the gate input,
//   b_scale * sigmoid to beta, the per-token L2 norm of q and k (Palimpsa-D,
//   slide 10) - and, in the v* mode of slide 11, writes v as given instead of
//   beta v. It runs once per chunk and CTA, outside the token loop.
#include <algorithm>
#include <cmath>

#include "fwd_staging.cuh"

namespace palimpsa {
namespace {

using namespace fwd;

// ------------------------------------------------------------------ pass C
// The recurrence with the readout over one segment (the whole sequence when
// S = 1), from the segment's true initial state. The chunk length C is a
// compile-time constant (16 or 32 tokens), so that the per-token operand
// arrays lie at fixed distances from one another in shared memory and one
// address per token serves all of a token's loads.
template <int DK, bool BF16, int RG, int R, int C>
__global__ void __launch_bounds__(RG / (4 * R) * 32)
palimpsa_fwd_chunked_kernel(FwdArgs a, int nseg, int seg_len, const float* __restrict__ seg_state) {
  constexpr int NV = DK / 32;                 // float4 column blocks per thread
  constexpr int NTH = RG / (4 * R) * 32;      // threads per CTA
  constexpr int ES = BF16 ? 2 : 4;
  extern __shared__ __align__(128) unsigned char smem[];

  const int DV = a.d_v;
  const Tile tl = tile_of(a, RG, nseg, seg_len);
  if (tl.bad) {  // packed offsets out of order or range: touch nothing
    if (threadIdx.x == 0) latch_status(a.status, kStatusDomain);
    return;
  }
  if (tl.seg > tl.last_seg) return;  // past the end of a shorter packed sequence
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cg = lane & (kLanesPerRow - 1);
  const int rt = lane >> 3;
  const int lr0 = (warp * 4 + rt) * R;  // first local row of this thread

  const FwdSmem L(C, DK, DV, RG, ES);
  float* kf = reinterpret_cast<float*>(smem + L.kf);
  float* k2f = reinterpret_cast<float*>(smem + L.k2f);
  float* qf = reinterpret_cast<float*>(smem + L.qf);
  float* bvf = reinterpret_cast<float*>(smem + L.bvf);
  float* bfv = reinterpret_cast<float*>(smem + L.bf);
  // the chunk's gates as (alpha, (1 - alpha) I_prior) pairs, one load per token:
  // they fill the alf and omf arrays, which are adjacent (C * 4 bytes each, a
  // multiple of 16)
  float2* gate = reinterpret_cast<float2*>(smem + L.alf);

  const float A_h = a.A[tl.h];
  const float Ip = a.I_prior[tl.h];
  const float bsc = a.pro.b_scale ? a.pro.b_scale[tl.h] : 1.f;
  bool domain_bad = !(pos_finite(A_h) && pos_finite(Ip));

  const size_t head_tok = tl.head_tok;
  ChunkPipe<DK, ES> pipe(L, smem, static_cast<const char*>(a.q) + head_tok * DK * ES,
                         static_cast<const char*>(a.k) + head_tok * DK * ES,
                         static_cast<const char*>(a.v) + head_tok * DV * ES,
                         static_cast<const char*>(a.beta) + head_tok * DV * ES, C, tl.tb, tl.tn, DV, false);
  pipe.init(a.withhold_first_copy != 0);

  // In a time split this kernel follows the carry kernel with programmatic
  // dependent launch: the first chunks' copies above read only the caller's
  // inputs; the carried state, and every write below, wait for the carry.
  // (Launched normally, the wait returns at once.)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- initial state: M = I0 (.) mu0, I = I0 for the first segment (defaults
  // mu0 = 0, I0 = I_prior); M = carried M, I = I_prior + carried Ibar otherwise.
  float2 Ist[R][2 * NV], Mst[R][2 * NV];
  const size_t state_base = ((size_t)tl.bh * DV + tl.row0) * DK;
  const float* carried = nullptr;
  const float* init = nullptr;  // the first segment of a split reads the carry's copy of (M_0, I_0)
  if (tl.seg > 0) carried = seg_state + ((size_t)tl.bh * (nseg - 1) + (tl.seg - 1)) * 2 * DV * DK;
  else if (nseg > 1)
    init = seg_state + SplitScratch((long long)a.B * a.H, nseg, (long long)DV * DK).init + (size_t)tl.bh * 2 * DV * DK;
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int s = 0; s < NV; ++s) {
      const size_t e = (size_t)(tl.row0 + lr0 + r) * DK + 32 * s + 4 * cg;
      float4 i4, m4;
      if (carried) {
        m4 = *reinterpret_cast<const float4*>(carried + e);
        const float4 ib = *reinterpret_cast<const float4*>(carried + (size_t)DV * DK + e);
        i4 = make_float4(Ip + ib.x, Ip + ib.y, Ip + ib.z, Ip + ib.w);
      } else if (init) {
        m4 = *reinterpret_cast<const float4*>(init + e);
        i4 = *reinterpret_cast<const float4*>(init + (size_t)DV * DK + e);
        domain_bad |= !(pos_finite(i4.x) && pos_finite(i4.y) && pos_finite(i4.z) && pos_finite(i4.w));
      } else {
        const size_t off = state_base + (size_t)(lr0 + r) * DK + 32 * s + 4 * cg;
        i4 = a.I0 ? *reinterpret_cast<const float4*>(a.I0 + off) : make_float4(Ip, Ip, Ip, Ip);
        const float4 u = a.mu0 ? *reinterpret_cast<const float4*>(a.mu0 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
        domain_bad |= !(pos_finite(i4.x) && pos_finite(i4.y) && pos_finite(i4.z) && pos_finite(i4.w));
        m4 = make_float4(i4.x * u.x, i4.y * u.y, i4.z * u.z, i4.w * u.w);
      }
      Ist[r][2 * s] = make_float2(i4.x, i4.y);
      Ist[r][2 * s + 1] = make_float2(i4.z, i4.w);
      Mst[r][2 * s] = make_float2(m4.x, m4.y);
      Mst[r][2 * s + 1] = make_float2(m4.z, m4.w);
    }
  }

  float* gy = a.y + (head_tok + tl.tb) * DV + tl.row0 + lr0;
  const float* gd = a.d_t + head_tok + tl.tb;
  // training checkpoints: the state before every 32nd token of the sequence
  float* ckh = nullptr;
  if (a.ckpt) {
    const long long slot0 =
        a.cu_seqlens ? packed_checkpoint_slot0(tl.h, tl.bh / a.H, (long long)(tl.head_tok - (size_t)tl.h * a.total_T),
                                               a.total_T, a.B)
                     : tl.bh * (long long)((a.T + kCheckpointTokens - 1) / kCheckpointTokens);
    ckh = a.ckpt + (size_t)slot0 * DV * 2 * DK;
  }
  // d_t is read one chunk ahead (thread t holds token t of the next chunk; C <= 32), so
  // that its global load lands during a chunk of compute instead of in front of the
  // barrier that ends the next chunk's conversion
  float d_next = 0.f;
  if (pipe.nch > 0 && (int)threadIdx.x < pipe.tc_of(0)) d_next = gd[pipe.t0_of(0) + threadIdx.x];
  for (int c = 0; c < pipe.nch; ++c) {
    const int t0 = pipe.t0_of(c), tc = pipe.tc_of(c);
    const float d_cur = d_next;
    if (c + 1 < pipe.nch && (int)threadIdx.x < pipe.tc_of(c + 1)) d_next = gd[pipe.t0_of(c + 1) + threadIdx.x];
    if (ckh && (tl.tb + t0) % kCheckpointTokens == 0) {
      float* ck = ckh + (size_t)((tl.tb + t0) / kCheckpointTokens) * DV * 2 * DK;
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int s = 0; s < NV; ++s) {
          const size_t e = (size_t)(tl.row0 + lr0 + r) * 2 * DK + 32 * s + 4 * cg;
          const float2 m01 = Mst[r][2 * s], m23 = Mst[r][2 * s + 1], i01 = Ist[r][2 * s], i23 = Ist[r][2 * s + 1];
          *reinterpret_cast<float4*>(ck + e) = make_float4(m01.x, m01.y, m23.x, m23.y);
          *reinterpret_cast<float4*>(ck + DK + e) = make_float4(i01.x, i01.y, i23.x, i23.y);
        }
      }
    }
    if (!pipe.wait(c, a.wait_timeout_ns, a.status)) return;
    // ---- convert the staged chunk to fp32 operands shared by all rows
    const unsigned char* raw = pipe.raw(c);
    convert_keys<DK, BF16, true, NTH>(raw, L, smem, tc, a.pro.qk_norm);
    auto row_item = [&](const int it) {
      const int t = it / RG, r = it % RG;
      const size_t e = (size_t)t * DV + tl.row0 + r;
      const float vv = raw_elem<BF16>(raw + L.raw_v, e);
      float bb = raw_elem<BF16>(raw + L.raw_b, e);
      if (a.pro.on) bb = bsc * sigmoid_f(bb);
      domain_bad |= !nonneg_finite(bb);
      bvf[it] = a.pro.v_star ? vv : bb * vv;
      bfv[it] = bb;
    };
    if (tc == C) {  // a whole chunk: a fixed count per thread, unrolled so the loads go out together
      static_assert(C * RG % NTH == 0, "whole chunks split evenly over the threads");
#pragma unroll
      for (int i = 0; i < C * RG / NTH; ++i) row_item((int)threadIdx.x + i * NTH);
    } else {
      for (int it = threadIdx.x; it < tc * RG; it += NTH) row_item(it);
    }
    for (int t = threadIdx.x; t < tc; t += NTH) {  // one token per thread at most (tc <= 32 <= NTH)
      float d = d_cur;
      if (a.pro.on) d = softplus_f(d);
      domain_bad |= !nonneg_finite(d);
      const float x = -A_h * d;
      gate[t] = make_float2(expf(x), -expm1f(x) * Ip);  // (1 - alpha) I_prior without cancellation
    }
    __syncthreads();
    pipe.refill(c);

    // ---- the recurrence over the chunk's tokens, state in registers
    for (int t = 0; t < tc; ++t) {
      const float2 gt = gate[t];
      const float2 a2 = f2(gt.x), om2 = f2(gt.y);
      float brow[R], bvrow[R];
      if constexpr (R == 2) {
        const float2 bb = *reinterpret_cast<const float2*>(bfv + t * RG + lr0);
        const float2 bv = *reinterpret_cast<const float2*>(bvf + t * RG + lr0);
        brow[0] = bb.x; brow[1] = bb.y; bvrow[0] = bv.x; bvrow[1] = bv.y;
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) { brow[r] = bfv[t * RG + lr0 + r]; bvrow[r] = bvf[t * RG + lr0 + r]; }
      }
      float2 acc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
      for (int s = 0; s < NV; ++s) {
        const int col = 32 * s + 4 * cg;
        const float4 k4 = *reinterpret_cast<const float4*>(kf + t * DK + col);
        const float4 kk4 = *reinterpret_cast<const float4*>(k2f + t * DK + col);
        const float4 q4 = *reinterpret_cast<const float4*>(qf + t * DK + col);
        const float2 kp[2] = {make_float2(k4.x, k4.y), make_float2(k4.z, k4.w)};
        const float2 kkp[2] = {make_float2(kk4.x, kk4.y), make_float2(kk4.z, kk4.w)};
        const float2 qp[2] = {make_float2(q4.x, q4.y), make_float2(q4.z, q4.w)};
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float2& I2 = Ist[r][2 * s + p];
            float2& M2 = Mst[r][2 * s + p];
            const float2 c2 = __ffma2_rn(f2(brow[r]), kkp[p], om2);
            I2 = __ffma2_rn(a2, I2, c2);
            M2 = __ffma2_rn(a2, M2, __fmul2_rn(f2(bvrow[r]), kp[p]));
            const float2 rc = make_float2(rcp_approx(I2.x), rcp_approx(I2.y));
            acc[r] = __ffma2_rn(__fmul2_rn(M2, rc), qp[p], acc[r]);
          }
        }
      }
      if constexpr (R == 2) {
        // both rows' sums over the row's 8 lanes: the first level hands each half
        // of the lanes one row (lane bit 2), the last two complete the sums
        const float y0 = acc[0].x + acc[0].y, y1 = acc[1].x + acc[1].y;
        const bool hi = (lane & 4) != 0;
        float yk = (hi ? y1 : y0) + __shfl_xor_sync(0xffffffffu, hi ? y0 : y1, 4);
        yk += __shfl_xor_sync(0xffffffffu, yk, 2);
        yk += __shfl_xor_sync(0xffffffffu, yk, 1);
        // the four lanes of each half hold the same sum (a butterfly; IEEE addition
        // commutes), so all of them store it: no branch around the store
        gy[(size_t)(t0 + t) * DV + (cg >> 2)] = yk;
      } else {
        float yv = acc[0].x + acc[0].y;
#pragma unroll
        for (int m = 1; m < kLanesPerRow; m <<= 1) yv += __shfl_xor_sync(0xffffffffu, yv, m);
        gy[(size_t)(t0 + t) * DV] = yv;  // every lane of the team holds the same sum
      }
    }
    // (the barrier at the top of the next chunk orders these reads before the
    // next conversion overwrites the operands)
  }

  // ---- final state (the sequence's last segment only): mu_T = M / I, I_T = I.
  if (tl.seg == tl.last_seg) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int s = 0; s < NV; ++s) {
        const size_t off = state_base + (size_t)(lr0 + r) * DK + 32 * s + 4 * cg;
        const float2 i01 = Ist[r][2 * s], i23 = Ist[r][2 * s + 1];
        float4 m4;
        if (tl.L == 0) {  // pass the initial state through unchanged
          m4 = a.mu0 ? *reinterpret_cast<const float4*>(a.mu0 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          const float2 m01 = Mst[r][2 * s], m23 = Mst[r][2 * s + 1];
          m4 = make_float4(m01.x / i01.x, m01.y / i01.y, m23.x / i23.x, m23.y / i23.y);
        }
        *reinterpret_cast<float4*>(a.mu_T + off) = m4;
        *reinterpret_cast<float4*>(a.I_T + off) = make_float4(i01.x, i01.y, i23.x, i23.y);
      }
    }
  }
  if (__any_sync(0xffffffffu, domain_bad) && lane == 0) latch_status(a.status, kStatusDomain);
}

// ------------------------------------------------------------------ pass A
// Segment summary for segments 0 .. S-2: with W_t = prod_{u > t in segment} alpha_u,
//   dM    = sum_t W_t (beta_t v_t) (x) k_t,
//   dIbar = sum_t W_t beta_t (x) k_t^2,
//   Gamma = prod_{t in segment} alpha_t,
// so that the state after the segment is Gamma * state_before + (dM, dIbar)
// (slide 9: both natural-parameter recurrences are affine with the shared
// scalar decay alpha). Chunks are staged and processed from the segment's end
// backwards, so W is a running suffix product (it only ever shrinks; no
// quotients of products).
// Output: seg_state[(bh, seg)] = (dM, dIbar), seg_gamma[(bh, seg)] = Gamma.
template <int DK, bool BF16, int RG, int R>
__global__ void __launch_bounds__(RG / (4 * R) * 32)
palimpsa_fwd_summary_kernel(FwdArgs a, int C, int nseg, int seg_len, float* __restrict__ seg_state,
                            float* __restrict__ seg_gamma) {
  constexpr int NV = DK / 32;
  constexpr int NTH = RG / (4 * R) * 32;
  constexpr int ES = BF16 ? 2 : 4;
  extern __shared__ __align__(128) unsigned char smem[];

  const int DV = a.d_v;
  // the grid covers segments 0 .. nseg - 2; a packed sequence needs only the
  // summaries of the segments before its own last one (a bad packed sequence
  // is reported by pass C)
  const Tile tl = tile_of(a, RG, nseg - 1, seg_len);
  if (tl.bad || (a.cu_seqlens && tl.seg >= tl.last_seg)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cg = lane & (kLanesPerRow - 1);
  const int rt = lane >> 3;
  const int lr0 = (warp * 4 + rt) * R;

  const FwdSmem L(C, DK, DV, RG, ES);
  const float* kf = reinterpret_cast<const float*>(smem + L.kf);
  const float* k2f = reinterpret_cast<const float*>(smem + L.k2f);
  float* wbvf = reinterpret_cast<float*>(smem + L.bvf);   // W_t beta_t v_t
  float* wbf = reinterpret_cast<float*>(smem + L.bf);     // W_t beta_t
  float* wf = reinterpret_cast<float*>(smem + L.alf);     // W_t
  float* carry = reinterpret_cast<float*>(smem + L.omf);  // [0] = product of alpha after this chunk

  const float A_h = a.A[tl.h];
  const float bsc = a.pro.b_scale ? a.pro.b_scale[tl.h] : 1.f;
  const size_t head_tok = tl.head_tok;
  ChunkPipe<DK, ES> pipe(L, smem, static_cast<const char*>(a.q) + head_tok * DK * ES,
                         static_cast<const char*>(a.k) + head_tok * DK * ES,
                         static_cast<const char*>(a.v) + head_tok * DV * ES,
                         static_cast<const char*>(a.beta) + head_tok * DV * ES, C, tl.tb, tl.tn, DV, true);
  if (threadIdx.x == 0) carry[0] = 1.f;
  pipe.init(a.withhold_first_copy != 0);

  float2 dI[R][2 * NV], dM[R][2 * NV];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int j = 0; j < 2 * NV; ++j) { dI[r][j] = make_float2(0.f, 0.f); dM[r][j] = make_float2(0.f, 0.f); }

  const float* gd = a.d_t + head_tok + tl.tb;
  // d_t one chunk ahead (warp 0, lane t = token t), so its load lands during a chunk of compute
  float d_next = 0.f;
  if (warp == 0 && pipe.nch > 0 && lane < pipe.tc_of(0)) d_next = gd[pipe.t0_of(0) + lane];
  for (int c = 0; c < pipe.nch; ++c) {
    const int tc = pipe.tc_of(c);
    const float d_cur = d_next;
    if (warp == 0 && c + 1 < pipe.nch && lane < pipe.tc_of(c + 1)) d_next = gd[pipe.t0_of(c + 1) + lane];
    if (!pipe.wait(c, a.wait_timeout_ns, a.status)) return;
    const unsigned char* raw = pipe.raw(c);
    // suffix products inside the chunk (warp 0; at most 32 tokens per chunk):
    // W_t = carry * prod_{t < u < tc} alpha_u
    if (warp == 0) {
      float d = lane < tc ? d_cur : 0.f;
      if (a.pro.on) d = softplus_f(d);
      const float al = lane < tc ? expf(-A_h * d) : 1.f;
      float p = al;  // inclusive suffix product prod_{u >= lane}
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_down_sync(0xffffffffu, p, off);
        if (lane + off < 32) p *= o;
      }
      const float excl = __shfl_down_sync(0xffffffffu, p, 1);
      const float cin = carry[0];
      if (lane < tc) wf[lane] = cin * (lane + 1 < tc ? excl : 1.f);
      __syncwarp();
      if (lane == 0) carry[0] = cin * p;  // lane 0 holds the product over the whole chunk
    }
    convert_keys<DK, BF16, false, NTH>(raw, L, smem, tc, a.pro.qk_norm);
    __syncthreads();  // W_t ready
    for (int it = threadIdx.x; it < tc * RG; it += NTH) {
      const int t = it / RG, r = it % RG;
      const size_t e = (size_t)t * DV + tl.row0 + r;
      const float vv = raw_elem<BF16>(raw + L.raw_v, e);
      float bb = raw_elem<BF16>(raw + L.raw_b, e);
      if (a.pro.on) bb = bsc * sigmoid_f(bb);
      const float w = wf[t];
      wbvf[it] = w * (a.pro.v_star ? vv : bb * vv);
      wbf[it] = w * bb;
    }
    __syncthreads();
    pipe.refill(c);
    for (int t = tc - 1; t >= 0; --t) {
      float wb[R], wbv[R];
#pragma unroll
      for (int r = 0; r < R; ++r) { wb[r] = wbf[t * RG + lr0 + r]; wbv[r] = wbvf[t * RG + lr0 + r]; }
#pragma unroll
      for (int s = 0; s < NV; ++s) {
        const int col = 32 * s + 4 * cg;
        const float4 k4 = *reinterpret_cast<const float4*>(kf + t * DK + col);
        const float4 kk4 = *reinterpret_cast<const float4*>(k2f + t * DK + col);
        const float2 kp[2] = {make_float2(k4.x, k4.y), make_float2(k4.z, k4.w)};
        const float2 kkp[2] = {make_float2(kk4.x, kk4.y), make_float2(kk4.z, kk4.w)};
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            dM[r][2 * s + p] = __ffma2_rn(f2(wbv[r]), kp[p], dM[r][2 * s + p]);
            dI[r][2 * s + p] = __ffma2_rn(f2(wb[r]), kkp[p], dI[r][2 * s + p]);
          }
        }
      }
    }
    // (the barrier at the top of the next chunk orders these reads before the
    // next conversion overwrites the operands)
  }

  float* out = seg_state + ((size_t)tl.bh * (nseg - 1) + tl.seg) * 2 * DV * DK;
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int s = 0; s < NV; ++s) {
      const size_t e = (size_t)(tl.row0 + lr0 + r) * DK + 32 * s + 4 * cg;
      const float2 m01 = dM[r][2 * s], m23 = dM[r][2 * s + 1], i01 = dI[r][2 * s], i23 = dI[r][2 * s + 1];
      *reinterpret_cast<float4*>(out + e) = make_float4(m01.x, m01.y, m23.x, m23.y);
      *reinterpret_cast<float4*>(out + (size_t)DV * DK + e) = make_float4(i01.x, i01.y, i23.x, i23.y);
    }
  }
  __syncthreads();  // carry[0] final (written by warp 0 in the last chunk)
  if (threadIdx.x == 0 && tl.row0 == 0) seg_gamma[(size_t)tl.bh * (nseg - 1) + tl.seg] = carry[0];
}

// ------------------------------------------------------------------ pass B
// Carry across segments, per state element (in place over the summaries):
//   (M, Ibar)_0 = (I0 mu0, I0 - I_prior)   (mu0 = 0 and I0 = I_prior when absent)
//   (M, Ibar)_{s+1} = Gamma_s (M, Ibar)_s + summary_s,   s = 0 .. S-2,
// leaving in slot s the state at the start of segment s + 1.
__global__ void __launch_bounds__(256)
palimpsa_fwd_carry_kernel(FwdArgs a, int nseg, int seg_len, float* __restrict__ seg_state,
                          const float* __restrict__ seg_gamma) {
  const long per_head = (long)a.d_v * a.d_k / 4;  // float4 quads per array
  const long q = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= (long)a.B * a.H * per_head) return;
  const long bh = q / per_head;
  const long e = (q % per_head) * 4;
  const int h = (int)(bh % a.H);
  int L = 0;
  size_t first_tok = 0;
  if (!seq_extent(a, bh, &L, &first_tok)) return;  // reported by pass C
  // boundaries this sequence uses: those before its last segment
  const int nb = min(nseg - 1, L > 0 ? (L - 1) / seg_len : 0);
  const float Ip = a.I_prior[h];
  const size_t DVK = (size_t)a.d_v * a.d_k;
  const size_t off = (size_t)bh * DVK + e;
  const float4 i0 = a.I0 ? *reinterpret_cast<const float4*>(a.I0 + off) : make_float4(Ip, Ip, Ip, Ip);
  const float4 u = a.mu0 ? *reinterpret_cast<const float4*>(a.mu0 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 m = make_float4(i0.x * u.x, i0.y * u.y, i0.z * u.z, i0.w * u.w);
  float4 ib = make_float4(i0.x - Ip, i0.y - Ip, i0.z - Ip, i0.w - Ip);
  float* init = seg_state + SplitScratch((long long)a.B * a.H, nseg, (long long)DVK).init + (size_t)bh * 2 * DVK;
  *reinterpret_cast<float4*>(init + e) = m;
  *reinterpret_cast<float4*>(init + DVK + e) = i0;
  // the summaries come from pass A, which may still be running (programmatic
  // dependent launch); pass C may be scheduled from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int s = 0; s < nb; ++s) {
    const float g = seg_gamma[(size_t)bh * (nseg - 1) + s];
    float* slot = seg_state + ((size_t)bh * (nseg - 1) + s) * 2 * DVK;
    const float4 dm = *reinterpret_cast<const float4*>(slot + e);
    const float4 di = *reinterpret_cast<const float4*>(slot + DVK + e);
    m = make_float4(fmaf(g, m.x, dm.x), fmaf(g, m.y, dm.y), fmaf(g, m.z, dm.z), fmaf(g, m.w, dm.w));
    ib = make_float4(fmaf(g, ib.x, di.x), fmaf(g, ib.y, di.y), fmaf(g, ib.z, di.z), fmaf(g, ib.w, di.w));
    *reinterpret_cast<float4*>(slot + e) = m;
    *reinterpret_cast<float4*>(slot + DVK + e) = ib;
  }
}

// ------------------------------------------------------------------ host side

// A launch that may start while the kernel before it in the stream drains
// (programmatic dependent launch); the kernel waits (griddepcontrol.wait)
// before it reads what that kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr int kRowsPerThread = 2;

template <int DK, bool BF16, int RG>
struct Kernels {
  static constexpr int kThreads = RG / (4 * kRowsPerThread) * 32;
  static size_t smem(const FwdArgs& a, int C) { return FwdSmem(C, DK, a.d_v, RG, BF16 ? 2 : 4).total; }

  static int ctas_per_sm(const FwdArgs& a, int C) {
    return C == 16 ? ctas_per_sm_c<16>(a) : ctas_per_sm_c<32>(a);
  }
  template <int CC>
  static int ctas_per_sm_c(const FwdArgs& a) {
    auto kern = palimpsa_fwd_chunked_kernel<DK, BF16, RG, kRowsPerThread, CC>;
    const size_t sm = smem(a, CC);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess) return 1;
    int n = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, sm) != cudaSuccess || n < 1) n = 1;
    return n;
  }

  // The chunk is 16 or 32 tokens (the planner's choice).
  static cudaError_t run(const FwdArgs& a, int C, int nseg, int seg_len, float* scratch, cudaStream_t s) {
    return C == 16 ? run_c<16>(a, nseg, seg_len, scratch, s) : run_c<32>(a, nseg, seg_len, scratch, s);
  }
  template <int CC>
  static cudaError_t run_c(const FwdArgs& a, int nseg, int seg_len, float* scratch, cudaStream_t s) {
    const size_t sm = smem(a, CC);
    const long groups = a.d_v / RG;
    const long heads = (long)a.B * a.H;
    auto main_k = palimpsa_fwd_chunked_kernel<DK, BF16, RG, kRowsPerThread, CC>;
    cudaError_t e = cudaFuncSetAttribute(main_k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    if (nseg > 1 && (e = prefix(a, CC, nseg, seg_len, scratch, s)) != cudaSuccess) return e;
    if (nseg > 1) {
      e = launch_dependent(main_k, dim3((unsigned)(heads * nseg * groups)), dim3(kThreads), sm, s, a, nseg, seg_len,
                           (const float*)scratch);
      return e != cudaSuccess ? e : cudaGetLastError();
    }
    main_k<<<(unsigned)(heads * nseg * groups), kThreads, sm, s>>>(a, nseg, seg_len, scratch);
    return cudaGetLastError();
  }

  // Passes A and B: the state at the start of segments 1 .. nseg - 1 of every
  // head into scratch[(bh, seg - 1)] as (M, Ibar).
  static cudaError_t prefix(const FwdArgs& a, int C, int nseg, int seg_len, float* scratch, cudaStream_t s) {
    const long heads = (long)a.B * a.H;
    float* seg_gamma = scratch + SplitScratch(heads, nseg, (long long)a.d_v * a.d_k).gammas;
    cudaError_t e = summaries(a, C, nseg - 1, seg_len, scratch, seg_gamma, s);
    if (e != cudaSuccess) return e;
    const long quads = heads * a.d_v * a.d_k / 4;
    e = launch_dependent(palimpsa_fwd_carry_kernel, dim3((unsigned)((quads + 255) / 256)), dim3(256), 0, s, a, nseg,
                         seg_len, scratch, (const float*)seg_gamma);
    return e != cudaSuccess ? e : cudaGetLastError();
  }

  // Pass A over segments 0 .. nseg - 1 of every head (summary slots [bh][seg]):
  // on the tensor cores where the inputs allow, else with FFMA.
  static cudaError_t summaries(const FwdArgs& a, int C, int nseg, int seg_len, float* st, float* gm,
                               cudaStream_t s) {
    if (summary_tc_eligible(a)) return launch_summary_tc(a, nseg, seg_len, st, gm, s);
    const size_t sm = smem(a, C);
    auto sum_k = palimpsa_fwd_summary_kernel<DK, BF16, RG, kRowsPerThread>;
    cudaError_t e = cudaFuncSetAttribute(sum_k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    const long units = (long)a.B * a.H * nseg * (a.d_v / RG);
    sum_k<<<(unsigned)units, kThreads, sm, s>>>(a, C, nseg + 1, seg_len, st, gm);
    return cudaGetLastError();
  }
};

struct Plan {
  int RG, C, nseg, seg_len;
};

// Rows per CTA: 64 where d_v allows (the staging work per CTA is then shared
// by the most rows), else the largest of {32, 16, 8} dividing d_v.
int rows_per_cta(int d_v) {
  for (int c : {64, 32, 16, 8})
    if (d_v % c == 0) return c;
  return 8;
}

// Segments: minimise a cost model of the whole forward, in units of one pass-C
// token-step of one wave of resident CTAs. Constants were measured on GB300
// (two 256-thread CTAs per SM): a pass-A token-step costs 0.46 of a pass-C one;
// each wave of either pass pays ~3 units of fill and drain; the carry kernel
// streams (read + write) 16 d_v d_k bytes per head and segment boundary at
// ~6.3 TB/s (2.24e-7 units per byte); the two extra launches cost ~15 units.
// A pass over U CTAs on `slots` resident CTA slots takes ceil(U / slots) waves.
void choose_segments(const FwdArgs& a, long units_per_seg, int slots, int C, Plan* p) {
  constexpr double kPassA = 0.46, kWave = 3.0, kCarryPerByte = 2.24e-7, kSplitFixed = 15.0;
  const long T = a.T;
  p->nseg = 1;
  p->seg_len = a.T > 0 ? a.T : 1;
  if (T <= 2L * C) return;
  const double carry_bytes_per_boundary = 16.0 * a.d_v * a.d_k * ((double)a.B * a.H);
  double best = 1e300;
  const int max_seg = (int)std::min<long>(256, T / C);
  for (int S = 1; S <= max_seg; ++S) {
    const long len = (T + S - 1) / S;
    const long len_c = (len + C - 1) / C * C;  // whole chunks per segment
    const long nseg = (T + len_c - 1) / len_c;
    if (nseg != S) continue;
    const double wC = std::ceil((double)units_per_seg * nseg / slots);
    double cost = wC * ((double)len_c + kWave);
    if (nseg > 1) {
      const double wA = std::ceil((double)units_per_seg * (nseg - 1) / slots);
      cost += wA * (kPassA * (double)len_c + kWave) + kCarryPerByte * carry_bytes_per_boundary * (nseg - 1) +
              kSplitFixed;
    }
    if (cost < best) {
      best = cost;
      p->nseg = (int)nseg;
      p->seg_len = (int)len_c;
    }
  }
}

template <int DK, bool BF16>
Plan plan_segments(const FwdArgs& a, Plan p) {
  int dev = 0, num_sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  int per_sm = 1;
  switch (p.RG) {
    case 64: per_sm = Kernels<DK, BF16, 64>::ctas_per_sm(a, p.C); break;
    case 32: per_sm = Kernels<DK, BF16, 32>::ctas_per_sm(a, p.C); break;
    case 16: per_sm = Kernels<DK, BF16, 16>::ctas_per_sm(a, p.C); break;
    default: per_sm = Kernels<DK, BF16, 8>::ctas_per_sm(a, p.C); break;
  }
  const long heads = (long)a.B * a.H;
  const long units = heads * (a.d_v / p.RG);
  if (a.force_segments > 0 && a.T > 0) {
    const long len = ((long)a.T + a.force_segments - 1) / a.force_segments;
    p.seg_len = (int)((len + p.C - 1) / p.C * p.C);
    p.nseg = (int)(((long)a.T + p.seg_len - 1) / p.seg_len);
  } else {
    choose_segments(a, units, num_sms * per_sm, p.C, &p);
  }
  return p;
}

template <int DK, bool BF16>
cudaError_t plan_and_run(const FwdArgs& a, Plan p, cudaStream_t s, ScratchProvider* sp) {
  p = plan_segments<DK, BF16>(a, p);
  const long heads = (long)a.B * a.H;
  float* scratch = nullptr;
  if (p.nseg > 1) {
    const size_t bytes = SplitScratch(heads, p.nseg, (long long)a.d_v * a.d_k).total * sizeof(float);
    cudaError_t e = sp->acquire(bytes, s, &scratch);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e;
  switch (p.RG) {
    case 64: e = Kernels<DK, BF16, 64>::run(a, p.C, p.nseg, p.seg_len, scratch, s); break;
    case 32: e = Kernels<DK, BF16, 32>::run(a, p.C, p.nseg, p.seg_len, scratch, s); break;
    case 16: e = Kernels<DK, BF16, 16>::run(a, p.C, p.nseg, p.seg_len, scratch, s); break;
    default: e = Kernels<DK, BF16, 8>::run(a, p.C, p.nseg, p.seg_len, scratch, s); break;
  }
  if (scratch) {
    const cudaError_t e2 = sp->release(scratch, s);
    if (e == cudaSuccess) e = e2;
  }
  return e;
}

// The summary of each head's whole range: pass A over the planned segments
// straight into (summary, gamma) when there is one segment, else into scratch
// and then folded.
template <int DK, bool BF16>
cudaError_t summary_plan_and_run(const FwdArgs& a, Plan p, float* summary, float* gamma, cudaStream_t s,
                                 ScratchProvider* sp) {
  p = plan_segments<DK, BF16>(a, p);
  auto pass_a = [&](float* st, float* gm) -> cudaError_t {
    switch (p.RG) {
      case 64: return Kernels<DK, BF16, 64>::summaries(a, p.C, p.nseg, p.seg_len, st, gm, s);
      case 32: return Kernels<DK, BF16, 32>::summaries(a, p.C, p.nseg, p.seg_len, st, gm, s);
      case 16: return Kernels<DK, BF16, 16>::summaries(a, p.C, p.nseg, p.seg_len, st, gm, s);
      default: return Kernels<DK, BF16, 8>::summaries(a, p.C, p.nseg, p.seg_len, st, gm, s);
    }
  };
  if (p.nseg == 1) return pass_a(summary, gamma);
  const long heads = (long)a.B * a.H;
  const long long DVK = (long long)a.d_v * a.d_k;
  float* scratch = nullptr;
  cudaError_t e = sp->acquire((size_t)heads * p.nseg * (2 * DVK + 1) * sizeof(float), s, &scratch);
  if (e != cudaSuccess) return e;
  float* gm = scratch + (size_t)heads * p.nseg * 2 * DVK;
  e = pass_a(scratch, gm);
  if (e == cudaSuccess) {
    // slot (bh, seg) of the scratch: states at (bh * nseg + seg) * 2 DVK, gammas at bh * nseg + seg
    const FoldArgs f{scratch, gm, 2 * DVK, (long long)p.nseg * 2 * DVK, 1, p.nseg, p.nseg, heads, a.H,
                     (int)DVK, false, a.I_prior, nullptr, nullptr, summary, summary + DVK, gamma, 2 * DVK};
    e = launch_fold(f, s);
  }
  const cudaError_t e2 = sp->release(scratch, s);
  return e != cudaSuccess ? e : e2;
}

Plan base_plan(const FwdArgs& a, int max_smem, bool* ok) {
  Plan p;
  p.RG = rows_per_cta(a.d_v);
  const int es = a.bf16 ? 2 : 4;
  // Chunk: at most 32 tokens (pass A computes a chunk's suffix products in one
  // warp), shrunk until two CTAs' staging (with the per-CTA reserve) fits an
  // SM: registers allow two pass-C CTAs per SM, and longer chunks halve the
  // barriers per token (32 against 16 tokens: 3-4 % faster on GB300).
  p.C = std::min(a.chunk, 32);
  while (p.C > 16 && FwdSmem(p.C, a.d_k, a.d_v, p.RG, es).total + 1024 > (size_t)max_smem / 2) p.C /= 2;
  *ok = FwdSmem(p.C, a.d_k, a.d_v, p.RG, es).total <= (size_t)max_smem;
  p.nseg = 1;
  p.seg_len = a.T;
  return p;
}

int max_smem_optin() {
  int dev = 0, max_smem = 227 * 1024;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return max_smem;
}

}  // namespace

cudaError_t launch_forward_chunked(const FwdArgs& a, cudaStream_t s, ScratchProvider* sp) {
  bool ok = false;
  const Plan p = base_plan(a, max_smem_optin(), &ok);
  if (!ok) return cudaErrorInvalidConfiguration;
  if (a.d_k == 128) return a.bf16 ? plan_and_run<128, true>(a, p, s, sp) : plan_and_run<128, false>(a, p, s, sp);
  return a.bf16 ? plan_and_run<64, true>(a, p, s, sp) : plan_and_run<64, false>(a, p, s, sp);
}

cudaError_t launch_split_prefix(const FwdArgs& a, int nseg, int seg_len, float* scratch, cudaStream_t s) {
  bool ok = false;
  const Plan p = base_plan(a, max_smem_optin(), &ok);
  if (!ok) return cudaErrorInvalidConfiguration;
  auto go = [&](auto tag) -> cudaError_t {
    using K = decltype(tag);
    return K::prefix(a, p.C, nseg, seg_len, scratch, s);
  };
  if (a.d_k == 128) {
    if (a.bf16) {
      switch (p.RG) {
        case 64: return go(Kernels<128, true, 64>{});
        case 32: return go(Kernels<128, true, 32>{});
        case 16: return go(Kernels<128, true, 16>{});
        default: return go(Kernels<128, true, 8>{});
      }
    }
    switch (p.RG) {
      case 64: return go(Kernels<128, false, 64>{});
      case 32: return go(Kernels<128, false, 32>{});
      case 16: return go(Kernels<128, false, 16>{});
      default: return go(Kernels<128, false, 8>{});
    }
  }
  if (a.bf16) {
    switch (p.RG) {
      case 64: return go(Kernels<64, true, 64>{});
      case 32: return go(Kernels<64, true, 32>{});
      case 16: return go(Kernels<64, true, 16>{});
      default: return go(Kernels<64, true, 8>{});
    }
  }
  switch (p.RG) {
    case 64: return go(Kernels<64, false, 64>{});
    case 32: return go(Kernels<64, false, 32>{});
    case 16: return go(Kernels<64, false, 16>{});
    default: return go(Kernels<64, false, 8>{});
  }
}

cudaError_t plan_forward(const FwdArgs& a, int* nseg, int* seg_len) {
  bool ok = false;
  Plan p = base_plan(a, max_smem_optin(), &ok);
  if (!ok) return cudaErrorInvalidConfiguration;
  if (a.d_k == 128) p = a.bf16 ? plan_segments<128, true>(a, p) : plan_segments<128, false>(a, p);
  else p = a.bf16 ? plan_segments<64, true>(a, p) : plan_segments<64, false>(a, p);
  *nseg = p.nseg;
  *seg_len = p.seg_len;
  return cudaGetLastError();
}

cudaError_t launch_segment_summary(const FwdArgs& a, float* summary, float* gamma, cudaStream_t s,
                                   ScratchProvider* sp) {
  bool ok = false;
  const Plan p = base_plan(a, max_smem_optin(), &ok);
  if (!ok) return cudaErrorInvalidConfiguration;
  if (a.d_k == 128)
    return a.bf16 ? summary_plan_and_run<128, true>(a, p, summary, gamma, s, sp)
                  : summary_plan_and_run<128, false>(a, p, summary, gamma, s, sp);
  return a.bf16 ? summary_plan_and_run<64, true>(a, p, summary, gamma, s, sp)
                : summary_plan_and_run<64, false>(a, p, summary, gamma, s, sp);
}

}  // namespace palimpsa
