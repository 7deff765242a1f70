// Chunked forward of the Palimpsa recurrence on sm_103a.
//
// Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
// Attention-Based Models" — slide 7 (paper Eq. 5) for the update, slide 4
// (Eq. 2) for the readout, slide 9 (App. A.12) for the natural parameters
// M = I (.) mu and the chunked scan with a sequential carry between chunks.
//
// Design (GB300-first, not the pages' Triton kernel):
// * The state of one value row i is 2 x d_k fp32 numbers (M_ij and I_ij). A CTA
//   owns RG rows of one head for the whole sequence and keeps their state in
//   registers: nothing of the state touches HBM between the first read and
//   the final write, so there is no per-chunk state traffic at all.
// * Thread tile: 2 rows x (d_k / 8) columns. The 8 lanes of a "row team" split
//   the key dimension; lane cg owns the float4 column blocks 32 s + 4 cg, so a
//   warp's shared-memory reads of k, k^2 and q are one 128-byte wavefront that
//   every row team of the warp shares (broadcast).
// * The inputs of a chunk of C tokens are staged by the bulk-copy (TMA) engine
//   into a double buffer (cp.async.bulk + mbarrier with a bounded wait), then
//   converted once per CTA into fp32 k, k^2, q, beta v, beta, alpha and
//   (1 - alpha) I_prior, shared by all the CTA's rows.
// * Per state element and token the arithmetic is
//       c = beta_i k_j^2 + (1 - alpha) I_prior      (FFMA)
//       I = alpha I + c                             (FFMA)
//       M = alpha M + (beta_i v_i) k_j              (FMUL + FFMA)
//       y_i += (M * rcp(I)) q_j                     (MUFU.RCP, FMUL + FFMA)
//   issued as packed f32x2 instructions over adjacent key columns, so the
//   kernel is bound by the reciprocal (SFU) pipe, not by issue.
// * y_{t,i} is reduced over the row team with three butterfly shuffles,
//   staged per chunk in shared memory and stored with coalesced 16-byte stores.
#include "palimpsa_internal.cuh"

namespace palimpsa {
namespace {

constexpr int kRowsPerThread = 2;
constexpr int kLanesPerRow = 8;

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory carve-up for one CTA (all offsets 16-byte aligned).
struct FwdSmem {
  size_t raw_bytes;  // one raw buffer (q, k, v, beta of one chunk)
  size_t raw_q, raw_k, raw_v, raw_b;  // offsets inside a raw buffer
  size_t kf, k2f, qf, bvf, bf, alf, omf, ys, bars, flag, total;

  __host__ __device__ FwdSmem(int C, int DK, int DV, int RG, int es) {
    raw_q = 0;
    raw_k = align_up(raw_q + (size_t)C * DK * es, 16);
    raw_v = align_up(raw_k + (size_t)C * DK * es, 16);
    raw_b = align_up(raw_v + (size_t)C * DV * es, 16);
    raw_bytes = align_up(raw_b + (size_t)C * DV * es, 128);
    size_t o = 2 * raw_bytes;
    kf = o;  o = align_up(o + (size_t)C * DK * 4, 16);
    k2f = o; o = align_up(o + (size_t)C * DK * 4, 16);
    qf = o;  o = align_up(o + (size_t)C * DK * 4, 16);
    bvf = o; o = align_up(o + (size_t)C * RG * 4, 16);
    bf = o;  o = align_up(o + (size_t)C * RG * 4, 16);
    alf = o; o = align_up(o + (size_t)C * 4, 16);
    omf = o; o = align_up(o + (size_t)C * 4, 16);
    ys = o;  o = align_up(o + (size_t)C * RG * 4, 16);
    bars = o; o += 2 * sizeof(uint64_t);
    flag = o; o += 16;
    total = align_up(o, 128);
  }
};

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// Producer side (one thread): stage chunk n's q, k, v, beta into one raw
// buffer with four bulk copies whose bytes complete on `bar`.
template <int DK, int ES>
__device__ __forceinline__ void stage_chunk(unsigned char* base, const FwdSmem& L, uint64_t* bar,
                                            const char* gq, const char* gk, const char* gv,
                                            const char* gb, int n, int C, int T, int DV) {
  const int t0 = n * C;
  const int tc = min(C, T - t0);
  const uint32_t bq = (uint32_t)tc * DK * ES, bvb = (uint32_t)tc * DV * ES;
  mbar_arrive_expect_tx(bar, 2 * bq + 2 * bvb);
  bulk_g2s(base + L.raw_q, gq + (size_t)t0 * DK * ES, bq, bar);
  bulk_g2s(base + L.raw_k, gk + (size_t)t0 * DK * ES, bq, bar);
  bulk_g2s(base + L.raw_v, gv + (size_t)t0 * DV * ES, bvb, bar);
  bulk_g2s(base + L.raw_b, gb + (size_t)t0 * DV * ES, bvb, bar);
}

template <int DK, bool BF16, int RG>
__global__ void __launch_bounds__(RG * 4)
palimpsa_fwd_chunked_kernel(FwdArgs a, int C) {
  constexpr int NV = DK / 32;          // float4 column blocks per thread
  constexpr int NTH = RG * 4;          // threads per CTA
  constexpr int ES = BF16 ? 2 : 4;     // input element size
  extern __shared__ __align__(128) unsigned char smem[];

  const int DV = a.d_v, T = a.T;
  const int groups = DV / RG;
  const long bh = blockIdx.x / groups;
  const int row0 = (blockIdx.x % groups) * RG;
  const int h = (int)(bh % a.H);
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int cg = lane & (kLanesPerRow - 1);
  const int rt = lane >> 3;
  const int lr0 = warp * 8 + rt * kRowsPerThread;  // first local row of this thread

  const FwdSmem L(C, DK, DV, RG, ES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  volatile int* sflag = reinterpret_cast<volatile int*>(smem + L.flag);
  float* kf = reinterpret_cast<float*>(smem + L.kf);
  float* k2f = reinterpret_cast<float*>(smem + L.k2f);
  float* qf = reinterpret_cast<float*>(smem + L.qf);
  float* bvf = reinterpret_cast<float*>(smem + L.bvf);
  float* bfv = reinterpret_cast<float*>(smem + L.bf);
  float* alf = reinterpret_cast<float*>(smem + L.alf);
  float* omf = reinterpret_cast<float*>(smem + L.omf);
  float* ys = reinterpret_cast<float*>(smem + L.ys);

  const float A_h = a.A[h];
  const float Ip = a.I_prior[h];
  bool domain_bad = !(pos_finite(A_h) && pos_finite(Ip));

  const int nchunks = (T + C - 1) / C;
  const char* gq = static_cast<const char*>(a.q) + (size_t)bh * T * DK * ES;
  const char* gk = static_cast<const char*>(a.k) + (size_t)bh * T * DK * ES;
  const char* gv = static_cast<const char*>(a.v) + (size_t)bh * T * DV * ES;
  const char* gb = static_cast<const char*>(a.beta) + (size_t)bh * T * DV * ES;
  const float* gd = a.d_t + (size_t)bh * T;

  // Thread 0's record of copies issued but not yet consumed, per raw buffer,
  // with the barrier phase that will signal them.
  bool pending0 = false, pending1 = false;
  uint32_t parity0 = 0u, parity1 = 0u;
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *sflag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    if (nchunks > 0 && !a.withhold_first_copy) {
      stage_chunk<DK, ES>(smem, L, &bars[0], gq, gk, gv, gb, 0, C, T, DV);
      pending0 = true; parity0 = 0u;
    }
    if (nchunks > 1) {
      stage_chunk<DK, ES>(smem + L.raw_bytes, L, &bars[1], gq, gk, gv, gb, 1, C, T, DV);
      pending1 = true; parity1 = 0u;
    }
  }

  // ---- initial state: M = I0 (.) mu0, I = I0 (defaults mu0 = 0, I0 = I_prior)
  float2 Ist[kRowsPerThread][2 * NV], Mst[kRowsPerThread][2 * NV];
  const size_t state_base = ((size_t)bh * DV + row0) * DK;
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
#pragma unroll
    for (int s = 0; s < NV; ++s) {
      const size_t off = state_base + (size_t)(lr0 + r) * DK + 32 * s + 4 * cg;
      float4 i4 = a.I0 ? *reinterpret_cast<const float4*>(a.I0 + off) : make_float4(Ip, Ip, Ip, Ip);
      float4 m4 = a.mu0 ? *reinterpret_cast<const float4*>(a.mu0 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
      domain_bad |= !(pos_finite(i4.x) && pos_finite(i4.y) && pos_finite(i4.z) && pos_finite(i4.w));
      Ist[r][2 * s] = make_float2(i4.x, i4.y);
      Ist[r][2 * s + 1] = make_float2(i4.z, i4.w);
      Mst[r][2 * s] = make_float2(i4.x * m4.x, i4.y * m4.y);
      Mst[r][2 * s + 1] = make_float2(i4.z * m4.z, i4.w * m4.w);
    }
  }

  for (int n = 0; n < nchunks; ++n) {
    const int t0 = n * C;
    const int tc = min(C, T - t0);
    const int buf = n & 1;
    if (!mbar_wait_bounded(&bars[buf], (n >> 1) & 1, a.wait_timeout_ns)) *sflag = 1;
    __syncthreads();
    if (*sflag) {
      // A staged copy never arrived: report, let copies still in flight land, leave.
      if (tid == 0) {
        latch_status(a.status, kStatusTimeout);
        const unsigned long long drain_ns = 1000000000ull;
        if (pending0) mbar_wait_bounded(&bars[0], parity0, drain_ns);
        if (pending1) mbar_wait_bounded(&bars[1], parity1, drain_ns);
      }
      __syncthreads();
      return;
    }

    // ---- convert the staged chunk to fp32 operands shared by all rows
    const unsigned char* raw = smem + (size_t)buf * L.raw_bytes;
    {
      constexpr int PER = 8;  // elements per work item (16 B of bf16, 32 B of fp32)
      const int items = tc * DK / PER;
      for (int it = tid; it < items; it += NTH) {
        float qv[PER], kv[PER];
        if constexpr (BF16) {
          const uint4 q8 = *reinterpret_cast<const uint4*>(raw + L.raw_q + (size_t)it * 16);
          const uint4 k8 = *reinterpret_cast<const uint4*>(raw + L.raw_k + (size_t)it * 16);
          const uint32_t qw[4] = {q8.x, q8.y, q8.z, q8.w}, kw[4] = {k8.x, k8.y, k8.z, k8.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qv[2 * e] = bf16_lo(qw[e]); qv[2 * e + 1] = bf16_hi(qw[e]);
            kv[2 * e] = bf16_lo(kw[e]); kv[2 * e + 1] = bf16_hi(kw[e]);
          }
        } else {
          const float4* q4 = reinterpret_cast<const float4*>(raw + L.raw_q) + 2 * it;
          const float4* k4 = reinterpret_cast<const float4*>(raw + L.raw_k) + 2 * it;
          const float4 qa = q4[0], qb = q4[1], ka = k4[0], kb = k4[1];
          qv[0] = qa.x; qv[1] = qa.y; qv[2] = qa.z; qv[3] = qa.w;
          qv[4] = qb.x; qv[5] = qb.y; qv[6] = qb.z; qv[7] = qb.w;
          kv[0] = ka.x; kv[1] = ka.y; kv[2] = ka.z; kv[3] = ka.w;
          kv[4] = kb.x; kv[5] = kb.y; kv[6] = kb.z; kv[7] = kb.w;
        }
        float4* qo = reinterpret_cast<float4*>(qf) + 2 * it;
        float4* ko = reinterpret_cast<float4*>(kf) + 2 * it;
        float4* k2o = reinterpret_cast<float4*>(k2f) + 2 * it;
        qo[0] = make_float4(qv[0], qv[1], qv[2], qv[3]);
        qo[1] = make_float4(qv[4], qv[5], qv[6], qv[7]);
        ko[0] = make_float4(kv[0], kv[1], kv[2], kv[3]);
        ko[1] = make_float4(kv[4], kv[5], kv[6], kv[7]);
        k2o[0] = make_float4(kv[0] * kv[0], kv[1] * kv[1], kv[2] * kv[2], kv[3] * kv[3]);
        k2o[1] = make_float4(kv[4] * kv[4], kv[5] * kv[5], kv[6] * kv[6], kv[7] * kv[7]);
      }
      for (int it = tid; it < tc * RG; it += NTH) {
        const int t = it / RG, r = it % RG;
        const size_t e = (size_t)t * DV + row0 + r;
        float vv, bb;
        if constexpr (BF16) {
          vv = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(raw + L.raw_v)[e]);
          bb = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(raw + L.raw_b)[e]);
        } else {
          vv = reinterpret_cast<const float*>(raw + L.raw_v)[e];
          bb = reinterpret_cast<const float*>(raw + L.raw_b)[e];
        }
        domain_bad |= !nonneg_finite(bb);
        bvf[it] = bb * vv;
        bfv[it] = bb;
      }
      for (int t = tid; t < tc; t += NTH) {
        const float d = gd[t0 + t];
        domain_bad |= !nonneg_finite(d);
        const float x = -A_h * d;
        alf[t] = expf(x);
        omf[t] = -expm1f(x) * Ip;  // (1 - alpha) I_prior without cancellation
      }
    }
    __syncthreads();
    // raw[buf] is consumed: refill it with chunk n + 2 while this chunk computes.
    if (tid == 0) {
      const bool more = n + 2 < nchunks;
      if (more) stage_chunk<DK, ES>(smem + (size_t)buf * L.raw_bytes, L, &bars[buf], gq, gk, gv, gb, n + 2, C, T, DV);
      const uint32_t par = (uint32_t)((n + 2) >> 1) & 1u;
      if (buf == 0) { pending0 = more; parity0 = par; } else { pending1 = more; parity1 = par; }
    }

    // ---- the recurrence over the chunk's tokens, state in registers
    for (int t = 0; t < tc; ++t) {
      const float al = alf[t], om = omf[t];
      const float2 a2 = f2(al), om2 = f2(om);
      const float2 bb = *reinterpret_cast<const float2*>(bfv + t * RG + lr0);
      const float2 bv = *reinterpret_cast<const float2*>(bvf + t * RG + lr0);
      const float brow[2] = {bb.x, bb.y}, bvrow[2] = {bv.x, bv.y};
      float2 acc[kRowsPerThread];
#pragma unroll
      for (int r = 0; r < kRowsPerThread; ++r) acc[r] = make_float2(0.f, 0.f);
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
        for (int r = 0; r < kRowsPerThread; ++r) {
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
      float y0 = acc[0].x + acc[0].y, y1 = acc[1].x + acc[1].y;
#pragma unroll
      for (int m = 1; m < kLanesPerRow; m <<= 1) {
        y0 += __shfl_xor_sync(0xffffffffu, y0, m);
        y1 += __shfl_xor_sync(0xffffffffu, y1, m);
      }
      if (cg == 0) *reinterpret_cast<float2*>(ys + t * RG + lr0) = make_float2(y0, y1);
    }
    __syncthreads();

    // ---- store the chunk's y rows (RG contiguous fp32 per token)
    {
      float* gy = a.y + ((size_t)bh * T + t0) * DV + row0;
      const int per_t = RG / 4;
      for (int it = tid; it < tc * per_t; it += NTH) {
        const int t = it / per_t, c4 = it % per_t;
        *reinterpret_cast<float4*>(gy + (size_t)t * DV + 4 * c4) =
            *reinterpret_cast<const float4*>(ys + t * RG + 4 * c4);
      }
    }
  }

  // ---- final state: mu_T = M / I, I_T = I (T = 0 passes the initial state through)
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
#pragma unroll
    for (int s = 0; s < NV; ++s) {
      const size_t off = state_base + (size_t)(lr0 + r) * DK + 32 * s + 4 * cg;
      const float2 i01 = Ist[r][2 * s], i23 = Ist[r][2 * s + 1];
      float4 m4;
      if (nchunks == 0) {
        m4 = a.mu0 ? *reinterpret_cast<const float4*>(a.mu0 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        const float2 m01 = Mst[r][2 * s], m23 = Mst[r][2 * s + 1];
        m4 = make_float4(m01.x / i01.x, m01.y / i01.y, m23.x / i23.x, m23.y / i23.y);
      }
      *reinterpret_cast<float4*>(a.mu_T + off) = m4;
      *reinterpret_cast<float4*>(a.I_T + off) = make_float4(i01.x, i01.y, i23.x, i23.y);
    }
  }
  if (domain_bad) latch_status(a.status, kStatusDomain);
}

template <int DK, bool BF16, int RG>
cudaError_t launch_t(const FwdArgs& a, int C, cudaStream_t s) {
  const FwdSmem L(C, DK, a.d_v, RG, BF16 ? 2 : 4);
  auto kern = palimpsa_fwd_chunked_kernel<DK, BF16, RG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
  if (e != cudaSuccess) return e;
  const long ctas = (long)a.B * a.H * (a.d_v / RG);
  kern<<<(unsigned)ctas, RG * 4, L.total, s>>>(a, C);
  return cudaGetLastError();
}

template <int DK, bool BF16>
cudaError_t launch_rg(const FwdArgs& a, int RG, int C, cudaStream_t s) {
  switch (RG) {
    case 64: return launch_t<DK, BF16, 64>(a, C, s);
    case 32: return launch_t<DK, BF16, 32>(a, C, s);
    case 16: return launch_t<DK, BF16, 16>(a, C, s);
    default: return launch_t<DK, BF16, 8>(a, C, s);
  }
}

}  // namespace

// Rows per CTA: the largest of {64, 32, 16, 8} that divides d_v while the grid
// still fills every SM about twice; smaller groups trade duplicated staging
// work for a better balance of CTAs over the 152 SMs.
static int choose_rows_per_cta(const FwdArgs& a, int num_sms) {
  const long heads = (long)a.B * a.H;
  const int cands[4] = {64, 32, 16, 8};
  for (int c : cands) {
    if (a.d_v % c) continue;
    if (heads * (a.d_v / c) >= 2L * num_sms || c == 8) return c;
  }
  return 8;
}

static size_t fwd_smem_bytes(int C, int DK, int DV, int RG, int es) {
  return FwdSmem(C, DK, DV, RG, es).total;
}

cudaError_t launch_forward_chunked(const FwdArgs& a, cudaStream_t s) {
  int dev = 0, num_sms = 152, max_smem = 227 * 1024;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  int RG = choose_rows_per_cta(a, num_sms);
  const int es = a.bf16 ? 2 : 4;
  int C = a.chunk;
  while (C > 16 && fwd_smem_bytes(C, a.d_k, a.d_v, RG, es) > (size_t)max_smem) C /= 2;
  while (RG > 8 && fwd_smem_bytes(C, a.d_k, a.d_v, RG, es) > (size_t)max_smem) RG /= 2;
  if (fwd_smem_bytes(C, a.d_k, a.d_v, RG, es) > (size_t)max_smem) return cudaErrorInvalidConfiguration;
  if (a.d_k == 128) return a.bf16 ? launch_rg<128, true>(a, RG, C, s) : launch_rg<128, false>(a, RG, C, s);
  return a.bf16 ? launch_rg<64, true>(a, RG, C, s) : launch_rg<64, false>(a, RG, C, s);
}

}  // namespace palimpsa
