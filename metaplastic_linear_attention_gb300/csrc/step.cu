// Recurrent (decode) step of the Palimpsa recurrence on sm_103a.
//
// Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
// Attention-Based Models" — slide 22 (paper App. A.13, Fig. 7): recurrent
// inference performs the dual-state update of Eq. (5) (slide 7) and the read
// y = mu q (slide 4, Eq. 2) once per generated token.
//
// The step is a stream over the state: each of the B*H*d_v*d_k elements of mu
// and I is read once and written once (16 bytes per element), against ~1 KB of
// per-head inputs and outputs. It is therefore bound by HBM bandwidth, and the
// kernel is built as a copy kernel with arithmetic in the middle:
// * a CTA is one warp (measured fastest against 2, 4 and 8 warps on GB300:
//   CTAs start and retire independently) and owns 8 value rows of one head;
//   a lane owns 4 consecutive key columns (one 16-byte vector of mu and one
//   of I per row, d_k = 128) or two rows are interleaved per warp instruction
//   (d_k = 64);
// * all 16 state loads of a lane are issued before any arithmetic, so every
//   SM keeps well over the ~45 KB in flight that 6.8 TB/s needs at ~1 us of
//   latency; loads and most stores use the streaming (evict-first) cache
//   policy, because the state (537 MB at B=256, H=32) is far larger than L2;
// * consecutive steps walk the state in opposite orders, and the CTAs that run
//   last store with an evict-last L2 policy instead of streaming: the next
//   step starts on those rows and finds them in L2 (129 MB), saving their DRAM
//   read. The order changes nothing in the results (every row is computed the
//   same way). The kept rows come back interleaved with fresh ones, so DRAM
//   keeps reading while they hit. Measured on GB300 at B=256, H=32: 6 % less
//   time per step with 96 MiB kept;
// * q, k of the head are loaded once per warp; k^2, alpha and (1 - alpha)
//   I_prior once per lane; beta_i (through the prologue when it is on) and
//   beta_i v_i of the warp's 8 rows are formed by 8 lanes, one row each, and
//   handed to the row loop by shuffles, so no lane waits on a load or repeats
//   a gate inside it;
// * y_i is a butterfly shuffle reduction over the lanes of the row;
// * steps are launched with programmatic dependent launch: a step's CTAs can be
//   scheduled while the previous launch drains, and each waits for it
//   (griddepcontrol.wait) before its first read; each triggers the next once
//   its state loads are issued (1-2 % faster per step on GB300).
// The update uses the mean/precision form of Eq. (5) directly:
//   I' = alpha I + (1 - alpha) I_prior + beta_i k_j^2
//   mu' = (alpha I mu + beta_i v_i k_j) / I'
// with IEEE division in the plain step and the fast division (within 2 ulp)
// in the fused one, whose launch bounds also hold it to 128 registers: on
// GB300 each of these choices measured fastest for its variant (the fused
// step compiles to over 128 registers otherwise and loses its second CTA per
// SM).
// The fused variant (PRO, palimpsa_step_fused) first applies the layer's
// prologue to the token's raw inputs: softplus to the gate input, b_scale *
// sigmoid to beta, optionally the L2 norm of q and k (one more butterfly over
// the row's lanes) and the v* write of slide 11.
#include <atomic>

#include "palimpsa_internal.cuh"

namespace palimpsa {
namespace {

constexpr int kRowsPerWarp = 8;
constexpr int kWarpsPerBlock = 1;

template <bool BF16>
__device__ __forceinline__ float4 load4(const void* base, size_t idx) {
  if constexpr (BF16) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + idx);
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
  } else {
    return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
  }
}

template <bool BF16>
__device__ __forceinline__ float load1(const void* base, size_t idx) {
  if constexpr (BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
  else return static_cast<const float*>(base)[idx];
}

// 16-byte store that L2 keeps in preference to streamed lines (evict_last).
__device__ __forceinline__ void st_evict_last(float* p, float4 v, unsigned long long pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w), "l"(pol)
               : "memory");
}

template <int DK, bool BF16, bool PRO>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, PRO ? 2 : 1)
palimpsa_step_kernel(StepArgs a, bool reverse, long keep_from) {
  constexpr int LPR = DK / 4;       // lanes per row
  constexpr int RPI = 32 / LPR;     // rows per warp instruction
  constexpr int NIT = kRowsPerWarp / RPI;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long total_rows = (long)a.B * a.H * a.d_v;
  // CTAs start roughly in index order (pos). The walk visits the row blocks
  // forwards or backwards (rank -> block), and the CTAs from keep_from on, the
  // last K of the walk, keep their rows in L2. The previous launch kept the K
  // blocks that this walk reaches first; over its first 2K positions they
  // alternate with the K blocks after them, so that DRAM has reads to serve
  // while those hit in L2.
  const long n_blk = (long)gridDim.x, pos = (long)blockIdx.x, K = n_blk - keep_from;
  long rank = pos;
  if (K > 0 && 2 * K <= keep_from && pos < 2 * K) rank = (pos & 1) ? K + (pos >> 1) : (pos >> 1);
  const long blk = reverse ? n_blk - 1 - rank : rank;
  const bool keep = pos >= keep_from;
  unsigned long long keep_pol = 0;
  if (keep) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep_pol));
  const long row_base = (blk * kWarpsPerBlock + warp) * kRowsPerWarp;
  if (row_base >= total_rows) return;
  // Launched with programmatic dependent launch, this CTA may start while the
  // kernel before it in the stream is still running; everything it reads may
  // come from that kernel (the state from the previous step, the token's
  // inputs from the layer's projections), so it waits for it before any read.
  // Without the launch attribute the wait returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long bh = row_base / a.d_v;
  const int h = (int)(bh % a.H);
  const int sub = lane / LPR;
  const int col = 4 * (lane % LPR);

  // The rows' beta and v: lane r (r < 8) takes row r's, forms the row's gate
  // values once for the warp (through the prologue when it is on), and the
  // row loop reads them back by shuffle.
  // (With the prologue each lane still loads v for every row: on GB300 that
  // measured faster than shuffling beta_i v_i, which would wait on the gate.)
  const int i_base = (int)(row_base - bh * a.d_v);
  const size_t row_in = (size_t)bh * a.d_v + i_base + (lane % kRowsPerWarp);
  float b_row = load1<BF16>(a.beta, row_in);
  float v_row = 0.f, v_in[NIT];
  if constexpr (PRO) {
#pragma unroll
    for (int it = 0; it < NIT; ++it) v_in[it] = load1<BF16>(a.v, (size_t)bh * a.d_v + i_base + it * RPI + sub);
  } else {
    v_row = load1<BF16>(a.v, row_in);
  }

  float4 q4 = load4<BF16>(a.q, (size_t)bh * DK + col);
  float4 k4 = load4<BF16>(a.k, (size_t)bh * DK + col);
  float d = a.d_t[bh];
  // Issue the state loads, 2 * NIT independent 16-byte loads per lane, and let
  // the next step's CTAs be scheduled.
  float4 mu4[NIT], I4[NIT];
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const size_t off = (size_t)(row_base + it * RPI + sub) * DK + col;
    mu4[it] = __ldcs(reinterpret_cast<const float4*>(a.mu + off));
    I4[it] = __ldcs(reinterpret_cast<const float4*>(a.I + off));
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  float bsc = 1.f;
  if constexpr (PRO) {
    d = softplus_f(d);
    if (a.pro.b_scale) bsc = a.pro.b_scale[h];
    b_row = bsc * sigmoid_f(b_row);
    if (a.pro.qk_norm) {  // the LPR lanes of a row hold the whole q and k of the head
      float sq = q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w;
      float sk = k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w;
#pragma unroll
      for (int m = 1; m < LPR; m <<= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, m);
        sk += __shfl_xor_sync(0xffffffffu, sk, m);
      }
      const float iq = rsqrtf(fmaxf(sq, kNormFloorSq)), ik = rsqrtf(fmaxf(sk, kNormFloorSq));
      q4 = make_float4(q4.x * iq, q4.y * iq, q4.z * iq, q4.w * iq);
      k4 = make_float4(k4.x * ik, k4.y * ik, k4.z * ik, k4.w * ik);
    }
  }
  const float bv_row = b_row * v_row;  // beta_i v_i of the lane's row (without the prologue)
  const float A_h = a.A[h], Ip = a.I_prior[h];
  bool bad = !(pos_finite(A_h) && pos_finite(Ip) && nonneg_finite(d));
  const float x = -A_h * d;
  const float al = expf(x);
  const float om = -expm1f(x) * Ip;  // (1 - alpha) I_prior
  const float kj[4] = {k4.x, k4.y, k4.z, k4.w};
  const float qj[4] = {q4.x, q4.y, q4.z, q4.w};
  float kk[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) kk[e] = kj[e] * kj[e];

#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const long row = row_base + it * RPI + sub;
    const float b = __shfl_sync(0xffffffffu, b_row, it * RPI + sub);
    float bv;
    if constexpr (PRO) bv = a.pro.v_star ? v_in[it] : b * v_in[it];
    else bv = __shfl_sync(0xffffffffu, bv_row, it * RPI + sub);
    bad |= !nonneg_finite(b);
    float Io[4] = {I4[it].x, I4[it].y, I4[it].z, I4[it].w};
    float mo[4] = {mu4[it].x, mu4[it].y, mu4[it].z, mu4[it].w};
    float In[4], mn[4];
    float yp = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      bad |= !pos_finite(Io[e]);
      In[e] = fmaf(al, Io[e], fmaf(b, kk[e], om));
      const float num = fmaf(al * Io[e], mo[e], bv * kj[e]);
      if constexpr (PRO) mn[e] = __fdividef(num, In[e]);
      else mn[e] = num / In[e];
      yp = fmaf(mn[e], qj[e], yp);
    }
#pragma unroll
    for (int m = 1; m < LPR; m <<= 1) yp += __shfl_xor_sync(0xffffffffu, yp, m);
    const size_t off = (size_t)row * DK + col;
    const float4 mu_new = make_float4(mn[0], mn[1], mn[2], mn[3]), I_new = make_float4(In[0], In[1], In[2], In[3]);
    if (keep) {  // stays in L2 for the next step
      st_evict_last(a.mu + off, mu_new, keep_pol);
      st_evict_last(a.I + off, I_new, keep_pol);
    } else {
      __stcs(reinterpret_cast<float4*>(a.mu + off), mu_new);
      __stcs(reinterpret_cast<float4*>(a.I + off), I_new);
    }
    if ((lane % LPR) == 0) a.y[row] = yp;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) latch_status(a.status, kStatusDomain);
}

}  // namespace

// Direction of the next step's walk: flips at every launch, process-wide. With
// one decode state this alternates its steps; any interleaving is still
// correct, only the L2 reuse is lost.
std::atomic<unsigned> g_step_parity{0};

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
  const long rows = (long)a.B * a.H * a.d_v;
  const long rows_per_block = (long)kWarpsPerBlock * kRowsPerWarp;
  const unsigned blocks = (unsigned)((rows + rows_per_block - 1) / rows_per_block);
  const dim3 g(blocks), b(kWarpsPerBlock * 32);
  bool reverse = false;
  long keep_from = (long)blocks;  // no CTA keeps its rows in L2
  if (a.l2_keep_bytes > 0) {
    reverse = (g_step_parity.fetch_add(1, std::memory_order_relaxed) & 1u) != 0;
    const long long block_bytes = rows_per_block * (long long)a.d_k * 2 * sizeof(float);
    const long long keep_blocks = a.l2_keep_bytes / block_bytes;
    keep_from = keep_blocks >= (long long)blocks ? 0 : (long)(blocks - keep_blocks);
  }
  // programmatic dependent launch: this step's CTAs may be scheduled while the
  // previous step drains; they wait for it before reading the state
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = g;
  cfg.blockDim = b;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (a.pro.on) {
    if (a.d_k == 128) e = a.bf16 ? cudaLaunchKernelEx(&cfg, palimpsa_step_kernel<128, true, true>, a, reverse, keep_from)
                                 : cudaLaunchKernelEx(&cfg, palimpsa_step_kernel<128, false, true>, a, reverse, keep_from);
    else e = a.bf16 ? cudaLaunchKernelEx(&cfg, palimpsa_step_kernel<64, true, true>, a, reverse, keep_from)
                    : cudaLaunchKernelEx(&cfg, palimpsa_step_kernel<64, false, true>, a, reverse, keep_from);
  } else if (a.d_k == 128) {
    e = a.bf16 ? cudaLaunchKernelEx(&cfg, palimpsa_step_kernel<128, true, false>, a, reverse, keep_from)
               : cudaLaunchKernelEx(&cfg, palimpsa_step_kernel<128, false, false>, a, reverse, keep_from);
  } else {
    e = a.bf16 ? cudaLaunchKernelEx(&cfg, palimpsa_step_kernel<64, true, false>, a, reverse, keep_from)
               : cudaLaunchKernelEx(&cfg, palimpsa_step_kernel<64, false, false>, a, reverse, keep_from);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace palimpsa
