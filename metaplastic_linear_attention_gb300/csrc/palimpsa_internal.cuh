// Internal declarations shared by the kernels and the C ABI layer: launch
// argument structs, the device status bits, and thin inline-PTX wrappers for
// the sm_103a features the kernels use (mbarrier, bulk async copies, packed
// fp32x2 arithmetic, the hardware reciprocal).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace palimpsa {

// Bits latched into the per-device status word.
enum : unsigned int {
  kStatusTimeout = 1u << 0,
  kStatusDomain = 1u << 1,
};

// The fused layer prologue (palimpsa_forward_fused / palimpsa_step_fused):
// raw projections are turned into the recurrence's inputs as they are staged.
struct Prologue {
  bool on = false;                 // d_t = softplus(raw), beta = b_scale[h] * sigmoid(raw)
  bool qk_norm = false;            // q, k divided by their L2 norm per token
  bool v_star = false;             // v holds v* = beta (.) v: the content write takes it as is
  const float* b_scale = nullptr;  // [H]; NULL means 1
};

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* beta;
  const float* d_t;
  const float* A;
  const float* I_prior;
  const float* mu0;  // may be null
  const float* I0;   // may be null
  float* y;
  float* mu_T;
  float* I_T;
  int B, H, T, d_k, d_v, chunk;
  bool bf16;
  unsigned int* status;
  unsigned long long wait_timeout_ns;
  int withhold_first_copy;
  int force_segments;  // 0: the library chooses the time split
  Prologue pro{};
  float* ckpt = nullptr;  // training checkpoints out (dense layout only), or null
  // Packed variable-length batch (palimpsa_forward_varlen): B counts sequences,
  // T is the longest sequence, and sequence n is tokens [cu[n], cu[n+1]) of each
  // head's total_T tokens. NULL for the dense [B, H, T] layout.
  const int* cu_seqlens = nullptr;
  long long total_T = 0;
};

struct StepArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* beta;
  const float* d_t;
  const float* A;
  const float* I_prior;
  float* mu;
  float* I;
  float* y;
  int B, H, d_k, d_v;
  bool bf16;
  unsigned int* status;
  Prologue pro{};
  // Bytes of the state that the step stores last and leaves in L2 for the
  // next step, which walks the state in the opposite order (0: every step
  // streams the whole state in the same order).
  long long l2_keep_bytes = 0;
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* beta;
  const float* d_t;
  const float* A;
  const float* I_prior;
  const float* mu0;    // may be null
  const float* I0;     // may be null
  const float* dy;
  const float* dmu_T;  // may be null
  const float* dI_T;   // may be null
  float* dq;           // zeroed by the caller of the launcher (accumulated)
  float* dk;           // zeroed (accumulated)
  float* dv;
  float* dbeta;
  float* dd_t;         // zeroed (accumulated)
  float* dA;           // zeroed (accumulated)
  float* dI_prior;     // zeroed (accumulated)
  float* dmu0;         // may be null
  float* dI0;          // may be null
  int B, H, T, d_k, d_v;
  bool bf16;
  // Training checkpoints written by the forward (layout of kCheckpointTokens
  // below), or null: the backward then recomputes them with a forward sweep.
  const float* ckpt_in = nullptr;
  // Packed variable-length batch, as in FwdArgs (B counts sequences, T is the
  // longest); null for the dense layout.
  const int* cu_seqlens = nullptr;
  long long total_T = 0;
  unsigned int* status = nullptr;  // device status word (bad packed offsets)
};

// Training checkpoints: the state (M, I) of every head before tokens 0, 32,
// 64, ... laid out [head][checkpoint][value row i][M_i0 .. M_i(d_k-1), I_i0 ..
// I_i(d_k-1)], fp32. Written by the forward when asked, read by the backward.
constexpr int kCheckpointTokens = 32;
inline size_t checkpoint_floats(long long heads, long long T, int d_k, int d_v) {
  const long long n = (T + kCheckpointTokens - 1) / kCheckpointTokens;
  return (size_t)heads * n * d_v * 2 * d_k;
}
// Packed batches keep their checkpoints without padding to the longest
// sequence: per head, total_T / 32 + N slots, and head h of the sequence that
// starts at token s0 (the n-th) owns the slots from
//   h (total_T / 32 + N) + s0 / 32 + n.
// A sequence of L tokens needs ceil(L / 32) slots, and the next one starts
// floor((s0 + L) / 32) + 1 >= floor(s0 / 32) + ceil(L / 32) slots on, so
// sequences never share a slot.
__host__ __device__ inline long long packed_checkpoint_slots(long long total_T, long long N) {
  return total_T / kCheckpointTokens + N;
}
__host__ __device__ inline long long packed_checkpoint_slot0(int h, long long n, long long s0, long long total_T,
                                                             long long N) {
  return (long long)h * packed_checkpoint_slots(total_T, N) + s0 / kCheckpointTokens + n;
}

// Source of temporary device memory for a launch that needs scratch (the time
// split of the forward). acquire/release are stream-ordered on `s`.
struct ScratchProvider {
  virtual cudaError_t acquire(size_t bytes, cudaStream_t s, float** p) = 0;
  virtual cudaError_t release(float* p, cudaStream_t s) = 0;
  virtual ~ScratchProvider() = default;
};

// Launchers (return the launch error, cudaSuccess on success). Arguments are
// validated by the caller.
cudaError_t launch_forward_chunked(const FwdArgs& a, cudaStream_t s, ScratchProvider* sp);
// Scratch of a time split, in floats: the carried states [heads][nseg - 1][2][d_v d_k]
// (summaries until the carry turns them into segment-start states), the gammas
// [heads][nseg - 1], then, 16-byte aligned, each head's initial state (M_0, I_0)
// [heads][2][d_v d_k], copied there by the carry so that the first segment never
// reads mu0 / I0, which the caller may alias with mu_T / I_T.
struct SplitScratch {
  size_t gammas, init, total;  // offsets and size in floats
  __host__ __device__ SplitScratch(long long heads, int nseg, long long dvk) {
    gammas = (size_t)heads * (nseg - 1) * 2 * dvk;
    init = (gammas + (size_t)heads * (nseg - 1) + 3) / 4 * 4;
    total = init + (size_t)heads * 2 * dvk;
  }
};

// The time-split plan launch_forward_chunked would use (queries the device; launches nothing).
cudaError_t plan_forward(const FwdArgs& a, int* nseg, int* seg_len);
// Passes A and B of a time split with that plan into scratch laid out as
// SplitScratch: the (M, Ibar) state at the start of segments 1 .. nseg - 1 of
// every head, and each head's initial (M_0, I_0).
cudaError_t launch_split_prefix(const FwdArgs& a, int nseg, int seg_len, float* scratch, cudaStream_t s);
cudaError_t launch_step(const StepArgs& a, cudaStream_t s);
// Summary of the whole token range of each head from a zero state (pass A over
// the planned segments, then folded): summary [B,H,2,d_v,d_k] = (dM, dIbar),
// gamma [B,H] = prod alpha.
cudaError_t launch_segment_summary(const FwdArgs& a, float* summary, float* gamma, cudaStream_t s,
                                   ScratchProvider* sp);

// Pass A on the tensor cores (fwd_summary_tc.cu): bf16 inputs, d_k = 128,
// d_v a multiple of 32 up to 128. Summaries of segments 0 ..
// nslot - 1 of every head, laid out as the FFMA pass A writes them.
bool summary_tc_eligible(const FwdArgs& a);
cudaError_t launch_summary_tc(const FwdArgs& a, int nslot, int seg_len, float* seg_state, float* seg_gamma,
                              cudaStream_t s);

// Affine fold of R segment summaries, in order (fold.cu):
//   (M, Ibar) <- Gamma_s (M, Ibar) + (dM_s, dIbar_s),   s = 0 .. R-1.
// Summary element (s, bh, part, e) is at sum[s*sum_ss + bh*sum_sh + part*DVK + e],
// gamma (s, bh) at gam[s*gam_ss + bh*gam_sh]. With to_state the fold starts
// from (I0 mu0, I0 - I_prior) (defaults mu0 = 0, I0 = I_prior) and writes the
// state as (mu, I) to out_a, out_b; otherwise it starts from zero and writes
// (dM, dIbar) to out_a, out_b and prod Gamma to out_gamma [heads]. Output
// element (bh, e) is at out_*[bh*out_sh + e]; mu0 and I0 are [heads, DVK].
struct FoldArgs {
  const float* sum;
  const float* gam;
  long long sum_ss, sum_sh, gam_ss, gam_sh;
  int R;
  long long heads;
  int H, DVK;
  bool to_state;
  const float* I_prior;
  const float* mu0;
  const float* I0;
  float* out_a;
  float* out_b;
  float* out_gamma;
  long long out_sh;
};
cudaError_t launch_fold(const FoldArgs& f, cudaStream_t s);
// The "without Meta" comparator (importance frozen at I_prior); uses a.mu0,
// a.y, a.mu_T and ignores a.I0, a.I_T; time split as the forward plans it.
cudaError_t launch_forward_without_meta(const FwdArgs& a, cudaStream_t s, ScratchProvider* sp);
// Backward: scratch of backward_scratch_bytes(a) bytes holds the checkpoints.
size_t backward_scratch_bytes(const BwdArgs& a);
cudaError_t launch_backward(const BwdArgs& a, float* scratch, cudaStream_t s);

// The domain preconditions of a call's inputs, checked by a separate pass for
// the entry points whose kernels do not test them as they read them.
struct DomainArgs {
  const void* beta;       // [n_beta] in the call's input dtype
  size_t n_beta;
  bool bf16;
  const float* d_t;       // [n_dt]
  size_t n_dt;
  const float* I0;        // [n_state], or null
  size_t n_state;
  const float* A;         // [H], or null
  const float* I_prior;   // [H]
  int H;
  unsigned int* status;   // latched: kStatusDomain
};
cudaError_t launch_domain_check(const DomainArgs& a, cudaStream_t s);

// ------------------------------------------------------------------ device helpers
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Waits until phase `parity` of `bar` completes or `timeout_ns` elapses.
// Returns false on timeout. Every wait in this library goes through here.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 >= timeout_ns) return mbar_try_wait(bar, parity);
  }
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xffff0000u); }

__device__ __forceinline__ void latch_status(unsigned int* status, unsigned int bits) {
  atomicOr(status, bits);
}

// fp32 "is a usable positive number" / "is a usable non-negative number".
__device__ __forceinline__ bool pos_finite(float x) { return x > 0.f && x <= 3.0e38f; }
__device__ __forceinline__ bool nonneg_finite(float x) { return x >= 0.f && x <= 3.0e38f; }

// Prologue activations. softplus(x) = log(1 + e^x) as max(x, 0) + log1p(e^-|x|)
// (no overflow for large x, no lost tail for very negative x); sigmoid(x) =
// 1 / (1 + e^-x), which tends to 0 when e^-x overflows.
__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// Squared-norm floor of the q/k L2 norm: x / max(||x||, 1e-12).
constexpr float kNormFloorSq = 1e-24f;

#endif  // __CUDACC__

}  // namespace palimpsa
