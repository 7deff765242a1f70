// C ABI layer: argument validation, the per-device status word, debug
// controls, and dispatch to the kernels' launchers. Declared in palimpsa.h.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "palimpsa.h"
#include "palimpsa_internal.cuh"

namespace palimpsa {

// One status word per device, latched by kernels (kStatus* bits).
__device__ unsigned int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};
std::atomic<unsigned long long> g_wait_timeout_ns{2000000000ull};
std::atomic<int> g_withhold_first_copy{0};
std::atomic<int> g_forward_segments{0};
// Bytes of state each decode step leaves in L2 for the next one.
std::atomic<long long> g_step_l2_keep_bytes{96ll << 20};

// Bytes of freed scratch each device's pool keeps mapped between calls.
std::atomic<unsigned long long> g_scratch_keep_bytes{512ull << 20};
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

// The library's own stream-ordered memory pool on the current device, created
// on first use. Memory freed by one call stays mapped for the next, up to the
// pool's release threshold (g_scratch_keep_bytes; 512 MiB by default): at the
// next synchronisation the pool gives back what it holds above that. The
// forward's time-split scratch (tens to a few hundred MiB) therefore stays
// mapped from call to call (re-mapping fresh pages cost the time-split passes
// a few percent), while a large backward's scratch goes back to the driver
// once the caller synchronises.
cudaError_t scratch_pool(cudaMemPool_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  if (!g_pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return e;
    unsigned long long keep = g_scratch_keep_bytes.load();
    if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return e;
    }
    g_pools[dev] = pool;
  }
  *out = g_pools[dev];
  return cudaSuccess;
}

// The current device's pool if one was created, else nullptr.
palimpsa_status existing_pool(cudaMemPool_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PALIMPSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  *out = g_pools[dev];
  return PALIMPSA_OK;
}

// Scratch from that pool, allocated and freed in stream order on the launch
// stream: no synchronisation, and reuse across calls.
struct StreamOrderedScratch final : ScratchProvider {
  cudaError_t acquire(size_t bytes, cudaStream_t s, float** p) override {
    cudaMemPool_t pool = nullptr;
    cudaError_t e = scratch_pool(&pool);
    if (e != cudaSuccess) return e;
    void* v = nullptr;
    e = cudaMallocFromPoolAsync(&v, bytes, pool, s);
    *p = static_cast<float*>(v);
    return e;
  }
  cudaError_t release(float* p, cudaStream_t s) override { return cudaFreeAsync(p, s); }
};

// Device address of the current device's status word (looked up once per
// device with that device current).
palimpsa_status status_word(unsigned int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PALIMPSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return PALIMPSA_ERR_CUDA;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_status_ptr[dev];
  return PALIMPSA_OK;
}

// The caller's chunk: 0 (library default) or one of 16, 32, 64, 128 tokens. The
// result does not depend on it (slide 9: the chunk only sets how many tokens are
// staged on chip at a time); the kernels stage at most 32 tokens per chunk, so
// longer chunks are staged as 32-token chunks.
bool chunk_ok(int c) { return c == 0 || c == 16 || c == 32 || c == 64 || c == 128; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool supported_dims(int d_k, int d_v) {
  return (d_k == 64 || d_k == 128) && d_v >= 8 && d_v <= 256 && d_v % 8 == 0;
}

// Element counts must fit comfortably in 63 bits and per-head token counts in int.
bool sizes_ok(long long B, long long H, long long T, int d_k, int d_v) {
  if (B < 1 || H < 1 || T < 0) return false;
  const long long lim = 1LL << 40;
  if (B * H > lim / 256) return false;
  if (B * H * (T > 0 ? T : 1) > lim) return false;
  (void)d_k;
  (void)d_v;
  return true;
}

// Validation and launch shared by palimpsa_forward_chunked and
// palimpsa_forward_fused (pro.on only for the latter).
palimpsa_status forward_impl(const void* q, const void* k, const void* v, const void* beta, const float* d_t,
                             const float* A, const float* I_prior, const float* mu0, const float* I0, float* y,
                             float* mu_T, float* I_T, int B, int H, int T, int d_k, int d_v, int chunk,
                             palimpsa_dtype in_dtype, void* cuda_stream, const Prologue& pro,
                             float* ckpt = nullptr) {
  if (!A || !I_prior || !mu_T || !I_T) return PALIMPSA_ERR_NULL;
  // With T == 0 the per-token arrays are empty and may be NULL.
  if (T != 0 && (!q || !k || !v || !beta || !d_t || !y)) return PALIMPSA_ERR_NULL;
  if (in_dtype != PALIMPSA_F32 && in_dtype != PALIMPSA_BF16) return PALIMPSA_ERR_DTYPE;
  if (!sizes_ok(B, H, T, d_k, d_v)) return PALIMPSA_ERR_SHAPE;
  if (!supported_dims(d_k, d_v)) return PALIMPSA_ERR_UNSUPPORTED;
  if (!chunk_ok(chunk)) return PALIMPSA_ERR_UNSUPPORTED;
  const void* a16[] = {q, k, v, beta, y, mu_T, I_T, mu0, I0, ckpt};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return PALIMPSA_ERR_ALIGN;
  const void* a4[] = {d_t, A, I_prior};
  for (const void* p : a4)
    if (p && !aligned(p, 4)) return PALIMPSA_ERR_ALIGN;
  unsigned int* st = nullptr;
  if (palimpsa_status s = status_word(&st)) return s;
  FwdArgs a{q, k, v, beta, d_t, A, I_prior, mu0, I0, y, mu_T, I_T, B, H, T, d_k, d_v,
            chunk == 0 ? 32 : chunk, in_dtype == PALIMPSA_BF16, st,
            g_wait_timeout_ns.load(), g_withhold_first_copy.load(), g_forward_segments.load(), pro};
  a.ckpt = ckpt;
  StreamOrderedScratch scratch;
  if (launch_forward_chunked(a, static_cast<cudaStream_t>(cuda_stream), &scratch) != cudaSuccess)
    return PALIMPSA_ERR_CUDA;
  return PALIMPSA_OK;
}

// Validation and launch shared by palimpsa_step and palimpsa_step_fused.
palimpsa_status step_impl(const void* q, const void* k, const void* v, const void* beta, const float* d_t,
                          const float* A, const float* I_prior, float* mu, float* I, float* y, int B, int H,
                          int d_k, int d_v, palimpsa_dtype in_dtype, void* cuda_stream, const Prologue& pro) {
  if (!q || !k || !v || !beta || !d_t || !A || !I_prior || !mu || !I || !y) return PALIMPSA_ERR_NULL;
  if (in_dtype != PALIMPSA_F32 && in_dtype != PALIMPSA_BF16) return PALIMPSA_ERR_DTYPE;
  if (!sizes_ok(B, H, 1, d_k, d_v)) return PALIMPSA_ERR_SHAPE;
  if (!supported_dims(d_k, d_v)) return PALIMPSA_ERR_UNSUPPORTED;
  const void* a16[] = {q, k, v, beta, mu, I, y};
  for (const void* p : a16)
    if (!aligned(p, 16)) return PALIMPSA_ERR_ALIGN;
  const void* a4[] = {d_t, A, I_prior, pro.b_scale};
  for (const void* p : a4)
    if (p && !aligned(p, 4)) return PALIMPSA_ERR_ALIGN;
  unsigned int* st = nullptr;
  if (palimpsa_status s = status_word(&st)) return s;
  StepArgs a{q, k, v, beta, d_t, A, I_prior, mu, I, y, B, H, d_k, d_v, in_dtype == PALIMPSA_BF16, st, pro};
  a.l2_keep_bytes = g_step_l2_keep_bytes.load();
  if (launch_step(a, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  return PALIMPSA_OK;
}

// S tokens in order (palimpsa_step_sequence, palimpsa_step_sequence_fused):
// the arguments are validated once, on the first token (every token's slice
// has the same sizes and alignment, since a token of q, k is 2 or 4 * d_k bytes
// and of v, beta, y d_v * 2 or 4 bytes, both multiples of 16; d_t only needs
// 4), then one step launch per token is enqueued.
palimpsa_status step_sequence_impl(const void* q, const void* k, const void* v, const void* beta, const float* d_t,
                                   const float* A, const float* I_prior, float* mu, float* I, float* y, int S,
                                   int B, int H, int d_k, int d_v, palimpsa_dtype in_dtype, void* cuda_stream,
                                   const Prologue& pro) {
  if (S < 0) return PALIMPSA_ERR_SHAPE;
  if (S == 0) return PALIMPSA_OK;
  palimpsa_status st = step_impl(q, k, v, beta, d_t, A, I_prior, mu, I, y, B, H, d_k, d_v, in_dtype, cuda_stream,
                                 pro);
  if (st != PALIMPSA_OK) return st;
  if ((long long)S * B * H > (1LL << 40)) return PALIMPSA_ERR_SHAPE;
  unsigned int* sw = nullptr;
  if (palimpsa_status s2 = status_word(&sw)) return s2;
  const size_t es = in_dtype == PALIMPSA_BF16 ? 2 : 4;
  const size_t bh = (size_t)B * H;
  const char* cq = static_cast<const char*>(q);
  const char* ck = static_cast<const char*>(k);
  const char* cv = static_cast<const char*>(v);
  const char* cb = static_cast<const char*>(beta);
  const long long keep = g_step_l2_keep_bytes.load();
  for (int s = 1; s < S; ++s) {
    StepArgs a{cq + s * bh * d_k * es, ck + s * bh * d_k * es, cv + s * bh * d_v * es, cb + s * bh * d_v * es,
               d_t + s * bh, A, I_prior, mu, I, y + s * bh * d_v, B, H, d_k, d_v, in_dtype == PALIMPSA_BF16, sw,
               pro};
    a.l2_keep_bytes = keep;
    if (launch_step(a, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  }
  return PALIMPSA_OK;
}

constexpr unsigned int kKnownFuseFlags = PALIMPSA_FUSE_QK_NORM | PALIMPSA_FUSE_V_STAR;

Prologue fused_prologue(const float* b_scale, unsigned int flags) {
  Prologue p;
  p.on = true;
  p.qk_norm = (flags & PALIMPSA_FUSE_QK_NORM) != 0;
  p.v_star = (flags & PALIMPSA_FUSE_V_STAR) != 0;
  p.b_scale = b_scale;
  return p;
}

}  // namespace
}  // namespace palimpsa

using namespace palimpsa;

extern "C" {

palimpsa_status palimpsa_forward_chunked(const void* q, const void* k, const void* v, const void* beta,
                                         const float* d_t, const float* A, const float* I_prior,
                                         const float* mu0, const float* I0, float* y, float* mu_T,
                                         float* I_T, int B, int H, int T, int d_k, int d_v, int chunk,
                                         palimpsa_dtype in_dtype, void* cuda_stream) {
  return forward_impl(q, k, v, beta, d_t, A, I_prior, mu0, I0, y, mu_T, I_T, B, H, T, d_k, d_v, chunk, in_dtype,
                      cuda_stream, Prologue{});
}

palimpsa_status palimpsa_forward_plan(int B, int H, int T, int d_k, int d_v, int chunk, palimpsa_dtype in_dtype,
                                      int* segments, int* segment_len, int* launches, size_t* scratch_bytes) {
  if (!segments || !segment_len || !launches || !scratch_bytes) return PALIMPSA_ERR_NULL;
  if (in_dtype != PALIMPSA_F32 && in_dtype != PALIMPSA_BF16) return PALIMPSA_ERR_DTYPE;
  if (!sizes_ok(B, H, T, d_k, d_v)) return PALIMPSA_ERR_SHAPE;
  if (!supported_dims(d_k, d_v)) return PALIMPSA_ERR_UNSUPPORTED;
  if (!chunk_ok(chunk)) return PALIMPSA_ERR_UNSUPPORTED;
  FwdArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
            nullptr, B, H, T, d_k, d_v, chunk == 0 ? 32 : chunk, in_dtype == PALIMPSA_BF16, nullptr, 0, 0,
            g_forward_segments.load(), Prologue{}};
  int nseg = 1, seg_len = 0;
  if (plan_forward(a, &nseg, &seg_len) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  *segments = nseg;
  *segment_len = seg_len;
  *launches = nseg > 1 ? 3 : 1;
  *scratch_bytes = nseg > 1 ? SplitScratch((long long)B * H, nseg, (long long)d_v * d_k).total * sizeof(float) : 0;
  return PALIMPSA_OK;
}

// Validation and launch shared by palimpsa_forward_varlen and _varlen_fused.
static palimpsa_status varlen_impl(const void* q, const void* k, const void* v, const void* beta, const float* d_t,
                                   const float* A, const float* I_prior, const float* mu0, const float* I0, float* y,
                                   float* mu_T, float* I_T, const int* cu_seqlens, int N, int H, int total_T,
                                   int max_seqlen, int d_k, int d_v, int chunk, palimpsa_dtype in_dtype,
                                   void* cuda_stream, const Prologue& pro, float* ckpt = nullptr) {
  if (!A || !I_prior || !mu_T || !I_T || !cu_seqlens) return PALIMPSA_ERR_NULL;
  if (total_T != 0 && (!q || !k || !v || !beta || !d_t || !y)) return PALIMPSA_ERR_NULL;
  if (in_dtype != PALIMPSA_F32 && in_dtype != PALIMPSA_BF16) return PALIMPSA_ERR_DTYPE;
  if (total_T < 0 || max_seqlen < 0 || max_seqlen > total_T) return PALIMPSA_ERR_SHAPE;
  if (!sizes_ok(N, H, max_seqlen, d_k, d_v) || !sizes_ok(1, H, total_T, d_k, d_v)) return PALIMPSA_ERR_SHAPE;
  if (!supported_dims(d_k, d_v)) return PALIMPSA_ERR_UNSUPPORTED;
  if (!chunk_ok(chunk)) return PALIMPSA_ERR_UNSUPPORTED;
  const void* a16[] = {q, k, v, beta, y, mu_T, I_T, mu0, I0, ckpt};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return PALIMPSA_ERR_ALIGN;
  const void* a4[] = {d_t, A, I_prior, cu_seqlens, pro.b_scale};
  for (const void* p : a4)
    if (p && !aligned(p, 4)) return PALIMPSA_ERR_ALIGN;
  unsigned int* st = nullptr;
  if (palimpsa_status s = status_word(&st)) return s;
  FwdArgs a{q, k, v, beta, d_t, A, I_prior, mu0, I0, y, mu_T, I_T, N, H, max_seqlen, d_k, d_v,
            chunk == 0 ? 32 : chunk, in_dtype == PALIMPSA_BF16, st,
            g_wait_timeout_ns.load(), g_withhold_first_copy.load(), g_forward_segments.load(), pro};
  a.cu_seqlens = cu_seqlens;
  a.total_T = total_T;
  a.ckpt = ckpt;
  StreamOrderedScratch scratch;
  if (launch_forward_chunked(a, static_cast<cudaStream_t>(cuda_stream), &scratch) != cudaSuccess)
    return PALIMPSA_ERR_CUDA;
  return PALIMPSA_OK;
}

palimpsa_status palimpsa_forward_varlen(const void* q, const void* k, const void* v, const void* beta,
                                        const float* d_t, const float* A, const float* I_prior, const float* mu0,
                                        const float* I0, float* y, float* mu_T, float* I_T, const int* cu_seqlens,
                                        int N, int H, int total_T, int max_seqlen, int d_k, int d_v, int chunk,
                                        palimpsa_dtype in_dtype, void* cuda_stream) {
  return varlen_impl(q, k, v, beta, d_t, A, I_prior, mu0, I0, y, mu_T, I_T, cu_seqlens, N, H, total_T, max_seqlen,
                     d_k, d_v, chunk, in_dtype, cuda_stream, Prologue{});
}

palimpsa_status palimpsa_forward_varlen_fused(const void* q, const void* k, const void* v, const void* beta_raw,
                                              const float* d_raw, const float* A, const float* I_prior,
                                              const float* b_scale, const float* mu0, const float* I0, float* y,
                                              float* mu_T, float* I_T, const int* cu_seqlens, int N, int H,
                                              int total_T, int max_seqlen, int d_k, int d_v, int chunk,
                                              unsigned int flags, palimpsa_dtype in_dtype, void* cuda_stream) {
  if (flags & ~kKnownFuseFlags) return PALIMPSA_ERR_UNSUPPORTED;
  return varlen_impl(q, k, v, beta_raw, d_raw, A, I_prior, mu0, I0, y, mu_T, I_T, cu_seqlens, N, H, total_T,
                     max_seqlen, d_k, d_v, chunk, in_dtype, cuda_stream, fused_prologue(b_scale, flags));
}

palimpsa_status palimpsa_forward_varlen_checkpointed(const void* q, const void* k, const void* v, const void* beta,
                                                     const float* d_t, const float* A, const float* I_prior,
                                                     const float* mu0, const float* I0, float* y, float* mu_T,
                                                     float* I_T, float* ckpt, const int* cu_seqlens, int N, int H,
                                                     int total_T, int max_seqlen, int d_k, int d_v, int chunk,
                                                     palimpsa_dtype in_dtype, void* cuda_stream) {
  if (!ckpt && max_seqlen != 0) return PALIMPSA_ERR_NULL;
  return varlen_impl(q, k, v, beta, d_t, A, I_prior, mu0, I0, y, mu_T, I_T, cu_seqlens, N, H, total_T, max_seqlen,
                     d_k, d_v, chunk, in_dtype, cuda_stream, Prologue{}, ckpt);
}

palimpsa_status palimpsa_segment_summary(const void* q, const void* k, const void* v, const void* beta,
                                         const float* d_t, const float* A, const float* I_prior, float* summary,
                                         float* gamma, int B, int H, int T, int d_k, int d_v, int chunk,
                                         palimpsa_dtype in_dtype, void* cuda_stream) {
  if (!A || !I_prior || !summary || !gamma) return PALIMPSA_ERR_NULL;
  if (T != 0 && (!q || !k || !v || !beta || !d_t)) return PALIMPSA_ERR_NULL;
  if (in_dtype != PALIMPSA_F32 && in_dtype != PALIMPSA_BF16) return PALIMPSA_ERR_DTYPE;
  if (!sizes_ok(B, H, T, d_k, d_v)) return PALIMPSA_ERR_SHAPE;
  if (!supported_dims(d_k, d_v)) return PALIMPSA_ERR_UNSUPPORTED;
  if (!chunk_ok(chunk)) return PALIMPSA_ERR_UNSUPPORTED;
  const void* a16[] = {q, k, v, beta, summary};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return PALIMPSA_ERR_ALIGN;
  const void* a4[] = {d_t, A, I_prior, gamma};
  for (const void* p : a4)
    if (p && !aligned(p, 4)) return PALIMPSA_ERR_ALIGN;
  unsigned int* st = nullptr;
  if (palimpsa_status s = status_word(&st)) return s;
  FwdArgs a{q, k, v, beta, d_t, A, I_prior, nullptr, nullptr, nullptr, nullptr, nullptr, B, H, T, d_k, d_v,
            chunk == 0 ? 32 : chunk, in_dtype == PALIMPSA_BF16, st,
            g_wait_timeout_ns.load(), g_withhold_first_copy.load(), g_forward_segments.load(), Prologue{}};
  // pass A does not test the preconditions as it reads the inputs (the forward's pass C does):
  // a separate pass does
  const DomainArgs dom{beta, (size_t)B * H * T * d_v, in_dtype == PALIMPSA_BF16, d_t, (size_t)B * H * T, nullptr,
                       0, A, I_prior, H, st};
  if (launch_domain_check(dom, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  StreamOrderedScratch scratch;
  if (launch_segment_summary(a, summary, gamma, static_cast<cudaStream_t>(cuda_stream), &scratch) != cudaSuccess)
    return PALIMPSA_ERR_CUDA;
  return PALIMPSA_OK;
}

palimpsa_status palimpsa_state_combine(const float* summaries, const float* gammas, int R, const float* I_prior,
                                       const float* mu0, const float* I0, float* mu_out, float* I_out, int B, int H,
                                       int d_k, int d_v, void* cuda_stream) {
  if (!I_prior || !mu_out || !I_out) return PALIMPSA_ERR_NULL;
  if (R > 0 && (!summaries || !gammas)) return PALIMPSA_ERR_NULL;
  if (R < 0 || !sizes_ok(B, H, R > 0 ? R : 1, d_k, d_v)) return PALIMPSA_ERR_SHAPE;
  if (!supported_dims(d_k, d_v)) return PALIMPSA_ERR_UNSUPPORTED;
  const void* a16[] = {summaries, mu0, I0, mu_out, I_out};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return PALIMPSA_ERR_ALIGN;
  const void* a4[] = {gammas, I_prior};
  for (const void* p : a4)
    if (p && !aligned(p, 4)) return PALIMPSA_ERR_ALIGN;
  const long long heads = (long long)B * H, DVK = (long long)d_v * d_k;
  unsigned int* st = nullptr;
  if (palimpsa_status s = status_word(&st)) return s;
  // the preconditions this call reads (I_prior > 0, I0 > 0), checked by a separate pass
  const DomainArgs dom{nullptr, 0, false, nullptr, 0, I0, I0 ? (size_t)(heads * DVK) : 0, nullptr, I_prior, H, st};
  if (launch_domain_check(dom, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  const FoldArgs f{summaries, gammas, heads * 2 * DVK, 2 * DVK, heads, 1, R, heads, H, (int)DVK, true, I_prior,
                   mu0, I0, mu_out, I_out, nullptr, DVK};
  if (launch_fold(f, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  return PALIMPSA_OK;
}

palimpsa_status palimpsa_forward_fused(const void* q, const void* k, const void* v, const void* beta_raw,
                                       const float* d_raw, const float* A, const float* I_prior,
                                       const float* b_scale, const float* mu0, const float* I0, float* y,
                                       float* mu_T, float* I_T, int B, int H, int T, int d_k, int d_v, int chunk,
                                       unsigned int flags, palimpsa_dtype in_dtype, void* cuda_stream) {
  if (flags & ~kKnownFuseFlags) return PALIMPSA_ERR_UNSUPPORTED;
  if (b_scale && !aligned(b_scale, 4)) return PALIMPSA_ERR_ALIGN;
  return forward_impl(q, k, v, beta_raw, d_raw, A, I_prior, mu0, I0, y, mu_T, I_T, B, H, T, d_k, d_v, chunk,
                      in_dtype, cuda_stream, fused_prologue(b_scale, flags));
}

palimpsa_status palimpsa_step_fused(const void* q, const void* k, const void* v, const void* beta_raw,
                                    const float* d_raw, const float* A, const float* I_prior, const float* b_scale,
                                    float* mu, float* I, float* y, int B, int H, int d_k, int d_v,
                                    unsigned int flags, palimpsa_dtype in_dtype, void* cuda_stream) {
  if (flags & ~kKnownFuseFlags) return PALIMPSA_ERR_UNSUPPORTED;
  return step_impl(q, k, v, beta_raw, d_raw, A, I_prior, mu, I, y, B, H, d_k, d_v, in_dtype, cuda_stream,
                   fused_prologue(b_scale, flags));
}

palimpsa_status palimpsa_forward_without_meta(const void* q, const void* k, const void* v, const void* beta,
                                              const float* d_t, const float* A, const float* I_prior,
                                              const float* mu0, float* y, float* mu_T, int B, int H, int T,
                                              int d_k, int d_v, int chunk, palimpsa_dtype in_dtype,
                                              void* cuda_stream) {
  if (!A || !I_prior || !mu_T) return PALIMPSA_ERR_NULL;
  if (T != 0 && (!q || !k || !v || !beta || !d_t || !y)) return PALIMPSA_ERR_NULL;
  if (in_dtype != PALIMPSA_F32 && in_dtype != PALIMPSA_BF16) return PALIMPSA_ERR_DTYPE;
  if (!sizes_ok(B, H, T, d_k, d_v)) return PALIMPSA_ERR_SHAPE;
  if (!supported_dims(d_k, d_v)) return PALIMPSA_ERR_UNSUPPORTED;
  if (!chunk_ok(chunk)) return PALIMPSA_ERR_UNSUPPORTED;
  const void* a16[] = {q, k, v, beta, y, mu_T, mu0};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return PALIMPSA_ERR_ALIGN;
  const void* a4[] = {d_t, A, I_prior};
  for (const void* p : a4)
    if (p && !aligned(p, 4)) return PALIMPSA_ERR_ALIGN;
  unsigned int* st = nullptr;
  if (palimpsa_status s = status_word(&st)) return s;
  FwdArgs a{q, k, v, beta, d_t, A, I_prior, mu0, nullptr, y, mu_T, nullptr, B, H, T, d_k, d_v,
            chunk == 0 ? 32 : chunk, in_dtype == PALIMPSA_BF16, st,
            g_wait_timeout_ns.load(), g_withhold_first_copy.load(), g_forward_segments.load()};
  StreamOrderedScratch scratch;
  if (launch_forward_without_meta(a, static_cast<cudaStream_t>(cuda_stream), &scratch) != cudaSuccess)
    return PALIMPSA_ERR_CUDA;
  return PALIMPSA_OK;
}

}  // extern "C"

namespace palimpsa {
namespace {

palimpsa_status backward_impl(const void* q, const void* k, const void* v, const void* beta, const float* d_t,
                              const float* A, const float* I_prior, const float* mu0, const float* I0,
                              const float* dy, const float* dmu_T, const float* dI_T, float* dq, float* dk,
                              float* dv, float* dbeta, float* dd_t, float* dA, float* dI_prior, float* dmu0,
                              float* dI0, const float* ckpt, int B, int H, int T, int d_k, int d_v,
                              palimpsa_dtype in_dtype, void* cuda_stream, const int* cu_seqlens = nullptr,
                              int total_T = 0) {
  // Dense layout: B sequences of T tokens each. Packed layout (cu_seqlens set):
  // B sequences, at most T tokens each, total_T tokens in all.
  const bool packed = cu_seqlens != nullptr;
  const long long ntok = packed ? total_T : (long long)B * T;
  if (!A || !I_prior || !dA || !dI_prior) return PALIMPSA_ERR_NULL;
  if (ntok != 0 && (!q || !k || !v || !beta || !d_t || !dy || !dq || !dk || !dv || !dbeta || !dd_t))
    return PALIMPSA_ERR_NULL;
  if (in_dtype != PALIMPSA_F32 && in_dtype != PALIMPSA_BF16) return PALIMPSA_ERR_DTYPE;
  if (!sizes_ok(B, H, T, d_k, d_v)) return PALIMPSA_ERR_SHAPE;
  if (packed && (total_T < 0 || T > total_T || !sizes_ok(1, H, total_T, d_k, d_v))) return PALIMPSA_ERR_SHAPE;
  if (!supported_dims(d_k, d_v)) return PALIMPSA_ERR_UNSUPPORTED;
  const void* a16[] = {q, k, v, beta, mu0, I0, dy, dmu_T, dI_T, dq, dk, dv, dbeta, dmu0, dI0, ckpt};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return PALIMPSA_ERR_ALIGN;
  const void* a4[] = {d_t, A, I_prior, dd_t, dA, dI_prior, cu_seqlens};
  for (const void* p : a4)
    if (p && !aligned(p, 4)) return PALIMPSA_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  BwdArgs a{q, k, v, beta, d_t, A, I_prior, mu0, I0, dy, dmu_T, dI_T, dq, dk, dv, dbeta, dd_t, dA, dI_prior,
            dmu0, dI0, B, H, T, d_k, d_v, in_dtype == PALIMPSA_BF16};
  a.ckpt_in = ckpt;
  if (palimpsa_status st = status_word(&a.status)) return st;
  if (packed) {
    a.cu_seqlens = cu_seqlens;
    a.total_T = total_T;
  }
  const size_t tok = packed ? (size_t)H * total_T : (size_t)B * H * T;
  // outputs that the kernel accumulates into start at zero
  if (tok != 0 && (cudaMemsetAsync(dq, 0, tok * d_k * sizeof(float), s) != cudaSuccess ||
                 cudaMemsetAsync(dk, 0, tok * d_k * sizeof(float), s) != cudaSuccess ||
                 cudaMemsetAsync(dd_t, 0, tok * sizeof(float), s) != cudaSuccess))
    return PALIMPSA_ERR_CUDA;
  if (cudaMemsetAsync(dA, 0, (size_t)H * sizeof(float), s) != cudaSuccess ||
      cudaMemsetAsync(dI_prior, 0, (size_t)H * sizeof(float), s) != cudaSuccess)
    return PALIMPSA_ERR_CUDA;
  // the kernel does not test the preconditions as it reads the inputs: a separate pass does
  const DomainArgs dom{beta, tok * (size_t)d_v, in_dtype == PALIMPSA_BF16, d_t, tok, I0,
                       (size_t)B * H * d_v * d_k, A, I_prior, H, a.status};
  if (launch_domain_check(dom, s) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  StreamOrderedScratch scratch;
  float* ck = nullptr;
  const size_t bytes = backward_scratch_bytes(a);
  if (bytes && scratch.acquire(bytes, s, &ck) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  const cudaError_t e = launch_backward(a, ck, s);
  const cudaError_t e2 = ck ? scratch.release(ck, s) : cudaSuccess;
  if (e != cudaSuccess || e2 != cudaSuccess) return PALIMPSA_ERR_CUDA;
  return PALIMPSA_OK;
}

}  // namespace
}  // namespace palimpsa

extern "C" {

palimpsa_status palimpsa_backward(const void* q, const void* k, const void* v, const void* beta, const float* d_t,
                                  const float* A, const float* I_prior, const float* mu0, const float* I0,
                                  const float* dy, const float* dmu_T, const float* dI_T, float* dq, float* dk,
                                  float* dv, float* dbeta, float* dd_t, float* dA, float* dI_prior, float* dmu0,
                                  float* dI0, int B, int H, int T, int d_k, int d_v, palimpsa_dtype in_dtype,
                                  void* cuda_stream) {
  return backward_impl(q, k, v, beta, d_t, A, I_prior, mu0, I0, dy, dmu_T, dI_T, dq, dk, dv, dbeta, dd_t, dA,
                       dI_prior, dmu0, dI0, nullptr, B, H, T, d_k, d_v, in_dtype, cuda_stream);
}

palimpsa_status palimpsa_backward_checkpointed(const void* q, const void* k, const void* v, const void* beta,
                                               const float* d_t, const float* A, const float* I_prior,
                                               const float* mu0, const float* I0, const float* dy,
                                               const float* dmu_T, const float* dI_T, float* dq, float* dk,
                                               float* dv, float* dbeta, float* dd_t, float* dA, float* dI_prior,
                                               float* dmu0, float* dI0, const float* ckpt, int B, int H, int T,
                                               int d_k, int d_v, palimpsa_dtype in_dtype, void* cuda_stream) {
  if (!ckpt && T != 0) return PALIMPSA_ERR_NULL;
  return backward_impl(q, k, v, beta, d_t, A, I_prior, mu0, I0, dy, dmu_T, dI_T, dq, dk, dv, dbeta, dd_t, dA,
                       dI_prior, dmu0, dI0, ckpt, B, H, T, d_k, d_v, in_dtype, cuda_stream);
}

palimpsa_status palimpsa_backward_varlen(const void* q, const void* k, const void* v, const void* beta,
                                         const float* d_t, const float* A, const float* I_prior, const float* mu0,
                                         const float* I0, const float* dy, const float* dmu_T, const float* dI_T,
                                         float* dq, float* dk, float* dv, float* dbeta, float* dd_t, float* dA,
                                         float* dI_prior, float* dmu0, float* dI0, const float* ckpt,
                                         const int* cu_seqlens, int N, int H, int total_T, int max_seqlen, int d_k,
                                         int d_v, palimpsa_dtype in_dtype, void* cuda_stream) {
  if (!cu_seqlens) return PALIMPSA_ERR_NULL;
  return backward_impl(q, k, v, beta, d_t, A, I_prior, mu0, I0, dy, dmu_T, dI_T, dq, dk, dv, dbeta, dd_t, dA,
                       dI_prior, dmu0, dI0, ckpt, N, H, max_seqlen, d_k, d_v, in_dtype, cuda_stream, cu_seqlens,
                       total_T);
}

size_t palimpsa_checkpoint_bytes(int B, int H, int T, int d_k, int d_v) {
  if (B < 1 || H < 1 || T < 0 || d_k < 1 || d_v < 1) return 0;
  return checkpoint_floats((long long)B * H, T, d_k, d_v) * sizeof(float);
}

size_t palimpsa_checkpoint_bytes_varlen(int N, int H, int total_T, int d_k, int d_v) {
  if (N < 1 || H < 1 || total_T < 0 || d_k < 1 || d_v < 1) return 0;
  return (size_t)H * packed_checkpoint_slots(total_T, N) * d_v * 2 * d_k * sizeof(float);
}

palimpsa_status palimpsa_forward_checkpointed(const void* q, const void* k, const void* v, const void* beta,
                                              const float* d_t, const float* A, const float* I_prior,
                                              const float* mu0, const float* I0, float* y, float* mu_T, float* I_T,
                                              float* ckpt, int B, int H, int T, int d_k, int d_v, int chunk,
                                              palimpsa_dtype in_dtype, void* cuda_stream) {
  if (!ckpt && T != 0) return PALIMPSA_ERR_NULL;
  return forward_impl(q, k, v, beta, d_t, A, I_prior, mu0, I0, y, mu_T, I_T, B, H, T, d_k, d_v, chunk, in_dtype,
                      cuda_stream, Prologue{}, ckpt);
}

palimpsa_status palimpsa_step(const void* q, const void* k, const void* v, const void* beta,
                              const float* d_t, const float* A, const float* I_prior, float* mu, float* I,
                              float* y, int B, int H, int d_k, int d_v, palimpsa_dtype in_dtype,
                              void* cuda_stream) {
  return step_impl(q, k, v, beta, d_t, A, I_prior, mu, I, y, B, H, d_k, d_v, in_dtype, cuda_stream, Prologue{});
}

palimpsa_status palimpsa_step_sequence(const void* q, const void* k, const void* v, const void* beta,
                                       const float* d_t, const float* A, const float* I_prior, float* mu, float* I,
                                       float* y, int S, int B, int H, int d_k, int d_v, palimpsa_dtype in_dtype,
                                       void* cuda_stream) {
  return palimpsa::step_sequence_impl(q, k, v, beta, d_t, A, I_prior, mu, I, y, S, B, H, d_k, d_v, in_dtype,
                                      cuda_stream, palimpsa::Prologue{});
}

palimpsa_status palimpsa_step_sequence_fused(const void* q, const void* k, const void* v, const void* beta_raw,
                                             const float* d_raw, const float* A, const float* I_prior,
                                             const float* b_scale, float* mu, float* I, float* y, int S, int B,
                                             int H, int d_k, int d_v, unsigned int flags, palimpsa_dtype in_dtype,
                                             void* cuda_stream) {
  if (flags & ~kKnownFuseFlags) return PALIMPSA_ERR_UNSUPPORTED;
  return palimpsa::step_sequence_impl(q, k, v, beta_raw, d_raw, A, I_prior, mu, I, y, S, B, H, d_k, d_v,
                                      in_dtype, cuda_stream, fused_prologue(b_scale, flags));
}

const char* palimpsa_status_string(palimpsa_status s) {
  switch (s) {
    case PALIMPSA_OK: return "ok";
    case PALIMPSA_ERR_NULL: return "a required pointer is NULL";
    case PALIMPSA_ERR_SHAPE: return "a size is out of range";
    case PALIMPSA_ERR_ALIGN: return "a pointer is not aligned as required";
    case PALIMPSA_ERR_DTYPE: return "unknown input dtype";
    case PALIMPSA_ERR_DOMAIN: return "an input broke a precondition (A, I_prior, I0 > 0; d_t, beta >= 0)";
    case PALIMPSA_ERR_UNSUPPORTED: return "d_k, d_v or chunk not supported";
    case PALIMPSA_ERR_CUDA: return "a CUDA runtime call failed";
    case PALIMPSA_ERR_TIMEOUT: return "a bounded device wait gave up";
    case PALIMPSA_ERR_SCRATCH_LIMIT: return "the call needs more scratch than the fixed no-allocation buffer holds";
  }
  return "unknown status";
}

palimpsa_status palimpsa_get_device_status(void* cuda_stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  unsigned int* st = nullptr;
  if (palimpsa_status s = status_word(&st)) return s;
  unsigned int bits = 0;
  if (cudaMemcpy(&bits, st, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  if (bits) {
    const unsigned int zero = 0;
    if (cudaMemcpy(st, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  }
  if (bits & kStatusTimeout) return PALIMPSA_ERR_TIMEOUT;
  if (bits & kStatusDomain) return PALIMPSA_ERR_DOMAIN;
  return PALIMPSA_OK;
}

int palimpsa_abi_version(void) { return PALIMPSA_ABI_VERSION; }

void palimpsa_set_wait_timeout_ns(uint64_t ns) { g_wait_timeout_ns.store(ns); }

void palimpsa_debug_withhold_first_copy(int on) { g_withhold_first_copy.store(on ? 1 : 0); }

void palimpsa_set_forward_segments(int segments) { g_forward_segments.store(segments > 0 ? segments : 0); }

void palimpsa_set_step_l2_keep_bytes(long long bytes) { g_step_l2_keep_bytes.store(bytes > 0 ? bytes : 0); }

palimpsa_status palimpsa_set_scratch_retention(unsigned long long bytes) {
  g_scratch_keep_bytes.store(bytes);
  std::lock_guard<std::mutex> lock(g_pool_mu);
  for (cudaMemPool_t pool : g_pools) {
    if (!pool) continue;
    unsigned long long keep = bytes;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  }
  return PALIMPSA_OK;
}

palimpsa_status palimpsa_release_scratch(void) {
  cudaMemPool_t pool = nullptr;
  if (palimpsa_status s = existing_pool(&pool)) return s;
  if (!pool) return PALIMPSA_OK;
  // every call's scratch is freed in stream order; once the device is idle
  // none of it backs work in flight and all of it can go
  if (cudaDeviceSynchronize() != cudaSuccess) return PALIMPSA_ERR_CUDA;
  if (cudaMemPoolTrimTo(pool, 0) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  return PALIMPSA_OK;
}

palimpsa_status palimpsa_scratch_reserved_bytes(size_t* bytes) {
  if (!bytes) return PALIMPSA_ERR_NULL;
  *bytes = 0;
  cudaMemPool_t pool = nullptr;
  if (palimpsa_status s = existing_pool(&pool)) return s;
  if (!pool) return PALIMPSA_OK;
  unsigned long long v = 0;  // cuuint64_t
  if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &v) != cudaSuccess) return PALIMPSA_ERR_CUDA;
  *bytes = (size_t)v;
  return PALIMPSA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// palimpsa_forward_chunked_noalloc: the chunked forward for callers that must
// not allocate device memory. Its time-split scratch lives in one fixed,
// file-scope device array instead of coming from the stream-ordered
// allocator.
namespace palimpsa {
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB per device, held until the process exits

// The shared scratch. Device code never names it directly: the host looks up
// its device address (once per device) and passes that pointer to the kernels.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the current device's scratch array. The first call on a
// device does the lookup with that device current.
palimpsa_status noalloc_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PALIMPSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PALIMPSA_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return PALIMPSA_OK;
}

// Hands out the fixed array; a request larger than the array is refused before
// any kernel is launched. Nothing is allocated and nothing is freed.
struct FixedScratch final : ScratchProvider {
  float* base = nullptr;
  bool too_large = false;
  cudaError_t acquire(size_t bytes, cudaStream_t, float** p) override {
    if (bytes > kNoAllocScratchBytes) {
      too_large = true;
      return cudaErrorMemoryAllocation;
    }
    *p = base;
    return cudaSuccess;
  }
  cudaError_t release(float*, cudaStream_t) override { return cudaSuccess; }
};

}  // namespace
}  // namespace palimpsa

extern "C" palimpsa_status palimpsa_forward_chunked_noalloc(
    const void* q, const void* k, const void* v, const void* beta, const float* d_t, const float* A,
    const float* I_prior, const float* mu0, const float* I0, float* y, float* mu_T, float* I_T, int B, int H,
    int T, int d_k, int d_v, int chunk, palimpsa_dtype in_dtype, void* cuda_stream) {
  if (!A || !I_prior || !mu_T || !I_T) return PALIMPSA_ERR_NULL;
  if (T != 0 && (!q || !k || !v || !beta || !d_t || !y)) return PALIMPSA_ERR_NULL;
  if (in_dtype != PALIMPSA_F32 && in_dtype != PALIMPSA_BF16) return PALIMPSA_ERR_DTYPE;
  if (!sizes_ok(B, H, T, d_k, d_v)) return PALIMPSA_ERR_SHAPE;
  if (!supported_dims(d_k, d_v)) return PALIMPSA_ERR_UNSUPPORTED;
  if (!chunk_ok(chunk)) return PALIMPSA_ERR_UNSUPPORTED;
  const void* a16[] = {q, k, v, beta, y, mu_T, I_T, mu0, I0};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return PALIMPSA_ERR_ALIGN;
  const void* a4[] = {d_t, A, I_prior};
  for (const void* p : a4)
    if (p && !aligned(p, 4)) return PALIMPSA_ERR_ALIGN;
  unsigned int* st = nullptr;
  if (palimpsa_status s = status_word(&st)) return s;
  FixedScratch scratch;
  if (palimpsa_status s = noalloc_scratch(&scratch.base)) return s;
  FwdArgs a{q, k, v, beta, d_t, A, I_prior, mu0, I0, y, mu_T, I_T, B, H, T, d_k, d_v,
            chunk == 0 ? 32 : chunk, in_dtype == PALIMPSA_BF16, st,
            g_wait_timeout_ns.load(), g_withhold_first_copy.load(), g_forward_segments.load()};
  const cudaError_t e = launch_forward_chunked(a, static_cast<cudaStream_t>(cuda_stream), &scratch);
  if (scratch.too_large) return PALIMPSA_ERR_SCRATCH_LIMIT;
  if (e != cudaSuccess) return PALIMPSA_ERR_CUDA;
  return PALIMPSA_OK;
}
