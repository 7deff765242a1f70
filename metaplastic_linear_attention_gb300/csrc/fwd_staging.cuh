// Chunk staging shared by the chunked forward kernels: the shared-memory
// carve-up, the bulk-copy ring with bounded mbarrier waits, the tile a CTA
// works on, and the conversion of a staged chunk into fp32 key/query operands.
#pragma once

#include "palimpsa_internal.cuh"

namespace palimpsa {
namespace fwd {

constexpr int kLanesPerRow = 8;

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory carve-up for one CTA (all offsets 16-byte aligned).
struct FwdSmem {
  size_t raw_q, raw_k, raw_v, raw_b, raw_bytes;  // one raw stage (q, k, v, beta of a chunk)
  size_t kf, k2f, qf, bvf, bf, alf, omf, bars, flag, total;

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
    bars = o; o += 2 * sizeof(uint64_t);
    flag = o; o += 16;
    total = align_up(o, 128);
  }
};

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// One thread: stage tokens [t0, t0 + tc) of q, k, v, beta into one raw buffer
// with four bulk copies whose bytes complete on `bar`.
template <int DK, int ES>
__device__ __forceinline__ void stage_chunk(unsigned char* base, const FwdSmem& L, uint64_t* bar,
                                            const char* gq, const char* gk, const char* gv,
                                            const char* gb, int t0, int tc, int DV) {
  const uint32_t bq = (uint32_t)tc * DK * ES, bvb = (uint32_t)tc * DV * ES;
  mbar_arrive_expect_tx(bar, 2 * bq + 2 * bvb);
  bulk_g2s(base + L.raw_q, gq + (size_t)t0 * DK * ES, bq, bar);
  bulk_g2s(base + L.raw_k, gk + (size_t)t0 * DK * ES, bq, bar);
  bulk_g2s(base + L.raw_v, gv + (size_t)t0 * DV * ES, bvb, bar);
  bulk_g2s(base + L.raw_b, gb + (size_t)t0 * DV * ES, bvb, bar);
}

// Where a CTA works: head bh (sequence n = bh / H of a packed batch), segment
// seg, rows [row0, row0 + RG), tokens [tb, tb + tn) of that sequence, whose
// first token is head_tok in the token-major input arrays and whose length is
// L; last_seg is the sequence's final segment. A packed sequence whose offsets
// are out of order or out of range is `bad`: the CTA must touch nothing.
struct Tile {
  long bh;
  int h, seg, row0, tb, tn, L, last_seg;
  size_t head_tok;
  bool bad;
};

// Length and first token (in the token-major input arrays) of head bh's
// sequence. Returns false, with L = 0, when packed offsets are out of order or
// out of range; nothing of that sequence may then be touched.
__device__ __forceinline__ bool seq_extent(const FwdArgs& a, long bh, int* L, size_t* head_tok) {
  if (!a.cu_seqlens) {
    *L = a.T;
    *head_tok = (size_t)bh * a.T;
    return true;
  }
  const long n = bh / a.H;
  const int h = (int)(bh % a.H);
  const int s0 = a.cu_seqlens[n], s1 = a.cu_seqlens[n + 1];
  const bool ok = s0 >= 0 && s1 >= s0 && (long long)s1 <= a.total_T && s1 - s0 <= a.T;
  *L = ok ? s1 - s0 : 0;
  *head_tok = ok ? (size_t)h * (size_t)a.total_T + (size_t)s0 : 0;
  return ok;
}

__device__ __forceinline__ Tile tile_of(const FwdArgs& a, int RG, int nseg, int seg_len) {
  const int groups = a.d_v / RG;
  Tile t;
  const long cta = blockIdx.x;
  const int rg = (int)(cta % groups);
  const long rest = cta / groups;
  t.seg = (int)(rest % nseg);
  t.bh = rest / nseg;
  t.h = (int)(t.bh % a.H);
  t.row0 = rg * RG;
  t.bad = !seq_extent(a, t.bh, &t.L, &t.head_tok);
  t.tb = t.seg * seg_len;
  t.tn = max(0, min(t.L, t.tb + seg_len) - t.tb);
  t.last_seg = t.L > 0 ? (t.L - 1) / seg_len : 0;
  return t;
}

// The staged-chunk pipeline shared by pass A and pass C: chunk order, the raw
// ring, bounded waits and the timeout exit. Chunk c (0-based in processing
// order) is segment-local chunk `reverse ? nch - 1 - c : c`.
template <int DK, int ES>
struct ChunkPipe {
  const FwdSmem& L;
  unsigned char* smem;
  uint64_t* bars;
  volatile int* flag;
  const char *gq, *gk, *gv, *gb;
  int C, tb, tn, DV, nch;
  bool reverse;
  // thread 0's record of copies in flight, for a clean exit after a timeout
  bool pend0 = false, pend1 = false;
  uint32_t par0 = 0, par1 = 0;

  __device__ ChunkPipe(const FwdSmem& L_, unsigned char* s, const char* q, const char* k, const char* v,
                       const char* b, int C_, int tb_, int tn_, int DV_, bool rev)
      : L(L_), smem(s), bars(reinterpret_cast<uint64_t*>(s + L_.bars)),
        flag(reinterpret_cast<volatile int*>(s + L_.flag)), gq(q), gk(k), gv(v), gb(b), C(C_), tb(tb_),
        tn(tn_), DV(DV_), nch((tn_ + C_ - 1) / C_), reverse(rev) {}

  __device__ int t0_of(int c) const { return (reverse ? nch - 1 - c : c) * C; }  // segment-local
  __device__ int tc_of(int c) const { return min(C, tn - t0_of(c)); }
  __device__ unsigned char* raw(int c) const { return smem + (size_t)(c & 1) * L.raw_bytes; }

  __device__ void issue(int c) {  // thread 0 only
    stage_chunk<DK, ES>(raw(c), L, &bars[c & 1], gq, gk, gv, gb, tb + t0_of(c), tc_of(c), DV);
    const uint32_t par = (uint32_t)(c >> 1) & 1u;
    if ((c & 1) == 0) { pend0 = true; par0 = par; } else { pend1 = true; par1 = par; }
  }

  __device__ void init(bool withhold_first) {  // all threads; thread 0 does the work
    if (threadIdx.x == 0) {
      mbar_init(&bars[0], 1);
      mbar_init(&bars[1], 1);
      *flag = 0;
      fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int c = 0; c < 2 && c < nch; ++c) {
        if (c == 0 && withhold_first) continue;
        issue(c);
      }
    }
  }

  // All threads: wait until chunk c has landed. Returns false (for every
  // thread, consistently) after a timeout; the caller must then return.
  __device__ bool wait(int c, unsigned long long timeout_ns, unsigned int* status) {
    if (!mbar_wait_bounded(&bars[c & 1], (uint32_t)(c >> 1) & 1u, timeout_ns)) *flag = 1;
    __syncthreads();
    if (*flag) {
      if (threadIdx.x == 0) {
        latch_status(status, kStatusTimeout);
        const unsigned long long drain_ns = 1000000000ull;
        if (pend0) mbar_wait_bounded(&bars[0], par0, drain_ns);
        if (pend1) mbar_wait_bounded(&bars[1], par1, drain_ns);
      }
      __syncthreads();
      return false;
    }
    if (threadIdx.x == 0) { if ((c & 1) == 0) pend0 = false; else pend1 = false; }
    return true;
  }

  // After the CTA-wide barrier that ends the conversion of chunk c: refill its
  // raw buffer with chunk c + 2 (thread 0).
  __device__ void refill(int c) {
    if (threadIdx.x == 0 && c + 2 < nch) issue(c + 2);
  }
};

// Convert the landed raw chunk to fp32 k, k^2 (and q when WITH_Q) shared by all
// rows. NTH threads cooperate. With `norm` (uniform over the CTA) each token's
// k and q are divided by their L2 norm first: the G = d_k / 8 items of a token
// sit on G consecutive, G-aligned lanes of one warp (NTH is a multiple of 32),
// which sum their squares with a butterfly inside that lane group.
template <int DK, bool BF16, bool WITH_Q, int NTH>
__device__ __forceinline__ void convert_keys(const unsigned char* raw, const FwdSmem& L, unsigned char* smem,
                                             int tc, bool norm) {
  float* kf = reinterpret_cast<float*>(smem + L.kf);
  float* k2f = reinterpret_cast<float*>(smem + L.k2f);
  float* qf = reinterpret_cast<float*>(smem + L.qf);
  constexpr int PER = 8;
  constexpr int G = DK / PER;  // items (lanes) per token
  static_assert(32 % G == 0 && NTH % 32 == 0, "a token's items must fill aligned lane groups");
  const int items = tc * DK / PER;
  for (int it = threadIdx.x; it < items; it += NTH) {
    float kv[PER], qv[PER];
    if constexpr (BF16) {
      const uint4 k8 = *reinterpret_cast<const uint4*>(raw + L.raw_k + (size_t)it * 16);
      const uint32_t kw[4] = {k8.x, k8.y, k8.z, k8.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) { kv[2 * e] = bf16_lo(kw[e]); kv[2 * e + 1] = bf16_hi(kw[e]); }
      if constexpr (WITH_Q) {
        const uint4 q8 = *reinterpret_cast<const uint4*>(raw + L.raw_q + (size_t)it * 16);
        const uint32_t qw[4] = {q8.x, q8.y, q8.z, q8.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) { qv[2 * e] = bf16_lo(qw[e]); qv[2 * e + 1] = bf16_hi(qw[e]); }
      }
    } else {
      const float4* k4 = reinterpret_cast<const float4*>(raw + L.raw_k) + 2 * it;
      const float4 ka = k4[0], kb = k4[1];
      kv[0] = ka.x; kv[1] = ka.y; kv[2] = ka.z; kv[3] = ka.w;
      kv[4] = kb.x; kv[5] = kb.y; kv[6] = kb.z; kv[7] = kb.w;
      if constexpr (WITH_Q) {
        const float4* q4 = reinterpret_cast<const float4*>(raw + L.raw_q) + 2 * it;
        const float4 qa = q4[0], qb = q4[1];
        qv[0] = qa.x; qv[1] = qa.y; qv[2] = qa.z; qv[3] = qa.w;
        qv[4] = qb.x; qv[5] = qb.y; qv[6] = qb.z; qv[7] = qb.w;
      }
    }
    if (norm) {
      const unsigned lane = threadIdx.x & 31u;
      const unsigned gmask = G == 32 ? 0xffffffffu : ((1u << G) - 1u) << (lane & ~(unsigned)(G - 1));
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        sk = fmaf(kv[e], kv[e], sk);
        if constexpr (WITH_Q) sq = fmaf(qv[e], qv[e], sq);
      }
#pragma unroll
      for (int m = 1; m < G; m <<= 1) {
        sk += __shfl_xor_sync(gmask, sk, m);
        if constexpr (WITH_Q) sq += __shfl_xor_sync(gmask, sq, m);
      }
      const float ik = rsqrtf(fmaxf(sk, kNormFloorSq));
#pragma unroll
      for (int e = 0; e < PER; ++e) kv[e] *= ik;
      if constexpr (WITH_Q) {
        const float iq = rsqrtf(fmaxf(sq, kNormFloorSq));
#pragma unroll
        for (int e = 0; e < PER; ++e) qv[e] *= iq;
      }
    }
    float4* ko = reinterpret_cast<float4*>(kf) + 2 * it;
    float4* k2o = reinterpret_cast<float4*>(k2f) + 2 * it;
    ko[0] = make_float4(kv[0], kv[1], kv[2], kv[3]);
    ko[1] = make_float4(kv[4], kv[5], kv[6], kv[7]);
    k2o[0] = make_float4(kv[0] * kv[0], kv[1] * kv[1], kv[2] * kv[2], kv[3] * kv[3]);
    k2o[1] = make_float4(kv[4] * kv[4], kv[5] * kv[5], kv[6] * kv[6], kv[7] * kv[7]);
    if constexpr (WITH_Q) {
      float4* qo = reinterpret_cast<float4*>(qf) + 2 * it;
      qo[0] = make_float4(qv[0], qv[1], qv[2], qv[3]);
      qo[1] = make_float4(qv[4], qv[5], qv[6], qv[7]);
    }
  }
}

template <bool BF16>
__device__ __forceinline__ float raw_elem(const unsigned char* base, size_t e) {
  if constexpr (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[e]);
  else return reinterpret_cast<const float*>(base)[e];
}

}  // namespace fwd
}  // namespace palimpsa
