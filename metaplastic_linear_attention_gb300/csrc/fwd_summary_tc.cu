// Pass A of the forward's time split on the 5th-generation tensor cores
// (tcgen05, sm_103a): the segment summaries as dense contractions over tokens.
//
// Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
// Attention-Based Models" — slide 9 (App. A.12): both natural-parameter
// recurrences are affine in the state with the shared decay alpha, so a
// segment acts on the state as (M, Ibar) -> Gamma (M, Ibar) + (dM, dIbar) with
//   dM[i][j]    = sum_t W_t beta_ti v_ti k_tj,   dIbar[i][j] = sum_t W_t beta_ti k_tj^2,
//   W_t = prod_{u > t in segment} alpha_u,       Gamma = prod_t alpha_t.
// Both sums are matrix products over the segment's tokens, computed here as
//   D_M^T = K^T X,  D_I^T = (K^2)^T Y,   X[t][i] = W_t beta_ti v_ti,  Y[t][i] = W_t beta_ti,
// with M = d_k = 128 key columns on the TMEM lanes, N = d_v, K = tokens.
//
// Precision (fp32 results from bf16 operands): k is exact in bf16 (bf16
// inputs); k^2 has at most 16 significant bits and is split exactly into
// hi + lo bf16 parts; X and Y are fp32 and are split into hi + lo bf16 parts
// (about 2^-17 relative error). Per 16 tokens that is five MMAs:
//   D_M += K^T X_hi + K^T X_lo,   D_I += (K^2)_hi^T Y_hi + (K^2)_hi^T Y_lo + (K^2)_lo^T Y_hi
// (the dropped (K^2)_lo^T Y_lo term is below 2^-16 relative).
//
// Structure: one CTA per (head, segment), 8 warps with two roles. The raw k,
// v, beta of each 32-token chunk arrive by bulk async copy into a 2-deep ring.
// Warp 0 is the control warp: one of its threads issues the copies, and the
// MMAs of a chunk once its operand tiles are complete, followed by a
// tcgen05.commit that frees the operand buffer again. Warps 1-7 build the
// tiles: each forms the chunk's suffix products W itself (a warp scan over the
// 32 tokens), so no CTA barrier sits in the chunk loop; the roles meet only at
// mbarriers (raw stage full, operand buffer full, operand buffer free, and
// among the builders the key-norm scales of the fused prologue). The
// tiles are MN-major without swizzle, the layout in which the staged rows
// already lie: a 16-byte row holds 8 consecutive key columns (or value rows)
// of one token, so building a tile moves whole 16-byte pieces of the staged k,
// v and beta and never transposes within one. The accumulators stay in TMEM
// (2 d_v columns) for the whole segment and are read back once with
// tcgen05.ld. Every wait is bounded; on a timeout the CTA records it, drains
// its copies and MMAs (bounded), frees its TMEM and returns.
#include <cuda_bf16.h>

#include "fwd_staging.cuh"

namespace palimpsa {
namespace {

using namespace fwd;

constexpr int kTcThreads = 256;
constexpr int kTcBuilders = kTcThreads - 32;  // warps 1-7 build the operand tiles
constexpr int kTcC = 32;     // tokens per chunk: two K = 16 MMA steps
constexpr int kTcDK = 128;   // key columns = MMA M

// Shared-memory carve-up (byte offsets).
struct TcSmem {
  size_t raw_k, raw_v, raw_b, raw_bytes;    // one raw stage (k, v, beta of a chunk)
  size_t ops, op_bytes;                      // two operand buffers
  size_t kt, k2h, k2l, xh, xl, yh, yl;       // tiles inside an operand buffer (one chunk each)
  size_t a_tile, b_tile;                     // bytes of one chunk's M- / N-side tile
  size_t ns, gam, bars, fbars, mbars, nbars, slot, flag, issued, total;

  __host__ __device__ explicit TcSmem(int DV) {
    raw_k = 0;
    raw_v = align_up(raw_k + (size_t)kTcC * kTcDK * 2, 16);
    raw_b = align_up(raw_v + (size_t)kTcC * DV * 2, 16);
    raw_bytes = align_up(raw_b + (size_t)kTcC * DV * 2, 128);
    ops = align_up(2 * raw_bytes, 1024);
    a_tile = (size_t)kTcDK * kTcC * 2;
    b_tile = (size_t)DV * kTcC * 2;
    kt = 0;
    k2h = kt + a_tile;
    k2l = k2h + a_tile;
    xh = k2l + a_tile;
    xl = xh + b_tile;
    yh = xl + b_tile;
    yl = yh + b_tile;
    op_bytes = align_up(yl + b_tile, 1024);
    size_t o = ops + 2 * op_bytes;
    ns = o;    o += 2 * kTcC * 4;  // per-token 1 / ||k_t|| (q/k norm), two chunks
    gam = o;   o += 16;            // Gamma of the segment
    bars = o;  o += 2 * 8;         // raw stage full (copy bytes)
    fbars = o; o += 2 * 8;         // operand buffer full (builder arrivals)
    mbars = o; o += 2 * 8;         // operand buffer free (MMA completion)
    nbars = o; o += 2 * 8;         // key-norm scales of a chunk written (builder arrivals)
    slot = o;  o += 16;            // TMEM base address
    flag = o;  o += 16;            // a wait timed out
    issued = o; o += 16;           // chunks whose MMAs were issued
    total = align_up(o, 128);
  }
};

// A chunk's operand tile, MN-major without swizzle: the 16-byte row of 8
// consecutive MN elements (key columns j = 8 grp .. 8 grp + 7, or value rows)
// of token t sits at grp * 512 + t * 16. Along K (tokens), core matrices of
// 8 tokens x 16 bytes are 128 bytes apart (leading byte offset); along MN,
// groups of 8 elements are 512 bytes apart (stride byte offset). One K = 16
// step of the MMA starts 256 bytes further per step.
constexpr uint32_t kMnGroupBytes = kTcC * 16;
__device__ __forceinline__ uint32_t mn_off(int grp, int t) { return (uint32_t)(grp * kMnGroupBytes + t * 16); }

// tcgen05 shared-memory matrix descriptor: start address, leading byte offset
// 128 (next 8 tokens along K), stride byte offset 512 (next 8 MN elements), the
// sm_100-family version field (bits 46-47 = 1), no swizzle.
__device__ __forceinline__ uint64_t smem_desc(const void* p) {
  const uint64_t a = (smem_u32(p) & 0x3FFFFu) >> 4;
  return a | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(kMnGroupBytes >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both MN-major
// (bits 15 and 16), N = n (multiple of 16), M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}

// Item it of a tile build -> (token t, 8-element group grp) such that the 8
// items of a shared-memory access phase (consecutive it) have distinct t mod 8
// (the tile stores, 16 bytes each at t * 16) and distinct grp mod 8 (the staged
// reads at t * row_bytes + grp * 16, row_bytes a multiple of 128): both
// conflict-free. Needs the group count G to be a multiple of 8; otherwise
// group-major order.
__device__ __forceinline__ void tile_item(int it, int G, int& t, int& grp) {
  if (G % 8 == 0) {
    const int i = it & 7, j = it >> 3;
    t = 8 * (j & 3) + i;
    grp = 8 * (j >> 5) + ((i + (j >> 2)) & 7);
  } else {
    t = it % kTcC;
    grp = it / kTcC;
  }
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(r[q]);
}

// Two fp32 values as packed bf16 pairs (x0 in the low half): each rounded to
// nearest even, and the rounding remainders, rounded again. One paired
// conversion per pair instead of one per value.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Thread 0: copy segment-local tokens [t0, t0 + tc) of k, v, beta into a raw stage.
__device__ __forceinline__ void tc_stage(unsigned char* st, const TcSmem& L, uint64_t* bar, const FwdArgs& a,
                                         size_t tok0, int tc) {
  const int DV = a.d_v;
  const uint32_t bk = (uint32_t)tc * kTcDK * 2, bv = (uint32_t)tc * DV * 2;
  mbar_arrive_expect_tx(bar, bk + 2 * bv);
  bulk_g2s(st + L.raw_k, static_cast<const char*>(a.k) + tok0 * kTcDK * 2, bk, bar);
  bulk_g2s(st + L.raw_v, static_cast<const char*>(a.v) + tok0 * DV * 2, bv, bar);
  bulk_g2s(st + L.raw_b, static_cast<const char*>(a.beta) + tok0 * DV * 2, bv, bar);
}

// All threads: the M-side tiles of one chunk (tokens >= tc are zero): K^T, and
// k^2 split into bf16 hi + lo. One item = 8 key columns of one token = one
// 16-byte row of each tile, read from the staged k as one 16-byte piece.
__device__ __forceinline__ void build_key_tiles(const unsigned char* raw, unsigned char* ob, const TcSmem& L,
                                                int tc, int btid) {
  constexpr int G = kTcDK / 8;
  for (int it = btid; it < G * kTcC; it += kTcBuilders) {
    int t, grp;
    tile_item(it, G, t, grp);
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (t < tc) w = *reinterpret_cast<const uint4*>(raw + L.raw_k + (size_t)t * kTcDK * 2 + grp * 16);
    const uint32_t kw[4] = {w.x, w.y, w.z, w.w};
    uint32_t kh[4], kl[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float k0 = __uint_as_float(kw[q] << 16), k1 = __uint_as_float(kw[q] & 0xffff0000u);
      split_bf16x2(k0 * k0, k1 * k1, kh[q], kl[q]);  // k^2 is exact in fp32 and in hi + lo
    }
    const uint32_t off = mn_off(grp, t);
    *reinterpret_cast<uint4*>(ob + L.kt + off) = w;
    *reinterpret_cast<uint4*>(ob + L.k2h + off) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
    *reinterpret_cast<uint4*>(ob + L.k2l + off) = make_uint4(kl[0], kl[1], kl[2], kl[3]);
  }
}

// All threads: the N-side tiles of one chunk: X = W s beta v (or W s v* in the
// v* mode) and Y = W s^2 beta, each split into bf16 hi + lo, where s_t is the
// token's key-norm scale (1 without the q/k norm: normalising k_t scales its
// row of K by s_t and of K^2 by s_t^2, which moves onto the token side and
// keeps K exact in bf16); beta through the fused prologue when it is on.
// Tokens >= tc are zero.
__device__ __forceinline__ void build_row_tiles(const unsigned char* raw, unsigned char* ob, const TcSmem& L,
                                                float w_lane, const float* ns, int tc, int DV, const Prologue& pro,
                                                float bsc, int btid) {
  const int G = DV / 8;
  // the same trip count on every lane: W_t comes from lane t of the warp by a shuffle
  for (int base = 0; base < G * kTcC; base += kTcBuilders) {
    const int it = base + btid;
    int t, grp;
    tile_item(it, G, t, grp);
    const float wt = __shfl_sync(0xffffffffu, w_lane, t & (kTcC - 1));
    if (it >= G * kTcC) continue;
    uint32_t xh[4] = {0u, 0u, 0u, 0u}, xl[4] = {0u, 0u, 0u, 0u}, yh[4] = {0u, 0u, 0u, 0u}, yl[4] = {0u, 0u, 0u, 0u};
    if (t < tc) {
      const size_t ro = (size_t)t * DV * 2 + grp * 16;
      const uint4 vw = *reinterpret_cast<const uint4*>(raw + L.raw_v + ro);
      const uint4 bw = *reinterpret_cast<const uint4*>(raw + L.raw_b + ro);
      const uint32_t vv[4] = {vw.x, vw.y, vw.z, vw.w}, bb[4] = {bw.x, bw.y, bw.z, bw.w};
      const float s = ns ? ns[t] : 1.f, ws = wt * s, wss = ws * s;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float b0 = __uint_as_float(bb[q] << 16), b1 = __uint_as_float(bb[q] & 0xffff0000u);
        const float v0 = __uint_as_float(vv[q] << 16), v1 = __uint_as_float(vv[q] & 0xffff0000u);
        if (pro.on) {
          b0 = bsc * sigmoid_f(b0);
          b1 = bsc * sigmoid_f(b1);
        }
        const float x0 = pro.v_star ? ws * v0 : ws * b0 * v0, x1 = pro.v_star ? ws * v1 : ws * b1 * v1;
        split_bf16x2(x0, x1, xh[q], xl[q]);
        split_bf16x2(wss * b0, wss * b1, yh[q], yl[q]);
      }
    }
    const uint32_t off = mn_off(grp, t);
    *reinterpret_cast<uint4*>(ob + L.xh + off) = make_uint4(xh[0], xh[1], xh[2], xh[3]);
    *reinterpret_cast<uint4*>(ob + L.xl + off) = make_uint4(xl[0], xl[1], xl[2], xl[3]);
    *reinterpret_cast<uint4*>(ob + L.yh + off) = make_uint4(yh[0], yh[1], yh[2], yh[3]);
    *reinterpret_cast<uint4*>(ob + L.yl + off) = make_uint4(yl[0], yl[1], yl[2], yl[3]);
  }
}

// Thread 0: the ten MMAs of one chunk (two K = 16 steps) on operand buffer ob.
__device__ __forceinline__ void issue_chunk_mmas(const unsigned char* ob, const TcSmem& L, uint32_t tmem, int DV,
                                                 bool first) {
  const uint32_t idesc = idesc_bf16(DV);
  const uint32_t dM = tmem, dI = tmem + (uint32_t)DV;
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const unsigned char* a0 = ob + ks * 256;  // tokens 16 ks .. 16 ks + 15 of every 8-element group
    const unsigned char* b0 = ob + ks * 256;
    const int acc = (first && ks == 0) ? 0 : 1;
    tc_mma(dM, smem_desc(a0 + L.kt), smem_desc(b0 + L.xh), idesc, acc);
    tc_mma(dM, smem_desc(a0 + L.kt), smem_desc(b0 + L.xl), idesc, 1);
    tc_mma(dI, smem_desc(a0 + L.k2h), smem_desc(b0 + L.yh), idesc, acc);
    tc_mma(dI, smem_desc(a0 + L.k2h), smem_desc(b0 + L.yl), idesc, 1);
    tc_mma(dI, smem_desc(a0 + L.k2l), smem_desc(b0 + L.yh), idesc, 1);
  }
}

// Summaries of segments 0 .. nslot - 1 of every head (grid: heads x nslot).
// Output as pass A: seg_state[(bh * nslot + seg)] = (dM [d_v][d_k], dIbar), seg_gamma[...] = Gamma.
__global__ void __launch_bounds__(kTcThreads)
palimpsa_fwd_summary_tc_kernel(FwdArgs a, int nslot, int seg_len, float* __restrict__ seg_state,
                               float* __restrict__ seg_gamma) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int DV = a.d_v;
  const Tile tl = tile_of(a, DV, nslot, seg_len);
  // a packed sequence needs only the summaries before its own last segment
  if (tl.bad || (a.cu_seqlens && tl.seg >= tl.last_seg)) return;
  const TcSmem L(DV);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* fbars = reinterpret_cast<uint64_t*>(smem + L.fbars);
  uint64_t* mbars = reinterpret_cast<uint64_t*>(smem + L.mbars);
  uint64_t* nbars = reinterpret_cast<uint64_t*>(smem + L.nbars);
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + L.slot);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + L.flag);
  int* issued_s = reinterpret_cast<int*>(smem + L.issued);
  float* gam = reinterpret_cast<float*>(smem + L.gam);
  const float A_h = a.A[tl.h];
  const float bsc = a.pro.b_scale ? a.pro.b_scale[tl.h] : 1.f;
  const int nch = (tl.tn + kTcC - 1) / kTcC;
  const uint32_t ncols = DV * 2 <= 64 ? 64u : DV * 2 <= 128 ? 128u : 256u;
  const size_t tok_base = tl.head_tok + tl.tb;
  const float* gd = a.d_t + tok_base;
  // builders: d_t one chunk ahead (lane t = token t); the first chunk's load is
  // issued before the set-up below, so that it lands meanwhile
  float d_next = 0.f;
  if (warp > 0 && nch > 0) {
    const int t0n = (nch - 1) * kTcC;
    if (lane < min(kTcC, tl.tn - t0n)) d_next = gd[t0n + lane];
  }

  // thread 0: raw copies in flight per stage (for a clean exit), and their phases
  bool pend[2] = {false, false};
  uint32_t ppar[2] = {0u, 0u};
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[i], 1);
      mbar_init(&fbars[i], kTcBuilders / 32);  // one arrival per builder warp
      mbar_init(&mbars[i], 1);
      mbar_init(&nbars[i], kTcBuilders / 32);
    }
    *flag = 0;
    *issued_s = 0;
    gam[0] = 1.f;
    fence_mbar_init();
    // the first two chunks' copies go out now and land during the set-up below
    // (processing chunk c is segment-local chunk nch - 1 - c: W is a suffix product)
    for (int c = 0; c < 2 && c < nch; ++c) {
      if (c == 0 && a.withhold_first_copy) continue;
      const int t0 = (nch - 1 - c) * kTcC;
      tc_stage(smem + (size_t)(c & 1) * L.raw_bytes, L, &bars[c & 1], a, tok_base + t0, min(kTcC, tl.tn - t0));
      pend[c & 1] = true;
      ppar[c & 1] = (uint32_t)(c >> 1) & 1u;
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (warp == 0) {
    // ---- control: copies into the raw ring, and the MMAs of each complete chunk
    if (lane == 0) {
      int c = 0;
      for (; c < nch && !*flag; ++c) {
        // the builders are done with raw stage c & 1 and operand buffer c & 1 is complete
        if (!mbar_wait_bounded(&fbars[c & 1], (uint32_t)(c >> 1) & 1u, a.wait_timeout_ns)) {
          *flag = 1;
          break;
        }
        pend[c & 1] = false;  // the builders waited for this stage's bytes
        if (c + 2 < nch) {
          const int t2 = (nch - 1 - (c + 2)) * kTcC;
          tc_stage(smem + (size_t)(c & 1) * L.raw_bytes, L, &bars[c & 1], a, tok_base + t2, min(kTcC, tl.tn - t2));
          pend[c & 1] = true;
          ppar[c & 1] = (uint32_t)((c + 2) >> 1) & 1u;
        }
        tc_fence_after();
        issue_chunk_mmas(smem + L.ops + (size_t)(c & 1) * L.op_bytes, L, tmem, DV, c == 0);
        tc_commit(&mbars[c & 1]);
      }
      *issued_s = c;
      // copies still in flight (a timeout upstream) land before the CTA may exit
      if (*flag) {
        if (pend[0]) mbar_wait_bounded(&bars[0], ppar[0], 1000000000ull);
        if (pend[1]) mbar_wait_bounded(&bars[1], ppar[1], 1000000000ull);
      }
    }
  } else {
    // ---- builders (warps 1-7)
    const int btid = threadIdx.x - 32;
    float carry = 1.f;  // product of the alphas of the chunks already processed (later tokens)
    for (int c = 0; c < nch; ++c) {
      const int t0 = (nch - 1 - c) * kTcC, tc = min(kTcC, tl.tn - t0);
      const float d_cur = d_next;
      if (c + 1 < nch) d_next = gd[(nch - 2 - c) * kTcC + lane];  // chunks before the last are whole
      // W_t = carry * prod_{t < u < tc} alpha_u (lane t), while the copies land
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
      const float w_lane = lane < tc ? carry * (lane + 1 < tc ? excl : 1.f) : 0.f;
      carry *= __shfl_sync(0xffffffffu, p, 0);
      bool ok = mbar_wait_bounded(&bars[c & 1], (uint32_t)(c >> 1) & 1u, a.wait_timeout_ns);
      // operand buffer c & 1 was last read by the MMAs of chunk c - 2
      if (ok && c >= 2) ok = mbar_wait_bounded(&mbars[c & 1], (uint32_t)((c - 2) >> 1) & 1u, a.wait_timeout_ns);
      // leave together (the loop holds warp shuffles); the arrivals of this chunk then
      // never come, and the control warp's wait for them times out too
      if (__any_sync(0xffffffffu, !ok || *flag)) {
        *flag = 1;
        break;
      }
      const unsigned char* raw = smem + (size_t)(c & 1) * L.raw_bytes;
      unsigned char* ob = smem + L.ops + (size_t)(c & 1) * L.op_bytes;
      const float* nsc = nullptr;
      if (a.pro.qk_norm) {
        // key-norm scales of the chunk (builder warp b takes tokens b - 1, b + 6, ...; each lane
        // 4 of the 128 columns), two chunks' worth so that a slow warp still reads its own
        float* ns = reinterpret_cast<float*>(smem + L.ns) + (c & 1) * kTcC;
        for (int t = warp - 1; t < kTcC; t += kTcBuilders / 32) {
          float sc = 1.f;
          if (t < tc) {
            const uint2 w2 = *reinterpret_cast<const uint2*>(raw + L.raw_k + ((size_t)t * kTcDK + 4 * lane) * 2);
            const float k0 = bf16_lo(w2.x), k1 = bf16_hi(w2.x), k2 = bf16_lo(w2.y), k3 = bf16_hi(w2.y);
            float ss = fmaf(k0, k0, fmaf(k1, k1, fmaf(k2, k2, k3 * k3)));
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            sc = rsqrtf(fmaxf(ss, kNormFloorSq));
          }
          if (lane == 0) ns[t] = sc;
        }
        // every builder's scales are in place (a bounded wait, as every wait here)
        __syncwarp();
        if (lane == 0)
          asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&nbars[c & 1]))
                       : "memory");
        if (__any_sync(0xffffffffu, !mbar_wait_bounded(&nbars[c & 1], (uint32_t)(c >> 1) & 1u, a.wait_timeout_ns))) {
          *flag = 1;
          break;
        }
        nsc = ns;
      }
      build_key_tiles(raw, ob, L, tc, btid);
      build_row_tiles(raw, ob, L, w_lane, nsc, tc, DV, a.pro, bsc, btid);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic-proxy writes -> tensor cores
      __syncwarp();  // the warp's tiles (and its reads of the raw stage) are done: one arrival for the warp
      if (lane == 0)
        asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&fbars[c & 1]))
                     : "memory");
    }
    if (warp == 1 && lane == 0) gam[0] = carry;
  }
  __syncthreads();
  const bool failed = *flag != 0;
  const int issued = *issued_s;

  // MMAs of chunks max(0, issued - 2) .. issued - 1 may still run: wait (bounded)
  // before reading or freeing the accumulators.
  const unsigned long long drain_ns = failed ? 1000000000ull : a.wait_timeout_ns;
  bool mma_ok = true;
  for (int k = issued - 2 > 0 ? issued - 2 : 0; k < issued; ++k)
    if (!mbar_wait_bounded(&mbars[k & 1], (uint32_t)(k >> 1) & 1u, drain_ns)) mma_ok = false;
  if (threadIdx.x == 0 && (failed || !mma_ok)) latch_status(a.status, kStatusTimeout);
  __syncthreads();
  tc_fence_after();
  if (!failed && __syncthreads_and(mma_ok)) {
    // warps 0-3 read dM^T, warps 4-7 dIbar^T; TMEM lane = key column j
    const int part = warp >> 2;
    const int j = 32 * (warp & 3) + lane;
    float* out = seg_state + ((size_t)tl.bh * nslot + tl.seg) * 2 * DV * kTcDK + (size_t)part * DV * kTcDK;
    for (int cb = 0; cb < DV; cb += 32) {
      float v[32];
      if (nch > 0) {
        tc_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(part * DV + cb), v);
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < 32; ++q) out[(size_t)(cb + q) * kTcDK + j] = v[q];
    }
    if (threadIdx.x == 0) seg_gamma[(size_t)tl.bh * nslot + tl.seg] = gam[0];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
}

}  // namespace

bool summary_tc_eligible(const FwdArgs& a) {
  return a.bf16 && a.d_k == kTcDK && a.d_v % 32 == 0 && a.d_v <= 128;
}

cudaError_t launch_summary_tc(const FwdArgs& a, int nslot, int seg_len, float* seg_state, float* seg_gamma,
                              cudaStream_t s) {
  const TcSmem L(a.d_v);
  cudaError_t e = cudaFuncSetAttribute(palimpsa_fwd_summary_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L.total);
  if (e != cudaSuccess) return e;
  const long ctas = (long)a.B * a.H * nslot;
  palimpsa_fwd_summary_tc_kernel<<<(unsigned)ctas, kTcThreads, L.total, s>>>(a, nslot, seg_len, seg_state,
                                                                              seg_gamma);
  return cudaGetLastError();
}

}  // namespace palimpsa
