// gp_attn_mma.cu -- paged GQA decode attention for bf16 pages, head_dim 128,
// with GrowPage's summary upkeep and summary scoring fused in.
//
// What it computes is the same as the fp32 kernel (gp_attn.cu), following
// "GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning Serving"
// (evolve.pub review, Summary: two exponentially smoothed query summaries,
// beta 0.9 / 0.999, kept pre-RoPE; Top-p working sets of both at each
// PagedAttention capacity boundary):
//   * the step's key, rotated to its position in fp64 and rounded once to
//     bf16 (the staged token), and its value;
//   * the fp32 fold of the mean of the G query heads into both summaries;
//   * out = softmax(RoPE(q)·K^T/sqrt(d))·V over the resident tokens plus the
//     staged token, for the G query heads of the kv head;
//   * at a boundary, u = RoPE(s)·k/sqrt(d) of both updated summaries for every
//     resident key, written for the working-set and compaction kernels.
//
// How.  The G query heads and, at boundary steps, the two summaries form the
// rows of one 16-row operand; each 16-token block of keys is the other
// operand, so Q·K^T and P·V run as warp-level bf16 tensor-core products
// (mma.sync m16n8k16, fp32 accumulation).  The contraction is a real dense
// one (G heads x d per key); the tensor pipe is used to cut the instruction
// count per byte so that the kernel stays bound by HBM, not by issue.
// Accuracy: bf16 operands hold fp32 values as exact-sum splits -- a query as
// hi + lo (rows g and g+8, summed by the same thread), a summary as
// hi + mid + lo, softmax weights as hi + lo -- so the scores and the output
// carry close to fp32 precision although the pages are bf16.
//
// Memory.  Each warp owns a ring of S shared-memory stages; its lane 0 fills
// a stage with four 2-D tensor-map copies (TMA, 128-byte swizzle: K and V,
// two 64-column halves each) that complete on the stage's mbarrier.  The
// swizzle makes the ldmatrix reads of both operands bank-conflict free.
// Work is split over a persistent grid as in the fp32 kernel (equal ranges
// of blocks per warp; a cut (request, head) is merged by the warp that
// finishes its last piece).  Every wait is bounded and on the warp's own
// copies.
#include <cuda.h>

#include "gp_attn_common.cuh"

namespace gp {

constexpr int kMmaD = 128;
constexpr int kMmaStageB = 8192;           // 16 tokens x (K 4 KiB + V 4 KiB)
#ifndef GP_MMA_WARPS
#define GP_MMA_WARPS 4
#endif
#ifndef GP_MMA_STAGES
#define GP_MMA_STAGES 3
#endif
constexpr int kMmaWarps = GP_MMA_WARPS;
constexpr int kMmaStages = GP_MMA_STAGES;
constexpr int kObFloats = 4 * (kMmaD + 2);  // per-warp merge buffer: [G<=4][D] + m + l
// prep and combine run one warp per CTA: their CTAs are launched early (see
// griddepcontrol) and must fit beside two resident attention CTAs.
constexpr int kSmallWarps = 1;

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Round to nearest-even bf16 (bit pattern) and the value it stands for.
__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_val(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ uint32_t pack2(uint32_t lo_col, uint32_t hi_col) {
  return lo_col | (hi_col << 16);
}

// x = hi + lo exactly up to the rounding of lo (x - hi is exact in fp32).
__device__ __forceinline__ void split2(float x, uint32_t& hi, uint32_t& lo) {
  hi = bf16_bits(x);
  lo = bf16_bits(x - bf16_val(hi));
}
// x = hi + mid + lo, each residual exact in fp32.
__device__ __forceinline__ void split3(float x, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  hi = bf16_bits(x);
  const float r1 = x - bf16_val(hi);
  mid = bf16_bits(r1);
  lo = bf16_bits(r1 - bf16_val(mid));
}

// Byte offset, inside a 2 KiB TMA box written with the 128-byte swizzle, of
// 16-byte chunk `lc` (0..7) of row `r`: the chunk index is XORed with r mod 8.
__device__ __forceinline__ uint32_t swz(int r, int lc) {
  return (uint32_t)(r * 128 + ((lc ^ (r & 7)) << 4));
}

__device__ __forceinline__ void issue_block_tma(const PoolDev& p, const CUtensorMap* map, int layer,
                                                const Cursor& c, int page, uint8_t* stage,
                                                uint64_t* bar) {
  const int t0 = c.blk * kBlockTok;
  // row of the pool viewed as [num_pages * L * Hk * 2 * P][d]
  const int row = (((page * p.L + layer) * p.Hk + c.h) * 2) * p.P + (t0 % p.P);
  mbar_expect_tx(bar, kMmaStageB);
  tma_load_2d(stage, map, 0, row, bar);
  tma_load_2d(stage + 2048, map, 64, row, bar);
  tma_load_2d(stage + 4096, map, 0, row + p.P, bar);
  tma_load_2d(stage + 6144, map, 64, row + p.P, bar);
}

// Summary fold (fp32, exact order): s' = fl(fl(b*s) + fl((1-b)*qbar)), or
// qbar on the request's first step; qbar = (sum of the G heads in order)/G.
template <int G>
__device__ __forceinline__ float fold_summary(const __nv_bfloat16* qrow0, int dim, const float* srowp,
                                              int X, float beta, int first) {
  float qb = __bfloat162float(qrow0[dim]);
#pragma unroll
  for (int g = 1; g < G; ++g) qb = __fadd_rn(qb, __bfloat162float(qrow0[g * kMmaD + dim]));
  const float qm = __fdiv_rn(qb, (float)G);
  if (first) return qm;
  const float a = __fsub_rn(1.0f, beta);
  return __fadd_rn(__fmul_rn(beta, srowp[X * kMmaD + dim]), __fmul_rn(a, qm));
}

// ---------------------------------------------------------------- prep ---
//
// One warp per (request i of the step, kv head h), before the attention
// launch of the layer.  Everything here depends on the step's inputs only,
// not on the resident keys, so it is kept off the streaming warps:
//   1. the tensor-core operand rows of the attention kernel, laid out as the
//      registers of lane (g = lane / 4, t = lane % 4) will hold them: rows
//      g < G = query head g rotated to the current position, scaled by
//      log2(e)/sqrt(d), bf16 hi (row g) + lo (row g+8); at a boundary, rows
//      4/5 = short/long summary (after this step's fold) rotated and scaled
//      by 1/sqrt(d), hi (rows 4/5) + mid (rows 12/13), lo in rows 6/7;
//   2. the staged token: key rotated in fp64 and rounded once to bf16, value
//      copied; and each query head's score against it;
//   3. the fold of the step's query mean into both summaries.
// Operands are written to scratch ([i][h][kk][lane] as 16-byte words).
// bf16 pair at element `di` (even) of a row, as two floats.
__device__ __forceinline__ float2 ld_bf2(const __nv_bfloat16* row, int di) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(row + di);
  return make_float2(bf16lo(w), bf16hi(w));
}

template <int G>
__global__ void __launch_bounds__(kSmallWarps * 32)
prep_kernel(PoolDev p, int layer, const __nv_bfloat16* __restrict__ q,
            const __nv_bfloat16* __restrict__ knew, const __nv_bfloat16* __restrict__ vnew) {
  using Gm = Geo<__nv_bfloat16, kMmaD>;
  constexpr int D = kMmaD, NE = Gm::NE, H2 = NE / 2;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.plan_misc[0];
  const int gw = blockIdx.x * kSmallWarps + warp;
  if (gw >= n * p.Hk) return;
  const int i = gw / p.Hk, h = gw % p.Hk;
  const int slot = p.plan_slot[i], flags = p.plan_flags[i];
  const int pos = p.req[slot].pos;
  const int first = flags & kPlanFirst;
  const bool score = (flags & kPlanScore) != 0;
  const size_t srow = (((size_t)slot * p.L + layer) * p.Hk + h) * 2;
  float* srowp = p.summary + srow * D;
  const int g = lane >> 2, t = lane & 3;         // operand-row layout
  const int sigma = lane & 7, grp = lane >> 3;   // 8 lanes per row layout
  const bool head_row = g < G;
  const bool sum_row = score && g >= 4;
  const int X = g & 1;
  // ---- loads of what was final before this step began (plan, positions,
  // rotary tables, this layer's summaries), while the previous kernel in the
  // stream may still run.  fd(j): operand dim 16*(j/4) + 2t + 8*((j/2)%2) + j%2.
  float rc[16], rs[16];              // fp32 rotation at the 16 operand dims
  float so[16], so2[16];             // old summary X at the operand dims, +64
  double c64[H2], s64[H2];           // fp64 rotation at this lane's row dims
  float c32r[H2], s32r[H2];          // fp32 rotation at this lane's row dims
  float fs[4], fl[4];                // old summaries at dims 4*lane + e
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int di = 16 * (j / 4) + 2 * t + 8 * ((j / 2) % 2) + (j % 2);
    rc[j] = p.rope ? p.cos32[(size_t)pos * (D / 2) + di] : 1.f;
    rs[j] = p.rope ? p.sin32[(size_t)pos * (D / 2) + di] : 0.f;
    so[j] = sum_row ? srowp[X * D + di] : 0.f;
    so2[j] = sum_row ? srowp[X * D + di + 64] : 0.f;
  }
#pragma unroll
  for (int e = 0; e < H2; ++e) {
    const int di = dim_of<Gm>(e, sigma);
    c64[e] = p.rope ? p.cos64[(size_t)pos * (D / 2) + di] : 1.0;
    s64[e] = p.rope ? p.sin64[(size_t)pos * (D / 2) + di] : 0.0;
    c32r[e] = p.rope ? p.cos32[(size_t)pos * (D / 2) + di] : 1.f;
    s32r[e] = p.rope ? p.sin32[(size_t)pos * (D / 2) + di] : 0.f;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    fs[e] = srowp[lane * 4 + e];
    fl[e] = srowp[D + lane * 4 + e];
  }
  // ---- the step's inputs may come from the previous kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const __nv_bfloat16* q0 = q + ((size_t)i * p.Hq + h * G) * D;
  const float bX = X ? p.beta_l : p.beta_s, aX = __fsub_rn(1.0f, bX);

  // ---- 1. operand rows
  {
    const float qscale = 1.4426950408889634f / sqrtf((float)D);  // log2(e)/sqrt(d)
    const float sscale = 1.0f / sqrtf((float)D);
    float a[16], b[16];
    if (head_row) {
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const int di = 16 * (j / 4) + 2 * t + 8 * ((j / 2) % 2);
        const float2 lo = ld_bf2(q0 + g * D, di), hi = ld_bf2(q0 + g * D, di + 64);
        a[j] = lo.x; a[j + 1] = lo.y; b[j] = hi.x; b[j + 1] = hi.y;
      }
    } else if (sum_row) {
      float qa[16], qb[16];   // head-order sums of the G heads at the operand dims
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const int di = 16 * (j / 4) + 2 * t + 8 * ((j / 2) % 2);
          const float2 lo = ld_bf2(q0 + gg * D, di), hi = ld_bf2(q0 + gg * D, di + 64);
          if (gg == 0) {
            qa[j] = lo.x; qa[j + 1] = lo.y; qb[j] = hi.x; qb[j + 1] = hi.y;
          } else {
            qa[j] = __fadd_rn(qa[j], lo.x); qa[j + 1] = __fadd_rn(qa[j + 1], lo.y);
            qb[j] = __fadd_rn(qb[j], hi.x); qb[j + 1] = __fadd_rn(qb[j + 1], hi.y);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {   // the fold, as in step 3
        const float ma = __fdiv_rn(qa[j], (float)G), mb = __fdiv_rn(qb[j], (float)G);
        a[j] = first ? ma : __fadd_rn(__fmul_rn(bX, so[j]), __fmul_rn(aX, ma));
        b[j] = first ? mb : __fadd_rn(__fmul_rn(bX, so2[j]), __fmul_rn(aX, mb));
      }
    }
    uint32_t afr[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) afr[kk][0] = afr[kk][1] = afr[kk][2] = afr[kk][3] = 0u;
    if (head_row || sum_row) {
      const float sc = head_row ? qscale : sscale;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (p.rope) {
          const float xa = a[j] * rc[j] - b[j] * rs[j];
          const float yb = b[j] * rc[j] + a[j] * rs[j];
          a[j] = xa;
          b[j] = yb;
        }
        a[j] *= sc;
        b[j] *= sc;
      }
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const int kk = j / 4, half = (j / 2) % 2;
        // registers: [0] row g, cols 2t..; [1] row g+8; [2] row g, cols 2t+8..; [3] row g+8
        uint32_t xh[2], xl[2], yh[2], yl[2];
        if (head_row) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            split2(a[j + u], xh[u], xl[u]);
            split2(b[j + u], yh[u], yl[u]);
          }
        } else {
          uint32_t xm[2], ym[2], xlo[2], ylo[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            split3(a[j + u], xh[u], xm[u], xlo[u]);
            split3(b[j + u], yh[u], ym[u], ylo[u]);
          }
          if (g >= 6) {  // rows 6/7 carry the lo parts; rows 14/15 stay zero
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              xh[u] = xlo[u]; yh[u] = ylo[u]; xl[u] = 0u; yl[u] = 0u;
            }
          } else {  // rows 4/5 hi, rows 12/13 mid
#pragma unroll
            for (int u = 0; u < 2; ++u) { xl[u] = xm[u]; yl[u] = ym[u]; }
          }
        }
        afr[kk][2 * half + 0] = pack2(xh[0], xh[1]);
        afr[kk][2 * half + 1] = pack2(xl[0], xl[1]);
        afr[kk + 4][2 * half + 0] = pack2(yh[0], yh[1]);
        afr[kk + 4][2 * half + 1] = pack2(yl[0], yl[1]);
      }
    }
    uint4* fr = p.frag + (size_t)gw * 8 * 32;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      fr[kk * 32 + lane] = make_uint4(afr[kk][0], afr[kk][1], afr[kk][2], afr[kk][3]);
  }

  // ---- 2. staged token and the query heads' scores against it
  {
    float vraw[NE], kst[NE];
    load_row<__nv_bfloat16, Gm>(reinterpret_cast<const uint8_t*>(knew + ((size_t)i * p.Hk + h) * D),
                                sigma, kst);
    load_row<__nv_bfloat16, Gm>(reinterpret_cast<const uint8_t*>(vnew + ((size_t)i * p.Hk + h) * D),
                                sigma, vraw);
    float qr[NE];
    if (grp < G)
      load_row<__nv_bfloat16, Gm>(
          reinterpret_cast<const uint8_t*>(q0 + (size_t)grp * D), sigma, qr);
    if (p.rope) {
#pragma unroll
      for (int e = 0; e < H2; ++e) {
        const double x = (double)kst[e], y = (double)kst[e + H2];
        const double ra = __dsub_rn(__dmul_rn(x, c64[e]), __dmul_rn(y, s64[e]));
        const double rb = __dadd_rn(__dmul_rn(y, c64[e]), __dmul_rn(x, s64[e]));
        kst[e] = __uint_as_float((uint32_t)f64_to_bf16_rne(ra) << 16);
        kst[e + H2] = __uint_as_float((uint32_t)f64_to_bf16_rne(rb) << 16);
      }
    }
    if (grp == 0) {
      __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(p.staging) + srow * D;
      store_row<__nv_bfloat16, Gm>(st, sigma, kst);  // exact: already on the bf16 grid
      store_row<__nv_bfloat16, Gm>(st + D, sigma, vraw);
    }
    const float qscale = 1.4426950408889634f / sqrtf((float)D);
    float sa = 0.f;
    if (grp < G) {  // one query head per 8-lane group
      if (p.rope) {
#pragma unroll
        for (int e = 0; e < H2; ++e) {
          const float x = qr[e], y = qr[e + H2];
          qr[e] = x * c32r[e] - y * s32r[e];
          qr[e + H2] = y * c32r[e] + x * s32r[e];
        }
      }
#pragma unroll
      for (int e = 0; e < NE; ++e) sa = fmaf(qr[e] * qscale, kst[e], sa);
    }
    sa += __shfl_xor_sync(0xffffffffu, sa, 1);
    sa += __shfl_xor_sync(0xffffffffu, sa, 2);
    sa += __shfl_xor_sync(0xffffffffu, sa, 4);
    if (grp < G && sigma == 0) p.sstage[gw * 4 + grp] = sa;
  }

  // ---- 3. summaries: 4 dims per lane (old values were read before the wait)
  {
    const float aS = __fsub_rn(1.0f, p.beta_s), aL = __fsub_rn(1.0f, p.beta_l);
    float qs[4];
    {
      const uint2 w0 = *reinterpret_cast<const uint2*>(q0 + lane * 4);
      qs[0] = bf16lo(w0.x); qs[1] = bf16hi(w0.x); qs[2] = bf16lo(w0.y); qs[3] = bf16hi(w0.y);
    }
#pragma unroll
    for (int gg = 1; gg < G; ++gg) {
      const uint2 w1 = *reinterpret_cast<const uint2*>(q0 + gg * D + lane * 4);
      qs[0] = __fadd_rn(qs[0], bf16lo(w1.x)); qs[1] = __fadd_rn(qs[1], bf16hi(w1.x));
      qs[2] = __fadd_rn(qs[2], bf16lo(w1.y)); qs[3] = __fadd_rn(qs[3], bf16hi(w1.y));
    }
    float4 ns, nl;
    float* nsp = &ns.x;
    float* nlp = &nl.x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float qm = __fdiv_rn(qs[e], (float)G);
      nsp[e] = first ? qm : __fadd_rn(__fmul_rn(p.beta_s, fs[e]), __fmul_rn(aS, qm));
      nlp[e] = first ? qm : __fadd_rn(__fmul_rn(p.beta_l, fl[e]), __fmul_rn(aL, qm));
    }
    *reinterpret_cast<float4*>(srowp + lane * 4) = ns;
    *reinterpret_cast<float4*>(srowp + D + lane * 4) = nl;
  }
}

// Output of one (request, kv head) from the merged attention state in the
// warp's buffer ob ([G][D] unnormalised output, then m[G] in the log2
// domain, l[G]): the staged token (value from the staging rows, score from
// the prep kernel) is merged in and the rows are normalised and stored.
template <int G>
__device__ __forceinline__ void finish_mma(const PoolDev& p, int layer, int i, int h, int slot,
                                           __nv_bfloat16* __restrict__ out, const float* ob,
                                           int lane) {
  using Gm = Geo<__nv_bfloat16, kMmaD>;
  constexpr int D = kMmaD, NE = Gm::NE;
  const int sigma = lane & 7, g = lane >> 3;  // one query head per 8-lane group
  if (g >= G) return;
  const size_t srow = (((size_t)slot * p.L + layer) * p.Hk + h) * 2;
  float vraw[NE];
  load_row<__nv_bfloat16, Gm>(p.staging + (srow + 1) * D * sizeof(__nv_bfloat16), sigma, vraw);
  const float a = p.sstage[(i * p.Hk + h) * 4 + g];
  const float mg = ob[G * D + g], lg = ob[G * D + G + g];
  const float mn = fmaxf(mg, a);
  const float al = (mg == -INFINITY) ? 0.f : exp2f(mg - mn);
  const float be = exp2f(a - mn);
  const float inv = 1.0f / (lg * al + be);
  uint8_t* orow = reinterpret_cast<uint8_t*>(out + ((size_t)i * p.Hq + h * G + g) * D);
#pragma unroll
  for (int c = 0; c < Gm::VEC; ++c) {
    uint32_t wv[4];
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {
      const int e0 = c * 8 + 2 * k2;
      const float r0 = (ob[g * D + dim_of<Gm>(e0, sigma)] * al + be * vraw[e0]) * inv;
      const float r1 = (ob[g * D + dim_of<Gm>(e0 + 1, sigma)] * al + be * vraw[e0 + 1]) * inv;
      const __nv_bfloat162 pr = __floats2bfloat162_rn(r0, r1);
      wv[k2] = *reinterpret_cast<const uint32_t*>(&pr);
    }
    *reinterpret_cast<uint4*>(orow + (c * 8 + sigma) * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
}

template <int G, int S>
__global__ void __launch_bounds__(kMmaWarps * 32)
attn_mma_kernel(const __grid_constant__ CUtensorMap kvmap, PoolDev p, int layer,
                __nv_bfloat16* __restrict__ out) {
  static_assert(G == 1 || G == 2 || G == 4, "G");
  constexpr int D = kMmaD;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint8_t* ring = smem + (size_t)warp * S * kMmaStageB;
  float* ob = reinterpret_cast<float*>(smem + (size_t)kMmaWarps * S * kMmaStageB) + warp * kObFloats;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kMmaWarps * S * kMmaStageB +
                                               (size_t)kMmaWarps * kObFloats * 4) + warp * S;

  const int n = p.plan_misc[0];
  const int64_t Tb = (int64_t)p.plan_misc[2] * p.Hk;
  const int64_t W = (int64_t)gridDim.x * kMmaWarps;
  const int64_t Weff = W < Tb ? W : Tb;
  const int64_t w = (int64_t)blockIdx.x * kMmaWarps + warp;
  // Programmatic dependent launch: the next kernel in the stream may start
  // its own prologue now.  Everything before griddepcontrol.wait below reads
  // only what was final before this step's first attention launch (plan,
  // block tables, K/V pages).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (n <= 0 || w >= Weff) return;  // warp-uniform: warps never synchronise
  const int64_t start = (w * Tb) / Weff, end = ((w + 1) * Tb) / Weff;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  Cursor pc;
  cursor_start(p, w, pc);
  PageWin win;
  const int first_seg = pc.i * p.Hk + pc.h;
  {
    int64_t b = start;
    for (int s = 0; s < S && b < end; ++s, ++b) {
      const int page = page_of(p, win, pc, lane);
      if (lane == 0) issue_block_tma(p, &kvmap, layer, pc, page, ring + s * kMmaStageB, &bars[s]);
      if (b + 1 < end) cursor_next(p, pc);
    }
  }
  int64_t issued = start + S < end ? start + S : end;
  // The operand rows and staged tokens (prep kernel), the split-K scratch
  // and the outputs belong to earlier kernels: wait for them to finish.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // per-lane ldmatrix row offsets (within a stage): K (non-transposed) and V
  const int mi = lane >> 3, ri = lane & 7;
  const int k_tok = 8 * (mi >> 1) + ri, k_half = mi & 1;   // K: token, chunk parity
  const int v_tok = 8 * (mi & 1) + ri, v_nt = mi >> 1;      // V: token, n-tile parity
  const uint32_t ring_u32 = smem_u32(ring);

  bool failed = false;
  Cursor cc;
  cursor_start(p, w, cc);
  int64_t j = start;
  while (j < end && !failed) {
    const int i = cc.i, h = cc.h, slot = cc.slot, nb = cc.nb;
    const int64_t len = ((int64_t)(nb - cc.blk) < end - j) ? (int64_t)(nb - cc.blk) : end - j;
    const bool full = (cc.blk == 0) && (len == nb);
    const int R = p.plan_R[i];
    const bool score = (p.plan_flags[i] & kPlanScore) != 0;

    // ---- A operand rows, prepared by prep_kernel (see there)
    uint32_t afr[8][4];
    {
      const uint4* fr = p.frag + (size_t)(i * p.Hk + h) * 8 * 32;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint4 v = fr[kk * 32 + lane];
        afr[kk][0] = v.x; afr[kk][1] = v.y; afr[kk][2] = v.z; afr[kk][3] = v.w;
      }
    }
    const bool head_row = g < G;
    float* lgS = p.logits + ((((size_t)slot * p.L + layer) * p.Hk + h) * 2) * p.logit_width;
    float* lgX = lgS + (g & 1) * p.logit_width;

    float m = -INFINITY, l = 0.f;
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    for (int64_t k = 0; k < len; ++k, ++j) {
      const int64_t jl = j - start;
      const int s = (int)(jl % S);
      const bool ok = __all_sync(0xffffffffu,
                                 mbar_wait_bounded(&bars[s], (uint32_t)((jl / S) & 1), kWaitLimitNs));
      if (!ok) {
        if (lane == 0) set_status(p, GP_ST_TIMEOUT, slot);
        failed = true;
        break;
      }
      const uint32_t sK = ring_u32 + s * kMmaStageB, sV = sK + 4096;
      // ---- scores: S[16 rows][16 tokens] = A · K^T
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int ch = 2 * kk + k_half;   // 16-byte chunk of the key row
        uint32_t b[4];
        ldsm_x4(b, sK + (ch >> 3) * 2048 + swz(k_tok, ch & 7));
        mma_bf16(c0, afr[kk], b[0], b[1]);
        mma_bf16(c1, afr[kk], b[2], b[3]);
      }
      // this thread's tokens of the block: 2t, 2t+1, 8+2t, 9+2t
      float sv[4] = {c0[0] + c0[2], c0[1] + c0[3], c1[0] + c1[2], c1[1] + c1[3]};
      const int t0 = (cc.blk + (int)k) * kBlockTok;
      const int nvalid = R - t0;
      const int tok[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
      // summary scores: rows 4/5 (+ rows 12/13 in the same thread) plus the
      // lo rows 6/7 held 8 lanes up
      {
        float other[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) other[u] = __shfl_xor_sync(0xffffffffu, sv[u], 8);
        if (score && (g == 4 || g == 5)) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (tok[u] < nvalid) lgX[t0 + tok[u]] = sv[u] + other[u];
        }
      }
      // ---- online softmax (log2 domain) for head row g
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (!head_row || tok[u] >= nvalid) sv[u] = -INFINITY;
        mx = fmaxf(mx, sv[u]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      // the running max moves only when a score exceeds it by more than 2^8:
      // weights stay <= 256, and the final normalisation uses the same m
      if (mx > m + 8.0f) {
        const float al = exp2f(m - mx);   // 0 when m == -inf
        l *= al;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          o[nt][0] *= al; o[nt][1] *= al; o[nt][2] *= al; o[nt][3] *= al;
        }
        m = mx;
      }
      float pv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        pv[u] = (sv[u] == -INFINITY) ? 0.f : exp2f(sv[u] - m);
        l += pv[u];
      }
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) split2(pv[u], ph[u], pl[u]);
      const uint32_t ap[4] = {pack2(ph[0], ph[1]), pack2(pl[0], pl[1]), pack2(ph[2], ph[3]),
                              pack2(pl[2], pl[3])};
      // ---- O += P · V
#pragma unroll
      for (int q2 = 0; q2 < 8; ++q2) {
        const int ch = 2 * q2 + v_nt;     // 16-byte chunk = 8 output dims
        uint32_t b[4];
        ldsm_x4_t(b, sV + (ch >> 3) * 2048 + swz(v_tok, ch & 7));
        mma_bf16(o[2 * q2], ap, b[0], b[1]);
        mma_bf16(o[2 * q2 + 1], ap, b[2], b[3]);
      }
      // refill this stage with the block S ahead
      __syncwarp();
      if (issued < end) {
        const int page = page_of(p, win, pc, lane);
        if (lane == 0) {
          fence_proxy_async_smem();
          issue_block_tma(p, &kvmap, layer, pc, page, ring + s * kMmaStageB, &bars[s]);
        }
        if (issued + 1 < end) cursor_next(p, pc);
        ++issued;
      }
    }
    if (failed) break;

    // ---- piece totals into the warp buffer: ob[g][dim], m[g], l[g]
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (head_row) {
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        ob[g * D + 8 * nt + 2 * t] = o[nt][0] + o[nt][2];
        ob[g * D + 8 * nt + 2 * t + 1] = o[nt][1] + o[nt][3];
      }
      if (t == 0) {
        ob[G * D + g] = m;
        ob[G * D + G + g] = l;
      }
    }
    __syncwarp();
    if (full) {
      finish_mma<G>(p, layer, i, h, slot, out, ob, lane);
    } else {
      // a cut (request, head): leave this piece's state for combine_kernel
      const int seg = i * p.Hk + h;
      const int pslot = (seg == first_seg) ? 0 : 1;
      constexpr int PW = G * (D + 2);
      float* part = p.partials + (size_t)(w * 2 + pslot) * PW;
      for (int x = lane; x < G * D; x += 32) part[(x / D) * (D + 2) + (x % D)] = ob[x];
      if (lane < 2 * G) part[(lane % G) * (D + 2) + D + lane / G] = ob[G * D + lane];
    }
    __syncwarp();  // the buffer is reused by the next piece
    if (j < end) {
      cc.blk = cc.nb - 1;
      cursor_next(p, cc);
    }
  }
  if (failed) {
    for (int64_t jl = j - start; jl < issued - start; ++jl)
      (void)mbar_wait_bounded(&bars[jl % S], (uint32_t)((jl / S) & 1), kWaitLimitNs);
  }
}

// ------------------------------------------------------------- combine ---
//
// One warp per (request, kv head) of the step.  A (request, head) whose
// blocks were cut between several attention workers is merged here: the
// workers' states (m, l, unnormalised output per query head) are combined
// with weights 2^(m_k - max m), then finished like an uncut one.  Runs after
// the attention kernel has completed, so no worker waits for another.
template <int G>
__global__ void __launch_bounds__(kSmallWarps * 32)
combine_kernel(PoolDev p, int layer, __nv_bfloat16* __restrict__ out) {
  constexpr int D = kMmaD, PW = G * (D + 2);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // which workers cut this (request, head): from the plan, final before the step
  const int n = p.plan_misc[0];
  const int gw = blockIdx.x * kSmallWarps + warp;
  if (gw >= n * p.Hk) return;
  const int i = gw / p.Hk, h = gw % p.Hk;
  const int nb = p.plan_nb[i];
  const int slot = p.plan_slot[i];
  const int64_t Tb = (int64_t)p.plan_misc[2] * p.Hk;
  const int64_t W = (int64_t)p.num_workers;
  const int64_t Weff = W < Tb ? W : Tb;
  const int64_t seg_b0 = (int64_t)p.Hk * p.plan_cum[i] + (int64_t)h * nb;
  const int64_t w_first = ((seg_b0 + 1) * Weff - 1) / Tb;
  const int64_t w_last = ((seg_b0 + nb) * Weff - 1) / Tb;
  if (w_first == w_last) return;  // finished by the attention kernel
  const bool first_is_second = (w_first * Tb) / Weff != seg_b0;  // its 2nd state slot
  const int nparts = (int)(w_last - w_first + 1);
  auto part_of = [&](int k) -> const float* {
    const int64_t wk = w_first + k;
    const int ps = (k == 0 && first_is_second) ? 1 : 0;
    return p.partials + (size_t)(wk * 2 + ps) * PW;
  };
  // the workers' states and the staged token come from earlier kernels
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const size_t srow = (((size_t)slot * p.L + layer) * p.Hk + h) * 2;
  const __nv_bfloat16* vst = reinterpret_cast<const __nv_bfloat16*>(p.staging) + (srow + 1) * D;
  float vs[4], sst[G];
#pragma unroll
  for (int e = 0; e < 4; ++e) vs[e] = __bfloat162float(vst[lane + 32 * e]);
#pragma unroll
  for (int g = 0; g < G; ++g) sst[g] = p.sstage[(i * p.Hk + h) * 4 + g];
  float mmax[G], lsum[G], acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    mmax[g] = -INFINITY;
    lsum[g] = 0.f;
    acc[g][0] = acc[g][1] = acc[g][2] = acc[g][3] = 0.f;
  }
  // online merge over the parts: every lane holds dims lane + 32e of each head
  for (int k = 0; k < nparts; ++k) {
    const float* pk = part_of(k);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mk = __ldcg(pk + g * (D + 2) + D);
      const float lk = __ldcg(pk + g * (D + 2) + D + 1);
      float ov[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) ov[e] = __ldcg(pk + g * (D + 2) + lane + 32 * e);
      if (mk == -INFINITY) continue;
      const float mn = fmaxf(mmax[g], mk);
      const float al = (mmax[g] == -INFINITY) ? 0.f : exp2f(mmax[g] - mn);
      const float be = exp2f(mk - mn);
      lsum[g] = lsum[g] * al + lk * be;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[g][e] = acc[g][e] * al + ov[e] * be;
      mmax[g] = mn;
    }
  }
  // the staged token, normalisation, store
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float mn = fmaxf(mmax[g], sst[g]);
    const float al = (mmax[g] == -INFINITY) ? 0.f : exp2f(mmax[g] - mn);
    const float be = exp2f(sst[g] - mn);
    const float inv = 1.0f / (lsum[g] * al + be);
    __nv_bfloat16* orow = out + ((size_t)i * p.Hq + h * G + g) * D;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      orow[lane + 32 * e] = __float2bfloat16_rn((acc[g][e] * al + be * vs[e]) * inv);
  }
}

size_t mma_smem_bytes() {
  return (size_t)kMmaWarps * kMmaStages * kMmaStageB + (size_t)kMmaWarps * kObFloats * 4 +
         (size_t)kMmaWarps * kMmaStages * 8 + 1024;
}

// Both kernels are launched as programmatic dependents of the previous
// kernel in the stream (see griddepcontrol in the kernels): the attention
// kernel's prologue (cursors, first K/V copies) overlaps the prep kernel.
static cudaLaunchConfig_t pdl_config(cudaLaunchAttribute* attr, dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int G>
static cudaError_t launch_mma_t(const PoolDev& p, const CUtensorMap* map, int layer, int n,
                                const void* q, const void* k, const void* v, void* out, int grid,
                                cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  const int warps = n * p.Hk;
  const dim3 sgrid((warps + kSmallWarps - 1) / kSmallWarps), sblock(kSmallWarps * 32);
  cudaLaunchConfig_t c1 = pdl_config(attr, sgrid, sblock, 0, st);
  cudaError_t e = cudaLaunchKernelEx(&c1, prep_kernel<G>, p, layer, (const __nv_bfloat16*)q,
                                     (const __nv_bfloat16*)k, (const __nv_bfloat16*)v);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t c2 = pdl_config(attr, dim3(grid), dim3(kMmaWarps * 32), mma_smem_bytes(), st);
  e = cudaLaunchKernelEx(&c2, attn_mma_kernel<G, kMmaStages>, *map, p, layer, (__nv_bfloat16*)out);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t c3 = pdl_config(attr, sgrid, sblock, 0, st);
  return cudaLaunchKernelEx(&c3, combine_kernel<G>, p, layer, (__nv_bfloat16*)out);
}

template <int G>
static cudaError_t occupancy_mma_t(int* blocks) {
  auto kern = attn_mma_kernel<G, kMmaStages>;
  const size_t smem = mma_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, kern, kMmaWarps * 32, smem);
}

int mma_warps_per_cta() { return kMmaWarps; }

// Three launches: prep_kernel, attn_mma_kernel, combine_kernel.
cudaError_t launch_attention_mma(const PoolDev& p, const CUtensorMap* map, int layer, int n,
                                 const void* q, const void* k, const void* v, void* out, int grid,
                                 cudaStream_t st) {
  if (p.G == 1) return launch_mma_t<1>(p, map, layer, n, q, k, v, out, grid, st);
  if (p.G == 2) return launch_mma_t<2>(p, map, layer, n, q, k, v, out, grid, st);
  if (p.G == 4) return launch_mma_t<4>(p, map, layer, n, q, k, v, out, grid, st);
  return cudaErrorInvalidValue;
}

cudaError_t attention_mma_occupancy(const PoolDev& p, int* blocks) {
  if (p.G == 1) return occupancy_mma_t<1>(blocks);
  if (p.G == 2) return occupancy_mma_t<2>(blocks);
  if (p.G == 4) return occupancy_mma_t<4>(blocks);
  return cudaErrorInvalidValue;
}

}  // namespace gp
