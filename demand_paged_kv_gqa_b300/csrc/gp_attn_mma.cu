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
// operand, so Q·K^T runs as warp-level bf16 tensor-core products (mma.sync
// m16n8k16, fp32 accumulation).  The output is accumulated transposed,
// O^T = V^T·P^T: the block's values are the 16-row operand (16 dims at a
// time) and the softmax weights, hi and lo parts of the G heads, are the
// 8 columns, taken straight from the score accumulators' layout.  The contraction is a real dense
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
// Ahead of every piece, the same ring carries a "meta"
// item (bulk copies of the query rows, the new key and value, the summaries
// and the rotary rows), so building a piece's operands never waits on a
// dependent global load.
// Work is split over a persistent grid: contiguous ranges of blocks per warp,
// weighted so that each (request, head) start counts as a few blocks (the
// plan kernel computes them).  A (request, head) cut between warps leaves one
// state per warp, and combine_kernel merges them after the attention grid has
// finished.  Every wait is bounded and on the warp's own copies.
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
#ifndef GP_PREF_L2
#define GP_PREF_L2 3  // blocks a warp prefetches into L2 before the dependency wait
#endif
constexpr int kMmaWarps = GP_MMA_WARPS;
constexpr int kMmaStages = GP_MMA_STAGES;
constexpr int kObFloats = 4 * (kMmaD + 2);  // per-warp merge buffer: [G<=4][D] + m + l
// prep and combine run one warp per CTA: their CTAs are launched early (see
// griddepcontrol) and must fit beside two resident attention CTAs.
constexpr int kSmallWarps = 1;

// An L2 prefetch of bytes (a multiple of 16) at a 16-byte aligned address.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The K and V rows of the cursor's block (page given) into L2.
__device__ __forceinline__ void prefetch_block_l2(const PoolDev& p, int layer, const Cursor& c, int page) {
  const int t0 = c.base + c.blk * kBlockTok;
  const int in_page = p.P_log2 >= 0 ? (t0 & (p.P - 1)) : t0 % p.P;
  const size_t krow = ((((size_t)page * p.L + layer) * p.Hk + c.h) * 2) * p.P + in_page;
  prefetch_l2(p.kv + krow * (kMmaD * 2), kBlockTok * kMmaD * 2);
  prefetch_l2(p.kv + (krow + p.P) * (kMmaD * 2), kBlockTok * kMmaD * 2);
}

// One 16-token block (K and V, both 64-column halves) of a (page, layer,
// head) in one copy: the block map's box (64, 16, 2, 2, 1) at token offset
// tok within the page and row index (page * L + layer) * Hk + head.
__device__ __forceinline__ void tma_load_block(void* dst, const CUtensorMap* map, int tok, int prow,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(tok), "r"(0), "r"(0), "r"(prow),
      "r"(smem_u32(bar))
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
  const int t0 = c.base + c.blk * kBlockTok;  // resident token of the block's first row
  const int in_page = p.P_log2 >= 0 ? (t0 & (p.P - 1)) : t0 % p.P;
  mbar_expect_tx(bar, kMmaStageB);
  tma_load_block(stage, map, in_page, (page * p.L + layer) * p.Hk + c.h, bar);
}

// ------------------------------------------------------------ meta items ---
//
// Besides K/V blocks, a warp's ring carries one "meta" item in front of each
// piece: what the piece needs besides the keys, copied by the bulk-copy
// engine with the blocks.  Offsets inside a stage:
constexpr int kQPitch = kMmaD;      // query row pitch (elements): the G rows are one copy
constexpr int kMetaQ = 0;       // the G query rows, bf16 (<= 4 x 256 B)
constexpr int kMetaK = 1088;    // the step's new key, bf16
constexpr int kMetaV = 1344;    // the step's new value, bf16
constexpr int kMetaS = 1600;    // short and long summary before this step, fp32
// kMetaC32 .. kMetaSF: the position's RoPE row, as laid out in the pool
constexpr int kMetaC32 = 2624;  // rotary cos / sin rows of the position, fp32
constexpr int kMetaS32 = 2880;
constexpr int kMetaC32lo = 3136;  // their fp32 residuals (cos, sin: c32 + c32lo ~ fp64)
constexpr int kMetaS32lo = 3392;
constexpr int kMetaC64 = 3648;  // the fp64 rows (the rare pairs the fp32 evaluation leaves open)
constexpr int kMetaS64 = 4160;
constexpr int kMetaSF = 4672;   // written in place: both summaries after this step's fold
static_assert(kMetaS32 == kMetaC32 + 2 * kMmaD && kMetaC32lo == kMetaC32 + 4 * kMmaD &&
                  kMetaS32lo == kMetaC32 + 6 * kMmaD && kMetaC64 == kMetaC32 + 8 * kMmaD &&
                  kMetaS64 == kMetaC64 + 4 * kMmaD && kMetaSF == kMetaC32 + 16 * kMmaD,
              "the meta item holds the RoPE row as laid out in the pool");

// Per-warp extra buffer (after ob): the staged-token score of each query
// head and the staged value (fp32), for finishing a piece in place.
constexpr int kObxFloats = 4 + kMmaD;
constexpr int kWarpBufFloats = ((kObFloats + kObxFloats + 3) / 4) * 4;

// The step's plan entries of 32 consecutive requests, one per lane, so that a
// cursor crossing into the next request reads registers, not memory.
struct PlanWin {
  int base = -(1 << 30);
  int nb = 1, slot = 0, R = 0, flags = 0, pos = 0, tb = 0;
};
struct PlanEntry {
  int nb, slot, R, flags, pos, tb;  // tb: first resident token the kernel attends
};

__device__ __forceinline__ PlanEntry plan_at(const PoolDev& p, PlanWin& w, int i, int n, int lane) {
  if (i < w.base || i >= w.base + 32) {  // warp-uniform
    w.base = i;
    const int k = i + lane;
    if (k < n) {
      w.nb = p.plan_nb[k]; w.slot = p.plan_slot[k]; w.R = p.plan_R[k];
      w.flags = p.plan_flags[k]; w.pos = p.plan_pos[k]; w.tb = p.plan_base[k];
    } else {
      w.nb = 1; w.slot = 0; w.R = 0; w.flags = 0; w.pos = 0; w.tb = 0;
    }
  }
  const int src = i - w.base;
  PlanEntry e;
  e.nb = __shfl_sync(0xffffffffu, w.nb, src);
  e.slot = __shfl_sync(0xffffffffu, w.slot, src);
  e.R = __shfl_sync(0xffffffffu, w.R, src);
  e.flags = __shfl_sync(0xffffffffu, w.flags, src);
  e.pos = __shfl_sync(0xffffffffu, w.pos, src);
  e.tb = __shfl_sync(0xffffffffu, w.tb, src);
  return e;
}

// Block-table windows for the producer: the window in use and the one it
// will need next, loaded when the current one is installed, so that crossing
// into it (the next 32 pages of a segment, the next head's or the next
// request's first pages) is a register swap instead of a dependent load.
struct PageWinAhead {
  int slot = -1, base = 0, page = 0;     // entries base .. base+31 of slot's table, one per lane
  int nslot = -1, nbase = 0, npage = 0;  // the expected next window (nslot -1: none)
};

__device__ __forceinline__ int page_index(const PoolDev& p, int tok) {
  return p.P_log2 >= 0 ? (tok >> p.P_log2) : tok / p.P;
}

__device__ __forceinline__ int load_window(const PoolDev& p, int slot, int base, int lane) {
  const int e = base + lane;
  return e < p.block_width ? p.block[(size_t)slot * p.block_width + e] : 0;
}

// The window the cursor's walk needs after (c.slot, base): the segment's next
// 32 pages; else the next head's first window (the same table) unless it is
// this one; else the next request's first window, when its plan entry is in
// the plan window w.  False when unknown.  Warp-uniform.
__device__ __forceinline__ bool next_window(const PoolDev& p, const PlanWin& w, const Cursor& c,
                                            int base, int n, int& nslot, int& nbase) {
  const int last = page_index(p, c.base + (c.nb - 1) * kBlockTok);
  if (base + 32 <= last) { nslot = c.slot; nbase = base + 32; return true; }
  const int first = page_index(p, c.base);
  if (c.h + 1 < p.Hk && first != base) { nslot = c.slot; nbase = first; return true; }
  const int i1 = c.i + 1;
  if (i1 >= n || i1 < w.base || i1 >= w.base + 32) return false;
  nslot = __shfl_sync(0xffffffffu, w.slot, i1 - w.base);
  nbase = page_index(p, __shfl_sync(0xffffffffu, w.tb, i1 - w.base));
  return true;
}

// Page id of the cursor's block; all lanes call it with the same cursor.
__device__ __forceinline__ int page_of_ahead(const PoolDev& p, PageWinAhead& win, const PlanWin& w,
                                             const Cursor& c, int n, int lane) {
  const int pidx = page_index(p, c.base + c.blk * kBlockTok);  // prefix pages first, then private
  if (c.slot != win.slot || pidx < win.base || pidx >= win.base + 32) {
    if (c.slot == win.nslot && pidx >= win.nbase && pidx < win.nbase + 32) {
      win.slot = win.nslot; win.base = win.nbase; win.page = win.npage;
    } else {
      win.slot = c.slot; win.base = pidx; win.page = load_window(p, c.slot, pidx, lane);
    }
    int ns, nb;
    if (next_window(p, w, c, win.base, n, ns, nb)) {
      win.nslot = ns; win.nbase = nb; win.npage = load_window(p, ns, nb, lane);
    } else {
      win.nslot = -1;
    }
  }
  int page = __shfl_sync(0xffffffffu, win.page, pidx - win.base);
  if ((unsigned)page >= (unsigned)p.num_pages) {
    if (lane == 0) set_status(p, GP_ST_BAD_PAGE, c.slot);
    page = 0;
  }
  return page;
}

__device__ __forceinline__ void walk_next(const PoolDev& p, PlanWin& w, Cursor& c, int n, int lane) {
  if (++c.blk == c.nb) {
    c.blk = 0;
    if (++c.h == p.Hk) {
      c.h = 0;
      if (++c.i < n) {
        const PlanEntry e = plan_at(p, w, c.i, n, lane);
        c.nb = e.nb;
        c.slot = e.slot;
        c.base = e.tb;
      }
    }
  }
}

// A meta item in two halves on one mbarrier: the part that is final before
// the step (the summaries and the position's RoPE row; it arms the barrier
// for the whole item) and the step's inputs (query rows, new key, value).
template <int G>
__device__ __forceinline__ void issue_meta_state(const PoolDev& p, int layer, int h, int slot, int pos,
                                                 uint8_t* st, uint64_t* bar) {
  constexpr int D = kMmaD;
  const uint32_t bytes = G * D * 2 + 2 * D * 2 + 2 * D * 4 + (p.rope ? 2 * D * 4 + D * 8 : 0);
  mbar_expect_tx(bar, bytes);
  bulk_g2s(st + kMetaS, p.summary + ((((size_t)slot * p.L + layer) * p.Hk + h) * 2) * D, 2 * D * 4, bar);
  if (p.rope) {
    // the position's RoPE row: c32, s32, their residuals, c64, s64 (one copy)
    bulk_g2s(st + kMetaC32, rope_c32(p, pos), 16 * D, bar);
  }
}

template <int G>
__device__ __forceinline__ void issue_meta_inputs(const PoolDev& p, int i, int h, const __nv_bfloat16* q,
                                                  const __nv_bfloat16* knew, const __nv_bfloat16* vnew,
                                                  uint8_t* st, uint64_t* bar) {
  constexpr int D = kMmaD;
  bulk_g2s(st + kMetaQ, q + ((size_t)i * p.Hq + h * G) * D, G * D * 2, bar);  // the G query rows
  bulk_g2s(st + kMetaK, knew + ((size_t)i * p.Hk + h) * D, D * 2, bar);
  bulk_g2s(st + kMetaV, vnew + ((size_t)i * p.Hk + h) * D, D * 2, bar);
}

// The same rows as issue_meta_inputs, prefetched into L2 only.
template <int G>
__device__ __forceinline__ void prefetch_inputs_l2(const PoolDev& p, int i, int h, const __nv_bfloat16* q,
                                                   const __nv_bfloat16* knew, const __nv_bfloat16* vnew) {
  constexpr int D = kMmaD;
  prefetch_l2(q + ((size_t)i * p.Hq + h * G) * D, G * D * 2);
  prefetch_l2(knew + ((size_t)i * p.Hk + h) * D, D * 2);
  prefetch_l2(vnew + ((size_t)i * p.Hk + h) * D, D * 2);
}

template <int G>
__device__ __forceinline__ void issue_meta(const PoolDev& p, int layer, int i, int h, int slot,
                                           int pos, const __nv_bfloat16* q,
                                           const __nv_bfloat16* knew, const __nv_bfloat16* vnew,
                                           uint8_t* st, uint64_t* bar) {
  issue_meta_state<G>(p, layer, h, slot, pos, st, bar);
  issue_meta_inputs<G>(p, i, h, q, knew, vnew, st, bar);
}

// Pointers to what a piece needs (a meta item in shared memory).
struct PieceIn {
  const __nv_bfloat16* q;  // [G][kQPitch]
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* s;          // [2][d] before this step
  const float* c32;
  const float* s32;
  const float* c32lo;      // fp32 residuals of the rotary rows
  const float* s32lo;
  const double* c64;       // the fp64 rotary rows
  const double* s64;
  const float* sf;         // [2][d] after this step's fold (set when needed)
};

// Both summaries after this step's fold, all d dims (4 per lane), in fp32 and
// in exact order: q̄ = (sum of the G heads in head order) / G;
// s' = fl(fl(b*s) + fl((1-b)*q̄)), or q̄ on the request's first step.
template <int G>
__device__ __forceinline__ void fold_rows(const PoolDev& p, const PieceIn& in, int flags, int lane,
                                          float* sf) {
  constexpr int D = kMmaD;
  const int d0 = lane * 4;
  float qb[4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint2 w = *reinterpret_cast<const uint2*>(in.q + g * kQPitch + d0);
    const float v[4] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y)};
#pragma unroll
    for (int e = 0; e < 4; ++e) qb[e] = g == 0 ? v[e] : __fadd_rn(qb[e], v[e]);
  }
  const float4 os = *reinterpret_cast<const float4*>(in.s + d0);
  const float4 ol = *reinterpret_cast<const float4*>(in.s + D + d0);
  const float osv[4] = {os.x, os.y, os.z, os.w}, olv[4] = {ol.x, ol.y, ol.z, ol.w};
  const float aS = __fsub_rn(1.0f, p.beta_s), aL = __fsub_rn(1.0f, p.beta_l);
  const int first = flags & kPlanFirst;
  float ns[4], nl[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float qm = __fdiv_rn(qb[e], (float)G);
    ns[e] = first ? qm : __fadd_rn(__fmul_rn(p.beta_s, osv[e]), __fmul_rn(aS, qm));
    nl[e] = first ? qm : __fadd_rn(__fmul_rn(p.beta_l, olv[e]), __fmul_rn(aL, qm));
  }
  *reinterpret_cast<float4*>(sf + d0) = make_float4(ns[0], ns[1], ns[2], ns[3]);
  *reinterpret_cast<float4*>(sf + D + d0) = make_float4(nl[0], nl[1], nl[2], nl[3]);
}

// Pair of fp32 values -> packed bf16 (hi) and the packed rounded residual.
__device__ __forceinline__ void split2x(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ void split3x(float a, float b, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float ra = a - __low2float(h), rb = b - __high2float(h);
  const __nv_bfloat162 m = __floats2bfloat162_rn(ra, rb);
  const __nv_bfloat162 l = __floats2bfloat162_rn(ra - __low2float(m), rb - __high2float(m));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  mid = *reinterpret_cast<const uint32_t*>(&m);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// The tensor-core operand rows of lane (g = lane / 4, t = lane % 4): rows
// g < G = query head g rotated to the position and scaled by log2(e)/sqrt(d),
// bf16 hi (row g) + lo (row g+8); at a boundary rows 4/5 = short/long summary
// after this step's fold, rotated and scaled by 1/sqrt(d), hi (rows 4/5) +
// mid (rows 12/13) with the lo parts in rows 6/7.  Other rows are zero.
template <int G>
__device__ __forceinline__ void build_rows(const PoolDev& p, const PieceIn& in, int flags, int lane,
                                           uint32_t (&afr)[8][4]) {
  constexpr int D = kMmaD;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) afr[kk][0] = afr[kk][1] = afr[kk][2] = afr[kk][3] = 0u;
  const bool head_row = g < G;
  const bool sum_row = (flags & kPlanScore) && g >= 4;
  if (!(head_row || sum_row)) return;
  const int X = g & 1;
  const float sc = head_row ? 1.4426950408889634f / sqrtf((float)D)   // log2(e)/sqrt(d)
                            : 1.0f / sqrtf((float)D);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // dims di, di+1 and their partners +64
      const int di = 16 * kk + 2 * t + 8 * half;
      float x0, x1, y0, y1;
      if (head_row) {
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(in.q + g * kQPitch + di);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(in.q + g * kQPitch + di + 64);
        x0 = bf16lo(wa); x1 = bf16hi(wa); y0 = bf16lo(wb); y1 = bf16hi(wb);
      } else {
        const float2 fa = *reinterpret_cast<const float2*>(in.sf + X * D + di);
        const float2 fb = *reinterpret_cast<const float2*>(in.sf + X * D + di + 64);
        x0 = fa.x; x1 = fa.y; y0 = fb.x; y1 = fb.y;
      }
      if (p.rope) {
        const float2 c = *reinterpret_cast<const float2*>(in.c32 + di);
        const float2 s = *reinterpret_cast<const float2*>(in.s32 + di);
        const float a0 = x0 * c.x - y0 * s.x, b0 = y0 * c.x + x0 * s.x;
        const float a1 = x1 * c.y - y1 * s.y, b1 = y1 * c.y + x1 * s.y;
        x0 = a0; y0 = b0; x1 = a1; y1 = b1;
      }
      x0 *= sc; x1 *= sc; y0 *= sc; y1 *= sc;
      // registers: [0] row g, cols 2t..; [1] row g+8; [2] row g, cols 2t+8..; [3] row g+8
      uint32_t xh, xl, yh, yl;
      if (head_row) {
        split2x(x0, x1, xh, xl);
        split2x(y0, y1, yh, yl);
      } else {
        uint32_t xm, ym, xlo, ylo;
        split3x(x0, x1, xh, xm, xlo);
        split3x(y0, y1, yh, ym, ylo);
        if (g >= 6) {  // rows 6/7 carry the lo parts; rows 14/15 stay zero
          xh = xlo; yh = ylo; xl = 0u; yl = 0u;
        } else {       // rows 4/5 hi, rows 12/13 mid
          xl = xm; yl = ym;
        }
      }
      afr[kk][2 * half + 0] = xh;
      afr[kk][2 * half + 1] = xl;
      afr[kk + 4][2 * half + 0] = yh;
      afr[kk + 4][2 * half + 1] = yl;
    }
  }
}

// Once per (request, kv head) and step, by the piece holding its first block:
//   the staged token (key rotated in fp64 and rounded once to bf16, value)
//   into the staging rows; each query head's score against it (log2 domain)
//   into sstage and obx[g]; the staged value into obx[4..]; and both folded
//   summaries into the next-summary rows (copied over the summaries by the
//   commit kernel once every layer has been read).
template <int G>
__device__ void segment_duties(const PoolDev& p, int layer, int i, int h, int slot, int flags,
                               const PieceIn& in, float* obx, int lane) {
  using Gm = Geo<__nv_bfloat16, kMmaD>;
  constexpr int D = kMmaD, NE = Gm::NE, H2 = NE / 2;
  const int sigma = lane & 7, grp = lane >> 3;
  const size_t srow = (((size_t)slot * p.L + layer) * p.Hk + h) * 2;
  float vraw[NE], kst[NE];
  load_row<__nv_bfloat16, Gm>(reinterpret_cast<const uint8_t*>(in.k), sigma, kst);
  load_row<__nv_bfloat16, Gm>(reinterpret_cast<const uint8_t*>(in.v), sigma, vraw);
  if (p.rope) {
    // x·c - y·s and y·c + x·s rounded once to bf16, as in fp64.  The lane
    // slice sigma holds 8 pairs (dims 8·sigma + e and +64, e < 8); lane
    // (grp, sigma) rotates pairs 2·grp and 2·grp + 1 -- by the certified fp32
    // evaluation, or the fp64 expression for a pair it leaves open -- and the
    // 8 results are gathered from the lanes (e / 2, sigma) by shuffles.
    static_assert(H2 == 8, "8 rotate-half pairs per lane slice");
    uint32_t rot[2];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      float x = kst[jj], y = kst[jj + H2];
#pragma unroll
      for (int g2 = 1; g2 < 4; ++g2)
        if (grp == g2) { x = kst[2 * g2 + jj]; y = kst[2 * g2 + jj + H2]; }
      const int di = 8 * sigma + 2 * grp + jj;
      const float c1 = in.c32[di], c2 = in.c32lo[di], s1 = in.s32[di], s2 = in.s32lo[di];
      uint16_t ra, rb;
      if (!(rope_bf16_certified(x, y, c1, c2, -s1, -s2, ra) &&
            rope_bf16_certified(y, x, c1, c2, s1, s2, rb))) {
        const double c = in.c64[di], sn = in.s64[di];
        const double xd = (double)x, yd = (double)y;
        ra = f64_to_bf16_rne(__dsub_rn(__dmul_rn(xd, c), __dmul_rn(yd, sn)));
        rb = f64_to_bf16_rne(__dadd_rn(__dmul_rn(yd, c), __dmul_rn(xd, sn)));
      }
      rot[jj] = (uint32_t)ra | ((uint32_t)rb << 16);
    }
#pragma unroll
    for (int e = 0; e < H2; ++e) {
      const uint32_t v = __shfl_sync(0xffffffffu, rot[e & 1], (e >> 1) * 8 + sigma);
      kst[e] = __uint_as_float(v << 16);
      kst[e + H2] = __uint_as_float(v & 0xffff0000u);
    }
  }
  if (grp == 0) {
    // both rows with 16-byte stores: elements 8c .. 8c+7 are the 16-byte
    // chunk c·8 + sigma of the row (all values already on the bf16 grid)
    uint8_t* st = p.staging + srow * D * 2;
#pragma unroll
    for (int c = 0; c < Gm::VEC; ++c) {
      uint32_t wk[4], wv[4];
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        wk[k2] = (__float_as_uint(kst[c * 8 + 2 * k2]) >> 16) | (__float_as_uint(kst[c * 8 + 2 * k2 + 1]) & 0xffff0000u);
        wv[k2] = (__float_as_uint(vraw[c * 8 + 2 * k2]) >> 16) | (__float_as_uint(vraw[c * 8 + 2 * k2 + 1]) & 0xffff0000u);
      }
      *reinterpret_cast<uint4*>(st + (c * 8 + sigma) * 16) = make_uint4(wk[0], wk[1], wk[2], wk[3]);
      *reinterpret_cast<uint4*>(st + D * 2 + (c * 8 + sigma) * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
#pragma unroll
    for (int e = 0; e < NE; ++e) obx[4 + dim_of<Gm>(e, sigma)] = vraw[e];
  }
  {
    const float qscale = 1.4426950408889634f / sqrtf((float)D);
    float sa = 0.f;
    if (grp < G) {  // one query head per 8-lane group
      float qr[NE];
      load_row<__nv_bfloat16, Gm>(reinterpret_cast<const uint8_t*>(in.q + grp * kQPitch), sigma, qr);
      if (p.rope) {
#pragma unroll
        for (int e = 0; e < H2; ++e) {
          const int di = dim_of<Gm>(e, sigma);
          const float c = in.c32[di], s = in.s32[di];
          const float x = qr[e], y = qr[e + H2];
          qr[e] = x * c - y * s;
          qr[e + H2] = y * c + x * s;
        }
      }
#pragma unroll
      for (int e = 0; e < NE; ++e) sa = fmaf(qr[e] * qscale, kst[e], sa);
    }
    sa += __shfl_xor_sync(0xffffffffu, sa, 1);
    sa += __shfl_xor_sync(0xffffffffu, sa, 2);
    sa += __shfl_xor_sync(0xffffffffu, sa, 4);
    if (grp < G && sigma == 0) {
      p.sstage[(i * p.Hk + h) * 4 + grp] = sa;
      obx[grp] = sa;
    }
  }
  // The folded summaries.  A request at a boundary has them read again,
  // unfolded, by the other pieces of its (request, head) for their summary
  // scores, so its fold goes to summary_next and commit_kernel makes it
  // current.  No other piece uses the summaries of any other request (its
  // meta items load them unused), so its fold is written in place.
  float* nxt = ((flags & kPlanScore) ? p.summary_next : p.summary) + srow * D;
  reinterpret_cast<float4*>(nxt)[lane] = reinterpret_cast<const float4*>(in.sf)[lane];
  reinterpret_cast<float4*>(nxt + D)[lane] = reinterpret_cast<const float4*>(in.sf + D)[lane];
}

// Output of one (request, kv head) from the attention state in the warp's
// buffer ob ([G][D] unnormalised output, then m[G] in the log2 domain, l[G])
// and the staged token in obx: merged, normalised, stored (16-byte stores).
template <int G>
__device__ __forceinline__ void finish_mma(const PoolDev& p, int i, int h,
                                           __nv_bfloat16* __restrict__ out, const float* ob,
                                           const float* obx, int lane) {
  using Gm = Geo<__nv_bfloat16, kMmaD>;
  constexpr int D = kMmaD;
  const int sigma = lane & 7, g = lane >> 3;  // one query head per 8-lane group
  if (g >= G) return;
  const float a = obx[g];
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
      const int d0 = dim_of<Gm>(c * 8 + 2 * k2, sigma);
      const float r0 = (ob[g * D + d0] * al + be * obx[4 + d0]) * inv;
      const float r1 = (ob[g * D + d0 + 1] * al + be * obx[4 + d0 + 1]) * inv;
      const __nv_bfloat162 pr = __floats2bfloat162_rn(r0, r1);
      wv[k2] = *reinterpret_cast<const uint32_t*>(&pr);
    }
    *reinterpret_cast<uint4*>(orow + (c * 8 + sigma) * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
}

// One 16-token block of keys and values (a ring stage at sK: K then V) for
// the 16 operand rows afr: scores, the boundary summary scores (rows 4/5,
// written to lgX[t0 + token] for tokens below nvalid when `score`), the
// online softmax of the G head rows (running max m, sum l, log2 domain) and
// O^T += V^T · P^T into o.
// 2^x by the hardware approximation (ex2.approx.ftz: relative error about
// 2^-22, flushes subnormal results to 0, 2^-inf = 0).  The softmax weights
// it produces are split into bf16 hi + lo parts (16 bits) right after.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// This lane's shared-memory offsets (inside a ring stage) of the 16
// ldmatrix loads of one block: [0..7] the keys, [8..15] the values.  They
// depend on the lane only, so a kernel computes them once.
struct LdsmOffsets {
  uint32_t k[8], v[8];
};
__device__ __forceinline__ LdsmOffsets ldsm_offsets(int lane) {
  const int mi = lane >> 3, ri = lane & 7;
  const int k_tok = 8 * (mi >> 1) + ri, k_half = mi & 1;   // K: token, chunk parity
  // V^T as the 16 x 16 operand (rows: dims, columns: tokens), by transposing
  // loads of V[token][dims]: matrices (tokens 0-7 | 8-15) x (dims +0 | +8)
  const int v_tok = 8 * (mi >> 1) + ri, v_half = mi & 1;
  LdsmOffsets o;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int ch = 2 * kk + k_half;   // 16-byte chunk of the key row
    o.k[kk] = (uint32_t)((ch >> 3) * 2048) + swz(k_tok, ch & 7);
    const int cv = 2 * kk + v_half;   // 16-byte chunk = 8 dims
    o.v[kk] = 4096u + (uint32_t)((cv >> 3) * 2048) + swz(v_tok, cv & 7);
  }
  return o;
}

template <int G>
__device__ __forceinline__ void attend_block(const uint32_t (&afr)[8][4], float (&o)[8][4], float& m,
                                             float& l, uint32_t sK, int t0, int nvalid, bool score,
                                             float* lgX, const LdsmOffsets& lo, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const bool head_row = g < G;
  // the lane whose softmax weights feed this lane's weight column: column
  // n < G is head n (hi part), G <= n < 2G is head n - G (lo part)
  const int p_src = ((g >= G && g < 2 * G) ? (g - G) : g) * 4 + t;
  // ---- scores: S[16 rows][16 tokens] = A · K^T
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    uint32_t b[4];
    ldsm_x4(b, sK + lo.k[kk]);
    mma_bf16(c0, afr[kk], b[0], b[1]);
    mma_bf16(c1, afr[kk], b[2], b[3]);
  }
  // this thread's tokens of the block: 2t, 2t+1, 8+2t, 9+2t
  float sv[4] = {c0[0] + c0[2], c0[1] + c0[3], c1[0] + c1[2], c1[1] + c1[3]};
  const int tok[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
  // summary scores: rows 4/5 (+ rows 12/13 in the same thread) plus the
  // lo rows 6/7 held 8 lanes up
  if (score) {
    float other[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) other[u] = __shfl_xor_sync(0xffffffffu, sv[u], 8);
    if (g == 4 || g == 5) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (tok[u] < nvalid) lgX[t0 + tok[u]] = sv[u] + other[u];
    }
  }
  // ---- online softmax (log2 domain) for head row g
  // rows beyond the G heads, and tokens beyond the resident count (the last
  // block of a segment only), take no part in the softmax
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (!head_row) sv[u] = -INFINITY;
  if (nvalid < kBlockTok) {  // warp-uniform
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (tok[u] >= nvalid) sv[u] = -INFINITY;
  }
  float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  // the running max moves only when a score exceeds it by more than 2^8:
  // weights stay <= 256, and the final normalisation uses the same m.
  // The accumulator columns of a head sit in other lanes, so the rescale
  // is taken by the whole warp (rare: a few times per piece).
  if (__any_sync(0xffffffffu, mx > m + 8.0f)) {
    float al = 1.0f;
    if (mx > m + 8.0f) {
      al = ex2_approx(m - mx);        // 0 when m == -inf
      l *= al;
      m = mx;
    }
    // column c holds head c mod G (columns >= 2G are zero)
    const float a0 = __shfl_sync(0xffffffffu, al, ((2 * t) % G) * 4);
    const float a1 = __shfl_sync(0xffffffffu, al, ((2 * t + 1) % G) * 4);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
    }
  }
  float pv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    pv[u] = (sv[u] == -INFINITY) ? 0.f : ex2_approx(sv[u] - m);
    l += pv[u];
  }
  uint32_t ph[4], pl[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) split2(pv[u], ph[u], pl[u]);
  // P^T as the 16 x 8 operand: this lane's column g, tokens 2t, 2t+1 and
  // 2t+8, 2t+9 -- hi parts for g < G, lo parts of head g - G for
  // G <= g < 2G (fetched from that head's lane), zero beyond
  const uint32_t xl0 = __shfl_sync(0xffffffffu, pack2(pl[0], pl[1]), p_src);
  const uint32_t xl1 = __shfl_sync(0xffffffffu, pack2(pl[2], pl[3]), p_src);
  const uint32_t bp0 = g < G ? pack2(ph[0], ph[1]) : (g < 2 * G ? xl0 : 0u);
  const uint32_t bp1 = g < G ? pack2(ph[2], ph[3]) : (g < 2 * G ? xl1 : 0u);
  // ---- O^T += V^T · P^T, 16 dims at a time
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t a[4];
    ldsm_x4_t(a, sK + lo.v[mt]);
    mma_bf16(o[mt], a, bp0, bp1);
  }
}

// A piece's totals into the warp buffer ob: [G][D] unnormalised output,
// then m[G] (log2 domain), l[G].  l is reduced over the row's four lanes.
template <int G>
__device__ __forceinline__ void piece_totals(const float (&o)[8][4], float m, float l, float* ob,
                                             int lane) {
  constexpr int D = kMmaD;
  const int g = lane >> 2, t = lane & 3;
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  // head h = column h (hi) + column G + h (lo): for G = 4 the lo columns
  // sit two lanes up, for G = 2 one lane up, for G = 1 in the same lane
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    float r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (G == 1) r[u] = o[mt][u & 2] + o[mt][(u & 2) + 1];
      else r[u] = o[mt][u] + __shfl_xor_sync(0xffffffffu, o[mt][u], G == 4 ? 2 : 1);
    }
    const int d0 = 16 * mt + g;
    if (G == 1) {
      if (t == 0) { ob[d0] = r[0]; ob[d0 + 8] = r[2]; }
    } else if (2 * t < G) {
      ob[(2 * t) * D + d0] = r[0];
      ob[(2 * t + 1) * D + d0] = r[1];
      ob[(2 * t) * D + d0 + 8] = r[2];
      ob[(2 * t + 1) * D + d0 + 8] = r[3];
    }
  }
  if (g < G && t == 0) {
    ob[G * D + g] = m;
    ob[G * D + G + g] = l;
  }
}

// Merge the shared-prefix states of (request i, kv head h) -- one per prefix
// range, written by prefix_attn_kernel -- into a piece's totals in ob.
template <int G>
__device__ __forceinline__ void merge_prefix(const PoolDev& p, int i, int h, float* ob, int lane) {
  constexpr int D = kMmaD, PW = G * (D + 4);
  const int nr = p.prefix_batch ? p.pranges[i] : 0;
  if (nr <= 0) return;
  const float* ps = p.pstate + ((size_t)i * p.Hk + h) * p.max_pranges * PW;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float m = ob[G * D + g], l = ob[G * D + G + g];
    float4 acc = *reinterpret_cast<const float4*>(ob + g * D + 4 * lane);
    for (int r = 0; r < nr; ++r) {
      const float* pr = ps + (size_t)r * PW + g * (D + 4);
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(pr + D));
      const float4 ov = __ldcg(reinterpret_cast<const float4*>(pr) + lane);
      if (ml.x == -INFINITY) continue;
      const float mn = fmaxf(m, ml.x);
      const float al = (m == -INFINITY) ? 0.f : exp2f(m - mn);
      const float be = exp2f(ml.x - mn);
      l = l * al + ml.y * be;
      acc.x = acc.x * al + ov.x * be; acc.y = acc.y * al + ov.y * be;
      acc.z = acc.z * al + ov.z * be; acc.w = acc.w * al + ov.w * be;
      m = mn;
    }
    __syncwarp();
    *reinterpret_cast<float4*>(ob + g * D + 4 * lane) = acc;
    if (lane == 0) { ob[G * D + g] = m; ob[G * D + G + g] = l; }
  }
  __syncwarp();
}

// ----------------------------------------------------------- attention ---
// ------------------------------------------------------ cut segments ---
//
// The output of a cut (request, head) from its pieces' states (workers
// w_first .. w_last of si), its shared-prefix range states and the staged
// token: the states are combined with weights 2^(m_k - max m), then the
// staged token is merged in and the result normalised and stored.  Every
// state must be final and visible (the caller orders it).
template <int G>
__device__ __forceinline__ void merge_segment(const PoolDev& p, int layer, int i, int h, int slot,
                                              int4 si, __nv_bfloat16* __restrict__ out, int lane) {
  constexpr int D = kMmaD, PW = G * (D + 4);
  const int64_t w_first = si.x, w_last = si.y;
  const bool first_is_second = si.z != 0;  // the first worker's second state slot
  const int nparts = (int)(w_last - w_first + 1);
  auto part_of = [&](int k) -> const float* {
    const int64_t wk = w_first + k;
    const int ps = (k == 0 && first_is_second) ? 1 : 0;
    return p.partials + (size_t)(wk * 2 + ps) * PW;
  };
  // every lane holds dims 4*lane .. 4*lane+3 of each head: 16-byte loads of
  // the states, 8-byte loads and stores of the bf16 rows
  const size_t srow = (((size_t)slot * p.L + layer) * p.Hk + h) * 2;
  const uint2 vraw = __ldcg(reinterpret_cast<const uint2*>(p.staging + (srow + 1) * D * 2) + lane);
  const float vs[4] = {__uint_as_float(vraw.x << 16), __uint_as_float(vraw.x & 0xffff0000u),
                       __uint_as_float(vraw.y << 16), __uint_as_float(vraw.y & 0xffff0000u)};
  float sst[G];
#pragma unroll
  for (int g = 0; g < G; ++g) sst[g] = __ldcg(p.sstage + (i * p.Hk + h) * 4 + g);
  float mmax[G], lsum[G], acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    mmax[g] = -INFINITY;
    lsum[g] = 0.f;
    acc[g][0] = acc[g][1] = acc[g][2] = acc[g][3] = 0.f;
  }
  // online merge over the parts, four at a time with all their loads issued
  // first: the workers' states, then the shared-prefix ranges' states
  constexpr int CH = 4;
  const int nr = p.prefix_batch ? p.pranges[i] : 0;
  const float* pst = p.pstate + ((size_t)i * p.Hk + h) * p.max_pranges * PW;
  auto part_or_prefix = [&](int k) -> const float* {
    return k < nparts ? part_of(k) : pst + (size_t)(k - nparts) * PW;
  };
  const int ntot = nparts + nr;
  for (int base = 0; base < ntot; base += CH) {
    float2 ml[CH][G];
    float4 ov[CH][G];
#pragma unroll
    for (int u = 0; u < CH; ++u) {
      const bool ok = base + u < ntot;
      const float* pk = part_or_prefix(ok ? base + u : base);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        ml[u][g] = ok ? __ldcg(reinterpret_cast<const float2*>(pk + g * (D + 4) + D))
                      : make_float2(-INFINITY, 0.f);
        ov[u][g] = ok ? __ldcg(reinterpret_cast<const float4*>(pk + g * (D + 4)) + lane)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < CH; ++u) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mk = ml[u][g].x;
        if (mk == -INFINITY) continue;
        const float mn = fmaxf(mmax[g], mk);
        const float al = (mmax[g] == -INFINITY) ? 0.f : exp2f(mmax[g] - mn);
        const float be = exp2f(mk - mn);
        lsum[g] = lsum[g] * al + ml[u][g].y * be;
        acc[g][0] = acc[g][0] * al + ov[u][g].x * be;
        acc[g][1] = acc[g][1] * al + ov[u][g].y * be;
        acc[g][2] = acc[g][2] * al + ov[u][g].z * be;
        acc[g][3] = acc[g][3] * al + ov[u][g].w * be;
        mmax[g] = mn;
      }
    }
  }
  // the staged token, normalisation, store
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float mn = fmaxf(mmax[g], sst[g]);
    const float al = (mmax[g] == -INFINITY) ? 0.f : exp2f(mmax[g] - mn);
    const float be = exp2f(sst[g] - mn);
    const float inv = 1.0f / (lsum[g] * al + be);
    const __nv_bfloat162 lo = __floats2bfloat162_rn((acc[g][0] * al + be * vs[0]) * inv,
                                                    (acc[g][1] * al + be * vs[1]) * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn((acc[g][2] * al + be * vs[2]) * inv,
                                                    (acc[g][3] * al + be * vs[3]) * inv);
    uint2 wv;
    wv.x = *reinterpret_cast<const uint32_t*>(&lo);
    wv.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(out + ((size_t)i * p.Hq + h * G + g) * D)[lane] = wv;
  }
}

template <int G, int S>
__global__ void __launch_bounds__(kMmaWarps * 32)
attn_mma_kernel(const __grid_constant__ CUtensorMap kvblk, PoolDev p, int layer,
                const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ knew,
                const __nv_bfloat16* __restrict__ vnew, __nv_bfloat16* __restrict__ out) {
  static_assert(G == 1 || G == 2 || G == 4, "G");
  constexpr int D = kMmaD;
  // The stages must start on 1024-byte boundaries (128-byte swizzle).  A
  // CTA's dynamic shared memory starts 1024-byte aligned when, as here, the
  // kernel declares no static shared memory; no slack is allocated for it
  // (that keeps three CTAs per SM), and a misaligned base is reported below
  // instead of run.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2;
  uint8_t* ring = smem + (size_t)warp * S * kMmaStageB;
  float* ob = reinterpret_cast<float*>(smem + (size_t)kMmaWarps * S * kMmaStageB) + warp * kWarpBufFloats;
  float* obx = ob + kObFloats;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kMmaWarps * S * kMmaStageB +
                                               (size_t)kMmaWarps * kWarpBufFloats * 4) + warp * S;

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
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) set_status(p, GP_ST_SMEM_ALIGN, (int)(smem_u32(smem_raw) & 1023u));
    return;
  }
  if (n <= 0 || w >= Weff) return;  // warp-uniform: warps never synchronise
  const int start = p.wblk[w], end = p.wblk[w + 1];  // the plan's (weighted) share
  if (start >= end) return;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // ---- the warp's item sequence: the blocks of its range, with a meta item
  // in front of every piece.  Item c lives in stage c % S.  Producer state:
  Cursor pc;
  cursor_start(p, w, pc);
  PlanWin pwin, cwin;
  PageWinAhead win;
  const int first_seg = pc.i * p.Hk + pc.h;
  const int i_first = pc.i, h_first = pc.h;
  (void)plan_at(p, pwin, pc.i, n, lane);  // lets the first page window see the next request
  // the consumer starts where the producer starts: its cursor and plan window
  // are copies (no loads after the wait)
  const Cursor c_first = pc;
  cwin = pwin;
  int pblk = start;       // next block to issue
  bool pmeta = false;     // next item is a meta item
  // Ring bookkeeping in 32 bits: the producer's next stage ps; items issued
  // and not yet released (item 0, the first meta, is reserved: it is issued
  // after the wait); the consumer's stage cs and phase cph.
  int ps = 1, inflight = 1;
  auto emit = [&](bool allow_meta) -> bool {
    if (pblk >= end && !pmeta) return false;
    if (pmeta && !allow_meta) return false;
    const int s = ps;
    uint8_t* st = ring + s * kMmaStageB;
    if (pmeta) {
      const PlanEntry e = plan_at(p, pwin, pc.i, n, lane);
      if (lane == 0) {
        fence_proxy_async_smem();
        issue_meta<G>(p, layer, pc.i, pc.h, e.slot, e.pos, q, knew, vnew, st, &bars[s]);
      }
      pmeta = false;
    } else {
      const int page = page_of_ahead(p, win, pwin, pc, n, lane);
      if (lane == 0) {
        fence_proxy_async_smem();
        issue_block_tma(p, &kvblk, layer, pc, page, st, &bars[s]);
      }
      if (++pblk < end) {
        walk_next(p, pwin, pc, n, lane);
        if (pc.blk == 0) pmeta = true;
      }
    }
    ps = (ps + 1 == S) ? 0 : ps + 1;
    ++inflight;
    return true;
  };
  // prologue: the first meta item's state half, then blocks only (meta
  // items read this step's inputs)
  {
    const PlanEntry e = plan_at(p, pwin, i_first, n, lane);
    if (lane == 0) issue_meta_state<G>(p, layer, h_first, e.slot, e.pos, ring, &bars[0]);
  }
  while (inflight < S && emit(false)) {}
  // The next GP_PREF_L2 blocks of the range into L2 (pages are final before
  // the step): the blocks issued right after the wait then come from L2,
  // fetched while the previous kernels finish.
  {
    Cursor pa = pc;
    PlanWin wa = pwin;
    PageWinAhead wina = win;
    for (int k = 0, b2 = pblk; k < GP_PREF_L2 && b2 < end; ++k) {
      const int page = page_of_ahead(p, wina, wa, pa, n, lane);
      if (lane == 0) prefetch_block_l2(p, layer, pa, page);
      if (++b2 < end) walk_next(p, wa, pa, n, lane);
    }
  }
  // The first piece's input rows into L2 as well.  They may still be being
  // written by the kernel before this one; a prefetch only warms L2, which
  // every writer updates, and nothing is read from them before the wait.
  if (lane == 0) prefetch_inputs_l2<G>(p, i_first, h_first, q, knew, vnew);
  // The step's inputs, the split-K scratch and the outputs belong to earlier
  // kernels: wait for them.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (lane == 0) issue_meta_inputs<G>(p, i_first, h_first, q, knew, vnew, ring, &bars[0]);
  while (inflight < S && emit(true)) {}

  const uint32_t ring_u32 = smem_u32(ring);
  const LdsmOffsets lofs = ldsm_offsets(lane);

  bool failed = false;
  int cs = 0;         // the consumer's stage
  uint32_t cph = 0;   // and its phase
  auto wait_item = [&](int slot) -> bool {
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[cs], cph, kWaitLimitNs));
    if (!ok && lane == 0) set_status(p, GP_ST_TIMEOUT, slot);
    return ok;
  };
  auto release_item = [&]() {
    __syncwarp();
    if (++cs == S) { cs = 0; cph ^= 1u; }
    --inflight;
    if (inflight < S) emit(true);
  };

  Cursor cc = c_first;
  int j = start;
  while (j < end && !failed) {
    const int i = cc.i, h = cc.h, slot = cc.slot, nb = cc.nb;
    const int len = (nb - cc.blk < end - j) ? nb - cc.blk : end - j;
    const bool full = (cc.blk == 0) && (len == nb);
    const PlanEntry pe = plan_at(p, cwin, i, n, lane);
    const int R = pe.R;
    const bool score = (pe.flags & kPlanScore) != 0;

    // ---- operand rows, and the once-per-(request, head) duties
    uint32_t afr[8][4];
    {
      if (!wait_item(slot)) { failed = true; break; }
      const uint8_t* st = ring + cs * kMmaStageB;
      PieceIn in;
      in.q = reinterpret_cast<const __nv_bfloat16*>(st + kMetaQ);
      in.k = reinterpret_cast<const __nv_bfloat16*>(st + kMetaK);
      in.v = reinterpret_cast<const __nv_bfloat16*>(st + kMetaV);
      in.s = reinterpret_cast<const float*>(st + kMetaS);
      in.c32 = reinterpret_cast<const float*>(st + kMetaC32);
      in.s32 = reinterpret_cast<const float*>(st + kMetaS32);
      in.c32lo = reinterpret_cast<const float*>(st + kMetaC32lo);
      in.s32lo = reinterpret_cast<const float*>(st + kMetaS32lo);
      in.c64 = reinterpret_cast<const double*>(st + kMetaC64);
      in.s64 = reinterpret_cast<const double*>(st + kMetaS64);
      float* sf = reinterpret_cast<float*>(ring + cs * kMmaStageB + kMetaSF);
      in.sf = sf;
      if (score || cc.blk == 0) {  // the folded summaries are needed
        fold_rows<G>(p, in, pe.flags, lane, sf);
        __syncwarp();
      }
      build_rows<G>(p, in, pe.flags, lane, afr);
      if (cc.blk == 0) segment_duties<G>(p, layer, i, h, slot, pe.flags, in, obx, lane);
      release_item();
    }
    float* lgS = p.logits + ((((size_t)slot * p.L + layer) * p.Hk + h) * 2) * p.logit_width;
    float* lgX = lgS + (g & 1) * p.logit_width;

    float m = -INFINITY, l = 0.f;
    // O^T: o[mt][0..1] = dims 16mt + g, columns 2t, 2t+1; o[mt][2..3] = dims + 8
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    for (int k = 0; k < len; ++k, ++j) {
      if (!wait_item(slot)) { failed = true; break; }
      const uint32_t sK = ring_u32 + (uint32_t)cs * kMmaStageB;
      const int t0 = pe.tb + (cc.blk + (int)k) * kBlockTok;
      attend_block<G>(afr, o, m, l, sK, t0, R - t0, score, lgX, lofs, lane);
      release_item();
    }
    if (failed) break;

    // ---- piece totals into the warp buffer: ob[g][dim], m[g], l[g]
    piece_totals<G>(o, m, l, ob, lane);
    __syncwarp();
    if (full) {
      merge_prefix<G>(p, i, h, ob, lane);  // the shared prefix, attended beforehand
      finish_mma<G>(p, i, h, out, ob, obx, lane);
    } else {
      // a cut (request, head): leave this piece's state for combine_kernel
      const int seg = i * p.Hk + h;
      const int pslot = (seg == first_seg) ? 0 : 1;
      constexpr int PW = G * (D + 4);  // per head: D outputs, m, l, 2 pad (16-byte rows)
      float* part = p.partials + (size_t)(w * 2 + pslot) * PW;
      for (int x = lane; x < G * D; x += 32) part[(x / D) * (D + 4) + (x % D)] = ob[x];
      if (lane < 2 * G) part[(lane % G) * (D + 4) + D + lane / G] = ob[G * D + lane];
    }
    __syncwarp();  // the buffers are reused by the next piece
    if (j < end) {  // next piece: block 0 of the following (request, head)
      cc.blk = cc.nb - 1;
      walk_next(p, cwin, cc, n, lane);
    }
  }
  if (failed) {
    // let the copies this warp has in flight land before the CTA may exit
    for (; inflight > 0; --inflight) {
      (void)mbar_wait_bounded(&bars[cs], cph, kWaitLimitNs);
      if (++cs == S) { cs = 0; cph ^= 1u; }
    }
  }
}

// ------------------------------------------------------------- combine ---
//
// One warp per (request, kv head) of the step.  A (request, head) whose
// blocks were cut between several attention workers is merged here
// (merge_segment), after the attention kernel has completed, so no worker
// waits for another.
template <int G>
__global__ void __launch_bounds__(kSmallWarps * 32)
combine_kernel(PoolDev p, int layer, __nv_bfloat16* __restrict__ out) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // which workers cut this (request, head): from the plan, final before the step
  const int n = p.plan_misc[0];
  const int gw = blockIdx.x * kSmallWarps + warp;
  if (gw >= n * p.Hk) return;
  const int i = gw / p.Hk, h = gw % p.Hk;
  const int slot = p.plan_slot[i];
  const int4 si = p.seginfo[gw];   // first and last worker of this (request, head)
  if (si.x == si.y) return;        // finished by the attention kernel
  // the workers' states and the staged token come from earlier kernels
  asm volatile("griddepcontrol.wait;" ::: "memory");
  merge_segment<G>(p, layer, i, h, slot, si, out, lane);
}

// ------------------------------------------------------ shared prefixes ---
//
// prefix_attn_kernel: the attention of the step's requests over the shared
// prefixes they use, computed once per group instead of once per request.
// A unit is (prefix, chunk of up to kPrefChunk of its members in this step,
// kv head, range of kPrefRangeBlocks 16-token blocks).  The CTA's four warps
// share one ring of K/V blocks, so each prefix block is read from HBM once
// per chunk; warp w runs members w and w + 4 through the same tensor-core
// steps as the attention kernel (attend_block).  Each member leaves, per
// range, its unnormalised output, running max (log2 domain) and sum per
// query head in pstate[member][head][range]; the attention kernel (uncut
// segments) or combine_kernel (cut ones) merges them.  A member at a
// boundary also gets its summary scores of the prefix tokens.  Every wait is
// bounded and on the CTA's own copies.
constexpr int kPrefWarps = 4;
constexpr int kPrefStages = 3;
// per member: q rows [G][kQPitch] bf16, the summaries before the step, the
// rotary rows of its position (fp32), the summaries after the fold
constexpr int kPmQ = 0, kPmS = 1088, kPmC32 = 2112, kPmS32 = 2368, kPmSF = 2624;
constexpr int kPrefMemberB = 3648;

size_t prefix_smem_bytes() {
  return (size_t)kPrefStages * kMmaStageB + (size_t)kPrefWarps * 2 * kPrefMemberB +
         (size_t)kPrefWarps * kObFloats * 4 + (size_t)kPrefStages * 8;
}

template <int G>
__global__ void __launch_bounds__(kPrefWarps * 32)
prefix_attn_kernel(const __grid_constant__ CUtensorMap kvblk, PoolDev p, int layer,
                   const __nv_bfloat16* __restrict__ q) {
  constexpr int D = kMmaD, S = kPrefStages, PW = G * (D + 4);
  // stages on 1024-byte boundaries (128-byte swizzle); see attn_mma_kernel
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* const after_ring = smem_raw + (size_t)S * kMmaStageB;
  uint8_t* mbuf = after_ring + (size_t)warp * 2 * kPrefMemberB;
  float* ob = reinterpret_cast<float*>(after_ring + (size_t)kPrefWarps * 2 * kPrefMemberB) +
              warp * kObFloats;
  uint64_t* bars = reinterpret_cast<uint64_t*>(after_ring + (size_t)kPrefWarps * 2 * kPrefMemberB +
                                               (size_t)kPrefWarps * kObFloats * 4);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) set_status(p, GP_ST_SMEM_ALIGN, (int)(smem_u32(smem_raw) & 1023u));
    return;
  }
  const int units = p.plan_misc[3];  // final before the step's first attention launch
  if ((int)blockIdx.x >= units) return;
  // the units' prefix table, once per CTA (final before the step's first launch)
  __shared__ int s_ucum[kMaxPrefixBatch + 1];
  const int np = p.max_prefixes;
  for (int k = threadIdx.x; k <= np; k += blockDim.x) s_ucum[k] = p.unit_cum[k];
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  // q, the summaries and the score rows belong to earlier kernels
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t ring_u32 = smem_u32(ring);
  const LdsmOffsets lofs = ldsm_offsets(lane);
  int64_t issued = 0, used = 0;  // ring items over the CTA's life (issued: thread 0)
  bool failed = false;
  for (int u = blockIdx.x; u < units && !failed; u += gridDim.x) {
    // the unit: the prefix whose units contain u, then chunk, head, range
    int lo = 0, hi = np - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_ucum[mid] <= u) lo = mid; else hi = mid - 1;
    }
    const int pid = lo;
    const int npb = p.prefix[pid].len / kBlockTok;
    const int nr = (npb + kPrefRangeBlocks - 1) / kPrefRangeBlocks;
    int local = u - s_ucum[pid];
    const int r = local % nr;
    local /= nr;
    const int h = local % p.Hk;
    const int m0 = (local / p.Hk) * kPrefChunk;
    const int cs = min(kPrefChunk, p.pref_cnt[pid] - m0);
    const int b0 = r * kPrefRangeBlocks;
    const int nblk = min(npb - b0, kPrefRangeBlocks);
    const int32_t* ppages = p.prefix_pages + (size_t)pid * p.max_prefix_pages;
    auto issue = [&](int b) {  // thread 0: block b of the prefix into the next stage
      const int s = (int)(issued % S);
      int page = ppages[(b * kBlockTok) / p.P];
      if ((unsigned)page >= (unsigned)p.num_pages) {
        set_status(p, GP_ST_BAD_PAGE, page);
        page = 0;
      }
      uint8_t* st = ring + s * kMmaStageB;
      fence_proxy_async_smem();
      mbar_expect_tx(&bars[s], kMmaStageB);
      tma_load_block(st, &kvblk, (b * kBlockTok) % p.P, (page * p.L + layer) * p.Hk + h, &bars[s]);
      ++issued;
    };
    if (threadIdx.x == 0)
      for (int b = 0; b < min(nblk, S); ++b) issue(b0 + b);
    // this warp's members: chunk positions warp and warp + kPrefWarps
    int mi[2], mslot[2], mflags[2];
    bool has[2];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int k = warp + kPrefWarps * kk;
      has[kk] = k < cs;
      mi[kk] = has[kk] ? p.pmem[p.pref_off[pid] + m0 + k] : 0;
      mslot[kk] = has[kk] ? p.plan_slot[mi[kk]] : 0;
      mflags[kk] = has[kk] ? p.plan_flags[mi[kk]] : 0;
      if (!has[kk]) continue;
      uint8_t* mb = mbuf + kk * kPrefMemberB;
      for (int x = lane; x < G * 16; x += 32) {  // q rows, 16 chunks of 16 bytes each
        const int row = x >> 4, c = x & 15;
        *reinterpret_cast<uint4*>(mb + kPmQ + row * kQPitch * 2 + c * 16) =
            *reinterpret_cast<const uint4*>(q + ((size_t)mi[kk] * p.Hq + h * G + row) * D + c * 8);
      }
      const float4* srow = reinterpret_cast<const float4*>(
          p.summary + ((((size_t)mslot[kk] * p.L + layer) * p.Hk + h) * 2) * D);
      for (int x = lane; x < 2 * D / 4; x += 32) reinterpret_cast<float4*>(mb + kPmS)[x] = srow[x];
      if (p.rope) {  // cos in lanes 0-15, sin in lanes 16-31 (D/2 floats each)
        const int pos_k = p.plan_pos[mi[kk]];
        const float4* src = reinterpret_cast<const float4*>(lane < 16 ? rope_c32(p, pos_k) : rope_s32(p, pos_k));
        reinterpret_cast<float4*>(mb + (lane < 16 ? kPmC32 : kPmS32))[lane & 15] = src[lane & 15];
      }
    }
    __syncwarp();
    uint32_t afr[2][8][4];
    float* lg[2];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint8_t* mb = mbuf + kk * kPrefMemberB;
      PieceIn in;
      in.q = reinterpret_cast<const __nv_bfloat16*>(mb + kPmQ);
      in.k = nullptr;
      in.v = nullptr;
      in.s = reinterpret_cast<const float*>(mb + kPmS);
      in.c32 = reinterpret_cast<const float*>(mb + kPmC32);
      in.s32 = reinterpret_cast<const float*>(mb + kPmS32);
      in.c32lo = nullptr;
      in.s32lo = nullptr;
      in.c64 = nullptr;
      in.s64 = nullptr;
      in.sf = reinterpret_cast<float*>(mb + kPmSF);
      if (has[kk] && (mflags[kk] & kPlanScore)) {  // the summaries after this step's fold
        fold_rows<G>(p, in, mflags[kk], lane, reinterpret_cast<float*>(mb + kPmSF));
        __syncwarp();
      }
      if (has[kk]) {
        build_rows<G>(p, in, mflags[kk], lane, afr[kk]);
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) afr[kk][c][0] = afr[kk][c][1] = afr[kk][c][2] = afr[kk][c][3] = 0u;
      }
      lg[kk] = p.logits + ((((size_t)mslot[kk] * p.L + layer) * p.Hk + h) * 2) * p.logit_width +
               ((lane >> 2) & 1) * p.logit_width;
    }
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[2][8][4];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[kk][mt][0] = o[kk][mt][1] = o[kk][mt][2] = o[kk][mt][3] = 0.f;
    for (int jb = 0; jb < nblk; ++jb) {
      const int s = (int)(used % S);
      const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)((used / S) & 1), kWaitLimitNs);
      if (__syncthreads_or(!ok)) {
        if (threadIdx.x == 0) set_status(p, GP_ST_TIMEOUT, -1);
        failed = true;
        break;
      }
      const uint32_t sK = ring_u32 + (uint32_t)s * kMmaStageB;
      const int t0 = (b0 + jb) * kBlockTok;  // prefix tokens: every one resident
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        if (has[kk])  // warp-uniform
          attend_block<G>(afr[kk], o[kk], m[kk], l[kk], sK, t0, 1 << 30,
                          (mflags[kk] & kPlanScore) != 0, lg[kk], lofs, lane);
      __syncthreads();  // every warp is done with stage s
      ++used;
      if (threadIdx.x == 0 && jb + S < nblk) issue(b0 + jb + S);
    }
    if (failed) break;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      if (!has[kk]) continue;
      piece_totals<G>(o[kk], m[kk], l[kk], ob, lane);
      __syncwarp();
      float* dst = p.pstate + (((size_t)mi[kk] * p.Hk + h) * p.max_pranges + r) * PW;
      for (int x = lane; x < G * D; x += 32) dst[(x / D) * (D + 4) + (x % D)] = ob[x];
      if (lane < 2 * G) dst[(lane % G) * (D + 4) + D + lane / G] = ob[G * D + lane];
      __syncwarp();
    }
    __syncthreads();  // the member buffers are reused by the next unit
  }
  if (failed && threadIdx.x == 0) {
    // let this CTA's copies in flight land before it exits
    for (int64_t c = used; c < issued; ++c)
      (void)mbar_wait_bounded(&bars[c % S], (uint32_t)((c / S) & 1), kWaitLimitNs);
  }
}

size_t mma_smem_bytes() {
  return (size_t)kMmaWarps * kMmaStages * kMmaStageB + (size_t)kMmaWarps * kWarpBufFloats * 4 +
         (size_t)kMmaWarps * kMmaStages * 8;
}

// Both kernels are launched as programmatic dependents of the previous
// kernel in the stream (see griddepcontrol in the kernels): the attention
// kernel's prologue (cursors, first K/V copies) overlaps what runs before it.
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
                                bool prefix, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaError_t e = cudaSuccess;
  if (prefix) {  // the shared prefixes first; the attention kernel merges their states
    cudaLaunchConfig_t c0 = pdl_config(attr, dim3(grid), dim3(kPrefWarps * 32), prefix_smem_bytes(), st);
    e = cudaLaunchKernelEx(&c0, prefix_attn_kernel<G>, *map, p, layer, (const __nv_bfloat16*)q);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t c1 = pdl_config(attr, dim3(grid), dim3(kMmaWarps * 32), mma_smem_bytes(), st);
  e = cudaLaunchKernelEx(&c1, attn_mma_kernel<G, kMmaStages>, *map, p, layer,
                                     (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                     (const __nv_bfloat16*)v, (__nv_bfloat16*)out);
  if (e != cudaSuccess) return e;
  const int warps = n * p.Hk;
  cudaLaunchConfig_t c2 = pdl_config(attr, dim3((warps + kSmallWarps - 1) / kSmallWarps),
                                     dim3(kSmallWarps * 32), 0, st);
  return cudaLaunchKernelEx(&c2, combine_kernel<G>, p, layer, (__nv_bfloat16*)out);
}

int attention_mma_launches(bool prefix) { return prefix ? 3 : 2; }

template <int G>
static cudaError_t occupancy_mma_t(int* blocks) {
  auto kern = attn_mma_kernel<G, kMmaStages>;
  const size_t smem = mma_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefix_attn_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)prefix_smem_bytes());
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, kern, kMmaWarps * 32, smem);
}

int mma_warps_per_cta() { return kMmaWarps; }

// Two launches, attn_mma_kernel then combine_kernel, or three with the
// shared-prefix kernel in front of them.
cudaError_t launch_attention_mma(const PoolDev& p, const CUtensorMap* map, int layer, int n,
                                 const void* q, const void* k, const void* v, void* out, int grid,
                                 bool prefix, cudaStream_t st) {
  if (p.G == 1) return launch_mma_t<1>(p, map, layer, n, q, k, v, out, grid, prefix, st);
  if (p.G == 2) return launch_mma_t<2>(p, map, layer, n, q, k, v, out, grid, prefix, st);
  if (p.G == 4) return launch_mma_t<4>(p, map, layer, n, q, k, v, out, grid, prefix, st);
  return cudaErrorInvalidValue;
}

cudaError_t attention_mma_occupancy(const PoolDev& p, int* blocks) {
  if (p.G == 1) return occupancy_mma_t<1>(blocks);
  if (p.G == 2) return occupancy_mma_t<2>(blocks);
  if (p.G == 4) return occupancy_mma_t<4>(blocks);
  return cudaErrorInvalidValue;
}

}  // namespace gp
