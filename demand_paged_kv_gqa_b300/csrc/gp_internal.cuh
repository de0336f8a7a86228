// gp_internal.cuh -- device-side view of a GrowPage pool and shared helpers.
//
// Everything here is private to libgrowpage.so.  The public contract is
// include/growpage.h; this file mirrors its structs and adds the scratch
// regions (per-step plan, split partials, move lists) the kernels use.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "growpage.h"

namespace gp {

constexpr int kBlockTok = 16;     // tokens per attention block (one bulk-copy unit)
constexpr int kAttnWarps = 4;     // warps per attention CTA (independent workers)
constexpr int kMaxWorkersBound = 160 * 8 * kAttnWarps;  // sizing bound

enum Decision : int32_t {
  kNone = 0, kGrow = 1, kCompact = 2, kCompactDenied = 3, kStarved = 4, kShrink = 5
};

// Flags of a request in the current step's plan.
constexpr int32_t kPlanBoundary = 1;  // all private pages full at step start
constexpr int32_t kPlanFirst = 2;     // first decode step: summaries start at qbar
constexpr int32_t kPlanScore = 4;     // boundary in GROWPAGE mode: score summaries

struct PoolDev {
  // configuration
  int32_t L, Hq, Hk, D, G, P;
  int32_t P_log2;         // log2(P) when P is a power of two, else -1
  int32_t num_pages, max_req, max_pages_per_req, max_prefixes, max_prefix_pages;
  int32_t block_width, logit_width, max_seq_len, dtype, mode, recent_window;
  int32_t num_workers;
  float beta_s, beta_l, top_p, tau;
  float random_grow_rate;
  int32_t rope;  // 1: rotary embedding on
  int32_t elem_bytes;
  uint64_t page_bytes, layer_bytes, head_bytes, half_bytes;  // kv strides
  // public regions
  uint8_t* kv;
  int32_t* tok_pos;
  int32_t* block;
  gp_req_meta* req;
  float* summary;
  uint8_t* staging;
  float* logits;
  int32_t* wset;
  int32_t* free_stack;
  gp_ctrl* ctrl;
  gp_prefix_meta* prefix;
  int32_t* prefix_pages;
  // RoPE rows, one per position (rope_row_bytes = 16 d): cos, sin fp32 [d/2]
  // each (the fp64 values rounded once), their fp32 residuals fp32(x64 - x32)
  // (x32 + residual carries ~48 bits), then cos, sin fp64 [d/2] each
  const uint8_t* rope_rows;
  int32_t rope_row_bytes;
  // scratch: per-step plan
  int32_t* plan_slot;     // [max_req] slot of request i
  int32_t* plan_R;        // [max_req] resident tokens (prefix + private)
  int32_t* plan_nb;       // [max_req] attention blocks (>= 1)
  int32_t* plan_cum;      // [max_req + 1] prefix sums of plan_nb
  int32_t* plan_flags;    // [max_req]
  int32_t* plan_commit;   // [max_req] private slot receiving the staged token
  int32_t* plan_cpos;     // [max_req] its position
  int32_t* plan_dec;      // [max_req] decision of this step
  int32_t* plan_bnd;      // [max_req] indices i of scoring boundaries
  int32_t* plan_pos;      // [max_req] position of the step's token
  int32_t* plan_misc;     // [0] n, [1] n scoring boundaries, [2] total blocks/Hk,
                          // [3] shared-prefix units
  int32_t* plan_base;     // [max_req] resident tokens the attention kernel skips (a
                          // shared prefix handled by prefix_attn_kernel), else 0
  long long* plan_delta;  // [max_req] Delta accumulators
  // scratch: attention split-K
  float* partials;        // [num_workers][2][G][D + 2]
  int32_t* seg_count;     // [max_req][Hk]
  float* summary_next;    // [max_req][L][Hk][2][d] this step's folded summaries
                          // of the requests at a boundary (bf16 attention path),
                          // copied over `summary` by the commit kernel
  float* sstage;          // [max_req][Hk][4] each query head's score against the
                          // staged token (log2 domain)
  int32_t summary_via_next;  // 1: the attention kernel writes the folds of requests
                             // at a boundary to summary_next (bf16 path)
  int32_t* wblk;          // [kMaxWorkersBound + 1] first block of each worker's share
                          // (bf16 path; the last entry is the total)
  int4* seginfo;          // [max_req][Hk] first and last worker of each (request,
                          // head) and whether it is the first worker's second state
  int32_t seg_cost;       // extra blocks' worth of work a (request, head) start costs
  int4* wstart;           // [kMaxWorkersBound] first block of each attention worker:
                          // request index, (head << 20) | block, blocks of the
                          // segment, slot (written by the plan kernel)
  // scratch: compaction moves
  int32_t* moves;         // [max_req][L][Hk][P][2] (dst, src) private slots
  int32_t* moves_n;       // [max_req][L][Hk]
  // asynchronous boundary work: 1 while a request's boundary work of an
  // earlier step still runs on the second stream (the plan refuses it)
  int32_t* busy;          // [max_req]
  // shared prefixes (bf16 attention path): the attention over a prefix is
  // computed once per group of the step's requests that share it
  int32_t prefix_batch;   // 1: enabled
  int32_t max_pranges;    // prefix ranges per request at most
  int32_t* pmem;          // [max_req] plan indices grouped by prefix
  int32_t* pranges;       // [max_req] prefix ranges of request i (0: none)
  int32_t* pref_off;      // [max_prefixes] first member of prefix k in pmem
  int32_t* pref_cnt;      // [max_prefixes] members of prefix k in this step
  int32_t* unit_cum;      // [max_prefixes + 1] first unit of prefix k
  float* pstate;          // [max_req][Hk][max_pranges][G][D + 4] attention state of
                          // each prefix range: output, then max (log2), sum
};

// Shared-prefix work: a unit is (prefix, chunk of up to kPrefChunk members,
// kv head, range of kPrefRangeBlocks 16-token blocks).
constexpr int kPrefChunk = 8;
constexpr int kPrefRangeBlocks = 64;
constexpr int kMaxPrefixBatch = 512;  // prefixes the plan kernel groups (in shared memory)

// Which requests a boundary-phase kernel (decide, commit) handles: every
// request of the step, only those not at a boundary (their token appended on
// the pool's stream), or only those at a boundary (their boundary work on the
// second stream).
enum Part : int32_t { kPartAll = 0, kPartPlain = 1, kPartBoundary = 2 };

// ------------------------------------------------------------ helpers ---

__device__ __forceinline__ void set_status(const PoolDev& p, uint32_t bit, int32_t info) {
  uint32_t old = atomicOr(&p.ctrl->status, bit);
  if (old == 0u) atomicExch(&p.ctrl->status_info, info);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round an fp64 value once, to nearest-even, to a bfloat16 bit pattern.
// Written from the IEEE-754 definition: bf16 keeps 8 significant bits and the
// fp32 exponent range; below 2^-126 its spacing is 2^-133.
__device__ __forceinline__ uint16_t f64_to_bf16_rne(double x) {
  uint64_t u = (uint64_t)__double_as_longlong(x);
  uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
  uint64_t a = u & 0x7fffffffffffffffull;
  if (a >= 0x7ff0000000000000ull) {  // inf or nan
    if (a == 0x7ff0000000000000ull) return sign | 0x7f80u;
    return sign | 0x7fc0u;
  }
  int e = (int)(a >> 52);  // biased fp64 exponent
  if (e >= 1023 - 126) {   // normal in bf16 (or overflows)
    // keep 1 + 7 mantissa bits: drop the low 45 bits with ties-to-even
    uint64_t lsb = (a >> 45) & 1ull;
    uint64_t r = a + ((1ull << 44) - 1ull) + lsb;
    r >>= 45;                          // exponent(11) | mantissa(7)
    int eb = (int)(r >> 7) - 1023 + 127;
    if (eb >= 255) return sign | 0x7f80u;
    return sign | (uint16_t)((eb << 7) | (int)(r & 0x7f));
  }
  // subnormal bf16 range: value / 2^-133 rounded to an integer (0..128);
  // 128 is the bit pattern of the smallest normal.  Scaling by 2^133 is exact.
  double s = fabs(x) * 0x1p133;
  double r = rint(s);
  return sign | (uint16_t)r;
}

// One output of a rotate-half RoPE pair for a bf16 key, rounded once to bf16:
// the value a·c + b·w of bf16 inputs a, b and fp64 table values c, w, as the
// fp64 expression fl(fl(a·c) + fl(b·w)) followed by f64_to_bf16_rne would give
// it (w = -s for x·c - y·s, w = s for y·c + x·s), without fp64 arithmetic.
// c and w arrive as fp32 pairs (c1 + c2, w1 + w2 with c1 = fl32(c),
// c2 = fl32(c - c1), so |c - c1 - c2| <= 2^-48 |c1|).  With M = |a| + |b|:
//   - a·c1 = p1 + e1 exactly (Dekker's product via fma), b·w1 = q1 + f1;
//     s + t = p1 + q1 exactly (Knuth's two-sum);
//   - lo = t + ((e1 + f1) + (p2 + q2)), p2 = fl(a·c2), q2 = fl(b·w2): four
//     roundings of terms below 3·2^-24 M, two product roundings and the
//     dropped c, w residuals keep |s + lo - (a·c + b·w)| <= 9·2^-48 M;
//   - the fp64 expression is within 2^-52 M (1 + 2^-50) of a·c + b·w.
// So when s + lo lies more than 2^-44 M = 16·2^-48 M inside the rounding
// interval of its bf16 neighbour B (distances taken after an exact Sterbenz
// subtraction and one rounding), the fp64 expression rounds to B as well.
// Returns false otherwise (that close to a rounding boundary, tiny or huge
// inputs, non-finite values): the caller evaluates the fp64 expression.
__device__ __forceinline__ bool rope_bf16_certified(float a, float b, float c1, float c2, float w1,
                                                    float w2, uint16_t& out) {
  if (a == 0.f && b == 0.f) {
    // fl(a·c) and fl(b·w) are zeros carrying the products' signs; their sum
    // is -0 only when both are -0 (round to nearest)
    const uint32_t na = (__float_as_uint(a) ^ __float_as_uint(c1)) >> 31;
    const uint32_t nb = (__float_as_uint(b) ^ __float_as_uint(w1)) >> 31;
    out = (na & nb) ? 0x8000u : 0u;
    return true;
  }
  const float M = __fadd_rn(fabsf(a), fabsf(b));
  if (!(M >= 0x1p-60f && M <= 0x1p120f)) return false;  // NaN fails too
  // a·c1 = p1 + e1 and b·w1 = q1 + f1 exactly; a·c2, b·w2 rounded
  const float p1 = __fmul_rn(a, c1), e1 = __fmaf_rn(a, c1, -p1);
  const float q1 = __fmul_rn(b, w1), f1 = __fmaf_rn(b, w1, -q1);
  const float p2 = __fmul_rn(a, c2), q2 = __fmul_rn(b, w2);
  // s + t = p1 + q1 exactly
  const float s = __fadd_rn(p1, q1);
  const float sb = __fsub_rn(s, p1);
  const float t = __fadd_rn(__fsub_rn(p1, __fsub_rn(s, sb)), __fsub_rn(q1, sb));
  const float lo = __fadd_rn(t, __fadd_rn(__fadd_rn(e1, f1), __fadd_rn(p2, q2)));
  // hi + r = s + lo exactly
  const float hi = __fadd_rn(s, lo);
  const float hb_ = __fsub_rn(hi, s);
  const float r = __fadd_rn(__fsub_rn(s, __fsub_rn(hi, hb_)), __fsub_rn(lo, hb_));
  const float ah = fabsf(hi);
  if (!(ah >= 0x1p-100f)) return false;
  const float ar = hi < 0.f ? -r : r;  // |value| = ah + ar
  // B: |hi| rounded to nearest-even on the bf16 grid; its two neighbours
  const uint32_t hbits = __float_as_uint(ah);
  const uint32_t rb = (hbits + 0x7fffu + ((hbits >> 16) & 1u)) >> 16;
  const float B = __uint_as_float(rb << 16);
  const float up = __fmul_rn(__fadd_rn(B, __uint_as_float((rb + 1u) << 16)), 0.5f);
  const float dn = __fmul_rn(__fadd_rn(B, __uint_as_float((rb - 1u) << 16)), 0.5f);
  const float margin = __fmul_rn(M, 0x1p-44f);
  const float d_up = __fsub_rn(__fsub_rn(up, ah), ar);
  const float d_dn = __fadd_rn(__fsub_rn(ah, dn), ar);
  if (!(d_up > margin && d_dn > margin)) return false;
  out = (uint16_t)(rb | (hi < 0.f ? 0x8000u : 0u));
  return true;
}

// The parts of the RoPE row of position pos.
__device__ __forceinline__ const float* rope_c32(const PoolDev& p, int pos) {
  return reinterpret_cast<const float*>(p.rope_rows + (size_t)pos * p.rope_row_bytes);
}
__device__ __forceinline__ const float* rope_s32(const PoolDev& p, int pos) { return rope_c32(p, pos) + p.D / 2; }
__device__ __forceinline__ const float* rope_c32lo(const PoolDev& p, int pos) { return rope_c32(p, pos) + p.D; }
__device__ __forceinline__ const float* rope_s32lo(const PoolDev& p, int pos) { return rope_c32(p, pos) + 3 * (p.D / 2); }
__device__ __forceinline__ const double* rope_c64(const PoolDev& p, int pos) {
  return reinterpret_cast<const double*>(rope_c32(p, pos) + 2 * p.D);
}
__device__ __forceinline__ const double* rope_s64(const PoolDev& p, int pos) { return rope_c64(p, pos) + p.D / 2; }

template <typename T> struct ElemIO;
template <> struct ElemIO<float> {
  static __device__ __forceinline__ float load(const float* p, int i) { return p[i]; }
};
template <> struct ElemIO<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p, int i) {
    return __bfloat162float(p[i]);
  }
};

// ------------------------------------------------- mbarrier / bulk copy ---

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared, completing on an mbarrier (TMA engine).
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, "
      "0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after ~limit_ns of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && global_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------- reductions ---

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace gp
