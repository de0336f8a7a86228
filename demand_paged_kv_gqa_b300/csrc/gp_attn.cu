// gp_attn.cu -- paged GQA decode attention fused with GrowPage's summary upkeep.
//
// One launch per layer.  For every request i of the step and kv head h it
//   * rotates the step's key to the request's position in fp64 and rounds it
//     once to the storage dtype (the staged token), copies the value;
//   * folds the mean of the G query heads into the short and long summaries
//     (fp32, "GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning
//     Serving", evolve.pub review, Summary: two exponentially smoothed query
//     summaries, beta 0.9 / 0.999, kept pre-RoPE);
//   * computes softmax(RoPE(q)·K^T/sqrt(d))·V over the resident tokens
//     (shared prefix + private pages) and the staged token, for the G query
//     heads that share the kv head;
//   * at a capacity boundary, scores both summaries, rotated to the current
//     position, against every resident key (the same K pass, no re-read) and
//     writes the scores for the working-set and compaction kernels.
//
// Work decomposition (split-K, balanced): the resident tokens of every
// (request, kv head) are cut into 16-token blocks; all blocks of the step are
// laid end to end and split into equal contiguous ranges, one per warp of a
// persistent grid.  Each warp streams its blocks through a private ring of
// shared-memory stages filled by 1-D bulk copies (TMA) that complete on
// mbarriers, keeping several blocks in flight.  A (request, head) cut between
// warps is merged by the warp that finishes its last piece (atomic arrival
// counter; nobody waits).  Warps never synchronise with each other, so every
// wait in this kernel is on the warp's own copies.
#include "gp_attn_common.cuh"

namespace gp {

template <class Gm>
__device__ __forceinline__ void issue_block(const PoolDev& p, int layer, const Cursor& c,
                                            uint8_t* stage, uint64_t* bar) {
  const int t0 = c.blk * kBlockTok;
  int page = p.block[(size_t)c.slot * p.block_width + t0 / p.P];
  if ((unsigned)page >= (unsigned)p.num_pages) {
    set_status(p, GP_ST_BAD_PAGE, c.slot);
    page = 0;
  }
  const uint8_t* src = p.kv + (size_t)page * p.page_bytes + (size_t)layer * p.layer_bytes +
                       (size_t)c.h * p.head_bytes + (size_t)(t0 % p.P) * Gm::ROWB;
  mbar_expect_tx(bar, Gm::STAGEB);
  bulk_g2s(stage, src, Gm::BLKB, bar);
  bulk_g2s(stage + Gm::BLKB, src + p.half_bytes, Gm::BLKB, bar);
}

// Staged token, summary update and output of one (request, kv head), given
// the attention state over its resident tokens (all lanes hold the totals for
// their slice).
template <typename T, class Gm, int G>
__device__ __forceinline__ void finalize(const PoolDev& p, int layer, int i, int h, int slot,
                                         int pos, int flags, const T* __restrict__ q,
                                         const T* __restrict__ knew,
                                         const T* __restrict__ vnew, T* __restrict__ out,
                                         float (&m)[G], float (&l)[G],
                                         float (&o)[G][Gm::NE],
                                         const float (&qreg)[G][Gm::NE], int lane) {
  constexpr int NE = Gm::NE, D = Gm::ROWB / Gm::EB, H2 = NE / 2;
  const int sigma = lane & 7, tg = lane >> 3;
  // A1: the step's key rotated in fp64, rounded once to the storage dtype.
  float kraw[NE], vraw[NE], kst[NE];
  load_row<T, Gm>(reinterpret_cast<const uint8_t*>(knew + ((size_t)i * p.Hk + h) * D), sigma, kraw);
  load_row<T, Gm>(reinterpret_cast<const uint8_t*>(vnew + ((size_t)i * p.Hk + h) * D), sigma, vraw);
  if (p.rope) {
    const double* c64 = rope_c64(p, pos);
    const double* s64 = rope_s64(p, pos);
#pragma unroll
    for (int e = 0; e < H2; ++e) {
      const int di = dim_of<Gm>(e, sigma);
      const double c = c64[di], s = s64[di];
      const double x = (double)kraw[e], y = (double)kraw[e + H2];
      const double a = __dsub_rn(__dmul_rn(x, c), __dmul_rn(y, s));
      const double b = __dadd_rn(__dmul_rn(y, c), __dmul_rn(x, s));
      if constexpr (sizeof(T) == 2) {
        kst[e] = __uint_as_float((uint32_t)f64_to_bf16_rne(a) << 16);
        kst[e + H2] = __uint_as_float((uint32_t)f64_to_bf16_rne(b) << 16);
      } else {
        kst[e] = __double2float_rn(a);
        kst[e + H2] = __double2float_rn(b);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < NE; ++e) kst[e] = kraw[e];
  }
  const size_t srow = (((size_t)slot * p.L + layer) * p.Hk + h) * 2;
  if (tg == 0) {
    T* st = reinterpret_cast<T*>(p.staging) + srow * D;
    store_row<T, Gm>(st, sigma, kst);       // exact: kst already on the dtype grid
    store_row<T, Gm>(st + D, sigma, vraw);
  }
  // A3: merge the staged token into the attention state.
  float sst[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float a = 0.f;
#pragma unroll
    for (int e = 0; e < NE; ++e) a = fmaf(qreg[g][e], kst[e], a);
    a += __shfl_xor_sync(0xffffffffu, a, 1);
    a += __shfl_xor_sync(0xffffffffu, a, 2);
    a += __shfl_xor_sync(0xffffffffu, a, 4);
    sst[g] = a;
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float mn = fmaxf(m[g], sst[g]);
    const float al = (m[g] == -INFINITY) ? 0.f : exp2f(m[g] - mn);
    const float be = exp2f(sst[g] - mn);
    const float ll = l[g] * al + be;
    const float inv = 1.0f / ll;
    float res[NE];
#pragma unroll
    for (int e = 0; e < NE; ++e) res[e] = (o[g][e] * al + be * vraw[e]) * inv;
    if (tg == 0) store_row<T, Gm>(out + ((size_t)i * p.Hq + h * G + g) * D, sigma, res);
  }
  // A2: fold this step's query mean into both summaries (fp32, exact order).
  if (tg == 0) {
    float qb[NE];
    float qr[NE];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      load_row<T, Gm>(reinterpret_cast<const uint8_t*>(q + ((size_t)i * p.Hq + h * G + g) * D),
                      sigma, qr);
#pragma unroll
      for (int e = 0; e < NE; ++e) qb[e] = (g == 0) ? qr[e] : __fadd_rn(qb[e], qr[e]);
    }
    float* srowp = p.summary + srow * D;
    const float bS = p.beta_s, bL = p.beta_l;
    const float aS = __fsub_rn(1.0f, bS), aL = __fsub_rn(1.0f, bL);
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const int dd = dim_of<Gm>(e, sigma);
      const float qm = __fdiv_rn(qb[e], (float)G);
      float ns, nl;
      if (flags & kPlanFirst) {
        ns = qm; nl = qm;
      } else {
        ns = __fadd_rn(__fmul_rn(bS, srowp[dd]), __fmul_rn(aS, qm));
        nl = __fadd_rn(__fmul_rn(bL, srowp[D + dd]), __fmul_rn(aL, qm));
      }
      srowp[dd] = ns;
      srowp[D + dd] = nl;
    }
  }
}

template <typename T, int D, int G, int S>
__global__ void __launch_bounds__(kAttnWarps * 32)
attn_kernel(PoolDev p, int layer, const T* __restrict__ q, const T* __restrict__ knew,
            const T* __restrict__ vnew, T* __restrict__ out) {
  using Gm = Geo<T, D>;
  constexpr int NE = Gm::NE, H2 = NE / 2;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sigma = lane & 7, tg = lane >> 3;
  uint8_t* ring = smem + (size_t)warp * S * Gm::STAGEB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kAttnWarps * S * Gm::STAGEB) + warp * S;

  const int n = p.plan_misc[0];
  const int64_t Tb = (int64_t)p.plan_misc[2] * p.Hk;
  const int64_t W = (int64_t)gridDim.x * kAttnWarps;
  const int64_t Weff = W < Tb ? W : Tb;
  const int64_t w = (int64_t)blockIdx.x * kAttnWarps + warp;
  if (n <= 0 || w >= Weff) return;  // warp-uniform: warps never synchronise
  const int64_t start = (w * Tb) / Weff, end = ((w + 1) * Tb) / Weff;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // producer cursor (lane 0 issues; every lane walks the same sequence)
  Cursor pc;
  cursor_at(p, n, start, pc);
  const int first_seg = pc.i * p.Hk + pc.h;
  {
    int64_t b = start;
    for (int s = 0; s < S && b < end; ++s, ++b) {
      if (lane == 0) issue_block<Gm>(p, layer, pc, ring + s * Gm::STAGEB, &bars[s]);
      if (b + 1 < end) cursor_next(p, pc);
    }
  }
  int64_t issued = start + S < end ? start + S : end;

  const float qscale = 1.4426950408889634f / sqrtf((float)D);  // log2(e)/sqrt(d)
  const float sscale = 1.0f / sqrtf((float)D);
  bool failed = false;
  Cursor cc;
  cursor_at(p, n, start, cc);
  int64_t j = start;
  while (j < end && !failed) {
    // ---- begin a piece: blocks [cc.blk, cc.blk + len) of (cc.i, cc.h)
    const int i = cc.i, h = cc.h, slot = cc.slot, nb = cc.nb;
    const int64_t len = ((int64_t)(nb - cc.blk) < end - j) ? (int64_t)(nb - cc.blk) : end - j;
    const bool full = (cc.blk == 0) && (len == nb);
    const int R = p.plan_R[i];
    const int flags = p.plan_flags[i];
    const bool score = (flags & kPlanScore) != 0;
    const int pos = p.req[slot].pos;

    float qreg[G][NE];
#pragma unroll
    for (int g = 0; g < G; ++g)
      load_row<T, Gm>(reinterpret_cast<const uint8_t*>(q + ((size_t)i * p.Hq + h * G + g) * D),
                      sigma, qreg[g]);
    float sreg[2][NE];
#pragma unroll
    for (int e = 0; e < NE; ++e) { sreg[0][e] = 0.f; sreg[1][e] = 0.f; }
    if (score) {
      // A2 ahead of scoring: the summaries this step folds in (recomputed
      // identically by the warp that finalises, which also stores them).
      const float* srowp = p.summary + (((size_t)slot * p.L + layer) * p.Hk + h) * 2 * D;
      const float bS = p.beta_s, bL = p.beta_l;
      const float aS = __fsub_rn(1.0f, bS), aL = __fsub_rn(1.0f, bL);
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        float qb = qreg[0][e];
#pragma unroll
        for (int g = 1; g < G; ++g) qb = __fadd_rn(qb, qreg[g][e]);
        const float qm = __fdiv_rn(qb, (float)G);
        const int dd = dim_of<Gm>(e, sigma);
        if (flags & kPlanFirst) {
          sreg[0][e] = qm; sreg[1][e] = qm;
        } else {
          sreg[0][e] = __fadd_rn(__fmul_rn(bS, srowp[dd]), __fmul_rn(aS, qm));
          sreg[1][e] = __fadd_rn(__fmul_rn(bL, srowp[D + dd]), __fmul_rn(aL, qm));
        }
      }
    }
    // RoPE(q) and RoPE(s) at the current position (fp32 table), then scale.
    if (p.rope) {
      const float* c32 = rope_c32(p, pos);
      const float* s32 = rope_s32(p, pos);
#pragma unroll
      for (int e = 0; e < H2; ++e) {
        const int di = dim_of<Gm>(e, sigma);
        const float c = c32[di], s = s32[di];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float x = qreg[g][e], y = qreg[g][e + H2];
          qreg[g][e] = x * c - y * s;
          qreg[g][e + H2] = y * c + x * s;
        }
        if (score) {
#pragma unroll
          for (int X = 0; X < 2; ++X) {
            const float x = sreg[X][e], y = sreg[X][e + H2];
            sreg[X][e] = x * c - y * s;
            sreg[X][e + H2] = y * c + x * s;
          }
        }
      }
    }
#pragma unroll
    for (int e = 0; e < NE; ++e) {
#pragma unroll
      for (int g = 0; g < G; ++g) qreg[g][e] *= qscale;
      sreg[0][e] *= sscale;
      sreg[1][e] *= sscale;
    }
    float* lgS = p.logits + ((((size_t)slot * p.L + layer) * p.Hk + h) * 2) * p.logit_width;
    float* lgL = lgS + p.logit_width;

    float m[G], l[G], o[G][NE];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY; l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < NE; ++e) o[g][e] = 0.f;
    }

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
      const uint8_t* sK = ring + s * Gm::STAGEB;
      const uint8_t* sV = sK + Gm::BLKB;
      const int t0 = (cc.blk + (int)k) * kBlockTok;
      const int nvalid = R - t0;  // tokens of this block that are resident
      float sc[4][G];
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int tk = it * 4 + tg;
        float kf[NE];
        load_row<T, Gm>(sK + tk * Gm::ROWB, sigma, kf);
        float acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < NE; ++e) a = fmaf(qreg[g][e], kf[e], a);
          acc[g] = a;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 1);
          acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 2);
          acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 4);
        }
        const bool valid = tk < nvalid;
#pragma unroll
        for (int g = 0; g < G; ++g) sc[it][g] = valid ? acc[g] : -INFINITY;
        if (score) {
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int e = 0; e < NE; ++e) {
            a0 = fmaf(sreg[0][e], kf[e], a0);
            a1 = fmaf(sreg[1][e], kf[e], a1);
          }
          a0 += __shfl_xor_sync(0xffffffffu, a0, 1);
          a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
          a0 += __shfl_xor_sync(0xffffffffu, a0, 2);
          a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
          a0 += __shfl_xor_sync(0xffffffffu, a0, 4);
          a1 += __shfl_xor_sync(0xffffffffu, a1, 4);
          if (sigma == 0 && valid) {
            lgS[t0 + tk] = a0;
            lgL[t0 + tk] = a1;
          }
        }
      }
      // online softmax (log2 domain), running max shared by the whole warp
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mb = fmaxf(fmaxf(sc[0][g], sc[1][g]), fmaxf(sc[2][g], sc[3][g]));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
        if (mb > m[g]) {
          const float al = (m[g] == -INFINITY) ? 0.f : exp2f(m[g] - mb);
          l[g] *= al;
#pragma unroll
          for (int e = 0; e < NE; ++e) o[g][e] *= al;
          m[g] = mb;
        }
      }
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int tk = it * 4 + tg;
        float vf[NE];
        load_row<T, Gm>(sV + tk * Gm::ROWB, sigma, vf);
        const bool valid = tk < nvalid;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pr = (valid && m[g] != -INFINITY) ? exp2f(sc[it][g] - m[g]) : 0.f;
          l[g] += pr;
#pragma unroll
          for (int e = 0; e < NE; ++e) o[g][e] = fmaf(pr, valid ? vf[e] : 0.f, o[g][e]);
        }
      }
      // refill this stage with the block S ahead
      __syncwarp();
      if (issued < end) {
        if (lane == 0) {
          fence_proxy_async_smem();
          issue_block<Gm>(p, layer, pc, ring + s * Gm::STAGEB, &bars[s]);
        }
        if (issued + 1 < end) cursor_next(p, pc);
        ++issued;
      }
    }
    if (failed) break;

    // ---- end of the piece: totals over the 4 token groups of the warp
#pragma unroll
    for (int g = 0; g < G; ++g) {
      l[g] += __shfl_xor_sync(0xffffffffu, l[g], 8);
      l[g] += __shfl_xor_sync(0xffffffffu, l[g], 16);
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 8);
        o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 16);
      }
    }
    if (full) {
      finalize<T, Gm, G>(p, layer, i, h, slot, pos, flags, q, knew, vnew, out, m, l, o, qreg, lane);
    } else {
      const int seg = i * p.Hk + h;
      const int pslot = (seg == first_seg) ? 0 : 1;
      float* part = p.partials + ((size_t)(w * 2 + pslot) * G) * (D + 2);
      if (tg == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int e = 0; e < NE; ++e) part[g * (D + 2) + dim_of<Gm>(e, sigma)] = o[g][e];
          if (sigma == 0) {
            part[g * (D + 2) + D] = m[g];
            part[g * (D + 2) + D + 1] = l[g];
          }
        }
      }
      __threadfence();
      __syncwarp();
      const int64_t seg_b0 = (int64_t)p.Hk * p.plan_cum[i] + (int64_t)h * nb;
      const int64_t w_first = ((seg_b0 + 1) * Weff - 1) / Tb;
      const int64_t w_last = ((seg_b0 + nb) * Weff - 1) / Tb;
      int old = 0;
      if (lane == 0) old = atomicAdd(&p.seg_count[seg], 1);
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old == (int)(w_last - w_first)) {
        __threadfence();
        const int64_t sfirst = (w_first * Tb) / Weff;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float mm = -INFINITY;
          for (int64_t k = w_first; k <= w_last; ++k) {
            const int ps = (k == w_first && sfirst != seg_b0) ? 1 : 0;
            const float* pk = p.partials + ((size_t)(k * 2 + ps) * G + g) * (D + 2);
            mm = fmaxf(mm, __ldcg(pk + D));
          }
          float ll = 0.f, oo[NE];
#pragma unroll
          for (int e = 0; e < NE; ++e) oo[e] = 0.f;
          for (int64_t k = w_first; k <= w_last; ++k) {
            const int ps = (k == w_first && sfirst != seg_b0) ? 1 : 0;
            const float* pk = p.partials + ((size_t)(k * 2 + ps) * G + g) * (D + 2);
            const float mk = __ldcg(pk + D);
            if (mk == -INFINITY) continue;
            const float wk = exp2f(mk - mm);
            ll = fmaf(__ldcg(pk + D + 1), wk, ll);
#pragma unroll
            for (int e = 0; e < NE; ++e) oo[e] = fmaf(__ldcg(pk + dim_of<Gm>(e, sigma)), wk, oo[e]);
          }
          m[g] = mm; l[g] = ll;
#pragma unroll
          for (int e = 0; e < NE; ++e) o[g][e] = oo[e];
        }
        finalize<T, Gm, G>(p, layer, i, h, slot, pos, flags, q, knew, vnew, out, m, l, o, qreg, lane);
        if (lane == 0) p.seg_count[seg] = 0;
      }
    }
    if (j < end) {  // next piece starts at block 0 of the following segment
      cc.blk = cc.nb - 1;
      cursor_next(p, cc);
    }
  }
  if (failed) {
    // let the copies this warp has in flight land before the CTA may exit
    for (int64_t jl = j - start; jl < issued - start; ++jl)
      (void)mbar_wait_bounded(&bars[jl % S], (uint32_t)((jl / S) & 1), kWaitLimitNs);
  }
}

template <typename T, int D>
constexpr int stages_for() { return (Geo<T, D>::STAGEB <= 8192) ? 3 : 2; }

template <typename T, int D, int G>
static cudaError_t launch_attn_t(const PoolDev& p, int layer, const void* q, const void* k,
                                 const void* v, void* out, int grid, cudaStream_t st) {
  using Gm = Geo<T, D>;
  constexpr int S = stages_for<T, D>();
  const size_t smem = (size_t)kAttnWarps * S * Gm::STAGEB + (size_t)kAttnWarps * S * 8;
  auto kern = attn_kernel<T, D, G, S>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kAttnWarps * 32, smem, st>>>(p, layer, (const T*)q, (const T*)k, (const T*)v, (T*)out);
  return cudaGetLastError();
}

template <typename T, int D, int G>
static cudaError_t occupancy_t(int* blocks) {
  using Gm = Geo<T, D>;
  constexpr int S = stages_for<T, D>();
  const size_t smem = (size_t)kAttnWarps * S * Gm::STAGEB + (size_t)kAttnWarps * S * 8;
  auto kern = attn_kernel<T, D, G, S>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, kern, kAttnWarps * 32, smem);
}

#define GP_DISPATCH(FN, ...)                                                          \
  do {                                                                                \
    if (p.dtype == GP_DTYPE_BF16 && p.D == 128) {                                     \
      if (p.G == 1) return FN<__nv_bfloat16, 128, 1>(__VA_ARGS__);                    \
      if (p.G == 2) return FN<__nv_bfloat16, 128, 2>(__VA_ARGS__);                    \
      if (p.G == 4) return FN<__nv_bfloat16, 128, 4>(__VA_ARGS__);                    \
    } else if (p.dtype == GP_DTYPE_F32 && p.D == 64) {                                \
      if (p.G == 1) return FN<float, 64, 1>(__VA_ARGS__);                             \
      if (p.G == 2) return FN<float, 64, 2>(__VA_ARGS__);                             \
      if (p.G == 4) return FN<float, 64, 4>(__VA_ARGS__);                             \
    } else if (p.dtype == GP_DTYPE_F32 && p.D == 128) {                               \
      if (p.G == 1) return FN<float, 128, 1>(__VA_ARGS__);                            \
      if (p.G == 2) return FN<float, 128, 2>(__VA_ARGS__);                            \
      if (p.G == 4) return FN<float, 128, 4>(__VA_ARGS__);                            \
    }                                                                                 \
    return cudaErrorInvalidValue;                                                     \
  } while (0)

cudaError_t launch_attention(const PoolDev& p, int layer, const void* q, const void* k,
                             const void* v, void* out, int grid, cudaStream_t st) {
  GP_DISPATCH(launch_attn_t, p, layer, q, k, v, out, grid, st);
}

cudaError_t attention_occupancy(const PoolDev& p, int* blocks) {
  GP_DISPATCH(occupancy_t, blocks);
}

}  // namespace gp
