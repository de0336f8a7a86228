// gp_step.cu -- the per-step kernels around the attention kernel.
//
//   plan_kernel     once per step (before layer 0): per request, resident
//                   tokens, attention blocks, boundary flags; prefix sums;
//                   the attention workers' weighted ranges and each cut
//                   (request, head)'s first and last worker.
//   select_kernel   per (boundary request, layer, kv head): softmax of both
//                   summaries' scores, Top-p working-set size by radix select
//                   with exact integer mass, Delta contribution, and the
//                   compaction plan (which private tokens to drop); for the
//                   SHRINK ablation a second launch re-plans the requests
//                   that release a page.
//   decide_kernel   one CTA: grow, compact or (SHRINK) release a page per
//                   request; pages popped from the lock-free stack in
//                   ascending slot order, released pages pushed after every
//                   pop; metadata.
//   commit_kernel   per (request, layer, kv head): the step's folded
//                   summaries of a request at a boundary made current (the
//                   attention kernel writes the others in place), compaction
//                   moves, then the staged token written into its slot.
// For the asynchronous boundary path, decide and commit run twice: once on
// the pool's stream for the requests not at a boundary, once on a second
// stream for those at a boundary (which sit out the next step).
//
// Method: "GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning
// Serving" -- abstract (capacity boundaries; compress within the current
// allocation or acquire one more physical page) and evolve.pub review,
// Summary (Top-p working sets of the two summaries; a larger recent set grows
// the request by one page, otherwise compaction by the maximum of both
// importance scores) and FAQ (Top-p, tau, local retention quota).
#include "gp_internal.cuh"

namespace gp {

// ------------------------------------------------------- block helpers ---

// Exclusive scan of one int per thread over the block (<= 1024 threads).
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int t = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
    int u = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, u, o);
      if (lane >= o) u += y;
    }
    s_warp[lane] = u - t;  // exclusive prefix of warp totals
    if (lane == 31) s_warp[32] = u;
  }
  __syncthreads();
  const int res = s_warp[wid] + x - v;
  *total = s_warp[32];
  __syncthreads();
  return res;
}

// ---------------------------------------------------------------- plan ---

// count == 0: lay out the plan without touching the pool's step counters
// (used by the read-ceiling measurement between steps).
constexpr int kPlanSmemReq = 2048;

__global__ void __launch_bounds__(1024) plan_kernel(PoolDev p, int n, const int32_t* slots, int count) {
  // Launched as a programmatic dependent of the kernel before it: wait for it.
  // No early trigger: the attention kernel after this one reads the plan
  // before its own wait, so it may start only once this kernel has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ int s_warp[33];
  __shared__ int s_bad;
  __shared__ unsigned long long s_tok, s_btok;
  // per-request block counts and prefix sums for the searches below (up to
  // kPlanSmemReq requests; beyond that the searches read the global copies)
  __shared__ int s_cum[kPlanSmemReq], s_nb[kPlanSmemReq];
  const bool in_smem = n <= kPlanSmemReq;
  const int* cum = in_smem ? s_cum : p.plan_cum;
  const int* nbs = in_smem ? s_nb : p.plan_nb;
  if (threadIdx.x == 0) { s_bad = 0; s_tok = 0ull; s_btok = 0ull; }
  __syncthreads();
  int carry = 0, bcarry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    int nb = 0, isb = 0;
    if (i < n) {
      const int slot = slots[i];
      bool ok = (unsigned)slot < (unsigned)p.max_req;
      if (ok) {  // boundary work still running on the second stream: refused
        int b;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(b) : "l"(p.busy + slot) : "memory");
        ok = b == 0;
      }
      if (ok) ok = p.req[slot].active != 0;
      if (ok && i > 0) ok = slots[i - 1] < slot;
      if (ok && p.req[slot].pos >= p.max_seq_len) {
        ok = false;
        set_status(p, GP_ST_POS_RANGE, slot);
      }
      if (!ok) {
        s_bad = 1;
        set_status(p, GP_ST_BAD_SLOTS, i);
        p.plan_slot[i] = 0; p.plan_R[i] = 0; p.plan_nb[i] = 1; p.plan_flags[i] = 0;
        p.plan_pos[i] = 0; p.plan_base[i] = 0;
        nb = 1;
      } else {
        const gp_req_meta m = p.req[slot];
        const int R = m.n_pre_pages * p.P + m.seq_priv;
        // a shared prefix is attended by prefix_attn_kernel, once per group
        // of requests sharing it: the attention kernel starts after it
        const int base = (count && p.prefix_batch && m.prefix_id >= 0 && m.n_pre_pages > 0)
                             ? m.n_pre_pages * p.P : 0;
        nb = (R - base + kBlockTok - 1) / kBlockTok;
        if (nb < 1) nb = 1;
        p.plan_base[i] = base;
        const bool at_b = m.seq_priv == m.n_pages * p.P;
        int flags = 0;
        if (at_b) flags |= kPlanBoundary;
        if (m.steps == 0) flags |= kPlanFirst;
        if (at_b && p.mode != GP_MODE_FULL_KV) flags |= kPlanScore;
        isb = (flags & kPlanScore) ? 1 : 0;
        p.plan_slot[i] = slot; p.plan_R[i] = R; p.plan_nb[i] = nb; p.plan_flags[i] = flags;
        p.plan_pos[i] = m.pos;
        p.plan_delta[i] = 0;
        atomicAdd(&s_tok, (unsigned long long)R);
        if (at_b) atomicAdd(&s_btok, (unsigned long long)R);
      }
    }
    int tot, btot;
    const int ex = block_excl_scan(nb, s_warp, &tot);
    const int bex = block_excl_scan(isb, s_warp, &btot);
    if (i < n) {
      p.plan_cum[i] = carry + ex;
      if (in_smem) { s_cum[i] = carry + ex; s_nb[i] = nb; }
      if (isb) p.plan_bnd[bcarry + bex] = i;
    }
    carry += tot;
    bcarry += btot;
  }
  __syncthreads();
  // Shares of the attention workers.  The blocks of all (request, head)
  // segments are laid end to end (request-major, then head, then block);
  // each segment start also costs seg_cost extra units (its piece set-up).
  // Worker w of Weff = min(workers, total blocks) takes the blocks whose
  // units fall in [w*U/Weff, (w+1)*U/Weff), U = blocks + seg_cost * segments.
  // With seg_cost = 0 this is an equal split of the blocks.
  __shared__ int s_wblk[kMaxWorkersBound + 1];
  if (!s_bad && n > 0) {
    const long long Tb = (long long)carry * p.Hk;
    const long long W = p.num_workers;
    const long long Weff = W < Tb ? W : Tb;
    const long long c = p.seg_cost;
    const int nseg = n * p.Hk;
    // the merge counters of cut (request, head)s start the step at zero (the
    // last piece of each resets its own after every layer)
    for (int k = threadIdx.x; count && k < nseg; k += blockDim.x) p.seg_count[k] = 0;
    const long long U = Tb + c * nseg;
    for (int w = threadIdx.x; w < Weff; w += blockDim.x) {
      const long long u = ((long long)w * U) / Weff;
      // largest segment k with (start block of k) + c*k <= u
      int lo = 0, hi = nseg - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int mi = mid / p.Hk, mh = mid % p.Hk;
        const long long cb = (long long)p.Hk * cum[mi] + (long long)mh * nbs[mi] + c * mid;
        if (cb <= u) lo = mid; else hi = mid - 1;
      }
      const int i = lo / p.Hk, h = lo % p.Hk;
      const int nb = nbs[i];
      const long long sb = (long long)p.Hk * cum[i] + (long long)h * nb;
      const long long off = u - sb - c * lo;
      const int blk = off < c ? 0 : (int)(off - c);
      p.wstart[w] = make_int4(i, (h << 20) | blk, nb, p.plan_slot[i]);
      p.wblk[w] = (int)(sb + blk);
      s_wblk[w] = (int)(sb + blk);
    }
    if (threadIdx.x == 0) {
      p.wblk[Weff] = (int)Tb;
      s_wblk[Weff] = (int)Tb;
    }
    __syncthreads();
    // each segment's first and last worker: the last worker whose share
    // starts at or before the segment's first (last) block (not needed by
    // the read-ceiling measurement, count == 0)
    for (int k = threadIdx.x; count && k < nseg; k += blockDim.x) {
      const int i = k / p.Hk, h = k % p.Hk;
      const int nb = nbs[i];
      const long long sb = (long long)p.Hk * cum[i] + (long long)h * nb;
      int wf = 0, wl = 0;
      for (int pass = 0; pass < 2; ++pass) {
        const long long b = pass ? sb + nb - 1 : sb;
        int lo = 0, hi = (int)Weff - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_wblk[mid] <= b) lo = mid; else hi = mid - 1;
        }
        if (pass) wl = lo; else wf = lo;
      }
      p.seginfo[k] = make_int4(wf, wl, s_wblk[wf] != sb ? 1 : 0, 0);
    }
  }
  // Shared-prefix units: the step's requests grouped by prefix (pmem, in an
  // arbitrary order inside a group: each member's result is its own), then
  // per prefix ceil(members / kPrefChunk) chunks x Hk heads x ranges of
  // kPrefRangeBlocks blocks, laid end to end (unit_cum).
  __shared__ int s_pcnt[kMaxPrefixBatch];
  int punits = 0;
  const bool batch = count && p.prefix_batch && !s_bad && n > 0;
  if (batch) {
    const int np = p.max_prefixes;  // <= kMaxPrefixBatch when batching is on
    for (int k = threadIdx.x; k < np; k += blockDim.x) s_pcnt[k] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      if (p.plan_base[i] > 0) p.pranges[i] = atomicAdd(&s_pcnt[p.req[p.plan_slot[i]].prefix_id], 1);
    __syncthreads();
    int tot_m, tot_u;
    const int k = threadIdx.x;  // np <= blockDim.x
    const int cnt = k < np ? s_pcnt[k] : 0;
    const int nr = (k < np && cnt) ? (p.prefix[k].len / kBlockTok + kPrefRangeBlocks - 1) / kPrefRangeBlocks : 0;
    const int units = cnt ? ((cnt + kPrefChunk - 1) / kPrefChunk) * p.Hk * nr : 0;
    const int off = block_excl_scan(cnt, s_warp, &tot_m);
    const int uoff = block_excl_scan(units, s_warp, &tot_u);
    if (k < np) { p.pref_off[k] = off; p.pref_cnt[k] = cnt; p.unit_cum[k] = uoff; }
    if (k == 0) p.unit_cum[np] = tot_u;
    punits = tot_u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      if (p.plan_base[i] > 0) {
        const int pid = p.req[p.plan_slot[i]].prefix_id;
        p.pmem[p.pref_off[pid] + p.pranges[i]] = i;
        p.pranges[i] = (p.prefix[pid].len / kBlockTok + kPrefRangeBlocks - 1) / kPrefRangeBlocks;
      } else {
        p.pranges[i] = 0;
      }
    }
  } else if (count && !s_bad && p.prefix_batch) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) p.pranges[i] = 0;
  }
  if (threadIdx.x == 0) {
    p.plan_cum[n] = carry;
    const int good = s_bad ? 0 : n;
    p.plan_misc[0] = good;
    p.plan_misc[1] = s_bad ? 0 : bcarry;
    p.plan_misc[2] = carry;
    p.plan_misc[3] = punits;
    if (count) {  // a rejected step (bad slot list) is not counted
      p.ctrl->plan_n = good;
      if (!s_bad) {
        p.ctrl->steps += 1;
        p.ctrl->tokens_attended += (long long)s_tok;
        p.ctrl->boundary_tokens += (long long)s_btok;
      }
    }
  }
}

// -------------------------------------------------------------- select ---

#ifndef GP_SEL_THREADS
#define GP_SEL_THREADS 256
#endif
#ifndef GP_SEL_TOK
#define GP_SEL_TOK 4096
#endif
#ifndef GP_SEL_MINB
#define GP_SEL_MINB 4
#endif
constexpr int kSelThreads = GP_SEL_THREADS;

// Block-wide max of two values at once (one per summary).
__device__ __forceinline__ float2 block_max2(float a, float b, float2* red) {
  a = warp_max(a);
  b = warp_max(b);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) red[wid] = make_float2(a, b);
  __syncthreads();
  if (wid == 0) {
    const bool in = lane < (int)(blockDim.x >> 5);
    float x = in ? red[lane].x : -INFINITY, y = in ? red[lane].y : -INFINITY;
    x = warp_max(x);
    y = warp_max(y);
    if (lane == 0) red[32] = make_float2(x, y);
  }
  __syncthreads();
  const float2 r = red[32];
  __syncthreads();
  return r;
}

// Block-wide sums of two 64-bit values at once.
__device__ __forceinline__ void block_sum2_ull(unsigned long long& a, unsigned long long& b,
                                               ulonglong2* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) red[wid] = make_ulonglong2(a, b);
  __syncthreads();
  if (wid == 0) {
    const bool in = lane < (int)(blockDim.x >> 5);
    unsigned long long x = in ? red[lane].x : 0ull, y = in ? red[lane].y : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      x += __shfl_xor_sync(0xffffffffu, x, o);
      y += __shfl_xor_sync(0xffffffffu, y, o);
    }
    if (lane == 0) red[32] = make_ulonglong2(x, y);
  }
  __syncthreads();
  a = red[32].x;
  b = red[32].y;
  __syncthreads();
}

// Probability mass of a token in fixed point: e * 2^40 rounded to nearest,
// ties to even (e in [0, 1]; the same value as converting the exact fp32
// product e * 2^40 to an integer).  Worked on the bit pattern with integer
// operations: e = m * 2^(E - 150), so e * 2^40 = m * 2^(E - 110).
__device__ __forceinline__ unsigned long long mass_q(float e) {
  const uint32_t b = __float_as_uint(e);
  const int E = (int)(b >> 23);  // biased exponent (e >= 0)
  if (E == 0) return 0ull;       // zero or subnormal: e * 2^40 < 2^-86
  const uint32_t m = (b & 0x7fffffu) | 0x800000u;
  const int sh = 110 - E;
  if (sh <= 0) return (-sh <= 40) ? (unsigned long long)m << (-sh) : 0ull;
  if (sh > 25) return 0ull;      // m < 2^24 < half of 2^sh
  const uint32_t q = m >> sh, rem = m & ((1u << sh) - 1u), half = 1u << (sh - 1);
  return (unsigned long long)(q + ((rem > half || (rem == half && (q & 1u))) ? 1u : 0u));
}

// ceil(top_p * T) exactly, top_p an fp32 value in (0, 1].
__device__ __forceinline__ unsigned long long ceil_mul(float top_p, unsigned long long T) {
  const uint32_t b = __float_as_uint(top_p);
  const int E = (int)((b >> 23) & 0xff);
  unsigned long long M = (E == 0) ? (b & 0x7fffffu) : ((b & 0x7fffffu) | 0x800000u);
  const int sh = (E == 0 ? 1 : E) - 150;  // top_p = M * 2^sh, sh < 0
  const unsigned long long lo = M * T, hi = __umul64hi(M, T);
  const int r = -sh;
  if (r >= 128) return (lo | hi) ? 1ull : 0ull;
  unsigned long long qv, rem;
  if (r >= 64) {
    qv = (r == 64) ? hi : (hi >> (r - 64));
    rem = lo | ((r == 64) ? 0ull : (hi & ((1ull << (r - 64)) - 1ull)));
  } else if (r == 0) {
    qv = lo; rem = 0;
  } else {
    qv = (lo >> r) | (hi << (64 - r));
    rem = lo & ((1ull << r) - 1ull);
  }
  return qv + (rem ? 1ull : 0ull);
}

// Histograms for both summaries.
struct SelShared {
  unsigned int cnt[2][256];
  // the 64-bit masses as two 32-bit words, added with native 32-bit atomics
  // (the low word's carry goes to the high word)
  unsigned int mlo[2][256], mhi[2][256];
  ulonglong2 red[33];
  float2 redf[33];
  unsigned int pick_d[2], pick_c[2];  // picked digit and how many elements it holds
  unsigned long long pick_a[2], pick_b[2];
  int done;
  int hcount[32];   // compaction holes per warp
  float inv[2];     // 2^40 / total mass of each summary
};

// x as fp32: the high word (exact below 2^24) times 2^32 plus the low word,
// rounded once more by the fused multiply-add (within an ulp of x).
__device__ __forceinline__ float u64_to_f32(unsigned long long x) {
  return __fmaf_rn(__uint2float_rn((unsigned int)(x >> 32)), 0x1p32f, __uint2float_rn((unsigned int)x));
}

__device__ __forceinline__ unsigned long long mass_at(const SelShared& sh, int X, int d) {
  return ((unsigned long long)sh.mhi[X][d] << 32) | sh.mlo[X][d];
}

// Sources of e_j = exp(u_j - max) for one summary's scores: computed from the
// scores in global memory, or read from shared memory where the kernel has
// staged them once (rows of up to kSelSmemTok tokens).  Both give the same
// value for every j.
struct EGlobal {
  const float* u;
  float mx;
  __device__ __forceinline__ float operator()(int j) const { return expf(u[j] - mx); }
};
struct ESmem {
  const float* e;
  __device__ __forceinline__ float operator()(int j) const { return e[j]; }
};
// Absolute position of private slot s: gathered through the block table, or
// staged in shared memory.
struct PosGlobal {
  const int32_t* bt;
  const int32_t* tok_pos;
  int P, L, Hk, layer, h, num_pages;
  __device__ __forceinline__ int operator()(int s) const {
    int page = bt[s / P];
    if ((unsigned)page >= (unsigned)num_pages) page = 0;
    return tok_pos[(((size_t)page * L + layer) * Hk + h) * P + (s % P)];
  }
};
struct PosSmem {
  const int* pos;
  __device__ __forceinline__ int operator()(int s) const { return pos[s]; }
};

// Top-p working-set sizes of both summaries: for each, the smallest k with
// (mass of the k largest) >= thr, by a 4-pass radix select (8 bits per pass,
// most significant first) on the fp32 bit patterns of e_j, weighting each by
// its fixed-point mass.  The two selects share their passes: warp X scans
// summary X's histogram.  A summary whose picked digit holds one element is
// settled there: that element is the last one the set needs (the mass still
// needed is positive and at most its own), so k = (count above it) + 1, which
// is what the remaining passes would give; it takes no part in them.
__device__ __forceinline__ void bin_add(SelShared& sh, int X, int d, unsigned int c, unsigned long long v) {
  atomicAdd(&sh.cnt[X][d], c);
  const unsigned int vlo = (unsigned int)v, vhi = (unsigned int)(v >> 32);
  const unsigned int old = atomicAdd(&sh.mlo[X][d], vlo);
  const unsigned int up = vhi + ((old + vlo < old) ? 1u : 0u);
  if (up) atomicAdd(&sh.mhi[X][d], up);
}

// Adds each lane's (digit d, mass mq) to the histogram X (d = 256: nothing).
// A lane alone with its digit adds its own; lanes sharing a digit are summed
// first, one group at a time, by full-warp reductions (a reduction over a
// partial mask costs a pass per group anyway, and more).
__device__ __forceinline__ void hist_add(SelShared& sh, int X, int d, unsigned long long mq) {
  const int lane = threadIdx.x & 31;
  const unsigned int peers = __match_any_sync(0xffffffffu, d);
  const bool valid = d < 256;
  const bool alone = __popc(peers) == 1;
  if (valid && alone) bin_add(sh, X, d, 1u, mq);
  unsigned int todo = __ballot_sync(0xffffffffu, valid && !alone);
  while (todo) {  // warp-uniform
    const int src = __ffs(todo) - 1;
    const unsigned int members = __shfl_sync(0xffffffffu, peers, src);
    const bool in = (members >> lane) & 1u;
    const unsigned int hi = __reduce_add_sync(0xffffffffu, in ? (unsigned int)(mq >> 20) : 0u);
    const unsigned int lo = __reduce_add_sync(0xffffffffu, in ? (unsigned int)(mq & 0xfffffull) : 0u);
    if (lane == src) bin_add(sh, X, d, (unsigned int)__popc(members), ((unsigned long long)hi << 20) + lo);
    todo &= ~members;
  }
}

template <class ES, class EL>
__device__ int2 topp_radix2(ES eS, EL eL, int R, unsigned long long thr0, unsigned long long thr1,
                            SelShared& sh, uint32_t* wbins_a = nullptr,
                            uint32_t* wbins_b = nullptr) {
  uint32_t prefix[2] = {0u, 0u}, pmask = 0u;
  unsigned long long mass_above[2] = {0ull, 0ull}, cnt_above[2] = {0ull, 0ull};
  bool settled[2] = {false, false};  // block-uniform (from shared picks)
  for (int d = threadIdx.x; d < 512; d += blockDim.x) {
    (&sh.cnt[0][0])[d] = 0u;
    (&sh.mlo[0][0])[d] = 0u;
    (&sh.mhi[0][0])[d] = 0u;
  }
  __syncthreads();
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (pass == 0 && wbins_a) {
      // The top byte of e in [0, 1] is one of 64 digits (sign 0, exponent
      // <= 127).  Each warp counts into bins of its own (cnt, mass low and
      // high words: [warp][X][64] each, in shared memory the caller leaves
      // free), so only lanes of one warp ever meet on a bin; the warps' bins
      // are then summed into the histogram.
      const int nw = blockDim.x >> 5, wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
      uint32_t* wc = wbins_a;               // [nw][2][64] counts
      uint32_t* wl = wbins_a + nw * 128;    // mass low words
      uint32_t* wh = wbins_b;               // mass high words
      for (int k = lane; k < 128; k += 32) {
        wc[wid * 128 + k] = 0u;
        wl[wid * 128 + k] = 0u;
        wh[wid * 128 + k] = 0u;
      }
      __syncwarp();
      for (int base = 0; base < R; base += blockDim.x) {
        const int j = base + threadIdx.x;
        if (j < R) {
#pragma unroll
          for (int X = 0; X < 2; ++X) {
            const float e = X ? eL(j) : eS(j);
            const int b = wid * 128 + X * 64 + (int)min(__float_as_uint(e) >> 24, 63u);
            const unsigned long long mq = mass_q(e);
            atomicAdd(&wc[b], 1u);
            const unsigned int vlo = (unsigned int)mq, vhi = (unsigned int)(mq >> 32);
            const unsigned int old = atomicAdd(&wl[b], vlo);
            const unsigned int up = vhi + ((old + vlo < old) ? 1u : 0u);
            if (up) atomicAdd(&wh[b], up);
          }
        }
      }
      __syncthreads();
      for (int k = threadIdx.x; k < 128; k += blockDim.x) {
        unsigned int c = 0u;
        unsigned long long m = 0ull;
        for (int w2 = 0; w2 < nw; ++w2) {
          c += wc[w2 * 128 + k];
          m += ((unsigned long long)wh[w2 * 128 + k] << 32) | wl[w2 * 128 + k];
        }
        const int X = k >> 6, d = k & 63;
        sh.cnt[X][d] = c;
        sh.mlo[X][d] = (unsigned int)m;
        sh.mhi[X][d] = (unsigned int)(m >> 32);
      }
      __syncthreads();
    } else {
    // Most weights share their top digits, so lanes with the same digit are
    // combined inside the warp first and one lane per digit does the atomics.
    for (int base = 0; base < R; base += blockDim.x) {
      const int j = base + threadIdx.x;
      int d0 = 256, d1 = 256;  // 256: "no digit"
      unsigned long long m0 = 0ull, m1 = 0ull;
      if (j < R) {
        const float e0 = eS(j), e1 = eL(j);
        const uint32_t b0 = __float_as_uint(e0), b1 = __float_as_uint(e1);
        if (!settled[0] && (b0 & pmask) == prefix[0]) { d0 = (b0 >> shift) & 255; m0 = mass_q(e0); }
        if (!settled[1] && (b1 & pmask) == prefix[1]) { d1 = (b1 >> shift) & 255; m1 = mass_q(e1); }
      }
      if (!settled[0]) hist_add(sh, 0, d0, m0);
      if (!settled[1]) hist_add(sh, 1, d1, m1);
    }
    __syncthreads();
    }
    const int wid = threadIdx.x >> 5;
    if (wid < 2 && !(wid ? settled[1] : settled[0])) {  // (no indexing: registers)
      // descending digits: lane L owns digits 255-8L .. 248-8L and is the
      // only lane that reads them, so it clears them for the next pass
      const int X = wid, lane = threadIdx.x & 31;
      unsigned long long mloc = 0ull, cloc = 0ull;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        mloc += mass_at(sh, X, 255 - 8 * lane - t);
        cloc += sh.cnt[X][255 - 8 * lane - t];
      }
      unsigned long long mex = mloc, cex = cloc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        unsigned long long y = __shfl_up_sync(0xffffffffu, mex, o);
        unsigned long long z = __shfl_up_sync(0xffffffffu, cex, o);
        if (lane >= o) { mex += y; cex += z; }
      }
      mex -= mloc; cex -= cloc;  // mass / count of the digits above this lane's
      // (register selects, not indexing: the arrays stay in registers)
      const unsigned long long need = X ? thr1 - mass_above[1] : thr0 - mass_above[0];
      const bool here = (mex < need) && (mex + mloc >= need);
      const unsigned int bal = __ballot_sync(0xffffffffu, here);
      if (bal == 0u && lane == 0) {
        sh.pick_d[X] = 0u; sh.pick_c[X] = 0u; sh.pick_a[X] = 0ull; sh.pick_b[X] = 0ull;
      }
      if (here && lane == __ffs(bal) - 1) {
        unsigned long long macc = mex, cacc = cex;
        for (int t = 0; t < 8; ++t) {
          const int d = 255 - 8 * lane - t;
          if (macc + mass_at(sh, X, d) >= need || t == 7) {
            sh.pick_d[X] = (unsigned)d;
            sh.pick_c[X] = sh.cnt[X][d];
            sh.pick_a[X] = macc;
            sh.pick_b[X] = cacc;
            break;
          }
          macc += mass_at(sh, X, d);
          cacc += sh.cnt[X][d];
        }
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        sh.mlo[X][255 - 8 * lane - t] = 0u;
        sh.mhi[X][255 - 8 * lane - t] = 0u;
        sh.cnt[X][255 - 8 * lane - t] = 0u;
      }
    }
    __syncthreads();
    // the picks are rewritten only after the next pass's histogram barrier
#pragma unroll
    for (int X = 0; X < 2; ++X) {
      if (settled[X]) continue;
      prefix[X] |= sh.pick_d[X] << shift;
      mass_above[X] += sh.pick_a[X];
      cnt_above[X] += sh.pick_b[X];
      settled[X] = sh.pick_c[X] == 1u;
    }
    pmask |= 255u << shift;
    if (settled[0] && settled[1]) break;
  }
  int W[2];
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    if (settled[X]) {
      W[X] = (int)(cnt_above[X] + 1ull);
      continue;
    }
    const unsigned long long thr = X ? thr1 : thr0;
    const unsigned long long qstar = mass_q(__uint_as_float(prefix[X]));
    const unsigned long long rest = thr > mass_above[X] ? thr - mass_above[X] : 0ull;
    const unsigned long long k = qstar ? (rest + qstar - 1ull) / qstar : 1ull;
    W[X] = (int)(cnt_above[X] + (k ? k : 1ull));
  }
  return make_int2(W[0], W[1]);
}

// Compaction key of private slot s: (importance bits << 32 | position), with
// importance = max(p_S, p_L); *cand: the token is older than the window.
template <class ES, class EL, class PF>
struct KeyOf {
  ES eS;
  EL eL;
  PF posf;
  float invS, invL;
  int npre, cut_pos;
  __device__ __forceinline__ unsigned long long operator()(int s, bool* cand) const {
    const int pos = posf(s);
    *cand = pos < cut_pos;
    const float I = fmaxf(eS(npre + s) * invS, eL(npre + s) * invL);
    return ((unsigned long long)__float_as_uint(I) << 32) | (unsigned long long)(uint32_t)pos;
  }
};

// Threshold key such that exactly `k` candidates have key <= threshold (keys
// are distinct: they end with the token position).  Radix select, 8 bits per
// pass from the top, stopping as soon as the chosen bucket is taken whole.
// The bucket is found by warp 0: lane L owns digits 8L .. 8L+7.
template <class KF>
__device__ unsigned long long kth_smallest(const KF& key_of, int C, int k, SelShared& sh) {
  unsigned long long prefix = 0ull, pmask = 0ull;
  unsigned int below = 0u;
  for (int d = threadIdx.x; d < 256; d += blockDim.x) sh.cnt[0][d] = 0u;
  __syncthreads();
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int base = 0; base < C; base += blockDim.x) {
      const int s = base + threadIdx.x;
      int d = 256;
      if (s < C) {
        bool cand;
        const unsigned long long key = key_of(s, &cand);
        if (cand && (key & pmask) == prefix) d = (int)((key >> shift) & 255);
      }
      const unsigned int peers = __match_any_sync(0xffffffffu, d);
      if (d < 256 && (threadIdx.x & 31) == __ffs(peers) - 1)
        atomicAdd(&sh.cnt[0][d], (unsigned int)__popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      unsigned int c[8], cloc = 0u;
#pragma unroll
      for (int t = 0; t < 8; ++t) { c[t] = sh.cnt[0][8 * lane + t]; cloc += c[t]; }
      unsigned int cex = cloc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, cex, o);
        if (lane >= o) cex += y;
      }
      cex = below + cex - cloc;  // candidates below this lane's digits
      const bool here = (cex < (unsigned)k) && (cex + cloc >= (unsigned)k);
      const unsigned int bal = __ballot_sync(0xffffffffu, here);
      // no crossing (fewer than k candidates): the last digit, as a scan would end
      const int owner = bal ? __ffs(bal) - 1 : 31;
      if (lane == owner) {
        unsigned int acc = cex;
        int t = 0;
        for (; t < 7; ++t) {
          if (acc + c[t] >= (unsigned)k) break;
          acc += c[t];
        }
        sh.pick_d[0] = (unsigned)(8 * lane + t);
        sh.pick_a[0] = acc;
        sh.done = (acc + c[t] == (unsigned)k) ? 1 : 0;
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) sh.cnt[0][8 * lane + t] = 0u;
    }
    __syncthreads();
    // the picks are rewritten only after the next pass's histogram barrier
    const unsigned int d = sh.pick_d[0];
    below = (unsigned int)sh.pick_a[0];
    prefix |= (unsigned long long)d << shift;
    pmask |= 255ull << shift;
    if (sh.done) return prefix | ((shift == 0) ? 0ull : ((1ull << shift) - 1ull));
  }
  return prefix;
}

// Working sets, Delta and the compaction plan of one (request, layer, head).
// The plan frees nfree private slots of a request holding C: it drops the
// nfree lowest (importance, position) candidates older than the window and
// moves the survivors at or above C - nfree into the holes below it.  With
// replan set (the SHRINK ablation's second pass, after the decisions), only
// the plan is computed.
template <class ES, class EL, class PF>
__device__ void select_item(const PoolDev& p, int i, int slot, size_t row, const gp_req_meta& m,
                            int R, ES eS, EL eL, unsigned long long TS, unsigned long long TL,
                            PF posf, int C, int pos, int nfree, bool replan, SelShared& sh,
                            uint32_t* wbins_a = nullptr, uint32_t* wbins_b = nullptr) {
  // the importance scales 2^40 / T in fp32 (T >= 2^40: the largest e_j is 1),
  // once per item by one thread, published by the next barrier
  if (threadIdx.x == 0) {
    sh.inv[0] = __fdiv_rn(0x1p40f, u64_to_f32(TS ? TS : 1ull));
    sh.inv[1] = __fdiv_rn(0x1p40f, u64_to_f32(TL ? TL : 1ull));
  }
  if (!replan) {
    // Top-p counts from the fixed-point total masses TS, TL
    const int2 Wv = topp_radix2(eS, eL, R, ceil_mul(p.top_p, TS), ceil_mul(p.top_p, TL), sh, wbins_a,
                                wbins_b);
    if (threadIdx.x == 0) {
      p.wset[row * 2 + 0] = Wv.x;
      p.wset[row * 2 + 1] = Wv.y;
      atomicAdd((unsigned long long*)&p.plan_delta[i], (unsigned long long)(long long)(Wv.x - Wv.y));
    }
  } else {
    __syncthreads();
  }
  const int keep = C - nfree;
  const int weff = min(p.recent_window, keep);
  KeyOf<ES, EL, PF> key_of{eS, eL, posf, sh.inv[0], sh.inv[1], m.n_pre_pages * p.P, pos - weff};
  const unsigned long long thr_key = kth_smallest(key_of, C, nfree, sh);
  // holes below C - nfree and the survivors above it, both ascending, paired
  // in order straight into the move list.  The holes: every warp counts those
  // of its chunk of slots, then writes them after the chunks before it.
  int32_t* mv = p.moves + row * (size_t)p.P * 4;  // room for 2P moves
  {
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int chunk = ((keep + nw - 1) / nw + 31) & ~31;
    const int s0 = wid * chunk, s1 = min(keep, s0 + chunk);
    auto dropped_at = [&](int s) -> bool {
      if (s >= s1) return false;
      bool cand;
      const unsigned long long key = key_of(s, &cand);
      return cand && key <= thr_key;
    };
    int cnt = 0;
    for (int base = s0; base < s1; base += 32) cnt += __popc(__ballot_sync(0xffffffffu, dropped_at(base + lane)));
    if (lane == 0) sh.hcount[wid] = cnt;
    __syncthreads();
    int nh = 0;
    for (int w2 = 0; w2 < wid; ++w2) nh += sh.hcount[w2];
    for (int base = s0; base < s1; base += 32) {
      const bool dropped = dropped_at(base + lane);
      const unsigned int bal = __ballot_sync(0xffffffffu, dropped);
      if (dropped) {
        const int r = nh + __popc(bal & ((1u << lane) - 1u));
        if (r < nfree) mv[2 * r] = base + lane;
      }
      nh += __popc(bal);
    }
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int nh = 0;
    for (int w2 = 0; w2 < (int)(blockDim.x >> 5); ++w2) nh += sh.hcount[w2];
    int ns = 0;
    for (int base = keep; base < C; base += 32) {
      const int s = base + lane;
      bool kept = false;
      if (s < C) {
        bool cand;
        const unsigned long long key = key_of(s, &cand);
        kept = !(cand && key <= thr_key);
      }
      const unsigned int bal = __ballot_sync(0xffffffffu, kept);
      if (kept) {
        const int r = ns + __popc(bal & ((1u << lane) - 1u));
        if (r < nfree) mv[2 * r + 1] = s;
      }
      ns += __popc(bal);
    }
    if (nh != ns || nh > nfree) {
      if (lane == 0) set_status(p, GP_ST_BAD_PLAN, slot);
      nh = 0;
    }
    if (lane == 0) p.moves_n[row] = nh;
  }
  __syncthreads();
}

// Rows of up to this many tokens are staged in shared memory: both
// summaries' e_j and the private slots' positions (48 KiB).
constexpr int kSelSmemTok = GP_SEL_TOK;
constexpr size_t kSelSmemBytes = (size_t)kSelSmemTok * (4 + 4 + 4);

// Two shapes of the same kernel: 256 threads, 4 CTAs per SM (many items:
// throughput) and 512 threads, 2 CTAs per SM (few items: latency per item).
template <int T, int MINB>
__global__ void __launch_bounds__(T, MINB) select_kernel(PoolDev p, int replan) {
  // programmatic dependent of the kernel before it; lets the next one launch
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ SelShared sh;
  extern __shared__ float sel_dyn[];
  float* eSs = sel_dyn;
  float* eLs = sel_dyn + kSelSmemTok;
  int* poss = reinterpret_cast<int*>(sel_dyn + 2 * kSelSmemTok);
  const int nb = p.plan_misc[1];
  const int items = nb * p.L * p.Hk;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int bi = item / (p.L * p.Hk);
    const int rem = item % (p.L * p.Hk);
    const int layer = rem / p.Hk, h = rem % p.Hk;
    const int i = p.plan_bnd[bi];
    if (replan && p.plan_dec[i] != kShrink) continue;  // uniform over the CTA
    const int slot = p.plan_slot[i];
    const int R = p.plan_R[i];
    const gp_req_meta m = p.req[slot];
    // the replan runs after the decisions, which have moved n_pages and pos
    const int C = replan ? p.plan_commit[i] + 2 * p.P : m.n_pages * p.P;
    const int pos = replan ? p.plan_cpos[i] : m.pos;
    const int nfree = replan ? 2 * p.P : p.P;
    const size_t row = ((size_t)slot * p.L + layer) * p.Hk + h;
    const float* uS = p.logits + row * 2 * p.logit_width;
    const float* uL = uS + p.logit_width;
    // rows of up to kSelSmemTok tokens are staged: the scores now, e_j below
    // (each thread rewrites its own entries)
    const bool staged = R <= kSelSmemTok && C <= kSelSmemTok;
    float a = -INFINITY, b = -INFINITY;
    for (int j = threadIdx.x; j < R; j += blockDim.x) {
      const float x = uS[j], y = uL[j];
      a = fmaxf(a, x);
      b = fmaxf(b, y);
      if (staged) { eSs[j] = x; eLs[j] = y; }
    }
    const float2 mx = block_max2(a, b, sh.redf);
    PosGlobal pg{p.block + (size_t)slot * p.block_width + m.n_pre_pages, p.tok_pos, p.P, p.L, p.Hk,
                 layer, h, p.num_pages};
    // fixed-point total masses; the staged path stages e_j in the same loop
    // (the sums' barriers also publish the staged rows)
    unsigned long long TS = 0ull, TL = 0ull;
    for (int j = threadIdx.x; j < R; j += blockDim.x) {
      const float eS = expf((staged ? eSs[j] : uS[j]) - mx.x), eL = expf((staged ? eLs[j] : uL[j]) - mx.y);
      TS += mass_q(eS);
      TL += mass_q(eL);
      if (staged) { eSs[j] = eS; eLs[j] = eL; }
    }
    if (staged)
      for (int s = threadIdx.x; s < C; s += blockDim.x) poss[s] = pg(s);
    block_sum2_ull(TS, TL, sh.red);
    // rows of up to half the staging size leave the upper halves of the two
    // e_j arrays free: the first Top-p pass keeps its per-warp bins there
    const bool wide = staged && R <= kSelSmemTok / 2 && 2 * T / 32 * 128 <= kSelSmemTok / 2;
    if (staged)
      select_item(p, i, slot, row, m, R, ESmem{eSs}, ESmem{eLs}, TS, TL, PosSmem{poss}, C, pos,
                  nfree, replan != 0, sh,
                  wide ? reinterpret_cast<uint32_t*>(eSs + kSelSmemTok / 2) : nullptr,
                  wide ? reinterpret_cast<uint32_t*>(eLs + kSelSmemTok / 2) : nullptr);
    else
      select_item(p, i, slot, row, m, R, EGlobal{uS, mx.x}, EGlobal{uL, mx.y}, TS, TL, pg, C, pos,
                  nfree, replan != 0, sh);
  }
}

// -------------------------------------------------------------- decide ---

// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", 2014): the output for state x.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void __launch_bounds__(1024) decide_kernel(PoolDev p, int part) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int s_warp[33];
  __shared__ int s_avail;
  __shared__ unsigned long long s_cnt[6];
  const int n = p.plan_misc[0];
  if (threadIdx.x < 6) s_cnt[threadIdx.x] = 0ull;
  __syncthreads();
  for (int base = 0; base < n; base += blockDim.x) {
    if (threadIdx.x == 0) s_avail = p.ctrl->free_top;
    __syncthreads();
    const int avail = s_avail;
    const int i = base + threadIdx.x;
    int wg = 0, want = 0, at_b = 0, slot = 0;
    gp_req_meta m;
    bool mine = false;
    if (i < n) {
      slot = p.plan_slot[i];
      at_b = (p.plan_flags[i] & kPlanBoundary) != 0;
      mine = part == kPartAll || (part == kPartBoundary) == (at_b != 0);
      if (part == kPartPlain && at_b) p.busy[slot] = 1;  // its work goes to the second stream
    }
    if (mine) {
      m = p.req[slot];
      if (at_b) {
        const double delta = (double)p.plan_delta[i];
        switch (p.mode) {
          case GP_MODE_GROWPAGE:
          case GP_MODE_SHRINK: want = delta > (double)p.tau; break;
          case GP_MODE_FULL_KV: want = 1; break;
          case GP_MODE_FIXED: want = 0; break;
          case GP_MODE_INVERSE: want = -delta > (double)p.tau; break;
          default: {  // GP_MODE_RANDOM
            const uint64_t x = ((uint64_t)(uint32_t)slot << 32) | (uint32_t)m.n_boundaries;
            want = (double)(splitmix64(x) >> 11) * 0x1p-53 < (double)p.random_grow_rate;
          }
        }
        wg = (want && m.n_pages < p.max_pages_per_req) ? 1 : 0;
      }
    }
    int total;
    const int rank = block_excl_scan(wg, s_warp, &total);
    if (mine) {
      const int C = m.n_pages * p.P;
      int dec, commit;
      if (wg && rank < avail) {
        const int page = p.free_stack[avail - 1 - rank];
        p.block[(size_t)slot * p.block_width + m.n_pre_pages + m.n_pages] = page;
        m.n_pages += 1;
        dec = kGrow; commit = C;
        m.n_grows += 1;
        atomicAdd(&s_cnt[1], 1ull);
      } else if (at_b) {
        if (p.mode == GP_MODE_SHRINK && !want && m.n_pages >= 2 &&
            (m.n_pages - 2) * p.P >= p.recent_window) {
          // release the last private page (pushed after this step's grows)
          dec = kShrink;
          commit = C - 2 * p.P;
          m.n_pages -= 1;
          m.n_shrinks += 1;
          atomicAdd(&s_cnt[5], 1ull);
        } else if (p.mode != GP_MODE_FULL_KV) {
          dec = want ? kCompactDenied : kCompact;
          commit = C - p.P;
          m.n_compacts += 1;
          atomicAdd(&s_cnt[2], 1ull);
          if (want) { m.n_denied += 1; atomicAdd(&s_cnt[3], 1ull); }
        } else {
          // full KV and no page (none free, or the request at its cap): the
          // step's token is dropped; counted, not a fault
          dec = kStarved; commit = -1;
          m.n_starved += 1;
          atomicAdd(&s_cnt[4], 1ull);
        }
      } else {
        dec = kNone; commit = m.seq_priv;
      }
      if (at_b) {
        m.n_boundaries += 1;
        m.last_decision = dec;
        m.delta = p.plan_delta[i];
        atomicAdd(&s_cnt[0], 1ull);
      }
      p.plan_dec[i] = dec;
      p.plan_commit[i] = commit;
      p.plan_cpos[i] = m.pos;
      if (commit >= 0) m.seq_priv = commit + 1;
      m.pos += 1;
      m.steps += 1;
      p.req[slot] = m;
    }
    __syncthreads();
    if (threadIdx.x == 0 && part != kPartPlain) {  // the plain part never pops
      const int g = total < avail ? total : avail;
      atomicSub(&p.ctrl->free_top, g);
    }
    __syncthreads();
  }
  // Pages released by SHRINK go on the free stack after every pop of the
  // step, in ascending slot order: a page released now is not handed out
  // before the next step (its tokens are still read by the commit's moves).
  if (p.mode == GP_MODE_SHRINK && part != kPartPlain) {
    for (int base = 0; base < n; base += blockDim.x) {
      if (threadIdx.x == 0) s_avail = p.ctrl->free_top;
      __syncthreads();
      const int top = s_avail;
      const int i = base + threadIdx.x;
      const int sh = (i < n && p.plan_dec[i] == kShrink) ? 1 : 0;
      int total;
      const int rank = block_excl_scan(sh, s_warp, &total);
      if (sh) {
        const int slot = p.plan_slot[i];
        const gp_req_meta& m = p.req[slot];
        // the released page still sits in the block table, just past the
        // request's (already reduced) page count
        p.free_stack[top + rank] = p.block[(size_t)slot * p.block_width + m.n_pre_pages + m.n_pages];
      }
      __syncthreads();
      if (threadIdx.x == 0) p.ctrl->free_top = top + total;
      __syncthreads();
    }
  }
  if (threadIdx.x == 0 && part != kPartPlain) {  // the two parts may run concurrently
    atomicAdd((unsigned long long*)&p.ctrl->boundaries, s_cnt[0]);
    atomicAdd((unsigned long long*)&p.ctrl->grows, s_cnt[1]);
    atomicAdd((unsigned long long*)&p.ctrl->compacts, s_cnt[2]);
    atomicAdd((unsigned long long*)&p.ctrl->denied, s_cnt[3]);
    atomicAdd((unsigned long long*)&p.ctrl->starved, s_cnt[4]);
    atomicAdd((unsigned long long*)&p.ctrl->shrinks, s_cnt[5]);
  }
}

// End of a step's boundary work on the second stream: its requests may take
// part in steps again.  Runs after the commit kernel has completed, so the
// release makes every write of the boundary work visible to a plan kernel
// that reads the flag with acquire.
__global__ void release_busy_kernel(PoolDev p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = p.plan_misc[0];
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    if (p.plan_flags[i] & kPlanBoundary)
      asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.busy + p.plan_slot[i]), "r"(0)
                   : "memory");
}

// -------------------------------------------------------------- commit ---

__device__ __forceinline__ uint8_t* slot_row(const PoolDev& p, const int32_t* bt, int s, int layer,
                                             int h, int rowb, int* page_out) {
  int page = bt[s / p.P];
  if ((unsigned)page >= (unsigned)p.num_pages) {
    set_status(p, GP_ST_BAD_PAGE, page);
    page = 0;
  }
  *page_out = page;
  return p.kv + (size_t)page * p.page_bytes + (size_t)layer * p.layer_bytes +
         (size_t)h * p.head_bytes + (size_t)(s % p.P) * rowb;
}

__global__ void __launch_bounds__(256, 4) commit_kernel(PoolDev p, int part) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int n = p.plan_misc[0];
  const int rowb = p.D * p.elem_bytes;
  const int chunks = rowb / 16;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int items = n * p.L * p.Hk;
  unsigned long long moved = 0ull;
  for (int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items; item += warps) {
    const int i = item / (p.L * p.Hk);
    const int rem = item % (p.L * p.Hk);
    const int layer = rem / p.Hk, h = rem % p.Hk;
    if (part != kPartAll &&
        (part == kPartBoundary) != ((p.plan_flags[i] & kPlanBoundary) != 0))
      continue;
    const int slot = p.plan_slot[i];
    const int dec = p.plan_dec[i];
    const int commit = p.plan_commit[i];
    const int npre = p.req[slot].n_pre_pages;
    const int32_t* bt = p.block + (size_t)slot * p.block_width + npre;
    const size_t row = ((size_t)slot * p.L + layer) * p.Hk + h;
    if (p.summary_via_next && (p.plan_flags[i] & kPlanScore)) {
      // the folded summaries of a request at a boundary become current (the
      // attention kernel wrote every other request's in place)
      const float4* src = reinterpret_cast<const float4*>(p.summary_next + row * 2 * p.D);
      float4* dst = reinterpret_cast<float4*>(p.summary + row * 2 * p.D);
      for (int c = lane; c < 2 * p.D / 4; c += 32) dst[c] = src[c];
    }
    if (dec == kCompact || dec == kCompactDenied || dec == kShrink) {
      // Four moves at a time, eight lanes each, every load of a group issued
      // before its stores.  Moves never overlap: holes lie below C - P and
      // survivors at or above it.
      const int nm = p.moves_n[row];
      const int32_t* mv = p.moves + row * (size_t)p.P * 4;
      const int sub = lane & 7;
      for (int base = 0; base < nm; base += 4) {
        const int t = base + (lane >> 3);
        if (t < nm) {
          const int dst = mv[2 * t], src = mv[2 * t + 1];
          int pd, ps;
          uint8_t* rd = slot_row(p, bt, dst, layer, h, rowb, &pd);
          const uint8_t* rs = slot_row(p, bt, src, layer, h, rowb, &ps);
          const int per = chunks / 8;  // 2 or 4 chunks per lane, two at a time
          int tpos = 0;
          if (sub == 0) tpos = p.tok_pos[(((size_t)ps * p.L + layer) * p.Hk + h) * p.P + (src % p.P)];
          for (int j0 = 0; j0 < per; j0 += 2) {
            uint4 kx[2], vx[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              kx[j] = *reinterpret_cast<const uint4*>(rs + 16 * (sub + 8 * (j0 + j)));
              vx[j] = *reinterpret_cast<const uint4*>(rs + p.half_bytes + 16 * (sub + 8 * (j0 + j)));
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              *reinterpret_cast<uint4*>(rd + 16 * (sub + 8 * (j0 + j))) = kx[j];
              *reinterpret_cast<uint4*>(rd + p.half_bytes + 16 * (sub + 8 * (j0 + j))) = vx[j];
            }
          }
          if (sub == 0) p.tok_pos[(((size_t)pd * p.L + layer) * p.Hk + h) * p.P + (dst % p.P)] = tpos;
        }
      }
      moved += (unsigned long long)nm;
    }
    __syncwarp();
    if (commit >= 0) {
      int pg;
      uint8_t* rd = slot_row(p, bt, commit, layer, h, rowb, &pg);
      const uint8_t* st = p.staging + row * 2 * rowb;
      for (int c = lane; c < chunks; c += 32) {
        *reinterpret_cast<uint4*>(rd + 16 * c) = *reinterpret_cast<const uint4*>(st + 16 * c);
        *reinterpret_cast<uint4*>(rd + p.half_bytes + 16 * c) =
            *reinterpret_cast<const uint4*>(st + rowb + 16 * c);
      }
      if (lane == 0)
        p.tok_pos[(((size_t)pg * p.L + layer) * p.Hk + h) * p.P + (commit % p.P)] = p.plan_cpos[i];
    }
  }
  if (lane == 0 && moved) atomicAdd((unsigned long long*)&p.ctrl->moved_tokens, moved);
}

// --------------------------------------------------------------- admin ---

__global__ void init_kernel(PoolDev p) {
  const int stride = gridDim.x * blockDim.x;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < p.num_pages; j += stride)
    p.free_stack[j] = p.num_pages - 1 - j;  // top holds page 0
  if (blockIdx.x == 0 && threadIdx.x == 0) p.ctrl->free_top = p.num_pages;
}

// Pop `count` pages (the host checked availability) into dst[0..count).
__global__ void pop_pages_kernel(PoolDev p, int32_t* dst, int count) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int top = p.ctrl->free_top;
  for (int k = 0; k < count; ++k) dst[k] = p.free_stack[--top];
  p.ctrl->free_top = top;
}

__global__ void prefix_meta_kernel(PoolDev p, int pid, int npages, int len) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  gp_prefix_meta m;
  m.refs = 1; m.n_pages = npages; m.len = len; m.reserved = 0;
  p.prefix[pid] = m;
}

// New request: block-table row = prefix pages + budget private pages.
__global__ void admit_kernel(PoolDev p, int slot, int budget, int prefix_id, int prompt_len) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int32_t* bt = p.block + (size_t)slot * p.block_width;
  int npre = 0, plen = 0;
  if (prefix_id >= 0) {
    gp_prefix_meta& pm = p.prefix[prefix_id];
    npre = pm.n_pages;
    plen = pm.len;
    for (int k = 0; k < npre; ++k) bt[k] = p.prefix_pages[(size_t)prefix_id * p.max_prefix_pages + k];
    pm.refs += 1;
  }
  int top = p.ctrl->free_top;
  for (int k = 0; k < budget; ++k) bt[npre + k] = p.free_stack[--top];
  p.ctrl->free_top = top;
  gp_req_meta m = {};
  m.active = 1;
  m.prefix_id = prefix_id;
  m.n_pre_pages = npre;
  m.n_pages = budget;
  m.seq_priv = prompt_len;
  m.pos = plen + prompt_len;
  p.req[slot] = m;
}

// Store tokens 0..count-1 of k, v ([L][count][Hk][d], keys not yet rotated)
// into the pages listed in `pages` (token t -> page t/P, slot t%P), keys
// rotated to position pos0 + t in fp64 and rounded once to the dtype (bf16:
// by rope_bf16_certified, which gives the same bits without fp64 arithmetic
// except for the rare pairs it leaves open).
template <typename T>
__global__ void write_tokens_kernel(PoolDev p, const int32_t* pages, const T* k, const T* v,
                                    int count, int pos0) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int D = p.D, H = D / 2;
  const long long items = (long long)p.L * count * p.Hk;
  for (long long it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
    const int layer = (int)(it / ((long long)count * p.Hk));
    const int rem = (int)(it % ((long long)count * p.Hk));
    const int t = rem / p.Hk, h = rem % p.Hk;
    int page = pages[t / p.P];
    if ((unsigned)page >= (unsigned)p.num_pages) { set_status(p, GP_ST_BAD_PAGE, page); continue; }
    T* dst = reinterpret_cast<T*>(p.kv + (size_t)page * p.page_bytes + (size_t)layer * p.layer_bytes +
                                  (size_t)h * p.head_bytes) + (size_t)(t % p.P) * D;
    T* dstv = reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(dst) + p.half_bytes);
    const T* src = k + (((size_t)layer * count + t) * p.Hk + h) * D;
    const T* srcv = v + (((size_t)layer * count + t) * p.Hk + h) * D;
    const int pos = pos0 + t;
    for (int e = lane; e < H; e += 32) {
      if constexpr (sizeof(T) == 2) {
        if (p.rope) {  // the certified fp32 evaluation of the fp64 expression below
          const float x = ElemIO<T>::load(src, e), y = ElemIO<T>::load(src, e + H);
          const float c1 = rope_c32(p, pos)[e], c2 = rope_c32lo(p, pos)[e];
          const float s1 = rope_s32(p, pos)[e], s2 = rope_s32lo(p, pos)[e];
          uint16_t ra, rb;
          if (rope_bf16_certified(x, y, c1, c2, -s1, -s2, ra) &&
              rope_bf16_certified(y, x, c1, c2, s1, s2, rb)) {
            reinterpret_cast<uint16_t*>(dst)[e] = ra;
            reinterpret_cast<uint16_t*>(dst)[e + H] = rb;
            continue;
          }
        }
      }
      const double x = (double)ElemIO<T>::load(src, e), y = (double)ElemIO<T>::load(src, e + H);
      double a = x, b = y;
      if (p.rope) {
        const double c = rope_c64(p, pos)[e], s = rope_s64(p, pos)[e];
        a = __dsub_rn(__dmul_rn(x, c), __dmul_rn(y, s));
        b = __dadd_rn(__dmul_rn(y, c), __dmul_rn(x, s));
      }
      if constexpr (sizeof(T) == 2) {
        reinterpret_cast<uint16_t*>(dst)[e] = f64_to_bf16_rne(a);
        reinterpret_cast<uint16_t*>(dst)[e + H] = f64_to_bf16_rne(b);
      } else {
        dst[e] = __double2float_rn(a);
        dst[e + H] = __double2float_rn(b);
      }
    }
    for (int e = lane; e < D; e += 32) dstv[e] = srcv[e];
    if (lane == 0) p.tok_pos[(((size_t)page * p.L + layer) * p.Hk + h) * p.P + (t % p.P)] = pos;
  }
}

__global__ void free_kernel(PoolDev p, int slot) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  gp_req_meta& m = p.req[slot];
  const int32_t* bt = p.block + (size_t)slot * p.block_width;
  int top = p.ctrl->free_top;
  for (int k = 0; k < m.n_pages; ++k) p.free_stack[top++] = bt[m.n_pre_pages + k];
  if (m.prefix_id >= 0) {
    gp_prefix_meta& pm = p.prefix[m.prefix_id];
    pm.refs -= 1;
    if (pm.refs == 0)
      for (int k = 0; k < pm.n_pages; ++k)
        p.free_stack[top++] = p.prefix_pages[(size_t)m.prefix_id * p.max_prefix_pages + k];
  }
  p.ctrl->free_top = top;
  m.active = 0;
}

__global__ void release_prefix_kernel(PoolDev p, int pid) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  gp_prefix_meta& pm = p.prefix[pid];
  pm.refs -= 1;
  if (pm.refs == 0) {
    int top = p.ctrl->free_top;
    for (int k = 0; k < pm.n_pages; ++k)
      p.free_stack[top++] = p.prefix_pages[(size_t)pid * p.max_prefix_pages + k];
    p.ctrl->free_top = top;
  }
}

// ------------------------------------------------------------ launchers ---

// The per-step kernels are launched as programmatic dependents of the kernel
// before them in the stream (each waits for it with griddepcontrol.wait
// before touching memory), so a launch overlaps its predecessor's tail.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

cudaError_t launch_plan(const PoolDev& p, int n, const int32_t* slots, int count, cudaStream_t st) {
  return launch_pdl(plan_kernel, 1, 1024, 0, st, p, n, slots, count);
}
constexpr int kSelBigThreads = 512;
cudaError_t select_setup() {
  cudaError_t e = cudaFuncSetAttribute(select_kernel<kSelThreads, GP_SEL_MINB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(select_kernel<kSelBigThreads, 2>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelSmemBytes);
}
cudaError_t select_occupancy(int* blocks, bool big) {
  return big ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, select_kernel<kSelBigThreads, 2>,
                                                             kSelBigThreads, kSelSmemBytes)
             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, select_kernel<kSelThreads, GP_SEL_MINB>,
                                                             kSelThreads, kSelSmemBytes);
}
cudaError_t launch_select(const PoolDev& p, int grid, int replan, bool big, cudaStream_t st) {
  return big ? launch_pdl(select_kernel<kSelBigThreads, 2>, grid, kSelBigThreads, kSelSmemBytes, st, p,
                          replan)
             : launch_pdl(select_kernel<kSelThreads, GP_SEL_MINB>, grid, kSelThreads, kSelSmemBytes, st, p,
                          replan);
}
cudaError_t launch_decide(const PoolDev& p, int part, cudaStream_t st) {
  return launch_pdl(decide_kernel, 1, 1024, 0, st, p, part);
}
cudaError_t launch_commit(const PoolDev& p, int grid, int part, cudaStream_t st) {
  return launch_pdl(commit_kernel, grid, 256, 0, st, p, part);
}
cudaError_t launch_release_busy(const PoolDev& p, cudaStream_t st) {
  return launch_pdl(release_busy_kernel, 1, 256, 0, st, p);
}
cudaError_t launch_init(const PoolDev& p, cudaStream_t st) {
  init_kernel<<<256, 256, 0, st>>>(p);
  return cudaGetLastError();
}
cudaError_t launch_pop_pages(const PoolDev& p, int32_t* dst, int count, cudaStream_t st) {
  pop_pages_kernel<<<1, 32, 0, st>>>(p, dst, count);
  return cudaGetLastError();
}
cudaError_t launch_prefix_meta(const PoolDev& p, int pid, int npages, int len, cudaStream_t st) {
  prefix_meta_kernel<<<1, 32, 0, st>>>(p, pid, npages, len);
  return cudaGetLastError();
}
cudaError_t launch_admit(const PoolDev& p, int slot, int budget, int prefix_id, int prompt_len,
                         cudaStream_t st) {
  admit_kernel<<<1, 32, 0, st>>>(p, slot, budget, prefix_id, prompt_len);
  return cudaGetLastError();
}
cudaError_t launch_write_tokens(const PoolDev& p, const int32_t* pages, const void* k, const void* v,
                                int count, int pos0, cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  const long long items = (long long)p.L * count * p.Hk;
  long long blocks = (items + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  if (p.dtype == GP_DTYPE_BF16)
    write_tokens_kernel<__nv_bfloat16><<<(int)blocks, 256, 0, st>>>(
        p, pages, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, count, pos0);
  else
    write_tokens_kernel<float><<<(int)blocks, 256, 0, st>>>(p, pages, (const float*)k,
                                                            (const float*)v, count, pos0);
  return cudaGetLastError();
}
cudaError_t launch_free(const PoolDev& p, int slot, cudaStream_t st) {
  free_kernel<<<1, 32, 0, st>>>(p, slot);
  return cudaGetLastError();
}
cudaError_t launch_release_prefix(const PoolDev& p, int pid, cudaStream_t st) {
  release_prefix_kernel<<<1, 32, 0, st>>>(p, pid);
  return cudaGetLastError();
}

}  // namespace gp
