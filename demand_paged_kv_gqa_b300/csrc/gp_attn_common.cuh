// gp_attn_common.cuh -- pieces shared by the two attention kernels.
//
// Work decomposition (both kernels): the resident tokens of every
// (request, kv head) are cut into 16-token blocks; all blocks of a layer
// launch are laid end to end and split into contiguous ranges, one per warp
// of a persistent grid: equal ranges for the fp32 kernel, ranges weighted by
// (request, head) starts for the bf16 kernel (the plan kernel computes both).
// A Cursor walks that sequence.
#pragma once

#include "gp_internal.cuh"

namespace gp {

template <typename T, int D>
struct Geo {
  static constexpr int EB = (int)sizeof(T);
  static constexpr int EPC = 16 / EB;            // elements per 16-byte chunk
  static constexpr int ROWB = D * EB;            // bytes of one token row
  static constexpr int VEC = ROWB / (8 * 16);    // 16-byte chunks per lane per row
  static constexpr int NE = VEC * EPC;           // elements per lane per row
  static constexpr int BLKB = kBlockTok * ROWB;  // 16 rows
  static constexpr int STAGEB = 2 * BLKB;        // K block + V block
  static_assert(VEC == 2 || VEC == 4, "unsupported (dtype, head_dim)");
};

// Lane slice `sigma` (0..7) holds, of each row, the 16-byte chunks
// c*8 + sigma, c < VEC.  Chunk c < VEC/2 lies in the first half of the row and
// chunk c + VEC/2 holds its rotate-half partners, so RoPE is lane-local, and
// 8 lanes reading one row touch 128 contiguous bytes (no bank conflicts).
template <class Gm>
__device__ __forceinline__ int dim_of(int e, int sigma) {
  return ((e / Gm::EPC) * 8 + sigma) * Gm::EPC + (e % Gm::EPC);
}

template <typename T, class Gm>
__device__ __forceinline__ void load_row(const uint8_t* row, int sigma, float (&f)[Gm::NE]) {
#pragma unroll
  for (int c = 0; c < Gm::VEC; ++c) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + (c * 8 + sigma) * 16);
    if constexpr (sizeof(T) == 2) {
      f[c * 8 + 0] = bf16lo(w.x); f[c * 8 + 1] = bf16hi(w.x);
      f[c * 8 + 2] = bf16lo(w.y); f[c * 8 + 3] = bf16hi(w.y);
      f[c * 8 + 4] = bf16lo(w.z); f[c * 8 + 5] = bf16hi(w.z);
      f[c * 8 + 6] = bf16lo(w.w); f[c * 8 + 7] = bf16hi(w.w);
    } else {
      f[c * 4 + 0] = __uint_as_float(w.x); f[c * 4 + 1] = __uint_as_float(w.y);
      f[c * 4 + 2] = __uint_as_float(w.z); f[c * 4 + 3] = __uint_as_float(w.w);
    }
  }
}

template <typename T, class Gm>
__device__ __forceinline__ void store_row(T* row, int sigma, const float (&f)[Gm::NE]) {
#pragma unroll
  for (int e = 0; e < Gm::NE; ++e) {
    const int dd = dim_of<Gm>(e, sigma);
    if constexpr (sizeof(T) == 2) row[dd] = __float2bfloat16_rn(f[e]);
    else row[dd] = f[e];
  }
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per bounded wait

// Block `blk` of (request i, kv head h) covers the request's resident tokens
// base + 16*blk .. base + 16*blk + 15 (base: a shared prefix attended
// elsewhere, else 0).
struct Cursor {
  int i, h, blk, nb, slot, base;
};

__device__ __forceinline__ int find_req(const int32_t* cum, int n, int64_t x) {
  // largest i in [0, n) with cum[i] <= x
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((int64_t)cum[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void cursor_at(const PoolDev& p, int n, int64_t b, Cursor& c) {
  const int i = find_req(p.plan_cum, n, b / p.Hk);
  const int nb = p.plan_nb[i];
  const int64_t r = b - (int64_t)p.Hk * p.plan_cum[i];
  c.i = i; c.nb = nb; c.h = (int)(r / nb); c.blk = (int)(r % nb); c.slot = p.plan_slot[i];
  c.base = p.plan_base[i];
}

// Cursor at worker w's first block, as the plan kernel laid it out.
__device__ __forceinline__ void cursor_start(const PoolDev& p, int64_t w, Cursor& c) {
  const int4 s = p.wstart[w];
  c.i = s.x; c.h = s.y >> 20; c.blk = s.y & 0xfffff; c.nb = s.z; c.slot = s.w;
  c.base = p.plan_base[s.x];
}

// 32 consecutive block-table entries of one request, one per lane, so that
// the page of the next block is a register shuffle instead of a dependent
// global load.  All lanes must call page_of with the same cursor.
struct PageWin {
  int slot = -1, base = 0, page = 0;
};

__device__ __forceinline__ int page_of(const PoolDev& p, PageWin& win, const Cursor& c, int lane) {
  const int pidx = (c.base + c.blk * kBlockTok) / p.P;  // entry: prefix pages first, then private
  if (c.slot != win.slot || pidx < win.base || pidx >= win.base + 32) {
    win.slot = c.slot;
    win.base = pidx;
    const int e = pidx + lane;
    win.page = e < p.block_width ? p.block[(size_t)c.slot * p.block_width + e] : 0;
  }
  int page = __shfl_sync(0xffffffffu, win.page, pidx - win.base);
  if ((unsigned)page >= (unsigned)p.num_pages) {
    if (lane == 0) set_status(p, GP_ST_BAD_PAGE, c.slot);
    page = 0;
  }
  return page;
}

__device__ __forceinline__ void cursor_next(const PoolDev& p, Cursor& c) {
  if (++c.blk == c.nb) {
    c.blk = 0;
    if (++c.h == p.Hk) {
      c.h = 0; ++c.i;
      c.nb = p.plan_nb[c.i]; c.slot = p.plan_slot[c.i]; c.base = p.plan_base[c.i];
    }
  }
}

}  // namespace gp
