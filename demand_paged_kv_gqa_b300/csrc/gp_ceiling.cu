// gp_ceiling.cu -- read-only streaming of a layer's resident K/V: the
// bandwidth ceiling the attention kernel is measured against.
//
// kv_read_kernel walks exactly the blocks the bf16 attention kernel walks for
// one layer (same persistent grid, same per-warp split, the same one-copy
// tensor-map loads of a block into a per-warp ring of stages) but does no
// arithmetic: it folds one word of each stage into a checksum so the copies
// cannot be elided.
//   mode 0  paged:       the request's own pages, in block-table order;
//   mode 1  sequential:  the same number of 8 KiB blocks, taken in address
//                        order from the start of the K/V region (TMA);
//   mode 2  sequential:  the same bytes read with plain 16-byte loads.
// The three together separate the cost of the paged access pattern from the
// cost of the arithmetic.  Not part of the decode path.
#include <cuda.h>

#include "gp_attn_common.cuh"

namespace gp {

constexpr int kCeilWarps = 4;
constexpr int kCeilStages = 3;
constexpr int kCeilStageB = 8192;

// A 16-token block (K and V, both 64-column halves) of row index
// (page * L + layer) * Hk + head, token offset tok, through the pool's 5-D
// block map: one copy.
__device__ __forceinline__ void tma_block(void* dst, const CUtensorMap* map, int tok, int prow,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(tok), "r"(0), "r"(0), "r"(prow),
      "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kCeilWarps * 32)
kv_read_kernel(const __grid_constant__ CUtensorMap kvblk, PoolDev p, int layer, int mode,
               uint32_t* sink) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int S = kCeilStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + (size_t)warp * S * kCeilStageB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kCeilWarps * S * kCeilStageB) + warp * S;
  const int n = p.plan_misc[0];
  const int64_t Tb = (int64_t)p.plan_misc[2] * p.Hk;
  const int64_t W = (int64_t)p.num_workers;
  const int64_t Weff = W < Tb ? W : Tb;
  const int64_t w = (int64_t)blockIdx.x * kCeilWarps + warp;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const unsigned long long bytes = (unsigned long long)Tb * kCeilStageB;
    sink[2] = (uint32_t)bytes;
    sink[3] = (uint32_t)(bytes >> 32);
  }
  if (n <= 0 || w >= Weff) return;
  const int64_t start = p.wblk[w], end = p.wblk[w + 1];  // the attention kernel's shares
  if (start >= end) return;
  uint32_t acc = 0u;
  // sequential modes wrap inside the K/V region (it holds num_pages * L * Hk blocks)
  const int64_t region_blocks = (int64_t)p.num_pages * p.L * p.Hk * (p.P / kBlockTok);
  if (mode == 2) {
    const uint4* base = reinterpret_cast<const uint4*>(p.kv);
    for (int64_t b = start; b < end; ++b) {
      const uint4* blk = base + (b % region_blocks) * (kCeilStageB / 16);
      uint4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = __ldcs(blk + lane + 32 * u);
#pragma unroll
      for (int u = 0; u < 16; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
  } else {
    if (lane == 0) {
      for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
      fence_barrier_init();
    }
    __syncwarp();
    Cursor pc;
    cursor_start(p, w, pc);
    PageWin win;
    int64_t issued = start;
    const int bpp = p.P / kBlockTok;  // blocks per page
    auto issue = [&](int s) {
      int prow, tok;
      if (mode == 0) {
        const int page = page_of(p, win, pc, lane);
        prow = (page * p.L + layer) * p.Hk + pc.h;
        tok = (pc.blk * kBlockTok) % p.P;
      } else {
        const int64_t b = issued % region_blocks;
        prow = (int)(b / bpp);
        tok = (int)(b % bpp) * kBlockTok;
      }
      if (lane == 0) {
        fence_proxy_async_smem();
        mbar_expect_tx(&bars[s], kCeilStageB);
        tma_block(ring + s * kCeilStageB, &kvblk, tok, prow, &bars[s]);
      }
      if (issued + 1 < end) cursor_next(p, pc);
      ++issued;
    };
    for (int s = 0; s < S && issued < end; ++s) issue(s);
    for (int64_t j = start; j < end; ++j) {
      const int64_t jl = j - start;
      const int s = (int)(jl % S);
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars[s], (uint32_t)((jl / S) & 1), kWaitLimitNs))) {
        if (lane == 0) set_status(p, GP_ST_TIMEOUT, -1);
        for (int64_t k = jl + 1; k < issued - start; ++k)
          (void)mbar_wait_bounded(&bars[k % S], (uint32_t)((k / S) & 1), kWaitLimitNs);
        break;
      }
      acc ^= reinterpret_cast<const uint32_t*>(ring + s * kCeilStageB)[lane * 64];
      __syncwarp();
      if (issued < end) issue(s);
    }
  }
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 16);
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 8);
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 4);
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 2);
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 1);
  if (lane == 0) atomicXor(sink, acc);
}

size_t ceiling_smem_bytes() {
  return (size_t)kCeilWarps * kCeilStages * kCeilStageB + (size_t)kCeilWarps * kCeilStages * 8 + 1024;
}

cudaError_t ceiling_setup() {
  return cudaFuncSetAttribute(kv_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)ceiling_smem_bytes());
}

int ceiling_warps_per_cta() { return kCeilWarps; }

cudaError_t launch_kv_read(const PoolDev& p, const CUtensorMap* map, int layer, int mode,
                           uint32_t* sink, int grid, cudaStream_t st) {
  kv_read_kernel<<<grid, kCeilWarps * 32, ceiling_smem_bytes(), st>>>(*map, p, layer, mode, sink);
  return cudaGetLastError();
}

}  // namespace gp
