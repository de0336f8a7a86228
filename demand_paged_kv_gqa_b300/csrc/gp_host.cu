// gp_host.cu -- the C ABI (include/growpage.h): validation, layout of the
// caller's buffer, host-side bookkeeping and kernel launches.
//
// The library never allocates device memory: every region, scratch included,
// lives in the buffer the caller passes to gp_create_pool.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gp_internal.cuh"

namespace gp {
cudaError_t launch_attention(const PoolDev& p, int layer, const void* q, const void* k,
                             const void* v, void* out, int grid, cudaStream_t st);
cudaError_t attention_occupancy(const PoolDev& p, int* blocks);
cudaError_t launch_attention_mma(const PoolDev& p, const CUtensorMap* map, int layer, int n,
                                 const void* q, const void* k, const void* v, void* out, int grid,
                                 bool prefix, cudaStream_t st);
cudaError_t attention_mma_occupancy(const PoolDev& p, int* blocks);
int attention_mma_launches(bool prefix);
int mma_warps_per_cta();
cudaError_t launch_plan(const PoolDev& p, int n, const int32_t* slots, int count, cudaStream_t st);
cudaError_t ceiling_setup();
int ceiling_warps_per_cta();
cudaError_t launch_kv_read(const PoolDev& p, const CUtensorMap* map, int layer, int mode,
                           uint32_t* sink, int grid, cudaStream_t st);
cudaError_t launch_select(const PoolDev& p, int grid, int replan, bool big, cudaStream_t st);
cudaError_t select_setup();
cudaError_t select_occupancy(int* blocks, bool big);
cudaError_t launch_decide(const PoolDev& p, int part, cudaStream_t st);
cudaError_t launch_commit(const PoolDev& p, int grid, int part, cudaStream_t st);
cudaError_t launch_release_busy(const PoolDev& p, cudaStream_t st);
cudaError_t launch_init(const PoolDev& p, cudaStream_t st);
cudaError_t launch_pop_pages(const PoolDev& p, int32_t* dst, int count, cudaStream_t st);
cudaError_t launch_prefix_meta(const PoolDev& p, int pid, int npages, int len, cudaStream_t st);
cudaError_t launch_admit(const PoolDev& p, int slot, int budget, int prefix_id, int prompt_len,
                         cudaStream_t st);
cudaError_t launch_write_tokens(const PoolDev& p, const int32_t* pages, const void* k,
                                const void* v, int count, int pos0, cudaStream_t st);
cudaError_t launch_free(const PoolDev& p, int slot, cudaStream_t st);
cudaError_t launch_release_prefix(const PoolDev& p, int pid, cudaStream_t st);
}  // namespace gp

struct gp_pool {
  CUtensorMap kvblk;  // (64-byte aligned type) K/V pages as 5-D boxes of one 16-token block
                      // (K and V, both column halves), 128-byte swizzle
  bool use_mma = false;           // bf16 pages, head_dim 128: tensor-core kernel
  gp_config cfg;
  gp::PoolDev dev;
  gp_layout lay;
  uint8_t* base = nullptr;
  cudaStream_t stream = nullptr;
  std::string err;
  int next_layer = 0;
  int step_n = -1;
  const int32_t* step_slots = nullptr;
  int attn_grid = 0, select_grid = 0, select_grid_big = 0, commit_grid = 0;
  int64_t launches = 0;
  std::vector<char> slot_active;
  std::vector<int> slot_prefix;
  std::vector<int> prefix_refs;  // host mirror of the device reference counts
  std::vector<char> prefix_held;
  std::vector<int> prefix_len;
  int prefixed_active = 0;  // active requests that use a shared prefix
  // Plan buffers: steps alternate between two, so that a step's boundary
  // work on a second stream (gp_boundary_async) can still read its own plan
  // while the next step runs.  plan_set[b][k] / delta_set[b] are buffer b's
  // twelve plan arrays and Delta accumulators; `parity` is the current one.
  int32_t* plan_set[2][12] = {};
  long long* delta_set[2] = {};
  int parity = 0;
  cudaEvent_t side_ev[2] = {nullptr, nullptr};  // boundary work of a buffer's step done
  bool side_pending[2] = {false, false};
  cudaEvent_t main_ev = nullptr;                // the plain part of a boundary done
};

// Work of starting a (request, head) segment in the bf16 attention kernel
// (meta item, operand rows, staged token), in blocks' worth: the plan
// weighs it when it splits the blocks between workers.
#ifndef GP_SEG_COST
#define GP_SEG_COST 4
#endif

namespace {

constexpr uint64_t kAlign = 256;

uint64_t align_up(uint64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int fail(gp_pool* p, int code, const std::string& msg) {
  if (p) p->err = msg;
  return code;
}

int cuda_fail(gp_pool* p, cudaError_t e, const char* what) {
  return fail(p, GP_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Shared prefixes are attended once per group of requests (bf16 pages,
// head_dim 128, the tensor-core path) when the pool holds prefixes.  Built
// with GP_PREFIX_BATCH=0, every request attends its prefix itself.
#ifndef GP_PREFIX_BATCH
#define GP_PREFIX_BATCH 1
#endif
bool prefix_batch_on(const gp_config* c) {
  return GP_PREFIX_BATCH && c->dtype == GP_DTYPE_BF16 && c->head_dim == 128 && c->max_prefixes > 0 &&
         c->max_prefixes <= gp::kMaxPrefixBatch && c->max_prefix_len > 0;
}
int prefix_ranges_max(const gp_config* c) {
  return (c->max_prefix_len / gp::kBlockTok + gp::kPrefRangeBlocks - 1) / gp::kPrefRangeBlocks;
}

const char* check_config(const gp_config* c) {
  if (!c) return "null config";
  if (c->num_layers < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1) return "bad head/layer counts";
  if (c->num_q_heads % c->num_kv_heads) return "num_q_heads must be a multiple of num_kv_heads";
  const int G = c->num_q_heads / c->num_kv_heads;
  if (G != 1 && G != 2 && G != 4) return "G = Hq/Hk must be 1, 2 or 4";
  if (c->dtype != GP_DTYPE_F32 && c->dtype != GP_DTYPE_BF16) return "unknown dtype";
  if (!((c->head_dim == 64 && c->dtype == GP_DTYPE_F32) || c->head_dim == 128))
    return "head_dim must be 128, or 64 with fp32 storage";
  if (c->page_size < 16 || c->page_size % 16 || c->page_size > 256)
    return "page_size must be a multiple of 16, at most 256";
  if (c->num_pages < 1 || c->max_requests < 1 || c->max_pages_per_req < 1) return "bad pool sizes";
  if (c->max_prefixes < 0 || c->max_prefix_len < 0 || c->max_prefix_len % c->page_size)
    return "max_prefix_len must be a non-negative multiple of page_size";
  if (c->max_seq_len < 1) return "bad max_seq_len";
  if (c->mode < GP_MODE_GROWPAGE || c->mode > GP_MODE_SHRINK) return "unknown mode";
  if (c->mode == GP_MODE_RANDOM && !(c->random_grow_rate >= 0.f && c->random_grow_rate <= 1.f))
    return "random_grow_rate must be in [0, 1]";
  if (c->recent_window < 0) return "recent_window < 0";
  if (!(c->beta_s >= 0.f && c->beta_s < 1.f && c->beta_l >= 0.f && c->beta_l < 1.f))
    return "betas must be in [0, 1)";
  if (!(c->top_p > 0.f && c->top_p <= 1.f)) return "top_p must be in (0, 1]";
  if (!(c->rope_theta >= 0.0)) return "rope_theta < 0";
  if (c->flags != 0) return "flags must be 0";
  const long long logit_w = (long long)c->max_prefix_len + (long long)c->max_pages_per_req * c->page_size;
  if (logit_w > (1ll << 24)) return "max_prefix_len + max_pages_per_req * page_size > 2^24 tokens";
  const long long rows = (long long)c->num_pages * c->num_layers * c->num_kv_heads * 2 * c->page_size;
  if (rows >= (1ll << 31)) return "pool too large: pages x layers x kv heads x 2 x page_size >= 2^31";
  return nullptr;
}

void compute_layout(const gp_config* c, gp_layout* l) {
  const uint64_t eb = c->dtype == GP_DTYPE_BF16 ? 2 : 4;
  const uint64_t L = c->num_layers, Hk = c->num_kv_heads, D = c->head_dim, P = c->page_size;
  const uint64_t G = c->num_q_heads / c->num_kv_heads;
  const uint64_t R = c->max_requests;
  std::memset(l, 0, sizeof(*l));
  l->max_prefix_pages = c->max_prefix_len / c->page_size;
  l->block_width = l->max_prefix_pages + c->max_pages_per_req;
  l->logit_width = c->max_prefix_len + c->max_pages_per_req * c->page_size;
  l->page_bytes = L * Hk * 2 * P * D * eb;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) { uint64_t o = off; off = align_up(off + bytes); return o; };
  l->kv = take((uint64_t)c->num_pages * l->page_bytes);
  l->tok_pos = take((uint64_t)c->num_pages * L * Hk * P * 4);
  l->block = take(R * (uint64_t)l->block_width * 4);
  l->req = take(R * sizeof(gp_req_meta));
  l->summary = take(R * L * Hk * 2 * D * 4);
  l->staging = take(R * L * Hk * 2 * D * eb);
  l->logits = take(c->mode != GP_MODE_FULL_KV ? R * L * Hk * 2 * (uint64_t)l->logit_width * 4 : 0);
  l->wset = take(R * L * Hk * 2 * 4);
  l->free_stack = take((uint64_t)c->num_pages * 4);
  l->ctrl = take(sizeof(gp_ctrl));
  l->prefix = take((uint64_t)c->max_prefixes * sizeof(gp_prefix_meta));
  l->prefix_pages = take((uint64_t)c->max_prefixes * l->max_prefix_pages * 4);
  l->rope = take((uint64_t)c->max_seq_len * (D / 2) * (8 + 8 + 4 + 4 + 4 + 4));
  l->scratch = off;
  for (int b = 0; b < 2; ++b) {                                // two plan buffers
    for (int k = 0; k < 12; ++k) take((R + 1) * 4);           //   plan arrays
    take(R * 8);                                               //   plan_delta
  }
  take((uint64_t)gp::kMaxWorkersBound * 2 * G * (D + 4) * 4);  // partials
  take(R * Hk * 4);                                            // seg_count
  take((uint64_t)gp::kMaxWorkersBound * 16);                   // wstart
  take((uint64_t)(gp::kMaxWorkersBound + 1) * 4);              // wblk
  take(R * Hk * 16);                                           // seginfo
  take(R * L * Hk * 2 * D * 4);                                // summary_next
  take(R * Hk * 4 * 4);                                        // sstage
  take(R * L * Hk * P * 4 * 4);                                // moves (up to 2P pairs)
  take(R * L * Hk * 4);                                        // moves_n
  take(R * 4);                                                 // busy
  if (prefix_batch_on(c)) {                                    // shared prefixes
    const uint64_t NP = c->max_prefixes;
    take(R * 4);                                               //   pmem
    take(R * 4);                                               //   pranges
    take(NP * 4);                                              //   pref_off
    take(NP * 4);                                              //   pref_cnt
    take((NP + 1) * 4);                                        //   unit_cum
    take(R * Hk * (uint64_t)prefix_ranges_max(c) * G * (D + 4) * 4);  // pstate
  }
  l->total = off;
}

void fill_dev(gp_pool* p) {
  const gp_config& c = p->cfg;
  const gp_layout& l = p->lay;
  gp::PoolDev& d = p->dev;
  std::memset(&d, 0, sizeof(d));
  d.L = c.num_layers; d.Hq = c.num_q_heads; d.Hk = c.num_kv_heads; d.D = c.head_dim;
  d.G = c.num_q_heads / c.num_kv_heads; d.P = c.page_size;
  d.P_log2 = -1;
  for (int k = 0; k < 31; ++k)
    if (c.page_size == (1 << k)) d.P_log2 = k;
  d.num_pages = c.num_pages; d.max_req = c.max_requests; d.max_pages_per_req = c.max_pages_per_req;
  d.max_prefixes = c.max_prefixes; d.max_prefix_pages = l.max_prefix_pages;
  d.block_width = l.block_width; d.logit_width = l.logit_width; d.max_seq_len = c.max_seq_len;
  d.dtype = c.dtype; d.mode = c.mode; d.recent_window = c.recent_window;
  d.beta_s = c.beta_s; d.beta_l = c.beta_l; d.top_p = c.top_p; d.tau = c.tau;
  d.random_grow_rate = c.random_grow_rate;
  d.rope = c.rope_theta != 0.0 ? 1 : 0;
  d.elem_bytes = c.dtype == GP_DTYPE_BF16 ? 2 : 4;
  d.half_bytes = (uint64_t)c.page_size * c.head_dim * d.elem_bytes;
  d.head_bytes = 2 * d.half_bytes;
  d.layer_bytes = (uint64_t)c.num_kv_heads * d.head_bytes;
  d.page_bytes = l.page_bytes;
  uint8_t* b = p->base;
  d.kv = b + l.kv;
  d.tok_pos = (int32_t*)(b + l.tok_pos);
  d.block = (int32_t*)(b + l.block);
  d.req = (gp_req_meta*)(b + l.req);
  d.summary = (float*)(b + l.summary);
  d.staging = b + l.staging;
  d.logits = (float*)(b + l.logits);
  d.wset = (int32_t*)(b + l.wset);
  d.free_stack = (int32_t*)(b + l.free_stack);
  d.ctrl = (gp_ctrl*)(b + l.ctrl);
  d.prefix = (gp_prefix_meta*)(b + l.prefix);
  d.prefix_pages = (int32_t*)(b + l.prefix_pages);
  d.rope_rows = b + l.rope;
  d.rope_row_bytes = 16 * c.head_dim;
  const uint64_t R = c.max_requests;
  uint64_t off = l.scratch;
  auto take = [&](uint64_t bytes) { uint64_t o = off; off = align_up(off + bytes); return b + o; };
  for (int b = 0; b < 2; ++b) {
    for (int k = 0; k < 12; ++k) p->plan_set[b][k] = (int32_t*)take((R + 1) * 4);
    p->delta_set[b] = (long long*)take(R * 8);
  }
  d.partials = (float*)take((uint64_t)gp::kMaxWorkersBound * 2 * d.G * (c.head_dim + 4) * 4);
  d.seg_count = (int32_t*)take(R * c.num_kv_heads * 4);
  d.wstart = (int4*)take((uint64_t)gp::kMaxWorkersBound * 16);
  d.wblk = (int32_t*)take((uint64_t)(gp::kMaxWorkersBound + 1) * 4);
  d.seginfo = (int4*)take(R * c.num_kv_heads * 16);
  d.summary_next = (float*)take(R * c.num_layers * c.num_kv_heads * 2 * c.head_dim * 4);
  d.sstage = (float*)take(R * c.num_kv_heads * 4 * 4);
  d.moves = (int32_t*)take(R * c.num_layers * c.num_kv_heads * c.page_size * 4 * 4);
  d.moves_n = (int32_t*)take(R * c.num_layers * c.num_kv_heads * 4);
  d.busy = (int32_t*)take(R * 4);
  if (prefix_batch_on(&c)) {
    const uint64_t NP = c.max_prefixes;
    d.prefix_batch = 1;
    d.max_pranges = prefix_ranges_max(&c);
    d.pmem = (int32_t*)take(R * 4);
    d.pranges = (int32_t*)take(R * 4);
    d.pref_off = (int32_t*)take(NP * 4);
    d.pref_cnt = (int32_t*)take(NP * 4);
    d.unit_cum = (int32_t*)take((NP + 1) * 4);
    d.pstate = (float*)take(R * c.num_kv_heads * (uint64_t)d.max_pranges * d.G * (c.head_dim + 4) * 4);
  }
}

// Point the device view at plan buffer b.
void use_plan(gp_pool* p, int b) {
  gp::PoolDev& d = p->dev;
  int32_t** arrays[12] = {&d.plan_slot, &d.plan_R,      &d.plan_nb,   &d.plan_cum,
                          &d.plan_flags, &d.plan_commit, &d.plan_cpos, &d.plan_dec,
                          &d.plan_bnd,  &d.plan_misc,   &d.plan_pos,  &d.plan_base};
  for (int k = 0; k < 12; ++k) *arrays[k] = p->plan_set[b][k];
  d.plan_delta = p->delta_set[b];
  p->parity = b;
}

// Make the pool's stream wait for every boundary work still pending on a
// second stream (device-side wait, no host sync).
cudaError_t join_side(gp_pool* p) {
  for (int b = 0; b < 2; ++b) {
    if (!p->side_pending[b]) continue;
    cudaError_t e = cudaStreamWaitEvent(p->stream, p->side_ev[b], 0);
    if (e != cudaSuccess) return e;
    p->side_pending[b] = false;
  }
  return cudaSuccess;
}

int sync_status(gp_pool* p) {
  cudaError_t e = cudaStreamSynchronize(p->stream);
  if (e != cudaSuccess) return cuda_fail(p, e, "cudaStreamSynchronize");
  uint32_t st[2] = {0, 0};
  e = cudaMemcpy(st, &p->dev.ctrl->status, 8, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(p, e, "read status");
  if (st[0]) {
    char buf[200];
    std::snprintf(buf, sizeof(buf), "device status 0x%x (info %d):%s%s%s%s%s%s%s", st[0], (int)st[1],
                  (st[0] & GP_ST_BAD_SLOTS) ? " bad-slot-list" : "",
                  (st[0] & GP_ST_BAD_PAGE) ? " page-out-of-range" : "",
                  (st[0] & GP_ST_TIMEOUT) ? " wait-timeout" : "",
                  (st[0] & GP_ST_STARVED) ? " full-kv-starved" : "",
                  (st[0] & GP_ST_BAD_PLAN) ? " bad-plan" : "",
                  (st[0] & GP_ST_POS_RANGE) ? " position-beyond-max_seq_len" : "",
                  (st[0] & GP_ST_SMEM_ALIGN) ? " shared-memory-misaligned" : "");
    return fail(p, GP_ERR_DEVICE, buf);
  }
  return GP_OK;
}

int read_free_top(gp_pool* p, int* out) {
  cudaError_t e = cudaMemcpyAsync(out, &p->dev.ctrl->free_top, 4, cudaMemcpyDeviceToHost, p->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(p->stream);
  if (e != cudaSuccess) return cuda_fail(p, e, "read free_top");
  return GP_OK;
}

#define GP_JOIN(pool)                                                        \
  do {                                                                       \
    cudaError_t _e = join_side(pool);                                        \
    if (_e != cudaSuccess) return cuda_fail(pool, _e, "wait for second stream"); \
  } while (0)

#define GP_LAUNCH(pool, expr)                                   \
  do {                                                          \
    cudaError_t _e = (expr);                                    \
    if (_e != cudaSuccess) return cuda_fail(pool, _e, #expr);   \
    (pool)->launches += 1;                                      \
  } while (0)

}  // namespace

extern "C" {

int gp_pool_bytes(const gp_config* cfg, size_t* bytes) {
  if (!bytes) return GP_ERR_INVALID;
  if (check_config(cfg)) return GP_ERR_INVALID;
  gp_layout l;
  compute_layout(cfg, &l);
  *bytes = (size_t)l.total;
  return GP_OK;
}

int gp_create_pool(const gp_config* cfg, void* dev_buf, size_t bytes, void* stream, gp_pool** out) {
  if (!out || !cfg) return GP_ERR_INVALID;
  *out = nullptr;
  if (check_config(cfg)) return GP_ERR_INVALID;
  gp_layout l;
  compute_layout(cfg, &l);
  if (!dev_buf || bytes < l.total || ((uintptr_t)dev_buf % kAlign)) return GP_ERR_INVALID;
  gp_pool* p = new gp_pool();
  p->cfg = *cfg;
  p->lay = l;
  p->base = (uint8_t*)dev_buf;
  p->stream = (cudaStream_t)stream;
  p->slot_active.assign(cfg->max_requests, 0);
  p->slot_prefix.assign(cfg->max_requests, -1);
  p->prefix_refs.assign(cfg->max_prefixes, 0);
  p->prefix_held.assign(cfg->max_prefixes, 0);
  p->prefix_len.assign(cfg->max_prefixes, 0);
  fill_dev(p);
  use_plan(p, 0);
  auto bail = [&](int code) { delete p; return code; };
  cudaError_t e = cudaMemsetAsync(dev_buf, 0, l.total, p->stream);
  if (e != cudaSuccess) return bail(GP_ERR_CUDA);
  if (cfg->rope_theta != 0.0) {
    // fp64 values from the C library (pow, cos, sin); fp32 copies rounded
    // once, and the fp32 residuals fp32(x64 - x32) (the difference is exact);
    // one row per position: c32 | s32 | c32 residual | s32 residual | c64 | s64
    const int H = cfg->head_dim / 2;
    const size_t row = 16 * (size_t)cfg->head_dim;
    std::vector<uint8_t> rows((size_t)cfg->max_seq_len * row);
    std::vector<double> inv(H);
    for (int i = 0; i < H; ++i) inv[i] = std::pow(cfg->rope_theta, -(2.0 * i) / cfg->head_dim);
    for (int pos = 0; pos < cfg->max_seq_len; ++pos) {
      uint8_t* r = rows.data() + (size_t)pos * row;
      float* f32 = reinterpret_cast<float*>(r);
      double* f64 = reinterpret_cast<double*>(r + 16 * (size_t)H);
      for (int i = 0; i < H; ++i) {
        const double a = (double)pos * inv[i];
        const double c = std::cos(a), sn = std::sin(a);
        const float c32 = (float)c, s32 = (float)sn;
        f32[i] = c32;
        f32[H + i] = s32;
        f32[2 * H + i] = (float)(c - (double)c32);
        f32[3 * H + i] = (float)(sn - (double)s32);
        f64[i] = c;
        f64[H + i] = sn;
      }
    }
    e = cudaMemcpyAsync((void*)p->dev.rope_rows, rows.data(), rows.size(), cudaMemcpyHostToDevice, p->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->stream);
    if (e != cudaSuccess) return bail(GP_ERR_CUDA);
  }
  if (gp::select_setup() != cudaSuccess) return bail(GP_ERR_CUDA);
  e = gp::launch_init(p->dev, p->stream);
  if (e != cudaSuccess) return bail(GP_ERR_CUDA);
  p->launches += 1;
  p->use_mma = cfg->dtype == GP_DTYPE_BF16 && cfg->head_dim == 128;
  p->dev.summary_via_next = p->use_mma ? 1 : 0;
  p->dev.seg_cost = p->use_mma ? GP_SEG_COST : 0;
  if (p->use_mma) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr);
    if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn) return bail(GP_ERR_CUDA);
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    // The pool's K/V pages as a 5-D bf16 tensor, one 16-token block of a
    // (page, layer, head) per copy: dims (inner first) 64 columns, P tokens
    // (256-byte stride), 2 column halves (128 B), K|V (P * 256 B), and
    // page * L * Hk + layer * Hk + head (2 * P * 256 B).  The box
    // (64, 16, 2, 2, 1) lands in shared memory as [K|V][half][token][64],
    // 128-byte rows 128B-swizzled by token.
    const cuuint64_t P = (cuuint64_t)cfg->page_size, rb = (cuuint64_t)cfg->head_dim * 2;
    const cuuint64_t dims5[5] = {64, P, 2, 2,
                                 (cuuint64_t)cfg->num_pages * cfg->num_layers * cfg->num_kv_heads};
    const cuuint64_t strides5[4] = {rb, 128, P * rb, 2 * P * rb};
    const cuuint32_t box5[5] = {64, (cuuint32_t)gp::kBlockTok, 2, 2, 1};
    const cuuint32_t estr5[5] = {1, 1, 1, 1, 1};
    const CUresult r = encode(&p->kvblk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, (void*)p->dev.kv, dims5, strides5, box5,
               estr5, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return bail(GP_ERR_CUDA);
    if (gp::ceiling_setup() != cudaSuccess) return bail(GP_ERR_CUDA);
  }
  int dev = 0, sms = 0, blocks = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = p->use_mma ? gp::attention_mma_occupancy(p->dev, &blocks) : gp::attention_occupancy(p->dev, &blocks);
  if (e != cudaSuccess || sms <= 0 || blocks <= 0) return bail(GP_ERR_CUDA);
  const int wpc = p->use_mma ? gp::mma_warps_per_cta() : gp::kAttnWarps;
  int grid = sms * blocks;
  if (grid * wpc > gp::kMaxWorkersBound) grid = gp::kMaxWorkersBound / wpc;
  p->attn_grid = grid;
  p->dev.num_workers = grid * wpc;
  int sel_blocks = 0;
  if (gp::select_occupancy(&sel_blocks, false) != cudaSuccess || sel_blocks < 1) return bail(GP_ERR_CUDA);
  p->select_grid = sms * sel_blocks;
  if (gp::select_occupancy(&sel_blocks, true) != cudaSuccess || sel_blocks < 1) return bail(GP_ERR_CUDA);
  p->select_grid_big = sms * sel_blocks;
  p->commit_grid = sms * 4;
  e = cudaStreamSynchronize(p->stream);
  if (e != cudaSuccess) return bail(GP_ERR_CUDA);
  for (int b = 0; b < 2 && e == cudaSuccess; ++b)
    e = cudaEventCreateWithFlags(&p->side_ev[b], cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->main_ev, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    for (int b = 0; b < 2; ++b)
      if (p->side_ev[b]) cudaEventDestroy(p->side_ev[b]);
    return bail(GP_ERR_CUDA);
  }
  *out = p;
  return GP_OK;
}

int gp_destroy_pool(gp_pool* pool) {
  if (!pool) return GP_ERR_INVALID;
  for (int b = 0; b < 2; ++b)
    if (pool->side_ev[b]) cudaEventDestroy(pool->side_ev[b]);
  if (pool->main_ev) cudaEventDestroy(pool->main_ev);
  delete pool;
  return GP_OK;
}

int gp_set_stream(gp_pool* pool, void* stream) {
  if (!pool) return GP_ERR_INVALID;
  GP_JOIN(pool);
  pool->stream = (cudaStream_t)stream;
  return GP_OK;
}

int gp_get_layout(const gp_pool* pool, gp_layout* out) {
  if (!pool || !out) return GP_ERR_INVALID;
  *out = pool->lay;
  out->num_workers = pool->dev.num_workers;
  return GP_OK;
}

int gp_add_prefix(gp_pool* pool, const void* k_prefix, const void* v_prefix, int32_t len,
                  int32_t* prefix_id) {
  if (!pool || !prefix_id) return GP_ERR_INVALID;
  const gp_config& c = pool->cfg;
  if (pool->next_layer != 0) return fail(pool, GP_ERR_INVALID, "add_prefix inside a step");
  if (len <= 0 || len % c.page_size || len > c.max_prefix_len || !k_prefix || !v_prefix)
    return fail(pool, GP_ERR_INVALID, "prefix length must be a positive multiple of page_size <= max_prefix_len");
  if (len >= c.max_seq_len) return fail(pool, GP_ERR_INVALID, "prefix beyond max_seq_len");
  GP_JOIN(pool);
  int pid = -1;
  for (int k = 0; k < c.max_prefixes; ++k)
    if (pool->prefix_refs[k] == 0) { pid = k; break; }
  if (pid < 0) return fail(pool, GP_ERR_INVALID, "no free prefix slot");
  const int npages = len / c.page_size;
  int free_top = 0;
  int rc = read_free_top(pool, &free_top);
  if (rc) return rc;
  if (free_top < npages) return fail(pool, GP_ERR_NO_PAGES, "not enough free pages for the prefix");
  int32_t* row = pool->dev.prefix_pages + (size_t)pid * pool->lay.max_prefix_pages;
  GP_LAUNCH(pool, gp::launch_pop_pages(pool->dev, row, npages, pool->stream));
  GP_LAUNCH(pool, gp::launch_prefix_meta(pool->dev, pid, npages, len, pool->stream));
  GP_LAUNCH(pool, gp::launch_write_tokens(pool->dev, row, k_prefix, v_prefix, len, 0, pool->stream));
  rc = sync_status(pool);
  if (rc) return rc;
  pool->prefix_refs[pid] = 1;
  pool->prefix_held[pid] = 1;
  pool->prefix_len[pid] = len;
  *prefix_id = pid;
  return GP_OK;
}

int gp_release_prefix(gp_pool* pool, int32_t prefix_id) {
  if (!pool) return GP_ERR_INVALID;
  if (prefix_id < 0 || prefix_id >= pool->cfg.max_prefixes || !pool->prefix_held[prefix_id])
    return fail(pool, GP_ERR_INVALID, "prefix not held");
  GP_JOIN(pool);
  GP_LAUNCH(pool, gp::launch_release_prefix(pool->dev, prefix_id, pool->stream));
  pool->prefix_held[prefix_id] = 0;
  pool->prefix_refs[prefix_id] -= 1;
  return GP_OK;
}

int gp_add_request(gp_pool* pool, int32_t slot, const void* k_prompt, const void* v_prompt,
                   int32_t prompt_len, int32_t budget_pages, int32_t prefix_id) {
  if (!pool) return GP_ERR_INVALID;
  const gp_config& c = pool->cfg;
  if (pool->next_layer != 0) return fail(pool, GP_ERR_INVALID, "add_request inside a step");
  if (slot < 0 || slot >= c.max_requests || pool->slot_active[slot])
    return fail(pool, GP_ERR_INVALID, "slot out of range or in use");
  if (budget_pages < 1 || budget_pages > c.max_pages_per_req)
    return fail(pool, GP_ERR_INVALID, "budget_pages out of range");
  if (prompt_len < 0 || prompt_len > budget_pages * c.page_size)
    return fail(pool, GP_ERR_INVALID, "prompt does not fit the budget");
  if (prompt_len > 0 && (!k_prompt || !v_prompt)) return fail(pool, GP_ERR_INVALID, "null prompt");
  int plen = 0;
  if (prefix_id >= 0) {
    if (prefix_id >= c.max_prefixes || pool->prefix_refs[prefix_id] <= 0)
      return fail(pool, GP_ERR_INVALID, "unknown prefix");
    plen = pool->prefix_len[prefix_id];
  } else if (prefix_id != -1) {
    return fail(pool, GP_ERR_INVALID, "bad prefix id");
  }
  if ((long long)plen + prompt_len >= c.max_seq_len)
    return fail(pool, GP_ERR_INVALID, "position beyond max_seq_len");
  GP_JOIN(pool);
  int free_top = 0;
  int rc = read_free_top(pool, &free_top);
  if (rc) return rc;
  if (free_top < budget_pages) return fail(pool, GP_ERR_NO_PAGES, "not enough free pages for the budget");
  GP_LAUNCH(pool, gp::launch_admit(pool->dev, slot, budget_pages, prefix_id, prompt_len, pool->stream));
  const int npre = prefix_id >= 0 ? plen / c.page_size : 0;
  const int32_t* row = pool->dev.block + (size_t)slot * pool->lay.block_width + npre;
  if (prompt_len > 0)
    GP_LAUNCH(pool, gp::launch_write_tokens(pool->dev, row, k_prompt, v_prompt, prompt_len, plen,
                                            pool->stream));
  rc = sync_status(pool);
  if (rc) return rc;
  pool->slot_active[slot] = 1;
  pool->slot_prefix[slot] = prefix_id;
  if (prefix_id >= 0) {
    pool->prefix_refs[prefix_id] += 1;
    pool->prefixed_active += 1;
  }
  return GP_OK;
}

int gp_decode_step(gp_pool* pool, int32_t layer, int32_t n, const int32_t* slots_dev,
                   const void* q, const void* k_new, const void* v_new, void* out) {
  if (!pool) return GP_ERR_INVALID;
  const gp_config& c = pool->cfg;
  if (layer != pool->next_layer || layer >= c.num_layers)
    return fail(pool, GP_ERR_INVALID, "layers must be called 0..L-1, then gp_boundary");
  if (n < 0 || n > c.max_requests) return fail(pool, GP_ERR_INVALID, "n out of range");
  if (n > 0 && (!slots_dev || !q || !k_new || !v_new || !out))
    return fail(pool, GP_ERR_INVALID, "null tensor");
  if (((uintptr_t)q | (uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)out) % 16)
    return fail(pool, GP_ERR_INVALID, "q, k_new, v_new and out must be 16-byte aligned");
  if (layer == 0) {
    // steps alternate between the two plan buffers; this one was last used
    // two steps ago, whose boundary work may still run on a second stream
    const int b = pool->parity ^ 1;
    if (pool->side_pending[b]) {
      cudaError_t e = cudaStreamWaitEvent(pool->stream, pool->side_ev[b], 0);
      if (e != cudaSuccess) return cuda_fail(pool, e, "wait for second stream");
      pool->side_pending[b] = false;
    }
    use_plan(pool, b);
    GP_LAUNCH(pool, gp::launch_plan(pool->dev, n, slots_dev, 1, pool->stream));
    pool->step_n = n;
    pool->step_slots = slots_dev;
  } else if (n != pool->step_n || slots_dev != pool->step_slots) {
    return fail(pool, GP_ERR_INVALID, "every layer of a step must get the same slot list");
  }
  if (n > 0) {
    if (pool->use_mma) {
      const bool prefix = pool->dev.prefix_batch && pool->prefixed_active > 0;
      GP_LAUNCH(pool, gp::launch_attention_mma(pool->dev, &pool->kvblk, layer, n, q, k_new, v_new,
                                               out, pool->attn_grid, prefix, pool->stream));
      pool->launches += gp::attention_mma_launches(prefix) - 1;  // beyond the one counted above
    }
    else
      GP_LAUNCH(pool, gp::launch_attention(pool->dev, layer, q, k_new, v_new, out, pool->attn_grid,
                                           pool->stream));
  }
  pool->next_layer = layer + 1;
  return GP_OK;
}

// The select kernel's shape for a boundary call over n requests: at most
// n * L * Hk items (those at a boundary); when that many fit one wave of the
// 512-thread shape, per-item latency decides and it is taken.
bool select_big(const gp_pool* pool, int n) {
  return (int64_t)n * pool->cfg.num_layers * pool->cfg.num_kv_heads <= pool->select_grid_big;
}

int gp_boundary(gp_pool* pool, int32_t n, const int32_t* slots_dev) {
  if (!pool) return GP_ERR_INVALID;
  if (pool->next_layer != pool->cfg.num_layers)
    return fail(pool, GP_ERR_INVALID, "gp_boundary before all layers of the step");
  if (n != pool->step_n || slots_dev != pool->step_slots)
    return fail(pool, GP_ERR_INVALID, "gp_boundary must get the step's slot list");
  pool->next_layer = 0;
  if (n == 0) return GP_OK;
  GP_JOIN(pool);  // pages are popped below: after any earlier step's boundary work
  const bool big = select_big(pool, n);
  const int sgrid = big ? pool->select_grid_big : pool->select_grid;
  if (pool->cfg.mode != GP_MODE_FULL_KV)
    GP_LAUNCH(pool, gp::launch_select(pool->dev, sgrid, 0, big, pool->stream));
  GP_LAUNCH(pool, gp::launch_decide(pool->dev, gp::kPartAll, pool->stream));
  // SHRINK: the requests that release a page drop 2P tokens, not P; their
  // plans are redone once the decisions are known
  if (pool->cfg.mode == GP_MODE_SHRINK)
    GP_LAUNCH(pool, gp::launch_select(pool->dev, sgrid, 1, big, pool->stream));
  GP_LAUNCH(pool, gp::launch_commit(pool->dev, pool->commit_grid, gp::kPartAll, pool->stream));
  return GP_OK;
}

int gp_boundary_async(gp_pool* pool, int32_t n, const int32_t* slots_dev, void* side_stream) {
  if (!pool) return GP_ERR_INVALID;
  if (pool->next_layer != pool->cfg.num_layers)
    return fail(pool, GP_ERR_INVALID, "gp_boundary_async before all layers of the step");
  if (n != pool->step_n || slots_dev != pool->step_slots)
    return fail(pool, GP_ERR_INVALID, "gp_boundary_async must get the step's slot list");
  cudaStream_t side = (cudaStream_t)side_stream;
  if (!side || side == pool->stream)
    return fail(pool, GP_ERR_INVALID, "gp_boundary_async needs a second stream");
  pool->next_layer = 0;
  if (n == 0) return GP_OK;
  const int b = pool->parity;
  cudaError_t e;
  // the requests not at a boundary: decision-free bookkeeping and their
  // token appended, on the pool's stream; those at a boundary are marked busy
  GP_LAUNCH(pool, gp::launch_decide(pool->dev, gp::kPartPlain, pool->stream));
  GP_LAUNCH(pool, gp::launch_commit(pool->dev, pool->commit_grid, gp::kPartPlain, pool->stream));
  e = cudaEventRecord(pool->main_ev, pool->stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side, pool->main_ev, 0);
  // one step's boundary work after the previous one's (page pops in step order)
  if (e == cudaSuccess && pool->side_pending[b ^ 1]) e = cudaStreamWaitEvent(side, pool->side_ev[b ^ 1], 0);
  if (e != cudaSuccess) return cuda_fail(pool, e, "order the second stream");
  // the requests at a boundary, on the second stream
  const bool big = select_big(pool, n);
  const int sgrid = big ? pool->select_grid_big : pool->select_grid;
  if (pool->cfg.mode != GP_MODE_FULL_KV)
    GP_LAUNCH(pool, gp::launch_select(pool->dev, sgrid, 0, big, side));
  GP_LAUNCH(pool, gp::launch_decide(pool->dev, gp::kPartBoundary, side));
  if (pool->cfg.mode == GP_MODE_SHRINK)
    GP_LAUNCH(pool, gp::launch_select(pool->dev, sgrid, 1, big, side));
  GP_LAUNCH(pool, gp::launch_commit(pool->dev, pool->commit_grid, gp::kPartBoundary, side));
  GP_LAUNCH(pool, gp::launch_release_busy(pool->dev, side));
  e = cudaEventRecord(pool->side_ev[b], side);
  if (e != cudaSuccess) return cuda_fail(pool, e, "record second stream");
  pool->side_pending[b] = true;
  return GP_OK;
}

int gp_free(gp_pool* pool, int32_t slot) {
  if (!pool) return GP_ERR_INVALID;
  if (pool->next_layer != 0) return fail(pool, GP_ERR_INVALID, "free inside a step");
  if (slot < 0 || slot >= pool->cfg.max_requests || !pool->slot_active[slot])
    return fail(pool, GP_ERR_INVALID, "slot not active");
  GP_JOIN(pool);
  GP_LAUNCH(pool, gp::launch_free(pool->dev, slot, pool->stream));
  pool->slot_active[slot] = 0;
  const int pid = pool->slot_prefix[slot];
  if (pid >= 0) {
    pool->prefix_refs[pid] -= 1;
    pool->prefixed_active -= 1;
  }
  pool->slot_prefix[slot] = -1;
  return GP_OK;
}

int gp_kv_read_ceiling(gp_pool* pool, int32_t layer0, int32_t count, int32_t mode, int32_t n,
                       const int32_t* slots_dev, uint32_t* sink_dev) {
  if (!pool) return GP_ERR_INVALID;
  if (!pool->use_mma) return fail(pool, GP_ERR_INVALID, "read ceiling needs bf16 pages with head_dim 128");
  if (pool->next_layer != 0) return fail(pool, GP_ERR_INVALID, "read ceiling inside a step");
  if (layer0 < 0 || count < 1 || layer0 + count > pool->cfg.num_layers || mode < 0 || mode > 2 ||
      n < 0 || n > pool->cfg.max_requests || !sink_dev || (n > 0 && !slots_dev))
    return fail(pool, GP_ERR_INVALID, "bad read-ceiling arguments");
  GP_JOIN(pool);
  GP_LAUNCH(pool, gp::launch_plan(pool->dev, n, slots_dev, 0, pool->stream));
  const int wpc = gp::ceiling_warps_per_cta();
  const int grid = (pool->dev.num_workers + wpc - 1) / wpc;
  for (int l = layer0; l < layer0 + count; ++l)
    GP_LAUNCH(pool, gp::launch_kv_read(pool->dev, &pool->kvblk, l, mode, sink_dev, grid, pool->stream));
  return GP_OK;
}

}  // extern "C"

// ---- read ceiling without caller scratch -------------------------------
//
// Scratch of gp_kv_read_ceiling_static: the step plan (twelve arrays of
// kStaticMaxRequests + 1 ints, the Delta accumulators), the per-worker
// start cursors and the per-worker first blocks.  It is a file-scope device array, so every GPU that loads
// the library holds these bytes until the process exits.
namespace {
constexpr int kStaticMaxRequests = 1024;
constexpr size_t kStaticPlanArrayBytes = ((size_t)(kStaticMaxRequests + 1) * 4 + 255) / 256 * 256;
constexpr size_t kStaticDeltaBytes = (size_t)kStaticMaxRequests * 8;
constexpr size_t kStaticWblkBytes = ((size_t)(gp::kMaxWorkersBound + 1) * 4 + 255) / 256 * 256;
constexpr size_t kStaticBytes = 12 * kStaticPlanArrayBytes + kStaticDeltaBytes +
                                (size_t)gp::kMaxWorkersBound * 16 + kStaticWblkBytes;
}  // namespace

static __device__ __align__(256) uint8_t g_static_scratch[kStaticBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
uint8_t* g_static_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (set up once per
// device; the host-side name of the array is not a device address).  The
// address stays valid while the device's primary context lives, which the
// header asks callers to keep for the life of the process.
cudaError_t static_scratch(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_addr[dev] = static_cast<uint8_t*>(ptr);
  }
  *out = g_static_addr[dev];
  return cudaSuccess;
}
}  // namespace

extern "C" {

int gp_kv_read_ceiling_static(gp_pool* pool, int32_t layer0, int32_t count, int32_t mode,
                              int32_t n, const int32_t* slots_dev, uint32_t* sink_dev) {
  if (!pool) return GP_ERR_INVALID;
  if (!pool->use_mma) return fail(pool, GP_ERR_INVALID, "read ceiling needs bf16 pages with head_dim 128");
  if (layer0 < 0 || count < 1 || layer0 + count > pool->cfg.num_layers || mode < 0 || mode > 2 ||
      n < 0 || n > pool->cfg.max_requests || !sink_dev || (n > 0 && !slots_dev))
    return fail(pool, GP_ERR_INVALID, "bad read-ceiling arguments");
  if (n > kStaticMaxRequests)
    return fail(pool, GP_ERR_INVALID, "gp_kv_read_ceiling_static: n exceeds the static scratch limit of 1024 requests");
  if (pool->dev.num_workers > gp::kMaxWorkersBound)
    return fail(pool, GP_ERR_INVALID, "gp_kv_read_ceiling_static: too many attention workers");
  uint8_t* base = nullptr;
  cudaError_t e = static_scratch(&base);
  if (e != cudaSuccess) return cuda_fail(pool, e, "cudaGetSymbolAddress(g_static_scratch)");
  // the pool's view with its per-call scratch moved into the static array
  gp::PoolDev d = pool->dev;
  int32_t** arrays[12] = {&d.plan_slot, &d.plan_R,    &d.plan_nb,  &d.plan_cum,
                          &d.plan_flags, &d.plan_commit, &d.plan_cpos, &d.plan_dec,
                          &d.plan_bnd,  &d.plan_misc, &d.plan_pos, &d.plan_base};
  for (int k = 0; k < 12; ++k) *arrays[k] = (int32_t*)(base + k * kStaticPlanArrayBytes);
  d.plan_delta = (long long*)(base + 12 * kStaticPlanArrayBytes);
  d.wstart = (int4*)(base + 12 * kStaticPlanArrayBytes + kStaticDeltaBytes);
  d.wblk = (int32_t*)(base + 12 * kStaticPlanArrayBytes + kStaticDeltaBytes +
                      (size_t)gp::kMaxWorkersBound * 16);
  d.seginfo = nullptr;  // not written by the plan in measurement calls
  GP_LAUNCH(pool, gp::launch_plan(d, n, slots_dev, 0, pool->stream));
  const int wpc = gp::ceiling_warps_per_cta();
  const int grid = (d.num_workers + wpc - 1) / wpc;
  for (int l = layer0; l < layer0 + count; ++l)
    GP_LAUNCH(pool, gp::launch_kv_read(d, &pool->kvblk, l, mode, sink_dev, grid, pool->stream));
  return GP_OK;
}

int gp_sync(gp_pool* pool) {
  if (!pool) return GP_ERR_INVALID;
  GP_JOIN(pool);
  return sync_status(pool);
}

int gp_clear_status(gp_pool* pool, uint32_t* status_out, int32_t* info_out) {
  if (!pool) return GP_ERR_INVALID;
  GP_JOIN(pool);
  cudaError_t e = cudaStreamSynchronize(pool->stream);
  uint32_t st[2] = {0u, 0u};  // status, status_info (adjacent in gp_ctrl)
  if (e == cudaSuccess) e = cudaMemcpy(st, &pool->dev.ctrl->status, 8, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemsetAsync(&pool->dev.ctrl->status, 0, 8, pool->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(pool->stream);
  if (e != cudaSuccess) return cuda_fail(pool, e, "gp_clear_status");
  if (status_out) *status_out = st[0];
  if (info_out) *info_out = (int32_t)st[1];
  pool->err.clear();
  return GP_OK;
}

int gp_get_stats(gp_pool* pool, gp_ctrl* out) {
  if (!pool || !out) return GP_ERR_INVALID;
  GP_JOIN(pool);
  cudaError_t e = cudaStreamSynchronize(pool->stream);
  if (e == cudaSuccess) e = cudaMemcpy(out, pool->dev.ctrl, sizeof(gp_ctrl), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(pool, e, "gp_get_stats");
  return GP_OK;
}

int gp_get_request(gp_pool* pool, int32_t slot, gp_req_meta* meta, int32_t* block_table, int32_t cap) {
  if (!pool || !meta || slot < 0 || slot >= pool->cfg.max_requests || cap < 0)
    return GP_ERR_INVALID;
  GP_JOIN(pool);
  cudaError_t e = cudaStreamSynchronize(pool->stream);
  if (e == cudaSuccess)
    e = cudaMemcpy(meta, pool->dev.req + slot, sizeof(gp_req_meta), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && block_table && cap > 0) {
    const int w = cap < pool->lay.block_width ? cap : pool->lay.block_width;
    e = cudaMemcpy(block_table, pool->dev.block + (size_t)slot * pool->lay.block_width, (size_t)w * 4,
                   cudaMemcpyDeviceToHost);
  }
  if (e != cudaSuccess) return cuda_fail(pool, e, "gp_get_request");
  return GP_OK;
}

int gp_get_state(gp_pool* pool, gp_state_view* out) {
  if (!pool || !out) return GP_ERR_INVALID;
  const gp_config& c = pool->cfg;
  const gp::PoolDev& d = pool->dev;
  const size_t R = (size_t)c.max_requests;
  GP_JOIN(pool);
  cudaError_t e = cudaStreamSynchronize(pool->stream);
  auto copy = [&](void* dst, const void* src, size_t bytes) {
    if (e == cudaSuccess && dst) e = cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost);
  };
  copy(out->req, d.req, R * sizeof(gp_req_meta));
  copy(out->block, d.block, R * (size_t)pool->lay.block_width * 4);
  copy(out->ctrl, d.ctrl, sizeof(gp_ctrl));
  copy(out->wset, d.wset, R * c.num_layers * c.num_kv_heads * 2 * 4);
  copy(out->tok_pos, d.tok_pos, (size_t)c.num_pages * c.num_layers * c.num_kv_heads * c.page_size * 4);
  copy(out->free_stack, d.free_stack, (size_t)c.num_pages * 4);
  if (e != cudaSuccess) return cuda_fail(pool, e, "gp_get_state");
  return GP_OK;
}

const char* gp_last_error(const gp_pool* pool) { return pool ? pool->err.c_str() : "null pool"; }

int64_t gp_launch_count(const gp_pool* pool) { return pool ? pool->launches : 0; }

}  // extern "C"
