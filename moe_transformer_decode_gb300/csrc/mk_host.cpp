// Host side of libmk: context and workspace, the task scheduler, tensor maps and launches.
//
// Scheduling follows the task-list design of the Cohere megakernel news pages
// (aimodeling.com "cohere-megakernel-north-mini-code-h100", section "One persistent kernel
// for the whole decode step"; aibriefing.imbch.dev article 8171681, section "Scheduling and
// Performance Benchmarks": a mostly static per-SM schedule built on the host). Every task
// of a layer is listed in dependency order (router, QKV, attention, expert gate/up, O-proj,
// expert down) and given to the SM with the least bytes assigned so far, so parallel-layer
// work backfills SMs that would otherwise wait; each SM's list is in that global order,
// which is what keeps the counter waits deadlock-free.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <queue>
#include <tuple>
#include <string>
#include <vector>

#include "mk_internal.h"

namespace mk {
int kernel_smem_bytes();
cudaError_t launch_decode(const Params& p, const TensorMaps& tm, cudaStream_t st);
cudaError_t max_blocks_per_sm(int B, int* n);
cudaError_t configure_kernels();
}  // namespace mk

using namespace mk;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct mk_ctx {
  mk_model_cfg cfg;
  mk_weight_ptrs w;
  int device, n_sm;
  int mode;
  long long wait_ns = 2000000000LL;  // device-side wait limit
  std::string err;
  // workspace (device)
  float *xs, *q, *knew, *vnew, *attn_o, *attn_out, *rlogits, *moe_out, *moe_part, *apart, *lm_best_v, *css;
  uint16_t* attn_hl;
  uint8_t* hsw;
  int32_t* lm_best_i;
  int32_t* topk_ids;
  float* topk_w;
  Route* route;
  float2* rope;
  uint32_t* counters;
  int32_t* status;
  int32_t* status_host;  // mapped pinned copy of the status code (written by the device on error)
  int32_t* status_host_dev;
  int max_pos;
  // schedule
  bool scheduled;
  int B;
  const int32_t* block_table;
  Task* d_tasks;
  int32_t* d_sm_begin;  // megakernel: [n_sm+1]; then per-op launches, each [n_sm+1]
  int32_t* d_cnt;
  int32_t *d_chunk_pages, *d_n_chunks;
  int max_chunks, n_lm_sm, n_tasks, n_counters;
  int n_op_launches;
  uint32_t epoch;
  // tensor maps cache
  void *tm_k_ptr, *tm_v_ptr;
  int tm_pages;
  TensorMaps tm;
  EncodeTiledFn encode;
  // trace
  mk_trace_entry* trace;
  unsigned long long* trace_count;
  long long trace_cap;
};

// The expert weights as 3D bf16 views {64, rows, K / 64} (strides: a row, 128 bytes) with 128B
// swizzle: a gate/up box lands kGuRows rows x 64 columns, a down box kDnRows rows x 128 columns
// as two [rows][128 bytes] chunks, the layout of the tcgen05 B operand. The O-proj weights as a
// 3D view {256, od / 256, rows} (strides: 512 bytes, a row) without swizzle: a box of RS rows x
// KS / 256 column blocks lands a row-major GEMV stage in one copy (a bulk copy per row would
// take RS copies, and a copy's issue time grows with their number).
mk_status mk::encode_weight_maps(void* encode_fn, const mk_model_cfg& m, const mk_weight_ptrs* w, TensorMaps& tm) {
  EncodeTiledFn enc = (EncodeTiledFn)encode_fn;
  const uint64_t gu_rows = (uint64_t)m.n_layers * m.n_experts * 2 * m.expert_inter;
  const uint64_t dn_rows = (uint64_t)m.n_layers * m.n_experts * m.hidden;
  if (gu_rows >= (1ull << 31) || dn_rows >= (1ull << 31)) return MK_ERR_UNSUPPORTED;
  cuuint32_t estr[3] = {1, 1, 1};
  {
    cuuint64_t dims[3] = {64, (cuuint64_t)gu_rows, (cuuint64_t)m.hidden / 64};
    cuuint64_t strides[2] = {(cuuint64_t)m.hidden * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kGuRows, 1};
    if (enc(&tm.gu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w->w_gate_up), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MK_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {64, (cuuint64_t)dn_rows, (cuuint64_t)m.expert_inter / 64};
    cuuint64_t strides[2] = {(cuuint64_t)m.expert_inter * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kDnRows, (cuuint32_t)(kStageK / 64)};
    if (enc(&tm.dn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w->w_down), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MK_ERR_CUDA;
  }
  {
    // the GEMV geometry of K = od (KS = min(od, 2048) columns, RS = 8 * 8 / (KS / 256) rows; od is a
    // multiple of 256): the box is RS x KS elements, 32 KB
    const uint64_t od = (uint64_t)m.n_q_heads * m.head_dim;
    const uint64_t o_rows = (uint64_t)m.n_layers * m.hidden;
    const uint32_t ks = od < 2048 ? (uint32_t)od : 2048u, kw = ks / 256, rs = 8u * (8u / kw);
    if (o_rows >= (1ull << 31)) return MK_ERR_UNSUPPORTED;
    cuuint64_t dims[3] = {256, (cuuint64_t)(od / 256), (cuuint64_t)o_rows};
    cuuint64_t strides[2] = {512, (cuuint64_t)od * 2};
    cuuint32_t box[3] = {256, kw, rs};
    if (enc(&tm.wo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w->w_o), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MK_ERR_CUDA;
  }
  return MK_OK;
}

static mk_status fail(mk_ctx* c, mk_status s, const std::string& msg) {
  if (c) c->err = msg;
  return s;
}
static mk_status cuda_fail(mk_ctx* c, cudaError_t e, const char* what) {
  return fail(c, MK_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define CK(call)                                          \
  do {                                                    \
    cudaError_t e_ = (call);                              \
    if (e_ != cudaSuccess) return cuda_fail(c, e_, #call); \
  } while (0)

template <typename T>
static cudaError_t dalloc(T** p, size_t n) {
  *p = nullptr;
  if (n == 0) n = 1;
  return cudaMalloc((void**)p, n * sizeof(T));
}

static void free_schedule(mk_ctx* c) {
  cudaFree(c->d_tasks);
  cudaFree(c->d_sm_begin);
  cudaFree(c->d_cnt);
  cudaFree(c->d_chunk_pages);
  cudaFree(c->d_n_chunks);
  cudaFree(c->apart);
  cudaFree(c->counters);
  c->d_tasks = nullptr;
  c->d_sm_begin = c->d_cnt = c->d_chunk_pages = c->d_n_chunks = nullptr;
  c->apart = nullptr;
  c->counters = nullptr;
  c->scheduled = false;
}

extern "C" void mk_destroy(mk_ctx* c) {
  if (!c) return;
  free_schedule(c);
  cudaFree(c->xs); cudaFree(c->q); cudaFree(c->knew); cudaFree(c->vnew); cudaFree(c->attn_o); cudaFree(c->attn_out);
  cudaFree(c->rlogits); cudaFree(c->hsw); cudaFree(c->attn_hl); cudaFree(c->moe_out); cudaFree(c->moe_part); cudaFree(c->css); cudaFree(c->lm_best_v); cudaFree(c->lm_best_i);
  cudaFree(c->route); cudaFree(c->rope); cudaFree(c->status); cudaFree(c->topk_ids); cudaFree(c->topk_w);
  if (c->status_host) cudaFreeHost(c->status_host);
  delete c;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// The one check of a model config and its weight pointers, shared by every entry point that
// takes them (mk_create, mk_decode_step_noalloc), so their limits cannot drift apart. It runs
// before any size or offset is computed from the config. *why (may be NULL) gets a static
// description of the first failed check.
mk_status mk::validate_model(const mk_model_cfg* cfg, const mk_weight_ptrs* w, const char** why) {
  auto no = [&](mk_status s, const char* text) {
    if (why) *why = text;
    return s;
  };
  if (!cfg || !w) return no(MK_ERR_INVALID_ARG, "null config or weight pointers");
  const mk_model_cfg& m = *cfg;
  if (m.n_layers <= 0 || m.hidden <= 0 || m.n_q_heads <= 0 || m.n_kv_heads <= 0 || m.head_dim <= 0 ||
      m.n_experts <= 0 || m.top_k <= 0 || m.top_k > m.n_experts || m.expert_inter <= 0 || m.vocab <= 0 ||
      m.max_batch <= 0 || m.max_pages_per_seq <= 0 || m.n_q_heads % m.n_kv_heads != 0 || m.n_layers > 65535)
    return no(MK_ERR_INVALID_ARG, "inconsistent model config (a size <= 0, top_k > n_experts, or n_kv_heads not "
                                  "dividing n_q_heads)");
  if (!(m.rms_eps >= 0.f) || !(m.rope_theta > 0.f) || !std::isfinite(m.rms_eps) || !std::isfinite(m.rope_theta))
    return no(MK_ERR_INVALID_ARG, "rms_eps must be finite and >= 0, rope_theta finite and > 0");
  if (!w->embed || !w->norm_gain || !w->w_qkv || !w->w_o || !w->w_router || !w->w_gate_up || !w->w_down ||
      !w->final_gain || !w->lm_head)
    return no(MK_ERR_INVALID_ARG, "null weight pointer");
  const void* ptrs[] = {w->embed, w->norm_gain, w->w_qkv, w->w_o, w->w_router, w->w_gate_up, w->w_down,
                        w->final_gain, w->lm_head, w->router_bias};
  for (const void* p : ptrs)
    if (!aligned16(p)) return no(MK_ERR_INVALID_ARG, "weight pointer not 16-byte aligned");
  const int od = m.n_q_heads * m.head_dim;
  const bool shape_ok = (m.hidden == 256 || m.hidden == 512 || m.hidden == 1024 || m.hidden == 2048) &&
                        (m.head_dim == 64 || m.head_dim == 128) && m.n_q_heads / m.n_kv_heads <= 8 &&
                        od % 256 == 0 && (od <= 2048 || od % 2048 == 0) && m.expert_inter % 256 == 0 &&
                        m.expert_inter <= 2048 && m.top_k <= kMaxK && m.max_batch <= kMaxB &&
                        m.page_size == kPage && m.n_experts <= kMaxExperts && m.n_experts % 8 == 0 &&
                        m.vocab % 64 == 0 &&
                        // an expert's activations for the whole batch fit one ring stage
                        2 * m.max_batch * 2 * m.expert_inter <= kStagePayload;
  if (!shape_ok) return no(MK_ERR_UNSUPPORTED, "model shape not supported by this build");
  return MK_OK;
}

extern "C" mk_status mk_create(const mk_model_cfg* cfg, const mk_weight_ptrs* w, mk_ctx** out) {
  if (!cfg || !w || !out) return MK_ERR_INVALID_ARG;
  *out = nullptr;
  const mk_status vs = validate_model(cfg, w, nullptr);
  if (vs != MK_OK) return vs;
  const mk_model_cfg& m = *cfg;
  const int od = m.n_q_heads * m.head_dim;

  mk_ctx* c = new mk_ctx();  // value-initialized: every pointer starts null
  c->cfg = m;
  c->w = *w;
  c->mode = MK_MODE_MEGAKERNEL;
  c->scheduled = false;
  c->d_tasks = nullptr;
  c->d_sm_begin = c->d_cnt = c->d_chunk_pages = c->d_n_chunks = nullptr;
  c->trace = nullptr;
  c->trace_count = nullptr;
  c->trace_cap = 0;
  c->tm_k_ptr = c->tm_v_ptr = nullptr;
  c->tm_pages = -1;
  c->epoch = 0;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e != cudaSuccess) { mk_destroy(c); return MK_ERR_CUDA; }
  cudaDeviceGetAttribute(&c->n_sm, cudaDevAttrMultiProcessorCount, c->device);
  int coop = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device);
  int smem_optin = 0;
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
  if (!coop || smem_optin < kernel_smem_bytes()) {
    c->err = "device lacks cooperative launch or enough shared memory";
    mk_destroy(c);
    return MK_ERR_UNSUPPORTED;
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess || !fn) {
    mk_destroy(c);
    return MK_ERR_CUDA;
  }
  c->encode = (EncodeTiledFn)fn;

  const size_t L = m.n_layers, Bm = kMaxB, H = m.hidden, d = m.head_dim;
  c->max_pos = m.max_pages_per_seq * kPage;
  bool okm = dalloc(&c->xs, (L + 1) * Bm * H) == cudaSuccess && dalloc(&c->q, L * Bm * m.n_q_heads * d) == cudaSuccess &&
             dalloc(&c->knew, L * Bm * m.n_kv_heads * d) == cudaSuccess &&
             dalloc(&c->vnew, L * Bm * m.n_kv_heads * d) == cudaSuccess && dalloc(&c->attn_o, L * Bm * od) == cudaSuccess && dalloc(&c->attn_hl, L * 2 * Bm * od) == cudaSuccess &&
             dalloc(&c->attn_out, L * Bm * H) == cudaSuccess && dalloc(&c->moe_out, L * Bm * H) == cudaSuccess &&
             dalloc(&c->rlogits, L * Bm * m.n_experts) == cudaSuccess &&
             dalloc(&c->hsw, L * kMaxActive * hsw_slot_bytes(m.expert_inter)) == cudaSuccess &&
             dalloc(&c->moe_part, L * kMoeParts * Bm * H) == cudaSuccess &&
             dalloc(&c->css, (L + 1) * kMaxCombineSlices * Bm) == cudaSuccess &&
             dalloc(&c->route, L) == cudaSuccess && dalloc(&c->lm_best_v, (size_t)c->n_sm * kMaxB) == cudaSuccess &&
             dalloc(&c->lm_best_i, (size_t)c->n_sm * kMaxB) == cudaSuccess &&
             dalloc(&c->rope, (size_t)c->max_pos * (d / 2)) == cudaSuccess && dalloc(&c->status, ST_WORDS) == cudaSuccess &&
             dalloc(&c->topk_ids, L * Bm * m.top_k) == cudaSuccess && dalloc(&c->topk_w, L * Bm * m.top_k) == cudaSuccess;
  if (!okm) {
    cudaGetLastError();
    mk_destroy(c);
    return MK_ERR_OOM;
  }
  if (cudaHostAlloc((void**)&c->status_host, 4 * sizeof(int32_t), cudaHostAllocMapped) != cudaSuccess) {
    c->status_host = nullptr;
    mk_destroy(c);
    return MK_ERR_CUDA;
  }
  memset(c->status_host, 0, 4 * sizeof(int32_t));
  if (cudaHostGetDevicePointer((void**)&c->status_host_dev, c->status_host, 0) != cudaSuccess) {
    mk_destroy(c);
    return MK_ERR_CUDA;
  }
  cudaMemset(c->status, 0, ST_WORDS * sizeof(int32_t));
  cudaMemset(c->xs, 0, (L + 1) * Bm * H * sizeof(float));
  // RoPE table: angle pos * theta^(-2i/d), computed in fp64, stored as fp32 (cos, sin)
  {
    std::vector<float2> tab((size_t)c->max_pos * (d / 2));
    for (int pos = 0; pos < c->max_pos; ++pos)
      for (size_t i = 0; i < d / 2; ++i) {
        const double ang = (double)pos * std::pow((double)m.rope_theta, -2.0 * (double)i / (double)d);
        tab[(size_t)pos * (d / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    e = cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) { mk_destroy(c); return MK_ERR_CUDA; }
  }
  // the expert weights as tcgen05 B operand tiles (3D views {64, rows, K / 64}, 128B swizzle) and
  // the O-proj weights as whole GEMV stages
  {
    const mk_status ts = encode_weight_maps((void*)c->encode, m, w, c->tm);
    if (ts != MK_OK) {
      mk_destroy(c);
      return ts;
    }
  }
  e = configure_kernels();
  if (e != cudaSuccess) {
    c->err = std::string("kernel configuration: ") + cudaGetErrorString(e);
    mk_destroy(c);
    return MK_ERR_CUDA;
  }
  for (int nb : {1, 2, 4, 8}) {
    int blocks = 0;
    e = max_blocks_per_sm(nb, &blocks);
    if (e != cudaSuccess || blocks < 1) {
      mk_destroy(c);
      return MK_ERR_UNSUPPORTED;
    }
  }
  *out = c;
  return MK_OK;
}

// ------------------------------------------------------------------ scheduler

namespace {

struct Geo {
  int KS, KW, RG, RS, NCS;
};
Geo geo_of(int K) {
  Geo g;
  g.KS = K < 2048 ? K : 2048;
  g.KW = g.KS / 256;
  g.RG = kConsumerWarps / g.KW;
  g.RS = 8 * g.RG;
  g.NCS = K / g.KS;
  return g;
}

// Least-loaded assignment within a partition of the SMs. Loads are counted per phase
// (new_layer() restarts them), so each phase's work is spread evenly over the partition; ties
// go to the SM with the least bytes over the whole step (`total`), so no SM takes the extra
// task in every phase. `layer` counts each SM's bytes since begin_layer(): put_layer breaks the
// phase's ties by it instead, so a phase's extra tasks land on the SMs with the least work in the
// layer so far.
struct Assigner {
  int n_sm;
  std::vector<int> part;  // partition of each SM
  std::vector<long long> load, total, layer;
  std::vector<std::vector<Task>> lists;
  typedef std::tuple<long long, long long, int> Key;
  std::vector<std::priority_queue<Key, std::vector<Key>, std::greater<>>> heaps;
  Assigner(int n, std::vector<int> part_, int n_parts)
      : n_sm(n), part(std::move(part_)), load(n, 0), total(n, 0), layer(n, 0), lists(n), heaps(n_parts) {
    new_layer();
  }
  void begin_layer() { std::fill(layer.begin(), layer.end(), 0LL); }
  void new_layer() {
    for (auto& h : heaps) h = std::priority_queue<Key, std::vector<Key>, std::greater<>>();
    for (int s = 0; s < n_sm; ++s) {
      load[s] = 0;
      heaps[part[s]].push(Key(0, total[s], s));
    }
  }
  // onto SM s (kept in s's heap position)
  void put_on(const Task& t, long long bytes, int s) {
    lists[s].push_back(t);
    load[s] += bytes;
    total[s] += bytes;
    layer[s] += bytes;
    auto& heap = heaps[part[s]];
    std::vector<Key> keep;
    while (!heap.empty()) {
      Key k = heap.top();
      heap.pop();
      if (std::get<2>(k) == s) k = Key(load[s], total[s], s);
      keep.push_back(k);
    }
    for (auto& k : keep) heap.push(k);
  }
  // onto the least-loaded SM of any partition, except those marked in `skip`
  int put_any(const Task& t, long long bytes, const std::vector<char>& skip) {
    int best = -1;
    for (int s = 0; s < n_sm; ++s)
      if (!skip[s] && (best < 0 || std::make_tuple(load[s], total[s], s) < std::make_tuple(load[best], total[best], best)))
        best = s;
    if (best < 0) best = 0;
    put_on(t, bytes, best);
    return best;
  }
  int put(const Task& t, long long bytes, int pt) {
    auto& heap = heaps[pt];
    const int s = std::get<2>(heap.top());
    heap.pop();
    lists[s].push_back(t);
    load[s] += bytes;
    total[s] += bytes;
    layer[s] += bytes;
    heap.push(Key(load[s], total[s], s));
    return s;
  }
  // onto the least-loaded SM of partition pt in this phase, ties to the least bytes in the layer
  int put_layer(const Task& t, long long bytes, int pt) {
    int best = -1;
    for (int s = 0; s < n_sm; ++s)
      if (part[s] == pt && (best < 0 || std::make_tuple(load[s], layer[s], s) < std::make_tuple(load[best], layer[best], best)))
        best = s;
    put_on(t, bytes, best);
    return best;
  }
};

Task mkt(int op, int layer, int a, int b, int c, int flags = 0) {
  Task t;
  t.op = (uint8_t)op;
  t.flags = (uint8_t)flags;
  t.layer = (uint16_t)layer;
  t.a = a;
  t.b = b;
  t.c = c;
  return t;
}

}  // namespace

mk_status mk::plan_schedule(const mk_model_cfg& m, int n_sm, int B, const int32_t* seq_lens, Plan& P) {
  if (n_sm < 1 || B < 1 || B > m.max_batch || !seq_lens) return MK_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] < 0 || seq_lens[b] >= m.max_pages_per_seq * kPage) return MK_ERR_INVALID_ARG;
  const int L = m.n_layers, H = m.hidden, d = m.head_dim, nkv = m.n_kv_heads, G = m.n_q_heads / nkv;
  const int E = m.n_experts, I = m.expert_inter, V = m.vocab, od = m.n_q_heads * d;
  const Geo gh = geo_of(H), go = geo_of(od);
  const int pps = kStagePayload / (4096 * (d / 64));
  CounterMap cmap{L, nkv, B};
  std::vector<int32_t>& cnt = P.cnt;
  cnt.assign(cmap.count(), 0);

  long long group_pages = 0;
  std::vector<int> npg(B);
  for (int b = 0; b < B; ++b) {
    npg[b] = (seq_lens[b] + kPage - 1) / kPage;
    group_pages += (long long)npg[b] * nkv;
  }
  const int maxa = std::min(B * m.top_k, E);
  // expected live fraction of the planned expert slots (1 at batch 1)
  const double live = maxa == m.top_k ? 1.0 : std::min(1.0, (double)E * (1.0 - std::pow(1.0 - (double)m.top_k / E, B)) / maxa);

  // At batch 1, when the two branches of a layer (attention: QKV, attention, O-proj; experts:
  // router, gate/up, down) stream comparable bytes, they run on disjoint SM partitions sized by
  // those bytes, so neither branch's tasks queue behind the other's on an SM. At larger batches,
  // or when one branch dominates (the KV of a long context), every SM takes both: measured faster.
  const double attn_bytes = (double)(m.n_q_heads + 2 * nkv) * d * H * 2 + (double)H * od * 2 +
                            (double)group_pages * 2 * kPage * d * 2;
  const double moe_bytes = (double)E * H * 2 + live * maxa * 3.0 * I * H * 2;
  int n_attn = n_sm;  // every SM takes both branches
  if (n_sm >= 8 && B == 1 && attn_bytes <= 1.5 * moe_bytes) {
    // The expert branch has one more dependent hand-off per layer (router -> routing -> gate/up ->
    // down) than the attention branch, and QKV runs on every SM, so the attention partition is
    // 0.82 x the attention branch's byte share: 52 of 152 SMs at 8K context, the smallest count
    // at which the attention chunks take 10 stages and the O-proj tasks 5 row blocks (measured
    // best among 0.65-0.85 on the 30B-shaped model; 0.75 and 0.85 are 2 % slower).
    n_attn = (int)std::lround(0.82 * n_sm * attn_bytes / (attn_bytes + moe_bytes));
    n_attn = std::min(std::max(n_attn, 1), n_sm - 1);
  }
  std::vector<int> part(n_sm, 0);
  for (int s = n_attn; s < n_sm; ++s) part[s] = 1;
  const int PA = 0, PM = n_attn < n_sm ? 1 : 0;
  const int n_moe = n_attn < n_sm ? n_sm - n_attn : n_sm;
  P.n_attn_sm = n_attn;

  // attention chunks: whole stages each, the smallest size for which the (sequence, group,
  // chunk) tasks number at most one per attention SM (a second task on one SM would double the
  // attention phase); unless that size is impractically large (more than twice the even share)
  int cp = (int)((group_pages + n_attn - 1) / n_attn);
  cp = std::max(cp, pps);
  cp = (cp + pps - 1) / pps * pps;
  auto n_attn_tasks = [&](int c) {
    long long n = 0;
    for (int b = 0; b < B; ++b) n += (long long)nkv * std::max(1, (npg[b] + c - 1) / c);
    return n;
  };
  for (int c = cp; c <= 2 * cp; c += pps)
    if (n_attn_tasks(c) <= n_attn) {
      cp = c;
      break;
    }
  P.chunk_pages.assign(B, cp);
  P.n_chunks.assign(B, 1);
  P.max_chunks = 1;
  for (int b = 0; b < B; ++b) {
    P.n_chunks[b] = std::max(1, (npg[b] + cp - 1) / cp);
    P.max_chunks = std::max(P.max_chunks, P.n_chunks[b]);
  }

  // expert GEMVs (tcgen05): gate/up units of kGuRows gate rows + the matching up rows over H;
  // down units of kDnRows output rows for one of `parts` partials (experts of rank j mod parts)
  const int tiles = I / kGuRows;
  const int parts = moe_parts_for(B, m.top_k, E);
  // Per layer, gate/up tasks are sized to about two per expert SM and QKV tasks to about two
  // per SM (whole stages each, rounded up so that no SM gets a third). When the SMs are
  // partitioned, QKV runs on every SM but the router's, about one task each: it needs only the
  // layer's input, and the expert SMs would otherwise wait idle for the routing. Unpartitioned,
  // batch 1 (a long context) takes one QKV task per SM too (256K: 6.16 -> 6.13 ms per step);
  // larger batches take about two smaller ones (one per SM measured 0.5-1.2 % slower at batch 8).
  const int upg_ = (G + 2) * (d / 8);
  const int qkv_tasks = n_attn < n_sm ? n_sm - (E + gh.RS - 1) / gh.RS : (B == 1 ? n_sm : 2 * n_attn);
  int qkv_per_task = std::max(1, (nkv * upg_ + qkv_tasks - 1) / qkv_tasks);
  qkv_per_task = std::max(gh.RG, (qkv_per_task + gh.RG - 1) / gh.RG * gh.RG);
  // gate/up tasks: at most one per expert SM; each takes an equal share of the units of the
  // experts the step actually routes to (known on the device only), see the kernel's op_gu
  const int n_gu_tasks = std::max(1, std::min(n_moe, maxa * tiles));
  const long long row_h = 2LL * H;

  Assigner as(n_sm, part, PM + 1);
  std::vector<std::vector<std::vector<Task>>> per_op;  // [launch][sm] tasks for the per-op mode
  // Each phase (the tasks of one op kind in a layer) becomes ready at once, after a dependency
  // every SM shares, so it is balanced on its own: loads restart at every phase (ties still go
  // to the SM with the fewest bytes over the step).
  // SMs holding a router task of the current layer (QKV avoids them: one of them computes the
  // routing right after its router task)
  std::vector<char> router_sm(n_sm, 0);
  // pt < 0: any SM; by_layer: least bytes in the layer so far (put_layer), not in the phase
  auto emit = [&](std::vector<std::pair<Task, long long>>& ts, int pt, bool by_layer = false) {
    as.new_layer();
    for (auto& x : ts) {
      if (pt < 0) {
        as.put_any(x.first, x.second, router_sm);
      } else if (by_layer) {
        as.put_layer(x.first, x.second, pt);
      } else {
        const int s = as.put(x.first, x.second, pt);
        if (x.first.op == OP_ROUTER) router_sm[s] = 1;
      }
    }
    std::vector<std::vector<Task>> lists(n_sm);
    for (size_t i = 0; i < ts.size(); ++i) lists[i % n_sm].push_back(ts[i].first);
    if (!ts.empty()) per_op.push_back(std::move(lists));
    ts.clear();
  };

  std::vector<std::pair<Task, long long>> ts;
  // Batch 5-8: the input of layer l >= 1 (and the final norm's) is combined once, by column
  // slices, before the layer's other tasks: slice s writes the residual x = x + attn + sum of the
  // expert partials for its columns and each token's square sum over them; every norm then reads
  // only x and those sums (at batch 8 each block would otherwise read every input of every token)
  const int n_slices = combine_slices_for(B, H);
  auto emit_combine = [&](int l) {
    if (n_slices == 0) return;
    for (int sl = 0; sl < n_slices; ++sl)
      ts.push_back({mkt(OP_COMBINE, l, sl, n_slices, 0), (long long)(2 + kMoeParts) * kCombineCols * B * 4});
    cnt[cmap.combine(l)] = n_slices;
    emit(ts, PA);
  };
  for (int l = 0; l < L; ++l) {
    std::fill(router_sm.begin(), router_sm.end(), 0);
    as.new_layer();
    as.begin_layer();
    if (l > 0) emit_combine(l);
    // Per layer, in an order that is a topological order of the dependencies (so no SM can
    // wait on work listed after its own): router, QKV, expert gate/up (needs the routing),
    // attention (needs its group's QKV), expert down (needs all gate/up), O-proj (needs
    // attention). Expert work sits between QKV and attention so that it covers the time the
    // QKV results take to complete everywhere.
    // router: one stage per task; the first task stores x of this layer
    int n_router = 0;
    for (int r0 = 0; r0 < E; r0 += gh.RS, ++n_router)
      ts.push_back({mkt(OP_ROUTER, l, r0, std::min(gh.RS, E - r0), 0, r0 == 0 ? TF_WRITE_X : 0),
                    std::min(gh.RS, E - r0) * row_h});
    cnt[cmap.router_arrive(l)] = n_router;
    cnt[cmap.route(l)] = 1;
    emit(ts, PM);
    // QKV units, group-major, a few stages per task
    const int upg = (G + 2) * (d / 8);
    for (int g = 0; g < nkv; ++g) {
      int n = 0;
      for (int u = g * upg; u < (g + 1) * upg; u += qkv_per_task, ++n)
        ts.push_back({mkt(OP_QKV, l, u, std::min(qkv_per_task, (g + 1) * upg - u), g),
                      std::min(qkv_per_task, (g + 1) * upg - u) * 8 * row_h});
      cnt[cmap.qkv(l, g)] = n;
    }
    emit(ts, n_attn < n_sm ? -1 : PA);
    // expert gate/up: task k of n takes units [k U / n, (k + 1) U / n) of the U = active experts
    // x tiles units of the step
    const int n_gu = n_gu_tasks;
    for (int k = 0; k < n_gu; ++k)
      ts.push_back({mkt(OP_GU, l, k, n_gu, 0), (long long)(live * maxa * tiles * 2 * kGuRows * row_h / n_gu)});
    cnt[cmap.gu(l)] = n_gu;
    emit(ts, PM);
    // attention chunks: task i of every layer on the same attention SM (i mod n_attn), which then
    // reads the same pages, so their ids stay cached there
    {
      int i = 0;
      std::vector<std::vector<Task>> lists(n_sm);
      for (int b = 0; b < B; ++b)
        for (int g = 0; g < nkv; ++g)
          for (int ch = 0; ch < P.n_chunks[b]; ++ch, ++i) {
            const int p0 = ch * cp, p1 = (ch == P.n_chunks[b] - 1) ? npg[b] : std::min(npg[b], p0 + cp);
            const Task t = mkt(OP_ATTN, l, b, g, ch);
            as.put_on(t, std::max(0, p1 - p0) * 2LL * kPage * d * 2, i % n_attn);
            lists[i % n_sm].push_back(t);
          }
      per_op.push_back(std::move(lists));
    }
    for (int g = 0; g < nkv; ++g) cnt[cmap.attn(l, g)] = B;
    // expert down: units u = row block * parts + part (kDnRows rows over the routed experts of
    // rank part, part + parts, ...), one per task; without a partition, the SMs with the fewest
    // bytes in the layer so far take the phase's extra tasks (as for O-proj below)
    int n_down = 0;
    for (int u = 0; u < (H / kDnRows) * parts; ++u, ++n_down)
      ts.push_back({mkt(OP_DOWN, l, u, 1, 0), (long long)((double)kDnRows * I * 2 * live * maxa / parts)});
    emit(ts, PM, n_attn == n_sm);
    // O-proj: blocks of RS rows; at batch <= 4 (and at most two 2048-column chunks) a task takes
    // several blocks, reusing one load of the attention output, about one task per SM
    const int o_blocks = (H + go.RS - 1) / go.RS;
    const int o_per = (B <= 4 && go.NCS <= 2) ? (o_blocks + n_attn - 1) / n_attn : 1;
    int n_o = 0;
    for (int r0 = 0; r0 < H; r0 += o_per * go.RS, ++n_o)
      ts.push_back({mkt(OP_O, l, r0, std::min(o_per * go.RS, H - r0), 0), std::min(o_per * go.RS, H - r0) * 2LL * od});
    // when every SM takes both branches, O-proj is the layer's last phase and each SM reaches it
    // after its own gate/up, attention and down work: the SMs with the fewest bytes in the layer
    // so far take the phase's extra tasks (by step totals, the SMs whose down work ended last
    // took two O-proj tasks each at batch 8, ~10 us after the others)
    emit(ts, PA, n_attn == n_sm);
    cnt[cmap.layer(l)] = n_o + n_down;
  }
  as.new_layer();
  emit_combine(L);
  as.new_layer();
  // LM head: contiguous row ranges of whole stages, at most one task per SM (on the least
  // loaded SMs): the argmax takes one candidate per LM task
  {
    const int stages = (V + gh.RS - 1) / gh.RS;
    const int per = (stages + n_sm - 1) / n_sm;
    int slot = 0;
    for (int s0 = 0; s0 < stages; s0 += per, ++slot) {
      const int r0 = s0 * gh.RS, r1 = std::min(V, (s0 + per) * gh.RS);
      ts.push_back({mkt(OP_LM, L, r0, r1 - r0, slot, TF_LAST_LM | (slot == 0 ? TF_WRITE_X : 0)), (r1 - r0) * row_h});
    }
    P.n_lm_sm = slot;
    cnt[cmap.lm_arrive()] = slot;
    std::vector<int> order(n_sm);
    for (int i = 0; i < n_sm; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return as.total[x] < as.total[y]; });
    std::vector<std::vector<Task>> lists(n_sm);
    for (size_t i = 0; i < ts.size(); ++i) {
      const int sm = order[i % n_sm];
      as.lists[sm].push_back(ts[i].first);
      as.load[sm] += ts[i].second;
      as.total[sm] += ts[i].second;
      lists[i % n_sm].push_back(ts[i].first);
    }
    per_op.push_back(std::move(lists));
    ts.clear();
  }

  // flatten: megakernel lists, then per-op launches
  P.all.clear();
  P.begin.clear();
  for (int s = 0; s < n_sm; ++s) {
    P.begin.push_back((int32_t)P.all.size());
    P.all.insert(P.all.end(), as.lists[s].begin(), as.lists[s].end());
  }
  P.begin.push_back((int32_t)P.all.size());
  P.n_tasks = (int)P.all.size();
  for (auto& launch : per_op) {
    for (int s = 0; s < n_sm; ++s) {
      P.begin.push_back((int32_t)P.all.size());
      P.all.insert(P.all.end(), launch[s].begin(), launch[s].end());
    }
    P.begin.push_back((int32_t)P.all.size());
  }
  P.n_op_launches = (int)per_op.size();
  P.load = as.total;
  return MK_OK;
}

extern "C" mk_status mk_plan_schedule(const mk_model_cfg* cfg, int32_t n_sm, int32_t batch, const int32_t* seq_lens,
                                      mk_plan_info* info, void* tasks, int32_t tasks_cap, int32_t* sm_begin,
                                      int64_t* sm_bytes) {
  if (!cfg || !info) return MK_ERR_INVALID_ARG;
  Plan P;
  mk_status s = plan_schedule(*cfg, n_sm, batch, seq_lens, P);
  if (s != MK_OK) return s;
  info->n_tasks = P.n_tasks;
  info->n_counters = (int32_t)P.cnt.size();
  info->max_chunks = P.max_chunks;
  info->n_lm_sm = P.n_lm_sm;
  info->n_attn_sm = P.n_attn_sm;
  info->n_op_launches = P.n_op_launches;
  if (tasks) {
    if (tasks_cap < P.n_tasks) return MK_ERR_INVALID_ARG;
    memcpy(tasks, P.all.data(), sizeof(Task) * (size_t)P.n_tasks);
  }
  if (sm_begin) memcpy(sm_begin, P.begin.data(), sizeof(int32_t) * (size_t)(n_sm + 1));
  if (sm_bytes)
    for (int i = 0; i < n_sm; ++i) sm_bytes[i] = P.load[i];
  return MK_OK;
}

extern "C" mk_status mk_build_schedule(mk_ctx* c, int32_t batch, const int32_t* seq_lens, const int32_t* block_tables) {
  if (!c) return MK_ERR_INVALID_ARG;
  const mk_model_cfg& m = c->cfg;
  if (batch < 1 || batch > m.max_batch || !seq_lens || !block_tables)
    return fail(c, MK_ERR_INVALID_ARG, "batch outside 1..max_batch or null array");
  Plan P;
  if (plan_schedule(m, c->n_sm, batch, seq_lens, P) != MK_OK)
    return fail(c, MK_ERR_INVALID_ARG, "sequence length negative or beyond the block table");
  cudaDeviceSynchronize();
  free_schedule(c);
  const int B = batch;
  const size_t part = (size_t)m.n_layers * B * m.n_kv_heads * P.max_chunks * (16 + 8 * (size_t)m.head_dim);
  bool okm = dalloc(&c->d_tasks, P.all.size()) == cudaSuccess && dalloc(&c->d_sm_begin, P.begin.size()) == cudaSuccess &&
             dalloc(&c->d_cnt, P.cnt.size()) == cudaSuccess && dalloc(&c->d_chunk_pages, B) == cudaSuccess &&
             dalloc(&c->d_n_chunks, B) == cudaSuccess && dalloc(&c->apart, part) == cudaSuccess &&
             dalloc(&c->counters, P.cnt.size() * kCounterStride) == cudaSuccess;
  if (!okm) {
    cudaGetLastError();
    free_schedule(c);
    return fail(c, MK_ERR_OOM, "schedule allocation failed");
  }
  CK(cudaMemcpy(c->d_tasks, P.all.data(), P.all.size() * sizeof(Task), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(c->d_sm_begin, P.begin.data(), P.begin.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(c->d_cnt, P.cnt.data(), P.cnt.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(c->d_chunk_pages, P.chunk_pages.data(), B * sizeof(int32_t), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(c->d_n_chunks, P.n_chunks.data(), B * sizeof(int32_t), cudaMemcpyHostToDevice));
  CK(cudaMemset(c->counters, 0, P.cnt.size() * kCounterStride * sizeof(uint32_t)));
  CK(cudaMemset(c->status, 0, ST_WORDS * sizeof(int32_t)));
  c->n_tasks = P.n_tasks;
  c->n_counters = (int)P.cnt.size();
  c->max_chunks = P.max_chunks;
  c->n_lm_sm = P.n_lm_sm;
  c->n_op_launches = P.n_op_launches;
  c->B = B;
  c->block_table = block_tables;
  c->epoch = 0;
  c->scheduled = true;
  return MK_OK;
}

// ------------------------------------------------------------------ launches

static mk_status tensor_maps(mk_ctx* c, const mk_kv_pages* kv) {
  if (c->tm_k_ptr == kv->k && c->tm_v_ptr == kv->v && c->tm_pages == kv->num_pages) return MK_OK;
  const mk_model_cfg& m = c->cfg;
  const uint64_t rows = (uint64_t)m.n_layers * kv->num_pages * m.n_kv_heads * kPage;
  if (rows >= (1ull << 31)) return fail(c, MK_ERR_UNSUPPORTED, "KV pool too large for 32-bit TMA coordinates");
  const cuuint32_t halves = (cuuint32_t)m.head_dim / 64;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, halves};
  cuuint64_t strides[2] = {(cuuint64_t)m.head_dim * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)kPage, halves};
  cuuint32_t estr[3] = {1, 1, 1};
  for (int i = 0; i < 2; ++i) {
    CUresult r = c->encode(i ? &c->tm.v : &c->tm.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, i ? kv->v : kv->k, dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(c, MK_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV pool");
  }
  c->tm_k_ptr = kv->k;
  c->tm_v_ptr = kv->v;
  c->tm_pages = kv->num_pages;
  return MK_OK;
}

static Params make_params(mk_ctx* c, const int32_t* tokens, const int32_t* positions, const mk_kv_pages* kv,
                          float* logits, int32_t* argmax, int pos_offset) {
  const mk_model_cfg& m = c->cfg;
  Params p;
  memset(&p, 0, sizeof(p));
  p.L = m.n_layers; p.H = m.hidden; p.nq = m.n_q_heads; p.nkv = m.n_kv_heads; p.d = m.head_dim;
  p.E = m.n_experts; p.topk = m.top_k; p.I = m.expert_inter; p.V = m.vocab; p.B = c->B;
  p.max_pages = m.max_pages_per_seq; p.num_pages = kv->num_pages; p.n_sm = c->n_sm;
  p.qkv_rows = (m.n_q_heads + 2 * m.n_kv_heads) * m.head_dim; p.od = m.n_q_heads * m.head_dim;
  p.group = m.n_q_heads / m.n_kv_heads; p.max_chunks = c->max_chunks; p.n_lm_sm = c->n_lm_sm; p.max_pos = c->max_pos;
  p.eps = m.rms_eps;
  p.pos_offset = pos_offset;
  p.timeout_ns = c->wait_ns;
  p.embed = (const uint16_t*)c->w.embed; p.norm_gain = (const uint16_t*)c->w.norm_gain;
  p.w_qkv = (const uint16_t*)c->w.w_qkv; p.w_o = (const uint16_t*)c->w.w_o; p.w_router = (const uint16_t*)c->w.w_router;
  p.w_gate_up = (const uint16_t*)c->w.w_gate_up; p.w_down = (const uint16_t*)c->w.w_down;
  p.final_gain = (const uint16_t*)c->w.final_gain; p.lm_head = (const uint16_t*)c->w.lm_head;
  p.router_bias = c->w.router_bias;
  p.rope = c->rope;
  p.kpool = (uint16_t*)kv->k; p.vpool = (uint16_t*)kv->v; p.block_table = c->block_table;
  p.token_ids = tokens; p.positions = positions; p.logits = logits; p.argmax_out = argmax;
  p.tasks = c->d_tasks; p.sm_begin = c->d_sm_begin; p.cnt_per_step = c->d_cnt;
  p.chunk_pages = c->d_chunk_pages; p.n_chunks = c->d_n_chunks;
  p.xs = c->xs; p.q = c->q; p.knew = c->knew; p.vnew = c->vnew; p.apart = c->apart; p.attn_o = c->attn_o;
  p.attn_out = c->attn_out; p.rlogits = c->rlogits; p.hsw = c->hsw; p.attn_hl = c->attn_hl; p.moe_out = c->moe_out;
  p.moe_part = c->moe_part; p.moe_parts = moe_parts_for(c->B, m.top_k, m.n_experts); p.route = c->route;
  p.combine_slices = combine_slices_for(c->B, m.hidden); p.css = c->css;
  p.lm_best_v = c->lm_best_v; p.lm_best_i = c->lm_best_i; p.counters = c->counters; p.status = c->status;
  p.status_host = c->status_host_dev; p.topk_ids = c->topk_ids; p.topk_w = c->topk_w;
  p.trace = c->trace; p.trace_count = c->trace_count; p.trace_cap = c->trace_cap;
  return p;
}

static mk_status check_latched(mk_ctx* c) {
  const int code = *(volatile int32_t*)c->status_host;
  if (code != 0) return fail(c, (mk_status)code, "device error latched by an earlier step (call mk_status_sync)");
  return MK_OK;
}

static mk_status run_step(mk_ctx* c, Params& p, cudaStream_t st) {
  ++c->epoch;
  p.epoch = c->epoch;
  if (c->trace) CK(cudaMemsetAsync(c->trace_count, 0, sizeof(unsigned long long), st));
  if (c->mode == MK_MODE_MEGAKERNEL) {
    p.sm_begin = c->d_sm_begin;
    CK(launch_decode(p, c->tm, st));
  } else {
    for (int i = 0; i < c->n_op_launches; ++i) {
      p.sm_begin = c->d_sm_begin + (size_t)(i + 1) * (c->n_sm + 1);
      CK(launch_decode(p, c->tm, st));
    }
  }
  return MK_OK;
}

static mk_status step_checks(mk_ctx* c, const mk_kv_pages* kv) {
  if (!c->scheduled) return fail(c, MK_ERR_NO_SCHEDULE, "mk_build_schedule has not succeeded");
  if (!kv || !kv->k || !kv->v || kv->num_pages <= 0 || !aligned16(kv->k) || !aligned16(kv->v))
    return fail(c, MK_ERR_INVALID_ARG, "bad KV pages");
  mk_status s = check_latched(c);
  if (s != MK_OK) return s;
  return tensor_maps(c, kv);
}

extern "C" mk_status mk_decode_step(mk_ctx* c, const int32_t* token_ids, const int32_t* positions, const mk_kv_pages* kv,
                                    float* logits_out, int32_t* argmax_out, void* stream) {
  if (!c) return MK_ERR_INVALID_ARG;
  if (!token_ids || !positions) return fail(c, MK_ERR_INVALID_ARG, "null token_ids or positions");
  mk_status s = step_checks(c, kv);
  if (s != MK_OK) return s;
  Params p = make_params(c, token_ids, positions, kv, logits_out, argmax_out, 0);
  return run_step(c, p, (cudaStream_t)stream);
}

extern "C" mk_status mk_decode_greedy(mk_ctx* c, int32_t n_steps, const int32_t* token_ids, const int32_t* positions,
                                      const mk_kv_pages* kv, float* logits_out, int32_t* tokens_out, void* stream) {
  if (!c) return MK_ERR_INVALID_ARG;
  if (!token_ids || !positions || !tokens_out || n_steps < 1)
    return fail(c, MK_ERR_INVALID_ARG, "null argument or n_steps < 1");
  mk_status s = step_checks(c, kv);
  if (s != MK_OK) return s;
  for (int i = 0; i < n_steps; ++i) {
    const int32_t* tok = i == 0 ? token_ids : tokens_out + (size_t)(i - 1) * c->B;
    Params p = make_params(c, tok, positions, kv, i == n_steps - 1 ? logits_out : nullptr,
                           tokens_out + (size_t)i * c->B, i);
    s = run_step(c, p, (cudaStream_t)stream);
    if (s != MK_OK) return s;
  }
  return MK_OK;
}

extern "C" mk_status mk_status_sync(mk_ctx* c) {
  if (!c) return MK_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaDeviceSynchronize");
  int32_t st[ST_WORDS];
  e = cudaMemcpy(st, c->status, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "status copy");
  if (st[ST_CODE] == 0) return MK_OK;
  char buf[200];
  const char* what = st[ST_CODE] == MK_ERR_BAD_PAGE        ? "page id out of range (sequence, page index)"
                     : st[ST_CODE] == MK_ERR_DEVICE_TIMEOUT ? "a device-side wait ran out of time (wait, progress)"
                     : st[ST_CODE] == MK_ERR_BAD_TOKEN      ? "token id out of range (sequence, token)"
                                                            : "device error";
  snprintf(buf, sizeof(buf), "device error %d: %s = (%d, %d)", st[ST_CODE], what, st[ST_AUX0], st[ST_AUX1]);
  c->err = buf;
  cudaMemset(c->status, 0, ST_WORDS * sizeof(int32_t));
  *(volatile int32_t*)c->status_host = 0;
  if (c->counters) cudaMemset(c->counters, 0, (size_t)c->n_counters * kCounterStride * sizeof(uint32_t));
  c->epoch = 0;
  cudaDeviceSynchronize();
  return (mk_status)st[ST_CODE];
}

extern "C" const char* mk_last_error(const mk_ctx* c) { return c ? c->err.c_str() : "null context"; }

extern "C" mk_status mk_set_mode(mk_ctx* c, int mode) {
  if (!c || (mode != MK_MODE_MEGAKERNEL && mode != MK_MODE_PER_OP)) return MK_ERR_INVALID_ARG;
  c->mode = mode;
  return MK_OK;
}

extern "C" mk_status mk_set_wait_limit(mk_ctx* c, int64_t ns) {
  if (!c || ns < 1000 || ns > 60000000000LL) return MK_ERR_INVALID_ARG;
  c->wait_ns = ns;
  return MK_OK;
}

extern "C" mk_status mk_enable_trace(mk_ctx* c, void* buf, size_t bytes) {
  if (!c) return MK_ERR_INVALID_ARG;
  if (!buf) {
    c->trace = nullptr;
    c->trace_count = nullptr;
    c->trace_cap = 0;
    return MK_OK;
  }
  if (bytes < 16 + sizeof(mk_trace_entry) || !aligned16(buf)) return fail(c, MK_ERR_INVALID_ARG, "trace buffer too small");
  c->trace_count = (unsigned long long*)buf;
  c->trace = (mk_trace_entry*)((char*)buf + 16);
  c->trace_cap = (long long)((bytes - 16) / sizeof(mk_trace_entry));
  return MK_OK;
}

extern "C" mk_status mk_get_activations(const mk_ctx* c, mk_activations* out) {
  if (!c || !out) return MK_ERR_INVALID_ARG;
  out->x = c->xs;
  out->q = c->q;
  out->attn = c->attn_o;
  out->attn_out = c->attn_out;
  out->moe_out = c->moe_out;
  out->router = c->rlogits;
  out->topk_ids = c->topk_ids;
  out->topk_w = c->topk_w;
  return MK_OK;
}

extern "C" mk_status mk_get_launch_info(const mk_ctx* c, int32_t* n_sm, int32_t* tasks, int32_t* launches) {
  if (!c) return MK_ERR_INVALID_ARG;
  if (n_sm) *n_sm = c->n_sm;
  if (tasks) *tasks = c->scheduled ? c->n_tasks : 0;
  if (launches) *launches = c->mode == MK_MODE_MEGAKERNEL ? 1 : c->n_op_launches;
  return MK_OK;
}
