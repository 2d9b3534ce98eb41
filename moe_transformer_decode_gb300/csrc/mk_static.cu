// mk_decode_step_noalloc: the decode step for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: code running under a memory pool or arena that owns
// every device allocation, plugins whose host process forbids allocation after start-up,
// and paths that must not take the allocator's locks or trigger its implicit device
// synchronisation. This entry point runs the same persistent kernel as mk_decode_step, but
// keeps its whole workspace (activations, schedule, counters, RoPE table) in one file-scope
// device array of fixed size, so it allocates nothing. The caller passes weights, KV pages,
// inputs and outputs exactly as for the context-based API.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "mk_internal.h"

namespace mk {
int kernel_smem_bytes();
cudaError_t launch_decode(const Params& p, const TensorMaps& tm, cudaStream_t st);
cudaError_t configure_kernels();
}  // namespace mk

using namespace mk;

// Every GPU that loads the library reserves this much device memory until the process exits.
static constexpr size_t kScratchBytes = (size_t)MK_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char mk_noalloc_scratch[kScratchBytes];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace {

constexpr int kMaxDevices = 64;

// Per-device set-up, done by the first call on each device with that device current.
struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of mk_noalloc_scratch on this device
  int n_sm = 0;
};
DeviceSetup g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
std::mutex g_mu;

void set_msg(char* msg, int32_t len, const char* text) {
  if (msg && len > 0) snprintf(msg, (size_t)len, "%s", text);
}

// Bump allocator over the scratch array (offsets only; nothing is allocated).
struct Carve {
  size_t off = 0;
  template <typename T>
  size_t take(size_t count) {
    off = (off + 255) & ~(size_t)255;
    const size_t at = off;
    off += (count ? count : 1) * sizeof(T);
    return at;
  }
};

}  // namespace

extern "C" mk_status mk_decode_step_noalloc(const mk_model_cfg* cfg, const mk_weight_ptrs* w, int32_t batch,
                                            const int32_t* seq_lens, const int32_t* block_tables,
                                            const int32_t* token_ids, const int32_t* positions, const mk_kv_pages* kv,
                                            float* logits_out, int32_t* argmax_out, void* stream, char* msg,
                                            int32_t msg_len) {
  if (!cfg || !w || !seq_lens || !block_tables || !token_ids || !positions || !kv) {
    set_msg(msg, msg_len, "null argument");
    return MK_ERR_INVALID_ARG;
  }
  // the same checks as mk_create, before any size or offset is derived from the config
  const char* why = "";
  const mk_status vs = validate_model(cfg, w, &why);
  if (vs != MK_OK) {
    set_msg(msg, msg_len, why);
    return vs;
  }
  if (!kv->k || !kv->v || kv->num_pages <= 0 || ((uintptr_t)kv->k & 15u) != 0 || ((uintptr_t)kv->v & 15u) != 0) {
    set_msg(msg, msg_len, "KV pools null, empty or not 16-byte aligned");
    return MK_ERR_INVALID_ARG;
  }
  const mk_model_cfg& m = *cfg;
  const int od = m.n_q_heads * m.head_dim;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_msg(msg, msg_len, "no current CUDA device");
    return MK_ERR_CUDA;
  }
  DeviceSetup& ds = g_dev[dev];
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!ds.ready) {
      void* addr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&addr, mk_noalloc_scratch);
      if (e != cudaSuccess || !addr) {
        set_msg(msg, msg_len, "cudaGetSymbolAddress of the scratch array failed");
        return MK_ERR_CUDA;
      }
      int coop = 0, smem = 0;
      cudaDeviceGetAttribute(&ds.n_sm, cudaDevAttrMultiProcessorCount, dev);
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
      cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      if (!coop || smem < kernel_smem_bytes()) {
        set_msg(msg, msg_len, "device lacks cooperative launch or enough shared memory");
        return MK_ERR_UNSUPPORTED;
      }
      if (configure_kernels() != cudaSuccess) {
        set_msg(msg, msg_len, "kernel configuration failed");
        return MK_ERR_CUDA;
      }
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || !fn) {
          set_msg(msg, msg_len, "cuTensorMapEncodeTiled not available");
          return MK_ERR_CUDA;
        }
        g_encode = (EncodeTiledFn)fn;
      }
      ds.scratch = (unsigned char*)addr;
      ds.ready = true;
    }
  }

  // host-side plan (host memory only)
  Plan P;
  if (plan_schedule(m, ds.n_sm, batch, seq_lens, P) != MK_OK) {
    set_msg(msg, msg_len, "batch outside 1..max_batch, or a sequence length negative or beyond the block table");
    return MK_ERR_INVALID_ARG;
  }
  const size_t L = m.n_layers, B = batch, H = m.hidden, d = m.head_dim, nkv = m.n_kv_heads;
  const int max_pos = m.max_pages_per_seq * kPage;

  // workspace layout inside the scratch array
  Carve cv;
  const size_t o_xs = cv.take<float>((L + 1) * B * H), o_q = cv.take<float>(L * B * m.n_q_heads * d);
  const size_t o_knew = cv.take<float>(L * B * nkv * d), o_vnew = cv.take<float>(L * B * nkv * d);
  const size_t o_apart = cv.take<float>(L * B * nkv * P.max_chunks * (16 + 8 * d));
  const size_t o_attn_o = cv.take<float>(L * B * od), o_attn_out = cv.take<float>(L * B * H);
  const size_t o_rl = cv.take<float>(L * B * m.n_experts);
  const size_t o_hsw = cv.take<uint8_t>(L * kMaxActive * hsw_slot_bytes(m.expert_inter));
  const size_t o_moep = cv.take<float>(L * kMoeParts * B * H);
  const size_t o_css = cv.take<float>((L + 1) * kMaxCombineSlices * kMaxB);
  const size_t o_attn_hl = cv.take<uint16_t>(L * 2 * B * od);
  const size_t o_moe = cv.take<float>(L * B * H), o_route = cv.take<Route>(L);
  const size_t o_lmv = cv.take<float>((size_t)ds.n_sm * kMaxB), o_lmi = cv.take<int32_t>((size_t)ds.n_sm * kMaxB);
  const size_t o_tki = cv.take<int32_t>(L * B * m.top_k), o_tkw = cv.take<float>(L * B * m.top_k);
  const size_t o_cnt = cv.take<uint32_t>(P.cnt.size() * kCounterStride), o_status = cv.take<int32_t>(ST_WORDS);
  const size_t o_rope = cv.take<float2>((size_t)max_pos * (d / 2));
  const size_t o_tasks = cv.take<Task>((size_t)P.n_tasks), o_begin = cv.take<int32_t>((size_t)ds.n_sm + 1);
  const size_t o_cps = cv.take<int32_t>(P.cnt.size());
  const size_t o_chp = cv.take<int32_t>(B), o_nch = cv.take<int32_t>(B);
  if (cv.off > kScratchBytes) {
    char buf[200];
    snprintf(buf, sizeof(buf), "workspace of %zu bytes exceeds the %zu-byte static scratch (smaller model, batch or context)",
             cv.off, kScratchBytes);
    set_msg(msg, msg_len, buf);
    return MK_ERR_UNSUPPORTED;
  }
  const uint64_t rows = (uint64_t)m.n_layers * kv->num_pages * m.n_kv_heads * kPage;
  if (rows >= (1ull << 31)) {
    set_msg(msg, msg_len, "KV pool too large for 32-bit TMA coordinates");
    return MK_ERR_UNSUPPORTED;
  }

  cudaStream_t st = (cudaStream_t)stream;
  unsigned char* s = ds.scratch;
  std::vector<float2> rope((size_t)max_pos * (d / 2));
  for (int pos = 0; pos < max_pos; ++pos)
    for (size_t i = 0; i < d / 2; ++i) {
      const double ang = (double)pos * std::pow((double)m.rope_theta, -2.0 * (double)i / (double)d);
      rope[(size_t)pos * (d / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
  // pageable host sources: each copy has read its source when the call returns
  cudaError_t e = cudaMemcpyAsync(s + o_rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(s + o_tasks, P.all.data(), (size_t)P.n_tasks * sizeof(Task), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(s + o_begin, P.begin.data(), ((size_t)ds.n_sm + 1) * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(s + o_cps, P.cnt.data(), P.cnt.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(s + o_chp, P.chunk_pages.data(), B * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(s + o_nch, P.n_chunks.data(), B * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  // the scratch keeps the previous call's contents: counters and status must start at zero
  if (e == cudaSuccess) e = cudaMemsetAsync(s + o_cnt, 0, P.cnt.size() * kCounterStride * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(s + o_status, 0, ST_WORDS * sizeof(int32_t), st);
  if (e != cudaSuccess) {
    set_msg(msg, msg_len, cudaGetErrorString(e));
    return MK_ERR_CUDA;
  }

  TensorMaps tm;
  if (encode_weight_maps((void*)g_encode, m, w, tm) != MK_OK) {
    set_msg(msg, msg_len, "cuTensorMapEncodeTiled failed for the expert or O-proj weights");
    return MK_ERR_INVALID_ARG;
  }
  {
    const cuuint32_t halves = (cuuint32_t)m.head_dim / 64;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, halves};
    cuuint64_t strides[2] = {(cuuint64_t)m.head_dim * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kPage, halves};
    cuuint32_t estr[3] = {1, 1, 1};
    for (int i = 0; i < 2; ++i)
      if (g_encode(i ? &tm.v : &tm.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, i ? kv->v : kv->k, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        set_msg(msg, msg_len, "cuTensorMapEncodeTiled failed for the KV pool (alignment?)");
        return MK_ERR_INVALID_ARG;
      }
  }

  Params p;
  memset(&p, 0, sizeof(p));
  p.L = m.n_layers; p.H = m.hidden; p.nq = m.n_q_heads; p.nkv = m.n_kv_heads; p.d = m.head_dim;
  p.E = m.n_experts; p.topk = m.top_k; p.I = m.expert_inter; p.V = m.vocab; p.B = batch;
  p.max_pages = m.max_pages_per_seq; p.num_pages = kv->num_pages; p.n_sm = ds.n_sm;
  p.qkv_rows = (m.n_q_heads + 2 * m.n_kv_heads) * m.head_dim; p.od = od; p.group = m.n_q_heads / m.n_kv_heads;
  p.max_chunks = P.max_chunks; p.n_lm_sm = P.n_lm_sm; p.max_pos = max_pos; p.eps = m.rms_eps;
  p.epoch = 1;  // counters were zeroed above
  p.pos_offset = 0;
  p.timeout_ns = 2000000000LL;
  p.embed = (const uint16_t*)w->embed; p.norm_gain = (const uint16_t*)w->norm_gain; p.w_qkv = (const uint16_t*)w->w_qkv;
  p.w_o = (const uint16_t*)w->w_o; p.w_router = (const uint16_t*)w->w_router; p.w_gate_up = (const uint16_t*)w->w_gate_up;
  p.w_down = (const uint16_t*)w->w_down; p.final_gain = (const uint16_t*)w->final_gain;
  p.lm_head = (const uint16_t*)w->lm_head; p.router_bias = w->router_bias;
  p.rope = (const float2*)(s + o_rope);
  p.kpool = (uint16_t*)kv->k; p.vpool = (uint16_t*)kv->v; p.block_table = block_tables;
  p.token_ids = token_ids; p.positions = positions; p.logits = logits_out; p.argmax_out = argmax_out;
  p.tasks = (const Task*)(s + o_tasks); p.sm_begin = (const int32_t*)(s + o_begin);
  p.cnt_per_step = (const int32_t*)(s + o_cps); p.chunk_pages = (const int32_t*)(s + o_chp);
  p.n_chunks = (const int32_t*)(s + o_nch);
  p.xs = (float*)(s + o_xs); p.q = (float*)(s + o_q); p.knew = (float*)(s + o_knew); p.vnew = (float*)(s + o_vnew);
  p.apart = (float*)(s + o_apart); p.attn_o = (float*)(s + o_attn_o); p.attn_out = (float*)(s + o_attn_out);
  p.rlogits = (float*)(s + o_rl); p.hsw = (uint8_t*)(s + o_hsw);
  p.moe_part = (float*)(s + o_moep); p.moe_parts = moe_parts_for(batch, m.top_k, m.n_experts);
  p.combine_slices = combine_slices_for(batch, m.hidden); p.css = (float*)(s + o_css); p.attn_hl = (uint16_t*)(s + o_attn_hl); p.moe_out = (float*)(s + o_moe);
  p.route = (Route*)(s + o_route); p.lm_best_v = (float*)(s + o_lmv); p.lm_best_i = (int32_t*)(s + o_lmi);
  p.topk_ids = (int32_t*)(s + o_tki); p.topk_w = (float*)(s + o_tkw);
  p.counters = (uint32_t*)(s + o_cnt); p.status = (int32_t*)(s + o_status);
  p.status_host = nullptr;
  p.trace = nullptr; p.trace_count = nullptr; p.trace_cap = 0;

  e = launch_decode(p, tm, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    set_msg(msg, msg_len, cudaGetErrorString(e));
    return MK_ERR_CUDA;
  }
  int32_t status[ST_WORDS];
  e = cudaMemcpy(status, s + o_status, sizeof(status), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    set_msg(msg, msg_len, cudaGetErrorString(e));
    return MK_ERR_CUDA;
  }
  if (status[ST_CODE] != 0) {
    char buf[120];
    snprintf(buf, sizeof(buf), "device error %d (aux %d, %d)", status[ST_CODE], status[ST_AUX0], status[ST_AUX1]);
    set_msg(msg, msg_len, buf);
    return (mk_status)status[ST_CODE];
  }
  set_msg(msg, msg_len, "");
  return MK_OK;
}
