// Internal layout shared by the host scheduler (mk_host.cpp) and the persistent kernel
// (mk_kernel.cu): task descriptors, dependency counters, routing records, kernel params.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include <vector>

#include "../../include/mk.h"

namespace mk {

constexpr int kConsumerWarps = 8;
// Two consumer warpgroups and one producer warpgroup (one thread of it issues the copies).
// Whole warpgroups let the producer hand its registers to the consumers (setmaxnreg).
constexpr int kThreads = (kConsumerWarps + 4) * 32;
constexpr int kProducerRegs = 56;
constexpr int kConsumerRegs = 224;
static_assert(kConsumerWarps == 8, "two consumer warpgroups");
static_assert(kProducerRegs * 128 + kConsumerRegs * 256 <= (65536 / kThreads) / 8 * 8 * kThreads,
              "register split exceeds the launch's allotment");
constexpr int kStagePayload = 32768;                 // data bytes of a ring stage
// ring slot: a stage, plus room for the tcgen05 A chunks (up to 4 KB) an expert-down stage carries
constexpr int kStageBytes = kStagePayload + 4096;
constexpr int kStages = 4;
// Expert GEMVs on tcgen05 (weights as the N operand, tokens x {hi, lo} as M). A stage holds
// kStageK = 128 columns of its weight rows as two 64-column (128-byte, swizzled) chunks. A gate/up
// unit is kGuRows gate rows and the matching up rows (two N = 64 products per k-step); a down unit
// is kDnRows output rows (N = 128) over the experts of one of kMoeParts partials.
constexpr int kTcK = 64;
constexpr int kStageK = 2 * kTcK;
constexpr int kGuRows = 64;
constexpr int kDnRows = 128;
constexpr int kMoeParts = 9;
// Expert-down partials of a step: partial j sums the routed experts of rank j, j + parts, ... in
// rank order, and the next layer's norm adds the partials in order. More partials give down more
// units (parallelism); fewer make the norm read less. At batch <= 4 kMoePartsSmall, at batch 8
// kMoeParts; never more than the experts a step can route to.
constexpr int kMoePartsSmall = 4;
__host__ __device__ constexpr int moe_parts_for(int batch, int top_k, int n_experts) {
  return (batch <= 4 ? kMoePartsSmall : kMoeParts) < (batch * top_k < n_experts ? batch * top_k : n_experts)
             ? (batch <= 4 ? kMoePartsSmall : kMoeParts)
             : (batch * top_k < n_experts ? batch * top_k : n_experts);
}
constexpr int kTmemCols = 512;
// the A operand (tokens x {hi, lo}, 8 rows per group, groups of 4 tokens) for one 64-column
// chunk: kMaxB / 4 groups of 1 KB
constexpr int kAChunkMax = (8 / 4) * 1024;  // 8 = kMaxB
constexpr int kABufBytes = 32 * kAChunkMax;          // the normalized input, hidden <= 2048
// Counters sit kCounterStride words (128 bytes) apart, so the lines that waiting warps poll spread
// over the L2 slices instead of all landing on one.
constexpr int kCounterStride = 32;
constexpr int kMaxB = 8;
constexpr int kMaxK = 8;
constexpr int kMaxActive = kMaxB * kMaxK;  // distinct experts a batch can route to
constexpr int kMaxExperts = 256;
constexpr int kPage = 16;

// Opcodes of the decode graph.
enum Op : uint8_t {
  OP_ROUTER = 1,  // router logits for a block of experts; last one computes top-k routing
  OP_QKV = 2,     // QKV rows + RoPE + KV append, a range of 8-row units of one KV group
  OP_ATTN = 3,    // paged GQA attention of one (sequence, KV group, chunk); last chunk combines
  OP_GU = 4,      // expert gate/up + SiLU*mul, a range of (row block, active expert) units
  OP_O = 5,       // O-proj rows, each warp released by its KV group's counter
  OP_DOWN = 6,    // expert down: (row block, partial) units, each over its share of the experts
  OP_LM = 7,      // LM-head rows + running argmax; the last LM task of the step reduces
  OP_COMBINE = 8  // batch 5-8: the residual of a layer's input for one column slice, written once
};
// Combine slices (batch 5-8): kCombineCols columns of the residual stream each. At batch <= 4
// there are none: every block combines the whole residual itself (small enough at that batch).
constexpr int kCombineCols = 16;
constexpr int kMaxCombineSlices = 2048 / kCombineCols;  // hidden <= 2048
__host__ __device__ constexpr int combine_slices_for(int batch, int hidden) {
  return batch > 4 ? hidden / kCombineCols : 0;
}
enum TaskFlag : uint8_t {
  TF_WRITE_X = 1,  // this task's block stores the residual stream x of its layer
  TF_LAST_LM = 2   // this SM's last LM task: publish its argmax candidate
};

struct Task {
  uint8_t op, flags;
  uint16_t layer;
  int32_t a, b, c;
};
static_assert(sizeof(Task) == 16, "task descriptor is 16 bytes");

// Routing of one layer for the whole batch (written by the last router task).
struct Route {
  int32_t n_active;
  int32_t pad[3];
  int32_t expert[kMaxActive];        // distinct routed experts, ascending id
  uint32_t mask[kMaxActive];         // bit b: token b routed to it
  float w[kMaxActive][kMaxB];        // routing weight (0 where not routed)
  int32_t ids[kMaxB][kMaxK];         // per token, top-k in rank order
  float wk[kMaxB][kMaxK];
};

// Counter indices (uint32, compared wrap-safely against epoch * per-step count).
struct CounterMap {
  int L, nkv, B;
  __host__ __device__ int layer(int l) const { return l; }
  __host__ __device__ int qkv(int l, int g) const { return L + l * nkv + g; }
  __host__ __device__ int router_arrive(int l) const { return L + L * nkv + l; }
  __host__ __device__ int route(int l) const { return 2 * L + L * nkv + l; }
  __host__ __device__ int gu(int l) const { return 3 * L + L * nkv + l; }
  __host__ __device__ int attn(int l, int g) const { return 4 * L + L * nkv + l * nkv + g; }
  __host__ __device__ int attn_arrive(int l, int b, int g) const { return 4 * L + 2 * L * nkv + (l * B + b) * nkv + g; }
  __host__ __device__ int lm_arrive() const { return 4 * L + 2 * L * nkv + L * B * nkv; }
  // combine slices done for the input of layer l, l = 1 .. L (L: the final norm's input)
  __host__ __device__ int combine(int l) const { return lm_arrive() + l; }
  __host__ __device__ int count() const { return lm_arrive() + L + 1; }
};

// Device status words.
enum { ST_CODE = 0, ST_AUX0 = 1, ST_AUX1 = 2, ST_ABORT = 3, ST_WORDS = 8 };

struct Params {
  // shape
  int L, H, nq, nkv, d, E, topk, I, V, B, max_pages, num_pages, n_sm;
  int qkv_rows, od, group, max_chunks, n_lm_sm, max_pos;
  float eps;
  uint32_t epoch;
  int pos_offset;  // added to positions[b] (greedy loop)
  long long timeout_ns;
  // weights (bf16 bits)
  const uint16_t *embed, *norm_gain, *w_qkv, *w_o, *w_router, *w_gate_up, *w_down, *final_gain, *lm_head;
  const float* router_bias;
  const float2* rope;  // [max_pos][d/2] (cos, sin)
  // KV cache
  uint16_t *kpool, *vpool;
  const int32_t* block_table;  // [B][max_pages]
  // step inputs / outputs
  const int32_t* token_ids;
  const int32_t* positions;
  float* logits;
  int32_t* argmax_out;
  // schedule
  const Task* tasks;
  const int32_t* sm_begin;     // [n_sm + 1] offsets into tasks
  const int32_t* cnt_per_step; // [counters] increments per step
  const int32_t* chunk_pages;  // [B] pages per attention chunk
  const int32_t* n_chunks;     // [B]
  // workspace
  float *xs, *q, *knew, *vnew, *apart, *attn_o, *attn_out, *rlogits, *moe_out;
  // expert down outputs as kMoeParts partials [L][kMoeParts][B][H] (part j sums the routed
  // experts of rank j mod parts), added in order by the next layer's residual + norm
  float* moe_part;
  int moe_parts;
  // batch 5-8: combine slices per layer input (0: every block combines the whole residual
  // itself) and their per-token square sums, [L + 1][kMaxCombineSlices][kMaxB]
  int combine_slices;
  float* css;
  // activations stored as bf16 hi/lo planes (hi = bf16(v), lo = bf16(v - hi)), the form the
  // tensor-core GEMV consumes: attention output [L][2][B][n_q d]
  uint16_t* attn_hl;
  // expert activations SiLU(gate) * up * routing weight as the tcgen05 A operand, per (layer,
  // active-expert rank): [I / 64 chunks][B > 4 ? 2 : 1 groups][8 rows = 4 tokens x {hi, lo}]
  // [128 bytes, 16-byte units XOR-swizzled by row], a slot of kHSlotBytes(I)
  uint8_t* hsw;
  Route* route;
  float* lm_best_v;
  int32_t* lm_best_i;
  int32_t* topk_ids;  // [L][B][topk]
  float* topk_w;
  uint32_t* counters;
  int32_t* status;
  int32_t* status_host;  // mapped host copy of the status code (written only on error)
  mk_trace_entry* trace;
  unsigned long long* trace_count;
  long long trace_cap;
};

// The host scheduler's output for one batch (see mk_host.cpp).
struct Plan {
  std::vector<Task> all;          // megakernel lists (per SM), then the per-op launches' lists
  std::vector<int32_t> begin;     // [n_sm + 1] offsets, then [n_sm + 1] per per-op launch
  std::vector<int32_t> cnt;       // counter increments per step
  std::vector<int32_t> chunk_pages, n_chunks;
  std::vector<long long> load;    // planned bytes per SM (megakernel lists)
  int max_chunks = 1, n_lm_sm = 0, n_tasks = 0, n_op_launches = 0;
  int n_attn_sm = 0;               // SMs [0, n_attn_sm) take the attention branch, the rest the experts
};
mk_status plan_schedule(const mk_model_cfg& m, int n_sm, int B, const int32_t* seq_lens, Plan& P);
// Checks a model config and its weight pointers (sizes, supported shapes, 16-byte alignment)
// for every entry point that takes them; *why (may be NULL) receives a static reason.
mk_status validate_model(const mk_model_cfg* cfg, const mk_weight_ptrs* w, const char** why);

struct TensorMaps {
  // KV pools as 3D {64, rows, head_dim / 64} bf16 views (a row is 2 head_dim bytes, a 64-wide
  // half of it 128 bytes), box {64, 16, head_dim / 64}, 128B swizzle: one copy lands a page's
  // rows as [half][row][128 bytes]
  CUtensorMap k, v;
  // expert weights as 3D {64, rows, K / 64} bf16 views with 128B swizzle (the tcgen05 operand
  // layout): gate/up rows [L][E][2I] over K = hidden, box {64, kGuRows, 1}; down rows [L][E][H]
  // over K = I, box {64, kDnRows, 2}
  CUtensorMap gu, dn;
  // O-proj weights [L][H][od] as a 3D {256, od / 256, L H} bf16 view without swizzle, box
  // {256, KS / 256, RS}: one copy lands a GEMV stage (RS rows x KS columns, row-major)
  CUtensorMap wo;
};
// bytes of one expert's activation slot in Params::hsw
inline __host__ __device__ size_t hsw_slot_bytes(int I) { return (size_t)(I / 64) * kAChunkMax; }
// encodes TensorMaps::gu, ::dn and ::wo over the caller's weights (encode_fn: cuTensorMapEncodeTiled)
mk_status encode_weight_maps(void* encode_fn, const mk_model_cfg& m, const mk_weight_ptrs* w, TensorMaps& tm);

}  // namespace mk
