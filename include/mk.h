/*
 * libmk — one decode step of a parallel-layer Mixture-of-Experts transformer as ONE
 * persistent CUDA kernel on an sm_103a GPU (GB300).
 *
 * The step (Cohere megakernel news pages; aimodeling.com "cohere-megakernel-north-mini-code-
 * h100", sections "One persistent kernel for the whole decode step" and "From demo to a full
 * serving system"; aibriefing.imbch.dev article 8171681, sections "Key Technologies and
 * Architecture" and "Scheduling and Performance Benchmarks"): for each sequence b with token
 * t_b at position p_b (= tokens already cached),
 *   x = E[t_b];  n = RMSNorm(x) * g_0
 *   per layer l:  q,k,v = W_qkv n; RoPE(q, k; p_b); append bf16 k, v to the paged cache;
 *                 o = GQA attention of q over cache positions 0..p_b;  a = W_o o
 *                 r = W_r n + bias; top-k experts, softmax over the k selected;
 *                 m = sum_j w_j W_down[e_j] (silu(W_gate[e_j] n) * W_up[e_j] n)
 *                 x = x + a + m;  n = RMSNorm(x) * g_{l+1}   (g_final after the last layer)
 *   logits = W_lm n;  next = argmax(logits)  (lowest id on ties)
 * Attention and the MoE read the same normalized input n (parallel layer). Readings taken
 * where the pages are silent: RMSNorm eps from the config (1e-6 in the shipped workloads),
 * rotate-half RoPE over the full head, contiguous GQA groups (q head h reads kv head
 * h / (n_q / n_kv)), router bias added before both top-k and softmax, untied LM head.
 *
 * Numerics: bf16 weights and KV; fp32 residual stream, norms, softmax and accumulation. Every
 * matrix product on the tensor cores takes its activation operand as a bf16 pair (hi = bf16(x),
 * lo = bf16(x - hi): at least 16 significant bits), so results stay close to fp32 products.
 *
 * Threading and streams: a context is used by one host thread at a time. Calls that take
 * a stream are asynchronous on it; host-detectable errors return at once, device-detected
 * errors (bad page id, bad token id, a dependency wait that timed out) are latched in the
 * context and returned by mk_status_sync() or by the next call.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MK_OK = 0,
  MK_ERR_INVALID_ARG = 1,     /* null pointer, size out of range, inconsistent config      */
  MK_ERR_UNSUPPORTED = 2,     /* valid model, but a shape this build does not implement    */
  MK_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed (see mk_last_error)     */
  MK_ERR_OOM = 4,             /* device workspace allocation failed                        */
  MK_ERR_NO_SCHEDULE = 5,     /* mk_decode_step before a successful mk_build_schedule      */
  MK_ERR_BAD_PAGE = 6,        /* device saw a page id outside [0, num_pages) or past the table */
  MK_ERR_DEVICE_TIMEOUT = 7,  /* a device-side dependency wait exceeded its time limit      */
  MK_ERR_BAD_TOKEN = 8        /* device saw a token id outside [0, vocab)                   */
} mk_status;

/* Model shape. Supported by this build: hidden in {256, 512, 1024, 2048}; head_dim in
 * {64, 128}; n_q_heads / n_kv_heads <= 8 and n_kv_heads divides n_q_heads; n_q_heads *
 * head_dim a multiple of 256 (and of 2048 when above 2048); expert_inter a multiple of 256,
 * at most 2048, with 4 * max_batch * expert_inter <= 32768 (one expert's hi/lo activations
 * for the batch fit a ring stage: any max_batch up to expert_inter 1024, max_batch <= 4 at
 * 2048); top_k <= 8; n_experts <= 256 and a multiple of 8; vocab a multiple of 64;
 * max_batch <= 8; page_size == 16. */
typedef struct {
  int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim;
  int32_t n_experts, top_k, expert_inter, vocab;
  int32_t page_size;          /* tokens per KV page; must be 16                             */
  int32_t max_batch;          /* 1..8                                                       */
  int32_t max_pages_per_seq;  /* columns of the block table; positions < this * page_size  */
  float rope_theta, rms_eps;
} mk_model_cfg;

/* Device pointers, caller-owned, never copied by the library; bf16 (bit pattern of the
 * upper half of an IEEE fp32) unless noted, row-major, stacked over layers:
 *   embed      [vocab][hidden]          norm_gain  [n_layers][hidden]
 *   w_qkv      [n_layers][(n_q + 2 n_kv) head_dim][hidden]   rows: q heads, k heads, v heads
 *   w_o        [n_layers][hidden][n_q head_dim]
 *   w_router   [n_layers][n_experts][hidden]    router_bias fp32 [n_layers][n_experts] or NULL
 *   w_gate_up  [n_layers][n_experts][2 expert_inter][hidden]  rows: gate, then up
 *   w_down     [n_layers][n_experts][hidden][expert_inter]
 *   final_gain [hidden]                 lm_head    [vocab][hidden]
 * Every pointer must be 16-byte aligned. */
typedef struct {
  const void *embed, *norm_gain, *w_qkv, *w_o, *w_router;
  const float* router_bias;
  const void *w_gate_up, *w_down, *final_gain, *lm_head;
} mk_weight_ptrs;

/* Paged KV cache (aimodeling.com "cohere-megakernel-north-mini-code-h100", section "From demo
 * to a full serving system": paged attention over ragged sequence lengths), caller-owned device
 * memory, bf16:
 *   k, v  [n_layers][num_pages][n_kv_heads][page_size][head_dim]
 * Page ids come from the block table given to mk_build_schedule. 16-byte aligned. */
typedef struct {
  void *k, *v;
  int32_t num_pages;
} mk_kv_pages;

typedef struct mk_ctx mk_ctx;

/* Defined by: aimodeling.com "cohere-megakernel-north-mini-code-h100", section "One persistent
 * kernel for the whole decode step" (one kernel resident on every SM for the whole step, over
 * the model's bf16 weights), and "Decode is a bandwidth game" (the weights are streamed once per
 * step, never copied).
 * Validates cfg and the weight pointers (the same check mk_decode_step_noalloc makes), queries
 * the current device (SM count, shared memory), allocates the device workspace (activations,
 * counters, RoPE cos/sin table built on the host in fp64) and returns a context in *out. Weights stay caller-owned and must outlive the context.
 * Errors: MK_ERR_INVALID_ARG, MK_ERR_UNSUPPORTED, MK_ERR_OOM, MK_ERR_CUDA. */
mk_status mk_create(const mk_model_cfg* cfg, const mk_weight_ptrs* weights, mk_ctx** out);

/* Defined by: aibriefing.imbch.dev article 8171681, section "Scheduling and Performance
 * Benchmarks" (a mostly static schedule built on the host, with dynamic work stealing), and
 * aimodeling.com "cohere-megakernel-north-mini-code-h100", section "One persistent kernel for the
 * whole decode step" (a task list in global memory, idle SMs backfilled deterministically); the
 * block tables are the paged KV cache of section "From demo to a full serving system".
 * Host-side scheduler: builds the per-SM task lists and dependency-counter targets for a
 * batch of `batch` sequences whose current lengths are seq_lens[b] (host array) and
 * uploads them (synchronously). block_tables is a device int32 array [batch][max_pages_per_seq]
 * that must stay valid while this schedule is used. Attention work is split in chunks
 * sized from seq_lens; the last chunk of each sequence is open-ended, so the schedule stays
 * valid as sequences grow, until they leave their pages. Resets the device counters.
 * Errors: MK_ERR_INVALID_ARG (batch outside 1..max_batch, negative length, length beyond
 * the table), MK_ERR_OOM, MK_ERR_CUDA. */
mk_status mk_build_schedule(mk_ctx* ctx, int32_t batch, const int32_t* seq_lens, const int32_t* block_tables);

/* Defined by: aimodeling.com "cohere-megakernel-north-mini-code-h100", section "One persistent
 * kernel for the whole decode step" (embedding to LM head in one launch: parallel attention and
 * MoE branches over one normalized input, fused residual + RMSNorm, O-proj released per KV
 * group); RoPE and SiLU-multiply fused per aibriefing.imbch.dev article 8171681, section "Key
 * Technologies and Architecture"; the paged cache of "From demo to a full serving system".
 * One decode step on `stream` (a cudaStream_t, NULL = legacy default stream), a single
 * kernel launch in MK_MODE_MEGAKERNEL. token_ids and positions are device int32 [batch];
 * positions[b] is the new token's position (= its sequence's current length). Writes the
 * bf16 K/V of the new token into kv at (block_tables[b][p / 16], p % 16), fp32 logits to
 * logits_out [batch][vocab] (device, may be NULL) and the greedy next token to argmax_out
 * [batch] (device, may be NULL). Errors: MK_ERR_INVALID_ARG, MK_ERR_NO_SCHEDULE,
 * MK_ERR_CUDA, or a device error latched by an earlier step. */
mk_status mk_decode_step(mk_ctx* ctx, const int32_t* token_ids, const int32_t* positions, const mk_kv_pages* kv,
                         float* logits_out, int32_t* argmax_out, void* stream);

/* Greedy decoding as the pages benchmark it (aibriefing.imbch.dev article 8171681, section
 * "Scheduling and Performance Benchmarks": 1K output tokens per sequence, token fed back).
 * n_steps greedy steps with the token fed back on the device: step i decodes at
 * positions[b] + i the token chosen by step i - 1 (token_ids for i = 0) and writes it to
 * tokens_out [n_steps][batch] (device). logits_out [batch][vocab] (device, may be NULL)
 * receives the last step's logits. One kernel launch per step, no host synchronization. */
mk_status mk_decode_greedy(mk_ctx* ctx, int32_t n_steps, const int32_t* token_ids, const int32_t* positions,
                           const mk_kv_pages* kv, float* logits_out, int32_t* tokens_out, void* stream);

/* Synchronizes the device and returns the latched device status (MK_OK, MK_ERR_BAD_PAGE,
 * MK_ERR_BAD_TOKEN, MK_ERR_DEVICE_TIMEOUT) or MK_ERR_CUDA. Clears it. After
 * MK_ERR_DEVICE_TIMEOUT the counters are reset, so the context stays usable. */
mk_status mk_status_sync(mk_ctx* ctx);

/* Human-readable description of the last error on this context (never NULL). */
const char* mk_last_error(const mk_ctx* ctx);

/* Execution mode: MK_MODE_MEGAKERNEL (default, one persistent kernel per step) or
 * MK_MODE_PER_OP (ablation of aimodeling.com "cohere-megakernel-north-mini-code-h100", section
 * "Decode is a bandwidth game": kernel boundaries between ops. The same opcodes and task lists,
 * one launch of the persistent kernel per layer and opcode kind, so every boundary becomes a
 * full drain of the GPU; it is not a pipeline of separately written small kernels). */
#define MK_MODE_MEGAKERNEL 0
#define MK_MODE_PER_OP 1
mk_status mk_set_mode(mk_ctx* ctx, int mode);

/* Failure detection (no counterpart on the pages): time limit of every device-side wait of a
 * step (a dependency counter, a ring slot, the blocks' own barrier), in nanoseconds; default
 * 2e9 (2 s), accepted range [1e3, 6e10]. A
 * wait that runs out latches MK_ERR_DEVICE_TIMEOUT and every block of the step leaves
 * early, its copies in flight drained (the error is returned by mk_status_sync, which
 * also resets the counters so the context stays usable). Errors: MK_ERR_INVALID_ARG. */
mk_status mk_set_wait_limit(mk_ctx* ctx, int64_t ns);

/* Tracing (no counterpart on the pages): when dev_buf is non-NULL, each step records one
 * 32-byte entry per task (mk_trace_entry) into dev_buf (device memory, caller-owned, `bytes` long; entries past
 * the end are dropped). The first 16 bytes of dev_buf hold the entry count (uint64) and
 * are reset at every step. NULL disables tracing. */
typedef struct {
  uint64_t t_start_ns;   /* %globaltimer when the task was taken           */
  uint32_t wait_ns;      /* time spent waiting for producers               */
  uint32_t run_ns;       /* time from the end of the wait to the release   */
  uint16_t sm, op, layer, pad;
  int32_t a, b;          /* task operands (op-specific)                    */
} mk_trace_entry;
mk_status mk_enable_trace(mk_ctx* ctx, void* dev_buf, size_t bytes);

/* Inspection (no counterpart on the pages): device pointers to the library-owned per-layer
 * activations of the last step (fp32 unless noted; valid until mk_destroy or the next
 * mk_build_schedule):
 *   x [n_layers+1][batch][hidden]  residual stream entering layer l (x[n_layers] final)
 *   q [n_layers][batch][n_q][head_dim] before RoPE (attention applies it when it loads q)
 *   attn [n_layers][batch][n_q][head_dim] attention output per head
 *   attn_out, moe_out [n_layers][batch][hidden]
 *   router [n_layers][batch][n_experts] logits with bias
 *   topk_ids int32 [n_layers][batch][top_k], topk_w [n_layers][batch][top_k]        */
typedef struct {
  const float *x, *q, *attn, *attn_out, *moe_out, *router;
  const int32_t* topk_ids;
  const float* topk_w;
} mk_activations;
mk_status mk_get_activations(const mk_ctx* ctx, mk_activations* out);

/* Host-only view of the scheduler of mk_build_schedule (same passages; no device needed): plans the step for `batch`
 * sequences of lengths seq_lens (host) on n_sm SMs, as mk_build_schedule would. Writes
 * the plan's sizes to *info; if `tasks` is non-NULL, copies the megakernel's task list
 * (info->n_tasks 16-byte descriptors {uint8 op, uint8 flags, uint16 layer, int32 a, b, c},
 * grouped by SM) when tasks_cap >= info->n_tasks, else returns MK_ERR_INVALID_ARG; if
 * sm_begin is non-NULL, writes the n_sm + 1 list offsets; if sm_bytes is non-NULL, the
 * planned bytes per SM. Opcodes: 1 router, 2 QKV, 3 attention, 4 expert gate/up, 5 O-proj,
 * 6 expert down, 7 LM head. At batch 1 (n_sm >= 8), when the attention branch streams at most
 * 1.5x the expert branch's bytes, the two branches of each layer run on disjoint SM partitions:
 * SMs [0, n_attn_sm) take attention and O-proj, the others router, gate/up and down, and QKV
 * spreads over all SMs; otherwise n_attn_sm == n_sm and every SM takes both branches. The LM
 * head spreads over all SMs.
 * Errors: MK_ERR_INVALID_ARG. */
typedef struct {
  int32_t n_tasks, n_counters, max_chunks, n_lm_sm, n_op_launches, n_attn_sm;
} mk_plan_info;
mk_status mk_plan_schedule(const mk_model_cfg* cfg, int32_t n_sm, int32_t batch, const int32_t* seq_lens,
                           mk_plan_info* info, void* tasks, int32_t tasks_cap, int32_t* sm_begin, int64_t* sm_bytes);

/* Number of SMs the persistent kernel runs on and tasks per step of the current schedule. */
mk_status mk_get_launch_info(const mk_ctx* ctx, int32_t* n_sm, int32_t* tasks_per_step, int32_t* launches_per_step);

/* One decode step without allocating device memory. No counterpart on the pages that
 * describe the method: this is a library convenience. For callers that cannot call
 * cudaMalloc (a memory pool or arena that owns every device allocation, a host process
 * that forbids allocation after start-up, code that must not take the allocator's locks or
 * trigger its implicit synchronisation), this runs the same kernel as mk_decode_step with
 * its whole workspace (activations, task lists, counters, RoPE table) placed in one static
 * device array of MK_NOALLOC_SCRATCH_BYTES that every GPU loading the library reserves
 * until the process exits. Nothing else is allocated: weights, KV pages, inputs and outputs
 * come from the caller, with the same meaning and layout as for mk_create, mk_build_schedule
 * and mk_decode_step (positions[b] must equal seq_lens[b], the lengths the step is planned
 * for). The call plans the step on the host, copies the plan into the array, launches on
 * `stream` and waits for that stream, so device errors (bad page, bad token, timeout) are
 * returned directly; the call is synchronous with respect to `stream`. Every device-side
 * wait of this entry point has a fixed limit of 2 s (mk_set_wait_limit, which acts on a
 * context, does not apply here). The first call on a device, with that device current,
 * looks up the array's device address and configures the kernel; make that first call
 * before any stream capture. Every call shares the array and overwrites it (counters and status are cleared
 * at each call), so calls that overlap on the GPU, from any thread or stream, race and must
 * be serialised by the caller. The config and weight pointers get the same checks as in mk_create
 * (MK_ERR_INVALID_ARG or MK_ERR_UNSUPPORTED before any device work), the KV pools must be
 * non-null and 16-byte aligned, and workloads whose workspace exceeds the array (for example
 * the 30B-shaped model) are rejected with MK_ERR_UNSUPPORTED; msg (may be NULL) receives a
 * NUL-terminated explanation of at most msg_len bytes. */
#define MK_NOALLOC_SCRATCH_BYTES (32u << 20)
mk_status mk_decode_step_noalloc(const mk_model_cfg* cfg, const mk_weight_ptrs* weights, int32_t batch,
                                 const int32_t* seq_lens, const int32_t* block_tables, const int32_t* token_ids,
                                 const int32_t* positions, const mk_kv_pages* kv, float* logits_out,
                                 int32_t* argmax_out, void* stream, char* msg, int32_t msg_len);

/* Releases the workspace. Safe on NULL. Does not free caller-owned memory. */
void mk_destroy(mk_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif
