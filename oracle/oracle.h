/*
 * CPU oracle for one autoregressive decode step of a parallel-layer MoE transformer.
 *
 * TEST INFRASTRUCTURE ONLY. Tests, the smoke check and the benchmark's CPU-baseline
 * leg call this code; the decode library never does, and this code shares nothing with it.
 *
 * What it computes (Cohere megakernel news pages: aimodeling.com "cohere-megakernel-north-
 * mini-code-h100", section "One persistent kernel for the whole decode step" (parallel
 * layers: attention and MoE read the same normalized input and are rejoined by a fused
 * residual add + RMSNorm; O-proj per KV group), section "From demo to a full serving
 * system" (paged attention, ragged lengths); aibriefing.imbch.dev article 8171681,
 * "Key Technologies and Architecture" (fused RoPE and SiLU-multiply); BF16 weights and
 * KV on all three pages). The pages give no dims, norm epsilon, RoPE layout or router
 * rule. Readings taken where they are silent: one RMSNorm per layer shared by both branches,
 * gain after normalization, eps from the config; residual x + attn + moe with no scaling;
 * rotate-half RoPE over the full head (pairs i, i + d/2; angle pos * theta^(-2i/d)) on q and
 * k only; contiguous GQA groups; scale 1/sqrt(d), no soft-cap or window; router bias added
 * before top-k and softmax, softmax over the k selected, ties to the lower id; routing
 * weight applied to the expert's down output, summed in rank order; untied LM head, argmax
 * ties to the lowest id; the new token's k and v rounded to bf16 before attention reads
 * them. Each reading is repeated at the function that takes it.
 *
 * Arithmetic: weights and the KV cache are bf16 (as stored); every other value is
 * carried in fp64. Decisions that produce integers (router top-k, LM-head argmax) are
 * taken on the fp32-rounded values, the precision the GPU path decides in.
 *
 * Parity status: every function below is pinned by closed forms, invariants or
 * library routines in tests/test_oracle_pins.py except the whole 30B-shaped step,
 * whose logits have no printed worked example (parity unpinned beyond the parts).
 */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t L, H, nq, nkv, d, E, topk, I, V;
  double rope_theta, eps;
} orc_cfg;

enum orc_kind {
  ORC_EMBED = 1,      /* row `index` of [V][H]          */
  ORC_GAIN = 2,       /* [H] input gain of layer        */
  ORC_FINAL_GAIN = 3, /* [H]                            */
  ORC_QKV = 4,        /* [(nq+2nkv)d][H] of layer       */
  ORC_O = 5,          /* [H][nq d]                      */
  ORC_ROUTER = 6,     /* [E][H]                         */
  ORC_GATE_UP = 7,    /* [2I][H] of expert `index`      */
  ORC_DOWN = 8,       /* [H][I] of expert `index`       */
  ORC_LM = 9          /* [V][H]                         */
};

/* Where the oracle reads weights and keeps its KV cache. weight() returns bf16 bits that
 * stay valid until the next weight() call of the same kind; kv_read/kv_write copy d
 * values of head group g at logical position pos of sequence b (thread-safe). */
typedef struct {
  void* ctx;
  const uint16_t* (*weight)(void* ctx, int kind, int layer, int index);
  const float* (*router_bias)(void* ctx, int layer); /* fp32 [E] or NULL (zero bias) */
  int (*kv_read)(void* ctx, int kind /*0 K, 1 V*/, int layer, int b, int pos, int g, uint16_t* dst);
  int (*kv_write)(void* ctx, int kind, int layer, int b, int pos, int g, const uint16_t* src);
} orc_source;

/* Optional per-layer record of intermediate values (any pointer may be NULL). */
typedef struct {
  float* x;          /* [L+1][B][H] residual stream entering layer l (x[L] = final)      */
  float* q;          /* [L][B][nq][d] after RoPE                                           */
  uint16_t* k_new;   /* [L][B][nkv][d] appended key (bf16)                                 */
  uint16_t* v_new;   /* [L][B][nkv][d]                                                     */
  float* attn;       /* [L][B][nq][d] attention output per head                            */
  float* attn_out;   /* [L][B][H] O-projection output                                      */
  float* router;     /* [L][B][E] router logits (bias included)                            */
  int32_t* topk_ids; /* [L][B][topk]                                                       */
  float* topk_w;     /* [L][B][topk]                                                       */
  float* moe_out;    /* [L][B][H]                                                          */
} orc_trace;

/* Status codes */
#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_SOURCE 2

/* One decode step for B sequences: token_ids[b] at position positions[b] (= tokens
 * already cached). Appends each layer's k,v (bf16) through kv_write, writes fp32 logits
 * [B][V] and the greedy next token [B] (lowest index on ties). */
/* Host threads the oracle's parallel loops use. */
int orc_threads(void);

int orc_decode_step(const orc_cfg* cfg, const orc_source* src, int B, const int32_t* token_ids,
                    const int32_t* positions, float* logits, int32_t* next_token, orc_trace* trace);

/* ---- the step's parts, exported so that tests can pin each one ---- */
double orc_bf16_to_double(uint16_t h);
uint16_t orc_double_to_bf16(double v);
/* y = W x for W bf16 [rows][cols] row-major */
void orc_matvec(const uint16_t* W, int rows, int cols, const double* x, double* y);
/* out = x / sqrt(mean(x^2) + eps) * gain */
void orc_rmsnorm(const double* x, const uint16_t* gain, int n, double eps, double* out);
/* rotate-half RoPE of one head vector (d even) at position pos, in place */
void orc_rope(double* v, int d, int pos, double theta);
/* one query head over keys/values [n][d] (bf16): out = softmax(q K^T / sqrt(d)) V */
void orc_attention_head(const double* q, const uint16_t* K, const uint16_t* V, int n, int d, double* out);
/* top-k of logits rounded to fp32 (the GPU decides in fp32), descending, lower index
 * first on equal values; w = softmax over the k selected fp64 logits */
void orc_route(const double* logits, int E, int k, int32_t* ids, double* w);
/* one SwiGLU expert: y = Wd (silu(Wg x) * (Wu x)); Wgu = [gate rows; up rows] [2I][H], Wd [H][I] */
void orc_expert(const uint16_t* Wgu, const uint16_t* Wd, int H, int I, const double* x, double* y);
/* expert weights by id: which 0 -> Wgu [2I][H], 1 -> Wd [H][I] */
typedef const uint16_t* (*orc_expert_fetch)(void* ctx, int expert, int which);
/* router + top-k + weighted experts for one token: y = sum_j w_j expert_{ids_j}(x), j in rank order */
void orc_moe(const double* x, const uint16_t* Wr, const float* bias, int H, int I, int E, int k,
             orc_expert_fetch fetch, void* fetch_ctx, double* y, double* logits_out, int32_t* ids_out,
             double* w_out);

#ifdef __cplusplus
}
#endif
#endif
