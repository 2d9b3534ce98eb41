/*
 * CPU oracle: one decode step of a parallel-layer MoE transformer, written out plainly.
 * TEST INFRASTRUCTURE ONLY (see oracle.h): only the tests, the smoke check and the
 * benchmark's CPU-baseline leg run it.
 *
 * Sources: aimodeling.com "cohere-megakernel-north-mini-code-h100", section "One
 * persistent kernel for the whole decode step" (the parallel layer: attention and MoE
 * read one normalized input; a fused residual add + RMSNorm rejoins them; O-proj per KV
 * group) and section "From demo to a full serving system" (paged attention, ragged
 * lengths); aibriefing.imbch.dev article 8171681, section "Key Technologies and
 * Architecture" (RoPE and SiLU-multiply are part of the step). Where the pages are
 * silent the plainest reading is taken and named at the function.
 */
#include "oracle.h"

#include <math.h>
#include <omp.h>
#include <stdlib.h>
#include <string.h>

double orc_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round to the nearest bf16 (ties to even) directly from fp64. */
uint16_t orc_double_to_bf16(double v) {
  if (v != v) return 0x7FC0;
  uint64_t u;
  memcpy(&u, &v, 8);
  const uint16_t sign = (uint16_t)((u >> 63) << 15);
  const double a = fabs(v);
  if (a == 0.0) return sign;
  if (a >= 0x1p128) return sign | 0x7F80;
  if (a >= 0x1p-126) {
    u += ((uint64_t)1 << 44) - 1 + ((u >> 45) & 1);
    const int e = (int)((u >> 52) & 0x7FF) - 1023;
    if (e > 127) return sign | 0x7F80;
    return sign | (uint16_t)((e + 127) << 7) | (uint16_t)((u >> 45) & 0x7F);
  }
  /* bf16 subnormal: multiples of 2^-133, rounded half to even */
  double q = nearbyint(a * 0x1p133);
  return sign | (uint16_t)q;
}

/* y = W x, W row-major bf16 [rows][cols]. */
void orc_matvec(const uint16_t* W, int rows, int cols, const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    const uint16_t* w = W + (size_t)r * cols;
    double acc = 0.0;
    for (int c = 0; c < cols; ++c) acc += orc_bf16_to_double(w[c]) * x[c];
    y[r] = acc;
  }
}

/* RMSNorm with the gain applied after normalization. eps is not given by the pages;
 * 1e-6 is the configured default. */
void orc_rmsnorm(const double* x, const uint16_t* gain, int n, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  const double r = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * r * orc_bf16_to_double(gain[i]);
}

/* Rotary position embedding, rotate-half layout: element i pairs with i + d/2 and turns
 * by pos * theta^(-2i/d). The pages name RoPE without a layout; this is the plainest
 * full-head reading. */
void orc_rope(double* v, int d, int pos, double theta) {
  const int h = d / 2;
  for (int i = 0; i < h; ++i) {
    const double ang = (double)pos * pow(theta, -2.0 * i / d);
    const double c = cos(ang), s = sin(ang);
    const double a = v[i], b = v[i + h];
    v[i] = a * c - b * s;
    v[i + h] = a * s + b * c;
  }
}

/* softmax(q K^T / sqrt(d)) V for one query head over n cached positions. */
void orc_attention_head(const double* q, const uint16_t* K, const uint16_t* V, int n, int d, double* out) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  const double scale = 1.0 / sqrt((double)d);
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += q[i] * orc_bf16_to_double(K[(size_t)j * d + i]);
    s[j] = acc * scale;
    if (s[j] > m) m = s[j];
  }
  double z = 0.0;
  for (int j = 0; j < n; ++j) {
    s[j] = exp(s[j] - m);
    z += s[j];
  }
  for (int i = 0; i < d; ++i) out[i] = 0.0;
  for (int j = 0; j < n; ++j)
    for (int i = 0; i < d; ++i) out[i] += s[j] * orc_bf16_to_double(V[(size_t)j * d + i]);
  for (int i = 0; i < d; ++i) out[i] /= z;
  free(s);
}

/* Router decision: the k largest logits (compared as fp32, lower expert id first on
 * equal values), then a softmax over the k selected logits. Bias, if any, is already in
 * the logits, so it shapes both the selection and the weights. */
void orc_route(const double* logits, int E, int k, int32_t* ids, double* w) {
  char* taken = (char*)calloc((size_t)E, 1);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    float bv = 0.0f;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      const float v = (float)logits[e];
      if (best < 0 || v > bv) {
        best = e;
        bv = v;
      }
    }
    taken[best] = 1;
    ids[j] = best;
  }
  double m = logits[ids[0]];
  for (int j = 1; j < k; ++j)
    if (logits[ids[j]] > m) m = logits[ids[j]];
  double z = 0.0;
  for (int j = 0; j < k; ++j) {
    w[j] = exp(logits[ids[j]] - m);
    z += w[j];
  }
  for (int j = 0; j < k; ++j) w[j] /= z;
  free(taken);
}

/* SwiGLU expert with SiLU(a) = a / (1 + e^-a) applied to the gate projection. */
void orc_expert(const uint16_t* Wgu, const uint16_t* Wd, int H, int I, const double* x, double* y) {
  double* gu = (double*)malloc(sizeof(double) * 2 * (size_t)I);
  orc_matvec(Wgu, 2 * I, H, x, gu);
  for (int i = 0; i < I; ++i) {
    const double g = gu[i];
    gu[i] = g / (1.0 + exp(-g)) * gu[I + i];
  }
  orc_matvec(Wd, H, I, gu, y);
  free(gu);
}

void orc_moe(const double* x, const uint16_t* Wr, const float* bias, int H, int I, int E, int k,
             orc_expert_fetch fetch, void* fetch_ctx, double* y, double* logits_out, int32_t* ids_out,
             double* w_out) {
  double* r = (double*)malloc(sizeof(double) * (size_t)E);
  double* ye = (double*)malloc(sizeof(double) * (size_t)H);
  orc_matvec(Wr, E, H, x, r);
  if (bias)
    for (int e = 0; e < E; ++e) r[e] += (double)bias[e];
  orc_route(r, E, k, ids_out, w_out);
  for (int i = 0; i < H; ++i) y[i] = 0.0;
  for (int j = 0; j < k; ++j) {
    const uint16_t* wgu = fetch(fetch_ctx, ids_out[j], 0);
    const uint16_t* wd = fetch(fetch_ctx, ids_out[j], 1);
    orc_expert(wgu, wd, H, I, x, ye);
    for (int i = 0; i < H; ++i) y[i] += w_out[j] * ye[i];
  }
  if (logits_out) memcpy(logits_out, r, sizeof(double) * (size_t)E);
  free(r);
  free(ye);
}

typedef struct {
  const orc_source* src;
  int layer;
} fetch_ctx_t;

static const uint16_t* fetch_expert(void* ctx, int expert, int which) {
  fetch_ctx_t* f = (fetch_ctx_t*)ctx;
  return f->src->weight(f->src->ctx, which ? ORC_DOWN : ORC_GATE_UP, f->layer, expert);
}

#define TR(ptr, idx) ((ptr) ? &(ptr)[idx] : NULL)

int orc_decode_step(const orc_cfg* c, const orc_source* src, int B, const int32_t* token_ids,
                    const int32_t* positions, float* logits, int32_t* next_token, orc_trace* tr) {
  if (!c || !src || B <= 0 || !token_ids || !positions) return ORC_ERR_ARG;
  if (c->nq % c->nkv || c->d % 2 || c->topk > c->E) return ORC_ERR_ARG;
  const int L = c->L, H = c->H, nq = c->nq, nkv = c->nkv, d = c->d, E = c->E, K = c->topk, I = c->I;
  const int V = c->V, qkv_rows = (nq + 2 * nkv) * d, group = nq / nkv;
  for (int b = 0; b < B; ++b)
    if (token_ids[b] < 0 || token_ids[b] >= V || positions[b] < 0) return ORC_ERR_ARG;

  double* x = (double*)calloc((size_t)B * H, sizeof(double));
  double* n = (double*)calloc((size_t)B * H, sizeof(double));
  double* qkv = (double*)calloc((size_t)B * qkv_rows, sizeof(double));
  double* o = (double*)calloc((size_t)B * nq * d, sizeof(double));
  double* attn = (double*)calloc((size_t)B * H, sizeof(double));
  double* moe = (double*)calloc((size_t)B * H, sizeof(double));
  double* rl = (double*)calloc((size_t)E, sizeof(double));
  double* wk = (double*)calloc((size_t)K, sizeof(double));
  int32_t* ids = (int32_t*)calloc((size_t)K, sizeof(int32_t));
  uint16_t* kb = (uint16_t*)calloc((size_t)d, sizeof(uint16_t));
  uint16_t* vb = (uint16_t*)calloc((size_t)d, sizeof(uint16_t));
  int status = ORC_OK;

  /* token embedding, then the layer-0 input norm */
  for (int b = 0; b < B; ++b) {
    const uint16_t* row = src->weight(src->ctx, ORC_EMBED, 0, token_ids[b]);
    if (!row) { status = ORC_ERR_SOURCE; goto done; }
    for (int i = 0; i < H; ++i) x[(size_t)b * H + i] = orc_bf16_to_double(row[i]);
  }
  {
    const uint16_t* g0 = src->weight(src->ctx, ORC_GAIN, 0, 0);
    if (!g0) { status = ORC_ERR_SOURCE; goto done; }
    for (int b = 0; b < B; ++b) orc_rmsnorm(&x[(size_t)b * H], g0, H, c->eps, &n[(size_t)b * H]);
  }

  for (int l = 0; l < L; ++l) {
    if (tr && tr->x)
      for (size_t i = 0; i < (size_t)B * H; ++i) tr->x[(size_t)l * B * H + i] = (float)x[i];

    /* attention branch: QKV projection, RoPE on q and k, append bf16 k and v */
    const uint16_t* Wqkv = src->weight(src->ctx, ORC_QKV, l, 0);
    if (!Wqkv) { status = ORC_ERR_SOURCE; goto done; }
    for (int b = 0; b < B; ++b) {
      double* r = &qkv[(size_t)b * qkv_rows];
      orc_matvec(Wqkv, qkv_rows, H, &n[(size_t)b * H], r);
      for (int h = 0; h < nq + nkv; ++h) orc_rope(&r[(size_t)h * d], d, positions[b], c->rope_theta);
      for (int g = 0; g < nkv; ++g) {
        for (int i = 0; i < d; ++i) {
          kb[i] = orc_double_to_bf16(r[(size_t)(nq + g) * d + i]);
          vb[i] = orc_double_to_bf16(r[(size_t)(nq + nkv + g) * d + i]);
        }
        if (src->kv_write(src->ctx, 0, l, b, positions[b], g, kb) ||
            src->kv_write(src->ctx, 1, l, b, positions[b], g, vb)) {
          status = ORC_ERR_SOURCE;
          goto done;
        }
        if (tr && tr->k_new) memcpy(&tr->k_new[(((size_t)l * B + b) * nkv + g) * d], kb, 2 * (size_t)d);
        if (tr && tr->v_new) memcpy(&tr->v_new[(((size_t)l * B + b) * nkv + g) * d], vb, 2 * (size_t)d);
      }
      if (tr && tr->q)
        for (int i = 0; i < nq * d; ++i) tr->q[((size_t)l * B + b) * nq * d + i] = (float)r[i];
    }

    /* paged GQA attention over positions 0..pos (the new token included, read back from
     * the cache): q head h reads KV group h / (nq / nkv) */
    for (int b = 0; b < B; ++b) {
      const int cnt = positions[b] + 1;
      uint16_t* Kc = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)cnt * d);
      uint16_t* Vc = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)cnt * d);
      for (int g = 0; g < nkv && status == ORC_OK; ++g) {
        int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
        for (int j = 0; j < cnt; ++j) {
          bad |= src->kv_read(src->ctx, 0, l, b, j, g, &Kc[(size_t)j * d]) != 0;
          bad |= src->kv_read(src->ctx, 1, l, b, j, g, &Vc[(size_t)j * d]) != 0;
        }
        if (bad) { status = ORC_ERR_SOURCE; break; }
#pragma omp parallel for schedule(static)
        for (int hh = 0; hh < group; ++hh) {
          const int h = g * group + hh;
          orc_attention_head(&qkv[(size_t)b * qkv_rows + (size_t)h * d], Kc, Vc, cnt, d,
                             &o[((size_t)b * nq + h) * d]);
        }
      }
      free(Kc);
      free(Vc);
      if (status != ORC_OK) goto done;
      if (tr && tr->attn)
        for (int i = 0; i < nq * d; ++i) tr->attn[((size_t)l * B + b) * nq * d + i] = (float)o[(size_t)b * nq * d + i];
    }
    const uint16_t* Wo = src->weight(src->ctx, ORC_O, l, 0);
    if (!Wo) { status = ORC_ERR_SOURCE; goto done; }
    for (int b = 0; b < B; ++b) orc_matvec(Wo, H, nq * d, &o[(size_t)b * nq * d], &attn[(size_t)b * H]);

    /* MoE branch on the same normalized input */
    const uint16_t* Wr = src->weight(src->ctx, ORC_ROUTER, l, 0);
    if (!Wr) { status = ORC_ERR_SOURCE; goto done; }
    const float* bias = src->router_bias ? src->router_bias(src->ctx, l) : NULL;
    fetch_ctx_t fc = {src, l};
    for (int b = 0; b < B; ++b) {
      orc_moe(&n[(size_t)b * H], Wr, bias, H, I, E, K, fetch_expert, &fc, &moe[(size_t)b * H], rl, ids, wk);
      if (tr && tr->router)
        for (int e = 0; e < E; ++e) tr->router[((size_t)l * B + b) * E + e] = (float)rl[e];
      if (tr && tr->topk_ids) memcpy(&tr->topk_ids[((size_t)l * B + b) * K], ids, sizeof(int32_t) * K);
      if (tr && tr->topk_w)
        for (int j = 0; j < K; ++j) tr->topk_w[((size_t)l * B + b) * K + j] = (float)wk[j];
    }

    /* rejoin: residual add of both branches, then the next input norm */
    const uint16_t* gn = (l + 1 < L) ? src->weight(src->ctx, ORC_GAIN, l + 1, 0)
                                     : src->weight(src->ctx, ORC_FINAL_GAIN, 0, 0);
    if (!gn) { status = ORC_ERR_SOURCE; goto done; }
    for (int b = 0; b < B; ++b) {
      for (int i = 0; i < H; ++i) x[(size_t)b * H + i] += attn[(size_t)b * H + i] + moe[(size_t)b * H + i];
      orc_rmsnorm(&x[(size_t)b * H], gn, H, c->eps, &n[(size_t)b * H]);
      if (tr && tr->attn_out)
        for (int i = 0; i < H; ++i) tr->attn_out[((size_t)l * B + b) * H + i] = (float)attn[(size_t)b * H + i];
      if (tr && tr->moe_out)
        for (int i = 0; i < H; ++i) tr->moe_out[((size_t)l * B + b) * H + i] = (float)moe[(size_t)b * H + i];
    }
  }
  if (tr && tr->x)
    for (size_t i = 0; i < (size_t)B * H; ++i) tr->x[(size_t)L * B * H + i] = (float)x[i];

  /* LM head (untied from the embedding) and greedy argmax on the fp32 logits */
  {
    const uint16_t* Wlm = src->weight(src->ctx, ORC_LM, 0, 0);
    if (!Wlm) { status = ORC_ERR_SOURCE; goto done; }
    double* lg = (double*)malloc(sizeof(double) * (size_t)V);
    for (int b = 0; b < B; ++b) {
      orc_matvec(Wlm, V, H, &n[(size_t)b * H], lg);
      int best = 0;
      float bv = (float)lg[0];
      for (int v = 0; v < V; ++v) {
        const float f = (float)lg[v];
        if (logits) logits[(size_t)b * V + v] = f;
        if (f > bv) {
          bv = f;
          best = v;
        }
      }
      if (next_token) next_token[b] = best;
    }
    free(lg);
  }

done:
  free(x); free(n); free(qkv); free(o); free(attn); free(moe); free(rl); free(wk); free(ids); free(kb); free(vb);
  return status;
}

/* Host threads the oracle's parallel loops use (reported next to its timings). */
int orc_threads(void) { return omp_get_max_threads(); }
