/*
 * Where the oracle reads its inputs. TEST INFRASTRUCTURE ONLY.
 *
 * dense source: host arrays in the decode library's documented layouts (weights stacked
 *   over layers; KV pools [L][num_pages][n_kv][page][d] with a block table [B][max_pages],
 *   or, with no block table, a contiguous cache [L][B][n_kv][max_len][d]).
 * synth source: the same model and prefilled cache produced on demand from the seeded
 *   generator (synth.h), so that a 30B-shaped model is never held in host memory; new
 *   tokens' K/V (positions >= the prefill length) are kept in an overlay.
 */
#include <stdlib.h>
#include <string.h>

#include "../synth/synth.h"
#include "oracle.h"

/* ------------------------------------------------------------------ dense */
typedef struct {
  orc_cfg c;
  const uint16_t *embed, *gain, *final_gain, *qkv, *o, *router, *gate_up, *down, *lm;
  const float* bias;
  uint16_t *kpool, *vpool;
  const int32_t* block_table; /* NULL: contiguous layout */
  int32_t B, max_pages, page, num_pages, max_len;
} dense_src;

static const uint16_t* dense_weight(void* ctx, int kind, int l, int idx) {
  dense_src* s = (dense_src*)ctx;
  const orc_cfg* c = &s->c;
  const size_t H = (size_t)c->H, I = (size_t)c->I, E = (size_t)c->E;
  const size_t qkv_rows = (size_t)(c->nq + 2 * c->nkv) * c->d, od = (size_t)c->nq * c->d;
  switch (kind) {
    case ORC_EMBED: return (idx >= 0 && idx < c->V) ? s->embed + (size_t)idx * H : NULL;
    case ORC_GAIN: return s->gain + (size_t)l * H;
    case ORC_FINAL_GAIN: return s->final_gain;
    case ORC_QKV: return s->qkv + (size_t)l * qkv_rows * H;
    case ORC_O: return s->o + (size_t)l * H * od;
    case ORC_ROUTER: return s->router + (size_t)l * E * H;
    case ORC_GATE_UP: return s->gate_up + ((size_t)l * E + idx) * 2 * I * H;
    case ORC_DOWN: return s->down + ((size_t)l * E + idx) * H * I;
    case ORC_LM: return s->lm;
  }
  return NULL;
}
static const float* dense_bias(void* ctx, int l) {
  dense_src* s = (dense_src*)ctx;
  return s->bias ? s->bias + (size_t)l * s->c.E : NULL;
}
static uint16_t* dense_slot(dense_src* s, int kind, int l, int b, int pos, int g) {
  const orc_cfg* c = &s->c;
  uint16_t* pool = kind ? s->vpool : s->kpool;
  if (b < 0 || b >= s->B || pos < 0 || g < 0 || g >= c->nkv) return NULL;
  if (!s->block_table) {
    if (pos >= s->max_len) return NULL;
    return pool + ((((size_t)l * s->B + b) * c->nkv + g) * s->max_len + pos) * c->d;
  }
  const int pi = pos / s->page;
  if (pi >= s->max_pages) return NULL;
  const int pg = s->block_table[(size_t)b * s->max_pages + pi];
  if (pg < 0 || pg >= s->num_pages) return NULL;
  return pool + ((((size_t)l * s->num_pages + pg) * c->nkv + g) * s->page + pos % s->page) * c->d;
}
static int dense_kv_read(void* ctx, int kind, int l, int b, int pos, int g, uint16_t* dst) {
  dense_src* s = (dense_src*)ctx;
  uint16_t* p = dense_slot(s, kind, l, b, pos, g);
  if (!p) return 1;
  memcpy(dst, p, sizeof(uint16_t) * (size_t)s->c.d);
  return 0;
}
static int dense_kv_write(void* ctx, int kind, int l, int b, int pos, int g, const uint16_t* src) {
  dense_src* s = (dense_src*)ctx;
  uint16_t* p = dense_slot(s, kind, l, b, pos, g);
  if (!p) return 1;
  memcpy(p, src, sizeof(uint16_t) * (size_t)s->c.d);
  return 0;
}

/* Creates a dense source; all arrays stay owned by the caller. */
void* orc_dense_source_create(const orc_cfg* c, const uint16_t* embed, const uint16_t* gain,
                              const uint16_t* final_gain, const uint16_t* qkv, const uint16_t* o,
                              const uint16_t* router, const float* bias, const uint16_t* gate_up,
                              const uint16_t* down, const uint16_t* lm, uint16_t* kpool, uint16_t* vpool,
                              const int32_t* block_table, int32_t B, int32_t max_pages, int32_t page,
                              int32_t num_pages, int32_t max_len, orc_source* out) {
  dense_src* s = (dense_src*)calloc(1, sizeof(dense_src));
  s->c = *c;
  s->embed = embed; s->gain = gain; s->final_gain = final_gain; s->qkv = qkv; s->o = o; s->router = router;
  s->bias = bias; s->gate_up = gate_up; s->down = down; s->lm = lm; s->kpool = kpool; s->vpool = vpool;
  s->block_table = block_table; s->B = B; s->max_pages = max_pages; s->page = page; s->num_pages = num_pages;
  s->max_len = max_len;
  out->ctx = s;
  out->weight = dense_weight;
  out->router_bias = dense_bias;
  out->kv_read = dense_kv_read;
  out->kv_write = dense_kv_write;
  return s;
}
void orc_dense_source_destroy(void* s) { free(s); }

/* ------------------------------------------------------------------ synth */
typedef struct {
  int kind, layer, index;
  uint16_t* data;
  size_t n;
} cache_ent;

typedef struct {
  orc_cfg c;
  uint64_t seed;
  int32_t B, max_new;
  int32_t* ctx_len;   /* prefill length per sequence */
  float* bias;        /* [L][E] or NULL */
  uint16_t* overlay;  /* [2][L][B][nkv][max_new][d] */
  uint16_t *embed_row, *gain, *final_gain, *qkv, *o, *router, *lm;
  int qkv_l, o_l, router_l, gain_l;
  uint16_t **qkv_all, **o_all, **router_all; /* keep_all: every layer's dense weights */
  cache_ent* experts; /* (kind, layer, expert) cache */
  int n_exp, cap_exp;
  int keep_all;       /* 0: drop cached experts of other layers */
} synth_src;

static void gen(synth_src* s, int skind, int layer, int sub, size_t count, float sigma, float offset,
                uint16_t* dst) {
  synth_fill_bf16(s->seed, synth_tid(skind, layer, sub), 0, count, sigma, offset, dst);
}

static const uint16_t* cached_dense(synth_src* s, uint16_t** tab, int skind, int l, size_t n) {
  if (!tab[l]) {
    tab[l] = (uint16_t*)malloc(sizeof(uint16_t) * n);
    gen(s, skind, l, 0, n, 0.02f, 0.0f, tab[l]);
  }
  return tab[l];
}

static const uint16_t* synth_weight(void* ctx, int kind, int l, int idx) {
  synth_src* s = (synth_src*)ctx;
  const orc_cfg* c = &s->c;
  const size_t H = (size_t)c->H, I = (size_t)c->I;
  const size_t qkv_rows = (size_t)(c->nq + 2 * c->nkv) * c->d, od = (size_t)c->nq * c->d;
  switch (kind) {
    case ORC_EMBED:
      if (idx < 0 || idx >= c->V) return NULL;
      synth_fill_bf16(s->seed, synth_tid(SYNTH_EMBED, 0, 0), (uint64_t)idx * H, H, 0.02f, 0.0f, s->embed_row);
      return s->embed_row;
    case ORC_GAIN:
      if (s->gain_l != l) { gen(s, SYNTH_GAIN, l, 0, H, 0.05f, 1.0f, s->gain); s->gain_l = l; }
      return s->gain;
    case ORC_FINAL_GAIN: return s->final_gain;
    case ORC_QKV:
      if (s->keep_all) return cached_dense(s, s->qkv_all, SYNTH_QKV, l, qkv_rows * H);
      if (s->qkv_l != l) { gen(s, SYNTH_QKV, l, 0, qkv_rows * H, 0.02f, 0.0f, s->qkv); s->qkv_l = l; }
      return s->qkv;
    case ORC_O:
      if (s->keep_all) return cached_dense(s, s->o_all, SYNTH_O, l, H * od);
      if (s->o_l != l) { gen(s, SYNTH_O, l, 0, H * od, 0.02f, 0.0f, s->o); s->o_l = l; }
      return s->o;
    case ORC_ROUTER:
      if (s->keep_all) return cached_dense(s, s->router_all, SYNTH_ROUTER, l, (size_t)c->E * H);
      if (s->router_l != l) { gen(s, SYNTH_ROUTER, l, 0, (size_t)c->E * H, 0.02f, 0.0f, s->router); s->router_l = l; }
      return s->router;
    case ORC_LM:
      if (!s->lm) {
        s->lm = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)c->V * H);
        gen(s, SYNTH_LM, 0, 0, (size_t)c->V * H, 0.02f, 0.0f, s->lm);
      }
      return s->lm;
    case ORC_GATE_UP:
    case ORC_DOWN: {
      if (idx < 0 || idx >= c->E) return NULL;
      for (int i = 0; i < s->n_exp; ++i)
        if (s->experts[i].kind == kind && s->experts[i].layer == l && s->experts[i].index == idx)
          return s->experts[i].data;
      if (!s->keep_all) { /* forget other layers' experts */
        int w = 0;
        for (int i = 0; i < s->n_exp; ++i) {
          if (s->experts[i].layer == l) s->experts[w++] = s->experts[i];
          else free(s->experts[i].data);
        }
        s->n_exp = w;
      }
      if (s->n_exp == s->cap_exp) {
        s->cap_exp = s->cap_exp ? 2 * s->cap_exp : 64;
        s->experts = (cache_ent*)realloc(s->experts, sizeof(cache_ent) * (size_t)s->cap_exp);
      }
      cache_ent* e = &s->experts[s->n_exp++];
      e->kind = kind; e->layer = l; e->index = idx; e->n = (kind == ORC_GATE_UP ? 2 : 1) * I * H;
      e->data = (uint16_t*)malloc(sizeof(uint16_t) * e->n);
      gen(s, kind == ORC_GATE_UP ? SYNTH_GATE_UP : SYNTH_DOWN, l, idx, e->n, 0.02f, 0.0f, e->data);
      return e->data;
    }
  }
  return NULL;
}
static const float* synth_bias(void* ctx, int l) {
  synth_src* s = (synth_src*)ctx;
  return s->bias ? s->bias + (size_t)l * s->c.E : NULL;
}
static uint16_t* overlay_slot(synth_src* s, int kind, int l, int b, int pos, int g) {
  const int k = pos - s->ctx_len[b];
  if (k < 0 || k >= s->max_new) return NULL;
  const orc_cfg* c = &s->c;
  return s->overlay + (((((size_t)kind * c->L + l) * s->B + b) * c->nkv + g) * s->max_new + k) * c->d;
}
static int synth_kv_read(void* ctx, int kind, int l, int b, int pos, int g, uint16_t* dst) {
  synth_src* s = (synth_src*)ctx;
  const orc_cfg* c = &s->c;
  if (b < 0 || b >= s->B || pos < 0 || g < 0 || g >= c->nkv) return 1;
  if (pos < s->ctx_len[b]) {
    synth_fill_bf16(s->seed, synth_tid(kind ? SYNTH_V : SYNTH_K, l, b * c->nkv + g), (uint64_t)pos * c->d,
                    (uint64_t)c->d, 1.0f, 0.0f, dst);
    return 0;
  }
  uint16_t* p = overlay_slot(s, kind, l, b, pos, g);
  if (!p) return 1;
  memcpy(dst, p, sizeof(uint16_t) * (size_t)c->d);
  return 0;
}
static int synth_kv_write(void* ctx, int kind, int l, int b, int pos, int g, const uint16_t* src) {
  synth_src* s = (synth_src*)ctx;
  if (b < 0 || b >= s->B || g < 0 || g >= s->c.nkv) return 1;
  uint16_t* p = overlay_slot(s, kind, l, b, pos, g);
  if (!p) return 1;
  memcpy(p, src, sizeof(uint16_t) * (size_t)s->c.d);
  return 0;
}

/* Creates a synth source for B sequences prefilled to ctx_len[b] positions with room
 * for max_new appended tokens each. bias ([L][E] fp32) is copied; NULL = zero bias.
 * keep_all != 0 keeps every generated weight (dense per-layer weights and experts) so that
 * a repeated step times the oracle's arithmetic rather than the generator. */
void* orc_synth_source_create(const orc_cfg* c, uint64_t seed, int32_t B, const int32_t* ctx_len,
                              int32_t max_new, const float* bias, int32_t keep_all_experts, orc_source* out) {
  synth_src* s = (synth_src*)calloc(1, sizeof(synth_src));
  const size_t H = (size_t)c->H;
  s->c = *c;
  s->seed = seed;
  s->B = B;
  s->max_new = max_new;
  s->keep_all = keep_all_experts;
  s->ctx_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)B);
  memcpy(s->ctx_len, ctx_len, sizeof(int32_t) * (size_t)B);
  if (bias) {
    s->bias = (float*)malloc(sizeof(float) * (size_t)c->L * c->E);
    memcpy(s->bias, bias, sizeof(float) * (size_t)c->L * c->E);
  }
  s->overlay = (uint16_t*)calloc((size_t)2 * c->L * B * c->nkv * (size_t)max_new * c->d, sizeof(uint16_t));
  s->embed_row = (uint16_t*)malloc(sizeof(uint16_t) * H);
  s->gain = (uint16_t*)malloc(sizeof(uint16_t) * H);
  s->final_gain = (uint16_t*)malloc(sizeof(uint16_t) * H);
  synth_fill_bf16(seed, synth_tid(SYNTH_FINAL_GAIN, 0, 0), 0, H, 0.05f, 1.0f, s->final_gain);
  s->qkv = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(c->nq + 2 * c->nkv) * c->d * H);
  s->o = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)c->nq * c->d * H);
  s->router = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)c->E * H);
  s->qkv_l = s->o_l = s->router_l = s->gain_l = -1;
  s->qkv_all = (uint16_t**)calloc((size_t)c->L, sizeof(uint16_t*));
  s->o_all = (uint16_t**)calloc((size_t)c->L, sizeof(uint16_t*));
  s->router_all = (uint16_t**)calloc((size_t)c->L, sizeof(uint16_t*));
  out->ctx = s;
  out->weight = synth_weight;
  out->router_bias = synth_bias;
  out->kv_read = synth_kv_read;
  out->kv_write = synth_kv_write;
  return s;
}
void orc_synth_source_destroy(void* p) {
  synth_src* s = (synth_src*)p;
  if (!s) return;
  for (int i = 0; i < s->n_exp; ++i) free(s->experts[i].data);
  for (int l = 0; l < s->c.L; ++l) { free(s->qkv_all[l]); free(s->o_all[l]); free(s->router_all[l]); }
  free(s->qkv_all); free(s->o_all); free(s->router_all);
  free(s->experts); free(s->ctx_len); free(s->bias); free(s->overlay); free(s->embed_row); free(s->gain);
  free(s->final_gain); free(s->qkv); free(s->o); free(s->router); free(s->lm);
  free(s);
}
