/*
 * Seeded synthetic inputs for the decode step: weights, gains, KV pages, token ids.
 *
 * This module only makes numbers. It holds none of the decode step's arithmetic and
 * is shared by the host-side checker and the GPU-side benchmark/tests, which both
 * need the same model and KV cache without storing 60+ GB of it anywhere.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used counter-style: draw n of stream `key` is
 * mix(key + (n+1)*GOLDEN), with mix() the published SplitMix64 finaliser.
 *   key(seed, tid) = splitmix(splitmix(seed) ^ tid)
 * Normal draws use the Irwin-Hall sum of 12 uniforms: element i takes draws 3i..3i+2,
 * splits them into twelve 16-bit integers u_j and returns (sum u_j - 6*65536) / 65536.
 * That value is exact in fp32, so host and device agree bit for bit. A bf16 value is
 * then bf16_rne(sigma * z) (one fp32 multiply), or bf16_rne(offset + sigma * z) with
 * two separately rounded fp32 operations when an offset is given (gains: 1 + 0.05 z).
 * The distribution has the mean and std of N(0,1) but tails bounded at +-6.
 *
 * Tensor ids: tid = kind << 32 | layer << 16 | sub, with `sub` the expert (weights)
 * or b * n_kv + g (KV streams). The element index within a tensor is row-major.
 */
#ifndef SYNTH_H
#define SYNTH_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum synth_kind {
  SYNTH_EMBED = 1,      /* [V][H]             sigma 0.02          */
  SYNTH_GAIN = 2,       /* [H] per layer      1 + 0.05 z          */
  SYNTH_FINAL_GAIN = 3, /* [H]                1 + 0.05 z          */
  SYNTH_QKV = 4,        /* [(nq+2nkv)d][H]    sigma 0.02          */
  SYNTH_O = 5,          /* [H][nq d]          sigma 0.02          */
  SYNTH_ROUTER = 6,     /* [E][H]             sigma 0.02          */
  SYNTH_GATE_UP = 7,    /* [2I][H] per expert sigma 0.02          */
  SYNTH_DOWN = 8,       /* [H][I] per expert  sigma 0.02          */
  SYNTH_LM = 9,         /* [V][H]             sigma 0.02          */
  SYNTH_K = 10,         /* logical [pos][d] per (layer, b, g), N(0,1) */
  SYNTH_V = 11,
  SYNTH_TOKENS = 12,    /* uniform ids                            */
  SYNTH_CTX = 13,       /* uniform context lengths                */
  SYNTH_PAGES = 14,     /* page-pool permutation draws            */
  SYNTH_ZIPF = 15       /* router-bias expert permutation draws   */
};

uint64_t synth_tid(int kind, int layer, int sub);
uint64_t synth_key(uint64_t seed, uint64_t tid);
/* raw 64-bit draw n of a stream */
uint64_t synth_draw(uint64_t key, uint64_t n);
/* one normal value (exact fp32) */
float synth_normal(uint64_t key, uint64_t i);
/* fp32 -> bf16 bits, round to nearest even (NaN kept quiet) */
uint16_t synth_bf16(float f);

/* out[i] = bf16(offset + sigma * z(start+i)), i < count; offset 0 means bf16(sigma * z). */
void synth_fill_bf16(uint64_t seed, uint64_t tid, uint64_t start, uint64_t count, float sigma,
                     float offset, uint16_t* out);
/* out[i] = uniform integer in [lo, hi] from draw (start+i) */
void synth_fill_uniform_int(uint64_t seed, uint64_t tid, uint64_t start, uint64_t count, int64_t lo,
                            int64_t hi, int64_t* out);
/* Fisher-Yates permutation of [0, n) driven by stream tid */
void synth_permutation(uint64_t seed, uint64_t tid, int64_t n, int32_t* out);

#ifdef __cplusplus
}
#endif
#endif
