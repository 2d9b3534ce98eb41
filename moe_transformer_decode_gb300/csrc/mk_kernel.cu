// The persistent decode-step kernel for sm_103a: one CTA per SM, one producer warp that
// streams weights and KV pages into a shared-memory ring with bulk / tensor TMA copies,
// and eight consumer warps that run the opcodes. Dependencies between tasks on different
// SMs are acquire/release counters in global memory with bounded waits (no grid barrier).
//
// Decode step and fused opcodes: Cohere megakernel news pages, aimodeling.com
// "cohere-megakernel-north-mini-code-h100", section "One persistent kernel for the whole
// decode step" (task list in global memory, per-producer counters, O-proj released per KV
// group, weight prefetch ahead of dependencies, parallel-layer backfill) and
// aibriefing.imbch.dev article 8171681, section "Key Technologies and Architecture"
// (fused RoPE and SiLU-multiply, fixed-size task descriptors).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mk_internal.h"

namespace mk {

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// waits up to about `ns` nanoseconds with the warp suspended (woken when the phase completes)
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// 1D bulk copy global -> shared, completion counted on an mbarrier (16-byte aligned, size % 16 == 0),
// with an L2 cache policy
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}
// 2D tiled tensor copy global -> shared (x: innermost coordinate in elements), with an L2 cache policy
__device__ __forceinline__ void tma_2d_g2s(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}
// L2 policy for data read once per step (weights, KV pages): evicted first, so that the code,
// activations and counters the step keeps touching stay resident
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}
// pack two floats as bf16 (lo in the low half), with their rounding residuals as a second pair
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  uint16_t h0 = f2bf(x0), h1 = f2bf(x1);
  uint16_t l0 = f2bf(x0 - bf2f(h0)), l1 = f2bf(x1 - bf2f(h1));
  hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
  lo = (uint32_t)l0 | ((uint32_t)l1 << 16);
}

// ------------------------------------------------------------------ errors and waits

__device__ __noinline__ void report(const Params& p, int code, int aux0, int aux1) {
  if (atomicCAS(&p.status[ST_CODE], 0, code) == 0) {
    atomicExch(&p.status[ST_AUX0], aux0);
    atomicExch(&p.status[ST_AUX1], aux1);
    if (p.status_host) *reinterpret_cast<volatile int32_t*>(p.status_host) = code;
  }
  if (code == MK_ERR_DEVICE_TIMEOUT) atomicExch(&p.status[ST_ABORT], 1);
}
__device__ __forceinline__ bool aborted(const Params& p) {
  return *reinterpret_cast<volatile int*>(&p.status[ST_ABORT]) != 0;
}
__device__ __forceinline__ uint32_t target_of(const Params& p, int idx) {
  return p.epoch * (uint32_t)p.cnt_per_step[idx];
}

// Slow-path checks of every bounded wait are time based, on the SM cycle counter: the
// abort flag (an L2 read) is looked at only every kAbortPollCycles of waiting, so a wait that
// is about to succeed is not held up by that read; the time limit uses %globaltimer.
constexpr long long kAbortPollCycles = 40000;  // ~20 us at 2 GHz

struct WaitClock {
  long long next_poll;
  uint64_t t0;
  bool started;
  __device__ WaitClock() : next_poll(0), t0(0), started(false) {}
  // false when the wait must give up (abort seen or time limit passed)
  __device__ bool keep_going(const Params& p, int idx, int aux) {
    const long long now = clock64();
    if (!started) {
      started = true;
      next_poll = now + kAbortPollCycles;
      t0 = gtimer();
      return true;
    }
    if ((long long)(gtimer() - t0) > p.timeout_ns) {
      report(p, MK_ERR_DEVICE_TIMEOUT, idx, aux);
      return false;
    }
    if (now < next_poll) return true;
    next_poll = now + kAbortPollCycles;
    return !aborted(p);
  }
};

// single-thread bounded wait; false on timeout or abort
__device__ bool wait_counter(const Params& p, int idx) {
  const uint32_t tgt = target_of(p, idx);
  const uint32_t* c = p.counters + idx;
  WaitClock wc;
  for (;;) {
    const uint32_t v = ld_acquire(c);
    if ((int32_t)(v - tgt) >= 0) return true;
    if (!wc.keep_going(p, idx, (int)(v - (tgt - (uint32_t)p.cnt_per_step[idx])))) return false;
  }
}
// whole-warp wait (every lane performs the acquire)
__device__ bool warp_wait(const Params& p, int idx) {
  const uint32_t tgt = target_of(p, idx);
  const uint32_t* c = p.counters + idx;
  WaitClock wc;
  for (;;) {
    const uint32_t v = ld_acquire(c);
    if (__all_sync(0xffffffffu, (int32_t)(v - tgt) >= 0)) return true;
    int stop = 0;
    if ((threadIdx.x & 31) == 0) stop = !wc.keep_going(p, idx, (int)(v - (tgt - (uint32_t)p.cnt_per_step[idx])));
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
  }
}
// bounded mbarrier wait
__device__ bool mbar_wait(const Params& p, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  WaitClock wc;
  for (;;) {  // suspended between checks, so waiting warps leave the issue slots to working ones
    if (mbar_try_wait_sleep(bar, parity, 2000)) return true;
    if (!wc.keep_going(p, -1, (int)parity)) return false;
  }
}

// For the consumer warps' own barrier: re-test with the default short blocking wait instead of
// a long suspend, so the warps resume as soon as the last one arrives.
__device__ bool mbar_wait_cta(const Params& p, uint32_t bar, uint32_t parity) {
  WaitClock wc;
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (!wc.keep_going(p, -1, (int)parity)) return false;
  }
}

// ------------------------------------------------------------------ geometry

// A GEMV stage is RS rows x KS columns (row-major bf16 in shared memory). Each consumer warp
// owns 8 rows ("row group") and a 256-column slice; a lane owns 8 consecutive columns.
struct Geo {
  int KS, KW, RG, RS, NCS;
};
__device__ __forceinline__ Geo geo_of(int K) {
  Geo g;
  g.KS = K < 2048 ? K : 2048;
  g.KW = g.KS / 256;
  g.RG = kConsumerWarps / g.KW;
  g.RS = 8 * g.RG;
  g.NCS = K / g.KS;
  return g;
}

// QKV unit u (8 output rows). Units are group-major: for KV group g, the q heads of g, then
// k head g, then v head g; each q/k head has d/8 units of 4 RoPE pairs (i, i + d/2).
struct QkvUnit {
  int kind;   // 0 q, 1 k, 2 v
  int head;   // q head, or kv head for k / v
  int j;      // unit index within the head
  int row0;   // first row in W_qkv
};
__device__ __forceinline__ QkvUnit qkv_unit(const Params& p, int u) {
  const int dd8 = p.d / 8, upg = (p.group + 2) * dd8;
  const int g = u / upg, r = u % upg;
  QkvUnit q;
  if (r < p.group * dd8) {
    q.kind = 0; q.head = g * p.group + r / dd8; q.j = r % dd8; q.row0 = q.head * p.d + 4 * q.j;
  } else if (r < (p.group + 1) * dd8) {
    q.kind = 1; q.head = g; q.j = r - p.group * dd8; q.row0 = (p.nq + g) * p.d + 4 * q.j;
  } else {
    q.kind = 2; q.head = g; q.j = r - (p.group + 1) * dd8; q.row0 = (p.nq + p.nkv + g) * p.d + 8 * q.j;
  }
  return q;
}

__device__ __forceinline__ int pos_of(const Params& p, int b) { return p.positions[b] + p.pos_offset; }

struct AttnRange {
  int cp0, cp1, pos_end;
};
__device__ __forceinline__ AttnRange attn_range(int pos, int cpp, int nch, int c) {
  const int npg = (pos + kPage - 1) / kPage;
  AttnRange r;
  r.cp0 = c * cpp;
  r.cp1 = (c == nch - 1) ? npg : min(r.cp0 + cpp, npg);
  if (r.cp1 < r.cp0) r.cp1 = r.cp0;
  r.pos_end = pos;
  return r;
}
__device__ __forceinline__ int attn_pps(const Params& p) { return kStageBytes / (4096 * (p.d / 64)); }

__device__ __forceinline__ int max_active(const Params& p) { return min(p.B * p.topk, p.E); }

// ------------------------------------------------------------------ shared memory

struct Misc {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t cbar;                     // consumer-warps barrier (8 arrivals per phase)
  alignas(16) float red[2][kConsumerWarps][64];  // cross-warp partial sums, double-buffered by stage
  alignas(16) float res[64 * kMaxB];             // reduced stage results [RS][B]
  float norm[kConsumerWarps][kMaxB]; // sum of squares partials
  int flag;
  // routing scratch of the warp that computes a layer's routing
  uint32_t em[kMaxExperts];  // bit b: token b picked the expert
  int ids[kMaxB][kMaxK];
  float wk[kMaxB][kMaxK];
  // per step (consumers): new token's position, page of its KV slot (-1 if invalid), RoPE at it,
  // attention chunking
  int st_pos[kMaxB];
  int st_page[kMaxB];
  int st_cpp[kMaxB];
  int st_nch[kMaxB];
  alignas(16) float2 st_rope[kMaxB][64];
  // per layer (consumers): routing of layer rc_layer
  int rc_n;
  int rc_expert[kMaxActive];
  uint32_t rc_mask[kMaxActive];
  float rc_w[kMaxActive][kMaxB];
  // producer-private: routed experts of layer pr_layer
  int pr_n;
  int pr_expert[kMaxActive];
  // batch 1: the normalized input of the current layer, and per-warp LM argmax candidates
  alignas(16) float nsm[2048];
  float lmw_v[kConsumerWarps];
  int lmw_i[kConsumerWarps];
};
constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + ((int)sizeof(Misc) + 127) / 128 * 128;
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds the sm_103a opt-in limit");
static_assert(offsetof(Misc, red) % 16 == 0 && offsetof(Misc, res) % 16 == 0 && offsetof(Misc, st_rope) % 16 == 0 &&
                  offsetof(Misc, nsm) % 16 == 0,
              "vector-accessed shared arrays must be 16-byte aligned");

struct Ring {
  uint32_t data;  // shared address of stage 0
  uint32_t full, empty;
  uint32_t it;
};
__device__ __forceinline__ uint32_t slot_addr(const Ring& r) { return r.data + (r.it % kStages) * kStageBytes; }

// ------------------------------------------------------------------ producer

struct Producer {
  const Params& p;
  const TensorMaps& tm;
  Misc& m;
  Ring r;
  bool ok;
  uint32_t bar, dst;
  int pos[kMaxB], cpp[kMaxB], nch[kMaxB];  // per step
  int route_layer;
  uint64_t pol;  // L2 policy of every copy

  __device__ Producer(const Params& p_, const TensorMaps& tm_, Misc& m_, Ring r_)
      : p(p_), tm(tm_), m(m_), r(r_), ok(true), route_layer(-1) {
    pol = policy_evict_first();
#pragma unroll 1
    for (int b = 0; b < kMaxB; ++b) {
      pos[b] = b < p.B ? pos_of(p, b) : 0;
      cpp[b] = b < p.B ? p.chunk_pages[b] : 1;
      nch[b] = b < p.B ? p.n_chunks[b] : 1;
    }
  }

  // the routed experts of layer l, loaded once per layer
  __device__ bool route(int l) {
    if (route_layer == l) return true;
    if (!wait_counter(p, CounterMap{p.L, p.nkv, p.B}.route(l))) return false;
    const Route* rt = p.route + l;
    const int na = __ldcg(&rt->n_active);
#pragma unroll 1
    for (int a = 0; a < na; ++a) m.pr_expert[a] = __ldcg(&rt->expert[a]);
    m.pr_n = na;
    route_layer = l;
    return true;
  }

  __device__ bool begin(uint32_t bytes) {
    const uint32_t s = r.it % kStages;
    const uint32_t parity = ((r.it / kStages) & 1u) ^ 1u;
    if (!mbar_wait(p, r.empty + 8 * s, parity)) return false;
    bar = r.full + 8 * s;
    dst = r.data + s * kStageBytes;
    mbar_expect_tx(bar, bytes);
    return true;
  }
  __device__ void end() { ++r.it; }

  __device__ bool gemv_rows(const uint16_t* base, int rows, int row_bytes) {
    const uint32_t bytes = (uint32_t)rows * row_bytes;
    if (!begin(bytes)) return false;
    bulk_g2s(dst, base, bytes, bar, pol);
    end();
    return true;
  }

  __device__ bool run_task(const Task& t) {
    const int l = t.layer;
    switch (t.op) {
      case OP_ROUTER:
      case OP_LM: {
        const Geo g = geo_of(p.H);
        const uint16_t* W = t.op == OP_ROUTER ? p.w_router + (size_t)l * p.E * p.H : p.lm_head;
#pragma unroll 1
        for (int r0 = t.a; r0 < t.a + t.b; r0 += g.RS)
          if (!gemv_rows(W + (size_t)r0 * p.H, min(g.RS, t.a + t.b - r0), p.H * 2)) return false;
        return true;
      }
      case OP_QKV: {
        const Geo g = geo_of(p.H);
        const int us = g.RG;  // units per stage
        const uint16_t* W = p.w_qkv + (size_t)l * p.qkv_rows * p.H;
#pragma unroll 1
        for (int u0 = t.a; u0 < t.a + t.b; u0 += us) {
          const int nu = min(us, t.a + t.b - u0);
          if (!begin((uint32_t)nu * 8 * p.H * 2)) return false;
#pragma unroll 1
          for (int i = 0; i < nu; ++i) {
            const QkvUnit q = qkv_unit(p, u0 + i);
            const uint32_t d0 = dst + (uint32_t)i * 8 * p.H * 2;
            if (q.kind == 2) {
              bulk_g2s(d0, W + (size_t)q.row0 * p.H, 8 * p.H * 2, bar, pol);
            } else {
              bulk_g2s(d0, W + (size_t)q.row0 * p.H, 4 * p.H * 2, bar, pol);
              bulk_g2s(d0 + 4 * p.H * 2, W + (size_t)(q.row0 + p.d / 2) * p.H, 4 * p.H * 2, bar, pol);
            }
          }
          end();
        }
        return true;
      }
      case OP_ATTN: {
        const int b = t.a, g = t.b;
        const AttnRange ar = attn_range(pos[b], cpp[b], nch[b], t.c);
        const int pps = attn_pps(p), halves = p.d / 64;
        int ids[64];  // page ids of up to 64 pages, loaded together (one round trip per 64 pages)
#pragma unroll 1
        for (int base = ar.cp0; base < ar.cp1; base += 64) {
          const int nb = min(64, ar.cp1 - base);
#pragma unroll 1
          for (int i0 = 0; i0 < nb; i0 += 8) {
            int v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int pg = base + i0 + j;
              v[j] = (i0 + j < nb && pg < p.max_pages) ? __ldg(&p.block_table[b * p.max_pages + pg]) : -1;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (i0 + j < nb) ids[i0 + j] = v[j];
          }
#pragma unroll 1
          for (int i = 0; i < nb; ++i)
            if (ids[i] < 0 || ids[i] >= p.num_pages) {
              report(p, MK_ERR_BAD_PAGE, b, base + i);
              ids[i] = -1;
            }
#pragma unroll 1
          for (int s0 = 0; s0 < nb; s0 += pps) {
            const int np = min(pps, nb - s0);
            if (!begin((uint32_t)np * 2 * halves * 2048)) return false;
#pragma unroll 1
            for (int i = 0; i < np; ++i) {
              // an invalid page (reported above) is loaded as zeros: a tile load at an
              // out-of-range row fills the box, so the stage never holds stale bytes
              const int id = ids[s0 + i];
              const int row = id >= 0 ? ((l * p.num_pages + id) * p.nkv + g) * kPage : -kPage;
              const uint32_t pb = dst + (uint32_t)i * 4096 * halves;
#pragma unroll 1
              for (int h = 0; h < halves; ++h) {
                tma_2d_g2s(pb + h * 2048, &tm.k, h * 64, row, bar, pol);
                tma_2d_g2s(pb + (halves + h) * 2048, &tm.v, h * 64, row, bar, pol);
              }
            }
            end();
          }
        }
        return true;
      }
      case OP_GU: {
        if (!route(l)) return false;
        const int na = m.pr_n, maxa = max_active(p);
        const Geo g = geo_of(p.H);
#pragma unroll 1
        for (int u = t.a; u < t.a + t.b; ++u) {
          const int a = u % maxa, tile = u / maxa;
          if (a >= na) continue;
          const int e = m.pr_expert[a];
          const uint16_t* W = p.w_gate_up + ((size_t)l * p.E + e) * 2 * p.I * p.H;
          if (!begin((uint32_t)g.RS * p.H * 2)) return false;
          bulk_g2s(dst, W + (size_t)tile * g.RS * p.H, (uint32_t)g.RS * p.H * 2, bar, pol);
          end();
        }
        return true;
      }
      case OP_O: {
        const Geo g = geo_of(p.od);
        const uint16_t* W = p.w_o + ((size_t)l * p.H + t.a) * p.od;
#pragma unroll 1
        for (int cs = 0; cs < g.NCS; ++cs) {
          if (g.NCS == 1) {
            if (!gemv_rows(W, t.b, p.od * 2)) return false;
          } else {
            if (!begin((uint32_t)t.b * g.KS * 2)) return false;
#pragma unroll 1
            for (int r = 0; r < t.b; ++r)
              bulk_g2s(dst + (uint32_t)r * g.KS * 2, W + (size_t)r * p.od + cs * g.KS, g.KS * 2, bar, pol);
            end();
          }
        }
        return true;
      }
      case OP_DOWN: {
        if (!route(l)) return false;
        const int na = m.pr_n;
#pragma unroll 1
        for (int a = 0; a < na; ++a) {
          const int e = m.pr_expert[a];
          const uint16_t* W = p.w_down + (((size_t)l * p.E + e) * p.H + t.a) * p.I;
          if (!gemv_rows(W, t.b, p.I * 2)) return false;
        }
        return true;
      }
    }
    return true;
  }

  // Abort path: wait until every copy this warp issued has landed. Bounded, but by its own
  // limit (1 s), not the caller's wait limit: a copy in flight completes in microseconds, and
  // the block must not leave while one still writes its shared memory.
  __device__ void drain() {
    const uint32_t n = r.it < (uint32_t)kStages ? r.it : (uint32_t)kStages;
    for (uint32_t k = 0; k < n; ++k) {
      const uint32_t it = r.it - 1 - k;
      const uint32_t s = it % kStages, parity = (it / kStages) & 1u;
      const uint64_t t0 = gtimer();
      while (!mbar_try_wait(r.full + 8 * s, parity)) {
        if (gtimer() - t0 > 1000000000ull) break;
      }
    }
  }
};

// ------------------------------------------------------------------ consumer building blocks

// Halving butterfly: sums v[N] over the 32 lanes. For N <= 32 the lane ends with the total
// of index lane >> (5 - log2 N) in v[0]; for N = 64 with indices 2*lane and 2*lane+1.
template <int C, int O>
struct LaneReduce {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (O > 0) {
      if constexpr (C > 1) {
        const bool up = (lane & O) != 0;
#pragma unroll
        for (int i = 0; i < C / 2; ++i) {
          const float send = up ? v[i] : v[i + C / 2];
          const float keep = up ? v[i + C / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
        }
        LaneReduce<C / 2, O / 2>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
        LaneReduce<1, O / 2>::run(v, lane);
      }
    }
  }
};

template <int NB>
__device__ __forceinline__ void warp_partials_to_smem(float (&acc)[8][NB], float* red_w, int lane) {
  constexpr int N = 8 * NB;
  float v[N];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) v[r * NB + b] = acc[r][b];
  LaneReduce<N, 16>::run(v, lane);
  if constexpr (N <= 32) {
    constexpr int rep = 32 / N;
    if ((lane & (rep - 1)) == 0) red_w[lane / rep] = v[0];
  } else {
    red_w[2 * lane] = v[0];
    red_w[2 * lane + 1] = v[1];
  }
}

// Sum the row groups' k-slices of red into res[row * NB + b] for rows < rows, using threads
// [t0, t0 + nthreads). Caller syncs around.
template <int NB>
__device__ __forceinline__ void cross_warp_reduce(const float (*red)[64], float* res, const Geo& g, int rows, int t,
                                                  int nthreads) {
  for (int e = t; e < rows * NB; e += nthreads) {
    const int r = e / NB, b = e % NB, rg = r / 8;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < g.KW) s += red[rg * g.KW + k][(r % 8) * NB + b];
    res[e] = s;
  }
}

// Accumulate one stage's rows for this warp: acc[r][b] += W[row][cols] . act[b][cols]
template <int NB>
__device__ __forceinline__ void gemv_stage(const uint8_t* stage, const Geo& g, int rg, int ks, int lane, int rows_valid,
                                           const float (&act)[NB][8], float (&acc)[8][NB], uint32_t bmask) {
  const uint8_t* base = stage + (size_t)(rg * 8) * g.KS * 2 + (size_t)(ks * 256 + lane * 8) * 2;
  constexpr int RB = NB <= 2 ? 8 : (NB == 4 ? 4 : 2);  // rows whose loads are in flight together
#pragma unroll
  for (int r0 = 0; r0 < 8; r0 += RB) {
    uint4 w[RB];
#pragma unroll
    for (int j = 0; j < RB; ++j)
      w[j] = r0 + j < rows_valid ? *reinterpret_cast<const uint4*>(base + (size_t)(r0 + j) * g.KS * 2)
                                 : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      const int r = r0 + j;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (bmask & (1u << b)) {  // two accumulation chains per row
          float s0 = fmaf(bf_lo(w[j].x), act[b][0], acc[r][b]);
          float s1 = bf_hi(w[j].x) * act[b][1];
          s0 = fmaf(bf_lo(w[j].y), act[b][2], s0);
          s1 = fmaf(bf_hi(w[j].y), act[b][3], s1);
          s0 = fmaf(bf_lo(w[j].z), act[b][4], s0);
          s1 = fmaf(bf_hi(w[j].z), act[b][5], s1);
          s0 = fmaf(bf_lo(w[j].w), act[b][6], s0);
          s1 = fmaf(bf_hi(w[j].w), act[b][7], s1);
          acc[r][b] = s0 + s1;
        }
      }
    }
  }
}

template <int NB>
__device__ __forceinline__ void zero_acc(float (&acc)[8][NB]) {
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;
}

__device__ __forceinline__ void load8(const float* src, float (&dst)[8]) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(src));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(src) + 1);
  dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
  dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
}

__device__ __forceinline__ void trace_task(const Params& p, const Task& t, uint64_t t0, uint64_t t1) {
  if (!p.trace || threadIdx.x != 0) return;
  const uint64_t t2 = gtimer();
  const unsigned long long i = atomicAdd(p.trace_count, 1ull);
  if ((long long)i >= p.trace_cap) return;
  mk_trace_entry e;
  e.t_start_ns = t0;
  e.wait_ns = (uint32_t)(t1 - t0);
  e.run_ns = (uint32_t)(t2 - t1);
  e.sm = (uint16_t)blockIdx.x;
  e.op = t.op;
  e.layer = t.layer;
  e.pad = 0;
  e.a = t.a;
  e.b = t.b;
  p.trace[i] = e;
}

// ------------------------------------------------------------------ consumer

template <int NB>
struct Consumer {
  const Params& p;
  Misc& m;
  Ring r;
  CounterMap cm;
  int warp, lane;
  bool ok;
  uint32_t cbar, cphase;
  int rpar;             // which half of m.red the next reduction uses
  int n_layer;          // layer whose normalized input is held in `nact` (-1 none)
  int route_layer;      // layer whose routing is cached in m.rc_*
  int gu_layer;         // layer whose expert gate/up work is known complete
  int attn_layer;       // layer of attn_ok
  uint32_t attn_ok;     // KV groups whose attention is known complete in attn_layer
  float nact[NB][8];    // this lane's 8 columns of the normalized input, per token
  float lm_best[NB];    // running LM-head argmax (threads < B)
  int lm_idx[NB];
  uint64_t t_start, t_ready;

  __device__ Consumer(const Params& p_, Misc& m_, Ring r_)
      : p(p_), m(m_), r(r_), cm{p_.L, p_.nkv, p_.B}, ok(true), n_layer(-1), route_layer(-1), gu_layer(-1),
        attn_layer(-1), attn_ok(0) {
    warp = threadIdx.x / 32;
    lane = threadIdx.x % 32;
    cbar = smem_addr(&m_.cbar);
    cphase = 0;
    rpar = 0;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      lm_best[b] = -INFINITY;
      lm_idx[b] = 0x7fffffff;
    }
  }

  __device__ const uint8_t* acquire() {
    const uint32_t s = r.it % kStages, parity = (r.it / kStages) & 1u;
    if (!mbar_wait(p, r.full + 8 * s, parity)) {
      ok = false;
      return nullptr;
    }
    return reinterpret_cast<const uint8_t*>(__cvta_shared_to_generic(r.data + s * kStageBytes));
  }
  __device__ void release() {
    __syncwarp();
    if (lane == 0) mbar_arrive(r.empty + 8 * (r.it % kStages));
    ++r.it;
  }
  __device__ uint32_t bmask_all() const { return (1u << p.B) - 1u; }
  // h holds, per (layer, active expert, token), the raw gate then up projections [2I]
  __device__ __forceinline__ size_t h_index(int l, int a, int b) const {
    return (((size_t)l * kMaxActive + a) * kMaxB + b) * 2 * (size_t)p.I;
  }
  // SiLU(gate) * up * routing weight for 8 consecutive intermediate columns
  __device__ __forceinline__ void load_h8(int l, int a, int b, int col, float wgt, float (&dst)[8]) const {
    float gt[8], up[8];
    load8(p.h + h_index(l, a, b) + col, gt);
    load8(p.h + h_index(l, a, b) + p.I + col, up);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = gt[i] / (1.0f + expf(-gt[i])) * up[i] * wgt;
  }

  // Barrier of the 8 consumer warps on an mbarrier, with the same time limit as every other
  // wait: a warp that gives up (timeout or abort) leaves the kernel and the rest follow.
  __device__ bool csync() {
    __syncwarp();
    if (lane == 0) mbar_arrive(cbar);
    const bool done = mbar_wait_cta(p, cbar, cphase);
    cphase ^= 1u;
    if (!done) ok = false;
    return done;
  }

  // The normalized input of layer l (l == L: the final norm before the LM head), for this
  // lane's 8 columns: x = residual stream (embedding at l = 0), n = x / rms(x) * gain.
  __device__ void load_norm(int l, bool write_x) {
    const Geo g = geo_of(p.H);
    const int ks = warp % g.KW;
    const int col = ks * 256 + lane * 8;
    if (l > 0 && !warp_wait(p, cm.layer(l - 1))) {
      ok = false;
      return;
    }
    float x[NB][8];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[b][i] = 0.f;
      if (b >= p.B) continue;
      if (l == 0) {
        int tok = p.token_ids[b];
        if (tok < 0 || tok >= p.V) {
          if (lane == 0 && warp == 0) report(p, MK_ERR_BAD_TOKEN, b, tok);
          tok = 0;
        }
        const uint4 w = *reinterpret_cast<const uint4*>(p.embed + (size_t)tok * p.H + col);
        x[b][0] = bf_lo(w.x); x[b][1] = bf_hi(w.x); x[b][2] = bf_lo(w.y); x[b][3] = bf_hi(w.y);
        x[b][4] = bf_lo(w.z); x[b][5] = bf_hi(w.z); x[b][6] = bf_lo(w.w); x[b][7] = bf_hi(w.w);
      } else {
        float a[8], mo[8];
        const size_t o = ((size_t)(l - 1) * p.B + b) * p.H + col;
        load8(p.xs + o, x[b]);
        load8(p.attn_out + o, a);
        load8(p.moe_out + o, mo);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[b][i] = (x[b][i] + a[i]) + mo[i];
      }
    }
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) s = fmaf(x[b][i], x[b][i], s);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      ss[b] = s;
    }
    if (lane == 0 && warp < g.KW)
#pragma unroll
      for (int b = 0; b < NB; ++b) m.norm[warp][b] = ss[b];
    if (!csync()) return;
    const uint16_t* gain = (l < p.L) ? p.norm_gain + (size_t)l * p.H : p.final_gain;
    const uint4 gw = *reinterpret_cast<const uint4*>(gain + col);
    const float gf[8] = {bf_lo(gw.x), bf_hi(gw.x), bf_lo(gw.y), bf_hi(gw.y),
                         bf_lo(gw.z), bf_hi(gw.z), bf_lo(gw.w), bf_hi(gw.w)};
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float tot = 0.f;
      for (int k = 0; k < g.KW; ++k) tot += m.norm[k][b];
      const float rinv = 1.0f / sqrtf(tot / (float)p.H + p.eps);
#pragma unroll
      for (int i = 0; i < 8; ++i) nact[b][i] = x[b][i] * rinv * gf[i];
    }
    if constexpr (NB == 1) {
      if (warp < g.KW) {
        float4* dn = reinterpret_cast<float4*>(&m.nsm[col]);
        dn[0] = make_float4(nact[0][0], nact[0][1], nact[0][2], nact[0][3]);
        dn[1] = make_float4(nact[0][4], nact[0][5], nact[0][6], nact[0][7]);
      }
    }
    if (write_x && warp < g.KW) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= p.B) continue;
        float4* dst = reinterpret_cast<float4*>(p.xs + ((size_t)l * p.B + b) * p.H + col);
        __stcg(dst, make_float4(x[b][0], x[b][1], x[b][2], x[b][3]));
        __stcg(dst + 1, make_float4(x[b][4], x[b][5], x[b][6], x[b][7]));
      }
    }
    if (!csync()) return;
    n_layer = l;
  }

  __device__ void ensure_norm(int l, bool write_x) {
    if (n_layer != l) load_norm(l, write_x);
  }

  // One GEMV stage against the held normalized input. All warps add their partials to one
  // half of m.red and meet once; warp 0 then reduces them into m.res [rows][NB] and runs
  // `epi` (its lanes), while the other warps go on to the next stage.
  template <typename Epi>
  __device__ bool norm_gemv_stage(const Geo& g, int rows, uint32_t bmask, Epi&& epi) {
    const int rg = warp / g.KW, ks = warp % g.KW;
    float acc[8][NB];
    zero_acc(acc);
    const uint8_t* st = acquire();
    if (!st) return false;
    if (rg < g.RG) gemv_stage<NB>(st, g, rg, ks, lane, min(8, rows - rg * 8), nact, acc, bmask);
    release();
    if (rg < g.RG) warp_partials_to_smem<NB>(acc, m.red[rpar][warp], lane);
    if (!csync()) return false;
    if (warp == 0) {
      cross_warp_reduce<NB>(m.red[rpar], m.res, g, rows, lane, 32);
      __syncwarp();
      epi();
    }
    rpar ^= 1;
    return true;
  }

  __device__ void release_counter(int idx) {
    if (!csync()) return;
    // the barrier orders every consumer's writes before thread 0's gpu-scope release
    if (threadIdx.x == 0) red_release_add(p.counters + idx, 1u);
  }
  // arrival on `idx`; true in every consumer thread of the task that arrived last
  __device__ bool arrive_last(int idx, int count) {
    if (!csync()) return false;
    if (threadIdx.x == 0) {
      const uint32_t old = atom_acq_rel_add(p.counters + idx, 1u);
      m.flag = ((old + 1u) % (uint32_t)count) == 0u;
    }
    if (!csync()) return false;
    return m.flag != 0;
  }

  // Per-step values every block needs, read once: positions, the new slots' pages, RoPE at the
  // positions, attention chunking.
  __device__ bool load_step_cache() {
    const int hd = p.d / 2;
    if (threadIdx.x < p.B) {
      const int b = threadIdx.x;
      const int pos = pos_of(p, b);
      int page = -1;
      if (pos >= 0 && pos / kPage < p.max_pages) {
        page = p.block_table[b * p.max_pages + pos / kPage];
        if (page < 0 || page >= p.num_pages) page = -1;
      }
      m.st_pos[b] = pos;
      m.st_page[b] = page;
      m.st_cpp[b] = p.chunk_pages[b];
      m.st_nch[b] = p.n_chunks[b];
    }
    for (int i = threadIdx.x; i < p.B * hd; i += 256) {
      const int b = i / hd, j = i % hd;
      const int pos = pos_of(p, b);
      m.st_rope[b][j] = (pos >= 0 && pos < p.max_pos) ? p.rope[(size_t)pos * hd + j] : make_float2(1.f, 0.f);
    }
    return csync();
  }

  // Routing of layer l in shared memory, loaded once per layer and block.
  __device__ bool load_route(int l) {
    if (route_layer == l) return true;
    if (!warp_wait(p, cm.route(l))) { ok = false; return false; }
    const Route* rt = p.route + l;
    const int na = __ldcg(&rt->n_active);
    for (int i = threadIdx.x; i < na; i += 256) {
      m.rc_expert[i] = __ldcg(&rt->expert[i]);
      m.rc_mask[i] = __ldcg(&rt->mask[i]);
    }
    for (int i = threadIdx.x; i < na * kMaxB; i += 256) m.rc_w[i / kMaxB][i % kMaxB] = __ldcg(&rt->w[i / kMaxB][i % kMaxB]);
    if (threadIdx.x == 0) m.rc_n = na;
    if (!csync()) return false;
    route_layer = l;
    return true;
  }
  __device__ bool wait_gu(int l) {
    if (gu_layer == l) return true;
    if (!warp_wait(p, cm.gu(l))) { ok = false; return false; }
    gu_layer = l;
    return true;
  }
  __device__ bool wait_attn_group(int l, int gg) {
    if (attn_layer != l) { attn_layer = l; attn_ok = 0; }
    if (attn_ok & (1u << gg)) return true;
    if (!warp_wait(p, cm.attn(l, gg))) { ok = false; return false; }
    attn_ok |= 1u << gg;
    return true;
  }

  // ---------------------------------------------------------------- opcodes

  __device__ void op_router(const Task& t) {
    const int l = t.layer;
    t_ready = gtimer();
    const Geo g = geo_of(p.H);
    for (int r0 = t.a; r0 < t.a + t.b && ok; r0 += g.RS) {
      const int rows = min(g.RS, t.a + t.b - r0);
      const bool st_ok = norm_gemv_stage(g, rows, bmask_all(), [&] {
        for (int i = lane; i < rows * NB; i += 32) {
          const int rr = i / NB, b = i % NB;
          if (b >= p.B) continue;
          const int e = r0 + rr;
          const float bias = p.router_bias ? p.router_bias[(size_t)l * p.E + e] : 0.f;
          __stcg(&p.rlogits[((size_t)l * p.B + b) * p.E + e], m.res[i] + bias);
        }
      });
      if (!st_ok) return;
    }
    if (arrive_last_w0(cm.router_arrive(l), p.cnt_per_step[cm.router_arrive(l)])) publish_routing(l);
  }

  // Arrival on `idx` once every consumer warp's writes are done; true in warp 0 of the task
  // that arrived last (the other warps get false and go on to their next task).
  __device__ bool arrive_last_w0(int idx, int count) {
    if (!csync()) return false;
    if (warp != 0) return false;
    uint32_t last = 0;
    if (lane == 0) last = ((atom_acq_rel_add(p.counters + idx, 1u) + 1u) % (uint32_t)count) == 0u;
    return __shfl_sync(0xffffffffu, last, 0) != 0u;
  }

  // Routing of layer l by warp 0 alone, then published with one release of the route counter.
  // Per token: top-k (value descending, lower expert id first on ties), softmax over the k
  // selected logits. Then the distinct routed experts in ascending id, each with its token
  // mask and per-token weights. Lane owns experts lane + 32 i.
  __device__ void publish_routing(int l) {
    constexpr int NE = kMaxExperts / 32;
    const int E = p.E, K = p.topk, B = p.B;
    float v[NB][NE];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        const int e = lane + 32 * i;
        const float x = (b < B && e < E) ? __ldcg(&p.rlogits[((size_t)l * B + b) * E + e]) : -INFINITY;
        v[b][i] = x == x ? x : -INFINITY;  // a NaN logit ranks last
      }
    uint32_t emask[NE];
#pragma unroll
    for (int i = 0; i < NE; ++i) emask[i] = 0u;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b >= B) break;
      float top0 = 0.f, z = 0.f;
      uint32_t taken = 0u;  // bit i: expert lane + 32 i already picked for token b
      for (int j = 0; j < K; ++j) {
        // every pick is a valid, distinct expert: -inf ties go to the lowest free id
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NE; ++i) {
          const int e = lane + 32 * i;
          if (e < E && !((taken >> i) & 1u) && (v[b][i] > bv || (v[b][i] == bv && e < be))) { bv = v[b][i]; be = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
#pragma unroll
        for (int i = 0; i < NE; ++i)
          if (lane + 32 * i == be) { taken |= 1u << i; emask[i] |= 1u << b; }
        if (j == 0) top0 = bv;
        const float w = expf(bv - top0);
        z += w;
        if (lane == 0) { m.ids[b][j] = be; m.wk[b][j] = w; }
      }
      __syncwarp();
      if (lane < K) m.wk[b][lane] /= z;
    }
    __syncwarp();
    // token masks per expert, then the distinct experts in ascending id (32 per round)
#pragma unroll 1
    for (int e = lane; e < E; e += 32) m.em[e] = 0u;
    __syncwarp();
#pragma unroll 1
    for (int i = lane; i < B * K; i += 32) atomicOr(&m.em[m.ids[i / K][i % K]], 1u << (i / K));
    __syncwarp();
    Route* rt = p.route + l;
    int na = 0;
#pragma unroll 1
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const uint32_t mask = e < E ? m.em[e] : 0u;
      const uint32_t act = __ballot_sync(0xffffffffu, mask != 0u);
      if (mask != 0u) {
        const int r = na + __popc(act & ((1u << lane) - 1u));
        __stcg(&rt->expert[r], e);
        __stcg(&rt->mask[r], mask);
#pragma unroll 1
        for (int b = 0; b < kMaxB; ++b) {
          float w = 0.f;
          if (mask & (1u << b)) {
#pragma unroll 1
            for (int j = 0; j < K; ++j) w = m.ids[b][j] == e ? m.wk[b][j] : w;
          }
          __stcg(&rt->w[r][b], w);
        }
      }
      na += __popc(act);
    }
    if (lane == 0) __stcg(&rt->n_active, na);
    for (int i = lane; i < B * K; i += 32) {
      const int b = i / K, j = i % K;
      __stcg(&rt->ids[b][j], m.ids[b][j]);
      __stcg(&rt->wk[b][j], m.wk[b][j]);
      __stcg(&p.topk_ids[((size_t)l * B + b) * K + j], m.ids[b][j]);
      __stcg(&p.topk_w[((size_t)l * B + b) * K + j], m.wk[b][j]);
    }
    __syncwarp();
    if (lane == 0) red_release_add(p.counters + cm.route(l), 1u);
  }

  __device__ void op_qkv(const Task& t) {
    const int l = t.layer;
    t_ready = gtimer();
    const Geo g = geo_of(p.H);
    const int hd = p.d / 2;
    for (int u0 = t.a; u0 < t.a + t.b && ok; u0 += g.RG) {
      const int nu = min(g.RG, t.a + t.b - u0);
      const bool st_ok = norm_gemv_stage(g, nu * 8, bmask_all(), [&] {
      // epilogue: RoPE on q/k pairs, bf16 K/V append
      for (int i = lane; i < nu * 8 * NB; i += 32) {
        const int unit = i / (8 * NB), rem = i % (8 * NB), tt = rem / NB, b = rem % NB;
        if (b >= p.B) continue;
        const QkvUnit q = qkv_unit(p, u0 + unit);
        const int pos = m.st_pos[b];
        const int page = q.kind != 0 ? m.st_page[b] : -1;
        if (q.kind != 0 && page < 0 && tt == 0 && unit == 0) report(p, MK_ERR_BAD_PAGE, b, pos);
        const float* res = m.res + unit * 8 * NB;
        if (q.kind == 2) {  // v: 8 consecutive elements
          const int e = 8 * q.j + tt;
          const uint16_t vb = f2bf(res[tt * NB + b]);
          __stcg(&p.vnew[(((size_t)l * p.B + b) * p.nkv + q.head) * p.d + e], bf2f(vb));
          if (page >= 0)
            p.vpool[((((size_t)l * p.num_pages + page) * p.nkv + q.head) * kPage + pos % kPage) * p.d + e] = vb;
          continue;
        }
        if (q.kind == 0) {  // q is stored before RoPE; attention rotates it when it loads it
          const int e = 4 * q.j + (tt & 3) + (tt >= 4 ? hd : 0);
          __stcg(&p.q[(((size_t)l * p.B + b) * p.nq + q.head) * p.d + e], res[tt * NB + b]);
          continue;
        }
        if (tt >= 4) continue;  // k pair (tt, tt + 4) handled by the lower row
        const int pi2 = 4 * q.j + tt;  // pair index in [0, d/2)
        const float a = res[tt * NB + b], c = res[(tt + 4) * NB + b];
        const float2 cs = m.st_rope[b][pi2];
        const float lo = a * cs.x - c * cs.y;
        const float hi = a * cs.y + c * cs.x;
        {
          const uint16_t kl = f2bf(lo), kh = f2bf(hi);
          float* dst = p.knew + (((size_t)l * p.B + b) * p.nkv + q.head) * p.d;
          __stcg(dst + pi2, bf2f(kl));
          __stcg(dst + pi2 + hd, bf2f(kh));
          if (page >= 0) {
            uint16_t* kp = p.kpool + ((((size_t)l * p.num_pages + page) * p.nkv + q.head) * kPage + pos % kPage) * p.d;
            kp[pi2] = kl;
            kp[pi2 + hd] = kh;
          }
        }
      }
      });
      if (!st_ok) return;
    }
    if (ok) release_counter(cm.qkv(l, t.c));
  }

  __device__ void op_gu(const Task& t) {
    const int l = t.layer;
    if (!load_route(l)) return;
    t_ready = gtimer();
    const int na = m.rc_n, maxa = max_active(p);
    const Geo g = geo_of(p.H);
    for (int u = t.a; u < t.a + t.b && ok; ++u) {
      const int a = u % maxa, tile = u / maxa;
      if (a >= na) continue;
      const uint32_t bm = m.rc_mask[a];
      const bool st_ok = norm_gemv_stage(g, g.RS, bm, [&] {
        for (int i = lane; i < g.RS * NB; i += 32) {
          const int rr = i / NB, b = i % NB;
          if (bm & (1u << b)) __stcg(&p.h[h_index(l, a, b) + tile * g.RS + rr], m.res[i]);
        }
      });
      if (!st_ok) return;
    }
    if (ok) release_counter(cm.gu(l));
  }

  __device__ void op_o(const Task& t) {
    const int l = t.layer;
    const Geo g = geo_of(p.od);
    const int rg = warp / g.KW, ks = warp % g.KW;
    const int gw = p.group * p.d;  // columns per KV group
    float acc[8][NB];
    zero_acc(acc);
    t_ready = 0;
    for (int cs = 0; cs < g.NCS; ++cs) {
      const int c0 = cs * g.KS + ks * 256;
      float act[NB][8];
      if (rg < g.RG) {
        for (int gg = c0 / gw; gg <= (c0 + 255) / gw; ++gg)
          if (!wait_attn_group(l, gg)) return;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b < p.B) load8(p.attn_o + ((size_t)l * p.B + b) * p.od + c0 + lane * 8, act[b]);
          else
#pragma unroll
            for (int i = 0; i < 8; ++i) act[b][i] = 0.f;
        }
      }
      if (!t_ready) t_ready = gtimer();
      const uint8_t* st = acquire();
      if (!st) return;
      if (rg < g.RG) gemv_stage<NB>(st, g, rg, ks, lane, min(8, t.b - rg * 8), act, acc, bmask_all());
      release();
    }
    if (rg < g.RG) warp_partials_to_smem<NB>(acc, m.red[rpar][warp], lane);
    if (!csync()) return;
    cross_warp_reduce<NB>(m.red[rpar], m.res, g, t.b, threadIdx.x, 256);
    rpar ^= 1;
    if (!csync()) return;
    for (int i = threadIdx.x; i < t.b * NB; i += 256) {
      const int rr = i / NB, b = i % NB;
      if (b < p.B) __stcg(&p.attn_out[((size_t)l * p.B + b) * p.H + t.a + rr], m.res[i]);
    }
    release_counter(cm.layer(l));
  }

  __device__ void op_down(const Task& t) {
    const int l = t.layer;
    if (!load_route(l) || !wait_gu(l)) return;
    t_ready = gtimer();
    const Geo g = geo_of(p.I);
    const int rg = warp / g.KW, ks = warp % g.KW;
    const int na = m.rc_n;
    float acc[8][NB];
    zero_acc(acc);
    for (int a = 0; a < na; ++a) {
      const uint32_t bm = m.rc_mask[a];
      float act[NB][8];
      if (rg < g.RG) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (bm & (1u << b)) {
            load_h8(l, a, b, ks * 256 + lane * 8, m.rc_w[a][b], act[b]);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) act[b][i] = 0.f;
          }
        }
      }
      const uint8_t* st = acquire();
      if (!st) return;
      if (rg < g.RG) gemv_stage<NB>(st, g, rg, ks, lane, min(8, t.b - rg * 8), act, acc, bm);
      release();
    }
    if (rg < g.RG) warp_partials_to_smem<NB>(acc, m.red[rpar][warp], lane);
    if (!csync()) return;
    cross_warp_reduce<NB>(m.red[rpar], m.res, g, t.b, threadIdx.x, 256);
    rpar ^= 1;
    if (!csync()) return;
    for (int i = threadIdx.x; i < t.b * NB; i += 256) {
      const int rr = i / NB, b = i % NB;
      if (b < p.B) __stcg(&p.moe_out[((size_t)l * p.B + b) * p.H + t.a + rr], m.res[i]);
    }
    release_counter(cm.layer(l));
  }

  __device__ void op_lm(const Task& t) {
    t_ready = gtimer();
    const Geo g = geo_of(p.H);
    for (int r0 = t.a; r0 < t.a + t.b && ok; r0 += g.RS) {
      const int rows = min(g.RS, t.a + t.b - r0);
      const bool st_ok = norm_gemv_stage(g, rows, bmask_all(), [&] {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int e = lane; e < rows * NB; e += 32) {  // e % NB == lane % NB since 32 % NB == 0
          const int rr = e / NB, b = e % NB;
          const float v = m.res[e];
          if (b < p.B && p.logits) __stcg(&p.logits[(size_t)b * p.V + r0 + rr], v);
          if (v > bv || (v == bv && r0 + rr < bi)) { bv = v; bi = r0 + rr; }
        }
#pragma unroll
        for (int o = 16; o >= NB; o >>= 1) {  // combine lanes of the same token, lowest id on ties
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (bv > lm_best[0] || (bv == lm_best[0] && bi < lm_idx[0])) { lm_best[0] = bv; lm_idx[0] = bi; }
      });
      if (!st_ok) return;
    }
    if (!(t.flags & TF_LAST_LM) || !ok) return;
    if (threadIdx.x < NB && threadIdx.x < p.B) {  // warp 0, lane b: token b
      __stcg(&p.lm_best_v[t.c * kMaxB + threadIdx.x], lm_best[0]);
      __stcg(&p.lm_best_i[t.c * kMaxB + threadIdx.x], lm_idx[0]);
    }
    if (!arrive_last(cm.lm_arrive(), p.n_lm_sm)) return;
    if (threadIdx.x < p.B) {
      const int b = threadIdx.x;
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int s = 0; s < p.n_lm_sm; ++s) {
        const float v = __ldcg(&p.lm_best_v[s * kMaxB + b]);
        const int i = __ldcg(&p.lm_best_i[s * kMaxB + b]);
        if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
      }
      if (p.argmax_out) p.argmax_out[b] = bi;
    }
  }


  // ---------------------------------------------------------------- batch-1 row-per-warp opcodes
  // With one token, a warp owns whole rows of a stage (all H columns, the normalized input in
  // registers), so each row needs only a warp reduction and its epilogue runs in that warp: no
  // block-wide barrier per stage.

  // this lane's columns pp*256 + lane*8 + i of the normalized input held in m.nsm
  __device__ __forceinline__ void rows_act(float (&a)[64]) const {
    const int np = p.H / 256;
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) {
      if (pp < np) {
        const float4 x = *reinterpret_cast<const float4*>(&m.nsm[pp * 256 + lane * 8]);
        const float4 y = *reinterpret_cast<const float4*>(&m.nsm[pp * 256 + lane * 8 + 4]);
        a[pp * 8 + 0] = x.x; a[pp * 8 + 1] = x.y; a[pp * 8 + 2] = x.z; a[pp * 8 + 3] = x.w;
        a[pp * 8 + 4] = y.x; a[pp * 8 + 5] = y.y; a[pp * 8 + 6] = y.z; a[pp * 8 + 7] = y.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) a[pp * 8 + i] = 0.f;
      }
    }
  }
  // full-warp dot of one shared-memory row (np * 256 bf16 columns) with a
  __device__ __forceinline__ float rdot(const uint8_t* row, int np, const float (&a)[64]) const {
    uint4 w[8];
#pragma unroll
    for (int pp = 0; pp < 8; ++pp)
      w[pp] = pp < np ? *reinterpret_cast<const uint4*>(row + (size_t)(pp * 256 + lane * 8) * 2) : make_uint4(0, 0, 0, 0);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) {
      s0 = fmaf(bf_lo(w[pp].x), a[pp * 8 + 0], s0);
      s1 = fmaf(bf_hi(w[pp].x), a[pp * 8 + 1], s1);
      s0 = fmaf(bf_lo(w[pp].y), a[pp * 8 + 2], s0);
      s1 = fmaf(bf_hi(w[pp].y), a[pp * 8 + 3], s1);
      s0 = fmaf(bf_lo(w[pp].z), a[pp * 8 + 4], s0);
      s1 = fmaf(bf_hi(w[pp].z), a[pp * 8 + 5], s1);
      s0 = fmaf(bf_lo(w[pp].w), a[pp * 8 + 6], s0);
      s1 = fmaf(bf_hi(w[pp].w), a[pp * 8 + 7], s1);
    }
    float s = s0 + s1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
  }

  __device__ void op_router_r(const Task& t) {
    const int l = t.layer;
    t_ready = gtimer();
    float a[64];
    rows_act(a);
    const int np = p.H / 256;
    const Geo g = geo_of(p.H);
    for (int r0 = t.a; r0 < t.a + t.b; r0 += g.RS) {
      const int rows = min(g.RS, t.a + t.b - r0);
      const uint8_t* st = acquire();
      if (!st) return;
      for (int r = warp; r < rows; r += kConsumerWarps) {
        const float s = rdot(st + (size_t)r * p.H * 2, np, a);
        if (lane == 0) {
          const int e = r0 + r;
          const float bias = p.router_bias ? p.router_bias[(size_t)l * p.E + e] : 0.f;
          __stcg(&p.rlogits[(size_t)l * p.E + e], s + bias);
        }
      }
      release();
    }
    if (arrive_last_w0(cm.router_arrive(l), p.cnt_per_step[cm.router_arrive(l)])) publish_routing(l);
  }

  __device__ void op_qkv_r(const Task& t) {
    const int l = t.layer;
    t_ready = gtimer();
    float a[64];
    rows_act(a);
    const Geo g = geo_of(p.H);
    const int np = p.H / 256, hd = p.d / 2;
    const int pos = m.st_pos[0], page = m.st_page[0];
    for (int u0 = t.a; u0 < t.a + t.b; u0 += g.RG) {
      const int nu = min(g.RG, t.a + t.b - u0);
      const uint8_t* st = acquire();
      if (!st) return;
      int item = 0;
      for (int i = 0; i < nu; ++i) {
        const QkvUnit q = qkv_unit(p, u0 + i);
        const uint8_t* ub = st + (size_t)i * 8 * p.H * 2;
        if (q.kind == 0) {  // q: 8 rows, stored before RoPE (attention rotates q when it loads it)
          for (int tt = 0; tt < 8; ++tt, ++item) {
            if (item % kConsumerWarps != warp) continue;
            const float s = rdot(ub + (size_t)tt * p.H * 2, np, a);
            if (lane == 0) __stcg(&p.q[((size_t)l * p.nq + q.head) * p.d + 4 * q.j + (tt & 3) + (tt >= 4 ? hd : 0)], s);
          }
        } else if (q.kind == 2) {  // v: 8 rows = 8 consecutive elements of v head q.head
          for (int tt = 0; tt < 8; ++tt, ++item) {
            if (item % kConsumerWarps != warp) continue;
            const float s = rdot(ub + (size_t)tt * p.H * 2, np, a);
            if (lane == 0) {
              const int e = 8 * q.j + tt;
              const uint16_t vb = f2bf(s);
              __stcg(&p.vnew[((size_t)l * p.nkv + q.head) * p.d + e], bf2f(vb));
              if (page >= 0)
                p.vpool[((((size_t)l * p.num_pages + page) * p.nkv + q.head) * kPage + pos % kPage) * p.d + e] = vb;
            }
          }
        } else {  // k: RoPE pair (4 j + tt, 4 j + tt + d/2) from rows tt and tt + 4, for the cache
          for (int tt = 0; tt < 4; ++tt, ++item) {
            if (item % kConsumerWarps != warp) continue;
            const float x0 = rdot(ub + (size_t)tt * p.H * 2, np, a);
            const float x1 = rdot(ub + (size_t)(tt + 4) * p.H * 2, np, a);
            if (lane == 0) {
              const int pi2 = 4 * q.j + tt;
              const float2 cs = m.st_rope[0][pi2];
              const float lo = x0 * cs.x - x1 * cs.y;
              const float hi = x0 * cs.y + x1 * cs.x;
              {
                const uint16_t kl = f2bf(lo), kh = f2bf(hi);
                float* dst = p.knew + ((size_t)l * p.nkv + q.head) * p.d;
                __stcg(dst + pi2, bf2f(kl));
                __stcg(dst + pi2 + hd, bf2f(kh));
                if (page >= 0) {
                  uint16_t* kp = p.kpool + ((((size_t)l * p.num_pages + page) * p.nkv + q.head) * kPage + pos % kPage) * p.d;
                  kp[pi2] = kl;
                  kp[pi2 + hd] = kh;
                }
              }
            }
          }
        }
      }
      release();
    }
    if (page < 0 && threadIdx.x == 0) report(p, MK_ERR_BAD_PAGE, 0, pos);
    release_counter(cm.qkv(l, t.c));
  }

  __device__ void op_gu_r(const Task& t) {
    const int l = t.layer;
    if (!load_route(l)) return;
    t_ready = gtimer();
    float a[64];
    rows_act(a);
    const int na = m.rc_n, maxa = max_active(p);
    const Geo g = geo_of(p.H);
    const int np = p.H / 256;
    for (int u = t.a; u < t.a + t.b; ++u) {
      const int ar = u % maxa, tile = u / maxa;
      if (ar >= na) continue;
      const uint8_t* st = acquire();
      if (!st) return;
      for (int rr = warp; rr < g.RS; rr += kConsumerWarps) {
        const float s = rdot(st + (size_t)rr * p.H * 2, np, a);
        if (lane == 0) __stcg(&p.h[h_index(l, ar, 0) + tile * g.RS + rr], s);
      }
      release();
    }
    release_counter(cm.gu(l));
  }

  __device__ void op_lm_r(const Task& t) {
    t_ready = gtimer();
    float a[64];
    rows_act(a);
    const int np = p.H / 256;
    const Geo g = geo_of(p.H);
    for (int r0 = t.a; r0 < t.a + t.b; r0 += g.RS) {
      const int rows = min(g.RS, t.a + t.b - r0);
      const uint8_t* st = acquire();
      if (!st) return;
      for (int r = warp; r < rows; r += kConsumerWarps) {  // ascending rows per warp
        const float s = rdot(st + (size_t)r * p.H * 2, np, a);
        if (lane == 0) {
          const int v = r0 + r;
          if (p.logits) __stcg(&p.logits[v], s);
          if (s > lm_best[0] || (s == lm_best[0] && v < lm_idx[0])) { lm_best[0] = s; lm_idx[0] = v; }
        }
      }
      release();
    }
    if (!(t.flags & TF_LAST_LM)) return;
    if (lane == 0) { m.lmw_v[warp] = lm_best[0]; m.lmw_i[warp] = lm_idx[0]; }
    if (!csync()) return;
    if (threadIdx.x == 0) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int w = 0; w < kConsumerWarps; ++w)
        if (m.lmw_v[w] > bv || (m.lmw_v[w] == bv && m.lmw_i[w] < bi)) { bv = m.lmw_v[w]; bi = m.lmw_i[w]; }
      __stcg(&p.lm_best_v[t.c * kMaxB], bv);
      __stcg(&p.lm_best_i[t.c * kMaxB], bi);
    }
    if (!arrive_last(cm.lm_arrive(), p.n_lm_sm)) return;
    if (threadIdx.x == 0) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int s = 0; s < p.n_lm_sm; ++s) {
        const float v = __ldcg(&p.lm_best_v[s * kMaxB]);
        const int i = __ldcg(&p.lm_best_i[s * kMaxB]);
        if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
      }
      if (p.argmax_out) p.argmax_out[0] = bi;
    }
  }

  // Paged GQA attention of one (sequence b, KV group g, chunk). The G <= 8 query heads of the
  // group are the 16 rows of an mma A operand: rows 0..7 hold the bf16 "hi" part of q and rows
  // 8..15 its rounding residual, so S = q K^T comes out at ~fp32 accuracy; P is split the same
  // way for P V. K/V tiles arrive 128B-swizzled from the tensor maps (conflict-free ldmatrix).
  __device__ void op_attn(const Task& t) {
    const int l = t.layer, b = t.a, g = t.b;
    if (!warp_wait(p, cm.qkv(l, g))) { ok = false; return; }
    t_ready = gtimer();
    const AttnRange ar = attn_range(m.st_pos[b], m.st_cpp[b], m.st_nch[b], t.c);
    const int pps = attn_pps(p), halves = p.d / 64, ksteps = p.d / 16;
    const int pi = warp % pps, dp = warp / pps;
    const int head = lane >> 2, tig = lane & 3;
    const float qscale = rsqrtf((float)p.d) * 1.4426950408889634f;  // scores in log2 units
    uint32_t qa[8][4];
    {
      // q arrives before RoPE: element d pairs with d + d/2, which this lane also holds (k-step
      // kk + ksteps/2), so the rotation happens here in registers
      const float* qh = p.q + (((size_t)l * p.B + b) * p.nq + g * p.group + head) * p.d;
      const bool hv = head < p.group;
      float x[8][4];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int d0 = kk * 16 + tig * 2;
#pragma unroll
        for (int e = 0; e < 4; ++e) x[kk][e] = (kk < ksteps && hv) ? __ldcg(qh + d0 + (e & 1) + (e >> 1) * 8) : 0.f;
      }
      const int half = ksteps / 2, hd = p.d / 2;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (kk < half) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d0 = kk * 16 + tig * 2 + (e & 1) + (e >> 1) * 8;  // < d/2
            const float2 cs = m.st_rope[b][d0];
            const float lo = x[kk][e], hi = x[kk + half][e];
            x[kk][e] = lo * cs.x - hi * cs.y;
            x[kk + half][e] = lo * cs.y + hi * cs.x;
          }
        }
      }
      (void)hd;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        if (kk < ksteps) {
          split_pack(x[kk][0] * qscale, x[kk][1] * qscale, qa[kk][0], qa[kk][1]);
          split_pack(x[kk][2] * qscale, x[kk][3] * qscale, qa[kk][2], qa[kk][3]);
        }
      }
    }
    float mrun = -INFINITY, lsum = 0.f;
    float oacc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) oacc[i][j] = 0.f;

    const int nst = (ar.cp1 - ar.cp0 + pps - 1) / pps;
    uint32_t last_slot = 0;
    for (int s = 0; s < nst; ++s) {
      const uint8_t* st = acquire();
      if (!st) return;
      const int page = ar.cp0 + s * pps + pi;
      if (page < ar.cp1) {
        const uint32_t kt = smem_addr(st) + (uint32_t)pi * 4096 * halves;
        const uint32_t vt = kt + (uint32_t)halves * 2048;
        float sc[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) sc[i][j] = 0.f;
        const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if (kk < ksteps) {
            const int prow = (mi >> 1) * 8 + rr;           // position within the page
            const int chunk = 2 * kk + (mi & 1);          // 16-byte chunk of the head dim
            const uint32_t addr = kt + (chunk >> 3) * 2048 + prow * 128 + (((chunk & 7) ^ (prow & 7)) << 4);
            uint32_t bk[4];
            ldsm_x4(addr, bk);
            mma_bf16(sc[0], qa[kk], bk[0], bk[1]);
            mma_bf16(sc[1], qa[kk], bk[2], bk[3]);
          }
        }
        float sv[2][2];
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pos = page * kPage + nt * 8 + tig * 2 + e;
            const float s_ = sc[nt][e] + sc[nt][e + 2];
            sv[nt][e] = pos < ar.pos_end ? s_ : -INFINITY;
            mx = fmaxf(mx, sv[nt][e]);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mnew = fmaxf(mrun, mx);
        if (mnew != -INFINITY) {
          const float alpha = exp2f(mrun - mnew);
          lsum *= alpha;
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) oacc[i][j] *= alpha;
          mrun = mnew;
          float pr[2][2];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              pr[nt][e] = exp2f(sv[nt][e] - mnew);
              lsum += pr[nt][e];
            }
          uint32_t pa[4];
          split_pack(pr[0][0], pr[0][1], pa[0], pa[1]);
          split_pack(pr[1][0], pr[1][1], pa[2], pa[3]);
#pragma unroll
          for (int c2 = 0; c2 < 4; ++c2) {  // two 8-wide d tiles per ldmatrix.x4.trans
            const int chunk = dp * 8 + c2 * 2 + (mi >> 1);
            const int prow = (mi & 1) * 8 + rr;
            const uint32_t addr = vt + (chunk >> 3) * 2048 + prow * 128 + (((chunk & 7) ^ (prow & 7)) << 4);
            uint32_t bv[4];
            ldsm_x4_t(addr, bv);
            mma_bf16(oacc[c2 * 2], pa, bv[0], bv[1]);
            mma_bf16(oacc[c2 * 2 + 1], pa, bv[2], bv[3]);
          }
        }
      }
      if (s + 1 < nst) release();
      else last_slot = smem_addr(st);
    }
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);

    // merge the warps that share a d range (different pages), using the last slot as scratch
    const size_t pidx = (((size_t)l * p.B + b) * p.nkv + g) * p.max_chunks + t.c;
    float* part = p.apart + pidx * (16 + 8 * (size_t)p.d);
    if (nst > 0) {
      if (!csync()) return;
      float* scr = reinterpret_cast<float*>(__cvta_shared_to_generic(last_slot));
      // per warp: m[8], l[8], O[8][64]
      float* mine = scr + warp * (16 + 8 * 64);
      if (tig == 0) { mine[head] = mrun; mine[8 + head] = lsum; }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) mine[16 + head * 64 + nt * 8 + tig * 2 + e] = oacc[nt][e] + oacc[nt][e + 2];
      if (!csync()) return;
      for (int i = threadIdx.x; i < 8 * p.d; i += 256) {
        const int h = i / p.d, dd = i % p.d, dpi = dd / 64, dl = dd % 64;
        float M = -INFINITY;
        for (int w = dpi * pps; w < (dpi + 1) * pps; ++w) M = fmaxf(M, scr[w * (16 + 512) + h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY)
          for (int w = dpi * pps; w < (dpi + 1) * pps; ++w) {
            const float* src = scr + w * (16 + 512);
            if (src[h] == -INFINITY) continue;
            const float f = exp2f(src[h] - M);
            L += src[8 + h] * f;
            O += src[16 + h * 64 + dl] * f;
          }
        if (dd == 0) { __stcg(part + h, M); __stcg(part + 8 + h, L); }
        __stcg(part + 16 + i, O);
      }
      if (!csync()) return;
      release();
    } else {
      for (int i = threadIdx.x; i < 16 + 8 * p.d; i += 256) __stcg(part + i, i < 8 ? -INFINITY : 0.f);
    }
    const int arr = cm.attn_arrive(l, b, g);
    if (!arrive_last(arr, m.st_nch[b])) return;

    // combine the chunks of (b, g) with the new token (position pos, read from knew / vnew)
    const int nch = m.st_nch[b];
    const float* pbase = p.apart + (((size_t)l * p.B + b) * p.nkv + g) * p.max_chunks * (16 + 8 * (size_t)p.d);
    // s_new per head: warp h < group
    if (warp < p.group) {
      const float* qh = p.q + (((size_t)l * p.B + b) * p.nq + g * p.group + warp) * p.d;
      const float* kn = p.knew + (((size_t)l * p.B + b) * p.nkv + g) * p.d;
      float s = 0.f;
      const int hd = p.d / 2;
      for (int i = lane; i < hd; i += 32) {  // q before RoPE: rotate pair (i, i + d/2)
        const float2 cs = m.st_rope[b][i];
        const float q0 = __ldcg(qh + i), q1 = __ldcg(qh + i + hd);
        s = fmaf(q0 * cs.x - q1 * cs.y, __ldcg(kn + i), s);
        s = fmaf(q0 * cs.y + q1 * cs.x, __ldcg(kn + i + hd), s);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) m.res[warp] = s * qscale;
    }
    if (!csync()) return;
    const float* vn = p.vnew + (((size_t)l * p.B + b) * p.nkv + g) * p.d;
    const size_t cstride = 16 + 8 * (size_t)p.d;
    if (nch <= 64) {
      // chunk maxima and sums in one parallel load round, scale factors in shared memory, then
      // independent loads of the chunk outputs
      float* sm_m = &m.red[0][0][0];  // [nch][8]: chunk max, then its scale factor
      float* sm_l = &m.red[1][0][0];  // [nch][8]: chunk sum
      for (int i = threadIdx.x; i < nch * 8; i += 256) {
        const float* src = pbase + (size_t)(i / 8) * cstride;
        sm_m[i] = __ldcg(src + (i % 8));
        sm_l[i] = __ldcg(src + 8 + (i % 8));
      }
      if (!csync()) return;
      if (threadIdx.x < p.group) {
        const int h = threadIdx.x;
        const float sn = m.res[h];
        float M = sn;
        for (int c = 0; c < nch; ++c) M = fmaxf(M, sm_m[c * 8 + h]);
        const float fn = exp2f(sn - M);
        float L = fn;
        for (int c = 0; c < nch; ++c) {
          const float mc = sm_m[c * 8 + h];
          const float f = mc == -INFINITY ? 0.f : exp2f(mc - M);
          L += sm_l[c * 8 + h] * f;
          sm_m[c * 8 + h] = f;
        }
        m.res[8 + h] = fn;
        m.res[16 + h] = 1.0f / L;
      }
      if (!csync()) return;
      for (int i = threadIdx.x; i < p.group * p.d; i += 256) {
        const int h = i / p.d, dd = i % p.d;
        const float* src = pbase + 16 + h * p.d + dd;
        float O = m.res[8 + h] * __ldcg(vn + dd);
        int c = 0;
        for (; c + 8 <= nch; c += 8) {
          float v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + (size_t)(c + j) * cstride);
#pragma unroll
          for (int j = 0; j < 8; ++j) O = fmaf(v[j], sm_m[(c + j) * 8 + h], O);
        }
        for (; c < nch; ++c) O = fmaf(__ldcg(src + (size_t)c * cstride), sm_m[c * 8 + h], O);
        __stcg(&p.attn_o[((size_t)l * p.B + b) * p.od + (g * p.group + h) * p.d + dd], O * m.res[16 + h]);
      }
    } else {
      for (int i = threadIdx.x; i < p.group * p.d; i += 256) {
        const int h = i / p.d, dd = i % p.d;
        const float sn = m.res[h];
        float M = sn;
        for (int c = 0; c < nch; ++c) M = fmaxf(M, __ldcg(pbase + (size_t)c * cstride + h));
        float fn = exp2f(sn - M);
        float L = fn, O = fn * __ldcg(vn + dd);
        for (int c = 0; c < nch; ++c) {
          const float* src = pbase + (size_t)c * cstride;
          const float mc = __ldcg(src + h);
          if (mc == -INFINITY) continue;
          const float f = exp2f(mc - M);
          L += __ldcg(src + 8 + h) * f;
          O += __ldcg(src + 16 + h * p.d + dd) * f;
        }
        __stcg(&p.attn_o[((size_t)l * p.B + b) * p.od + (g * p.group + h) * p.d + dd], O / L);
      }
    }
    release_counter(cm.attn(l, g));
  }

  __device__ void run_task(const Task& t) {
    t_start = gtimer();
    t_ready = t_start;
    // ops that read the normalized input of their layer (the final norm for the LM head) get it
    // here, at one call site
    if (t.op == OP_ROUTER || t.op == OP_QKV || t.op == OP_GU || t.op == OP_LM) {
      ensure_norm(t.op == OP_LM ? p.L : (int)t.layer, (t.flags & TF_WRITE_X) != 0);
      if (!ok) return;
    }
    if constexpr (NB == 1) {
      switch (t.op) {
        case OP_ROUTER: op_router_r(t); break;
        case OP_QKV: op_qkv_r(t); break;
        case OP_ATTN: op_attn(t); break;
        case OP_GU: op_gu_r(t); break;
        case OP_O: op_o(t); break;
        case OP_DOWN: op_down(t); break;
        case OP_LM: op_lm_r(t); break;
      }
    } else {
      switch (t.op) {
        case OP_ROUTER: op_router(t); break;
        case OP_QKV: op_qkv(t); break;
        case OP_ATTN: op_attn(t); break;
        case OP_GU: op_gu(t); break;
        case OP_O: op_o(t); break;
        case OP_DOWN: op_down(t); break;
        case OP_LM: op_lm(t); break;
      }
    }
    if (ok) trace_task(p, t, t_start, t_ready ? t_ready : t_start);
  }
};

// ------------------------------------------------------------------ kernel

template <int NB>
__global__ void __launch_bounds__(kThreads, 1) mk_decode_kernel(const __grid_constant__ Params p,
                                                                const __grid_constant__ TensorMaps tm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& misc = *reinterpret_cast<Misc*>(base + kStages * kStageBytes);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&misc.full[s]), 1);
      mbar_init(smem_addr(&misc.empty[s]), kConsumerWarps);
    }
    mbar_init(smem_addr(&misc.cbar), kConsumerWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  Ring ring;
  ring.data = smem_addr(base);
  ring.full = smem_addr(&misc.full[0]);
  ring.empty = smem_addr(&misc.empty[0]);
  ring.it = 0;
  const int t0 = p.sm_begin[blockIdx.x], t1 = p.sm_begin[blockIdx.x + 1];

  if (threadIdx.x / 32 >= kConsumerWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    if (threadIdx.x != kConsumerWarps * 32) return;
    Producer pr(p, tm, misc, ring);
    // descriptors in a 4-deep register queue, refilled as tasks are taken (one call site, so
    // the task code is inlined once)
    const uint4* src = reinterpret_cast<const uint4*>(p.tasks);
    const uint4 zero = make_uint4(0, 0, 0, 0);
    uint4 q0 = t0 < t1 ? __ldg(src + t0) : zero, q1 = t0 + 1 < t1 ? __ldg(src + t0 + 1) : zero;
    uint4 q2 = t0 + 2 < t1 ? __ldg(src + t0 + 2) : zero, q3 = t0 + 3 < t1 ? __ldg(src + t0 + 3) : zero;
    bool fine = true;
    for (int i = t0; i < t1 && fine; ++i) {
      const uint4 nx = i + 4 < t1 ? __ldg(src + i + 4) : zero;
      fine = pr.run_task(*reinterpret_cast<const Task*>(&q0));
      q0 = q1;
      q1 = q2;
      q2 = q3;
      q3 = nx;
    }
    pr.drain();  // never leave while a copy into this CTA's shared memory is in flight
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
  Consumer<NB> c(p, misc, ring);
  if (!c.load_step_cache()) return;
  // descriptors in batches of 32 (lane j holds descriptor base + j), the next batch loaded
  // while the current one runs; each task is broadcast from its lane
  const uint4* src = reinterpret_cast<const uint4*>(p.tasks);
  const int lane = threadIdx.x & 31;
  uint4 cur = t0 + lane < t1 ? __ldg(src + t0 + lane) : make_uint4(0, 0, 0, 0);
  for (int base = t0; base < t1 && c.ok; base += 32) {
    const uint4 nxt = base + 32 + lane < t1 ? __ldg(src + base + 32 + lane) : make_uint4(0, 0, 0, 0);
    const int n = min(32, t1 - base);
    for (int j = 0; j < n && c.ok; ++j) {
      uint4 v;
      v.x = __shfl_sync(0xffffffffu, cur.x, j);
      v.y = __shfl_sync(0xffffffffu, cur.y, j);
      v.z = __shfl_sync(0xffffffffu, cur.z, j);
      v.w = __shfl_sync(0xffffffffu, cur.w, j);
      c.run_task(*reinterpret_cast<const Task*>(&v));
    }
    cur = nxt;
  }
}

}  // namespace mk

// ------------------------------------------------------------------ launch entry (host)

namespace mk {
int kernel_smem_bytes() { return kSmemBytes; }

cudaError_t configure_kernels() {
  cudaError_t e = cudaFuncSetAttribute(mk_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mk_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mk_decode_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mk_decode_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  return e;
}

template <int NB>
static cudaError_t launch_nb(const Params& p, const TensorMaps& tm, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_sm);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mk_decode_kernel<NB>, p, tm);
}

cudaError_t launch_decode(const Params& p, const TensorMaps& tm, cudaStream_t st) {
  if (p.B <= 1) return launch_nb<1>(p, tm, st);
  if (p.B <= 2) return launch_nb<2>(p, tm, st);
  if (p.B <= 4) return launch_nb<4>(p, tm, st);
  return launch_nb<8>(p, tm, st);
}

cudaError_t max_blocks_per_sm(int B, int* n) {
  if (B <= 1) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, mk_decode_kernel<1>, kThreads, kSmemBytes);
  if (B <= 2) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, mk_decode_kernel<2>, kThreads, kSmemBytes);
  if (B <= 4) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, mk_decode_kernel<4>, kThreads, kSmemBytes);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, mk_decode_kernel<8>, kThreads, kSmemBytes);
}
}  // namespace mk
