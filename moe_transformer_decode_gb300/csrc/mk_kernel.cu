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
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
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
// 3D tiled tensor copy global -> shared (coordinates innermost first), with an L2 cache policy
__device__ __forceinline__ void tma_3d_g2s(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar,
                                           uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}
// ------------------------------------------------------------------ tcgen05 (5th-generation tensor cores)
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle (rows of 128 bytes, 16-byte
// units XOR-swizzled by row within 1 KB groups of 8 rows), sbo = byte distance between 8-row
// groups along M or N (0 makes every group alias the first: 8 distinct rows).
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t addr, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(sbo >> 4) << 32;         // stride byte offset
  d |= (uint64_t)1 << 46;                  // descriptor version
  d |= (uint64_t)2 << 61;                  // 128-byte swizzle
  return d;
}
// instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32 accumulator, M x N
__host__ __device__ constexpr uint32_t tc_idesc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// The same, issued from a converged warp: every lane computes the (warp-uniform) operands and
// the elected lane (the lowest, lane 0) issues. In isolation (one warp issuing back to back) this
// form issued about 30 % faster than lane 0 alone under a branch (measured).
__device__ __forceinline__ void tc_mma_warp(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.u32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// arrive once on the mbarrier when every tcgen05.mma this thread issued so far has completed
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// the same from a converged warp, by the elected lane (the one that issued the products)
__device__ __forceinline__ void tc_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (lane i of the warp reads lane
// 32 (warp % 4) + i); the wait is in the same statement, so no register is read before it lands
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(n) : "memory");
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
// Cross-proxy ordering. Bulk and tensor copies run in the async proxy; plain loads and stores
// in the generic proxy. Global data written by generic stores (on any SM) and read here by a
// bulk copy needs this fence after the acquire that made the writes visible, and a shared-memory
// region written by generic stores and then overwritten by a copy needs the shared-memory form.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
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
// explicit shared-memory loads (a generic load of shared data waits on the long scoreboard)
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
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

constexpr uint32_t kPollSuspendNs = 200;  // suspend limit of the producer's free-slot waits

// single-thread bounded wait; false on timeout or abort
__device__ bool wait_counter(const Params& p, int idx) {
  const uint32_t tgt = target_of(p, idx);
  const uint32_t* c = p.counters + (size_t)idx * kCounterStride;
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
  const uint32_t* c = p.counters + (size_t)idx * kCounterStride;
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
  if (mbar_test_wait(bar, parity)) return true;
  WaitClock wc;
  for (;;) {  // suspended between checks, so waiting warps leave the issue slots to working ones
    if (mbar_try_wait_sleep(bar, parity, 2000)) return true;
    if (!wc.keep_going(p, -1, (int)parity)) return false;
  }
}

// Spinning bounded mbarrier wait, for barriers whose phases complete by asynchronous arrivals
// (tensor-core commits, copy completions) that the waiter must see at once: a warp suspended in
// try_wait is not woken early by them.
__device__ bool mbar_wait_spin(const Params& p, uint32_t bar, uint32_t parity) {
  WaitClock wc;
  for (int i = 0;; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((i & 63) == 63 && !wc.keep_going(p, -1, (int)parity)) return false;
  }
}

// Bounded wait with a short suspend limit, for the producer's free-slot waits: a slot of a
// tensor-core stage is freed by a commit (an asynchronous arrival), which does not wake a warp
// suspended in try_wait, so the suspension must end by itself soon; the consumers' own arrivals
// wake it at once.
__device__ bool mbar_wait_poll(const Params& p, uint32_t bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  WaitClock wc;
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kPollSuspendNs)) return true;
    if (!wc.keep_going(p, -1, (int)parity)) return false;
  }
}

// For the consumer warps' own barrier: re-test with the default short blocking wait instead of
// a long suspend, so the warps resume as soon as the last one arrives.
__device__ bool mbar_wait_cta(const Params& p, uint32_t bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  WaitClock wc;
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (!wc.keep_going(p, -1, (int)parity)) return false;
  }
}

// ------------------------------------------------------------------ geometry

// A GEMV stage is RS rows x KS columns of bf16, row-major in shared memory (RST = 2 KS bytes
// apart, as in global memory, so a stage of consecutive rows is one bulk copy). Each consumer
// warp owns 8 rows ("row group") and a 256-column slice (16 mma k-steps).
struct Geo {
  int KS, KW, RG, RS, NCS, RST;
};
__device__ __forceinline__ Geo geo_of(int K) {
  Geo g;
  g.KS = K < 2048 ? K : 2048;
  g.KW = g.KS / 256;
  g.RG = kConsumerWarps / g.KW;
  g.RS = 8 * g.RG;
  g.NCS = K / g.KS;
  g.RST = g.KS * 2;
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
__device__ __forceinline__ int attn_pps(const Params& p) { return kStagePayload / (4096 * (p.d / 64)); }

// Gate/up task t.a of t.b (a layer's tasks) takes units [v0, v1) of the step's na x tiles units,
// unit v = (routed expert rank v % na, row block v / na): an equal share of the experts the step
// actually routes to, however many that is. Producer and consumers compute it alike from the
// layer's routing, so the split is deterministic and needs no claim counter.
struct GuRange {
  int v0, v1;
};
__device__ __forceinline__ GuRange gu_range(const Task& t, int na, int tiles) {
  const long long total = (long long)na * tiles;
  return GuRange{(int)(total * t.a / t.b), (int)(total * (t.a + 1) / t.b)};
}

__device__ __forceinline__ int max_active(const Params& p) { return min(p.B * p.topk, p.E); }

// ------------------------------------------------------------------ shared memory

constexpr int kRedBufs = 4;    // GEMV partial-sum buffers in flight
constexpr int kIdCache = 128;  // page ids the producer keeps (the same pages serve every layer)

struct Misc {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t cbar;                     // consumer-warps barrier (8 arrivals per phase)
  uint64_t tc_acc;                   // tcgen05: a unit's products have all completed (commit)
  uint64_t acc_full[2];              // gate/up: accumulator buffer b holds a unit's finished products
  uint64_t acc_empty[2];             // gate/up: the epilogue warps have read buffer b
  uint32_t tmem_base;                // tcgen05: the block's tensor memory (kTmemCols columns)
  uint64_t gpart[kRedBufs];          // GEMV pass buffers: every consumer warp's partials are in
  uint64_t gfree[kRedBufs];          // ... and: the pass's epilogue warp has read them
  union {
    // GEMV partial sums [buffer][warp][row * 8 + token]; also scratch of the attention combine
    alignas(16) float red[kRedBufs][kConsumerWarps][64];
    // per-warp exchange area (256 floats each) for building the norm input's mma fragments; used
    // only between the norm load's block barriers, when no GEMV pass is in flight
    alignas(16) float nsm[kConsumerWarps * 256];
  };
  float norm[kConsumerWarps][kMaxB]; // sum of squares partials
  int flag;
  int wait_failed;  // set by the polling warp of a block-wide wait that gave up
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
  alignas(16) float rc_w[kMaxActive][kMaxB];
  // producer-private: routed experts of layer pr_layer, and a window of one sequence's page ids
  int pr_n;
  int pr_expert[kMaxActive];
  int pr_ids[kIdCache];
  // expert-down stages whose weight copy is out but whose activation copy waits for gate/up
  uint32_t pend_dst[kStages], pend_bar[kStages];
  const uint8_t* pend_src[kStages];
  // per-warp LM argmax candidates per token
  float lmw_v[kConsumerWarps][kMaxB];
  int lmw_i[kConsumerWarps][kMaxB];
};
// shared memory: the ring, the tcgen05 A operand of the normalized input, then Misc
constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + kABufBytes + ((int)sizeof(Misc) + 127) / 128 * 128;
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds the sm_103a opt-in limit");
static_assert(offsetof(Misc, red) % 16 == 0 && offsetof(Misc, st_rope) % 16 == 0 &&
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
  int lane;
  uint32_t bar, dst;
  int pos[kMaxB], cpp[kMaxB], nch[kMaxB];  // per step
  int route_layer;
  int id_b, id_p0, id_n;  // m.pr_ids holds the page ids of sequence id_b, pages [id_p0, id_p0 + id_n)
  uint64_t pol;           // L2 policy of every copy

  __device__ Producer(const Params& p_, const TensorMaps& tm_, Misc& m_, Ring r_)
      : p(p_), tm(tm_), m(m_), r(r_), route_layer(-1), id_b(-1), id_p0(0), id_n(0) {
    lane = threadIdx.x & 31;
    pol = policy_evict_first();
#pragma unroll 1
    for (int b = 0; b < kMaxB; ++b) {
      pos[b] = b < p.B ? pos_of(p, b) : 0;
      cpp[b] = b < p.B ? p.chunk_pages[b] : 1;
      nch[b] = b < p.B ? p.n_chunks[b] : 1;
    }
  }

  // the routed experts of layer l, loaded once per layer (lane 0 waits, the warp loads)
  __device__ bool route(int l) {
    if (route_layer == l) return true;
    int fine = 1;
    const Route* rt = p.route + l;
    if (lane == 0) fine = wait_counter(p, CounterMap{p.L, p.nkv, p.B}.route(l));
    if (!__shfl_sync(0xffffffffu, fine, 0)) return false;
    __syncwarp();
    // the count and the whole list in one round of loads (entries past the count are unused)
    const int na = __ldcg(&rt->n_active);
#pragma unroll
    for (int a = lane; a < kMaxActive; a += 32) m.pr_expert[a] = __ldcg(&rt->expert[a]);
    if (lane == 0) m.pr_n = na;
    __syncwarp();
    route_layer = l;
    return true;
  }

  // the next ring slot: lane 0 waits until it is free and arms its barrier with `bytes`
  __device__ bool begin(uint32_t bytes) {
    const uint32_t s = r.it % kStages;
    const uint32_t parity = ((r.it / kStages) & 1u) ^ 1u;
    bar = r.full + 8 * s;
    dst = r.data + s * kStageBytes;
    int fine = 1;
    if (lane == 0) {
      fine = mbar_wait_poll(p, r.empty + 8 * s, parity);
      if (fine) mbar_expect_tx(bar, bytes);
    }
    fine = __shfl_sync(0xffffffffu, fine, 0);
    __syncwarp();
    return fine != 0;
  }
  __device__ void end() { ++r.it; }

  // `rows` rows of row_bytes each, src_stride elements apart in global memory, into one stage
  // (rows row_bytes apart): one copy when the rows are contiguous, else one per row, spread over
  // the lanes (a bulk copy costs about the same to issue whatever its size)
  __device__ bool gemv_rows(const uint16_t* base, int rows, size_t src_stride, int row_bytes) {
    if (!begin((uint32_t)rows * row_bytes)) return false;
    if (src_stride * 2 == (size_t)row_bytes) {
      if (lane == 0) bulk_g2s(dst, base, (uint32_t)rows * row_bytes, bar, pol);
    } else {
#pragma unroll 1
      for (int rr = lane; rr < rows; rr += 32)
        bulk_g2s(dst + (uint32_t)(rr * row_bytes), base + (size_t)rr * src_stride, row_bytes, bar, pol);
    }
    end();
    return true;
  }

  // page ids of sequence b, pages [p0, p0 + n) (n <= kIdCache), into m.pr_ids, one per lane;
  // invalid ids are reported and kept as -1 (their pages are skipped)
  __device__ void fill_ids(int b, int p0, int n) {
    id_b = b;
    id_p0 = p0;
    id_n = n;
#pragma unroll 1
    for (int i = lane; i < n; i += 32) {
      const int pg = p0 + i;
      int v = pg < p.max_pages ? __ldg(&p.block_table[b * p.max_pages + pg]) : -1;
      if (v < 0 || v >= p.num_pages) {
        report(p, MK_ERR_BAD_PAGE, b, pg);
        v = -1;
      }
      m.pr_ids[i] = v;
    }
    __syncwarp();
  }

  // Issues every copy of task t into the ring, in order. Warp-uniform; false once a wait gave up.
  __device__ bool run_task(const Task& t) {
    const int l = t.layer;
    switch (t.op) {  // (combine tasks carry no weights: nothing of theirs goes through the ring)
      case OP_ROUTER:
      case OP_LM: {
        const Geo g = geo_of(p.H);
        const uint16_t* W = t.op == OP_ROUTER ? p.w_router + (size_t)l * p.E * p.H : p.lm_head;
#pragma unroll 1
        for (int r0 = t.a; r0 < t.a + t.b; r0 += g.RS)
          if (!gemv_rows(W + (size_t)r0 * p.H, min(g.RS, t.a + t.b - r0), p.H, p.H * 2)) return false;
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
          for (int i = lane; i < nu; i += 32) {  // unit i: v rows are consecutive; q/k rows are
            const QkvUnit q = qkv_unit(p, u0 + i);  // 4 at row0 and 4 at row0 + d/2 (RoPE pairs)
            const uint32_t d0 = dst + (uint32_t)(i * 8 * g.RST);
            if (q.kind == 2) {
              bulk_g2s(d0, W + (size_t)q.row0 * p.H, 8 * p.H * 2, bar, pol);
            } else {
              bulk_g2s(d0, W + (size_t)q.row0 * p.H, 4 * p.H * 2, bar, pol);
              bulk_g2s(d0 + 4 * g.RST, W + (size_t)(q.row0 + p.d / 2) * p.H, 4 * p.H * 2, bar, pol);
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
#pragma unroll 1
        for (int s0 = ar.cp0; s0 < ar.cp1; s0 += pps) {
          const int np = min(pps, ar.cp1 - s0);
          if (!(id_b == b && s0 >= id_p0 && s0 + np <= id_p0 + id_n)) fill_ids(b, s0, min(kIdCache, ar.cp1 - s0));
          const int* ids = m.pr_ids + (s0 - id_p0);
          if (!begin((uint32_t)np * 2 * halves * 2048)) return false;
          // copy j: page j / 2, K (0) or V (1): one 3D box of the page's 16 rows x all head-dim
          // halves (each half 16 x 128 bytes, 128-byte swizzled). A bulk copy costs about the
          // same to issue whatever its size, so one copy per page and pool instead of one per
          // half. An invalid page (reported when its id was read) loads as zeros: a tile load at
          // an out-of-range row fills the box, so the stage never holds stale bytes.
          if (lane < np * 2) {
            const int i = lane / 2, kv = lane & 1;
            const int id = ids[i];
            const int row = id >= 0 ? ((l * p.num_pages + id) * p.nkv + g) * kPage : -kPage;
            const uint32_t pb = dst + (uint32_t)i * 4096 * halves + (uint32_t)(kv * halves) * 2048;
            tma_3d_g2s(pb, kv ? &tm.v : &tm.k, 0, row, 0, bar, pol);
          }
          end();
        }
        return true;
      }
      case OP_GU: {
        // unit u = (row block j = u / maxa, active expert a = u % maxa): kGuRows gate rows and the
        // matching up rows over the hidden dim; stage s = columns [128 s, 128 s + 128) as two
        // 64-column chunks, each [kGuRows gate rows | kGuRows up rows][128 bytes] (swizzled), the
        // same B layout as a down stage: four tensor copies, lane 2 c + g for chunk c, gate (0) or up (1)
        if (!route(l)) return false;
        const int na = m.pr_n, nst = p.H / kStageK;
        const GuRange gr = gu_range(t, na, p.I / kGuRows);
#pragma unroll 1
        for (int v = gr.v0; v < gr.v1; ++v) {
          const int a = v % na, j = v / na;
          const int grow = ((l * p.E + m.pr_expert[a]) * 2 * p.I) + j * kGuRows;
#pragma unroll 1
          for (int st = 0; st < nst; ++st) {
            if (!begin(kStagePayload)) return false;
            if (lane < 4)  // up rows are I rows after their gate rows
              tma_3d_g2s(dst + (uint32_t)(lane >> 1) * (kStagePayload / 2) + (uint32_t)(lane & 1) * (kGuRows * 128), &tm.gu,
                         0, grow + (lane & 1) * p.I, 2 * st + (lane >> 1), bar, pol);
            end();
          }
        }
        return true;
      }
      case OP_O: {
        // row blocks, each over the column chunks; a stage is one tensor copy of RS rows x KS
        // columns (rows past the task's last one land too and are not read)
        const Geo g = geo_of(p.od);
#pragma unroll 1
        for (int r0 = 0; r0 < t.b; r0 += g.RS)
#pragma unroll 1
          for (int cs = 0; cs < g.NCS; ++cs) {
            if (!begin(kStagePayload)) return false;
            if (lane == 0) tma_3d_g2s(dst, &tm.wo, 0, cs * g.KW, l * p.H + t.a + r0, bar, pol);
            end();
          }
        return true;
      }
      case OP_DOWN: {
        // unit u = (row block rb = u / parts, partial j = u % parts): output rows [kDnRows rb, +kDnRows)
        // over the routed experts of rank j, j + parts, ...; per expert I / kStageK stages, stage s
        // holding the rows' columns [128 s, 128 s + 128) as two swizzled 64-column chunks and,
        // after them, the expert's activations of those columns (two A chunks), so no stage
        // outlives its own products.
        // The weight copy of a stage goes out as soon as its slot is free, before the layer's
        // gate/up is complete; the activation copy (other blocks' gate/up output) only after it.
        // Until then the activation copies wait in a list of at most kStages - 1 stages, so the
        // slot the next stage needs never holds a stage whose copy is still pending.
        if (!route(l)) return false;
        const int na = m.pr_n, parts = p.moe_parts, nst = p.I / kStageK;
        const uint32_t abytes = 2u * (p.B > 4 ? 2048u : 1024u);
        int npend = 0;
        bool gu_done = false;
        auto flush = [&]() -> bool {
          if (!gu_done) {
            int fine = 1;
            if (lane == 0) fine = wait_counter(p, CounterMap{p.L, p.nkv, p.B}.gu(l));
            if (!__shfl_sync(0xffffffffu, fine, 0)) return false;
            // p.hsw was written by the gate/up epilogues' generic stores (other SMs) and published
            // by their release; lane 0's acquire made it visible to the warp, and this fence
            // orders it before the bulk copies below, which read it through the async proxy
            __syncwarp();
            fence_proxy_async_global();
            gu_done = true;
          }
          if (lane == 1)
            for (int i = 0; i < npend; ++i) bulk_g2s(m.pend_dst[i], m.pend_src[i], abytes, m.pend_bar[i], pol);
          npend = 0;
          __syncwarp();
          return true;
        };
#pragma unroll 1
        for (int u = t.a; u < t.a + t.b; ++u) {
          const int rb = u / parts, part = u % parts;
#pragma unroll 1
          for (int a = part; a < na; a += parts) {
            const int row = (l * p.E + m.pr_expert[a]) * p.H + rb * kDnRows;
            const uint8_t* hs = p.hsw + ((size_t)l * kMaxActive + a) * hsw_slot_bytes(p.I);
#pragma unroll 1
            for (int st = 0; st < nst; ++st) {
              if (!gu_done && npend == kStages - 1 && !flush()) return false;
              if (!begin(kStagePayload + abytes)) return false;
              if (lane == 0) tma_3d_g2s(dst, &tm.dn, 0, row, 2 * st, bar, pol);
              const uint8_t* src = hs + (size_t)st * abytes;
              if (gu_done) {
                if (lane == 1) bulk_g2s(dst + kStagePayload, src, abytes, bar, pol);
              } else {
                if (lane == 1) {
                  m.pend_dst[npend] = dst + kStagePayload;
                  m.pend_bar[npend] = bar;
                  m.pend_src[npend] = src;
                }
                ++npend;
              }
              end();
            }
          }
        }
        return npend == 0 || flush();
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

// bf16 pair (lower column in the low half) of the high or the low part of two fp32 values:
// hi = bf16(x), lo = bf16(x - hi), so hi + lo carries about 16 significant bits of x
__device__ __forceinline__ uint32_t pack_part(float x0, float x1, int lo) {
  const uint16_t h0 = f2bf(x0), h1 = f2bf(x1);
  const uint16_t v0 = lo ? f2bf(x0 - bf2f(h0)) : h0;
  const uint16_t v1 = lo ? f2bf(x1 - bf2f(h1)) : h1;
  return (uint32_t)v0 | ((uint32_t)v1 << 16);
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
  static constexpr int AR = NB > 4 ? 4 : 2;  // mma A-fragment registers per k-step
  uint32_t gv;          // GEMV passes done (every consumer warp counts the same sequence)
  int n_layer;          // layer whose normalized input is held in the A buffer (-1 none)
  int route_layer;      // layer whose routing is cached in m.rc_*
  int attn_layer;       // layer of attn_ok
  uint32_t attn_ok;     // KV groups whose attention is known complete in attn_layer
  float lm_best[NB];    // running LM-head argmax of the stages whose epilogue this lane ran
  int lm_idx[NB];
  uint64_t t_start, t_ready;
  // tcgen05 state (used by warp 0, which runs the expert GEMVs): the A operand of the normalized
  // input in shared memory (chunks of kAChunk bytes), the block's tensor memory, and the parity
  // of the next completion of m.tc_acc
  static constexpr uint32_t kAChunk = (NB > 4 ? 2u : 1u) * 1024u;
  static constexpr int kAGroups = NB > 4 ? 2 : 1;
  uint32_t abuf, tmem, tc_phase;
  uint32_t gu_units;  // gate/up units run so far (unit n uses accumulator buffer n & 1)

  __device__ Consumer(const Params& p_, Misc& m_, Ring r_, uint32_t abuf_)
      : p(p_), m(m_), r(r_), cm{p_.L, p_.nkv, p_.B}, ok(true), n_layer(-1), route_layer(-1),
        attn_layer(-1), attn_ok(0), abuf(abuf_), tmem(m_.tmem_base), tc_phase(0), gu_units(0) {
    warp = threadIdx.x / 32;
    lane = threadIdx.x % 32;
    cbar = smem_addr(&m_.cbar);
    cphase = 0;
    gv = 0;
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
  // For a warp that takes only some of a task's stages: stage `it` explicitly, and `n` of the
  // slot's kConsumerWarps arrivals at once. The ring position is moved past the task by the caller.
  // Parity waits stay exact as long as every slot a warp waits on is one whose previous stage it
  // also waited on (or that was consumed before a block barrier the warp passed).
  __device__ const uint8_t* acquire_at(uint32_t it) {
    const uint32_t s = it % kStages, parity = (it / kStages) & 1u;
    if (!mbar_wait(p, r.full + 8 * s, parity)) {
      ok = false;
      return nullptr;
    }
    return reinterpret_cast<const uint8_t*>(__cvta_shared_to_generic(r.data + s * kStageBytes));
  }
  __device__ void release_at(uint32_t it, uint32_t n) {
    __syncwarp();
    if (lane == 0) mbar_arrive_n(r.empty + 8 * (it % kStages), n);
  }
  __device__ uint32_t bmask_all() const { return (1u << p.B) - 1u; }

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

  // Block-wide wait on counter idx. One warp polls and the others wait at the block barrier,
  // which orders their later reads after the poller's acquire: every consumer warp of every SM
  // polling the same line would make that L2 slice a hot spot.
  __device__ bool block_wait(int idx) {
    if (warp == 0) {
      const bool done = warp_wait(p, idx);
      if (lane == 0) m.wait_failed = done ? 0 : 1;
    }
    if (!csync()) return false;
    if (m.wait_failed) ok = false;  // every warp learns that the poller gave up
    return ok;
  }

  // The normalized input of layer l (l == L: the final norm before the LM head), for this
  // lane's 8 columns: x = residual stream (embedding at l = 0), n = x / rms(x) * gain.
  __device__ void load_norm(int l, bool write_x) {
    const Geo g = geo_of(p.H);
    const int ks = warp % g.KW;
    const int col = ks * 256 + lane * 8;
    // batch 5-8, layer input past the embedding: the combine slices wrote the residual and the
    // per-slice square sums; only those are read here
    const bool combined = NB > 4 && l > 0 && p.combine_slices > 0;  // (batch <= 4: compiled out)
    // the gain (static) is read before the wait, off the layer's dependency chain
    const uint16_t* gain = (l < p.L) ? p.norm_gain + (size_t)l * p.H : p.final_gain;
    const uint4 gw = __ldg(reinterpret_cast<const uint4*>(gain + col));
    if (l > 0 && !block_wait(combined ? cm.combine(l) : cm.layer(l - 1))) return;
    // combined: token `warp`'s per-slice square sums (lane j: slices j, j + 32, ...), all in one
    // round of loads right after the wait
    constexpr int kCsPerLane = kMaxCombineSlices / 32;
    float csq[kCsPerLane];
#pragma unroll
    for (int j = 0; j < kCsPerLane; ++j) {
      const int sl = lane + 32 * j;
      csq[j] = (combined && warp < NB && warp < p.B && sl < p.combine_slices)
                   ? __ldcg(&p.css[((size_t)l * kMaxCombineSlices + sl) * kMaxB + warp])
                   : 0.f;
    }
    if (combined) {
      // warp b normalizes token b over every column: its square sum is the slices' sums in slice
      // order within a lane, then a fixed shuffle tree (the same order in every block), so no
      // block barrier sits between the sums and the normalization; tokens past the batch write
      // zero rows of the A operand
      const int b = warp;
      float tot = 0.f;
#pragma unroll
      for (int j = 0; j < kCsPerLane; ++j) tot += csq[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
      const float rinv = 1.0f / sqrtf(tot / (float)p.H + p.eps);
      const bool live = b < p.B;
      const int q = b >> 2, r0 = 2 * (b & 3);
      const float* xrow = p.xs + ((size_t)l * p.B + (live ? b : 0)) * p.H;
#pragma unroll 4
      for (int c = lane * 8; c < p.H; c += 256) {
        float xv[8];
        if (live) load8(xrow + c, xv);
        const uint4 gc = __ldg(reinterpret_cast<const uint4*>(gain + c));
        const float gf[8] = {bf_lo(gc.x), bf_hi(gc.x), bf_lo(gc.y), bf_hi(gc.y),
                             bf_lo(gc.z), bf_hi(gc.z), bf_lo(gc.w), bf_hi(gc.w)};
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (live) split_pack(xv[2 * i] * rinv * gf[2 * i], xv[2 * i + 1] * rinv * gf[2 * i + 1], hw[i], lw[i]);
          else hw[i] = lw[i] = 0u;
        }
        const int u16 = (c & 63) >> 3;
        const uint32_t base = abuf + (uint32_t)(c >> 6) * kAChunk + (uint32_t)q * 1024u;
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + r0 * 128 + ((u16 ^ r0) << 4)), "r"(hw[0]),
                     "r"(hw[1]), "r"(hw[2]), "r"(hw[3]) : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + (r0 + 1) * 128 + ((u16 ^ (r0 + 1)) << 4)),
                     "r"(lw[0]), "r"(lw[1]), "r"(lw[2]), "r"(lw[3]) : "memory");
      }
      fence_proxy_async_smem();  // generic stores that the tensor cores read through the async proxy
      if (!csync()) return;
      n_layer = l;
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
        float a[8], mo[8], mp[8];
        const size_t o = ((size_t)(l - 1) * p.B + b) * p.H + col;
        load8(p.xs + o, x[b]);
        load8(p.attn_out + o, a);
        // the expert branch's output is the sum of its partials, added in part order
        load8(p.moe_part + ((size_t)(l - 1) * kMoeParts * p.B + b) * p.H + col, mo);
        for (int j = 1; j < p.moe_parts; ++j) {
          load8(p.moe_part + (((size_t)(l - 1) * kMoeParts + j) * p.B + b) * p.H + col, mp);
#pragma unroll
          for (int i = 0; i < 8; ++i) mo[i] += mp[i];
        }
        if (write_x && warp < g.KW) {
          float4* dm = reinterpret_cast<float4*>(p.moe_out + o);
          __stcg(dm, make_float4(mo[0], mo[1], mo[2], mo[3]));
          __stcg(dm + 1, make_float4(mo[4], mo[5], mo[6], mo[7]));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) x[b][i] = (x[b][i] + a[i]) + mo[i];
      }
    }
    {
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
    }
    if (!csync()) return;
    const float gf[8] = {bf_lo(gw.x), bf_hi(gw.x), bf_lo(gw.y), bf_hi(gw.y),
                         bf_lo(gw.z), bf_hi(gw.z), bf_lo(gw.w), bf_hi(gw.w)};
    // the normalized input into the A buffer (the GEMVs and the tensor-core products read it there)
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float tot = 0.f;
      for (int k = 0; k < g.KW; ++k) tot += m.norm[k][b];
      const float rinv = 1.0f / sqrtf(tot / (float)p.H + p.eps);
      float xn[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) xn[i] = x[b][i] * rinv * gf[i];
      if (warp < g.KW) {
        // tcgen05 A operand (expert gate/up): row 2 (b % 4) + {hi, lo} of group b / 4, this lane's
        // 8 columns as one 16-byte unit of chunk col / 64 (tokens past the batch are zero rows)
        const int q = b >> 2, r0 = 2 * (b & 3), u16 = (col & 63) >> 3;
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (b < p.B) split_pack(xn[2 * i], xn[2 * i + 1], hw[i], lw[i]);
          else hw[i] = lw[i] = 0u;
        }
        const uint32_t base = abuf + (uint32_t)(col >> 6) * kAChunk + (uint32_t)q * 1024u;
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + r0 * 128 + ((u16 ^ r0) << 4)), "r"(hw[0]),
                     "r"(hw[1]), "r"(hw[2]), "r"(hw[3]) : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + (r0 + 1) * 128 + ((u16 ^ (r0 + 1)) << 4)),
                     "r"(lw[0]), "r"(lw[1]), "r"(lw[2]), "r"(lw[3]) : "memory");
      }
    }
    __syncwarp();
    // the A operand's groups beyond the batch's last token are zero rows too
    if constexpr (NB % 4 != 0) {
      if (warp < g.KW) {
        const int u16 = (col & 63) >> 3;
        const uint32_t base = abuf + (uint32_t)(col >> 6) * kAChunk;
#pragma unroll
        for (int r = 2 * NB; r < 8; ++r)
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(base + r * 128 + ((u16 ^ r) << 4)), "r"(0u) : "memory");
      }
    }
    fence_proxy_async_smem();  // generic stores that the tensor cores read through the async proxy
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

  // ---------------------------------------------------------------- tensor-core GEMV
  // A GEMV pass accumulates one or more stages into per-warp mma accumulators: warp (rg, ks)
  // multiplies rows [8 rg, 8 rg + 8) x columns [256 ks, 256 ks + 256) of each stage (the B
  // operand, 8 rows = n8) by activation fragments (the A operand: up to 8 tokens x hi/lo = m16),
  // in four accumulation chains. post_pass / run_epi then add the warps' k-slices.
  //
  // Column map: a dot product may sum its columns in any order, so the k order inside the mma
  // is permuted to suit the loads. In each 32-column group, lane t (= lane & 3) holds columns
  // [8t, 8t + 8) of its row as one 16-byte word w: k-step 2j of group j takes columns (w.x, w.y)
  // as its (2t, 2t + 1) and (2t + 8, 2t + 9) pairs, k-step 2j + 1 takes (w.z, w.w). The A
  // fragments (af[s][0], af[s][1] = a0, a2) follow the same map. Rows are 2 KS bytes apart
  // (a multiple of 128), so the two rows that share a load phase (g even and odd) read the two
  // 64-byte halves of a 128-byte block in opposite orders and hit distinct banks.

  __device__ __forceinline__ void afrag(const uint32_t (&f)[AR], uint32_t (&a)[4]) const {
    a[0] = f[0];
    a[2] = f[1];
    if constexpr (AR == 4) {
      a[1] = f[2];
      a[3] = f[3];
    } else {
      a[1] = 0u;
      a[3] = 0u;
    }
  }
  // this lane's 16-byte words of column groups 2jj and 2jj + 1 from its row (rowp: the row's
  // slice start + 16 t); odd rows load the two groups in the other order (distinct banks)
  __device__ __forceinline__ void ld_pair(const uint8_t* rowp, int jj, uint4& w0, uint4& w1) const {
    const int odd = (lane >> 2) & 1;
    const uint32_t ra = (uint32_t)__cvta_generic_to_shared(rowp);
    const uint4 x = lds128(ra + (2 * jj + odd) * 64);
    const uint4 y = lds128(ra + (2 * jj + (odd ^ 1)) * 64);
    w0 = odd ? y : x;
    w1 = odd ? x : y;
  }
  __device__ __forceinline__ const uint8_t* b_row(const uint8_t* st, const Geo& g, int rg, int ks) const {
    return st + (size_t)(rg * 8 + (lane >> 2)) * g.RST + ks * 512 + (lane & 3) * 16;
  }
  __device__ __forceinline__ void mma_rows(const uint8_t* st, const Geo& g, int rg, int ks, const uint32_t (&af)[16][AR],
                                           float (&c)[4][4]) const {
    const uint8_t* rowp = b_row(st, g, rg, ks);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint4 w0, w1;
      ld_pair(rowp, jj, w0, w1);
      uint32_t a[4];
      afrag(af[4 * jj], a);
      mma_bf16(c[0], a, w0.x, w0.y);
      afrag(af[4 * jj + 1], a);
      mma_bf16(c[1], a, w0.z, w0.w);
      afrag(af[4 * jj + 2], a);
      mma_bf16(c[2], a, w1.x, w1.y);
      afrag(af[4 * jj + 3], a);
      mma_bf16(c[3], a, w1.z, w1.w);
    }
  }
  // End of a GEMV pass: each warp leaves its partial sums (rows [8 rg, 8 rg + 8) x tokens) in
  // buffer pid % kRedBufs and goes on; returns the pass id. The buffers are handed over by
  // mbarriers: gpart (all 8 warps posted) and gfree (the pass's epilogue warp has read them).
  __device__ uint32_t post_pass(bool active, const float (&c)[4][4]) {
    const uint32_t pid = gv++;
    const int buf = pid % kRedBufs;
    const uint32_t ph = (pid / kRedBufs) & 1u;
    float s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s[i] = (c[0][i] + c[1][i]) + (c[2][i] + c[3][i]);
      s[i] += __shfl_xor_sync(0xffffffffu, s[i], 4);  // hi part (even g) + lo part (odd g)
    }
    if (!mbar_wait_cta(p, smem_addr(&m.gfree[buf]), ph ^ 1u)) {
      ok = false;
      return pid;
    }
    const int g8 = lane >> 2, t4 = lane & 3;
    if (active && !(g8 & 1)) {  // rows 2 t4, 2 t4 + 1 of token g8/2 (and g8/2 + 4)
      float* rw = m.red[buf][warp];
      rw[(2 * t4) * 8 + (g8 >> 1)] = s[0];
      rw[(2 * t4 + 1) * 8 + (g8 >> 1)] = s[1];
      if constexpr (NB > 4) {
        rw[(2 * t4) * 8 + (g8 >> 1) + 4] = s[2];
        rw[(2 * t4 + 1) * 8 + (g8 >> 1) + 4] = s[3];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&m.gpart[buf]));
    return pid;
  }
  // The epilogue of pass pid, in its epilogue warp (pid % 8: the duty rotates): epi(R) with
  // R(row, token) the pass's result, summed over the k-slices from the partials. Callers run it
  // one pass late (after posting the next pass), so it neither waits for the other warps nor
  // holds up the next stage.
  template <typename Epi>
  __device__ void run_epi(uint32_t pid, const Geo& g, Epi&& epi) {
    if (warp != (int)(pid % kConsumerWarps) || !ok) return;
    const int buf = pid % kRedBufs;
    if (!mbar_wait_cta(p, smem_addr(&m.gpart[buf]), (pid / kRedBufs) & 1u)) {
      ok = false;
      return;
    }
    const float(*rb)[64] = m.red[buf];
    const int kw = g.KW;
    auto R = [&](int rr, int b) -> float {
      const int rg = rr >> 3;
      float v = 0.f;
      for (int q = 0; q < kw; ++q) v += rb[rg * kw + q][(rr & 7) * 8 + b];
      return v;
    };
    epi(R);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&m.gfree[buf]));
  }
  // batch 1: as mma_rows, A fragments of the normalized input read from the tcgen05 A operand in
  // shared memory, two k-steps per 16-byte load: lane (g, t) < 8 of k-step pair q (columns
  // [32 q, 32 q + 32) of this warp's slice) takes 16-byte unit 4 (q % 2) + t of row g (0: hi,
  // 1: lo of token 0) of 64-column chunk 4 ks + q / 2, which holds its (a0, a2) registers of
  // k-steps 2 q and 2 q + 1 in the column map above; every other lane's are zero
  // The GEMV core with its A fragments read from the A buffer (the tensor-core A layout: per
  // 64-column chunk, 8-row groups of 4 tokens x {hi, lo}, 128-byte swizzled) instead of registers:
  // mma row g < 8 is row g of token group 0 (tokens 0-3), row g + 8 row g of group 1 (tokens 4-7),
  // the row order of the C fragments' epilogue. One 16-byte load gives a lane its 8 columns of
  // two k-steps; lanes whose rows hold no token load nothing. cbase: the A-buffer chunk of the
  // stage's first column, for inputs wider than one stage.
  __device__ __forceinline__ void mma_rows_sm(const uint8_t* st, const Geo& g, int rg, int ks, float (&c)[4][4],
                                              int cbase = 0) const {
    constexpr int kRows = 2 * (NB < 4 ? NB : 4);  // rows of a token group that hold tokens
    const uint8_t* rowp = b_row(st, g, rg, ks);
    const int r = lane >> 2, t4 = lane & 3;
    const uint32_t fr = abuf + (uint32_t)(cbase + 4 * ks) * kAChunk + r * 128;
    const bool has = r < kRows;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint4 w0, w1;
      ld_pair(rowp, jj, w0, w1);
      const uint32_t bw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int hp = 0; hp < 2; ++hp) {  // k-steps 4 jj + 2 hp and 4 jj + 2 hp + 1
        const int q = 2 * jj + hp, unit = 4 * (q & 1) + t4;
        const uint32_t off = (uint32_t)(q >> 1) * kAChunk + ((unit ^ r) << 4);
        const uint4 f0 = has ? lds128(fr + off) : make_uint4(0u, 0u, 0u, 0u);
        uint4 f1 = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (NB > 4) f1 = lds128(fr + 1024u + off);
        const uint32_t a0[4] = {f0.x, f1.x, f0.y, f1.y}, a1[4] = {f0.z, f1.z, f0.w, f1.w};
        mma_bf16(c[2 * hp], a0, bw[4 * hp], bw[4 * hp + 1]);
        mma_bf16(c[2 * hp + 1], a1, bw[4 * hp + 2], bw[4 * hp + 3]);
      }
    }
  }
  // One stage against the normalized input, as one pass; returns its id.
  __device__ uint32_t norm_pass(const Geo& g) {
    const int rg = warp / g.KW, ks = warp % g.KW;
    const bool active = rg < g.RG;
    float c[4][4] = {};
    const uint8_t* st = acquire();
    if (!st) return gv;
    if (active) mma_rows_sm(st, g, rg, ks, c);
    release();
    return post_pass(active, c);
  }

  __device__ void release_counter(int idx) {
    if (!csync()) return;
    // the barrier orders every consumer's writes before thread 0's gpu-scope release
    if (threadIdx.x == 0) red_release_add(p.counters + (size_t)idx * kCounterStride, 1u);
  }
  // arrival on `idx`; true in every consumer thread of the task that arrived last
  __device__ bool arrive_last(int idx, int count) {
    if (!csync()) return false;
    if (threadIdx.x == 0) {
      const uint32_t old = atom_acq_rel_add(p.counters + (size_t)idx * kCounterStride, 1u);
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
    if (!block_wait(cm.route(l))) return false;
    const Route* rt = p.route + l;
    // the count and the whole tables in one round of loads (rows past the count are unused)
    if (threadIdx.x == 0) m.rc_n = __ldcg(&rt->n_active);
    for (int i = threadIdx.x; i < kMaxActive; i += 256) {
      m.rc_expert[i] = __ldcg(&rt->expert[i]);
      m.rc_mask[i] = __ldcg(&rt->mask[i]);
    }
    for (int i = threadIdx.x; i < kMaxActive * kMaxB / 4; i += 256)
      reinterpret_cast<float4*>(&m.rc_w[0][0])[i] = __ldcg(reinterpret_cast<const float4*>(&rt->w[0][0]) + i);
    if (!csync()) return false;
    route_layer = l;
    return true;
  }
  __device__ bool wait_attn_group(int l, int gg) {
    if (attn_layer != l) { attn_layer = l; attn_ok = 0; }
    if (attn_ok & (1u << gg)) return true;
    if (!warp_wait(p, cm.attn(l, gg))) { ok = false; return false; }
    attn_ok |= 1u << gg;
    return true;
  }

  // hi/lo bf16 planes of an activation value (hi = bf16(v), lo = bf16(v - hi))
  __device__ __forceinline__ void store_hl(uint16_t* hi, size_t plane, float v) const {
    const uint16_t h = f2bf(v);
    hi[0] = h;
    hi[plane] = f2bf(v - bf2f(h));
  }
  // attention output of token b, column col of layer l: fp32 and the GEMV's hi/lo planes
  __device__ __forceinline__ void store_attn(int l, int b, int col, float v) const {
    __stcg(&p.attn_o[((size_t)l * p.B + b) * p.od + col], v);
    store_hl(p.attn_hl + ((size_t)l * 2 * p.B + b) * p.od + col, (size_t)p.B * p.od, v);
  }
  // A fragments from hi/lo bf16 planes (no conversion): token b's row of this warp's slice in
  // plane hl starts at element base + hl * plane + b * row (16-byte aligned); tokens outside
  // bmask are zero. One 16-byte load per 32-column group (the column map above).
  __device__ __forceinline__ void ld_frags_hl(const uint16_t* base, size_t plane, size_t row, uint32_t bmask,
                                              uint32_t (&af)[16][AR]) const {
    const int g8 = lane >> 2, t4 = lane & 3, hl = g8 & 1, b0 = g8 >> 1;
    const bool v0 = (bmask >> b0) & 1u;
    const uint4* s0 = reinterpret_cast<const uint4*>(base + hl * plane + (size_t)b0 * row) + t4;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 w = v0 ? __ldcg(s0 + 4 * j) : make_uint4(0u, 0u, 0u, 0u);
      af[2 * j][0] = w.x; af[2 * j][1] = w.y; af[2 * j + 1][0] = w.z; af[2 * j + 1][1] = w.w;
    }
    if constexpr (AR == 4) {
      const bool v1 = (bmask >> (b0 + 4)) & 1u;
      const uint4* s1 = reinterpret_cast<const uint4*>(base + hl * plane + (size_t)(b0 + 4) * row) + t4;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 w = v1 ? __ldcg(s1 + 4 * j) : make_uint4(0u, 0u, 0u, 0u);
        af[2 * j][2] = w.x; af[2 * j][3] = w.y; af[2 * j + 1][2] = w.z; af[2 * j + 1][3] = w.w;
      }
    }
  }

  // ---------------------------------------------------------------- opcodes

  __device__ void op_router(const Task& t) {
    const int l = t.layer;
    t_ready = gtimer();
    const Geo g = geo_of(p.H);
    auto epi = [&](uint32_t pid, int r0, int rows) {
      run_epi(pid, g, [&](auto&& R) {
        for (int i = lane; i < rows * NB; i += 32) {
          const int rr = i / NB, b = i % NB;
          if (b >= p.B) continue;
          const int e = r0 + rr;
          const float bias = p.router_bias ? p.router_bias[(size_t)l * p.E + e] : 0.f;
          __stcg(&p.rlogits[((size_t)l * p.B + b) * p.E + e], R(rr, b) + bias);
        }
      });
    };
    uint32_t prev = 0;
    int pr0 = -1, prows = 0;
    for (int r0 = t.a; r0 < t.a + t.b && ok; r0 += g.RS) {
      const int rows = min(g.RS, t.a + t.b - r0);
      const uint32_t pid = norm_pass(g);
      if (!ok) return;
      if (pr0 >= 0) epi(prev, pr0, prows);
      prev = pid, pr0 = r0, prows = rows;
    }
    if (pr0 >= 0) epi(prev, pr0, prows);
    if (!ok) return;
    if (arrive_last(cm.router_arrive(l), p.cnt_per_step[cm.router_arrive(l)])) publish_routing(l);
  }

  // Routing of layer l by the block whose router task arrived last, then published with one
  // release of the route counter. Per token (warp b takes token b): top-k (value descending,
  // lower expert id first on ties), softmax over the k selected logits. Then (warp 0) the
  // distinct routed experts in ascending id, each with its token mask and per-token weights.
  // Lane owns experts lane + 32 i. This runs on the critical path of every layer, so each pick
  // is two warp reductions (redux.sync) on an order-preserving integer image of the logit, and
  // the lists are built with ballots, not per-lane loops.
  __device__ static __forceinline__ uint32_t order_key(float x) {
    // +0 and -0 compare equal as logits, so both map to the image of +0
    const uint32_t u = x == 0.f ? 0u : __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  __device__ static __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
  }
  __device__ void publish_routing(int l) {
    constexpr int NE = kMaxExperts / 32;
    const int E = p.E, K = p.topk, B = p.B;
    // every consumer warp of the block that arrived last: warp b routes token b (the tokens are
    // independent, and a token's picks are a serial chain of warp reductions), marking its picks
    // in m.em (bit b per expert); warp 0 then builds the distinct list
    for (int i = threadIdx.x; i < kMaxExperts; i += kConsumerWarps * 32) m.em[i] = 0u;
    if (!csync()) return;
    if (warp < B) {
      const int b = warp;
      uint32_t key[NE];
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        const int e = lane + 32 * i;
        const float x = e < E ? __ldcg(&p.rlogits[((size_t)l * B + b) * E + e]) : -INFINITY;
        // a NaN logit ranks last (with -inf); 0 marks "no expert" and is never picked
        key[i] = e < E ? order_key(x == x ? x : -INFINITY) : 0u;
      }
      float top0 = 0.f, z = 0.f, my_w = 0.f;
      int my_id = 0;
      for (int j = 0; j < K; ++j) {
        uint32_t bk = 0u;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NE; ++i)
          if (key[i] > bk) { bk = key[i]; be = lane + 32 * i; }  // ascending e: ties keep the lower id
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        const int pick = (int)__reduce_min_sync(0xffffffffu, bk == kmax ? (uint32_t)be : 0xffffffffu);
        if ((pick & 31) == lane) {
#pragma unroll
          for (int i = 0; i < NE; ++i)
            if (i == (pick >> 5)) key[i] = 0u;
          atomicOr(&m.em[pick], 1u << b);
        }
        const float bv = key_value(kmax);
        if (j == 0) top0 = bv;
        const float w = expf(bv - top0);
        z += w;
        if (lane == j) { my_id = pick; my_w = w; }
      }
      if (lane < K) { m.ids[b][lane] = my_id; m.wk[b][lane] = my_w / z; }
    }
    if (!csync() || warp != 0) return;
    uint32_t emask[NE];  // bit b: token b picked expert lane + 32 i
#pragma unroll
    for (int i = 0; i < NE; ++i) emask[i] = m.em[lane + 32 * i];
    __syncwarp();
    // the distinct experts in ascending id; m.em[e] holds e's rank for the weight scatter
    Route* rt = p.route + l;
    int na = 0;
#pragma unroll
    for (int i = 0; i < NE; ++i) {
      const uint32_t act = __ballot_sync(0xffffffffu, emask[i] != 0u);
      if (emask[i] != 0u) {
        const int r = na + __popc(act & ((1u << lane) - 1u));
        __stcg(&rt->expert[r], lane + 32 * i);
        __stcg(&rt->mask[r], emask[i]);
        m.em[lane + 32 * i] = (uint32_t)r;
      }
      na += __popc(act);
    }
    static_assert(offsetof(Route, w) % 16 == 0 && sizeof(Route) % 16 == 0, "Route rows must be 16-byte aligned");
    float4* w4 = reinterpret_cast<float4*>(&rt->w[0][0]);
    for (int i = lane; i < na * (kMaxB / 4); i += 32) __stcg(w4 + i, make_float4(0.f, 0.f, 0.f, 0.f));
    __syncwarp();
    for (int i = lane; i < B * K; i += 32) {
      const int b = i / K, j = i % K;
      const int e = m.ids[b][j];
      const float w = m.wk[b][j];
      __stcg(&rt->w[m.em[e]][b], w);
      __stcg(&rt->ids[b][j], e);
      __stcg(&rt->wk[b][j], w);
      __stcg(&p.topk_ids[((size_t)l * B + b) * K + j], e);
      __stcg(&p.topk_w[((size_t)l * B + b) * K + j], w);
    }
    if (lane == 0) __stcg(&rt->n_active, na);
    __syncwarp();
    if (lane == 0) red_release_add(p.counters + (size_t)cm.route(l) * kCounterStride, 1u);
  }

  __device__ void op_qkv(const Task& t) {
    const int l = t.layer;
    t_ready = gtimer();
    const Geo g = geo_of(p.H);
    const int hd = p.d / 2;
    // epilogue: RoPE on k pairs, bf16 K/V append, q stored before RoPE
    auto epi = [&](uint32_t pid, int u0, int nu) {
      run_epi(pid, g, [&](auto&& R) {
      for (int i = lane; i < nu * 8 * NB; i += 32) {
        const int unit = i / (8 * NB), rem = i % (8 * NB), tt = rem / NB, b = rem % NB;
        if (b >= p.B) continue;
        const QkvUnit q = qkv_unit(p, u0 + unit);
        const int pos = m.st_pos[b];
        const int page = q.kind != 0 ? m.st_page[b] : -1;
        if (q.kind != 0 && page < 0 && tt == 0 && unit == 0) report(p, MK_ERR_BAD_PAGE, b, pos);
        if (q.kind == 2) {  // v: 8 consecutive elements
          const int e = 8 * q.j + tt;
          const uint16_t vb = f2bf(R(unit * 8 + tt, b));
          __stcg(&p.vnew[(((size_t)l * p.B + b) * p.nkv + q.head) * p.d + e], bf2f(vb));
          if (page >= 0)
            p.vpool[((((size_t)l * p.num_pages + page) * p.nkv + q.head) * kPage + pos % kPage) * p.d + e] = vb;
          continue;
        }
        if (q.kind == 0) {  // q is stored before RoPE; attention rotates it when it loads it
          const int e = 4 * q.j + (tt & 3) + (tt >= 4 ? hd : 0);
          __stcg(&p.q[(((size_t)l * p.B + b) * p.nq + q.head) * p.d + e], R(unit * 8 + tt, b));
          continue;
        }
        if (tt >= 4) continue;  // k pair (tt, tt + 4) handled by the lower row
        const int pi2 = 4 * q.j + tt;  // pair index in [0, d/2)
        const float a = R(unit * 8 + tt, b), c = R(unit * 8 + tt + 4, b);
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
    };
    uint32_t prev = 0;
    int pu0 = -1, pnu = 0;
    for (int u0 = t.a; u0 < t.a + t.b && ok; u0 += g.RG) {
      const int nu = min(g.RG, t.a + t.b - u0);
      const uint32_t pid = norm_pass(g);
      if (!ok) return;
      if (pu0 >= 0) epi(prev, pu0, pnu);
      prev = pid, pu0 = u0, pnu = nu;
    }
    if (pu0 >= 0) epi(prev, pu0, pnu);
    if (ok) release_counter(cm.qkv(l, t.c));
  }

  // ---------------------------------------------------------------- expert GEMVs on tcgen05
  // Warp 0 runs them: lane 0 issues the products (A: tokens x {hi, lo} from shared memory, 8 rows
  // per group with the descriptor's group stride 0; B: the stage's weight rows; D: fp32 in
  // tensor memory, 128 columns per token group) and frees each ring slot by a commit when its products complete; the warp
  // then reads the accumulators for the epilogue. The other warps step their ring position over
  // the task's stages and wait for warp 0 at the block barrier that ends the task: ring waits
  // test a phase's parity, so a warp must never wait on a slot more than one ring cycle ahead
  // of the stages that are actually in it.


  // Product issue and commits of warp 0 (converged). At batch 8 the elected lane issues from
  // warp-uniform operands; at batch <= 4 lane 0 issues under a branch. Both run the same products
  // from lane 0; measured on the 30B-shaped model, each form is the faster one at its batch size
  // (batch 1 at 8K: 1.995 vs 2.250 ms per step; batch 8: 9.97 vs 10.68 ms).
  __device__ __forceinline__ void tc_issue(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if constexpr (NB > 4) {
      tc_mma_warp(d, a, b, idesc, acc);
    } else {
      if (lane == 0) tc_mma(d, a, b, idesc, acc);
    }
  }
  __device__ __forceinline__ void tc_commit_w0(uint32_t bar) {
    if constexpr (NB > 4) {
      tc_commit_warp(bar);
    } else {
      if (lane == 0) tc_commit(bar);
    }
  }
  // free ring stage `it` once the products issued so far have read it (warp 0, converged)
  __device__ void tc_free(uint32_t it) {
    const uint32_t bar = r.empty + 8 * (it % kStages);
    tc_commit_w0(bar);
    if (lane == 0) mbar_arrive_n(bar, kConsumerWarps - 1);
    __syncwarp();
  }



  // The products of one unit, issued by warp 0 (converged; lane 0 waits and issues, see tc_issue):
  // nst ring stages, each as soon as it lands, then (if `last`) every product completed. A stage
  // holds kStageK columns as two 64-column chunks of 4 k-steps of 16; B = the chunk's 128 weight
  // rows (gate/up: kGuRows gate rows then kGuRows up rows; down: kDnRows output rows), one N = 128
  // product per chunk and k-step. A is the token rows: at batch <= 4 one group of 8 rows (4 tokens
  // x {hi, lo}) that a group stride of 0 repeats in every 8-row group of M; at batch 8 two groups,
  // 1 KB apart, as rows 0-15 of M (the rows after them read whatever follows in shared memory and
  // are never read back). So one product serves all tokens, and the tensor pipe takes 512 cycles
  // per 32 KB stage (measured). A of stage st: the chunks at a_base + st * a_step (a_base 0: the
  // activations riding in the stage after its payload). Gate/up and down share this one loop, so
  // its instructions stay cached from one to the other.
  // Accumulation restarts at the unit's first product unless `accumulate` (down: the next expert
  // of the same partial). D starts at tensor-memory column dcol. With done_bar set, the last
  // products' completion is signalled there by a commit and not awaited. The warp's ring
  // position moves past the stages.
  __device__ bool tc_products(int nst, uint32_t a_base, uint32_t a_step, bool accumulate, bool last,
                              uint32_t dcol = 0, uint32_t done_bar = 0) {
    static_assert(kGuRows * 2 == 128 && kDnRows == 128, "one N = 128 product per chunk");
    constexpr uint32_t idesc = tc_idesc(64, 128);
    constexpr uint32_t kASbo = NB > 4 ? 1024u : 0u;
    int done = 1;
#pragma unroll 1
    for (int st = 0; st < nst; ++st) {
      const uint32_t it = r.it + st;
      int fine = 1;
      if (lane == 0) fine = mbar_wait_spin(p, r.full + 8 * (it % kStages), (it / kStages) & 1u);
      if (!__shfl_sync(0xffffffffu, fine, 0)) {
        done = 0;
        break;
      }
      tc_fence_after();
      const uint32_t wb = r.data + (it % kStages) * kStageBytes;
      const uint32_t ab = a_base ? a_base + (uint32_t)st * a_step : wb + kStagePayload;
      // descriptors built once per stage; offsets go into the 14-bit address field (byte address
      // / 16; shared addresses stay below 256 KB, so the field never carries)
      const uint64_t a0 = tc_sdesc(ab, kASbo), b0 = tc_sdesc(wb, 1024);
#pragma unroll
      for (int c = 0; c < kStageK / kTcK; ++c)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_issue(tmem + dcol, a0 + (uint64_t)((c * kAChunk + k * 32) >> 4),
                   b0 + (uint64_t)((c * 128 * 128 + k * 32) >> 4), idesc,
                   (accumulate || st != 0 || c != 0 || k != 0) ? 1u : 0u);
      tc_free(it);
    }
    if (done && last) {
      if (done_bar) {
        tc_commit_w0(done_bar);
      } else {
        tc_commit_w0(smem_addr(&m.tc_acc));
        int fine = 1;
        if (lane == 0) fine = mbar_wait_spin(p, smem_addr(&m.tc_acc), tc_phase);
        done = __shfl_sync(0xffffffffu, fine, 0);
      }
    }
    r.it += nst;
    if (last && !done_bar) tc_phase ^= 1u;
    tc_fence_after();
    if (!done) ok = false;
    return done != 0;
  }

  __device__ void op_gu(const Task& t) {
    const int l = t.layer;
    if (!load_route(l)) return;
    t_ready = gtimer();
    const int na = m.rc_n, nst = p.H / kStageK;
    const size_t slot_bytes = hsw_slot_bytes(p.I);
    const GuRange gr = gu_range(t, na, p.I / kGuRows);
    // Units alternate between two accumulator buffers, tensor-memory columns [256 b, 256 b + 256):
    // warp 0 issues unit n's products into buffer n & 1 (D of token group q at 128 q: the unit's
    // gate rows, then its up rows) and signals acc_full[n & 1] by a commit without waiting, while
    // warps 4-7 run unit n - 1's epilogue from the other buffer and hand it back through
    // acc_empty. The j-th use of a buffer completes phase j of both its barriers (parity j & 1).
    // Warps 1-7 step their ring position over the stages; the block barrier at the end keeps the
    // ring waits of the next task exact.
    auto epilogue = [&](uint32_t n, int a, int j) {
      // D row r holds token 4 (r / 8) + (r % 8) / 2, part r % 2 (hi, lo). At batch <= 4 the A
      // group stride 0 repeats rows 0-7 in every 16-lane group of D, so warp w (4-7) reads them
      // from its own lane quarter (tensor-memory lanes 32 (w - 4) + r) and takes gate/up columns
      // [16 (w - 4), +16); at batch 8 rows 0-15 sit in lane quarter 0 only, and warp 4 takes all
      // 64 columns (acc_empty then counts one arrival per phase instead of four).
      constexpr int kRows = NB > 4 ? 16 : 8;
      const uint32_t buf = n & 1u, wq = (uint32_t)warp & 3u;
      if (NB > 4 && wq != 0) return;
      int fine = 1;
      if (lane == 0) fine = mbar_wait_spin(p, smem_addr(&m.acc_full[buf]), (n >> 1) & 1u);
      if (!__shfl_sync(0xffffffffu, fine, 0)) {
        ok = false;
        return;
      }
      tc_fence_after();
      uint8_t* hs = p.hsw + ((size_t)l * kMaxActive + a) * slot_bytes;
      const uint32_t tq = tmem + buf * 256u + ((32u * wq) << 16);
      const int q = (lane >> 3) & 1, rr = lane & 7, tok = 4 * q + (rr >> 1), hl = rr & 1;
      const bool row_ok = lane < kRows && tok < p.B;
      const float wgt = row_ok ? m.rc_w[a][tok] : 0.f;
      const int c0 = NB > 4 ? 0 : 16 * (int)wq, c1 = NB > 4 ? kGuRows : c0 + 16;
#pragma unroll 1
      for (int i0 = c0; i0 < c1; i0 += 16) {
        uint32_t gv_[16], uv[16];
        tc_ld16(tq + i0, gv_);
        tc_ld16(tq + kGuRows + i0, uv);
        // hi + lo of each gate and up value (lanes 2 t and 2 t + 1 hold the two parts of token
        // t); lanes past the token rows hold tensor-memory words no product wrote
        float gs[16], us[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          gs[c] = lane < kRows ? __uint_as_float(gv_[c]) : 0.f;
          us[c] = lane < kRows ? __uint_as_float(uv[c]) : 0.f;
          gs[c] += __shfl_xor_sync(0xffffffffu, gs[c], 1);
          us[c] += __shfl_xor_sync(0xffffffffu, us[c], 1);
        }
        if (row_ok) {
          uint32_t packed[8];
#pragma unroll
          for (int c = 0; c < 16; c += 2) {
            float hv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e)  // SiLU(g) = g / (1 + e^-g), times up and the routing weight
              hv[e] = __fdividef(gs[c + e], 1.0f + __expf(-gs[c + e])) * us[c + e] * wgt;
            uint32_t hi, lo;
            split_pack(hv[0], hv[1], hi, lo);
            packed[c / 2] = hl ? lo : hi;
          }
          // columns kc = j kGuRows + i0 + 0..15: chunk kc / 64, 16-byte units (kc % 64) / 8 + 0..1
          const int kc = j * kGuRows + i0;
          uint8_t* rowp = hs + (size_t)(kc >> 6) * kAChunk + q * 1024 + rr * 128;
#pragma unroll
          for (int m4 = 0; m4 < 2; ++m4) {
            const int u16 = ((kc & 63) >> 3) + m4;
            __stcg(reinterpret_cast<uint4*>(rowp + ((u16 ^ rr) << 4)),
                   make_uint4(packed[4 * m4], packed[4 * m4 + 1], packed[4 * m4 + 2], packed[4 * m4 + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&m.acc_empty[buf]));
    };
    uint32_t n = gu_units;
    int pa = -1, pj = 0;
#pragma unroll 1
    for (int v = gr.v0; v < gr.v1 && ok; ++v) {
      const int a = v % na, j = v / na;
      if (warp == 0) {
        // buffer n & 1 is free once unit n - 2's epilogue has read it
        int fine = 1;
        if (lane == 0 && n >= 2) fine = mbar_wait_spin(p, smem_addr(&m.acc_empty[n & 1u]), ((n >> 1) & 1u) ^ 1u);
        if (!__shfl_sync(0xffffffffu, fine, 0)) {
          ok = false;
          return;
        }
        tc_fence_after();
        tc_products(nst, abuf, 2 * kAChunk, false, true, (n & 1u) * 256u, smem_addr(&m.acc_full[n & 1u]));
      } else {
        r.it += nst;
      }
      if (warp >= 4 && pa >= 0) epilogue(n - 1, pa, pj);
      pa = a, pj = j;
      ++n;
    }
    if (warp >= 4 && pa >= 0 && ok) epilogue(n - 1, pa, pj);
    gu_units = n;
    if (!csync()) return;
    release_counter(cm.gu(l));
  }

  __device__ void op_o(const Task& t) {
    const int l = t.layer;
    const Geo g = geo_of(p.od);
    const int rg = warp / g.KW, ks = warp % g.KW;
    const bool active = rg < g.RG;
    const int gw = p.group * p.d;  // columns per KV group
    const uint16_t* base = p.attn_hl + (size_t)l * 2 * p.B * p.od + ks * 256;
    const size_t plane = (size_t)p.B * p.od;
    // waits for the KV groups behind chunk cs's columns of this warp's slice
    auto wait_chunk = [&](int cs) -> bool {
      const int c0 = cs * g.KS + ks * 256;
      for (int gg = c0 / gw; gg <= (c0 + 255) / gw; ++gg)
        if (!wait_attn_group(l, gg)) return false;
      return true;
    };
    auto epi = [&](uint32_t pid, int r0, int rows) {
      run_epi(pid, g, [&](auto&& R) {
        for (int i = lane; i < rows * NB; i += 32) {
          const int rr = i / NB, b = i % NB;
          if (b < p.B) __stcg(&p.attn_out[((size_t)l * p.B + b) * p.H + t.a + r0 + rr], R(rr, b));
        }
      });
    };
    t_ready = 0;
    if (NB == 1 && p.od / 64 * kAChunk <= kABufBytes) {
      // Batch 1: the attention output (hi, lo) goes into the A buffer once, as rows 0 and 1 of its
      // 64-column chunks (the layout mma_rows_nf1 reads). Nothing in the layer reads the buffer
      // after attention, and the next layer's norm rebuilds it.
      for (int gg = 0; gg < p.nkv; ++gg)
        if (!wait_attn_group(l, gg)) return;
      t_ready = gtimer();
      const uint16_t* src = p.attn_hl + (size_t)l * 2 * p.od;  // [hi | lo][od] of token 0
      for (int i = threadIdx.x; i < p.od / 4; i += kConsumerWarps * 32) {
        const int hl = i / (p.od / 8), col = (i % (p.od / 8)) * 8;
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(src + (size_t)hl * p.od + col));
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(abuf + (uint32_t)(col >> 6) * kAChunk + hl * 128 +
                                                                      ((((col & 63) >> 3) ^ hl) << 4)),
                     "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
      }
      n_layer = -1;
      if (!csync()) return;
      uint32_t prev = 0;
      int pr0 = -1, prows = 0;
      for (int r0 = 0; r0 < t.b && ok; r0 += g.RS) {
        float c[4][4] = {};
        for (int cs = 0; cs < g.NCS; ++cs) {
          const uint8_t* st = acquire();
          if (!st) return;
          if (active) mma_rows_sm(st, g, rg, ks, c, cs * (g.KS / 64));
          release();
        }
        const uint32_t pid = post_pass(active, c);
        if (!ok) return;
        if (pr0 >= 0) epi(prev, pr0, prows);
        prev = pid, pr0 = r0, prows = min(g.RS, t.b - r0);
      }
      if (pr0 >= 0) epi(prev, pr0, prows);
      if (ok) release_counter(cm.layer(l));
      return;
    }
    // At batch <= 4 with at most two column chunks, both chunks' fragments are loaded once and
    // reused by every row block of the task; otherwise (one block per task) chunk by chunk.
    constexpr bool kHold = AR == 2;
    const bool hold = kHold && g.NCS <= 2;
    uint32_t af[kHold ? 2 : 1][16][AR];
    if (hold && active) {
      for (int cs = 0; cs < g.NCS; ++cs)
        if (!wait_chunk(cs)) return;
      ld_frags_hl(base, plane, p.od, bmask_all(), af[0]);
      if (g.NCS > 1) ld_frags_hl(base + g.KS, plane, p.od, bmask_all(), af[kHold ? 1 : 0]);
    }
    uint32_t prev = 0;
    int pr0 = -1, prows = 0;
    for (int r0 = 0; r0 < t.b && ok; r0 += g.RS) {
      float c[4][4] = {};
      for (int cs = 0; cs < g.NCS; ++cs) {
        if (!hold && active) {
          if (!wait_chunk(cs)) return;
          ld_frags_hl(base + cs * g.KS, plane, p.od, bmask_all(), af[0]);
        }
        if (!t_ready) t_ready = gtimer();
        const uint8_t* st = acquire();
        if (!st) return;
        if (active) mma_rows(st, g, rg, ks, af[hold ? (cs & 1) : 0], c);
        release();
      }
      const uint32_t pid = post_pass(active, c);
      if (!ok) return;
      if (pr0 >= 0) epi(prev, pr0, prows);
      prev = pid, pr0 = r0, prows = min(g.RS, t.b - r0);
    }
    if (pr0 >= 0) epi(prev, pr0, prows);
    if (ok) release_counter(cm.layer(l));
  }

  __device__ void op_down(const Task& t) {
    const int l = t.layer;
    if (!load_route(l)) return;
    t_ready = gtimer();
    const int na = m.rc_n, parts = p.moe_parts, nst = p.I / kStageK;
#pragma unroll 1
    for (int u = t.a; u < t.a + t.b; ++u) {
      const int rb = u / parts, part = u % parts;
      // partial `part` of output rows [kDnRows rb, +kDnRows): the routed experts of rank part,
      // part + parts, ..., accumulated in rank order; stage st carries the expert's weight rows'
      // columns [128 st, +128) (B) and, after them in the slot, its activations of those columns (A)
      int ne = 0;
      for (int a = part; a < na; a += parts) ++ne;
      if (warp == 0) {
        int i = 0;
        for (int a = part; a < na && ok; a += parts, ++i) tc_products(nst, 0, 0, i > 0, i + 1 == ne);
      } else {
        r.it += ne * nst;
      }
      tc_fence_before();
      if (!csync() || !ok) return;
      tc_fence_after();
      // epilogue (D rows as in op_gu): at batch <= 4 warps 0-3, each from its own tensor-memory
      // lane quarter, output columns [32 w, 32 w + 32); at batch 8 warp 0 (rows 0-15 in lane
      // quarter 0) all kDnRows columns. Zero when no routed expert falls in this partial.
      constexpr int kRows = NB > 4 ? 16 : 8;
      if (NB > 4 ? warp == 0 : warp < 4) {
        const uint32_t tq = tmem + ((uint32_t)(32 * warp) << 16);
        const int q = (lane >> 3) & 1, rr = lane & 7, hl = rr & 1, tok = 4 * q + (rr >> 1);
        float* dst = p.moe_part + (((size_t)l * kMoeParts + part) * p.B + tok) * p.H + rb * kDnRows;
        const int c0 = NB > 4 ? 0 : 32 * warp, c1 = NB > 4 ? kDnRows : c0 + 32;
#pragma unroll 1
        for (int i0 = c0; i0 < c1; i0 += 16) {
          uint32_t v[16];
          if (ne > 0) tc_ld16(tq + i0, v);
          float o[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            float x = (ne == 0 || lane >= kRows) ? 0.f : __uint_as_float(v[c]);
            x += __shfl_xor_sync(0xffffffffu, x, 1);  // hi + lo
            o[c] = x;
          }
          if (lane < kRows && hl == 0 && tok < p.B)
#pragma unroll
            for (int c = 0; c < 16; c += 4)
              __stcg(reinterpret_cast<float4*>(dst + i0 + c), make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]));
        }
      }
      // the accumulator is read before warp 0 issues the next products into it (the next unit's,
      // or those of the block's next tensor-core task)
      tc_fence_before();
      if (!csync()) return;
    }
    release_counter(cm.layer(l));
  }

  __device__ void op_lm(const Task& t) {
    t_ready = gtimer();
    const Geo g = geo_of(p.H);
    auto epi = [&](uint32_t pid, int r0, int rows) {
      run_epi(pid, g, [&](auto&& R) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int e = lane; e < rows * NB; e += 32) {  // e % NB == lane % NB since 32 % NB == 0
          const int rr = e / NB, b = e % NB;
          const float v = R(rr, b);
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
    };
    uint32_t prev = 0;
    int pr0 = -1, prows = 0;
    for (int r0 = t.a; r0 < t.a + t.b && ok; r0 += g.RS) {
      const int rows = min(g.RS, t.a + t.b - r0);
      const uint32_t pid = norm_pass(g);
      if (!ok) return;
      if (pr0 >= 0) epi(prev, pr0, prows);
      prev = pid, pr0 = r0, prows = rows;
    }
    if (pr0 >= 0) epi(prev, pr0, prows);
    if (!(t.flags & TF_LAST_LM) || !ok) return;
    // lanes < NB of every warp hold that warp's candidate for token lane; combine over warps
    if (lane < NB) {
      m.lmw_v[warp][lane] = lm_best[0];
      m.lmw_i[warp][lane] = lm_idx[0];
    }
    if (!csync()) return;
    if (threadIdx.x < p.B) {  // warp 0, lane b: token b
      const int b = threadIdx.x;
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int w = 0; w < kConsumerWarps; ++w)
        if (m.lmw_v[w][b] > bv || (m.lmw_v[w][b] == bv && m.lmw_i[w][b] < bi)) { bv = m.lmw_v[w][b]; bi = m.lmw_i[w][b]; }
      __stcg(&p.lm_best_v[t.c * kMaxB + b], bv);
      __stcg(&p.lm_best_i[t.c * kMaxB + b], bi);
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

  // Paged GQA attention of one (sequence b, KV group g, chunk). The G <= 8 query heads of the
  // group are the 16 rows of an mma A operand: rows 0..7 hold the bf16 "hi" part of q and rows
  // 8..15 its rounding residual, so S = q K^T comes out at ~fp32 accuracy; P is split the same
  // way for P V. K/V tiles arrive 128B-swizzled from the tensor maps (conflict-free ldmatrix).
  // One attention chunk; KS = head_dim / 16 (mma k-steps over the head dim: 8 at d = 128, 4 at
  // d = 64) is a template parameter so that every loop and register index below is static.
  template <int KS>
  __device__ void attn_chunk(const Task& t) {
    constexpr int halves = KS / 4, pps = kStagePayload / (4096 * halves);
    const int l = t.layer, b = t.a, g = t.b;
    if (!block_wait(cm.qkv(l, g))) return;
    t_ready = gtimer();
    const AttnRange ar = attn_range(m.st_pos[b], m.st_cpp[b], m.st_nch[b], t.c);
    // warp (pi, sp) takes page pi of every stage s with s % npar == sp, over the whole head dim
    // (2 stage parities at d = 128, 1 at d = 64), so no two warps compute the same scores
    constexpr int npar = kConsumerWarps / pps;
    const int pi = warp % pps, sp = warp / pps;
    const int head = lane >> 2, tig = lane & 3;
    const float qscale = rsqrtf((float)p.d) * 1.4426950408889634f;  // scores in log2 units
    uint32_t qa[KS][4];
    {
      // this lane's q elements straight from global memory (one round of 8-byte loads); q
      // arrives before RoPE: element d pairs with d + d/2, which this lane also holds (k-step
      // kk + ksteps/2), so the rotation happens here in registers
      const bool hv = head < p.group;
      const float* qh = p.q + (((size_t)l * p.B + b) * p.nq + g * p.group + (hv ? head : 0)) * p.d;
      float x[KS][4];
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const int d0 = kk * 16 + tig * 2;
        const float2 lo = hv ? __ldcg(reinterpret_cast<const float2*>(qh + d0)) : make_float2(0.f, 0.f);
        const float2 hi = hv ? __ldcg(reinterpret_cast<const float2*>(qh + d0 + 8)) : make_float2(0.f, 0.f);
        x[kk][0] = lo.x; x[kk][1] = lo.y; x[kk][2] = hi.x; x[kk][3] = hi.y;
      }
      constexpr int half = KS / 2;
#pragma unroll
      for (int kk = 0; kk < half; ++kk) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d0 = kk * 16 + tig * 2 + (e & 1) + (e >> 1) * 8;  // < d/2
          const float2 cs = m.st_rope[b][d0];
          const float lo = x[kk][e], hi = x[kk + half][e];
          x[kk][e] = lo * cs.x - hi * cs.y;
          x[kk + half][e] = lo * cs.y + hi * cs.x;
        }
      }
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        split_pack(x[kk][0] * qscale, x[kk][1] * qscale, qa[kk][0], qa[kk][1]);
        split_pack(x[kk][2] * qscale, x[kk][3] * qscale, qa[kk][2], qa[kk][3]);
      }
    }
    float mrun = -INFINITY, lsum = 0.f;
    float oacc[2 * KS][4];
#pragma unroll
    for (int i = 0; i < 2 * KS; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) oacc[i][j] = 0.f;

    // Warp (pi, sp) waits only on the stages of its parity sp and gives each slot its group's
    // share of the arrivals. With 4 slots and 2 parities, stages s and s + 4 of one slot have the
    // same parity, so each slot is waited on by one group of warps only (and the block barrier of
    // the q load precedes the loop), which keeps every parity wait exact.
    static_assert(kStages % npar == 0, "a ring slot must serve stages of one parity");
    const int nst = (ar.cp1 - ar.cp0 + pps - 1) / pps;
    const uint32_t it0 = r.it;
    for (int s = sp; s < nst; s += npar) {
      const uint8_t* st = acquire_at(it0 + s);
      if (!st) return;
      const int page = ar.cp0 + s * pps + pi;
      if (page < ar.cp1) {
        const uint32_t kt = smem_addr(st) + (uint32_t)pi * 4096 * halves;
        const uint32_t vt = kt + (uint32_t)halves * 2048;
        // Rows of the sequence's last page at or past the new token's position are masked out of
        // the scores, but their V bytes still enter P V (with weight 0), and 0 * NaN is NaN: the
        // cache there holds whatever the caller left. This warp alone reads this page, so it
        // zeroes those V rows (whole 128-byte rows: the swizzle only permutes within a row).
        const int live = ar.pos_end - page * kPage;
        if (live < kPage) {
          const int nz = (kPage - max(live, 0)) * 8 * halves;  // 16-byte words to clear
          for (int i = lane; i < nz; i += 32) {
            const int h = i / ((kPage - max(live, 0)) * 8), rem = i % ((kPage - max(live, 0)) * 8);
            const int row = max(live, 0) + rem / 8;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vt + h * 2048 + row * 128 + (rem % 8) * 16),
                         "r"(0u)
                         : "memory");
          }
          fence_proxy_async_smem();  // generic stores into a ring slot the producer refills later
          __syncwarp();
        }
        float sc[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) sc[i][j] = 0.f;
        const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int prow = (mi >> 1) * 8 + rr;           // position within the page
          const int chunk = 2 * kk + (mi & 1);          // 16-byte chunk of the head dim
          const uint32_t addr = kt + (chunk >> 3) * 2048 + prow * 128 + (((chunk & 7) ^ (prow & 7)) << 4);
          uint32_t bk[4];
          ldsm_x4(addr, bk);
          mma_bf16(sc[0], qa[kk], bk[0], bk[1]);
          mma_bf16(sc[1], qa[kk], bk[2], bk[3]);
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
          for (int i = 0; i < 2 * KS; ++i)
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
          for (int c2 = 0; c2 < KS; ++c2) {  // two 8-wide d tiles per ldmatrix.x4.trans
            const int chunk = c2 * 2 + (mi >> 1);
            const int prow = (mi & 1) * 8 + rr;
            const uint32_t addr = vt + (chunk >> 3) * 2048 + prow * 128 + (((chunk & 7) ^ (prow & 7)) << 4);
            uint32_t bv[4];
            ldsm_x4_t(addr, bv);
            mma_bf16(oacc[c2 * 2], pa, bv[0], bv[1]);
            mma_bf16(oacc[c2 * 2 + 1], pa, bv[2], bv[3]);
          }
        }
      }
      release_at(it0 + s, npar);
    }
    r.it = it0 + nst;
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);

    // merge the 8 warps (disjoint pages) in one round through the A buffer: within a layer no
    // task after attention reads the normalized input (down carries its activations in the ring,
    // O-proj reads the attention output), and the next task that needs it rebuilds it
    const size_t pidx = (((size_t)l * p.B + b) * p.nkv + g) * p.max_chunks + t.c;
    float* part = p.apart + pidx * (16 + 8 * (size_t)p.d);
    if (nst > 0) {
      constexpr int d = 16 * KS, q4 = d / 4, kW = 16 + 8 * d;  // per warp: m[8], l[8], O[8][d]
      static_assert(kConsumerWarps * kW * 4 <= kABufBytes, "merge scratch exceeds the A buffer");
      float* scr = reinterpret_cast<float*>(__cvta_shared_to_generic(abuf));
      float* mine = scr + warp * kW;
      // (every earlier reader of the buffer finished before the block barrier that ended its task)
      if (tig == 0) { mine[head] = mrun; mine[8 + head] = lsum; }
#pragma unroll
      for (int nt = 0; nt < 2 * KS; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) mine[16 + head * d + nt * 8 + tig * 2 + e] = oacc[nt][e] + oacc[nt][e + 2];
      n_layer = -1;
      if (!csync()) return;
      if (threadIdx.x < 8 * q4) {  // head h, dims [dd, dd + 4)
        const int h = threadIdx.x / q4, dd = 4 * (threadIdx.x % q4);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, scr[w * kW + h]);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY)
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = scr[w * kW + h];
            const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
            L += scr[w * kW + 8 + h] * f;
            const float4 v = *reinterpret_cast<const float4*>(scr + w * kW + 16 + h * d + dd);
            O.x = fmaf(v.x, f, O.x);
            O.y = fmaf(v.y, f, O.y);
            O.z = fmaf(v.z, f, O.z);
            O.w = fmaf(v.w, f, O.w);
          }
        if (dd == 0) { __stcg(part + h, M); __stcg(part + 8 + h, L); }
        __stcg(reinterpret_cast<float4*>(part + 16 + h * d + dd), O);
      }
    } else {
      for (int i = threadIdx.x; i < 16 + 8 * p.d; i += 256) __stcg(part + i, i < 8 ? -INFINITY : 0.f);
    }
    const int arr = cm.attn_arrive(l, b, g);
    if (!arrive_last(arr, m.st_nch[b])) return;

    // combine the chunks of (b, g) with the new token (position pos, read from knew / vnew)
    const int nch = m.st_nch[b];
    const float* pbase = p.apart + (((size_t)l * p.B + b) * p.nkv + g) * p.max_chunks * (16 + 8 * (size_t)p.d);
    const size_t cstride = 16 + 8 * (size_t)p.d;
    const float* vn = p.vnew + (((size_t)l * p.B + b) * p.nkv + g) * p.d;
    const float* kn = p.knew + (((size_t)l * p.B + b) * p.nkv + g) * p.d;
    const int hd = p.d / 2;
    if (nch <= 64) {
      // Warp h combines head h on its own, with no block barrier: one round of loads brings the
      // new token's q and k, every chunk's max and sum (lane j: chunks j and j + 32) and the
      // first 16 chunks' outputs of the lane's 4 columns; the scale factors reach the other
      // lanes by shuffles. (group <= 8: one head per warp at most)
      const int h = warp;
      if (h < p.group) {
        const float* qh = p.q + (((size_t)l * p.B + b) * p.nq + g * p.group + h) * p.d;
        const int dd = 4 * lane;
        const bool has = dd < p.d;
        const float* src = pbase + 16 + h * p.d + dd;
        float4 v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          v[j] = (j < nch && has) ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)j * cstride))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        const float m0 = lane < nch ? __ldcg(pbase + (size_t)lane * cstride + h) : -INFINITY;
        const float l0 = lane < nch ? __ldcg(pbase + (size_t)lane * cstride + 8 + h) : 0.f;
        const float m1 = lane + 32 < nch ? __ldcg(pbase + (size_t)(lane + 32) * cstride + h) : -INFINITY;
        const float l1 = lane + 32 < nch ? __ldcg(pbase + (size_t)(lane + 32) * cstride + 8 + h) : 0.f;
        const float4 vv = has ? __ldcg(reinterpret_cast<const float4*>(vn + dd)) : make_float4(0.f, 0.f, 0.f, 0.f);
        float s = 0.f;
        for (int i = lane; i < hd; i += 32) {  // q before RoPE: rotate pair (i, i + d/2)
          const float2 cs = m.st_rope[b][i];
          const float q0 = __ldcg(qh + i), q1 = __ldcg(qh + i + hd);
          s = fmaf(q0 * cs.x - q1 * cs.y, __ldcg(kn + i), s);
          s = fmaf(q0 * cs.y + q1 * cs.x, __ldcg(kn + i + hd), s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float sn = s * qscale;
        float M = fmaxf(sn, fmaxf(m0, m1));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float fn = exp2f(sn - M);
        const float f0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M);
        const float f1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
        float L = l0 * f0 + l1 * f1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        L += fn;
        float4 O = make_float4(fn * vv.x, fn * vv.y, fn * vv.z, fn * vv.w);
        for (int c0 = 0; c0 < nch; c0 += 16) {
          if (c0 > 0)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              v[j] = (c0 + j < nch && has) ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)(c0 + j) * cstride))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
          const float fsrc = c0 < 32 ? f0 : f1;  // chunks [c0, c0 + 16) lie in one half
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float f = __shfl_sync(0xffffffffu, fsrc, (c0 + j) & 31);
            O.x = fmaf(v[j].x, f, O.x);
            O.y = fmaf(v[j].y, f, O.y);
            O.z = fmaf(v[j].z, f, O.z);
            O.w = fmaf(v[j].w, f, O.w);
          }
        }
        if (has) {
          const float inv = 1.0f / L;
          const int col = (g * p.group + h) * p.d + dd;
          store_attn(l, b, col, O.x * inv);
          store_attn(l, b, col + 1, O.y * inv);
          store_attn(l, b, col + 2, O.z * inv);
          store_attn(l, b, col + 3, O.w * inv);
        }
      }
    } else {
      // many chunks: the new token's scores first (warp h: head h), then one thread per output
      float* sc = &m.red[2][0][0];
      if (warp < p.group) {
        const float* qh = p.q + (((size_t)l * p.B + b) * p.nq + g * p.group + warp) * p.d;
        float s = 0.f;
        for (int i = lane; i < hd; i += 32) {
          const float2 cs = m.st_rope[b][i];
          const float q0 = __ldcg(qh + i), q1 = __ldcg(qh + i + hd);
          s = fmaf(q0 * cs.x - q1 * cs.y, __ldcg(kn + i), s);
          s = fmaf(q0 * cs.y + q1 * cs.x, __ldcg(kn + i + hd), s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) sc[warp] = s * qscale;
      }
      if (!csync()) return;
      for (int i = threadIdx.x; i < p.group * p.d; i += 256) {
        const int h = i / p.d, dd = i % p.d;
        const float sn = sc[h];
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
        store_attn(l, b, (g * p.group + h) * p.d + dd, O / L);
      }
    }
    release_counter(cm.attn(l, g));
  }

  // Combine slice t.a of layer t.layer's input (batch 5-8): for its kCombineCols columns and every
  // token, the residual x = (x + attn_out) + (sum of the expert partials in part order) of the
  // previous layer, stored once, and each token's square sum over those columns. Warp 0: lane
  // (b, q) takes token b = lane / 4, columns [c0 + 4 q, + 4).
  __device__ void op_combine(const Task& t) {
    const int l = t.layer, c0 = t.a * kCombineCols;
    if (!block_wait(cm.layer(l - 1))) return;
    t_ready = gtimer();
    if (warp == 0) {
      const int b = lane >> 2, c = c0 + 4 * (lane & 3);
      float sq = 0.f;
      if (b < p.B) {
        const size_t o = ((size_t)(l - 1) * p.B + b) * p.H + c;
        float4 x = __ldcg(reinterpret_cast<const float4*>(p.xs + o));
        const float4 a = __ldcg(reinterpret_cast<const float4*>(p.attn_out + o));
        float4 mo = __ldcg(reinterpret_cast<const float4*>(p.moe_part + ((size_t)(l - 1) * kMoeParts * p.B + b) * p.H + c));
        float4 mp[kMoeParts - 1];
#pragma unroll
        for (int j = 1; j < kMoeParts; ++j)
          if (j < p.moe_parts)
            mp[j - 1] = __ldcg(reinterpret_cast<const float4*>(p.moe_part + (((size_t)(l - 1) * kMoeParts + j) * p.B + b) * p.H + c));
#pragma unroll
        for (int j = 1; j < kMoeParts; ++j)
          if (j < p.moe_parts) {
            mo.x += mp[j - 1].x; mo.y += mp[j - 1].y; mo.z += mp[j - 1].z; mo.w += mp[j - 1].w;
          }
        __stcg(reinterpret_cast<float4*>(p.moe_out + o), mo);
        x.x = (x.x + a.x) + mo.x; x.y = (x.y + a.y) + mo.y; x.z = (x.z + a.z) + mo.z; x.w = (x.w + a.w) + mo.w;
        __stcg(reinterpret_cast<float4*>(p.xs + ((size_t)l * p.B + b) * p.H + c), x);
        sq = fmaf(x.x, x.x, sq); sq = fmaf(x.y, x.y, sq); sq = fmaf(x.z, x.z, sq); sq = fmaf(x.w, x.w, sq);
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sq += __shfl_xor_sync(0xffffffffu, sq, 2);
      if ((lane & 3) == 0 && b < p.B) __stcg(&p.css[((size_t)l * kMaxCombineSlices + t.a) * kMaxB + b], sq);
    }
    release_counter(cm.combine(l));
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
    switch (t.op) {
      case OP_ROUTER: op_router(t); break;
      case OP_QKV: op_qkv(t); break;
      case OP_ATTN:
        if (p.d == 128) attn_chunk<8>(t);
        else attn_chunk<4>(t);
        break;
      case OP_GU: op_gu(t); break;
      case OP_O: op_o(t); break;
      case OP_DOWN: op_down(t); break;
      case OP_LM: op_lm(t); break;
      case OP_COMBINE:
        if constexpr (NB > 4) op_combine(t);  // only batch 5-8 plans hold combine tasks
        break;
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
  Misc& misc = *reinterpret_cast<Misc*>(base + kStages * kStageBytes + kABufBytes);
  if (threadIdx.x < 32) {  // warp 0 takes the block's tensor memory (one block per SM, so it is free)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&misc.tmem_base)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&misc.full[s]), 1);
      mbar_init(smem_addr(&misc.empty[s]), kConsumerWarps);
    }
    mbar_init(smem_addr(&misc.cbar), kConsumerWarps);
    mbar_init(smem_addr(&misc.tc_acc), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&misc.acc_full[b]), 1);
      mbar_init(smem_addr(&misc.acc_empty[b]), NB > 4 ? 1 : 4);  // the epilogue's reading warps
    }
    for (int i = 0; i < kRedBufs; ++i) {
      mbar_init(smem_addr(&misc.gpart[i]), kConsumerWarps);
      mbar_init(smem_addr(&misc.gfree[i]), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  Ring ring;
  ring.data = smem_addr(base);
  ring.full = smem_addr(&misc.full[0]);
  ring.empty = smem_addr(&misc.empty[0]);
  ring.it = 0;
  const int t0 = p.sm_begin[blockIdx.x], t1 = p.sm_begin[blockIdx.x + 1];

  if (threadIdx.x / 32 >= kConsumerWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    // the copies go out from warp 9, on a different SM sub-partition (warp % 4) than the
    // tensor-core issue (warp 0) and the batch-8 expert epilogue (warp 4); measured ~1 % faster
    // at batch 8 than warp 8, neutral at batch 1
    if (threadIdx.x / 32 != kConsumerWarps + 1) return;
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
    if ((threadIdx.x & 31) == 0) pr.drain();  // never leave while a copy into shared memory is in flight
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
  Consumer<NB> c(p, misc, ring, smem_addr(base + kStages * kStageBytes));
  // The task loop, inline in the kernel (a call after setmaxnreg would hand the callee a register
  // budget of its own): descriptors in batches of 32, lane j holding descriptor base + j, the next
  // batch loaded while the current one runs; each task broadcast from its lane.
  if (c.load_step_cache()) {
    const uint4* src = reinterpret_cast<const uint4*>(p.tasks);
    const int lane = threadIdx.x & 31;
    uint4 cur = t0 + lane < t1 ? __ldg(src + t0 + lane) : make_uint4(0, 0, 0, 0);
    for (int tb = t0; tb < t1 && c.ok; tb += 32) {
      const uint4 nxt = tb + 32 + lane < t1 ? __ldg(src + tb + 32 + lane) : make_uint4(0, 0, 0, 0);
      const int n = min(32, t1 - tb);
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
  if (threadIdx.x < 32) {
    // warp 0 issued every tensor-core product of the block: wait (bounded) until they have all
    // completed, also on an abort path, then give the tensor memory back
    __syncwarp();
    if (!c.ok) {
      if (threadIdx.x == 0) tc_commit(smem_addr(&misc.tc_acc));
      __syncwarp();
      const uint64_t tw0 = gtimer();
      while (!mbar_try_wait(smem_addr(&misc.tc_acc), c.tc_phase) && gtimer() - tw0 < 1000000000ull) {
      }
      __syncwarp();
    }
    tc_fence_before();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(misc.tmem_base), "r"(kTmemCols));
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
