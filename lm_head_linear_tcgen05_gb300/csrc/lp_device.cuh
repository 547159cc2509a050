// lp_device.cuh - device helpers shared by the linear-logp kernels (sm_103a).
//
//  * thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor) and the
//    5th-generation tensor core (tcgen05: TMEM alloc, mma, commit, ld);
//  * bounded waits: every spin on an mbarrier gives up after a time limit, records
//    LP_ERR_DEVICE_TIMEOUT in the device error word and lets the kernel tear down;
//  * the per-row statistics fold used by every path. Statistics are kept in base-2
//    units of the scaled logit, u = z * log2(e), z = (x.w + b) / tau:
//        m = max u,  s = sum 2^(u - m),  a = sum 2^(u - m) (u - m)
//    so that LSE = ln2 (m + log2 s) and entropy = ln2 (log2 s - a / s). An empty set
//    is (m, s, a) = (-inf, 0, 0)
//    and is skipped by every merge, so no -inf - -inf is ever formed (the
//    empty-shard rule of page "Perf/cuda compact top p replay", Walkthrough).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "lp_internal.h"

namespace lp {

// ----------------------------------------------------------------- basics

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// hardware 2^x (ex2.approx, flush-to-zero); 2^-inf = +0
__device__ __forceinline__ float hw_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void record_error(unsigned int* err, unsigned int code) {
  if (err) atomicCAS(err, 0u, code);  // first error wins
}

// Device-side bounds checks of the bounds-checked build (LP_DEBUG_BOUNDS=1): in_bounds(ok,
// err) returns ok and, when ok is false, records LP_ERR_BOUNDS, so that the caller skips the
// access. In the regular build it returns true and the comparison compiles away.
#ifndef LP_DEBUG_BOUNDS
#define LP_DEBUG_BOUNDS 0
#endif
__device__ __forceinline__ bool in_bounds(bool ok, unsigned int* err) {
#if LP_DEBUG_BOUNDS
  if (!ok) record_error(err, LP_ERR_BOUNDS);
  return ok;
#else
  (void)ok;
  (void)err;
  return true;
#endif
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// --------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete. Gives up (returns
// false) when `*abort` is raised by another role or when `limit_ns` has elapsed; in
// the latter case it raises `*abort` and records LP_ERR_DEVICE_TIMEOUT. Each try_wait may
// suspend the thread for a while in hardware, so the flag and the clock are checked after
// every unsuccessful try: the limit holds to within one suspension.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns, unsigned int* err) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_test(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort = 1;
      record_error(err, LP_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// mbar_wait for a barrier that threads of another CTA of the cluster arrive on (acquire at
// cluster scope).
__device__ __forceinline__ bool mbar_test_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  uint64_t limit_ns, unsigned int* err) {
  if (mbar_test_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_test_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort = 1;
      record_error(err, LP_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait used on teardown paths: ignores the abort flag, gives up at `deadline`
// (global timer, ns).
__device__ __forceinline__ void drain_until(uint64_t* bar, uint32_t parity, uint64_t deadline) {
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() > deadline) break;
  }
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  drain_until(bar, parity, global_timer_ns() + limit_ns);
}

// -------------------------------------------------------------------- TMA

// 2-D tiled bulk tensor copy global -> shared, completing on `bar` (tx bytes).
// (x, y) = (innermost, outer) element coordinates of the box origin; x is always a
// multiple of the 64-element box width here, so x * 2 bytes is 16-byte aligned.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int32_t x,
                                            int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// The same copy for a CTA pair running paired-SM MMAs (.cta_group::2): the box lands in
// this CTA's shared memory and completes on the mbarrier at shared::cluster address
// `bar_cl`, which may be the pair's other CTA's (the one that issues the MMAs).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* tmap, uint32_t bar_cl, int32_t x, int32_t y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(bar_cl), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// shared::cluster address of the variable at `local` in the shared memory of cluster CTA `rank`
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

// Arrive on an mbarrier of any CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cl) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster: release/acquire barrier.
// Programmatic dependent launch: a kernel launched with programmatic stream serialisation
// may start before the kernel it follows on the stream has finished, once every CTA of that
// kernel has signalled launch_dependents (or exited); grid_dependency_wait then blocks
// until that kernel has completed and its memory operations are visible. Without such a
// launch both are no-ops.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- tcgen05

// TMEM allocation by one warp of the CTA (CG = 1), or collectively by one warp of each CTA
// of a pair (CG = 2: the same columns in both CTAs).
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (CG == 1)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate. CG = 1: one CTA. CG = 2:
// issued by one thread of a CTA pair; A's M rows and B's N rows are split evenly between
// the two CTAs' shared memory (same offsets in both) and each CTA's TMEM receives its half
// of the rows for all N columns.
template <int CG>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  if constexpr (CG == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` (this CTA's) when every tcgen05.mma issued so far by this thread is done.
template <int CG>
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// As umma_commit, arriving on the mbarrier at the same offset in both CTAs of the pair.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(uint16_t(3))
               : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile stored as the 128-byte
// swizzled layout TMA writes (rows of 64 elements = 128 B, 8-row atoms of 1024 B):
// start address >> 4 in bits [0,14), leading byte offset (unused for this layout,
// 16 B) in [16,30), stride byte offset 1024 B (next 8-row group) in [32,46),
// descriptor version 1 in [46,48), swizzle mode 2 (128 B) in [61,64).
// The tile base must be 1024-byte aligned; advancing along K by 16 elements adds
// 32 bytes (2 in the encoded address).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Descriptor of an MN-major bf16 operand in the 128-byte swizzled layout TMA writes
// for boxes of 64 MN-elements x 64 K-rows: each K row is 128 bytes (64 consecutive
// MN elements), 8 K rows form a 1024-byte swizzle atom, consecutive 8-row K groups
// are 1024 bytes apart (stride byte offset) and consecutive 64-element MN atoms are
// `mn_atom_bytes` apart (leading byte offset). Advancing along K by 16 rows adds
// 2048 bytes (128 in the encoded address).
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr, uint32_t mn_atom_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(mn_atom_bytes >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits [4,6) = 1),
// A and B bf16 (bits [7,10) = 1, [10,13) = 1), A / B major-ness in bits 15 / 16
// (0 = K-major, 1 = MN-major), N >> 3 in bits [17,23), M >> 4 in bits [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool a_mn = false,
                                                      bool b_mn = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

// 32 TMEM lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// columns [col, col + 32) of lane (lane_base + i); taddr = (lane_base << 16) | col.
// The load and its tcgen05.wait::ld sit in one asm statement, so no use of the
// destination registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// ------------------------------------------------------------ statistics

// Running base-2 statistics of a set of scaled logits (see the file comment).
struct Stat {
  float m, s, a;
};

__device__ __forceinline__ Stat stat_empty() { return Stat{-INFINITY, 0.f, 0.f}; }

// Merge B into A: both are statistics of disjoint sets; the result is that of the union.
// Written with explicit round-to-nearest intrinsics so that every caller gets the
// same bits for the same operands, whatever the surrounding code.
__device__ __forceinline__ void stat_merge(Stat& A, const Stat& B) {
  if (B.m == -INFINITY) return;
  if (A.m == -INFINITY) {
    A = B;
    return;
  }
  const float M = fmaxf(A.m, B.m);
  const float da = __fsub_rn(A.m, M);
  const float db = __fsub_rn(B.m, M);
  const float ea = hw_ex2(da);
  const float eb = hw_ex2(db);
  const float s = __fadd_rn(__fmul_rn(A.s, ea), __fmul_rn(B.s, eb));
  const float a = __fadd_rn(__fmul_rn(ea, __fmaf_rn(da, A.s, A.a)), __fmul_rn(eb, __fmaf_rn(db, B.s, B.a)));
  A = Stat{M, s, a};
}

// Fold one scaled logit u (base-2 units) into A, sequentially.
__device__ __forceinline__ void stat_push(Stat& A, float u) {
  if (A.m == -INFINITY) {
    A = Stat{u, 1.f, 0.f};
    return;
  }
  if (u > A.m) {
    const float d = __fsub_rn(A.m, u);
    const float e = hw_ex2(d);
    A.a = __fmul_rn(e, __fmaf_rn(d, A.s, A.a));
    A.s = __fadd_rn(__fmul_rn(A.s, e), 1.f);
    A.m = u;
  } else {
    const float d = __fsub_rn(u, A.m);
    const float e = hw_ex2(d);
    A.s = __fadd_rn(A.s, e);
    A.a = __fmaf_rn(e, d, A.a);
  }
}

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;

// LSE in nats of a statistic (-inf for the empty set).
__device__ __forceinline__ float stat_lse(const Stat& A) {
  if (A.m == -INFINITY) return -INFINITY;
  return __fmul_rn(kLn2, __fadd_rn(A.m, log2f(A.s)));
}

// Entropy in nats (0 for the empty set).
__device__ __forceinline__ float stat_entropy(const Stat& A) {
  if (A.m == -INFINITY) return 0.f;
  return __fmul_rn(kLn2, __fsub_rn(log2f(A.s), __fdiv_rn(A.a, A.s)));
}

// ------------------------------------------------- rank-ordered shard reduction
// What a vocabulary shard reports for the rank-ordered reduction (page "Perf/cuda
// compact top p replay", Summary), in nats: its local LSE (-inf when it holds no id of
// the support), its own entropy h (0 when empty) and its target logit t. The merged row
// follows from these alone:
//     LSE     = M + ln sum_k e^(lse_k - M),             M = max_k lse_k
//     entropy = sum_k w_k (h_k + LSE - lse_k),          w_k = e^(lse_k - LSE)
//     logp    = t_o - LSE, o the shard holding y; -inf when no shard holds y or o is
//               empty (the empty-shard rule), and -inf when t_o is (an excluded id).
// Every path folds its shards through row_finish, and lp_merge_shard_stats folds
// statistics exchanged between ranks through it as well, so one call over K shards and
// K rank-local calls merged afterwards give the same bits. With a single shard the
// result is that shard's own (LSE, h) exactly.

struct RowOut {
  float logp, lse, entropy;
};

// e^d for d <= 0; exactly 1 at d = 0
__device__ __forceinline__ float nat_exp(float d) { return d == 0.f ? 1.f : hw_ex2(__fmul_rn(d, kLog2e)); }

// lse, h, t: [n] per-shard statistics in ascending shard order (n <= LP_MAX_SHARDS);
// owner: index of the shard holding the row's target, or -1.
__device__ __forceinline__ RowOut row_finish(const float* lse, const float* h, const float* t, int n, int owner) {
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < LP_MAX_SHARDS; ++k)
    if (k < n) M = fmaxf(M, lse[k]);
  if (M == -INFINITY) return RowOut{-INFINITY, -INFINITY, 0.f};
  float S = 0.f;
#pragma unroll
  for (int k = 0; k < LP_MAX_SHARDS; ++k)
    if (k < n && lse[k] != -INFINITY) S = __fadd_rn(S, nat_exp(__fsub_rn(lse[k], M)));
  const float L = S == 1.f ? M : __fadd_rn(M, __fmul_rn(kLn2, log2f(S)));
  float E = 0.f;
#pragma unroll
  for (int k = 0; k < LP_MAX_SHARDS; ++k) {
    if (k < n && lse[k] != -INFINITY) {
      const float gap = __fsub_rn(L, lse[k]);
      E = __fmaf_rn(nat_exp(-gap), __fadd_rn(h[k], gap), E);
    }
  }
  float lp = -INFINITY;
#pragma unroll
  for (int k = 0; k < LP_MAX_SHARDS; ++k)
    if (k == owner && lse[k] != -INFINITY) lp = __fsub_rn(t[k], L);
  return RowOut{lp, L, E};
}

}  // namespace lp
