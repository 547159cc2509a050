// lp_replay.cu - compact top-p replay and the dense keep-mask route it replaces.
//
// Page "Perf/cuda compact top p replay", Summary and Walkthrough ("CUDA kernel and
// empty-shard handling"): instead of materialising a full-vocabulary keep mask, the
// kernel validates the replay ids of each row, sorts and deduplicates up to 64 of
// them, scores only those ids with temperature applied, and returns local target
// logits and LSE reduced over shards in rank order; a shard without candidates
// contributes zero probability (LSE -inf, target logit 0) and never a NaN.
//
// One CTA (256 threads) per row, six rows resident per SM (a launch-shape sweep: 4-16
// rows per SM, 128-512 threads, 2-8 vectors per lane in flight; 4.6 % faster than four
// rows with eight vectors, and every variant gives the same bits):
//   1. warp 0 reads the 64 slots, checks every id, sorts them with a bitonic network
//      across its lanes (two per lane) and writes the distinct ids in ascending order;
//   2. the row of X is staged in shared memory;
//   3. each warp scores ids i = warp, warp+8, ...: a canonical fp32 dot product
//      (lane l accumulates 16-byte vectors l, l+32, ... in order, then a fixed
//      shuffle tree) of x with the gathered row W[id] - a gather GEMV;
//   4. warp 0 folds the scores shard by shard - each lane two adjacent ids of the shard's
//      run of the ascending list, then a fixed shuffle tree - and the shards are reduced
//      in ascending order. The order depends only on each shard's own ids.
// The dense keep-mask route compacts each mask row into the same canonical slots
// and runs this very kernel, so both routes produce identical bits for equal sets.
// The logits-gather variant (reused unscaled logits instead of x . W) runs one warp per
// row: the same steps 1 and 4 (the same device functions), and one gather per id in place
// of steps 2 and 3.
#include <cuda_bf16.h>

#include <atomic>

#include "lp_device.cuh"

namespace lp {

namespace {

#ifndef LP_REPLAY_MIN_BLOCKS
#define LP_REPLAY_MIN_BLOCKS 6  // rows resident per SM (40 registers a thread)
#endif
#ifndef LP_REPLAY_UNROLL
#define LP_REPLAY_UNROLL 4      // 16-byte vectors of a W row per lane in flight
#endif
constexpr int kReplayThreads = 256;
constexpr int kDotUnroll = LP_REPLAY_UNROLL;
constexpr int kReplayWarps = kReplayThreads / 32;

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float fma8(float acc, const uint4 x, const uint4 w) {
  acc = __fmaf_rn(bf16_lo(x.x), bf16_lo(w.x), acc);
  acc = __fmaf_rn(bf16_hi(x.x), bf16_hi(w.x), acc);
  acc = __fmaf_rn(bf16_lo(x.y), bf16_lo(w.y), acc);
  acc = __fmaf_rn(bf16_hi(x.y), bf16_hi(w.y), acc);
  acc = __fmaf_rn(bf16_lo(x.z), bf16_lo(w.z), acc);
  acc = __fmaf_rn(bf16_hi(x.z), bf16_hi(w.z), acc);
  acc = __fmaf_rn(bf16_lo(x.w), bf16_lo(w.w), acc);
  acc = __fmaf_rn(bf16_hi(x.w), bf16_hi(w.w), acc);
  return acc;
}

// Canonical dot product of the staged x (shared memory, nvec 16-byte vectors) with a
// row of W; every lane returns the same value.
__device__ __forceinline__ float warp_dot(const uint4* __restrict__ w, const uint4* xs, int nvec, int lane) {
  float acc = 0.f;
  for (int base = 0; base < nvec; base += 32 * kDotUnroll) {
    uint4 wv[kDotUnroll];
#pragma unroll
    for (int u = 0; u < kDotUnroll; ++u) {
      const int v = base + u * 32 + lane;
      wv[u] = v < nvec ? ld_nc(w + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kDotUnroll; ++u) {
      const int v = base + u * 32 + lane;
      if (v < nvec) acc = fma8(acc, xs[v], wv[u]);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float o = __shfl_down_sync(0xffffffffu, acc, off);
    if (lane < off) acc = __fadd_rn(acc, o);
  }
  return __shfl_sync(0xffffffffu, acc, 0);
}

// Warp-wide bitonic sort of 64 unsigned keys, two per lane: element e = 2 * lane + j
// holds k[j]; on return the keys ascend with e. Stage (size, d) compare-exchanges e with
// e ^ d, keeping the smaller key at the lower index inside blocks of `size` whose index
// has bit `size` clear and the larger one elsewhere.
__device__ __forceinline__ void warp_sort64(uint32_t& k0, uint32_t& k1, int lane) {
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
    const bool asc = ((2 * lane) & size) == 0;  // bit 0 (the j of e) never reaches `size`
#pragma unroll
    for (int d = size >> 1; d >= 1; d >>= 1) {
      if (d == 1) {  // both elements in this lane
        const uint32_t lo = min(k0, k1), hi = max(k0, k1);
        k0 = asc ? lo : hi;
        k1 = asc ? hi : lo;
      } else {  // partner lane = lane ^ (d / 2), same j
        const int ld = d >> 1;
        const uint32_t p0 = __shfl_xor_sync(0xffffffffu, k0, ld);
        const uint32_t p1 = __shfl_xor_sync(0xffffffffu, k1, ld);
        const bool take_min = ((lane & ld) == 0) == asc;
        k0 = take_min ? min(k0, p0) : max(k0, p0);
        k1 = take_min ? min(k1, p1) : max(k1, p1);
      }
    }
  }
}

__device__ __forceinline__ int shard_of(const ReplayParams& p, int64_t v) {
  int k = 0;
  while (k + 1 < p.n_shards && v >= p.shard_end[k]) ++k;
  return k;
}

}  // namespace

// 1. Canonicalise one row's replay slots (one warp): unused and invalid slots, and valid
// ids outside this call's range [lo, hi) (another rank's ids in a rank-local partition),
// become the key 0xFFFFFFFF, above every id; the 64 keys are sorted ascending, a key is
// kept if it differs from its predecessor, and its rank is the number of kept keys before
// it. Writes the distinct ids ascending to uniq[0..n) and returns n (0 for a row with an
// invalid id, which is recorded as a device error and fails closed).
__device__ __forceinline__ int canon_row(const ReplayParams& p, int row, int lane, int32_t* uniq) {
  const int32_t* ids = p.ids + size_t(row) * LP_REPLAY_SLOTS;
  const int32_t v0 = __ldg(ids + 2 * lane), v1 = __ldg(ids + 2 * lane + 1);
  const bool bad0 = v0 != -1 && (v0 < 0 || int64_t(v0) >= p.vocab_real);
  const bool bad1 = v1 != -1 && (v1 < 0 || int64_t(v1) >= p.vocab_real);
  const unsigned any_bad = __ballot_sync(0xffffffffu, bad0 || bad1);
  const int64_t lo = p.shard_start[0], hi = p.shard_end[p.n_shards - 1];
  const bool here0 = int64_t(v0) >= lo && int64_t(v0) < hi, here1 = int64_t(v1) >= lo && int64_t(v1) < hi;
  uint32_t k0 = (bad0 || v0 < 0 || !here0) ? 0xFFFFFFFFu : uint32_t(v0);
  uint32_t k1 = (bad1 || v1 < 0 || !here1) ? 0xFFFFFFFFu : uint32_t(v1);
  warp_sort64(k0, k1, lane);
  const uint32_t prev0 = __shfl_up_sync(0xffffffffu, k1, 1);
  const bool keep0 = k0 != 0xFFFFFFFFu && (lane == 0 || k0 != prev0);
  const bool keep1 = k1 != 0xFFFFFFFFu && k1 != k0;
  const unsigned b0 = __ballot_sync(0xffffffffu, keep0), b1 = __ballot_sync(0xffffffffu, keep1);
  const unsigned lower = (1u << lane) - 1u;
  const int before = __popc(b0 & lower) + __popc(b1 & lower);
  if (keep0) uniq[before] = int32_t(k0);
  if (keep1) uniq[before + (keep0 ? 1 : 0)] = int32_t(k1);
  if (any_bad && lane == 0) record_error(p.err, LP_ERR_REPLAY_ID_OUT_OF_RANGE);
  __syncwarp();
  return any_bad ? 0 : __popc(b0) + __popc(b1);
}

// 4. Fold one row's scores (one warp), shard by shard: the shard's ids are a contiguous
// run [i0, i1) of the ascending list; lane l takes its ids i0 + 2l and i0 + 2l + 1, the
// lanes' statistics combine by a fixed shuffle tree, and the shards are reduced in
// ascending order by row_finish - an order fixed by each shard's own ids alone, so a
// rank-local call that holds only some of the shards folds each of them exactly as a call
// holding all does, and every route that produces the same scores gives the same bits.
// A row that failed closed arrives with n = 0: every shard is empty, LSE = logp = -inf.
__device__ __forceinline__ void fold_row(const ReplayParams& p, int row, int lane, const int32_t* uniq,
                                         const float* zs, int n) {
  const size_t T = size_t(p.T);
  const int yv = __ldg(p.y + row);
  const bool y_ok = yv >= 0 && int64_t(yv) < p.vocab_real;
  if (lane == 0 && !y_ok) record_error(p.err, LP_ERR_TARGET_OUT_OF_RANGE);
  const int64_t id0 = 2 * lane < n ? int64_t(uniq[2 * lane]) : INT64_MAX;
  const int64_t id1 = 2 * lane + 1 < n ? int64_t(uniq[2 * lane + 1]) : INT64_MAX;
  // the target logit, if y is in the set: the lane holding it says which of its two ids
  const bool own0 = y_ok && id0 == yv, own1 = y_ok && id1 == yv;
  const unsigned tb = __ballot_sync(0xffffffffu, own0 || own1);
  const bool t_found = tb != 0u;
  const int src = t_found ? __ffs(tb) - 1 : 0;
  const int t_idx = 2 * src + __shfl_sync(0xffffffffu, own0 ? 0 : 1, src);
  const float t_val = t_found ? zs[t_idx] : 0.f;
  int owner = -1;
  float lse[LP_MAX_SHARDS], hz[LP_MAX_SHARDS], t[LP_MAX_SHARDS];
#pragma unroll
  for (int k = 0; k < LP_MAX_SHARDS; ++k) {
    lse[k] = -INFINITY;
    hz[k] = 0.f;
    t[k] = 0.f;
    if (k < p.n_shards) {
      const int64_t s0 = p.shard_start[k], s1 = p.shard_end[k];
      const int i0 = __popc(__ballot_sync(0xffffffffu, id0 < s0)) + __popc(__ballot_sync(0xffffffffu, id1 < s0));
      const int i1 = __popc(__ballot_sync(0xffffffffu, id0 < s1)) + __popc(__ballot_sync(0xffffffffu, id1 < s1));
      Stat loc = stat_empty();
      if (i1 > i0) {
        const int j0 = i0 + 2 * lane, j1 = j0 + 1;
        if (j0 < i1) stat_push(loc, __fmul_rn(zs[j0], kLog2e));
        if (j1 < i1) stat_push(loc, __fmul_rn(zs[j1], kLog2e));
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
          const Stat o{__shfl_down_sync(0xffffffffu, loc.m, off), __shfl_down_sync(0xffffffffu, loc.s, off),
                       __shfl_down_sync(0xffffffffu, loc.a, off)};
          if (lane < off) stat_merge(loc, o);
        }
      }
      lse[k] = stat_lse(loc);
      if (y_ok && yv >= s0 && yv < s1) {
        owner = k;
        // the target's logit over the support: z_y if kept, -inf if the shard keeps
        // other ids but not y (an excluded id), 0 if the shard keeps none (empty shard)
        t[k] = t_found ? t_val : (i1 > i0 ? -INFINITY : 0.f);
      }
    }
  }
  if (lane == 0) {
    if (p.shard_stats != nullptr) {
#pragma unroll
      for (int k = 0; k < LP_MAX_SHARDS; ++k) {
        if (k < p.n_shards) {
          float* ss = p.shard_stats + size_t(k) * 3 * T;
          ss[row] = lse[k];
          ss[T + row] = t[k];
          ss[2 * T + row] = 0.f;
        }
      }
    }
    const RowOut o = row_finish(lse, hz, t, p.n_shards, owner);
    p.lse[row] = o.lse;
    p.logp[row] = o.logp;
  }
}

// Gather-GEMV replay: one CTA per row. Warp 0 canonicalises the slots while all threads
// stage x; the warps then score the row's distinct ids (2, 3); warp 0 folds (4).
__global__ void __launch_bounds__(kReplayThreads, LP_REPLAY_MIN_BLOCKS) replay_kernel(const __grid_constant__ ReplayParams p) {
  extern __shared__ uint4 xs[];  // the row of X, H / 8 vectors
  __shared__ int32_t uniq[LP_REPLAY_SLOTS];
  __shared__ float zs[LP_REPLAY_SLOTS];
  __shared__ int n_uniq;

  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nvec = p.H >> 3;

  if (warp == 0) {
    const int n = canon_row(p, row, lane, uniq);
    if (lane == 0) n_uniq = n;
  }
  // 2. stage x
  const uint4* xrow = reinterpret_cast<const uint4*>(p.X) + size_t(row) * size_t(nvec);
  for (int v = tid; v < nvec; v += kReplayThreads) xs[v] = __ldg(xrow + v);
  __syncthreads();

  const int n = n_uniq;
  // 3. gather GEMV
  for (int i = warp; i < n; i += kReplayWarps) {
    const int64_t v = uniq[i];
    const int k = shard_of(p, v);
    const int64_t local = v - p.shard_start[k];
    // the gathered row lies inside shard k's weight (the same for every lane)
    if (!in_bounds(local >= 0 && v < p.shard_end[k] && v < p.vocab_real, p.err)) {
      if (lane == 0) zs[i] = 0.f;
      continue;
    }
    const uint4* wrow = reinterpret_cast<const uint4*>(p.W[k]) + size_t(local) * size_t(nvec);
    const float dot = warp_dot(wrow, xs, nvec, lane);
    if (lane == 0) {
      const float b = p.bias[k] != nullptr ? __bfloat162float(p.bias[k][local]) : 0.f;
      zs[i] = __fmul_rn(__fadd_rn(dot, b), p.inv_tau);
    }
  }
  __syncthreads();

  if (warp == 0) fold_row(p, row, lane, uniq, zs, n);
}

// Logits-gather replay: one warp per row (kReplayWarps rows per CTA), every step warp-wide -
// canonicalise, one gather of the reused unscaled logit per distinct id (temperature
// applied here, once), fold - so many rows' dependent loads are in flight per SM.
__global__ void __launch_bounds__(kReplayThreads) replay_logits_kernel(const __grid_constant__ ReplayParams p) {
  __shared__ int32_t uniq_s[kReplayWarps][LP_REPLAY_SLOTS];
  __shared__ float zs_s[kReplayWarps][LP_REPLAY_SLOTS];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int row = int(blockIdx.x) * kReplayWarps + warp;
  if (row >= p.T) return;
  int32_t* uniq = uniq_s[warp];
  float* zs = zs_s[warp];
  const int n = canon_row(p, row, lane, uniq);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = 2 * lane + h;
    if (i < n) {
      const int64_t v = uniq[i];
      const int k = shard_of(p, v);
      const int64_t col = v - p.shard_start[k];
      const bool ok = in_bounds(col >= 0 && v < p.shard_end[k] && col < p.ld[k] && v < p.vocab_real, p.err);
      const float l = ok ? __bfloat162float(p.logits[k][size_t(row) * size_t(p.ld[k]) + size_t(col)]) : 0.f;
      zs[i] = __fmul_rn(l, p.inv_tau);
    }
  }
  __syncwarp();
  fold_row(p, row, lane, uniq, zs, n);
}

// Dense keep-mask route: one CTA (256 threads) per row scans the masks of all shards
// in ascending id order and writes the kept real ids, ascending, into canonical
// replay slots (-1 padded). More than 64 kept ids in a row is a device error, and the
// row fails closed: its first slot is overwritten with an out-of-range id, so the
// replay kernel reports LSE = logp = -inf for it.
__global__ void __launch_bounds__(256) mask_compact_kernel(const __grid_constant__ MaskParams p) {
  __shared__ int warp_counts[8];
  __shared__ int base_s;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  int32_t* out = p.ids_out + size_t(row) * LP_REPLAY_SLOTS;
  if (tid < LP_REPLAY_SLOTS) out[tid] = -1;
  if (tid == 0) base_s = 0;
  __syncthreads();
  for (int k = 0; k < p.n_shards; ++k) {
    int64_t width = p.shard_width[k];
    if (p.vocab_real - p.shard_start[k] < width) width = p.vocab_real - p.shard_start[k];
    if (width <= 0) continue;
    const uint8_t* m = p.mask[k] + size_t(row) * size_t(p.shard_width[k]);
    for (int64_t c0 = 0; c0 < width; c0 += 256) {
      const int64_t c = c0 + tid;
      const bool keep = c < width && m[c] != 0;
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      if (lane == 0) warp_counts[warp] = __popc(bal);
      __syncthreads();
      int before = base_s;
      for (int w = 0; w < warp; ++w) before += warp_counts[w];
      const int pos = before + __popc(bal & ((1u << lane) - 1u));
      if (keep) {
        if (pos < LP_REPLAY_SLOTS)
          out[pos] = int32_t(p.shard_start[k] + c);
        else
          record_error(p.err, LP_ERR_REPLAY_TOO_MANY_IDS);
      }
      __syncthreads();
      if (tid == 0) {
        int tot = 0;
        for (int w = 0; w < 8; ++w) tot += warp_counts[w];
        base_s += tot;
      }
      __syncthreads();
    }
  }
  if (tid == 0 && base_s > LP_REPLAY_SLOTS) out[0] = INT32_MIN;
}

cudaError_t launch_replay(const ReplayParams& p, cudaStream_t s) {
  const size_t smem = size_t(p.H / 8) * sizeof(uint4);
  if (smem > 48 * 1024) {
    // the opt-in for the largest x row (H = 65536: 128 KB) once per device
    static std::atomic<bool> ready[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev].load(std::memory_order_acquire)) {
      cudaError_t e = cudaFuncSetAttribute(replay_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536 / 8 * 16);
      if (e != cudaSuccess) return e;
      ready[dev].store(true, std::memory_order_release);
    }
  }
  replay_kernel<<<p.T, kReplayThreads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_replay_from_logits(const ReplayParams& p, cudaStream_t s) {
  replay_logits_kernel<<<(p.T + kReplayWarps - 1) / kReplayWarps, kReplayThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_mask_compact(const MaskParams& p, cudaStream_t s) {
  mask_compact_kernel<<<p.T, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace lp
