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
//   1. warp 0 reads the 64 slots, checks every id, and writes the distinct ids in
//      ascending order (rank of each first occurrence among the distinct values);
//   2. the row of X is staged in shared memory;
//   3. each warp scores ids i = warp, warp+8, ...: a canonical fp32 dot product
//      (lane l accumulates 16-byte vectors l, l+32, ... in order, then a fixed
//      shuffle tree) of x with the gathered row W[id] - a gather GEMV;
//   4. thread 0 folds the scores in ascending id order, shard by shard, and merges
//      the shards in ascending order.
// The dense keep-mask route compacts each mask row into the same canonical slots
// and runs this very kernel, so both routes produce identical bits for equal sets.
// The logits-gather variant (reused unscaled logits instead of x . W) replaces step 3
// by one gather per id and keeps steps 1 and 4.
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

__device__ __forceinline__ int shard_of(const ReplayParams& p, int64_t v) {
  int k = 0;
  while (k + 1 < p.n_shards && v >= p.shard_end[k]) ++k;
  return k;
}

}  // namespace

template <bool kFromLogits>
__global__ void __launch_bounds__(kReplayThreads, LP_REPLAY_MIN_BLOCKS) replay_kernel(const __grid_constant__ ReplayParams p) {
  extern __shared__ uint4 xs[];  // the row of X, H / 8 vectors
  __shared__ int32_t slots[LP_REPLAY_SLOTS];
  __shared__ uint8_t dup[LP_REPLAY_SLOTS];
  __shared__ int32_t uniq[LP_REPLAY_SLOTS];
  __shared__ float zs[LP_REPLAY_SLOTS];
  __shared__ int n_uniq;
  __shared__ int bad_row;

  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const size_t T = size_t(p.T);
  const int nvec = p.H >> 3;

  // 1. validate, sort ascending, deduplicate
  if (warp == 0) {
    const int32_t* ids = p.ids + size_t(row) * LP_REPLAY_SLOTS;
    const int32_t v0 = __ldg(ids + lane), v1 = __ldg(ids + 32 + lane);
    const bool bad0 = v0 != -1 && (v0 < 0 || int64_t(v0) >= p.vocab_real);
    const bool bad1 = v1 != -1 && (v1 < 0 || int64_t(v1) >= p.vocab_real);
    const unsigned any_bad = __ballot_sync(0xffffffffu, bad0 || bad1);
    slots[lane] = (bad0 || v0 < 0) ? -1 : v0;
    slots[32 + lane] = (bad1 || v1 < 0) ? -1 : v1;
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      const int32_t v = slots[i];
      bool d = v == -1;
      for (int j = 0; j < i && !d; ++j) d = slots[j] == v;
      dup[i] = d ? 1 : 0;
    }
    __syncwarp();
    int kept = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      const int32_t v = slots[i];
      if (!dup[i]) {
        int rank = 0;
        for (int j = 0; j < LP_REPLAY_SLOTS; ++j) rank += (!dup[j] && slots[j] < v) ? 1 : 0;
        uniq[rank] = v;
        ++kept;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, off);
    if (lane == 0) {
      n_uniq = kept;
      bad_row = any_bad != 0u;
      if (any_bad) record_error(p.err, LP_ERR_REPLAY_ID_OUT_OF_RANGE);
    }
  }
  if constexpr (!kFromLogits) {
    // 2. stage x
    const uint4* xrow = reinterpret_cast<const uint4*>(p.X) + size_t(row) * size_t(nvec);
    for (int v = tid; v < nvec; v += kReplayThreads) xs[v] = __ldg(xrow + v);
  }
  __syncthreads();

  const int n = bad_row ? 0 : n_uniq;
  if constexpr (!kFromLogits) {
    // 3. gather GEMV
    for (int i = warp; i < n; i += kReplayWarps) {
      const int64_t v = uniq[i];
      const int k = shard_of(p, v);
      const int64_t local = v - p.shard_start[k];
      const uint4* wrow = reinterpret_cast<const uint4*>(p.W[k]) + size_t(local) * size_t(nvec);
      const float dot = warp_dot(wrow, xs, nvec, lane);
      if (lane == 0) {
        const float b = p.bias[k] != nullptr ? __bfloat162float(p.bias[k][local]) : 0.f;
        zs[i] = __fmul_rn(__fadd_rn(dot, b), p.inv_tau);
      }
    }
  } else {
    // 3. gather of the reused logits, temperature applied here (once)
    if (tid < n) {
      const int64_t v = uniq[tid];
      const int k = shard_of(p, v);
      const float l = __bfloat162float(p.logits[k][size_t(row) * size_t(p.ld[k]) + size_t(v - p.shard_start[k])]);
      zs[tid] = __fmul_rn(l, p.inv_tau);
    }
  }
  __syncthreads();

  // 4. fold in ascending id order, shard by shard, shards in ascending order
  if (tid == 0) {
    const int yv = __ldg(p.y + row);
    const bool y_ok = yv >= 0 && int64_t(yv) < p.vocab_real;
    if (!y_ok) record_error(p.err, LP_ERR_TARGET_OUT_OF_RANGE);
    Stat tot = stat_empty();
    float t_val = 0.f;
    bool t_found = false;
    int i = 0;
    for (int k = 0; k < p.n_shards; ++k) {
      Stat loc = stat_empty();
      float tk = 0.f;
      for (; i < n && uniq[i] < p.shard_end[k]; ++i) {
        const float z = zs[i];
        stat_push(loc, __fmul_rn(z, kLog2e));
        if (uniq[i] == yv) {
          tk = z;
          t_val = z;
          t_found = true;
        }
      }
      if (p.shard_stats != nullptr) {
        float* ss = p.shard_stats + size_t(k) * 3 * T;
        ss[row] = stat_lse(loc);
        ss[T + row] = tk;
        ss[2 * T + row] = 0.f;
      }
      stat_merge(tot, loc);
    }
    const float lse = stat_lse(tot);
    p.lse[row] = bad_row ? -INFINITY : lse;
    p.logp[row] = (!bad_row && y_ok && t_found) ? __fsub_rn(t_val, lse) : -INFINITY;
  }
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
      cudaError_t e =
          cudaFuncSetAttribute(replay_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536 / 8 * 16);
      if (e != cudaSuccess) return e;
      ready[dev].store(true, std::memory_order_release);
    }
  }
  replay_kernel<false><<<p.T, kReplayThreads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_replay_from_logits(const ReplayParams& p, cudaStream_t s) {
  replay_kernel<true><<<p.T, kReplayThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_mask_compact(const MaskParams& p, cudaStream_t s) {
  mask_compact_kernel<<<p.T, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace lp
