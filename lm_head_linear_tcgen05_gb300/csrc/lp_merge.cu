// lp_merge.cu - the steps a vocabulary-parallel run adds between ranks: the rank-ordered
// reduction of exchanged per-shard statistics, and the rank-ordered sum of partial
// results (page "Perf/cuda compact top p replay", Summary: rank-ordered reductions, and
// tensor-parallel shards with no replay candidates handled without NaN).
//
// merge_stats_kernel folds, per row, the (local LSE, target logit, own entropy) of every
// shard in ascending order through row_finish - the very function each entry point uses
// on its own shards - so statistics gathered from rank-local calls merge to the bits one
// call over every shard returns. One thread per row: the [K][3][T] statistics are read
// with consecutive threads on consecutive rows (whole sectors).
//
// sum_partials_kernel adds n partial arrays elementwise in ascending order, four
// elements per thread (16-byte loads), rounding once to bf16 when asked.
#include <cuda_bf16.h>

#include "lp_device.cuh"

namespace lp {

namespace {

constexpr int kMergeStatsThreads = 256;
constexpr int kSumThreads = 256;

}  // namespace

__global__ void __launch_bounds__(kMergeStatsThreads) merge_stats_kernel(const __grid_constant__ MergeStatsParams p) {
  const int row = int(blockIdx.x) * kMergeStatsThreads + int(threadIdx.x);
  if (row >= p.T) return;
  const size_t T = size_t(p.T);
  const int yv = __ldg(p.y + row);
  const bool y_ok = yv >= 0 && int64_t(yv) < p.vocab_real;
  int owner = -1;
  float lse[LP_MAX_SHARDS], h[LP_MAX_SHARDS], t[LP_MAX_SHARDS];
#pragma unroll
  for (int k = 0; k < LP_MAX_SHARDS; ++k) {
    lse[k] = -INFINITY;
    h[k] = 0.f;
    t[k] = 0.f;
    if (k < p.n_shards) {
      const float* sk = p.stats + size_t(k) * 3 * T;
      lse[k] = __ldg(sk + row);
      t[k] = __ldg(sk + T + row);
      h[k] = __ldg(sk + 2 * T + row);
      if (y_ok && yv >= p.shard_start[k] && yv < p.shard_end[k]) owner = k;
    }
  }
  const RowOut o = row_finish(lse, h, t, p.n_shards, owner);
  p.lse[row] = o.lse;
  if (p.entropy != nullptr) p.entropy[row] = o.entropy;
  if (!y_ok) record_error(p.err, LP_ERR_TARGET_OUT_OF_RANGE);
  p.logp[row] = o.logp;
}

__global__ void __launch_bounds__(kSumThreads) sum_partials_kernel(const __grid_constant__ SumPartsParams p) {
  const int64_t n4 = p.count >> 2;
  const int64_t i = int64_t(blockIdx.x) * kSumThreads + threadIdx.x;
  if (i < n4) {
    float4 acc = __ldg(reinterpret_cast<const float4*>(p.parts[0]) + i);
    for (int s = 1; s < p.n_parts; ++s) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(p.parts[s]) + i);
      acc.x = __fadd_rn(acc.x, v.x);
      acc.y = __fadd_rn(acc.y, v.y);
      acc.z = __fadd_rn(acc.z, v.z);
      acc.w = __fadd_rn(acc.w, v.w);
    }
    if (p.out_bf16) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
      reinterpret_cast<uint2*>(p.out)[i] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    } else {
      reinterpret_cast<float4*>(p.out)[i] = acc;
    }
  }
  // the count % 4 trailing elements, by the first threads of the grid
  const int64_t j = (n4 << 2) + i;
  if (i < 4 && j < p.count) {
    float acc = p.parts[0][j];
    for (int s = 1; s < p.n_parts; ++s) acc = __fadd_rn(acc, p.parts[s][j]);
    if (p.out_bf16)
      static_cast<__nv_bfloat16*>(p.out)[j] = __float2bfloat16_rn(acc);
    else
      static_cast<float*>(p.out)[j] = acc;
  }
}

cudaError_t launch_merge_stats(const MergeStatsParams& p, cudaStream_t s) {
  merge_stats_kernel<<<unsigned((p.T + kMergeStatsThreads - 1) / kMergeStatsThreads), kMergeStatsThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_sum_partials(const SumPartsParams& p, cudaStream_t s) {
  const int64_t threads = (p.count >> 2) > 4 ? (p.count >> 2) : 4;
  sum_partials_kernel<<<unsigned((threads + kSumThreads - 1) / kSumThreads), kSumThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace lp
