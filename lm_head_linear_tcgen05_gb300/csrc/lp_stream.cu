// lp_stream.cu - logits-reuse path: LSE, target logp and entropy from precomputed
// local logits, streamed once from HBM.
//
// Page "feat(rl-kernel): add CUDA linear logp provider integration", Changes /
// Megatron integration: strict LM-head local logits are reused when available,
// avoiding a second projection. Page "Perf/cuda compact top p replay", Summary:
// temperature scaling happens exactly once for reused logits - the logits given
// here are unscaled and 1/tau is applied in this kernel only.
//
// One CTA (256 threads) per row, four per SM. Each thread loads its 16-byte vectors
// j = tid, tid+256, ... of a shard's row straight into registers, eight at a time
// (128 KB in flight per SM, streaming cache hint), takes the maximum of the whole batch
// with max.bf16x2 and rescales its running statistic at most once per batch, then
// folds the 64 logits in packed f32x2 arithmetic. Logits far below the running maximum
// are first raised to a floor whose scaled value is at least 200 binary orders below it:
// 2^d flushes to 0 there exactly as it would for the original logit, and a -inf logit
// (an entry the caller masked out) never forms 0 * inf. The threads of a shard are
// combined by a fixed shuffle tree per warp; the per-warp results of every shard wait in
// shared memory until the row is done, and thread 0 then merges warp after warp into each
// shard's own (LSE, entropy) and reduces the shards in ascending order (row_finish). The
// work split depends only on the shard width, so a row's result never depends on T. No
// thread waits on another while streaming.
#include <cuda_bf16.h>

#include "lp_device.cuh"
#include "lp_f32x2.cuh"

namespace lp {

namespace {

#ifndef LP_STREAM_UNROLL
#define LP_STREAM_UNROLL 8       // 16-byte vectors per thread in flight
#endif
#ifndef LP_STREAM_MIN_BLOCKS
#define LP_STREAM_MIN_BLOCKS 4   // rows resident per SM
#endif
constexpr int kStreamThreads = 256;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kUnroll = LP_STREAM_UNROLL;
// the most negative finite bf16, exactly
constexpr float kBf16Lowest = -3.38953138925153547590470800371487866880e38f;
// padding for the vectors of a partial batch: eight bf16 -inf
constexpr uint32_t kNegInfPair = 0xFF80FF80u;

// Per-thread online statistic over raw (unscaled) logits x: the running maximum is
// tracked on x, m = max(x) * c2 and d = x * c2 - m, so u = x * c2 is never rounded
// separately from the subtraction. Sums are kept as two interleaved partial sums
// (even / odd elements of each 16-byte vector) in packed fp32 pairs and added at the
// end. floor2 holds, twice in bf16, the largest bf16 value <= max(x) - 200 / c2 (never
// below the lowest finite bf16): a logit below it is folded as if it were the floor,
// which changes nothing - both give 2^d < 2^-126, flushed to 0 - but keeps d finite.
struct RawStat {
  float xmax;       // running max of x (-inf while empty)
  float m;          // xmax * c2
  uint64_t s2;      // {even, odd} partial sums of 2^(u - m)
  uint64_t a2;      // {even, odd} partial sums of 2^(u - m) (u - m)
  uint32_t floor2;  // {floor, floor} in bf16
};

// span = 200 / c2 rounded up, so that floor * c2 <= max(x) * c2 - 200
__device__ __forceinline__ void raw_rescale(RawStat& st, float new_xmax, float c2, float span) {
  const float nm = __fmul_rn(new_xmax, c2);
  if (st.xmax == -INFINITY) {
    st.s2 = 0ull;
    st.a2 = 0ull;
  } else {
    const float d = __fsub_rn(st.m, nm);
    const float e = hw_ex2(d);
    const uint64_t d2 = pack2(d, d), e2 = pack2(e, e);
    st.a2 = mul2(e2, fma2(d2, st.s2, st.a2));
    st.s2 = mul2(st.s2, e2);
  }
  st.xmax = new_xmax;
  st.m = nm;
  const __nv_bfloat16 f = __float2bfloat16_rd(fmaxf(__fsub_rd(new_xmax, span), kBf16Lowest));
  const uint32_t fb = *reinterpret_cast<const uint16_t*>(&f);
  st.floor2 = fb | (fb << 16);
}

// fold the pair (lo, hi) of one bf16x2 word; nm2 = {-m, -m}
__device__ __forceinline__ void raw_pair(RawStat& st, uint32_t w, uint64_t c22, uint64_t nm2) {
  const uint32_t wc = max_bf16x2(w, st.floor2);
  const uint64_t d2 = fma2(pack2(bf16_lo(wc), bf16_hi(wc)), c22, nm2);
  float d0, d1;
  unpack2(d2, d0, d1);
  const uint64_t e2 = pack2(hw_ex2(d0), hw_ex2(d1));
  st.s2 = add2(st.s2, e2);
  st.a2 = fma2(e2, d2, st.a2);
}

__device__ __forceinline__ uint32_t vec_max(const uint4& v) {
  return max_bf16x2(max_bf16x2(v.x, v.y), max_bf16x2(v.z, v.w));
}

// Fold one batch of vectors, in order; only the first n_valid are folded (the rest are
// -inf padding). The running maximum is raised once, to the maximum of the batch.
__device__ __forceinline__ void raw_fold_batch(RawStat& st, const uint4 (&v)[kUnroll], int n_valid, float c2,
                                               float span) {
  uint32_t mm = vec_max(v[0]);
#pragma unroll
  for (int u = 1; u < kUnroll; ++u) mm = max_bf16x2(mm, vec_max(v[u]));
  const float vmax = fmaxf(bf16_lo(mm), bf16_hi(mm));
  if (vmax > st.xmax) raw_rescale(st, vmax, c2, span);
  if (st.xmax == -INFINITY) return;  // every logit so far is -inf: nothing to add
  const uint64_t c22 = pack2(c2, c2);
  const uint64_t nm2 = pack2(-st.m, -st.m);
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    if (u < n_valid) {
      raw_pair(st, v[u].x, c22, nm2);
      raw_pair(st, v[u].y, c22, nm2);
      raw_pair(st, v[u].z, c22, nm2);
      raw_pair(st, v[u].w, c22, nm2);
    }
  }
}

// one element, folded into the even partial sums
__device__ __forceinline__ void raw_push1(RawStat& st, float x, float c2, float span) {
  if (x > st.xmax) raw_rescale(st, x, c2, span);
  const float d = fmaxf(__fmaf_rn(x, c2, -st.m), -256.f);
  const float e = hw_ex2(d);
  st.s2 = add2(st.s2, pack2(e, 0.f));
  st.a2 = fma2(pack2(e, 0.f), pack2(d, 0.f), st.a2);
}

__device__ __forceinline__ Stat raw_to_stat(const RawStat& st) {
  float s0, s1, a0, a1;
  unpack2(st.s2, s0, s1);
  unpack2(st.a2, a0, a1);
  return Stat{st.m, __fadd_rn(s0, s1), __fadd_rn(a0, a1)};
}

}  // namespace

__global__ void __launch_bounds__(kStreamThreads, LP_STREAM_MIN_BLOCKS) stream_logits_kernel(const __grid_constant__ StreamParams p) {
  __shared__ Stat red[LP_MAX_SHARDS][kStreamWarps];  // per shard, per warp
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const float c2 = p.scale_log2;
  const float span = __fdiv_ru(200.f, c2);
  const int yv = __ldg(p.y + row);
  const bool y_ok = yv >= 0 && int64_t(yv) < p.vocab_real;
  const size_t T = size_t(p.T);
  constexpr int64_t kBatch = int64_t(kUnroll) * kStreamThreads;

  for (int k = 0; k < p.n_shards; ++k) {
    const int64_t width = p.shard_width[k];
    const __nv_bfloat16* L = p.logits[k] + size_t(row) * size_t(p.ld[k]);
    const uint4* src = reinterpret_cast<const uint4*>(L);
    const int64_t nvec = width > 0 ? (width >> 3) : 0;
    RawStat st{-INFINITY, -INFINITY, 0ull, 0ull, 0u};
    int64_t j0 = tid;  // this thread's vectors: j0, j0 + 256, ...
    for (; j0 + kBatch - kStreamThreads < nvec; j0 += kBatch) {
      // the batch's last vector ends inside the shard's real columns
      if (!in_bounds(8 * (j0 + kBatch - kStreamThreads + 1) <= width, p.err)) break;
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(src + j0 + int64_t(u) * kStreamThreads);
      raw_fold_batch(st, v, kUnroll, c2, span);
    }
    if (j0 < nvec) {  // the last, partial batch: fewer than kUnroll vectors for this thread
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + int64_t(u) * kStreamThreads;
        v[u] = j < nvec && in_bounds(8 * (j + 1) <= width, p.err)
                   ? __ldcs(src + j)
                   : make_uint4(kNegInfPair, kNegInfPair, kNegInfPair, kNegInfPair);
      }
      raw_fold_batch(st, v, int((nvec - j0 + kStreamThreads - 1) / kStreamThreads), c2, span);
    }
    // ragged tail (width % 8 elements) by the first threads, in ascending order
    const int64_t tail0 = nvec << 3;
    if (width > 0 && tail0 + tid < width && in_bounds(tail0 + tid < p.ld[k], p.err))
      raw_push1(st, __bfloat162float(L[tail0 + tid]), c2, span);

    Stat loc = raw_to_stat(st);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const Stat o{__shfl_down_sync(0xffffffffu, loc.m, off), __shfl_down_sync(0xffffffffu, loc.s, off),
                   __shfl_down_sync(0xffffffffu, loc.a, off)};
      if (lane < off) stat_merge(loc, o);
    }
    if (lane == 0) red[k][warp] = loc;
  }
  __syncthreads();
  if (tid != 0) return;
  // shard by shard: the warps' statistics merged in ascending order, then the shards
  // reduced in ascending order by row_finish
  int owner = -1;  // the shard holding y (none: y belongs to another rank's range)
  float lse[LP_MAX_SHARDS], h[LP_MAX_SHARDS], t[LP_MAX_SHARDS];
#pragma unroll
  for (int k = 0; k < LP_MAX_SHARDS; ++k) {
    lse[k] = -INFINITY;
    h[k] = 0.f;
    t[k] = 0.f;
    if (k < p.n_shards) {
      Stat sh = red[k][0];
      for (int w = 1; w < kStreamWarps; ++w) stat_merge(sh, red[k][w]);
      lse[k] = stat_lse(sh);
      h[k] = stat_entropy(sh);
      if (y_ok && yv >= p.shard_start[k] && yv < p.shard_end[k]) {
        owner = k;
        if (in_bounds(yv - p.shard_start[k] < p.shard_width[k], p.err)) {
          const __nv_bfloat16* L = p.logits[k] + size_t(row) * size_t(p.ld[k]);
          t[k] = __fmul_rn(__bfloat162float(L[yv - p.shard_start[k]]), p.inv_tau);
        }
      }
      if (p.shard_stats != nullptr) {
        float* ss = p.shard_stats + size_t(k) * 3 * T;
        ss[row] = lse[k];
        ss[T + row] = t[k];
        ss[2 * T + row] = h[k];
      }
    }
  }
  const RowOut o = row_finish(lse, h, t, p.n_shards, owner);
  p.lse[row] = o.lse;
  if (p.entropy != nullptr) p.entropy[row] = o.entropy;
  if (!y_ok) record_error(p.err, LP_ERR_TARGET_OUT_OF_RANGE);
  p.logp[row] = o.logp;
}

cudaError_t launch_stream_logits(const StreamParams& p, cudaStream_t s) {
  stream_logits_kernel<<<p.T, kStreamThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace lp
