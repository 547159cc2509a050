// lp_stream.cu - logits-reuse path: LSE, target logp and entropy from precomputed
// local logits, streamed once from HBM.
//
// Page "feat(rl-kernel): add CUDA linear logp provider integration", Changes /
// Megatron integration: strict LM-head local logits are reused when available,
// avoiding a second projection. Page "Perf/cuda compact top p replay", Summary:
// temperature scaling happens exactly once for reused logits - the logits given
// here are unscaled and 1/tau is applied in this kernel only.
//
// One CTA (256 threads) per row, three CTAs per SM. Thread 0 streams the row through
// a 2-stage ring of 32 KB shared-memory chunks with 1-D bulk copies (cp.async.bulk,
// completion on mbarriers, L2 evict-first), so up to 192 KB per SM are in flight
// without holding registers (the ring shape was chosen by measurement: 6.18 TB/s on
// 8192 x 151936 bf16 logits, against 5.96 TB/s for 3 x 16 KB at four rows per SM). Each thread folds the 16-byte vectors j = tid, tid+256,
// ... of every chunk into an online base-2 statistic; the threads are combined by a
// fixed shuffle tree per warp and then warp by warp in ascending order, shard after
// shard in ascending order. The work split depends only on the shard width, so a
// row's result never depends on T.
#include <cuda_bf16.h>

#include <atomic>

#include "lp_device.cuh"
#include "lp_f32x2.cuh"

namespace lp {

namespace {

#ifndef LP_STREAM_STAGES
#define LP_STREAM_STAGES 2        // 64 KB of copies in flight per row
#endif
#ifndef LP_STREAM_CHUNK_VECS
#define LP_STREAM_CHUNK_VECS 2048  // 32 KB of logits per stage
#endif
#ifndef LP_STREAM_MIN_BLOCKS
#define LP_STREAM_MIN_BLOCKS 3     // rows resident per SM
#endif
constexpr int kStreamThreads = 256;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kChunkVecs = LP_STREAM_CHUNK_VECS;
constexpr int kStages = LP_STREAM_STAGES;

// Per-thread online statistic over raw (unscaled) logits x: the running maximum is
// tracked on x, m = max(x) * c2 and d = x * c2 - m, so u = x * c2 is never rounded
// separately from the subtraction. Sums are kept as two interleaved partial sums
// (even / odd elements of each 16-byte vector) in packed fp32 pairs and added at the
// end. -inf logits (entries a caller masked out) add nothing; a thread that saw only
// -inf stays empty.
struct RawStat {
  float xmax;   // running max of x (-inf while empty)
  float m;      // xmax * c2
  uint64_t s2;  // {even, odd} partial sums of 2^(u - m)
  uint64_t a2;  // {even, odd} partial sums of 2^(u - m) (u - m)
};

__device__ __forceinline__ void raw_rescale(RawStat& st, float new_xmax, float c2) {
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
}

// fold the pair (lo, hi) of one bf16x2 word
__device__ __forceinline__ void raw_pair(RawStat& st, uint32_t w, uint64_t c22, uint64_t nm2) {
  float d0, d1;
  unpack2(fma2(pack2(bf16_lo(w), bf16_hi(w)), c22, nm2), d0, d1);
  // clamping at -256 (2^-256 flushes to 0) keeps -inf (masked) logits from
  // producing 0 * -inf in the entropy sum
  d0 = fmaxf(d0, -256.f);
  d1 = fmaxf(d1, -256.f);
  const uint64_t e2 = pack2(hw_ex2(d0), hw_ex2(d1));
  st.s2 = add2(st.s2, e2);
  st.a2 = fma2(e2, pack2(d0, d1), st.a2);
}

__device__ __forceinline__ void raw_push8(RawStat& st, const uint4 v, float c2) {
  const uint32_t mm = max_bf16x2(max_bf16x2(v.x, v.y), max_bf16x2(v.z, v.w));
  const float vmax = fmaxf(bf16_lo(mm), bf16_hi(mm));
  if (vmax > st.xmax) raw_rescale(st, vmax, c2);
  const uint64_t c22 = pack2(c2, c2);
  const uint64_t nm2 = pack2(-st.m, -st.m);
  raw_pair(st, v.x, c22, nm2);
  raw_pair(st, v.y, c22, nm2);
  raw_pair(st, v.z, c22, nm2);
  raw_pair(st, v.w, c22, nm2);
}

// one element, folded into the even partial sums
__device__ __forceinline__ void raw_push1(RawStat& st, float x, float c2) {
  if (x > st.xmax) raw_rescale(st, x, c2);
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
  extern __shared__ uint4 sbuf[];  // kStages x kChunkVecs vectors of 8 bf16
  __shared__ uint64_t full[kStages];
  __shared__ Stat red[kStreamWarps];
  __shared__ int abort_flag;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const float c2 = p.scale_log2;
  const int yv = __ldg(p.y + row);
  const bool y_ok = yv >= 0 && int64_t(yv) < p.vocab_real;
  const size_t T = size_t(p.T);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const uint64_t pol = l2_policy_evict_first();

  Stat tot = stat_empty();  // meaningful in thread 0 only
  float t_val = 0.f;
  uint32_t g0 = 0;          // chunks of this row consumed so far (all shards): fixes stage and parity
  bool ok = true;

  for (int k = 0; k < p.n_shards && ok; ++k) {
    const int64_t width = p.shard_width[k];
    const __nv_bfloat16* L = p.logits[k] + size_t(row) * size_t(p.ld[k]);
    const uint4* src = reinterpret_cast<const uint4*>(L);
    const int64_t nvec = width > 0 ? (width >> 3) : 0;
    const int nchunks = int((nvec + kChunkVecs - 1) / kChunkVecs);
    RawStat st{-INFINITY, -INFINITY, 0ull, 0ull};
    // thread 0 streams the row through the stage ring; the other threads consume
    auto issue = [&](int c) {
      const int64_t v0 = int64_t(c) * kChunkVecs;
      const int64_t nv = nvec - v0 < kChunkVecs ? nvec - v0 : kChunkVecs;
      const uint32_t s = (g0 + c) % kStages;
      mbar_arrive_expect_tx(&full[s], uint32_t(nv) * 16u);
      bulk_load(sbuf + size_t(s) * kChunkVecs, src + v0, uint32_t(nv) * 16u, &full[s], pol);
    };
    if (tid == 0)
      for (int c = 0; c < nchunks && c < kStages; ++c) issue(c);
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t g = g0 + c;
      const uint32_t s = g % kStages;
      const bool got = mbar_wait(&full[s], (g / kStages) & 1u, &abort_flag, kDefaultWaitLimitNs, p.err);
      if (!__syncthreads_and(got)) {
        ok = false;
        if (tid == 0)  // let the copies already issued land before the CTA exits
          for (int d = c; d < nchunks && d < c + kStages; ++d)
            drain_wait(&full[(g0 + d) % kStages], ((g0 + d) / kStages) & 1u, kDefaultWaitLimitNs);
        break;
      }
      const int64_t v0 = int64_t(c) * kChunkVecs;
      const int nv = int(nvec - v0 < kChunkVecs ? nvec - v0 : kChunkVecs);
      const uint4* chunk = sbuf + size_t(s) * kChunkVecs;
#pragma unroll 4
      for (int j = tid; j < nv; j += kStreamThreads) raw_push8(st, chunk[j], c2);
      __syncthreads();  // stage s fully read
      if (tid == 0 && c + kStages < nchunks) issue(c + kStages);
    }
    g0 += uint32_t(nchunks);
    if (!ok) break;
    // ragged tail (width % 8 elements) by the first threads, in ascending order
    const int64_t tail0 = nvec << 3;
    if (width > 0 && tail0 + tid < width) raw_push1(st, __bfloat162float(L[tail0 + tid]), c2);

    Stat loc = raw_to_stat(st);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const Stat o{__shfl_down_sync(0xffffffffu, loc.m, off), __shfl_down_sync(0xffffffffu, loc.s, off),
                   __shfl_down_sync(0xffffffffu, loc.a, off)};
      if (lane < off) stat_merge(loc, o);
    }
    if (lane == 0) red[warp] = loc;
    __syncthreads();
    if (tid == 0) {
      Stat sh = red[0];
      for (int w = 1; w < kStreamWarps; ++w) stat_merge(sh, red[w]);
      const bool own = y_ok && yv >= p.shard_start[k] && yv < p.shard_end[k];
      float tk = 0.f;
      if (own) {
        tk = __fmul_rn(__bfloat162float(L[yv - p.shard_start[k]]), p.inv_tau);
        t_val = tk;
      }
      if (p.shard_stats != nullptr) {
        float* ss = p.shard_stats + size_t(k) * 3 * T;
        ss[row] = stat_lse(sh);
        ss[T + row] = tk;
        ss[2 * T + row] = stat_mean(sh);
      }
      stat_merge(tot, sh);
    }
    __syncthreads();
  }
  if (tid == 0) {
    const float lse = stat_lse(tot);
    if (!ok) {
      p.lse[row] = -INFINITY;
      p.logp[row] = -INFINITY;
      if (p.entropy != nullptr) p.entropy[row] = 0.f;
      return;
    }
    p.lse[row] = lse;
    if (p.entropy != nullptr) p.entropy[row] = stat_entropy(tot);
    if (!y_ok) record_error(p.err, LP_ERR_TARGET_OUT_OF_RANGE);
    p.logp[row] = (y_ok && tot.m != -INFINITY) ? __fsub_rn(t_val, lse) : -INFINITY;
  }
}

cudaError_t launch_stream_logits(const StreamParams& p, cudaStream_t s) {
  const int smem = kStages * kChunkVecs * int(sizeof(uint4));
  static std::atomic<bool> ready[64];  // shared-memory opt-in done on this device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(stream_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    ready[dev].store(true, std::memory_order_release);
  }
  stream_logits_kernel<<<p.T, kStreamThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace lp
