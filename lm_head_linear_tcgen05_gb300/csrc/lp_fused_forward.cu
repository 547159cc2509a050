// lp_fused_forward.cu - fused linear-logp forward on the 5th-generation tensor core.
//
// Page "feat(rl-kernel): add CUDA linear logp provider integration", Changes: the
// selected-token log probability and optional entropy of softmax((X W^T + b) / tau)
// from the output-layer hidden states and the local projection weight and bias,
// without a second logits tensor.
//
// The projection runs on the tcgen05 pipeline of lp_tcgemm.cuh (A = X, B = W_k, K =
// H) with tiles of 128 rows x 256 vocabulary ids enumerated row-block fastest: all
// row blocks of one vocabulary block run together, so every W block is read from HBM
// once and then served from L2 while X stays L2-resident. The epilogue below turns
// each accumulator row straight from TMEM into base-2 statistics
//     m = max u,  s = sum 2^(u - m),  a = sum 2^(u - m)(u - m),   u = (acc + b) log2(e) / tau
// over the tile's valid columns, plus the target logit z[y] = (acc + b) / tau when y
// falls in the tile; the logits never leave the SM. Each tile's statistics go to
// their own workspace slot and merge_kernel combines them per row in a fixed order
// (vocabulary blocks ascending within a shard, then shards ascending), so the result
// is bitwise deterministic and independent of T, the grid size and the row position.
#include <cuda_bf16.h>

#include "lp_tcgemm.cuh"

namespace lp {

namespace {

constexpr int kChunks = kGemmBlockN / 32;  // 32-column TMEM loads per tile row

__device__ __forceinline__ float f32(uint32_t r) { return __uint_as_float(r); }

// Four interleaved partial sums (column j goes to partial j % 4), combined at the
// end as (p0 + p1) + (p2 + p3): a fixed order that shortens the dependency chains.
struct Sums4 {
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  float a[4] = {0.f, 0.f, 0.f, 0.f};
};

__device__ __forceinline__ float chunk_max_full(const uint32_t (&r)[32]) {
  float m[4] = {f32(r[0]), f32(r[1]), f32(r[2]), f32(r[3])};
#pragma unroll
  for (int j = 4; j < 32; ++j) m[j & 3] = fmaxf(m[j & 3], f32(r[j]));
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// columns j < lim of (acc + b); the bias of column j is lane j's `bl`
__device__ __forceinline__ float chunk_max_masked(const uint32_t (&r)[32], float bl, int lim) {
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float v = __fadd_rn(f32(r[j]), __shfl_sync(0xffffffffu, bl, j));
    mx = j < lim ? fmaxf(mx, v) : mx;
  }
  return mx;
}

__device__ __forceinline__ void chunk_sums_full(const uint32_t (&r)[32], float c2, float m_u, Sums4& acc) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float d = __fmaf_rn(f32(r[j]), c2, -m_u);
    const float e = hw_ex2(d);
    acc.s[j & 3] = __fadd_rn(acc.s[j & 3], e);
    acc.a[j & 3] = __fmaf_rn(e, d, acc.a[j & 3]);
  }
}

// A bias of -inf masks its id out (p = 0). The scaled difference is clamped at -256, where
// 2^d is 0 either way, so such an id never forms 0 * -inf (nor -inf - -inf when a whole
// block is masked); for every finite d below -256 the sums are unchanged.
__device__ __forceinline__ void chunk_sums_masked(const uint32_t (&r)[32], float bl, int lim, float c2, float m_u,
                                                  Sums4& acc) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float v = __fadd_rn(f32(r[j]), __shfl_sync(0xffffffffu, bl, j));
    const float d = fmaxf(__fmaf_rn(v, c2, -m_u), -256.f);
    const float e = hw_ex2(d);
    const bool in = j < lim;
    acc.s[j & 3] = in ? __fadd_rn(acc.s[j & 3], e) : acc.s[j & 3];
    acc.a[j & 3] = in ? __fmaf_rn(e, d, acc.a[j & 3]) : acc.a[j & 3];
  }
}

// r[i] for a run-time i in [0, 32) without indexing the register array
__device__ __forceinline__ float pick(const uint32_t (&r)[32], int i) {
  float v = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) v = (j == i) ? f32(r[j]) : v;
  return v;
}

struct TileCoord {
  int shard, nb_local, nb_global, mb;
};

__device__ __forceinline__ TileCoord fwd_coord(const FwdParams& p, int tile) {
  TileCoord c;
  proj_raster(tile, p.num_m_blocks, p.m_chunk, p.nb_start[p.n_shards], c.mb, c.nb_global);
  int k = 0;
  while (k + 1 < p.n_shards && c.nb_global >= p.nb_start[k + 1]) ++k;
  c.shard = k;
  c.nb_local = c.nb_global - p.nb_start[k];
  return c;
}

}  // namespace

// CM CTAs per cluster along M: kFwdClusterM in general, 1 when the batch is a single row
// block (the second row block of a pair would be padding only). Both compute every tile
// identically - only who fetches the W box differs - so a row's bits do not depend on it.
template <int CM>
struct LogpEpi : GemmEpiBase {
  using Params = FwdParams;
  static constexpr int kClusterM = CM;
  // a single row block loads only its T (rounded up to 16) rows of X: a 128-row box that is
  // nearly all out-of-bounds fill slowed the W stream of tiny batches (T <= 8) by ~20 %
  static constexpr bool kVarABox = CM == 1;

  static __device__ __forceinline__ TileJob job(const Params& p, int tile) {
    const TileCoord c = fwd_coord(p, tile);
    TileJob j;
    j.a_map = 0;
    j.a_y = c.mb * kGemmBlockM;
    j.b_map = 1 + c.shard;
    j.b_y = c.nb_local * kGemmBlockN;
    j.kb0 = 0;
    j.nkb = p.num_k_blocks;
    return j;
  }

  static __device__ __forceinline__ void run(const Params& p, int tile, int /*half*/, uint32_t tbase, int q,
                                             int lane) {
    const TileCoord c = fwd_coord(p, tile);
    const int row = c.mb * kGemmBlockM + q * 32 + lane;
    const int64_t n0 = int64_t(c.nb_local) * kGemmBlockN;
    const int64_t gid0 = p.shard_start[c.shard] + n0;
    int64_t lim64 = int64_t(p.shard_width[c.shard]) - n0;
    if (p.vocab_real - gid0 < lim64) lim64 = p.vocab_real - gid0;
    const int valid = lim64 < 0 ? 0 : (lim64 > kGemmBlockN ? kGemmBlockN : int(lim64));
    const int yv = row < p.T ? __ldg(p.y + row) : -1;
    const int64_t ycol = int64_t(yv) - gid0;
    const __nv_bfloat16* bias = p.bias[c.shard];
    const float c2 = p.scale_log2;

    // bias of column 32*ch + j sits in lane j of bl[ch]
    float bl[kChunks];
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      const int col = ch * 32 + lane;
      bl[ch] = (bias != nullptr && col < valid && in_bounds(n0 + col < p.shard_width[c.shard], p.err))
                   ? __bfloat162float(bias[n0 + col])
                   : 0.f;
    }

    // pass 1: row maximum of (acc + b) over the valid columns
    float mx = -INFINITY;
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      if (ch * 32 < valid) {
        uint32_t r[32];
        tmem_ld32(tbase + ch * 32, r);
        const int lim = valid - ch * 32;
        if (bias == nullptr && lim >= 32)
          mx = fmaxf(mx, chunk_max_full(r));
        else
          mx = fmaxf(mx, chunk_max_masked(r, bl[ch], lim));
      }
    }

    // pass 2: sums of 2^(u - m) and 2^(u - m)(u - m), four interleaved partial sums
    const float m_u = __fmul_rn(mx, c2);
    Sums4 acc4;
    float t_val = 0.f;
    bool t_here = false;
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      if (ch * 32 < valid) {
        uint32_t r[32];
        tmem_ld32(tbase + ch * 32, r);
        const int lim = valid - ch * 32;
        if (bias == nullptr && lim >= 32)
          chunk_sums_full(r, c2, m_u, acc4);
        else
          chunk_sums_masked(r, bl[ch], lim, c2, m_u, acc4);
        // target logit z[y] = (acc + b) / tau when y falls in this chunk
        const int64_t tc = ycol - ch * 32;
        if (tc >= 0 && tc < 32 && tc < lim) {
          const float v = pick(r, int(tc));
          const float b = (bias != nullptr && in_bounds(n0 + ch * 32 + tc < p.shard_width[c.shard], p.err))
                              ? __bfloat162float(bias[n0 + ch * 32 + tc])
                              : 0.f;
          t_val = __fmul_rn(__fadd_rn(v, b), p.inv_tau);
          t_here = true;
        }
      }
    }
    const float s_tot = __fadd_rn(__fadd_rn(acc4.s[0], acc4.s[1]), __fadd_rn(acc4.s[2], acc4.s[3]));
    const float a_tot = __fadd_rn(__fadd_rn(acc4.a[0], acc4.a[1]), __fadd_rn(acc4.a[2], acc4.a[3]));

    // the statistics arrays hold nb_total x T slots
    if (row < p.T && in_bounds(c.nb_global < p.nb_start[p.n_shards], p.err)) {
      const size_t slot = size_t(c.nb_global) * size_t(p.T) + size_t(row);
      p.ws_m[slot] = valid > 0 ? m_u : -INFINITY;
      p.ws_s[slot] = s_tot;
      p.ws_a[slot] = a_tot;
      if (t_here) p.ws_t[row] = t_val;
    }
  }
};

// ------------------------------------------------------------------ merge
// The statistics of vocabulary block nb for row t sit at slot nb * T + t, so consecutive
// rows are adjacent. A block of 256 threads takes 8 rows: thread (g, r) with r = tid % 8
// and g = tid / 8 folds, for row r, the blocks nb = g, g + 32, ... of each shard in
// ascending order, so every load instruction of a warp reads whole 32-byte sectors (4
// groups x 8 adjacent rows). The 32 partials of a row are then combined in a fixed order:
// a shuffle tree over the warp's 4 groups, then the 8 warps in ascending order, giving
// the shard's own (LSE, entropy); the shards are then reduced in ascending order by
// row_finish (the rank-ordered reduction of page "Perf/cuda compact top p replay",
// Summary). The order depends only on the vocabulary layout, never on T.
constexpr int kMergeRows = 8;
constexpr int kMergeThreads = 256;
constexpr int kMergeGroups = kMergeThreads / kMergeRows;  // 32
constexpr int kMergeWarps = kMergeThreads / 32;           // 8
constexpr int kMergeBatch = 8;                            // blocks per thread loaded ahead of folding

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ MergeParams p) {
  __shared__ Stat part[kMergeWarps][kMergeRows];
  __shared__ float sh_lse[LP_MAX_SHARDS][kMergeRows];
  __shared__ float sh_h[LP_MAX_SHARDS][kMergeRows];
  // launched as the GEMM's programmatic dependent: its statistics are complete and visible
  // once this returns
  grid_dependency_wait();
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int r = tid % kMergeRows;
  const int g = tid / kMergeRows;
  const int row = int(blockIdx.x) * kMergeRows + r;
  const bool in_rows = row < p.T;
  const size_t T = size_t(p.T);
  for (int k = 0; k < p.n_shards; ++k) {
    Stat loc = stat_empty();
    if (in_rows) {
      const int nb_end = p.nb_start[k + 1];
      // batches of kMergeBatch blocks: all their loads are issued before the (dependent) folds
      for (int nb0 = p.nb_start[k] + g; nb0 < nb_end; nb0 += kMergeBatch * kMergeGroups) {
        float m[kMergeBatch], sm[kMergeBatch], am[kMergeBatch];
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
          const int nb = nb0 + i * kMergeGroups;
          const size_t slot = size_t(nb < nb_end ? nb : nb0) * T + size_t(row);
          m[i] = __ldg(p.ws_m + slot);
          sm[i] = __ldg(p.ws_s + slot);
          am[i] = __ldg(p.ws_a + slot);
        }
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i)
          if (nb0 + i * kMergeGroups < nb_end) stat_merge(loc, Stat{m[i], sm[i], am[i]});
      }
    }
    // the warp's four groups of this row: lanes r, r + 8, r + 16, r + 24
#pragma unroll
    for (int off = 16; off >= kMergeRows; off >>= 1) {
      const Stat o{__shfl_down_sync(0xffffffffu, loc.m, off), __shfl_down_sync(0xffffffffu, loc.s, off),
                   __shfl_down_sync(0xffffffffu, loc.a, off)};
      if (lane < off) stat_merge(loc, o);
    }
    if (lane < kMergeRows) part[warp][lane] = loc;
    __syncthreads();
    if (tid < kMergeRows) {
      Stat sh = part[0][tid];
      for (int w = 1; w < kMergeWarps; ++w) stat_merge(sh, part[w][tid]);
      sh_lse[k][tid] = stat_lse(sh);
      sh_h[k][tid] = stat_entropy(sh);
    }
    __syncthreads();  // part is rewritten for the next shard
  }
  if (tid < kMergeRows && in_rows) {
    const int yv = __ldg(p.y + row);
    const bool y_ok = yv >= 0 && int64_t(yv) < p.vocab_real;
    int owner = -1;  // the shard holding y (none: y belongs to another rank's range)
    for (int k = 0; k < p.n_shards; ++k)
      if (y_ok && yv >= p.shard_start[k] && yv < p.shard_end[k]) owner = k;
    const float tv = owner >= 0 ? p.ws_t[row] : 0.f;
    float lse[LP_MAX_SHARDS], h[LP_MAX_SHARDS], t[LP_MAX_SHARDS];
#pragma unroll
    for (int k = 0; k < LP_MAX_SHARDS; ++k) {
      lse[k] = k < p.n_shards ? sh_lse[k][tid] : -INFINITY;
      h[k] = k < p.n_shards ? sh_h[k][tid] : 0.f;
      t[k] = k == owner ? tv : 0.f;
    }
    if (p.shard_stats != nullptr) {
#pragma unroll
      for (int k = 0; k < LP_MAX_SHARDS; ++k) {
        if (k < p.n_shards) {
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
}

cudaError_t launch_fused_forward(const FwdParams& p, int num_sms, cudaStream_t s) {
  // the W maps were encoded with boxes of kGemmBlockN / cluster rows to match (lp_api.cu)
  if (p.num_m_blocks == 1) return launch_tc_gemm<LogpEpi<1>>(p, num_sms, s);
  return launch_tc_gemm<LogpEpi<kFwdClusterM>>(p, num_sms, s);
}

// Launched with programmatic stream serialisation, so that its launch overlaps the end of the
// GEMM that precedes it on the stream (merge_kernel waits for that GEMM's completion first).
cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((p.T + kMergeRows - 1) / kMergeRows), 1, 1);
  cfg.blockDim = dim3(kMergeThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, merge_kernel, p);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

}  // namespace lp
