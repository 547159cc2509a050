// lp_backward.cu - deterministic backward of the linear-logp operator.
//
// Gradient of sum_t g_t * logp_t (+ sum_t h_t * entropy_t), the quantity whose
// autograd the provider contract of page "feat(rl-kernel): add CUDA linear logp
// provider integration" (Summary: logp and optional entropy, detached gradients
// rejected) requires. With p = softmax(z) over the real vocabulary, the merged LSE
// and entropy of the forward and mu = LSE - entropy:
//     G[t, v] = (g_t (1[v = y_t] - p_tv) - h_t p_tv (z_tv - mu_t)) / tau   (0 on padded ids)
//     dX = sum_k G_k W_k,   dW_k = G_k^T X,   db_k = sum_t G_k.
//
// Steps (all in the caller's workspace; nothing is allocated):
//   1. the G kernel: the forward's projection X W_k^T recomputed tile by tile on the
//      tensor core (CTA pairs on the paired-SM MMA); its epilogue forms G from the
//      accumulator and the saved LSE and writes it once, bf16 [T, Vc];
//   2. dW_k^T = X^T G_k: tcgen05 GEMM with both operands read MN-major straight from
//      X [T, H] and G [T, Vc] (K = T), CTA pairs each holding half of the G tile; the
//      epilogue stores each accumulator row h as column h of dW_k;
//   3. dX = G W: tcgen05 GEMM, A = G (K-major), B = W_k read MN-major from each
//      shard's own weight (K = every shard's columns in ascending order), split into
//      a fixed number of K ranges (a function of the vocabulary only) whose fp32
//      partials are then summed in ascending order;
//   4. db_k: the G kernel's epilogue also sums each 32-row slice of every G column (a
//      fixed butterfly across the warp) into a partial; the partials of a column are then
//      added in ascending row order.
// Column layout of G: shard k occupies columns [coff_k, coff_k + real_k) with coff_k a
// multiple of 64 and zero columns up to coff_{k+1}, so K blocks never straddle shards
// and padded ids contribute exactly zero.
#include <cuda_bf16.h>

#include <cstring>

#include "lp_tcgemm.cuh"

namespace lp {

namespace {

constexpr int kSplitChunkCols = 32768;  // dX splits K into Vc / 32768 ranges (1..8)
constexpr int kDbRows = 32;             // rows per db partial sum (one epilogue warp)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct BwdLayout {
  int64_t Vc;
  int64_t coff[LP_MAX_SHARDS + 1];
  int split;
  int64_t db_chunks;
  size_t off_g, off_part, off_db, total;
};

BwdLayout bwd_layout(int64_t T, int64_t H, const Shards& sh) {
  BwdLayout L;
  int64_t c = 0;
  for (int k = 0; k < sh.n; ++k) {
    L.coff[k] = c;
    c += (sh.real[k] + 63) / 64 * 64;
  }
  L.coff[sh.n] = c;
  L.Vc = c;
  int split = int(c / kSplitChunkCols);
  L.split = split < 1 ? 1 : (split > 8 ? 8 : split);
  // one partial per 32-row warp slice of every 128-row block, blocks counted in whole clusters
  L.db_chunks = (T + kFwdBlockM * kFwdClusterM - 1) / (kFwdBlockM * kFwdClusterM) * kFwdClusterM *
                (kFwdBlockM / kDbRows);
  size_t off = 0;
  L.off_g = off;
  off += align_up(size_t(T) * size_t(L.Vc) * 2, 256);
  L.off_part = off;
  if (L.split > 1) off += align_up(size_t(L.split) * size_t(T) * size_t(H) * 4, 256);
  L.off_db = off;
  off += align_up(size_t(L.db_chunks) * size_t(L.Vc) * 4, 256);
  L.total = off;
  return L;
}

__device__ __forceinline__ float f32(uint32_t r) { return __uint_as_float(r); }

// The backward's large outputs (G, 1.2 GB at the headline size, and dW) stream through L2
// once; storing them with an evict-first policy keeps the GEMM operands (X, W, G slices)
// resident instead. LP_BWD_STORE_EVICT_FIRST=0 stores them with the default policy.
#ifndef LP_BWD_STORE_EVICT_FIRST
#define LP_BWD_STORE_EVICT_FIRST 1
#endif

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// one 32-byte store (a whole sector per lane); p must be 32-byte aligned
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* v, uint64_t pol) {
#if LP_BWD_STORE_EVICT_FIRST
  asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "l"(pol)
               : "memory");
#else
  (void)pol;
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
#endif
}

__device__ __forceinline__ void st_global_f32(float* p, float v, uint64_t pol) {
#if LP_BWD_STORE_EVICT_FIRST
  asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(__float_as_uint(v)), "l"(pol) : "memory");
#else
  (void)pol;
  *p = v;
#endif
}

__device__ __forceinline__ void st_global_bf16(__nv_bfloat16* p, float v, uint64_t pol) {
#if LP_BWD_STORE_EVICT_FIRST
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(p), "h"(*reinterpret_cast<const uint16_t*>(&b)),
               "l"(pol)
               : "memory");
#else
  (void)pol;
  *p = __float2bfloat16_rn(v);
#endif
}

// r[i] for a run-time i in [0, 32) without indexing the register array
__device__ __forceinline__ float reg_pick(const uint32_t (&r)[32], int i) {
  float v = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) v = j == i ? __uint_as_float(r[j]) : v;
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Column sums of a 32 x 32 block held one row per lane (v[j] = column j of this lane's
// row): a butterfly that halves the columns each lane keeps at every step (16, 8, 4, 2,
// 1 columns exchanged with lane ^ 16, ^ 8, ...), so after 31 shuffles lane l holds the
// sum of column l over the 32 rows. The order of the additions is fixed.
__device__ __forceinline__ float warp_column_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int j = 0; j < s; ++j) {
      const float send = up ? v[j] : v[j + s];
      const float keep = up ? v[j + s] : v[j];
      v[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, s));
    }
  }
  return v[0];
}

// dX = sum_s part[s] in ascending s (vectors of 4), stored as fp32, or rounded once to
// bf16 when kBf16
template <bool kBf16>
__global__ void __launch_bounds__(256) reduce_split_kernel(const float4* __restrict__ part, int split, size_t n4,
                                                            void* __restrict__ out) {
  const size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  float4 acc = part[i];
  for (int s = 1; s < split; ++s) {
    const float4 v = part[size_t(s) * n4 + i];
    acc.x = __fadd_rn(acc.x, v.x);
    acc.y = __fadd_rn(acc.y, v.y);
    acc.z = __fadd_rn(acc.z, v.z);
    acc.w = __fadd_rn(acc.w, v.w);
  }
  if (kBf16) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    reinterpret_cast<uint2*>(out)[i] =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  } else {
    reinterpret_cast<float4*>(out)[i] = acc;
  }
}

// db[v] = sum_c part[c][col0 + v] in ascending c for v < real; 0 for real <= v < width.
// With accumulate the sum is added to db[v] and padded ids keep their value.
__global__ void __launch_bounds__(256) db_reduce_kernel(const float* __restrict__ part, int64_t Vc, int64_t chunks,
                                                         int64_t col0, int64_t real, int64_t width, int accumulate,
                                                         float* __restrict__ db) {
  const int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (v >= width) return;
  float acc = 0.f;
  if (v < real)
    for (int64_t c = 0; c < chunks; ++c) acc = __fadd_rn(acc, part[c * Vc + col0 + v]);
  if (!accumulate)
    db[v] = acc;
  else if (v < real)
    db[v] = __fadd_rn(db[v], acc);
}

}  // namespace

// ------------------------------------------------------------- G epilogue
struct GradParams {
  CUtensorMap maps[kGemmMaps];  // [0] X; [1 + k] W_k
  uint32_t keep_maps;
  int32_t total_tiles;
  unsigned int* err;
  uint64_t wait_limit_ns;
  const __nv_bfloat16* bias[LP_MAX_SHARDS];
  const int32_t* y;
  const float* lse;
  const float* grad;
  const float* entropy;       // or NULL
  const float* grad_entropy;  // or NULL
  uint16_t* G;  // [T][Vc]
  float* dbp;   // [4 * num_m_blocks][Vc] per-warp column sums of G, or NULL (no bias gradient)
  int64_t Vc;
  int64_t db_chunks;  // rows of dbp (the extent the bounds-checked build compares with)
  int64_t coff[LP_MAX_SHARDS + 1];
  int64_t shard_start[LP_MAX_SHARDS];
  int32_t real[LP_MAX_SHARDS];
  int32_t width[LP_MAX_SHARDS];  // ids of each shard: the length of its bias
  int32_t nb_start[LP_MAX_SHARDS + 1];
  int64_t vocab_real;
  int32_t n_shards;
  int32_t T;
  int32_t num_m_blocks;
  int32_t num_k_blocks;
  int32_t m_chunk;  // row blocks per tile-order chunk
  float scale_log2;
  float inv_tau;
};

struct GradEpi : GemmEpiBase {
  using Params = GradParams;
  static constexpr int kClusterM = kFwdClusterM;

  struct Coord {
    int shard, nb_local, mb;
  };

  static __device__ __forceinline__ Coord coord(const Params& p, int tile) {
    Coord c;
    int nbg;
    proj_raster(tile, p.num_m_blocks, p.m_chunk, p.nb_start[p.n_shards], c.mb, nbg);
    int k = 0;
    while (k + 1 < p.n_shards && nbg >= p.nb_start[k + 1]) ++k;
    c.shard = k;
    c.nb_local = nbg - p.nb_start[k];
    return c;
  }

  static __device__ __forceinline__ TileJob job(const Params& p, int tile) {
    const Coord c = coord(p, tile);
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
    const Coord c = coord(p, tile);
    const int row = c.mb * kGemmBlockM + q * 32 + lane;
    const int64_t n0 = int64_t(c.nb_local) * kGemmBlockN;
    const int64_t real = p.real[c.shard];
    const int valid = int(real - n0 < kGemmBlockN ? real - n0 : kGemmBlockN);
    const int64_t span = (real + 63) / 64 * 64 - n0;  // columns up to the next shard
    const int wlim = int(span < kGemmBlockN ? span : kGemmBlockN);
    const bool in_rows = row < p.T;
    float gi = 0.f, lse2 = 0.f, hi = 0.f, mu = 0.f;
    int64_t ycol = -1;
    bool live = false;
    if (in_rows) {
      const float l = __ldg(p.lse + row);
      const float g = __ldg(p.grad + row);
      const int yv = __ldg(p.y + row);
      // rows without a finite LSE or a valid target get no gradient
      if (isfinite(l) && isfinite(g) && yv >= 0 && int64_t(yv) < p.vocab_real) {
        live = true;
        gi = __fmul_rn(g, p.inv_tau);
        lse2 = __fmul_rn(l, kLog2e);
        ycol = int64_t(yv) - p.shard_start[c.shard] - n0;
        if (p.grad_entropy != nullptr) {
          const float h = __ldg(p.grad_entropy + row);
          const float e = __ldg(p.entropy + row);
          if (isfinite(h) && isfinite(e)) {
            hi = __fmul_rn(h, p.inv_tau);
            mu = __fsub_rn(l, e);  // sum_v p_v z_v = LSE - entropy
          }
        }
      }
    }
    const __nv_bfloat16* bias = p.bias[c.shard];
    const uint64_t pol = l2_policy_evict_first();
    const int64_t col_base = p.coff[c.shard] + n0;
    uint16_t* grow = p.G + size_t(in_rows ? row : 0) * size_t(p.Vc) + size_t(col_base);
    float* dbrow = p.dbp != nullptr ? p.dbp + (size_t(c.mb) * 4 + size_t(q)) * size_t(p.Vc) + size_t(col_base) : nullptr;
    // the bias of column 32 ch + j sits in lane j; the next chunk's is fetched while this
    // chunk is formed
    auto bias_of = [&](int ch) {
      return (bias != nullptr && ch * 32 + lane < valid &&
              in_bounds(n0 + ch * 32 + lane < p.width[c.shard], p.err))
                 ? __bfloat162float(bias[n0 + ch * 32 + lane])
                 : 0.f;
    };
    float bl_next = bias_of(0);
#pragma unroll 1
    for (int ch = 0; ch < kGemmBlockN / 32; ++ch) {
      if (ch * 32 >= wlim) break;
      const float bl = bl_next;
      if (ch + 1 < kGemmBlockN / 32) bl_next = bias_of(ch + 1);
      float gv[32];
      if (ch * 32 < valid) {
        uint32_t r[32];
        tmem_ld32(tbase + ch * 32, r);
        if (p.grad_entropy == nullptr) {
          // logp term only. Every column first takes the non-target value g (0 - p) / tau
          // (the same two roundings as the general form below, so the bits agree with it);
          // the lane whose target falls in this chunk then replaces that one column.
          if (bias != nullptr) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float v = __fadd_rn(f32(r[j]), __shfl_sync(0xffffffffu, bl, j));
              gv[j] = __fmul_rn(gi, __fsub_rn(0.f, hw_ex2(__fmaf_rn(v, p.scale_log2, -lse2))));
            }
          } else {  // acc + 0 differs from acc only in the sign of a zero, which 2^d ignores
#pragma unroll
            for (int j = 0; j < 32; ++j)
              gv[j] = __fmul_rn(gi, __fsub_rn(0.f, hw_ex2(__fmaf_rn(f32(r[j]), p.scale_log2, -lse2))));
          }
          // (a target in a later shard can fall past `valid` of this shard's last block;
          // that column is masked below and its bias is not read)
          const int64_t tc = ycol - ch * 32;
          if (tc >= 0 && tc < 32 && ch * 32 + tc < valid) {
            const int t = int(tc);
            const float b = (bias != nullptr && in_bounds(n0 + ch * 32 + t < p.width[c.shard], p.err))
                                ? __bfloat162float(bias[n0 + ch * 32 + t])
                                : 0.f;
            const float pr = hw_ex2(__fmaf_rn(__fadd_rn(reg_pick(r, t), b), p.scale_log2, -lse2));
            const float gt = __fmul_rn(gi, __fsub_rn(1.f, pr));
#pragma unroll
            for (int j = 0; j < 32; ++j) gv[j] = j == t ? gt : gv[j];
          }
          if (!live || ch * 32 + 32 > valid) {
#pragma unroll
            for (int j = 0; j < 32; ++j) gv[j] = (live && ch * 32 + j < valid) ? gv[j] : 0.f;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = ch * 32 + j;
            const float v = __fadd_rn(f32(r[j]), __shfl_sync(0xffffffffu, bl, j));
            const float pr = hw_ex2(__fmaf_rn(v, p.scale_log2, -lse2));
            const float oh = (int64_t(col) == ycol) ? 1.f : 0.f;
            // logp term g (1[v = y] - p) / tau, entropy term - h p (z - mu) / tau
            float gval = __fmul_rn(gi, __fsub_rn(oh, pr));
            // (p = 0 adds nothing; skipping it keeps a -inf-biased id from forming 0 * -inf)
            if (hi != 0.f && pr != 0.f)
              gval = __fsub_rn(gval, __fmul_rn(__fmul_rn(hi, pr), __fsub_rn(__fmul_rn(v, p.inv_tau), mu)));
            gv[j] = (col < valid && live) ? gval : 0.f;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) gv[j] = 0.f;
      }
      // 64 bytes of this row (two whole-sector stores) inside its Vc columns
      if (in_rows && in_bounds(col_base + ch * 32 + 32 <= p.Vc, p.err)) {
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) packed[j] = pack_bf16(gv[2 * j], gv[2 * j + 1]);
        st_global_v8(grow + ch * 32, packed, pol);
        st_global_v8(grow + ch * 32 + 16, packed + 8, pol);
      }
      // bias gradient: this warp's 32 rows of the chunk's 32 columns, summed in fp32
      if (dbrow != nullptr &&
          in_bounds(int64_t(c.mb) * 4 + q < p.db_chunks && col_base + ch * 32 + 32 <= p.Vc, p.err))
        dbrow[ch * 32 + lane] = warp_column_sum(gv, lane);
    }
  }
};

// ------------------------------------------------------------------- dW
// Tile = (vocabulary block of one shard, row block of H), row blocks fastest. The
// accumulator holds dW_k^T: TMEM lane = h, column = vocabulary id, so each thread
// stores its row h into column h of 256 rows of dW_k (a warp writes 128 contiguous
// bytes of one dW row per store).
struct DwParams {
  CUtensorMap maps[kGemmMaps];  // [0] X [T, H] (MN-major boxes 64 h x 64 t); [1] G [T, Vc] (64 v x 64 t)
  uint32_t keep_maps;
  int32_t total_tiles;
  unsigned int* err;
  uint64_t wait_limit_ns;
  void* dW[LP_MAX_SHARDS];  // float, or bf16 with dw_bf16
  int64_t width[LP_MAX_SHARDS];  // rows of dW_k
  int64_t coff[LP_MAX_SHARDS];
  int32_t real[LP_MAX_SHARDS];
  int32_t nb_start[LP_MAX_SHARDS + 1];
  int32_t n_shards;
  int32_t num_m_blocks;  // row blocks of H, counted in whole clusters
  int32_t nkb;           // K blocks over T
  int32_t accumulate;    // dW += G^T X instead of dW = G^T X
  int32_t dw_bf16;       // store dW rounded to bf16
  int64_t H;
};

struct DwEpi : GemmEpiBase {
  using Params = DwParams;
  static constexpr int kClusterM = kFwdClusterM;
  static constexpr bool kAMN = true;
  static constexpr bool kBMN = true;

  struct Coord {
    int shard, nb_local, mb;
  };

  static __device__ __forceinline__ Coord coord(const Params& p, int tile) {
    Coord c;
    c.mb = tile % p.num_m_blocks;
    const int nbg = tile / p.num_m_blocks;
    int k = 0;
    while (k + 1 < p.n_shards && nbg >= p.nb_start[k + 1]) ++k;
    c.shard = k;
    c.nb_local = nbg - p.nb_start[k];
    return c;
  }

  static __device__ __forceinline__ TileJob job(const Params& p, int tile) {
    const Coord c = coord(p, tile);
    TileJob j;
    j.a_map = 0;
    j.a_y = c.mb * kGemmBlockM;
    j.b_map = 1;
    j.b_y = int(p.coff[c.shard]) + c.nb_local * kGemmBlockN;
    j.kb0 = 0;
    j.nkb = p.nkb;
    return j;
  }

  static __device__ __forceinline__ void run(const Params& p, int tile, int /*half*/, uint32_t tbase, int q,
                                             int lane) {
    const Coord c = coord(p, tile);
    const int64_t h = int64_t(c.mb) * kGemmBlockM + q * 32 + lane;
    const int64_t v0 = int64_t(c.nb_local) * kGemmBlockN;
    const int64_t left = p.real[c.shard] - v0;
    const int valid = int(left < kGemmBlockN ? left : kGemmBlockN);
    // rows v0 .. v0 + valid of dW_k: within its width rows
    const bool ok = h < p.H && in_bounds(v0 + valid <= p.width[c.shard], p.err);
    const size_t off = size_t(v0) * size_t(p.H) + size_t(ok ? h : 0);
    const uint64_t pol = l2_policy_evict_first();
    if (p.dw_bf16) {  // a warp stores 64 contiguous bytes of one dW row per instruction
      __nv_bfloat16* b16 = static_cast<__nv_bfloat16*>(p.dW[c.shard]) + off;
#pragma unroll 1
      for (int ch = 0; ch < kGemmBlockN / 32; ++ch) {
        if (ch * 32 >= valid) break;
        uint32_t r[32];
        tmem_ld32(tbase + ch * 32, r);
        if (ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (ch * 32 + j < valid) st_global_bf16(b16 + size_t(ch * 32 + j) * size_t(p.H), f32(r[j]), pol);
        }
      }
      return;
    }
    float* base = static_cast<float*>(p.dW[c.shard]) + off;
#pragma unroll 1
    for (int ch = 0; ch < kGemmBlockN / 32; ++ch) {
      if (ch * 32 >= valid) break;
      uint32_t r[32];
      tmem_ld32(tbase + ch * 32, r);
      if (ok && p.accumulate) {
        // read-add-write in groups of 8 rows (8 loads in flight, few live registers)
#pragma unroll
        for (int j0 = 0; j0 < 32; j0 += 8) {
          float old[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (ch * 32 + j0 + j < valid) old[j] = base[size_t(ch * 32 + j0 + j) * size_t(p.H)];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (ch * 32 + j0 + j < valid)
              st_global_f32(base + size_t(ch * 32 + j0 + j) * size_t(p.H), __fadd_rn(old[j], f32(r[j0 + j])), pol);
        }
      } else if (ok) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (ch * 32 + j < valid) st_global_f32(base + size_t(ch * 32 + j) * size_t(p.H), f32(r[j]), pol);
      }
    }
  }
};

// ------------------------------------------------------------------- dX
// Tile = (block of 256 rows of T, column block of H, K range s): each CTA accumulates
// two 128-row halves into all 512 TMEM columns (the K loop over a ~38K-long range dwarfs
// the epilogue, so no second accumulator is needed), which halves the A-tile loads per
// FLOP and doubles the output each wave of tiles covers. Within a K range, row blocks go
// in groups of kDxGroupM: inside a group the row block runs fastest, then the column
// block, so the tiles in flight share both operands' K slices through L2. A = G (K-major,
// K = global column), B = W_k read MN-major from the shard holding each K block; partial
// s goes to out + s*T*H.
struct DxParams {
  CUtensorMap maps[kGemmMaps];  // [0] G [T, Vc] (boxes 64 v x 128 t); [1 + k] W_k [real_k, H] (64 h x 64 v)
  uint32_t keep_maps;
  int32_t total_tiles;
  unsigned int* err;
  uint64_t wait_limit_ns;
  float* out;            // fp32 partial s at out + s*T*H, or (one K range) dX itself
  uint16_t* out_bf16;    // one K range and bf16 dX: dX rounded in the epilogue (out unused)
  int64_t coff[LP_MAX_SHARDS + 1];
  int32_t n_shards;
  int32_t num_m_blocks;  // row blocks of T, counted in whole clusters
  int32_t num_n;
  int32_t nkb_total;
  int32_t kb_per_split;
  int32_t splits;  // fp32 partials in out (the extent the bounds-checked build compares with)
  int64_t T, H;
};

struct DxEpi : GemmEpiBase {
  using Params = DxParams;
  static constexpr int kClusterM = kFwdClusterM;
  static constexpr bool kBMN = true;
  static constexpr int kMHalves = 2;  // 256-row tiles: the K loop (a K range of ~38K) dwarfs the epilogue
  static constexpr int kRows = kMHalves * kGemmBlockM;

  struct Coord {
    int mb, nb, s;
  };

  static constexpr int kDxGroupM = 8;  // row blocks of 256 per group; even, so cluster pairs never straddle groups

  static __device__ __forceinline__ Coord coord(const Params& p, int tile) {
    Coord c;
    const int per_split = p.num_m_blocks * p.num_n;
    c.s = tile / per_split;
    const int r = tile - c.s * per_split;
    const int g = r / (kDxGroupM * p.num_n);
    const int within = r - g * kDxGroupM * p.num_n;
    const int left = p.num_m_blocks - g * kDxGroupM;
    const int gs = left < kDxGroupM ? left : kDxGroupM;
    c.nb = within / gs;
    c.mb = g * kDxGroupM + within % gs;
    return c;
  }

  static __device__ __forceinline__ TileJob job(const Params& p, int tile) {
    const Coord c = coord(p, tile);
    TileJob j;
    j.a_map = 0;
    j.a_y = c.mb * kRows;
    j.b_map = 1;
    j.b_y = c.nb * kGemmBlockN;
    j.kb0 = c.s * p.kb_per_split;
    const int left = p.nkb_total - j.kb0;
    j.nkb = left < p.kb_per_split ? left : p.kb_per_split;
    return j;
  }

  // the W map and local row of global K block kb0 + kb: the shard whose columns hold it
  static __device__ __forceinline__ void b_k(const void* pp, const TileJob& j, int kb, int& map, int& k) {
    const Params& p = *static_cast<const Params*>(pp);
    const int64_t col = int64_t(j.kb0 + kb) * kFwdBlockK;
    int s = 0;
    while (s + 1 < p.n_shards && col >= p.coff[s + 1]) ++s;
    map = 1 + s;
    k = int(col - p.coff[s]);
  }

  static __device__ __forceinline__ void run(const Params& p, int tile, int half, uint32_t tbase, int q,
                                             int lane) {
    const Coord c = coord(p, tile);
    const int64_t row = int64_t(c.mb) * kRows + half * kGemmBlockM + q * 32 + lane;
    const int64_t c0 = int64_t(c.nb) * kGemmBlockN;
    const int64_t cols = p.H - c0 < kGemmBlockN ? p.H - c0 : kGemmBlockN;
    const bool ok = row < p.T && in_bounds(c.s < p.splits && c0 + cols <= p.H, p.err);
    if (p.out_bf16 != nullptr) {
      // H % 8 == 0, so 8-column groups are whole: one 16-byte store per group
      uint16_t* dst = p.out_bf16 + size_t(ok ? row : 0) * size_t(p.H) + size_t(c0);
#pragma unroll 1
      for (int ch = 0; ch < kGemmBlockN / 32; ++ch) {
        if (ch * 32 >= cols) break;
        uint32_t r[32];
        tmem_ld32(tbase + ch * 32, r);
        if (ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (ch * 32 + v * 8 >= cols) break;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 b = __floats2bfloat162_rn(f32(r[8 * v + 2 * e]), f32(r[8 * v + 2 * e + 1]));
              w[e] = *reinterpret_cast<const uint32_t*>(&b);
            }
            *reinterpret_cast<uint4*>(dst + ch * 32 + v * 8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      return;
    }
    float* dst = p.out + size_t(c.s) * size_t(p.T) * size_t(p.H) + size_t(ok ? row : 0) * size_t(p.H);
#pragma unroll 1
    for (int ch = 0; ch < kGemmBlockN / 32; ++ch) {
      if (ch * 32 >= cols) break;
      uint32_t r[32];
      tmem_ld32(tbase + ch * 32, r);
      if (ok) {
        float4* d4 = reinterpret_cast<float4*>(dst + c0 + ch * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          if (ch * 32 + v * 4 < cols)
            d4[v] = make_float4(f32(r[4 * v]), f32(r[4 * v + 1]), f32(r[4 * v + 2]), f32(r[4 * v + 3]));
      }
    }
  }
};

namespace {

// bf16 [rows, inner] with row stride ld as MN-major atoms: boxes of 64 (inner) x 64 rows
bool encode_mn_atoms(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t ld) {
  return encode_bf16_2d(m, base, inner, rows, ld, 64);
}

int32_t pad_to_cluster(int64_t blocks) {
  return int32_t((blocks + kFwdClusterM - 1) / kFwdClusterM * kFwdClusterM);
}

}  // namespace

size_t backward_ws_bytes(int64_t T, int64_t H, const Shards& sh) { return bwd_layout(T, H, sh).total; }

lp_status run_backward(const BackwardArgs& a, const Shards& sh, cudaStream_t s) {
  const BwdLayout L = bwd_layout(a.T, a.H, sh);
  char* ws = static_cast<char*>(a.workspace);
  uint16_t* G = reinterpret_cast<uint16_t*>(ws + L.off_g);
  float* part = reinterpret_cast<float*>(ws + L.off_part);
  float* dbp = reinterpret_cast<float*>(ws + L.off_db);
  const int64_t T = a.T, H = a.H;

  // 1. G
  {
    GradParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_bf16_2d(&p.maps[0], a.X, uint64_t(H), uint64_t(T), uint64_t(H), kFwdBlockM)) return LP_ERR_CUDA;
    int nb = 0;
    for (int k = 0; k < sh.n; ++k) {
      if (sh.real[k] > 0 && !encode_bf16_2d(&p.maps[1 + k], a.W[k], uint64_t(H), uint64_t(sh.width[k]),
                                            uint64_t(H), kFwdBlockN / kFwdClusterM))
        return LP_ERR_CUDA;
      p.bias[k] = static_cast<const __nv_bfloat16*>(a.bias[k]);
      p.coff[k] = L.coff[k];
      p.shard_start[k] = sh.start[k];
      p.real[k] = int32_t(sh.real[k]);
      p.width[k] = int32_t(sh.width[k]);
      p.nb_start[k] = nb;
      nb += int((sh.real[k] + kFwdBlockN - 1) / kFwdBlockN);
    }
    p.coff[sh.n] = L.coff[sh.n];
    p.nb_start[sh.n] = nb;
    p.keep_maps = 1u;
    p.n_shards = sh.n;
    p.T = int32_t(T);
    p.num_m_blocks = pad_to_cluster((T + kFwdBlockM - 1) / kFwdBlockM);
    p.num_k_blocks = int32_t((H + kFwdBlockK - 1) / kFwdBlockK);
    p.m_chunk = proj_row_chunk(H, p.num_m_blocks);
    p.total_tiles = nb * p.num_m_blocks;
    p.err = a.err;
    p.wait_limit_ns = wait_limit_ns();
    p.y = a.y;
    p.lse = a.lse;
    p.grad = a.grad;
    p.entropy = a.entropy;
    p.grad_entropy = a.grad_entropy;
    p.G = G;
    p.Vc = L.Vc;
    p.db_chunks = L.db_chunks;
    bool any_db = false;
    for (int k = 0; k < sh.n; ++k) any_db = any_db || (a.db[k] != nullptr && sh.width[k] > 0);
    p.dbp = any_db ? dbp : nullptr;
    p.vocab_real = sh.vocab_real;
    p.scale_log2 = float(1.4426950408889634 / double(a.tau));
    p.inv_tau = float(1.0 / double(a.tau));
    if (launch_tc_gemm<GradEpi>(p, a.num_sms, s) != cudaSuccess) return LP_ERR_CUDA;
  }

  // 2. dW_k (and zero rows of padded ids)
  {
    DwParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_mn_atoms(&p.maps[0], a.X, uint64_t(H), uint64_t(T), uint64_t(H)) ||
        !encode_mn_atoms(&p.maps[1], G, uint64_t(L.Vc), uint64_t(T), uint64_t(L.Vc)))
      return LP_ERR_CUDA;
    p.keep_maps = 1u;  // X is re-read by every vocabulary block
    int nb = 0;
    for (int k = 0; k < sh.n; ++k) {
      p.dW[k] = a.dW[k];
      p.width[k] = sh.width[k];
      p.coff[k] = L.coff[k];
      p.real[k] = int32_t(sh.real[k]);
      p.nb_start[k] = nb;
      nb += int((sh.real[k] + kFwdBlockN - 1) / kFwdBlockN);
    }
    p.nb_start[sh.n] = nb;
    p.n_shards = sh.n;
    p.num_m_blocks = pad_to_cluster((H + kFwdBlockM - 1) / kFwdBlockM);
    p.nkb = int32_t((T + kFwdBlockK - 1) / kFwdBlockK);
    p.H = H;
    p.total_tiles = nb * p.num_m_blocks;
    p.accumulate = a.accumulate;
    p.dw_bf16 = a.dw_bf16;
    p.err = a.err;
    p.wait_limit_ns = wait_limit_ns();
    if (launch_tc_gemm<DwEpi>(p, a.num_sms, s) != cudaSuccess) return LP_ERR_CUDA;
    const size_t esz = a.dw_bf16 ? 2 : 4;
    for (int k = 0; k < sh.n && !a.accumulate; ++k) {
      const int64_t pad = sh.width[k] - sh.real[k];
      if (pad > 0 && cudaMemsetAsync(static_cast<char*>(a.dW[k]) + size_t(sh.real[k]) * size_t(H) * esz, 0,
                                     size_t(pad) * size_t(H) * esz, s) != cudaSuccess)
        return LP_ERR_CUDA;
    }
  }

  // 3. dX = G W
  {
    DxParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_bf16_2d(&p.maps[0], G, uint64_t(L.Vc), uint64_t(T), uint64_t(L.Vc), kFwdBlockM)) return LP_ERR_CUDA;
    for (int k = 0; k < sh.n; ++k)
      if (sh.real[k] > 0 && !encode_mn_atoms(&p.maps[1 + k], a.W[k], uint64_t(H), uint64_t(sh.real[k]), uint64_t(H)))
        return LP_ERR_CUDA;
    for (int k = 0; k <= sh.n; ++k) p.coff[k] = L.coff[k];
    p.keep_maps = 0u;
    p.n_shards = sh.n;
    p.num_m_blocks = pad_to_cluster((T + DxEpi::kRows - 1) / DxEpi::kRows);
    p.num_n = int32_t((H + kFwdBlockN - 1) / kFwdBlockN);
    p.nkb_total = int32_t(L.Vc / kFwdBlockK);
    p.kb_per_split = (p.nkb_total + L.split - 1) / L.split;
    const int splits = (p.nkb_total + p.kb_per_split - 1) / p.kb_per_split;
    p.splits = splits;
    p.T = T;
    p.H = H;
    p.out = splits > 1 ? part : static_cast<float*>(a.dX);
    p.out_bf16 = (splits == 1 && a.dx_bf16) ? static_cast<uint16_t*>(a.dX) : nullptr;
    p.total_tiles = p.num_m_blocks * p.num_n * splits;
    p.err = a.err;
    p.wait_limit_ns = wait_limit_ns();
    if (launch_tc_gemm<DxEpi>(p, a.num_sms, s) != cudaSuccess) return LP_ERR_CUDA;
    if (splits > 1) {
      const size_t n4 = size_t(T) * size_t(H) / 4;
      const unsigned blocks = unsigned((n4 + 255) / 256);
      if (a.dx_bf16)
        reduce_split_kernel<true><<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(part), splits, n4, a.dX);
      else
        reduce_split_kernel<false><<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(part), splits, n4, a.dX);
      if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
    }
  }

  // 4. db: the G kernel wrote per-warp column sums; add them in ascending row order
  {
    for (int k = 0; k < sh.n; ++k) {
      if (a.db[k] == nullptr || sh.width[k] == 0) continue;
      db_reduce_kernel<<<unsigned((sh.width[k] + 255) / 256), 256, 0, s>>>(dbp, L.Vc, L.db_chunks, L.coff[k],
                                                                           sh.real[k], sh.width[k], a.accumulate,
                                                                           a.db[k]);
      if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
    }
  }
  return LP_OK;
}

}  // namespace lp
