// lp_backward.cu - deterministic backward of the linear-logp operator.
//
// Gradient of sum_t g_t * logp_t, the quantity whose autograd the provider contract
// of page "feat(rl-kernel): add CUDA linear logp provider integration" (Summary:
// detached gradients are rejected) requires. With p = softmax(z) over the real
// vocabulary and the merged LSE of the forward:
//     G[t, v] = g_t (1[v = y_t] - exp(z[t, v] - LSE_t)) / tau        (0 on padded ids)
//     dX = sum_k G_k W_k,   dW_k = G_k^T X,   db_k = sum_t G_k.
//
// Steps (all in the caller's workspace; nothing is allocated):
//   1. X^T and W^T (bf16) by tiled transposes, so that every GEMM below has both
//      operands K-major and runs on the same tcgen05 pipeline as the forward;
//   2. the G kernel: the forward's projection X W_k^T recomputed tile by tile on the
//      tensor core; its epilogue forms G from the accumulator and the saved LSE and
//      writes it in bf16 twice, as G [T, Vc] and G^T [Vc, Tp];
//   3. dW_k = G_k^T X: tcgen05 GEMM, A = G^T rows of shard k, B = X^T, K = T;
//   4. dX = G W: tcgen05 GEMM, A = G, B = W^T, K = every shard's columns in
//      ascending order, split into a fixed number of K ranges (a function of the
//      vocabulary only) whose fp32 partials are then summed in ascending order;
//   5. db_k: sums of the rows of G^T, each in a fixed order.
// Column layout of G and W^T: shard k occupies columns [coff_k, coff_k + real_k) with
// coff_k a multiple of 64 and zero columns up to coff_{k+1}, so K blocks never read
// another shard's data and padded ids contribute exactly zero.
#include <cuda_bf16.h>

#include <cstring>

#include "lp_tcgemm.cuh"

namespace lp {

namespace {

constexpr int kSplitChunkCols = 32768;  // dX splits K into Vc / 32768 ranges (1..8)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct BwdLayout {
  int64_t Tp, Vc;
  int64_t coff[LP_MAX_SHARDS + 1];
  int split;
  size_t off_xt, off_wt, off_g, off_gt, off_part, total;
};

BwdLayout bwd_layout(int64_t T, int64_t H, const Shards& sh) {
  BwdLayout L;
  L.Tp = (T + 7) / 8 * 8;
  int64_t c = 0;
  for (int k = 0; k < sh.n; ++k) {
    L.coff[k] = c;
    c += (sh.real[k] + 63) / 64 * 64;
  }
  L.coff[sh.n] = c;
  L.Vc = c;
  int split = int(c / kSplitChunkCols);
  L.split = split < 1 ? 1 : (split > 8 ? 8 : split);
  size_t off = 0;
  L.off_xt = off;
  off += align_up(size_t(H) * size_t(L.Tp) * 2, 256);
  L.off_wt = off;
  off += align_up(size_t(H) * size_t(L.Vc) * 2, 256);
  L.off_g = off;
  off += align_up(size_t(T) * size_t(L.Vc) * 2, 256);
  L.off_gt = off;
  off += align_up(size_t(L.Vc) * size_t(L.Tp) * 2, 256);
  L.off_part = off;
  if (L.split > 1) off += align_up(size_t(L.split) * size_t(T) * size_t(H) * 4, 256);
  L.total = off;
  return L;
}

__device__ __forceinline__ float f32(uint32_t r) { return __uint_as_float(r); }

// out[c][col0 + r] = in[r][c] for r < rows, c < cols (bf16, 32 x 32 tiles through
// shared memory); out[c][col0 + r] = 0 for rows <= r < rows_pad.
__global__ void __launch_bounds__(256) transpose_kernel(const uint16_t* __restrict__ in, int64_t ld_in, int64_t rows,
                                                         int64_t rows_pad, int64_t cols, uint16_t* __restrict__ out,
                                                         int64_t ld_out, int64_t col0) {
  __shared__ uint16_t tile[32][33];
  const int64_t r0 = int64_t(blockIdx.y) * 32;
  const int64_t c0 = int64_t(blockIdx.x) * 32;
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;  // 0..7
  for (int i = ty; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + tx;
    tile[i][tx] = (r < rows && c < cols) ? in[r * ld_in + c] : uint16_t(0);
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + tx;
    if (c < cols && r < rows_pad) out[c * ld_out + col0 + r] = tile[tx][i];
  }
}

// fp32 dX = sum_s part[s] in ascending s (vectors of 4)
__global__ void __launch_bounds__(256) reduce_split_kernel(const float4* __restrict__ part, int split, size_t n4,
                                                            float4* __restrict__ out) {
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
  out[i] = acc;
}

// db[v] = sum_t G^T[row0 + v][t], one warp per v: lane l adds the 8-element vectors
// l, l+32, ... in order, then a fixed shuffle tree.
__global__ void __launch_bounds__(256) bias_grad_kernel(const uint16_t* __restrict__ gt, int64_t ld, int64_t row0,
                                                         int64_t rows, int64_t T, float* __restrict__ db) {
  const int64_t v = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (v >= rows) return;
  const uint4* row = reinterpret_cast<const uint4*>(gt + (row0 + v) * ld);
  const int64_t nvec = (T + 7) / 8;
  float acc = 0.f;
  for (int64_t i = lane; i < nvec; i += 32) {
    const uint4 q = row[i];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t t = i * 8 + j;
      const float x = (j & 1) ? bf16_hi(w[j >> 1]) : bf16_lo(w[j >> 1]);
      if (t < T) acc = __fadd_rn(acc, x);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float o = __shfl_down_sync(0xffffffffu, acc, off);
    if (lane < off) acc = __fadd_rn(acc, o);
  }
  if (lane == 0) db[v] = acc;
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
  uint16_t* G;   // [T][Vc]
  uint16_t* Gt;  // [Vc][Tp]
  int64_t Vc, Tp;
  int64_t coff[LP_MAX_SHARDS + 1];
  int64_t shard_start[LP_MAX_SHARDS];
  int32_t real[LP_MAX_SHARDS];
  int32_t nb_start[LP_MAX_SHARDS + 1];
  int64_t vocab_real;
  int32_t n_shards;
  int32_t T;
  int32_t num_m_blocks;
  int32_t num_k_blocks;
  float scale_log2;
  float inv_tau;
};

struct GradEpi {
  using Params = GradParams;
  static constexpr int kClusterM = kFwdClusterM;

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
    j.b_map = 1 + c.shard;
    j.b_y = c.nb_local * kGemmBlockN;
    j.kb0 = 0;
    j.nkb = p.num_k_blocks;
    return j;
  }

  static __device__ __forceinline__ void run(const Params& p, int tile, uint32_t tbase, int q, int lane) {
    const Coord c = coord(p, tile);
    const int row = c.mb * kGemmBlockM + q * 32 + lane;
    const int64_t n0 = int64_t(c.nb_local) * kGemmBlockN;
    const int64_t real = p.real[c.shard];
    const int valid = int(real - n0 < kGemmBlockN ? real - n0 : kGemmBlockN);
    const int64_t span = (real + 63) / 64 * 64 - n0;  // columns up to the next shard
    const int wlim = int(span < kGemmBlockN ? span : kGemmBlockN);
    const bool in_rows = row < p.T;
    float gi = 0.f, lse2 = 0.f;
    int64_t ycol = -1;
    if (in_rows) {
      const float l = __ldg(p.lse + row);
      const float g = __ldg(p.grad + row);
      const int yv = __ldg(p.y + row);
      // rows without a finite LSE or a valid target get no gradient
      if (isfinite(l) && isfinite(g) && yv >= 0 && int64_t(yv) < p.vocab_real) {
        gi = __fmul_rn(g, p.inv_tau);
        lse2 = __fmul_rn(l, kLog2e);
        ycol = int64_t(yv) - p.shard_start[c.shard] - n0;
      }
    }
    const __nv_bfloat16* bias = p.bias[c.shard];
    const int64_t col_base = p.coff[c.shard] + n0;
    uint16_t* grow = p.G + size_t(in_rows ? row : 0) * size_t(p.Vc) + size_t(col_base);
#pragma unroll 1
    for (int ch = 0; ch < kGemmBlockN / 32; ++ch) {
      if (ch * 32 >= wlim) break;
      float bl = 0.f;
      if (bias != nullptr && ch * 32 + lane < valid) bl = __bfloat162float(bias[n0 + ch * 32 + lane]);
      uint32_t r[32];
      uint32_t packed[16];
      if (ch * 32 < valid) {
        tmem_ld32(tbase + ch * 32, r);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float gv[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = ch * 32 + j + h;
            const float v = __fadd_rn(f32(r[j + h]), __shfl_sync(0xffffffffu, bl, j + h));
            const float pr = hw_ex2(__fmaf_rn(v, p.scale_log2, -lse2));
            const float oh = (int64_t(col) == ycol) ? 1.f : 0.f;
            gv[h] = (col < valid && gi != 0.f) ? __fmul_rn(gi, __fsub_rn(oh, pr)) : 0.f;
          }
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(gv[0], gv[1]);
          packed[j >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) packed[j] = 0u;
      }
      if (in_rows) {
        uint4* dst = reinterpret_cast<uint4*>(grow + ch * 32);
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        dst[2] = make_uint4(packed[8], packed[9], packed[10], packed[11]);
        dst[3] = make_uint4(packed[12], packed[13], packed[14], packed[15]);
        // G^T: column (col_base + ch*32 + j), row `row`; lanes write consecutive rows
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (ch * 32 + j < valid) {
            const uint16_t h = uint16_t((j & 1) ? (packed[j >> 1] >> 16) : (packed[j >> 1] & 0xFFFFu));
            p.Gt[size_t(col_base + ch * 32 + j) * size_t(p.Tp) + size_t(row)] = h;
          }
        }
      }
    }
  }
};

// --------------------------------------------------------- fp32 GEMM store
// mode 0 (dW): tile = (row block of one shard's G^T rows, column block of H),
//              column blocks fastest; K = T.
// mode 1 (dX): tile = (row block of T, column block of H, K range s), row blocks
//              fastest, then column blocks, then s; partial s goes to part[s].
struct StoreParams {
  CUtensorMap maps[kGemmMaps];  // [0] A, [1] B
  uint32_t keep_maps;
  int32_t total_tiles;
  unsigned int* err;
  uint64_t wait_limit_ns;
  int32_t mode;
  int32_t num_m, num_n;
  int32_t nkb_total, kb_per_split;
  int64_t H;
  // mode 0
  float* dW[LP_MAX_SHARDS];
  int32_t mb_start[LP_MAX_SHARDS + 1];
  int64_t coff[LP_MAX_SHARDS];
  int64_t real[LP_MAX_SHARDS];
  int32_t n_shards;
  // mode 1
  float* out;     // dX (split == 1) or partials [split][T][H]
  int64_t T;
};

struct StoreEpi {
  using Params = StoreParams;
  static constexpr int kClusterM = 1;

  struct Coord {
    int shard, mb, nb, s;
  };

  static __device__ __forceinline__ Coord coord(const Params& p, int tile) {
    Coord c;
    if (p.mode == 0) {
      c.nb = tile % p.num_n;
      const int mbg = tile / p.num_n;
      int k = 0;
      while (k + 1 < p.n_shards && mbg >= p.mb_start[k + 1]) ++k;
      c.shard = k;
      c.mb = mbg - p.mb_start[k];
      c.s = 0;
    } else {
      c.mb = tile % p.num_m;
      const int rest = tile / p.num_m;
      c.nb = rest % p.num_n;
      c.s = rest / p.num_n;
      c.shard = 0;
    }
    return c;
  }

  static __device__ __forceinline__ TileJob job(const Params& p, int tile) {
    const Coord c = coord(p, tile);
    TileJob j;
    j.a_map = 0;
    j.b_map = 1;
    j.b_y = c.nb * kGemmBlockN;
    if (p.mode == 0) {
      j.a_y = int(p.coff[c.shard]) + c.mb * kGemmBlockM;
      j.kb0 = 0;
      j.nkb = p.nkb_total;
    } else {
      j.a_y = c.mb * kGemmBlockM;
      j.kb0 = c.s * p.kb_per_split;
      const int left = p.nkb_total - j.kb0;
      j.nkb = left < p.kb_per_split ? left : p.kb_per_split;
    }
    return j;
  }

  static __device__ __forceinline__ void run(const Params& p, int tile, uint32_t tbase, int q, int lane) {
    const Coord c = coord(p, tile);
    const int64_t rloc = int64_t(c.mb) * kGemmBlockM + q * 32 + lane;
    float* dst;
    bool ok;
    if (p.mode == 0) {
      ok = rloc < p.real[c.shard];
      dst = p.dW[c.shard] + size_t(ok ? rloc : 0) * size_t(p.H);
    } else {
      ok = rloc < p.T;
      dst = p.out + size_t(c.s) * size_t(p.T) * size_t(p.H) + size_t(ok ? rloc : 0) * size_t(p.H);
    }
    const int64_t c0 = int64_t(c.nb) * kGemmBlockN;
    const int64_t cols = p.H - c0 < kGemmBlockN ? p.H - c0 : kGemmBlockN;
#pragma unroll 1
    for (int ch = 0; ch < kGemmBlockN / 32; ++ch) {
      if (ch * 32 >= cols) break;
      uint32_t r[32];
      tmem_ld32(tbase + ch * 32, r);
      if (ok) {
        float4* d4 = reinterpret_cast<float4*>(dst + c0 + ch * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          if (ch * 32 + v * 4 < cols) d4[v] = make_float4(f32(r[4 * v]), f32(r[4 * v + 1]), f32(r[4 * v + 2]), f32(r[4 * v + 3]));
      }
    }
  }
};

size_t backward_ws_bytes(int64_t T, int64_t H, const Shards& sh) { return bwd_layout(T, H, sh).total; }

lp_status run_backward(const BackwardArgs& a, const Shards& sh, cudaStream_t s) {
  const BwdLayout L = bwd_layout(a.T, a.H, sh);
  char* ws = static_cast<char*>(a.workspace);
  uint16_t* Xt = reinterpret_cast<uint16_t*>(ws + L.off_xt);
  uint16_t* Wt = reinterpret_cast<uint16_t*>(ws + L.off_wt);
  uint16_t* G = reinterpret_cast<uint16_t*>(ws + L.off_g);
  uint16_t* Gt = reinterpret_cast<uint16_t*>(ws + L.off_gt);
  float* part = reinterpret_cast<float*>(ws + L.off_part);
  const int64_t T = a.T, H = a.H;

  // 1. transposes
  {
    dim3 grid(unsigned((H + 31) / 32), unsigned((T + 31) / 32));
    transpose_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(a.X), H, T, T, H, Xt, L.Tp, 0);
    if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
    for (int k = 0; k < sh.n; ++k) {
      const int64_t rp = L.coff[k + 1] - L.coff[k];
      if (rp == 0) continue;
      dim3 g2(unsigned((H + 31) / 32), unsigned((rp + 31) / 32));
      transpose_kernel<<<g2, 256, 0, s>>>(static_cast<const uint16_t*>(a.W[k]), H, sh.real[k], rp, H, Wt, L.Vc,
                                           L.coff[k]);
      if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
    }
  }

  // 2. G and G^T
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
      p.nb_start[k] = nb;
      nb += int((sh.real[k] + kFwdBlockN - 1) / kFwdBlockN);
    }
    p.coff[sh.n] = L.coff[sh.n];
    p.nb_start[sh.n] = nb;
    p.keep_maps = 1u;
    p.n_shards = sh.n;
    p.T = int32_t(T);
    const int64_t mblocks = (T + kFwdBlockM - 1) / kFwdBlockM;
    p.num_m_blocks = int32_t((mblocks + kFwdClusterM - 1) / kFwdClusterM * kFwdClusterM);
    p.num_k_blocks = int32_t((H + kFwdBlockK - 1) / kFwdBlockK);
    p.total_tiles = nb * p.num_m_blocks;
    p.err = a.err;
    p.wait_limit_ns = kDefaultWaitLimitNs;
    p.y = a.y;
    p.lse = a.lse;
    p.grad = a.grad;
    p.G = G;
    p.Gt = Gt;
    p.Vc = L.Vc;
    p.Tp = L.Tp;
    p.vocab_real = sh.vocab_real;
    p.scale_log2 = float(1.4426950408889634 / double(a.tau));
    p.inv_tau = float(1.0 / double(a.tau));
    if (launch_tc_gemm<GradEpi>(p, a.num_sms, s) != cudaSuccess) return LP_ERR_CUDA;
  }

  // 3. dW_k = G_k^T X  (and zero rows of padded ids)
  {
    StoreParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_bf16_2d(&p.maps[0], Gt, uint64_t(T), uint64_t(L.Vc), uint64_t(L.Tp), kFwdBlockM) ||
        !encode_bf16_2d(&p.maps[1], Xt, uint64_t(T), uint64_t(H), uint64_t(L.Tp), kFwdBlockN))
      return LP_ERR_CUDA;
    p.keep_maps = 2u;  // X^T is reused by every row block
    p.mode = 0;
    p.num_n = int32_t((H + kFwdBlockN - 1) / kFwdBlockN);
    p.nkb_total = int32_t((T + kFwdBlockK - 1) / kFwdBlockK);
    p.H = H;
    int mb = 0;
    for (int k = 0; k < sh.n; ++k) {
      p.dW[k] = a.dW[k];
      p.mb_start[k] = mb;
      p.coff[k] = L.coff[k];
      p.real[k] = sh.real[k];
      mb += int((sh.real[k] + kFwdBlockM - 1) / kFwdBlockM);
    }
    p.mb_start[sh.n] = mb;
    p.n_shards = sh.n;
    p.total_tiles = mb * p.num_n;
    p.err = a.err;
    p.wait_limit_ns = kDefaultWaitLimitNs;
    if (launch_tc_gemm<StoreEpi>(p, a.num_sms, s) != cudaSuccess) return LP_ERR_CUDA;
    for (int k = 0; k < sh.n; ++k) {
      const int64_t pad = sh.width[k] - sh.real[k];
      if (pad > 0 && cudaMemsetAsync(a.dW[k] + sh.real[k] * H, 0, size_t(pad) * size_t(H) * 4, s) != cudaSuccess)
        return LP_ERR_CUDA;
    }
  }

  // 4. dX = G W
  {
    StoreParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_bf16_2d(&p.maps[0], G, uint64_t(L.Vc), uint64_t(T), uint64_t(L.Vc), kFwdBlockM) ||
        !encode_bf16_2d(&p.maps[1], Wt, uint64_t(L.Vc), uint64_t(H), uint64_t(L.Vc), kFwdBlockN))
      return LP_ERR_CUDA;
    p.keep_maps = 0u;
    p.mode = 1;
    p.num_m = int32_t((T + kFwdBlockM - 1) / kFwdBlockM);
    p.num_n = int32_t((H + kFwdBlockN - 1) / kFwdBlockN);
    p.nkb_total = int32_t(L.Vc / kFwdBlockK);
    p.kb_per_split = (p.nkb_total + L.split - 1) / L.split;
    const int splits = (p.nkb_total + p.kb_per_split - 1) / p.kb_per_split;
    p.H = H;
    p.T = T;
    p.out = splits > 1 ? part : a.dX;
    p.total_tiles = p.num_m * p.num_n * splits;
    p.err = a.err;
    p.wait_limit_ns = kDefaultWaitLimitNs;
    if (launch_tc_gemm<StoreEpi>(p, a.num_sms, s) != cudaSuccess) return LP_ERR_CUDA;
    if (splits > 1) {
      const size_t n4 = size_t(T) * size_t(H) / 4;
      reduce_split_kernel<<<unsigned((n4 + 255) / 256), 256, 0, s>>>(reinterpret_cast<const float4*>(part), splits,
                                                                      n4, reinterpret_cast<float4*>(a.dX));
      if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
    }
  }

  // 5. db
  for (int k = 0; k < sh.n; ++k) {
    if (a.db[k] == nullptr) continue;
    if (sh.real[k] > 0) {
      const unsigned blocks = unsigned((sh.real[k] * 32 + 255) / 256);
      bias_grad_kernel<<<blocks, 256, 0, s>>>(Gt, L.Tp, L.coff[k], sh.real[k], T, a.db[k]);
      if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
    }
    const int64_t pad = sh.width[k] - sh.real[k];
    if (pad > 0 && cudaMemsetAsync(a.db[k] + sh.real[k], 0, size_t(pad) * 4, s) != cudaSuccess) return LP_ERR_CUDA;
  }
  return LP_OK;
}

}  // namespace lp
