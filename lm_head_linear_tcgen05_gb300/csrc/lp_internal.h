// lp_internal.h - declarations shared by the translation units of liblp.so
// (kernel parameter blocks, tile constants and the launchers lp_api.cu calls).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lp.h"

namespace lp {

// Tile of the tcgen05 GEMM pipeline: 128 rows x 256 columns, K walked in 64s.
constexpr int kFwdBlockM = 128;
constexpr int kFwdBlockN = 256;
constexpr int kFwdBlockK = 64;
// CTAs per cluster along M in the projection GEMMs (forward and backward): a CTA pair
// on the paired-SM MMA, which takes the two row blocks of one vocabulary block and holds
// half of its W box in each CTA, so row blocks are counted in pairs and W maps have boxes
// of kFwdBlockN / 2 rows. 1 runs every tile on one CTA.
#ifndef LP_CLUSTER_M
#define LP_CLUSTER_M 2
#endif
constexpr int kFwdClusterM = LP_CLUSTER_M;
static_assert(kFwdClusterM == 1 || kFwdClusterM == 2, "one CTA or a CTA pair per tile pair");

// Validated vocabulary partition (host side).
struct Shards {
  int n;
  int64_t vocab_real, vocab_padded;
  int64_t start[LP_MAX_SHARDS], end[LP_MAX_SHARDS];
  int64_t width[LP_MAX_SHARDS];  // vocab_end - vocab_start
  int64_t real[LP_MAX_SHARDS];   // ids of the shard below vocab_real
};

// ------------------------------------------------------------- fused forward
// Tensor-map slots of the GEMM kernels: maps[0] is the row operand (X, or G / G^T
// in the backward), maps[1 + k] the operand of shard k.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait (lp_set_wait_limit)
// Teardown after a wait gave up: the time a CTA allows its own copies and MMAs already in
// flight to finish. Those always finish, so this is generous and independent of the limit.
constexpr uint64_t kDrainLimitNs = 2000000000ull;

// The pipeline wait limit every launch carries (lp_set_wait_limit; kDefaultWaitLimitNs).
uint64_t wait_limit_ns();

struct FwdParams {
  CUtensorMap maps[LP_MAX_SHARDS + 1];  // [0] X [T, H]; [1 + k] W_k [V_k, H]; 128B swizzle
  uint32_t keep_maps;                   // maps loaded with an L2 evict-last hint
  int32_t total_tiles;
  unsigned int* err;
  uint64_t wait_limit_ns;
  const __nv_bfloat16* bias[LP_MAX_SHARDS];
  const int32_t* y;
  float* ws_m;                          // [nb_total][T]
  float* ws_s;                          // [nb_total][T]
  float* ws_a;                          // [nb_total][T]
  float* ws_t;                          // [T] target logit z[y], written by the tile holding y
  int64_t vocab_real;
  int64_t shard_start[LP_MAX_SHARDS];
  int32_t shard_width[LP_MAX_SHARDS];   // real (unpadded) width of each shard
  int32_t nb_start[LP_MAX_SHARDS + 1];  // first global vocabulary block of each shard
  int32_t n_shards;
  int32_t T;
  int32_t num_m_blocks;
  int32_t num_k_blocks;
  int32_t m_chunk;                      // row blocks per tile-order chunk (proj_row_chunk)
  int32_t a_box_rows;                   // rows of the X boxes (a batch of one row block: T rounded up to 16)
  float scale_log2;                     // log2(e) / tau
  float inv_tau;                        // 1 / tau
};

// Row blocks per chunk of the projection GEMMs' tile order: every vocabulary block of a
// chunk is visited before the next chunk starts, so a chunk's rows of X (at most 32 MiB)
// stay in L2 while W streams past them once per chunk. A multiple of the cluster size.
inline int32_t proj_row_chunk(int64_t H, int64_t num_m_blocks) {
  const int64_t per_block = int64_t(kFwdBlockM) * H * 2;
  int64_t m = (int64_t(32) << 20) / per_block / kFwdClusterM * kFwdClusterM;
  if (m < kFwdClusterM) m = kFwdClusterM;
  if (m > num_m_blocks) m = num_m_blocks;
  return int32_t(m);
}

// Merge of per-tile (or per-chunk) statistics, one warp per row.
struct MergeParams {
  const float* ws_m;
  const float* ws_s;
  const float* ws_a;
  const float* ws_t;
  const int32_t* y;
  float* logp;
  float* lse;
  float* entropy;
  float* shard_stats;
  unsigned int* err;
  int64_t vocab_real;
  int64_t shard_start[LP_MAX_SHARDS];
  int64_t shard_end[LP_MAX_SHARDS];
  int32_t nb_start[LP_MAX_SHARDS + 1];
  int32_t n_shards;
  int32_t T;
};

// Logits-reuse streaming kernel, one CTA per row.
struct StreamParams {
  const __nv_bfloat16* logits[LP_MAX_SHARDS];
  int64_t ld[LP_MAX_SHARDS];
  int64_t shard_start[LP_MAX_SHARDS];
  int64_t shard_width[LP_MAX_SHARDS];   // real (unpadded) columns of each shard
  int64_t shard_end[LP_MAX_SHARDS];
  const int32_t* y;
  float* logp;
  float* lse;
  float* entropy;
  float* shard_stats;
  unsigned int* err;
  int64_t vocab_real;
  int32_t n_shards;
  int32_t T;
  float scale_log2;
  float inv_tau;
};

// Gradient with respect to reused logits, one CTA per row.
struct LogitsGradParams {
  const __nv_bfloat16* logits[LP_MAX_SHARDS];
  void* out[LP_MAX_SHARDS];              // bf16 or fp32 [T, width], row stride ld_out
  int64_t ld[LP_MAX_SHARDS];
  int64_t ld_out[LP_MAX_SHARDS];
  int64_t shard_start[LP_MAX_SHARDS];
  int64_t width[LP_MAX_SHARDS];          // all columns of the shard (padded ids included)
  int64_t real[LP_MAX_SHARDS];           // columns below vocab_real
  const int32_t* y;
  const float* lse;
  const float* grad;
  const float* entropy;                  // with grad_entropy, else NULL
  const float* grad_entropy;
  int64_t vocab_real;
  int32_t n_shards;
  int32_t T;
  int32_t out_bf16;
  float scale_log2;                      // log2(e) / tau
  float inv_tau;
  unsigned int* err;                     // device error word (bounds-checked builds)
};

// Compact top-p replay, one CTA per row. Scores come from x . W[v] + b[v] (X, W, bias)
// or, in the logits-gather variant, from reused unscaled logits (logits, ld).
struct ReplayParams {
  const __nv_bfloat16* X;
  const __nv_bfloat16* W[LP_MAX_SHARDS];
  const __nv_bfloat16* bias[LP_MAX_SHARDS];
  const __nv_bfloat16* logits[LP_MAX_SHARDS];
  int64_t ld[LP_MAX_SHARDS];
  const int32_t* ids;                   // [T][64]
  const int32_t* y;
  float* logp;
  float* lse;
  float* shard_stats;
  unsigned int* err;
  int64_t vocab_real;
  int64_t shard_start[LP_MAX_SHARDS];
  int64_t shard_end[LP_MAX_SHARDS];
  int32_t n_shards;
  int32_t T;
  int32_t H;
  float inv_tau;
};

// Dense keep-mask compaction into canonical replay slots.
struct MaskParams {
  const uint8_t* mask[LP_MAX_SHARDS];
  int64_t shard_start[LP_MAX_SHARDS];
  int64_t shard_width[LP_MAX_SHARDS];
  int32_t* ids_out;                     // [T][64]
  unsigned int* err;
  int64_t vocab_real;
  int32_t n_shards;
  int32_t T;
};

// Rank-ordered reduction of exchanged per-shard statistics, one thread per row.
struct MergeStatsParams {
  const float* stats;                   // [n_shards][3][T]: lse, t, h
  const int32_t* y;
  float* logp;
  float* lse;
  float* entropy;                       // or NULL
  unsigned int* err;
  int64_t vocab_real;
  int64_t shard_start[LP_MAX_SHARDS];
  int64_t shard_end[LP_MAX_SHARDS];
  int32_t n_shards;
  int32_t T;
};

// Ordered elementwise sum of partial results.
struct SumPartsParams {
  const float* parts[LP_MAX_PARTS];
  void* out;
  int64_t count;
  int32_t n_parts;
  int32_t out_bf16;
};

// Backward: everything lp_backward validated, handed to the backward translation unit.
struct BackwardArgs {
  const void* X;
  int64_t T, H;
  const int32_t* y;
  float tau;
  const float* lse;
  const float* grad;
  const float* entropy;       // with grad_entropy: the forward's entropy, else NULL
  const float* grad_entropy;  // upstream gradient of the entropy, or NULL
  void* dX;                   // float or bf16 [T, H] (dx_bf16)
  int dx_bf16;
  int accumulate;             // add into dW and db instead of overwriting them
  int dw_bf16;                // dW in bf16 (not with accumulate)
  const void* W[LP_MAX_SHARDS];
  const void* bias[LP_MAX_SHARDS];
  void* dW[LP_MAX_SHARDS];    // float or bf16 [V_k, H] (dw_bf16)
  float* db[LP_MAX_SHARDS];
  void* workspace;
  unsigned int* err;
  int num_sms;
};

size_t backward_ws_bytes(int64_t T, int64_t H, const Shards& sh);
lp_status run_backward(const BackwardArgs& a, const Shards& sh, cudaStream_t s);

// bf16 row-major [rows, inner] (row stride ld elements) as a TMA map with boxes of
// 64 x box_rows elements, 128-byte swizzle and zero fill out of bounds.
bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t ld,
                    uint32_t box_rows);

cudaError_t launch_fused_forward(const FwdParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t s);
cudaError_t launch_stream_logits(const StreamParams& p, cudaStream_t s);
cudaError_t launch_replay(const ReplayParams& p, cudaStream_t s);
cudaError_t launch_replay_from_logits(const ReplayParams& p, cudaStream_t s);
cudaError_t launch_mask_compact(const MaskParams& p, cudaStream_t s);
cudaError_t launch_logits_backward(const LogitsGradParams& p, cudaStream_t s);
cudaError_t launch_merge_stats(const MergeStatsParams& p, cudaStream_t s);
cudaError_t launch_sum_partials(const SumPartsParams& p, cudaStream_t s);

}  // namespace lp
