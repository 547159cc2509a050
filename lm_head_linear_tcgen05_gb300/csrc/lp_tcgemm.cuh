// lp_tcgemm.cuh - persistent warp-specialised bf16 GEMM pipeline on tcgen05/TMEM.
//
// C_tile[128 x 256] = sum_k A[rows, k] * B[cols, k]  (K-major or MN-major bf16 operands,
// fp32 accumulation in tensor memory), followed by an epilogue supplied by the caller
// that reads the accumulator straight out of TMEM. The kernel is persistent (one CTA per
// SM, tiles handed out round-robin) and warp specialised:
//
//   warp 0      TMA producer: A and B boxes (64 K-elements wide, 128-byte swizzle)
//               into a shared-memory ring of S::kStages stages (mbarrier full/empty);
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and
//               issues tcgen05.mma kind::f16 (K=16) from one thread, committing each
//               stage back to the producers and each finished tile to the epilogue;
//   warps 2..5  epilogue: warp w may read TMEM lanes 32*(w%4)..+31, so each thread
//               owns one row of the tile; the callback runs while the MMA warp
//               fills the other accumulator.
//
// kClusterM = 2 runs the CTAs as pairs on the paired-SM MMA (tcgen05 .cta_group::2). The
// two CTAs of a pair take the two row blocks of one column block (tiles 2j and 2j+1):
// each loads its own 128 rows of A and one half (128 rows) of the shared B box into its
// own shared memory, and the pair's even CTA issues M = 256, N = 256 MMAs that read A and
// B from both CTAs' shared memory and leave each CTA's 128 rows in its own TMEM. Every SM
// thus receives 32 KB of operands per 64-deep K step instead of 48 KB, and no operand is
// copied to more than one SM. Both CTAs' copies complete on the even CTA's full barrier
// (it expects the pair's bytes); each MMA commit arrives on the empty barrier of both
// CTAs, each finished tile on both CTAs' accumulator barriers, and all eight epilogue
// warps of the pair release an accumulator on the even CTA's barrier.
//
// Every mbarrier wait is bounded in time (see lp_device.cuh): a wait that runs past
// the limit (p.wait_limit_ns) records LP_ERR_DEVICE_TIMEOUT, raises a CTA-wide abort flag
// and every role leaves its loop; the producer then waits for its copies in flight and the
// MMA thread for its MMAs (up to kDrainLimitNs, whatever the limit), a cluster barrier keeps
// both CTAs of a pair alive until neither can touch the other, and TMEM is freed before the
// CTA exits.
//
// An epilogue type E derives from GemmEpiBase and provides
//   static constexpr int kClusterM;       1, or 2 for the CTA pairs above
//   kAMN / kBMN                           operand major-ness (default K-major)
//   a_k / b_k                             per-k-block map and K coordinate (default above)
//   struct E::Params           with members `CUtensorMap maps[kGemmMaps]`,
//                              `uint32_t keep_maps` (bit i: map i is small and
//                              reused, loaded with an L2 evict-last hint),
//                              `int total_tiles` (a multiple of kClusterM),
//                              `unsigned int* err`, `uint64_t wait_limit_ns`;
//   kMHalves                              1, or 2 for 256-row tiles (see GemmShape)
//   static TileJob E::job(const Params&, int tile);
//   static void E::run(const Params&, int tile, int half, uint32_t tmem_row_base, int quarter, int lane);
// `tmem_row_base` addresses column 0 of the accumulator of rows [128 half, 128 half + 128)
// of the tile at this warp's first lane; column c of this thread's row is at
// tmem_row_base + c. Boxes: K-major A 64 x 128, K-major B 64 x 256 (64 x 128 in a pair:
// each CTA loads its half), MN-major operands 64 x 64 atoms (a pair's CTAs load half of
// B's atoms each).
#pragma once

#include <atomic>

#include "lp_device.cuh"

namespace lp {

constexpr int kGemmBlockM = kFwdBlockM;
constexpr int kGemmBlockN = kFwdBlockN;
constexpr int kGemmBlockK = kFwdBlockK;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int kGemmThreads = 192;
constexpr int kGemmTmemCols = 512;
constexpr int kGemmMaps = LP_MAX_SHARDS + 1;

constexpr uint32_t kGemmStageA = kGemmBlockM * kGemmBlockK * 2;  // 16 KB per 128-row half
constexpr uint32_t kGemmStageB = kGemmBlockN * kGemmBlockK * 2;  // 32 KB

constexpr uint32_t kMNAtomBytes = 64 * kGemmBlockK * 2;  // 64 MN elements x 64 K rows: 8 KB

// Tile order of the projection GEMMs: row blocks in chunks of m_chunk (see
// proj_row_chunk), and inside a chunk row blocks fastest, then vocabulary blocks. Pairs
// of tiles (2j, 2j+1) stay two row blocks of one vocabulary block, as clusters need.
__device__ __forceinline__ void proj_raster(int tile, int num_m_blocks, int m_chunk, int nb_total, int& mb,
                                            int& nb) {
  const int per_chunk = m_chunk * nb_total;
  const int c = tile / per_chunk;
  const int r = tile - c * per_chunk;
  const int m0 = c * m_chunk;
  const int rows = num_m_blocks - m0 < m_chunk ? num_m_blocks - m0 : m_chunk;
  mb = m0 + r % rows;
  nb = r / rows;
}

// What one tile reads: rows (MN indices) a_y.. of map a_map and b_y.. of map b_map,
// for k blocks kb0 .. kb0 + nkb - 1; nkb >= 1. A K-major operand is one box at
// (x = k, y = row); an MN-major one is a row of 64-wide atoms at (x = mn, y = k).
struct TileJob {
  int a_map, b_map;
  int a_y, b_y;
  int kb0, nkb;
};

// Default K coordinates: the tile's own maps, k = (kb0 + kb) * 64. An epilogue type
// overrides a_k / b_k when an operand's K range spans several maps (shards).
struct GemmEpiBase {
  static constexpr bool kAMN = false;  // A operand MN-major
  static constexpr bool kBMN = false;  // B operand MN-major
  static constexpr int kMHalves = 1;   // 128-row halves per CTA tile (2: 256 rows, single accumulator)
  // K-major A boxes of p.a_box_rows (<= 128) rows instead of 128: the rows of the A tile
  // past them keep stale shared memory, so only output rows < a_box_rows are meaningful
  static constexpr bool kVarABox = false;
  static __device__ __forceinline__ void a_k(const void*, const TileJob& j, int kb, int& map, int& k) {
    map = j.a_map;
    k = (j.kb0 + kb) * kFwdBlockK;
  }
  static __device__ __forceinline__ void b_k(const void*, const TileJob& j, int kb, int& map, int& k) {
    map = j.b_map;
    k = (j.kb0 + kb) * kFwdBlockK;
  }
};

#ifndef LP_GEMM_MAX_STAGES
#define LP_GEMM_MAX_STAGES 8
#endif

struct GemmSync {
  uint64_t full[LP_GEMM_MAX_STAGES];
  uint64_t empty[LP_GEMM_MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
};

// Ring geometry of an epilogue type: a stage holds kMHalves 128-row halves of A and this
// CTA's rows of B (all 256, or 128 in a CTA pair); as many stages as fit the shared memory
// (up to LP_GEMM_MAX_STAGES). 128-row tiles keep two TMEM accumulators, so the epilogue of
// one tile overlaps the MMAs of the next; 256-row tiles fill all 512 TMEM columns with
// their two halves (meant for tiles whose K loop is long enough that the epilogue gap does
// not matter).
template <class E>
struct GemmShape {
  static constexpr int kCG = E::kClusterM;
  static_assert(kCG == 1 || kCG == 2, "one CTA, or a CTA pair");
  static constexpr int kMH = E::kMHalves;
  static_assert(kMH == 1 || kMH == 2, "one or two 128-row halves");
  static constexpr uint32_t kStageA = kMH * kGemmStageA;
  static constexpr uint32_t kStageB = kGemmStageB / kCG;
  static constexpr uint32_t kStageBytes = kStageA + kStageB;
  static constexpr size_t kFixed = 1024 + sizeof(GemmSync);
  static constexpr int kFit = int((232448 - kFixed) / kStageBytes);
  static constexpr int kStages = kFit < LP_GEMM_MAX_STAGES ? kFit : LP_GEMM_MAX_STAGES;
  static constexpr int kAcc = kMH == 1 ? 2 : 1;  // accumulators in flight
  static constexpr size_t kSmemBytes = kFixed + size_t(kStages) * kStageBytes;
  static_assert(kStages >= 2 && kSmemBytes <= 232448, "shared memory budget");
};

template <class E>
__global__ void __launch_bounds__(kGemmThreads, 1) tc_gemm_kernel(const __grid_constant__ typename E::Params p) {
  using S = GemmShape<E>;
  constexpr int kCG = S::kCG;
  constexpr int kStages = S::kStages;
  constexpr int kMH = S::kMH;
  static_assert(kMH == 1 || !E::kAMN, "256-row tiles take a K-major A operand");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * S::kStageA;
  GemmSync* sync = reinterpret_cast<GemmSync*>(smem + kStages * S::kStageBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kCG > 1 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;  // the CTA that issues the MMAs
  const int cluster_id = int(blockIdx.x) / kCG;
  const int num_clusters = int(gridDim.x) / kCG;
  const int cluster_tiles = p.total_tiles / kCG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sync->full[s], 1);
      mbar_init(&sync->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sync->tfull[b], 1);
      mbar_init(&sync->tempty[b], 4 * kCG);
    }
    mbar_init(&sync->done, 1);
    sync->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc<kCG>(&sync->tmem_base, kGemmTmemCols);
    tmem_relinquish<kCG>();
  }
  tc_fence_before();
  if constexpr (kCG > 1)
    cluster_sync();  // the pair's barriers and TMEM exist before anything targets them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sync->tmem_base;
  volatile int* abort = &sync->abort;

  if (warp == 0) {
    if (lane == 0) {
      // --------------------------------------------------------- TMA producer
      const uint64_t pol_keep = l2_policy_evict_last();
      const uint64_t pol_norm = l2_policy_evict_normal();
      uint32_t stage_tx = S::kStageBytes;  // bytes this CTA's copies deliver per stage
      if constexpr (E::kVarABox) {
        static_assert(kMH == 1 && !E::kAMN && kCG == 1, "short A boxes: one K-major 128-row half, one CTA");
        stage_tx = kGemmStageB + uint32_t(p.a_box_rows) * (kGemmBlockK * 2);
      }
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0, armed_phase = 0;  // stages with a copy issued, and its phase
      bool ok = true;
      for (int ct = cluster_id; ok && ct < cluster_tiles; ct += num_clusters) {
        const TileJob j = E::job(p, ct * kCG + int(rank));
        const uint64_t pa = ((p.keep_maps >> j.a_map) & 1u) ? pol_keep : pol_norm;
        const uint64_t pb = ((p.keep_maps >> j.b_map) & 1u) ? pol_keep : pol_norm;
        for (int kb = 0; kb < j.nkb; ++kb) {
          if (!mbar_wait(&sync->empty[stage], phase ^ 1u, abort, p.wait_limit_ns, p.err)) {
            ok = false;
            break;
          }
          int am, ak, bm, bk;
          E::a_k(&p, j, kb, am, ak);
          E::b_k(&p, j, kb, bm, bk);
          // the pair's copies all complete on the leader's barrier, which expects both CTAs' bytes
          if (leader) mbar_arrive_expect_tx(&sync->full[stage], stage_tx * kCG);
          uint8_t* dA = sA + stage * S::kStageA;
          uint8_t* dB = sB + stage * S::kStageB;
          const uint32_t bar_cl = kCG > 1 ? cluster_addr(&sync->full[stage], 0) : 0u;
          auto load = [&](void* dst, int map, int32_t x, int32_t y, uint64_t pol) {
            if constexpr (kCG > 1)
              tma_load_2d_pair(dst, &p.maps[map], bar_cl, x, y, pol);
            else
              tma_load_2d(dst, &p.maps[map], &sync->full[stage], x, y, pol);
          };
          if constexpr (!E::kAMN) {
#pragma unroll
            for (int h = 0; h < kMH; ++h) load(dA + h * kGemmStageA, am, ak, j.a_y + h * kGemmBlockM, pa);
          } else {  // MN-major: 64-element atoms of 64 K rows each
#pragma unroll
            for (int i = 0; i < kGemmBlockM / 64; ++i) load(dA + i * kMNAtomBytes, am, j.a_y + 64 * i, ak, pa);
          }
          if constexpr (!E::kBMN) {
            load(dB, bm, bk, j.b_y + int(rank) * (kGemmBlockN / kCG), pb);
          } else {
            constexpr int kAtoms = kGemmBlockN / 64 / kCG;  // this CTA's atoms of B
#pragma unroll
            for (int i = 0; i < kAtoms; ++i)
              load(dB + i * kMNAtomBytes, bm, j.b_y + 64 * (int(rank) * kAtoms + i), bk, pb);
          }
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // the leader's barriers count the pair's bytes, so its drain waits for both CTAs'
        // armed copies; the other CTA cannot observe its own, and gives any copy still in
        // flight (a few microseconds at most) time to land before the CTAs leave
        if (leader) {
          const uint64_t deadline = global_timer_ns() + kDrainLimitNs;
          for (int s = 0; s < kStages; ++s)
            if (armed & (1u << s)) drain_until(&sync->full[s], (armed_phase >> s) & 1u, deadline);
        } else {
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 100000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kGemmBlockM * kCG, kGemmBlockN, E::kAMN, E::kBMN);
      // per 16-deep K step: +32 bytes inside a K-major row, +2048 bytes (16 rows) in MN-major
      constexpr uint32_t a_step = E::kAMN ? 128u : 2u;
      constexpr uint32_t b_step = E::kBMN ? 128u : 2u;
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int ct = cluster_id; ok && ct < cluster_tiles; ct += num_clusters) {
        const TileJob j = E::job(p, ct * kCG);
        const bool free_acc = kCG > 1
                                  ? mbar_wait_cluster(&sync->tempty[acc], acc_phase ^ 1u, abort, p.wait_limit_ns, p.err)
                                  : mbar_wait(&sync->tempty[acc], acc_phase ^ 1u, abort, p.wait_limit_ns, p.err);
        if (!free_acc) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * kGemmBlockN;  // half h at + h * kGemmBlockN
        for (int kb = 0; kb < j.nkb; ++kb) {
          if (!mbar_wait(&sync->full[stage], phase, abort, p.wait_limit_ns, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aa = smem_u32(sA + stage * S::kStageA);
          const uint32_t ba = smem_u32(sB + stage * S::kStageB);
          const uint64_t b_desc = E::kBMN ? sw128_mnmajor_desc(ba, kMNAtomBytes) : sw128_kmajor_desc(ba);
#pragma unroll
          for (int h = 0; h < kMH; ++h) {
            const uint32_t ah = aa + h * kGemmStageA;
            const uint64_t a_desc = E::kAMN ? sw128_mnmajor_desc(ah, kMNAtomBytes) : sw128_kmajor_desc(ah);
#pragma unroll
            for (int k = 0; k < kGemmBlockK / 16; ++k)
              umma_bf16<kCG>(d_tmem + h * kGemmBlockN, a_desc + a_step * k, b_desc + b_step * k, idesc,
                             (kb | k) != 0 ? 1u : 0u);
          }
          if constexpr (kCG > 1)
            umma_commit_pair(&sync->empty[stage]);
          else
            umma_commit<1>(&sync->empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (kCG > 1)
          umma_commit_pair(&sync->tfull[acc]);
        else
          umma_commit<1>(&sync->tfull[acc]);
        if (++acc == uint32_t(S::kAcc)) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit<kCG>(&sync->done);
      drain_wait(&sync->done, 0, kDrainLimitNs);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    for (int ct = cluster_id; ct < cluster_tiles; ct += num_clusters) {
      // every lane waits; the warp proceeds only if all saw the accumulator ready
      if (!__all_sync(0xffffffffu, mbar_wait(&sync->tfull[acc], acc_phase, abort, p.wait_limit_ns, p.err)))
        break;
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < kMH; ++h)
        E::run(p, ct * kCG + int(rank), h, tmem + (uint32_t(q * 32) << 16) + (acc + h) * kGemmBlockN, q, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kCG > 1)
          mbar_arrive_cluster(cluster_addr(&sync->tempty[acc], 0));  // the leader's barrier
        else
          mbar_arrive(&sync->tempty[acc]);
      }
      if (++acc == uint32_t(S::kAcc)) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  if constexpr (kCG > 1)
    cluster_sync();  // no CTA leaves while the pair's MMAs or copies may still touch it
  else
    __syncthreads();
  // this CTA's work is done: a kernel launched as this grid's programmatic dependent (the
  // forward's row merge) may be scheduled once every CTA gets here; it waits for the grid's
  // completion itself
  if (threadIdx.x == 0) grid_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kCG>(tmem, kGemmTmemCols);
  }
}

// Per-device launch set-up of one GEMM kernel, resolved on the first launch on each
// device (dynamic shared memory opt-in, clusters that can be co-resident) so that later
// launches - including launches captured into a CUDA graph - issue nothing but the
// kernel launch itself.
template <class E>
int gemm_clusters_for_device(int num_sms) {
  constexpr int kCM = E::kClusterM;
  static_assert(kCM == 1 || kCM == 2, "one CTA or a CTA pair");
  static std::atomic<int> cache[64];  // 0 = unresolved, > 0 = clusters, < 0 = error
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  int c = cache[dev].load(std::memory_order_acquire);
  if (c != 0) return c;
  if (cudaFuncSetAttribute(tc_gemm_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(GemmShape<E>::kSmemBytes)) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  int clusters = num_sms / kCM;
  if (kCM > 1) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCM;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = GemmShape<E>::kSmemBytes;
    cfg.gridDim = dim3(kCM * clusters, 1, 1);
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, tc_gemm_kernel<E>, &cfg) == cudaSuccess && active > 0 &&
        active < clusters)
      clusters = active;
    cudaGetLastError();
  }
  if (clusters < 1) clusters = 1;
  cache[dev].store(clusters, std::memory_order_release);
  return clusters;
}

// Launches one CTA per SM (rounded to whole clusters) over p.total_tiles tiles.
template <class E>
cudaError_t launch_tc_gemm(const typename E::Params& p, int num_sms, cudaStream_t s) {
  constexpr int kCM = E::kClusterM;
  int clusters = gemm_clusters_for_device<E>(num_sms);
  if (clusters < 0) return cudaErrorInvalidConfiguration;
  if (p.total_tiles < kCM) return cudaSuccess;
  const int cluster_tiles = p.total_tiles / kCM;
  if (clusters > cluster_tiles) clusters = cluster_tiles;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = GemmShape<E>::kSmemBytes;
  cfg.stream = s;
  cfg.gridDim = dim3(kCM * clusters, 1, 1);
  if (kCM > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCM;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<E>, p);
}

}  // namespace lp
