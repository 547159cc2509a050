// lp_api.cu - the C ABI of liblp.so: argument validation, per-device set-up, tensor
// maps, workspace carving and kernel dispatch. Declarations and the contract of every
// entry point are in include/lp.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "lp_device.cuh"
#include "lp_internal.h"

namespace lp {

// Sticky per-device error word: the first device-detected error since the last
// lp_get_device_error(). Kernels receive its device address as a parameter.
__device__ unsigned int g_error_word;

__global__ void probe_kernel() {}

// One warp waits on an mbarrier that nothing arrives on; the bounded wait must give
// up after limit_ns, record LP_ERR_DEVICE_TIMEOUT and return.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, unsigned int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort, limit_ns, err);
  __syncthreads();
}

// One thread checks an index equal to its extent: a bounds-checked build records
// LP_ERR_BOUNDS, the regular build nothing. No memory is read or written.
__global__ void bounds_selftest_kernel(int64_t extent, unsigned int* err) {
  if (threadIdx.x == 0) (void)in_bounds(extent < extent, err);
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool init = false;
  bool supported = false;
  int num_sms = 0;
  unsigned int* err = nullptr;
  // lp_forward_host's copy stream and its three events, created on its first call; a
  // call holds host_mu while it records and waits on them, so that calls from several
  // host threads never wait on one another's records
  bool copy_init = false;
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  std::mutex host_mu;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_wait_limit{kDefaultWaitLimitNs};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Resolves, once per device (with that device current), whether this library's
// sm_103a code can run there, the SM count and the device address of the error word.
lp_status device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return LP_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.init) {
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, probe_kernel) != cudaSuccess) {
      cudaGetLastError();
      st.supported = false;
    } else {
      int sms = 0;
      void* err = nullptr;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaGetSymbolAddress(&err, g_error_word) != cudaSuccess) {
        cudaGetLastError();
        return LP_ERR_CUDA;
      }
      st.num_sms = sms;
      st.err = static_cast<unsigned int*>(err);
      st.supported = true;
    }
    st.init = true;
  }
  if (!st.supported) return LP_ERR_UNSUPPORTED_DEVICE;
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      cudaGetLastError();
      return LP_ERR_CUDA;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = &st;
  return LP_OK;
}

// The copy stream of lp_forward_host on the current device (created once, with that
// device current): a non-blocking stream and three events without timing.
lp_status device_copy_stream(DeviceState* st) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!st->copy_init) {
    if (cudaStreamCreateWithFlags(&st->copy_stream, cudaStreamNonBlocking) != cudaSuccess) {
      cudaGetLastError();
      return LP_ERR_CUDA;
    }
    for (auto& e : st->ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return LP_ERR_CUDA;
      }
    st->copy_init = true;
  }
  return LP_OK;
}

}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit.load(std::memory_order_relaxed); }

// bf16 row-major matrix [rows, inner] with row stride ld elements, boxes of
// 64 (inner) x box_rows, 128-byte swizzle, out-of-bounds elements read as zero.
bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t ld,
                    uint32_t box_rows) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

// A partition is valid when its shards are contiguous and ascending and tile
// [0, vocab_padded) (local = 0) or a range [lo, hi) inside it (local = 1, one
// tensor-parallel rank's ids). The kernels need no mode of their own: an id outside the
// shards is simply not here (another rank's target or replay id).
lp_status check_partition(const lp_vocab_partition* part, Shards* sh) {
  if (part == nullptr || part->shards == nullptr) return LP_ERR_INVALID_ARG;
  const int n = part->n_shards;
  if (n < 1 || n > LP_MAX_SHARDS) return LP_ERR_INVALID_ARG;
  if (part->vocab_real < 1 || part->vocab_real > part->vocab_padded || part->vocab_padded > INT32_MAX)
    return LP_ERR_INVALID_ARG;
  if (part->local != 0 && part->local != 1) return LP_ERR_INVALID_ARG;
  const bool local = part->local == 1;
  int64_t expect = local ? part->shards[0].vocab_start : 0;
  if (expect < 0) return LP_ERR_INVALID_ARG;
  for (int k = 0; k < n; ++k) {
    const int64_t s = part->shards[k].vocab_start, e = part->shards[k].vocab_end;
    if (s != expect || e < s) return LP_ERR_INVALID_ARG;
    expect = e;
    sh->start[k] = s;
    sh->end[k] = e;
    sh->width[k] = e - s;
    const int64_t r = (e < part->vocab_real ? e : part->vocab_real) - s;
    sh->real[k] = r > 0 ? r : 0;
  }
  if (local ? expect > part->vocab_padded : expect != part->vocab_padded) return LP_ERR_INVALID_ARG;
  sh->n = n;
  sh->vocab_real = part->vocab_real;
  sh->vocab_padded = part->vocab_padded;
  return LP_OK;
}

// T = 0 (an empty batch) is valid: the call succeeds without touching any pointer,
// except lp_backward, which still zeroes dW and db (the gradient of an empty sum).
bool valid_rows(int64_t T) { return T >= 0 && T <= (int64_t(1) << 30); }
bool valid_hidden(int64_t H) { return H >= 8 && H <= 65536 && H % 8 == 0; }
bool valid_tau(float tau) { return std::isfinite(tau) && tau > 0.f; }

// lp_forward_host splits batches of at least this many rows in two halves
constexpr int64_t kHostSplitRows = 4096;

size_t forward_ws_bytes(int64_t T, const Shards& sh) {
  int64_t nb = 0;
  for (int k = 0; k < sh.n; ++k) nb += (sh.real[k] + kFwdBlockN - 1) / kFwdBlockN;
  const size_t per = align_up(size_t(nb) * size_t(T) * sizeof(float), 256);
  return 3 * per + align_up(size_t(T) * sizeof(float), 256);
}

// Workspace of lp_forward_host: the forward's own, then device staging for X, y and
// every output (logp, LSE, entropy, shard statistics), each 256-byte aligned.
struct HostLayout {
  size_t off_x, off_y, off_logp, off_lse, off_ent, off_ss, total;
};

HostLayout host_layout(int64_t T, int64_t H, const Shards& sh) {
  HostLayout L;
  size_t off = forward_ws_bytes(T, sh);
  L.off_x = off;
  off += align_up(size_t(T) * size_t(H) * 2, 256);
  L.off_y = off;
  off += align_up(size_t(T) * 4, 256);
  L.off_logp = off;
  off += align_up(size_t(T) * 4, 256);
  L.off_lse = off;
  off += align_up(size_t(T) * 4, 256);
  L.off_ent = off;
  off += align_up(size_t(T) * 4, 256);
  L.off_ss = off;
  off += align_up(size_t(sh.n) * 3 * size_t(T) * 4, 256);
  L.total = off;
  return L;
}

}  // namespace lp

using namespace lp;

extern "C" {

const char* lp_status_string(lp_status s) {
  switch (s) {
    case LP_OK: return "LP_OK";
    case LP_ERR_INVALID_ARG: return "LP_ERR_INVALID_ARG: invalid argument";
    case LP_ERR_ALIGNMENT: return "LP_ERR_ALIGNMENT: a pointer or row stride is not 16-byte aligned";
    case LP_ERR_UNSUPPORTED_DEVICE: return "LP_ERR_UNSUPPORTED_DEVICE: no sm_103 device is current";
    case LP_ERR_WORKSPACE_TOO_SMALL: return "LP_ERR_WORKSPACE_TOO_SMALL: workspace smaller than lp_workspace_size()";
    case LP_ERR_TARGET_OUT_OF_RANGE: return "LP_ERR_TARGET_OUT_OF_RANGE: a target id is outside [0, vocab_real)";
    case LP_ERR_REPLAY_ID_OUT_OF_RANGE: return "LP_ERR_REPLAY_ID_OUT_OF_RANGE: a replay id is outside [0, vocab_real)";
    case LP_ERR_DEVICE_TIMEOUT: return "LP_ERR_DEVICE_TIMEOUT: a pipeline wait exceeded its time limit";
    case LP_ERR_CUDA: return "LP_ERR_CUDA: a CUDA runtime call failed";
    case LP_ERR_REPLAY_TOO_MANY_IDS: return "LP_ERR_REPLAY_TOO_MANY_IDS: a keep-mask row keeps more than 64 ids";
    case LP_ERR_BOUNDS: return "LP_ERR_BOUNDS: a device bounds check failed (bounds-checked build)";
  }
  return "unknown lp_status";
}

int lp_device_supported(void) {
  DeviceState* st = nullptr;
  return device_state(&st) == LP_OK ? 1 : 0;
}

size_t lp_workspace_size(lp_op op, int64_t T, int64_t H, const lp_vocab_partition* part) {
  Shards sh;
  if (!valid_rows(T) || check_partition(part, &sh) != LP_OK) return 0;
  switch (op) {
    case LP_OP_FORWARD: return forward_ws_bytes(T, sh);
    case LP_OP_FORWARD_FROM_LOGITS: return 0;
    case LP_OP_TOP_P_REPLAY: return 0;
    case LP_OP_TOP_P_REPLAY_DENSE_MASK: return align_up(size_t(T) * LP_REPLAY_SLOTS * sizeof(int32_t), 256);
    case LP_OP_BACKWARD: return valid_hidden(H) ? backward_ws_bytes(T, H, sh) : 0;
    case LP_OP_BACKWARD_FROM_LOGITS: return 0;
    case LP_OP_FORWARD_HOST: return valid_hidden(H) ? host_layout(T, H, sh).total : 0;
  }
  return 0;
}

lp_status lp_forward(const void* X, int64_t T, int64_t H, const void* const* W, const void* const* bias,
                     const lp_vocab_partition* part, const int32_t* y, float tau, const lp_outputs* out,
                     void* workspace, size_t ws_bytes, lp_stream_t stream) {
  Shards sh;
  if (check_partition(part, &sh) != LP_OK) return LP_ERR_INVALID_ARG;
  if (!valid_rows(T) || !valid_hidden(H) || !valid_tau(tau)) return LP_ERR_INVALID_ARG;
  if (T == 0) return LP_OK;
  if (X == nullptr || W == nullptr || y == nullptr || out == nullptr || out->logp == nullptr ||
      out->lse == nullptr)
    return LP_ERR_INVALID_ARG;
  for (int k = 0; k < sh.n; ++k)
    if (sh.real[k] > 0 && W[k] == nullptr) return LP_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(workspace)) return LP_ERR_ALIGNMENT;
  for (int k = 0; k < sh.n; ++k)
    if (sh.real[k] > 0 && !aligned16(W[k])) return LP_ERR_ALIGNMENT;
  {
    // tiles are counted in 32-bit integers on the device
    int64_t nb_total = 0;
    for (int k = 0; k < sh.n; ++k) nb_total += (sh.real[k] + kFwdBlockN - 1) / kFwdBlockN;
    if (nb_total * ((T + kFwdBlockM - 1) / kFwdBlockM + kFwdClusterM) > int64_t(INT32_MAX)) return LP_ERR_INVALID_ARG;
  }
  const size_t need = forward_ws_bytes(T, sh);
  if (workspace == nullptr || ws_bytes < need) return LP_ERR_WORKSPACE_TOO_SMALL;

  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;

  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  // a batch of a single row block runs without clusters (launch_fused_forward): each CTA
  // fetches its whole W box, instead of half of it for a partner CTA with padding rows, and
  // its X boxes hold only the batch's rows (rounded up to 16)
  const int64_t mblocks = (T + kFwdBlockM - 1) / kFwdBlockM;
  const int cm = mblocks == 1 ? 1 : kFwdClusterM;
  p.a_box_rows = cm == 1 ? int32_t((T + 15) / 16 * 16) : kFwdBlockM;
  if (!encode_bf16_2d(&p.maps[0], X, uint64_t(H), uint64_t(T), uint64_t(H), uint32_t(p.a_box_rows)))
    return LP_ERR_CUDA;
  int nb = 0;
  for (int k = 0; k < sh.n; ++k) {
    if (sh.real[k] > 0 && !encode_bf16_2d(&p.maps[1 + k], W[k], uint64_t(H), uint64_t(sh.width[k]), uint64_t(H),
                                          uint32_t(kFwdBlockN / cm)))
      return LP_ERR_CUDA;
    p.bias[k] = bias != nullptr ? static_cast<const __nv_bfloat16*>(bias[k]) : nullptr;
    p.shard_start[k] = sh.start[k];
    p.shard_width[k] = int32_t(sh.real[k]);
    p.nb_start[k] = nb;
    nb += int((sh.real[k] + kFwdBlockN - 1) / kFwdBlockN);
  }
  p.nb_start[sh.n] = nb;
  p.keep_maps = 1u;  // X is re-read by every vocabulary block: keep it in L2
  p.n_shards = sh.n;
  p.T = int32_t(T);
  p.num_m_blocks = int32_t((mblocks + cm - 1) / cm * cm);  // row blocks, counted in whole clusters
  p.num_k_blocks = int32_t((H + kFwdBlockK - 1) / kFwdBlockK);
  p.m_chunk = proj_row_chunk(H, p.num_m_blocks);
  p.total_tiles = nb * p.num_m_blocks;
  p.err = dev->err;
  p.wait_limit_ns = wait_limit_ns();
  p.y = y;
  p.vocab_real = sh.vocab_real;
  p.scale_log2 = float(1.4426950408889634 / double(tau));
  p.inv_tau = float(1.0 / double(tau));
  const size_t per = align_up(size_t(nb) * size_t(T) * sizeof(float), 256);
  char* ws = static_cast<char*>(workspace);
  p.ws_m = reinterpret_cast<float*>(ws);
  p.ws_s = reinterpret_cast<float*>(ws + per);
  p.ws_a = reinterpret_cast<float*>(ws + 2 * per);
  p.ws_t = reinterpret_cast<float*>(ws + 3 * per);

  MergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  mp.ws_m = p.ws_m;
  mp.ws_s = p.ws_s;
  mp.ws_a = p.ws_a;
  mp.ws_t = p.ws_t;
  mp.y = y;
  mp.logp = out->logp;
  mp.lse = out->lse;
  mp.entropy = out->entropy;
  mp.shard_stats = out->shard_stats;
  mp.err = dev->err;
  mp.vocab_real = sh.vocab_real;
  for (int k = 0; k < sh.n; ++k) {
    mp.shard_start[k] = sh.start[k];
    mp.shard_end[k] = sh.end[k];
    mp.nb_start[k] = p.nb_start[k];
  }
  mp.nb_start[sh.n] = nb;
  mp.n_shards = sh.n;
  mp.T = int32_t(T);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (launch_fused_forward(p, dev->num_sms, s) != cudaSuccess) return LP_ERR_CUDA;
  if (launch_merge(mp, s) != cudaSuccess) return LP_ERR_CUDA;
  return LP_OK;
}

lp_status lp_forward_host(const void* X_host, int64_t T, int64_t H, const void* const* W, const void* const* bias,
                          const lp_vocab_partition* part, const int32_t* y_host, float tau, const lp_outputs* out_host,
                          void* workspace, size_t ws_bytes, lp_stream_t stream) {
  Shards sh;
  if (check_partition(part, &sh) != LP_OK) return LP_ERR_INVALID_ARG;
  if (!valid_rows(T) || !valid_hidden(H) || !valid_tau(tau)) return LP_ERR_INVALID_ARG;
  if (T == 0) return LP_OK;
  if (X_host == nullptr || y_host == nullptr || out_host == nullptr || out_host->logp == nullptr ||
      out_host->lse == nullptr)
    return LP_ERR_INVALID_ARG;
  const HostLayout L = host_layout(T, H, sh);
  if (workspace == nullptr || ws_bytes < L.total) return LP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return LP_ERR_ALIGNMENT;
  DeviceState* dev = nullptr;
  lp_status dst = device_state(&dev);
  if (dst != LP_OK) return dst;
  // Large batches run as two halves (rows split at a multiple of 256): the second half's
  // rows cross the host link on the copy stream while the first half's GEMM runs. A
  // row's bits do not depend on the batch it is computed in, so the results are those of
  // one call over all rows.
  const int64_t T0 = T >= kHostSplitRows ? (T / 2 + 255) / 256 * 256 : T;
  const int nparts = T0 < T ? 2 : 1;
  if (nparts == 2 && (dst = device_copy_stream(dev)) != LP_OK) return dst;
  // the shared events are recorded and waited on under the device's lock (only enqueueing
  // happens while it is held)
  std::unique_lock<std::mutex> host_lock(dev->host_mu, std::defer_lock);
  if (nparts == 2) host_lock.lock();
  char* ws = static_cast<char*>(workspace);
  char* dX = ws + L.off_x;
  int32_t* dy = reinterpret_cast<int32_t*>(ws + L.off_y);
  float* d_logp = reinterpret_cast<float*>(ws + L.off_logp);
  float* d_lse = reinterpret_cast<float*>(ws + L.off_lse);
  float* d_ent = out_host->entropy != nullptr ? reinterpret_cast<float*>(ws + L.off_ent) : nullptr;
  float* d_ss = out_host->shard_stats != nullptr ? reinterpret_cast<float*>(ws + L.off_ss) : nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t cs = nparts == 2 ? dev->copy_stream : s;
  const size_t row_x = size_t(H) * 2;
  auto fail = [] {
    cudaGetLastError();
    return LP_ERR_CUDA;
  };
  // copies: on the caller's stream (one part), or on the copy stream after the caller's
  // earlier work (which may still use the staging), one event per part
  if (nparts == 2 && (cudaEventRecord(dev->ev[0], s) != cudaSuccess || cudaStreamWaitEvent(cs, dev->ev[0], 0) != cudaSuccess))
    return fail();
  for (int c = 0; c < nparts; ++c) {
    const int64_t r0 = c == 0 ? 0 : T0, rows = (c == 0 ? T0 : T) - r0;
    if (cudaMemcpyAsync(dX + size_t(r0) * row_x, static_cast<const char*>(X_host) + size_t(r0) * row_x,
                        size_t(rows) * row_x, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(dy + r0, y_host + r0, size_t(rows) * 4, cudaMemcpyHostToDevice, cs) != cudaSuccess)
      return fail();
    if (nparts == 2 && cudaEventRecord(dev->ev[1 + c], cs) != cudaSuccess) return fail();
  }
  // the forward of each part on the caller's stream, once its rows have arrived. lp_forward
  // validates W, bias and the device before it launches anything, so a rejected call has
  // enqueued at most the input copies.
  const size_t fws = forward_ws_bytes(T0, sh);
  for (int c = 0; c < nparts; ++c) {
    const int64_t r0 = c == 0 ? 0 : T0, rows = (c == 0 ? T0 : T) - r0;
    if (nparts == 2 && cudaStreamWaitEvent(s, dev->ev[1 + c], 0) != cudaSuccess) return fail();
    lp_outputs o;
    o.logp = d_logp + r0;
    o.lse = d_lse + r0;
    o.entropy = d_ent != nullptr ? d_ent + r0 : nullptr;
    o.shard_stats = d_ss != nullptr ? d_ss + size_t(sh.n) * 3 * size_t(r0) : nullptr;  // [K][3][rows] per part
    const lp_status st = lp_forward(dX + size_t(r0) * row_x, rows, H, W, bias, part, dy + r0, tau, &o, ws, fws, stream);
    if (st != LP_OK) return st;
  }
  // outputs back on the caller's stream
  const size_t tb = size_t(T) * 4;
  if (cudaMemcpyAsync(out_host->logp, d_logp, tb, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(out_host->lse, d_lse, tb, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      (d_ent != nullptr && cudaMemcpyAsync(out_host->entropy, d_ent, tb, cudaMemcpyDeviceToHost, s) != cudaSuccess))
    return fail();
  if (d_ss != nullptr) {
    // part c's statistics are [K * 3][rows_c] rows of floats; host rows are T floats apart
    for (int c = 0; c < nparts; ++c) {
      const int64_t r0 = c == 0 ? 0 : T0, rows = (c == 0 ? T0 : T) - r0;
      if (cudaMemcpy2DAsync(out_host->shard_stats + r0, tb, d_ss + size_t(sh.n) * 3 * size_t(r0), size_t(rows) * 4,
                            size_t(rows) * 4, size_t(sh.n) * 3, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return fail();
    }
  }
  return LP_OK;
}

lp_status lp_forward_from_logits(const void* const* logits, const int64_t* ld, int64_t T,
                                 const lp_vocab_partition* part, const int32_t* y, float tau,
                                 const lp_outputs* out, void* workspace, size_t ws_bytes, lp_stream_t stream) {
  (void)workspace;
  (void)ws_bytes;
  Shards sh;
  if (check_partition(part, &sh) != LP_OK) return LP_ERR_INVALID_ARG;
  if (!valid_rows(T) || !valid_tau(tau)) return LP_ERR_INVALID_ARG;
  if (T == 0) return LP_OK;
  if (logits == nullptr || ld == nullptr || y == nullptr || out == nullptr || out->logp == nullptr ||
      out->lse == nullptr)
    return LP_ERR_INVALID_ARG;
  for (int k = 0; k < sh.n; ++k) {
    if (sh.real[k] == 0) continue;
    if (logits[k] == nullptr || ld[k] < sh.width[k]) return LP_ERR_INVALID_ARG;
    if (!aligned16(logits[k]) || ld[k] % 8 != 0) return LP_ERR_ALIGNMENT;
  }
  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;

  StreamParams p;
  std::memset(&p, 0, sizeof(p));
  for (int k = 0; k < sh.n; ++k) {
    p.logits[k] = static_cast<const __nv_bfloat16*>(logits[k]);
    p.ld[k] = ld[k];
    p.shard_start[k] = sh.start[k];
    p.shard_width[k] = sh.real[k];
    p.shard_end[k] = sh.end[k];
  }
  p.y = y;
  p.logp = out->logp;
  p.lse = out->lse;
  p.entropy = out->entropy;
  p.shard_stats = out->shard_stats;
  p.err = dev->err;
  p.vocab_real = sh.vocab_real;
  p.n_shards = sh.n;
  p.T = int32_t(T);
  p.scale_log2 = float(1.4426950408889634 / double(tau));
  p.inv_tau = float(1.0 / double(tau));
  if (launch_stream_logits(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LP_ERR_CUDA;
  return LP_OK;
}

static lp_status replay_common(const void* X, int64_t T, int64_t H, const void* const* W, const void* const* bias,
                               const lp_vocab_partition* part, const int32_t* y, float tau, const lp_outputs* out,
                               Shards* sh, ReplayParams* p, DeviceState** dev) {
  if (check_partition(part, sh) != LP_OK) return LP_ERR_INVALID_ARG;
  if (!valid_rows(T) || !valid_hidden(H) || !valid_tau(tau)) return LP_ERR_INVALID_ARG;
  if (T == 0) return LP_OK;  // callers check T before using the filled parameters
  if (X == nullptr || W == nullptr || y == nullptr || out == nullptr || out->logp == nullptr ||
      out->lse == nullptr || out->entropy != nullptr)
    return LP_ERR_INVALID_ARG;
  for (int k = 0; k < sh->n; ++k) {
    if (sh->real[k] == 0) continue;
    if (W[k] == nullptr) return LP_ERR_INVALID_ARG;
    if (!aligned16(W[k])) return LP_ERR_ALIGNMENT;
  }
  if (!aligned16(X)) return LP_ERR_ALIGNMENT;
  lp_status st = device_state(dev);
  if (st != LP_OK) return st;
  std::memset(p, 0, sizeof(*p));
  p->X = static_cast<const __nv_bfloat16*>(X);
  for (int k = 0; k < sh->n; ++k) {
    p->W[k] = static_cast<const __nv_bfloat16*>(W[k]);
    p->bias[k] = bias != nullptr ? static_cast<const __nv_bfloat16*>(bias[k]) : nullptr;
    p->shard_start[k] = sh->start[k];
    p->shard_end[k] = sh->end[k];
  }
  p->y = y;
  p->logp = out->logp;
  p->lse = out->lse;
  p->shard_stats = out->shard_stats;
  p->err = (*dev)->err;
  p->vocab_real = sh->vocab_real;
  p->n_shards = sh->n;
  p->T = int32_t(T);
  p->H = int32_t(H);
  p->inv_tau = float(1.0 / double(tau));
  return LP_OK;
}

lp_status lp_top_p_replay(const void* X, int64_t T, int64_t H, const void* const* W, const void* const* bias,
                          const lp_vocab_partition* part, const int32_t* replay_ids, const int32_t* y, float tau,
                          const lp_outputs* out, void* workspace, size_t ws_bytes, lp_stream_t stream) {
  (void)workspace;
  (void)ws_bytes;
  Shards sh;
  ReplayParams p;
  DeviceState* dev = nullptr;
  lp_status st = replay_common(X, T, H, W, bias, part, y, tau, out, &sh, &p, &dev);
  if (st != LP_OK || T == 0) return st;
  if (replay_ids == nullptr) return LP_ERR_INVALID_ARG;
  p.ids = replay_ids;
  if (launch_replay(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LP_ERR_CUDA;
  return LP_OK;
}

lp_status lp_top_p_replay_from_logits(const void* const* logits, const int64_t* ld, int64_t T,
                                      const lp_vocab_partition* part, const int32_t* replay_ids, const int32_t* y,
                                      float tau, const lp_outputs* out, void* workspace, size_t ws_bytes,
                                      lp_stream_t stream) {
  (void)workspace;
  (void)ws_bytes;
  Shards sh;
  if (check_partition(part, &sh) != LP_OK) return LP_ERR_INVALID_ARG;
  if (!valid_rows(T) || !valid_tau(tau)) return LP_ERR_INVALID_ARG;
  if (T == 0) return LP_OK;
  if (logits == nullptr || ld == nullptr || replay_ids == nullptr || y == nullptr || out == nullptr ||
      out->logp == nullptr || out->lse == nullptr || out->entropy != nullptr)
    return LP_ERR_INVALID_ARG;
  for (int k = 0; k < sh.n; ++k)
    if (sh.real[k] > 0 && (logits[k] == nullptr || ld[k] < sh.width[k])) return LP_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;
  ReplayParams p;
  std::memset(&p, 0, sizeof(p));
  for (int k = 0; k < sh.n; ++k) {
    p.logits[k] = static_cast<const __nv_bfloat16*>(logits[k]);
    p.ld[k] = ld[k];
    p.shard_start[k] = sh.start[k];
    p.shard_end[k] = sh.end[k];
  }
  p.ids = replay_ids;
  p.y = y;
  p.logp = out->logp;
  p.lse = out->lse;
  p.shard_stats = out->shard_stats;
  p.err = dev->err;
  p.vocab_real = sh.vocab_real;
  p.n_shards = sh.n;
  p.T = int32_t(T);
  p.inv_tau = float(1.0 / double(tau));
  if (launch_replay_from_logits(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LP_ERR_CUDA;
  return LP_OK;
}

lp_status lp_top_p_replay_dense_mask(const void* X, int64_t T, int64_t H, const void* const* W,
                                     const void* const* bias, const lp_vocab_partition* part,
                                     const uint8_t* const* keep_mask, const int32_t* y, float tau,
                                     const lp_outputs* out, void* workspace, size_t ws_bytes, lp_stream_t stream) {
  Shards sh;
  ReplayParams p;
  DeviceState* dev = nullptr;
  lp_status st = replay_common(X, T, H, W, bias, part, y, tau, out, &sh, &p, &dev);
  if (st != LP_OK || T == 0) return st;
  if (keep_mask == nullptr) return LP_ERR_INVALID_ARG;
  for (int k = 0; k < sh.n; ++k)
    if (sh.real[k] > 0 && keep_mask[k] == nullptr) return LP_ERR_INVALID_ARG;
  const size_t need = align_up(size_t(T) * LP_REPLAY_SLOTS * sizeof(int32_t), 256);
  if (workspace == nullptr || ws_bytes < need) return LP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return LP_ERR_ALIGNMENT;
  MaskParams mp;
  std::memset(&mp, 0, sizeof(mp));
  for (int k = 0; k < sh.n; ++k) {
    mp.mask[k] = keep_mask[k];
    mp.shard_start[k] = sh.start[k];
    mp.shard_width[k] = sh.width[k];
  }
  mp.ids_out = static_cast<int32_t*>(workspace);
  mp.err = dev->err;
  mp.vocab_real = sh.vocab_real;
  mp.n_shards = sh.n;
  mp.T = int32_t(T);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (launch_mask_compact(mp, s) != cudaSuccess) return LP_ERR_CUDA;
  p.ids = mp.ids_out;
  if (launch_replay(p, s) != cudaSuccess) return LP_ERR_CUDA;
  return LP_OK;
}

lp_status lp_backward(const void* X, int64_t T, int64_t H, const void* const* W, const void* const* bias,
                      const lp_vocab_partition* part, const int32_t* y, float tau, const float* lse,
                      const float* grad_logp, const float* entropy, const float* grad_entropy, float* dX,
                      float* const* dW, float* const* db, void* workspace, size_t ws_bytes, lp_stream_t stream) {
  return lp_backward_ex(X, T, H, W, bias, part, y, tau, lse, grad_logp, entropy, grad_entropy, dX,
                        reinterpret_cast<void* const*>(dW), db, nullptr, workspace, ws_bytes, stream);
}

lp_status lp_backward_ex(const void* X, int64_t T, int64_t H, const void* const* W, const void* const* bias,
                         const lp_vocab_partition* part, const int32_t* y, float tau, const float* lse,
                         const float* grad_logp, const float* entropy, const float* grad_entropy, void* dX,
                         void* const* dW, float* const* db, const lp_backward_options* opts, void* workspace,
                         size_t ws_bytes, lp_stream_t stream) {
  Shards sh;
  if (check_partition(part, &sh) != LP_OK) return LP_ERR_INVALID_ARG;
  if (!valid_rows(T) || !valid_hidden(H) || !valid_tau(tau) || dW == nullptr) return LP_ERR_INVALID_ARG;
  const int dx_bf16 = opts != nullptr && opts->dx_dtype == LP_DTYPE_BF16;
  const int accumulate = opts != nullptr ? opts->accumulate : 0;
  const int dw_bf16 = opts != nullptr && opts->dw_dtype == LP_DTYPE_BF16;
  if (opts != nullptr && ((opts->dx_dtype != LP_DTYPE_F32 && opts->dx_dtype != LP_DTYPE_BF16) ||
                          (opts->dw_dtype != LP_DTYPE_F32 && opts->dw_dtype != LP_DTYPE_BF16) ||
                          (accumulate != 0 && accumulate != 1) || (accumulate && dw_bf16)))
    return LP_ERR_INVALID_ARG;
  if (T == 0) {
    // the gradient of an empty sum: dW and db are zero (or unchanged when accumulating),
    // dX has no rows
    for (int k = 0; k < sh.n; ++k)
      if (sh.width[k] > 0 && (dW[k] == nullptr || (db != nullptr && db[k] == nullptr))) return LP_ERR_INVALID_ARG;
    if (accumulate) return LP_OK;
    DeviceState* dev = nullptr;
    lp_status st = device_state(&dev);
    if (st != LP_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int k = 0; k < sh.n; ++k) {
      if (sh.width[k] == 0) continue;
      if (cudaMemsetAsync(dW[k], 0, size_t(sh.width[k]) * size_t(H) * (dw_bf16 ? 2 : 4), s) != cudaSuccess)
        return LP_ERR_CUDA;
      if (db != nullptr && cudaMemsetAsync(db[k], 0, size_t(sh.width[k]) * 4, s) != cudaSuccess) return LP_ERR_CUDA;
    }
    return LP_OK;
  }
  if (X == nullptr || W == nullptr || y == nullptr || lse == nullptr || grad_logp == nullptr || dX == nullptr ||
      ((entropy == nullptr) != (grad_entropy == nullptr)))
    return LP_ERR_INVALID_ARG;
  for (int k = 0; k < sh.n; ++k) {
    if (sh.width[k] == 0) continue;
    if ((sh.real[k] > 0 && W[k] == nullptr) || dW[k] == nullptr || (db != nullptr && db[k] == nullptr))
      return LP_ERR_INVALID_ARG;
    if ((sh.real[k] > 0 && !aligned16(W[k])) || !aligned16(dW[k])) return LP_ERR_ALIGNMENT;
  }
  if (!aligned16(X) || !aligned16(dX) || !aligned16(workspace)) return LP_ERR_ALIGNMENT;
  {
    // tiles are counted in 32-bit integers on the device
    int64_t nb_total = 0;
    for (int k = 0; k < sh.n; ++k) nb_total += (sh.real[k] + kFwdBlockN - 1) / kFwdBlockN;
    if (nb_total * ((T + kFwdBlockM - 1) / kFwdBlockM + kFwdClusterM) > int64_t(INT32_MAX)) return LP_ERR_INVALID_ARG;
  }
  const size_t need = backward_ws_bytes(T, H, sh);
  if (workspace == nullptr || ws_bytes < need) return LP_ERR_WORKSPACE_TOO_SMALL;
  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;
  BackwardArgs a;
  a.X = X;
  a.T = T;
  a.H = H;
  a.y = y;
  a.tau = tau;
  a.lse = lse;
  a.grad = grad_logp;
  a.entropy = entropy;
  a.grad_entropy = grad_entropy;
  a.dX = dX;
  a.dx_bf16 = dx_bf16;
  a.accumulate = accumulate;
  a.dw_bf16 = dw_bf16;
  for (int k = 0; k < sh.n; ++k) {
    a.W[k] = W[k];
    a.bias[k] = bias != nullptr ? bias[k] : nullptr;
    a.dW[k] = dW[k];
    a.db[k] = db != nullptr ? db[k] : nullptr;
  }
  a.workspace = workspace;
  a.err = dev->err;
  a.num_sms = dev->num_sms;
  return run_backward(a, sh, reinterpret_cast<cudaStream_t>(stream));
}

// byte range [lo, hi) spanned by rows of `width` elements of `esz` bytes at stride ld
struct Span {
  uintptr_t lo, hi;
};

static Span row_span(const void* base, int64_t T, int64_t width, int64_t ld, int64_t esz) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(base);
  return Span{lo, lo + uintptr_t(((T - 1) * ld + width) * esz)};
}

static bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

lp_status lp_backward_from_logits(const void* const* logits, const int64_t* ld, int64_t T,
                                  const lp_vocab_partition* part, const int32_t* y, float tau, const float* lse,
                                  const float* grad_logp, const float* entropy, const float* grad_entropy,
                                  void* const* dlogits, const int64_t* ld_out, lp_dtype out_dtype,
                                  lp_stream_t stream) {
  Shards sh;
  if (check_partition(part, &sh) != LP_OK) return LP_ERR_INVALID_ARG;
  if (!valid_rows(T) || !valid_tau(tau)) return LP_ERR_INVALID_ARG;
  if (out_dtype != LP_DTYPE_F32 && out_dtype != LP_DTYPE_BF16) return LP_ERR_INVALID_ARG;
  if (T == 0) return LP_OK;
  if (logits == nullptr || ld == nullptr || y == nullptr || lse == nullptr || grad_logp == nullptr ||
      dlogits == nullptr || ld_out == nullptr || ((entropy == nullptr) != (grad_entropy == nullptr)))
    return LP_ERR_INVALID_ARG;
  const bool bf16 = out_dtype == LP_DTYPE_BF16;
  const int64_t esz = bf16 ? 2 : 4;
  for (int k = 0; k < sh.n; ++k) {
    if (sh.width[k] == 0) continue;
    if (sh.real[k] > 0) {
      if (logits[k] == nullptr || ld[k] < sh.width[k]) return LP_ERR_INVALID_ARG;
      if (!aligned16(logits[k]) || ld[k] % 8 != 0) return LP_ERR_ALIGNMENT;
    }
    if (dlogits[k] == nullptr || ld_out[k] < sh.width[k]) return LP_ERR_INVALID_ARG;
    if (!aligned16(dlogits[k]) || ld_out[k] % (16 / esz) != 0) return LP_ERR_ALIGNMENT;
  }
  // outputs may not overlap each other, nor any shard's logits except their own shard's
  // exactly (the in-place form)
  for (int k = 0; k < sh.n; ++k) {
    if (sh.width[k] == 0) continue;
    const Span o = row_span(dlogits[k], T, sh.width[k], ld_out[k], esz);
    for (int j = 0; j < sh.n; ++j) {
      if (sh.width[j] == 0) continue;
      if (j != k && overlap(o, row_span(dlogits[j], T, sh.width[j], ld_out[j], esz))) return LP_ERR_INVALID_ARG;
      if (sh.real[j] == 0) continue;
      const bool in_place = j == k && bf16 && dlogits[k] == logits[k] && ld_out[k] == ld[k];
      if (!in_place && overlap(o, row_span(logits[j], T, sh.width[j], ld[j], 2))) return LP_ERR_INVALID_ARG;
    }
  }
  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;

  LogitsGradParams p;
  std::memset(&p, 0, sizeof(p));
  for (int k = 0; k < sh.n; ++k) {
    p.logits[k] = static_cast<const __nv_bfloat16*>(logits[k]);
    p.out[k] = dlogits[k];
    p.ld[k] = ld[k];
    p.ld_out[k] = ld_out[k];
    p.shard_start[k] = sh.start[k];
    p.width[k] = sh.width[k];
    p.real[k] = sh.real[k];
  }
  p.y = y;
  p.lse = lse;
  p.grad = grad_logp;
  p.entropy = entropy;
  p.grad_entropy = grad_entropy;
  p.vocab_real = sh.vocab_real;
  p.n_shards = sh.n;
  p.T = int32_t(T);
  p.out_bf16 = bf16 ? 1 : 0;
  p.err = dev->err;
  p.scale_log2 = float(1.4426950408889634 / double(tau));
  p.inv_tau = float(1.0 / double(tau));
  if (launch_logits_backward(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LP_ERR_CUDA;
  return LP_OK;
}

lp_status lp_merge_shard_stats(const float* shard_stats, int64_t T, const lp_vocab_partition* part,
                               const int32_t* y, const lp_outputs* out, lp_stream_t stream) {
  Shards sh;
  if (check_partition(part, &sh) != LP_OK) return LP_ERR_INVALID_ARG;
  if (!valid_rows(T)) return LP_ERR_INVALID_ARG;
  if (T == 0) return LP_OK;
  if (shard_stats == nullptr || y == nullptr || out == nullptr || out->logp == nullptr || out->lse == nullptr ||
      out->shard_stats != nullptr)
    return LP_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;
  MergeStatsParams p;
  std::memset(&p, 0, sizeof(p));
  p.stats = shard_stats;
  p.y = y;
  p.logp = out->logp;
  p.lse = out->lse;
  p.entropy = out->entropy;
  p.err = dev->err;
  p.vocab_real = sh.vocab_real;
  for (int k = 0; k < sh.n; ++k) {
    p.shard_start[k] = sh.start[k];
    p.shard_end[k] = sh.end[k];
  }
  p.n_shards = sh.n;
  p.T = int32_t(T);
  if (launch_merge_stats(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LP_ERR_CUDA;
  return LP_OK;
}

lp_status lp_sum_partials(const float* const* parts, int32_t n_parts, int64_t count, void* out, lp_dtype out_dtype,
                          lp_stream_t stream) {
  if (n_parts < 1 || n_parts > LP_MAX_PARTS || count < 0 || parts == nullptr) return LP_ERR_INVALID_ARG;
  if (out_dtype != LP_DTYPE_F32 && out_dtype != LP_DTYPE_BF16) return LP_ERR_INVALID_ARG;
  if (count == 0) return LP_OK;
  if (out == nullptr) return LP_ERR_INVALID_ARG;
  const int64_t esz = out_dtype == LP_DTYPE_BF16 ? 2 : 4;
  const Span o = row_span(out, 1, count, count, esz);
  for (int i = 0; i < n_parts; ++i) {
    if (parts[i] == nullptr) return LP_ERR_INVALID_ARG;
    if (!aligned16(parts[i])) return LP_ERR_ALIGNMENT;
    const bool in_place = i == 0 && parts[0] == out && out_dtype == LP_DTYPE_F32;
    if (!in_place && overlap(o, row_span(parts[i], 1, count, count, 4))) return LP_ERR_INVALID_ARG;
  }
  if (!aligned16(out)) return LP_ERR_ALIGNMENT;
  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;
  SumPartsParams p;
  std::memset(&p, 0, sizeof(p));
  for (int i = 0; i < n_parts; ++i) p.parts[i] = parts[i];
  p.out = out;
  p.count = count;
  p.n_parts = n_parts;
  p.out_bf16 = out_dtype == LP_DTYPE_BF16 ? 1 : 0;
  if (launch_sum_partials(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LP_ERR_CUDA;
  return LP_OK;
}

int lp_debug_bounds_build(void) { return LP_DEBUG_BOUNDS ? 1 : 0; }

#ifndef LP_SOURCE_HASH
#define LP_SOURCE_HASH "unknown"
#endif
const char* lp_build_id(void) { return LP_SOURCE_HASH; }

lp_status lp_selftest_bounds(lp_stream_t stream) {
  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;
  bounds_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(int64_t(1), dev->err);
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

lp_status lp_set_wait_limit(uint64_t limit_ns) {
  if (limit_ns == 0) limit_ns = kDefaultWaitLimitNs;
  if (limit_ns < 1000ull || limit_ns > 10000000000ull) return LP_ERR_INVALID_ARG;
  g_wait_limit.store(limit_ns, std::memory_order_relaxed);
  return LP_OK;
}

lp_status lp_selftest_wait_timeout(uint64_t limit_ns, lp_stream_t stream) {
  if (limit_ns < 1000ull || limit_ns > 2000000000ull) return LP_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;
  wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, dev->err);
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

lp_status lp_get_device_error(lp_stream_t stream) {
  DeviceState* dev = nullptr;
  lp_status st = device_state(&dev);
  if (st != LP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int word = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LP_ERR_CUDA;
  if (cudaMemcpyAsync(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return LP_ERR_CUDA;
  if (cudaMemsetAsync(dev->err, 0, sizeof(word), s) != cudaSuccess) return LP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LP_ERR_CUDA;
  return static_cast<lp_status>(word);
}

}  // extern "C"
