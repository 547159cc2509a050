// lp_logits_backward.cu - gradient of the logits-reuse route with respect to the
// reused logits.
//
// Page "feat(rl-kernel): add CUDA linear logp provider integration", Megatron
// integration: local LM-head logits are reused instead of a second projection, and the
// provider's outputs carry gradients, so the gradient has to flow back into those
// logits. With z = L / tau (temperature applied once), p = exp(z - LSE) and mu = LSE -
// entropy, the gradient of sum_t g_t logp_t + h_t entropy_t is
//     dL[t, v] = (g_t (1[v = y_t] - p_tv) - h_t p_tv (z_tv - mu_t)) / tau,   0 on padded ids.
//
// Purely elementwise once the row's LSE is known, so the kernel is a stream: one CTA
// of 256 threads per row walks each shard's row in 16-byte vectors (8 logits), eight
// vectors in flight per thread, and writes each gradient vector right after reading
// its logits. Per row the gradient is rewritten as
//     dL = g/tau 1[v = y] - p (A + B x),   A = (g - h mu)/tau,  B = h/tau^2,  x = L[t, v],
// so an element costs one ex2 and three packed f32x2 operations (two elements per
// instruction); the one-hot term is added by the thread holding the target. Logits are
// first raised to a per-row floor x_lo, below which 2^(x c2 - LSE log2 e) flushes to 0:
// that leaves every nonzero p unchanged and keeps -inf logits from forming 0 * inf.
// Loads and stores use the streaming cache hints and ordinary (coherent) global
// accesses, so the gradient may overwrite the logits in place. Every element's value
// depends only on its own logit and its row's scalars: the result is deterministic and
// batch invariant by construction.
#include <cuda_bf16.h>

#include "lp_device.cuh"
#include "lp_f32x2.cuh"

namespace lp {

namespace {

#ifndef LP_LG_THREADS
#define LP_LG_THREADS 256  // threads per row
#endif
#ifndef LP_LG_UNROLL
#define LP_LG_UNROLL 8     // 16-byte vectors per thread in flight
#endif
constexpr int kLgThreads = LP_LG_THREADS;
constexpr int kLgUnroll = LP_LG_UNROLL;

struct RowGrad {
  uint64_t c2x2;    // {c2, c2}, c2 = log2(e) / tau
  uint64_t nl2x2;   // {-LSE log2 e, ...}
  uint64_t nbx2;    // {-B, -B}
  uint64_t nax2;    // {-A, -A}
  uint32_t floor2;  // {x_lo, x_lo} in bf16
  float gi;         // g / tau (the one-hot term)
};

// gradients of the 8 logits of one vector (all real ids) into gv[8]
__device__ __forceinline__ void grad8(const RowGrad& r, const uint4 v, float (&gv)[8]) {
  const uint32_t w[4] = {max_bf16x2(v.x, r.floor2), max_bf16x2(v.y, r.floor2), max_bf16x2(v.z, r.floor2),
                         max_bf16x2(v.w, r.floor2)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t x2 = pack2(bf16_lo(w[i]), bf16_hi(w[i]));
    float u0, u1;
    unpack2(fma2(x2, r.c2x2, r.nl2x2), u0, u1);
    const uint64_t p2 = pack2(hw_ex2(u0), hw_ex2(u1));
    unpack2(mul2(p2, fma2(x2, r.nbx2, r.nax2)), gv[2 * i], gv[2 * i + 1]);
  }
}

// gradient of one real logit (scalar form of grad8, same operations and rounding)
__device__ __forceinline__ float grad1(const RowGrad& r, float x) {
  float fl, c2, nl, nb, na;
  unpack2(r.c2x2, c2, c2);
  unpack2(r.nl2x2, nl, nl);
  unpack2(r.nbx2, nb, nb);
  unpack2(r.nax2, na, na);
  fl = bf16_lo(r.floor2);
  const float xc = fmaxf(x, fl);
  return __fmul_rn(hw_ex2(__fmaf_rn(xc, c2, nl)), __fmaf_rn(xc, nb, na));
}

// store 8 gradients at element offset c of an output row (16-byte aligned)
__device__ __forceinline__ void store8(void* row_out, bool bf16, int64_t c, const float (&g)[8]) {
  if (bf16) {
    const uint4 v = make_uint4(cvt_bf16x2(g[0], g[1]), cvt_bf16x2(g[2], g[3]), cvt_bf16x2(g[4], g[5]),
                               cvt_bf16x2(g[6], g[7]));
    __stcs(reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(row_out) + c), v);
  } else {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(row_out) + c);
    __stcs(o, make_float4(g[0], g[1], g[2], g[3]));
    __stcs(o + 1, make_float4(g[4], g[5], g[6], g[7]));
  }
}

__device__ __forceinline__ void store1(void* row_out, bool bf16, int64_t c, float g) {
  if (bf16)
    static_cast<__nv_bfloat16*>(row_out)[c] = __float2bfloat16_rn(g);
  else
    static_cast<float*>(row_out)[c] = g;
}

}  // namespace

__global__ void __launch_bounds__(kLgThreads) logits_backward_kernel(const __grid_constant__ LogitsGradParams p) {
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  const float l = __ldg(p.lse + row);
  const float g = __ldg(p.grad + row);
  const int yv = __ldg(p.y + row);
  // rows without a finite LSE or gradient, or without a valid target, get zeros
  const bool live = isfinite(l) && isfinite(g) && yv >= 0 && int64_t(yv) < p.vocab_real;
  RowGrad r;
  {
    const float gi = __fmul_rn(g, p.inv_tau);
    float hi = 0.f, mu = 0.f;
    if (live && p.grad_entropy != nullptr) {
      const float h = __ldg(p.grad_entropy + row);
      const float e = __ldg(p.entropy + row);
      if (isfinite(h) && isfinite(e)) {
        hi = __fmul_rn(h, p.inv_tau);
        mu = __fsub_rn(l, e);
      }
    }
    const float a = __fsub_rn(gi, __fmul_rn(hi, mu));
    const float b = __fmul_rn(hi, p.inv_tau);
    const float lse2 = __fmul_rn(l, kLog2e);
    // x_lo: 2^(x_lo c2 - lse2) <= 2^-140 flushes to 0; kept finite (also in bf16)
    const float xlo = fmaxf(__fdiv_rn(__fsub_rn(lse2, 140.f), p.scale_log2), -3.0e38f);
    const __nv_bfloat16 flo = __float2bfloat16_rd(live ? xlo : 0.f);
    const uint32_t f16 = *reinterpret_cast<const uint16_t*>(&flo);
    r.c2x2 = pack2(p.scale_log2, p.scale_log2);
    r.nl2x2 = pack2(-lse2, -lse2);
    r.nbx2 = pack2(-b, -b);
    r.nax2 = pack2(-a, -a);
    r.floor2 = f16 | (f16 << 16);
    r.gi = gi;
  }
  const bool bf16 = p.out_bf16 != 0;
  const int esz = bf16 ? 2 : 4;

  for (int k = 0; k < p.n_shards; ++k) {
    const int64_t width = p.width[k];
    if (width == 0) continue;
    const int64_t real = live ? p.real[k] : 0;  // columns that get a computed gradient
    const __nv_bfloat16* L = p.logits[k] + size_t(row) * size_t(p.ld[k]);
    void* O = static_cast<char*>(p.out[k]) + size_t(row) * size_t(p.ld_out[k]) * size_t(esz);
    const int64_t ycol = int64_t(yv) - p.shard_start[k];  // the one-hot column, if in this shard
    const int64_t nfull = real >> 3;                     // vectors of real ids only
    for (int64_t j0 = tid; j0 < nfull; j0 += int64_t(kLgThreads) * kLgUnroll) {
      uint4 v[kLgUnroll];
#pragma unroll
      for (int u = 0; u < kLgUnroll; ++u) {
        const int64_t j = j0 + int64_t(u) * kLgThreads;
        if (j < nfull && in_bounds(8 * (j + 1) <= real && real <= width && width <= p.ld[k], p.err))
          v[u] = __ldcs(reinterpret_cast<const uint4*>(L) + j);
      }
#pragma unroll
      for (int u = 0; u < kLgUnroll; ++u) {
        const int64_t j = j0 + int64_t(u) * kLgThreads;
        if (j >= nfull) break;
        float gv[8];
        grad8(r, v[u], gv);
        const int64_t d = ycol - (j << 3);
        if (d >= 0 && d < 8) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e == d) gv[e] = __fadd_rn(gv[e], r.gi);
        }
        if (in_bounds(8 * (j + 1) <= width && width <= p.ld_out[k], p.err)) store8(O, bf16, j << 3, gv);
      }
    }
    // the rest of the row: the vector holding the last real ids, vectors of padded ids,
    // and the ragged tail (width % 8 columns)
    const int64_t nvec = width >> 3;
    for (int64_t j = nfull + tid; j < nvec; j += kLgThreads) {
      const int64_t c0 = j << 3;
      float gv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int64_t c = c0 + e;
        gv[e] = c < real ? __fadd_rn(grad1(r, __bfloat162float(L[c])), c == ycol ? r.gi : 0.f) : 0.f;
      }
      store8(O, bf16, c0, gv);
    }
    const int64_t c = (nvec << 3) + tid;
    if (c < width)
      store1(O, bf16, c, c < real ? __fadd_rn(grad1(r, __bfloat162float(L[c])), c == ycol ? r.gi : 0.f) : 0.f);
  }
}

cudaError_t launch_logits_backward(const LogitsGradParams& p, cudaStream_t s) {
  logits_backward_kernel<<<unsigned(p.T), kLgThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace lp
