// Conv-state window of the layer's short causal convolution, and its rollback
// on commit (LightLLM PR #1690 "feat: add ReplaySSM state modes for GDN and
// KDA", commit messages: the accepted conv window is the per-request conv
// state that page save, PD and DP copy; SGLang fork PR jianc99/sglang#2, fifth
// commit: the ring commit rolls the conv back with the cursor and the fold).
//
// Per request row and channel c, with the kept window of K-1 inputs:
//     y_t[c] = act(bias[c] + sum_{i<K} w[c][i] * xp[t + i][c]),
//     xp = [window, x_0, ..., x_{T-1}],  act = identity or SiLU.
// A verify window leaves the window as it is and keeps its T inputs as drafts;
// the commit makes the window the last K-1 rows of [window, x_0 .. x_{a-1}].
// Decode commits its token at once.
//
// One thread per (row, four consecutive channels): every access is one vector
// (8 bytes of bf16, 16 of fp32) and a warp's accesses are consecutive; a
// thread issues the loads of up to four tokens before it uses them and keeps
// the window, the taps and the bias in registers across the tokens, few
// enough that many threads, and their loads, are in flight. The work is a few
// flops per byte: HBM-bound.
#include "rssm_common.cuh"
#include "rssm_launch.h"

#include <type_traits>

namespace rssm {

constexpr int kConvThreads = 128;
constexpr int kConvTok = 4;  // tokens whose loads are in flight together

// VW 32-bit words of values (bf16 pairs or fp32) <-> fp32
template <int VW, bool BF>
struct ConvVec {
  static constexpr int kVals = BF ? 2 * VW : VW;
  using T = typename std::conditional<VW == 4, uint4, uint2>::type;
  static __device__ __forceinline__ void unpack(const T& u, float (&v)[kVals]) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&u);
#pragma unroll
    for (int t = 0; t < VW; ++t) {
      if (BF) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[t]));
        v[(2 * t) % kVals] = f.x;
        v[(2 * t + 1) % kVals] = f.y;
      } else {
        v[t % kVals] = __uint_as_float(w[t]);
      }
    }
  }
  static __device__ __forceinline__ T pack(const float (&v)[kVals]) {
    T u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int t = 0; t < VW; ++t) {
      if (BF) {
        const __nv_bfloat162 hh = __floats2bfloat162_rn(v[(2 * t) % kVals], v[(2 * t + 1) % kVals]);
        w[t] = *reinterpret_cast<const uint32_t*>(&hh);
      } else {
        w[t] = __float_as_uint(v[t % kVals]);
      }
    }
    return u;
  }
};

// One thread per (row, group of EPV consecutive channels) in VW-word vectors.
template <int K, int VW, bool BF>
__global__ void __launch_bounds__(kConvThreads) conv_window_kernel(const ConvParams p) {
  using Vec = ConvVec<VW, BF>;
  using VT = typename Vec::T;
  constexpr int EPV = Vec::kVals;
  const int D = p.D, T = p.T;
  const int g = blockIdx.x * kConvThreads + threadIdx.x, r = blockIdx.y;
  if (g * EPV >= D) return;
  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (g == 0 && p.err != nullptr) atomicOr(p.err, DEVERR_SLOT);
    return;
  }
  const int c0 = g * EPV, nv = D / EPV;  // vectors per row of D channels
  const VT* x = static_cast<const VT*>(p.x);
  VT* y = static_cast<VT*>(p.y);
  VT* win_g = static_cast<VT*>(p.window) + (size_t)s * (K - 1) * nv + g;
  VT* draft = static_cast<VT*>(p.draft);

  float taps[EPV][K], b[EPV], win[K - 1][EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) {
#pragma unroll
    for (int i = 0; i < K; ++i) taps[e][i] = p.w[(size_t)(c0 + e) * K + i];
    b[e] = p.bias != nullptr ? p.bias[c0 + e] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < K - 1; ++i) Vec::unpack(win_g[(size_t)i * nv], win[i]);

  for (int t0 = 0; t0 < T; t0 += kConvTok) {
    VT xr[kConvTok];
#pragma unroll
    for (int u = 0; u < kConvTok; ++u) {
      if (t0 + u < T) xr[u] = __ldg(x + ((size_t)r * T + t0 + u) * nv + g);
    }
#pragma unroll
    for (int u = 0; u < kConvTok; ++u) {
      if (t0 + u < T) {
        const size_t xi = ((size_t)r * T + t0 + u) * nv + g;
        float xv[EPV], yv[EPV];
        Vec::unpack(xr[u], xv);
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          float acc = b[e];
#pragma unroll
          for (int i = 0; i < K - 1; ++i) acc = fmaf(taps[e][i], win[i][e], acc);
          acc = fmaf(taps[e][K - 1], xv[e], acc);
          if (p.act == CONV_ACT_SILU) acc = acc / (1.f + __expf(-acc));
          yv[e] = acc;
        }
        y[xi] = Vec::pack(yv);
        if (!p.commit_now) draft[((size_t)s * T + t0 + u) * nv + g] = xr[u];
#pragma unroll
        for (int i = 0; i < K - 2; ++i) {
#pragma unroll
          for (int e = 0; e < EPV; ++e) win[i][e] = win[i + 1][e];
        }
#pragma unroll
        for (int e = 0; e < EPV; ++e) win[K - 2][e] = xv[e];
      }
    }
  }
  if (p.commit_now) {
#pragma unroll
    for (int i = 0; i < K - 1; ++i) win_g[(size_t)i * nv] = Vec::pack(win[i]);
  }
}

// window <- the last K-1 rows of [window, draft_0 .. draft_{a-1}] (raw copies)
template <int K>
__global__ void __launch_bounds__(kConvThreads) conv_commit_kernel(const ConvParams p) {
  const int nv = p.D * dtype_bytes(p.dt) / 16;
  const int g = blockIdx.x * kConvThreads + threadIdx.x, r = blockIdx.y;
  if (g >= nv) return;
  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (g == 0 && p.err != nullptr) atomicOr(p.err, DEVERR_SLOT);
    return;
  }
  const int a = p.accept[r];
  if (a < 0 || a > p.T) {
    if (g == 0 && p.err != nullptr) atomicOr(p.err, DEVERR_ACCEPT);
    return;
  }
  uint4* win_g = static_cast<uint4*>(p.window) + (size_t)s * (K - 1) * nv + g;
  const uint4* draft = static_cast<const uint4*>(p.draft);
  uint4 nw[K - 1];
#pragma unroll
  for (int i = 0; i < K - 1; ++i) {
    const int idx = a + i;  // position in [window (K-1 rows), drafts]
    nw[i] = idx < K - 1 ? win_g[(size_t)idx * nv]
                        : draft[((size_t)s * p.T + idx - (K - 1)) * nv + g];
  }
#pragma unroll
  for (int i = 0; i < K - 1; ++i) win_g[(size_t)i * nv] = nw[i];
}

cudaError_t conv_launch(const ConvParams& p, bool commit, cudaStream_t st) {
  const bool f32 = p.dt == DT_F32;
  const int nv = p.D * (f32 ? 4 : 2) / 16;
  const dim3 grid((unsigned)((nv + kConvThreads - 1) / kConvThreads), (unsigned)p.B, 1);
  const int nw = p.D / 4;  // four channels per window thread
  const dim3 wgrid((unsigned)((nw + kConvThreads - 1) / kConvThreads), (unsigned)p.B, 1);
#define RSSM_CONV_CASE(KV)                                                        \
  case KV:                                                                        \
    if (commit) {                                                                 \
      conv_commit_kernel<KV><<<grid, kConvThreads, 0, st>>>(p);                   \
    } else if (f32) {                                                             \
      conv_window_kernel<KV, 4, false><<<wgrid, kConvThreads, 0, st>>>(p);        \
    } else {                                                                      \
      conv_window_kernel<KV, 2, true><<<wgrid, kConvThreads, 0, st>>>(p);         \
    }                                                                             \
    break;
  switch (p.K) {
    RSSM_CONV_CASE(2)
    RSSM_CONV_CASE(3)
    RSSM_CONV_CASE(4)
    RSSM_CONV_CASE(5)
    RSSM_CONV_CASE(6)
    RSSM_CONV_CASE(7)
    RSSM_CONV_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef RSSM_CONV_CASE
  return cudaGetLastError();
}

}  // namespace rssm
