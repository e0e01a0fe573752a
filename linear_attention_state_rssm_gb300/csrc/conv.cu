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
// One thread per (row, 16 bytes of consecutive channels): every access is a
// 16-byte vector and a warp's accesses are consecutive; a thread issues the
// loads of up to eight tokens before it uses them, and keeps the window, the
// taps and the bias in registers across the tokens. The work is a few flops
// per byte: HBM-bound.
#include "rssm_common.cuh"
#include "rssm_launch.h"

namespace rssm {

constexpr int kConvThreads = 128;
constexpr int kConvTok = 8;  // tokens whose loads are in flight together

// 16 bytes of EPV values (bf16 when EPV = 8, fp32 when EPV = 4) <-> fp32
template <int EPV>
__device__ __forceinline__ void unpack16(const uint4& u, float (&v)[EPV]) {
  if (EPV == 4) {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[EPV - 1] = __uint_as_float(u.w);
  } else {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[t]));
      v[(2 * t) % EPV] = f.x;
      v[(2 * t + 1) % EPV] = f.y;
    }
  }
}

template <int EPV>
__device__ __forceinline__ uint4 pack16(const float (&v)[EPV]) {
  if (EPV == 4) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[EPV - 1]));
  }
  uint32_t w[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[(2 * t) % EPV], v[(2 * t + 1) % EPV]);
    w[t] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One thread per (row, group of EPV consecutive channels).
template <int K, int EPV>
__global__ void __launch_bounds__(kConvThreads) conv_window_kernel(const ConvParams p) {
  const int D = p.D, T = p.T;
  const int g = blockIdx.x * kConvThreads + threadIdx.x, r = blockIdx.y;
  if (g * EPV >= D) return;
  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (g == 0 && p.err != nullptr) atomicOr(p.err, DEVERR_SLOT);
    return;
  }
  const int c0 = g * EPV, nv = D / EPV;  // 16-byte vectors per row of D channels
  const uint4* x = static_cast<const uint4*>(p.x);
  uint4* y = static_cast<uint4*>(p.y);
  uint4* win_g = static_cast<uint4*>(p.window) + (size_t)s * (K - 1) * nv + g;
  uint4* draft = static_cast<uint4*>(p.draft);

  float taps[EPV][K], b[EPV], win[K - 1][EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) {
#pragma unroll
    for (int i = 0; i < K; ++i) taps[e][i] = p.w[(size_t)(c0 + e) * K + i];
    b[e] = p.bias != nullptr ? p.bias[c0 + e] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < K - 1; ++i) unpack16<EPV>(win_g[(size_t)i * nv], win[i]);

  for (int t0 = 0; t0 < T; t0 += kConvTok) {
    uint4 xr[kConvTok];
#pragma unroll
    for (int u = 0; u < kConvTok; ++u) {
      if (t0 + u < T) xr[u] = __ldg(x + ((size_t)r * T + t0 + u) * nv + g);
    }
#pragma unroll
    for (int u = 0; u < kConvTok; ++u) {
      if (t0 + u < T) {
        const size_t xi = ((size_t)r * T + t0 + u) * nv + g;
        float xv[EPV], yv[EPV];
        unpack16<EPV>(xr[u], xv);
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          float acc = b[e];
#pragma unroll
          for (int i = 0; i < K - 1; ++i) acc = fmaf(taps[e][i], win[i][e], acc);
          acc = fmaf(taps[e][K - 1], xv[e], acc);
          if (p.act == CONV_ACT_SILU) acc = acc / (1.f + __expf(-acc));
          yv[e] = acc;
        }
        y[xi] = pack16<EPV>(yv);
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
    for (int i = 0; i < K - 1; ++i) win_g[(size_t)i * nv] = pack16<EPV>(win[i]);
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
#define RSSM_CONV_CASE(KV)                                                        \
  case KV:                                                                        \
    if (commit) {                                                                 \
      conv_commit_kernel<KV><<<grid, kConvThreads, 0, st>>>(p);                   \
    } else if (f32) {                                                             \
      conv_window_kernel<KV, 4><<<grid, kConvThreads, 0, st>>>(p);                \
    } else {                                                                      \
      conv_window_kernel<KV, 8><<<grid, kConvThreads, 0, st>>>(p);                \
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
