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
// One thread per (row, channel): consecutive channels are consecutive
// addresses in every buffer, so each access of a warp is one coalesced line;
// the window and the taps stay in registers across the tokens. The work is a
// few flops per byte: HBM-bound.
#include "rssm_common.cuh"
#include "rssm_launch.h"

namespace rssm {

constexpr int kConvThreads = 128;

template <int K>
__global__ void __launch_bounds__(kConvThreads) conv_window_kernel(const ConvParams p) {
  const int c = blockIdx.x * kConvThreads + threadIdx.x, r = blockIdx.y;
  if (c >= p.D) return;
  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (c == 0 && p.err != nullptr) atomicOr(p.err, DEVERR_SLOT);
    return;
  }
  const int D = p.D, T = p.T;
  float taps[K], win[K - 1];
#pragma unroll
  for (int i = 0; i < K; ++i) taps[i] = p.w[(size_t)c * K + i];
  const size_t wbase = (size_t)s * (K - 1) * D + c;
#pragma unroll
  for (int i = 0; i < K - 1; ++i) win[i] = ld_f32(p.window, wbase + (size_t)i * D, p.dt);
  const float b = p.bias != nullptr ? p.bias[c] : 0.f;
  for (int t = 0; t < T; ++t) {
    const size_t xi = ((size_t)r * T + t) * D + c;
    const float xt = ld_f32(p.x, xi, p.dt);
    float acc = b;
#pragma unroll
    for (int i = 0; i < K - 1; ++i) acc = fmaf(taps[i], win[i], acc);
    acc = fmaf(taps[K - 1], xt, acc);
    if (p.act == CONV_ACT_SILU) acc = acc / (1.f + __expf(-acc));
    st_f32(p.y, xi, p.dt, acc);
    if (!p.commit_now) st_f32(p.draft, ((size_t)s * T + t) * D + c, p.dt, xt);
#pragma unroll
    for (int i = 0; i < K - 2; ++i) win[i] = win[i + 1];
    win[K - 2] = xt;
  }
  if (p.commit_now) {
#pragma unroll
    for (int i = 0; i < K - 1; ++i) st_f32(p.window, wbase + (size_t)i * D, p.dt, win[i]);
  }
}

// window <- the last K-1 rows of [window, draft_0 .. draft_{a-1}]
template <int K>
__global__ void __launch_bounds__(kConvThreads) conv_commit_kernel(const ConvParams p) {
  const int c = blockIdx.x * kConvThreads + threadIdx.x, r = blockIdx.y;
  if (c >= p.D) return;
  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (c == 0 && p.err != nullptr) atomicOr(p.err, DEVERR_SLOT);
    return;
  }
  const int a = p.accept[r];
  if (a < 0 || a > p.T) {
    if (c == 0 && p.err != nullptr) atomicOr(p.err, DEVERR_ACCEPT);
    return;
  }
  const int D = p.D;
  const size_t wbase = (size_t)s * (K - 1) * D + c;
  float nw[K - 1];
#pragma unroll
  for (int i = 0; i < K - 1; ++i) {
    const int idx = a + i;  // position in [window (K-1 rows), drafts]
    nw[i] = idx < K - 1 ? ld_f32(p.window, wbase + (size_t)idx * D, p.dt)
                        : ld_f32(p.draft, ((size_t)s * p.T + idx - (K - 1)) * D + c, p.dt);
  }
#pragma unroll
  for (int i = 0; i < K - 1; ++i) st_f32(p.window, wbase + (size_t)i * D, p.dt, nw[i]);
}

cudaError_t conv_launch(const ConvParams& p, bool commit, cudaStream_t st) {
  const dim3 grid((unsigned)((p.D + kConvThreads - 1) / kConvThreads), (unsigned)p.B, 1);
#define RSSM_CONV_CASE(KV)                                                        \
  case KV:                                                                        \
    if (commit) {                                                                 \
      conv_commit_kernel<KV><<<grid, kConvThreads, 0, st>>>(p);                   \
    } else {                                                                      \
      conv_window_kernel<KV><<<grid, kConvThreads, 0, st>>>(p);                   \
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
