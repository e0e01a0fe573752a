// Instantiation and launch of the replay kernel for one (algorithm, state
// dtype) pair; included by one small translation unit per pair so the build
// compiles them in parallel.
#pragma once

#include "replay_impl.cuh"
#include "rssm_launch.h"

namespace rssm {

// One CTA per (value head, request row).
template <int ALGO, typename ST, int NT, bool RAGGED, bool TC = false, bool LONG = false>
static cudaError_t replay_launch_one(const ReplayParams& p, cudaStream_t st) {
  const dim3 grid((unsigned)p.HV, (unsigned)p.B, 1);
  replay_kernel<ALGO, ST, NT, RAGGED, TC, LONG><<<grid, kThreads, p.sm.total, st>>>(p);
  return cudaGetLastError();
}

template <int ALGO, typename ST, int NT, bool RAGGED, bool TC = false, bool LONG = false>
static cudaError_t replay_prepare_one(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(replay_kernel<ALGO, ST, NT, RAGGED, TC, LONG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(replay_kernel<ALGO, ST, NT, RAGGED, TC, LONG>,
                              cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

// Decode and verify windows of four and eight tokens: GDN takes the
// tensor-core stream kernel when p.tc is set, and on rings longer than 16
// records the kernel whose tensor-core folds take longer histories.
template <int ALGO, typename ST, int NT>
static cudaError_t replay_launch_wide(const ReplayParams& p, cudaStream_t st) {
  if constexpr (ALGO == ALGO_GDN) {
    if constexpr (NT != 1) {
      if (p.tc) return replay_launch_one<ALGO, ST, NT, false, true>(p, st);
    }
    if (p.L > 16) return replay_launch_one<ALGO, ST, NT, false, false, true>(p, st);
  }
  return replay_launch_one<ALGO, ST, NT, false>(p, st);
}

template <int ALGO, typename ST, int NT>
static cudaError_t replay_prepare_wide(int max_smem) {
  if constexpr (ALGO == ALGO_GDN) {
    cudaError_t e;
    if constexpr (NT != 1) {
      if ((e = replay_prepare_one<ALGO, ST, NT, false, true>(max_smem)) != cudaSuccess) return e;
    }
    e = replay_prepare_one<ALGO, ST, NT, false, false, true>(max_smem);
    if (e != cudaSuccess) return e;
  }
  return replay_prepare_one<ALGO, ST, NT, false>(max_smem);
}

}  // namespace rssm

#define RSSM_DEFINE_REPLAY(NAME, ALGO, ST)                                                  \
  namespace rssm {                                                                          \
  cudaError_t NAME##_launch(const ReplayParams& p, int NT, cudaStream_t st) {             \
    switch (NT) {                                                                           \
      case 1: return replay_launch_wide<ALGO, ST, 1>(p, st);                                \
      case 2: return replay_launch_one<ALGO, ST, 2, false>(p, st);                          \
      case 4: return replay_launch_wide<ALGO, ST, 4>(p, st);                                \
      case 8: return replay_launch_wide<ALGO, ST, 8>(p, st);                                \
      case 16: return replay_launch_one<ALGO, ST, 16, false>(p, st);                        \
      default: return cudaErrorInvalidValue;                                                \
    }                                                                                       \
  }                                                                                         \
  cudaError_t NAME##_prepare(int max_smem) {                                                \
    cudaError_t e;                                                                          \
    if ((e = replay_prepare_wide<ALGO, ST, 1>(max_smem)) != cudaSuccess) return e;          \
    if ((e = replay_prepare_one<ALGO, ST, 2, false>(max_smem)) != cudaSuccess) return e;    \
    if ((e = replay_prepare_wide<ALGO, ST, 4>(max_smem)) != cudaSuccess) return e;          \
    if ((e = replay_prepare_wide<ALGO, ST, 8>(max_smem)) != cudaSuccess) return e;          \
    return replay_prepare_one<ALGO, ST, 16, false>(max_smem);                               \
  }                                                                                         \
  }

// Ragged windows (cu_seqlens): the verify widths 2..16; a ragged launch of
// windows of at most one token takes width 2.
#define RSSM_DEFINE_REPLAY_RAGGED(NAME, ALGO, ST)                                           \
  namespace rssm {                                                                          \
  cudaError_t NAME##_launch(const ReplayParams& p, int NT, cudaStream_t st) {             \
    switch (NT) {                                                                           \
      case 2: return replay_launch_one<ALGO, ST, 2, true>(p, st);                           \
      case 4: return replay_launch_one<ALGO, ST, 4, true>(p, st);                           \
      case 8: return replay_launch_one<ALGO, ST, 8, true>(p, st);                           \
      case 16: return replay_launch_one<ALGO, ST, 16, true>(p, st);                         \
      default: return cudaErrorInvalidValue;                                                \
    }                                                                                       \
  }                                                                                         \
  cudaError_t NAME##_prepare(int max_smem) {                                                \
    cudaError_t e;                                                                          \
    if ((e = replay_prepare_one<ALGO, ST, 2, true>(max_smem)) != cudaSuccess) return e;     \
    if ((e = replay_prepare_one<ALGO, ST, 4, true>(max_smem)) != cudaSuccess) return e;     \
    if ((e = replay_prepare_one<ALGO, ST, 8, true>(max_smem)) != cudaSuccess) return e;     \
    return replay_prepare_one<ALGO, ST, 16, true>(max_smem);                                \
  }                                                                                         \
  }
