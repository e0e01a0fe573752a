// Instantiation and launch of the replay kernel for one (algorithm, state
// dtype) pair; included by one small translation unit per pair so the build
// compiles them in parallel.
#pragma once

#include "replay_impl.cuh"
#include "rssm_launch.h"

namespace rssm {

// One CTA per (value head, request row).
template <int ALGO, typename ST, int NT, bool RAGGED, bool LONG = false, bool TC = false>
static cudaError_t replay_launch_one(const ReplayParams& p, cudaStream_t st) {
  const dim3 grid((unsigned)p.HV, (unsigned)p.B, 1);
  replay_kernel<ALGO, ST, NT, RAGGED, LONG, TC><<<grid, kThreads, p.sm.total, st>>>(p);
  return cudaGetLastError();
}

template <int ALGO, typename ST, int NT, bool RAGGED, bool LONG = false, bool TC = false>
static cudaError_t replay_prepare_one(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(replay_kernel<ALGO, ST, NT, RAGGED, LONG, TC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(replay_kernel<ALGO, ST, NT, RAGGED, LONG, TC>,
                              cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

// Verify windows of four and eight tokens: GDN takes the tensor-core stream
// kernel when p.tc is set.
template <int ALGO, typename ST, int NT>
static cudaError_t replay_launch_wide(const ReplayParams& p, cudaStream_t st) {
  if constexpr (ALGO == ALGO_GDN) {
    if (p.tc) return replay_launch_one<ALGO, ST, NT, false, false, true>(p, st);
  }
  return replay_launch_one<ALGO, ST, NT, false>(p, st);
}

template <int ALGO, typename ST, int NT>
static cudaError_t replay_prepare_wide(int max_smem) {
  if constexpr (ALGO == ALGO_GDN) {
    const cudaError_t e = replay_prepare_one<ALGO, ST, NT, false, false, true>(max_smem);
    if (e != cudaSuccess) return e;
  }
  return replay_prepare_one<ALGO, ST, NT, false>(max_smem);
}

// Decode: GDN rings longer than 16 records take the kernel without the
// tensor-core fold (their folds carry more than 16 records).
template <int ALGO, typename ST>
static cudaError_t replay_launch_decode(const ReplayParams& p, cudaStream_t st) {
  if constexpr (ALGO == ALGO_GDN) {
    if (p.L > 16) return replay_launch_one<ALGO, ST, 1, false, true>(p, st);
  }
  return replay_launch_one<ALGO, ST, 1, false>(p, st);
}

template <int ALGO, typename ST>
static cudaError_t replay_prepare_decode(int max_smem) {
  if constexpr (ALGO == ALGO_GDN) {
    const cudaError_t e = replay_prepare_one<ALGO, ST, 1, false, true>(max_smem);
    if (e != cudaSuccess) return e;
  }
  return replay_prepare_one<ALGO, ST, 1, false>(max_smem);
}

}  // namespace rssm

#define RSSM_DEFINE_REPLAY(NAME, ALGO, ST)                                                  \
  namespace rssm {                                                                          \
  cudaError_t NAME##_launch(const ReplayParams& p, int NT, cudaStream_t st) {             \
    switch (NT) {                                                                           \
      case 1: return replay_launch_decode<ALGO, ST>(p, st);                                 \
      case 2: return replay_launch_one<ALGO, ST, 2, false>(p, st);                          \
      case 4: return replay_launch_wide<ALGO, ST, 4>(p, st);                                \
      case 8: return replay_launch_wide<ALGO, ST, 8>(p, st);                                \
      case 16: return replay_launch_one<ALGO, ST, 16, false>(p, st);                        \
      default: return cudaErrorInvalidValue;                                                \
    }                                                                                       \
  }                                                                                         \
  cudaError_t NAME##_prepare(int max_smem) {                                                \
    cudaError_t e;                                                                          \
    if ((e = replay_prepare_decode<ALGO, ST>(max_smem)) != cudaSuccess) return e;           \
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
