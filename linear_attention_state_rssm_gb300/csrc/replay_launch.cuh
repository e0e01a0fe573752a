// Instantiation and launch of the replay kernel for one (algorithm, state
// dtype) pair; included by one small translation unit per pair so the build
// compiles them in parallel.
#pragma once

#include "replay_impl.cuh"
#include "rssm_launch.h"

namespace rssm {

// One CTA per (value head, request row).
template <int ALGO, typename ST, int NT>
static cudaError_t replay_launch_one(const ReplayParams& p, cudaStream_t st) {
  const dim3 grid((unsigned)p.HV, (unsigned)p.B, 1);
  replay_kernel<ALGO, ST, NT><<<grid, kThreads, p.sm.total, st>>>(p);
  return cudaGetLastError();
}

template <int ALGO, typename ST, int NT>
static cudaError_t replay_prepare_one(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(replay_kernel<ALGO, ST, NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(replay_kernel<ALGO, ST, NT>,
                              cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

}  // namespace rssm

#define RSSM_DEFINE_REPLAY(NAME, ALGO, ST)                                                  \
  namespace rssm {                                                                          \
  cudaError_t NAME##_launch(const ReplayParams& p, int NT, cudaStream_t st) {             \
    switch (NT) {                                                                           \
      case 1: return replay_launch_one<ALGO, ST, 1>(p, st);                                 \
      case 2: return replay_launch_one<ALGO, ST, 2>(p, st);                                 \
      case 4: return replay_launch_one<ALGO, ST, 4>(p, st);                                 \
      case 8: return replay_launch_one<ALGO, ST, 8>(p, st);                                 \
      case 16: return replay_launch_one<ALGO, ST, 16>(p, st);                               \
      default: return cudaErrorInvalidValue;                                                \
    }                                                                                       \
  }                                                                                         \
  cudaError_t NAME##_prepare(int max_smem) {                                                \
    cudaError_t e;                                                                          \
    if ((e = replay_prepare_one<ALGO, ST, 1>(max_smem)) != cudaSuccess) return e;           \
    if ((e = replay_prepare_one<ALGO, ST, 2>(max_smem)) != cudaSuccess) return e;           \
    if ((e = replay_prepare_one<ALGO, ST, 4>(max_smem)) != cudaSuccess) return e;           \
    if ((e = replay_prepare_one<ALGO, ST, 8>(max_smem)) != cudaSuccess) return e;           \
    return replay_prepare_one<ALGO, ST, 16>(max_smem);                                      \
  }                                                                                         \
  }
