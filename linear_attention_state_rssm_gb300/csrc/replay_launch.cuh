// Instantiation and launch of the replay kernel for one (algorithm, state
// dtype) pair; included by one small translation unit per pair so the build
// compiles them in parallel.
#pragma once

#include "replay_impl.cuh"
#include "rssm_launch.h"

namespace rssm {

template <int ALGO, typename ST, int NT>
static cudaError_t replay_launch_one(const ReplayParams& p, int cluster, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.HV, (unsigned)p.B, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.sm.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (cluster > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  }
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, replay_kernel<ALGO, ST, NT>, p);
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
  cudaError_t NAME##_launch(const ReplayParams& p, int NT, int cluster, cudaStream_t st) {  \
    switch (NT) {                                                                           \
      case 1: return replay_launch_one<ALGO, ST, 1>(p, cluster, st);                        \
      case 2: return replay_launch_one<ALGO, ST, 2>(p, cluster, st);                        \
      case 4: return replay_launch_one<ALGO, ST, 4>(p, cluster, st);                        \
      case 8: return replay_launch_one<ALGO, ST, 8>(p, cluster, st);                        \
      case 16: return replay_launch_one<ALGO, ST, 16>(p, cluster, st);                      \
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
