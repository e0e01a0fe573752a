// Pipelined replay kernel (pipe_impl.cuh), GDN heads of 128 x 128: fp32 and
// bf16 checkpoints, windows of 1, 2, 4 and 8 tokens (a window of T tokens runs
// in the smallest width >= T).
#include "pipe_impl.cuh"
#include "rssm_launch.h"

namespace rssm {
namespace {

template <typename ST, int NT>
cudaError_t launch_one(const ReplayParams& p, const PipeSmem& sm, int grid, cudaStream_t st) {
  pipe_kernel<ALGO_GDN, ST, NT><<<grid, kPipeThreads, sm.total, st>>>(p, sm);
  return cudaGetLastError();
}

template <typename ST, int NT>
cudaError_t prepare_one(int max_smem) {
  return cudaFuncSetAttribute(pipe_kernel<ALGO_GDN, ST, NT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

template <typename ST>
cudaError_t launch_t(int NT, const ReplayParams& p, const PipeSmem& sm, int grid,
                     cudaStream_t st) {
  switch (NT) {
    case 1: return launch_one<ST, 1>(p, sm, grid, st);
    case 2: return launch_one<ST, 2>(p, sm, grid, st);
    case 4: return launch_one<ST, 4>(p, sm, grid, st);
    case 8: return launch_one<ST, 8>(p, sm, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

template <typename ST>
cudaError_t prepare_t(int max_smem) {
  cudaError_t e;
  if ((e = prepare_one<ST, 1>(max_smem)) != cudaSuccess) return e;
  if ((e = prepare_one<ST, 2>(max_smem)) != cudaSuccess) return e;
  if ((e = prepare_one<ST, 4>(max_smem)) != cudaSuccess) return e;
  return prepare_one<ST, 8>(max_smem);
}

}  // namespace

cudaError_t pipe_launch(int state_dt, int NT, const ReplayParams& p, const PipeSmem& sm, int grid,
                        cudaStream_t st) {
  return state_dt == DT_F32 ? launch_t<float>(NT, p, sm, grid, st)
                            : launch_t<__nv_bfloat16>(NT, p, sm, grid, st);
}

cudaError_t pipe_prepare(int state_dt, int max_smem) {
  return state_dt == DT_F32 ? prepare_t<float>(max_smem) : prepare_t<__nv_bfloat16>(max_smem);
}

}  // namespace rssm
