// Native fused-recurrent decode kernels (comparison point of the replay path).
#include "native_impl.cuh"
#include "rssm_launch.h"

namespace rssm {

namespace {

template <int ALGO, typename ST>
cudaError_t launch_one(const ReplayParams& p, const NativeSmem& sm, cudaStream_t st) {
  const dim3 grid((unsigned)p.HV, (unsigned)p.B, 1);
  native_decode_kernel<ALGO, ST><<<grid, kThreads, sm.total, st>>>(p, sm);
  return cudaGetLastError();
}

template <int ALGO, typename ST>
cudaError_t prepare_one(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(native_decode_kernel<ALGO, ST>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(native_decode_kernel<ALGO, ST>,
                              cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

}  // namespace

cudaError_t native_launch(int algo, int state_dt, const ReplayParams& p, const NativeSmem& sm,
                          cudaStream_t st) {
  if (algo == ALGO_GDN) {
    return state_dt == DT_F32 ? launch_one<ALGO_GDN, float>(p, sm, st)
                              : launch_one<ALGO_GDN, __nv_bfloat16>(p, sm, st);
  }
  return state_dt == DT_F32 ? launch_one<ALGO_KDA, float>(p, sm, st)
                            : launch_one<ALGO_KDA, __nv_bfloat16>(p, sm, st);
}

cudaError_t native_prepare(int algo, int state_dt, int max_smem) {
  if (algo == ALGO_GDN) {
    return state_dt == DT_F32 ? prepare_one<ALGO_GDN, float>(max_smem)
                              : prepare_one<ALGO_GDN, __nv_bfloat16>(max_smem);
  }
  return state_dt == DT_F32 ? prepare_one<ALGO_KDA, float>(max_smem)
                            : prepare_one<ALGO_KDA, __nv_bfloat16>(max_smem);
}

}  // namespace rssm
