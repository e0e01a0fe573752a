// Host-side entry points of the kernel translation units (internal to librssm).
#pragma once

#include <cuda_runtime.h>

#include "rssm_common.cuh"

namespace rssm {

// Window widths the replay kernel is built for; a window of T tokens runs in
// the smallest width >= T.
inline int nt_for(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16; }
// Ragged windows of at most T tokens (kernels built for the verify widths).
inline int nt_for_ragged(int T) { return T <= 2 ? 2 : nt_for(T); }

#define RSSM_DECLARE_REPLAY(NAME)                                                      \
  cudaError_t NAME##_launch(const ReplayParams& p, int NT, cudaStream_t st); \
  cudaError_t NAME##_prepare(int max_smem);

RSSM_DECLARE_REPLAY(replay_gdn_f32)
RSSM_DECLARE_REPLAY(replay_gdn_bf16)
RSSM_DECLARE_REPLAY(replay_kda_f32)
RSSM_DECLARE_REPLAY(replay_kda_bf16)
RSSM_DECLARE_REPLAY(replay_gdn_f32_ragged)
RSSM_DECLARE_REPLAY(replay_gdn_bf16_ragged)
RSSM_DECLARE_REPLAY(replay_kda_f32_ragged)
RSSM_DECLARE_REPLAY(replay_kda_bf16_ragged)
#undef RSSM_DECLARE_REPLAY

// Pipelined replay kernel (GDN, dk = dv = 128, rings of at most 16 records,
// windows of at most 8 tokens, uniform windows): NT in {1, 2, 4, 8}.
cudaError_t pipe_launch(int state_dt, int NT, const ReplayParams& p, const PipeSmem& sm, int grid,
                        cudaStream_t st);
cudaError_t pipe_prepare(int state_dt, int max_smem);
inline int pipe_nt(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8; }

cudaError_t fold_launch(int algo, int state_dt, const FoldParams& p, int n_layers,
                        cudaStream_t st);
cudaError_t fold_prepare(int algo, int state_dt, int max_smem);
cudaError_t native_launch(int algo, int state_dt, const ReplayParams& p, const NativeSmem& sm,
                          cudaStream_t st);
cudaError_t native_prepare(int algo, int state_dt, int max_smem);
cudaError_t prefill_launch(int algo, int state_dt, const PrefillParams& p, cudaStream_t st);
cudaError_t prefill_prepare(int algo, int state_dt, int max_smem);
cudaError_t conv_launch(const ConvParams& p, bool commit, cudaStream_t st);
cudaError_t cursor_launch(int32_t* cursor, const int32_t* slot, const uint8_t* force,
                          const int32_t* accept, const int32_t* cu, int B, int T, int L,
                          int n_slots, int mode, uint32_t* err, cudaStream_t st);

}  // namespace rssm
