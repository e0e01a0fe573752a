// Replay kernel, KDA with a bf16 checkpoint.
#include "replay_launch.cuh"

RSSM_DEFINE_REPLAY(replay_kda_bf16, rssm::ALGO_KDA, __nv_bfloat16)
