// Replay kernel for ragged windows, KDA with a bf16 checkpoint.
#include "replay_launch.cuh"

RSSM_DEFINE_REPLAY_RAGGED(replay_kda_bf16_ragged, rssm::ALGO_KDA, __nv_bfloat16)
