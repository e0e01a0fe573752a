// Replay kernel for ragged windows, KDA with a f32 checkpoint.
#include "replay_launch.cuh"

RSSM_DEFINE_REPLAY_RAGGED(replay_kda_f32_ragged, rssm::ALGO_KDA, float)
