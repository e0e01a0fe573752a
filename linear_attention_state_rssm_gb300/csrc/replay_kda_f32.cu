// Replay kernel, KDA with a f32 checkpoint.
#include "replay_launch.cuh"

RSSM_DEFINE_REPLAY(replay_kda_f32, rssm::ALGO_KDA, float)
