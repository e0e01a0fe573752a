// Replay kernel for ragged windows, GDN with a f32 checkpoint.
#include "replay_launch.cuh"

RSSM_DEFINE_REPLAY_RAGGED(replay_gdn_f32_ragged, rssm::ALGO_GDN, float)
