// Replay kernel, GDN with a f32 checkpoint.
#include "replay_launch.cuh"

RSSM_DEFINE_REPLAY(replay_gdn_f32, rssm::ALGO_GDN, float)
