// Replay kernel, GDN with a bf16 checkpoint.
#include "replay_launch.cuh"

RSSM_DEFINE_REPLAY(replay_gdn_bf16, rssm::ALGO_GDN, __nv_bfloat16)
