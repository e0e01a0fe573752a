// Replay kernel for ragged windows, GDN with a bf16 checkpoint.
#include "replay_launch.cuh"

RSSM_DEFINE_REPLAY_RAGGED(replay_gdn_bf16_ragged, rssm::ALGO_GDN, __nv_bfloat16)
