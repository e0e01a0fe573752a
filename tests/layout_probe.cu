// Host program for tests/test_layout.py (test infrastructure): prints the
// replay kernel's shared-memory plan, one JSON line per configuration given on
// the command line as groups of eleven integers
//   algo state_bytes NT T L dk dv in_dtype ring_k_dtype ring_d_dtype tc
// It runs no device code.
#include <cstdio>
#include <cstdlib>

#include "rssm_common.cuh"

using namespace rssm;

int main(int argc, char** argv) {
  for (int i = 1; i + 10 < argc; i += 11) {
    int v[11];
    for (int j = 0; j < 11; ++j) v[j] = std::atoi(argv[i + j]);
    const ReplaySmem m =
        replay_layout(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], v[8], v[9], v[10] != 0);
    std::printf(
        "{\"ring\": %u, \"mbar\": %u, \"wq\": %u, \"wk\": %u, \"wv\": %u, \"wraw\": %u, "
        "\"wb\": %u, \"wg\": %u, \"yk\": %u, \"yq\": %u, \"scal\": %u, \"xh\": %u, \"xl\": %u, "
        "\"am\": %u, \"fm\": %u, \"hk\": %u, \"kl\": %u, \"hkraw\": %u, \"hd\": %u, "
        "\"hdraw\": %u, \"hg\": %u, \"hf\": %u, \"hdot\": %u, \"red\": %u, \"rank\": %u, "
        "\"kip\": %u, \"ns\": %u, \"total\": %u, \"ctas\": %u, \"rank_bytes\": %u}\n",
        m.ring, m.mbar, m.wq, m.wk, m.wv, m.wraw, m.wb, m.wg, m.yk, m.yq, m.scal, m.xh, m.xl,
        m.am, m.fm, m.hk, m.kl, m.hkraw, m.hd, m.hdraw, m.hg, m.hf, m.hdot, m.red, m.rank,
        m.kip, m.ns, m.total, ctas_per_sm(m.total), kRankBytes);
  }
  return 0;
}
