// Commit/fold kernel and cursor kernel.
//
// Fold (SGLang fork PR jianc99/sglang#2, fourth commit: a fold-every commit
// makes the checkpoint the committed state after each step; LightLLM PR #1690
// "feat: add ReplaySSM state modes for GDN and KDA": materialising the
// canonical state): S0 <- exp(Gam) S0 + sum_{m<n} k~_m d_m^T over the first n
// ring records, for every layer, one CTA per (layer, row, value head). Only
// loads of ring records are masked to the committed history [0, n), so records
// of rejected drafts are never read (same PR, commit on selects).
//
// Cursor advance (LightLLM PR #1690 commit messages: the cursor moves once per
// step, after the last layer, so every layer reads the same value; SGLang fork
// PR jianc99/sglang#2, first commit: rows whose state slot is null are skipped).
#include "rssm_common.cuh"
#include "rssm_history.cuh"
#include "rssm_launch.h"

namespace rssm {

template <int ALGO, typename ST>
__global__ void __launch_bounds__(kThreads) fold_kernel(const FoldParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int h = blockIdx.x, r = blockIdx.y, layer = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dk = p.dk, dv = p.dv, L = p.L, HV = p.HV;

  const int s = p.slot[r];
  if (s < 0) return;
  const bool reporter = (h == 0 && layer == 0 && tid == 0);
  if (s >= p.n_slots) {
    if (reporter) atomicOr(p.err, DEVERR_SLOT);
    return;
  }
  const int c = p.cursor[s];
  if (c < 0 || c > L) {
    if (reporter) atomicOr(p.err, DEVERR_CURSOR);
    return;
  }
  int n = c;
  if (p.mode == FOLD_COMMIT) {
    size_t tok0;
    int T;
    if (!row_window(p.cu, r, p.T, tok0, T)) {
      if (reporter) atomicOr(p.err, DEVERR_SEQLEN);
      return;
    }
    if (T == 0) return;  // an idle row keeps its checkpoint
    const int a = p.accept[r];
    if (a < 0 || a > T) {
      if (reporter) atomicOr(p.err, DEVERR_ACCEPT);
      return;
    }
    const bool fold = (p.force != nullptr && p.force[r] != 0) || (c + T > L);
    n = (fold ? 0 : c) + a;
  }
  if (n == 0) return;

  const ColMap cm(dk, dv, tid);
  ST* gtile = static_cast<ST*>(p.state) + layer * p.layer_state +
              ((size_t)s * HV + h) * (size_t)dk * dv;
  ST* gcol = gtile + cm.col;

  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + p.sm.mbar);
  float* hk = reinterpret_cast<float*>(smem + p.sm.hk);
  float* hd = reinterpret_cast<float*>(smem + p.sm.hd);
  float* hg = reinterpret_cast<float*>(smem + p.sm.hg);
  float* hf = reinterpret_cast<float*>(smem + p.sm.hf);
  float* scal = reinterpret_cast<float*>(smem + p.sm.scal);
  unsigned char* hkraw = smem + p.sm.hkraw;
  unsigned char* hdraw = smem + p.sm.hdraw;
  // GDN: scal[0] = Gam, scal[1] = exp(Gam). KDA: egam[dk] = exp(Gam[ch]).
  float* egam = scal;

  const size_t kbase = layer * p.layer_k + ((size_t)s * HV + h) * L * dk;
  const size_t dbase = layer * p.layer_d + ((size_t)s * HV + h) * L * dv;
  const size_t gbase = layer * p.layer_g + ((size_t)s * HV + h) * L * (ALGO == ALGO_GDN ? 1 : dk);

  const TilePipe<ST> pipe(reinterpret_cast<ST*>(smem + p.sm.ring), mbar, gtile, dk, dv, kStages,
                          p.hook);
  constexpr unsigned long long lim = kWaitLimitNs;
  if (tid == 0) {
    mbar_init(&mbar[kMbarWin], 1);
    mbar_init(&mbar[kMbarHist], 1);
    pipe.init();
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    pipe.prime();
    issue_history<ALGO>(n, dk, dv, p.ring_k, kbase, p.rk_dt,
                        p.rk_dt == DT_F32 ? static_cast<void*>(hk) : hkraw, p.ring_d, dbase,
                        p.rd_dt, p.rd_dt == DT_F32 ? static_cast<void*>(hd) : hdraw, p.ring_g,
                        gbase, hg, &mbar[kMbarHist], p.hook.extra(WH_HIST));
  }
  if (ALGO == ALGO_GDN) {
    for (int m = tid; m < n; m += kThreads) hf[m] = p.ring_g[gbase + m];
  }
  // the history copy did not arrive in time: the checkpoint is left as it is
  if (!__syncthreads_and(mbar_wait_bounded(&mbar[kMbarHist], 0, lim))) {
    if (tid == 0) {
      atomicOr(p.err, DEVERR_TIMEOUT);
      mbar_wait_bounded(&mbar[kMbarHist], 0, lim);
      pipe.drain();
    }
    return;
  }
  widen_history(n, dk, dv, p.rk_dt, p.rd_dt, hk, hkraw, hd, hdraw, tid);
  __syncthreads();
  if (ALGO == ALGO_GDN) {
    if (warp == 0) gdn_history_scan(n, hf, scal, lane);
  } else {
    for (int ch = tid; ch < dk; ch += kThreads) {
      egam[ch] = __expf(kda_history_channel(n, dk, ch, hk, hg));
    }
  }
  __syncthreads();
  // a chunk that did not arrive in time: no chunk from there on is stored (the
  // ones before it hold the folded state), and the copies issued are waited for
  float unused[1] = {0.f};
  const bool ok = stream_tile<ALGO, ST, 0, true>(pipe, unused, gcol, cm, dk, dv, n, hk, hd, hf,
                                                 scal[1], egam, nullptr, tid, lane);
  if (!__syncthreads_and(ok) && tid == 0) {
    atomicOr(p.err, DEVERR_TIMEOUT);
    pipe.drain_tail();
  }
}

__global__ void cursor_kernel(int32_t* cursor, const int32_t* slot, const uint8_t* force,
                              const int32_t* accept, const int32_t* cu, int B, int maxT, int L,
                              int n_slots, int mode, uint32_t* err) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= B) return;
  const int s = slot[r];
  if (s < 0) return;
  if (s >= n_slots) {
    atomicOr(err, DEVERR_SLOT);
    return;
  }
  const int c = cursor[s];
  if (mode == CURSOR_ZERO) {
    cursor[s] = 0;
    return;
  }
  if (mode == CURSOR_PREFILL) {
    const int a0 = cu[r], a1 = cu[r + 1];
    if (a0 < 0 || a1 < a0) {
      atomicOr(err, DEVERR_SEQLEN);
      return;
    }
    if (a1 > a0 && c >= 0 && c <= L) cursor[s] = 0;
    return;
  }
  if (c < 0 || c > L) {
    atomicOr(err, DEVERR_CURSOR);
    return;
  }
  const bool f = force != nullptr && force[r] != 0;
  if (mode == CURSOR_DECODE) {
    const bool fold = f || (c + 1 > L);
    cursor[s] = (fold ? 0 : c) + 1;
    return;
  }
  size_t tok0;
  int T;
  if (!row_window(cu, r, maxT, tok0, T)) {
    atomicOr(err, DEVERR_SEQLEN);
    return;
  }
  if (T == 0) return;  // an idle row keeps its cursor
  const int a = accept[r];
  if (a < 0 || a > T) {
    atomicOr(err, DEVERR_ACCEPT);
    return;
  }
  if (mode == CURSOR_COMMIT_FOLD) {
    cursor[s] = 0;
    return;
  }
  const bool fold = f || (c + T > L);
  cursor[s] = (fold ? 0 : c) + a;
}

template <int ALGO, typename ST>
static cudaError_t fold_launch_t(const FoldParams& p, int n_layers, cudaStream_t st) {
  dim3 grid((unsigned)p.HV, (unsigned)p.B, (unsigned)n_layers);
  fold_kernel<ALGO, ST><<<grid, kThreads, p.sm.total, st>>>(p);
  return cudaGetLastError();
}

template <int ALGO, typename ST>
static cudaError_t fold_prepare_t(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(fold_kernel<ALGO, ST>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fold_kernel<ALGO, ST>,
                              cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

cudaError_t fold_launch(int algo, int state_dt, const FoldParams& p, int n_layers,
                        cudaStream_t st) {
  if (algo == ALGO_GDN) {
    return state_dt == DT_F32 ? fold_launch_t<ALGO_GDN, float>(p, n_layers, st)
                              : fold_launch_t<ALGO_GDN, __nv_bfloat16>(p, n_layers, st);
  }
  return state_dt == DT_F32 ? fold_launch_t<ALGO_KDA, float>(p, n_layers, st)
                            : fold_launch_t<ALGO_KDA, __nv_bfloat16>(p, n_layers, st);
}

cudaError_t fold_prepare(int algo, int state_dt, int max_smem) {
  if (algo == ALGO_GDN) {
    return state_dt == DT_F32 ? fold_prepare_t<ALGO_GDN, float>(max_smem)
                              : fold_prepare_t<ALGO_GDN, __nv_bfloat16>(max_smem);
  }
  return state_dt == DT_F32 ? fold_prepare_t<ALGO_KDA, float>(max_smem)
                            : fold_prepare_t<ALGO_KDA, __nv_bfloat16>(max_smem);
}

cudaError_t cursor_launch(int32_t* cursor, const int32_t* slot, const uint8_t* force,
                          const int32_t* accept, const int32_t* cu, int B, int T, int L,
                          int n_slots, int mode, uint32_t* err, cudaStream_t st) {
  const int threads = 128;
  const int blocks = (B + threads - 1) / threads;
  cursor_kernel<<<blocks, threads, 0, st>>>(cursor, slot, force, accept, cu, B, T, L, n_slots,
                                            mode, err);
  return cudaGetLastError();
}

}  // namespace rssm
