// Replay kernel: decode (T = 1) and speculative verify (T <= 16) of one layer,
// with the ring-overflow fold fused in.
//
// One CTA of 4 warps per (request row, value head); for GQA the G value heads
// of a key head form a thread-block cluster, whose barrier orders their reads
// of the shared key records before a folding window overwrites them (LightLLM
// PR #1690 "feat: add ReplaySSM state modes for GDN and KDA", commit message on
// waiting until every value tile has read the old prefix before slot 0 is
// rewritten; here the wait is a hardware cluster barrier, which always makes
// progress because cluster CTAs are co-scheduled).
//
// The (slot, head) checkpoint tile S0 [dk][dv] streams through a ring of four
// shared-memory stages (8 KB row chunks, one bulk async copy each, full/empty
// mbarriers); thread tid consumes value column tid % dv of every chunk. The
// small ring lets several CTAs share an SM, each with 32 KB of the tile in
// flight from its first microsecond.
//
// Per CTA, with c = cursor[slot], fold = force || c + T > L:
//  1. bulk async copies: the first tile chunks and the window rows (they need
//     only the slot) and, once the cursor is known, the c history records;
//  2. gates: history decay factors and in-window inclusive prefixes G_i;
//  3. window coefficients for j <= i < T (per key channel for KDA)
//        A_ij = beta_i sum_ch e^{G_i-G_j} k_j k_i   (j < i)
//        F_ij =        sum_ch e^{G_i-G_j} k_j q_i   (j <= i)
//     and, without a fold, history dot coefficients H[m][x] = k~_m . (e^{G_i} x)
//     for every window vector x in {k_i, q_i};
//  4. stream the tile: on a fold S0 <- e^{Gam} S0 + sum_m k~_m d_m^T (stored
//     back), and y_x = S0^T (e^{Gam_e + G_i} x) for all 2T vectors in one pass
//     (a GDN window without a fold streams first, while its history lands);
//  5. per column: a_i, b_i = y + sum_m H d_m; the triangular solve
//     d_i = beta_i (v_i - a_i) - sum_{j<i} A_ij d_j (forward substitution of
//     (I + A) D = R) and o_i = scale (b_i + sum_{j<=i} F_ij d_j); the records of
//     the window go to ring positions base + i (base = fold ? 0 : c).
// Every window sum runs over j <= i only, so a NaN or Inf at a later (rejected)
// position is never read by an earlier output: the causal selection is
// structural, never a multiplication by zero (SGLang fork PR jianc99/sglang#2,
// "Modifications" and the commit on fused selects).
#pragma once

#include "rssm_common.cuh"
#include "rssm_history.cuh"

namespace rssm {

template <int ALGO, typename ST, int NT>
__global__ void __launch_bounds__(kThreads) replay_kernel(const ReplayParams p) {
  constexpr int NV = 2 * NT;             // mat-vec vectors: k_i at [0, NT), q_i at [NT, 2NT)
  extern __shared__ __align__(128) unsigned char smem[];

  const int h = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = p.T, dk = p.dk, dv = p.dv, L = p.L, HV = p.HV, HK = p.HK;
  const int kh = h / p.G;

  // ---- row resolve (uniform over the CTA and its cluster)
  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (h == 0 && tid == 0) atomicOr(p.err, DEVERR_SLOT);
    return;
  }

  const ColMap cm(dk, dv, tid);
  ST* gtile = static_cast<ST*>(p.state) + ((size_t)s * HV + h) * dk * dv;
  ST* gcol = gtile + cm.col;

  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + p.sm.mbar);
  float* wq = reinterpret_cast<float*>(smem + p.sm.wq);
  float* wk = reinterpret_cast<float*>(smem + p.sm.wk);
  float* wv = reinterpret_cast<float*>(smem + p.sm.wv);
  float* wb = reinterpret_cast<float*>(smem + p.sm.wb);
  float* wg = reinterpret_cast<float*>(smem + p.sm.wg);
  float* yk = reinterpret_cast<float*>(smem + p.sm.yk);
  float* yq = reinterpret_cast<float*>(smem + p.sm.yq);
  float* scal = reinterpret_cast<float*>(smem + p.sm.scal);
  float* xh = reinterpret_cast<float*>(smem + p.sm.xh);
  float* am = reinterpret_cast<float*>(smem + p.sm.am);
  float* fm = reinterpret_cast<float*>(smem + p.sm.fm);
  float* hk = reinterpret_cast<float*>(smem + p.sm.hk);
  float* hd = reinterpret_cast<float*>(smem + p.sm.hd);
  float* hg = reinterpret_cast<float*>(smem + p.sm.hg);
  float* hf = reinterpret_cast<float*>(smem + p.sm.hf);
  float* hdot = reinterpret_cast<float*>(smem + p.sm.hdot);
  float* red = reinterpret_cast<float*>(smem + p.sm.red);
  unsigned char* wraw = smem + p.sm.wraw;
  unsigned char* hkraw = smem + p.sm.hkraw;
  unsigned char* hdraw = smem + p.sm.hdraw;
  // GDN scalars: es[i] = e^{Gam_e + G_i}, eG[i] = e^{G_i}, hscal = {Gam, e^Gam}.
  // KDA vectors: egam[ch] = e^{Gam[ch]}, gam[ch] = Gam[ch].
  float* es = scal;
  float* eG = scal + NT;
  float* hscal = scal + 2 * NT;
  float* egam = scal;
  float* gam = scal + dk;

  const size_t tok0 = (size_t)r * T;
  const int s_in = dtype_bytes(p.in_dt);
  const uint32_t qrow = (uint32_t)(dk * s_in), vrow = (uint32_t)(dv * s_in);

  // ---- 1. bulk async copies: window rows now, history once the cursor is
  //         known. One thread issues every copy of a barrier after registering
  //         its byte count.
  const TilePipe<ST> pipe(reinterpret_cast<ST*>(smem + p.sm.ring), mbar, gtile, dk, dv);
  if (tid == 0) {
    mbar_init(&mbar[kMbarWin], 1);
    mbar_init(&mbar[kMbarHist], 1);
    pipe.init();
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    pipe.prime();
    const bool f32in = p.in_dt == DT_F32;
    mbar_expect_tx(&mbar[kMbarWin],
                   T * (2 * qrow + vrow) + (ALGO == ALGO_KDA ? (uint32_t)(T * dk * 4) : 0u));
    for (int i = 0; i < T; ++i) {
      const size_t tok = tok0 + i;
      const size_t qoff = ((tok * HK + kh) * dk) * s_in;
      const size_t voff = ((tok * HV + h) * dv) * s_in;
      bulk_g2s(f32in ? static_cast<void*>(wq + i * dk) : wraw + i * qrow,
               static_cast<const char*>(p.q) + qoff, qrow, &mbar[kMbarWin]);
      bulk_g2s(f32in ? static_cast<void*>(wk + i * dk) : wraw + (T + i) * qrow,
               static_cast<const char*>(p.k) + qoff, qrow, &mbar[kMbarWin]);
      bulk_g2s(f32in ? static_cast<void*>(wv + i * dv) : wraw + 2 * T * qrow + i * vrow,
               static_cast<const char*>(p.v) + voff, vrow, &mbar[kMbarWin]);
      if (ALGO == ALGO_KDA) {
        bulk_g2s(wg + i * dk, p.g + (tok * HV + h) * dk, (uint32_t)(dk * 4), &mbar[kMbarWin]);
      }
    }
  }
  const int c = p.cursor[s];
  if (tid < T) {
    wb[tid] = p.beta[(tok0 + tid) * HV + h];
    if (ALGO == ALGO_GDN) wg[tid] = p.g[(tok0 + tid) * HV + h];
  }
  if (c < 0 || c > L) {
    if (h == 0 && tid == 0) atomicOr(p.err, DEVERR_CURSOR);
    // copies are in flight into this CTA's shared memory: let them land
    mbar_wait_bounded(&mbar[kMbarWin], 0);
    pipe.drain();
    return;
  }
  // fold decision (uniform over the CTA and its cluster)
  const bool fold = (p.force != nullptr && p.force[r] != 0) || (c + T > L);
  const int base = fold ? 0 : c;
  const int nh = c;
  const bool group_sync = fold && p.G > 1;
  const size_t kbase = ((size_t)s * HK + kh) * L * dk;
  const size_t dbase = ((size_t)s * HV + h) * L * dv;
  const size_t gbase = ((size_t)s * HV + h) * L * (ALGO == ALGO_GDN ? 1 : dk);
  if (nh > 0 && tid == 0) {
    issue_history<ALGO>(nh, dk, dv, p.ring_k, kbase, p.rk_dt, p.ring_d, dbase, p.rd_dt, p.ring_g,
                        gbase, hk, hkraw, hd, hdraw, hg, &mbar[kMbarHist]);
  }
  if (ALGO == ALGO_GDN) {
    for (int m = tid; m < nh; m += kThreads) hf[m] = p.ring_g[gbase + m];
  }
  bool copies_ok = mbar_wait_bounded(&mbar[kMbarWin], 0);
  if (p.in_dt != DT_F32) {
    widen16(wq, wraw, T * dk, p.in_dt, tid, kThreads);
    widen16(wk, wraw + T * qrow, T * dk, p.in_dt, tid, kThreads);
    widen16(wv, wraw + 2 * T * qrow, T * dv, p.in_dt, tid, kThreads);
  }
  __syncthreads();

  // ---- records that need no result of the window: keys (once per key head),
  //      gates and betas, at ring positions base + i. Each thread writes the
  //      key channels it owns in step 2 below. A folding window writes over
  //      positions [0, T) of the history it reads: it first waits for its own
  //      history copy, then until the whole key group has read the old keys.
  if (fold && nh > 0) copies_ok = mbar_wait_bounded(&mbar[kMbarHist], 0) && copies_ok;
  if (group_sync) {
    cluster_arrive_release();
    cluster_wait_acquire();
  }
  for (int ch = tid; ch < dk; ch += kThreads) {
    for (int i = 0; i < T; ++i) {
      if (h % p.G == 0) {
        st_f32(p.ring_k, kbase + (size_t)(base + i) * dk + ch, p.rk_dt, wk[i * dk + ch]);
      }
      if (ALGO == ALGO_KDA) p.ring_g[gbase + (size_t)(base + i) * dk + ch] = wg[i * dk + ch];
    }
  }
  if (tid < T) {
    p.ring_beta[((size_t)s * HV + h) * L + base + tid] = wb[tid];
    if (ALGO == ALGO_GDN) p.ring_g[gbase + base + tid] = wg[tid];
  }

  float y[NV];
#pragma unroll
  for (int vv = 0; vv < NV; ++vv) y[vv] = 0.f;
  // GDN mat-vec inputs are the raw window vectors (their scalar decay goes on
  // the column results); without a fold the tile streams now, before the
  // history is needed.
  const bool early = ALGO == ALGO_GDN && !fold;
  if (ALGO == ALGO_GDN) {
    for (int e = tid; e < dk * NV; e += kThreads) {
      const int ch = e / NV, vv = e - ch * NV;
      const int i = vv < NT ? vv : vv - NT;
      xh[e] = i < T ? (vv < NT ? wk[i * dk + ch] : wq[i * dk + ch]) : 0.f;
    }
    if (early) {
      __syncthreads();
      copies_ok = stream_tile<ALGO, ST, NV, false>(pipe, y, gcol, cm, dk, dv, 0, hk, hd, hf, 1.f,
                                                   egam, xh, tid, lane) && copies_ok;
    }
  }
  if (nh > 0 && !fold) copies_ok = mbar_wait_bounded(&mbar[kMbarHist], 0) && copies_ok;
  if (nh > 0) widen_history(nh, dk, dv, p.rk_dt, p.rd_dt, hk, hkraw, hd, hdraw, tid);
  if (!copies_ok) atomicOr(p.err, DEVERR_TIMEOUT);
  __syncthreads();

  // ---- 2. gates
  if (ALGO == ALGO_GDN) {
    if (warp == 0) {
      if (nh > 0) {
        gdn_history_scan(nh, hf, hscal, lane);
      } else if (lane == 0) {
        hscal[0] = 0.f;
        hscal[1] = 1.f;
      }
      __syncwarp();
      // in-window inclusive prefix of the gates (T <= 16 lanes)
      const float gv = lane < T ? wg[lane] : 0.f;
      float incl = gv;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float t = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += t;
      }
      const float gam_e = fold ? 0.f : hscal[0];
      if (lane < T) {
        wg[lane] = incl;
        eG[lane] = __expf(incl);
        es[lane] = __expf(gam_e + incl);
      }
    }
  } else {
    // one thread per key channel: history decay, window prefix, scaled vectors
    for (int ch = tid; ch < dk; ch += kThreads) {
      const float gm = nh > 0 ? kda_history_channel(nh, dk, ch, hk, hg) : 0.f;
      gam[ch] = gm;
      egam[ch] = __expf(gm);
      const float gam_e = fold ? 0.f : gm;
      float G = 0.f;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        float xk = 0.f, xq = 0.f;
        if (i < T) {
          G += wg[i * dk + ch];
          wg[i * dk + ch] = G;
          const float eg = __expf(G);
          yk[i * dk + ch] = eg * wk[i * dk + ch];
          yq[i * dk + ch] = eg * wq[i * dk + ch];
          const float ex = __expf(gam_e + G);
          xk = ex * wk[i * dk + ch];
          xq = ex * wq[i * dk + ch];
        }
        xh[ch * NV + i] = xk;
        xh[ch * NV + NT + i] = xq;
      }
    }
  }
  __syncthreads();

  // ---- 3. window coefficients A, F (j <= i only) and history dot coefficients
  {
    int pi = 0;
    for (int i = 0; i < T; ++i) {
      for (int j = 0; j <= i; ++j, ++pi) {
        if ((pi & (kWarps - 1)) != warp) continue;
        float skk = 0.f, skq = 0.f;
        for (int ch = lane; ch < dk; ch += 32) {
          float kj = wk[j * dk + ch];
          if (ALGO == ALGO_KDA) kj *= __expf(wg[i * dk + ch] - wg[j * dk + ch]);
          skk = fmaf(kj, wk[i * dk + ch], skk);
          skq = fmaf(kj, wq[i * dk + ch], skq);
        }
        skk = warp_sum(skk);
        skq = warp_sum(skq);
        if (lane == 0) {
          const float w = (ALGO == ALGO_GDN) ? __expf(wg[i] - wg[j]) : 1.f;
          fm[i * NT + j] = w * skq;
          am[i * NT + j] = (j < i) ? wb[i] * w * skk : 0.f;
        }
      }
    }
  }
  if (!fold) {
    // GDN: raw keys, coefficient hf[m] * e^{G_i}; KDA: decayed keys and e^{G_i} x
    const float* xk = ALGO == ALGO_GDN ? wk : yk;
    const float* xq = ALGO == ALGO_GDN ? wq : yq;
    for (int m = warp; m < nh; m += kWarps) {
      float part[NV];
#pragma unroll
      for (int vv = 0; vv < NV; ++vv) part[vv] = 0.f;
      for (int ch = lane; ch < dk; ch += 32) {
        const float km = hk[m * dk + ch];
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) {
          const int i = vv < NT ? vv : vv - NT;
          if (i < T) part[vv] = fmaf(km, (vv < NT ? xk : xq)[i * dk + ch], part[vv]);
        }
      }
#pragma unroll
      for (int vv = 0; vv < NV; ++vv) part[vv] = warp_sum(part[vv]);
      if (lane == 0) {
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) {
          const int i = vv < NT ? vv : vv - NT;
          float hv = 0.f;
          if (i < T) hv = (ALGO == ALGO_GDN) ? part[vv] * hf[m] * eG[i] : part[vv];
          hdot[m * NV + vv] = hv;
        }
      }
    }
  }
  __syncthreads();

  // ---- 4. stream the checkpoint tile (unless done early): fold, then S^T x
  if (!early) {
    bool ok;
    if (fold && nh > 0) {
      ok = stream_tile<ALGO, ST, NV, true>(pipe, y, gcol, cm, dk, dv, nh, hk, hd, hf, hscal[1],
                                           egam, xh, tid, lane);
    } else {
      ok = stream_tile<ALGO, ST, NV, false>(pipe, y, gcol, cm, dk, dv, 0, hk, hd, hf, 1.f, egam,
                                            xh, tid, lane);
    }
    if (!ok) {
      atomicOr(p.err, DEVERR_TIMEOUT);
      copies_ok = false;
    }
  }
  if (cm.RG > 1) {
    // dv < kThreads: several row groups share a column; add their sums
#pragma unroll
    for (int vv = 0; vv < NV; ++vv) red[(cm.rg * NV + vv) * dv + cm.col] = y[vv];
    __syncthreads();
    if (cm.rg == 0) {
      for (int g2 = 1; g2 < cm.RG; ++g2) {
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) y[vv] += red[(g2 * NV + vv) * dv + cm.col];
      }
    }
  }

  // ---- 5. per value column: corrections, triangular solve, outputs, deltas
  if (cm.rg == 0) {
    const int col = cm.col;
    if (ALGO == ALGO_GDN) {
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        if (i < T) {
          y[i] *= es[i];
          y[NT + i] *= es[i];
        }
      }
    }
    if (!fold) {
      for (int m = 0; m < nh; ++m) {
        const float dm = hd[m * dv + col];
        const float* hm = hdot + m * NV;
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) y[vv] = fmaf(hm[vv], dm, y[vv]);
      }
    }
    float d[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      d[i] = 0.f;
      if (i < T) {
        float acc = wb[i] * (wv[i * dv + col] - y[i]);
#pragma unroll
        for (int j = 0; j < i; ++j) acc = fmaf(-am[i * NT + j], d[j], acc);
        d[i] = acc;
        float o = y[NT + i];
#pragma unroll
        for (int j = 0; j <= i; ++j) o = fmaf(fm[i * NT + j], d[j], o);
        o *= p.scale;
        const size_t tok = tok0 + i;
        st_f32(p.o, (tok * HV + h) * dv + col, p.in_dt, o);
        const size_t rec = dbase + (size_t)(base + i) * dv + col;
        st_f32(p.ring_d, rec, p.rd_dt, acc);
        st_f32(p.ring_v, rec, p.in_dt, wv[i * dv + col]);
      }
    }
  }
  if (h == 0 && tid == 0 && p.fold_out != nullptr) p.fold_out[r] = fold ? 1 : 0;
  if (!copies_ok) {
    // give copies that did not arrive a second bounded chance before exit
    mbar_wait_bounded(&mbar[kMbarWin], 0);
    if (nh > 0) mbar_wait_bounded(&mbar[kMbarHist], 0);
  }
}

}  // namespace rssm
