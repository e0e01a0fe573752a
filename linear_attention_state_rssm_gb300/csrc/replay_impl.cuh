// Replay kernel: decode (T = 1) and speculative verify (T <= 16) of one layer,
// with the ring-overflow fold fused in.
//
// One CTA of 4 warps per (request row, value head). The (slot, head)
// checkpoint tile S0 [dk][dv] streams through a ring of four shared-memory
// stages (8 KB row chunks, one bulk async copy each, full/empty mbarriers); a
// lane owns CW consecutive value columns of some rows of every chunk, so one
// vector load feeds CW x 2T fused multiply-adds. The stream is the only
// O(dk dv) work, and the kernel keeps the instructions spent around it small.
//
// Ring keys are stored per value head, so every CTA reads and writes only its
// own records: a folding window (which writes positions [0, T) of the history
// it reads) waits for nothing but its own history copy. (LightLLM PR #1690
// "feat: add ReplaySSM state modes for GDN and KDA" shares one key buffer
// across the value heads of a key group and needs a counted cross-CTA barrier
// for that reason; its author notes the barrier has no progress guarantee.)
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
//  5. per value column: a_i, b_i = y + sum_m H d_m; the triangular solve
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

// Dot products of key-channel vectors: lanes take float4 groups of channels,
// then a warp reduction.
__device__ __forceinline__ float4 ld4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

// Narrow windows keep four CTAs per SM (at most 128 registers per thread);
// wide verify windows trade occupancy for their larger accumulator tiles.
template <int ALGO, typename ST, int NT>
__global__ void __launch_bounds__(kThreads, NT <= 4 ? 4 : 2) replay_kernel(const ReplayParams p) {
  constexpr int NV = 2 * NT;             // mat-vec vectors: k_i at [0, NT), q_i at [NT, 2NT)
  constexpr int CW = quad_width(NT);     // value columns per lane in the tile stream
  extern __shared__ __align__(128) unsigned char smem[];

  const int h = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = p.T, dk = p.dk, dv = p.dv, L = p.L, HV = p.HV, HK = p.HK;
  const int kh = h / p.G;

  // ---- row resolve
  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (h == 0 && tid == 0) atomicOr(p.err, DEVERR_SLOT);
    return;
  }

  ST* gtile = static_cast<ST*>(p.state) + ((size_t)s * HV + h) * dk * dv;
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

  // ---- 1. bulk async copies. One thread issues every copy of a barrier after
  //         registering its byte count.
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
  // fold decision (uniform over the CTA)
  const bool fold = (p.force != nullptr && p.force[r] != 0) || (c + T > L);
  const int base = fold ? 0 : c;
  const int nh = c;
  const size_t kbase = ((size_t)s * HV + h) * L * dk;
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
  // A folding window writes over positions [0, T) of the history it reads:
  // its history copy must have landed before the records below.
  if (fold && nh > 0) copies_ok = mbar_wait_bounded(&mbar[kMbarHist], 0) && copies_ok;
  __syncthreads();

  // ---- records that need no result of the window: keys, gates and betas at
  //      ring positions base + i. Each thread writes the key channels it owns
  //      in step 2 below.
  for (int ch = tid; ch < dk; ch += kThreads) {
    for (int i = 0; i < T; ++i) {
      st_f32(p.ring_k, kbase + (size_t)(base + i) * dk + ch, p.rk_dt, wk[i * dk + ch]);
      if (ALGO == ALGO_KDA) p.ring_g[gbase + (size_t)(base + i) * dk + ch] = wg[i * dk + ch];
    }
  }
  if (tid < T) {
    p.ring_beta[((size_t)s * HV + h) * L + base + tid] = wb[tid];
    if (ALGO == ALGO_GDN) p.ring_g[gbase + base + tid] = wg[tid];
  }

  const QuadLayout qlay(dv, CW);
  const QuadLane qlane(qlay, CW, warp, lane);
  float acc[NV][CW];
#pragma unroll
  for (int vv = 0; vv < NV; ++vv) {
#pragma unroll
    for (int cc = 0; cc < CW; ++cc) acc[vv][cc] = 0.f;
  }
  // GDN mat-vec inputs are the raw window vectors (their scalar decay goes on
  // the column results); without a fold the tile streams now.
  const bool early = ALGO == ALGO_GDN && !fold;
  if (ALGO == ALGO_GDN) {
    for (int e = tid; e < dk * NV; e += kThreads) {
      const int ch = e / NV, vv = e - ch * NV;
      const int i = vv < NT ? vv : vv - NT;
      xh[e] = i < T ? (vv < NT ? wk[i * dk + ch] : wq[i * dk + ch]) : 0.f;
    }
    if (early) {
      __syncthreads();
      copies_ok = stream_quads<ALGO, ST, NV, CW, false>(pipe, qlane, acc, gtile, dk, dv, 0, hk,
                                                        hd, hf, 1.f, egam, xh, tid, lane) &&
                  copies_ok;
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
        for (int c4 = 4 * lane; c4 < dk; c4 += 128) {
          float4 kj = ld4(wk + j * dk + c4);
          if (ALGO == ALGO_KDA) {
            const float4 gi = ld4(wg + i * dk + c4), gj = ld4(wg + j * dk + c4);
            kj.x *= __expf(gi.x - gj.x);
            kj.y *= __expf(gi.y - gj.y);
            kj.z *= __expf(gi.z - gj.z);
            kj.w *= __expf(gi.w - gj.w);
          }
          const float4 ki = ld4(wk + i * dk + c4), qi = ld4(wq + i * dk + c4);
          skk = fmaf(kj.x, ki.x, fmaf(kj.y, ki.y, fmaf(kj.z, ki.z, fmaf(kj.w, ki.w, skk))));
          skq = fmaf(kj.x, qi.x, fmaf(kj.y, qi.y, fmaf(kj.z, qi.z, fmaf(kj.w, qi.w, skq))));
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
      for (int c4 = 4 * lane; c4 < dk; c4 += 128) {
        const float4 km = ld4(hk + m * dk + c4);
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) {
          const int i = vv < NT ? vv : vv - NT;
          if (i < T) {
            const float4 x = ld4((vv < NT ? xk : xq) + i * dk + c4);
            part[vv] = fmaf(km.x, x.x, fmaf(km.y, x.y, fmaf(km.z, x.z, fmaf(km.w, x.w, part[vv]))));
          }
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

  // ---- 4. stream the checkpoint tile (unless done early): fold, then S^T x
  if (!early) {
    __syncthreads();
    bool ok;
    if (fold && nh > 0) {
      ok = stream_quads<ALGO, ST, NV, CW, true>(pipe, qlane, acc, gtile, dk, dv, nh, hk, hd, hf,
                                                hscal[1], egam, xh, tid, lane);
    } else {
      ok = stream_quads<ALGO, ST, NV, CW, false>(pipe, qlane, acc, gtile, dk, dv, 0, hk, hd, hf,
                                                 1.f, egam, xh, tid, lane);
    }
    if (!ok) {
      atomicOr(p.err, DEVERR_TIMEOUT);
      copies_ok = false;
    }
  }
  // partial column sums of the warp row groups -> shared memory (the ring is
  // free once every warp has consumed the last chunk)
  __syncthreads();
  if (qlane.first) {
#pragma unroll
    for (int vv = 0; vv < NV; ++vv) {
#pragma unroll
      for (int cc = 0; cc < CW; ++cc) red[(qlane.rg * NV + vv) * dv + qlane.col0 + cc] = acc[vv][cc];
    }
  }
  __syncthreads();

  // ---- 5. per value column: corrections, triangular solve, outputs, deltas
  if (tid < dv) {
    const int col = tid;
    float y[NV];
#pragma unroll
    for (int vv = 0; vv < NV; ++vv) {
      float sum = 0.f;
      for (int g2 = 0; g2 < qlay.rgw; ++g2) sum += red[(g2 * NV + vv) * dv + col];
      y[vv] = sum;
    }
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
        float a = wb[i] * (wv[i * dv + col] - y[i]);
#pragma unroll
        for (int j = 0; j < i; ++j) a = fmaf(-am[i * NT + j], d[j], a);
        d[i] = a;
        float o = y[NT + i];
#pragma unroll
        for (int j = 0; j <= i; ++j) o = fmaf(fm[i * NT + j], d[j], o);
        o *= p.scale;
        const size_t tok = tok0 + i;
        st_f32(p.o, (tok * HV + h) * dv + col, p.in_dt, o);
        const size_t rec = dbase + (size_t)(base + i) * dv + col;
        st_f32(p.ring_d, rec, p.rd_dt, a);
        st_f32(p.ring_v, rec, p.in_dt, wv[i * dv + col]);
      }
    }
  }
  if (h == 0 && tid == 0 && p.fold_out != nullptr) p.fold_out[r] = fold ? 1 : 0;
  if (!copies_ok) {
    // give copies that did not arrive a second bounded chance before exit
    mbar_wait_bounded(&mbar[kMbarWin], 0);
    if (nh > 0) mbar_wait_bounded(&mbar[kMbarHist], 0);
    pipe.drain();
  }
}

}  // namespace rssm
