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
// Per CTA, with c = cursor[slot], fold = force || c + T > L:
//  1. the checkpoint tile S0 [dk][dv] streams into shared memory by bulk async
//     copies (one row chunk per warp), overlapped with loading the window and
//     the c history records;
//  2. history gates become decay-scaled keys k~_m (rssm_history.cuh);
//  3. window coefficients, for j <= i < T, G_i the inclusive in-window gate
//     prefix (per channel for KDA):
//        A_ij = beta_i sum_ch e^{G_i-G_j} k_j k_i   (j < i)
//        F_ij =        sum_ch e^{G_i-G_j} k_j q_i   (j <= i)
//  4. fold: S0 <- exp(Gam) S0 + sum_m k~_m d_m^T, written back, history emptied;
//     no fold: history dot coefficients H[m][x] = k~_m . (e^{G_i} x) for every
//     window vector x in {k_i, q_i};
//  5. one pass over the tile computes S0^T (e^{Gam_e + G_i} x) for all 2T
//     vectors at once (the only O(dk dv) work);
//  6. per value column: a_i, b_i = state part + sum_m H d_m; the triangular
//     solve d_i = beta_i (v_i - a_i) - sum_{j<i} A_ij d_j (forward
//     substitution of (I + A) D = R) and o_i = scale (b_i + sum_{j<=i} F_ij d_j);
//  7. the T records go to ring positions base + i (base = fold ? 0 : c).
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
  constexpr int NV = 2 * NT;     // mat-vec vectors: k_i at [0, NT), q_i at [NT, 2NT)
  constexpr int VB = vblock(NT);  // vectors per accumulator block
  extern __shared__ __align__(128) unsigned char smem[];

  const int h = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = p.T, dk = p.dk, dv = p.dv, L = p.L, HV = p.HV, HK = p.HK;
  const int kh = h / p.G;

  // ---- row resolve and fold decision (uniform over the CTA and its cluster)
  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (h == 0 && tid == 0) atomicOr(p.err, DEVERR_SLOT);
    return;
  }
  const int c = p.cursor[s];
  if (c < 0 || c > L) {
    if (h == 0 && tid == 0) atomicOr(p.err, DEVERR_CURSOR);
    return;
  }
  const bool fold = (p.force != nullptr && p.force[r] != 0) || (c + T > L);
  const int base = fold ? 0 : c;
  const int nh = c;
  const bool group_sync = fold && p.G > 1;

  ST* tile = reinterpret_cast<ST*>(smem);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + p.sm.mbar);
  float* wq = reinterpret_cast<float*>(smem + p.sm.wq);
  float* wk = reinterpret_cast<float*>(smem + p.sm.wk);
  float* wv = reinterpret_cast<float*>(smem + p.sm.wv);
  float* wb = reinterpret_cast<float*>(smem + p.sm.wb);
  float* wg = reinterpret_cast<float*>(smem + p.sm.wg);
  float* scal = reinterpret_cast<float*>(smem + p.sm.scal);
  float* xh = reinterpret_cast<float*>(smem + p.sm.xh);
  float* am = reinterpret_cast<float*>(smem + p.sm.am);
  float* fm = reinterpret_cast<float*>(smem + p.sm.fm);
  float* hk = reinterpret_cast<float*>(smem + p.sm.hk);
  float* hd = reinterpret_cast<float*>(smem + p.sm.hd);
  float* hf = reinterpret_cast<float*>(smem + p.sm.hf);
  float* hdot = reinterpret_cast<float*>(smem + p.sm.hdot);
  // GDN scalars: es[NT] = e^{Gam_e + G_i}, eG[NT] = e^{G_i}, scal[2NT..] = Gam, e^Gam.
  // KDA vectors: egam[dk] = e^{Gam[ch]}, gam[dk] = Gam[ch].
  float* es = scal;
  float* eG = scal + NT;
  float* hscal = scal + 2 * NT;
  float* egam = scal;
  float* gam = scal + dk;

  const size_t tile_elems = (size_t)dk * dv;
  ST* gtile = static_cast<ST*>(p.state) + ((size_t)s * HV + h) * tile_elems;

  // ---- 1. checkpoint tile -> shared memory (async), window + history loads
  if (tid == 0) {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mbar_init(&mbar[w], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) load_tile_async(tile, gtile, dk, dv, mbar);

  const size_t tok0 = (size_t)r * T;
  for (int e = tid; e < T * dk; e += kThreads) {
    const int i = e / dk, ch = e - i * dk;
    const size_t gi = ((tok0 + i) * HK + kh) * dk + ch;
    wq[e] = ld_f32(p.q, gi, p.in_dt);
    wk[e] = ld_f32(p.k, gi, p.in_dt);
  }
  for (int e = tid; e < T * dv; e += kThreads) {
    const int i = e / dv, col = e - i * dv;
    wv[e] = ld_f32(p.v, ((tok0 + i) * HV + h) * dv + col, p.in_dt);
  }
  if (tid < T) wb[tid] = p.beta[(tok0 + tid) * HV + h];
  if (ALGO == ALGO_GDN) {
    if (tid < T) wg[tid] = p.g[(tok0 + tid) * HV + h];
  } else {
    for (int e = tid; e < T * dk; e += kThreads) {
      const int i = e / dk, ch = e - i * dk;
      wg[e] = p.g[((tok0 + i) * HV + h) * dk + ch];
    }
  }
  const size_t kbase = ((size_t)s * HK + kh) * L * dk;
  const size_t dbase = ((size_t)s * HV + h) * L * dv;
  const size_t gbase = ((size_t)s * HV + h) * L * (ALGO == ALGO_GDN ? 1 : dk);
  if (nh > 0) {
    stage_history<ALGO>(nh, dk, dv, p.ring_k, kbase, p.rk_dt, p.ring_d, dbase, p.rd_dt,
                        p.ring_g, gbase, hk, hd, hf, tid);
  }
  __syncthreads();
  // This CTA has read every old key record it needs; a folding sibling may
  // overwrite them once all of the key group has arrived.
  if (group_sync) cluster_arrive_release();

  // ---- 2. gates: history decay factors, in-window prefixes
  if (nh > 0) {
    history_decay<ALGO>(nh, dk, hk, hf, hscal, gam, egam, p.ring_g, gbase, tid, warp, lane);
  } else {
    if (ALGO == ALGO_GDN) {
      if (tid == 0) {
        hscal[0] = 0.f;
        hscal[1] = 1.f;
      }
    } else {
      for (int ch = tid; ch < dk; ch += kThreads) {
        gam[ch] = 0.f;
        egam[ch] = 1.f;
      }
    }
    __syncthreads();
  }
  if (ALGO == ALGO_GDN) {
    if (warp == 0) {
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
    for (int ch = tid; ch < dk; ch += kThreads) {
      float G = 0.f;
      for (int i = 0; i < T; ++i) {
        G += wg[i * dk + ch];
        wg[i * dk + ch] = G;
      }
    }
  }
  __syncthreads();

  // ---- 3. window coefficients A, F (j <= i only) and mat-vec inputs
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
  for (int e = tid; e < dk * NV; e += kThreads) {
    const int ch = e / NV, vv = e - ch * NV;
    const int i = vv < NT ? vv : vv - NT;
    float x = 0.f;
    if (i < T) {
      x = vv < NT ? wk[i * dk + ch] : wq[i * dk + ch];
      if (ALGO == ALGO_KDA) x *= __expf((fold ? 0.f : gam[ch]) + wg[i * dk + ch]);
    }
    xh[e] = x;
  }
  __syncthreads();
  if (ALGO == ALGO_KDA && !fold && nh > 0) {
    // history dots use e^{G_i} x (the history keys carry their own decay)
    for (int e = tid; e < T * dk; e += kThreads) {
      const float eg = __expf(wg[e]);
      wk[e] *= eg;
      wq[e] *= eg;
    }
    __syncthreads();
  }

  // ---- 4. fold, or history dot coefficients
  bool tile_ok = true;
  bool waited = false;
  if (fold) {
    if (nh > 0) {
      tile_ok = mbar_wait_bounded(&mbar[warp], 0);
      waited = true;
      fold_rows<ALGO, ST>(tile, gtile, nh, dk, dv, hk, hd, hscal[1], egam, warp, lane);
      __syncwarp();
    }
  } else if (nh > 0) {
    for (int m = warp; m < nh; m += kWarps) {
      float part[NV];
#pragma unroll
      for (int vv = 0; vv < NV; ++vv) part[vv] = 0.f;
      for (int ch = lane; ch < dk; ch += 32) {
        const float km = hk[m * dk + ch];
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) {
          const int i = vv < NT ? vv : vv - NT;
          if (i < T) part[vv] = fmaf(km, (vv < NT ? wk : wq)[i * dk + ch], part[vv]);
        }
      }
#pragma unroll
      for (int vv = 0; vv < NV; ++vv) part[vv] = warp_sum(part[vv]);
      if (lane == 0) {
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) {
          const int i = vv < NT ? vv : vv - NT;
          float hv = 0.f;
          if (i < T) hv = (ALGO == ALGO_GDN) ? part[vv] * eG[i] : part[vv];
          hdot[m * NV + vv] = hv;
        }
      }
    }
  }

  // ---- 5. S^T x for all window vectors, one pass over the tile
  if (!waited) tile_ok = mbar_wait_bounded(&mbar[warp], 0);
  if (!tile_ok) atomicOr(p.err, DEVERR_TIMEOUT);

  const TileMap tm(dk, dv, warp, lane);
  float y[NV];  // per value column (thread tid < dv): reduced S^T x
#pragma unroll
  for (int vv = 0; vv < NV; ++vv) y[vv] = 0.f;

#pragma unroll
  for (int v0 = 0; v0 < NV; v0 += VB) {
    float acc[VB][4];
#pragma unroll
    for (int v = 0; v < VB; ++v) acc[v][0] = acc[v][1] = acc[v][2] = acc[v][3] = 0.f;
    for (int t = 0; t < tm.rpt; ++t) {
      const int row = tm.row0 + t;
      const float4 s4 = StateIO<ST>::load4(tile + (size_t)row * dv + 4 * tm.cc);
      const float* xr = xh + (size_t)row * NV + v0;
      if constexpr (VB % 4 == 0) {
#pragma unroll
        for (int q4 = 0; q4 < VB / 4; ++q4) {
          const float4 x = reinterpret_cast<const float4*>(xr)[q4];
          const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            acc[4 * q4 + u][0] = fmaf(xs[u], s4.x, acc[4 * q4 + u][0]);
            acc[4 * q4 + u][1] = fmaf(xs[u], s4.y, acc[4 * q4 + u][1]);
            acc[4 * q4 + u][2] = fmaf(xs[u], s4.z, acc[4 * q4 + u][2]);
            acc[4 * q4 + u][3] = fmaf(xs[u], s4.w, acc[4 * q4 + u][3]);
          }
        }
      } else {
        const float2 x = *reinterpret_cast<const float2*>(xr);
        const float xs[2] = {x.x, x.y};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          acc[u][0] = fmaf(xs[u], s4.x, acc[u][0]);
          acc[u][1] = fmaf(xs[u], s4.y, acc[u][1]);
          acc[u][2] = fmaf(xs[u], s4.z, acc[u][2]);
          acc[u][3] = fmaf(xs[u], s4.w, acc[u][3]);
        }
      }
    }
    // reduce over the lanes that share columns (row sub-lanes)
    for (int off = tm.ccw; off < 32; off <<= 1) {
#pragma unroll
      for (int v = 0; v < VB; ++v) {
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[v][u] += __shfl_xor_sync(kFull, acc[v][u], off);
      }
    }
    float* red = p.sm.red_alias
                     ? reinterpret_cast<float*>(smem + (size_t)warp * (dk / kWarps) * dv * sizeof(ST))
                     : reinterpret_cast<float*>(smem + p.sm.red) + (size_t)warp * VB * dv;
    if (p.sm.red_alias) __syncwarp();  // every lane is done with this warp's tile rows
    if (tm.rs == 0) {
#pragma unroll
      for (int v = 0; v < VB; ++v) {
        *reinterpret_cast<float4*>(red + (size_t)v * dv + 4 * tm.cc) =
            make_float4(acc[v][0], acc[v][1], acc[v][2], acc[v][3]);
      }
    }
    __syncthreads();
    if (tid < dv) {
      const size_t wstride =
          p.sm.red_alias ? (size_t)(dk / kWarps) * dv * sizeof(ST) / sizeof(float) : (size_t)VB * dv;
      const float* red0 = p.sm.red_alias ? reinterpret_cast<const float*>(smem)
                                         : reinterpret_cast<const float*>(smem + p.sm.red);
#pragma unroll
      for (int v = 0; v < VB; ++v) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += red0[w * wstride + (size_t)v * dv + tid];
        y[v0 + v] = sum;
      }
    }
    if (v0 + VB < NV) __syncthreads();
  }

  // ---- 6. per value column: corrections, triangular solve, outputs, deltas
  if (tid < dv) {
    const int col = tid;
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

  // ---- 7. remaining records: keys (once per key head), gates, beta
  if (group_sync) cluster_wait_acquire();
  if (h % p.G == 0) {
    for (int e = tid; e < T * dk; e += kThreads) {
      const int i = e / dk, ch = e - i * dk;
      const float kv = ld_f32(p.k, ((tok0 + i) * HK + kh) * dk + ch, p.in_dt);
      st_f32(p.ring_k, kbase + (size_t)(base + i) * dk + ch, p.rk_dt, kv);
    }
  }
  if (tid < T) p.ring_beta[((size_t)s * HV + h) * L + base + tid] = p.beta[(tok0 + tid) * HV + h];
  if (ALGO == ALGO_GDN) {
    if (tid < T) p.ring_g[gbase + base + tid] = p.g[(tok0 + tid) * HV + h];
  } else {
    for (int e = tid; e < T * dk; e += kThreads) {
      const int i = e / dk, ch = e - i * dk;
      p.ring_g[gbase + (size_t)(base + i) * dk + ch] = p.g[((tok0 + i) * HV + h) * dk + ch];
    }
  }
  if (h == 0 && tid == 0 && p.fold_out != nullptr) p.fold_out[r] = fold ? 1 : 0;
  if (!tile_ok) {
    // give the copy that did not arrive a second bounded chance before exit
    mbar_wait_bounded(&mbar[warp], 0);
  }
}

}  // namespace rssm
