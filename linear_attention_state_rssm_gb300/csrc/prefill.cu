// Replay prefill: the prompt runs through the gated delta rule and the
// checkpoint takes the resulting state; the cursor is then cleared (LightLLM
// PR #1690 "feat: add ReplaySSM state modes for GDN and KDA", commit messages:
// prefill writes the canonical state directly and leaves the cursor at zero).
//
// One CTA per (request row, value head, block of CB value columns): the
// columns of the delta rule evolve independently given the keys, gates and
// betas, so a CTA keeps its [dk][CB] slice of the state in shared memory (fp32)
// for the whole prompt and never writes it to HBM until the end. The row's
// committed state is built first: the checkpoint slice, then the c ring
// records replayed into it (S <- e^{g_m} S + k_m d_m^T, 16 records at a time).
//
// The prompt is scanned in chunks of C = 16 tokens, each in the triangular
// form of the replay window:
//     A_ij = beta_i e^{G_i-G_j} k_i.k_j (j < i),  F_ij = e^{G_i-G_j} q_i.k_j (j <= i)
//     a_i = S^T (e^{G_i} k_i),  b_i = S^T (e^{G_i} q_i)
//     d_i = beta_i (v_i - a_i) - sum_{j<i} A_ij d_j,  o_i = scale (b_i + sum_{j<=i} F_ij d_j)
//     S <- e^{G_last} S + sum_j e^{G_last-G_j} k_j d_j^T
// (G_i the in-chunk inclusive gate prefix; per key channel for KDA). Each
// chunk's inputs are loaded into registers (16-byte coalesced loads) while the
// chunk before is computed, and widened to fp32 as they are stored to shared
// memory. The O(dk CB) work per token runs on CUDA cores in fp32: the
// two mat-vec passes (one column and 16 vectors per thread, inputs broadcast
// from a per-channel row) and the rank-16 update (four columns and sixteen
// rows per step of a thread).
#include "replay_impl.cuh"
#include "rssm_launch.h"

namespace rssm {

// Sixteen bytes of 16-bit (INB = 2) or fp32 (INB = 4) values -> fp32 in shared memory.
template <int INB>
__device__ __forceinline__ void widen_store(float* dst, const uint4& u, int in_dt) {
  if (INB == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(u.x), __uint_as_float(u.y),
                                                  __uint_as_float(u.z), __uint_as_float(u.w));
  } else {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float f[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float2 x;
      if (in_dt == DT_F16) {
        x = __half22float2(*reinterpret_cast<const __half2*>(&w[t]));
      } else {
        x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[t]));
      }
      f[2 * t] = x.x;
      f[2 * t + 1] = x.y;
    }
    *reinterpret_cast<float4*>(dst) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
}

template <int ALGO, typename ST, int CB, int INB>
__global__ void __launch_bounds__(kPrefillThreads, 2) prefill_kernel(const PrefillParams p) {
  constexpr int PT = kPrefillThreads, PW = PT / 32;
  constexpr int C = kPrefillChunk;
  constexpr int CQ = CB / 4;                  // column quads
  constexpr int VT = 2 * C * CQ / PT;         // mat-vec vectors per thread (4 columns each)
  constexpr int NRG = PT / CQ;                // row groups of the update
  constexpr int XS = kPrefillXS, KS = kPrefillKS;
  constexpr int EPU = 16 / INB;               // input values per 16-byte unit
  // 16-byte units of one chunk per thread (dk <= 128): q and k rows, v
  // columns, KDA gates
  constexpr int MQ = (C * 128 / EPU + PT - 1) / PT;
  constexpr int MV = (C * CB / EPU + PT - 1) / PT;
  constexpr int MG = ALGO == ALGO_KDA ? (C * 128 / 4 + PT - 1) / PT : 0;
  static_assert((VT == 1 || VT == 2) && PT % CQ == 0, "prefill lane layout");
  extern __shared__ __align__(128) unsigned char smem[];

  const int nb = p.dv / CB;
  const int h = blockIdx.x / nb, cb0 = (blockIdx.x - h * nb) * CB, r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dk = p.dk, dv = p.dv, L = p.L, HV = p.HV, HK = p.HK, kh = h / p.G;
  const bool reporter = tid == 0 && blockIdx.x == 0;

  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (reporter) atomicOr(p.err, DEVERR_SLOT);
    return;
  }
  const int a0 = p.cu[r], a1 = p.cu[r + 1];
  if (a0 < 0 || a1 < a0) {
    if (reporter) atomicOr(p.err, DEVERR_SEQLEN);
    return;
  }
  const int n = a1 - a0;
  if (n == 0) return;  // no prompt tokens: the row is left as it is
  const int c = p.cursor[s];
  if (c < 0 || c > L) {
    if (reporter) atomicOr(p.err, DEVERR_CURSOR);
    return;
  }

  float* S = reinterpret_cast<float*>(smem + p.sm.S);
  float* wq = reinterpret_cast<float*>(smem + p.sm.wq);
  float* wk = reinterpret_cast<float*>(smem + p.sm.wk);
  float* wv = reinterpret_cast<float*>(smem + p.sm.wv);
  float* xT = reinterpret_cast<float*>(smem + p.sm.xT);
  float* kdT = xT;  // the update's decayed keys replace the mat-vec inputs
  float* y = reinterpret_cast<float*>(smem + p.sm.y);
  float* part = y;  // GDN pair partial sums [PW][2C][C], before y is written
  float* dch = reinterpret_cast<float*>(smem + p.sm.dch);
  float* am = reinterpret_cast<float*>(smem + p.sm.am);
  float* fm = reinterpret_cast<float*>(smem + p.sm.fm);
  float* G = reinterpret_cast<float*>(smem + p.sm.G);
  float* eG = reinterpret_cast<float*>(smem + p.sm.eG);
  float* ekd = reinterpret_cast<float*>(smem + p.sm.ekd);
  float* wb = reinterpret_cast<float*>(smem + p.sm.wb);
  float* decr = reinterpret_cast<float*>(smem + p.sm.decr);

  const int uq = dk / EPU, uv = CB / EPU, ug = dk / 4;  // 16-byte units per row
  const int nchunks = (n + C - 1) / C;

  // ---- the next chunk's inputs, loaded into registers one chunk ahead
  uint4 rq[MQ], rk[MQ], rv[MV], rg[MG > 0 ? MG : 1];
  float rb = 0.f, rgg = 0.f;  // beta and GDN gate of token tid of the chunk
  auto prefetch = [&](int ch) {
    const int t0 = ch * C, cn = min(C, n - t0);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
      const int u = tid + m * PT, i = u / uq, pu = u - i * uq;
      rq[m] = z;
      rk[m] = z;
      if (u < C * uq && i < cn) {
        const size_t row = ((size_t)a0 + t0 + i) * HK + kh;
        rq[m] = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(p.q) +
                                                     (row * dk) * INB) + pu);
        rk[m] = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(p.k) +
                                                     (row * dk) * INB) + pu);
      }
    }
#pragma unroll
    for (int m = 0; m < MV; ++m) {
      const int u = tid + m * PT, i = u / uv, pu = u - i * uv;
      rv[m] = z;
      if (u < C * uv && i < cn) {
        const size_t off = ((((size_t)a0 + t0 + i) * HV + h) * dv + cb0) * INB;
        rv[m] = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(p.v) + off) + pu);
      }
    }
#pragma unroll
    for (int m = 0; m < MG; ++m) {
      const int u = tid + m * PT, i = u / ug, pu = u - i * ug;
      rg[m] = z;
      if (u < C * ug && i < cn) {
        const size_t off = (((size_t)a0 + t0 + i) * HV + h) * dk;
        rg[m] = __ldg(reinterpret_cast<const uint4*>(p.g + off) + pu);
      }
    }
    rb = 0.f;
    rgg = 0.f;
    if (tid < cn) {
      const size_t tok = (size_t)a0 + t0 + tid;
      rb = __ldg(p.beta + tok * HV + h);
      if (ALGO == ALGO_GDN) rgg = __ldg(p.g + tok * HV + h);
    }
  };
  // registers -> fp32 chunk arrays (rows past the chunk are zero)
  auto stage = [&]() {
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
      const int u = tid + m * PT, i = u / uq, pu = u - i * uq;
      if (u < C * uq) {
        widen_store<INB>(wq + i * dk + pu * EPU, rq[m], p.in_dt);
        widen_store<INB>(wk + i * dk + pu * EPU, rk[m], p.in_dt);
      }
    }
#pragma unroll
    for (int m = 0; m < MV; ++m) {
      const int u = tid + m * PT, i = u / uv, pu = u - i * uv;
      if (u < C * uv) widen_store<INB>(wv + i * CB + pu * EPU, rv[m], p.in_dt);
    }
#pragma unroll
    for (int m = 0; m < MG; ++m) {
      const int u = tid + m * PT, i = u / ug, pu = u - i * ug;
      if (u < C * ug) widen_store<4>(G + i * dk + pu * 4, rg[m], DT_F32);
    }
    if (tid < C) wb[tid] = rb;
  };
  // GDN, warp 0: inclusive prefix of the nm gates x (lane i holds gate i),
  // G[i], eG[i] = e^{G_i}, ekd[i] = e^{G_last - G_i}
  auto gdn_scan = [&](float x, int nm) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += u;
    }
    const float gl = __shfl_sync(kFull, x, nm - 1);
    if (lane < C) {
      G[lane] = x;
      eG[lane] = __expf(x);
      ekd[lane] = lane < nm ? __expf(gl - x) : 0.f;
    }
  };
  // KDA, one thread per key channel: in-place inclusive prefix of G rows
  // [0, nm) and the channel's total decay
  auto kda_scan = [&](int nm) {
    for (int ch = tid; ch < dk; ch += PT) {
      float acc = 0.f;
      for (int i = 0; i < nm; ++i) {
        acc += G[i * dk + ch];
        G[i * dk + ch] = acc;
      }
      decr[ch] = __expf(acc);
    }
  };
  // decayed keys of the update, one key channel per thread:
  // kdT[row][j] = e^{G_last - G_j} k_j[row] (per channel for KDA), zero for j >= nm
  auto build_kd = [&](int nm, int t, int nt) {
    for (int row = t; row < dk; row += nt) {
      float kd[C];
#pragma unroll
      for (int j = 0; j < C; ++j) {
        float f = 0.f;
        if (j < nm) {
          f = ALGO == ALGO_KDA ? __expf(G[(nm - 1) * dk + row] - G[j * dk + row]) : ekd[j];
        }
        kd[j] = f * wk[j * dk + row];
      }
#pragma unroll
      for (int j4 = 0; j4 < C; j4 += 4) {
        *reinterpret_cast<float4*>(kdT + row * KS + j4) =
            make_float4(kd[j4], kd[j4 + 1], kd[j4 + 2], kd[j4 + 3]);
      }
    }
  };
  // S <- e^{G_last} S + sum_j kd_j d_j^T (dch rows past the chunk are zero)
  auto update = [&](float dec) {
    const int q4 = tid % CQ, rg0 = tid / CQ;
    float4 dq[C];
#pragma unroll
    for (int j = 0; j < C; ++j) dq[j] = ld4(dch + j * CB + 4 * q4);
#pragma unroll 2
    for (int row = rg0; row < dk; row += NRG) {
      float4 s4 = ld4(S + row * CB + 4 * q4);
      const float f = ALGO == ALGO_KDA ? decr[row] : dec;
      s4.x *= f;
      s4.y *= f;
      s4.z *= f;
      s4.w *= f;
#pragma unroll
      for (int j4 = 0; j4 < C; j4 += 4) {
        const float4 kd = ld4(kdT + row * KS + j4);
        const float kv[4] = {kd.x, kd.y, kd.z, kd.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          s4.x = fmaf(kv[u], dq[j4 + u].x, s4.x);
          s4.y = fmaf(kv[u], dq[j4 + u].y, s4.y);
          s4.z = fmaf(kv[u], dq[j4 + u].z, s4.z);
          s4.w = fmaf(kv[u], dq[j4 + u].w, s4.w);
        }
      }
      *reinterpret_cast<float4*>(S + row * CB + 4 * q4) = s4;
    }
  };

  prefetch(0);

  // ---- the checkpoint slice -> fp32 S [dk][CB]
  ST* gtile = static_cast<ST*>(p.state) + ((size_t)s * HV + h) * dk * dv + cb0;
  for (int e = tid; e < dk * CQ; e += PT) {
    const int row = e / CQ, q4 = e - row * CQ;
    float v4[4];
    ld_cols<ST, 4>(gtile + (size_t)row * dv + 4 * q4, v4);
    *reinterpret_cast<float4*>(S + row * CB + 4 * q4) = make_float4(v4[0], v4[1], v4[2], v4[3]);
  }

  // ---- committed state: replay the c ring records into S, 16 at a time
  const size_t sh = (size_t)s * HV + h;
  for (int m0 = 0; m0 < c; m0 += C) {
    const int nm = min(C, c - m0);
    for (int e = tid; e < C * dk; e += PT) {
      const int j = e / dk, ch = e - j * dk;
      wk[e] = j < nm ? ld_f32(p.ring_k, (sh * L + m0 + j) * dk + ch, p.rk_dt) : 0.f;
      if (ALGO == ALGO_KDA && j < nm) G[e] = p.ring_g[(sh * L + m0 + j) * dk + ch];
    }
    for (int e = tid; e < C * CB; e += PT) {
      const int j = e / CB, col = e - j * CB;
      dch[e] = j < nm ? ld_f32(p.ring_d, (sh * L + m0 + j) * dv + cb0 + col, p.rd_dt) : 0.f;
    }
    if (ALGO == ALGO_GDN && warp == 0) gdn_scan(lane < nm ? p.ring_g[sh * L + m0 + lane] : 0.f, nm);
    __syncthreads();
    if (ALGO == ALGO_KDA) {
      kda_scan(nm);
      __syncthreads();
    }
    build_kd(nm, tid, PT);
    __syncthreads();
    update(ALGO == ALGO_GDN ? __expf(G[nm - 1]) : 1.f);
    __syncthreads();
  }

  // ---- the prompt, chunk by chunk
  const int cq = tid % CQ, vg = tid / CQ;  // mat-vec: columns 4cq.., vectors vg*VT..
  for (int ch = 0; ch < nchunks; ++ch) {
    const int t0 = ch * C, cn = min(C, n - t0);
    stage();
    if (ALGO == ALGO_GDN && warp == 0) gdn_scan(rgg, cn);
    if (ch + 1 < nchunks) prefetch(ch + 1);
    __syncthreads();
    if (ALGO == ALGO_KDA) {
      kda_scan(cn);
      __syncthreads();
    }

    // ---- mat-vec inputs per key channel: k_i at [0, C), q_i at [C, 2C)
    //      (KDA: decayed by e^{G_i} per channel); half the threads each
    for (int e = tid; e < 2 * dk; e += PT) {
      const int row = e >> 1, half = e & 1;
      const float* src = half ? wq : wk;
      float x[C];
#pragma unroll
      for (int i = 0; i < C; ++i) {
        const float f = (ALGO == ALGO_KDA && i < cn) ? __expf(G[i * dk + row]) : 1.f;
        x[i] = f * src[i * dk + row];
      }
#pragma unroll
      for (int i4 = 0; i4 < C; i4 += 4) {
        *reinterpret_cast<float4*>(xT + row * XS + half * C + i4) =
            make_float4(x[i4], x[i4 + 1], x[i4 + 2], x[i4 + 3]);
      }
    }
    if (ALGO == ALGO_KDA) {
      window_pairs<ALGO, C>(cn, dk, wk, wq, G, wb, am, fm, warp, PW, lane);
    }
    __syncthreads();

    // ---- GDN window coefficients: lane j of a half warp accumulates k_i.k_j
    //      and q_i.k_j for every i over its channels (raw vectors; the
    //      in-window decay and beta go on when the partial sums are combined)
    if (ALGO == ALGO_GDN) {
      {
        const int j = tid & 15, cgrp = tid >> 4;  // 16 channel groups
        float kk[C], qk[C];
#pragma unroll
        for (int i = 0; i < C; ++i) {
          kk[i] = 0.f;
          qk[i] = 0.f;
        }
        for (int ch = cgrp; ch < dk; ch += PT / 16) {
          const float* xr = xT + ch * XS;
          const float kj = xr[j];
#pragma unroll
          for (int i4 = 0; i4 < C; i4 += 4) {
            const float4 k4 = ld4(xr + i4), q4v = ld4(xr + C + i4);
            kk[i4] = fmaf(k4.x, kj, kk[i4]);
            kk[i4 + 1] = fmaf(k4.y, kj, kk[i4 + 1]);
            kk[i4 + 2] = fmaf(k4.z, kj, kk[i4 + 2]);
            kk[i4 + 3] = fmaf(k4.w, kj, kk[i4 + 3]);
            qk[i4] = fmaf(q4v.x, kj, qk[i4]);
            qk[i4 + 1] = fmaf(q4v.y, kj, qk[i4 + 1]);
            qk[i4 + 2] = fmaf(q4v.z, kj, qk[i4 + 2]);
            qk[i4 + 3] = fmaf(q4v.w, kj, qk[i4 + 3]);
          }
        }
#pragma unroll
        for (int i = 0; i < C; ++i) {
          kk[i] += __shfl_xor_sync(kFull, kk[i], 16);
          qk[i] += __shfl_xor_sync(kFull, qk[i], 16);
        }
        // partial sums [warp][2C][C]: lane j of the lower half stores column j
        if (lane < 16) {
          float* pw = part + warp * 2 * C * C + j;
#pragma unroll
          for (int i = 0; i < C; ++i) {
            pw[i * C] = kk[i];
            pw[(C + i) * C] = qk[i];
          }
        }
      }
      __syncthreads();
      // A_ij = beta_i e^{G_i - G_j} k_i.k_j (j < i), F_ij = e^{G_i - G_j} q_i.k_j (j <= i)
      {
        const int i = tid >> 4, j = tid & 15;
        float skk = 0.f, sqk = 0.f;
#pragma unroll
        for (int w = 0; w < PW; ++w) {
          skk += part[(w * 2 * C + i) * C + j];
          sqk += part[(w * 2 * C + C + i) * C + j];
        }
        const bool on = i < cn && j <= i;
        const float wgt = on ? __expf(G[i] - G[j]) : 0.f;
        fm[i * C + j] = on ? wgt * sqk : 0.f;
        am[i * C + j] = (on && j < i) ? wb[i] * wgt * skk : 0.f;
      }
      __syncthreads();
    }

    // ---- y_v = S^T x_v
    if (CB == 64) {
      // four columns x eight vectors per thread over a quarter of the rows
      // (rows kq, kq + 4, ...: the four quarters of a step read four
      // consecutive rows, on distinct banks), summed over the quarters by
      // shuffles; lane = column quad (low 3 bits) + 8 quarter, warp = column
      // half + 2 vector octet
      const int cqm = (warp & 1) * 8 + (lane & 7), kq = lane >> 3, vo = warp >> 1;
      float acc[8][4];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[u][q] = 0.f;
      }
      const float* sp = S + 4 * cqm;
      const float* xp = xT + 8 * vo;
#pragma unroll 2
      for (int row = kq; row < dk; row += 4) {
        const float4 s4 = ld4(sp + row * CB);
        const float4 xa = ld4(xp + row * XS), xb = ld4(xp + row * XS + 4);
        const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc[u][0] = fmaf(s4.x, xv[u], acc[u][0]);
          acc[u][1] = fmaf(s4.y, xv[u], acc[u][1]);
          acc[u][2] = fmaf(s4.z, xv[u], acc[u][2]);
          acc[u][3] = fmaf(s4.w, xv[u], acc[u][3]);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[u][q] += __shfl_xor_sync(kFull, acc[u][q], 8);
          acc[u][q] += __shfl_xor_sync(kFull, acc[u][q], 16);
        }
      }
      // quarter kq stores vectors 2kq, 2kq + 1 of the octet
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if ((u >> 1) == kq) {
          const int vv = 8 * vo + u;
          const float f = ALGO == ALGO_GDN ? eG[vv < C ? vv : vv - C] : 1.f;
          *reinterpret_cast<float4*>(y + vv * CB + 4 * cqm) =
              make_float4(f * acc[u][0], f * acc[u][1], f * acc[u][2], f * acc[u][3]);
        }
      }
    } else {
      // four columns and VT vectors per thread over all rows
      float acc[VT][4];
#pragma unroll
      for (int u = 0; u < VT; ++u) {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[u][q] = 0.f;
      }
      const float* sp = S + 4 * cq;
      const float* xp = xT + vg * VT;
#pragma unroll 4
      for (int row = 0; row < dk; ++row) {
        const float4 s4 = ld4(sp + row * CB);
        float xv[VT];
        if (VT == 2) {
          const float2 x2 = *reinterpret_cast<const float2*>(xp + row * XS);
          xv[0] = x2.x;
          xv[VT - 1] = x2.y;
        } else {
          xv[0] = xp[row * XS];
        }
#pragma unroll
        for (int u = 0; u < VT; ++u) {
          acc[u][0] = fmaf(s4.x, xv[u], acc[u][0]);
          acc[u][1] = fmaf(s4.y, xv[u], acc[u][1]);
          acc[u][2] = fmaf(s4.z, xv[u], acc[u][2]);
          acc[u][3] = fmaf(s4.w, xv[u], acc[u][3]);
        }
      }
#pragma unroll
      for (int u = 0; u < VT; ++u) {
        const int vv = vg * VT + u;
        const float f = ALGO == ALGO_GDN ? eG[vv < C ? vv : vv - C] : 1.f;
        *reinterpret_cast<float4*>(y + vv * CB + 4 * cq) =
            make_float4(f * acc[u][0], f * acc[u][1], f * acc[u][2], f * acc[u][3]);
      }
    }
    __syncthreads();

    // ---- per column: triangular solve and outputs; meanwhile the other
    //      threads build the update's decayed keys (over xT, now free)
    if (tid < CB) {
      float d[C];
#pragma unroll
      for (int i = 0; i < C; ++i) {
        d[i] = 0.f;
        if (i < cn) {
          float di = wb[i] * (wv[i * CB + tid] - y[i * CB + tid]);
#pragma unroll
          for (int j = 0; j < i; ++j) di = fmaf(-am[i * C + j], d[j], di);
          d[i] = di;
          float oi = y[(C + i) * CB + tid];
#pragma unroll
          for (int j = 0; j <= i; ++j) oi = fmaf(fm[i * C + j], d[j], oi);
          st_f32(p.o, (((size_t)a0 + t0 + i) * HV + h) * dv + cb0 + tid, p.in_dt, p.scale * oi);
        }
        dch[i * CB + tid] = d[i];
      }
    } else {
      build_kd(cn, tid - CB, PT - CB);
    }
    // the chunk's decay, read before warp 0 may scan the next chunk's gates
    const float dec = ALGO == ALGO_GDN ? eG[cn - 1] : 1.f;
    __syncthreads();
    // (the next chunk's staging writes none of what the update reads)
    update(dec);
  }
  __syncthreads();

  // ---- the checkpoint takes the state (rounded to its dtype)
  for (int e = tid; e < dk * CQ; e += PT) {
    const int row = e / CQ, q4 = e - row * CQ;
    const float4 s4 = ld4(S + row * CB + 4 * q4);
    float v4[4] = {s4.x, s4.y, s4.z, s4.w};
    st_cols<ST, 4>(gtile + (size_t)row * dv + 4 * q4, v4);
  }
}

template <int ALGO, typename ST, int CB, int INB>
static cudaError_t prefill_prepare_one(int max_smem) {
  return cudaFuncSetAttribute(prefill_kernel<ALGO, ST, CB, INB>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

template <int ALGO, typename ST>
static cudaError_t prefill_launch_t(const PrefillParams& p, cudaStream_t st) {
  const dim3 grid((unsigned)(p.HV * (p.dv / p.CB)), (unsigned)p.B, 1);
  const bool f32in = p.in_dt == DT_F32;
  if (p.CB == 64) {
    if (f32in) prefill_kernel<ALGO, ST, 64, 4><<<grid, kPrefillThreads, p.sm.total, st>>>(p);
    else prefill_kernel<ALGO, ST, 64, 2><<<grid, kPrefillThreads, p.sm.total, st>>>(p);
  } else if (p.CB == 32) {
    if (f32in) prefill_kernel<ALGO, ST, 32, 4><<<grid, kPrefillThreads, p.sm.total, st>>>(p);
    else prefill_kernel<ALGO, ST, 32, 2><<<grid, kPrefillThreads, p.sm.total, st>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int ALGO, typename ST>
static cudaError_t prefill_prepare_t(int max_smem) {
  cudaError_t e;
  if ((e = prefill_prepare_one<ALGO, ST, 64, 4>(max_smem)) != cudaSuccess) return e;
  if ((e = prefill_prepare_one<ALGO, ST, 64, 2>(max_smem)) != cudaSuccess) return e;
  if ((e = prefill_prepare_one<ALGO, ST, 32, 4>(max_smem)) != cudaSuccess) return e;
  return prefill_prepare_one<ALGO, ST, 32, 2>(max_smem);
}

cudaError_t prefill_launch(int algo, int state_dt, const PrefillParams& p, cudaStream_t st) {
  if (algo == ALGO_GDN) {
    return state_dt == DT_F32 ? prefill_launch_t<ALGO_GDN, float>(p, st)
                              : prefill_launch_t<ALGO_GDN, __nv_bfloat16>(p, st);
  }
  return state_dt == DT_F32 ? prefill_launch_t<ALGO_KDA, float>(p, st)
                            : prefill_launch_t<ALGO_KDA, __nv_bfloat16>(p, st);
}

cudaError_t prefill_prepare(int algo, int state_dt, int max_smem) {
  if (algo == ALGO_GDN) {
    return state_dt == DT_F32 ? prefill_prepare_t<ALGO_GDN, float>(max_smem)
                              : prefill_prepare_t<ALGO_GDN, __nv_bfloat16>(max_smem);
  }
  return state_dt == DT_F32 ? prefill_prepare_t<ALGO_KDA, float>(max_smem)
                            : prefill_prepare_t<ALGO_KDA, __nv_bfloat16>(max_smem);
}

}  // namespace rssm
