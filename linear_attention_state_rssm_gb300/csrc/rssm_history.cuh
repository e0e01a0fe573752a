// Device helpers shared by the replay kernel and the fold kernel: staging the
// ring history, turning its gates into decay factors, and folding it into the
// checkpoint tile.
//
// Replay identity (LightLLM PR #1690 "feat: add ReplaySSM state modes for GDN
// and KDA": the checkpoint is the canonical state and the ring holds the
// accepted records): after n records (k_m, g_m, d_m) on top of checkpoint S0,
//   S = exp(Gam) * S0 + sum_m k~_m d_m^T,   k~_m = exp(sum_{m < m' < n} g_m') * k_m,
// with Gam = sum_{m < n} g_m (a scalar for GDN, a per-key-channel vector for KDA,
// where exp(Gam) scales row ch of S0).
#pragma once

#include "rssm_common.cuh"

namespace rssm {

// Stage n history records of one (slot, key head, value head) into shared
// memory as fp32: keys [n][dk], deltas [n][dv]; GDN raw gates [n] into hf.
template <int ALGO>
__device__ __forceinline__ void stage_history(int n, int dk, int dv, const void* ring_k,
                                              size_t kbase, int rk_dt, const void* ring_d,
                                              size_t dbase, int rd_dt, const float* ring_g,
                                              size_t gbase, float* hk, float* hd, float* hf,
                                              int tid) {
  for (int e = tid; e < n * dk; e += kThreads) hk[e] = ld_f32(ring_k, kbase + e, rk_dt);
  for (int e = tid; e < n * dv; e += kThreads) hd[e] = ld_f32(ring_d, dbase + e, rd_dt);
  if (ALGO == ALGO_GDN) {
    for (int m = tid; m < n; m += kThreads) hf[m] = ring_g[gbase + m];
  }
}

// Turn staged history into decay-scaled keys k~_m (in place in hk) and the total
// decay. Needs a __syncthreads() between stage_history and this call; ends with
// one. GDN: scal[0] <- Gam, scal[1] <- exp(Gam). KDA: gam[ch] <- Gam[ch],
// egam[ch] <- exp(Gam[ch]); the KDA record gates are read from global memory
// (ring_g + gbase, [n][dk]).
template <int ALGO>
__device__ __forceinline__ void history_decay(int n, int dk, float* hk, float* hf, float* scal,
                                              float* gam, float* egam, const float* ring_g,
                                              size_t gbase, int tid, int warp, int lane) {
  if (ALGO == ALGO_GDN) {
    if (warp == 0) {
      // Exclusive suffix sums of the record gates, 32 records at a time from
      // the newest: hf[m] <- exp(sum_{m' > m} g_m').
      float carry = 0.f;
      for (int hi = n; hi > 0; hi -= 32) {
        const int m = hi - 1 - lane;
        const float gv = (m >= 0) ? hf[m] : 0.f;
        float incl = gv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float t = __shfl_up_sync(kFull, incl, off);
          if (lane >= off) incl += t;
        }
        float excl = __shfl_up_sync(kFull, incl, 1);
        if (lane == 0) excl = 0.f;
        if (m >= 0) hf[m] = __expf(carry + excl);
        carry += __shfl_sync(kFull, incl, 31);
      }
      if (lane == 0) {
        scal[0] = carry;
        scal[1] = __expf(carry);
      }
    }
    __syncthreads();
    for (int e = tid; e < n * dk; e += kThreads) hk[e] *= hf[e / dk];
    __syncthreads();
  } else {
    for (int ch = tid; ch < dk; ch += kThreads) {
      float suf = 0.f;
      for (int m = n - 1; m >= 0; --m) {
        hk[m * dk + ch] *= __expf(suf);
        suf += ring_g[gbase + (size_t)m * dk + ch];
      }
      gam[ch] = suf;
      egam[ch] = __expf(suf);
    }
    __syncthreads();
  }
}

// Thread mapping of one warp over its quarter of the state tile: rows
// [warp*dk/4, (warp+1)*dk/4), a lane owning 4 consecutive columns of
// `rows_per_thread` consecutive rows.
struct TileMap {
  int cc, rs, ccw, rsw, rpt, row0;
  __device__ __forceinline__ TileMap(int dk, int dv, int warp, int lane) {
    const int rpw = dk / kWarps;
    ccw = dv / 4 < 32 ? dv / 4 : 32;
    rsw = 32 / ccw;
    cc = lane % ccw;
    rs = lane / ccw;
    rpt = rpw / rsw;
    row0 = warp * rpw + rs * rpt;
  }
};

// Fold n staged records into this warp's rows of the tile:
//   S[row][:] <- decay(row) S[row][:] + sum_m k~_m[row] d_m[:]
// and write the folded rows to shared memory and to the checkpoint in global
// memory. decay(row) = exp(Gam) (GDN) or exp(Gam[row]) (KDA).
template <int ALGO, typename ST>
__device__ __forceinline__ void fold_rows(ST* tile, ST* gtile, int n, int dk, int dv,
                                          const float* hk, const float* hd, float gdn_decay,
                                          const float* egam, int warp, int lane) {
  const TileMap tm(dk, dv, warp, lane);
  for (int t0 = 0; t0 < tm.rpt; t0 += 8) {
    const int nr = tm.rpt - t0 < 8 ? tm.rpt - t0 : 8;
    const int rbase = tm.row0 + t0;
    float4 acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < nr) {
        const int row = rbase + j;
        const float4 s4 = StateIO<ST>::load4(tile + (size_t)row * dv + 4 * tm.cc);
        const float dec = (ALGO == ALGO_GDN) ? gdn_decay : egam[row];
        acc[j] = make_float4(dec * s4.x, dec * s4.y, dec * s4.z, dec * s4.w);
      }
    }
    for (int m = 0; m < n; ++m) {
      const float4 d4 = *reinterpret_cast<const float4*>(hd + (size_t)m * dv + 4 * tm.cc);
      const float* km = hk + (size_t)m * dk + rbase;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < nr) {
          const float kt = km[j];
          acc[j].x = fmaf(kt, d4.x, acc[j].x);
          acc[j].y = fmaf(kt, d4.y, acc[j].y);
          acc[j].z = fmaf(kt, d4.z, acc[j].z);
          acc[j].w = fmaf(kt, d4.w, acc[j].w);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < nr) {
        const size_t off = (size_t)(rbase + j) * dv + 4 * tm.cc;
        StateIO<ST>::store4(tile + off, acc[j]);
        StateIO<ST>::store4(gtile + off, acc[j]);
      }
    }
  }
}

// Issue the bulk copies of one (slot, head) state tile: one row chunk per warp,
// each completing on its own mbarrier. Called by one thread after the
// mbarriers are initialised and the initialisation is visible to the CTA.
template <typename ST>
__device__ __forceinline__ void load_tile_async(ST* tile, const ST* gtile, int dk, int dv,
                                                uint64_t* mbar) {
  const int rpw = dk / kWarps;
  const uint32_t bytes = (uint32_t)(rpw * dv * (int)sizeof(ST));
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    mbar_expect_tx(&mbar[w], bytes);
    bulk_g2s(tile + (size_t)w * rpw * dv, gtile + (size_t)w * rpw * dv, bytes, &mbar[w]);
  }
}

}  // namespace rssm
