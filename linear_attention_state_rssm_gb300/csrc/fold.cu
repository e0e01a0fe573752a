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
#include "rssm_tc.cuh"

namespace rssm {

// Two consecutive checkpoint values <-> fp32 (shared loads, global stores in
// the checkpoint dtype).
__device__ __forceinline__ float2 ld_pair(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
__device__ __forceinline__ float2 ld_pair(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void st_pair(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
__device__ __forceinline__ void st_pair(__nv_bfloat16* p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}

// The tile stream of the fold. Thread tid owns the column pair (c0, c0 + 1),
// c0 = 2 (tid % (dv / 2)), and the rows rg, rg + RG, ... of every chunk
// (rg = tid / (dv / 2), RG = kThreads / (dv / 2)); it holds d~_m = f_m d_m[c]
// of both columns for the NB records in registers (zero past n) and, per
// row, adds sum_m k~_m[row] d~_m to decay(row) S[row][c], with the row's
// keys read four records at a time from hkt [dk][NB] (one load serves both
// columns); the pair goes back in the checkpoint dtype. GDN: decay e^Gam,
// f_m = hf[m]; KDA: decay egam[row] and the decayed keys, f_m = 1.
template <int ALGO, typename ST, int NB>
__device__ __forceinline__ bool fold_stream(const TilePipe<ST>& pipe, ST* gtile, int dv, int n,
                                            const float* hkt, const float* hd, const float* hf,
                                            float decay, const float* egam, int tid, int lane) {
  const int half = dv / 2;
  const int c0 = 2 * (tid % half), rg = tid / half, RG = kThreads / half;
  float d0[NB], d1[NB];
#pragma unroll
  for (int m = 0; m < NB; ++m) {
    const float f = ALGO == ALGO_GDN && m < n ? hf[m] : 1.f;
    const float2 d = m < n ? *reinterpret_cast<const float2*>(hd + m * dv + c0)
                           : make_float2(0.f, 0.f);
    d0[m] = f * d.x;
    d1[m] = f * d.y;
  }
  const int cr = pipe.tr.cr, rpc = cr / RG;  // this thread's rows per chunk
  bool ok = true;
  for (int j = 0; j < pipe.tr.nchunk; ++j) {
    // a warp stores no chunk once one of its waits has run out
    ok = __all_sync(kFull, pipe.wait_full(j) && ok);
    const ST* stg = pipe.ring + (size_t)(j % pipe.tr.ns) * cr * dv + (size_t)rg * dv + c0;
#pragma unroll 4
    for (int u = 0; u < rpc; ++u) {
      const int row = j * cr + rg + RG * u;
      const float2 sv = ld_pair(stg + (size_t)RG * u * dv);
      const float dec = ALGO == ALGO_GDN ? decay : egam[row];
      float a0 = dec * sv.x, a1 = dec * sv.y;
      const float4* kr = reinterpret_cast<const float4*>(hkt + (size_t)row * NB);
#pragma unroll
      for (int q = 0; q < NB / 4; ++q) {
        const float4 k4 = kr[q];
        a0 = fmaf(k4.x, d0[4 * q], a0);
        a1 = fmaf(k4.x, d1[4 * q], a1);
        a0 = fmaf(k4.y, d0[4 * q + 1], a0);
        a1 = fmaf(k4.y, d1[4 * q + 1], a1);
        a0 = fmaf(k4.z, d0[4 * q + 2], a0);
        a1 = fmaf(k4.z, d1[4 * q + 2], a1);
        a0 = fmaf(k4.w, d0[4 * q + 3], a0);
        a1 = fmaf(k4.w, d1[4 * q + 3], a1);
      }
      if (ok) st_pair(gtile + (size_t)row * dv + c0, a0, a1);
    }
    pipe.release(j, tid, lane);
    if (tid == 0 && ok) ok = pipe.refill(j);
  }
  return ok;
}

// Records per fold stream: n rounded up to 4, 8, 16, 32 or 64.
__host__ __device__ constexpr int fold_nb(int n) {
  return n <= 4 ? 4 : n <= 8 ? 8 : n <= 16 ? 16 : n <= 32 ? 32 : 64;
}

// NBMAX: fold_nb(L), the most records a fold of this store carries (its
// stream variants are the only ones compiled in, which keeps registers low).
template <int ALGO, typename ST, int NBMAX>
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

  ST* gtile = static_cast<ST*>(p.state) + layer * p.layer_state +
              ((size_t)s * HV + h) * (size_t)dk * dv;

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
  // 16-bit deltas widened; KDA's 16-bit keys widened (GDN's are read from
  // the landing zone when they are transposed below)
  if (p.rd_dt != DT_F32) widen16(hd, hdraw, n * dv, p.rd_dt, tid, kThreads);
  if (ALGO == ALGO_KDA && p.rk_dt != DT_F32) widen16(hk, hkraw, n * dk, p.rk_dt, tid, kThreads);
  __syncthreads();
  if (ALGO == ALGO_GDN) {
    if (warp == 0) gdn_history_scan(n, hf, scal, lane);
  } else {
    for (int ch = tid; ch < dk; ch += kThreads) {
      egam[ch] = __expf(kda_history_channel(n, dk, ch, hk, hg));
    }
    __syncthreads();
  }
  // keys transposed to [dk][NB] (zero past n) for the stream's row-wise reads
  const int NB = fold_nb(n);
  float* hkt = reinterpret_cast<float*>(smem + p.sm.hkt);
  const bool raw16 = ALGO == ALGO_GDN && p.rk_dt != DT_F32;
  for (int e = tid; e < NB * dk; e += kThreads) {
    const int m = e / dk, row = e - m * dk;
    float k = 0.f;
    if (m < n) k = raw16 ? ld_f32(hkraw, (size_t)m * dk + row, p.rk_dt) : hk[m * dk + row];
    hkt[row * NB + m] = k;
  }
  __syncthreads();
  // a chunk that did not arrive in time: no chunk from there on is stored (the
  // ones before it hold the folded state), and the copies issued are waited for
  const float decay = scal[1];
  bool ok;
  if (NB <= 4) {
    ok = fold_stream<ALGO, ST, 4>(pipe, gtile, dv, n, hkt, hd, hf, decay, egam, tid, lane);
  } else if (NB <= 8) {
    ok = fold_stream<ALGO, ST, 8>(pipe, gtile, dv, n, hkt, hd, hf, decay, egam, tid, lane);
  } else if (NBMAX <= 16 || NB <= 16) {
    ok = fold_stream<ALGO, ST, 16>(pipe, gtile, dv, n, hkt, hd, hf, decay, egam, tid, lane);
  } else if (NBMAX <= 32 || NB <= 32) {
    ok = fold_stream<ALGO, ST, (NBMAX < 32 ? 16 : 32)>(pipe, gtile, dv, n, hkt, hd, hf, decay,
                                                       egam, tid, lane);
  } else {
    ok = fold_stream<ALGO, ST, (NBMAX < 64 ? 16 : 64)>(pipe, gtile, dv, n, hkt, hd, hf, decay,
                                                       egam, tid, lane);
  }
  if (!__syncthreads_and(ok) && tid == 0) {
    atomicOr(p.err, DEVERR_TIMEOUT);
    pipe.drain_tail();
  }
}

// GDN fold on the 5th-generation tensor cores (128 value columns, at most 32
// records; same rows, records and timeout behaviour as fold_kernel):
//     S^T <- e^Gam S^T + (F D)^T K     (F D)[m][col] = f_m d_m[col], K[m][row] = k_m[row]
// The rank-n product does not depend on S: it is computed 32 rows at a time
// (a quarter of the tile, two tensor-memory buffers, each quarter issued as
// soon as its buffer is free) by kind::tf32 MMAs with (F D)^T in tensor memory
// (tf32 hi/lo) and the keys K-major in shared memory (16-bit keys exact, fp32
// keys as hi/lo). The tile streams through the ring once: thread tid (value
// column tid) adds e^Gam S from the stage to the product of its rows and stores
// the rows. A wait that runs out stops the stores from that chunk on.
constexpr int kFoldQuarter = 32;  // rows per fold product

template <typename ST>
__device__ __forceinline__ void fold_tc_issue(uint32_t tbase, const float* bf, const float* bl,
                                              int K, int dk, int quarter, uint64_t* bar) {
  constexpr uint32_t idesc = tf32_idesc(128, kFoldQuarter);
  const uint32_t lbo = (uint32_t)(dk / 8) * 128u;  // 4 records further along K
  const uint32_t d = tbase + (uint32_t)(quarter & 1) * kFoldQuarter;
  const uint32_t boff = (uint32_t)quarter * (kFoldQuarter / 8) * 128u;
  for (int kk = 0; kk < K / 8; ++kk) {
    const uint32_t off = boff + (uint32_t)(2 * kk) * lbo;
    const uint64_t bh = kmajor_desc(smem_addr(bf) + off, lbo, 128u);
    const uint32_t ah = tbase + 64 + 8 * kk, al = ah + K;
    mma_ts(d, ah, bh, idesc, kk > 0);
    mma_ts(d, al, bh, idesc, true);
    if (bl != nullptr) mma_ts(d, ah, kmajor_desc(smem_addr(bl) + off, lbo, 128u), idesc, true);
  }
  mma_commit(bar);
}

template <typename ST>
__global__ void __launch_bounds__(kThreads) fold_tc_kernel(const FoldParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int h = blockIdx.x, r = blockIdx.y, layer = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dk = p.dk, dv = p.dv, L = p.L, HV = p.HV;
  constexpr int DV = 128;

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
  const int K = (n + 7) & ~7;  // records, padded to whole MMA steps

  ST* gtile = static_cast<ST*>(p.state) + layer * p.layer_state +
              ((size_t)s * HV + h) * (size_t)dk * dv;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + p.sm.mbar);
  float* hd = reinterpret_cast<float*>(smem + p.sm.hd);
  float* hf = reinterpret_cast<float*>(smem + p.sm.hf);
  float* scal = reinterpret_cast<float*>(smem + p.sm.scal);
  float* bf = reinterpret_cast<float*>(smem + p.sm.bf);
  float* bl = p.rk_dt == DT_F32 ? reinterpret_cast<float*>(smem + p.sm.bl) : nullptr;
  unsigned char* hkraw = smem + p.sm.hkraw;
  unsigned char* hdraw = smem + p.sm.hdraw;
  uint64_t* fbar = &mbar[kMbarAFull];   // [2] fold product of a quarter done
  uint64_t* dfree = &mbar[kMbarAEmpty];  // [2] every warp has read a quarter's product
  uint32_t* tslot = reinterpret_cast<uint32_t*>(&mbar[kMbarTmem]);

  const size_t kbase = layer * p.layer_k + ((size_t)s * HV + h) * L * dk;
  const size_t dbase = layer * p.layer_d + ((size_t)s * HV + h) * L * dv;
  const size_t gbase = layer * p.layer_g + ((size_t)s * HV + h) * L;

  const TilePipe<ST> pipe(reinterpret_cast<ST*>(smem + p.sm.ring), mbar, gtile, dk, dv, kStages,
                          p.hook);
  constexpr unsigned long long lim = kWaitLimitNs;
  if (tid == 0) {
    mbar_init(&mbar[kMbarWin], 1);
    mbar_init(&mbar[kMbarHist], 1);
    pipe.init();
    for (int b = 0; b < 2; ++b) {
      mbar_init(&fbar[b], 1);
      mbar_init(&dfree[b], kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    pipe.prime();
    issue_history<ALGO_GDN>(n, dk, dv, p.ring_k, kbase, p.rk_dt, hkraw, p.ring_d, dbase, p.rd_dt,
                            p.rd_dt == DT_F32 ? static_cast<void*>(hd) : hdraw, p.ring_g, gbase,
                            nullptr, &mbar[kMbarHist], p.hook.extra(WH_HIST));
  }
  for (int m = tid; m < n; m += kThreads) hf[m] = p.ring_g[gbase + m];
  if (!__syncthreads_and(mbar_wait_bounded(&mbar[kMbarHist], 0, lim))) {
    if (tid == 0) {
      atomicOr(p.err, DEVERR_TIMEOUT);
      mbar_wait_bounded(&mbar[kMbarHist], 0, lim);
      pipe.drain();
    }
    return;
  }
  if (p.rd_dt != DT_F32) widen16(hd, hdraw, n * dv, p.rd_dt, tid, kThreads);
  // fold keys, K-major [K records x dk rows]; records >= n are zero
  for (int e = tid; e < K * dk; e += kThreads) {
    const int row = e % dk, m = e / dk;
    const float k = m < n ? ld_f32(hkraw, (size_t)m * dk + row, p.rk_dt) : 0.f;
    const uint32_t off = kmajor_off(row, m, dk / 8) >> 2;
    bf[off] = bl != nullptr ? tf32_hi(k) : k;
    if (bl != nullptr) bl[off] = k - tf32_hi(k);
  }
  fence_async_smem();
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tslot);
  }
  __syncthreads();
  if (warp == 0) gdn_history_scan(n, hf, scal, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t ta = tmem_lane(tbase, warp);
  // (F D)^T: lane col holds f_m d_m[col] (hi at column 64 + m, lo at 64 + K + m)
  for (int m0 = 0; m0 < K; m0 += 16) {
    float hi[16], lo[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int m = m0 + i;
      const float a = m < n ? hf[m] * hd[m * dv + tid] : 0.f;
      hi[i] = tf32_hi(a);
      lo[i] = a - hi[i];
    }
    // K is a multiple of 8: a last half block stores its first 8 columns only
    if (m0 + 16 <= K) {
      tmem_st16(ta + 64 + m0, hi);
      tmem_st16(ta + 64 + K + m0, lo);
    } else {
      float h8[8], l8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        h8[i] = hi[i];
        l8[i] = lo[i];
      }
      tmem_st8(ta + 64 + m0, h8);
      tmem_st8(ta + 64 + K + m0, l8);
    }
  }
  tmem_st_wait();
  tc_fence_before();
  __syncthreads();
  const int nq = dk / kFoldQuarter;
  if (tid == 0) {
    tc_fence_after();
    fold_tc_issue<ST>(tbase, bf, bl, K, dk, 0, &fbar[0]);
    if (nq > 1) fold_tc_issue<ST>(tbase, bf, bl, K, dk, 1, &fbar[1]);
  }
  const float eg = scal[1];
  const int cr = pipe.tr.cr;  // 16 (fp32) or 32 (bf16) rows per chunk
  bool ok = true;
  for (int j = 0; j < pipe.tr.nchunk; ++j) {
    const int r0 = j * cr, q = r0 / kFoldQuarter, b = q & 1, o = r0 % kFoldQuarter;
    ok = __all_sync(kFull, pipe.wait(j) && ok);
    if (o == 0) {
      ok = __all_sync(kFull, mbar_wait_bounded(&fbar[b], (uint32_t)((q >> 1) & 1)) && ok);
      tc_fence_after();
    }
    const ST* stg = pipe.stage(j);
    const uint32_t dcol = ta + (uint32_t)(b * kFoldQuarter + o);
    for (int u = 0; u < cr; u += 16) {
      float d[16];
      __syncwarp();
      tmem_ld16(dcol + u, d);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float v = fmaf(eg, tc_f32(stg[(u + i) * DV + tid]), d[i]);
        if (ok) gtile[(size_t)(r0 + u + i) * DV + tid] = tc_st<ST>(v);
      }
    }
    ok = pipe.done(j, tid, lane, ok) && ok;
    if (o + cr == kFoldQuarter) {
      // quarter q has been read: its buffer takes quarter q + 2
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dfree[b]);
      if (tid == 0 && q + 2 < nq) {
        ok = mbar_wait_bounded(&dfree[b], (uint32_t)((q >> 1) & 1)) && ok;
        tc_fence_after();
        fold_tc_issue<ST>(tbase, bf, bl, K, dk, q + 2, &fbar[b]);
      }
    }
  }
  if (!__syncthreads_and(ok) && tid == 0) {
    atomicOr(p.err, DEVERR_TIMEOUT);
    pipe.drain_tail();
  }
  // the last quarters' products were read (their waits precede the loads)
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase);
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
  if constexpr (ALGO == ALGO_GDN) {
    if (p.tc) {
      fold_tc_kernel<ST><<<grid, kThreads, p.sm.total, st>>>(p);
      return cudaGetLastError();
    }
  }
  if (p.L <= 16) {
    fold_kernel<ALGO, ST, 16><<<grid, kThreads, p.sm.total, st>>>(p);
  } else if (p.L <= 32) {
    fold_kernel<ALGO, ST, 32><<<grid, kThreads, p.sm.total, st>>>(p);
  } else {
    fold_kernel<ALGO, ST, 64><<<grid, kThreads, p.sm.total, st>>>(p);
  }
  return cudaGetLastError();
}

template <int ALGO, typename ST, int NBMAX>
static cudaError_t fold_prepare_nb(int max_smem) {
  const cudaError_t e = cudaFuncSetAttribute(fold_kernel<ALGO, ST, NBMAX>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fold_kernel<ALGO, ST, NBMAX>,
                              cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

template <int ALGO, typename ST>
static cudaError_t fold_prepare_t(int max_smem) {
  cudaError_t e;
  if constexpr (ALGO == ALGO_GDN) {
    e = cudaFuncSetAttribute(fold_tc_kernel<ST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             max_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fold_tc_kernel<ST>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             100);
    if (e != cudaSuccess) return e;
  }
  if ((e = fold_prepare_nb<ALGO, ST, 16>(max_smem)) != cudaSuccess) return e;
  if ((e = fold_prepare_nb<ALGO, ST, 32>(max_smem)) != cudaSuccess) return e;
  return fold_prepare_nb<ALGO, ST, 64>(max_smem);
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
