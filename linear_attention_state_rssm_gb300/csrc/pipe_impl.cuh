// Pipelined replay kernel: decode and speculative verify of one layer for
// Gated DeltaNet heads of 128 x 128, the ring-overflow fold fused in, as one
// persistent CTA per SM that walks a list of (request row, value head) items.
//
// What it computes is what the per-row replay kernel computes (replay_impl.cuh,
// after LightLLM PR #1690 "feat: add ReplaySSM state modes for GDN and KDA" and
// SGLang fork PR jianc99/sglang#2): per item, with c = cursor, fold = force ||
// c + T > L, the checkpoint S0 and the c history records give the replayed
// state S~ = e^Gam S0 + sum_m f_m k_m d_m^T (f_m = e^{Gam - Gam_m}); a folding
// item stores S~ back as the checkpoint; the window of T tokens is solved in
// the (I + A)^-1 form with every sum over j <= i only (a NaN or Inf at a later,
// rejected, position never reaches an earlier output), and its records go to
// ring positions base + i (base = fold ? 0 : c).
//
// How the work is laid out. A CTA of the per-row kernel spends most of its
// life outside the checkpoint stream (window set-up, window solve), and with
// three or four CTAs per SM the stream of one is not enough to keep HBM busy.
// Here the three kinds of work run on separate warps, one item apart:
//  - warp 8 (one thread) issues the 8 KB checkpoint chunks of item after item
//    into a ring of up to 16 stages, so the SM's stream never stops at an item
//    boundary;
//  - warps 0-3 ("math") consume the chunks on the tensor cores: for a folding
//    item S^T <- e^Gam S^T + D~^T K (D~ = f_m d_m, stored back), then the
//    mat-vec Y^T = S^T X for the 2T window vectors (X = raw k_i, q_i); for an
//    item with history that does not fold, Y^T <- e^Gam Y^T + D~^T H with
//    H = K X the history dots (the correction term of the replayed state);
//  - warps 4-7 ("prep") prepare item k + 1 (gate scans, X and D~ in fragment
//    order, fold keys or H, the window coefficients A and F) while the math
//    warps stream item k, then solve item k - 1 per value column (outputs and
//    records), and issue the window and history copies of item k + 2.
// Items are dealt round-robin from one order that every CTA computes alike:
// folding rows first, so every CTA gets an equal share of the heavier items.
// Each product uses warp-level mma.sync m16n8k8 with tf32 operands and fp32
// accumulation; fp32 operands are split into tf32 head and tail (hi*hi +
// hi*lo + lo*hi), 16-bit values are exact in tf32 and take one product.
//
// Waits: every mbarrier wait is bounded (the launch's limit) and also gives up
// once another role has given up (abort word). A CTA whose wait ran out sets
// RSSM_DEVERR_TIMEOUT and processes no further item: the rows of those items
// are left untouched; the item in progress writes no output or record (a
// folding item may have stored the chunks it had folded). Before the CTA
// leaves, every copy it issued is waited for again (bounded).
#pragma once

#include <type_traits>

#include "rssm_common.cuh"
#include "rssm_history.cuh"
#include "rssm_mma.cuh"

namespace rssm {

enum : int { PF_LIVE = 1, PF_FOLD = 2 };
constexpr int kPipeDK = 128, kPipeDV = 128;
constexpr int kPipeGroups = kPipeMaxRows / 32;

// Bounded wait that also returns false once the CTA's abort word is set.
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long lim, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > lim) return false;
  }
}

// AND of `pred` over the `count` threads that name barrier `id`.
__device__ __forceinline__ bool named_and(int id, int count, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

// Four consecutive values of a 16-bit or fp32 array in shared memory as fp32.
__device__ __forceinline__ float4 ld4_as_f32(const void* base, int i, int dt) {
  if (dt == DT_F32) return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
  const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + i);
  float2 a, b;
  if (dt == DT_BF16) {
    a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  } else {
    a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  }
  return make_float4(a.x, a.y, b.x, b.y);
}

// Two consecutive values as fp32 (i even).
__device__ __forceinline__ float2 ld2_as_f32(const void* base, int i, int dt) {
  if (dt == DT_F32) return *reinterpret_cast<const float2*>(static_cast<const float*>(base) + i);
  const uint32_t u = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(base) + i);
  if (dt == DT_BF16) return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

// ---------------------------------------------------------------- math warps
// One item's stream on math warp `warp` (columns 32 warp + 4g .. + 3 of every
// eight-row step, rows 2t and 2t + 1; see stream_mma in replay_impl.cuh for
// the fragment relabelling this shares). q is the global index of the item's
// first chunk. Returns false if a wait gave up (the item is then abandoned:
// nothing more is stored, the stages it did not release stay held).
template <typename ST, int NTN, bool EXACT_X, bool EXACT_K>
__device__ __forceinline__ bool pipe_stream(const PipeItem& I, const ST* ring, uint64_t* mb, int NS,
                                            int q, const float* xf, const float* kf,
                                            const float* dfp, const float* hh, ST* gtile,
                                            unsigned long long lim, const volatile int* abort,
                                            int warp, int lane, float (&y)[16]) {
  constexpr int DV = kPipeDV, DK = kPipeDK;
  constexpr int CR = kChunkBytes / (DV * (int)sizeof(ST));  // rows per chunk
  constexpr int NCH = DK / CR;
  constexpr bool EXACT_S = !std::is_same<ST, float>::value;
  const int g = lane >> 2, t = lane & 3, col = 32 * warp + 4 * g;
  const bool fold = I.fold != 0;
  const int n = I.n, nkq = n > 8 ? 2 : (n > 0 ? 1 : 0);
  const float decay = I.egam;
  // f_m d_m as A fragments [m-tile][record block][4] (zero past the history)
  Tf32 df[2][2][4];
  if (n > 0) {
    const float4* d4 = reinterpret_cast<const float4*>(dfp) + (warp * 32 + lane) * 4;
#pragma unroll
    for (int mk = 0; mk < 4; ++mk) {
      const float4 v = d4[mk];
      df[mk >> 1][mk & 1][0] = tf32_split<false>(v.x);
      df[mk >> 1][mk & 1][1] = tf32_split<false>(v.y);
      df[mk >> 1][mk & 1][2] = tf32_split<false>(v.z);
      df[mk >> 1][mk & 1][3] = tf32_split<false>(v.w);
    }
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) y[e] = 0.f;
  const float4* kf4 = reinterpret_cast<const float4*>(kf);
  for (int j = 0; j < NCH; ++j, ++q) {
    const int st = q % NS;
    if (!__all_sync(kFull, pipe_wait(&mb[PB_FULL + st], (uint32_t)((q / NS) & 1), lim, abort)))
      return false;
    const ST* stg = ring + (size_t)st * CR * DV;
#pragma unroll 2
    for (int kb = 0; kb < CR; kb += 8) {
      const int r0 = j * CR + kb + 2 * t;        // this lane's tile rows r0, r0 + 1
      const int fi = ((j * CR + kb) >> 3) * 32 + lane;
      float s0[4], s1[4];
      ld_cols<ST, 4>(stg + (size_t)(kb + 2 * t) * DV + col, s0);
      ld_cols<ST, 4>(stg + (size_t)(kb + 2 * t + 1) * DV + col, s1);
      if (fold) {
        const float4 k4 = kf4[fi];  // row j*CR + kb + g: records t, t + 4, 8 + t, 12 + t
        const Tf32 kb0[2] = {tf32_split<EXACT_K>(k4.x), tf32_split<EXACT_K>(k4.y)};
        const Tf32 kb1[2] = {tf32_split<EXACT_K>(k4.z), tf32_split<EXACT_K>(k4.w)};
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          float c[4] = {decay * s0[2 * mt], decay * s1[2 * mt], decay * s0[2 * mt + 1],
                        decay * s1[2 * mt + 1]};
          if (nkq > 0) mma_split<false, EXACT_K>(c, df[mt][0], kb0);
          if (nkq > 1) mma_split<false, EXACT_K>(c, df[mt][1], kb1);
          s0[2 * mt] = c[0];
          s1[2 * mt] = c[1];
          s0[2 * mt + 1] = c[2];
          s1[2 * mt + 1] = c[3];
        }
        // the mat-vec takes the stored (rounded) checkpoint values
        st_cols<ST, 4>(gtile + (size_t)r0 * DV + col, s0);
        st_cols<ST, 4>(gtile + (size_t)(r0 + 1) * DV + col, s1);
      }
      Tf32 xb[NTN][2];
      if constexpr (NTN == 2) {
        const float4 x4 = reinterpret_cast<const float4*>(xf)[fi];
        xb[0][0] = tf32_split<EXACT_X>(x4.x);
        xb[0][1] = tf32_split<EXACT_X>(x4.y);
        xb[NTN - 1][0] = tf32_split<EXACT_X>(x4.z);
        xb[NTN - 1][1] = tf32_split<EXACT_X>(x4.w);
      } else {
        const float2 x2 = reinterpret_cast<const float2*>(xf)[fi];
        xb[0][0] = tf32_split<EXACT_X>(x2.x);
        xb[0][1] = tf32_split<EXACT_X>(x2.y);
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int h2 = 2 * mt;
        const Tf32 af[4] = {tf32_split<EXACT_S>(s0[h2]), tf32_split<EXACT_S>(s0[h2 + 1]),
                            tf32_split<EXACT_S>(s1[h2]), tf32_split<EXACT_S>(s1[h2 + 1])};
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
          float(&c)[4] = *reinterpret_cast<float(*)[4]>(&y[4 * (NTN * mt + nt)]);
          mma_split<EXACT_S, EXACT_X>(c, af, xb[nt]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&mb[PB_FULL + NS + st]);  // stage released
  }
  if (!fold && n > 0) {
    // replayed state of a window that does not fold: e^Gam S0^T x + sum_m f_m d_m (k_m . x)
#pragma unroll
    for (int e = 0; e < 16; ++e) y[e] *= decay;
#pragma unroll
    for (int kq = 0; kq < 2; ++kq) {
      if (kq < nkq) {
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
          const Tf32 hb[2] = {tf32_split<false>(hh[(8 * kq + t) * kPipeHist + 8 * nt + g]),
                              tf32_split<false>(hh[(8 * kq + t + 4) * kPipeHist + 8 * nt + g])};
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            float(&c)[4] = *reinterpret_cast<float(*)[4]>(&y[4 * (NTN * mt + nt)]);
            mma_split<false, false>(c, df[mt][kq], hb);
          }
        }
      }
    }
  }
  return true;
}

// ---------------------------------------------------------------- kernel
template <int ALGO, typename ST, int NT>
__global__ void __launch_bounds__(kPipeThreads, 1)
    pipe_kernel(const ReplayParams p, const PipeSmem sm) {
  static_assert(ALGO == ALGO_GDN, "the pipelined kernel serves GDN heads");
  constexpr int DK = kPipeDK, DV = kPipeDV, NTN = pipe_ntn(NT), NV = 2 * NT;
  constexpr int CR = kChunkBytes / (DV * (int)sizeof(ST));
  constexpr int NCH = DK / CR;
  constexpr int PT = 32 * kPipePrep;       // prep threads
  constexpr int kPrepBar = 1;              // named barrier of the prep warps
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, T = p.T, L = p.L, HV = p.HV, NS = sm.ns;
  const unsigned long long lim = p.hook.limit_ns;
  uint64_t* mb = reinterpret_cast<uint64_t*>(smem + sm.mbar);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + sm.mbar + 8 * kPipeMbars);
  int* r_slot = reinterpret_cast<int*>(smem + sm.rows);
  int* r_cur = r_slot + sm.maxb;
  int* r_order = r_cur + sm.maxb;
  int* r_flag = r_order + sm.maxb;
  int* gcnt = r_flag + sm.maxb;  // [2][kPipeGroups]: folding / other live rows per group
  ST* ring = reinterpret_cast<ST*>(smem + sm.ring);

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&mb[PB_WIN + b], 1);
      mbar_init(&mb[PB_PREP + b], 1);
      mbar_init(&mb[PB_MATH + b], kPipeMath);
      mbar_init(&mb[PB_YFREE + b], 1);
    }
    for (int st = 0; st < NS; ++st) {
      mbar_init(&mb[PB_FULL + st], 1);
      mbar_init(&mb[PB_FULL + NS + st], kPipeMath);
    }
    *abort = 0;
    fence_mbar_init();
  }

  // ---- rows: slot, cursor and fold decision of every request row, then one
  //      order shared by every CTA: folding rows first, each group by row
  const int ngrp = sm.maxb / 32;
  for (int r = tid; r < sm.maxb; r += kPipeThreads) {
    int s = -1, c = 0, f = 0;
    if (r < B) {
      s = p.slot[r];
      if (s >= p.n_slots) {
        if (blockIdx.x == 0) atomicOr(p.err, DEVERR_SLOT);
        s = -1;
      } else if (s >= 0) {
        c = p.cursor[s];
        if (c < 0 || c > L) {
          if (blockIdx.x == 0) atomicOr(p.err, DEVERR_CURSOR);
          s = -1;
        } else {
          const bool fl = (p.force != nullptr && p.force[r] != 0) || c + T > L;
          f = PF_LIVE | (fl ? PF_FOLD : 0);
        }
      }
    }
    r_slot[r] = s;
    r_cur[r] = c;
    r_flag[r] = f;
  }
  __syncthreads();
  for (int gi = warp; gi < ngrp; gi += kPipeThreads / 32) {
    const int f = r_flag[gi * 32 + lane];
    const unsigned mf = __ballot_sync(kFull, f == (PF_LIVE | PF_FOLD));
    const unsigned mo = __ballot_sync(kFull, f == PF_LIVE);
    if (lane == 0) {
      gcnt[gi] = __popc(mf);
      gcnt[kPipeGroups + gi] = __popc(mo);
    }
  }
  __syncthreads();
  int nfold = 0, nlive = 0;
  for (int gi = 0; gi < ngrp; ++gi) {
    nfold += gcnt[gi];
    nlive += gcnt[gi] + gcnt[kPipeGroups + gi];
  }
  for (int gi = warp; gi < ngrp; gi += kPipeThreads / 32) {
    const int r = gi * 32 + lane, f = r_flag[r];
    const unsigned mf = __ballot_sync(kFull, f == (PF_LIVE | PF_FOLD));
    const unsigned mo = __ballot_sync(kFull, f == PF_LIVE);
    const unsigned lt = (1u << lane) - 1u;
    if (f & PF_LIVE) {
      int rank = (f & PF_FOLD) ? __popc(mf & lt) : nfold + __popc(mo & lt);
      for (int g2 = 0; g2 < gi; ++g2) rank += (f & PF_FOLD) ? gcnt[g2] : gcnt[kPipeGroups + g2];
      r_order[rank] = r;
    }
  }
  __syncthreads();
  const int n_items = nlive * HV;
  const int P = gridDim.x, b0 = blockIdx.x;
  const int nk = b0 < n_items ? (n_items - b0 + P - 1) / P : 0;
  auto item_of = [&](int k, int& row, int& h) {
    const int i = b0 + k * P;
    row = r_order[i / HV];
    h = i - (i / HV) * HV;
  };

  if (warp == kPipeProd) {
    // ================= producer: checkpoint chunks of every item, in order
    int q = 0;
    if (lane == 0) {
      bool ok = true;
      for (int k = 0; ok && k < nk; ++k) {
        int row, h;
        item_of(k, row, h);
        const ST* tile = static_cast<const ST*>(p.state) + ((size_t)r_slot[row] * HV + h) * DK * DV;
        for (int j = 0; j < NCH; ++j) {
          const int st = q % NS;
          if (q >= NS &&
              !pipe_wait(&mb[PB_FULL + NS + st], (uint32_t)(((q / NS) - 1) & 1), lim, abort)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&mb[PB_FULL + st],
                         (uint32_t)kChunkBytes + (k == 0 ? p.hook.extra(WH_CHUNK0 + j) : 0u));
          bulk_g2s(ring + (size_t)st * CR * DV, tile + (size_t)j * CR * DV, kChunkBytes,
                   &mb[PB_FULL + st]);
          ++q;
        }
      }
      if (!ok && !*abort) {
        *abort = 1;
        atomicOr(p.err, DEVERR_TIMEOUT);
      }
    }
    __syncwarp();
    __syncthreads();
    // every chunk issued has landed before the CTA leaves (bounded)
    if (lane == 0) {
      for (int qq = q > NS ? q - NS : 0; qq < q; ++qq)
        mbar_wait_bounded(&mb[PB_FULL + qq % NS], (uint32_t)((qq / NS) & 1), lim);
    }
    return;
  }

  if (warp < kPipeMath) {
    // ================= math: stream every item's tile on the tensor cores
    const bool xk = p.in_dt != DT_F32, kk = p.rk_dt != DT_F32;
    int q = 0;
    for (int k = 0; k < nk; ++k) {
      const int b = k & 1;
      if (!__all_sync(kFull, pipe_wait(&mb[PB_PREP + b], (uint32_t)((k >> 1) & 1), lim, abort))) {
        if (lane == 0 && !*abort) {
          *abort = 1;
          atomicOr(p.err, DEVERR_TIMEOUT);
        }
        break;
      }
      const PipeItem& I = *reinterpret_cast<const PipeItem*>(smem + sm.item[b]);
      ST* gtile = static_cast<ST*>(p.state) + ((size_t)I.s * HV + I.h) * DK * DV;
      const float* xf = reinterpret_cast<const float*>(smem + sm.xf[b]);
      const float* kf = reinterpret_cast<const float*>(smem + sm.kf[b]);
      const float* dfp = reinterpret_cast<const float*>(smem + sm.df[b]);
      const float* hh = reinterpret_cast<const float*>(smem + sm.hh[b]);
      float y[16];
      bool ok;
      if (xk) {
        ok = kk ? pipe_stream<ST, NTN, true, true>(I, ring, mb, NS, q, xf, kf, dfp, hh, gtile, lim,
                                                   abort, warp, lane, y)
                : pipe_stream<ST, NTN, true, false>(I, ring, mb, NS, q, xf, kf, dfp, hh, gtile,
                                                    lim, abort, warp, lane, y);
      } else {
        ok = kk ? pipe_stream<ST, NTN, false, true>(I, ring, mb, NS, q, xf, kf, dfp, hh, gtile,
                                                    lim, abort, warp, lane, y)
                : pipe_stream<ST, NTN, false, false>(I, ring, mb, NS, q, xf, kf, dfp, hh, gtile,
                                                     lim, abort, warp, lane, y);
      }
      q += NCH;
      // the column sums of item k - 2 (same buffer) have been read
      if (ok && k >= 2)
        ok = __all_sync(kFull,
                        pipe_wait(&mb[PB_YFREE + b], (uint32_t)(((k >> 1) - 1) & 1), lim, abort));
      if (!ok) {
        if (lane == 0 && !*abort) {
          *abort = 1;
          atomicOr(p.err, DEVERR_TIMEOUT);
        }
        break;
      }
      float* yo = reinterpret_cast<float*>(smem + sm.y[b]);
      const int g = lane >> 2, t = lane & 3;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
          const int c0 = 32 * warp + 4 * g + 2 * mt, v = 8 * nt + 2 * t;
          const float* c = &y[4 * (NTN * mt + nt)];
          if (v < NV) {
            yo[v * DV + c0] = c[0];
            yo[v * DV + c0 + 1] = c[2];
          }
          if (v + 1 < NV) {
            yo[(v + 1) * DV + c0] = c[1];
            yo[(v + 1) * DV + c0 + 1] = c[3];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&mb[PB_MATH + b]);
    }
    __syncthreads();
    return;
  }

  // ================= prep warps: prepare item k, solve item k - 1
  const int pt = tid - 32 * kPipeMath, pw = pt >> 5;
  const int s_in = dtype_bytes(p.in_dt);
  const uint32_t qrow = (uint32_t)(DK * s_in);
  int kw = 0;  // windows issued (by prep thread 0)
  auto issue_window = [&](int k) {
    int row, h;
    item_of(k, row, h);
    const int b = k & 1, s = r_slot[row], n = r_cur[row];
    const size_t tok0 = (size_t)row * T;
    const int kh = h / p.G;
    unsigned char* wr = smem + sm.wraw[b];
    const int sk = dtype_bytes(p.rk_dt), sd = dtype_bytes(p.rd_dt);
    uint32_t bytes = 2u * T * qrow;
    if (n > 0) bytes += (uint32_t)(n * (DK * sk + DV * sd) + 4 * round4(n));
    const uint32_t extra =
        k == 0 ? p.hook.extra(WH_WINDOW) + (n > 0 ? p.hook.extra(WH_HIST) : 0u) : 0u;
    mbar_expect_tx(&mb[PB_WIN + b], bytes + extra);
    for (int i = 0; i < T; ++i) {
      const size_t off = ((tok0 + i) * p.HK + kh) * (size_t)qrow;
      bulk_g2s(wr + i * qrow, static_cast<const char*>(p.q) + off, qrow, &mb[PB_WIN + b]);
      bulk_g2s(wr + (T + i) * qrow, static_cast<const char*>(p.k) + off, qrow, &mb[PB_WIN + b]);
    }
    if (n > 0) {
      const size_t sh = (size_t)s * HV + h;
      bulk_g2s(smem + sm.hkr[b], static_cast<const char*>(p.ring_k) + sh * L * DK * sk,
               (uint32_t)(n * DK * sk), &mb[PB_WIN + b]);
      bulk_g2s(smem + sm.hdr[b], static_cast<const char*>(p.ring_d) + sh * L * DV * sd,
               (uint32_t)(n * DV * sd), &mb[PB_WIN + b]);
      bulk_g2s(smem + sm.hgr[b], p.ring_g + sh * L, (uint32_t)(4 * round4(n)), &mb[PB_WIN + b]);
    }
  };
  if (pt == 0) {
    for (; kw < 2 && kw < nk; ++kw) issue_window(kw);
  }
  __syncwarp();
  bool alive = true;  // no wait of the prep warps has run out
  int nprep = 0;      // items prepared (handed to the math warps)
  for (int k = 0; k <= nk; ++k) {
    // ---- prepare item k
    if (named_and(kPrepBar, PT, alive && k < nk && !*abort)) {
      const int b = k & 1;
      int row, h;
      item_of(k, row, h);
      const int s = r_slot[row], c = r_cur[row];
      const bool fold = (r_flag[row] & PF_FOLD) != 0;
      const int n = c;
      const size_t tok0 = (size_t)row * T;
      PipeItem& I = *reinterpret_cast<PipeItem*>(smem + sm.item[b]);
      float bet = 0.f, gw = 0.f;
      if (pt < T) {
        bet = p.beta[(tok0 + pt) * HV + h];
        gw = p.g[(tok0 + pt) * HV + h];
      }
      const bool landed = named_and(kPrepBar, PT,
                                    pipe_wait(&mb[PB_WIN + b], (uint32_t)((k >> 1) & 1), lim,
                                              abort));
      if (!landed) {
        if (pt == 0 && !*abort) {
          *abort = 1;
          atomicOr(p.err, DEVERR_TIMEOUT);
        }
        __syncwarp();
        alive = false;
      } else {
        const unsigned char* wr = smem + sm.wraw[b];
        const void* wq = wr;                      // q rows [T][dk]
        const void* wkr = wr + T * qrow;          // k rows [T][dk]
        float* xf = reinterpret_cast<float*>(smem + sm.xf[b]);
        // P1 (prep warp 0): gates, item scalars
        if (pw == 0) {
          const float* hg = reinterpret_cast<const float*>(smem + sm.hgr[b]);
          // history: hf[m] = e^{sum_{m' > m} g_m'} (n <= 16 records: one pass)
          const int m = n - 1 - lane;
          float incl = (m >= 0) ? hg[m] : 0.f;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float tv = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += tv;
          }
          float excl = __shfl_up_sync(kFull, incl, 1);
          if (lane == 0) excl = 0.f;
          if (lane < kPipeHist) I.hf[lane] = 0.f;
          __syncwarp();
          if (m >= 0) I.hf[m] = __expf(excl);
          const float gam = __shfl_sync(kFull, incl, 31);
          // window: inclusive gate prefixes G_i
          float gi = lane < T ? gw : 0.f;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float tv = __shfl_up_sync(kFull, gi, off);
            if (lane >= off) gi += tv;
          }
          if (lane < kPipeMaxNT) {
            I.G[lane] = lane < T ? gi : 0.f;
            I.eG[lane] = lane < T ? __expf(gi) : 0.f;
            I.beta[lane] = lane < T ? bet : 0.f;
          }
          if (lane == 0) {
            I.row = row;
            I.h = h;
            I.s = s;
            I.c = c;
            I.base = fold ? 0 : c;
            I.fold = fold ? 1 : 0;
            I.n = n;
            I.egam = __expf(gam);
          }
        }
        // P2 (all prep threads): mat-vec inputs in fragment order
        for (int e = pt; e < DK * 8 * NTN; e += PT) {
          int ch, v;
          x_slot<NTN>(e, ch, v);
          const int i = v < NT ? v : v - NT;
          float x = 0.f;
          if (v < NV && i < T) x = ld_f32(v < NT ? wkr : wq, (size_t)i * DK + ch, p.in_dt);
          xf[e] = x;
        }
        named_sync(kPrepBar, PT);
        // P3: window coefficients, one warp per pair (j <= i < T)
        {
          int pi = 0;
          for (int i = 0; i < T; ++i) {
            for (int j = 0; j <= i; ++j, ++pi) {
              if (pi % kPipePrep != pw) continue;
              const float4 kj = ld4_as_f32(wkr, j * DK + 4 * lane, p.in_dt);
              const float4 ki = ld4_as_f32(wkr, i * DK + 4 * lane, p.in_dt);
              const float4 qi = ld4_as_f32(wq, i * DK + 4 * lane, p.in_dt);
              float skk = fmaf(kj.x, ki.x, fmaf(kj.y, ki.y, fmaf(kj.z, ki.z, kj.w * ki.w)));
              float skq = fmaf(kj.x, qi.x, fmaf(kj.y, qi.y, fmaf(kj.z, qi.z, kj.w * qi.w)));
              skk = warp_sum(skk);
              skq = warp_sum(skq);
              if (lane == 0) {
                const float wgt = __expf(I.G[i] - I.G[j]);
                I.fm[i * kPipeMaxNT + j] = wgt * skq;
                I.am[i * kPipeMaxNT + j] = j < i ? I.beta[i] * wgt * skk : 0.f;
              }
            }
          }
        }
        // P4: history operands. f_m d_m in the math lanes' A-fragment order
        if (n > 0) {
          float* dfp = reinterpret_cast<float*>(smem + sm.df[b]);
          const void* hd = smem + sm.hdr[b];
          const int w = pt >> 5, l = pt & 31, g = l >> 2, t = l & 3;
          float v16[16];
#pragma unroll
          for (int mk = 0; mk < 4; ++mk) {
            const int mt = mk >> 1, kq = mk & 1, c0 = 32 * w + 4 * g + 2 * mt;
            const int m0 = 8 * kq + t, m1 = m0 + 4;
            float2 d0 = make_float2(0.f, 0.f), d1 = make_float2(0.f, 0.f);
            if (m0 < n) d0 = ld2_as_f32(hd, m0 * DV + c0, p.rd_dt);
            if (m1 < n) d1 = ld2_as_f32(hd, m1 * DV + c0, p.rd_dt);
            const float f0 = m0 < n ? I.hf[m0] : 0.f, f1 = m1 < n ? I.hf[m1] : 0.f;
            v16[4 * mk + 0] = f0 * d0.x;
            v16[4 * mk + 1] = f0 * d0.y;
            v16[4 * mk + 2] = f1 * d1.x;
            v16[4 * mk + 3] = f1 * d1.y;
          }
          float4* o4 = reinterpret_cast<float4*>(dfp) + pt * 4;
#pragma unroll
          for (int mk = 0; mk < 4; ++mk)
            o4[mk] = make_float4(v16[4 * mk], v16[4 * mk + 1], v16[4 * mk + 2], v16[4 * mk + 3]);
          if (fold) {
            // fold keys in the B-fragment order of the tile rows
            frag_keys16(reinterpret_cast<float*>(smem + sm.kf[b]), smem + sm.hkr[b], n, DK,
                        p.rk_dt, pt, PT);
          } else if (pw == kPipePrep - 1) {
            // history dots H[m][v] = k_m . x_v on the tensor cores: records as m,
            // window vectors as n, key channels as k (relabelled as in x_slot)
            const void* hk = smem + sm.hkr[b];
            const bool xk = p.in_dt != DT_F32, kk = p.rk_dt != DT_F32;
            const int g = lane >> 2, t = lane & 3;
            float hc[NTN][4];
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt) hc[nt][0] = hc[nt][1] = hc[nt][2] = hc[nt][3] = 0.f;
            for (int s8 = 0; s8 < DK / 8; ++s8) {
              const int ch = 8 * s8 + 2 * t;
              float2 ka = make_float2(0.f, 0.f), kb = make_float2(0.f, 0.f);
              if (g < n) ka = ld2_as_f32(hk, g * DK + ch, p.rk_dt);
              if (g + 8 < n) kb = ld2_as_f32(hk, (g + 8) * DK + ch, p.rk_dt);
              const int fi = s8 * 32 + lane;
#pragma unroll
              for (int nt = 0; nt < NTN; ++nt) {
                const float x0 = xf[2 * NTN * fi + 2 * nt], x1 = xf[2 * NTN * fi + 2 * nt + 1];
                if (kk && xk) {
                  const Tf32 a[4] = {tf32_split<true>(ka.x), tf32_split<true>(kb.x),
                                     tf32_split<true>(ka.y), tf32_split<true>(kb.y)};
                  const Tf32 bb[2] = {tf32_split<true>(x0), tf32_split<true>(x1)};
                  mma_split<true, true>(hc[nt], a, bb);
                } else {
                  const Tf32 a[4] = {tf32_split<false>(ka.x), tf32_split<false>(kb.x),
                                     tf32_split<false>(ka.y), tf32_split<false>(kb.y)};
                  const Tf32 bb[2] = {tf32_split<false>(x0), tf32_split<false>(x1)};
                  mma_split<false, false>(hc[nt], a, bb);
                }
              }
            }
            float* hh = reinterpret_cast<float*>(smem + sm.hh[b]);
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt) {
              hh[g * kPipeHist + 8 * nt + 2 * t] = hc[nt][0];
              hh[g * kPipeHist + 8 * nt + 2 * t + 1] = hc[nt][1];
              hh[(g + 8) * kPipeHist + 8 * nt + 2 * t] = hc[nt][2];
              hh[(g + 8) * kPipeHist + 8 * nt + 2 * t + 1] = hc[nt][3];
            }
            if (NTN == 1) {
              hh[g * kPipeHist + 8 + 2 * t] = 0.f;
              hh[g * kPipeHist + 8 + 2 * t + 1] = 0.f;
              hh[(g + 8) * kPipeHist + 8 + 2 * t] = 0.f;
              hh[(g + 8) * kPipeHist + 8 + 2 * t + 1] = 0.f;
            }
          }
        }
        named_sync(kPrepBar, PT);
        if (pt == 0) {
          if (kw < nk) issue_window(kw++);  // into the buffer item k's copies used
          mbar_arrive(&mb[PB_PREP + b]);
        }
        __syncwarp();
        nprep = k + 1;
      }
    }
    // ---- solve item k - 1 per value column: outputs and records (an item
    //      the math warps finished is solved even after another wait ran out)
    if (k >= 1 && k - 1 < nprep) {
      const int kp = k - 1, b = kp & 1;
      const bool streamed = named_and(
          kPrepBar, PT, mbar_wait_bounded(&mb[PB_MATH + b], (uint32_t)((kp >> 1) & 1), lim));
      if (!streamed) {
        if (pt == 0 && !*abort) {
          *abort = 1;
          atomicOr(p.err, DEVERR_TIMEOUT);
        }
        alive = false;
        nprep = 0;
      } else {
        const PipeItem& I = *reinterpret_cast<const PipeItem*>(smem + sm.item[b]);
        const float* yo = reinterpret_cast<const float*>(smem + sm.y[b]);
        const int row = I.row, h = I.h, s = I.s, base = I.base;
        const size_t tok0 = (size_t)row * T;
        const size_t sh = (size_t)s * HV + h;
        const int col = pt;  // dv = 128 = prep threads
        float y[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) y[v] = yo[v * DV + col];
        float d[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          d[i] = 0.f;
          if (i < T) {
            const float eg = I.eG[i];
            const size_t tok = tok0 + i;
            const float vi = ld_f32(p.v, (tok * HV + h) * DV + col, p.in_dt);
            float a = I.beta[i] * (vi - eg * y[i]);
#pragma unroll
            for (int j = 0; j < i; ++j) a = fmaf(-I.am[i * kPipeMaxNT + j], d[j], a);
            d[i] = a;
            float o = eg * y[NT + i];
#pragma unroll
            for (int j = 0; j <= i; ++j) o = fmaf(I.fm[i * kPipeMaxNT + j], d[j], o);
            st_f32(p.o, (tok * HV + h) * DV + col, p.in_dt, o * p.scale);
            const size_t rec = (sh * L + base + i) * DV + col;
            st_f32(p.ring_d, rec, p.rd_dt, a);
            st_f32(p.ring_v, rec, p.in_dt, vi);
            const float kv = ld_f32(p.k, (tok * p.HK + h / p.G) * DK + col, p.in_dt);
            st_f32(p.ring_k, (sh * L + base + i) * DK + col, p.rk_dt, kv);
          }
        }
        if (pt < T) {
          p.ring_beta[sh * L + base + pt] = I.beta[pt];
          p.ring_g[sh * L + base + pt] = p.g[(tok0 + pt) * HV + h];
        }
        if (pt == 0 && h == 0 && p.fold_out != nullptr) p.fold_out[row] = (uint8_t)I.fold;
        named_sync(kPrepBar, PT);  // the column sums are read
        if (pt == 0) mbar_arrive(&mb[PB_YFREE + b]);
        __syncwarp();
      }
    }
  }
  __syncthreads();
  // the window copies issued have landed before the CTA leaves (bounded)
  if (pt == 0) {
    for (int kk2 = kw > 2 ? kw - 2 : 0; kk2 < kw; ++kk2)
      mbar_wait_bounded(&mb[PB_WIN + (kk2 & 1)], (uint32_t)((kk2 >> 1) & 1), lim);
  }
}

}  // namespace rssm
