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
// Here the kinds of work run on separate warps, one item apart:
//  - warps 8-11 issue every async copy as 16-byte cp.async pieces spread over
//    their 128 threads: the 8 KB checkpoint chunks of item after item into a
//    ring of up to 16 stages (each as soon as its stage is released), and the
//    window and history rows of item k + 2 as soon as item k is prepared;
//    each barrier counts one arrival per copying thread, made when that
//    thread's copies have landed. They poll and wait, never release: a
//    release waits for the issuing thread's copies in flight, and one thread
//    issuing whole-chunk bulk copies reached one chunk per ~900 cycles, a
//    fifth of an SM's share of HBM;
//  - warps 0-3 ("math"), one value column per thread, consume the chunks: for
//    a folding item S[row] <- e^Gam S[row] + sum_m k_m[row] f_m d_m (stored
//    back), then y_v += x_v[row] S[row] for the 2T window vectors (raw k_i,
//    q_i); for an item with history that does not fold, y_v <- e^Gam y_v +
//    sum_m (k_m . x_v) f_m d_m (the correction term of the replayed state);
//  - warps 4-7 ("prep") prepare item k + 1 (gate scans, the mat-vec inputs,
//    transposed history keys, f_m d_m, the history dots k_m . x_v, the window
//    coefficients A and F) while the math warps stream item k, then solve item
//    k - 1 per value column (outputs and records).
// All of it runs on the CUDA cores: every sum is short or split across
// threads, so no thread waits on a long chain of dependent products (the
// warp-level tensor-core product takes hundreds of cycles from operands to a
// usable accumulator on this part, and a 128-row mat-vec made of them was
// four times slower than the stream of its chunks).
// Items are dealt round-robin from one order that every CTA computes alike:
// folding rows first, so every CTA gets an equal share of the heavier items.
//
// Waits: every mbarrier wait is bounded (the launch's limit) and also gives up
// once another role has given up (abort word). A CTA whose wait ran out sets
// RSSM_DEVERR_TIMEOUT and processes no further item: the rows of those items
// are left untouched; the item in progress writes no output or record (a
// folding item may have stored the chunks it had folded). Before the CTA
// leaves, every copy it issued is waited for again (bounded).
#pragma once

#include "rssm_common.cuh"
#include "rssm_history.cuh"

namespace rssm {

enum : int { PF_LIVE = 1, PF_FOLD = 2 };
constexpr int kPipeDK = 128, kPipeDV = 128;
constexpr int kPipeGroups = kPipeMaxRows / 32;

// Bounded wait that also returns false once the CTA's abort word is set. The
// thread is parked by the hardware between polls (a suspend-time hint), so a
// waiting warp leaves the issue slots of its sub-partition to the warps that
// have work: with short sleeps instead, the waiting and polling warps issued
// most of a launch's instructions.
constexpr uint32_t kPipeParkNs = 1000;
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long lim, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait_hint(bar, parity, kPipeParkNs)) return true;
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

// Eight consecutive 16-bit values (bf16 or fp16) or fp32 values in shared
// memory as fp32 (i a multiple of 8).
__device__ __forceinline__ void ld8_as_f32(const void* base, int i, int dt, float (&v)[8]) {
  if (dt == DT_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    const float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    return;
  }
  const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float2 f;
    if (dt == DT_BF16) {
      f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
    } else {
      f = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
    }
    v[2 * q] = f.x;
    v[2 * q + 1] = f.y;
  }
}

// y[v] += x_v[row] s over the NV mat-vec inputs of one row (xr: [NV] floats)
template <int NV>
__device__ __forceinline__ void matvec_row(const float* xr, float s, float (&y)[NV]) {
  const float4* x4 = reinterpret_cast<const float4*>(xr);
#pragma unroll
  for (int v4 = 0; v4 < NV / 4; ++v4) {
    const float4 x = x4[v4];
    y[4 * v4] = fmaf(x.x, s, y[4 * v4]);
    y[4 * v4 + 1] = fmaf(x.y, s, y[4 * v4 + 1]);
    y[4 * v4 + 2] = fmaf(x.z, s, y[4 * v4 + 2]);
    y[4 * v4 + 3] = fmaf(x.w, s, y[4 * v4 + 3]);
  }
  if constexpr (NV % 4 != 0) {
    const float2 x = reinterpret_cast<const float2*>(xr)[NV / 2 - 1];
    y[NV - 2] = fmaf(x.x, s, y[NV - 2]);
    y[NV - 1] = fmaf(x.y, s, y[NV - 1]);
  }
}

// ---------------------------------------------------------------- math warps
// One item's stream, thread `col` owning value column col. q is the global
// index of the item's first chunk. Returns false if a wait gave up (the item
// is then abandoned: nothing more is stored, the stages it did not release
// stay held).
template <typename ST, int NV>
__device__ __forceinline__ bool pipe_stream(const PipeItem& I, const ST* ring, uint64_t* mb, int NS,
                                            int q, const float* xh, const float* hkt,
                                            const float* dtm, const float* hh, ST* gtile,
                                            unsigned long long lim, const volatile int* abort,
                                            int col, int lane, float (&y)[NV]) {
  constexpr int DV = kPipeDV, DK = kPipeDK;
  constexpr int CR = kChunkBytes / (DV * (int)sizeof(ST));  // rows per chunk
  constexpr int NCH = DK / CR;
  const bool fold = I.fold != 0;
  const int n = I.n;
  const float decay = I.egam;
  // f_m d_m of this column (zero past the history)
  float dm[kPipeHist];
#pragma unroll
  for (int m = 0; m < kPipeHist; ++m) dm[m] = n > 0 ? dtm[m * DV + col] : 0.f;
#pragma unroll
  for (int v = 0; v < NV; ++v) y[v] = 0.f;
  for (int j = 0; j < NCH; ++j, ++q) {
    const int st = q % NS;
    if (!__all_sync(kFull, pipe_wait(&mb[PB_FULL + st], (uint32_t)((q / NS) & 1), lim, abort)))
      return false;
    const ST* stg = ring + (size_t)st * CR * DV + col;
    if (fold) {
#pragma unroll 4
      for (int u = 0; u < CR; ++u) {
        const int row = j * CR + u;
        float s = decay * st_load<ST>(stg + (size_t)u * DV);
        if (n > 0) {  // (an empty history folds to the checkpoint itself)
          const float4* kr = reinterpret_cast<const float4*>(hkt + row * kPipeHist);
#pragma unroll
          for (int q4 = 0; q4 < kPipeHist / 4; ++q4) {
            const float4 k4 = kr[q4];
            s = fmaf(k4.x, dm[4 * q4], s);
            s = fmaf(k4.y, dm[4 * q4 + 1], s);
            s = fmaf(k4.z, dm[4 * q4 + 2], s);
            s = fmaf(k4.w, dm[4 * q4 + 3], s);
          }
        }
        // the mat-vec takes the stored (rounded) checkpoint value
        s = st_store<ST>(gtile + (size_t)row * DV + col, s);
        matvec_row<NV>(xh + row * NV, s, y);
      }
    } else {
#pragma unroll 8
      for (int u = 0; u < CR; ++u) {
        const int row = j * CR + u;
        matvec_row<NV>(xh + row * NV, st_load<ST>(stg + (size_t)u * DV), y);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&mb[PB_FULL + NS + st]);  // stage released
  }
  if (!fold && n > 0) {
    // replayed state of a window that does not fold: e^Gam S0^T x + sum_m f_m d_m (k_m . x)
#pragma unroll
    for (int v = 0; v < NV; ++v) y[v] *= decay;
#pragma unroll
    for (int m = 0; m < kPipeHist; ++m) {
      if (m < n) {
#pragma unroll
        for (int v = 0; v < NV; ++v) y[v] = fmaf(hh[m * NV + v], dm[m], y[v]);
      }
    }
  }
  return true;
}

// The items of one CTA: item k is (row, value head) number b0 + k P of the
// launch's order (rows as ranked, value heads fastest).
struct PipeItems {
  const int* order;
  int b0, P, HV;
  __device__ __forceinline__ void at(int k, int& row, int& h) const {
    const int i = b0 + k * P;
    row = order[i / HV];
    h = i - (i / HV) * HV;
  }
};

// Copies of item k's window into buffer k & 1: q, k, v rows, and the
// history's keys, deltas and gates; copying thread pp of NP takes the 16-byte
// pieces pp, pp + NP, ... of the whole list, then arrives on the buffer's
// barrier once its copies have landed. The thread that withholds its arrival
// (test hook) leaves the barrier one arrival short.
template <int NP>
__device__ __forceinline__ void pipe_copy_window(const ReplayParams& p, const PipeSmem& sm,
                                                 unsigned char* smem, uint64_t* mb,
                                                 const PipeItems& it, const int* r_slot,
                                                 const int* r_cur, int k, int pp) {
  constexpr int DK = kPipeDK, DV = kPipeDV;
  int row, h;
  it.at(k, row, h);
  const int T = p.T, L = p.L, HV = p.HV;
  const int b = k & 1, s = r_slot[row], n = r_cur[row];
  const size_t tok0 = (size_t)row * T;
  const int kh = h / p.G;
  const uint32_t qrow = (uint32_t)(DK * dtype_bytes(p.in_dt));
  unsigned char* wr = smem + sm.buf + b * sm.bufsz + sm.wraw;
  const int sk = dtype_bytes(p.rk_dt), sd = dtype_bytes(p.rd_dt);
  const int rowp = (int)(qrow / 16);  // pieces of one q, k or v row
  const int nwin = 3 * T * rowp;
  const int nkey = n * DK * sk / 16, ndel = n * DV * sd / 16, ngat = n > 0 ? round4(n) / 4 : 0;
  const size_t sh = (size_t)s * HV + h;
  const char* kbase = static_cast<const char*>(p.ring_k) + sh * L * DK * sk;
  const char* dbase = static_cast<const char*>(p.ring_d) + sh * L * DV * sd;
  const char* gbase = reinterpret_cast<const char*>(p.ring_g + sh * L);
  for (int e = pp; e < nwin + nkey + ndel + ngat; e += NP) {
    if (e < nwin) {
      const int r3 = e / rowp, off = (e - r3 * rowp) * 16;  // row r3 of [q | k | v][T]
      const int which = r3 / T, i = r3 - which * T;
      const char* src;
      if (which == 2) {
        src = static_cast<const char*>(p.v) + ((tok0 + i) * HV + h) * (size_t)qrow;
      } else {
        src = static_cast<const char*>(which == 0 ? p.q : p.k) +
              ((tok0 + i) * p.HK + kh) * (size_t)qrow;
      }
      cp_async16(wr + r3 * qrow + off, src + off);
    } else if (e < nwin + nkey) {
      const int off = (e - nwin) * 16;
      cp_async16(smem + sm.buf + b * sm.bufsz + sm.hkr + off, kbase + off);
    } else if (e < nwin + nkey + ndel) {
      const int off = (e - nwin - nkey) * 16;
      cp_async16(smem + sm.buf + b * sm.bufsz + sm.hdr + off, dbase + off);
    } else {
      const int off = (e - nwin - nkey - ndel) * 16;
      cp_async16(smem + sm.buf + b * sm.bufsz + sm.hgr + off, gbase + off);
    }
  }
  const bool held = k == 0 && pp == 0 &&
                    (p.hook.withhold == WH_WINDOW || (n > 0 && p.hook.withhold == WH_HIST));
  if (!held) cp_async_arrive(&mb[PB_WIN + b]);
}

// Chunk qq of the CTA's stream (chunk qq % NCH of item qq / NCH) into ring
// stage qq % NS, copying thread pp's share of its 16-byte pieces.
template <typename ST, int NP>
__device__ __forceinline__ void pipe_copy_chunk(const ReplayParams& p, const PipeSmem& sm,
                                                unsigned char* smem, uint64_t* mb,
                                                const PipeItems& it, const int* r_slot, int qq,
                                                int pp) {
  constexpr int DK = kPipeDK, DV = kPipeDV;
  constexpr int NCH = DK * DV * (int)sizeof(ST) / kChunkBytes;
  const int k = qq / NCH, j = qq - k * NCH;
  int row, h;
  it.at(k, row, h);
  const char* src = reinterpret_cast<const char*>(static_cast<const ST*>(p.state) +
                                                  ((size_t)r_slot[row] * p.HV + h) * DK * DV) +
                    (size_t)j * kChunkBytes;
  const int st = qq % sm.ns;
  unsigned char* dst = smem + sm.ring + (size_t)st * kChunkBytes;
#pragma unroll
  for (int e = pp; e < kChunkBytes / 16; e += NP) cp_async16(dst + e * 16, src + e * 16);
  const bool held = k == 0 && pp == 0 && p.hook.withhold == WH_CHUNK0 + j;
  if (!held) cp_async_arrive(&mb[PB_FULL + st]);
}

// ---------------------------------------------------------------- kernel
template <int ALGO, typename ST, int NT>
__global__ void __launch_bounds__(kPipeThreads, 1)
    pipe_kernel(const ReplayParams p, const PipeSmem sm) {
  static_assert(ALGO == ALGO_GDN, "the pipelined kernel serves GDN heads");
  constexpr int DK = kPipeDK, DV = kPipeDV, NV = 2 * NT;
  constexpr int CR = kChunkBytes / (DV * (int)sizeof(ST));
  constexpr int NCH = DK / CR;
  constexpr int PT = 32 * kPipePrep;       // prep threads (one per value column)
  constexpr int kPrepBar = 1;              // named barrier of the prep warps
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, T = p.T, L = p.L, HV = p.HV, NS = sm.ns;
  constexpr unsigned long long lim = kWaitLimitNs;
  uint64_t* mb = reinterpret_cast<uint64_t*>(smem + sm.mbar);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + sm.mbar + 8 * kPipeMbars);
  int* r_slot = reinterpret_cast<int*>(smem + sm.rows);
  int* r_cur = r_slot + sm.maxb;
  int* r_order = r_cur + sm.maxb;
  int* r_flag = r_order + sm.maxb;
  int* gcnt = r_flag + sm.maxb;  // [2][kPipeGroups]: folding / other live rows per group
  ST* ring = reinterpret_cast<ST*>(smem + sm.ring);

  constexpr int NP = 32 * kPipeProdWarps;  // copying threads
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&mb[PB_WIN + b], NP);
      mbar_init(&mb[PB_PREP + b], 1);
      mbar_init(&mb[PB_MATH + b], kPipeMath);
      mbar_init(&mb[PB_YFREE + b], 1);
    }
    for (int st = 0; st < NS; ++st) {
      mbar_init(&mb[PB_FULL + st], NP);
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
  const PipeItems items{r_order, b0, P, HV};
  const int pt = tid - 32 * kPipeMath;  // prep thread (negative on the math warps)
  const int s_in = dtype_bytes(p.in_dt);
  const uint32_t qrow = (uint32_t)(DK * s_in);
  const int nq = nk * NCH;  // chunks of this CTA's stream
  // the window betas and gates of every item of this CTA, staged once: the
  // prep warps then read no global memory on their critical path
  float2* bgt = reinterpret_cast<float2*>(smem + sm.bg);
  for (int e = tid; e < nk * T; e += kPipeThreads) {
    const int k = e / T, i = e - k * T;
    int row, h;
    items.at(k, row, h);
    const size_t ix = ((size_t)row * T + i) * HV + h;
    bgt[k * NT + i] = make_float2(p.beta[ix], p.g[ix]);
  }
  __syncthreads();

  if (warp >= kPipeProd) {
    // ================= copying threads: every async copy, as its buffer frees
    const int pp = tid - 32 * kPipeProd;
    int kw = 0, qq = 0;  // windows and chunks issued
    unsigned long long t_last = global_ns();
    while (kw < nk || qq < nq) {
      bool progress = false;
      // window and history rows of item kw into buffer kw & 1, once item kw - 2
      // (the buffer's last user) is prepared
      while (kw < nk && (kw < 2 || mbar_test(&mb[PB_PREP + (kw & 1)],
                                             (uint32_t)(((kw - 2) >> 1) & 1)))) {
        pipe_copy_window<NP>(p, sm, smem, mb, items, r_slot, r_cur, kw++, pp);
        progress = true;
      }
      // every chunk whose stage is free, each once the chunk NS before it is released
      while (qq < nq && (qq < NS || mbar_test(&mb[PB_FULL + NS + qq % NS],
                                              (uint32_t)(((qq / NS) - 1) & 1)))) {
        pipe_copy_chunk<ST, NP>(p, sm, smem, mb, items, r_slot, qq++, pp);
        progress = true;
      }
      if (progress) {
        t_last = global_ns();
        continue;
      }
      if (*abort) break;
      if (global_ns() - t_last > lim) {
        if (!*abort) {
          *abort = 1;
          atomicOr(p.err, DEVERR_TIMEOUT);
        }
        break;
      }
      // park until the next stage is released (or the window buffer frees, the
      // next time round)
      if (qq < nq) {
        mbar_try_wait_hint(&mb[PB_FULL + NS + qq % NS], (uint32_t)(((qq / NS) - 1) & 1),
                           kPipeParkNs);
      } else {
        mbar_try_wait_hint(&mb[PB_PREP + (kw & 1)], (uint32_t)(((kw - 2) >> 1) & 1),
                           kPipeParkNs);
      }
    }
    // every copy this thread issued has landed before the CTA leaves
    cp_async_wait_all();
    __syncwarp();
    __syncthreads();
    return;
  }

  if (warp < kPipeMath) {
    // ================= math: stream every item's tile, one value column per thread
    const int col = tid;
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
      const PipeItem& I = *reinterpret_cast<const PipeItem*>(smem + sm.buf + b * sm.bufsz + sm.item);
      ST* gtile = static_cast<ST*>(p.state) + ((size_t)I.s * HV + I.h) * DK * DV;
      float y[NV];
      bool ok = pipe_stream<ST, NV>(
          I, ring, mb, NS, q, reinterpret_cast<const float*>(smem + sm.buf + b * sm.bufsz + sm.xh),
          reinterpret_cast<const float*>(smem + sm.buf + b * sm.bufsz + sm.hkt),
          reinterpret_cast<const float*>(smem + sm.buf + b * sm.bufsz + sm.dt),
          reinterpret_cast<const float*>(smem + sm.buf + b * sm.bufsz + sm.hh), gtile, lim, abort, col, lane, y);
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
      float* yo = reinterpret_cast<float*>(smem + sm.buf + b * sm.bufsz + sm.y);
#pragma unroll
      for (int v = 0; v < NV; ++v) yo[v * DV + col] = y[v];
      __syncwarp();
      if (lane == 0) mbar_arrive(&mb[PB_MATH + b]);
    }
    __syncwarp();
    __syncthreads();
    return;
  }

  // ================= prep warps: prepare item k, solve item k - 1
  const int pw = pt >> 5;
  bool alive = true;  // no wait of the prep warps has run out
  int nprep = 0;      // items prepared (handed to the math warps)
  for (int k = 0; k <= nk; ++k) {
    // ---- prepare item k
    if (named_and(kPrepBar, PT, alive && k < nk && !*abort)) {
      const int b = k & 1;
      int row, h;
      items.at(k, row, h);
      const int s = r_slot[row], c = r_cur[row];
      const bool fold = (r_flag[row] & PF_FOLD) != 0;
      const int n = c;
      PipeItem& I = *reinterpret_cast<PipeItem*>(smem + sm.buf + b * sm.bufsz + sm.item);
      float bet = 0.f, gw = 0.f;
      if (pt < T) {
        const float2 e = bgt[k * NT + pt];
        bet = e.x;
        gw = e.y;
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
        const unsigned char* wr = smem + sm.buf + b * sm.bufsz + sm.wraw;
        const void* wq = wr;                      // q rows [T][dk]
        const void* wkr = wr + T * qrow;          // k rows [T][dk]
        float* xh = reinterpret_cast<float*>(smem + sm.buf + b * sm.bufsz + sm.xh);
        const int ch = pt;                        // key channel / value column of this thread
        // P1 (prep warp 0): gates, item scalars
        if (pw == 0) {
          const float* hg = reinterpret_cast<const float*>(smem + sm.buf + b * sm.bufsz + sm.hgr);
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
        // P2 (thread = key channel): the window's k and v rows kept for the
        // solve (the landing buffer takes item k + 2's copies), the mat-vec
        // inputs of this channel, and its history keys transposed
        {
          const uint4* src = reinterpret_cast<const uint4*>(wkr);
          uint4* dst = reinterpret_cast<uint4*>(smem + sm.buf + b * sm.bufsz + sm.ep);
          for (int e = pt; e < (int)(2 * T * qrow / 16); e += PT) dst[e] = src[e];
        }
        {
          float xv[NV];
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            xv[i] = i < T ? ld_f32(wkr, (size_t)i * DK + ch, p.in_dt) : 0.f;
            xv[NT + i] = i < T ? ld_f32(wq, (size_t)i * DK + ch, p.in_dt) : 0.f;
          }
          float* xr = xh + ch * NV;
#pragma unroll
          for (int v = 0; v < NV; ++v) xr[v] = xv[v];
        }
        if (fold && n > 0) {
          const void* hk = smem + sm.buf + b * sm.bufsz + sm.hkr;
          float kt[kPipeHist];
#pragma unroll
          for (int m = 0; m < kPipeHist; ++m)
            kt[m] = m < n ? ld_f32(hk, (size_t)m * DK + ch, p.rk_dt) : 0.f;
          float4* kr = reinterpret_cast<float4*>(smem + sm.buf + b * sm.bufsz + sm.hkt) + ch * (kPipeHist / 4);
#pragma unroll
          for (int q4 = 0; q4 < kPipeHist / 4; ++q4)
            kr[q4] = make_float4(kt[4 * q4], kt[4 * q4 + 1], kt[4 * q4 + 2], kt[4 * q4 + 3]);
        }
        named_sync(kPrepBar, PT);
        // P3: f_m d_m of this column (the fold's and the correction's deltas)
        if (n > 0) {
          const void* hd = smem + sm.buf + b * sm.bufsz + sm.hdr;
          float* dtm = reinterpret_cast<float*>(smem + sm.buf + b * sm.bufsz + sm.dt);
#pragma unroll
          for (int m = 0; m < kPipeHist; ++m)
            dtm[m * DV + ch] = m < n ? I.hf[m] * ld_f32(hd, (size_t)m * DV + ch, p.rd_dt) : 0.f;
        }
        // P4: window coefficients, two threads per pair (j <= i < T), half the
        // key channels each
        {
          const int pr2 = pt >> 1, half = pt & 1;
          const int i = pr2 / kPipeMaxNT, j = pr2 - i * kPipeMaxNT;
          float skk = 0.f, skq = 0.f;
          if (i < T && j <= i) {
            for (int c8 = 64 * half; c8 < 64 * half + 64; c8 += 8) {
              float kj[8], ki[8], qi[8];
              ld8_as_f32(wkr, j * DK + c8, p.in_dt, kj);
              ld8_as_f32(wkr, i * DK + c8, p.in_dt, ki);
              ld8_as_f32(wq, i * DK + c8, p.in_dt, qi);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                skk = fmaf(kj[e], ki[e], skk);
                skq = fmaf(kj[e], qi[e], skq);
              }
            }
          }
          skk += __shfl_xor_sync(kFull, skk, 1);
          skq += __shfl_xor_sync(kFull, skq, 1);
          if (half == 0 && i < T && j <= i) {
            const float wgt = __expf(I.G[i] - I.G[j]);
            I.fm[i * kPipeMaxNT + j] = wgt * skq;
            I.am[i * kPipeMaxNT + j] = j < i ? I.beta[i] * wgt * skk : 0.f;
          }
        }
        // P5: history dots k_m . x_v of a window that does not fold, one
        // thread per (record, pair of vectors)
        if (!fold && n > 0) {
          const void* hk = smem + sm.buf + b * sm.bufsz + sm.hkr;
          float* hh = reinterpret_cast<float*>(smem + sm.buf + b * sm.bufsz + sm.hh);
          constexpr int VP = NV / 2;  // vector pairs
          for (int o = pt; o < kPipeHist * VP; o += PT) {
            const int m = o / VP, v0 = 2 * (o - m * VP);
            float a0 = 0.f, a1 = 0.f;
            if (m < n) {
              for (int c8 = 0; c8 < DK; c8 += 8) {
                float km[8];
                ld8_as_f32(hk, m * DK + c8, p.rk_dt, km);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float2 x = *reinterpret_cast<const float2*>(xh + (c8 + e) * NV + v0);
                  a0 = fmaf(km[e], x.x, a0);
                  a1 = fmaf(km[e], x.y, a1);
                }
              }
            }
            hh[m * NV + v0] = a0;
            hh[m * NV + v0 + 1] = a1;
          }
        }
        named_sync(kPrepBar, PT);
        if (pt == 0) mbar_arrive(&mb[PB_PREP + b]);  // (frees the landing buffer too)
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
        const PipeItem& I = *reinterpret_cast<const PipeItem*>(smem + sm.buf + b * sm.bufsz + sm.item);
        const float* yo = reinterpret_cast<const float*>(smem + sm.buf + b * sm.bufsz + sm.y);
        const void* ek = smem + sm.buf + b * sm.bufsz + sm.ep;               // k rows [T][dk]
        const void* ev = smem + sm.buf + b * sm.bufsz + sm.ep + T * qrow;    // v rows [T][dv]
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
            const float vi = ld_f32(ev, (size_t)i * DV + col, p.in_dt);
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
            const float kv = ld_f32(ek, (size_t)i * DK + col, p.in_dt);
            st_f32(p.ring_k, (sh * L + base + i) * DK + col, p.rk_dt, kv);
          }
        }
        if (pt < T) {
          p.ring_beta[sh * L + base + pt] = I.beta[pt];
          p.ring_g[sh * L + base + pt] = bgt[kp * NT + pt].y;
        }
        if (pt == 0 && h == 0 && p.fold_out != nullptr) p.fold_out[row] = (uint8_t)I.fold;
        named_sync(kPrepBar, PT);  // the column sums are read
        if (pt == 0) mbar_arrive(&mb[PB_YFREE + b]);
        __syncwarp();
      }
    }
  }
  __syncthreads();
}

}  // namespace rssm
