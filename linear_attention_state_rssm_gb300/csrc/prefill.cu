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
// memory. The chunk's dense products run on the tensor cores (warp-level
// mma.sync m16n8k8, tf32 head/tail operand splits, fp32 accumulation): the
// mat-vecs Y = X^T S for its 2C vectors, the GDN pair dots [K; Q] K^T, the
// outputs O = Y_q + F D and the rank-16 update of the state slice. The forward
// substitution for the deltas (one column per thread, on warps 0-1) and the
// gate scans run on CUDA cores while warps 2-7 prepare the next chunk.
#include "replay_impl.cuh"
#include "rssm_mma.cuh"
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
  constexpr int CQ = CB / 4;                  // column quads of the state slice
  constexpr int XS = kPrefillXS, KS = kPrefillKS;
  constexpr int SS = CB + 8, DS = CB + 8, YS = CB + 8;  // row strides: S, deltas, y
  constexpr int FS = kPrefillKS;              // row stride of the coefficients A, F
  constexpr int NTN = CB / 8;                 // 8-column tiles of a CB-wide product
  // GDN mat-vec and pair inputs are the raw bf16 k, q: exact in tf32
  constexpr bool EXACT_X = ALGO == ALGO_GDN && INB == 2;
  // Warps 0-1 solve a chunk while warps 2-7 (the preparing warps) stage the
  // next one and build its mat-vec inputs and window coefficients.
  constexpr int PREP0 = 2 * 32, NP = PT - PREP0;
  constexpr int EPU = 16 / INB;               // input values per 16-byte unit
  // 16-byte units of one chunk per preparing thread (dk <= 128): q and k
  // rows, v columns, KDA gates
  constexpr int MQ = (C * 128 / EPU + NP - 1) / NP;
  constexpr int MV = (C * CB / EPU + NP - 1) / NP;
  constexpr int MG = ALGO == ALGO_KDA ? (C * 128 / 4 + NP - 1) / NP : 0;
  static_assert(PW == 8 && CB % 8 == 0, "prefill warp layout");
  extern __shared__ __align__(128) unsigned char smem[];

  const int nb = p.dv / CB;
  const int h = blockIdx.x / nb, cb0 = (blockIdx.x - h * nb) * CB, r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dk = p.dk, dv = p.dv, L = p.L, HV = p.HV, HK = p.HK, kh = h / p.G;
  const bool reporter = tid == 0 && blockIdx.x == 0;
  const bool prep = tid >= PREP0;
  const int lt = tid - PREP0;  // index among the preparing threads

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
  float* wv2 = reinterpret_cast<float*>(smem + p.sm.wv);
  float* xT = reinterpret_cast<float*>(smem + p.sm.xT);
  float* kdT = reinterpret_cast<float*>(smem + p.sm.kdT);
  float* y = reinterpret_cast<float*>(smem + p.sm.y);
  float* part = reinterpret_cast<float*>(smem + p.sm.part);
  float* dch = reinterpret_cast<float*>(smem + p.sm.dch);
  float* am2 = reinterpret_cast<float*>(smem + p.sm.am);
  float* fm2 = reinterpret_cast<float*>(smem + p.sm.fm);
  float* G = reinterpret_cast<float*>(smem + p.sm.G);
  float* eG = reinterpret_cast<float*>(smem + p.sm.eG);
  float* ekd = reinterpret_cast<float*>(smem + p.sm.ekd);
  float* wb2 = reinterpret_cast<float*>(smem + p.sm.wb);
  float* decr2 = reinterpret_cast<float*>(smem + p.sm.decr);

  const int uq = dk / EPU, uv = CB / EPU, ug = dk / 4;  // 16-byte units per row
  const int nchunks = (n + C - 1) / C;
  const int fg = lane >> 2, ft = lane & 3;  // fragment row group, thread in group

  // ---- a chunk's inputs, loaded into registers of the preparing threads
  //      one chunk ahead
  uint4 rq[MQ], rk[MQ], rv[MV], rg[MG > 0 ? MG : 1];
  float rb = 0.f, rgg = 0.f;  // beta and GDN gate of token lt of the chunk
  auto prefetch = [&](int ch) {
    const int t0 = ch * C, cn = min(C, n - t0);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
      const int u = lt + m * NP, i = u / uq, pu = u - i * uq;
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
      const int u = lt + m * NP, i = u / uv, pu = u - i * uv;
      rv[m] = z;
      if (u < C * uv && i < cn) {
        const size_t off = ((((size_t)a0 + t0 + i) * HV + h) * dv + cb0) * INB;
        rv[m] = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(p.v) + off) + pu);
      }
    }
#pragma unroll
    for (int m = 0; m < MG; ++m) {
      const int u = lt + m * NP, i = u / ug, pu = u - i * ug;
      rg[m] = z;
      if (u < C * ug && i < cn) {
        const size_t off = (((size_t)a0 + t0 + i) * HV + h) * dk;
        rg[m] = __ldg(reinterpret_cast<const uint4*>(p.g + off) + pu);
      }
    }
    rb = 0.f;
    rgg = 0.f;
    if (lt < cn) {
      const size_t tok = (size_t)a0 + t0 + lt;
      rb = __ldg(p.beta + tok * HV + h);
      if (ALGO == ALGO_GDN) rgg = __ldg(p.g + tok * HV + h);
    }
  };
  // registers -> fp32 chunk arrays (rows past the chunk are zero)
  auto stage = [&](float* wv, float* wb) {
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
      const int u = lt + m * NP, i = u / uq, pu = u - i * uq;
      if (u < C * uq) {
        widen_store<INB>(wq + i * dk + pu * EPU, rq[m], p.in_dt);
        widen_store<INB>(wk + i * dk + pu * EPU, rk[m], p.in_dt);
      }
    }
#pragma unroll
    for (int m = 0; m < MV; ++m) {
      const int u = lt + m * NP, i = u / uv, pu = u - i * uv;
      if (u < C * uv) widen_store<INB>(wv + i * CB + pu * EPU, rv[m], p.in_dt);
    }
#pragma unroll
    for (int m = 0; m < MG; ++m) {
      const int u = lt + m * NP, i = u / ug, pu = u - i * ug;
      if (u < C * ug) widen_store<4>(G + i * dk + pu * 4, rg[m], DT_F32);
    }
    if (lt < C) wb[lt] = rb;
  };
  // GDN, one warp: inclusive prefix of the nm gates x (lane i holds gate i),
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
  auto kda_scan = [&](int nm, float* decr, int t, int nt) {
    for (int ch = t; ch < dk; ch += nt) {
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
  // S <- e^{G_last} S + sum_j kd_j d_j^T (dch rows past the chunk are zero):
  // a [dk x C] x [C x CB] product on the tensor cores, the S tile as the fp32
  // accumulator; warp w takes 8-column tile w % NTN of every 16-row tile
  auto update = [&](float dec, const float* decr) {
    const int ntiles = (dk / 16) * NTN;
    const int nt = warp % NTN;
    Tf32 bf[2][2];  // deltas: k-steps j0 = 0, 8
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      bf[ks][0] = tf32_split<false>(dch[(8 * ks + ft) * DS + nt * 8 + fg]);
      bf[ks][1] = tf32_split<false>(dch[(8 * ks + ft + 4) * DS + nt * 8 + fg]);
    }
    for (int id = warp; id < ntiles; id += PW) {
      const int m0 = (id / NTN) * 16;
      float* s0 = S + (m0 + fg) * SS + nt * 8 + 2 * ft;
      float* s1 = s0 + 8 * SS;
      const float2 u0 = *reinterpret_cast<const float2*>(s0);
      const float2 u1 = *reinterpret_cast<const float2*>(s1);
      const float f0 = ALGO == ALGO_KDA ? decr[m0 + fg] : dec;
      const float f1 = ALGO == ALGO_KDA ? decr[m0 + fg + 8] : dec;
      float acc[4] = {f0 * u0.x, f0 * u0.y, f1 * u1.x, f1 * u1.y};
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const float* kr = kdT + (m0 + fg) * KS + 8 * ks + ft;
        const Tf32 af[4] = {tf32_split<false>(kr[0]), tf32_split<false>(kr[8 * KS]),
                            tf32_split<false>(kr[4]), tf32_split<false>(kr[8 * KS + 4])};
        mma_split<false, false>(acc, af, bf[ks]);
      }
      *reinterpret_cast<float2*>(s0) = make_float2(acc[0], acc[1]);
      *reinterpret_cast<float2*>(s1) = make_float2(acc[2], acc[3]);
    }
  };
  // The next chunk on the preparing warps (named barrier 1): stage it, its gate
  // prefixes, mat-vec inputs per key channel (k_i at [0, C), q_i at [C, 2C);
  // KDA: decayed by e^{G_i}), and its window coefficients
  //     A_ij = beta_i e^{G_i - G_j} k_i.k_j (j < i), F_ij = e^{G_i - G_j} q_i.k_j (j <= i)
  auto prepare = [&](int ch) {
    const int b = ch & 1, cn = min(C, n - ch * C);
    float* am = am2 + b * C * FS;
    float* fm = fm2 + b * C * FS;
    float* wb = wb2 + b * C;
    stage(wv2 + b * C * CB, wb);
    if (ALGO == ALGO_GDN && warp == 2) gdn_scan(rgg, cn);
    if (ch + 1 < nchunks) prefetch(ch + 1);  // after the scan has read this chunk's gates
    named_sync(1, NP);
    if (ALGO == ALGO_KDA) {
      kda_scan(cn, decr2 + b * dk, lt, NP);
      named_sync(1, NP);
    }
    for (int e = lt; e < 2 * dk; e += NP) {
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
      // (writes rows i < cn, entries j <= i; F's other entries stay zero)
      for (int e = lt; e < C * FS; e += NP) {
        const int i = e / FS, j = e - i * FS;
        if (i >= cn || j > i) fm[e] = 0.f;
      }
      window_pairs<ALGO, FS>(cn, dk, wk, wq, G, wb, am, fm, warp - 2, PW - 2, lane);
      return;
    }
    named_sync(1, NP);
    // [K; Q] K^T over the key channels on the tensor cores (raw vectors):
    // warps 2-5, one 16 x 8 tile each
    if (warp < 6) {
      const int tile = warp - 2;
      const int mq = (tile >> 1) * C, n8 = (tile & 1) * 8;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k0 = 0; k0 < dk; k0 += 8) {
        const float* x0 = xT + (k0 + ft) * XS;
        const float* x4 = x0 + 4 * XS;
        const Tf32 af[4] = {tf32_split<EXACT_X>(x0[mq + fg]), tf32_split<EXACT_X>(x0[mq + fg + 8]),
                            tf32_split<EXACT_X>(x4[mq + fg]), tf32_split<EXACT_X>(x4[mq + fg + 8])};
        const Tf32 bf[2] = {tf32_split<EXACT_X>(x0[n8 + fg]), tf32_split<EXACT_X>(x4[n8 + fg])};
        mma_split<EXACT_X, EXACT_X>(acc, af, bf);
      }
      float* pw = part + (mq + fg) * C + n8 + 2 * ft;
      *reinterpret_cast<float2*>(pw) = make_float2(acc[0], acc[1]);
      *reinterpret_cast<float2*>(pw + 8 * C) = make_float2(acc[2], acc[3]);
    }
    named_sync(1, NP);
    for (int e = lt; e < C * C; e += NP) {
      const int i = e >> 4, j = e & 15;
      const bool on = i < cn && j <= i;
      const float wgt = on ? __expf(G[i] - G[j]) : 0.f;
      fm[i * FS + j] = on ? wgt * part[(C + i) * C + j] : 0.f;
      am[i * FS + j] = (on && j < i) ? wb[i] * wgt * part[i * C + j] : 0.f;
    }
  };

  if (prep) prefetch(0);

  // ---- the checkpoint slice -> fp32 S [dk][CB]
  ST* gtile = static_cast<ST*>(p.state) + ((size_t)s * HV + h) * dk * dv + cb0;
  for (int e = tid; e < dk * CQ; e += PT) {
    const int row = e / CQ, q4 = e - row * CQ;
    float v4[4];
    ld_cols<ST, 4>(gtile + (size_t)row * dv + 4 * q4, v4);
    *reinterpret_cast<float4*>(S + row * SS + 4 * q4) = make_float4(v4[0], v4[1], v4[2], v4[3]);
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
      dch[j * DS + col] =
          j < nm ? ld_f32(p.ring_d, (sh * L + m0 + j) * dv + cb0 + col, p.rd_dt) : 0.f;
    }
    if (ALGO == ALGO_GDN && warp == 0) gdn_scan(lane < nm ? p.ring_g[sh * L + m0 + lane] : 0.f, nm);
    __syncthreads();
    if (ALGO == ALGO_KDA) {
      kda_scan(nm, decr2, tid, PT);
      __syncthreads();
    }
    build_kd(nm, tid, PT);
    __syncthreads();
    update(ALGO == ALGO_GDN ? __expf(G[nm - 1]) : 1.f, decr2);
    __syncthreads();
  }

  // ---- the prompt, chunk by chunk: (A) mat-vec, (B) solve || prepare the
  //      next chunk, (C) update
  if (prep) prepare(0);
  __syncthreads();
  for (int ch = 0; ch < nchunks; ++ch) {
    const int b = ch & 1, t0 = ch * C, cn = min(C, n - t0);
    // ---- (A) y_v = S^T x_v for the 2C vectors: Y [2C x CB] = X^T S on the
    //      tensor cores; warp w takes the 16-vector block and the 8-column
    //      blocks TPW w, TPW w + 1, ...
    {
      constexpr int TPW = 2 * NTN / PW > 0 ? 2 * NTN / PW : 1;
      const int id0 = warp * TPW;
      const int v0 = (id0 / NTN) * 16;
      float acc[TPW][4];
#pragma unroll
      for (int u = 0; u < TPW; ++u) {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[u][q] = 0.f;
      }
      if (id0 < 2 * NTN) {
        for (int k0 = 0; k0 < dk; k0 += 8) {
          const float* x0 = xT + (k0 + ft) * XS + v0 + fg;
          const float* x4 = x0 + 4 * XS;
          const Tf32 af[4] = {tf32_split<EXACT_X>(x0[0]), tf32_split<EXACT_X>(x0[8]),
                              tf32_split<EXACT_X>(x4[0]), tf32_split<EXACT_X>(x4[8])};
#pragma unroll
          for (int u = 0; u < TPW; ++u) {
            const int n0 = ((id0 + u) % NTN) * 8;
            const float* s0 = S + (k0 + ft) * SS + n0 + fg;
            const Tf32 bf[2] = {tf32_split<false>(s0[0]), tf32_split<false>(s0[4 * SS])};
            mma_split<EXACT_X, false>(acc[u], af, bf);
          }
        }
#pragma unroll
        for (int u = 0; u < TPW; ++u) {
          const int n0 = ((id0 + u) % NTN) * 8 + 2 * ft;
          const int va = v0 + fg, vb = va + 8;
          const float fa = ALGO == ALGO_GDN ? eG[va < C ? va : va - C] : 1.f;
          const float fb = ALGO == ALGO_GDN ? eG[vb < C ? vb : vb - C] : 1.f;
          *reinterpret_cast<float2*>(y + va * YS + n0) = make_float2(fa * acc[u][0], fa * acc[u][1]);
          *reinterpret_cast<float2*>(y + vb * YS + n0) = make_float2(fb * acc[u][2], fb * acc[u][3]);
        }
      }
    }
    // the chunk's decay, read before the next chunk's gate scan
    const float dec = ALGO == ALGO_GDN ? eG[cn - 1] : 1.f;
    __syncthreads();

    // ---- (B) per column: the deltas by forward substitution, on warps 0-1
    //      (four partial sums per step); the preparing warps build this
    //      chunk's decayed keys, then prepare the next chunk
    if (tid < CB) {
      const float* am = am2 + b * C * FS;
      const float* wv = wv2 + b * C * CB;
      const float* wb = wb2 + b * C;
      float d[C];
#pragma unroll
      for (int i = 0; i < C; ++i) {
        d[i] = 0.f;
        if (i < cn) {
          float sj[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < i; ++j) sj[j & 3] = fmaf(am[i * FS + j], d[j], sj[j & 3]);
          d[i] = wb[i] * (wv[i * CB + tid] - y[i * YS + tid]) - ((sj[0] + sj[1]) + (sj[2] + sj[3]));
        }
        dch[i * DS + tid] = d[i];
      }
    } else if (prep) {
      build_kd(cn, lt, NP);
      if (ch + 1 < nchunks) {
        named_sync(1, NP);  // the keys of this chunk are read before the next lands
        prepare(ch + 1);
      }
    }
    __syncthreads();
    // ---- (C) outputs O = Y_q + F D on the tensor cores (warp w < NTN: the
    //      8 columns of tile w), then the rank-16 update of the state slice
    if (warp < NTN) {
      const float* fm = fm2 + b * C * FS;
      const int n0 = warp * 8;
      const float* yq = y + (C + fg) * YS + n0 + 2 * ft;
      const float2 q0 = *reinterpret_cast<const float2*>(yq);
      const float2 q1 = *reinterpret_cast<const float2*>(yq + 8 * YS);
      float acc[4] = {q0.x, q0.y, q1.x, q1.y};
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const float* fr = fm + fg * FS + 8 * ks + ft;
        const Tf32 af[4] = {tf32_split<false>(fr[0]), tf32_split<false>(fr[8 * FS]),
                            tf32_split<false>(fr[4]), tf32_split<false>(fr[8 * FS + 4])};
        const Tf32 bf[2] = {tf32_split<false>(dch[(8 * ks + ft) * DS + n0 + fg]),
                            tf32_split<false>(dch[(8 * ks + ft + 4) * DS + n0 + fg])};
        mma_split<false, false>(acc, af, bf);
      }
      const size_t col = (size_t)cb0 + n0 + 2 * ft;
      if (fg < cn) {
        const size_t ob = (((size_t)a0 + t0 + fg) * HV + h) * dv + col;
        st_f32(p.o, ob, p.in_dt, p.scale * acc[0]);
        st_f32(p.o, ob + 1, p.in_dt, p.scale * acc[1]);
      }
      if (fg + 8 < cn) {
        const size_t ob = (((size_t)a0 + t0 + fg + 8) * HV + h) * dv + col;
        st_f32(p.o, ob, p.in_dt, p.scale * acc[2]);
        st_f32(p.o, ob + 1, p.in_dt, p.scale * acc[3]);
      }
    }
    update(dec, decr2 + b * dk);
    __syncthreads();
  }

  // ---- the checkpoint takes the state (rounded to its dtype)
  for (int e = tid; e < dk * CQ; e += PT) {
    const int row = e / CQ, q4 = e - row * CQ;
    const float4 s4 = ld4(S + row * SS + 4 * q4);
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
