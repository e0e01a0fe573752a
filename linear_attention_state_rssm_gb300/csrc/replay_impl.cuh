// Replay kernel: decode (T = 1) and speculative verify (T <= 16) of one layer,
// with the ring-overflow fold fused in.
//
// One CTA of 4 warps per (request row, value head). The (slot, head)
// checkpoint tile S0 [dk][dv] streams through a ring of four shared-memory
// stages (8 KB row chunks, one bulk async copy each, full/empty mbarriers); a
// lane owns CW consecutive value columns of some rows of every chunk, so one
// vector load feeds CW x 2T fused multiply-adds. The stream is the only
// O(dk dv) work; everything else is arranged so that a CTA spends as little
// time as possible outside it.
//
// Ring keys are stored per value head, so every CTA reads and writes only its
// own records: a folding window (which writes positions [0, T) of the history
// it reads) waits for nothing but its own history copy. (LightLLM PR #1690
// "feat: add ReplaySSM state modes for GDN and KDA" shares one key buffer
// across the value heads of a key group and needs a counted cross-CTA barrier
// for that reason; its author notes the barrier has no progress guarantee.)
//
// Per CTA, with c = cursor[slot], fold = force || c + T > L:
//  0. bulk async copies: the window rows first (they need only the request
//     row), then the first tile chunks (once the slot is known) and the c
//     history records (once the cursor is known);
//  1. gates: history decay factors and in-window inclusive prefixes G_i;
//  2. window coefficients for j <= i < T (per key channel for KDA)
//        A_ij = beta_i sum_ch e^{G_i-G_j} k_j k_i   (j < i)
//        F_ij =        sum_ch e^{G_i-G_j} k_j q_i   (j <= i)
//     and, without a fold, history dot coefficients H[m][x] = k~_m . (e^{G_i} x)
//     for every window vector x in {k_i, q_i};
//  3. stream the tile: on a fold S0 <- e^{Gam} S0 + sum_m k~_m d_m^T (stored
//     back), and y_x = S0^T (e^{Gam_e + G_i} x) for all 2T vectors in one pass;
//  4. per value column: a_i, b_i = y + sum_m H d_m; the triangular solve
//     d_i = beta_i (v_i - a_i) - sum_{j<i} A_ij d_j (forward substitution of
//     (I + A) D = R) and o_i = scale (b_i + sum_{j<=i} F_ij d_j); the records of
//     the window go to ring positions base + i (base = fold ? 0 : c).
// A narrow GDN window without a fold runs steps 1-2 (and the history part of
// step 4) on two warps while the other two stream the tile: its mat-vec inputs
// are the raw window vectors, whose scalar decay goes on the column results.
// Every window sum runs over j <= i only, so a NaN or Inf at a later (rejected)
// position is never read by an earlier output: the causal selection is
// structural, never a multiplication by zero (SGLang fork PR jianc99/sglang#2,
// "Modifications" and the commit on fused selects).
#pragma once

#include "rssm_common.cuh"
#include "rssm_history.cuh"
#include "rssm_mma.cuh"
#include "rssm_tc.cuh"

#include <type_traits>

namespace rssm {

__device__ __forceinline__ float4 ld4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

// GDN, one warp: history decay factors (hf, hscal = {Gam, e^Gam}) and the
// in-window inclusive gate prefixes gp[i] = G_i of the raw gates wg (T <= 16
// lanes; wg itself is left as it is, the ring records copy it) with eG[i] =
// e^{G_i} and es[i] = e^{Gam_e + G_i} (Gam_e = Gam unless the window folds).
__device__ __forceinline__ void gdn_gates(int nh, int T, bool fold, float* hf, float* hscal,
                                          const float* wg, float* gp, float* eG, float* es,
                                          int lane) {
  if (nh > 0) {
    gdn_history_scan(nh, hf, hscal, lane);
  } else if (lane == 0) {
    hscal[0] = 0.f;
    hscal[1] = 1.f;
  }
  __syncwarp();
  const float gv = lane < T ? wg[lane] : 0.f;
  float incl = gv;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float t = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += t;
  }
  const float gam_e = fold ? 0.f : hscal[0];
  if (lane < T) {
    gp[lane] = incl;
    eG[lane] = __expf(incl);
    es[lane] = __expf(gam_e + incl);
  }
}

// Window coefficients A_ij (j < i) and F_ij (j <= i) of the pairs that fall to
// warp w of nw; lanes take float4 groups of key channels, then a warp sum.
// wg holds the inclusive gate prefixes (GDN [T], KDA [T][dk]).
template <int ALGO, int NT>
__device__ __forceinline__ void window_pairs(int T, int dk, const float* wk, const float* wq,
                                             const float* wg, const float* wb, float* am,
                                             float* fm, int w, int nw, int lane) {
  int pi = 0;
  for (int i = 0; i < T; ++i) {
    for (int j = 0; j <= i; ++j, ++pi) {
      if (pi % nw != w) continue;
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
        const float wgt = (ALGO == ALGO_GDN) ? __expf(wg[i] - wg[j]) : 1.f;
        fm[i * NT + j] = wgt * skq;
        am[i * NT + j] = (j < i) ? wb[i] * wgt * skk : 0.f;
      }
    }
  }
}

// Four consecutive ring keys (as stored: fp32, fp16 or bf16) as fp32.
__device__ __forceinline__ float4 ld4_key(const void* raw, size_t i, int dt) {
  if (dt == DT_F32) return *reinterpret_cast<const float4*>(static_cast<const float*>(raw) + i);
  const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(raw) + i);
  float2 a, b;
  if (dt == DT_F16) {
    a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  } else {
    a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  }
  return make_float4(a.x, a.y, b.x, b.y);
}

// Warp reduce-scatter of 32 values: afterwards lane l holds the sum over the
// warp of value l (31 shuffles in five independent levels).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int lvl = 0; lvl < 5; ++lvl) {
    const int off = 16 >> lvl, half = 16 >> lvl;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, off);
    }
  }
  return v[0];
}

// Decode (one window token), one warp: raw history dots hraw[m][0] = k_m . k,
// hraw[m][1] = k_m . q for m < nh (keys as stored in the ring, 16 records per
// pass of one reduce-scatter) and the window pair F_00 = k . q (A_00 = 0).
__device__ __forceinline__ void decode_dots(int nh, int dk, const void* hkraw, int rk_dt,
                                            const float* wk, const float* wq, float* hraw,
                                            float* am, float* fm, int lane) {
  const int c4 = 4 * lane;
  const bool has = c4 < dk;
  const float4 xk = has ? ld4(wk + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 xq = has ? ld4(wq + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int m0 = 0; m0 < nh; m0 += 16) {
    float v[32];
#pragma unroll
    for (int mm = 0; mm < 16; ++mm) {
      v[2 * mm] = 0.f;
      v[2 * mm + 1] = 0.f;
      if (m0 + mm < nh && has) {
        const float4 km = ld4_key(hkraw, (size_t)(m0 + mm) * dk + c4, rk_dt);
        v[2 * mm] = fmaf(km.x, xk.x, fmaf(km.y, xk.y, fmaf(km.z, xk.z, km.w * xk.w)));
        v[2 * mm + 1] = fmaf(km.x, xq.x, fmaf(km.y, xq.y, fmaf(km.z, xq.z, km.w * xq.w)));
      }
    }
    const float r = warp_reduce_scatter32(v, lane);
    if (m0 + lane / 2 < nh) hraw[2 * m0 + lane] = r;
  }
  const float kq = warp_sum(fmaf(xk.x, xq.x, fmaf(xk.y, xq.y, fmaf(xk.z, xq.z, xk.w * xq.w))));
  if (lane == 0) {
    fm[0] = kq;
    am[0] = 0.f;
  }
}

// GDN window coefficients, four consecutive threads per pair (i, j), j <= i:
// thread q of a pair takes the channels 4q + 16 s (so the four read one 64-byte
// span of a row) of copies of the window keys and queries whose rows are
// padded to `pitch` floats; two shuffles finish each sum. gp holds the
// inclusive gate prefixes. Every thread of the CTA (t < nt, nt a multiple of
// 32) runs the same number of rounds.
template <int NT>
__device__ __forceinline__ void window_pairs_flat(int T, int dk, const float* kp,
                                                  const float* qp, int pitch, const float* gp,
                                                  const float* wb, float* am, float* fm, int t,
                                                  int nt) {
  constexpr int S = 4;  // threads per pair
  const int npairs = T * (T + 1) / 2;
  for (int base = 0; base < npairs * S; base += nt) {
    const int pidx = (base + t) / S, q = (base + t) % S;
    const bool act = pidx < npairs;
    int i = 0, j = 0;
    float sk = 0.f, sq = 0.f;
    if (act) {
      while ((i + 1) * (i + 2) / 2 <= pidx) ++i;
      j = pidx - i * (i + 1) / 2;
      const float* kj = kp + j * pitch;
      const float* ki = kp + i * pitch;
      const float* qi = qp + i * pitch;
      float sk1 = 0.f, sq1 = 0.f;
      for (int c4 = 4 * q; c4 < dk; c4 += 8 * S) {
        const float4 a = ld4(kj + c4), b = ld4(ki + c4), c = ld4(qi + c4);
        sk = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, sk))));
        sq = fmaf(a.x, c.x, fmaf(a.y, c.y, fmaf(a.z, c.z, fmaf(a.w, c.w, sq))));
        if (c4 + 4 * S < dk) {
          const float4 a2 = ld4(kj + c4 + 4 * S), b2 = ld4(ki + c4 + 4 * S),
                       c2 = ld4(qi + c4 + 4 * S);
          sk1 = fmaf(a2.x, b2.x, fmaf(a2.y, b2.y, fmaf(a2.z, b2.z, fmaf(a2.w, b2.w, sk1))));
          sq1 = fmaf(a2.x, c2.x, fmaf(a2.y, c2.y, fmaf(a2.z, c2.z, fmaf(a2.w, c2.w, sq1))));
        }
      }
      sk += sk1;
      sq += sq1;
    }
#pragma unroll
    for (int off = 1; off < S; off <<= 1) {
      sk += __shfl_xor_sync(kFull, sk, off);
      sq += __shfl_xor_sync(kFull, sq, off);
    }
    if (act && q == 0) {
      const float wgt = __expf(gp[i] - gp[j]);
      fm[i * NT + j] = wgt * sq;
      am[i * NT + j] = (j < i) ? wb[i] * wgt * sk : 0.f;
    }
  }
}

// History dot coefficients hdot[m][v]: GDN: raw keys against raw window
// vectors, times hf[m] e^{G_i}; KDA: decayed keys against e^{G_i} x (xk, xq =
// yk, yq). Warp w takes the groups of 32 / NV records starting at record
// (w + k nw) 32 / NV; each lane sums its channels' products for every (record,
// vector) of the group and one reduce-scatter leaves the full sum of value l in
// lane l (31 shuffles per group instead of five per value).
template <int ALGO, int NT>
__device__ __forceinline__ void history_dots(int nh, int T, int dk, const float* hk,
                                             const float* xk, const float* xq, const float* hf,
                                             const float* eG, float* hdot, int w, int nw,
                                             int lane) {
  constexpr int NV = 2 * NT;
  static_assert(32 % NV == 0, "vectors per record divide the warp");
  constexpr int RPI = 32 / NV;  // records per reduce-scatter
  for (int m0 = w * RPI; m0 < nh; m0 += nw * RPI) {
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = 0.f;
    for (int c4 = 4 * lane; c4 < dk; c4 += 128) {
#pragma unroll
      for (int vv = 0; vv < NV; ++vv) {
        const int i = vv < NT ? vv : vv - NT;
        if (i < T) {
          const float4 x = ld4((vv < NT ? xk : xq) + i * dk + c4);
#pragma unroll
          for (int r = 0; r < RPI; ++r) {
            if (m0 + r < nh) {
              const float4 km = ld4(hk + (m0 + r) * dk + c4);
              float& a = v[r * NV + vv];
              a = fmaf(km.x, x.x, fmaf(km.y, x.y, fmaf(km.z, x.z, fmaf(km.w, x.w, a))));
            }
          }
        }
      }
    }
    const float sum = warp_reduce_scatter32(v, lane);
    const int m = m0 + lane / NV, vv = lane % NV, i = vv < NT ? vv : vv - NT;
    if (m < nh) {
      float hv = 0.f;
      if (i < T) hv = (ALGO == ALGO_GDN) ? sum * hf[m] * eG[i] : sum;
      hdot[m * NV + vv] = hv;
    }
  }
}

// Decode row order: with fmask holding one bit per request row (set for a row
// that folds; kWarps words, row = 32 word + bit) and F folding rows, the
// position-y CTA takes row y, except that the i-th non-folding row in front of
// F and the i-th folding row at or behind F trade places. Uniform over the CTA.
__device__ __forceinline__ int nth_row(const unsigned* fmask, int k, bool folding) {
  for (int w = 0; w < kWarps; ++w) {
    unsigned m = folding ? fmask[w] : ~fmask[w];
    const int n = __popc(m);
    if (k < n) {
      for (; k > 0; --k) m &= m - 1u;
      return w * 32 + __ffs(m) - 1;
    }
    k -= n;
  }
  return 0;  // not reached: k is below the count it is taken from
}

__device__ __forceinline__ int folding_below(const unsigned* fmask, int row) {
  int n = 0;
  for (int w = 0; w < (row >> 5); ++w) n += __popc(fmask[w]);
  if (row & 31) n += __popc(fmask[row >> 5] & ((1u << (row & 31)) - 1u));
  return n;
}

__device__ __forceinline__ int swap_rank(const unsigned* fmask, int y) {
  int F = 0;
  for (int w = 0; w < kWarps; ++w) F += __popc(fmask[w]);
  const bool fy = (fmask[y >> 5] >> (y & 31)) & 1u;
  if (y < F && !fy) {
    // the (y - folding_below(y))-th non-folding row in front of F
    return nth_row(fmask, folding_below(fmask, F) + (y - folding_below(fmask, y)), true);
  }
  if (y >= F && fy) return nth_row(fmask, folding_below(fmask, y) - folding_below(fmask, F), false);
  return y;
}

// Decode fold of a GDN window with at most 16 history records (LONG: up to
// kMmaFoldRecords) and 128 value columns on the tensor cores: each 16-row tile
// of the checkpoint is folded as
//     S <- e^Gam S + K~^T D~,   K~^T [16 rows x n records], D~ [n records x 128]
// with the keys transposed in hkt (row stride round4(n); records >= n read as
// zero; LONG with kdt 16-bit: the ring's keys transposed in place, which are
// exact in tf32), D~ = f_m d_m (f_m = hf[m], the decay from record m to the
// end of the history), the tile rows from the ring stage as the fp32 accumulator, the
// folded rows stored back to the checkpoint and fed to the mat-vec
// y_v = S^T x_v (x from xh [dk][2]). The D~ fragments of records [0, 16) stay
// in registers for the whole tile; those of later records (LONG) come from
// hd, which holds f_m d_m in place for m >= 16. Warp w owns value columns
// [32w, 32w + 32); y[nt][c][v] ends as the column sums of its columns
// 32w + 8nt + 2t + c in the lanes with g = 0. Keys from a 16-bit ring are
// exact in tf32 (EXACT_K).
template <typename ST, bool EXACT_K, bool LONG>
__device__ __forceinline__ bool fold_stream_mma(const TilePipe<ST>& pipe, const float* hkt,
                                                const float* hd, const float* hf, int n,
                                                float decay, const float* xh, ST* gtile, int tid,
                                                int warp, int lane, float (&y)[4][2][2],
                                                int kdt = DT_F32) {
  constexpr int DV = 128, NV = 2;
  const int g = lane >> 2, t = lane & 3, c0 = warp * 32, ks = round4(n);
  Tf32 bf[2][4][2];
#pragma unroll
  for (int kq = 0; kq < 2; ++kq) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int m = 8 * kq + t + 4 * hh;
        bf[kq][nt][hh] = tf32_split<false>(m < n ? hf[m] * hd[m * DV + c0 + 8 * nt + g] : 0.f);
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      y[nt][c][0] = 0.f;
      y[nt][c][1] = 0.f;
    }
  }
  // transposed key i: fp32, or (LONG, kdt 16-bit) the ring's own 16-bit keys
  auto key = [&](int i) -> float {
    if constexpr (LONG) {
      if (kdt != DT_F32) return ld_f32(hkt, (size_t)i, kdt);
    }
    return hkt[i];
  };
  // A fragment of records ma = 8 kq + t and ma + 4 for rows ra and ra + 8
  auto key_frag = [&](int ra, int kq, Tf32 (&a)[4]) {
    const int rb = ra + 8, ma = 8 * kq + t, mb = ma + 4;
    a[0] = tf32_split<EXACT_K>(ma < n ? key(ra * ks + ma) : 0.f);
    a[1] = tf32_split<EXACT_K>(ma < n ? key(rb * ks + ma) : 0.f);
    a[2] = tf32_split<EXACT_K>(mb < n ? key(ra * ks + mb) : 0.f);
    a[3] = tf32_split<EXACT_K>(mb < n ? key(rb * ks + mb) : 0.f);
  };
  bool ok = true;
  const int cr = pipe.tr.cr;
  for (int j = 0; j < pipe.tr.nchunk; ++j) {
    ok = __all_sync(kFull, pipe.wait(j) && ok);  // no store-back once a wait has run out
    const ST* stg = pipe.stage(j);
    for (int m0 = 0; m0 < cr; m0 += 16) {
      const int ra = j * cr + m0 + g, rb = ra + 8;  // this lane's two tile rows
      Tf32 af[2][4];
#pragma unroll
      for (int kq = 0; kq < 2; ++kq) key_frag(ra, kq, af[kq]);
      const float xa0 = xh[ra * NV], xa1 = xh[ra * NV + 1];
      const float xb0 = xh[rb * NV], xb1 = xh[rb * NV + 1];
      // fold of one n-tile's accumulator done: store it back, mat-vec
      auto finish = [&](int nt, const float (&acc)[4]) {
        const int col = c0 + 8 * nt + 2 * t;
        float wa[2] = {acc[0], acc[1]}, wb[2] = {acc[2], acc[3]};
        if (ok) {
          st_cols<ST, 2>(gtile + (size_t)ra * DV + col, wa);
          st_cols<ST, 2>(gtile + (size_t)rb * DV + col, wb);
        }
        // the mat-vec takes the stored (rounded) checkpoint values
        y[nt][0][0] = fmaf(wa[0], xa0, fmaf(wb[0], xb0, y[nt][0][0]));
        y[nt][0][1] = fmaf(wa[0], xa1, fmaf(wb[0], xb1, y[nt][0][1]));
        y[nt][1][0] = fmaf(wa[1], xa0, fmaf(wb[1], xb0, y[nt][1][0]));
        y[nt][1][1] = fmaf(wa[1], xa1, fmaf(wb[1], xb1, y[nt][1][1]));
      };
      if constexpr (!LONG) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int col = c0 + 8 * nt + 2 * t;
          float sa[2], sb[2];
          ld_cols<ST, 2>(stg + (size_t)(m0 + g) * DV + col, sa);
          ld_cols<ST, 2>(stg + (size_t)(m0 + g + 8) * DV + col, sb);
          float acc[4] = {decay * sa[0], decay * sa[1], decay * sb[0], decay * sb[1]};
          mma_split<EXACT_K, false>(acc, af[0], bf[0][nt]);
          if (n > 8) mma_split<EXACT_K, false>(acc, af[1], bf[1][nt]);
          finish(nt, acc);
        }
      } else {
        // all four n-tiles' accumulators stay live over the later records
        float acc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int col = c0 + 8 * nt + 2 * t;
          float sa[2], sb[2];
          ld_cols<ST, 2>(stg + (size_t)(m0 + g) * DV + col, sa);
          ld_cols<ST, 2>(stg + (size_t)(m0 + g + 8) * DV + col, sb);
          acc[nt][0] = decay * sa[0];
          acc[nt][1] = decay * sa[1];
          acc[nt][2] = decay * sb[0];
          acc[nt][3] = decay * sb[1];
          mma_split<EXACT_K, false>(acc[nt], af[0], bf[0][nt]);
          if (n > 8) mma_split<EXACT_K, false>(acc[nt], af[1], bf[1][nt]);
        }
        for (int kq = 2; 8 * kq < n; ++kq) {
          Tf32 ak[4];
          key_frag(ra, kq, ak);
          const int ma = 8 * kq + t, mb = ma + 4;
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            const int cb = c0 + 8 * nt + g;
            const Tf32 b[2] = {tf32_split<false>(ma < n ? hd[ma * DV + cb] : 0.f),
                               tf32_split<false>(mb < n ? hd[mb * DV + cb] : 0.f)};
            mma_split<EXACT_K, false>(acc[nt], ak, b);
          }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) finish(nt, acc[nt]);
      }
    }
    ok = pipe.done(j, tid, lane, ok) && ok;
  }
  // sum over the eight row groups (lanes with the same t)
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        float s = y[nt][c][v];
        s += __shfl_xor_sync(kFull, s, 4);
        s += __shfl_xor_sync(kFull, s, 8);
        s += __shfl_xor_sync(kFull, s, 16);
        y[nt][c][v] = s;
      }
    }
  }
  return ok;
}

// Tile stream of a GDN window with 8 NTN mat-vec vectors (four or eight
// tokens) and 128 value columns on the tensor cores, with the fold of a
// history of n records when FOLD. Both products take the value columns as
// the m index and the checkpoint rows as the reduction or n index, so the
// fold's accumulator fragment is the mat-vec's A fragment as it stands:
//     fold     S^T <- e^Gam S^T + D~^T K~     D~^T [128 x n records], K~ [n x rows]
//     mat-vec  Y^T += S^T X                   X [rows x 8 NTN]
// with D~ = f_m d_m (f_m = hf[m]). The raw keys (hkf, from frag_keys) and the
// window vectors X (xf, see x_slot) are stored in fragment order: one load
// per lane and step gives all of the step's fragments of each (of one group
// of 16 records, for the keys). The D~ fragments of records [0, 16) stay in
// registers for the whole tile; a longer history (LONG) reads those of each
// later group at every step from hd, which holds f_m d_m in place for m >= 16.
// The 128 / (16 MT) streaming warps own 16 MT columns each; lane (g, t) of warp
// w reads, for each of its MT / 2 column quads q, the four columns
// 16 MT w + 32 q + 4g .. + 3 of rows 2t and 2t + 1 of each eight-row step (one
// 16-byte load per row and quad; eight lanes cover 128 contiguous bytes); in
// m-tile mt (quad mt / 2), m = g is column 16 MT w + 32 (mt / 2) + 4g +
// 2 (mt % 2) and m = g + 8 the column after it; the step's reduction index
// k = t is row 2t and k = t + 4 row 2t + 1. Folded rows are stored back
// (rounded to the checkpoint dtype) and the mat-vec takes the stored values.
// y[4 (NTN mt + nt) + e] ends as the fragment of Y^T: e = 0 (column of m = g,
// vector 8 nt + 2t), 1 (same column, next vector), 2 and 3 (the next column).
// 16-bit checkpoint values, 16-bit inputs (EXACT_X) and 16-bit ring keys
// (EXACT_K) are exact in tf32. A fold runs on four warps (MT = 2).
template <typename ST, int NTN, int MT, bool FOLD, bool EXACT_X, bool EXACT_K, bool LONG>
__device__ __forceinline__ bool stream_mma(const TilePipe<ST>& pipe, const float* hkf,
                                           const float* hd, const float* hf, int n, float decay,
                                           const float* xf, ST* gtile, int tid, int warp,
                                           int lane, float (&y)[16]) {
  static_assert(NTN * MT * 4 <= 16 && (MT == 2 || MT == 4) && (!FOLD || MT == 2),
                "tensor-core stream shape");
  constexpr int DV = 128, NQ = MT / 2;
  constexpr bool EXACT_S = !std::is_same<ST, float>::value;
  const int g = lane >> 2, t = lane & 3, col = warp * 16 * MT + 4 * g;
  const float4* kf4 = reinterpret_cast<const float4*>(hkf);
  const int ng = FOLD && LONG ? (n + 15) >> 4 : 1;  // groups of 16 history records
  // fold A fragments of records m0 = t (+ 8 kq), m0 + 4 and value columns c,
  // c + 1: one float4 of hd row m holds columns [col, col + 4), i.e. both
  // m-tiles; f scales the rows that hd does not hold scaled
  auto d_frag = [&](int m0, float f0, float f1, Tf32 (&a)[2][4]) {
    const int m1 = m0 + 4;
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f), w = u;
    if (m0 < n) u = *reinterpret_cast<const float4*>(hd + m0 * DV + col);
    if (m1 < n) w = *reinterpret_cast<const float4*>(hd + m1 * DV + col);
    a[0][0] = tf32_split<false>(f0 * u.x);
    a[0][1] = tf32_split<false>(f0 * u.y);
    a[0][2] = tf32_split<false>(f1 * w.x);
    a[0][3] = tf32_split<false>(f1 * w.y);
    a[1][0] = tf32_split<false>(f0 * u.z);
    a[1][1] = tf32_split<false>(f0 * u.w);
    a[1][2] = tf32_split<false>(f1 * w.z);
    a[1][3] = tf32_split<false>(f1 * w.w);
  };
  Tf32 df[2][2][4];  // fold A fragments of records [0, 16): [record step][m-tile][4]
  if (FOLD && LONG) {
#pragma unroll
    for (int kq = 0; kq < 2; ++kq) {
      const int m0 = 8 * kq + t, m1 = m0 + 4;
      d_frag(m0, m0 < n ? hf[m0] : 0.f, m1 < n ? hf[m1] : 0.f, df[kq]);
    }
  } else if (FOLD) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int kq = 0; kq < 2; ++kq) {
        const int m0 = 8 * kq + t, m1 = m0 + 4, c0 = col + 2 * mt;
        const float f0 = m0 < n ? hf[m0] : 0.f, f1 = m1 < n ? hf[m1] : 0.f;
        df[kq][mt][0] = tf32_split<false>(m0 < n ? f0 * hd[m0 * DV + c0] : 0.f);
        df[kq][mt][1] = tf32_split<false>(m0 < n ? f0 * hd[m0 * DV + c0 + 1] : 0.f);
        df[kq][mt][2] = tf32_split<false>(m1 < n ? f1 * hd[m1 * DV + c0] : 0.f);
        df[kq][mt][3] = tf32_split<false>(m1 < n ? f1 * hd[m1 * DV + c0 + 1] : 0.f);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) y[e] = 0.f;
  bool ok = true;
  const int cr = pipe.tr.cr;
  for (int j = 0; j < pipe.tr.nchunk; ++j) {
    ok = pipe.wait(j) && ok;
    if (FOLD) ok = __all_sync(kFull, ok);  // no store-back once a wait has run out
    const ST* stg = pipe.stage(j);
    for (int kb = 0; kb < cr; kb += 8) {
      const int r0 = j * cr + kb + 2 * t, r1 = r0 + 1;  // this lane's two tile rows
      const int step = (j * cr + kb) >> 3;
      const int fi = step * 32 + lane;                    // fragment slot of this step
      float s0[NQ][4], s1[NQ][4];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        ld_cols<ST, 4>(stg + (size_t)(kb + 2 * t) * DV + col + 32 * q, s0[q]);
        ld_cols<ST, 4>(stg + (size_t)(kb + 2 * t + 1) * DV + col + 32 * q, s1[q]);
      }
      if constexpr (FOLD && !LONG) {
        const float4 k4 = kf4[fi];  // row kb + g: records t, t + 4, 8 + t, 12 + t
        const Tf32 kf[2][2] = {{tf32_split<EXACT_K>(k4.x), tf32_split<EXACT_K>(k4.y)},
                               {tf32_split<EXACT_K>(k4.z), tf32_split<EXACT_K>(k4.w)}};
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          float c[4] = {decay * s0[0][2 * mt], decay * s1[0][2 * mt], decay * s0[0][2 * mt + 1],
                        decay * s1[0][2 * mt + 1]};
          mma_split<false, EXACT_K>(c, df[0][mt], kf[0]);
          if (n > 8) mma_split<false, EXACT_K>(c, df[1][mt], kf[1]);
          s0[0][2 * mt] = c[0];
          s1[0][2 * mt] = c[1];
          s0[0][2 * mt + 1] = c[2];
          s1[0][2 * mt + 1] = c[3];
        }
        if (ok) {
          st_cols<ST, 4>(gtile + (size_t)r0 * DV + col, s0[0]);
          st_cols<ST, 4>(gtile + (size_t)r1 * DV + col, s1[0]);
        }
      } else if constexpr (FOLD) {
        float c[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          c[mt][0] = decay * s0[0][2 * mt];
          c[mt][1] = decay * s1[0][2 * mt];
          c[mt][2] = decay * s0[0][2 * mt + 1];
          c[mt][3] = decay * s1[0][2 * mt + 1];
        }
        {
          // row kb + g: records t, t + 4, t + 8, t + 12
          const float4 k4 = kf4[step * ng * 32 + lane];
          const Tf32 kf[2][2] = {{tf32_split<EXACT_K>(k4.x), tf32_split<EXACT_K>(k4.y)},
                                 {tf32_split<EXACT_K>(k4.z), tf32_split<EXACT_K>(k4.w)}};
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            mma_split<false, EXACT_K>(c[mt], df[0][mt], kf[0]);
            if (n > 8) mma_split<false, EXACT_K>(c[mt], df[1][mt], kf[1]);
          }
        }
        for (int q = 1; q < ng; ++q) {
          // records 16q + t, + t + 4, + t + 8, + t + 12
          const float4 k4 = kf4[(step * ng + q) * 32 + lane];
          const Tf32 kf[2][2] = {{tf32_split<EXACT_K>(k4.x), tf32_split<EXACT_K>(k4.y)},
                                 {tf32_split<EXACT_K>(k4.z), tf32_split<EXACT_K>(k4.w)}};
#pragma unroll
          for (int kq = 0; kq < 2; ++kq) {
            if (16 * q + 8 * kq < n) {
              Tf32 a[2][4];
              d_frag(16 * q + 8 * kq + t, 1.f, 1.f, a);
#pragma unroll
              for (int mt = 0; mt < 2; ++mt) mma_split<false, EXACT_K>(c[mt], a[mt], kf[kq]);
            }
          }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          s0[0][2 * mt] = c[mt][0];
          s1[0][2 * mt] = c[mt][1];
          s0[0][2 * mt + 1] = c[mt][2];
          s1[0][2 * mt + 1] = c[mt][3];
        }
        if (ok) {
          st_cols<ST, 4>(gtile + (size_t)r0 * DV + col, s0[0]);
          st_cols<ST, 4>(gtile + (size_t)r1 * DV + col, s1[0]);
        }
      }
      Tf32 xb[NTN][2];  // vectors 8 nt + g of rows 2t, 2t + 1
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
      for (int mt = 0; mt < MT; ++mt) {
        const int q = mt >> 1, h = 2 * (mt & 1);
        const Tf32 af[4] = {tf32_split<EXACT_S>(s0[q][h]), tf32_split<EXACT_S>(s0[q][h + 1]),
                            tf32_split<EXACT_S>(s1[q][h]), tf32_split<EXACT_S>(s1[q][h + 1])};
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
          float(&c)[4] = *reinterpret_cast<float(*)[4]>(&y[4 * (NTN * mt + nt)]);
          mma_split<EXACT_S, EXACT_X>(c, af, xb[nt]);
        }
      }
    }
    ok = pipe.done(j, tid, lane, ok) && ok;
  }
  return ok;
}

// The column sums of stream_mma -> red[v][col] (dv = 128), each (column,
// vector) from the one lane that holds it.
template <int NTN, int MT>
__device__ __forceinline__ void red_mma(float* red, const float (&y)[16], int warp, int lane) {
  constexpr int DV = 128;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt) {
      const int col = warp * 16 * MT + 32 * (mt >> 1) + 4 * g + 2 * (mt & 1), v = 8 * nt + 2 * t;
      const float* c = &y[4 * (NTN * mt + nt)];
      red[v * DV + col] = c[0];
      red[(v + 1) * DV + col] = c[1];
      red[v * DV + col + 1] = c[2];
      red[(v + 1) * DV + col + 1] = c[3];
    }
  }
}

// stream_mma with the exact-operand variants chosen by the input and ring-key
// dtypes.
template <typename ST, int NTN, int MT, bool FOLD, bool LONG = false>
__device__ __forceinline__ bool stream_mma_dt(const TilePipe<ST>& pipe, int in_dt, int rk_dt,
                                              const float* hkf, const float* hd, const float* hf,
                                              int n, float decay, const float* xf, ST* gtile,
                                              int tid, int warp, int lane, float (&y)[16]) {
  const bool xk = in_dt != DT_F32, kk = FOLD && rk_dt != DT_F32;
  if (xk) {
    return kk ? stream_mma<ST, NTN, MT, FOLD, true, true, LONG>(pipe, hkf, hd, hf, n, decay, xf,
                                                                gtile, tid, warp, lane, y)
              : stream_mma<ST, NTN, MT, FOLD, true, false, LONG>(pipe, hkf, hd, hf, n, decay, xf,
                                                                 gtile, tid, warp, lane, y);
  }
  return kk ? stream_mma<ST, NTN, MT, FOLD, false, true, LONG>(pipe, hkf, hd, hf, n, decay, xf,
                                                               gtile, tid, warp, lane, y)
            : stream_mma<ST, NTN, MT, FOLD, false, false, LONG>(pipe, hkf, hd, hf, n, decay, xf,
                                                                gtile, tid, warp, lane, y);
}

// Narrow windows keep four CTAs per SM (at most 128 registers per thread),
// eight-token windows three (two value columns per lane, a three-stage ring);
// the widest trade occupancy for their larger accumulator tiles.
// RAGGED: windows of different lengths from p.cu (verify widths only); the
// uniform kernels keep the window length a launch constant.
// TC: GDN windows of 3..8 tokens (NT 4 and 8) with 128 value columns stream on
// the 5th-generation tensor cores when p.tc is set (stream_tc).
// LONG: GDN decode and four- and eight-token windows on rings longer than 16
// records: their tensor-core folds take up to kMmaFoldRecords records (the
// kernels of shorter rings keep the tighter code of folds of at most 16).
template <int ALGO, typename ST, int NT, bool RAGGED, bool TC = false, bool LONG = false>
__global__ void __launch_bounds__(kThreads, NT <= 4 ? 4 : NT == 8 ? 3 : 2)
    replay_kernel(const ReplayParams p) {
  constexpr int NV = 2 * NT;             // mat-vec vectors: k_i at [0, NT), q_i at [NT, 2NT)
  constexpr int CW = quad_width(NT);     // value columns per lane in the tile stream
  constexpr int MR = fold_reg_records(NT);
  extern __shared__ __align__(128) unsigned char smem[];

  const int h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dk = p.dk, dv = p.dv, L = p.L, HV = p.HV, HK = p.HK;
  int T = p.T;  // this row's window (RAGGED: set once the row is known)
  const int kh = h / p.G;
  constexpr unsigned long long lim = kWaitLimitNs;

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
  float* hc = reinterpret_cast<float*>(smem + p.sm.hkraw);  // split windows, after widening
  // GDN scalars: es[i] = e^{Gam_e + G_i}, eG[i] = e^{G_i}, hscal = {Gam, e^Gam}.
  // KDA vectors: egam[ch] = e^{Gam[ch]}, gam[ch] = Gam[ch].
  float* es = scal;
  float* eG = scal + NT;
  float* hscal = scal + 2 * NT;
  float* gp = scal + 2 * NT + 4;  // GDN in-window gate prefixes
  float* egam = scal;
  float* gam = scal + dk;

  const int s_in = dtype_bytes(p.in_dt);
  const bool f32in = p.in_dt == DT_F32;
  const uint32_t qrow = (uint32_t)(dk * s_in), vrow = (uint32_t)(dv * s_in);

  // ---- copies of one request row: the window rows (they need only the row),
  //      the first tile chunks of a slot, the n history records of a slot
  auto tile_of = [&](int slot) {
    return static_cast<ST*>(p.state) + ((size_t)slot * HV + h) * dk * dv;
  };
  auto issue_window = [&](size_t t0) {
    mbar_expect_tx(&mbar[kMbarWin], T * (2 * qrow + vrow) +
                                        (ALGO == ALGO_KDA ? (uint32_t)(T * dk * 4) : 0u) +
                                        p.hook.extra(WH_WINDOW));
    for (int i = 0; i < T; ++i) {
      const size_t tok = t0 + i;
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
  };
  auto issue_hist = [&](int slot, int n) {
    const size_t sh = (size_t)slot * HV + h;
    // (KDA's gates land in hk, where they become the decayed keys)
    issue_history<ALGO>(n, dk, dv, p.ring_k, sh * L * dk, p.rk_dt, hkraw, p.ring_d, sh * L * dv,
                        p.rd_dt, p.rd_dt == DT_F32 ? static_cast<void*>(hd) : hdraw, p.ring_g,
                        sh * L * (ALGO == ALGO_GDN ? 1 : dk), ALGO == ALGO_KDA ? hk : hg,
                        &mbar[kMbarHist], p.hook.extra(WH_HIST));
  };
  // ---- row order. A folding row's CTAs live several times longer than the
  //      others; started last they would set the end of the launch. For
  //      decode (about one row in L folds) with up to kThreads rows, every CTA
  //      computes the same order from one load of every row's slot, cursor
  //      and force flag: each folding row behind position F (the number of
  //      folding rows) trades places with a non-folding row in front of it,
  //      the i-th with the i-th, and every other row keeps its place. Its own
  //      slot and cursor come out of the same loads. (Wider verify windows
  //      fold a large share of their rows, and the ranking's extra latency
  //      does not pay there.)
  const int y = blockIdx.y;
  int r = y, s, c = 0;
  bool have_c = false;
  if (NT == 1 && !RAGGED && p.B <= kThreads) {
    int2* rsc = reinterpret_cast<int2*>(smem + p.sm.rank);  // [kThreads] (slot, cursor)
    unsigned* fmask = reinterpret_cast<unsigned*>(rsc + kThreads);  // [kWarps] folding rows
    int sv = -1, cv = 0, fv = 0;
    if (tid < p.B) {
      sv = p.slot[tid];
      if (p.force != nullptr) fv = p.force[tid];
    }
    const bool sv_ok = sv >= 0 && sv < p.n_slots;
    if (sv_ok) cv = p.cursor[sv];
    const bool fr = sv_ok && (fv != 0 || cv + T > L);
    if (tid < p.B) rsc[tid] = make_int2(sv, cv);
    const unsigned m = __ballot_sync(kFull, fr);
    if (lane == 0) fmask[warp] = m;
    __syncthreads();
    r = swap_rank(fmask, y);
    const int2 e = rsc[r];
    s = e.x;
    c = e.y;
    have_c = true;
  } else {
    s = p.slot[r];
  }
  size_t tok0 = (size_t)r * T;
  if (RAGGED) {
    if (!row_window(p.cu, r, p.T, tok0, T)) {
      if (tid == 0 && h == 0) atomicOr(p.err, DEVERR_SEQLEN);
      return;
    }
    if (T == 0) return;  // no tokens for this row in this step: left as it is
  }

  // ---- 0. bulk async copies; one thread issues every copy of a barrier after
  //         registering its byte count.
  if (tid == 0) {
    mbar_init(&mbar[kMbarWin], 1);
    mbar_init(&mbar[kMbarHist], 1);
    TilePipe<ST>::init_full(mbar);
    if (TC) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&mbar[kMbarAFull + b], kWarps);
        mbar_init(&mbar[kMbarAEmpty + b], 1);
      }
      mbar_init(&mbar[kMbarFoldTc], 1);
      mbar_init(&mbar[kMbarYDone], 1);
    }
    fence_mbar_init();
    issue_window(tok0);
  }
  float wbeta = 0.f, wgate = 0.f;
  if (tid < T) {
    wbeta = p.beta[(tok0 + tid) * HV + h];
    if (ALGO == ALGO_GDN) wgate = p.g[(tok0 + tid) * HV + h];
  }
  if (s < 0 || s >= p.n_slots) {
    // null row (or a slot out of range): let the window copies land, leave
    if (tid == 0) {
      if (s >= p.n_slots && h == 0) atomicOr(p.err, DEVERR_SLOT);
      mbar_wait_bounded(&mbar[kMbarWin], 0, lim);
    }
    return;
  }
  ST* gtile = tile_of(s);
  const TilePipe<ST> pipe(reinterpret_cast<ST*>(smem + p.sm.ring), mbar, gtile, dk, dv,
                          (int)p.sm.ns, p.hook);
  if (tid == 0) pipe.prime();
  if (!have_c) c = p.cursor[s];
  if (c < 0 || c > L) {
    if (tid == 0) {
      if (h == 0) atomicOr(p.err, DEVERR_CURSOR);
      mbar_wait_bounded(&mbar[kMbarWin], 0, lim);
      pipe.drain();
    }
    return;
  }
  // fold decision (uniform over the CTA)
  const bool fold = (p.force != nullptr && p.force[r] != 0) || (c + T > L);
  const int base = fold ? 0 : c;
  const int nh = c;
  // the 5th-generation tensor-core stream: one thread per value column
  const bool tc = TC && p.tc != 0 && dv == kThreads && dk % 32 == 0 &&
                  (!fold || (nh <= 16 && L >= 16));
  const bool split = can_split(ALGO, NT) && !fold && !tc;
  const int sw = split ? kSplitWarps : kWarps;  // warps that stream the tile
  // Four- and eight-token GDN windows with 128 value columns stream on the
  // tensor cores (mat-vec inputs and fold keys in fragment order, column sums
  // in ymm); a fold there takes at most 16 records (LONG: up to
  // kMmaFoldRecords, as many groups of 16 as the key buffer holds).
  constexpr bool kMmaNT = ALGO == ALGO_GDN && (NT == 4 || NT == 8);
  constexpr int NTN = NV >= 8 ? NV / 8 : 1;  // n-tiles of eight vectors
  constexpr int kFoldMax = LONG ? kMmaFoldRecords : 16;
  const bool mmas = !TC && kMmaNT && dv == 128 && pipe.tr.cr % 8 == 0 &&
                    (!fold || (LONG ? nh <= kFoldMax && ((nh + 15) & ~15) <= round4(L)
                                    : nh <= 16 && L >= 16));
  const size_t kbase = ((size_t)s * HV + h) * L * dk;
  const size_t dbase = ((size_t)s * HV + h) * L * dv;
  const size_t gbase = ((size_t)s * HV + h) * L * (ALGO == ALGO_GDN ? 1 : dk);
  if (tid == 0) {
    pipe.init_empty(sw);
    if (nh > 0) issue_hist(s, nh);
  }
  // GDN history gates: loaded now, stored once the window has landed
  float hgate = 0.f;
  if (ALGO == ALGO_GDN && tid < nh) hgate = p.ring_g[gbase + tid];
  __syncthreads();  // every mbarrier is initialised

  // ---- window rows -> fp32; GDN mat-vec inputs xh[ch][v] are the raw window
  //      vectors (their scalar decay goes on the column results)
  bool copies_ok = mbar_wait_bounded(&mbar[kMbarWin], 0, lim);
  if (!f32in) {
    if constexpr (NT >= 4) {  // (dk and dv are multiples of 32)
      widen16x8(wq, wraw, T * dk, p.in_dt, tid, kThreads);
      widen16x8(wk, wraw + T * qrow, T * dk, p.in_dt, tid, kThreads);
      widen16x8(wv, wraw + 2 * T * qrow, T * dv, p.in_dt, tid, kThreads);
    } else {
      widen16(wq, wraw, T * dk, p.in_dt, tid, kThreads);
      widen16(wk, wraw + T * qrow, T * dk, p.in_dt, tid, kThreads);
      widen16(wv, wraw + 2 * T * qrow, T * dv, p.in_dt, tid, kThreads);
    }
  }
  if (TC && tc) {
    // K-major X [16 vectors x dk rows]; fp32 inputs split into hi (xh) and lo
    const void* qsrc = f32in ? static_cast<const void*>(wq) : wraw;
    const void* ksrc = f32in ? static_cast<const void*>(wk) : wraw + T * qrow;
    float* xl = reinterpret_cast<float*>(smem + p.sm.xl);
    for (int e = tid; e < dk * kTcN; e += kThreads) {
      int ch, vv;
      x_slot_tc(e, ch, vv);
      const int i = vv < NT ? vv : vv - NT;
      const float x = vv < NV && i < T ? ld_f32(vv < NT ? ksrc : qsrc, (size_t)i * dk + ch, p.in_dt)
                                       : 0.f;
      if (f32in) {
        xh[e] = tf32_hi(x);
        xl[e] = x - tf32_hi(x);
      } else {
        xh[e] = x;
      }
    }
    fence_async_smem();
  } else if (ALGO == ALGO_GDN && mmas) {
    if constexpr (kMmaNT) {
      // fragment order (x_slot): a lane-step of 2 NTN consecutive slots holds
      // the channel pair (c, c + 1) of NTN vectors, one paired load each
      const void* qsrc = f32in ? static_cast<const void*>(wq) : wraw;
      const void* ksrc = f32in ? static_cast<const void*>(wk) : wraw + T * qrow;
      constexpr int CPL = 2 * NTN;
      for (int st = tid; st < dk * NV / CPL; st += kThreads) {
        const int ln = st & 31, c = 8 * (st >> 5) + 2 * (ln & 3), vl = ln >> 2;
        float x[CPL];
#pragma unroll
        for (int m = 0; m < NTN; ++m) {
          const int v = 8 * m + vl, i = v < NT ? v : v - NT;
          float2 pr = make_float2(0.f, 0.f);
          if (i < T) pr = ld2_f32(v < NT ? ksrc : qsrc, (size_t)i * dk + c, p.in_dt);
          x[2 * m] = pr.x;
          x[2 * m + 1] = pr.y;
        }
        if constexpr (CPL == 4) {
          *reinterpret_cast<float4*>(xh + 4 * st) = make_float4(x[0], x[1], x[2], x[3]);
        } else {
          *reinterpret_cast<float2*>(xh + 2 * st) = make_float2(x[0], x[1]);
        }
      }
    }
  } else if (ALGO == ALGO_GDN) {
    const void* qsrc = f32in ? static_cast<const void*>(wq) : wraw;
    const void* ksrc = f32in ? static_cast<const void*>(wk) : wraw + T * qrow;
    for (int e = tid; e < dk * NV; e += kThreads) {
      // slot e holds (row ch, vector vv), row-major
      const int ch = e / NV, vv = e - ch * NV;
      const int i = vv < NT ? vv : vv - NT;
      xh[e] = i < T ? ld_f32(vv < NT ? ksrc : qsrc, (size_t)i * dk + ch, p.in_dt) : 0.f;
    }
  }
  if (tid < T) {
    wb[tid] = wbeta;
    if (ALGO == ALGO_GDN) wg[tid] = wgate;
  }
  if (ALGO == ALGO_GDN) {
    if (tid < nh) hf[tid] = hgate;
    for (int m = tid + kThreads; m < nh; m += kThreads) hf[m] = p.ring_g[gbase + m];
  }
  // A folding window streams its fold right away: its history must be here.
  if (fold && nh > 0) copies_ok = mbar_wait_bounded(&mbar[kMbarHist], 0, lim) && copies_ok;
  if (!__syncthreads_and(copies_ok)) {
    // a copy of the window (or of a folding window's history) did not arrive
    // in time: the row is left as it is
    if (tid == 0) {
      atomicOr(p.err, DEVERR_TIMEOUT);
      mbar_wait_bounded(&mbar[kMbarWin], 0, lim);
      if (nh > 0) mbar_wait_bounded(&mbar[kMbarHist], 0, lim);
      pipe.drain();
    }
    return;
  }

  // tensor memory of the tensor-core stream (freed at the end of the kernel)
  TcStream tcs{};
  if (TC && tc) {
    uint32_t* tslot = reinterpret_cast<uint32_t*>(&mbar[kMbarTmem]);
    if (warp == 0) {
      __syncwarp();
      tmem_alloc(tslot);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tcs.tbase = *tslot;
    tcs.afull = &mbar[kMbarAFull];
    tcs.aempty = &mbar[kMbarAEmpty];
    tcs.fbar = &mbar[kMbarFoldTc];
    tcs.ydone = &mbar[kMbarYDone];
    tcs.xh = xh;
    tcs.xl = f32in ? reinterpret_cast<const float*>(smem + p.sm.xl) : nullptr;
    tcs.kh = hk;
    tcs.kl = p.rk_dt == DT_F32 ? reinterpret_cast<const float*>(smem + p.sm.kl) : nullptr;
  }

  // ---- records that need no result of the solve: keys, gates and betas at
  //      ring positions base + i (KDA's raw gates were turned into prefixes in
  //      shared memory: they are copied from the input). A window that does
  //      not fold writes them now, past the history it reads ([0, c)).
  auto write_kgb = [&]() {
    for (int ch = tid; ch < dk; ch += kThreads) {
      for (int i = 0; i < T; ++i) {
        st_f32(p.ring_k, kbase + (size_t)(base + i) * dk + ch, p.rk_dt, wk[i * dk + ch]);
        if (ALGO == ALGO_KDA) {
          p.ring_g[gbase + (size_t)(base + i) * dk + ch] = p.g[((tok0 + i) * HV + h) * dk + ch];
        }
      }
    }
    if (tid < T) {
      p.ring_beta[((size_t)s * HV + h) * L + base + tid] = wb[tid];
      if (ALGO == ALGO_GDN) p.ring_g[gbase + base + tid] = wg[tid];
    }
  };
  if (!fold) write_kgb();

  const QuadLayout qlay(dv, CW, sw);
  const QuadLane qlane(qlay, CW, warp, lane);
  bool mma_fold = false;     // decode fold on the tensor cores (column sums in ymma)
  float ymma[4][2][2];
  float ymm[16];             // column sums of the tensor-core stream (stream_mma)
  float acc[NV][CW];
#pragma unroll
  for (int vv = 0; vv < NV; ++vv) {
#pragma unroll
    for (int cc = 0; cc < CW; ++cc) acc[vv][cc] = 0.f;
  }

  if (split) {
    if (warp < sw) {
      // ---- 3. stream warps: y_x = S0^T x for the raw window vectors (decode
      //         with 128 value columns takes the unrolled fixed-geometry loop)
      constexpr int kFixedRpl = 8192 / (128 * (int)sizeof(ST)) / (2 * kSplitWarps / 2);
      if (NT == 1 && dv == 128 && qlane.rstep == kSplitWarps &&
          pipe.tr.cr / qlane.rstep == kFixedRpl) {
        copies_ok = stream_fixed<ST, NV, CW, kFixedRpl, kSplitWarps, 128>(pipe, qlane, acc, xh,
                                                                         tid, lane) &&
                    copies_ok;
      } else if (mmas) {
        if constexpr (kMmaNT && NT == 4) {
          copies_ok = stream_mma_dt<ST, NTN, 4, false>(pipe, p.in_dt, p.rk_dt, hk, hd, hf, 0, 1.f,
                                                       xh, gtile, tid, warp, lane, ymm) &&
                      copies_ok;
        }
      } else {
        copies_ok = stream_quads<ALGO, ST, NV, CW, MR, false>(pipe, qlane, acc, gtile, dk, dv, 0,
                                                              hk, hd, hf, 1.f, egam, xh, tid,
                                                              lane) &&
                    copies_ok;
      }
    } else {
      // ---- 1, 2 and the history part of 4 on the other warps
      const int ht = tid - sw * 32, hw = warp - sw;
      const int nht = kThreads - sw * 32, nhw = kWarps - sw;
      // decode: the gate scan on one history warp while the other takes every
      // raw history dot straight from the ring keys (gate factors go on in the
      // column correction below)
      const bool decode1 = NT == 1 && nhw == 2;
      if (nh > 0) {
        copies_ok = mbar_wait_bounded(&mbar[kMbarHist], 0, lim) && copies_ok;
        if (!decode1) widen_keys(hk, hkraw, nh * dk, p.rk_dt, ht, nht);
        if (p.rd_dt != DT_F32) widen16(hd, hdraw, nh * dv, p.rd_dt, ht, nht);
      }
      if (decode1) {
        if (p.rd_dt != DT_F32) named_sync(1, nht);
        if (hw == 0) {
          gdn_gates(nh, T, false, hf, hscal, wg, gp, eG, es, lane);
        } else {
          decode_dots(nh, dk, hkraw, p.rk_dt, wk, wq, hdot, am, fm, lane);
        }
      } else {
        named_sync(1, nht);
        if (hw == 0) gdn_gates(nh, T, false, hf, hscal, wg, gp, eG, es, lane);
        named_sync(1, nht);
        window_pairs<ALGO, NT>(T, dk, wk, wq, gp, wb, am, fm, hw, nhw, lane);
        history_dots<ALGO, NT>(nh, T, dk, hk, wk, wq, hf, eG, hdot, hw, nhw, lane);
      }
      named_sync(1, nht);
      // history correction of every column: hc[v][col] = sum_m H[m][v] d_m[col]
      // (hc reuses the landing zone of the keys, widened above)
      for (int col = ht; col < dv; col += nht) {
        float y[NV];
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) y[vv] = 0.f;
        for (int m = 0; m < nh; ++m) {
          const float dm = decode1 ? hd[m * dv + col] * hf[m] : hd[m * dv + col];
#pragma unroll
          for (int vv = 0; vv < NV; ++vv) y[vv] = fmaf(hdot[m * NV + vv], dm, y[vv]);
        }
        const float f = decode1 ? eG[0] : 1.f;
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) hc[vv * dv + col] = f * y[vv];
      }
    }
  } else {
    // A wide GDN window without a fold streams first, while its history lands.
    const bool early = ALGO == ALGO_GDN && !fold;
    if (early && TC && tc) {
      if constexpr (TC) {
        copies_ok = stream_tc<ST, false>(pipe, tcs, gtile, 1.f, tid, warp, lane) && copies_ok;
      }
    } else if (early) {
      if (mmas) {
        if constexpr (kMmaNT) {
          copies_ok = stream_mma_dt<ST, NTN, 2, false>(pipe, p.in_dt, p.rk_dt, hk, hd, hf, 0, 1.f,
                                                       xh, gtile, tid, warp, lane, ymm) &&
                      copies_ok;
        }
      } else {
        copies_ok = stream_quads<ALGO, ST, NV, CW, MR, false>(pipe, qlane, acc, gtile, dk, dv, 0,
                                                              hk, hd, hf, 1.f, egam, xh, tid,
                                                              lane) &&
                    copies_ok;
      }
    }
    if (nh > 0 && !fold) copies_ok = mbar_wait_bounded(&mbar[kMbarHist], 0, lim) && copies_ok;
    if (nh > 0) {
      // (KDA reads fp16 deltas as they landed)
      if (p.rd_dt != DT_F32 && ALGO == ALGO_GDN) widen16(hd, hdraw, nh * dv, p.rd_dt, tid, kThreads);
      if (ALGO == ALGO_GDN) {
        if (fold && TC && tc) {
          float* kl = p.rk_dt == DT_F32 ? reinterpret_cast<float*>(smem + p.sm.kl) : nullptr;
          tc_fold_keys(hk, kl, hkraw, nh, dk, p.rk_dt, tid, kThreads);
          fence_async_smem();
        } else if (fold && LONG && p.sm.kip) {
          // (every fold of this plan runs on the tensor cores: mma_fold below)
          transpose_keys16_inplace(reinterpret_cast<uint16_t*>(hkraw), nh, dk, tid, kThreads);
        } else if (fold && mmas) {
          if (LONG) {
            frag_keys(hk, hkraw, nh, dk, p.rk_dt, tid, kThreads);
          } else {
            frag_keys16(hk, hkraw, nh, dk, p.rk_dt, tid, kThreads);
          }
        } else if (fold) {
          transpose_keys(hk, hkraw, nh, dk, p.rk_dt, tid, kThreads);
        } else {
          widen_keys(hk, hkraw, nh * dk, p.rk_dt, tid, kThreads);
        }
      }
    }
    __syncthreads();

    // Windows of four or more tokens compute the GDN window coefficients one
    // thread per pair on padded copies of the window keys and queries in the
    // drained tile ring: a window without a fold has streamed already; a
    // folding one computes them after its stream (only the per-column solve
    // needs them).
    const int wpitch = dk + 4;
    float* kpad = reinterpret_cast<float*>(smem + p.sm.ring);
    float* qpad = kpad + T * wpitch;
    const bool flat = ALGO == ALGO_GDN && NT >= 4 &&
                      (uint32_t)(8 * T * wpitch) <= pipe.tr.ns * pipe.tr.chunk_bytes;
    auto pad_window = [&]() {
      for (int e = tid; e < T * dk / 4; e += kThreads) {
        const int i = e / (dk / 4), c4 = 4 * (e - i * (dk / 4));
        *reinterpret_cast<float4*>(kpad + i * wpitch + c4) = ld4(wk + i * dk + c4);
        *reinterpret_cast<float4*>(qpad + i * wpitch + c4) = ld4(wq + i * dk + c4);
      }
    };

    // ---- 1. gates
    if (ALGO == ALGO_GDN) {
      if (warp == 0) gdn_gates(nh, T, fold, hf, hscal, wg, gp, eG, es, lane);
      if (flat && early) pad_window();
    } else {
      // one thread per key channel: decayed history keys k~ (in hk, [nh][dk],
      // over the record gates that landed there), history decay, window
      // prefix, scaled window vectors
      for (int ch = tid; ch < dk; ch += kThreads) {
        float suf = 0.f;
        for (int m = nh - 1; m >= 0; --m) {
          const float kraw = ld_f32(hkraw, (size_t)m * dk + ch, p.rk_dt);
          const float gm = hk[m * dk + ch];
          hk[m * dk + ch] = kraw * __expf(suf);
          suf += gm;
        }
        gam[ch] = suf;
        egam[ch] = __expf(suf);
        const float gam_e = fold ? 0.f : suf;
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

    // ---- 2. window coefficients A, F (j <= i only) and history dot coefficients
    if (flat) {
      if (early) window_pairs_flat<NT>(T, dk, kpad, qpad, wpitch, gp, wb, am, fm, tid, kThreads);
    } else {
      window_pairs<ALGO, NT>(T, dk, wk, wq, ALGO == ALGO_GDN ? gp : wg, wb, am, fm, warp, kWarps,
                             lane);
    }
    if (!fold) {
      history_dots<ALGO, NT>(nh, T, dk, hk, ALGO == ALGO_GDN ? wk : yk,
                             ALGO == ALGO_GDN ? wq : yq, hf, eG, hdot, warp, kWarps, lane);
    }

    // ---- 3. stream the checkpoint tile (unless done early): fold, then S^T x
    if (!early) {
      __syncthreads();
      if (fold && nh > 0) {
        if constexpr (NT == 1 && ALGO == ALGO_GDN) {
          mma_fold = nh <= kFoldMax && dv == 128 && pipe.tr.cr % 16 == 0;
        }
        // the tensor-core folds read the deltas of records m >= 16 as f_m d_m,
        // scaled in place over the gate factors of step 1 (a folding window
        // reads hd nowhere else)
        if (LONG && (mmas || mma_fold) && nh > 16) {
          for (int e = 16 * (dv / 4) + tid; e < nh * (dv / 4); e += kThreads) {
            const float f = hf[e / (dv / 4)];
            float4 d4 = reinterpret_cast<float4*>(hd)[e];
            d4.x *= f;
            d4.y *= f;
            d4.z *= f;
            d4.w *= f;
            reinterpret_cast<float4*>(hd)[e] = d4;
          }
          __syncthreads();
        }
        if (TC && tc) {
          if constexpr (TC) {
            tc_fold_a(tcs, hd, hf, nh, dv, tid, warp);
            tc_fence_before();
            __syncthreads();
            copies_ok = stream_tc<ST, true>(pipe, tcs, gtile, hscal[1], tid, warp, lane) &&
                        copies_ok;
          }
        } else if (mmas) {
          if constexpr (kMmaNT) {
            copies_ok = stream_mma_dt<ST, NTN, 2, true, LONG>(pipe, p.in_dt, p.rk_dt, hk, hd, hf,
                                                              nh, hscal[1], xh, gtile, tid, warp,
                                                              lane, ymm) &&
                        copies_ok;
          }
        } else if (mma_fold) {
          if constexpr (NT == 1 && ALGO == ALGO_GDN) {
            const bool kip = LONG && p.sm.kip;
            const float* hkt = kip ? reinterpret_cast<const float*>(hkraw) : hk;
            copies_ok = (p.rk_dt == DT_F32
                             ? fold_stream_mma<ST, false, LONG>(pipe, hkt, hd, hf, nh, hscal[1], xh,
                                                                gtile, tid, warp, lane, ymma)
                             : fold_stream_mma<ST, true, LONG>(pipe, hkt, hd, hf, nh, hscal[1], xh,
                                                               gtile, tid, warp, lane, ymma,
                                                               kip ? p.rk_dt : (int)DT_F32)) &&
                        copies_ok;
          }
        } else {
          copies_ok = stream_quads<ALGO, ST, NV, CW, MR, true>(
                          pipe, qlane, acc, gtile, dk, dv, nh, hk, hd, hf, hscal[1], egam, xh, tid,
                          lane, ALGO == ALGO_KDA ? p.rd_dt : (int)DT_F32) &&
                      copies_ok;
        }
      } else if (TC && tc) {
        if constexpr (TC) {
          copies_ok = stream_tc<ST, false>(pipe, tcs, gtile, 1.f, tid, warp, lane) && copies_ok;
        }
      } else if (mmas) {
        if constexpr (kMmaNT) {
          copies_ok = stream_mma_dt<ST, NTN, 2, false>(pipe, p.in_dt, p.rk_dt, hk, hd, hf, 0, 1.f,
                                                       xh, gtile, tid, warp, lane, ymm) &&
                      copies_ok;
        }
      } else {
        copies_ok = stream_quads<ALGO, ST, NV, CW, MR, false>(pipe, qlane, acc, gtile, dk, dv, 0,
                                                              hk, hd, hf, 1.f, egam, xh, tid,
                                                              lane) &&
                    copies_ok;
      }
      if (flat) {
        __syncthreads();  // the ring is drained
        pad_window();
        __syncthreads();
        window_pairs_flat<NT>(T, dk, kpad, qpad, wpitch, gp, wb, am, fm, tid, kThreads);
      }
    }
  }
  // partial column sums of the warp row groups -> shared memory (the ring is
  // free once every warp has consumed the last chunk); the tensor-core streams
  // leave whole column sums, in the first row-group slot
  __syncthreads();
  if (TC && tc) {
    if constexpr (TC) {
      copies_ok = tc_read_y<NV>(tcs, red, dv, tid, warp) && copies_ok;
    }
  } else if (mma_fold) {
    if constexpr (NT == 1) {
      if (lane < 4) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int col = warp * 32 + 8 * nt + 2 * lane + cc;
            red[0 * dv + col] = ymma[nt][cc][0];
            red[1 * dv + col] = ymma[nt][cc][1];
          }
        }
      }
    }
  } else if (mmas) {
    if constexpr (kMmaNT) {
      if constexpr (can_split(ALGO, NT)) {
        if (!split) {
          red_mma<NTN, 2>(red, ymm, warp, lane);
        } else if (warp < sw) {
          red_mma<NTN, 4>(red, ymm, warp, lane);
        }
      } else {
        red_mma<NTN, 2>(red, ymm, warp, lane);
      }
    }
  } else if (warp < sw && qlane.first) {
#pragma unroll
    for (int vv = 0; vv < NV; ++vv) {
#pragma unroll
      for (int cc = 0; cc < CW; ++cc) red[(qlane.rg * NV + vv) * dv + qlane.col0 + cc] = acc[vv][cc];
    }
  }
  // every wait of the CTA succeeded, or the row's outputs and records are not
  // written (a folding row may have stored back the chunks folded before the
  // wait that failed)
  const bool all_ok = __syncthreads_and(copies_ok);

  // a folding window writes its keys, gates and betas only now: positions
  // [0, T) are the ones its history was read from
  if (fold && all_ok) write_kgb();

  // ---- 4. per value column: corrections, triangular solve, outputs, deltas
  //      (the tensor-core streams leave whole column sums in row group 0)
  const int rgu = (tc || mma_fold || mmas) ? 1 : qlay.rgw;
  if (tid < dv && all_ok) {
    const int col = tid;
    float y[NV];
#pragma unroll
    for (int vv = 0; vv < NV; ++vv) {
      float sum = 0.f;
      for (int g2 = 0; g2 < rgu; ++g2) sum += red[(g2 * NV + vv) * dv + col];
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
    if (split) {
#pragma unroll
      for (int vv = 0; vv < NV; ++vv) y[vv] += hc[vv * dv + col];
    } else if (!fold) {
      const bool d16 = ALGO == ALGO_KDA && p.rd_dt != DT_F32;
      for (int m = 0; m < nh; ++m) {
        const float dm = d16 ? __half2float(reinterpret_cast<const __half*>(hd)[m * dv + col])
                             : hd[m * dv + col];
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
  if (all_ok) {
    if (h == 0 && tid == 0 && p.fold_out != nullptr) p.fold_out[r] = fold ? 1 : 0;
  } else if (tid == 0) {
    atomicOr(p.err, DEVERR_TIMEOUT);
    // copies that did not arrive in time get a second bounded wait before the
    // CTA leaves (the window's waited above, or the row would not be here)
    if (nh > 0) mbar_wait_bounded(&mbar[kMbarHist], 0, lim);
    pipe.drain_tail();
  }
  if (TC && tc) {
    // every read of tensor memory is done (tc_read_y waited for the last MMA)
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tcs.tbase);
    }
  }
}

}  // namespace rssm
