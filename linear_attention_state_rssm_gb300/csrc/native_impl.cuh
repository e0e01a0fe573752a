// Native fused-recurrent decode: the state is read and written every token.
//
// This is the path ReplaySSM replaces (LightLLM PR #1690 "feat: add ReplaySSM
// state modes for GDN and KDA", PR description: the native mode keeps the
// recurrent state current by writing it back each step; SGLang fork PR
// jianc99/sglang#2, "Motivation": per-draft state snapshots). It is built here
// as the comparison point of the replay kernel on the same hardware and
// shapes: one decode token per (request row, value head) applied to the
// store's checkpoint tile as the live state,
//     S <- decay(g) S;  d = beta (v - S^T k);  S <- S + k d^T;  o = scale S^T q,
// with decay e^g (GDN) or diag(e^g) (KDA). The ring and the cursor are not
// used.
//
// One CTA of 4 warps per (row, value head). The whole tile lands in shared
// memory (one bulk copy and one mbarrier per 8 KB chunk); pass 1 computes
// S^T (decay k) and S^T (decay q) for the tile with the replay kernel's
// 4-column lanes; then d = beta (v - .) and o = scale (S^T (decay q) + (k.q) d);
// pass 2 writes decay(row) S + k d^T back from shared memory, rounded to the
// state dtype.
#pragma once

#include "rssm_common.cuh"
#include "rssm_history.cuh"

namespace rssm {

// The whole tile in shared memory: chunk j in stage j, waited on once.
template <typename ST>
struct WholeTile {
  const ST* ring;
  uint64_t* full;
  TileRing tr;
  int dv;
  __device__ __forceinline__ const ST* stage(int j) const {
    return ring + (size_t)j * tr.cr * dv;
  }
  __device__ __forceinline__ bool wait(int j) const { return mbar_wait_bounded(&full[j], 0); }
  __device__ __forceinline__ bool done(int, int, int, bool) const { return true; }
};

template <int ALGO, typename ST>
__global__ void __launch_bounds__(kThreads) native_decode_kernel(const ReplayParams p,
                                                                 const NativeSmem sm) {
  constexpr int NV = 2, CW = 4;
  extern __shared__ __align__(128) unsigned char smem[];
  const int h = blockIdx.x, r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dk = p.dk, dv = p.dv, HV = p.HV, HK = p.HK, kh = h / p.G;

  const int s = p.slot[r];
  if (s < 0) return;
  if (s >= p.n_slots) {
    if (h == 0 && tid == 0) atomicOr(p.err, DEVERR_SLOT);
    return;
  }
  ST* gtile = static_cast<ST*>(p.state) + ((size_t)s * HV + h) * dk * dv;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + sm.mbar);  // [0]: window, [1 + j]: chunk j
  ST* ring = reinterpret_cast<ST*>(smem + sm.ring);
  float* wq = reinterpret_cast<float*>(smem + sm.wq);
  float* wk = reinterpret_cast<float*>(smem + sm.wk);
  float* wv = reinterpret_cast<float*>(smem + sm.wv);
  float* wg = reinterpret_cast<float*>(smem + sm.wg);
  float* xh = reinterpret_cast<float*>(smem + sm.xh);
  float* red = reinterpret_cast<float*>(smem + sm.red);
  float* dsh = reinterpret_cast<float*>(smem + sm.dsh);
  float* scal = reinterpret_cast<float*>(smem + sm.scal);  // [kWarps] k.q partials
  unsigned char* wraw = smem + sm.wraw;
  const TileRing tr(dk, dv, (int)sizeof(ST), 1 << 30);  // every chunk has a stage
  const WholeTile<ST> tile{ring, mbar + 1, tr, dv};
  const int s_in = dtype_bytes(p.in_dt);
  const bool f32in = p.in_dt == DT_F32;
  const uint32_t qrow = (uint32_t)(dk * s_in), vrow = (uint32_t)(dv * s_in);

  if (tid == 0) {
    for (int j = 0; j <= tr.nchunk; ++j) mbar_init(&mbar[j], 1);
    fence_mbar_init();
    const size_t qoff = (((size_t)r * HK + kh) * dk) * s_in;
    const size_t voff = (((size_t)r * HV + h) * dv) * s_in;
    mbar_expect_tx(&mbar[0], 2 * qrow + vrow + (ALGO == ALGO_KDA ? (uint32_t)(dk * 4) : 0u));
    bulk_g2s(f32in ? static_cast<void*>(wq) : wraw, static_cast<const char*>(p.q) + qoff, qrow,
             &mbar[0]);
    bulk_g2s(f32in ? static_cast<void*>(wk) : wraw + qrow, static_cast<const char*>(p.k) + qoff,
             qrow, &mbar[0]);
    bulk_g2s(f32in ? static_cast<void*>(wv) : wraw + 2 * qrow,
             static_cast<const char*>(p.v) + voff, vrow, &mbar[0]);
    if (ALGO == ALGO_KDA) bulk_g2s(wg, p.g + ((size_t)r * HV + h) * dk, (uint32_t)(dk * 4), &mbar[0]);
    for (int j = 0; j < tr.nchunk; ++j) {
      mbar_expect_tx(&mbar[1 + j], tr.chunk_bytes);
      bulk_g2s(ring + (size_t)j * tr.cr * dv, gtile + (size_t)j * tr.cr * dv, tr.chunk_bytes,
               &mbar[1 + j]);
    }
  }
  const float beta = p.beta[(size_t)r * HV + h];
  const float eg = ALGO == ALGO_GDN ? __expf(p.g[(size_t)r * HV + h]) : 1.f;
  __syncthreads();
  bool ok = mbar_wait_bounded(&mbar[0], 0);
  if (!f32in) {
    widen16(wq, wraw, dk, p.in_dt, tid, kThreads);
    widen16(wk, wraw + qrow, dk, p.in_dt, tid, kThreads);
    widen16(wv, wraw + 2 * qrow, dv, p.in_dt, tid, kThreads);
  }
  __syncthreads();
  // mat-vec inputs: decay(k), decay(q) per key channel (GDN: the scalar decay
  // goes on the column results); k . q for the output correction
  float kq = 0.f;
  for (int ch = tid; ch < dk; ch += kThreads) {
    const float e = ALGO == ALGO_KDA ? __expf(wg[ch]) : 1.f;
    if (ALGO == ALGO_KDA) wg[ch] = e;
    xh[ch * NV + 0] = e * wk[ch];
    xh[ch * NV + 1] = e * wq[ch];
    kq = fmaf(wk[ch], wq[ch], kq);
  }
  kq = warp_sum(kq);
  if (lane == 0) scal[warp] = kq;

  // ---- pass 1: y_k = S^T decay(k), y_q = S^T decay(q)
  const QuadLayout qlay(dv, CW, kWarps);
  const QuadLane qlane(qlay, CW, warp, lane);
  float acc[NV][CW];
#pragma unroll
  for (int vv = 0; vv < NV; ++vv) {
#pragma unroll
    for (int cc = 0; cc < CW; ++cc) acc[vv][cc] = 0.f;
  }
  __syncthreads();
  ok = stream_quads<ALGO, ST, NV, CW, 4, false>(tile, qlane, acc, gtile, dk, dv, 0, nullptr,
                                                nullptr, nullptr, 1.f, nullptr, xh, tid, lane) &&
       ok;
  if (qlane.first) {
#pragma unroll
    for (int vv = 0; vv < NV; ++vv) {
#pragma unroll
      for (int cc = 0; cc < CW; ++cc) red[(qlane.rg * NV + vv) * dv + qlane.col0 + cc] = acc[vv][cc];
    }
  }
  __syncthreads();

  // ---- per value column: delta and output
  if (tid < dv) {
    const int col = tid;
    float yk = 0.f, yq = 0.f;
    for (int g2 = 0; g2 < qlay.rgw; ++g2) {
      yk += red[(g2 * NV + 0) * dv + col];
      yq += red[(g2 * NV + 1) * dv + col];
    }
    float kqs = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) kqs += scal[w2];
    const float d = beta * (wv[col] - eg * yk);
    dsh[col] = d;
    st_f32(p.o, ((size_t)r * HV + h) * dv + col, p.in_dt, p.scale * (eg * yq + kqs * d));
  }
  __syncthreads();

  // ---- pass 2: S <- decay(row) S + k d^T, from shared memory to the state
  const int rpl = tr.cr / qlane.rstep;
  for (int j = 0; j < tr.nchunk; ++j) {
    const ST* stg = tile.stage(j) + qlane.col0;
    float dcol[CW];
#pragma unroll
    for (int c = 0; c < CW; ++c) dcol[c] = dsh[qlane.col0 + c];
    for (int u = 0; u < rpl; ++u) {
      const int lr = qlane.lr0 + u * qlane.rstep;
      const int row = j * tr.cr + lr;
      float v[CW];
      ld_cols<ST, CW>(stg + (size_t)lr * dv, v);
      const float dec = ALGO == ALGO_GDN ? eg : wg[row];
      const float kr = wk[row];
#pragma unroll
      for (int c = 0; c < CW; ++c) v[c] = fmaf(kr, dcol[c], dec * v[c]);
      st_cols<ST, CW>(gtile + (size_t)row * dv + qlane.col0, v);
    }
  }
  if (!ok) {
    atomicOr(p.err, DEVERR_TIMEOUT);
    for (int j = 0; j <= tr.nchunk; ++j) mbar_wait_bounded(&mbar[j], 0);
  }
}

}  // namespace rssm
