// Device helpers shared by the replay kernel and the fold kernel: staging the
// ring history with bulk async copies, turning its gates into decay factors,
// and streaming the checkpoint tile through a ring of shared-memory stages,
// each thread consuming one value column (with the fold and the mat-vecs of
// the window fused in).
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

// Issue the bulk copies of n history records of one (slot, value head),
// completing on `bar` (one thread, after the mbarrier is initialised): keys
// [n][dk] -> kdst and deltas [n][dv] -> ddst, both as stored in the ring; KDA
// gates [n][dk] -> hg. The ring is head-major, so each run is contiguous;
// every run is a multiple of 16 bytes (dk, dv >= 32).
template <int ALGO>
__host__ __device__ __forceinline__ uint32_t history_bytes(int n, int dk, int dv, int rk_dt,
                                                           int rd_dt) {
  return (uint32_t)(n * (dk * dtype_bytes(rk_dt) + dv * dtype_bytes(rd_dt) +
                         (ALGO == ALGO_KDA ? dk * 4 : 0)));
}

// The copies alone; the caller has registered history_bytes() on `bar`.
template <int ALGO>
__device__ __forceinline__ void history_copies(int n, int dk, int dv, const void* ring_k,
                                               size_t kbase, int rk_dt, void* kdst,
                                               const void* ring_d, size_t dbase, int rd_dt,
                                               void* ddst, const float* ring_g, size_t gbase,
                                               float* hg, uint64_t* bar) {
  const int sk = dtype_bytes(rk_dt), sd = dtype_bytes(rd_dt);
  bulk_g2s(kdst, static_cast<const char*>(ring_k) + kbase * sk, (uint32_t)(n * dk * sk), bar);
  bulk_g2s(ddst, static_cast<const char*>(ring_d) + dbase * sd, (uint32_t)(n * dv * sd), bar);
  if (ALGO == ALGO_KDA) bulk_g2s(hg, ring_g + gbase, (uint32_t)(n * dk * 4), bar);
}

template <int ALGO>
__device__ __forceinline__ void issue_history(int n, int dk, int dv, const void* ring_k,
                                              size_t kbase, int rk_dt, void* kdst,
                                              const void* ring_d, size_t dbase, int rd_dt,
                                              void* ddst, const float* ring_g, size_t gbase,
                                              float* hg, uint64_t* bar, uint32_t extra = 0u) {
  mbar_expect_tx(bar, history_bytes<ALGO>(n, dk, dv, rk_dt, rd_dt) + extra);
  history_copies<ALGO>(n, dk, dv, ring_k, kbase, rk_dt, kdst, ring_d, dbase, rd_dt, ddst, ring_g,
                       gbase, hg, bar);
}

// Once the history copies have landed: widen 16-bit records to fp32 (fold
// kernel: fp32 records land in place).
__device__ __forceinline__ void widen_history(int n, int dk, int dv, int rk_dt, int rd_dt,
                                              float* hk, const void* hkraw, float* hd,
                                              const void* hdraw, int tid) {
  if (rk_dt != DT_F32) widen16(hk, hkraw, n * dk, rk_dt, tid, kThreads);
  if (rd_dt != DT_F32) widen16(hd, hdraw, n * dv, rd_dt, tid, kThreads);
}

// Ring keys [n][dk] as stored (any dtype) -> fp32 [n][dk]; threads t of nt.
__device__ __forceinline__ void widen_keys(float* hk, const void* raw, int count, int dt, int t,
                                           int nt) {
  if (dt == DT_F32) {
    const float4* s = static_cast<const float4*>(raw);
    float4* d = reinterpret_cast<float4*>(hk);
    for (int e = t; e < count / 4; e += nt) d[e] = s[e];
  } else {
    widen16(hk, raw, count, dt, t, nt);
  }
}

// Keys [n][dk] (any dtype) -> transposed fp32 keys hkt[ch][m] with row stride
// ks = round4(n); the padding entries m in [n, ks) are zero.
__device__ __forceinline__ void transpose_keys(float* hkt, const void* raw, int n, int dk, int dt,
                                               int t, int nt) {
  const int ks = round4(n);
  for (int e = t; e < dk * (ks / 4); e += nt) {
    const int ch = e % dk, m0 = 4 * (e / dk);
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = m0 + j < n ? ld_f32(raw, (size_t)(m0 + j) * dk + ch, dt) : 0.f;
    *reinterpret_cast<float4*>(hkt + (size_t)ch * ks + m0) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// Keys of n records as they landed, [n][dk] 16-bit, transposed in place to
// [dk][ks] 16-bit (ks = round4(n), entries m in [n, ks) zero). Every one of
// the nt threads of the CTA (t its index) takes part, with two CTA barriers:
// each first holds at most kKipVec 16-byte rows of eight keys in registers,
// so n * dk <= 8 * kKipVec * nt. Consecutive threads take consecutive
// records, so the 2-byte stores of a warp land in consecutive halves.
constexpr int kKipVec = 8;
__device__ __forceinline__ void transpose_keys16_inplace(uint16_t* raw, int n, int dk, int t,
                                                         int nt) {
  const int ks = round4(n), c8n = dk / 8, nvec = n * c8n;
  uint4 v[kKipVec];
#pragma unroll
  for (int i = 0; i < kKipVec; ++i) {
    const int e = t + i * nt;
    if (e < nvec) {
      const int m = e % n, c8 = e / n;
      v[i] = reinterpret_cast<const uint4*>(raw)[m * c8n + c8];
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kKipVec; ++i) {
    const int e = t + i * nt;
    if (e < nvec) {
      const int m = e % n, c8 = e / n;
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        raw[(8 * c8 + j) * ks + m] = (uint16_t)(w[j >> 1] >> (16 * (j & 1)));
      }
    }
  }
  const int pad = ks - n;
  for (int e = t; e < dk * pad; e += nt) raw[(e / pad) * ks + n + e % pad] = 0;
  __syncthreads();
}

// The raw keys of n <= 16 records in the order of the B fragments of an
// m16n8k8 product with the records as k and eight rows as n: for rows
// [8s, 8s + 8) lane (g, t) finds at hkf[4 (32 s + 4 g + t)] the keys of row
// 8s + g from records t, t + 4, 8 + t and 12 + t (zero for records >= n).
// hkf holds dk * 16 floats.
__device__ __forceinline__ void frag_keys16(float* hkf, const void* raw, int n, int dk, int dt,
                                            int t, int nt) {
  for (int e = t; e < dk * 4; e += nt) {
    const int s8 = e >> 5, ln = e & 31, row = 8 * s8 + (ln >> 2), m0 = ln & 3;
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + 4 * j;
      v[j] = m < n ? ld_f32(raw, (size_t)m * dk + row, dt) : 0.f;
    }
    *reinterpret_cast<float4*>(hkf + 4 * e) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// The same for any n, in ng = ceil(n / 16) groups of 16 records: for rows
// [8s, 8s + 8) and group q lane (g, t) finds at
// hkf[4 (32 (ng s + q) + 4 g + t)] the keys of row 8s + g from records
// 16q + t, 16q + t + 4, 16q + t + 8 and 16q + t + 12 (zero for records >= n).
// hkf holds dk * 16 * ng floats.
__device__ __forceinline__ void frag_keys(float* hkf, const void* raw, int n, int dk, int dt,
                                          int t, int nt) {
  const int ng = (n + 15) >> 4;
  for (int e = t; e < dk * 4 * ng; e += nt) {
    const int blk = e >> 5, ln = e & 31, s8 = blk / ng, q = blk - s8 * ng;
    const int row = 8 * s8 + (ln >> 2), m0 = 16 * q + (ln & 3);
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + 4 * j;
      v[j] = m < n ? ld_f32(raw, (size_t)m * dk + row, dt) : 0.f;
    }
    *reinterpret_cast<float4*>(hkf + 4 * e) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// GDN, warp 0: hf[m] holds the raw record gates g_m; replaces them with
// exp(sum_{m' > m} g_m') and writes Gam, exp(Gam) to scal[0], scal[1].
__device__ __forceinline__ void gdn_history_scan(int n, float* hf, float* scal, int lane) {
  float carry = 0.f;
  for (int hi = n; hi > 0; hi -= 32) {
    const int m = hi - 1 - lane;  // newest record first
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

// KDA, one key channel: scale the staged keys of channel ch by their decay to
// the end of the history (k~_m[ch], in place) and return Gam[ch]. hg holds the
// record gates [n][dk].
__device__ __forceinline__ float kda_history_channel(int n, int dk, int ch, float* hk,
                                                     const float* hg) {
  float suf = 0.f;
  for (int m = n - 1; m >= 0; --m) {
    hk[m * dk + ch] *= __expf(suf);
    suf += hg[m * dk + ch];
  }
  return suf;
}

// Column mapping of a CTA over one (slot, head) checkpoint tile [dk][dv]:
// thread tid owns value column col = tid % dv and rows rg, rg + RG, ... with
// RG = kThreads / dv row groups. A warp's load of one row is 32 consecutive
// columns (128 bytes for fp32).
struct ColMap {
  int col, rg, RG, nrow;
  __device__ __forceinline__ ColMap(int dk, int dv, int tid) {
    RG = kThreads / dv;
    col = tid % dv;
    rg = tid / dv;
    nrow = dk / RG;
  }
  __device__ __forceinline__ int row(int j) const { return rg + RG * j; }
};

template <typename ST>
__device__ __forceinline__ float st_load(const ST* p);
template <>
__device__ __forceinline__ float st_load<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float st_load<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// Round to the checkpoint dtype, store, and return the stored value.
template <typename ST>
__device__ __forceinline__ float st_store(ST* p, float x);
template <>
__device__ __forceinline__ float st_store<float>(float* p, float x) {
  *p = x;
  return x;
}
template <>
__device__ __forceinline__ float st_store<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  const __nv_bfloat16 b = __float2bfloat16_rn(x);
  *p = b;
  return __bfloat162float(b);
}

// Consume one register batch of this thread's column:
//  - FOLD: S[row] <- decay(row) S[row] + sum_m k~_m[row] d~_m   (d~_m = f_m d_m[col]),
//    stored back to the checkpoint in its dtype; the stored value is used below;
//  - NV > 0: y[v] += x_v[row] S[row] for every mat-vec vector (xh [dk][NV]).
// GDN: hk holds raw keys and f_m = hf[m], decay = gdn_decay; KDA: hk holds k~
// and f_m = 1, decay(row) = egam[row].
template <int ALGO, typename ST, int RB, int NV, bool FOLD>
__device__ __forceinline__ void consume_rows(float (&buf)[RB], float (&y)[NV > 0 ? NV : 1],
                                             ST* gcol, int j0, const ColMap& cm, int dk, int dv,
                                             int n, const float* hk, const float* hd,
                                             const float* hf, float gdn_decay,
                                             const float* egam, const float* xh) {
  if (FOLD) {
    float acc[RB];
#pragma unroll
    for (int u = 0; u < RB; ++u) {
      const int row = cm.row(min(j0 + u, cm.nrow - 1));
      const float dec = (ALGO == ALGO_GDN) ? gdn_decay : egam[row];
      acc[u] = dec * buf[u];
    }
    for (int m = 0; m < n; ++m) {
      float dm = hd[m * dv + cm.col];
      if (ALGO == ALGO_GDN) dm *= hf[m];
      const float* km = hk + (size_t)m * dk;
#pragma unroll
      for (int u = 0; u < RB; ++u) {
        acc[u] = fmaf(km[cm.row(min(j0 + u, cm.nrow - 1))], dm, acc[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < RB; ++u) {
      const int j = j0 + u;
      if (j < cm.nrow) buf[u] = st_store<ST>(gcol + (size_t)cm.row(j) * dv, acc[u]);
    }
  }
  if constexpr (NV > 0) {
#pragma unroll
    for (int u = 0; u < RB; ++u) {
      const int j = j0 + u;
      if (j < cm.nrow) {
        const float* xr = xh + (size_t)cm.row(j) * NV;
        if constexpr (NV % 4 == 0) {
#pragma unroll
          for (int q4 = 0; q4 < NV / 4; ++q4) {
            const float4 x = reinterpret_cast<const float4*>(xr)[q4];
            y[4 * q4 + 0] = fmaf(x.x, buf[u], y[4 * q4 + 0]);
            y[4 * q4 + 1] = fmaf(x.y, buf[u], y[4 * q4 + 1]);
            y[4 * q4 + 2] = fmaf(x.z, buf[u], y[4 * q4 + 2]);
            y[4 * q4 + 3] = fmaf(x.w, buf[u], y[4 * q4 + 3]);
          }
        } else {
          const float2 x = *reinterpret_cast<const float2*>(xr);
          y[0] = fmaf(x.x, buf[u], y[0]);
          y[1] = fmaf(x.y, buf[u], y[1]);
        }
      }
    }
  }
}

// Ring of shared-memory stages over the row chunks of one checkpoint tile.
// One thread produces (bulk async copies), every warp consumes; stage
// j % ns holds chunk j; "full" completes when a chunk has landed, "empty"
// when all warps have consumed it.
template <typename ST>
struct TilePipe {
  ST* ring;
  uint64_t* full;
  uint64_t* empty;
  const ST* gtile;
  int dv;
  TileRing tr;
  WaitHook hook;
  __device__ __forceinline__ TilePipe(ST* ring_, uint64_t* mbar, const ST* gtile_, int dk, int dv_,
                                      int stages, const WaitHook& hook_)
      : ring(ring_), full(mbar + kMbarFull), empty(mbar + kMbarEmpty), gtile(gtile_), dv(dv_),
        tr(dk, dv_, (int)sizeof(ST), stages), hook(hook_) {}
  // mbarrier set-up (one thread): "full" before the first copy (and the fence
  // that makes initialisation visible to the copies), "empty" with the number
  // of consuming warps before the CTA barrier that precedes the stream.
  static __device__ __forceinline__ void init_full(uint64_t* mbar) {
    for (int st = 0; st < kStages; ++st) mbar_init(&mbar[kMbarFull + st], 1);
  }
  __device__ __forceinline__ void init_empty(int warps) const {
    for (int st = 0; st < tr.ns; ++st) mbar_init(&empty[st], warps);
  }
  __device__ __forceinline__ void init() const {
    for (int st = 0; st < tr.ns; ++st) mbar_init(&full[st], 1);
    init_empty(kWarps);
  }
  __device__ __forceinline__ void issue(int j) const {
    const int st = j % tr.ns;
    mbar_expect_tx(&full[st], tr.chunk_bytes + hook.extra(WH_CHUNK0 + j));
    bulk_g2s(ring + (size_t)st * tr.cr * dv, gtile + (size_t)j * tr.cr * dv, tr.chunk_bytes,
             &full[st]);
  }
  // producer: the first ns chunks
  __device__ __forceinline__ void prime() const {
    for (int j = 0; j < tr.ns; ++j) issue(j);
  }
  __device__ __forceinline__ bool wait_full(int j) const {
    return mbar_wait_bounded(&full[j % tr.ns], (uint32_t)((j / tr.ns) & 1));
  }
  // every warp, once it has consumed chunk j (thread 0, the producer, whose own
  // reads come before its refill in program order, arrives without release
  // semantics, which would wait for its copies in flight)
  __device__ __forceinline__ void release(int j, int tid, int lane) const {
    __syncwarp();
    if (lane == 0) {
      if (tid == 0) {
        mbar_arrive_relaxed(&empty[j % tr.ns]);
      } else {
        mbar_arrive(&empty[j % tr.ns]);
      }
    }
  }
  // producer, after its own release of chunk j: refill that stage with chunk j + ns
  __device__ __forceinline__ bool refill(int j) const {
    if (j + tr.ns >= tr.nchunk) return true;
    const bool ok = mbar_wait_bounded(&empty[j % tr.ns], (uint32_t)((j / tr.ns) & 1));
    if (ok) issue(j + tr.ns);
    return ok;
  }
  // a CTA that leaves early lets the primed chunks land first
  __device__ __forceinline__ void drain() const {
    for (int j = 0; j < tr.ns; ++j) mbar_wait_bounded(&full[j], 0);
  }
  // a CTA whose stream failed lets the chunks that may still be in flight (the
  // last ns issued) land before it leaves; each wait is bounded again
  __device__ __forceinline__ void drain_tail() const {
    const int j0 = tr.nchunk > tr.ns ? tr.nchunk - tr.ns : 0;
    for (int j = j0; j < tr.nchunk; ++j) wait_full(j);
  }
  // interface of stream_quads: stage data of chunk j, wait for it, hand it back
  __device__ __forceinline__ const ST* stage(int j) const {
    return ring + (size_t)(j % tr.ns) * tr.cr * dv;
  }
  __device__ __forceinline__ bool wait(int j) const { return wait_full(j); }
  // (the producer issues nothing more once one of its own waits has run out,
  // so every copy it issued can be waited for before the CTA leaves)
  __device__ __forceinline__ bool done(int j, int tid, int lane, bool ok) const {
    release(j, tid, lane);
    return tid == 0 && ok ? refill(j) : true;
  }
};

// Stream the checkpoint tile through the ring; each thread consumes its
// column's rows of every chunk (fold and/or mat-vecs, see consume_rows).
// Returns false if a bounded wait ran out.
template <int ALGO, typename ST, int NV, bool FOLD>
__device__ __forceinline__ bool stream_tile(const TilePipe<ST>& pipe, float (&y)[NV > 0 ? NV : 1],
                                            ST* gcol, const ColMap& cm, int dk, int dv, int n,
                                            const float* hk, const float* hd, const float* hf,
                                            float gdn_decay, const float* egam, const float* xh,
                                            int tid, int lane) {
  constexpr int RB = 8;  // rows of a chunk held in registers at a time
  const int rpc = pipe.tr.cr / cm.RG;  // this thread's rows per chunk (a multiple of 8)
  bool ok = true;
  for (int j = 0; j < pipe.tr.nchunk; ++j) {
    // a warp stores no chunk once one of its waits has run out
    ok = __all_sync(kFull, pipe.wait_full(j) && ok);
    const ST* stg = pipe.ring + (size_t)(j % pipe.tr.ns) * pipe.tr.cr * dv +
                    (size_t)cm.rg * dv + cm.col;
    for (int u0 = 0; ok && u0 < rpc; u0 += RB) {
      float buf[RB];
#pragma unroll
      for (int u = 0; u < RB; ++u) buf[u] = st_load<ST>(stg + (size_t)cm.RG * (u0 + u) * dv);
      consume_rows<ALGO, ST, RB, NV, FOLD>(buf, y, gcol, j * rpc + u0, cm, dk, dv, n, hk, hd, hf,
                                           gdn_decay, egam, xh);
    }
    pipe.release(j, tid, lane);
    if (tid == 0 && ok) ok = pipe.refill(j);
  }
  return ok;
}

// CW consecutive checkpoint values <-> fp32 (shared-memory loads, global stores
// that round to the checkpoint dtype and return the stored values).
template <typename ST, int CW>
__device__ __forceinline__ void ld_cols(const ST* p, float (&v)[CW]);
template <>
__device__ __forceinline__ void ld_cols<float, 4>(const float* p, float (&v)[4]) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
template <>
__device__ __forceinline__ void ld_cols<float, 2>(const float* p, float (&v)[2]) {
  const float2 x = *reinterpret_cast<const float2*>(p);
  v[0] = x.x; v[1] = x.y;
}
template <>
__device__ __forceinline__ void ld_cols<__nv_bfloat16, 4>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
template <>
__device__ __forceinline__ void ld_cols<__nv_bfloat16, 2>(const __nv_bfloat16* p, float (&v)[2]) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
  v[0] = a.x; v[1] = a.y;
}

template <typename ST, int CW>
__device__ __forceinline__ void st_cols(ST* p, float (&v)[CW]);
template <>
__device__ __forceinline__ void st_cols<float, 4>(float* p, float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void st_cols<float, 2>(float* p, float (&v)[2]) {
  *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
}
template <>
__device__ __forceinline__ void st_cols<__nv_bfloat16, 4>(__nv_bfloat16* p, float (&v)[4]) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&a);
  u.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
}
template <>
__device__ __forceinline__ void st_cols<__nv_bfloat16, 2>(__nv_bfloat16* p, float (&v)[2]) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  *reinterpret_cast<__nv_bfloat162*>(p) = a;
  const float2 fa = __bfloat1622float2(a);
  v[0] = fa.x; v[1] = fa.y;
}

// Lane position in the tile stream (see QuadLayout).
struct QuadLane {
  int col0;   // first of this lane's CW columns
  int lr0;    // first local row of a chunk handled by this lane
  int rstep;  // distance between this lane's rows
  int rg;     // warp row group (index of the partial sum)
  int first;  // 1 on the lane that holds the row group's sum after the reduction
  int lanes;  // lanes of one row within a warp
  __device__ __forceinline__ QuadLane(const QuadLayout& ql, int CW, int warp, int lane) {
    lanes = ql.lpr < 32 ? ql.lpr : 32;
    const int cb = warp % ql.wcb;
    rg = warp / ql.wcb;
    col0 = CW * (cb * 32 + lane % lanes);
    const int rl = lane / lanes;
    lr0 = rg * ql.rsw + rl;
    rstep = ql.rgw * ql.rsw;
    first = rl == 0;
  }
};

// Stream the checkpoint tile through the ring: each lane takes CW columns of
// some rows of every chunk, a few rows at a time. FOLD: S[row] <- decay(row)
// S[row] + sum_m k~_m[row] d_m, stored back to the checkpoint rounded to its
// dtype; hkt holds the keys transposed ([dk][round4(n)], zero padded; GDN: raw
// keys with k~_m = hf[m] k_m and decay = gdn_decay; KDA: k~ itself, decay =
// egam[row]). A lane's columns never change, so the deltas of the first MR
// records stay in registers for the whole tile and every row costs one
// broadcast vector load per four records; records past MR come from hd
// [n][dv]. Then acc[v] += x_v[row] S[row] for the NV mat-vec vectors (xh
// [dk][NV]). Sums over the rows of one warp instruction are reduced before
// returning.
// hd_dt: the dtype of the deltas at hd (fp32, or fp16 read as they landed).
template <int ALGO, typename ST, int NV, int CW, int MR, bool FOLD, class PIPE>
__device__ __forceinline__ bool stream_quads(const PIPE& pipe, const QuadLane& ql,
                                             float (&acc)[NV][CW], ST* gtile, int dk, int dv,
                                             int n, const float* hkt, const float* hd,
                                             const float* hf, float gdn_decay,
                                             const float* egam, const float* xh, int tid,
                                             int lane, int hd_dt = DT_F32) {
  auto hd_at = [&](size_t i) {
    return hd_dt == DT_F32 ? hd[i] : __half2float(reinterpret_cast<const __half*>(hd)[i]);
  };
  constexpr int RS = FOLD ? 2 : 4;  // rows held in registers at a time
  constexpr int MRR = FOLD ? MR : 1;
  const int ks = round4(n);
  float dr[MRR][CW];
  if (FOLD) {
#pragma unroll
    for (int m = 0; m < MRR; ++m) {
#pragma unroll
      for (int c = 0; c < CW; ++c) dr[m][c] = 0.f;
      if (m < n) {
        const float f = ALGO == ALGO_GDN ? hf[m] : 1.f;
#pragma unroll
        for (int c = 0; c < CW; ++c) dr[m][c] = f * hd_at((size_t)m * dv + ql.col0 + c);
      }
    }
  }
  const int rpl = pipe.tr.cr / ql.rstep;  // this lane's rows per chunk
  bool ok = true;
  for (int j = 0; j < pipe.tr.nchunk; ++j) {
    ok = pipe.wait(j) && ok;
    if (FOLD) ok = __all_sync(kFull, ok);  // no store-back once a wait has run out
    const ST* stg = pipe.stage(j) + ql.col0;
    const int row0 = j * pipe.tr.cr;
    for (int u0 = 0; u0 < rpl; u0 += RS) {
      float s[RS][CW];
      int rows[RS];
#pragma unroll
      for (int u = 0; u < RS; ++u) {
        const int uu = u0 + u < rpl ? u0 + u : rpl - 1;  // a repeated row is never used
        const int lr = ql.lr0 + uu * ql.rstep;
        rows[u] = row0 + lr;
        ld_cols<ST, CW>(stg + (size_t)lr * dv, s[u]);
      }
      if (FOLD && ALGO == ALGO_KDA) {
        // KDA: the decayed keys as computed, [n][dk] (one broadcast load per
        // record and row)
#pragma unroll
        for (int u = 0; u < RS; ++u) {
          const float dec = egam[rows[u]];
#pragma unroll
          for (int c = 0; c < CW; ++c) s[u][c] *= dec;
#pragma unroll
          for (int m = 0; m < MRR; ++m) {
            if (m < n) {
              const float k = hkt[(size_t)m * dk + rows[u]];
#pragma unroll
              for (int c = 0; c < CW; ++c) s[u][c] = fmaf(k, dr[m][c], s[u][c]);
            }
          }
          for (int m = MRR; m < n; ++m) {
            float dv4[CW];
            if (hd_dt == DT_F32) {
              ld_cols<float, CW>(hd + (size_t)m * dv + ql.col0, dv4);
            } else {
#pragma unroll
              for (int c = 0; c < CW; ++c) dv4[c] = hd_at((size_t)m * dv + ql.col0 + c);
            }
            const float k = hkt[(size_t)m * dk + rows[u]];
#pragma unroll
            for (int c = 0; c < CW; ++c) s[u][c] = fmaf(k, dv4[c], s[u][c]);
          }
        }
#pragma unroll
        for (int u = 0; u < RS; ++u) {
          if (ok && u0 + u < rpl) st_cols<ST, CW>(gtile + (size_t)rows[u] * dv + ql.col0, s[u]);
        }
      } else if (FOLD) {
#pragma unroll
        for (int u = 0; u < RS; ++u) {
          const float dec = ALGO == ALGO_GDN ? gdn_decay : egam[rows[u]];
          const float* kr = hkt + (size_t)rows[u] * ks;
#pragma unroll
          for (int c = 0; c < CW; ++c) s[u][c] *= dec;
#pragma unroll
          for (int q4 = 0; q4 < MRR / 4; ++q4) {
            if (4 * q4 < n) {
              const float4 k4 = *reinterpret_cast<const float4*>(kr + 4 * q4);
#pragma unroll
              for (int c = 0; c < CW; ++c) {
                s[u][c] = fmaf(k4.x, dr[4 * q4 + 0][c], s[u][c]);
                s[u][c] = fmaf(k4.y, dr[4 * q4 + 1][c], s[u][c]);
                s[u][c] = fmaf(k4.z, dr[4 * q4 + 2][c], s[u][c]);
                s[u][c] = fmaf(k4.w, dr[4 * q4 + 3][c], s[u][c]);
              }
            }
          }
          for (int m0 = MRR; m0 < n; m0 += 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(kr + m0);
            const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              if (m0 + m < n) {
                float dv4[CW];
                ld_cols<float, CW>(hd + (size_t)(m0 + m) * dv + ql.col0, dv4);
                const float kf = (ALGO == ALGO_GDN ? hf[m0 + m] : 1.f) * kv[m];
#pragma unroll
                for (int c = 0; c < CW; ++c) s[u][c] = fmaf(kf, dv4[c], s[u][c]);
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < RS; ++u) {
          if (ok && u0 + u < rpl) st_cols<ST, CW>(gtile + (size_t)rows[u] * dv + ql.col0, s[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < RS; ++u) {
        if (u0 + u < rpl) {
          const float* xr = xh + (size_t)rows[u] * NV;
          if constexpr (NV % 4 == 0) {
#pragma unroll
            for (int q4 = 0; q4 < NV / 4; ++q4) {
              const float4 x = reinterpret_cast<const float4*>(xr)[q4];
#pragma unroll
              for (int c = 0; c < CW; ++c) {
                acc[4 * q4 + 0][c] = fmaf(x.x, s[u][c], acc[4 * q4 + 0][c]);
                acc[4 * q4 + 1][c] = fmaf(x.y, s[u][c], acc[4 * q4 + 1][c]);
                acc[4 * q4 + 2][c] = fmaf(x.z, s[u][c], acc[4 * q4 + 2][c]);
                acc[4 * q4 + 3][c] = fmaf(x.w, s[u][c], acc[4 * q4 + 3][c]);
              }
            }
          } else {
            const float2 x = *reinterpret_cast<const float2*>(xr);
#pragma unroll
            for (int c = 0; c < CW; ++c) {
              acc[0][c] = fmaf(x.x, s[u][c], acc[0][c]);
              acc[1][c] = fmaf(x.y, s[u][c], acc[1][c]);
            }
          }
        }
      }
    }
    ok = pipe.done(j, tid, lane, ok) && ok;
  }
  for (int off = ql.lanes; off < 32; off <<= 1) {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
      for (int c = 0; c < CW; ++c) acc[v][c] += __shfl_xor_sync(kFull, acc[v][c], off);
    }
  }
  return ok;
}

// stream_quads without a fold for a fixed geometry: RPL rows per lane per
// chunk, RSTEP rows between a lane's rows, DV value columns. Every offset is a
// compile-time constant and a chunk is one fully unrolled block of loads and
// FMAs, which halves the instructions per row of the general loop.
template <typename ST, int NV, int CW, int RPL, int RSTEP, int DV, class PIPE>
__device__ __forceinline__ bool stream_fixed(const PIPE& pipe, const QuadLane& ql,
                                             float (&acc)[NV][CW], const float* xh, int tid,
                                             int lane) {
  bool ok = true;
  const int cr = pipe.tr.cr;
  for (int j = 0; j < pipe.tr.nchunk; ++j) {
    ok = pipe.wait(j) && ok;
    const ST* stg = pipe.stage(j) + ql.col0 + ql.lr0 * DV;
    const float* xr = xh + (size_t)(j * cr + ql.lr0) * NV;
    float sv[RPL][CW];
#pragma unroll
    for (int u = 0; u < RPL; ++u) ld_cols<ST, CW>(stg + u * RSTEP * DV, sv[u]);
#pragma unroll
    for (int u = 0; u < RPL; ++u) {
      if constexpr (NV == 2) {
        const float2 x = *reinterpret_cast<const float2*>(xr + u * RSTEP * NV);
#pragma unroll
        for (int c = 0; c < CW; ++c) {
          acc[0][c] = fmaf(x.x, sv[u][c], acc[0][c]);
          acc[1][c] = fmaf(x.y, sv[u][c], acc[1][c]);
        }
      } else {
#pragma unroll
        for (int q4 = 0; q4 < NV / 4; ++q4) {
          const float4 x = *reinterpret_cast<const float4*>(xr + u * RSTEP * NV + 4 * q4);
#pragma unroll
          for (int c = 0; c < CW; ++c) {
            acc[4 * q4 + 0][c] = fmaf(x.x, sv[u][c], acc[4 * q4 + 0][c]);
            acc[4 * q4 + 1][c] = fmaf(x.y, sv[u][c], acc[4 * q4 + 1][c]);
            acc[4 * q4 + 2][c] = fmaf(x.z, sv[u][c], acc[4 * q4 + 2][c]);
            acc[4 * q4 + 3][c] = fmaf(x.w, sv[u][c], acc[4 * q4 + 3][c]);
          }
        }
      }
    }
    ok = pipe.done(j, tid, lane, ok) && ok;
  }
  for (int off = ql.lanes; off < 32; off <<= 1) {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
      for (int c = 0; c < CW; ++c) acc[v][c] += __shfl_xor_sync(kFull, acc[v][c], off);
    }
  }
  return ok;
}

}  // namespace rssm
