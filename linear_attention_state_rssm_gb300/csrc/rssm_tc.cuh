// 5th-generation tensor-core (tcgen05) building blocks and the tile stream of
// a GDN verify window built on them.
//
// Operand layouts (checked element by element against a host product on a
// GB300 before any kernel used them):
//  - shared-memory operands are K-major without swizzle: 8 x 16-byte core
//    matrices (8 rows of the M or N index, 4 tf32 along K, 128 contiguous
//    bytes); the descriptor's leading byte offset is the distance between
//    core matrices along K, its stride byte offset the distance between
//    8-row groups along M or N;
//  - an A operand in tensor memory holds row m of A in lane m, K along the
//    columns (one tf32 per column);
//  - the fp32 accumulator D[m][n] sits in lane m, column n;
//  - warp w of the CTA reaches lanes [32 (w % 4), 32 (w % 4) + 32).
// An fp32 value x enters a tf32 product as hi = x with its 13 low mantissa
// bits cleared plus lo = x - hi (exact in fp32): the pair carries x to about
// 2^-21 relative, and 16-bit values are exact in tf32 as they stand.
#pragma once

#include "rssm_common.cuh"
#include "rssm_history.cuh"

namespace rssm {

// Tensor-memory columns of one replay CTA: the mat-vec accumulator, two A
// stages of one 16-row slice each (hi, lo), the fold accumulator of one slice
// and the fold's A operand (hi, lo). At most four CTAs per SM fit in 512.
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kTcY = 0;     // [0, 16)   Y^T = S^T X, lane = value column
constexpr uint32_t kTcDf = 16;   // [16, 32)  fold D~^T K~ of one slice, lane = value column
constexpr uint32_t kTcA = 32;    // [32, 96)  A stages: 32 s + [0, 16) hi, [16, 32) lo
constexpr uint32_t kTcAf = 96;   // [96, 128) fold A = (f_m d_m)^T: [0, 16) hi, [16, 32) lo

__device__ __forceinline__ void tmem_alloc(uint32_t* slot) {  // one whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(kTmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {  // the allocating warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(kTmemCols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// generic-proxy writes to shared memory -> visible to the tensor core
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 consecutive columns of this thread's lane
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// this warp's first lane, as a tensor-memory address
__device__ __forceinline__ uint32_t tmem_lane(uint32_t tbase, int warp) {
  return tbase + ((uint32_t)(32 * (warp & 3)) << 16);
}

// K-major, no swizzle: lbo = bytes between core matrices along K, sbo = bytes
// between 8-row groups along M or N; bit 46 is the descriptor version.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// kind::tf32 instruction descriptor: fp32 accumulator, tf32 A and B, both
// K-major, M x N
__host__ __device__ constexpr uint32_t tf32_idesc(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// D (+)= A B with A and B in shared memory
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       bool acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)acc)
      : "memory");
}
// D (+)= A B with A in tensor memory
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                       bool acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"((uint32_t)acc)
      : "memory");
}
// one arrival on bar once every MMA this thread issued so far has completed
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// checkpoint values <-> fp32
__device__ __forceinline__ float tc_f32(float x) { return x; }
__device__ __forceinline__ float tc_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename ST>
__device__ __forceinline__ ST tc_st(float x);
template <>
__device__ __forceinline__ float tc_st<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 tc_st<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// Byte offset of element (row n of the N or M index, k) of a K-major operand
// with nb = N / 8 core-matrix rows per K step of four.
__device__ __forceinline__ uint32_t kmajor_off(int n, int k, int nb) {
  return (uint32_t)((((k >> 2) * nb + (n >> 3)) << 7) + ((n & 7) << 4) + ((k & 3) << 2));
}

// The mat-vec operand X always has kTcN = 16 vectors (an M = 128 product
// takes N in steps of 16): windows of four tokens leave vectors 8..15 zero.
constexpr int kTcN = 16;

// Slot e of the K-major mat-vec operand X [kTcN vectors x dk rows] -> (row ch,
// vector v); consecutive slots are consecutive 4-byte words.
__device__ __forceinline__ void x_slot_tc(int e, int& ch, int& v) {
  constexpr int NB = kTcN / 8;
  const int core = e >> 5;
  v = 8 * (core % NB) + ((e >> 2) & 7);
  ch = 4 * (core / NB) + (e & 3);
}

// Barriers and tensor memory of one CTA's tensor-core stream.
struct TcStream {
  uint32_t tbase;     // tensor-memory base address (column 0, lane 0)
  uint64_t* afull;    // [2] an A stage has been written (one arrival per warp)
  uint64_t* aempty;   // [2] the MMAs that read an A stage have completed
  uint64_t* fbar;     // the fold MMA of a slice has completed
  uint64_t* ydone;    // every mat-vec MMA has completed
  const float* xh;    // X (hi) [dk rows x kTcN vectors], K-major
  const float* xl;    // X lo (fp32 inputs) or null
  const float* kh;    // fold keys B~ [16 records x dk rows], K-major (hi)
  const float* kl;    // fold keys lo (fp32 ring keys) or null
};

// Fold operand A~ = (f_m d_m)^T, m < 16 (records >= n are zero), into tensor
// memory columns kTcAf: the lane of value column col holds f_m d_m[col] as hi
// in [0, 16) and lo in [16, 32).
__device__ __forceinline__ void tc_fold_a(const TcStream& tc, const float* hd, const float* hf,
                                          int n, int dv, int col, int warp) {
  float hi[16], lo[16];
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    const float a = m < n ? hf[m] * hd[m * dv + col] : 0.f;
    hi[m] = tf32_hi(a);
    lo[m] = a - hi[m];
  }
  const uint32_t ta = tmem_lane(tc.tbase, warp) + kTcAf;
  tmem_st16(ta, hi);
  tmem_st16(ta + 16, lo);
  tmem_st_wait();
}

// Fold keys B~ [K = 16 records x N = dk rows], K-major (row r at n, record m
// at k), from the n ring records (16-bit or fp32, [n][dk]); records >= n are
// zero. fp32 keys leave their lo part in kl.
__device__ __forceinline__ void tc_fold_keys(float* kh, float* kl, const void* raw, int n, int dk,
                                             int dt, int tid, int nthr) {
  const int nb = dk / 8;
  for (int e = tid; e < 16 * dk; e += nthr) {
    const int r = e % dk, m = e / dk;
    const float k = m < n ? ld_f32(raw, (size_t)m * dk + r, dt) : 0.f;
    const uint32_t off = kmajor_off(r, m, nb) >> 2;
    if (kl != nullptr) {
      kh[off] = tf32_hi(k);
      kl[off] = k - tf32_hi(k);
    } else {
      kh[off] = k;
    }
  }
}

// One thread (tid 0): the fold MMAs of 16-row slice q, D~f = A~ B~[rows of q]
// in columns kTcDf, then a commit on fbar.
__device__ __forceinline__ void tc_issue_fold(const TcStream& tc, int q, int dk) {
  constexpr uint32_t idesc = tf32_idesc(128, 16);
  const uint32_t lbo = (uint32_t)(dk / 8) * 128u;  // 4 records further along K
  for (int kk = 0; kk < 2; ++kk) {
    // rows [16q, 16q + 16): two 8-row groups past the start; records [8kk, 8kk + 8)
    const uint32_t boff = (uint32_t)(2 * q) * 128u + (uint32_t)(2 * kk) * lbo;
    const uint64_t bh = kmajor_desc(smem_addr(tc.kh) + boff, lbo, 128u);
    const uint32_t ah = tc.tbase + kTcAf + 8 * kk, al = ah + 16;
    mma_ts(tc.tbase + kTcDf, ah, bh, idesc, kk > 0);
    mma_ts(tc.tbase + kTcDf, al, bh, idesc, true);
    if (tc.kl != nullptr) {
      const uint64_t bl = kmajor_desc(smem_addr(tc.kl) + boff, lbo, 128u);
      mma_ts(tc.tbase + kTcDf, ah, bl, idesc, true);
    }
  }
  mma_commit(tc.fbar);
}

// One thread (tid 0): the mat-vec MMAs of slice q (A stage s), Y^T += S_q^T X_q.
template <bool EXACT_S>
__device__ __forceinline__ void tc_issue_matvec(const TcStream& tc, int q, int s) {
  constexpr uint32_t idesc = tf32_idesc(128, kTcN);
  constexpr uint32_t lbo = (uint32_t)(kTcN / 8) * 128u;  // 4 rows further along K
  for (int kk = 0; kk < 2; ++kk) {
    const uint32_t boff = (uint32_t)(4 * q + 2 * kk) * lbo;  // rows 16q + 8kk ..
    const uint64_t bh = kmajor_desc(smem_addr(tc.xh) + boff, lbo, 128u);
    const uint32_t ah = tc.tbase + kTcA + 32 * s + 8 * kk;
    mma_ts(tc.tbase + kTcY, ah, bh, idesc, q > 0 || kk > 0);
    if (!EXACT_S) mma_ts(tc.tbase + kTcY, ah + 16, bh, idesc, true);
    if (tc.xl != nullptr) {
      const uint64_t bl = kmajor_desc(smem_addr(tc.xl) + boff, lbo, 128u);
      mma_ts(tc.tbase + kTcY, ah, bl, idesc, true);
    }
  }
  mma_commit(&tc.aempty[s]);
}

// Tile stream of a GDN window (at most kTcN mat-vec vectors) and 128 value columns
// on the tensor cores. Thread tid owns value column tid. Each chunk's rows of
// the column are read from the ring stage (which is then handed back), and
// for each 16-row slice q:
//   FOLD: S'[r][col] = decay S[r][col] + (D~^T K~)[col][r] (fold MMA of slice
//         q, issued one slice ahead), rounded to the checkpoint dtype and
//         stored back; the mat-vec takes the stored values;
//   the slice goes, split into tf32 hi and lo, into A stage q % 2 of tensor
//   memory; thread 0 issues Y^T += S_q^T X_q (after the fold MMA of slice q + 1).
// Y^T ends in columns kTcY once ydone completes. Returns false if a bounded
// wait ran out (no store-back from then on).
template <typename ST, bool FOLD>
__device__ __forceinline__ bool stream_tc(const TilePipe<ST>& pipe, const TcStream& tc, ST* gtile,
                                          float decay, int tid, int warp, int lane) {
  constexpr int DV = 128;
  constexpr bool EXACT_S = !std::is_same<ST, float>::value;
  constexpr int CR = 8192 / (DV * (int)sizeof(ST));  // rows per chunk: 16 (fp32) or 32
  constexpr int NSL = CR / 16;                        // 16-row slices per chunk
  static_assert(NSL * 16 == CR, "chunk rows");
  const int col = tid;
  const int dk = pipe.tr.nchunk * CR;
  const int nslice = dk / 16;
  const uint32_t ta = tmem_lane(tc.tbase, warp);
  bool ok = true;
  if (FOLD && tid == 0) {
    tc_fence_after();
    tc_issue_fold(tc, 0, dk);
  }
  for (int j = 0; j < pipe.tr.nchunk; ++j) {
    ok = __all_sync(kFull, pipe.wait(j) && ok);
    const ST* stg = pipe.stage(j);
    float v[CR];
#pragma unroll
    for (int r = 0; r < CR; ++r) v[r] = tc_f32(stg[r * DV + col]);
    ok = pipe.done(j, tid, lane, ok) && ok;  // the stage goes back to the producer
#pragma unroll
    for (int h = 0; h < NSL; ++h) {
      const int q = j * NSL + h, s = q & 1;
      float* vs = v + 16 * h;
      if (FOLD) {
        ok = __all_sync(kFull, mbar_wait_bounded(tc.fbar, (uint32_t)(q & 1)) && ok);
        tc_fence_after();
        float d[16];
        tmem_ld16(ta + kTcDf, d);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const ST sv = tc_st<ST>(fmaf(decay, vs[r], d[r]));
          vs[r] = tc_f32(sv);
          if (ok) gtile[(size_t)(16 * q + r) * DV + col] = sv;
        }
      }
      // the MMAs of slice q - 2 have read A stage s
      if (q >= 2) {
        ok = __all_sync(kFull, mbar_wait_bounded(&tc.aempty[s], (uint32_t)(((q - 2) >> 1) & 1)) &&
                                   ok);
        tc_fence_after();
      }
      float hi[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) hi[r] = EXACT_S ? vs[r] : tf32_hi(vs[r]);
      __syncwarp();
      tmem_st16(ta + kTcA + 32 * s, hi);
      if (!EXACT_S) {
#pragma unroll
        for (int r = 0; r < 16; ++r) hi[r] = vs[r] - hi[r];
        tmem_st16(ta + kTcA + 32 * s + 16, hi);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tc.afull[s]);
      if (tid == 0) {
        ok = mbar_wait_bounded(&tc.afull[s], (uint32_t)((q >> 1) & 1)) && ok;
        tc_fence_after();
        if (FOLD && q + 1 < nslice) tc_issue_fold(tc, q + 1, dk);
        tc_issue_matvec<EXACT_S>(tc, q, s);
      }
    }
  }
  if (tid == 0) mma_commit(tc.ydone);
  return ok;
}

// Column sums of the tensor-core stream -> red[v][col] (thread tid = column).
template <int NV>
__device__ __forceinline__ bool tc_read_y(const TcStream& tc, float* red, int dv, int tid,
                                          int warp) {
  const bool ok = mbar_wait_bounded(tc.ydone, 0);
  tc_fence_after();
  const uint32_t ta = tmem_lane(tc.tbase, warp) + kTcY;
  if constexpr (NV == 16) {
    float y[16];
    tmem_ld16(ta, y);
#pragma unroll
    for (int v = 0; v < 16; ++v) red[v * dv + tid] = y[v];
  } else {
    float y[8];
    tmem_ld8(ta, y);  // columns [0, 8) of the 16
#pragma unroll
    for (int v = 0; v < 8; ++v) red[v * dv + tid] = y[v];
  }
  return ok;
}

}  // namespace rssm
