// Shared definitions of the ReplaySSM kernels: launch parameters, the shared
// memory plans, dtype helpers and the inline-PTX primitives (mbarrier, bulk
// async copy) used on sm_103a.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace rssm {

enum : int { ALGO_GDN = 0, ALGO_KDA = 1 };
enum : int { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };
enum : uint32_t {
  DEVERR_SLOT = 1u,
  DEVERR_CURSOR = 2u,
  DEVERR_ACCEPT = 4u,
  DEVERR_TIMEOUT = 8u,
  DEVERR_SEQLEN = 16u,
};
enum : int {
  CURSOR_DECODE = 0,
  CURSOR_COMMIT_LAZY = 1,
  CURSOR_ZERO = 2,
  CURSOR_COMMIT_FOLD = 3,
  CURSOR_PREFILL = 4  // cursor <- 0 for rows with prompt tokens (cu)
};
enum : int { FOLD_ALL = 0, FOLD_COMMIT = 1 };

constexpr int kThreads = 128;  // 4 warps per CTA, one CTA per (row, value head)
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;
// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 500ull * 1000ull * 1000ull;

// Test hook of the bounded waits, off (withhold < 0) in every ordinary call:
// the copies that complete on barrier `withhold` (0 the window rows, 1 the
// history records, 2 + j chunk j of the checkpoint tile) register 16 more
// bytes than they carry, so no copy can complete that barrier and every wait
// on it runs out. Nothing faults: the copies themselves all land.
enum : int { WH_OFF = -1, WH_WINDOW = 0, WH_HIST = 1, WH_CHUNK0 = 2 };
struct WaitHook {
  int withhold;
  __host__ __device__ uint32_t extra(int barrier) const {
    return withhold == barrier ? 16u : 0u;
  }
};

__host__ __device__ constexpr int dtype_bytes(int dt) { return dt == DT_F32 ? 4 : 2; }
__host__ __device__ constexpr uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

// The checkpoint tile streams through a ring of kStages shared-memory stages,
// each holding one chunk of whole rows (at most kChunkBytes) moved by one bulk
// async copy.
constexpr int kStages = 4;
constexpr int kChunkBytes = 8192;

// mbarriers of one CTA: the window rows, the history records, then one "full"
// and one "empty" barrier per stage of the tile ring.
constexpr int kMbarWin = 0;
constexpr int kMbarHist = 1;
constexpr int kMbarFull = 2;
constexpr int kMbarEmpty = 2 + kStages;
// tensor-core stream (rssm_tc.cuh): A stage written [2], A stage read [2], fold
// slice done, mat-vec done, and an 8-byte slot for the tensor-memory address
constexpr int kMbarAFull = 2 + 2 * kStages;
constexpr int kMbarAEmpty = kMbarAFull + 2;
constexpr int kMbarFoldTc = kMbarAFull + 4;
constexpr int kMbarYDone = kMbarAFull + 5;
constexpr int kMbarTmem = kMbarAFull + 6;
constexpr int kMbars = kMbarAFull + 7;

// Geometry of the tile ring for a [dk][dv] tile of `state_bytes`-byte elements.
struct TileRing {
  int cr;       // rows per chunk
  int nchunk;   // chunks per tile
  int ns;       // stages in use
  uint32_t chunk_bytes;
  __host__ __device__ TileRing(int dk, int dv, int state_bytes, int stages = kStages) {
    const int rowb = dv * state_bytes;
    cr = kChunkBytes / rowb < dk ? kChunkBytes / rowb : dk;
    nchunk = dk / cr;
    ns = nchunk < stages ? nchunk : stages;
    chunk_bytes = (uint32_t)(cr * rowb);
  }
};

// Byte offsets into the dynamic shared memory of the replay kernel.
struct ReplaySmem {
  uint32_t ring;   // tile ring: ns stages of one chunk each (offset 0)
  uint32_t mbar;   // kMbars mbarriers
  uint32_t wq;     // [T][dk]  window q (fp32)
  uint32_t wk;     // [T][dk]  window k (fp32)
  uint32_t wv;     // [T][dv]  window v (fp32)
  uint32_t wraw;   // raw 16-bit window rows q [T][dk], k [T][dk], v [T][dv] (16-bit inputs)
  uint32_t wb;     // [NT]     window beta
  uint32_t wg;     // [T] (GDN) | [T][dk] (KDA): window gates -> inclusive prefix
  uint32_t yk;     // KDA [T][dk]: e^{G_i} * k_i (history dots)
  uint32_t yq;     // KDA [T][dk]: e^{G_i} * q_i
  uint32_t scal;   // GDN: es[NT], eG[NT], Gam, e^Gam, G[NT]; KDA: egam[dk], gam[dk]
  uint32_t xh;     // [dk][2NT] mat-vec inputs (tensor-core stream: K-major, 16 vectors)
  uint32_t xl;     // tensor-core stream, fp32 inputs: the lo parts of xh
  uint32_t am;     // [NT][NT] window coefficients A (strictly lower)
  uint32_t fm;     // [NT][NT] window coefficients F (lower incl. diagonal)
  uint32_t hk;     // [L][dk] fp32 history keys (KDA: decay-scaled), or for a GDN fold the
                   // transposed keys [dk][round4(n)] (tensor-core stream: K-major, 16 records)
  uint32_t kl;     // tensor-core stream, fp32 ring keys: the lo parts of the fold keys
  uint32_t hkraw;  // [L][dk]  history keys as stored in the ring (landing zone of the copy;
                   // KDA fp32 keys land in hk); split GDN windows reuse it for the history
                   // correction hc [NV][dv]
  uint32_t hd;     // [L][dv]  history deltas (fp32)
  uint32_t hdraw;  // [L][dv]  raw 16-bit history deltas (16-bit ring deltas)
  uint32_t hg;     // [L][dk]  KDA history gates (a fold: transposed decayed keys)
  uint32_t hf;     // [L]      GDN: raw gates -> exp(suffix sums)
  uint32_t hdot;   // [L][2NT] history dot coefficients
  uint32_t red;    // [row groups][2NT][dv] partial column sums (on the ring when it fits)
  uint32_t rank;   // decode row order: [kThreads] (slot, cursor), [kWarps] fold masks
  uint32_t kip;    // 1: GDN decode on a long ring with 16-bit keys; a fold transposes the
                   // landed keys in place ([dk][round4(n)], 16-bit) and hk is empty
  uint32_t ns;     // tile ring stages
  uint32_t total;
};

// Lane layout of the tile stream: a lane owns CW consecutive value columns
// (one vector load per row); the lanes of a row may span several warps
// (column blocks) and a warp instruction may cover several rows.
struct QuadLayout {
  int lpr;   // lanes per row (dv / CW)
  int wcb;   // warps per row (column blocks)
  int rsw;   // rows covered by one warp instruction
  int rgw;   // warp row groups (warps / wcb): partial sums to add
  __host__ __device__ QuadLayout(int dv, int CW, int warps) {
    lpr = dv / CW;
    wcb = lpr > 32 ? lpr / 32 : 1;
    rsw = lpr < 32 ? 32 / lpr : 1;
    rgw = warps / wcb;
  }
};

// Columns per lane in the tile stream for a window width.
__host__ __device__ constexpr int quad_width(int NT) { return NT <= 4 ? 4 : 2; }

// Stages of the tile ring for a window width and ring length: decode on rings
// of up to 16 records keeps four (a 64 KB fp32 tile in two round trips);
// verify windows and longer rings take three, which with their larger window
// or history arrays keeps more CTAs per SM (the width-16 window keeps four:
// its partial sums fill the drained ring). Measured on 128-row verify: T = 8
// 219 -> 173 us, T = 3 127 -> 101 us per launch.
__host__ __device__ constexpr int ring_stages(int NT, int L) {
  return (NT == 1 && L <= 16) || NT == 16 ? 4 : 3;
}

// Narrow GDN windows without a fold split the CTA: kSplitWarps warps stream
// the checkpoint tile while the others stage the history and compute the
// window and history coefficients.
constexpr int kSplitWarps = 2;
// longest history the verify kernel's tensor-core fold takes (in groups of 16)
constexpr int kMmaFoldRecords = 64;
__host__ __device__ constexpr bool can_split(int algo, int NT) {
  return algo == ALGO_GDN && NT <= 4;
}

// Fused fold: the deltas of the first fold_reg_records(NT) history records
// stay in registers for the whole tile.
__host__ __device__ constexpr int fold_reg_records(int NT) {
  return NT == 1 ? 16 : NT <= 4 ? 8 : 16;
}

__host__ __device__ constexpr int round4(int x) { return (x + 3) & ~3; }

struct ReplayParams {
  // store (layer offset already applied)
  void* state;
  void* ring_k;
  void* ring_d;
  float* ring_g;
  void* ring_v;
  float* ring_beta;
  const int32_t* cursor;
  uint32_t* err;
  // window
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* g;
  const int32_t* slot;
  const uint8_t* force;
  const int32_t* cu;  // ragged windows: row r's tokens [cu[r], cu[r+1]); null: r*T + [0, T)
  void* o;
  uint8_t* fold_out;
  int B, T, L, n_slots, HK, HV, G, dk, dv;  // T: the window (ragged: the widest allowed)
  int in_dt, rk_dt, rd_dt;
  float scale;
  WaitHook hook;
  int tc;  // GDN windows of 3..8 tokens stream on the 5th-generation tensor cores
  ReplaySmem sm;
};

struct FoldSmem {
  uint32_t ring, mbar, hk, hkraw, hd, hdraw, hg, hf, scal, hkt, bf, bl, total;
};

struct FoldParams {
  void* state;
  const void* ring_k;
  const void* ring_d;
  const float* ring_g;
  const int32_t* cursor;
  uint32_t* err;
  const int32_t* slot;
  const uint8_t* force;
  const int32_t* accept;
  const int32_t* cu;  // ragged windows (as in ReplayParams), or null
  size_t layer_state, layer_k, layer_d, layer_g;  // per-layer strides (elements)
  int B, T, L, n_slots, HK, HV, G, dk, dv;
  int rk_dt, rd_dt, mode;
  WaitHook hook;
  int tc;  // GDN folds on the 5th-generation tensor cores (fold_tc_kernel)
  FoldSmem sm;
};



// Window of request row r: its first token and length. Uniform windows hold
// T tokens at r*T; ragged ones cu[r+1] - cu[r] tokens at cu[r] (at most T).
// Returns false for offsets out of order or a window wider than T.
__device__ __forceinline__ bool row_window(const int32_t* cu, int r, int T, size_t& tok0,
                                           int& n) {
  if (cu == nullptr) {
    tok0 = (size_t)r * T;
    n = T;
    return true;
  }
  const int a = cu[r], b = cu[r + 1];
  tok0 = (size_t)(a < 0 ? 0 : a);
  n = b - a;
  return a >= 0 && n >= 0 && n <= T;
}

// --------------------------------------------------------------- conv window
enum : int { CONV_ACT_NONE = 0, CONV_ACT_SILU = 1 };
constexpr int kConvMaxK = 8;  // widest causal convolution built

struct ConvParams {
  const void* x;       // [B*T][D]
  const float* w;      // [D][K]
  const float* bias;   // [D] or null
  void* window;        // [n_slots][K-1][D]
  void* draft;         // [n_slots][T][D]
  const int32_t* slot;
  const int32_t* accept;
  void* y;             // [B*T][D]
  uint32_t* err;       // may be null
  int B, T, D, K, n_slots, dt, act, commit_now;
};

// ------------------------------------------------------------------ prefill
constexpr int kPrefillChunk = 16;     // prompt tokens per step of the prefill scan
constexpr int kPrefillThreads = 256;  // threads of a prefill CTA

// Chunk arrays marked x2 have one copy per chunk parity: the next chunk is
// prepared while the current one is solved.
struct PrefillSmem {
  uint32_t S;     // [dk][CB + 8]  fp32 state columns of this CTA (row stride CB + 8)
  uint32_t wq;    // [C][dk]   fp32 chunk q
  uint32_t wk;    // [C][dk]   fp32 chunk k (history replay: ring keys)
  uint32_t wv;    // x2 [C][CB]  fp32 chunk v columns
  uint32_t xT;    // [dk][kPrefillXS] mat-vec and pair inputs per key channel
  uint32_t kdT;   // [dk][kPrefillKS] the update's decayed keys
  uint32_t y;     // [2C][CB + 8]  S^T k_i, S^T q_i (decay applied)
  uint32_t part;  // [2C][C]   GDN pair sums k_i.k_j, q_i.k_j
  uint32_t dch;   // [C][CB + 8]  chunk deltas (history replay: ring deltas)
  uint32_t am;    // x2 [C][kPrefillKS]  window coefficients A (row stride kPrefillKS)
  uint32_t fm;    // x2 [C][kPrefillKS]  window coefficients F
  uint32_t G;     // GDN [C] / KDA [C][dk] in-chunk inclusive gate prefixes
  uint32_t eG;    // GDN [C] e^{G_i}
  uint32_t ekd;   // GDN [C] e^{G_last - G_i}
  uint32_t wb;    // x2 [C] betas
  uint32_t decr;  // KDA x2 [dk] e^{G_last} per key channel
  uint32_t total;
};

struct PrefillParams {
  void* state;
  const void* ring_k;
  const void* ring_d;
  const float* ring_g;
  const int32_t* cursor;
  uint32_t* err;
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* g;
  const int32_t* cu;
  const int32_t* slot;
  void* o;
  int B, L, n_slots, HK, HV, G, dk, dv, CB;
  int in_dt, rk_dt, rd_dt;
  float scale;
  PrefillSmem sm;
};

// Value columns per prefill CTA (the columns of the delta rule are independent).
__host__ __device__ constexpr int prefill_cb(int dv) { return dv < 64 ? dv : 64; }

// Row strides (floats) of the per-channel arrays. The padding puts the
// tensor-core fragment loads (lanes over 4 rows x 8 columns) on 32 distinct
// banks: row strides of 8 (mod 32) floats for the mat-vec and pair inputs,
// of 20 for the update's keys and the coefficients F, and CB + 8 for the
// state, the deltas and the mat-vec results.
constexpr int kPrefillXS = 2 * kPrefillChunk + 8;
constexpr int kPrefillKS = kPrefillChunk + 4;

__host__ __device__ inline PrefillSmem prefill_layout(int algo, int dk, int dv) {
  constexpr int C = kPrefillChunk;
  const int CB = prefill_cb(dv);
  const bool kda = algo == ALGO_KDA;
  PrefillSmem m{};
  uint32_t off = 0;
  m.S = off;     off = align16(off + 4u * dk * (CB + 8));
  m.wq = off;    off = align16(off + 4u * C * dk);
  m.wk = off;    off = align16(off + 4u * C * dk);
  m.wv = off;    off = align16(off + 2u * 4u * C * CB);
  m.xT = off;    off = align16(off + 4u * dk * kPrefillXS);
  m.kdT = off;   off = align16(off + 4u * dk * kPrefillKS);
  m.y = off;     off = align16(off + 4u * 2 * C * (CB + 8));
  m.part = off;  off = align16(off + 4u * 2 * C * C);
  m.dch = off;   off = align16(off + 4u * C * (CB + 8));
  m.am = off;    off = align16(off + 2u * 4u * C * kPrefillKS);
  m.fm = off;    off = align16(off + 2u * 4u * C * kPrefillKS);
  m.G = off;     off = align16(off + 4u * (kda ? C * dk : C));
  m.eG = off;    off = align16(off + 4u * C);
  m.ekd = off;   off = align16(off + 4u * C);
  m.wb = off;    off = align16(off + 2u * 4u * C);
  m.decr = off;  off = align16(off + 2u * 4u * dk);
  m.total = off;
  return m;
}

constexpr uint32_t kRankBytes = 8u * kThreads + 4u * kWarps;

// Shared memory plan of the replay kernel for a window of T <= NT tokens, a
// ring of L records and a tile ring of `stages` stages.
__host__ __device__ inline ReplaySmem replay_layout_ns(int algo, int state_bytes, int NT, int T,
                                                       int L, int dk, int dv, int in_dt,
                                                       int rk_dt, int rd_dt, bool tc,
                                                       int stages) {
  ReplaySmem m{};
  const int NV = 2 * NT;
  const bool kda = algo == ALGO_KDA;
  const TileRing tr(dk, dv, state_bytes, stages);
  m.ns = (uint32_t)tr.ns;
  const QuadLayout ql(dv, quad_width(NT), kWarps);
  uint32_t off = 0;
  m.ring = off;  off = align16(off + tr.ns * tr.chunk_bytes);
  m.mbar = off;  off = align16(off + 8u * kMbars);
  m.wq = off;    off = align16(off + 4u * T * dk);
  m.wk = off;    off = align16(off + 4u * T * dk);
  m.wv = off;    off = align16(off + 4u * T * dv);
  m.wraw = off;  if (in_dt != DT_F32) off = align16(off + 2u * T * (2 * dk + dv));
  m.wb = off;    off = align16(off + 4u * NT);
  m.wg = off;    off = align16(off + 4u * (kda ? T * dk : NT));
  m.yk = off;    if (kda) off = align16(off + 4u * T * dk);
  m.yq = off;    if (kda) off = align16(off + 4u * T * dk);
  m.scal = off;  off = align16(off + 4u * (kda ? 2 * dk : 3 * NT + 4));
  m.xh = off;    off = align16(off + 4u * dk * (tc ? 16 : NV));
  m.xl = off;    if (tc && in_dt == DT_F32) off = align16(off + 4u * dk * 16);
  m.am = off;    off = align16(off + 4u * NT * NT);
  m.fm = off;    off = align16(off + 4u * NT * NT);
  // GDN decode on a ring of 17..kMmaFoldRecords records with 16-bit keys and
  // 128 value columns: every fold runs on the tensor cores, which take the
  // keys transposed in place in their landing zone (at most eight 16-byte
  // rows of keys per thread), so the fp32 key region is left out
  const bool kip = algo == ALGO_GDN && NT == 1 && L > 16 && L <= kMmaFoldRecords &&
                   rk_dt != DT_F32 && dv == 128 && dk % 16 == 0 && dk >= 32 &&
                   round4(L) * dk <= 64 * kThreads;
  m.kip = kip ? 1u : 0u;
  m.hk = off;    if (!kip) off = align16(off + 4u * round4(L) * dk);
  m.kl = off;    if (tc && rk_dt == DT_F32) off = align16(off + 4u * 16 * dk);
  {
    // ring keys land in hkraw; KDA's record gates land in hk and become the
    // decayed keys there
    const uint32_t raw = (uint32_t)(kip ? 2 * round4(L) * dk : dtype_bytes(rk_dt) * L * dk);
    const uint32_t hc = can_split(algo, NT) ? 4u * NV * dv : 0u;
    m.hkraw = off; off = align16(off + (raw > hc ? raw : hc));
  }
  // (KDA reads 16-bit deltas where they landed: no widened copy)
  const bool kda_d16 = kda && rd_dt != DT_F32;
  m.hd = off;    if (!kda_d16) off = align16(off + 4u * L * dv);
  m.hdraw = off; if (rd_dt != DT_F32) off = align16(off + 2u * L * dv);
  if (kda_d16) m.hd = m.hdraw;
  m.hg = off;
  m.hf = off;    off = align16(off + 4u * L);
  m.hdot = off;  off = align16(off + 4u * L * NV);
  // partial column sums go to the ring once the tile is consumed, if they fit
  const uint32_t red_bytes = 4u * ql.rgw * NV * dv;
  if (red_bytes <= tr.ns * tr.chunk_bytes) {
    m.red = m.ring;
  } else {
    m.red = off;
    off = align16(off + red_bytes);
  }
  // The decode row order sits in the fp32 history keys: nothing writes there
  // before the CTA barrier that follows the copies (ring keys land in hkraw),
  // unless KDA's gates land there (they get a region of their own).
  m.rank = m.hk;
  if (NT == 1 && (kda || kip || 4u * round4(L) * dk < kRankBytes)) {
    m.rank = off;
    off = align16(off + kRankBytes);
  }
  // the tensor-core stream holds kTmemCols of the SM's 512 tensor-memory
  // columns: at most four such CTAs may share an SM
  if (tc && off < 47u * 1024u) off = 47u * 1024u;
  m.total = off;
  return m;
}

// CTAs of one kernel that fit an SM's 228 KB of shared memory (1 KB of which
// each CTA's launch reserves)
__host__ __device__ constexpr uint32_t ctas_per_sm(uint32_t smem) {
  return 233472u / (smem + 1024u);
}

// The replay kernel's plan: ring_stages(NT, L) stages, or one fewer where that
// fits one more CTA per SM (long KDA rings with 16-bit deltas or checkpoints).
__host__ __device__ inline ReplaySmem replay_layout(int algo, int state_bytes, int NT, int T,
                                                    int L, int dk, int dv, int in_dt, int rk_dt,
                                                    int rd_dt, bool tc = false) {
  const int st = ring_stages(NT, L);
  const ReplaySmem m = replay_layout_ns(algo, state_bytes, NT, T, L, dk, dv, in_dt, rk_dt, rd_dt,
                                        tc, st);
  if (st <= 2) return m;
  const ReplaySmem m2 = replay_layout_ns(algo, state_bytes, NT, T, L, dk, dv, in_dt, rk_dt,
                                         rd_dt, tc, st - 1);
  return ctas_per_sm(m2.total) > ctas_per_sm(m.total) ? m2 : m;
}

// ----------------------------------------------------------- pipelined replay
// Persistent replay kernel (pipe_impl.cuh): one CTA per SM walks a list of
// (row, value head) items. Warps 0-3 stream the checkpoint tiles, warps 4-7
// prepare the next item and solve the previous one, warps 8-11 issue every
// async copy (checkpoint chunks into a ring that runs across items, window
// and history rows into two item buffers).
constexpr int kPipeMath = 4;                       // warps streaming the tile
constexpr int kPipePrep = 4;                       // warps preparing / solving items
constexpr int kPipeProd = kPipeMath + kPipePrep;   // first copy-issuing warp
constexpr int kPipeProdWarps = 4;                  // copy-issuing warps
constexpr int kPipeThreads = 32 * (kPipeProd + kPipeProdWarps);
constexpr int kPipeMaxRows = 512;                  // request rows ranked in shared memory
constexpr int kPipeMaxStages = 16;                 // chunk ring stages at most
constexpr int kPipeHist = 16;                      // history records an item folds / corrects
constexpr int kPipeMaxNT = 8;                      // widest window

// barriers: window copies [2], item prepared [2], item streamed [2], column sums
// read [2], then "full" and "empty" per ring stage
enum : int { PB_WIN = 0, PB_PREP = 2, PB_MATH = 4, PB_YFREE = 6, PB_FULL = 8 };
constexpr int kPipeMbars = PB_FULL + 2 * kPipeMaxStages;

// Per-item scalars shared by the roles (one copy per item buffer).
struct PipeItem {
  int row, h, s, c, base, fold, n, pad;
  float egam;                    // e^Gam of the history (the fold's decay, or the scale of
                                 // the checkpoint term of a window that does not fold)
  float beta[kPipeMaxNT], eG[kPipeMaxNT], G[kPipeMaxNT];
  float hf[kPipeHist];           // e^{Gam - Gam_m}: decay of record m to the end of the history
  float am[kPipeMaxNT * kPipeMaxNT], fm[kPipeMaxNT * kPipeMaxNT];
};

// Shared memory of the pipelined kernel. The two item buffers have the same
// layout: buffer b starts at buf + b * bufsz and its arrays sit at the offsets
// below within it (so a buffer is chosen by arithmetic, not by indexing a
// kernel parameter, which would put the parameter block in local memory).
struct PipeSmem {
  uint32_t ring;                 // ns stages of one 8 KB chunk
  uint32_t mbar;                 // kPipeMbars barriers, then the abort word
  uint32_t rows;                 // slot, cursor, order, flags [maxb] (int32), group counts
  uint32_t bg;                   // window beta and gate of every item of the CTA [nkmax][NT][2]
  uint32_t buf, bufsz;           // item buffer 0, size of one buffer
  uint32_t item;                 // PipeItem
  uint32_t wraw;                 // window q, k, v rows as stored [3][NT][dk]
  uint32_t ep;                   // window k, v rows kept for the solve [2][NT][dk]
  uint32_t hkr;                  // history keys as stored [16][dk]
  uint32_t hdr;                  // history deltas as stored [16][dv]
  uint32_t hgr;                  // history gates [16] fp32
  uint32_t xh;                   // mat-vec inputs [dk][2 NT] fp32 (k_i at i, q_i at NT + i)
  uint32_t hkt;                  // history keys transposed [dk][16] fp32 (a fold)
  uint32_t dt;                   // f_m d_m [16][dv] fp32
  uint32_t hh;                   // history dots k_m . x_v [16][2 NT] fp32
  uint32_t y;                    // column sums [2 NT][dv]
  uint32_t total;
  int ns;                        // ring stages
  int maxb;                      // rows the ranking tables hold (a multiple of 32, >= B)
  int nkmax;                     // items of one CTA at most
};

// Layout for windows of up to NT tokens; the ring takes what is left of
// max_smem (at most kPipeMaxStages stages). ns < 2 means it does not fit.
__host__ __device__ inline PipeSmem pipe_layout(int NT, int B, int dk, int dv, int in_dt,
                                                int rk_dt, int rd_dt, int max_smem, int nkmax) {
  PipeSmem m{};
  const int nv = 2 * NT;
  m.maxb = (B + 31) & ~31;
  m.nkmax = nkmax;
  uint32_t off = 0;
  m.mbar = off;  off = align16(off + 8u * kPipeMbars + 16u);
  m.rows = off;  off = align16(off + 16u * m.maxb + 8u * (kPipeMaxRows / 32));
  m.bg = off;    off = align16(off + 8u * nkmax * NT);
  m.buf = off;
  uint32_t o = 0;  // within one buffer
  m.item = o;  o = align16(o + (uint32_t)sizeof(PipeItem));
  m.wraw = o;  o = align16(o + 3u * NT * dk * dtype_bytes(in_dt));
  m.ep = o;    o = align16(o + 2u * NT * dk * dtype_bytes(in_dt));
  m.hkr = o;   o = align16(o + (uint32_t)(kPipeHist * dk * dtype_bytes(rk_dt)));
  m.hdr = o;   o = align16(o + (uint32_t)(kPipeHist * dv * dtype_bytes(rd_dt)));
  m.hgr = o;   o = align16(o + 4u * kPipeHist);
  m.xh = o;    o = align16(o + 4u * dk * nv);
  m.hkt = o;   o = align16(o + 4u * dk * kPipeHist);
  m.dt = o;    o = align16(o + 4u * kPipeHist * dv);
  m.hh = o;    o = align16(o + 4u * kPipeHist * nv);
  m.y = o;     o = align16(o + 4u * nv * dv);
  m.bufsz = o;
  off += 2u * o;
  off = (off + 127u) & ~127u;
  m.ring = off;
  const int room = (max_smem - (int)off) / kChunkBytes;
  m.ns = room < kPipeMaxStages ? room : kPipeMaxStages;
  m.total = off + (uint32_t)(m.ns > 0 ? m.ns : 0) * kChunkBytes;
  return m;
}

// Native fused-recurrent decode: the whole tile, one mbarrier for the window
// and one per chunk, the window, the mat-vec inputs and the partial sums.
struct NativeSmem {
  uint32_t ring, mbar, wq, wk, wv, wraw, wg, xh, red, dsh, scal, total;
};

__host__ __device__ inline NativeSmem native_layout(int algo, int state_bytes, int dk, int dv,
                                                    int in_dt) {
  NativeSmem m{};
  const TileRing tr(dk, dv, state_bytes, 1 << 30);
  const QuadLayout ql(dv, 4, kWarps);
  uint32_t off = 0;
  m.ring = off;  off = align16(off + tr.nchunk * tr.chunk_bytes);
  m.mbar = off;  off = align16(off + 8u * (1 + tr.nchunk));
  m.wq = off;    off = align16(off + 4u * dk);
  m.wk = off;    off = align16(off + 4u * dk);
  m.wv = off;    off = align16(off + 4u * dv);
  m.wraw = off;  if (in_dt != DT_F32) off = align16(off + 2u * (2 * dk + dv));
  m.wg = off;    if (algo == ALGO_KDA) off = align16(off + 4u * dk);
  m.xh = off;    off = align16(off + 8u * dk);
  m.red = off;   off = align16(off + 8u * ql.rgw * dv);
  m.dsh = off;   off = align16(off + 4u * dv);
  m.scal = off;  off = align16(off + 4u * kWarps);
  m.total = off;
  return m;
}

__host__ __device__ inline FoldSmem fold_layout(int algo, int state_bytes, int L, int dk, int dv,
                                                int rk_dt, int rd_dt) {
  FoldSmem m{};
  const bool kda = algo == ALGO_KDA;
  const TileRing tr(dk, dv, state_bytes);
  // the fold stream reads the keys transposed, [dk][nb] with the record count
  // rounded up to 4 .. 64: in hk for GDN 16-bit keys (read from the landing
  // zone), else in hg (GDN fp32 keys land in hk; KDA's gates are consumed
  // before its decayed keys are transposed)
  const int nb = L <= 4 ? 4 : L <= 8 ? 8 : L <= 16 ? 16 : L <= 32 ? 32 : 64;
  const bool own_hkt = kda || rk_dt == DT_F32;
  uint32_t off = 0;
  m.ring = off;  off = align16(off + tr.ns * tr.chunk_bytes);
  m.mbar = off;  off = align16(off + 8u * kMbars);
  m.hk = off;    off = align16(off + 4u * nb * dk);
  m.hkraw = off; if (rk_dt != DT_F32) off = align16(off + 2u * L * dk);
  m.hd = off;    off = align16(off + 4u * L * dv);
  m.hdraw = off; if (rd_dt != DT_F32) off = align16(off + 2u * L * dv);
  m.hg = off;    if (own_hkt) off = align16(off + 4u * nb * dk);
  m.hkt = own_hkt ? m.hg : m.hk;
  m.hf = off;    off = align16(off + 4u * L);
  m.scal = off;  off = align16(off + 4u * (kda ? 2 * dk : 4));
  m.total = off;
  return m;
}

// Fold on the tensor cores (GDN): ring, barriers, the ring records as copied
// (keys in any dtype land in hkraw), fp32 deltas, gates, and the fold keys
// K-major for up to round8(L) records (hi in bf, lo in bl for fp32 keys).
__host__ __device__ inline FoldSmem fold_tc_layout(int state_bytes, int L, int dk, int dv,
                                                   int rk_dt, int rd_dt) {
  FoldSmem m{};
  const TileRing tr(dk, dv, state_bytes);
  const int K = (L + 7) & ~7;
  uint32_t off = 0;
  m.ring = off;  off = align16(off + tr.ns * tr.chunk_bytes);
  m.mbar = off;  off = align16(off + 8u * kMbars);
  m.hkraw = off; off = align16(off + (uint32_t)(dtype_bytes(rk_dt) * L * dk));
  m.hk = m.hkraw;
  m.hd = off;    off = align16(off + 4u * L * dv);
  m.hdraw = off; if (rd_dt != DT_F32) off = align16(off + 2u * L * dv);
  m.hg = off;
  m.hf = off;    off = align16(off + 4u * L);
  m.scal = off;  off = align16(off + 16u);
  m.bf = off;    off = align16(off + 4u * K * dk);
  m.bl = off;    if (rk_dt == DT_F32) off = align16(off + 4u * K * dk);
  // kTmemCols of the SM's 512 tensor-memory columns: at most four CTAs per SM
  if (off < 47u * 1024u) off = 47u * 1024u;
  m.total = off;
  return m;
}

#if defined(__CUDACC__)

// ------------------------------------------------------------------ dtypes
__device__ __forceinline__ float ld_f32(const void* base, size_t i, int dt) {
  if (dt == DT_F32) return static_cast<const float*>(base)[i];
  if (dt == DT_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
  return __half2float(static_cast<const __half*>(base)[i]);
}

// Two consecutive values at element i (i even) as fp32.
__device__ __forceinline__ float2 ld2_f32(const void* base, size_t i, int dt) {
  if (dt == DT_F32) return *reinterpret_cast<const float2*>(static_cast<const float*>(base) + i);
  if (dt == DT_BF16) {
    return __bfloat1622float2(
        *reinterpret_cast<const __nv_bfloat162*>(static_cast<const __nv_bfloat16*>(base) + i));
  }
  return __half22float2(*reinterpret_cast<const __half2*>(static_cast<const __half*>(base) + i));
}

// Widen n 16-bit values (bf16 or fp16) in shared memory to fp32, eight at a
// time (n a multiple of 8, both buffers 16-byte aligned).
__device__ __forceinline__ void widen16x8(float* dst, const void* src, int n, int dt, int tid,
                                          int nthreads) {
  {
    const uint4* s8 = static_cast<const uint4*>(src);
    float4* d4 = reinterpret_cast<float4*>(dst);
    for (int e = tid; e < n / 8; e += nthreads) {
      const uint4 u = s8[e];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      float f[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 t;
        if (dt == DT_BF16) {
          t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        } else {
          t = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
        }
        f[2 * k] = t.x;
        f[2 * k + 1] = t.y;
      }
      d4[2 * e] = make_float4(f[0], f[1], f[2], f[3]);
      d4[2 * e + 1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
}

// Widen n 16-bit values (bf16 or fp16) in shared memory to fp32.
__device__ __forceinline__ void widen16(float* dst, const void* src, int n, int dt, int tid,
                                        int nthreads) {
  if (dt == DT_BF16) {
    const __nv_bfloat16* s = static_cast<const __nv_bfloat16*>(src);
    for (int e = tid; e < n; e += nthreads) dst[e] = __bfloat162float(s[e]);
  } else {
    const __half* s = static_cast<const __half*>(src);
    for (int e = tid; e < n; e += nthreads) dst[e] = __half2float(s[e]);
  }
}

__device__ __forceinline__ void st_f32(void* base, size_t i, int dt, float x) {
  if (dt == DT_F32) {
    static_cast<float*>(base)[i] = x;
  } else if (dt == DT_BF16) {
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(x);
  } else {
    static_cast<__half*>(base)[i] = __float2half_rn(x);
  }
}

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive with an expected byte count, without release semantics: for a
// thread that only issues async copies (a release would order it behind the
// copies it already has in flight).
__device__ __forceinline__ void mbar_expect_tx_relaxed(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// 16-byte async copy global -> shared (cache at L2 only), and an arrive on
// `bar` once every such copy this thread has issued so far has completed
// (the barrier's expected count includes the arrival).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Wait for phase `parity` of `bar` for up to about hint_ns, the thread parked
// by the hardware meanwhile (it resumes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking test of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The arrival that registers a copy's byte count is made by the thread that
// issues the copies, and it carries no release semantics: nothing the thread
// wrote before is published through it (the data comes with the copy), and on
// this part a release by a thread waits for the copies that thread has in
// flight, which serialised each refill of a tile ring behind the copy before.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  mbar_expect_tx_relaxed(bar, bytes);
}

// One bulk (non-tensor) async copy global -> shared, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar`, giving up after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}



// Barrier over the `count` threads (a multiple of 32) that name barrier `id`
// (id 0 is the one __syncthreads uses).
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
  return x;
}

#endif  // __CUDACC__

}  // namespace rssm
