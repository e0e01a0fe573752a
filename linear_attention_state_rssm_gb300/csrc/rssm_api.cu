// C ABI of librssm: host-side validation, per-layer addressing and launches.
// See include/rssm.h for the contract of every entry point.
#include <cmath>
#include <cstring>
#include <new>

#include "../../include/rssm.h"
#include "rssm_common.cuh"
#include "rssm_launch.h"

using namespace rssm;

struct rssm_handle {
  rssm_config cfg;
  rssm_buffers buf;
  int G;
  int max_smem;
  int num_sms;
  size_t layer_state, layer_k, layer_d, layer_g, layer_v, layer_beta;  // elements
  WaitHook hook;  // bounded-wait test hook (off unless rssm_debug_withhold set it)
  bool pipe_cfg;  // the configuration is one the pipelined kernel serves
  int plan;       // RSSM_PLAN_*
};

namespace {

// Rings of up to 64 records: a fold (rssm_fold, a fold-every commit after
// decode history) carries the whole history, and the fold kernel's streams
// take at most 64 records.
constexpr int kMaxL = 64;
constexpr int kMaxT = 16;
constexpr int kMaxGrid = 65535;

bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

int n_gate(const rssm_config& c) { return c.algo == RSSM_ALGO_GDN ? 1 : c.dk; }

rssm_status check_config(const rssm_config* c) {
  if (c == nullptr) return RSSM_ERR_INVALID_ARG;
  if (c->algo != RSSM_ALGO_GDN && c->algo != RSSM_ALGO_KDA) return RSSM_ERR_INVALID_ARG;
  if (c->n_layers < 1 || c->n_slots < 1 || c->HK < 1 || c->HV < 1) return RSSM_ERR_INVALID_ARG;
  if (c->HV % c->HK != 0) return RSSM_ERR_INVALID_ARG;
  if (c->max_T < 1 || c->L < 1) return RSSM_ERR_INVALID_ARG;
  // A ring that cannot hold the widest window is refused up front.
  if (c->max_T > c->L) return RSSM_ERR_INVALID_ARG;
  if (c->dk < 1 || c->dv < 1) return RSSM_ERR_INVALID_ARG;
  if (!(c->in_dtype == RSSM_F32 || c->in_dtype == RSSM_BF16 || c->in_dtype == RSSM_F16))
    return RSSM_ERR_INVALID_ARG;
  if (!(c->state_dtype == RSSM_F32 || c->state_dtype == RSSM_BF16 ||
        c->state_dtype == RSSM_F16))
    return RSSM_ERR_INVALID_ARG;
  if (!(c->ring_k_dtype == RSSM_F32 || c->ring_k_dtype == RSSM_BF16 ||
        c->ring_k_dtype == RSSM_F16))
    return RSSM_ERR_INVALID_ARG;
  if (!(c->ring_d_dtype == RSSM_F32 || c->ring_d_dtype == RSSM_BF16 ||
        c->ring_d_dtype == RSSM_F16))
    return RSSM_ERR_INVALID_ARG;
  if (c->commit_mode != RSSM_COMMIT_LAZY && c->commit_mode != RSSM_COMMIT_FOLD_EVERY)
    return RSSM_ERR_INVALID_ARG;
  if (!std::isfinite(c->scale)) return RSSM_ERR_INVALID_ARG;
  // Valid but not built.
  if (!dim_ok(c->dk) || !dim_ok(c->dv)) return RSSM_ERR_UNSUPPORTED;
  if (c->max_T > kMaxT || c->L > kMaxL) return RSSM_ERR_UNSUPPORTED;
  if (c->in_dtype == RSSM_F16 || c->state_dtype == RSSM_F16 || c->ring_d_dtype == RSSM_BF16)
    return RSSM_ERR_UNSUPPORTED;
  if (c->HV > kMaxGrid || c->n_layers > kMaxGrid) return RSSM_ERR_UNSUPPORTED;
  return RSSM_OK;
}

size_t esize(int dt) { return dt == RSSM_F32 ? 4 : 2; }

void sizes_of(const rssm_config& c, rssm_sizes* s) {
  const size_t ls = (size_t)c.n_layers * c.n_slots;
  s->state = ls * c.HV * c.dk * c.dv * esize(c.state_dtype);
  s->ring_k = ls * c.HV * c.L * c.dk * esize(c.ring_k_dtype);
  s->ring_d = ls * c.HV * c.L * c.dv * esize(c.ring_d_dtype);
  s->ring_g = ls * c.HV * c.L * n_gate(c) * sizeof(float);
  s->ring_v = ls * c.HV * c.L * c.dv * esize(c.in_dtype);
  s->ring_beta = ls * c.HV * c.L * sizeof(float);
  s->cursor = (size_t)c.n_slots * sizeof(int32_t);
  s->err_word = sizeof(uint32_t);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

rssm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA; }

int state_dt(const rssm_config& c) { return c.state_dtype == RSSM_F32 ? DT_F32 : DT_BF16; }

cudaError_t replay_launch(const rssm_config& c, const ReplayParams& p, int NT,
                          cudaStream_t st) {
  const bool f32 = c.state_dtype == RSSM_F32;
  if (p.cu != nullptr) {
    if (c.algo == RSSM_ALGO_GDN) {
      return f32 ? replay_gdn_f32_ragged_launch(p, NT, st)
                 : replay_gdn_bf16_ragged_launch(p, NT, st);
    }
    return f32 ? replay_kda_f32_ragged_launch(p, NT, st)
               : replay_kda_bf16_ragged_launch(p, NT, st);
  }
  if (c.algo == RSSM_ALGO_GDN) {
    return f32 ? replay_gdn_f32_launch(p, NT, st) : replay_gdn_bf16_launch(p, NT, st);
  }
  return f32 ? replay_kda_f32_launch(p, NT, st) : replay_kda_bf16_launch(p, NT, st);
}

cudaError_t replay_prepare(const rssm_config& c, int max_smem) {
  const bool f32 = c.state_dtype == RSSM_F32;
  cudaError_t e;
  if (c.algo == RSSM_ALGO_GDN) {
    e = f32 ? replay_gdn_f32_prepare(max_smem) : replay_gdn_bf16_prepare(max_smem);
    if (e != cudaSuccess) return e;
    return f32 ? replay_gdn_f32_ragged_prepare(max_smem)
               : replay_gdn_bf16_ragged_prepare(max_smem);
  }
  e = f32 ? replay_kda_f32_prepare(max_smem) : replay_kda_bf16_prepare(max_smem);
  if (e != cudaSuccess) return e;
  return f32 ? replay_kda_f32_ragged_prepare(max_smem) : replay_kda_bf16_ragged_prepare(max_smem);
}

ReplaySmem layout_for(const rssm_config& c, int T, int NT, bool tc = false) {
  return replay_layout(c.algo, (int)esize(c.state_dtype), NT, T, c.L, c.dk, c.dv, c.in_dtype,
                       c.ring_k_dtype, c.ring_d_dtype, tc);
}

// the tensor-core stream serves GDN windows of 3..8 tokens with 128 value columns
bool tc_config(const rssm_config& c) {
  return c.algo == RSSM_ALGO_GDN && c.dv == 128 && c.dk % 32 == 0;
}

// the tensor-core fold serves GDN stores with 128 value columns and rings of
// at most 32 records
bool fold_tc_config(const rssm_config& c) {
  return tc_config(c) && c.L <= 32;
}

ReplaySmem layout_for(const rssm_config& c, int T) { return layout_for(c, T, nt_for(T)); }

FoldSmem fold_layout_for(const rssm_config& c) {
  return fold_layout(c.algo, (int)esize(c.state_dtype), c.L, c.dk, c.dv, c.ring_k_dtype,
                     c.ring_d_dtype);
}

template <typename T>
T* at(void* base, size_t elems, size_t esz) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + elems * esz);
}

// Validates the window arguments shared by decode, verify and native decode
// and fills the launch parameters (all but the shared memory plan).
rssm_status window_params(const rssm_handle* h, int32_t layer, const void* q, const void* k,
                          const void* v, const float* beta, const float* g,
                          const int32_t* slot, const uint8_t* force, int32_t B, int32_t T,
                          void* o, uint8_t* fold_out, ReplayParams* out) {
  if (h == nullptr) return RSSM_ERR_INVALID_ARG;
  const rssm_config& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers) return RSSM_ERR_INVALID_ARG;
  if (B < 0 || B > kMaxGrid) return RSSM_ERR_INVALID_ARG;
  if (T < 1 || T > c.max_T) return RSSM_ERR_INVALID_ARG;
  if (B == 0) return RSSM_OK;
  if (!q || !k || !v || !beta || !g || !slot || !o) return RSSM_ERR_INVALID_ARG;
  if (!aligned4(beta) || !aligned4(slot)) return RSSM_ERR_INVALID_ARG;
  // window rows move by bulk copies: 16-byte aligned sources
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return RSSM_ERR_INVALID_ARG;
  if (c.algo == RSSM_ALGO_KDA ? !aligned16(g) : !aligned4(g)) return RSSM_ERR_INVALID_ARG;

  ReplayParams& p = *out;
  p = ReplayParams{};
  const rssm_buffers& b = h->buf;
  p.state = at<char>(b.state, layer * h->layer_state, esize(c.state_dtype));
  p.ring_k = at<char>(b.ring_k, layer * h->layer_k, esize(c.ring_k_dtype));
  p.ring_d = at<char>(b.ring_d, layer * h->layer_d, esize(c.ring_d_dtype));
  p.ring_g = b.ring_g + layer * h->layer_g;
  p.ring_v = at<char>(b.ring_v, layer * h->layer_v, esize(c.in_dtype));
  p.ring_beta = b.ring_beta + layer * h->layer_beta;
  p.cursor = b.cursor;
  p.err = b.err_word;
  p.q = q;
  p.k = k;
  p.v = v;
  p.beta = beta;
  p.g = g;
  p.slot = slot;
  p.force = force;
  p.o = o;
  p.fold_out = fold_out;
  p.B = B;
  p.T = T;
  p.L = c.L;
  p.n_slots = c.n_slots;
  p.HK = c.HK;
  p.HV = c.HV;
  p.G = h->G;
  p.dk = c.dk;
  p.dv = c.dv;
  p.in_dt = c.in_dtype;
  p.rk_dt = c.ring_k_dtype;
  p.rd_dt = c.ring_d_dtype;
  p.scale = c.scale;
  p.hook = h->hook;
  return RSSM_OK;
}

// Whether a store configuration is one the pipelined kernel serves: GDN heads
// of 128 x 128, a ring of at most 16 records (multiple of 4), fp32 or fp16
// deltas.
bool pipe_config(const rssm_config& c) {
  return c.algo == RSSM_ALGO_GDN && c.dk == 128 && c.dv == 128 && c.L <= kPipeHist &&
         c.L % 4 == 0 && (c.ring_d_dtype == RSSM_F32 || c.ring_d_dtype == RSSM_F16);
}

rssm_status window(rssm_handle* h, int32_t layer, const void* q, const void* k, const void* v,
                   const float* beta, const float* g, const int32_t* slot,
                   const uint8_t* force, int32_t B, int32_t T, void* o, uint8_t* fold_out,
                   void* stream, const int32_t* cu = nullptr) {
  ReplayParams p;
  const rssm_status st = window_params(h, layer, q, k, v, beta, g, slot, force, B, T, o,
                                       fold_out, &p);
  if (st != RSSM_OK || B == 0) return st;
  p.cu = cu;
  const rssm_config& c = h->cfg;
  if (cu == nullptr && h->plan == RSSM_PLAN_PIPE && h->pipe_cfg && T <= kPipeMaxNT &&
      B <= kPipeMaxRows) {
    const int NT = pipe_nt(T);
    const long long items = (long long)B * c.HV;
    const int grid = (int)(items < h->num_sms ? items : h->num_sms);
    const int nkmax = (int)((items + grid - 1) / grid);
    const PipeSmem sm = pipe_layout(NT, B, c.dk, c.dv, c.in_dtype, c.ring_k_dtype,
                                    c.ring_d_dtype, h->max_smem, nkmax);
    if (sm.ns >= 4) {
      return from_cuda(pipe_launch(state_dt(c), NT, p, sm, grid, static_cast<cudaStream_t>(stream)));
    }
  }
  const int NT = cu != nullptr ? nt_for_ragged(T) : nt_for(T);
  p.tc = h->plan == RSSM_PLAN_TC && cu == nullptr && tc_config(c) && (NT == 4 || NT == 8);
  p.sm = layout_for(h->cfg, T, NT, p.tc != 0);
  if ((int)p.sm.total > h->max_smem) return RSSM_ERR_UNSUPPORTED;
  return from_cuda(replay_launch(h->cfg, p, NT, static_cast<cudaStream_t>(stream)));
}

NativeSmem native_layout_for(const rssm_config& c) {
  return native_layout(c.algo, (int)esize(c.state_dtype), c.dk, c.dv, c.in_dtype);
}

FoldParams fold_params(const rssm_handle* h, const int32_t* slot, const uint8_t* force,
                       const int32_t* accept, int B, int T, int mode) {
  const rssm_config& c = h->cfg;
  FoldParams p{};
  p.state = h->buf.state;
  p.ring_k = h->buf.ring_k;
  p.ring_d = h->buf.ring_d;
  p.ring_g = h->buf.ring_g;
  p.cursor = h->buf.cursor;
  p.err = h->buf.err_word;
  p.slot = slot;
  p.force = force;
  p.accept = accept;
  p.layer_state = h->layer_state;
  p.layer_k = h->layer_k;
  p.layer_d = h->layer_d;
  p.layer_g = h->layer_g;
  p.B = B;
  p.T = T;
  p.L = c.L;
  p.n_slots = c.n_slots;
  p.HK = c.HK;
  p.HV = c.HV;
  p.G = h->G;
  p.dk = c.dk;
  p.dv = c.dv;
  p.rk_dt = c.ring_k_dtype;
  p.rd_dt = c.ring_d_dtype;
  p.mode = mode;
  p.hook = h->hook;
  p.tc = h->plan == RSSM_PLAN_TC && fold_tc_config(c);
  p.sm = p.tc ? fold_tc_layout((int)esize(c.state_dtype), c.L, c.dk, c.dv, c.ring_k_dtype,
                               c.ring_d_dtype)
              : fold_layout_for(c);
  return p;
}

// Commit of uniform (cu == null, T tokens per row) or ragged windows (at most
// T tokens per row).
rssm_status commit(rssm_handle* h, const int32_t* slot, const uint8_t* force,
                   const int32_t* accept_len, const int32_t* cu, int32_t B, int32_t T,
                   void* stream) {
  if (h == nullptr) return RSSM_ERR_INVALID_ARG;
  const rssm_config& c = h->cfg;
  if (B < 0 || B > kMaxGrid || T < 1 || T > c.max_T) return RSSM_ERR_INVALID_ARG;
  if (B == 0) return RSSM_OK;
  if (!slot || !accept_len) return RSSM_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c.commit_mode == RSSM_COMMIT_FOLD_EVERY) {
    FoldParams p = fold_params(h, slot, force, accept_len, B, T, FOLD_COMMIT);
    p.cu = cu;
    const cudaError_t e = fold_launch(c.algo, state_dt(c), p, c.n_layers, st);
    if (e != cudaSuccess) return RSSM_ERR_CUDA;
    return from_cuda(cursor_launch(h->buf.cursor, slot, force, accept_len, cu, B, T, c.L,
                                   c.n_slots, CURSOR_COMMIT_FOLD, h->buf.err_word, st));
  }
  return from_cuda(cursor_launch(h->buf.cursor, slot, force, accept_len, cu, B, T, c.L,
                                 c.n_slots, CURSOR_COMMIT_LAZY, h->buf.err_word, st));
}

}  // namespace

extern "C" {

rssm_status rssm_required_bytes(const rssm_config* cfg, rssm_sizes* out) {
  if (out == nullptr) return RSSM_ERR_INVALID_ARG;
  const rssm_status st = check_config(cfg);
  if (st != RSSM_OK) return st;
  sizes_of(*cfg, out);
  return RSSM_OK;
}

rssm_status rssm_alloc(const rssm_config* cfg, const rssm_buffers* buf, rssm_handle** out) {
  if (out == nullptr || buf == nullptr) return RSSM_ERR_INVALID_ARG;
  *out = nullptr;
  const rssm_status st = check_config(cfg);
  if (st != RSSM_OK) return st;
  const rssm_buffers& b = *buf;
  if (!b.state || !b.ring_k || !b.ring_d || !b.ring_g || !b.ring_v || !b.ring_beta ||
      !b.cursor || !b.err_word)
    return RSSM_ERR_INVALID_ARG;
  if (!aligned16(b.state) || !aligned16(b.ring_k) || !aligned16(b.ring_d) ||
      !aligned16(b.ring_v) || !aligned16(b.ring_g) || !aligned4(b.ring_beta) ||
      !aligned4(b.cursor) || !aligned4(b.err_word))
    return RSSM_ERR_INVALID_ARG;

  int dev = 0, max_smem = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RSSM_ERR_CUDA;
  if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
      cudaSuccess)
    return RSSM_ERR_CUDA;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return RSSM_ERR_CUDA;
  // The widest window this store allows must fit in shared memory.
  const ReplaySmem worst = layout_for(*cfg, cfg->max_T);
  const FoldSmem fworst = fold_layout_for(*cfg);
  if ((int)worst.total > max_smem || (int)fworst.total > max_smem) return RSSM_ERR_UNSUPPORTED;
  if (replay_prepare(*cfg, max_smem) != cudaSuccess) return RSSM_ERR_CUDA;
  if (fold_prepare(cfg->algo, state_dt(*cfg), max_smem) != cudaSuccess) return RSSM_ERR_CUDA;
  // the comparison kernel needs the whole tile in shared memory; configurations
  // where it does not fit still allocate, and rssm_native_decode reports
  // RSSM_ERR_UNSUPPORTED for them
  if ((int)native_layout_for(*cfg).total <= max_smem &&
      native_prepare(cfg->algo, state_dt(*cfg), max_smem) != cudaSuccess)
    return RSSM_ERR_CUDA;
  if ((int)prefill_layout(cfg->algo, cfg->dk, cfg->dv).total <= max_smem &&
      prefill_prepare(cfg->algo, state_dt(*cfg), max_smem) != cudaSuccess)
    return RSSM_ERR_CUDA;
  const bool pipe_cfg = pipe_config(*cfg);
  if (pipe_cfg && pipe_prepare(state_dt(*cfg), max_smem) != cudaSuccess) return RSSM_ERR_CUDA;

  rssm_handle* h = new (std::nothrow) rssm_handle;
  if (h == nullptr) return RSSM_ERR_INVALID_ARG;
  h->cfg = *cfg;
  h->buf = b;
  h->G = cfg->HV / cfg->HK;
  h->max_smem = max_smem;
  h->num_sms = num_sms;
  const size_t slots = (size_t)cfg->n_slots;
  h->layer_state = slots * cfg->HV * cfg->dk * cfg->dv;
  h->layer_k = slots * cfg->HV * cfg->L * cfg->dk;
  h->layer_d = slots * cfg->HV * cfg->L * cfg->dv;
  h->layer_g = slots * cfg->HV * cfg->L * n_gate(*cfg);
  h->layer_v = slots * cfg->HV * cfg->L * cfg->dv;
  h->layer_beta = slots * cfg->HV * cfg->L;
  h->hook = WaitHook{WH_OFF};
  h->pipe_cfg = pipe_cfg;
  h->plan = RSSM_PLAN_AUTO;
  *out = h;
  return RSSM_OK;
}

void rssm_free(rssm_handle* h) { delete h; }

rssm_status rssm_decode(rssm_handle* h, int32_t layer, const void* q, const void* k,
                        const void* v, const float* beta, const float* g, const int32_t* slot,
                        const uint8_t* force, int32_t B, void* o, uint8_t* fold_out,
                        int32_t advance_cursor, void* stream) {
  const rssm_status st = window(h, layer, q, k, v, beta, g, slot, force, B, 1, o, fold_out,
                                stream);
  if (st != RSSM_OK || B == 0 || !advance_cursor) return st;
  const rssm_config& c = h->cfg;
  return from_cuda(cursor_launch(h->buf.cursor, slot, force, nullptr, nullptr, B, 1, c.L, c.n_slots,
                                 CURSOR_DECODE, h->buf.err_word,
                                 static_cast<cudaStream_t>(stream)));
}

rssm_status rssm_verify(rssm_handle* h, int32_t layer, const void* q, const void* k,
                        const void* v, const float* beta, const float* g, const int32_t* slot,
                        const uint8_t* force, int32_t B, int32_t T, void* o, uint8_t* fold_out,
                        void* stream) {
  return window(h, layer, q, k, v, beta, g, slot, force, B, T, o, fold_out, stream);
}

rssm_status rssm_verify_ragged(rssm_handle* h, int32_t layer, const void* q, const void* k,
                               const void* v, const float* beta, const float* g,
                               const int32_t* cu_seqlens, const int32_t* slot,
                               const uint8_t* force, int32_t B, int32_t max_T, void* o,
                               uint8_t* fold_out, void* stream) {
  if (B > 0 && (cu_seqlens == nullptr || !aligned4(cu_seqlens))) return RSSM_ERR_INVALID_ARG;
  return window(h, layer, q, k, v, beta, g, slot, force, B, max_T, o, fold_out, stream,
                cu_seqlens);
}

rssm_status rssm_prefill(rssm_handle* h, int32_t layer, const void* q, const void* k,
                         const void* v, const float* beta, const float* g,
                         const int32_t* cu_seqlens, const int32_t* slot, int32_t B, void* o,
                         int32_t reset_cursor, void* stream) {
  // the window rules of a one-token window cover the pointers and alignment
  ReplayParams w;
  const rssm_status st = window_params(h, layer, q, k, v, beta, g, slot, nullptr, B, 1, o,
                                       nullptr, &w);
  if (st != RSSM_OK || B == 0) return st;
  if (cu_seqlens == nullptr || !aligned4(cu_seqlens)) return RSSM_ERR_INVALID_ARG;
  const rssm_config& c = h->cfg;
  PrefillParams p{};
  p.state = w.state;
  p.ring_k = w.ring_k;
  p.ring_d = w.ring_d;
  p.ring_g = w.ring_g;
  p.cursor = w.cursor;
  p.err = w.err;
  p.q = q;
  p.k = k;
  p.v = v;
  p.beta = beta;
  p.g = g;
  p.cu = cu_seqlens;
  p.slot = slot;
  p.o = o;
  p.B = B;
  p.L = c.L;
  p.n_slots = c.n_slots;
  p.HK = c.HK;
  p.HV = c.HV;
  p.G = h->G;
  p.dk = c.dk;
  p.dv = c.dv;
  p.CB = prefill_cb(c.dv);
  p.in_dt = w.in_dt;
  p.rk_dt = w.rk_dt;
  p.rd_dt = w.rd_dt;
  p.scale = c.scale;
  p.sm = prefill_layout(c.algo, c.dk, c.dv);
  if ((int)p.sm.total > h->max_smem) return RSSM_ERR_UNSUPPORTED;
  if ((long long)c.HV * (c.dv / p.CB) > kMaxGrid) return RSSM_ERR_UNSUPPORTED;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = prefill_launch(c.algo, state_dt(c), p, s);
  if (e != cudaSuccess || !reset_cursor) return from_cuda(e);
  return from_cuda(cursor_launch(h->buf.cursor, slot, nullptr, nullptr, cu_seqlens, B, 1, c.L,
                                 c.n_slots, CURSOR_PREFILL, h->buf.err_word, s));
}

static rssm_status conv_params(const void* x, void* window, void* draft, const int32_t* slot,
                               int32_t B, int32_t T, int32_t D, int32_t K, int32_t n_slots,
                               int32_t dtype, ConvParams* out) {
  if (B < 0 || B > kMaxGrid || T < 1 || D < 1 || n_slots < 1) return RSSM_ERR_INVALID_ARG;
  if (K < 2 || K > kConvMaxK) return RSSM_ERR_UNSUPPORTED;
  if (dtype != RSSM_F32 && dtype != RSSM_BF16) return RSSM_ERR_UNSUPPORTED;
  if (!window || !slot) return RSSM_ERR_INVALID_ARG;
  if (!aligned4(slot)) return RSSM_ERR_INVALID_ARG;
  // 16-byte vectors of channels: D a multiple of 16 bytes, buffers 16-byte aligned
  if ((D * (dtype == RSSM_F32 ? 4 : 2)) % 16 != 0) return RSSM_ERR_UNSUPPORTED;
  if (!aligned16(window) || (x && !aligned16(x)) || (draft && !aligned16(draft)))
    return RSSM_ERR_INVALID_ARG;
  ConvParams& p = *out;
  p = ConvParams{};
  p.window = window;
  p.slot = slot;
  p.B = B;
  p.T = T;
  p.D = D;
  p.K = K;
  p.n_slots = n_slots;
  p.dt = dtype == RSSM_F32 ? DT_F32 : DT_BF16;
  return RSSM_OK;
}

rssm_status rssm_conv_window(const void* x, const float* w, const float* bias, void* window,
                             void* draft, const int32_t* slot, int32_t B, int32_t T, int32_t D,
                             int32_t K, int32_t n_slots, int32_t dtype, int32_t act,
                             int32_t commit_now, void* y, uint32_t* err_word, void* stream) {
  ConvParams p;
  const rssm_status st = conv_params(x, window, draft, slot, B, T, D, K, n_slots, dtype, &p);
  if (st != RSSM_OK) return st;
  if (act != RSSM_CONV_ACT_NONE && act != RSSM_CONV_ACT_SILU) return RSSM_ERR_INVALID_ARG;
  if (B == 0) return RSSM_OK;
  if (!x || !w || !y || (!commit_now && !draft)) return RSSM_ERR_INVALID_ARG;
  if (!aligned16(y)) return RSSM_ERR_INVALID_ARG;
  p.x = x;
  p.w = w;
  p.bias = bias;
  p.draft = draft;
  p.y = y;
  p.err = err_word;
  p.act = act;
  p.commit_now = commit_now ? 1 : 0;
  return from_cuda(conv_launch(p, false, static_cast<cudaStream_t>(stream)));
}

rssm_status rssm_conv_commit(void* window, const void* draft, const int32_t* slot,
                             const int32_t* accept_len, int32_t B, int32_t T, int32_t D,
                             int32_t K, int32_t n_slots, int32_t dtype, uint32_t* err_word,
                             void* stream) {
  ConvParams p;
  const rssm_status st = conv_params(nullptr, window, nullptr, slot, B, T, D, K, n_slots, dtype,
                                     &p);
  if (st != RSSM_OK) return st;
  if (B == 0) return RSSM_OK;
  if (!draft || !accept_len || !aligned4(accept_len)) return RSSM_ERR_INVALID_ARG;
  p.draft = const_cast<void*>(draft);
  p.accept = accept_len;
  p.err = err_word;
  return from_cuda(conv_launch(p, true, static_cast<cudaStream_t>(stream)));
}

rssm_status rssm_native_decode(rssm_handle* h, int32_t layer, const void* q, const void* k,
                               const void* v, const float* beta, const float* g,
                               const int32_t* slot, int32_t B, void* o, void* stream) {
  ReplayParams p;
  const rssm_status st = window_params(h, layer, q, k, v, beta, g, slot, nullptr, B, 1, o,
                                       nullptr, &p);
  if (st != RSSM_OK || B == 0) return st;
  const NativeSmem sm = native_layout_for(h->cfg);
  if ((int)sm.total > h->max_smem) return RSSM_ERR_UNSUPPORTED;
  return from_cuda(native_launch(h->cfg.algo, state_dt(h->cfg), p, sm,
                                 static_cast<cudaStream_t>(stream)));
}

rssm_status rssm_commit(rssm_handle* h, const int32_t* slot, const uint8_t* force,
                        const int32_t* accept_len, int32_t B, int32_t T, void* stream) {
  return commit(h, slot, force, accept_len, nullptr, B, T, stream);
}

rssm_status rssm_commit_ragged(rssm_handle* h, const int32_t* slot, const uint8_t* force,
                               const int32_t* accept_len, const int32_t* cu_seqlens, int32_t B,
                               int32_t max_T, void* stream) {
  if (B > 0 && (cu_seqlens == nullptr || !aligned4(cu_seqlens))) return RSSM_ERR_INVALID_ARG;
  return commit(h, slot, force, accept_len, cu_seqlens, B, max_T, stream);
}

rssm_status rssm_fold(rssm_handle* h, const int32_t* slot, int32_t B, void* stream) {
  if (h == nullptr) return RSSM_ERR_INVALID_ARG;
  if (B < 0 || B > kMaxGrid) return RSSM_ERR_INVALID_ARG;
  if (B == 0) return RSSM_OK;
  if (!slot) return RSSM_ERR_INVALID_ARG;
  const rssm_config& c = h->cfg;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const FoldParams p = fold_params(h, slot, nullptr, nullptr, B, 1, FOLD_ALL);
  const cudaError_t e = fold_launch(c.algo, state_dt(c), p, c.n_layers, st);
  if (e != cudaSuccess) return RSSM_ERR_CUDA;
  return from_cuda(cursor_launch(h->buf.cursor, slot, nullptr, nullptr, nullptr, B, 1, c.L, c.n_slots,
                                 CURSOR_ZERO, h->buf.err_word, st));
}

rssm_status rssm_reset_slots(rssm_handle* h, const int32_t* slot, int32_t B, void* stream) {
  if (h == nullptr) return RSSM_ERR_INVALID_ARG;
  if (B < 0 || B > kMaxGrid) return RSSM_ERR_INVALID_ARG;
  if (B == 0) return RSSM_OK;
  if (!slot) return RSSM_ERR_INVALID_ARG;
  const rssm_config& c = h->cfg;
  return from_cuda(cursor_launch(h->buf.cursor, slot, nullptr, nullptr, nullptr, B, 1, c.L, c.n_slots,
                                 CURSOR_ZERO, h->buf.err_word,
                                 static_cast<cudaStream_t>(stream)));
}

rssm_status rssm_get_device_error(rssm_handle* h, uint32_t* out, int32_t clear, void* stream) {
  if (h == nullptr || out == nullptr) return RSSM_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return RSSM_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, h->buf.err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return RSSM_ERR_CUDA;
  if (clear) {
    if (cudaMemsetAsync(h->buf.err_word, 0, sizeof(uint32_t), st) != cudaSuccess)
      return RSSM_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return RSSM_ERR_CUDA;
  }
  *out = word;
  return word == 0 ? RSSM_OK : RSSM_ERR_DEVICE;
}

rssm_status rssm_set_plan(rssm_handle* h, int32_t plan) {
  if (h == nullptr) return RSSM_ERR_INVALID_ARG;
  if (plan != RSSM_PLAN_AUTO && plan != RSSM_PLAN_ROWS && plan != RSSM_PLAN_PIPE &&
      plan != RSSM_PLAN_TC)
    return RSSM_ERR_INVALID_ARG;
  if (plan == RSSM_PLAN_PIPE && !h->pipe_cfg) return RSSM_ERR_UNSUPPORTED;
  if (plan == RSSM_PLAN_TC && !tc_config(h->cfg)) return RSSM_ERR_UNSUPPORTED;
  h->plan = plan;
  return RSSM_OK;
}

rssm_status rssm_debug_withhold(rssm_handle* h, int32_t barrier) {
  if (h == nullptr) return RSSM_ERR_INVALID_ARG;
  if (barrier < WH_OFF || barrier >= WH_CHUNK0 + 256) return RSSM_ERR_INVALID_ARG;
  h->hook = WaitHook{barrier};
  return RSSM_OK;
}

const char* rssm_status_string(rssm_status s) {
  switch (s) {
    case RSSM_OK: return "ok";
    case RSSM_ERR_INVALID_ARG: return "invalid argument";
    case RSSM_ERR_UNSUPPORTED: return "unsupported configuration";
    case RSSM_ERR_CUDA: return "CUDA runtime error";
    case RSSM_ERR_DEVICE: return "device error word set";
  }
  return "unknown status";
}

int32_t rssm_version(void) { return 1; }

}  // extern "C"
