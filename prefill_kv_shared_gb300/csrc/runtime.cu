// Runtime behind the C ABI (include/prefill.h): context creation (weight
// repack and upload, KV cache and activation buffers), the ubatch schedule
// with the pruning decision, and the KV image save/restore.
//
// The pruning follows the Gemma 4 prefill change (devotd.net llama.cpp Gemma 4
// prefill news, section 1 and its listing): when 0 < n_layer_kv_from_start <
// n_layer, one sequence, no embeddings output, the rows no output needs are
// dropped before the first KV-shared layer; an intermediate ubatch ends there
// and the final ubatch carries its last row only.  The KV image follows the
// PicoLM KV cache article ("file" and "rules" paragraphs).
#include "../../include/prefill.h"
#include "common.cuh"
#include "kernels.h"

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <string>
#include <vector>

using namespace pf;

namespace {

struct DevBuf {
  void* p = nullptr;
  size_t bytes = 0;
};

struct LayerW {
  WeightMat qkv;  // writing layers: [Wq; Wk; Wv]; KV-shared layers: Wq
  WeightMat o, gu, down, pg, pp;
  float* attn_norm = nullptr;
  float* ffn_norm = nullptr;
};

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// The epilogue of a projection moved from its launch's row 0 to row r: the
// outputs, the per-layer-embedding multipliers and the Q rows advance by r
// rows, and the position (RoPE angle, K/V cache row) by r.
EpiParams shift_rows(const EpiParams& e, int r) {
  EpiParams s = e;
  if (s.out_f32) s.out_f32 += static_cast<size_t>(r) * s.ld_f32;
  if (s.out_bf16) s.out_bf16 += static_cast<size_t>(r) * s.ld_bf16;
  if (s.ple) s.ple += static_cast<size_t>(r) * s.ple_stride;
  if (s.q_out) s.q_out += static_cast<size_t>(r) * s.q_dim;
  if (s.row_pos) s.row_pos += r;
  if (s.row_slot) s.row_slot += r;
  s.pos0 += r;
  return s;
}

}  // namespace

struct prefill_ctx {
  prefill_model_desc d{};
  std::vector<int32_t> kv_src;
  std::vector<int32_t> layer_inp;  // [n_layer + 1] requests of hidden-state outputs (empty: none)
  std::vector<float*> layer_out;   // [n_layer + 1] their device buffers
  float* embd_out = nullptr;       // the embeddings output's buffer
  int L = 0, S = 0, L_w = 0, D = 0, Hq = 0, Hkv = 0, hd = 0, q = 0, kv = 0, F = 0, V = 0, P = 0;
  int rows_alloc = 0;
  cudaStream_t stream = nullptr;
  int device = 0;
  std::vector<void*> allocs;

  std::vector<LayerW> layers;
  WeightMat head;
  const void* tok_table = nullptr;  // gather copy (original Q4_0 rows or fp32)
  const void* ple_table = nullptr;
  float* out_norm = nullptr;

  int32_t* tok = nullptr;
  float* x = nullptr;
  float* xr = nullptr;
  __nv_bfloat16 *y = nullptr, *att = nullptr, *h = nullptr, *xb = nullptr, *pg = nullptr, *ple = nullptr;
  __half* q16 = nullptr;
  float* partials = nullptr;
  float* row_partials = nullptr;  // range states of the single-row attention
  __half* cache = nullptr;  // [2][L_w][max_ctx][kv]
  float2* rope = nullptr;
  int* err = nullptr;
  ActMat a_y, a_att, a_h, a_xb, a_pg;

  std::vector<int64_t> seq_pos;  // positions in the cache, per sequence
  int* rowinfo = nullptr;        // several sequences: row positions, cache rows, output rows and positions
  std::vector<int> rowinfo_host;
  __nv_bfloat16* ple_g = nullptr;  // per-layer-embedding rows of the gathered output rows
  int prune_enable = 1;  // PF_PRUNE_ON / PF_PRUNE_OFF / PF_PRUNE_OFF_PLAIN
  // a recorded ubatch (prefill_graph_capture) and the positions it covers
  cudaGraphExec_t graph = nullptr;
  int64_t graph_pos0 = -1;
  int graph_T = 0;
  std::string last_error;

  // launch accounting
  prefill_stats stats{};
  bool timing = false;
  struct Timed {
    int kc;
    cudaEvent_t e0, e1;
  };
  std::vector<Timed> timed;
  std::vector<cudaEvent_t> event_pool;

  prefill_ctx() = default;
  prefill_ctx(const prefill_ctx&) = delete;
  prefill_ctx& operator=(const prefill_ctx&) = delete;
  // Frees the events and device buffers the context holds.  Also runs when
  // prefill_create gives up half way, so a failed create leaves no device
  // memory behind.
  ~prefill_ctx() {
    if (graph) cudaGraphExecDestroy(graph);
    for (auto& t : timed) {
      cudaEventDestroy(t.e0);
      cudaEventDestroy(t.e1);
    }
    for (cudaEvent_t e : event_pool) cudaEventDestroy(e);
    for (void* p : allocs) cudaFree(p);
  }
};

namespace {

thread_local std::string g_last_error;

// A named range for profilers (ncu --nvtx --nvtx-include, nsys): one per
// ubatch, one per layer, one for the head and for each KV image copy.
// Without a tool attached a push/pop is a cheap no-op.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

int fail(prefill_ctx* c, int code, const std::string& msg) {
  if (c)
    c->last_error = msg;
  else
    g_last_error = msg;
  return code;
}

int cuda_fail(prefill_ctx* c, cudaError_t e, const char* what) {
  return fail(c, PF_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define PF_CUDA(ctx, call)                                    \
  do {                                                        \
    cudaError_t e_ = (call);                                  \
    if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #call); \
  } while (0)

template <class T>
int dev_alloc(prefill_ctx* c, T** out, size_t bytes, bool zero = true) {
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, bytes ? bytes : 16);
  if (e != cudaSuccess)  // out of memory is PF_E_NOMEM; no device or driver is a CUDA failure
    return fail(c, e == cudaErrorMemoryAllocation ? PF_E_NOMEM : PF_E_CUDA,
                std::string("cudaMalloc: ") + cudaGetErrorString(e));
  c->allocs.push_back(p);
  if (zero) {
    e = cudaMemset(p, 0, bytes ? bytes : 16);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemset");
  }
  *out = static_cast<T*>(p);
  return PF_OK;
}

template <class T>
int upload(prefill_ctx* c, T** out, const void* host, size_t bytes) {
  int rc = dev_alloc(c, out, bytes, false);
  if (rc) return rc;
  PF_CUDA(c, cudaMemcpy(*out, host, bytes, cudaMemcpyHostToDevice));
  return PF_OK;
}

size_t row_bytes(int wtype, int K) { return wtype == PF_W_Q4_0 ? static_cast<size_t>(K / 32) * 18 : static_cast<size_t>(K) * 4; }

// rows: sources of the stored rows in tile order (null = zero row)
// split_as: 0 = choose the k-split for this shape; otherwise use that split
int build_weight(prefill_ctx* c, WeightMat& w, const std::vector<const void*>& rows, int K, int BN, int split_as = 0) {
  w.K = K;
  w.BN = BN;
  w.N_rows = static_cast<int>(rows.size());
  if (w.N_rows % BN != 0 || K % 64 != 0) return fail(c, PF_E_ARG, "weight shape not tileable");
  const int kind = c->d.wtype == PF_W_Q4_0 ? W_Q4 : W_BF16;
  w.split = split_as > 0 ? split_as : choose_split(kind, w.N_rows, BN, K, c->d.ubatch_max);
  w.pair = choose_pair(kind, w.N_rows, BN, K, c->d.ubatch_max, w.split);
  std::string err;
  if (c->d.wtype == PF_W_Q4_0) {
    w.kind = W_Q4;
    std::vector<const uint8_t*> r(rows.size());
    for (size_t i = 0; i < rows.size(); ++i) r[i] = static_cast<const uint8_t*>(rows[i]);
    std::vector<uint8_t> t = repack_q4_tiles(r, K, BN);
    w.bytes = t.size();
    int rc = upload(c, &w.dev, t.data(), t.size());
    if (rc) return rc;
  } else {
    w.kind = W_BF16;
    std::vector<const float*> r(rows.size());
    for (size_t i = 0; i < rows.size(); ++i) r[i] = static_cast<const float*>(rows[i]);
    std::vector<uint16_t> t = repack_bf16_rows(r, K);
    w.bytes = t.size() * 2;
    int rc = upload(c, &w.dev, t.data(), w.bytes);
    if (rc) return rc;
  }
  if (!make_weight_map(w, &err)) return fail(c, PF_E_CUDA, err);
  return PF_OK;
}

// plain matrix [N][K], rows in order, padded to BN
std::vector<const void*> plain_rows(const void* m, int N, int K, int wtype, int BN) {
  std::vector<const void*> r(round_up(N, BN), nullptr);
  const uint8_t* b = static_cast<const uint8_t*>(m);
  for (int n = 0; n < N; ++n) r[n] = b + n * row_bytes(wtype, K);
  return r;
}

int check_desc(const prefill_model_desc* d, std::string* why) {
  auto bad = [&](const char* m) {
    *why = m;
    return PF_E_ARG;
  };
  if (!d) return bad("null description");
  if (d->n_layer < 1) return bad("n_layer < 1");
  if (d->n_layer_kv_from_start < 0 || d->n_layer_kv_from_start > d->n_layer)
    return bad("n_layer_kv_from_start outside [0, n_layer]");
  if (d->n_layer_kv_from_start == 0) return bad("at least one layer must write the KV cache");
  if (d->head_dim != 64 && d->head_dim != 256) return bad("head_dim must be 64 or 256");
  if (d->n_head < 1 || d->n_head_kv < 1 || d->n_head % d->n_head_kv) return bad("n_head must be a multiple of n_head_kv");
  const int G = d->n_head / d->n_head_kv;
  if (G > 16 || 16 % G) return bad("n_head / n_head_kv must divide 16");
  if (d->d_model < 64 || d->d_model % 64) return bad("d_model must be a multiple of 64");
  if (d->ffn_dim < 64 || d->ffn_dim % 64) return bad("ffn_dim must be a multiple of 64");
  if (d->ple_dim < 0 || d->ple_dim % 64) return bad("ple_dim must be 0 or a multiple of 64");
  if (d->vocab < 1) return bad("vocab < 1");
  if (d->ffn_kind != PF_FFN_GEGLU && d->ffn_kind != PF_FFN_SWIGLU) return bad("ffn_kind");
  if (d->wtype != PF_W_F32 && d->wtype != PF_W_Q4_0) return bad("wtype");
  if (d->max_ctx < 1 || d->ubatch_max < 1) return bad("max_ctx and ubatch_max must be >= 1");
  // the gathered output rows (one per finishing sequence) share the
  // 128-row buffer of the pruned rows
  if (d->n_seq_max < 1 || d->n_seq_max > 128) return bad("n_seq_max outside [1, 128]");
  // Sizes whose products the kernels index with 32-bit integers: a row of
  // any activation, a weight matrix, and one layer's cache stay below 2^31
  // elements (far above any model this library targets).
  constexpr int64_t kMaxElems = int64_t(1) << 31;
  if (d->n_layer > 4096 || d->n_head > 1024 || d->ubatch_max > (1 << 20) || d->max_ctx > (1 << 26))
    return bad("n_layer, n_head, ubatch_max or max_ctx too large");
  {
    const int64_t rows = (int64_t(d->ubatch_max) + 127) / 128 * 128;
    const int64_t kv = int64_t(d->n_head_kv) * d->head_dim, q = int64_t(d->n_head) * d->head_dim;
    const int64_t width = std::max({int64_t(d->d_model), int64_t(d->ffn_dim), q, 2 * kv,
                                    int64_t(d->n_layer) * d->ple_dim});
    if (rows * width >= kMaxElems) return bad("ubatch_max times the widest activation reaches 2^31 elements");
    if (int64_t(d->vocab) * d->d_model >= kMaxElems || 2 * int64_t(d->ffn_dim) * d->d_model >= kMaxElems ||
        (q + 2 * kv) * d->d_model >= kMaxElems || int64_t(d->vocab) * d->n_layer * d->ple_dim >= kMaxElems)
      return bad("a weight matrix reaches 2^31 elements");
    if (int64_t(d->max_ctx) * kv * (d->n_seq_max > 0 ? d->n_seq_max : 1) >= kMaxElems)
      return bad("n_seq_max times max_ctx times the KV width reaches 2^31 elements");
  }
  if (!d->kv_src) return bad("kv_src is null");
  for (int il = 0; il < d->n_layer; ++il) {
    const int s = d->kv_src[il];
    if (il < d->n_layer_kv_from_start) {
      if (s != -1) return bad("kv_src of a writing layer must be -1");
    } else if (s < 0 || s >= d->n_layer_kv_from_start) {
      return bad("kv_src of a KV-shared layer must name a writing layer");
    }
  }
  return PF_OK;
}

// The pruning condition of the Gemma 4 prefill change (devotd.net news,
// section 1 listing).  The NextN crop is always allowed here (no
// multi-token-prediction head); a per-layer input embedding requested for
// any layer from the first KV-shared one up to the final state (index
// n_layer) needs every row there.
bool predicate(const prefill_model_desc& d, int enable) {
  if (!(enable && d.n_layer_kv_from_start > 0 && d.n_layer_kv_from_start < d.n_layer && !d.embeddings &&
        d.n_seq_max == 1))
    return false;
  if (d.embd_layer_inp)
    for (int il = d.n_layer_kv_from_start; il <= d.n_layer; ++il)
      if (d.embd_layer_inp[il]) return false;
  return true;
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int check_device_error(prefill_ctx* c) {
  int e = 0;
  PF_CUDA(c, cudaMemcpy(&e, c->err, sizeof(int), cudaMemcpyDeviceToHost));
  if (e == 0) return PF_OK;
  PF_CUDA(c, cudaMemset(c->err, 0, sizeof(int)));
  if (e == PF_DEV_BAD_TOKEN) return fail(c, PF_E_DEVICE_TOKEN, "a token id was outside [0, vocab)");
  return fail(c, PF_E_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (code " + std::to_string(e) + ")");
}

cudaEvent_t take_event(prefill_ctx* c) {
  if (!c->event_pool.empty()) {
    cudaEvent_t e = c->event_pool.back();
    c->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Launch one step's kernel(s) through `fn`, counting them (n kernels) and
// their algorithmic work; with timing on, bracket them with events.
template <class F>
cudaError_t counted(prefill_ctx* c, int kc, int n, double flops, double bytes, F&& fn) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (c->timing) {
    e0 = take_event(c);
    e1 = take_event(c);
    cudaEventRecord(e0, c->stream);
  }
  const cudaError_t e = fn();
  if (c->timing) {
    cudaEventRecord(e1, c->stream);
    c->timed.push_back({kc, e0, e1});
  }
  if (e == cudaSuccess) {
    c->stats.launches[kc] += n;
    c->stats.flops[kc] += flops;
    c->stats.bytes[kc] += bytes;
  }
  return e;
}

// launch class of a projection: at most 16 rows stream the weights once and
// are bound by them, more rows are bound by the tensor cores
int gemm_class(int M) { return M <= 16 ? PF_KC_GEMM_ROW : PF_KC_GEMM; }

double gemm_wbytes(const prefill_ctx* c, double n, double k) {
  return c->d.wtype == PF_W_Q4_0 ? n * k * 18.0 / 32.0 : n * k * 4.0;
}

}  // namespace

// ---------------------------------------------------------------------------
// create / destroy

extern "C" int prefill_create(const prefill_model_desc* desc, const prefill_weights* w, void* stream,
                              prefill_ctx** out) {
  if (!out) return fail(nullptr, PF_E_ARG, "out is null");
  *out = nullptr;
  std::string why;
  if (check_desc(desc, &why) != PF_OK) return fail(nullptr, PF_E_ARG, why);
  if (!w || !w->tok_embd || !w->out_norm || !w->layers) return fail(nullptr, PF_E_ARG, "missing weights");
  if (desc->ple_dim > 0 && !w->ple_embd) return fail(nullptr, PF_E_ARG, "missing ple_embd");

  std::unique_ptr<prefill_ctx> c(new prefill_ctx());
  prefill_ctx* C = c.get();
  C->d = *desc;
  C->kv_src.assign(desc->kv_src, desc->kv_src + desc->n_layer);
  C->d.kv_src = C->kv_src.data();
  if (desc->embd_layer_inp) {
    C->layer_inp.assign(desc->embd_layer_inp, desc->embd_layer_inp + desc->n_layer + 1);
    C->d.embd_layer_inp = C->layer_inp.data();
    C->layer_out.assign(desc->n_layer + 1, nullptr);
  }
  C->L = desc->n_layer;
  C->S = desc->n_layer_kv_from_start;
  C->L_w = C->S;
  C->D = desc->d_model;
  C->Hq = desc->n_head;
  C->Hkv = desc->n_head_kv;
  C->hd = desc->head_dim;
  C->q = C->Hq * C->hd;
  C->kv = C->Hkv * C->hd;
  C->F = desc->ffn_dim;
  C->V = desc->vocab;
  C->P = desc->ple_dim;
  C->stream = static_cast<cudaStream_t>(stream);
  C->prune_enable = desc->prune_shared_enable ? 1 : 0;
  C->rows_alloc = round_up(desc->ubatch_max, 128);
  cudaGetDevice(&C->device);
  const int wt = desc->wtype;
  int rc;

  // layers
  C->layers.resize(C->L);
  for (int il = 0; il < C->L; ++il) {
    const prefill_layer_weights& lw = w->layers[il];
    LayerW& L = C->layers[il];
    const bool writes = il < C->S;
    if (!lw.attn_norm || !lw.wq || !lw.wo || !lw.ffn_norm || !lw.w_gate || !lw.w_up || !lw.w_down)
      return fail(nullptr, PF_E_ARG, "missing layer weight");
    if (writes && (!lw.wk || !lw.wv)) return fail(nullptr, PF_E_ARG, "writing layer without wk/wv");
    if (C->P > 0 && (!lw.ple_gate || !lw.ple_proj)) return fail(nullptr, PF_E_ARG, "missing ple_gate/ple_proj");
    // QKV (or Q): one tile holds whole heads so RoPE pairs stay in the tile
    {
      std::vector<const void*> rows = qkv_tile_rows(lw.wq, writes ? lw.wk : nullptr, writes ? lw.wv : nullptr, C->Hq,
                                                    C->Hkv, C->hd, row_bytes(wt, C->D), QKV_BN);
      if ((rc = build_weight(C, L.qkv, rows, C->D, QKV_BN))) return fail(nullptr, rc, C->last_error);
    }
    if ((rc = build_weight(C, L.o, plain_rows(lw.wo, C->D, C->q, wt, 128), C->q, 128)))
      return fail(nullptr, rc, C->last_error);
    {
      // gate/up interleaved per tile: BN/2 gate rows, then the same BN/2 up rows
      auto gu_rows = [&](int bn) {
        const int half = bn / 2;
        const size_t rb = row_bytes(wt, C->D);
        std::vector<const void*> rows;
        for (int t = 0; t < C->F / half; ++t) {
          for (int i = 0; i < half; ++i) rows.push_back(static_cast<const uint8_t*>(lw.w_gate) + (t * half + i) * rb);
          for (int i = 0; i < half; ++i) rows.push_back(static_cast<const uint8_t*>(lw.w_up) + (t * half + i) * rb);
        }
        return rows;
      };
      // Q4_0: 192-row tiles (96 gate + 96 up rows) when they give the
      // ubatch's gate/up launch more CTAs than 256-row tiles and still fit
      // one wave on the SMs (two 128-row M tiles per CTA); else 256 or 128
      int bn = C->F % 128 == 0 ? 256 : 128;
      if (wt == PF_W_Q4_0 && C->F % 96 == 0 && C->d.ubatch_max > 128) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, C->device);
        const int pairs = (C->d.ubatch_max + 255) / 256;
        const int u192 = (2 * C->F / 192) * pairs, u256 = C->F % 128 == 0 ? (2 * C->F / 256) * pairs : 0;
        if (u192 > u256 && u192 <= sms) bn = 192;
      }
      if ((rc = build_weight(C, L.gu, gu_rows(bn), C->D, bn))) return fail(nullptr, rc, C->last_error);
    }
    if ((rc = build_weight(C, L.down, plain_rows(lw.w_down, C->D, C->F, wt, 128), C->F, 128)))
      return fail(nullptr, rc, C->last_error);
    if (C->P > 0) {
      // the PLE gate has few output rows: 64-row tiles give it more CTAs
      const int bn_pg = C->P <= 512 ? 64 : 128;
      if ((rc = build_weight(C, L.pg, plain_rows(lw.ple_gate, C->P, C->D, wt, bn_pg), C->D, bn_pg)))
        return fail(nullptr, rc, C->last_error);
      // the PLE projection (K = P, a few k-blocks) is bound by its epilogue:
      // 64-row tiles halve each CTA's share of it when the launch still fits
      // one wave
      int sms_pp = 0;
      cudaDeviceGetAttribute(&sms_pp, cudaDevAttrMultiProcessorCount, C->device);
      const int bn_pp = (C->D % 64 == 0 && (C->D / 64) * ((C->d.ubatch_max + 127) / 128) <= sms_pp) ? 64 : 128;
      if ((rc = build_weight(C, L.pp, plain_rows(lw.ple_proj, C->D, C->P, wt, bn_pp), C->P, bn_pp)))
        return fail(nullptr, rc, C->last_error);
    }
    if ((rc = upload(C, &L.attn_norm, lw.attn_norm, C->D * 4))) return fail(nullptr, rc, C->last_error);
    if ((rc = upload(C, &L.ffn_norm, lw.ffn_norm, C->D * 4))) return fail(nullptr, rc, C->last_error);
  }
  // head (tied embedding), gather tables, final norm
  if ((rc = build_weight(C, C->head, plain_rows(w->tok_embd, C->V, C->D, wt, 128), C->D, 128)))
    return fail(nullptr, rc, C->last_error);
  {
    void* p = nullptr;
    if ((rc = upload(C, &p, w->tok_embd, static_cast<size_t>(C->V) * row_bytes(wt, C->D))))
      return fail(nullptr, rc, C->last_error);
    C->tok_table = p;
    if (C->P > 0) {
      if ((rc = upload(C, &p, w->ple_embd, static_cast<size_t>(C->V) * row_bytes(wt, C->L * C->P))))
        return fail(nullptr, rc, C->last_error);
      C->ple_table = p;
    }
    if ((rc = upload(C, &C->out_norm, w->out_norm, C->D * 4))) return fail(nullptr, rc, C->last_error);
  }

  // buffers
  const size_t R = C->rows_alloc;
  if ((rc = dev_alloc(C, &C->tok, R * 4)) || (rc = dev_alloc(C, &C->x, R * C->D * 4)) ||
      (rc = dev_alloc(C, &C->xr, 128 * C->D * 4)) || (rc = dev_alloc(C, &C->y, R * C->D * 2)) ||
      (rc = dev_alloc(C, &C->att, R * C->q * 2)) || (rc = dev_alloc(C, &C->h, R * C->F * 2)) ||
      (rc = dev_alloc(C, &C->xb, R * C->D * 2)) || (rc = dev_alloc(C, &C->q16, R * C->q * 2)) ||
      (rc = dev_alloc(C, &C->err, 16)))
    return fail(nullptr, rc, C->last_error);
  if (C->P > 0) {
    if ((rc = dev_alloc(C, &C->pg, R * C->P * 2)) || (rc = dev_alloc(C, &C->ple, R * C->L * C->P * 2)))
      return fail(nullptr, rc, C->last_error);
  }
  if ((rc = dev_alloc(C, &C->partials, attn_partials_floats(R, C->Hq, C->hd, C->d.max_ctx) * 4)))
    return fail(nullptr, rc, C->last_error);
  if ((rc = dev_alloc(C, &C->row_partials,
                      attn_split_partials_floats(C->Hq, C->Hkv, C->hd, static_cast<int>(C->d.max_ctx) - 1) * 4)))
    return fail(nullptr, rc, C->last_error);
  if ((rc = dev_alloc(C, &C->cache,
                      static_cast<size_t>(2) * C->L_w * C->d.n_seq_max * C->d.max_ctx * C->kv * 2)))
    return fail(nullptr, rc, C->last_error);
  C->seq_pos.assign(C->d.n_seq_max, 0);
  if ((rc = dev_alloc(C, &C->rowinfo, static_cast<size_t>(4) * C->rows_alloc * 4)))
    return fail(nullptr, rc, C->last_error);
  if (C->P > 0 && C->d.n_seq_max > 1 &&
      (rc = dev_alloc(C, &C->ple_g, static_cast<size_t>(C->d.n_seq_max) * C->L * C->P * 2)))
    return fail(nullptr, rc, C->last_error);
  {
    // RoPE table: angle pos * base^(-2i/hd) in double, cos/sin rounded to fp32
    const int half = C->hd / 2;
    std::vector<float2> tab(static_cast<size_t>(C->d.max_ctx) * half);
    for (int p = 0; p < C->d.max_ctx; ++p)
      for (int i = 0; i < half; ++i) {
        const double th = static_cast<double>(p) * std::pow(static_cast<double>(C->d.rope_base), -2.0 * i / C->hd);
        tab[static_cast<size_t>(p) * half + i] = make_float2(static_cast<float>(std::cos(th)), static_cast<float>(std::sin(th)));
      }
    if ((rc = upload(C, &C->rope, tab.data(), tab.size() * sizeof(float2)))) return fail(nullptr, rc, C->last_error);
  }
  std::string err;
  auto mk = [&](ActMat& a, const __nv_bfloat16* p, int K) {
    a.dev = p;
    a.rows = C->rows_alloc;
    a.K = K;
    return make_act_map(a, &err);
  };
  if (!mk(C->a_y, C->y, C->D) || !mk(C->a_att, C->att, C->q) || !mk(C->a_h, C->h, C->F) ||
      !mk(C->a_xb, C->xb, C->D) || (C->P > 0 && !mk(C->a_pg, C->pg, C->P)))
    return fail(nullptr, PF_E_CUDA, err);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "create");
  *out = c.release();
  return PF_OK;
}

extern "C" int prefill_set_timing(prefill_ctx* c, int32_t enable) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  c->timing = enable != 0;
  return PF_OK;
}

extern "C" int prefill_get_stats(prefill_ctx* c, prefill_stats* out) {
  if (!c || !out) return fail(c, PF_E_ARG, "null argument");
  if (!c->timed.empty()) {
    PF_CUDA(c, cudaStreamSynchronize(c->stream));
    for (auto& t : c->timed) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, t.e0, t.e1) == cudaSuccess) {
        c->stats.ms[t.kc] += ms;
        c->stats.timed[t.kc] += 1;
      }
      c->event_pool.push_back(t.e0);
      c->event_pool.push_back(t.e1);
    }
    c->timed.clear();
  }
  *out = c->stats;
  return PF_OK;
}

extern "C" int prefill_reset_stats(prefill_ctx* c) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  prefill_stats tmp;
  prefill_get_stats(c, &tmp);
  c->stats = prefill_stats{};
  return PF_OK;
}

extern "C" void prefill_destroy(prefill_ctx* c) {
  if (!c) return;
  cudaStreamSynchronize(c->stream);
  delete c;
}

extern "C" const char* prefill_last_error(const prefill_ctx* c) {
  return c ? c->last_error.c_str() : g_last_error.c_str();
}

// ---------------------------------------------------------------------------
// the ubatch

namespace {

// One run of a ubatch: n consecutive rows of sequence `seq`, continuing it at
// position pos0; `last`: the run ends that sequence's prompt (its last row's
// logits are an output).
struct Run {
  int seq = 0, n = 0, last = 0, row0 = 0;
  int64_t pos0 = 0;
};

// The pruning condition without its single-sequence clause: a KV-shared
// split inside the model and no output that needs every row there.  With
// several sequences in a ubatch, this decides the per-sequence gather (one
// row kept per finishing sequence), the variant of the page's pruning that
// its server setting would need.
bool gather_possible(const prefill_model_desc& d) {
  prefill_model_desc one = d;
  one.n_seq_max = 1;
  return predicate(one, 1);
}

// The ubatch of one or more sequence runs (the runs' positions already
// checked).  `multi`: the call came through prefill_ubatch_seqs; a single
// run of sequence 0 then computes what prefill_ubatch computes, but takes the
// tensor-core projections for its output row (the one-row stream kernel
// serves single-sequence ubatches only).
int run_ubatch(prefill_ctx* c, const int32_t* tokens, int T, std::vector<Run>& runs, bool multi, float* logits) {
  int n_out = 0;
  for (const Run& r : runs) n_out += r.last ? 1 : 0;
  const bool is_last = n_out > 0;
  if (is_last && !logits) return fail(c, PF_E_ARG, "logits is null for a ubatch that ends a prompt");
  // the head kernel writes the logits: they must be device (or managed) memory
  if (is_last && !is_device_ptr(logits)) return fail(c, PF_E_ARG, "logits is not device memory");
  if (c->d.embeddings && !c->embd_out) return fail(c, PF_E_ARG, "the embeddings output has no buffer");
  for (size_t il = 0; il < c->layer_inp.size(); ++il)
    if (c->layer_inp[il] && !c->layer_out[il])
      return fail(c, PF_E_ARG, "the hidden state of layer " + std::to_string(il) + " has no buffer");
  const bool dev_tokens = is_device_ptr(tokens);
  if (!dev_tokens)
    for (int i = 0; i < T; ++i)
      if (tokens[i] < 0 || tokens[i] >= c->V) return fail(c, PF_E_ARG, "token id outside [0, vocab)");
  NvtxRange r_ubatch(is_last ? "ubatch (last)" : "ubatch");
  cudaStream_t s = c->stream;
  PF_CUDA(c, cudaMemcpyAsync(c->tok, tokens, T * 4, dev_tokens ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, s));

  const int L = c->L, S = c->S, D = c->D, LP = L * c->P;
  const int max_ctx = c->d.max_ctx;
  // per layer the cache holds every sequence's cells: sequence q at rows
  // [q * max_ctx, (q + 1) * max_ctx)
  const size_t seg = static_cast<size_t>(c->d.n_seq_max) * max_ctx * c->kv;
  const size_t seq_cells = static_cast<size_t>(max_ctx) * c->kv;
  const bool prune = multi ? (c->prune_enable == PF_PRUNE_ON && gather_possible(c->d))
                           : predicate(c->d, c->prune_enable == PF_PRUNE_ON);
  // the output row of the KV-shared layers takes the single-row kernels
  // unless the plain unpruned pass was asked for
  const bool row_kernels = c->prune_enable != PF_PRUNE_OFF_PLAIN;
  const int64_t pos0 = runs[0].pos0;
  const int kv_len = static_cast<int>(pos0) + T;  // single-sequence ubatches

  // several sequences: each row's position and cache row, the output rows
  // and their positions, uploaded once for the ubatch
  int* d_row_pos = c->rowinfo;
  int* d_row_slot = c->rowinfo + c->rows_alloc;
  int* d_out_rows = c->rowinfo + 2 * c->rows_alloc;
  int* d_out_pos = c->rowinfo + 3 * c->rows_alloc;
  std::vector<int> out_rows, out_pos, out_run;
  for (size_t k = 0; k < runs.size(); ++k)
    if (runs[k].last) {
      out_rows.push_back(runs[k].row0 + runs[k].n - 1);
      out_pos.push_back(static_cast<int>(runs[k].pos0) + runs[k].n - 1);
      out_run.push_back(static_cast<int>(k));
    }
  if (multi) {
    std::vector<int>& h = c->rowinfo_host;
    h.assign(static_cast<size_t>(4) * c->rows_alloc, 0);
    for (const Run& r : runs)
      for (int i = 0; i < r.n; ++i) {
        h[r.row0 + i] = static_cast<int>(r.pos0) + i;
        h[c->rows_alloc + r.row0 + i] = r.seq * max_ctx + static_cast<int>(r.pos0) + i;
      }
    for (int j = 0; j < n_out; ++j) {
      h[2 * c->rows_alloc + j] = out_rows[j];
      h[3 * c->rows_alloc + j] = out_pos[j];
    }
    PF_CUDA(c, cudaMemcpyAsync(c->rowinfo, h.data(), h.size() * 4, cudaMemcpyHostToDevice, s));
  }

  EmbedArgs ea;
  ea.tok = c->tok;
  ea.T = T;
  ea.vocab = c->V;
  ea.D = D;
  ea.wq4 = c->d.wtype == PF_W_Q4_0;
  ea.tok_table = c->tok_table;
  ea.x = c->x;
  ea.ple_table = c->P > 0 ? c->ple_table : nullptr;
  ea.LP = LP;
  ea.ple_scale = c->P > 0 ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(c->P))) : 1.0f;
  ea.ple = c->ple;
  ea.err = c->err;
  PF_CUDA(c, counted(c, PF_KC_OTHER, 1, 0.0, T * (4.0 + D * 4.0 + LP * 2.0), [&] { return launch_embed(ea, s); }));

  float* xcur = c->x;
  int M = T;
  int pos_base = static_cast<int>(pos0);
  const __nv_bfloat16* ple_view = c->ple;
  bool gathered = false;
  // One projection of a layer over the launch's `rows` rows.  With
  // `out_row`, the last row streams through the one-row kernel
  // (launch_gemv) and the rows before it (if any) take the tensor cores;
  // otherwise every row takes the tensor cores.  The output row of a
  // KV-shared layer in the final ubatch takes the one-row kernel in both
  // pruning modes (alone after the pruning, beside the other rows without
  // it), so its bits do not depend on the mode; a one-token ubatch (a decode
  // step) takes it in every layer.  Work counted per row: flops_row FLOPs and
  // io_row activation bytes, plus the weight bytes once per launch.  (The
  // tensor-core kernel's rows are independent of each other bit for bit, so
  // the rows of several sequences keep their bits whether the launch holds
  // every row or only the gathered output rows.)
  // norm_src / norm_gain: the projection's input is the RMS norm of these
  // residual rows; the one-row kernel then forms its row's norm itself
  // (the launch's A rows still serve the tensor-core part).
  auto project = [&](const ActMat& A, int rows, bool out_row, const WeightMat& Wm, const EpiParams& e,
                     double flops_row, double io_row, double wbytes, const float* norm_src = nullptr,
                     const float* norm_gain = nullptr) -> cudaError_t {
    const int m_tc = out_row ? rows - 1 : rows;
    if (m_tc > 0) {
      const cudaError_t err = counted(c, gemm_class(m_tc), 1, flops_row * m_tc, wbytes + io_row * m_tc,
                                      [&] { return launch_gemm(A, m_tc, Wm, e, c->err, s); });
      if (err != cudaSuccess) return err;
    }
    if (!out_row) return cudaSuccess;
    ActMat a1 = A;
    a1.dev = A.dev + static_cast<size_t>(rows - 1) * A.K;
    const EpiParams e1 = shift_rows(e, rows - 1);
    const float* nx = norm_src ? norm_src + static_cast<size_t>(rows - 1) * D : nullptr;
    return counted(c, PF_KC_GEMM_ROW, 1, flops_row, wbytes + io_row, [&] {
      return launch_gemv(a1, Wm, e1, c->err, s, nx, norm_gain, c->d.rms_eps);
    });
  };
  // the single-row attention of one output row
  auto row_attention = [&](const AttnArgs& base, int row, int seq, int pos) -> cudaError_t {
    AttnArgs r = base;
    r.M = 1;
    r.q = c->q16 + static_cast<size_t>(row) * c->q;
    r.out = c->att + static_cast<size_t>(row) * c->q;
    r.k = base.k + static_cast<size_t>(seq) * seq_cells;
    r.v = base.v + static_cast<size_t>(seq) * seq_cells;
    r.pos_base = pos;
    r.kv_len = pos + 1;
    const int n_keys = pos + 1;
    return counted(c, PF_KC_ATTN_ROW, 1, static_cast<double>(n_keys) * c->Hq * 4.0 * c->hd,
                   n_keys * c->kv * 4.0 + c->q * 4.0, [&] { return launch_attn_split(r, c->row_partials, s); });
  };
  // the prefill attention of rows [row0, row0 + n) of sequence seq at positions pos .. pos + n - 1
  auto rows_attention = [&](const AttnArgs& base, int row0, int n, int seq, int pos, int keys) -> cudaError_t {
    AttnArgs r = base;
    r.M = n;
    r.q = c->q16 + static_cast<size_t>(row0) * c->q;
    r.out = c->att + static_cast<size_t>(row0) * c->q;
    r.k = base.k + static_cast<size_t>(seq) * seq_cells;
    r.v = base.v + static_cast<size_t>(seq) * seq_cells;
    r.pos_base = pos;
    r.kv_len = keys;
    // (query head, visible key) pairs: rows at positions pos .. pos+n-1
    const double pairs = static_cast<double>(n) * pos + 0.5 * n * (n + 1.0);
    return counted(c, PF_KC_ATTN, attn_launch_count(r), pairs * c->Hq * 4.0 * c->hd, keys * c->kv * 4.0 + n * c->q * 4.0,
                   [&] { return launch_attn_prefill(r, c->partials, s); });
  };

  for (int il = 0; il < L; ++il) {
    const LayerW& W = c->layers[il];
    char range_name[32];
    std::snprintf(range_name, sizeof range_name, "layer %d", il);
    NvtxRange r_layer(range_name);
    if (prune && il == S) {
      if (!is_last) {
        break;
      }
      if (!multi) {
        // keep the output row only: the rest of the pass works on row T-1 of
        // the residual in place, and its one-row projections form their
        // norms themselves
        xcur = c->x + static_cast<size_t>(T - 1) * D;
        M = 1;
        pos_base = static_cast<int>(pos0) + T - 1;
        ple_view = c->ple + static_cast<size_t>(T - 1) * LP;
      } else {
        // keep one row per finishing sequence (the norm gathers them), and
        // their per-layer-embedding rows
        PF_CUDA(c, counted(c, PF_KC_NORM, 1, 0.0, n_out * D * 10.0, [&] {
                   return launch_rmsnorm(c->x, 0, n_out, D, W.attn_norm, c->d.rms_eps, c->y, c->xr, s, nullptr,
                                         d_out_rows);
                 }));
        if (c->P > 0)
          PF_CUDA(c, counted(c, PF_KC_OTHER, 1, 0.0, n_out * LP * 4.0, [&] {
                     return launch_gather_rows(c->ple, c->ple_g, d_out_rows, n_out, static_cast<size_t>(LP) * 2, s);
                   }));
        M = n_out;
        ple_view = c->ple_g;
        xcur = c->xr;
      }
      gathered = true;
    } else {
      // a requested hidden state entering this layer leaves as the norm's
      // input copy; a one-row launch needs the norm for nothing else
      float* inp = c->layer_inp.empty() || !c->layer_inp[il] ? nullptr : c->layer_out[il];
      if (multi || M > 1 || inp)
        PF_CUDA(c, counted(c, PF_KC_NORM, 1, 0.0, M * D * (6.0 + (inp ? 4.0 : 0.0)), [&] {
                   return launch_rmsnorm(xcur, 0, M, D, W.attn_norm, c->d.rms_eps, c->y, inp, s);
                 }));
    }
    const bool writes = il < S;
    const int src = writes ? il : c->kv_src[il];
    // the output row of a KV-shared layer in the final ubatch, and the one
    // row of a one-row launch, take the single-row kernels (see project);
    // ubatches of several sequences keep every projection on the tensor cores
    const bool out_row = !multi && (M == 1 || (!writes && is_last && row_kernels));
    {
      EpiParams e;
      e.kind = EPI_QKV;
      e.q_out = c->q16;
      e.q_dim = c->q;
      e.kv_dim = writes ? c->kv : 0;
      e.head_dim = c->hd;
      e.pos0 = pos_base;
      e.rope = c->rope;
      e.k_cache = c->cache + static_cast<size_t>(il) * seg;
      e.v_cache = c->cache + static_cast<size_t>(c->L_w + il) * seg;
      if (multi) {
        e.row_pos = gathered ? d_out_pos : d_row_pos;
        e.row_slot = gathered ? nullptr : d_row_slot;
      }
      const double n_out_cols = c->q + 2.0 * e.kv_dim;
      PF_CUDA(c, project(c->a_y, M, out_row, W.qkv, e, 2.0 * n_out_cols * D, D * 2.0 + n_out_cols * 2.0,
                         gemm_wbytes(c, n_out_cols, D), xcur, W.attn_norm));
    }
    {
      AttnArgs a;
      a.q = c->q16;
      a.k = c->cache + static_cast<size_t>(src) * seg;
      a.v = c->cache + static_cast<size_t>(c->L_w + src) * seg;
      a.out = c->att;
      a.M = M;
      a.Hq = c->Hq;
      a.Hkv = c->Hkv;
      a.hd = c->hd;
      a.pos_base = pos_base;
      a.kv_len = kv_len;
      a.err = c->err;
      if (!multi) {
        // the output row takes the single-row attention, as in project()
        const int m_rest = out_row ? M - 1 : M;  // rows for the prefill kernels
        if (m_rest > 0) PF_CUDA(c, rows_attention(a, 0, m_rest, 0, pos_base, kv_len));
        if (out_row) PF_CUDA(c, row_attention(a, M - 1, 0, pos_base + M - 1));
      } else if (gathered) {
        for (int j = 0; j < n_out; ++j) PF_CUDA(c, row_attention(a, j, runs[out_run[j]].seq, out_pos[j]));
      } else {
        // each sequence attends to its own cells; the output row of a
        // finishing sequence takes the single-row attention in the KV-shared
        // layers, as it does after the gather
        for (const Run& r : runs) {
          const bool single = !writes && r.last && row_kernels;
          const int n_pre = single ? r.n - 1 : r.n;
          const int keys = static_cast<int>(r.pos0) + r.n;
          if (n_pre > 0) PF_CUDA(c, rows_attention(a, r.row0, n_pre, r.seq, static_cast<int>(r.pos0), keys));
          if (single) PF_CUDA(c, row_attention(a, r.row0 + r.n - 1, r.seq, keys - 1));
        }
      }
    }
    {
      EpiParams e;
      e.kind = EPI_RESID;
      e.N = D;
      e.out_f32 = xcur;
      e.ld_f32 = D;
      PF_CUDA(c, project(c->a_att, M, out_row, W.o, e, 2.0 * D * c->q, c->q * 2.0 + D * 8.0, gemm_wbytes(c, D, c->q)));
    }
    if (multi || M > 1)
      PF_CUDA(c, counted(c, PF_KC_NORM, 1, 0.0, M * D * 6.0, [&] {
                 return launch_rmsnorm(xcur, 0, M, D, W.ffn_norm, c->d.rms_eps, c->y, nullptr, s);
               }));
    {
      EpiParams e;
      e.kind = EPI_GLU;
      e.N = c->F;
      e.out_bf16 = c->h;
      e.ld_bf16 = c->F;
      e.act = c->d.ffn_kind == PF_FFN_GEGLU ? 0 : 1;
      PF_CUDA(c, project(c->a_y, M, out_row, W.gu, e, 4.0 * c->F * D, D * 2.0 + c->F * 2.0,
                         gemm_wbytes(c, 2.0 * c->F, D), xcur, W.ffn_norm));
    }
    {
      EpiParams e;
      e.kind = EPI_RESID;
      e.N = D;
      e.out_f32 = xcur;
      e.ld_f32 = D;
      if (c->P > 0) {
        e.out_bf16 = c->xb;
        e.ld_bf16 = D;
      }
      PF_CUDA(c, project(c->a_h, M, out_row, W.down, e, 2.0 * D * c->F, c->F * 2.0 + D * 8.0, gemm_wbytes(c, D, c->F)));
    }
    if (c->P > 0) {
      EpiParams e;
      e.kind = EPI_PLE;
      e.N = c->P;
      e.out_bf16 = c->pg;
      e.ld_bf16 = c->P;
      e.ple = ple_view + static_cast<size_t>(il) * c->P;
      e.ple_stride = LP;
      PF_CUDA(c, project(c->a_xb, M, out_row, W.pg, e, 2.0 * c->P * D, D * 2.0 + c->P * 4.0, gemm_wbytes(c, c->P, D)));
      EpiParams r;
      r.kind = EPI_RESID;
      r.N = D;
      r.out_f32 = xcur;
      r.ld_f32 = D;
      PF_CUDA(c, project(c->a_pg, M, out_row, W.pp, r, 2.0 * D * c->P, c->P * 2.0 + D * 8.0, gemm_wbytes(c, D, c->P)));
    }
  }
  {
    // the final hidden state (index L) and the embeddings output of every
    // row; requesting either turns the pruning off, so all T rows are here
    float* fin = c->layer_inp.empty() || !c->layer_inp[L] ? nullptr : c->layer_out[L];
    float* embd = c->d.embeddings ? c->embd_out : nullptr;
    if ((fin || embd) && !gathered && !(prune && !is_last))
      PF_CUDA(c, counted(c, PF_KC_NORM, 1, 0.0, M * D * (4.0 + (fin ? 4.0 : 0.0) + (embd ? 4.0 : 0.0)), [&] {
                 return launch_rmsnorm(xcur, 0, M, D, c->out_norm, c->d.rms_eps, nullptr, fin, s, embd);
               }));
  }
  if (is_last && !multi) {
    // the head projects the output row's final norm, formed inside the launch
    NvtxRange r_head("head");
    const int row = gathered ? 0 : T - 1;
    const float* xrow = xcur + static_cast<size_t>(row) * D;
    EpiParams e;
    e.kind = EPI_F32;
    e.N = c->V;
    e.out_f32 = logits;
    e.ld_f32 = c->V;
    PF_CUDA(c, counted(c, gemm_class(1), 1, 2.0 * c->V * D, D * 4.0 + gemm_wbytes(c, c->V, D) + c->V * 4.0, [&] {
      return launch_gemv(c->a_y, c->head, e, c->err, s, xrow, c->out_norm, c->d.rms_eps);
    }));
  } else if (is_last) {
    // one logits row per finishing sequence, in run order: their rows are
    // normed into y (gathered: rows 0 .. n_out-1 of xr; else picked out of x)
    // and projected together on the tensor cores
    NvtxRange r_head("head");
    PF_CUDA(c, counted(c, PF_KC_NORM, 1, 0.0, n_out * D * 6.0, [&] {
               return launch_rmsnorm(xcur, 0, n_out, D, c->out_norm, c->d.rms_eps, c->y, nullptr, s, nullptr,
                                     gathered ? nullptr : d_out_rows);
             }));
    EpiParams e;
    e.kind = EPI_F32;
    e.N = c->V;
    e.out_f32 = logits;
    e.ld_f32 = c->V;
    PF_CUDA(c, counted(c, gemm_class(n_out), 1, 2.0 * n_out * c->V * D,
                       n_out * D * 2.0 + gemm_wbytes(c, c->V, D) + n_out * c->V * 4.0,
                       [&] { return launch_gemm(c->a_y, n_out, c->head, e, c->err, s); }));
  }
  for (const Run& r : runs) c->seq_pos[r.seq] = r.pos0 + r.n;
  return PF_OK;
}

}  // namespace

extern "C" int prefill_ubatch(prefill_ctx* c, const int32_t* tokens, int32_t T, int64_t pos0, int32_t is_last,
                              float* logits) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  if (!tokens || T < 1 || T > c->d.ubatch_max) return fail(c, PF_E_ARG, "n_tokens outside [1, ubatch_max]");
  if (pos0 != c->seq_pos[0]) return fail(c, PF_E_ARG, "pos0 must equal the cached position count");
  if (pos0 + T > c->d.max_ctx) return fail(c, PF_E_ARG, "positions would exceed max_ctx");
  std::vector<Run> runs(1);
  runs[0].seq = 0;
  runs[0].n = T;
  runs[0].last = is_last ? 1 : 0;
  runs[0].row0 = 0;
  runs[0].pos0 = pos0;
  return run_ubatch(c, tokens, T, runs, false, logits);
}

extern "C" int prefill_ubatch_seqs(prefill_ctx* c, const int32_t* tokens, const prefill_seq_run* runs, int32_t n_runs,
                                   float* logits) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  if (!tokens || !runs || n_runs < 1 || n_runs > c->d.n_seq_max)
    return fail(c, PF_E_ARG, "n_runs outside [1, n_seq_max]");
  std::vector<Run> rs(n_runs);
  std::vector<char> seen(c->d.n_seq_max, 0);
  int T = 0;
  for (int k = 0; k < n_runs; ++k) {
    const prefill_seq_run& r = runs[k];
    if (r.seq_id < 0 || r.seq_id >= c->d.n_seq_max) return fail(c, PF_E_ARG, "seq_id outside [0, n_seq_max)");
    if (seen[r.seq_id]) return fail(c, PF_E_ARG, "a sequence appears in two runs of one ubatch");
    seen[r.seq_id] = 1;
    if (r.n_tokens < 1) return fail(c, PF_E_ARG, "a run without tokens");
    if (c->seq_pos[r.seq_id] + r.n_tokens > c->d.max_ctx) return fail(c, PF_E_ARG, "positions would exceed max_ctx");
    rs[k].seq = r.seq_id;
    rs[k].n = r.n_tokens;
    rs[k].last = r.is_last ? 1 : 0;
    rs[k].row0 = T;
    rs[k].pos0 = c->seq_pos[r.seq_id];
    T += r.n_tokens;
    if (T > c->d.ubatch_max) return fail(c, PF_E_ARG, "the runs hold more than ubatch_max tokens");
  }
  return run_ubatch(c, tokens, T, rs, true, logits);
}

extern "C" int prefill_graph_capture(prefill_ctx* c, const int32_t* tokens, int32_t T, int64_t pos0,
                                     int32_t is_last, float* logits) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  if (!c->stream) return fail(c, PF_E_ARG, "recording needs a context created on a non-default stream");
  if (c->timing) return fail(c, PF_E_ARG, "per-launch timing is on");
  if (!tokens || !is_device_ptr(tokens)) return fail(c, PF_E_ARG, "recorded tokens must be device memory");
  if (c->graph) {
    cudaGraphExecDestroy(c->graph);
    c->graph = nullptr;
  }
  const std::vector<int64_t> saved = c->seq_pos;
  const prefill_stats saved_stats = c->stats;
  // relaxed: the host-side queries the call makes (pointer kinds, device
  // attributes) are allowed while the stream records
  PF_CUDA(c, cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeRelaxed));
  const int rc = prefill_ubatch(c, tokens, T, pos0, is_last, logits);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(c->stream, &g);
  // recording runs nothing: the positions and the launch counts stay as they were
  c->seq_pos = saved;
  c->stats = saved_stats;
  if (rc != PF_OK) {
    if (g) cudaGraphDestroy(g);
    return rc;
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaStreamEndCapture");
  cudaGraphExec_t x = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&x, g, 0);
  cudaGraphDestroy(g);
  if (ei != cudaSuccess) return cuda_fail(c, ei, "cudaGraphInstantiate");
  c->graph = x;
  c->graph_pos0 = pos0;
  c->graph_T = T;
  return PF_OK;
}

extern "C" int prefill_graph_launch(prefill_ctx* c) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  if (!c->graph) return fail(c, PF_E_ARG, "no recorded ubatch");
  if (c->seq_pos[0] != c->graph_pos0) return fail(c, PF_E_ARG, "the recorded ubatch starts at another position");
  PF_CUDA(c, cudaGraphLaunch(c->graph, c->stream));
  c->seq_pos[0] = c->graph_pos0 + c->graph_T;
  return PF_OK;
}

extern "C" int64_t prefill_seq_n_pos(const prefill_ctx* c, int32_t seq_id) {
  if (!c || seq_id < 0 || seq_id >= c->d.n_seq_max) return -1;
  return c->seq_pos[seq_id];
}

extern "C" int prefill_seq_reset(prefill_ctx* c, int32_t seq_id) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  if (seq_id < 0 || seq_id >= c->d.n_seq_max) return fail(c, PF_E_ARG, "seq_id outside [0, n_seq_max)");
  c->seq_pos[seq_id] = 0;
  return PF_OK;
}

extern "C" int prefill_set_output(prefill_ctx* c, int32_t which, float* dst) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  if (dst && !is_device_ptr(dst)) return fail(c, PF_E_ARG, "output buffer is not device memory");
  if (which == PF_OUT_EMBD) {
    if (!c->d.embeddings) return fail(c, PF_E_ARG, "the description requests no embeddings output");
    c->embd_out = dst;
    return PF_OK;
  }
  if (which < 0 || which > c->L || c->layer_inp.empty() || !c->layer_inp[which])
    return fail(c, PF_E_ARG, "the description requests no hidden state for that layer");
  c->layer_out[which] = dst;
  return PF_OK;
}

extern "C" int prefill_sync(prefill_ctx* c) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  PF_CUDA(c, cudaStreamSynchronize(c->stream));
  return check_device_error(c);
}

extern "C" int64_t prefill_n_pos(const prefill_ctx* c) { return c ? c->seq_pos[0] : -1; }

extern "C" int prefill_reset(prefill_ctx* c) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  std::fill(c->seq_pos.begin(), c->seq_pos.end(), 0);
  return PF_OK;
}

extern "C" int prefill_set_prune(prefill_ctx* c, int32_t enable) {
  if (!c) return fail(nullptr, PF_E_ARG, "null context");
  if (enable != PF_PRUNE_OFF && enable != PF_PRUNE_ON && enable != PF_PRUNE_OFF_PLAIN)
    return fail(c, PF_E_ARG, "pruning mode must be PF_PRUNE_OFF, PF_PRUNE_ON or PF_PRUNE_OFF_PLAIN");
  c->prune_enable = enable;
  return PF_OK;
}

extern "C" int prefill_prune_active(const prefill_ctx* c) {
  return c ? (predicate(c->d, c->prune_enable == PF_PRUNE_ON) ? 1 : 0) : 0;
}

// ---------------------------------------------------------------------------
// KV image

extern "C" int64_t prefill_kv_image_bytes_for(int32_t n_layers_written, int64_t n_pos, int32_t kv_dim) {
  if (n_layers_written < 0 || n_pos < 0 || kv_dim < 0) return -1;
  return 16 + 2 * static_cast<int64_t>(n_layers_written) * n_pos * kv_dim * 2;
}

extern "C" int64_t prefill_kv_image_bytes(const prefill_ctx* c, int64_t n_pos) {
  if (!c) return -1;
  return prefill_kv_image_bytes_for(c->L_w, n_pos, c->kv);
}

extern "C" int prefill_kv_header_check(const void* header16, int32_t n_layers_written, int32_t kv_dim, int64_t n_pos,
                                       int64_t max_ctx, size_t image_bytes) {
  if (!header16 || image_bytes < 16) return PF_E_KV_MAGIC;
  const uint8_t* h = static_cast<const uint8_t*>(header16);
  if (std::memcmp(h, "KVCP", 4) != 0) return PF_E_KV_MAGIC;
  int32_t f[3];
  for (int i = 0; i < 3; ++i)
    f[i] = static_cast<int32_t>(static_cast<uint32_t>(h[4 + 4 * i]) | (static_cast<uint32_t>(h[5 + 4 * i]) << 8) |
                                (static_cast<uint32_t>(h[6 + 4 * i]) << 16) | (static_cast<uint32_t>(h[7 + 4 * i]) << 24));
  const int32_t n_img = f[0], l_img = f[1], kv_img = f[2];
  if (l_img != n_layers_written || kv_img != kv_dim) return PF_E_KV_SHAPE;
  if (n_img < 0 || n_pos < 0 || n_pos > n_img || n_pos > max_ctx) return PF_E_KV_RANGE;
  if (static_cast<int64_t>(image_bytes) < prefill_kv_image_bytes_for(l_img, n_img, kv_img)) return PF_E_KV_RANGE;
  return PF_OK;
}

extern "C" int kv_save(prefill_ctx* c, void* dst, size_t dst_bytes) {
  if (!c || !dst) return fail(c, PF_E_ARG, "null argument");
  NvtxRange r_save("kv_save");
  const int64_t n = c->seq_pos[0];
  const int64_t need = prefill_kv_image_bytes(c, n);
  if (static_cast<int64_t>(dst_bytes) < need) return fail(c, PF_E_ARG, "destination smaller than the image");
  if (reinterpret_cast<uintptr_t>(dst) % 16 != 0) return fail(c, PF_E_ARG, "destination not 16-byte aligned");
  int32_t h4[4];
  std::memcpy(h4, "KVCP", 4);
  h4[1] = static_cast<int32_t>(n);
  h4[2] = c->L_w;
  h4[3] = c->kv;
  const size_t seg_bytes = static_cast<size_t>(n) * c->kv * 2;
  // sequence 0's cells of each layer; a layer holds n_seq_max sequences' cells
  const int64_t layer_halves = static_cast<int64_t>(c->d.n_seq_max) * c->d.max_ctx * c->kv;
  const size_t cache_pitch = static_cast<size_t>(layer_halves) * 2;
  if (is_device_ptr(dst)) {
    PF_CUDA(c, counted(c, PF_KC_OTHER, 1, 0.0, 2.0 * seg_bytes * 2 * c->L_w, [&] {
               return launch_kv_copy(0, c->cache, layer_halves, static_cast<uint8_t*>(dst),
                                     static_cast<int64_t>(seg_bytes), 2 * c->L_w, static_cast<int64_t>(seg_bytes), h4,
                                     c->stream);
             }));
  } else {
    std::memcpy(dst, h4, 16);
    if (seg_bytes > 0)
      PF_CUDA(c, cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + 16, seg_bytes, c->cache, cache_pitch, seg_bytes,
                                   2 * c->L_w, cudaMemcpyDeviceToHost, c->stream));
    PF_CUDA(c, cudaStreamSynchronize(c->stream));
  }
  if (std::getenv("PREFILL_LOG")) std::fprintf(stderr, "KV cache saved: %lld positions\n", (long long)n);
  return PF_OK;
}

extern "C" int kv_load(prefill_ctx* c, const void* src, size_t src_bytes, int64_t n_pos) {
  if (!c || !src) return fail(c, PF_E_ARG, "null argument");
  NvtxRange r_load("kv_load");
  const bool dev = is_device_ptr(src);
  uint8_t hdr[16] = {0};
  if (src_bytes >= 16) {
    if (dev) {
      PF_CUDA(c, cudaStreamSynchronize(c->stream));
      PF_CUDA(c, cudaMemcpy(hdr, src, 16, cudaMemcpyDeviceToHost));
    } else {
      std::memcpy(hdr, src, 16);
    }
  }
  const int rc = prefill_kv_header_check(hdr, c->L_w, c->kv, n_pos, c->d.max_ctx, src_bytes);
  if (rc == PF_E_KV_MAGIC) return fail(c, rc, "not a KV image (magic)");
  if (rc == PF_E_KV_SHAPE) return fail(c, rc, "KV image layers or kv_dim do not match the model");
  if (rc != PF_OK) return fail(c, rc, "KV image position count out of range");
  if (dev && reinterpret_cast<uintptr_t>(src) % 16 != 0) return fail(c, PF_E_ARG, "source not 16-byte aligned");
  int32_t n_img;
  std::memcpy(&n_img, hdr + 4, 4);
  const size_t img_seg = static_cast<size_t>(n_img) * c->kv * 2;
  const size_t copy = static_cast<size_t>(n_pos) * c->kv * 2;
  // sequence 0's cells of each layer; a layer holds n_seq_max sequences' cells
  const int64_t layer_halves = static_cast<int64_t>(c->d.n_seq_max) * c->d.max_ctx * c->kv;
  const size_t cache_pitch = static_cast<size_t>(layer_halves) * 2;
  if (copy > 0) {
    if (dev) {
      PF_CUDA(c, counted(c, PF_KC_OTHER, 1, 0.0, 2.0 * copy * 2 * c->L_w, [&] {
                 return launch_kv_copy(1, c->cache, layer_halves,
                                       const_cast<uint8_t*>(static_cast<const uint8_t*>(src)),
                                       static_cast<int64_t>(img_seg), 2 * c->L_w, static_cast<int64_t>(copy),
                                       reinterpret_cast<const int32_t*>(hdr), c->stream);
               }));
    } else {
      PF_CUDA(c, cudaMemcpy2DAsync(c->cache, cache_pitch, static_cast<const uint8_t*>(src) + 16, img_seg, copy,
                                   2 * c->L_w, cudaMemcpyHostToDevice, c->stream));
    }
  }
  c->seq_pos[0] = n_pos;
  if (std::getenv("PREFILL_LOG"))
    std::fprintf(stderr, "KV cache loaded: %lld positions; skipping %lld cached prompt tokens\n", (long long)n_pos,
                 (long long)n_pos);
  return PF_OK;
}

// ---------------------------------------------------------------------------
// KV image files (PicoLM KV cache article, "usage", "file" and "rules"): one
// image per file, written and read through host memory

namespace {

struct FileCloser {
  std::FILE* f;
  ~FileCloser() {
    if (f) std::fclose(f);
  }
};

// size of an open file, or -1
int64_t file_size(std::FILE* f) {
  if (std::fseek(f, 0, SEEK_END) != 0) return -1;
  const long n = std::ftell(f);
  if (n < 0 || std::fseek(f, 0, SEEK_SET) != 0) return -1;
  return static_cast<int64_t>(n);
}

// header checks of kv_load_file; *n_img = the file's position count
int check_file(std::FILE* f, int32_t n_layers_written, int32_t kv_dim, int64_t n_pos, int64_t max_ctx,
               int64_t* n_img, int64_t* bytes) {
  const int64_t size = file_size(f);
  if (size < 0) return PF_E_IO;
  uint8_t hdr[16] = {0};
  if (size >= 16 && std::fread(hdr, 1, 16, f) != 16) return PF_E_IO;
  int32_t n_file = 0;
  std::memcpy(&n_file, hdr + 4, 4);
  const int64_t want = n_pos < 0 ? n_file : n_pos;
  const int rc = prefill_kv_header_check(hdr, n_layers_written, kv_dim, want, max_ctx, static_cast<size_t>(size));
  if (rc != PF_OK) return rc;
  *n_img = n_file;
  *bytes = size;
  return PF_OK;
}

}  // namespace

extern "C" int prefill_kv_file_check(const char* path, int32_t n_layers_written, int32_t kv_dim, int64_t max_ctx,
                                     int64_t* n_pos_out) {
  if (!path) return PF_E_ARG;
  FileCloser fc{std::fopen(path, "rb")};
  if (!fc.f) return PF_E_IO;
  int64_t n = 0, bytes = 0;
  const int rc = check_file(fc.f, n_layers_written, kv_dim, -1, max_ctx, &n, &bytes);
  if (rc == PF_OK && n_pos_out) *n_pos_out = n;
  return rc;
}

extern "C" int kv_save_file(prefill_ctx* c, const char* path) {
  if (!c || !path) return fail(c, PF_E_ARG, "null argument");
  const int64_t bytes = prefill_kv_image_bytes(c, c->seq_pos[0]);
  std::vector<uint8_t> img(static_cast<size_t>(bytes) + 16);
  // 16-byte aligned staging inside the vector
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(img.data()) + 15) & ~uintptr_t(15));
  const int rc = kv_save(c, p, static_cast<size_t>(bytes));
  if (rc != PF_OK) return rc;
  FileCloser fc{std::fopen(path, "wb")};
  if (!fc.f) return fail(c, PF_E_IO, std::string("cannot open ") + path + " for writing");
  if (std::fwrite(p, 1, static_cast<size_t>(bytes), fc.f) != static_cast<size_t>(bytes))
    return fail(c, PF_E_IO, std::string("short write to ") + path);
  if (std::fclose(fc.f) != 0) {
    fc.f = nullptr;
    return fail(c, PF_E_IO, std::string("cannot close ") + path);
  }
  fc.f = nullptr;
  return PF_OK;
}

extern "C" int kv_load_file(prefill_ctx* c, const char* path, int64_t n_pos) {
  if (!c || !path) return fail(c, PF_E_ARG, "null argument");
  FileCloser fc{std::fopen(path, "rb")};
  if (!fc.f) return fail(c, PF_E_IO, std::string("cannot open ") + path);
  int64_t n_img = 0, bytes = 0;
  int rc = check_file(fc.f, c->L_w, c->kv, n_pos, c->d.max_ctx, &n_img, &bytes);
  if (rc == PF_E_IO) return fail(c, rc, std::string("cannot read ") + path);
  if (rc == PF_E_KV_MAGIC) return fail(c, rc, "not a KV image file (magic)");
  if (rc == PF_E_KV_SHAPE) return fail(c, rc, "KV image file layers or kv_dim do not match the model");
  if (rc != PF_OK) return fail(c, rc, "KV image file position count out of range");
  const int64_t img_bytes = prefill_kv_image_bytes(c, n_img);
  std::vector<uint8_t> img(static_cast<size_t>(img_bytes) + 16);
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(img.data()) + 15) & ~uintptr_t(15));
  if (std::fseek(fc.f, 0, SEEK_SET) != 0 ||
      std::fread(p, 1, static_cast<size_t>(img_bytes), fc.f) != static_cast<size_t>(img_bytes))
    return fail(c, PF_E_IO, std::string("cannot read ") + path);
  rc = kv_load(c, p, static_cast<size_t>(img_bytes), n_pos < 0 ? n_img : n_pos);
  if (rc != PF_OK) return rc;
  PF_CUDA(c, cudaStreamSynchronize(c->stream));  // the staging buffer is released on return
  return PF_OK;
}

extern "C" int prefill_prune_predicate(const prefill_model_desc* d) {
  if (!d) return PF_E_ARG;
  return predicate(*d, d->prune_shared_enable) ? 1 : 0;
}
