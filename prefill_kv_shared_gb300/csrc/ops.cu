// Per-kernel entry points (include/prefill_ops.h): each uploads what it
// needs, runs one launcher of the prefill pass, waits and reports.
#include "../../include/prefill_ops.h"
#include "common.cuh"
#include "kernels.h"

#include <atomic>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

using namespace pf;

namespace {

thread_local std::string g_err;
// CTA pairs for the op entry points' GEMMs (pfop_set_gemm_pairs)
std::atomic<int> g_pairs{0};

int op_fail(int code, const std::string& m) {
  g_err = m;
  return code;
}

struct Scope {  // frees device memory on exit
  std::vector<void*> ptrs;
  ~Scope() {
    for (void* p : ptrs) cudaFree(p);
  }
  template <class T>
  cudaError_t alloc(T** out, size_t bytes) {
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, bytes ? bytes : 16);
    if (e == cudaSuccess) ptrs.push_back(p);
    *out = static_cast<T*>(p);
    return e;
  }
};

#define OP_CUDA(call)                                                                 \
  do {                                                                                \
    cudaError_t e_ = (call);                                                          \
    if (e_ != cudaSuccess) return op_fail(PF_E_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
  } while (0)

size_t rbytes(int wtype, int K) { return wtype == PF_W_Q4_0 ? static_cast<size_t>(K / 32) * 18 : static_cast<size_t>(K) * 4; }
int rup(int x, int m) { return (x + m - 1) / m * m; }

int make_weight(Scope& sc, WeightMat& w, int wtype, const std::vector<const void*>& rows, int K, int BN) {
  if (wtype != PF_W_Q4_0 && wtype != PF_W_F32) return op_fail(PF_E_ARG, "wtype");
  if (K <= 0 || K % 64 || rows.size() % BN) return op_fail(PF_E_ARG, "weight shape not tileable");
  w.K = K;
  w.BN = BN;
  w.N_rows = static_cast<int>(rows.size());
  // the split depends on the matrix shape only (as in a context with
  // ubatch_max = 512), so one row gives the same bits whatever M is
  const int kind = wtype == PF_W_Q4_0 ? W_Q4 : W_BF16;
  w.split = choose_split(kind, w.N_rows, BN, K, 512);
  const int pm = g_pairs.load();
  if (pm > 0 && kind == W_Q4 && (BN == 128 || BN == 192 || BN == 256)) {
    w.split = 1;
    w.pair = 1;
  } else {
    w.pair = pm == 0 ? choose_pair(kind, w.N_rows, BN, K, 512, w.split) : 0;
  }
  if (wtype == PF_W_Q4_0) {
    w.kind = W_Q4;
    std::vector<const uint8_t*> r(rows.size());
    for (size_t i = 0; i < rows.size(); ++i) r[i] = static_cast<const uint8_t*>(rows[i]);
    std::vector<uint8_t> t = repack_q4_tiles(r, K, BN);
    OP_CUDA(sc.alloc(&w.dev, t.size()));
    OP_CUDA(cudaMemcpy(w.dev, t.data(), t.size(), cudaMemcpyHostToDevice));
  } else {
    w.kind = W_BF16;
    std::vector<const float*> r(rows.size());
    for (size_t i = 0; i < rows.size(); ++i) r[i] = static_cast<const float*>(rows[i]);
    std::vector<uint16_t> t = repack_bf16_rows(r, K);
    OP_CUDA(sc.alloc(&w.dev, t.size() * 2));
    OP_CUDA(cudaMemcpy(w.dev, t.data(), t.size() * 2, cudaMemcpyHostToDevice));
  }
  std::string err;
  if (!make_weight_map(w, &err)) return op_fail(PF_E_CUDA, err);
  return PF_OK;
}

std::vector<const void*> rows_of(const void* m, int N, int K, int wtype, int BN) {
  std::vector<const void*> r(rup(N, BN), nullptr);
  for (int n = 0; n < N; ++n) r[n] = static_cast<const uint8_t*>(m) + n * rbytes(wtype, K);
  return r;
}

int make_act(ActMat& a, const void* dev, int rows, int K) {
  if (rows < 128) return op_fail(PF_E_ARG, "a_rows must be >= 128");
  a.dev = static_cast<const __nv_bfloat16*>(dev);
  a.rows = rows;
  a.K = K;
  std::string err;
  if (!make_act_map(a, &err)) return op_fail(PF_E_CUDA, err);
  return PF_OK;
}

int run_gemm(Scope& sc, const ActMat& A, int M, const WeightMat& W, const EpiParams& e, cudaStream_t s) {
  int* err = nullptr;
  OP_CUDA(sc.alloc(&err, 16));
  OP_CUDA(cudaMemsetAsync(err, 0, 16, s));
  OP_CUDA(launch_gemm(A, M, W, e, err, s));
  OP_CUDA(cudaStreamSynchronize(s));
  int h = 0;
  OP_CUDA(cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost));
  if (h) return op_fail(PF_E_DEVICE_TIMEOUT, "GEMM gave up a bounded wait, code " + std::to_string(h));
  return PF_OK;
}

}  // namespace

extern "C" const char* pfop_last_error(void) { return g_err.c_str(); }

extern "C" int pfop_set_gemm_pairs(int32_t mode) {
  if (mode < -1 || mode > 1) return op_fail(PF_E_ARG, "mode must be -1, 0 or 1");
  g_pairs.store(mode);
  return PF_OK;
}

void pf::set_op_error(const std::string& m) { g_err = m; }

extern "C" int32_t pfop_qkv_row_order(int32_t Hq, int32_t Hkv, int32_t hd, int32_t with_kv, int32_t* order,
                                      int32_t cap) {
  if (Hq < 1 || Hkv < 1 || hd < 2 || hd % 2 || (hd > QKV_BN && hd % QKV_BN) || !order || cap < 0)
    return op_fail(PF_E_ARG, "bad argument");
  const size_t q = static_cast<size_t>(Hq) * hd, kv = static_cast<size_t>(Hkv) * hd;
  // one byte per source row: a stored row's source is its offset from base
  std::vector<uint8_t> base(q + 2 * kv);
  const uint8_t* b = base.data();
  const std::vector<const void*> rows =
      qkv_tile_rows(b, with_kv ? b + q : nullptr, with_kv ? b + q + kv : nullptr, Hq, Hkv, hd, 1, QKV_BN);
  if (rows.size() > static_cast<size_t>(cap)) return op_fail(PF_E_ARG, "order holds fewer than the stored rows");
  for (size_t i = 0; i < rows.size(); ++i)
    order[i] = rows[i] ? static_cast<int32_t>(static_cast<const uint8_t*>(rows[i]) - b) : -1;
  return static_cast<int32_t>(rows.size());
}

extern "C" int64_t pfop_repack_q4(const void* w_host, int32_t N, int32_t K, int32_t bn, void* dst, int64_t dst_bytes) {
  if (!w_host || N < 1 || K < 64 || K % 64 || (bn != 64 && bn != 128 && bn != 192 && bn != 256))
    return op_fail(PF_E_ARG, "bad argument");
  const size_t rb = static_cast<size_t>(K / 32) * 18;
  std::vector<const uint8_t*> rows(static_cast<size_t>(rup(N, bn)), nullptr);
  for (int n = 0; n < N; ++n) rows[n] = static_cast<const uint8_t*>(w_host) + n * rb;
  const std::vector<uint8_t> t = repack_q4_tiles(rows, K, bn);
  const int64_t need = static_cast<int64_t>(t.size());
  if (!dst) return need;
  if (dst_bytes < need) return op_fail(PF_E_ARG, "dst smaller than the stored matrix");
  std::memcpy(dst, t.data(), t.size());
  return need;
}

extern "C" int pfop_linear_f32(int32_t wtype, const void* w_host, int32_t N, int32_t K, int32_t bn, const void* a_dev,
                               int32_t a_rows, int32_t M, float* out_dev, void* stream) {
  if (!w_host || !a_dev || !out_dev || N < 1 || M < 1 || M > a_rows ||
      (bn != 64 && bn != 128 && bn != 256 && !(bn == 192 && wtype == PF_W_Q4_0)))
    return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  WeightMat W;
  ActMat A;
  int rc;
  if ((rc = make_weight(sc, W, wtype, rows_of(w_host, N, K, wtype, bn), K, bn))) return rc;
  if ((rc = make_act(A, a_dev, a_rows, K))) return rc;
  EpiParams e;
  e.kind = EPI_F32;
  e.N = N;
  e.out_f32 = out_dev;
  e.ld_f32 = N;
  if (N % 4) return op_fail(PF_E_ARG, "N must be a multiple of 4");
  return run_gemm(sc, A, M, W, e, static_cast<cudaStream_t>(stream));
}

extern "C" int pfop_linear_row(int32_t wtype, const void* w_host, int32_t N, int32_t K, int32_t bn,
                               const void* a_dev, float* out_dev, int32_t iters, float* us, void* stream) {
  if (!w_host || !a_dev || !out_dev || N < 1 || N % 4 || K % 64 ||
      (bn != 64 && bn != 128 && bn != 256 && !(bn == 192 && wtype == PF_W_Q4_0)) || iters < 0 || (iters > 0 && !us))
    return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  WeightMat W;
  ActMat A;
  int rc;
  if ((rc = make_weight(sc, W, wtype, rows_of(w_host, N, K, wtype, bn), K, bn))) return rc;
  A.dev = static_cast<const __nv_bfloat16*>(a_dev);
  A.rows = 1;
  A.K = K;
  EpiParams e;
  e.kind = EPI_F32;
  e.N = N;
  e.out_f32 = out_dev;
  e.ld_f32 = N;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = nullptr;
  OP_CUDA(sc.alloc(&err, 16));
  OP_CUDA(cudaMemsetAsync(err, 0, 16, s));
  OP_CUDA(launch_gemv(A, W, e, err, s));
  if (iters > 0) {
    cudaEvent_t e0, e1;
    OP_CUDA(cudaEventCreate(&e0));
    OP_CUDA(cudaEventCreate(&e1));
    OP_CUDA(cudaEventRecord(e0, s));
    for (int i = 0; i < iters; ++i) OP_CUDA(launch_gemv(A, W, e, err, s));
    OP_CUDA(cudaEventRecord(e1, s));
    OP_CUDA(cudaEventSynchronize(e1));
    float ms = 0.f;
    OP_CUDA(cudaEventElapsedTime(&ms, e0, e1));
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    *us = ms * 1000.f / iters;
  }
  OP_CUDA(cudaStreamSynchronize(s));
  int h = 0;
  OP_CUDA(cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost));
  if (h) return op_fail(PF_E_DEVICE_TIMEOUT, "one-row projection gave up a bounded wait, code " + std::to_string(h));
  return PF_OK;
}

extern "C" int pfop_linear_bench(int32_t wtype, const void* w_host, int32_t N, int32_t K, int32_t bn, int32_t split,
                                 const void* a_dev, int32_t a_rows, int32_t M, float* out_dev, int32_t warmup,
                                 int32_t iters, float* us, void* stream) {
  if (!w_host || !a_dev || !out_dev || !us || N < 1 || N % 4 || M < 1 || M > a_rows ||
      (bn != 64 && bn != 128 && bn != 256 && !(bn == 192 && wtype == PF_W_Q4_0)) || iters < 1 || warmup < 0 ||
      split < -1 || (split == -1 && (wtype != PF_W_Q4_0 || bn == 64)))
    return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  WeightMat W;
  ActMat A;
  int rc;
  if ((rc = make_weight(sc, W, wtype, rows_of(w_host, N, K, wtype, bn), K, bn))) return rc;
  if (split > 0) {
    if ((K / 64) % split) return op_fail(PF_E_ARG, "split must divide K/64");
    W.split = split;
    W.pair = 0;
  } else if (split == -1) {
    W.split = 1;
    W.pair = 1;
  }
  if ((rc = make_act(A, a_dev, a_rows, K))) return rc;
  EpiParams e;
  e.kind = EPI_F32;
  e.N = N;
  e.out_f32 = out_dev;
  e.ld_f32 = N;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = nullptr;
  OP_CUDA(sc.alloc(&err, 16));
  OP_CUDA(cudaMemsetAsync(err, 0, 16, s));
  for (int i = 0; i < warmup; ++i) OP_CUDA(launch_gemm(A, M, W, e, err, s));
  cudaEvent_t e0, e1;
  OP_CUDA(cudaEventCreate(&e0));
  OP_CUDA(cudaEventCreate(&e1));
  OP_CUDA(cudaEventRecord(e0, s));
  for (int i = 0; i < iters; ++i) OP_CUDA(launch_gemm(A, M, W, e, err, s));
  OP_CUDA(cudaEventRecord(e1, s));
  OP_CUDA(cudaEventSynchronize(e1));
  float ms = 0.f;
  OP_CUDA(cudaEventElapsedTime(&ms, e0, e1));
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  *us = ms * 1000.f / iters;
  int h = 0;
  OP_CUDA(cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost));
  if (h) return op_fail(PF_E_DEVICE_TIMEOUT, "GEMM gave up a bounded wait, code " + std::to_string(h));
  return PF_OK;
}

extern "C" int pfop_linear_wait_test(int32_t wtype, const void* w_host, int32_t N, int32_t K, int32_t bn,
                                     const void* a_dev, int32_t a_rows, int32_t M, float* out_dev,
                                     int32_t withhold_stage, void* stream) {
  if (!w_host || !a_dev || !out_dev || N < 1 || N % 4 || M < 1 || M > a_rows || (bn != 64 && bn != 128 && bn != 256))
    return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  WeightMat W;
  ActMat A;
  int rc;
  if ((rc = make_weight(sc, W, wtype, rows_of(w_host, N, K, wtype, bn), K, bn))) return rc;
  W.split = 1;  // no cluster: the withheld stage belongs to one CTA alone
  if ((rc = make_act(A, a_dev, a_rows, K))) return rc;
  EpiParams e;
  e.kind = EPI_F32;
  e.N = N;
  e.out_f32 = out_dev;
  e.ld_f32 = N;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = nullptr;
  OP_CUDA(sc.alloc(&err, 16));
  OP_CUDA(cudaMemsetAsync(err, 0, 16, s));
  OP_CUDA(launch_gemm(A, M, W, e, err, s, withhold_stage < 0 ? -1 : withhold_stage));
  OP_CUDA(cudaStreamSynchronize(s));
  int h = 0;
  OP_CUDA(cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost));
  if (h) return op_fail(PF_E_DEVICE_TIMEOUT, "GEMM gave up a bounded wait, code " + std::to_string(h));
  return PF_OK;
}

extern "C" int pfop_linear_resid(int32_t wtype, const void* w_host, int32_t N, int32_t K, const void* a_dev,
                                 int32_t a_rows, int32_t M, float* x_dev, void* xb_dev, void* stream) {
  if (!w_host || !a_dev || !x_dev || N < 32 || N % 32 || M < 1 || M > a_rows) return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  WeightMat W;
  ActMat A;
  int rc;
  if ((rc = make_weight(sc, W, wtype, rows_of(w_host, N, K, wtype, 128), K, 128))) return rc;
  if ((rc = make_act(A, a_dev, a_rows, K))) return rc;
  EpiParams e;
  e.kind = EPI_RESID;
  e.N = N;
  e.out_f32 = x_dev;
  e.ld_f32 = N;
  e.out_bf16 = static_cast<__nv_bfloat16*>(xb_dev);
  e.ld_bf16 = N;
  return run_gemm(sc, A, M, W, e, static_cast<cudaStream_t>(stream));
}

extern "C" int pfop_linear_glu(int32_t wtype, const void* wg_host, const void* wu_host, int32_t F, int32_t K,
                               int32_t act, const void* a_dev, int32_t a_rows, int32_t M, void* h_dev, void* stream) {
  if (!wg_host || !wu_host || !a_dev || !h_dev || F < 64 || F % 64 || M < 1 || M > a_rows)
    return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  WeightMat W;
  ActMat A;
  int rc;
  const size_t rb = rbytes(wtype, K);
  // tiles of 256 rows (128 gate + 128 up), of 192 for Q4_0 when F is a
  // multiple of 96 but not of 128, else of 128
  const int bn = F % 128 == 0 ? 256 : (wtype == PF_W_Q4_0 && F % 96 == 0) ? 192 : 128, half = bn / 2;
  std::vector<const void*> rows;
  for (int t = 0; t < F / half; ++t) {
    for (int i = 0; i < half; ++i) rows.push_back(static_cast<const uint8_t*>(wg_host) + (t * half + i) * rb);
    for (int i = 0; i < half; ++i) rows.push_back(static_cast<const uint8_t*>(wu_host) + (t * half + i) * rb);
  }
  if ((rc = make_weight(sc, W, wtype, rows, K, bn))) return rc;
  if ((rc = make_act(A, a_dev, a_rows, K))) return rc;
  EpiParams e;
  e.kind = EPI_GLU;
  e.N = F;
  e.out_bf16 = static_cast<__nv_bfloat16*>(h_dev);
  e.ld_bf16 = F;
  e.act = act ? 1 : 0;
  return run_gemm(sc, A, M, W, e, static_cast<cudaStream_t>(stream));
}

extern "C" int pfop_linear_ple(int32_t wtype, const void* w_host, int32_t P, int32_t K, const void* a_dev,
                               int32_t a_rows, int32_t M, const void* ple_dev, int32_t ple_stride, void* out_dev,
                               void* stream) {
  if (!w_host || !a_dev || !ple_dev || !out_dev || P < 32 || P % 32 || M < 1 || M > a_rows)
    return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  WeightMat W;
  ActMat A;
  int rc;
  if ((rc = make_weight(sc, W, wtype, rows_of(w_host, P, K, wtype, 128), K, 128))) return rc;
  if ((rc = make_act(A, a_dev, a_rows, K))) return rc;
  EpiParams e;
  e.kind = EPI_PLE;
  e.N = P;
  e.out_bf16 = static_cast<__nv_bfloat16*>(out_dev);
  e.ld_bf16 = P;
  e.ple = static_cast<const __nv_bfloat16*>(ple_dev);
  e.ple_stride = ple_stride;
  return run_gemm(sc, A, M, W, e, static_cast<cudaStream_t>(stream));
}

extern "C" int pfop_linear_qkv(int32_t wtype, const void* wq_host, const void* wk_host, const void* wv_host,
                               int32_t Hq, int32_t Hkv, int32_t hd, int32_t K, float rope_base, const void* a_dev,
                               int32_t a_rows, int32_t M, int32_t pos0, int32_t max_ctx, void* q_dev, void* kc_dev,
                               void* vc_dev, void* stream) {
  const bool kvw = wk_host && wv_host;
  if (!wq_host || !a_dev || !q_dev || (kvw && (!kc_dev || !vc_dev)) || (hd != 64 && hd != 256) || Hq < 1 || Hkv < 1 ||
      M < 1 || M > a_rows || pos0 < 0 || pos0 + M > max_ctx)
    return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  WeightMat W;
  ActMat A;
  int rc;
  const int q = Hq * hd, kv = Hkv * hd;
  const int bn = QKV_BN;
  std::vector<const void*> rows =
      qkv_tile_rows(wq_host, kvw ? wk_host : nullptr, kvw ? wv_host : nullptr, Hq, Hkv, hd, rbytes(wtype, K), bn);
  if ((rc = make_weight(sc, W, wtype, rows, K, bn))) return rc;
  if ((rc = make_act(A, a_dev, a_rows, K))) return rc;
  const int half = hd / 2;
  std::vector<float2> tab(static_cast<size_t>(pos0 + M) * half);
  for (int p = 0; p < pos0 + M; ++p)
    for (int i = 0; i < half; ++i) {
      const double th = static_cast<double>(p) * std::pow(static_cast<double>(rope_base), -2.0 * i / hd);
      tab[static_cast<size_t>(p) * half + i] = make_float2(static_cast<float>(std::cos(th)), static_cast<float>(std::sin(th)));
    }
  float2* rope = nullptr;
  OP_CUDA(sc.alloc(&rope, tab.size() * sizeof(float2)));
  OP_CUDA(cudaMemcpy(rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice));
  EpiParams e;
  e.kind = EPI_QKV;
  e.q_out = static_cast<__half*>(q_dev);
  e.k_cache = static_cast<__half*>(kc_dev);
  e.v_cache = static_cast<__half*>(vc_dev);
  e.q_dim = q;
  e.kv_dim = kvw ? kv : 0;
  e.head_dim = hd;
  e.pos0 = pos0;
  e.rope = rope;
  return run_gemm(sc, A, M, W, e, static_cast<cudaStream_t>(stream));
}

extern "C" int pfop_attention(int32_t mode, const void* q_dev, const void* k_dev, const void* v_dev, int32_t M,
                              int32_t Hq, int32_t Hkv, int32_t hd, int32_t pos_base, int32_t kv_len, void* out_dev,
                              void* stream) {
  if (!q_dev || !k_dev || !v_dev || !out_dev || M < 1 || Hq < 1 || Hkv < 1 || pos_base < 0 || pos_base + M > kv_len)
    return op_fail(PF_E_ARG, "bad argument");
  if (mode == 1 && M != 1) return op_fail(PF_E_ARG, "split mode takes one row");
  AttnArgs a;
  a.q = static_cast<const __half*>(q_dev);
  a.k = static_cast<const __half*>(k_dev);
  a.v = static_cast<const __half*>(v_dev);
  a.out = static_cast<__nv_bfloat16*>(out_dev);
  a.M = M;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.hd = hd;
  a.pos_base = pos_base;
  a.kv_len = kv_len;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Scope sc;
  float* part = nullptr;
  int* err = nullptr;
  OP_CUDA(sc.alloc(&part, (mode == 1 ? attn_split_partials_floats(Hq, Hkv, hd, pos_base)
                                     : attn_partials_floats(M, Hq, hd, kv_len)) * 4));
  OP_CUDA(sc.alloc(&err, 16));
  OP_CUDA(cudaMemsetAsync(err, 0, 16, s));
  if (mode == 1) OP_CUDA(cudaMemsetAsync(part, 0, attn_split_ticket_bytes(Hkv), s));  // the tickets start at zero
  a.err = err;
  if (mode == 0) {
    OP_CUDA(launch_attn_prefill(a, part, s));
  } else {
    OP_CUDA(launch_attn_split(a, part, s));
  }
  OP_CUDA(cudaStreamSynchronize(s));
  int h = 0;
  OP_CUDA(cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost));
  if (h) return op_fail(PF_E_DEVICE_TIMEOUT, "attention gave up a bounded wait, code " + std::to_string(h));
  return PF_OK;
}

extern "C" int pfop_rmsnorm(const float* x_dev, int32_t row0, int32_t M, int32_t D, const float* g_host, float eps,
                            void* y_dev, float* xcopy_dev, void* stream) {
  if (!x_dev || !g_host || !y_dev || M < 1 || D < 4 || D % 4 || row0 < 0) return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  float* g = nullptr;
  OP_CUDA(sc.alloc(&g, D * 4));
  OP_CUDA(cudaMemcpy(g, g_host, D * 4, cudaMemcpyHostToDevice));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  OP_CUDA(launch_rmsnorm(x_dev, row0, M, D, g, eps, static_cast<__nv_bfloat16*>(y_dev), xcopy_dev, s));
  OP_CUDA(cudaStreamSynchronize(s));
  return PF_OK;
}

extern "C" int pfop_embed(int32_t wtype, const void* tok_host, const void* ple_host, int32_t vocab, int32_t D,
                          int32_t LP, float ple_scale, const int32_t* tok_dev, int32_t T, float* x_dev, void* ple_dev,
                          void* stream) {
  if (!tok_host || !tok_dev || !x_dev || T < 1 || D < 32 || D % 32 || vocab < 1 ||
      (ple_host && (!ple_dev || LP % 32 || LP < 32)))
    return op_fail(PF_E_ARG, "bad argument");
  Scope sc;
  void* tt = nullptr;
  void* pt = nullptr;
  int* err = nullptr;
  OP_CUDA(sc.alloc(&tt, static_cast<size_t>(vocab) * rbytes(wtype, D)));
  OP_CUDA(cudaMemcpy(tt, tok_host, static_cast<size_t>(vocab) * rbytes(wtype, D), cudaMemcpyHostToDevice));
  if (ple_host) {
    OP_CUDA(sc.alloc(&pt, static_cast<size_t>(vocab) * rbytes(wtype, LP)));
    OP_CUDA(cudaMemcpy(pt, ple_host, static_cast<size_t>(vocab) * rbytes(wtype, LP), cudaMemcpyHostToDevice));
  }
  OP_CUDA(sc.alloc(&err, 16));
  OP_CUDA(cudaMemset(err, 0, 16));
  EmbedArgs a;
  a.tok = tok_dev;
  a.T = T;
  a.vocab = vocab;
  a.D = D;
  a.wq4 = wtype == PF_W_Q4_0;
  a.tok_table = tt;
  a.x = x_dev;
  a.ple_table = pt;
  a.LP = ple_host ? LP : 0;
  a.ple_scale = ple_scale;
  a.ple = static_cast<__nv_bfloat16*>(ple_dev);
  a.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  OP_CUDA(launch_embed(a, s));
  OP_CUDA(cudaStreamSynchronize(s));
  int h = 0;
  OP_CUDA(cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost));
  if (h == PF_DEV_BAD_TOKEN) return op_fail(PF_E_DEVICE_TOKEN, "token id outside [0, vocab)");
  return PF_OK;
}

namespace {
// the copy kernel moves 16-byte vectors on both sides
bool kv_copy_layout_ok(const void* cache, int64_t cache_seg_halves, const void* image, int64_t img_seg_bytes,
                       int64_t copy_bytes) {
  return ((reinterpret_cast<uintptr_t>(cache) | reinterpret_cast<uintptr_t>(image)) % 16) == 0 &&
         cache_seg_halves % 8 == 0 && img_seg_bytes % 16 == 0 && copy_bytes % 16 == 0;
}
}  // namespace

extern "C" int pfop_kv_copy(int32_t dir, void* cache_dev, int64_t cache_seg_halves, void* image_dev,
                            int64_t img_seg_bytes, int32_t n_seg, int64_t copy_bytes, const int32_t* header4,
                            void* stream) {
  if (!cache_dev || !image_dev || n_seg < 0 || copy_bytes < 0 || (dir != 0 && dir != 1))
    return op_fail(PF_E_ARG, "bad argument");
  if (!kv_copy_layout_ok(cache_dev, cache_seg_halves, image_dev, img_seg_bytes, copy_bytes))
    return op_fail(PF_E_ARG, "KV copy layout not 16-byte aligned");
  const int32_t zero[4] = {0, 0, 0, 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  OP_CUDA(launch_kv_copy(dir, static_cast<__half*>(cache_dev), cache_seg_halves, static_cast<uint8_t*>(image_dev),
                         img_seg_bytes, n_seg, copy_bytes, header4 ? header4 : zero, s));
  OP_CUDA(cudaStreamSynchronize(s));
  return PF_OK;
}

namespace {

// Mean device time of `iters` timed repetitions of `launch` on s, each
// bracketed by its own pair of events; with a scrub buffer, a memset of it
// runs before every repetition (outside the events) so that the timed
// kernels start with their operands evicted from L2.
template <class F>
int time_launches(F&& launch, void* scrub, int64_t scrub_bytes, int warmup, int iters, float* us, cudaStream_t s) {
  for (int i = 0; i < warmup; ++i) OP_CUDA(launch());
  std::vector<cudaEvent_t> ev(2 * static_cast<size_t>(iters), nullptr);
  struct Ev {
    std::vector<cudaEvent_t>& v;
    ~Ev() {
      for (cudaEvent_t e : v)
        if (e) cudaEventDestroy(e);
    }
  } guard{ev};
  for (auto& e : ev) OP_CUDA(cudaEventCreate(&e));
  for (int i = 0; i < iters; ++i) {
    if (scrub && scrub_bytes > 0) OP_CUDA(cudaMemsetAsync(scrub, i & 0xff, static_cast<size_t>(scrub_bytes), s));
    OP_CUDA(cudaEventRecord(ev[2 * i], s));
    OP_CUDA(launch());
    OP_CUDA(cudaEventRecord(ev[2 * i + 1], s));
  }
  OP_CUDA(cudaStreamSynchronize(s));
  double total = 0.0;
  for (int i = 0; i < iters; ++i) {
    float ms = 0.f;
    OP_CUDA(cudaEventElapsedTime(&ms, ev[2 * i], ev[2 * i + 1]));
    total += ms;
  }
  *us = static_cast<float>(total * 1000.0 / iters);
  return PF_OK;
}

}  // namespace

extern "C" int pfop_attention_bench(int32_t mode, const void* q_dev, const void* k_dev, const void* v_dev, int32_t M,
                                    int32_t Hq, int32_t Hkv, int32_t hd, int32_t pos_base, int32_t kv_len,
                                    void* out_dev, void* scrub_dev, int64_t scrub_bytes, int32_t warmup,
                                    int32_t iters, float* us, void* stream) {
  if (!q_dev || !k_dev || !v_dev || !out_dev || !us || M < 1 || Hq < 1 || Hkv < 1 || pos_base < 0 ||
      pos_base + M > kv_len || iters < 1 ||
      warmup < 0 || scrub_bytes < 0)
    return op_fail(PF_E_ARG, "bad argument");
  if (mode != 0 && mode != 1) return op_fail(PF_E_ARG, "mode");
  if (mode == 1 && M != 1) return op_fail(PF_E_ARG, "split mode takes one row");
  AttnArgs a;
  a.q = static_cast<const __half*>(q_dev);
  a.k = static_cast<const __half*>(k_dev);
  a.v = static_cast<const __half*>(v_dev);
  a.out = static_cast<__nv_bfloat16*>(out_dev);
  a.M = M;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.hd = hd;
  a.pos_base = pos_base;
  a.kv_len = kv_len;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Scope sc;
  float* part = nullptr;
  int* err = nullptr;
  OP_CUDA(sc.alloc(&part, (mode == 1 ? attn_split_partials_floats(Hq, Hkv, hd, pos_base)
                                     : attn_partials_floats(M, Hq, hd, kv_len)) * 4));
  OP_CUDA(sc.alloc(&err, 16));
  OP_CUDA(cudaMemsetAsync(err, 0, 16, s));
  if (mode == 1) OP_CUDA(cudaMemsetAsync(part, 0, attn_split_ticket_bytes(Hkv), s));  // the tickets start at zero
  a.err = err;
  int rc = time_launches([&] { return mode == 0 ? launch_attn_prefill(a, part, s) : launch_attn_split(a, part, s); },
                         scrub_dev, scrub_bytes, warmup, iters, us, s);
  if (rc) return rc;
  int h = 0;
  OP_CUDA(cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost));
  if (h) return op_fail(PF_E_DEVICE_TIMEOUT, "attention gave up a bounded wait, code " + std::to_string(h));
  return PF_OK;
}

extern "C" int pfop_kv_copy_bench(int32_t dir, void* cache_dev, int64_t cache_seg_halves, void* image_dev,
                                  int64_t img_seg_bytes, int32_t n_seg, int64_t copy_bytes, void* scrub_dev,
                                  int64_t scrub_bytes, int32_t warmup, int32_t iters, float* us, void* stream) {
  if (!cache_dev || !image_dev || !us || n_seg < 0 || copy_bytes < 0 || (dir != 0 && dir != 1) || iters < 1 ||
      warmup < 0 || scrub_bytes < 0)
    return op_fail(PF_E_ARG, "bad argument");
  if (!kv_copy_layout_ok(cache_dev, cache_seg_halves, image_dev, img_seg_bytes, copy_bytes))
    return op_fail(PF_E_ARG, "KV copy layout not 16-byte aligned");
  const int32_t hdr[4] = {0, 0, 0, 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return time_launches(
      [&] {
        return launch_kv_copy(dir, static_cast<__half*>(cache_dev), cache_seg_halves, static_cast<uint8_t*>(image_dev),
                              img_seg_bytes, n_seg, copy_bytes, hdr, s);
      },
      scrub_dev, scrub_bytes, warmup, iters, us, s);
}
