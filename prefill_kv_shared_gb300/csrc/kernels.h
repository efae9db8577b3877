// Host-side declarations of the CUDA kernels' launchers and the data layouts
// they share with the runtime.  Internal to the library (not part of the
// C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

namespace pf {

// ---------------------------------------------------------------------------
// GEMM: out = A[M, K] (bf16, row-major) x W[N, K]^T, fused epilogues

enum WKind : int { W_BF16 = 0, W_Q4 = 1 };

enum EpiKind : int {
  EPI_F32 = 0,    // out_f32[m, n] = acc
  EPI_RESID = 1,  // out_f32[m, n] += acc; if out_bf16: out_bf16[m, n] = bf16(new value)
  EPI_GLU = 2,    // W rows interleaved per tile (gate half, up half):
                  //   out_bf16[m, f] = act(gate) * up
  EPI_QKV = 3,    // columns [0,q) Q, [q,q+kv) K, [q+kv,q+2kv) V; RoPE on Q and K;
                  //   Q -> q_out fp16 [m][q], K/V -> fp16 cache rows at pos0+m
  EPI_PLE = 4,    // out_bf16[m, n] = bf16(gelu_tanh(acc) * ple[m*ple_stride + n])
};

struct EpiParams {
  int kind = EPI_F32;
  int N = 0;  // logical output columns (GLU: ffn dim)
  float* out_f32 = nullptr;
  int ld_f32 = 0;
  __nv_bfloat16* out_bf16 = nullptr;
  int ld_bf16 = 0;
  const __nv_bfloat16* ple = nullptr;
  int ple_stride = 0;
  int act = 0;  // GLU: 0 = gelu_tanh, 1 = silu
  __half* q_out = nullptr;
  __half* k_cache = nullptr;  // row p = position p, kv_dim halves per row
  __half* v_cache = nullptr;
  int q_dim = 0, kv_dim = 0, head_dim = 0;
  int pos0 = 0;                  // position of GEMM row 0
  const float2* rope = nullptr;  // [position][head_dim/2] = (cos, sin)
  // rows of several sequences in one launch: row m's position (RoPE angle)
  // and its K/V cache row; null: pos0 + m for both
  const int* row_pos = nullptr;
  const int* row_slot = nullptr;
};

// A weight matrix in device memory, in the GEMM's tile order.
//  W_BF16: bf16 [N_rows][K] row-major (rows already in tile order), TMA-read.
//  W_Q4:   tiles (n-tile t, k-block kb) at byte (t*nkb + kb) * BN*36:
//          [half h][row r] 16 nibble bytes, then [half h][row r] fp16 scales,
//          where half h is the Q4_0 block of k in [64kb+32h, 64kb+32h+32).
struct WeightMat {
  int kind = W_Q4;
  int N_rows = 0;  // stored rows (multiple of BN)
  int K = 0;
  int BN = 128;
  int split = 1;   // k-splits (fixed per matrix shape; K/64 divisible by it)
  int pair = 0;    // 1: launches run in 2-CTA clusters sharing 256-row MMAs (Q4_0 only, split 1)
  void* dev = nullptr;
  size_t bytes = 0;
  CUtensorMap tmap;
};

// A bf16 activation matrix used as the GEMM's A operand.
struct ActMat {
  const __nv_bfloat16* dev = nullptr;
  int rows = 0, K = 0;
  CUtensorMap tmap;        // 128-row boxes
  CUtensorMap tmap_small;  // 16-row boxes, for launches of at most 16 rows
  CUtensorMap tmap_wide;   // 256-row boxes: two 128-row M tiles in one copy
};

bool make_act_map(ActMat& a, std::string* err);
// fp16 tensor map with the 128-byte swizzle (rank 2..5; strides of dims 1..)
bool encode_fp16_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, std::string* err);
bool make_weight_map(WeightMat& w, std::string* err);

// k-splits (cluster size) for a weight shape, chosen from the shape and the
// largest M the context runs; never from a launch's M
int choose_split(int kind, int N_rows, int BN, int K, int max_rows);
// 1 if the matrix's launches run in CTA pairs (tcgen05 .cta_group::2),
// chosen like the split; a matrix with a k-split never does
int choose_pair(int kind, int N_rows, int BN, int K, int max_rows, int split);
// Q|K|V weight rows in GEMM tile order (128-row tiles; heads wider than a
// tile are cut so that RoPE pairs share a tile; V in plain order), padded to
// BN with NULL rows.  wk/wv may be NULL (a Q-only projection).
constexpr int QKV_BN = 128;
std::vector<const void*> qkv_tile_rows(const void* wq, const void* wk, const void* wv, int Hq, int Hkv, int hd,
                                       size_t row_bytes, int BN);

// withhold_stage >= 0 only in the failure-path check (pfop_linear_wait_test):
// CTA 0's copy producer issues nothing from that pipeline stage on.
cudaError_t launch_gemm(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err_word,
                        cudaStream_t s, int withhold_stage = -1);
// the one-unit launches of launch_gemm (Q4_0, every CTA one work unit);
// two: two 128-row M tiles per unit
cudaError_t launch_gemm_solo(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err_word,
                             cudaStream_t s, int withhold_stage, bool two);
// whether a split's partial tiles fit the one-unit form's A ring (they must
// stay clear of its epilogue staging in the B ring)
bool gemm_solo_fits(int BN, bool two, int split);
// the CTA-pair launches of launch_gemm (W.pair set); two: two 256-row MMA
// tiles per pair
cudaError_t launch_gemm_pair(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err_word,
                             cudaStream_t s, int withhold_stage, bool two);

// One row (a one-token ubatch): out = A[0] W^T with the same fused epilogue,
// streamed by CUDA cores over (tile, k-part) CTAs, the k-parts of a tile
// one thread-block cluster (no scratch memory).  err: device error word (a
// weight copy that never lands flags it after the bounded wait).  With
// norm_x (fp32 [K], 16-byte aligned) the row is not read from A: it is the
// RMS norm of norm_x with gain (1 + norm_g) and eps, formed inside the
// launch and rounded to bf16.
cudaError_t launch_gemv(const ActMat& A, const WeightMat& W, const EpiParams& ep, int* err, cudaStream_t s,
                        const float* norm_x = nullptr, const float* norm_g = nullptr, float eps = 0.f);

// Host repack.  `rows[i]` points at the i-th stored row's source (Q4_0: K/32
// blocks of 18 bytes; F32: K floats) or is null for a zero padding row.
std::vector<uint8_t> repack_q4_tiles(const std::vector<const uint8_t*>& rows, int K, int BN);
std::vector<uint16_t> repack_bf16_rows(const std::vector<const float*>& rows, int K);

// ---------------------------------------------------------------------------
// attention (fp16 Q and KV cache, fp32 accumulation, 64-key chunks)

struct AttnArgs {
  const __half* q = nullptr;  // [M][Hq*hd]
  const __half* k = nullptr;  // [position][Hkv*hd]
  const __half* v = nullptr;
  __nv_bfloat16* out = nullptr;  // [M][Hq*hd]
  int M = 0, Hq = 0, Hkv = 0, hd = 0;
  int pos_base = 0;  // position of row 0
  int kv_len = 0;    // keys [0, kv_len) exist in the cache
  int* err = nullptr;  // device error word (bounded waits that give up set it)
};

// Causal attention over (64-row block, chunk group) CTAs; rows whose keys span
// several groups go through the partials buffer (attn_partials_floats) and an
// ordered merge.  launch_attn_split is the single-row form of the KV-shared
// layers (M == 1, position pos_base, keys [0, pos_base]): key ranges spread
// over clusters of CTAs, one launch; `partials` holds
// attn_split_partials_floats floats (enough for any position up to the one
// it was sized for), whose first attn_split_ticket_bytes bytes are tickets
// that must be zero before the first launch (each launch leaves them zero).
cudaError_t launch_attn_prefill(const AttnArgs& a, float* partials, cudaStream_t s);
cudaError_t launch_attn_split(const AttnArgs& a, float* partials, cudaStream_t s);
// floats of partials a launch of M rows over kv_len keys needs (0: none)
size_t attn_partials_floats(int M, int Hq, int hd, int kv_len);
size_t attn_split_partials_floats(int Hq, int Hkv, int hd, int pos);
size_t attn_split_ticket_bytes(int Hkv);
int attn_group_chunks(int kv_len, int row_ctas);  // row_ctas: (128-row block, KV head) pairs
int attn_launch_count(const AttnArgs& a);  // kernels launch_attn_prefill starts (1 or 2)

// ---------------------------------------------------------------------------
// per-row kernels

struct EmbedArgs {
  const int32_t* tok = nullptr;
  int T = 0, vocab = 0, D = 0;
  int wq4 = 1;
  const void* tok_table = nullptr;  // Q4_0 rows [V][D/32][18] or f32 [V][D]
  float* x = nullptr;               // [T][D]
  const void* ple_table = nullptr;  // Q4_0 rows [V][LP/32][18] or f32 [V][LP] (null: none)
  int LP = 0;
  float ple_scale = 1.0f;
  __nv_bfloat16* ple = nullptr;  // [T][LP]
  int* err = nullptr;
};
cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t s);

// y[i] = rmsnorm(x[r_i]) * (1 + g) for i < M as bf16 (y) and/or fp32 (y32),
// r_i = rows[i] when rows is given, else row0 + i; optionally x_copy[i] =
// x[r_i].  Null outputs are skipped.
cudaError_t launch_rmsnorm(const float* x, int row0, int M, int D, const float* g, float eps,
                           __nv_bfloat16* y, float* x_copy, cudaStream_t s, float* y32 = nullptr,
                           const int* rows = nullptr);

// dst[i] = src[rows[i]] for i < n, rows of row_bytes bytes (a multiple of 16,
// both bases 16-byte aligned)
cudaError_t launch_gather_rows(const void* src, void* dst, const int* rows, int n, size_t row_bytes, cudaStream_t s);

// KV image body <-> cache.  n_seg segments (keys of each writing layer, then
// values); each copies copy_bytes, from/to the cache at seg * cache_seg_stride
// halves and the image body (16 bytes after `image`) at seg * img_seg_bytes.
// dir 0: cache -> image (also writes the 16-byte header), dir 1: image -> cache.
cudaError_t launch_kv_copy(int dir, __half* cache, int64_t cache_seg_stride, uint8_t* image, int64_t img_seg_bytes,
                           int n_seg, int64_t copy_bytes, const int32_t header[4], cudaStream_t s);

// message returned by pfop_last_error() on this thread
void set_op_error(const std::string& m);

}  // namespace pf
