/*
 * prefill_ops.h -- per-kernel entry points of the KV-shared prefill library.
 *
 * Each call runs ONE of the library's CUDA kernels (the same launchers the
 * prefill pass uses) on caller-provided device buffers, waits for it, and
 * returns a status (PF_OK or a negative PF_E_* from prefill.h).  They exist
 * so that every step of the pass can be checked on its own against a
 * reference.  Weights are passed as host pointers and uploaded for the call.
 * Calls are synchronous on `stream` (a cudaStream_t or NULL).
 *
 * Matrices are row-major.  bf16/fp16 buffers hold raw 16-bit values.  The A
 * operand of every GEMM (a_dev, bf16 [a_rows][K]) must have a_rows >= 128
 * rows allocated (rows beyond M are read but their results are dropped) and
 * K a multiple of 64.
 */
#ifndef PREFILL_OPS_H
#define PREFILL_OPS_H

#include <stdint.h>

#include "prefill.h"

#ifdef __cplusplus
extern "C" {
#endif

/* out[m][n] = sum_k A[m][k] W[n][k] (fp32 [M][N]); W [N][K] in wtype
   (PF_W_Q4_0 blocks or fp32, computed as bf16).  bn: N-tile, 64, 128 or 256
   (192 with Q4_0). */
int pfop_linear_f32(int32_t wtype, const void* w_host, int32_t N, int32_t K, int32_t bn, const void* a_dev,
                    int32_t a_rows, int32_t M, float* out_dev, void* stream);

/* x[m][n] += (A W^T)[m][n] (fp32 [M][N], in place); if xb_dev != NULL also
   xb[m][n] = bf16(new x[m][n]).  N must be a multiple of 32. */
int pfop_linear_resid(int32_t wtype, const void* w_host, int32_t N, int32_t K, const void* a_dev, int32_t a_rows,
                      int32_t M, float* x_dev, void* xb_dev, void* stream);

/* h[m][f] = act(A Wg^T)[m][f] * (A Wu^T)[m][f] (bf16 [M][F]); act 0 =
   gelu_tanh (GeGLU), 1 = silu (SwiGLU).  F a multiple of 64.  Gate and up
   rows are interleaved in tiles of 256 rows when F is a multiple of 128, of
   192 (Q4_0) when F is a multiple of 96, else of 128. */
int pfop_linear_glu(int32_t wtype, const void* wg_host, const void* wu_host, int32_t F, int32_t K, int32_t act,
                    const void* a_dev, int32_t a_rows, int32_t M, void* h_dev, void* stream);

/* out[m][p] = bf16(gelu_tanh((A W^T)[m][p]) * ple[m*ple_stride + p]) (bf16
   [M][P]); ple bf16.  P a multiple of 32 (the per-layer-embedding gate). */
int pfop_linear_ple(int32_t wtype, const void* w_host, int32_t P, int32_t K, const void* a_dev, int32_t a_rows,
                    int32_t M, const void* ple_dev, int32_t ple_stride, void* out_dev, void* stream);

/* Q/K/V projection with half-split RoPE at positions pos0+m (angle
   pos * base^(-2i/hd), i < hd/2, pairing i with i+hd/2):
   q_out fp16 [M][Hq*hd]; if wk_host/wv_host are not NULL, K (rotated) and V
   go to the fp16 caches kc/vc [max_ctx][Hkv*hd] at rows pos0+m. */
int pfop_linear_qkv(int32_t wtype, const void* wq_host, const void* wk_host, const void* wv_host, int32_t Hq,
                    int32_t Hkv, int32_t hd, int32_t K, float rope_base, const void* a_dev, int32_t a_rows,
                    int32_t M, int32_t pos0, int32_t max_ctx, void* q_dev, void* kc_dev, void* vc_dev, void* stream);

/* Causal GQA attention: q fp16 [M][Hq*hd] at positions pos_base+m, K/V fp16
   [positions][Hkv*hd] with keys [0, kv_len) valid; out bf16 [M][Hq*hd].
   mode 0: any M.  The (query row, query head of a KV head's group) pairs
   form 128-row blocks; keys are folded in 64-key chunks, the chunks in at
   most four groups (as many as keep the launch to one wave of CTAs, at
   least four chunks a group); one CTA per (row block, KV head, group),
   then an ordered merge of the group states of rows whose keys span
   several groups.
   mode 1: one row (M == 1) at position pos_base, the form the KV-shared
   layers use for the output row (G4 section 1: after the pruning those
   layers carry that row only): the keys [0, pos_base] are cut into 64-key
   tiles and the tiles into ranges over up to 144 CTAs in clusters of four;
   each CTA streams its range once (online softmax, fp32 accumulation), a
   cluster folds its four range states in rank order, and the last cluster
   of each KV head merges the cluster states in cluster order, all in one
   launch.  Its bits depend on pos_base only, not on the launch; they differ
   from mode 0's in rounding. */
int pfop_attention(int32_t mode, const void* q_dev, const void* k_dev, const void* v_dev, int32_t M, int32_t Hq,
                   int32_t Hkv, int32_t hd, int32_t pos_base, int32_t kv_len, void* out_dev, void* stream);

/* y[i] = bf16(rmsnorm(x[row0+i]) * (1 + g)) for i < M (x fp32 [.][D]); if
   xcopy_dev != NULL, xcopy[i] = x[row0+i]. */
int pfop_rmsnorm(const float* x_dev, int32_t row0, int32_t M, int32_t D, const float* g_host, float eps, void* y_dev,
                 float* xcopy_dev, void* stream);

/* x[t] = E[tok_t] (fp32 [T][D]); if ple_host != NULL, ple[t] = bf16(E_ple[tok_t] *
   ple_scale) (bf16 [T][LP]).  Tables in wtype.  tok_dev: int32 device. */
int pfop_embed(int32_t wtype, const void* tok_host, const void* ple_host, int32_t vocab, int32_t D, int32_t LP,
               float ple_scale, const int32_t* tok_dev, int32_t T, float* x_dev, void* ple_dev, void* stream);

/* The KV image copy kernel.  dir 0: cache -> image (writes the 16-byte header
   `header`, then n_seg segments of copy_bytes); dir 1: image -> cache.
   Segment s is at s*cache_seg_halves halves in the cache and at
   16 + s*img_seg_bytes bytes in the image.  The kernel moves 16-byte
   vectors: cache_dev and image_dev 16-byte aligned, cache_seg_halves a
   multiple of 8, img_seg_bytes and copy_bytes multiples of 16, else
   PF_E_ARG (checked before any CUDA call). */
int pfop_kv_copy(int32_t dir, void* cache_dev, int64_t cache_seg_halves, void* image_dev, int64_t img_seg_bytes,
                 int32_t n_seg, int64_t copy_bytes, const int32_t* header4, void* stream);

/* out[n] = sum_k a[k] W[n][k] (fp32 [N]) for ONE row a (bf16 [K]) with the
   one-token projection kernel that a one-token ubatch uses (generation
   after the prompt): CUDA cores stream W once (wtype as in pfop_linear_f32,
   bn its tile width: 64, 128, 256, or 192 for Q4_0), fp32 dot products,
   k-part sums added in a fixed order.  If iters > 0 the call is then repeated `iters` times and *us
   receives the mean device time per launch (CUDA events on `stream`). */
int pfop_linear_row(int32_t wtype, const void* w_host, int32_t N, int32_t K, int32_t bn, const void* a_dev,
                    float* out_dev, int32_t iters, float* us, void* stream);

/* Check of the failure path of the bounded waits (the library's own error
   convention; the pages have no counterpart).  Runs the GEMM of
   pfop_linear_f32 (no k-split) with the copy producer of CTA 0 issuing
   nothing from pipeline stage `withhold_stage` on, so no copy is left in
   flight for the tensor-core and dequantisation warps that wait for that
   stage: their waits give up after their bound (about 2 s of SM clock),
   every warp unwinds (copies already issued are drained, TMEM is freed), and
   the call returns PF_E_DEVICE_TIMEOUT with the GPU context still usable.
   withhold_stage < 0 (or past the CTA's last stage) runs the plain GEMM and
   returns PF_OK.  Synchronous on `stream`. */
int pfop_linear_wait_test(int32_t wtype, const void* w_host, int32_t N, int32_t K, int32_t bn, const void* a_dev,
                          int32_t a_rows, int32_t M, float* out_dev, int32_t withhold_stage, void* stream);

/* Time the GEMM kernel: upload W once, run `warmup` then `iters` launches of
   out = A W^T (fp32 [M][N]) and return the mean device time per launch in
   *us (CUDA events on `stream`).  split: k-splits on single CTAs (0 = the
   library's choice for this shape; -1 = no split, 2-CTA pairs sharing
   256-row tcgen05 MMAs, Q4_0 with bn 128, 192 or 256 only).  bn 192 takes
   Q4_0 weights only. */
int pfop_linear_bench(int32_t wtype, const void* w_host, int32_t N, int32_t K, int32_t bn, int32_t split,
                      const void* a_dev, int32_t a_rows, int32_t M, float* out_dev, int32_t warmup, int32_t iters,
                      float* us, void* stream);

/* Time the attention kernels of pfop_attention (same arguments and modes):
   `warmup` untimed calls, then `iters` timed ones, each bracketed by its own
   CUDA events on `stream`; *us = mean device time per call (the single-row
   kernel, or the prefill kernel plus the group-state merge when it runs).  If scrub_dev is
   not NULL, scrub_bytes of it (a caller-owned device buffer larger than L2)
   are overwritten before every timed call, outside the events, so that each
   call reads K/V from HBM (cold L2).  Reading K/V once is the op's
   algorithmic traffic: kv_len * Hkv * hd * 2 bytes for each of K and V.
   Returns PF_E_DEVICE_TIMEOUT if a bounded wait gave up. */
int pfop_attention_bench(int32_t mode, const void* q_dev, const void* k_dev, const void* v_dev, int32_t M, int32_t Hq,
                         int32_t Hkv, int32_t hd, int32_t pos_base, int32_t kv_len, void* out_dev, void* scrub_dev,
                         int64_t scrub_bytes, int32_t warmup, int32_t iters, float* us, void* stream);

/* Time the KV image copy kernel of pfop_kv_copy (same layout arguments and
   alignment rules; the image header written by dir 0 is all zeros here)
   like pfop_attention_bench: mean device time per launch in *us, optional
   L2 scrub of scrub_dev before every timed launch.  The copy reads and
   writes n_seg * copy_bytes bytes each. */
int pfop_kv_copy_bench(int32_t dir, void* cache_dev, int64_t cache_seg_halves, void* image_dev, int64_t img_seg_bytes,
                       int32_t n_seg, int64_t copy_bytes, void* scrub_dev, int64_t scrub_bytes, int32_t warmup,
                       int32_t iters, float* us, void* stream);

/* The single-row split-K attention of pfop_attention (mode 1) without any
   memory allocation, for callers that may not allocate device memory at this
   point (a fixed memory budget already handed out, a server that forbids
   allocation after start-up, an embedder whose allocator owns the device).
   The page set this library follows has no counterpart for this call.
   q fp16 [Hq*hd] at position pos; K/V fp16 [positions][Hkv*hd] with keys
   [0, kv_len) valid, pos < kv_len; out bf16 [Hq*hd].
   Scratch: one fixed device array of 2^19 floats (2 MiB) per GPU that loads
   the library, kept until exit.  A call needs the merge tickets (Hkv ints,
   rounded up to 4) and Hkv*C*(Hq/Hkv*hd + 32) floats of folded states, C
   being the clusters of four key ranges per KV head (at most 36/Hkv, at
   least 1), plus 4 for an error word: any shape of up to 1024 query heads
   of 256 fits; larger requests return PF_E_ARG without touching the GPU,
   and so do
   shapes the kernels do not take (head_dim other than 64 or 256, n_head not
   a multiple of n_head_kv, a group size not dividing 16, q/k/v not 16-byte
   aligned).  All calls share the array, so calls that overlap on the GPU
   race: order them on one stream or with events.  Each call clears the
   tickets it uses.  The first call on a device looks up the array's device
   address with that device current (cudaGetSymbolAddress); make that first
   call before capturing any stream.  Synchronous on `stream`. */
int pfop_attention_split_noalloc(const void* q_dev, const void* k_dev, const void* v_dev, int32_t Hq, int32_t Hkv,
                                 int32_t hd, int32_t pos, int32_t kv_len, void* out_dev, void* stream);

/* How the GEMMs of the pfop_* calls run (process-wide, for every later
   call): 0 = as the library picks per matrix shape (the default), 1 = every
   Q4_0 matrix with 128-, 192- or 256-row tiles in 2-CTA pairs (tcgen05
   .cta_group::2, no k-split), -1 = never in pairs.  Lets the same checks run
   on both forms; no effect on prefill contexts.  PF_E_ARG for other modes. */
int pfop_set_gemm_pairs(int32_t mode);

/* ---- host-only: the stored form of the weights (no GPU needed) ----
   The library repacks every matrix at create into the order and layout its
   kernels read; these two calls return that form so that it can be checked
   on its own.

   pfop_qkv_row_order: the stored row order of a layer's Q|K|V projection
   (128-row tiles).  order[i] = the source row of stored row i, counting
   rows of [Wq; Wk; Wv] (Wq: Hq*hd rows, then Wk and Wv: Hkv*hd rows each;
   with_kv = 0: a Q-only projection), or -1 for a zero row padding the last
   tile.  A Q or K head wider than a tile is cut into hd/128 tiles: tile j
   of the head holds dims j*64 .. j*64+63 of each half of the head, so that
   every RoPE pair (i, i + hd/2) lies in one tile; narrower heads and V rows
   stay in order.  Returns the number of stored
   rows (a multiple of 128), or PF_E_ARG (hd odd, hd above 128 and not a
   multiple of it, cap too small).

   pfop_repack_q4: a Q4_0 matrix [N][K] (K a multiple of 64) in tiles of bn
   rows (64, 128, 192 or 256; N padded with zero rows to a multiple of bn).
   Tile (t, kb), for t < ceil(N/bn) and 64-wide k-block kb < K/64, is bn*36
   contiguous bytes at ((t * K/64) + kb) * bn*36: first the 16 nibble bytes
   of 32-element block h (h = 0, 1: elements kb*64 + h*32 ..) of row r at
   (h*bn + r)*16, then that block's fp16 scale at bn*32 + (h*bn + r)*2.
   Padding rows hold nibble bytes 0x88 and scale 0 (value 0).  With dst NULL
   returns the byte count; otherwise writes it to dst (host memory,
   dst_bytes at least that) and returns it; PF_E_ARG for bad shapes. */
int32_t pfop_qkv_row_order(int32_t Hq, int32_t Hkv, int32_t hd, int32_t with_kv, int32_t* order, int32_t cap);
int64_t pfop_repack_q4(const void* w_host, int32_t N, int32_t K, int32_t bn, void* dst, int64_t dst_bytes);

/* Last error message of a pfop_* call on this thread. */
const char* pfop_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PREFILL_OPS_H */
