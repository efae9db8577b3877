/*
 * prefill.h -- C ABI of the KV-shared prompt-prefill library (GB300, sm_103a).
 *
 * What it computes.  The prompt-prefill forward pass of a decoder-only
 * transformer whose last layers are KV-shared:
 *   - layers il < n_layer_kv_from_start compute Q/K/V for every prompt row and
 *     write FP16 K/V into the KV cache;
 *   - layers il >= n_layer_kv_from_start write nothing and attend to the cache
 *     of an earlier layer (kv_src[il]); so, before the first such layer, the
 *     rows no output needs are pruned: an intermediate ubatch stops there and
 *     the final ubatch carries exactly one row (its last) through them.
 *   ("llama.cpp Gemma 4 prefill KV graph optimization", devotd.net news,
 *   section 1, with its listing of the pruning condition; outputs unchanged,
 *   end of section 3.)
 * The per-layer-embedding scaling (same page, section 1) is part of the pass,
 * and the FP16 KV cache can be saved to and restored from a "KVCP" image to
 * reuse a fixed system-prompt prefix ("PicoLM KV Cache persistence",
 * xxqk.cn news 668802, "usage", "file" and "rules" paragraphs).
 *
 * Model, per layer (pre-norm):  y = rmsnorm(x)*(1+g);  q,k,v = y W^T;
 * half-split RoPE on q,k;  o = causal GQA attention;  x += o Wo^T;
 * y = rmsnorm(x)*(1+g);  x += (act(y Wg^T) * (y Wu^T)) Wd^T  (act = GELU-tanh
 * or SiLU);  if ple_dim > 0:  x += (gelu(x Wpg^T) * ple[il]) Wpp^T, with
 * ple[il] = E_ple[token, il, :] / sqrt(ple_dim).  Logits = rmsnorm(x_last)*(1+g)
 * times the tied token-embedding matrix.
 *
 * Conventions.
 *   - Every call returns an int status: 0 = PF_OK, negative = PF_E_*.  No
 *     exception crosses the ABI; kernels never trap.  prefill_last_error()
 *     gives a message for the last failure on a context.
 *   - Device work is ordered on the stream given at create (or the legacy
 *     default stream when NULL).  prefill_ubatch, kv_save and kv_load return
 *     once the work is enqueued; prefill_sync() waits for it and reports a
 *     device-side error (a bad token, a timed-out pipeline wait).
 *   - A context holds one sequence, unless its description sets n_seq_max
 *     above 1 (then prefill_ubatch_seqs feeds several; see there).
 */
#ifndef PREFILL_KV_SHARED_H
#define PREFILL_KV_SHARED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define PF_OK 0
#define PF_E_ARG (-1)            /* bad argument, token, position or size */
#define PF_E_KV_MAGIC (-2)       /* KV image does not start with "KVCP" */
#define PF_E_KV_SHAPE (-3)       /* KV image layer count or kv_dim differs from the model */
#define PF_E_KV_RANGE (-4)       /* n_pos beyond the image or the context; image too short */
#define PF_E_CUDA (-5)           /* a CUDA call failed */
#define PF_E_DEVICE_TIMEOUT (-6) /* a kernel gave up a bounded wait; results are invalid */
#define PF_E_DEVICE_TOKEN (-7)   /* a device-resident token id was out of range */
#define PF_E_NOMEM (-8)          /* device memory exhausted (a cudaMalloc that failed for another reason is PF_E_CUDA) */
#define PF_E_IO (-9)             /* a KV image file could not be opened, read or written */

/* weight storage types */
#define PF_W_F32 0  /* fp32 matrices (computed as bf16 on the GPU) */
#define PF_W_Q4_0 2 /* Q4_0: 32-element blocks of 18 bytes: fp16 scale d (little
                       endian), 16 bytes; byte j = element j (low nibble), element
                       j+16 (high nibble); value d*(nibble-8) */

/* feed-forward gate activation */
#define PF_FFN_GEGLU 0  /* gelu_tanh(g) * u */
#define PF_FFN_SWIGLU 1 /* silu(g) * u */

typedef struct prefill_ctx prefill_ctx; /* opaque */

typedef struct prefill_model_desc {
  int32_t n_layer;
  int32_t n_layer_kv_from_start; /* first KV-shared layer (== n_layer: none) */
  int32_t d_model;
  int32_t n_head;
  int32_t n_head_kv;
  int32_t head_dim; /* 64 or 256 */
  int32_t ffn_dim;
  int32_t vocab;
  int32_t ple_dim; /* per-layer embedding width; 0 = no per-layer embeddings */
  int32_t ffn_kind;  /* PF_FFN_* */
  int32_t wtype;     /* PF_W_* for every matrix and embedding table */
  float rms_eps;
  float rope_base;
  const int32_t* kv_src; /* [n_layer]: -1 for writing layers, else the writing layer
                            whose cache the layer reads; copied at create */
  int32_t max_ctx;        /* positions the KV cache holds */
  int32_t ubatch_max;     /* largest n_tokens per prefill_ubatch */
  int32_t prune_shared_enable; /* 1: prune before the first KV-shared layer when the
                                  condition holds; 0: every row passes every layer */
  int32_t n_seq_max;      /* sequences sharing the context (1 .. 128; see
                             prefill_ubatch_seqs); the page's pruning needs 1 */
  int32_t embeddings;     /* nonzero: the embeddings output of every row is requested
                             (PF_OUT_EMBD of prefill_set_output; disables pruning) */
  const int32_t* embd_layer_inp; /* NULL, or [n_layer + 1] flags: nonzero at il requests the
                                    hidden state entering layer il for every row (il ==
                                    n_layer: the final hidden state, before the output
                                    norm); copied at create.  A request at any il >=
                                    n_layer_kv_from_start disables pruning. */
} prefill_model_desc;

/* host pointers; the library copies (and repacks) everything at create.
   Matrices are [out][in] row-major in the model's wtype; norm gains are fp32.
   Absent tensors (wk/wv of KV-shared layers, ple_* when ple_dim == 0) are NULL. */
typedef struct prefill_layer_weights {
  const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down, *ple_gate, *ple_proj;
} prefill_layer_weights;

typedef struct prefill_weights {
  const void* tok_embd; /* [vocab][d_model]; also the LM head (tied) */
  const void* ple_embd; /* [vocab][n_layer * ple_dim] or NULL */
  const void* out_norm; /* fp32 [d_model] */
  const prefill_layer_weights* layers; /* [n_layer] */
} prefill_weights;

/* Build a context on the current CUDA device.  (The model the pass runs:
   "llama.cpp Gemma 4 prefill KV graph optimization", section 1: writing
   layers below n_layer_kv_from_start, KV-shared layers from it up that
   read kv_src's cache; the pruning condition of that section's listing is
   evaluated from prune_shared_enable, n_seq_max and embeddings.)  Contexts of
   one process may sit on different devices (the kernels' shared-memory
   opt-in is made once per kernel and device); each context's calls must be
   made with its own device current.  Validates the description,
   uploads and repacks the weights, allocates the FP16 KV cache
   (2 x writing layers x max_ctx x kv_dim) and the activation buffers for
   ubatch_max rows.  cuda_stream: a cudaStream_t or NULL.  On failure *out is
   NULL, nothing stays allocated, and the status says why: PF_E_ARG for a
   description outside the supported shapes (head_dim 64 or 256, n_head /
   n_head_kv dividing 16, d_model / ffn_dim / ple_dim multiples of 64) or
   too large to index with 32-bit integers (ubatch_max rounded up to 128
   times the widest activation row, any weight matrix, or max_ctx x kv_dim
   reaching 2^31 elements; ubatch_max above 2^20; max_ctx above 2^26),
   checked before any CUDA call; PF_E_NOMEM when device memory runs out;
   PF_E_CUDA for any other CUDA failure. */
int prefill_create(const prefill_model_desc* desc, const prefill_weights* weights, void* cuda_stream,
                   prefill_ctx** out);

/* Run one ubatch of n_tokens tokens at positions pos0 .. pos0+n_tokens-1.
   ("llama.cpp Gemma 4 prefill KV graph optimization", section 1: every row
   passes the writing layers; before the first KV-shared layer the rows no
   output needs are dropped, so an intermediate ubatch stops there and the
   final ubatch carries only its last row through the KV-shared layers.)
   tokens: host memory (validated on the host: PF_E_ARG on an id outside
   [0, vocab)) or device memory (validated on the device: PF_E_DEVICE_TOKEN at
   prefill_sync).  pos0 must equal the context's position count (ubatches
   continue the sequence), and pos0 + n_tokens <= max_ctx, 1 <= n_tokens <=
   ubatch_max.  is_last: this ubatch ends the prompt; its last row's logits
   (fp32 [vocab]) are written to `logits`, which must then be device (or
   managed) memory, else PF_E_ARG, and may be NULL otherwise.  With pruning active, a non-final ubatch runs only the writing
   layers.  Enqueue only: call prefill_sync to wait. */
int prefill_ubatch(prefill_ctx* ctx, const int32_t* tokens, int32_t n_tokens, int64_t pos0, int32_t is_last,
                   float* logits);

/* Hidden-state outputs ("llama.cpp Gemma 4 prefill KV graph optimization",
   section 1 listing: with embeddings requested, or a per-layer input
   embedding requested for a layer from n_layer_kv_from_start up to the
   final state, every row is needed there and the pruning is off).
   which = PF_OUT_EMBD: the embeddings output, rmsnorm(final hidden
   state) * (1 + out_norm) of every row, fp32 [n_tokens][d_model]; needs
   desc.embeddings.  which = il in [0, n_layer]: the hidden state entering
   layer il (il == n_layer: the final one, before the output norm), fp32
   [n_tokens][d_model]; needs desc.embd_layer_inp[il].  dst: device memory
   with room for ubatch_max rows (each later ubatch writes its rows from
   dst[0]), or NULL to clear.  PF_E_ARG for an output the description did not
   request or a dst that is not device memory; prefill_ubatch refuses
   (PF_E_ARG) while a requested output has no buffer. */
#define PF_OUT_EMBD (-1)
int prefill_set_output(prefill_ctx* ctx, int32_t which, float* dst);

/* ---- several sequences in one ubatch (unified KV cache) ----
   ("llama.cpp Gemma 4 prefill KV graph optimization", section 5: the server
   setting, where several sequences share one KV cache and one batch.)  A
   context with n_seq_max > 1 gives every sequence q the cache cells
   [q * max_ctx, (q + 1) * max_ctx) of each writing layer, and its own
   position count.  A ubatch of several sequences is a list of runs: run k
   holds runs[k].n_tokens consecutive tokens of sequence runs[k].seq_id
   (each sequence at most once per ubatch, 0 <= seq_id < n_seq_max),
   continuing it at prefill_seq_n_pos(seq_id); tokens holds the runs'
   tokens one after another (host memory, validated on the host, or device
   memory), at most ubatch_max in all.  Every row attends only to its own
   sequence's cells.  A run with is_last nonzero ends its sequence's prompt:
   its last row's logits go to row j of `logits` (fp32 [n_last][vocab],
   device memory), j counting the is_last runs in order.
   The page's pruning condition asks for one sequence, so with several
   sequences it never holds; this call instead applies the variant the
   server setting would need when pruning is on (PF_PRUNE_ON) and the rest
   of the condition holds (a KV-shared split inside the model, no embeddings
   or per-layer hidden-state outputs): before the first KV-shared layer only
   the output rows (one per is_last run) are kept.  Pruned and unpruned
   (PF_PRUNE_OFF) calls give bit-identical logits.  Enqueue only.
   PF_E_ARG for a bad run list, positions past max_ctx, more than
   ubatch_max tokens, or a missing/host logits buffer when a run ends. */
typedef struct prefill_seq_run {
  int32_t seq_id;
  int32_t n_tokens;
  int32_t is_last;
} prefill_seq_run;
int prefill_ubatch_seqs(prefill_ctx* ctx, const int32_t* tokens, const prefill_seq_run* runs, int32_t n_runs,
                        float* logits);

/* Positions of sequence seq_id in the cache (-1 for a bad id); forget one
   sequence (prefill_reset forgets all of them).  prefill_n_pos, kv_save and
   kv_load work on sequence 0. */
int64_t prefill_seq_n_pos(const prefill_ctx* ctx, int32_t seq_id);
int prefill_seq_reset(prefill_ctx* ctx, int32_t seq_id);

/* ---- a recorded ubatch (CUDA graph) ----
   prefill_graph_capture records one prefill_ubatch call (same arguments;
   tokens must be device memory) into a CUDA graph held by the context,
   without running it; prefill_graph_launch replays it on the context's
   stream.  A replay computes what the recorded call computes for the
   current contents of the tokens buffer: the same positions (pos0 ..
   pos0 + n_tokens - 1), the same logits buffer, the pruning mode and
   outputs in force when it was recorded; it needs the context's position
   count to be pos0 (PF_E_ARG otherwise) and advances it like the call.
   The ubatch's few hundred kernel launches become one graph launch.
   Recording needs a context created on a non-default stream and per-launch
   timing off; the launch counts of prefill_get_stats do not include
   replays.  A new recording replaces the previous one. */
int prefill_graph_capture(prefill_ctx* ctx, const int32_t* tokens, int32_t n_tokens, int64_t pos0, int32_t is_last,
                          float* logits);
int prefill_graph_launch(prefill_ctx* ctx);

/* Wait for the context's stream and report device-side errors. */
int prefill_sync(prefill_ctx* ctx);

/* Positions currently in the cache. */
int64_t prefill_n_pos(const prefill_ctx* ctx);

/* Forget the sequence (position count 0; with several sequences, all of
   them); the cache memory is kept.  (The
   fallback of "PicoLM KV Cache persistence", "rules": a request whose
   prefix cannot be restored starts from an empty cache.) */
int prefill_reset(prefill_ctx* ctx);

/* Switch pruning on or off for later ubatches (the A/B switch); the pruning
   condition itself still has to hold.  prefill_prune_active() says whether
   ubatches are pruned with the current settings.
     PF_PRUNE_ON:        prune when the condition holds (the default when the
                         description's prune_shared_enable is nonzero);
     PF_PRUNE_OFF:       every row passes every layer; in the KV-shared layers
                         of the final ubatch the output row takes the same
                         single-row kernels as with pruning, so its logits are
                         bit-identical to the pruned pass's;
     PF_PRUNE_OFF_PLAIN: every row passes every layer through the prefill
                         kernels (the fastest unpruned pass; the output row's
                         logits then differ from the pruned pass's in
                         rounding).
   Any other value is PF_E_ARG. */
#define PF_PRUNE_OFF 0
#define PF_PRUNE_ON 1
#define PF_PRUNE_OFF_PLAIN 2
int prefill_set_prune(prefill_ctx* ctx, int32_t enable);
int prefill_prune_active(const prefill_ctx* ctx);

/* Size in bytes of a KV image of n_pos positions for this model:
   16-byte header + 2 * writing_layers * n_pos * kv_dim * 2.  ("PicoLM KV
   Cache persistence", "file": a header, then the FP16 keys and values of
   the cached positions of every layer; 25 positions of a 22-layer,
   kv_dim-256 model are about 550 KB.)  -1 for a NULL context or n_pos < 0. */
int64_t prefill_kv_image_bytes(const prefill_ctx* ctx, int64_t n_pos);

/* ("PicoLM KV Cache persistence", "usage" and "file": after the prompt
   prefix has been prefilled its FP16 cache is saved, to be restored by
   later runs with the same prefix; "rules": only prompt positions are
   saved, never generated ones.)
   Write the cache's first prefill_n_pos() positions as a KV image to dst
   (device or host memory, 16-byte aligned, dst_bytes >= the image size).
   Image: "KVCP", int32 n_pos, int32 writing layers, int32 kv_dim (little
   endian), then FP16 keys [layer][pos][kv_dim], then FP16 values.  Only
   prompt positions are ever in the cache. */
int kv_save(prefill_ctx* ctx, void* dst, size_t dst_bytes);

/* ("PicoLM KV Cache persistence", "usage": a saved prefix is restored and
   its positions are skipped by the next prefill; "rules": the image must
   match the model's layers and kv_dim, the restored count may not exceed
   the image or the context, and a refused image means a full prefill.)
   Restore the first n_pos positions of a KV image (device or host memory; a
   device image 16-byte aligned, else PF_E_ARG) and set the position count
   to n_pos; the next ubatch continues at n_pos.  A
   wrong magic (PF_E_KV_MAGIC), a layer/kv_dim mismatch (PF_E_KV_SHAPE), or
   n_pos beyond the image's positions or max_ctx (PF_E_KV_RANGE) is refused
   and leaves the cache and position count unchanged: the caller then runs a
   full prefill.  Whether the image was made from the same prompt prefix is
   the caller's contract (the image stores no tokens). */
int kv_load(prefill_ctx* ctx, const void* src, size_t src_bytes, int64_t n_pos);

/* ---- KV image files (PicoLM KV cache article, "usage" and "file") ----
   A file holds exactly one KV image (the layout above).  kv_save_file
   writes the cache's first prefill_n_pos() positions to `path` (created or
   replaced; PF_E_IO when the file cannot be written).  kv_load_file checks
   the file's header against this model and the file's size first
   (PF_E_IO: cannot open or read; PF_E_KV_MAGIC / PF_E_KV_SHAPE /
   PF_E_KV_RANGE: as kv_load) and only then restores its first n_pos
   positions (n_pos < 0: all of them); any refusal leaves the cache and the
   position count unchanged, so the caller falls back to a full prefill.
   Both are synchronous and stage the image through host memory. */
int kv_save_file(prefill_ctx* ctx, const char* path);
int kv_load_file(prefill_ctx* ctx, const char* path, int64_t n_pos);

/* Host-only check of a KV image file against a model (writing layers,
   kv_dim) and a context length: PF_OK and *n_pos_out = the file's position
   count, or the refusal kv_load_file would give.  No GPU needed. */
int prefill_kv_file_check(const char* path, int32_t n_layers_written, int32_t kv_dim, int64_t max_ctx,
                          int64_t* n_pos_out);

/* ---- launch accounting and per-class kernel timing ----
   Every kernel the context launches is counted by class, with the
   algorithmic work it does (FLOPs: 2*M*N*K for a projection, 4*hd per
   (query head, visible key) for attention; bytes: what the step must move
   at least).  With timing on, each launch is bracketed by CUDA events on
   the context's stream (this adds host overhead; use it on a separate run
   from throughput measurements). */
#define PF_KC_GEMM 0      /* projections of launches with more than 16 rows (tcgen05, tensor-bound) */
#define PF_KC_ATTN 1      /* prefill attention and its group-state merge */
#define PF_KC_NORM 2      /* RMSNorm (+ row gather) */
#define PF_KC_OTHER 3     /* embedding gather, KV image copies */
#define PF_KC_GEMM_ROW 4  /* projections of at most 16 rows: the one-row stream projections of the output row and
                           of one-token ubatches, the LM head (weight-bound) */
#define PF_KC_ATTN_ROW 5  /* the single-row attention: the output row in the KV-shared layers, every layer of a
                           one-token ubatch (HBM-bound) */
#define PF_KC_COUNT 6

typedef struct prefill_stats {
  int64_t launches[PF_KC_COUNT];
  double flops[PF_KC_COUNT];
  double bytes[PF_KC_COUNT];
  int64_t timed[PF_KC_COUNT]; /* launches with event timing */
  double ms[PF_KC_COUNT];     /* summed device time of the timed launches */
} prefill_stats;

int prefill_set_timing(prefill_ctx* ctx, int32_t enable);
/* Waits for the stream when timing is on; fills *out with the totals since
   the last prefill_reset_stats. */
int prefill_get_stats(prefill_ctx* ctx, prefill_stats* out);
int prefill_reset_stats(prefill_ctx* ctx);

/* Free the context: waits for its stream, then releases the weights, the
   KV cache and every buffer it holds.  NULL is ignored.  (The library's
   own resource handling; the pages describe no counterpart.) */
void prefill_destroy(prefill_ctx* ctx);

/* Message of the last failed call on ctx (or, with ctx NULL, of the last
   failed prefill_create on this thread).  The returned string stays valid
   until the next call on the same context. */
const char* prefill_last_error(const prefill_ctx* ctx);

/* ---- host-only helpers (no GPU needed) ---- */

/* The pruning condition for a description (n_seq_max == 1, no embeddings,
   no embd_layer_inp request at a layer from n_layer_kv_from_start to
   n_layer, 0 < n_layer_kv_from_start < n_layer, pruning enabled).  Returns 1
   or 0, or PF_E_ARG for a NULL description. */
int prefill_prune_predicate(const prefill_model_desc* desc);

/* Validate a 16-byte KV image header against a model (writing layers, kv_dim),
   a requested n_pos, the context length and the image size.  Returns PF_OK or
   PF_E_KV_MAGIC / PF_E_KV_SHAPE / PF_E_KV_RANGE. */
int prefill_kv_header_check(const void* header16, int32_t n_layers_written, int32_t kv_dim, int64_t n_pos,
                            int64_t max_ctx, size_t image_bytes);

/* 16 + 2 * n_layers_written * n_pos * kv_dim * 2, or -1 on negative input. */
int64_t prefill_kv_image_bytes_for(int32_t n_layers_written, int64_t n_pos, int32_t kv_dim);

#ifdef __cplusplus
}
#endif

#endif /* PREFILL_KV_SHARED_H */
