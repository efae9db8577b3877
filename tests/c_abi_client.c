/* A plain C99 client of the library's C ABI (include/prefill.h), built and
   run by tests/test_library_host.py: the header is usable from C without
   any Python or C++ in between, and the host-only calls answer as the
   pages fix them.  With the argument "nogpu" it also checks that creating a
   context on a machine without a GPU fails with a status and a message
   instead of falling back to a host path.  Exit status 0 = every check held;
   otherwise the number of the first failed check. */
#include <stdio.h>
#include <string.h>

#include "prefill.h"

static void put_le32(unsigned char* p, int32_t v) {
  uint32_t u = (uint32_t)v;
  p[0] = (unsigned char)(u & 0xFF);
  p[1] = (unsigned char)((u >> 8) & 0xFF);
  p[2] = (unsigned char)((u >> 16) & 0xFF);
  p[3] = (unsigned char)((u >> 24) & 0xFF);
}

int main(int argc, char** argv) {
  /* "PicoLM KV Cache persistence", "file": 25 positions of a 22-layer model
     with kv_dim 256 in FP16 keys and values, about 550 KB, plus the header */
  const int64_t bytes = prefill_kv_image_bytes_for(22, 25, 256);
  if (bytes != 16 + 2 * 22 * 25 * 256 * 2) return 1;
  if (prefill_kv_image_bytes_for(22, -1, 256) != -1) return 2;

  /* the pruning condition of "llama.cpp Gemma 4 prefill KV graph
     optimization", section 1 listing, on an E2B-shaped description */
  int32_t kv_src[24];
  for (int il = 0; il < 24; ++il) kv_src[il] = il < 16 ? -1 : (il % 2 == 0 ? 14 : 15);
  prefill_model_desc d;
  memset(&d, 0, sizeof d);
  d.n_layer = 24;
  d.n_layer_kv_from_start = 16;
  d.d_model = 1536;
  d.n_head = 8;
  d.n_head_kv = 1;
  d.head_dim = 256;
  d.ffn_dim = 6144;
  d.vocab = 32768;
  d.ple_dim = 256;
  d.ffn_kind = PF_FFN_GEGLU;
  d.wtype = PF_W_Q4_0;
  d.rms_eps = 1e-6f;
  d.rope_base = 10000.0f;
  d.kv_src = kv_src;
  d.max_ctx = 512;
  d.ubatch_max = 512;
  d.prune_shared_enable = 1;
  d.n_seq_max = 1;
  if (prefill_prune_predicate(&d) != 1) return 3;
  d.n_seq_max = 2;
  if (prefill_prune_predicate(&d) != 0) return 4;
  d.n_seq_max = 1;
  d.embeddings = 1;
  if (prefill_prune_predicate(&d) != 0) return 5;
  d.embeddings = 0;
  int32_t layer_inp[25];
  memset(layer_inp, 0, sizeof layer_inp);
  layer_inp[15] = 1; /* below the first KV-shared layer: pruning still holds */
  d.embd_layer_inp = layer_inp;
  if (prefill_prune_predicate(&d) != 1) return 6;
  layer_inp[24] = 1; /* the final hidden state of every row */
  if (prefill_prune_predicate(&d) != 0) return 7;
  d.embd_layer_inp = NULL;
  if (prefill_prune_predicate(NULL) != PF_E_ARG) return 8;

  /* KV image header ("PicoLM KV Cache persistence", "file" and "rules") */
  unsigned char h[16];
  memcpy(h, "KVCP", 4);
  put_le32(h + 4, 25);
  put_le32(h + 8, 22);
  put_le32(h + 12, 256);
  if (prefill_kv_header_check(h, 22, 256, 25, 2048, (size_t)bytes) != PF_OK) return 9;
  if (prefill_kv_header_check(h, 22, 256, 26, 2048, (size_t)bytes) != PF_E_KV_RANGE) return 10;
  if (prefill_kv_header_check(h, 22, 256, 25, 24, (size_t)bytes) != PF_E_KV_RANGE) return 11;
  if (prefill_kv_header_check(h, 22, 256, 25, 2048, (size_t)bytes - 1) != PF_E_KV_RANGE) return 12;
  if (prefill_kv_header_check(h, 16, 256, 25, 2048, (size_t)bytes) != PF_E_KV_SHAPE) return 13;
  h[3] = 'Q';
  if (prefill_kv_header_check(h, 22, 256, 25, 2048, (size_t)bytes) != PF_E_KV_MAGIC) return 14;

  if (argc > 1 && strcmp(argv[1], "nogpu") == 0) {
    /* a complete 2-layer fp32 model (layer 0 writes, layer 1 reads it), so
       that only the missing device can stop the create */
    static float zeros[64 * 64];
    int32_t src2[2] = {-1, 0};
    prefill_model_desc t;
    memset(&t, 0, sizeof t);
    t.n_layer = 2;
    t.n_layer_kv_from_start = 1;
    t.d_model = 64;
    t.n_head = 1;
    t.n_head_kv = 1;
    t.head_dim = 64;
    t.ffn_dim = 64;
    t.vocab = 8;
    t.ffn_kind = PF_FFN_SWIGLU;
    t.wtype = PF_W_F32;
    t.rms_eps = 1e-6f;
    t.rope_base = 10000.0f;
    t.kv_src = src2;
    t.max_ctx = 16;
    t.ubatch_max = 16;
    t.prune_shared_enable = 1;
    t.n_seq_max = 1;
    prefill_layer_weights lw[2];
    for (int il = 0; il < 2; ++il) {
      lw[il].attn_norm = lw[il].wq = lw[il].wo = lw[il].ffn_norm = zeros;
      lw[il].w_gate = lw[il].w_up = lw[il].w_down = zeros;
      lw[il].wk = lw[il].wv = il == 0 ? zeros : NULL;
      lw[il].ple_gate = lw[il].ple_proj = NULL;
    }
    prefill_weights w;
    w.tok_embd = zeros;
    w.ple_embd = NULL;
    w.out_norm = zeros;
    w.layers = lw;
    prefill_ctx* ctx = (prefill_ctx*)&t; /* must be overwritten with NULL */
    const int rc = prefill_create(&t, &w, NULL, &ctx);
    if (rc != PF_E_CUDA) return 15;
    if (ctx != NULL) return 16;
    const char* msg = prefill_last_error(NULL);
    if (!msg || !msg[0]) return 17;
    printf("create without a GPU: status %d (%s)\n", rc, msg);
  }
  printf("ok\n");
  return 0;
}
