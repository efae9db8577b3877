// Host side of the tensor-core GEMM (the kernel and its configurations are
// in gemm_tc.cuh): tensor maps, the k-split and CTA-pair choices, the QKV
// tile order, launch dispatch for single CTAs (one-unit launches in
// gemm_solo.cu, CTA pairs in gemm_pair.cu), and the host repack of weights
// into tile order.
#include "gemm_tc.cuh"

namespace pf {

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                      CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);

static PFN_encodeTiled_t get_encode_fn(std::string* err) {
  static PFN_encodeTiled_t fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled_t>(p);
  });
  if (!fn && err) *err = "cuTensorMapEncodeTiled is not available";
  return fn;
}

bool encode_fp16_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, std::string* err) {
  PFN_encodeTiled_t enc = get_encode_fn(err);
  if (!enc) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st,
                   b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")";
    return false;
  }
  return true;
}

static bool encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                           uint32_t box_outer, std::string* err) {
  PFN_encodeTiled_t enc = get_encode_fn(err);
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")";
    return false;
  }
  return true;
}

bool make_act_map(ActMat& a, std::string* err) {
  if (a.K % 64 != 0) {
    if (err) *err = "GEMM K must be a multiple of 64";
    return false;
  }
  std::memset(&a.tmap, 0, sizeof(a.tmap));
  std::memset(&a.tmap_small, 0, sizeof(a.tmap_small));
  std::memset(&a.tmap_wide, 0, sizeof(a.tmap_wide));
  return encode_2d_bf16(&a.tmap, a.dev, (uint64_t)a.K, (uint64_t)a.rows, 64, 128, err) &&
         encode_2d_bf16(&a.tmap_small, a.dev, (uint64_t)a.K, (uint64_t)a.rows, 64, 16, err) &&
         encode_2d_bf16(&a.tmap_wide, a.dev, (uint64_t)a.K, (uint64_t)a.rows, 64, 256, err);
}

bool make_weight_map(WeightMat& w, std::string* err) {
  std::memset(&w.tmap, 0, sizeof(w.tmap));
  if (w.kind != W_BF16) return true;
  return encode_2d_bf16(&w.tmap, w.dev, (uint64_t)w.K, (uint64_t)w.N_rows, 64, (uint32_t)w.BN, err);
}

static size_t ring_bytes_mt1(int kind, int BN) {
  if (kind == W_Q4)
    return BN == 256   ? ring_bytes<W_Q4, 256, 1>()
           : BN == 192 ? ring_bytes<W_Q4, 192, 1>()
           : BN == 64  ? ring_bytes<W_Q4, 64, 1>()
                       : ring_bytes<W_Q4, 128, 1>();
  return BN == 256 ? ring_bytes<W_BF16, 256, 1>() : BN == 64 ? ring_bytes<W_BF16, 64, 1>() : ring_bytes<W_BF16, 128, 1>();
}

int choose_split(int kind, int N_rows, int BN, int K, int max_rows) {
  // Split the k-range over a cluster of 2 CTAs while the split tile grid
  // (one 128-row block per tile) still fits on the SMs at once, each part
  // keeps at least 4 k-blocks, and rank 0's ring holds the other rank's
  // partial tile.  (A 3-way split of the 1536 x 6144 down projection, which
  // also fits one wave, made the E2B pass slower.)  Depends on the matrix
  // shape and the context's largest ubatch only, never on a launch's M.
  const int units1 = (N_rows / BN) * ((max_rows + 127) / 128);
  const int nkb = K / 64;
  const size_t ring = ring_bytes_mt1(kind, BN);
  // Matrices with very few output tiles (the 256-row per-layer-embedding
  // gate: 16 units at 512 rows) are bound by the length of each CTA's
  // k-loop, not by tile counts: they take a 4-way split when it fits.
  if (units1 <= 16 && units1 * 4 <= sm_count() && nkb % 4 == 0 && nkb / 4 >= 4 &&
      static_cast<size_t>(3) * 128 * BN * 4 <= ring)
    return 4;
  if (units1 * 2 <= sm_count() && nkb % 2 == 0 && nkb / 2 >= 4 && static_cast<size_t>(128) * BN * 4 <= ring) return 2;
  return 1;
}

int choose_pair(int kind, int N_rows, int BN, int K, int max_rows, int split) {
  // CTA pairs halve each SM's B-operand traffic, dequant work and MMA
  // instructions, but on GB300 every measured projection shape (E2B and E4B
  // QKV, O, gate/up, down at 512 and 1024 rows) ran 15-55 % slower in pairs
  // than on single CTAs: the main loop waits on operand latency, not on B
  // traffic, and a pair adds a cross-SM hop to every stage.  The library
  // therefore never picks them; pfop_set_gemm_pairs runs them on request.
  (void)kind;
  (void)N_rows;
  (void)BN;
  (void)K;
  (void)max_rows;
  (void)split;
  return 0;
}

std::vector<const void*> qkv_tile_rows(const void* wq, const void* wk, const void* wv, int Hq, int Hkv, int hd,
                                       size_t row_bytes, int BN) {
  std::vector<const void*> rows;
  auto region = [&](const void* w, int heads, bool rotated) {
    const uint8_t* b = static_cast<const uint8_t*>(w);
    if (!rotated || hd <= BN) {
      for (int n = 0; n < heads * hd; ++n) rows.push_back(b + n * row_bytes);
      return;
    }
    // heads wider than a tile: tile j of a head holds dims j*BN/2 .. +BN/2 of
    // each half, so that every RoPE pair (i, i + hd/2) stays in one tile
    const int half = hd / 2, per = BN / 2;
    for (int h = 0; h < heads; ++h)
      for (int j = 0; j < hd / BN; ++j) {
        for (int i = 0; i < per; ++i) rows.push_back(b + (size_t)(h * hd + j * per + i) * row_bytes);
        for (int i = 0; i < per; ++i) rows.push_back(b + (size_t)(h * hd + half + j * per + i) * row_bytes);
      }
  };
  region(wq, Hq, true);
  if (wk) region(wk, Hkv, true);
  if (wv) region(wv, Hkv, false);
  rows.resize((rows.size() + BN - 1) / BN * BN, nullptr);
  return rows;
}

cudaError_t launch_gemm(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err, cudaStream_t s,
                        int withhold_stage) {
  if (M <= 0) return cudaSuccess;
  if (A.K != W.K || W.K % 64 != 0 || W.N_rows % W.BN != 0 || M > A.rows || W.split < 1 ||
      (W.K / 64) % W.split != 0)
    return cudaErrorInvalidValue;
  // two 128-row M tiles per CTA for large M on wide tiles, and on narrower
  // tiles when one M tile per CTA would need a second wave of CTAs (not in
  // split mode, whose partial slots hold one); otherwise one M tile, so
  // that more CTAs share the work.  A row's result does not depend on it.
  const int units_one = (W.N_rows / W.BN) * ((M + 127) / 128);
  const bool two = M > 128 && W.split == 1 && (W.BN >= 192 || (W.BN == 128 && units_one > sm_count()));
  if (W.pair) {
    // CTA pairs: 256-row MMA tiles; two of them per pair when one would need
    // a second wave of pairs
    if (W.kind != W_Q4 || W.split != 1) return cudaErrorInvalidValue;
    const int units_pair = (W.N_rows / W.BN) * ((M + 255) / 256);
    return launch_gemm_pair(A, M, W, ep, err, s, withhold_stage, M > 256 && units_pair > sm_count() / 2);
  }
  if (W.kind == W_Q4) {
    // one work unit per CTA: the epilogue stages in the B ring, and the A
    // ring gets the room (gemm_solo.cu)
    const int unit_rows = two ? 256 : 128;
    const int units = (W.N_rows / W.BN) * ((M + unit_rows - 1) / unit_rows) * W.split;
    if (units <= sm_count() && gemm_solo_fits(W.BN, two, W.split))
      return launch_gemm_solo(A, M, W, ep, err, s, withhold_stage, two);
  }
#define PF_GEMM_CASE(WKV, BNV)                                                        \
  if (W.kind == WKV && W.BN == BNV)                                                   \
    return two ? launch_t<WKV, BNV, 2, false>(A, M, W, ep, err, s, withhold_stage)   \
               : launch_t<WKV, BNV, 1, false>(A, M, W, ep, err, s, withhold_stage);
  PF_GEMM_CASE(W_Q4, 64)
  PF_GEMM_CASE(W_Q4, 128)
  PF_GEMM_CASE(W_Q4, 192)
  PF_GEMM_CASE(W_Q4, 256)
  PF_GEMM_CASE(W_BF16, 64)
  PF_GEMM_CASE(W_BF16, 128)
  PF_GEMM_CASE(W_BF16, 256)
#undef PF_GEMM_CASE
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// repack

std::vector<uint8_t> repack_q4_tiles(const std::vector<const uint8_t*>& rows, int K, int BN) {
  const int n_rows = static_cast<int>(rows.size());
  const int n_tiles = n_rows / BN;
  const int nkb = K / 64;
  const size_t tile_bytes = static_cast<size_t>(BN) * 36;
  std::vector<uint8_t> out(static_cast<size_t>(n_tiles) * nkb * tile_bytes, 0);
  for (int t = 0; t < n_tiles; ++t) {
    for (int kb = 0; kb < nkb; ++kb) {
      uint8_t* tile = out.data() + (static_cast<size_t>(t) * nkb + kb) * tile_bytes;
      for (int h = 0; h < 2; ++h) {
        for (int r = 0; r < BN; ++r) {
          const uint8_t* src = rows[static_cast<size_t>(t) * BN + r];
          uint8_t* nib = tile + (static_cast<size_t>(h) * BN + r) * 16;
          uint8_t* sc = tile + static_cast<size_t>(BN) * 32 + (static_cast<size_t>(h) * BN + r) * 2;
          if (!src) {
            std::memset(nib, 0x88, 16);  // nibble 8 -> value 0
            sc[0] = sc[1] = 0;
            continue;
          }
          const uint8_t* blk = src + static_cast<size_t>(2 * kb + h) * 18;
          sc[0] = blk[0];
          sc[1] = blk[1];
          std::memcpy(nib, blk + 2, 16);
        }
      }
    }
  }
  return out;
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return static_cast<uint16_t>((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

std::vector<uint16_t> repack_bf16_rows(const std::vector<const float*>& rows, int K) {
  std::vector<uint16_t> out(rows.size() * static_cast<size_t>(K), 0);
  for (size_t i = 0; i < rows.size(); ++i) {
    if (!rows[i]) continue;
    for (int k = 0; k < K; ++k) out[i * K + k] = f32_to_bf16_rne(rows[i][k]);
  }
  return out;
}

}  // namespace pf
