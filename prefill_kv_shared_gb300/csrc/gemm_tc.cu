// Dense GEMM on the 5th-generation tensor cores (tcgen05, TMEM accumulators)
// for the projections of the prefill pass: QKV, O, gate/up, down, the
// per-layer-embedding gate and projection, and the tied LM head.
//
//   out = A[M, K] (bf16, K-major) x W[N, K]^T, fp32 accumulation in TMEM.
//
// Weights are Q4_0 (32-element blocks, fp16 scale d, value d*(nibble-8)) or
// bf16.  Q4_0 tiles are fetched with one bulk copy per k-block and expanded
// to bf16 in shared memory by eight dequant warps, written directly in the
// 128-byte-swizzled K-major layout the MMA reads; A (and bf16 W) tiles come
// in by TMA with the same swizzle.
//
// CTA: 128*MT rows x BN columns, K in blocks of 64.
//   warp 0      TMA / bulk-copy producer (one lane issues)
//   warp 1      TMEM allocation, MMA issue (one lane), commits
//   warps 2..9  Q4_0 -> bf16 dequant per stage, then the fused epilogue
//               (TMEM -> registers -> global), 4 lane quarters x 2
//
// Determinism: every output element is produced by the same sequence of
// MMAs over k (64-wide blocks in ascending order, four K=16 steps each)
// whatever M is, so a row's result does not depend on how many rows the
// launch carries (M = 1 and M = 512 give bit-identical rows).
#include "common.cuh"
#include "kernels.h"

#include <cstring>
#include <mutex>

namespace pf {

constexpr int GEMM_THREADS = 320;

template <int WK, int BN, int MT>
struct GemmCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int RAW_BYTES = (WK == W_Q4) ? BN * 36 : 0;
  static constexpr int RAW_SLOT = (RAW_BYTES + 1023) / 1024 * 1024;
  static constexpr int STAGE_BYTES = MT * A_BYTES + B_BYTES + RAW_SLOT;
  static constexpr int SMEM_BUDGET = 232448 - 2048;
  static constexpr int STAGES_FIT = SMEM_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int ACC_COLS = MT * BN;
  static constexpr int TMEM_COLS = ACC_COLS <= 32 ? 32 : ACC_COLS <= 64 ? 64 : ACC_COLS <= 128 ? 128
                                                                      : ACC_COLS <= 256 ? 256 : 512;
  static_assert(STAGES >= 2, "shared memory too small for two stages");
  static_assert(ACC_COLS <= 512, "accumulators exceed TMEM");
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "MMA N");
};

// ---------------------------------------------------------------------------
// Q4_0 -> bf16

// bf16x2 with value 128 + n in each half, from nibbles in bits [0,4) and [16,20)
__device__ __forceinline__ uint32_t nib_pair_to_bf16x2_biased(uint32_t t) {
  uint32_t r;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(r) : "r"(t));  // (t & m) | c
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_scale(uint32_t biased, __nv_bfloat162 d2) {
  const __nv_bfloat162 c136 = __floats2bfloat162_rn(136.0f, 136.0f);
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&biased);
  v = __hmul2(__hsub2(v, c136), d2);  // (128 + n - 136) is exact; one rounding in the product
  return *reinterpret_cast<uint32_t*>(&v);
}

// One 32-element Q4_0 block (16 nibble bytes + fp16 scale) of row r -> four
// 16-byte chunks (8 bf16 each) of the swizzled row, chunks 4h .. 4h+3.
__device__ __forceinline__ void dequant_block32(uint4 nib, __half d, uint8_t* row_ptr, int h, int sw) {
  const __nv_bfloat16 db = __float2bfloat16_rn(__half2float(d));
  const __nv_bfloat162 d2 = __halves2bfloat162(db, db);
  const uint32_t w[4] = {nib.x, nib.y, nib.z, nib.w};
  uint32_t lo[8], hi[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t01 = __byte_perm(w[i], 0u, 0x4140);  // byte0 -> bits 0..7, byte1 -> bits 16..23
    const uint32_t t23 = __byte_perm(w[i], 0u, 0x4342);  // byte2, byte3
    lo[2 * i] = bf16x2_scale(nib_pair_to_bf16x2_biased(t01), d2);
    lo[2 * i + 1] = bf16x2_scale(nib_pair_to_bf16x2_biased(t23), d2);
    hi[2 * i] = bf16x2_scale(nib_pair_to_bf16x2_biased(t01 >> 4), d2);
    hi[2 * i + 1] = bf16x2_scale(nib_pair_to_bf16x2_biased(t23 >> 4), d2);
  }
  // elements 0..7 | 8..15 are the low nibbles of bytes 0..7 | 8..15,
  // elements 16..23 | 24..31 the high nibbles
  *reinterpret_cast<uint4*>(row_ptr + (((4 * h + 0) ^ sw) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  *reinterpret_cast<uint4*>(row_ptr + (((4 * h + 1) ^ sw) << 4)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  *reinterpret_cast<uint4*>(row_ptr + (((4 * h + 2) ^ sw) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(row_ptr + (((4 * h + 3) ^ sw) << 4)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
}

// ---------------------------------------------------------------------------
// epilogue helpers

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// store 32 packed 16-bit values (16 words) to a 16-byte aligned address
__device__ __forceinline__ void store32x16(void* dst, const uint32_t (&w)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

template <int BN>
__device__ __forceinline__ void epilogue(const EpiParams& ep, uint32_t tmem_acc, int m, bool row_ok,
                                         int n_tile, int ew) {
  constexpr int NCH = BN / 32;
  const int n0 = n_tile * BN;
  uint32_t v[32], u[32];
  if (ep.kind == EPI_GLU) {
    constexpr int HALF_CH = NCH / 2;
    for (int c = ew; c < HALF_CH; c += 2) {
      tmem_ld32(tmem_acc + 32 * c, v);
      tmem_ld32(tmem_acc + 32 * (c + HALF_CH), u);
      tmem_ld_wait();
      if (!row_ok) continue;
      const int f0 = n_tile * (BN / 2) + 32 * c;
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float g0 = u2f(v[2 * j]), g1 = u2f(v[2 * j + 1]);
        float a0 = ep.act == 0 ? gelu_tanh_f(g0) : silu_f(g0);
        float a1 = ep.act == 0 ? gelu_tanh_f(g1) : silu_f(g1);
        w[j] = pack_bf16x2(a0 * u2f(u[2 * j]), a1 * u2f(u[2 * j + 1]));
      }
      if (f0 + 32 <= ep.N) store32x16(ep.out_bf16 + (size_t)m * ep.ld_bf16 + f0, w);
    }
    return;
  }
  if (ep.kind == EPI_QKV) {
    const int hd = ep.head_dim, half = hd / 2, pair_ch = half / 32;
    const int q_end = ep.q_dim, k_end = ep.q_dim + ep.kv_dim, v_end = ep.q_dim + 2 * ep.kv_dim;
    const int pos = ep.pos0 + m;
    for (int c = ew; c < NCH; c += 2) {
      const int n = n0 + 32 * c;
      if (n >= v_end) break;  // padding columns (uniform across the warp)
      if (n >= k_end) {       // V: no rotation
        tmem_ld32(tmem_acc + 32 * c, v);
        tmem_ld_wait();
        if (!row_ok) continue;
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = pack_half2(u2f(v[2 * j]), u2f(v[2 * j + 1]));
        store32x16(ep.v_cache + (size_t)pos * ep.kv_dim + (n - k_end), w);
        continue;
      }
      const bool is_q = n < q_end;
      const int rel = is_q ? n : n - q_end;
      const int i0 = rel % hd;
      if (i0 >= half) continue;  // handled together with its partner chunk
      tmem_ld32(tmem_acc + 32 * c, v);
      tmem_ld32(tmem_acc + 32 * (c + pair_ch), u);
      tmem_ld_wait();
      if (!row_ok) continue;
      const int head = rel / hd;
      const float2* cs = ep.rope + (size_t)pos * half + i0;
      uint32_t w1[16], w2[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float2 c0 = cs[2 * j], c1 = cs[2 * j + 1];
        const float x0 = u2f(v[2 * j]), x1 = u2f(v[2 * j + 1]);
        const float y0 = u2f(u[2 * j]), y1 = u2f(u[2 * j + 1]);
        w1[j] = pack_half2(x0 * c0.x - y0 * c0.y, x1 * c1.x - y1 * c1.y);
        w2[j] = pack_half2(x0 * c0.y + y0 * c0.x, x1 * c1.y + y1 * c1.x);
      }
      __half* dst = is_q ? ep.q_out + (size_t)m * ep.q_dim + head * hd
                         : ep.k_cache + (size_t)pos * ep.kv_dim + head * hd;
      store32x16(dst + i0, w1);
      store32x16(dst + i0 + half, w2);
    }
    return;
  }
  // F32, RESID, PLE: one 32-column chunk at a time
  for (int c = ew; c < NCH; c += 2) {
    const int n = n0 + 32 * c;
    if (n >= ep.N) break;
    tmem_ld32(tmem_acc + 32 * c, v);
    tmem_ld_wait();
    if (!row_ok) continue;
    const bool full = n + 32 <= ep.N;
    if (ep.kind == EPI_F32) {
      float* dst = ep.out_f32 + (size_t)m * ep.ld_f32 + n;
      if (full) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          reinterpret_cast<float4*>(dst)[j] =
              make_float4(u2f(v[4 * j]), u2f(v[4 * j + 1]), u2f(v[4 * j + 2]), u2f(v[4 * j + 3]));
      } else {
        for (int j = 0; j < 32 && n + j < ep.N; ++j) dst[j] = u2f(v[j]);
      }
    } else if (ep.kind == EPI_RESID) {
      float* xr = ep.out_f32 + (size_t)m * ep.ld_f32 + n;
      float nv[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float4 x4 = reinterpret_cast<const float4*>(xr)[j];
        nv[4 * j] = x4.x + u2f(v[4 * j]);
        nv[4 * j + 1] = x4.y + u2f(v[4 * j + 1]);
        nv[4 * j + 2] = x4.z + u2f(v[4 * j + 2]);
        nv[4 * j + 3] = x4.w + u2f(v[4 * j + 3]);
        reinterpret_cast<float4*>(xr)[j] = make_float4(nv[4 * j], nv[4 * j + 1], nv[4 * j + 2], nv[4 * j + 3]);
      }
      if (ep.out_bf16) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(nv[2 * j], nv[2 * j + 1]);
        store32x16(ep.out_bf16 + (size_t)m * ep.ld_bf16 + n, w);
      }
    } else {  // EPI_PLE
      const __nv_bfloat16* pl = ep.ple + (size_t)m * ep.ple_stride + n;
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const __nv_bfloat162 p2 = reinterpret_cast<const __nv_bfloat162*>(pl)[j];
        w[j] = pack_bf16x2(gelu_tanh_f(u2f(v[2 * j])) * __low2float(p2),
                           gelu_tanh_f(u2f(v[2 * j + 1])) * __high2float(p2));
      }
      store32x16(ep.out_bf16 + (size_t)m * ep.ld_bf16 + n, w);
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel

// wait with a time limit but without giving up on another thread's error:
// used to let in-flight copies land before the CTA exits on an error path
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;  // 200 ms
  }
}

template <int WK, int BN, int MT>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ wq4, int M, int K, const __grid_constant__ EpiParams ep,
                   int* err) {
  using C = GemmCfg<WK, BN, MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* bready = empty + C::STAGES;
  uint64_t* accum = bready + C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x;
  const int m_base = blockIdx.y * (MT * 128);
  const int nkb = K / 64;
  int mt_valid = (M - m_base + 127) / 128;
  if (mt_valid > MT) mt_valid = MT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&bready[s], 8);
    }
    mbar_init(accum, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    if (WK == W_BF16) prefetch_tensormap(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- producer
    int issued = 0;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % C::STAGES;
      const uint32_t ph = (kb / C::STAGES) & 1;
      if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1, err, PF_DEV_TIMEOUT_PRODUCER);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        uint8_t* st = smem + s * C::STAGE_BYTES;
        const uint32_t tx = mt_valid * C::A_BYTES + (WK == W_BF16 ? C::B_BYTES : C::RAW_BYTES);
        mbar_arrive_expect_tx(&full[s], tx);
        for (int mt = 0; mt < mt_valid; ++mt)
          tma_load_2d(st + mt * C::A_BYTES, &tmA, &full[s], kb * 64, m_base + mt * 128);
        if (WK == W_BF16) {
          tma_load_2d(st + MT * C::A_BYTES, &tmB, &full[s], kb * 64, n_tile * BN);
        } else {
          bulk_load(st + MT * C::A_BYTES + C::B_BYTES, wq4 + ((size_t)n_tile * nkb + kb) * C::RAW_BYTES,
                    C::RAW_BYTES, &full[s]);
        }
      }
      __syncwarp();
      issued = kb + 1;
    }
    if (!ok && lane == 0) {
      // let the copies already issued land before shared memory goes away
      const int first = issued > C::STAGES ? issued - C::STAGES : 0;
      for (int kb = first; kb < issued; ++kb) mbar_drain(&full[kb % C::STAGES], (kb / C::STAGES) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue
    constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % C::STAGES;
      const uint32_t ph = (kb / C::STAGES) & 1;
      if (lane == 0) {
        ok = mbar_wait(&full[s], ph, err, PF_DEV_TIMEOUT_MMA);
        if (ok && WK == W_Q4) ok = mbar_wait(&bready[s], ph, err, PF_DEV_TIMEOUT_MMA);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint8_t* st = smem + s * C::STAGE_BYTES;
        const uint32_t a0 = smem_u32(st);
        const uint32_t b0 = smem_u32(st + MT * C::A_BYTES);
        for (int mt = 0; mt < mt_valid; ++mt) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sdesc_sw128(a0 + mt * C::A_BYTES + kk * 32);
            const uint64_t bd = sdesc_sw128(b0 + kk * 32);
            tc_mma_f16(tmem_base + mt * BN, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
        }
        tc_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(accum);  // fires once every MMA issued above has completed
    __syncwarp();
  } else {
    // ---------------- dequant, then epilogue
    const int t = threadIdx.x - 64;  // 0..255
    bool ok = true;
    if (WK == W_Q4) {
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % C::STAGES;
        const uint32_t ph = (kb / C::STAGES) & 1;
        const bool w_ok = mbar_wait(&full[s], ph, err, PF_DEV_TIMEOUT_DEQUANT);
        ok = __all_sync(0xffffffffu, w_ok);
        if (!ok) break;
        uint8_t* bt = smem + s * C::STAGE_BYTES + MT * C::A_BYTES;
        const uint8_t* raw = bt + C::B_BYTES;
#pragma unroll
        for (int it = t; it < BN * 2; it += 256) {
          const int r = it % BN, h = it / BN;
          const uint4 nib = *reinterpret_cast<const uint4*>(raw + (size_t)(h * BN + r) * 16);
          const __half d = *reinterpret_cast<const __half*>(raw + BN * 32 + (h * BN + r) * 2);
          dequant_block32(nib, d, bt + r * 128, h, r & 7);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bready[s]);
      }
    }
    bool acc_ok = ok ? mbar_wait(accum, 0, err, PF_DEV_TIMEOUT_EPILOGUE) : false;
    acc_ok = __all_sync(0xffffffffu, acc_ok);
    if (acc_ok) {
      tc_fence_after();
      const int qw = warp & 3;         // TMEM lane quarter this warp may access
      const int ew = (warp - 2) >> 2;  // which of the two warps on that quarter
      const int r = 32 * qw + lane;
      for (int mt = 0; mt < mt_valid; ++mt) {
        const int m = m_base + mt * 128 + r;
        const uint32_t tacc = tmem_base + (static_cast<uint32_t>(32 * qw) << 16) + mt * BN;
        epilogue<BN>(ep, tacc, m, m < M, n_tile, ew);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side

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
  return encode_2d_bf16(&a.tmap, a.dev, (uint64_t)a.K, (uint64_t)a.rows, 64, 128, err);
}

bool make_weight_map(WeightMat& w, std::string* err) {
  std::memset(&w.tmap, 0, sizeof(w.tmap));
  if (w.kind != W_BF16) return true;
  return encode_2d_bf16(&w.tmap, w.dev, (uint64_t)w.K, (uint64_t)w.N_rows, 64, (uint32_t)w.BN, err);
}

template <int WK, int BN, int MT>
static cudaError_t launch_t(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err,
                            cudaStream_t s) {
  using C = GemmCfg<WK, BN, MT>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_tc_kernel<WK, BN, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  dim3 grid(W.N_rows / BN, (M + MT * 128 - 1) / (MT * 128));
  gemm_tc_kernel<WK, BN, MT><<<grid, GEMM_THREADS, C::SMEM_BYTES, s>>>(
      A.tmap, W.tmap, static_cast<const uint8_t*>(W.dev), M, W.K, ep, err);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err,
                        cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (A.K != W.K || W.K % 64 != 0 || W.N_rows % W.BN != 0 || M > A.rows) return cudaErrorInvalidValue;
  const bool two = M > 128;
#define PF_GEMM_CASE(WKV, BNV)                                                    \
  if (W.kind == WKV && W.BN == BNV)                                               \
    return two ? launch_t<WKV, BNV, 2>(A, M, W, ep, err, s) : launch_t<WKV, BNV, 1>(A, M, W, ep, err, s);
  PF_GEMM_CASE(W_Q4, 128)
  PF_GEMM_CASE(W_Q4, 256)
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
