// Per-row kernels of the prefill pass and the KV image copies.
//
//  embed    x[t] = E[tok_t] (fp32, exact Q4_0 decode) and the per-layer
//           embeddings ple[t] = E_ple[tok_t] * (1/sqrt(P)) (bf16), written
//           once as [T][L*P]; each layer reads its [P] slice through a strided
//           view, with no contiguous copy (Gemma 4 prefill news, section 1:
//           per-layer embedding scaling, no contiguous copies).
//  rmsnorm  y = x / sqrt(mean(x^2) + eps) * (1 + g) -> bf16, optionally
//           gathering rows (the output-row gather before the first KV-shared
//           layer) and copying the gathered fp32 residual rows.  One CTA per
//           row with a fixed thread->element map and reduction tree, so a
//           row's result does not depend on how many rows are normalised.
//  kv_copy  KV image body <-> cache segments (PicoLM KV cache article, "file"
//           paragraph: FP16 keys of the first N positions, then the values).
#include "common.cuh"
#include "kernels.h"

namespace pf {

// ---------------------------------------------------------------------------
// embed

__device__ __forceinline__ void decode_q4_block(const uint8_t* blk, float (&out)[32]) {
  const uint16_t dbits = static_cast<uint16_t>(blk[0]) | (static_cast<uint16_t>(blk[1]) << 8);
  const float d = __half2float(__ushort_as_half(dbits));
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int b = blk[2 + j];
    out[j] = d * static_cast<float>((b & 0x0F) - 8);
    out[j + 16] = d * static_cast<float>((b >> 4) - 8);
  }
}

__global__ void __launch_bounds__(128) embed_kernel(EmbedArgs a) {
  pdl_launch();
  pdl_wait();
  const int t = blockIdx.x;
  int tok = a.tok[t];
  if (tok < 0 || tok >= a.vocab) {
    if (threadIdx.x == 0) set_error(a.err, PF_DEV_BAD_TOKEN);
    tok = 0;
  }
  // token row -> x (fp32)
  if (a.wq4) {
    const int nb = a.D / 32;
    const uint8_t* row = static_cast<const uint8_t*>(a.tok_table) + (size_t)tok * nb * 18;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
      float v[32];
      decode_q4_block(row + (size_t)b * 18, v);
      float4* dst = reinterpret_cast<float4*>(a.x + (size_t)t * a.D + b * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(a.tok_table) + (size_t)tok * a.D);
    float4* dst = reinterpret_cast<float4*>(a.x + (size_t)t * a.D);
    for (int i = threadIdx.x; i < a.D / 4; i += blockDim.x) dst[i] = src[i];
  }
  if (!a.ple_table) return;
  // per-layer embeddings -> ple (bf16), scaled
  __nv_bfloat16* prow = a.ple + (size_t)t * a.LP;
  if (a.wq4) {
    const int nb = a.LP / 32;
    const uint8_t* row = static_cast<const uint8_t*>(a.ple_table) + (size_t)tok * nb * 18;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
      float v[32];
      decode_q4_block(row + (size_t)b * 18, v);
      uint4* dst = reinterpret_cast<uint4*>(prow + b * 32);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * j + 2 * k] * a.ple_scale, v[8 * j + 2 * k + 1] * a.ple_scale);
          w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  } else {
    const float* src = static_cast<const float*>(a.ple_table) + (size_t)tok * a.LP;
    for (int i = threadIdx.x; i < a.LP / 2; i += blockDim.x) {
      const float2 v = reinterpret_cast<const float2*>(src)[i];
      reinterpret_cast<__nv_bfloat162*>(prow)[i] = __floats2bfloat162_rn(v.x * a.ple_scale, v.y * a.ple_scale);
    }
  }
}

cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.D % 32 != 0 || a.LP % 32 != 0) return cudaErrorInvalidValue;
  return launch_k(embed_kernel, dim3(a.T), dim3(128), 0, s, 1, a);
}

// ---------------------------------------------------------------------------
// rmsnorm

constexpr int NORM_THREADS = 128;

// One CTA per row.  Rows of up to NORM_THREADS*4*NORM_VEC elements are read
// once and kept in registers between the sum of squares and the scaling;
// longer rows are read twice.  The reduction order (per-thread fmaf over the
// thread's vectors in index order, xor-shuffle tree, warps in order) is the
// same either way.
constexpr int NORM_VEC = 8;

// Outputs (each optional): y bf16 (the next projection's operand), y32 fp32
// (the embeddings output), x_copy (the input rows themselves).
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_kernel(const float* __restrict__ x, int row0, int D,
                                                               const float* __restrict__ gain, float eps,
                                                               __nv_bfloat16* __restrict__ y,
                                                               float* __restrict__ x_copy, float* __restrict__ y32,
                                                               const int* __restrict__ rows) {
  __shared__ float red[NORM_THREADS / 32];
  pdl_launch();
  pdl_wait();
  const int i = blockIdx.x;
  const int src_row = rows ? rows[i] : row0 + i;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)src_row * D);
  const int nv = D / 4;
  const bool in_regs = nv <= NORM_THREADS * NORM_VEC;
  float4 keep[NORM_VEC];
  float ss = 0.f;
  if (in_regs) {
#pragma unroll
    for (int k = 0; k < NORM_VEC; ++k) {
      const int v = threadIdx.x + k * NORM_THREADS;
      keep[k] = v < nv ? xr[v] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < NORM_VEC; ++k) {
      if (threadIdx.x + k * NORM_THREADS >= nv) break;
      const float4 a = keep[k];
      ss = __fmaf_rn(a.x, a.x, ss);
      ss = __fmaf_rn(a.y, a.y, ss);
      ss = __fmaf_rn(a.z, a.z, ss);
      ss = __fmaf_rn(a.w, a.w, ss);
    }
  } else {
    for (int v = threadIdx.x; v < nv; v += NORM_THREADS) {
      const float4 a = xr[v];
      ss = __fmaf_rn(a.x, a.x, ss);
      ss = __fmaf_rn(a.y, a.y, ss);
      ss = __fmaf_rn(a.z, a.z, ss);
      ss = __fmaf_rn(a.w, a.w, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = red[0];
#pragma unroll
  for (int w = 1; w < NORM_THREADS / 32; ++w) tot = __fadd_rn(tot, red[w]);
  const float r = rsqrtf(__fadd_rn(__fdiv_rn(tot, static_cast<float>(D)), eps));
  const float4* g4 = reinterpret_cast<const float4*>(gain);
  auto emit = [&](int v, const float4 a) {
    const float4 g = g4[v];
    const float4 n = make_float4(a.x * r * (1.f + g.x), a.y * r * (1.f + g.y), a.z * r * (1.f + g.z),
                                 a.w * r * (1.f + g.w));
    if (y) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(n.x, n.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(n.z, n.w);
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t*>(&lo);
      w.y = *reinterpret_cast<const uint32_t*>(&hi);
      reinterpret_cast<uint2*>(y + (size_t)i * D)[v] = w;
    }
    if (y32) reinterpret_cast<float4*>(y32 + (size_t)i * D)[v] = n;
    if (x_copy) reinterpret_cast<float4*>(x_copy + (size_t)i * D)[v] = a;
  };
  if (in_regs) {
#pragma unroll
    for (int k = 0; k < NORM_VEC; ++k) {
      const int v = threadIdx.x + k * NORM_THREADS;
      if (v >= nv) break;
      emit(v, keep[k]);
    }
  } else {
    for (int v = threadIdx.x; v < nv; v += NORM_THREADS) emit(v, xr[v]);
  }
}

cudaError_t launch_rmsnorm(const float* x, int row0, int M, int D, const float* g, float eps, __nv_bfloat16* y,
                           float* x_copy, cudaStream_t s, float* y32, const int* rows) {
  if (M <= 0) return cudaSuccess;
  if (D % 4 != 0) return cudaErrorInvalidValue;
  return launch_k(rmsnorm_kernel, dim3(M), dim3(NORM_THREADS), 0, s, 1, x, row0, D, g, eps, y, x_copy, y32, rows);
}

// one CTA per gathered row, 16-byte vectors
__global__ void __launch_bounds__(128) gather_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          const int* __restrict__ rows, int row_vec) {
  pdl_launch();
  pdl_wait();
  const uint4* s = src + (size_t)rows[blockIdx.x] * row_vec;
  uint4* d = dst + (size_t)blockIdx.x * row_vec;
  for (int v = threadIdx.x; v < row_vec; v += blockDim.x) d[v] = s[v];
}

cudaError_t launch_gather_rows(const void* src, void* dst, const int* rows, int n, size_t row_bytes, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (row_bytes % 16 != 0 || ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 16) != 0)
    return cudaErrorInvalidValue;
  return launch_k(gather_rows_kernel, dim3(n), dim3(128), 0, s, 1, static_cast<const uint4*>(src),
                  static_cast<uint4*>(dst), rows, static_cast<int>(row_bytes / 16));
}

// ---------------------------------------------------------------------------
// KV image copy: a grid-stride loop over 16-byte vectors, up to four
// vectors in flight per thread.  Segment s (s = kind * L_w + layer) is copy_vec vectors
// long; it sits at s * cache_stride_vec in the cache and s * img_stride_vec
// in the image body.

__device__ __forceinline__ void kv_vec_index(int64_t v, int64_t copy_vec, int64_t cache_stride_vec,
                                             int64_t img_stride_vec, int64_t& ci, int64_t& ii) {
  const int64_t seg = v / copy_vec, off = v - seg * copy_vec;
  ci = seg * cache_stride_vec + off;
  ii = seg * img_stride_vec + off;
}

__global__ void __launch_bounds__(256) kv_copy_kernel(int dir, uint4* __restrict__ cache, int64_t cache_stride_vec,
                                                      uint8_t* __restrict__ image, int64_t img_stride_vec,
                                                      int64_t copy_vec, int64_t n_vec, int4 header) {
  pdl_launch();
  pdl_wait();
  if (dir == 0 && blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<int4*>(image) = header;
  uint4* body = reinterpret_cast<uint4*>(image + 16);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // up to four vectors per thread in flight, the last group predicated, so
  // that an image with only a few vectors per thread still issues all its
  // loads before the first store
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n_vec; v += 4 * stride) {
    int64_t ci[4], ii[4];
    uint4 tmp[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (v + u * stride < n_vec) {
        kv_vec_index(v + u * stride, copy_vec, cache_stride_vec, img_stride_vec, ci[u], ii[u]);
        tmp[u] = dir == 0 ? cache[ci[u]] : body[ii[u]];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (v + u * stride < n_vec) {
        if (dir == 0)
          body[ii[u]] = tmp[u];
        else
          cache[ci[u]] = tmp[u];
      }
    }
  }
}

cudaError_t launch_kv_copy(int dir, __half* cache, int64_t cache_seg_stride, uint8_t* image, int64_t img_seg_bytes,
                           int n_seg, int64_t copy_bytes, const int32_t header[4], cudaStream_t s) {
  // both sides move 16-byte vectors
  if (copy_bytes % 16 != 0 || img_seg_bytes % 16 != 0 || cache_seg_stride % 8 != 0 ||
      ((reinterpret_cast<uintptr_t>(image) | reinterpret_cast<uintptr_t>(cache)) % 16) != 0)
    return cudaErrorInvalidValue;
  const int64_t copy_vec = copy_bytes / 16;
  const int64_t n_vec = copy_vec * n_seg;
  const int4 h = make_int4(header[0], header[1], header[2], header[3]);
  if (n_vec == 0) {
    if (dir == 0) return cudaMemcpyAsync(image, &h, 16, cudaMemcpyHostToDevice, s);
    return cudaSuccess;
  }
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n_vec + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  return launch_k(kv_copy_kernel, dim3((unsigned)blocks), dim3(256), 0, s, 1, dir, reinterpret_cast<uint4*>(cache),
                  static_cast<int64_t>(cache_seg_stride / 8), image, static_cast<int64_t>(img_seg_bytes / 16), copy_vec,
                  n_vec, h);
}

}  // namespace pf
