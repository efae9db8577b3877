// One-row projections on CUDA cores (kernels.h launch_gemv): a one-token
// ubatch, the output row of the KV-shared layers, the LM head.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

#include <mutex>

namespace pf {

// ---------------------------------------------------------------------------
// one-token projections
//
// A ubatch of one token (generation after the prompt) reads every weight
// once for one row, which the tensor-core kernel serves badly (its MMAs are
// 128 rows tall and it is bound per pipeline stage).  Here CTAs take
// (tile, k-part) pairs of a weight matrix in the GEMM's tile layout: the
// tile's BN rows over 32-row groups of lanes, the k-part's 64-wide k-blocks
// over the remaining warps, plain 16-byte loads of the Q4_0 tiles (or bf16
// rows), fp32 dot products (a Q4_0 value d*(n-8) is exact in fp32).  The
// k-parts of a tile form a thread-block cluster: after a cluster barrier,
// rank 0 adds the parts' row sums in part order through distributed shared
// memory and runs the GEMM's fused epilogue on the tile's one output row
// (no global partials, fences or tickets on the path).  The bits depend
// only on the matrix shape and the part count (a function of the shape).
constexpr int GV_WARPS = 8;
constexpr int GV_THREADS = GV_WARPS * 32;
constexpr int GV_TARGET_CTAS = 304;  // about two CTAs per SM
constexpr int GV_MAX_PARTS = 8;      // k-parts of a tile: one cluster, at most the portable cluster size

// Two fp32 lanes in one 64-bit register pair, for the packed arithmetic
// of sm_100-class SMs (sub.rn.f32x2 / fma.rn.f32x2: one instruction for two
// independent fp32 operations, each rounded as its scalar form would be).
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// sum over one 32-element Q4_0 block: byte j holds element j (low nibble)
// and element j + 16 (high nibble); x: the block's 32 activations.  A
// nibble n becomes the float 2^23 + n by placing it under the exponent byte
// of 2^23 (one byte permute, no integer-to-float conversion), and
// (2^23 + n) - (2^23 + 8) = n - 8 exactly.  The subtraction and the
// multiply-add run two elements per instruction (packed f32x2) on two
// chains: the even and the odd elements of each group of four, added at
// the end.
__device__ __forceinline__ float q4_block_dot(uint4 nib, const float* x) {
  const uint32_t wds[4] = {nib.x, nib.y, nib.z, nib.w};
  const unsigned long long bias = f2_pack(8388616.0f, 8388616.0f);  // 2^23 + 8
  unsigned long long s = 0ull;  // (+0, +0)
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 xl = *reinterpret_cast<const float4*>(x + 4 * q);
    const float4 xh = *reinterpret_cast<const float4*>(x + 16 + 4 * q);
    const uint32_t lo = wds[q] & 0x0F0F0F0Fu, hi = (wds[q] >> 4) & 0x0F0F0F0Fu;
    const unsigned long long l01 = f2_pack(__int_as_float(__byte_perm(lo, 0x4B000000u, 0x7440)),
                                           __int_as_float(__byte_perm(lo, 0x4B000000u, 0x7441)));
    const unsigned long long l23 = f2_pack(__int_as_float(__byte_perm(lo, 0x4B000000u, 0x7442)),
                                           __int_as_float(__byte_perm(lo, 0x4B000000u, 0x7443)));
    const unsigned long long h01 = f2_pack(__int_as_float(__byte_perm(hi, 0x4B000000u, 0x7440)),
                                           __int_as_float(__byte_perm(hi, 0x4B000000u, 0x7441)));
    const unsigned long long h23 = f2_pack(__int_as_float(__byte_perm(hi, 0x4B000000u, 0x7442)),
                                           __int_as_float(__byte_perm(hi, 0x4B000000u, 0x7443)));
    s = f2_fma(f2_sub(l01, bias), f2_pack(xl.x, xl.y), s);
    s = f2_fma(f2_sub(l23, bias), f2_pack(xl.z, xl.w), s);
    s = f2_fma(f2_sub(h01, bias), f2_pack(xh.x, xh.y), s);
    s = f2_fma(f2_sub(h23, bias), f2_pack(xh.z, xh.w), s);
  }
  const float2 r = f2_unpack(s);
  return r.x + r.y;
}

// Shared memory of a CTA: the row as fp32 [K] (only the part's columns are
// filled), then (Q4_0 weights) the CTA's weight slice: the tile's k-blocks
// kb0 .. kb1-1, contiguous in the tile layout, brought in by one bulk copy
// that is issued before the wait for the previous kernel (weights never
// depend on it), so the fetch overlaps that kernel's tail.
template <int WK, int BN>
__global__ void __launch_bounds__(GV_THREADS) gemv_kernel(const __nv_bfloat16* __restrict__ a, int K,
                                                          const uint8_t* __restrict__ w, int parts,
                                                          const EpiParams ep_in, int* err,
                                                          const float* __restrict__ nx, const float* __restrict__ ng,
                                                          float eps) {
  constexpr int RG = BN / 32;          // 32-row groups of a tile
  constexpr int KW = GV_WARPS / RG;    // warps along k inside the CTA
  static_assert(KW >= 1 && RG * KW <= GV_WARPS, "row groups x k-slices must fit the CTA's warps");
  constexpr int TILE = BN * 36;        // bytes of one (tile, k-block) of Q4_0
  extern __shared__ __align__(16) float xs[];  // the row, fp32 [K]; then the weight slice
  __shared__ float part_s[GV_WARPS][32];
  __shared__ float yp[BN];  // this part's row sums
  __shared__ float yv[BN];  // the tile's row (rank 0)
  __shared__ EpiParams ep;
  __shared__ __align__(8) uint64_t wbar;
  __shared__ __align__(16) uint8_t stage[2][EPI_STAGE_BYTES];
  const int nt = blockIdx.x / parts, kp = blockIdx.x % parts;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkb = K / 64;
  const int kb0 = kp * nkb / parts, kb1 = (kp + 1) * nkb / parts;
  uint8_t* wsl = reinterpret_cast<uint8_t*>(xs + K);
  if constexpr (WK == W_Q4) {
    if (tid == 0) {
      mbar_init(&wbar, 1);
      fence_mbar_init();
      if (kb1 > kb0) {
        const uint32_t bytes = static_cast<uint32_t>(kb1 - kb0) * TILE;
        mbar_arrive_expect_tx(&wbar, bytes);
        bulk_load(wsl, w + ((size_t)nt * nkb + kb0) * TILE, bytes, &wbar);
      } else {
        mbar_arrive(&wbar);
      }
    }
  }
  pdl_launch();
  if (tid == 0) ep = ep_in;
  pdl_wait();
  if (nx) {
    // The row is the RMS norm of the residual row nx (fp32 [K]) with gain
    // (1 + ng): every CTA forms it for itself (a fixed-order sum of squares,
    // the same in every CTA and every launch) and rounds it to bf16 as the
    // norm kernel would hand it over.
    __shared__ float red[GV_WARPS];
    const float4* x4 = reinterpret_cast<const float4*>(nx);
    float ss = 0.f;
    for (int v = tid; v < K / 4; v += GV_THREADS) {
      const float4 q = x4[v];
      ss = __fmaf_rn(q.x, q.x, ss);
      ss = __fmaf_rn(q.y, q.y, ss);
      ss = __fmaf_rn(q.z, q.z, ss);
      ss = __fmaf_rn(q.w, q.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = red[0];
#pragma unroll
    for (int w2 = 1; w2 < GV_WARPS; ++w2) tot = __fadd_rn(tot, red[w2]);
    const float rr = rsqrtf(__fadd_rn(__fdiv_rn(tot, static_cast<float>(K)), eps));
    const float4* g4 = reinterpret_cast<const float4*>(ng);
    for (int v = kb0 * 16 + tid; v < kb1 * 16; v += GV_THREADS) {  // the part's columns, 4 at a time
      const float4 q = x4[v], g = g4[v];
      const __nv_bfloat162 lo = __floats2bfloat162_rn(q.x * rr * (1.f + g.x), q.y * rr * (1.f + g.y));
      const __nv_bfloat162 hi = __floats2bfloat162_rn(q.z * rr * (1.f + g.z), q.w * rr * (1.f + g.w));
      *reinterpret_cast<float4*>(xs + 4 * v) =
          make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
    }
  } else {
    for (int i = kb0 * 8 + tid; i < kb1 * 8; i += GV_THREADS) {  // the part's columns, 8 at a time
      const uint4 u = reinterpret_cast<const uint4*>(a)[i];
      *reinterpret_cast<float4*>(xs + 8 * i) = bf16x4_to_f32(make_uint2(u.x, u.y));
      *reinterpret_cast<float4*>(xs + 8 * i + 4) = bf16x4_to_f32(make_uint2(u.z, u.w));
    }
  }
  __syncthreads();
  const int rg = warp % RG, kw = warp / RG;
  const int r = rg * 32 + lane;
  const int nk = kb1 - kb0;
  // warps past RG * KW (BN = 192: six row groups, one k-slice, warps 6 and
  // 7) take no k-blocks
  const int c0 = kw < KW ? kb0 + kw * nk / KW : kb0, c1 = kw < KW ? kb0 + (kw + 1) * nk / KW : kb0;
  float acc = 0.f;
  if constexpr (WK == W_Q4) {
    // bounded: a copy that never lands flags the error word; the sums are
    // then meaningless, but the launch still ends
    const bool landed = mbar_wait(&wbar, 0, err, PF_DEV_TIMEOUT_PRODUCER);
    if (landed) {
#pragma unroll 4
      for (int kb = c0; kb < c1; ++kb) {
        const uint8_t* t = wsl + (size_t)(kb - kb0) * TILE;
        const uint4 n0 = *reinterpret_cast<const uint4*>(t + r * 16);
        const uint4 n1 = *reinterpret_cast<const uint4*>(t + (BN + r) * 16);
        const float d0 = __half2float(*reinterpret_cast<const __half*>(t + BN * 32 + r * 2));
        const float d1 = __half2float(*reinterpret_cast<const __half*>(t + BN * 32 + (BN + r) * 2));
        acc = fmaf(d0, q4_block_dot(n0, xs + kb * 64), acc);
        acc = fmaf(d1, q4_block_dot(n1, xs + kb * 64 + 32), acc);
      }
    }
  } else {
    const __nv_bfloat16* wr = reinterpret_cast<const __nv_bfloat16*>(w) + (size_t)(nt * BN + r) * K;
#pragma unroll 2
    for (int k = c0 * 64; k < c1 * 64; k += 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(wr + k);
      const float4 w0 = bf16x4_to_f32(make_uint2(u.x, u.y)), w1 = bf16x4_to_f32(make_uint2(u.z, u.w));
      const float4 x0 = *reinterpret_cast<const float4*>(xs + k), x1 = *reinterpret_cast<const float4*>(xs + k + 4);
      acc = fmaf(w0.x, x0.x, acc);
      acc = fmaf(w0.y, x0.y, acc);
      acc = fmaf(w0.z, x0.z, acc);
      acc = fmaf(w0.w, x0.w, acc);
      acc = fmaf(w1.x, x1.x, acc);
      acc = fmaf(w1.y, x1.y, acc);
      acc = fmaf(w1.z, x1.z, acc);
      acc = fmaf(w1.w, x1.w, acc);
    }
  }
  part_s[warp][lane] = acc;
  __syncthreads();
  if (tid < BN) {
    const int g = tid >> 5, l = tid & 31;
    float t = part_s[g][l];
    for (int q = 1; q < KW; ++q) t += part_s[q * RG + g][l];
    yp[tid] = t;
  }
  if (parts > 1) {
    // the cluster's CTAs are the tile's k-parts, rank = part: rank 0 adds
    // the parts in order once every rank's sums are in its shared memory,
    // and the others stay until rank 0 has read them
    cluster_sync_all();
    if (kp == 0 && tid < BN) {
      float t = yp[tid];
      const uint32_t own = smem_u32(&yp[tid]);
      for (int q = 1; q < parts; ++q) t += ld_cluster_f32(map_to_rank(own, static_cast<uint32_t>(q)));
      yv[tid] = t;
    }
    cluster_sync_all();
    if (kp != 0) return;
  } else if (tid < BN) {
    yv[tid] = yp[tid];
  }
  __syncthreads();
  if (warp < 2)
    run_epilogue<BN>(ep, 0, 1, nt, warp, stage[warp], 0, [&](int c, float(&v)[32]) {
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = lane == 0 ? yv[32 * c + q] : 0.f;
    });
}

int gemv_parts(const WeightMat& W) {
  const int n_tiles = W.N_rows / W.BN, nkb = W.K / 64;
  int p = (GV_TARGET_CTAS + n_tiles - 1) / n_tiles;
  if (p > nkb) p = nkb;
  if (p > GV_MAX_PARTS) p = GV_MAX_PARTS;
  return p < 1 ? 1 : p;
}

// dynamic shared memory of a launch: the row (K floats) and, for Q4_0, the
// largest weight slice of a k-part
static size_t gemv_smem(const WeightMat& W, int parts) {
  const int nkb = W.K / 64;
  const size_t slice = W.kind == W_Q4 ? static_cast<size_t>((nkb + parts - 1) / parts) * W.BN * 36 : 0;
  return static_cast<size_t>(W.K) * 4 + slice;
}

constexpr size_t GV_SMEM_MAX = 160 * 1024;

template <int WK, int BN>
static cudaError_t launch_gemv_t(const ActMat& A, const WeightMat& W, const EpiParams& ep, int* err, cudaStream_t s,
                                 const float* nx, const float* ng, float eps) {
  {
    const cudaError_t e = smem_opt_in<gemv_kernel<WK, BN>>(static_cast<int>(GV_SMEM_MAX));
    if (e != cudaSuccess) return e;
  }
  const int parts = gemv_parts(W);
  const size_t smem = gemv_smem(W, parts);
  if (smem > GV_SMEM_MAX) return cudaErrorInvalidValue;
  const int grid = (W.N_rows / BN) * parts;  // clusters of `parts` CTAs: one tile each
  return launch_k(gemv_kernel<WK, BN>, dim3(grid), dim3(GV_THREADS), smem, s, parts, A.dev, W.K,
                  static_cast<const uint8_t*>(W.dev), parts, ep, err, nx, ng, eps);
}

cudaError_t launch_gemv(const ActMat& A, const WeightMat& W, const EpiParams& ep, int* err, cudaStream_t s,
                        const float* norm_x, const float* norm_g, float eps) {
  if (A.K != W.K || W.K % 64 != 0 || W.N_rows % W.BN != 0) return cudaErrorInvalidValue;
  if (norm_x && (!norm_g || (reinterpret_cast<uintptr_t>(norm_x) | reinterpret_cast<uintptr_t>(norm_g)) % 16 != 0))
    return cudaErrorInvalidValue;
#define PF_GEMV_CASE(WKV, BNV) \
  if (W.kind == WKV && W.BN == BNV) return launch_gemv_t<WKV, BNV>(A, W, ep, err, s, norm_x, norm_g, eps);
  PF_GEMV_CASE(W_Q4, 64)
  PF_GEMV_CASE(W_Q4, 128)
  PF_GEMV_CASE(W_Q4, 192)
  PF_GEMV_CASE(W_Q4, 256)
  PF_GEMV_CASE(W_BF16, 64)
  PF_GEMV_CASE(W_BF16, 128)
  PF_GEMV_CASE(W_BF16, 256)
#undef PF_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pf
