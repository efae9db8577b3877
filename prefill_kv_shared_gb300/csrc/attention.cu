// Causal grouped-query attention over the FP16 KV cache.
//
// Keys are cut into absolute 64-key chunks.  For one query row the result is
// a left fold, in ascending chunk order, of per-chunk partials
//     (m_j, l_j, o_j):  m_j = max_k s_k,  p_k = fp16(2^((s_k - m_j) c)),
//                       l_j = sum_k p_k,  o_j = sum_k p_k V_k
// (s = q.k, c = log2(e)/sqrt(hd)) combined by merge_state().  Two launch forms
// compute exactly the same fold:
//   attn_prefill  every row of a ubatch; a CTA walks the chunks in order and
//                 merges each partial into registers (writing layers, and the
//                 KV-shared layers when pruning is off);
//   attn_split    one output row (KV-shared layers after pruning): one CTA per
//                 chunk writes its partial to global memory, then a warp per
//                 head folds them in order (a split-K warp reduction).
// Both run the same warp routine, attn_chunk(), for a chunk, and the same
// merge_state(); a row's partial does not depend on the other rows in its MMA
// tile.  So the pruned output row is bit-identical to the unpruned one.
//
// MMA rows are (query, head-within-group) pairs: row R = t*G + g for query t
// and query head kvh*G + g, so the G query heads that share a KV head share
// the K/V tiles.
#include "common.cuh"
#include "kernels.h"

namespace pf {

constexpr int CHUNK = 64;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0: fill the 16 bytes with zeros
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Fold partial (mj, lj) into state (m, l); returns the scale factors a (old
// state) and b (partial).  The state's o is updated by the caller as
// o = a*o + b*o_j with merge_o().  An empty state (m = -inf, l = 0, o = 0)
// merged with a partial gives the partial exactly.
struct MergeAB {
  float a, b;
};
template <int HD>
__device__ __forceinline__ MergeAB merge_state(float& m, float& l, float mj, float lj) {
  constexpr float c = 1.4426950408889634f / (HD == 256 ? 16.0f : HD == 128 ? 11.313708498984761f : 8.0f);
  const float mn = fmaxf(m, mj);
  MergeAB r;
  r.a = ex2_approx(__fmul_rn(__fsub_rn(m, mn), c));
  r.b = ex2_approx(__fmul_rn(__fsub_rn(mj, mn), c));
  l = __fadd_rn(__fmul_rn(r.a, l), __fmul_rn(r.b, lj));
  m = mn;
  return r;
}
__device__ __forceinline__ float merge_o(float o, float oj, MergeAB ab) {
  return __fadd_rn(__fmul_rn(ab.a, o), __fmul_rn(ab.b, oj));
}

template <int HD>
struct ChunkSmem {
  static constexpr int LD = HD + 8;  // halves per row; the pad removes ldmatrix bank conflicts
  static constexpr int ROW_BYTES = LD * 2;
  static constexpr int KV_BYTES = CHUNK * ROW_BYTES;  // one K or V chunk
};

// Stage chunk `ch` of K and V (keys [64ch, 64ch+64)) into shared memory;
// keys >= kv_len read as zeros.
template <int HD>
__device__ __forceinline__ void load_kv_chunk(uint32_t sk, uint32_t sv, const __half* k, const __half* v,
                                              int kv_stride, int kv_len, int ch, int tid, int nthreads) {
  using S = ChunkSmem<HD>;
  constexpr int VPR = HD / 8;  // 16-byte vectors per key row
  for (int i = tid; i < CHUNK * VPR; i += nthreads) {
    const int r = i / VPR, c = i % VPR;
    const int key = ch * CHUNK + r;
    const bool ok = key < kv_len;
    const size_t off = (size_t)(ok ? key : 0) * kv_stride + c * 8;
    cp_async16(sk + r * S::ROW_BYTES + c * 16, k + off, ok);
    cp_async16(sv + r * S::ROW_BYTES + c * 16, v + off, ok);
  }
}

// One warp, 16 MMA rows (q in shared memory, ld = HD+8), one 64-key chunk.
// pos0/pos1: positions of the thread's rows g and g+8 (-1: row unused).
// Produces, for both rows, mj/lj (identical across the row's 4 lanes) and the
// fp16 probabilities; then calls sink(dt0, o) for each 64-dim group with the
// group's o_j fragments o[8][4].
template <int HD, class Sink>
__device__ __forceinline__ void attn_chunk(uint32_t sq, uint32_t sk, uint32_t sv, int ch, int pos0, int pos1,
                                           float (&mj)[2], float (&lj)[2], Sink&& sink) {
  using S = ChunkSmem<HD>;
  const int lane = threadIdx.x & 31;
  const int tq = lane & 3;
  const int lm = lane >> 3, lr = lane & 7;

  // s = q k^T for 16 rows x 64 keys
  float s[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < HD / 16; ks += 2) {
    uint32_t qa[4], qb[4];
    ldsm_x4(qa, sq + (lr + ((lm & 1) << 3)) * S::ROW_BYTES + (16 * ks + ((lm >> 1) << 3)) * 2);
    ldsm_x4(qb, sq + (lr + ((lm & 1) << 3)) * S::ROW_BYTES + (16 * (ks + 1) + ((lm >> 1) << 3)) * 2);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      uint32_t kb[4];  // b0,b1 for k-step ks, then b0,b1 for ks+1
      ldsm_x4(kb, sk + (8 * nt + lr) * S::ROW_BYTES + (16 * ks + 8 * lm) * 2);
      mma16816(s[nt], qa, kb[0], kb[1]);
      mma16816(s[nt], qb, kb[2], kb[3]);
    }
  }

  // causal mask, row max
  const int kbase = ch * CHUNK + 2 * tq;
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = kbase + 8 * nt + e;
      if (key > pos0) s[nt][e] = -INFINITY;
      if (key > pos1) s[nt][2 + e] = -INFINITY;
      mx0 = fmaxf(mx0, s[nt][e]);
      mx1 = fmaxf(mx1, s[nt][2 + e]);
    }
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));

  // probabilities, rounded to fp16; the sum adds the rounded values
  constexpr float c = 1.4426950408889634f / (HD == 256 ? 16.0f : HD == 128 ? 11.313708498984761f : 8.0f);
  uint32_t p[8][2];
  float sum0 = 0.f, sum1 = 0.f;
  const bool act0 = mx0 != -INFINITY, act1 = mx1 != -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const float p0 = act0 ? ex2_approx(__fmul_rn(__fsub_rn(s[nt][0], mx0), c)) : 0.f;
    const float p1 = act0 ? ex2_approx(__fmul_rn(__fsub_rn(s[nt][1], mx0), c)) : 0.f;
    const float p2 = act1 ? ex2_approx(__fmul_rn(__fsub_rn(s[nt][2], mx1), c)) : 0.f;
    const float p3 = act1 ? ex2_approx(__fmul_rn(__fsub_rn(s[nt][3], mx1), c)) : 0.f;
    const __half2 h01 = __floats2half2_rn(p0, p1);
    const __half2 h23 = __floats2half2_rn(p2, p3);
    p[nt][0] = *reinterpret_cast<const uint32_t*>(&h01);
    p[nt][1] = *reinterpret_cast<const uint32_t*>(&h23);
    sum0 = __fadd_rn(__fadd_rn(sum0, __low2float(h01)), __high2float(h01));
    sum1 = __fadd_rn(__fadd_rn(sum1, __low2float(h23)), __high2float(h23));
  }
  sum0 = __fadd_rn(sum0, __shfl_xor_sync(0xffffffffu, sum0, 1));
  sum0 = __fadd_rn(sum0, __shfl_xor_sync(0xffffffffu, sum0, 2));
  sum1 = __fadd_rn(sum1, __shfl_xor_sync(0xffffffffu, sum1, 1));
  sum1 = __fadd_rn(sum1, __shfl_xor_sync(0xffffffffu, sum1, 2));
  mj[0] = mx0;
  mj[1] = mx1;
  lj[0] = sum0;
  lj[1] = sum1;

  // o_j = P V, 64 output dims at a time
#pragma unroll
  for (int grp = 0; grp < HD / 64; ++grp) {
    float o[8][4];
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t pa[4] = {p[2 * kk][0], p[2 * kk][1], p[2 * kk + 1][0], p[2 * kk + 1][1]};
#pragma unroll
      for (int dp = 0; dp < 4; ++dp) {
        const int dt = 2 * dp;
        uint32_t vb[4];  // (keys +0, dims dt) (keys +8, dims dt) (keys +0, dims dt+1) (keys +8, dims dt+1)
        ldsm_x4_t(vb, sv + (16 * kk + lr + ((lm & 1) << 3)) * S::ROW_BYTES +
                          (64 * grp + 8 * dt + ((lm >> 1) << 3)) * 2);
        mma16816(o[dt], pa, vb[0], vb[1]);
        mma16816(o[dt + 1], pa, vb[2], vb[3]);
      }
    }
    sink(grp, o);
  }
}

// ---------------------------------------------------------------------------
// attn_prefill: every row, in-CTA ordered fold

template <int HD, int NW>
struct PrefillCfg {
  using S = ChunkSmem<HD>;
  static constexpr int ROWS = 16 * NW;
  static constexpr int Q_BYTES = ROWS * S::ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * S::KV_BYTES;
  static constexpr int SMEM = Q_BYTES + 2 * STAGE_BYTES;
};

template <int HD, int NW>
__global__ void __launch_bounds__(NW * 32, 1) attn_prefill_kernel(AttnArgs a) {
  using S = ChunkSmem<HD>;
  using C = PrefillCfg<HD, NW>;
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_launch();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int G = a.Hq / a.Hkv;
  const int kvh = blockIdx.y;
  const int R0 = blockIdx.x * C::ROWS;
  const int q_stride = a.Hq * HD, kv_stride = a.Hkv * HD;
  const __half* kbase = a.k + kvh * HD;
  const __half* vbase = a.v + kvh * HD;

  // queries of this CTA
  const uint32_t sq = smem_u32(smem);
  for (int i = tid; i < C::ROWS * (HD / 8); i += NW * 32) {
    const int r = i / (HD / 8), c = i % (HD / 8);
    const int R = R0 + r, t = R / G, head = kvh * G + R % G;
    const bool ok = t < a.M;
    cp_async16(sq + r * S::ROW_BYTES + c * 16, a.q + (size_t)(ok ? t : 0) * q_stride + head * HD + c * 8, ok);
  }
  const int t_last = min(a.M - 1, (R0 + C::ROWS - 1) / G);
  const int last_ch = (a.pos_base + t_last) / CHUNK;
  const uint32_t skv0 = sq + C::Q_BYTES;
  load_kv_chunk<HD>(skv0, skv0 + S::KV_BYTES, kbase, vbase, kv_stride, a.kv_len, 0, tid, NW * 32);
  cp_async_commit();

  // this thread's two rows
  const int Rw = R0 + warp * 16;
  const int ta = (Rw + g) / G, tb = (Rw + g + 8) / G;
  const int posa = ta < a.M ? a.pos_base + ta : -1;
  const int posb = tb < a.M ? a.pos_base + tb : -1;
  const int warp_tmax = min(a.M - 1, (Rw + 15) / G);
  const int warp_pmax = (Rw / G) < a.M ? a.pos_base + warp_tmax : -1;

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int ch = 0; ch <= last_ch; ++ch) {
    if (ch + 1 <= last_ch) {
      const uint32_t nst = skv0 + ((ch + 1) & 1) * C::STAGE_BYTES;
      load_kv_chunk<HD>(nst, nst + S::KV_BYTES, kbase, vbase, kv_stride, a.kv_len, ch + 1, tid, NW * 32);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (warp_pmax >= ch * CHUNK) {
      const uint32_t st = skv0 + (ch & 1) * C::STAGE_BYTES;
      float mj[2], lj[2];
      MergeAB ab[2];
      bool act[2];
      attn_chunk<HD>(sq + warp * 16 * S::ROW_BYTES, st, st + S::KV_BYTES, ch, posa, posb, mj, lj,
                     [&](int grp, float(&oj)[8][4]) {
                       if (grp == 0) {
                         act[0] = mj[0] != -INFINITY;
                         act[1] = mj[1] != -INFINITY;
                         if (act[0]) ab[0] = merge_state<HD>(m[0], l[0], mj[0], lj[0]);
                         if (act[1]) ab[1] = merge_state<HD>(m[1], l[1], mj[1], lj[1]);
                       }
#pragma unroll
                       for (int dt = 0; dt < 8; ++dt) {
                         float* od = o[grp * 8 + dt];
                         if (act[0]) {
                           od[0] = merge_o(od[0], oj[dt][0], ab[0]);
                           od[1] = merge_o(od[1], oj[dt][1], ab[0]);
                         }
                         if (act[1]) {
                           od[2] = merge_o(od[2], oj[dt][2], ab[1]);
                           od[3] = merge_o(od[3], oj[dt][3], ab[1]);
                         }
                       }
                     });
    }
    __syncthreads();
  }

  // out = o / l
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int t = half ? tb : ta;
    if (t >= a.M) continue;
    const int R = Rw + g + 8 * half;
    const int head = kvh * G + R % G;
    __nv_bfloat16* dst = a.out + (size_t)t * q_stride + head * HD;
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt) {
      const float x0 = __fdiv_rn(o[dt][2 * half], l[half]);
      const float x1 = __fdiv_rn(o[dt][2 * half + 1], l[half]);
      *reinterpret_cast<__nv_bfloat162*>(dst + 8 * dt + 2 * tq) = __floats2bfloat162_rn(x0, x1);
    }
  }
}

// ---------------------------------------------------------------------------
// attn_split: one row; a CTA (one warp) per (chunk, KV head) writes its
// partial, then attn_merge folds the partials of each head in chunk order.
// partial layout: [head][chunk][HD + 2] = o_j[HD], m_j, l_j

template <int HD>
struct SplitCfg {
  using S = ChunkSmem<HD>;
  static constexpr int Q_BYTES = 16 * S::ROW_BYTES;
  static constexpr int SMEM = Q_BYTES + 2 * S::KV_BYTES;
};

template <int HD>
__global__ void __launch_bounds__(32) attn_split_kernel(AttnArgs a, float* __restrict__ part, int n_chunks) {
  using S = ChunkSmem<HD>;
  using C = SplitCfg<HD>;
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_launch();
  pdl_wait();
  const int lane = threadIdx.x;
  const int g = lane >> 2, tq = lane & 3;
  const int ch = blockIdx.x, kvh = blockIdx.y;
  const int G = a.Hq / a.Hkv;
  const int kv_stride = a.Hkv * HD;
  const uint32_t sq = smem_u32(smem);
  const uint32_t sk = sq + C::Q_BYTES, sv = sk + S::KV_BYTES;
  for (int i = lane; i < 16 * (HD / 8); i += 32) {
    const int r = i / (HD / 8), c = i % (HD / 8);
    const bool ok = r < G;
    cp_async16(sq + r * S::ROW_BYTES + c * 16, a.q + (ok ? (kvh * G + r) * HD : 0) + c * 8, ok);
  }
  load_kv_chunk<HD>(sk, sv, a.k + kvh * HD, a.v + kvh * HD, kv_stride, a.kv_len, ch, lane, 32);
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();

  const int pos = a.pos_base;  // the single row's position
  const int pa = g < G ? pos : -1, pb = g + 8 < G ? pos : -1;
  float mj[2], lj[2];
  attn_chunk<HD>(sq, sk, sv, ch, pa, pb, mj, lj, [&](int grp, float(&oj)[8][4]) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = g + 8 * half;
      if (r >= G) continue;
      float* dst = part + ((size_t)(kvh * G + r) * n_chunks + ch) * (HD + 2);
#pragma unroll
      for (int dt = 0; dt < 8; ++dt)
        *reinterpret_cast<float2*>(dst + 64 * grp + 8 * dt + 2 * tq) =
            make_float2(oj[dt][2 * half], oj[dt][2 * half + 1]);
    }
  });
  if (tq == 0) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = g + 8 * half;
      if (r >= G) continue;
      float* dst = part + ((size_t)(kvh * G + r) * n_chunks + ch) * (HD + 2);
      dst[HD] = mj[half];
      dst[HD + 1] = lj[half];
    }
  }
}

// one warp per head; lane owns HD/32 consecutive dims
template <int HD>
__global__ void __launch_bounds__(32) attn_merge_kernel(const float* __restrict__ part, int n_chunks, int Hq,
                                                        __nv_bfloat16* __restrict__ out) {
  constexpr int PER = HD / 32;
  pdl_launch();
  pdl_wait();
  const int head = blockIdx.x, lane = threadIdx.x;
  const float* base = part + (size_t)head * n_chunks * (HD + 2);
  float m = -INFINITY, l = 0.f, o[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) o[i] = 0.f;
  for (int ch = 0; ch < n_chunks; ++ch) {
    const float* p = base + (size_t)ch * (HD + 2);
    const float mj = p[HD], lj = p[HD + 1];
    float oj[PER];
#pragma unroll
    for (int i = 0; i < PER; i += 2) {
      const float2 v = *reinterpret_cast<const float2*>(p + lane * PER + i);
      oj[i] = v.x;
      oj[i + 1] = v.y;
    }
    if (mj == -INFINITY) continue;
    const MergeAB ab = merge_state<HD>(m, l, mj, lj);
#pragma unroll
    for (int i = 0; i < PER; ++i) o[i] = merge_o(o[i], oj[i], ab);
  }
  __nv_bfloat16* dst = out + (size_t)head * HD + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + i) = __floats2bfloat162_rn(__fdiv_rn(o[i], l), __fdiv_rn(o[i + 1], l));
}

// ---------------------------------------------------------------------------
// launchers

template <int HD, int NW>
static cudaError_t launch_prefill_t(const AttnArgs& a, cudaStream_t s) {
  using C = PrefillCfg<HD, NW>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<HD, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int G = a.Hq / a.Hkv;
  const int rows = a.M * G;
  dim3 grid((rows + C::ROWS - 1) / C::ROWS, a.Hkv);
  return launch_k(attn_prefill_kernel<HD, NW>, grid, dim3(NW * 32), C::SMEM, s, 1, a);
}

static bool attn_shape_ok(const AttnArgs& a) {
  if (a.Hkv <= 0 || a.Hq % a.Hkv != 0) return false;
  const int G = a.Hq / a.Hkv;
  if (G > 16 || (16 % G) != 0) return false;
  return a.hd == 64 || a.hd == 256;
}

cudaError_t launch_attn_prefill(const AttnArgs& a, cudaStream_t s) {
  if (a.M <= 0) return cudaSuccess;
  if (!attn_shape_ok(a)) return cudaErrorInvalidValue;
  if (a.hd == 256) return launch_prefill_t<256, 4>(a, s);
  return launch_prefill_t<64, 4>(a, s);
}

template <int HD>
static cudaError_t launch_split_t(const AttnArgs& a, float* part, cudaStream_t s) {
  using C = SplitCfg<HD>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_split_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int n_chunks = a.pos_base / CHUNK + 1;
  cudaError_t e = launch_k(attn_split_kernel<HD>, dim3(n_chunks, a.Hkv), dim3(32), C::SMEM, s, 1, a, part, n_chunks);
  if (e != cudaSuccess) return e;
  return launch_k(attn_merge_kernel<HD>, dim3(a.Hq), dim3(32), 0, s, 1, static_cast<const float*>(part), n_chunks,
                  a.Hq, a.out);
}

cudaError_t launch_attn_split(const AttnArgs& a, float* part, cudaStream_t s) {
  if (a.M != 1 || !attn_shape_ok(a)) return cudaErrorInvalidValue;
  if (a.hd == 256) return launch_split_t<256>(a, part, s);
  return launch_split_t<64>(a, part, s);
}

size_t attn_partials_floats(int Hq, int hd, int max_ctx) {
  const size_t n_chunks = (static_cast<size_t>(max_ctx) + CHUNK - 1) / CHUNK;
  return static_cast<size_t>(Hq) * n_chunks * (hd + 2);
}

}  // namespace pf
