// Causal grouped-query attention over the FP16 KV cache.
//
// Keys are cut into absolute 64-key chunks.  For one query row the result is
// a left fold, in ascending chunk order, of per-chunk partials
//     (m_j, l_j, o_j):  m_j = max_k s_k,  p_k = fp16(2^((s_k - m_j) c)),
//                       l_j = sum_k p_k,  o_j = sum_k p_k V_k
// (s = q.k, c = log2(e)/sqrt(hd)) combined by merge_state().
//
// The chunks are taken in groups of gc consecutive chunks, gc fixed by the
// number of keys in the launch (attn_group_chunks: at most 4 groups).  A CTA
// handles one (64-row block, group) pair: it folds the group's chunks in
// ascending order into a state (m, l, o).  A row whose keys lie in one group
// writes o / l directly; otherwise each group's state goes to a partials
// buffer and attn_merge folds the row's group states in ascending order.  So
// the causal work spreads over many CTAs instead of piling up on the CTAs of
// the last rows.
//
// A row's result depends only on its own position, the keys and gc: the MMA
// rows of a tile are independent, chunks past a row's position leave its
// state unchanged, and gc is the same for the ubatch's last row whether the
// launch carries the whole ubatch (M = T) or that row alone (M = 1, the
// KV-shared layers after pruning), because both see the same number of keys.
// So the pruned output row is bit-identical to the unpruned one.
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

// partials layout: [row t][query head][group (ATTN_MAX_GROUPS)][HD + 2] =
// o[HD] (not normalised), m, l
constexpr int ATTN_MAX_GROUPS = 4;

int attn_group_chunks(int kv_len) {
  const int n_chunks = (kv_len + CHUNK - 1) / CHUNK;
  const int gc = (n_chunks + ATTN_MAX_GROUPS - 1) / ATTN_MAX_GROUPS;
  return gc < 1 ? 1 : gc;
}

// groups that hold keys of the row at position pos
__host__ __device__ __forceinline__ int attn_row_groups(int pos, int gc) { return (pos / CHUNK) / gc + 1; }

template <int HD, int NW>
struct PrefillCfg {
  using S = ChunkSmem<HD>;
  static constexpr int ROWS = 16 * NW;
  static constexpr int Q_BYTES = ROWS * S::ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * S::KV_BYTES;
  static constexpr int SMEM = Q_BYTES + STAGE_BYTES;  // one K/V stage: two CTAs fit on an SM
};

template <int HD, int NW>
__global__ void __launch_bounds__(NW * 32, 2) attn_prefill_kernel(AttnArgs a, float* __restrict__ part, int gc) {
  using S = ChunkSmem<HD>;
  using C = PrefillCfg<HD, NW>;
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_launch();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int G = a.Hq / a.Hkv;
  const int kvh = blockIdx.y, grp = blockIdx.z;
  const int R0 = blockIdx.x * C::ROWS;
  const int q_stride = a.Hq * HD, kv_stride = a.Hkv * HD;
  const __half* kbase = a.k + kvh * HD;
  const __half* vbase = a.v + kvh * HD;
  const int t_last = min(a.M - 1, (R0 + C::ROWS - 1) / G);
  const int last_ch = (a.pos_base + t_last) / CHUNK;
  const int ch_first = grp * gc;
  if (ch_first > last_ch) return;  // no keys of this group reach the block's rows
  const int ch_end = min(last_ch, ch_first + gc - 1);

  // queries of this CTA
  const uint32_t sq = smem_u32(smem);
  for (int i = tid; i < C::ROWS * (HD / 8); i += NW * 32) {
    const int r = i / (HD / 8), c = i % (HD / 8);
    const int R = R0 + r, t = R / G, head = kvh * G + R % G;
    const bool ok = t < a.M;
    cp_async16(sq + r * S::ROW_BYTES + c * 16, a.q + (size_t)(ok ? t : 0) * q_stride + head * HD + c * 8, ok);
  }
  const uint32_t sk = sq + C::Q_BYTES, sv = sk + S::KV_BYTES;

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

  for (int ch = ch_first; ch <= ch_end; ++ch) {
    if (ch != ch_first) __syncthreads();  // every warp is done with the previous chunk
    load_kv_chunk<HD>(sk, sv, kbase, vbase, kv_stride, a.kv_len, ch, tid, NW * 32);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    if (warp_pmax >= ch * CHUNK) {
      float mj[2], lj[2];
      MergeAB ab[2];
      bool act[2];
      attn_chunk<HD>(sq + warp * 16 * S::ROW_BYTES, sk, sv, ch, posa, posb, mj, lj, [&](int dg, float(&oj)[8][4]) {
        if (dg == 0) {
          act[0] = mj[0] != -INFINITY;
          act[1] = mj[1] != -INFINITY;
          if (act[0]) ab[0] = merge_state<HD>(m[0], l[0], mj[0], lj[0]);
          if (act[1]) ab[1] = merge_state<HD>(m[1], l[1], mj[1], lj[1]);
        }
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
          float* od = o[dg * 8 + dt];
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
  }

  // a row with one group: out = o / l; otherwise the group state
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int t = half ? tb : ta;
    if (t >= a.M) continue;
    const int R = Rw + g + 8 * half;
    const int head = kvh * G + R % G;
    const int n_g = attn_row_groups(a.pos_base + t, gc);
    if (n_g == 1) {
      __nv_bfloat16* dst = a.out + (size_t)t * q_stride + head * HD;
#pragma unroll
      for (int dt = 0; dt < HD / 8; ++dt) {
        const float x0 = __fdiv_rn(o[dt][2 * half], l[half]);
        const float x1 = __fdiv_rn(o[dt][2 * half + 1], l[half]);
        *reinterpret_cast<__nv_bfloat162*>(dst + 8 * dt + 2 * tq) = __floats2bfloat162_rn(x0, x1);
      }
    } else if (grp < n_g) {
      float* dst = part + (((size_t)t * a.Hq + head) * ATTN_MAX_GROUPS + grp) * (HD + 2);
#pragma unroll
      for (int dt = 0; dt < HD / 8; ++dt)
        *reinterpret_cast<float2*>(dst + 8 * dt + 2 * tq) = make_float2(o[dt][2 * half], o[dt][2 * half + 1]);
      if (tq == 0) {
        dst[HD] = m[half];
        dst[HD + 1] = l[half];
      }
    }
  }
}

// Rows t0 .. M-1 (two or more groups): a warp per (row, query head) combines
// the group states (m_g, l_g, o_g): m = max m_g, w_g = 2^((m_g - m) c),
// l = sum w_g l_g, out = (sum w_g o_g) / l, sums in ascending group order.
// Every load is issued before the values it feeds are combined, so a row
// costs two memory round trips however many groups it has.  (The single-row
// form of the KV-shared layers runs this same kernel, so the pruned row's
// bits do not depend on the combination order chosen here.)  Lane owns HD/32
// consecutive dims.
template <int HD>
__global__ void __launch_bounds__(128) attn_merge_kernel(const float* __restrict__ part, int M, int Hq, int pos_base,
                                                         int gc, int t0, __nv_bfloat16* __restrict__ out) {
  constexpr int PER = HD / 32;
  constexpr float c = 1.4426950408889634f / (HD == 256 ? 16.0f : HD == 128 ? 11.313708498984761f : 8.0f);
  pdl_launch();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int t = t0 + pair / Hq, head = pair % Hq;
  if (t >= M) return;
  const int n_g = attn_row_groups(pos_base + t, gc);  // 2 .. ATTN_MAX_GROUPS
  const float* base = part + ((size_t)t * Hq + head) * ATTN_MAX_GROUPS * (HD + 2);
  // lane g < n_g fetches group g's (m, l)
  float mg = -INFINITY, lg = 0.f;
  if (lane < n_g) {
    const float2 ml = *reinterpret_cast<const float2*>(base + (size_t)lane * (HD + 2) + HD);
    mg = ml.x;
    lg = ml.y;
  }
  float m = mg;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float wg = mg == -INFINITY ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(mg, m), c));
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float l = 0.f;
  for (int g0 = 0; g0 < n_g; g0 += 4) {
    float oj[4][PER];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float* p = base + (size_t)(g0 + k) * (HD + 2) + lane * PER;
#pragma unroll
      for (int i = 0; i < PER; i += 2) {
        float2 v = make_float2(0.f, 0.f);
        if (g0 + k < n_g) v = *reinterpret_cast<const float2*>(p + i);
        oj[k][i] = v.x;
        oj[k][i + 1] = v.y;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float w = __shfl_sync(0xffffffffu, wg, (g0 + k) & 31);
      const float lk = __shfl_sync(0xffffffffu, lg, (g0 + k) & 31);
      if (g0 + k >= n_g) continue;
      l = __fadd_rn(l, __fmul_rn(w, lk));
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(w, oj[k][i]));
    }
  }
  __nv_bfloat16* dst = out + (size_t)t * Hq * HD + (size_t)head * HD + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + i) =
        __floats2bfloat162_rn(__fdiv_rn(acc[i], l), __fdiv_rn(acc[i + 1], l));
}

// ---------------------------------------------------------------------------
// launchers

template <int HD, int NW>
static cudaError_t launch_prefill_t(const AttnArgs& a, float* part, cudaStream_t s) {
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
  const int gc = attn_group_chunks(a.kv_len);
  const int last_pos = a.pos_base + a.M - 1;
  const int n_groups = attn_row_groups(last_pos, gc);
  if (n_groups > 1 && !part) return cudaErrorInvalidValue;
  dim3 grid((rows + C::ROWS - 1) / C::ROWS, a.Hkv, n_groups);
  cudaError_t e = launch_k(attn_prefill_kernel<HD, NW>, grid, dim3(NW * 32), C::SMEM, s, 1, a, part, gc);
  if (e != cudaSuccess || n_groups == 1) return e;
  const int t0 = a.pos_base >= CHUNK * gc ? 0 : CHUNK * gc - a.pos_base;  // first row with two groups
  const int pairs = (a.M - t0) * a.Hq;
  return launch_k(attn_merge_kernel<HD>, dim3((pairs + 3) / 4), dim3(128), 0, s, 1,
                  static_cast<const float*>(part), a.M, a.Hq, a.pos_base, gc, t0, a.out);
}

static bool attn_shape_ok(const AttnArgs& a) {
  if (a.Hkv <= 0 || a.Hq % a.Hkv != 0) return false;
  const int G = a.Hq / a.Hkv;
  if (G > 16 || (16 % G) != 0) return false;
  if (a.pos_base < 0 || a.pos_base + a.M > a.kv_len) return false;
  return a.hd == 64 || a.hd == 256;
}

cudaError_t launch_attn_prefill(const AttnArgs& a, float* partials, cudaStream_t s) {
  if (a.M <= 0) return cudaSuccess;
  if (!attn_shape_ok(a)) return cudaErrorInvalidValue;
  if (a.hd == 256) return launch_prefill_t<256, 4>(a, partials, s);
  return launch_prefill_t<64, 4>(a, partials, s);
}

cudaError_t launch_attn_split(const AttnArgs& a, float* partials, cudaStream_t s) {
  if (a.M != 1) return cudaErrorInvalidValue;
  return launch_attn_prefill(a, partials, s);
}

int attn_launch_count(const AttnArgs& a) {
  if (a.M <= 0) return 0;
  return attn_row_groups(a.pos_base + a.M - 1, attn_group_chunks(a.kv_len)) > 1 ? 2 : 1;
}

size_t attn_partials_floats(int M, int Hq, int hd, int kv_len) {
  const int gc = attn_group_chunks(kv_len > 0 ? kv_len : 1);
  const int n_groups = attn_row_groups(kv_len > 0 ? kv_len - 1 : 0, gc);
  if (n_groups <= 1) return 0;
  return static_cast<size_t>(M > 0 ? M : 0) * Hq * ATTN_MAX_GROUPS * (hd + 2);
}

}  // namespace pf
