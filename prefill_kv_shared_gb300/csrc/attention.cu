// Causal grouped-query attention over the FP16 KV cache, on the 5th-generation
// tensor cores.
//
// MMA rows are (query, head-within-group) pairs: row R = t*G + g for query t
// and query head kvh*G + g, so the G query heads that share a KV head share
// the K/V tiles.  A CTA takes 128 rows (128/G queries) of one KV head.
//
// Keys are cut into absolute 64-key chunks, and the chunks into groups of gc
// consecutive chunks, gc fixed by the launch's key count and its number of
// row blocks (attn_group_chunks: at most ATTN_MAX_GROUPS groups, as many as
// keep the launch to one wave, at least ATTN_GC_MIN chunks a group).  A CTA handles one
// (128-row block, group) pair and runs the online softmax over the group's
// chunks in ascending order:
//     S = Q K^T (tcgen05.mma, TMEM), m' = max(m, max_k s_k),
//     p_k = fp16(2^((s_k - m') c)), l' = l 2^((m - m') c) + sum_k p_k,
//     O' = O 2^((m - m') c) + P V (the rescale in TMEM, P V by tcgen05.mma)
// with c = log2(e)/sqrt(hd).  A row whose keys lie in one group writes
// O * (1/l);
// otherwise each group's (O, m, l) goes to a partials buffer and
// attn_merge_kernel combines the row's group states.  So the causal work
// spreads over many CTAs instead of piling up on those of the last rows.
//
// A row's result depends only on its own position, the keys and gc: the MMA
// rows of a tile are independent and chunks past a row's position leave its
// state unchanged.  (Rows of a prompt cut into ubatches differently can see
// different gc, so such runs agree to rounding.)  The output row of a
// KV-shared layer does not come from this kernel in either pruning mode: the
// single-row kernels at the end of this file (attn_row_kernel) compute it, so
// that its bits are the same whether the layer carries one row or the whole
// ubatch.
//
// CTA roles: warp 1 lane 0 issues the TMA copies of Q (once) and of K, warp
// 6 lane 0 those of V (K on a 3-stage ring, V double-buffered, on separate
// barriers: a K buffer is free again once S = Q K^T has read it, a V buffer
// once P V has); warp 0 allocates TMEM and its lane 0 issues the MMAs;
// warps 2..5 own the 128 rows (thread = TMEM lane = row): softmax, the P
// tile (fp16, written to TMEM next to O: the A operand of P V comes from
// TMEM, which leaves the shared memory of a P tile to the K ring), the O
// rescale and the output.  The MMA thread issues S(j+1) = Q K(j+1)^T before P(j) V(j), so
// the tensor cores work while the row warps run the softmax of chunk j.  All
// waits are bounded (PF_WAIT_CYCLES); a timed-out wait flags the error word
// and the CTA unwinds.
#include "common.cuh"
#include "kernels.h"

#include <string>

namespace pf {

constexpr int CHUNK = 64;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// partials layout: [row t][query head][group (ATTN_MAX_GROUPS)][HD + 4] =
// o[HD] (not normalised), m, l, 2 pad (16-byte aligned rows)
constexpr int ATTN_MAX_GROUPS = 4;
__host__ __device__ constexpr int attn_part_stride(int hd) { return hd + 4; }

// A group holds at least this many chunks: a group's partial state and its
// merge cost more than a short chain of chunks (E2B, 512 rows over 512 keys:
// two groups of four chunks 21.0 us, four groups of two 22.3 us).
constexpr int ATTN_GC_MIN = 4;

static int attn_sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

int attn_group_chunks(int kv_len, int row_ctas) {
  const int n_chunks = (kv_len + CHUNK - 1) / CHUNK;
  // as many groups as keep the launch to one wave of CTAs (E4B, 1024 rows
  // over 1024 keys: 128 CTAs in two groups 26.9 us, 256 in four 36.0 us)
  int groups = ATTN_MAX_GROUPS;
  const int sms = attn_sm_count();
  while (groups > 1 && row_ctas * groups > sms) --groups;
  int gc = (n_chunks + groups - 1) / groups;
  if (gc < ATTN_GC_MIN) gc = ATTN_GC_MIN;
  return gc;
}

// CTAs over (128-row block, KV head) of a prefill launch
static int attn_row_ctas(const AttnArgs& a) { return (a.M * (a.Hq / a.Hkv) + 127) / 128 * a.Hkv; }

// groups that hold keys of the row at position pos
__host__ __device__ __forceinline__ int attn_row_groups(int pos, int gc) { return (pos / CHUNK) / gc + 1; }

template <int HD>
__host__ __device__ constexpr float attn_c() {
  return 1.4426950408889634f / (HD == 256 ? 16.0f : HD == 128 ? 11.313708498984761f : 8.0f);
}

// ---------------------------------------------------------------------------
// the tcgen05 kernel

template <int HD>
struct AttnTcCfg {
  static constexpr int NB = HD / 64;               // 64-dim (128-byte) boxes per row
  static constexpr int Q_BYTES = 128 * HD * 2;      // [box][128 rows][128 B]
  static constexpr int KV_BYTES = CHUNK * HD * 2;   // one K or V chunk: [box][64 keys][128 B]
  static constexpr int NK = 3;                      // K ring stages (V: 2)
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + 2 * KV_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + barriers, + alignment slack
  static constexpr int TMEM_S = 0;                  // two S buffers of 64 columns
  static constexpr int TMEM_O = 2 * CHUNK;          // O: HD columns
  static constexpr int TMEM_P = TMEM_O + HD;        // two P buffers of 32 columns (64 fp16 a row)
  static constexpr int TMEM_COLS = (TMEM_P + CHUNK) <= 256 ? 256 : 512;
  static_assert(TMEM_P + CHUNK <= 512, "TMEM");
  static constexpr int THREADS = 224;
  static_assert(SMEM <= 232448, "shared memory");
};

// 128-byte-swizzled operand descriptor with explicit leading / stride byte
// offsets (MN-major: LBO = bytes between 64-element atoms along MN, SBO =
// bytes between 8-row groups along K)
__device__ __forceinline__ uint64_t sdesc_sw128_lbo_sbo(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(lbo >> 4) << 16;
  d |= static_cast<uint64_t>(sbo >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// D[tmem] (+)= A[tmem] * B[smem] (kind::f16), A in TMEM: its rows are the
// TMEM lanes, two 16-bit elements of a row per 32-bit column (the lower k
// in the low half), K = 16 per instruction (8 columns)
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// kind::f16 instruction descriptor, fp16 A and B, fp32 accumulator; b_mn:
// B is MN-major (V stored [key][dim] is the B operand of P V)
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool b_mn) {
  return (1u << 4) | (b_mn ? (1u << 16) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// 32 lanes x 32 consecutive 32-bit columns from registers (thread i -> lane i)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// let issued MMAs finish before TMEM is freed on an error path (bounded;
// `bar` completes once, on the commit that follows them)
__device__ __forceinline__ void attn_drain(uint64_t* bar) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, 0)) {
    if (clock64() - t0 > 400000000ll) return;  // about 0.2 s
  }
}

struct AttnTcShape {
  int M, Hq, Hkv, pos_base, gc;
};

template <int HD>
__global__ void __launch_bounds__(AttnTcCfg<HD>::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnTcShape sh, __nv_bfloat16* __restrict__ out,
                   float* __restrict__ part, int* err) {
  using C = AttnTcCfg<HD>;
  constexpr float cexp = attn_c<HD>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;        // 1
  uint64_t* k_full = bars + 1;    // NK
  uint64_t* k_empty = bars + 4;   // NK
  uint64_t* v_full = bars + 7;    // 2
  uint64_t* v_empty = bars + 9;   // 2
  uint64_t* s_full = bars + 11;   // 2
  uint64_t* s_free = bars + 13;   // 2
  uint64_t* p_full = bars + 15;   // 2
  uint64_t* pv_done = bars + 17;  // 2
  uint64_t* drain = bars + 19;    // 1, error path only
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  static_assert(C::NK == 3, "barrier layout");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = sh.Hq / sh.Hkv;
  const int kvh = blockIdx.y, grp = blockIdx.z;
  const int R0 = blockIdx.x * 128;
  const int t0 = R0 / G;
  const int t_last = min(sh.M - 1, (R0 + 127) / G);
  const int last_ch = (sh.pos_base + t_last) / CHUNK;
  const int ch_first = grp * sh.gc;
  pdl_launch();
  if (ch_first > last_ch) return;  // no keys of this group reach the block's rows
  const int ch_end = min(last_ch, ch_first + sh.gc - 1);
  const int n = ch_end - ch_first + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int b = 0; b < C::NK; ++b) {
      mbar_init(&k_full[b], 1);
      mbar_init(&k_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&v_full[b], 1);
      mbar_init(&v_empty[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 4);
      mbar_init(&p_full[b], 4);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == 0) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp == 1 || warp == 6) {
    // ---------------- TMA producers: Q and K (warp 1), V (warp 6)
    if (lane == 0) {
      const bool is_k = warp == 1;
      bool ok = true;
      // one copy per tile: the maps list the 64-dim box index last, so a
      // copy lands as [box][rows][128 B]
      if (is_k) {
        mbar_arrive_expect_tx(q_full, C::Q_BYTES);
        tma_load_4d(smem, &tmQ, q_full, 0, kvh * G, t0, 0);
      }
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = smem + (is_k ? C::OFF_K : C::OFF_V);
      const CUtensorMap* map = is_k ? &tmK : &tmV;
      const int ns = is_k ? C::NK : 2;  // ring stages
      for (int j = 0; j < n && ok; ++j) {
        const int s = j % ns;
        if (j >= ns) ok = mbar_wait(&empty[s], ((j - ns) / ns) & 1, err, PF_DEV_TIMEOUT_PRODUCER);
        if (!ok) break;
        mbar_arrive_expect_tx(&full[s], C::KV_BYTES);
        tma_load_3d(ring + s * C::KV_BYTES, map, &full[s], kvh * HD, (ch_first + j) * CHUNK, 0);
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    // ---------------- MMA issue: the whole warp runs the loop in step
    // (waits and decisions warp-uniform), one lane elected once issues the
    // MMAs and commits (its commits track the MMAs it issued); an issue
    // from a lone lane's divergent loop costs several times as much
    {
      const bool leader = elect_one();
      constexpr uint32_t id_qk = idesc_f16_f32(128, CHUNK, false);
      constexpr uint32_t id_pv = idesc_f16_f32(128, HD, true);
      const uint32_t sq = smem_u32(smem);
      bool ok = mbar_wait(q_full, 0, err, PF_DEV_TIMEOUT_MMA);
      ok = __all_sync(0xffffffffu, ok);
      bool issued = false;
      // step i: S(i) = Q K(i)^T (if i < n), then O (+)= P(i-1) V(i-1)
      for (int i = 0; i <= n && ok; ++i) {
        if (i < n) {
          const int s = i & 1, sk_i = i % C::NK;
          ok = mbar_wait(&k_full[sk_i], (i / C::NK) & 1, err, PF_DEV_TIMEOUT_MMA);
          if (ok && i >= 2) ok = mbar_wait(&s_free[s], ((i - 2) >> 1) & 1, err, PF_DEV_TIMEOUT_MMA);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sk = smem_u32(smem + C::OFF_K + sk_i * C::KV_BYTES);
          // descriptors built once per tile, constant offsets per step (the
          // address field holds any shared-memory address: no carry)
          const uint64_t qd0 = sdesc_sw128(sq), kd0 = sdesc_sw128(sk);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
              const int b = kk >> 2, w = kk & 3;  // 64-dim box, 16-dim step within it
              tc_mma_f16(tmem + C::TMEM_S + s * CHUNK, qd0 + ((b * (128 * 128) + w * 32) >> 4),
                         kd0 + ((b * (CHUNK * 128) + w * 32) >> 4), id_qk, kk > 0 ? 1u : 0u);
            }
            tc_commit(&s_full[s]);
            tc_commit(&k_empty[sk_i]);  // K(i) has been read
          }
          __syncwarp();
          issued = true;
        }
        if (i >= 1) {
          const int j = i - 1, s = j & 1;
          ok = mbar_wait(&p_full[s], (j >> 1) & 1, err, PF_DEV_TIMEOUT_MMA);
          if (ok) ok = mbar_wait(&v_full[s], (j >> 1) & 1, err, PF_DEV_TIMEOUT_MMA);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sv = smem_u32(smem + C::OFF_V + s * C::KV_BYTES);
          const uint64_t vd0 = sdesc_sw128_lbo_sbo(sv, CHUNK * 128, 1024);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < CHUNK / 16; ++kk)  // 16 keys a step: 8 TMEM columns of P
              tc_mma_f16_ts(tmem + C::TMEM_O, tmem + C::TMEM_P + s * (CHUNK / 2) + kk * 8,
                            vd0 + ((kk * 16 * 128) >> 4), id_pv, (j > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&pv_done[s]);
            tc_commit(&v_empty[s]);
          }
          __syncwarp();
        }
      }
      if (!ok && issued && leader) {
        // the MMAs already issued finish before TMEM is freed
        tc_commit(drain);
        attn_drain(drain);
      }
    }
    __syncwarp();
  } else {
    // ---------------- rows (warps 2..5: TMEM lane quarter warp % 4)
    const int qw = warp & 3;
    const int r = 32 * qw + lane;
    const int R = R0 + r;
    const int t = R / G, head = kvh * G + R % G;
    const int pos = t < sh.M ? sh.pos_base + t : -1;
    const uint32_t lane_base = static_cast<uint32_t>(32 * qw) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      const int s = j & 1;
      const int ch = ch_first + j;
      if (lane == 0) ok = mbar_wait(&s_full[s], (j >> 1) & 1, err, PF_DEV_TIMEOUT_EPILOGUE);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(tmem + lane_base + C::TMEM_S + s * CHUNK, sr[0]);
      tmem_ld32(tmem + lane_base + C::TMEM_S + s * CHUNK + 32, sr[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[s]);
      // keys ch*64 + k visible to this row: k < nvis
      const int nvis = pos < 0 ? 0 : min(CHUNK, pos - ch * CHUNK + 1);
      // the chunk's max and sum over eight interleaved partials (fixed
      // combination order): one thread owns the row, and a 64-long chain
      // of dependent operations would set the softmax's pace
      float mx[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mx[q] = -INFINITY;
#pragma unroll
      for (int k = 0; k < CHUNK; ++k)
        if (k < nvis) mx[k & 7] = fmaxf(mx[k & 7], __uint_as_float(sr[k >> 5][k & 31]));
      const float mj =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // The running max moves only when this chunk's max passes it by more
      // than 2^8 in the exponent (or on the row's first visible keys): then
      // O and l are rescaled; otherwise P is taken against the old max
      // (p <= 2^8, exact in fp16 range) and O needs no touch, so the P V of
      // successive chunks go to the tensor cores back to back.  O / l is the
      // same softmax either way.
      const bool grow = mj != -INFINITY && (m == -INFINITY || __fmul_rn(__fsub_rn(mj, m), cexp) > 8.f);
      const float mn = grow ? mj : m;
      float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pw[32];  // 64 fp16 probabilities, two per word
#pragma unroll
      for (int k2 = 0; k2 < 32; ++k2) {
        const int k = 2 * k2;
        const float s0 = __uint_as_float(sr[k >> 5][k & 31]), s1 = __uint_as_float(sr[(k + 1) >> 5][(k + 1) & 31]);
        const float p0 = k < nvis ? ex2_approx(__fmul_rn(__fsub_rn(s0, mn), cexp)) : 0.f;
        const float p1 = k + 1 < nvis ? ex2_approx(__fmul_rn(__fsub_rn(s1, mn), cexp)) : 0.f;
        const __half2 h = __floats2half2_rn(p0, p1);
        pw[k2] = *reinterpret_cast<const uint32_t*>(&h);
        ls[k2 & 7] = __fadd_rn(ls[k2 & 7], __fadd_rn(__low2float(h), __high2float(h)));
      }
      const float lc = __fadd_rn(__fadd_rn(__fadd_rn(ls[0], ls[1]), __fadd_rn(ls[2], ls[3])),
                                 __fadd_rn(__fadd_rn(ls[4], ls[5]), __fadd_rn(ls[6], ls[7])));
      const bool resc = grow && m != -INFINITY;  // an earlier max to move away from
      const float scale = resc ? ex2_approx(__fmul_rn(__fsub_rn(m, mn), cexp)) : 1.f;
      l = __fadd_rn(__fmul_rn(l, scale), lc);
      m = mn;
      // P(j) goes to buffer s once P V(j-2) has read it
      if (j >= 2) {
        if (lane == 0) ok = mbar_wait(&pv_done[s], ((j - 2) >> 1) & 1, err, PF_DEV_TIMEOUT_EPILOGUE);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      tmem_st32(tmem + lane_base + C::TMEM_P + s * (CHUNK / 2), pw);
      tmem_st_wait();
      // O *= scale once P V(j-1) has landed (chunk 0 overwrites O), only in
      // the warps where a row moved its max.  (Skipping the wait elsewhere is
      // safe: P V(j+1) cannot complete before P(j+1) is written, so the next
      // wait on this barrier still finds the phase it expects.)
      if (j >= 1 && __any_sync(0xffffffffu, resc)) {
        if (lane == 0) ok = mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, err, PF_DEV_TIMEOUT_EPILOGUE);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t x[32];
          tmem_ld32(tmem + lane_base + C::TMEM_O + 32 * c, x);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 32; ++q) x[q] = __float_as_uint(__fmul_rn(__uint_as_float(x[q]), scale));
          tmem_st32(tmem + lane_base + C::TMEM_O + 32 * c, x);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[s]);
    }
    // the group's state of each row
    if (ok) {
      if (lane == 0) ok = mbar_wait(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, err, PF_DEV_TIMEOUT_EPILOGUE);
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (ok) {
      // Each 32 x 32 block of O goes through a warp-private staging buffer
      // in the (now idle) K ring, so that the global stores cover whole row
      // segments: lane l stores rows 4i + l/8, columns 4(l%8) .. +3.
      tc_fence_after();
      // this lane's row: 0 = nothing to write, 1 = output row, 2 = group state
      const int n_g = pos >= 0 ? attn_row_groups(pos, sh.gc) : 0;
      const int kind_own = pos < 0 ? 0 : (n_g == 1 ? 1 : (grp < n_g ? 2 : 0));
      const float inv_l = kind_own == 1 ? __frcp_rn(l) : 1.f;  // output rows: O * (1/l)
      // destinations of the rows this lane writes in the transposed layout
      // (rows 4i + lane/8), fetched once from the rows' own lanes
      const size_t own_off = kind_own == 1 ? (size_t)t * sh.Hq * HD + (size_t)head * HD
                                           : (((size_t)t * sh.Hq + head) * ATTN_MAX_GROUPS + grp) * attn_part_stride(HD);
      const int rs = lane >> 3, pc = lane & 7;
      size_t dst_off[8];
      int dst_kind[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + rs;
        dst_kind[i] = __shfl_sync(0xffffffffu, kind_own, rr);
        const uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(own_off), rr);
        const uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(own_off >> 32), rr);
        dst_off[i] = (static_cast<size_t>(hi) << 32) | lo;
      }
      uint8_t* stg = smem + C::OFF_K + qw * 4096;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t x[32];
        tmem_ld32(tmem + lane_base + C::TMEM_O + 32 * c, x);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(stg + lane * 128 + ((q ^ (lane & 7)) << 4)) =
              make_float4(__fmul_rn(__uint_as_float(x[4 * q]), inv_l), __fmul_rn(__uint_as_float(x[4 * q + 1]), inv_l),
                          __fmul_rn(__uint_as_float(x[4 * q + 2]), inv_l), __fmul_rn(__uint_as_float(x[4 * q + 3]), inv_l));
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = 4 * i + rs;
          if (dst_kind[i] == 0) continue;
          const float4 v = *reinterpret_cast<const float4*>(stg + rr * 128 + ((pc ^ (rr & 7)) << 4));
          if (dst_kind[i] == 1) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
            *reinterpret_cast<uint2*>(out + dst_off[i] + 32 * c + 4 * pc) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
          } else {
            *reinterpret_cast<float4*>(part + dst_off[i] + 32 * c + 4 * pc) = v;
          }
        }
        __syncwarp();
      }
      if (kind_own == 2) *reinterpret_cast<float2*>(part + own_off + HD) = make_float2(m, l);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// merge

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
  constexpr float c = attn_c<HD>();
  pdl_launch();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int t = t0 + pair / Hq, head = pair % Hq;
  if (t >= M) return;
  const int n_g = attn_row_groups(pos_base + t, gc);  // 2 .. ATTN_MAX_GROUPS
  const float* base = part + ((size_t)t * Hq + head) * ATTN_MAX_GROUPS * attn_part_stride(HD);
  // lane g < n_g fetches group g's (m, l)
  float mg = -INFINITY, lg = 0.f;
  if (lane < n_g) {
    const float2 ml = *reinterpret_cast<const float2*>(base + (size_t)lane * attn_part_stride(HD) + HD);
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
      const float* p = base + (size_t)(g0 + k) * attn_part_stride(HD) + lane * PER;
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
  const float inv_l = __frcp_rn(l);
#pragma unroll
  for (int i = 0; i < PER; i += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + i) =
        __floats2bfloat162_rn(__fmul_rn(acc[i], inv_l), __fmul_rn(acc[i + 1], inv_l));
}

// ---------------------------------------------------------------------------
// launchers

template <int HD>
static cudaError_t launch_tc_t(const AttnArgs& a, float* part, cudaStream_t s) {
  using C = AttnTcCfg<HD>;
  {
    const cudaError_t e = smem_opt_in<attn_tc_kernel<HD>>(C::SMEM);
    if (e != cudaSuccess) return e;
  }
  const int G = a.Hq / a.Hkv;
  // Q viewed as [64-dim box][query][head][64 dims]; K and V as [64-dim
  // box][key][64 dims] (the box dimension listed last, its stride 128 B), so
  // that one copy brings a whole tile as [box][rows][128 B]; keys past kv_len
  // read as zeros
  CUtensorMap tq, tk, tv;
  std::string err;
  {
    const uint64_t dims[4] = {64, static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(a.M),
                              static_cast<uint64_t>(HD / 64)};
    const uint64_t st[3] = {static_cast<uint64_t>(HD) * 2, static_cast<uint64_t>(a.Hq) * HD * 2, 128};
    const uint32_t box[4] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(128 / G),
                             static_cast<uint32_t>(HD / 64)};
    if (!encode_fp16_sw128(&tq, a.q, 4, dims, st, box, &err)) return cudaErrorInvalidValue;
  }
  {
    // the KV head's dims start at column kvh*HD: coordinate 0 of the
    // innermost dimension spans the whole row so the head offset fits in it
    const uint64_t dims[3] = {static_cast<uint64_t>(a.Hkv) * HD, static_cast<uint64_t>(a.kv_len),
                              static_cast<uint64_t>(HD / 64)};
    const uint64_t st[2] = {static_cast<uint64_t>(a.Hkv) * HD * 2, 128};
    const uint32_t box[3] = {64, CHUNK, static_cast<uint32_t>(HD / 64)};
    if (!encode_fp16_sw128(&tk, a.k, 3, dims, st, box, &err)) return cudaErrorInvalidValue;
    if (!encode_fp16_sw128(&tv, a.v, 3, dims, st, box, &err)) return cudaErrorInvalidValue;
  }
  AttnTcShape sh;
  sh.M = a.M;
  sh.Hq = a.Hq;
  sh.Hkv = a.Hkv;
  sh.pos_base = a.pos_base;
  sh.gc = attn_group_chunks(a.kv_len, attn_row_ctas(a));
  const int last_pos = a.pos_base + a.M - 1;
  const int n_groups = attn_row_groups(last_pos, sh.gc);
  if (n_groups > 1 && !part) return cudaErrorInvalidValue;
  const int rows = a.M * G;
  dim3 grid((rows + 127) / 128, a.Hkv, n_groups);
  cudaError_t e =
      launch_k(attn_tc_kernel<HD>, grid, dim3(C::THREADS), C::SMEM, s, 1, tq, tk, tv, sh, a.out, part, a.err);
  if (e != cudaSuccess || n_groups == 1) return e;
  const int t0 = a.pos_base >= CHUNK * sh.gc ? 0 : CHUNK * sh.gc - a.pos_base;  // first row with two groups
  const int pairs = (a.M - t0) * a.Hq;
  return launch_k(attn_merge_kernel<HD>, dim3((pairs + 3) / 4), dim3(128), 0, s, 1,
                  static_cast<const float*>(part), a.M, a.Hq, a.pos_base, sh.gc, t0, a.out);
}

static bool attn_shape_ok(const AttnArgs& a) {
  if (a.Hkv <= 0 || a.Hq <= 0 || a.Hq % a.Hkv != 0 || !a.err) return false;
  const int G = a.Hq / a.Hkv;
  if (G > 16 || (16 % G) != 0) return false;
  if (a.pos_base < 0 || a.pos_base + a.M > a.kv_len) return false;
  // TMA bases must be 16-byte aligned
  if ((reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.v)) & 15)
    return false;
  return a.hd == 64 || a.hd == 256;
}

cudaError_t launch_attn_prefill(const AttnArgs& a, float* partials, cudaStream_t s) {
  if (a.M <= 0) return cudaSuccess;
  if (!attn_shape_ok(a)) return cudaErrorInvalidValue;
  if (a.hd == 256) return launch_tc_t<256>(a, partials, s);
  return launch_tc_t<64>(a, partials, s);
}


// ---------------------------------------------------------------------------
// single-row attention: the output row of the KV-shared layers
//
// One query row at position pos reads keys [0, pos] of one layer's cache
// once, so its cost is the K/V bytes (G4 section 1: after the pruning the
// KV-shared layers carry only the output row).  The keys are cut into 64-key
// tiles and the tiles of each KV head into `splits` consecutive ranges, sized
// so that the clusters that fit on the GPU at once stream the cache together.  A CTA (range,
// KV head) copies its K and V tiles through a TMA ring, forms the scores of
// the KV head's G query heads and P V with mma.sync (m16n8k16: rows are the
// G query heads, zero rows above G; fp32 accumulation), runs the online
// softmax over its tiles and keeps its state (o unnormalised, m, l) per
// query head.  The states are then combined inside the same launch: the
// CTAs of a thread-block cluster (ATTN_ROW_CL consecutive ranges) fold their
// states through distributed shared memory, each rank one slice of the
// heads' dims, in rank order, into a cluster state in global memory; the
// last cluster of a KV head to finish (a ticket) merges the cluster states
// slice by slice, in cluster order, and writes the output row.  The range
// cut depends only on pos and the fold order is fixed, so the row gets the
// same bits from every pass that computes it.

constexpr int ATTN_ROW_THREADS = 256;
constexpr int ATTN_ROW_CL = 4;         // CTAs (ranges) per cluster
constexpr int ATTN_ROW_CLUSTERS = 36;  // clusters of 4 resident at once with this kernel's shared memory
                                       // (cudaOccupancyMaxActiveClusters on the GB300: 36)

template <int HD>
struct AttnRowCfg {
  static constexpr int KV_BYTES = CHUNK * HD * 2;  // one 64-key K or V tile: [64-dim box][key][128 B]
  static constexpr int STAGE = 2 * KV_BYTES;
  static constexpr int NST = HD >= 256 ? 3 : 4;    // ring stages
  static constexpr int S_LD = CHUNK + 4;           // score row stride, floats
  static constexpr int P_LD = CHUNK + 8;           // P row stride, halves (conflict-free fragment loads)
  // scores, P and the rescale factors are double-buffered by tile parity,
  // so one tile's P V overlaps the next tile's scores
  static constexpr int OFF_S = NST * STAGE;
  static constexpr int OFF_P = OFF_S + 2 * 16 * S_LD * 4;
  static constexpr int OFF_H = OFF_P + 2 * 16 * P_LD * 2;  // per head: m, l, then alpha x 2
  static constexpr int OFF_Q = OFF_H + 4 * 16 * 4;  // the KV head's query rows, fp16 [16][HD]
  static constexpr int OFF_BAR = OFF_Q + 16 * HD * 2;
  static constexpr int SMEM = OFF_BAR + NST * 8 + 1024;
  static_assert(STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(SMEM <= 232448, "shared memory");
};

struct AttnRowShape {
  int Hq, Hkv, pos, n_tiles, tps, splits;  // splits = n_cl * ATTN_ROW_CL ranges per KV head
  int n_cl;                                // clusters per KV head
};

// Work buffer of the single-row attention (floats): a ticket per KV head
// (ints, attn_row_ticket_words of them, zero before the first launch; every
// launch leaves them zero), then per (KV head, cluster) a cluster state:
// o [G][HD], then (m, l) per head, attn_row_cst_stride floats in all.
__host__ __device__ __forceinline__ int attn_row_ticket_words(int Hkv) { return (Hkv + 3) / 4 * 4; }
__host__ __device__ __forceinline__ int attn_row_cst_stride(int G, int HD) { return G * HD + 32; }

__device__ __forceinline__ uint32_t row_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void row_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// this CTA's shared-memory address as seen from cluster rank `rank`
__device__ __forceinline__ uint32_t row_mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_cluster_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// byte offset of (key r, dims d .. d+7) in a swizzled [64-dim box][64 keys][128 B] tile
__device__ __forceinline__ uint32_t tile_off(int r, int d) {
  return static_cast<uint32_t>((d >> 6) * (CHUNK * 128) + r * 128 + ((((d & 63) >> 3) ^ (r & 7)) << 4));
}

// bounded wait for a copy still in flight (error path: its shared memory
// must not be released while the copy writes it)
__device__ __forceinline__ void row_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (clock64() - t0 > 400000000ll) return;  // about 0.2 s
  }
}

template <int HD>
__global__ void __launch_bounds__(ATTN_ROW_THREADS, 1)
    attn_row_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __half* __restrict__ q, const AttnRowShape sh, float* __restrict__ work,
                    __nv_bfloat16* __restrict__ out, int* err) {
  using C = AttnRowCfg<HD>;
  constexpr float cexp = attn_c<HD>();
  constexpr int KS = HD / 16;  // 16-dim steps of Q K^T
  constexpr int NG = HD / 64;  // 8-dim column groups of P V per warp (the 8 warps split the dims)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sS0 = reinterpret_cast<float*>(smem + C::OFF_S);
  __half* sP0 = reinterpret_cast<__half*>(smem + C::OFF_P);
  float* sM = reinterpret_cast<float*>(smem + C::OFF_H);
  float* sL = sM + 16;
  float* sA0 = sL + 16;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y;
  const int G = sh.Hq / sh.Hkv;
  const int tile0 = split * sh.tps;
  const int nt = min(sh.n_tiles, tile0 + sh.tps) - tile0;

  pdl_launch();
  if (tid == 0) {
    for (int i = 0; i < C::NST; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (tid < 16) {
    sM[tid] = -INFINITY;
    sL[tid] = 0.f;
    sA0[tid] = 1.f;
    sA0[tid + 16] = 1.f;
  }
  for (int i = tid; i < 2 * 16 * C::P_LD / 2; i += ATTN_ROW_THREADS) reinterpret_cast<uint32_t*>(sP0)[i] = 0u;
  __syncthreads();
  pdl_wait();
  if (tid == 0) {
    for (int i = 0; i < nt && i < C::NST; ++i) {
      mbar_arrive_expect_tx(&full[i], C::STAGE);
      tma_load_3d(smem + i * C::STAGE, &tmK, &full[i], kvh * HD, (tile0 + i) * CHUNK, 0);
      tma_load_3d(smem + i * C::STAGE + C::KV_BYTES, &tmV, &full[i], kvh * HD, (tile0 + i) * CHUNK, 0);
    }
  }
  // Q fragments (A of Q K^T): row g is query head kvh*G + g, row g + 8 head
  // kvh*G + g + 8; rows past G are zero.  The KV head's G query rows come
  // in with one 16-byte load per thread and are read back from shared memory.
  uint32_t qa[KS][4];
  {
    __half* sQ = reinterpret_cast<__half*>(smem + C::OFF_Q);
    const uint4* qg = reinterpret_cast<const uint4*>(q + (size_t)kvh * G * HD);
    for (int i = tid; i < 16 * HD / 8; i += ATTN_ROW_THREADS)
      reinterpret_cast<uint4*>(sQ)[i] = i < G * HD / 8 ? qg[i] : make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const __half* q0 = sQ + g * HD;
    const __half* q1 = sQ + (g + 8) * HD;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d = ks * 16 + 2 * t4;
      qa[ks][0] = *reinterpret_cast<const uint32_t*>(q0 + d);
      qa[ks][1] = *reinterpret_cast<const uint32_t*>(q1 + d);
      qa[ks][2] = *reinterpret_cast<const uint32_t*>(q0 + d + 8);
      qa[ks][3] = *reinterpret_cast<const uint32_t*>(q1 + d + 8);
    }
  }
  float o[NG][4];
#pragma unroll
  for (int n = 0; n < NG; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  const int dw = warp * (HD / 8);  // the warp's first P V column
  int i = 0;
  bool ok = true;
  for (; i < nt; ++i) {
    const int st = i % C::NST;
    float* sS = sS0 + (i & 1) * 16 * C::S_LD;
    __half* sP = sP0 + (i & 1) * 16 * C::P_LD;
    float* sA = sA0 + (i & 1) * 16;
    ok = mbar_wait(&full[st], (i / C::NST) & 1, err, PF_DEV_TIMEOUT_MMA);
    // every warp is past its P V of tile i-1: that tile's stage is free
    ok = __syncthreads_and(ok);
    if (!ok) break;
    if (tid == 0 && i >= 1 && i - 1 + C::NST < nt) {
      const int sp = (i - 1) % C::NST;
      mbar_arrive_expect_tx(&full[sp], C::STAGE);
      tma_load_3d(smem + sp * C::STAGE, &tmK, &full[sp], kvh * HD, (tile0 + i - 1 + C::NST) * CHUNK, 0);
      tma_load_3d(smem + sp * C::STAGE + C::KV_BYTES, &tmV, &full[sp], kvh * HD, (tile0 + i - 1 + C::NST) * CHUNK,
                  0);
    }
    const uint8_t* kt = smem + st * C::STAGE;
    const uint32_t vt = smem_u32(kt + C::KV_BYTES);
    const int key0 = (tile0 + i) * CHUNK;
    {
      // scores of the warp's 8 keys (tile rows 8 warp .. +7): two
      // accumulation chains (even and odd 16-dim steps), added at the end
      float c[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      const int r = warp * 8 + g;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int d = ks * 16 + 2 * t4;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kt + tile_off(r, d) + (d & 7) * 2);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kt + tile_off(r, d + 8) + (d & 7) * 2);
        if (ks & 1)
          mma_16816(c1, qa[ks], b0, b1);
        else
          mma_16816(c, qa[ks], b0, b1);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) c[e] = __fadd_rn(c[e], c1[e]);
      const int kc = warp * 8 + 2 * t4;  // tile column of c[0] / c[2]
      const bool v0 = key0 + kc <= sh.pos, v1 = key0 + kc + 1 <= sh.pos;
      *reinterpret_cast<float2*>(sS + g * C::S_LD + kc) = make_float2(v0 ? c[0] : -INFINITY, v1 ? c[1] : -INFINITY);
      *reinterpret_cast<float2*>(sS + (g + 8) * C::S_LD + kc) =
          make_float2(v0 ? c[2] : -INFINITY, v1 ? c[3] : -INFINITY);
    }
    __syncthreads();
    // online softmax: warp w takes query heads w and w + 8 of the KV head
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = warp + 8 * hh;
      if (h >= G) continue;
      const float s0 = sS[h * C::S_LD + lane], s1 = sS[h * C::S_LD + lane + 32];
      float mt = fmaxf(s0, s1);
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, x));
      const float m_old = sM[h];
      const float m_new = fmaxf(m_old, mt);
      float p0 = 0.f, p1 = 0.f, alpha = 1.f;
      if (m_new != -INFINITY) {
        p0 = ex2_approx(__fmul_rn(__fsub_rn(s0, m_new), cexp));
        p1 = ex2_approx(__fmul_rn(__fsub_rn(s1, m_new), cexp));
        alpha = m_old == -INFINITY ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(m_old, m_new), cexp));
      }
      const __half h0 = __float2half_rn(p0), h1 = __float2half_rn(p1);
      float ps = __fadd_rn(__half2float(h0), __half2float(h1));  // the row sum adds the rounded values
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) ps = __fadd_rn(ps, __shfl_xor_sync(0xffffffffu, ps, x));
      sP[h * C::P_LD + lane] = h0;
      sP[h * C::P_LD + lane + 32] = h1;
      __syncwarp();
      if (lane == 0) {
        sL[h] = __fadd_rn(__fmul_rn(sL[h], alpha), ps);
        sM[h] = m_new;
        sA[h] = alpha;
      }
    }
    __syncthreads();
    {
      // O = O * alpha + P V over the warp's columns
      const float a0 = sA[g], a1 = sA[g + 8];
#pragma unroll
      for (int n = 0; n < NG; ++n) {
        o[n][0] = __fmul_rn(o[n][0], a0);
        o[n][1] = __fmul_rn(o[n][1], a0);
        o[n][2] = __fmul_rn(o[n][2], a1);
        o[n][3] = __fmul_rn(o[n][3], a1);
      }
#pragma unroll
      for (int kk = 0; kk < CHUNK / 16; ++kk) {
        uint32_t pa[4];
        pa[0] = *reinterpret_cast<const uint32_t*>(sP + g * C::P_LD + kk * 16 + 2 * t4);
        pa[1] = *reinterpret_cast<const uint32_t*>(sP + (g + 8) * C::P_LD + kk * 16 + 2 * t4);
        pa[2] = *reinterpret_cast<const uint32_t*>(sP + g * C::P_LD + kk * 16 + 8 + 2 * t4);
        pa[3] = *reinterpret_cast<const uint32_t*>(sP + (g + 8) * C::P_LD + kk * 16 + 8 + 2 * t4);
        if constexpr (NG >= 2) {
#pragma unroll
          for (int n = 0; n < NG; n += 2) {
            // matrices: (keys 0-7, cols d0), (keys 8-15, d0), (keys 0-7, d0+8), (keys 8-15, d0+8)
            const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int d = dw + 8 * n + (lane >> 4) * 8;
            uint32_t v0, v1, v2, v3;
            ldsm_x4_trans(vt + tile_off(r, d), v0, v1, v2, v3);
            mma_16816(o[n], pa, v0, v1);
            mma_16816(o[n + 1], pa, v2, v3);
          }
        } else {
          const int r = kk * 16 + (lane & 15);
          uint32_t v0, v1;
          ldsm_x2_trans(vt + tile_off(r, dw), v0, v1);
          mma_16816(o[0], pa, v0, v1);
        }
      }
    }
  }
  __syncthreads();  // the last tile's P V is done everywhere
  if (!ok) {
    // copies issued for tiles i .. (i == 0 ? NST : i - 1 + NST) - 1 may still be landing
    const int issued = i == 0 ? C::NST : i - 1 + C::NST;
    if (tid == 0)
      for (int j = i; j < nt && j < issued; ++j) row_drain(&full[j % C::NST], (j / C::NST) & 1);
    __syncthreads();
  }
  // This range's state in shared memory (the K/V ring is free now): o
  // [G][HD] (room for 16 heads), then (m, l) per head.  A range that gave up
  // a wait, or holds no keys, adds nothing (m = -inf).  Every CTA takes part
  // in the cluster steps below whatever happened before.
  __shared__ int s_last;
  float* sO = reinterpret_cast<float*>(smem);
  float* sML = sO + 16 * HD;
#pragma unroll
  for (int n = 0; n < NG; ++n) {
    const int d = dw + 8 * n + 2 * t4;
    if (g < G)
      *reinterpret_cast<float2*>(sO + g * HD + d) = ok ? make_float2(o[n][0], o[n][1]) : make_float2(0.f, 0.f);
    if (g + 8 < G)
      *reinterpret_cast<float2*>(sO + (g + 8) * HD + d) = ok ? make_float2(o[n][2], o[n][3]) : make_float2(0.f, 0.f);
  }
  if (tid < G) {
    sML[2 * tid] = ok ? sM[tid] : -INFINITY;
    sML[2 * tid + 1] = ok ? sL[tid] : 0.f;
  }
  __syncthreads();
  row_cluster_sync();  // the cluster's range states are in shared memory
  const uint32_t rank = row_cluster_rank();
  const int cl = split / ATTN_ROW_CL;
  const int GH = G * HD, SL = GH / ATTN_ROW_CL;  // rank r folds elements [r SL, (r+1) SL) of [G][HD]
  const int CST = attn_row_cst_stride(G, HD);
  float* cstates = work + attn_row_ticket_words(sh.Hkv);
  {
    float* cs = cstates + ((size_t)kvh * sh.n_cl + cl) * CST;
    uint32_t ro[ATTN_ROW_CL], rml[ATTN_ROW_CL];
#pragma unroll
    for (int r = 0; r < ATTN_ROW_CL; ++r) {
      ro[r] = row_mapa(smem_u32(sO), r);
      rml[r] = row_mapa(smem_u32(sML), r);
    }
    for (int e = static_cast<int>(rank) * SL + 2 * tid; e < static_cast<int>(rank + 1) * SL;
         e += 2 * ATTN_ROW_THREADS) {
      const int h = e / HD;
      float2 ml[ATTN_ROW_CL];
      float mx = -INFINITY;
#pragma unroll
      for (int r = 0; r < ATTN_ROW_CL; ++r) {
        ml[r] = ld_cluster_f32x2(rml[r] + 8u * h);
        mx = fmaxf(mx, ml[r].x);
      }
      float2 acc = make_float2(0.f, 0.f);
      float lacc = 0.f;
#pragma unroll
      for (int r = 0; r < ATTN_ROW_CL; ++r) {  // ranks in order
        const float w = ml[r].x == -INFINITY ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(ml[r].x, mx), cexp));
        const float2 v = ld_cluster_f32x2(ro[r] + 4u * e);
        acc.x = __fadd_rn(acc.x, __fmul_rn(w, v.x));
        acc.y = __fadd_rn(acc.y, __fmul_rn(w, v.y));
        lacc = __fadd_rn(lacc, __fmul_rn(w, ml[r].y));
      }
      *reinterpret_cast<float2*>(cs + e) = acc;
      if (e % HD == 0) *reinterpret_cast<float2*>(cs + GH + 2 * h) = make_float2(mx, lacc);
    }
  }
  __threadfence();
  __syncthreads();
  row_cluster_sync();  // the cluster state is in global memory; no rank reads another's shared memory after this
  if (rank == 0 && tid == 0) {
    int* tickets = reinterpret_cast<int*>(work);
    const int last = atomicAdd(&tickets[kvh], 1) == sh.n_cl - 1;
    if (last) tickets[kvh] = 0;  // every cluster of this KV head has counted: ready for the next launch
#pragma unroll
    for (int r = 0; r < ATTN_ROW_CL; ++r) st_cluster_u32(row_mapa(smem_u32(&s_last), r), last ? 1u : 0u);
  }
  row_cluster_sync();  // every rank holds the flag
  if (!s_last) return;
  __threadfence();
  // The last cluster: rank r merges slice r over the KV head's cluster
  // states, in cluster order; (m, l) of the clusters first go to shared memory.
  const float* cb = cstates + (size_t)kvh * sh.n_cl * CST;
  float2* sCML = reinterpret_cast<float2*>(smem);  // [n_cl][G]
  for (int i2 = tid; i2 < sh.n_cl * G; i2 += ATTN_ROW_THREADS) {
    const int c = i2 / G, h = i2 % G;
    sCML[i2] = __ldcg(reinterpret_cast<const float2*>(cb + (size_t)c * CST + GH + 2 * h));
  }
  __syncthreads();
  for (int e = static_cast<int>(rank) * SL + 2 * tid; e < static_cast<int>(rank + 1) * SL; e += 2 * ATTN_ROW_THREADS) {
    const int h = e / HD;
    float mx = -INFINITY;
    for (int c = 0; c < sh.n_cl; ++c) mx = fmaxf(mx, sCML[c * G + h].x);
    float2 acc = make_float2(0.f, 0.f);
    float lacc = 0.f;
    for (int c0 = 0; c0 < sh.n_cl; c0 += 8) {  // clusters in order, eight loads in flight
      float2 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = c0 + u < sh.n_cl ? __ldcg(reinterpret_cast<const float2*>(cb + (size_t)(c0 + u) * CST + e))
                                : make_float2(0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c0 + u >= sh.n_cl) break;
        const float2 ml = sCML[(c0 + u) * G + h];
        const float w = ml.x == -INFINITY ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(ml.x, mx), cexp));
        acc.x = __fadd_rn(acc.x, __fmul_rn(w, v[u].x));
        acc.y = __fadd_rn(acc.y, __fmul_rn(w, v[u].y));
        lacc = __fadd_rn(lacc, __fmul_rn(w, ml.y));
      }
    }
    const float inv = __frcp_rn(lacc);
    *reinterpret_cast<__nv_bfloat162*>(out + (size_t)kvh * GH + e) =
        __floats2bfloat162_rn(__fmul_rn(acc.x, inv), __fmul_rn(acc.y, inv));
  }
}

// tiles per range, ranges and clusters per KV head for a row at position
// pos: the ranges of all KV heads aim at the clusters that fit at once
static void attn_row_split(int pos, int Hkv, int* n_tiles, int* tps, int* splits, int* n_cl) {
  const int nt = pos / CHUNK + 1;
  int per_head = (ATTN_ROW_CLUSTERS / (Hkv > 0 ? Hkv : 1)) * ATTN_ROW_CL;
  if (per_head < ATTN_ROW_CL) per_head = ATTN_ROW_CL;
  const int t = (nt + per_head - 1) / per_head;
  const int ranges = (nt + t - 1) / t;
  *n_tiles = nt;
  *tps = t;
  *n_cl = (ranges + ATTN_ROW_CL - 1) / ATTN_ROW_CL;
  *splits = *n_cl * ATTN_ROW_CL;
}

// Enough for a row at any position up to pos: a row's ranges are at most
// its tile count and at most the per-head share, whatever the cut.
size_t attn_split_partials_floats(int Hq, int Hkv, int hd, int pos) {
  if (pos < 0 || Hkv < 1 || Hq < Hkv) return 0;
  const int nt = pos / CHUNK + 1;
  int per_head = (ATTN_ROW_CLUSTERS / Hkv) * ATTN_ROW_CL;
  if (per_head < ATTN_ROW_CL) per_head = ATTN_ROW_CL;
  const int ranges_max = nt < per_head ? nt : per_head;
  const int n_cl_max = (ranges_max + ATTN_ROW_CL - 1) / ATTN_ROW_CL;
  return static_cast<size_t>(attn_row_ticket_words(Hkv)) +
         static_cast<size_t>(Hkv) * n_cl_max * attn_row_cst_stride(Hq / Hkv, hd);
}

size_t attn_split_ticket_bytes(int Hkv) { return static_cast<size_t>(attn_row_ticket_words(Hkv)) * 4; }

template <int HD>
static cudaError_t launch_row_t(const AttnArgs& a, float* part, cudaStream_t s) {
  using C = AttnRowCfg<HD>;
  {
    const cudaError_t e = smem_opt_in<attn_row_kernel<HD>>(C::SMEM);
    if (e != cudaSuccess) return e;
  }
  // K and V as [64-dim box][key][64 dims] (the box dimension last, stride
  // 128 B): one copy brings a 64-key tile of one KV head as [box][key][128 B]
  CUtensorMap tk, tv;
  std::string err;
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(a.Hkv) * HD, static_cast<uint64_t>(a.kv_len),
                              static_cast<uint64_t>(HD / 64)};
    const uint64_t st[2] = {static_cast<uint64_t>(a.Hkv) * HD * 2, 128};
    const uint32_t box[3] = {64, CHUNK, static_cast<uint32_t>(HD / 64)};
    if (!encode_fp16_sw128(&tk, a.k, 3, dims, st, box, &err)) return cudaErrorInvalidValue;
    if (!encode_fp16_sw128(&tv, a.v, 3, dims, st, box, &err)) return cudaErrorInvalidValue;
  }
  AttnRowShape sh;
  sh.Hq = a.Hq;
  sh.Hkv = a.Hkv;
  sh.pos = a.pos_base;
  attn_row_split(a.pos_base, a.Hkv, &sh.n_tiles, &sh.tps, &sh.splits, &sh.n_cl);
  return launch_k(attn_row_kernel<HD>, dim3(sh.splits, a.Hkv), dim3(ATTN_ROW_THREADS), C::SMEM, s, ATTN_ROW_CL, tk,
                  tv, a.q, sh, part, a.out, a.err);
}

cudaError_t launch_attn_split(const AttnArgs& a, float* partials, cudaStream_t s) {
  if (a.M != 1 || !partials) return cudaErrorInvalidValue;
  if (!attn_shape_ok(a)) return cudaErrorInvalidValue;
  if (a.hd == 256) return launch_row_t<256>(a, partials, s);
  return launch_row_t<64>(a, partials, s);
}

int attn_launch_count(const AttnArgs& a) {
  if (a.M <= 0) return 0;
  return attn_row_groups(a.pos_base + a.M - 1, attn_group_chunks(a.kv_len, attn_row_ctas(a))) > 1 ? 2 : 1;
}

size_t attn_partials_floats(int M, int Hq, int hd, int kv_len) {
  // a launch of up to M rows over up to kv_len keys: several groups are
  // possible once the keys need more than one group of the minimum size
  if (kv_len <= CHUNK * ATTN_GC_MIN) return 0;
  return static_cast<size_t>(M > 0 ? M : 0) * Hq * ATTN_MAX_GROUPS * attn_part_stride(hd);
}

}  // namespace pf
