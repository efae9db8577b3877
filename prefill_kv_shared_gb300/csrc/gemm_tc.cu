// Dense GEMM on the 5th-generation tensor cores (tcgen05, TMEM accumulators)
// for the projections of the prefill pass: QKV, O, gate/up, down, the
// per-layer-embedding gate and projection, and the tied LM head.
//
//   out = A[M, K] (bf16, K-major) x W[N, K]^T, fp32 accumulation in TMEM.
//
// Weights are Q4_0 (32-element blocks, fp16 scale d, value d*(nibble-8)) or
// bf16.  Q4_0 tiles arrive by one bulk copy per 64-wide k-block into a raw
// ring; dequant warps expand them to bf16 straight into the 128-byte-swizzled
// K-major layout the MMA reads (B ring).  A (and bf16 W) tiles come in by TMA
// with the same swizzle (A ring).  The three rings are released separately:
// the raw ring by the dequant warps, the A and B rings by the MMA commits,
// so weight fetches run far ahead of the tensor cores.
//
// Persistent CTAs (one per SM) walk work units (m-block, n-tile, k-split):
//   warp 0        TMA / bulk-copy producer
//   warp 1        TMEM allocation, MMA issue (one lane), commits
//   warps 4..11   epilogue (two per TMEM lane quarter, splitting the column
//                 chunks): TMEM -> registers -> shared-memory staging ->
//                 fused epilogue with coalesced global accesses; TMEM
//                 accumulators are double buffered when they fit, so a
//                 unit's epilogue overlaps the next unit's main loop
//   warps 2, 3, 12..15  Q4_0 -> bf16 dequant
//
// Split-K: a weight matrix may be cut into S k-ranges (S fixed per matrix
// shape, never per M), run by the S CTAs of a thread-block cluster; ranks
// 1..S-1 stage their fp32 partial tiles in their own shared memory and move
// the real rows into rank 0's with bulk copies (distributed shared memory),
// and rank 0 adds them to its own in ascending rank order before the
// epilogue.
//
// Determinism: every output element is produced by the same sequence of
// MMAs over k (64-wide blocks in ascending order, four K=16 steps each, the
// same split boundaries and the same split order) whatever M is, so a row's
// result does not depend on how many rows the launch carries.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

#include <cstring>
#include <mutex>

namespace pf {

// Roles sit on warpgroup boundaries so that registers can be moved between
// them (setmaxnreg): warpgroups 1 and 2 (warps 4..11) run the epilogue with
// EPI_REGS registers a thread; warpgroups 0 and 3 (producer, MMA and the
// dequant warps 2, 3, 12..15) give theirs up down to LEAN_REGS.  The launch
// holds GEMM_THREADS x 128 = 65536 registers, and
// 2 x 128 x (LEAN_REGS + EPI_REGS) must not exceed that.
constexpr int GEMM_WARPS = 16;
constexpr int GEMM_THREADS = GEMM_WARPS * 32;
constexpr int EPI_WARP0 = 4;  // warps 4..11: epilogue, two per TMEM lane quarter
constexpr int EPI_WARPS = 8;
constexpr int DQ_THREADS = 192;  // warps 2, 3, 12..15: Q4_0 dequant
constexpr int EPI_REGS = 176;
constexpr int LEAN_REGS = 80;
static_assert(2 * 128 * (EPI_REGS + LEAN_REGS) <= GEMM_THREADS * 128, "register split exceeds the launch's registers");
static_assert(EPI_REGS % 8 == 0 && LEAN_REGS % 8 == 0 && LEAN_REGS >= 24 && EPI_REGS <= 256, "setmaxnreg range");

__device__ __forceinline__ bool is_epi_warp(int w) { return w >= EPI_WARP0 && w < EPI_WARP0 + EPI_WARPS; }
// dequant thread index 0..DQ_THREADS-1 of a thread in warps 2, 3, 12..15
__device__ __forceinline__ int dq_index(int w, int lane) { return (w < 4 ? w - 2 : w - 10) * 32 + lane; }
constexpr int SMEM_LIMIT = 232448;

__host__ __device__ constexpr int pow2_cols(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

template <int WK, int BN, int MT>
struct GemmCfg {
  static constexpr bool Q4 = WK == W_Q4;
  // 64-wide k-blocks per pipeline stage: every stage costs the copy engine,
  // the barriers and the dequant warps a fixed amount whatever its size, so
  // narrow tiles take two k-blocks a stage where shared memory allows.
  static constexpr int KS = (Q4 && BN <= 128 && MT == 1) ? 2 : 1;
  static constexpr int A_KB = MT * 128 * 128;  // one k-block of A: MT tiles of 128 rows x 64 bf16
  static constexpr int BT_KB = BN * 128;       // one k-block of bf16 B (BN rows x 64)
  static constexpr int RAW_KB = Q4 ? BN * 36 : 0;
  static constexpr int A_BYTES = KS * A_KB;    // stage layouts: [k-block][M tile][128 x 128 B], [k-block][BN x 128 B]
  static constexpr int BT_BYTES = KS * BT_KB;
  static constexpr int RAW_BYTES = KS * RAW_KB;
  static constexpr int A_STAGE = A_BYTES + (Q4 ? 0 : BT_BYTES);
  // The dequantised B ring bounds how far the dequant warps run ahead of the
  // MMAs (B stage k+S_B is written once the MMAs of stage k are done); the
  // A ring takes what the B and raw rings and the epilogue staging leave.
  static constexpr int S_B =
      Q4 ? (BN >= 256 ? (MT == 2 ? 2 : 3) : BN == 192 ? 2 : KS == 2 ? (BN == 64 ? 4 : 2) : 4) : 0;
  static constexpr int S_R = Q4 ? (BN >= 192 ? 3 : KS == 2 ? (BN == 64 ? 6 : 3) : 6) : 0;
  static constexpr int NB = S_B > 0 ? S_B : 1;  // ring moduli (the rings are unused without Q4)
  static constexpr int NR = S_R > 0 ? S_R : 1;
  static constexpr int RAW_RING = (S_R * RAW_BYTES + 1023) / 1024 * 1024;
  static constexpr int EPI_BYTES = EPI_WARPS * 32 * 32 * 4;  // one 4 KB staging buffer per epilogue warp
  static constexpr int FIXED = S_B * BT_BYTES + RAW_RING + EPI_BYTES + 1024 + 512;
  static constexpr int S_A_FIT = (SMEM_LIMIT - FIXED) / A_STAGE;
  static constexpr int S_A = S_A_FIT > 8 ? 8 : S_A_FIT;
  static constexpr int SMEM_BYTES = S_A * A_STAGE + FIXED;
  static constexpr int ACC = MT * BN;
  static constexpr int ACC_BUFS = (2 * ACC <= 512) ? 2 : 1;
  static constexpr int TMEM_COLS = pow2_cols(ACC * ACC_BUFS);
  static_assert(S_A >= 2, "shared memory too small for two A stages");
  static_assert(ACC <= 512, "accumulators exceed TMEM");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "MMA N");
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
// the kernel

// Let copies already issued land before the CTA exits on an error path
// (bounded in time, ignoring the error flag).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (clock64() - t0 > 400000000ll) return;  // about 0.2 s
  }
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_smem, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem), "r"(rank));
  return r;
}
// Bulk copy from this CTA's shared memory to a cluster peer's, completing
// on the peer's mbarrier (both destination addresses from mapa).
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst),
               "r"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// barrier among the epilogue warps only
__device__ __forceinline__ void epi_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(EPI_WARPS * 32) : "memory");
}

struct GemmShape {
  int M, K;
  int n_tiles, m_blocks, splits, kb_per_split, n_units;
  int a_box_rows;  // rows of A one TMA box brings (16 for launches of at most 16 rows, else 128)
  // Failure-path check only (-1 otherwise): CTA 0's copy producer issues
  // nothing from this pipeline stage on, so a consumer's bounded wait has to
  // run out (no copy is left in flight for it).
  int withhold_stage;
};

// Byte offset of (chunk c, row r, 16-byte piece q) in a split partial slot:
// [chunk][row][32 floats], pieces XOR-swizzled by row so that a warp's
// 16-byte accesses hit all banks.
__device__ __forceinline__ uint32_t slot_off(int c, int r, int q) {
  return static_cast<uint32_t>(((c * 128 + r) << 7) + ((q ^ (r & 7)) << 4));
}

template <int WK, int BN, int MT>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ wq4, const GemmShape sh_in, const EpiParams ep_in, int* err) {
  using C = GemmCfg<WK, BN, MT>;
  // The launch parameters are read from shared-memory copies: fields of a
  // kernel parameter used through a reference are re-read from parameter
  // memory inside the loops, and a local copy of a struct this size lands in
  // local memory; both are slow next to a 220 KB shared-memory carve-out.
  __shared__ GemmShape s_sh;
  __shared__ EpiParams s_ep;
  if (threadIdx.x == 0) {
    s_sh = sh_in;
    s_ep = ep_in;
  }
  __syncthreads();
  const GemmShape& sh = s_sh;
  const EpiParams& ep = s_ep;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_ring = smem;
  uint8_t* b_ring = a_ring + C::S_A * C::A_STAGE;
  uint8_t* r_ring = b_ring + C::S_B * C::BT_BYTES;
  uint8_t* epi_stage = r_ring + C::RAW_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + C::EPI_BYTES);
  uint64_t* full_a = bars;
  uint64_t* empty_a = full_a + C::S_A;
  uint64_t* full_r = empty_a + C::S_A;
  uint64_t* empty_r = full_r + C::NR;
  uint64_t* bfull = empty_r + C::NR;
  uint64_t* bempty = bfull + C::NB;
  uint64_t* tfull = bempty + C::NB;
  uint64_t* tempty = tfull + 2;
  uint64_t* red_full = tempty + 2;  // split-K: rank 0's partials have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = sh.kb_per_split;
  const bool split_mode = sh.splits > 1;  // one unit per CTA, a cluster per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S_A; ++s) {
      mbar_init(&full_a[s], 1);
      mbar_init(&empty_a[s], 1);
    }
    for (int s = 0; s < C::S_R; ++s) {
      mbar_init(&full_r[s], 1);
      mbar_init(&empty_r[s], DQ_THREADS / 32);
    }
    for (int s = 0; s < C::S_B; ++s) {
      mbar_init(&bfull[s], DQ_THREADS / 32);
      mbar_init(&bempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], EPI_WARPS);
    }
    mbar_init(red_full, 1);
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
  bool epi_ok = true;
  pdl_launch();
  // split-K: bytes of one column chunk's real rows in a partial tile (one
  // 128-row unit per CTA in split mode)
  uint32_t split_chunk_bytes = 0;
  if (split_mode) {
    const int mb = (blockIdx.x / sh.splits) / sh.n_tiles;
    const int rows = sh.M - mb * 128 < 128 ? sh.M - mb * 128 : 128;
    split_chunk_bytes = static_cast<uint32_t>(rows) * 128u;
  }
  const int wg = warp >> 2;
  if (wg == 1 || wg == 2) {
    // ================ epilogue warpgroups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(EPI_REGS));
    {
      // ---------------- epilogue
      pdl_wait();
      const int qw = warp & 3;                 // TMEM lane quarter this warp may access
      const int ew = (warp - EPI_WARP0) >> 2;  // which of the quarter's two epilogue warps
      uint8_t* stage = epi_stage + (warp - EPI_WARP0) * EPI_STAGE_BYTES;
      uint32_t j = 0;
      for (int u = blockIdx.x; u < sh.n_units; u += gridDim.x, ++j) {
        const int t = u / sh.splits;
        const int nt = t % sh.n_tiles, mb = t / sh.n_tiles;
        const int m_base = mb * MT * 128;
        int mt_valid = (sh.M - m_base + 127) / 128;
        if (mt_valid > MT) mt_valid = MT;
        const int buf = C::ACC_BUFS == 2 ? (j & 1) : 0;
        bool ok = mbar_wait_sleep(&tfull[buf], (j / C::ACC_BUFS) & 1, err, PF_DEV_TIMEOUT_EPILOGUE, 128);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          epi_ok = false;
          break;
        }
        tc_fence_after();
        if (split_mode) break;  // the cluster reduction below takes it from here
        const uint32_t tq = tmem_base + (static_cast<uint32_t>(32 * qw) << 16) + buf * C::ACC;
        for (int mt = 0; mt < mt_valid; ++mt) {
          const int m0 = m_base + mt * 128 + 32 * qw;
          const int rv = sh.M - m0 < 32 ? sh.M - m0 : 32;
          run_epilogue<BN>(ep, m0, rv, nt, ew, stage, [&](int c, float(&v)[32]) {
            uint32_t x[32];
            tmem_ld32(tq + mt * BN + 32 * c, x);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(x[q]);
          });
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
    }
    if (split_mode) {
      // Split-K over the cluster: CTA rank r holds the partial of k-range r.
      // Ranks 1.. stage theirs in their own (now idle) ring memory and send the
      // real rows to rank 0's ring with bulk copies; rank 0 adds them to its
      // own in ascending rank order and runs the epilogue.
      const uint32_t rank = cluster_ctarank();
      const int t = blockIdx.x / sh.splits;
      const int nt = t % sh.n_tiles, mb = t / sh.n_tiles;
      const int m_base = mb * 128;  // one 128-row tile per unit in split mode
      const int rows = sh.M - m_base < 128 ? sh.M - m_base : 128;
      const uint32_t chunk_bytes = split_chunk_bytes;
      const uint32_t slot_bytes = 128u * BN * 4u;
      cluster_sync_all();  // rank 0's expected byte count is posted by its producer warp
      const bool epi_warp = true;
      const int qw = warp & 3;
      const int ew = (warp - EPI_WARP0) >> 2;
      const int r = 32 * qw + lane;
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(32 * qw) << 16);
      if (epi_warp && rank != 0) {
        if (epi_ok && 32 * qw < rows) {
          for (int c = ew; c < BN / 32; c += 2) {
            uint32_t x[32];
            tmem_ld32(tq + 32 * c, x);
            tmem_ld_wait();
            if (r < rows) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(a_ring + slot_off(c, r, q)) =
                    make_float4(__uint_as_float(x[4 * q]), __uint_as_float(x[4 * q + 1]), __uint_as_float(x[4 * q + 2]),
                                __uint_as_float(x[4 * q + 3]));
            }
          }
        }
        fence_proxy_async_smem();
        epi_bar_sync();
        if (warp == EPI_WARP0 && lane == 0) {
          // sent even after a failed wait, so that rank 0 is not left waiting
          const uint32_t dst = map_to_rank(smem_u32(a_ring), 0) + (rank - 1) * slot_bytes;
          const uint32_t bar = map_to_rank(smem_u32(red_full), 0);
          for (int c = 0; c < BN / 32; ++c)
            bulk_copy_to_cluster(dst + c * 16384u, smem_u32(a_ring) + c * 16384u, chunk_bytes, bar);
        }
      }
      if (epi_warp && rank == 0) {
        bool ok = mbar_wait(red_full, 0, err, PF_DEV_TIMEOUT_EPILOGUE);
        ok = __all_sync(0xffffffffu, ok);
        if (ok && epi_ok) {
          const uint8_t* slots = a_ring;
          uint8_t* stage = epi_stage + (warp - EPI_WARP0) * EPI_STAGE_BYTES;
          const int m0 = m_base + 32 * qw;
          const int rv = sh.M - m0 < 32 ? sh.M - m0 : 32;
          run_epilogue<BN>(ep, m0, rv, nt, ew, stage, [&](int c, float(&v)[32]) {
            uint32_t x[32];
            tmem_ld32(tq + 32 * c, x);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(x[q]);
            for (int s = 1; s < sh.splits; ++s) {
              const uint8_t* sl = slots + (s - 1) * slot_bytes;
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 p = *reinterpret_cast<const float4*>(sl + slot_off(c, r, q));
                v[4 * q] += p.x;
                v[4 * q + 1] += p.y;
                v[4 * q + 2] += p.z;
                v[4 * q + 3] += p.w;
              }
            }
          });
        }
      }
      // ranks 1.. keep their shared memory (the copies' source) until rank 0
      // has received everything
      cluster_sync_all();
    }
  } else {
    // ================ producer, MMA and dequant warpgroups
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(LEAN_REGS));
    if (warp == 0) {
      // ---------------- producer
      // Weights do not depend on the previous kernel: the first raw stages are
      // fetched before waiting for it.
      const int nst = (nkb + C::KS - 1) / C::KS;  // pipeline stages per unit
      const uint32_t pre = (C::Q4 && blockIdx.x < sh.n_units) ? (nst < C::S_R ? nst : C::S_R) : 0;
      // one stage per lane: copies issued by one thread are served one after
      // another, copies issued by different threads overlap
      if (C::Q4 && static_cast<uint32_t>(lane) < pre) {
        const int u = blockIdx.x;
        const int ks = u % sh.splits, t = u / sh.splits;
        const int nt = t % sh.n_tiles;
        const int kc = nkb - lane * C::KS < C::KS ? nkb - lane * C::KS : C::KS;
        mbar_arrive_expect_tx(&full_r[lane], kc * C::RAW_KB);
        bulk_load(r_ring + lane * C::RAW_BYTES,
                  wq4 + ((size_t)nt * (sh.splits * nkb) + ks * nkb + lane * C::KS) * C::RAW_KB, kc * C::RAW_KB,
                  &full_r[lane]);
      }
      __syncwarp();
      pdl_wait();
      // The main loop runs in lane 0 alone: no warp-wide step per k-block.
      if (lane == 0) {
        uint32_t g = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < sh.n_units && ok; u += gridDim.x) {
          const int ks = u % sh.splits, t = u / sh.splits;
          const int nt = t % sh.n_tiles, mb = t / sh.n_tiles;
          const int m_base = mb * MT * 128;
          int mt_valid = (sh.M - m_base + 127) / 128;
          if (mt_valid > MT) mt_valid = MT;
          for (int i = 0; i < nst; ++i, ++g) {
            const int kb = ks * nkb + i * C::KS;  // first k-block of the stage
            const int kc = nkb - i * C::KS < C::KS ? nkb - i * C::KS : C::KS;
            const int sa = g % C::S_A;
            if (blockIdx.x == 0 && static_cast<int>(g) == sh.withhold_stage) {
              ok = false;  // stop issuing; the stages already issued are drained below
              break;
            }
            ok = mbar_wait(&empty_a[sa], ((g / C::S_A) & 1) ^ 1, err, PF_DEV_TIMEOUT_PRODUCER);
            const bool raw_now = C::Q4 && g >= pre;
            const int sr = g % C::NR;
            if (ok && raw_now) ok = mbar_wait(&empty_r[sr], ((g / C::NR) & 1) ^ 1, err, PF_DEV_TIMEOUT_PRODUCER);
            if (!ok) break;
            uint8_t* st = a_ring + sa * C::A_STAGE;
            mbar_arrive_expect_tx(&full_a[sa], kc * mt_valid * sh.a_box_rows * 128 + (C::Q4 ? 0 : C::BT_BYTES));
            for (int j = 0; j < kc; ++j)
              for (int mt = 0; mt < mt_valid; ++mt)
                tma_load_2d(st + (j * MT + mt) * 128 * 128, &tmA, &full_a[sa], (kb + j) * 64, m_base + mt * 128);
            if (raw_now) {
              mbar_arrive_expect_tx(&full_r[sr], kc * C::RAW_KB);
              bulk_load(r_ring + sr * C::RAW_BYTES, wq4 + ((size_t)nt * (sh.splits * nkb) + kb) * C::RAW_KB,
                        kc * C::RAW_KB, &full_r[sr]);
            } else if (!C::Q4) {
              tma_load_2d(st + C::A_BYTES, &tmB, &full_a[sa], kb * 64, nt * BN);
            }
          }
        }
        if (!ok) {
          // the last S_A / S_R issues may still be in flight
          const uint32_t ga = g > (uint32_t)C::S_A ? g - C::S_A : 0;
          for (uint32_t x = ga; x < g; ++x) mbar_drain(&full_a[x % C::S_A], (x / C::S_A) & 1);
          if (C::Q4) {
            const uint32_t gr = g > (uint32_t)C::S_R ? g - C::S_R : 0;
            for (uint32_t x = gr; x < g; ++x) mbar_drain(&full_r[x % C::NR], (x / C::NR) & 1);
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------- MMA issue (lane 0 alone)
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
        uint32_t g = 0, j = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < sh.n_units && ok; u += gridDim.x, ++j) {
          const int t = u / sh.splits;
          const int mb = t / sh.n_tiles;
          int mt_valid = (sh.M - mb * MT * 128 + 127) / 128;
          if (mt_valid > MT) mt_valid = MT;
          const int buf = C::ACC_BUFS == 2 ? (j & 1) : 0;
          const uint32_t tacc = tmem_base + buf * C::ACC;
          ok = mbar_wait(&tempty[buf], ((j / C::ACC_BUFS) & 1) ^ 1, err, PF_DEV_TIMEOUT_MMA);
          if (!ok) break;
          tc_fence_after();
          const int nst = (nkb + C::KS - 1) / C::KS;
          for (int i = 0; i < nst; ++i, ++g) {
            const int kc = nkb - i * C::KS < C::KS ? nkb - i * C::KS : C::KS;
            const int sa = g % C::S_A;
            const int sb = C::Q4 ? g % C::NB : 0;
            ok = mbar_wait_spin(&full_a[sa], (g / C::S_A) & 1, err, PF_DEV_TIMEOUT_MMA);
            if (ok && C::Q4) ok = mbar_wait_spin(&bfull[sb], (g / C::NB) & 1, err, PF_DEV_TIMEOUT_MMA);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a0 = smem_u32(a_ring + sa * C::A_STAGE);
            const uint32_t b0 = C::Q4 ? smem_u32(b_ring + sb * C::BT_BYTES) : a0 + C::A_BYTES;
            // The stage's descriptors are built once; an operand's address
            // sits in the low bits (16-byte units, 14 bits) and every step
            // adds a constant offset that cannot carry out of that field.
            // A single issuing thread pays for every instruction between
            // two MMAs, so the common full stage is unrolled completely.
            const uint64_t ad0 = sdesc_sw128(a0), bd0 = sdesc_sw128(b0);
            if (kc == C::KS && mt_valid == MT) {
#pragma unroll
              for (int j = 0; j < C::KS; ++j)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16(tacc + mt * BN, ad0 + (((j * MT + mt) * 128 * 128 + kk * 32) >> 4),
                               bd0 + ((j * C::BT_KB + kk * 32) >> 4), idesc, (i | j | kk) != 0 ? 1u : 0u);
            } else {
              for (int j = 0; j < kc; ++j) {
                const int kbl = i * C::KS + j;  // k-block within the unit
                for (int mt = 0; mt < mt_valid; ++mt) {
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16(tacc + mt * BN, ad0 + (((j * MT + mt) * 128 * 128 + kk * 32) >> 4),
                               bd0 + ((j * C::BT_KB + kk * 32) >> 4), idesc, (kbl | kk) != 0 ? 1u : 0u);
                }
              }
            }
            tc_commit(&empty_a[sa]);
            if (C::Q4) tc_commit(&bempty[sb]);
          }
          if (ok) tc_commit(&tfull[buf]);  // the unit's accumulator is complete
        }
        if (!ok) {
          // wait for the MMAs already issued before TMEM is freed
          tc_commit(&tfull[0]);
          mbar_drain(&tfull[0], 0);
          mbar_drain(&tfull[0], 1);
        }
      }
      __syncwarp();
    } else if (C::Q4) {
      // ---------------- dequant
      const int t = dq_index(warp, lane);
      uint32_t g = 0;
      bool ok = true;
      const int nst = (nkb + C::KS - 1) / C::KS;
      for (int u = blockIdx.x; u < sh.n_units && ok; u += gridDim.x) {
        for (int i = 0; i < nst; ++i, ++g) {
          const int kc = nkb - i * C::KS < C::KS ? nkb - i * C::KS : C::KS;
          const int sr = g % C::NR, sb = g % C::NB;
          bool w_ok = mbar_wait(&full_r[sr], (g / C::NR) & 1, err, PF_DEV_TIMEOUT_DEQUANT);
          if (w_ok) w_ok = mbar_wait(&bempty[sb], ((g / C::NB) & 1) ^ 1, err, PF_DEV_TIMEOUT_DEQUANT);
          ok = __all_sync(0xffffffffu, w_ok);
          if (!ok) break;
          uint8_t* bt = b_ring + sb * C::BT_BYTES;
          const uint8_t* raw = r_ring + sr * C::RAW_BYTES;
          // items: (k-block j, half h, row rr); a thread takes two at a time
          // so that their shared-memory loads overlap
          const int items = kc * BN * 2;
          for (int it = t; it < items; it += 2 * DQ_THREADS) {
            const int it2 = it + DQ_THREADS;
            const int j = it / (BN * 2), rr = it % BN, h = (it / BN) & 1;
            const uint8_t* rj = raw + j * C::RAW_KB;
            const uint4 nib = *reinterpret_cast<const uint4*>(rj + (size_t)(h * BN + rr) * 16);
            const __half d = *reinterpret_cast<const __half*>(rj + BN * 32 + (h * BN + rr) * 2);
            if (it2 < items) {
              const int j2 = it2 / (BN * 2), rr2 = it2 % BN, h2 = (it2 / BN) & 1;
              const uint8_t* rj2 = raw + j2 * C::RAW_KB;
              const uint4 nib2 = *reinterpret_cast<const uint4*>(rj2 + (size_t)(h2 * BN + rr2) * 16);
              const __half d2 = *reinterpret_cast<const __half*>(rj2 + BN * 32 + (h2 * BN + rr2) * 2);
              dequant_block32(nib, d, bt + j * C::BT_KB + rr * 128, h, rr & 7);
              dequant_block32(nib2, d2, bt + j2 * C::BT_KB + rr2 * 128, h2, rr2 & 7);
            } else {
              dequant_block32(nib, d, bt + j * C::BT_KB + rr * 128, h, rr & 7);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bfull[sb]);
            mbar_arrive(&empty_r[sr]);
          }
        }
      }
    }
    if (split_mode) {
      // the epilogue warpgroups run the cluster reduction; these warps
      // take part in its two cluster barriers
      if (warp == 0 && lane == 0 && cluster_ctarank() == 0)
        mbar_arrive_expect_tx(red_full, static_cast<uint32_t>(sh.splits - 1) * (BN / 32) * split_chunk_bytes);
      cluster_sync_all();
      cluster_sync_all();
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
  return encode_2d_bf16(&a.tmap, a.dev, (uint64_t)a.K, (uint64_t)a.rows, 64, 128, err) &&
         encode_2d_bf16(&a.tmap_small, a.dev, (uint64_t)a.K, (uint64_t)a.rows, 64, 16, err);
}

bool make_weight_map(WeightMat& w, std::string* err) {
  std::memset(&w.tmap, 0, sizeof(w.tmap));
  if (w.kind != W_BF16) return true;
  return encode_2d_bf16(&w.tmap, w.dev, (uint64_t)w.K, (uint64_t)w.N_rows, 64, (uint32_t)w.BN, err);
}

// SM count of the current device (looked up per call: contexts of one
// process may sit on different devices)
static int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

template <int WK, int BN, int MT>
static size_t ring_bytes() {
  using C = GemmCfg<WK, BN, MT>;
  return static_cast<size_t>(C::S_A) * C::A_STAGE + static_cast<size_t>(C::S_B) * C::BT_BYTES + C::RAW_RING;
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
  if (units1 * 2 <= sm_count() && nkb % 2 == 0 && nkb / 2 >= 4 && static_cast<size_t>(128) * BN * 4 <= ring) return 2;
  return 1;
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

template <int WK, int BN, int MT>
static cudaError_t launch_t(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err,
                            cudaStream_t s, int withhold_stage) {
  using C = GemmCfg<WK, BN, MT>;
  {
    const cudaError_t e = smem_opt_in<gemm_tc_kernel<WK, BN, MT>>(C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  GemmShape sh;
  sh.M = M;
  sh.K = W.K;
  sh.n_tiles = W.N_rows / BN;
  sh.m_blocks = (M + MT * 128 - 1) / (MT * 128);
  sh.splits = W.split;
  sh.kb_per_split = (W.K / 64) / W.split;
  sh.n_units = sh.n_tiles * sh.m_blocks * sh.splits;
  // A launch of at most 16 rows fetches 16-row A boxes: the MMA still reads
  // 128 rows, and rows 16..127 (stale shared memory) only reach accumulator
  // rows that are never stored.
  const bool small = MT == 1 && M <= 16;
  sh.a_box_rows = small ? 16 : 128;
  sh.withhold_stage = withhold_stage;
  if (W.split > 1 && static_cast<size_t>(W.split - 1) * 128 * BN * 4 > ring_bytes<WK, BN, MT>())
    return cudaErrorInvalidValue;
  const int cluster = W.split > 1 ? W.split : 1;
  const int grid = W.split > 1 ? sh.n_units : (sh.n_units < sm_count() ? sh.n_units : sm_count());
  return launch_k(gemm_tc_kernel<WK, BN, MT>, dim3(grid), dim3(GEMM_THREADS), C::SMEM_BYTES, s, cluster,
                  small ? A.tmap_small : A.tmap, W.tmap, static_cast<const uint8_t*>(W.dev), sh, ep, err);
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
#define PF_GEMM_CASE(WKV, BNV)                                                    \
  if (W.kind == WKV && W.BN == BNV)                                               \
    return two ? launch_t<WKV, BNV, 2>(A, M, W, ep, err, s, withhold_stage)      \
               : launch_t<WKV, BNV, 1>(A, M, W, ep, err, s, withhold_stage);
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
