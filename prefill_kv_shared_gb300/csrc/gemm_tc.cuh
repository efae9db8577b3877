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
// result does not depend on how many rows the launch carries.  Whether a
// matrix runs in CTA pairs is fixed per matrix shape, like its k-split.
//
// CTA pairs (PAIR): a 2-CTA cluster shares each tcgen05.mma of 256 rows
// (.cta_group::2).  Each CTA stages its own 128 rows of A and one half of the
// weight tile (BN/2 rows, fetched as four bulk copies per k-block from the
// unchanged tile layout and dequantised by its own warps), so per SM the
// shared-memory operand traffic of B, the dequant work and the MMA
// instructions per FLOP are halved.  The even CTA issues the MMAs and the
// commits (one to each CTA's barrier); the odd CTA forwards "my A
// stage has landed" and "my B stage is dequantised" to the even CTA's
// barriers and returns "my accumulator is drained" from its epilogue.  Each
// CTA's TMA and bulk copies complete on its own barriers only.
#pragma once

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

#include <cstring>
#include <mutex>
#include <string>

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
// one-unit launches: the eight epilogue warps dequantise too until the
// unit's last stage (their epilogue cannot start before it)
constexpr int DQ_THREADS_SOLO = DQ_THREADS + 256;
constexpr int EPI_REGS = 176;
constexpr int LEAN_REGS = 80;
static_assert(2 * 128 * (EPI_REGS + LEAN_REGS) <= GEMM_THREADS * 128, "register split exceeds the launch's registers");
static_assert(EPI_REGS % 8 == 0 && LEAN_REGS % 8 == 0 && LEAN_REGS >= 24 && EPI_REGS <= 256, "setmaxnreg range");

__device__ __forceinline__ bool is_epi_warp(int w) { return w >= EPI_WARP0 && w < EPI_WARP0 + EPI_WARPS; }
// dequant thread index 0..DQ_THREADS-1 of a thread in warps 2, 3, 12..15
__device__ __forceinline__ int dq_index(int w, int lane) { return (w < 4 ? w - 2 : w - 10) * 32 + lane; }
constexpr int SMEM_LIMIT = 232448;

__host__ __device__ constexpr int pow2_cols(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

// SOLO: a launch whose CTAs take one work unit each.  The epilogue then
// stages in the dequantised-B ring, idle once the unit's last MMA has
// completed, instead of a dedicated area, and the 32 KB go to the A ring
// (one more A stage: the A operand's latency against the ring's depth paces
// the main loop).
template <int WK, int BN, int MT, bool PAIR = false, bool SOLO = false>
struct GemmCfg {
  static constexpr bool Q4 = WK == W_Q4;
  static_assert(!PAIR || Q4, "CTA pairs take Q4_0 weights");
  static_assert(!SOLO || (Q4 && !PAIR), "one-unit launches: Q4_0 weights on single CTAs");
  static constexpr int BNL = PAIR ? BN / 2 : BN;  // weight rows this CTA stages
  static constexpr int MMA_M = PAIR ? 256 : 128;  // rows of one MMA (over both CTAs of a pair)
  static constexpr int ROWS = MT * MMA_M;         // rows of A in one work unit
  // 64-wide k-blocks per pipeline stage: every stage costs the copy engine,
  // the barriers and the dequant warps a fixed amount whatever its size, so
  // narrow tiles take two k-blocks a stage where shared memory allows.
  static constexpr int KS = (Q4 && BNL <= 128 && MT == 1) ? 2 : 1;
  static constexpr int A_KB = MT * 128 * 128;  // one k-block of this CTA's A: MT tiles of 128 rows x 64 bf16
  static constexpr int BT_KB = BNL * 128;      // one k-block of bf16 B (BNL rows x 64)
  static constexpr int RAW_KB = Q4 ? BNL * 36 : 0;
  static constexpr int A_BYTES = KS * A_KB;    // stage layouts: [k-block][M tile][128 x 128 B], [k-block][BN x 128 B]
  static constexpr int BT_BYTES = KS * BT_KB;
  static constexpr int RAW_BYTES = KS * RAW_KB;
  static constexpr int A_STAGE = A_BYTES + (Q4 ? 0 : BT_BYTES);
  // The dequantised B ring bounds how far the dequant warps run ahead of the
  // MMAs (B stage k+S_B is written once the MMAs of stage k are done); the
  // A ring takes what the B and raw rings and the epilogue staging leave.
  static constexpr int S_B =
      !Q4    ? 0
      : PAIR ? (BT_BYTES >= 32768 ? 2 : 3)
             : (BN >= 256 ? (MT == 2 ? 2 : 3) : BN == 192 ? 2 : KS == 2 ? (BN == 64 ? 4 : 2) : 4);
  // (192-row tiles over two M tiles: two raw stages leave room for a
  // fourth A stage, which paces the main loop there)
  static constexpr int S_R =
      !Q4 ? 0 : PAIR ? S_B + 1 : (BN == 192 && MT == 2 ? 2 : BN >= 192 ? 3 : KS == 2 ? (BN == 64 ? 6 : 3) : 6);
  static constexpr int NB = S_B > 0 ? S_B : 1;  // ring moduli (the rings are unused without Q4)
  static constexpr int NR = S_R > 0 ? S_R : 1;
  static constexpr int RAW_RING = (S_R * RAW_BYTES + 1023) / 1024 * 1024;
  static constexpr int EPI_STAGING = EPI_WARPS * 32 * 32 * 4;  // one 4 KB staging buffer per epilogue warp
  static constexpr int EPI_BYTES = SOLO ? 0 : EPI_STAGING;      // (SOLO: in the B ring)
  static_assert(!SOLO || S_B * BT_BYTES >= EPI_STAGING, "the B ring holds the epilogue staging");
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
  static_assert(!PAIR || (BNL % 16 == 0 && BNL >= 32), "pair: each CTA's half of B in whole 16-row steps");
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

template <int WK, int BN, int MT, bool PAIR, bool SOLO>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB, const uint8_t* __restrict__ wq4, const GemmShape sh_in,
                   const EpiParams ep_in, int* err) {
  using C = GemmCfg<WK, BN, MT, PAIR, SOLO>;
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
  // one-unit launches stage the epilogue in the B ring: every MMA that read
  // it has completed (tfull) before the epilogue writes there, and no
  // dequant follows the unit's last stage
  uint8_t* epi_stage = SOLO ? b_ring : r_ring + C::RAW_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(r_ring + C::RAW_RING + C::EPI_BYTES);
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
  // CTA pairs: rank in the pair, the pair's first unit and the unit stride
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool issuer = rank == 0;  // this CTA issues the MMAs (always, without pairs)
  const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ustep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // The issuing CTA's full_a, bfull and tempty also count the odd CTA's
  // forwarded arrivals (remote arrives, released at cluster scope): its MMA
  // thread waits on them with cluster-scope acquire.  Barriers that only
  // tcgen05.commit completes (empty_a, bempty, tfull, one commit to each of both
  // CTAs) order the tensor cores' accesses by themselves and are waited on
  // at CTA scope.
  const uint32_t peers = PAIR && issuer ? 2u : 1u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S_A; ++s) {
      mbar_init(&full_a[s], peers);
      mbar_init(&empty_a[s], 1);
    }
    for (int s = 0; s < C::S_R; ++s) {
      mbar_init(&full_r[s], 1);
      mbar_init(&empty_r[s], (SOLO ? DQ_THREADS_SOLO : DQ_THREADS) / 32);
    }
    for (int s = 0; s < C::S_B; ++s) {
      mbar_init(&bfull[s], peers * ((SOLO ? DQ_THREADS_SOLO : DQ_THREADS) / 32));
      mbar_init(&bempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], peers * EPI_WARPS);
    }
    mbar_init(red_full, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    if (MT == 2 && !PAIR) prefetch_tensormap(&tmA2);
    if (WK == W_BF16) prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    else
      tmem_alloc(tmem_slot, C::TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // both CTAs' barriers are initialised before any arrive crosses the pair
  if constexpr (PAIR) cluster_sync_all();
  const uint32_t tmem_base = *tmem_slot;
  // shared::cluster address of one of the issuing CTA's barriers
  auto issuer_bar = [&](uint64_t* bar) -> uint32_t { return map_to_rank(smem_u32(bar), 0); };
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
  // Q4_0 -> bf16 over every stage of this CTA's units, by `nthreads` threads
  // (t = this thread's index among them), each warp arriving on the ring
  // barriers once per stage
  constexpr int DQ_THREADS_ALL = SOLO ? DQ_THREADS_SOLO : DQ_THREADS;
  auto dequant_loop = [&](const int t, const int nthreads) {
    uint32_t g = 0;
    bool ok = true;
    const int nst = (nkb + C::KS - 1) / C::KS;
    for (int u = unit0; u < sh.n_units && ok; u += ustep) {
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
        constexpr int R = C::BNL;  // weight rows staged by this CTA
        const int items = kc * R * 2;
        for (int it = t; it < items; it += 2 * nthreads) {
          const int it2 = it + nthreads;
          const int j = it / (R * 2), rr = it % R, h = (it / R) & 1;
          const uint8_t* rj = raw + j * C::RAW_KB;
          const uint4 nib = *reinterpret_cast<const uint4*>(rj + (size_t)(h * R + rr) * 16);
          const __half d = *reinterpret_cast<const __half*>(rj + R * 32 + (h * R + rr) * 2);
          if (it2 < items) {
            const int j2 = it2 / (R * 2), rr2 = it2 % R, h2 = (it2 / R) & 1;
            const uint8_t* rj2 = raw + j2 * C::RAW_KB;
            const uint4 nib2 = *reinterpret_cast<const uint4*>(rj2 + (size_t)(h2 * R + rr2) * 16);
            const __half d2 = *reinterpret_cast<const __half*>(rj2 + R * 32 + (h2 * R + rr2) * 2);
            dequant_block32(nib, d, bt + j * C::BT_KB + rr * 128, h, rr & 7);
            dequant_block32(nib2, d2, bt + j2 * C::BT_KB + rr2 * 128, h2, rr2 & 7);
          } else {
            dequant_block32(nib, d, bt + j * C::BT_KB + rr * 128, h, rr & 7);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(issuer_bar(&bfull[sb]));
          else
            mbar_arrive(&bfull[sb]);
          mbar_arrive(&empty_r[sr]);
        }
      }
    }
  };
  const int wg = warp >> 2;
  if (wg == 1 || wg == 2) {
    // ================ epilogue warpgroups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(EPI_REGS));
    if constexpr (SOLO) dequant_loop(DQ_THREADS + (warp - EPI_WARP0) * 32 + lane, DQ_THREADS_ALL);
    {
      // ---------------- epilogue
      pdl_wait();
      const int qw = warp & 3;                 // TMEM lane quarter this warp may access
      const int ew = (warp - EPI_WARP0) >> 2;  // which of the quarter's two epilogue warps
      uint8_t* stage = epi_stage + (warp - EPI_WARP0) * EPI_STAGE_BYTES;
      uint32_t j = 0;
      for (int u = unit0; u < sh.n_units; u += ustep, ++j) {
        const int t = u / sh.splits;
        const int nt = t % sh.n_tiles, mb = t / sh.n_tiles;
        const int m_base = mb * C::ROWS;
        int mt_valid = (sh.M - m_base + C::MMA_M - 1) / C::MMA_M;
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
          // this CTA's accumulator rows (lanes) of MMA tile mt; rv <= 0 when
          // they are all past M
          const int m0 = m_base + mt * C::MMA_M + static_cast<int>(rank) * 128 + 32 * qw;
          const int rv = sh.M - m0 < 32 ? sh.M - m0 : 32;
          run_epilogue<BN>(ep, m0, rv, nt, ew, stage, mt, [&](int c, float(&v)[32]) {
            uint32_t x[32];
            tmem_ld32(tq + mt * BN + 32 * c, x);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(x[q]);
          });
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(issuer_bar(&tempty[buf]));
          else
            mbar_arrive(&tempty[buf]);
        }
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
          run_epilogue<BN>(ep, m0, rv, nt, ew, stage, 0, [&](int c, float(&v)[32]) {
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
      // kc k-blocks of weight tile nt from k-block kb into raw stage `dst`:
      // the whole tile, or with pairs this CTA's half of its rows (nibbles
      // of both Q4_0 halves, then their scales: four pieces a k-block)
      auto issue_raw = [&](uint8_t* dst, int nt, int kb, int kc, uint64_t* bar) {
        const size_t tkb = (size_t)nt * (sh.splits * nkb) + kb;  // (tile, k-block) index
        mbar_arrive_expect_tx(bar, kc * C::RAW_KB);
        if constexpr (!PAIR) {
          bulk_load(dst, wq4 + tkb * C::RAW_KB, kc * C::RAW_KB, bar);
        } else {
          constexpr int H = C::BNL;
          for (int j = 0; j < kc; ++j) {
            const uint8_t* src = wq4 + (tkb + j) * (size_t)(BN * 36);
            uint8_t* d = dst + j * C::RAW_KB;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              bulk_load(d + h * H * 16, src + (h * BN + rank * H) * 16, H * 16, bar);
              bulk_load(d + H * 32 + h * H * 2, src + BN * 32 + (h * BN + rank * H) * 2, H * 2, bar);
            }
          }
        }
      };
      const uint32_t pre = (C::Q4 && unit0 < sh.n_units) ? (nst < C::S_R ? nst : C::S_R) : 0;
      // one stage per lane: copies issued by one thread are served one after
      // another, copies issued by different threads overlap
      if (C::Q4 && static_cast<uint32_t>(lane) < pre) {
        const int u = unit0;
        const int ks = u % sh.splits, t = u / sh.splits;
        const int nt = t % sh.n_tiles;
        const int kc = nkb - lane * C::KS < C::KS ? nkb - lane * C::KS : C::KS;
        issue_raw(r_ring + lane * C::RAW_BYTES, nt, ks * nkb + lane * C::KS, kc, &full_r[lane]);
      }
      __syncwarp();
      pdl_wait();
      // The whole warp runs the main loop in step (waits and decisions
      // uniform); one elected lane issues the copies.
      {
        uint32_t g = 0;
        bool ok = true;
        for (int u = unit0; u < sh.n_units && ok; u += ustep) {
          const int ks = u % sh.splits, t = u / sh.splits;
          const int nt = t % sh.n_tiles, mb = t / sh.n_tiles;
          const int m_base = mb * C::ROWS;
          int mt_valid = (sh.M - m_base + C::MMA_M - 1) / C::MMA_M;
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
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (elect_one()) {
              uint8_t* st = a_ring + sa * C::A_STAGE;
              mbar_arrive_expect_tx(&full_a[sa], kc * mt_valid * sh.a_box_rows * 128 + (C::Q4 ? 0 : C::BT_BYTES));
              // two adjacent 128-row M tiles come in one 256-row box (the
              // same shared-memory layout as two boxes); every async copy
              // costs the issuing thread a fixed amount
              if (!PAIR && MT == 2 && mt_valid == 2) {
                for (int j = 0; j < kc; ++j)
                  tma_load_2d(st + j * MT * 128 * 128, &tmA2, &full_a[sa], (kb + j) * 64, m_base);
              } else {
                for (int j = 0; j < kc; ++j)
                  for (int mt = 0; mt < mt_valid; ++mt)
                    tma_load_2d(st + (j * MT + mt) * 128 * 128, &tmA, &full_a[sa], (kb + j) * 64,
                                m_base + mt * C::MMA_M + static_cast<int>(rank) * 128);
              }
              if (raw_now) {
                issue_raw(r_ring + sr * C::RAW_BYTES, nt, kb, kc, &full_r[sr]);
              } else if (!C::Q4) {
                tma_load_2d(st + C::A_BYTES, &tmB, &full_a[sa], kb * 64, nt * BN);
              }
            }
            __syncwarp();
          }
        }
        if (!ok && elect_one()) {
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
      // ---------------- MMA issue (lane 0 alone); with pairs, in the odd
      // CTA: forward each landed A stage to the issuing CTA
      if (lane == 0 && !issuer) {
        uint32_t g = 0;
        bool ok = true;
        const int nst = (nkb + C::KS - 1) / C::KS;
        for (int u = unit0; u < sh.n_units && ok; u += ustep)
          for (int i = 0; i < nst; ++i, ++g) {
            const int sa = g % C::S_A;
            ok = mbar_wait_spin(&full_a[sa], (g / C::S_A) & 1, err, PF_DEV_TIMEOUT_MMA);
            if (!ok) break;
            mbar_arrive_cluster(issuer_bar(&full_a[sa]));
          }
      }
      if (issuer) {
        // the whole warp runs the loop in step; one lane, elected once (its
        // commits track the MMAs it issued), issues
        const bool leader = elect_one();
        constexpr uint32_t idesc = idesc_bf16_f32(C::MMA_M, BN);
        uint32_t g = 0, j = 0;
        bool ok = true;
        for (int u = unit0; u < sh.n_units && ok; u += ustep, ++j) {
          const int t = u / sh.splits;
          const int mb = t / sh.n_tiles;
          int mt_valid = (sh.M - mb * C::ROWS + C::MMA_M - 1) / C::MMA_M;
          if (mt_valid > MT) mt_valid = MT;
          const int buf = C::ACC_BUFS == 2 ? (j & 1) : 0;
          const uint32_t tacc = tmem_base + buf * C::ACC;
          ok = mbar_wait<PAIR>(&tempty[buf], ((j / C::ACC_BUFS) & 1) ^ 1, err, PF_DEV_TIMEOUT_MMA);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const int nst = (nkb + C::KS - 1) / C::KS;
          for (int i = 0; i < nst; ++i, ++g) {
            const int kc = nkb - i * C::KS < C::KS ? nkb - i * C::KS : C::KS;
            const int sa = g % C::S_A;
            const int sb = C::Q4 ? g % C::NB : 0;
            ok = mbar_wait_spin<PAIR>(&full_a[sa], (g / C::S_A) & 1, err, PF_DEV_TIMEOUT_MMA);
            if (ok && C::Q4) ok = mbar_wait_spin<PAIR>(&bfull[sb], (g / C::NB) & 1, err, PF_DEV_TIMEOUT_MMA);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a0 = smem_u32(a_ring + sa * C::A_STAGE);
            const uint32_t b0 = C::Q4 ? smem_u32(b_ring + sb * C::BT_BYTES) : a0 + C::A_BYTES;
            // The stage's descriptors are built once; an operand's address
            // sits in the low bits (16-byte units, 14 bits) and every step
            // adds a constant offset that cannot carry out of that field.
            // With pairs the same descriptors address both CTAs' shared
            // memory (identical layouts).
            const uint64_t ad0 = sdesc_sw128(a0), bd0 = sdesc_sw128(b0);
            auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
              if constexpr (PAIR)
                tc_mma_f16_pair(d, a, b, idesc, acc);
              else
                tc_mma_f16(d, a, b, idesc, acc);
            };
            if (leader) {
              if (kc == C::KS && mt_valid == MT) {
#pragma unroll
                for (int j = 0; j < C::KS; ++j)
#pragma unroll
                  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                      mma(tacc + mt * BN, ad0 + (((j * MT + mt) * 128 * 128 + kk * 32) >> 4),
                          bd0 + ((j * C::BT_KB + kk * 32) >> 4), (i | j | kk) != 0 ? 1u : 0u);
              } else {
                for (int j = 0; j < kc; ++j) {
                  const int kbl = i * C::KS + j;  // k-block within the unit
                  for (int mt = 0; mt < mt_valid; ++mt) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                      mma(tacc + mt * BN, ad0 + (((j * MT + mt) * 128 * 128 + kk * 32) >> 4),
                          bd0 + ((j * C::BT_KB + kk * 32) >> 4), (kbl | kk) != 0 ? 1u : 0u);
                  }
                }
              }
              if constexpr (PAIR) {  // both CTAs' rings
                for (uint32_t r2 = 0; r2 < 2; ++r2) {
                  tc_commit_pair(map_to_rank(smem_u32(&empty_a[sa]), r2));
                  tc_commit_pair(map_to_rank(smem_u32(&bempty[sb]), r2));
                }
              } else {
                tc_commit(&empty_a[sa]);
                if (C::Q4) tc_commit(&bempty[sb]);
              }
            }
            __syncwarp();
          }
          if (ok && leader) {  // the unit's accumulator is complete
            if constexpr (PAIR) {
              tc_commit_pair(map_to_rank(smem_u32(&tfull[buf]), 0));
              tc_commit_pair(map_to_rank(smem_u32(&tfull[buf]), 1));
            } else {
              tc_commit(&tfull[buf]);
            }
          }
          __syncwarp();
        }
        if (!ok && leader) {
          // wait for the MMAs already issued before TMEM is freed (and,
          // with pairs, before the odd CTA may leave)
          if constexpr (PAIR)
            tc_commit_pair(map_to_rank(smem_u32(&tfull[0]), 0));
          else
            tc_commit(&tfull[0]);
          mbar_drain(&tfull[0], 0);
          mbar_drain(&tfull[0], 1);
        }
      }
      __syncwarp();
    } else if (C::Q4) {
      // ---------------- dequant
      dequant_loop(dq_index(warp, lane), DQ_THREADS_ALL);
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
  // with pairs neither CTA leaves (or frees TMEM) while the pair's MMAs may
  // still read its shared memory or write its TMEM
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host-side launch of one instantiation

// SM count of the current device (looked up per call: contexts of one
// process may sit on different devices)
inline int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

template <int WK, int BN, int MT, bool PAIR = false, bool SOLO = false>
inline size_t ring_bytes() {
  using C = GemmCfg<WK, BN, MT, PAIR, SOLO>;
  return static_cast<size_t>(C::S_A) * C::A_STAGE + static_cast<size_t>(C::S_B) * C::BT_BYTES + C::RAW_RING;
}

// 2-CTA clusters of this kernel that fit on the device at once (a GPC with
// an odd number of free SMs leaves one out), looked up once per device
template <auto Kernel>
inline int max_pairs(int smem_bytes) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static int n_pairs[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return sm_count() / 2;
  std::lock_guard<std::mutex> g(mu);
  if (n_pairs[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = smem_bytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, Kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sm_count() / 2;
    }
    n_pairs[dev] = n < sm_count() / 2 ? n : sm_count() / 2;
  }
  return n_pairs[dev];
}

template <int WK, int BN, int MT, bool PAIR, bool SOLO = false>
inline cudaError_t launch_t(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err,
                            cudaStream_t s, int withhold_stage) {
  using C = GemmCfg<WK, BN, MT, PAIR, SOLO>;
  {
    const cudaError_t e = smem_opt_in<gemm_tc_kernel<WK, BN, MT, PAIR, SOLO>>(C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  if (PAIR && W.split != 1) return cudaErrorInvalidValue;
  GemmShape sh;
  sh.M = M;
  sh.K = W.K;
  sh.n_tiles = W.N_rows / BN;
  sh.m_blocks = (M + C::ROWS - 1) / C::ROWS;
  sh.splits = W.split;
  sh.kb_per_split = (W.K / 64) / W.split;
  sh.n_units = sh.n_tiles * sh.m_blocks * sh.splits;
  // A launch of at most 16 rows fetches 16-row A boxes: the MMA still reads
  // 128 rows, and rows 16..127 (stale shared memory) only reach accumulator
  // rows that are never stored.
  const bool small = !PAIR && MT == 1 && M <= 16;
  sh.a_box_rows = small ? 16 : 128;
  sh.withhold_stage = withhold_stage;
  if (W.split > 1 && static_cast<size_t>(W.split - 1) * 128 * BN * 4 > ring_bytes<WK, BN, MT, PAIR, SOLO>())
    return cudaErrorInvalidValue;
  // one-unit launches: the split partials (A ring) must not reach the
  // epilogue staging (B ring), and every CTA takes one unit
  if (SOLO && (static_cast<size_t>(W.split - 1) * 128 * BN * 4 > static_cast<size_t>(C::S_A) * C::A_STAGE ||
               sh.n_units > (W.split > 1 ? sh.n_units : sm_count())))
    return cudaErrorInvalidValue;
  int cluster = 1, grid = 0;
  if (PAIR) {  // persistent 2-CTA clusters, as many as fit at once
    const int pairs = max_pairs<gemm_tc_kernel<WK, BN, MT, PAIR, SOLO>>(C::SMEM_BYTES);
    cluster = 2;
    grid = 2 * (sh.n_units < pairs ? sh.n_units : pairs);
  } else if (W.split > 1) {
    cluster = W.split;
    grid = sh.n_units;
  } else {
    grid = sh.n_units < sm_count() ? sh.n_units : sm_count();
  }
  return launch_k(gemm_tc_kernel<WK, BN, MT, PAIR, SOLO>, dim3(grid), dim3(GEMM_THREADS), C::SMEM_BYTES, s, cluster,
                  small ? A.tmap_small : A.tmap, A.tmap_wide, W.tmap, static_cast<const uint8_t*>(W.dev), sh, ep,
                  err);
}

}  // namespace pf
