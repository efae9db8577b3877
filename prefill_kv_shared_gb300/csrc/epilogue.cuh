// The fused epilogue shared by the tensor-core GEMM (gemm_tc.cu) and the
// one-row stream projection (gemv.cu): QKV with RoPE and the FP16 KV write,
// GeGLU/SwiGLU, the per-layer-embedding gate, the residual add, plain fp32.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace pf {

// ---------------------------------------------------------------------------
// Epilogue.
//
// tcgen05.ld (32x32b) gives each thread one accumulator row: a warp holds a
// 32-row x 32-column block, one row per lane.  Written to global memory in
// that layout every 16-byte access of a warp instruction falls in a
// different row, so a 128-byte row segment costs eight separate
// transactions.  Each block therefore goes through a warp-private 4 KB
// staging buffer in shared memory, and global memory is touched with lane l
// at row 4i + l/8, columns 4(l%8) .. 4(l%8)+3 (i = 0..7): every instruction
// covers four whole 128-byte (fp32) or 64-byte (16-bit) row segments.

constexpr int EPI_STAGE_BYTES = 32 * 32 * 4;

// Row r's 16-byte piece p (columns 4p .. 4p+3) sits at r*128 + 16*(p ^ (r & 7)):
// both the row-per-lane writes and the transposed reads are free of bank
// conflicts.
__device__ __forceinline__ void stage_put(uint8_t* st, int r, const float (&v)[32]) {
#pragma unroll
  for (int p = 0; p < 8; ++p)
    *reinterpret_cast<float4*>(st + r * 128 + ((p ^ (r & 7)) << 4)) =
        make_float4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
}
__device__ __forceinline__ float4 stage_get(const uint8_t* st, int r, int p) {
  return *reinterpret_cast<const float4*>(st + r * 128 + ((p ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint2 pack_bf16x4(float4 a) {
  return make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
}
__device__ __forceinline__ uint2 pack_half4(float4 a) { return make_uint2(pack_half2(a.x, a.y), pack_half2(a.z, a.w)); }
__device__ __forceinline__ float comp(const float4& a, int e) { return e == 0 ? a.x : e == 1 ? a.y : e == 2 ? a.z : a.w; }
__device__ __forceinline__ float4 bf16x4_to_f32(uint2 p) {
  return make_float4(__uint_as_float(p.x << 16), __uint_as_float(p.x & 0xFFFF0000u), __uint_as_float(p.y << 16),
                     __uint_as_float(p.y & 0xFFFF0000u));
}

// The fused epilogue for one warp's 32 rows of one tile: output rows
// m0 .. m0+31, of which the first rv are real (warp-uniform).  load(c, v)
// fills v with this lane's row (m0 + lane) of the tile's column chunk c
// (columns 32c .. 32c+31) and is called in a warp-uniform way.  The two
// epilogue warps of a lane quarter (ew = 0, 1) take alternate work items;
// `par` (0 or 1) flips which of them takes the first, so that over the M
// tiles of a unit (par = tile index & 1) an odd item count still splits
// evenly.  st: the warp's staging buffer.
template <int BN, class Load>
__device__ __forceinline__ void run_epilogue(const EpiParams& ep, int m0, int rv, int n_tile, int ew, uint8_t* st,
                                             int par, Load&& load) {
  constexpr int NCH = BN / 32;
  if (rv <= 0) return;
  const int ew0 = ew ^ (par & 1);  // parity of this warp's items
  const int lane = threadIdx.x & 31;
  const int rs = lane >> 3, p = lane & 7;  // transposed position: rows 4i + rs, columns 4p .. 4p+3
  const int n0 = n_tile * BN;
  float v[32];
  // Every kind below first computes all of a block's values into registers
  // and only then stores them: a global load placed after a store in
  // program order waits for it, which would put one memory round trip on
  // every row of the block.

  if (ep.kind == EPI_GLU) {
    // gate chunk c and up chunk c + NCH/2 of the interleaved tile -> output
    // columns f0 .. f0+31
    constexpr int HALF_CH = NCH / 2;
    for (int c = ew0; c < HALF_CH; c += 2) {
      const int f0 = n_tile * (BN / 2) + 32 * c;
      if (f0 >= ep.N) break;
      load(c, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = ep.act == 0 ? gelu_tanh_f(v[j]) : silu_f(v[j]);
      {
        float u[32];
        load(c + HALF_CH, u);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= u[j];
      }
      stage_put(st, lane, v);
      __syncwarp();
      uint2 h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = pack_bf16x4(stage_get(st, 4 * i + rs, p));
      __syncwarp();
      const int col = f0 + 4 * p;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 4 * i + rs;
        if (r >= rv || col >= ep.N) continue;
        __nv_bfloat16* dst = ep.out_bf16 + (size_t)(m0 + r) * ep.ld_bf16 + col;
        if (col + 4 <= ep.N) {
          *reinterpret_cast<uint2*>(dst) = h[i];
        } else {
          for (int e = 0; col + e < ep.N; ++e) {
            const uint32_t w = e < 2 ? h[i].x : h[i].y;
            dst[e] = __ushort_as_bfloat16(static_cast<unsigned short>(w >> (16 * (e & 1))));
          }
        }
      }
    }
    return;
  }

  if (ep.kind == EPI_QKV) {
    // Q | K | V columns; Q and K rotated (half-split RoPE at position
    // pos0 + row) and written as fp16, V written as fp16 to the cache.  A
    // rotated chunk is handled together with its partner half a head away:
    // with whole heads in a tile (hd <= BN) the partner is half/32 chunks
    // further; with heads wider than the tile, a tile holds BN/2 dims of the
    // head's first half and the same BN/2 dims of its second half
    // (qkv_tile_rows), and the partner is NCH/2 chunks further.
    const int hd = ep.head_dim, half = hd / 2, pair_ch = half / 32;
    const bool split_heads = hd > BN;
    const int q_end = ep.q_dim, k_end = ep.q_dim + ep.kv_dim, v_end = ep.q_dim + 2 * ep.kv_dim;
    int item = 0;
    for (int c = 0; c < NCH; ++c) {
      const int n = n0 + 32 * c;
      if (n >= v_end) break;  // padding columns
      if (n >= k_end) {       // V: no rotation
        if ((item++ & 1) != ew0) continue;
        load(c, v);
        stage_put(st, lane, v);
        __syncwarp();
        uint2 h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = pack_half4(stage_get(st, 4 * i + rs, p));
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 4 * i + rs;
          if (r >= rv) continue;
          const int slot = ep.row_slot ? ep.row_slot[m0 + r] : ep.pos0 + m0 + r;
          *reinterpret_cast<uint2*>(ep.v_cache + (size_t)slot * ep.kv_dim + (n - k_end) + 4 * p) = h[i];
        }
        continue;
      }
      const bool is_q = n < q_end;
      const int rel = is_q ? n : n - q_end;
      int i0, head, partner;
      if (split_heads) {
        const int tile = rel / BN, x = rel % BN;
        if (x >= BN / 2) continue;  // handled together with its partner chunk
        head = tile / (hd / BN);
        i0 = (tile % (hd / BN)) * (BN / 2) + x;
        partner = c + NCH / 2;
      } else {
        i0 = rel % hd;
        if (i0 >= half) continue;  // handled together with its partner chunk
        head = rel / hd;
        partner = c + pair_ch;
      }
      if ((item++ & 1) != ew0) continue;
      // two passes of 16 rows each keep the transposed halves in registers
      for (int hp = 0; hp < 2; ++hp) {
        float4 c01[4], c23[4];  // (cos, sin) of columns i0+4p .. i0+4p+3 at each row's position
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 16 * hp + 4 * i + rs;
          const int m = m0 + (r < rv ? r : 0);
          const int pos = ep.row_pos ? ep.row_pos[m] : ep.pos0 + m;
          const float4* cs = reinterpret_cast<const float4*>(ep.rope + (size_t)pos * half + i0 + 4 * p);
          c01[i] = cs[0];
          c23[i] = cs[1];
        }
        float4 vt[4], ut[4];
        load(c, v);
        stage_put(st, lane, v);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) vt[i] = stage_get(st, 16 * hp + 4 * i + rs, p);
        __syncwarp();
        load(partner, v);
        stage_put(st, lane, v);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) ut[i] = stage_get(st, 16 * hp + 4 * i + rs, p);
        __syncwarp();
        uint2 o1[4], o2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 a = vt[i], b = ut[i], x = c01[i], y = c23[i];
          o1[i] = pack_half4(make_float4(a.x * x.x - b.x * x.y, a.y * x.z - b.y * x.w, a.z * y.x - b.z * y.y,
                                         a.w * y.z - b.w * y.w));
          o2[i] = pack_half4(make_float4(a.x * x.y + b.x * x.x, a.y * x.w + b.y * x.z, a.z * y.y + b.z * y.x,
                                         a.w * y.w + b.w * y.z));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 16 * hp + 4 * i + rs;
          if (r >= rv) continue;
          const int m = m0 + r;
          const int slot = ep.row_slot ? ep.row_slot[m] : ep.pos0 + m;
          __half* dst = is_q ? ep.q_out + (size_t)m * ep.q_dim + head * hd
                             : ep.k_cache + (size_t)slot * ep.kv_dim + head * hd;
          *reinterpret_cast<uint2*>(dst + i0 + 4 * p) = o1[i];
          *reinterpret_cast<uint2*>(dst + i0 + half + 4 * p) = o2[i];
        }
        if (rv <= 16) break;
      }
    }
    return;
  }

  // F32, RESID, PLE: one 32-column chunk at a time.  The chunk's global
  // operand (RESID: the residual rows; PLE: the multipliers) is requested
  // before the TMEM load so that its latency overlaps the staging.  (Asking
  // for the next chunk's operand before this chunk's stores does not fit
  // the registers: the epilogue then spills.)
  auto load_side = [&](int c, float4(&sd)[8]) {
    const int col = n0 + 32 * c + 4 * p;
    const bool full = col + 4 <= ep.N;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + rs;
      sd[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r >= rv || col >= ep.N) continue;
      if (ep.kind == EPI_RESID) {
        const float* xr = ep.out_f32 + (size_t)(m0 + r) * ep.ld_f32 + col;
        if (full) {
          sd[i] = *reinterpret_cast<const float4*>(xr);
        } else {
          sd[i].x = xr[0];
          if (col + 1 < ep.N) sd[i].y = xr[1];
          if (col + 2 < ep.N) sd[i].z = xr[2];
        }
      } else if (ep.kind == EPI_PLE) {
        const __nv_bfloat16* pl = ep.ple + (size_t)(m0 + r) * ep.ple_stride + col;
        if (full) {
          sd[i] = bf16x4_to_f32(*reinterpret_cast<const uint2*>(pl));
        } else {
          sd[i].x = __bfloat162float(pl[0]);
          if (col + 1 < ep.N) sd[i].y = __bfloat162float(pl[1]);
          if (col + 2 < ep.N) sd[i].z = __bfloat162float(pl[2]);
        }
      }
    }
  };
  for (int c = ew0; c < NCH; c += 2) {
    const int n = n0 + 32 * c;
    if (n >= ep.N) break;
    const int col = n + 4 * p;
    const bool full = col + 4 <= ep.N;
    float4 side[8];
    load_side(c, side);
    load(c, v);
    stage_put(st, lane, v);
    __syncwarp();
    // values of the block in the transposed layout (RESID: the new residual;
    // PLE: gelu(acc) * multiplier, before rounding)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 a = stage_get(st, 4 * i + rs, p);
      const float4 g = side[i];
      if (ep.kind == EPI_RESID) {
        side[i] = make_float4(g.x + a.x, g.y + a.y, g.z + a.z, g.w + a.w);
      } else if (ep.kind == EPI_PLE) {
        side[i] = make_float4(gelu_tanh_f(a.x) * g.x, gelu_tanh_f(a.y) * g.y, gelu_tanh_f(a.z) * g.z,
                              gelu_tanh_f(a.w) * g.w);
      } else {
        side[i] = a;
      }
    }
    __syncwarp();
    if (col < ep.N) {
      float* of = ep.kind != EPI_PLE ? ep.out_f32 : nullptr;                        // fp32 result
      __nv_bfloat16* ob = ep.kind != EPI_F32 ? ep.out_bf16 : nullptr;               // bf16 result (RESID: optional copy)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 4 * i + rs;
        if (r >= rv) continue;
        const size_t m = static_cast<size_t>(m0 + r);
        const float4 a = side[i];
        if (full) {
          if (of) *reinterpret_cast<float4*>(of + m * ep.ld_f32 + col) = a;
          if (ob) *reinterpret_cast<uint2*>(ob + m * ep.ld_bf16 + col) = pack_bf16x4(a);
        } else {
          for (int e = 0; col + e < ep.N; ++e) {
            if (of) of[m * ep.ld_f32 + col + e] = comp(a, e);
            if (ob) ob[m * ep.ld_bf16 + col + e] = __float2bfloat16_rn(comp(a, e));
          }
        }
      }
    }
  }
}

}  // namespace pf
