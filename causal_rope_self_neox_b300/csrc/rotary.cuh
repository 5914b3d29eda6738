// rotary.cuh -- NeoX rotate-half rotary embedding on shared-memory tiles.
//
// The rotation (GPT-NeoX on FasterTransformer guide, sections "背景" and "模型配置":
// Neox-style rotary on both Query and Key, rotary_embedding of the head dims) pairs dim i
// with dim i + r/2 for i < r/2 and turns the pair by the angle p * base^(-2i/r), p the
// token position.  Dims >= r pass through.
//
// The kernel keeps the tensor-core operands in bf16.  A rotated value y is computed in
// fp32 and split as hi = bf16(y), lo = bf16(y - hi); the score is then accumulated as
// q_hi.k_hi + q_hi.k_lo + q_lo.k_hi over the rotated dims (relative error ~2^-16, the
// lo.lo term ~2^-18 is dropped), while a plain bf16 rounding of y (~2^-9) would cost up
// to ~3e-3 in the row logsumexp.  "hi" overwrites y's slot in the tile itself; "lo" goes
// to a side tile whose columns >= r stay zero.
#pragma once

#include <cstdint>

#include "tile_layout.cuh"

namespace neox {

// cos/sin table, fp64 arithmetic stored as fp32: tab[p * h + i] = (cos, sin)(p * base^(-2i/r)).
__global__ void rope_table_kernel(float2* __restrict__ tab, int S, int h, int r, double base) {
  const int64_t n = static_cast<int64_t>(S) * h;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = idx / h;
    const int i = static_cast<int>(idx - p * h);
    const double inv_freq = pow(base, -2.0 * static_cast<double>(i) / static_cast<double>(r));
    double s, c;
    sincos(static_cast<double>(p) * inv_freq, &s, &c);
    tab[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
  }
}

__device__ __forceinline__ void split_hi_lo(float y, uint16_t& hi, uint16_t& lo) {
  hi = f32_to_bf16_bits(y);
  lo = f32_to_bf16_bits(y - bf16_bits_to_f32(hi));
}

// Rotate the first r dims of one tile row in place (hi) and write lo to the side tile.
// pos < 0 marks a row past the end of the sequence (TMA filled it with zeros): lo = 0.
__device__ __forceinline__ void rotate_row(uint8_t* tile, uint8_t* side, int row, int64_t pos,
                                           const float2* __restrict__ cs, int r) {
  const int h = r >> 1;
  if ((h & 1) == 0) {
    // two pairs per step with 32-bit shared accesses: (i, i+1) and (i+h, i+h+1)
    for (int i = 0; i < h; i += 2) {
      uint32_t* pa = reinterpret_cast<uint32_t*>(tile + sw64_off(row, i));
      uint32_t* pb = reinterpret_cast<uint32_t*>(tile + sw64_off(row, i + h));
      const uint32_t a = *pa, b = *pb;
      float x0 = bf16_bits_to_f32(static_cast<uint16_t>(a & 0xFFFF));
      float x1 = bf16_bits_to_f32(static_cast<uint16_t>(a >> 16));
      float z0 = bf16_bits_to_f32(static_cast<uint16_t>(b & 0xFFFF));
      float z1 = bf16_bits_to_f32(static_cast<uint16_t>(b >> 16));
      float y0 = x0, y1 = x1, w0 = z0, w1 = z1;
      if (pos >= 0) {
        const float4 t = *reinterpret_cast<const float4*>(cs + pos * h + i);  // (c0, s0, c1, s1)
        y0 = fmaf(x0, t.x, -z0 * t.y);
        w0 = fmaf(z0, t.x, x0 * t.y);
        y1 = fmaf(x1, t.z, -z1 * t.w);
        w1 = fmaf(z1, t.z, x1 * t.w);
      }
      uint16_t hy0, ly0, hy1, ly1, hw0, lw0, hw1, lw1;
      split_hi_lo(y0, hy0, ly0);
      split_hi_lo(y1, hy1, ly1);
      split_hi_lo(w0, hw0, lw0);
      split_hi_lo(w1, hw1, lw1);
      *pa = static_cast<uint32_t>(hy0) | (static_cast<uint32_t>(hy1) << 16);
      *pb = static_cast<uint32_t>(hw0) | (static_cast<uint32_t>(hw1) << 16);
      *reinterpret_cast<uint32_t*>(side + sw64_off(row, i)) =
          static_cast<uint32_t>(ly0) | (static_cast<uint32_t>(ly1) << 16);
      *reinterpret_cast<uint32_t*>(side + sw64_off(row, i + h)) =
          static_cast<uint32_t>(lw0) | (static_cast<uint32_t>(lw1) << 16);
    }
  } else {
    for (int i = 0; i < h; ++i) {
      uint16_t* pa = reinterpret_cast<uint16_t*>(tile + sw64_off(row, i));
      uint16_t* pb = reinterpret_cast<uint16_t*>(tile + sw64_off(row, i + h));
      const float x = bf16_bits_to_f32(*pa), z = bf16_bits_to_f32(*pb);
      float y = x, w = z;
      if (pos >= 0) {
        const float2 t = cs[pos * h + i];
        y = fmaf(x, t.x, -z * t.y);
        w = fmaf(z, t.x, x * t.y);
      }
      uint16_t hy, ly, hw, lw;
      split_hi_lo(y, hy, ly);
      split_hi_lo(w, hw, lw);
      *pa = hy;
      *pb = hw;
      *reinterpret_cast<uint16_t*>(side + sw64_off(row, i)) = ly;
      *reinterpret_cast<uint16_t*>(side + sw64_off(row, i + h)) = lw;
    }
  }
}

// ---- register-staged variant: the table loads of a whole chunk are issued together
// (and can be issued ahead of the shared-memory data), so a row costs one L2 round trip
// per chunk of pairs instead of one per pair.  Needs r/2 even (float4 = two pairs).
constexpr int kCsChunkPairs = 12;

struct CsChunk {
  float4 v[2][kCsChunkPairs / 2];  // two rows x (cos_i, sin_i, cos_i+1, sin_i+1) per pair of pairs
};

// Table entries for pairs [i0, i0 + kCsChunkPairs) of two rows at positions p0, p1 (< 0: past the
// end of the sequence, loaded as the identity rotation).
__device__ __forceinline__ void cs_load(CsChunk& c, const float2* __restrict__ cs, int h, int i0, int64_t p0,
                                        int64_t p1) {
#pragma unroll
  for (int q = 0; q < kCsChunkPairs / 2; ++q) {
    const int i = i0 + 2 * q;
    float4 a = make_float4(1.0f, 0.0f, 1.0f, 0.0f), b = a;
    if (i < h) {
      if (p0 >= 0) a = __ldg(reinterpret_cast<const float4*>(cs + p0 * h + i));
      if (p1 >= 0) b = __ldg(reinterpret_cast<const float4*>(cs + p1 * h + i));
    }
    c.v[0][q] = a;
    c.v[1][q] = b;
  }
}

// Rotate pairs [i0, i0 + kCsChunkPairs) of one row with table entries already in registers.
__device__ __forceinline__ void rotate_chunk(uint8_t* __restrict__ tile, uint8_t* __restrict__ side, int row, int h,
                                             int i0, const float4 (&t)[kCsChunkPairs / 2]) {
#pragma unroll
  for (int q = 0; q < kCsChunkPairs / 2; ++q) {
    const int i = i0 + 2 * q;
    if (i >= h) break;
    uint32_t* pa = reinterpret_cast<uint32_t*>(tile + sw64_off(row, i));
    uint32_t* pb = reinterpret_cast<uint32_t*>(tile + sw64_off(row, i + h));
    const uint32_t a = *pa, b = *pb;
    const float x0 = bf16_bits_to_f32(static_cast<uint16_t>(a & 0xFFFF));
    const float x1 = bf16_bits_to_f32(static_cast<uint16_t>(a >> 16));
    const float z0 = bf16_bits_to_f32(static_cast<uint16_t>(b & 0xFFFF));
    const float z1 = bf16_bits_to_f32(static_cast<uint16_t>(b >> 16));
    const float y0 = fmaf(x0, t[q].x, -z0 * t[q].y), w0 = fmaf(z0, t[q].x, x0 * t[q].y);
    const float y1 = fmaf(x1, t[q].z, -z1 * t[q].w), w1 = fmaf(z1, t[q].z, x1 * t[q].w);
    uint16_t hy0, ly0, hy1, ly1, hw0, lw0, hw1, lw1;
    split_hi_lo(y0, hy0, ly0);
    split_hi_lo(y1, hy1, ly1);
    split_hi_lo(w0, hw0, lw0);
    split_hi_lo(w1, hw1, lw1);
    *pa = static_cast<uint32_t>(hy0) | (static_cast<uint32_t>(hy1) << 16);
    *pb = static_cast<uint32_t>(hw0) | (static_cast<uint32_t>(hw1) << 16);
    *reinterpret_cast<uint32_t*>(side + sw64_off(row, i)) = static_cast<uint32_t>(ly0) | (static_cast<uint32_t>(ly1) << 16);
    *reinterpret_cast<uint32_t*>(side + sw64_off(row, i + h)) =
        static_cast<uint32_t>(lw0) | (static_cast<uint32_t>(lw1) << 16);
  }
}

// Two rows of a tile, every chunk: loads of a chunk in flight together.
__device__ __forceinline__ void rotate_two_rows(uint8_t* tile, uint8_t* side, int row0, int row1, int64_t p0,
                                                int64_t p1, const float2* __restrict__ cs, int r) {
  const int h = r >> 1;
  if ((h & 1) == 0) {
    for (int i0 = 0; i0 < h; i0 += kCsChunkPairs) {
      CsChunk c;
      cs_load(c, cs, h, i0, p0, p1);
      rotate_chunk(tile, side, row0, h, i0, c.v[0]);
      rotate_chunk(tile, side, row1, h, i0, c.v[1]);
    }
  } else {
    rotate_row(tile, side, row0, p0, cs, r);
    rotate_row(tile, side, row1, p1, cs, r);
  }
}

// ---- vectorised variants: whole 16-byte chunks (8 dims) per shared access --------
// bf16x8 <-> fp32 helpers
__device__ __forceinline__ void unpack8(const uint4 v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}
// hi = bf16(y), lo = bf16(y - hi) for 8 values, packed
__device__ __forceinline__ void split8(const float* y, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    h[k] = pack_bf16x2(y[2 * k], y[2 * k + 1]);
    const float r0 = y[2 * k] - __uint_as_float(h[k] << 16);
    const float r1 = y[2 * k + 1] - __uint_as_float(h[k] & 0xFFFF0000u);
    l[k] = pack_bf16x2(r0, r1);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Table entries of pairs [i0, i0 + 2n) of a row at position pos (< 0: identity), as n
// float4 = (cos_i, sin_i, cos_i+1, sin_i+1).  Needs r/2 and i0 even.
template <int N>
__device__ __forceinline__ void cs_load_n(float4* t, const float2* __restrict__ cs, int h, int i0, int64_t pos) {
#pragma unroll
  for (int q = 0; q < N; ++q)
    t[q] = pos >= 0 ? __ldg(reinterpret_cast<const float4*>(cs + pos * h + i0 + 2 * q)) : make_float4(1.f, 0.f, 1.f, 0.f);
}

// r = 8 * NCH <= 32: the whole rotated prefix of the row lives in registers; NCH chunk
// loads, then NCH hi stores (in place) and NCH lo stores (side tile).
//
// Packed last chunk (NCH odd, i.e. r % 16 == 8; pack != 0): the side tile's last 16-column
// chunk holds both halves of the cross terms of the final 8 dims, so that one MMA chunk
// accumulates q_lo.k_hi + q_hi.k_lo there instead of two half-empty chunks.  For a query
// row (pack = 1) it is [lo | hi], for a key row (pack = 2) [hi | lo].
template <int NCH>
__device__ __forceinline__ void rotate_row_small(uint8_t* __restrict__ tile, uint8_t* __restrict__ side, int row,
                                                 const float4* t, int pack = 0) {
  constexpr int R = 8 * NCH, HH = R / 2;
  float x[R], y[R];
#pragma unroll
  for (int c = 0; c < NCH; ++c) unpack8(*reinterpret_cast<const uint4*>(tile + sw64_off(row, 8 * c)), x + 8 * c);
#pragma unroll
  for (int i = 0; i < HH; ++i) {
    const float cth = (i & 1) ? t[i >> 1].z : t[i >> 1].x;
    const float sth = (i & 1) ? t[i >> 1].w : t[i >> 1].y;
    y[i] = fmaf(x[i], cth, -x[i + HH] * sth);
    y[i + HH] = fmaf(x[i + HH], cth, x[i] * sth);
  }
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    uint4 hi, lo;
    split8(y + 8 * c, hi, lo);
    *reinterpret_cast<uint4*>(tile + sw64_off(row, 8 * c)) = hi;
    if ((NCH & 1) && c == NCH - 1 && pack != 0) {
      *reinterpret_cast<uint4*>(side + sw64_off(row, 8 * c)) = pack == 1 ? lo : hi;
      *reinterpret_cast<uint4*>(side + sw64_off(row, 8 * c + 8)) = pack == 1 ? hi : lo;
    } else {
      *reinterpret_cast<uint4*>(side + sw64_off(row, 8 * c)) = lo;
    }
  }
}

// Eight pairs (x_i, z_i) turned by the angles in t (four float4 = (cos, sin) of two
// consecutive pairs each): y = x cos - z sin, w = z cos + x sin, in fp32.  The one place
// this arithmetic is written, so the in-kernel rotation and the pre-rotation pass give
// bit-identical results.
__device__ __forceinline__ void rotate_pairs8(const float* x, const float* z, const float4* t, float* y, float* w) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float cth = (i & 1) ? t[i >> 1].z : t[i >> 1].x;
    const float sth = (i & 1) ? t[i >> 1].w : t[i >> 1].y;
    y[i] = fmaf(x[i], cth, -z[i] * sth);
    w[i] = fmaf(z[i], cth, x[i] * sth);
  }
}

// r % 16 == 0: eight pairs (i0..i0+7 with partners i0+h..i0+h+7) per step, two chunks
// in, four chunks out.
__device__ __forceinline__ void rotate_group8(uint8_t* __restrict__ tile, uint8_t* __restrict__ side, int row, int i0,
                                              int h, const float4* t) {
  float x[8], z[8], y[8], w[8];
  unpack8(*reinterpret_cast<const uint4*>(tile + sw64_off(row, i0)), x);
  unpack8(*reinterpret_cast<const uint4*>(tile + sw64_off(row, i0 + h)), z);
  rotate_pairs8(x, z, t, y, w);
  uint4 hi, lo;
  split8(y, hi, lo);
  *reinterpret_cast<uint4*>(tile + sw64_off(row, i0)) = hi;
  *reinterpret_cast<uint4*>(side + sw64_off(row, i0)) = lo;
  split8(w, hi, lo);
  *reinterpret_cast<uint4*>(tile + sw64_off(row, i0 + h)) = hi;
  *reinterpret_cast<uint4*>(side + sw64_off(row, i0 + h)) = lo;
}

// ---- fp16 operands for the rotated chunks (rotary_dim 16, 24, 32, in-kernel rotation) ----
// The rotated values, and for rotary_dim 24 dims 24..31 as they are, are rounded once to fp16
// in place, so the first rotary_dim/16 (rounded up) 16-column MMA chunks run as fp16 x fp16
// (the others bf16 x bf16) with no lo products: fp16 keeps 11 significant bits to bf16's 8.
// fp16 holds |v| <= 65504; each call returns false when a value it wrote is beyond that.
__device__ __forceinline__ uint4 pack8_f16(const float* v) {
  return make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]), pack_f16x2(v[6], v[7]));
}
__device__ __forceinline__ float absmax8(const float* v) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  return m;
}
constexpr float kF16Max = 65504.0f;

// rotary_dim 24: dims 0..23 rotated and 24..31 unchanged, as fp16 (MMA chunks 0 and 1).
__device__ __forceinline__ bool rotate_row_r24_f16(uint8_t* __restrict__ tile, int row, const float4* t) {
  float x[32], y[24];
#pragma unroll
  for (int c = 0; c < 4; ++c) unpack8(*reinterpret_cast<const uint4*>(tile + sw64_off(row, 8 * c)), x + 8 * c);
#pragma unroll
  for (int i = 0; i < 12; ++i) {  // the expressions of rotate_row_small
    const float cth = (i & 1) ? t[i >> 1].z : t[i >> 1].x;
    const float sth = (i & 1) ? t[i >> 1].w : t[i >> 1].y;
    y[i] = fmaf(x[i], cth, -x[i + 12] * sth);
    y[i + 12] = fmaf(x[i + 12], cth, x[i] * sth);
  }
  float m = absmax8(x + 24);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float* v = c < 3 ? y + 8 * c : x + 24;
    if (c < 3) m = fmaxf(m, absmax8(v));
    *reinterpret_cast<uint4*>(tile + sw64_off(row, 8 * c)) = pack8_f16(v);
  }
  return !(m > kF16Max);
}

// r % 16 == 0 (16 or 32): eight pairs (i0..i0+7 with partners i0+h..i0+h+7), as fp16.
__device__ __forceinline__ bool rotate_group8_f16(uint8_t* __restrict__ tile, int row, int i0, int h,
                                                  const float4* t) {
  float x[8], z[8], y[8], w[8];
  unpack8(*reinterpret_cast<const uint4*>(tile + sw64_off(row, i0)), x);
  unpack8(*reinterpret_cast<const uint4*>(tile + sw64_off(row, i0 + h)), z);
  rotate_pairs8(x, z, t, y, w);
  *reinterpret_cast<uint4*>(tile + sw64_off(row, i0)) = pack8_f16(y);
  *reinterpret_cast<uint4*>(tile + sw64_off(row, i0 + h)) = pack8_f16(w);
  return !(fmaxf(absmax8(y), absmax8(w)) > kF16Max);
}

// Two rows of a tile for r % 16 == 0, any size: group g's table loads are issued while
// group g-1 is being rotated.  t0 / t1 (8 float4 each) are the caller's buffers for
// rows row0 / row1: entries [0, 4) and [4, 8) alternate between groups.
__device__ __forceinline__ void rotate_two_rows_groups(uint8_t* tile, uint8_t* side, int row0, int row1, int64_t p0,
                                                       int64_t p1, const float2* __restrict__ cs, int h, float4* t0,
                                                       float4* t1) {
  cs_load_n<4>(t0, cs, h, 0, p0);
  cs_load_n<4>(t1, cs, h, 0, p1);
  for (int i0 = 0; i0 < h; i0 += 16) {
    if (i0 + 8 < h) {
      cs_load_n<4>(t0 + 4, cs, h, i0 + 8, p0);
      cs_load_n<4>(t1 + 4, cs, h, i0 + 8, p1);
    }
    rotate_group8(tile, side, row0, i0, h, t0);
    rotate_group8(tile, side, row1, i0, h, t1);
    if (i0 + 8 >= h) break;
    if (i0 + 16 < h) {
      cs_load_n<4>(t0, cs, h, i0 + 16, p0);
      cs_load_n<4>(t1, cs, h, i0 + 16, p1);
    }
    rotate_group8(tile, side, row0, i0 + 8, h, t0 + 4);
    rotate_group8(tile, side, row1, i0 + 8, h, t1 + 4);
  }
}

// Pre-rotation pass (the alternative to rotating K tiles inside the attention kernel for
// every query unit): writes rot[B, S, H, 4, D] bf16 with slot 0 = hi(q'), 1 = lo(q'),
// 2 = hi(k'), 3 = lo(k') where q' = R(s) q, k' = R(s) k and lo is zero at dims >= r, so
// the attention kernel can load the split operands with TMA and rotate nothing.  Needs
// r % 16 == 0 (the side tiles then hold plain lo columns).  One warp per (b, s, h) row:
// lanes 0..15 do q, lanes 16..31 do k, lane c of a half owns the 8-dim chunk c; a chunk
// of the first half of the rotated dims also writes its partner chunk.
// rotary_dim 24 (the GPT-NeoX-20B setting): the 24 rotated dims of a row in registers, as
// rotate_row_small<3> does, and the lo slot laid out as the attention kernel's side tile
// for r = 24: lo of dims 0..15, then one chunk holding the cross terms of dims 16..23 packed
// ([lo | hi] for q', [hi | lo] for k'), zero beyond.  One thread per (row, q or k).
template <int D>
__device__ __forceinline__ void prerotate_r24(const uint16_t* __restrict__ src, uint16_t* __restrict__ hi,
                                              uint16_t* __restrict__ lo, const float2* __restrict__ cs, int64_t pos,
                                              bool is_q) {
  constexpr int HH = 12;
  float x[24], y[24];
#pragma unroll
  for (int c = 0; c < 3; ++c) unpack8(*reinterpret_cast<const uint4*>(src + 8 * c), x + 8 * c);
  float4 t[6];
  cs_load_n<6>(t, cs, HH, 0, pos);
#pragma unroll
  for (int i0 = 0; i0 < HH; i0 += 4) {  // same expressions as rotate_pairs8, four pairs at a time
#pragma unroll
    for (int i = i0; i < i0 + 4; ++i) {
      const float cth = (i & 1) ? t[i >> 1].z : t[i >> 1].x;
      const float sth = (i & 1) ? t[i >> 1].w : t[i >> 1].y;
      y[i] = fmaf(x[i], cth, -x[i + HH] * sth);
      y[i + HH] = fmaf(x[i + HH], cth, x[i] * sth);
    }
  }
  uint4 h4[3], l4[3];
#pragma unroll
  for (int c = 0; c < 3; ++c) split8(y + 8 * c, h4[c], l4[c]);
#pragma unroll
  for (int c = 0; c < 3; ++c) *reinterpret_cast<uint4*>(hi + 8 * c) = h4[c];
#pragma unroll
  for (int c = 3; c < D / 8; ++c) *reinterpret_cast<uint4*>(hi + 8 * c) = *reinterpret_cast<const uint4*>(src + 8 * c);
  *reinterpret_cast<uint4*>(lo + 0) = l4[0];
  *reinterpret_cast<uint4*>(lo + 8) = l4[1];
  *reinterpret_cast<uint4*>(lo + 16) = is_q ? l4[2] : h4[2];
  *reinterpret_cast<uint4*>(lo + 24) = is_q ? h4[2] : l4[2];
#pragma unroll
  for (int c = 4; c < D / 8; ++c) *reinterpret_cast<uint4*>(lo + 8 * c) = make_uint4(0, 0, 0, 0);
}

// r = 24: one thread per (row, q or k), 256 threads = 128 rows per block.
template <int D>
__global__ void __launch_bounds__(256) rope_prerotate_r24_kernel(const uint16_t* __restrict__ qkv,
                                                                 uint16_t* __restrict__ rot,
                                                                 const float2* __restrict__ cs, int64_t rows, int S,
                                                                 int H) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 128 + (threadIdx.x >> 1);
  if (row >= rows) return;
  const int which = threadIdx.x & 1;  // 0: q, 1: k
  const int64_t pos = (row / H) % S;
  uint16_t* hi = rot + row * 4 * D + 2 * which * D;
  prerotate_r24<D>(qkv + row * 3 * D + which * D, hi, hi + D, cs, pos, which == 0);
}

template <int D>
__global__ void __launch_bounds__(256) rope_prerotate_kernel(const uint16_t* __restrict__ qkv, uint16_t* __restrict__ rot,
                                                             const float2* __restrict__ cs, int64_t rows, int S, int H,
                                                             int r) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int which = lane >> 4;  // 0: q, 1: k
  const int c = lane & 15;      // 8-dim chunk
  if (c >= D / 8) return;
  const int h = r >> 1;
  const int64_t pos = (row / H) % S;  // row = (b * S + s) * H + hd
  const uint16_t* src = qkv + row * 3 * D + which * D;
  uint16_t* hi = rot + row * 4 * D + 2 * which * D;
  uint16_t* lo = hi + D;
  if (8 * c < h) {
    const int i0 = 8 * c;
    float x[8], z[8], y[8], w[8];
    unpack8(*reinterpret_cast<const uint4*>(src + i0), x);
    unpack8(*reinterpret_cast<const uint4*>(src + i0 + h), z);
    float4 t[4];
    cs_load_n<4>(t, cs, h, i0, pos);
    rotate_pairs8(x, z, t, y, w);
    uint4 a, b;
    split8(y, a, b);
    *reinterpret_cast<uint4*>(hi + i0) = a;
    *reinterpret_cast<uint4*>(lo + i0) = b;
    split8(w, a, b);
    *reinterpret_cast<uint4*>(hi + i0 + h) = a;
    *reinterpret_cast<uint4*>(lo + i0 + h) = b;
  } else if (8 * c >= r) {
    *reinterpret_cast<uint4*>(hi + 8 * c) = *reinterpret_cast<const uint4*>(src + 8 * c);
    *reinterpret_cast<uint4*>(lo + 8 * c) = make_uint4(0, 0, 0, 0);
  }
}

}  // namespace neox
