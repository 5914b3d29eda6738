// decode.cuh -- incremental decode: one new token per sequence against a key/value cache.
//
// GPT-NeoX serving runs a per-token decoder against a growing context ("GPT-NeoX on
// FasterTransformer" guide, section "背景").  This op: sequence b already holds pos[b]
// tokens in the cache (keys as projected, NOT rotated; head-major [B, H, Smax, D]); the
// new token's packed projection qkv_new[b, h, 0|1|2, :] sits at position pos[b].  Its
// query, rotated at pos[b], attends to keys 0..pos[b], each rotated at its own position,
// with 1/sqrt(D) scaling; the new key and value are appended to the cache at row pos[b].
//
// One query per head makes this a matrix-vector product: HBM-bound (every cached key and
// value is read once), so the tensor cores have no part in it.  Layout of the work:
//   attn_decode_kernel: CTA (split, h, b) streams 128-key tiles [t0, t1) of its head's
//     K and V through a shared-memory ring: a head's cache rows are contiguous, so each
//     tile is one bulk copy per operand (row-major [128][D] in shared memory, rows past
//     Smax not copied).  Warp 0 issues the copies; 256 consumer threads
//     work in pairs on the key rows of every tile, each thread owning half of the head
//     dims: rotate, partial score (four independent FMA chains), pair sum, online
//     softmax, accumulate p * v for its dims in registers.  The CTA then reduces its 128
//     partial states and writes (m, l, o[D]) for its split.
//   attn_decode_combine_kernel: merges the splits of a head into out (bf16) and lse.
// Rotation: dims i < r/2 pair with i + r/2.  For r <= 32 the angle of key p = 128 t + row
// comes from angle addition, (cos, sin)(p w) = (cos, sin)(128 t w) x (cos, sin)(row w),
// with the row factor held in registers and the tile factor read once per tile (both are
// table entries, fp64-computed and stored fp32; the product is within ~3e-7 of the exact
// value, far below the 2^-9 of the bf16 inputs); for larger r each key reads its own
// table row.
#pragma once

#include "attn_common.cuh"

namespace neox {

struct DecodeParams {
  const uint16_t* qkv_new;  // bf16 [B, H, 3, D]
  uint16_t* k_cache;        // bf16 [B, H, Smax, D]
  uint16_t* v_cache;
  const int* pos;           // int32 [B]
  const float2* cs;         // cos/sin table [>= Smax rows][r/2]
  float* part;              // fp32 [B, H, splits, D + 2]: o[D], m, l  (m in log2 units)
  uint16_t* out;            // bf16 [B, H, D]
  float* lse;               // fp32 [B, H]
  int B, H, Smax, r;
  int splits, tiles_per_split;
  float scale_log2;         // log2(e) / sqrt(D)
  uint64_t wait_limit_ns;
};

constexpr int kDecThreads = 288;  // warp 0: TMA; warps 1-8: two threads per key row
// One CTA per SM (registers), with a deep ring: 4 stages of K + V tiles (3 for D = 128),
// 192 KB of loads in flight.
__host__ __device__ constexpr int dec_stages(int D) { return D == 128 ? 3 : 4; }
constexpr int kDecMaxStages = 4;

__host__ __device__ constexpr int dec_tile_bytes(int D) { return tile_bytes(D); }
// smem: stages x (K tile + V tile), q' (fp32 D), per stage the tile's angle factor (16
// float2), barriers; the tiles double as the reduction buffer [D][128] fp32 at the end
// (D * 512 bytes <= stages x 2 tiles).
__host__ __device__ constexpr int dec_smem_bytes(int D) {
  return dec_stages(D) * 2 * dec_tile_bytes(D) + D * 4 + kDecMaxStages * 16 * 8 + 2 * kDecMaxStages * 8 + 16 + 512;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// dim e (0..31) of four 8-dim chunks held in registers (e a compile-time constant after
// unrolling: no address is taken, so the chunks stay in registers)
__device__ __forceinline__ float dim_of(const uint4 (&k)[4], int e) {
  const uint4& c = k[e >> 3];
  const int q = (e & 7) >> 1;
  const uint32_t w = q == 0 ? c.x : q == 1 ? c.y : q == 2 ? c.z : c.w;
  return (e & 1) ? bf16hi(w) : bf16lo(w);
}
__device__ __forceinline__ float dim_of(const uint4& c, int e) {  // dim e (0..7) of one chunk
  const int q = e >> 1;
  const uint32_t w = q == 0 ? c.x : q == 1 ? c.y : q == 2 ? c.z : c.w;
  return (e & 1) ? bf16hi(w) : bf16lo(w);
}

// H2 = rotary_dim / 2 when it is 0, 4, 8, 12 or 16 (compile-time pairing, angle addition),
// or -1 for any other rotary_dim (runtime pairing, one table row per key).
template <int D, int H2>
__global__ void __launch_bounds__(kDecThreads, 1)
    attn_decode_kernel(const DecodeParams p) {
  constexpr bool SMALL_R = H2 >= 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 511) & ~uintptr_t(511));
  constexpr int TB = dec_tile_bytes(D);
  constexpr int kDecStages = dec_stages(D);
  float* qs = reinterpret_cast<float*>(smem + kDecStages * 2 * TB);  // q' scaled by log2(e)/sqrt(D)
  float2* tf = reinterpret_cast<float2*>(qs + D);                      // [stages][16] angle of 128 t
  uint64_t* bars = reinterpret_cast<uint64_t*>(tf + kDecStages * 16);  // full[stages], empty[stages]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kDecStages);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kDecStages + s]); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int h2 = SMALL_R ? H2 : (p.r >> 1);
  const uint64_t lim = p.wait_limit_ns;

  const int P = p.pos[b];
  const bool pos_ok = P >= 0 && P < p.Smax;
  const int n_tiles = pos_ok ? P / kRows + 1 : 0;
  const int t0 = split * p.tiles_per_split;
  const int t1 = min(t0 + p.tiles_per_split, n_tiles);
  float* part = p.part + ((static_cast<int64_t>(b) * p.H + h) * p.splits + split) * (D + 2);
  if (!pos_ok && split == 0 && tid == 0) record_error(kErrBadInput, 0);
  if (t0 >= t1) {  // nothing to do for this split: an empty partial state
    for (int d = tid; d < D; d += kDecThreads) part[d] = 0.0f;
    if (tid == 0) {
      part[D] = -INFINITY;
      part[D + 1] = 0.0f;
    }
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 256);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  // q' = rotate(q_new, P) * log2(e)/sqrt(D), by the consumer threads
  const uint16_t* qn = p.qkv_new + (static_cast<int64_t>(b) * p.H + h) * 3 * D;
  if (tid >= 32) {
    const int d = tid - 32;
    if (d < h2) {
      const float2 c = p.cs[static_cast<int64_t>(P) * h2 + d];
      const float x1 = bf16_bits_to_f32(qn[d]), x2 = bf16_bits_to_f32(qn[d + h2]);
      qs[d] = (x1 * c.x - x2 * c.y) * p.scale_log2;
      qs[d + h2] = (x2 * c.x + x1 * c.y) * p.scale_log2;
    }
    if (p.r + d < D) qs[p.r + d] = bf16_bits_to_f32(qn[p.r + d]) * p.scale_log2;
  }
  __syncthreads();

  if (warp == 0) {
    // ================================================================ producer ====
    if (lane == 0) {
      bool ok = true;
      int armed = 0;  // bitmask of stages with a load in flight, and their parities
      uint32_t par_bits = 0;
      for (int t = t0; t < t1 && ok; ++t) {
        const int s = (t - t0) % kDecStages;
        const uint32_t lap = static_cast<uint32_t>((t - t0) / kDecStages) & 1u;
        if (!wait_phase(empty(s), lap ^ 1, abort_flag, lim, 50)) { ok = false; break; }
        const int rows = min(kRows, p.Smax - t * kRows);  // never past the head's last row
        const uint32_t bytes = static_cast<uint32_t>(rows) * D * 2;
        if (SMALL_R)  // the tile's angle factor, published with the arrival below
          for (int i = 0; i < h2; ++i) tf[s * 16 + i] = p.cs[static_cast<int64_t>(t) * kRows * h2 + i];
        mbar_arrive_expect_tx(full(s), 2 * bytes);
        armed |= 1 << s;
        par_bits = (par_bits & ~(1u << s)) | (lap << s);
        const int64_t row0 = (static_cast<int64_t>(b) * p.H + h) * p.Smax + static_cast<int64_t>(t) * kRows;
        bulk_load(smem_u32(smem + (2 * s) * TB), p.k_cache + row0 * D, bytes, full(s));
        bulk_load(smem_u32(smem + (2 * s + 1) * TB), p.v_cache + row0 * D, bytes, full(s));
      }
      if (!ok || *abort_flag)
        for (int s = 0; s < kDecStages; ++s)
          if (armed & (1 << s)) drain_phase(full(s), (par_bits >> s) & 1, lim);
    }
    __syncwarp();
  } else {
    // =============================================================== consumers ====
    constexpr int DH = D / 2;           // output dims per thread
    const int c = tid - 32;             // 0..255
    const int row = c >> 1, half = c & 1;  // key row of every tile; which half of the dims
    // score dims: half 0 takes the rotated dims [0, r) and pass-through chunks up to `mid`,
    // half 1 the pass-through chunks from `mid` (8-dim chunks; r is even)
    const int r8 = p.r >> 3;  // first chunk holding a pass-through dim
    const int mid8 = r8 + (D / 8 - r8) / 2;
    const int cb0 = half == 0 ? r8 : mid8, cb1 = half == 0 ? mid8 : D / 8;
    // row factor of the rotation angle: (cos, sin)(row * w_i), i < r/2 (r <= 32, half 0)
    float2 off[SMALL_R && H2 > 0 ? H2 : 1];
    if constexpr (SMALL_R) {
#pragma unroll
      for (int i = 0; i < H2; ++i) off[i] = half == 0 ? p.cs[static_cast<int64_t>(row) * H2 + i] : make_float2(1.f, 0.f);
    }
    float m = -INFINITY, l = 0.0f;
    float o[DH];
#pragma unroll
    for (int d = 0; d < DH; ++d) o[d] = 0.0f;
    const uint16_t* kn = qn + D;
    const uint16_t* vn = qn + 2 * D;
    const float4* q4 = reinterpret_cast<const float4*>(qs);
    for (int t = t0; t < t1; ++t) {
      const int s = (t - t0) % kDecStages;
      const uint32_t lap = static_cast<uint32_t>((t - t0) / kDecStages) & 1u;
      // warp-uniform exit: the pair sum below is a warp-synchronous shuffle
      if (!__all_sync(0xffffffffu, wait_phase(full(s), lap, abort_flag, lim, 51))) break;
      const uint8_t* kt = smem + (2 * s) * TB;
      const uint8_t* vt = smem + (2 * s + 1) * TB;
      const int key = t * kRows + row;
      // lanes with a key in range (both threads of a pair agree): the shuffle's members
      const unsigned active = __ballot_sync(0xffffffffu, key <= P);
      if (key <= P) {
        const bool is_new = key == P;
        auto kchunk = [&](int c8) -> uint4 {  // dims [8 c8, 8 c8 + 8) of the key
          return is_new ? reinterpret_cast<const uint4*>(kn)[c8]
                        : reinterpret_cast<const uint4*>(kt + row * (2 * D))[c8];
        };
        float sa = 0.0f, sb = 0.0f, sc2 = 0.0f, sd = 0.0f;  // four independent chains
        if (half == 0 && h2 > 0) {
          if constexpr (SMALL_R) {
            const float2* tb = tf + s * 16;  // angle of 128 t
            uint4 kc[4];
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) kc[c8] = c8 * 8 < 2 * H2 ? kchunk(c8) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < H2; ++i) {
              {
                const float2 bt = tb[i];
                const float cth = bt.x * off[i].x - bt.y * off[i].y, sth = bt.y * off[i].x + bt.x * off[i].y;
                const int j2 = i + H2;
                const float x1 = dim_of(kc, i), x2 = dim_of(kc, j2);
                if (i & 1) {
                  sa = fmaf(qs[i], x1 * cth - x2 * sth, sa);
                  sb = fmaf(qs[j2], x2 * cth + x1 * sth, sb);
                } else {
                  sc2 = fmaf(qs[i], x1 * cth - x2 * sth, sc2);
                  sd = fmaf(qs[j2], x2 * cth + x1 * sth, sd);
                }
              }
            }
          } else {
            const float2* cr = p.cs + static_cast<int64_t>(key) * h2;
            for (int i = 0; i < h2; ++i) {
              const float2 cs = cr[i];
              const int j2 = i + h2;
              const uint4 ci = kchunk(i >> 3), cj = kchunk(j2 >> 3);
              const int ei = i & 7, ej = j2 & 7;
              float x1 = 0.0f, x2 = 0.0f;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                if (e == ei) x1 = dim_of(ci, e);
                if (e == ej) x2 = dim_of(cj, e);
              }
              sa = fmaf(qs[i], x1 * cs.x - x2 * cs.y, sa);
              sb = fmaf(qs[j2], x2 * cs.x + x1 * cs.y, sb);
            }
          }
        }
        // pass-through dims of this half, a chunk at a time
        for (int c8 = cb0; c8 < cb1; ++c8) {
          const uint4 kc = kchunk(c8);
          const float4 qa = q4[2 * c8], qb = q4[2 * c8 + 1];
          const int d0 = 8 * c8;
          if (d0 >= p.r) {
            sa = fmaf(qa.x, bf16lo(kc.x), sa);
            sb = fmaf(qa.y, bf16hi(kc.x), sb);
            sc2 = fmaf(qa.z, bf16lo(kc.y), sc2);
            sd = fmaf(qa.w, bf16hi(kc.y), sd);
            sa = fmaf(qb.x, bf16lo(kc.z), sa);
            sb = fmaf(qb.y, bf16hi(kc.z), sb);
            sc2 = fmaf(qb.z, bf16lo(kc.w), sc2);
            sd = fmaf(qb.w, bf16hi(kc.w), sd);
          } else {  // the chunk holding dim r: only its dims >= r
            const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (d0 + e >= p.r) sa = fmaf(qv[e], dim_of(kc, e), sa);
          }
        }
        float sc = (sa + sb) + (sc2 + sd);
        sc += __shfl_xor_sync(active, sc, 1);  // the pair's two halves
        // online softmax of this pair's keys (log2 units), lazy rescale beyond 2^8
        if (sc > m + 8.0f || m == -INFINITY) {
          const float mn = fmaxf(sc, m);
          const float f = ex2_approx(m - mn);
          l *= f;
#pragma unroll
          for (int d = 0; d < DH; ++d) o[d] *= f;
          m = mn;
        }
        const float pw = ex2_approx(sc - m);
        l += pw;
#pragma unroll
        for (int c8 = 0; c8 < DH / 8; ++c8) {
          const int cv = half * (DH / 8) + c8;
          const uint4 vc = is_new ? reinterpret_cast<const uint4*>(vn)[cv]
                                  : reinterpret_cast<const uint4*>(vt + row * (2 * D))[cv];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[8 * c8 + e] = fmaf(pw, dim_of(vc, e), o[8 * c8 + e]);
        }
        if (is_new) {  // append the new token's raw key and value (its tile has landed)
          uint4* kd = reinterpret_cast<uint4*>(p.k_cache + ((static_cast<int64_t>(b) * p.H + h) * p.Smax + P) * D);
          uint4* vd = reinterpret_cast<uint4*>(p.v_cache + ((static_cast<int64_t>(b) * p.H + h) * p.Smax + P) * D);
#pragma unroll
          for (int c8 = half * (D / 16); c8 < (half + 1) * (D / 16); ++c8) {
            kd[c8] = reinterpret_cast<const uint4*>(kn)[c8];
            vd[c8] = reinterpret_cast<const uint4*>(vn)[c8];
          }
        }
      }
      mbar_arrive(empty(s));  // this thread is done with stage s
    }
    // ---- CTA reduction of the 128 partial states -> (o, m, l) of this split
    // (the ring becomes the [D][128] buffer once every consumer has passed its last
    // tile, which the first barrier below ensures)
    float* red = reinterpret_cast<float*>(smem);
    float* mred = qs;  // 8 warp maxima, then 8 warp sums (q' is dead after the barrier)
    float wm = m;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, k));
    asm volatile("bar.sync 1, 256;" ::: "memory");  // consumers only: every tile consumed
    if (lane == 0) mred[warp - 1] = wm;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    float M = mred[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) M = fmaxf(M, mred[w]);
    const float f = (m == -INFINITY) ? 0.0f : ex2_approx(m - M);
    float lf = half == 0 ? l * f : 0.0f;  // each key's l counted once
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) lf += __shfl_xor_sync(0xffffffffu, lf, k);
#pragma unroll
    for (int d = 0; d < DH; ++d) red[(half * DH + d) * 128 + row] = o[d] * f;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (lane == 0) mred[8 + warp - 1] = lf;
    if (c < D) {
      float acc = 0.0f;
      for (int k = 0; k < 128; ++k) acc += red[c * 128 + (k + c) % 128];
      part[c] = acc;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (c == 0) {
      float L = 0.0f;
      for (int w = 0; w < 8; ++w) L += mred[8 + w];
      part[D] = M;
      part[D + 1] = L;
    }
  }
  __syncthreads();
}

// Merge the splits of head (b, h): M = max m_s, L = sum l_s 2^(m_s - M),
// out = sum o_s 2^(m_s - M) / L, lse = ln 2 * (M + log2 L).
template <int D>
__global__ void __launch_bounds__(128) attn_decode_combine_kernel(const DecodeParams p) {
  const int h = blockIdx.x, b = blockIdx.y;
  const float* part = p.part + (static_cast<int64_t>(b) * p.H + h) * p.splits * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < p.splits; ++s) M = fmaxf(M, part[s * (D + 2) + D]);
  float L = 0.0f;
  for (int s = 0; s < p.splits; ++s) {
    const float ms = part[s * (D + 2) + D];
    if (ms != -INFINITY) L += part[s * (D + 2) + D + 1] * ex2_approx(ms - M);
  }
  const float inv_l = 1.0f / L;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.0f;
    for (int s = 0; s < p.splits; ++s) {
      const float ms = part[s * (D + 2) + D];
      if (ms != -INFINITY) acc += part[s * (D + 2) + d] * ex2_approx(ms - M);
    }
    p.out[(static_cast<int64_t>(b) * p.H + h) * D + d] = f32_to_bf16_bits(acc * inv_l);
  }
  if (threadIdx.x == 0) p.lse[static_cast<int64_t>(b) * p.H + h] = (M + log2f(L)) * 0.69314718055994530942f;
}

}  // namespace neox
