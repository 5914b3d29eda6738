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
//     K and V through a 2-stage shared-memory ring (TMA, the same 64-byte-swizzled
//     [128][32] blocks as the prefill, which makes one-key-row-per-thread reads free of
//     bank conflicts).  Warp 0 issues the copies; 128 consumer threads each own one key
//     row of every tile: rotate, score, online softmax, accumulate p * v into registers.
//     The CTA then reduces its 128 partial states and writes (m, l, o[D]) for its split.
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

constexpr int kDecThreads = 160;  // warp 0: TMA; warps 1-4: one key row each
constexpr int kDecStages = 2;

__host__ __device__ constexpr int dec_tile_bytes(int D) { return tile_bytes(D); }
// smem: stages x (K tile + V tile), q' (fp32 D), barriers; the tiles double as the
// reduction buffer [D][128] fp32 at the end (D * 512 bytes <= 2 stages x 2 tiles).
__host__ __device__ constexpr int dec_smem_bytes(int D) {
  return kDecStages * 2 * dec_tile_bytes(D) + D * 4 + 64 + 512;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int D, bool SMALL_R>
__global__ void __launch_bounds__(kDecThreads, 2)
    attn_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 511) & ~uintptr_t(511));
  constexpr int TB = dec_tile_bytes(D);
  float* qs = reinterpret_cast<float*>(smem + kDecStages * 2 * TB);  // q' scaled by log2(e)/sqrt(D)
  uint64_t* bars = reinterpret_cast<uint64_t*>(qs + D);               // full[2], empty[2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kDecStages);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kDecStages + s]); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int h2 = p.r >> 1;
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
      mbar_init(empty(s), 128);
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
    for (int e = p.r + d; e < D; e += 128) qs[e] = bf16_bits_to_f32(qn[e]) * p.scale_log2;
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
        mbar_arrive_expect_tx(full(s), 2 * TB);
        armed |= 1 << s;
        par_bits = (par_bits & ~(1u << s)) | (lap << s);
        uint8_t* kt = smem + (2 * s) * TB;
        uint8_t* vt = smem + (2 * s + 1) * TB;
        for (int cb = 0; cb < D / kBlkCols; ++cb) {
          tma_load_4d(smem_u32(kt + cb * kBlkBytes), &kmap, full(s), cb * kBlkCols, t * kRows, h, b);
          tma_load_4d(smem_u32(vt + cb * kBlkBytes), &vmap, full(s), cb * kBlkCols, t * kRows, h, b);
        }
      }
      if (!ok || *abort_flag)
        for (int s = 0; s < kDecStages; ++s)
          if (armed & (1 << s)) drain_phase(full(s), (par_bits >> s) & 1, lim);
    }
    __syncwarp();
  } else {
    // =============================================================== consumers ====
    const int row = tid - 32;  // key row of every tile
    // row factor of the rotation angle: (cos, sin)(row * w_i), i < r/2 (r <= 32)
    float2 off[SMALL_R ? 16 : 1];
    if (SMALL_R) {
#pragma unroll
      for (int i = 0; i < 16; ++i) off[i] = i < h2 ? p.cs[static_cast<int64_t>(row) * h2 + i] : make_float2(1.f, 0.f);
    }
    float m = -INFINITY, l = 0.0f;
    float o[D];
#pragma unroll
    for (int d = 0; d < D; ++d) o[d] = 0.0f;
    const uint16_t* kn = qn + D;
    const uint16_t* vn = qn + 2 * D;
    bool ok = true;
    for (int t = t0; t < t1; ++t) {
      const int s = (t - t0) % kDecStages;
      const uint32_t lap = static_cast<uint32_t>((t - t0) / kDecStages) & 1u;
      if (!wait_phase(full(s), lap, abort_flag, lim, 51)) { ok = false; break; }
      const uint8_t* kt = smem + (2 * s) * TB;
      const uint8_t* vt = smem + (2 * s + 1) * TB;
      const int key = t * kRows + row;
      if (key <= P) {
        const bool is_new = key == P;
        // k row: the new token's from global, a cached one from the tile
        auto kword = [&](int c8, int q) -> uint32_t {  // 32-bit word q (0..3) of 8-dim chunk c8
          if (is_new) return reinterpret_cast<const uint32_t*>(kn)[c8 * 4 + q];
          return reinterpret_cast<const uint32_t*>(kt + sw64_off(row, 8 * c8))[q];
        };
        auto vword = [&](int c8, int q) -> uint32_t {
          if (is_new) return reinterpret_cast<const uint32_t*>(vn)[c8 * 4 + q];
          return reinterpret_cast<const uint32_t*>(vt + sw64_off(row, 8 * c8))[q];
        };
        float sc = 0.0f;
        // rotated dims: pairs (i, i + r/2)
        if (p.r > 0) {
          if (SMALL_R) {
            const float2* tb = p.cs + static_cast<int64_t>(t) * kRows * h2;  // angle of 128 t
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (i < h2) {
                const float2 bt = tb[i];
                const float c = bt.x * off[i].x - bt.y * off[i].y, sn = bt.y * off[i].x + bt.x * off[i].y;
                const uint32_t w1 = kword(i >> 3, (i & 7) >> 1), w2 = kword((i + h2) >> 3, ((i + h2) & 7) >> 1);
                const float x1 = (i & 1) ? bf16hi(w1) : bf16lo(w1);
                const float x2 = ((i + h2) & 1) ? bf16hi(w2) : bf16lo(w2);
                sc = fmaf(qs[i], x1 * c - x2 * sn, sc);
                sc = fmaf(qs[i + h2], x2 * c + x1 * sn, sc);
              }
            }
          } else {
            const float2* cr = p.cs + static_cast<int64_t>(key) * h2;
            for (int i = 0; i < h2; ++i) {
              const float2 cs = cr[i];
              const uint32_t w1 = kword(i >> 3, (i & 7) >> 1), w2 = kword((i + h2) >> 3, ((i + h2) & 7) >> 1);
              const float x1 = (i & 1) ? bf16hi(w1) : bf16lo(w1);
              const float x2 = ((i + h2) & 1) ? bf16hi(w2) : bf16lo(w2);
              sc = fmaf(qs[i], x1 * cs.x - x2 * cs.y, sc);
              sc = fmaf(qs[i + h2], x2 * cs.x + x1 * cs.y, sc);
            }
          }
        }
        // pass-through dims, 8 at a time (r is even; chunks from r rounded down)
        for (int c8 = p.r >> 3; c8 < D / 8; ++c8) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int d0 = 8 * c8 + 2 * q;
            const uint32_t w = kword(c8, q);
            if (d0 >= p.r) sc = fmaf(qs[d0], bf16lo(w), sc);
            if (d0 + 1 >= p.r) sc = fmaf(qs[d0 + 1], bf16hi(w), sc);
          }
        }
        // online softmax of this thread's keys (log2 units), lazy rescale beyond 2^8
        float pw;
        if (sc > m + 8.0f || m == -INFINITY) {
          const float mn = fmaxf(sc, m);
          const float f = ex2_approx(m - mn);
          l *= f;
#pragma unroll
          for (int d = 0; d < D; ++d) o[d] *= f;
          m = mn;
        }
        pw = ex2_approx(sc - m);
        l += pw;
#pragma unroll
        for (int c8 = 0; c8 < D / 8; ++c8) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t w = vword(c8, q);
            o[8 * c8 + 2 * q] = fmaf(pw, bf16lo(w), o[8 * c8 + 2 * q]);
            o[8 * c8 + 2 * q + 1] = fmaf(pw, bf16hi(w), o[8 * c8 + 2 * q + 1]);
          }
        }
        if (is_new) {  // append the new token's raw key and value (its tile has landed)
          uint4* kd = reinterpret_cast<uint4*>(p.k_cache + ((static_cast<int64_t>(b) * p.H + h) * p.Smax + P) * D);
          uint4* vd = reinterpret_cast<uint4*>(p.v_cache + ((static_cast<int64_t>(b) * p.H + h) * p.Smax + P) * D);
          const uint4* ks = reinterpret_cast<const uint4*>(kn);
          const uint4* vs = reinterpret_cast<const uint4*>(vn);
#pragma unroll
          for (int c8 = 0; c8 < D / 8; ++c8) {
            kd[c8] = ks[c8];
            vd[c8] = vs[c8];
          }
        }
      }
      mbar_arrive(empty(s));  // this thread is done with stage s
    }
    // ---- CTA reduction of the 128 partial states -> (o, m, l) of this split
    // (all tiles are consumed; the ring becomes the [D][128] buffer once every thread
    // has passed its last tile, ensured by the barrier below)
    float* red = reinterpret_cast<float*>(smem);
    float* mred = qs;  // 4 warp maxima (q' is no longer needed after the barrier)
    float wm = m;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, k));
    asm volatile("bar.sync 1, 128;" ::: "memory");  // consumers only: every tile consumed
    if (lane == 0) mred[warp - 1] = wm;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const float M = fmaxf(fmaxf(mred[0], mred[1]), fmaxf(mred[2], mred[3]));
    const float f = (m == -INFINITY) ? 0.0f : ex2_approx(m - M);
    float lf = l * f;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) lf += __shfl_xor_sync(0xffffffffu, lf, k);
#pragma unroll
    for (int d = 0; d < D; ++d) red[d * 128 + row] = o[d] * f;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (lane == 0) mred[4 + warp - 1] = lf;
    for (int d = row; d < D; d += 128) {
      float acc = 0.0f;
      for (int k = 0; k < 128; ++k) acc += red[d * 128 + (k + d) % 128];
      part[d] = acc;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (row == 0) {
      part[D] = M;
      part[D + 1] = mred[4] + mred[5] + mred[6] + mred[7];
    }
    (void)ok;
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
