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
//   attn_decode_kernel: persistent, one CTA per SM.  The B*H*ceil(Smax/128) key tiles of
//     all heads, taken head after head, are cut into one contiguous range per CTA (equal
//     to within one tile, whatever B, H and Smax are); the run of a range inside one head
//     is a work item.
//     Warp 0 streams the items' K and V tiles (one bulk copy per operand: a head's cache
//     rows are contiguous) through a shared-memory ring that runs on across items, and
//     each item's new-token row (q, k, v) and query angle into one of two item slots.
//     The 8 consumer warps form NG = 32 row groups of 8 lanes; group g takes rows g,
//     g + 32, g + 64, g + 96 of every tile, and
//     lane l of a group owns D/8 dims of the row (16-byte chunk l, plus chunk l+8 for
//     D = 128 or the 8-byte piece l of dims 64..95 for D = 96), so the 8
//     lanes reading one row touch 8 distinct bank groups.  Partial dot products meet in
//     three shuffles; each group keeps its own online softmax; at the end of an item the
//     groups merge by shuffles inside a warp and through shared memory across warps.
//   A head inside one CTA's range is written out by that CTA; a head spanning several
//   ranges leaves one partial state per range, and the last of its CTAs to finish (a
//   per-head arrival counter, reset to zero by that CTA) merges them into out and lse.
// Rotation, with the cache keys unrotated: for pair (i, i + r/2) and key angle phi,
//   q'_i k'_i + q'_{i+r/2} k'_{i+r/2} = k_i Re(z e^{-j phi}) + k_{i+r/2} Im(z e^{-j phi}),
// z = q'_i + j q'_{i+r/2}, so the query is turned instead of the key.  For r = 8..32 all
// rotated dims sit in chunk 0 of lanes 0..r/8-1, and e^{-j phi} of key 128 t + row splits
// into a tile factor (applied to z once per tile) and a row factor (held in registers:
// each lane sees the same rows in every tile); the product of the two fp32 table entries
// is within ~3e-7 of the exact value, far below the 2^-9 of the bf16 inputs.  Other r
// read each key's angle from the table.
#pragma once

#include "attn_common.cuh"

namespace neox {

struct DecodeParams {
  const uint16_t* qkv_new;  // bf16 [B, H, 3, D]
  uint16_t* k_cache;        // bf16 [B, H, Smax, D]
  uint16_t* v_cache;
  const int* pos;           // int32 [B]
  const float2* cs;         // cos/sin table [max(Smax, 128) rows][r/2]
  float* part;              // fp32 [B*H][runs_per_head][D + 2]: o[D], m, l  (m in log2 units)
  int* counters;            // int32 [B*H], zero between calls: runs of a head merged so far
  uint16_t* out;            // bf16 [B, H, D]
  float* lse;               // fp32 [B, H]
  int B, H, Smax, r;
  int tiles_per_head;       // ceil(Smax / 128)
  int runs_per_head;        // partial-state slots per head (CTAs one head's tiles can span)
  long long total_tiles;    // B * H * tiles_per_head
  float scale_log2;         // log2(e) / sqrt(D)
  uint64_t wait_limit_ns;
};

// warp 0: copies; then CW consumer warps = 4 CW row groups of 8 lanes, each group 128/(4 CW)
// rows of every tile.  CW = 8 for every D: 16 warps (2 rows per group) measured 16% slower
// for D = 64 (a 544-thread CTA caps a thread at 96 registers, and the per-tile work of a
// group is spread over fewer rows).
__host__ __device__ constexpr int dec_consumer_warps(int) { return 8; }
__host__ __device__ constexpr int dec_threads(int D) { return 32 + 32 * dec_consumer_warps(D); }
constexpr int kDecRingBytes = 192 * 1024;
// ring stages of K + V tiles in 192 KB: 6 (D = 64), 4 (D = 96), 3 (D = 128)
__host__ __device__ constexpr int dec_stages(int D) { return kDecRingBytes / (2 * tile_bytes(D)); }
__host__ __device__ constexpr int dec_slot_bytes(int D) { return 3 * D * 2 + 16 * 8; }  // q|k|v, query angle
// row factors of rows 0..127: per row 8 entries of 2 pairs (cos 2q, cos 2q+1, sin 2q,
// sin 2q+1) and the identity (1, 1, 0, 0)
constexpr int kDecRowTabBytes = kRows * 9 * 16;
// smem: ring, 2 item slots, per stage the tile factor (16 float2 + the identity), the
// cross-warp merge buffer [2][8][D + 2], the row factors, barriers, abort flag and the
// slots' positions
__host__ __device__ constexpr int dec_smem_bytes(int D) {
  return kDecRingBytes + 2 * dec_slot_bytes(D) + dec_stages(D) * 18 * 8 + 2 * dec_consumer_warps(D) * (D + 2) * 4 +
         kDecRowTabBytes +
         (2 * dec_stages(D) + 4) * 8 + 16 + 512;
}

// The CTA whose tile range holds global tile x (ranges [N c / G, N (c + 1) / G)).
__host__ __device__ __forceinline__ long long dec_cta_of(long long x, long long N, int G) {
  return ((x + 1) * G - 1) / N;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float word_dim(uint32_t w, int odd) { return odd ? bf16hi(w) : bf16lo(w); }
// two bf16 (lo, hi) as an fp32 pair, and fp32 pair helpers
__device__ __forceinline__ uint64_t bf16x2_f32x2(uint32_t w) { return f32x2_pack(bf16lo(w), bf16hi(w)); }
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float f2lo(uint64_t x) { return __uint_as_float(static_cast<uint32_t>(x)); }
__device__ __forceinline__ float f2hi(uint64_t x) { return __uint_as_float(static_cast<uint32_t>(x >> 32)); }

// The D/8 dims lane l8 of a row group owns: v < 8 -> 8 l8 + v (chunk l8); v >= 8 ->
// 64 + 8 l8 + (v - 8) (chunk l8 + 8, D = 128) or 64 + 4 l8 + (v - 8) (piece l8, D = 96).
template <int D>
__device__ __forceinline__ int lane_dim(int l8, int v) {
  return v < 8 ? 8 * l8 + v : (D == 128 ? 64 + 8 * l8 + (v - 8) : 64 + 4 * l8 + (v - 8));
}

// One row's share of a lane, as loaded from a row-major [*][D] bf16 row in shared memory.
template <int D>
struct LaneRow {
  uint4 c0;
  uint4 c1;  // D = 128
  uint2 pc;  // D = 96
  __device__ __forceinline__ void load(const uint8_t* row, int l8) {
    c0 = *reinterpret_cast<const uint4*>(row + 16 * l8);
    if constexpr (D == 128) c1 = *reinterpret_cast<const uint4*>(row + 128 + 16 * l8);
    if constexpr (D == 96) pc = *reinterpret_cast<const uint2*>(row + 128 + 8 * l8);
  }
  // dim v of the lane (v a compile-time constant after unrolling)
  __device__ __forceinline__ float at(int v) const {
    if (v < 8) {
      const int q = (v & 7) >> 1;
      return word_dim(q == 0 ? c0.x : q == 1 ? c0.y : q == 2 ? c0.z : c0.w, v & 1);
    }
    if constexpr (D == 128) {
      const int q = (v & 7) >> 1;
      return word_dim(q == 0 ? c1.x : q == 1 ? c1.y : q == 2 ? c1.z : c1.w, v & 1);
    }
    return word_dim(((v - 8) >> 1) == 0 ? pc.x : pc.y, v & 1);
  }
  // dims (2u, 2u + 1) of the lane as an fp32 pair
  __device__ __forceinline__ uint64_t pair(int u) const {
    if (u < 4) return bf16x2_f32x2(u == 0 ? c0.x : u == 1 ? c0.y : u == 2 ? c0.z : c0.w);
    if constexpr (D == 128) return bf16x2_f32x2(u == 4 ? c1.x : u == 5 ? c1.y : u == 6 ? c1.z : c1.w);
    return bf16x2_f32x2(u == 4 ? pc.x : pc.y);
  }
};

template <int N>
__device__ __forceinline__ float dec_max(const float (&x)[N]) {
  if constexpr (N == 2) return fmaxf(x[0], x[1]);
  return fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
}
template <int N>
__device__ __forceinline__ float dec_sum(const float (&x)[N]) {
  if constexpr (N == 2) return x[0] + x[1];
  return (x[0] + x[1]) + (x[2] + x[3]);
}

// Final output of head `head`, dim c, from a merged state (m in log2 units):
// out = o / l (bf16), lse = ln 2 * (m + log2 l); a head with no valid position (l = 0,
// reported through the device error word) gets out = 0, lse = -inf.
template <int D>
__device__ __forceinline__ void dec_write_out(const DecodeParams& p, long long head, int c, float o, float m,
                                              float l) {
  p.out[head * D + c] = f32_to_bf16_bits(l > 0.0f ? o * (1.0f / l) : 0.0f);
  if (c == 0) p.lse[head] = l > 0.0f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
}

// Named barrier 1 over the NT consumer threads, plain and OR-reducing a flag.
template <int NT>
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}
template <int NT>
__device__ __forceinline__ bool consumers_sync_or(bool flag) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(res)
      : "r"(static_cast<uint32_t>(flag)), "n"(NT)
      : "memory");
  return res != 0;
}

// H2 = rotary_dim / 2 when it is 0, 4, 8, 12 or 16 (tile x row factorisation of the
// angle), or -1 for any other rotary_dim (one table read per key and rotated dim).
template <int D, int H2>
__global__ void __launch_bounds__(dec_threads(D), 1)
    attn_decode_kernel(const DecodeParams p) {
  constexpr bool SMALL_R = H2 >= 0;
  constexpr int CW = dec_consumer_warps(D);  // consumer warps
  constexpr int NCT = 32 * CW;               // consumer threads
  constexpr int NG = 4 * CW;                 // row groups
  constexpr int RPG = kRows / NG;            // rows of a tile per group
  constexpr int NV = D / 8;  // dims per lane
  constexpr int S = dec_stages(D);
  constexpr int TB = tile_bytes(D);
  constexpr int SLOT = dec_slot_bytes(D);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 511) & ~uintptr_t(511));
  uint8_t* slots = smem + kDecRingBytes;                                  // [2][SLOT]
  float2* tf = reinterpret_cast<float2*>(slots + 2 * SLOT);              // [S][18]
  float* red = reinterpret_cast<float*>(tf + S * 18);                    // [2][CW][D + 2]
  float4* rtab = reinterpret_cast<float4*>(red + 2 * CW * (D + 2));      // [128][H2/2 + 1]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(rtab) + kDecRowTabBytes);
  int* misc = reinterpret_cast<int*>(bars + 2 * S + 4);                  // abort flag, slot positions
  volatile int* abort_flag = misc;
  int* slot_pos = misc + 1;
  volatile int* last_flag = misc + 3;
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[S + s]); };
  auto qfull = [&](int i) { return smem_u32(&bars[2 * S + i]); };
  auto qempty = [&](int i) { return smem_u32(&bars[2 * S + 2 + i]); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t lim = p.wait_limit_ns;
  const int G = gridDim.x, cta = blockIdx.x;
  const long long N = p.total_tiles;
  const long long lo = N * cta / G, hi = N * (cta + 1) / G;
  const int Th = p.tiles_per_head;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), CW);
      tf[s * 18 + 16] = make_float2(1.0f, 0.0f);  // identity factor for unrotated dims
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(qfull(i), 1);
      mbar_init(qempty(i), CW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ================================================================ producer ====
    bool ok = true;
    uint32_t armed = 0, par_bits = 0, qarmed = 0, qpar_bits = 0;
    uint32_t n = 0;  // tiles issued by this CTA
    int k = 0;       // items
    for (long long g = lo; g < hi && ok; ++k) {
      const long long head = g / Th;
      const int tb = static_cast<int>(g - head * Th);
      const long long gend = min(hi, (head + 1) * Th);
      const int te = tb + static_cast<int>(gend - g);
      g = gend;
      const int b = static_cast<int>(head / p.H);
      const int P = p.pos[b];
      const bool valid = P >= 0 && P < p.Smax;
      if (!valid && tb == 0 && lane == 0) record_error(kErrBadInput, 0);
      const int t1 = min(te, valid ? P / kRows + 1 : 0);
      const int slot = k & 1;
      const uint32_t qlap = static_cast<uint32_t>(k >> 1) & 1u;
      if (!__all_sync(0xffffffffu, wait_phase(qempty(slot), qlap ^ 1, abort_flag, lim, 52))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        slot_pos[slot] = P;  // published by the arrival below
        const bool tab = SMALL_R && H2 > 0 && valid;
        constexpr uint32_t kAngBytes = (SMALL_R ? H2 : 0) * 8;
        mbar_arrive_expect_tx(qfull(slot), 3 * D * 2 + (tab ? kAngBytes : 0));
        bulk_load(smem_u32(slots + slot * SLOT), p.qkv_new + head * 3 * D, 3 * D * 2, qfull(slot));
        if (tab)
          bulk_load(smem_u32(slots + slot * SLOT + 6 * D), p.cs + static_cast<long long>(P) * (SMALL_R ? H2 : 0),
                    kAngBytes, qfull(slot));
      }
      qarmed |= 1u << slot;
      qpar_bits = (qpar_bits & ~(1u << slot)) | (qlap << slot);
      for (int t = tb; t < t1; ++t, ++n) {
        const int s = static_cast<int>(n % S);
        const uint32_t lap = (n / S) & 1u;
        float2 fac = make_float2(1.0f, 0.0f);
        if (SMALL_R && lane < H2) fac = p.cs[static_cast<long long>(t) * kRows * (SMALL_R ? H2 : 0) + lane];
        if (!__all_sync(0xffffffffu, wait_phase(empty(s), lap ^ 1, abort_flag, lim, 50))) {
          ok = false;
          break;
        }
        if (SMALL_R && lane < H2) tf[s * 18 + lane] = fac;  // the tile factor, published below
        __syncwarp();
        if (lane == 0) {
          const int rows = min(kRows, p.Smax - t * kRows);  // never past the head's last row
          const uint32_t bytes = static_cast<uint32_t>(rows) * D * 2;
          mbar_arrive_expect_tx(full(s), 2 * bytes);
          const long long row0 = head * p.Smax + static_cast<long long>(t) * kRows;
          bulk_load(smem_u32(smem + (2 * s) * TB), p.k_cache + row0 * D, bytes, full(s));
          bulk_load(smem_u32(smem + (2 * s + 1) * TB), p.v_cache + row0 * D, bytes, full(s));
        }
        armed |= 1u << s;
        par_bits = (par_bits & ~(1u << s)) | (lap << s);
      }
    }
    if (lane == 0 && (!ok || *abort_flag)) {  // let every copy in flight land before exit
      for (int s = 0; s < S; ++s)
        if (armed & (1u << s)) drain_phase(full(s), (par_bits >> s) & 1, lim);
      for (int i = 0; i < 2; ++i)
        if (qarmed & (1u << i)) drain_phase(qfull(i), (qpar_bits >> i) & 1, lim);
    }
    __syncwarp();
  } else {
    // =============================================================== consumers ====
    const int cw = warp - 1;                  // consumer warp 0..7
    const int l8 = lane & 7;                  // lane of the row group
    const int grp = cw * 4 + (lane >> 3);     // row group: rows grp + NG jj of every tile
    const int h2 = SMALL_R ? H2 : (p.r >> 1);
    // lanes whose chunk 0 holds rotated dims (r = 8..32: chunks 0..r/8-1, all 8 dims)
    const bool rot_lane = SMALL_R && 8 * l8 < 2 * h2;
    // pair index of chunk-0 dim v, or 16 (the identity factor) on unrotated lanes
    auto pair0 = [&](int v) { return rot_lane ? (8 * l8 + v < h2 ? 8 * l8 + v : 8 * l8 + v - h2) : 16; };
    auto is_a0 = [&](int v) { return !rot_lane || 8 * l8 + v < h2; };  // first half of its pair
    // row factors e^{j row w}: (cos, sin)(row w_pair) for rows grp + 32 jj
    // row factors e^{j row w} of rows 0..127 into shared memory; lane entry u of a row
    // covers chunk-0 dims (2u, 2u + 1): pairs 2q, 2q + 1 with q = qo[u] (dims 2u, 2u + 1
    // of a rotated lane belong to consecutive pairs since r/2 is even), the identity on
    // unrotated lanes
    constexpr int RQ = (SMALL_R && H2 > 0 ? H2 / 2 : 0) + 1;  // entries per row
    int qo[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) qo[u] = rot_lane ? pair0(2 * u) / 2 : RQ - 1;
    if constexpr (SMALL_R && H2 > 0) {
      for (int e = tid - 32; e < kRows * RQ; e += NCT) {
        const int row = e / RQ, q = e - row * RQ;
        float4 f = make_float4(1.0f, 1.0f, 0.0f, 0.0f);
        if (q < RQ - 1) {
          const float2 a = p.cs[row * H2 + 2 * q], b = p.cs[row * H2 + 2 * q + 1];
          f = make_float4(a.x, b.x, a.y, b.y);
        }
        rtab[e] = f;
      }
      consumers_sync<NCT>();
    }
    // (cos, sin) of chunk-0 dims (2u, 2u + 1) of row `row`, packed over the two dims
    auto row_factor = [&](int row, int u, uint64_t& c2, uint64_t& s2) {
      const float4 f = rtab[row * RQ + qo[u]];
      c2 = f32x2_pack(f.x, f.y);
      s2 = f32x2_pack(f.z, f.w);
    };
    uint32_t n = 0;
    int k = 0;
    for (long long g = lo; g < hi; ++k) {
      const long long head = g / Th;
      const int tb = static_cast<int>(g - head * Th);
      const long long gend = min(hi, (head + 1) * Th);
      const int te = tb + static_cast<int>(gend - g);
      g = gend;
      const int slot = k & 1;
      const uint32_t qlap = static_cast<uint32_t>(k >> 1) & 1u;
      bool ok = __all_sync(0xffffffffu, wait_phase(qfull(slot), qlap, abort_flag, lim, 53));
      const int P = ok ? slot_pos[slot] : -1;
      const bool valid = P >= 0 && P < p.Smax;
      const int t1 = min(te, valid ? P / kRows + 1 : 0);
      const uint16_t* sq = reinterpret_cast<const uint16_t*>(slots + slot * SLOT);  // q | k | v
      const float2* sang = reinterpret_cast<const float2*>(slots + slot * SLOT + 6 * D);
      // the lane's query dims, rotated at P and scaled by log2(e)/sqrt(D): z = (q'_i, q'_{i+h2})
      // of each rotated dim's pair; q'_d (and 0) for the others
      float zr[NV], zi[NV];
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int d = lane_dim<D>(l8, v);
        zr[v] = bf16_bits_to_f32(sq[d]) * p.scale_log2;
        zi[v] = 0.0f;
        const bool rot = SMALL_R ? (v < 8 && rot_lane) : d < p.r;
        if (rot && valid) {
          const int i = d < h2 ? d : d - h2;
          const float2 c = SMALL_R ? sang[i] : p.cs[static_cast<long long>(P) * h2 + i];
          const float x1 = bf16_bits_to_f32(sq[i]), x2 = bf16_bits_to_f32(sq[i + h2]);
          zr[v] = (x1 * c.x - x2 * c.y) * p.scale_log2;
          zi[v] = (x2 * c.x + x1 * c.y) * p.scale_log2;
        }
      }
      float m = -INFINITY, l = 0.0f;
      uint64_t o2[NV / 2];  // o over dims (2u, 2u + 1)
#pragma unroll
      for (int u = 0; u < NV / 2; ++u) o2[u] = 0;

      for (int t = tb; ok && t < t1; ++t, ++n) {
        const int s = static_cast<int>(n % S);
        const uint32_t lap = (n / S) & 1u;
        if (!__all_sync(0xffffffffu, wait_phase(full(s), lap, abort_flag, lim, 51))) {
          ok = false;
          break;
        }
        // chunk-0 coefficients of this tile: w = z e^{-j 128 t w}; dim i of a pair takes
        // Re(w e^{-j row w}) = wr c + wi s, dim i + h2 takes Im(...) = wi c - wr s
        uint64_t ca2[4], cb2[4];
        if constexpr (SMALL_R && H2 > 0) {
          float ca[8], cb[8];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float2 f = tf[s * 18 + pair0(v)];
            const float wr = zr[v] * f.x + zi[v] * f.y, wi = zi[v] * f.x - zr[v] * f.y;
            ca[v] = is_a0(v) ? wr : wi;
            cb[v] = is_a0(v) ? wi : -wr;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            ca2[u] = f32x2_pack(ca[2 * u], ca[2 * u + 1]);
            cb2[u] = f32x2_pack(cb[2 * u], cb[2 * u + 1]);
          }
        }
        const uint8_t* kt = smem + (2 * s) * TB;
        const uint8_t* vt = kt + TB;
        const bool whole = t * kRows + kRows - 1 < P;  // every row valid, none is the new token
        if (SMALL_R && whole) {
          // ---- a full tile of cached keys: all loads first, then packed fp32 math
          LaneRow<D> kr[RPG];
#pragma unroll
          for (int jj = 0; jj < RPG; ++jj) kr[jj].load(kt + (grp + NG * jj) * (2 * D), l8);
          float sc[RPG];
#pragma unroll
          for (int jj = 0; jj < RPG; ++jj) {
            uint64_t acc = 0;
#pragma unroll
            for (int u = 0; u < NV / 2; ++u) {
              uint64_t coef;
              if (H2 > 0 && u < 4) {
                uint64_t c2, s2;
                row_factor(grp + NG * jj, u, c2, s2);
                coef = ffma2(cb2[u], s2, fmul2(ca2[u], c2));
              } else
                coef = f32x2_pack(zr[2 * u], zr[2 * u + 1]);
              acc = ffma2(coef, kr[jj].pair(u), acc);
            }
            sc[jj] = f2lo(acc) + f2hi(acc);
          }
          LaneRow<D> vr[RPG];
#pragma unroll
          for (int jj = 0; jj < RPG; ++jj) vr[jj].load(vt + (grp + NG * jj) * (2 * D), l8);
#pragma unroll
          for (int x = 1; x <= 4; x <<= 1)
#pragma unroll
            for (int jj = 0; jj < RPG; ++jj) sc[jj] += __shfl_xor_sync(0xffffffffu, sc[jj], x);
          const float mx = dec_max<RPG>(sc);
          if (mx > m + 8.0f) {
            const float f = ex2_approx(m - mx);
            l *= f;
            const uint64_t f2 = f32x2_pack(f, f);
#pragma unroll
            for (int u = 0; u < NV / 2; ++u) o2[u] = fmul2(o2[u], f2);
            m = mx;
          }
          float pw[RPG];
#pragma unroll
          for (int jj = 0; jj < RPG; ++jj) pw[jj] = ex2_approx(sc[jj] - m);
          l += dec_sum<RPG>(pw);
#pragma unroll
          for (int jj = 0; jj < RPG; ++jj) {
            const uint64_t pp = f32x2_pack(pw[jj], pw[jj]);
#pragma unroll
            for (int u = 0; u < NV / 2; ++u) o2[u] = ffma2(vr[jj].pair(u), pp, o2[u]);
          }
        } else {
        // ---- general tile: masked rows past P, the new token's row, any rotary_dim
        float sc[RPG];
        LaneRow<D> kr[RPG];
#pragma unroll
        for (int jj = 0; jj < RPG; ++jj) {
          const int row = grp + NG * jj;
          const int key = t * kRows + row;
          const bool use = whole || key <= P;
          const uint8_t* src = (!whole && key == P) ? reinterpret_cast<const uint8_t*>(sq + D) : kt + row * (2 * D);
          if (use) kr[jj].load(src, l8);
          float a0 = 0.0f, a1 = 0.0f;
          if (use) {
#pragma unroll
            for (int v = 0; v < NV; ++v) {
              const float x = kr[jj].at(v);
              float coef;
              if constexpr (SMALL_R && H2 > 0) {
                if (v < 8) {
                  uint64_t c2, s2;
                  row_factor(row, v >> 1, c2, s2);
                  const float crv = (v & 1) ? f2hi(c2) : f2lo(c2), srv = (v & 1) ? f2hi(s2) : f2lo(s2);
                  const float cav = (v & 1) ? f2hi(ca2[v >> 1]) : f2lo(ca2[v >> 1]);
                  const float cbv = (v & 1) ? f2hi(cb2[v >> 1]) : f2lo(cb2[v >> 1]);
                  coef = fmaf(cbv, srv, cav * crv);
                } else {
                  coef = zr[v];
                }
              } else if constexpr (SMALL_R) {
                coef = zr[v];
              } else {
                const int d = lane_dim<D>(l8, v);
                coef = zr[v];
                if (d < p.r) {
                  const int i = d < h2 ? d : d - h2;
                  const float2 c = p.cs[static_cast<long long>(key) * h2 + i];
                  coef = d < h2 ? zr[v] * c.x + zi[v] * c.y : zi[v] * c.x - zr[v] * c.y;
                }
              }
              if (v & 1)
                a1 = fmaf(coef, x, a1);
              else
                a0 = fmaf(coef, x, a0);
            }
          }
          sc[jj] = a0 + a1;
        }
#pragma unroll
        for (int jj = 0; jj < RPG; ++jj) {
          sc[jj] += __shfl_xor_sync(0xffffffffu, sc[jj], 1);
          sc[jj] += __shfl_xor_sync(0xffffffffu, sc[jj], 2);
          sc[jj] += __shfl_xor_sync(0xffffffffu, sc[jj], 4);
          if (!whole && t * kRows + grp + NG * jj > P) sc[jj] = -INFINITY;
        }
        // online softmax of the group's rows (log2 units), lazy rescale beyond 2^8
        const float mx = dec_max<RPG>(sc);
        if (mx > m + 8.0f) {
          const float f = ex2_approx(m - mx);
          l *= f;
          const uint64_t f2 = f32x2_pack(f, f);
#pragma unroll
          for (int u = 0; u < NV / 2; ++u) o2[u] = fmul2(o2[u], f2);
          m = mx;
        }
        float pw[RPG];
#pragma unroll
        for (int jj = 0; jj < RPG; ++jj) pw[jj] = sc[jj] == -INFINITY ? 0.0f : ex2_approx(sc[jj] - m);
        l += dec_sum<RPG>(pw);
#pragma unroll
        for (int jj = 0; jj < RPG; ++jj) {
          const int row = grp + NG * jj;
          const int key = t * kRows + row;
          if (whole || key <= P) {
            const bool is_new = !whole && key == P;
            const uint8_t* src = is_new ? reinterpret_cast<const uint8_t*>(sq + 2 * D) : vt + row * (2 * D);
            LaneRow<D> vr;
            vr.load(src, l8);
            const uint64_t pp = f32x2_pack(pw[jj], pw[jj]);
#pragma unroll
            for (int u = 0; u < NV / 2; ++u) o2[u] = ffma2(vr.pair(u), pp, o2[u]);
            if (is_new) {  // append the new token's raw key and value to the cache
              const long long crow = (head * p.Smax + P) * D;
              uint8_t* kd = reinterpret_cast<uint8_t*>(p.k_cache + crow);
              uint8_t* vd = reinterpret_cast<uint8_t*>(p.v_cache + crow);
              const uint8_t* ks = reinterpret_cast<const uint8_t*>(sq + D);
              *reinterpret_cast<uint4*>(kd + 16 * l8) = *reinterpret_cast<const uint4*>(ks + 16 * l8);
              *reinterpret_cast<uint4*>(vd + 16 * l8) = *reinterpret_cast<const uint4*>(src + 16 * l8);
              if constexpr (D == 128) {
                *reinterpret_cast<uint4*>(kd + 128 + 16 * l8) = *reinterpret_cast<const uint4*>(ks + 128 + 16 * l8);
                *reinterpret_cast<uint4*>(vd + 128 + 16 * l8) = *reinterpret_cast<const uint4*>(src + 128 + 16 * l8);
              }
              if constexpr (D == 96) {
                *reinterpret_cast<uint2*>(kd + 128 + 8 * l8) = *reinterpret_cast<const uint2*>(ks + 128 + 8 * l8);
                *reinterpret_cast<uint2*>(vd + 128 + 8 * l8) = *reinterpret_cast<const uint2*>(src + 128 + 8 * l8);
              }
            }
          }
        }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));  // this warp is done with stage s
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty(slot));  // and with the item slot

      // ---- merge the row groups: the warp's 4 groups by shuffles, then the CW warps
#pragma unroll
      for (int x = 8; x <= 16; x <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, x), lo2 = __shfl_xor_sync(0xffffffffu, l, x);
        const float M = fmaxf(m, mo);
        const float fs = m == -INFINITY ? 0.0f : ex2_approx(m - M);
        const float fo = mo == -INFINITY ? 0.0f : ex2_approx(mo - M);
        l = l * fs + lo2 * fo;
#pragma unroll
        for (int u = 0; u < NV / 2; ++u) {
          const float a = f2lo(o2[u]), b = f2hi(o2[u]);
          o2[u] = f32x2_pack(a * fs + __shfl_xor_sync(0xffffffffu, a, x) * fo,
                             b * fs + __shfl_xor_sync(0xffffffffu, b, x) * fo);
        }
        m = M;
      }
      float* rb = red + ((k & 1) * CW + cw) * (D + 2);
      if (lane < 8) {
#pragma unroll
        for (int v = 0; v < NV; ++v) rb[lane_dim<D>(l8, v)] = (v & 1) ? f2hi(o2[v >> 1]) : f2lo(o2[v >> 1]);
      }
      if (lane == 0) {
        rb[D] = m;
        rb[D + 1] = l;
      }
      const bool stop = consumers_sync_or<NCT>(!ok || *abort_flag != 0);
      if (stop) break;
      const int c = tid - 32;
      float M = -INFINITY, acc = 0.0f, L = 0.0f;
      if (c < D) {
        const float* r0 = red + (k & 1) * CW * (D + 2);
#pragma unroll
        for (int w = 0; w < CW; ++w) M = fmaxf(M, r0[w * (D + 2) + D]);
#pragma unroll
        for (int w = 0; w < CW; ++w) {
          const float mw = r0[w * (D + 2) + D];
          const float f = mw == -INFINITY ? 0.0f : ex2_approx(mw - M);
          acc = fmaf(r0[w * (D + 2) + c], f, acc);
          L = fmaf(r0[w * (D + 2) + D + 1], f, L);
        }
      }
      // the CTAs whose tile ranges hold part of this head (the same for every thread)
      const long long cfirst = dec_cta_of(head * Th, N, G);
      const int runs = static_cast<int>(dec_cta_of(head * Th + Th - 1, N, G) - cfirst) + 1;
      if (runs == 1) {  // the whole head is this item
        if (c < D) dec_write_out<D>(p, head, c, acc, M, L);
      } else if (runs <= p.runs_per_head) {
        // partial state to this run's slot; the last of the head's CTAs to arrive merges
        float* hp = p.part + head * p.runs_per_head * (D + 2);
        if (c < D) {
          float* pp = hp + (cta - cfirst) * (D + 2);
          pp[c] = acc;
          if (c == 0) {
            pp[D] = M;
            pp[D + 1] = L;
          }
          __threadfence();
        }
        consumers_sync<NCT>();
        if (c == 0) {
          const bool last = atomicAdd(p.counters + head, 1) == runs - 1;
          if (last) p.counters[head] = 0;  // every run has arrived: ready for the next call
          *last_flag = last ? 1 : 0;
        }
        consumers_sync<NCT>();
        if (*last_flag && c < D) {
          __threadfence();
          float Mh = -INFINITY;
          for (int r = 0; r < runs; ++r) Mh = fmaxf(Mh, __ldcg(hp + r * (D + 2) + D));
          float a = 0.0f, Lh = 0.0f;
          for (int r = 0; r < runs; ++r) {
            const float mr = __ldcg(hp + r * (D + 2) + D);
            if (mr != -INFINITY) {
              const float f = ex2_approx(mr - Mh);
              a = fmaf(__ldcg(hp + r * (D + 2) + c), f, a);
              Lh = fmaf(__ldcg(hp + r * (D + 2) + D + 1), f, Lh);
            }
          }
          dec_write_out<D>(p, head, c, a, Mh, Lh);
        }
      } else if (c == 0) {
        record_error(kErrBadInput, 1);
      }
    }
  }
  __syncthreads();
}

}  // namespace neox
