// attn_ws.cuh -- the persistent, warp-specialised causal rotary attention kernel.
//
// One CTA per SM (persistent).  A work unit is (b, h, t): the two 128-row query tiles
// 2t and 2t+1 of one head, which share one stream of 128-key K/V blocks.  Units are
// taken longest first (descending t), dealt to the CTAs in a snake order.
//
// Roles (384 threads):
//   warp 0        TMA producer: Q tiles once per unit, then K_j / V_j into rings
//   warp 1        tcgen05 issuer (one lane) and TMEM owner
//   warps 2-3     rotary transform: rotate-half of Q (per unit) and of K_j (per block)
//                 in shared memory (rotary_dim 16/24/32: the rotated chunks as fp16 in
//                 place; otherwise hi in place, lo to the side tiles).  A unit's K_0 is
//                 loaded and rotated before its query tiles: K_0's ring slot frees a few
//                 blocks before the previous unit releases the query buffers, so only the
//                 query load and rotation remain between two units (the producer also
//                 prefetches the next unit's query tiles into L2)
//   warps 4-7     softmax + lazy correction + epilogue of query tile 0
//   warps 8-11    the same for query tile 1
//
// TMEM (512 columns): S/P of tile 0 at [0,128), S/P of tile 1 at [128,256),
// O of tile 0 at [256, 256+D), O of tile 1 at [384, 384+D).  P (bf16) overwrites the
// first 64 columns of its S block; the PV MMA reads it from TMEM as operand A.
//
// MMA order per block step j (for each tile tau with work):
//   PV_tau(j-1): O_tau (+)= P_tau V_{j-1}, after softmax tau published P_tau(j-1)
//   S_tau(j)   : S_tau  = Q'_tau K'_j^T   (commit -> s_full[tau])
// so the softmax of one tile overlaps the MMAs of the other.  Because a commit tracks
// every earlier MMA of the issuing thread, s_full[tau] for block j also means that
// PV_tau(j-1) has landed: the softmax may rescale O_tau in place right then.
//
// Causality: tile q visits KV blocks 0..q only, and masks keys > row on block q.
//
// Code size matters here: every role shares the SM's instruction caches, so the
// rotation variant is a template parameter (one path per kernel) and each role has a
// single copy of its inner loop.
#pragma once

#include "attn_common.cuh"

namespace neox {

constexpr int kWsThreads = 384;
constexpr int kRegsControl = 136;  // producer, MMA and rotary warps (warpgroup 0)
constexpr int kRegsSoftmax = 184;  // the two softmax warpgroups
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kWsThreads * 168, "register split exceeds the launch");
constexpr int kMaxRing = 4;

// Descriptor words for the 64-byte-swizzled tiles: the high word is the same for every
// operand (SBO = 512 B, version 1, layout SW64); the low word is (address >> 4) plus
// the leading-byte-offset field (16 B for K-major, 8 KB between 32-column blocks for V).
constexpr uint32_t kDescHi = (512u >> 4) | (1u << 14) | (4u << 29);
__device__ __forceinline__ uint32_t desc_lo_k(uint32_t saddr) { return (saddr >> 4) | (1u << 16); }
__device__ __forceinline__ uint32_t desc_lo_v(uint32_t saddr) { return (saddr >> 4) | ((kBlkBytes >> 4) << 16); }
__device__ __forceinline__ uint64_t desc_of(uint32_t lo) { return (static_cast<uint64_t>(kDescHi) << 32) | lo; }
// Offset (in 16-byte units) of K chunk kc (16 columns) inside a column-blocked tile.
__host__ __device__ constexpr uint32_t kchunk_off(int kc) { return (kc >> 1) * (kBlkBytes >> 4) + (kc & 1) * 2; }

// How the rotary warps rotate a row (fixed per kernel instance):
//   kRotNone: no rotary dims.  kRotR16 / kRotR32: r = 16 / 32, groups of 8 pairs with the
//   next tile's table entries loaded ahead.  kRotR24: r = 24, the 24-dim prefix in
//   registers, table loaded ahead.  kRotGroups: r % 16 == 0 and r > 32, groups of 8 pairs
//   with double-buffered table loads inside the tile.  kRotScalar: any other even r.
enum : int { kRotNone = 0, kRotR16 = 1, kRotR24 = 2, kRotR32 = 3, kRotGroups = 4, kRotScalar = 5 };
__host__ __device__ constexpr int rot_kind(int r) {
  return r == 0 ? kRotNone : r == 16 ? kRotR16 : r == 24 ? kRotR24 : r == 32 ? kRotR32 : (r % 16 == 0 ? kRotGroups : kRotScalar);
}
// float4 table entries per row loaded ahead of a tile's data.
__host__ __device__ constexpr int rot_ahead(int rk) { return rk == kRotR16 ? 4 : rk == kRotR24 ? 6 : rk == kRotR32 ? 8 : 0; }
// In-kernel rotation with fp16 operands for the rotated chunks (rotary_dim 16, 24, 32): the
// first rot_f16_chunks 16-column chunks of Q' and K' are fp16, the S MMA has no lo products.
// The other rotary_dims (and pre-rotated operands) keep the bf16 hi/lo split.
__host__ __device__ constexpr bool rot_f16(int rk, bool pre) {
  return !pre && (rk == kRotR16 || rk == kRotR24 || rk == kRotR32);
}
__host__ __device__ constexpr int rot_f16_chunks(int rk) { return rk == kRotR16 ? 1 : 2; }

// Shared-memory carve-up, identical on host and device: the two query tiles (each followed
// by its side tile), the K ring (each slot a tile and its side tile), the V ring, then the
// barrier block.  Offsets are closed forms of the slot index (no arrays, so no local memory).
struct WsLayout {
  int tb, sb;    // bytes of a D-column tile and of a side tile
  int nk, nv;
  __host__ __device__ int q_raw(int t) const { return t * (tb + sb); }
  __host__ __device__ int q_side(int t) const { return t * (tb + sb) + tb; }
  __host__ __device__ int k_raw(int s) const { return (2 + s) * (tb + sb); }
  __host__ __device__ int k_side(int s) const { return (2 + s) * (tb + sb) + tb; }
  __host__ __device__ int v(int s) const { return (2 + nk) * (tb + sb) + s * tb; }
  __host__ __device__ int bars() const { return (2 + nk) * (tb + sb) + nv * tb; }
  __host__ __device__ int total() const { return bars() + 64 * 8 + 16 + 1024; }  // + TMEM slot, flag, alignment slack
};
__host__ __device__ inline WsLayout ws_layout(int D, int side_cols, int NK, int NV) {
  return WsLayout{tile_bytes(D), tile_bytes(side_cols), NK, NV};
}

// Barrier indices inside the barrier block.
enum : int {
  BAR_Q_FULL = 0, BAR_Q_READY = 1, BAR_Q_EMPTY = 2, BAR_DRAIN = 3,
  BAR_S_FULL = 4,   // +tau
  BAR_P_FULL = 6,   // +tau
  BAR_O_FINAL = 8,  // +tau
  BAR_K_FULL = 10,  // +slot (4)
  BAR_K_READY = 14, // +slot
  BAR_K_EMPTY = 18, // +slot
  BAR_V_FULL = 22,  // +slot (4)
  BAR_V_EMPTY = 26, // +slot
  BAR_Q_READY1 = 30,  // query tile 1 rotated (BAR_Q_READY: tile 0)
  BAR_COUNT = 31
};

struct Unit {
  int b, h, t;
  int n0, n1;    // KV blocks of tile 0 / tile 1 (n1 = 0: no tile 1)
  int nkv;       // max(n0, n1)
};

__device__ __forceinline__ Unit decode_unit(int k, int B, int H, int S) {
  const int T = (S + 255) / 256;
  const int bh_count = B * H;
  Unit u;
  u.t = T - 1 - k / bh_count;
  const int bh = k % bh_count;
  u.b = bh / H;
  u.h = bh % H;
  u.n0 = 2 * u.t + 1;
  u.n1 = ((2 * u.t + 1) * kRows < S) ? 2 * u.t + 2 : 0;
  u.nkv = u.n1 > u.n0 ? u.n1 : u.n0;
  return u;
}

// Units in the order of decreasing work (t descending, then head), dealt to the CTAs in
// a snake: round r covers units [rG, rG + G); even rounds go to CTAs 0..G-1, odd rounds
// to CTAs G-1..0, which balances the longest-first list about as well as a greedy
// dynamic scheduler would, with no atomics (so concurrent launches cannot interfere).
__device__ __forceinline__ int snake_unit(int round, int cta, int G) {
  return round * G + ((round & 1) ? (G - 1 - cta) : cta);
}

// PRE: the operands come pre-rotated (the pre-rotation pass: hi and lo of q' and k' in the
// copy that tmap_rot views as [B, S, 4H, D], the lo slot in the side-tile layout); the
// query tiles and K tiles are then loaded with their side tiles by TMA and nothing is
// rotated here (rotary_dim % 16 == 0, or 24).
//
// ALIBI: no rotation; the scores get the linear position bias -m_h (i - j) of the ALiBi
// scheme instead (m_h the head's slope: 2^(-8k/n), k = 1..n, for the n = largest power of
// two <= H heads, then 2^(-8k/(2n)) for odd k for the rest).
template <int D, int RK, bool PRE, bool ALIBI = false>
__global__ void __launch_bounds__(kWsThreads, 1)
    attn_fwd_ws_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_rot,
                       const AttnParams p) {
  static_assert(!PRE || RK != kRotScalar, "pre-rotated operands need rotary_dim % 16 == 0 or rotary_dim == 24");
  static_assert(!ALIBI || (RK == kRotNone && !PRE), "the ALiBi bias replaces the rotary embedding");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NK = p.nk, NV = p.nv;
  const WsLayout L = ws_layout(D, p.side_cols, NK, NV);
  // barrier block: 64 mbarriers, then the TMEM address slot and the abort flag (32-bit
  // shared addresses throughout)
  const uint32_t bar0 = smem_u32(smem) + static_cast<uint32_t>(L.bars());
  const uint32_t tmem_slot_a = bar0 + 64 * 8, abort_a = tmem_slot_a + 4;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t lim = p.wait_limit_ns;

  // ---------------------------------------------------------------- setup ----
  if (tid == 0) {
    mbar_init(bar(BAR_Q_FULL), 1);
    mbar_init(bar(BAR_Q_READY), 64);
    mbar_init(bar(BAR_Q_READY1), 64);
    mbar_init(bar(BAR_Q_EMPTY), 1);
    mbar_init(bar(BAR_DRAIN), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(BAR_S_FULL + t), 1);
      mbar_init(bar(BAR_P_FULL + t), 128);
      mbar_init(bar(BAR_O_FINAL + t), 1);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(BAR_K_FULL + s), 1);
      mbar_init(bar(BAR_K_READY + s), 64);
      mbar_init(bar(BAR_K_EMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(BAR_V_FULL + s), 1);
      mbar_init(bar(BAR_V_EMPTY + s), 1);
    }
    flag_st(abort_a, 0);
    fence_barrier_init();
    tma_prefetch_map(&tmap);
    if (PRE) tma_prefetch_map(&tmap_rot);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot_a, 512);
    tmem_relinquish();
  }
  // side tiles start at zero; columns >= r are never written again
  if (RK != kRotNone) {
    const int sb = tile_bytes(p.side_cols);
    for (int i = tid * 16; i < sb; i += kWsThreads * 16) {
      for (int t = 0; t < 2; ++t) *reinterpret_cast<uint4*>(smem + L.q_side(t) + i) = make_uint4(0, 0, 0, 0);
      for (int s = 0; s < NK; ++s) *reinterpret_cast<uint4*>(smem + L.k_side(s) + i) = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = static_cast<uint32_t>(flag_ld(tmem_slot_a));
  // register split: the softmax warpgroups hold a whole 128-column S row per thread
  // (launch: 384 x 168 = 128 x 136 + 256 x 184)

  const int G = gridDim.x;
  if (warp < 4) {
   regs_release<kRegsControl>();
   if (warp == 0) {
    // ============================================================ producer ====
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      int ks = 0, vs = 0;        // next K / V ring slot
      uint32_t kph = 0, vph = 0;  // ring lap parity of that slot
      uint32_t u_local = 0;
      // for the abort path: which ring slots have a load armed, and its phase parity
      uint32_t k_armed = 0, k_par = 0, v_armed = 0, v_par = 0;
      int last_q_par = -1;
      bool ok = true;
      auto load_k = [&](const Unit& u, int j) {
        const int s = ks;
        const uint32_t par = kph;
        if (!wait_phase_s(bar(BAR_K_EMPTY + s), par ^ 1, abort_a, lim, 11)) return false;
        mbar_arrive_expect_tx(bar(BAR_K_FULL + s), tile_bytes(D) + (PRE ? tile_bytes(p.side_cols) : 0));
        k_armed |= 1u << s;
        k_par = (k_par & ~(1u << s)) | (par << s);
        if (PRE) {  // hi into the tile, lo into its side tile
          for (int cb = 0; cb < D / kBlkCols; ++cb)
            tma_load_4d_hint(smem_u32(smem + L.k_raw(s) + cb * kBlkBytes), &tmap_rot, bar(BAR_K_FULL + s),
                             cb * kBlkCols, 4 * u.h + 2, j * kRows, u.b, pol_kv);
          for (int cb = 0; cb < p.side_cols / kBlkCols; ++cb)
            tma_load_4d_hint(smem_u32(smem + L.k_side(s) + cb * kBlkBytes), &tmap_rot, bar(BAR_K_FULL + s),
                             cb * kBlkCols, 4 * u.h + 3, j * kRows, u.b, pol_kv);
        } else {
          for (int cb = 0; cb < D / kBlkCols; ++cb)
            tma_load_4d_hint(smem_u32(smem + L.k_raw(s) + cb * kBlkBytes), &tmap, bar(BAR_K_FULL + s), cb * kBlkCols,
                             3 * u.h + 1, j * kRows, u.b, pol_kv);
        }
        if (++ks == NK) { ks = 0; kph ^= 1; }
        return true;
      };
      for (int rd = 0; rd * G < p.num_units && ok; ++rd) {
        const int k = snake_unit(rd, blockIdx.x, G);
        if (k >= p.num_units) continue;
        const Unit u = decode_unit(k, p.B, p.H, p.S);
        // K_0 first: its ring slot frees a few blocks before the previous unit's last S
        // MMA releases the query buffers, so it is loaded (and rotated) off the boundary
        if (!load_k(u, 0)) { ok = false; break; }
        if (!wait_phase_s(bar(BAR_Q_EMPTY), (u_local & 1) ^ 1, abort_a, lim, 10)) { ok = false; break; }
        const int nq = u.n1 > 0 ? 2 : 1;
        mbar_arrive_expect_tx(bar(BAR_Q_FULL), (tile_bytes(D) + (PRE ? tile_bytes(p.side_cols) : 0)) * nq);
        last_q_par = u_local & 1;
        for (int t = 0; t < nq; ++t) {
          if (PRE) {
            for (int cb = 0; cb < D / kBlkCols; ++cb)
              tma_load_4d_hint(smem_u32(smem + L.q_raw(t) + cb * kBlkBytes), &tmap_rot, bar(BAR_Q_FULL),
                               cb * kBlkCols, 4 * u.h + 0, (2 * u.t + t) * kRows, u.b, pol_q);
            for (int cb = 0; cb < p.side_cols / kBlkCols; ++cb)
              tma_load_4d_hint(smem_u32(smem + L.q_side(t) + cb * kBlkBytes), &tmap_rot, bar(BAR_Q_FULL),
                               cb * kBlkCols, 4 * u.h + 1, (2 * u.t + t) * kRows, u.b, pol_q);
          } else {
            for (int cb = 0; cb < D / kBlkCols; ++cb)
              tma_load_4d_hint(smem_u32(smem + L.q_raw(t) + cb * kBlkBytes), &tmap, bar(BAR_Q_FULL), cb * kBlkCols,
                               3 * u.h + 0, (2 * u.t + t) * kRows, u.b, pol_q);
          }
        }
        // the next unit's query tiles into L2 now, so their load at the next boundary is short
        {
          const int kn = snake_unit(rd + 1, blockIdx.x, G);
          if (kn < p.num_units) {
            const Unit un = decode_unit(kn, p.B, p.H, p.S);
            for (int t = 0; t < (un.n1 > 0 ? 2 : 1); ++t)
              for (int cb = 0; cb < D / kBlkCols; ++cb) {
                if (PRE)
                  tma_prefetch_l2_4d(&tmap_rot, cb * kBlkCols, 4 * un.h + 0, (2 * un.t + t) * kRows, un.b);
                else
                  tma_prefetch_l2_4d(&tmap, cb * kBlkCols, 3 * un.h + 0, (2 * un.t + t) * kRows, un.b);
              }
          }
        }
        // K_j before V_{j-1}: the order in which the MMA warp consumes them
        for (int j = 1; j <= u.nkv && ok; ++j) {
          if (j < u.nkv && !load_k(u, j)) { ok = false; break; }
          {
            const int s = vs;
            const uint32_t par = vph;
            if (!wait_phase_s(bar(BAR_V_EMPTY + s), par ^ 1, abort_a, lim, 12)) { ok = false; break; }
            mbar_arrive_expect_tx(bar(BAR_V_FULL + s), tile_bytes(D));
            v_armed |= 1u << s;
            v_par = (v_par & ~(1u << s)) | (par << s);
            for (int cb = 0; cb < D / kBlkCols; ++cb)
              tma_load_4d_hint(smem_u32(smem + L.v(s) + cb * kBlkBytes), &tmap, bar(BAR_V_FULL + s), cb * kBlkCols,
                               3 * u.h + 2, (j - 1) * kRows, u.b, pol_kv);
            if (++vs == NV) { vs = 0; vph ^= 1; }
          }
        }
        ++u_local;
      }
      if (!ok || flag_ld(abort_a)) {
        // let every load this thread armed land before the CTA's shared memory goes away
        if (last_q_par >= 0) drain_phase(bar(BAR_Q_FULL), last_q_par, lim);
        for (int s = 0; s < NK; ++s)
          if (k_armed & (1u << s)) drain_phase(bar(BAR_K_FULL + s), (k_par >> s) & 1, lim);
        for (int s = 0; s < NV; ++s)
          if (v_armed & (1u << s)) drain_phase(bar(BAR_V_FULL + s), (v_par >> s) & 1, lim);
      }
    }
   } else if (warp == 1) {
    // ============================================================ MMA issuer ====
    // The whole warp walks the schedule, so its control flow and descriptors stay
    // warp-uniform (a single-lane issue loop runs markedly slower once the softmax warps
    // on the same SM sub-partition are busy); one elected lane starts each tensor-core
    // operation.  Ring slots and query buffers are released by commits, i.e. as soon as
    // the MMAs reading them have completed.
    {
      const uint32_t lead = elect_lane();
      const uint32_t idesc_s = idesc_bf16_f32(128, 128, false);
      const uint32_t idesc_s16 = idesc_f16_f32(128, 128, false);  // fp16 chunks (rot_f16)
      const uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      // Every operand buffer sits at a fixed shared address for the whole kernel, so each
      // descriptor is a base below plus a constant: the issue loop is adds and MMAs only.
      const uint64_t dq[2] = {desc_of(desc_lo_k(smem_u32(smem + L.q_raw(0)))),
                              desc_of(desc_lo_k(smem_u32(smem + L.q_raw(1))))};
      // query descriptors of every 16-column chunk, both tiles (fixed for the kernel)
      uint64_t qd[2][D / 16];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int kc = 0; kc < D / 16; ++kc) qd[t][kc] = dq[t] + kchunk_off(kc);
      const uint64_t dqs[2] = {desc_of(desc_lo_k(smem_u32(smem + L.q_side(0)))),
                               desc_of(desc_lo_k(smem_u32(smem + L.q_side(1))))};
      const uint64_t dk0 = desc_of(desc_lo_k(smem_u32(smem + L.k_raw(0))));
      const uint64_t dks0 = desc_of(desc_lo_k(smem_u32(smem + L.k_side(0))));
      const uint64_t dv0 = desc_of(desc_lo_v(smem_u32(smem + L.v(0))));
      const uint32_t kstep = static_cast<uint32_t>(tile_bytes(D) + tile_bytes(p.side_cols)) >> 4;
      const uint32_t vstep = static_cast<uint32_t>(tile_bytes(D)) >> 4;
      int kslot = 0, vslot = 0;
      uint32_t kph = 0, vph = 0, u_local = 0;
      uint32_t p_cnt[2] = {0, 0};
      uint32_t q1_cnt = 0;  // units with a query tile 1 (a ragged last block may have none)
      const int nside = p.r16 / 16;  // 16-column chunks of lo products (<= 8)
      bool ok = true, issued = false;
      auto wait_all = [&](int b, uint32_t par, unsigned int site) {
        return __all_sync(0xffffffffu, wait_phase_s(bar(b), par, abort_a, lim, site));
      };
      for (int rd = 0; rd * G < p.num_units && ok; ++rd) {
        const int k = snake_unit(rd, blockIdx.x, G);
        if (k >= p.num_units) continue;
        const Unit u = decode_unit(k, p.B, p.H, p.S);
        for (int j = 0; j <= u.nkv && ok; ++j) {
          const int ks = kslot, vs = vslot;
          if (j < u.nkv && !wait_all(BAR_K_READY + ks, kph, 31)) { ok = false; break; }
          if (j >= 1 && !wait_all(BAR_V_FULL + vs, vph, 32)) { ok = false; break; }
          // this step's K and V descriptors, computed once for both tiles
          const uint64_t dk = dk0 + ks * kstep, dks = dks0 + ks * kstep, dv = dv0 + vs * vstep;
          uint64_t kd[D / 16], vd[kRows / 16];
#pragma unroll
          for (int kc = 0; kc < D / 16; ++kc) kd[kc] = dk + kchunk_off(kc);
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk) vd[kk] = dv + kk * 64;
#pragma unroll
          for (int tau = 0; tau < 2; ++tau) {
            const int n = tau == 0 ? u.n0 : u.n1;
            if (n == 0) continue;
            const uint32_t tS = tmem + tau * 128, tO = tmem + 256 + tau * 128;
            if (j >= 1 && j <= n) {
              if (!wait_all(BAR_P_FULL + tau, p_cnt[tau] & 1, 33)) { ok = false; break; }
              ++p_cnt[tau];
              tc_fence_after_sync();
              mma_ts_x8_l(lead, tO, tS, vd, idesc_pv, j > 1);
              issued = true;
              if (j == n) tc_commit_l(lead, bar(BAR_O_FINAL + tau));
            }
            if (j < n) {
              if (j == 0) {
                const uint32_t par = tau == 0 ? (u_local & 1) : (q1_cnt++ & 1);
                if (!wait_all(tau == 0 ? BAR_Q_READY : BAR_Q_READY1, par, 30)) { ok = false; break; }
                tc_fence_after_sync();
              }
              const uint64_t q = dq[tau], qs = dqs[tau];
              if constexpr (rot_f16(RK, PRE)) {
                // the rotated chunks as fp16 x fp16, the rest bf16 x bf16, one accumulator
                constexpr int NF = rot_f16_chunks(RK);
                mma_ss_l(lead, tS, qd[tau][0], kd[0], idesc_s16, 0);
#pragma unroll
                for (int kc = 1; kc < D / 16; ++kc)
                  mma_ss_acc_l(lead, tS, qd[tau][kc], kd[kc], kc < NF ? idesc_s16 : idesc_s);
              } else {
              mma_ss_l(lead, tS, qd[tau][0], kd[0], idesc_s, 0);
#pragma unroll
              for (int kc = 1; kc < D / 16; ++kc) mma_ss_acc_l(lead, tS, qd[tau][kc], kd[kc], idesc_s);
              if constexpr (RK == kRotR24) {
                // cross terms: dims 0..15 as q_lo.k_hi and q_hi.k_lo, dims 16..23 packed into
                // one chunk of the two side tiles ([lo | hi] . [hi | lo])
                mma_ss_acc_l(lead, tS, qs, dk, idesc_s);
                mma_ss_acc_l(lead, tS, q, dks, idesc_s);
                mma_ss_acc_l(lead, tS, qs + kchunk_off(1), dks + kchunk_off(1), idesc_s);
              } else {
                // a plain runtime loop: the same issue written as an unrolled loop of 8 with a
                // `kc < nside` guard produced wrong scores for nside >= 2 on the GPU
                for (int kc = 0; kc < nside; ++kc) {
                  mma_ss_acc_l(lead, tS, qs + kchunk_off(kc), dk + kchunk_off(kc), idesc_s);
                  mma_ss_acc_l(lead, tS, q + kchunk_off(kc), dks + kchunk_off(kc), idesc_s);
                }
              }
              }
              issued = true;
              tc_commit_l(lead, bar(BAR_S_FULL + tau));
            }
          }
          if (!ok) break;
          if (j < u.nkv) {
            tc_commit_l(lead, bar(BAR_K_EMPTY + ks));
            if (++kslot == NK) { kslot = 0; kph ^= 1; }
          }
          if (j >= 1) {
            tc_commit_l(lead, bar(BAR_V_EMPTY + vs));
            if (++vslot == NV) { vslot = 0; vph ^= 1; }
          }
          // the unit's last S MMAs are issued: its query buffers may be refilled
          if (j == u.nkv - 1) tc_commit_l(lead, bar(BAR_Q_EMPTY));
        }
        ++u_local;
      }
      if (issued && __any_sync(0xffffffffu, !ok || flag_ld(abort_a))) {
        tc_commit_l(lead, bar(BAR_DRAIN));
        drain_phase(bar(BAR_DRAIN), 0, lim);
      }
      __syncwarp();
    }
   } else {
    // ======================================================= rotary transform ====
    // Per unit the tiles arrive as: K_0, query tile 0, query tile 1 (if any), K_1, K_2, ...
    // (the producer's order).  One loop over that list, one rotation call site.
    const int tt = tid - 64;  // 0..63: rows tt and tt + 64 of every tile
    const int h = p.r >> 1;
    constexpr int AH = PRE ? 0 : rot_ahead(RK);
    float4 ta0[8], ta1[8];  // table entries of rows tt / tt + 64, loaded one tile ahead
    auto pos_of = [&](int blk, int row) -> int64_t {
      const int64_t pos = static_cast<int64_t>(blk) * kRows + row;
      return pos < p.S ? pos : -1;
    };
    auto load_ahead = [&](int blk) {
      if (AH > 0) {
        cs_load_n<AH>(ta0, p.cs, h, 0, pos_of(blk, tt));
        cs_load_n<AH>(ta1, p.cs, h, 0, pos_of(blk, tt + 64));
      }
    };
    int kslot = 0;
    uint32_t kph = 0, u_local = 0;
    bool ok = true;
    if (AH > 0) load_ahead(0);  // every unit starts with K_0
    for (int rd = 0; rd * G < p.num_units && ok; ++rd) {
      const int k = snake_unit(rd, blockIdx.x, G);
      if (k >= p.num_units) continue;
      const Unit u = decode_unit(k, p.B, p.H, p.S);
      const int nq = u.n1 > 0 ? 2 : 1;
      // item it: 0 -> K_0, 1..nq -> query tile it-1, then K_(it - nq)
      auto blk_of = [&](int it) { return it == 0 ? 0 : it <= nq ? 2 * u.t + it - 1 : it - nq; };
#pragma unroll 1
      for (int it = 0; it < nq + u.nkv; ++it) {
        const bool isq = it >= 1 && it <= nq;
        const int qt = it - 1;  // query tile (when isq)
        const int s = kslot;
        const int blk = blk_of(it);  // 128-row block of the sequence
        if (isq ? (qt == 0 && !wait_phase_s(bar(BAR_Q_FULL), u_local & 1, abort_a, lim, 20))
                : !wait_phase_s(bar(BAR_K_FULL + s), kph, abort_a, lim, 21)) {
          ok = false;
          break;
        }
        uint8_t* tile = smem + (isq ? L.q_raw(qt) : L.k_raw(s));
        uint8_t* side = smem + (isq ? L.q_side(qt) : L.k_side(s));
        if (PRE) {
          // operands arrive rotated: only hand them on
        } else if (RK == kRotR24) {  // fp16 chunks 0 and 1 (see rot_f16)
          const bool in0 = rotate_row_r24_f16(tile, tt, ta0);
          const bool in1 = rotate_row_r24_f16(tile, tt + 64, ta1);
          if (!(in0 && in1)) record_error(kErrRange, 23);
        } else if (RK == kRotR16 || RK == kRotR32) {  // fp16 chunk(s) 0 (and 1)
          bool in = true;
#pragma unroll
          for (int g = 0; g < AH / 4; ++g) {
            in &= rotate_group8_f16(tile, tt, 8 * g, h, ta0 + 4 * g);
            in &= rotate_group8_f16(tile, tt + 64, 8 * g, h, ta1 + 4 * g);
          }
          if (!in) record_error(kErrRange, 23);
        } else if (RK == kRotGroups) {
          rotate_two_rows_groups(tile, side, tt, tt + 64, pos_of(blk, tt), pos_of(blk, tt + 64), p.cs, h, ta0, ta1);
        } else if (RK == kRotScalar) {
          rotate_row(tile, side, tt, pos_of(blk, tt), p.cs, p.r);
          rotate_row(tile, side, tt + 64, pos_of(blk, tt + 64), p.cs, p.r);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(isq ? (qt == 0 ? BAR_Q_READY : BAR_Q_READY1) : BAR_K_READY + s));
        if (!isq && ++kslot == NK) {
          kslot = 0;
          kph ^= 1;
        }
        // table entries of the next tile in this list, or of the next unit's K_0
        if (AH > 0) load_ahead(it + 1 < nq + u.nkv ? blk_of(it + 1) : 0);
      }
      ++u_local;
    }
   }
  } else {
    regs_acquire<kRegsSoftmax>();
    // ========================================== softmax / correction / epilogue ====
    const int tau = (warp - 4) >> 2;          // query tile of this warpgroup
    const int row = tid - 128 * (tau + 1);     // 0..127: this thread's row / TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + tau * 128 + lane_off, tO = tmem + 256 + tau * 128 + lane_off;
    const float sl2 = p.scale_log2;
    uint32_t s_use = 0, o_use = 0;
    for (int rd = 0; rd * G < p.num_units; ++rd) {
      const int k = snake_unit(rd, blockIdx.x, G);
      if (k >= p.num_units) continue;
      const Unit u = decode_unit(k, p.B, p.H, p.S);
      const int n = tau == 0 ? u.n0 : u.n1;
      if (n == 0) continue;
      const int qt = 2 * u.t + tau;
      float m_used = -INFINITY, l_run = 0.0f;
      // ALiBi: the head's slope in log2 units, and the bias of column 0 of block 0 for this
      // thread's row (the bias of key k is bh * (k - row), at most 0 on the causal side)
      float bh = 0.0f, row0 = 0.0f;
      if constexpr (ALIBI) {
        int n2 = 1;
        while (n2 * 2 <= p.H) n2 *= 2;
        const double e = u.h < n2 ? -8.0 * (u.h + 1) / n2 : -8.0 * (2 * (u.h - n2) + 1) / (2.0 * n2);
        bh = static_cast<float>(exp2(e) * 1.4426950408889634);
        row0 = -bh * static_cast<float>(qt * kRows + row);
      }
      // every exit decision is warp-uniform: the TMEM loads and stores below are
      // warp-collective, so no lane may leave while the others go on
      bool ok = true;
#pragma unroll 1
      for (int j = 0; j < n; ++j) {
        if (!__all_sync(0xffffffffu, wait_phase_s(bar(BAR_S_FULL + tau), s_use & 1, abort_a, lim, 40))) {
          ok = false;
          break;
        }
        ++s_use;
        tc_fence_after_sync();
        uint32_t sr[128];
        float mx;
        if constexpr (ALIBI) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr + c * 32);
          tmem_wait_ld();
          // biased scores in log2 units: s * log2(e)/sqrt(D) + bh * (128 j + c - row)
          const uint64_t sc2 = f32x2_pack(sl2, sl2), bh2 = f32x2_pack(bh, bh);
          const float off = fmaf(bh, static_cast<float>(j * kRows), row0);
          const uint64_t off2 = f32x2_pack(off, off);
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const uint64_t b = ffma2(f32x2_pack(static_cast<float>(2 * c), static_cast<float>(2 * c + 1)), bh2, off2);
            const uint64_t v = ffma2(f32x2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc2, b);
            float v0, v1;
            f32x2_unpack(v, v0, v1);
            sr[2 * c] = __float_as_uint(v0);
            sr[2 * c + 1] = __float_as_uint(v1);
          }
          if (j == qt) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c > row) sr[c] = __float_as_uint(-INFINITY);
          }
          float mc[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint32_t* v = sr + 16 * g;
            float m = fmax3f(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
            for (int q = 3; q < 15; q += 2) m = fmax3f(m, __uint_as_float(v[q]), __uint_as_float(v[q + 1]));
            mc[g] = fmaxf(m, __uint_as_float(v[15]));
          }
          mx = fmaxf(fmax3f(mc[0], mc[1], mc[2]), fmax3f(fmax3f(mc[3], mc[4], mc[5]), mc[6], mc[7]));
        } else if (j != qt) {
          // below the diagonal: the loads return each 32-column chunk's max as well
          float mq[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) mq[c] = tmem_ld32_max(tS + c * 32, sr + c * 32);
          tmem_wait_ld();
          mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr + c * 32);
          tmem_wait_ld();
          // the diagonal block: keys > row get -inf (the block's keys are 128*qt + c, its
          // rows 128*qt + row), then the row max in eight chains of 3-input max
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > row) sr[c] = __float_as_uint(-INFINITY);
          float mc[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint32_t* v = sr + 16 * g;
            float m = fmax3f(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
            for (int q = 3; q < 15; q += 2) m = fmax3f(m, __uint_as_float(v[q]), __uint_as_float(v[q + 1]));
            mc[g] = fmaxf(m, __uint_as_float(v[15]));
          }
          mx = fmaxf(fmax3f(mc[0], mc[1], mc[2]), fmax3f(fmax3f(mc[3], mc[4], mc[5]), mc[6], mc[7]));
        }
        const float mx_s = ALIBI ? mx : mx * sl2;  // the biased scores are in log2 units already
        float m_new = m_used;
        bool rescale = false;
        if (j == 0) {
          m_new = mx_s;
        } else if (mx_s > m_used + 8.0f) {
          m_new = mx_s;
          rescale = true;
        }
        const float alpha = rescale ? ex2_approx(m_used - m_new) : 1.0f;
        // p = 2^(s * log2(e)/sqrt(D) - m): packed fp32 FMA, MUFU exp2, four packed partial sums
        const float sc = ALIBI ? 1.0f : sl2;
        const uint64_t sc2 = f32x2_pack(sc, sc), nm2 = f32x2_pack(-m_new, -m_new);
        uint64_t acc[4] = {0, 0, 0, 0};
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const uint64_t t = ffma2(f32x2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc2, nm2);
          float t0, t1;
          f32x2_unpack(t, t0, t1);
          const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
          acc[c & 3] = fadd2(acc[c & 3], f32x2_pack(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        acc[0] = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
        float rs0, rs1;
        f32x2_unpack(acc[0], rs0, rs1);
        const float rowsum = rs0 + rs1;
        l_run = l_run * alpha + rowsum;
        m_used = m_new;
        // lazy correction: O holds sum over blocks < j (landed, see s_full); rescale it only
        // when some row's running max grew by more than 2^8
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tO + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tmem_st32(tO + c0, o);
          }
        }
        tmem_st32(tS, pk);
        tmem_st32(tS + 32, pk + 32);
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(bar(BAR_P_FULL + tau));
      }
      if (!ok) break;
      if (!__all_sync(0xffffffffu, wait_phase_s(bar(BAR_O_FINAL + tau), o_use & 1, abort_a, lim, 41))) break;
      ++o_use;
      tc_fence_after_sync();
      const int qrow = qt * kRows + row;
      const float inv_l = 1.0f / l_run;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tO + c0, o);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q)
          pk[q] = pack_bf16x2(__uint_as_float(o[2 * q]) * inv_l, __uint_as_float(o[2 * q + 1]) * inv_l);
        if (qrow < p.S) {  // 32-byte stores: a row is 2D bytes, 32-byte aligned
          uint16_t* dst = p.out + ((static_cast<int64_t>(u.b) * p.S + qrow) * p.H + u.h) * D + c0;
          st_global_v8(dst, pk);
          st_global_v8(dst + 16, pk + 8);
        }
      }
      if (qrow < p.S)
        p.lse[(static_cast<int64_t>(u.b) * p.H + u.h) * p.S + qrow] = (m_used + log2f(l_run)) * 0.69314718055994530942f;
      tc_fence_before_sync();
    }
  }

  // ------------------------------------------------------------- teardown ----
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

constexpr int kSmemLimit = 227 * 1024;

// Ring depths: the deepest (K, V) pair that fits next to the two query tiles, preferring
// the per-head-dim defaults (at D = 128 a K ring of 3 once there are no side tiles).
inline void pick_rings(int D, int side_cols, int* nk, int* nv) {
  const bool side = side_cols > 0;
  const int pref_k = D == 64 ? 4 : D == 96 ? 3 : (side ? 2 : 3);  // D = 96: (4, 3) measured slower
  const int pref_v = D == 64 ? 4 : 2;
  const int cand[][2] = {{pref_k, pref_v}, {3, 2}, {2, 2}, {2, 1}, {1, 1}};
  for (const auto& c : cand) {
    if (ws_layout(D, side_cols, c[0], c[1]).total() <= kSmemLimit) {
      *nk = c[0];
      *nv = c[1];
      return;
    }
  }
  *nk = *nv = 1;
}

template <int D, int RK, bool PRE, bool ALIBI = false>
int launch_ws_impl(const CUtensorMap& map, const CUtensorMap& map_rot, AttnParams p, int num_sms, cudaStream_t stream,
                   int* last_err) {
  if (rot_f16(RK, PRE)) p.side_cols = 0;  // fp16 rotated chunks: no lo side tiles
  pick_rings(D, p.side_cols, &p.nk, &p.nv);
  const WsLayout L = ws_layout(D, p.side_cols, p.nk, p.nv);
  auto kern = attn_fwd_ws_kernel<D, RK, PRE, ALIBI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total());
  if (e != cudaSuccess) { *last_err = static_cast<int>(e); return -4; }
  const int T = (p.S + 255) / 256;
  p.num_units = p.B * p.H * T;
  const int grid = p.num_units < num_sms ? p.num_units : num_sms;
  kern<<<grid, kWsThreads, L.total(), stream>>>(map, map_rot, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) { *last_err = static_cast<int>(e); return -4; }
  return 0;
}

// The ALiBi variant (rotary_dim 0 in p).
template <int D>
int launch_attn_ws_alibi(const CUtensorMap& map, const AttnParams& p, int num_sms, cudaStream_t stream,
                         int* last_err) {
  return launch_ws_impl<D, kRotNone, false, true>(map, map, p, num_sms, stream, last_err);
}

// pre_rotated: map_rot views the rotated copy written by the pre-rotation pass (the caller
// checks rotary_dim % 16 == 0 or rotary_dim == 24, rotary_dim > 0); otherwise map_rot is
// not read.
template <int D>
int launch_attn_ws(const CUtensorMap& map, const CUtensorMap& map_rot, bool pre_rotated, const AttnParams& p,
                   int num_sms, cudaStream_t stream, int* last_err) {
  if (pre_rotated) {
    switch (rot_kind(p.r)) {
      case kRotR16: return launch_ws_impl<D, kRotR16, true>(map, map_rot, p, num_sms, stream, last_err);
      case kRotR24: return launch_ws_impl<D, kRotR24, true>(map, map_rot, p, num_sms, stream, last_err);
      case kRotR32: return launch_ws_impl<D, kRotR32, true>(map, map_rot, p, num_sms, stream, last_err);
      case kRotGroups: return launch_ws_impl<D, kRotGroups, true>(map, map_rot, p, num_sms, stream, last_err);
      default: return -1;
    }
  }
  switch (rot_kind(p.r)) {
    case kRotNone: return launch_ws_impl<D, kRotNone, false>(map, map_rot, p, num_sms, stream, last_err);
    case kRotR16: return launch_ws_impl<D, kRotR16, false>(map, map_rot, p, num_sms, stream, last_err);
    case kRotR24: return launch_ws_impl<D, kRotR24, false>(map, map_rot, p, num_sms, stream, last_err);
    case kRotR32: return launch_ws_impl<D, kRotR32, false>(map, map_rot, p, num_sms, stream, last_err);
    case kRotGroups: return launch_ws_impl<D, kRotGroups, false>(map, map_rot, p, num_sms, stream, last_err);
    default: return launch_ws_impl<D, kRotScalar, false>(map, map_rot, p, num_sms, stream, last_err);
  }
}

}  // namespace neox
