// qkv_proj.cuh -- the fused query_key_value projection that produces the packed qkv, on the
// tcgen05 tensor cores, with the bias add and (optionally) the NeoX rotary embedding of the
// query and key slots in the epilogue.
//
// "GPT-NeoX on FasterTransformer" guide, "从 HuggingFace 检查点部署": the weight is stored
// [hidden, num_heads, 3, head_hidden], so with the token rows x[M = B*S, K = hidden] and the
// weight read as w[K, N = 3*H*D] the product x * w (+ bias[N]) is, row by row, the packed
// [B, S, H, 3, D] qkv the attention reads; section "模型配置（config.ini）" gives the
// 20B shape (64 heads x 96, hidden 6144, rotary_embedding 24).
//
// Kernel: persistent, one CTA per SM, 192 threads in three roles.
//   warp 0      TMA producer: per 64-wide K step, a 128 x 64 tile of x (K-major) and a
//               64 x NT tile of w (N contiguous, so MN-major for the MMA), both 128-byte
//               swizzled, into a ring of ST stages.
//   warp 1      MMA issuer: four 128 x NT x 16 tcgen05.mma per stage into one of two TMEM
//               accumulators (columns 0 and 256), so the epilogue of tile i overlaps the
//               main loop of tile i + 1.
//   warps 2..5  epilogue, one TMEM lane quadrant (32 token rows) each, half a tile at a
//               time: fp32 accumulator + bias -> bf16 into a staging slab of 32 x 32 blocks
//               (64-byte swizzle); then, when rotary_dim > 0, each query/key slot's rotary
//               pairs (d, d + r/2) are rotated in fp32 from those bf16 values and rounded
//               again (the rotation the model applies to its bf16 q and k); then TMA stores.
// NT is a whole number of D-wide slots (192 for D = 96, 256 for D = 64 and 128) and so is
// NT/2, so every slot's rotary pairs lie inside one half-tile.  Staging half a tile (6 or
// 8 KB a warp) leaves the shared memory to a deeper operand ring: 5 stages of 40 KB at
// NT = 192, 4 of 48 KB at NT = 256.  Tiles run m-fastest: the CTAs working at one time
// share a few NT-wide column blocks of w and all of x, which stays in L2.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "attn_common.cuh"
#include "ptx.cuh"

namespace neox {

struct ProjParams {
  const uint16_t* bias;  // bf16 [N] or nullptr
  const float2* cs;      // cos/sin table [>= S][r/2] (r > 0 only)
  int M, N, K;           // token rows (B*S), 3*H*D, hidden
  int S, D, r;           // sequence length (positions restart every S rows), head dim, rotary_dim
  int num_m, num_tiles;  // 128-row tiles, all tiles
  uint64_t wait_limit_ns;
};

constexpr int kProjThreads = 192;

__host__ __device__ constexpr int proj_tile_n(int D) { return D == 96 ? 192 : 256; }
__host__ __device__ constexpr int proj_stages(int NT) { return NT == 192 ? 5 : 4; }
__host__ __device__ constexpr uint32_t proj_stage_bytes(int NT) { return 128u * 128u + static_cast<uint32_t>(NT) * 128u; }
// one warp's staging: 32 rows x NT/2 columns of bf16, as NT/64 blocks of 32 x 32 (2 KB)
__host__ __device__ constexpr uint32_t proj_slab_bytes(int NT) { return 32u * static_cast<uint32_t>(NT); }
// ring, four staging slabs, barrier block (256 bytes), 1 KB alignment slack
__host__ __device__ constexpr uint32_t proj_smem_bytes(int NT) {
  return proj_stages(NT) * proj_stage_bytes(NT) + 4u * proj_slab_bytes(NT) + 256u + 1024u;
}

// Byte address of element (row, col) of a staging slab: 32-column blocks of 32 rows x 64
// bytes, the 16-byte chunks of a row swizzled by bits 1..2 of the row (the TMA 64-byte
// swizzle), which keeps eight consecutive rows' chunk stores on distinct banks.
__device__ __forceinline__ uint32_t slab_chunk(uint32_t slab, int row, int col) {
  return slab + static_cast<uint32_t>((col >> 5) * 2048 + row * 64 + ((((col >> 3) & 3) ^ ((row >> 1) & 3)) << 4));
}
__device__ __forceinline__ uint32_t slab_addr(uint32_t slab, int row, int col) {
  return slab_chunk(slab, row, col) + static_cast<uint32_t>((col & 7) << 1);
}
__device__ __forceinline__ uint16_t ld_shared_u16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_u16(uint32_t a, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ void prefetch_l1(const void* ptr) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)));
}

// One slot's rotary pairs (c0 + i, c0 + i + rh), i < rh, of row `row` of a staging slab, W
// pairs per step (W = 8: 16-byte accesses, needs rh % 8 == 0; W = 4: 8-byte, rh % 4 == 0;
// W = 1: any rh).  cs = the row's (cos, sin) entries; the slab holds bf16 values in place.
template <int W>
__device__ __forceinline__ void rotate_slot(uint32_t slab, int row, int c0, int rh, const float2* cs) {
#pragma unroll 1
  for (int i = 0; i < rh; i += W) {
    const uint32_t aa = slab_addr(slab, row, c0 + i), ab = slab_addr(slab, row, c0 + i + rh);
    uint32_t xa[W > 1 ? W / 2 : 1], xb[W > 1 ? W / 2 : 1];
    float2 t[W];
    if constexpr (W == 8) {
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(xa[0]), "=r"(xa[1]), "=r"(xa[2]), "=r"(xa[3]) : "r"(aa) : "memory");
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(xb[0]), "=r"(xb[1]), "=r"(xb[2]), "=r"(xb[3]) : "r"(ab) : "memory");
    } else if constexpr (W == 4) {
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(xa[0]), "=r"(xa[1]) : "r"(aa) : "memory");
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(xb[0]), "=r"(xb[1]) : "r"(ab) : "memory");
    } else {
      xa[0] = ld_shared_u16(aa);
      xb[0] = ld_shared_u16(ab);
    }
    if constexpr (W > 1) {
#pragma unroll
      for (int e = 0; e < W; e += 2) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(cs + i + e));
        t[e] = make_float2(v.x, v.y);
        t[e + 1] = make_float2(v.z, v.w);
      }
    } else {
      t[0] = __ldg(cs + i);
    }
    uint32_t ya[W > 1 ? W / 2 : 1], yb[W > 1 ? W / 2 : 1];
#pragma unroll
    for (int e = 0; e < W; ++e) {
      const uint32_t wa = W > 1 ? xa[e >> 1] : xa[0], wb = W > 1 ? xb[e >> 1] : xb[0];
      const int sh = (W > 1 && (e & 1)) ? 16 : 0;
      const float x = __uint_as_float(((wa >> sh) & 0xFFFFu) << 16), z = __uint_as_float(((wb >> sh) & 0xFFFFu) << 16);
      const uint32_t ra = f32_to_bf16_bits(fmaf(x, t[e].x, -z * t[e].y));
      const uint32_t rb = f32_to_bf16_bits(fmaf(z, t[e].x, x * t[e].y));
      if (W == 1) {
        ya[0] = ra;
        yb[0] = rb;
      } else if (e & 1) {
        ya[e >> 1] |= ra << 16;
        yb[e >> 1] |= rb << 16;
      } else {
        ya[e >> 1] = ra;
        yb[e >> 1] = rb;
      }
    }
    if constexpr (W == 8) {
      st_shared_v4(aa, ya[0], ya[1], ya[2], ya[3]);
      st_shared_v4(ab, yb[0], yb[1], yb[2], yb[3]);
    } else if constexpr (W == 4) {
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(aa), "r"(ya[0]), "r"(ya[1]) : "memory");
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(ab), "r"(yb[0]), "r"(yb[1]) : "memory");
    } else {
      st_shared_u16(aa, static_cast<uint16_t>(ya[0]));
      st_shared_u16(ab, static_cast<uint16_t>(yb[0]));
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kProjThreads, 1)
    qkv_proj_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                    const __grid_constant__ CUtensorMap map_out, const ProjParams p) {
  static_assert(NT == 192 || NT == 256, "tile width");
  constexpr int ST = proj_stages(NT);
  constexpr uint32_t A_BYTES = 128u * 128u, STAGE = proj_stage_bytes(NT), SLAB = proj_slab_bytes(NT);
  constexpr int NB = NT / 64;  // 64-column blocks of w per stage; 32-column slab blocks per half-tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t slab0 = s0 + ST * STAGE;
  const uint32_t bar0 = slab0 + 4 * SLAB;
  // barriers: full[ST], empty[ST], acc_full[2], acc_empty[2], drain; then the TMEM address
  // slot and the abort flag
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (ST + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * ST + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * ST + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * ST + 4);
  const uint32_t tmem_slot_a = bar0 + 128, abort_a = tmem_slot_a + 4;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t lim = p.wait_limit_ns;
  const int KT = (p.K + 63) / 64;

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);
    }
    mbar_init(drain_bar, 1);
    flag_st(abort_a, 0);
    fence_barrier_init();
    tma_prefetch_map(&map_x);
    tma_prefetch_map(&map_w);
    tma_prefetch_map(&map_out);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot_a, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = static_cast<uint32_t>(flag_ld(tmem_slot_a));

  if (warp == 0) {
    // ============================================================ producer ====
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      uint32_t armed = 0, armed_par = 0;  // stages with a load issued, and that load's parity
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int m0 = (tile % p.num_m) * 128, n0 = (tile / p.num_m) * NT;
        for (int kt = 0; kt < KT; ++kt) {
          if (!wait_phase_s(empty(st), ph ^ 1, abort_a, lim, 60)) {
            ok = false;
            break;
          }
          const uint32_t a = s0 + st * STAGE;
          mbar_arrive_expect_tx(full(st), STAGE);
          tma_load_2d(a, &map_x, full(st), kt * 64, m0);
#pragma unroll
          for (int j = 0; j < NB; ++j) tma_load_2d(a + A_BYTES + j * 8192u, &map_w, full(st), n0 + 64 * j, kt * 64);
          armed |= 1u << st;
          armed_par = (armed_par & ~(1u << st)) | (ph << st);
          if (++st == ST) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      // loads still landing (only after an abort: otherwise the MMA consumed them all)
      for (int s = 0; s < ST; ++s)
        if ((armed >> s) & 1) drain_phase(full(s), (armed_par >> s) & 1, lim);
    }
  } else if (warp == 1) {
    // ================================================================= MMA ====
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NT, true);
      int st = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
        const int b = it & 1;
        if (!wait_phase_s(acc_empty(b), ((it >> 1) & 1) ^ 1, abort_a, lim, 61)) break;
        tc_fence_after_sync();
        const uint32_t d = tmem + static_cast<uint32_t>(b) * 256u;
        for (int kt = 0; kt < KT; ++kt) {
          if (!wait_phase_s(full(st), ph, abort_a, lim, 62)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a = s0 + st * STAGE, bb = a + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(d, sdesc_sw128(a + 32u * kk, 16, 1024), sdesc_sw128(bb + 2048u * kk, 8192, 1024), idesc,
                   (kt | kk) != 0);
          tc_commit(empty(st));
          if (++st == ST) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(acc_full(b));
      }
      // every MMA this thread issued has completed before the TMEM is freed
      tc_commit(drain_bar);
      drain_phase(drain_bar, 0, lim);
    }
  } else {
    // ============================================================ epilogue ====
    const int q = warp & 3;  // TMEM lane quadrant = rows 32q .. 32q + 31 of the tile
    const uint32_t slab = slab0 + q * SLAB;
    const int row = 32 * q + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
      const int b = it & 1;
      const int m0 = (tile % p.num_m) * 128, n0 = (tile / p.num_m) * NT;
      // this row's cos/sin entries, pulled toward L1 while the main loop runs
      const float2* cs = p.cs + static_cast<int64_t>((m0 + row) % p.S) * (p.r >> 1);
      for (int o = 0; o < 4 * (p.r >> 1); o += 64) prefetch_l1(reinterpret_cast<const char*>(cs) + 2 * o);
      if (!__all_sync(0xffffffffu, wait_phase_s(acc_full(b), (it >> 1) & 1, abort_a, lim, 63))) break;
      tc_fence_after_sync();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b) * 256u;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int h0 = half * (NT / 2);  // first column of this half-tile
        // the slab's previous stores have read it
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        // two 32-column chunks per TMEM round trip (their bias words fetched meanwhile)
#pragma unroll 1
        for (int c2 = 0; c2 < NB; c2 += 2) {
          const int nc = NB - c2 < 2 ? NB - c2 : 2;
          uint32_t v[2][32];
          uint4 bw[2][4];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (k < nc) tmem_ld32(taddr + static_cast<uint32_t>(h0 + 32 * (c2 + k)), v[k]);
            const int n = n0 + h0 + 32 * (c2 + k);
            const bool has_bias = k < nc && p.bias != nullptr && n < p.N;
#pragma unroll
            for (int u = 0; u < 4; ++u)
              bw[k][u] = has_bias ? __ldg(reinterpret_cast<const uint4*>(p.bias + n) + u) : make_uint4(0, 0, 0, 0);
          }
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (k >= nc) break;
            const int c = c2 + k;
            uint32_t pk[16];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t ws[4] = {bw[k][u].x, bw[k][u].y, bw[k][u].z, bw[k][u].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int q2 = 4 * u + e;  // packed pair index: columns 2 q2, 2 q2 + 1
                pk[q2] = pack_bf16x2(__uint_as_float(v[k][2 * q2]) + __uint_as_float(ws[e] << 16),
                                     __uint_as_float(v[k][2 * q2 + 1]) + __uint_as_float(ws[e] & 0xFFFF0000u));
              }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              st_shared_v4(slab_chunk(slab, lane, 32 * c + 8 * u), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                           pk[4 * u + 3]);
          }
        }
        if (half == 1) {
          // the accumulator is read: hand it back to the MMA warp
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty(b));
        }
        if (p.r > 0) {
          // rotate-half on the bf16 query/key values: pair (i, i + r/2) of each slot, angle
          // pos * inv_freq[i], pos = the token's place in its sequence
          const int rh = p.r >> 1;
#pragma unroll 1
          for (int c0 = 0; c0 < NT / 2; c0 += p.D) {
            const int g = (n0 + h0 + c0) / p.D;  // global slot index h*3 + {0: q, 1: k, 2: v}
            if (n0 + h0 + c0 >= p.N || g % 3 == 2) continue;
            if ((rh & 7) == 0)
              rotate_slot<8>(slab, lane, c0, rh, cs);
            else if ((rh & 3) == 0)
              rotate_slot<4>(slab, lane, c0, rh, cs);
            else
              rotate_slot<1>(slab, lane, c0, rh, cs);
          }
        }
        // generic-proxy writes of the slab -> visible to the TMA store
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && m0 + 32 * q < p.M) {
#pragma unroll
          for (int j = 0; j < NB; ++j)
            if (n0 + h0 + 32 * j < p.N) tma_store_2d(&map_out, slab + j * 2048u, n0 + h0 + 32 * j, m0 + 32 * q);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int NT>
int launch_qkv_proj_impl(const CUtensorMap& mx, const CUtensorMap& mw, const CUtensorMap& mo, const ProjParams& p,
                         int num_sms, cudaStream_t stream, int* last_err) {
  auto kern = qkv_proj_kernel<NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, proj_smem_bytes(NT));
  if (e != cudaSuccess) {
    *last_err = static_cast<int>(e);
    return -4;
  }
  const int grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
  kern<<<grid, kProjThreads, proj_smem_bytes(NT), stream>>>(mx, mw, mo, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    *last_err = static_cast<int>(e);
    return -4;
  }
  return 0;
}

// x map: [M, K] box {64, 128} and w map: [K, N] box {64, 64}, both with the 128-byte
// swizzle; out map: [M, N] box {32, 32} with the 64-byte swizzle.  All bf16.
inline int launch_qkv_proj(const CUtensorMap& mx, const CUtensorMap& mw, const CUtensorMap& mo, const ProjParams& p,
                           int num_sms, cudaStream_t stream, int* last_err) {
  if (proj_tile_n(p.D) == 192) return launch_qkv_proj_impl<192>(mx, mw, mo, p, num_sms, stream, last_err);
  return launch_qkv_proj_impl<256>(mx, mw, mo, p, num_sms, stream, last_err);
}

}  // namespace neox
