// attn_bwd.cuh -- backward of the causal NeoX-rotary attention: dq, dk, dv of the packed
// qkv from dout, given the forward's out and lse.
//
// GPT-NeoX is a training library ("gpt-neox - 模型与框架" page: the framework trains the
// 20B model and moved its attention to the exact, tiled Flash Attention, section
// "问题二：注意力计算太慢"), so the attention's gradient is the training-side twin of the
// forward.  With s_ij = q'_i.k'_j / sqrt(D) (keys j <= i), p_ij = exp(s_ij - lse_i):
//   dv_j  = sum_i p_ij dout_i                 dp_ij = dout_i . v_j
//   ds_ij = p_ij (dp_ij - delta_i),  delta_i = dout_i . out_i
//   dq'_i = sum_j ds_ij k'_j / sqrt(D)         dk'_j = sum_i ds_ij q'_i / sqrt(D)
//   dq_i = R(i)^T dq'_i,  dk_j = R(j)^T dk'_j  (the rotation back by -theta).
// Three kernels on the caller's stream:
//   attn_bwd_prep_kernel   the rotated q', k' (bf16, rounded once) into a scratch copy of
//                          qkv, delta_i (fp32) and a zeroed fp32 dq' accumulator;
//   attn_bwd_kernel        persistent, one CTA per SM taking work items (key block j,
//                          head) in a fixed order from a counter: K'_j, V_j stay in shared
//                          memory while query blocks i >= j stream through (the next
//                          item's K'/V, and its first Q'/dO, load under the epilogue); per block
//                          five tcgen05 MMAs (S = Q'K'^T and dP = dO V^T into TMEM, then
//                          dV += P^T dO and dK += dS^T Q' accumulating in TMEM over i, and
//                          dQ'_i = dS K' added to the fp32 accumulator by D/32 TMA tensor
//                          reductions of 128 x 32 boxes, staged, with two query-side
//                          buffers, in block i's own (then free) Q'/dO buffer and reduced
//                          while block i+1 computes its P/dS);
//                          at the end dk (rotated back) and dv go out as bf16 tiles by
//                          TMA tensor stores;
//   attn_bwd_dq_kernel     rotates the accumulated dq' back and writes dq as bf16.
// P and dS enter the MMAs as bf16 (fp32 accumulation), as do the rotated q', k' (rounded
// once, no hi/lo split); the transposed operands P^T, dS^T, dO and Q' are read through
// MN-major descriptors of the same swizzled tiles.
#pragma once

#include "attn_common.cuh"

namespace neox {

struct BwdParams {
  const uint16_t* qkv;   // bf16 [B, S, H, 3, D]
  const uint16_t* out;   // bf16 [B, S, H, D]  (the forward's)
  const float* lse;      // fp32 [B, H, S]     (the forward's, natural log)
  const uint16_t* dout;  // bf16 [B, S, H, D]
  uint16_t* dqkv;        // bf16 [B, S, H, 3, D]
  uint16_t* qkv_rot;     // bf16 [B, S, H, 3, D]  scratch: rotated q', k' in slots 0, 1 (slot 2 unused)
  float* dq_acc;         // fp32 [B, S, H, D]  scratch: dq' before the rotation back
  float* delta;          // fp32 [B, H, S]     scratch
  const float2* cs;      // cos/sin table [>= S rows][r/2]
  int B, S, H, r, nblk;
  int heads_per_group;   // work-item order: groups of heads whose Q'/dO tiles fit in L2 together
  float scale_log2;      // log2(e) / sqrt(D)
  float scale;           // 1 / sqrt(D)
  uint64_t wait_limit_ns;
};

constexpr float kLog2e = 1.4426950408889634f;

// Programmatic dependent launch between the three kernels of a call: a kernel lets the next
// one launch early (its CTAs set up while this grid drains), and the next one waits for
// this grid's completion and memory before it reads anything this grid wrote.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Work counter of the main kernel (items past the grid's first), zeroed by the prep kernel
// of the same call (calls on one device are serialised by the shared scratch anyway).
__device__ unsigned int g_bwd_next;

// Per row (one warp per row): slots 0, 1 of qkv_rot = R(s) q, R(s) k in bf16 (the
// rotation rounded once, as the MMAs take it), delta = dout . out (fp32), and dq_acc
// zeroed.  16-byte loads and stores; the row's q and k wait in shared memory (fp32) so
// that a rotated dim can read its pair partner.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p) {
  constexpr int C8 = D / 8;  // 16-byte chunks per D-vector
  __shared__ float xbuf[8][2 * D];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0) g_bwd_next = 0u;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + w;  // [b][s][h]
  if (row >= static_cast<long long>(p.B) * p.S * p.H) return;
  const long long s = (row / p.H) % p.S;
  const int h2 = p.r >> 1;
  float* x = xbuf[w];
  const uint16_t* src = p.qkv + row * 3 * D;
  uint16_t* dst = p.qkv_rot + row * 3 * D;
  for (int c = lane; c < 2 * C8; c += 32) {  // q chunks then k chunks
    const uint4 v = *reinterpret_cast<const uint4*>(src + 8 * c);
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[8 * c + 2 * k] = __uint_as_float(wd[k] << 16);
      x[8 * c + 2 * k + 1] = __uint_as_float(wd[k] & 0xFFFF0000u);
    }
  }
  __syncwarp();
  for (int c = lane; c < 2 * C8; c += 32) {
    const int base = c < C8 ? 0 : D;  // this chunk's vector (q or k) in x
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int d = 8 * c + e - base;
      float v = x[base + d];
      if (d < p.r) {  // y_i = x_i c - x_{i+h} s,  y_{i+h} = x_{i+h} c + x_i s
        const bool first = d < h2;
        const int i = first ? d : d - h2;
        const float2 cs = p.cs[s * h2 + i];
        const float partner = x[base + (first ? d + h2 : d - h2)];
        v = fmaf(v, cs.x, (first ? -partner : partner) * cs.y);
      }
      y[e] = v;
    }
    *reinterpret_cast<uint4*>(dst + 8 * c) = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                                        pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
  }
  const uint16_t* o = p.out + row * D;
  const uint16_t* g = p.dout + row * D;
  float acc = 0.0f;
  for (int c = lane; c < C8; c += 32) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + 8 * c), gg = *reinterpret_cast<const uint4*>(g + 8 * c);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wg[4] = {gg.x, gg.y, gg.z, gg.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = fmaf(__uint_as_float(wa[k] << 16), __uint_as_float(wg[k] << 16), acc);
      acc = fmaf(__uint_as_float(wa[k] & 0xFFFF0000u), __uint_as_float(wg[k] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
  float4* dq = reinterpret_cast<float4*>(p.dq_acc + row * D);
  for (int c = lane; c < D / 4; c += 32) dq[c] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (lane == 0) {
    const long long h = row % p.H, b = row / (static_cast<long long>(p.H) * p.S);
    p.delta[(b * p.H + h) * p.S + s] = acc;
  }
}

// dq = R(s)^T dq' (bf16) into slot 0 of dqkv, one warp per row:
//   dq_i = dq'_i c + dq'_{i+h} s,  dq_{i+h} = dq'_{i+h} c - dq'_i s  (i < h = r/2).
// When r/2 is a multiple of 4 no 4-dim chunk straddles i = h or i = r, and lane l handles
// chunk l with 16-byte loads (the partner chunk too) and an 8-byte store; otherwise lane
// l handles dims l, l + 32, ...
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(const BwdParams p) {
  pdl_wait_prior();  // the main kernel's dq' reductions
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);  // [b][s][h]
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<long long>(p.B) * p.S * p.H) return;
  const long long s = (row / p.H) % p.S;
  const float* src = p.dq_acc + row * D;
  const int h2 = p.r >> 1;
  uint16_t* dst = p.dqkv + row * 3 * D;
  if ((h2 & 3) == 0) {
    for (int c = lane; c < D / 4; c += 32) {
      const int d = 4 * c;
      float4 v = *reinterpret_cast<const float4*>(src + d);
      if (d < p.r) {
        const bool first = d < h2;
        const float4 w = *reinterpret_cast<const float4*>(src + (first ? d + h2 : d - h2));
        const float sg = first ? 1.0f : -1.0f;
        const float2* cs = p.cs + s * h2 + (first ? d : d - h2);
        const float2 c0 = cs[0], c1 = cs[1], c2 = cs[2], c3 = cs[3];
        v = make_float4(fmaf(v.x, c0.x, sg * w.x * c0.y), fmaf(v.y, c1.x, sg * w.y * c1.y),
                        fmaf(v.z, c2.x, sg * w.z * c2.y), fmaf(v.w, c3.x, sg * w.w * c3.y));
      }
      *reinterpret_cast<uint2*>(dst + d) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
    return;
  }
  for (int d = lane; d < D; d += 32) {
    float v = src[d];
    if (d < h2) {
      const float2 c = p.cs[s * h2 + d];
      v = fmaf(v, c.x, src[d + h2] * c.y);
    } else if (d < p.r) {
      const float2 c = p.cs[s * h2 + (d - h2)];
      v = fmaf(v, c.x, -src[d - h2] * c.y);
    }
    dst[d] = f32_to_bf16_bits(v);
  }
}

// kind::f16 instruction descriptor with the A major-ness as well (bit 15: 1 = MN-major).
__host__ __device__ constexpr uint32_t idesc_bwd(int M, int N, bool a_mn, bool b_mn) {
  return idesc_bf16_f32(M, N, b_mn) | ((a_mn ? 1u : 0u) << 15);
}

// Query-side buffers (Q'_i and dO_i tile pairs): two for D <= 96, so the next block's
// tiles load (TMA) while the current block's MMAs run; one for D = 128, where
// a second pair does not fit next to K', V, P and dS.
__host__ __device__ constexpr int bwd_qbufs(int D) { return D == 128 ? 1 : 2; }
// smem: K'_j, V_j, then per buffer Q'_i and dO_i, then P_i and dS_i [128][128] tiles
// (1 KB aligned), barriers, the TMEM address and the abort flag.
// dq' staging for the tensor reductions: D/32 boxes of [128 rows][32 floats] (16 KB each,
// the TMA 128-byte swizzle: 16-byte chunk k of row r at chunk k ^ (r & 7)) in the block's
// Q'/dO buffer (two buffers) or in the P/dS tiles (one buffer), both free once the block's
// dV/dK/dQ MMAs have completed.
__host__ __device__ constexpr int bwd_stage_bytes(int D) { return D / 32 * 16384; }
__host__ __device__ constexpr int bwd_stage_extra(int D) {
  return bwd_stage_bytes(D) > 2 * tile_bytes(128) ? bwd_stage_bytes(D) - 2 * tile_bytes(128) : 0;
}
// Columns of dk' that the epilogue stages in fp32 for the rotation: the 32-column blocks
// holding rotated dims (the rest goes from TMEM straight into the bf16 dk tile).
__host__ __device__ constexpr int bwd_rot_cols(int r) { return (r + 31) / 32 * 32; }
// Where that staging goes: beside the dk and dv tiles in the P/dS area when it fits there,
// else in the query-side tiles (whose next loads then wait for the end of the epilogue).
template <int D>
__host__ __device__ constexpr bool bwd_stage_in_qbuf(int r) {
  return bwd_qbufs(D) == 1 || bwd_rot_cols(r) * kRows * 4 > 2 * tile_bytes(128) - 2 * tile_bytes(D);
}
__host__ __device__ constexpr int bwd_smem_bytes(int D) {
  return 1024 + (2 + 2 * bwd_qbufs(D)) * tile_bytes(D) + 2 * tile_bytes(128) + bwd_stage_extra(D) + 128;
}
constexpr int kBwdThreads = 512;  // four threads per tile row (each a quarter of the columns)

__device__ __forceinline__ uint64_t bwd_fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float bwd_lo(uint64_t x) { return __uint_as_float(static_cast<uint32_t>(x)); }
__device__ __forceinline__ float bwd_hi(uint64_t x) { return __uint_as_float(static_cast<uint32_t>(x >> 32)); }

// Element-wise add of a shared-memory box into the tensor at (c0, c1, c2) (fp32 per the
// tensor map), tracked in this thread's bulk async-group; rows past the tensor's extent
// are skipped.
__device__ __forceinline__ void tma_reduce_add_3d(const void* map, uint32_t ssrc, int c0, int c1, int c2) {
  asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(ssrc), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// Tensor store of a tile from shared memory (4-D map, coordinates innermost first), tracked
// in this thread's bulk async-group; rows past the tensor's extent are skipped.
__device__ __forceinline__ void tma_store_4d(const void* map, uint32_t ssrc, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(ssrc), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tg, const __grid_constant__ CUtensorMap tdq,
                    const __grid_constant__ CUtensorMap tdo, const BwdParams p) {
  constexpr int NB = bwd_qbufs(D);
  constexpr int TB = tile_bytes(D);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Kt = smem;
  uint8_t* Vt = Kt + TB;
  auto Qb = [&](int k) { return Vt + TB + 2 * k * TB; };
  auto Gb = [&](int k) { return Vt + TB + (2 * k + 1) * TB; };
  uint8_t* Pt = Vt + TB + 2 * NB * TB;
  uint8_t* St = Pt + tile_bytes(128);
  // barriers kv, ld[2], mma, rel (the block's dV and dK MMAs done), then the TMEM address
  uint64_t* bars = reinterpret_cast<uint64_t*>(St + tile_bytes(128) + bwd_stage_extra(D));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  int* next_slot = reinterpret_cast<int*>(tmem_slot + 2);  // the CTA's next work item
  volatile int* kv_pending = reinterpret_cast<volatile int*>(tmem_slot + 3);  // K'/V copies in flight

  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & (kRows - 1), part = tid >> 7;  // tile row, quarter of the row
  // Work items (key block j, head), taken in order: heads in groups of heads_per_group
  // (their Q'/dO tiles, read by every key block of a head, stay in L2 while the group
  // runs); inside a group the heaviest key blocks (j = 0, every query block) come first.
  // A CTA's first item is its block index, every later one comes from the work counter.
  const int BH = p.B * p.H;
  const int total = p.nblk * BH;
  auto item_jbh = [&](int it, int& jj, int& bb, int& hh) {
    const int per_group = p.heads_per_group * p.nblk;
    const int grp_id = it / per_group;
    const int g0 = grp_id * p.heads_per_group;
    const int gh = min(p.heads_per_group, BH - g0);  // heads in this group (the last may be short)
    const int rem = it - grp_id * per_group;
    jj = rem / gh;
    const int bh = g0 + (rem - jj * gh);
    bb = bh / p.H;
    hh = bh - bb * p.H;
  };
  int item = blockIdx.x;
  int j, b, h;
  item_jbh(item, j, b, h);
  const uint32_t bar_kv = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[3]), bar_rel = smem_u32(&bars[4]);
  auto bar_ld = [&](int k) { return smem_u32(&bars[1 + k]); };
  const uint64_t lim = p.wait_limit_ns;

  if (tid == 0) {
    mbar_init(bar_kv, 1);
    mbar_init(bar_ld(0), 1);
    mbar_init(bar_ld(1), 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_rel, 1);
    *abort_flag = 0;
    *kv_pending = 0;
    fence_barrier_init();
    tma_prefetch_map(&tq);
    tma_prefetch_map(&tg);
    tma_prefetch_map(&tv);
    tma_prefetch_map(&tdq);
    tma_prefetch_map(&tdo);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  pdl_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  pdl_wait_prior();  // the prep kernel's q', k', delta, zeroed dq' and work counter
  const uint32_t tS = tbase, tdP = tbase + 128, tdV = tbase + 256, tdK = tbase + 256 + D, tdQ = tbase;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  constexpr uint32_t idesc_s = idesc_bwd(128, 128, false, false);  // S, dP
  constexpr uint32_t idesc_t = idesc_bwd(128, D, true, true);      // dV, dK: A = P^T / dS^T
  constexpr uint32_t idesc_q = idesc_bwd(128, D, false, true);     // dQ: A = dS, B = K'

  // thread 0 only: copies and MMAs in flight, for the abort path (the K'/V flag lives in
  // shared memory: an epilogue's K'/V copies may be issued by another thread)
  bool mma_pending = false;
  bool ld_pending[2] = {false, false};
  uint32_t ph_kv = 0, ph_ld[2] = {0, 0}, ph_mma = 0, ph_rel = 0;
  auto issue_qg_of = [&](int k, int blk, int bb, int hh) {  // Q'_blk and dO_blk of head (bb, hh) into buffer k
    mbar_arrive_expect_tx(bar_ld(k), 2 * TB);
    for (int cb = 0; cb < D / kBlkCols; ++cb) {
      tma_load_4d(smem_u32(Qb(k) + cb * kBlkBytes), &tq, bar_ld(k), cb * kBlkCols, 3 * hh + 0, blk * kRows, bb);
      tma_load_4d(smem_u32(Gb(k) + cb * kBlkBytes), &tg, bar_ld(k), cb * kBlkCols, hh, blk * kRows, bb);
    }
    ld_pending[k] = true;
  };
  auto issue_qg = [&](int k, int blk) { issue_qg_of(k, blk, b, h); };
  auto issue_kv = [&](int jj, int bb, int hh) {  // K'_jj and V_jj of head (bb, hh)
    mbar_arrive_expect_tx(bar_kv, 2 * TB);
    for (int cb = 0; cb < D / kBlkCols; ++cb) {
      tma_load_4d(smem_u32(Kt + cb * kBlkBytes), &tq, bar_kv, cb * kBlkCols, 3 * hh + 1, jj * kRows, bb);
      tma_load_4d(smem_u32(Vt + cb * kBlkBytes), &tv, bar_kv, cb * kBlkCols, 3 * hh + 2, jj * kRows, bb);
    }
    *kv_pending = 1;
  };
  // wait for buffer k's tiles (the query rows arrive rotated)
  auto land = [&](int k, unsigned int site) -> bool {
    wait_phase(bar_ld(k), ph_ld[k], abort_flag, lim, site);
    __syncthreads();
    if (*abort_flag) return false;
    ph_ld[k] ^= 1;
    if (tid == 0) ld_pending[k] = false;
    return true;
  };

  bool ok = true;
  if (tid == 0) {
    issue_kv(j, b, h);
    issue_qg(0, j);
    if (NB == 2 && j + 1 < p.nblk) issue_qg(1, j + 1);
  }
  // ---- one work item per pass; the next item's K'/V (and, with two query-side buffers,
  //      its first Q'/dO tiles) load under this item's epilogue
  for (;;) {
  wait_phase(bar_kv, ph_kv, abort_flag, lim, 42);
  __syncthreads();
  const long long key = static_cast<long long>(j) * kRows + row;
  if (*abort_flag) {
    ok = false;
  } else {
    ph_kv ^= 1;
    if (tid == 0) *kv_pending = 0;
    ok = land(0, 43);
  }
  // the previous item's dk/dv tensor stores have read their tiles before P/dS overwrites them
  if (tid == 0) bulk_wait_read_all();
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  if (!ok) break;

  for (int i = j; i < p.nblk && ok; ++i) {
    const int bi = NB == 2 ? ((i - j) & 1) : 0;
    const bool next = i + 1 < p.nblk;
    // ---- S = Q' K'^T and dP = dO V^T
    if (tid == 0) {
      tc_fence_after_sync();
      const uint32_t qa = smem_u32(Qb(bi)), ka = smem_u32(Kt), ga = smem_u32(Gb(bi)), va = smem_u32(Vt);
      for (int kc = 0; kc < D / 16; ++kc) mma_ss(tS, kmajor_desc(qa, kc), kmajor_desc(ka, kc), idesc_s, kc > 0);
      for (int kc = 0; kc < D / 16; ++kc) mma_ss(tdP, kmajor_desc(ga, kc), kmajor_desc(va, kc), idesc_s, kc > 0);
      tc_commit(bar_mma);
      mma_pending = true;
    }
    const long long q = static_cast<long long>(i) * kRows + row;
    const bool qvalid = q < p.S;
    // this row's lse and delta, loaded while the MMAs run
    const float lse2 = qvalid ? p.lse[(static_cast<long long>(b) * p.H + h) * p.S + q] * kLog2e : 0.0f;
    const float dl = qvalid ? p.delta[(static_cast<long long>(b) * p.H + h) * p.S + q] : 0.0f;
    wait_phase(bar_mma, ph_mma, abort_flag, lim, 40);
    __syncthreads();
    if (*abort_flag) { ok = false; break; }
    ph_mma ^= 1;
    if (tid == 0) mma_pending = false;
    tc_fence_after_sync();

    // ---- the previous block's dq' reductions run under this block's P/dS (two buffers:
    //      staged in that block's Q'/dO buffer); with one buffer they were staged in the
    //      P/dS tiles, which must have been read before P/dS overwrite them
    if (NB == 2) {
      if (tid == 0 && i > j) {
        for (int c = 0; c < D / 32; ++c)
          tma_reduce_add_3d(&tdq, smem_u32(Qb(bi ^ 1) + c * 16384), h * D + 32 * c, (i - 1) * kRows, b);
        bulk_commit_group();
      }
    } else {
      bulk_wait_read_all();
      __syncthreads();
    }
    // ---- P = exp(S/sqrt(D) - lse), dS = P (dP - delta) / sqrt(D) for this thread's 32
    //      keys of the row, to shared memory as bf16
    uint32_t sr2[1][32], dr2[1][32];
    tmem_ld32(tS + lane_off + 32 * part, sr2[0]);
    tmem_ld32(tdP + lane_off + 32 * part, dr2[0]);
    tmem_wait_ld();
    // dS = P (dP - delta) / sqrt(D) = P * (dP / sqrt(D) - delta / sqrt(D)), in fp32 pairs
    const uint64_t sc2 = f32x2_pack(p.scale_log2, p.scale_log2), nl2 = f32x2_pack(-lse2, -lse2);
    const uint64_t ds2 = f32x2_pack(p.scale, p.scale), nd2 = f32x2_pack(-dl * p.scale, -dl * p.scale);
#pragma unroll
    for (int ch = 0; ch < 1; ++ch) {
      const int c0 = 32 * part;
      const uint32_t* sr = sr2[ch];
      const uint32_t* dr = dr2[ch];
      uint32_t pk[16], dk[16];
      const bool full = qvalid && static_cast<long long>(j) * kRows + c0 + 31 <= q;  // no key past the row
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const uint64_t t = ffma2(f32x2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sc2, nl2);
        float p0 = ex2_approx(bwd_lo(t)), p1 = ex2_approx(bwd_hi(t));
        if (!full) {
          const long long kk = static_cast<long long>(j) * kRows + c0 + e;
          if (!(qvalid && kk <= q)) p0 = 0.0f;
          if (!(qvalid && kk + 1 <= q)) p1 = 0.0f;
        }
        const uint64_t pp = f32x2_pack(p0, p1);
        const uint64_t d2 = bwd_fmul2(pp, ffma2(f32x2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), ds2, nd2));
        pk[e / 2] = pack_bf16x2(p0, p1);
        dk[e / 2] = pack_bf16x2(bwd_lo(d2), bwd_hi(d2));
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        *reinterpret_cast<uint4*>(Pt + sw64_off(row, c0 + 8 * k)) =
            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        *reinterpret_cast<uint4*>(St + sw64_off(row, c0 + 8 * k)) =
            make_uint4(dk[4 * k], dk[4 * k + 1], dk[4 * k + 2], dk[4 * k + 3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();

    // ---- dV += P^T dO, dK += dS^T Q' (accumulating over i), dQ'_i = dS K'
    if (tid == 0) {
      // two buffers: the other one, whose staging the previous block's reductions have read
      // by now, takes the next block's tiles first, so they load under these MMAs (the
      // first block's were loaded up front)
      if (NB == 2 && next && i > j) {
        bulk_wait_read_all();
        issue_qg(bi ^ 1, i + 1);
      }
      tc_fence_after_sync();
      const uint32_t pa = smem_u32(Pt), sa = smem_u32(St), ga = smem_u32(Gb(bi)), qa = smem_u32(Qb(bi)),
                     ka = smem_u32(Kt);
      for (int kk = 0; kk < kRows / 16; ++kk)
        mma_ss(tdV, vmajor_desc(pa, kk), vmajor_desc(ga, kk), idesc_t, (i > j || kk > 0) ? 1u : 0u);
      for (int kk = 0; kk < kRows / 16; ++kk)
        mma_ss(tdK, vmajor_desc(sa, kk), vmajor_desc(qa, kk), idesc_t, (i > j || kk > 0) ? 1u : 0u);
      // single query-side buffer: it is free once dV and dK have read dO and Q'
      const bool early = NB == 1 && next;
      if (early) tc_commit(bar_rel);
      for (int kc = 0; kc < kRows / 16; ++kc) mma_ss(tdQ, kmajor_desc(sa, kc), vmajor_desc(ka, kc), idesc_q, kc > 0);
      tc_commit(bar_mma);
      mma_pending = true;
      // ... so the next block's tiles load while dQ' is computed and staged
      if (early && wait_phase(bar_rel, ph_rel, abort_flag, lim, 46)) {
        ph_rel ^= 1;
        issue_qg(0, i + 1);
      }
    }
    wait_phase(bar_mma, ph_mma, abort_flag, lim, 41);
    __syncthreads();
    if (*abort_flag) { ok = false; break; }
    ph_mma ^= 1;
    if (tid == 0) mma_pending = false;
    tc_fence_after_sync();

    // ---- dq' of the block into the fp32 accumulator: this thread's 16-column chunks staged as
    //      128 x 32 boxes, then one tensor reduction per box that runs on while the next
    //      block proceeds (query rows past S fall outside the tensor and are skipped)
    uint8_t* stg = NB == 2 ? Qb(bi) : Pt;
    for (int c0 = 16 * part; c0 < D; c0 += 64) {
      uint32_t r[16];
      tmem_ld16(tdQ + lane_off + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 16; k += 4) {
        const int col = c0 + k;
        *reinterpret_cast<float4*>(stg + (col >> 5) * 16384 + row * 128 + ((((col & 31) >> 2) ^ (row & 7)) << 4)) =
            make_float4(__uint_as_float(r[k]), __uint_as_float(r[k + 1]), __uint_as_float(r[k + 2]),
                        __uint_as_float(r[k + 3]));
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    // one buffer: reduce now; two: at the next block's P/dS (or now, after the last block)
    if (tid == 0 && (NB == 1 || !next)) {
      for (int c = 0; c < D / 32; ++c) tma_reduce_add_3d(&tdq, smem_u32(stg + c * 16384), h * D + 32 * c, i * kRows, b);
      bulk_commit_group();
    }
    if (NB == 1 && next && !land(0, 45)) { ok = false; break; }  // single buffer: issued above
    if (NB == 2 && next && !land(bi ^ 1, 44)) { ok = false; break; }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
  }

  if (!ok) break;
  // ---- the next work item, taken now: its K'/V go into tiles that this item's last MMAs
  //      have finished reading, and load while the epilogue below runs.  The counter's round
  //      trip is taken by a thread with the least staging below (row 0 of the last quarter:
  //      one 16-column chunk of dk' and of dv where D < 128), so that it does not hold up
  //      the barrier after the staging
  if (tid == (D < 128 ? 3 * kRows : 0)) {
    const int nxt = static_cast<int>(gridDim.x) + static_cast<int>(atomicAdd(&g_bwd_next, 1u));
    *next_slot = nxt;
    if (nxt < total) {
      int jn, bn, hn;
      item_jbh(nxt, jn, bn, hn);
      issue_kv(jn, bn, hn);
    }
  }

  // ---- dk = R(key)^T dk' and dv for the rows of key block j, bf16 into slots 1 and 2.
  // staging in the query-side tiles (and, with one buffer, the output tiles over that
  // block's dq' staging): the last reductions must have read theirs
  if (bwd_stage_in_qbuf<D>(p.r)) {
    bulk_wait_read_all();
    __syncthreads();
  }
  if (!*abort_flag) {
    tc_fence_after_sync();
    const bool kvalid = key < p.S;
    const int h2 = p.r >> 1;
    // the table entries of this thread's first 8-dim group, requested before the staging
    float2 cs0[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int d = 8 * part + e;
      cs0[e] = kvalid && d < p.r ? p.cs[key * h2 + (d < h2 ? d : d - h2)] : make_float2(1.0f, 0.0f);
    }
    // dk and dv leave as bf16 tiles (the loads' 64-byte-swizzled layout) from the P/dS tiles,
    // free now (this item's MMAs are done; with one buffer its last reduction has read them).
    // Only the 32-column blocks holding rotated dims go through the fp32 staging, where the
    // rotation finds the pair partners held by the row's other threads.
    uint8_t* const tk = Pt;
    uint8_t* const tvo = Pt + TB;
    const int rc = bwd_rot_cols(p.r);
    float* xs = bwd_stage_in_qbuf<D>(p.r) ? reinterpret_cast<float*>(Qb(0)) + row * rc
                                          : reinterpret_cast<float*>(Pt + 2 * TB) + row * rc;
    auto xcol = [&](int c) { return c ^ (row & 31); };  // a warp's 32 rows on one column: 32 banks
    for (int c0 = 16 * part; c0 < D; c0 += 64) {
      uint32_t r[16];
      tmem_ld16(tdK + lane_off + c0, r);
      tmem_wait_ld();
      if (c0 < rc) {
#pragma unroll
        for (int k = 0; k < 16; ++k) xs[xcol(c0 + k)] = __uint_as_float(r[k]);
      } else {
#pragma unroll
        for (int k = 0; k < 16; k += 8)
          *reinterpret_cast<uint4*>(tk + sw64_off(row, c0 + k)) =
              make_uint4(pack_bf16x2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                         pack_bf16x2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])),
                         pack_bf16x2(__uint_as_float(r[k + 4]), __uint_as_float(r[k + 5])),
                         pack_bf16x2(__uint_as_float(r[k + 6]), __uint_as_float(r[k + 7])));
      }
    }
    for (int c0 = 16 * part; c0 < D; c0 += 64) {
      uint32_t r[16];
      tmem_ld16(tdV + lane_off + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 16; k += 8)
        *reinterpret_cast<uint4*>(tvo + sw64_off(row, c0 + k)) =
            make_uint4(pack_bf16x2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                       pack_bf16x2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])),
                       pack_bf16x2(__uint_as_float(r[k + 4]), __uint_as_float(r[k + 5])),
                       pack_bf16x2(__uint_as_float(r[k + 6]), __uint_as_float(r[k + 7])));
    }
    // two buffers with the staging beside the output tiles: both buffers are free once the
    // last reductions have read their staging (thread 0's bulk groups); the next item's first
    // Q'/dO tiles load under the rotation
    const bool early_qg = NB == 2 && !bwd_stage_in_qbuf<D>(p.r);
    if (early_qg && tid == 0) bulk_wait_read_all();
    __syncthreads();
    if (early_qg && tid == 0) {
      const int nxt = *next_slot;
      if (nxt < total) {
        int jn, bn, hn;
        item_jbh(nxt, jn, bn, hn);
        issue_qg_of(0, jn, bn, hn);
        if (jn + 1 < p.nblk) issue_qg_of(1, jn + 1, bn, hn);
      }
    }
    // dk = R(key)^T dk' on the staged columns, this thread's 8-dim groups (rows past S are
    // zeros: the tensor stores skip them)
    for (int d0 = 8 * part; d0 < rc; d0 += 32) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int d = d0 + e;
        float v = kvalid ? xs[xcol(d)] : 0.0f;
        if (kvalid && d < h2) {
          const float2 c = d0 == 8 * part ? cs0[e] : p.cs[key * h2 + d];
          v = fmaf(v, c.x, xs[xcol(d + h2)] * c.y);
        } else if (kvalid && d < p.r) {
          const float2 c = d0 == 8 * part ? cs0[e] : p.cs[key * h2 + (d - h2)];
          v = fmaf(v, c.x, -xs[xcol(d - h2)] * c.y);
        }
        y[e] = v;
      }
      *reinterpret_cast<uint4*>(tk + sw64_off(row, d0)) = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                                                     pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
    }
    fence_proxy_async_smem();
    __syncthreads();
    // slots 1 and 2 of the key block's rows by tensor stores (the next item waits for them
    // to have read the tiles before its first P/dS)
    if (tid == 0) {
      for (int cb = 0; cb < D / kBlkCols; ++cb) {
        tma_store_4d(&tdo, smem_u32(tk + cb * kBlkBytes), cb * kBlkCols, 3 * h + 1, j * kRows, b);
        tma_store_4d(&tdo, smem_u32(tvo + cb * kBlkBytes), cb * kBlkCols, 3 * h + 2, j * kRows, b);
      }
      bulk_commit_group();
    }
  }
  // ---- this item's TMEM and staging reads done: hand over to the next item (one buffer:
  //      its first Q'/dO tiles go into the query-side tiles the dk' staging used)
  tc_fence_before_sync();
  __syncthreads();
  if (*abort_flag) {
    ok = false;
    break;
  }
  item = *next_slot;
  if (item >= total) break;
  item_jbh(item, j, b, h);
  if (bwd_stage_in_qbuf<D>(p.r) && tid == 0) {  // its staging used the query-side tiles
    issue_qg(0, j);
    if (NB == 2 && j + 1 < p.nblk) issue_qg(1, j + 1);
  }
  }  // work items

  // ---- teardown: let the copies, reductions and MMAs in flight land, then free TMEM
  bulk_wait_all();
  if (tid == 0) {
    if (*kv_pending) drain_phase(bar_kv, ph_kv, lim);
    for (int k = 0; k < 2; ++k)
      if (ld_pending[k]) drain_phase(bar_ld(k), ph_ld[k], lim);
    if (mma_pending) drain_phase(bar_mma, ph_mma, lim);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace neox
