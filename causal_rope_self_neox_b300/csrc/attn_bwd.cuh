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
//   attn_bwd_delta_kernel  delta_i (fp32) and a zeroed fp32 dq' accumulator;
//   attn_bwd_kernel        one CTA per (key block j, head): K'_j, V_j stay in shared
//                          memory while query blocks i >= j stream through; per block
//                          five tcgen05 MMAs (S = Q'K'^T and dP = dO V^T into TMEM, then
//                          dV += P^T dO and dK += dS^T Q' accumulating in TMEM over i, and
//                          dQ'_i = dS K' added to the fp32 accumulator with vector reds);
//                          at the end dk (rotated back) and dv are written as bf16;
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
  float* dq_acc;         // fp32 [B, S, H, D]  scratch: dq' before the rotation back
  float* delta;          // fp32 [B, H, S]     scratch
  const float2* cs;      // cos/sin table [>= S rows][r/2]
  int B, S, H, r, nblk;
  float scale_log2;      // log2(e) / sqrt(D)
  float scale;           // 1 / sqrt(D)
  uint64_t wait_limit_ns;
};

constexpr float kLog2e = 1.4426950408889634f;

// delta[b, h, s] = dout . out for every row (one warp per row), and dq_acc zeroed.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_delta_kernel(const BwdParams p) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);  // [b][s][h]
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<long long>(p.B) * p.S * p.H) return;
  const uint16_t* o = p.out + row * D;
  const uint16_t* g = p.dout + row * D;
  float acc = 0.0f;
  for (int d = lane; d < D; d += 32) acc = fmaf(bf16_bits_to_f32(o[d]), bf16_bits_to_f32(g[d]), acc);
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
  float* dq = p.dq_acc + row * D;
  for (int d = lane; d < D; d += 32) dq[d] = 0.0f;
  if (lane == 0) {
    const long long h = row % p.H, s = (row / p.H) % p.S, b = row / (static_cast<long long>(p.H) * p.S);
    p.delta[(b * p.H + h) * p.S + s] = acc;
  }
}

// dq = R(s)^T dq' (bf16) into slot 0 of dqkv, one thread per row:
//   dq_i = dq'_i c + dq'_{i+h} s,  dq_{i+h} = dq'_{i+h} c - dq'_i s  (i < h = r/2).
template <int D>
__global__ void __launch_bounds__(128) attn_bwd_dq_kernel(const BwdParams p) {
  const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;  // [b][s][h]
  if (row >= static_cast<long long>(p.B) * p.S * p.H) return;
  const long long s = (row / p.H) % p.S;
  const float* src = p.dq_acc + row * D;
  const int h2 = p.r >> 1;
  uint4* dst = reinterpret_cast<uint4*>(p.dqkv + row * 3 * D);
  for (int d0 = 0; d0 < D; d0 += 8) {
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int d = d0 + e;
      float v = src[d];
      if (d < h2) {
        const float2 c = p.cs[s * h2 + d];
        v = fmaf(v, c.x, src[d + h2] * c.y);
      } else if (d < p.r) {
        const float2 c = p.cs[s * h2 + (d - h2)];
        v = fmaf(v, c.x, -src[d - h2] * c.y);
      }
      y[e] = v;
    }
    dst[d0 / 8] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                             pack_bf16x2(y[6], y[7]));
  }
}

// Rows [128 blk, 128 blk + 128) of one head of a row-major [B, S, H, stride] bf16 tensor
// (head offset `col0` elements into the row) into a swizzled [128][D] tile; rows >= S
// are zero.  Consecutive threads read consecutive 16-byte chunks of a row; every
// thread's loads are issued before its first store (one memory latency per tile).
template <int D>
__device__ __forceinline__ void bwd_load_tile(uint8_t* tile, const uint16_t* base, long long row_stride, int col0,
                                              const BwdParams& p, int b, int h, int blk) {
  constexpr int CH = D / 8;
  constexpr int PER = kRows * CH / 128;  // 128 threads
  uint4 v[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int idx = threadIdx.x + 128 * k;
    const int row = idx / CH, ch = idx - row * CH;
    const int s = blk * kRows + row;
    v[k] = make_uint4(0, 0, 0, 0);
    if (s < p.S)
      v[k] = *reinterpret_cast<const uint4*>(base + ((static_cast<long long>(b) * p.S + s) * p.H + h) * row_stride +
                                             col0 + ch * 8);
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int idx = threadIdx.x + 128 * k;
    const int row = idx / CH, ch = idx - row * CH;
    *reinterpret_cast<uint4*>(tile + sw64_off(row, ch * 8)) = v[k];
  }
}

// Rotate the first r dims of one tile row in place at position pos (rounded to bf16).
__device__ __forceinline__ void bwd_rotate_row(uint8_t* tile, int row, long long pos, const float2* cs, int r) {
  const int h2 = r >> 1;
  for (int i = 0; i < h2; ++i) {
    uint16_t* pa = reinterpret_cast<uint16_t*>(tile + sw64_off(row, i));
    uint16_t* pb = reinterpret_cast<uint16_t*>(tile + sw64_off(row, i + h2));
    const float x1 = bf16_bits_to_f32(*pa), x2 = bf16_bits_to_f32(*pb);
    const float2 c = cs[pos * h2 + i];
    *pa = f32_to_bf16_bits(fmaf(x1, c.x, -x2 * c.y));
    *pb = f32_to_bf16_bits(fmaf(x2, c.x, x1 * c.y));
  }
}

// kind::f16 instruction descriptor with the A major-ness as well (bit 15: 1 = MN-major).
__host__ __device__ constexpr uint32_t idesc_bwd(int M, int N, bool a_mn, bool b_mn) {
  return idesc_bf16_f32(M, N, b_mn) | ((a_mn ? 1u : 0u) << 15);
}

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// smem: K'_j, V_j, Q'_i, dO_i tiles [128][D], P_i and dS_i tiles [128][128], a barrier,
// the TMEM address and the abort flag (tiles 1 KB aligned).
__host__ __device__ constexpr int bwd_smem_bytes(int D) { return 1024 + 4 * tile_bytes(D) + 2 * tile_bytes(128) + 64; }

template <int D>
__global__ void __launch_bounds__(128, 1) attn_bwd_kernel(const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Kt = smem;
  uint8_t* Vt = Kt + tile_bytes(D);
  uint8_t* Qt = Vt + tile_bytes(D);
  uint8_t* Gt = Qt + tile_bytes(D);
  uint8_t* Pt = Gt + tile_bytes(D);
  uint8_t* St = Pt + tile_bytes(128);
  uint64_t* bar = reinterpret_cast<uint64_t*>(St + tile_bytes(128));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int BH = p.B * p.H;
  const int j = blockIdx.x / BH;  // key block; the heaviest (j = 0) blocks are launched first
  const int bh = blockIdx.x - j * BH;
  const int b = bh / p.H, h = bh - b * p.H;
  const uint32_t bar_mma = smem_u32(bar);

  if (tid == 0) {
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  // K'_j (rotated) and V_j
  bwd_load_tile<D>(Kt, p.qkv, 3 * D, D, p, b, h, j);
  bwd_load_tile<D>(Vt, p.qkv, 3 * D, 2 * D, p, b, h, j);
  __syncthreads();
  const long long key = static_cast<long long>(j) * kRows + tid;
  if (p.r > 0 && key < p.S) bwd_rotate_row(Kt, tid, key, p.cs, p.r);
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tbase = *tmem_slot;
  const uint32_t tS = tbase, tdP = tbase + 128, tdV = tbase + 256, tdK = tbase + 256 + D, tdQ = tbase;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  constexpr uint32_t idesc_s = idesc_bwd(128, 128, false, false);  // S, dP
  constexpr uint32_t idesc_t = idesc_bwd(128, D, true, true);      // dV, dK: A = P^T / dS^T
  constexpr uint32_t idesc_q = idesc_bwd(128, D, false, true);     // dQ: A = dS, B = K'
  uint32_t ph = 0;
  bool pending = false;  // thread 0: an MMA commit not yet waited for
  bool ok = true;

  for (int i = j; i < p.nblk && ok; ++i) {
    // ---- Q'_i (rotated) and dO_i
    bwd_load_tile<D>(Qt, p.qkv, 3 * D, 0, p, b, h, i);
    bwd_load_tile<D>(Gt, p.dout, D, 0, p, b, h, i);
    __syncthreads();
    const long long q = static_cast<long long>(i) * kRows + tid;
    const bool qvalid = q < p.S;
    if (p.r > 0 && qvalid) bwd_rotate_row(Qt, tid, q, p.cs, p.r);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();

    // ---- S = Q' K'^T, dP = dO V^T
    if (tid == 0) {
      tc_fence_after_sync();
      const uint32_t qa = smem_u32(Qt), ka = smem_u32(Kt), ga = smem_u32(Gt), va = smem_u32(Vt);
      for (int kc = 0; kc < D / 16; ++kc) mma_ss(tS, kmajor_desc(qa, kc), kmajor_desc(ka, kc), idesc_s, kc > 0);
      for (int kc = 0; kc < D / 16; ++kc) mma_ss(tdP, kmajor_desc(ga, kc), kmajor_desc(va, kc), idesc_s, kc > 0);
      tc_commit(bar_mma);
      pending = true;
    }
    wait_phase(bar_mma, ph, abort_flag, p.wait_limit_ns, 40);
    __syncthreads();
    if (*abort_flag) { ok = false; break; }
    ph ^= 1;
    if (tid == 0) pending = false;
    tc_fence_after_sync();

    // ---- P = exp(S/sqrt(D) - lse), dS = P (dP - delta) / sqrt(D), both to smem as bf16
    const float lse2 = qvalid ? p.lse[(static_cast<long long>(b) * p.H + h) * p.S + q] * kLog2e : 0.0f;
    const float dl = qvalid ? p.delta[(static_cast<long long>(b) * p.H + h) * p.S + q] : 0.0f;
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t sr[32], dr[32];
      tmem_ld32(tS + lane_off + c0, sr);
      tmem_ld32(tdP + lane_off + c0, dr);
      tmem_wait_ld();
      uint32_t pk[16], dk[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float pe[2], de[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const long long kk = static_cast<long long>(j) * kRows + c0 + e + u;
          const bool use = qvalid && kk <= q;
          const float pv = use ? ex2_approx(fmaf(__uint_as_float(sr[e + u]), p.scale_log2, -lse2)) : 0.0f;
          pe[u] = pv;
          de[u] = pv * (__uint_as_float(dr[e + u]) - dl) * p.scale;
        }
        pk[e / 2] = pack_bf16x2(pe[0], pe[1]);
        dk[e / 2] = pack_bf16x2(de[0], de[1]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        *reinterpret_cast<uint4*>(Pt + sw64_off(tid, c0 + 8 * k)) =
            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        *reinterpret_cast<uint4*>(St + sw64_off(tid, c0 + 8 * k)) =
            make_uint4(dk[4 * k], dk[4 * k + 1], dk[4 * k + 2], dk[4 * k + 3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();

    // ---- dV += P^T dO, dK += dS^T Q' (accumulating over i), dQ'_i = dS K'
    if (tid == 0) {
      tc_fence_after_sync();
      const uint32_t pa = smem_u32(Pt), sa = smem_u32(St), ga = smem_u32(Gt), qa = smem_u32(Qt), ka = smem_u32(Kt);
      for (int kk = 0; kk < kRows / 16; ++kk)
        mma_ss(tdV, vmajor_desc(pa, kk), vmajor_desc(ga, kk), idesc_t, (i > j || kk > 0) ? 1u : 0u);
      for (int kk = 0; kk < kRows / 16; ++kk)
        mma_ss(tdK, vmajor_desc(sa, kk), vmajor_desc(qa, kk), idesc_t, (i > j || kk > 0) ? 1u : 0u);
      for (int kc = 0; kc < kRows / 16; ++kc) mma_ss(tdQ, kmajor_desc(sa, kc), vmajor_desc(ka, kc), idesc_q, kc > 0);
      tc_commit(bar_mma);
      pending = true;
    }
    wait_phase(bar_mma, ph, abort_flag, p.wait_limit_ns, 41);
    __syncthreads();
    if (*abort_flag) { ok = false; break; }
    ph ^= 1;
    if (tid == 0) pending = false;
    tc_fence_after_sync();

    // ---- dq' rows of this query block into the fp32 accumulator
    float* dq = p.dq_acc + ((static_cast<long long>(b) * p.S + (qvalid ? q : 0)) * p.H + h) * D;
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tdQ + lane_off + c0, r);
      tmem_wait_ld();
      if (qvalid) {
#pragma unroll
        for (int k = 0; k < 32; k += 4)
          red_add_v4(dq + c0 + k, __uint_as_float(r[k]), __uint_as_float(r[k + 1]), __uint_as_float(r[k + 2]),
                     __uint_as_float(r[k + 3]));
      }
    }
    tc_fence_before_sync();
    __syncthreads();
  }

  // ---- dk = R(key)^T dk', dv: rows of key block j, bf16 into slots 1 and 2
  if (ok && !*abort_flag) {
    tc_fence_after_sync();
    const bool kvalid = key < p.S;
    uint16_t* dst = p.dqkv + ((static_cast<long long>(b) * p.S + (kvalid ? key : 0)) * p.H + h) * 3 * D;
    // dk' row staged in shared memory (the Q'/dO/P/dS tiles are free now), one padded
    // row per thread, so the rotation can pick its pair partners by index
    float* xs = reinterpret_cast<float*>(Qt) + tid * (D + 1);
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tdK + lane_off + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 32; ++k) xs[c0 + k] = __uint_as_float(r[k]);
    }
    const int h2 = p.r >> 1;
    if (kvalid) {
      for (int d0 = 0; d0 < D; d0 += 8) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int d = d0 + e;
          float v = xs[d];
          if (d < h2) {
            const float2 c = p.cs[key * h2 + d];
            v = fmaf(v, c.x, xs[d + h2] * c.y);
          } else if (d < p.r) {
            const float2 c = p.cs[key * h2 + (d - h2)];
            v = fmaf(v, c.x, -xs[d - h2] * c.y);
          }
          y[e] = v;
        }
        *reinterpret_cast<uint4*>(dst + D + d0) = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                                             pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
      }
    }
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tdV + lane_off + c0, r);
      tmem_wait_ld();
      if (kvalid) {
#pragma unroll
        for (int k = 0; k < 32; k += 8)
          *reinterpret_cast<uint4*>(dst + 2 * D + c0 + k) =
              make_uint4(pack_bf16x2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                         pack_bf16x2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])),
                         pack_bf16x2(__uint_as_float(r[k + 4]), __uint_as_float(r[k + 5])),
                         pack_bf16x2(__uint_as_float(r[k + 6]), __uint_as_float(r[k + 7])));
      }
    }
  }

  // ---- teardown: let an MMA in flight land, then free TMEM
  if (tid == 0 && pending) drain_phase(bar_mma, ph, p.wait_limit_ns);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace neox
