// attn_simple.cuh -- the plain tcgen05 attention kernel: one CTA (one warpgroup) per
// 128-row query tile, every stage in sequence (TMA -> rotary -> S MMA -> softmax -> PV MMA).
// It exists to check the operand layouts, descriptors and TMEM formats on their own; the
// warp-specialised persistent kernel (attn_ws.cuh) is the fast path.
#pragma once

#include "attn_common.cuh"

namespace neox {

template <int D>
__global__ void __launch_bounds__(128, 1)
    attn_fwd_simple_kernel(const __grid_constant__ CUtensorMap tmap, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int RS = p.side_cols;
  uint8_t* Qraw = smem;
  uint8_t* Qside = Qraw + tile_bytes(D);
  uint8_t* Kraw = Qside + tile_bytes(RS);
  uint8_t* Kside = Kraw + tile_bytes(D);
  uint8_t* Vt = Kside + tile_bytes(RS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(Vt + tile_bytes(D));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int m = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int row0 = m * kRows;
  const uint32_t bar_tma = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);

  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmap);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  for (int i = tid * 16; i < tile_bytes(RS); i += 128 * 16) {
    *reinterpret_cast<uint4*>(Qside + i) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(Kside + i) = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tS = tbase, tO = tbase + 128;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t idesc_s = idesc_bf16_f32(128, 128, false);
  const uint32_t idesc_pv = idesc_bf16_f32(128, D, true);

  uint32_t ph_tma = 0, ph_mma = 0;
  bool pending_tma = false, pending_mma = false;  // meaningful in thread 0 only
  bool ok = true;

  // ---- Q tile: load, rotate
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_tma, tile_bytes(D));
    for (int cb = 0; cb < D / kBlkCols; ++cb)
      tma_load_4d(smem_u32(Qraw + cb * kBlkBytes), &tmap, bar_tma, cb * kBlkCols, 3 * h + 0, row0, b);
    pending_tma = true;
  }
  wait_phase(bar_tma, ph_tma, abort_flag, p.wait_limit_ns, 1);
  __syncthreads();
  ok = !*abort_flag;
  if (ok) {
    ph_tma ^= 1;
    pending_tma = false;
    if (p.r > 0) {
      const int64_t pos = row0 + tid;
      rotate_row(Qraw, Qside, tid, pos < p.S ? pos : -1, p.cs, p.r);
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  float m_used = -INFINITY, l_run = 0.0f;
  const int row = tid;
  for (int j = 0; j <= m && ok; ++j) {
    if (tid == 0) {
      mbar_arrive_expect_tx(bar_tma, 2 * tile_bytes(D));
      for (int cb = 0; cb < D / kBlkCols; ++cb) {
        tma_load_4d(smem_u32(Kraw + cb * kBlkBytes), &tmap, bar_tma, cb * kBlkCols, 3 * h + 1, j * kRows, b);
        tma_load_4d(smem_u32(Vt + cb * kBlkBytes), &tmap, bar_tma, cb * kBlkCols, 3 * h + 2, j * kRows, b);
      }
      pending_tma = true;
    }
    wait_phase(bar_tma, ph_tma, abort_flag, p.wait_limit_ns, 2);
    __syncthreads();
    if (*abort_flag) { ok = false; break; }
    ph_tma ^= 1;
    pending_tma = false;
    if (p.r > 0) {
      const int64_t pos = static_cast<int64_t>(j) * kRows + tid;
      rotate_row(Kraw, Kside, tid, pos < p.S ? pos : -1, p.cs, p.r);
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- S = Q' K'^T  (pass + hi.hi over D columns, then lo.hi and hi.lo over r16 columns)
    if (tid == 0) {
      tc_fence_after_sync();
      const uint32_t q = smem_u32(Qraw), qs = smem_u32(Qside), k = smem_u32(Kraw), ks = smem_u32(Kside);
      for (int kc = 0; kc < D / 16; ++kc) mma_ss(tS, kmajor_desc(q, kc), kmajor_desc(k, kc), idesc_s, kc > 0);
      for (int kc = 0; kc < p.r16 / 16; ++kc) {
        mma_ss(tS, kmajor_desc(qs, kc), kmajor_desc(k, kc), idesc_s, 1);
        mma_ss(tS, kmajor_desc(q, kc), kmajor_desc(ks, kc), idesc_s, 1);
      }
      tc_commit(bar_mma);
      pending_mma = true;
    }
    wait_phase(bar_mma, ph_mma, abort_flag, p.wait_limit_ns, 3);
    __syncthreads();
    if (*abort_flag) { ok = false; break; }
    ph_mma ^= 1;
    if (tid == 0) pending_mma = false;
    tc_fence_after_sync();

    // ---- softmax of this row block
    uint32_t sr[128];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, sr + c * 32);
    tmem_wait_ld();
    const bool diag = (j == m);
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 128; ++c) {
      float v = __uint_as_float(sr[c]);
      if (diag && c > row) v = -INFINITY;
      sr[c] = __float_as_uint(v);
      mx = fmaxf(mx, v);
    }
    const float mx_s = mx * p.scale_log2;
    float m_new = m_used;
    bool rescale = false;
    if (j == 0) {
      m_new = mx_s;
    } else if (mx_s > m_used + 8.0f) {
      m_new = mx_s;
      rescale = true;
    }
    const float alpha = rescale ? ex2_approx(m_used - m_new) : 1.0f;
    float rowsum = 0.0f;
    uint32_t pk[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), p.scale_log2, -m_new));
      const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), p.scale_log2, -m_new));
      rowsum += p0 + p1;
      pk[c] = pack_bf16x2(p0, p1);
    }
    l_run = l_run * alpha + rowsum;
    m_used = m_new;
    if (__any_sync(0xffffffffu, rescale)) {
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c0, o);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
        tmem_st32(tO + lane_off + c0, o);
      }
    }
    tmem_st32(tS + lane_off, pk);
    tmem_st32(tS + lane_off + 32, pk + 32);
    tmem_wait_st();
    tc_fence_before_sync();
    __syncthreads();

    // ---- O += P V   (P from TMEM, V as an MN-major smem operand)
    if (tid == 0) {
      tc_fence_after_sync();
      const uint32_t v = smem_u32(Vt);
      for (int kk = 0; kk < kRows / 16; ++kk) mma_ts(tO, tS + kk * 8, vmajor_desc(v, kk), idesc_pv, (j > 0 || kk > 0));
      tc_commit(bar_mma);
      pending_mma = true;
    }
    wait_phase(bar_mma, ph_mma, abort_flag, p.wait_limit_ns, 4);
    __syncthreads();
    if (*abort_flag) { ok = false; break; }
    ph_mma ^= 1;
    if (tid == 0) pending_mma = false;
    tc_fence_after_sync();
  }

  // ---- epilogue: out = O / l (bf16), lse = ln 2 * (m + log2 l)
  if (ok && !*abort_flag) {
    const int qrow = row0 + row;
    const float inv_l = 1.0f / l_run;
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t o[32];
      tmem_ld32(tO + lane_off + c0, o);
      tmem_wait_ld();
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        pk[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
      if (qrow < p.S) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((static_cast<int64_t>(b) * p.S + qrow) * p.H + h) * D + c0);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
    }
    if (qrow < p.S)
      p.lse[(static_cast<int64_t>(b) * p.H + h) * p.S + qrow] = (m_used + log2f(l_run)) * 0.69314718055994530942f;
  }

  // ---- teardown: let in-flight async work land, then free TMEM
  if (tid == 0) {
    if (pending_tma) drain_phase(bar_tma, ph_tma, p.wait_limit_ns);
    if (pending_mma) drain_phase(bar_mma, ph_mma, p.wait_limit_ns);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 256);
  }
}

__host__ __device__ constexpr int simple_smem_bytes(int D, int side_cols) {
  return 1024 + 3 * tile_bytes(D) + 2 * tile_bytes(side_cols) + 64;
}

}  // namespace neox
