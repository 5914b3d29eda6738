// neox_attn.cu -- the C ABI (include/neox_attn.h): argument validation, the cached
// cos/sin table, TMA descriptor encoding and kernel launch.  No torch types anywhere.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "neox_attn.h"
#include "attn_common.cuh"
#include "attn_simple.cuh"
#include "attn_ws.cuh"
#include "decode.cuh"
#include "attn_bwd.cuh"
#include "qkv_proj.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return NEOX_ERR_CUDA;
}

// ---------------------------------------------------------------- validation ----
bool ranges_overlap(uintptr_t a, uint64_t na, uintptr_t b, uint64_t nb) { return a < b + nb && b < a + na; }

int validate(const void* qkv, int B, int S, int H, int D, int r, float base, const void* out, const float* lse) {
  if (!qkv || !out || !lse) return NEOX_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1) return NEOX_ERR_INVALID_ARG;
  if (D != 64 && D != 96 && D != 128) return NEOX_ERR_UNSUPPORTED_HEAD_DIM;
  if (r < 0 || r > D || (r & 1)) return NEOX_ERR_INVALID_ARG;
  if (!(base > 0.0f) || !std::isfinite(base)) return NEOX_ERR_INVALID_ARG;
  const uint64_t elems = static_cast<uint64_t>(B) * S * H * 3 * D;
  if (elems >= (1ull << 40)) return NEOX_ERR_INVALID_ARG;
  if (static_cast<uint64_t>(B) * H > 0x7FFFFFFFull) return NEOX_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return NEOX_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(lse) & 3) return NEOX_ERR_MISALIGNED;
  const uint64_t qkv_bytes = elems * 2, out_bytes = elems / 3 * 2, lse_bytes = static_cast<uint64_t>(B) * H * S * 4;
  const uintptr_t q = reinterpret_cast<uintptr_t>(qkv), o = reinterpret_cast<uintptr_t>(out),
                  l = reinterpret_cast<uintptr_t>(lse);
  if (ranges_overlap(q, qkv_bytes, o, out_bytes) || ranges_overlap(q, qkv_bytes, l, lse_bytes) ||
      ranges_overlap(o, out_bytes, l, lse_bytes))
    return NEOX_ERR_INVALID_ARG;
  return NEOX_OK;
}

// --------------------------------------------------------- device properties ----
struct DeviceInfo {
  bool known = false;
  bool supported = false;
  int num_sms = 0;
  bool smem_configured = false;
};
std::mutex g_dev_mu;
std::vector<DeviceInfo> g_devs;

int current_device(int* dev, DeviceInfo* info) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (static_cast<int>(g_devs.size()) <= *dev) g_devs.resize(*dev + 1);
  DeviceInfo& d = g_devs[*dev];
  if (!d.known) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, *dev)) != cudaSuccess) return cuda_fail(e);
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.known = true;
  }
  *info = d;
  return d.supported ? NEOX_OK : NEOX_ERR_NO_DEVICE_SUPPORT;
}

// ------------------------------------------------------------ cos/sin tables ----
struct Table {
  int device;
  int r;
  float base;
  int64_t rows;  // positions covered
  float2* ptr;
};
std::mutex g_tab_mu;
std::vector<Table> g_tables;

int get_table(int device, int S, int r, float base, cudaStream_t stream, const float2** out) {
  std::lock_guard<std::mutex> lk(g_tab_mu);
  for (auto it = g_tables.begin(); it != g_tables.end(); ++it) {
    if (it->device == device && it->r == r && it->base == base) {
      if (it->rows >= S) {
        *out = it->ptr;
        return NEOX_OK;
      }
      // too short: in-flight kernels may still read it, so let the device go idle first
      cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return cuda_fail(e);
      cudaFree(it->ptr);
      g_tables.erase(it);
      break;
    }
  }
  const int h = r / 2;
  const int64_t rows = ((static_cast<int64_t>(S) + 2047) / 2048) * 2048;
  float2* ptr = nullptr;
  cudaError_t e = cudaMalloc(&ptr, sizeof(float2) * rows * h);
  if (e != cudaSuccess) return cuda_fail(e);
  const int64_t n = rows * h;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<int64_t>((n + threads - 1) / threads, 65535));
  neox::rope_table_kernel<<<blocks, threads, 0, stream>>>(ptr, static_cast<int>(rows), h, r, static_cast<double>(base));
  if ((e = cudaGetLastError()) != cudaSuccess || (e = cudaStreamSynchronize(stream)) != cudaSuccess) {
    cudaFree(ptr);
    return cuda_fail(e);
  }
  g_tables.push_back(Table{device, r, base, rows, ptr});
  *out = ptr;
  return NEOX_OK;
}

// -------------------------------------------------------------- tensor maps ----
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// cuTensorMapEncodeTiled through the runtime's driver entry point, resolved once.
bool resolve_encode() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

int encode_qkv_map(CUtensorMap* map, const void* qkv, int B, int S, int H, int D) {
  if (!resolve_encode()) return cuda_fail(cudaErrorNotSupported);
  // dims (innermost first): head dim, (head, slot), sequence, batch.
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(3) * H, static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(3) * H * D * 2,
                           static_cast<cuuint64_t>(S) * 3 * H * D * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(neox::kBlkCols), 1, static_cast<cuuint32_t>(neox::kRows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(qkv), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return NEOX_OK;
}

// 2-D bf16 map over a row-major [outer, inner] matrix.
int encode_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swizzle) {
  if (!resolve_encode()) return cuda_fail(cudaErrorNotSupported);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return NEOX_OK;
}

int validate_proj(const void* x, const void* w, const void* bias, int B, int S, int hidden, int H, int D, int r,
                  float base, const void* qkv) {
  if (!x || !w || !qkv) return NEOX_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || hidden < 8 || (hidden & 7)) return NEOX_ERR_INVALID_ARG;
  if (D != 64 && D != 96 && D != 128) return NEOX_ERR_UNSUPPORTED_HEAD_DIM;
  if (r < 0 || r > D || (r & 1)) return NEOX_ERR_INVALID_ARG;
  if (!(base > 0.0f) || !std::isfinite(base)) return NEOX_ERR_INVALID_ARG;
  const uint64_t M = static_cast<uint64_t>(B) * S, N = static_cast<uint64_t>(3) * H * D;
  if (M > 0x7FFFFFFFull || N > 0x7FFFFFFFull) return NEOX_ERR_INVALID_ARG;
  if (M * hidden >= (1ull << 40) || N * hidden >= (1ull << 40) || M * N >= (1ull << 40)) return NEOX_ERR_INVALID_ARG;
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x), wa = reinterpret_cast<uintptr_t>(w),
                  ba = reinterpret_cast<uintptr_t>(bias), oa = reinterpret_cast<uintptr_t>(qkv);
  if ((xa & 15) || (wa & 15) || (ba & 15) || (oa & 15)) return NEOX_ERR_MISALIGNED;
  const uint64_t out_bytes = M * N * 2;
  if (ranges_overlap(oa, out_bytes, xa, M * hidden * 2) || ranges_overlap(oa, out_bytes, wa, N * hidden * 2) ||
      (bias && ranges_overlap(oa, out_bytes, ba, N * 2)))
    return NEOX_ERR_INVALID_ARG;
  return NEOX_OK;
}

// ------------------------------------------------------------------ launches ----
struct Prepared {
  CUtensorMap map;
  CUtensorMap map_rot;  // the pre-rotated copy (pre == true only)
  bool pre = false;
  neox::AttnParams p;
  DeviceInfo dev;
  int device;
};

int prepare(const void* qkv, int B, int S, int H, int D, int r, float base, void* out, float* lse, cudaStream_t stream,
            Prepared* P) {
  int rc = validate(qkv, B, S, H, D, r, base, out, lse);
  if (rc != NEOX_OK) return rc;
  rc = current_device(&P->device, &P->dev);
  if (rc != NEOX_OK) return rc;
  const float2* cs = nullptr;
  if (r > 0) {
    rc = get_table(P->device, S, r, base, stream, &cs);
    if (rc != NEOX_OK) return rc;
  }
  rc = encode_qkv_map(&P->map, qkv, B, S, H, D);
  if (rc != NEOX_OK) return rc;
  neox::AttnParams& p = P->p;
  p.cs = cs;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.B = B;
  p.S = S;
  p.H = H;
  p.r = r;
  p.r16 = (r + 15) / 16 * 16;
  p.side_cols = r > 0 ? (p.r16 + 31) / 32 * 32 : 0;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  p.num_units = 0;
  p.wait_limit_ns = neox::kWaitLimitNs;
  return NEOX_OK;
}

template <int D>
int launch_simple(const Prepared& P, cudaStream_t stream) {
  const int smem = neox::simple_smem_bytes(D, P.p.side_cols);
  cudaError_t e = cudaFuncSetAttribute(neox::attn_fwd_simple_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  if (P.p.H > 65535 || P.p.B > 65535) return NEOX_ERR_INVALID_ARG;
  dim3 grid((P.p.S + neox::kRows - 1) / neox::kRows, P.p.H, P.p.B);
  neox::attn_fwd_simple_kernel<D><<<grid, 128, smem, stream>>>(P.map, P.p);
  e = cudaGetLastError();
  return e == cudaSuccess ? NEOX_OK : cuda_fail(e);
}

template <int D>
int launch_ws(Prepared& P, cudaStream_t stream) {
  const int rc = neox::launch_attn_ws<D>(P.map, P.pre ? P.map_rot : P.map, P.pre, P.p, P.dev.num_sms, stream,
                                         &g_last_cuda_error);
  return rc == 0 ? NEOX_OK : rc == -1 ? NEOX_ERR_INVALID_ARG : NEOX_ERR_CUDA;
}

// ------------------------------------------------------------------- decode ----
// Per-device decode scratch: fp32 partial states of heads that span several CTAs, and one
// int32 arrival counter per head (zeroed when allocated; every launch leaves them zero,
// except one that gave up on a timed-out wait, after which the error report re-zeroes them).
struct Scratch {
  int device;
  size_t bytes;
  float* ptr;
  size_t counters;  // entries
  int* cnt;
};
std::vector<Scratch> g_scratch;  // guarded by g_tab_mu

int get_scratch(int device, size_t bytes, size_t heads, float** out, int** cnt) {
  std::lock_guard<std::mutex> lk(g_tab_mu);
  for (auto it = g_scratch.begin(); it != g_scratch.end(); ++it) {
    if (it->device == device) {
      if (it->bytes >= bytes && it->counters >= heads) {
        *out = it->ptr;
        *cnt = it->cnt;
        return NEOX_OK;
      }
      cudaError_t e = cudaDeviceSynchronize();  // in-flight kernels may still use it
      if (e != cudaSuccess) return cuda_fail(e);
      cudaFree(it->ptr);
      cudaFree(it->cnt);
      bytes = std::max(bytes, it->bytes);
      heads = std::max(heads, it->counters);
      g_scratch.erase(it);
      break;
    }
  }
  const size_t grown = std::max<size_t>(bytes, size_t(1) << 20);
  const size_t ncnt = std::max<size_t>(heads, 4096);
  float* ptr = nullptr;
  int* c = nullptr;
  cudaError_t e = cudaMalloc(&ptr, grown);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMalloc(&c, ncnt * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(c, 0, ncnt * sizeof(int));
  if (e != cudaSuccess) {
    cudaFree(ptr);
    if (c) cudaFree(c);
    return cuda_fail(e);
  }
  g_scratch.push_back(Scratch{device, grown, ptr, ncnt, c});
  *out = ptr;
  *cnt = c;
  return NEOX_OK;
}

// TMA view of the pre-rotated copy [B, S, H, 4, D] bf16 (slots: q hi, q lo, k hi, k lo)
// as 4-D {D, 4H, S, B} with the same {32, 1, 128, 1} box and swizzle as the qkv view.
int encode_rot_map(CUtensorMap* map, const void* rot, int B, int S, int H, int D) {
  if (!resolve_encode()) return cuda_fail(cudaErrorNotSupported);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(4) * H, static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(4) * H * D * 2,
                           static_cast<cuuint64_t>(S) * 4 * H * D * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(neox::kBlkCols), 1, static_cast<cuuint32_t>(neox::kRows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(rot), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return NEOX_OK;
}

// The separate pre-rotation pass: q' and k' of every row, split hi/lo, into the library's
// per-device scratch, then the tensor map the attention kernel loads them through.
template <int D>
int prerotate(Prepared& P, const void* qkv, cudaStream_t stream) {
  const neox::AttnParams& p = P.p;
  const int64_t rows = static_cast<int64_t>(p.B) * p.S * p.H;
  float* scratch = nullptr;
  int* counters = nullptr;
  int rc = get_scratch(P.device, static_cast<size_t>(rows) * 4 * D * 2, 1, &scratch, &counters);
  if (rc != NEOX_OK) return rc;
  uint16_t* rot = reinterpret_cast<uint16_t*>(scratch);
  if (p.r == 24) {
    const int64_t blocks = (rows + 127) / 128;
    if (blocks > 0x7FFFFFFF) return NEOX_ERR_INVALID_ARG;
    neox::rope_prerotate_r24_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(qkv), rot, p.cs, rows, p.S, p.H);
  } else {
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7FFFFFFF) return NEOX_ERR_INVALID_ARG;
    neox::rope_prerotate_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(qkv), rot, p.cs, rows, p.S, p.H, p.r);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  rc = encode_rot_map(&P.map_rot, rot, p.B, p.S, p.H, D);
  if (rc != NEOX_OK) return rc;
  P.pre = true;
  return NEOX_OK;
}

// After a wait timed out, heads may have been left half-counted: zero every counter.
void reset_decode_counters() {
  std::lock_guard<std::mutex> lk(g_tab_mu);
  for (auto& t : g_scratch) {
    int cur = 0;
    if (cudaGetDevice(&cur) == cudaSuccess && cur == t.device) cudaMemset(t.cnt, 0, t.counters * sizeof(int));
  }
}

int validate_decode(const void* qkv_new, const void* k_cache, const void* v_cache, const int* pos, int B, int H,
                    int Smax, int D, int r, float base, const void* out, const float* lse) {
  if (!qkv_new || !k_cache || !v_cache || !pos || !out || !lse) return NEOX_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Smax < 1 || B > 65535 || H > 65535) return NEOX_ERR_INVALID_ARG;
  if (D != 64 && D != 96 && D != 128) return NEOX_ERR_UNSUPPORTED_HEAD_DIM;
  if (r < 0 || r > D || (r & 1)) return NEOX_ERR_INVALID_ARG;
  if (!(base > 0.0f) || !std::isfinite(base)) return NEOX_ERR_INVALID_ARG;
  const uint64_t cache_elems = static_cast<uint64_t>(B) * H * Smax * D;
  if (cache_elems >= (1ull << 40)) return NEOX_ERR_INVALID_ARG;
  for (const void* ptr : {qkv_new, k_cache, v_cache, out})
    if (reinterpret_cast<uintptr_t>(ptr) & 15) return NEOX_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(lse) & 3) || (reinterpret_cast<uintptr_t>(pos) & 3)) return NEOX_ERR_MISALIGNED;
  const uint64_t bh = static_cast<uint64_t>(B) * H;
  const struct {
    const void* p;
    uint64_t n;
  } buf[6] = {{qkv_new, bh * 3 * D * 2}, {k_cache, cache_elems * 2}, {v_cache, cache_elems * 2},
              {pos, static_cast<uint64_t>(B) * 4}, {out, bh * D * 2}, {lse, bh * 4}};
  for (int i = 0; i < 6; ++i)
    for (int j = i + 1; j < 6; ++j) {
      if (i == 0 && j == 3) continue;  // the read-only inputs may share memory
      if (ranges_overlap(reinterpret_cast<uintptr_t>(buf[i].p), buf[i].n, reinterpret_cast<uintptr_t>(buf[j].p),
                         buf[j].n))
        return NEOX_ERR_INVALID_ARG;
    }
  return NEOX_OK;
}

template <int D, int H2>
int launch_decode_h2(const neox::DecodeParams& p, int ctas, cudaStream_t stream) {
  const int smem = neox::dec_smem_bytes(D);
  cudaError_t e = cudaFuncSetAttribute(neox::attn_decode_kernel<D, H2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return cuda_fail(e);
  neox::attn_decode_kernel<D, H2><<<ctas, neox::dec_threads(D), smem, stream>>>(p);
  e = cudaGetLastError();
  return e == cudaSuccess ? NEOX_OK : cuda_fail(e);
}

// rotary_dim 0, 8, 16, 24, 32: tile x row factorisation of the angle; others: the general path
template <int D>
int launch_decode(const neox::DecodeParams& p, int r, int ctas, cudaStream_t stream) {
  switch (r) {
    case 0: return launch_decode_h2<D, 0>(p, ctas, stream);
    case 8: return launch_decode_h2<D, 4>(p, ctas, stream);
    case 16: return launch_decode_h2<D, 8>(p, ctas, stream);
    case 24: return launch_decode_h2<D, 12>(p, ctas, stream);
    case 32: return launch_decode_h2<D, 16>(p, ctas, stream);
    default: return launch_decode_h2<D, -1>(p, ctas, stream);
  }
}

__global__ void selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    neox::mbar_init(neox::smem_u32(&bar), 1);
    abort_flag = 0;
    neox::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) neox::wait_phase(neox::smem_u32(&bar), 0, &abort_flag, limit_ns, 0xEE);
}

// ------------------------------------------------- allocation-free variant ----
// The cos/sin table of neox_attn_fwd_noalloc lives in this fixed device array instead of
// memory the library allocates: S * rotary_dim/2 entries at most (8 MiB).  Every GPU that
// loads the library holds it until the process exits.  In host code the name is only a
// host-side stand-in; the kernels get its device address from cudaGetSymbolAddress.
constexpr int64_t kNoAllocTableEntries = int64_t(1) << 20;
static __device__ __align__(256) float2 g_noalloc_table[kNoAllocTableEntries];

std::mutex g_noalloc_mu;
std::vector<float2*> g_noalloc_addr;  // per device ordinal; nullptr until looked up

// Device address of g_noalloc_table on `device`, which must be the current device.
int noalloc_table_address(int device, float2** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (static_cast<int>(g_noalloc_addr.size()) <= device) g_noalloc_addr.resize(device + 1, nullptr);
  if (!g_noalloc_addr[device]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_table);
    if (e != cudaSuccess) return cuda_fail(e);
    g_noalloc_addr[device] = static_cast<float2*>(ptr);
  }
  *out = g_noalloc_addr[device];
  return NEOX_OK;
}

// ------------------------------------------------------------------ backward ----
int validate_bwd(const void* qkv, const void* out, const float* lse, const void* dout, int B, int S, int H, int D,
                 int r, float base, const void* dqkv) {
  int rc = validate(qkv, B, S, H, D, r, base, out, lse);
  if (rc != NEOX_OK) return rc;
  if (!dout || !dqkv) return NEOX_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dout) & 15) || (reinterpret_cast<uintptr_t>(dqkv) & 15)) return NEOX_ERR_MISALIGNED;
  const uint64_t rows = static_cast<uint64_t>(B) * S * H;
  const uintptr_t g = reinterpret_cast<uintptr_t>(dout), d = reinterpret_cast<uintptr_t>(dqkv);
  const uint64_t gb = rows * D * 2, db = rows * 3 * D * 2;
  // dqkv is written: it may overlap no input; dout may alias nothing written either
  if (ranges_overlap(d, db, reinterpret_cast<uintptr_t>(qkv), db) ||
      ranges_overlap(d, db, reinterpret_cast<uintptr_t>(out), rows * D * 2) ||
      ranges_overlap(d, db, reinterpret_cast<uintptr_t>(lse), static_cast<uint64_t>(B) * H * S * 4) ||
      ranges_overlap(d, db, g, gb))
    return NEOX_ERR_INVALID_ARG;
  return NEOX_OK;
}

// TMA view of a row-major [B, S, H, D] bf16 tensor (dout): dims {D, H, S, B}, the same
// {32, 1, 128, 1} box and swizzle as the qkv view.
int encode_rows_map(CUtensorMap* map, const void* ptr, int B, int S, int H, int D) {
  if (!resolve_encode()) return cuda_fail(cudaErrorNotSupported);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                           static_cast<cuuint64_t>(S) * H * D * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(neox::kBlkCols), 1, static_cast<cuuint32_t>(neox::kRows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return NEOX_OK;
}

// The fp32 dq' accumulator [B, S, H, D] as a 3-D tensor {H*D, S, B}: a box of 32 columns
// of 128 query rows of one batch, 128-byte swizzle, for the backward's tensor reductions.
int encode_dq_map(CUtensorMap* map, const float* ptr, int B, int S, int H, int D) {
  if (!resolve_encode()) return cuda_fail(cudaErrorNotSupported);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(H) * D, static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(H) * D * 4, static_cast<cuuint64_t>(S) * H * D * 4};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(neox::kRows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult res = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return NEOX_OK;
}

template <int D>
int launch_bwd(const neox::BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tv, const CUtensorMap& tg,
               const CUtensorMap& tdq, const CUtensorMap& tdo, int num_sms, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.S * p.H;
  neox::attn_bwd_prep_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  const int smem = neox::bwd_smem_bytes(D);
  e = cudaFuncSetAttribute(neox::attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  // persistent: one CTA per SM (at most one per work item), later items from the work counter.
  // The main and dq kernels are launched as programmatic dependents of the kernel before
  // them (each waits in-kernel for that grid's completion before reading its results).
  const long long ctas = std::min<long long>(static_cast<long long>(p.nblk) * p.B * p.H, std::max(num_sms, 1));
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(neox::kBwdThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, neox::attn_bwd_kernel<D>, tq, tv, tg, tdq, tdo, p);
  if (e != cudaSuccess) return cuda_fail(e);
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, neox::attn_bwd_dq_kernel<D>, p);
  return e == cudaSuccess ? NEOX_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int neox_attn_fwd_ex(const void* qkv, int B, int S, int H, int D, int rotary_dim, float rotary_base, void* out,
                     float* lse, int rotation, void* stream) {
  try {
    if (rotation != NEOX_ROTATION_AUTO && rotation != NEOX_ROTATION_FUSED && rotation != NEOX_ROTATION_PRE)
      return NEOX_ERR_INVALID_ARG;
    const bool pre_ok = rotary_dim > 0 && (rotary_dim % 16 == 0 || rotary_dim == 24);
    if (rotation == NEOX_ROTATION_PRE && !pre_ok) return NEOX_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Prepared P;
    int rc = prepare(qkv, B, S, H, D, rotary_dim, rotary_base, out, lse, st, &P);
    if (rc != NEOX_OK) return rc;
    const bool pre = rotation == NEOX_ROTATION_PRE || (rotation == NEOX_ROTATION_AUTO && pre_ok && rotary_dim >= 64);
    if (pre) {
      switch (D) {
        case 64: rc = prerotate<64>(P, qkv, st); break;
        case 96: rc = prerotate<96>(P, qkv, st); break;
        default: rc = prerotate<128>(P, qkv, st); break;
      }
      if (rc != NEOX_OK) return rc;
    }
    switch (D) {
      case 64: return launch_ws<64>(P, st);
      case 96: return launch_ws<96>(P, st);
      default: return launch_ws<128>(P, st);
    }
  } catch (...) {
    return NEOX_ERR_CUDA;
  }
}

int neox_attn_fwd(const void* qkv, int B, int S, int H, int D, int rotary_dim, float rotary_base, void* out, float* lse,
                  void* stream) {
  return neox_attn_fwd_ex(qkv, B, S, H, D, rotary_dim, rotary_base, out, lse, NEOX_ROTATION_AUTO, stream);
}

int neox_attn_fwd_alibi(const void* qkv, int B, int S, int H, int D, void* out, float* lse, void* stream) {
  try {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Prepared P;
    // no rotary dims (so no table): the base is only validated, never used
    int rc = prepare(qkv, B, S, H, D, 0, 10000.0f, out, lse, st, &P);
    if (rc != NEOX_OK) return rc;
    int r2 = 0;
    switch (D) {
      case 64: r2 = neox::launch_attn_ws_alibi<64>(P.map, P.p, P.dev.num_sms, st, &g_last_cuda_error); break;
      case 96: r2 = neox::launch_attn_ws_alibi<96>(P.map, P.p, P.dev.num_sms, st, &g_last_cuda_error); break;
      default: r2 = neox::launch_attn_ws_alibi<128>(P.map, P.p, P.dev.num_sms, st, &g_last_cuda_error); break;
    }
    return r2 == 0 ? NEOX_OK : NEOX_ERR_CUDA;
  } catch (...) {
    return NEOX_ERR_CUDA;
  }
}

int neox_attn_qkv_proj(const void* x, const void* w, const void* bias, int B, int S, int hidden, int H, int D,
                       int rotary_dim, float rotary_base, void* qkv, void* stream) {
  try {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = validate_proj(x, w, bias, B, S, hidden, H, D, rotary_dim, rotary_base, qkv);
    if (rc != NEOX_OK) return rc;
    int device = 0;
    DeviceInfo dev;
    if ((rc = current_device(&device, &dev)) != NEOX_OK) return rc;
    neox::ProjParams p{};
    p.bias = static_cast<const uint16_t*>(bias);
    p.cs = nullptr;
    if (rotary_dim > 0 && (rc = get_table(device, S, rotary_dim, rotary_base, st, &p.cs)) != NEOX_OK) return rc;
    p.M = B * S;
    p.N = 3 * H * D;
    p.K = hidden;
    p.S = S;
    p.D = D;
    p.r = rotary_dim;
    p.num_m = (p.M + 127) / 128;
    const int NT = neox::proj_tile_n(D);
    p.num_tiles = p.num_m * ((p.N + NT - 1) / NT);
    p.wait_limit_ns = neox::kWaitLimitNs;
    CUtensorMap mx, mw, mo;
    if ((rc = encode_2d(&mx, x, hidden, p.M, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) != NEOX_OK) return rc;
    if ((rc = encode_2d(&mw, w, p.N, hidden, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != NEOX_OK) return rc;
    if ((rc = encode_2d(&mo, qkv, p.N, p.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) != NEOX_OK) return rc;
    return neox::launch_qkv_proj(mx, mw, mo, p, dev.num_sms, st, &g_last_cuda_error) == 0 ? NEOX_OK : NEOX_ERR_CUDA;
  } catch (...) {
    return NEOX_ERR_CUDA;
  }
}

int neox_attn_fwd_simple(const void* qkv, int B, int S, int H, int D, int rotary_dim, float rotary_base, void* out,
                         float* lse, void* stream) {
  try {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Prepared P;
    int rc = prepare(qkv, B, S, H, D, rotary_dim, rotary_base, out, lse, st, &P);
    if (rc != NEOX_OK) return rc;
    switch (D) {
      case 64: return launch_simple<64>(P, st);
      case 96: return launch_simple<96>(P, st);
      default: return launch_simple<128>(P, st);
    }
  } catch (...) {
    return NEOX_ERR_CUDA;
  }
}

int neox_attn_decode(const void* qkv_new, void* k_cache, void* v_cache, const int* pos, int B, int H, int Smax,
                     int D, int rotary_dim, float rotary_base, void* out, float* lse, void* stream_) {
  try {
    int rc = validate_decode(qkv_new, k_cache, v_cache, pos, B, H, Smax, D, rotary_dim, rotary_base, out, lse);
    if (rc != NEOX_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int device = 0;
    DeviceInfo dev;
    rc = current_device(&device, &dev);
    if (rc != NEOX_OK) return rc;
    const float2* cs = nullptr;
    if (rotary_dim > 0) {  // rows 0..127 (row factors) and every position < Smax
      rc = get_table(device, std::max(Smax, neox::kRows), rotary_dim, rotary_base, stream, &cs);
      if (rc != NEOX_OK) return rc;
    }
    // one CTA per SM, each with an equal contiguous range of the B*H*ceil(Smax/128) key
    // tiles; a head's tiles fall into the ranges of at most runs_per_head CTAs (every range
    // but the first and last inside the head covers at least N / G of its tiles)
    const int tiles = (Smax + neox::kRows - 1) / neox::kRows;
    const long long heads = static_cast<long long>(B) * H;
    const long long N = heads * tiles;
    const int ctas = static_cast<int>(std::min<long long>(dev.num_sms, N));
    const long long q = N / ctas;
    const int runs = tiles >= 2 ? static_cast<int>(std::min<long long>(tiles, (tiles - 2) / q + 2)) : 1;
    float* part = nullptr;
    int* counters = nullptr;
    rc = get_scratch(device, static_cast<size_t>(heads) * runs * (D + 2) * sizeof(float), static_cast<size_t>(heads),
                     &part, &counters);
    if (rc != NEOX_OK) return rc;
    neox::DecodeParams p{};
    p.qkv_new = static_cast<const uint16_t*>(qkv_new);
    p.k_cache = static_cast<uint16_t*>(k_cache);
    p.v_cache = static_cast<uint16_t*>(v_cache);
    p.pos = pos;
    p.cs = cs;
    p.part = part;
    p.counters = counters;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.Smax = Smax;
    p.r = rotary_dim;
    p.tiles_per_head = tiles;
    p.runs_per_head = runs;
    p.total_tiles = N;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    p.wait_limit_ns = neox::kWaitLimitNs;
    switch (D) {
      case 64: return launch_decode<64>(p, rotary_dim, ctas, stream);
      case 96: return launch_decode<96>(p, rotary_dim, ctas, stream);
      default: return launch_decode<128>(p, rotary_dim, ctas, stream);
    }
  } catch (...) {
    return NEOX_ERR_CUDA;
  }
}

int neox_attn_bwd(const void* qkv, const void* out, const float* lse, const void* dout, int B, int S, int H, int D,
                  int rotary_dim, float rotary_base, void* dqkv, void* stream_) {
  try {
    int rc = validate_bwd(qkv, out, lse, dout, B, S, H, D, rotary_dim, rotary_base, dqkv);
    if (rc != NEOX_OK) return rc;
    const long long nblk = (static_cast<long long>(S) + neox::kRows - 1) / neox::kRows;
    if (nblk * B * H > 0x7FFFFFFFll) return NEOX_ERR_INVALID_ARG;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int device = 0;
    DeviceInfo dev;
    rc = current_device(&device, &dev);
    if (rc != NEOX_OK) return rc;
    const float2* cs = nullptr;
    if (rotary_dim > 0) {
      rc = get_table(device, S, rotary_dim, rotary_base, stream, &cs);
      if (rc != NEOX_OK) return rc;
    }
    // scratch: the fp32 dq' accumulator [B,S,H,D], delta [B,H,S], then (256-byte aligned)
    // the rotated copy of qkv [B,S,H,3,D] bf16
    const size_t rows = static_cast<size_t>(B) * S * H;
    const size_t rot_off = (rows * D * sizeof(float) + rows * sizeof(float) + 255) / 256 * 256;
    float* scratch = nullptr;
    int* counters = nullptr;
    rc = get_scratch(device, rot_off + rows * 3 * D * 2, 1, &scratch, &counters);
    if (rc != NEOX_OK) return rc;
    uint16_t* qkv_rot = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(scratch) + rot_off);
    CUtensorMap tq, tv, tg;  // rotated q', k'; v from the input; dout
    rc = encode_qkv_map(&tq, qkv_rot, B, S, H, D);
    if (rc != NEOX_OK) return rc;
    rc = encode_qkv_map(&tv, qkv, B, S, H, D);
    if (rc != NEOX_OK) return rc;
    rc = encode_rows_map(&tg, dout, B, S, H, D);
    if (rc != NEOX_OK) return rc;
    CUtensorMap tdq;  // the fp32 dq' accumulator at the start of the scratch
    rc = encode_dq_map(&tdq, scratch, B, S, H, D);
    if (rc != NEOX_OK) return rc;
    CUtensorMap tdo;  // dqkv, for the tensor stores of dk and dv
    rc = encode_qkv_map(&tdo, dqkv, B, S, H, D);
    if (rc != NEOX_OK) return rc;
    neox::BwdParams p{};
    p.qkv = static_cast<const uint16_t*>(qkv);
    p.out = static_cast<const uint16_t*>(out);
    p.lse = lse;
    p.dout = static_cast<const uint16_t*>(dout);
    p.dqkv = static_cast<uint16_t*>(dqkv);
    p.qkv_rot = qkv_rot;
    p.dq_acc = scratch;
    p.delta = scratch + rows * D;
    p.cs = cs;
    p.B = B;
    p.S = S;
    p.H = H;
    p.r = rotary_dim;
    p.nblk = static_cast<int>(nblk);
    // about 48 MB of Q and dO per group of heads (half of L2), at least one head
    p.heads_per_group = static_cast<int>(std::max<long long>(
        1, std::min<long long>(static_cast<long long>(B) * H, (48ll << 20) / (static_cast<long long>(S) * D * 4))));
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    p.wait_limit_ns = neox::kWaitLimitNs;
    switch (D) {
      case 64: return launch_bwd<64>(p, tq, tv, tg, tdq, tdo, dev.num_sms, stream);
      case 96: return launch_bwd<96>(p, tq, tv, tg, tdq, tdo, dev.num_sms, stream);
      default: return launch_bwd<128>(p, tq, tv, tg, tdq, tdo, dev.num_sms, stream);
    }
  } catch (...) {
    return NEOX_ERR_CUDA;
  }
}

int neox_attn_get_device_error(void) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, neox::g_device_error, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v == 0) return NEOX_OK;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(neox::g_device_error, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v & neox::kErrTimeout) reset_decode_counters();
  if (v & neox::kErrTimeout) return NEOX_ERR_DEVICE_TIMEOUT;
  return (v & neox::kErrRange) ? NEOX_ERR_DEVICE_RANGE : NEOX_ERR_DEVICE_BAD_POSITION;
}

const char* neox_attn_status_string(int status) {
  switch (status) {
    case NEOX_OK: return "ok";
    case NEOX_ERR_INVALID_ARG: return "invalid argument";
    case NEOX_ERR_UNSUPPORTED_HEAD_DIM: return "unsupported head dim (64, 96 or 128)";
    case NEOX_ERR_MISALIGNED: return "misaligned pointer";
    case NEOX_ERR_CUDA: return "CUDA error";
    case NEOX_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case NEOX_ERR_NO_DEVICE_SUPPORT: return "device is not compute capability 10.3";
    case NEOX_ERR_TOO_LARGE: return "S * rotary_dim/2 exceeds the fixed 1048576-entry table of neox_attn_fwd_noalloc";
    case NEOX_ERR_DEVICE_BAD_POSITION: return "a decode position was outside [0, Smax)";
    case NEOX_ERR_DEVICE_RANGE: return "a rotated query/key value exceeded the fp16 operand range (65504)";
    default: return "unknown status";
  }
}

int neox_attn_last_cuda_error(void) { return g_last_cuda_error; }

void neox_attn_release(void) {
  std::lock_guard<std::mutex> lk(g_tab_mu);
  if (!g_tables.empty()) {
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& t : g_tables) {
      cudaSetDevice(t.device);
      cudaDeviceSynchronize();
      cudaFree(t.ptr);
    }
    cudaSetDevice(cur);
    g_tables.clear();
  }
  if (!g_scratch.empty()) {
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& t : g_scratch) {
      cudaSetDevice(t.device);
      cudaDeviceSynchronize();
      cudaFree(t.ptr);
      cudaFree(t.cnt);
    }
    cudaSetDevice(cur);
    g_scratch.clear();
  }
}

int neox_attn_selftest_wait_timeout(int64_t timeout_ns, void* stream) {
  if (timeout_ns < 1000 || timeout_ns > 1000000000) return NEOX_ERR_INVALID_ARG;
  int dev = 0;
  DeviceInfo info;
  int rc = current_device(&dev, &info);
  if (rc != NEOX_OK) return rc;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(timeout_ns));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? NEOX_OK : cuda_fail(e);
}

int neox_attn_version(void) { return 100; }

int neox_attn_fwd_noalloc(const void* qkv, int B, int S, int H, int D, int rotary_dim, float rotary_base, void* out,
                          float* lse, void* stream) {
  try {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = validate(qkv, B, S, H, D, rotary_dim, rotary_base, out, lse);
    if (rc != NEOX_OK) return rc;
    if (static_cast<int64_t>(S) * (rotary_dim / 2) > kNoAllocTableEntries) return NEOX_ERR_TOO_LARGE;
    Prepared P;
    rc = current_device(&P.device, &P.dev);
    if (rc != NEOX_OK) return rc;
    float2* table = nullptr;
    if (rotary_dim > 0) {
      rc = noalloc_table_address(P.device, &table);
      if (rc != NEOX_OK) return rc;
    }
    rc = encode_qkv_map(&P.map, qkv, B, S, H, D);
    if (rc != NEOX_OK) return rc;
    neox::AttnParams& p = P.p;
    p.cs = table;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.B = B;
    p.S = S;
    p.H = H;
    p.r = rotary_dim;
    p.r16 = (rotary_dim + 15) / 16 * 16;
    p.side_cols = rotary_dim > 0 ? (p.r16 + 31) / 32 * 32 : 0;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    p.num_units = 0;
    p.wait_limit_ns = neox::kWaitLimitNs;
    if (rotary_dim > 0) {
      // rebuilt on every call, rows [0, S): the array keeps whatever the last call left
      const int h = rotary_dim / 2;
      const int64_t n = static_cast<int64_t>(S) * h;
      const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 65535));
      neox::rope_table_kernel<<<blocks, 256, 0, st>>>(table, S, h, rotary_dim, static_cast<double>(rotary_base));
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e);
    }
    switch (D) {
      case 64: return launch_ws<64>(P, st);
      case 96: return launch_ws<96>(P, st);
      default: return launch_ws<128>(P, st);
    }
  } catch (...) {
    return NEOX_ERR_CUDA;
  }
}

}  // extern "C"
