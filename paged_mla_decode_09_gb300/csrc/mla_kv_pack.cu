// The cache write that precedes a decode step (see include/mla_kv_pack.h):
// the new tokens' latent rows, quantised to e4m3 (or copied for a bf16
// cache), scattered through the page table.  One warp per row; a row is
// 72 chunks of 16 bytes (8 bf16 values) read once and written once, so the
// kernel streams at the copy rate of HBM and does no other work.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>

#include "mla_kv_pack.h"

namespace {

constexpr int kRowVals = 576;              // c_kv (512) | k_pe (64)
constexpr int kPageRows = 64;              // tokens per page
constexpr int kChunks = kRowVals * 2 / 16;  // 16-byte chunks of a bf16 row
constexpr int kWarps = 8;                  // rows per block

__device__ __forceinline__ uint4 ldg_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(reinterpret_cast<uint64_t>(p)));
  return v;
}

// e4m3 code nearest to x / scale when x * inv_scale * (1 - 2^-20) rounds to
// code ca and x * inv_scale * (1 + 2^-20) to code cb != ca: the two codes are
// neighbours and the quotient lies on one side of their midpoint m, or on
// it.  x - m * scale has the sign of (x / scale - m) for scale > 0, and one
// fma gives that sign exactly (one rounding never changes a sign; only an
// exact zero is zero).  A tie goes to the even code (mantissa bit 0 clear).
__device__ __noinline__ uint32_t e4m3_resolve(uint32_t ca, uint32_t cb, float x, float scale) {
  const float va = __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(ca), __NV_E4M3)));
  const float vb = __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(cb), __NV_E4M3)));
  const float m = 0.5f * (va + vb);  // exact: neighbouring e4m3 values have at most 5 significant bits together
  const float t = __fmaf_rn(-m, scale, x);
  if (t > 0.f) return va > vb ? ca : cb;
  if (t < 0.f) return va > vb ? cb : ca;
  return (ca & 1u) ? cb : ca;
}

// e4m3 codes of two bf16 values (packed as in memory, the lower address in
// the low half) divided by kv_scale: the nearest code to the exact quotient
// x / kv_scale, ties to even, saturated to +-448.  The quotient is
// bracketed without a division: with r = fp32(1 / kv_scale), x * r is
// within 2^-23 (relative) of x / kv_scale, so x * r * (1 -+ 2^-20) lie on
// either side of it; when both round to the same code, so does the
// quotient (rounding is monotone), and otherwise (a midpoint within about
// 2^-20 of the quotient: rare) e4m3_resolve decides.
__device__ __forceinline__ uint32_t e4m3x2(uint32_t bf2, float inv_scale, float scale) {
  const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bf2));
  const float q0 = __fmul_rn(x.x, inv_scale), q1 = __fmul_rn(x.y, inv_scale);
  constexpr float kDown = 1.0f - 0x1p-20f, kUp = 1.0f + 0x1p-20f;
  const uint32_t lo = static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(q0, kDown), __fmul_rn(q1, kDown)), __NV_SATFINITE, __NV_E4M3));
  const uint32_t hi = static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(q0, kUp), __fmul_rn(q1, kUp)), __NV_SATFINITE, __NV_E4M3));
  if (lo == hi) return lo;
  const uint32_t c0 = (lo & 0xFFu) == (hi & 0xFFu) ? (lo & 0xFFu) : e4m3_resolve(lo & 0xFFu, hi & 0xFFu, x.x, scale);
  const uint32_t c1 = (lo >> 8) == (hi >> 8) ? (lo >> 8) : e4m3_resolve(lo >> 8, hi >> 8, x.y, scale);
  return c0 | (c1 << 8);
}

}  // namespace

namespace mla {

template <bool kF8>
__global__ void __launch_bounds__(kWarps * 32)
    mla_kv_pack_kernel(const uint4* __restrict__ rows, const int32_t* __restrict__ page_table,
                       const int32_t* __restrict__ seq_lens, int batch, int num_new, int num_pages, int max_pages,
                       int stride, float inv_scale, float scale, uint8_t* __restrict__ cache, int32_t* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (row >= static_cast<int64_t>(batch) * num_new) return;
  const int b = static_cast<int>(row / num_new), i = static_cast<int>(row % num_new);
  const int L = seq_lens[b];
  if (L < num_new || L > max_pages * kPageRows) {
    if (lane == 0) atomicOr(status, MLA_DEV_BAD_SEQ_LEN);
    return;
  }
  const int t = L - num_new + i;  // position of the token in its sequence
  const int page = page_table[static_cast<int64_t>(b) * stride + t / kPageRows];
  if (page < 0 || page >= num_pages) {
    if (lane == 0) atomicOr(status, MLA_DEV_BAD_PAGE_ID);
    return;
  }
  const int64_t slot = static_cast<int64_t>(page) * kPageRows + t % kPageRows;
  const uint4* src = rows + row * kChunks;
  // all loads of the lane first (chunks lane, lane + 32 and, for lanes
  // 0-7, lane + 64), then the conversions and stores
  constexpr int kPer = (kChunks + 31) / 32;
  uint4 v[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    if (lane + 32 * k < kChunks) v[k] = ldg_nc_v4(src + lane + 32 * k);
  if constexpr (kF8) {
    uint2* dst = reinterpret_cast<uint2*>(cache + slot * kRowVals);  // 8 codes per chunk
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (lane + 32 * k >= kChunks) break;
      const uint32_t lo = e4m3x2(v[k].x, inv_scale, scale) | (e4m3x2(v[k].y, inv_scale, scale) << 16);
      const uint32_t hi = e4m3x2(v[k].z, inv_scale, scale) | (e4m3x2(v[k].w, inv_scale, scale) << 16);
      dst[lane + 32 * k] = make_uint2(lo, hi);
    }
  } else {
    uint4* dst = reinterpret_cast<uint4*>(cache + slot * kRowVals * 2);
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (lane + 32 * k < kChunks) dst[lane + 32 * k] = v[k];
  }
}

}  // namespace mla

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int mla_kv_pack(const mla_kv_pack_dims* d, const void* rows, const int32_t* page_table,
                           const int32_t* seq_lens, float kv_scale, void* kv_cache, int32_t* status, void* stream) {
  if (!d || !rows || !page_table || !seq_lens || !kv_cache || !status) return MLA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->num_new < 1 || d->num_pages < 1 || d->max_pages_per_req < 1 ||
      d->page_table_stride < d->max_pages_per_req)
    return MLA_ERR_INVALID_ARG;
  if (d->kv_dtype != MLA_KV_BF16 && d->kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_UNSUPPORTED;
  const bool f8 = d->kv_dtype == MLA_KV_FP8_E4M3;
  // a normal, finite scale whose reciprocal is finite too
  if (f8 && !(kv_scale >= FLT_MIN && std::isfinite(kv_scale) && std::isfinite(1.0f / kv_scale)))
    return MLA_ERR_INVALID_ARG;
  if (!aligned(rows, 16) || !aligned(kv_cache, 16) || !aligned(page_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(status, 4))
    return MLA_ERR_ALIGNMENT;
  if (static_cast<int64_t>(d->max_pages_per_req) * kPageRows > INT_MAX) return MLA_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(d->batch) * d->num_new;
  const int64_t blocks = (n + kWarps - 1) / kWarps;
  if (blocks > INT_MAX) return MLA_ERR_INVALID_ARG;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (major != 10 || minor != 3) return MLA_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float inv_scale = f8 ? 1.0f / kv_scale : 1.0f;  // IEEE fp32 division, once per call
  const uint4* src = static_cast<const uint4*>(rows);
  uint8_t* dst = static_cast<uint8_t*>(kv_cache);
  if (f8)
    mla::mla_kv_pack_kernel<true><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(
        src, page_table, seq_lens, d->batch, d->num_new, d->num_pages, d->max_pages_per_req, d->page_table_stride,
        inv_scale, kv_scale, dst, status);
  else
    mla::mla_kv_pack_kernel<false><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(
        src, page_table, seq_lens, d->batch, d->num_new, d->num_pages, d->max_pages_per_req, d->page_table_stride,
        inv_scale, kv_scale, dst, status);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
