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

// Rounding x / scale to e4m3 without a division.  q = x * r, r = fp32(1 /
// scale), is within 2^-23 (relative) of x / scale, so both round to the same
// code unless an e4m3 midpoint lies within that distance of q.  In e4m3's
// normal range (2^-6 .. 448: 3 mantissa bits) the midpoints are the fp32
// numbers whose mantissa bits 19..0 are 0x80000, and q is near one when
// those bits are within 8 units of it (2^-23 relative is at most 2 units).
// Nonzero q below 2^-6 (the subnormal grid) are always sent to the exact
// path; zero converts exactly.
__device__ __forceinline__ bool needs_exact(float q) {
  const uint32_t b = __float_as_uint(q) & 0x7FFFFFFFu;
  return (b - 1u) < 0x3C7FFFFFu || ((b + 8u) & 0xFFFF0u) == 0x80000u;
}

// The code nearest to x / scale: m is the midpoint nearest q (the only one
// that x / scale can lie across), and x - m * scale, formed by one fma, has
// exactly the sign of x / scale - m for scale > 0 (one rounding never
// changes a sign; only an exact zero is zero).  A value just past m on that
// side (or m itself on a tie, which the conversion sends to the even code)
// is then converted.  The subnormal range [0, 2^-6) has the grid step of the
// binade [2^-6, 2^-5) (2^-9), so |q| + 2^-6 locates its midpoint there.
__device__ __noinline__ uint32_t e4m3_exact(float x, float scale, float inv_scale) {
  const float q = __fmul_rn(x, inv_scale);
  const float shift = fabsf(q) < 0x1p-6f ? 0x1p-6f : 0.f;
  // g may round (by at most 2^-30), which can only move it across a code
  // value, never across a midpoint; the midpoint found on either side of a
  // code value still lies between x / scale and the code it does not round to
  const float g = fabsf(q) + shift;
  const float mi = __uint_as_float((__float_as_uint(g) & ~0xFFFFFu) | 0x80000u);
  const float m = copysignf(mi - shift, q);
  const float t = __fmaf_rn(-m, scale, x);
  const float v = t > 0.f ? m + fabsf(m) * 0x1p-10f : (t < 0.f ? m - fabsf(m) * 0x1p-10f : m);
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// e4m3 codes of the 8 bf16 values of a 16-byte chunk divided by kv_scale:
// one rounding of x * (1 / kv_scale) each, then, for a chunk holding a value
// that needs it (rare), the exact code of every value
__device__ __forceinline__ uint2 e4m3x8(uint4 v, float inv_scale, float scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
  bool flag = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    const float q0 = __fmul_rn(x.x, inv_scale), q1 = __fmul_rn(x.y, inv_scale);
    flag |= needs_exact(q0) | needs_exact(q1);
    c[k] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(q0, q1), __NV_SATFINITE, __NV_E4M3));
  }
  if (flag) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      c[k] = e4m3_exact(x.x, scale, inv_scale) | (e4m3_exact(x.y, scale, inv_scale) << 8);
    }
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
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
    // the code nearest to x / kv_scale (see e4m3x8)
    uint2* dst = reinterpret_cast<uint2*>(cache + slot * kRowVals);  // 8 codes per chunk
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (lane + 32 * k < kChunks) dst[lane + 32 * k] = e4m3x8(v[k], inv_scale, scale);
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
