// The cache write that precedes a decode step (see include/mla_kv_pack.h):
// the new tokens' latent rows, quantised to e4m3 (or copied for a bf16
// cache), scattered through the page table.  One warp per 4 rows: a row is
// 72 chunks of 16 bytes (8 bf16 values), so each lane reads and writes 9
// chunks, all loads first; the kernel streams at close to the copy rate of
// HBM.
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
constexpr int kRowsPerWarp = 4;            // 4 x 72 chunks = 9 per lane
constexpr int kPer = kRowsPerWarp * kChunks / 32;
constexpr int kWarps = 8;                  // warps per block

__device__ __forceinline__ uint4 ldg_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(reinterpret_cast<uint64_t>(p)));
  return v;
}

// Rounding x / scale to e4m3 without a division.  With r = fp32(1 /
// scale), x * r is within 2^-23 (relative) of x / scale; r_dn = fp32(r (1 -
// 2^-20)) and r_up = fp32(r (1 + 2^-20)) put x * r_dn and x * r_up on either
// side of x / scale.  When both round to the same code, so does the
// quotient (rounding is monotone); otherwise an e4m3 midpoint lies within
// about 2^-20 of it (rare) and e4m3_exact decides.
//
// e4m3_exact: the code nearest to x / scale.  m is the midpoint nearest q =
// x * r (the only one that x / scale can lie across), and x - m * scale,
// formed by one fma, has exactly the sign of x / scale - m for scale > 0
// (one rounding never changes a sign; only an exact zero is zero).  A value
// just past m on that side (or m itself on a tie, which the conversion
// sends to the even code) is then converted.  In e4m3's normal range (2^-6
// .. 448: 3 mantissa bits) the midpoints are the fp32 numbers whose
// mantissa bits 19..0 are 0x80000; the subnormal range [0, 2^-6) has the
// grid step of the binade [2^-6, 2^-5) (2^-9), so |q| + 2^-6 locates its
// midpoint there (g may round by at most 2^-30, which can move it across
// a code value but never across a midpoint, and the midpoint found on
// either side of a code value still separates x / scale from the code it
// does not round to).
__device__ __noinline__ uint32_t e4m3_exact(float x, float scale, float inv_scale) {
  const float q = __fmul_rn(x, inv_scale);
  const float shift = fabsf(q) < 0x1p-6f ? 0x1p-6f : 0.f;
  const float g = fabsf(q) + shift;
  const float mi = __uint_as_float((__float_as_uint(g) & ~0xFFFFFu) | 0x80000u);
  const float m = copysignf(mi - shift, q);
  const float t = __fmaf_rn(-m, scale, x);
  const float v = t > 0.f ? m + fabsf(m) * 0x1p-10f : (t < 0.f ? m - fabsf(m) * 0x1p-10f : m);
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

struct E4m3Scale {
  float scale, r, r_dn, r_up;
};

// e4m3 codes of two bf16 values (packed as in memory, the lower address in
// the low half) times a factor: the lower address goes to the low byte
__device__ __forceinline__ uint32_t cvt2(uint32_t bf2, float f) {
  const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bf2));
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(x.x, f), __fmul_rn(x.y, f)), __NV_SATFINITE, __NV_E4M3));
}

// the codes nearest to x / scale of the 8 bf16 values of a 16-byte chunk
__device__ __forceinline__ uint2 e4m3x8(uint4 v, const E4m3Scale& k) {
  const uint2 dn = make_uint2(cvt2(v.x, k.r_dn) | (cvt2(v.y, k.r_dn) << 16), cvt2(v.z, k.r_dn) | (cvt2(v.w, k.r_dn) << 16));
  const uint2 up = make_uint2(cvt2(v.x, k.r_up) | (cvt2(v.y, k.r_up) << 16), cvt2(v.z, k.r_up) | (cvt2(v.w, k.r_up) << 16));
  if (dn.x == up.x && dn.y == up.y) return dn;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    c[e] = e4m3_exact(x.x, k.scale, k.r) | (e4m3_exact(x.y, k.scale, k.r) << 8);
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

}  // namespace

namespace mla {

template <bool kF8>
__global__ void __launch_bounds__(kWarps * 32)
    mla_kv_pack_kernel(const uint4* __restrict__ rows, const int32_t* __restrict__ page_table,
                       const int32_t* __restrict__ seq_lens, int batch, int num_new, int num_pages, int max_pages,
                       int stride, E4m3Scale sc, uint8_t* __restrict__ cache, int32_t* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nrows = static_cast<int64_t>(batch) * num_new;
  const int64_t row0 = (static_cast<int64_t>(blockIdx.x) * kWarps + warp) * kRowsPerWarp;
  if (row0 >= nrows) return;
  // lanes 0..3 find the cache slot of rows row0 .. row0 + 3 (-1: not written)
  int64_t my_slot = -1;
  if (lane < kRowsPerWarp && row0 + lane < nrows) {
    const int64_t row = row0 + lane;
    const int b = static_cast<int>(row / num_new), i = static_cast<int>(row % num_new);
    const int L = seq_lens[b];
    if (L < num_new || L > max_pages * kPageRows) {
      atomicOr(status, MLA_DEV_BAD_SEQ_LEN);
    } else {
      const int t = L - num_new + i;  // position of the token in its sequence
      const int page = page_table[static_cast<int64_t>(b) * stride + t / kPageRows];
      if (page < 0 || page >= num_pages) atomicOr(status, MLA_DEV_BAD_PAGE_ID);
      else my_slot = static_cast<int64_t>(page) * kPageRows + t % kPageRows;
    }
  }
  // chunk c = lane + 32 k of the warp's 4 rows (they are contiguous in the
  // input): row c / 72, chunk c % 72 of it; all loads first
  const uint4* src = rows + row0 * kChunks;
  const int64_t avail = (nrows - row0) * kChunks;  // chunks of this warp that exist
  uint4 v[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    if (lane + 32 * k < avail) v[k] = ldg_nc_v4(src + lane + 32 * k);
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int c = lane + 32 * k;
    const int rq = c / kChunks, cc = c % kChunks;
    const int64_t sl = __shfl_sync(0xffffffffu, my_slot, rq);  // the slot of this chunk's row
    if (c >= avail || sl < 0) continue;
    if constexpr (kF8) {
      reinterpret_cast<uint2*>(cache + sl * kRowVals)[cc] = e4m3x8(v[k], sc);  // 8 codes per chunk
    } else {
      reinterpret_cast<uint4*>(cache + sl * kRowVals * 2)[cc] = v[k];
    }
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
  const int64_t blocks = (n + kWarps * kRowsPerWarp - 1) / (kWarps * kRowsPerWarp);
  if (blocks > INT_MAX) return MLA_ERR_INVALID_ARG;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (major != 10 || minor != 3) return MLA_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  E4m3Scale sc;
  sc.scale = f8 ? kv_scale : 1.0f;
  sc.r = f8 ? 1.0f / kv_scale : 1.0f;  // IEEE fp32 division, once per call
  sc.r_dn = sc.r * (1.0f - 0x1p-20f);
  sc.r_up = sc.r * (1.0f + 0x1p-20f);
  const uint4* src = static_cast<const uint4*>(rows);
  uint8_t* dst = static_cast<uint8_t*>(kv_cache);
  if (f8)
    mla::mla_kv_pack_kernel<true><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(
        src, page_table, seq_lens, d->batch, d->num_new, d->num_pages, d->max_pages_per_req, d->page_table_stride,
        sc, dst, status);
  else
    mla::mla_kv_pack_kernel<false><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(
        src, page_table, seq_lens, d->batch, d->num_new, d->num_pages, d->max_pages_per_req, d->page_table_stride,
        sc, dst, status);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
