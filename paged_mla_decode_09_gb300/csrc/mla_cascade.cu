// Cascade decode over a shared prefix (see include/mla_cascade.h): a prefix
// pass with several requests' query rows per row block, a suffix pass, and a
// log-sum-exp merge.  The two passes are the paged decode of mla_decode.h,
// called with rearranged dimensions on the caller's buffers.
//
// Workspace: [status | prefix lengths [B] | suffix lengths [B] | prefix out
// (fp32 [B][q_len][H][512]) | prefix lse (fp32 [B][q_len][H]) | suffix out
// (fp32, same shape) | decode workspace (shared by the passes, which run in
// order on one stream)].  Both passes write fp32 results, so that the only
// rounding to bf16 is the merged output's, as in the plain decode's combine.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>

#include "mla_cascade.h"
#include "mla_decode.h"
#include "mla_internal.h"

namespace {

constexpr int kPageRows = 64;
constexpr int kDL = 512;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

namespace mla {

// one block per request: its prefix and suffix lengths, and a check that
// its prefix columns name the same pages as request 0's
__global__ void __launch_bounds__(128)
    mla_cascade_prep_kernel(const int32_t* __restrict__ page_table, const int32_t* __restrict__ seq_lens,
                            int stride, int prefix_pages, int q_len, int32_t* __restrict__ len_pre,
                            int32_t* __restrict__ len_suf, int32_t* status) {
  const int b = blockIdx.x;
  bool same = true;
  for (int c = threadIdx.x; c < prefix_pages; c += blockDim.x)
    same &= page_table[static_cast<int64_t>(b) * stride + c] == page_table[c];
  if (!__syncthreads_and(same) && threadIdx.x == 0) atomicOr(status, MLA_DEV_BAD_PREFIX);
  if (threadIdx.x == 0) {
    const int pre = prefix_pages * kPageRows;
    const int L = seq_lens[b];
    if (L < pre + q_len) atomicOr(status, MLA_DEV_BAD_SEQ_LEN);
    len_pre[b] = pre;
    len_suf[b] = L - pre;  // the suffix pass flags and clamps a bad length
  }
}

__global__ void mla_cascade_or_status_kernel(const int32_t* __restrict__ pass_status, int32_t* status) {
  const int32_t s = pass_status[0];
  if (s != 0) atomicOr(status, s);
}

// one warp per query row: out = (e^lp op + e^ls os) / (e^lp + e^ls),
// lse = ln(e^lp + e^ls), from the two passes' fp32 results; the suffix lse
// is in lse and is replaced
__global__ void __launch_bounds__(256)
    mla_cascade_merge_kernel(const float* __restrict__ out_pre, const float* __restrict__ lse_pre,
                             const float* __restrict__ out_suf, __nv_bfloat16* out, float* lse, int64_t rows) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const float lp = lse_pre[r], ls = lse[r];
  const float m = fmaxf(lp, ls);
  const float wp = (lp == -INFINITY) ? 0.f : __expf(lp - m);
  const float ws = (ls == -INFINITY) ? 0.f : __expf(ls - m);
  const float z = wp + ws;
  const float ap = z > 0.f ? wp / z : 0.f, as = z > 0.f ? ws / z : 0.f;
  // 16 values per lane: four float4 of each pass, two 16-byte bf16 chunks out
  const float4* src_p = reinterpret_cast<const float4*>(out_pre + r * kDL);
  const float4* src_s = reinterpret_cast<const float4*>(out_suf + r * kDL);
  uint2* dst = reinterpret_cast<uint2*>(out + r * kDL);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = lane + 32 * k;
    const float4 a = src_p[c], b = src_s[c];
    const __nv_bfloat162 y0 = __floats2bfloat162_rn(ap * a.x + as * b.x, ap * a.y + as * b.y);
    const __nv_bfloat162 y1 = __floats2bfloat162_rn(ap * a.z + as * b.z, ap * a.w + as * b.w);
    dst[c] = make_uint2(*reinterpret_cast<const uint32_t*>(&y0), *reinterpret_cast<const uint32_t*>(&y1));
  }
  if (lane == 0) lse[r] = z > 0.f ? m + __logf(z) : -INFINITY;
}

}  // namespace mla

namespace {

struct Plan {
  int g;                                // requests per prefix-pass row block
  int b_main, b_tail;                   // requests in the grouped / ungrouped prefix pass
  mla_dims main, tail, suffix;          // the passes' dimensions
  size_t status, len_pre, len_suf, out_pre, lse_pre, out_suf, dec, dec_bytes, total;
};

bool make_plan(const mla_dims* d, int32_t prefix_pages, int device, Plan* p) {
  if (!d || d->batch < 1 || d->num_heads < 1 || d->q_len < 1 || d->num_pages < 1 || d->page_size != kPageRows)
    return false;
  if (prefix_pages < 1 || prefix_pages >= d->max_pages_per_req || d->page_table_stride < d->max_pages_per_req)
    return false;
  const int rows = d->num_heads * d->q_len;
  if (rows > 256) return false;
  p->g = (rows <= 128 && 128 % rows == 0) ? 128 / rows : 1;
  p->b_main = d->batch / p->g * p->g;
  p->b_tail = d->batch - p->b_main;
  if (static_cast<int64_t>(p->g) * d->page_table_stride > INT_MAX) return false;
  p->main = *d;
  p->main.batch = p->b_main / p->g;
  p->main.num_heads = p->g * rows;
  p->main.q_len = 1;
  p->main.max_pages_per_req = prefix_pages;
  p->main.page_table_stride = p->g * d->page_table_stride;
  p->tail = *d;
  p->tail.batch = std::max(p->b_tail, 1);
  p->tail.num_heads = rows;
  p->tail.q_len = 1;
  p->tail.max_pages_per_req = prefix_pages;
  p->suffix = *d;
  p->suffix.max_pages_per_req = d->max_pages_per_req - prefix_pages;
  size_t dec = 0;
  for (const mla_dims* pd : {&p->main, &p->tail, &p->suffix}) {
    if (pd == &p->main && p->b_main == 0) continue;
    if (pd == &p->tail && p->b_tail == 0) continue;
    const size_t n = mla_decode_workspace_size(pd, device);
    if (n == 0) return false;
    dec = std::max(dec, n);
  }
  const size_t B = static_cast<size_t>(d->batch);
  const size_t qrows = B * d->q_len * d->num_heads;
  p->status = 0;
  p->len_pre = 256;
  p->len_suf = align_up(p->len_pre + B * 4, 256);
  p->out_pre = align_up(p->len_suf + B * 4, 256);
  p->lse_pre = align_up(p->out_pre + qrows * kDL * 4, 256);
  p->out_suf = align_up(p->lse_pre + qrows * 4, 256);
  p->dec = align_up(p->out_suf + qrows * kDL * 4, 256);
  p->dec_bytes = dec;
  p->total = p->dec + dec;
  return true;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace

extern "C" {

size_t mla_decode_cascade_workspace_size(const mla_dims* d, int32_t prefix_pages, int device) {
  Plan p;
  return make_plan(d, prefix_pages, device, &p) ? p.total : 0;
}

int mla_decode_cascade(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                       const int32_t* page_table, const int32_t* seq_lens, int32_t prefix_pages, int32_t q_len,
                       float scale, float kv_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                       void* stream_v) {
  if (!d || !q_nope || !q_pe || !kv_cache || !page_table || !seq_lens || !out || !lse || !workspace)
    return MLA_ERR_INVALID_ARG;
  if (q_len != d->q_len) return MLA_ERR_INVALID_ARG;
  if (d->page_size != kPageRows) return MLA_ERR_UNSUPPORTED;
  if (!aligned(workspace, 256) || !aligned(page_table, 4) || !aligned(seq_lens, 4)) return MLA_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  Plan p;
  if (!make_plan(d, prefix_pages, dev, &p)) return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < p.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws + p.status);
  int32_t* len_pre = reinterpret_cast<int32_t*>(ws + p.len_pre);
  int32_t* len_suf = reinterpret_cast<int32_t*>(ws + p.len_suf);
  float* out_pre = reinterpret_cast<float*>(ws + p.out_pre);
  float* lse_pre = reinterpret_cast<float*>(ws + p.lse_pre);
  float* out_suf = reinterpret_cast<float*>(ws + p.out_suf);
  uint8_t* dec = ws + p.dec;
  const int32_t* dec_status = reinterpret_cast<const int32_t*>(dec);
  if (cudaMemsetAsync(status, 0, 4, stream) != cudaSuccess) return MLA_ERR_CUDA;
  mla::mla_cascade_prep_kernel<<<d->batch, 128, 0, stream>>>(page_table, seq_lens, d->page_table_stride,
                                                              prefix_pages, d->q_len, len_pre, len_suf, status);
  if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
  const size_t row_q = static_cast<size_t>(d->q_len) * d->num_heads;  // query rows per request
  int rc;
  // 1. prefix pass: every draft sees the whole prefix (q_len folded into heads)
  if (p.b_main > 0) {
    rc = mla_decode_f32_out(&p.main, q_nope, q_pe, kv_cache, page_table, len_pre, 1, scale, kv_scale, out_pre,
                            lse_pre, dec, p.dec_bytes, stream_v);
    if (rc != MLA_OK) return rc;
    mla::mla_cascade_or_status_kernel<<<1, 1, 0, stream>>>(dec_status, status);
  }
  if (p.b_tail > 0) {
    const size_t r0 = static_cast<size_t>(p.b_main) * row_q;
    rc = mla_decode_f32_out(&p.tail, static_cast<const uint8_t*>(q_nope) + r0 * kDL * 2,
                            static_cast<const uint8_t*>(q_pe) + r0 * 64 * 2, kv_cache,
                            page_table + static_cast<int64_t>(p.b_main) * d->page_table_stride, len_pre, 1, scale,
                            kv_scale, out_pre + r0 * kDL, lse_pre + r0, dec, p.dec_bytes, stream_v);
    if (rc != MLA_OK) return rc;
    mla::mla_cascade_or_status_kernel<<<1, 1, 0, stream>>>(dec_status, status);
  }
  // 2. suffix pass: fp32 out in the workspace, lse in the caller's lse
  rc = mla_decode_f32_out(&p.suffix, q_nope, q_pe, kv_cache, page_table + prefix_pages, len_suf, d->q_len, scale,
                          kv_scale, out_suf, lse, dec, p.dec_bytes, stream_v);
  if (rc != MLA_OK) return rc;
  mla::mla_cascade_or_status_kernel<<<1, 1, 0, stream>>>(dec_status, status);
  // 3. merge
  const int64_t rows = static_cast<int64_t>(d->batch) * row_q;
  mla::mla_cascade_merge_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      out_pre, lse_pre, out_suf, static_cast<__nv_bfloat16*>(out), lse, rows);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode_cascade_query_status(const mla_dims* d, int32_t prefix_pages, const void* workspace, void* stream_v,
                                    int32_t* status) {
  if (!workspace || !status) return MLA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  Plan p;
  if (!make_plan(d, prefix_pages, dev, &p)) return MLA_ERR_INVALID_ARG;
  return mla_query_status(workspace, stream_v, status);  // the passes' bits are OR-ed into word 0
}

}  // extern "C"
