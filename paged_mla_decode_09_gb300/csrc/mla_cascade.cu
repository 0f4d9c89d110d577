// Cascade decode over a shared prefix (see include/mla_cascade.h): a prefix
// pass with several requests' query rows per row block, a suffix pass, and a
// log-sum-exp merge.  The two passes are the paged decode of mla_decode.h,
// called with rearranged dimensions on the caller's buffers; the prefix pass
// sees every request's length as the prefix length and the suffix pass the
// length minus the prefix (internal length controls of the decode, so no
// kernel rewrites the lengths).
//
// Workspace: [prefix out (fp32 [B][q_len][H][512]) | prefix lse (fp32
// [B][q_len][H]) | suffix out (fp32, same shape) | one decode workspace per
// pass (main prefix pass, leftover prefix pass, suffix pass)].  Both passes
// write fp32 results, so that the only rounding to bf16 is the merged
// output's, as in the plain decode's combine.  Each pass keeps its own
// status word; the merge adds the shared-prefix check to the suffix pass's.
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

// one warp per query row: out = (e^lp op + e^ls os) / (e^lp + e^ls),
// lse = ln(e^lp + e^ls), from the two passes' fp32 results; the suffix lse
// is in lse and is replaced.  The warp of a request's first row also checks
// that the request's prefix columns name the same pages as request 0's.
__global__ void __launch_bounds__(256)
    mla_cascade_merge_kernel(const float* __restrict__ out_pre, const float* __restrict__ lse_pre,
                             const float* __restrict__ out_suf, __nv_bfloat16* out, float* lse, int64_t rows,
                             int rows_per_req, const int32_t* __restrict__ page_table, int stride, int prefix_pages,
                             int32_t* status) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  if (r % rows_per_req == 0) {
    const int64_t b = r / rows_per_req;
    bool same = true;
    for (int c = lane; c < prefix_pages; c += 32) same &= page_table[b * stride + c] == page_table[c];
    if (!__all_sync(0xffffffffu, same) && lane == 0) atomicOr(status, MLA_DEV_BAD_PREFIX);
  }
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
  size_t out_pre, lse_pre, out_suf, dec_main, dec_tail, dec_suf, total;
  size_t n_main, n_tail, n_suf;         // bytes of each pass's decode workspace (0: the pass does not run)
};

bool make_plan(const mla_dims* d, int32_t prefix_pages, int device, Plan* p) {
  if (!d || d->batch < 1 || d->num_heads < 1 || d->q_len < 1 || d->num_pages < 1 || d->page_size != kPageRows)
    return false;
  if (prefix_pages < 1 || prefix_pages >= d->max_pages_per_req || d->page_table_stride < d->max_pages_per_req)
    return false;
  if (static_cast<int64_t>(prefix_pages) * kPageRows > INT_MAX) return false;
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
  p->n_main = p->b_main > 0 ? mla_decode_workspace_size(&p->main, device) : 0;
  p->n_tail = p->b_tail > 0 ? mla_decode_workspace_size(&p->tail, device) : 0;
  p->n_suf = mla_decode_workspace_size(&p->suffix, device);
  if ((p->b_main > 0 && p->n_main == 0) || (p->b_tail > 0 && p->n_tail == 0) || p->n_suf == 0) return false;
  const size_t B = static_cast<size_t>(d->batch);
  const size_t qrows = B * d->q_len * d->num_heads;
  p->out_pre = 0;
  p->lse_pre = align_up(p->out_pre + qrows * kDL * 4, 256);
  p->out_suf = align_up(p->lse_pre + qrows * 4, 256);
  p->dec_main = align_up(p->out_suf + qrows * kDL * 4, 256);
  p->dec_tail = align_up(p->dec_main + p->n_main, 256);
  p->dec_suf = align_up(p->dec_tail + p->n_tail, 256);
  p->total = p->dec_suf + p->n_suf;
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
  float* out_pre = reinterpret_cast<float*>(ws + p.out_pre);
  float* lse_pre = reinterpret_cast<float*>(ws + p.lse_pre);
  float* out_suf = reinterpret_cast<float*>(ws + p.out_suf);
  const int32_t pre_len = prefix_pages * kPageRows;
  const size_t row_q = static_cast<size_t>(d->q_len) * d->num_heads;  // query rows per request
  int rc;
  // 1. prefix pass: every draft sees the whole prefix (q_len folded into heads)
  if (p.b_main > 0) {
    rc = mla_decode_f32_out(&p.main, q_nope, q_pe, kv_cache, page_table, seq_lens, 0, pre_len, 1, scale, kv_scale,
                            out_pre, lse_pre, ws + p.dec_main, p.n_main, stream_v);
    if (rc != MLA_OK) return rc;
  }
  if (p.b_tail > 0) {
    const size_t r0 = static_cast<size_t>(p.b_main) * row_q;
    rc = mla_decode_f32_out(&p.tail, static_cast<const uint8_t*>(q_nope) + r0 * kDL * 2,
                            static_cast<const uint8_t*>(q_pe) + r0 * 64 * 2, kv_cache,
                            page_table + static_cast<int64_t>(p.b_main) * d->page_table_stride, seq_lens, 0, pre_len,
                            1, scale, kv_scale, out_pre + r0 * kDL, lse_pre + r0, ws + p.dec_tail, p.n_tail,
                            stream_v);
    if (rc != MLA_OK) return rc;
  }
  // 2. suffix pass (lengths minus the prefix): fp32 out in the workspace, lse in the caller's lse
  rc = mla_decode_f32_out(&p.suffix, q_nope, q_pe, kv_cache, page_table + prefix_pages, seq_lens, pre_len, 0,
                          d->q_len, scale, kv_scale, out_suf, lse, ws + p.dec_suf, p.n_suf, stream_v);
  if (rc != MLA_OK) return rc;
  // 3. merge, and the check that the prefix is shared
  const int64_t rows = static_cast<int64_t>(d->batch) * row_q;
  mla::mla_cascade_merge_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      out_pre, lse_pre, out_suf, static_cast<__nv_bfloat16*>(out), lse, rows, static_cast<int>(row_q), page_table,
      d->page_table_stride, prefix_pages, reinterpret_cast<int32_t*>(ws + p.dec_suf));
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode_cascade_query_status(const mla_dims* d, int32_t prefix_pages, const void* workspace, void* stream_v,
                                    int32_t* status) {
  if (!workspace || !status) return MLA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  Plan p;
  if (!make_plan(d, prefix_pages, dev, &p)) return MLA_ERR_INVALID_ARG;
  // the OR of the passes' status words
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  int32_t all = 0;
  const size_t offs[3] = {p.dec_main, p.dec_tail, p.dec_suf};
  const size_t lens[3] = {p.n_main, p.n_tail, p.n_suf};
  for (int k = 0; k < 3; ++k) {
    if (lens[k] == 0) continue;
    int32_t w = 0;
    const int rc = mla_query_status(ws + offs[k], stream_v, &w);
    if (rc != MLA_OK) return rc;
    all |= w;
  }
  *status = all;
  return MLA_OK;
}

}  // extern "C"
