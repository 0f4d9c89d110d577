// Top-k sparse decode (see include/mla_sparse.h): a gather kernel packs the
// selected latent rows of every (request, draft position) into pages of the
// workspace, then the paged decode runs over them as B * q_len requests of
// one draft position each.
//
// Workspace: [per-block status bits | packed lengths | empty flags | packed
// page table | packed rows | decode workspace].  The gather's blocks each
// write their status bits to a word of their own (no word needs clearing
// first); the decode's schedule kernel ORs them into its status word, and
// its combine kernel gives the lists without a valid entry lse = -inf.
// Packed request b' = b * q_len + i owns pages b' * P .. b' * P + P - 1,
// P = ceil(topk / 64), and its k-th valid entry is its packed row k.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "mla_decode.h"
#include "mla_internal.h"
#include "mla_sparse.h"

namespace {

constexpr int kPageRows = 64;
constexpr int kChunkEntries = 256;  // top-k entries per gather block
constexpr int64_t kMaxPacked = 65535;  // (b, i) pairs: the gather grid's y extent
constexpr int kRowsInFlight = 2;    // rows a warp copies per round (all loads first; 1-8 measured, 1-2 best)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__device__ __forceinline__ uint4 ldg_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(reinterpret_cast<uint64_t>(p)));
  return v;
}

}  // namespace

namespace mla {

// grid (ceil(topk / 256), B * q_len), 256 threads: block (c, b') ranks the
// valid entries c*256 .. c*256+255 of b' after those of the chunks before it
// and copies their rows to the packed rows of those ranks.
template <int kRowBytes>
__global__ void __launch_bounds__(kChunkEntries)
    mla_topk_gather_kernel(const uint8_t* __restrict__ cache, const int32_t* __restrict__ page_table,
                           const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ indices, int q_len,
                           int topk, int num_pages, int max_pages, int pt_stride, int p_per,
                           uint8_t* __restrict__ packed, int32_t* __restrict__ packed_pt,
                           int32_t* __restrict__ packed_len, int32_t* __restrict__ packed_empty,
                           int32_t* __restrict__ block_bits) {
  constexpr int kChunks = kRowBytes / 16;
  constexpr int kPer = (kChunks + 31) / 32;
  __shared__ int warp_cnt[kChunkEntries / 32];
  __shared__ int red[kChunkEntries / 32];
  __shared__ int32_t list_t[kChunkEntries];
  __shared__ int32_t list_slot[kChunkEntries];
  __shared__ int bits;  // this block's status bits
  int32_t* status = &bits;
  if (threadIdx.x == 0) bits = 0;
  __syncthreads();
  const int bq = blockIdx.y, chunk = blockIdx.x;
  const int b = bq / q_len, i = bq % q_len;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = seq_lens[b];
  const bool len_ok = L >= q_len && L <= max_pages * kPageRows;
  if (!len_ok && chunk == 0 && threadIdx.x == 0) atomicOr(status, MLA_DEV_BAD_SEQ_LEN);
  const int nvis = len_ok ? L - q_len + i + 1 : 0;  // positions draft i may see
  const int32_t* idx = indices + static_cast<int64_t>(bq) * topk;

  // valid entries of the chunks before this one
  int before = 0;
  for (int e = threadIdx.x; e < chunk * kChunkEntries; e += kChunkEntries) {
    const int t = idx[e];
    before += (t >= 0 && t < nvis) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  if (lane == 0) red[warp] = before;

  // this chunk: rank the valid entries in list order
  const int e = chunk * kChunkEntries + threadIdx.x;
  const int t = e < topk ? idx[e] : -1;
  const bool valid = t >= 0 && t < nvis;
  const bool bad = e < topk && t != -1 && !valid;
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, MLA_DEV_BAD_INDEX);
  const unsigned m = __ballot_sync(0xffffffffu, valid);
  if (lane == 0) warp_cnt[warp] = __popc(m);
  __syncthreads();
  int base = 0, wbase = 0, total_chunk = 0;
#pragma unroll
  for (int w = 0; w < kChunkEntries / 32; ++w) {
    base += red[w];
    if (w < warp) wbase += warp_cnt[w];
    total_chunk += warp_cnt[w];
  }
  const int rank_w = __popc(m & ((1u << lane) - 1u));
  if (valid) {
    list_t[warp * 32 + rank_w] = t;
    list_slot[warp * 32 + rank_w] = base + wbase + rank_w;
  }
  const int64_t row0 = static_cast<int64_t>(bq) * p_per * kPageRows;  // packed row 0 of b'
  if (chunk == 0)
    for (int p = threadIdx.x; p < p_per; p += kChunkEntries) packed_pt[static_cast<int64_t>(bq) * p_per + p] =
        bq * p_per + p;
  const bool last = chunk == static_cast<int>(gridDim.x) - 1;
  const int total = base + total_chunk;
  if (last && total == 0) {  // nothing to attend: one zero row (out = 0; lse is set afterwards)
    if (threadIdx.x == 0) atomicOr(status, MLA_DEV_BAD_INDEX);
    uint4* dst = reinterpret_cast<uint4*>(packed + row0 * kRowBytes);
    for (int c = threadIdx.x; c < kChunks; c += kChunkEntries) dst[c] = make_uint4(0, 0, 0, 0);
  }
  if (last && threadIdx.x == 0) {
    packed_len[bq] = total > 0 ? total : 1;
    packed_empty[bq] = total == 0 ? 1 : 0;
  }
  __syncwarp();

  // copy this warp's rows, kRowsInFlight at a time
  const int n = __popc(m);
  for (int r0 = 0; r0 < n; r0 += kRowsInFlight) {
    uint4 v[kRowsInFlight][kPer];
    int64_t dst_row[kRowsInFlight];
    bool ok[kRowsInFlight];
#pragma unroll
    for (int r = 0; r < kRowsInFlight; ++r) {
      ok[r] = false;
      dst_row[r] = 0;
      if (r0 + r >= n) continue;
      const int tt = list_t[warp * 32 + r0 + r];
      dst_row[r] = row0 + list_slot[warp * 32 + r0 + r];
      const int pid = page_table[static_cast<int64_t>(b) * pt_stride + tt / kPageRows];
      ok[r] = pid >= 0 && pid < num_pages;
      if (!ok[r]) continue;
      const uint4* src =
          reinterpret_cast<const uint4*>(cache + (static_cast<int64_t>(pid) * kPageRows + tt % kPageRows) * kRowBytes);
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        if (lane + 32 * k < kChunks) v[r][k] = ldg_nc_v4(src + lane + 32 * k);
    }
#pragma unroll
    for (int r = 0; r < kRowsInFlight; ++r) {
      if (r0 + r >= n) continue;
      if (!ok[r] && lane == 0) atomicOr(status, MLA_DEV_BAD_PAGE_ID);
      uint4* dst = reinterpret_cast<uint4*>(packed + dst_row[r] * kRowBytes);
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        if (lane + 32 * k < kChunks) dst[lane + 32 * k] = ok[r] ? v[r][k] : make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) block_bits[static_cast<int64_t>(bq) * gridDim.x + chunk] = bits;
}

}  // namespace mla

namespace {

struct SparseLayout {
  size_t status, plen, pempty, ppt, rows, dec, total;
};

bool packed_dims(const mla_dims* d, int32_t topk, mla_dims* pd) {
  if (!d || topk < 1 || topk > 65536) return false;
  if (d->batch < 1 || d->q_len < 1 || d->num_heads < 1) return false;
  const int64_t bq = static_cast<int64_t>(d->batch) * d->q_len;
  const int64_t p_per = (topk + kPageRows - 1) / kPageRows;
  if (bq > kMaxPacked || bq * p_per > INT_MAX / kPageRows) return false;
  *pd = *d;
  pd->batch = static_cast<int32_t>(bq);
  pd->q_len = 1;
  pd->num_pages = static_cast<int32_t>(bq * p_per);
  pd->max_pages_per_req = static_cast<int32_t>(p_per);
  pd->page_table_stride = static_cast<int32_t>(p_per);
  return true;
}

bool sparse_layout(const mla_dims* d, int32_t topk, int device, SparseLayout* l, mla_dims* pd) {
  if (!packed_dims(d, topk, pd)) return false;
  const size_t dec = mla_decode_workspace_size(pd, device);
  if (dec == 0) return false;
  const size_t row_bytes = d->kv_dtype == MLA_KV_FP8_E4M3 ? 576 : 1152;
  l->status = 0;  // block status bits: [B * q_len][ceil(topk / 256)]
  l->plen = align_up(static_cast<size_t>(pd->batch) * ((topk + kChunkEntries - 1) / kChunkEntries) * 4, 256);
  l->pempty = align_up(l->plen + static_cast<size_t>(pd->batch) * 4, 256);
  l->ppt = align_up(l->pempty + static_cast<size_t>(pd->batch) * 4, 256);
  l->rows = align_up(l->ppt + static_cast<size_t>(pd->num_pages) * 4, 1024);
  l->dec = align_up(l->rows + static_cast<size_t>(pd->num_pages) * kPageRows * row_bytes, 256);
  l->total = l->dec + dec;
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" {

size_t mla_decode_sparse_workspace_size(const mla_dims* d, int32_t topk, int device) {
  SparseLayout l;
  mla_dims pd;
  return sparse_layout(d, topk, device, &l, &pd) ? l.total : 0;
}

int mla_decode_sparse(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                      const int32_t* page_table, const int32_t* seq_lens, const int32_t* indices, int32_t topk,
                      int32_t q_len, float scale, float kv_scale, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, void* stream_v) {
  if (!d || !indices || !workspace || !kv_cache || !page_table || !seq_lens) return MLA_ERR_INVALID_ARG;
  if (topk < 1 || topk > 65536 || q_len != d->q_len) return MLA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->num_heads < 1 || d->q_len < 1 || d->num_pages < 1 || d->max_pages_per_req < 1 ||
      d->page_table_stride < d->max_pages_per_req)
    return MLA_ERR_INVALID_ARG;
  if (d->page_size != kPageRows) return MLA_ERR_UNSUPPORTED;
  if (d->kv_dtype != MLA_KV_BF16 && d->kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_UNSUPPORTED;
  if (!aligned(indices, 4) || !aligned(workspace, 256) || !aligned(kv_cache, 16) || !aligned(page_table, 4) ||
      !aligned(seq_lens, 4))
    return MLA_ERR_ALIGNMENT;
  if (static_cast<int64_t>(d->batch) * d->q_len > kMaxPacked) return MLA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  SparseLayout l;
  mla_dims pd;
  if (!sparse_layout(d, topk, dev, &l, &pd)) return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < l.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (major != 10 || minor != 3) return MLA_ERR_DEVICE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* block_bits = reinterpret_cast<int32_t*>(ws + l.status);
  int32_t* plen = reinterpret_cast<int32_t*>(ws + l.plen);
  int32_t* pempty = reinterpret_cast<int32_t*>(ws + l.pempty);
  int32_t* ppt = reinterpret_cast<int32_t*>(ws + l.ppt);
  uint8_t* rows = ws + l.rows;
  const dim3 grid((topk + kChunkEntries - 1) / kChunkEntries, pd.batch);
  const uint8_t* cache = static_cast<const uint8_t*>(kv_cache);
  if (d->kv_dtype == MLA_KV_FP8_E4M3)
    mla::mla_topk_gather_kernel<576><<<grid, kChunkEntries, 0, stream>>>(
        cache, page_table, seq_lens, indices, d->q_len, topk, d->num_pages, d->max_pages_per_req,
        d->page_table_stride, pd.max_pages_per_req, rows, ppt, plen, pempty, block_bits);
  else
    mla::mla_topk_gather_kernel<1152><<<grid, kChunkEntries, 0, stream>>>(
        cache, page_table, seq_lens, indices, d->q_len, topk, d->num_pages, d->max_pages_per_req,
        d->page_table_stride, pd.max_pages_per_req, rows, ppt, plen, pempty, block_bits);
  if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
  // the packed problem: request b * q_len + i has one draft position; its
  // queries and outputs are those of (b, i), already laid out that way.  The
  // decode's status word (cleared by its schedule kernel) collects the
  // gather's bits too, and lists without a valid pick get lse = -inf.
  return mla_decode_topk_packed(&pd, q_nope, q_pe, rows, ppt, plen, scale, kv_scale, out, lse, ws + l.dec,
                                workspace_bytes - l.dec, block_bits, static_cast<int32_t>(grid.x), pempty, stream_v);
}

int mla_decode_sparse_query_status(const mla_dims* d, int32_t topk, const void* workspace, void* stream_v,
                                   int32_t* status) {
  if (!workspace || !status) return MLA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  SparseLayout l;
  mla_dims pd;
  if (!sparse_layout(d, topk, dev, &l, &pd)) return MLA_ERR_INVALID_ARG;
  return mla_query_status(static_cast<const uint8_t*>(workspace) + l.dec, stream_v, status);
}

}  // extern "C"
