// Host side of the paged MLA decode C ABI (see include/mla_decode.h):
// argument checks, workspace layout, TMA tensor maps and the three launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mla_decode.h"
#include "mla_internal.h"
#include "mla_kernels.cuh"

namespace {

using mla::Cfg;
using mla::Params;

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per pipeline wait

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Launches a kernel with programmatic stream serialization: it may start
// while the previous kernel in the stream is finishing and waits for it
// (griddep_wait) before reading that kernel's output.
template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Workspace: [status words | page prefix sums | cluster slices | each
// request's first and last cluster | the requests cut into pieces, each with
// its pieces' partial slots | fp32 partial outputs | partial log-sum-exps |
// e4m3 query scales | e4m3 query terms (1152 bytes a row)].  Sized by B,
// the cluster count, the number of row blocks and the cache type only.
struct Layout {
  size_t status, prefix, cinfo, rrange, splits, o_part, lse_part, qscale, qterms, total;
};

Layout workspace_layout(int B, int C, int G, bool qterms) {
  Layout l;
  l.status = 0;
  l.prefix = 256;
  l.cinfo = l.prefix + align256(static_cast<size_t>(B + 1) * 4);
  l.rrange = l.cinfo + align256(static_cast<size_t>(C) * 3 * 4);
  l.splits = l.rrange + align256(static_cast<size_t>(B) * 2 * 4);
  l.o_part = l.splits + align256(static_cast<size_t>(1 + (B < C ? B : C)) * 8 * 4);
  l.lse_part = l.o_part + align256(static_cast<size_t>(2 * C) * G * mla::kRows * mla::kDL * 4);
  l.qscale = l.lse_part + align256(static_cast<size_t>(2 * C) * G * mla::kRows * 4);
  l.qterms = l.qscale + align256(static_cast<size_t>(B) * G * mla::kRows * 4);  // e4m3 query scales
  l.total = l.qterms + (qterms ? align256(static_cast<size_t>(B) * G * mla::kRows * 1152) : 0);
  return l;
}

int check_dims(const mla_dims* d) {
  if (!d) return MLA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->num_heads < 1 || d->q_len < 1 || d->num_pages < 1 || d->max_pages_per_req < 1 ||
      d->page_table_stride < d->max_pages_per_req)
    return MLA_ERR_INVALID_ARG;
  if (d->page_size != 64) return MLA_ERR_UNSUPPORTED;
  if (d->kv_dtype != MLA_KV_BF16 && d->kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->num_heads) * d->q_len > 256) return MLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->num_pages) * 64 > (1ll << 31) - 1) return MLA_ERR_UNSUPPORTED;
  // token positions of one request and the schedule's page prefix sums over
  // all requests are int32 on the device
  if (static_cast<int64_t>(d->max_pages_per_req) * 64 > (1ll << 31) - 1) return MLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->batch) * d->max_pages_per_req > (1ll << 31) - 1) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

int device_ok(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (major != 10 || minor != 3) return MLA_ERR_DEVICE;  // built for sm_103a only
  return MLA_OK;
}

// Slices of the attention kernel's work: the clusters of one S/O pair that
// fit at once, divided by G (each slice is computed by G clusters, one per
// row block).
struct ShapeCache {
  std::mutex mu;
  int clusters[64][2][3] = {};  // [device][fp8][G]
  int smem_sm[64] = {};         // shared memory per SM, reserved per block, a block's maximum
  int smem_rsv[64] = {};
  int smem_blk[64] = {};
};
ShapeCache g_shapes;

int launch_shape(int device, bool f8, int G, int* clusters_out) {
  if (device < 0 || device >= 64 || G < 1 || G > 2) return MLA_ERR_INVALID_ARG;
  {
    std::lock_guard<std::mutex> lk(g_shapes.mu);
    if (g_shapes.clusters[device][f8][G]) {
      *clusters_out = g_shapes.clusters[device][f8][G];
      return MLA_OK;
    }
  }
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return MLA_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return MLA_ERR_CUDA;
  int rc = device_ok(device);
  int n = 0;
  if (rc == MLA_OK) {
    const void* fn = f8 ? reinterpret_cast<const void*>(&mla::mla_decode_kernel<true, true>)
                        : reinterpret_cast<const void*>(&mla::mla_decode_kernel<false, false>);
    const int smem = f8 ? Cfg<true>::kSmem : Cfg<false>::kSmem;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        (f8 && cudaFuncSetAttribute(reinterpret_cast<const void*>(&mla::mla_decode_kernel<true, false>),
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)) {
      rc = MLA_ERR_CUDA;
    } else {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * 64, 1, 1);
      cfg.blockDim = dim3(mla::kThreads, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < G) rc = MLA_ERR_CUDA;
      n /= G;
    }
  }
  // the combine kernel takes dynamic shared memory that it does not use
  // (up to a block's maximum) to cap its blocks per SM
  int smem_sm = 0, smem_rsv = 0, smem_blk = 0;
  if (rc == MLA_OK &&
      (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess ||
       cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, device) != cudaSuccess ||
       cudaDeviceGetAttribute(&smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
       cudaFuncSetAttribute(mla::mla_combine_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_blk) !=
           cudaSuccess ||
       cudaFuncSetAttribute(mla::mla_combine_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_blk) !=
           cudaSuccess ||
       cudaFuncSetAttribute(mla::mla_combine_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_blk) !=
           cudaSuccess))
    rc = MLA_ERR_CUDA;
  if (prev != device) cudaSetDevice(prev);
  if (rc != MLA_OK) {
    cudaGetLastError();
    return rc;
  }
  std::lock_guard<std::mutex> lk(g_shapes.mu);
  g_shapes.smem_sm[device] = smem_sm;
  g_shapes.smem_rsv[device] = smem_rsv;
  g_shapes.smem_blk[device] = smem_blk;
  g_shapes.clusters[device][f8][G] = n;
  *clusters_out = n;
  return MLA_OK;
}

// Dynamic shared memory that lets at most k blocks of a kernel that uses
// none share an SM (0: no cap).
size_t spread_smem(int device, int k) {
  std::lock_guard<std::mutex> lk(g_shapes.mu);
  if (k >= mla::kCombineBlocksPerSm || g_shapes.smem_sm[device] <= 0) return 0;
  int s = g_shapes.smem_sm[device] / k - g_shapes.smem_rsv[device];
  if (s > g_shapes.smem_blk[device]) s = g_shapes.smem_blk[device];
  return s > 0 ? static_cast<size_t>(s) & ~static_cast<size_t>(127) : 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Tensor maps over the cache.  Each page is fetched with one 3-D box whose
// dimensions are (64 or 128 values of a row, 64 token rows 576 values apart,
// box index 128 bytes apart): the box lands in shared memory as [box][row]
// [128 bytes] with 128-byte swizzle, the K-major / MN-major layout the MMAs
// read.  tm_s: the S CTA's page (bf16: all 9 boxes; e4m3: the 4 c_kv boxes),
// tm_o: the O CTA's c_kv boxes, tm_pe: the e4m3 k_pe part (64-byte rows,
// 64-byte swizzle, 2-D).
struct Maps {
  CUtensorMap s, o, pe, qn, qp;
};

int make_maps(const void* kv, int num_pages, bool f8, Maps* m) {
  auto enc = encode_fn();
  if (!enc) return MLA_ERR_CUDA;
  const cuuint64_t rows = static_cast<cuuint64_t>(num_pages) * 64;
  const cuuint64_t row_bytes = f8 ? 576 : 1152;
  const cuuint32_t box_vals = f8 ? 128 : 64;  // one 128-byte swizzle row
  cuuint64_t gdim[3] = {box_vals, rows, f8 ? 4u : 9u};
  cuuint64_t gstr[2] = {row_bytes, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // one copy = one ring part: kBoxesPartS / kBoxesPartO 128-byte columns of 64 token rows
  cuuint32_t box_s[3] = {box_vals, 64, static_cast<cuuint32_t>(f8 ? Cfg<true>::kBoxesPartS : Cfg<false>::kBoxesPartS)};
  CUresult r = enc(&m->s, dt, 3, const_cast<void*>(kv), gdim, gstr, box_s, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
  cuuint32_t box_o[3] = {box_vals, 64, static_cast<cuuint32_t>(f8 ? Cfg<true>::kBoxesPartO : Cfg<false>::kBoxesPartO)};
  r = enc(&m->o, dt, 3, const_cast<void*>(kv), gdim, gstr, box_o, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
  if (f8) {
    cuuint64_t gdim2[2] = {576, rows};
    cuuint64_t gstr2[1] = {576};
    cuuint32_t box2[2] = {64u, 64u};
    r = enc(&m->pe, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv), gdim2, gstr2, box2, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
  } else {
    m->pe = m->s;
  }
  return MLA_OK;
}

// Query rows as copied into the S CTA's ring (64 rows per copy, laid out
// like a page): q_nope as 8 boxes of 64 values, q_pe as one.
// Tensor maps of the queries: q_nope as 8 boxes and q_pe as one box of 64
// rows (the bf16 S CTA's ring entries).  With e4m3 query terms the first map
// instead covers the terms, [rows][1152] bytes read as 9 boxes of 128 bytes
// of 32 rows (36 KB, an e4m3 ring slot).
int make_qmaps(const void* q_nope, const void* q_pe, const uint8_t* qterms, int64_t rows, Maps* m) {
  auto enc = encode_fn();
  if (!enc) return MLA_ERR_CUDA;
  cuuint32_t estr[3] = {1, 1, 1};
  if (qterms) {
    cuuint64_t gdim[3] = {128, static_cast<cuuint64_t>(rows), 9};
    cuuint64_t gstr[2] = {1152, 128};
    cuuint32_t box[3] = {128, 32, 9};
    const CUresult r = enc(&m->qn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(qterms), gdim, gstr, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
    m->qp = m->qn;  // unused with terms
    return MLA_OK;
  }
  cuuint64_t gdim[3] = {64, static_cast<cuuint64_t>(rows), 8};
  cuuint64_t gstr[2] = {1024, 128};
  cuuint32_t box[3] = {64, 64, 8};
  CUresult r = enc(&m->qn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q_nope), gdim, gstr, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
  cuuint64_t gdim2[2] = {64, static_cast<cuuint64_t>(rows)};
  cuuint64_t gstr2[1] = {128};
  cuuint32_t box2[2] = {64, 64};
  r = enc(&m->qp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q_pe), gdim2, gstr2, box2, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int current_device(int* dev) { return cudaGetDevice(dev) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

// The launch sequence of both decode entry points.  `ws` is the scratch
// (status words, schedule, split partials): the caller's workspace for
// mla_decode, the library's static array for mla_decode_noalloc.  With
// shrink_to_fit the attention kernel runs on fewer clusters when the split
// partials of every cluster the device could hold would not fit in
// ws_bytes (none at all: MLA_ERR_SCRATCH_TOO_SMALL); without it a workspace
// below the full size is MLA_ERR_WORKSPACE_TOO_SMALL.  status_out (device,
// may be null) receives a copy of the status word at the end, on `stream`.
// Checks of a decode call's arguments that need no device.
int check_call(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
               const int32_t* page_table, const int32_t* seq_lens, int32_t q_len, float scale, float kv_scale,
               const void* out, const float* lse, const int32_t* status_out) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (q_len != d->q_len) return MLA_ERR_INVALID_ARG;
  if (!q_nope || !q_pe || !kv_cache || !page_table || !seq_lens || !out || !lse) return MLA_ERR_INVALID_ARG;
  // the softmax scale (and an e4m3 cache's scale) must be positive and finite
  if (!(scale > 0.f) || scale > 3.0e38f) return MLA_ERR_INVALID_ARG;
  if (d->kv_dtype == MLA_KV_FP8_E4M3 && (!(kv_scale > 0.f) || kv_scale > 3.0e38f)) return MLA_ERR_INVALID_ARG;
  if (!aligned(q_nope, 32) || !aligned(q_pe, 32) || !aligned(kv_cache, 16) || !aligned(out, 32) ||
      !aligned(lse, 4) || !aligned(page_table, 4) || !aligned(seq_lens, 4) || (status_out && !aligned(status_out, 4)))
    return MLA_ERR_ALIGNMENT;
  return MLA_OK;
}

int decode_impl(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                const int32_t* page_table, const int32_t* seq_lens, int32_t q_len, float scale, float kv_scale,
                void* out, float* lse, uint8_t* ws, size_t ws_bytes, bool shrink_to_fit, int32_t* status_out,
                void* stream_v, void* const* events, bool out_f32 = false, int32_t len_offset = 0,
                int32_t len_fixed = 0, const int32_t* topk_bits = nullptr, const int32_t* topk_empty = nullptr,
                int32_t topk_nchunk = 0) {
  int rc = check_call(d, q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, scale, kv_scale, out, lse, status_out);
  if (rc != MLA_OK) return rc;
  if (!ws) return MLA_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return MLA_ERR_ALIGNMENT;
  int dev = 0;
  if ((rc = current_device(&dev)) != MLA_OK) return rc;
  if ((rc = device_ok(dev)) != MLA_OK) return rc;
  const bool f8 = d->kv_dtype == MLA_KV_FP8_E4M3;
  const int R = d->num_heads * d->q_len;
  const int G = (R + mla::kRows - 1) / mla::kRows;
  int C = 0;
  if ((rc = launch_shape(dev, f8, G, &C)) != MLA_OK) return rc;
  // e4m3: the query terms prepared by the scale pre-pass when the workspace
  // has room for them, else the attention kernel splits the rows itself
  bool terms = f8 && workspace_layout(d->batch, C, G, true).total <= ws_bytes;
  if (shrink_to_fit) {
    while (C > 0 && workspace_layout(d->batch, C, G, terms).total > ws_bytes) --C;
    if (C < 1) return MLA_ERR_SCRATCH_TOO_SMALL;
  }
  const Layout lay = workspace_layout(d->batch, C, G, terms);
  if (ws_bytes < lay.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  Maps maps;
  if ((rc = make_maps(kv_cache, d->num_pages, f8, &maps)) != MLA_OK) return rc;
  if ((rc = make_qmaps(q_nope, q_pe, terms ? ws + lay.qterms : nullptr, static_cast<int64_t>(d->batch) * R, &maps)) !=
      MLA_OK)
    return rc;

  Params p;
  p.q_nope = static_cast<const uint8_t*>(q_nope);
  p.q_pe = static_cast<const uint8_t*>(q_pe);
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.out = static_cast<uint8_t*>(out);
  p.lse = lse;
  p.o_part = reinterpret_cast<float*>(ws + lay.o_part);
  p.lse_part = reinterpret_cast<float*>(ws + lay.lse_part);
  p.status = reinterpret_cast<int32_t*>(ws + lay.status);
  p.prefix = reinterpret_cast<int32_t*>(ws + lay.prefix);
  p.cinfo = reinterpret_cast<int32_t*>(ws + lay.cinfo);
  p.rrange = reinterpret_cast<int32_t*>(ws + lay.rrange);
  p.splits = reinterpret_cast<int32_t*>(ws + lay.splits);
  p.qscale = reinterpret_cast<float*>(ws + lay.qscale);
  p.qterms = terms ? ws + lay.qterms : nullptr;
  p.B = d->batch;
  p.H = d->num_heads;
  p.Q = d->q_len;
  p.R = R;
  p.G = G;
  p.C = C;
  p.num_pages = d->num_pages;
  p.max_pages = d->max_pages_per_req;
  p.pt_stride = d->page_table_stride;
  p.unit_cost = mla::unit_cost_pages(f8, R < mla::kRows ? R : mla::kRows);
  p.out_f32 = out_f32 ? 1 : 0;
  p.len_offset = len_offset;
  p.len_fixed = len_fixed;
  p.topk_bits = topk_bits;
  p.topk_empty = topk_empty;
  p.topk_nchunk = topk_nchunk;
  p.scale = scale;
  p.kv_scale = f8 ? kv_scale : 1.f;
  p.timeout_ns = kTimeoutNs;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  auto mark = [&](int k) {
    return !events || cudaEventRecord(static_cast<cudaEvent_t>(events[k]), stream) == cudaSuccess;
  };
  if (!mark(0)) return MLA_ERR_CUDA;
  mla::mla_schedule_kernel<<<1, (d->batch < 256 && C < 256) ? 256 : 1024, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
  if (f8) {  // per-row e4m3 query scales
    if (launch_pdl(mla::mla_qscale_kernel, dim3(static_cast<unsigned>((static_cast<int64_t>(d->batch) * R + 7) / 8)),
                   dim3(256), 0, stream, p) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
  }
  if (!mark(1)) return MLA_ERR_CUDA;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * G * C, 1, 1);  // G clusters of one S/O pair per slice
  cfg.blockDim = dim3(mla::kThreads, 1, 1);
  cfg.dynamicSmemBytes = f8 ? Cfg<true>::kSmem : Cfg<false>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // prologue overlaps the schedule
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = f8 ? (terms ? cudaLaunchKernelEx(&cfg, mla::mla_decode_kernel<true, true>, p, maps.s, maps.o,
                                                     maps.pe, maps.qn, maps.qp)
                             : cudaLaunchKernelEx(&cfg, mla::mla_decode_kernel<true, false>, p, maps.s, maps.o,
                                                     maps.pe, maps.qn, maps.qp))
                     : cudaLaunchKernelEx(&cfg, mla::mla_decode_kernel<false, false>, p, maps.s, maps.o, maps.pe,
                                          maps.qn, maps.qp);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (!mark(2)) return MLA_ERR_CUDA;
  // one block column per request that may be cut into pieces: at most one
  // per cluster boundary
  const unsigned nsplit_max = static_cast<unsigned>(d->batch < C ? d->batch : C);
  // rows per row block that exist (R < 128: only the first R)
  const unsigned zrows = static_cast<unsigned>(((R < mla::kRows ? R : mla::kRows) + mla::kCombineWarps - 1) /
                                               mla::kCombineWarps);
  // A batch of few requests splits each row's columns over two or four
  // blocks (more partial rows in flight per warp) while the grid still fits
  // the GPU at once.  Under programmatic dependent launch the blocks go to
  // the SMs that the attention kernel frees first, as many to each as fit:
  // one 131K-token request's 32 blocks, packed onto the first five SMs, took
  // twice as long as spread over 32.  Shared memory that the kernel does not
  // use caps the blocks per SM at what spreads the grid over the attention
  // kernel's SMs.
  const unsigned sms = 2u * G * C;  // the attention kernel's CTAs, one per SM
  const unsigned resident = static_cast<unsigned>(mla::kCombineBlocksPerSm) * sms;
  const unsigned base = nsplit_max * G * zrows;
  const int parts = base * 4 <= resident ? 4 : base * 2 <= resident ? 2 : 1;
  const unsigned per_sm = (base * parts + sms - 1) / sms;
  const size_t csmem = spread_smem(dev, static_cast<int>(per_sm));
  const dim3 cgrid(nsplit_max, G, zrows * parts), cblock(mla::kCombineWarps * 32);
  const cudaError_t ce = parts == 4   ? launch_pdl(mla::mla_combine_kernel<4>, cgrid, cblock, csmem, stream, p)
                         : parts == 2 ? launch_pdl(mla::mla_combine_kernel<2>, cgrid, cblock, csmem, stream, p)
                                      : launch_pdl(mla::mla_combine_kernel<1>, cgrid, cblock, csmem, stream, p);
  if (ce != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (!mark(3)) return MLA_ERR_CUDA;
  if (status_out && cudaMemcpyAsync(status_out, p.status, 4, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_ALIGNMENT: return "pointer alignment";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_DEVICE: return "device is not sm_103a";
    case MLA_ERR_SCRATCH_TOO_SMALL: return "dimensions exceed the 40 MiB static scratch of mla_decode_noalloc";
    default: return "unknown status";
  }
}

int mla_decode_launch_shape(const mla_dims* d, int device, int32_t* clusters, int32_t* cluster_size) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!clusters || !cluster_size) return MLA_ERR_INVALID_ARG;
  const int G = (d->num_heads * d->q_len + mla::kRows - 1) / mla::kRows;
  int n = 0;
  rc = launch_shape(device, d->kv_dtype == MLA_KV_FP8_E4M3, G, &n);
  if (rc != MLA_OK) return rc;
  *clusters = n * G;
  *cluster_size = 2;
  return MLA_OK;
}

size_t mla_decode_workspace_size(const mla_dims* d, int device) {
  if (check_dims(d) != MLA_OK) return 0;
  const int G = (d->num_heads * d->q_len + mla::kRows - 1) / mla::kRows;
  int C = 0;
  if (launch_shape(device, d->kv_dtype == MLA_KV_FP8_E4M3, G, &C) != MLA_OK) return 0;
  return workspace_layout(d->batch, C, G, d->kv_dtype == MLA_KV_FP8_E4M3).total;
}

int mla_decode(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
               const int32_t* page_table, const int32_t* seq_lens, int32_t q_len, float scale, float kv_scale,
               void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(d, q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, scale, kv_scale, out, lse,
                     static_cast<uint8_t*>(workspace), workspace_bytes, false, nullptr, stream, nullptr);
}

int mla_decode_profiled(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                        const int32_t* page_table, const int32_t* seq_lens, int32_t q_len, float scale,
                        float kv_scale, void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream,
                        void* const* events) {
  if (!events || !events[0] || !events[1] || !events[2] || !events[3]) return MLA_ERR_INVALID_ARG;
  return decode_impl(d, q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, scale, kv_scale, out, lse,
                     static_cast<uint8_t*>(workspace), workspace_bytes, false, nullptr, stream, events);
}

int mla_decode_topk_packed(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                           const int32_t* page_table, const int32_t* seq_lens, float scale, float kv_scale, void* out,
                           float* lse, void* workspace, size_t workspace_bytes, const int32_t* gather_bits,
                           int32_t gather_nchunk, const int32_t* list_empty, void* stream) {
  if (!gather_bits || !list_empty || gather_nchunk < 1) return MLA_ERR_INVALID_ARG;
  return decode_impl(d, q_nope, q_pe, kv_cache, page_table, seq_lens, 1, scale, kv_scale, out, lse,
                     static_cast<uint8_t*>(workspace), workspace_bytes, false, nullptr, stream, nullptr, false, 0, 0,
                     gather_bits, list_empty, gather_nchunk);
}

int mla_decode_f32_out(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                       const int32_t* page_table, const int32_t* seq_lens, int32_t len_offset, int32_t len_fixed,
                       int32_t q_len, float scale, float kv_scale, float* out, float* lse, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (len_offset < 0 || len_fixed < 0) return MLA_ERR_INVALID_ARG;
  return decode_impl(d, q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, scale, kv_scale, out, lse,
                     static_cast<uint8_t*>(workspace), workspace_bytes, false, nullptr, stream, nullptr, true,
                     len_offset, len_fixed);
}

int mla_query_status(const void* workspace, void* stream_v, int32_t* device_status) {
  if (!workspace || !device_status) return MLA_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  if (cudaMemcpyAsync(device_status, workspace, 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_gather_rows(const mla_dims* d, const void* kv_cache, const int32_t* page_table, const int32_t* seq_lens,
                    const int64_t* row_offsets, void* rows_out, void* workspace, void* stream_v) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!kv_cache || !page_table || !seq_lens || !row_offsets || !rows_out || !workspace) return MLA_ERR_INVALID_ARG;
  if (!aligned(kv_cache, 16) || !aligned(rows_out, 16) || !aligned(workspace, 256) || !aligned(row_offsets, 8))
    return MLA_ERR_ALIGNMENT;
  if (d->batch > 65535) return MLA_ERR_UNSUPPORTED;  // the grid's y extent; refused before anything is enqueued
  int dev = 0;
  if ((rc = current_device(&dev)) != MLA_OK) return rc;
  if ((rc = device_ok(dev)) != MLA_OK) return rc;
  const bool f8 = d->kv_dtype == MLA_KV_FP8_E4M3;
  Maps maps;
  if ((rc = make_maps(kv_cache, d->num_pages, f8, &maps)) != MLA_OK) return rc;
  mla::GatherParams gp;
  gp.page_table = page_table;
  gp.seq_lens = seq_lens;
  gp.row_offsets = row_offsets;
  gp.rows_out = static_cast<uint8_t*>(rows_out);
  gp.status = static_cast<int32_t*>(workspace);
  gp.B = d->batch;
  gp.num_pages = d->num_pages;
  gp.max_pages = d->max_pages_per_req;
  gp.pt_stride = d->page_table_stride;
  gp.timeout_ns = kTimeoutNs;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const int smem = 64 + 1024 + (f8 ? Cfg<true>::kSlotS : Cfg<false>::kSlotS);
  if (cudaMemsetAsync(workspace, 0, 16, stream) != cudaSuccess) return MLA_ERR_CUDA;
  cudaError_t e;
  dim3 grid(d->max_pages_per_req, d->batch);
  if (f8) {
    e = cudaFuncSetAttribute(mla::mla_gather_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) mla::mla_gather_kernel<true><<<grid, 128, smem, stream>>>(gp, maps.s, maps.pe);
  } else {
    e = cudaFuncSetAttribute(mla::mla_gather_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) mla::mla_gather_kernel<false><<<grid, 128, smem, stream>>>(gp, maps.s, maps.pe);
  }
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_selftest_wait_timeout(void* workspace, uint32_t timeout_us, void* stream_v) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  if (timeout_us == 0 || timeout_us > 10000000u) return MLA_ERR_INVALID_ARG;
  int dev = 0, rc;
  if ((rc = current_device(&dev)) != MLA_OK) return rc;
  if ((rc = device_ok(dev)) != MLA_OK) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  if (cudaMemsetAsync(workspace, 0, 16, stream) != cudaSuccess) return MLA_ERR_CUDA;
  mla::mla_wait_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<int32_t*>(workspace),
                                                      static_cast<uint64_t>(timeout_us) * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Allocation-free decode.  Some callers cannot call cudaMalloc: code that
// runs where a device allocation is not allowed or not wanted (an inference
// server that must not allocate in its serving loop, a process that hands
// every byte of device memory to its own pool up front, plug-ins that only
// receive buffers from their host).  mla_decode_noalloc serves them by
// taking its scratch (status words, schedule, split partials) from a static
// device array that lives in this library's module instead of a
// caller-provided workspace.  Every GPU that loads the library holds this
// array until the process exits.
namespace {

// 40 MiB: the split partials of every slice a GB300 runs at once (2 slots
// of 128 x 512 fp32 per slice and row block, 38 MiB) plus the schedule and
// query scales of a batch of about two thousand requests; larger batches
// run on fewer slices
constexpr size_t kNoAllocScratchBytes = size_t(40) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up with the device current (in
// host code the symbol itself is only a stand-in).  It is cached per device
// together with the id of the context it was found in: a device reset
// (cudaDeviceReset, a primary-context reset) creates a new context in which
// the module, and this array, are loaded again, possibly elsewhere, and the
// next call then looks the address up again.
struct NoAllocScratch {
  std::mutex mu;
  void* ptr[64] = {};
  unsigned long long ctx_id[64] = {};
};
NoAllocScratch g_noalloc;

// Id of the current context (unique within the process, never reused), or 0
// when there is none yet or the driver cannot be asked.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

int noalloc_scratch(int device, uint8_t** out) {
  if (device < 0 || device >= 64) return MLA_ERR_INVALID_ARG;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lk(g_noalloc.mu);
  if (!g_noalloc.ptr[device] || id == 0 || g_noalloc.ctx_id[device] != id) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_noalloc.ptr[device] = ptr;
    g_noalloc.ctx_id[device] = current_context_id();  // the lookup made the context current if it was not
  }
  *out = static_cast<uint8_t*>(g_noalloc.ptr[device]);
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_noalloc(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                                  const int32_t* page_table, const int32_t* seq_lens, int32_t q_len, float scale,
                                  float kv_scale, void* out, float* lse, int32_t* status_out, void* stream) {
  int rc = check_call(d, q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, scale, kv_scale, out, lse, status_out);
  if (rc != MLA_OK) return rc;
  int dev = 0;
  if ((rc = current_device(&dev)) != MLA_OK) return rc;
  if ((rc = device_ok(dev)) != MLA_OK) return rc;
  uint8_t* ws = nullptr;
  if ((rc = noalloc_scratch(dev, &ws)) != MLA_OK) return rc;
  // the status words start at zero (the schedule kernel clears them); everything
  // else in the scratch is written before it is read within the call
  return decode_impl(d, q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, scale, kv_scale, out, lse, ws,
                     kNoAllocScratchBytes, true, status_out, stream, nullptr);
}

#ifdef MLA_TRACE
// Trace builds only: copies the event stamps of cluster 0 to host memory.
extern "C" int mla_trace_set_cluster(int cid) {
  return cudaMemcpyToSymbol(mla::g_mla_trace_cid, &cid, sizeof(int)) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
extern "C" int mla_trace_cluster_times(void* host_dst, size_t bytes) {
  if (bytes > sizeof(mla::g_mla_cluster_times)) bytes = sizeof(mla::g_mla_cluster_times);
  return cudaMemcpyFromSymbol(host_dst, mla::g_mla_cluster_times, bytes) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
extern "C" int mla_trace_kernel_times(void* host_dst, int reset) {
  if (cudaMemcpyFromSymbol(host_dst, mla::g_mla_kernel_times, sizeof(mla::g_mla_kernel_times)) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (reset) {
    unsigned long long init[8] = {0, 0, ~0ull, 0, ~0ull, ~0ull, 0, 0};
    if (cudaMemcpyToSymbol(mla::g_mla_kernel_times, init, sizeof(init)) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}
extern "C" int mla_trace_combine_times(void* host_dst, int reset) {
  if (cudaMemcpyFromSymbol(host_dst, mla::g_mla_combine_times, sizeof(mla::g_mla_combine_times)) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (reset) {
    static unsigned long long zeros[4096][4];
    if (cudaMemcpyToSymbol(mla::g_mla_combine_times, zeros, sizeof(zeros)) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}
extern "C" int mla_trace_copy(void* host_dst, size_t bytes) {
  if (bytes > sizeof(mla::g_mla_trace)) bytes = sizeof(mla::g_mla_trace);
  return cudaMemcpyFromSymbol(host_dst, mla::g_mla_trace, bytes) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
#endif
