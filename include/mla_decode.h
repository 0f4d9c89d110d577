/*
 * Paged MLA decode for GB300 (sm_103a): C ABI.
 *
 * The operation (TokenSpeed code audit, mlqm.cn/news/403565, section
 * 完整技术清单 > MLA): every cached token is one latent row of 576 values,
 * [c_kv (512) | k_pe (64)], stored once and used both as the key (all 576
 * values) and as the value (the 512 latent values).  Each query head arrives
 * already absorbed into that space (q_nope 512, q_pe 64).  For request b,
 * draft position i and head h, with n = seq_lens[b] - q_len + i + 1 visible
 * keys:
 *
 *     s_t = (q_nope . c_kv[t] + q_pe . k_pe[t]) * scale
 *     out = sum_t softmax(s)_t * c_kv[t]            (512-d latent, bf16)
 *     lse = ln sum_t exp(s_t)                        (fp32, natural log)
 *
 * The keys are gathered through a page table of 64-token pages (guijiagi.com
 * "推理优化" tag page, KV-cache article, PagedAttention); pages shared by
 * several requests are the same page ids in several table rows and are read
 * in place.  Long contexts are split over the keys and merged by
 * log-sum-exp in a second kernel (same audit section: two-stage split-KV
 * decode with fp32 partials in a workspace).
 *
 * Conventions for every entry point:
 *   - all buffers are owned by the caller; the library never allocates,
 *     frees or synchronises inside mla_decode and never writes the cache,
 *     the page table or the sequence lengths;
 *   - device pointers are CUDA device addresses on the current device;
 *     `stream` is a cudaStream_t passed as void* (NULL = legacy stream);
 *   - work is enqueued on `stream` and runs asynchronously; the call's last
 *     kernel completes only after all of its earlier ones, so a kernel the
 *     caller launches next on `stream` as a programmatic dependent sees all
 *     of the call's output once its griddepcontrol.wait returns;
 *   - the return value is an mla_status; no C++ exception crosses the ABI;
 *   - errors that only the device can see (a page id outside the pool, a
 *     sequence length outside [q_len, max_pages_per_req * 64], a wait that
 *     ran out) are OR-ed into a status word inside the workspace and read
 *     with mla_query_status after the stream is synchronised.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side return codes. */
typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,      /* null pointer, bad dimension, q_len mismatch */
  MLA_ERR_UNSUPPORTED = -2,      /* page_size != 64, num_heads * q_len > 256, unknown cache type */
  MLA_ERR_ALIGNMENT = -3,        /* a pointer breaks the alignment rule of its argument */
  MLA_ERR_WORKSPACE_TOO_SMALL = -4,
  MLA_ERR_CUDA = -5,             /* a CUDA runtime/driver call failed */
  MLA_ERR_DEVICE = -6,           /* the current device is not sm_103a */
  MLA_ERR_SCRATCH_TOO_SMALL = -7 /* mla_decode_noalloc: dimensions need more than its static scratch */
} mla_status;

/* Device-side status bits (word 0 of the workspace). */
enum {
  MLA_DEV_BAD_PAGE_ID = 1,  /* a page id outside [0, num_pages); page 0 was read instead */
  MLA_DEV_BAD_SEQ_LEN = 2,  /* seq_lens[b] outside [q_len, max_pages_per_req*64]; clamped */
  MLA_DEV_TIMEOUT = 4,      /* a bounded wait inside a kernel gave up; outputs are garbage.
                               Words 1..3 of the workspace then hold which wait (an internal
                               tag), its page counter and (cluster << 16 | rank << 8 | warp) */
  MLA_DEV_INTERNAL = 8      /* an internal index check failed (a bug); the write was skipped */
};

typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1 } mla_kv_dtype;

typedef struct {
  int32_t batch;             /* B >= 1 requests */
  int32_t num_heads;         /* H >= 1 absorbed query heads */
  int32_t q_len;             /* draft positions per request; H*q_len <= 256 */
  int32_t page_size;         /* must be 64 */
  int32_t num_pages;         /* pool size; valid page ids are [0, num_pages) */
  int32_t max_pages_per_req; /* columns of the page table a request may use; max_pages_per_req * 64
                                and batch * max_pages_per_req must fit in int32 (else
                                MLA_ERR_UNSUPPORTED) */
  int32_t page_table_stride; /* int32 elements between page-table rows (>= max_pages_per_req) */
  int32_t kv_dtype;          /* mla_kv_dtype */
} mla_dims;

/*
 * Bytes of workspace mla_decode needs for these dimensions on `device`.
 * Depends on the dimensions (cache type included) and the device's SM count
 * only, never on the values in seq_lens, so one allocation serves every step
 * of a batch shape.  With an e4m3 cache it includes 1152 bytes per query row
 * (128 per row block at least) for the queries' e4m3 terms; a workspace
 * without room for them still works, with the attention kernel splitting the
 * queries itself, more slowly.  Returns 0 on invalid dimensions or if the
 * device cannot be queried.
 */
size_t mla_decode_workspace_size(const mla_dims* d, int device);

/*
 * One decode step: three kernels on `stream` (schedule, split-KV attention,
 * log-sum-exp combine; with an e4m3 cache a fourth, the queries' scales and
 * e4m3 terms, beside the schedule).
 *
 *   q_nope      bf16 [B][q_len][H][512], contiguous, 32-byte aligned
 *   q_pe        bf16 [B][q_len][H][64],  contiguous, 32-byte aligned
 *   kv_cache    bf16 or e4m3 [num_pages][64][576]: per token [c_kv | k_pe];
 *               an e4m3 value means code * kv_scale; 16-byte aligned
 *   page_table  int32 [B][page_table_stride]; entries beyond a request's
 *               ceil(seq_len/64) pages are never read
 *   seq_lens    int32 [B]; L_b counts the q_len new tokens, already in the
 *               cache; position i sees keys 0 .. L_b - q_len + i
 *   q_len       must equal d->q_len
 *   scale       softmax scale applied to the whole score (e.g. 1/sqrt(192)); > 0
 *   kv_scale    per-tensor dequantisation scale of an e4m3 cache, > 0 (ignored for bf16)
 *   out         bf16 [B][q_len][H][512], 32-byte aligned (rows are read and written
 *               32 bytes per access)
 *   lse         fp32 [B][q_len][H], natural log of sum exp(score)
 *   workspace   >= mla_decode_workspace_size bytes, 256-byte aligned device memory;
 *               holds the status words, the schedule, fp32 split partials and
 *               (e4m3 cache) the queries' scales and e4m3 terms;
 *               must not be shared by calls that may run concurrently
 */
int mla_decode(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
               const int32_t* page_table, const int32_t* seq_lens, int32_t q_len, float scale,
               float kv_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
               void* stream);

/*
 * mla_decode plus timing marks: records events[0] before the schedule
 * kernel, events[1] before the attention kernel, events[2] after it and
 * events[3] after the combine kernel, all on `stream`.  `events` holds four
 * caller-created cudaEvent_t handles (as void*).  Used by the benchmark to
 * time the attention kernel alone; results are identical to mla_decode.
 */
int mla_decode_profiled(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                        const int32_t* page_table, const int32_t* seq_lens, int32_t q_len, float scale,
                        float kv_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                        void* stream, void* const* events);

/*
 * Copies the device status word of the last mla_decode / mla_gather_rows
 * call that used `workspace` into *device_status (a bitmask of MLA_DEV_*).
 * Synchronises `stream` (it is a diagnostic call, not for the hot path).
 */
int mla_query_status(const void* workspace, void* stream, int32_t* device_status);

/*
 * Test hook for the page-table gather: copies, for every request in order,
 * the raw cache rows of its tokens 0 .. seq_lens[b]-1 into rows_out
 * (row-major [sum_b seq_lens[b]][576] of the cache's element type), using
 * the same tensor-map TMA page loads as the decode kernel.  `row_offsets`
 * is int64 [B+1] (device) with row_offsets[b] = sum_{c<b} seq_lens[c].
 * Device errors go to the status word of `workspace` (>= 256 bytes).
 * batch > 65535 is refused (MLA_ERR_UNSUPPORTED) before anything is enqueued.
 */
int mla_gather_rows(const mla_dims* d, const void* kv_cache, const int32_t* page_table,
                    const int32_t* seq_lens, const int64_t* row_offsets, void* rows_out,
                    void* workspace, void* stream);

/*
 * Self-test of the bounded wait used by every pipeline wait in the kernels:
 * launches one CTA that waits on an mbarrier nothing ever completes, with a
 * limit of `timeout_us` microseconds (1 .. 10^7), then returns.  The
 * workspace status word must read MLA_DEV_TIMEOUT afterwards and the
 * context stays usable.
 */
int mla_selftest_wait_timeout(void* workspace, uint32_t timeout_us, void* stream);

/*
 * Allocation-free variant of mla_decode (no counterpart in the pages: it
 * exists for callers that cannot call cudaMalloc, such as a serving loop
 * that must not allocate, a process whose device memory is all handed to
 * its own pool, or a plug-in that only receives buffers from its host).
 * Same arguments and results as mla_decode, but there is no workspace: the
 * status words, schedule and split partials live in a static 40 MiB device
 * array inside this library (every GPU that loads the library holds it
 * until the process exits).  The caller still passes all inputs and
 * outputs.  Nothing is allocated or freed.
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *     A device reset (cudaDeviceReset, a primary-context reset) loads the
 *     library's device code again: the next call looks the address up
 *     again, so it too belongs outside a capture.
 *   - Each slice of the work needs about G * 0.5 MiB of split partials
 *     (G = ceil(num_heads * q_len / 128)), so the 76 slices (G = 1) or 38
 *     (G = 2) that mla_decode runs on GB300 fit, together with the schedule
 *     of a batch of up to about two thousand requests: there the call runs
 *     as fast as mla_decode.  Larger batches leave less room for partials
 *     and are decoded on fewer slices, more slowly; if even one slice's
 *     partials do not fit (very large batches), the call returns
 *     MLA_ERR_SCRATCH_TOO_SMALL.  With an e4m3 cache the queries' e4m3
 *     terms (147 KB per request and row block) are prepared in the array
 *     only when they fit beside the full partials (about a dozen requests
 *     on GB300); otherwise
 *     the attention kernel splits the queries itself, as fast as mla_decode
 *     with a workspace without room for the terms.
 *   - All calls share the one array, which keeps the last call's contents:
 *     calls that may overlap on the GPU (other streams, other threads)
 *     race and must be serialised by the caller.
 *   - status_out (device int32, may be NULL) receives a copy of the device
 *     status word (MLA_DEV_* bits) at the end of the call, on `stream`.
 */
int mla_decode_noalloc(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                       const int32_t* page_table, const int32_t* seq_lens, int32_t q_len, float scale,
                       float kv_scale, void* out, float* lse, int32_t* status_out, void* stream);

/* Static description of a status code. */
const char* mla_status_string(int status);

/* Number of clusters and CTAs per cluster the attention kernel launches for
 * `d` on `device` (reported by the benchmark): clusters of one S/O CTA pair,
 * G of them per slice of the work (G = ceil(num_heads * q_len / 128)). */
int mla_decode_launch_shape(const mla_dims* d, int device, int32_t* clusters, int32_t* cluster_size);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
