/*
 * Paged MLA decode for GB300 (sm_103a): cascade decode over a shared
 * prefix.  C ABI.
 *
 * The operation is exactly the decode of mla_decode.h; only the way it is
 * computed differs.  It serves batches whose requests share a prefix of
 * their sequences, stored once (TokenSpeed code audit, mlqm.cn/news/403565,
 * section 调度器 / KV 缓存: prefix pages shared by reference through the
 * page table, a ~91 % prefix-cache hit rate on agentic traffic).  The first
 * prefix_pages columns of every page-table row hold the same page ids, so
 * every request's first prefix_pages * 64 tokens are the same rows.
 *
 * How it runs:
 *   1. prefix pass: the decode of mla_decode.h over the prefix pages only,
 *      with the query rows of g = 128 / (q_len * H) consecutive requests
 *      (when that divides; else g = 1) as the rows of one request (every
 *      draft sees the whole prefix, so no causal mask applies there): with
 *      H = 64 two requests fill the 128 rows the MMA computes, instead of
 *      one request and 64 padding rows;
 *   2. suffix pass: the decode of mla_decode.h over each request's pages
 *      after the prefix (lengths seq_lens[b] - prefix_pages * 64, causal
 *      between drafts as usual);
 *   3. a merge of the two (out, lse) per query row by log-sum-exp (the
 *      split-KV merge: section 完整技术清单 > MLA), which also checks that
 *      every row's prefix columns equal row 0's.
 * The passes keep their results in fp32 until the merge, which rounds to
 * bf16 once.  The three run on `stream` in this order.  Conventions as in
 * mla_decode.h.
 */
#ifndef MLA_CASCADE_H_
#define MLA_CASCADE_H_

#include <stddef.h>
#include <stdint.h>

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

enum { MLA_DEV_BAD_PREFIX = 32 /* a page-table row's prefix columns differ from row 0's */ };

/* Workspace bytes for mla_decode_cascade; 0 for invalid arguments. */
size_t mla_decode_cascade_workspace_size(const mla_dims* d, int32_t prefix_pages, int device);

/*
 *   d, q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, scale,
 *   kv_scale, out, lse, stream: as for mla_decode
 *   prefix_pages  1 .. max_pages_per_req - 1 shared leading page-table
 *                 columns; every seq_lens[b] must be at least
 *                 prefix_pages * 64 + q_len (the drafts are not in the
 *                 prefix), else MLA_DEV_BAD_SEQ_LEN is raised
 *   workspace     256-byte aligned, >= mla_decode_cascade_workspace_size
 *
 * Device errors (including MLA_DEV_BAD_PREFIX) are read with
 * mla_decode_cascade_query_status after the stream is synchronised.
 */
int mla_decode_cascade(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                       const int32_t* page_table, const int32_t* seq_lens, int32_t prefix_pages, int32_t q_len,
                       float scale, float kv_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                       void* stream);

/* The OR of every pass's device status bits (synchronises `stream`). */
int mla_decode_cascade_query_status(const mla_dims* d, int32_t prefix_pages, const void* workspace, void* stream,
                                    int32_t* status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_CASCADE_H_ */
