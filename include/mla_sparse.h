/*
 * Paged MLA decode for GB300 (sm_103a): top-k sparse decode.  C ABI.
 *
 * The operation (TokenSpeed code audit, mlqm.cn/news/403565, section
 * 完整技术清单 > Attention 接入 / KV: DeepSeek sparse attention, an indexer
 * selects the top-k latent rows and the decode attends to those only).  The
 * indexer is the caller's; this entry point takes its output, a list of
 * token positions per request and draft position, and computes the decode
 * of mla_decode.h over exactly the listed rows of the paged cache:
 *
 *     for request b, draft position i and head h, with S = the valid
 *     entries of indices[b][i][0 .. topk) (a multiset, in list order):
 *     s_t = (q_nope . c_kv[t] + q_pe . k_pe[t]) * scale       for t in S
 *     out = sum_{t in S} softmax(s)_t * c_kv[t],  lse = ln sum_{t in S} exp(s_t)
 *
 * An entry t is valid when 0 <= t < n, n = seq_lens[b] - q_len + i + 1 the
 * positions draft i may see (causal between drafts, as in mla_decode);
 * -1 marks an unused entry and is skipped silently; any other entry is
 * skipped and raises MLA_DEV_BAD_INDEX.  A repeated position counts as
 * often as it is listed.  A (b, i) with no valid entry raises
 * MLA_DEV_BAD_INDEX and gets out = 0 and lse = -inf (the log of an empty
 * sum: the result under which an empty key set drops out of a log-sum-exp
 * merge).
 *
 * How it runs: a gather kernel packs the selected rows of every (b, i)
 * (the cache's own bytes, bf16 or e4m3) into pages of the workspace; the
 * decode of mla_decode.h then runs over those pages with B * q_len requests
 * of one draft position each, on the caller's queries and outputs in place.
 * Conventions as in mla_decode.h (caller-owned buffers, asynchronous on
 * `stream`, mla_status return, device errors in a status word).
 */
#ifndef MLA_SPARSE_H_
#define MLA_SPARSE_H_

#include <stddef.h>
#include <stdint.h>

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

enum { MLA_DEV_BAD_INDEX = 16 /* a top-k entry outside [-1, n), or no valid entry for a (b, i) */ };

/*
 * Workspace bytes for mla_decode_sparse with dimensions d (as for
 * mla_decode) and `topk` entries per (b, i); depends on d, topk and the
 * device's SM count only.  0 for invalid dimensions or topk < 1.
 */
size_t mla_decode_sparse_workspace_size(const mla_dims* d, int32_t topk, int device);

/*
 *   d, q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, scale,
 *   kv_scale, out, lse, stream: as for mla_decode (same shapes, layouts,
 *               alignment and errors)
 *   indices     int32 [B][q_len][topk] token positions (device), 4-byte aligned
 *   topk        entries per (b, i), 1 .. 65536
 *   B * q_len   at most 65535 (MLA_ERR_UNSUPPORTED beyond; the workspace
 *               size is then 0)
 *   workspace   device, 256-byte aligned, at least
 *               mla_decode_sparse_workspace_size(d, topk) bytes
 *
 * Device-side errors (bad page id, bad sequence length, bad index, a wait
 * that gave up) are read with mla_decode_sparse_query_status after the
 * stream is synchronised.
 */
int mla_decode_sparse(const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache,
                      const int32_t* page_table, const int32_t* seq_lens, const int32_t* indices, int32_t topk,
                      int32_t q_len, float scale, float kv_scale, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, void* stream);

/* The OR of the gather's and the decode's device status bits (synchronises `stream`). */
int mla_decode_sparse_query_status(const mla_dims* d, int32_t topk, const void* workspace, void* stream,
                                   int32_t* status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_SPARSE_H_ */
