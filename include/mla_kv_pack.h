/*
 * Paged MLA decode for GB300 (sm_103a): the cache write that precedes a
 * decode step.  C ABI.
 *
 * The operation (TokenSpeed code audit, mlqm.cn/news/403565, section
 * 完整技术清单 > Attention 接入 / KV: the fused FP8 KV-pack kernel quantises
 * the new tokens' latent rows and scatters them into the paged cache in one
 * launch).  Request b brings num_new new tokens, the last num_new positions
 * of its sequence (seq_lens[b] already counts them, as mla_decode expects):
 * token i of request b sits at position t = seq_lens[b] - num_new + i, in
 * slot t % 64 of page page_table[b * page_table_stride + t / 64].  Its row
 * [c_kv (512) | k_pe (64)] is written there:
 *
 *     e4m3 cache: code = e4m3(x * r) for every value x of the row, with
 *                 r = 1 / kv_scale rounded to fp32 and x * r an fp32
 *                 product rounded to nearest-even, e4m3 the OCP-FP8 E4M3
 *                 encoding rounded to nearest-even and saturated to +-448
 *                 (a NaN value gives a NaN code); one per-tensor kv_scale,
 *                 the one mla_decode multiplies back;
 *     bf16 cache: the row is copied unchanged (kv_scale is ignored).
 *
 * Nothing else of the cache is written; rows are independent, so the order
 * of the writes does not matter (two new rows mapped to one slot leave one
 * of them there).  Conventions as in mla_decode.h: the
 * caller owns every buffer, device pointers are on the current device,
 * `stream` is a cudaStream_t passed as void*, work is enqueued
 * asynchronously and the return value is an mla_status.
 */
#ifndef MLA_KV_PACK_H_
#define MLA_KV_PACK_H_

#include <stddef.h>
#include <stdint.h>

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t batch;             /* B >= 1 requests */
  int32_t num_new;           /* new tokens per request, >= 1 */
  int32_t num_pages;         /* pool size; valid page ids are [0, num_pages) */
  int32_t max_pages_per_req; /* columns of the page table a request may use */
  int32_t page_table_stride; /* int32 elements between page-table rows (>= max_pages_per_req) */
  int32_t kv_dtype;          /* mla_kv_dtype of the cache */
} mla_kv_pack_dims;

/*
 * Quantises (e4m3 cache) or copies (bf16 cache) the new rows into the cache.
 *
 *   d           dimensions; read on the host during the call
 *   rows        bf16 [B][num_new][576], contiguous, 16-byte aligned (device)
 *   page_table  int32 [B][page_table_stride] (device)
 *   seq_lens    int32 [B] (device); each in [num_new, max_pages_per_req * 64]
 *   kv_scale    e4m3 cache: > 0 and finite; bf16 cache: ignored
 *   kv_cache    [num_pages][64][576] of the cache type, 16-byte aligned (device);
 *               only the num_new rows of every request are written
 *   status      int32 [1] (device): MLA_DEV_BAD_PAGE_ID / MLA_DEV_BAD_SEQ_LEN
 *               are OR-ed in for a row whose page id or position is invalid,
 *               and that row is not written; the caller clears it
 *   stream      cudaStream_t as void*
 *
 * Returns MLA_ERR_INVALID_ARG for a null pointer, a dimension below 1, a
 * stride below max_pages_per_req or a bad kv_scale; MLA_ERR_UNSUPPORTED for
 * an unknown cache type; MLA_ERR_ALIGNMENT when rows or kv_cache is not
 * 16-byte aligned; MLA_ERR_CUDA when the launch fails.  With B * num_new
 * rows the launch is one kernel of one warp per row.
 */
int mla_kv_pack(const mla_kv_pack_dims* d, const void* rows, const int32_t* page_table, const int32_t* seq_lens,
                float kv_scale, void* kv_cache, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_KV_PACK_H_ */
