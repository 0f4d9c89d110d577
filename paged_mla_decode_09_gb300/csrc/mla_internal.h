// Library-internal entry points shared between the translation units of
// libmla_decode.so (hidden: not part of the C ABI in include/).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "mla_decode.h"

extern "C" {

// mla_decode writing fp32 out [B][q_len][H][512] (32-byte aligned) instead
// of bf16: the cascade's passes keep their partial results unrounded until
// their merge.  Request b's length is seq_lens[b] - len_offset, or len_fixed
// for every request when len_fixed > 0 (seq_lens is then not read): the
// cascade's suffix pass and prefix pass, without a kernel to rewrite the
// lengths.
__attribute__((visibility("hidden"))) int mla_decode_f32_out(
    const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache, const int32_t* page_table,
    const int32_t* seq_lens, int32_t len_offset, int32_t len_fixed, int32_t q_len, float scale, float kv_scale,
    float* out, float* lse, void* workspace, size_t workspace_bytes, void* stream);

// mla_decode (q_len 1) over the top-k path's packed pick lists, which also
// finishes that path: the gather's status bits (gather_nchunk words per
// list, in workspace the gather wrote before this call's kernels run) are
// OR-ed into the decode's status word, and each list flagged in list_empty
// (no valid pick: decoded over one all-zero key, out = 0) gets lse = -inf.
__attribute__((visibility("hidden"))) int mla_decode_topk_packed(
    const mla_dims* d, const void* q_nope, const void* q_pe, const void* kv_cache, const int32_t* page_table,
    const int32_t* seq_lens, float scale, float kv_scale, void* out, float* lse, void* workspace,
    size_t workspace_bytes, const int32_t* gather_bits, int32_t gather_nchunk, const int32_t* list_empty,
    void* stream);

}  // extern "C"
