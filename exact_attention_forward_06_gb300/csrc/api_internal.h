// api_internal.h -- host-side helpers shared between the C-ABI translation
// units (not part of the public interface).
#pragma once

#include <cstdint>

#include "attn.h"

namespace attn {

// Checks every argument of a paged decode step except its workspace: null or
// misaligned pointers, shapes, Hq % Hkv, scale (ATTN_ERR_INVALID_ARG) and
// d / page_size (ATTN_ERR_UNSUPPORTED).  Touches no device state.
attn_status_t check_decode_args(const void *q, const void *k_pages, const void *v_pages, const int32_t *block_table,
                                const int32_t *seqlens, const void *out, const float *lse, int B, int Hq, int Hkv,
                                int d, int page_size, int num_pages, int max_blocks_per_seq, float scale);

}  // namespace attn
