// a8. KV commit / rollback of one request, for a whole CTA.
//
// Source: "Introspective Diffusion Language Models" (project page), section
// "Serving (SGLang)": paged KV cache.  Only the rows an ISD step keeps -- the
// anchor and its accepted drafts, or a FRESH request's one clean row -- are
// appended; rejected drafts and MASK rows are never written, so rolling them
// back costs nothing.  The CTA first checks every page and slot the commit
// would touch (all-or-nothing per request), then copies the rows with 16-byte
// vectors and advances the length.  Used by idlm_kv_commit (one CTA per
// request) and by the fused accept + commit (a work item of the accept's
// residual kernel).
#pragma once

#include "common.cuh"

namespace idlm {

struct CommitArgs {
  uint8_t* k_cache;
  uint8_t* v_cache;
  const int32_t* page_table;
  int max_pages;
  const int32_t* seq_lens_in;
  int32_t* seq_lens_out;
  const uint8_t* k_new;
  const uint8_t* v_new;
  const int32_t* qo_indptr;
  int T, Hkv, row_bytes, page_size, num_pages;
  int32_t* releasable_from;   // or null
  int32_t* status;
};

// Every thread of the CTA calls this with the same c and n.
__device__ __forceinline__ void commit_request(const CommitArgs& a, int c, int n) {
  const int L = a.seq_lens_in[c];
  const int t0 = a.qo_indptr[c];
  const int rows = a.qo_indptr[c + 1] - t0;
  int bad = 0;
  if (L < 0 || n < 0 || n > rows || t0 < 0 || t0 + rows > a.T) bad = IDLM_DEV_BAD_LAYOUT;
  for (int j = threadIdx.x; j < n && !bad; j += blockDim.x) {
    const int slot = L + j;
    const int pi = slot / a.page_size;
    if (pi >= a.max_pages) {
      bad = IDLM_DEV_SLOT_OVERFLOW;
    } else {
      const int page = a.page_table[static_cast<size_t>(c) * a.max_pages + pi];
      if (page < 0 || page >= a.num_pages) bad = IDLM_DEV_BAD_PAGE;
    }
  }
  if (bad) set_status(a.status, bad);
  if (__syncthreads_or(bad)) return;

  // copy n rows x Hkv heads of row_bytes each, in 16-byte vectors
  const int vec_per_row = a.row_bytes / 16;
  const int total = n * a.Hkv * vec_per_row;
  for (int v = threadIdx.x; v < total; v += blockDim.x) {
    const int j = v / (a.Hkv * vec_per_row);
    const int rem = v % (a.Hkv * vec_per_row);
    const int h = rem / vec_per_row;
    const int x = rem % vec_per_row;
    const int slot = L + j;
    const int page = a.page_table[static_cast<size_t>(c) * a.max_pages + slot / a.page_size];
    const size_t dst = ((static_cast<size_t>(page) * a.Hkv + h) * a.page_size + slot % a.page_size) *
                           static_cast<size_t>(a.row_bytes) + x * 16;
    const size_t src =
        (static_cast<size_t>(t0 + j) * a.Hkv + h) * static_cast<size_t>(a.row_bytes) + x * 16;
    *reinterpret_cast<uint4*>(a.k_cache + dst) = *reinterpret_cast<const uint4*>(a.k_new + src);
    *reinterpret_cast<uint4*>(a.v_cache + dst) = *reinterpret_cast<const uint4*>(a.v_new + src);
  }
  __syncthreads();   // every thread has read L before the length moves
  if (threadIdx.x == 0) {
    a.seq_lens_out[c] = L + n;
    if (a.releasable_from) a.releasable_from[c] = (L + n + a.page_size - 1) / a.page_size;
  }
}

// Host-side checks shared by the commit entry points.
inline idlm_status commit_check(void* k_cache, void* v_cache, const int32_t* page_table,
                                int max_pages, const int32_t* seq_lens_in,
                                int32_t* seq_lens_out, const void* k_new, const void* v_new,
                                int Hkv, int D, int page_size, int num_pages, int dtype,
                                int* row_bytes) {
  if (!k_cache || !v_cache || !page_table || !seq_lens_in || !seq_lens_out || !k_new || !v_new)
    return IDLM_ERR_INVALID_ARG;
  if (Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages <= 0 || max_pages <= 0)
    return IDLM_ERR_INVALID_ARG;
  if (dtype != IDLM_BF16 && dtype != IDLM_F32) return IDLM_ERR_INVALID_ARG;
  *row_bytes = D * (dtype == IDLM_BF16 ? 2 : 4);
  if (*row_bytes % 16) return IDLM_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return IDLM_ERR_INVALID_ARG;
  return IDLM_OK;
}

}  // namespace idlm
