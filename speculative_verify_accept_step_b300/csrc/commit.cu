// a8. KV commit / rollback.
//
// Source: "Introspective Diffusion Language Models" (project page), section
// "Serving (SGLang)": paged KV cache.  Only the rows an ISD step keeps -- the
// anchor and its accepted drafts, or a FRESH request's one clean row -- are
// appended; rejected drafts and MASK rows are never written, so rolling them
// back costs nothing.  One CTA per request: it first checks every page and
// slot the commit would touch (all-or-nothing per request), then copies the
// rows with 16-byte vectors and advances the length.
#include "common.cuh"
#include "host_util.h"

namespace idlm {
namespace kvc {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
commit_kernel(uint8_t* k_cache, uint8_t* v_cache, const int32_t* page_table, int max_pages,
              const int32_t* seq_lens_in, int32_t* seq_lens_out, const uint8_t* k_new,
              const uint8_t* v_new, const int32_t* qo_indptr, const int32_t* n_commit,
              int T, int Hkv, int row_bytes, int page_size, int num_pages,
              int32_t* releasable_from, int32_t* status) {
  const int c = blockIdx.x;
  const int L = seq_lens_in[c];
  const int n = n_commit[c];
  const int t0 = qo_indptr[c];
  const int rows = qo_indptr[c + 1] - t0;
  int bad = 0;
  if (L < 0 || n < 0 || n > rows || t0 < 0 || t0 + rows > T) bad = IDLM_DEV_BAD_LAYOUT;
  for (int j = threadIdx.x; j < n && !bad; j += kThreads) {
    const int slot = L + j;
    const int pi = slot / page_size;
    if (pi >= max_pages) {
      bad = IDLM_DEV_SLOT_OVERFLOW;
    } else {
      const int page = page_table[static_cast<size_t>(c) * max_pages + pi];
      if (page < 0 || page >= num_pages) bad = IDLM_DEV_BAD_PAGE;
    }
  }
  if (bad) set_status(status, bad);
  if (__syncthreads_or(bad)) return;

  // copy n rows x Hkv heads of row_bytes each, in 16-byte vectors
  const int vec_per_row = row_bytes / 16;
  const int total = n * Hkv * vec_per_row;
  for (int v = threadIdx.x; v < total; v += kThreads) {
    const int j = v / (Hkv * vec_per_row);
    const int rem = v % (Hkv * vec_per_row);
    const int h = rem / vec_per_row;
    const int x = rem % vec_per_row;
    const int slot = L + j;
    const int page = page_table[static_cast<size_t>(c) * max_pages + slot / page_size];
    const size_t dst = ((static_cast<size_t>(page) * Hkv + h) * page_size + slot % page_size) *
                           static_cast<size_t>(row_bytes) + x * 16;
    const size_t src = (static_cast<size_t>(t0 + j) * Hkv + h) * static_cast<size_t>(row_bytes) + x * 16;
    *reinterpret_cast<uint4*>(k_cache + dst) = *reinterpret_cast<const uint4*>(k_new + src);
    *reinterpret_cast<uint4*>(v_cache + dst) = *reinterpret_cast<const uint4*>(v_new + src);
  }
  __syncthreads();   // every thread has read L before the length moves
  if (threadIdx.x == 0) {
    seq_lens_out[c] = L + n;
    if (releasable_from) releasable_from[c] = (L + n + page_size - 1) / page_size;
  }
}

}  // namespace kvc
}  // namespace idlm

using namespace idlm;

extern "C" idlm_status idlm_kv_commit(
    void* k_cache, void* v_cache, const int32_t* page_table, int max_pages,
    const int32_t* seq_lens_in, int32_t* seq_lens_out, const void* k_new, const void* v_new,
    const int32_t* qo_indptr, const int32_t* n_commit, int C, int T, int Hkv, int D, int page_size,
    int num_pages, int dtype, int32_t* releasable_from, int32_t* status, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!k_cache || !v_cache || !page_table || !seq_lens_in || !seq_lens_out || !k_new || !v_new ||
      !qo_indptr || !n_commit || !status)
    return IDLM_ERR_INVALID_ARG;
  if (C <= 0 || T <= 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages <= 0 || max_pages <= 0)
    return IDLM_ERR_INVALID_ARG;
  if (dtype != IDLM_BF16 && dtype != IDLM_F32) return IDLM_ERR_INVALID_ARG;
  const int row_bytes = D * (dtype == IDLM_BF16 ? 2 : 4);
  if (row_bytes % 16) return IDLM_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return IDLM_ERR_INVALID_ARG;
  kvc::commit_kernel<<<C, kvc::kThreads, 0, stream>>>(
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), page_table, max_pages,
      seq_lens_in, seq_lens_out, static_cast<const uint8_t*>(k_new),
      static_cast<const uint8_t*>(v_new), qo_indptr, n_commit, T, Hkv, row_bytes, page_size,
      num_pages, releasable_from, status);
  return cuda_status(cudaGetLastError());
}
