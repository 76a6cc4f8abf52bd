// a8. KV commit / rollback.
//
// Source: "Introspective Diffusion Language Models" (project page), section
// "Serving (SGLang)": paged KV cache.  Only the rows an ISD step keeps -- the
// anchor and its accepted drafts, or a FRESH request's one clean row -- are
// appended; rejected drafts and MASK rows are never written, so rolling them
// back costs nothing.  One CTA per request: it first checks every page and
// slot the commit would touch (all-or-nothing per request), then copies the
// rows with 16-byte vectors and advances the length.
#include "commit.cuh"
#include "host_util.h"

namespace idlm {
namespace kvc {

constexpr int kThreads = 256;

// One CTA per request.
__global__ void __launch_bounds__(kThreads) commit_kernel(const CommitArgs a, const int32_t* n_commit) {
  commit_request(a, blockIdx.x, n_commit[blockIdx.x]);
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
  if (!qo_indptr || !n_commit || !status || C <= 0 || T <= 0) return IDLM_ERR_INVALID_ARG;
  int row_bytes = 0;
  const idlm_status rc = commit_check(k_cache, v_cache, page_table, max_pages, seq_lens_in,
                                      seq_lens_out, k_new, v_new, Hkv, D, page_size, num_pages,
                                      dtype, &row_bytes);
  if (rc != IDLM_OK) return rc;
  CommitArgs a;
  a.k_cache = static_cast<uint8_t*>(k_cache);
  a.v_cache = static_cast<uint8_t*>(v_cache);
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.seq_lens_in = seq_lens_in;
  a.seq_lens_out = seq_lens_out;
  a.k_new = static_cast<const uint8_t*>(k_new);
  a.v_new = static_cast<const uint8_t*>(v_new);
  a.qo_indptr = qo_indptr;
  a.T = T;
  a.Hkv = Hkv;
  a.row_bytes = row_bytes;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.releasable_from = releasable_from;
  a.status = status;
  kvc::commit_kernel<<<C, kvc::kThreads, 0, stream>>>(a, n_commit);
  return cuda_status(cudaGetLastError());
}
