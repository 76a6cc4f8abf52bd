// Stationary-batch hand-off between two ISD steps: the next step's row
// layout and row inputs, from this step's accept and commit results.
//
// Sources: "Introspective Diffusion Language Models" (project page), sections
// "Serving (SGLang)" (stationary-batch decode loop: the batch keeps its
// shape from step to step and the step is replayed from a CUDA graph) and
// "Inference & ISD" (MASK rows propose, clean rows verify); the abstract
// ("stationary-batch scheduler").  A request whose step accepted every
// draft continues FULL: rows [anchor, d_1 .. d_{N-1}, MASK x (N-1)] at
// positions L .. L + 2N - 2, where L is its committed length after this
// step's commit, the anchor is the token it emitted last (not yet in the KV
// cache) and d_k the MASK proposals of this step.  After a rejection it
// continues FRESH: rows [anchor, MASK x (N-1)] at positions L .. L + N - 1.
//
// One kernel: every CTA scans the row counts of all requests (so that no CTA
// waits for another), CTA 0 writes qo_indptr, and each CTA fills the rows of
// its 64 requests (request, position, input token; -1 at MASK rows) and
// advances their counters and token history.
#include <algorithm>

#include "common.cuh"
#include "host_util.h"

namespace idlm {
namespace adv {

constexpr int kThreads = 256;
constexpr int kReqPerCta = 64;

struct Params {
  int C, N, T;
  const uint8_t* mode;         // [C] this step's modes (counters only; may be null)
  const uint8_t* next_mode;    // [C]
  const int32_t* out_tokens;   // [C, N]
  const int32_t* n_out;        // [C]
  const int32_t* n_accepted;   // [C] (counters only; may be null)
  const int32_t* next_drafts;  // [C, N-1]
  const int32_t* seq_lens;     // [C] committed length after this step
  int32_t* qo;                 // [C+1]
  int32_t* row_req;            // [T]
  int32_t* row_pos;            // [T]
  int32_t* row_token;          // [T]
  int32_t* counters;           // [4][C] or null: tokens, forwards, accepted drafts, drafts tested
  int32_t* history;            // [C, hist_cap] or null
  int32_t* hist_len;           // [C]
  int hist_cap;
  int count;                   // 0: first layout of a loop (no step to count)
  int32_t* status;
};

__device__ __forceinline__ int rows_of(const Params& p, int c) {
  return p.next_mode[c] == IDLM_MODE_FULL ? 2 * p.N - 1 : p.N;
}

__global__ void __launch_bounds__(kThreads) advance_kernel(const Params p) {
  __shared__ int warp_sum[kThreads / 32];
  __shared__ int cta_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c_lo = blockIdx.x * kReqPerCta;
  const int c_hi = min(p.C, c_lo + kReqPerCta);
  // rows of requests [0, c_lo): every thread sums a strided share
  int before = 0;
  for (int c = tid; c < c_lo; c += kThreads) before += rows_of(p, c);
#pragma unroll
  for (int o = 16; o; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  if (lane == 0) warp_sum[warp] = before;
  __syncthreads();
  if (tid == 0) {
    int s = 0;
    for (int w = 0; w < kThreads / 32; ++w) s += warp_sum[w];
    cta_base = s;
  }
  __syncthreads();
  // exclusive scan of this CTA's requests (at most 64: two warps' worth)
  __shared__ int first_row[kReqPerCta + 1];
  if (tid == 0) {
    int acc = cta_base;
    for (int c = c_lo; c < c_hi; ++c) {
      first_row[c - c_lo] = acc;
      acc += rows_of(p, c);
    }
    first_row[c_hi - c_lo] = acc;
  }
  __syncthreads();
  if (blockIdx.x == 0 && tid == 0) p.qo[0] = 0;
  for (int c = c_lo + tid; c < c_hi; c += kThreads) p.qo[c + 1] = first_row[c - c_lo + 1];
  // the rows of each request: one warp per request
  const int M = p.N - 1;
  for (int c = c_lo + warp; c < c_hi; c += kThreads / 32) {
    const int r0 = first_row[c - c_lo];
    const bool full = p.next_mode[c] == IDLM_MODE_FULL;
    const int rows = full ? 2 * p.N - 1 : p.N;
    const int ncl = full ? p.N : 1;
    const int no = p.n_out[c];
    const int L = p.seq_lens[c];
    if (no < 1 || no > p.N || L < 0 || r0 + rows > p.T) {
      if (lane == 0) set_status(p.status, IDLM_DEV_BAD_LAYOUT);
      continue;
    }
    const int anchor = p.out_tokens[c * p.N + no - 1];
    for (int r = lane; r < rows; r += 32) {
      int tok;
      if (r == 0) tok = anchor;
      else if (r < ncl) tok = p.next_drafts[c * M + r - 1];
      else tok = -1;
      p.row_req[r0 + r] = c;
      p.row_pos[r0 + r] = L + r;
      p.row_token[r0 + r] = tok;
    }
    if (p.count && lane == 0) {
      if (p.counters) {
        const int na = p.n_accepted ? p.n_accepted[c] : no - 1;
        const bool was_full = p.mode ? p.mode[c] == IDLM_MODE_FULL : false;
        p.counters[c] += no;
        p.counters[p.C + c] += 1;
        p.counters[2 * p.C + c] += na;
        p.counters[3 * p.C + c] += was_full ? min(na + 1, M) : 0;
      }
    }
    if (p.count && p.history && lane < no) {
      const int at = p.hist_len[c] + lane;
      if (at < p.hist_cap) p.history[static_cast<size_t>(c) * p.hist_cap + at] = p.out_tokens[c * p.N + lane];
    }
    __syncwarp();
    if (p.count && p.history && lane == 0) p.hist_len[c] = min(p.hist_len[c] + no, p.hist_cap);
  }
  // rows past the last request: no request
  if (blockIdx.x == gridDim.x - 1) {
    const int used = first_row[c_hi - c_lo];
    for (int t = used + tid; t < p.T; t += kThreads) {
      p.row_req[t] = 0;
      p.row_pos[t] = 0;
      p.row_token[t] = -2;
    }
  }
}

}  // namespace adv
}  // namespace idlm

using namespace idlm;

extern "C" idlm_status idlm_isd_advance(
    int C, int N, int T, const uint8_t* mode, const uint8_t* next_mode, const int32_t* out_tokens,
    const int32_t* n_out, const int32_t* n_accepted, const int32_t* next_drafts,
    const int32_t* seq_lens, int32_t* qo_indptr, int32_t* row_req, int32_t* row_pos,
    int32_t* row_token, int32_t* counters, int32_t* history, int hist_cap, int32_t* hist_len,
    int count, int32_t* status, void* stream) {
  if (!next_mode || !out_tokens || !n_out || !next_drafts || !seq_lens || !qo_indptr ||
      !row_req || !row_pos || !row_token || !status)
    return IDLM_ERR_INVALID_ARG;
  if (C <= 0 || N < 2 || N > 16 || T < C * (2 * N - 1)) return IDLM_ERR_INVALID_ARG;
  if (history && (!hist_len || hist_cap <= 0)) return IDLM_ERR_INVALID_ARG;
  adv::Params p;
  p.C = C;
  p.N = N;
  p.T = T;
  p.mode = mode;
  p.next_mode = next_mode;
  p.out_tokens = out_tokens;
  p.n_out = n_out;
  p.n_accepted = n_accepted;
  p.next_drafts = next_drafts;
  p.seq_lens = seq_lens;
  p.qo = qo_indptr;
  p.row_req = row_req;
  p.row_pos = row_pos;
  p.row_token = row_token;
  p.counters = counters;
  p.history = history;
  p.hist_len = hist_len;
  p.hist_cap = hist_cap;
  p.count = count;
  p.status = status;
  const int grid = (C + adv::kReqPerCta - 1) / adv::kReqPerCta;
  adv::advance_kernel<<<grid, adv::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cuda_status(cudaGetLastError());
}
