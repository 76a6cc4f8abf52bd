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
// One kernel: every CTA sums the row counts of the requests before its own
// (so that no CTA waits for another), CTA 0 writes qo_indptr[0], and each CTA
// fills the rows of its 256 requests (request, position, input token; -1 at
// MASK rows) and advances their counters and token history.
#include <algorithm>

#include "common.cuh"
#include "host_util.h"

namespace idlm {
namespace adv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kReqPerCta = kThreads;  // one thread per request in the scalar phase

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

// Two phases per CTA of 256 requests.  Scalar phase: thread j owns request
// c_lo + j and issues all of its loads (mode, emitted count, length) before
// using any, so the CTA pays one memory latency where a serial walk over
// the requests paid one per request; the rows before this CTA come from a
// strided sum over the earlier requests' modes, the rows within it from a
// shuffle scan.  Row phase: the CTA's (request, row) pairs are spread flat
// over its threads, so consecutive threads write consecutive rows.
__global__ void __launch_bounds__(kThreads) advance_kernel(const Params p) {
  __shared__ int warp_rows[kWarps];
  __shared__ int warp_before[kWarps];
  __shared__ int s_r0[kReqPerCta];
  __shared__ int s_rows[kReqPerCta];  // 0 for a request whose inputs are out of range
  __shared__ int s_ncl[kReqPerCta];
  __shared__ int s_pos[kReqPerCta];
  __shared__ int s_anchor[kReqPerCta];
  __shared__ int s_used;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c_lo = blockIdx.x * kReqPerCta;
  const int n_here = min(p.C - c_lo, kReqPerCta);
  const int c = c_lo + tid;
  const bool mine = tid < n_here;
  int nm = 0, no = 0, L = 0;
  if (mine) {
    nm = p.next_mode[c];
    no = p.n_out[c];
    L = p.seq_lens[c];
  }
  int before = 0;
#pragma unroll 4
  for (int k = tid; k < c_lo; k += kThreads) before += rows_of(p, k);
  const bool full = nm == IDLM_MODE_FULL;
  const int rows = mine ? (full ? 2 * p.N - 1 : p.N) : 0;
  int incl = rows;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  if (lane == 31) warp_rows[warp] = incl;
  if (lane == 0) warp_before[warp] = before;
  __syncthreads();
  int r0 = incl - rows;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) r0 += warp_before[w] + (w < warp ? warp_rows[w] : 0);
  if (blockIdx.x == 0 && tid == 0) p.qo[0] = 0;
  if (mine) {
    p.qo[c + 1] = r0 + rows;
    if (tid == n_here - 1) s_used = r0 + rows;
    const bool bad = no < 1 || no > p.N || L < 0 || r0 + rows > p.T;
    if (bad) set_status(p.status, IDLM_DEV_BAD_LAYOUT);
    s_r0[tid] = r0;
    s_rows[tid] = bad ? 0 : rows;
    s_ncl[tid] = full ? p.N : 1;
    s_pos[tid] = L;
    s_anchor[tid] = bad ? 0 : p.out_tokens[c * p.N + no - 1];
    if (!bad && p.count) {
      if (p.counters) {
        const int M = p.N - 1;
        const int na = p.n_accepted ? p.n_accepted[c] : no - 1;
        const bool was_full = p.mode ? p.mode[c] == IDLM_MODE_FULL : false;
        p.counters[c] += no;
        p.counters[p.C + c] += 1;
        p.counters[2 * p.C + c] += na;
        p.counters[3 * p.C + c] += was_full ? min(na + 1, M) : 0;
      }
      if (p.history) {
        const int h = max(p.hist_len[c], 0);
        int32_t* hist = p.history + static_cast<size_t>(c) * p.hist_cap;
        for (int k = 0; k < no && h + k < p.hist_cap; ++k) hist[h + k] = p.out_tokens[c * p.N + k];
        p.hist_len[c] = min(h + no, p.hist_cap);
      }
    }
  }
  __syncthreads();
  const int M = p.N - 1, R = 2 * p.N - 1;
  for (int idx = tid; idx < n_here * R; idx += kThreads) {
    const int j = idx / R, r = idx - j * R;
    if (r >= s_rows[j]) continue;
    const int cj = c_lo + j;
    int tok;
    if (r == 0) tok = s_anchor[j];
    else if (r < s_ncl[j]) tok = p.next_drafts[cj * M + r - 1];
    else tok = -1;
    const int t = s_r0[j] + r;
    p.row_req[t] = cj;
    p.row_pos[t] = s_pos[j] + r;
    p.row_token[t] = tok;
  }
  // rows past the last request: no request
  if (blockIdx.x == gridDim.x - 1) {
    for (int t = s_used + tid; t < p.T; t += kThreads) {
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
