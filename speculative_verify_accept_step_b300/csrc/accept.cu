// a4-a7. ISD accept: vocab pass, p/q acceptance scan, residual resample,
// bonus / fresh draw, proposals and next state.
//
// Sources: "Introspective Diffusion Language Models" (project page), section
// "Inference & ISD" (MASK positions propose from q, clean positions verify
// with the anchor distribution p, a draft x passes with probability
// min(1, p(x)/q(x))), "Serving (SGLang)" (argmax proposals); "I-DLM -
// Icgozlemsel Difuzyon Dil Modelleri" (GeekNews), sections "I-DLM Yontemi"
// and "Inference & ISD".  Row layout: a FULL request has N clean rows
// [anchor, d_1..d_{N-1}] then N-1 MASK rows; clean row i-1 gives p_i for
// draft d_i, clean row N-1 gives p_N for the bonus slot, MASK row k gives q
// for the next step's draft k.  A FRESH request has one clean row then N-1
// MASK rows.
//
// Kernel 1 (vocab_kernel): one CTA per (row, 8192-entry chunk) streams the
// bf16 logits once with 128-bit loads and keeps the chunk's max (log2 domain),
// sum of 2^(z - max) and argmax; the partials go to the workspace.  The last
// CTA of a request to arrive (atomic count, no waiting) combines the partials
// of the request's rows and runs the per-request tail: Philox uniforms, the
// ratios p_i(d_i)/q_i(d_i) from two single-element gathers, the first
// rejection, the bonus / fresh draw (inverse CDF: pick the chunk from the
// partial sums, then re-read that one chunk), argmax proposals and next state.
// Kernel 2 (residual_kernel): only for requests with a rejection at draft j,
// one CTA per chunk sums max(0, p_j - q_j) over the re-read rows p_j (this
// step) and q_j (the previous step's MASK row); the last CTA draws the token
// by inverse CDF the same way.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "host_util.h"
#include "philox.cuh"

namespace idlm {
namespace acc {

constexpr int kThreads = 256;
constexpr int kVec = 4;                          // 16-byte vectors per thread
constexpr int kSpan = kThreads * 8;              // elements per vector sweep
constexpr int kChunk = kSpan * kVec;             // 8192 elements per CTA
constexpr int kMaxRows = 31;                     // 2N-1 with N <= 16
constexpr float kNegInf = -__builtin_inff();
constexpr float kInf = __builtin_inff();

struct __align__(16) Partial {
  float m;     // max of z = x * log2(e) / T over the chunk (greedy: max x)
  float s;     // sum of 2^(z - m)
  float amax;  // max x
  int aidx;    // first index of the max
};

struct RejInfo {
  int row_p, row_q, j, pad;
  float mp, sp, mq, sq;   // log2-domain max and sum of the two rows
};

struct Params {
  const void* logits;
  const void* prev_logits;
  const int32_t* qo;
  const uint8_t* mode;
  const int32_t* drafts;
  const float* dq_stats;
  const int32_t* prev_row0;
  int32_t* n_accepted;
  int32_t* out_tokens;
  int32_t* n_out;
  int32_t* n_commit;
  int32_t* next_drafts;
  float* next_q_stats;
  uint8_t* next_mode;
  int32_t* next_mask_row0;
  float* row_stats;
  float* dbg;
  Partial* part;      // [T][CH]
  int32_t* req_cnt;   // [C]
  int32_t* rej_flag;  // [C]
  int32_t* res_cnt;   // [C]
  RejInfo* rej;       // [C]
  float* res_part;    // [C][CH]
  int32_t* status;
  uint64_t seed, step;
  int V, C, T, N, CH, greedy, propose, prev_rows;
  float s2;           // log2(e) / T
};

// 8 consecutive logits as floats (V % 8 == 0 keeps vectors inside a row).
template <typename T>
__device__ __forceinline__ void load8(const T* p, float* v);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float* v) {
  const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
  v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
  v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* v) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename T>
__device__ __forceinline__ float load1(const T* p);
template <>
__device__ __forceinline__ float load1<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <>
__device__ __forceinline__ float load1<float>(const float* p) { return *p; }

// ------------------------------------------------------------ block reductions

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = red[0];
  for (int i = 1; i < kThreads / 32; ++i) v = fmaxf(v, red[i]);
  return v;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = 0.f;
  for (int i = 0; i < kThreads / 32; ++i) v += red[i];
  return v;
}

// (value, index) with the larger value, the lower index on ties.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void block_argmax(float& v, int& idx, float* redv, int* redi) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    argmax_merge(v, idx, v2, i2);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    redv[w] = v;
    redi[w] = idx;
  }
  __syncthreads();
  v = redv[0];
  idx = redi[0];
  for (int i = 1; i < kThreads / 32; ++i) argmax_merge(v, idx, redv[i], redi[i]);
}

// Prefix sums over the block in thread order.  Thread t gets the interval
// [lo, hi) of the running sum its value covers; adjacent threads share the
// boundary value bit for bit (no gaps or overlaps from rounding).  Returns the
// block total, which equals the last thread's hi.
__device__ __forceinline__ float block_interval_scan(float v, float* lo, float* hi, float* red) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  float inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, inc, o);
    if (l >= o) inc += n;
  }
  float exc = __shfl_up_sync(0xffffffffu, inc, 1);
  if (l == 0) exc = 0.f;
  __syncthreads();
  if (l == 31) red[w] = inc;
  __syncthreads();
  float before = 0.f;
  for (int i = 0; i < w; ++i) before += red[i];
  float total = before;
  for (int i = w; i < kThreads / 32; ++i) total += red[i];
  *lo = before + exc;
  *hi = before + inc;
  return total;
}

// ----------------------------------------------------- inverse-CDF in a chunk
//
// Weight of element e given its logit(s): Kind 0 = 2^(z - m) (a softmax row),
// Kind 1 = max(0, 2^(zp - mp)/sp - 2^(zq - mq)/sq) (the residual).
struct WeightFn {
  int kind;
  float s2, m, mp, sp, mq, sq;
  __device__ __forceinline__ float operator()(float x, float y) const {
    if (kind == 0) return fast_exp2(x * s2 - m);
    return fmaxf(0.f, fast_exp2(x * s2 - mp) / sp - fast_exp2(y * s2 - mq) / sq);
  }
};

struct SampleSmem {
  float red[kThreads / 32];
  int found;
  int last_pos;
};

// First element e of chunk `ch` (in index order) whose running weight sum
// exceeds `target`; if rounding leaves none, the last element with positive
// weight.  Every thread of the block calls this and gets the answer.
template <typename T>
__device__ int chunk_search(const T* rowx, const T* rowy, int V, int ch, float target,
                            const WeightFn& wf, SampleSmem* sm) {
  if (threadIdx.x == 0) {
    sm->found = 0x7fffffff;
    sm->last_pos = -1;
  }
  __syncthreads();
  float run = 0.f;
  for (int it = 0; it < kVec; ++it) {
    const int e0 = ch * kChunk + it * kSpan + threadIdx.x * 8;
    float w[8];
    float tsum = 0.f;
    if (e0 < V) {
      float xv[8], yv[8];
      load8(rowx + e0, xv);
      if (rowy) load8(rowy + e0, yv);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        w[k] = wf(xv[k], rowy ? yv[k] : 0.f);
        tsum += w[k];
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = 0.f;
    }
    float tlo, thi;
    const float total = block_interval_scan(tsum, &tlo, &thi, sm->red);
    const float lo_abs = run + tlo, hi_abs = run + thi;
    if (lo_abs <= target && target < hi_abs) {
      // the target lies in this thread's 8 elements
      float acc = lo_abs;
      int pick = -1;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc += w[k];
        if (w[k] > 0.f) {
          pick = e0 + k;
          if (acc > target) break;
        }
      }
      if (pick >= 0) atomicMin(&sm->found, pick);
    }
    for (int k = 7; k >= 0; --k)
      if (w[k] > 0.f) {
        atomicMax(&sm->last_pos, e0 + k);
        break;
      }
    run += total;
  }
  __syncthreads();
  const int r = sm->found != 0x7fffffff ? sm->found : sm->last_pos;
  __syncthreads();
  return r;
}

// Walk the chunk masses in order: chunk holding u * total and the offset
// into it.  Thread 0 only.
__device__ __forceinline__ void pick_chunk(const float* mass, int CH, float u, int* ch_out,
                                           float* off_out) {
  float total = 0.f;
  for (int k = 0; k < CH; ++k) total += mass[k];
  const float target = u * total;
  float acc = 0.f;
  int last = -1;
  for (int k = 0; k < CH; ++k) {
    if (mass[k] > 0.f) {
      if (acc + mass[k] > target) {
        *ch_out = k;
        *off_out = target - acc;
        return;
      }
      last = k;
    }
    acc += mass[k];
  }
  *ch_out = last < 0 ? 0 : last;
  *off_out = last < 0 ? 0.f : mass[last];
}

struct DecideSmem {
  float rm[kMaxRows], rs[kMaxRows];
  int ridx[kMaxRows];
  int acc_ok[16];
  float mass[1024];
  int pick_ch;
  float pick_off;
  int n_acc;
  SampleSmem ss;
};

// Inverse-CDF draw from the softmax of local row i of the request.
template <typename T>
__device__ int sample_softmax_row(const Params& p, const T* row, const Partial* parts, float m,
                                  float u, DecideSmem* sm) {
  for (int k = threadIdx.x; k < p.CH; k += kThreads) {
    const float4 q = __ldcg(reinterpret_cast<const float4*>(parts) + k);
    sm->mass[k] = q.y * fast_exp2(q.x - m);
  }
  __syncthreads();
  if (threadIdx.x == 0) pick_chunk(sm->mass, p.CH, u, &sm->pick_ch, &sm->pick_off);
  __syncthreads();
  WeightFn wf{0, p.s2, m, 0.f, 1.f, 0.f, 1.f};
  return chunk_search<T>(row, nullptr, p.V, sm->pick_ch, sm->pick_off, wf, &sm->ss);
}

template <typename T>
__device__ void decide(const Params& p, int c, DecideSmem* sm) {
  const int N = p.N, M = N - 1, V = p.V;
  const int row0 = p.qo[c];
  const int rows = p.qo[c + 1] - row0;
  const bool full = p.mode[c] == IDLM_MODE_FULL;
  const int ncl = full ? N : 1;
  const int prow0 = full ? p.prev_row0[c] : 0;
  if (rows != ncl + M || row0 < 0 || row0 + rows > p.T ||
      (full && (prow0 < 0 || prow0 + M > p.prev_rows))) {
    if (threadIdx.x == 0) set_status(p.status, IDLM_DEV_BAD_LAYOUT);
    return;
  }
  const T* logits = static_cast<const T*>(p.logits);
  const T* prev = static_cast<const T*>(p.prev_logits);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;

  // 1. per-row softmax normaliser and argmax from the chunk partials
  for (int i = w; i < rows; i += kThreads / 32) {
    const float4* pr = reinterpret_cast<const float4*>(p.part + static_cast<size_t>(row0 + i) * p.CH);
    float m = kNegInf;
    for (int k = l; k < p.CH; k += 32) m = fmaxf(m, __ldcg(pr + k).x);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f, av = kNegInf;
    int ai = 0x7fffffff;
    for (int k = l; k < p.CH; k += 32) {
      const float4 q = __ldcg(pr + k);   // (m, s, amax, aidx)
      s += q.y * fast_exp2(q.x - m);
      argmax_merge(av, ai, q.z, __float_as_int(q.w));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, ai, o);
      argmax_merge(av, ai, v2, i2);
    }
    if (l == 0) {
      sm->rm[i] = m;
      sm->rs[i] = p.greedy ? 1.f : s;
      sm->ridx[i] = ai;
    }
  }
  __syncthreads();

  // 2. row statistics in natural units: (max x / T, sum exp(x/T - max))
  const float to_nat = p.greedy ? 1.f : (1.f / kLog2e);
  if (p.row_stats && threadIdx.x < rows) {
    p.row_stats[2 * (row0 + threadIdx.x)] = sm->rm[threadIdx.x] * to_nat;
    p.row_stats[2 * (row0 + threadIdx.x) + 1] = sm->rs[threadIdx.x];
  }
  if (threadIdx.x < M) {
    const int k = threadIdx.x;
    p.next_q_stats[2 * (c * M + k)] = sm->rm[ncl + k] * to_nat;
    p.next_q_stats[2 * (c * M + k) + 1] = sm->rs[ncl + k];
  }

  // 3. verification of the drafts (FULL)
  if (threadIdx.x < 16) sm->acc_ok[threadIdx.x] = 0;
  __syncthreads();
  if (full && threadIdx.x < M) {
    const int i = threadIdx.x;   // draft i+1, verified by clean row i
    const int d = p.drafts[c * M + i];
    float u = isd_uniform(p.seed, p.step, c, kPurposeAccept, i);
    float pv = 0.f, qv = 0.f, ratio = 0.f;
    int ok = 0;
    if (d < 0 || d >= V) {
      set_status(p.status, IDLM_DEV_BAD_TOKEN);
    } else {
      const float xp = load1(logits + static_cast<size_t>(row0 + i) * V + d);
      const float yq = load1(prev + static_cast<size_t>(prow0 + i) * V + d);
      const float mq = p.dq_stats[2 * (c * M + i)];
      const float sq = p.dq_stats[2 * (c * M + i) + 1];
      if (p.greedy) {
        pv = (d == sm->ridx[i]) ? 1.f : 0.f;
        qv = (yq == mq) ? 1.f : 0.f;
      } else {
        pv = fast_exp2(xp * p.s2 - sm->rm[i]) / sm->rs[i];
        qv = fast_exp2(yq * p.s2 - mq * kLog2e) / sq;
      }
      ratio = qv > 0.f ? pv / qv : kInf;
      ok = u < fminf(1.f, ratio);
    }
    sm->acc_ok[i] = ok;
    if (p.dbg) {
      float* db = p.dbg + 4 * (c * M + i);
      db[0] = u;
      db[1] = pv;
      db[2] = qv;
      db[3] = ratio;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    if (full)
      while (n < M && sm->acc_ok[n]) ++n;
    sm->n_acc = n;
  }
  __syncthreads();
  const int n_acc = sm->n_acc;
  const bool rejected = full && n_acc < M;

  // 4. the token that ends the step
  int final_tok = -1;
  if (!rejected) {
    const int i = ncl - 1;   // bonus row (FULL) or the fresh row
    if (p.greedy) {
      final_tok = sm->ridx[i];
    } else {
      const float u = isd_uniform(p.seed, p.step, c, kPurposeSample, 0);
      final_tok = sample_softmax_row<T>(p, logits + static_cast<size_t>(row0 + i) * V,
                                        p.part + static_cast<size_t>(row0 + i) * p.CH, sm->rm[i],
                                        u, sm);
    }
  } else if (p.greedy) {
    final_tok = sm->ridx[n_acc];   // residual of one-hots = argmax of p_j
  } else if (threadIdx.x == 0) {
    RejInfo ri;
    ri.row_p = row0 + n_acc;
    ri.row_q = prow0 + n_acc;
    ri.j = n_acc + 1;
    ri.pad = 0;
    ri.mp = sm->rm[n_acc];
    ri.sp = sm->rs[n_acc];
    ri.mq = p.dq_stats[2 * (c * M + n_acc)] * kLog2e;
    ri.sq = p.dq_stats[2 * (c * M + n_acc) + 1];
    p.rej[c] = ri;
    p.rej_flag[c] = 1;
  }

  // 5. proposals for the next step from the MASK rows
  for (int k = 0; k < M; ++k) {
    int tok;
    if (rejected) {
      tok = -1;
    } else if (p.propose == IDLM_PROPOSE_ARGMAX || p.greedy) {
      tok = sm->ridx[ncl + k];
    } else {
      const float u = isd_uniform(p.seed, p.step, c, kPurposePropose, k);
      tok = sample_softmax_row<T>(p, logits + static_cast<size_t>(row0 + ncl + k) * V,
                                  p.part + static_cast<size_t>(row0 + ncl + k) * p.CH,
                                  sm->rm[ncl + k], u, sm);
    }
    if (threadIdx.x == 0) p.next_drafts[c * M + k] = tok;
  }

  // 6. outputs
  if (threadIdx.x == 0) {
    p.n_accepted[c] = n_acc;
    p.n_out[c] = n_acc + 1;
    p.n_commit[c] = full ? 1 + n_acc : 1;
    p.next_mode[c] = rejected ? IDLM_MODE_FRESH : IDLM_MODE_FULL;
    p.next_mask_row0[c] = row0 + ncl;
  }
  if (threadIdx.x < N) {
    const int t = threadIdx.x;
    int v = -1;
    if (t < n_acc) v = p.drafts[c * M + t];
    else if (t == n_acc) v = final_tok;
    p.out_tokens[c * N + t] = v;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) vocab_kernel(const Params p) {
  __shared__ float redv[kThreads / 32];
  __shared__ int redi[kThreads / 32];
  __shared__ int is_last;
  __shared__ DecideSmem dsm;
  const int row = blockIdx.x / p.CH;
  const int ch = blockIdx.x % p.CH;
  const T* rowp = static_cast<const T*>(p.logits) + static_cast<size_t>(row) * p.V;

  float z[kVec][8];
  float mx = kNegInf, av = kNegInf;
  int ai = 0x7fffffff;
#pragma unroll
  for (int it = 0; it < kVec; ++it) {
    const int e0 = ch * kChunk + it * kSpan + threadIdx.x * 8;
    if (e0 < p.V) {
      float x[8];
      load8(rowp + e0, x);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (x[k] > av) {
          av = x[k];
          ai = e0 + k;
        }
        z[it][k] = p.greedy ? x[k] : x[k] * p.s2;
        mx = fmaxf(mx, z[it][k]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) z[it][k] = kNegInf;
    }
  }
  block_argmax(av, ai, redv, redi);
  const float m = block_max(mx, redv);
  float s = 0.f;
  if (!p.greedy) {
#pragma unroll
    for (int it = 0; it < kVec; ++it)
#pragma unroll
      for (int k = 0; k < 8; ++k) s += fast_exp2(z[it][k] - m);
  }
  s = block_sum(s, redv);

  // request of this row
  int lo = 0, hi = p.C - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.qo[mid] <= row) lo = mid; else hi = mid - 1;
  }
  const int c = lo;
  if (threadIdx.x == 0) {
    Partial pt;
    pt.m = m;
    pt.s = s;
    pt.amax = av;
    pt.aidx = ai;
    p.part[static_cast<size_t>(row) * p.CH + ch] = pt;
    __threadfence();
    const int expect = (p.qo[c + 1] - p.qo[c]) * p.CH;
    const int old = atomicAdd(&p.req_cnt[c], 1);
    is_last = (old == expect - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  decide<T>(p, c, &dsm);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) residual_kernel(const Params p) {
  __shared__ float red[kThreads / 32];
  __shared__ int is_last;
  __shared__ DecideSmem dsm;
  const int c = blockIdx.x / p.CH;
  const int ch = blockIdx.x % p.CH;
  if (p.rej_flag[c] == 0) return;
  const RejInfo ri = p.rej[c];
  const T* rp = static_cast<const T*>(p.logits) + static_cast<size_t>(ri.row_p) * p.V;
  const T* rq = static_cast<const T*>(p.prev_logits) + static_cast<size_t>(ri.row_q) * p.V;
  const WeightFn wf{1, p.s2, 0.f, ri.mp, ri.sp, ri.mq, ri.sq};
  float s = 0.f;
#pragma unroll
  for (int it = 0; it < kVec; ++it) {
    const int e0 = ch * kChunk + it * kSpan + threadIdx.x * 8;
    if (e0 < p.V) {
      float x[8], y[8];
      load8(rp + e0, x);
      load8(rq + e0, y);
#pragma unroll
      for (int k = 0; k < 8; ++k) s += wf(x[k], y[k]);
    }
  }
  s = block_sum(s, red);
  if (threadIdx.x == 0) {
    p.res_part[static_cast<size_t>(c) * p.CH + ch] = s;
    __threadfence();
    const int old = atomicAdd(&p.res_cnt[c], 1);
    is_last = (old == p.CH - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const float u = isd_uniform(p.seed, p.step, c, kPurposeSample, 1);
  for (int k = threadIdx.x; k < p.CH; k += kThreads)
    dsm.mass[k] = __ldcg(p.res_part + static_cast<size_t>(c) * p.CH + k);
  __syncthreads();
  __shared__ int empty_res;
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int k = 0; k < p.CH; ++k) tot += dsm.mass[k];
    empty_res = !(tot > 0.f);
  }
  __syncthreads();
  int tok;
  if (!empty_res) {
    if (threadIdx.x == 0) pick_chunk(dsm.mass, p.CH, u, &dsm.pick_ch, &dsm.pick_off);
    __syncthreads();
    tok = chunk_search<T>(rp, rq, p.V, dsm.pick_ch, dsm.pick_off, wf, &dsm.ss);
  } else {
    // p_j == q_j everywhere: draw from p_j
    tok = sample_softmax_row<T>(p, rp, p.part + static_cast<size_t>(ri.row_p) * p.CH, ri.mp, u,
                                &dsm);
  }
  if (threadIdx.x == 0) {
    p.out_tokens[c * p.N + ri.j - 1] = tok;
    p.rej_flag[c] = 0;
  }
}

inline int chunks_for(int V) { return (V + kChunk - 1) / kChunk; }

size_t workspace_bytes(int C, int T, int V, Params* p, void* base) {
  const int CH = chunks_for(V);
  Carver cv(base);
  Partial* part = cv.take<Partial>(static_cast<size_t>(T) * CH);
  int32_t* cnt = cv.take<int32_t>(static_cast<size_t>(3) * C);   // req_cnt | rej_flag | res_cnt
  RejInfo* rej = cv.take<RejInfo>(C);
  float* res_part = cv.take<float>(static_cast<size_t>(C) * CH);
  if (p) {
    p->part = part;
    p->req_cnt = cnt;
    p->rej_flag = cnt ? cnt + C : nullptr;
    p->res_cnt = cnt ? cnt + 2 * C : nullptr;
    p->rej = rej;
    p->res_part = res_part;
  }
  return cv.used;
}

}  // namespace acc
}  // namespace idlm

using namespace idlm;

extern "C" size_t idlm_isd_accept_workspace_size(int C, int T, int N, int V) {
  if (C <= 0 || T <= 0 || N < 2 || V <= 0) return 0;
  return acc::workspace_bytes(C, T, V, nullptr, nullptr);
}

extern "C" idlm_status idlm_isd_accept(
    const void* logits, int dtype, int V, const int32_t* qo_indptr, const uint8_t* mode,
    const int32_t* drafts, const float* draft_q_stats, const void* prev_logits, int prev_rows,
    const int32_t* prev_mask_row0, int C, int T, int N, float temperature, int proposal_mode,
    uint64_t seed, uint64_t step, int32_t* n_accepted, int32_t* out_tokens, int32_t* n_out,
    int32_t* n_commit, int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
    int32_t* next_mask_row0, float* row_stats, float* dbg, void* workspace,
    size_t workspace_bytes, int32_t* status, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!logits || !qo_indptr || !mode || !drafts || !draft_q_stats || !prev_logits ||
      !prev_mask_row0 || !n_accepted || !out_tokens || !n_out || !n_commit || !next_drafts ||
      !next_q_stats || !next_mode || !next_mask_row0 || !status)
    return IDLM_ERR_INVALID_ARG;
  if (C <= 0 || T <= 0 || V <= 0 || N < 2 || N > 16 || prev_rows <= 0 || !(temperature >= 0.f) ||
      (proposal_mode != IDLM_PROPOSE_ARGMAX && proposal_mode != IDLM_PROPOSE_SAMPLE))
    return IDLM_ERR_INVALID_ARG;
  if (dtype != IDLM_BF16 && dtype != IDLM_F32) return IDLM_ERR_INVALID_ARG;
  if (V % 8) return IDLM_ERR_UNSUPPORTED;
  const int CH = acc::chunks_for(V);
  if (CH > 1024) return IDLM_ERR_UNSUPPORTED;
  const size_t elem = dtype == IDLM_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(prev_logits)) & 15)
    return IDLM_ERR_INVALID_ARG;
  (void)elem;
  acc::Params p;
  if (!workspace || workspace_bytes < acc::workspace_bytes(C, T, V, nullptr, nullptr))
    return IDLM_ERR_WORKSPACE;
  acc::workspace_bytes(C, T, V, &p, workspace);
  p.logits = logits;
  p.prev_logits = prev_logits;
  p.qo = qo_indptr;
  p.mode = mode;
  p.drafts = drafts;
  p.dq_stats = draft_q_stats;
  p.prev_row0 = prev_mask_row0;
  p.n_accepted = n_accepted;
  p.out_tokens = out_tokens;
  p.n_out = n_out;
  p.n_commit = n_commit;
  p.next_drafts = next_drafts;
  p.next_q_stats = next_q_stats;
  p.next_mode = next_mode;
  p.next_mask_row0 = next_mask_row0;
  p.row_stats = row_stats;
  p.dbg = dbg;
  p.status = status;
  p.seed = seed;
  p.step = step;
  p.V = V;
  p.C = C;
  p.T = T;
  p.N = N;
  p.CH = CH;
  p.greedy = temperature == 0.f;
  p.propose = proposal_mode;
  p.prev_rows = prev_rows;
  p.s2 = p.greedy ? 1.f : kLog2e / temperature;

  cudaError_t e = cudaMemsetAsync(p.req_cnt, 0, sizeof(int32_t) * 3 * static_cast<size_t>(C), stream);
  if (e != cudaSuccess) return IDLM_ERR_CUDA;
  if (dtype == IDLM_BF16) {
    acc::vocab_kernel<__nv_bfloat16><<<T * CH, acc::kThreads, 0, stream>>>(p);
    acc::residual_kernel<__nv_bfloat16><<<C * CH, acc::kThreads, 0, stream>>>(p);
  } else {
    acc::vocab_kernel<float><<<T * CH, acc::kThreads, 0, stream>>>(p);
    acc::residual_kernel<float><<<C * CH, acc::kThreads, 0, stream>>>(p);
  }
  return cuda_status(cudaGetLastError());
}

// ------------------------------------------------------- allocation-free entry
//
// Some callers cannot allocate device memory at all: a plugin whose host
// process owns every byte of the GPU and hands out no scratch, or a decode
// loop that runs under a fixed memory budget and must not call the allocator
// once it is running.  For them, idlm_isd_accept_noalloc runs the same accept
// step with its scratch in a fixed array compiled into this library.

namespace idlm {
namespace acc {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;   // 4 MiB, per GPU
static __device__ __align__(256) uint8_t g_accept_scratch[kStaticScratchBytes];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};
}  // namespace

// Device address of g_accept_scratch on the current device, looked up once
// per device.  In host code the array's name is only a host-side handle; the
// kernels need the address cudaGetSymbolAddress returns.
void* static_scratch() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace acc
}  // namespace idlm

extern "C" idlm_status idlm_isd_accept_noalloc(
    const void* logits, int dtype, int V, const int32_t* qo_indptr, const uint8_t* mode,
    const int32_t* drafts, const float* draft_q_stats, const void* prev_logits, int prev_rows,
    const int32_t* prev_mask_row0, int C, int T, int N, float temperature, int proposal_mode,
    uint64_t seed, uint64_t step, int32_t* n_accepted, int32_t* out_tokens, int32_t* n_out,
    int32_t* n_commit, int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
    int32_t* next_mask_row0, float* row_stats, float* dbg, int32_t* status, void* stream) {
  if (C <= 0 || T <= 0 || V <= 0) return IDLM_ERR_INVALID_ARG;
  if (acc::workspace_bytes(C, T, V, nullptr, nullptr) > acc::kStaticScratchBytes)
    return IDLM_ERR_WORKSPACE;
  void* scratch = acc::static_scratch();
  if (!scratch) return IDLM_ERR_CUDA;
  return idlm_isd_accept(logits, dtype, V, qo_indptr, mode, drafts, draft_q_stats, prev_logits,
                         prev_rows, prev_mask_row0, C, T, N, temperature, proposal_mode, seed,
                         step, n_accepted, out_tokens, n_out, n_commit, next_drafts,
                         next_q_stats, next_mode, next_mask_row0, row_stats, dbg, scratch,
                         acc::kStaticScratchBytes, status, stream);
}
