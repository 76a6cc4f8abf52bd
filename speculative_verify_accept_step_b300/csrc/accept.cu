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
// Kernel 1 (vocab_stream_kernel) is the only pass over all logits.  A
// persistent grid (one CTA per SM) splits the list of 8 KB chunks of all rows
// evenly; a producer thread streams each CTA's chunks into a 26-stage
// shared-memory ring with 1-D bulk copies (cp.async.bulk, mbarrier
// completion), and eight consumer warps each take whole chunks: packed
// bf16x2 maxima per group of 64 values, one exp2 per value for the sum, and
// the first index of the chunk maximum.  Every chunk leaves one partial
// (max, sum, max value, argmax) in the workspace; nothing is decided here.
//
// Kernels 2 and 3 are launched as programmatic dependents of the kernel
// before them (they start early and wait in griddepcontrol.wait).
// Kernel 2 (decide_kernel), one CTA per request, gathers the draft logits
// before the wait, then combines the request's partials, runs the acceptance
// scan, writes every output and draws the bonus / fresh token (and
// SAMPLE-mode proposals): the draw picks the chunk from kernel 1's partial
// sums and searches only that chunk.  After a rejection at draft j it leaves
// a decision record instead, and kernel 3 (residual_kernel), one CTA per
// (request, chunk), sums the residual max(0, p_j - q_j) over each chunk; the
// last CTA of the request to finish picks the chunk from those sums and
// searches it.  Kernel-3 CTAs of other requests leave after one read.  Draws
// are inverse-CDF in vocabulary order.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "host_util.h"
#include "philox.cuh"

namespace idlm {
namespace acc {

constexpr int kItemBytes = 8192;                 // one chunk of a row
constexpr int kStages = 26;                      // kernel-1 ring depth
constexpr int kCWarps = 8;                       // kernel-1 consumer warps
constexpr int kK1Threads = 32 * (kCWarps + 1);
constexpr size_t kK1Smem = 1024 + size_t(kStages) * kItemBytes + 2 * kStages * 8;
constexpr int kK2Threads = 128;
constexpr int kRounds = kItemBytes / 16 / kK2Threads;   // vectors of a chunk per kernel-2 thread
constexpr int kMaxRows = 31;                     // 2N-1 with N <= 16
constexpr int kMaxChunks = 1024;
constexpr float kNegInf = -__builtin_inff();
constexpr float kInf = __builtin_inff();
constexpr uint32_t kNegInfBf2 = 0xff80ff80u;     // two bf16 -inf

struct __align__(16) Partial {
  float m;     // max of z = x * log2(e) / T over the chunk (greedy: max x)
  float s;     // sum of 2^(z - m) (greedy: 1)
  float amax;  // max x
  int aidx;    // first index of the max
};

struct __align__(16) Decision {
  int residual;         // 1: a rejection whose token comes from the residual
  int row_p, row_q, n_acc;
  float mp, isp, mq, isq;
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
  float* res_part;    // [C][CH] residual mass per chunk
  int32_t* res_cnt;   // [C] residual chunks finished (zeroed by kernel 2)
  Decision* dec;      // [C] acceptance result, kernel 2 -> kernel 3
  int32_t* status;
  uint64_t seed, step;
  int V, C, T, N, CH, chunk, greedy, propose, prev_rows;
  float s2;           // log2(e) / T
};

template <typename T>
__device__ __forceinline__ float load1(const T* p);
template <>
__device__ __forceinline__ float load1<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <>
__device__ __forceinline__ float load1<float>(const float* p) { return *p; }

// (value, index) with the larger value, the lower index on ties.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// Values of one 16-byte vector as floats: 8 bf16 or 4 fp32.
template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ __forceinline__ static void get(const uint4& w, float* v) {
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
    v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
    v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  }
  __device__ __forceinline__ static uint4 neg_inf() {
    return make_uint4(kNegInfBf2, kNegInfBf2, kNegInfBf2, kNegInfBf2);
  }
};
template <>
struct Vec<float> {
  static constexpr int kN = 4;
  __device__ __forceinline__ static void get(const uint4& w, float* v) {
    v[0] = __uint_as_float(w.x); v[1] = __uint_as_float(w.y);
    v[2] = __uint_as_float(w.z); v[3] = __uint_as_float(w.w);
  }
  __device__ __forceinline__ static uint4 neg_inf() {
    const uint32_t n = __float_as_uint(kNegInf);
    return make_uint4(n, n, n, n);
  }
};

// Maximum of the 32 values of one lane's group (8 vectors).
template <typename T>
__device__ __forceinline__ float group_max(const uint4* v);
template <>
__device__ __forceinline__ float group_max<__nv_bfloat16>(const uint4* v) {
  uint32_t a = bmax2(bmax2(v[0].x, v[0].y), bmax2(v[0].z, v[0].w));
  uint32_t b = bmax2(bmax2(v[1].x, v[1].y), bmax2(v[1].z, v[1].w));
#pragma unroll
  for (int j = 2; j < 8; j += 2) {
    a = bmax2(a, bmax2(bmax2(v[j].x, v[j].y), bmax2(v[j].z, v[j].w)));
    b = bmax2(b, bmax2(bmax2(v[j + 1].x, v[j + 1].y), bmax2(v[j + 1].z, v[j + 1].w)));
  }
  a = bmax2(a, b);
  return fmaxf(bf16_lo(a), bf16_hi(a));
}
template <>
__device__ __forceinline__ float group_max<float>(const uint4* v) {
  float a = kNegInf, b = kNegInf;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    a = fmaxf(a, fmaxf(__uint_as_float(v[j].x), __uint_as_float(v[j].y)));
    b = fmaxf(b, fmaxf(__uint_as_float(v[j].z), __uint_as_float(v[j].w)));
  }
  return fmaxf(a, b);
}

// ----------------------------------------------------------------- kernel 1
//
// One warp reduces one chunk held in shared memory at `sbase` (cnt values,
// element e0 of the row first).  Lane l reads vectors l, l+32, ... (no bank
// conflicts) in groups of 8 vectors; each group updates the lane's running
// (max, sum) with one rescale and records where the lane's maximum first
// rose.  The chunk's argmax is found afterwards by re-reading only that
// group in the lanes that hold the chunk maximum.
template <typename T>
__device__ __forceinline__ Partial consume_chunk(uint32_t sbase, int cnt, int e0, float s2,
                                                 bool greedy, int lane) {
  constexpr int EV = Vec<T>::kN;
  const int nvec = cnt / EV;
  float m_run = kNegInf, s_run = 0.f, bx = kNegInf;
  int bg = -1;
  for (int g0 = 0; g0 < nvec; g0 += 256) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int idx = g0 + j * 32 + lane;
      v[j] = idx < nvec ? lds128(sbase + idx * 16) : Vec<T>::neg_inf();
    }
    const float gm = group_max<T>(v);
    if (gm > bx) {
      bx = gm;
      bg = g0;
    }
    if (!greedy) {
      const float mz = gm * s2;
      if (mz > m_run) {
        s_run = s_run * fast_exp2(m_run - mz);
        m_run = mz;
      }
      if (m_run > kNegInf) {
        const float nm = -m_run;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float x[EV];
          Vec<T>::get(v[j], x);
#pragma unroll
          for (int k = 0; k < EV; ++k) a[k & 3] += fast_exp2(fmaf(x[k], s2, nm));
        }
        s_run += (a[0] + a[1]) + (a[2] + a[3]);
      }
    }
  }
  // (max, sum) over the warp
  float M = m_run;
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float S = m_run > kNegInf ? s_run * fast_exp2(m_run - M) : 0.f;
#pragma unroll
  for (int o = 16; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  // first index of the chunk maximum
  float BX = bx;
#pragma unroll
  for (int o = 16; o; o >>= 1) BX = fmaxf(BX, __shfl_xor_sync(0xffffffffu, BX, o));
  int idx = 0x7fffffff;
  if (bg >= 0 && bx == BX) {
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      const int vi = bg + j * 32 + lane;
      if (vi < nvec) {
        float x[EV];
        Vec<T>::get(lds128(sbase + vi * 16), x);
#pragma unroll
        for (int k = EV - 1; k >= 0; --k)
          if (x[k] == BX) idx = vi * EV + k;
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
  Partial pt;
  pt.m = greedy ? BX : M;
  pt.s = greedy ? 1.f : S;
  pt.amax = BX;
  pt.aidx = idx == 0x7fffffff ? idx : e0 + idx;
  return pt;
}

template <typename T>
__global__ void __launch_bounds__(kK1Threads, 1) vocab_stream_kernel(const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + size_t(kStages) * kItemBytes);
  uint64_t* empty = full + kStages;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  griddep_launch_dependents();

  const long long W = static_cast<long long>(p.T) * p.CH;
  const long long lo = W * blockIdx.x / gridDim.x;
  const long long hi = W * (blockIdx.x + 1) / gridDim.x;
  const int n = static_cast<int>(hi - lo);
  const T* logits = static_cast<const T*>(p.logits);

  if (warp == kCWarps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      int row = static_cast<int>(lo / p.CH), ch = static_cast<int>(lo % p.CH);
      for (int j = 0; j < n; ++j, ++ch) {
        if (ch == p.CH) {
          ch = 0;
          ++row;
        }
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!mbar_wait_bounded(&empty[s], ph ^ 1, &abort_flag, p.status)) break;
        const int e0 = ch * p.chunk;
        const uint32_t bytes = static_cast<uint32_t>(min(p.chunk, p.V - e0) * sizeof(T));
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(base + size_t(s) * kItemBytes, logits + static_cast<size_t>(row) * p.V + e0,
                 bytes, &full[s]);
        ++issued;
      }
      // every issued copy must land before the CTA may exit
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, nullptr, p.status);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  int row = static_cast<int>(lo / p.CH), ch = static_cast<int>(lo % p.CH) + warp;
  for (int j = warp; j < n; j += kCWarps, ch += kCWarps) {
    while (ch >= p.CH) {
      ch -= p.CH;
      ++row;
    }
    const int s = j % kStages;
    const uint32_t ph = (j / kStages) & 1;
    if (!mbar_wait_bounded(&full[s], ph, &abort_flag, p.status)) break;
    const size_t item = static_cast<size_t>(row) * p.CH + ch;
    const int e0 = ch * p.chunk;
    const int cnt = min(p.chunk, p.V - e0);
    const Partial pt =
        consume_chunk<T>(smem_u32(base + size_t(s) * kItemBytes), cnt, e0, p.s2, p.greedy, lane);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty[s]);
      p.part[item] = pt;
    }
  }
}

// ----------------------------------------------------------------- kernel 2

// Weight of an element given its logit(s): kind 0 = 2^(x s2 - m) (a softmax
// row), kind 1 = max(0, 2^(x s2 - mp) / sp - 2^(y s2 - mq) / sq) (the
// residual of p_j over q_j).
struct WeightFn {
  int kind;
  float s2, m, mp, isp, mq, isq;
  __device__ __forceinline__ float operator()(float x, float y) const {
    if (kind == 0) return fast_exp2(fmaf(x, s2, -m));
    return fmaxf(0.f, fast_exp2(fmaf(x, s2, -mp)) * isp - fast_exp2(fmaf(y, s2, -mq)) * isq);
  }
};

struct DecideSmem {
  float rm[kMaxRows], rs[kMaxRows];
  int ridx[kMaxRows];
  float xp[16], yq[16];
  int dtok[16];
  int acc_ok[16];
  float mass[kMaxChunks];
  float red[kRounds][kK2Threads / 32];
  int found, last_pos;
  int pick_ch;
  float pick_off;
  int n_acc;
  int is_last;
};

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = 0.f;
  for (int i = 0; i < kK2Threads / 32; ++i) v += red[i];
  return v;
}

// Weights of the values in vector `vi` of a chunk (row y optional).
template <typename T>
__device__ __forceinline__ void vec_weights(const uint4* xs, const uint4* ys, int vi,
                                            const WeightFn& wf, float* w) {
  constexpr int EV = Vec<T>::kN;
  float x[EV], y[EV];
  Vec<T>::get(__ldg(xs + vi), x);
  if (ys) {
    Vec<T>::get(__ldg(ys + vi), y);
  } else {
#pragma unroll
    for (int k = 0; k < EV; ++k) y[k] = 0.f;
  }
#pragma unroll
  for (int k = 0; k < EV; ++k) w[k] = wf(x[k], y[k]);
}

// Inverse CDF inside one chunk (global memory, `cnt` values from xs[0]):
// the first element in index order whose running weight sum exceeds
// `target`; if rounding leaves none, the last element with positive weight.
// Element order is (round k, thread t, value): round k covers vectors
// [128k, 128k + 128).  Adjacent intervals share their boundary value bit for
// bit, so no target falls in a gap.  Every thread returns the answer
// (chunk-relative index, or -1 if every weight is zero).
template <typename T>
__device__ int chunk_search(const uint4* xs, const uint4* ys, int cnt, float target,
                            const WeightFn& wf, DecideSmem& sm) {
  constexpr int EV = Vec<T>::kN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvec = cnt / EV;
  float w[kRounds][EV];
  float inc[kRounds], exc[kRounds];
#pragma unroll
  for (int k = 0; k < kRounds; ++k) {
    const int vi = k * kK2Threads + tid;
    if (vi < nvec) {
      vec_weights<T>(xs, ys, vi, wf, w[k]);
    } else {
#pragma unroll
      for (int e = 0; e < EV; ++e) w[k][e] = 0.f;
    }
  }
#pragma unroll
  for (int k = 0; k < kRounds; ++k) {
    float t = 0.f;
#pragma unroll
    for (int e = 0; e < EV; ++e) t += w[k][e];
    inc[k] = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float nb = __shfl_up_sync(0xffffffffu, inc[k], o);
      if (lane >= o) inc[k] += nb;
    }
    exc[k] = __shfl_up_sync(0xffffffffu, inc[k], 1);
    if (lane == 0) exc[k] = 0.f;
  }
  if (tid == 0) {
    sm.found = 0x7fffffff;
    sm.last_pos = -1;
  }
  __syncthreads();
  if (lane == 31)
#pragma unroll
    for (int k = 0; k < kRounds; ++k) sm.red[k][warp] = inc[k];
  __syncthreads();
  float base = 0.f;
#pragma unroll
  for (int k = 0; k < kRounds; ++k) {
    float before = 0.f, total = 0.f;
    for (int i = 0; i < kK2Threads / 32; ++i) {
      if (i == warp) before = total;
      total += sm.red[k][i];
    }
    const float lo = base + (before + exc[k]);
    const float hi = base + (before + inc[k]);
    const int vi = k * kK2Threads + tid;
    if (lo <= target && target < hi) {
      float acc = lo;
      int pick = -1;
#pragma unroll
      for (int e = 0; e < EV; ++e) {
        acc += w[k][e];
        if (w[k][e] > 0.f) {
          pick = e;
          if (acc > target) break;
        }
      }
      if (pick >= 0) atomicMin(&sm.found, vi * EV + pick);
    }
#pragma unroll
    for (int e = EV - 1; e >= 0; --e)
      if (w[k][e] > 0.f) {
        atomicMax(&sm.last_pos, vi * EV + e);
        break;
      }
    base = base + total;
  }
  __syncthreads();
  const int r = sm.found != 0x7fffffff ? sm.found : sm.last_pos;
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

// Softmax masses of the chunks of one row from kernel 1's partials.
__device__ __forceinline__ void row_masses(const Params& p, int row, float m, DecideSmem& sm) {
  const float4* pr = reinterpret_cast<const float4*>(p.part + static_cast<size_t>(row) * p.CH);
  for (int k = threadIdx.x; k < p.CH; k += kK2Threads) {
    const float4 q = __ldcg(pr + k);
    sm.mass[k] = q.y * fast_exp2(q.x - m);
  }
  __syncthreads();
}

// Inverse-CDF draw from the softmax of `row` (row max m, log2 domain): pick
// the chunk from the partial masses, then search that chunk.
template <typename T>
__device__ int draw_softmax(const Params& p, const T* rowp, int row, float m, float u,
                            DecideSmem& sm) {
  row_masses(p, row, m, sm);
  if (threadIdx.x == 0) pick_chunk(sm.mass, p.CH, u, &sm.pick_ch, &sm.pick_off);
  __syncthreads();
  const int ch = sm.pick_ch;
  const float target = sm.pick_off;
  const int e0 = ch * p.chunk;
  const WeightFn wp{0, p.s2, m, 0.f, 1.f, 0.f, 1.f};
  const int e = chunk_search<T>(reinterpret_cast<const uint4*>(rowp + e0), nullptr,
                                min(p.chunk, p.V - e0), target, wp, sm);
  return e >= 0 ? e0 + e : 0;
}

// (max, sum, argmax) of one row from its chunk partials: one warp.
__device__ __forceinline__ void combine_row(const Params& p, int row, int i, DecideSmem& sm) {
  const int lane = threadIdx.x & 31;
  const float4* pr = reinterpret_cast<const float4*>(p.part + static_cast<size_t>(row) * p.CH);
  float m = kNegInf;
  for (int k = lane; k < p.CH; k += 32) m = fmaxf(m, __ldcg(pr + k).x);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f, av = kNegInf;
  int ai = 0x7fffffff;
  for (int k = lane; k < p.CH; k += 32) {
    const float4 q = __ldcg(pr + k);   // (m, s, amax, aidx); an L1 hit after the first loop
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
  if (lane == 0) {
    sm.rm[i] = m;
    sm.rs[i] = p.greedy ? 1.f : s;
    sm.ridx[i] = ai;
  }
}

// Kernel 2: one CTA per request.  Combines the request's chunk partials,
// runs the acceptance scan, writes every output except a residual token and
// the decision record for kernel 3, then draws the bonus / fresh token and
// any SAMPLE-mode proposals (nothing is drawn after a rejection here).
template <typename T>
__global__ void __launch_bounds__(kK2Threads) decide_kernel(const Params p) {
  __shared__ DecideSmem sm;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int c = blockIdx.x;
  const int N = p.N, M = N - 1, V = p.V;
  const T* logits = static_cast<const T*>(p.logits);
  const T* prev = static_cast<const T*>(p.prev_logits);
  griddep_launch_dependents();

  const int row0 = p.qo[c];
  const int rows = p.qo[c + 1] - row0;
  const bool full = p.mode[c] == IDLM_MODE_FULL;
  const int ncl = full ? N : 1;
  const int prow0 = full ? p.prev_row0[c] : 0;
  if (rows != ncl + M || row0 < 0 || row0 + rows > p.T ||
      (full && (prow0 < 0 || prow0 + M > p.prev_rows))) {
    if (tid == 0) {
      set_status(p.status, IDLM_DEV_BAD_LAYOUT);
      p.dec[c].residual = 0;
    }
    return;
  }
  // draft logits and q statistics: inputs of this call, not kernel 1's
  // results, so they are read before waiting for kernel 1
  float mq_i = 0.f, sq_i = 1.f;
  if (full && tid < M) {
    const int d = p.drafts[c * M + tid];
    sm.dtok[tid] = d;
    mq_i = p.dq_stats[2 * (c * M + tid)];
    sq_i = p.dq_stats[2 * (c * M + tid) + 1];
    if (d >= 0 && d < V) {
      sm.xp[tid] = load1(logits + static_cast<size_t>(row0 + tid) * V + d);
      sm.yq[tid] = load1(prev + static_cast<size_t>(prow0 + tid) * V + d);
    }
  }
  if (tid < 16) sm.acc_ok[tid] = 0;
  griddep_wait();

  // 1. row statistics of every row of the request
  for (int i = warp; i < rows; i += kK2Threads / 32) combine_row(p, row0 + i, i, sm);
  __syncthreads();

  // 2. verification of the drafts (FULL)
  if (full && tid < M) {
    const int i = tid;   // draft i+1, verified by clean row i
    const int d = sm.dtok[i];
    const float u = isd_uniform(p.seed, p.step, c, kPurposeAccept, i);
    float pv = 0.f, qv = 0.f, ratio = 0.f;
    int ok = 0;
    if (d < 0 || d >= V) {
      set_status(p.status, IDLM_DEV_BAD_TOKEN);
    } else {
      if (p.greedy) {
        pv = (d == sm.ridx[i]) ? 1.f : 0.f;
        qv = (sm.yq[i] == mq_i) ? 1.f : 0.f;
      } else {
        pv = fast_exp2(sm.xp[i] * p.s2 - sm.rm[i]) / sm.rs[i];
        qv = fast_exp2(sm.yq[i] * p.s2 - mq_i * kLog2e) / sq_i;
      }
      ratio = qv > 0.f ? pv / qv : kInf;
      ok = u < fminf(1.f, ratio);
    }
    sm.acc_ok[i] = ok;
    if (p.dbg) {
      float* db = p.dbg + 4 * (c * M + i);
      db[0] = u;
      db[1] = pv;
      db[2] = qv;
      db[3] = ratio;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int n = 0;
    if (full)
      while (n < M && sm.acc_ok[n]) ++n;
    sm.n_acc = n;
  }
  __syncthreads();
  const int n_acc = sm.n_acc;
  const bool rejected = full && n_acc < M;

  // 3. the decision record and every output that needs no draw
  if (tid == 0) {
    Decision dr;
    dr.residual = rejected && !p.greedy;
    dr.row_p = row0 + n_acc;
    dr.row_q = prow0 + n_acc;
    dr.n_acc = n_acc;
    dr.mp = sm.rm[n_acc];
    dr.isp = 1.f / sm.rs[n_acc];
    dr.mq = 0.f;
    dr.isq = 1.f;
    if (dr.residual) {
      dr.mq = p.dq_stats[2 * (c * M + n_acc)] * kLog2e;
      dr.isq = 1.f / p.dq_stats[2 * (c * M + n_acc) + 1];
    }
    p.dec[c] = dr;
    p.res_cnt[c] = 0;
    p.n_accepted[c] = n_acc;
    p.n_out[c] = n_acc + 1;
    p.n_commit[c] = full ? 1 + n_acc : 1;
    p.next_mode[c] = rejected ? IDLM_MODE_FRESH : IDLM_MODE_FULL;
    p.next_mask_row0[c] = row0 + ncl;
  }
  const float to_nat = p.greedy ? 1.f : (1.f / kLog2e);
  if (p.row_stats && tid < rows) {
    p.row_stats[2 * (row0 + tid)] = sm.rm[tid] * to_nat;
    p.row_stats[2 * (row0 + tid) + 1] = sm.rs[tid];
  }
  if (tid < M) {
    p.next_q_stats[2 * (c * M + tid)] = sm.rm[ncl + tid] * to_nat;
    p.next_q_stats[2 * (c * M + tid) + 1] = sm.rs[ncl + tid];
  }
  if (tid < N) {
    if (tid < n_acc) p.out_tokens[c * N + tid] = sm.dtok[tid];
    else if (tid > n_acc) p.out_tokens[c * N + tid] = -1;
    else if (p.greedy) p.out_tokens[c * N + tid] = sm.ridx[rejected ? n_acc : ncl - 1];
  }
  if (tid < M) {
    if (rejected) p.next_drafts[c * M + tid] = -1;
    else if (p.greedy || p.propose == IDLM_PROPOSE_ARGMAX)
      p.next_drafts[c * M + tid] = sm.ridx[ncl + tid];
  }

  // 4. draws from p: bonus / fresh token (t = 0), SAMPLE proposals (t >= 1)
  if (!rejected && !p.greedy) {
    const int ntask = p.propose == IDLM_PROPOSE_SAMPLE ? N : 1;
    for (int t = 0; t < ntask; ++t) {
      const int li = t == 0 ? ncl - 1 : ncl + t - 1;
      const float u = t == 0 ? isd_uniform(p.seed, p.step, c, kPurposeSample, 0)
                             : isd_uniform(p.seed, p.step, c, kPurposePropose, t - 1);
      const int tok = draw_softmax<T>(p, logits + static_cast<size_t>(row0 + li) * V, row0 + li,
                                      sm.rm[li], u, sm);
      if (tid == 0) {
        if (t == 0) p.out_tokens[c * N + n_acc] = tok;
        else p.next_drafts[c * M + t - 1] = tok;
      }
    }
  }
}

// Kernel 3: one CTA per (request, chunk).  For a request rejected at draft
// j, CTA k sums the residual max(0, p_j - q_j) over chunk k; the last CTA of
// the request to finish picks the chunk from those sums and searches it (or
// draws from p_j when the residual is zero everywhere).  Every other CTA
// leaves after reading the decision record.
template <typename T>
__global__ void __launch_bounds__(kK2Threads) residual_kernel(const Params p) {
  __shared__ DecideSmem sm;
  __shared__ Decision dr;
  const int tid = threadIdx.x;
  const int c = blockIdx.x / p.CH;
  const int k = blockIdx.x % p.CH;
  const int V = p.V;
  griddep_wait();
  if (tid == 0) dr = p.dec[c];
  __syncthreads();
  if (!dr.residual) return;
  const T* rp = static_cast<const T*>(p.logits) + static_cast<size_t>(dr.row_p) * V;
  const T* rq = static_cast<const T*>(p.prev_logits) + static_cast<size_t>(dr.row_q) * V;
  const WeightFn wres{1, p.s2, 0.f, dr.mp, dr.isp, dr.mq, dr.isq};
  constexpr int EV = Vec<T>::kN;
  const int e0 = k * p.chunk;
  const int nvec = min(p.chunk, V - e0) / EV;
  const uint4* xs = reinterpret_cast<const uint4*>(rp + e0);
  const uint4* ys = reinterpret_cast<const uint4*>(rq + e0);
  float acc = 0.f;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int vi = r * kK2Threads + tid;
    if (vi < nvec) {
      float w[EV];
      vec_weights<T>(xs, ys, vi, wres, w);
#pragma unroll
      for (int e = 0; e < EV; ++e) acc += w[e];
    }
  }
  acc = block_sum(acc, sm.red[0]);
  if (tid == 0) {
    p.res_part[static_cast<size_t>(c) * p.CH + k] = acc;
    __threadfence();
    sm.is_last = atomicAdd(&p.res_cnt[c], 1) == p.CH - 1;
  }
  __syncthreads();
  if (!sm.is_last) return;
  __threadfence();
  const float u = isd_uniform(p.seed, p.step, c, kPurposeSample, 1);
  for (int j = tid; j < p.CH; j += kK2Threads)
    sm.mass[j] = __ldcg(p.res_part + static_cast<size_t>(c) * p.CH + j);
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f;
    for (int j = 0; j < p.CH; ++j) tot += sm.mass[j];
    sm.n_acc = tot > 0.f;
    if (tot > 0.f) pick_chunk(sm.mass, p.CH, u, &sm.pick_ch, &sm.pick_off);
  }
  __syncthreads();
  int tok;
  if (sm.n_acc) {
    const int ch = sm.pick_ch;
    const float target = sm.pick_off;
    const int f0 = ch * p.chunk;
    const int e = chunk_search<T>(reinterpret_cast<const uint4*>(rp + f0),
                                  reinterpret_cast<const uint4*>(rq + f0), min(p.chunk, V - f0),
                                  target, wres, sm);
    tok = e >= 0 ? f0 + e : 0;
  } else {
    tok = draw_softmax<T>(p, rp, dr.row_p, dr.mp, u, sm);   // p_j == q_j: draw from p_j
  }
  if (tid == 0) p.out_tokens[c * p.N + dr.n_acc] = tok;
}

inline int chunk_elems(int dtype) { return dtype == IDLM_BF16 ? kItemBytes / 2 : kItemBytes / 4; }
inline int chunks_for(int V, int dtype) { return (V + chunk_elems(dtype) - 1) / chunk_elems(dtype); }

size_t workspace_bytes(int C, int T, int V, int dtype, Params* p, void* base) {
  const int CH = chunks_for(V, dtype);
  Carver cv(base);
  Partial* part = cv.take<Partial>(static_cast<size_t>(T) * CH);
  float* res_part = cv.take<float>(static_cast<size_t>(C) * CH);
  int32_t* res_cnt = cv.take<int32_t>(C);
  Decision* dec = cv.take<Decision>(C);
  if (p) {
    p->part = part;
    p->res_part = res_part;
    p->res_cnt = res_cnt;
    p->dec = dec;
  }
  return cv.used;
}

template <typename T>
idlm_status launch(const Params& p, int dev, int sm_count, cudaStream_t stream) {
  // shared-memory opt-in, once per device
  static std::mutex mu;
  static bool done[64] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return IDLM_ERR_CUDA;
    if (!done[dev]) {
      if (cudaFuncSetAttribute(vocab_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kK1Smem)) != cudaSuccess)
        return IDLM_ERR_CUDA;
      done[dev] = true;
    }
  }
  const long long W = static_cast<long long>(p.T) * p.CH;
  const int grid1 = static_cast<int>(std::min<long long>(sm_count, W));
  vocab_stream_kernel<T><<<grid1, kK1Threads, kK1Smem, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return IDLM_ERR_CUDA;

  // kernels 2 and 3 start early as programmatic dependents and wait in
  // griddepcontrol.wait for the results of the kernel before them
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kK2Threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.C);
  e = cudaLaunchKernelEx(&cfg, decide_kernel<T>, p);
  if (e != cudaSuccess) {
    // a stream that does not take programmatic serialisation: plain order
    (void)cudaGetLastError();
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, decide_kernel<T>, p);
  }
  if (e != cudaSuccess) return IDLM_ERR_CUDA;
  cfg.gridDim = dim3(p.C * p.CH);
  e = cudaLaunchKernelEx(&cfg, residual_kernel<T>, p);
  return cuda_status(e);
}

}  // namespace acc
}  // namespace idlm

using namespace idlm;

extern "C" size_t idlm_isd_accept_workspace_size(int C, int T, int N, int V) {
  if (C <= 0 || T <= 0 || N < 2 || V <= 0) return 0;
  // an fp32 chunk holds fewer values than a bf16 one: size for fp32
  return acc::workspace_bytes(C, T, V, IDLM_F32, nullptr, nullptr);
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
  const int CH = acc::chunks_for(V, dtype);
  if (CH > acc::kMaxChunks) return IDLM_ERR_UNSUPPORTED;
  // bulk copies and vector loads start on 16-byte boundaries
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(prev_logits)) & 15)
    return IDLM_ERR_INVALID_ARG;
  acc::Params p;
  if (!workspace || workspace_bytes < acc::workspace_bytes(C, T, V, dtype, nullptr, nullptr))
    return IDLM_ERR_WORKSPACE;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return IDLM_ERR_CUDA;
  acc::workspace_bytes(C, T, V, dtype, &p, workspace);
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
  p.chunk = acc::chunk_elems(dtype);
  p.greedy = temperature == 0.f;
  p.propose = proposal_mode;
  p.prev_rows = prev_rows;
  p.s2 = p.greedy ? 1.f : kLog2e / temperature;
  if (dtype == IDLM_BF16) return acc::launch<__nv_bfloat16>(p, dev.device, dev.sm_count, stream);
  return acc::launch<float>(p, dev.device, dev.sm_count, stream);
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
  if (acc::workspace_bytes(C, T, V, IDLM_F32, nullptr, nullptr) > acc::kStaticScratchBytes)
    return IDLM_ERR_WORKSPACE;
  void* scratch = acc::static_scratch();
  if (!scratch) return IDLM_ERR_CUDA;
  return idlm_isd_accept(logits, dtype, V, qo_indptr, mode, drafts, draft_q_stats, prev_logits,
                         prev_rows, prev_mask_row0, C, T, N, temperature, proposal_mode, seed,
                         step, n_accepted, out_tokens, n_out, n_commit, next_drafts,
                         next_q_stats, next_mode, next_mask_row0, row_stats, dbg, scratch,
                         acc::kStaticScratchBytes, status, stream);
}
