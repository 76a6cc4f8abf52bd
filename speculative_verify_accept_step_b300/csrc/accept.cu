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
// evenly; a producer thread streams each CTA's chunks into a 22-stage
// shared-memory ring with 1-D bulk copies (cp.async.bulk, mbarrier
// completion), and eleven consumer warps each take whole chunks (copied to registers, so
// the stage is free again at once): packed
// bf16x2 maxima per group of 64 values, one exp2 per value for the sum, and
// the first index of the chunk maximum.  Every chunk leaves one partial
// (max, sum, max value, argmax) in the workspace; nothing is decided here.
//
// A 13th warp of kernel 1 gathers each request's inputs that do not depend
// on the pass (draft tokens and their two logits, the proposing rows' (m, S),
// every Philox uniform) while the logits stream.
//
// The decide kernel (one CTA per request), a programmatic dependent of
// kernel 1, combines the request's chunk partials, runs the acceptance scan,
// writes every output that needs no draw and appends the open draws to a
// work list.  The work kernel (a persistent grid, a programmatic dependent
// of the decide kernel) takes the list: after a rejection at draft j, one
// item per two chunks sums the residual max(0, p_j - q_j), and the last item
// of the request to finish picks the chunk from those sums and searches it;
// otherwise an item draws the bonus / fresh token or a SAMPLE-mode proposal,
// picking the chunk from kernel 1's partial sums and searching only that
// chunk.  Draws are inverse-CDF in vocabulary order.
#include <algorithm>
#include <mutex>

#include "commit.cuh"
#include "common.cuh"
#include "host_util.h"
#include "philox.cuh"

namespace idlm {
namespace acc {

constexpr int kItemBytes = 8192;                 // one chunk of a row
constexpr int kCWarps = 11;                      // kernel-1 consumer warps
// Kernel-1 ring depth, a multiple of kCWarps: consumer warp w takes chunks
// j = w, w + kCWarps, ..., so stage j % kStages is only ever read by warp w
// and a warp waits on a stage's next phase only after it consumed the one
// before.  With another depth, warp w could wait on stage s for chunk j while
// chunk j - kStages (another warp's) has not landed yet, and the parity test
// would pass on the older phase.
constexpr int kStages = 2 * kCWarps;
static_assert(kStages % kCWarps == 0, "a stage must return to the warp that read it");
constexpr int kK1Threads = 32 * (kCWarps + 2);   // + producer warp + request warp
constexpr size_t kK1Smem = 1024 + size_t(kStages) * kItemBytes + 2 * kStages * 8;
constexpr int kDThreads = 256;                   // decide kernel
constexpr int kWThreads = 256;                   // work kernel
constexpr int kWorkPerSM = 4;                    // work-kernel CTAs per SM
constexpr int kSliceChunks = 2;                  // chunks per residual slice
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

// Per-request inputs gathered by kernel 1's request warp while the logits
// stream: draft tokens, their logits in this step's verifying row (xp) and
// in the previous step's proposing row (yq), the proposing rows' (m, S), and
// every uniform the request may use.
struct __align__(16) PreRecord {
  int dtok[16];
  float xp[16], yq[16], mq[16], sq[16];
  float u_acc[16];   // acceptance test of draft i+1
  float u_draw[16];  // t = 0: bonus / fresh token; t >= 1: SAMPLE proposal t
  float u_res;       // residual draw
  int pad[3];
};

// One unit of the work kernel, written by the decide kernel.
struct __align__(16) WorkItem {
  int c, kind, idx, n_acc;   // kind 0: residual slice idx; kind 1: softmax draw t = idx;
                             // kind 2: KV commit of idx rows
  int row_x, row_y;          // residual: rows of p_j (this step) and q_j (previous step);
                             // draw: the row drawn from (row_y unused)
  float mx, isx;             // log2-domain max and 1/sum of row x
  float my, isy;             // the same for row y (residual only)
  float u;                   // uniform of the draw
  int pad;
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
  int32_t* res_cnt;   // [C] residual slices finished (zeroed by kernel 1)
  PreRecord* pre;     // [C] kernel 1 -> decide kernel
  WorkItem* work;     // [C * max(nslice, N)] decide kernel -> work kernel
  int32_t* work_cnt;  // [1] items in `work` (zeroed by kernel 1)
  int32_t* status;
  uint64_t seed, step;
  int V, C, T, N, CH, nslice, chunk, greedy, propose, prev_rows;
  float s2;           // log2(e) / T
  int part_given;     // 1: `part` already holds every chunk record (the fused LM head
                      // wrote them); kernel 1 then only gathers the requests' inputs
  int do_commit;      // 1: each request's KV commit is a work item (fused accept + commit)
  CommitArgs cm;
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

// Atomic add at GPU scope with acquire-release ordering: the caller's earlier
// writes are visible to whoever sees the new count, and the caller sees the
// writes of everyone who counted before it.
__device__ __forceinline__ int atomic_add_acq_rel(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Packed fp32x2 arithmetic (two lanes of values per instruction).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Sum of 2^(x s2 - m) over the 8 values of a vector, into two packed
// accumulators (bf16: one packed FMA, two exp2 and one packed add per pair).
template <typename T>
__device__ __forceinline__ void exp_sum_vec(const uint4& v, uint64_t s2x2, uint64_t nmx2,
                                            uint64_t& acc0, uint64_t& acc1);
template <>
__device__ __forceinline__ void exp_sum_vec<__nv_bfloat16>(const uint4& v, uint64_t s2x2,
                                                           uint64_t nmx2, uint64_t& acc0,
                                                           uint64_t& acc1) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint64_t z = fma2(pack2(bf16_lo(w[q]), bf16_hi(w[q])), s2x2, nmx2);
    float z0, z1;
    unpack2(z, z0, z1);
    const uint64_t e = pack2(fast_exp2(z0), fast_exp2(z1));
    if (q & 1) acc1 = add2(acc1, e);
    else acc0 = add2(acc0, e);
  }
}
template <>
__device__ __forceinline__ void exp_sum_vec<float>(const uint4& v, uint64_t s2x2, uint64_t nmx2,
                                                   uint64_t& acc0, uint64_t& acc1) {
  const uint64_t z0 = fma2(pack2(__uint_as_float(v.x), __uint_as_float(v.y)), s2x2, nmx2);
  const uint64_t z1 = fma2(pack2(__uint_as_float(v.z), __uint_as_float(v.w)), s2x2, nmx2);
  float a, b, c, d;
  unpack2(z0, a, b);
  unpack2(z1, c, d);
  acc0 = add2(acc0, pack2(fast_exp2(a), fast_exp2(b)));
  acc1 = add2(acc1, pack2(fast_exp2(c), fast_exp2(d)));
}

// Running (max, sum) of one lane over 8 vectors: packed bf16x2 maxima first,
// one rescale when the lane maximum rises, then one exp2 per value.
template <typename T>
__device__ __forceinline__ void lane_group(const uint4* v, float s2, bool greedy, int g,
                                           float& m_run, uint64_t& acc0, uint64_t& acc1,
                                           float& bx, int& bg) {
  const float gm = group_max<T>(v);
  if (gm > bx) {
    bx = gm;
    bg = g;
  }
  if (greedy) return;
  const float mz = gm * s2;
  if (mz > m_run) {
    const float f = fast_exp2(m_run - mz);
    const uint64_t f2 = pack2(f, f), zero = pack2(0.f, 0.f);
    acc0 = fma2(acc0, f2, zero);
    acc1 = fma2(acc1, f2, zero);
    m_run = mz;
  }
  if (m_run > kNegInf) {
    const uint64_t s2x2 = pack2(s2, s2), nmx2 = pack2(-m_run, -m_run);
#pragma unroll
    for (int j = 0; j < 8; ++j) exp_sum_vec<T>(v[j], s2x2, nmx2, acc0, acc1);
  }
}

// One warp reduces one 8 KB chunk (element e0 of its row first) that it has
// copied from shared memory into registers: lane l holds vectors
// l, l+32, ..., l+480 (unused ones hold -inf).  The chunk's argmax is the
// first index of the chunk maximum among the lanes that hold it.
template <typename T>
__device__ __forceinline__ Partial reduce_chunk(const uint4 (&v)[16], int e0, float s2,
                                                bool greedy, int lane) {
  constexpr int EV = Vec<T>::kN;
  float m_run = kNegInf, bx = kNegInf;
  uint64_t acc0 = pack2(0.f, 0.f), acc1 = acc0;
  int bg = -1;
  lane_group<T>(v, s2, greedy, 0, m_run, acc0, acc1, bx, bg);
  lane_group<T>(v + 8, s2, greedy, 1, m_run, acc0, acc1, bx, bg);
  float a0, a1, a2, a3;
  unpack2(acc0, a0, a1);
  unpack2(acc1, a2, a3);
  const float s_run = (a0 + a1) + (a2 + a3);
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
    for (int j = 15; j >= 0; --j) {
      if ((j >> 3) == bg) {
        float x[EV];
        Vec<T>::get(v[j], x);
#pragma unroll
        for (int k = EV - 1; k >= 0; --k)
          if (x[k] == BX) idx = (j * 32 + lane) * EV + k;
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

// Layout of request c as its inputs state it; false if they disagree.
struct Layout {
  int row0, rows, ncl, prow0;
  bool full;
};
__device__ __forceinline__ bool request_layout(const Params& p, int c, Layout& L) {
  const int M = p.N - 1;
  L.row0 = p.qo[c];
  L.rows = p.qo[c + 1] - L.row0;
  L.full = p.mode[c] == IDLM_MODE_FULL;
  L.ncl = L.full ? p.N : 1;
  L.prow0 = L.full ? p.prev_row0[c] : 0;
  return L.rows == L.ncl + M && L.row0 >= 0 && L.row0 + L.rows <= p.T &&
         (!L.full || (L.prow0 >= 0 && L.prow0 + M <= p.prev_rows));
}

// Kernel 1's request warp: everything request c needs that does not depend
// on the vocab pass (one warp; lanes in parallel).
template <typename T>
__device__ void request_inputs(const Params& p, int c, int lane) {
  const int N = p.N, M = N - 1, V = p.V;
  PreRecord* pr = p.pre + c;
  Layout L;
  const bool ok = request_layout(p, c, L);
  if (lane == 0) p.res_cnt[c] = 0;
  if (lane == 0 && c == 0) *p.work_cnt = 0;
  if (!ok) {
    if (lane == 0) set_status(p.status, IDLM_DEV_BAD_LAYOUT);
    return;
  }
  if (lane < M) {
    int d = -1;
    float xp = 0.f, yq = 0.f, mq = 0.f, sq = 1.f;
    if (L.full) {
      d = p.drafts[c * M + lane];
      mq = p.dq_stats[2 * (c * M + lane)];
      sq = p.dq_stats[2 * (c * M + lane) + 1];
      if (d >= 0 && d < V) {
        xp = load1(static_cast<const T*>(p.logits) + static_cast<size_t>(L.row0 + lane) * V + d);
        yq = load1(static_cast<const T*>(p.prev_logits) + static_cast<size_t>(L.prow0 + lane) * V + d);
      } else {
        set_status(p.status, IDLM_DEV_BAD_TOKEN);
      }
    }
    pr->dtok[lane] = d;
    pr->xp[lane] = xp;
    pr->yq[lane] = yq;
    pr->mq[lane] = mq;
    pr->sq[lane] = sq;
    pr->u_acc[lane] = isd_uniform(p.seed, p.step, c, kPurposeAccept, lane);
  }
  if (lane >= 16 && lane < 16 + N) {
    const int t = lane - 16;
    pr->u_draw[t] = t == 0 ? isd_uniform(p.seed, p.step, c, kPurposeSample, 0)
                           : isd_uniform(p.seed, p.step, c, kPurposePropose, t - 1);
  }
  if (lane == 31) pr->u_res = isd_uniform(p.seed, p.step, c, kPurposeSample, 1);
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
  // launched as a programmatic dependent of the kernel before it: its
  // results (the logits, the previous step's state) are read only after it
  // has finished
  griddep_wait();
  griddep_launch_dependents();

  // rows in use: qo_indptr[C] (T is the capacity of the logits buffer, so a
  // fixed-shape loop can pass its largest row count every step)
  const int T_used = min(max(__ldg(p.qo + p.C), 0), p.T);
  const long long W = p.part_given ? 0 : static_cast<long long>(T_used) * p.CH;
  const long long lo = W * blockIdx.x / gridDim.x;
  const long long hi = W * (blockIdx.x + 1) / gridDim.x;
  const int n = static_cast<int>(hi - lo);
  const T* logits = static_cast<const T*>(p.logits);

  if (warp == kCWarps + 1) {
    // ------------------------------------------------------ request warp
    for (int c = blockIdx.x; c < p.C; c += gridDim.x) request_inputs<T>(p, c, lane);
    return;
  }
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
    const int nvec = min(p.chunk, p.V - e0) / Vec<T>::kN;
    // copy the chunk to registers and hand the stage back at once
    const uint32_t sb = smem_u32(base + size_t(s) * kItemBytes);
    uint4 v[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int idx = q * 32 + lane;
      v[q] = idx < nvec ? lds128(sb + idx * 16) : Vec<T>::neg_inf();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    const Partial pt = reduce_chunk<T>(v, e0, p.s2, p.greedy, lane);
    if (lane == 0) p.part[item] = pt;
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

constexpr int kMaxRounds = 4;       // vectors of a chunk per thread in a search
constexpr int kMaxWarps = 8;

struct DecideSmem {
  float rm[kMaxRows], rs[kMaxRows];
  int ridx[kMaxRows];
  int acc_ok[16];
  float red[kMaxRounds][kMaxWarps];
  int found, last_pos;
  int pick_ch;
  float pick_off;
  int flag;
  float mass[kMaxChunks];
};

template <int THREADS>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = 0.f;
#pragma unroll
  for (int i = 0; i < THREADS / 32; ++i) v += red[i];
  return v;
}

// Inverse CDF inside one chunk (global memory, `cnt` values from xs[0]):
// the first element in index order whose running weight sum exceeds
// `target`; if rounding leaves none, the last element with positive weight.
// Element order is (round r, thread t, value): round r covers vectors
// [THREADS r, THREADS (r + 1)).  Adjacent intervals share their boundary
// value bit for bit, so no target falls in a gap.  Every thread returns the
// answer (chunk-relative index, or -1 if every weight is zero).
template <typename T, int THREADS>
__device__ int chunk_search(const uint4* xs, const uint4* ys, int cnt, float target,
                            const WeightFn& wf, DecideSmem& sm) {
  constexpr int EV = Vec<T>::kN;
  constexpr int R = kItemBytes / 16 / THREADS;
  constexpr int NW = THREADS / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvec = cnt / EV;
  float w[R][EV];
  float inc[R], exc[R];
  {
    // every load of the chunk in flight before any weight is computed
    uint4 vx[R], vy[R];
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int vi = k * THREADS + tid;
      vx[k] = vi < nvec ? __ldg(xs + vi) : make_uint4(0u, 0u, 0u, 0u);
      vy[k] = (ys && vi < nvec) ? __ldg(ys + vi) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int vi = k * THREADS + tid;
      float x[EV], y[EV];
      Vec<T>::get(vx[k], x);
      Vec<T>::get(vy[k], y);
#pragma unroll
      for (int e = 0; e < EV; ++e) w[k][e] = vi < nvec ? wf(x[e], y[e]) : 0.f;
    }
  }
#pragma unroll
  for (int k = 0; k < R; ++k) {
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
    for (int k = 0; k < R; ++k) sm.red[k][warp] = inc[k];
  __syncthreads();
  float base = 0.f;
  int last = -1;
#pragma unroll
  for (int k = 0; k < R; ++k) {
    float before = 0.f, total = 0.f;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      if (i == warp) before = total;
      total += sm.red[k][i];
    }
    const float lo = base + (before + exc[k]);
    const float hi = base + (before + inc[k]);
    const int vi = k * THREADS + tid;
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
        last = max(last, vi * EV + e);
        break;
      }
    base = base + total;
  }
  // last element with positive weight: one shared atomic per warp
#pragma unroll
  for (int o = 16; o; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  if (lane == 0 && last >= 0) atomicMax(&sm.last_pos, last);
  __syncthreads();
  const int r = sm.found != 0x7fffffff ? sm.found : sm.last_pos;
  __syncthreads();
  return r;
}

// Chunk holding u * total of the masses, and the offset into it: the first
// chunk k with positive mass whose running sum (index order) exceeds the
// target; if rounding leaves none, the last chunk with positive mass.  One
// warp: lane l holds a contiguous run of chunks, so lane order is index
// order.  Writes sm.pick_ch / sm.pick_off (read them after a barrier).
__device__ __forceinline__ float pick_chunk_warp(const float* mass, int CH, float u,
                                                 DecideSmem& sm) {
  const int lane = threadIdx.x & 31;
  const int per = (CH + 31) / 32;
  const int k0 = min(CH, lane * per), k1 = min(CH, k0 + per);
  float mine = 0.f;
  int last = -1;
  for (int k = k0; k < k1; ++k) {
    mine += mass[k];
    if (mass[k] > 0.f) last = k;
  }
  float inc = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float nb = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += nb;
  }
  const float total = __shfl_sync(0xffffffffu, inc, 31);
  const float target = u * total;
  float acc = inc - mine;   // sum before this lane's run
  int pick = -1;
  float off = 0.f;
  if (acc <= target && target < inc) {
    for (int k = k0; k < k1; ++k) {
      if (mass[k] > 0.f && acc + mass[k] > target) {
        pick = k;
        off = target - acc;
        break;
      }
      acc += mass[k];
    }
    if (pick < 0 && last >= 0) {   // rounding inside the run: its last positive chunk
      pick = last;
      off = mass[last];
    }
  }
  // first lane with a pick; else the last positive chunk
  const unsigned hit = __ballot_sync(0xffffffffu, pick >= 0);
  if (hit) {
    const int src = __ffs(hit) - 1;
    pick = __shfl_sync(0xffffffffu, pick, src);
    off = __shfl_sync(0xffffffffu, off, src);
  } else {
    int lp = last;
#pragma unroll
    for (int o = 16; o; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
    pick = lp < 0 ? 0 : lp;
    off = lp < 0 ? 0.f : mass[lp];
  }
  if (lane == 0) {
    sm.pick_ch = pick;
    sm.pick_off = off;
  }
  return total;
}

// Inverse-CDF draw from the softmax of `row` (row max m, log2 domain), with
// the chunk masses already in `mass`: pick the chunk, then search it.
template <typename T, int THREADS>
__device__ int draw_softmax(const Params& p, const T* rowp, const float* mass, float m, float u,
                            DecideSmem& sm) {
  if (threadIdx.x < 32) pick_chunk_warp(mass, p.CH, u, sm);
  __syncthreads();
  const int ch = sm.pick_ch;
  const float target = sm.pick_off;
  const int e0 = ch * p.chunk;
  const WeightFn wp{0, p.s2, m, 0.f, 1.f, 0.f, 1.f};
  const int e = chunk_search<T, THREADS>(reinterpret_cast<const uint4*>(rowp + e0), nullptr,
                                         min(p.chunk, p.V - e0), target, wp, sm);
  return e >= 0 ? e0 + e : 0;
}

// Softmax masses of the chunks of one row from kernel 1's partials.
template <int THREADS>
__device__ __forceinline__ void row_masses(const Params& p, int row, float m, float* mass) {
  const float4* pr = reinterpret_cast<const float4*>(p.part + static_cast<size_t>(row) * p.CH);
  for (int k = threadIdx.x; k < p.CH; k += THREADS) {
    const float4 q = __ldcg(pr + k);
    mass[k] = q.y * fast_exp2(q.x - m);
  }
  __syncthreads();
}

// (max, sum, argmax) of one row from its chunk partials: one warp, one round
// of loads for up to 128 chunks.
__device__ __forceinline__ void combine_row(const Params& p, int row, int i, DecideSmem& sm) {
  const int lane = threadIdx.x & 31;
  const float4* pr = reinterpret_cast<const float4*>(p.part + static_cast<size_t>(row) * p.CH);
  float4 q[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int k = lane + 32 * r;
    q[r] = k < p.CH ? __ldcg(pr + k) : make_float4(kNegInf, 0.f, kNegInf, __int_as_float(0x7fffffff));
  }
  float m = fmaxf(fmaxf(q[0].x, q[1].x), fmaxf(q[2].x, q[3].x));
  for (int k = lane + 128; k < p.CH; k += 32) m = fmaxf(m, __ldcg(pr + k).x);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f, av = kNegInf;
  int ai = 0x7fffffff;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int k = lane + 32 * r;
    if (k < p.CH) {
      s += q[r].y * fast_exp2(q[r].x - m);
      argmax_merge(av, ai, q[r].z, __float_as_int(q[r].w));
    }
  }
  for (int k = lane + 128; k < p.CH; k += 32) {
    const float4 t = __ldcg(pr + k);
    s += t.y * fast_exp2(t.x - m);
    argmax_merge(av, ai, t.z, __float_as_int(t.w));
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

// Decide kernel: one CTA per request, launched as a programmatic dependent
// of kernel 1.  Combines the request's chunk partials (one warp per row, one
// round of loads), runs the acceptance scan, writes every output that needs
// no draw, and appends the draws it leaves open to the work list: after a
// rejection at draft j, one residual slice per two chunks of p_j / q_j;
// otherwise the bonus / fresh token and any SAMPLE-mode proposals.
template <typename T>
__global__ void __launch_bounds__(kDThreads) decide_kernel(const Params p) {
  __shared__ DecideSmem sm;
  __shared__ int base;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int c = blockIdx.x;
  const int N = p.N, M = N - 1, V = p.V;
  griddep_launch_dependents();
  Layout L;
  if (!request_layout(p, c, L)) return;   // kernel 1 has set the status
  const int ncl = L.ncl;
  if (tid < 16) sm.acc_ok[tid] = 0;
  griddep_wait();

  // kernel 1's request record and the row partials, in one round
  const PreRecord* pr = p.pre + c;
  int d = -1;
  float u = 0.f, mq = 0.f, sq = 1.f, xp = 0.f, yq = 0.f;
  if (L.full && tid < M) {
    d = pr->dtok[tid];
    u = pr->u_acc[tid];
    mq = pr->mq[tid];
    sq = pr->sq[tid];
    xp = pr->xp[tid];
    yq = pr->yq[tid];
  }
  for (int i = warp; i < L.rows; i += kDThreads / 32) combine_row(p, L.row0 + i, i, sm);
  __syncthreads();

  // verification of the drafts (FULL)
  if (L.full && tid < M) {
    const int i = tid;   // draft i+1, verified by clean row i
    float pv = 0.f, qv = 0.f, ratio = 0.f;
    int ok = 0;
    if (d >= 0 && d < V) {
      if (p.greedy) {
        pv = (d == sm.ridx[i]) ? 1.f : 0.f;
        qv = (yq == mq) ? 1.f : 0.f;
      } else {
        pv = fast_exp2(xp * p.s2 - sm.rm[i]) / sm.rs[i];
        qv = fast_exp2(yq * p.s2 - mq * kLog2e) / sq;
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
  int n_acc = 0;
  if (L.full)
    while (n_acc < M && sm.acc_ok[n_acc]) ++n_acc;
  const bool rejected = L.full && n_acc < M;
  const bool residual = rejected && !p.greedy;
  const int ndraw = (rejected || p.greedy) ? 0 : (p.propose == IDLM_PROPOSE_SAMPLE ? N : 1);
  const int nitems = residual ? p.nslice : ndraw;
  const int nall = nitems + (p.do_commit ? 1 : 0);

  // work items for the draws left open (and the request's KV commit)
  if (tid == 0 && nall) base = atomicAdd(p.work_cnt, nall);
  __syncthreads();
  if (p.do_commit && tid == 0) {
    WorkItem it;
    it.c = c;
    it.kind = 2;
    it.idx = L.full ? 1 + n_acc : 1;
    it.n_acc = n_acc;
    it.row_x = it.row_y = 0;
    it.mx = it.isx = it.my = it.isy = it.u = 0.f;
    it.pad = 0;
    p.work[base + nitems] = it;
  }
  if (tid < nitems) {
    WorkItem it;
    it.c = c;
    it.idx = tid;
    it.n_acc = n_acc;
    it.pad = 0;
    if (residual) {
      it.kind = 0;
      it.row_x = L.row0 + n_acc;
      it.row_y = L.prow0 + n_acc;
      it.mx = sm.rm[n_acc];
      it.isx = 1.f / sm.rs[n_acc];
      it.my = pr->mq[n_acc] * kLog2e;
      it.isy = 1.f / pr->sq[n_acc];
      it.u = pr->u_res;
    } else {
      const int li = tid == 0 ? ncl - 1 : ncl + tid - 1;
      it.kind = 1;
      it.row_x = L.row0 + li;
      it.row_y = 0;
      it.mx = sm.rm[li];
      it.isx = 1.f / sm.rs[li];
      it.my = 0.f;
      it.isy = 1.f;
      it.u = pr->u_draw[tid];
    }
    p.work[base + tid] = it;
  }

  // every output that needs no draw
  if (tid == 0) {
    p.n_accepted[c] = n_acc;
    p.n_out[c] = n_acc + 1;
    p.n_commit[c] = L.full ? 1 + n_acc : 1;
    p.next_mode[c] = rejected ? IDLM_MODE_FRESH : IDLM_MODE_FULL;
    p.next_mask_row0[c] = L.row0 + ncl;
  }
  const float to_nat = p.greedy ? 1.f : (1.f / kLog2e);
  if (p.row_stats && tid < L.rows) {
    p.row_stats[2 * (L.row0 + tid)] = sm.rm[tid] * to_nat;
    p.row_stats[2 * (L.row0 + tid) + 1] = sm.rs[tid];
  }
  if (tid < M) {
    p.next_q_stats[2 * (c * M + tid)] = sm.rm[ncl + tid] * to_nat;
    p.next_q_stats[2 * (c * M + tid) + 1] = sm.rs[ncl + tid];
  }
  if (tid < N) {
    if (tid < n_acc) p.out_tokens[c * N + tid] = pr->dtok[tid];
    else if (tid > n_acc) p.out_tokens[c * N + tid] = -1;
    else if (p.greedy) p.out_tokens[c * N + tid] = sm.ridx[rejected ? n_acc : ncl - 1];
  }
  if (tid < M) {
    if (rejected) p.next_drafts[c * M + tid] = -1;
    else if (p.greedy || p.propose == IDLM_PROPOSE_ARGMAX)
      p.next_drafts[c * M + tid] = sm.ridx[ncl + tid];
  }
}

// Work kernel: a persistent grid (kWorkPerSM CTAs per SM), launched as a
// programmatic dependent of the decide kernel, takes the work list in order.
// A residual slice sums max(0, p_j - q_j) over its two chunks; the last
// slice of a request to finish picks the chunk from the sums and searches it
// (or draws from p_j when the residual is zero everywhere).  A softmax draw
// picks the chunk from kernel 1's partial sums and searches only that chunk.
template <typename T>
__global__ void __launch_bounds__(kWThreads) work_kernel(const Params p) {
  __shared__ DecideSmem sm;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int N = p.N, M = N - 1, V = p.V;
  const T* logits = static_cast<const T*>(p.logits);
  constexpr int EV = Vec<T>::kN;
  constexpr int R = kItemBytes / 16 / kWThreads;
  griddep_wait();
  const int count = __ldcg(p.work_cnt);
  for (int i = blockIdx.x; i < count; i += gridDim.x) {
    const WorkItem it = p.work[i];
    const int c = it.c;
    if (it.kind == 2) {
      commit_request(p.cm, c, it.idx);
      __syncthreads();
      continue;
    }
    const T* rx = logits + static_cast<size_t>(it.row_x) * V;
    if (it.kind == 1) {
      row_masses<kWThreads>(p, it.row_x, it.mx, sm.mass);
      const int tok = draw_softmax<T, kWThreads>(p, rx, sm.mass, it.mx, it.u, sm);
      if (tid == 0) {
        if (it.idx == 0) p.out_tokens[c * N + it.n_acc] = tok;
        else p.next_drafts[c * M + it.idx - 1] = tok;
      }
      __syncthreads();
      continue;
    }
    // residual slice idx over chunks [2 idx, 2 idx + 2)
    const T* ry = static_cast<const T*>(p.prev_logits) + static_cast<size_t>(it.row_y) * V;
    const WeightFn wres{1, p.s2, 0.f, it.mx, it.isx, it.my, it.isy};
    const int ch0 = it.idx * kSliceChunks;
    float part[kSliceChunks];
    {
      uint4 vx[kSliceChunks][R], vy[kSliceChunks][R];
#pragma unroll
      for (int h = 0; h < kSliceChunks; ++h) {
        const int ch = ch0 + h;
        const int e0 = ch * p.chunk;
        const int nvec = ch < p.CH ? min(p.chunk, V - e0) / EV : 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int vi = r * kWThreads + tid;
          vx[h][r] = vi < nvec ? __ldg(reinterpret_cast<const uint4*>(rx + e0) + vi) : make_uint4(0u, 0u, 0u, 0u);
          vy[h][r] = vi < nvec ? __ldg(reinterpret_cast<const uint4*>(ry + e0) + vi) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int h = 0; h < kSliceChunks; ++h) {
        const int ch = ch0 + h;
        const int nvec = ch < p.CH ? min(p.chunk, V - ch * p.chunk) / EV : 0;
        float a = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (r * kWThreads + tid < nvec) {
            float x[EV], y[EV];
            Vec<T>::get(vx[h][r], x);
            Vec<T>::get(vy[h][r], y);
#pragma unroll
            for (int e = 0; e < EV; ++e) a += wres(x[e], y[e]);
          }
        }
        part[h] = a;
      }
    }
#pragma unroll
    for (int h = 0; h < kSliceChunks; ++h) {
#pragma unroll
      for (int o = 16; o; o >>= 1) part[h] += __shfl_xor_sync(0xffffffffu, part[h], o);
    }
    if ((tid & 31) == 0)
#pragma unroll
      for (int h = 0; h < kSliceChunks; ++h) sm.red[h][warp] = part[h];
    __syncthreads();
    if (tid < kSliceChunks && ch0 + tid < p.CH) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kWThreads / 32; ++w) a += sm.red[tid][w];
      p.res_part[static_cast<size_t>(c) * p.CH + ch0 + tid] = a;
      __threadfence();
    }
    __syncthreads();
    if (tid == 0) sm.flag = atomic_add_acq_rel(&p.res_cnt[c], 1) == p.nslice - 1;
    __syncthreads();
    if (!sm.flag) continue;
    // the last slice of the request: every chunk's mass is visible now
    for (int j = tid; j < p.CH; j += kWThreads)
      sm.mass[j] = __ldcg(p.res_part + static_cast<size_t>(c) * p.CH + j);
    __syncthreads();
    if (tid < 32) {
      const float tot = pick_chunk_warp(sm.mass, p.CH, it.u, sm);
      if (tid == 0) sm.flag = tot > 0.f;
    }
    __syncthreads();
    int tok;
    if (sm.flag) {
      const int ch = sm.pick_ch;
      const float target = sm.pick_off;
      const int f0 = ch * p.chunk;
      const int e = chunk_search<T, kWThreads>(reinterpret_cast<const uint4*>(rx + f0),
                                               reinterpret_cast<const uint4*>(ry + f0),
                                               min(p.chunk, V - f0), target, wres, sm);
      tok = e >= 0 ? f0 + e : 0;
    } else {
      // p_j == q_j everywhere: draw from p_j
      row_masses<kWThreads>(p, it.row_x, it.mx, sm.mass);
      tok = draw_softmax<T, kWThreads>(p, rx, sm.mass, it.mx, it.u, sm);
    }
    if (tid == 0) p.out_tokens[c * N + it.n_acc] = tok;
    __syncthreads();
  }
}

// Chunk records from the fused LM head's tile records: the tiles of 128
// vocabulary entries that make up each 4096-entry chunk (bf16), merged in one
// warp per (row, chunk): max of the maxima, the sums rescaled to it, the
// largest value with the lowest index.
constexpr int kLmTile = 128;
__global__ void __launch_bounds__(256) lm_combine_kernel(const Partial* ts, int tiles, Partial* part,
                                                        int rows, int CH, int greedy) {
  const int w = static_cast<int>((blockIdx.x * 256u + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (w >= rows * CH) return;   // whole warps
  const int row = w / CH, ch = w % CH;
  constexpr int per = kItemBytes / 2 / kLmTile;   // tiles per chunk
  static_assert(per == 32, "one lane per tile of a chunk");
  const int tile = ch * per + lane;
  Partial t;
  t.m = kNegInf;
  t.s = 0.f;
  t.amax = kNegInf;
  t.aidx = 0x7fffffff;
  if (tile < tiles) t = ts[static_cast<size_t>(row) * tiles + tile];
  float M = t.m;
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float S = (greedy || t.m == kNegInf) ? 0.f : t.s * fast_exp2(t.m - M);
#pragma unroll
  for (int o = 16; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  float BX = t.amax;
  int BI = t.aidx;
#pragma unroll
  for (int o = 16; o; o >>= 1)
    argmax_merge(BX, BI, __shfl_xor_sync(0xffffffffu, BX, o), __shfl_xor_sync(0xffffffffu, BI, o));
  if (lane == 0) {
    Partial r;
    r.m = greedy ? BX : M;
    r.s = greedy ? 1.f : S;
    r.amax = BX;
    r.aidx = BI;
    part[static_cast<size_t>(row) * CH + ch] = r;
  }
}

inline int chunk_elems(int dtype) { return dtype == IDLM_BF16 ? kItemBytes / 2 : kItemBytes / 4; }
inline int chunks_for(int V, int dtype) { return (V + chunk_elems(dtype) - 1) / chunk_elems(dtype); }

size_t workspace_bytes(int C, int T, int V, int dtype, Params* p, void* base) {
  const int CH = chunks_for(V, dtype);
  Carver cv(base);
  Partial* part = cv.take<Partial>(static_cast<size_t>(T) * CH);
  float* res_part = cv.take<float>(static_cast<size_t>(C) * CH);
  int32_t* res_cnt = cv.take<int32_t>(C);
  PreRecord* pre = cv.take<PreRecord>(C);
  const int nslice = (CH + kSliceChunks - 1) / kSliceChunks;
  WorkItem* work = cv.take<WorkItem>(static_cast<size_t>(C) * (std::max(nslice, 16) + 1));
  int32_t* work_cnt = cv.take<int32_t>(1);
  if (p) {
    p->part = part;
    p->res_part = res_part;
    p->res_cnt = res_cnt;
    p->pre = pre;
    p->work = work;
    p->work_cnt = work_cnt;
  }
  return cv.used;
}

template <typename T>
idlm_status launch(const Params& p, int dev, int sm_count, cudaStream_t stream) {
  // shared-memory opt-in, once per device and context (a reset context
  // forgets function attributes)
  static std::mutex mu;
  static unsigned long long done[64] = {};
  const unsigned long long ctx = current_context_id();
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return IDLM_ERR_CUDA;
    if (done[dev] != ctx || ctx == 0) {
      // all three kernels ask for the largest shared-memory carveout, so that
      // CTAs of kernels 2 and 3 may share an SM with a kernel-1 CTA
      if (cudaFuncSetAttribute(vocab_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kK1Smem)) != cudaSuccess ||
          cudaFuncSetAttribute(vocab_stream_kernel<T>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
          cudaFuncSetAttribute(decide_kernel<T>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
          cudaFuncSetAttribute(work_kernel<T>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return IDLM_ERR_CUDA;
      done[dev] = ctx;
    }
  }
  const long long W = static_cast<long long>(p.T) * p.CH;
  const int grid1 = static_cast<int>(std::min<long long>(sm_count, W));
  // all three kernels start early as programmatic dependents and wait in
  // griddepcontrol.wait for the results of the kernel before them
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(grid1);
  cfg.blockDim = dim3(kK1Threads);
  cfg.dynamicSmemBytes = kK1Smem;
  cudaError_t e = cudaLaunchKernelEx(&cfg, vocab_stream_kernel<T>, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, vocab_stream_kernel<T>, p);
    cfg.numAttrs = 1;
  }
  if (e != cudaSuccess) return IDLM_ERR_CUDA;
  cfg.dynamicSmemBytes = 0;
  cfg.gridDim = dim3(p.C);
  cfg.blockDim = dim3(kDThreads);
  e = cudaLaunchKernelEx(&cfg, decide_kernel<T>, p);
  if (e != cudaSuccess) {
    // a stream that does not take programmatic serialisation: plain order
    (void)cudaGetLastError();
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, decide_kernel<T>, p);
  }
  if (e != cudaSuccess) return IDLM_ERR_CUDA;
  cfg.gridDim = dim3(sm_count * kWorkPerSM);
  cfg.blockDim = dim3(kWThreads);
  e = cudaLaunchKernelEx(&cfg, work_kernel<T>, p);
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

namespace {

// Checks the accept call's arguments, carves its workspace and fills the
// kernels' parameters (part_given = 0).
idlm_status accept_prepare(acc::Params& p, DeviceInfo& dev, const void* logits, int dtype, int V,
                           const int32_t* qo_indptr, const uint8_t* mode, const int32_t* drafts,
                           const float* draft_q_stats, const void* prev_logits, int prev_rows,
                           const int32_t* prev_mask_row0, int C, int T, int N, float temperature,
                           int proposal_mode, uint64_t seed, uint64_t step, int32_t* n_accepted,
                           int32_t* out_tokens, int32_t* n_out, int32_t* n_commit,
                           int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
                           int32_t* next_mask_row0, float* row_stats, float* dbg, void* workspace,
                           size_t workspace_bytes, int32_t* status) {
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
  if (!workspace || workspace_bytes < acc::workspace_bytes(C, T, V, dtype, nullptr, nullptr))
    return IDLM_ERR_WORKSPACE;
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
  p.nslice = (CH + acc::kSliceChunks - 1) / acc::kSliceChunks;
  p.chunk = acc::chunk_elems(dtype);
  p.greedy = temperature == 0.f;
  p.propose = proposal_mode;
  p.prev_rows = prev_rows;
  p.s2 = p.greedy ? 1.f : kLog2e / temperature;
  p.part_given = 0;
  p.do_commit = 0;
  return IDLM_OK;
}

idlm_status accept_launch(const acc::Params& p, const DeviceInfo& dev, int dtype,
                          cudaStream_t stream) {
  if (dtype == IDLM_BF16) return acc::launch<__nv_bfloat16>(p, dev.device, dev.sm_count, stream);
  return acc::launch<float>(p, dev.device, dev.sm_count, stream);
}

}  // namespace

extern "C" idlm_status idlm_isd_accept(
    const void* logits, int dtype, int V, const int32_t* qo_indptr, const uint8_t* mode,
    const int32_t* drafts, const float* draft_q_stats, const void* prev_logits, int prev_rows,
    const int32_t* prev_mask_row0, int C, int T, int N, float temperature, int proposal_mode,
    uint64_t seed, uint64_t step, int32_t* n_accepted, int32_t* out_tokens, int32_t* n_out,
    int32_t* n_commit, int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
    int32_t* next_mask_row0, float* row_stats, float* dbg, void* workspace,
    size_t workspace_bytes, int32_t* status, void* stream) {
  acc::Params p;
  DeviceInfo dev;
  const idlm_status rc = accept_prepare(
      p, dev, logits, dtype, V, qo_indptr, mode, drafts, draft_q_stats, prev_logits, prev_rows,
      prev_mask_row0, C, T, N, temperature, proposal_mode, seed, step, n_accepted, out_tokens,
      n_out, n_commit, next_drafts, next_q_stats, next_mode, next_mask_row0, row_stats, dbg,
      workspace, workspace_bytes, status);
  if (rc != IDLM_OK) return rc;
  return accept_launch(p, dev, dtype, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------- fused accept + commit
//
// The accept step and the KV commit of its kept rows in one call: the
// decision kernel appends one commit item per request to the residual
// kernel's work list, so the copies run beside the residual and draw items
// (on CTAs that have no other item) instead of as a kernel after them.

extern "C" idlm_status idlm_isd_accept_commit(
    const void* logits, int dtype, int V, const int32_t* qo_indptr, const uint8_t* mode,
    const int32_t* drafts, const float* draft_q_stats, const void* prev_logits, int prev_rows,
    const int32_t* prev_mask_row0, int C, int T, int N, float temperature, int proposal_mode,
    uint64_t seed, uint64_t step, int32_t* n_accepted, int32_t* out_tokens, int32_t* n_out,
    int32_t* n_commit, int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
    int32_t* next_mask_row0, float* row_stats, float* dbg, void* k_cache, void* v_cache,
    const int32_t* page_table, int max_pages, const int32_t* seq_lens_in,
    int32_t* seq_lens_out, const void* k_new, const void* v_new, int Hkv, int D,
    int page_size, int num_pages, int kv_dtype, int32_t* releasable_from, void* workspace,
    size_t workspace_bytes, int32_t* status, void* stream) {
  int row_bytes = 0;
  idlm_status rc = commit_check(k_cache, v_cache, page_table, max_pages, seq_lens_in,
                                seq_lens_out, k_new, v_new, Hkv, D, page_size, num_pages,
                                kv_dtype, &row_bytes);
  if (rc != IDLM_OK) return rc;
  acc::Params p;
  DeviceInfo dev;
  rc = accept_prepare(p, dev, logits, dtype, V, qo_indptr, mode, drafts, draft_q_stats,
                      prev_logits, prev_rows, prev_mask_row0, C, T, N, temperature,
                      proposal_mode, seed, step, n_accepted, out_tokens, n_out, n_commit,
                      next_drafts, next_q_stats, next_mode, next_mask_row0, row_stats, dbg,
                      workspace, workspace_bytes, status);
  if (rc != IDLM_OK) return rc;
  p.do_commit = 1;
  p.cm.k_cache = static_cast<uint8_t*>(k_cache);
  p.cm.v_cache = static_cast<uint8_t*>(v_cache);
  p.cm.page_table = page_table;
  p.cm.max_pages = max_pages;
  p.cm.seq_lens_in = seq_lens_in;
  p.cm.seq_lens_out = seq_lens_out;
  p.cm.k_new = static_cast<const uint8_t*>(k_new);
  p.cm.v_new = static_cast<const uint8_t*>(v_new);
  p.cm.qo_indptr = qo_indptr;
  p.cm.T = T;
  p.cm.Hkv = Hkv;
  p.cm.row_bytes = row_bytes;
  p.cm.page_size = page_size;
  p.cm.num_pages = num_pages;
  p.cm.releasable_from = releasable_from;
  p.cm.status = status;
  return accept_launch(p, dev, dtype, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------- fused LM head + accept
//
// The forward pass's last product and the accept step in one call: the LM
// head's GEMM writes the logits once and, in the same epilogue, the softmax
// statistics of every logits row per 128-entry tile of the vocabulary; a
// small kernel merges them into the accept's per-chunk records, and the
// accept runs on them without its own pass over the logits (kernel 1 only
// gathers the requests' inputs).  The logits are still written: the draws
// (inverse-CDF searches of one chunk, the residual of a rejected draft) read
// the rows and chunks they need from them.

extern "C" size_t idlm_lm_head_accept_workspace_size(int C, int T, int N, int H, int V) {
  if (C <= 0 || T <= 0 || N < 2 || H <= 0 || V <= 0) return 0;
  Carver cv(nullptr);
  cv.take<uint8_t>(acc::workspace_bytes(C, T, V, IDLM_BF16, nullptr, nullptr));
  cv.take<acc::Partial>(static_cast<size_t>(T) * ((V + acc::kLmTile - 1) / acc::kLmTile));
  cv.take<uint8_t>(lm_head_gemm_workspace(T, H, V));
  return cv.used;
}

extern "C" idlm_status idlm_lm_head_accept(
    const void* hidden, const void* w_vocab, int H, void* logits, int V,
    const int32_t* qo_indptr, const uint8_t* mode, const int32_t* drafts,
    const float* draft_q_stats, const void* prev_logits, int prev_rows,
    const int32_t* prev_mask_row0, int C, int T, int N, float temperature, int proposal_mode,
    uint64_t seed, uint64_t step, int32_t* n_accepted, int32_t* out_tokens, int32_t* n_out,
    int32_t* n_commit, int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
    int32_t* next_mask_row0, float* row_stats, float* dbg, void* workspace,
    size_t workspace_bytes, int32_t* status, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!hidden || !w_vocab || !logits) return IDLM_ERR_INVALID_ARG;
  if (H <= 0 || H % 8) return IDLM_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < idlm_lm_head_accept_workspace_size(C, T, N, H, V))
    return IDLM_ERR_WORKSPACE;
  Carver cv(workspace);
  void* acc_ws = cv.take<uint8_t>(acc::workspace_bytes(C, T, V, IDLM_BF16, nullptr, nullptr));
  const int tiles = (V + acc::kLmTile - 1) / acc::kLmTile;
  acc::Partial* tstat = cv.take<acc::Partial>(static_cast<size_t>(T) * tiles);
  const size_t gemm_bytes = lm_head_gemm_workspace(T, H, V);
  void* gemm_ws = cv.take<uint8_t>(gemm_bytes);
  acc::Params p;
  DeviceInfo dev;
  idlm_status rc = accept_prepare(
      p, dev, logits, IDLM_BF16, V, qo_indptr, mode, drafts, draft_q_stats, prev_logits,
      prev_rows, prev_mask_row0, C, T, N, temperature, proposal_mode, seed, step, n_accepted,
      out_tokens, n_out, n_commit, next_drafts, next_q_stats, next_mode, next_mask_row0,
      row_stats, dbg, acc_ws, acc::workspace_bytes(C, T, V, IDLM_BF16, nullptr, nullptr), status);
  if (rc != IDLM_OK) return rc;
  // logits = H W^T and the tile statistics of every row
  rc = lm_head_gemm(hidden, w_vocab, T, H, V, logits, gemm_ws, gemm_bytes, tstat, p.s2,
                    p.greedy, status, stream);
  if (rc != IDLM_OK) return rc;
  const long long warps = static_cast<long long>(T) * p.CH;
  acc::lm_combine_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(
      tstat, tiles, p.part, T, p.CH, p.greedy);
  if (cudaGetLastError() != cudaSuccess) return IDLM_ERR_CUDA;
  p.part_given = 1;
  return accept_launch(p, dev, IDLM_BF16, stream);
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
unsigned long long g_scratch_ctx[64] = {};
}  // namespace

// Device address of g_accept_scratch in the current context, looked up once
// per context.  In host code the array's name is only a host-side handle; the
// kernels need the address cudaGetSymbolAddress returns.  The cache is keyed
// on the context's unique id, so after cudaDeviceReset (or under another
// context on the same device) the address is looked up again instead of
// reusing one from a context that no longer exists.  Where the driver gives
// no context id, every call looks the address up.
void* static_scratch() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] && ctx != 0 && g_scratch_ctx[dev] == ctx) return g_scratch_ptr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess) return nullptr;
  if (ctx == 0) ctx = current_context_id();   // the look-up made the context current
  g_scratch_ptr[dev] = p;
  g_scratch_ctx[dev] = ctx;
  return p;
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
