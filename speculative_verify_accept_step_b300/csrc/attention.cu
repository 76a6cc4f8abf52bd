// a2. Paged strict-causal GQA attention of the ISD step rows.
//
// Source: "Introspective Diffusion Language Models" (project page), sections
// "Training" (strict causal masking over all positions) and "Serving
// (SGLang)" (paged KV cache, paged-only attention kernel).  Row r of request
// c sits at position L_c + r and attends to committed slots 0..L_c-1 (through
// the page table) and to this step's own new rows 0..r; query head h reads
// KV head h / G with G = Hq / Hkv.
//
// Fast path (bf16, D = 128, 16-token pages): one work unit is a (request,
// kv head) pair.  Its G * R query rows (R rows per request, G query heads per
// kv head; 28 at N = 4) are packed into MT m-tiles of 16 rows, so every KV
// byte is read from HBM once per unit and reused by all of them.  Work is the
// list of 16-key blocks of all units (every cached page, then ceil(R / 16)
// blocks of the step's own new rows); a persistent grid splits that list evenly
// (balanced split-KV), so long and short contexts load the SMs equally.
// Units cut by a CTA boundary write partial (max, sum, O) triples to the
// workspace, and a small second kernel, launched as a programmatic dependent,
// merges them once the grid is done: no CTA waits for another, no counter
// or fence sits at the end of a CTA's range, and the sums do not depend on
// timing.
//
// Per CTA: one producer warp issues TMA tile loads (cp.async.bulk.tensor,
// 128-byte swizzle) into an 8-stage shared-memory ring guarded by mbarriers:
// one 4 KB box per K page and one per V page, the two 64-column halves of D
// being the box's outer dimension, with each page id read one block ahead.
// 2*MT consumer warps each own one m-tile and every other pair of blocks (two
// parity groups, 32 keys per step), compute S = Q K^T and O += P V with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) and an fp32 online softmax in
// the log2 domain, release a pair's first stage as soon as its V is read, and
// merge the two parity halves at the end of a unit.
//
// The general path (fp32, or any other D / page size) is a plain kernel with
// one warp per (row, head) walking the keys in order.
#include <algorithm>

#include "common.cuh"
#include "host_util.h"

namespace idlm {
namespace attn {

constexpr int D = 128;
constexpr int PS = 16;
// Ring depth, a multiple of 4: block i is consumed by parity group
// (i >> 1) & 1 from stage i % STAGES, so a stage only ever serves one group,
// whose warps wait on its phases in order, and a pair (i even) sits in two
// stages of one phase.  With another depth a fast warp could wait on stage s
// for block i while block i - STAGES (the other group's) has not landed, and
// the parity test would pass on that older phase.
constexpr int STAGES = 8;
static_assert(STAGES % 4 == 0, "a stage must return to the parity group that read it");
constexpr int BOX_BYTES = PS * 64 * 2;       // 16 rows x 128 bytes
constexpr int STAGE_BYTES = 4 * BOX_BYTES;   // K lo/hi half, V lo/hi half
constexpr int kMaxRequests = 8192;           // prefix array lives in shared memory
constexpr float kNegInf = -__builtin_inff();

struct Params {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* qo_indptr;
  float* ws_o;       // [B][2][MT*16][D]: partial O of a cut unit's part
  float* ws_ml;      // [B][2][MT*16][2]: its (max, sum) per row
  int32_t* status;
  int max_pages, C, T, Hq, Hkv, G, num_pages, max_rows;
  float scale_log2;  // sm_scale * log2(e)
};

template <int MT>
struct Layout {
  static constexpr int kConsumers = 2 * MT;
  static constexpr int kThreads = 32 * (1 + kConsumers);
  static constexpr size_t kStageOff = 0;
  static constexpr size_t kMergeOOff = kStageOff + size_t(STAGES) * STAGE_BYTES;
  static constexpr size_t kMergeMLOff = kMergeOOff + size_t(16) * D * 4;   // one m-tile's O
  static constexpr size_t kBarOff = kMergeMLOff + size_t(MT) * 16 * 2 * 4;
  static constexpr size_t kFlagOff = kBarOff + 2 * STAGES * 8;
  static constexpr size_t kPrefOff = kFlagOff + 16;
  static size_t bytes(int C) { return 1024 + kPrefOff + size_t(C + 1) * 4; }
};

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Position in the global block list -> (request, kv head, block-in-unit).
// A unit's blocks are its nbc cached pages, then its blocks of new rows.
struct Cursor {
  int c, g, k, nb, nbc;
  long long unit_start;
};

// Cached 16-key blocks of request c: ceil(L_c / 16), L_c clamped to the
// request's page-table row.
__device__ __forceinline__ int cached_blocks(const Params& p, int c) {
  const int L = min(max(p.seq_lens[c], 0), p.max_pages * PS);
  return (L + PS - 1) / PS;
}

__device__ __forceinline__ Cursor locate(const Params& p, const int* pref, int C, int Hkv,
                                         long long j) {
  // largest c with Hkv * pref[c] <= j
  int lo = 0, hi = C - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<long long>(Hkv) * pref[mid] <= j) lo = mid; else hi = mid - 1;
  }
  Cursor cur;
  cur.c = lo;
  cur.nb = pref[lo + 1] - pref[lo];
  const long long rel = j - static_cast<long long>(Hkv) * pref[lo];
  cur.g = static_cast<int>(rel / cur.nb);
  cur.k = static_cast<int>(rel % cur.nb);
  cur.unit_start = static_cast<long long>(Hkv) * pref[lo] + static_cast<long long>(cur.g) * cur.nb;
  cur.nbc = cached_blocks(p, lo);
  return cur;
}

// Next block; past the last request's last block the cursor is not read.
__device__ __forceinline__ void advance(Cursor& cur, const Params& p, const int* pref, int C,
                                        int Hkv) {
  if (++cur.k < cur.nb) return;
  cur.k = 0;
  cur.unit_start += cur.nb;
  if (++cur.g < Hkv) return;
  cur.g = 0;
  if (++cur.c >= C) return;
  cur.nb = pref[cur.c + 1] - pref[cur.c];
  cur.nbc = cached_blocks(p, cur.c);
}

// pref[c] = blocks of requests 0 .. c-1: ceil(L / 16) cached pages plus
// ceil(R / 16) blocks of new rows (at least one, so that every unit has a
// block).  Every thread of the CTA calls it; a barrier must follow before
// pref is read.  With check set, bad layouts and lengths go to the status.
template <int NT>
__device__ __forceinline__ void block_prefix(const Params& p, int* pref, bool check) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int C = p.C;
  const int per = (C + NT - 1) / NT;
  const int c0 = min(C, tid * per), c1 = min(C, c0 + per);
  int sum = 0;
  for (int c = c0; c < c1; ++c) {
    int L = p.seq_lens[c];
    const int rows = p.qo_indptr[c + 1] - p.qo_indptr[c];
    if (check) {
      if (L < 0 || rows < 0 || rows > p.max_rows || p.qo_indptr[c] < 0 ||
          p.qo_indptr[c + 1] > p.T)
        set_status(p.status, IDLM_DEV_BAD_LAYOUT);
      if (L > p.max_pages * PS) set_status(p.status, IDLM_DEV_SLOT_OVERFLOW);
    }
    L = min(max(L, 0), p.max_pages * PS);
    const int R = min(max(rows, 0), p.max_rows);
    pref[c + 1] = (L + PS - 1) / PS + max(1, (R + PS - 1) / PS);   // temporarily the count
    sum += pref[c + 1];
  }
  // exclusive scan of the per-thread sums: shuffles within a warp, then the
  // warp totals
  __shared__ int wsum[NT / 32];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  if (tid == 0) pref[0] = 0;
  __syncthreads();
  int acc = incl - sum;
  for (int w = 0; w < warp; ++w) acc += wsum[w];
  for (int c = c0; c < c1; ++c) {
    acc += pref[c + 1];
    pref[c + 1] = acc;
  }
}

__device__ __forceinline__ long long range_lo(long long W, int B, int b) {
  return W * b / B;
}

// Index of the CTA whose range holds block x.
__device__ __forceinline__ int owner_of(long long W, int B, long long x) {
  return static_cast<int>(((x + 1) * B - 1) / W);
}

template <int MT>
__global__ void __launch_bounds__(Layout<MT>::kThreads, MT <= 2 ? 2 : 1)
paged_attn_kernel(const __grid_constant__ CUtensorMap kc_map,
                  const __grid_constant__ CUtensorMap vc_map,
                  const __grid_constant__ CUtensorMap kn_map,
                  const __grid_constant__ CUtensorMap vn_map, const Params p) {
  using LY = Layout<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = base + LY::kStageOff;
  float* merge_o = reinterpret_cast<float*>(base + LY::kMergeOOff);
  float* merge_ml = reinterpret_cast<float*>(base + LY::kMergeMLOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + LY::kBarOff);
  uint64_t* empty = full + STAGES;
  volatile int* flags = reinterpret_cast<volatile int*>(base + LY::kFlagOff);
  int* pref = reinterpret_cast<int*>(base + LY::kPrefOff);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int C = p.C;

  // ---- blocks per request: ceil(L / 16) cached pages + ceil(R / 16) blocks
  // of new rows (at least one, so that every unit has a block)
  if (tid == 0) {
    flags[0] = 0;
    flags[1] = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MT);
    }
    fence_barrier_init();
  }
  block_prefix<LY::kThreads>(p, pref, true);
  fence_proxy_async();
  __syncthreads();

  const long long W = static_cast<long long>(p.Hkv) * pref[C];
  const int B = gridDim.x;
  const long long lo = range_lo(W, B, blockIdx.x);
  const long long hi = range_lo(W, B, blockIdx.x + 1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && lo < hi) {
      prefetch_tensormap(&kc_map);
      prefetch_tensormap(&vc_map);
      prefetch_tensormap(&kn_map);
      prefetch_tensormap(&vn_map);
      Cursor cur = locate(p, pref, C, p.Hkv, lo);
      int issued = 0;
      // the next block's page id is read while this block waits for its stage
      auto page_of = [&](const Cursor& cc) {
        return cc.k < cc.nbc ? p.page_table[static_cast<size_t>(cc.c) * p.max_pages + cc.k] : 0;
      };
      int page_nx = page_of(cur);
      for (long long j = lo; j < hi; ++j) {
        const int page = page_nx;
        Cursor nx = cur;
        advance(nx, p, pref, C, p.Hkv);
        if (j + 1 < hi) page_nx = page_of(nx);
        const int s = issued % STAGES;
        const uint32_t ph = (issued / STAGES) & 1;
        if (!mbar_wait_bounded(&empty[s], ph ^ 1, flags, p.status)) break;
        uint8_t* dst = stages + s * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
        if (cur.k < cur.nbc) {
          int y;
          if (page < 0 || page >= p.num_pages) {
            set_status(p.status, IDLM_DEV_BAD_PAGE);
            y = -2 * PS;   // wholly outside the tensor: the copy fills zeros
          } else {
            y = (page * p.Hkv + cur.g) * PS;
          }
          tma_load_3d(dst, &kc_map, &full[s], 0, y, 0);
          tma_load_3d(dst + 2 * BOX_BYTES, &vc_map, &full[s], 0, y, 0);
        } else {
          // new rows 16 b .. 16 b + 15 of the request (rows past T read zeros)
          const int t0 = p.qo_indptr[cur.c] + PS * (cur.k - cur.nbc);
          tma_load_4d(dst, &kn_map, &full[s], 0, cur.g, t0, 0);
          tma_load_4d(dst + 2 * BOX_BYTES, &vn_map, &full[s], 0, cur.g, t0, 0);
        }
        ++issued;
        cur = nx;
      }
      // every issued copy must land before the CTA may exit
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        mbar_wait_bounded(&full[i % STAGES], (i / STAGES) & 1, nullptr, p.status);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int mt = cw % MT;
  const int par = cw / MT;
  const int qr = lane >> 2;       // fragment row within the m-tile (and +8)
  const int qc = (lane & 3) * 2;  // fragment column pair
  const int G = p.G;
  const int row_a = 16 * mt + qr, row_b = row_a + 8;   // packed rows m
  const int r_a = row_a / G, hl_a = row_a % G;
  const int r_b = row_b / G, hl_b = row_b % G;
  const int key_ld = (lane & 7) + ((lane >> 4) << 3);
  const int kch_off = (lane >> 3) & 1;
  const int vkey = lane & 15;
  const int vch_off = lane >> 4;

  Cursor cur = locate(p, pref, C, p.Hkv, lo < hi ? lo : 0);
  long long j = lo;
  int i = 0;
  while (j < hi) {
    const long long unit_end = cur.unit_start + cur.nb;
    const long long seg_start = j;
    const long long seg_end = min(hi, unit_end);
    const bool whole = (seg_start == cur.unit_start) && (seg_end == unit_end);
    const int c = cur.c, g = cur.g;
    const int L = min(max(p.seq_lens[c], 0), p.max_pages * PS);
    const int t0 = min(max(p.qo_indptr[c], 0), p.T);
    const int R = min(min(max(p.qo_indptr[c + 1] - t0, 0), p.max_rows), p.T - t0);
    const bool va = r_a < R, vb = r_b < R;
    const int nbc = cur.nbc, nb = cur.nb;
    // The unit stays the same within a segment, so the loop below counts
    // only the block within it and moves the cursor once, at the end.
    int kb = cur.k;

    // Q fragments of this m-tile (rows past R are zero)
    uint32_t qa[8][4];
    {
      const uint32_t* qa_ptr = reinterpret_cast<const uint32_t*>(
          p.q + (static_cast<size_t>(t0 + r_a) * p.Hq + g * G + hl_a) * D);
      const uint32_t* qb_ptr = reinterpret_cast<const uint32_t*>(
          p.q + (static_cast<size_t>(t0 + r_b) * p.Hq + g * G + hl_b) * D);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int col = (16 * ks + qc) >> 1;
        qa[ks][0] = va ? __ldg(qa_ptr + col) : 0u;
        qa[ks][1] = vb ? __ldg(qb_ptr + col) : 0u;
        qa[ks][2] = va ? __ldg(qa_ptr + col + 4) : 0u;
        qa[ks][3] = vb ? __ldg(qb_ptr + col + 4) : 0u;
      }
    }

    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;

    // Blocks i and i + 1 (i even) go to parity group (i >> 1) & 1 together
    // when both lie in this segment: 32 keys per step, four independent
    // score chains and one max / rescale for both.  A block whose partner
    // lies in another segment goes alone.
    while (j < seg_end) {
      const bool two = ((i & 1) == 0) && (j + 1 < seg_end);
      const int nblk = two ? 2 : 1;
      if (((i >> 1) & 1) != par) {
        j += nblk;
        i += nblk;
        kb += nblk;
        continue;
      }
      const int s0 = i % STAGES;
      // a pair starts at an even stage, so both blocks share one ring phase
      const uint32_t ph = (i / STAGES) & 1;
      const uint32_t kb0 = smem_u32(stages + s0 * STAGE_BYTES);
      const uint32_t kb1 = kb0 + STAGE_BYTES;
      // S = Q K^T: n-tiles 0, 1 are block i, n-tiles 2, 3 block i + 1; the
      // second stage is awaited only once block i's chain is issued
      float sc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
      auto scores = [&](uint32_t kb, float (&s0_)[4], float (&s1_)[4]) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int ch = 2 * ks + kch_off;
          const uint32_t off = (ch >> 3) * BOX_BYTES + key_ld * 128 +
                               (((ch & 7) ^ (key_ld & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + off, b0, b1, b2, b3);
          mma_bf16_16816(s0_, qa[ks], b0, b1);
          mma_bf16_16816(s1_, qa[ks], b2, b3);
        }
      };
      bool ok = mbar_wait_bounded(&full[s0], ph, flags, p.status);
      if (ok) scores(kb0, sc[0], sc[1]);
      if (two && ok) {
        ok = mbar_wait_bounded(&full[s0 + 1], ph, flags, p.status);
        if (ok) scores(kb1, sc[2], sc[3]);
      }
      bool released = false;
      if (ok) {
        // mask keys past the request's context (cached pages) or past the
        // row's own position (the step's new rows, block b = k - nbc holds
        // rows 16 b ..); a full cached page needs no mask.  Column key =
        // 8n + qc + e within its block.
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int k = kb + bb;
          if (bb == 1 && !two) {
#pragma unroll
            for (int n = 2; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = kNegInf;
            continue;
          }
          const bool full_page = k < nbc && (k + 1) * PS <= L;
          if (!full_page) {
#pragma unroll
            for (int n = 0; n < 2; ++n) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int key = 8 * n + qc + e;
                bool ka, kb;
                if (k < nbc) {
                  ka = kb = (k * PS + key) < L;
                } else {
                  const int nr = PS * (k - nbc) + key;
                  ka = nr <= r_a;
                  kb = nr <= r_b;
                }
                if (!ka) sc[2 * bb + n][e] = kNegInf;
                if (!kb) sc[2 * bb + n][2 + e] = kNegInf;
              }
            }
          }
        }
        // online softmax in the log2 domain: p = 2^(s * scale - m)
        float mx_a = fmaxf(fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1])),
                           fmaxf(fmaxf(sc[2][0], sc[2][1]), fmaxf(sc[3][0], sc[3][1])));
        float mx_b = fmaxf(fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3])),
                           fmaxf(fmaxf(sc[2][2], sc[2][3]), fmaxf(sc[3][2], sc[3][3])));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a * p.scale_log2), mn_b = fmaxf(m_b, mx_b * p.scale_log2);
        const float base_a = mn_a == kNegInf ? 0.f : mn_a;
        const float base_b = mn_b == kNegInf ? 0.f : mn_b;
        // rescale O only when some row's maximum rose (otherwise the factor is 1)
        if (__any_sync(0xffffffffu, mn_a != m_a || mn_b != m_b)) {
          const float corr_a = fast_exp2(m_a - base_a), corr_b = fast_exp2(m_b - base_b);
          l_a *= corr_a;
          l_b *= corr_b;
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            o[n][0] *= corr_a;
            o[n][1] *= corr_a;
            o[n][2] *= corr_b;
            o[n][3] *= corr_b;
          }
          m_a = mn_a;
          m_b = mn_b;
        }
        float pr[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          pr[n][0] = fast_exp2(fmaf(sc[n][0], p.scale_log2, -base_a));
          pr[n][1] = fast_exp2(fmaf(sc[n][1], p.scale_log2, -base_a));
          pr[n][2] = fast_exp2(fmaf(sc[n][2], p.scale_log2, -base_b));
          pr[n][3] = fast_exp2(fmaf(sc[n][3], p.scale_log2, -base_b));
        }
        l_a += ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1])) +
               ((pr[2][0] + pr[2][1]) + (pr[3][0] + pr[3][1]));
        l_b += ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3])) +
               ((pr[2][2] + pr[2][3]) + (pr[3][2] + pr[3][3]));
        uint32_t pa[4], pb[4];
        pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
        pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
        pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
        pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
        pb[0] = pack_bf16x2(pr[2][0], pr[2][1]);
        pb[1] = pack_bf16x2(pr[2][2], pr[2][3]);
        pb[2] = pack_bf16x2(pr[3][0], pr[3][1]);
        pb[3] = pack_bf16x2(pr[3][2], pr[3][3]);
        // O += P V, block i (whose stage is then released) and block i + 1
        auto pv = [&](uint32_t kb, const uint32_t (&pp)[4]) {
#pragma unroll
          for (int dp = 0; dp < 8; ++dp) {
            const int ch = 2 * dp + vch_off;
            const uint32_t off = 2 * BOX_BYTES + (ch >> 3) * BOX_BYTES + vkey * 128 +
                                 (((ch & 7) ^ (vkey & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(kb + off, b0, b1, b2, b3);
            mma_bf16_16816(o[2 * dp], pp, b0, b1);
            mma_bf16_16816(o[2 * dp + 1], pp, b2, b3);
          }
        };
        pv(kb0, pa);
        if (two) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s0]);
          released = true;
          pv(kb1, pb);
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (!released) mbar_arrive(&empty[s0]);
        if (two) mbar_arrive(&empty[s0 + 1]);
      }
      j += nblk;
      i += nblk;
      kb += nblk;
    }
    // on to the next unit's first block
    cur.k = nb - 1;
    advance(cur, p, pref, C, p.Hkv);

    // ---- end of this unit's segment: merge the two parity halves
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    // the m-tiles take turns through one O buffer (all consumer warps meet
    // at named barrier 2 + MT); a smaller CTA footprint and fewer live
    // values measured faster than one buffer per m-tile
    float* mo = merge_o;
    float* mml = merge_ml + mt * 32;
    for (int r = 0; r < MT; ++r) {
      if (mt == r && par == 1) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          *reinterpret_cast<float2*>(mo + qr * D + 8 * n + qc) = make_float2(o[n][0], o[n][1]);
          *reinterpret_cast<float2*>(mo + (qr + 8) * D + 8 * n + qc) = make_float2(o[n][2], o[n][3]);
        }
        if ((lane & 3) == 0) {
          mml[2 * qr] = m_a;
          mml[2 * qr + 1] = l_a;
          mml[2 * (qr + 8)] = m_b;
          mml[2 * (qr + 8) + 1] = l_b;
        }
      }
      named_bar(2 + MT, 64 * MT);
      if (mt == r && par == 0) {
        const float m2a = mml[2 * qr], l2a = mml[2 * qr + 1];
        const float m2b = mml[2 * (qr + 8)], l2b = mml[2 * (qr + 8) + 1];
        const float Ma = fmaxf(m_a, m2a), Mb = fmaxf(m_b, m2b);
        const float ba = Ma == kNegInf ? 0.f : Ma, bb = Mb == kNegInf ? 0.f : Mb;
        const float fa1 = fast_exp2(m_a - ba), fa2 = fast_exp2(m2a - ba);
        const float fb1 = fast_exp2(m_b - bb), fb2 = fast_exp2(m2b - bb);
        l_a = l_a * fa1 + l2a * fa2;
        l_b = l_b * fb1 + l2b * fb2;
        m_a = Ma;
        m_b = Mb;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          const float2 xa = *reinterpret_cast<const float2*>(mo + qr * D + 8 * n + qc);
          const float2 xb = *reinterpret_cast<const float2*>(mo + (qr + 8) * D + 8 * n + qc);
          o[n][0] = o[n][0] * fa1 + xa.x * fa2;
          o[n][1] = o[n][1] * fa1 + xa.y * fa2;
          o[n][2] = o[n][2] * fb1 + xb.x * fb2;
          o[n][3] = o[n][3] * fb1 + xb.y * fb2;
        }
      }
      named_bar(2 + MT, 64 * MT);
    }

    if (par == 0) {
      const int h_a = g * G + hl_a, h_b = g * G + hl_b;
      uint32_t* out_a = reinterpret_cast<uint32_t*>(p.out + (static_cast<size_t>(t0 + r_a) * p.Hq + h_a) * D);
      uint32_t* out_b = reinterpret_cast<uint32_t*>(p.out + (static_cast<size_t>(t0 + r_b) * p.Hq + h_b) * D);
      if (whole) {
        const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          if (va) out_a[(8 * n + qc) >> 1] = pack_bf16x2(o[n][0] * ia, o[n][1] * ia);
          if (vb) out_b[(8 * n + qc) >> 1] = pack_bf16x2(o[n][2] * ib, o[n][3] * ib);
        }
      } else {
        // a part of a unit cut by a CTA boundary: (max, sum, O) for the merge
        // kernel, in slot 0 if this segment opened the CTA's range, else slot 1
        const int slot = (seg_start == lo) ? 0 : 1;
        const size_t sbase = (static_cast<size_t>(blockIdx.x) * 2 + slot) * (MT * 16);
        float* wo = p.ws_o + sbase * D;
        float* wml = p.ws_ml + sbase * 2;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          *reinterpret_cast<float2*>(wo + row_a * D + 8 * n + qc) = make_float2(o[n][0], o[n][1]);
          *reinterpret_cast<float2*>(wo + row_b * D + 8 * n + qc) = make_float2(o[n][2], o[n][3]);
        }
        if ((lane & 3) == 0) {
          wml[2 * row_a] = m_a;
          wml[2 * row_a + 1] = l_a;
          wml[2 * row_b] = m_b;
          wml[2 * row_b + 1] = l_b;
        }
        named_bar(1 + MT, 32 * MT);
      }
    }
  }
}

// ------------------------------------------------------------ merge of cuts
// CTA b merges the unit that CTA b of the attention grid opens at the end of
// its range when that unit goes on into later CTAs (the CTAs bf = b .. bl
// hold its parts): per (row, 4 columns) item, M = the parts' largest max,
// then the sum and O weighted by 2^(max - M), added in CTA order, and O /
// sum.  It is a programmatic dependent of the attention kernel: the block
// prefix and the unit are found before griddepcontrol.wait, the parts read
// after it.  Each thread issues the loads of four items before using any,
// so the merge is one round of loads.  (Measured: 256 threads and one CTA
// per unit beat 128 or 512 threads, four CTAs per unit, and an early launch
// of this grid.)
constexpr int kMergeThreads = 256;
constexpr int kMergeRegParts = 2;   // parts held in registers; more go round a loop
constexpr int kMergeItems = 4;

template <int MT>
__global__ void __launch_bounds__(kMergeThreads)
attn_merge_kernel(const Params p) {
  extern __shared__ int pref[];
  block_prefix<kMergeThreads>(p, pref, false);
  __syncthreads();
  const int C = p.C, B = gridDim.x, b = blockIdx.x;
  const long long W = static_cast<long long>(p.Hkv) * pref[C];
  const long long lo = range_lo(W, B, b), hi = range_lo(W, B, b + 1);
  bool mine = lo < hi;
  Cursor cur;
  if (mine) {
    cur = locate(p, pref, C, p.Hkv, hi - 1);
    mine = cur.unit_start >= lo && cur.unit_start + cur.nb > hi;
  }
  griddep_wait();
  griddep_launch_dependents();
  if (!mine) return;
  const long long ustart = cur.unit_start;
  const int bl = owner_of(W, B, ustart + cur.nb - 1);
  const int c = cur.c, g = cur.g, G = p.G;
  const int t0 = min(max(p.qo_indptr[c], 0), p.T);
  const int R = min(min(max(p.qo_indptr[c + 1] - t0, 0), p.max_rows), p.T - t0);
  // the slot of CTA x's part: 1 for the opener when its range began earlier
  auto part_row = [&](int x) -> size_t {
    const int sl = (x == b && ustart > lo) ? 1 : 0;
    return (static_cast<size_t>(x) * 2 + sl) * (MT * 16);
  };
  auto has_part = [&](int x) { return range_lo(W, B, x) < range_lo(W, B, x + 1); };
  constexpr int Q4 = D / 4;
  const int n = G * R * Q4;
  // the first kMergeRegParts parts: whether they exist and their first rows
  bool okp[kMergeRegParts];
  size_t rowp[kMergeRegParts];
#pragma unroll
  for (int k = 0; k < kMergeRegParts; ++k) {
    okp[k] = b + k <= bl && has_part(b + k);
    rowp[k] = okp[k] ? part_row(b + k) : 0;
  }
  // kMergeItems items per thread at a time: all their loads issued before
  // any of them is used
  for (int i0 = threadIdx.x; i0 < n; i0 += kMergeItems * kMergeThreads) {
    float mp[kMergeItems][kMergeRegParts], lp[kMergeItems][kMergeRegParts];
    float4 xp[kMergeItems][kMergeRegParts];
#pragma unroll
    for (int it = 0; it < kMergeItems; ++it) {
      const int item = i0 + it * kMergeThreads;
      const int m = item / Q4, q4 = item % Q4;
#pragma unroll
      for (int k = 0; k < kMergeRegParts; ++k) {
        if (item < n && okp[k]) {
          const size_t pr = rowp[k] + m;
          mp[it][k] = __ldcg(p.ws_ml + pr * 2);
          lp[it][k] = __ldcg(p.ws_ml + pr * 2 + 1);
          xp[it][k] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + pr * D) + q4);
        }
      }
    }
#pragma unroll
    for (int it = 0; it < kMergeItems; ++it) {
      const int item = i0 + it * kMergeThreads;
      if (item >= n) break;
      const int m = item / Q4, q4 = item % Q4;
      float M = kNegInf;
#pragma unroll
      for (int k = 0; k < kMergeRegParts; ++k)
        if (okp[k]) M = fmaxf(M, mp[it][k]);
      for (int x = b + kMergeRegParts; x <= bl; ++x)
        if (has_part(x)) M = fmaxf(M, __ldcg(p.ws_ml + (part_row(x) + m) * 2));
      const float base = M == kNegInf ? 0.f : M;
      float L = 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      auto add = [&](float mx, float l, float4 x) {
        const float f = fast_exp2(mx - base);
        L = fmaf(f, l, L);
        o.x = fmaf(f, x.x, o.x);
        o.y = fmaf(f, x.y, o.y);
        o.z = fmaf(f, x.z, o.z);
        o.w = fmaf(f, x.w, o.w);
      };
#pragma unroll
      for (int k = 0; k < kMergeRegParts; ++k)
        if (okp[k]) add(mp[it][k], lp[it][k], xp[it][k]);
      for (int x = b + kMergeRegParts; x <= bl; ++x) {
        if (!has_part(x)) continue;
        const size_t pr = part_row(x) + m;
        add(__ldcg(p.ws_ml + pr * 2), __ldcg(p.ws_ml + pr * 2 + 1),
            __ldcg(reinterpret_cast<const float4*>(p.ws_o + pr * D) + q4));
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const int r = m / G, h = g * G + m % G;
      uint2 v;
      v.x = pack_bf16x2(o.x * inv, o.y * inv);
      v.y = pack_bf16x2(o.z * inv, o.w * inv);
      reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(t0 + r) * p.Hq + h) * D)[q4] = v;
    }
  }
}

// --------------------------------------------------------------- general path
// One warp per (row, query head); lanes split D; keys visited in order with
// an online softmax in fp32.  Any page size, D a multiple of 32 up to 256.
template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st_f(T* p, float v);
template <>
__device__ __forceinline__ void st_f<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

template <typename T>
__global__ void __launch_bounds__(128)
simple_attn_kernel(const T* q, const T* k_new, const T* v_new, const T* k_cache,
                   const T* v_cache, const int32_t* page_table, int max_pages,
                   const int32_t* seq_lens, const int32_t* qo_indptr, int C, int T_rows,
                   int Hq, int Hkv, int D_, int page_size, int num_pages, int max_rows,
                   float scale, T* out, int32_t* status) {
  const int t = blockIdx.x;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T_rows || h >= Hq) return;
  // request of row t
  int lo = 0, hi = C - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qo_indptr[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int c = lo;
  const int t0 = qo_indptr[c];
  const int r = t - t0;
  const int rows = qo_indptr[c + 1] - t0;
  if (rows > max_rows || seq_lens[c] < 0) set_status(status, IDLM_DEV_BAD_LAYOUT);
  const int L = max(seq_lens[c], 0);
  const int g = h / (Hq / Hkv);
  const int per = D_ / 32;  // elements per lane
  float qv[8], acc[8];
  for (int e = 0; e < per; ++e) {
    qv[e] = ld_f(q + (static_cast<size_t>(t) * Hq + h) * D_ + lane * per + e);
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int total = L + r + 1;
  for (int s = 0; s < total; ++s) {
    const T* kp;
    const T* vp;
    if (s < L) {
      const int pi = s / page_size;
      int page = pi < max_pages ? page_table[static_cast<size_t>(c) * max_pages + pi] : -1;
      if (page < 0 || page >= num_pages) {
        set_status(status, IDLM_DEV_BAD_PAGE);
        continue;
      }
      const size_t off = ((static_cast<size_t>(page) * Hkv + g) * page_size + s % page_size) * D_;
      kp = k_cache + off;
      vp = v_cache + off;
    } else {
      const size_t off = (static_cast<size_t>(t0 + (s - L)) * Hkv + g) * D_;
      kp = k_new + off;
      vp = v_new + off;
    }
    float dot = 0.f;
    for (int e = 0; e < per; ++e) dot += qv[e] * ld_f(kp + lane * per + e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const float sc = dot * scale;
    const float mn = fmaxf(m, sc);
    const float corr = expf(m - mn);
    const float pr = expf(sc - mn);
    l = l * corr + pr;
    for (int e = 0; e < per; ++e) acc[e] = acc[e] * corr + pr * ld_f(vp + lane * per + e);
    m = mn;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  for (int e = 0; e < per; ++e)
    st_f(out + (static_cast<size_t>(t) * Hq + h) * D_ + lane * per + e, acc[e] * inv);
}

template <int MT>
size_t workspace_for(int C, int Hkv, int B) {
  Carver cv(nullptr);
  cv.take<float>(static_cast<size_t>(B) * 2 * MT * 16 * D);
  cv.take<float>(static_cast<size_t>(B) * 2 * MT * 16 * 2);
  return cv.used;
}

template <int MT>
int grid_for(const DeviceInfo& dev, int C) {
  const size_t smem = Layout<MT>::bytes(C);
  int per_sm = 0;
  if (cudaFuncSetAttribute(paged_attn_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, paged_attn_kernel<MT>,
                                                    Layout<MT>::kThreads, smem) != cudaSuccess)
    return 0;
  return dev.sm_count * std::max(per_sm, 1);
}

inline int mtiles_for(int G, int max_rows) { return (G * max_rows + 15) / 16; }

bool use_fast_path(int dtype, int D_, int page_size, int G, int max_rows, int C) {
  const int mtl = mtiles_for(G, max_rows);
  return dtype == IDLM_BF16 && D_ == D && page_size == PS && mtl >= 1 && mtl <= 4 &&
         C <= kMaxRequests;
}

template <int MT>
idlm_status launch_fast(const DeviceInfo& dev, const void* q, const void* k_new,
                        const void* v_new, const void* k_cache, const void* v_cache,
                        const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                        const int32_t* qo_indptr, int C, int T, int Hq, int Hkv,
                        int num_pages, int max_rows, float sm_scale, void* out,
                        void* workspace, size_t ws_bytes, int32_t* status,
                        cudaStream_t stream) {
  const int B = grid_for<MT>(dev, C);
  if (B <= 0) return IDLM_ERR_CUDA;
  if (ws_bytes < workspace_for<MT>(C, Hkv, B) || !workspace) return IDLM_ERR_WORKSPACE;
  Carver cv(workspace);
  Params p;
  p.ws_o = cv.take<float>(static_cast<size_t>(B) * 2 * MT * 16 * D);
  p.ws_ml = cv.take<float>(static_cast<size_t>(B) * 2 * MT * 16 * 2);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.qo_indptr = qo_indptr;
  p.status = status;
  p.max_pages = max_pages;
  p.C = C;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.num_pages = num_pages;
  p.max_rows = max_rows;
  p.scale_log2 = sm_scale * kLog2e;

  CUtensorMap kc, vc, kn, vn;
  // Dimensions: 64 columns, rows, then the half of D (stride 128 bytes) as
  // the outermost, so one box of a 16-row page lands as [half][row][64
  // columns], 128-byte swizzled: the layout the consumers' ldmatrix reads.
  const uint64_t cdims[3] = {64, static_cast<uint64_t>(num_pages) * Hkv * PS, 2};
  const uint64_t cstr[2] = {D * 2, 128};
  const uint32_t cbox[3] = {64, PS, 2};
  const uint64_t ndims[4] = {64, static_cast<uint64_t>(Hkv), static_cast<uint64_t>(T), 2};
  const uint64_t nstr[3] = {D * 2, static_cast<uint64_t>(Hkv) * D * 2, 128};
  const uint32_t nbox[4] = {64, 1, PS, 2};
  if (!encode_bf16_map(&kc, const_cast<void*>(k_cache), 3, cdims, cstr, cbox) ||
      !encode_bf16_map(&vc, const_cast<void*>(v_cache), 3, cdims, cstr, cbox) ||
      !encode_bf16_map(&kn, const_cast<void*>(k_new), 4, ndims, nstr, nbox) ||
      !encode_bf16_map(&vn, const_cast<void*>(v_new), 4, ndims, nstr, nbox))
    return IDLM_ERR_CUDA;

  paged_attn_kernel<MT><<<B, Layout<MT>::kThreads, Layout<MT>::bytes(C), stream>>>(kc, vc, kn, vn, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  // the merge starts as the attention CTAs finish (a programmatic
  // dependent), or after the whole grid where the stream does not allow it
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(C + 1) * sizeof(int);
  e = cudaLaunchKernelEx(&cfg, attn_merge_kernel<MT>, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, attn_merge_kernel<MT>, p);
  }
  return cuda_status(e);
}

}  // namespace attn
}  // namespace idlm

using namespace idlm;

extern "C" size_t idlm_isd_attention_workspace_size(int C, int Hq, int Hkv, int D_,
                                                    int page_size, int max_rows, int dtype) {
  if (C <= 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv) return 0;
  const int G = Hq / Hkv;
  if (!attn::use_fast_path(dtype, D_, page_size, G, max_rows, C)) return 256;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return 0;
  switch (attn::mtiles_for(G, max_rows)) {
    case 1: return attn::workspace_for<1>(C, Hkv, attn::grid_for<1>(dev, C));
    case 2: return attn::workspace_for<2>(C, Hkv, attn::grid_for<2>(dev, C));
    case 3: return attn::workspace_for<3>(C, Hkv, attn::grid_for<3>(dev, C));
    default: return attn::workspace_for<4>(C, Hkv, attn::grid_for<4>(dev, C));
  }
}

extern "C" idlm_status idlm_isd_attention(
    const void* q, const void* k_new, const void* v_new, const void* k_cache,
    const void* v_cache, const int32_t* page_table, int max_pages, const int32_t* seq_lens,
    const int32_t* qo_indptr, int C, int T, int Hq, int Hkv, int D_, int page_size,
    int num_pages, int max_rows, float sm_scale, int dtype, void* out, void* workspace,
    size_t workspace_bytes, int32_t* status, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !page_table || !seq_lens ||
      !qo_indptr || !out || !status)
    return IDLM_ERR_INVALID_ARG;
  if (C <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D_ <= 0 || page_size <= 0 ||
      num_pages <= 0 || max_pages <= 0 || max_rows <= 0 || !(sm_scale > 0.f))
    return IDLM_ERR_INVALID_ARG;
  if (dtype != IDLM_BF16 && dtype != IDLM_F32) return IDLM_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (attn::use_fast_path(dtype, D_, page_size, G, max_rows, C)) {
    DeviceInfo dev;
    if (!current_device_info(&dev)) return IDLM_ERR_CUDA;
    // TMA needs 16-byte aligned bases
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
         reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
      return IDLM_ERR_INVALID_ARG;
#define IDLM_FAST(MT)                                                                          \
  return attn::launch_fast<MT>(dev, q, k_new, v_new, k_cache, v_cache, page_table, max_pages, \
                               seq_lens, qo_indptr, C, T, Hq, Hkv, num_pages, max_rows,       \
                               sm_scale, out, workspace, workspace_bytes, status, stream)
    switch (attn::mtiles_for(G, max_rows)) {
      case 1: IDLM_FAST(1);
      case 2: IDLM_FAST(2);
      case 3: IDLM_FAST(3);
      default: IDLM_FAST(4);
    }
#undef IDLM_FAST
  }
  if (D_ % 32 || D_ > 256) return IDLM_ERR_UNSUPPORTED;
  dim3 grid(T, (Hq + 3) / 4);
  if (dtype == IDLM_BF16) {
    attn::simple_attn_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_new),
        static_cast<const __nv_bfloat16*>(v_new), static_cast<const __nv_bfloat16*>(k_cache),
        static_cast<const __nv_bfloat16*>(v_cache), page_table, max_pages, seq_lens, qo_indptr,
        C, T, Hq, Hkv, D_, page_size, num_pages, max_rows, sm_scale,
        static_cast<__nv_bfloat16*>(out), status);
  } else {
    attn::simple_attn_kernel<float><<<grid, 128, 0, stream>>>(
        static_cast<const float*>(q), static_cast<const float*>(k_new),
        static_cast<const float*>(v_new), static_cast<const float*>(k_cache),
        static_cast<const float*>(v_cache), page_table, max_pages, seq_lens, qo_indptr, C, T,
        Hq, Hkv, D_, page_size, num_pages, max_rows, sm_scale, static_cast<float*>(out),
        status);
  }
  return cuda_status(cudaGetLastError());
}
