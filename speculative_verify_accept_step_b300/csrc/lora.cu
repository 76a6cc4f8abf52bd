// a3. Gated-LoRA projection: Y = X W^T + g_row * s * (X A^T) B^T, the LoRA
// term present only at MASK rows (g = 1) and absent at clean rows (g = 0).
//
// Source: "Introspective Diffusion Language Models" (project page), section
// "Lossless R-ISD" (a LoRA adapter applied only at MASK positions; verify
// positions keep the base weights, so their outputs equal the base model's
// bit for bit) and the speedup panel (R-ISD overhead alpha = 1.12).
//
// The step's token rows are few (M = C (2N - 1) = 448 at C = 64, N = 4) and
// the weights are large (N x K up to 12288 x 4096), so the tensor-core tile
// puts the weight rows on the MMA's M side and the tokens on its N side:
// one CTA accumulates a [128 weight rows x M tokens] tile of Y^T in tensor
// memory (up to 448 tokens per launch: two MMAs of N <= 256 per K step in
// 512 TMEM columns), reading each weight byte once from HBM while X stays in L2.
//
// The LoRA term is one more K step of the same accumulation: the operands
// of that step are B (the weight side, [N x r]) and T = g s X A^T (the token
// side, [M x r]), both copied to the workspace as rows of 64 values (zeros
// past r) so they load like any other K block.  Rows with g = 0 have T = 0,
// which adds exact zeros to their fp32 accumulators: their outputs are
// bit-identical to the base projection computed by this kernel without the
// adapter.
//
// Kernels:
//   lora_t_kernel     T = g s X A^T in fp32 on CUDA cores, stored as bf16
//                     (a [M x r] product, 0.03% of the flops), and B padded
//                     to 64 columns.
//   lora_gemm_kernel  tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in
//                     TMEM), operands staged by TMA (cp.async.bulk.tensor,
//                     128-byte swizzle) in a 3-stage ring.  Warp 0 issues
//                     the loads, warp 1 owns TMEM and issues the MMAs (one
//                     thread), warps 2-5 drain TMEM with tcgen05.ld and
//                     write Y.  A programmatic dependent of lora_t_kernel:
//                     only the load of T waits for it.
// Every mbarrier wait is bounded; a wait that runs out records
// IDLM_DEV_TIMEOUT, and the CTA drains its copies and MMAs and frees its
// tensor memory before it leaves.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace idlm {
namespace lora {

constexpr int kBK = 64;                    // K values per stage (128 bytes of bf16)
constexpr int kTileN = 128;                // weight rows per tile (MMA M)
constexpr int kStages = 3;
constexpr int kMaxTokens = 448;            // tokens per launch: TMEM columns (<= 512) and a
                                           // 3-stage ring of 72 KB stages
constexpr int kThreads = 192;              // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kTmemCols = 512;        // allocation: a power of two >= the tokens
constexpr uint32_t kWBytes = kTileN * kBK * 2;   // 16 KB

struct Params {
  __nv_bfloat16* y;
  const uint8_t* row_gate;
  int32_t* status;
  int M, K, N, r;
  int m16;        // tokens rounded up to 16
  int n1, n2;     // MMA N of the two token blocks (n1 <= 256, n2 = m16 - n1)
  int tiles, kb;  // weight-row tiles, K blocks
  uint32_t stage_bytes;
};

// ------------------------------------------------------------- tcgen05 PTX

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has finished.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes: v[j] = column col + j
// of lane (32 * (warp % 4) + lane id).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A
// and B, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 4)                              // D format: fp32
         | (1u << 7)                            // A format: bf16
         | (1u << 10)                           // B format: bf16
         | (static_cast<uint32_t>(n >> 3) << 17)
         | (static_cast<uint32_t>(m >> 4) << 24);
}

// Shared-memory matrix descriptor: K-major operand written by TMA with the
// 128-byte swizzle (rows of 128 bytes, 8-row groups 1024 bytes apart).
// `saddr` must sit in a 1024-byte aligned group.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3ffff) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
  return d;
}

// ------------------------------------------------------------------ T = g s X A^T
//
// The first ceil(M / 4) CTAs: one CTA per 4 token rows; each thread
// accumulates the 4 x r partial dots of its K-slice, then the block sums
// them.  Rows with g = 0 get zeros.  T is stored [M x 64] (zeros past r).
// The remaining CTAs copy B [N x r] to B64 [N x 64] (zeros past r), so that
// both operands of the LoRA step are plain 128-byte rows for TMA.
constexpr int kTRows = 4;
constexpr int kTThreads = 256;
constexpr int kPadW = 64;   // padded LoRA rank

__global__ void __launch_bounds__(kTThreads) lora_t_kernel(const __nv_bfloat16* x,
                                                           const __nv_bfloat16* a,
                                                           const __nv_bfloat16* b,
                                                           const uint8_t* gate, float scale,
                                                           int M, int K, int N, int r,
                                                           __nv_bfloat16* t64,
                                                           __nv_bfloat16* b64) {
  __shared__ float red[kTThreads / 32][kTRows][16];
  griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tblocks = (M + kTRows - 1) / kTRows;
  if (static_cast<int>(blockIdx.x) >= tblocks) {
    const int n = (blockIdx.x - tblocks) * kTThreads + tid;
    if (n < N)
      for (int j = 0; j < kPadW; ++j)
        b64[static_cast<size_t>(n) * kPadW + j] =
            j < r ? b[static_cast<size_t>(n) * r + j] : __float2bfloat16_rn(0.f);
    return;
  }
  const int m0 = blockIdx.x * kTRows;
  // zero the padding and the ungated rows
  for (int e = tid; e < kTRows * kPadW; e += kTThreads) {
    const int i = e / kPadW, j = e % kPadW;
    if (m0 + i < M && (j >= r || !gate[m0 + i]))
      t64[static_cast<size_t>(m0 + i) * kPadW + j] = __float2bfloat16_rn(0.f);
  }
  bool any = false;
  for (int i = 0; i < kTRows; ++i) any |= (m0 + i < M) && gate[m0 + i];
  if (!any) return;
  for (int j0 = 0; j0 < r; j0 += 16) {
    const int nj = min(16, r - j0);
    float acc[kTRows][16];
#pragma unroll
    for (int i = 0; i < kTRows; ++i)
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[i][j] = 0.f;
    for (int k = tid * 8; k < K; k += kTThreads * 8) {
      float xv[kTRows][8];
#pragma unroll
      for (int i = 0; i < kTRows; ++i) {
        if (m0 + i < M) {
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(m0 + i) * K + k));
          xv[i][0] = bf16_lo(w.x); xv[i][1] = bf16_hi(w.x);
          xv[i][2] = bf16_lo(w.y); xv[i][3] = bf16_hi(w.y);
          xv[i][4] = bf16_lo(w.z); xv[i][5] = bf16_hi(w.z);
          xv[i][6] = bf16_lo(w.w); xv[i][7] = bf16_hi(w.w);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) xv[i][e] = 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (j < nj) {
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(a + static_cast<size_t>(j0 + j) * K + k));
          const float av[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                               bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
          for (int i = 0; i < kTRows; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][j] = fmaf(xv[i][e], av[e], acc[i][j]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kTRows; ++i)
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float v = acc[i][j];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp][i][j] = v;
      }
    __syncthreads();
    if (tid < kTRows * 16) {
      const int i = tid / 16, j = tid % 16;
      if (j < nj && m0 + i < M && gate[m0 + i]) {
        float v = 0.f;
        for (int w = 0; w < kTThreads / 32; ++w) v += red[w][i][j];
        t64[static_cast<size_t>(m0 + i) * kPadW + j0 + j] = __float2bfloat16_rn(v * scale);
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------ the GEMM

// Dynamic shared memory: the stage ring (1024-byte aligned), then barriers.
__host__ __device__ inline size_t bar_offset(uint32_t stage_bytes) {
  return size_t(kStages) * stage_bytes;
}
inline size_t smem_bytes(uint32_t stage_bytes) { return 1024 + bar_offset(stage_bytes) + 256; }

__global__ void __launch_bounds__(kThreads, 1)
lora_gemm_kernel(const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap x_map1,
                 const __grid_constant__ CUtensorMap x_map2, const __grid_constant__ CUtensorMap b_map,
                 const __grid_constant__ CUtensorMap t_map1, const __grid_constant__ CUtensorMap t_map2,
                 const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + bar_offset(p.stage_bytes));
  uint64_t* full = bars;                    // [kStages] TMA -> MMA
  uint64_t* empty = bars + kStages;         // [kStages] MMA -> TMA
  uint64_t* tmem_full = bars + 2 * kStages; // MMA -> epilogue
  uint64_t* tmem_empty = tmem_full + 1;     // epilogue -> MMA
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(tmem_empty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 4);   // one arrival per epilogue warp
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base;
  const int nsteps = p.kb + 1;   // K blocks, then the LoRA block

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&w_map);
      prefetch_tensormap(&x_map1);
      prefetch_tensormap(&x_map2);
      int issued = 0;
      bool ok = true;
      bool t_ready = false;
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
        for (int k = 0; k < nsteps; ++k, ++issued) {
          const int s = issued % kStages;
          const uint32_t ph = (issued / kStages) & 1;
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* st = base + size_t(s) * p.stage_bytes;
          mbar_arrive_expect_tx(&full[s], p.stage_bytes);
          if (k < p.kb) {
            tma_load_2d(st, &w_map, &full[s], k * kBK, tile * kTileN);
            tma_load_2d(st + kWBytes, &x_map1, &full[s], k * kBK, 0);
            if (p.n2) tma_load_2d(st + kWBytes + p.n1 * 128, &x_map2, &full[s], k * kBK, p.n1);
          } else {
            if (!t_ready) {   // T comes from lora_t_kernel
              griddep_wait();
              t_ready = true;
            }
            tma_load_2d(st, &b_map, &full[s], 0, tile * kTileN);
            tma_load_2d(st + kWBytes, &t_map1, &full[s], 0, 0);
            if (p.n2) tma_load_2d(st + kWBytes + p.n1 * 128, &t_map2, &full[s], 0, p.n1);
          }
        }
      }
      // every issued copy lands before the CTA may leave
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, nullptr, p.status);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc1 = make_idesc(kTileN, p.n1);
      const uint32_t idesc2 = make_idesc(kTileN, p.n2 ? p.n2 : 16);
      const int ksub_lora = (p.r + 15) / 16;
      int consumed = 0, t_iter = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, ++t_iter) {
        // the epilogue has drained the previous tile's accumulator
        if (!mbar_wait_bounded(tmem_empty, (t_iter & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        for (int k = 0; k < nsteps; ++k, ++consumed) {
          const int s = consumed % kStages;
          const uint32_t ph = (consumed / kStages) & 1;
          if (!mbar_wait_bounded(&full[s], ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(base + size_t(s) * p.stage_bytes);
          const uint64_t a_desc = make_sdesc(sa);
          const uint64_t b1_desc = make_sdesc(sa + kWBytes);
          const uint64_t b2_desc = make_sdesc(sa + kWBytes + p.n1 * 128);
          const int nsub = k < p.kb ? kBK / 16 : ksub_lora;
          for (int j = 0; j < nsub; ++j) {
            // advance 16 values (32 bytes) along K inside the swizzled rows
            const uint64_t off = static_cast<uint64_t>(j * 2);
            const uint32_t acc = (k > 0 || j > 0) ? 1u : 0u;
            mma_bf16(tmem, a_desc + off, b1_desc + off, idesc1, acc);
            if (p.n2) mma_bf16(tmem + p.n1, a_desc + off, b2_desc + off, idesc2, acc);
          }
          mma_commit(&empty[s]);   // the stage is free once these MMAs finish
        }
        mma_commit(tmem_full);     // the tile's accumulator is complete
      }
      // no MMA may still run when the tensor memory is freed
      if (*abort_flag) {
        mma_commit(tmem_full);
        mbar_wait_bounded(tmem_full, t_iter & 1, nullptr, p.status);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    int t_iter = 0;
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++t_iter) {
      if (!mbar_wait_bounded(tmem_full, t_iter & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const int n = tile * kTileN + q * 32 + lane;   // weight row = output column
      for (int c0 = 0; c0 < p.m16; c0 += 32) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, v);
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = c0 + j;
            if (m < p.M) p.y[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(v[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace lora
}  // namespace idlm

using namespace idlm;

namespace {

struct LoraPlan {
  int m16, n1, n2, tiles, kb;
  uint32_t stage_bytes;
  size_t smem;
};

LoraPlan plan_for(int M, int K, int N) {
  LoraPlan pl;
  pl.m16 = (M + 15) / 16 * 16;
  pl.n1 = std::min(256, pl.m16);
  pl.n2 = pl.m16 - pl.n1;
  pl.tiles = (N + lora::kTileN - 1) / lora::kTileN;
  pl.kb = (K + lora::kBK - 1) / lora::kBK;
  pl.stage_bytes = lora::kWBytes + static_cast<uint32_t>(pl.m16) * 128;
  pl.stage_bytes = (pl.stage_bytes + 1023) / 1024 * 1024;
  pl.smem = lora::smem_bytes(pl.stage_bytes);
  return pl;
}

}  // namespace

extern "C" size_t idlm_gated_lora_workspace_size(int M, int K, int N, int r) {
  if (M <= 0 || K <= 0 || N <= 0 || r <= 0) return 0;
  const int Ms = std::min(M, lora::kMaxTokens);
  return align_up(static_cast<size_t>(Ms) * lora::kPadW * 2, 256) +
         align_up(static_cast<size_t>(N) * lora::kPadW * 2, 256);
}

extern "C" idlm_status idlm_gated_lora(const void* x, const void* w, const void* lora_a,
                                       const void* lora_b, const uint8_t* row_gate,
                                       float lora_scale, int M, int K, int N, int r, void* y,
                                       void* workspace, size_t workspace_bytes, int32_t* status,
                                       void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!x || !w || !lora_a || !lora_b || !row_gate || !y || !status) return IDLM_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0 || N <= 0 || r <= 0) return IDLM_ERR_INVALID_ARG;
  if (K % 8 || r % 8 || r > 64) return IDLM_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) |
       reinterpret_cast<uintptr_t>(lora_a) | reinterpret_cast<uintptr_t>(lora_b)) & 15)
    return IDLM_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < idlm_gated_lora_workspace_size(M, K, N, r))
    return IDLM_ERR_WORKSPACE;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return IDLM_ERR_CUDA;
  static std::mutex mu;
  static bool done[64] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64) return IDLM_ERR_CUDA;
    if (!done[dev.device]) {
      if (cudaFuncSetAttribute(lora::lora_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               dev.max_smem_optin) != cudaSuccess)
        return IDLM_ERR_CUDA;
      done[dev.device] = true;
    }
  }
  __nv_bfloat16* t = static_cast<__nv_bfloat16*>(workspace);
  __nv_bfloat16* b64 = reinterpret_cast<__nv_bfloat16*>(
      static_cast<uint8_t*>(workspace) +
      align_up(static_cast<size_t>(std::min(M, lora::kMaxTokens)) * lora::kPadW * 2, 256));
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(y);
  // token rows in slices of at most 512 (the tensor-memory columns)
  for (int m0 = 0; m0 < M; m0 += lora::kMaxTokens) {
    const int Ms = std::min(lora::kMaxTokens, M - m0);
    const LoraPlan pl = plan_for(Ms, K, N);
    if (pl.smem > static_cast<size_t>(dev.max_smem_optin)) return IDLM_ERR_UNSUPPORTED;
    const __nv_bfloat16* xs = xb + static_cast<size_t>(m0) * K;
    CUtensorMap wm, xm1, xm2, bm, tm1, tm2;
    const uint64_t wdims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
    const uint64_t wstr[1] = {static_cast<uint64_t>(K) * 2};
    const uint32_t wbox[2] = {lora::kBK, lora::kTileN};
    const uint64_t xdims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(Ms)};
    const uint32_t xbox1[2] = {lora::kBK, static_cast<uint32_t>(pl.n1)};
    const uint32_t xbox2[2] = {lora::kBK, static_cast<uint32_t>(pl.n2 ? pl.n2 : 16)};
    const uint64_t bdims[2] = {static_cast<uint64_t>(lora::kPadW), static_cast<uint64_t>(N)};
    const uint64_t rstr[1] = {static_cast<uint64_t>(lora::kPadW) * 2};
    const uint64_t tdims[2] = {static_cast<uint64_t>(lora::kPadW), static_cast<uint64_t>(Ms)};
    if (!encode_bf16_map(&wm, const_cast<void*>(w), 2, wdims, wstr, wbox) ||
        !encode_bf16_map(&xm1, const_cast<__nv_bfloat16*>(xs), 2, xdims, wstr, xbox1) ||
        !encode_bf16_map(&xm2, const_cast<__nv_bfloat16*>(xs), 2, xdims, wstr, xbox2) ||
        !encode_bf16_map(&bm, b64, 2, bdims, rstr, wbox) ||
        !encode_bf16_map(&tm1, t, 2, tdims, rstr, xbox1) ||
        !encode_bf16_map(&tm2, t, 2, tdims, rstr, xbox2))
      return IDLM_ERR_CUDA;

    const int tblocks = (Ms + lora::kTRows - 1) / lora::kTRows;
    const int bblocks = (N + lora::kTThreads - 1) / lora::kTThreads;
    lora::lora_t_kernel<<<tblocks + bblocks, lora::kTThreads, 0, stream>>>(
        xs, static_cast<const __nv_bfloat16*>(lora_a), static_cast<const __nv_bfloat16*>(lora_b),
        row_gate + m0, lora_scale, Ms, K, N, r, t, b64);
    if (cudaGetLastError() != cudaSuccess) return IDLM_ERR_CUDA;

    lora::Params p;
    p.y = yb + static_cast<size_t>(m0) * N;
    p.row_gate = row_gate + m0;
    p.status = status;
    p.M = Ms;
    p.K = K;
    p.N = N;
    p.r = r;
    p.m16 = pl.m16;
    p.n1 = pl.n1;
    p.n2 = pl.n2;
    p.tiles = pl.tiles;
    p.kb = pl.kb;
    p.stage_bytes = pl.stage_bytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(pl.tiles, dev.sm_count));
    cfg.blockDim = dim3(lora::kThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lora::lora_gemm_kernel, wm, xm1, xm2, bm, tm1, tm2, p);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      cfg.numAttrs = 0;
      e = cudaLaunchKernelEx(&cfg, lora::lora_gemm_kernel, wm, xm1, xm2, bm, tm1, tm2, p);
    }
    if (e != cudaSuccess) return IDLM_ERR_CUDA;
  }
  return IDLM_OK;
}
