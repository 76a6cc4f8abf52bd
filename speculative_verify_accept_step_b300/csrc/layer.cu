// One R-ISD decoder layer over the step's rows: the gated-LoRA projections,
// the paged strict-causal attention and the elementwise work between them.
//
// Sources: "Introspective Diffusion Language Models" (project page),
// sections "Lossless R-ISD" (LoRA adapters of rank 128 applied only at MASK
// positions, so that clean positions reproduce the base model bit for bit;
// R-ISD overhead alpha = 1.12 in the speedup panel) and "Training" (strict
// causal attention).  The pages do not spell out the layer; this is the
// pre-norm layout of the Qwen3-style base models they convert:
//
//   n1  = RMSNorm(x)                        h   = x + o
//   qkv = n1 [Wq|Wk|Wv]^T (+ gated LoRA)    n2  = RMSNorm(h)
//   a   = attention(q, k, v, paged KV)      gu  = n2 [Wg|Wu]^T (+ gated LoRA)
//   o   = a Wo^T (+ gated LoRA)             out = h + (silu(g) * u) Wd^T (+ gated LoRA)
//
// RMSNorm(v) = v / sqrt(mean(v^2) + eps) * weight (weight 1 when absent).
// Every activation is stored in bf16 between the kernels; reductions and
// elementwise arithmetic run in fp32.
#include <algorithm>

#include "common.cuh"
#include "host_util.h"

namespace idlm {
namespace layer {

constexpr int kThreads = 256;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* v) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
  v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
  v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}
__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// One CTA per row: h = x (+ r), rounded to bf16 (written to h_out if given);
// n = h / sqrt(mean(h^2) + eps) * weight (written to n_out if given).
__global__ void __launch_bounds__(kThreads)
residual_rmsnorm_kernel(const __nv_bfloat16* x, const __nv_bfloat16* r, __nv_bfloat16* h_out,
                        __nv_bfloat16* n_out, const __nv_bfloat16* weight, int H, float eps) {
  __shared__ float red[kThreads / 32];
  const size_t row = blockIdx.x;
  const __nv_bfloat16* xr = x + row * H;
  const __nv_bfloat16* rr = r ? r + row * H : nullptr;
  float ss = 0.f;
  for (int i = threadIdx.x * 8; i < H; i += kThreads * 8) {
    float a[8], b[8];
    load8(xr + i, a);
    if (rr) {
      load8(rr + i, b);
#pragma unroll
      for (int e = 0; e < 8; ++e) a[e] = round_bf16(a[e] + b[e]);
    }
    if (h_out) store8(h_out + row * H + i, a);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(a[e], a[e], ss);
  }
  if (!n_out) return;
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) tot += red[w];
  const float inv = rsqrtf(tot / static_cast<float>(H) + eps);
  for (int i = threadIdx.x * 8; i < H; i += kThreads * 8) {
    float a[8], b[8], g[8];
    load8(xr + i, a);
    if (rr) {
      load8(rr + i, b);
#pragma unroll
      for (int e = 0; e < 8; ++e) a[e] = round_bf16(a[e] + b[e]);
    }
    if (weight) load8(weight + i, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] = a[e] * inv * (weight ? g[e] : 1.f);
    store8(n_out + row * H + i, a);
  }
}

// qkv [M, (Hq + 2 Hkv) D] -> q [M, Hq D], k [M, Hkv D], v [M, Hkv D].
__global__ void __launch_bounds__(kThreads)
split_qkv_kernel(const __nv_bfloat16* qkv, __nv_bfloat16* q, __nv_bfloat16* k, __nv_bfloat16* v,
                 int M, int nq, int nkv) {
  const int width = nq + 2 * nkv;
  const long long total = static_cast<long long>(M) * width / 8;
  for (long long i = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * kThreads) {
    const int m = static_cast<int>(i / (width / 8));
    const int c = static_cast<int>(i % (width / 8)) * 8;
    const uint4 w = *reinterpret_cast<const uint4*>(qkv + static_cast<size_t>(m) * width + c);
    __nv_bfloat16* dst;
    if (c < nq) dst = q + static_cast<size_t>(m) * nq + c;
    else if (c < nq + nkv) dst = k + static_cast<size_t>(m) * nkv + (c - nq);
    else dst = v + static_cast<size_t>(m) * nkv + (c - nq - nkv);
    *reinterpret_cast<uint4*>(dst) = w;
  }
}

// act[m][j] = silu(gu[m][j]) * gu[m][F + j], silu(g) = g / (1 + exp(-g)).
__global__ void __launch_bounds__(kThreads)
swiglu_kernel(const __nv_bfloat16* gu, __nv_bfloat16* act, int M, int F) {
  const long long total = static_cast<long long>(M) * F / 8;
  for (long long i = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * kThreads) {
    const int m = static_cast<int>(i / (F / 8));
    const int j = static_cast<int>(i % (F / 8)) * 8;
    float g[8], u[8], o[8];
    load8(gu + static_cast<size_t>(m) * 2 * F + j, g);
    load8(gu + static_cast<size_t>(m) * 2 * F + F + j, u);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = g[e] / (1.f + expf(-g[e])) * u[e];
    store8(act + static_cast<size_t>(m) * F + j, o);
  }
}

}  // namespace layer
}  // namespace idlm

using namespace idlm;

extern "C" idlm_status idlm_gated_lora_grouped(const void* x, const void* w, const void* lora_a,
                                               const void* lora_b, const uint8_t* row_gate,
                                               float lora_scale, int M, int K, int N, int r,
                                               int ngroups, const int* group_rows, void* y,
                                               void* workspace, size_t workspace_bytes,
                                               int32_t* status, void* stream);
extern "C" size_t idlm_gated_lora_grouped_workspace_size(int M, int K, int N, int r, int ngroups);
extern "C" size_t idlm_isd_attention_workspace_size(int C, int Hq, int Hkv, int D, int page_size,
                                                    int max_rows, int dtype);
extern "C" idlm_status idlm_isd_attention(
    const void* q, const void* k_new, const void* v_new, const void* k_cache, const void* v_cache,
    const int32_t* page_table, int max_pages, const int32_t* seq_lens, const int32_t* qo_indptr,
    int C, int T, int Hq, int Hkv, int D, int page_size, int num_pages, int max_rows,
    float sm_scale, int dtype, void* out, void* workspace, size_t workspace_bytes,
    int32_t* status, void* stream);

namespace {

struct LayerWs {
  size_t n1, qkv, q, k, v, att, o, h, n2, gu, act, d, gemm, attn, total;
  size_t gemm_bytes, attn_bytes;
};

bool valid_shape(const idlm_layer_weights* L) {
  return L && L->hidden > 0 && L->ffn > 0 && L->n_heads > 0 && L->n_kv_heads > 0 &&
         L->head_dim > 0 && L->n_heads % L->n_kv_heads == 0 && L->rank >= 0 &&
         L->hidden % 8 == 0 && L->ffn % 128 == 0 && (L->n_heads * L->head_dim) % 128 == 0 &&
         (L->n_kv_heads * L->head_dim) % 128 == 0;
}

LayerWs layer_ws(const idlm_layer_weights* L, int M, int C, int page_size, int max_rows) {
  const size_t H = L->hidden, F = L->ffn, nq = L->n_heads * L->head_dim,
               nkv = L->n_kv_heads * L->head_dim;
  const int r = L->rank;
  LayerWs w;
  size_t off = 0;
  auto put = [&](size_t bytes) {
    off = align_up(off, 256);
    const size_t at = off;
    off += bytes;
    return at;
  };
  w.n1 = put(M * H * 2);
  w.qkv = put(M * (nq + 2 * nkv) * 2);
  w.q = put(M * nq * 2);
  w.k = put(M * nkv * 2);
  w.v = put(M * nkv * 2);
  w.att = put(M * nq * 2);
  w.o = put(M * H * 2);
  w.h = put(M * H * 2);
  w.n2 = put(M * H * 2);
  w.gu = put(M * 2 * F * 2);
  w.act = put(M * F * 2);
  w.d = put(M * H * 2);
  w.gemm_bytes = std::max({idlm_gated_lora_grouped_workspace_size(M, H, nq + 2 * nkv, r, 3),
                           idlm_gated_lora_grouped_workspace_size(M, nq, H, r, 1),
                           idlm_gated_lora_grouped_workspace_size(M, H, 2 * F, r, 2),
                           idlm_gated_lora_grouped_workspace_size(M, F, H, r, 1)});
  w.gemm = put(w.gemm_bytes);
  w.attn_bytes = std::max<size_t>(
      idlm_isd_attention_workspace_size(C, L->n_heads, L->n_kv_heads, L->head_dim, page_size,
                                        max_rows, IDLM_BF16),
      256);
  w.attn = put(w.attn_bytes);
  w.total = align_up(off, 256);
  return w;
}

}  // namespace

extern "C" size_t idlm_risd_layer_workspace_size(const idlm_layer_weights* L, int M, int C,
                                                 int page_size, int max_rows) {
  if (!valid_shape(L) || M <= 0 || C <= 0 || page_size <= 0 || max_rows <= 0) return 0;
  return layer_ws(L, M, C, page_size, max_rows).total;
}

extern "C" idlm_status idlm_risd_layer(
    const idlm_layer_weights* L, const void* x, void* out, int M, const uint8_t* row_gate,
    const void* k_cache, const void* v_cache, const int32_t* page_table, int max_pages,
    const int32_t* seq_lens, const int32_t* qo_indptr, int C, int page_size, int num_pages,
    int max_rows, void* k_new_out, void* v_new_out, void* workspace, size_t workspace_bytes,
    int32_t* status, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!valid_shape(L)) return IDLM_ERR_INVALID_ARG;
  if (!x || !out || !row_gate || !k_cache || !v_cache || !page_table || !seq_lens || !qo_indptr ||
      !status || M <= 0 || C <= 0)
    return IDLM_ERR_INVALID_ARG;
  if (!L->w_qkv || !L->w_o || !L->w_gu || !L->w_down) return IDLM_ERR_INVALID_ARG;
  if (L->rank > 0 && (!L->a_qkv || !L->b_qkv || !L->a_o || !L->b_o || !L->a_gu || !L->b_gu ||
                      !L->a_down || !L->b_down))
    return IDLM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
    return IDLM_ERR_INVALID_ARG;
  const LayerWs w = layer_ws(L, M, C, page_size, max_rows);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return IDLM_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto at = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(ws + off); };
  const int H = L->hidden, F = L->ffn, nq = L->n_heads * L->head_dim,
            nkv = L->n_kv_heads * L->head_dim;
  const int r = L->rank;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return IDLM_ERR_CUDA;
  const int ew_grid = dev.sm_count * 4;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  __nv_bfloat16* k_new = k_new_out ? static_cast<__nv_bfloat16*>(k_new_out) : at(w.k);
  __nv_bfloat16* v_new = v_new_out ? static_cast<__nv_bfloat16*>(v_new_out) : at(w.v);

  auto gemm = [&](const void* xin, const void* wt, const void* a, const void* b, int K, int N,
                  int ngroups, const int* rows, void* y) {
    return idlm_gated_lora_grouped(xin, wt, a, b, row_gate, L->lora_scale, M, K, N, r, ngroups,
                                   rows, y, ws + w.gemm, w.gemm_bytes, status, stream);
  };
  idlm_status rc;
  layer::residual_rmsnorm_kernel<<<M, layer::kThreads, 0, stream>>>(
      xb, nullptr, nullptr, at(w.n1), static_cast<const __nv_bfloat16*>(L->norm1), H, L->rms_eps);
  if (cudaGetLastError() != cudaSuccess) return IDLM_ERR_CUDA;
  const int qkv_rows[3] = {nq, nkv, nkv};
  if ((rc = gemm(at(w.n1), L->w_qkv, L->a_qkv, L->b_qkv, H, nq + 2 * nkv, 3, qkv_rows, at(w.qkv))))
    return rc;
  layer::split_qkv_kernel<<<ew_grid, layer::kThreads, 0, stream>>>(at(w.qkv), at(w.q), k_new,
                                                                   v_new, M, nq, nkv);
  if (cudaGetLastError() != cudaSuccess) return IDLM_ERR_CUDA;
  if ((rc = idlm_isd_attention(at(w.q), k_new, v_new, k_cache, v_cache, page_table, max_pages,
                               seq_lens, qo_indptr, C, M, L->n_heads, L->n_kv_heads, L->head_dim,
                               page_size, num_pages, max_rows,
                               1.0f / sqrtf(static_cast<float>(L->head_dim)), IDLM_BF16,
                               at(w.att), ws + w.attn, w.attn_bytes, status, stream)))
    return rc;
  const int one_h[1] = {H};
  if ((rc = gemm(at(w.att), L->w_o, L->a_o, L->b_o, nq, H, 1, one_h, at(w.o)))) return rc;
  layer::residual_rmsnorm_kernel<<<M, layer::kThreads, 0, stream>>>(
      xb, at(w.o), at(w.h), at(w.n2), static_cast<const __nv_bfloat16*>(L->norm2), H, L->rms_eps);
  if (cudaGetLastError() != cudaSuccess) return IDLM_ERR_CUDA;
  const int gu_rows[2] = {F, F};
  if ((rc = gemm(at(w.n2), L->w_gu, L->a_gu, L->b_gu, H, 2 * F, 2, gu_rows, at(w.gu)))) return rc;
  layer::swiglu_kernel<<<ew_grid, layer::kThreads, 0, stream>>>(at(w.gu), at(w.act), M, F);
  if (cudaGetLastError() != cudaSuccess) return IDLM_ERR_CUDA;
  if ((rc = gemm(at(w.act), L->w_down, L->a_down, L->b_down, F, H, 1, one_h, at(w.d)))) return rc;
  layer::residual_rmsnorm_kernel<<<M, layer::kThreads, 0, stream>>>(
      at(w.h), at(w.d), static_cast<__nv_bfloat16*>(out), nullptr, nullptr, H, 0.f);
  return cuda_status(cudaGetLastError());
}
