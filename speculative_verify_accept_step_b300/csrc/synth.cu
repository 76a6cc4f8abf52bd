// Synthetic logit rows for a stationary-batch decode loop: the stand-in for
// the language model's forward pass in the seeded workloads.  Nothing of the
// ISD step is computed here; the kernel only writes input rows.
//
// Every row predicts one slot (its position + 1, the logit shift of
// "Introspective Diffusion Language Models", section "Training").  A clean
// row of request c that predicts slot s holds z(c, s); a MASK row holds
// z(c, s) + sigma_c * e(c, s, step), so that a draft proposed from the MASK
// row at one step is verified against z(c, s) at the next, with the overlap
// sum_v min(p_v, q_v) set by sigma_c.
//
// Values: each of z and e is the Irwin-Hall sum of the eight 16-bit halves
// of one Philox4x32-10 output (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11), centred: S - 4 * 65535, an integer
// of magnitude <= 262140 (exact in fp32), with variance (2/3) 65536^2.
//   counter = (v, s, c, d), key = (seed, 0x1D1A7E5D); d = 0 for z, 1 + step
//   for e.
//   z = fp32(S_z) * scale_z            (one round to nearest)
//   x = z + fp32(S_e) * scale_e[c]     (two roundings to nearest, no fma)
// then one round to nearest-even into bf16.  scale_z and scale_e are fp32
// numbers chosen by the caller (logit_std * sqrt(1.5) / 65536 gives unit
// variance times logit_std).  The arithmetic is exact integer work followed
// by IEEE-rounded fp32 products and sums, so a CPU implementation of the same
// definition reproduces every bit.
#include <algorithm>

#include "common.cuh"
#include "host_util.h"

namespace idlm {
namespace synth {

constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
constexpr uint32_t kKey1 = 0x1D1A7E5Du;
constexpr int kThreads = 256;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint32_t hi0 = __umulhi(kM0, c.x), lo0 = kM0 * c.x;
    const uint32_t hi1 = __umulhi(kM1, c.z), lo1 = kM1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Centred Irwin-Hall sum of the eight 16-bit halves.
__device__ __forceinline__ int ih8(uint4 w) {
  const int s = static_cast<int>((w.x & 0xffffu) + (w.x >> 16) + (w.y & 0xffffu) + (w.y >> 16) +
                                 (w.z & 0xffffu) + (w.z >> 16) + (w.w & 0xffffu) + (w.w >> 16));
  return s - 4 * 65535;
}

struct Params {
  __nv_bfloat16* logits;     // [T, V]
  const int32_t* qo;         // [C+1]
  const int32_t* row_req;    // [T]
  const int32_t* row_pos;    // [T]
  const int32_t* row_token;  // [T], -1 at MASK rows
  const float* scale_e;      // [C]
  float scale_z;
  uint32_t seed;
  uint32_t step;
  int C, T, V, vec_per_row;
};

// One thread writes 8 consecutive values (one 16-byte store) of one row.
__global__ void __launch_bounds__(kThreads) synth_logits_kernel(const Params p) {
  const int T_used = min(p.T, p.qo[p.C]);
  const long long total = static_cast<long long>(T_used) * p.vec_per_row;
  for (long long i = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * kThreads) {
    const int row = static_cast<int>(i / p.vec_per_row);
    const int v0 = static_cast<int>(i % p.vec_per_row) * 8;
    const int c = p.row_req[row];
    if (c < 0 || c >= p.C) continue;   // not a request's row (the layout was invalid)
    const uint32_t slot = static_cast<uint32_t>(p.row_pos[row] + 1);
    const bool mask = p.row_token[row] < 0;
    const float se = mask ? p.scale_e[c] : 0.f;
    uint32_t out[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float x[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t v = static_cast<uint32_t>(v0 + 2 * h + e);
        const int sz = ih8(philox4x32_10(make_uint4(v, slot, static_cast<uint32_t>(c), 0u), p.seed, kKey1));
        float val = __fmul_rn(__int2float_rn(sz), p.scale_z);
        if (mask) {
          const int sn = ih8(philox4x32_10(make_uint4(v, slot, static_cast<uint32_t>(c), 1u + p.step),
                                           p.seed, kKey1));
          val = __fadd_rn(val, __fmul_rn(__int2float_rn(sn), se));
        }
        x[e] = val;
      }
      out[h] = pack_bf16x2(x[0], x[1]);
    }
    *reinterpret_cast<uint4*>(p.logits + static_cast<size_t>(row) * p.V + v0) =
        make_uint4(out[0], out[1], out[2], out[3]);
  }
}

}  // namespace synth
}  // namespace idlm

using namespace idlm;

extern "C" idlm_status idlm_synth_logits(void* logits, int C, int T, int V, const int32_t* qo_indptr,
                                         const int32_t* row_req, const int32_t* row_pos,
                                         const int32_t* row_token, float scale_z,
                                         const float* scale_e, uint32_t seed, uint32_t step,
                                         void* stream) {
  if (!logits || !qo_indptr || !row_req || !row_pos || !row_token || !scale_e)
    return IDLM_ERR_INVALID_ARG;
  if (C <= 0 || T <= 0 || V <= 0 || step == 0xffffffffu) return IDLM_ERR_INVALID_ARG;
  if (V % 8 || (reinterpret_cast<uintptr_t>(logits) & 15)) return IDLM_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return IDLM_ERR_CUDA;
  synth::Params p;
  p.logits = static_cast<__nv_bfloat16*>(logits);
  p.qo = qo_indptr;
  p.row_req = row_req;
  p.row_pos = row_pos;
  p.row_token = row_token;
  p.scale_e = scale_e;
  p.scale_z = scale_z;
  p.seed = seed;
  p.step = step;
  p.C = C;
  p.T = T;
  p.V = V;
  p.vec_per_row = V / 8;
  const long long work = static_cast<long long>(T) * p.vec_per_row;
  const int grid = static_cast<int>(std::min<long long>(
      (work + synth::kThreads - 1) / synth::kThreads, static_cast<long long>(dev.sm_count) * 8));
  synth::synth_logits_kernel<<<grid, synth::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cuda_status(cudaGetLastError());
}
