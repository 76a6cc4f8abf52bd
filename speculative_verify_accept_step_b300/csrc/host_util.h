// Host-side helpers shared by the entry points: device properties, TMA tensor
// map encoding through the driver entry point (no link against libcuda), and
// workspace carving.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/idlm.h"

namespace idlm {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int max_smem_optin = 0;
};

// Properties of the current device (cached per device ordinal).
bool current_device_info(DeviceInfo* out);

// cuTensorMapEncodeTiled, resolved once from the driver.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Unique id (cuCtxGetId) of the calling thread's current CUDA context, or 0
// if there is none or the driver does not report one.  Ids are never reused
// within a process, so a cache keyed on it goes stale neither after
// cudaDeviceReset nor under another context on the same device.
unsigned long long current_context_id();

// Encode a tiled bf16 tensor map with a 128-, 64- or 32-byte swizzle, or
// none (swizzle_bytes = 0).
// dims/strides are innermost first; strides (bytes) exclude dimension 0.
bool encode_bf16_map(CUtensorMap* map, void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes = 128);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Carve consecutive 256-byte aligned regions out of a workspace.
struct Carver {
  uint8_t* base;
  size_t used = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <class T>
  T* take(size_t count) {
    used = align_up(used, 256);
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += count * sizeof(T);
    return p;
  }
};

inline idlm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? IDLM_OK : IDLM_ERR_CUDA; }

// The LM-head GEMM of the fused LM-head + accept call (lora.cu): logits =
// H W^T in bf16, [T][V], and the softmax statistics of every logits row per
// 128-entry tile of the vocabulary, 16-byte records (max z, sum, max x,
// first argmax) at tile_stats[row * ceil(V / 128) + tile].
size_t lm_head_gemm_workspace(int T, int H, int V);
idlm_status lm_head_gemm(const void* h, const void* w, int T, int H, int V, void* logits,
                         void* workspace, size_t workspace_bytes, void* tile_stats, float s2,
                         int greedy, int32_t* status, cudaStream_t stream);

}  // namespace idlm
