// Host helpers and the library-wide entry points (version, status text).
#include <mutex>

#include "host_util.h"

namespace idlm {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
unsigned long long g_ctx[kMaxDevices] = {};
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

bool current_device_info(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_info[dev].device != dev || g_ctx[dev] != ctx || ctx == 0) {
    DeviceInfo d;
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return false;
    g_info[dev] = d;
    g_ctx[dev] = ctx;
  }
  *out = g_info[dev];
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!get_current || !get_id) {
      void* f1 = nullptr;
      void* f2 = nullptr;
      cudaDriverEntryPointQueryResult q1, q2;
      if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
              cudaSuccess ||
          q1 != cudaDriverEntryPointSuccess ||
          cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
              cudaSuccess ||
          q2 != cudaDriverEntryPointSuccess) {
        (void)cudaGetLastError();
        return 0;
      }
      get_current = reinterpret_cast<GetCurrent>(f1);
      get_id = reinterpret_cast<GetId>(f2);
    }
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

bool encode_bf16_map(CUtensorMap* map, void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, gdim, gstride, bdim, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle_bytes == 0    ? CU_TENSOR_MAP_SWIZZLE_NONE
                   : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                   : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                         : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace idlm

extern "C" int idlm_version(void) { return 100; }

extern "C" const char* idlm_status_string(int s) {
  switch (s) {
    case IDLM_OK: return "ok";
    case IDLM_ERR_INVALID_ARG: return "invalid argument";
    case IDLM_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case IDLM_ERR_WORKSPACE: return "workspace missing or too small";
    case IDLM_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}
