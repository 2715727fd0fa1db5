// pa_api.cu — library-wide entry points: status word, error text, version,
// and the host helpers shared by the kernels (SM count, TMA tensor maps).
#include "pa_common.cuh"

#include <cudaTypedefs.h>
#include <mutex>
#include <set>
#include <stdio.h>
#include <utility>

namespace pa {

static thread_local char g_host_msg[256] = "";

void note_host_error(const char* what) { snprintf(g_host_msg, sizeof(g_host_msg), "%s", what); }

bool ck(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return true;
  snprintf(g_host_msg, sizeof(g_host_msg), "%s: %s", what, cudaGetErrorString(e));
  return false;
}

cudaError_t launch_after(const void* kernel, dim3 grid, dim3 block, void** args, cudaStream_t stream) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelExC(&cfg, kernel, args) == cudaSuccess) return cudaSuccess;
    (void)cudaGetLastError();      // not accepted here: a plain launch
  }
  return cudaLaunchKernel(kernel, grid, block, args, 0, stream);
}

bool raise_smem_limit(const void* kernel, int dev) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({kernel, dev})) return true;
  int optin = 0;
  if (!ck(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
          "cudaDeviceGetAttribute(MaxSharedMemoryPerBlockOptin)"))
    return false;
  if (!ck(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin),
          "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)"))
    return false;
  done.insert({kernel, dev});
  return true;
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
    cache[dev] = n;
  }
  return cache[dev];
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_map(CUtensorMap* map, const void* base, pa_dtype dt, int rank, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box, bool swizzle128) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  const CUtensorMapDataType ty = dt == PA_F32         ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dt == PA_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(map, ty, rank,
                  const_cast<void*>(base), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace pa

extern "C" int pa_last_error(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  const unsigned a = pa::fetch_status_cache_ops();
  const unsigned b0 = pa::fetch_status_decode(), b1 = pa::fetch_status_decode_fp8(), b2 = pa::fetch_status_shared();
  const unsigned b = (b0 == 0xffffffffu || b1 == 0xffffffffu || b2 == 0xffffffffu) ? 0xffffffffu : (b0 | b1 | b2);
  const unsigned c = pa::fetch_status_prefill();
  const unsigned d = pa::fetch_status_selftest();
  if (a == 0xffffffffu || b == 0xffffffffu || c == 0xffffffffu || d == 0xffffffffu) return PA_ERR_CUDA;
  return (int)(a | b | c | d);
}

extern "C" const char* pa_strerror(int code) {
  switch (code) {
    case PA_OK: return "success";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_SHAPE: return "unsupported or inconsistent sizes";
    case PA_ERR_DTYPE: return "unknown element type";
    case PA_ERR_ALIGN: return "a K/V/Q/output pointer is not 16-byte aligned";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CUDA: return "a CUDA runtime call failed";
    case (int)PA_DEV_BAD_BLOCK: return "device: block id outside the pool";
    case (int)PA_DEV_BAD_SLOT: return "device: slot outside the pool";
    case (int)PA_DEV_BAD_LEN: return "device: context length outside its block-table row";
    case (int)PA_DEV_TIMEOUT: return "device: pipeline wait timed out";
    case (int)PA_DEV_BAD_GROUP: return "device: shared-prefix group descriptor inconsistent with the block tables";
    default: return code > 0 ? "device: several conditions (bitmask)" : "unknown error";
  }
}

extern "C" int pa_version(void) { return 100; }

extern "C" const char* pa_last_host_error(void) { return pa::g_host_msg; }
