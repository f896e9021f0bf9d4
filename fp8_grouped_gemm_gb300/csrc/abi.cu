// Status strings, the per-device error word and host utilities of libmgq.
#include <cudaTypedefs.h>
#include <mutex>

#include "mgq_internal.h"

namespace {

// First device-side error since the last mgq_get_error (0 = none). A static
// device variable: every device that loads the library holds one int.
__device__ int g_mgq_error;

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices];
int g_sms[kMaxDevices];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool load_encode() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

}  // namespace

namespace mgq {

int* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mgq_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

bool encode_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch,
                       uint32_t box_inner, uint32_t box_outer) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!load_encode()) return false;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                    uint64_t pitch, uint32_t box_inner, uint32_t box_outer, bool sw128) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!load_encode()) return false;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mgq

extern "C" {

const char* mgq_status_string(int s) {
  switch (s) {
    case MGQ_OK: return "ok";
    case MGQ_ERR_INVALID_ARG: return "invalid argument";
    case MGQ_ERR_UNSUPPORTED: return "unsupported format or mode";
    case MGQ_ERR_CUDA: return "CUDA error";
    case MGQ_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MGQ_ERR_DEVICE_INDEX: return "expert index out of range";
    default: return "unknown status";
  }
}

int mgq_version(void) { return MGQ_VERSION; }

int mgq_get_error(void* stream, int* device_status) {
  if (!device_status) return MGQ_ERR_INVALID_ARG;
  int* p = mgq::error_word();
  if (!p) return MGQ_ERR_CUDA;
  cudaStream_t s = mgq::as_stream(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MGQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MGQ_ERR_CUDA;
  if (v != 0) {
    int zero = 0;
    if (cudaMemcpyAsync(p, &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess) return MGQ_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MGQ_ERR_CUDA;
  }
  *device_status = v;
  return MGQ_OK;
}

}  // extern "C"
