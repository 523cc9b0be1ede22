// api.cu -- library information and host-tier registration.
//
// [P4] "3.14M Context on 3x 3090 ...", "No Need to Rewrite the Kernel": the
// host KV is allocated with anonymous mmap, page-locked with
// cudaHostRegister(ptr, n, PORTABLE | MAPPED), and kernels read it through the
// returned device pointer.
#include "common.cuh"

using namespace skv;

SKV_EXPORT int skv_version(void) { return 1; }

SKV_EXPORT const char* skv_status_string(int status) {
  switch (status) {
    case SKV_OK: return "ok";
    case SKV_EINVAL: return "invalid argument";
    case SKV_EUNSUPPORTED: return "unsupported configuration";
    case SKV_ECUDA: return "CUDA error";
    case SKV_ENOMEM: return "buffer too small";
    default: return "unknown status";
  }
}

SKV_EXPORT int skv_device_sm_count(void) { return sm_count(); }

SKV_EXPORT int skv_host_register(void* host, size_t bytes, void** dev_alias) {
  if (!host || !bytes || !dev_alias) return SKV_EINVAL;
  if (cudaHostRegister(host, bytes, cudaHostRegisterPortable | cudaHostRegisterMapped) != cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  if (cudaHostGetDevicePointer(dev_alias, host, 0) != cudaSuccess) {
    cudaGetLastError();
    cudaHostUnregister(host);
    return SKV_ECUDA;
  }
  return SKV_OK;
}

SKV_EXPORT int skv_host_unregister(void* host) {
  if (!host) return SKV_EINVAL;
  if (cudaHostUnregister(host) != cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  return SKV_OK;
}
