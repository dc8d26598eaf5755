// Backward-over-backward for callers that cannot allocate device memory.
//
// Some callers of this library have no way to obtain device memory of their own:
// a plugin running inside a host application whose memory manager owns the whole
// device and forbids independent cudaMalloc calls, or a deployment with a fixed
// memory plan that rules out any allocation after start-up.  attn_bob needs a
// scratch workspace (one float4 of row statistics per (batch, head, row), the rows
// of each slice rounded up to an even count); this entry point supplies it from a
// file-scope device array instead, so the caller passes only its inputs and outputs.
//
// The array is a static device object: every GPU that loads this library holds
// its kStaticBobScratchBytes until the process exits.  With CUDA's lazy module
// loading (the default) that memory is committed when this file's module is first
// loaded on a device, which the set-up below triggers: the first call on a device.
// Host code sees the array's name only as a host-side stand-in, so its device
// address is looked up once per device with cudaGetSymbolAddress (that device
// current) and cached; the cache assumes the device is not reset while the
// library is in use.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "fbd.h"
#include "internal.h"

namespace {

constexpr size_t kStaticBobScratchBytes = size_t(16) << 20;  // 16 MiB: 1,048,576 rows of 16 bytes

static __device__ __align__(256) unsigned char g_bob_scratch[kStaticBobScratchBytes];

constexpr int kMaxDevices = 256;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Set-up, once per device: the device address of g_bob_scratch on the current device.
attn_status_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return fbd::set_last_error(ATTN_ERR_DEVICE, "attn_bob_static: no usable current CUDA device");
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bob_scratch);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return fbd::set_last_error(ATTN_ERR_DEVICE, "attn_bob_static: cudaGetSymbolAddress of the scratch array failed");
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_bob_static(const attn_desc_t* desc, const void* Q, const void* K, const void* V,
                                         const void* O, const void* dO, const float* lse, const void* gdQ,
                                         const void* gdK, const void* gdV, void* gQ, void* gK, void* gV,
                                         void* gdO, void* stream) {
  // The descriptor first, so that errors come in the order attn_bob reports them.
  attn_status_t s = fbd::validate_desc(desc);
  if (s != ATTN_OK) return s;
  const size_t need = attn_bob_workspace_bytes(desc, 0);  // plain BoB (no GProj)
  if (need > kStaticBobScratchBytes) {
    const long long np = (desc->N + 1) & ~static_cast<long long>(1);
    char msg[240];
    std::snprintf(msg, sizeof(msg),
                  "attn_bob_static: B*H*Np = %lld*%lld*%lld rows (Np = N rounded up to even) need %zu scratch "
                  "bytes; the static limit is %zu (1,048,576 rows); use attn_bob with a caller workspace",
                  static_cast<long long>(desc->B), static_cast<long long>(desc->H), np, need,
                  kStaticBobScratchBytes);
    return fbd::set_last_error(ATTN_ERR_WORKSPACE, msg);
  }
  // Set-up on the device's first call, an empty problem included (such a call serves
  // as the start-up call that loads the array; it launches nothing).
  void* scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != ATTN_OK) return s;
  return attn_bob(desc, Q, K, V, O, dO, lse, gdQ, gdK, gdV, gQ, gK, gV, gdO, 0, scratch, kStaticBobScratchBytes,
                  stream);
}
