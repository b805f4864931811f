// wb_logmel_static: the log-mel front end for callers that cannot allocate
// device memory.
//
// Some hosts of this library cannot call cudaMalloc: a real-time audio
// thread must not block in the allocator (cudaMalloc may synchronize the
// device), and plugin hosts or serving runtimes that own every device buffer
// forbid allocations from the plugins they load.  Such a caller still needs
// scratch space for the log-mel pipeline (the split-precision padded audio,
// the DFT basis, the power spectrum, the per-chunk maxima), so this entry
// point takes it from one fixed array that lives in the library's own device
// image instead of from a caller-provided workspace.
//
// The array below is created on every device that loads the library and
// stays there until the process exits.  Its size caps one call at
// WB_LOGMEL_STATIC_MAX_CHUNKS chunks of 30 s.
#include <mutex>

#include "../../include/wb.h"
#include "internal.h"

namespace {

// Scratch for WB_LOGMEL_STATIC_MAX_CHUNKS chunks of wb_logmel (13,268,992 bytes at two chunks,
// rounded up to 13 MiB).  In host code the name stands for a host-side shadow, not a device
// address; the device address comes from cudaGetSymbolAddress below.
constexpr size_t kScratchBytes = 13u << 20;
static __device__ __align__(256) unsigned char g_logmel_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of this device's copy of the array, looked up once per device (with that
// device current) on its first call.
wb_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WB_ECUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_logmel_scratch) != cudaSuccess || !p) return WB_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return WB_OK;
}

}  // namespace

extern "C" wb_status wb_logmel_static(const float* audio, int64_t n_samples, int64_t chunk_stride, int n_chunks,
                                      int n_mels, float* out, void* stream) {
  if (n_chunks < 0 || n_chunks > WB_LOGMEL_STATIC_MAX_CHUNKS) return WB_EINVAL;
  if (n_chunks == 0) return WB_OK;
  const size_t need = wb_logmel_workspace_bytes(n_chunks, n_mels);
  if (need > kScratchBytes) return WB_EINVAL;
  void* scratch = nullptr;
  const wb_status st = scratch_for_current_device(&scratch);
  if (st != WB_OK) return st;
  // wb_logmel itself zeroes the per-chunk maxima it accumulates, so nothing the previous call
  // left in the array leaks into this one.
  return wb_logmel(audio, n_samples, chunk_stride, n_chunks, n_mels, out, scratch, kScratchBytes, stream);
}
