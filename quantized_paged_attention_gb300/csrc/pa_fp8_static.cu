// pa_decode_fp8_static: the fp8 decode step for callers that cannot allocate
// device memory. The partition partials, which pa_decode_fp8 keeps in a
// caller-supplied workspace, live here in one file-scope device array that
// every GPU loading the library holds until the process exits.
#include <mutex>

#include "qpa.h"
#include "common.cuh"
#include "qpa_internal.h"

// The shared scratch. Host code sees only a host-side stand-in under this
// name; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char qpa_fp8_static_scratch[QPA_FP8_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, qpa_fp8_static_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}
}  // namespace

extern "C" int pa_decode_fp8_static(const void* q, const uint8_t* kv_cache, const int32_t* block_table,
                                    const int32_t* seq_lens, const float* k_scale, const float* v_scale,
                                    int num_partitions, void* out, const qpa_fp8_desc* d, void* stream) {
  const size_t need = pa_decode_fp8_workspace_size(d, num_partitions);
  if (need == 0)   // invalid arguments or nothing to do: let the regular entry point report which
    return pa_decode_fp8(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions, out, d,
                         nullptr, 0, stream);
  if (need > QPA_FP8_STATIC_SCRATCH_BYTES) return QPA_ERR_WORKSPACE;
  void* ws = scratch_on_current_device();
  if (!ws) return QPA_ERR_CUDA;
  return pa_decode_fp8(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions, out, d, ws,
                       QPA_FP8_STATIC_SCRATCH_BYTES, stream);
}
