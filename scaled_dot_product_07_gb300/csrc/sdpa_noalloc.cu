// sdpa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory themselves.
//
// Who needs it: code that is handed only its input and output buffers by a
// host framework that owns all device memory (a plugin or callback whose
// rules forbid private cudaMalloc calls, because they would bypass the
// framework's pool and memory accounting), and latency-critical loops where
// an allocation -- which may synchronise the device -- is not acceptable.
// sdpa_bwd needs a scratch workspace (an fp32 dQ accumulator and two fp32
// row vectors); this entry point takes it from a fixed array compiled into
// the library instead of from the caller.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds SDPA_BWD_NOALLOC_SCRATCH_BYTES of it until the process exits.
// In host code its name is only a host-side stand-in, so the device address
// is looked up once per device with cudaGetSymbolAddress and passed on.
#include <mutex>

#include "../../include/sdpa.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[SDPA_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_bwd_scratch on the current device (looked up once per
// device, with that device current). nullptr on failure.
void* scratch_address() {
  static void* addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" sdpa_status sdpa_bwd_noalloc(const sdpa_tensor* dout, const sdpa_tensor* q,
                                        const sdpa_tensor* k, const sdpa_tensor* v,
                                        const sdpa_tensor* out, const float* lse,
                                        double dropout_p, int is_causal, uint64_t seed,
                                        uint64_t offset, float scale, sdpa_tensor* dq,
                                        sdpa_tensor* dk, sdpa_tensor* dv,
                                        sdpa_stream_t stream) {
  if (!q || !k) return SDPA_ERR_INVALID_ARG;
  const size_t need =
      sdpa_bwd_workspace_size(q->size[0], q->size[1], q->size[2], k->size[2], q->size[3]);
  if (need > static_cast<size_t>(SDPA_BWD_NOALLOC_SCRATCH_BYTES)) return SDPA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_address();
    if (!scratch) return SDPA_ERR_CUDA;
  }
  // The backward's first kernel overwrites every scratch byte it later reads
  // (it zeroes the dQ accumulator and writes both row vectors), so what an
  // earlier call left in the array does not matter.
  return sdpa_bwd(dout, q, k, v, out, lse, dropout_p, is_causal, seed, offset, scale, dq, dk, dv,
                  scratch, static_cast<size_t>(SDPA_BWD_NOALLOC_SCRATCH_BYTES), stream);
}
