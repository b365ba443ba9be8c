// ekv_noalloc.cu — decode attention whose scratch lives in a fixed device array.
//
// ekv_decode_attn keeps its split-K partial results and merge tickets in
// scratch that ekv_create obtained through the caller's allocator.  Some
// callers cannot allocate device memory at all at the point where they need
// attention (for example a serving process that reserves every byte of device
// memory at start-up and forbids any later cudaMalloc, or a host library
// embedded in a runtime whose allocator is not reachable from it).  This file
// gives them ekv_decode_attn_noalloc: the same kernel and the same split
// schedule, with the scratch taken from one file-scope __device__ array instead.
//
// The array is a static global of the library: every GPU that loads the
// library holds EKV_NOALLOC_SCRATCH_BYTES of device memory until the process
// exits, and every call shares it.  Calls that overlap on the GPU (two streams,
// or two handles, at the same time) therefore race on it; serialize them.
#include <mutex>

#include "ekv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[EKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device.  The symbol name is only
// a host-side stand-in; the address comes from cudaGetSymbolAddress, looked up
// once per device with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" EKV_API int ekv_decode_attn_noalloc(ekv_cache* cache, int32_t layer, int32_t n_seqs,
                                               const int32_t* seq_slots, const void* q, void* o,
                                               void* stream) {
  using namespace ekv;
  DevState st;
  int splits = 0, vb = 0, pack = 1;
  // Same argument checks, split count and kernel as ekv_decode_attn.
  int rc = attn_plan(cache, layer, n_seqs, &st, &splits, &vb, &pack);
  if (rc != EKV_OK) return rc;
  if (n_seqs == 0) return EKV_OK;
  if (!seq_slots || !q || !o || (((uintptr_t)q | (uintptr_t)o) & 15)) return EKV_EINVAL;

  // Carve the array: [split numerators | split (max, sum) | merge tickets].
  const size_t parts = (size_t)n_seqs * st.Hkv * splits;
  const size_t acc_bytes = parts * MAX_G * st.D * sizeof(float);
  const size_t ml_bytes = parts * MAX_G * 2 * sizeof(float);
  const size_t tk_bytes = (size_t)n_seqs * st.Hkv * ATTN_TICKETS * sizeof(int32_t);
  const size_t acc_off = 0;
  const size_t ml_off = (acc_off + acc_bytes + 255) & ~(size_t)255;
  const size_t tk_off = (ml_off + ml_bytes + 255) & ~(size_t)255;
  if (tk_off + tk_bytes > (size_t)EKV_NOALLOC_SCRATCH_BYTES) return EKV_EINVAL;

  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return EKV_ECUDA;
  uint8_t* b = static_cast<uint8_t*>(base);
  st.attn_acc = reinterpret_cast<float*>(b + acc_off);
  st.attn_ml = reinterpret_cast<float*>(b + ml_off);
  st.attn_ticket = reinterpret_cast<int32_t*>(b + tk_off);
  st.attn_parts_cap = (int32_t)parts;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Each ticket returns to zero when the last CTA of its group arrives, so a
  // completed call leaves them clear; this clear only guards against a launch
  // that never completed (an aborted kernel would leave counts behind).
  if (cudaMemsetAsync(st.attn_ticket, 0, tk_bytes, s) != cudaSuccess) return EKV_ECUDA;
  cudaError_t e = launch_decode_attn(st, layer, n_seqs, seq_slots, static_cast<const __half*>(q),
                                     static_cast<__half*>(o), splits, vb, pack, s);
  return e == cudaSuccess ? EKV_OK : EKV_ECUDA;
}
