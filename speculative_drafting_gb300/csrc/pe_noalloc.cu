// LM head + greedy argmax for callers that cannot allocate device memory.
//
// pe_argmax needs a caller-allocated workspace for its per-row argmax keys and
// status word.  Some callers cannot provide one: a serving engine that has
// already reserved all device memory for weights and KV cache and hands a
// plugin only a stream, or a runtime bound to a fixed memory plan it cannot
// grow.  pe_argmax_noalloc runs the same LM-head plan and argmax finalisation
// with that scratch in a file-scope __device__ array instead, so it allocates
// nothing.
//
// The array is global state: every GPU that loads this library holds it
// (PE_NOALLOC_MAX_ROWS 64-bit keys, 32 KiB) until the process exits.  Every call
// on a device shares it and it keeps the last call's contents, so each call
// clears the keys it uses before its kernels run, and calls that overlap on the
// GPU (concurrent streams) race and must not be issued.  This variant keeps no
// status word: device-side problems are not reported.
#include <mutex>

#include "pe_internal.h"
#include "pe_prep.h"

namespace {

static __device__ __align__(256) unsigned long long g_noalloc_scratch[PE_NOALLOC_MAX_ROWS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.  The cache assumes one CUDA
// context per device for the life of the process: after a cudaDeviceReset the
// cached address would be stale, so a caller that resets a device must not
// call this entry point on it again.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PE_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return PE_OK;
}

}  // namespace

extern "C" int pe_argmax_noalloc(pe_handle* h, const void* z, int n_rows, int32_t* draft_tokens,
                                 float* logits, void* stream) {
  using namespace pe;
  if (!h || !handle_has_layer(h) || !z || !draft_tokens || n_rows < 1) return PE_ERR_ARG;
  if (n_rows > PE_NOALLOC_MAX_ROWS) return PE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(z) & 15u) != 0) return PE_ERR_ARG;
  void* base = nullptr;
  int rc = scratch_address(&base);
  if (rc != PE_OK) return rc;
  unsigned long long* keys = static_cast<unsigned long long*>(base);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_zero_keys(keys, n_rows, st) != PE_OK) return PE_ERR_CUDA;
  const pe_dims& d = *handle_dims(h);
  Epilogue e;
  e.mode = EPI_ARGMAX;
  e.amax = keys;
  e.logits = logits;
  e.ld_logits = d.vocab;
  if (d.dtype == PE_DTYPE_BF16) {
    // the plan pe_argmax takes: K splits, where the plan makes any, add their
    // partial tiles inside a thread-block cluster, so they need no global scratch
    const TcPlan p = plan_gemm_tc(d.vocab, d.d, n_rows, 0, 0, handle_num_sms(h), true);
    rc = launch_gemm_tc(p, handle_lm_map(h), nullptr, z, nullptr, nullptr, e, nullptr, st);
  } else {
    rc = launch_gemm_f32(static_cast<const float*>(handle_w_lm(h)), nullptr,
                         static_cast<const float*>(z), d.vocab, d.d, n_rows, nullptr, e, st);
  }
  if (rc != PE_OK) return rc;
  return launch_argmax_finalize(keys, n_rows, draft_tokens, st);
}
