// cpattn_fwd_noalloc: the fused ring-attention forward for callers that cannot
// allocate device memory.
//
// cpattn_fwd needs a caller-provided workspace (error word, per-sample prefix
// and work list).  Some callers have no way to provide one: a plug-in running
// inside a host program that owns the whole device-memory budget through its
// own pool and forbids further allocations, or latency-critical code that
// must not call cudaMalloc/cudaFree because those calls can synchronise the
// device.  For them this entry point uses a fixed scratch array that lives in
// the library's own device image instead of a workspace argument.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes; every
// GPU that loads the library holds it until the process exits.  Host code
// cannot pass the array's name to a kernel (on the host that name is only a
// stand-in for the device symbol), so the first call on each device, with
// that device current, looks up its device address with cudaGetSymbolAddress
// and caches it.  Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>

#include "cpattn.h"
#include "kernels.h"

// Size of the fixed scratch: enough for the work list of any problem with
// T / 256 + B * max_cp below about 130,000 (for example a 16M-token batch).
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace cpattn {

namespace {

std::mutex g_scratch_mu;
std::unordered_map<int, void*> g_scratch_ptr;  // device ordinal -> address

// Device address of g_noalloc_scratch on the current device (set up once per
// device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CPATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  auto it = g_scratch_ptr.find(dev);
  if (it == g_scratch_ptr.end()) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return CPATTN_ERR_CUDA;
    it = g_scratch_ptr.emplace(dev, ptr).first;
  }
  *out = it->second;
  return CPATTN_OK;
}

}  // namespace

}  // namespace cpattn

using namespace cpattn;

extern "C" int cpattn_fwd_noalloc(const void* q, const void* k, const void* v,
                                  const int32_t* cu_seqlens,
                                  const int32_t* cp_size, int32_t num_seqs,
                                  int64_t total_tokens, int32_t max_seqlen,
                                  int32_t max_cp, int32_t num_heads,
                                  int32_t head_dim, float softmax_scale,
                                  int32_t causal, void* out, float* lse,
                                  int32_t* status, void* stream) {
  FwdArgs a{q, k, v, cu_seqlens, cp_size, num_seqs, total_tokens, max_seqlen,
            max_cp, num_heads, head_dim, softmax_scale, causal};
  int st = check_fwd(a);
  if (st != CPATTN_OK) return st;
  if (total_tokens > 0 && (out == nullptr || !aligned(out, 16)))
    return CPATTN_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return CPATTN_ERR_INVALID_ARG;
  if (status != nullptr && !aligned(status, 4)) return CPATTN_ERR_INVALID_ARG;
  // The fixed scratch must hold what cpattn_fwd's workspace would.
  const size_t need =
      ws_layout(total_tokens, num_seqs, num_heads, head_dim, max_cp, false).total;
  if (need > kNoAllocScratchBytes) return CPATTN_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != CPATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The schedule kernel clears the error word and the work-item count at the
  // start of every call, so nothing left by an earlier call is read.
  st = run_attention(a, false, 0, static_cast<__nv_bfloat16*>(out), lse,
                     nullptr, nullptr, nullptr, scratch, s);
  if (st != CPATTN_OK) return st;
  if (status != nullptr &&
      cudaMemcpyAsync(status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      s) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  return CPATTN_OK;
}
