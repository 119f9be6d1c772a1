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
// stand-in for the device symbol), so the first call in each CUDA context
// (normally one per device: the primary context), with that device current,
// looks up its device address with cudaGetSymbolAddress and caches it under
// the context.  A context created later -- for example after
// cudaDeviceReset, which loads the module anew and may place the array
// elsewhere -- gets its own lookup.  Nothing here calls cudaMalloc, cudaFree
// or any allocating library routine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>

#include "cpattn.h"
#include "kernels.h"

// Size of the fixed scratch.  It must hold the fused forward's workspace
// (ws_layout in api.cu): a 256-byte header, 4 (B + 1) bytes of per-sample
// prefix, and 8 + 16 H bytes per work item, each part rounded up to 256 bytes,
// with n_items = T / 256 + B * max_cp + 1.  So a problem fits when
//   256 + 4 (B + 1) + (8 + 16 H) n_items  (+ up to 768 bytes of rounding)
// stays within 1 MiB.  At H = 32 that is about 2,000 work items: for example
// a 16,384-token batch of 7 samples at max_cp 4 needs 93 items (49 KB), and
// the largest micro-batch of the 256-sample sweep (max_cp 8) 154 items
// (81 KB); one call over the whole sweep (4.4 M tokens) or over about 510K
// tokens at H = 32 is refused.  At H = 1 the limit is about 43,000 items.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace cpattn {

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

std::mutex g_scratch_mu;
CtxGetCurrentFn g_ctx_get_current = nullptr;
std::unordered_map<CUcontext, void*> g_scratch_ptr;  // CUDA context -> address

// Device address of g_noalloc_scratch in the current device's context (looked
// up once per context).
int scratch_address(void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_ctx_get_current == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return CPATTN_ERR_CUDA;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return CPATTN_ERR_CUDA;
  if (ctx != nullptr) {
    auto it = g_scratch_ptr.find(ctx);
    if (it != g_scratch_ptr.end()) {
      *out = it->second;
      return CPATTN_OK;
    }
  }
  // Set-up for this context: the runtime makes the current device's primary
  // context current here if this thread had none yet.
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
    return CPATTN_ERR_CUDA;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return CPATTN_ERR_CUDA;
  g_scratch_ptr[ctx] = ptr;
  *out = ptr;
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
