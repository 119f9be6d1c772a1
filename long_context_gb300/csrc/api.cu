// Host side of the C ABI declared in include/cpattn.h: argument checks,
// workspace layout, TMA tensor maps and kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <unordered_map>

#include "cpattn.h"
#include "kernels.h"

namespace cpattn {

namespace {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct DeviceInfo {
  int num_sms = 0;
  int cc_major = 0;
  int cc_minor = 0;
};

std::mutex g_mu;
std::unordered_map<int, DeviceInfo> g_devices;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CPATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_devices.find(dev);
  if (it == g_devices.end()) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    it = g_devices.emplace(dev, d).first;
  }
  *out = it->second;
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return CPATTN_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return CPATTN_OK;
}

// Tensor map over a packed bf16 [T, H, D] tensor: dims (D, H, T), box
// (64, 1, 128) with 128-byte swizzle -- one 128-token x 64-feature slab of one
// head per copy, laid out as the tcgen05 128-byte-swizzle operand expects.
int make_qkv_map(CUtensorMap* map, const void* base, int64_t T, int H, int D) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T > 0 ? T : 1)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(H) * D * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CPATTN_OK : CPATTN_ERR_CUDA;
}

}  // namespace

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

int check_fwd(const FwdArgs& a) {
  if (a.B < 0 || a.T < 0 || a.H < 1 || a.max_cp < 1 || a.max_cp > kMaxCp)
    return CPATTN_ERR_INVALID_ARG;
  if (a.D != 64 && a.D != 128) return CPATTN_ERR_UNSUPPORTED;
  if (!(std::isfinite(a.scale) && a.scale > 0.f)) return CPATTN_ERR_INVALID_ARG;
  if (a.causal != 0 && a.causal != 1) return CPATTN_ERR_INVALID_ARG;
  if (a.T >= (int64_t(1) << 31) || a.H > 65535) return CPATTN_ERR_INVALID_ARG;
  if (a.T > 0 && (a.B < 1 || a.max_seqlen < 1)) return CPATTN_ERR_INVALID_ARG;
  if (a.cu == nullptr || !aligned(a.cu, 4)) return CPATTN_ERR_INVALID_ARG;
  if (a.cp != nullptr && !aligned(a.cp, 4)) return CPATTN_ERR_INVALID_ARG;
  if (a.T > 0) {
    if (a.q == nullptr || a.k == nullptr || a.v == nullptr) return CPATTN_ERR_INVALID_ARG;
    if (!aligned(a.q, 16) || !aligned(a.k, 16) || !aligned(a.v, 16)) return CPATTN_ERR_INVALID_ARG;
  }
  return CPATTN_OK;
}

// Builds the schedule and launches the attention kernel.
int run_attention(const FwdArgs& a, bool partials, int32_t num_steps,
                  __nv_bfloat16* out, float* lse, float* o_steps,
                  float* m_steps, float* l_steps, void* workspace,
                  cudaStream_t stream) {
  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != CPATTN_OK) return st;
  // The kernels are built for sm_103a only.
  if (dev.cc_major != 10 || dev.cc_minor != 3) return CPATTN_ERR_UNSUPPORTED;
  const WsLayout lay = ws_layout(a.T, a.B, a.H, a.D, a.max_cp, false);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);

  const long long grid = lay.max_items * a.H;
  if (grid > 0x7fffffffLL) return CPATTN_ERR_UNSUPPORTED;
  SchedParams sp;
  sp.cu_seqlens = a.cu;
  sp.cp_size = a.cp;
  sp.num_seqs = a.B;
  sp.num_heads = a.H;
  sp.total_tokens = a.T;
  sp.max_seqlen = a.max_seqlen;
  sp.max_cp = a.max_cp;
  sp.hdr = hdr;
  sp.first_cta = reinterpret_cast<int*>(ws + lay.prefix_off);
  sp.order = reinterpret_cast<int*>(ws + lay.items_off);
  sp.table = reinterpret_cast<CtaWork*>(ws + lay.table_off);
  sp.table_asc = nullptr;
  sp.max_ctas = grid;
  sp.rows_per_item = kRowsPerItem;
  if (launch_schedule(sp, stream) != cudaSuccess) return CPATTN_ERR_CUDA;
  if (a.T == 0 || a.B == 0) return CPATTN_OK;

  CUtensorMap tq, tk, tv;
  if (make_qkv_map(&tq, a.q, a.T, a.H, a.D) != CPATTN_OK ||
      make_qkv_map(&tk, a.k, a.T, a.H, a.D) != CPATTN_OK ||
      make_qkv_map(&tv, a.v, a.T, a.H, a.D) != CPATTN_OK)
    return CPATTN_ERR_CUDA;
  // O in the same layout (the fused epilogue stores full tiles with TMA);
  // the partials mode writes no O here, and takes Q's map as a placeholder.
  CUtensorMap to = tq;
  if (!partials && out != nullptr && make_qkv_map(&to, out, a.T, a.H, a.D) != CPATTN_OK)
    return CPATTN_ERR_CUDA;

  FwdParams fp;
  fp.table = sp.table;
  fp.num_heads = a.H;
  fp.num_steps = partials ? num_steps : a.max_cp;
  fp.causal = a.causal;
  fp.scale_log2 = a.scale * 1.4426950408889634f;
  fp.out = out;
  fp.lse = lse;
  fp.o_steps = o_steps;
  fp.m_steps = m_steps;
  fp.l_steps = l_steps;
  fp.total_tokens = a.T;
  fp.hdr = hdr;
  fp.num_sms = dev.num_sms;
  if (launch_attn(tq, tk, tv, to, fp, a.D, partials, grid, stream) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  return CPATTN_OK;
}

WsLayout ws_layout(int64_t T, int32_t B, int32_t H, int32_t D, int32_t max_cp,
                   bool with_partials) {
  WsLayout l;
  l.max_items = T / kRowsPerItem + static_cast<int64_t>(B) * max_cp + 1;
  size_t off = align_up(sizeof(WsHeader));
  l.prefix_off = off;
  off = align_up(off + sizeof(int) * (static_cast<size_t>(B) + 1));
  l.items_off = off;
  off = align_up(off + sizeof(int2) * static_cast<size_t>(l.max_items));
  l.table_off = off;
  off = align_up(off + sizeof(CtaWork) * static_cast<size_t>(l.max_items) * H);
  l.o_off = l.m_off = l.l_off = 0;
  if (with_partials) {
    const size_t rows = static_cast<size_t>(max_cp) * T * H;
    l.o_off = off;
    off = align_up(off + rows * D * sizeof(float));
    l.m_off = off;
    off = align_up(off + rows * sizeof(float));
    l.l_off = off;
    off = align_up(off + rows * sizeof(float));
  }
  l.total = off;
  return l;
}

}  // namespace cpattn

using namespace cpattn;

extern "C" size_t cpattn_fwd_workspace_size(int64_t total_tokens,
                                            int32_t num_seqs,
                                            int32_t num_heads, int32_t head_dim,
                                            int32_t max_cp, int32_t mode) {
  if (total_tokens < 0 || num_seqs < 0 || num_heads < 1 || max_cp < 1 ||
      max_cp > kMaxCp || (head_dim != 64 && head_dim != 128) ||
      (mode != CPATTN_MODE_FUSED && mode != CPATTN_MODE_UNFUSED))
    return 0;
  return ws_layout(total_tokens, num_seqs, num_heads, head_dim, max_cp,
                   mode == CPATTN_MODE_UNFUSED)
      .total;
}

extern "C" int cpattn_fwd(const void* q, const void* k, const void* v,
                          const int32_t* cu_seqlens, const int32_t* cp_size,
                          int32_t num_seqs, int64_t total_tokens,
                          int32_t max_seqlen, int32_t max_cp,
                          int32_t num_heads, int32_t head_dim,
                          float softmax_scale, int32_t causal, int32_t mode,
                          void* out, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream) {
  FwdArgs a{q, k, v, cu_seqlens, cp_size, num_seqs, total_tokens, max_seqlen,
            max_cp, num_heads, head_dim, softmax_scale, causal};
  int st = check_fwd(a);
  if (st != CPATTN_OK) return st;
  if (mode != CPATTN_MODE_FUSED && mode != CPATTN_MODE_UNFUSED)
    return CPATTN_ERR_INVALID_ARG;
  if (total_tokens > 0 && (out == nullptr || !aligned(out, 16)))
    return CPATTN_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return CPATTN_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, kAlign)) return CPATTN_ERR_INVALID_ARG;
  const bool unfused = mode == CPATTN_MODE_UNFUSED;
  const WsLayout lay = ws_layout(total_tokens, num_seqs, num_heads, head_dim,
                                 max_cp, unfused);
  if (workspace_bytes < lay.total) return CPATTN_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (!unfused)
    return run_attention(a, false, 0, static_cast<__nv_bfloat16*>(out), lse,
                         nullptr, nullptr, nullptr, workspace, s);
  float* o_steps = reinterpret_cast<float*>(ws + lay.o_off);
  float* m_steps = reinterpret_cast<float*>(ws + lay.m_off);
  float* l_steps = reinterpret_cast<float*>(ws + lay.l_off);
  st = run_attention(a, true, max_cp, nullptr, nullptr, o_steps, m_steps,
                     l_steps, workspace, s);
  if (st != CPATTN_OK || total_tokens == 0) return st;
  DeviceInfo dev;
  st = device_info(&dev);
  if (st != CPATTN_OK) return st;
  MergeParams mp{};
  mp.o_steps = o_steps;
  mp.m_steps = m_steps;
  mp.l_steps = l_steps;
  mp.num_steps = max_cp;
  mp.rows = total_tokens * num_heads;
  mp.out_bf16 = static_cast<__nv_bfloat16*>(out);
  mp.out_lse = lse;
  if (launch_merge(mp, head_dim, true, dev.num_sms, s) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  return CPATTN_OK;
}

extern "C" int cpattn_fwd_partials(
    const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
    const int32_t* cp_size, int32_t num_seqs, int64_t total_tokens,
    int32_t max_seqlen, int32_t max_cp, int32_t num_heads, int32_t head_dim,
    float softmax_scale, int32_t causal, int32_t num_steps, float* o_steps,
    float* m_steps, float* l_steps, void* workspace, size_t workspace_bytes,
    void* stream) {
  FwdArgs a{q, k, v, cu_seqlens, cp_size, num_seqs, total_tokens, max_seqlen,
            max_cp, num_heads, head_dim, softmax_scale, causal};
  int st = check_fwd(a);
  if (st != CPATTN_OK) return st;
  if (num_steps < max_cp || num_steps > kMaxCp) return CPATTN_ERR_INVALID_ARG;
  if (total_tokens > 0 &&
      (o_steps == nullptr || m_steps == nullptr || l_steps == nullptr ||
       !aligned(o_steps, 16) || !aligned(m_steps, 4) || !aligned(l_steps, 4)))
    return CPATTN_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, kAlign)) return CPATTN_ERR_INVALID_ARG;
  const WsLayout lay = ws_layout(total_tokens, num_seqs, num_heads, head_dim,
                                 max_cp, false);
  if (workspace_bytes < lay.total) return CPATTN_ERR_WORKSPACE_TOO_SMALL;
  return run_attention(a, true, num_steps, nullptr, nullptr, o_steps, m_steps,
                       l_steps, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" int cpattn_merge(const float* o_steps, const float* m_steps,
                            const float* l_steps, int32_t num_steps,
                            int64_t total_tokens, int32_t num_heads,
                            int32_t head_dim, float* out_o, float* out_m,
                            float* out_l, void* stream) {
  if (num_steps < 1 || num_steps > kMaxCp || total_tokens < 0 || num_heads < 1)
    return CPATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return CPATTN_ERR_UNSUPPORTED;
  if (total_tokens == 0) return CPATTN_OK;
  if (o_steps == nullptr || m_steps == nullptr || l_steps == nullptr ||
      out_o == nullptr)
    return CPATTN_ERR_INVALID_ARG;
  if (!aligned(o_steps, 16) || !aligned(out_o, 16) || !aligned(m_steps, 4) ||
      !aligned(l_steps, 4) || (out_m && !aligned(out_m, 4)) ||
      (out_l && !aligned(out_l, 4)))
    return CPATTN_ERR_INVALID_ARG;
  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != CPATTN_OK) return st;
  MergeParams mp{};
  mp.o_steps = o_steps;
  mp.m_steps = m_steps;
  mp.l_steps = l_steps;
  mp.num_steps = num_steps;
  mp.rows = total_tokens * num_heads;
  mp.out_o = out_o;
  mp.out_m = out_m;
  mp.out_l = out_l;
  if (launch_merge(mp, head_dim, false, dev.num_sms,
                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  return CPATTN_OK;
}

// ------------------------------------------------------------- backward --

namespace cpattn {
namespace {

constexpr int kBwdRows = 128;  // rows per backward work unit (one tile)

struct BwdLayout {
  size_t prefix_off, order_off, table_dq_off, table_kv_off, delta_off, total;
  int64_t max_items;
};

BwdLayout bwd_layout(int64_t T, int32_t B, int32_t H, int32_t max_cp) {
  BwdLayout l;
  l.max_items = T / kBwdRows + static_cast<int64_t>(B) * max_cp + 1;
  size_t off = align_up(sizeof(WsHeader));
  l.prefix_off = off;
  off = align_up(off + sizeof(int) * (static_cast<size_t>(B) + 1));
  l.order_off = off;
  off = align_up(off + sizeof(int) * (static_cast<size_t>(B) + 1));
  l.table_dq_off = off;
  off = align_up(off + sizeof(CtaWork) * static_cast<size_t>(l.max_items) * H);
  l.table_kv_off = off;
  off = align_up(off + sizeof(CtaWork) * static_cast<size_t>(l.max_items) * H);
  l.delta_off = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(T) * H);
  l.total = off;
  return l;
}

}  // namespace
}  // namespace cpattn

extern "C" size_t cpattn_bwd_workspace_size(int64_t total_tokens, int32_t num_seqs,
                                            int32_t num_heads, int32_t head_dim,
                                            int32_t max_cp) {
  if (total_tokens < 0 || num_seqs < 0 || num_heads < 1 || max_cp < 1 ||
      max_cp > kMaxCp || (head_dim != 64 && head_dim != 128))
    return 0;
  return bwd_layout(total_tokens, num_seqs, num_heads, max_cp).total;
}

extern "C" int cpattn_bwd(const void* q, const void* k, const void* v, const void* out,
                          const void* dout, const float* lse, const int32_t* cu_seqlens,
                          const int32_t* cp_size, int32_t num_seqs, int64_t total_tokens,
                          int32_t max_seqlen, int32_t max_cp, int32_t num_heads,
                          int32_t head_dim, float softmax_scale, int32_t causal, void* dq,
                          void* dk, void* dv, void* workspace, size_t workspace_bytes,
                          void* stream) {
  FwdArgs a{q, k, v, cu_seqlens, cp_size, num_seqs, total_tokens, max_seqlen,
            max_cp, num_heads, head_dim, softmax_scale, causal};
  int st = check_fwd(a);
  if (st != CPATTN_OK) return st;
  if (total_tokens > 0) {
    for (const void* ptr : {out, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                            static_cast<const void*>(dv)})
      if (ptr == nullptr || !aligned(ptr, 16)) return CPATTN_ERR_INVALID_ARG;
    if (lse == nullptr || !aligned(lse, 4)) return CPATTN_ERR_INVALID_ARG;
  }
  if (workspace == nullptr || !aligned(workspace, kAlign)) return CPATTN_ERR_INVALID_ARG;
  const BwdLayout lay = bwd_layout(total_tokens, num_seqs, num_heads, max_cp);
  if (workspace_bytes < lay.total) return CPATTN_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo dev;
  st = device_info(&dev);
  if (st != CPATTN_OK) return st;
  if (dev.cc_major != 10 || dev.cc_minor != 3) return CPATTN_ERR_UNSUPPORTED;
  const long long grid = lay.max_items * num_heads;
  if (grid > 0x7fffffffLL) return CPATTN_ERR_UNSUPPORTED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  float* delta = reinterpret_cast<float*>(ws + lay.delta_off);
  if (launch_bwd_delta(static_cast<const __nv_bfloat16*>(out),
                       static_cast<const __nv_bfloat16*>(dout), delta,
                       total_tokens * num_heads, head_dim, dev.num_sms, s) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  SchedParams sp;
  sp.cu_seqlens = cu_seqlens;
  sp.cp_size = cp_size;
  sp.num_seqs = num_seqs;
  sp.num_heads = num_heads;
  sp.total_tokens = total_tokens;
  sp.max_seqlen = max_seqlen;
  sp.max_cp = max_cp;
  sp.hdr = hdr;
  sp.first_cta = reinterpret_cast<int*>(ws + lay.prefix_off);
  sp.order = reinterpret_cast<int*>(ws + lay.order_off);
  sp.table = reinterpret_cast<CtaWork*>(ws + lay.table_dq_off);     // query blocks, costly first
  sp.table_asc = reinterpret_cast<CtaWork*>(ws + lay.table_kv_off); // key blocks, costly first
  sp.max_ctas = grid;
  sp.rows_per_item = kBwdRows;
  if (launch_schedule(sp, s) != cudaSuccess) return CPATTN_ERR_CUDA;
  if (total_tokens == 0 || num_seqs == 0) return CPATTN_OK;

  CUtensorMap tq, tk, tv, tdo;
  if (make_qkv_map(&tq, q, total_tokens, num_heads, head_dim) != CPATTN_OK ||
      make_qkv_map(&tk, k, total_tokens, num_heads, head_dim) != CPATTN_OK ||
      make_qkv_map(&tv, v, total_tokens, num_heads, head_dim) != CPATTN_OK ||
      make_qkv_map(&tdo, dout, total_tokens, num_heads, head_dim) != CPATTN_OK)
    return CPATTN_ERR_CUDA;
  BwdParams bp;
  bp.lse = lse;
  bp.delta = delta;
  bp.dq = static_cast<__nv_bfloat16*>(dq);
  bp.dk = static_cast<__nv_bfloat16*>(dk);
  bp.dv = static_cast<__nv_bfloat16*>(dv);
  bp.num_heads = num_heads;
  bp.causal = causal;
  bp.scale = softmax_scale;
  bp.scale_log2 = softmax_scale * 1.4426950408889634f;
  bp.hdr = hdr;
  bp.total_tokens = total_tokens;
  bp.table = sp.table_asc;
  if (launch_bwd_dkdv(tq, tk, tv, tdo, bp, head_dim, grid, s) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  bp.table = sp.table;
  if (launch_bwd_dq(tq, tk, tv, tdo, bp, head_dim, grid, s) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  return CPATTN_OK;
}

// ----------------------------------------------------------- decode CP --

extern "C" size_t cpattn_decode_workspace_size(int32_t num_seqs, int32_t num_heads,
                                               int32_t head_dim, int32_t cp) {
  if (num_seqs < 0 || num_heads < 1 || cp < 1 || cp > kMaxCp ||
      (head_dim != 64 && head_dim != 128))
    return 0;
  const size_t rows = static_cast<size_t>(cp) * num_seqs * num_heads;
  return align_up(rows * head_dim * sizeof(float)) + align_up(rows * sizeof(float)) + kAlign;
}

extern "C" int cpattn_decode_partials(const void* q, const void* k, const void* v,
                                      const int32_t* cu_seqlens, int32_t num_seqs,
                                      int64_t total_tokens, int32_t num_heads, int32_t head_dim,
                                      float softmax_scale, int32_t cp, float* o_steps,
                                      float* lse_steps, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || total_tokens >= (int64_t(1) << 31) ||
      num_heads < 1 || num_heads > 65535 || cp < 1 || cp > kMaxCp)
    return CPATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return CPATTN_ERR_UNSUPPORTED;
  if (!(std::isfinite(softmax_scale) && softmax_scale > 0.f)) return CPATTN_ERR_INVALID_ARG;
  if (num_seqs == 0) return CPATTN_OK;
  if (q == nullptr || cu_seqlens == nullptr || o_steps == nullptr || lse_steps == nullptr ||
      !aligned(q, 16) || !aligned(cu_seqlens, 4) || !aligned(o_steps, 16) ||
      !aligned(lse_steps, 4))
    return CPATTN_ERR_INVALID_ARG;
  if (total_tokens > 0 && (k == nullptr || v == nullptr || !aligned(k, 16) || !aligned(v, 16)))
    return CPATTN_ERR_INVALID_ARG;
  DecodeParams dp;
  dp.q = static_cast<const __nv_bfloat16*>(q);
  dp.k = static_cast<const __nv_bfloat16*>(k);
  dp.v = static_cast<const __nv_bfloat16*>(v);
  dp.cu_seqlens = cu_seqlens;
  dp.num_seqs = num_seqs;
  dp.num_heads = num_heads;
  dp.cp = cp;
  dp.total_tokens = total_tokens;
  dp.scale_log2 = softmax_scale * 1.4426950408889634f;
  dp.o_steps = o_steps;
  dp.lse_steps = lse_steps;
  return launch_decode_partials(dp, head_dim, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CPATTN_OK
             : CPATTN_ERR_CUDA;
}

static int merge_lse_common(const float* o_steps, const float* lse_steps, int32_t num_steps,
                            int64_t rows, int32_t head_dim, float* out_o,
                            __nv_bfloat16* out_bf16, float* out_lse, cudaStream_t stream) {
  DeviceInfo dev;
  const int st = device_info(&dev);
  if (st != CPATTN_OK) return st;
  MergeParams mp{};
  mp.o_steps = o_steps;
  mp.m_steps = lse_steps;
  mp.l_steps = nullptr;  // normalised partials: l_s = 1, m_s = lse_s
  mp.num_steps = num_steps;
  mp.rows = rows;
  mp.out_o = out_o;
  mp.out_bf16 = out_bf16;
  mp.out_lse = out_lse;
  return launch_merge(mp, head_dim, out_bf16 != nullptr, dev.num_sms, stream) == cudaSuccess
             ? CPATTN_OK
             : CPATTN_ERR_CUDA;
}

extern "C" int cpattn_merge_lse(const float* o_steps, const float* lse_steps, int32_t num_steps,
                                int64_t rows, int32_t head_dim, float* out_o, float* out_lse,
                                void* stream) {
  if (num_steps < 1 || num_steps > kMaxCp || rows < 0) return CPATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return CPATTN_ERR_UNSUPPORTED;
  if (rows == 0) return CPATTN_OK;
  if (o_steps == nullptr || lse_steps == nullptr || out_o == nullptr || !aligned(o_steps, 16) ||
      !aligned(lse_steps, 4) || !aligned(out_o, 16) || (out_lse && !aligned(out_lse, 4)))
    return CPATTN_ERR_INVALID_ARG;
  return merge_lse_common(o_steps, lse_steps, num_steps, rows, head_dim, out_o, nullptr, out_lse,
                          static_cast<cudaStream_t>(stream));
}

extern "C" int cpattn_decode(const void* q, const void* k, const void* v,
                             const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                             int32_t num_heads, int32_t head_dim, float softmax_scale, int32_t cp,
                             void* out, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream) {
  const size_t need = cpattn_decode_workspace_size(num_seqs, num_heads, head_dim, cp);
  if (need == 0) return (head_dim != 64 && head_dim != 128) ? CPATTN_ERR_UNSUPPORTED
                                                            : CPATTN_ERR_INVALID_ARG;
  if (num_seqs > 0 && (out == nullptr || !aligned(out, 16))) return CPATTN_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return CPATTN_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, kAlign)) return CPATTN_ERR_INVALID_ARG;
  if (workspace_bytes < need) return CPATTN_ERR_WORKSPACE_TOO_SMALL;
  const size_t rows = static_cast<size_t>(cp) * num_seqs * num_heads;
  float* o_steps = static_cast<float*>(workspace);
  float* lse_steps = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                              align_up(rows * head_dim * sizeof(float)));
  int st = cpattn_decode_partials(q, k, v, cu_seqlens, num_seqs, total_tokens, num_heads,
                                  head_dim, softmax_scale, cp, o_steps, lse_steps, stream);
  if (st != CPATTN_OK || num_seqs == 0) return st;
  return merge_lse_common(o_steps, lse_steps, cp, static_cast<int64_t>(num_seqs) * num_heads,
                          head_dim, nullptr, static_cast<__nv_bfloat16*>(out), lse,
                          static_cast<cudaStream_t>(stream));
}

extern "C" int cpattn_poll_error(const void* workspace, void* stream) {
  if (workspace == nullptr) return CPATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return CPATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  return word;
}

extern "C" const char* cpattn_status_string(int status) {
  switch (status) {
    case CPATTN_OK: return "ok";
    case CPATTN_ERR_INVALID_ARG: return "invalid argument";
    case CPATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case CPATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case CPATTN_ERR_PLAN_INFEASIBLE: return "plan infeasible";
    case CPATTN_ERR_CUDA: return "CUDA error";
    case CPATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case CPATTN_ERR_DEVICE_BOUNDS: return "device bounds check failed (debug build)";
    default: return "unknown status";
  }
}

extern "C" int cpattn_version(void) { return (0 << 16) | (1 << 8) | 0; }
