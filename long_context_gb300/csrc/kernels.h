// Internal interface between the host library (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace cpattn {

// Geometry of the attention kernel.
constexpr int kBM = 128;               // query rows per Q tile (= TMEM lanes)
constexpr int kBN = 128;               // keys per KV tile
constexpr int kNQ = 2;                 // Q tiles per CTA, ping-ponged
constexpr int kRowsPerItem = kBM * kNQ;
constexpr int kThreads = 384;          // 2 softmax warpgroups + control WG
// Register split (setmaxnreg): the kernel is launched at kLaunchRegs per
// thread; the control warpgroup drops to kCtrlRegs and the two softmax
// warpgroups rise to kSoftmaxRegs.  The shares add up to the launch total:
// 384 * 168 = 256 * 224 + 128 * 56.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 224;
constexpr int kCtrlRegs = 56;
static_assert(kThreads * kLaunchRegs == 256 * kSoftmaxRegs + 128 * kCtrlRegs,
              "register split must match the launch allocation");
constexpr int kMaxCp = 64;

// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)                 WsHeader
//   [256, +4*(B+1))          first CTA of each sample (in schedule order)
//   [.., +8*max_items)       schedule order of the samples (B ints used)
//   [.., +16*max_items*H)    work table: one CtaWork per attention CTA
//   [.., ...)                unfused mode only: o_steps, m_steps, l_steps
struct WsHeader {
  int error;    // cpattn_status of the last kernels run on this workspace
  int n_items;  // CTAs of the attention grid that have work
  int pad[62];
};

struct WsLayout {
  size_t prefix_off, items_off, table_off, o_off, m_off, l_off, total;
  int64_t max_items;
};

// One attention CTA's work, written by the schedule kernel so that a CTA
// finds it with a single 16-byte load:
//   x = first token of the sample, y = sample length L,
//   z = (head << 8) | CP size c,  w = (query block << 8) | CP rank.
// (head < 2^16, c <= 64, rank < c, block < 2^23 since L < 2^31.)
using CtaWork = int4;

WsLayout ws_layout(int64_t T, int32_t B, int32_t H, int32_t D, int32_t max_cp,
                   bool with_partials);

struct SchedParams {
  const int* cu_seqlens;
  const int* cp_size;  // may be null: every sample at CP 1
  int num_seqs;
  int num_heads;
  long long total_tokens;
  int max_seqlen;
  int max_cp;
  WsHeader* hdr;
  int* first_cta;      // [B + 1]: first CTA of the sample at each order position
  int* order;          // [B]: samples by decreasing length
  CtaWork* table;      // [max_ctas]: work of each CTA (first n_items used)
  // Optional second table over the same items in the opposite order within
  // each (sample, head): increasing item index (null: not written).
  CtaWork* table_asc;
  long long max_ctas;  // grid size the host launches
  int rows_per_item;   // query (or key) rows per item
};

struct FwdParams {
  const CtaWork* table;  // [grid]: written by the schedule kernel
  int num_heads;
  int num_steps;        // ring steps walked: max_cp (fused) or S (partials)
  int causal;
  float scale_log2;     // softmax_scale * log2(e)
  __nv_bfloat16* out;   // fused: [T, H, D]
  float* lse;           // fused: [T, H] or null
  float* o_steps;       // partials: [S, T, H, D]
  float* m_steps;       // partials: [S, T, H]
  float* l_steps;
  long long total_tokens;
  WsHeader* hdr;
  int num_sms;          // CTA x_cta + num_sms is, in table order, a likely next CTA
};

// Backward kernels (attn_bwd.cu).  Gradients are bf16 [T, H, D]; `lse` is
// the forward's natural-log LSE [T, H]; `delta` = rowsum(dO * O) [T, H].
struct BwdParams {
  const CtaWork* table;  // this kernel's work table (written by the schedule kernel)
  const float* lse;
  const float* delta;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int num_heads;
  int causal;
  float scale;       // softmax scale (applied to dQ and dK at the end)
  float scale_log2;  // softmax scale * log2(e)
  WsHeader* hdr;
  long long total_tokens;  // T (bounds of the debug build's checks)
};

struct MergeParams {
  const float* o_steps;
  const float* m_steps;
  const float* l_steps;  // null: every l_s is 1 (normalised partials, m_s = their LSE)
  int num_steps;
  long long rows;       // T * H
  float* out_o;         // public merge: O / l in fp32
  float* out_m;
  float* out_l;
  __nv_bfloat16* out_bf16;  // unfused forward: O / l in bf16
  float* out_lse;           // m + ln l (written when not null)
};

// Host-side forward arguments and the launch sequence shared by the entry
// points (api.cu).
struct FwdArgs {
  const void *q, *k, *v;
  const int32_t *cu, *cp;
  int32_t B;
  int64_t T;
  int32_t max_seqlen, max_cp, H, D;
  float scale;
  int32_t causal;
};

bool aligned(const void* p, size_t a);

// Host-checkable argument rules of the forward calls; a cpattn_status.
int check_fwd(const FwdArgs& a);

// Schedule kernel + attention kernel on `stream`, using `workspace` (at least
// ws_layout(T, B, H, D, max_cp, false).total bytes) for the error word and the
// work list; a cpattn_status.
int run_attention(const FwdArgs& a, bool partials, int32_t num_steps,
                  __nv_bfloat16* out, float* lse, float* o_steps,
                  float* m_steps, float* l_steps, void* workspace,
                  cudaStream_t stream);

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t stream);

// Dynamic shared memory the attention kernel needs for head_dim D.
int attn_smem_bytes(int D);

cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p, int D,
                        bool partials, long long grid, cudaStream_t stream);

// Decode-time CP partials (decode.cu): q [B, H, D] bf16 (one new token per
// sequence), the KV cache k, v [T, H, D] bf16 packed by cu_seqlens [B + 1];
// shard s of sequence b is its keys [s*ceil(L/c), min((s+1)*ceil(L/c), L)).
// Outputs the normalised partials o_steps [c, B, H, D] and their natural-log
// LSE lse_steps [c, B, H] (an empty shard: 0 and -inf).
struct DecodeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int* cu_seqlens;
  int num_seqs, num_heads, cp;
  long long total_tokens;
  float scale_log2;
  float* o_steps;
  float* lse_steps;
};

cudaError_t launch_decode_partials(const DecodeParams& p, int D, cudaStream_t stream);


// delta[r] = sum_d dO[r, d] * O[r, d] for rows r < rows (= T * H).
cudaError_t launch_bwd_delta(const __nv_bfloat16* out, const __nv_bfloat16* dout,
                             float* delta, long long rows, int D, int num_sms,
                             cudaStream_t stream);

// dK/dV kernel (one CTA per 128-key tile) and dQ kernel (one CTA per 128-query
// tile); the four tensor maps are Q, K, V, dO.
cudaError_t launch_bwd_dkdv(const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const BwdParams& p, int D, long long grid, cudaStream_t stream);
cudaError_t launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo,
                          const BwdParams& p, int D, long long grid, cudaStream_t stream);

cudaError_t launch_merge(const MergeParams& p, int D, bool bf16_out,
                         int num_sms, cudaStream_t stream);

}  // namespace cpattn
